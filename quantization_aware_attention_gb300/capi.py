"""ctypes binding of the C ABI in ``include/qat_attn.h`` (argument marshalling only).

Every function has the C name and argument order.  Tensor arguments may be torch
tensors (their ``data_ptr()`` is passed) or raw integer addresses; ``stream`` may be a
``torch.cuda.Stream``, a raw handle, or ``None`` for torch's current stream on the
current device.  Functions return the ``qat_status_t`` value as a ``Status``.
No computation happens here: the library's kernels do all of it, and a missing
library is an error, never a fallback.
"""

from __future__ import annotations

import ctypes
import enum
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libqat_attn.so")

# Every symbol include/qat_attn.h declares (checked by the CPU test suite).
EXPORTED = (
    "qat_attn_fwd",
    "qat_attn_bwd_workspace_bytes",
    "qat_attn_bwd",
    "qat_attn_bwd_noalloc",
    "qat_status_string",
    "qat_attn_device_status",
    "qat_debug_quant_tiles",
    "qat_debug_wait_timeout",
    "qat_channel_mean",
    "qat_fake_quant_tokens",
    "qat_attn_fwd_chunk",
    "qat_attn_merge",
    "qat_attn_bwd_smooth_k",
    "qat_subtract_mean",
    "qat_debug_set_wait_limit_us",
)


class Status(enum.IntEnum):
    OK = 0
    INVALID_ARG = 1
    UNSUPPORTED = 2
    CUDA = 3
    TIMEOUT = 4
    WORKSPACE = 5


QUANT_NONE = 0
QUANT_P_FP8E4M3_ROW_TILE64 = 1
QUANT_P_FP8E4M3_ROW_TILE64_PAGE_BWD = 2


class QatError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = Status(status)
        super().__init__(f"{what}: {qat_status_string(status)}" if what else qat_status_string(status))


_lib = None
_vp, _i, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t


def lib() -> ctypes.CDLL:
    """The loaded library (loaded once).  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it first "
                "(python -m quantization_aware_attention_gb300.build)")
        L = ctypes.CDLL(LIB_PATH)
        L.qat_attn_fwd.argtypes = [_vp] * 6 + [_i] * 5 + [_f, _i, _i, _vp]
        L.qat_attn_fwd.restype = _i
        L.qat_attn_bwd_workspace_bytes.argtypes = [_i] * 5
        L.qat_attn_bwd_workspace_bytes.restype = _sz
        L.qat_attn_bwd.argtypes = [_vp] * 9 + [_i] * 5 + [_f, _i, _i, _vp, _sz, _vp]
        L.qat_attn_bwd.restype = _i
        L.qat_attn_bwd_noalloc.argtypes = [_vp] * 9 + [_i] * 5 + [_f, _i, _i, _vp]
        L.qat_attn_bwd_noalloc.restype = _i
        L.qat_status_string.argtypes = [_i]
        L.qat_status_string.restype = ctypes.c_char_p
        L.qat_attn_device_status.argtypes = [_vp]
        L.qat_attn_device_status.restype = _i
        L.qat_debug_quant_tiles.argtypes = [_vp, _i, _i, _vp, _vp, _vp, _vp]
        L.qat_debug_quant_tiles.restype = _i
        L.qat_debug_wait_timeout.argtypes = [_i, _vp]
        L.qat_debug_wait_timeout.restype = _i
        L.qat_channel_mean.argtypes = [_vp, _vp] + [_i] * 4 + [_vp]
        L.qat_channel_mean.restype = _i
        L.qat_fake_quant_tokens.argtypes = [_vp] * 4 + [_i] * 4 + [_vp]
        L.qat_fake_quant_tokens.restype = _i
        L.qat_attn_fwd_chunk.argtypes = [_vp] * 6 + [_i] * 7 + [_f, _i, _vp]
        L.qat_attn_fwd_chunk.restype = _i
        L.qat_attn_merge.argtypes = [_vp] * 8 + [_i] * 4 + [_vp]
        L.qat_attn_merge.restype = _i
        L.qat_attn_bwd_smooth_k.argtypes = [_vp] * 10 + [_i] * 5 + [_f, _i, _i, _vp, _sz, _vp]
        L.qat_attn_bwd_smooth_k.restype = _i
        L.qat_subtract_mean.argtypes = [_vp] * 3 + [_i] * 4 + [_vp]
        L.qat_subtract_mean.restype = _i
        L.qat_debug_set_wait_limit_us.argtypes = [_i, _vp]
        L.qat_debug_set_wait_limit_us.restype = _i
        _lib = L
    return _lib


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s) -> int | None:
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def qat_status_string(status: int) -> str:
    return lib().qat_status_string(int(status)).decode()


def qat_attn_fwd(q, k, v, o_q, o_hp, lse, B, H, Nq, Nkv, D, sm_scale, causal, quant_mode,
                 stream=None) -> Status:
    return Status(lib().qat_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o_q), _ptr(o_hp), _ptr(lse),
                                     B, H, Nq, Nkv, D, float(sm_scale), int(causal),
                                     int(quant_mode), _stream(stream)))


def qat_attn_bwd_workspace_bytes(B, H, Nq, Nkv, D) -> int:
    return int(lib().qat_attn_bwd_workspace_bytes(B, H, Nq, Nkv, D))


def qat_attn_bwd(q, k, v, o_hp, lse, dO, dq, dk, dv, B, H, Nq, Nkv, D, sm_scale, causal,
                 quant_mode, workspace, workspace_bytes, stream=None) -> Status:
    return Status(lib().qat_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o_hp), _ptr(lse), _ptr(dO),
                                     _ptr(dq), _ptr(dk), _ptr(dv), B, H, Nq, Nkv, D,
                                     float(sm_scale), int(causal), int(quant_mode),
                                     _ptr(workspace), int(workspace_bytes), _stream(stream)))


def qat_attn_bwd_noalloc(q, k, v, o_hp, lse, dO, dq, dk, dv, B, H, Nq, Nkv, D, sm_scale, causal,
                         quant_mode, stream=None) -> Status:
    return Status(lib().qat_attn_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o_hp), _ptr(lse),
                                             _ptr(dO), _ptr(dq), _ptr(dk), _ptr(dv), B, H, Nq,
                                             Nkv, D, float(sm_scale), int(causal),
                                             int(quant_mode), _stream(stream)))


def qat_attn_bwd_smooth_k(q, k, v, o_hp, lse, dO, dq, dk, dv, k_mean, B, H, Nq, Nkv, D, sm_scale,
                          causal, quant_mode, workspace, workspace_bytes, stream=None) -> Status:
    return Status(lib().qat_attn_bwd_smooth_k(_ptr(q), _ptr(k), _ptr(v), _ptr(o_hp), _ptr(lse),
                                              _ptr(dO), _ptr(dq), _ptr(dk), _ptr(dv),
                                              _ptr(k_mean), B, H, Nq, Nkv, D, float(sm_scale),
                                              int(causal), int(quant_mode), _ptr(workspace),
                                              int(workspace_bytes), _stream(stream)))


def qat_subtract_mean(x, mean, out, B, H, N, D, stream=None) -> Status:
    return Status(lib().qat_subtract_mean(_ptr(x), _ptr(mean), _ptr(out), B, H, N, D,
                                          _stream(stream)))


def qat_debug_set_wait_limit_us(limit_us, stream=None) -> Status:
    return Status(lib().qat_debug_set_wait_limit_us(int(limit_us), _stream(stream)))


def qat_attn_device_status(stream=None) -> Status:
    return Status(lib().qat_attn_device_status(_stream(stream)))


def qat_debug_wait_timeout(limit_ms, stream=None) -> Status:
    return Status(lib().qat_debug_wait_timeout(limit_ms, _stream(stream)))


def qat_debug_quant_tiles(p, rows, cols, deq, scales, codes, stream=None) -> Status:
    return Status(lib().qat_debug_quant_tiles(_ptr(p), rows, cols, _ptr(deq), _ptr(scales),
                                              _ptr(codes), _stream(stream)))


def qat_channel_mean(x, mean, B, H, N, D, stream=None) -> Status:
    return Status(lib().qat_channel_mean(_ptr(x), _ptr(mean), B, H, N, D, _stream(stream)))


def qat_fake_quant_tokens(x, mean, out, scales, B, H, N, D, stream=None) -> Status:
    return Status(lib().qat_fake_quant_tokens(_ptr(x), _ptr(mean), _ptr(out), _ptr(scales), B, H,
                                              N, D, _stream(stream)))


def qat_attn_fwd_chunk(q, k, v, o_q, o_hp, lse, B, H, Nq, Nkv_total, kv_begin, kv_len, D,
                       sm_scale, quant_mode, stream=None) -> Status:
    return Status(lib().qat_attn_fwd_chunk(_ptr(q), _ptr(k), _ptr(v), _ptr(o_q), _ptr(o_hp),
                                           _ptr(lse), B, H, Nq, Nkv_total, kv_begin, kv_len, D,
                                           float(sm_scale), int(quant_mode), _stream(stream)))


def qat_attn_merge(o_q_acc, o_hp_acc, lse_acc, o_q_part, o_hp_part, lse_part, o_q_out, o_hp_out,
                   B, H, Nq, D, stream=None) -> Status:
    return Status(lib().qat_attn_merge(_ptr(o_q_acc), _ptr(o_hp_acc), _ptr(lse_acc),
                                       _ptr(o_q_part), _ptr(o_hp_part), _ptr(lse_part),
                                       _ptr(o_q_out), _ptr(o_hp_out), B, H, Nq, D,
                                       _stream(stream)))
