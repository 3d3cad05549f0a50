"""GB300-native (sm_103a) quantization-aware attention (QAT attention).

The computation lives in the C-ABI library ``libqat_attn.so`` (hand-written CUDA);
``capi`` binds it with ctypes and ``attention`` wraps it for torch tensors and
autograd.  Importing this package does not load the library; the first call does,
and fails loudly if it has not been built.
"""

from .capi import (QUANT_NONE, QUANT_P_FP8E4M3_ROW_TILE64,  # noqa: F401
                   QUANT_P_FP8E4M3_ROW_TILE64_PAGE_BWD, QatError, Status)
from .attention import (QATAttention, attention, check_device_status,  # noqa: F401
                        qat_attention_backward, qat_attention_forward, qat_prepare_qkv,
                        qat_subtract_mean)
