"""Helpers of the GPU parity tests: device transfer of seeded bf16 inputs and error
measures.  Tolerances are relative L2 over a whole tensor: 5e-3 for O_hp and lse,
1e-2 for O_q, dQ, dK and dV."""

import numpy as np
import torch

from oracle import qat_oracle as orc

TOL_HP = 5e-3
TOL_Q = 1e-2


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    a = np.ascontiguousarray(bits).view(np.int16)
    return torch.from_numpy(a).to("cuda").view(torch.bfloat16)


def host_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def oracle_f64(inp: dict) -> dict:
    return {k: orc.bf16_bits_to_f64(v) for k, v in inp.items()}


def rel_l2(got, want) -> float:
    got = np.asarray(got, np.float64).ravel()
    want = np.asarray(want, np.float64).ravel()
    den = np.linalg.norm(want)
    return float(np.linalg.norm(got - want) / (den if den > 0 else 1.0))
