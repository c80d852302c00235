"""Helpers shared by the GPU tests: host<->device views of raw bit patterns."""

import numpy as np
import torch

import oracle


def dev_words(a: np.ndarray, dev="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint32).view(np.int32)).to(dev)


def dev_bf16(a: np.ndarray, dev="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16)).to(dev).view(
        torch.bfloat16)


def host_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def host_words(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().cpu().numpy().view(np.uint32)


def poison_bf16(shape, dev="cuda") -> torch.Tensor:
    """bf16 buffer filled with a NaN payload no kernel produces (0x7FA5)."""
    return torch.full(shape, 0x7FA5, dtype=torch.int16, device=dev).view(torch.bfloat16)


POISON = 0x7FA5


def assert_gemv_parity(y: torch.Tensor, qw_h, st_h, x_h, rows=None):
    """Every (sampled) output within |y - y_ref| <= 2e-3 sum|w x| + ulp_bf16(y_ref)."""
    yb = host_bits(y)
    if rows is not None:
        yb = yb[:, rows]
        qw_h = qw_h[rows]
        st_h = st_h[rows]
    y_ref = oracle.gemv_ref(qw_h, st_h, x_h)
    a_ref = oracle.gemv_abs_ref(qw_h, st_h, x_h)
    bad = oracle.bound_violations(yb, y_ref, a_ref)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        detail = [(tuple(i), float(oracle.bf16_bits_to_f64(yb[tuple(i)])), float(y_ref[tuple(i)]),
                   float(a_ref[tuple(i)])) for i in idx]
        raise AssertionError(f"{int(bad.sum())} outputs outside the bound, e.g. {detail}")
    assert not np.any(yb == POISON), "unwritten outputs"
    return y_ref, a_ref
