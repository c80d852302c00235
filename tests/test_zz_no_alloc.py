"""w4a16_gemv_static_scratch: the GEMV for callers that cannot allocate.

Some callers cannot call cudaMalloc: a host framework that owns every device
allocation, a latency-critical loop where allocating could synchronise the
device, a plain C caller with nowhere to keep a workspace.  For them the
split-K scratch lives in a fixed array inside the library.  This file checks,
through the C ABI, that the call matches w4a16_gemv on shapes that use the
scratch, on two calls in a row (the array keeps the previous call's
contents), and that a shape needing more scratch than the array holds is
refused before any work.  It is collected last and also runs on its own.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle
from bit_weight_only_gemv_gb300 import lib, synth
from _helpers import POISON, dev_bf16, dev_words, host_bits, poison_bf16

pytestmark = pytest.mark.gpu

STATIC_SCRATCH_BYTES = 256 << 10   # W4_STATIC_SCRATCH_BYTES in include/w4a16.h


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _static_call(L, y, qw, st, x, M, N, K, status):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return L.w4a16_gemv_static_scratch(_ptr(y), _ptr(qw), _ptr(st), _ptr(x), M, N, K,
                                       _ptr(status), 0, stream)


@pytest.mark.parametrize("m,n,k", [(1, 16, 21504), (1, 64, 21504), (5, 40, 21504),
                                   (2, 300, 5376), (1, 2048, 2048), (16, 300, 2048),
                                   (100, 300, 2048)])
def test_static_scratch_matches_workspace_call(cuda_lib, m, n, k):
    L = cuda_lib
    rng = np.random.default_rng(100 + m + n + k)
    qw_h = synth.np_words(rng, (n, k // 8))
    st_h = synth.np_steps(rng, (n, k // 32))
    x_h = synth.np_x(rng, (m, k))
    qw, st, x = dev_words(qw_h), dev_bf16(st_h), dev_bf16(x_h)
    need = lib.workspace_bytes(m, n, k)
    assert need <= STATIC_SCRATCH_BYTES
    ws = torch.zeros(max(need, 16), dtype=torch.uint8, device="cuda") if need else None
    y_ref = lib.gemv(qw, st, x, workspace=ws)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = []
    for _ in range(2):                     # the array keeps the first call's contents
        y = poison_bf16((m, n))
        assert _static_call(L, y, qw, st, x, m, n, k, status) == 0
        outs.append(y)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref_bits = host_bits(y_ref)
    abs_sum = oracle.gemv_abs_ref(qw_h, st_h, x_h)
    ref_val = oracle.bf16_bits_to_f64(ref_bits)
    for y in outs:
        b = host_bits(y)
        assert not np.any(b == POISON)
        # within the parity tolerance of the workspace call's result
        assert oracle.within_bound(b, ref_val, abs_sum)


def test_static_scratch_refuses_shapes_beyond_the_array(cuda_lib):
    L = cuda_lib
    m, n, k = 4, 2000, 2208
    assert lib.workspace_bytes(m, n, k) > STATIC_SCRATCH_BYTES
    qw = torch.zeros((n, k // 8), dtype=torch.int32, device="cuda")
    st = torch.zeros((n, k // 32), dtype=torch.bfloat16, device="cuda")
    x = torch.zeros((m, k), dtype=torch.bfloat16, device="cuda")
    y = poison_bf16((m, n))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert lib.STATUS[_static_call(L, y, qw, st, x, m, n, k, status)] == "W4_ERR_WORKSPACE"
    torch.cuda.synchronize()
    assert np.all(host_bits(y) == POISON)   # nothing was enqueued
