"""w4a16_gemv_static_scratch: the GEMV for callers that cannot allocate.

Some callers cannot call cudaMalloc: a host framework that owns every device
allocation, a latency-critical loop where allocating could synchronise the
device, a plain C caller with nowhere to keep a workspace.  For them the
split-K scratch lives in a fixed array inside the library.  This file checks,
through the C ABI, on shapes whose plan really uses that array (and on two
that need none), over three calls in a row (the array keeps the previous
call's contents):

* every output is within the acceptance bound of the fp64 oracle;
* the bits equal those of w4a16_gemv with a caller workspace, as the header
  promises;
* the calls allocate no device memory (torch's allocator and the driver's
  free-memory count are unchanged across them);
* the gated activation flag works as in w4a16_gemv;
* a shape needing more scratch than the array holds is refused before any
  work.

It is collected last and also runs on its own in a fresh process.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle
from bit_weight_only_gemv_gb300 import lib, synth
from _helpers import POISON, assert_gemv_parity, dev_bf16, dev_words, host_bits, poison_bf16

pytestmark = pytest.mark.gpu

STATIC_SCRATCH_BYTES = 256 << 10   # W4_STATIC_SCRATCH_BYTES in include/w4a16.h
FLAG_SILU_MUL = 8                  # W4_FLAG_SILU_MUL

# shapes whose plan splits K and so uses the array: CUDA-core split-K at 1-5
# activation rows, and the tensor-core small-batch kernel's split-K at 16 rows
USES_ARRAY = [(1, 16, 21504), (1, 64, 21504), (5, 40, 21504), (2, 300, 5376), (3, 100, 8192),
              (16, 300, 2048)]
# shapes that need no scratch (whole rows; the prompt GEMM)
NO_ARRAY = [(1, 2048, 2048), (100, 300, 2048)]


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _static_call(L, y, qw, st, x, M, N, K, status, flags=0):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return L.w4a16_gemv_static_scratch(_ptr(y), _ptr(qw), _ptr(st), _ptr(x), M, N, K,
                                       _ptr(status), flags, stream)


def _check(outs, y_ws, y_ref, a_ref):
    ref_bits = host_bits(y_ws)
    for y in outs:
        b = host_bits(y)
        assert not np.any(b == POISON), "outputs left unwritten"
        assert np.array_equal(b, ref_bits), "not the bits of w4a16_gemv"
        assert oracle.within_bound(b, y_ref, a_ref), "outside the oracle bound"


@pytest.mark.parametrize("m,n,k", USES_ARRAY + NO_ARRAY)
def test_static_scratch_equals_gemv_and_oracle(cuda_lib, m, n, k):
    L = cuda_lib
    need = lib.workspace_bytes(m, n, k)
    if (m, n, k) in USES_ARRAY:
        assert 0 < need <= STATIC_SCRATCH_BYTES, need     # the array is really used
    else:
        assert need == 0
    rng = np.random.default_rng(100 + m + n + k)
    qw_h = synth.np_words(rng, (n, k // 8))
    st_h = synth.np_steps(rng, (n, k // 32))
    x_h = synth.np_x(rng, (m, k))
    qw, st, x = dev_words(qw_h), dev_bf16(st_h), dev_bf16(x_h)
    ws = torch.zeros(max(need, 16), dtype=torch.uint8, device="cuda") if need else None
    y_ws = lib.gemv(qw, st, x, workspace=ws)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    # the outputs are made up front, so that only the calls run between the reads
    ys = [poison_bf16((m, n)) for _ in range(3)]
    torch.cuda.synchronize()
    assert lib.STATUS[_static_call(L, ys[0], qw, st, x, m, n, k, status)] == "W4_OK"
    torch.cuda.synchronize()
    alloc0, free0 = torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0]
    for y in ys[1:]:
        assert lib.STATUS[_static_call(L, y, qw, st, x, m, n, k, status)] == "W4_OK"
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated() == alloc0
    assert torch.cuda.mem_get_info()[0] == free0
    assert int(status.item()) == 0
    _check(ys, y_ws, oracle.gemv_ref(qw_h, st_h, x_h), oracle.gemv_abs_ref(qw_h, st_h, x_h))


@pytest.mark.parametrize("m,n,k", [(1, 64, 21504), (2, 300, 5376)])
def test_static_scratch_gated_activation(cuda_lib, m, n, k):
    # W4_FLAG_SILU_MUL: x rows are [gate K | up K], as in w4a16_gemv
    L = cuda_lib
    need = lib.workspace_bytes(m, n, k, "cuda")
    assert 0 < need <= STATIC_SCRATCH_BYTES
    rng = np.random.default_rng(200 + m + n + k)
    qw_h = synth.np_words(rng, (n, k // 8))
    st_h = synth.np_steps(rng, (n, k // 32))
    x_h = synth.np_x(rng, (m, 2 * k))
    qw, st, x = dev_words(qw_h), dev_bf16(st_h), dev_bf16(x_h)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    y_ws = lib.gemv(qw, st, x, workspace=ws, silu_mul=True)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ys = [poison_bf16((m, n)) for _ in range(2)]
    for y in ys:
        assert lib.STATUS[_static_call(L, y, qw, st, x, m, n, k, status, FLAG_SILU_MUL)] == "W4_OK"
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    y_ref, a_ref = oracle.gemv_values_ref(qw_h, st_h, oracle.silu_mul_ref(x_h))
    _check(ys, y_ws, y_ref, a_ref)


def test_static_scratch_runs_the_plain_plan_of_balanced_shapes(cuda_lib):
    # A tensor-core shape whose full-speed plan cuts tiles between CTAs
    # (balanced runs, their hand-over slots well beyond the fixed array)
    # runs the plain plan here: the same bits as w4a16_gemv with the full
    # workspace, within the oracle bound on sampled rows, no device memory
    # taken.
    L = cuda_lib
    m, n, k = 16, 39680, 1024
    assert lib.plan(m, n, k)["dynamic_windows"] == 1
    assert lib.workspace_bytes(m, n, k) > STATIC_SCRATCH_BYTES
    rng = np.random.default_rng(321)
    qw_h = synth.np_words(rng, (n, k // 8))
    st_h = synth.np_steps(rng, (n, k // 32))
    x_h = synth.np_x(rng, (m, k))
    qw, st, x = dev_words(qw_h), dev_bf16(st_h), dev_bf16(x_h)
    ws = torch.zeros(lib.workspace_bytes(m, n, k), dtype=torch.uint8, device="cuda")
    y_ws = lib.gemv(qw, st, x, workspace=ws)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = poison_bf16((m, n))
    torch.cuda.synchronize()
    before = torch.cuda.memory_allocated()
    assert lib.STATUS[_static_call(L, y, qw, st, x, m, n, k, status)] == "W4_OK"
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated() == before
    assert int(status.item()) == 0
    assert torch.equal(y.view(torch.int16), y_ws.view(torch.int16))
    rows = np.unique(np.concatenate([np.arange(0, n, 97), np.arange(n - 130, n)]))
    assert_gemv_parity(y, qw_h, st_h, x_h, rows=rows)


def test_static_scratch_refuses_shapes_beyond_the_array(cuda_lib):
    L = cuda_lib
    for m, n, k in [(4, 2000, 2208), (8, 256, 8192)]:    # CUDA-core and tensor-core plans
        assert lib.workspace_bytes(m, n, k) > STATIC_SCRATCH_BYTES
        qw = torch.zeros((n, k // 8), dtype=torch.int32, device="cuda")
        st = torch.zeros((n, k // 32), dtype=torch.bfloat16, device="cuda")
        x = torch.zeros((m, k), dtype=torch.bfloat16, device="cuda")
        y = poison_bf16((m, n))
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        assert lib.STATUS[_static_call(L, y, qw, st, x, m, n, k, status)] == "W4_ERR_WORKSPACE"
        torch.cuda.synchronize()
        assert np.all(host_bits(y) == POISON)   # nothing was enqueued
