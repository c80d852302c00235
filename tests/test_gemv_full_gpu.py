"""GPU parity of w4a16_gemv at the full sizes of the decode workloads, through
the C ABI, in the launch configuration the benchmark times.

These launches hand their windows to the CTAs at run time (a window counter
per launch), so the tests also check that every row is written exactly as it
would be by a launch that owns a fixed share of rows:

* sampled rows against the fp64 oracle (|y - y_ref| <= 2e-3 sum|w x| + one
  bf16 ulp), no output left unwritten;
* the first and last rows bitwise equal to a small launch over just those
  rows (the per-row arithmetic depends on K alone);
* the counters re-armed: more launches than there are counter slots give the
  same bits every time.
"""

import numpy as np
import pytest
import torch

from bit_weight_only_gemv_gb300 import lib, synth
from _helpers import POISON, assert_gemv_parity, host_bits, host_words, poison_bf16

pytestmark = pytest.mark.gpu

# (N, K): lm_head of the hidden-2048 decoder, merged gate/up, down and lm_head
# of the hidden-5376 decoder
FULL = [(262144, 2048), (43008, 5376), (5376, 21504), (262144, 5376)]


def weights(n, k, seed):
    qw = synth.torch_words((n, k // 8), synth.seed_of(seed, 1), "cuda")
    st = synth.torch_steps((n, k // 32), synth.seed_of(seed, 2), "cuda")
    x = synth.torch_x((1, k), synth.seed_of(seed, 3), "cuda")
    return qw, st, x


def call(qw, st, x):
    n, k = qw.shape[0], qw.shape[1] * 8
    y = poison_bf16((x.shape[0], n))
    need = lib.workspace_bytes(x.shape[0], n, k)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda") if need else None
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib.gemv(qw, st, x, y=y, workspace=ws, status=status, pdl=True)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return y


@pytest.mark.parametrize("n,k", FULL)
def test_full_size_gemv_sampled_rows_and_edges(cuda_lib, n, k):
    assert lib.plan(1, n, k)["dynamic_windows"] == 1
    qw, st, x = weights(n, k, n + k)
    y = call(qw, st, x)
    yb = host_bits(y)
    assert not np.any(yb == POISON), "unwritten outputs"
    # sampled rows against the oracle, read back from the bytes the GPU used
    rng = np.random.default_rng(k)
    rows = np.unique(np.concatenate([rng.choice(n, 384, replace=False), [0, n - 1]]))
    qw_h = host_words(qw[rows])
    st_h = host_bits(st[rows])
    x_h = host_bits(x)
    assert_gemv_parity(y[:, rows], qw_h, st_h, x_h)
    # first and last rows: bitwise equal to a launch over just those rows
    for sl in (slice(0, 1000), slice(n - 777, n)):
        ys = call(qw[sl].contiguous(), st[sl].contiguous(), x)
        assert np.array_equal(host_bits(ys), yb[:, sl])


def test_window_counters_rearm_across_many_launches(cuda_lib):
    n, k = 65536, 2048
    assert lib.plan(1, n, k)["dynamic_windows"] == 1
    qw, st, x = weights(n, k, 99)
    ref = host_bits(call(qw, st, x))
    ys = [poison_bf16((1, n)) for _ in range(4)]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for i in range(1100):                       # more launches than counter slots
        lib.gemv(qw, st, x, y=ys[i % 4], status=status, pdl=True)
        if i % 275 == 274:
            torch.cuda.synchronize()
            assert np.array_equal(host_bits(ys[i % 4]), ref)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for y in ys:
        assert np.array_equal(host_bits(y), ref)


@pytest.mark.parametrize("m,n,k", [(2, 131072, 2048), (3, 65536, 5376), (4, 65536, 2048)])
def test_batched_rows_with_run_time_windows(cuda_lib, m, n, k):
    """Several activation rows (CUDA-core path) with windows handed out at run
    time: sampled rows against the oracle, and each activation row bitwise
    equal to the single-row call (the row arithmetic depends on K alone)."""
    assert lib.plan(m, n, k, path="cuda")["dynamic_windows"] == 1
    qw, st, _ = weights(n, k, 7 * m + k)
    x = synth.torch_x((m, k), synth.seed_of(m, k), "cuda")
    y = poison_bf16((m, n))
    lib.gemv(qw, st, x, y=y, pdl=True, path="cuda")
    torch.cuda.synchronize()
    yb = host_bits(y)
    assert not np.any(yb == POISON)
    rng = np.random.default_rng(m)
    rows = np.unique(np.concatenate([rng.choice(n, 192, replace=False), [0, n - 1]]))
    assert_gemv_parity(y[:, rows], host_words(qw[rows]), host_bits(st[rows]), host_bits(x))
    for i in range(m):
        yi = call(qw, st, x[i:i + 1].contiguous())
        assert np.array_equal(host_bits(yi)[0], yb[i])


# (M, N, K): the tensor-core small-batch kernel and the prompt GEMM on the
# merged gate/up and lm_head of the hidden-2048 decoder and the merged gate/up
# and down of the hidden-5376 decoder
FULL_BATCHED = [(16, 16384, 2048), (32, 262144, 2048), (8, 43008, 5376),
                (64, 5376, 21504), (256, 43008, 5376), (200, 16384, 2048)]


@pytest.mark.parametrize("m,n,k", FULL_BATCHED)
def test_full_size_tensor_core_paths(cuda_lib, m, n, k):
    """Batches of 8-256 activation rows at full size, on the path the plan
    picks (small-batch kernel up to 32 rows, prompt GEMM above): sampled rows
    against the oracle, no output unwritten, and the first and last weight
    rows bitwise equal to a launch over just those rows."""
    assert lib.plan(m, n, k)["path"] == (2 if m <= 32 else 3)
    qw, st, _ = weights(n, k, 3 * m + k)
    x = synth.torch_x((m, k), synth.seed_of(m + 1, k), "cuda")
    y = call(qw, st, x)
    yb = host_bits(y)
    assert not np.any(yb == POISON), "unwritten outputs"
    rng = np.random.default_rng(m + k)
    rows = np.unique(np.concatenate([rng.choice(n, 256, replace=False), [0, n - 1]]))
    assert_gemv_parity(y[:, rows], host_words(qw[rows]), host_bits(st[rows]), host_bits(x))
    for sl in (slice(0, 640), slice(n - 300, n)):
        ys = call(qw[sl].contiguous(), st[sl].contiguous(), x)
        assert np.array_equal(host_bits(ys), yb[:, sl])
