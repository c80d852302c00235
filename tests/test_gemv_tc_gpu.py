"""GPU parity of the tensor-core (tcgen05) path of w4a16_gemv against the fp64
oracle, through the C ABI.

The path is the default for 5 to 32 activation rows, and 3 to 4 rows of large
weights (K a multiple of 256), and
can be pinned at any M with the path flag.  Bar: every output within
|y - y_ref| <= 2e-3 * sum_k |w x| + one bf16 ulp of y_ref.
"""

import numpy as np
import pytest
import torch

import oracle
from bit_weight_only_gemv_gb300 import lib, synth
from _helpers import POISON, assert_gemv_parity, dev_bf16, dev_words, host_bits, poison_bf16

pytestmark = pytest.mark.gpu


def make(rng, n, k, m, step_scale=0.02 / 8):
    return (synth.np_words(rng, (n, k // 8)), synth.np_steps(rng, (n, k // 32), scale=step_scale),
            synth.np_x(rng, (m, k)))


def run(qw_h, st_h, x_h, path=None, pdl=False):
    n, k = qw_h.shape[0], qw_h.shape[1] * 8
    m = x_h.shape[0]
    qw, st, x = dev_words(qw_h), dev_bf16(st_h), dev_bf16(x_h)
    y = poison_bf16((m, n))
    need = lib.workspace_bytes(m, n, k, path)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda") if need else None
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib.gemv(qw, st, x, y=y, workspace=ws, status=status, pdl=pdl, path=path)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return y


# (n, k, m): one and several 128-row tiles, ragged last tile, K slices from one
# to many (split-K and not), 16 and 32 activation columns.
SHAPES = [
    (128, 256, 8), (300, 512, 8), (77, 256, 16), (640, 1024, 17), (2048, 2048, 16),
    (1000, 2048, 32), (129, 8192, 32), (4096, 2048, 8), (250, 5376, 24), (40, 21504, 9),
]


@pytest.mark.parametrize("n,k,m", SHAPES)
def test_tensor_core_path_matches_oracle(cuda_lib, n, k, m):
    assert lib.plan(min(m, 32), n, k)["path"] == 2
    rng = np.random.default_rng(n * 7 + k + m)
    qw_h, st_h, x_h = make(rng, n, k, m)
    y = run(qw_h, st_h, x_h)
    assert_gemv_parity(y, qw_h, st_h, x_h)


@pytest.mark.parametrize("m", [1, 2, 4])
def test_tensor_core_path_pinned_at_small_m(cuda_lib, m):
    rng = np.random.default_rng(40 + m)
    qw_h, st_h, x_h = make(rng, 384, 1024, m)
    y = run(qw_h, st_h, x_h, path="tensor")
    assert_gemv_parity(y, qw_h, st_h, x_h)


def test_cuda_core_path_pinned_at_large_m(cuda_lib):
    rng = np.random.default_rng(50)
    qw_h, st_h, x_h = make(rng, 300, 2048, 16)
    y = run(qw_h, st_h, x_h, path="cuda")
    assert_gemv_parity(y, qw_h, st_h, x_h)


@pytest.mark.parametrize("n,k,m", [(40900, 1024, 8), (39680, 1024, 16), (38990, 2048, 32),
                                   (43008, 5376, 16)])
def test_balanced_runs_equal_the_plain_plan(cuda_lib, n, k, m):
    # Row tiles that do not divide evenly over the CTAs: each CTA takes an
    # equal run of (tile, slice) work and a tile cut between two CTAs hands
    # its rows' running sums over.  With the full workspace the call runs
    # that plan, without it the plain one: the same bits, within the bound,
    # every output written (ragged last tile included), the workspace left
    # zero-filled, and again on a second call (the hand-over flags re-armed).
    p = lib.plan(m, n, k)
    assert p["path"] == 2 and p["dynamic_windows"] == 1
    rng = np.random.default_rng(n + k + m)
    qw_h, st_h, x_h = make(rng, n, k, m)
    qw, st, x = dev_words(qw_h), dev_bf16(st_h), dev_bf16(x_h)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    y0 = poison_bf16((m, n))
    lib.gemv(qw, st, x, y=y0, status=status)                 # no workspace: plain plan
    ws = torch.zeros(lib.workspace_bytes(m, n, k), dtype=torch.uint8, device="cuda")
    for _ in range(2):
        y = poison_bf16((m, n))
        lib.gemv(qw, st, x, y=y, workspace=ws, status=status, pdl=True)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.equal(y.view(torch.int16), y0.view(torch.int16))
        assert int(ws.count_nonzero().item()) == 0          # flags and prefix slots cleared
    rows = np.unique(np.concatenate([np.arange(0, n, max(1, n // 700)), np.arange(n - 200, n)]))
    assert_gemv_parity(y, qw_h, st_h, x_h, rows=rows)
    assert not np.any(host_bits(y) == POISON)


def test_tensor_core_rows_do_not_depend_on_n_or_split(cuda_lib):
    # The same 128 rows alone (16 K splits), among 8192 rows (4 splits) and
    # among 40960 rows (no split): the per-row association (groups in order
    # within 256-code slices, slices in order) must give the same bits.
    rng = np.random.default_rng(60)
    k, m = 4096, 16
    big_q, big_s, x_h = make(rng, 40960, k, m)
    splits = [lib.plan(m, n, k)["slices"] for n in (128, 8192, 40960)]
    assert splits[0] > splits[1] > splits[2] == 1
    outs = [host_bits(run(big_q[:n], big_s[:n], x_h))[:, :128] for n in (128, 8192, 40960)]
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])
    y = run(big_q[:128], big_s[:128], x_h)
    assert_gemv_parity(y, big_q[:128], big_s[:128], x_h)


def test_tensor_core_path_is_deterministic_and_rearms(cuda_lib):
    rng = np.random.default_rng(61)
    qw_h, st_h, x_h = make(rng, 256, 8192, 12)
    qw, st, x = dev_words(qw_h), dev_bf16(st_h), dev_bf16(x_h)
    need = lib.workspace_bytes(12, 256, 8192)
    assert need > 0
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    ys = [lib.gemv(qw, st, x, workspace=ws) for _ in range(3)]
    torch.cuda.synchronize()
    for y in ys[1:]:
        assert torch.equal(y.view(torch.int16), ys[0].view(torch.int16))
    assert int(ws[:4 * 2].view(torch.int32).abs().sum()) == 0    # counters re-armed
    assert_gemv_parity(ys[0], qw_h, st_h, x_h)


def test_tensor_core_path_dynamic_range_and_nonfinite(cuda_lib):
    rng = np.random.default_rng(62)
    n, k, m = 256, 1024, 8
    qw_h, st_h, x_h = make(rng, n, k, m)
    # steps over 40 decades, activations over 20
    st_h = oracle.bf16_rne(np.exp(rng.uniform(np.log(1e-20), np.log(1e20), size=st_h.shape)))
    xv = rng.standard_normal(x_h.shape) * np.exp(rng.uniform(-23, 23, size=x_h.shape))
    x_h = oracle.bf16_rne(xv)
    y = run(qw_h, st_h, x_h)
    assert_gemv_parity(y, qw_h, st_h, x_h)
    # an infinite step poisons its row, and only it
    st2 = st_h.copy()
    st2[5, 3] = 0x7F80
    y2 = run(qw_h, st2, x_h)
    ref = oracle.gemv_ref(qw_h, st2, x_h)
    got = oracle.bf16_bits_to_f64(host_bits(y2))
    assert np.array_equal(np.isfinite(got), np.isfinite(ref))


def test_tensor_core_pdl_chain(cuda_lib):
    rng = np.random.default_rng(63)
    qw_h, st_h, x_h = make(rng, 512, 2048, 8)
    qw, st, x = dev_words(qw_h), dev_bf16(st_h), dev_bf16(x_h)
    need = lib.workspace_bytes(8, 512, 2048)
    ws = torch.zeros(max(need, 16), dtype=torch.uint8, device="cuda")
    ys = [poison_bf16((8, 512)) for _ in range(4)]
    for y in ys:
        lib.gemv(qw, st, x, y=y, workspace=ws if need else None, pdl=True)
    torch.cuda.synchronize()
    for y in ys:
        assert not np.any(host_bits(y) == POISON)
        assert torch.equal(y.view(torch.int16), ys[0].view(torch.int16))
    assert_gemv_parity(ys[0], qw_h, st_h, x_h)


# one unit of all rows (4096 x 2048), and activation rows cut into tiles when
# the weight tiles are few, the last tile ragged (201 rows in 8 tiles of 26)
PROMPT_SHAPES = [(300, 2048, 64), (1000, 1024, 100), (256, 5376, 256), (129, 256, 33),
                 (200, 21504, 129), (4096, 2048, 256), (300, 1024, 201)]


@pytest.mark.parametrize("n,k,m", PROMPT_SHAPES)
def test_prompt_chunks_match_oracle(cuda_lib, n, k, m):
    """Prompt chunks (33 to 256 activation rows, one launch of the hi/lo-split
    GEMM): every output within the oracle bound, no output unwritten."""
    assert lib.plan(m, n, k)["path"] == 3
    rng = np.random.default_rng(n + k + m)
    qw_h, st_h, x_h = make(rng, n, k, m)
    y = run(qw_h, st_h, x_h)
    assert_gemv_parity(y, qw_h, st_h, x_h)


def test_prompt_rows_do_not_depend_on_m(cuda_lib):
    # the same activation row gives the same bits in chunks of 33, 100 and
    # 256 rows (different activation tiles and MMA widths)
    rng = np.random.default_rng(77)
    qw_h, st_h, x_h = make(rng, 384, 2048, 256)
    ref = host_bits(run(qw_h, st_h, x_h))
    for lo, hi in ((0, 33), (100, 200), (223, 256)):
        part = host_bits(run(qw_h, st_h, x_h[lo:hi]))
        assert np.array_equal(part, ref[lo:hi])


def test_prompt_extreme_values(cuda_lib):
    # steps over many decades and wide activations: the exact bf16 split
    # keeps every output within the bound
    rng = np.random.default_rng(78)
    qw_h, st_h, x_h = make(rng, 256, 1024, 48)
    st_h = oracle.bf16_rne(np.exp(rng.uniform(np.log(1e-20), np.log(1e20), size=st_h.shape)))
    x_h = oracle.bf16_rne(rng.standard_normal(x_h.shape) *
                          np.exp(rng.uniform(-23, 23, size=x_h.shape)))
    y = run(qw_h, st_h, x_h)
    assert_gemv_parity(y, qw_h, st_h, x_h)
    # an infinite step poisons its row, and only it
    st2 = st_h.copy()
    st2[5, 3] = 0x7F80
    ref = oracle.gemv_ref(qw_h, st2, x_h)
    got = oracle.bf16_bits_to_f64(host_bits(run(qw_h, st2, x_h)))
    assert np.array_equal(np.isfinite(got), np.isfinite(ref))


def test_prompt_chunks_on_cuda_cores(cuda_lib):
    # the CUDA-core path pinned at prompt size: 4 rows per launch
    rng = np.random.default_rng(79)
    qw_h, st_h, x_h = make(rng, 300, 2048, 40)
    yc = run(qw_h, st_h, x_h, path="cuda")
    assert_gemv_parity(yc, qw_h, st_h, x_h)
