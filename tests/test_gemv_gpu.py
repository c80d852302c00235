"""GPU parity of w4a16_gemv against the fp64 oracle (through the C ABI).

Bar: every output within |y - y_ref| <= 2e-3 * sum_k |w x| + one bf16 ulp of
y_ref; bit-exact where the result is a single rounding of an exact value.
"""

import numpy as np
import pytest
import torch

import oracle
from bit_weight_only_gemv_gb300 import lib, synth
from _helpers import (POISON, assert_gemv_parity, dev_bf16, dev_words, host_bits,
                      poison_bf16)

pytestmark = pytest.mark.gpu


def make(rng, n, k, m=1, step_scale=0.02 / 8):
    qw_h = synth.np_words(rng, (n, k // 8))
    st_h = synth.np_steps(rng, (n, k // 32), scale=step_scale)
    x_h = synth.np_x(rng, (m, k))
    return qw_h, st_h, x_h


def run(qw_h, st_h, x_h, pdl=False):
    n, k = qw_h.shape[0], qw_h.shape[1] * 8
    m = x_h.shape[0]
    qw, st, x = dev_words(qw_h), dev_bf16(st_h), dev_bf16(x_h)
    y = poison_bf16((m, n))
    ws = None
    need = lib.workspace_bytes(m, n, k)
    if need:
        ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib.gemv(qw, st, x, y=y, workspace=ws, status=status, pdl=pdl)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return y, ws


# Shapes spanning every tiling the plan picks (whole rows and K chunks, team
# sizes 8/16/32), several tiles and CTAs, ragged row and chunk tails, and the
# split-K path.
SHAPES = [
    (1, 32, 1), (7, 32, 1), (37, 96, 1), (16, 64, 1), (17, 2048, 1), (300, 2048, 1),
    (2048, 2048, 1), (129, 704, 1), (1000, 704, 1), (333, 2816, 1), (250, 5376, 1),
    (100, 8192, 1), (513, 8192, 1), (64, 21504, 1), (19, 65536, 1),
    (300, 2048, 2), (300, 2048, 3), (130, 2048, 4), (77, 2816, 5), (50, 1024, 8),
    (40, 5376, 32),
]


@pytest.mark.parametrize("n,k,m", SHAPES)
def test_gemv_matches_oracle(cuda_lib, n, k, m):
    rng = np.random.default_rng(n * 131 + k + m)
    qw_h, st_h, x_h = make(rng, n, k, m)
    y, _ = run(qw_h, st_h, x_h)
    assert_gemv_parity(y, qw_h, st_h, x_h)


def test_gemv_one_hot_is_bit_exact(cuda_lib):
    rng = np.random.default_rng(1)
    n, k = 333, 2816
    qw_h, st_h, _ = make(rng, n, k)
    w = oracle.dequant(qw_h, st_h)
    for kk in (0, 5, 31, 32, 1000, k - 1):
        x_h = np.zeros((1, k), np.uint16)
        x_h[0, kk] = 0x3F80
        y, _ = run(qw_h, st_h, x_h)
        assert np.array_equal(host_bits(y)[0], oracle.bf16_rne(w[:, kk]))


def test_gemv_code_eight_gives_zero_and_closed_form(cuda_lib):
    rng = np.random.default_rng(2)
    n, k = 200, 2048
    x_h = synth.np_x(rng, (1, k))
    st_h = synth.np_steps(rng, (n, k // 32))
    qw_h = np.full((n, k // 8), 0x88888888, np.uint32)
    y, _ = run(qw_h, st_h, x_h)
    assert np.all(host_bits(y) & 0x7FFF == 0)
    for c in (0, 3, 15):
        qw_c = np.full((n, k // 8), int(format(c, "x") * 8, 16), np.uint32)
        y, _ = run(qw_c, st_h, x_h)
        assert_gemv_parity(y, qw_c, st_h, x_h)


def test_gemv_is_deterministic_and_batch_rows_match(cuda_lib):
    rng = np.random.default_rng(3)
    n, k = 700, 5376
    qw_h, st_h, x_h = make(rng, n, k, 4)
    y4, _ = run(qw_h, st_h, x_h)
    y4b, _ = run(qw_h, st_h, x_h)
    assert torch.equal(y4.view(torch.int16), y4b.view(torch.int16))
    for m in range(4):
        y1, _ = run(qw_h, st_h, x_h[m:m + 1])
        assert np.array_equal(host_bits(y1)[0], host_bits(y4)[m])


def test_split_k_equals_unsplit_bitwise(cuda_lib):
    # N = 16, K = 21504 is planned with K slices; gemv_id over the same rows is
    # never split; the per-row arithmetic must not depend on the split.
    rng = np.random.default_rng(4)
    n, k = 16, 21504
    assert lib.plan(1, n, k)["slices"] > 1
    qw_h, st_h, x_h = make(rng, n, k)
    y, ws = run(qw_h, st_h, x_h)
    assert ws is not None and int(ws[:4].view(torch.int32).abs().sum()) == 0
    qw, st, x = dev_words(qw_h), dev_bf16(st_h), dev_bf16(x_h)
    ids = torch.zeros(1, dtype=torch.int32, device="cuda")
    y_id = lib.gemv_id(qw, st, ids, x, n, k, 1, n * k // 2, n * k // 16)
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(y), host_bits(y_id))
    assert_gemv_parity(y, qw_h, st_h, x_h)


def test_split_k_workspace_is_rearmed(cuda_lib):
    rng = np.random.default_rng(5)
    n, k = 64, 21504
    qw_h, st_h, x_h = make(rng, n, k)
    qw, st, x = dev_words(qw_h), dev_bf16(st_h), dev_bf16(x_h)
    need = lib.workspace_bytes(1, n, k)
    assert need > 0
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    ys = [lib.gemv(qw, st, x, workspace=ws) for _ in range(3)]
    torch.cuda.synchronize()
    for y in ys[1:]:
        assert torch.equal(y.view(torch.int16), ys[0].view(torch.int16))
    assert_gemv_parity(ys[0], qw_h, st_h, x_h)
    with pytest.raises(lib.W4Error) as ei:
        lib.gemv(qw, st, x, workspace=ws[:16])
    assert ei.value.name == "W4_ERR_WORKSPACE"


def test_gemv_wide_dynamic_range_and_extreme_steps(cuda_lib):
    rng = np.random.default_rng(6)
    n, k = 300, 2048
    qw_h = synth.np_words(rng, (n, k // 8))
    mags = 10.0 ** rng.uniform(-6, 4, size=(2, k))
    x_h = synth._to_bf16_bits(rng.choice([-1.0, 1.0], size=(2, k)) * mags)
    x_h[1, :64] = 0                       # an all-zero group
    st_h = synth._to_bf16_bits(10.0 ** rng.uniform(-30, 20, size=(n, k // 32)))
    y, _ = run(qw_h, st_h, x_h)
    assert_gemv_parity(y, qw_h, st_h, x_h)


def test_gemv_non_finite_activation_propagates(cuda_lib):
    rng = np.random.default_rng(7)
    n, k = 64, 2048
    qw_h, st_h, x_h = make(rng, n, k)
    x_h[0, 100] = 0x7F80                  # +inf
    y, _ = run(qw_h, st_h, x_h)
    y_ref = oracle.gemv_ref(qw_h, st_h, x_h)
    got = oracle.bf16_bits_to_f64(host_bits(y))
    assert np.array_equal(np.isfinite(got), np.isfinite(y_ref))


def test_gemv_pdl_flag_same_bits(cuda_lib):
    rng = np.random.default_rng(8)
    n, k = 1500, 2048
    qw_h, st_h, x_h = make(rng, n, k)
    qw, st, x = dev_words(qw_h), dev_bf16(st_h), dev_bf16(x_h)
    y0 = lib.gemv(qw, st, x)
    ys = []
    for _ in range(5):                    # back-to-back programmatic dependents
        ys.append(lib.gemv(qw, st, x, pdl=True))
    torch.cuda.synchronize()
    for y in ys:
        assert torch.equal(y.view(torch.int16), y0.view(torch.int16))


@pytest.mark.parametrize("m,n,k", [(1, 1500, 2048), (5, 300, 2048), (16, 2048, 2048),
                                   (1, 700, 21504)])
def test_prefetch_l2_same_bits(cuda_lib, m, n, k):
    # w4a16_gemv_prefetch_l2 changes timing only: the same bits as
    # w4a16_gemv on every path (CUDA cores with one and two launches, the
    # tensor-core small batch, split-K), whole and ragged ranges, and the
    # prefetched tensors are left as they were
    rng = np.random.default_rng(m * 7 + n + k)
    qw_h, st_h, x_h = make(rng, n, k, m)
    qw, st, x = dev_words(qw_h), dev_bf16(st_h), dev_bf16(x_h)
    nq, ns = dev_words(synth.np_words(rng, (900, 1024 // 8))), dev_bf16(
        synth.np_steps(rng, (900, 1024 // 32)))
    nq0, ns0 = nq.clone(), ns.clone()
    need = lib.workspace_bytes(m, n, k)
    ws = torch.zeros(max(need, 16), dtype=torch.uint8, device="cuda") if need else None
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    y0 = lib.gemv(qw, st, x, workspace=ws, status=status)
    for ranges in ([(nq, None), (ns, None)], [(nq, 1000), (ns, 37)], [(ns, 8)],
                   [(nq, None), (ns, None), (qw, None), (st, None)]):
        y = lib.gemv(qw, st, x, workspace=ws, status=status, pdl=True, l2_next=ranges)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.equal(y.view(torch.int16), y0.view(torch.int16))
    assert torch.equal(nq, nq0) and torch.equal(ns.view(torch.int16), ns0.view(torch.int16))


def test_gemv_unaligned_output_view_and_guard_band(cuda_lib):
    rng = np.random.default_rng(9)
    n, k = 100, 2048
    qw_h, st_h, x_h = make(rng, n, k)
    qw, st, x = dev_words(qw_h), dev_bf16(st_h), dev_bf16(x_h)
    big = poison_bf16((1, n + 3))
    y = big[:, 1:n + 1]                   # 2-byte aligned view inside a guard band
    assert y.is_contiguous() and y.data_ptr() % 4 == 2
    lib.gemv(qw, st, x, y=y)
    torch.cuda.synchronize()
    b = host_bits(big)[0]
    assert b[0] == POISON and np.all(b[n + 1:] == POISON)
    assert_gemv_parity(y, qw_h, st_h, x_h)


def test_merged_projection_rows_equal_separate_gemvs(cuda_lib):
    # q/k/v (and gate/up) read the same activation; stored row-concatenated
    # they run as one GEMV whose rows are bitwise those of the separate GEMVs
    rng = np.random.default_rng(10)
    k = 2048
    parts = [synth.np_words(rng, (n, k // 8)) for n in (2048, 512, 512)]
    steps = [synth.np_steps(rng, (n, k // 32)) for n in (2048, 512, 512)]
    x_h = synth.np_x(rng, (1, k))
    merged, _ = run(np.concatenate(parts), np.concatenate(steps), x_h)
    sep = [run(q, s_, x_h)[0] for q, s_ in zip(parts, steps)]
    assert np.array_equal(host_bits(merged), np.concatenate([host_bits(y) for y in sep], axis=1))


@pytest.mark.parametrize("m,n,k", [(1, 2048, 8192), (1, 300, 704), (2, 512, 2816),
                                   (4, 1000, 2048), (3, 77, 96), (1, 5376, 21504),
                                   (9, 300, 512)])
def test_silu_mul_gated_activation_matches_oracle(cuda_lib, m, n, k):
    """W4_FLAG_SILU_MUL: x rows are [gate K | up K]; the product takes
    h = silu(gate) * up formed while staging (fp32, staged as fp16 pairs)."""
    rng = np.random.default_rng(m * 13 + n + k)
    qw_h = synth.np_words(rng, (n, k // 8))
    st_h = synth.np_steps(rng, (n, k // 32))
    x_h = synth.np_x(rng, (m, 2 * k))
    y = poison_bf16((m, n))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    need = lib.workspace_bytes(m, n, k, "cuda")
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda") if need else None
    lib.gemv(dev_words(qw_h), dev_bf16(st_h), dev_bf16(x_h), y=y, workspace=ws, status=status,
             silu_mul=True)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    yb = host_bits(y)
    assert not np.any(yb == POISON)
    y_ref, a_ref = oracle.gemv_values_ref(qw_h, st_h, oracle.silu_mul_ref(x_h))
    assert oracle.within_bound(yb, y_ref, a_ref)


def test_merged_gate_up_feeds_the_gated_down_projection(cuda_lib):
    # the gated MLP of one decode step: merged gate/up GEMV, then the down
    # GEMV reading its [gate | up] output row directly
    rng = np.random.default_rng(90)
    hid, inter = 2048, 8192
    gu_q = synth.np_words(rng, (2 * inter, hid // 8))
    gu_s = synth.np_steps(rng, (2 * inter, hid // 32))
    dn_q = synth.np_words(rng, (hid, inter // 8))
    dn_s = synth.np_steps(rng, (hid, inter // 32))
    x_h = synth.np_x(rng, (1, hid))
    gu = lib.gemv(dev_words(gu_q), dev_bf16(gu_s), dev_bf16(x_h))
    y = lib.gemv(dev_words(dn_q), dev_bf16(dn_s), gu, silu_mul=True, pdl=True)
    torch.cuda.synchronize()
    y_ref, a_ref = oracle.gemv_values_ref(dn_q, dn_s, oracle.silu_mul_ref(host_bits(gu)))
    assert oracle.within_bound(host_bits(y), y_ref, a_ref)


# K whose groups do not split evenly: a short last chunk (37 and 13 groups
# with chunks of 4) and lane teams padded past the end of a row (101 and 443
# groups walked by 32 lanes); the generic kernel instantiation
RAGGED = [(300, 1184, 1), (129, 416, 3), (77, 3232, 1), (40, 14176, 2), (20, 65504, 1)]


@pytest.mark.parametrize("n,k,m", RAGGED)
def test_gemv_ragged_k_matches_oracle(cuda_lib, n, k, m):
    p = lib.plan(m, n, k)
    groups = k // 32
    lanes = -(-groups // p["team"])
    assert groups % p["team"] or lanes % p["chunk_steps"]     # the shape is ragged
    rng = np.random.default_rng(n + 3 * k + m)
    qw_h, st_h, x_h = make(rng, n, k, m)
    y, _ = run(qw_h, st_h, x_h)
    assert_gemv_parity(y, qw_h, st_h, x_h)
