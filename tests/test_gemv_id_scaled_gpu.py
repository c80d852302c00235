"""GPU parity of w4a16_gemv_id_scaled: routed GEMV whose outputs take
per-expert vectors indexed by the real expert id, while the weights may be
read through slot ids of a pool.

Page "Running a 26B MoE on an 8 GB Jetson by streaming experts from SSD",
section "Streaming without touching a single GPU kernel": only the expert
matmul may see slot ids; per-expert scales and biases keep the real ids; the
bar is bitwise identity with the full expert tensor.  Also here: the device
slot table kept by the pool catches slot ids fed where real ids belong, and a
full expert tensor held in host memory (read over the CPU-GPU link) fills the
pool with the same bytes.
"""

import numpy as np
import pytest
import torch

import oracle
from bit_weight_only_gemv_gb300 import lib, synth
from _helpers import POISON, dev_bf16, host_bits, poison_bf16

pytestmark = pytest.mark.gpu


def bf16_bits(rng, shape, lo=-2.0, hi=2.0):
    v = torch.from_numpy(rng.uniform(lo, hi, size=shape).astype(np.float32))
    return v.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def expert_set(rng, e, n, k):
    qw_h = synth.np_words(rng, (e, n, k // 8))
    st_h = synth.np_steps(rng, (e, n, k // 32))
    qw = torch.from_numpy(qw_h.view(np.int32).reshape(e, -1)).to("cuda")
    st = torch.from_numpy(st_h.view(np.int16).reshape(e, -1)).to("cuda").view(torch.bfloat16)
    return qw_h, st_h, qw, st


def status_word():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


@pytest.mark.parametrize("e,n,k,n_ids,x_rows,vec", [
    (6, 704, 2816, 8, 1, "both"), (6, 2816, 704, 8, 8, "both"), (5, 96, 704, 4, 4, "scale"),
    (5, 33, 2048, 5, 1, "bias"), (3, 100, 8192, 3, 3, "both"), (2, 40, 96, 1, 1, "both")])
def test_scaled_matches_oracle(cuda_lib, e, n, k, n_ids, x_rows, vec):
    rng = np.random.default_rng(e * 31 + n + k + n_ids)
    qw_h, st_h, qw, st = expert_set(rng, e, n, k)
    sc_h = bf16_bits(rng, (e, n)) if vec in ("both", "scale") else None
    bi_h = bf16_bits(rng, (e, n), -0.5, 0.5) if vec in ("both", "bias") else None
    ids_h = rng.integers(0, e, size=n_ids).astype(np.int32)
    x_h = synth.np_x(rng, (x_rows, k))
    ids = torch.from_numpy(ids_h).cuda()
    y = poison_bf16((n_ids, n))
    status = status_word()
    lib.gemv_id_scaled(qw, st, ids, dev_bf16(x_h), n, k, e, n * k // 2, n * k // 16, ids, e,
                       scale=None if sc_h is None else dev_bf16(sc_h),
                       bias=None if bi_h is None else dev_bf16(bi_h), y=y, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    yb = host_bits(y)
    assert not np.any(yb == POISON)
    y_ref, a_ref = oracle.gemv_id_scaled_ref(qw_h, st_h, ids_h, x_h, sc_h, bi_h)
    assert oracle.within_bound(yb, y_ref, a_ref)


@pytest.mark.parametrize("e,n,k,n_ids,x_rows", [(4, 72, 1184, 5, 5), (5, 136, 416, 6, 1),
                                                 (4, 40, 3232, 3, 1), (3, 24, 14176, 4, 4)])
def test_scaled_ragged_k_matches_oracle(cuda_lib, e, n, k, n_ids, x_rows):
    # K with a short last chunk (37, 13 groups) or a padded lane team (101,
    # 443 groups), real ids through a slot permutation with the slot table
    p = lib.plan(1, n, k)
    groups = k // 32
    assert groups % p["team"] or (-(-groups // p["team"])) % p["chunk_steps"]   # ragged
    rng = np.random.default_rng(e * 3 + n + k + n_ids)
    qw_h, st_h, qw, st = expert_set(rng, e, n, k)
    sc_h = bf16_bits(rng, (e, n))
    bi_h = bf16_bits(rng, (e, n), -0.5, 0.5)
    eids_h = rng.integers(0, e, size=n_ids).astype(np.int32)
    perm = rng.permutation(e).astype(np.int32)        # slot s holds expert perm[s]
    slot_of = np.argsort(perm).astype(np.int32)
    sids_h = slot_of[eids_h]
    qw_pool = qw[torch.from_numpy(perm).long().cuda()].contiguous()
    st_pool = st[torch.from_numpy(perm).long().cuda()].contiguous()
    x_h = synth.np_x(rng, (x_rows, k))
    y = poison_bf16((n_ids, n))
    status = status_word()
    lib.gemv_id_scaled(qw_pool, st_pool, torch.from_numpy(sids_h).cuda(), dev_bf16(x_h), n, k, e,
                       n * k // 2, n * k // 16, torch.from_numpy(eids_h).cuda(), e,
                       slot_expert=torch.from_numpy(perm).cuda(), scale=dev_bf16(sc_h),
                       bias=dev_bf16(bi_h), y=y, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    yb = host_bits(y)
    assert not np.any(yb == POISON)
    y_ref, a_ref = oracle.gemv_id_scaled_ref(qw_h, st_h, eids_h, x_h, sc_h, bi_h)
    assert oracle.within_bound(yb, y_ref, a_ref)


def test_no_vectors_is_bitwise_gemv_id(cuda_lib):
    rng = np.random.default_rng(5)
    e, n, k = 6, 704, 2816
    _, _, qw, st = expert_set(rng, e, n, k)
    ids = torch.from_numpy(rng.integers(0, e, size=8).astype(np.int32)).cuda()
    x = dev_bf16(synth.np_x(rng, (1, k)))
    a = lib.gemv_id(qw, st, ids, x, n, k, e, n * k // 2, n * k // 16)
    b = lib.gemv_id_scaled(qw, st, ids, x, n, k, e, n * k // 2, n * k // 16, ids, e)
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(a), host_bits(b))


@pytest.mark.parametrize("home", ["device", "pinned", "pageable"])
def test_pool_with_slot_table_is_bitwise_full_tensor(cuda_lib, home):
    """Weights through slot ids, vectors through real ids, slot table checked:
    every step bitwise equal to the full expert tensor; the table names what
    the host pool holds; the slots hold the source experts' bytes."""
    rng = np.random.default_rng(17)
    E, S, k_top = 32, 8, 4
    n, k = 704, 2816
    qs, ss = n * k // 2, n * k // 16
    full_q = synth.torch_words((E, qs // 4), seed=synth.seed_of(7, n), device="cuda")
    full_s = synth.torch_steps((E, ss // 2), seed=synth.seed_of(8, n), device="cuda")
    src_q, src_s = full_q, full_s
    if home != "device":
        src_q, src_s = full_q.cpu(), full_s.cpu()
        if home == "pinned":
            src_q, src_s = src_q.pin_memory(), src_s.pin_memory()
    sc = dev_bf16(bf16_bits(rng, (E, n)))
    bi = dev_bf16(bf16_bits(rng, (E, n), -0.25, 0.25))
    pool_q = torch.zeros((S, qs // 4), dtype=torch.int32, device="cuda")
    pool_s = torch.zeros((S, ss // 2), dtype=torch.bfloat16, device="cuda")
    table = torch.full((S,), -1, dtype=torch.int32, device="cuda")
    slot_ids = torch.zeros(k_top, dtype=torch.int32, device="cuda")
    eids = torch.zeros(k_top, dtype=torch.int32, device="cuda")
    pool = lib.SlotPool(E, S)
    ref_pool = oracle.LFUSlotPoolRef(E, S)
    x = dev_bf16(synth.np_x(rng, (1, k)))
    status = status_word()
    trace = synth.moe_trace(E, k_top, 30, 1.1, 0.7, seed=3)
    for req in trace:
        slots, _ = pool.stage(req, pool_q, src_q, qs, qs, pool_s, src_s, ss, ss, slot_ids,
                              slot_expert=table)
        want_slots, _ = ref_pool.step(req)
        assert slots == want_slots
        eids.copy_(torch.tensor(req, dtype=torch.int32))
        y_pool = poison_bf16((k_top, n))
        y_full = poison_bf16((k_top, n))
        lib.gemv_id_scaled(pool_q, pool_s, slot_ids, x, n, k, S, qs, ss, eids, E,
                           slot_expert=table, scale=sc, bias=bi, y=y_pool, status=status)
        lib.gemv_id_scaled(full_q, full_s, eids, x, n, k, E, qs, ss, eids, E,
                           scale=sc, bias=bi, y=y_full, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert host_bits(y_pool).tobytes() == host_bits(y_full).tobytes()
        assert table.cpu().tolist() == ref_pool.expert_in_slot
    for s_, ex in enumerate(ref_pool.expert_in_slot):
        if ex >= 0:
            assert torch.equal(pool_q[s_], full_q[ex]) and torch.equal(pool_s[s_], full_s[ex])


def test_slot_ids_fed_as_real_ids_are_caught(cuda_lib):
    rng = np.random.default_rng(19)
    E, S, k_top = 16, 4, 3
    n, k = 96, 704
    qs, ss = n * k // 2, n * k // 16
    full_q = synth.torch_words((E, qs // 4), seed=41, device="cuda")
    full_s = synth.torch_steps((E, ss // 2), seed=42, device="cuda")
    pool_q = torch.zeros((S, qs // 4), dtype=torch.int32, device="cuda")
    pool_s = torch.zeros((S, ss // 2), dtype=torch.bfloat16, device="cuda")
    table = torch.full((S,), -1, dtype=torch.int32, device="cuda")
    slot_ids = torch.zeros(k_top, dtype=torch.int32, device="cuda")
    pool = lib.SlotPool(E, S)
    req = [9, 12, 5]                      # experts >= S: no slot index names its own expert
    pool.stage(req, pool_q, full_q, qs, qs, pool_s, full_s, ss, ss, slot_ids, slot_expert=table)
    sc = dev_bf16(bf16_bits(rng, (E, n)))
    x = dev_bf16(synth.np_x(rng, (1, k)))
    # with the slot table: every row refused, none written
    y = poison_bf16((k_top, n))
    status = status_word()
    lib.gemv_id_scaled(pool_q, pool_s, slot_ids, x, n, k, S, qs, ss, slot_ids, E,
                       slot_expert=table, scale=sc, y=y, status=status)
    torch.cuda.synchronize()
    assert lib.STATUS[int(status.item())] == "W4_ERR_OWNER"
    assert np.all(host_bits(y) == POISON)
    # without it the mistake goes through, and the memcmp bar sees it
    eids = torch.tensor(req, dtype=torch.int32, device="cuda")
    bad = lib.gemv_id_scaled(pool_q, pool_s, slot_ids, x, n, k, S, qs, ss, slot_ids, E, scale=sc)
    good = lib.gemv_id_scaled(full_q, full_s, eids, x, n, k, E, qs, ss, eids, E, scale=sc)
    torch.cuda.synchronize()
    assert host_bits(bad).tobytes() != host_bits(good).tobytes()


def test_bad_real_ids_leave_rows_unwritten(cuda_lib):
    rng = np.random.default_rng(23)
    e, n, k = 4, 64, 2048
    qw_h, st_h, qw, st = expert_set(rng, e, n, k)
    sc_h = bf16_bits(rng, (e, n))
    ids_h = np.array([1, 2, 3, 0], np.int32)
    eids_h = np.array([1, 4, 3, -2], np.int32)
    x_h = synth.np_x(rng, (1, k))
    y = poison_bf16((4, n))
    status = status_word()
    lib.gemv_id_scaled(qw, st, torch.from_numpy(ids_h).cuda(), dev_bf16(x_h), n, k, e,
                       n * k // 2, n * k // 16, torch.from_numpy(eids_h).cuda(), e,
                       scale=dev_bf16(sc_h), y=y, status=status)
    torch.cuda.synchronize()
    assert lib.STATUS[int(status.item())] == "W4_ERR_INDEX"
    yb = host_bits(y)
    assert np.all(yb[1] == POISON) and np.all(yb[3] == POISON)
    y_ref, a_ref = oracle.gemv_id_scaled_ref(qw_h, st_h, eids_h[[0, 2]], x_h, sc_h)
    assert oracle.within_bound(yb[[0, 2]], y_ref, a_ref)
