"""GPU parity of w4a16_gemv_id: oracle bound, the slot-pool memcmp bar, and
row-for-row identity with w4a16_gemv on the selected expert."""

import numpy as np
import pytest
import torch

import oracle
from bit_weight_only_gemv_gb300 import lib, synth
from _helpers import POISON, dev_bf16, dev_words, host_bits, poison_bf16

pytestmark = pytest.mark.gpu


def experts(rng, e, n, k, pad_qw=0, pad_st=0):
    """Expert tensors as one byte buffer each, expert stride = size + padding."""
    qw_bytes, st_bytes = n * k // 2, n * k // 16
    qs, ss = qw_bytes + pad_qw, st_bytes + pad_st
    qw_buf = np.zeros(e * qs, np.uint8)
    st_buf = np.zeros(e * ss, np.uint8)
    qw_h = synth.np_words(rng, (e, n, k // 8))
    st_h = synth.np_steps(rng, (e, n, k // 32))
    for i in range(e):
        qw_buf[i * qs:i * qs + qw_bytes] = qw_h[i].view(np.uint8).ravel()
        st_buf[i * ss:i * ss + st_bytes] = st_h[i].view(np.uint8).ravel()
    return qw_h, st_h, qw_buf, st_buf, qs, ss


def dev_bytes(a):
    return torch.from_numpy(a).to("cuda")


@pytest.mark.parametrize("e,n,k,n_ids,x_rows,pad", [
    (6, 96, 704, 4, 4, 0), (6, 96, 704, 4, 1, 32), (5, 704, 2816, 8, 1, 0),
    (5, 2816, 704, 8, 8, 16), (3, 33, 2048, 5, 5, 48), (4, 100, 8192, 3, 1, 0),
    (2, 40, 96, 1, 1, 0)])
def test_gemv_id_matches_oracle(cuda_lib, e, n, k, n_ids, x_rows, pad):
    rng = np.random.default_rng(e * 7 + n + k + n_ids + pad)
    qw_h, st_h, qwb, stb, qs, ss = experts(rng, e, n, k, pad, pad)
    ids_h = rng.integers(0, e, size=n_ids).astype(np.int32)
    if n_ids > 1:
        ids_h[1] = ids_h[0]                       # repeated id
    x_h = synth.np_x(rng, (x_rows, k))
    ids = torch.from_numpy(ids_h).to("cuda")
    y = poison_bf16((n_ids, n))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib.gemv_id(dev_bytes(qwb), dev_bytes(stb), ids, dev_bf16(x_h), n, k, e, qs, ss, y=y,
                status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    yb = host_bits(y)
    y_ref = oracle.gemv_id_ref(qw_h, st_h, ids_h, x_h)
    a_ref = np.stack([oracle.gemv_abs_ref(qw_h[d], st_h[d], x_h[0 if x_rows == 1 else i])[0]
                      for i, d in enumerate(ids_h)])
    assert oracle.within_bound(yb, y_ref, a_ref)
    # row i is bitwise the dense GEMV of expert ids[i] on its activation row
    for i, d in enumerate(ids_h):
        yd = lib.gemv(dev_words(qw_h[d]), dev_bf16(st_h[d]),
                      dev_bf16(x_h[0 if x_rows == 1 else i][None]),
                      workspace=torch.zeros(max(1, lib.workspace_bytes(1, n, k)),
                                            dtype=torch.uint8, device="cuda"))
        torch.cuda.synchronize()
        assert np.array_equal(host_bits(yd)[0], yb[i])


# K whose groups do not split evenly over a lane team's chunks: a short last
# chunk (37 and 13 groups, chunks of 4) and teams padded past the end of a row
# (101 and 443 groups walked by 32 lanes); broadcast and per-id activations,
# expert strides with and without padding
RAGGED_ROUTED = [(4, 70, 1184, 5, 5, 16), (5, 129, 416, 6, 1, 0), (4, 33, 3232, 3, 1, 32),
                 (3, 20, 14176, 4, 4, 48), (3, 45, 3232, 4, 4, 0)]


@pytest.mark.parametrize("e,n,k,n_ids,x_rows,pad", RAGGED_ROUTED)
def test_gemv_id_ragged_k_matches_oracle(cuda_lib, e, n, k, n_ids, x_rows, pad):
    p = lib.plan(1, n, k)
    groups = k // 32
    assert groups % p["team"] or (-(-groups // p["team"])) % p["chunk_steps"]   # ragged
    rng = np.random.default_rng(e + 5 * n + k + n_ids + pad)
    # expert strides: the sizes rounded up to 16 bytes, plus the padding
    qw_h, st_h, qwb, stb, qs, ss = experts(rng, e, n, k, (-(n * k // 2)) % 16 + pad,
                                           (-(n * k // 16)) % 16 + pad)
    ids_h = rng.integers(0, e, size=n_ids).astype(np.int32)
    ids_h[-1] = ids_h[0]                          # repeated id
    x_h = synth.np_x(rng, (x_rows, k))
    y = poison_bf16((n_ids, n))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib.gemv_id(dev_bytes(qwb), dev_bytes(stb), torch.from_numpy(ids_h).to("cuda"),
                dev_bf16(x_h), n, k, e, qs, ss, y=y, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    yb = host_bits(y)
    assert not np.any(yb == POISON)
    y_ref = oracle.gemv_id_ref(qw_h, st_h, ids_h, x_h)
    a_ref = np.stack([oracle.gemv_abs_ref(qw_h[d], st_h[d], x_h[0 if x_rows == 1 else i])[0]
                      for i, d in enumerate(ids_h)])
    assert oracle.within_bound(yb, y_ref, a_ref)
    # and row i is bitwise the dense GEMV of expert ids[i]
    for i, d in enumerate(ids_h):
        need = lib.workspace_bytes(1, n, k)
        yd = lib.gemv(dev_words(qw_h[d]), dev_bf16(st_h[d]),
                      dev_bf16(x_h[0 if x_rows == 1 else i][None]),
                      workspace=torch.zeros(max(16, need), dtype=torch.uint8, device="cuda")
                      if need else None)
        torch.cuda.synchronize()
        assert np.array_equal(host_bits(yd)[0], yb[i])


# calls with enough windows take them at run time, within one id each, on
# the dense walk's loop (compiled team shapes with 4, 2 and 1 rows per lane,
# and the generic loop); shared and per-id activation rows
RUN_TIME = [(10, 5376, 5376, 8, 1), (8, 4096, 2048, 6, 6), (34, 2816, 704, 32, 32),
            (10, 9000, 1184, 8, 1), (12, 3000, 1184, 10, 10), (14, 4000, 2816, 12, 1),
            (9, 3000, 3232, 8, 1)]


@pytest.mark.parametrize("e,n,k,n_ids,x_rows", RUN_TIME)
def test_gemv_id_run_time_windows(cuda_lib, e, n, k, n_ids, x_rows):
    plan = lib.id_plan(n_ids, x_rows, n, k)
    assert plan["dynamic_windows"] == 1
    rng = np.random.default_rng(e * 3 + n + k)
    qw = synth.torch_words((e, n * k // 8), synth.seed_of(71, n, k), "cuda")
    st = synth.torch_steps((e, n * k // 32), synth.seed_of(72, n, k), "cuda")
    ids_h = rng.integers(0, e, size=n_ids).astype(np.int32)
    ids_h[-1] = ids_h[0]                                   # a repeated id
    x_h = synth.np_x(rng, (x_rows, k))
    y = poison_bf16((n_ids, n))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib.gemv_id(qw, st, torch.from_numpy(ids_h).to("cuda"), dev_bf16(x_h), n, k, e, n * k // 2,
                n * k // 16, y=y, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    yb = host_bits(y)
    assert not np.any(yb == POISON)
    # sampled rows of every id (the item's last rows: a short window) against
    # the oracle, and every row bitwise the dense GEMV of its expert
    rows = np.unique(np.concatenate([rng.choice(n, 40, replace=False), np.arange(n - 5, n)]))
    for i, d in enumerate(ids_h):
        xi = x_h[0 if x_rows == 1 else i][None]
        qe = qw[int(d)].view(n, k // 8)
        se = st[int(d)].view(n, k // 32)
        need = lib.workspace_bytes(1, n, k)
        yd = lib.gemv(qe, se, dev_bf16(xi), workspace=torch.zeros(
            max(16, need), dtype=torch.uint8, device="cuda") if need else None)
        torch.cuda.synchronize()
        assert np.array_equal(host_bits(yd)[0], yb[i])
        idx = torch.from_numpy(rows).to("cuda")
        q_h = qe[idx].cpu().numpy().view(np.uint32)
        s_h = se[idx].view(torch.int16).cpu().numpy().view(np.uint16)
        assert oracle.within_bound(yb[i][rows][None], oracle.gemv_ref(q_h, s_h, xi),
                                   oracle.gemv_abs_ref(q_h, s_h, xi))


def test_gemv_id_run_time_windows_bad_ids(cuda_lib):
    e, n, k = 6, 4096, 2048
    assert lib.id_plan(6, 1, n, k)["dynamic_windows"] == 1
    qw = synth.torch_words((e, n * k // 8), synth.seed_of(73), "cuda")
    st = synth.torch_steps((e, n * k // 32), synth.seed_of(74), "cuda")
    ids_h = np.array([1, 6, 3, -2, 5, 1], np.int32)
    x = dev_bf16(synth.np_x(np.random.default_rng(3), (1, k)))
    y = poison_bf16((6, n))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib.gemv_id(qw, st, torch.from_numpy(ids_h).to("cuda"), x, n, k, e, n * k // 2, n * k // 16,
                y=y, status=status)
    torch.cuda.synchronize()
    assert lib.STATUS[int(status.item())] == "W4_ERR_INDEX"
    yb = host_bits(y)
    for i, d in enumerate(ids_h):
        if 0 <= d < e:
            ref = lib.gemv(qw[int(d)].view(n, k // 8), st[int(d)].view(n, k // 32), x)
            torch.cuda.synchronize()
            assert np.array_equal(yb[i], host_bits(ref)[0])
        else:
            assert np.all(yb[i] == POISON)


def test_gemv_id_bad_ids_leave_rows_unwritten(cuda_lib):
    rng = np.random.default_rng(11)
    e, n, k = 4, 64, 2048
    qw_h, st_h, qwb, stb, qs, ss = experts(rng, e, n, k)
    ids_h = np.array([1, 4, -1, 3], np.int32)
    x_h = synth.np_x(rng, (1, k))
    y = poison_bf16((4, n))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib.gemv_id(dev_bytes(qwb), dev_bytes(stb), torch.from_numpy(ids_h).cuda(), dev_bf16(x_h),
                n, k, e, qs, ss, y=y, status=status)
    torch.cuda.synchronize()
    assert lib.STATUS[int(status.item())] == "W4_ERR_INDEX"
    yb = host_bits(y)
    assert np.all(yb[1] == POISON) and np.all(yb[2] == POISON)
    assert not np.any(yb[0] == POISON) and not np.any(yb[3] == POISON)
    ref = oracle.gemv_id_ref(qw_h, st_h, ids_h[[0, 3]], x_h)
    a = np.stack([oracle.gemv_abs_ref(qw_h[d], st_h[d], x_h)[0] for d in ids_h[[0, 3]]])
    assert oracle.within_bound(yb[[0, 3]], ref, a)


def test_slot_pool_is_bitwise_equal_to_full_tensor(cuda_lib):
    """The page's memcmp bar: the pool changes only where the kernel reads the
    expert from, so the outputs must be identical bit for bit."""
    rng = np.random.default_rng(12)
    cfg = synth.moe_2816()
    E, S, H, I = 32, 8, cfg.hidden, cfg.expert_inter
    n_layers, steps = 2, 40
    for proj, (n, k) in (("gate", (I, H)), ("down", (H, I))):
        for layer in range(n_layers):
            qs, ss = n * k // 2, n * k // 16
            full_q = synth.torch_words((E, qs // 4), seed=synth.seed_of(3, layer, n), device="cuda")
            full_s = synth.torch_steps((E, ss // 2), seed=synth.seed_of(4, layer, n), device="cuda")
            pool_q = torch.zeros((S, qs // 4), dtype=torch.int32, device="cuda")
            pool_s = torch.zeros((S, ss // 2), dtype=torch.bfloat16, device="cuda")
            pool = lib.SlotPool(E, S)
            slot_ids = torch.zeros(4, dtype=torch.int32, device="cuda")
            trace = synth.moe_trace(E, 4, steps, 1.1, 0.7, seed=layer)
            for t in range(steps):
                x_rows = 1 if proj == "gate" else 4
                x = synth.torch_x((x_rows, k), seed=synth.seed_of(5, layer, t), device="cuda")
                pool.stage(trace[t], pool_q, full_q, qs, qs, pool_s, full_s, ss, ss, slot_ids)
                ids_full = torch.from_numpy(trace[t].astype(np.int32)).cuda()
                y_pool = lib.gemv_id(pool_q, pool_s, slot_ids, x, n, k, S, qs, ss)
                y_full = lib.gemv_id(full_q, full_s, ids_full, x, n, k, E, qs, ss)
                assert torch.equal(y_pool.view(torch.int16), y_full.view(torch.int16)), (proj, t)
            st = pool.stats()
            assert st["hits"] > 0 and st["misses"] >= S
    torch.cuda.synchronize()


def test_bound_calls_and_side_by_side_slots(cuda_lib):
    """Pre-marshalled calls (bind_stage, bind_gemv_id) over slots that hold two
    projections side by side give the same slots and bits as the plain calls
    on separate per-projection tensors."""
    cfg = synth.moe_2816()
    E, S, H, I, k_top = 16, 6, cfg.hidden, cfg.expert_inter, 4
    shapes = {"gate_up": (2 * I, H), "down": (H, I)}
    qoff, soff, qcomb, scomb = {}, {}, 0, 0
    for name, (n, k) in shapes.items():
        qoff[name], soff[name] = qcomb, scomb
        qcomb += n * k // 2
        scomb += n * k // 16
    full_q = synth.torch_words((E, qcomb // 4), seed=synth.seed_of(6, 1), device="cuda")
    full_s = synth.torch_steps((E, scomb // 2), seed=synth.seed_of(6, 2), device="cuda")
    pool_q = torch.zeros((S, qcomb // 4), dtype=torch.int32, device="cuda")
    pool_s = torch.zeros((S, scomb // 2), dtype=torch.bfloat16, device="cuda")
    slot_ids = torch.zeros(k_top, dtype=torch.int32, device="cuda")
    xs = {"gate_up": synth.torch_x((1, H), seed=7, device="cuda"),
          "down": synth.torch_x((k_top, I), seed=8, device="cuda")}
    ys = {name: torch.empty((k_top, n), dtype=torch.bfloat16, device="cuda")
          for name, (n, k) in shapes.items()}
    calls = {name: lib.bind_gemv_id(pool_q[:, qoff[name] // 4:], pool_s[:, soff[name] // 2:],
                                    slot_ids, xs[name], n, k, S, qcomb, scomb, ys[name])
             for name, (n, k) in shapes.items()}
    pool, ref_pool = lib.SlotPool(E, S), lib.SlotPool(E, S)
    stage = pool.bind_stage(k_top, pool_q, full_q, qcomb, qcomb, pool_s, full_s, scomb, scomb,
                            slot_ids)
    ref_slots = torch.zeros(k_top, dtype=torch.int32, device="cuda")
    trace = synth.moe_trace(E, k_top, 30, 1.1, 0.7, seed=3)
    for t in range(30):
        nm = stage(trace[t])
        _, nm_ref = ref_pool.stage(trace[t], pool_q, full_q, qcomb, qcomb, pool_s, full_s, scomb,
                                   scomb, ref_slots)
        assert nm == nm_ref
        assert torch.equal(slot_ids, ref_slots)
        for name, (n, k) in shapes.items():
            calls[name](pdl=name == "down")
            # the same product from this projection's weights of the named experts
            q = full_q[:, qoff[name] // 4:(qoff[name] + n * k // 2) // 4].contiguous()
            st = full_s[:, soff[name] // 2:(soff[name] + n * k // 16) // 2].contiguous()
            ids = torch.from_numpy(trace[t].astype(np.int32)).cuda()
            y_ref = lib.gemv_id(q, st, ids, xs[name], n, k, E, n * k // 2, n * k // 16)
            assert torch.equal(ys[name].view(torch.int16), y_ref.view(torch.int16)), (name, t)
    torch.cuda.synchronize()


@pytest.mark.parametrize("e,n,k,n_ids,x_rows", [(8, 2816, 704, 8, 8), (8, 1408, 2816, 8, 1),
                                                (6, 5376, 5376, 8, 1)])
def test_ids_final_same_bits_in_a_pdl_chain(cuda_lib, e, n, k, n_ids, x_rows):
    # A routed call launched as a programmatic dependent of another kernel
    # with W4_FLAG_IDS_FINAL (its ids written before that kernel) starts its
    # weight copies early: the same bits as without the flag, and as the
    # oracle bound, on fixed-share and run-time-window plans alike.
    rng = np.random.default_rng(e + n + k)
    qw_h, st_h, qwb, stb, qs, ss = experts(rng, e, n, k)
    ids_h = rng.permutation(e)[:n_ids].astype(np.int32) if n_ids <= e else \
        rng.integers(0, e, size=n_ids).astype(np.int32)
    x_h = synth.np_x(rng, (x_rows, k))
    qw, st, ids, x = dev_bytes(qwb), dev_bytes(stb), torch.from_numpy(ids_h).to("cuda"), dev_bf16(x_h)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    y0 = lib.gemv_id(qw, st, ids, x, n, k, e, qs, ss, status=status)
    # a kernel before it in the stream: another routed call on the same ids
    other = poison_bf16((n_ids, n))
    ys = []
    for _ in range(3):
        lib.gemv_id(qw, st, ids, x, n, k, e, qs, ss, y=other, status=status, pdl=True)
        y = poison_bf16((n_ids, n))
        lib.gemv_id(qw, st, ids, x, n, k, e, qs, ss, y=y, status=status, pdl=True, ids_final=True)
        ys.append(y)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for y in ys:
        assert torch.equal(y.view(torch.int16), y0.view(torch.int16))
    y_ref = oracle.gemv_id_ref(qw_h, st_h, ids_h, x_h)
    a_ref = np.stack([oracle.gemv_abs_ref(qw_h[d], st_h[d], x_h[0 if x_rows == 1 else i])[0]
                      for i, d in enumerate(ids_h)])
    assert oracle.within_bound(host_bits(ys[-1]), y_ref, a_ref)
