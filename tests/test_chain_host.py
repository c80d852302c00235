"""Host-side checks of w4a16_gemv_chain (no GPU): argument checks before any
launch, the launch plan of the decoder chains, and a CPU model of every
shared-memory access and copy the kernel makes for those plans (each stays
inside its buffer, and every (row, group) of a window is read exactly once).
"""

import ctypes

import pytest

from bit_weight_only_gemv_gb300 import lib, synth

MAX_SMEM = 232448          # largest dynamic shared memory of a GB300 CTA
HDR = 1024                 # barriers, flags, window records, finished windows
WARPS = 7                  # warps of a consumer group


@pytest.fixture(scope="module")
def L():
    return lib.load()


def task(N, K, dep=-1, ids=False, n_ids=1, x_rows=1, gated=False, base=1 << 30):
    t = lib.GemvTask()
    t.y, t.qw, t.st, t.x = base, base + (1 << 26), base + (2 << 26), base + (3 << 26)
    t.ids = base + (4 << 26) if ids else None
    t.qw_stride = N * K // 2 if ids else 0
    t.st_stride = N * K // 16 if ids else 0
    t.num_experts = 128 if ids else 0
    t.n_ids, t.x_rows = n_ids, x_rows
    t.N, t.K, t.dep = N, K, dep
    t.flags = lib.W4_TASK_SILU_MUL if gated else 0
    return t


def arr(ts):
    a = (lib.GemvTask * len(ts))()
    for i, t in enumerate(ts):
        a[i] = t
    return a


def dense_pass(model):
    ts = []
    for _ in range(model.layers):
        h = model.hidden
        for n, k in ((sum(p.n for p in model.projs[:3]), h), (model.projs[3].n, h),
                     (model.projs[4].n + model.projs[5].n, h), (model.projs[6].n, model.projs[6].k)):
            ts.append(task(n, k, dep=len(ts) - 1))
    ts.append(task(model.vocab, model.hidden, dep=len(ts) - 1))
    return ts


def moe_layer():
    cfg = synth.moe_2816()
    I, H, k = cfg.expert_inter, cfg.hidden, cfg.top_k
    return [task(2 * I, H, ids=True, n_ids=k, x_rows=1),
            task(H, I, dep=0, ids=True, n_ids=k, x_rows=k, gated=True)]


def plans(L, ts):
    a = arr(ts)
    info = lib.ChainPlanInfo()
    assert L.w4a16_gemv_chain_plan(a, len(ts), ctypes.byref(info)) == 0
    per = []
    for i in range(len(ts)):
        ti = lib.ChainTaskInfo()
        assert L.w4a16_gemv_chain_task_plan(a, len(ts), i, ctypes.byref(ti)) == 0
        per.append({n: getattr(ti, n) for n, _ in lib.ChainTaskInfo._fields_})
    return {n: getattr(info, n) for n, _ in lib.ChainPlanInfo._fields_}, per


def model_windows(ts, plan, per):
    """Replay the kernel's index arithmetic for the first, a middle and the
    last (short) window of every task shape; return the number of checks."""
    nst, stage = plan["stages"], plan["stage_bytes"]
    kgp_max = max(p["team"] * (-(-(t.K // 32) // p["team"])) for t, p in zip(ts, per))
    xs_off = HDR + nst * stage
    xsc_off = xs_off + kgp_max * 64
    red_off = (xsc_off + kgp_max * 4 + 15) & ~15
    red_slot = max([p["rows_per_window"] * p["chunks"] for p in per if p["chunks"] > 1] or [0])
    smem = red_off + nst * red_slot * 4
    assert smem == plan["smem_bytes"] and smem <= MAX_SMEM
    checks = 0
    seen = set()
    for t, p in zip(ts, per):
        key = (t.N, t.K, p["rows_per_window"])
        if key in seen:
            continue
        seen.add(key)
        K, N = t.K, t.N
        Kg, kg2 = K // 32, K // 16
        T, CL, nch, RW, RB = p["team"], p["chunk_steps"], p["chunks"], p["rows_per_lane"], \
            p["rows_per_window"]
        NI = -(-Kg // T)
        Kgp = NI * T
        nsw, gpc, rstep = 32 // T, CL * T, (32 // T) * RW
        assert RB % rstep == 0 and p["windows_per_item"] == -(-N // RB)
        step_off = RB * (K // 2) + (T - 1) * 16
        wins = sorted({0, p["windows_per_item"] // 2, p["windows_per_item"] - 1})
        for w in wins:
            for tile in (HDR, HDR + (nst - 1) * stage):
                row0 = w * RB
                nrows = min(RB, N - row0)
                # copies: codes, the steps' 16-byte superset, the hand-stored tail
                assert nrows * (K // 2) <= step_off
                for sbase in (0, 48):           # the step array's offset mod 16 of an item
                    a0 = sbase + row0 * kg2
                    e = sbase + (row0 + nrows) * kg2
                    a = a0 & ~15
                    assert step_off + (e - a) <= stage
                # consumer reads
                soff0 = 0 if kg2 % 16 == 0 else ((row0 & 7) * (kg2 & 15)) & 15
                nrs = -(-nrows // rstep)
                covered = set()
                for ci in range(nch):
                    ns = min(CL, NI - ci * CL)
                    for rs in range(nrs):
                        for lane in range(32):
                            st_, tt = lane // T, lane % T
                            for j in range(RW):
                                r = rs * rstep + j * nsw + st_
                                assert r < RB
                                for s in range(ns):
                                    g = ci * gpc + tt + s * T
                                    co = tile + r * (K // 2) + g * 16
                                    so = tile + step_off + soff0 + r * kg2 + g * 2
                                    assert HDR <= co and co + 16 <= tile + stage
                                    assert so + 2 <= tile + stage
                                    assert xs_off + g * 16 + 3 * Kgp * 16 + 16 <= xsc_off
                                    assert xsc_off + g * 4 + 4 <= red_off or red_slot == 0
                                    if r < nrows and g < Kg:
                                        assert (r, g) not in covered
                                        covered.add((r, g))
                                        checks += 1
                                if r < nrows and nch > 1:
                                    assert r * nch + ci < red_slot
                assert len(covered) == nrows * Kg
    return checks


@pytest.mark.parametrize("name", ["dense-60L-h5376", "dense-35L-h2048"])
def test_decode_pass_chain_plan_and_bounds(L, name):
    model = {"dense-60L-h5376": synth.dense_5376, "dense-35L-h2048": synth.dense_2048}[name]()
    ts = dense_pass(model)
    plan, per = plans(L, ts)
    assert plan["instantiation"] == (0 if model.hidden == 5376 else 1)
    assert plan["threads"] == 512 and plan["stages"] >= 2
    # tasks with rows for many rounds of windows keep all 7 warps of a group busy
    for t, p in zip(ts, per):
        items = p["chunks"] * p["rows_per_window"] // ((32 // p["team"]) * p["rows_per_lane"])
        if p["windows_per_item"] >= 4 * plan["ctas"]:
            assert items % WARPS == 0, p
    assert model_windows(ts, plan, per) > 0


def test_routed_layer_chain_plan_and_bounds(L):
    ts = moe_layer()
    plan, per = plans(L, ts)
    assert plan["instantiation"] == 2
    assert model_windows(ts, plan, per) > 0


@pytest.mark.parametrize("ks", [(1184, 416), (3232, 14176), (96, 65536), (2048, 704)])
def test_generic_chain_plan_and_bounds(L, ks):
    # K outside the compiled pairs (ragged chunks, padded lane teams, the
    # largest K) run the generic dot loop
    ts = [task(300, ks[0]), task(77, ks[1], dep=0), task(129, ks[0], dep=1, gated=True)]
    plan, per = plans(L, ts)
    assert plan["instantiation"] == 3
    assert model_windows(ts, plan, per) > 0


def test_chain_host_checks(L):
    ts = dense_pass(synth.dense_2048())[:4]
    a = arr(ts)
    ws = ctypes.c_void_p(1 << 30)
    need = L.w4a16_gemv_chain_workspace_bytes(a, 4)
    assert need >= 6 * 4
    # one counter per task, one per id of a routed task
    routed = arr([task(64, 2048, ids=True, n_ids=100), task(64, 2048, dep=0)])
    assert L.w4a16_gemv_chain_workspace_bytes(routed, 2) == (((100 + 1 + 2) * 4 + 255) // 256) * 256
    assert L.w4a16_gemv_chain_workspace_bytes(arr([task(16, 48)]), 1) == 0
    assert L.w4a16_gemv_chain(a, 4, ws, need - 1, None, 0, None) == 4          # workspace
    assert L.w4a16_gemv_chain(a, 4, None, need, None, 0, None) == 4
    assert L.w4a16_gemv_chain(a, 4, ctypes.c_void_p((1 << 30) + 8), need, None, 0, None) == 2
    assert L.w4a16_gemv_chain(a, 4, ws, need, None, 2, None) == 1             # unknown flag
    assert L.w4a16_gemv_chain(a, 0, ws, need, None, 0, None) == 1
    bad = [task(16, 64), task(16, 64, dep=1)]                                  # dep not earlier
    assert L.w4a16_gemv_chain(arr(bad), 2, ws, need, None, 0, None) == 1
    bad = [task(16, 48)]                                                       # K % 32
    assert L.w4a16_gemv_chain(arr(bad), 1, ws, need, None, 0, None) == 3
    t = task(16, 64)
    t.x += 8                                                                   # misaligned x
    assert L.w4a16_gemv_chain(arr([t]), 1, ws, need, None, 0, None) == 2
    t = task(16, 64, ids=True, n_ids=3, x_rows=2)                              # x_rows
    assert L.w4a16_gemv_chain(arr([t]), 1, ws, need, None, 0, None) == 3
    t = task(16, 64, ids=True, n_ids=3)
    t.qw_stride += 8                                                           # stride % 16
    assert L.w4a16_gemv_chain(arr([t]), 1, ws, need, None, 0, None) == 2
    t = task(16, 64)
    t.flags = 2                                                                # unknown task flag
    assert L.w4a16_gemv_chain(arr([t]), 1, ws, need, None, 0, None) == 1
    many = [task(16, 64)] * (lib.CHAIN_MAX_TASKS + 1)
    assert L.w4a16_gemv_chain(arr(many), len(many), ws, 1 << 20, None, 0, None) == 3
