"""C-ABI checks that need no GPU: the library loads, exports every call the
header declares, validates arguments on the host, plans launches, and runs the
host-side slot pool exactly like the oracle's policy."""

import ctypes
import os
import re

import numpy as np
import pytest
import torch

import oracle
from bit_weight_only_gemv_gb300 import lib, synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    return lib.load()


def header_functions():
    text = open(os.path.join(ROOT, "include", "w4a16.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(w4\w*)\s*\(", text)))


def test_header_declares_the_calls():
    names = header_functions()
    for need in ("w4a16_gemv", "w4a16_gemv_id", "w4a16_gemv_id_scaled", "w4_embed_gather",
                 "w4_pack", "w4_quantize"):
        assert need in names


def test_library_exports_every_declared_call(L):
    for name in header_functions():
        assert hasattr(L, name), name
        assert isinstance(getattr(L, name), ctypes._CFuncPtr)
    assert set(lib.EXPORTS) <= set(header_functions())


def test_version_and_status_strings(L):
    assert L.w4_abi_version() == 4
    assert L.w4_status_str(0) == b"ok"
    assert L.w4_status_str(6) == b"id out of range"
    assert L.w4_status_str(11) == b"slot does not hold the named expert"
    assert L.w4_status_str(999) == b"unknown status"


def test_host_validation_rejects_before_any_launch(L):
    vp = ctypes.c_void_p
    good = vp(1 << 20)                      # never dereferenced: rejected earlier
    # K not a multiple of 32
    assert L.w4a16_gemv(good, good, good, good, 1, 16, 48, None, 0, None, 0, None) == 3
    # null pointer
    assert L.w4a16_gemv(None, good, good, good, 1, 16, 64, None, 0, None, 0, None) == 1
    # M out of range
    assert L.w4a16_gemv(good, good, good, good, 257, 16, 64, None, 0, None, 0, None) == 3
    # misaligned weights
    assert L.w4a16_gemv(good, vp((1 << 20) + 8), good, good, 1, 16, 64, None, 0, None, 0,
                        None) == 2
    # unknown flag bit
    assert L.w4a16_gemv(good, good, good, good, 1, 16, 64, None, 0, None, 16, None) == 1
    # the fused SiLU-mul activation runs on the CUDA cores only
    assert L.w4a16_gemv(good, good, good, good, 1, 16, 256, None, 0, None, 8 | 4, None) == 3
    assert L.w4a16_gemv(good, good, good, good, 1, 16, 256, None, 0, None, 6, None) == 1
    assert L.w4a16_gemv(good, good, good, good, 1, 16, 64, None, 0, None, 4, None) == 3
    # gemv_id: x_rows must be 1 or n_ids, strides multiples of 16 and >= an expert
    assert L.w4a16_gemv_id(good, good, 1024, good, 128, 4, good, 3, good, 2, 32, 64, None, 0,
                           None) == 3
    assert L.w4a16_gemv_id(good, good, 1032, good, 128, 4, good, 3, good, 1, 32, 64, None, 0,
                           None) == 2
    assert L.w4a16_gemv_id(good, good, 512, good, 128, 4, good, 3, good, 1, 32, 64, None, 0,
                           None) == 1
    # routed flags: W4_FLAG_PDL and W4_FLAG_IDS_FINAL only
    assert L.w4a16_gemv_id(good, good, 1024, good, 128, 4, good, 3, good, 1, 32, 64, None, 32,
                           None) == 1
    assert L.w4a16_gemv_id(good, good, 1024, good, 128, 4, good, 3, good, 1, 32, 64, None, 8,
                           None) == 1
    # gemv_id_scaled: real ids required, vectors 2-byte aligned, table 4-byte aligned
    def scaled(eids=good, n_real=8, table=None, scale=None, bias=None, x_rows=1):
        return L.w4a16_gemv_id_scaled(good, good, 1024, good, 128, 4, good, 3, good, x_rows, 32,
                                      64, eids, n_real, table, scale, bias, None, 0, None)
    assert scaled(eids=None) == 1
    assert scaled(n_real=0) == 1
    assert scaled(x_rows=2) == 3
    assert scaled(scale=vp((1 << 20) + 1)) == 2
    assert scaled(bias=vp((1 << 20) + 3)) == 2
    assert scaled(table=vp((1 << 20) + 2)) == 2
    # the no-allocation GEMV takes w4a16_gemv's flags (the gated flag on the
    # CUDA cores only) and refuses the rest before any launch
    sgemv = L.w4a16_gemv_static_scratch
    assert sgemv(good, good, good, good, 1, 16, 64, None, 16, None) == 1
    assert sgemv(good, good, good, good, 1, 16, 256, None, 6, None) == 1
    assert sgemv(good, good, good, good, 1, 16, 256, None, 8 | 4, None) == 3
    assert sgemv(good, good, good, good, 1, 16, 48, None, 8, None) == 3
    assert sgemv(None, good, good, good, 1, 16, 64, None, 8, None) == 1
    # the L2-prefetching GEMV: range count, null and misaligned ranges, then
    # w4a16_gemv's own checks
    pf = L.w4a16_gemv_prefetch_l2
    R = lib.l2_ranges
    ok2 = R([(1 << 22, 4096), (1 << 23, 100)])
    assert pf(good, good, good, good, 1, 16, 64, None, 0, None, 0, ok2, -1, None) == 1
    assert pf(good, good, good, good, 1, 16, 64, None, 0, None, 0, ok2, 5, None) == 1
    assert pf(good, good, good, good, 1, 16, 64, None, 0, None, 0, None, 1, None) == 1
    assert pf(good, good, good, good, 1, 16, 64, None, 0, None, 0,
              R([(0, 64)]), 1, None) == 1                                     # null with bytes
    assert pf(good, good, good, good, 1, 16, 64, None, 0, None, 0,
              R([((1 << 22) + 8, 64)]), 1, None) == 2                         # misaligned
    assert pf(good, good, good, good, 1, 16, 48, None, 0, None, 0, ok2, 2, None) == 3
    assert pf(None, good, good, good, 1, 16, 64, None, 0, None, 0, ok2, 2, None) == 1
    assert pf(good, good, good, good, 1, 16, 64, None, 0, None, 16, ok2, 2, None) == 1
    assert L.w4_embed_gather(good, good, good, good, 0, 10, 64, None, 0, None) == 1
    assert L.w4_pack(good, good, 4, 40, None, None) == 3
    assert L.w4_quantize(good, good, vp((1 << 20) + 4), 4, 64, None) == 2


def test_device_pool_host_checks(L):
    vp = ctypes.c_void_p
    good = vp(1 << 20)
    # state size: slots and experts within their limits
    assert L.w4_dev_pool_state_bytes(128, 32) > 0
    assert L.w4_dev_pool_state_bytes(128, 32) % 16 == 0
    assert L.w4_dev_pool_state_bytes(128, 65) == 0
    assert L.w4_dev_pool_state_bytes(3981, 8) == 0
    assert L.w4_dev_pool_state_bytes(0, 8) == 0
    # init: arguments checked before any launch
    assert L.w4_dev_pool_init(None, 128, 32, None) == 1
    assert L.w4_dev_pool_init(good, 8, 9, None) == 3          # more slots than experts
    assert L.w4_dev_pool_init(vp((1 << 20) + 8), 128, 32, None) == 2

    def stage(state=good, E=128, S=32, ids=good, k=8, qw_stride=1024, qw_bytes=1024,
              st_stride=128, st_bytes=128, slot_ids=good, flags=0):
        return L.w4_dev_pool_stage(state, E, S, ids, k, good, good, qw_stride, qw_bytes, good,
                                   good, st_stride, st_bytes, slot_ids, None, None, flags, None)
    assert stage(state=None) == 1
    assert stage(slot_ids=None) == 1
    assert stage(k=0) == 1
    assert stage(k=65) == 3
    assert stage(S=65) == 3
    assert stage(E=4000) == 3
    assert stage(qw_bytes=2048) == 1                           # expert larger than its stride
    assert stage(flags=2) == 1                                 # only W4_FLAG_PDL


@pytest.mark.parametrize("M,N,K", [(1, 2048, 2048), (1, 512, 2048), (1, 2048, 8192),
                                   (1, 5376, 21504), (1, 704, 2816), (1, 2816, 704),
                                   (4, 8192, 2048), (1, 262144, 2048), (1, 7, 32),
                                   (3, 100, 65536)])
def test_plan_is_valid(M, N, K):
    p = lib.plan(M, N, K, path="cuda")          # the CUDA-core plan (4 x 8192 x 2048 defaults
    assert p["path"] == 1                       # to the tensor cores)
    assert p["threads"] == 256                   # 7 consumer warps + 1 copy warp
    assert p["team"] in (1, 2, 4, 8, 16, 32) and (K // 32) % p["team"] == 0
    assert p["rows_per_lane"] in (1, 2, 4)
    assert p["unit_rows"] % ((32 // p["team"]) * p["rows_per_lane"]) == 0
    # groups per lane per chunk: all of a lane's groups when <= 4, else 4 or 3
    # when that divides them, else all of them up to 12, else 4
    ni = -(-(K // 32) // p["team"])
    want = (ni if ni <= 4 else 4 if ni % 4 == 0 else 3 if ni % 3 == 0 else ni if ni <= 12 else 4)
    assert p["chunk_steps"] == want
    assert p["chunk_groups"] == p["team"] * p["chunk_steps"]
    assert 1 <= p["ctas"] <= 2 * 152
    assert p["ctas_per_sm"] in (1, 2)
    assert 2 <= p["stages"] <= 8
    assert p["smem_bytes"] <= 232448
    if p["ctas_per_sm"] == 2:
        assert p["smem_bytes"] <= 233472 // 2 - 1024
    assert 1 <= p["rows_per_call"] <= min(M, 4)
    if K <= 21504:
        assert p["rows_per_call"] == min(M, 4)
    ws = lib.workspace_bytes(M, N, K, "cuda")
    assert (ws > 0) == (p["slices"] > 1)


@pytest.mark.parametrize("M,N,K", [(8, 2048, 2048), (16, 16384, 2048), (32, 2048, 8192),
                                   (17, 300, 256), (9, 5376, 21504)])
def test_tensor_core_plan_is_valid(M, N, K):
    p = lib.plan(M, N, K)
    assert p["path"] == 2 and p["threads"] == 320 and p["unit_rows"] == 128
    assert p["tmpl_team"] == (16 if M <= 16 else 32)      # MMA N: activation columns
    assert p["rows_per_call"] == min(M, 32)
    assert p["ctas_per_sm"] in (1, 2)
    assert 2 <= p["stages"] <= 8 and p["smem_bytes"] <= 233472 // p["ctas_per_sm"] - 1024
    assert 1 <= p["ctas"] <= p["ctas_per_sm"] * 152
    if p["ctas_per_sm"] == 1:      # all of tensor memory: no second CTA fits the SM
        assert p["smem_bytes"] > 233472 // 2
    tiles, slices = -(-N // 128), K // 256
    assert 1 <= p["slices"] <= slices
    assert (lib.workspace_bytes(M, N, K) > 0) == (p["slices"] > 1 or p["dynamic_windows"] == 1)
    assert lib.workspace_bytes(M, N, K, "tensor") == lib.workspace_bytes(M, N, K)


@pytest.mark.parametrize("M,N,K", [(33, 2048, 2048), (64, 16384, 2048), (100, 300, 256),
                                   (256, 43008, 5376), (256, 5376, 21504), (200, 7, 512)])
def test_prompt_plan_is_valid(M, N, K):
    p = lib.plan(M, N, K)
    assert p["path"] == 3 and p["threads"] == 320 and p["unit_rows"] == 128
    assert p["rows_per_call"] == M and p["ctas_per_sm"] == 1
    nt = p["tmpl_team"]                  # MMA N: the activation rows of a unit
    assert nt % 16 == 0 and 16 <= nt <= 256
    tiles = -(-N // 128)
    # activation rows stay in one unit unless the weight tiles are too few for
    # the SMs: then they are halved (tiles of at least 16 rows) while the
    # units fit one wave
    ttiles = 1
    while 2 * ttiles * tiles <= 152 and -(-M // (2 * ttiles)) >= 16:
        ttiles *= 2
    xrows = -(-M // ttiles)
    assert nt == -(-xrows // 16) * 16
    assert p["ctas"] == min(tiles * ttiles, 152)
    if tiles >= 76:
        assert ttiles == 1 and M <= nt < M + 16
    assert 2 <= p["stages"] <= 8
    # more than half the SM (one CTA holds all 512 tensor-memory columns), within the limit
    assert 233472 // 2 < p["smem_bytes"] <= 232448
    assert lib.workspace_bytes(M, N, K) == 0
    # K not a multiple of 256 stays on the CUDA cores
    assert lib.plan(M, N, K + 32)["path"] == 1


def test_tiling_depends_on_k_only():
    # the per-row arithmetic (team, chunk length) must not change with N or M
    for K in (704, 2048, 2816, 5376, 8192, 21504):
        ref = lib.plan(1, 4096, K)
        for N in (16, 704, 2048, 100000):
            p = lib.plan(1, N, K)
            assert (p["team"], p["chunk_groups"]) == (ref["team"], ref["chunk_groups"])


def test_slot_pool_matches_oracle_policy():
    rng = np.random.default_rng(0)
    for trial in range(20):
        e = int(rng.integers(2, 200))
        s = int(rng.integers(1, min(e, 48) + 1))
        k = int(rng.integers(1, s + 1))
        pool = lib.SlotPool(e, s)
        ref = oracle.LFUSlotPoolRef(e, s)
        if trial % 2:
            trace = synth.moe_trace(e, k, 60, 1.1, 0.7, seed=trial) if k <= e else None
        else:
            trace = [list(rng.integers(0, e, size=k)) for _ in range(60)]
        for req in trace:
            assert pool.remap(req) == ref.step(req)


def test_slot_pool_hand_traces_and_errors():
    import test_oracle_pins as pins
    for name, e, s, steps in pins._read_traces():
        pool = lib.SlotPool(e, s)
        for req, want_slots, want_miss in steps:
            assert pool.remap(req) == (want_slots, want_miss), name
    pool = lib.SlotPool(4, 2)
    with pytest.raises(lib.W4Error) as ei:
        pool.remap([0, 1, 2])
    assert ei.value.name == "W4_ERR_STATE"
    with pytest.raises(lib.W4Error) as ei:
        pool.remap([4])
    assert ei.value.name == "W4_ERR_INDEX"
    # rejected requests leave the pool unchanged
    assert pool.remap([1]) == ([0], [(1, 0)])
    st = pool.stats()
    assert st == {"requests": 1, "hits": 0, "misses": 1}


@pytest.mark.skipif(torch.cuda.is_available(), reason="uses the failure of copies without a GPU")
def test_slot_pool_failed_copy_forgets_the_slot():
    # Without a device every enqueue fails: the pool must report it and must not
    # keep the expert it could not load.
    pool = lib.SlotPool(8, 2)
    fake = torch.empty(1)
    fake_ptr = type("P", (), {"data_ptr": lambda self: 1 << 20})()
    with pytest.raises(lib.W4Error) as ei:
        pool.stage([3], fake_ptr, fake_ptr, 4096, 4096, fake_ptr, fake_ptr, 512, 512, fake_ptr,
                   stream=type("S", (), {"cuda_stream": 0})(), slot_expert=fake_ptr)
    assert ei.value.name == "W4_ERR_STATE"
    # the expert is not resident: the next request for it is a miss again
    assert pool.remap([3]) == ([0], [(3, 0)])
    del fake


def test_planner_sweep_of_random_shapes():
    """Every valid shape gets a plan on the path the rule names, within the
    SM's limits (seeded sample: M 1..256, N 1..300000, K 32..65536)."""
    rng = np.random.default_rng(2024)
    for _ in range(3000):
        M = int(rng.choice([1, 2, 3, 4, 5, 7, 8, 9, 16, 31, 32, 33, 64, 100, 255, 256])) \
            if rng.random() < 0.5 else int(rng.integers(1, 257))
        N = int(np.exp(rng.uniform(0, np.log(300000))))
        K = 32 * int(np.exp(rng.uniform(0, np.log(2048))))
        if rng.random() < 0.3:
            K = 256 * max(1, K // 256)
        p = lib.plan(M, N, K)
        tc_rows = M >= 5 or (M == 4 and N * K >= 1 << 24) or (M == 3 and N * K >= 1 << 27)
        want = 1 if (not tc_rows or K % 256) else (2 if M <= 32 else 3)
        assert p["path"] == want, (M, N, K, p)
        assert 1 <= p["ctas"] <= p["ctas_per_sm"] * 152, (M, N, K, p)
        assert p["smem_bytes"] <= 232448, (M, N, K, p)
        if p["ctas_per_sm"] == 2:
            assert p["smem_bytes"] <= 233472 // 2 - 1024, (M, N, K, p)
        if want == 1:
            assert p["threads"] == 256 and 1 <= p["rows_per_call"] <= min(M, 4)
            # a team of lanes shares a row: the largest power of two dividing
            # the groups that leaves each lane 4 or more (else the largest
            # dividing one); when a step of 32/team whole rows would pass
            # 40 KB, up to 32 lanes walk the row and the last are padded
            g = K // 32
            t = 1
            while t < 32 and g % (2 * t) == 0 and g // (2 * t) >= 4:
                t *= 2
            if g // t < 4:
                t = 1
                while t < 32 and g % (2 * t) == 0:
                    t *= 2
            if (32 // t) * (K // 2 + g * 2) > 40 << 10:
                t = 32
                while t > 1 and -(-g // t) < 4:
                    t //= 2
            assert p["team"] == t, (M, N, K, p)
            assert 1 <= p["chunk_steps"] <= min(-(-g // t), 12)
        elif want == 2:
            assert p["threads"] == 320 and p["rows_per_call"] == min(M, 32)
        else:
            assert p["threads"] == 320 and p["rows_per_call"] == M
            assert lib.workspace_bytes(M, N, K) == 0
        ws = lib.workspace_bytes(M, N, K)
        # CUDA cores: the size covers the largest plan a launch of up to 4
        # rows of this shape may take (a bound); tensor cores: exactly the
        # split-K scratch of the one launch
        if want == 1:
            assert ws > 0 or p["slices"] == 1, (M, N, K, p, ws)
        else:
            # (or the hand-over slots of balanced runs)
            assert (ws > 0) == (p["slices"] > 1 or p["dynamic_windows"] == 1), (M, N, K, p, ws)
        # a call pinned to either path is planned too (tensor cores: K % 256 == 0)
        assert lib.workspace_bytes(M, N, K, "cuda") >= 0
        if K % 256 == 0:
            assert lib.workspace_bytes(M, N, K, "tensor") == (ws if want != 1 else
                                                             lib.workspace_bytes(M, N, K, "tensor"))


def tc_segments(c, G, tiles, slices):
    """The tensor-core kernel's balanced runs for CTA c of G (its segment
    arithmetic, replayed): [(tile, first slice, end slice, kind)]."""
    W = tiles * slices
    w0, w1 = c * W // G, (c + 1) * W // G
    tf, k0 = divmod(w0, slices)
    tl = (w1 - 1) // slices
    j1 = w1 - tl * slices
    segs = []
    if j1 < slices:
        segs.append((tl, 0, j1, "head"))
    wb = tf + 1 if k0 > 0 else tf
    we = tl if j1 < slices else tl + 1
    segs += [(t, 0, slices, "whole") for t in range(wb, max(wb, we))]
    if k0 > 0:
        segs.append((tf, k0, slices, "tail"))
    return segs


@pytest.mark.parametrize("M,N,K", [(16, 43008, 5376), (32, 65536, 2048), (8, 40900, 1024),
                                   (16, 39680, 1024), (32, 131072, 2048), (9, 77824 - 64, 512),
                                   (32, 38990, 2048), (1, 43008, 5376)])
def test_tensor_core_balanced_runs_cover_every_item_once(M, N, K):
    p = lib.plan(M, N, K)
    if p["path"] != 2:   # batch 1 stays on the CUDA cores
        return
    tiles, slices, G = -(-N // 128), K // 256, p["ctas"]
    if not p["dynamic_windows"]:
        assert tiles <= G or 4 * -(-tiles // G) * G < 5 * tiles or slices < 2
        return
    assert p["ctas_per_sm"] == 2 and tiles > G and tiles * slices // G >= slices
    # workspace: one flag per CTA (256-byte aligned), then a prefix slot of
    # M x 128 fp32 per CTA
    assert lib.workspace_bytes(M, N, K) == (-(-G * 4 // 256)) * 256 + G * M * 128 * 4
    seen = {}
    heads, tails = {}, {}
    for c in range(G):
        segs = tc_segments(c, G, tiles, slices)
        kinds = [k for *_, k in segs]
        # the head (if any) first, the tail (if any) last, whole tiles between
        assert kinds.count("head") <= 1 and kinds.count("tail") <= 1
        if "head" in kinds:
            assert kinds[0] == "head"
        if "tail" in kinds:
            assert kinds[-1] == "tail" and c > 0
        for t, b, e, k in segs:
            assert 0 <= t < tiles and 0 <= b < e <= slices
            for sl in range(b, e):
                assert (t, sl) not in seen
                seen[(t, sl)] = c
            if k == "head":
                heads[c] = (t, e)
            if k == "tail":
                tails[c] = (t, b)
    assert len(seen) == tiles * slices
    # every cut tile: its head in CTA c (prefix slot c), its tail in CTA c + 1
    assert len(heads) == len(tails)
    for c, (t, b) in tails.items():
        assert heads[c - 1] == (t, b)
