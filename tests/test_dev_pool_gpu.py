"""GPU tests of the device-side expert slot pool (w4_dev_pool_*): the remap
decided on the GPU follows the reference LFU policy step for step, the pool
holds the source experts' bytes, and a routed step captured in a CUDA graph
(ids copied in, remap, fills, routed GEMV) is bitwise the product on the full
expert tensor.

Page "Running a 26B MoE on an 8 GB Jetson by streaming experts from SSD",
section "Streaming without touching a single GPU kernel": the LFU cache of
expert slots, the slot-id tensor and the memcmp bar.
"""

import numpy as np
import pytest
import torch

import oracle
from bit_weight_only_gemv_gb300 import lib, synth
from _helpers import POISON, host_bits, poison_bf16

pytestmark = pytest.mark.gpu


def experts(E, n, k, seed, home="device"):
    qs, ss = n * k // 2, n * k // 16
    full_q = synth.torch_words((E, qs // 4), seed=synth.seed_of(seed, 1), device="cuda")
    full_s = synth.torch_steps((E, ss // 2), seed=synth.seed_of(seed, 2), device="cuda")
    src_q, src_s = full_q, full_s
    if home == "pinned":
        src_q = torch.empty(full_q.shape, dtype=full_q.dtype, pin_memory=True)
        src_s = torch.empty(full_s.shape, dtype=full_s.dtype, pin_memory=True)
        src_q.copy_(full_q)
        src_s.copy_(full_s)
    return full_q, full_s, src_q, src_s, qs, ss


@pytest.mark.parametrize("E,S,k,kind", [(32, 8, 4, "zipf"), (128, 32, 8, "zipf"),
                                        (16, 4, 4, "repeats"), (9, 9, 3, "repeats"),
                                        (64, 2, 1, "zipf")])
def test_device_pool_follows_the_reference_policy(cuda_lib, E, S, k, kind):
    n, K = 64, 256
    full_q, full_s, _, _, qs, ss = experts(E, n, K, E + S)
    pool_q = torch.zeros((S, qs // 4), dtype=torch.int32, device="cuda")
    pool_s = torch.zeros((S, ss // 2), dtype=torch.bfloat16, device="cuda")
    ids = torch.zeros(k, dtype=torch.int32, device="cuda")
    slot_ids = torch.zeros(k, dtype=torch.int32, device="cuda")
    table = torch.full((S,), -1, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pool = lib.DevSlotPool(E, S)
    stage = pool.bind_stage(ids, pool_q, full_q, qs, qs, pool_s, full_s, ss, ss, slot_ids,
                            slot_expert=table, status=status)
    ref = oracle.LFUSlotPoolRef(E, S)
    rng = np.random.default_rng(E * S + k)
    if kind == "zipf":
        trace = synth.moe_trace(E, k, 60, 1.1, 0.7, seed=E + k)
    else:   # repeated ids inside a request, few distinct experts
        trace = [list(rng.integers(0, min(E, S + 2), size=k)) for _ in range(60)]
    misses = 0
    for req in trace:
        ids.copy_(torch.tensor([int(v) for v in req], dtype=torch.int32))
        stage()
        want, miss = ref.step(req)
        misses += len(miss)
        torch.cuda.synchronize()
        assert slot_ids.cpu().tolist() == want
        assert table.cpu().tolist() == ref.expert_in_slot
    assert int(status.item()) == 0
    st = pool.stats()
    assert st == {"requests": k * len(trace), "hits": k * len(trace) - misses, "misses": misses}
    for s_, ex in enumerate(ref.expert_in_slot):   # the slots hold the source bytes
        if ex >= 0:
            assert torch.equal(pool_q[s_], full_q[ex]) and torch.equal(pool_s[s_], full_s[ex])


@pytest.mark.parametrize("home", ["device", "pinned"])
def test_routed_step_in_a_graph_is_bitwise_the_full_tensor(cuda_lib, home):
    E, S, k = 64, 16, 8
    n, K = 704, 2816
    full_q, full_s, src_q, src_s, qs, ss = experts(E, n, K, 5, home)
    pool_q = torch.zeros((S, qs // 4), dtype=torch.int32, device="cuda")
    pool_s = torch.zeros((S, ss // 2), dtype=torch.bfloat16, device="cuda")
    ids_host = torch.zeros(k, dtype=torch.int32).pin_memory()
    ids = torch.zeros(k, dtype=torch.int32, device="cuda")
    slot_ids = torch.zeros(k, dtype=torch.int32, device="cuda")
    table = torch.full((S,), -1, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    x = synth.torch_x((1, K), 7, "cuda")
    scale = synth.torch_x((E, n), 8, "cuda")
    y_pool = torch.empty((k, n), dtype=torch.bfloat16, device="cuda")
    y_full = torch.empty((k, n), dtype=torch.bfloat16, device="cuda")
    pool = lib.DevSlotPool(E, S)
    stage = pool.bind_stage(ids, pool_q, src_q, qs, qs, pool_s, src_s, ss, ss, slot_ids,
                            slot_expert=table, status=status)
    routed = lib.bind_gemv_id_scaled(pool_q, pool_s, slot_ids, x, n, K, S, qs, ss, ids, E,
                                     y_pool, slot_expert=table, scale=scale, status=status)
    full = lib.bind_gemv_id_scaled(full_q, full_s, ids, x, n, K, E, qs, ss, ids, E, y_full,
                                   scale=scale, status=status)
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        ids.copy_(ids_host, non_blocking=True)
        stage(stream=stream)
        routed(pdl=True, stream=stream)
        full(pdl=True, stream=stream)
    ref = oracle.LFUSlotPoolRef(E, S)
    for req in synth.moe_trace(E, k, 40, 1.1, 0.7, seed=9):
        ids_host.copy_(torch.tensor([int(v) for v in req], dtype=torch.int32))
        g.replay()
        torch.cuda.synchronize()
        want, _ = ref.step(req)
        assert slot_ids.cpu().tolist() == want
        assert host_bits(y_pool).tobytes() == host_bits(y_full).tobytes()
    assert int(status.item()) == 0


def test_bad_requests_change_nothing(cuda_lib):
    E, S, k = 16, 2, 3
    n, K = 32, 256
    full_q, full_s, _, _, qs, ss = experts(E, n, K, 11)
    pool_q = torch.zeros((S, qs // 4), dtype=torch.int32, device="cuda")
    pool_s = torch.zeros((S, ss // 2), dtype=torch.bfloat16, device="cuda")
    ids = torch.zeros(k, dtype=torch.int32, device="cuda")
    slot_ids = torch.zeros(k, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pool = lib.DevSlotPool(E, S)
    stage = pool.bind_stage(ids, pool_q, full_q, qs, qs, pool_s, full_s, ss, ss, slot_ids,
                            status=status)
    ref = oracle.LFUSlotPoolRef(E, S)

    def run(req):
        ids.copy_(torch.tensor(req, dtype=torch.int32))
        stage()
        torch.cuda.synchronize()
        return slot_ids.cpu().tolist()

    assert run([3, 3, 5]) == ref.step([3, 3, 5])[0]
    # an id out of range: -1 slot ids, W4_ERR_INDEX, the pool unchanged
    assert run([3, 16, 5]) == [-1, -1, -1]
    assert lib.STATUS[int(status.item())] == "W4_ERR_INDEX"
    status.zero_()
    # more distinct ids than slots: W4_ERR_STATE, unchanged
    assert run([1, 2, 7]) == [-1, -1, -1]
    assert lib.STATUS[int(status.item())] == "W4_ERR_STATE"
    status.zero_()
    # the next valid request is served as if the bad ones had never come
    assert run([5, 9, 9]) == ref.step([5, 9, 9])[0]
    assert int(status.item()) == 0
    # a routed GEMV fed the -1 slot ids leaves its rows unwritten
    run([0, 40, 1])
    status.zero_()
    x = synth.torch_x((1, K), 3, "cuda")
    y = poison_bf16((k, n))
    lib.gemv_id(pool_q, pool_s, slot_ids, x, n, K, S, qs, ss, y=y, status=status)
    torch.cuda.synchronize()
    assert lib.STATUS[int(status.item())] == "W4_ERR_INDEX"
    assert np.all(host_bits(y) == POISON)


def test_device_pool_hand_traces(cuda_lib):
    """The hand-worked traces of the policy (tests/golden/lfu_traces.txt):
    slot ids, the slot table and the miss count at every step."""
    import test_oracle_pins as pins
    n, K = 64, 256
    for name, E, S, steps in pins._read_traces():
        full_q, full_s, _, _, qs, ss = experts(E, n, K, 7 * E + S)
        pool_q = torch.zeros((S, qs // 4), dtype=torch.int32, device="cuda")
        pool_s = torch.zeros((S, ss // 2), dtype=torch.bfloat16, device="cuda")
        table = torch.full((S,), -1, dtype=torch.int32, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        pool = lib.DevSlotPool(E, S)
        stages = {}
        resident = [-1] * S
        for req, want_slots, want_miss in steps:
            k = len(req)
            if k not in stages:      # one bound stage per request length, one pool state
                ids = torch.zeros(k, dtype=torch.int32, device="cuda")
                sl = torch.zeros(k, dtype=torch.int32, device="cuda")
                stages[k] = (ids, sl, pool.bind_stage(ids, pool_q, full_q, qs, qs, pool_s, full_s,
                                                      ss, ss, sl, slot_expert=table,
                                                      status=status))
            ids, sl, stage = stages[k]
            ids.copy_(torch.tensor(req, dtype=torch.int32))
            stage()
            torch.cuda.synchronize()
            for ex, s_ in want_miss:
                resident[s_] = ex
            assert sl.cpu().tolist() == want_slots, name
            assert table.cpu().tolist() == resident, name
        assert int(status.item()) == 0, name
        misses = sum(len(m) for _, _, m in steps)
        requests = sum(len(r) for r, _, _ in steps)
        assert pool.stats() == {"requests": requests, "hits": requests - misses, "misses": misses}
        for s_, ex in enumerate(resident):
            if ex >= 0:
                assert torch.equal(pool_q[s_], full_q[ex]) and torch.equal(pool_s[s_], full_s[ex])
