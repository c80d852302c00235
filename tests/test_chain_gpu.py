"""GPU parity of w4a16_gemv_chain: a list of GEMVs in one persistent launch.

Every task's outputs must be bitwise those of the same product made by the
single calls (w4a16_gemv, w4a16_gemv_id; the per-row arithmetic depends on K
alone), and within the acceptance bound of the fp64 oracle.  Covered: the
compiled dot pairs of the two decoders and of the routed-expert layer, the
generic loop (ragged chunks, padded lane teams), a down projection reading
its gate/up task's output through silu(gate) * up, a routed layer whose
down product reads each expert's own gate/up rows, ids out of range,
repeated launches on one workspace, CUDA-graph replay, and a two-layer slice
of the hidden-5376 decoder at full size.
"""

import numpy as np
import pytest
import torch

import oracle
from bit_weight_only_gemv_gb300 import lib, synth
from _helpers import POISON, dev_bf16, dev_words, host_bits, poison_bf16

pytestmark = pytest.mark.gpu


def workspace(tasks):
    return torch.zeros(lib.chain_workspace_bytes(tasks), dtype=torch.uint8, device="cuda")


def single_gemv(qw, st, x, silu_mul=False):
    n, k = qw.shape[0], qw.shape[1] * 8
    need = lib.workspace_bytes(1, n, k, "cuda" if silu_mul else None)
    ws = torch.zeros(max(16, need), dtype=torch.uint8, device="cuda") if need else None
    return lib.gemv(qw, st, x.view(1, -1), workspace=ws, silu_mul=silu_mul)


def dense_chain(rng, shapes, rows_checked=None):
    """Tasks of the given (N, K), each on its own activation row, each
    depending on the one before."""
    hosts, tasks = [], []
    for i, (n, k) in enumerate(shapes):
        qw_h = synth.np_words(rng, (n, k // 8))
        st_h = synth.np_steps(rng, (n, k // 32))
        x_h = synth.np_x(rng, (1, k))
        qw, st, x = dev_words(qw_h), dev_bf16(st_h), dev_bf16(x_h)
        y = poison_bf16((n,))
        hosts.append((qw_h, st_h, x_h))
        tasks.append(lib.gemv_task(qw, st, x, y, dep=i - 1))
    return hosts, tasks


def check_dense(hosts, tasks, sample=None):
    for (qw_h, st_h, x_h), t in zip(hosts, tasks):
        yb = host_bits(t["y"])
        assert not np.any(yb == POISON), "unwritten outputs"
        ref = host_bits(single_gemv(t["qw"], t["st"], t["x"]))[0]
        assert np.array_equal(yb, ref), "not the bits of w4a16_gemv"
        rows = np.arange(yb.size) if sample is None or yb.size <= sample else \
            np.random.default_rng(0).choice(yb.size, sample, replace=False)
        y_ref = oracle.gemv_ref(qw_h[rows], st_h[rows], x_h)[0]
        a_ref = oracle.gemv_abs_ref(qw_h[rows], st_h[rows], x_h)[0]
        assert oracle.within_bound(yb[rows], y_ref, a_ref)


@pytest.mark.parametrize("shapes", [
    [(600, 5376), (333, 5376), (140, 21504), (1000, 5376)],         # hidden-5376 dot pair
    [(700, 2048), (2048, 2048), (300, 8192), (5000, 2048)],         # hidden-2048 dot pair
    [(300, 1184), (77, 3232), (20, 14176), (129, 416), (64, 96)],   # generic loop
    [(1, 2048)],                                                    # one row, one task
])
def test_dense_chain_matches_single_calls_and_oracle(cuda_lib, shapes):
    rng = np.random.default_rng(sum(n + k for n, k in shapes))
    hosts, tasks = dense_chain(rng, shapes)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = workspace(tasks)
    lib.gemv_chain(tasks, ws, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert int(ws.view(torch.int32).abs().sum()) == 0      # counters re-armed
    check_dense(hosts, tasks)


def test_gated_down_reads_its_gate_up_task(cuda_lib):
    # merged gate/up, then the down projection on silu(gate) * up of its output
    rng = np.random.default_rng(21)
    hid, inter = 2048, 8192
    gu_q = synth.np_words(rng, (2 * inter, hid // 8))
    gu_s = synth.np_steps(rng, (2 * inter, hid // 32))
    dn_q = synth.np_words(rng, (hid, inter // 8))
    dn_s = synth.np_steps(rng, (hid, inter // 32))
    x_h = synth.np_x(rng, (1, hid))
    gu_y = poison_bf16((2 * inter,))
    dn_y = poison_bf16((hid,))
    tasks = [lib.gemv_task(dev_words(gu_q), dev_bf16(gu_s), dev_bf16(x_h), gu_y),
             lib.gemv_task(dev_words(dn_q), dev_bf16(dn_s), gu_y, dn_y, dep=0, silu_mul=True)]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib.gemv_chain(tasks, workspace(tasks), status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(host_bits(gu_y), host_bits(single_gemv(tasks[0]["qw"], tasks[0]["st"],
                                                                 tasks[0]["x"]))[0])
    ref = single_gemv(tasks[1]["qw"], tasks[1]["st"], gu_y, silu_mul=True)
    assert np.array_equal(host_bits(dn_y), host_bits(ref)[0])
    y_ref, a_ref = oracle.gemv_values_ref(dn_q, dn_s, oracle.silu_mul_ref(host_bits(gu_y)[None]))
    assert oracle.within_bound(host_bits(dn_y)[None], y_ref, a_ref)


def routed_layer(rng, E, H, I, ids_h, pad=0):
    """Experts of merged gate/up (2I x H) and down (H x I), each a byte block
    of its own with the given padding; the routed chain of one layer."""
    gq = synth.np_words(rng, (E, 2 * I, H // 8))
    gs = synth.np_steps(rng, (E, 2 * I, H // 32))
    dq = synth.np_words(rng, (E, H, I // 8))
    ds = synth.np_steps(rng, (E, H, I // 32))
    x_h = synth.np_x(rng, (1, H))
    k = len(ids_h)
    ids = torch.from_numpy(np.asarray(ids_h, np.int32)).cuda()
    gu_y = poison_bf16((k, 2 * I))
    dn_y = poison_bf16((k, H))
    tasks = [lib.gemv_id_task(dev_words(gq.reshape(E, -1)), dev_bf16(gs.reshape(E, -1)), ids,
                              dev_bf16(x_h), gu_y, 2 * I, H, E, 2 * I * H // 2, 2 * I * H // 16),
             lib.gemv_id_task(dev_words(dq.reshape(E, -1)), dev_bf16(ds.reshape(E, -1)), ids,
                              gu_y, dn_y, H, I, E, H * I // 2, H * I // 16, dep=0,
                              silu_mul=True)]
    return (gq, gs, dq, ds, x_h), tasks


@pytest.mark.parametrize("E,H,I,ids_h", [
    (16, 2816, 704, [3, 9, 0, 15, 3, 7, 11, 2]),     # the routed decoder's dot pair
    (6, 1024, 96, [5, 1, 1, 4]),                      # generic loop
])
def test_routed_layer_chain(cuda_lib, E, H, I, ids_h):
    rng = np.random.default_rng(E + H + I)
    (gq, gs, dq, ds, x_h), tasks = routed_layer(rng, E, H, I, ids_h)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib.gemv_chain(tasks, workspace(tasks), status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    gu = host_bits(tasks[0]["y"])
    dn = host_bits(tasks[1]["y"])
    assert not np.any(gu == POISON) and not np.any(dn == POISON)
    # gate/up rows: bitwise w4a16_gemv_id, and the oracle by expert id
    ref = lib.gemv_id(tasks[0]["qw"], tasks[0]["st"], tasks[0]["ids"], tasks[0]["x"], 2 * I, H,
                      E, 2 * I * H // 2, 2 * I * H // 16)
    torch.cuda.synchronize()
    assert np.array_equal(gu, host_bits(ref))
    a = np.stack([oracle.gemv_abs_ref(gq[e], gs[e], x_h)[0] for e in ids_h])
    assert oracle.within_bound(gu, oracle.gemv_id_ref(gq, gs, np.array(ids_h), x_h), a)
    # down rows: expert ids[i] on silu(gate_i) * up_i of its own gate/up row
    for i, e in enumerate(ids_h):
        r = single_gemv(dev_words(dq[e]), dev_bf16(ds[e]), tasks[0]["y"][i], silu_mul=True)
        assert np.array_equal(dn[i], host_bits(r)[0])
        y_ref, a_ref = oracle.gemv_values_ref(dq[e], ds[e], oracle.silu_mul_ref(gu[i][None]))
        assert oracle.within_bound(dn[i][None], y_ref, a_ref)


def test_routed_bad_id_leaves_rows_unwritten(cuda_lib):
    rng = np.random.default_rng(5)
    E, H, I = 6, 1024, 96
    ids_h = [2, 6, 1, -1]
    (gq, gs, dq, ds, x_h), tasks = routed_layer(rng, E, H, I, ids_h)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = workspace(tasks)
    lib.gemv_chain(tasks, ws, status)
    torch.cuda.synchronize()
    assert lib.STATUS[int(status.item())] == "W4_ERR_INDEX"
    gu, dn = host_bits(tasks[0]["y"]), host_bits(tasks[1]["y"])
    for i in (1, 3):
        assert np.all(gu[i] == POISON) and np.all(dn[i] == POISON)
    for i in (0, 2):
        assert not np.any(gu[i] == POISON) and not np.any(dn[i] == POISON)
    assert int(ws.view(torch.int32).abs().sum()) == 0      # the launch still completed


def test_repeated_launches_and_graph_replay(cuda_lib):
    rng = np.random.default_rng(8)
    hosts, tasks = dense_chain(rng, [(900, 2048), (3000, 2048), (700, 8192)])
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = workspace(tasks)
    call = lib.bind_gemv_chain(tasks, ws, status)
    call()
    torch.cuda.synchronize()
    first = [host_bits(t["y"]).copy() for t in tasks]
    for _ in range(20):                          # back to back, as programmatic dependents
        call(pdl=True)
    torch.cuda.synchronize()
    for t, f in zip(tasks, first):
        assert np.array_equal(host_bits(t["y"]), f)
    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        call(stream=stream)
    for t in tasks:
        t["y"].view(torch.int16).fill_(POISON)
    for _ in range(5):
        g.replay()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for t, f in zip(tasks, first):
        assert np.array_equal(host_bits(t["y"]), f)
    assert int(ws.view(torch.int32).abs().sum()) == 0
    check_dense(hosts, tasks)


def test_two_layers_of_the_hidden_5376_decoder_at_full_size(cuda_lib):
    # merged q/k/v, o, merged gate/up, down, twice, then the 262144 x 5376 lm_head
    shapes = [(9472, 5376), (5376, 5376), (43008, 5376), (5376, 21504)] * 2 + [(262144, 5376)]
    rng = np.random.default_rng(60)
    hosts, tasks = [], []
    for i, (n, k) in enumerate(shapes):
        qw = synth.torch_words((n, k // 8), synth.seed_of(60, i, 1), "cuda")
        st = synth.torch_steps((n, k // 32), synth.seed_of(60, i, 2), "cuda")
        x = synth.torch_x((k,), synth.seed_of(60, i, 3), "cuda")
        tasks.append(lib.gemv_task(qw, st, x, poison_bf16((n,)), dep=i - 1))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib.gemv_chain(tasks, workspace(tasks), status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for i, t in enumerate(tasks):
        yb = host_bits(t["y"])
        assert not np.any(yb == POISON)
        assert np.array_equal(yb, host_bits(single_gemv(t["qw"], t["st"], t["x"]))[0])
        rows = rng.choice(yb.size, 64, replace=False)
        qw_h = t["qw"][torch.from_numpy(rows).cuda()].cpu().numpy().view(np.uint32)
        st_h = t["st"][torch.from_numpy(rows).cuda()].view(torch.int16).cpu().numpy() \
            .view(np.uint16)
        x_h = host_bits(t["x"])[None]
        assert oracle.within_bound(yb[rows], oracle.gemv_ref(qw_h, st_h, x_h)[0],
                                   oracle.gemv_abs_ref(qw_h, st_h, x_h)[0])
