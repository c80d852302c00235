#!/usr/bin/env python3
"""Benchmark: batch-1 decode pass of a W4A16 decoder, by default the 60-layer
hidden-5376 one.

One step = one decode pass over the whole hot path, replayed as one CUDA
graph: the embed-row gather (tied 262144 x 5376 table), for each of 60 layers
the merged q/k/v (9472 x 5376), o (5376 x 5376), merged gate/up (43008 x 5376)
and down (5376 x 21504) GEMVs, and the lm_head GEMV over the tied table
(262144 x 5376); 242 kernels, chained with programmatic dependent launch.
All weights and activations are seeded synthetic data (uniform codes,
|N(0,1)|*0.02/8 steps, N(0,1) activations); each layer's q/k/v share one
activation row and gate/up share another.  A pass reads 15.2 GB of packed
weights, far more than the 129 MB L2, so every step streams from HBM.
`--workload dense-35L-h2048` runs the 35-layer hidden-2048 decoder (with its
per-layer table), `--workload moe-30L-h2816` the routed-expert decoder.

Prints one JSON line (see --help).  `--impl reference` times the fp64 CPU
oracle instead, on a bounded sample of the same pass.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from bit_weight_only_gemv_gb300 import metrics, synth  # noqa: E402

METRIC = "W4A16 GEMV HBM GB/s and % of GB300 peak; decode-equivalent tok/s at batch 1"
DENSE_WORKLOADS = {"dense-35L-h2048": synth.dense_2048, "dense-60L-h5376": synth.dense_5376}
UNIT = "tok/s"
# the arithmetic of the CUDA-core path (batch 1): exact fp16 products of
# (code - 8) and power-of-two-scaled activations, fp16 partial sums of 4
# products, fp32 accumulation
DTYPE = "w4a16: exact f16 products, f16 partial sums of 4 products, f32 accumulate"
NOMINAL_HBM_GBPS = 8000.0
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}


# ------------------------------------------------------------------ helpers
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK["hbm_gbs"], "fallback"


def max_over_ranks(value: float, device) -> float:
    """Largest value over all ranks (identity for one process)."""
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled in the background."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, period_ms: int = 100):
        self.index, self.period = index, period_ms
        self.proc = None
        self.path = None
        self.t0 = self.t1 = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.period)],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        rows = []
        if self.path and os.path.exists(self.path):
            for line in open(self.path):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
                except ValueError:
                    continue
            os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, flags in rows for i, f in enumerate(flags)
                          if f.lower() == "active"})
        sm = sorted(r[0] for r in rows)
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------ workload
class DecodePass:
    """Device-resident weights, inputs and outputs of one decode pass."""

    def __init__(self, model: synth.DenseDecoder, device, seed: int = 0, merge: bool = True,
                 gated: bool = False, l2_next_bytes: int = 0):
        from bit_weight_only_gemv_gb300 import lib
        self.lib = lib
        # each GEMV brings up to this many bytes of the next GEMV's weights
        # (its leading rows) into L2 once its own tiles are requested
        self.l2_next_bytes = l2_next_bytes
        # gated MLP: each layer's down projection reads the merged gate/up
        # output through silu(gate) * up instead of its own activation row
        self.gated = gated and merge
        self.model = model
        self.dev = device
        self.merge = merge
        h, V = model.hidden, model.vocab
        s = seed
        # tied embed / lm_head table and the per-layer table
        self.emb_qw = synth.torch_words((V, h // 8), synth.seed_of(s, 1), device)
        self.emb_st = synth.torch_steps((V, h // 32), synth.seed_of(s, 2), device)
        pw = model.per_layer_width
        self.ple_qw = synth.torch_words((V, pw // 8), synth.seed_of(s, 3), device) if pw else None
        self.ple_st = synth.torch_steps((V, pw // 32), synth.seed_of(s, 4), device) if pw else None
        # weight matrices per layer; projections that read the same activation
        # (q/k/v, gate/up) are stored as one row-concatenated matrix when merged
        groups = []
        for pr in model.projs:
            if merge and groups and groups[-1][0] == pr.x_key and groups[-1][1][0].k == pr.k:
                groups[-1][1].append(pr)
            else:
                groups.append((pr.x_key, [pr]))
        self.mats = []   # (layer, name, n, k, x_key, qw, st)
        for li in range(model.layers):
            for gi, (xk, prs) in enumerate(groups):
                n = sum(p.n for p in prs)
                k = prs[0].k
                name = "+".join(p.name for p in prs)
                qw = synth.torch_words((n, k // 8), synth.seed_of(s, 10, li, gi), device)
                st = synth.torch_steps((n, k // 32), synth.seed_of(s, 11, li, gi), device)
                self.mats.append((li, name, n, k, xk, qw, st))
        # activations: one row per distinct (layer, x_key), plus the final row
        self.x_keys = []
        self.k_of = {}
        for li, name, n, k, xk, _, _ in self.mats:
            if (li, xk) not in self.k_of:
                self.x_keys.append((li, xk))
                self.k_of[(li, xk)] = k
        total_x = sum(self.k_of[k] for k in self.x_keys) + h
        self.x_flat = synth.torch_x((total_x,), synth.seed_of(s, 20), device)
        self.x_off = {}
        off = 0
        for k in self.x_keys:
            self.x_off[k] = off
            off += self.k_of[k]
        self.x_off["final"] = off
        self.ids = torch.tensor([int(synth.seed_of(s, 30) % V)], dtype=torch.int32, device=device)
        # outputs, one region per launch
        self.y_off = {}
        off = 0
        for li, name, n, k, xk, _, _ in self.mats:
            self.y_off[(li, name)] = off
            off += n
        self.y_off["logits"] = off
        off += V
        self.y_flat = torch.empty(off, dtype=torch.bfloat16, device=device)
        self.emb_row = torch.empty((1, h), dtype=torch.bfloat16, device=device)
        self.ple_row = torch.empty((1, pw), dtype=torch.bfloat16, device=device) if pw else None
        ws = 0
        for li, name, n, k, xk, _, _ in self.mats:
            ws = max(ws, lib.workspace_bytes(1, n, k))
        ws = max(ws, lib.workspace_bytes(1, V, h))
        self.ws = torch.zeros(max(ws, 16), dtype=torch.uint8, device=device) if ws else None
        self.status = torch.zeros(1, dtype=torch.int32, device=device)

    def x(self, key, k):
        o = self.x_off[key]
        return self.x_flat[o:o + k].view(1, k)

    def launches(self):
        """(kind, shape, callable) for every kernel of the pass, in stream order."""
        lib, m = self.lib, self.model
        out = []
        out.append(("gather", (1, m.hidden), lambda pdl: lib.embed_gather(
            self.emb_qw, self.emb_st, self.ids, out=self.emb_row, status=self.status, pdl=pdl)))
        if m.per_layer_width:
            out.append(("gather", (1, m.per_layer_width), lambda pdl: lib.embed_gather(
                self.ple_qw, self.ple_st, self.ids, out=self.ple_row, status=self.status, pdl=pdl)))
        specs = []   # (n, k, qw, st, x, y, gated) of every GEMV in order
        for li, name, n, k, xk, qw, st in self.mats:
            x = self.x((li, xk), k)
            gated = self.gated and name == "down"
            if gated:
                og = self.y_off[(li, "gate+up")]
                x = self.y_flat[og:og + 2 * k].view(1, 2 * k)
            o = self.y_off[(li, name)]
            specs.append((n, k, qw, st, x, self.y_flat[o:o + n].view(1, n), gated))
        o = self.y_off["logits"]
        specs.append((m.vocab, m.hidden, self.emb_qw, self.emb_st, self.x("final", m.hidden),
                      self.y_flat[o:o + m.vocab].view(1, m.vocab), False))
        for i, (n, k, qw, st, x, y, gated) in enumerate(specs):
            nxt = specs[i + 1] if i + 1 < len(specs) else None
            l2 = self.next_ranges(nxt[0], nxt[1], nxt[2], nxt[3]) if nxt else None
            out.append(("gemv", (1, n, k), self._gemv(qw, st, x, y, gated, l2)))
        return out

    def next_ranges(self, n, k, qw, st):
        """The leading rows of an (n, k) matrix's codes and steps that fit
        l2_next_bytes, as w4_l2_range entries (None when disabled)."""
        if self.l2_next_bytes <= 0:
            return None
        rows = min(n, self.l2_next_bytes // (k // 2 + k // 16))
        if rows < 1:
            return None
        return self.lib.l2_ranges([(qw, rows * (k // 2)), (st, rows * (k // 16))])

    def chain_launches(self):
        """The same pass as the row gather(s) plus ONE w4a16_gemv_chain launch
        of every GEMV, each task depending on the one before (as in a
        decoder, where each projection reads what the previous produced)."""
        lib, m = self.lib, self.model
        out = [e for e in self.launches() if e[0] == "gather"]
        tasks, shapes = [], []
        for li, name, n, k, xk, qw, st in self.mats:
            x = self.x((li, xk), k).view(-1)
            gated = self.gated and name == "down"
            if gated:
                og = self.y_off[(li, "gate+up")]
                x = self.y_flat[og:og + 2 * k]
            o = self.y_off[(li, name)]
            tasks.append(lib.gemv_task(qw, st, x, self.y_flat[o:o + n], dep=len(tasks) - 1,
                                       silu_mul=gated))
            shapes.append((1, n, k))
        o = self.y_off["logits"]
        tasks.append(lib.gemv_task(self.emb_qw, self.emb_st, self.x("final", m.hidden).view(-1),
                                   self.y_flat[o:o + m.vocab], dep=len(tasks) - 1))
        shapes.append((1, m.vocab, m.hidden))
        self.chain_ws = torch.zeros(lib.chain_workspace_bytes(tasks), dtype=torch.uint8,
                                    device=self.dev)
        call = lib.bind_gemv_chain(tasks, self.chain_ws, self.status)
        self.chain_plan = lib.chain_plan(tasks)
        out.append(("chain", shapes, lambda pdl: call(pdl=pdl)))
        return out

    def _gemv(self, qw, st, x, y, gated=False, l2_next=None):
        lib = self.lib
        return lambda pdl: lib.gemv(qw, st, x, y=y, workspace=self.ws, status=self.status, pdl=pdl,
                                    silu_mul=gated, l2_next=l2_next)

    def step_bytes(self):
        return step_bytes_of(self.model)

    def host_inputs(self):
        """Pinned host copies of the per-step inputs (token id, activation rows)."""
        return (self.ids.cpu().pin_memory(), self.x_flat.cpu().pin_memory())

    def host_outputs(self):
        o = self.y_off["logits"]
        return torch.empty(self.model.vocab, dtype=torch.bfloat16).pin_memory(), o


def kernel_key(kind, shape, lib):  # ncu names the instantiation
    if kind == "gather":
        return "gather_kernel"
    if kind == "chain":
        return "chain_kernel"
    M, N, K = shape
    p = lib.plan(M, N, K)
    if p["path"] == 2:
        return "tc_kernel"
    dense = "1" if p["slices"] == 1 else "0"   # dense whole-row instantiation (as ncu prints it)
    return (f"gemv_kernel<{p['rows_per_call']}, {p['rows_per_lane']}, "
            f"{p['tmpl_team']}, {p['tmpl_chunk']}, {dense}>")


def capture(fns, stream, pdl=True):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i, f in enumerate(fns):
            f(pdl and i > 0)
    return g


def time_replays(g, stream, steps):
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def code_tokens(text: str) -> str:
    """C/C++/CUDA source with comments removed and each run of blank space
    outside string and character literals made one line break (if it held
    one: preprocessor lines keep their ends) or one space: the part of a
    source file that can change what it compiles to."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        elif c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif c.isspace():
            j = i
            while j < n and text[j].isspace():
                j += 1
            out.append("\n" if "\n" in text[i:j] else " ")
            i = j
        else:
            out.append(c)
            i += 1
    return re.sub(r"\s*\n\s*", "\n", re.sub(r"[ ]+", " ", "".join(out))).strip()


def kernel_source_digest() -> str:
    """sha256 over the code tokens of csrc/gemv.cu then csrc/common.cuh."""
    h = hashlib.sha256()
    for f in ("gemv.cu", "common.cuh"):
        path = os.path.join(ROOT, "bit_weight_only_gemv_gb300", "csrc", f)
        h.update(code_tokens(open(path, encoding="utf-8").read()).encode())
    return h.hexdigest()


def traffic_from_profile(kernel):
    """DRAM bytes per launch from the committed ncu summary, if still current."""
    path = os.path.join(ROOT, "profiles", "gemv_kernel_traffic.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"source_sha256:\s*([0-9a-f]+)", text)
    if not m or m.group(1) != kernel_source_digest():
        return None
    for line in text.splitlines():
        mm = re.match(r"\s*-\s*kernel:\s*(.+?)\s*\|\s*dram_bytes_per_launch:\s*([0-9.]+)\s*\|"
                      r"\s*workload:\s*(.+)$", line)
        if mm and mm.group(1) == kernel:
            return {"bytes": float(mm.group(2)), "workload": mm.group(3)}
    return None


# ------------------------------------------------------------------ CPU oracle
# One sample definition serves the main line's cpu_baseline and the
# --impl reference arm: a bounded slice of one decode pass of the same
# workload, run by the fp64 oracle, its time scaled to the whole pass by
# algorithmic bytes.
SAMPLE_ROWS = 256          # rows of each sampled matrix
CPU_BASELINE_SECONDS = 10.0


def merged_groups(model, merge=True):
    """Projections that one GEMV serves, in launch order: q/k/v and gate/up
    row-concatenated when merged (they read the same activation row)."""
    groups = []
    for pr in model.projs:
        if merge and groups and groups[-1][0] == pr.x_key and groups[-1][1][0].k == pr.k:
            groups[-1][1].append(pr)
        else:
            groups.append((pr.x_key, [pr]))
    return [("+".join(p.name for p in prs), sum(p.n for p in prs), prs[0].k) for _, prs in groups]


def sample_rows(n, rows=SAMPLE_ROWS):
    """Evenly spaced row indices of an n-row matrix."""
    r = min(rows, n)
    return np.arange(r, dtype=np.int64) * (n // r)


def dense_sample_from_recipe(model, merge=True, seed=0):
    """The sample drawn on the host by the workload's recipe (same shapes and
    distributions as the GPU arm's weights): layer 0's GEMVs as launched,
    SAMPLE_ROWS rows each, SAMPLE_ROWS lm_head rows, the row gathers."""
    rng = np.random.default_rng(seed)
    items = []
    for name, n, k in merged_groups(model, merge):
        r = len(sample_rows(n))
        items.append(("gemv", synth.np_words(rng, (r, k // 8)), synth.np_steps(rng, (r, k // 32)),
                      synth.np_x(rng, (1, k))))
    r = len(sample_rows(model.vocab))
    h = model.hidden
    items.append(("gemv", synth.np_words(rng, (r, h // 8)), synth.np_steps(rng, (r, h // 32)),
                  synth.np_x(rng, (1, h))))
    for w in (h, model.per_layer_width):
        if w:
            items.append(("gather", synth.np_words(rng, (1, w // 8)),
                          synth.np_steps(rng, (1, w // 32)), None))
    return items


def dense_sample_from_device(dp):
    """The same sample, read back from the bytes the GPU arm uses."""
    m = dp.model
    items = []

    def rows_of(qw, st, idx):
        t = torch.from_numpy(idx).to(dp.dev)
        return (qw[t].cpu().numpy().view(np.uint32),
                st[t].view(torch.int16).cpu().numpy().view(np.uint16))

    for li, name, n, k, xk, qw, st in dp.mats:
        if li != 0:
            continue
        q, s_ = rows_of(qw, st, sample_rows(n))
        items.append(("gemv", q, s_, dp.x((0, xk), k).view(torch.int16).cpu().numpy().view(np.uint16)))
    q, s_ = rows_of(dp.emb_qw, dp.emb_st, sample_rows(m.vocab))
    items.append(("gemv", q, s_, dp.x("final", m.hidden).view(torch.int16).cpu().numpy()
                  .view(np.uint16)))
    tid = np.array([int(dp.ids.item())])
    items.append(("gather",) + rows_of(dp.emb_qw, dp.emb_st, tid) + (None,))
    if m.per_layer_width:
        items.append(("gather",) + rows_of(dp.ple_qw, dp.ple_st, tid) + (None,))
    return items


def moe_sample_from_recipe(cfg, seed=0):
    """Routed workload: one layer's top-k experts, SAMPLE_ROWS // 2 rows of
    each expert's merged gate/up (shared activation row) and of its down
    projection (its own activation row)."""
    rng = np.random.default_rng(seed)
    items = []
    r = SAMPLE_ROWS // 2
    for n, k in ((2 * cfg.expert_inter, cfg.hidden), (cfg.hidden, cfg.expert_inter)):
        x = synth.np_x(rng, (1, k))
        for _ in range(cfg.top_k):
            items.append(("gemv", synth.np_words(rng, (min(r, n), k // 8)),
                          synth.np_steps(rng, (min(r, n), k // 32)), x))
    return items


def sample_bytes(items):
    nb = 0
    for kind, qw, st, x in items:
        if kind == "gemv":
            nb += metrics.gemv_bytes(1, qw.shape[0], qw.shape[1] * 8)
        else:
            nb += metrics.gather_bytes(1, qw.shape[1] * 8)
    return nb


def run_oracle_sample(items):
    """Seconds the fp64 oracle takes over the sample."""
    import oracle
    t0 = time.perf_counter()
    for kind, qw, st, x in items:
        if kind == "gemv":
            oracle.gemv_ref(qw, st, x)
        else:
            oracle.gather_ref(qw, st, np.array([0]))
    return time.perf_counter() - t0


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def sample_note(items, pass_bytes):
    return (f"{len(items)} pieces of one pass (layer 0's GEMVs as launched, {SAMPLE_ROWS} rows "
            f"each, {SAMPLE_ROWS} lm_head rows, the row gathers; {sample_bytes(items):,} of "
            f"{pass_bytes:,} algorithmic bytes), fp64 NumPy oracle; time scaled to the whole "
            "pass by algorithmic bytes; NumPy may use BLAS threads on the listed cores")


_ONE_CORE_CHILD = r"""
import os, sys, time
import numpy as np
sys.path.insert(0, sys.argv[1])
try:
    os.sched_setaffinity(0, {sorted(os.sched_getaffinity(0))[0]})
except Exception:
    pass
import oracle
z = np.load(sys.argv[2])
items = []
for i in range(int(z["n"])):
    items.append((str(z["k%d" % i]), z["q%d" % i], z["s%d" % i],
                  z["x%d" % i] if ("x%d" % i) in z.files else None))
reps, spent, seconds = 0, 0.0, float(sys.argv[3])
while reps == 0 or spent < seconds:
    t0 = time.perf_counter()
    for kind, qw, st, x in items:
        if kind == "gemv":
            oracle.gemv_ref(qw, st, x)
        else:
            oracle.gather_ref(qw, st, np.array([0]))
    spent += time.perf_counter() - t0
    reps += 1
print(spent / reps * 1e3, reps)
"""


def one_core_sample_ms(items, seconds=5.0):
    """ms per run of the same sample in a child process held to one core
    (its BLAS and OpenMP pools one thread each), or None if it failed."""
    with tempfile.TemporaryDirectory() as d:
        path = os.path.join(d, "sample.npz")
        arrays = {"n": np.array(len(items))}
        for i, (kind, qw, st, x) in enumerate(items):
            arrays[f"k{i}"], arrays[f"q{i}"], arrays[f"s{i}"] = np.array(kind), qw, st
            if x is not None:
                arrays[f"x{i}"] = x
        np.savez(path, **arrays)
        env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1",
                   MKL_NUM_THREADS="1", BLIS_NUM_THREADS="1")
        try:
            out = subprocess.run([sys.executable, "-c", _ONE_CORE_CHILD, ROOT, path,
                                  str(seconds)], env=env, capture_output=True, text=True,
                                 timeout=60 + 4 * seconds)
            ms, reps = out.stdout.split()[:2]
            return float(ms), int(reps)
        except Exception:
            return None


def cpu_baseline_of(items, pass_bytes, seconds=CPU_BASELINE_SECONDS, one_core=True,
                    one_core_seconds=5.0):
    """The oracle on the sample, repeated for about `seconds`; tok/s scaled
    to whole passes.  one_core: also the same sample on one core (for about
    one_core_seconds)."""
    reps, spent = 0, 0.0
    while reps == 0 or spent < seconds:
        spent += run_oracle_sample(items)
        reps += 1
    per_token = spent / reps * pass_bytes / sample_bytes(items)
    out = {"value": 1.0 / per_token, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
           "sample": sample_note(items, pass_bytes) + f"; {reps} repetitions, {spent:.1f} s",
           "sample_ms": spent / reps * 1e3, "extrapolated_ms_per_token": per_token * 1e3,
           "cpu_count": os.cpu_count(), "affinity_cores": cpu_cores()}
    if one_core:
        r = one_core_sample_ms(items, one_core_seconds)
        if r is not None:
            ms1, reps1 = r
            per1 = ms1 * 1e-3 * pass_bytes / sample_bytes(items)
            out["one_core"] = {"value": 1.0 / per1, "unit": UNIT, "sample_ms": ms1,
                               "extrapolated_ms_per_token": per1 * 1e3, "repetitions": reps1,
                               "note": "the same sample in a child process held to one core, "
                                       "BLAS and OpenMP pools of one thread"}
    return out


# ------------------------------------------------------------------ arms
def step_bytes_of(model):
    b = metrics.gather_bytes(1, model.hidden)
    if model.per_layer_width:
        b += metrics.gather_bytes(1, model.per_layer_width)
    for pr in model.projs:
        b += model.layers * metrics.gemv_bytes(1, pr.n, pr.k)
    return b + metrics.gemv_bytes(1, model.vocab, model.hidden)


def moe_step_bytes(cfg):
    I, H, k_top = cfg.expert_inter, cfg.hidden, cfg.top_k
    return cfg.layers * (metrics.gemv_id_bytes(k_top, 1, 2 * I, H) +
                         metrics.gemv_id_bytes(k_top, k_top, H, I))


def dense_config(model, args, world, step_bytes):
    """config object of a dense decode pass (shared by both arms)."""
    n_mats = len(merged_groups(model, not args.separate)) * model.layers
    return {"workload": f"{model.name} decode pass, batch 1 (gathers, {model.layers} "
                        f"layers of q/k/v/o/gate/up/down GEMVs, {model.vocab}x"
                        f"{model.hidden} lm_head)",
            "projections": f"separate ({len(model.projs) * model.layers} GEMVs)"
            if args.separate else
            f"merged: q/k/v and gate/up row-concatenated ({n_mats} GEMVs)",
            "gated_mlp": ("each down projection reads its layer's gate/up output "
                          "through silu(gate) * up (fused into its activation staging; "
                          "bytes_per_step counts one activation row)"
                          if args.gated_mlp and not args.separate else None),
            "launch": ("the row gather(s), then every GEMV of the pass in ONE w4a16_gemv_chain "
                       "launch, each task waiting for the one before"
                       if getattr(args, "chain", False) else
                       "one launch per GEMV, chained with programmatic dependent launch"),
            "l2_next": (f"each GEMV brings up to {args.l2_next_mb:g} MiB of the next GEMV's "
                        "weights into L2 once its own tiles are requested "
                        "(w4a16_gemv_prefetch_l2)"
                        if getattr(args, "l2_next_mb", 0) > 0 and not getattr(args, "chain", False)
                        else None),
            "global_batch": world, "parallelism": f"replicas x{world}",
            "bytes_per_step": step_bytes,
            "l2": f"inputs larger than L2 ({step_bytes / 1e9:.2f} GB of weights per step, "
                  "129 MB L2)"}


def moe_config(cfg, args, world):
    """config object of the routed-expert decode workload (shared by both arms)."""
    E, S, H, I, k_top, L = (cfg.experts, cfg.slots, cfg.hidden, cfg.expert_inter, cfg.top_k,
                            cfg.layers)
    device_pool = args.pool == "device"
    return {"workload": f"{cfg.name}: routed decode, batch 1, {L} layers, top-{k_top} of "
                        f"{E} experts (Zipf {cfg.zipf_s}, repeat {cfg.repeat_p}), "
                        f"{S}-slot LFU pool per layer; per layer merged gate/up "
                        f"{2 * I}x{H} and down {H}x{I} through w4a16_gemv_id",
            "global_batch": world, "parallelism": f"replicas x{world}",
            "timed": ("one CUDA graph replay per step: the step's router ids picked "
                      "on the device, per layer the device LFU remap, pool copies and "
                      "slot ids, 2 gemv_id (CUDA events)" if device_pool else
                      "eager steps: host LFU remap + pool copies + slot ids + 2 gemv_id "
                      "per layer (CUDA events)"),
            "pool_layout": "one 32-slot pool per layer; a slot holds an expert's gate/up "
                           "and down codes (and, in a second pool array, steps)",
            "expert_home": ("page-locked host memory, pool fills over NVLink-C2C"
                            if args.expert_home == "host" else "HBM"),
            "shared_ffn": {"none": None,
                           "serial": "dense FFN of one expert's shape per layer, after "
                                     "the pool fill on the same stream",
                           "overlap": "dense FFN of one expert's shape per layer, the "
                                      "pool fill beside it on a second stream, joined "
                                      "before the routed GEMVs"}[args.shared_ffn],
            "routed_ffn": ("one w4a16_gemv_chain launch per layer: routed gate/up, then each "
                           "expert's down product on silu(gate) * up of its own gate/up rows"
                           if getattr(args, "chain", False) else
                           "two w4a16_gemv_id launches per layer, down on its own activation "
                           "rows" + ("" if getattr(args, "no_ids_final", False) else
                                     "; the down call's weight copies start before its "
                                     "dependency wait (W4_FLAG_IDS_FINAL: its ids are the "
                                     "gate/up call's)")),
            "expert_vectors": ("per-expert output scales (gate/up, down) and down "
                               "biases by real id, slot table checked, "
                               "w4a16_gemv_id_scaled; real ids copied to the device "
                               "once per step" if args.expert_vectors else None)}


def run_reference(args, world, rank):
    """The CPU oracle, as it stands, on the host cores: each step one run of
    the bounded sample of the selected workload's pass."""
    if rank != 0:
        return 0
    if args.workload.startswith("moe"):
        cfg = synth.moe_2816()
        items = moe_sample_from_recipe(cfg)
        pass_bytes = moe_step_bytes(cfg)
        config = moe_config(cfg, args, world)
    else:
        model = DENSE_WORKLOADS[args.workload]()
        items = dense_sample_from_recipe(model, merge=not args.separate)
        pass_bytes = step_bytes_of(model)
        config = dense_config(model, args, world, pass_bytes)
    for _ in range(args.warmup):
        run_oracle_sample(items)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run_oracle_sample(items)
    spent = time.perf_counter() - t0
    sample_ms = spent / args.steps * 1e3
    per_token = spent / args.steps * pass_bytes / sample_bytes(items)
    value = 1.0 / per_token
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": sample_ms,
        "ms_per_step_note": "time actually spent per step: one oracle run of the sample",
        "extrapolated_ms_per_token": per_token * 1e3,
        "sample_fraction_of_pass": sample_bytes(items) / pass_bytes,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config,
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                         "sample": sample_note(items, pass_bytes)},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "hbm_gbs": metrics.gbps(pass_bytes, per_token),
    }
    print(json.dumps(line), flush=True)
    return 0


def run_gb300(args, world, rank, local):
    from bit_weight_only_gemv_gb300 import lib
    lib.load()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    model = DENSE_WORKLOADS[args.workload]()
    dp = DecodePass(model, dev, seed=0, merge=not args.separate, gated=args.gated_mlp,
                    l2_next_bytes=int(args.l2_next_mb * (1 << 20)))
    launches = dp.chain_launches() if args.chain else dp.launches()
    stream = torch.cuda.Stream(device=dev)
    # eager warm-up (plans, attributes), then capture the pass as one graph
    with torch.cuda.stream(stream):
        for i, (_, _, f) in enumerate(launches):
            f(i > 0)
    torch.cuda.synchronize()
    g = capture([f for _, _, f in launches], stream)
    step_bytes = dp.step_bytes()
    n_launch = len(launches)

    for _ in range(args.warmup):
        g.replay()
    torch.cuda.synchronize()
    sampler = ClockSampler(local).start()
    # settle under load so the clock samples of the timed region are steady
    t_end = time.time() + 0.5
    while time.time() < t_end:
        g.replay()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    ms = time_replays(g, stream, args.steps)
    torch.cuda.synchronize()
    ms = max_over_ranks(ms, dev)
    clocks = sampler.stop()
    if int(dp.status.item()) != 0:
        raise RuntimeError(f"device status {int(dp.status.item())}")

    tok_s = world * 1000.0 / ms

    # dominant kernel: time its launches of the pass on their own (same stream,
    # same arguments), CUDA events around whole-graph replays
    keys = [kernel_key(k, s, lib) for k, s, _ in launches]
    by_key = {}
    for (kind, shape, f), key in zip(launches, keys):
        b = (metrics.gemv_bytes(*shape) if kind == "gemv" else metrics.gather_bytes(*shape)
             if kind == "gather" else sum(metrics.gemv_bytes(*sh) for sh in shape))
        by_key.setdefault(key, []).append((f, b))
    key_time = {}
    for key, items in by_key.items():
        gk = capture([f for f, _ in items], stream)
        for _ in range(3):
            gk.replay()
        reps = max(3, min(args.steps, 50))
        key_time[key] = (time_replays(gk, stream, reps), len(items), sum(b for _, b in items))
        del gk
    dom = max(key_time, key=lambda k: key_time[k][0])
    dom_ms, dom_n, dom_bytes = key_time[dom]
    peak, peak_kind = load_peaks()
    achieved = metrics.gbps(dom_bytes / dom_n, dom_ms * 1e-3 / dom_n)
    traffic = traffic_from_profile(dom)

    # end to end: inputs from pinned host memory, logits back to the host
    h_ids, h_x = dp.host_inputs()
    h_logits, lo = dp.host_outputs()
    e2e_steps = max(3, min(args.steps, 50))
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(e2e_steps):
            dp.ids.copy_(h_ids, non_blocking=True)
            dp.x_flat.copy_(h_x, non_blocking=True)
            g.replay()
            h_logits.copy_(dp.y_flat[lo:lo + model.vocab], non_blocking=True)
        e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    h2d = h_ids.numel() * 4 + h_x.numel() * 2
    d2h = h_logits.numel() * 2

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline_of(dense_sample_from_device(dp), step_bytes)

    line = {
        "metric": METRIC, "value": tok_s, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": DTYPE,
        "data": "synthetic",
        "config": dense_config(model, args, world, step_bytes),
        "hbm_gbs": metrics.gbps(step_bytes, ms * 1e-3),
        "frac_of_nominal_8tbps": metrics.gbps(step_bytes, ms * 1e-3) / NOMINAL_HBM_GBPS,
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": None if traffic is None else traffic["bytes"],
                     "traffic_note": None if traffic is None else
                     "ncu dram read+write per launch, " + traffic["workload"],
                     "launches_per_step": dom_n, "ms_per_step": dom_ms},
        "kernels": {k: {"launches_per_step": v[1], "ms": v[0],
                        "gbps": metrics.gbps(v[2], v[0] * 1e-3)} for k, v in key_time.items()},
        "cpu_baseline": cpu,
        "e2e": {"value": world * 1000.0 / e2e_ms, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": n_launch * args.steps,
        "clocks": clocks,
    }
    if world == 1 and not args.no_side and not args.chain:
        # after the main measurement (its clocks, e2e and oracle are taken);
        # the decode pass's buffers are freed first
        del g, dp, launches
        torch.cuda.empty_cache()
        line["side_workloads"] = side_workloads(args, world, rank, local)
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def run_moe(args, world, rank, local, emit=True):
    """Routed-expert decode (30 layers, 128 experts, top-8, 32-slot LFU pool per
    layer): per step and layer, remap the step's experts to pool slots (host),
    copy the missed experts into the pool and write the slot ids (device),
    then w4a16_gemv_id for the merged gate/up (x broadcast) and for down (one
    x row per expert), addressing the pool.  An expert's gate/up and down
    weights sit side by side in its slot (and in the full tensor), so one
    remap and one copy of codes and one of steps per miss serve both."""
    from bit_weight_only_gemv_gb300 import lib
    lib.load()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    cfg = synth.moe_2816()
    E, S, H, I, k_top, L = (cfg.experts, cfg.slots, cfg.hidden, cfg.expert_inter, cfg.top_k,
                            cfg.layers)
    steps, warm = args.steps, args.warmup
    total = warm + steps
    shapes = {"gate_up": (2 * I, H), "down": (H, I)}
    # bytes per expert: codes and steps of each projection, and where they sit
    qoff, soff, qcomb, scomb = {}, {}, 0, 0
    for name, (n, k) in shapes.items():
        qoff[name], soff[name] = qcomb, scomb
        qcomb += n * k // 2
        scomb += n * k // 16
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    fill_stream = torch.cuda.Stream(device=dev)   # pool fills beside the dense FFN
    shared = args.shared_ffn
    host_home = args.expert_home == "host"
    vectors = args.expert_vectors
    # the router's real ids of every step, as it would leave them on the device
    eids_dev = torch.zeros((L, k_top), dtype=torch.int32, device=dev)
    eids_host = torch.zeros((total, L, k_top), dtype=torch.int32).pin_memory()
    layers = []
    for li in range(L):
        lay = {"trace": synth.moe_trace(E, k_top, total, cfg.zipf_s, cfg.repeat_p,
                                        seed=synth.seed_of(42, li)),
               "x": {"gate_up": synth.torch_x((1, H), synth.seed_of(43, li), dev),
                     "down": synth.torch_x((k_top, I), synth.seed_of(44, li), dev)},
               "slot_ids": torch.zeros(k_top, dtype=torch.int32, device=dev),
               "ids_full": torch.zeros(k_top, dtype=torch.int32, device=dev),
               "full_q": synth.torch_words((E, qcomb // 4), synth.seed_of(40, li), dev),
               "full_s": synth.torch_steps((E, scomb // 2), synth.seed_of(41, li), dev),
               "pool_q": torch.zeros((S, qcomb // 4), dtype=torch.int32, device=dev),
               "pool_s": torch.zeros((S, scomb // 2), dtype=torch.bfloat16, device=dev),
               "y": {}, "y_full": {}, "calls": [], "calls_full": []}
        eids_host[:, li] = torch.from_numpy(np.asarray(lay["trace"], dtype=np.int32))
        if shared != "none":
            # a dense FFN per layer of one expert's shape, on the layer's input
            lay["shared"] = [(synth.torch_words((n, k // 8), synth.seed_of(47, li, n), dev),
                              synth.torch_steps((n, k // 32), synth.seed_of(48, li, n), dev),
                              lay["x"]["gate_up"] if name == "gate_up" else
                              synth.torch_x((1, k), synth.seed_of(49, li), dev),
                              torch.empty((1, n), dtype=torch.bfloat16, device=dev))
                             for name, (n, k) in shapes.items()]
            lay["fill_done"] = torch.cuda.Event()
            lay["pool_free"] = torch.cuda.Event()
        lay["src_q"], lay["src_s"] = lay["full_q"], lay["full_s"]
        if host_home:   # the pool's source; the HBM copy only serves the bitwise check
            lay["src_q"] = torch.empty(lay["full_q"].shape, dtype=torch.int32, pin_memory=True)
            lay["src_s"] = torch.empty(lay["full_s"].shape, dtype=torch.bfloat16,
                                       pin_memory=True)
            lay["src_q"].copy_(lay["full_q"])
            lay["src_s"].copy_(lay["full_s"])
        if vectors:
            lay["table"] = torch.full((S,), -1, dtype=torch.int32, device=dev)
            lay["scale"] = {name: synth.torch_x((E, n), synth.seed_of(45, li, n), dev)
                            for name, (n, k) in shapes.items()}
            lay["bias"] = {"gate_up": None,
                           "down": synth.torch_x((E, H), synth.seed_of(46, li), dev)}
        for name, (n, k) in shapes.items():
            lay["y"][name] = torch.empty((k_top, n), dtype=torch.bfloat16, device=dev)
            lay["y_full"][name] = torch.empty((k_top, n), dtype=torch.bfloat16, device=dev)
        if args.chain:
            # one launch per layer: gate/up, then down on silu(gate) * up of
            # each expert's own gate/up rows (the fused routed FFN)
            for full, calls in ((False, lay["calls"]), (True, lay["calls_full"])):
                ys = lay["y_full" if full else "y"]
                src_q, src_s = lay["full_q" if full else "pool_q"], lay["full_s" if full else "pool_s"]
                ids = lay["ids_full" if full else "slot_ids"]
                ne = E if full else S
                tasks = [lib.gemv_id_task(src_q[:, qoff["gate_up"] // 4:], src_s[:, soff["gate_up"] // 2:],
                                          ids, lay["x"]["gate_up"], ys["gate_up"], 2 * I, H, ne,
                                          qcomb, scomb),
                         lib.gemv_id_task(src_q[:, qoff["down"] // 4:], src_s[:, soff["down"] // 2:],
                                          ids, ys["gate_up"], ys["down"], H, I, ne, qcomb, scomb,
                                          dep=0, silu_mul=True)]
                ws = torch.zeros(lib.chain_workspace_bytes(tasks), dtype=torch.uint8, device=dev)
                calls.append(lib.bind_gemv_chain(tasks, ws, status))
            layers.append(lay)
            continue
        for name, (n, k) in shapes.items():
            for full, calls in ((False, lay["calls"]), (True, lay["calls_full"])):
                q = lay["full_q" if full else "pool_q"][:, qoff[name] // 4:]
                st = lay["full_s" if full else "pool_s"][:, soff[name] // 2:]
                ids = lay["ids_full" if full else "slot_ids"]
                y = lay["y_full" if full else "y"][name]
                if vectors:
                    calls.append(lib.bind_gemv_id_scaled(
                        q, st, ids, lay["x"][name], n, k, E if full else S, qcomb, scomb,
                        ids if full else eids_dev[li], E, y,
                        slot_expert=None if full else lay["table"], scale=lay["scale"][name],
                        bias=lay["bias"][name], status=status))
                else:
                    calls.append(lib.bind_gemv_id(q, st, ids, lay["x"][name], n, k,
                                                  E if full else S, qcomb, scomb, y, status))
        layers.append(lay)

    device_pool = args.pool == "device"
    if args.chain and vectors:
        raise SystemExit("--chain runs without --expert-vectors")
    if device_pool and shared != "none":
        raise SystemExit("--pool device runs without --shared-ffn")
    # device pool: every step's router ids on the device; a device counter
    # picks the current step's into eids_dev, which the remap reads
    all_ids = eids_host.to(dev) if device_pool else None
    step_idx = torch.zeros(1, dtype=torch.int64, device=dev)

    def new_pools():
        for li, lay in enumerate(layers):
            if device_pool:
                if "dpool" not in lay:
                    lay["dpool"] = lib.DevSlotPool(E, S, device=dev)
                    lay["dstage"] = lay["dpool"].bind_stage(
                        eids_dev[li], lay["pool_q"], lay["src_q"], qcomb, qcomb, lay["pool_s"],
                        lay["src_s"], scomb, scomb, lay["slot_ids"], slot_expert=lay.get("table"),
                        status=status)
                else:
                    lay["dpool"].reset()
                if vectors:
                    lay["table"].fill_(-1)
                continue
            lay["pool"] = lib.SlotPool(E, S)
            lay["stage"] = lay["pool"].bind_stage(k_top, lay["pool_q"], lay["src_q"], qcomb,
                                                  qcomb, lay["pool_s"], lay["src_s"], scomb,
                                                  scomb, lay["slot_ids"],
                                                  slot_expert=lay.get("table"))
            if vectors:
                lay["table"].fill_(-1)
        torch.cuda.synchronize()

    ids_final = not getattr(args, "no_ids_final", False) and not args.chain

    def gemvs(lay, full=False, pdl=False):
        # programmatic dependent launch after the first kernel: the routed
        # kernel reads its ids and activations only after the previous one;
        # the down call's ids are the gate/up call's, written before it ran,
        # so its weight copies may start before that wait (W4_FLAG_IDS_FINAL)
        for i, call in enumerate(lay["calls_full" if full else "calls"]):
            if ids_final:
                call(pdl=pdl or i > 0, stream=stream, ids_final=i > 0)
            else:
                call(pdl=pdl or i > 0, stream=stream)

    def layer_step(lay, t):
        """One layer of one step: pool fill and slot ids, the dense FFN if any,
        the routed GEMVs.  Returns the misses (None for the device pool)."""
        if device_pool:
            lay["dstage"](pdl=True, stream=stream)
            gemvs(lay, pdl=True)
            return None
        if shared == "none":
            misses = lay["stage"](lay["trace"][t], stream=stream)
            gemvs(lay, pdl=True)
            return misses
        if shared == "overlap":
            # the fill may start once the layer's previous routed GEMVs are done
            fill_stream.wait_event(lay["pool_free"])
            misses = lay["stage"](lay["trace"][t], stream=fill_stream)
            lay["fill_done"].record(fill_stream)
        else:
            misses = lay["stage"](lay["trace"][t], stream=stream)
        for qw, st, x, y in lay["shared"]:
            lib.gemv(qw, st, x, y=y, status=status, pdl=True, stream=stream)
        if shared == "overlap":
            stream.wait_event(lay["fill_done"])
        gemvs(lay)
        if shared == "overlap":
            lay["pool_free"].record(stream)
        return misses

    kernel_bytes = L * sum(metrics.gemv_id_bytes(k_top, 1 if name == "gate_up" else k_top, n, k)
                           for name, (n, k) in shapes.items())

    def pool_stats():
        lfu = {"requests": 0, "hits": 0, "misses": 0}
        for lay in layers:
            st = (lay["dpool"] if device_pool else lay["pool"]).stats()
            for key in lfu:
                lfu[key] += st[key]
        return lfu

    # phase A (timed): the routed pass through the pools, eager steps (host
    # pool) or one graph replay per step (device pool)
    new_pools()
    copied = 0
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    if device_pool:
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            step_idx.zero_()
        torch.cuda.synchronize()
        gstep = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gstep, stream=stream):
            eids_dev.copy_(torch.index_select(all_ids, 0, step_idx).view(L, k_top))
            step_idx.add_(1)
            for lay in layers:
                layer_step(lay, 0)
        with torch.cuda.stream(stream):   # the capture ran nothing: start again
            step_idx.zero_()
        new_pools()
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            for t in range(total):
                if t == warm:
                    torch.cuda.synchronize()
                    miss0 = pool_stats()["misses"]
                    e0.record(stream)
                    t_host = time.perf_counter()
                gstep.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        copied = (pool_stats()["misses"] - miss0) * (qcomb + scomb)
    with torch.cuda.stream(stream):
        for t in range(0 if device_pool else total):
            if t == warm:
                torch.cuda.synchronize()
                e0.record(stream)
                t_host = time.perf_counter()
            misses = 0
            if vectors:
                eids_dev.copy_(eids_host[t], non_blocking=True)
            for lay in layers:
                misses += layer_step(lay, t)
            if t >= warm:
                copied += misses * (qcomb + scomb)
        e1.record(stream)
    torch.cuda.synchronize()
    host_s = time.perf_counter() - t_host
    ms = e0.elapsed_time(e1) / steps
    ms = max_over_ranks(ms, dev)
    lfu = pool_stats()

    # kernel only: the last step's 60 routed GEMVs (pool contents as left), as a graph
    fns = [(lambda lay: (lambda pdl: gemvs(lay, pdl=pdl)))(lay) for lay in layers]
    g = capture(fns, stream)
    for _ in range(3):
        g.replay()
    kms = time_replays(g, stream, max(3, min(steps, 50)))
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())}")

    # phase B (check): fresh pools, same traces; every step and layer the pool
    # call must equal the call on the full 128-expert tensor bit for bit
    new_pools()
    bad = torch.zeros((), dtype=torch.int64, device=dev)
    with torch.cuda.stream(stream):
        for t in range(total):
            if vectors or device_pool:
                eids_dev.copy_(eids_host[t], non_blocking=True)
            for lay in layers:
                layer_step(lay, t)
                lay["ids_full"].copy_(torch.from_numpy(lay["trace"][t].astype(np.int32)))
                gemvs(lay, full=True)
                for name in shapes:
                    bad += (lay["y"][name].view(torch.int16) !=
                            lay["y_full"][name].view(torch.int16)).sum()
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())}")

    peak, peak_kind = load_peaks()
    gbps = metrics.gbps(kernel_bytes, kms * 1e-3)
    line = {
        "metric": METRIC, "value": world * 1000.0 / ms, "unit": UNIT, "n_gpus": world,
        "steps": steps, "warmup": warm, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": DTYPE,
        "data": "synthetic",
        "config": moe_config(cfg, args, world),
        "host_seconds_per_step": host_s / steps,
        "kernel": {"ms_per_step": kms, "tok_s": 1000.0 / kms, "bytes_per_step": kernel_bytes,
                   "gbps": gbps, "frac": gbps / peak, "peak": peak, "peak_kind": peak_kind,
                   "note": ("the 30 w4a16_gemv_chain launches (routed gate/up, then down on "
                            "silu(gate) * up) of one step replayed as a graph, PDL-chained"
                            if args.chain else "the 60 gemv_id launches of one step replayed "
                            "as a graph, PDL-chained")},
        "pool": dict(lfu, hit_rate=lfu["hits"] / max(1, lfu["requests"]),
                     copy_bytes_per_step=copied / steps),
        "bitwise_pool_vs_full": {"steps": total, "layers": L, "mismatched_values": int(bad.item())},
        # per layer: pool fill / slot ids, 2 gemv_id (+ 2 dense GEMVs)
        "gpu_launches": steps * L * ((4 if device_pool else 3 if shared == "none" else 5) -
                                     (1 if args.chain else 0)),
    }
    if not emit:
        return line
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def shape_us(M, N, K, dev, copies=None, steps=20, warmup=3):
    """µs per launch of one (M, N, K) GEMV: `copies` weight copies (default:
    enough to exceed 600 MB, so every launch reads HBM) replayed in turn as
    one PDL-chained graph; copies=1 keeps the weights in L2."""
    from bit_weight_only_gemv_gb300 import lib
    per = metrics.gemv_bytes(M, N, K)
    n = copies or max(2, -(-600_000_000 // per))
    qws = [synth.torch_words((N, K // 8), synth.seed_of(7, i), dev) for i in range(n)]
    sts = [synth.torch_steps((N, K // 32), synth.seed_of(8, i), dev) for i in range(n)]
    x = synth.torch_x((M, K), synth.seed_of(9), dev)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    need = lib.workspace_bytes(M, N, K)
    ws = torch.zeros(max(need, 16), dtype=torch.uint8, device=dev) if need else None
    fns = [(lambda q, s_: (lambda pdl: lib.gemv(q, s_, x, y=y, workspace=ws, pdl=pdl)))(q, s_)
           for q, s_ in zip(qws, sts)]
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        for i, f in enumerate(fns):
            f(i > 0)
    torch.cuda.synchronize()
    g = capture(fns * max(1, 16 // n), stream)
    for _ in range(warmup):
        g.replay()
    ms = time_replays(g, stream, steps) / (n * max(1, 16 // n))
    return ms * 1e3, per


def side_workloads(args, world, rank, local):
    """Two smaller workloads measured after the main one, in the same run:
    the 2048 x 2048 batch-1 GEMV (HBM-cold over rotating copies, and
    L2-hot), and the routed decode (30 layers, 128 experts, top-8, 32-slot
    pools; 128 steps, every step and layer checked bitwise against the call
    on the full expert tensor)."""
    dev = torch.device("cuda", local)
    out = {}
    us_cold, per = shape_us(1, 2048, 2048, dev)
    us_hot, _ = shape_us(1, 2048, 2048, dev, copies=1)
    peak, peak_kind = load_peaks()
    out["gemv_2048x2048_batch1"] = {
        "us_hbm_cold": us_cold, "gbps_hbm_cold": metrics.gbps(per, us_cold * 1e-6),
        "frac_hbm_cold": metrics.gbps(per, us_cold * 1e-6) / peak, "us_l2_hot": us_hot,
        "gbps_l2_hot": metrics.gbps(per, us_hot * 1e-6), "bytes": per, "peak": peak,
        "peak_kind": peak_kind,
        "note": "rotating weight copies over 600 MB (HBM-cold) or one copy (L2-hot), "
                "PDL-chained graph, CUDA events"}
    margs = argparse.Namespace(**vars(args))
    margs.workload, margs.steps, margs.warmup = "moe-30L-h2816", 128, 3
    margs.pool, margs.expert_home, margs.expert_vectors = "host", "device", False
    margs.shared_ffn, margs.chain = "none", False
    m = run_moe(margs, world, rank, local, emit=False)
    out["routed_decode_moe_30L_h2816"] = {
        "tok_s": m["value"], "ms_per_step": m["ms_per_step"], "steps": m["steps"],
        "kernel_gbps": m["kernel"]["gbps"], "kernel_frac": m["kernel"]["frac"],
        "lfu_hit_rate": m["pool"]["hit_rate"],
        "bitwise_pool_vs_full": m["bitwise_pool_vs_full"],
        "note": "eager steps (host LFU remap, pool copies, slot ids, 2 w4a16_gemv_id per "
                "layer); kernel GB/s from the step's 60 routed launches replayed as a graph"}
    return out


def run_shape(args):
    """One GEMV shape, timed alone: rotating weight copies (over 4x the L2
    together, so every launch reads HBM), graph replay, CUDA events."""
    from bit_weight_only_gemv_gb300 import lib
    lib.load()
    M, N, K = (int(v) for v in args.shape.split(","))
    dev = torch.device("cuda", 0)
    per = metrics.gemv_bytes(M, N, K)
    copies = max(2, -(-600_000_000 // per))
    qws = [synth.torch_words((N, K // 8), synth.seed_of(7, i), dev) for i in range(copies)]
    sts = [synth.torch_steps((N, K // 32), synth.seed_of(8, i), dev) for i in range(copies)]
    x = synth.torch_x((M, K), synth.seed_of(9), dev)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    if args.path == "chain":
        # each launch a one-task w4a16_gemv_chain (batch 1), own workspace
        if M != 1:
            raise SystemExit("--path chain times batch-1 shapes")
        fns = []
        for q, s_ in zip(qws, sts):
            tasks = [lib.gemv_task(q, s_, x.view(-1), y.view(-1))]
            wsc = torch.zeros(lib.chain_workspace_bytes(tasks), dtype=torch.uint8, device=dev)
            fns.append((lambda c: (lambda pdl: c(pdl=pdl)))(lib.bind_gemv_chain(tasks, wsc)))
    else:
        path = None if args.path == "auto" else args.path
        need = lib.workspace_bytes(M, N, K, path)
        ws = torch.zeros(max(need, 16), dtype=torch.uint8, device=dev) if need else None
        # --l2-next-mb: each launch brings the next copy's leading rows into L2
        pf_rows = min(N, int(args.l2_next_mb * (1 << 20)) // (K // 2 + K // 16))
        nxt = [lib.l2_ranges([(qws[(i + 1) % copies], pf_rows * (K // 2)),
                              (sts[(i + 1) % copies], pf_rows * (K // 16))])
               if pf_rows > 0 else None for i in range(copies)]
        fns = [(lambda q, s_, l2: (lambda pdl: lib.gemv(q, s_, x, y=y, workspace=ws, pdl=pdl,
                                                        path=path, l2_next=l2)))(q, s_, l2)
               for q, s_, l2 in zip(qws, sts, nxt)]
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        for i, f in enumerate(fns):
            f(i > 0)
    torch.cuda.synchronize()
    g = capture(fns, stream, pdl=not args.no_pdl)
    for _ in range(args.warmup):
        g.replay()
    ms = time_replays(g, stream, args.steps) / copies
    print(json.dumps({"mode": "shape", "M": M, "N": N, "K": K, "pdl": not args.no_pdl,
                      "path": args.path, "l2_next_mb": args.l2_next_mb,
                      "us_per_launch": ms * 1e3, "gbps": metrics.gbps(per, ms * 1e-3),
                      "bytes_per_launch": per, "copies": copies, "plan": lib.plan(M, N, K)}),
          flush=True)
    return 0


def run_shape_id(args):
    """One routed call (w4a16_gemv_id), timed alone: n_ids distinct experts of
    an N x K expert tensor, one activation row (broadcast) or one per id,
    rotating expert tensors larger than L2, graph replay, CUDA events."""
    from bit_weight_only_gemv_gb300 import lib
    lib.load()
    parts = [int(v) for v in args.shape_id.split(",")]
    N, K, n_ids = parts[:3]
    x_rows = parts[3] if len(parts) > 3 else 1
    dev = torch.device("cuda", 0)
    per = metrics.gemv_id_bytes(n_ids, x_rows, N, K)
    copies = max(2, -(-600_000_000 // per))
    E = n_ids
    qws = [synth.torch_words((E, N * K // 8), synth.seed_of(17, i), dev) for i in range(copies)]
    sts = [synth.torch_steps((E, N * K // 32), synth.seed_of(18, i), dev) for i in range(copies)]
    ids = torch.randperm(E, generator=torch.Generator().manual_seed(0)).to(torch.int32).to(dev)
    x = synth.torch_x((x_rows, K), synth.seed_of(19), dev)
    y = torch.empty((n_ids, N), dtype=torch.bfloat16, device=dev)
    fns = [lib.bind_gemv_id(q, s_, ids, x, N, K, E, N * K // 2, N * K // 16, y, None)
           for q, s_ in zip(qws, sts)]
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        for i, f in enumerate(fns):
            f(pdl=i > 0, stream=stream)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i, f in enumerate(fns):
            f(pdl=i > 0, stream=stream)
    for _ in range(args.warmup):
        g.replay()
    ms = time_replays(g, stream, args.steps) / copies
    print(json.dumps({"mode": "shape_id", "N": N, "K": K, "n_ids": n_ids, "x_rows": x_rows,
                      "us_per_launch": ms * 1e3, "gbps": metrics.gbps(per, ms * 1e-3),
                      "bytes_per_launch": per, "copies": copies}), flush=True)
    return 0


def build_parser() -> argparse.ArgumentParser:
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default 200; 128 for the routed-expert workload)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("gb300", "reference"), default="gb300")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-ids-final", action="store_true",
                    help="routed-expert workload: the down call waits for the gate/up call "
                         "before reading its ids (without W4_FLAG_IDS_FINAL)")
    ap.add_argument("--no-side", action="store_true",
                    help="decode passes: skip the two side workloads measured after the main "
                         "one (the 2048 x 2048 batch-1 GEMV HBM-cold and L2-hot; the routed "
                         "decode's 128 steps with the bitwise pool-vs-full check)")
    ap.add_argument("--shape", default=None,
                    help="M,N,K: time one GEMV shape alone instead of the decode pass")
    ap.add_argument("--shape-id", default=None,
                    help="N,K,n_ids[,x_rows]: time one routed call (w4a16_gemv_id) over n_ids "
                         "experts of N x K alone")
    ap.add_argument("--no-pdl", action="store_true", help="with --shape: plain launches")
    ap.add_argument("--path", choices=("auto", "cuda", "tensor", "chain"), default="auto",
                    help="with --shape: the library's choice, CUDA cores, tensor cores, or "
                         "(batch 1) a one-task w4a16_gemv_chain launch")
    ap.add_argument("--separate", action="store_true",
                    help="one GEMV per projection instead of merged q/k/v and gate/up")
    ap.add_argument("--expert-home", choices=("device", "host"), default="device",
                    help="routed-expert workload: full expert tensors in HBM, or in page-locked "
                         "host (Grace) memory that the pool fills read over NVLink-C2C")
    ap.add_argument("--expert-vectors", action="store_true",
                    help="routed-expert workload: per-expert output scales (and down biases) "
                         "by real expert id, slot table checked (w4a16_gemv_id_scaled)")
    ap.add_argument("--chain", action="store_true",
                    help="decode passes: every GEMV of the pass in one w4a16_gemv_chain launch "
                         "(each task waiting for the one before) instead of one launch each")
    ap.add_argument("--l2-next-mb", type=float, default=0.0,
                    help="decode passes: each GEMV brings up to this many MiB of the next GEMV's "
                         "weights (its leading rows) into L2 once its own tiles are requested "
                         "(w4a16_gemv_prefetch_l2); 0 turns it off")
    ap.add_argument("--gated-mlp", action="store_true",
                    help="decode passes: each down projection reads its layer's merged gate/up "
                         "output through silu(gate) * up (W4_FLAG_SILU_MUL) instead of its own "
                         "activation row")
    ap.add_argument("--pool", choices=("host", "device"), default="host",
                    help="routed-expert workload: LFU remap on the host per layer (eager steps), "
                         "or on the device (w4_dev_pool_*), each step one CUDA graph replay")
    ap.add_argument("--shared-ffn", choices=("none", "serial", "overlap"), default="none",
                    help="routed-expert workload: add a dense FFN per layer of one expert's "
                         "shape (merged gate/up, down; w4a16_gemv) and run the pool fill "
                         "before it on the same stream (serial) or beside it on a second "
                         "stream, joined before the routed GEMVs (overlap)")
    ap.add_argument("--workload", default="dense-60L-h5376",
                    choices=sorted(DENSE_WORKLOADS) + ["moe-30L-h2816"],
                    help="decode pass to time (default: the 60-layer hidden-5376 decoder "
                         "with its 262144 x 5376 lm_head)")
    return ap


def main():
    ap = build_parser()
    args = ap.parse_args()
    if args.steps is None:
        args.steps = 128 if args.workload.startswith("moe") else 200
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world, rank, local = dist_env()
    if world > 1:
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        torch.distributed.init_process_group(backend)
    try:
        if args.impl == "reference":
            return run_reference(args, world, rank)
        if args.shape:
            return run_shape(args)
        if args.shape_id:
            return run_shape_id(args)
        if args.workload.startswith("moe"):
            return run_moe(args, world, rank, local)
        return run_gb300(args, world, rank, local)
    finally:
        if world > 1 and torch.distributed.is_initialized():
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
