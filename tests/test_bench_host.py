"""Host-side pieces of bench.py that need no GPU."""

import re

import bench


def test_code_tokens_ignore_comments_and_blank_space_only():
    a = "int f(int x) { // add one\n  return x + 1; /* done */ }\n#define A 1\n"
    b = "/* header */\nint f(int x)   {\n\n return x + 1;  }\n#define A 1 // note\n"
    assert bench.code_tokens(a) == bench.code_tokens(b)
    # a change of code, of a literal, or of where a preprocessor line ends counts
    assert bench.code_tokens(a) != bench.code_tokens(a.replace("x + 1", "x + 2"))
    s = 'const char* p = "// kept /* kept */ \\" kept";'
    assert bench.code_tokens(s) == s
    assert bench.code_tokens("char c = '\"'; int y;") == "char c = '\"'; int y;"
    assert bench.code_tokens("#define A 1\n#define B 2") != \
        bench.code_tokens("#define A 1 #define B 2")


def test_kernel_source_digest_is_a_sha256():
    d = bench.kernel_source_digest()
    assert len(d) == 64 and int(d, 16) >= 0


def _profile_commands():
    """Every `python bench.py ...` command quoted in profiles/ (line
    continuations joined), with its argument list."""
    import glob
    import os
    import re
    import shlex
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    for path in sorted(glob.glob(os.path.join(root, "profiles", "*.md"))):
        text = re.sub(r"\\\s*\n\s*", " ", open(path).read())
        for m in re.finditer(r"python bench\.py([^`\n]*)", text):
            tail = re.split(r"\s(?:>|&&|\|)", m.group(1))[0]
            yield os.path.basename(path), shlex.split(tail)


def test_profile_commands_parse_with_the_current_flags():
    seen = 0
    for name, argv in _profile_commands():
        # placeholders such as M,N,K or {cuda,tensor} stand for a sweep
        if any(re.search(r"[A-Z],|\{", a) for a in argv):
            continue
        try:
            bench.build_parser().parse_args(argv)
        except SystemExit:
            raise AssertionError(f"{name}: bench.py {' '.join(argv)} no longer parses")
        seen += 1
    assert seen >= 8


def test_reference_arm_reports_time_it_spent(capsys):
    """The oracle arm runs the selected workload's sample; steps x ms_per_step
    is the time it spent, the extrapolation to a whole pass is apart."""
    import json
    import time
    for workload in ("dense-60L-h5376", "dense-35L-h2048", "moe-30L-h2816"):
        args = bench.build_parser().parse_args(
            ["--impl", "reference", "--steps", "3", "--warmup", "3", "--workload", workload])
        t0 = time.perf_counter()
        assert bench.run_reference(args, 1, 0) == 0
        wall = time.perf_counter() - t0
        line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
        assert line["impl"] == "reference" and line["steps"] == 3
        assert line["steps"] * line["ms_per_step"] <= wall * 1e3
        assert workload.split("-")[0] in line["config"]["workload"]
        frac = line["sample_fraction_of_pass"]
        assert 0 < frac < 1
        # value is the extrapolated whole-pass rate
        assert abs(line["value"] * line["extrapolated_ms_per_token"] - 1e3) < 1e-6 * 1e3
        assert abs(line["extrapolated_ms_per_token"] * frac - line["ms_per_step"]) < \
            1e-6 * line["ms_per_step"]


def test_dense_sample_covers_each_launched_matrix():
    from bit_weight_only_gemv_gb300 import synth
    model = synth.dense_5376()
    groups = bench.merged_groups(model)
    assert [g[0] for g in groups] == ["q+k+v", "o", "gate+up", "down"]
    assert [g[1:] for g in groups] == [(9472, 5376), (5376, 5376), (43008, 5376), (5376, 21504)]
    items = bench.dense_sample_from_recipe(model)
    gemvs = [it for it in items if it[0] == "gemv"]
    assert len(gemvs) == len(groups) + 1                      # + the lm_head rows
    assert [it[1].shape[1] * 8 for it in gemvs] == [5376, 5376, 5376, 21504, 5376]
    assert all(it[1].shape[0] == bench.SAMPLE_ROWS for it in gemvs)
    assert sum(1 for it in items if it[0] == "gather") == 1    # no per-layer table


def test_cpu_baseline_times_the_sample_on_all_cores_and_on_one():
    import numpy as np
    from bit_weight_only_gemv_gb300 import synth
    rng = np.random.default_rng(0)
    items = [("gemv", synth.np_words(rng, (32, 256)), synth.np_steps(rng, (32, 64)),
              synth.np_x(rng, (1, 2048))),
             ("gather", synth.np_words(rng, (1, 256)), synth.np_steps(rng, (1, 64)), None)]
    out = bench.cpu_baseline_of(items, 10 ** 9, seconds=0.2, one_core_seconds=0.2)
    assert out["kind"] == "oracle" and out["value"] > 0 and out["cores"] >= 1
    assert out["cpu_count"] >= out["affinity_cores"] >= 1
    one = out["one_core"]                        # the child process held to one core
    assert one["value"] > 0 and one["repetitions"] >= 1
    # both rates scale the same sample to the same pass
    assert abs(one["extrapolated_ms_per_token"] * one["value"] - 1000.0) < 1e-6
    assert abs(out["extrapolated_ms_per_token"] * out["value"] - 1000.0) < 1e-6
