"""Planted mistakes in the CPU oracle must fail its pins (no GPU needed).

Each case below edits one line of an oracle function's source the way a
plausible slip would (a nibble order reversed, the zero code off by one, the
step of the wrong group, a dropped term, a transposed or reversed operand,
truncation for round-to-nearest-even, a bound made looser, an eviction rule
turned round), rebuilds the function from the edited source, puts it in
place of the original and runs the pins of ``test_oracle_pins.py``: at least
one pin must fail.  The edits live here, on the CPU, in the oracle only; the
oracle's own files are not changed.
"""

import inspect
import textwrap

import pytest

import oracle
import test_oracle_pins as pins
from oracle import lfu, ref

# (id, module, function or class, source fragment, its replacement)
MUTANTS = [
    ("nibble_order_high_first", ref, "unpack_codes",
     "shifts = (4 * np.arange(NIBBLES_PER_WORD, dtype=np.uint32))",
     "shifts = (4 * np.arange(NIBBLES_PER_WORD, dtype=np.uint32))[::-1]"),
    ("pack_order_high_first", ref, "pack_codes",
     "shifts = (4 * np.arange(NIBBLES_PER_WORD, dtype=np.uint32))",
     "shifts = (4 * np.arange(NIBBLES_PER_WORD, dtype=np.uint32))[::-1]"),
    ("zero_code_off_by_one", ref, "dequant", "(codes - CODE_ZERO)", "(codes - (CODE_ZERO - 1))"),
    ("step_of_group_k_mod_groups", ref, "dequant", "np.repeat(steps, GROUP, axis=-1)",
     "np.tile(steps, GROUP)"),
    ("dropped_last_group", ref, "gemv_ref", "return x @ w.T",
     "return x[:, :-GROUP] @ w[:, :-GROUP].T"),
    ("activation_reversed_along_k", ref, "gemv_ref",
     "x = bf16_bits_to_f64(np.atleast_2d(x_bits))",
     "x = bf16_bits_to_f64(np.atleast_2d(x_bits))[:, ::-1]"),
    ("abs_of_sum_for_sum_of_abs", ref, "gemv_abs_ref", "return x @ w.T",
     "return np.abs(bf16_bits_to_f64(np.atleast_2d(x_bits)) @ dequant(qw, st).T)"),
    ("values_rounded_to_bf16", ref, "gemv_values_ref",
     "x = np.atleast_2d(np.asarray(x, dtype=np.float64))",
     "x = bf16_bits_to_f64(bf16_rne(np.atleast_2d(np.asarray(x, dtype=np.float64))))"),
    ("bf16_truncates", ref, "bf16_rne", "r = np.rint(q) * ulp", "r = np.trunc(q) * ulp"),
    ("bf16_ties_away_from_zero", ref, "bf16_rne", "r = np.rint(q) * ulp",
     "r = np.floor(q + 0.5) * ulp"),
    ("bf16_no_subnormal_grid", ref, "bf16_rne", "e = np.maximum(e2 - 1, _BF16_MIN_EXP)",
     "e = e2 - 1"),
    ("bf16_overflow_kept_finite", ref, "bf16_rne",
     "out = np.where(finite & (out > _BF16_MAX), np.inf, out)",
     "out = np.where(finite & (out > _BF16_MAX), _BF16_MAX, out)"),
    ("ulp_twice_too_large", ref, "ulp_bf16", "return np.ldexp(1.0, e - 7)",
     "return np.ldexp(1.0, e - 6)"),
    ("bound_ten_times_looser", ref, "bound_violations",
     "ok = err <= rel * np.asarray(abs_ref) + ulp_bf16(y_ref)",
     "ok = err <= 10 * rel * np.asarray(abs_ref) + ulp_bf16(y_ref)"),
    ("bound_without_ulp_term", ref, "bound_violations",
     "ok = err <= rel * np.asarray(abs_ref) + ulp_bf16(y_ref)",
     "ok = err <= rel * np.asarray(abs_ref)"),
    ("bound_accepts_non_finite", ref, "bound_violations",
     "ok = np.where(ref_finite, ok & np.isfinite(y), same_class)",
     "ok = np.where(ref_finite, ok | ~np.isfinite(y), True)"),
    ("bound_any_non_finite_class", ref, "bound_violations",
     "ok = np.where(ref_finite, ok & np.isfinite(y), same_class)",
     "ok = np.where(ref_finite, ok & np.isfinite(y), ~np.isfinite(y))"),
    ("bound_infinity_sign_ignored", ref, "bound_violations",
     "(np.isinf(y_ref) & (y == y_ref))",
     "(np.isinf(y_ref) & np.isinf(y))"),
    ("silu_sign", ref, "silu_mul_ref", "g / (1.0 + np.exp(-g)) * u", "g / (1.0 + np.exp(g)) * u"),
    ("gate_and_up_swapped", ref, "silu_mul_ref", "g, u = x[:, :k], x[:, k:]",
     "u, g = x[:, :k], x[:, k:]"),
    ("routed_rows_always_broadcast", ref, "gemv_id_ref",
     "xi = x[0] if x.shape[0] == 1 else x[i]", "xi = x[0]"),
    ("routed_expert_by_position", ref, "gemv_id_ref",
     "rows.append(gemv_ref(qw_experts[e], st_experts[e], xi)[0])",
     "rows.append(gemv_ref(qw_experts[i], st_experts[i], xi)[0])"),
    ("expert_scale_dropped", ref, "gemv_id_scaled_ref", "y = s * y", "y = y"),
    ("expert_bias_by_position", ref, "gemv_id_scaled_ref",
     "y = y + bf16_bits_to_f64(np.asarray(bias_bits))[ids]",
     "y = y + bf16_bits_to_f64(np.asarray(bias_bits))[:ids.size]"),
    ("gather_steps_of_other_rows", ref, "gather_ref",
     "return bf16_rne(dequant(qw[ids], st[ids]))",
     "return bf16_rne(dequant(qw[ids], st[ids[::-1]]))"),
    ("quantize_step_sign", ref, "quantize_ref", "step_f32 = m / np.float32(-8.0)",
     "step_f32 = m / np.float32(8.0)"),
    ("quantize_floor", ref, "quantize_ref", "codes = np.clip(np.rint(q) + CODE_ZERO, 0, 15)",
     "codes = np.clip(np.floor(q) + CODE_ZERO, 0, 15)"),
    ("quantize_last_maximum", ref, "quantize_ref",
     "first_max = np.argmax(np.abs(g), axis=-1)",
     "first_max = g.shape[-1] - 1 - np.argmax(np.abs(g)[..., ::-1], axis=-1)"),
    ("quantize_step_from_fp32_truncation", ref, "quantize_ref",
     "st = bf16_rne(step_f32.astype(np.float64))",
     "st = (step_f32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)"),
    ("lfu_evicts_most_used", lfu, "LFUSlotPoolRef",
     "s = min(cands, key=lambda j: (self.count[self.expert_in_slot[j]],",
     "s = min(cands, key=lambda j: (-self.count[self.expert_in_slot[j]],"),
    ("lfu_ties_to_most_recent", lfu, "LFUSlotPoolRef", "self.last_use[j], j))",
     "-self.last_use[j], j))"),
    ("lfu_highest_free_slot", lfu, "LFUSlotPoolRef", "s = free[0]", "s = free[-1]"),
    ("lfu_may_evict_a_needed_expert", lfu, "LFUSlotPoolRef",
     "if self.expert_in_slot[j] not in needed]", "if True]"),
    ("lfu_hits_not_counted", lfu, "LFUSlotPoolRef",
     "for e in ids:\n            self.count[e] += 1",
     "for e in ids:\n            self.count[e] += 0 if e in self.slot_of_expert else 1"),
]


def _mutant(module, name, old, new):
    src = textwrap.dedent(inspect.getsource(getattr(module, name)))
    assert src.count(old) == 1, f"fragment not found once in {name}: {old!r}"
    ns = dict(vars(module))
    exec(compile(src.replace(old, new), f"<mutant of {name}>", "exec"), ns)
    return ns[name]


def _pin_cases():
    """Every pin of test_oracle_pins.py with its parameters, except the
    plain-C identity check (it does not run the Python oracle)."""
    for name, fn in vars(pins).items():
        if not (name.startswith("test_") and callable(fn)):
            continue
        if "tmp_path" in inspect.signature(fn).parameters:
            continue
        marks = [m for m in getattr(fn, "pytestmark", []) if m.name == "parametrize"]
        if not marks:
            yield name, fn, {}
            continue
        assert len(marks) == 1, name
        argnames, values = marks[0].args[0], marks[0].args[1]
        names = [a.strip() for a in argnames.split(",")]
        for v in values:
            v = tuple(v) if isinstance(v, (tuple, list)) else (v,)
            yield name, fn, dict(zip(names, v))


def test_pins_pass_on_the_oracle_as_it_stands():
    # the runner itself: with nothing planted every pin passes
    cases = list(_pin_cases())
    assert len(cases) > 30
    for _, fn, kw in cases:
        fn(**kw)


@pytest.mark.parametrize("mid,module,name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_fails_a_pin(monkeypatch, mid, module, name, old, new):
    bad = _mutant(module, name, old, new)
    monkeypatch.setattr(module, name, bad)
    if hasattr(oracle, name):
        monkeypatch.setattr(oracle, name, bad)
    for pin, fn, kw in _pin_cases():
        try:
            fn(**kw)
        except AssertionError:
            return          # a value check of this pin caught it (a crash would not count)
    pytest.fail(f"no pin fails with the planted mistake {mid}")
