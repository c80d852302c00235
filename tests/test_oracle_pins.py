"""Pins of the CPU oracle against facts fixed outside it (no GPU needed).

Each test checks the oracle against the pages' stated identities and worked
numbers, closed forms, exact rational brute force on tiny inputs, or a library
routine in a special case, chosen so that a dropped term, a wrong sign, a wrong
nibble or group index, or a transposed operand fails at least one of them.
"""

import os
import subprocess
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from oracle import ref
from bit_weight_only_gemv_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


# ---------------------------------------------------------------- helpers
def frac_bf16(bits: int) -> Fraction:
    """Exact value of a bf16 bit pattern, decoded field by field."""
    sign = -1 if bits >> 15 else 1
    e = (bits >> 7) & 0xFF
    m = bits & 0x7F
    assert e != 0xFF
    if e == 0:
        return sign * Fraction(m, 2 ** 133)
    return sign * Fraction(128 + m, 128) * Fraction(2) ** (e - 127)


def hex_codes(word: int):
    """Codes of a packed word read as hex digits, least significant first."""
    return [int(d, 16) for d in format(int(word), "08x")[::-1]]


def exact_gemv(qw, st, x):
    """Rational y[m][n] and sum|w x| from raw bits, independent of the oracle."""
    n_rows, n_words = qw.shape
    k = n_words * 8
    out = []
    out_abs = []
    for xm in np.atleast_2d(x):
        row, row_abs = [], []
        for n in range(n_rows):
            codes = [c for j in range(n_words) for c in hex_codes(qw[n, j])]
            acc = Fraction(0)
            acc_abs = Fraction(0)
            for kk in range(k):
                w = (codes[kk] - 8) * frac_bf16(int(st[n, kk // 32]))
                t = w * frac_bf16(int(xm[kk]))
                acc += t
                acc_abs += abs(t)
            row.append(acc)
            row_abs.append(acc_abs)
        out.append(row)
        out_abs.append(row_abs)
    return out, out_abs


def f32_to_bf16_bits_torch(v: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.asarray(v, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


# ---------------------------------------------------------------- dequant
def test_magic_identity_exhaustive_in_c(tmp_path):
    src = os.path.join(ROOT, "oracle", "magic_check.c")
    exe = os.path.join(ROOT, "oracle", "magic_check")
    if not os.path.exists(exe) or os.path.getmtime(exe) < os.path.getmtime(src):
        exe = str(tmp_path / "magic_check")
        subprocess.run(["gcc", "-O2", "-std=c11", "-o", exe, src], check=True)
    res = subprocess.run([exe], capture_output=True, text=True)
    assert res.returncode == 0, res.stdout
    got = [ln.rsplit(" ", 1)[0].split() for ln in res.stdout.strip().splitlines()]
    want = [ln.split() for ln in open(os.path.join(GOLDEN, "magic_dequant.txt"))
            if ln.strip() and not ln.startswith("#")]
    assert got == want


def test_packed_word_fixture():
    for line in open(os.path.join(GOLDEN, "packed_words.txt")):
        if not line.strip() or line.startswith("#"):
            continue
        word_s, codes_s, vals_s = line.split()
        word = int(word_s, 16)
        codes = [int(c) for c in codes_s.split(",")]
        vals = [int(v) for v in vals_s.split(",")]
        qw = np.array([[word, word, word, word]], dtype=np.uint32)
        step_bits = 0x3E80            # bf16 0.25
        st = np.array([[step_bits]], dtype=np.uint16)
        assert list(ref.unpack_codes(qw)[0, :8]) == codes
        w = ref.dequant(qw, st)[0, :8]
        assert list(w) == [0.25 * v for v in vals]
        assert list(ref.pack_codes(ref.unpack_codes(qw))[0]) == [word] * 4


def test_group_index_of_steps():
    # every word 0x00000000 (code 0 -> -8), steps 1, 2, 3 for groups 0, 1, 2
    qw = np.zeros((1, 12), dtype=np.uint32)
    st = f32_to_bf16_bits_torch(np.array([[1.0, 2.0, 3.0]]))
    w = ref.dequant(qw, st)[0]
    assert np.all(w[:32] == -8.0) and np.all(w[32:64] == -16.0) and np.all(w[64:] == -24.0)


def test_code_eight_is_exact_zero():
    rng = np.random.default_rng(1)
    qw = np.full((5, 16), 0x88888888, dtype=np.uint32)
    st = synth.np_steps(rng, (5, 4))
    x = synth.np_x(rng, (3, 128))
    assert np.all(ref.dequant(qw, st) == 0.0)
    y = ref.gemv_ref(qw, st, x)
    assert np.all(y == 0.0)
    assert np.all(ref.gather_ref(qw, st, np.arange(5)) & 0x7FFF == 0)


# ---------------------------------------------------------------- gemv
@pytest.mark.parametrize("n,k,m,seed", [(1, 32, 1, 0), (3, 32, 2, 1), (4, 64, 1, 2),
                                        (2, 64, 2, 3), (4, 32, 1, 4)])
def test_gemv_exact_bruteforce(n, k, m, seed):
    rng = np.random.default_rng(seed)
    qw = synth.np_words(rng, (n, k // 8))
    qw[0, 0] = 0x76543210          # make sure every code occurs
    qw[-1, -1] = 0xFEDCBA98
    st = synth.np_steps(rng, (n, k // 32), scale=1.0)
    x = synth.np_x(rng, (m, k))
    y = ref.gemv_ref(qw, st, x)
    ya = ref.gemv_abs_ref(qw, st, x)
    exact, exact_abs = exact_gemv(qw, st, x)
    for mi in range(m):
        for ni in range(n):
            e = exact[mi][ni]
            a = exact_abs[mi][ni]
            assert abs(Fraction(y[mi, ni]) - e) <= Fraction(k) * Fraction(2) ** -52 * a
            assert abs(Fraction(ya[mi, ni]) - a) <= Fraction(k) * Fraction(2) ** -52 * a
    assert y.shape == (m, n)


def test_one_hot_activation_selects_column():
    rng = np.random.default_rng(5)
    n, k = 6, 96
    qw = synth.np_words(rng, (n, k // 8))
    st = synth.np_steps(rng, (n, k // 32))
    w = ref.dequant(qw, st)
    one = 0x3F80                     # bf16 1.0
    for kk in (0, 7, 8, 31, 32, 95):
        x = np.zeros((1, k), dtype=np.uint16)
        x[0, kk] = one
        y = ref.gemv_ref(qw, st, x)[0]
        assert np.array_equal(y, w[:, kk])
        # and element-by-element from the raw bits
        for ni in range(n):
            c = hex_codes(qw[ni, kk // 8])[kk % 8]
            assert Fraction(y[ni]) == (c - 8) * frac_bf16(int(st[ni, kk // 32]))


@pytest.mark.parametrize("c", [0, 3, 8, 9, 15])
def test_all_equal_codes_closed_form(c):
    # all codes c: y[n] = (c - 8) * sum_g st[n, g] * sum_{k in g} x[k]
    rng = np.random.default_rng(10 + c)
    n, k = 5, 160
    word = int("".join([format(c, "x")] * 8), 16)
    qw = np.full((n, k // 8), word, dtype=np.uint32)
    st = synth.np_steps(rng, (n, k // 32))
    x = synth.np_x(rng, (1, k))
    y = ref.gemv_ref(qw, st, x)[0]
    for ni in range(n):
        want = Fraction(0)
        for g in range(k // 32):
            sx = sum((frac_bf16(int(v)) for v in x[0, 32 * g:32 * g + 32]), Fraction(0))
            want += frac_bf16(int(st[ni, g])) * sx
        want *= (c - 8)
        assert abs(Fraction(y[ni]) - want) <= Fraction(k) * Fraction(2) ** -52 * abs(want) + \
            Fraction(2) ** -200


def test_gemv_linearity_and_batch_rows():
    rng = np.random.default_rng(7)
    n, k = 9, 256
    qw = synth.np_words(rng, (n, k // 8))
    st = synth.np_steps(rng, (n, k // 32))
    x = synth.np_x(rng, (4, k))
    y = ref.gemv_ref(qw, st, x)
    for mi in range(4):
        assert np.array_equal(y[mi], ref.gemv_ref(qw, st, x[mi])[0])
    # transposed use of the operands would change the shape or the values
    w = ref.dequant(qw, st)
    xf = ref.bf16_bits_to_f64(x)
    assert np.allclose(y, np.einsum("mk,nk->mn", xf, w), rtol=1e-13, atol=0)


def test_gemv_id_addresses_experts_and_broadcasts():
    rng = np.random.default_rng(8)
    e, n, k = 5, 3, 64
    qw = synth.np_words(rng, (e, n, k // 8))
    st = synth.np_steps(rng, (e, n, k // 32), scale=1.0)
    ids = np.array([4, 0, 4, 2], dtype=np.int32)
    xb = synth.np_x(rng, (1, k))
    xr = synth.np_x(rng, (4, k))
    yb = ref.gemv_id_ref(qw, st, ids, xb)
    yr = ref.gemv_id_ref(qw, st, ids, xr)
    for i, ex in enumerate(ids):
        eb, _ = exact_gemv(qw[ex], st[ex], xb)
        er, _ = exact_gemv(qw[ex], st[ex], xr[i:i + 1])
        for ni in range(n):
            assert abs(Fraction(yb[i, ni]) - eb[0][ni]) <= Fraction(2) ** -40 * (abs(eb[0][ni]) + 1)
            assert abs(Fraction(yr[i, ni]) - er[0][ni]) <= Fraction(2) ** -40 * (abs(er[0][ni]) + 1)
    assert np.array_equal(yb[0], yb[2])          # repeated id, same activation
    with pytest.raises(ValueError):
        ref.gemv_id_ref(qw, st, ids, synth.np_x(rng, (2, k)))


def _bf16_bits(rng, shape, lo=-2.0, hi=2.0):
    return f32_to_bf16_bits_torch(rng.uniform(lo, hi, size=shape))


def test_gemv_id_scaled_exact_bruteforce_by_real_ids():
    # y[i][n] = scale[e][n] * (W_e x_i)[n] + bias[e][n], e the REAL expert id,
    # checked against rationals built from the raw bits
    rng = np.random.default_rng(21)
    e, n, k = 4, 3, 32
    qw = synth.np_words(rng, (e, n, k // 8))
    st = synth.np_steps(rng, (e, n, k // 32), scale=1.0)
    sc = _bf16_bits(rng, (e, n))
    bi = _bf16_bits(rng, (e, n))
    eids = np.array([3, 1, 3], dtype=np.int32)
    x = synth.np_x(rng, (3, k))
    y, a = ref.gemv_id_scaled_ref(qw, st, eids, x, sc, bi)
    for i, ex in enumerate(eids):
        dot, dot_abs = exact_gemv(qw[ex], st[ex], x[i:i + 1])
        for ni in range(n):
            s_ = frac_bf16(int(sc[ex, ni]))
            want = s_ * dot[0][ni] + frac_bf16(int(bi[ex, ni]))
            assert abs(Fraction(y[i, ni]) - want) <= Fraction(2) ** -45 * (abs(want) + 1)
            assert abs(Fraction(a[i, ni]) - abs(s_) * dot_abs[0][ni]) <= \
                Fraction(2) ** -45 * (abs(s_) * dot_abs[0][ni] + 1)


def test_gemv_id_scaled_special_cases():
    rng = np.random.default_rng(22)
    e, n, k = 6, 5, 64
    qw = synth.np_words(rng, (e, n, k // 8))
    st = synth.np_steps(rng, (e, n, k // 32), scale=1.0)
    eids = np.array([5, 0, 2, 5], dtype=np.int32)
    x = synth.np_x(rng, (1, k))
    plain = ref.gemv_id_ref(qw, st, eids, x)
    # no vectors: the plain routed product
    y, a = ref.gemv_id_scaled_ref(qw, st, eids, x)
    assert np.array_equal(y, plain)
    # zero activations: exactly the bias row of the real expert
    bi = _bf16_bits(rng, (e, n))
    y0, a0 = ref.gemv_id_scaled_ref(qw, st, eids, np.zeros((1, k), np.uint16), None, bi)
    for i, ex in enumerate(eids):
        for ni in range(n):
            assert Fraction(y0[i, ni]) == frac_bf16(int(bi[ex, ni]))
    assert not np.any(a0)
    # power-of-two scales: exact scaling of the plain product, row by row
    pw = rng.integers(-3, 4, size=(e, n))
    sc = f32_to_bf16_bits_torch(np.ldexp(1.0, pw).astype(np.float32))
    ys, _ = ref.gemv_id_scaled_ref(qw, st, eids, x, sc, None)
    assert np.array_equal(ys, plain * np.ldexp(1.0, pw[eids]))


def test_gemv_id_scaled_slot_ids_fed_to_the_vectors_change_the_result():
    # The page's hazard: a consumer of per-expert vectors given slot ids
    # instead of real ids.  With distinct per-expert biases the planted
    # mistake (vectors indexed by slot id) cannot pass for the real result.
    rng = np.random.default_rng(23)
    e, n, k = 8, 4, 32
    qw = synth.np_words(rng, (e, n, k // 8))
    st = synth.np_steps(rng, (e, n, k // 32), scale=1.0)
    bi = _bf16_bits(rng, (e, n), 1.0, 2.0)
    pool = oracle.LFUSlotPoolRef(e, 3)
    x = synth.np_x(rng, (1, k))
    for req in ([6, 2], [2, 7], [5, 6]):
        slots, _ = pool.step(req)
        good, _ = ref.gemv_id_scaled_ref(qw, st, np.array(req), x, None, bi)
        # weights by real id, vectors by slot id
        bad = ref.gemv_id_ref(qw, st, np.array(req), x) + \
            ref.bf16_bits_to_f64(bi)[np.array(slots)]
        assert not np.array_equal(good, bad)


def test_gemv_values_ref_reduces_to_the_bf16_product():
    rng = np.random.default_rng(31)
    qw = synth.np_words(rng, (5, 12))
    st = synth.np_steps(rng, (5, 3), scale=1.0)
    xb = synth.np_x(rng, (2, 96))
    y, a = ref.gemv_values_ref(qw, st, ref.bf16_bits_to_f64(xb))
    assert np.array_equal(y, ref.gemv_ref(qw, st, xb))
    assert np.array_equal(a, ref.gemv_abs_ref(qw, st, xb))


def test_gemv_values_ref_exact_on_real_valued_activations():
    # activations that are not bf16 values (the gated activation's fp64
    # products): rational brute force, each fp64 input taken exactly
    rng = np.random.default_rng(33)
    n, k = 3, 64
    qw = synth.np_words(rng, (n, k // 8))
    st = synth.np_steps(rng, (n, k // 32), scale=1.0)
    x = rng.standard_normal((2, k)) / 3.0
    y, a = ref.gemv_values_ref(qw, st, x)
    for m in range(2):
        for ni in range(n):
            codes = [c for j in range(k // 8) for c in hex_codes(qw[ni, j])]
            terms = [(codes[kk] - 8) * frac_bf16(int(st[ni, kk // 32])) * Fraction(float(x[m, kk]))
                     for kk in range(k)]
            exact, exact_abs = sum(terms, Fraction(0)), sum((abs(t) for t in terms), Fraction(0))
            tol = float(exact_abs) * k * 2.0 ** -52
            assert abs(Fraction(float(y[m, ni])) - exact) <= Fraction(tol)
            assert abs(Fraction(float(a[m, ni])) - exact_abs) <= Fraction(tol)


def test_silu_mul_special_values_and_library_form():
    from scipy.special import expit
    g = np.array([0.0, 1.0, -1.0, 20.0, -20.0, 3.5, -100.0, 88.0], dtype=np.float32)
    u = np.array([2.0, 1.0, 1.0, 0.5, 1.0, 0.0, 1.0, -1.0], dtype=np.float32)
    x_bits = f32_to_bf16_bits_torch(np.concatenate([g, u]))[None, :]
    gb = ref.bf16_bits_to_f64(x_bits[0, :8])
    ub = ref.bf16_bits_to_f64(x_bits[0, 8:])
    h = ref.silu_mul_ref(x_bits)[0]
    assert h[0] == 0.0 and h[5] == 0.0                  # silu(0) = 0; up = 0
    assert h[1] == pytest.approx(1.0 / (1.0 + np.exp(-1.0)), rel=1e-15)
    assert h[2] == pytest.approx(-1.0 / (1.0 + np.exp(1.0)), rel=1e-15)
    assert h[3] == pytest.approx(0.5 * 20.0, rel=3e-9)  # silu(g) -> g for large g
    assert abs(h[6]) < 1e-40                             # -> 0 for very negative g
    # the textbook form g * sigmoid(g) * u from the library's logistic function
    assert np.allclose(h, gb * expit(gb) * ub, rtol=1e-14, atol=0)
    rng = np.random.default_rng(32)
    xb = synth.np_x(rng, (3, 64))
    x = ref.bf16_bits_to_f64(xb)
    assert np.allclose(ref.silu_mul_ref(xb), x[:, :32] * expit(x[:, :32]) * x[:, 32:],
                       rtol=1e-14, atol=0)


# ---------------------------------------------------------------- bf16
def test_bf16_rne_hand_values():
    cases = [
        (1.0, 0x3F80),
        (1.0 + 2 ** -8, 0x3F80),                  # tie -> even (mantissa 0)
        (1.0 + 3 * 2 ** -8, 0x3F82),              # tie -> even (mantissa 2)
        (1.0 + 2 ** -8 + 2 ** -40, 0x3F81),       # just above the tie: up
        (-(1.0 + 2 ** -8 + 2 ** -40), 0xBF81),
        (2.0 ** -133, 0x0001),                    # smallest subnormal
        (2.0 ** -134, 0x0000),                    # tie with 0 -> even (0)
        (3 * 2.0 ** -134, 0x0002),                # tie 1.5 -> 2
        (float.fromhex("0x1.fep127"), 0x7F7F),    # largest finite
        (float.fromhex("0x1.ffp127"), 0x7F80),    # tie above it -> inf
        (float.fromhex("0x1.fefp127"), 0x7F7F),
        (float("inf"), 0x7F80),
        (-0.0, 0x8000),
        (0.0, 0x0000),
    ]
    for v, want in cases:
        assert int(ref.bf16_rne(np.array([v]))[0]) == want, (v, hex(want))
    assert int(ref.bf16_rne(np.array([float("nan")]))[0]) & 0x7FFF == 0x7FC0


def test_bf16_rne_matches_torch_on_fp32_values():
    rng = np.random.default_rng(11)
    v = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-30, 30, 20000),
                        rng.standard_normal(2000) * 1e-39]).astype(np.float32)
    assert np.array_equal(ref.bf16_rne(v.astype(np.float64)), f32_to_bf16_bits_torch(v))


def test_ulp_bf16():
    assert ref.ulp_bf16(np.array([1.0]))[0] == 2.0 ** -7
    assert ref.ulp_bf16(np.array([1.99]))[0] == 2.0 ** -7
    assert ref.ulp_bf16(np.array([-2.0]))[0] == 2.0 ** -6
    assert ref.ulp_bf16(np.array([0.0]))[0] == 2.0 ** -133
    assert ref.ulp_bf16(np.array([2.0 ** -130]))[0] == 2.0 ** -133


def test_bound_check_logic():
    y_ref = np.array([1.0, 1.0, 0.0, -0.0, 100.0, np.inf])
    abs_ref = np.array([1.0, 1.0, 0.0, 0.0, 100.0, np.inf])
    ok_bits = ref.bf16_rne(np.array([1.0 + 2 ** -7, 1.0 + 2 * 2 ** -7, 0.0, 0.0, 100.0, np.inf]))
    bad = ref.bound_violations(ok_bits, y_ref, abs_ref)
    assert list(bad) == [False, True, False, False, False, False]
    # +0 and -0 are equal
    assert not ref.bound_violations(np.array([0x8000], np.uint16), np.array([0.0]), np.array([0.0]))[0]
    # a finite result where the reference is infinite fails
    assert ref.bound_violations(np.array([0x3F80], np.uint16), np.array([np.inf]), np.array([np.inf]))[0]


def test_bound_non_finite_classes():
    # a non-finite reference takes a result of the same class: bf16 bit
    # patterns +inf 0x7F80, -inf 0xFF80, a quiet NaN 0x7FC0 (and one with the
    # sign bit set), against references +inf, -inf, NaN
    bits = np.array([0x7F80, 0xFF80, 0x7FC0, 0xFFC0], np.uint16)
    refs = np.array([np.inf, -np.inf, np.nan])
    got = np.array([[ref.bound_violations(np.array([b], np.uint16), np.array([r]),
                                          np.array([np.inf]))[0] for r in refs] for b in bits])
    expect = np.array([[False, True, True],     # +inf result
                       [True, False, True],     # -inf result
                       [True, True, False],     # NaN result
                       [True, True, False]])    # negative NaN result
    assert np.array_equal(got, expect)
    # and a non-finite result where the reference is finite fails
    for b in bits:
        assert ref.bound_violations(np.array([b], np.uint16), np.array([1.0]), np.array([1.0]))[0]


# ---------------------------------------------------------------- gather
def test_gather_matches_exact_products_rounded_by_torch():
    rng = np.random.default_rng(12)
    v, k = 40, 288
    qw = synth.np_words(rng, (v, k // 8))
    st = synth.np_steps(rng, (v, k // 32), scale=0.37)
    ids = np.array([39, 0, 17, 17, 5], dtype=np.int32)
    got = ref.gather_ref(qw, st, ids)
    # (c - 8) * step is exact in fp32, so torch's fp32 -> bf16 (nearest even)
    # is the one rounding
    for t, i in enumerate(ids):
        codes = np.array([c for j in range(k // 8) for c in hex_codes(qw[i, j])], dtype=np.float32)
        steps = np.repeat(np.array([float(frac_bf16(int(s))) for s in st[i]], np.float32), 32)
        prod = (codes - 8) * steps
        assert np.array_equal(got[t], f32_to_bf16_bits_to_u16(prod))


def f32_to_bf16_bits_to_u16(a):
    return f32_to_bf16_bits_torch(a)


def test_gather_one_hot_rows_and_tied_column():
    # a row whose codes are all c with step s gathers to bf16((c-8) s) everywhere,
    # and the GEMV of the table against e_k reproduces column k of the gather
    rng = np.random.default_rng(13)
    v, k = 16, 64
    qw = np.array([[int(format(c, "x") * 8, 16)] * (k // 8) for c in range(16)], dtype=np.uint32)
    st = f32_to_bf16_bits_torch(np.full((v, k // 32), 0.75, np.float32))
    g = ref.gather_ref(qw, st, np.arange(16))
    for c in range(16):
        assert np.all(ref.bf16_bits_to_f64(g[c]) == (c - 8) * 0.75)
    qw2 = synth.np_words(rng, (v, k // 8))
    st2 = synth.np_steps(rng, (v, k // 32))
    g2 = ref.gather_ref(qw2, st2, np.arange(v))
    for kk in (0, 33, 63):
        x = np.zeros((1, k), dtype=np.uint16)
        x[0, kk] = 0x3F80
        col = ref.bf16_rne(ref.gemv_ref(qw2, st2, x)[0])
        assert np.array_equal(col, g2[:, kk])


# ---------------------------------------------------------------- quantiser
def test_quantize_codes_are_nearest_grid_points():
    rng = np.random.default_rng(14)
    n, k = 7, 256
    w = (rng.standard_normal((n, k)) * 10.0 ** rng.integers(-3, 3, (n, 1))).astype(np.float32)
    w[0, :32] = 0.0                               # all-zero group -> step 0, codes 8
    w[1, 32:64] = 0.5                             # constant group
    qw, st = ref.quantize_ref(w)
    codes = ref.unpack_codes(qw).astype(np.int64)
    steps = ref.bf16_bits_to_f64(st)
    assert np.all(codes[0, :32] == 8) and steps[0, 0] == 0.0
    grid = np.arange(16) - 8
    for ni in range(n):
        for kk in range(k):
            s = steps[ni, kk // 32]
            if s == 0:
                continue
            errs = np.abs(w[ni, kk] - grid * s)
            chosen = errs[codes[ni, kk]]
            # nearest grid point, up to the fp32 division's last-bit error
            assert chosen <= errs.min() + abs(s) * 2.0 ** -20
    # the element of largest magnitude gets code 0 (value -8 * step)
    g = w.reshape(n, -1, 32)
    first = np.argmax(np.abs(g), axis=-1)
    for ni in range(n):
        for gi in range(k // 32):
            if steps[ni, gi] != 0:
                assert codes[ni, gi * 32 + first[ni, gi]] == 0


def test_quantize_step_is_bf16_of_signed_absmax_over_minus_eight():
    w = np.zeros((1, 32), np.float32)
    w[0, 3] = -3.0
    w[0, 9] = 3.0                      # same magnitude later in K: not chosen
    qw, st = ref.quantize_ref(w)
    assert ref.bf16_bits_to_f64(st)[0, 0] == 0.375          # -3 / -8
    assert ref.unpack_codes(qw)[0, 3] == 0 and ref.unpack_codes(qw)[0, 9] == 15   # 8 -> clamp 15
    w2 = np.zeros((1, 32), np.float32)
    w2[0, 0] = 1.01                     # 1.01 / -8 is not a bf16: rounded once
    _, st2 = ref.quantize_ref(w2)
    assert int(st2[0, 0]) == int(f32_to_bf16_bits_torch(np.array([np.float32(1.01) / np.float32(-8)]))[0])
    # steps that round up: 1.99 / -8 (bits past the 8th above one half) and
    # 8.09375 / -8 = -(1 + 3 * 2^-8), a tie resolved to the even neighbour
    # -(1 + 4 * 2^-8); truncation would give -(1 + 2^-7) and -(1 + 2 * 2^-8)
    for v, want in ((1.99, None), (8.09375, -1.015625)):
        w3 = np.zeros((1, 32), np.float32)
        w3[0, 7] = v
        _, st3 = ref.quantize_ref(w3)
        lib_bits = int(f32_to_bf16_bits_torch(np.array([np.float32(v) / np.float32(-8)]))[0])
        assert int(st3[0, 0]) == lib_bits
        if want is not None:
            assert ref.bf16_bits_to_f64(st3)[0, 0] == want


def test_quantize_round_trip_on_grid():
    rng = np.random.default_rng(15)
    n, k = 6, 128
    codes = synth.np_codes(rng, (n, k))
    codes.reshape(n, -1, 32)[:, :, 5] = 0            # code 0 in every group
    st = synth.np_steps(rng, (n, k // 32), scale=0.3)
    w = ref.dequant(ref.pack_codes(codes), st).astype(np.float32)
    qw2, st2 = ref.quantize_ref(w)
    assert np.array_equal(st2, st)
    assert np.array_equal(ref.unpack_codes(qw2), codes)


def test_pack_unpack_round_trip():
    rng = np.random.default_rng(16)
    codes = synth.np_codes(rng, (5, 64))
    assert np.array_equal(ref.unpack_codes(ref.pack_codes(codes)), codes)
    words = synth.np_words(rng, (5, 8))
    assert np.array_equal(ref.pack_codes(ref.unpack_codes(words)), words)
    with pytest.raises(ValueError):
        ref.pack_codes(np.full((1, 8), 16, np.uint8))


# ---------------------------------------------------------------- LFU pool
def _read_traces():
    traces = []
    cur = None
    for line in open(os.path.join(GOLDEN, "lfu_traces.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        if line.startswith("trace"):
            parts = line.split()
            kv = dict(p.split("=") for p in parts[2:])
            cur = (parts[1], int(kv["experts"]), int(kv["slots"]), [])
            traces.append(cur)
            continue
        req, slots, miss = [p.strip() for p in line.split("|")]
        misses = [] if miss == "-" else [tuple(int(v) for v in m.split(":")) for m in miss.split(",")]
        cur[3].append(([int(v) for v in req.split(",")], [int(v) for v in slots.split(",")], misses))
    return traces


def test_lfu_hand_traces():
    traces = _read_traces()
    assert len(traces) >= 5
    for name, e, s, steps in traces:
        pool = oracle.LFUSlotPoolRef(e, s)
        for req, want_slots, want_miss in steps:
            got_slots, got_miss = pool.step(req)
            assert (got_slots, got_miss) == (want_slots, want_miss), name


def test_lfu_pool_contents_follow_the_misses():
    # simulate the pool memory: after each step the slot named for every
    # requested expert holds that expert
    rng = np.random.default_rng(17)
    tr = synth.moe_trace(128, 8, 300, 1.1, 0.7, seed=3)
    pool = oracle.LFUSlotPoolRef(128, 32)
    content = [-1] * 32
    hits = 0
    for req in tr:
        slots, misses = pool.step(req)
        for ex, sl in misses:
            content[sl] = ex
        assert all(0 <= sl < 32 for sl in slots)
        assert [content[sl] for sl in slots] == list(req)
        hits += len(req) - len(misses)
    assert hits > 0
    with pytest.raises(ValueError):
        oracle.LFUSlotPoolRef(4, 2).step([0, 1, 2])
    del rng


def test_moe_trace_recipe():
    tr = synth.moe_trace(128, 8, 200, 1.1, 0.7, seed=9)
    assert tr.shape == (200, 8)
    assert all(len(set(r)) == 8 for r in tr)
    assert tr.min() >= 0 and tr.max() < 128
    kept = np.mean([len(set(tr[t]) & set(tr[t - 1])) for t in range(1, 200)])
    assert 5.0 < kept < 7.5          # about 0.7 * 8 kept plus Zipf re-draws


# ---------------------------------------------------------------- metric form
def test_bandwidth_formula_reproduces_the_pages_example():
    from bit_weight_only_gemv_gb300 import metrics
    vals = {}
    for line in open(os.path.join(GOLDEN, "bandwidth_example.txt")):
        if line.startswith("#") or not line.strip():
            continue
        parts = line.split()
        if parts[0] == "bytes_per_token_MiB":
            vals["mib"] = float(parts[1])
        elif parts[0] == "kernel":
            vals[parts[1]] = (float(parts[3]), float(parts[5]))
        elif parts[0] == "plain_read_GBps":
            vals["plain"] = float(parts[1])
        elif parts[0] == "kernel_fraction_percent":
            vals["pct"] = float(parts[1])
    nbytes = vals["mib"] * metrics.MIB
    for ver in ("v5", "v4"):
        ms, printed = vals[ver]
        digits = len(str(ms).split(".")[1])
        half = 0.5 * 10.0 ** -digits
        lo = metrics.gbps(nbytes, (ms + half) * 1e-3)
        hi = metrics.gbps(nbytes, (ms - half) * 1e-3)
        assert lo - 0.05 <= printed <= hi + 0.05, (ver, lo, hi, printed)
    v5 = metrics.gbps(nbytes, vals["v5"][0] * 1e-3)
    assert round(100 * v5 / vals["plain"]) == vals["pct"]


def test_gemv_byte_accounting():
    from bit_weight_only_gemv_gb300 import metrics
    # one 2048 x 2048 GEMV at batch 1: 2 MiB codes + 256 KiB steps + x + y
    assert metrics.gemv_bytes(1, 2048, 2048) == 2 * 1024 * 1024 + 256 * 1024 + 4096 + 4096
    assert metrics.gemv_bytes(1, 2048, 2048) == 2367488
    # per-layer table row: 35 x 256 values
    assert metrics.gather_bytes(1, 35 * 256) == 4480 + 560 + 17920 + 4
    assert metrics.gemv_id_bytes(8, 1, 704, 2816) == 8 * (991232 + 123904) + 5632 + 11264
