"""Plain fp64 CPU oracle for the W4A16 group-32 GEMV path.  TEST INFRASTRUCTURE.

Only the test-suite, the smoke check and the benchmark's CPU-baseline legs use
this module.  It shares no code with the CUDA library and imports nothing from
it.  Every function is the textbook definition written out with NumPy; a NumPy
matmul or reduction is used as a single step where the definition is a sum.

Sources (cited by page title and section):

* [G4] "Gemma 4 on a 4 GB GPU in Plain PyTorch: From Out of Memory to Faster
  Than llama.cpp" (dev.to).
    - "Step 1 — Load Google's QAT Weights Without Unpacking Them": the format
      is compressed-tensors W4A16, 4-bit weight codes in groups of 32 with a
      16-bit step per group and 16-bit activations.
    - "Step 2 — Keep the Vocabulary Tables in 4-Bit": the token table (shared
      with the output layer) and the per-layer table stay as 4-bit codes, a
      16-bit step for each group; a single copy on the device serves both the
      lookup by token id and the output GEMV.
    - "Step 3 — Multiply Straight From the Packed Weights": each decoded token
      needs the product of an activation vector with each weight matrix,
      taken from the packed words as stored; a code is turned into a float by
      placing it in the low mantissa bits of 2^23 and subtracting 2^23 + 8, so
      the dequantised value is (code - 8) * step.
    - "Why Doesn't 16-bit Fit?": the per-layer table holds, for every one of
      262,144 vocabulary ids, a row of 35 x 256 values.
* [MoE] "Running a 26B MoE on an 8 GB Jetson by streaming experts from SSD"
  (anyesh.me), section "Streaming without touching a single GPU kernel": the
  routed-expert matmul reads expert ``id`` at ``base + id * stride``; a slot
  pool plus a slot-id tensor must give bitwise the same logits as addressing
  the full expert tensor.

Readings where the pages are silent:

* nibble order inside a 32-bit word: low nibble first, so element ``k`` of a
  row lives in word ``k // 8`` at bits ``4*(k % 8) .. 4*(k % 8)+3``;
* 16-bit step and activation type: bfloat16 (the pages say "16-bit");
* output: bf16, round-to-nearest-even of the exact (fp64) sum;
* quantiser: signed absmax, step = bf16(m / -8) with ``m`` the group element of
  largest magnitude (first in K order on ties), code = clamp(rint(w / step) + 8,
  0, 15) with IEEE fp32 division and round-half-even (see ``quantize_ref``).

Array conventions (all little-endian, row-major):

* ``qw``  uint32 [N, K/8]   packed codes;
* ``st``  uint16 [N, K/32]  bf16 bit patterns of the per-group steps;
* ``x``   uint16 [M, K]     bf16 bit patterns of the activations;
* results are fp64 unless stated otherwise; bf16 results are uint16 bit
  patterns.
"""

from __future__ import annotations

import numpy as np

GROUP = 32            # codes per quantisation group along K ([G4] Step 1)
NIBBLES_PER_WORD = 8  # 4-bit codes per uint32 word
CODE_ZERO = 8         # the code that dequantises to exactly 0 ([G4] Step 3)

_BF16_MAX = float.fromhex("0x1.fep127")   # largest finite bfloat16
_BF16_MIN_EXP = -126                      # exponent of the smallest normal


# --------------------------------------------------------------------------
# bfloat16 helpers
# --------------------------------------------------------------------------
def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Value of bf16 bit patterns: a bf16 is the top half of an IEEE fp32."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def bf16_rne(v) -> np.ndarray:
    """Round fp64 values to bfloat16 (nearest, ties to even); return the bits.

    Done directly from the fp64 value, not through fp32, so that no double
    rounding occurs.  Magnitudes that round above the largest finite bf16 give
    infinity; NaN gives the quiet NaN 0x7FC0 with the input's sign.
    """
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    out = np.empty(v.shape, dtype=np.float64)
    finite = np.isfinite(a)
    nz = finite & (a > 0)
    # exponent of the leading bit, floored at the smallest normal exponent so
    # that subnormals are rounded on the fixed 2^-133 grid
    _, e2 = np.frexp(np.where(nz, a, 1.0))
    e = np.maximum(e2 - 1, _BF16_MIN_EXP)
    ulp = np.ldexp(1.0, e - 7)
    q = np.where(nz, a / ulp, 0.0)         # exact: division by a power of two
    r = np.rint(q) * ulp                   # np.rint rounds half to even
    out[...] = np.where(nz, r, 0.0)
    out = np.where(finite & (out > _BF16_MAX), np.inf, out)
    out = np.where(~finite, a, out)        # inf stays inf, nan stays nan
    out = np.copysign(out, v)
    f32 = out.astype(np.float32)           # exact: every bf16 is an fp32
    bits = (f32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    nan = np.isnan(v)
    if np.any(nan):
        sign = (np.signbit(v).astype(np.uint16) << np.uint16(15))
        bits = np.where(nan, np.uint16(0x7FC0) | sign, bits).astype(np.uint16)
    return bits


def ulp_bf16(v) -> np.ndarray:
    """Spacing of bf16 values at ``v``: 2^(floor(log2|v|) - 7) for normal v.

    Below the smallest normal (and at 0) it is the subnormal spacing 2^-133.
    """
    a = np.abs(np.asarray(v, dtype=np.float64))
    _, e2 = np.frexp(np.where(a > 0, a, 1.0))
    e = np.where(a > 0, np.maximum(e2 - 1, _BF16_MIN_EXP), _BF16_MIN_EXP)
    return np.ldexp(1.0, e - 7)


# --------------------------------------------------------------------------
# packing and dequantisation  ([G4] Step 1 and Step 3)
# --------------------------------------------------------------------------
def unpack_codes(qw: np.ndarray) -> np.ndarray:
    """uint32 [N, K/8] -> uint8 [N, K]; element k is nibble k % 8 of word k // 8."""
    qw = np.asarray(qw, dtype=np.uint32)
    shifts = (4 * np.arange(NIBBLES_PER_WORD, dtype=np.uint32))
    codes = (qw[..., :, None] >> shifts) & np.uint32(0xF)
    return codes.reshape(*qw.shape[:-1], qw.shape[-1] * NIBBLES_PER_WORD).astype(np.uint8)


def pack_codes(codes: np.ndarray) -> np.ndarray:
    """uint8 [N, K] (values 0..15) -> uint32 [N, K/8], low nibble first."""
    c = np.asarray(codes)
    if c.shape[-1] % NIBBLES_PER_WORD:
        raise ValueError("K must be a multiple of 8")
    if np.any(c > 15):
        raise ValueError("codes must be in 0..15")
    c = c.astype(np.uint32).reshape(*c.shape[:-1], -1, NIBBLES_PER_WORD)
    shifts = (4 * np.arange(NIBBLES_PER_WORD, dtype=np.uint32))
    return np.bitwise_or.reduce(c << shifts, axis=-1).astype(np.uint32)


def dequant(qw: np.ndarray, st: np.ndarray) -> np.ndarray:
    """W[n, k] = (code[n, k] - 8) * step[n, k // 32] in fp64 (exact)."""
    codes = unpack_codes(qw).astype(np.float64)
    steps = bf16_bits_to_f64(st)
    if codes.shape[-1] != steps.shape[-1] * GROUP:
        raise ValueError("st must have K/32 columns")
    return (codes - CODE_ZERO) * np.repeat(steps, GROUP, axis=-1)


# --------------------------------------------------------------------------
# GEMV, routed-expert GEMV, row gather
# --------------------------------------------------------------------------
def gemv_ref(qw: np.ndarray, st: np.ndarray, x_bits: np.ndarray) -> np.ndarray:
    """y[m, n] = sum_k W[n, k] * x[m, k] in fp64 ([G4] Step 3).

    ``x_bits`` is uint16 [M, K] (or [K]).  Each product is exact in fp64
    (at most 11 + 8 significant bits); the sum is one NumPy matmul.
    """
    w = dequant(qw, st)
    x = bf16_bits_to_f64(np.atleast_2d(x_bits))
    return x @ w.T


def gemv_abs_ref(qw: np.ndarray, st: np.ndarray, x_bits: np.ndarray) -> np.ndarray:
    """sum_k |W[n, k] * x[m, k]|: the scale of the acceptance bound."""
    w = np.abs(dequant(qw, st))
    x = np.abs(bf16_bits_to_f64(np.atleast_2d(x_bits)))
    return x @ w.T


def gemv_values_ref(qw: np.ndarray, st: np.ndarray, x: np.ndarray):
    """(W x, sum_k |w x|) for real-valued activations x [M, K] (fp64): the
    product gemv_ref takes, for activations that are not bf16 values."""
    w = dequant(qw, st)
    x = np.atleast_2d(np.asarray(x, dtype=np.float64))
    return x @ w.T, np.abs(x) @ np.abs(w).T


def silu_mul_ref(x_bits: np.ndarray) -> np.ndarray:
    """Gated activation of rows [gate K | up K] (bf16 bit patterns): h =
    silu(gate) * up = gate / (1 + e^-gate) * up, in fp64.

    The down projection of a gated MLP reads this product of the merged
    gate/up GEMV's two halves ([G4] tip "Merge the Small Projections" merges
    gate and up into one GEMV; the pages name no activation, SiLU is the
    reading taken here).
    """
    x = bf16_bits_to_f64(np.atleast_2d(x_bits))
    k = x.shape[1] // 2
    g, u = x[:, :k], x[:, k:]
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g)) * u


def gemv_id_ref(qw_experts: np.ndarray, st_experts: np.ndarray,
                ids: np.ndarray, x_bits: np.ndarray) -> np.ndarray:
    """Routed-expert GEMV ([MoE] "Streaming without touching a single GPU kernel").

    ``qw_experts`` uint32 [E, N, K/8], ``st_experts`` uint16 [E, N, K/32],
    ``ids`` int [n_ids], ``x_bits`` uint16 [x_rows, K] with x_rows either 1
    (one activation row shared by every id) or n_ids (row i goes with ids[i]).
    Output row i is expert ids[i] applied to its activation row; ids may repeat.
    """
    ids = np.asarray(ids).reshape(-1)
    x = np.atleast_2d(x_bits)
    if x.shape[0] not in (1, ids.size):
        raise ValueError("x must have 1 or n_ids rows")
    rows = []
    for i, e in enumerate(ids):
        xi = x[0] if x.shape[0] == 1 else x[i]
        rows.append(gemv_ref(qw_experts[e], st_experts[e], xi)[0])
    return np.stack(rows) if rows else np.zeros((0, qw_experts.shape[1]))


def gemv_id_scaled_ref(qw_experts: np.ndarray, st_experts: np.ndarray, expert_ids: np.ndarray,
                       x_bits: np.ndarray, scale_bits=None, bias_bits=None):
    """Routed-expert GEMV with per-expert output vectors, by REAL expert id.

    [MoE] "Streaming without touching a single GPU kernel": besides the
    expert matmul, per-expert scale vectors and biases consume the router's
    choice; those tables hold one row for every expert in memory at all
    times, so their row is chosen by the true expert number, and only the
    matmul is redirected to a slot pool.  So, with e = expert_ids[i]:

        y_ref[i, n] = scale[e, n] * (W_e x_i)[n] + bias[e, n]

    from the FULL expert tensor (a pool is an addressing detail that must not
    change the bits).  ``scale_bits`` / ``bias_bits`` are bf16 bit patterns
    [E, N] or None (1 and 0).  Returns (y_ref, abs_ref) in fp64, where
    abs_ref = |scale| * sum_k |w x| is the scale of the acceptance bound.
    """
    ids = np.asarray(expert_ids).reshape(-1)
    y = gemv_id_ref(qw_experts, st_experts, ids, x_bits)
    x = np.atleast_2d(x_bits)
    a = np.stack([gemv_abs_ref(qw_experts[e], st_experts[e],
                               x[0] if x.shape[0] == 1 else x[i])[0]
                  for i, e in enumerate(ids)])
    if scale_bits is not None:
        s = bf16_bits_to_f64(np.asarray(scale_bits))[ids]
        y = s * y
        a = np.abs(s) * a
    if bias_bits is not None:
        y = y + bf16_bits_to_f64(np.asarray(bias_bits))[ids]
    return y, a


def gather_ref(qw: np.ndarray, st: np.ndarray, ids: np.ndarray) -> np.ndarray:
    """out[t, k] = bf16((code[ids[t], k] - 8) * step[ids[t], k // 32]).

    [G4] Step 2: the 4-bit vocabulary tables are looked up by token id; the
    product is exact, so the only rounding is the one to bf16.
    """
    ids = np.asarray(ids).reshape(-1)
    return bf16_rne(dequant(qw[ids], st[ids]))


# --------------------------------------------------------------------------
# quantiser (pack/quantise helper)
# --------------------------------------------------------------------------
def quantize_ref(w: np.ndarray):
    """fp32 W [N, K] -> (qw uint32 [N, K/8], st uint16 [N, K/32]).

    [G4] Step 2 only says each group's step is recovered from the 4-bit grid.
    Plain signed-absmax reading, group by group:
      m     = the element of largest |w| (the first one in K order on ties);
      step  = bf16_rne(m / -8)     (fp32 division, then one rounding to bf16);
      code  = 8 everywhere if step == 0, else
              clamp(rint(w / step) + 8, 0, 15), fp32 IEEE division, rint half
              to even.
    With this step the element m gets code 0, i.e. the value -8 * step = m.
    Inputs must be finite.
    """
    w = np.asarray(w, dtype=np.float32)
    n, k = w.shape
    if k % GROUP:
        raise ValueError("K must be a multiple of 32")
    g = w.reshape(n, k // GROUP, GROUP)
    first_max = np.argmax(np.abs(g), axis=-1)          # first maximum
    m = np.take_along_axis(g, first_max[..., None], axis=-1)[..., 0]
    step_f32 = m / np.float32(-8.0)
    st = bf16_rne(step_f32.astype(np.float64))
    step = bf16_bits_to_f64(st).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        q = g / step[..., None]
    codes = np.clip(np.rint(q) + CODE_ZERO, 0, 15)
    codes = np.where(step[..., None] == 0, CODE_ZERO, codes)
    codes = codes.astype(np.uint8).reshape(n, k)
    return pack_codes(codes), st


# --------------------------------------------------------------------------
# acceptance bound
# --------------------------------------------------------------------------
REL_BOUND = 2e-3


def bound_violations(y_bits: np.ndarray, y_ref: np.ndarray, abs_ref: np.ndarray,
                     rel: float = REL_BOUND) -> np.ndarray:
    """Boolean mask of outputs outside |y - y_ref| <= rel * sum|w x| + ulp(y_ref).

    ``y_bits`` are the bf16 results, ``y_ref`` the unrounded fp64 sums and
    ``abs_ref`` the fp64 sums of |w x|.  +0 and -0 compare equal.  A
    non-finite reference requires a result of the same class: +inf for +inf,
    -inf for -inf, a NaN for a NaN.
    """
    y = bf16_bits_to_f64(y_bits)
    y_ref = np.asarray(y_ref, dtype=np.float64)
    ref_finite = np.isfinite(y_ref)
    with np.errstate(invalid="ignore"):
        err = np.abs(y - y_ref)
        ok = err <= rel * np.asarray(abs_ref) + ulp_bf16(y_ref)
    same_class = (np.isnan(y) & np.isnan(y_ref)) | (np.isinf(y_ref) & (y == y_ref))
    ok = np.where(ref_finite, ok & np.isfinite(y), same_class)
    return ~ok


def within_bound(y_bits, y_ref, abs_ref, rel: float = REL_BOUND) -> bool:
    return not bool(np.any(bound_violations(y_bits, y_ref, abs_ref, rel)))
