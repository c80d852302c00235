/*
 * Exhaustive check of the float-bit dequantisation identities.  TEST
 * INFRASTRUCTURE: built by __graft_entry__.build() and run by the CPU tests.
 *
 * Page "Gemma 4 on a 4 GB GPU in Plain PyTorch", section "Step 3 — Multiply
 * Straight From the Packed Weights": placing a 4-bit code c in the low
 * mantissa bits of the float 2^23 and then subtracting 2^23 + 8 yields c - 8
 * exactly.  The same idea works in 16-bit formats, where the magic constant
 * is 2^10 (fp16, mantissa 10 bits) or 2^7 (bf16, mantissa 7 bits).  The CUDA
 * kernels use the fp16 form on two codes at a time; this program checks every
 * code against the plain integer c - 8, decoding the 16-bit patterns by hand.
 *
 * Prints one line per code:  c  fp32-bits  fp32-result  fp16-lo  fp16-hi  bf16
 * and exits 0 when every identity holds, 1 otherwise.
 */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

static float f32_from_bits(uint32_t b) { float f; memcpy(&f, &b, 4); return f; }

/* value of an fp16 bit pattern (normal or zero only; enough for these cases) */
static double f16_value(uint16_t h) {
    int sign = (h >> 15) & 1, e = (h >> 10) & 0x1F, m = h & 0x3FF;
    double v;
    if (e == 0) v = (double)m / 1024.0 / 16384.0;          /* subnormal */
    else {
        v = 1.0 + (double)m / 1024.0;
        for (int i = 15; i < e; ++i) v *= 2.0;
        for (int i = e; i < 15; ++i) v /= 2.0;
    }
    return sign ? -v : v;
}

/* value of a bf16 bit pattern via its fp32 widening */
static double bf16_value(uint16_t b) { return (double)f32_from_bits((uint32_t)b << 16); }

int main(void) {
    int bad = 0;
    for (uint32_t c = 0; c < 16; ++c) {
        int want = (int)c - 8;
        /* fp32: (0x4B000000 | c) is 2^23 + c; minus (2^23 + 8) is c - 8 */
        uint32_t b32 = 0x4B000000u | c;
        float r32 = f32_from_bits(b32) - 8388616.0f;
        /* fp16, code in bits 0..3: 0x6400 | c is 1024 + c */
        double r16lo = f16_value((uint16_t)(0x6400u | c)) - 1032.0;
        /* fp16, code in bits 4..7: 0x6400 | (c << 4) is 1024 + 16 c */
        double r16hi = f16_value((uint16_t)(0x6400u | (c << 4))) / 16.0 - 72.0;
        /* bf16, code in bits 0..3: 0x4300 | c is 128 + c */
        double r16b = bf16_value((uint16_t)(0x4300u | c)) - 136.0;
        int ok = (r32 == (float)want) && (r16lo == want) && (r16hi == want) && (r16b == want);
        if (!ok) bad = 1;
        printf("%2u 0x%08X %+.1f %+.1f %+.1f %+.1f %s\n", c, b32, (double)r32, r16lo, r16hi,
               r16b, ok ? "ok" : "MISMATCH");
    }
    return bad;
}
