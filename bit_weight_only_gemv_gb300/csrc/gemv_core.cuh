// Device building blocks shared by the W4A16 GEMV kernels (gemv.cu, chain.cu):
// the staged activation format, the float-bit dequantisation of packed codes,
// the dot of one group of 32 codes and the fixed reductions.  The per-row
// arithmetic of every kernel that includes this file is therefore the same,
// which keeps their results bitwise equal.
#pragma once

#include "common.cuh"

namespace w4 {

// ---------------------------------------------------------------- staging
// Staged form of one group of 32 activations: four 16-byte chunks
// w = 0..3 of fp16 pairs (x[8w+p], x[8w+p+4]) for p = 0..3, at dst + w *
// plane, scaled by 2^e so that the group's largest magnitude lies in
// [2^9, 2^10) (exact for bf16 values within 2^26 of the group maximum), and
// the inverse scale 2^-e at *scale (0 for a padding group past the row's
// end, whose activations are zero).  `v` holds the group's 32 bf16 values
// in order (all zero for a padding group).
__device__ __forceinline__ void store_staged_group(const uint4 v[4], uint8_t* dst, int plane,
                                                   float* scale, bool valid) {
  uint32_t mx = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    mx = __vmaxu2(mx, v[i].x & 0x7FFF7FFFu);
    mx = __vmaxu2(mx, v[i].y & 0x7FFF7FFFu);
    mx = __vmaxu2(mx, v[i].z & 0x7FFF7FFFu);
    mx = __vmaxu2(mx, v[i].w & 0x7FFF7FFFu);
  }
  mx = max(mx & 0xFFFFu, mx >> 16);
  int e = 0;
  float inv = 1.0f;
  if (mx != 0) {
    const int ef = (int)(mx >> 7);                 // biased exponent, 0..255
    const int E = (ef == 0) ? -127 : ef - 127;     // unbiased (subnormal: -127)
    e = 9 - E;                                     // max * 2^e in [2^9, 2^10)
    const int ei = E - 9;                          // inverse scale exponent
    inv = (ei >= -126) ? __int_as_float((ei + 127) << 23) : __int_as_float(1 << (ei + 149));
  }
  const int ea = e >> 1, eb = e - ea;              // split so each factor is normal
  const float fa = __int_as_float((ea + 127) << 23);
  const float fb = __int_as_float((eb + 127) << 23);
  const uint32_t* wv = reinterpret_cast<const uint32_t*>(v);
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    float f[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t pair = wv[4 * w + i];       // elements 8w+2i, 8w+2i+1
      f[2 * i] = __uint_as_float(pair << 16) * fa * fb;
      f[2 * i + 1] = __uint_as_float(pair & 0xFFFF0000u) * fa * fb;
    }
    uint4 out;
    __half2 h;
    h = __floats2half2_rn(f[0], f[4]);
    out.x = *reinterpret_cast<uint32_t*>(&h);
    h = __floats2half2_rn(f[1], f[5]);
    out.y = *reinterpret_cast<uint32_t*>(&h);
    h = __floats2half2_rn(f[2], f[6]);
    out.z = *reinterpret_cast<uint32_t*>(&h);
    h = __floats2half2_rn(f[3], f[7]);
    out.w = *reinterpret_cast<uint32_t*>(&h);
    *reinterpret_cast<uint4*>(dst + w * plane) = out;
  }
  *scale = valid ? inv : 0.0f;
}

// The same for 32 fp32 values h (largest magnitude mx), each rounded once to
// fp16 after the power-of-two scaling.
__device__ __forceinline__ void store_staged_group_f32(const float h[32], float mx, uint8_t* dst,
                                                       int plane, float* scale, bool valid) {
  int e = 0;
  float inv = 1.0f;
  if (mx != 0.0f) {
    const int ef = (int)((__float_as_uint(mx) >> 23) & 0xFF);
    const int E = (ef == 0) ? -127 : ef - 127;
    e = 9 - E;                                     // max * 2^e in [2^9, 2^10)
    const int ei = E - 9;
    inv = (ei >= -126) ? __int_as_float((ei + 127) << 23) : __int_as_float(1 << (ei + 149));
  }
  const int ea = e >> 1, eb = e - ea;              // split so each factor is normal
  const float fa = __int_as_float((ea + 127) << 23);
  const float fb = __int_as_float((eb + 127) << 23);
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    uint4 out;
    __half2 hp;
    hp = __floats2half2_rn(h[8 * w] * fa * fb, h[8 * w + 4] * fa * fb);
    out.x = *reinterpret_cast<uint32_t*>(&hp);
    hp = __floats2half2_rn(h[8 * w + 1] * fa * fb, h[8 * w + 5] * fa * fb);
    out.y = *reinterpret_cast<uint32_t*>(&hp);
    hp = __floats2half2_rn(h[8 * w + 2] * fa * fb, h[8 * w + 6] * fa * fb);
    out.z = *reinterpret_cast<uint32_t*>(&hp);
    hp = __floats2half2_rn(h[8 * w + 3] * fa * fb, h[8 * w + 7] * fa * fb);
    out.w = *reinterpret_cast<uint32_t*>(&hp);
    *reinterpret_cast<uint4*>(dst + w * plane) = out;
  }
  *scale = valid ? inv : 0.0f;
}

// Gated activation of one group: h = silu(gate) * up = gate / (1 + e^-gate)
// * up in fp32, from the group's 32 bf16 gate values `gv` and up values
// `uv`; returns the largest |h|.
__device__ __forceinline__ float silu_mul_group(const uint4 gv[4], const uint4 uv[4],
                                                float h[32]) {
  float mx = 0.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t gw[4] = {gv[i].x, gv[i].y, gv[i].z, gv[i].w};
    const uint32_t uw[4] = {uv[i].x, uv[i].y, uv[i].z, uv[i].w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        const float gf = __uint_as_float(b ? (gw[q] & 0xFFFF0000u) : (gw[q] << 16));
        const float uf = __uint_as_float(b ? (uw[q] & 0xFFFF0000u) : (uw[q] << 16));
        // every CTA forms the whole row: the fast exponential and
        // division (relative error near 2^-21, below the staging's
        // 2^-11; 0 below gate = -87, where the product is under 2^-120)
        const float v = __fdividef(gf * uf, 1.0f + __expf(-gf));
        h[8 * i + 2 * q + b] = v;
        mx = fmaxf(mx, fabsf(v));
      }
    }
  }
  return mx;
}

// ---------------------------------------------------------------- the dot
__device__ __forceinline__ __half2 u2h(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

// Four fp16 pairs (c - 8) of one packed word, in pair order
// (nibble 0, 4), (1, 5), (2, 6), (3, 7).
__device__ __forceinline__ void unpack_word(uint32_t wd, __half2 h[4]) {
  const __half2 k1032 = u2h(0x64086408u);   // 1032
  const __half2 k16th = u2h(0x2C002C00u);   // 1/16
  const __half2 km72 = u2h(0xD480D480u);    // -72
  const uint32_t s8 = wd >> 8;
  h[0] = __hsub2(u2h(and_or(wd, 0x000F000Fu, 0x64006400u)), k1032);
  h[1] = __hfma2(u2h(and_or(wd, 0x00F000F0u, 0x64006400u)), k16th, km72);
  h[2] = __hsub2(u2h(and_or(s8, 0x000F000Fu, 0x64006400u)), k1032);
  h[3] = __hfma2(u2h(and_or(s8, 0x00F000F0u, 0x64006400u)), k16th, km72);
}

// c + lo + hi of an fp16 pair, each add in fp32 (exact widening).
__device__ __forceinline__ float add_pair_f32(float c, __half2 v) {
  float d;
  const uint32_t u = *reinterpret_cast<uint32_t*>(&v);
  asm("{\n\t.reg .f16 lo, hi;\n\t"
      "mov.b32 {lo, hi}, %1;\n\t"
      "add.rn.f32.f16 %0, lo, %2;\n\t"
      "add.rn.f32.f16 %0, hi, %0;\n\t}"
      : "=f"(d)
      : "r"(u), "f"(c));
  return d;
}

// Dot of one group (4 packed words) with one staged activation row.
__device__ __forceinline__ float group_sum(const uint4 q, const uint4 xv[4]) {
  __half2 h[4][4];
  unpack_word(q.x, h[0]);
  unpack_word(q.y, h[1]);
  unpack_word(q.z, h[2]);
  unpack_word(q.w, h[3]);
  __half2 a0 = u2h(0u), a1 = u2h(0u), a2 = u2h(0u), a3 = u2h(0u);
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    a0 = __hfma2(h[w][0], u2h(xv[w].x), a0);
    a1 = __hfma2(h[w][1], u2h(xv[w].y), a1);
    a2 = __hfma2(h[w][2], u2h(xv[w].z), a2);
    a3 = __hfma2(h[w][3], u2h(xv[w].w), a3);
  }
  float gs = add_pair_f32(0.0f, a0);
  gs = add_pair_f32(gs, a1);
  gs = add_pair_f32(gs, a2);
  return add_pair_f32(gs, a3);
}

// One chunk of a tile: for each of its `ns` groups per lane, the
// lane loads the group's staged activations (MR rows) once and applies them
// to its RW rows.  acc[j][m] = sum over the chunk's groups, in group order.
// TT, CLT > 0 fix the team size and the (always full) chunk length at compile
// time, so every shared-memory offset is an immediate.  gleft: groups of the
// row left from this lane's first one (fewer than the chunk only when the
// team pads K/32; the generic kernel then drops the padding groups).
template <int MR, int RW, int TT, int CLT>
__device__ __forceinline__ void tile_dot(const uint8_t* sm, uint32_t xo, uint32_t xso, int xplane,
                                         int xmrow, int xsmrow, const uint32_t co[RW],
                                         const uint32_t so[RW], int ns, int T, int gleft,
                                         float acc[RW][MR]) {
#pragma unroll
  for (int j = 0; j < RW; ++j)
#pragma unroll
    for (int m = 0; m < MR; ++m) acc[j][m] = 0.0f;
  const int gstep = (TT > 0 ? TT : T) * 16;          // bytes between a lane's groups
  const int sstep = gstep >> 3, xsstep = gstep >> 2;  // the same for steps, scales
  auto group = [&](int s) {
    uint4 xv[MR][4];
    float inv[MR];
#pragma unroll
    for (int m = 0; m < MR; ++m) {
#pragma unroll
      for (int w = 0; w < 4; ++w)
        xv[m][w] = *reinterpret_cast<const uint4*>(sm + xo + m * xmrow + w * xplane + s * gstep);
      inv[m] = *reinterpret_cast<const float*>(sm + xso + m * xsmrow + s * xsstep);
    }
#pragma unroll
    for (int j = 0; j < RW; ++j) {
      const uint4 q = *reinterpret_cast<const uint4*>(sm + co[j] + s * gstep);
      float stf = bf16_bits_to_float(*reinterpret_cast<const uint16_t*>(sm + so[j] + s * sstep));
      // padding groups (generic kernel only): their shared bytes belong to
      // the next row, so the step is dropped (activations there are zero)
      if (TT == 0 && s * T >= gleft) stf = 0.0f;
#pragma unroll
      for (int m = 0; m < MR; ++m) acc[j][m] = fmaf(group_sum(q, xv[m]) * inv[m], stf, acc[j][m]);
    }
  };
  if constexpr (CLT > 0) {
#pragma unroll
    for (int s = 0; s < CLT; ++s) group(s);
  } else {
#pragma unroll 4
    for (int s = 0; s < ns; ++s) group(s);
  }
}

// Sum over the T lanes of a team with a fixed xor tree (T a power of two;
// TT > 0: T = TT known at compile time).
template <int TT>
__device__ __forceinline__ float team_sum(float v, int T) {
  if (TT > 0) {
#pragma unroll
    for (int off = TT >> 1; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  } else {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
      if (off < T) v += __shfl_xor_sync(0xffffffffu, v, off);
  }
  return v;
}

}  // namespace w4
