// W4A16 group-32 GEMV and routed-expert GEMV for GB300 (sm_103a).
//
// Page "Gemma 4 on a 4 GB GPU in Plain PyTorch", section "Step 3 — Multiply
// Straight From the Packed Weights": a decode step multiplies one activation
// vector by every weight matrix straight from the packed 4-bit words, so the
// speed limit is how fast the weights stream from memory.  The routed-expert
// variant (page "Running a 26B MoE on an 8 GB Jetson by streaming experts from
// SSD", section "Streaming without touching a single GPU kernel") reads expert
// `id` at base + id * stride.
//
// Design (persistent CTAs of 8 warps, one or two per SM):
//  * The activation rows are staged once per CTA in shared memory as fp16
//    pairs scaled by a power of two per group of 32 (exact), next to the
//    group's inverse scale.
//  * A team of `team` lanes shares an output row (team = the largest power
//    of two <= 32 dividing K/32 that leaves each lane >= 8 groups of a row,
//    so no lane idles); each lane walks the groups lane, lane + team, ...
//  * Packed codes and steps go straight from HBM to registers with coalesced
//    128-bit (codes) loads that bypass L1; the weights never touch shared
//    memory, which keeps shared-memory bandwidth for the activations.
//  * Per group and row the lane turns each packed word into four fp16 pairs
//    (c - 8) with the float-bit trick of the page in its fp16 form
//    ((0x6400 | c) - 1032 = c - 8, exact), multiplies them with the fp16
//    activation pairs in packed fp16 (products exact), sums each pair lane
//    over the group's 4 words in fp16 (at most 3 roundings: 3 * 2^-11 of
//    sum|w x|), adds the 8 partial sums in fp32, rescales by the group's 2^-e
//    (exact), multiplies by the step and accumulates in fp32.
//  * K is cut into chunks of 8 groups per lane; the loads of the next chunk
//    are in flight (second register buffer) while a chunk is computed, and
//    the first chunk is requested before waiting on the previous kernel.
//    After each chunk the team reduces with a fixed xor-shuffle tree and
//    chunk sums are added in chunk order.  A row's arithmetic therefore
//    depends on K only, never on N, the row index, the split or the
//    addresses: results are bitwise reproducible and a gemv_id row equals
//    the gemv of that expert.
//  * Work unit = (row block of 32/team rows, K slice).  Each CTA owns a
//    balanced contiguous range of units; its warps take them round-robin.
//    Split-K (slices > 1): chunk sums go to the workspace and the warp that
//    finishes a row block last (atomic counter, no waiting) adds them in
//    chunk order, writes the rows and re-arms the counter.
//  * With W4_FLAG_PDL the launch may overlap the previous kernel in the
//    stream; all global reads and writes happen after waiting for it.
#include <algorithm>
#include <mutex>

#include "common.cuh"

namespace w4 {

constexpr int kWarps = 8;
constexpr int kThreads = 32 * kWarps;
constexpr int kCtasPerSm = 2;    // two resident CTAs per SM: this launch and the next
constexpr int kMaxMR = 4;        // activation rows per launch
constexpr int kChunkPerLane = 8; // groups per lane per chunk

struct GemvParams {
  const uint8_t* qw;
  const uint8_t* st;
  unsigned long long qw_item_stride;   // bytes between experts (0: dense)
  unsigned long long st_item_stride;
  const int32_t* ids;                  // nullptr for dense
  int num_experts;
  const __nv_bfloat16* x;
  int x_per_item;                      // 1: item i uses activation row i
  __nv_bfloat16* y;
  int MR;                              // activation rows per item in this launch
  int N, K, Kg;
  int n_items;
  int team, sets, R, rows_per_unit;    // lanes per row, row sets per warp, rows per lane
  int chunk, nch;                      // groups per chunk (team * 8), chunks per row
  int S, cps, upi;                     // slices, chunks per slice, row blocks per item
  int B, U;                            // row blocks, units (= S * B)
  int x_slots;                         // activation rows staged per CTA (per MR row)
  int* ws_count;                       // [B] at the start of the workspace
  float* ws_partial;                   // [B][nch][rows_per_unit][MR] after it
  int32_t* status;
};

// ---------------------------------------------------------------- activations
// Stage the activation rows of `nslots` items (or one shared row) as fp16
// pairs scaled by 2^e per group of 32 so that the group's largest magnitude
// lies in [2^9, 2^10).  Layout for staged row j (= slot * MR + m): 16-byte
// chunk (w, g) = pairs (x[8w+p], x[8w+p+4]) for p = 0..3 of group g, at
// ((j * 4 + w) * Kg + g) * 16; the inverse scale 2^-e of the group at
// xscale[j * Kg + g].
__device__ void stage_x(const GemvParams& p, int item0, int nslots, uint8_t* xs, float* xscale) {
  const int rows = nslots * p.MR;
  for (int idx = threadIdx.x; idx < rows * p.Kg; idx += kThreads) {
    const int j = idx / p.Kg;
    const int g = idx - j * p.Kg;
    const int slot = j / p.MR, m = j - slot * p.MR;
    const int xrow = (p.x_per_item ? (item0 + slot) * p.MR : 0) + m;
    const uint4* src =
        reinterpret_cast<const uint4*>(p.x + (long long)xrow * p.K + (long long)g * 32);
    uint4 v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = __ldg(src + i);
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
      *reinterpret_cast<uint4*>(xs + ((long long)(j * 4 + w) * p.Kg + g) * 16) = out;
    }
    xscale[(long long)j * p.Kg + g] = inv;
  }
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

__device__ __forceinline__ uint4 ldg_stream16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t ldg_stream2(const void* p) {
  unsigned short v;
  asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

// Lanes of one warp: ask L2 for the codes and steps of unit `u` (rows of the
// unit's row block, groups of its K slice).  Ranges are clipped to 16-byte
// lines inside the item's arrays; bytes outside them are simply not
// prefetched.
__device__ __forceinline__ void prefetch_unit(const GemvParams& p, int u, int lane) {
  if (u >= p.U) return;
  const int slice = u / p.B;
  const int rb = u - slice * p.B;
  const int item = rb / p.upi;
  const int row0 = (rb - item * p.upi) * p.rows_per_unit;
  const int rows = min(p.rows_per_unit, p.N - row0);
  long long blk = item;
  if (p.ids != nullptr) {
    const int e = __ldg(p.ids + item);
    if (e < 0 || e >= p.num_experts) return;
    blk = e;
  }
  const uint8_t* qw = p.qw + (unsigned long long)blk * p.qw_item_stride;
  const uint8_t* st = p.st + (unsigned long long)blk * p.st_item_stride;
  const long long row_bytes = (long long)p.K / 2, st_row = (long long)p.Kg * 2;
  const long long st_lim = ((long long)p.N * st_row) & ~15LL;
  const int g0 = slice * p.cps * p.chunk;
  const int g1 = min((slice + 1) * p.cps * p.chunk, p.Kg);
  if (p.S == 1) {   // whole rows: one contiguous range each for codes and steps
    if (lane == 0) {
      prefetch_l2_bulk(qw + row0 * row_bytes, (uint32_t)(rows * row_bytes));
      const long long b = (row0 * st_row) & ~15LL;
      const long long e = min((((long long)(row0 + rows) * st_row) + 15) & ~15LL, st_lim);
      if (e > b) prefetch_l2_bulk(st + b, (uint32_t)(e - b));
    }
  } else if (lane < rows) {
    const long long r = row0 + lane;
    prefetch_l2_bulk(qw + r * row_bytes + (long long)g0 * 16, (uint32_t)(g1 - g0) * 16);
    const long long b = (r * st_row + (long long)g0 * 2) & ~15LL;
    const long long e = min((r * st_row + (long long)g1 * 2 + 15) & ~15LL, st_lim);
    if (e > b) prefetch_l2_bulk(st + b, (uint32_t)(e - b));
  }
}

// ---------------------------------------------------------------- kernel
// A warp's position in its walk over (unit, chunk) pairs.  Chunk c of a unit
// holds, for this lane, the groups g = c*chunk + lane_in_team + s*team for
// s < steps (steps = chunk / team, smaller only in a ragged last chunk).
struct Cursor {
  int u;                // current unit (>= end when the walk is over)
  int c, c_end;         // chunk and end chunk of the unit's slice
  int steps;            // groups of this chunk per lane
  int g;                // this lane's first group of the chunk
  int item, rb, slice;
  int row;              // this lane's row
  const uint8_t* qrow;  // codes of the row
  const uint8_t* srow;  // steps of the row

  __device__ void set_chunk(const GemvParams& p, int lt) {
    g = c * p.chunk + lt;
    steps = (min((c + 1) * p.chunk, p.Kg) - c * p.chunk) / p.team;
  }
  // First unit at or after uu (stride kWarps) with a valid expert id.
  __device__ void seek(const GemvParams& p, int uu, int ue, int lt, int set, bool rep) {
    for (u = uu; u < ue; u += kWarps) {
      if (p.S == 1) {          // common cases without divisions
        slice = 0;
        rb = u;
      } else {
        slice = u / p.B;
        rb = u - slice * p.B;
      }
      item = (p.n_items == 1) ? 0 : rb / p.upi;
      row = (rb - item * p.upi) * p.rows_per_unit + set;
      long long blk = item;
      if (p.ids != nullptr) {
        const int e = __ldg(p.ids + item);
        if (e < 0 || e >= p.num_experts) {   // leave this unit's rows unwritten
          if (rep) report(p.status, W4_ERR_INDEX);
          continue;
        }
        blk = e;
      }
      c = slice * p.cps;
      c_end = min(c + p.cps, p.nch);
      set_chunk(p, lt);
      qrow = p.qw + (unsigned long long)blk * p.qw_item_stride + (long long)row * (p.K / 2);
      srow = p.st + (unsigned long long)blk * p.st_item_stride + (long long)row * (p.Kg * 2);
      return;
    }
  }
  __device__ void next_chunk(const GemvParams& p, int ue, int lt, int set, bool rep) {
    if (++c < c_end) {
      set_chunk(p, lt);
      return;
    }
    seek(p, u + kWarps, ue, lt, set, rep);
  }
};

// Chunk register buffer: CS groups of one row for this lane.  CS > 0: every
// chunk has exactly CS steps; CS == 0: up to kChunkPerLane, guarded.
template <int CS>
struct Buf {
  static constexpr int kN = CS > 0 ? CS : kChunkPerLane;
  uint4 code[kN];
  uint32_t sb[kN];
};

// Load the codes and steps of cursor c's chunk (rows past N and steps past a
// ragged chunk get code 8 and step 0, which contribute nothing).
template <int CS>
__device__ __forceinline__ void load_chunk(const GemvParams& p, const Cursor& c, Buf<CS>& b) {
  const uint8_t* q = c.qrow + c.g * 16;
  const uint8_t* st = c.srow + c.g * 2;
  const int qstep = p.team * 16, sstep = p.team * 2;
  if (c.row < p.N) {
#pragma unroll
    for (int s = 0; s < Buf<CS>::kN; ++s) {
      if (CS > 0 || s < c.steps) {
        b.code[s] = ldg_stream16(q + s * qstep);
        b.sb[s] = ldg_stream2(st + s * sstep);
      } else {
        b.code[s] = make_uint4(0x88888888u, 0x88888888u, 0x88888888u, 0x88888888u);
        b.sb[s] = 0;
      }
    }
  } else {
#pragma unroll
    for (int s = 0; s < Buf<CS>::kN; ++s) {
      b.code[s] = make_uint4(0x88888888u, 0x88888888u, 0x88888888u, 0x88888888u);
      b.sb[s] = 0;
    }
  }
}

// Sum over the chunk's steps, in step order, for every activation row.
template <int CS, int MR>
__device__ __forceinline__ void chunk_dot(const GemvParams& p, const Cursor& c, const Buf<CS>& b,
                                          const uint8_t* xrow, const float* srow, float acc[MR]) {
  const int kgs = p.Kg * 16;                 // bytes between the 4 word planes
  const uint8_t* x0 = xrow + c.g * 16;
  const float* s0 = srow + c.g;
  const int xstep = p.team * 16;
#pragma unroll
  for (int m = 0; m < MR; ++m) acc[m] = 0.0f;
#pragma unroll
  for (int s = 0; s < Buf<CS>::kN; ++s) {
    if (CS == 0 && s >= c.steps) break;
#pragma unroll
    for (int m = 0; m < MR; ++m) {
      const uint8_t* xp = x0 + m * 4 * kgs + s * xstep;
      uint4 xv[4];
#pragma unroll
      for (int w = 0; w < 4; ++w) xv[w] = *reinterpret_cast<const uint4*>(xp + w * kgs);
      const float sc = s0[m * p.Kg + s * p.team];
      acc[m] = fmaf(group_sum(b.code[s], xv) * sc, bf16_bits_to_float(b.sb[s]), acc[m]);
    }
  }
}

constexpr int kPrefetchUnits = 2;   // units per warp requested into L2 before the PDL wait

// Chunks longer than 8 steps, or several activation rows, need more
// registers: one CTA per SM.
constexpr int ctas_per_sm(int cs, int mr) { return (cs > 8 || mr > 1) ? 1 : kCtasPerSm; }

template <int MR, int CS>
__global__ void __launch_bounds__(kThreads, ctas_per_sm(CS, MR)) gemv_kernel(const __grid_constant__ GemvParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int team = p.team;
  const int set = lane / team;   // row set (= row of the unit) of this lane
  const int lt = lane - set * team;
  const int ub = (int)((long long)blockIdx.x * p.U / gridDim.x);
  const int ue = (int)((long long)(blockIdx.x + 1) * p.U / gridDim.x);

  // items whose activation rows this CTA needs (units are slice-major)
  int item0 = 0, nslots = 1;
  if (p.x_per_item) {
    const int rb_lo = ub % p.B, rb_hi = (ue - 1) % p.B;
    if (ue - ub >= p.B || rb_lo > rb_hi) {
      item0 = 0;
      nslots = p.n_items;
    } else {
      item0 = rb_lo / p.upi;
      nslots = rb_hi / p.upi - item0 + 1;
    }
  }
  uint8_t* xs = smem;
  float* xscale = reinterpret_cast<float*>(smem + (long long)p.x_slots * MR * 4 * p.Kg * 16);

  // Compute cursor `cp` and load cursor `ld` one chunk ahead; two register
  // buffers used in turn.  Dense weights do not depend on earlier kernels:
  // this warp's first units are requested into L2 and its first chunk into
  // registers before waiting for the previous kernel (W4_FLAG_PDL), so a
  // launch that is resident early has its weights in flight already.  Routed
  // ids may come from the previous kernel and are read after the wait.
  Cursor cp, ld;
  Buf<CS> ba, bb;
  const bool dense = p.ids == nullptr;
  if (!dense) pdl_wait();
  for (int d = 0; d < kPrefetchUnits; ++d)
    if (ub + warp + d * kWarps < ue) prefetch_unit(p, ub + warp + d * kWarps, lane);
  cp.seek(p, ub + warp, ue, lt, set, true);
  ld = cp;
  if (ld.u < ue) {
    load_chunk<CS>(p, ld, ba);
    ld.next_chunk(p, ue, lt, set, false);
  }
  if (dense) pdl_wait();     // activations and outputs follow earlier kernels
  pdl_launch_dependents();
  if (ub < ue) stage_x(p, item0, nslots, xs, xscale);
  __syncthreads();

  float rowsum[MR];
#pragma unroll
  for (int m = 0; m < MR; ++m) rowsum[m] = 0.0f;

  // End of a chunk: team reduction (fixed xor tree), then the chunk sum goes
  // to the row sum, or to the workspace under split-K.
  auto finish_chunk = [&](float acc[MR]) {
#pragma unroll
    for (int m = 0; m < MR; ++m)
      for (int off = team >> 1; off > 0; off >>= 1) acc[m] += __shfl_xor_sync(0xffffffffu, acc[m], off);
    const bool unit_end = cp.c + 1 == cp.c_end;
    if (p.S == 1) {
#pragma unroll
      for (int m = 0; m < MR; ++m) rowsum[m] += acc[m];
      if (unit_end) {
        if (lt == 0 && cp.row < p.N) {
#pragma unroll
          for (int m = 0; m < MR; ++m)
            p.y[((long long)cp.item * MR + m) * p.N + cp.row] = __float2bfloat16_rn(rowsum[m]);
        }
#pragma unroll
        for (int m = 0; m < MR; ++m) rowsum[m] = 0.0f;
      }
      return;
    }
    if (lt == 0) {
      float* dst = p.ws_partial + (((long long)cp.rb * p.nch + cp.c) * p.rows_per_unit + set) * MR;
#pragma unroll
      for (int m = 0; m < MR; ++m) dst[m] = acc[m];
    }
    if (unit_end) {
      // the last warp to finish this row block adds the chunk sums in chunk
      // order, writes the rows and re-arms the counter
      __threadfence();
      __syncwarp();
      int last = 0;
      if (lane == 0) last = atomicAdd(p.ws_count + cp.rb, 1) == p.S - 1;
      last = __shfl_sync(0xffffffffu, last, 0);
      if (last) {
        __threadfence();
        const int rbase = (cp.rb - cp.item * p.upi) * p.rows_per_unit;
        const float* src = p.ws_partial + (long long)cp.rb * p.nch * p.rows_per_unit * MR;
        for (int e = lane; e < p.rows_per_unit * MR; e += 32) {
          const int r = e / MR, m = e - r * MR;
          if (rbase + r >= p.N) continue;
          float v = 0.0f;
          for (int c = 0; c < p.nch; ++c) v += __ldcg(src + ((long long)c * p.rows_per_unit + r) * MR + m);
          p.y[((long long)cp.item * MR + m) * p.N + rbase + r] = __float2bfloat16_rn(v);
        }
        if (lane == 0) atomicExch(p.ws_count + cp.rb, 0);
      }
    }
  };

  while (cp.u < ue) {
#pragma unroll
    for (int phase = 0; phase < 2; ++phase) {   // buffers ba, bb in turn
      Buf<CS>& curb = phase == 0 ? ba : bb;
      Buf<CS>& nxtb = phase == 0 ? bb : ba;
      if (cp.u >= ue) break;
      if (ld.u < ue) {   // next chunk's loads fly while this one is computed
        load_chunk<CS>(p, ld, nxtb);
        ld.next_chunk(p, ue, lt, set, false);
      }
      const int xslot = p.x_per_item ? cp.item - item0 : 0;
      float acc[MR];
      chunk_dot<CS, MR>(p, cp, curb, xs + (long long)xslot * MR * 4 * p.Kg * 16,
                        xscale + (long long)xslot * MR * p.Kg, acc);
      finish_chunk(acc);
      cp.next_chunk(p, ue, lt, set, true);
    }
  }
}

// ================================================================= host side
namespace {

struct DeviceInfo {
  int sms = 0;
  int smem_optin = 0;
};

DeviceInfo device_info(int dev) {
  static std::mutex mu;
  static DeviceInfo cache[64];
  std::lock_guard<std::mutex> lock(mu);
  if (dev < 0 || dev >= 64) return DeviceInfo{};
  if (cache[dev].sms == 0) {
    int sms = 0, smem = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess) {
      cudaGetLastError();
      return DeviceInfo{};
    }
    cache[dev].sms = sms;
    cache[dev].smem_optin = smem;
  }
  return cache[dev];
}

struct Plan {
  int MR = 1;
  int team = 32, sets = 1, R = 1, rows_per_unit = 1;
  int chunk = 0, nch = 1, cs = 0;
  int S = 1, cps = 1, upi = 1;
  long long B = 0, U = 0;
  int x_slots = 1;
  int ctas = 0;
  long long smem = 0;
  size_t ws_bytes = 0;
  size_t ws_part_off = 0;
};

// The per-row arithmetic (team, chunk) comes from K alone.  team: the largest
// power of two <= 32 dividing K/32 that leaves each lane >= kChunkPerLane
// groups of a row.  Chunk steps per lane: the largest divisor of the lane's
// groups per row in 5..12, so every chunk is full (0 = none: chunks of
// kChunkPerLane steps, the last one ragged).
void row_shape(int K, int* team, int* chunk, int* nch, int* cs) {
  const int Kg = K / 32;
  int t = 1;
  while (t < 32 && Kg % (2 * t) == 0 && Kg / (2 * t) >= kChunkPerLane) t *= 2;
  *team = t;
  const int q = Kg / t;
  int c = 0;
  for (int d = 12; d >= 5 && c == 0; --d)
    if (q % d == 0) c = d;
  if (q <= 12) c = q;             // a whole row per chunk
  if (c != 0 && c != 7 && c != 8 && c != 11 && c != 12 && c != 5 && c != 6 && c != 9 && c != 10)
    c = 0;
  *cs = c;
  *chunk = t * (c > 0 ? c : kChunkPerLane);
  *nch = (Kg + *chunk - 1) / *chunk;
}

long long x_bytes(int slots, int MR, int Kg) {
  return (long long)slots * MR * Kg * (64 + 4);
}

bool make_plan(int MR, int N, int K, int n_items, int allow_split, int x_per_item,
               const DeviceInfo& di, Plan* out) {
  Plan pl;
  pl.MR = MR;
  const int Kg = K / 32;
  row_shape(K, &pl.team, &pl.chunk, &pl.nch, &pl.cs);
  pl.sets = 32 / pl.team;
  const int sms = di.sms > 0 ? di.sms : 1;
  const long long warps = (long long)sms * kWarps * kCtasPerSm;
  const long long want = 6 * warps;       // units for a balanced split over warps
  pl.R = 1;   // one row per lane
  pl.rows_per_unit = pl.sets;
  pl.upi = (N + pl.rows_per_unit - 1) / pl.rows_per_unit;
  pl.B = (long long)n_items * pl.upi;
  if (pl.B > (1LL << 30)) return false;
  int S = 1;
  if (allow_split && pl.nch > 1 && pl.B < want)
    S = (int)std::min<long long>(pl.nch, (want + pl.B - 1) / pl.B);
  pl.cps = (pl.nch + S - 1) / S;
  pl.S = (pl.nch + pl.cps - 1) / pl.cps;
  pl.U = (long long)pl.S * pl.B;
  if (pl.U > (1LL << 30)) return false;
  // One CTA per SM leaves room for the next launch's CTA (PDL); problems
  // with many units per warp fill two CTAs per SM instead.
  const int cap = ctas_per_sm(pl.cs, MR);
  const long long per_sm = (pl.U >= (long long)cap * sms * kWarps) ? cap : 1;
  pl.ctas = (int)std::min<long long>(pl.U, per_sm * sms);
  // activation rows a CTA stages: one, or the items its unit range touches
  pl.x_slots = 1;
  if (x_per_item) {
    for (int c = 0; c < pl.ctas; ++c) {
      const long long ub = (long long)c * pl.U / pl.ctas, ue = (long long)(c + 1) * pl.U / pl.ctas;
      if (ue <= ub) continue;
      const long long lo = ub % pl.B, hi = (ue - 1) % pl.B;
      const long long n = (ue - ub >= pl.B || lo > hi) ? n_items : hi / pl.upi - lo / pl.upi + 1;
      pl.x_slots = (int)std::max<long long>(pl.x_slots, n);
    }
  }
  pl.smem = x_bytes(pl.x_slots, MR, Kg);
  const long long smem_max = di.smem_optin > 0 ? di.smem_optin : 232448;
  if (pl.smem > smem_max) return false;
  if (pl.S > 1) {
    // counters first, so every plan of the same shape (any MR) finds them at
    // the same place; chunk partials after them
    const size_t part = (size_t)pl.B * pl.nch * pl.rows_per_unit * MR * sizeof(float);
    pl.ws_part_off = ((size_t)pl.B * sizeof(int) + 255) & ~size_t(255);
    pl.ws_bytes = pl.ws_part_off + part;
  }
  *out = pl;
  return true;
}

template <int MR, int CS>
cudaError_t launch_one(const GemvParams& prm, const Plan& pl, bool pdl, cudaStream_t stream, int dev) {
  static std::mutex mu;
  static long long attr_bytes[64] = {};
  auto kern = gemv_kernel<MR, CS>;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  {
    // raise the kernel's dynamic shared-memory limit to what this plan needs
    std::lock_guard<std::mutex> lock(mu);
    if (pl.smem > attr_bytes[dev]) {
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)pl.smem);
      if (e != cudaSuccess) return e;
      attr_bytes[dev] = pl.smem;
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)pl.ctas);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = (size_t)pl.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, prm);
}

template <int MR>
cudaError_t launch_cs(const GemvParams& prm, const Plan& pl, bool pdl, cudaStream_t s, int dev) {
  switch (pl.cs) {
    case 5: return launch_one<MR, 5>(prm, pl, pdl, s, dev);
    case 6: return launch_one<MR, 6>(prm, pl, pdl, s, dev);
    case 7: return launch_one<MR, 7>(prm, pl, pdl, s, dev);
    case 8: return launch_one<MR, 8>(prm, pl, pdl, s, dev);
    case 9: return launch_one<MR, 9>(prm, pl, pdl, s, dev);
    case 10: return launch_one<MR, 10>(prm, pl, pdl, s, dev);
    case 11: return launch_one<MR, 11>(prm, pl, pdl, s, dev);
    case 12: return launch_one<MR, 12>(prm, pl, pdl, s, dev);
    default: return launch_one<MR, 0>(prm, pl, pdl, s, dev);
  }
}

cudaError_t launch(const GemvParams& prm, const Plan& pl, bool pdl, cudaStream_t s, int dev) {
  switch (pl.MR) {
    case 1: return launch_cs<1>(prm, pl, pdl, s, dev);
    case 2: return launch_cs<2>(prm, pl, pdl, s, dev);
    case 3: return launch_cs<3>(prm, pl, pdl, s, dev);
    case 4: return launch_cs<4>(prm, pl, pdl, s, dev);
    default: return cudaErrorInvalidConfiguration;
  }
}

GemvParams base_params(const Plan& pl, int N, int K) {
  GemvParams p = {};
  p.N = N;
  p.K = K;
  p.Kg = K / 32;
  p.MR = pl.MR;
  p.team = pl.team;
  p.sets = pl.sets;
  p.R = pl.R;
  p.rows_per_unit = pl.rows_per_unit;
  p.chunk = pl.chunk;
  p.nch = pl.nch;
  p.S = pl.S;
  p.cps = pl.cps;
  p.upi = pl.upi;
  p.B = (int)pl.B;
  p.U = (int)pl.U;
  p.x_slots = pl.x_slots;
  return p;
}

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool current_device(int* dev, DeviceInfo* di) {
  if (cudaGetDevice(dev) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  *di = device_info(*dev);
  return di->sms > 0;
}

void planning_device(DeviceInfo* di) {
  int dev = 0;
  if (!current_device(&dev, di)) {
    di->sms = 152;              // planning without a device: GB300 figures
    di->smem_optin = 232448;
  }
}

// Plans are cached per shape: planning is cheap but not free, and decode
// loops call the same few shapes over and over.
struct PlanKey {
  int MR, N, K, n_items, split, xpi, sms;
  bool operator==(const PlanKey& o) const {
    return MR == o.MR && N == o.N && K == o.K && n_items == o.n_items && split == o.split &&
           xpi == o.xpi && sms == o.sms;
  }
};

bool cached_plan(int MR, int N, int K, int n_items, int split, int xpi, const DeviceInfo& di,
                 Plan* out) {
  static std::mutex mu;
  static PlanKey keys[256];
  static Plan plans[256];
  static int used = 0, next = 0;
  const PlanKey k{MR, N, K, n_items, split, xpi, di.sms};
  {
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i)
      if (keys[i] == k) {
        *out = plans[i];
        return true;
      }
  }
  if (!make_plan(MR, N, K, n_items, split, xpi, di, out)) return false;
  std::lock_guard<std::mutex> lock(mu);
  keys[next] = k;
  plans[next] = *out;
  next = (next + 1) % 256;
  used = std::min(used + 1, 256);
  return true;
}

// Activation rows per launch: up to kMaxMR, as many as fit shared memory.
int max_rows_per_launch(int K, const DeviceInfo& di) {
  const long long smem_max = di.smem_optin > 0 ? di.smem_optin : 232448;
  int mr = kMaxMR;
  while (mr > 0 && x_bytes(1, mr, K / 32) > smem_max) --mr;
  return mr;
}

}  // namespace
}  // namespace w4

// ================================================================= C ABI
using namespace w4;

extern "C" w4_status w4a16_gemv_plan(int M, int N, int K, w4_plan_info* info) {
  if (info == nullptr || M < 1 || N < 1) return W4_ERR_ARG;
  if (M > W4_MAX_M || K < 32 || K % 32 != 0 || K > W4_MAX_K) return W4_ERR_SHAPE;
  DeviceInfo di;
  planning_device(&di);
  Plan pl;
  const int mr_cap = max_rows_per_launch(K, di);
  if (mr_cap < 1 || !cached_plan(std::min(M, mr_cap), N, K, 1, 1, 0, di, &pl)) return W4_ERR_SHAPE;
  info->path = 0;
  info->ctas = pl.ctas;
  info->slices = pl.S;
  info->threads = kThreads;
  info->team = pl.team;
  info->unit_rows = pl.rows_per_unit;
  info->chunk_groups = pl.chunk;
  info->rows_per_lane = pl.R;
  info->smem_bytes = (int)pl.smem;
  info->rows_per_call = pl.MR;
  info->chunk_steps = pl.cs;
  return W4_OK;
}

extern "C" size_t w4a16_gemv_workspace_bytes(int M, int N, int K) {
  if (M < 1 || N < 1 || M > W4_MAX_M || K < 32 || K % 32 != 0 || K > W4_MAX_K) return 0;
  DeviceInfo di;
  planning_device(&di);
  Plan pl;
  const int mr_cap = max_rows_per_launch(K, di);
  if (mr_cap < 1 || !cached_plan(std::min(M, mr_cap), N, K, 1, 1, 0, di, &pl)) return 0;
  size_t ws = pl.ws_bytes;
  for (int mr = 1; mr < std::min(M, mr_cap); ++mr) {   // smaller tail launches
    Plan pm;
    if (cached_plan(mr, N, K, 1, 1, 0, di, &pm)) ws = std::max(ws, pm.ws_bytes);
  }
  return ws;
}

extern "C" w4_status w4a16_gemv(void* y, const void* qw, const void* st, const void* x, int M,
                                int N, int K, void* workspace, size_t workspace_bytes,
                                int32_t* status_dev, unsigned flags, w4_stream_t stream) {
  if (y == nullptr || qw == nullptr || st == nullptr || x == nullptr) return W4_ERR_ARG;
  if (M < 1 || N < 1 || (flags & ~W4_FLAG_PDL) != 0) return W4_ERR_ARG;
  if (M > W4_MAX_M || K < 32 || K % 32 != 0 || K > W4_MAX_K) return W4_ERR_SHAPE;
  if (!aligned(qw, 16) || !aligned(st, 16) || !aligned(x, 16) || !aligned(y, 2))
    return W4_ERR_ALIGN;
  int dev = 0;
  DeviceInfo di;
  if (!current_device(&dev, &di)) return W4_ERR_DEVICE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int mr_cap = max_rows_per_launch(K, di);
  if (mr_cap < 1) return W4_ERR_SHAPE;
  for (int m0 = 0; m0 < M; m0 += mr_cap) {
    const int mr = std::min(mr_cap, M - m0);
    Plan pm;
    if (!cached_plan(mr, N, K, 1, 1, 0, di, &pm)) return W4_ERR_SHAPE;
    if (pm.ws_bytes > 0 && (workspace == nullptr || workspace_bytes < pm.ws_bytes))
      return W4_ERR_WORKSPACE;
    if (pm.ws_bytes > 0 && !aligned(workspace, 16)) return W4_ERR_ALIGN;
    GemvParams p = base_params(pm, N, K);
    p.qw = static_cast<const uint8_t*>(qw);
    p.st = static_cast<const uint8_t*>(st);
    p.x = static_cast<const __nv_bfloat16*>(x) + (long long)m0 * K;
    p.y = static_cast<__nv_bfloat16*>(y) + (long long)m0 * N;
    p.n_items = 1;
    p.num_experts = 1;
    p.status = status_dev;
    if (pm.ws_bytes > 0) {
      p.ws_count = static_cast<int*>(workspace);
      p.ws_partial = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + pm.ws_part_off);
    }
    const cudaError_t e = launch(p, pm, (flags & W4_FLAG_PDL) != 0, s, dev);
    if (e != cudaSuccess) {
      note_cuda_error(e);
      cudaGetLastError();
      return W4_ERR_LAUNCH;
    }
  }
  return W4_OK;
}

extern "C" w4_status w4a16_gemv_id(void* y, const void* qw_base, size_t qw_stride_bytes,
                                   const void* st_base, size_t st_stride_bytes, int num_experts,
                                   const int32_t* ids, int n_ids, const void* x, int x_rows,
                                   int N, int K, int32_t* status_dev, unsigned flags,
                                   w4_stream_t stream) {
  if (y == nullptr || qw_base == nullptr || st_base == nullptr || ids == nullptr || x == nullptr)
    return W4_ERR_ARG;
  if (n_ids < 1 || N < 1 || num_experts < 1 || (flags & ~W4_FLAG_PDL) != 0) return W4_ERR_ARG;
  if (K < 32 || K % 32 != 0 || K > W4_MAX_K) return W4_ERR_SHAPE;
  if (x_rows != 1 && x_rows != n_ids) return W4_ERR_SHAPE;
  if (qw_stride_bytes < (size_t)N * K / 2 || st_stride_bytes < (size_t)N * (K / 32) * 2)
    return W4_ERR_ARG;
  if (!aligned(qw_base, 16) || !aligned(st_base, 16) || !aligned(x, 16) || !aligned(y, 2) ||
      qw_stride_bytes % 16 != 0 || st_stride_bytes % 16 != 0)
    return W4_ERR_ALIGN;
  int dev = 0;
  DeviceInfo di;
  if (!current_device(&dev, &di)) return W4_ERR_DEVICE;
  const int xpi = (x_rows == n_ids && n_ids > 1) ? 1 : 0;
  Plan pl;
  if (!cached_plan(1, N, K, n_ids, 0, xpi, di, &pl)) return W4_ERR_SHAPE;
  GemvParams p = base_params(pl, N, K);
  p.qw = static_cast<const uint8_t*>(qw_base);
  p.st = static_cast<const uint8_t*>(st_base);
  p.qw_item_stride = qw_stride_bytes;
  p.st_item_stride = st_stride_bytes;
  p.ids = ids;
  p.num_experts = num_experts;
  p.x = static_cast<const __nv_bfloat16*>(x);
  p.x_per_item = xpi;
  p.y = static_cast<__nv_bfloat16*>(y);
  p.n_items = n_ids;
  p.status = status_dev;
  const cudaError_t e =
      launch(p, pl, (flags & W4_FLAG_PDL) != 0, reinterpret_cast<cudaStream_t>(stream), dev);
  if (e != cudaSuccess) {
    note_cuda_error(e);
    cudaGetLastError();
    return W4_ERR_LAUNCH;
  }
  return W4_OK;
}

// ================================================================= no-allocation variant
// Split-K GEMV whose scratch lives in a fixed device array compiled into the
// library, for callers that cannot allocate device memory themselves (see
// w4a16_gemv_static_scratch in w4a16.h).  Every GPU that loads the library
// holds this array until the process exits.
static __device__ __align__(256) unsigned char w4_static_scratch[W4_STATIC_SCRATCH_BYTES];

namespace w4 {
namespace {

// Device address of w4_static_scratch on device `dev` (the host-side name is
// only a stand-in).  Looked up once per device, with that device current.
cudaError_t static_scratch_address(int dev, void** out) {
  static std::mutex mu;
  static void* addr[64] = {};
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, w4_static_scratch);
    if (e != cudaSuccess) return e;
    addr[dev] = p;
  }
  *out = addr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace w4

extern "C" w4_status w4a16_gemv_static_scratch(void* y, const void* qw, const void* st,
                                               const void* x, int M, int N, int K,
                                               int32_t* status_dev, unsigned flags,
                                               w4_stream_t stream) {
  if (y == nullptr || qw == nullptr || st == nullptr || x == nullptr) return W4_ERR_ARG;
  if (M < 1 || N < 1 || (flags & ~W4_FLAG_PDL) != 0) return W4_ERR_ARG;
  if (M > W4_MAX_M || K < 32 || K % 32 != 0 || K > W4_MAX_K) return W4_ERR_SHAPE;
  if (!aligned(qw, 16) || !aligned(st, 16) || !aligned(x, 16) || !aligned(y, 2))
    return W4_ERR_ALIGN;
  int dev = 0;
  DeviceInfo di;
  if (!current_device(&dev, &di)) return W4_ERR_DEVICE;
  const int mr_cap = max_rows_per_launch(K, di);
  if (mr_cap < 1) return W4_ERR_SHAPE;
  // every launch of this call must fit the fixed array: check before any work
  for (int m0 = 0; m0 < M; m0 += mr_cap) {
    Plan pm;
    if (!cached_plan(std::min(mr_cap, M - m0), N, K, 1, 1, 0, di, &pm)) return W4_ERR_SHAPE;
    if (pm.ws_bytes > (size_t)W4_STATIC_SCRATCH_BYTES) return W4_ERR_WORKSPACE;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  for (int m0 = 0; m0 < M; m0 += mr_cap) {
    const int mr = std::min(mr_cap, M - m0);
    Plan pm;
    cached_plan(mr, N, K, 1, 1, 0, di, &pm);
    GemvParams p = base_params(pm, N, K);
    p.qw = static_cast<const uint8_t*>(qw);
    p.st = static_cast<const uint8_t*>(st);
    p.x = static_cast<const __nv_bfloat16*>(x) + (long long)m0 * K;
    p.y = static_cast<__nv_bfloat16*>(y) + (long long)m0 * N;
    p.n_items = 1;
    p.num_experts = 1;
    p.status = status_dev;
    if (pm.ws_bytes > 0) {
      void* base = nullptr;
      cudaError_t e = static_scratch_address(dev, &base);
      // the counters must start at zero; the array keeps the previous call's
      // contents (and an aborted call may leave them armed)
      if (e == cudaSuccess) e = cudaMemsetAsync(base, 0, (size_t)pm.B * sizeof(int), s);
      if (e != cudaSuccess) {
        note_cuda_error(e);
        cudaGetLastError();
        return W4_ERR_LAUNCH;
      }
      p.ws_count = static_cast<int*>(base);
      p.ws_partial = reinterpret_cast<float*>(static_cast<uint8_t*>(base) + pm.ws_part_off);
    }
    const cudaError_t e = launch(p, pm, (flags & W4_FLAG_PDL) != 0, s, dev);
    if (e != cudaSuccess) {
      note_cuda_error(e);
      cudaGetLastError();
      return W4_ERR_LAUNCH;
    }
  }
  return W4_OK;
}
