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
// Design (one persistent CTA per SM):
//  * The weight matrix is split into row blocks of `tile_rows` rows; a row
//    block is cut along K into chunks of G groups (G = K/32 when whole rows fit
//    a stage).  A (row block, K slice) pair is a unit; every CTA owns a
//    contiguous, balanced range of units.
//  * Thread 0 streams each (row block, chunk) tile from HBM into a 4-deep ring
//    of shared-memory stages with 1-D bulk copies (cp.async.bulk, TMA engine),
//    completion tracked by one mbarrier per stage.  Codes of a whole-row tile
//    are one contiguous copy.  With W4_FLAG_PDL the first copies are issued
//    before waiting on the previous kernel in the stream.
//  * The activation rows are staged once per CTA into shared memory as fp16
//    pairs scaled by a power of two per group of 32 (exact), with the group's
//    inverse scale kept beside them.
//  * `TEAM` lanes share an output row.  Per 32-code group a lane turns each
//    packed word into four fp16 pairs (c - 8) with the float-bit trick of the
//    page (fp16 form: (0x6400 | c) - 1032 = c - 8, exact), multiplies them with
//    the fp16 activation pairs in packed fp16 (products exact), sums each lane
//    of a pair over the group's 4 words in fp16, converts and adds the 8
//    partial sums into fp32, scales by step * group scale and accumulates in
//    fp32.  Error: at most 3 fp16 roundings per 4-product partial, i.e.
//    3 * 2^-11 of sum|w x|, plus fp32 accumulation.
//  * After each chunk the team reduces its lanes with a fixed xor-shuffle
//    tree; chunk sums are added in chunk order.  The arithmetic of a row thus
//    depends on K only, never on N, the row index, the slice split or the
//    addresses (bitwise-reproducible and gemv_id == gemv per row).
//  * Split-K (slices > 1): every chunk sum goes to the workspace; the CTA that
//    finishes a row block last (atomic counter, no waiting) adds the chunk
//    sums in chunk order, writes the row block and re-arms the counter.
//  * Every wait is bounded; on expiry the kernel records W4_ERR_TIMEOUT, waits
//    (bounded) for its own copies in flight and leaves.
#include <algorithm>
#include <mutex>

#include "common.cuh"

namespace w4 {

constexpr int kThreads = 512;      // 16 warps, all compute; thread 0 also issues copies
constexpr int kStages = 4;         // shared-memory ring depth
constexpr int kMaxMR = 4;          // activation rows per launch on this path
constexpr long long kWaitCycles = 4000000000LL;   // ~2 s at GB300 clocks

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
  int tile_rows, G, nch, whole;        // tiling (depends on K only)
  int S, cps, bpi;                     // partition
  long long B, U;
  int xg_max;                          // groups of staged activations
  int stage_codes, stage_steps, seg_stride, stage_bytes;
  int* ws_count;                       // [B] at the start of the workspace
  float* ws_partial;                   // [B][nch][tile_rows][MR] after it
  int32_t* status;
};

// ---------------------------------------------------------------- tile walk
struct Walk {
  long long u, u_end;
  int c, c_end;
  int slice, item, row0, rows;
  long long rb;
  const uint8_t* qw_item;
  const uint8_t* st_item;

  __device__ void load(const GemvParams& p) {
    while (u < u_end) {
      slice = (int)(u / p.B);
      rb = u - (long long)slice * p.B;
      item = (int)(rb / p.bpi);
      const int rbi = (int)(rb - (long long)item * p.bpi);
      row0 = rbi * p.tile_rows;
      rows = min(p.tile_rows, p.N - row0);
      c = slice * p.cps;
      c_end = min(c + p.cps, p.nch);
      long long blk = item;
      if (p.ids != nullptr) {
        const int e = __ldg(p.ids + item);
        if (e < 0 || e >= p.num_experts) {   // id out of range: skip the unit
          report(p.status, W4_ERR_INDEX);
          ++u;
          continue;
        }
        blk = e;
      }
      qw_item = p.qw + (unsigned long long)blk * p.qw_item_stride;
      st_item = p.st + (unsigned long long)blk * p.st_item_stride;
      return;
    }
  }
  __device__ void init(const GemvParams& p, long long ub, long long ue) {
    u = ub;
    u_end = ue;
    load(p);
  }
  __device__ bool done() const { return u >= u_end; }
  __device__ void next(const GemvParams& p) {
    if (++c >= c_end) {
      ++u;
      load(p);
    }
  }
  __device__ int g0(const GemvParams& p) const { return c * p.G; }
  __device__ int glen(const GemvParams& p) const { return min(p.G, p.Kg - c * p.G); }
};

// Copy bytes [b, e) of a step array of `total` bytes to shared memory at
// `dst` (16-byte aligned), as the 16-byte-aligned superset [b & ~15, ...)
// clipped to the array; bytes past the last full 16-byte line of the array
// are loaded one by one.  Returns the number of bulk-copied bytes.
__device__ __forceinline__ uint32_t copy_steps(uint8_t* dst, const uint8_t* src, long long b,
                                               long long e, long long total, uint32_t bar,
                                               uint64_t pol, bool issue) {
  const long long lo = b & ~15LL;
  const long long lim = total & ~15LL;
  const long long hi = min((e + 15) & ~15LL, lim);
  uint32_t bytes = 0;
  if (hi > lo) {
    bytes = (uint32_t)(hi - lo);
    if (issue) bulk_g2s_evict_first(smem_addr(dst), src + lo, bytes, bar, pol);
  }
  if (!issue) {
    for (long long i = max(lo, lim); i < e; ++i) dst[i - lo] = src[i];
  }
  return bytes;
}

// Thread 0: start loading tile `w` into stage `slot`.
__device__ void issue_tile(const GemvParams& p, const Walk& w, uint8_t* stage, uint32_t bar,
                           uint64_t pol) {
  uint8_t* codes = stage;
  uint8_t* steps = stage + p.stage_codes;
  const long long row_bytes = (long long)p.K / 2;
  const long long st_total = (long long)p.N * p.Kg * 2;
  const int g0 = w.g0(p), gl = w.glen(p);
  uint32_t tx = 0;
  // scalar step tails first (generic stores), then one arrive with the byte
  // count, then the bulk copies
  for (int pass = 0; pass < 2; ++pass) {
    const bool issue = pass == 1;
    if (issue) {
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(bar, tx);
      const uint8_t* src = w.qw_item + (long long)w.row0 * row_bytes + (long long)g0 * 16;
      if (p.whole) {
        bulk_g2s_evict_first(smem_addr(codes), src, (uint32_t)(w.rows * row_bytes), bar, pol);
      } else {
        for (int r = 0; r < w.rows; ++r)
          bulk_g2s_evict_first(smem_addr(codes + r * p.G * 16), src + r * row_bytes,
                               (uint32_t)gl * 16, bar, pol);
      }
    }
    if (p.whole) {
      const long long b = (long long)w.row0 * p.Kg * 2;
      const uint32_t n = copy_steps(steps, w.st_item, b, b + (long long)w.rows * p.Kg * 2,
                                    st_total, bar, pol, issue);
      if (!issue) tx = (uint32_t)(w.rows * row_bytes) + n;
    } else {
      if (!issue) tx = 0;
      for (int r = 0; r < w.rows; ++r) {
        const long long b = ((long long)(w.row0 + r) * p.Kg + g0) * 2;
        const uint32_t n = copy_steps(steps + r * p.seg_stride, w.st_item, b, b + gl * 2,
                                      st_total, bar, pol, issue);
        if (!issue) tx += (uint32_t)gl * 16 + n;
      }
    }
  }
}

// ---------------------------------------------------------------- activations
// Stage activation rows as fp16 pairs, scaled by 2^e per group of 32 so that
// the group's largest magnitude lies in [2^9, 2^10).  Layout per row m:
// 16-byte chunk (w, g) = pairs (x[8w+p], x[8w+p+4]) for p = 0..3 of group g,
// stored at ((m * 4 + w) * xg_max + g) * 16; the inverse scale 2^-e of the
// group at xscale[m * xg_max + g].
__device__ void stage_x(const GemvParams& p, int xrow0, int gbeg, int gend, uint8_t* xs,
                        float* xscale) {
  const int ng = gend - gbeg;
  for (int idx = threadIdx.x; idx < p.MR * ng; idx += blockDim.x) {
    const int m = idx / ng;
    const int gi = idx - m * ng;
    const uint4* src = reinterpret_cast<const uint4*>(p.x + (long long)(xrow0 + m) * p.K +
                                                      (long long)(gbeg + gi) * 32);
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
      // elements 8w .. 8w+7 are bf16 halves of words wv[4w .. 4w+3]
      float f[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t pair = wv[4 * w + i];
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
      *reinterpret_cast<uint4*>(xs + ((long long)(m * 4 + w) * p.xg_max + gi) * 16) = out;
    }
    xscale[m * p.xg_max + gi] = inv;
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

template <int MR>
__device__ __forceinline__ void group_dot(uint4 q, const uint8_t* xg, int wstride, int mstride,
                                          float stf, const float* sc, int sc_mstride,
                                          float acc[MR]) {
  __half2 h[4][4];
  unpack_word(q.x, h[0]);
  unpack_word(q.y, h[1]);
  unpack_word(q.z, h[2]);
  unpack_word(q.w, h[3]);
#pragma unroll
  for (int m = 0; m < MR; ++m) {
    __half2 a0 = u2h(0u), a1 = u2h(0u), a2 = u2h(0u), a3 = u2h(0u);
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const uint4 xv = *reinterpret_cast<const uint4*>(xg + m * mstride + w * wstride);
      a0 = __hfma2(h[w][0], u2h(xv.x), a0);
      a1 = __hfma2(h[w][1], u2h(xv.y), a1);
      a2 = __hfma2(h[w][2], u2h(xv.z), a2);
      a3 = __hfma2(h[w][3], u2h(xv.w), a3);
    }
    float gs = add_pair_f32(0.0f, a0);
    gs = add_pair_f32(gs, a1);
    gs = add_pair_f32(gs, a2);
    gs = add_pair_f32(gs, a3);
    // gs * 2^-e is exact (power-of-two rescale), so the step multiply is the
    // only rounding before the fp32 accumulate
    acc[m] = fmaf(gs * sc[m * sc_mstride], stf, acc[m]);
  }
}

// ---------------------------------------------------------------- kernel
template <int TEAM, int MR>
__global__ void __launch_bounds__(kThreads, 1) gemv_kernel(const __grid_constant__ GemvParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* xs = smem;
  float* xscale = reinterpret_cast<float*>(xs + (long long)MR * 4 * p.xg_max * 16);
  uint8_t* stages =
      smem + (((long long)MR * 4 * p.xg_max * 16 + (long long)MR * p.xg_max * 4 + 127) & ~127LL);
  uint64_t* bars = reinterpret_cast<uint64_t*>(stages + (long long)kStages * p.stage_bytes);
  __shared__ int s_last;

  const int tid = threadIdx.x;
  const long long ub = (long long)blockIdx.x * p.U / gridDim.x;
  const long long ue = (long long)(blockIdx.x + 1) * p.U / gridDim.x;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(smem_addr(&bars[s]), 1);
    mbar_init_fence();
  }
  __syncthreads();

  // The ids (routed experts) may be written by the previous kernel: read them
  // only after it has completed.  Dense weights do not depend on earlier
  // kernels, so their first tiles are requested before the wait.
  if (p.ids != nullptr) pdl_wait();
  Walk it;
  it.init(p, ub, ue);
  Walk iss = it;          // thread 0's issue cursor, kStages tiles ahead
  long long issued = 0;
  uint64_t pol = 0;
  if (tid == 0) {
    pol = policy_evict_first();
    for (; issued < kStages && !iss.done(); ++issued, iss.next(p))
      issue_tile(p, iss, stages + issued * p.stage_bytes, smem_addr(&bars[issued]), pol);
  }
  if (p.ids == nullptr) pdl_wait();
  // Let the next kernel in the stream (if launched with PDL) get scheduled as
  // SMs free up: it can only start once every CTA of this grid has reached
  // this point, and it waits for this grid's completion before reading our
  // outputs.
  pdl_launch_dependents();

  const int team = tid / TEAM;   // row of the tile this lane works on
  const int lane_t = tid % TEAM;
  const int wstride = p.xg_max * 16;
  const int mstride = 4 * p.xg_max * 16;

  int cur_xrow = -1, cur_slice = -1, xg_base = 0;
  float row_acc[MR];
#pragma unroll
  for (int m = 0; m < MR; ++m) row_acc[m] = 0.0f;

  long long t = 0;
  bool timed_out = false;
  while (!it.done()) {
    const int xrow = p.x_per_item ? it.item * p.MR : 0;
    if (xrow != cur_xrow || it.slice != cur_slice) {
      xg_base = (p.S == 1) ? 0 : it.slice * p.cps * p.G;
      const int xg_end = (p.S == 1) ? p.Kg : min(p.Kg, (it.slice + 1) * p.cps * p.G);
      stage_x(p, xrow, xg_base, xg_end, xs, xscale);
      __syncthreads();
      cur_xrow = xrow;
      cur_slice = it.slice;
    }
    const int slot = (int)(t % kStages);
    const uint32_t parity = (uint32_t)((t / kStages) & 1);
    const bool ok = mbar_wait_bounded(smem_addr(&bars[slot]), parity, kWaitCycles);

    const uint8_t* stage = stages + (long long)slot * p.stage_bytes;
    const int g0 = it.g0(p);
    const int gl = it.glen(p);
    const bool first_chunk = it.c == it.slice * p.cps;
    const bool last_chunk = it.c + 1 == it.c_end;
    if (first_chunk) {
#pragma unroll
      for (int m = 0; m < MR; ++m) row_acc[m] = 0.0f;
    }
    float cs[MR];
#pragma unroll
    for (int m = 0; m < MR; ++m) cs[m] = 0.0f;
    if (ok && team < it.rows) {
      const uint8_t* codes = stage + (long long)team * p.G * 16;
      long long st_first;
      const uint8_t* steps;
      if (p.whole) {
        st_first = (long long)it.row0 * p.Kg * 2;
        steps = stage + p.stage_codes + (st_first & 15) + (long long)team * p.Kg * 2;
      } else {
        st_first = ((long long)(it.row0 + team) * p.Kg + g0) * 2;
        steps = stage + p.stage_codes + (long long)team * p.seg_stride + (st_first & 15);
      }
      const uint8_t* xg = xs + (long long)(g0 - xg_base) * 16;
      const float* sc = xscale + (g0 - xg_base);
#pragma unroll 2
      for (int g = lane_t; g < gl; g += TEAM) {
        const uint4 q = *reinterpret_cast<const uint4*>(codes + g * 16);
        const uint32_t sb = *reinterpret_cast<const uint16_t*>(steps + g * 2);
        group_dot<MR>(q, xg + g * 16, wstride, mstride, bf16_bits_to_float(sb), sc + g,
                      p.xg_max, cs);
      }
    }
    // team reduction, fixed xor tree
#pragma unroll
    for (int m = 0; m < MR; ++m) {
#pragma unroll
      for (int off = TEAM / 2; off > 0; off >>= 1) cs[m] += __shfl_xor_sync(0xffffffffu, cs[m], off);
    }
    const bool writer = ok && lane_t == 0 && team < it.rows;
    if (p.S == 1) {
#pragma unroll
      for (int m = 0; m < MR; ++m) row_acc[m] += cs[m];
      if (last_chunk && writer) {
#pragma unroll
        for (int m = 0; m < MR; ++m)
          p.y[((long long)it.item * p.MR + m) * p.N + it.row0 + team] =
              __float2bfloat16_rn(row_acc[m]);
      }
    } else if (writer) {
      float* dst = p.ws_partial + ((it.rb * p.nch + it.c) * p.tile_rows + team) * p.MR;
#pragma unroll
      for (int m = 0; m < MR; ++m) dst[m] = cs[m];
      __threadfence();
    }
    timed_out = __syncthreads_or(!ok) != 0;
    if (timed_out) break;

    if (p.S > 1 && last_chunk) {
      if (tid == 0) {
        const int old = atomicAdd(p.ws_count + it.rb, 1);
        s_last = (old == p.S - 1);
      }
      __syncthreads();
      if (s_last) {
        __threadfence();
        const float* src = p.ws_partial + it.rb * p.nch * p.tile_rows * p.MR;
        for (int i = tid; i < it.rows * p.MR; i += kThreads) {
          const int r = i / p.MR, m = i - r * p.MR;
          float v = 0.0f;
          for (int c = 0; c < p.nch; ++c) v += __ldcg(src + ((long long)c * p.tile_rows + r) * p.MR + m);
          p.y[((long long)it.item * p.MR + m) * p.N + it.row0 + r] = __float2bfloat16_rn(v);
        }
        if (tid == 0) atomicExch(p.ws_count + it.rb, 0);
      }
    }

    if (tid == 0 && !iss.done()) {
      issue_tile(p, iss, stages + (long long)slot * p.stage_bytes, smem_addr(&bars[slot]), pol);
      ++issued;
      iss.next(p);
    }
    it.next(p);
    ++t;
  }
  if (timed_out) {
    report(p.status, W4_ERR_TIMEOUT);
    if (tid == 0) {   // let this CTA's copies in flight land before leaving
      for (long long k = t; k < issued; ++k)
        mbar_wait_bounded(smem_addr(&bars[k % kStages]), (uint32_t)((k / kStages) & 1),
                          kWaitCycles);
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

struct Tiling {
  int team = 32;
  int tile_rows = 16;
  int G = 0;
  int nch = 1;
  int whole = 1;
  int stage_codes = 0, stage_steps = 0, seg_stride = 0, stage_bytes = 0;
};

inline long long align16(long long v) { return (v + 15) & ~15LL; }

Tiling make_tiling(int K) {
  const int Kg = K / 32;
  Tiling best;
  double best_score = -1.0;
  const int teams[3] = {32, 16, 8};
  for (int ti = 0; ti < 3; ++ti) {
    const int team = teams[ti];
    const int rows = kThreads / team;
    for (int u = 1; u <= 64; ++u) {
      int G = team * u;
      const bool whole = G >= Kg;
      if (whole) G = Kg;
      const int nch = whole ? 1 : (Kg + G - 1) / G;
      const int glast = Kg - (nch - 1) * G;
      const long long slots = (long long)team * ((long long)(nch - 1) * ((G + team - 1) / team) +
                                                 (glast + team - 1) / team);
      const double util = (double)Kg / (double)slots;
      Tiling t;
      t.team = team;
      t.tile_rows = rows;
      t.G = G;
      t.nch = nch;
      t.whole = whole ? 1 : 0;
      t.stage_codes = rows * G * 16;
      t.seg_stride = (int)(whole ? align16((long long)rows * Kg * 2 + 32) : align16(G * 2 + 32));
      t.stage_steps = whole ? t.seg_stride : rows * t.seg_stride;
      t.stage_bytes = t.stage_codes + t.stage_steps;
      const double kb = t.stage_bytes / 1024.0;
      const bool fits = kb <= 40.0;
      if (fits) {
        // utilisation first; then stages of 16-32 KB; then whole rows
        double score = util * 100.0;
        score -= (kb < 16.0) ? (16.0 - kb) * 0.15 : 0.0;
        score -= (kb > 32.0) ? (kb - 32.0) * 0.15 : 0.0;
        score += whole ? 0.5 : 0.0;
        score -= (double)(whole ? 0 : rows) * 0.01;   // one bulk copy per row segment
        if (score > best_score) {
          best_score = score;
          best = t;
        }
      }
      if (whole) break;
    }
  }
  if (best_score < 0) {   // no stage under the cap: smallest chunks of one warp per row
    Tiling t;
    t.team = 32;
    t.tile_rows = kThreads / 32;
    t.G = 32;
    t.nch = (Kg + 31) / 32;
    t.whole = (t.nch == 1) ? 1 : 0;
    if (t.whole) t.G = Kg;
    t.stage_codes = t.tile_rows * t.G * 16;
    t.seg_stride = (int)(t.whole ? align16((long long)t.tile_rows * Kg * 2 + 32) : align16(t.G * 2 + 32));
    t.stage_steps = t.whole ? t.seg_stride : t.tile_rows * t.seg_stride;
    t.stage_bytes = t.stage_codes + t.stage_steps;
    best = t;
  }
  return best;
}

struct Plan {
  Tiling t;
  int MR = 1;
  int S = 1, cps = 1, bpi = 1;
  long long B = 0, U = 0;
  int xg_max = 0;
  int ctas = 0;
  long long smem = 0;
  size_t ws_bytes = 0;
  size_t ws_part_off = 0;
};

long long smem_for(const Tiling& t, int MR, int xg_max) {
  long long x = (long long)MR * 4 * xg_max * 16 + (long long)MR * xg_max * 4;
  x = (x + 127) & ~127LL;
  return x + (long long)kStages * t.stage_bytes + kStages * 8;
}

// Plan for `rows_items` items of N rows, MR activation rows per item.
bool make_plan(int MR, int N, int K, int n_items, int allow_split, const DeviceInfo& di, Plan* out) {
  Plan pl;
  pl.t = make_tiling(K);
  pl.MR = MR;
  const int Kg = K / 32;
  pl.bpi = (N + pl.t.tile_rows - 1) / pl.t.tile_rows;
  pl.B = (long long)n_items * pl.bpi;
  const int sms = di.sms > 0 ? di.sms : 1;
  int S = 1;
  if (allow_split && pl.t.nch > 1 && pl.B < 8LL * sms)
    S = (int)std::min<long long>(pl.t.nch, (8LL * sms + pl.B - 1) / pl.B);
  while (true) {
    const int cps = (pl.t.nch + S - 1) / S;
    S = (pl.t.nch + cps - 1) / cps;
    const int xg = (S == 1) ? Kg : std::min(Kg, cps * pl.t.G);
    const long long sm = smem_for(pl.t, MR, xg);
    if (sm <= di.smem_optin || di.smem_optin == 0) {
      pl.S = S;
      pl.cps = cps;
      pl.xg_max = xg;
      pl.smem = sm;
      break;
    }
    if (!allow_split || S >= pl.t.nch) return false;
    ++S;
  }
  pl.U = (long long)pl.S * pl.B;
  pl.ctas = (int)std::min<long long>(pl.U, sms);
  if (pl.S > 1) {
    // counters first, so every plan of the same shape (any MR) finds them at
    // the same place; chunk partials after them
    const size_t part = (size_t)pl.B * pl.t.nch * pl.t.tile_rows * MR * sizeof(float);
    pl.ws_part_off = ((size_t)pl.B * sizeof(int) + 255) & ~size_t(255);
    pl.ws_bytes = pl.ws_part_off + part;
  }
  *out = pl;
  return true;
}

template <int TEAM, int MR>
cudaError_t launch_one(const GemvParams& prm, const Plan& pl, bool pdl, cudaStream_t stream, int dev) {
  static std::mutex mu;
  static long long attr_bytes[64] = {};
  auto kern = gemv_kernel<TEAM, MR>;
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

template <int TEAM>
cudaError_t launch_team(const GemvParams& prm, const Plan& pl, bool pdl, cudaStream_t s, int dev) {
  switch (pl.MR) {
    case 1: return launch_one<TEAM, 1>(prm, pl, pdl, s, dev);
    case 2: return launch_one<TEAM, 2>(prm, pl, pdl, s, dev);
    case 3: return launch_one<TEAM, 3>(prm, pl, pdl, s, dev);
    default: return launch_one<TEAM, 4>(prm, pl, pdl, s, dev);
  }
}

cudaError_t launch(const GemvParams& prm, const Plan& pl, bool pdl, cudaStream_t s, int dev) {
  switch (pl.t.team) {
    case 8: return launch_team<8>(prm, pl, pdl, s, dev);
    case 16: return launch_team<16>(prm, pl, pdl, s, dev);
    default: return launch_team<32>(prm, pl, pdl, s, dev);
  }
}

GemvParams base_params(const Plan& pl, int N, int K) {
  GemvParams p = {};
  p.N = N;
  p.K = K;
  p.Kg = K / 32;
  p.MR = pl.MR;
  p.tile_rows = pl.t.tile_rows;
  p.G = pl.t.G;
  p.nch = pl.t.nch;
  p.whole = pl.t.whole;
  p.S = pl.S;
  p.cps = pl.cps;
  p.bpi = pl.bpi;
  p.B = pl.B;
  p.U = pl.U;
  p.xg_max = pl.xg_max;
  p.stage_codes = pl.t.stage_codes;
  p.stage_steps = pl.t.stage_steps;
  p.seg_stride = pl.t.seg_stride;
  p.stage_bytes = pl.t.stage_bytes;
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

}  // namespace
}  // namespace w4

// ================================================================= C ABI
using namespace w4;

extern "C" w4_status w4a16_gemv_plan(int M, int N, int K, w4_plan_info* info) {
  if (info == nullptr || M < 1 || N < 1) return W4_ERR_ARG;
  if (M > W4_MAX_M || K < 32 || K % 32 != 0 || K > W4_MAX_K) return W4_ERR_SHAPE;
  int dev = 0;
  DeviceInfo di;
  if (!current_device(&dev, &di)) {
    di.sms = 152;              // planning without a device: GB300 figures
    di.smem_optin = 232448;
  }
  Plan pl;
  if (!make_plan(std::min(M, kMaxMR), N, K, 1, 1, di, &pl)) return W4_ERR_SHAPE;
  info->path = 0;
  info->ctas = pl.ctas;
  info->slices = pl.S;
  info->threads = kThreads;
  info->team = pl.t.team;
  info->tile_rows = pl.t.tile_rows;
  info->tile_groups = pl.t.G;
  info->stages = kStages;
  info->smem_bytes = (int)pl.smem;
  info->rows_per_call = pl.MR;
  return W4_OK;
}

extern "C" size_t w4a16_gemv_workspace_bytes(int M, int N, int K) {
  if (M < 1 || N < 1 || M > W4_MAX_M || K < 32 || K % 32 != 0 || K > W4_MAX_K) return 0;
  int dev = 0;
  DeviceInfo di;
  if (!current_device(&dev, &di)) {
    di.sms = 152;
    di.smem_optin = 232448;
  }
  Plan pl;
  if (!make_plan(std::min(M, kMaxMR), N, K, 1, 1, di, &pl)) return 0;
  return pl.ws_bytes;
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
  Plan pl;
  if (!make_plan(std::min(M, kMaxMR), N, K, 1, 1, di, &pl)) return W4_ERR_SHAPE;
  if (pl.ws_bytes > 0 && (workspace == nullptr || workspace_bytes < pl.ws_bytes))
    return W4_ERR_WORKSPACE;
  if (pl.ws_bytes > 0 && !aligned(workspace, 16)) return W4_ERR_ALIGN;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  for (int m0 = 0; m0 < M; m0 += kMaxMR) {
    const int mr = std::min(kMaxMR, M - m0);
    Plan pm = pl;
    if (mr != pl.MR && !make_plan(mr, N, K, 1, 1, di, &pm)) return W4_ERR_SHAPE;
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
  Plan pl;
  if (!make_plan(1, N, K, n_ids, 0, di, &pl)) return W4_ERR_SHAPE;
  GemvParams p = base_params(pl, N, K);
  p.qw = static_cast<const uint8_t*>(qw_base);
  p.st = static_cast<const uint8_t*>(st_base);
  p.qw_item_stride = qw_stride_bytes;
  p.st_item_stride = st_stride_bytes;
  p.ids = ids;
  p.num_experts = num_experts;
  p.x = static_cast<const __nv_bfloat16*>(x);
  p.x_per_item = (x_rows == n_ids && n_ids > 1) ? 1 : 0;
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
