// W4A16 group-32 GEMM for small batches on the 5th-generation tensor cores
// (tcgen05, sm_103a).
//
// Page "Gemma 4 on a 4 GB GPU in Plain PyTorch", section "Step 3 — Multiply
// Straight From the Packed Weights": the weights are multiplied straight from
// the packed 4-bit words.  With several activation rows (M up to 32) the
// product is a real dense contraction, and the tensor cores take the dot
// products while the CUDA cores only unpack codes:
//
//  * A CTA owns tiles of 128 weight rows (the MMA's M).  A copy warp streams
//    each (tile, 256-code K slice) stage into a shared-memory ring: the codes
//    as one 2-D TMA box with 128-byte swizzle (16 KB), the steps as one 2-D
//    box (2 KB), and the M activation rows of the slice as one 3-D box that
//    lands directly in the B-operand layout (bf16, K-major 8x8 core
//    matrices, 16-byte rows, K blocks M rows apart).
//  * Four warps (thread = weight row) turn each packed word into four bf16
//    pairs (c - 8) of consecutive codes with the page's float-bit trick in
//    bf16 form ((0x4300 | c) - 136 = c - 8, exact) and store them into
//    tensor memory with tcgen05.st: tensor memory holds the A operand.
//  * Per group of 32 codes one thread issues two tcgen05.mma (K = 16 each,
//    N = 16 or 32 activation columns, fp32 accumulate) into a fresh group
//    accumulator in tensor memory; the four warps read it back (tcgen05.ld)
//    and add step * dot to the row's running sum in fp32.  Products of bf16
//    (c - 8) and bf16 activations are exact; only fp32 additions round.
//  * Association: per row and activation row, groups are added in order
//    within each 256-code slice and the slice sums in slice order, starting
//    from 0.  Split-K (K slices over CTAs, for few row tiles) writes slice
//    sums to the workspace and the last CTA of a tile adds them in the same
//    order, so the result does not depend on N or on the split.
//  * Every wait is bounded; on expiry W4_ERR_TIMEOUT is recorded, the warps
//    leave their loops, in-flight copies and MMAs are waited for (bounded)
//    and the tensor memory is released before exit.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "gemv_tc.h"
#include "tc_common.cuh"

namespace w4 {
namespace tc {

constexpr int kRows = 128;          // weight rows per tile = MMA M
constexpr int kSliceK = 256;        // codes per row per stage
constexpr int kSliceGroups = 8;     // 32-code groups per stage
constexpr int kUnpackWarps = 4;     // one weight row per thread
constexpr int kFoldWarps = 4;       // one weight row per thread
constexpr int kCopyWarp = kUnpackWarps + kFoldWarps;
constexpr int kMmaWarp = kCopyWarp + 1;
constexpr int kThreads = 32 * (kMmaWarp + 1);
constexpr int kMaxStages = 8;
// Rounds of A and D held in tensor memory: 2 with two CTAs per SM (each
// half of the tensor memory), or 4 with one CTA per SM (all of it) for calls
// whose row tiles do not fill the SMs, where the rounds' hand-off latency,
// not the warps' issue, sets the pace.
constexpr int kMaxBufs = 4;
// shared-memory header: full[kMaxStages], empty[kMaxStages], then aready,
// afree, dready, dfree [kMaxBufs] each, then the flags and the tensor-memory base
constexpr int kFullOff = 0, kEmptyOff = 8 * kMaxStages;
constexpr int kAreadyOff = 16 * kMaxStages, kAfreeOff = kAreadyOff + 8 * kMaxBufs;
constexpr int kDreadyOff = kAfreeOff + 8 * kMaxBufs, kDfreeOff = kDreadyOff + 8 * kMaxBufs;
constexpr int kFlagOff = kDfreeOff + 8 * kMaxBufs;
constexpr int kBarBytes = kFlagOff + 16;
constexpr int kCodesBytes = kRows * 128;   // 16 KB, 1024-byte aligned (128-byte swizzle)
constexpr int kStepsBytes = kRows * 16;    // 2 KB

struct TcParams {
  CUtensorMap tm_codes;   // codes viewed as uint8 [N][K/2], box 128 x 128, 128-byte swizzle
  CUtensorMap tm_steps;   // steps viewed as uint16 [N][K/32], box 8 x 128
  CUtensorMap tm_x;       // activations viewed as uint16 [K/8][M][8], box 8 x NP x 32
  const __nv_bfloat16* x; // [M][K]
  __nv_bfloat16* y;       // [M][N]
  int M, N, K, slices;    // slices = K / 256
  int tiles, S, sps;      // row tiles, K splits, slices per split
  int units;              // tiles * S
  int nst, stage_bytes, off_b;
  int xrows;              // activation rows loaded per K block (M)
  float* ws_partial;      // [slices][M][N] under split-K
  int* ws_count;          // [tiles]
  int32_t* status;
  L2Ranges l2;            // brought into L2 after the launch's own tiles
  // Balanced runs (S == 1): the tiles x slices work items cut into equal
  // runs per CTA; a tile cut between CTAs c and c + 1 hands its rows' sum
  // over its first slices (exactly the prefix of the unsplit sum) from c to
  // c + 1 through prefix slot c.
  int sk;
  int* sk_flag;           // [ctas] 1 while prefix slot c holds a prefix
  float* sk_prefix;       // [ctas][M][128]
};

// The work of one CTA as a list of segments: (tile, slices [b, e), kind).
constexpr int kSegWhole = 0;   // a whole tile (or all of it a split covers, S == 1): write y
constexpr int kSegSplit = 1;   // a K split of a tile (S > 1): slice partials, last CTA adds
constexpr int kSegHead = 2;    // a tile's first slices: publish the prefix for the next CTA
constexpr int kSegTail = 3;    // a tile's last slices: continue from the published prefix
struct Seg {
  int t, b, e, kind;
};
struct Segs {
  int n;                  // segments of this CTA
  int u0;                 // first unit (K-split plans)
  int head_t, head_e;     // balanced runs: head tile (-1: none) and its end slice
  int wb;                 // first whole tile
  int nw;                 // whole tiles
  int tail_t, tail_b;     // tail tile (-1: none) and its first slice
};
// Balanced runs: the CTA's items [w0, w1) of tile-major (tile, slice) items.
// Its last tile, if cut, is processed FIRST (its prefix is published early,
// so that the next CTA never waits long), then the whole tiles, then its
// first tile's last slices (behind the previous CTA's prefix).  Each run
// holds at least one tile's worth of items, so a tile is cut at most once.
template <bool SK>
__device__ __forceinline__ Segs segs_of(const TcParams& p) {
  Segs g{};
  g.head_t = g.tail_t = -1;
  if constexpr (SK) {
    const long long W = (long long)p.tiles * p.slices;
    const int w0 = (int)((long long)blockIdx.x * W / gridDim.x);
    const int w1 = (int)((long long)(blockIdx.x + 1) * W / gridDim.x);
    const int tf = w0 / p.slices, k0 = w0 - tf * p.slices;
    const int tl = (w1 - 1) / p.slices, j1 = w1 - tl * p.slices;   // slices [0, j1) of tl
    if (j1 < p.slices) {
      g.head_t = tl;
      g.head_e = j1;
    }
    if (k0 > 0) {
      g.tail_t = tf;
      g.tail_b = k0;
    }
    g.wb = k0 > 0 ? tf + 1 : tf;
    g.nw = max(0, (j1 < p.slices ? tl : tl + 1) - g.wb);
    g.n = (g.head_t >= 0) + g.nw + (g.tail_t >= 0);
  } else {
    g.u0 = (int)((long long)blockIdx.x * p.units / gridDim.x);
    g.n = (int)((long long)(blockIdx.x + 1) * p.units / gridDim.x) - g.u0;
  }
  return g;
}
template <bool SK>
__device__ __forceinline__ Seg seg_at(const TcParams& p, const Segs& g, int i) {
  if constexpr (SK) {
    if (g.head_t >= 0) {
      if (i == 0) return Seg{g.head_t, 0, g.head_e, kSegHead};
      --i;
    }
    if (i < g.nw) return Seg{g.wb + i, 0, p.slices, kSegWhole};
    return Seg{g.tail_t, g.tail_b, p.slices, kSegTail};
  } else {
  const int u = g.u0 + i;
  const int s = u / p.tiles, t = u - s * p.tiles;
  const int b = s * p.sps;
  return Seg{t, b, min(b + p.sps, p.slices), p.S == 1 ? kSegWhole : kSegSplit};
  }
}

// Balanced runs' hand-over flag: a release store, and a bounded acquire
// wait (false after about a second, or once the CTA has aborted).
__device__ __forceinline__ void store_release_gpu(int* f, int v) {
  asm volatile("st.release.gpu.global.s32 [%0], %1;" ::"l"(f), "r"(v) : "memory");
}
__device__ __forceinline__ bool wait_flag_gpu(const int* f, volatile int* abort_flag) {
  const long long t0 = clock64();
  while (true) {
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
    if (v != 0) return true;
    if (*abort_flag != 0) return false;
    if (clock64() - t0 > kWaitCycles) return false;
    __nanosleep(64);
  }
}

// Row `tid`'s prefix from slot blockIdx.x - 1 (the previous CTA's part of
// this tile), its M values read once and cleared: the workspace is left
// zero-filled, as every completed call leaves it.
template <int MC>
__device__ __forceinline__ void take_prefix(const TcParams& p, int tid, float* v) {
  float* slot = p.sk_prefix + (long long)(blockIdx.x - 1) * p.M * kRows + tid;
#pragma unroll
  for (int m = 0; m < MC; ++m) {
    if (m < p.M) {
      v[m] = __ldcg(slot + (long long)m * kRows);
      slot[(long long)m * kRows] = 0.0f;
    }
  }
}

// MMA width (activation columns, 16 or 32) and groups per round for MC
// columns of results.
__host__ __device__ constexpr int np_of(int mc) { return mc <= 16 ? 16 : 32; }
__host__ __device__ constexpr int g_of(int mc) { return np_of(mc) == 16 ? 4 : 2; }
// Columns of tensor memory the kernel allocates (A and D of `bufs` rounds,
// and the running sums at 32 columns).
__host__ __device__ constexpr int tmem_cols(int np, int g, int bufs) {
  return bufs * g * (16 + np) + (np >= 32 ? 32 : 0) <= 128   ? 128
         : bufs * g * (16 + np) + (np >= 32 ? 32 : 0) <= 256 ? 256
                                                              : 512;
}

// MC: result columns read back (a power of two >= M, <= 32).
// Warps 0-3 unpack codes into A, warps 4-7 read results back and fold them,
// warp 8 copies, warp 9 issues MMAs.  Per round (G groups) the four roles
// hand off through mbarriers: aready (A stored), dready / afree (MMAs done:
// D ready, A free again), dfree (D read back).
// SK: balanced runs (p.sk); compiled only where the planner takes them
// (two CTAs per SM), so the other kernels carry none of their code.
template <int MC, int kBufs, bool SK>
__global__ void __launch_bounds__(kThreads, kBufs >= 4 ? 1 : 2)
    tc_kernel(const __grid_constant__ TcParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  constexpr int NP = np_of(MC), G = g_of(MC);
  constexpr int kCols = tmem_cols(NP, G, kBufs);
  constexpr int kACol = 0;                 // A buffers: [kBufs][G][16 columns]
  constexpr int kDCol = kBufs * G * 16;    // D buffers: [kBufs][G][NP columns]
  constexpr int kRounds = kSliceGroups / G;
  constexpr int kLdBatch = MC >= 16 ? 1 : (16 / MC < G ? 16 / MC : G);   // groups per read-back
  // 32 columns: the row's running sum over slices lives in tensor memory
  // (columns past A and D), which keeps the folding threads' registers for
  // two CTAs per SM
  constexpr bool kTmemSum = MC >= 32;
  constexpr int kSumCol = kDCol + kBufs * G * NP;
  static_assert(!kTmemSum || kSumCol + MC <= kCols, "tensor memory");
  // bytes between K-adjacent core matrices of B: the M loaded rows.  Rows
  // past M that the MMA's N reads belong to the next K block (or to the
  // stage's spare bytes); they only reach result columns past M, which are
  // never read.
  const uint32_t lbo = (uint32_t)p.xrows * 16;
  // instruction descriptor: D fp32, A and B bf16, both K-major, N = NP, M = 128
  constexpr uint32_t kIdesc =
      (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(NP >> 3) << 17) | ((uint32_t)(kRows >> 4) << 24);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t base = smem_addr(smem_raw);
  const uint32_t full0 = base + kFullOff, empty0 = base + kEmptyOff;
  const uint32_t aready0 = base + kAreadyOff, afree0 = base + kAfreeOff;
  const uint32_t dready0 = base + kDreadyOff, dfree0 = base + kDfreeOff;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem_raw + kFlagOff);
  volatile int* last_flag = reinterpret_cast<volatile int*>(smem_raw + kFlagOff + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem_raw + kFlagOff + 8);
  // stages start at the first 1024-byte boundary past the barriers
  const uint32_t st0 = (base + kBarBytes + 1023) & ~1023u;
  uint8_t* st0_ptr = smem_raw + (st0 - base);
  const int nst = p.nst;

  if (threadIdx.x == 0) {
    for (int s = 0; s < nst; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, kFoldWarps);
    }
    for (int b = 0; b < kBufs; ++b) {
      mbar_init(aready0 + 8 * b, kUnpackWarps);
      mbar_init(afree0 + 8 * b, 1);
      mbar_init(dready0 + 8 * b, 1);
      mbar_init(dfree0 + 8 * b, kFoldWarps);
    }
    *abort_flag = 0;
    mbar_init_fence();
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(tmem_slot)),
                 "n"(kCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_launch_dependents();
  // activations, outputs and the workspace follow earlier kernels; the
  // copy warp waits later, after requesting its first stages' weights
  if (warp != kCopyWarp) pdl_wait();

  const Segs segs = segs_of<SK>(p);

  if (warp == kCopyWarp) {
    // ------------------------------------------------------------ producer
    const uint64_t pol = policy_evict_first();
    int slot = 0, issued = 0;
    uint32_t phase = 0;
    bool ok = true;
    // Weights do not depend on earlier kernels (W4_FLAG_PDL's contract): the
    // first nst stages' codes and steps are requested before the wait, their
    // activation boxes (slice dsl[s] of stage s) after it.
    bool waited = false;
    int dsl[kMaxStages];
    auto wait_then_activations = [&]() {
      pdl_wait();
      waited = true;
      if (lane == 0)
        for (int s = 0; s < min(issued, nst); ++s)
          tma_load_3d(st0 + s * p.stage_bytes + p.off_b, &p.tm_x, 0, 0, dsl[s] * (kSliceK / 8),
                      full0 + 8 * s, pol);
      __syncwarp();
    };
    for (int i = 0; i < segs.n && ok; ++i) {
      const Seg sg = seg_at<SK>(p, segs, i);
      const int t = sg.t, sl0 = sg.b, sl1 = sg.e;
      for (int sl = sl0; sl < sl1; ++sl) {
        if (issued >= nst && !waited) wait_then_activations();
        if (issued >= nst && !wait_bar(empty0 + 8 * slot, phase ^ 1u, abort_flag)) {
          if (*abort_flag == 0) report(p.status, W4_ERR_TIMEOUT);
          *abort_flag = 1;
          ok = false;
          break;
        }
        const uint32_t stg = st0 + slot * p.stage_bytes;
        if (lane == 0) {
          mbar_arrive_expect_tx(full0 + 8 * slot,
                                (uint32_t)(kCodesBytes + kStepsBytes + p.xrows * kSliceK * 2));
          tma_load_2d(stg, &p.tm_codes, sl * (kSliceK / 2), t * kRows, full0 + 8 * slot, pol);
          tma_load_2d(stg + kCodesBytes, &p.tm_steps, sl * kSliceGroups, t * kRows,
                      full0 + 8 * slot, pol);
          if (waited)
            tma_load_3d(stg + p.off_b, &p.tm_x, 0, 0, sl * (kSliceK / 8), full0 + 8 * slot, pol);
          else
            dsl[slot] = sl;
        }
        __syncwarp();
        ++issued;
        if (++slot == nst) {
          slot = 0;
          phase ^= 1u;
        }
      }
    }
    // fewer stages than the ring holds (or a timed-out wait): the
    // activation boxes of the stages requested so far still go out
    if (!waited) wait_then_activations();
    // every tile of this CTA is requested: its share of the caller's L2
    // ranges (the next call's weights) goes out now, behind them
    if (p.l2.n > 0 && *abort_flag == 0) l2_prefetch_share(p.l2, blockIdx.x, gridDim.x, lane);
    // let the last copies land before the CTA may leave
    const int last = issued < nst ? issued : nst;
    for (int i = 1; i <= last; ++i) {
      const int sl = slot - i < 0 ? slot - i + nst : slot - i;
      const uint32_t ph = slot - i < 0 ? phase ^ 1u : phase;
      if (!mbar_wait_bounded(full0 + 8 * sl, ph, kWaitCycles)) {
        report(p.status, W4_ERR_TIMEOUT);
        break;
      }
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------- MMA issuer
    // Round r uses buffers b = r % kBufs for the (u = r / kBufs)-th time: its
    // MMAs go out once its A is stored and the D of use u - 1 has been read.
    int slot = 0;
    long long r = 0;
    bool ok = true;
    for (int i = 0; i < segs.n && ok; ++i) {
      const Seg sg = seg_at<SK>(p, segs, i);
      const int sl0 = sg.b, sl1 = sg.e;
      for (int sl = sl0; sl < sl1 && ok; ++sl) {
        const uint32_t stg = st0 + slot * p.stage_bytes;
        for (int q = 0; q < kRounds; ++q, ++r) {
          const int b = (int)(r % kBufs);
          const uint32_t use = (uint32_t)(r / kBufs);
          if (!wait_bar(aready0 + 8 * b, use & 1u, abort_flag) ||
              (use > 0 && !wait_bar(dfree0 + 8 * b, (use - 1) & 1u, abort_flag))) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (lane == 0) {
#pragma unroll
            for (int g = 0; g < G; ++g) {
              const int grp = q * G + g;
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                const uint32_t baddr = stg + p.off_b + (uint32_t)(4 * grp + 2 * h) * lbo;
                const uint64_t bdesc = (uint64_t)((baddr >> 4) & 0x3FFF) |
                                       ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
                                       ((uint64_t)(128 >> 4) << 32) | (1ull << 46);
                mma_f16(tmem + kDCol + (b * G + g) * NP, tmem + kACol + (b * G + g) * 16 + h * 8,
                        bdesc, kIdesc, (uint32_t)h);
              }
            }
            mma_commit(dready0 + 8 * b);
            mma_commit(afree0 + 8 * b);
          }
          __syncwarp();
        }
        if (++slot == nst) slot = 0;
      }
    }
    if (!ok) {
      if (*abort_flag == 0) report(p.status, W4_ERR_TIMEOUT);
      *abort_flag = 1;
    }
    // the last commits must land before the tensor memory is released
    for (int b = 0; b < kBufs && r > 0; ++b) {
      const long long uses = (r - b + kBufs - 1) / kBufs;   // rounds r' < r with r' % kBufs == b
      if (uses > 0) mbar_wait_bounded(afree0 + 8 * b, (uint32_t)((uses - 1) & 1), kWaitCycles);
    }
  } else if (warp < kUnpackWarps) {
    // -------------------------------------------------------- unpacking warps
    const int tid = threadIdx.x;                       // weight row within the tile
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    int slot = 0;
    uint32_t phase = 0;
    long long r = 0;
    bool ok = true;
    for (int i = 0; i < segs.n && ok; ++i) {
      const Seg sg = seg_at<SK>(p, segs, i);
      const int sl0 = sg.b, sl1 = sg.e;
      for (int sl = sl0; sl < sl1 && ok; ++sl) {
        if (!wait_bar(full0 + 8 * slot, phase, abort_flag)) {
          ok = false;
          break;
        }
        const uint8_t* stg_ptr = st0_ptr + slot * p.stage_bytes;
        for (int q = 0; q < kRounds; ++q, ++r) {
          const int b = (int)(r % kBufs);
          const uint32_t use = (uint32_t)(r / kBufs);
          // A[b] is free once the MMAs of its previous use are done
          if (use > 0 && !wait_bar(afree0 + 8 * b, (use - 1) & 1u, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll 2
          for (int g = 0; g < G; ++g) {
            const int grp = q * G + g;
            const uint4 w = *reinterpret_cast<const uint4*>(stg_ptr + tid * 128 + ((grp ^ (tid & 7)) << 4));
            uint32_t a[16];
            unpack_bf16(w.x, a);
            unpack_bf16(w.y, a + 4);
            unpack_bf16(w.z, a + 8);
            unpack_bf16(w.w, a + 12);
            tmem_st16(tmem + lane_base + kACol + (b * G + g) * 16, a);
          }
          asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(aready0 + 8 * b);   // this warp's rows are in
        }
        if (++slot == nst) {
          slot = 0;
          phase ^= 1u;
        }
      }
    }
    if (!ok) {
      if (*abort_flag == 0) report(p.status, W4_ERR_TIMEOUT);
      *abort_flag = 1;
    }
  } else if (warp < kUnpackWarps + kFoldWarps) {
    // ---------------------------------------------------------- folding warps
    const int tid = threadIdx.x - 32 * kUnpackWarps;   // weight row within the tile
    const uint32_t lane_base = (uint32_t)((warp - kUnpackWarps) * 32) << 16;
    int slot = 0;
    uint32_t phase = 0;
    long long r = 0;
    float acc[MC], rowsum[kTmemSum ? 1 : MC];
    bool ok = true;
    for (int i = 0; i < segs.n && ok; ++i) {
      const Seg sg = seg_at<SK>(p, segs, i);
      const int t = sg.t, sl0 = sg.b, sl1 = sg.e;
      const bool direct = sg.kind != kSegSplit;   // the row sum stays in this CTA
      const int row = t * kRows + tid;
      if constexpr (!kTmemSum) {
#pragma unroll
        for (int m = 0; m < MC; ++m) rowsum[m] = 0.0f;
      }
      for (int sl = sl0; sl < sl1 && ok; ++sl) {
        // the stage's data (steps) is visible once its copies have landed
        if (!wait_bar(full0 + 8 * slot, phase, abort_flag)) {
          ok = false;
          break;
        }
        const uint8_t* stg_ptr = st0_ptr + slot * p.stage_bytes;
        float stv[kSliceGroups];   // the row's 8 steps of the slice, one 16-byte load
        {
          const uint4 sv = *reinterpret_cast<const uint4*>(stg_ptr + kCodesBytes + tid * 16);
          const uint32_t wv[4] = {sv.x, sv.y, sv.z, sv.w};
#pragma unroll
          for (int j = 0; j < kSliceGroups; ++j)
            stv[j] = bf16_bits_to_float((wv[j >> 1] >> (16 * (j & 1))) & 0xFFFFu);
        }
#pragma unroll
        for (int m = 0; m < MC; ++m) acc[m] = 0.0f;
#pragma unroll
        for (int q = 0; q < kRounds; ++q) {
          const int b = (int)(r % kBufs);
          const uint32_t use = (uint32_t)(r / kBufs);
          if (!wait_bar(dready0 + 8 * b, use & 1u, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int g0 = 0; g0 < G; g0 += kLdBatch) {
            float d[kLdBatch][MC];
#pragma unroll
            for (int g = 0; g < kLdBatch; ++g)
              tmem_ld<MC>(tmem + lane_base + kDCol + (b * G + g0 + g) * NP, d[g]);
            tmem_wait_ld<kLdBatch * MC>(&d[0][0]);
#pragma unroll
            for (int g = 0; g < kLdBatch; ++g)
#pragma unroll
              for (int m = 0; m < MC; ++m) acc[m] = fmaf(stv[q * G + g0 + g], d[g][m], acc[m]);
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(dfree0 + 8 * b);   // this warp has read D[b]
          ++r;
        }
        if (!ok) break;
        // the slice is done: its sum goes on, its stage back to the copy warp
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * slot);
        // a tile's last slices continue from the previous CTA's prefix (the
        // same sum, in the same order, as if this CTA had run every slice)
        const bool from_prefix = SK && sg.kind == kSegTail && sl == sl0;
        if (SK && from_prefix) {
          if (tid == 0) *last_flag = wait_flag_gpu(p.sk_flag + blockIdx.x - 1, abort_flag) ? 1 : 0;
          asm volatile("bar.sync 1, %0;" ::"n"(kRows) : "memory");
          if (*last_flag == 0) {
            ok = false;
            break;
          }
        }
        if (direct) {
          if constexpr (kTmemSum) {
            // sum (from 0, or from the prefix) of the slices so far, kept
            // in tensor memory
            float sum[MC];
            if (sl == sl0) {
#pragma unroll
              for (int m = 0; m < MC; ++m) sum[m] = 0.0f;
              if (from_prefix) take_prefix<MC>(p, tid, sum);
            } else {
              tmem_ld<MC>(tmem + lane_base + kSumCol, sum);
              tmem_wait_ld<MC>(sum);
            }
            uint32_t v[MC];
#pragma unroll
            for (int m = 0; m < MC; ++m) v[m] = __float_as_uint(sum[m] + acc[m]);
#pragma unroll
            for (int c = 0; c < MC; c += 16) tmem_st16(tmem + lane_base + kSumCol + c, v + c);
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
          } else {
            if (from_prefix) take_prefix<MC>(p, tid, rowsum);
#pragma unroll
            for (int m = 0; m < MC; ++m) rowsum[m] += acc[m];
          }
        } else if (row < p.N) {
#pragma unroll
          for (int m = 0; m < MC; ++m)
            if (m < p.M) p.ws_partial[((long long)sl * p.M + m) * p.N + row] = acc[m];
        }
        if (++slot == nst) {
          slot = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      if (direct) {
        float* sum = rowsum;
        float tsum[kTmemSum ? MC : 1];
        if constexpr (kTmemSum) {
          tmem_ld<MC>(tmem + lane_base + kSumCol, tsum);
          tmem_wait_ld<MC>(tsum);
          sum = tsum;
        }
        if (SK && sg.kind == kSegHead) {
          // the tile's first slices: their sum (every row of the tile) goes
          // to prefix slot blockIdx.x for the next CTA.  The barrier orders
          // all rows' stores before thread 0's release of the flag.
          float* out = p.sk_prefix + (long long)blockIdx.x * p.M * kRows + tid;
#pragma unroll
          for (int m = 0; m < MC; ++m)
            if (m < p.M) out[(long long)m * kRows] = sum[m];
          __threadfence();
          asm volatile("bar.sync 1, %0;" ::"n"(kRows) : "memory");
          if (tid == 0) store_release_gpu(p.sk_flag + blockIdx.x, 1);
          continue;
        }
        if (row < p.N) {
#pragma unroll
          for (int m = 0; m < MC; ++m)
            if (m < p.M) p.y[(long long)m * p.N + row] = __float2bfloat16_rn(sum[m]);
        }
        if (SK && sg.kind == kSegTail) {
          // every row has read the prefix (at the first slice): the slot is
          // re-armed for the next call
          asm volatile("bar.sync 1, %0;" ::"n"(kRows) : "memory");
          if (tid == 0) p.sk_flag[blockIdx.x - 1] = 0;
        }
        continue;
      }
      // Split-K: the last CTA to finish this tile adds the slice sums in
      // slice order.  The barrier orders the partial stores of all rows
      // before thread 0's release; its acquire, then the second barrier,
      // order the other CTAs' partials before they are read.
      asm volatile("bar.sync 1, %0;" ::"n"(kRows) : "memory");
      if (tid == 0) *last_flag = atomic_add_acq_rel_gpu(p.ws_count + t, 1) == p.S - 1;
      asm volatile("bar.sync 1, %0;" ::"n"(kRows) : "memory");
      if (*last_flag) {
        if (row < p.N) {
          // CB activation columns at a time; for each, SB slices' partials
          // in flight at once, then added in slice order
          constexpr int CB = MC < 8 ? MC : 8, SB = 32 / CB;
#pragma unroll 1
          for (int m0 = 0; m0 < MC; m0 += CB) {
            if (m0 >= p.M) break;
            float fsum[CB];
#pragma unroll
            for (int c = 0; c < CB; ++c) fsum[c] = 0.0f;
            for (int sb = 0; sb < p.slices; sb += SB) {
              float v[SB][CB];
#pragma unroll
              for (int k2 = 0; k2 < SB; ++k2)
#pragma unroll
                for (int c = 0; c < CB; ++c)
                  v[k2][c] = (sb + k2 < p.slices && m0 + c < p.M)
                                 ? __ldcg(p.ws_partial + ((long long)(sb + k2) * p.M + m0 + c) * p.N + row)
                                 : 0.0f;
#pragma unroll
              for (int k2 = 0; k2 < SB; ++k2)
                if (sb + k2 < p.slices) {
#pragma unroll
                  for (int c = 0; c < CB; ++c) fsum[c] += v[k2][c];
                }
            }
#pragma unroll
            for (int c = 0; c < CB; ++c)
              if (m0 + c < p.M) p.y[(long long)(m0 + c) * p.N + row] = __float2bfloat16_rn(fsum[c]);
          }
        }
        if (tid == 0) atomicExch(p.ws_count + t, 0);
      }
      asm volatile("bar.sync 1, %0;" ::"n"(kRows) : "memory");
    }
    if (!ok) {
      if (*abort_flag == 0) report(p.status, W4_ERR_TIMEOUT);
      *abort_flag = 1;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kCols)
                 : "memory");
}

// ================================================================= host side
PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  static std::mutex mu;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static bool tried = false;
  std::lock_guard<std::mutex> lock(mu);
  if (!tried) {
    tried = true;
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    else
      cudaGetLastError();
  }
  return fn;
}

namespace {

// Stage: codes (16 KB, 1024-aligned for the swizzle), steps (2 KB), then the
// B operand (np x 256 bf16).
int stage_bytes_of(int np, int* off_b) {
  *off_b = kCodesBytes + kStepsBytes;
  return (*off_b + np * kSliceK * 2 + 1023) & ~1023;
}

struct DevInfo {
  int sms = 0, smem_optin = 0;
};

DevInfo dev_info(int dev) {
  static std::mutex mu;
  static DevInfo cache[64];
  std::lock_guard<std::mutex> lock(mu);
  if (dev < 0 || dev >= 64) return DevInfo{};
  if (cache[dev].sms == 0) {
    int sms = 0, optin = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess) {
      cudaGetLastError();
      return DevInfo{};
    }
    cache[dev].sms = sms;
    cache[dev].smem_optin = optin;
  }
  return cache[dev];
}

using TcFn = void (*)(TcParams);

int mc_of(int M) { return M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : M <= 8 ? 8 : M <= 16 ? 16 : 32; }

// Instantiations: (MC, 4 rounds), (MC, 2 rounds), (MC, 2 rounds, balanced
// runs); key = log2(MC) + 6 * variant.
TcFn kernel_of(int mc, int bufs, bool sk) {
  if (bufs >= 4) {
    switch (mc) {
      case 1: return tc_kernel<1, 4, false>;
      case 2: return tc_kernel<2, 4, false>;
      case 4: return tc_kernel<4, 4, false>;
      case 8: return tc_kernel<8, 4, false>;
      case 16: return tc_kernel<16, 4, false>;
      default: return tc_kernel<32, 4, false>;
    }
  }
  if (sk) {
    switch (mc) {
      case 1: return tc_kernel<1, 2, true>;
      case 2: return tc_kernel<2, 2, true>;
      case 4: return tc_kernel<4, 2, true>;
      case 8: return tc_kernel<8, 2, true>;
      case 16: return tc_kernel<16, 2, true>;
      default: return tc_kernel<32, 2, true>;
    }
  }
  switch (mc) {
    case 1: return tc_kernel<1, 2, false>;
    case 2: return tc_kernel<2, 2, false>;
    case 4: return tc_kernel<4, 2, false>;
    case 8: return tc_kernel<8, 2, false>;
    case 16: return tc_kernel<16, 2, false>;
    default: return tc_kernel<32, 2, false>;
  }
}
int kernel_key(int mc, int bufs, bool sk) {
  int l = 0;
  while ((1 << l) < mc && l < 5) ++l;
  return l + 6 * (bufs >= 4 ? 1 : (sk ? 2 : 0));
}

cudaError_t allow_smem(TcFn fn, int key, int smem, int dev) {
  static std::mutex mu;
  static int done[64][18] = {};
  if (dev < 0 || dev >= 64 || key < 0 || key >= 18) return cudaErrorInvalidDevice;
  const int k = key;
  std::lock_guard<std::mutex> lock(mu);
  if (done[dev][k] >= smem) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess) done[dev][k] = smem;
  return e;
}

}  // namespace

bool tc_supported(int M, int K) {
  return M >= 1 && M <= kTcMaxM && K >= kSliceK && K % kSliceK == 0 && encoder() != nullptr;
}

bool tc_plan(int M, int N, int K, int sms, TcPlan* out, bool allow_sk) {
  if (M < 1 || M > kTcMaxM || K % kSliceK != 0 || N < 1) return false;
  TcPlan pl;
  pl.np = M <= 16 ? 16 : 32;
  pl.slices = K / kSliceK;
  pl.tiles = (N + kRows - 1) / kRows;
  // K splits, only for few row tiles (the split-K fix-up costs more than
  // leaving part of the grid idle): as many as still give every CTA at most
  // one unit.  First with one CTA per SM, which holds all of the SM's tensor
  // memory for four rounds in flight (measured 7-18% faster when the units
  // fit the SMs, where the rounds' hand-off latency sets the pace); when the
  // units do not fit, two CTAs per SM of two rounds each (more warps issue).
  for (int per_sm = 1; per_sm <= 2; ++per_sm) {
    const int target = per_sm * std::max(1, sms);
    int S = 1;
    if (2 * pl.tiles <= std::max(1, sms)) S = std::max(1, std::min(pl.slices, target / pl.tiles));
    pl.sps = (pl.slices + S - 1) / S;
    pl.S = (pl.slices + pl.sps - 1) / pl.sps;
    pl.units = pl.tiles * pl.S;
    pl.per_sm = per_sm;
    if (per_sm == 1 && pl.units > std::max(1, sms)) continue;
    break;
  }
  pl.bufs = pl.per_sm == 1 ? 4 : 2;
  pl.ctas = std::min(pl.units, pl.per_sm * std::max(1, sms));
  int off_b;
  pl.stage_bytes = stage_bytes_of(pl.np, &off_b);
  pl.off_b = off_b;
  // each of the SM's CTAs keeps its share of the 228 KB of shared memory
  const int budget = pl.per_sm == 2 ? 232448 / 2 - 1024 : 232448 - 1024;
  pl.nst = std::min(pl.per_sm == 2 ? 4 : kMaxStages, (budget - kBarBytes - 1024) / pl.stage_bytes);
  if (pl.nst < 2) return false;
  pl.smem = kBarBytes + 1024 + pl.nst * pl.stage_bytes;
  // one CTA per SM must stay one: a second would wait in the tensor-memory
  // allocation for the first to finish (all 512 columns are taken)
  if (pl.per_sm == 1) pl.smem = std::max(pl.smem, 232448 / 2 + 1024);
  if (pl.S > 1) {
    pl.ws_part_off = ((size_t)pl.tiles * sizeof(int) + 255) & ~size_t(255);
    pl.ws_bytes = pl.ws_part_off + (size_t)pl.slices * M * N * sizeof(float);
  }
  // Balanced runs when whole tiles divide badly over the CTAs: the busiest
  // CTA's tiles at least 1.25x the mean (measured at 43008 x 5376, M = 16:
  // 336 tiles on 304 CTAs took 78.6 us, 304 tiles 48.3 us, 608 tiles
  // 82.2 us; balanced runs 56-57 us; near 1.19x the two plans are within
  // +-8% either way).  Every run covers at least one tile's slices, so a
  // tile is cut at most once; needs the hand-over slots.
  const long long busiest = (pl.tiles + pl.ctas - 1) / pl.ctas;
  if (allow_sk && pl.S == 1 && pl.slices >= 2 && pl.tiles > pl.ctas &&
      4LL * busiest * pl.ctas >= 5LL * pl.tiles &&
      (long long)pl.tiles * pl.slices / pl.ctas >= pl.slices) {
    pl.sk = 1;
    pl.ws_part_off = ((size_t)pl.ctas * sizeof(int) + 255) & ~size_t(255);
    pl.ws_bytes = pl.ws_part_off + (size_t)pl.ctas * M * kRows * sizeof(float);
  }
  *out = pl;
  return true;
}

cudaError_t tc_launch(const TcPlan& pl, void* y, const void* qw, const void* st, const void* x, int M,
                      int N, int K, void* workspace, int32_t* status, bool pdl, cudaStream_t stream,
                      int dev, const L2Ranges* l2) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
  if (enc == nullptr) return cudaErrorNotSupported;
  TcParams p = {};
  {
    const cuuint64_t dims[2] = {(cuuint64_t)K / 2, (cuuint64_t)N};
    const cuuint64_t strides[1] = {(cuuint64_t)K / 2};
    const cuuint32_t box[2] = {128, kRows};
    const cuuint32_t es[2] = {1, 1};
    if (enc(&p.tm_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(qw), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[2] = {(cuuint64_t)K / 32, (cuuint64_t)N};
    const cuuint64_t strides[1] = {(cuuint64_t)K / 32 * 2};
    const cuuint32_t box[2] = {kSliceGroups, kRows};
    const cuuint32_t es[2] = {1, 1};
    if (enc(&p.tm_steps, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(st), dims, strides,
            box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    // x [M][K] seen as (8 codes, M rows, K/8 blocks): a slice's box lands as
    // [block][row][8] = the K-major core-matrix layout of the B operand
    const cuuint64_t dims[3] = {8, (cuuint64_t)M, (cuuint64_t)K / 8};
    const cuuint64_t strides[2] = {(cuuint64_t)K * 2, 16};
    const cuuint32_t box[3] = {8, (cuuint32_t)M, kSliceK / 8};
    const cuuint32_t es[3] = {1, 1, 1};
    if (enc(&p.tm_x, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void*>(x), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  p.x = static_cast<const __nv_bfloat16*>(x);
  p.y = static_cast<__nv_bfloat16*>(y);
  p.M = M;
  p.N = N;
  p.K = K;
  p.slices = pl.slices;
  p.tiles = pl.tiles;
  p.S = pl.S;
  p.sps = pl.sps;
  p.units = pl.units;
  p.nst = pl.nst;
  p.stage_bytes = pl.stage_bytes;
  p.off_b = pl.off_b;
  p.xrows = M;
  p.status = status;
  if (l2 != nullptr) p.l2 = *l2;
  if (pl.sk) {
    p.sk = 1;
    p.sk_flag = static_cast<int*>(workspace);
    p.sk_prefix = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + pl.ws_part_off);
  }
  if (pl.S > 1) {
    p.ws_count = static_cast<int*>(workspace);
    p.ws_partial = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + pl.ws_part_off);
  }
  const TcFn fn = kernel_of(mc_of(M), pl.bufs, pl.sk != 0);
  const cudaError_t ea = allow_smem(fn, kernel_key(mc_of(M), pl.bufs, pl.sk != 0), pl.smem, dev);
  if (ea != cudaSuccess) return ea;
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
  return cudaLaunchKernelEx(&cfg, fn, p);
}

int tc_sms(int dev) { return dev_info(dev).sms; }

}  // namespace tc
}  // namespace w4
