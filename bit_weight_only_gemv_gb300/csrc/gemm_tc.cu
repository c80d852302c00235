// W4A16 group-32 GEMM for prompt chunks (33 to 256 activation rows) on the
// 5th-generation tensor cores (tcgen05, sm_103a).
//
// Page "Gemma 4 on a 4 GB GPU in Plain PyTorch", section "Step 6 — Read
// Prompts in 32-Bit on a Card Without Tensor Cores": prompts go through the
// model 256 tokens at a time, and for each product the weights are expanded
// to full precision first (fp32 for cuBLAS there, on a card with no tensor
// cores).
// Here the tensor cores take the product and the weights are unpacked on the
// fly, without rounding:
//
//  * w = (code - 8) * step has at most 11 significant bits, so it is exactly
//    hi + lo with hi = bf16(w) and lo = w - hi (at most 3 significant bits):
//    one bf16x2 multiply and one bf16x2 fused multiply-add per pair of codes.
//    Four warps (thread = weight row) unpack each 32-code group into hi and
//    lo and store both into tensor memory as the MMA's A operand; the MMA
//    warp issues per group two K = 16 MMAs for hi and two for lo into one
//    fp32 accumulator.  bf16 x bf16 products are exact; only the fp32 sums
//    round.  The step is inside A, so no per-group rescaling follows.
//  * A CTA owns units of 128 weight rows times all the activation rows (the
//    MMA's N, up to 256; when the weight tiles are too few for the SMs, a
//    tile of the activation rows).  The copy warp streams 256-code slices of
//    codes (2-D TMA box, 128-byte swizzle) and steps (2-D box), and per two
//    groups the unit's activations as one 2-D box of 64 codes x its rows
//    with 128-byte swizzle: the canonical K-major B-operand layout, each
//    16-code K step an address offset inside the 128-byte rows.
//  * Association: one fp32 accumulator per (weight row, activation row) over
//    the whole of K, groups in order; four epilogue warps round it to bf16
//    once.  Results depend on K only (not on N, M or the tiling).
//  * Tensor memory: eight A buffers (one group each, 32 columns), handed from
//    the unpacking warps to the MMA warp four groups at a time, and one
//    accumulator of up to 256 columns.  Below N = 256 an MMA of 128 rows
//    takes about as long whatever its N (measured: about 90 cycles), and
//    each hand-off costs a few hundred cycles of commits and waits, so the
//    widest N (all activation rows at once) and the largest hand-off the
//    ring allows do the most work per MMA.
//  * Every wait is bounded; on expiry W4_ERR_TIMEOUT is recorded, the warps
//    leave their loops, in-flight copies and MMAs are waited for (bounded)
//    and the tensor memory is released before exit.
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "gemv_tc.h"
#include "tc_common.cuh"

namespace w4 {
namespace tc {
namespace {

constexpr int kRows = 128;           // weight rows per unit = MMA M
constexpr int kSliceK = 256;         // codes per row per codes stage
constexpr int kSliceGroups = 8;
constexpr int kMaxTok = 256;         // activation rows per unit (MMA N <= 256)
constexpr int kUnpackWarps = 4;
constexpr int kEpiWarps = 4;
constexpr int kCopyWarp = kUnpackWarps + kEpiWarps;
constexpr int kMmaWarp = kCopyWarp + 1;
constexpr int kThreads = 32 * (kMmaWarp + 1);
constexpr int kCodeStages = 3;
constexpr int kMaxXStages = 8;        // activation stages of two groups each
constexpr int kABufs = 8;            // A operands in tensor memory (one group each)
constexpr int kHand = 4;             // groups handed over at a time
constexpr int kAPairs = kABufs / kHand;   // A hand-off units in the ring
constexpr int kDBufs = 1;            // accumulators
constexpr int kACol = 0;             // [kABufs][hi 16 | lo 16] columns
constexpr int kDCol = kABufs * 32;   // [kDBufs][kMaxTok]
constexpr int kCols = 512;
static_assert(kDCol + kDBufs * kMaxTok <= kCols, "tensor memory");
static_assert(kSliceGroups % kHand == 0 && kHand % 2 == 0, "hand-offs");
static_assert((kAPairs & (kAPairs - 1)) == 0 && (kDBufs & (kDBufs - 1)) == 0, "ring sizes");
static_assert(kTpMaxM <= kMaxTok, "one activation tile per unit");
constexpr int kCodesBytes = kRows * 128;                  // 16 KB, 128-byte swizzle
constexpr int kStepsBytes = kRows * 16;                   // 2 KB
constexpr int kCodeStageBytes = kCodesBytes + kStepsBytes;   // 18 KB, a multiple of 1024
// barriers: cfull[4] cempty[4] xfull[8] xempty[8] aready[8] afree[8]
// dready[2] dfree[2], abort flag, tensor-memory base
constexpr int kOffCFull = 0, kOffCEmpty = 32, kOffXFull = 64, kOffXEmpty = 128;
constexpr int kOffAReady = 192, kOffAFree = 256, kOffDReady = 320, kOffDFree = 336;
constexpr int kOffAbort = 352, kOffTmem = 356;
constexpr int kBarBytes = 384;

struct TpParams {
  CUtensorMap tm_codes;   // codes as uint8 [N][K/2], box 128 x 128, 128-byte swizzle
  CUtensorMap tm_steps;   // steps as uint16 [N][K/32], box 8 x 128
  CUtensorMap tm_x;       // activations as uint16 [M][K], box 64 x xrows, 128-byte swizzle
  __nv_bfloat16* y;       // [M][N]
  int M, N, K;
  int groups;             // K / 32
  int tiles;              // 128-row weight tiles
  int xrows;              // activation rows per unit tile
  int nt;                 // MMA N: xrows rounded up to 16
  int units;              // tiles x activation tiles
  int xs;                 // activation stages
  int x_stage_bytes;
  int32_t* status;
};

// Exact bf16 split of the eight weights of one packed word, in pairs of
// consecutive codes (the lower code in the low half): (c - 8) from the
// page's float-bit trick in bf16 form, then hi = (c - 8) * step by one bf16x2
// multiply (the product of two bf16 values is exact before its one
// rounding, so hi = bf16(w)) and lo = (c - 8) * step - hi by one fused
// multiply-add (exact: w - hi has at most 3 significant bits).
__device__ __forceinline__ void split_word(uint32_t wd, __nv_bfloat162 step2, uint32_t hi[4],
                                           uint32_t lo[4]) {
  uint32_t c8[4];
  unpack_bf16(wd, c8);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 c = *reinterpret_cast<const __nv_bfloat162*>(&c8[i]);
    const __nv_bfloat162 h = __hmul2(c, step2);
    const __nv_bfloat162 l = __hfma2(c, step2, __hneg2(h));
    hi[i] = *reinterpret_cast<const uint32_t*>(&h);
    lo[i] = *reinterpret_cast<const uint32_t*>(&l);
  }
}

// B-operand (shared memory) descriptor of a K-major tile with 128-byte
// swizzle: rows of 128 bytes (64 bf16 of K), 1024 bytes between 8-row
// groups; `addr` advances by 32 bytes per 16-code K step inside the rows.
__device__ __forceinline__ uint64_t b_desc_sw128(uint32_t addr) {
  return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         (1ull << 46) | (2ull << 61);
}

// Warps 0-3 unpack A, 4-7 add the slice sums and write y, 8 copies, 9
// issues MMAs.  Hand-offs: cfull/cempty (codes and steps stages), xfull /
// xempty (activation stages, released by MMA completion), aready / afree (A
// buffers), dready / dfree (accumulators).
__global__ void __launch_bounds__(kThreads, 1) tp_kernel(const __grid_constant__ TpParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t base = smem_addr(smem_raw);
  const uint32_t cfull0 = base + kOffCFull, cempty0 = base + kOffCEmpty;
  const uint32_t xfull0 = base + kOffXFull, xempty0 = base + kOffXEmpty;
  const uint32_t aready0 = base + kOffAReady, afree0 = base + kOffAFree;
  const uint32_t dready0 = base + kOffDReady, dfree0 = base + kOffDFree;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem_raw + kOffAbort);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem_raw + kOffTmem);
  // code stages from the first 1024-byte boundary past the barriers, then
  // the activation stages
  const uint32_t cst0 = (base + kBarBytes + 1023) & ~1023u;
  const uint8_t* cst0_ptr = smem_raw + (cst0 - base);
  const uint32_t xst0 = cst0 + kCodeStages * kCodeStageBytes;
  const int xs = p.xs;
  const int slices = p.groups / kSliceGroups;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kCodeStages; ++s) {
      mbar_init(cfull0 + 8 * s, 1);
      mbar_init(cempty0 + 8 * s, kUnpackWarps);
    }
    for (int s = 0; s < xs; ++s) {
      mbar_init(xfull0 + 8 * s, 1);
      mbar_init(xempty0 + 8 * s, 1);
    }
    for (int b = 0; b < kAPairs; ++b) {
      mbar_init(aready0 + 8 * b, kUnpackWarps);
      mbar_init(afree0 + 8 * b, 1);
    }
    for (int b = 0; b < kDBufs; ++b) {
      mbar_init(dready0 + 8 * b, 1);
      mbar_init(dfree0 + 8 * b, kEpiWarps);
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
  // activations and outputs follow earlier kernels; the copy warp waits
  // later, after requesting its first code stages
  if (warp != kCopyWarp) pdl_wait();

  const int u0 = (int)((long long)blockIdx.x * p.units / gridDim.x);
  const int u1 = (int)((long long)(blockIdx.x + 1) * p.units / gridDim.x);
  bool ok = true;

  if (warp == kCopyWarp) {
    // ------------------------------------------------------------ producer
    const uint64_t pol = policy_evict_first();
    int cslot = 0, xslot = 0;
    uint32_t cph = 0, xph = 0;
    long long cissued = 0, xissued = 0;
    auto issue_codes = [&](int t, int sl) {
      const uint32_t cst = cst0 + cslot * kCodeStageBytes;
      if (lane == 0) {
        mbar_arrive_expect_tx(cfull0 + 8 * cslot, (uint32_t)kCodeStageBytes);
        tma_load_2d(cst, &p.tm_codes, sl * (kSliceK / 2), t * kRows, cfull0 + 8 * cslot, pol);
        tma_load_2d(cst + kCodesBytes, &p.tm_steps, sl * kSliceGroups, t * kRows,
                    cfull0 + 8 * cslot, pol);
      }
      __syncwarp();
      ++cissued;
      if (++cslot == kCodeStages) {
        cslot = 0;
        cph ^= 1u;
      }
    };
    // Weights do not depend on earlier kernels (W4_FLAG_PDL's contract):
    // the first code stages are requested before the wait.
    long long pre = 0;
    for (int u = u0; u < u1 && pre < kCodeStages; ++u) {
      const int t = u - (u / p.tiles) * p.tiles;
      for (int sl = 0; sl < slices && pre < kCodeStages; ++sl, ++pre) issue_codes(t, sl);
    }
    pdl_wait();
    long long idx = 0;   // (unit, slice) pairs walked so far
    for (int u = u0; u < u1 && ok; ++u) {
      const int mt = u / p.tiles, t = u - mt * p.tiles;
      for (int sl = 0; sl < slices && ok; ++sl) {
        if (idx++ >= pre) {
          if (cissued >= kCodeStages && !wait_bar(cempty0 + 8 * cslot, cph ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          issue_codes(t, sl);
        }
        for (int g = 0; g < kSliceGroups; g += 2) {
          if (xissued >= xs && !wait_bar(xempty0 + 8 * xslot, xph ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          if (lane == 0) {
            mbar_arrive_expect_tx(xfull0 + 8 * xslot, (uint32_t)(p.xrows * 128));
            tma_load_2d(xst0 + xslot * p.x_stage_bytes, &p.tm_x, (sl * kSliceGroups + g) * 32,
                        mt * p.xrows, xfull0 + 8 * xslot, pol);
          }
          __syncwarp();
          ++xissued;
          if (++xslot == xs) {
            xslot = 0;
            xph ^= 1u;
          }
        }
      }
    }
    // let the last copies land before the CTA may leave
    const int clast = cissued < kCodeStages ? (int)cissued : kCodeStages;
    for (int i = 1; i <= clast; ++i) {
      const int s = cslot - i < 0 ? cslot - i + kCodeStages : cslot - i;
      if (!mbar_wait_bounded(cfull0 + 8 * s, cslot - i < 0 ? cph ^ 1u : cph, kWaitCycles)) break;
    }
    const int xlast = xissued < xs ? (int)xissued : xs;
    for (int i = 1; i <= xlast; ++i) {
      const int s = xslot - i < 0 ? xslot - i + xs : xslot - i;
      if (!mbar_wait_bounded(xfull0 + 8 * s, xslot - i < 0 ? xph ^ 1u : xph, kWaitCycles)) break;
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------- MMA issuer
    // instruction descriptor: D fp32, A and B bf16, both K-major, N = nt, M = 128
    const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(p.nt >> 3) << 17) |
                           ((uint32_t)(kRows >> 4) << 24);
    // A buffers go by hand-offs of kHand groups (two activation stages): one
    // wait per stage, 4 kHand MMAs and three or four commits per hand-off
    long long pi = 0, si = 0;   // hand-offs and units issued
    int xsl = 0;                 // next activation stage and its phase
    uint32_t xph = 0;
    const int hands = p.groups / kHand;
    for (int u = u0; u < u1 && ok; ++u, ++si) {
      for (int q = 0; q < hands; ++q, ++pi) {
        const int a = (int)(pi & (kAPairs - 1));
        const bool first = q == 0;
        const bool last = q == hands - 1;
        const int d = (int)(si & (kDBufs - 1));
        int xsv[kHand / 2];
        bool got = wait_bar(aready0 + 8 * a, (uint32_t)((pi / kAPairs) & 1), abort_flag);
#pragma unroll
        for (int k = 0; k < kHand / 2; ++k) {
          xsv[k] = xsl;
          got = got && wait_bar(xfull0 + 8 * xsl, xph, abort_flag);
          if (++xsl == xs) {
            xsl = 0;
            xph ^= 1u;
          }
        }
        if (!got || (first && si >= kDBufs &&
                     !wait_bar(dfree0 + 8 * d, (uint32_t)((si / kDBufs - 1) & 1), abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (lane == 0) {
          const uint32_t dcol = tmem + kDCol + d * kMaxTok;
#pragma unroll
          for (int j = 0; j < kHand; ++j) {   // the hand-off's groups, two per stage
            const uint32_t xst = xst0 + xsv[j >> 1] * p.x_stage_bytes + (uint32_t)(j & 1) * 64;
            const uint32_t acol = tmem + kACol + (kHand * a + j) * 32;
#pragma unroll
            for (int h = 0; h < 2; ++h)   // hi: K = 16h .. 16h + 15
              mma_f16(dcol, acol + h * 8, b_desc_sw128(xst + 32 * h), idesc,
                      (first && j == 0 && h == 0) ? 0u : 1u);
#pragma unroll
            for (int h = 0; h < 2; ++h)   // lo
              mma_f16(dcol, acol + 16 + h * 8, b_desc_sw128(xst + 32 * h), idesc, 1u);
          }
          mma_commit(afree0 + 8 * a);
#pragma unroll
          for (int k = 0; k < kHand / 2; ++k) mma_commit(xempty0 + 8 * xsv[k]);
          if (last) mma_commit(dready0 + 8 * d);
        }
        __syncwarp();
      }
    }
    // the last commits must land before the tensor memory is released
    if (pi > 0) {
      const long long pl = pi - 1;
      mbar_wait_bounded(afree0 + 8 * (int)(pl & (kAPairs - 1)), (uint32_t)((pl / kAPairs) & 1),
                        kWaitCycles);
    }
  } else if (warp < kUnpackWarps) {
    // -------------------------------------------------------- unpacking warps
    const int tid = threadIdx.x;                       // weight row within the unit
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    int cslot = 0;
    uint32_t cph = 0;
    long long pi = 0;   // pairs of groups unpacked
    for (int u = u0; u < u1 && ok; ++u) {
      for (int sl = 0; sl < slices && ok; ++sl) {
        if (!wait_bar(cfull0 + 8 * cslot, cph, abort_flag)) {
          ok = false;
          break;
        }
        const uint8_t* cst = cst0_ptr + cslot * kCodeStageBytes;
        // the row's 8 steps of the slice, one 16-byte load
        const uint4 sv = *reinterpret_cast<const uint4*>(cst + kCodesBytes + tid * 16);
#pragma unroll 1
        for (int q = 0; q < kSliceGroups / kHand; ++q, ++pi) {
          const int a = (int)(pi & (kAPairs - 1));
          // A buffers of hand-off a are free once the MMAs of their previous use are done
          if (pi >= kAPairs &&
              !wait_bar(afree0 + 8 * a, (uint32_t)((pi / kAPairs - 1) & 1), abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll 2
          for (int j = 0; j < kHand; ++j) {
            const int g = kHand * q + j;
            const uint4 w = *reinterpret_cast<const uint4*>(cst + tid * 128 + ((g ^ (tid & 7)) << 4));
            // steps of groups 2i and 2i + 1 share one 32-bit word of the row's
            // eight; the group's step goes to both halves
            const uint32_t sw = (g & 4) ? ((g & 2) ? sv.w : sv.z) : ((g & 2) ? sv.y : sv.x);
            const uint32_t sb = (sw >> (16 * (g & 1))) & 0xFFFFu;
            const uint32_t s2 = sb | (sb << 16);
            const __nv_bfloat162 step = *reinterpret_cast<const __nv_bfloat162*>(&s2);
            uint32_t hi[16], lo[16];
            split_word(w.x, step, hi, lo);
            split_word(w.y, step, hi + 4, lo + 4);
            split_word(w.z, step, hi + 8, lo + 8);
            split_word(w.w, step, hi + 12, lo + 12);
            tmem_st16(tmem + lane_base + kACol + (kHand * a + j) * 32, hi);
            tmem_st16(tmem + lane_base + kACol + (kHand * a + j) * 32 + 16, lo);
          }
          asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(aready0 + 8 * a);   // this warp's rows are in
        }
        if (!ok) break;
        __syncwarp();
        if (lane == 0) mbar_arrive(cempty0 + 8 * cslot);   // codes and steps read
        if (++cslot == kCodeStages) {
          cslot = 0;
          cph ^= 1u;
        }
      }
    }
  } else if (warp < kUnpackWarps + kEpiWarps) {
    // --------------------------------------------------------- epilogue warps
    const int tid = threadIdx.x - 32 * kUnpackWarps;   // weight row within the unit
    const uint32_t lane_base = (uint32_t)((warp - kUnpackWarps) * 32) << 16;
    const int ncol = (p.xrows + 31) & ~31;             // columns read back, <= kMaxTok
    long long si = 0;
    for (int u = u0; u < u1 && ok; ++u, ++si) {
      const int mt = u / p.tiles, t = u - mt * p.tiles;
      const int row = t * kRows + tid;
      const int d = (int)(si % kDBufs);
      if (!wait_bar(dready0 + 8 * d, (uint32_t)((si / kDBufs) & 1), abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll 1
      for (int c0 = 0; c0 < ncol; c0 += 32) {
        float v[32];
        tmem_ld<32>(tmem + lane_base + kDCol + d * kMaxTok + c0, v);
        tmem_wait_ld<32>(v);
        if (row < p.N) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int col = c0 + i, tok = mt * p.xrows + col;
            if (col < p.xrows && tok < p.M)
              p.y[(long long)tok * p.N + row] = __float2bfloat16_rn(0.0f + v[i]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(dfree0 + 8 * d);   // this warp has read D[d]
    }
  }
  if (!ok) {
    if (*abort_flag == 0) report(p.status, W4_ERR_TIMEOUT);
    *abort_flag = 1;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kCols)
                 : "memory");
}

}  // namespace

// ================================================================= host side
namespace {

cudaError_t allow_tp_smem(int smem, int dev) {
  static std::mutex mu;
  static int done[64] = {};
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (done[dev] >= smem) return cudaSuccess;
  const cudaError_t e =
      cudaFuncSetAttribute(tp_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess) done[dev] = smem;
  return e;
}

}  // namespace

bool tp_plan(int M, int N, int K, int sms, TpPlan* out) {
  if (M < 1 || M > kTpMaxM || N < 1 || K < kSliceK || K % kSliceK != 0) return false;
  TpPlan pl;
  pl.tiles = (N + kRows - 1) / kRows;
  // All the activation rows in one unit, unless the weight tiles are too
  // few for the SMs: then the rows are cut into equal tiles (of at least 16)
  // while the units still fit one wave.  The tiling changes no result: each
  // output is its own accumulator column.
  int ttiles = (M + kMaxTok - 1) / kMaxTok;   // 1: kTpMaxM <= kMaxTok
  while (2 * ttiles * pl.tiles <= std::max(1, sms) && (M + 2 * ttiles - 1) / (2 * ttiles) >= 16)
    ttiles *= 2;
  pl.xrows = (M + ttiles - 1) / ttiles;
  pl.nt = (pl.xrows + 15) & ~15;
  pl.units = pl.tiles * ttiles;
  pl.ctas = std::min(pl.units, std::max(1, sms));
  // an activation stage: 128-byte rows of the MMA's N (the rows past the
  // tile's are never written and only reach unused columns), 1024-aligned
  pl.x_stage_bytes = (pl.nt * 128 + 1023) & ~1023;
  const int fixed = kBarBytes + 1024 + kCodeStages * kCodeStageBytes;
  const int budget = 232448 - 1024;
  pl.xs = std::min(kMaxXStages, (budget - fixed) / pl.x_stage_bytes);
  if (pl.xs < 2) return false;
  // more than half the SM's shared memory: one CTA per SM (each holds all
  // 512 columns of tensor memory)
  pl.smem = std::max(fixed + pl.xs * pl.x_stage_bytes, 232448 / 2 + 1024);
  *out = pl;
  return true;
}

cudaError_t tp_launch(const TpPlan& pl, void* y, const void* qw, const void* st, const void* x,
                      int M, int N, int K, int32_t* status, bool pdl, cudaStream_t stream,
                      int dev) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
  if (enc == nullptr) return cudaErrorNotSupported;
  TpParams p = {};
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
    // x [M][K]: a box of 64 codes x the tile's rows, 128-byte swizzle (the
    // K-major B-operand layout)
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)pl.xrows};
    const cuuint32_t es[2] = {1, 1};
    if (enc(&p.tm_x, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(x), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  p.y = static_cast<__nv_bfloat16*>(y);
  p.M = M;
  p.N = N;
  p.K = K;
  p.groups = K / 32;
  p.tiles = pl.tiles;
  p.xrows = pl.xrows;
  p.nt = pl.nt;
  p.units = pl.units;
  p.xs = pl.xs;
  p.x_stage_bytes = pl.x_stage_bytes;
  p.status = status;
  const cudaError_t ea = allow_tp_smem(pl.smem, dev);
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
  return cudaLaunchKernelEx(&cfg, tp_kernel, p);
}

}  // namespace tc
}  // namespace w4
