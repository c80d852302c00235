// W4A16 group-32 GEMV and routed-expert GEMV for GB300 (sm_103a).
//
// Page "Gemma 4 on a 4 GB GPU in Plain PyTorch", section "Step 3 — Multiply
// Straight From the Packed Weights": every decoded token takes the product of
// one activation vector with each weight matrix, computed from the 4-bit words
// as stored; the time per token is then set by the rate at which those words
// can be read from memory.  The routed-expert
// variant (page "Running a 26B MoE on an 8 GB Jetson by streaming experts from
// SSD", section "Streaming without touching a single GPU kernel") reads expert
// `id` at base + id * stride.
//
// Design (CTAs of 7 consumer warps + 1 producer warp, one or two per SM):
//  * The producer warp streams weight tiles (a window of whole rows: packed
//    codes and bf16 steps, contiguous in memory) from HBM into a ring of
//    shared-memory stages with 1-D bulk copies on the TMA engine.  One mbarrier per stage
//    counts the bytes in ("full"), another the consumer warps done with it
//    ("empty").  The copies need no registers, so several tiles are in
//    flight per CTA while the consumers compute, and with W4_FLAG_PDL the
//    first tiles are requested before the previous kernel has finished.
//  * The activation rows are staged once per CTA in shared memory as fp16
//    pairs scaled by a power of two per group of 32 (exact), next to the
//    group's inverse scale.
//  * A team of T lanes shares an output row (T = a power of two dividing
//    K/32, chosen from K alone); lane t of the team owns groups t, t + T, ...
//    of the row.  The window's work items (a K chunk of a step of rows) are
//    dealt round-robin to the consumer warps; a lane loads one group's
//    activations once and applies them to RW rows (activation reuse),
//    reading each row's codes and steps from shared memory.
//  * Per group and row the lane turns each packed word into four fp16 pairs
//    (c - 8) with the float-bit trick of the page in its fp16 form
//    ((0x6400 | c) - 1032 = c - 8, exact), multiplies them with the fp16
//    activation pairs in packed fp16 (products exact), sums each pair lane
//    over the group's 4 words in fp16 (at most 3 roundings: 3 * 2^-11 of
//    sum|w x|), adds the 8 partial sums in fp32, rescales by the group's 2^-e
//    (exact), multiplies by the step and accumulates in fp32.
//  * K is cut into chunks of CL groups per lane (CL from K alone).  After
//    each chunk the team reduces with a fixed xor-shuffle tree; the chunk
//    sums of a row (kept in shared memory) are added in chunk order.  A row's arithmetic therefore
//    depends on K only, never on N, M, the row index, the tiling, the split
//    or the addresses: results are bitwise reproducible, a gemv_id row
//    equals the gemv of that expert, and merged projections equal separate
//    ones.
//  * Each CTA owns a balanced contiguous range of rows (split-K, for few
//    rows and long K: of (row block, K slice) units).  Split-K writes chunk
//    sums to the workspace; per row block, the last of the slices to finish
//    (atomic counter, no waiting) adds them in chunk order, writes the rows
//    and re-arms the counter.
//  * Every wait is bounded: on expiry the kernel records W4_ERR_TIMEOUT, the
//    warps leave without further waiting, and the producer lets its copies
//    in flight land (bounded) before the CTA exits.
#include <algorithm>
#include <cmath>
#include <mutex>

#include "common.cuh"
#include "gemv_core.cuh"
#include "gemv_host.h"
#include "gemv_tc.h"

// Window counters of dense launches that hand out their windows at run time:
// kWorkSlots slots of (windows taken, CTAs done), 64 bytes apart, used round
// robin by successive launches on a device.  A launch's last CTA re-arms its
// slot, so a slot is clean again long before it comes round (only a
// launch still running kWorkSlots launches later could see it in use).
constexpr int kWorkSlots = 1024;
static __device__ __align__(64) int w4_window_counters[kWorkSlots * 16];

namespace w4 {

constexpr int kConsumerWarps = 7;
constexpr int kConsumers = 32 * kConsumerWarps;
constexpr int kThreads = kConsumers + 32;   // + the producer warp
constexpr int kMaxMR = 4;                   // activation rows per launch
constexpr int kMaxStages = 8;
constexpr int kBarBytes = 256;              // full[8], empty[8], flags, windows[8]
constexpr int kWinOff = 160;                // (row0, rows) of each stage's window (dense calls)
constexpr int kItemOff = 224;               // item of each stage's window (routed run-time windows)
constexpr long long kWaitCycles = 1LL << 31;

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
  int Kgp;                             // groups per row padded to a whole team (>= Kg)
  int n_items;
  int T, nsw;                          // lanes per row, row sets per warp (32 / T)
  int NI, CL, nch;                     // groups per lane per row, per chunk; chunks
  int RB;                              // rows of a window (a multiple of nsw * RW)
  int S, cps, upi;                     // slices, chunks per slice, row blocks per item
  int B;                               // row blocks (split-K only)
  long long U;                         // work items: rows (S == 1) or units
  int x_slots;                         // activation rows staged per CTA (per MR row)
  int nst;                             // pipeline stages
  int tile_bytes, code_pitch, step_pitch, step_off;
  int* ws_count;                       // [B] at the start of the workspace
  float* ws_partial;                   // [B][nch][RB][MR] after it
  int32_t* status;
  int gated;                           // x rows are [gate K | up K]: the product takes silu(gate) * up
  int dyn;                             // windows handed out at run time (dense, whole rows)
  int* work;                           // [0] windows taken, [1] CTAs done (dyn only)
  // routed calls with real expert ids (all nullptr otherwise)
  const int32_t* eids;                 // [n_items] real expert of each item
  int num_real;                        // experts behind eids
  const int32_t* slot_expert;          // [num_experts] expert each slot holds, or nullptr
  const __nv_bfloat16* escale;         // [num_real][N] output scale, or nullptr
  const __nv_bfloat16* ebias;          // [num_real][N] output bias, or nullptr
  L2Ranges l2;                         // brought into L2 after the launch's own tiles
  int ids_final;                       // routed ids written before the previous kernel began
};

// ---------------------------------------------------------------- activations
// Stage the activation rows of `nslots` items (or one shared row) as fp16
// pairs scaled by 2^e per group of 32 so that the group's largest magnitude
// lies in [2^9, 2^10).  Layout for staged row j (= slot * MR + m): 16-byte
// chunk (w, g) = pairs (x[8w+p], x[8w+p+4]) for p = 0..3 of group g, at
// ((j * 4 + w) * Kgp + g) * 16; the inverse scale 2^-e of the group at
// xscale[j * Kgp + g].  Groups Kg .. Kgp-1 (padding of a team that does not
// divide K/32) are zero with a zero inverse scale.  Run by the consumer
// threads.
// Gated activations (W4_FLAG_SILU_MUL): row j of x holds gate[K] then
// up[K], and the activation is h = silu(gate) * up = gate / (1 + e^-gate) *
// up, computed in fp32 and staged as above (fp16 pairs scaled by 2^e per
// group, rounded to nearest: a relative error of at most 2^-11 per element,
// where bf16 inputs stage exactly).  Every CTA computes the whole row.
__device__ __noinline__ void stage_x_gated(const GemvParams& p, int nslots, uint8_t* xs,
                                           float* xscale) {
  const int rows = nslots * p.MR;
  for (int idx = threadIdx.x; idx < rows * p.Kgp; idx += kConsumers) {
    const int j = idx / p.Kgp;
    const int g = idx - j * p.Kgp;
    float h[32];
    float mx = 0.0f;
    if (g < p.Kg) {
      const uint4* gs = reinterpret_cast<const uint4*>(p.x + (long long)j * 2 * p.K + (long long)g * 32);
      const uint4* us = reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(gs) + p.K);
      uint4 gv[4], uv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        gv[i] = __ldg(gs + i);
        uv[i] = __ldg(us + i);
      }
      mx = silu_mul_group(gv, uv, h);
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) h[i] = 0.0f;
    }
    store_staged_group_f32(h, mx, xs + (long long)j * 4 * p.Kgp * 16 + g * 16, p.Kgp * 16,
                           xscale + (long long)j * p.Kgp + g, g < p.Kg);
  }
}

__device__ void stage_x(const GemvParams& p, int item0, int nslots, uint8_t* xs, float* xscale) {
  const int rows = nslots * p.MR;
  for (int idx = threadIdx.x; idx < rows * p.Kgp; idx += kConsumers) {
    const int j = idx / p.Kgp;
    const int g = idx - j * p.Kgp;
    const int slot = j / p.MR, m = j - slot * p.MR;
    const int xrow = (p.x_per_item ? (item0 + slot) * p.MR : 0) + m;
    uint4 v[4] = {};
    if (g < p.Kg) {
      const uint4* src =
          reinterpret_cast<const uint4*>(p.x + (long long)xrow * p.K + (long long)g * 32);
#pragma unroll
      for (int i = 0; i < 4; ++i) v[i] = __ldg(src + i);
    }
    store_staged_group(v, xs + (long long)j * 4 * p.Kgp * 16 + g * 16, p.Kgp * 16,
                       xscale + (long long)j * p.Kgp + g, g < p.Kg);
  }
}

// ---------------------------------------------------------------- work walk
// The producer and the consumers of a CTA walk the same sequence of windows
// (item, rows [row0, row0 + nrows), chunks [c0, c1)); each (window, chunk)
// is one tile of the stage ring.
struct Walk {
  long long pos, end;   // next work item, end of the CTA's range
  int item, row0, nrows, c0, c1, rb;

  __device__ void init(const GemvParams& p) {
    pos = (long long)blockIdx.x * p.U / gridDim.x;
    end = (long long)(blockIdx.x + 1) * p.U / gridDim.x;
  }
  __device__ bool next(const GemvParams& p) {
    if (pos >= end) return false;
    if (p.S == 1) {   // rows of the flattened (item, row) space
      const long long r = pos;
      item = (p.n_items == 1) ? 0 : (int)(r / p.N);
      row0 = (int)(r - (long long)item * p.N);
      nrows = (int)min(min((long long)p.RB, end - r), (long long)(p.N - row0));
      c0 = 0;
      c1 = p.nch;
      rb = 0;
      pos += nrows;
    } else {          // (slice, row block) units, slice-major
      const int slice = (int)(pos / p.B);
      rb = (int)(pos - (long long)slice * p.B);
      item = rb / p.upi;
      row0 = (rb - item * p.upi) * p.RB;
      nrows = min(p.RB, p.N - row0);
      c0 = slice * p.cps;
      c1 = min(c0 + p.cps, p.nch);
      pos += 1;
    }
    return true;
  }
};

// Codes and steps of `item` (false: routed id out of range; its rows are left
// unwritten).  The copy warp and the consumers take the same decision for
// every item.
__device__ __forceinline__ bool item_arrays(const GemvParams& p, int item, const uint8_t** q,
                                            const uint8_t** s) {
  long long blk = item;
  if (p.ids != nullptr) {
    const int e = __ldg(p.ids + item);
    if (e < 0 || e >= p.num_experts) return false;
    blk = e;
  }
  *q = p.qw + (unsigned long long)blk * p.qw_item_stride;
  *s = p.st + (unsigned long long)blk * p.st_item_stride;
  return true;
}

// Per-expert output vectors of a window (scale and bias from its first row),
// nullptr when absent: an output is fma(sum, scale, bias) in fp32.
struct OutVec {
  const __nv_bfloat16* s;
  const __nv_bfloat16* b;
};

__device__ __forceinline__ float out_value(const OutVec& o, int r, float v) {
  if (o.s == nullptr && o.b == nullptr) return v;
  const float sc = o.s != nullptr ? __bfloat162float(o.s[r]) : 1.0f;
  const float bi = o.b != nullptr ? __bfloat162float(o.b[r]) : 0.0f;
  return fmaf(v, sc, bi);
}

// Bounded wait on a stage barrier that also gives up once another warp of
// the CTA has aborted.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag != 0) return false;
    if (clock64() - t0 > kWaitCycles) return false;
  }
}

// ---------------------------------------------------------------- producer
// All 32 lanes of the producer warp: request the tile of window wk (its rows,
// chunks [c0, c1)) into the stage at shared address `stage` (generic pointer
// `stage_ptr`).
//  * A window of whole rows (all chunks) is contiguous in memory: one copy
//    for its codes, one for its steps.  A split-K window (a slice of the
//    chunks) takes one copy of each per row.
//  * steps: the 16-byte-aligned superset of the needed bytes, clipped to the
//    item's last full 16-byte line; the bytes past that line (at most 14, at
//    the very end of the item's step array) are stored by hand.  A row's
//    steps start at (row * Kg * 2 + first group * 2) mod 16 in its slot.
__device__ void issue_tile(const GemvParams& p, const Walk& wk, const uint8_t* qwi,
                           const uint8_t* sti, uint32_t stage, uint8_t* stage_ptr, uint32_t full,
                           int lane, uint64_t pol) {
  const int gpc = p.CL * p.T;
  const int gs0 = wk.c0 * gpc;
  const int gs1 = min(wk.c1 * gpc, p.Kg);
  const long long row_code = (long long)p.K / 2, row_st = (long long)p.Kg * 2;
  const uintptr_t sbase = reinterpret_cast<uintptr_t>(sti);
  const uintptr_t st_lim = (sbase + (uintptr_t)((long long)p.N * row_st)) & ~(uintptr_t)15;
  const bool whole = wk.c0 == 0 && wk.c1 == p.nch;
  const int copies = whole ? 1 : wk.nrows;
  const int rows = whole ? wk.nrows : 1;
  uint32_t bytes = 0;
  for (int r = lane; r < copies; r += 32) {
    const long long row = wk.row0 + r;
    bytes += (uint32_t)(rows * (gs1 - gs0) * 16);
    const uintptr_t a0 = sbase + (uintptr_t)(row * row_st + gs0 * 2);
    const uintptr_t e = whole ? sbase + (uintptr_t)((row + rows) * row_st) : a0 + (gs1 - gs0) * 2;
    const uintptr_t a = a0 & ~(uintptr_t)15;
    const uintptr_t b = min((e + 15) & ~(uintptr_t)15, st_lim);
    if (b > a) bytes += (uint32_t)(b - a);
    uint8_t* dst = stage_ptr + p.step_off + (whole ? 0 : r * p.step_pitch);
    for (uintptr_t q = max(a, b); q < e; q += 2)
      *reinterpret_cast<uint16_t*>(dst + (q - a)) = *reinterpret_cast<const uint16_t*>(q);
  }
  bytes = __reduce_add_sync(0xffffffffu, bytes);
  __syncwarp();
  if (lane == 0) mbar_arrive_expect_tx(full, bytes);   // also releases the hand-stored tails
  __syncwarp();
  for (int r = lane; r < copies; r += 32) {
    const long long row = wk.row0 + r;
    const uint8_t* src = qwi + row * row_code + (long long)gs0 * 16;
    bulk_g2s_evict_first(stage + (whole ? 0 : r * p.code_pitch), src,
                         (uint32_t)(rows * (gs1 - gs0) * 16), full, pol);
    const uintptr_t a0 = sbase + (uintptr_t)(row * row_st + gs0 * 2);
    const uintptr_t e = whole ? sbase + (uintptr_t)((row + rows) * row_st) : a0 + (gs1 - gs0) * 2;
    const uintptr_t a = a0 & ~(uintptr_t)15;
    const uintptr_t b = min((e + 15) & ~(uintptr_t)15, st_lim);
    if (b > a)
      bulk_g2s_evict_first(stage + p.step_off + (whole ? 0 : r * p.step_pitch),
                           reinterpret_cast<const void*>(a), (uint32_t)(b - a), full, pol);
  }
}

// ---------------------------------------------------------------- consumers
// Resident CTAs per SM the register budget allows: two (16 warps, 128
// registers a thread) for up to four accumulated (row, activation row)
// pairs, one otherwise.
constexpr int min_ctas(int mr, int rw) { return (mr * rw <= 4) ? 2 : 1; }

// ---------------------------------------------------------------- kernel
// End of a window of whole rows with several chunks, after the consumer
// threads have released its stage: once every warp has stored its chunk sums
// (CTA barrier), each row's are added in chunk order and the row is written.
// The chunk sums have a buffer per stage, and a warp can only write a stage's
// buffer again after every consumer thread has passed the barrier of a later
// window, i.e. has finished reading this one.
template <int MR>
__device__ __forceinline__ void finish_window(const GemvParams& p, const float* redw, int nrows,
                                              int ncw, __nv_bfloat16* yrow, OutVec ov) {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
  for (int i = threadIdx.x; i < nrows * MR; i += kConsumers) {
    const int r = i / MR, m = i - r * MR;
    float v = 0.0f;
    for (int cc = 0; cc < ncw; ++cc) v += redw[(r * p.nch + cc) * MR + m];
    yrow[(long long)m * p.N + r] = __float2bfloat16_rn(out_value(ov, r, v));
  }
}

// WALK kWalkDense: a dense call of whole rows (no routed ids, no split-K).
// Its CTAs walk their rows in windows of RB rows with every offset fixed for
// the launch; the other calls take the general walk (kWalkGeneral), which
// kWalkRealIds extends with the real-id checks and per-expert output vectors
// of w4a16_gemv_id_scaled, and kWalkGated with the gated activation staging
// (W4_FLAG_SILU_MUL).  kWalkRouted is the dense walk for routed calls whose
// windows (within one item) are handed out at run time: each stage also
// names its item, whose output rows (and activation row) the window uses.
constexpr int kWalkGeneral = 0, kWalkDense = 1, kWalkRealIds = 2, kWalkGated = 3,
              kWalkRouted = 4;

template <int MR, int RW, int TT, int CLT, int WALK>
__global__ void __launch_bounds__(kThreads, min_ctas(MR, RW))
    gemv_kernel(const __grid_constant__ GemvParams p) {
  constexpr bool DS = WALK == kWalkDense || WALK == kWalkRouted;
  constexpr bool RDS = WALK == kWalkRouted;
  constexpr bool RID = MR == 1 && WALK == kWalkRealIds;
  constexpr bool GATED = WALK == kWalkGated;   // general walk, gated activations
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t sbase = smem_addr(smem);
  const uint32_t full0 = sbase, empty0 = sbase + 8 * kMaxStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + 16 * kMaxStages);
  volatile int* last_flag = abort_flag + 1;
  volatile int* win = reinterpret_cast<volatile int*>(smem + kWinOff);
  const bool dense = p.ids == nullptr;
  const int nst = p.nst;

  if (threadIdx.x == 0) {
    for (int s = 0; s < nst; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, kConsumerWarps);
    }
    *abort_flag = 0;
    mbar_init_fence();
  }
  __syncthreads();
  pdl_launch_dependents();

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    // Dense weights do not depend on earlier kernels: their tiles are
    // requested at once.  Routed ids may come from the previous kernel,
    // unless the caller says they were final before it (W4_FLAG_IDS_FINAL).
    if (!dense && !p.ids_final) pdl_wait();
    const uint64_t pol = policy_evict_first();
    Walk wk;
    wk.init(p);
    long long issued = 0;
    int slot = 0;
    uint32_t phase = 0;   // use count of the slot, mod 2
    bool ended = false;   // the end of the windows went out in stage `slot`
    if constexpr (WALK == kWalkDense) {
      // Windows of RB rows: the CTA's range in order, or (dyn) window
      // blockIdx.x first, then whichever the launch's counter hands out next.
      // Each stage carries its window's (row0, rows) to the consumers; rows 0
      // tells them there is no more work.
      const long long nwin = (p.U + p.RB - 1) / p.RB;
      long long r0 = wk.pos, w = blockIdx.x;
      int grabbed = 0;      // lane 0: the counter's answer, in flight
      bool pending = false;
      while (true) {
        if (issued >= nst && !wait_phase(empty0 + 8 * slot, phase ^ 1u, abort_flag)) {
          if (*abort_flag == 0) report(p.status, W4_ERR_TIMEOUT);
          *abort_flag = 1;
          break;
        }
        long long row0;
        int nrows;
        if (p.dyn) {
          if (pending) w = (long long)__shfl_sync(0xffffffffu, grabbed, 0) + gridDim.x;
          row0 = w * p.RB;
          nrows = w < nwin ? (int)min((long long)p.RB, p.U - row0) : 0;
        } else {
          row0 = r0;
          nrows = (int)max(0LL, min((long long)p.RB, wk.end - r0));
          r0 += p.RB;
        }
        if (nrows == 0) {
          if (lane == 0) {
            win[2 * slot + 1] = 0;
            mbar_arrive(full0 + 8 * slot);
          }
          ended = true;
          break;
        }
        // the next window's number travels while this tile is requested
        if (p.dyn && lane == 0) grabbed = atomicAdd(p.work, 1);
        pending = p.dyn != 0;
        if (lane == 0) {
          win[2 * slot] = (int)row0;
          win[2 * slot + 1] = nrows;
        }
        Walk cur = wk;
        cur.item = 0;
        cur.row0 = (int)row0;
        cur.nrows = nrows;
        cur.c0 = 0;
        cur.c1 = p.nch;
        cur.rb = 0;
        const uint32_t st_off = kBarBytes + slot * p.tile_bytes;
        issue_tile(p, cur, p.qw, p.st, sbase + st_off, smem + st_off, full0 + 8 * slot, lane, pol);
        ++issued;
        if (++slot == nst) {
          slot = 0;
          phase ^= 1u;
        }
      }
    }
    if (WALK != kWalkDense && p.dyn) {
      // Routed calls of whole rows: windows of RB rows within one item,
      // numbered item-major, window blockIdx.x first, then whichever the
      // launch's counter hands out next.  Each stage carries its window's
      // (row0, rows, item); rows 0 ends the work, negative rows mark an
      // item whose id is out of range (nothing copied, rows left unwritten).
      const int wpi = (p.N + p.RB - 1) / p.RB;
      const long long nwin = (long long)p.n_items * wpi;
      long long w = blockIdx.x;
      int grabbed = 0;
      bool pending = false;
      volatile int* witem = reinterpret_cast<volatile int*>(smem + kItemOff);
      while (true) {
        if (issued >= nst && !wait_phase(empty0 + 8 * slot, phase ^ 1u, abort_flag)) {
          if (*abort_flag == 0) report(p.status, W4_ERR_TIMEOUT);
          *abort_flag = 1;
          break;
        }
        if (pending) w = (long long)__shfl_sync(0xffffffffu, grabbed, 0) + gridDim.x;
        if (w >= nwin) {
          if (lane == 0) {
            win[2 * slot + 1] = 0;
            mbar_arrive(full0 + 8 * slot);
          }
          ended = true;
          break;
        }
        if (lane == 0) grabbed = atomicAdd(p.work, 1);
        pending = true;
        Walk cur = wk;
        cur.item = (int)(w / wpi);
        cur.row0 = (int)(w - (long long)cur.item * wpi) * p.RB;
        cur.nrows = min(p.RB, p.N - cur.row0);
        cur.c0 = 0;
        cur.c1 = p.nch;
        cur.rb = 0;
        const uint8_t *qwi, *sti;
        const bool ok = item_arrays(p, cur.item, &qwi, &sti);
        if (lane == 0) {
          win[2 * slot] = cur.row0;
          win[2 * slot + 1] = ok ? cur.nrows : -cur.nrows;
          witem[slot] = cur.item;
        }
        const uint32_t st_off = kBarBytes + slot * p.tile_bytes;
        if (ok) {
          issue_tile(p, cur, qwi, sti, sbase + st_off, smem + st_off, full0 + 8 * slot, lane, pol);
        } else {
          __syncwarp();
          if (lane == 0) mbar_arrive(full0 + 8 * slot);
        }
        ++issued;
        if (++slot == nst) {
          slot = 0;
          phase ^= 1u;
        }
      }
    }
    while (!DS && !p.dyn && wk.next(p)) {
      const uint8_t *qwi, *sti;
      if (!item_arrays(p, wk.item, &qwi, &sti)) continue;
      // reuse of a slot waits for the consumers to release its last tile
      if (issued >= nst && !wait_phase(empty0 + 8 * slot, phase ^ 1u, abort_flag)) {
        if (*abort_flag == 0) report(p.status, W4_ERR_TIMEOUT);
        *abort_flag = 1;
        break;
      }
      const uint32_t st_off = kBarBytes + slot * p.tile_bytes;
      issue_tile(p, wk, qwi, sti, sbase + st_off, smem + st_off, full0 + 8 * slot, lane, pol);
      ++issued;
      if (++slot == nst) {
        slot = 0;
        phase ^= 1u;
      }
    }
    // Every tile of this CTA is requested: its share of the caller's L2
    // ranges (the next call's weights) goes out now, behind them.
    if (p.l2.n > 0 && *abort_flag == 0) l2_prefetch_share(p.l2, blockIdx.x, gridDim.x, lane);
    // Let the last copies land before the CTA may leave.  When the end went
    // out in stage `slot`, that stage's previous tile had been released by
    // the consumers (its barrier has moved on since): it is not waited for.
    const int inflight = ended ? nst - 1 : nst;
    const int last = issued < inflight ? (int)issued : inflight;
    for (int i = 1; i <= last; ++i) {
      const int sl = slot - i < 0 ? slot - i + nst : slot - i;
      const uint32_t ph = slot - i < 0 ? phase ^ 1u : phase;
      if (!mbar_wait_bounded(full0 + 8 * sl, ph, kWaitCycles)) {
        report(p.status, W4_ERR_TIMEOUT);
        break;
      }
    }
    // dyn: the last CTA to finish re-arms the launch's counters (every CTA
    // has taken its last window before it counts itself done)
    if (p.dyn && lane == 0) {
      __threadfence();
      if (atomicAdd(p.work + 1, 1) == (int)gridDim.x - 1) {
        __threadfence();
        atomicExch(p.work, 0);
        atomicExch(p.work + 1, 0);
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int T = TT > 0 ? TT : p.T;
  const int nsw = 32 / T;
  const int set = lane / T;          // row set of this lane within the warp
  const int t = lane - set * T;      // lane within the row's team

  // items whose activation rows this CTA needs
  int item0 = 0, nslots = 1;
  if (p.x_per_item && p.dyn) {
    nslots = p.n_items;   // run-time windows may come from any item
  } else if (p.x_per_item) {
    Walk r;
    r.init(p);
    if (p.S == 1) {
      item0 = (int)(r.pos / p.N);
      nslots = (r.end > r.pos) ? (int)((r.end - 1) / p.N) - item0 + 1 : 1;
    } else {
      const int rb_lo = (int)(r.pos % p.B), rb_hi = (int)((r.end - 1) % p.B);
      if (r.end - r.pos >= p.B || rb_lo > rb_hi) {
        nslots = p.n_items;
      } else {
        item0 = rb_lo / p.upi;
        nslots = rb_hi / p.upi - item0 + 1;
      }
    }
  }
  const uint32_t xs_off = kBarBytes + nst * p.tile_bytes;
  const uint32_t xsc_off = xs_off + (uint32_t)(p.x_slots * MR * 4 * p.Kgp * 16);
  float* red = reinterpret_cast<float*>(smem + xsc_off + p.x_slots * MR * p.Kgp * 4);
  pdl_wait();   // activations and outputs follow earlier kernels
  if constexpr (GATED)
    stage_x_gated(p, nslots, smem + xs_off, reinterpret_cast<float*>(smem + xsc_off));
  else
    stage_x(p, item0, nslots, smem + xs_off, reinterpret_cast<float*>(smem + xsc_off));
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");

  const int xplane = p.Kgp * 16, xmrow = 4 * p.Kgp * 16, xsmrow = p.Kgp * 4;
  const int kg_valid = p.Kgp != p.Kg ? p.Kg : 0x7fffffff;   // groups past it are padding
  const int gpc = p.CL * T;                  // groups per chunk
  const int kg2 = p.Kg * 2;
  const int rstep = nsw * RW;                // rows of one item
  const int nrs_full = p.RB / rstep;         // row steps of a full window
  const bool steps_aligned = (kg2 & 15) == 0;
  uint32_t lane_c[RW], lane_s[RW];           // lane offsets within a whole-row tile
#pragma unroll
  for (int j = 0; j < RW; ++j) {
    lane_c[j] = (uint32_t)((j * nsw + set) * p.code_pitch + t * 16);
    lane_s[j] = (uint32_t)(p.step_off + (j * nsw + set) * kg2 + t * 2);
  }
  Walk wk;
  wk.init(p);
  int slot = 0;
  uint32_t phase = 0;
  uint32_t tile = kBarBytes;   // shared offset of the current slot
  const int red_slot = p.RB * p.nch * MR;   // chunk sums of one stage's window

  if constexpr (DS) {
    // Each stage brings a window of whole rows (the copy warp's choice, up
    // to RB rows; none: no more work).  Rows of a short window past its end
    // read stale bytes of the stage (in bounds) and are dropped.
    // Every window is walked as a full one: item it = ci * nrs_full + rs
    // (chunk ci, row step rs); a warp takes items warp, warp + 7, ..., its
    // (chunk, row step) stepping by a fixed increment.
    const int ncw = p.nch;
    const int items = ncw * nrs_full;
    const int ci_first = warp / nrs_full, rs_first = warp - ci_first * nrs_full;
    const int dci = kConsumerWarps / nrs_full, drs = kConsumerWarps - dci * nrs_full;
    // routed calls (run-time windows within one item): the item's output
    // rows and, with one activation row per item, its staged row
    volatile int* witem = reinterpret_cast<volatile int*>(smem + kItemOff);
    bool reported = false;
    while (true) {
      if (!wait_phase(full0 + 8 * slot, phase, abort_flag)) {
        if (*abort_flag == 0) report(p.status, W4_ERR_TIMEOUT);
        *abort_flag = 1;
        return;
      }
      const int row0 = win[2 * slot];
      const int nrows = win[2 * slot + 1];
      if (nrows == 0) break;
      const int item = RDS ? witem[slot] : 0;
      if (RDS && nrows < 0) {   // an id out of range: rows left unwritten, stage handed back
        if (!reported && lane == 0) report(p.status, W4_ERR_INDEX);
        reported = true;
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * slot);
        if (++slot == nst) {
          slot = 0;
          phase ^= 1u;
          tile = kBarBytes;
        } else {
          tile += p.tile_bytes;
        }
        continue;
      }
      __nv_bfloat16* yrow = p.y + (long long)item * MR * p.N + row0;
      const int xslot = RDS && p.x_per_item ? item : 0;
      const uint32_t xo0 = xs_off + (uint32_t)(xslot * MR * 4 * p.Kgp * 16);
      const uint32_t xso0 = xsc_off + (uint32_t)(xslot * MR * p.Kgp * 4);
      const uint32_t soff0 = steps_aligned ? 0u : (uint32_t)(((row0 & 7) * (kg2 & 15)) & 15);
      float* redw = red + slot * red_slot;
      int ci = ci_first, rs = rs_first;
      for (int it = warp; it < items; it += kConsumerWarps) {
        const uint32_t ic = tile + (uint32_t)(rs * rstep * p.code_pitch + ci * gpc * 16);
        const uint32_t is = tile + soff0 + (uint32_t)(rs * rstep * kg2 + ci * gpc * 2);
        uint32_t co[RW], so[RW];
#pragma unroll
        for (int j = 0; j < RW; ++j) {
          co[j] = ic + lane_c[j];
          so[j] = is + lane_s[j];
        }
        const int g0 = ci * gpc + t;
        const int ns = CLT > 0 ? CLT : min(p.CL, p.NI - ci * p.CL);
        float acc[RW][MR];
        tile_dot<MR, RW, TT, CLT>(smem, xo0 + (uint32_t)(g0 * 16), xso0 + (uint32_t)(g0 * 4),
                                  xplane, xmrow, xsmrow, co, so, ns, T, kg_valid - g0, acc);
#pragma unroll
        for (int j = 0; j < RW; ++j)
#pragma unroll
          for (int m = 0; m < MR; ++m) acc[j][m] = team_sum<TT>(acc[j][m], T);
        if (t == 0) {
#pragma unroll
          for (int j = 0; j < RW; ++j) {
            const int rl = rs * rstep + j * nsw + set;
            if (rl >= nrows) continue;
            if (ncw == 1) {   // one chunk: the row is done (0 + chunk sum)
#pragma unroll
              for (int m = 0; m < MR; ++m)
                yrow[(long long)m * p.N + rl] = __float2bfloat16_rn(0.0f + acc[j][m]);
            } else {
#pragma unroll
              for (int m = 0; m < MR; ++m) redw[(rl * p.nch + ci) * MR + m] = acc[j][m];
            }
          }
        }
        ci += dci;
        rs += drs;
        if (rs >= nrs_full) {
          rs -= nrs_full;
          ++ci;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * slot);   // this warp is done with the stage
      if (++slot == nst) {
        slot = 0;
        phase ^= 1u;
        tile = kBarBytes;
      } else {
        tile += p.tile_bytes;
      }
      if (ncw > 1) finish_window<MR>(p, redw, nrows, ncw, yrow, OutVec{nullptr, nullptr});
    }
    return;
  } else {
    bool reported = false;
    volatile int* witem = reinterpret_cast<volatile int*>(smem + kItemOff);
    while (true) {
      const uint8_t *qwi, *sti;
      bool bad = false;
      if (p.dyn) {
        // routed run-time windows: the stage says which (rows 0: no more)
        if (!wait_phase(full0 + 8 * slot, phase, abort_flag)) {
          if (*abort_flag == 0) report(p.status, W4_ERR_TIMEOUT);
          *abort_flag = 1;
          return;
        }
        const int nr = win[2 * slot + 1];
        if (nr == 0) break;
        wk.item = witem[slot];
        wk.row0 = win[2 * slot];
        wk.nrows = nr < 0 ? -nr : nr;
        wk.c0 = 0;
        wk.c1 = p.nch;
        wk.rb = 0;
        bad = nr < 0;
      } else if (!wk.next(p)) {
        break;
      }
      int rid = 0;   // real expert id (RID), loaded together with the routed id
      if constexpr (RID) rid = __ldg(p.eids + wk.item);
      if (bad || (!p.dyn && !dense && !item_arrays(p, wk.item, &qwi, &sti))) {
        if (!reported && lane == 0) report(p.status, W4_ERR_INDEX);
        reported = true;
        if (bad) {   // its stage carried nothing: hand it back
          __syncwarp();
          if (lane == 0) mbar_arrive(empty0 + 8 * slot);
          if (++slot == nst) {
            slot = 0;
            phase ^= 1u;
            tile = kBarBytes;
          } else {
            tile += p.tile_bytes;
          }
        }
        continue;
      }
      // Real expert ids: a real id out of range (W4_ERR_INDEX) or a slot that
      // does not hold that expert (W4_ERR_OWNER) keeps the window's rows
      // unwritten; its tile is still read and released as usual.  The checks
      // are taken at the stores, so their loads (and those of the output
      // vectors, from a clamped row) overlap the dot product.
      OutVec ov = {nullptr, nullptr};
      int wcode = W4_OK;
      if constexpr (RID) {
        const bool in_range = rid >= 0 && rid < p.num_real;
        const int holder = p.slot_expert != nullptr ? __ldg(p.slot_expert + __ldg(p.ids + wk.item))
                                                    : rid;
        const long long rr = in_range ? rid : 0;
        if (p.escale != nullptr) ov.s = p.escale + rr * p.N + wk.row0;
        if (p.ebias != nullptr) ov.b = p.ebias + rr * p.N + wk.row0;
        wcode = !in_range ? W4_ERR_INDEX : (holder != rid ? W4_ERR_OWNER : W4_OK);
      }
      const int xslot = p.x_per_item ? wk.item - item0 : 0;
      const bool whole = p.S == 1;
      const bool full = wk.nrows == p.RB;
      // full windows of whole rows whose steps start on 16-byte lines: every
      // offset below is a lane constant plus a per-item term
      const bool fast = whole && full && steps_aligned;
      const int ncw = wk.c1 - wk.c0;                       // chunks in the window
      const int nrs = full ? nrs_full : (wk.nrows + rstep - 1) / rstep;   // row steps
      const int items = ncw * nrs;
      const int soff0 = whole ? (((wk.row0 & 7) * (kg2 & 15)) & 15) : 0;
      float* redw = red + slot * red_slot;
      __nv_bfloat16* yrow = p.y + (long long)wk.item * MR * p.N + wk.row0;
      const uint32_t xo0 = xs_off + (uint32_t)(xslot * MR * 4 * p.Kgp * 16);
      const uint32_t xso0 = xsc_off + (uint32_t)(xslot * MR * p.Kgp * 4);

      if (!p.dyn && !wait_phase(full0 + 8 * slot, phase, abort_flag)) {
        if (*abort_flag == 0) report(p.status, W4_ERR_TIMEOUT);
        *abort_flag = 1;
        return;
      }
      for (int it = warp; it < items; it += kConsumerWarps) {
        // item = (chunk ci of the window, row step rs), it = ci * nrs + rs
        int ci, rs;
        if (nrs == 1) {
          ci = it;
          rs = 0;
        } else if (ncw == 1) {
          ci = 0;
          rs = it;
        } else {
          ci = it / nrs;
          rs = it - ci * nrs;
        }
        const int c = wk.c0 + ci;
        uint32_t co[RW], so[RW];
        int rl[RW];
        bool rv[RW];
        if (fast) {
          const uint32_t ic = tile + (uint32_t)(rs * rstep * p.code_pitch + ci * gpc * 16);
          const uint32_t is = tile + (uint32_t)(rs * rstep * kg2 + ci * gpc * 2);
#pragma unroll
          for (int j = 0; j < RW; ++j) {
            rv[j] = true;
            rl[j] = rs * rstep + j * nsw + set;
            co[j] = ic + lane_c[j];
            so[j] = is + lane_s[j];
          }
        } else {
#pragma unroll
          for (int j = 0; j < RW; ++j) {
            // rows past the window read the window's last row (results dropped)
            const int r = rs * rstep + j * nsw + set;
            rv[j] = r < wk.nrows;
            rl[j] = rv[j] ? r : wk.nrows - 1;
            co[j] = tile + rl[j] * p.code_pitch + (ci * gpc + t) * 16;
            so[j] = tile + p.step_off + (ci * gpc + t) * 2 +
                    (whole ? soff0 + rl[j] * kg2
                           : rl[j] * p.step_pitch +
                                 ((((wk.row0 + rl[j]) & 7) * (kg2 & 15) + wk.c0 * gpc * 2) & 15));
          }
        }
        const int g0 = c * gpc + t;
        const int ns = CLT > 0 ? CLT : min(p.CL, p.NI - c * p.CL);
        // Rows finished by this item (one chunk) of a call with per-expert
        // vectors: their scale and bias are fetched now, so that the loads'
        // latency hides behind the dot product.
        const bool epi = RID && ncw == 1 && t == 0 && (ov.s != nullptr || ov.b != nullptr);
        float osc[RW], obi[RW];
#pragma unroll
        for (int j = 0; j < RW; ++j) {
          osc[j] = 1.0f;
          obi[j] = 0.0f;
          if (epi && rv[j]) {
            if (ov.s != nullptr) osc[j] = __bfloat162float(__ldg(ov.s + rl[j]));
            if (ov.b != nullptr) obi[j] = __bfloat162float(__ldg(ov.b + rl[j]));
          }
        }
        float acc[RW][MR];
        tile_dot<MR, RW, TT, CLT>(smem, xo0 + (uint32_t)(g0 * 16), xso0 + (uint32_t)(g0 * 4), xplane,
                                  xmrow, xsmrow, co, so, ns, T, kg_valid - g0, acc);
#pragma unroll
        for (int j = 0; j < RW; ++j)
#pragma unroll
          for (int m = 0; m < MR; ++m) acc[j][m] = team_sum<TT>(acc[j][m], T);
        if (t == 0) {
#pragma unroll
          for (int j = 0; j < RW; ++j) {
            if (!rv[j] || wcode != W4_OK) continue;
            if (!whole) {          // split-K: chunk sums to the workspace
              float* dst = p.ws_partial + (((long long)wk.rb * p.nch + c) * p.RB + rl[j]) * MR;
#pragma unroll
              for (int m = 0; m < MR; ++m) dst[m] = acc[j][m];
            } else if (ncw == 1) { // one chunk: the row is done (0 + chunk sum)
#pragma unroll
              for (int m = 0; m < MR; ++m)
                yrow[(long long)m * p.N + rl[j]] = __float2bfloat16_rn(
                    epi ? fmaf(0.0f + acc[j][m], osc[j], obi[j]) : 0.0f + acc[j][m]);
            } else {
#pragma unroll
              for (int m = 0; m < MR; ++m) redw[(rl[j] * p.nch + ci) * MR + m] = acc[j][m];
            }
          }
        }
      }
      __syncwarp();

      if (whole) {
        if (lane == 0) mbar_arrive(empty0 + 8 * slot);   // this warp is done with the stage
        if (++slot == nst) {
          slot = 0;
          phase ^= 1u;
          tile = kBarBytes;
        } else {
          tile += p.tile_bytes;
        }
        if (RID && wcode != W4_OK) {
          if (!reported && lane == 0) report(p.status, wcode);
          reported = true;
        }
        if (ncw > 1) finish_window<MR>(p, redw, wcode == W4_OK ? wk.nrows : 0, ncw, yrow, ov);
        continue;
      }
      if (lane == 0) mbar_arrive(empty0 + 8 * slot);
      if (++slot == nst) {
        slot = 0;
        phase ^= 1u;
        tile = kBarBytes;
      } else {
        tile += p.tile_bytes;
      }
      // Split-K: the last of the slices to finish this row block adds the chunk
      // sums in chunk order, writes the rows and re-arms the counter.  The CTA
      // barrier orders every thread's partial stores before thread 0's counter
      // update, whose release publishes them at GPU scope; its acquire side,
      // then the second barrier, order the other slices' partials before this
      // CTA reads them.
      asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
      if (threadIdx.x == 0)
        *last_flag = atomic_add_acq_rel_gpu(p.ws_count + wk.rb, 1) == p.S - 1;
      asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
      if (*last_flag) {
        for (int i = threadIdx.x; i < wk.nrows * MR; i += kConsumers) {
          const int r = i / MR, m = i - r * MR;
          const float* src = p.ws_partial + ((long long)wk.rb * p.nch * p.RB + r) * MR + m;
          float v = 0.0f;
          for (int cc = 0; cc < p.nch; ++cc) v += __ldcg(src + (long long)cc * p.RB * MR);
          yrow[(long long)m * p.N + r] = __float2bfloat16_rn(v);
        }
        if (threadIdx.x == 0) atomicExch(p.ws_count + wk.rb, 0);
      }
    }
  }
}

// ================================================================= host side
// Host helpers shared with the chain launches (declared in gemv_host.h).
constexpr long long kRowStepMax = 40 << 10;  // largest step of whole rows

DeviceInfo device_info(int dev) {
  static std::mutex mu;
  static DeviceInfo cache[64];
  std::lock_guard<std::mutex> lock(mu);
  if (dev < 0 || dev >= 64) return DeviceInfo{};
  if (cache[dev].sms == 0) {
    int sms = 0, optin = 0, per_sm = 0, reserved = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) !=
            cudaSuccess) {
      cudaGetLastError();
      return DeviceInfo{};
    }
    cache[dev].dev = dev;
    cache[dev].sms = sms;
    cache[dev].smem_optin = optin;
    cache[dev].smem_per_sm = per_sm;
    cache[dev].smem_reserved = reserved;
  }
  return cache[dev];
}

// The per-row arithmetic comes from K alone.  T: the largest power of two
// <= 32 dividing K/32 that leaves each lane >= 4 groups of a row (else the
// largest dividing one).  CL, groups per lane per chunk: all of the lane's
// groups when they are <= 4, else 4 or 3 when that divides them, else all of
// them up to 12, else 4 (the last chunk shorter).
void row_shape(int K, int* T, int* NI, int* CL, int* nch) {
  const int Kg = K / 32;
  int t = 1;
  while (t < 32 && Kg % (2 * t) == 0 && Kg / (2 * t) >= 4) t *= 2;
  if (Kg / t < 4) {   // short rows: the largest power of two that divides
    t = 1;
    while (t < 32 && Kg % (2 * t) == 0) t *= 2;
  }
  // A step of 32 / t whole rows must fit a stage; otherwise a team of up to
  // 32 lanes walks the row with the last groups padded.
  if ((long long)(32 / t) * (K / 2 + Kg * 2) > kRowStepMax) {
    t = 32;
    while (t > 1 && (Kg + t - 1) / t < 4) t /= 2;
  }
  *T = t;
  const int ni = (Kg + t - 1) / t;
  int cl = 4;
  if (ni <= 4) cl = ni;
  else if (ni % 4 == 0) cl = 4;
  else if (ni % 3 == 0) cl = 3;
  else if (ni <= 12) cl = ni;   // 5, 7, 10, 11: one chunk
  *NI = ni;
  *CL = cl;
  *nch = (ni + cl - 1) / cl;
}

// Stage geometry of a window of `rb` rows: whole rows (contiguous codes, then
// the steps' 16-byte superset), or `cps` chunks of each row (split-K: one
// slot per row for codes and for steps).
void tile_geometry(int K, int T, int CL, bool whole, int cps, int rb, int* code_pitch,
                   int* step_pitch, int* step_off, int* tile_bytes) {
  const int Kg = K / 32;
  const int pad = T - 1;   // padding groups a lane may read past a row's end
  *code_pitch = whole ? K / 2 : cps * CL * T * 16;
  *step_pitch = whole ? Kg * 2 : ((cps * CL * T * 2 + 30 + 15) & ~15);
  *step_off = rb * *code_pitch + pad * 16;
  const long long steps =
      whole ? (long long)rb * Kg * 2 + 32 + pad * 2 : (long long)rb * *step_pitch;
  *tile_bytes = (int)((*step_off + steps + 127) & ~127LL);
}

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
    di->smem_per_sm = 233472;
    di->smem_reserved = 1024;
  }
}

namespace {


struct Plan {
  bool routed = false;   // routed-expert call (ids), never split
  bool dyn = false;      // dense whole rows: windows handed out at run time
  int MR = 1;
  int Kg = 1;
  int T = 32, nsw = 1, NI = 1, CL = 1, nch = 1;
  int RW = 1, RB = 8;
  int S = 1, cps = 1, upi = 1;
  long long B = 0, U = 0;
  int x_slots = 1;
  int nst = 2, per_sm = 1;
  int tile_bytes = 0, code_pitch = 0, step_pitch = 0, step_off = 0;
  int ctas = 0;
  long long smem = 0;
  size_t ws_bytes = 0;
  size_t ws_part_off = 0;
};

constexpr long long kTileMax = 48 << 10;   // largest stage the planner picks
constexpr long long kTileGood = 24 << 10;  // stages this large amortise a window's overhead
constexpr long long kRoutedXMax = 64 << 10;  // staged activation rows of a routed call


long long x_bytes(int slots, int MR, int Kgp) { return (long long)slots * MR * Kgp * (64 + 4); }


// Chunk sums of a window of whole rows, one buffer per stage (none for one
// chunk).
long long red_bytes(int rb, int nch, int MR) { return nch > 1 ? (long long)rb * nch * MR * 4 : 0; }

using KernelFn = void (*)(GemvParams);
int occupancy(const struct Plan& pl, int dev);

bool make_plan(int MR, int N, int K, int n_items, int allow_split, int x_per_item, bool routed,
               const DeviceInfo& di, Plan* out, int force_per_sm = 0) {
  Plan pl;
  pl.routed = routed;
  pl.MR = MR;
  const int Kg = K / 32;
  pl.Kg = Kg;
  row_shape(K, &pl.T, &pl.NI, &pl.CL, &pl.nch);
  pl.nsw = 32 / pl.T;
  const int sms = di.sms > 0 ? di.sms : 1;
  const long long optin = di.smem_optin > 0 ? di.smem_optin : 232448;
  const long long per_sm_smem = di.smem_per_sm > 0 ? di.smem_per_sm : 233472;
  const long long reserved = di.smem_reserved > 0 ? di.smem_reserved : 1024;
  const long long rows_total = (long long)n_items * N;
  if (rows_total > (1LL << 40)) return false;
  const long long weight_bytes = rows_total * ((long long)K / 2 + Kg * 2);
  // Two CTAs per SM for large problems.  For smaller ones, one CTA per SM
  // leaves room for the next launch's CTA to start streaming its weights
  // (W4_FLAG_PDL), two shorten each CTA's share: take two unless that pads
  // the CTAs' last windows more (rows a CTA's windows could hold over the
  // rows it has).
  if (force_per_sm == 0 && weight_bytes < (16LL << 20) && min_ctas(MR, 1) == 2) {
    Plan one, two;
    const bool ok1 = make_plan(MR, N, K, n_items, allow_split, x_per_item, routed, di, &one, 1);
    const bool ok2 = make_plan(MR, N, K, n_items, allow_split, x_per_item, routed, di, &two, 2);
    if (!ok1 || !ok2) {
      if (!ok1 && !ok2) return false;
      *out = ok1 ? one : two;
      return true;
    }
    auto padding = [](const Plan& q) {
      const double rows = (double)q.U / q.ctas;   // rows (or units) per CTA
      const double win = q.S == 1 ? q.RB : 1.0;
      return std::ceil(rows / win) * win / rows;
    };
    *out = (two.per_sm == 2 && padding(two) <= 1.05 * padding(one)) ? two : one;
    return true;
  }
  pl.per_sm = (weight_bytes >= (16LL << 20)) ? min_ctas(MR, 1) : 1;
  if (force_per_sm > 0) pl.per_sm = force_per_sm;
  // shared memory a CTA may take and still leave room for a second one
  const long long half = per_sm_smem / 2 - reserved;
  // fewest rows a CTA should own: enough (row step, chunk) items for its warps
  const long long min_rows =
      std::max<long long>(pl.nsw, ((long long)kConsumerWarps * pl.nsw + pl.nch - 1) / pl.nch);
  const long long target = (long long)pl.per_sm * sms;
  const long long g1 = std::min(target, (rows_total + min_rows - 1) / min_rows);
  int rw_cap = MR == 1 ? 4 : (MR == 2 ? 2 : 1);
  // few rows, long K: split K across CTAs (windows of one row step)
  const long long blocks = (long long)n_items * ((N + pl.nsw - 1) / pl.nsw);
  // chunks per slice: few enough that a window (one row step) fits a stage
  const long long step_chunk = (long long)pl.nsw * pl.CL * pl.T * 18;
  const int cps_max = (int)std::max<long long>(1, kTileMax / step_chunk);
  int split = 1;
  if (allow_split && pl.nch > 1 && 2 * g1 < target) {
    split = (int)std::min<long long>(pl.nch, (target + blocks - 1) / blocks);
    split = std::max(split, (pl.nch + cps_max - 1) / cps_max);
  }
  if (split > 1) {
    pl.RB = pl.nsw;
    pl.upi = (int)((N + pl.RB - 1) / pl.RB);
    pl.B = blocks;
    if (pl.B > (1LL << 30)) return false;
    pl.cps = (pl.nch + split - 1) / split;
    pl.S = (pl.nch + pl.cps - 1) / pl.cps;
    pl.U = (long long)pl.S * pl.B;
    pl.ctas = (int)std::min<long long>(pl.U, target);
    rw_cap = 1;
  } else {
    pl.S = 1;
    pl.cps = pl.nch;
    pl.U = rows_total;
    pl.ctas = (int)std::max<long long>(1, g1);
  }
  // activation rows a CTA stages: one, or the items its range touches; a
  // routed call whose windows are handed out at run time stages every
  // item's row (when they fit kRoutedXMax)
  pl.x_slots = 1;
  const bool routed_dyn_ok =
      routed && pl.S == 1 &&
      (!x_per_item || x_bytes(n_items, MR, pl.NI * pl.T) <= kRoutedXMax);
  if (x_per_item && routed_dyn_ok) {
    pl.x_slots = n_items;
  } else if (x_per_item) {
    for (int c = 0; c < pl.ctas; ++c) {
      const long long ub = (long long)c * pl.U / pl.ctas, ue = (long long)(c + 1) * pl.U / pl.ctas;
      if (ue <= ub) continue;
      long long n;
      if (pl.S == 1) {
        n = (ue - 1) / N - ub / N + 1;
      } else {
        const long long lo = ub % pl.B, hi = (ue - 1) % pl.B;
        n = (ue - ub >= pl.B || lo > hi) ? n_items : hi / pl.upi - lo / pl.upi + 1;
      }
      pl.x_slots = (int)std::max<long long>(pl.x_slots, n);
    }
  }
  const long long xb = x_bytes(pl.x_slots, MR, pl.NI * pl.T);
  // Window shape: RW rows per lane and `rs` row steps per window (whole rows;
  // a split-K window is one row step).  Score: the share of warp slots the
  // window's (row step, chunk) items fill, stages of at least kTileGood
  // bytes, three or more stages, then activation reuse (RW).
  const long long rows_per_cta = (pl.U + pl.ctas - 1) / pl.ctas;
  bool found = false;
  const long long budgets[2] = {half, std::min(optin, per_sm_smem - reserved)};
  for (int bi = 0; bi < 2 && !found; ++bi) {
    double best = 0.0;
    for (int rw = rw_cap; rw >= 1; rw /= 2) {
      for (int rs = 1; rs <= 64; ++rs) {
        const int rb = rs * pl.nsw * rw;
        if (pl.S > 1 && (rs > 1 || rw > 1)) break;
        if (rs > 1 && rb > rows_per_cta) break;
        int cp, sp, so, tb;
        tile_geometry(K, pl.T, pl.CL, pl.S == 1, pl.cps, rb, &cp, &sp, &so, &tb);
        if (rs > 1 && tb > kTileMax) break;
        const long long rd = pl.S == 1 ? red_bytes(rb, pl.nch, MR) : 0;
        const long long room = budgets[bi] - kBarBytes - xb;
        if (room < 2LL * (tb + rd)) break;
        const int nst = (int)std::min<long long>(kMaxStages, room / (tb + rd));
        const long long items = (long long)(pl.S == 1 ? pl.nch : pl.cps) * rs;
        const double util =
            (double)items / (double)(kConsumerWarps * ((items + kConsumerWarps - 1) / kConsumerWarps));
        const double per_warp = (double)items / kConsumerWarps;   // items a warp takes
        const double score = util * std::min(1.0, (double)tb / kTileGood) *
                             (nst >= 3 ? 1.0 : 0.95) * (1.0 - 0.15 / std::max(1.0, per_warp)) *
                             (1.0 + 0.2 * (rw > 1) + 0.2 * (rw > 2));
        if (score > best + 1e-9) {
          best = score;
          pl.RW = rw;
          pl.RB = rb;
          pl.nst = nst;
          pl.code_pitch = cp;
          pl.step_pitch = sp;
          pl.step_off = so;
          pl.tile_bytes = tb;
          found = true;
        }
      }
    }
    if (found && bi == 1 && pl.per_sm > 1)   // only one CTA per SM fits
      return make_plan(MR, N, K, n_items, allow_split, x_per_item, routed, di, out, 1);
  }
  if (!found) return false;
  pl.smem = kBarBytes + (long long)pl.nst * pl.tile_bytes + xb +
            (pl.S == 1 ? pl.nst * red_bytes(pl.RB, pl.nch, MR) : 0);
  // resident CTAs the device really fits (registers, shared memory); fewer
  // than planned: the same work over fewer CTAs
  if (di.dev >= 0) {
    const int occ = occupancy(pl, di.dev);
    if (occ < 1) return false;
    if (occ < pl.per_sm)
      return make_plan(MR, N, K, n_items, allow_split, x_per_item, routed, di, out, occ);
  }
  // Dense whole-row launches with several windows per CTA take them from a
  // counter at run time: SMs stream at different speeds, and a fixed share of
  // rows per CTA would make the launch wait for the slowest.
  if (!routed && pl.S == 1) pl.dyn = (pl.U + pl.RB - 1) / pl.RB >= 4LL * pl.ctas;
  // Routed calls take windows of RB rows within one item; at run time too
  // once there are enough of them.
  if (routed_dyn_ok)
    pl.dyn = (long long)n_items * ((N + pl.RB - 1) / pl.RB) >= 2LL * pl.ctas;
  if (pl.S > 1) {
    // counters first, partials after them
    const size_t part = (size_t)pl.B * pl.nch * pl.RB * MR * sizeof(float);
    pl.ws_part_off = ((size_t)pl.B * sizeof(int) + 255) & ~size_t(255);
    pl.ws_bytes = pl.ws_part_off + part;
  }
  *out = pl;
  return true;
}

using KernelFn = void (*)(GemvParams);

// The instantiation that runs a plan: batch-1 plans whose chunks are all full
// get one compiled for their team size and chunk length (the common K);
// everything else the generic one.  *tt, *clt (if given) receive the
// compile-time team size and chunk length (0: generic).
// The instantiation that runs a plan.  Calls with real expert ids
// (w4a16_gemv_id_scaled) take their own kernels: the checks and output
// vectors stay out of every other launch.
KernelFn kernel_for(const Plan& pl, bool real_ids = false, int* tt = nullptr, int* clt = nullptr,
                    bool gated = false) {
  if (tt != nullptr) *tt = 0;
  if (clt != nullptr) *clt = 0;
  if (gated) {   // dense calls with gated activations: generic instantiations
    switch (pl.MR * 8 + pl.RW) {
      case 8 + 1: return gemv_kernel<1, 1, 0, 0, kWalkGated>;
      case 8 + 2: return gemv_kernel<1, 2, 0, 0, kWalkGated>;
      case 8 + 4: return gemv_kernel<1, 4, 0, 0, kWalkGated>;
      case 16 + 1: return gemv_kernel<2, 1, 0, 0, kWalkGated>;
      case 16 + 2: return gemv_kernel<2, 2, 0, 0, kWalkGated>;
      case 24 + 1: return gemv_kernel<3, 1, 0, 0, kWalkGated>;
      case 32 + 1: return gemv_kernel<4, 1, 0, 0, kWalkGated>;
      default: return nullptr;
    }
  }
  // the dense walk: dense calls of whole rows, and (its routed form) routed
  // calls whose windows within one item are handed out at run time
  const bool ds = !pl.routed && pl.S == 1;
  const bool rds = pl.routed && pl.dyn && pl.S == 1;
  const bool full = pl.NI % pl.CL == 0 && pl.NI * pl.T == pl.Kg;
  const int key = pl.T * 16 + pl.CL;
  if (real_ids) {
    if (pl.MR != 1) return nullptr;
#define W4_RID(t, cl)                                                                   \
  if (full && pl.RW <= 2 && key == (t) * 16 + (cl)) {                                   \
    if (tt != nullptr) *tt = t;                                                         \
    if (clt != nullptr) *clt = cl;                                                      \
    return pl.RW == 1 ? gemv_kernel<1, 1, t, cl, kWalkRealIds>                          \
                      : gemv_kernel<1, 2, t, cl, kWalkRealIds>;                         \
  }
    W4_RID(8, 11)   // K = 2816
    W4_RID(2, 11)   // K = 704
#undef W4_RID
    switch (pl.RW) {
      case 1: return gemv_kernel<1, 1, 0, 0, kWalkRealIds>;
      case 2: return gemv_kernel<1, 2, 0, 0, kWalkRealIds>;
      case 4: return gemv_kernel<1, 4, 0, 0, kWalkRealIds>;
      default: return nullptr;
    }
  }
  if (pl.MR == 1 && full && (pl.RW <= 2 || ((ds || rds) && pl.RW == 4))) {
#define W4_SPEC(t, cl)                                                                  \
  if (key == (t) * 16 + (cl)) {                                                         \
    if (tt != nullptr) *tt = t;                                                         \
    if (clt != nullptr) *clt = cl;                                                      \
    if (rds)                                                                            \
      return pl.RW == 1 ? gemv_kernel<1, 1, t, cl, kWalkRouted>                         \
             : pl.RW == 2 ? gemv_kernel<1, 2, t, cl, kWalkRouted>                       \
                          : gemv_kernel<1, 4, t, cl, kWalkRouted>;                      \
    if (ds && pl.RW == 4) return gemv_kernel<1, 4, t, cl, kWalkDense>;                  \
    if (ds)                                                                             \
      return pl.RW == 1 ? gemv_kernel<1, 1, t, cl, kWalkDense>                          \
                        : gemv_kernel<1, 2, t, cl, kWalkDense>;                         \
    return pl.RW == 1 ? gemv_kernel<1, 1, t, cl, kWalkGeneral>                          \
                      : gemv_kernel<1, 2, t, cl, kWalkGeneral>;                         \
  }
    W4_SPEC(16, 4)   // K = 2048
    W4_SPEC(8, 3)    // K = 5376
    W4_SPEC(32, 3)   // K = 21504
    W4_SPEC(32, 4)   // K = 4096 * n
    W4_SPEC(8, 11)   // K = 2816
    W4_SPEC(2, 11)   // K = 704
#undef W4_SPEC
  }
#define W4_GEN(mr, rw) \
  (ds ? gemv_kernel<mr, rw, 0, 0, kWalkDense> : gemv_kernel<mr, rw, 0, 0, kWalkGeneral>)
  if (rds) {
    switch (pl.RW) {
      case 1: return gemv_kernel<1, 1, 0, 0, kWalkRouted>;
      case 2: return gemv_kernel<1, 2, 0, 0, kWalkRouted>;
      case 4: return gemv_kernel<1, 4, 0, 0, kWalkRouted>;
      default: return nullptr;
    }
  }
  switch (pl.MR * 8 + pl.RW) {
    case 8 + 1: return W4_GEN(1, 1);
    case 8 + 2: return W4_GEN(1, 2);
    case 8 + 4: return W4_GEN(1, 4);
    case 16 + 1: return W4_GEN(2, 1);
    case 16 + 2: return gemv_kernel<2, 2, 0, 0, kWalkDense>;   // whole rows only (RW > 1)
    case 24 + 1: return W4_GEN(3, 1);
    case 32 + 1: return W4_GEN(4, 1);
    default: return nullptr;
  }
#undef W4_GEN
}

// Raise `fn`'s dynamic shared-memory limit on `dev` (current) to at least
// `smem` bytes.
cudaError_t allow_smem(KernelFn fn, long long smem, int dev) {
  struct Entry {
    KernelFn fn;
    int dev;
    long long bytes;
  };
  static std::mutex mu;
  static Entry seen[256];
  static int used = 0;
  std::lock_guard<std::mutex> lock(mu);
  Entry* e = nullptr;
  for (int i = 0; i < used; ++i)
    if (seen[i].fn == fn && seen[i].dev == dev) e = &seen[i];
  if (e != nullptr && e->bytes >= smem) return cudaSuccess;
  const cudaError_t r =
      cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (r != cudaSuccess) return r;
  if (e == nullptr && used < 256) e = &seen[used++];
  if (e != nullptr) *e = Entry{fn, dev, smem};
  return cudaSuccess;
}

// Resident CTAs per SM of the plan's instantiation (0: not launchable).
int occupancy(const Plan& pl, int dev) {
  const KernelFn fn = kernel_for(pl);
  int n = 0;
  if (fn == nullptr || allow_smem(fn, pl.smem, dev) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kThreads, (size_t)pl.smem) !=
          cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

// The next window-counter slot of device `dev` (current).
cudaError_t work_slot(int dev, int** out) {
  static std::mutex mu;
  static int* base[64] = {};
  static unsigned next[64] = {};
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (base[dev] == nullptr) {
    void* a = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&a, w4_window_counters);
    if (e != cudaSuccess) return e;
    base[dev] = static_cast<int*>(a);
  }
  *out = base[dev] + 16 * (next[dev]++ % kWorkSlots);
  return cudaSuccess;
}

cudaError_t launch(const GemvParams& prm, const Plan& pl, bool pdl, cudaStream_t stream, int dev) {
  const KernelFn fn = kernel_for(pl, prm.eids != nullptr, nullptr, nullptr, prm.gated != 0);
  if (fn == nullptr) return cudaErrorInvalidConfiguration;
  const cudaError_t ea = allow_smem(fn, pl.smem, dev);
  if (ea != cudaSuccess) return ea;
  GemvParams p = prm;
  if (pl.dyn && !prm.gated) {   // run-time windows: the dense walk only
    const cudaError_t ew = work_slot(dev, &p.work);
    if (ew != cudaSuccess) return ew;
    p.dyn = 1;
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
  return cudaLaunchKernelEx(&cfg, fn, p);
}

GemvParams base_params(const Plan& pl, int N, int K) {
  GemvParams p = {};
  p.N = N;
  p.K = K;
  p.Kg = K / 32;
  p.Kgp = pl.NI * pl.T;
  p.MR = pl.MR;
  p.T = pl.T;
  p.nsw = pl.nsw;
  p.NI = pl.NI;
  p.CL = pl.CL;
  p.nch = pl.nch;
  p.RB = pl.RB;
  p.S = pl.S;
  p.cps = pl.cps;
  p.upi = pl.upi;
  p.B = (int)pl.B;
  p.U = pl.U;
  p.x_slots = pl.x_slots;
  p.nst = pl.nst;
  p.tile_bytes = pl.tile_bytes;
  p.code_pitch = pl.code_pitch;
  p.step_pitch = pl.step_pitch;
  p.step_off = pl.step_off;
  return p;
}

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }


// Plans are cached per shape: planning is cheap but not free, and decode
// loops call the same few shapes over and over.
struct PlanKey {
  int MR, N, K, n_items, split, xpi, sms;
  bool routed;
  bool operator==(const PlanKey& o) const {
    return MR == o.MR && N == o.N && K == o.K && n_items == o.n_items && split == o.split &&
           xpi == o.xpi && sms == o.sms && routed == o.routed;
  }
};

bool cached_plan(int MR, int N, int K, int n_items, int split, int xpi, bool routed,
                 const DeviceInfo& di, Plan* out) {
  static std::mutex mu;
  static PlanKey keys[256];
  static Plan plans[256];
  static int used = 0, next = 0;
  const PlanKey k{MR, N, K, n_items, split, xpi, di.sms, routed};
  {
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i)
      if (keys[i] == k) {
        *out = plans[i];
        return true;
      }
  }
  if (!make_plan(MR, N, K, n_items, split, xpi, routed, di, out)) return false;
  std::lock_guard<std::mutex> lock(mu);
  keys[next] = k;
  plans[next] = *out;
  next = (next + 1) % 256;
  used = std::min(used + 1, 256);
  return true;
}

// Activation rows per launch: up to kMaxMR, as many as fit shared memory
// next to two stages of one row per lane.
int max_rows_per_launch(int K, const DeviceInfo& di) {
  const long long optin = di.smem_optin > 0 ? di.smem_optin : 232448;
  int T, NI, CL, nch, cp, sp, so, tb;
  row_shape(K, &T, &NI, &CL, &nch);
  tile_geometry(K, T, CL, true, nch, 32 / T, &cp, &sp, &so, &tb);
  int mr = kMaxMR;
  while (mr > 0 &&
         kBarBytes + 2LL * (tb + red_bytes(32 / T, nch, mr)) + x_bytes(1, mr, NI * T) > optin)
    --mr;
  return mr;
}

// Batches that use the tensor-core path (K a multiple of 256): from 5
// activation rows always (the CUDA cores take a second launch there), at 4
// rows for weights of 2^24 codes or more and at 3 rows from 2^27 (measured
// crossovers: at 4 rows 16384 x 2048 takes 13.3 us on the tensor cores
// against 14.6 on the CUDA cores, 3072 x 2048 7.2 against 5.7; at 3 rows
// 43008 x 5376 44.5 against 67.0, 9472 x 5376 20.4 against 18.9).
bool tc_rows(int M, int N, int K) {
  const long long codes = (long long)N * K;
  return M >= 5 || (M == 4 && codes >= (1LL << 24)) || (M == 3 && codes >= (1LL << 27));
}
constexpr unsigned kPathFlags = W4_FLAG_CUDA_CORES | W4_FLAG_TENSOR_CORES;

bool tc_shape(int K) { return K >= 256 && K % 256 == 0; }

// 1: tensor-core path, 0: CUDA-core path, -1: the flags ask for a path that
// cannot run this shape (or for both paths).
int path_of(int M, int N, int K, unsigned flags) {
  if ((flags & kPathFlags) == kPathFlags) return -1;
  if (flags & W4_FLAG_SILU_MUL) return (flags & W4_FLAG_TENSOR_CORES) ? -1 : 0;   // CUDA cores
  if (flags & W4_FLAG_CUDA_CORES) return 0;
  if (flags & W4_FLAG_TENSOR_CORES) return tc_shape(K) ? 1 : -1;
  return (tc_rows(M, N, K) && tc_shape(K)) ? 1 : 0;
}

// Largest workspace of the tensor-core launches of an (M, N, K) call: with
// allow_sk the size that lets every launch take balanced runs, without it
// the size the call cannot run without (split-K).
size_t tc_workspace(int M, int N, int K, int sms, bool allow_sk = true) {
  tc::TpPlan pp;
  if (M > tc::kTcMaxM && tc::tp_plan(M, N, K, sms, &pp)) return 0;   // one prompt launch
  size_t ws = 0;
  for (int m0 = 0; m0 < M; m0 += tc::kTcMaxM) {
    tc::TcPlan tp;
    if (tc::tc_plan(std::min(tc::kTcMaxM, M - m0), N, K, sms, &tp, allow_sk))
      ws = std::max(ws, tp.ws_bytes);
  }
  return ws;
}

// The plan of one small-batch launch: balanced runs when the workspace
// holds their hand-over slots, else the plain plan (the same bits).
bool tc_launch_plan(int M, int N, int K, int sms, const void* workspace, size_t workspace_bytes,
                    tc::TcPlan* tp) {
  if (!tc::tc_plan(M, N, K, sms, tp)) return false;
  if (tp->sk && (workspace == nullptr || workspace_bytes < tp->ws_bytes || !aligned(workspace, 16)))
    return tc::tc_plan(M, N, K, sms, tp, false);
  return true;
}

// Enqueue the tensor-core launches of a call (up to 32 activation rows each).
w4_status tc_enqueue(void* y, const void* qw, const void* st, const void* x, int M, int N, int K,
                     void* workspace, size_t workspace_bytes, int32_t* status_dev, bool pdl,
                     cudaStream_t s, int dev, int sms, const L2Ranges* l2 = nullptr) {
  // more rows than a small-batch launch takes: one launch of the prompt GEMM
  tc::TpPlan pp;
  if (M > tc::kTcMaxM && tc::tp_plan(M, N, K, sms, &pp)) {
    const cudaError_t e = tc::tp_launch(pp, y, qw, st, x, M, N, K, status_dev, pdl, s, dev);
    if (e != cudaSuccess) {
      note_cuda_error(e);
      cudaGetLastError();
      return W4_ERR_LAUNCH;
    }
    return W4_OK;
  }
  // every launch of the call is checked before the first one is enqueued
  for (int m0 = 0; m0 < M; m0 += tc::kTcMaxM) {
    tc::TcPlan tp;
    if (!tc_launch_plan(std::min(tc::kTcMaxM, M - m0), N, K, sms, workspace, workspace_bytes, &tp))
      return W4_ERR_SHAPE;
    if (tp.ws_bytes > 0 && (workspace == nullptr || workspace_bytes < tp.ws_bytes))
      return W4_ERR_WORKSPACE;
    if (tp.ws_bytes > 0 && !aligned(workspace, 16)) return W4_ERR_ALIGN;
  }
  for (int m0 = 0; m0 < M; m0 += tc::kTcMaxM) {
    const int mr = std::min(tc::kTcMaxM, M - m0);
    tc::TcPlan tp;
    tc_launch_plan(mr, N, K, sms, workspace, workspace_bytes, &tp);
    const cudaError_t e =
        tc::tc_launch(tp, static_cast<__nv_bfloat16*>(y) + (long long)m0 * N, qw, st,
                      static_cast<const __nv_bfloat16*>(x) + (long long)m0 * K, mr, N, K, workspace,
                      status_dev, pdl, s, dev, m0 + mr >= M ? l2 : nullptr);
    if (e != cudaSuccess) {
      note_cuda_error(e);
      cudaGetLastError();
      return W4_ERR_LAUNCH;
    }
  }
  return W4_OK;
}

}  // namespace
}  // namespace w4

// ================================================================= C ABI
using namespace w4;

extern "C" w4_status w4a16_gemv_plan(int M, int N, int K, w4_plan_info* info) {
  return w4a16_gemv_plan_flags(M, N, K, 0, info);
}

extern "C" w4_status w4a16_gemv_plan_flags(int M, int N, int K, unsigned flags,
                                           w4_plan_info* info) {
  if (info == nullptr || M < 1 || N < 1) return W4_ERR_ARG;
  if ((flags & ~(W4_FLAG_PDL | kPathFlags | W4_FLAG_SILU_MUL)) != 0) return W4_ERR_ARG;
  const int fpath = path_of(M, N, K, flags);
  if (fpath < 0) return W4_ERR_SHAPE;
  if (M > W4_MAX_M || K < 32 || K % 32 != 0 || K > W4_MAX_K) return W4_ERR_SHAPE;
  DeviceInfo di;
  planning_device(&di);
  tc::TpPlan pp;
  if (fpath == 1 && M > tc::kTcMaxM && tc::tp_plan(M, N, K, di.sms, &pp)) {
    *info = w4_plan_info{};
    info->path = 3;
    info->ctas = pp.ctas;
    info->slices = 1;
    info->threads = 320;   // 4 unpacking, 4 epilogue, copy and MMA warps
    info->team = 1;
    info->unit_rows = 128;
    info->chunk_groups = 32;
    info->rows_per_lane = 1;
    info->smem_bytes = pp.smem;
    info->rows_per_call = M;
    info->chunk_steps = 8;
    info->stages = pp.xs;
    info->ctas_per_sm = 1;
    info->tmpl_team = pp.nt;
    info->tmpl_chunk = 0;
    return W4_OK;
  }
  if (fpath == 1) {
    tc::TcPlan tp;
    if (!tc::tc_plan(std::min(M, tc::kTcMaxM), N, K, di.sms, &tp)) return W4_ERR_SHAPE;
    *info = w4_plan_info{};
    info->path = 2;
    info->ctas = tp.ctas;
    info->slices = tp.S;
    info->threads = 320;   // 4 unpacking, 4 folding, copy and MMA warps
    info->team = 1;
    info->unit_rows = 128;
    info->chunk_groups = 8;
    info->rows_per_lane = 1;
    info->smem_bytes = tp.smem;
    info->rows_per_call = std::min(M, tc::kTcMaxM);
    info->chunk_steps = 8;
    info->stages = tp.nst;
    info->ctas_per_sm = tp.per_sm;
    info->tmpl_team = tp.np;
    info->tmpl_chunk = 0;
    info->dynamic_windows = tp.sk;   // balanced runs (needs the full workspace)
    return W4_OK;
  }
  Plan pl;
  const int mr_cap = max_rows_per_launch(K, di);
  if (mr_cap < 1 || !cached_plan(std::min(M, mr_cap), N, K, 1, 1, 0, false, di, &pl)) return W4_ERR_SHAPE;
  info->path = 1;
  info->ctas = pl.ctas;
  info->slices = pl.S;
  info->threads = kThreads;
  info->team = pl.T;
  info->unit_rows = pl.RB;
  info->chunk_groups = pl.CL * pl.T;
  info->rows_per_lane = pl.RW;
  info->smem_bytes = (int)pl.smem;
  info->rows_per_call = pl.MR;
  info->chunk_steps = pl.CL;
  info->stages = pl.nst;
  info->ctas_per_sm = pl.per_sm;
  info->dynamic_windows = pl.dyn ? 1 : 0;
  // compile-time team size / chunk length of the instantiation (0: generic)
  kernel_for(pl, false, &info->tmpl_team, &info->tmpl_chunk);
  return W4_OK;
}

extern "C" w4_status w4a16_gemv_id_plan(int n_ids, int x_rows, int N, int K, w4_plan_info* info) {
  if (info == nullptr || n_ids < 1 || N < 1) return W4_ERR_ARG;
  if (K < 32 || K % 32 != 0 || K > W4_MAX_K) return W4_ERR_SHAPE;
  if (x_rows != 1 && x_rows != n_ids) return W4_ERR_SHAPE;
  DeviceInfo di;
  planning_device(&di);
  const int xpi = (x_rows == n_ids && n_ids > 1) ? 1 : 0;
  Plan pl;
  if (!cached_plan(1, N, K, n_ids, 0, xpi, true, di, &pl)) return W4_ERR_SHAPE;
  *info = w4_plan_info{};
  info->path = 1;
  info->ctas = pl.ctas;
  info->slices = pl.S;
  info->threads = kThreads;
  info->team = pl.T;
  info->unit_rows = pl.RB;
  info->chunk_groups = pl.CL * pl.T;
  info->rows_per_lane = pl.RW;
  info->smem_bytes = (int)pl.smem;
  info->rows_per_call = 1;
  info->chunk_steps = pl.CL;
  info->stages = pl.nst;
  info->ctas_per_sm = pl.per_sm;
  info->dynamic_windows = pl.dyn ? 1 : 0;
  kernel_for(pl, false, &info->tmpl_team, &info->tmpl_chunk);
  return W4_OK;
}

extern "C" size_t w4a16_gemv_workspace_bytes_flags(int M, int N, int K, unsigned flags) {
  if (M < 1 || N < 1 || M > W4_MAX_M || K < 32 || K % 32 != 0 || K > W4_MAX_K) return 0;
  const int path = path_of(M, N, K, flags);
  if (path < 0) return 0;
  DeviceInfo di;
  planning_device(&di);
  if (path == 1) return tc_workspace(M, N, K, di.sms);
  Plan pl;
  const int mr_cap = max_rows_per_launch(K, di);
  if (mr_cap < 1 || !cached_plan(std::min(M, mr_cap), N, K, 1, 1, 0, false, di, &pl)) return 0;
  size_t ws = pl.ws_bytes;
  for (int mr = 1; mr < std::min(M, mr_cap); ++mr) {   // smaller tail launches
    Plan pm;
    if (cached_plan(mr, N, K, 1, 1, 0, false, di, &pm)) ws = std::max(ws, pm.ws_bytes);
  }
  return ws;
}

extern "C" size_t w4a16_gemv_workspace_bytes(int M, int N, int K) {
  return w4a16_gemv_workspace_bytes_flags(M, N, K, 0);
}

// w4a16_gemv, and (l2 != nullptr) the caller's L2 ranges fetched by the
// call's last launch once its CTAs have requested their own tiles.
static w4_status gemv_call(void* y, const void* qw, const void* st, const void* x, int M, int N,
                           int K, void* workspace, size_t workspace_bytes, int32_t* status_dev,
                           unsigned flags, w4_stream_t stream, const L2Ranges* l2) {
  if (y == nullptr || qw == nullptr || st == nullptr || x == nullptr) return W4_ERR_ARG;
  if (M < 1 || N < 1 || (flags & ~(W4_FLAG_PDL | kPathFlags | W4_FLAG_SILU_MUL)) != 0)
    return W4_ERR_ARG;
  if ((flags & kPathFlags) == kPathFlags) return W4_ERR_ARG;
  if (M > W4_MAX_M || K < 32 || K % 32 != 0 || K > W4_MAX_K) return W4_ERR_SHAPE;
  if (!aligned(qw, 16) || !aligned(st, 16) || !aligned(x, 16) || !aligned(y, 2))
    return W4_ERR_ALIGN;
  const int path = path_of(M, N, K, flags);
  if (path < 0) return W4_ERR_SHAPE;
  const bool gated = (flags & W4_FLAG_SILU_MUL) != 0;   // x rows [gate K | up K]
  int dev = 0;
  DeviceInfo di;
  if (!current_device(&dev, &di)) return W4_ERR_DEVICE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (path == 1)
    return tc_enqueue(y, qw, st, x, M, N, K, workspace, workspace_bytes, status_dev,
                      (flags & W4_FLAG_PDL) != 0, s, dev, di.sms, l2);
  const int mr_cap = max_rows_per_launch(K, di);
  if (mr_cap < 1) return W4_ERR_SHAPE;
  // every launch of the call is checked before the first one is enqueued
  for (int m0 = 0; m0 < M; m0 += mr_cap) {
    Plan pm;
    if (!cached_plan(std::min(mr_cap, M - m0), N, K, 1, 1, 0, false, di, &pm))
      return W4_ERR_SHAPE;
    if (pm.ws_bytes > 0 && (workspace == nullptr || workspace_bytes < pm.ws_bytes))
      return W4_ERR_WORKSPACE;
    if (pm.ws_bytes > 0 && !aligned(workspace, 16)) return W4_ERR_ALIGN;
  }
  for (int m0 = 0; m0 < M; m0 += mr_cap) {
    const int mr = std::min(mr_cap, M - m0);
    Plan pm;
    cached_plan(mr, N, K, 1, 1, 0, false, di, &pm);
    GemvParams p = base_params(pm, N, K);
    p.qw = static_cast<const uint8_t*>(qw);
    p.st = static_cast<const uint8_t*>(st);
    p.x = static_cast<const __nv_bfloat16*>(x) + (long long)m0 * K * (gated ? 2 : 1);
    p.gated = gated ? 1 : 0;
    p.y = static_cast<__nv_bfloat16*>(y) + (long long)m0 * N;
    p.n_items = 1;
    p.num_experts = 1;
    p.status = status_dev;
    if (pm.ws_bytes > 0) {
      p.ws_count = static_cast<int*>(workspace);
      p.ws_partial = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + pm.ws_part_off);
    }
    if (l2 != nullptr && m0 + mr >= M) p.l2 = *l2;   // the call's last launch
    const cudaError_t e = launch(p, pm, (flags & W4_FLAG_PDL) != 0, s, dev);
    if (e != cudaSuccess) {
      note_cuda_error(e);
      cudaGetLastError();
      return W4_ERR_LAUNCH;
    }
  }
  return W4_OK;
}

extern "C" w4_status w4a16_gemv(void* y, const void* qw, const void* st, const void* x, int M,
                                int N, int K, void* workspace, size_t workspace_bytes,
                                int32_t* status_dev, unsigned flags, w4_stream_t stream) {
  return gemv_call(y, qw, st, x, M, N, K, workspace, workspace_bytes, status_dev, flags, stream,
                   nullptr);
}

extern "C" w4_status w4a16_gemv_prefetch_l2(void* y, const void* qw, const void* st,
                                            const void* x, int M, int N, int K, void* workspace,
                                            size_t workspace_bytes, int32_t* status_dev,
                                            unsigned flags, const w4_l2_range* ranges,
                                            int n_ranges, w4_stream_t stream) {
  if (n_ranges < 0 || n_ranges > W4_MAX_L2_RANGES || (n_ranges > 0 && ranges == nullptr))
    return W4_ERR_ARG;
  L2Ranges l2{};
  for (int i = 0; i < n_ranges; ++i) {
    if (ranges[i].bytes > 0 && ranges[i].ptr == nullptr) return W4_ERR_ARG;
    if (ranges[i].bytes > 0 && !aligned(ranges[i].ptr, 16)) return W4_ERR_ALIGN;
    if (ranges[i].bytes < 16) continue;   // less than one 16-byte unit: nothing to fetch
    l2.ptr[l2.n] = static_cast<const uint8_t*>(ranges[i].ptr);
    l2.bytes[l2.n] = ranges[i].bytes;
    ++l2.n;
  }
  return gemv_call(y, qw, st, x, M, N, K, workspace, workspace_bytes, status_dev, flags, stream,
                   l2.n > 0 ? &l2 : nullptr);
}

namespace w4 {
namespace {

// Real expert ids and per-expert output vectors of a routed call (all null
// for w4a16_gemv_id).
struct RealIds {
  const int32_t* eids = nullptr;
  int num_real = 0;
  const int32_t* slot_expert = nullptr;
  const void* scale = nullptr;
  const void* bias = nullptr;
};

w4_status routed(void* y, const void* qw_base, size_t qw_stride_bytes, const void* st_base,
                 size_t st_stride_bytes, int num_experts, const int32_t* ids, int n_ids,
                 const void* x, int x_rows, int N, int K, const RealIds& real,
                 int32_t* status_dev, unsigned flags, w4_stream_t stream) {
  if (y == nullptr || qw_base == nullptr || st_base == nullptr || ids == nullptr || x == nullptr)
    return W4_ERR_ARG;
  if (n_ids < 1 || N < 1 || num_experts < 1 || (flags & ~(W4_FLAG_PDL | W4_FLAG_IDS_FINAL)) != 0)
    return W4_ERR_ARG;
  if (K < 32 || K % 32 != 0 || K > W4_MAX_K) return W4_ERR_SHAPE;
  if (x_rows != 1 && x_rows != n_ids) return W4_ERR_SHAPE;
  if (qw_stride_bytes < (size_t)N * K / 2 || st_stride_bytes < (size_t)N * (K / 32) * 2)
    return W4_ERR_ARG;
  if (!aligned(qw_base, 16) || !aligned(st_base, 16) || !aligned(x, 16) || !aligned(y, 2) ||
      qw_stride_bytes % 16 != 0 || st_stride_bytes % 16 != 0)
    return W4_ERR_ALIGN;
  if (real.eids != nullptr &&
      (!aligned(real.slot_expert, 4) || !aligned(real.scale, 2) || !aligned(real.bias, 2)))
    return W4_ERR_ALIGN;
  int dev = 0;
  DeviceInfo di;
  if (!current_device(&dev, &di)) return W4_ERR_DEVICE;
  const int xpi = (x_rows == n_ids && n_ids > 1) ? 1 : 0;
  Plan pl;
  if (!cached_plan(1, N, K, n_ids, 0, xpi, true, di, &pl)) return W4_ERR_SHAPE;
  GemvParams p = base_params(pl, N, K);
  p.qw = static_cast<const uint8_t*>(qw_base);
  p.st = static_cast<const uint8_t*>(st_base);
  p.qw_item_stride = qw_stride_bytes;
  p.st_item_stride = st_stride_bytes;
  p.ids = ids;
  p.ids_final = (flags & W4_FLAG_IDS_FINAL) != 0 ? 1 : 0;
  p.num_experts = num_experts;
  p.x = static_cast<const __nv_bfloat16*>(x);
  p.x_per_item = xpi;
  p.y = static_cast<__nv_bfloat16*>(y);
  p.n_items = n_ids;
  p.status = status_dev;
  p.eids = real.eids;
  p.num_real = real.num_real;
  p.slot_expert = real.slot_expert;
  p.escale = static_cast<const __nv_bfloat16*>(real.scale);
  p.ebias = static_cast<const __nv_bfloat16*>(real.bias);
  const cudaError_t e =
      launch(p, pl, (flags & W4_FLAG_PDL) != 0, reinterpret_cast<cudaStream_t>(stream), dev);
  if (e != cudaSuccess) {
    note_cuda_error(e);
    cudaGetLastError();
    return W4_ERR_LAUNCH;
  }
  return W4_OK;
}

}  // namespace
}  // namespace w4

extern "C" w4_status w4a16_gemv_id(void* y, const void* qw_base, size_t qw_stride_bytes,
                                   const void* st_base, size_t st_stride_bytes, int num_experts,
                                   const int32_t* ids, int n_ids, const void* x, int x_rows,
                                   int N, int K, int32_t* status_dev, unsigned flags,
                                   w4_stream_t stream) {
  return routed(y, qw_base, qw_stride_bytes, st_base, st_stride_bytes, num_experts, ids, n_ids,
                x, x_rows, N, K, RealIds{}, status_dev, flags, stream);
}

extern "C" w4_status w4a16_gemv_id_scaled(void* y, const void* qw_base, size_t qw_stride_bytes,
                                          const void* st_base, size_t st_stride_bytes,
                                          int num_slots, const int32_t* ids, int n_ids,
                                          const void* x, int x_rows, int N, int K,
                                          const int32_t* expert_ids, int num_experts,
                                          const int32_t* slot_expert, const void* scale,
                                          const void* bias, int32_t* status_dev, unsigned flags,
                                          w4_stream_t stream) {
  if (expert_ids == nullptr || num_experts < 1) return W4_ERR_ARG;
  RealIds real;
  real.eids = expert_ids;
  real.num_real = num_experts;
  real.slot_expert = slot_expert;
  real.scale = scale;
  real.bias = bias;
  return routed(y, qw_base, qw_stride_bytes, st_base, st_stride_bytes, num_slots, ids, n_ids, x,
                x_rows, N, K, real, status_dev, flags, stream);
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
  if (M < 1 || N < 1 || (flags & ~(W4_FLAG_PDL | kPathFlags | W4_FLAG_SILU_MUL)) != 0)
    return W4_ERR_ARG;
  if ((flags & kPathFlags) == kPathFlags) return W4_ERR_ARG;
  if (M > W4_MAX_M || K < 32 || K % 32 != 0 || K > W4_MAX_K) return W4_ERR_SHAPE;
  if (!aligned(qw, 16) || !aligned(st, 16) || !aligned(x, 16) || !aligned(y, 2))
    return W4_ERR_ALIGN;
  const int path = path_of(M, N, K, flags);
  if (path < 0) return W4_ERR_SHAPE;
  const bool gated = (flags & W4_FLAG_SILU_MUL) != 0;   // x rows [gate K | up K]
  int dev = 0;
  DeviceInfo di;
  if (!current_device(&dev, &di)) return W4_ERR_DEVICE;
  if (path == 1) {
    // every launch of this call must fit the fixed array: check before any work
    // (the plain plans: balanced runs are not taken here)
    const size_t need = tc_workspace(M, N, K, di.sms, false);
    if (need > (size_t)W4_STATIC_SCRATCH_BYTES) return W4_ERR_WORKSPACE;
    void* base = nullptr;
    if (need > 0) {
      cudaError_t e = static_scratch_address(dev, &base);
      if (e == cudaSuccess) e = cudaMemsetAsync(base, 0, need, reinterpret_cast<cudaStream_t>(stream));
      if (e != cudaSuccess) {
        note_cuda_error(e);
        cudaGetLastError();
        return W4_ERR_LAUNCH;
      }
    }
    return tc_enqueue(y, qw, st, x, M, N, K, base, need, status_dev, (flags & W4_FLAG_PDL) != 0,
                      reinterpret_cast<cudaStream_t>(stream), dev, di.sms);
  }
  const int mr_cap = max_rows_per_launch(K, di);
  if (mr_cap < 1) return W4_ERR_SHAPE;
  // every launch of this call must fit the fixed array: check before any work
  for (int m0 = 0; m0 < M; m0 += mr_cap) {
    Plan pm;
    if (!cached_plan(std::min(mr_cap, M - m0), N, K, 1, 1, 0, false, di, &pm)) return W4_ERR_SHAPE;
    if (pm.ws_bytes > (size_t)W4_STATIC_SCRATCH_BYTES) return W4_ERR_WORKSPACE;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  for (int m0 = 0; m0 < M; m0 += mr_cap) {
    const int mr = std::min(mr_cap, M - m0);
    Plan pm;
    cached_plan(mr, N, K, 1, 1, 0, false, di, &pm);
    GemvParams p = base_params(pm, N, K);
    p.qw = static_cast<const uint8_t*>(qw);
    p.st = static_cast<const uint8_t*>(st);
    p.x = static_cast<const __nv_bfloat16*>(x) + (long long)m0 * K * (gated ? 2 : 1);
    p.gated = gated ? 1 : 0;
    p.y = static_cast<__nv_bfloat16*>(y) + (long long)m0 * N;
    p.n_items = 1;
    p.num_experts = 1;
    p.status = status_dev;
    if (pm.ws_bytes > 0) {
      void* base = nullptr;
      cudaError_t e = static_scratch_address(dev, &base);
      // the counters must start at zero; the array keeps the previous call's
      // contents (and an aborted call may leave them armed)
      if (e == cudaSuccess)
        e = cudaMemsetAsync(base, 0, (size_t)pm.B * sizeof(int), s);
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
