// A chain of W4A16 GEMVs in one persistent launch (w4a16_gemv_chain).
//
// Page "Gemma 4 on a 4 GB GPU in Plain PyTorch", section "Step 3 — Multiply
// Straight From the Packed Weights": a decoded token is one product of an
// activation vector with each weight matrix in turn, read from the packed
// words, and the token rate is set by how fast those words stream from
// memory.  Launched one by one, every product pays a start-up gap in which
// the weight stream is idle (the next launch's CTAs only start once the
// previous ones leave the SM).  Here one launch runs a whole list of
// products ("tasks": a decode pass, or a routed-expert layer's gate/up then
// down projection, page "Running a 26B MoE on an 8 GB Jetson by streaming
// experts from SSD", section "Streaming without touching a single GPU
// kernel"), and the weight stream never stops at a task boundary:
//
//  * One CTA per SM: 14 consumer warps and 1 copy warp.  The copy warp takes
//    windows (whole rows of one task, or of one expert of a routed task)
//    from a counter shared by the launch, in one global order, and streams
//    their packed codes and steps into a ring of shared-memory stages with
//    1-D bulk copies (TMA).  Weights do not depend on earlier tasks, so a
//    CTA keeps fetching the next task's windows while its consumers still
//    wait for the activations of that task.
//  * A task may name an earlier task whose output it reads (`dep`).  Each
//    window, once its rows are stored, adds one to its task's count (a
//    release add at GPU scope by the last consumer warp done with it).
//    Before the first window of a dependent task the consumers wait
//    (bounded) until the earlier task's count is complete, then stage its
//    activation row.  Windows are handed out in increasing order and each
//    CTA finishes its windows in that order, so the lowest unfinished window
//    always has every window it waits for finished: the launch cannot
//    deadlock, whatever the number of resident CTAs.
//  * The per-row arithmetic is that of w4a16_gemv (gemv_core.cuh, with the
//    team size and chunk length fixed by K alone), so every task's outputs
//    are bitwise those of the same call made on its own.
//  * Every wait is bounded; on expiry the kernel records W4_ERR_TIMEOUT and
//    the CTA leaves in order.  The launch's last CTA re-arms the counters.
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "gemv_core.cuh"
#include "gemv_host.h"

namespace w4 {
namespace chain {

constexpr int kGroups = 2;                  // consumer groups, alternate windows each
constexpr int kGroupWarps = 7;
constexpr int kGroupThreads = 32 * kGroupWarps;
constexpr int kWarps = kGroups * kGroupWarps;   // consumer warps
constexpr int kCons = 32 * kWarps;
constexpr int kCopyWarp = kWarps;          // warp 14
constexpr int kSignalWarp = kWarps + 1;     // warp 15
constexpr int kThreads = kCons + 64;        // + the copy warp and the signal warp
constexpr int kMaxStages = 8;
constexpr int kHdrBytes = 1024;             // barriers, flags, window records
constexpr int kEndOff = 132;                // windows of this CTA, once known (else -1)
constexpr int kXsOff = 136;                 // (task, item) whose activation row is staged
constexpr int kGdoneOff = 144;              // last window each group finished [2]
constexpr int kGflagOff = 152;              // a group's decision to restage [2]
constexpr int kInfoOff = 256;               // (task, item, row0, rows) per stage
constexpr int kSeqOff = 384;                // warps done with each of the last 16 windows
constexpr int kPendOff = 512;               // finished windows for the signal warp [32]
constexpr int kPend = 32;
constexpr long long kWaitCycles = 1LL << 31;
constexpr long long kStageMax = 96 << 10;   // largest stage the planner picks

constexpr unsigned kTaskGated = 1u;         // x rows are [gate K | up K]
constexpr unsigned kTaskXPerItem = 2u;      // routed: item i reads activation row i
constexpr unsigned kTaskDepPerItem = 4u;    // item i reads only item i of task `dep`

// One task as the kernel sees it (in the launch's parameter space).
struct Task {
  const uint8_t* qw;
  const uint8_t* st;
  const __nv_bfloat16* x;
  __nv_bfloat16* y;
  const int32_t* ids;                  // routed: ids[n_items]; nullptr: dense
  uint32_t qw_stride16, st_stride16;   // bytes between experts / 16
  int N, K;
  int wbase;                           // global number of the task's first window
  int wpi;                             // windows per item
  int n_items;
  int num_experts;
  int dep;                             // task whose outputs this one reads, or -1
  int cbase;                           // first of its n_items done-counters
  int16_t RB;                          // rows of a full window
  uint8_t spec;                        // 0: dot instantiation A, 1: B
  uint8_t T, CL, nch, flags;
  uint16_t NI;                         // groups per lane per row
};

struct Params {
  int n_tasks;
  int total;                           // windows of all tasks
  int nst;                             // stages
  int stage_bytes;
  int xs_off, xsc_off, red_off, red_slot;   // shared-memory offsets; floats per red slot
  int n_counters;                      // done-counters of all tasks (one per item)
  int* ws;                             // [0] windows taken, [1] CTAs done, [2 + c] done[c]
  int32_t* status;
  Task tasks[W4_CHAIN_MAX_TASKS];
};
static_assert(sizeof(Params) <= 32764, "kernel parameters must fit 32764 bytes");

__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag != 0) return false;
    if (clock64() - t0 > kWaitCycles) return false;
  }
}

__device__ __forceinline__ int load_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void red_release_gpu(int* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ int atom_add_acq_rel_cta(int* p, int v) {
  int old;
  asm volatile("atom.acq_rel.cta.shared::cta.add.s32 %0, [%1], %2;"
               : "=r"(old)
               : "r"(smem_addr(p)), "r"(v)
               : "memory");
  return old;
}

__device__ __forceinline__ void st_release_cta_s32(int* p, int v) {
  asm volatile("st.release.cta.shared::cta.s32 [%0], %1;" ::"r"(smem_addr(p)), "r"(v) : "memory");
}

__device__ __forceinline__ int ld_acquire_cta_s32(const int* p) {
  int v;
  asm volatile("ld.acquire.cta.shared::cta.s32 %0, [%1];" : "=r"(v) : "r"(smem_addr(p)) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_cta_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.release.cta.shared::cta.u64 [%0], %1;" ::"r"(smem_addr(p)), "l"(v) : "memory");
}

__device__ __forceinline__ unsigned long long ld_acquire_cta_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.cta.shared::cta.u64 %0, [%1];" : "=l"(v) : "r"(smem_addr(p)) : "memory");
  return v;
}

// Consumer warp of group g, after its stores of the CTA's window number
// `seq`: the last of the group's 7 warps to get here records that the group
// is done with the window (gdone[g] = seq: its staged activation row is no
// longer read for it) and hands the window (its done-counter `ctr`) to the
// signal warp through pend[seq % 32] = (seq + 1) << 32 | ctr.  The per-window
// warp count is reset by that warp; it is used again 16 windows later, which
// no warp can reach before every warp of the group has passed this point
// (the ring holds at most 8 windows, and the ring only turns once every warp
// of a window has released its stage).  A pend entry is reused 32 windows
// later, once the signal warp has cleared it (bounded wait).
__device__ __forceinline__ bool window_done(uint8_t* smem, int seq, int ctr, int g, int lane,
                                            volatile int* abort_flag) {
  __syncwarp();
  bool ok = true;
  if (lane == 0) {
    int* c = reinterpret_cast<int*>(smem + kSeqOff) + (seq & 15);
    if (atom_add_acq_rel_cta(c, 1) == kGroupWarps - 1) {
      *c = 0;
      st_release_cta_s32(reinterpret_cast<int*>(smem + kGdoneOff) + g, seq);
      unsigned long long* pe = reinterpret_cast<unsigned long long*>(smem + kPendOff) + (seq % kPend);
      const long long t0 = clock64();
      while (ld_acquire_cta_u64(pe) != 0ull) {
        if (*abort_flag != 0 || clock64() - t0 > kWaitCycles) {
          ok = false;
          break;
        }
      }
      st_release_cta_u64(pe, ((unsigned long long)(seq + 1) << 32) | (unsigned)ctr);
    }
  }
  return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

// Copy warp, lane 0: request the window's rows [row0, row0 + nrows) of the
// matrix at (qwi, sti) into the stage at shared address `stage` (generic
// pointer `stage_ptr`): one bulk copy of the codes (contiguous in memory)
// and one of the 16-byte-aligned superset of the steps, clipped to the
// matrix's last full 16-byte line; the bytes past that line (at most 14, at
// the very end of the step array) are stored by hand.
__device__ void issue_rows(const Task& tk, const uint8_t* qwi, const uint8_t* sti, int row0,
                           int nrows, int step_off, uint32_t stage, uint8_t* stage_ptr,
                           uint32_t full, uint64_t pol) {
  const long long row_code = tk.K / 2, row_st = (long long)(tk.K / 32) * 2;
  const uintptr_t sbase = reinterpret_cast<uintptr_t>(sti);
  const uintptr_t st_lim = (sbase + (uintptr_t)((long long)tk.N * row_st)) & ~(uintptr_t)15;
  const uint32_t code_bytes = (uint32_t)(nrows * row_code);
  const uintptr_t a0 = sbase + (uintptr_t)(row0 * row_st);
  const uintptr_t e = sbase + (uintptr_t)((row0 + nrows) * row_st);
  const uintptr_t a = a0 & ~(uintptr_t)15;
  const uintptr_t b = min((e + 15) & ~(uintptr_t)15, st_lim);
  const uint32_t step_bytes = b > a ? (uint32_t)(b - a) : 0u;
  uint8_t* dst = stage_ptr + step_off;
  for (uintptr_t q = max(a, b); q < e; q += 2)
    *reinterpret_cast<uint16_t*>(dst + (q - a)) = *reinterpret_cast<const uint16_t*>(q);
  mbar_arrive_expect_tx(full, code_bytes + step_bytes);   // also releases the hand-stored tail
  bulk_g2s_evict_first(stage, qwi + row0 * row_code, code_bytes, full, pol);
  if (step_bytes > 0)
    bulk_g2s_evict_first(stage + step_off, reinterpret_cast<const void*>(a), step_bytes, full, pol);
}

// Consumers: stage the activation row of (task, item) with loads that see
// the outputs of earlier tasks of this launch (L2, not the read-only path).
__device__ void stage_row(const Task& tk, int item, uint8_t* xs, float* xsc, int tid,
                          int nthreads) {
  const int K = tk.K, Kg = K / 32, Kgp = (int)tk.NI * tk.T;
  const int row = (tk.flags & kTaskXPerItem) ? item : 0;
  const bool gated = (tk.flags & kTaskGated) != 0;
  if (!gated) {
    // a thread issues the loads of two 32-value groups before converting
    // either: one trip to L2 per round
    for (int base = tid; base < Kgp; base += 2 * nthreads) {
      uint4 v[2][4];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int g = base + u * nthreads;
#pragma unroll
        for (int i = 0; i < 4; ++i) v[u][i] = make_uint4(0u, 0u, 0u, 0u);
        if (g < Kg) {
          const uint4* src = reinterpret_cast<const uint4*>(tk.x + (long long)row * K + g * 32);
#pragma unroll
          for (int i = 0; i < 4; ++i) v[u][i] = __ldcg(src + i);
        }
      }
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int g = base + u * nthreads;
        if (g < Kgp) store_staged_group(v[u], xs + g * 16, Kgp * 16, xsc + g, g < Kg);
      }
    }
    return;
  }
  for (int g = tid; g < Kgp; g += nthreads) {
    const bool valid = g < Kg;
    {   // gated: silu(gate) * up, one group at a time
      float h[32];
      float mx = 0.0f;
      if (valid) {
        const uint4* gs = reinterpret_cast<const uint4*>(tk.x + (long long)row * 2 * K + g * 32);
        const uint4* us = reinterpret_cast<const uint4*>(tk.x + (long long)row * 2 * K + K + g * 32);
        uint4 gv[4], uv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          gv[i] = __ldcg(gs + i);
          uv[i] = __ldcg(us + i);
        }
        mx = silu_mul_group(gv, uv, h);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) h[i] = 0.0f;
      }
      store_staged_group_f32(h, mx, xs + g * 16, Kgp * 16, xsc + g, valid);
    }
  }
}

// Consumer warp `warp` of its group: its share of a window's (chunk, row
// step) items, dealt round robin over the group's 7 warps.  Rows finished by one chunk are
// stored (0 + chunk sum, rounded once); otherwise each chunk sum goes to the
// window's buffer `redw` [rows][nch].  Rows of a short window past its end
// read stale stage bytes (in bounds) and are dropped.
template <int RW, int TT, int CLT>
__device__ __forceinline__ void window_dot(const Task& tk, const uint8_t* sm, uint32_t tile,
                                           uint32_t xs_off, uint32_t xsc_off, int row0, int nrows,
                                           __nv_bfloat16* yrow, float* redw, int warp, int lane) {
  const int T = TT > 0 ? TT : tk.T;
  const int nsw = 32 / T;
  const int set = lane / T, t = lane - set * T;
  const int K = tk.K, Kg = K / 32, kg2 = Kg * 2;
  const int NI = tk.NI, CL = tk.CL, nch = tk.nch;
  const int Kgp = NI * T;
  const int kg_valid = Kgp != Kg ? Kg : 0x7fffffff;   // groups past it are padding
  const int gpc = CL * T;
  const int rstep = nsw * RW;
  const int nrs = (nrows + rstep - 1) / rstep;
  const int items = nch * nrs;
  const int code_pitch = K / 2;
  const uint32_t step_base = (uint32_t)(tk.RB * code_pitch + (T - 1) * 16);
  const uint32_t soff0 = (kg2 & 15) == 0 ? 0u : (uint32_t)(((row0 & 7) * (kg2 & 15)) & 15);
  for (int it = warp; it < items; it += kGroupWarps) {
    const int ci = it / nrs, rs = it - ci * nrs;
    uint32_t co[RW], so[RW];
#pragma unroll
    for (int j = 0; j < RW; ++j) {
      const int r = rs * rstep + j * nsw + set;
      co[j] = tile + (uint32_t)(r * code_pitch + (ci * gpc + t) * 16);
      so[j] = tile + step_base + soff0 + (uint32_t)(r * kg2 + (ci * gpc + t) * 2);
    }
    const int g0 = ci * gpc + t;
    const int ns = CLT > 0 ? CLT : min(CL, NI - ci * CL);
    float acc[RW][1];
    tile_dot<1, RW, TT, CLT>(sm, xs_off + (uint32_t)(g0 * 16), xsc_off + (uint32_t)(g0 * 4),
                             Kgp * 16, 0, 0, co, so, ns, T, kg_valid - g0, acc);
#pragma unroll
    for (int j = 0; j < RW; ++j) acc[j][0] = team_sum<TT>(acc[j][0], T);
    if (t == 0) {
#pragma unroll
      for (int j = 0; j < RW; ++j) {
        const int rl = rs * rstep + j * nsw + set;
        if (rl >= nrows) continue;
        if (nch == 1)
          yrow[rl] = __float2bfloat16_rn(0.0f + acc[j][0]);
        else
          redw[rl * nch + ci] = acc[j][0];
      }
    }
  }
}

template <int RWA, int TTA, int CLA, int RWB, int TTB, int CLB>
__global__ void __launch_bounds__(kThreads, 1) chain_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t sbase = smem_addr(smem);
  const uint32_t full0 = sbase, empty0 = sbase + 8 * kMaxStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + 16 * kMaxStages);
  volatile int* info = reinterpret_cast<volatile int*>(smem + kInfoOff);
  int* seq_cnt = reinterpret_cast<int*>(smem + kSeqOff);
  const int nst = p.nst;
  int* const work = p.ws;
  int* const done = p.ws + 2;

  if (threadIdx.x == 0) {
    for (int s = 0; s < nst; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, kGroupWarps);   // the group that takes the window
    }
    *abort_flag = 0;
    *reinterpret_cast<volatile int*>(smem + kEndOff) = -1;
    *reinterpret_cast<volatile unsigned long long*>(smem + kXsOff) = ~0ull;   // no row staged
    reinterpret_cast<volatile int*>(smem + kGdoneOff)[0] = -1;
    reinterpret_cast<volatile int*>(smem + kGdoneOff)[1] = -1;
    for (int i = 0; i < 16; ++i) seq_cnt[i] = 0;
    for (int i = 0; i < kPend; ++i) reinterpret_cast<unsigned long long*>(smem + kPendOff)[i] = 0ull;
    mbar_init_fence();
  }
  __syncthreads();
  pdl_launch_dependents();
  pdl_wait();   // inputs, ids and counters follow earlier kernels

  if (warp == kSignalWarp) {
    // ------------------------------------------------------------ signal warp
    // Publishes finished windows in order: each done-counter gets one add
    // per window, release at GPU scope (the consumers' stores come before
    // it through the hand-over).  Runs of windows of one counter share one
    // add, so the release's wait for earlier stores to reach L2 stays off
    // the consumers' path.  Then the launch's last CTA re-arms the counters.
    if (lane != 0) return;
    unsigned long long* pend = reinterpret_cast<unsigned long long*>(smem + kPendOff);
    volatile int* end_seq = reinterpret_cast<volatile int*>(smem + kEndOff);
    int next = 0, run_ctr = -1, run_n = 0;
    long long t0 = clock64();
    bool ok = true;
    while (true) {
      const unsigned long long v = ld_acquire_cta_u64(pend + (next % kPend));
      if ((int)(v >> 32) == next + 1) {
        const int ctr = (int)(v & 0xffffffffu);
        st_release_cta_u64(pend + (next % kPend), 0ull);
        if (ctr != run_ctr && run_n > 0) {
          red_release_gpu(done + run_ctr, run_n);
          run_n = 0;
        }
        run_ctr = ctr;
        ++run_n;
        ++next;
        t0 = clock64();
        continue;
      }
      if (run_n > 0) {   // nothing more ready now: publish the run
        red_release_gpu(done + run_ctr, run_n);
        run_n = 0;
      }
      const int e = *end_seq;
      if (e >= 0 && next >= e) break;
      if (*abort_flag != 0 || clock64() - t0 > kWaitCycles) {
        ok = false;
        break;
      }
      __nanosleep(128);   // idle: leave the issue slots to the consumer warps
    }
    if (ok) {
      __threadfence();
      if (atomicAdd(work + 1, 1) == (int)gridDim.x - 1) {
        __threadfence();
        atomicExch(work, 0);
        for (int i = 0; i < p.n_counters; ++i) atomicExch(done + i, 0);
        atomicExch(work + 1, 0);
      }
    }
    return;
  }

  if (warp == kCopyWarp) {
    // ------------------------------------------------------------ copy warp
    const uint64_t pol = policy_evict_first();
    long long issued = 0;
    int slot = 0;
    uint32_t phase = 0;
    bool ended = false;
    int ends = 0;   // end records issued
    int ti = 0;   // task of the current window (windows come in increasing order)
    int w = 0, grabbed = 0;
    if (lane == 0) w = atomicAdd(work, 1);
    w = __shfl_sync(0xffffffffu, w, 0);
    while (true) {
      if (issued >= nst && !wait_phase(empty0 + 8 * slot, phase ^ 1u, abort_flag)) {
        if (*abort_flag == 0) report(p.status, W4_ERR_TIMEOUT);
        *abort_flag = 1;
        break;
      }
      volatile int* rec = info + 4 * slot;
      if (w >= p.total) {
        // one end record for each consumer group (the second in the next
        // stage, once it is free); the signal warp learns the window count
        if (lane == 0) {
          *reinterpret_cast<volatile int*>(smem + kEndOff) = (int)(issued - ends);
          rec[3] = 0;
          mbar_arrive(full0 + 8 * slot);
        }
        __syncwarp();
        ++issued;
        if (++slot == nst) {
          slot = 0;
          phase ^= 1u;
        }
        if (++ends == kGroups) {
          ended = true;
          break;
        }
        continue;
      }
      // the next window's number travels while this one is requested
      if (lane == 0) grabbed = atomicAdd(work, 1);
      while (ti + 1 < p.n_tasks && w >= p.tasks[ti + 1].wbase) ++ti;
      const Task& tk = p.tasks[ti];
      const int lw = w - tk.wbase;
      const int item = lw / tk.wpi;
      const int row0 = (lw - item * tk.wpi) * tk.RB;
      const int nrows = min((int)tk.RB, tk.N - row0);
      if (lane == 0) {
        const uint8_t* qwi = tk.qw;
        const uint8_t* sti = tk.st;
        bool ok = true;
        if (tk.ids != nullptr) {
          const int e = __ldg(tk.ids + item);
          ok = e >= 0 && e < tk.num_experts;
          qwi += (unsigned long long)(ok ? e : 0) * tk.qw_stride16 * 16ull;
          sti += (unsigned long long)(ok ? e : 0) * tk.st_stride16 * 16ull;
        }
        rec[0] = ti;
        rec[1] = item;
        rec[2] = row0;
        rec[3] = ok ? nrows : -nrows;   // negative: an id out of range, nothing copied
        const uint32_t st_off = kHdrBytes + slot * p.stage_bytes;
        const int step_off = tk.RB * (tk.K / 2) + (tk.T - 1) * 16;
        if (ok)
          issue_rows(tk, qwi, sti, row0, nrows, step_off, sbase + st_off, smem + st_off,
                     full0 + 8 * slot, pol);
        else
          mbar_arrive(full0 + 8 * slot);
      }
      __syncwarp();
      ++issued;
      if (++slot == nst) {
        slot = 0;
        phase ^= 1u;
      }
      w = __shfl_sync(0xffffffffu, grabbed, 0);
    }
    // let the last copies land before the CTA may leave (the end records
    // complete at once)
    const int last = issued < nst ? (int)issued : nst;
    for (int i = 1; i <= last; ++i) {
      const int sl = slot - i < 0 ? slot - i + nst : slot - i;
      const uint32_t ph = slot - i < 0 ? phase ^ 1u : phase;
      if (!mbar_wait_bounded(full0 + 8 * sl, ph, kWaitCycles)) {
        report(p.status, W4_ERR_TIMEOUT);
        break;
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  // Two groups of 7 warps take alternate windows (group g: the CTA's windows
  // g, g + 2, ...), each like one CTA of the per-launch kernel, and share one
  // staged activation row.  A group whose window needs another row than the
  // staged one waits until either the other group has staged it or the other
  // group is done with every earlier window, and in the latter case stages
  // it itself (after waiting for the task it depends on).  So a row is never
  // replaced while a window that needs it is still being computed.
  const int g = warp / kGroupWarps;               // consumer group
  const int gw = warp - g * kGroupWarps;          // warp within the group
  const int gtid = threadIdx.x - g * kGroupThreads;
  const int bar_id = 1 + g;
  uint8_t* xs = smem + p.xs_off;
  float* xsc = reinterpret_cast<float*>(smem + p.xsc_off);
  float* red = reinterpret_cast<float*>(smem + p.red_off);
  unsigned long long* xs_key = reinterpret_cast<unsigned long long*>(smem + kXsOff);
  int* gdone = reinterpret_cast<int*>(smem + kGdoneOff);
  volatile int* gflag = reinterpret_cast<volatile int*>(smem + kGflagOff);
  auto group_sync = [&]() {
    asm volatile("bar.sync %0, %1;" ::"r"(bar_id), "n"(kGroupThreads) : "memory");
  };
  int cur_task = -1, cur_item = -1;   // the row this group's windows last used
  bool reported = false;
  for (int seq = g;; seq += kGroups) {
    const int slot = seq % nst;
    const uint32_t phase = (uint32_t)((seq / nst) & 1);
    if (!wait_phase(full0 + 8 * slot, phase, abort_flag)) {
      if (*abort_flag == 0) report(p.status, W4_ERR_TIMEOUT);
      *abort_flag = 1;
      return;
    }
    const volatile int* rec = info + 4 * slot;
    const int t = rec[0], item = rec[1], row0 = rec[2], nr = rec[3];
    if (nr == 0) {   // no more windows: never make the other group wait for us
      if (gtid == 0) st_release_cta_s32(gdone + g, 0x7fffffff);
      return;
    }
    const Task& tk = p.tasks[t];
    const bool xpi = (tk.flags & kTaskXPerItem) != 0;
    const int want_item = xpi ? item : 0;
    const unsigned long long key = ((unsigned long long)(unsigned)t << 32) | (unsigned)want_item;
    if (t != cur_task || want_item != cur_item) {
      // the row this window needs: staged already, or stage it here
      if (gtid == 0) {
        const long long t0 = clock64();
        int restage = 0;
        while (true) {
          if (ld_acquire_cta_u64(xs_key) == key) break;           // staged by the other group
          if (ld_acquire_cta_s32(gdone + (1 - g)) >= seq - 1) {  // other group done before us
            restage = ld_acquire_cta_u64(xs_key) == key ? 0 : 1;
            break;
          }
          if (*abort_flag != 0 || clock64() - t0 > kWaitCycles) {
            if (*abort_flag == 0) report(p.status, W4_ERR_TIMEOUT);
            *abort_flag = 1;
            break;
          }
        }
        if (restage && tk.dep >= 0 && *abort_flag == 0) {
          // the earlier task's windows (all its items, or item `item`) are done
          const bool per_item = (tk.flags & kTaskDepPerItem) != 0;
          const Task& dk = p.tasks[tk.dep];
          const long long t1 = clock64();
          for (int i = per_item ? item : 0; i < (per_item ? item + 1 : dk.n_items); ++i) {
            while (load_acquire_gpu(done + dk.cbase + i) < dk.wpi) {
              if (*abort_flag != 0 || clock64() - t1 > kWaitCycles) {
                if (*abort_flag == 0) report(p.status, W4_ERR_TIMEOUT);
                *abort_flag = 1;
                break;
              }
              __nanosleep(32);
            }
            if (*abort_flag != 0) break;
          }
        }
        gflag[g] = restage;
      }
      group_sync();
      if (*abort_flag != 0) return;
      if (gflag[g]) {
        stage_row(tk, item, xs, xsc, gtid, kGroupThreads);
        group_sync();
        if (gtid == 0) st_release_cta_u64(xs_key, key);
      }
      cur_task = t;
      cur_item = want_item;
    }
    float* redw = red + slot * p.red_slot;
    const int nrows = nr < 0 ? -nr : nr;
    const uint32_t tile = kHdrBytes + (uint32_t)slot * p.stage_bytes;
    if (nr > 0) {
      __nv_bfloat16* yrow = tk.y + (long long)item * tk.N + row0;
      const uint32_t xs_off = (uint32_t)p.xs_off, xsc_off = (uint32_t)p.xsc_off;
      if (tk.spec == 0 || (RWA == RWB && TTA == TTB && CLA == CLB))
        window_dot<RWA, TTA, CLA>(tk, smem, tile, xs_off, xsc_off, row0, nrows, yrow, redw, gw,
                                  lane);
      else
        window_dot<RWB, TTB, CLB>(tk, smem, tile, xs_off, xsc_off, row0, nrows, yrow, redw, gw,
                                  lane);
    } else if (!reported && gtid == 0) {
      report(p.status, W4_ERR_INDEX);   // the item's rows stay unwritten
      reported = true;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * slot);   // this warp is done with the stage
    if (tk.nch > 1 && nr > 0) {
      // rows whose chunks were summed by different warps: added in chunk order
      group_sync();
      __nv_bfloat16* yrow = tk.y + (long long)item * tk.N + row0;
      for (int i = gtid; i < nrows; i += kGroupThreads) {
        float v = 0.0f;
        for (int c = 0; c < tk.nch; ++c) v += redw[i * tk.nch + c];
        yrow[i] = __float2bfloat16_rn(v);
      }
    }
    if (!window_done(smem, seq, tk.cbase + item, g, lane, abort_flag)) {
      if (*abort_flag == 0) report(p.status, W4_ERR_TIMEOUT);
      *abort_flag = 1;
      return;
    }
  }
}

// ================================================================= host side
// Dot instantiations: compile-time (rows per lane, team, chunk) for the two
// row lengths of the common decoders (hidden and intermediate), and a
// generic one for any K.
struct Spec {
  int RW, TT, CL;
};
struct Inst {
  Spec a, b;
  int Ka, Kb;   // the K each spec serves (0: any)
};
constexpr int kInsts = 4;
constexpr Inst kInst[kInsts] = {
    {{4, 8, 3}, {2, 32, 3}, 5376, 21504},   // hidden 5376, intermediate 21504
    {{2, 16, 4}, {1, 32, 4}, 2048, 8192},   // hidden 2048, intermediate 8192
    {{1, 8, 11}, {1, 2, 11}, 2816, 704},    // routed experts: hidden 2816, expert width 704
    {{1, 0, 0}, {1, 0, 0}, 0, 0},           // generic
};

using KernelFn = void (*)(Params);

KernelFn kernel_of(int inst) {
  switch (inst) {
    case 0: return chain_kernel<4, 8, 3, 2, 32, 3>;
    case 1: return chain_kernel<2, 16, 4, 1, 32, 4>;
    case 2: return chain_kernel<1, 8, 11, 1, 2, 11>;
    case 3: return chain_kernel<1, 0, 0, 1, 0, 0>;
    default: return nullptr;
  }
}

// Whether `spec` (compile-time team and chunk, or generic) computes rows of K.
bool spec_fits(const Spec& sp, int K) {
  if (sp.TT == 0) return true;
  int T, NI, CL, nch;
  row_shape(K, &T, &NI, &CL, &nch);
  return T == sp.TT && CL == sp.CL && NI % CL == 0 && NI * T == K / 32;
}

struct TaskPlan {
  int spec = 0, RW = 1, T = 1, NI = 1, CL = 1, nch = 1, RB = 1;
  int tile = 0;
  int windows = 0;   // per item
};

struct ChainPlan {
  int inst = 3;
  int nst = 2;
  int stage_bytes = 0;
  int xs_off = 0, xsc_off = 0, red_off = 0, red_slot = 0;
  long long smem = 0;
  int total = 0;
  TaskPlan t[W4_CHAIN_MAX_TASKS];
};

// Window (rows a multiple of the row step) of a task for stages of at most
// `cap` bytes.  Each warp of a consumer group takes at most ceil(items / 7)
// of a window's (chunk, row step) items, so a window lasts about as long as
// its copy (at half the SM's stream rate: two groups) or as its slowest
// warp's items, whichever is longer, and a task takes about
// ceil(windows / (2 SMs)) such rounds.  The SM's stream rate is its share of
// HBM, or less when the stages not held by the two groups cannot keep that
// share in flight over a copy's latency.  The window with the shortest
// estimate is taken (ties: the taller one): full 7-item windows for large
// tasks, more and smaller windows for tasks too small to reach every SM.
// `est` returns the estimate (microseconds).
constexpr double kSmBytesPerUs = 44.7e3;    // an SM's share of the HBM stream
constexpr double kCopyLatencyUs = 2.0;      // a stage's copy under load
// weight bytes a consumer warp dequantises per microsecond, by rows per lane
constexpr double warp_bytes_per_us(int rw) { return rw >= 4 ? 3.9e3 : rw == 2 ? 3.55e3 : 3.1e3; }
bool pick_window(int K, int N, int n_items, const TaskPlan& tp, long long cap, int nst, int sms,
                 int* rb_out, int* tile_out, double* est_out) {
  const int nsw = 32 / tp.T;
  const int rstep = nsw * tp.RW;
  const double row_bytes = K / 2 + K / 16;
  const double sm_rate =
      std::min(kSmBytesPerUs, std::max(0.5, (double)(nst - kGroups)) * cap / kCopyLatencyUs);
  double best = -1.0;
  for (int rs = 1; rs <= 64; ++rs) {
    const int rb = rs * rstep;
    int cp, sp, so, tb;
    tile_geometry(K, tp.T, tp.CL, true, tp.nch, rb, &cp, &sp, &so, &tb);
    if (tb > cap) break;
    if (rs > 1 && rb >= N + rstep) break;   // no taller than the rows there are
    const int items = tp.nch * rs;
    const double item_bytes = rstep * row_bytes / tp.nch;
    const double t_win =
        std::max(rb * row_bytes / (sm_rate / kGroups),
                 ((items + kGroupWarps - 1) / kGroupWarps) * item_bytes / warp_bytes_per_us(tp.RW));
    const long long wins = (long long)n_items * ((N + rb - 1) / rb);
    const long long slots = (long long)kGroups * sms;
    const double est = (double)((wins + slots - 1) / slots) * t_win;
    if (best < 0.0 || est <= best * (1.0 + 1e-9)) {
      best = est;
      *rb_out = rb;
      *tile_out = tb;
      *est_out = est;
    }
  }
  return best >= 0.0;
}

// The plan of one instantiation: stages and windows with the shortest
// estimated chain (more stages unless fewer are clearly faster).
double plan_inst(const w4_gemv_task* tasks, int n, const DeviceInfo& di, int inst, ChainPlan* out) {
  ChainPlan& pl = *out;
  pl.inst = inst;
  const Inst& in = kInst[inst];
  int kgp_max = 0;
  for (int j = 0; j < n; ++j) {
    TaskPlan& tp = pl.t[j];
    const int K = tasks[j].K;
    tp.spec = (in.a.TT == 0 || K == in.Ka) ? 0 : 1;
    const Spec& sp = tp.spec == 0 ? in.a : in.b;
    tp.RW = sp.RW;
    row_shape(K, &tp.T, &tp.NI, &tp.CL, &tp.nch);
    kgp_max = std::max(kgp_max, tp.NI * tp.T);
  }
  const long long optin = di.smem_optin > 0 ? di.smem_optin : 232448;
  const long long xbytes = (long long)kgp_max * (64 + 4);
  double best_est = -1.0;
  static thread_local TaskPlan trial[W4_CHAIN_MAX_TASKS];
  for (int nst = kMaxStages; nst >= 2; --nst) {
    const long long room = optin - kHdrBytes - xbytes;
    long long cap = std::min(kStageMax, room / nst);
    cap &= ~127LL;
    if (cap <= 0) continue;
    double est_sum = 0.0;
    int red_slot = 0, stage = 0;
    bool ok = true;
    for (int j = 0; j < n && ok; ++j) {
      trial[j] = pl.t[j];
      double est = 0.0;
      ok = pick_window(tasks[j].K, tasks[j].N, tasks[j].ids ? tasks[j].n_ids : 1, trial[j], cap,
                       nst, std::max(1, di.sms), &trial[j].RB, &trial[j].tile, &est);
      est_sum += est;
      if (trial[j].nch > 1) red_slot = std::max(red_slot, trial[j].RB * trial[j].nch);
      stage = std::max(stage, trial[j].tile);
    }
    if (!ok) continue;
    const long long red_bytes = ((long long)red_slot * 4 + 15) & ~15LL;
    const long long smem = kHdrBytes + (long long)nst * (stage + red_bytes) + xbytes;
    if (smem > optin) continue;
    if (best_est < 0.0 || est_sum < 0.99 * best_est) {
      best_est = est_sum;
      pl.nst = nst;
      pl.stage_bytes = stage;
      pl.red_slot = red_slot;
      pl.xs_off = (int)(kHdrBytes + (long long)nst * stage);
      pl.xsc_off = pl.xs_off + kgp_max * 64;
      pl.red_off = (int)(((long long)pl.xsc_off + (long long)kgp_max * 4 + 15) & ~15LL);
      pl.smem = pl.red_off + (long long)nst * red_slot * 4;
      for (int j = 0; j < n; ++j) pl.t[j] = trial[j];
    }
  }
  return best_est;
}

w4_status make_plan(const w4_gemv_task* tasks, int n, const DeviceInfo& di, ChainPlan* out) {
  // the compiled instantiations whose specs serve every task's K, the one
  // with the shortest estimate (the generic loop when none does)
  static thread_local ChainPlan trial;
  double best = -1.0;
  for (int i = 0; i < kInsts; ++i) {
    bool ok = true;
    for (int j = 0; j < n && ok; ++j) {
      const int K = tasks[j].K;
      ok = kInst[i].a.TT == 0 || (K == kInst[i].Ka && spec_fits(kInst[i].a, K)) ||
           (K == kInst[i].Kb && spec_fits(kInst[i].b, K));
    }
    if (!ok) continue;
    // the generic loop only when no compiled pair serves the tasks
    if (kInst[i].a.TT == 0 && best >= 0.0) continue;
    const double est = plan_inst(tasks, n, di, i, &trial);
    if (est >= 0.0 && (best < 0.0 || est < 0.99 * best)) {
      best = est;
      *out = trial;
    }
  }
  if (best < 0.0) return W4_ERR_SHAPE;
  ChainPlan& pl = *out;
  long long total = 0;
  for (int j = 0; j < n; ++j) {
    TaskPlan& tp = pl.t[j];
    tp.windows = (tasks[j].N + tp.RB - 1) / tp.RB;
    total += (long long)tp.windows * (tasks[j].ids ? tasks[j].n_ids : 1);
  }
  if (total >= (1LL << 30)) return W4_ERR_SHAPE;
  pl.total = (int)total;
  return W4_OK;
}

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

w4_status check_tasks(const w4_gemv_task* tasks, int n) {
  if (tasks == nullptr || n < 1) return W4_ERR_ARG;
  if (n > W4_CHAIN_MAX_TASKS) return W4_ERR_SHAPE;
  for (int j = 0; j < n; ++j) {
    const w4_gemv_task& t = tasks[j];
    if (t.y == nullptr || t.qw == nullptr || t.st == nullptr || t.x == nullptr) return W4_ERR_ARG;
    if ((t.flags & ~W4_TASK_SILU_MUL) != 0 || t.N < 1) return W4_ERR_ARG;
    if (t.dep < -1 || t.dep >= j) return W4_ERR_ARG;
    if (t.K < 32 || t.K % 32 != 0 || t.K > W4_MAX_K) return W4_ERR_SHAPE;
    if (!aligned(t.qw, 16) || !aligned(t.st, 16) || !aligned(t.x, 16) || !aligned(t.y, 2))
      return W4_ERR_ALIGN;
    if (t.ids != nullptr) {
      if (t.n_ids < 1 || t.num_experts < 1) return W4_ERR_ARG;
      if (t.x_rows != 1 && t.x_rows != t.n_ids) return W4_ERR_SHAPE;
      if (t.qw_stride < (size_t)t.N * t.K / 2 || t.st_stride < (size_t)t.N * (t.K / 32) * 2)
        return W4_ERR_ARG;
      if (t.qw_stride % 16 != 0 || t.st_stride % 16 != 0) return W4_ERR_ALIGN;
      if (t.qw_stride / 16 > 0xffffffffull || t.st_stride / 16 > 0xffffffffull)
        return W4_ERR_SHAPE;
      if ((long long)t.n_ids * t.N >= (1LL << 31)) return W4_ERR_SHAPE;
    }
  }
  return W4_OK;
}

// Task j may wait for item i of its `dep` alone when both route the same ids
// and item i's activation row is exactly item i's output row of `dep`.
bool dep_per_item(const w4_gemv_task* tasks, int j) {
  const w4_gemv_task& t = tasks[j];
  if (t.dep < 0 || t.ids == nullptr || t.n_ids < 2) return false;
  const w4_gemv_task& d = tasks[t.dep];
  const int row = t.K * ((t.flags & W4_TASK_SILU_MUL) ? 2 : 1);
  return d.ids == t.ids && d.n_ids == t.n_ids && t.x_rows == t.n_ids && t.x == d.y &&
         row == d.N;
}

cudaError_t allow_smem(KernelFn fn, long long smem, int dev) {
  static std::mutex mu;
  static long long seen[64][kInsts] = {};
  std::lock_guard<std::mutex> lock(mu);
  int idx = -1;
  for (int i = 0; i < kInsts; ++i)
    if (kernel_of(i) == fn) idx = i;
  if (dev < 0 || dev >= 64 || idx < 0) return cudaErrorInvalidValue;
  if (seen[dev][idx] >= smem) return cudaSuccess;
  const cudaError_t r =
      cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (r == cudaSuccess) seen[dev][idx] = smem;
  return r;
}

}  // namespace chain
}  // namespace w4

// ================================================================= C ABI
using namespace w4;

extern "C" size_t w4a16_gemv_chain_workspace_bytes(const w4_gemv_task* tasks, int n_tasks) {
  if (chain::check_tasks(tasks, n_tasks) != W4_OK) return 0;
  size_t counters = 0;
  for (int j = 0; j < n_tasks; ++j) counters += tasks[j].ids ? (size_t)tasks[j].n_ids : 1u;
  return ((counters + 2) * sizeof(int) + 255) & ~(size_t)255;
}

extern "C" w4_status w4a16_gemv_chain_plan(const w4_gemv_task* tasks, int n_tasks,
                                           w4_chain_plan_info* info) {
  if (info == nullptr) return W4_ERR_ARG;
  const w4_status c = chain::check_tasks(tasks, n_tasks);
  if (c != W4_OK) return c;
  DeviceInfo di;
  planning_device(&di);
  static thread_local chain::ChainPlan pl;
  const w4_status s = chain::make_plan(tasks, n_tasks, di, &pl);
  if (s != W4_OK) return s;
  *info = w4_chain_plan_info{};
  info->ctas = di.sms;
  info->threads = chain::kThreads;
  info->instantiation = pl.inst;
  info->stages = pl.nst;
  info->stage_bytes = pl.stage_bytes;
  info->smem_bytes = (int)pl.smem;
  info->windows = pl.total;
  return W4_OK;
}

extern "C" w4_status w4a16_gemv_chain_task_plan(const w4_gemv_task* tasks, int n_tasks, int task,
                                                w4_chain_task_info* info) {
  if (info == nullptr || task < 0 || task >= n_tasks) return W4_ERR_ARG;
  const w4_status c = chain::check_tasks(tasks, n_tasks);
  if (c != W4_OK) return c;
  DeviceInfo di;
  planning_device(&di);
  static thread_local chain::ChainPlan pl;
  const w4_status s = chain::make_plan(tasks, n_tasks, di, &pl);
  if (s != W4_OK) return s;
  const chain::TaskPlan& tp = pl.t[task];
  info->rows_per_window = tp.RB;
  info->rows_per_lane = tp.RW;
  info->team = tp.T;
  info->chunk_steps = tp.CL;
  info->chunks = tp.nch;
  info->windows_per_item = tp.windows;
  info->dot = tp.spec;
  return W4_OK;
}

extern "C" w4_status w4a16_gemv_chain(const w4_gemv_task* tasks, int n_tasks, void* workspace,
                                      size_t workspace_bytes, int32_t* status_dev, unsigned flags,
                                      w4_stream_t stream) {
  const w4_status c = chain::check_tasks(tasks, n_tasks);
  if (c != W4_OK) return c;
  if ((flags & ~W4_FLAG_PDL) != 0) return W4_ERR_ARG;
  if (workspace == nullptr || workspace_bytes < w4a16_gemv_chain_workspace_bytes(tasks, n_tasks))
    return W4_ERR_WORKSPACE;
  if (!chain::aligned(workspace, 16)) return W4_ERR_ALIGN;
  int dev = 0;
  DeviceInfo di;
  if (!current_device(&dev, &di)) return W4_ERR_DEVICE;
  static thread_local chain::ChainPlan pl;
  static thread_local chain::Params prm;
  const w4_status s = chain::make_plan(tasks, n_tasks, di, &pl);
  if (s != W4_OK) return s;
  prm.n_tasks = n_tasks;
  prm.n_counters = 0;
  for (int j = 0; j < n_tasks; ++j) prm.n_counters += tasks[j].ids ? tasks[j].n_ids : 1;
  prm.total = pl.total;
  prm.nst = pl.nst;
  prm.stage_bytes = pl.stage_bytes;
  prm.xs_off = pl.xs_off;
  prm.xsc_off = pl.xsc_off;
  prm.red_off = pl.red_off;
  prm.red_slot = pl.red_slot;
  prm.ws = static_cast<int*>(workspace);
  prm.status = status_dev;
  int wbase = 0, cbase = 0;
  for (int j = 0; j < n_tasks; ++j) {
    const w4_gemv_task& t = tasks[j];
    const chain::TaskPlan& tp = pl.t[j];
    chain::Task& d = prm.tasks[j];
    d = chain::Task{};
    d.qw = static_cast<const uint8_t*>(t.qw);
    d.st = static_cast<const uint8_t*>(t.st);
    d.x = static_cast<const __nv_bfloat16*>(t.x);
    d.y = static_cast<__nv_bfloat16*>(t.y);
    d.ids = t.ids;
    d.qw_stride16 = t.ids ? (uint32_t)(t.qw_stride / 16) : 0u;
    d.st_stride16 = t.ids ? (uint32_t)(t.st_stride / 16) : 0u;
    d.N = t.N;
    d.K = t.K;
    d.wbase = wbase;
    d.wpi = tp.windows;
    d.n_items = t.ids ? t.n_ids : 1;
    d.num_experts = t.ids ? t.num_experts : 1;
    d.dep = t.dep;
    d.cbase = cbase;
    cbase += d.n_items;
    d.RB = (int16_t)tp.RB;
    d.spec = (uint8_t)tp.spec;
    d.T = (uint8_t)tp.T;
    d.CL = (uint8_t)tp.CL;
    d.nch = (uint8_t)tp.nch;
    d.NI = (uint16_t)tp.NI;
    d.flags = (uint8_t)(((t.flags & W4_TASK_SILU_MUL) ? chain::kTaskGated : 0u) |
                        ((t.ids && t.x_rows == t.n_ids && t.n_ids > 1) ? chain::kTaskXPerItem : 0u) |
                        (chain::dep_per_item(tasks, j) ? chain::kTaskDepPerItem : 0u));
    wbase += tp.windows * d.n_items;
  }
  const chain::KernelFn fn = chain::kernel_of(pl.inst);
  cudaError_t e = chain::allow_smem(fn, pl.smem, dev);
  if (e == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)di.sms);
    cfg.blockDim = dim3(chain::kThreads);
    cfg.dynamicSmemBytes = (size_t)pl.smem;
    cfg.stream = reinterpret_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = (flags & W4_FLAG_PDL) ? 1 : 0;
    e = cudaLaunchKernelEx(&cfg, fn, prm);
  }
  if (e != cudaSuccess) {
    note_cuda_error(e);
    cudaGetLastError();
    return W4_ERR_LAUNCH;
  }
  return W4_OK;
}
