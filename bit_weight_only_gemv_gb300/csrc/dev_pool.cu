// Device-side expert slot pool: the LFU remap of a routed request runs on the
// GPU, so a routed decode step (router ids -> remap -> pool fills -> routed
// GEMVs) needs no host round trip per layer and can be captured in a CUDA
// graph.
//
// Page "Running a 26B MoE on an 8 GB Jetson by streaming experts from SSD",
// section "Streaming without touching a single GPU kernel": a per-layer LFU
// cache of expert slots is consulted when the router names the next token's
// experts; hits stay, misses are loaded into their assigned slots, and the
// slot indices are written for the expert matmul.  The page runs the policy
// in a host callback because its misses are disk reads; with the experts in
// HBM or in Grace memory the GPU can decide and copy by itself.
//
// The policy is the host pool's (slot_pool.cu), step for step: every
// requested id counts one use; hits stay; misses, in request order, take the
// lowest free slot, else the slot whose expert is not requested now with the
// fewest uses, then the least recently used, then the lowest index; a
// repeated id shares one slot.
#include <algorithm>

#include "common.cuh"
#include "pointer_view.h"

namespace w4 {
namespace {

constexpr int kMaxK = 64;       // ids per request
constexpr int kMaxSlots = 64;   // slots per pool
constexpr int kMaxExperts = 3980;   // experts per pool: the remap keeps a copy in 48 KB of shared memory

// Device state, 8-byte aligned:
//   int64 step, requests, hits, misses
//   int64 count[E], int64 last_use[S]
//   int32 slot_of_expert[E], int32 expert_in_slot[S]
//   int32 n_miss, miss_expert[kMaxK], miss_slot[kMaxK], ok
struct Layout {
  size_t count, last_use, slot_of, in_slot, n_miss, miss_e, miss_s, ok, bytes;
};

__host__ __device__ inline Layout layout(int E, int S) {
  Layout l;
  size_t o = 4 * sizeof(long long);
  l.count = o;
  o += (size_t)E * sizeof(long long);
  l.last_use = o;
  o += (size_t)S * sizeof(long long);
  l.slot_of = o;
  o += (size_t)E * sizeof(int);
  l.in_slot = o;
  o += (size_t)S * sizeof(int);
  l.n_miss = o;
  o += sizeof(int);
  l.miss_e = o;
  o += kMaxK * sizeof(int);
  l.miss_s = o;
  o += kMaxK * sizeof(int);
  l.ok = o;
  o += sizeof(int);
  l.bytes = (o + 15) & ~size_t(15);
  return l;
}

__global__ void dev_pool_init_kernel(uint8_t* st, int E, int S) {
  const Layout l = layout(E, S);
  long long* hdr = reinterpret_cast<long long*>(st);
  long long* count = reinterpret_cast<long long*>(st + l.count);
  long long* last_use = reinterpret_cast<long long*>(st + l.last_use);
  int* slot_of = reinterpret_cast<int*>(st + l.slot_of);
  int* in_slot = reinterpret_cast<int*>(st + l.in_slot);
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < E + S + 4; i += gridDim.x * blockDim.x) {
    if (i < 4) hdr[i] = 0;
    if (i < E) {
      count[i] = 0;
      slot_of[i] = -1;
    }
    if (i < S) {
      last_use[i] = -1;
      in_slot[i] = -1;
    }
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    *reinterpret_cast<int*>(st + l.n_miss) = 0;
    *reinterpret_cast<int*>(st + l.ok) = 0;
  }
}

// One block: the remap of one request.  The block loads the pool's state
// into shared memory, one thread takes the decisions there (the policy is
// sequential), the block writes the state back.  On an invalid request (an
// id out of range, more distinct ids than slots) the state is left
// unchanged, the slot ids become -1 (the routed GEMV then leaves those rows
// unwritten) and the error goes to *status.  Slots about to be refilled are
// marked as holding no expert in the slot table until the fill kernel has
// copied them.
__global__ void __launch_bounds__(256) dev_pool_remap_kernel(uint8_t* st, int E, int S,
                                                             const int32_t* ids, int k,
                                                             int32_t* slot_ids,
                                                             int32_t* slot_expert,
                                                             int32_t* status) {
  extern __shared__ __align__(16) uint8_t sm[];
  pdl_wait();   // the ids come from earlier kernels
  const Layout l = layout(E, S);
  long long* hdr = reinterpret_cast<long long*>(st);
  long long* g_count = reinterpret_cast<long long*>(st + l.count);
  long long* g_last = reinterpret_cast<long long*>(st + l.last_use);
  int* g_slot_of = reinterpret_cast<int*>(st + l.slot_of);
  int* g_in_slot = reinterpret_cast<int*>(st + l.in_slot);
  // shared copy: count[E], last_use[S], slot_of[E], in_slot[S], ids, flags
  long long* count = reinterpret_cast<long long*>(sm);
  long long* last_use = count + E;
  int* slot_of = reinterpret_cast<int*>(last_use + S);
  int* in_slot = slot_of + E;
  int* id = in_slot + S;
  int* flag = id + kMaxK;   // [0] valid request; the slots of the ids follow at flag + 4
  for (int i = threadIdx.x; i < E; i += blockDim.x) {
    count[i] = g_count[i];
    slot_of[i] = g_slot_of[i];
  }
  for (int i = threadIdx.x; i < S; i += blockDim.x) {
    last_use[i] = g_last[i];
    in_slot[i] = g_in_slot[i];
  }
  for (int i = threadIdx.x; i < k; i += blockDim.x) id[i] = ids[i];
  __syncthreads();
  // Warp 0 takes the decisions, its lanes side by side where the policy
  // allows (checks, hits, the free-slot and victim searches over the slots);
  // the misses themselves are placed one after another, in request order.
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int* n_miss = reinterpret_cast<int*>(st + l.n_miss);
    int* miss_e = reinterpret_cast<int*>(st + l.miss_e);
    int* miss_s = reinterpret_cast<int*>(st + l.miss_s);
    int* out = flag + 4;   // [kMaxK] slot of each id
    // validity: every id in range, at most S distinct ids
    int bad_range = 0, distinct = 0;
    for (int i0 = 0; i0 < k; i0 += 32) {
      const int i = i0 + lane;
      bool inr = true, first = false;
      if (i < k) {
        inr = id[i] >= 0 && id[i] < E;
        first = true;
        for (int j = 0; j < i; ++j) first = first && id[j] != id[i];
      }
      bad_range |= __any_sync(0xffffffffu, !inr);
      distinct += __popc(__ballot_sync(0xffffffffu, first));
    }
    const int bad = bad_range ? W4_ERR_INDEX : (distinct > S ? W4_ERR_STATE : 0);
    if (lane == 0) {
      *n_miss = 0;
      flag[0] = bad ? 0 : 1;
    }
    if (bad) {
      for (int i = lane; i < k; i += 32) slot_ids[i] = -1;
      if (lane == 0) report(status, bad);
    } else {
      const long long t = hdr[0];
      if (lane == 0)
        for (int i = 0; i < k; ++i) count[id[i]] += 1;   // repeats count each time
      __syncwarp();
      // hits: experts resident before this request
      long long hits = 0;
      for (int i0 = 0; i0 < k; i0 += 32) {
        const int i = i0 + lane;
        int s_ = -1;
        if (i < k) {
          s_ = slot_of[id[i]];
          out[i] = s_;
          if (s_ >= 0) last_use[s_] = t;
        }
        hits += __popc(__ballot_sync(0xffffffffu, s_ >= 0));
      }
      __syncwarp();
      int nm = 0;
      for (int i = 0; i < k; ++i) {
        if (out[i] >= 0) continue;   // warp-uniform: shared memory
        const int e = id[i];
        int sl = slot_of[e];         // loaded earlier in this request
        if (sl < 0) {
          // lowest free slot
          for (int j0 = 0; j0 < S; j0 += 32) {
            const int j = j0 + lane;
            const unsigned b = __ballot_sync(0xffffffffu, j < S && in_slot[j] < 0);
            if (sl < 0 && b != 0) sl = j0 + __ffs(b) - 1;
          }
          if (sl < 0) {
            // victim: the slot whose expert is not requested now with the
            // fewest uses, then the least recently used, then the lowest index
            long long bc = 0x7fffffffffffffffLL, bl = 0x7fffffffffffffffLL;
            int bj = 0x7fffffff;
            for (int j = lane; j < S; j += 32) {
              const int ej = in_slot[j];
              bool needed = false;
              for (int q = 0; q < k; ++q) needed = needed || id[q] == ej;
              if (needed) continue;
              const long long c = count[ej], lu = last_use[j];
              if (c < bc || (c == bc && (lu < bl || (lu == bl && j < bj)))) {
                bc = c;
                bl = lu;
                bj = j;
              }
            }
            for (int off = 16; off > 0; off >>= 1) {
              const long long oc = __shfl_xor_sync(0xffffffffu, bc, off);
              const long long ol = __shfl_xor_sync(0xffffffffu, bl, off);
              const int oj = __shfl_xor_sync(0xffffffffu, bj, off);
              if (oc < bc || (oc == bc && (ol < bl || (ol == bl && oj < bj)))) {
                bc = oc;
                bl = ol;
                bj = oj;
              }
            }
            sl = bj;
            if (lane == 0) slot_of[in_slot[sl]] = -1;
          }
          if (lane == 0) {
            in_slot[sl] = e;
            slot_of[e] = sl;
            miss_e[nm] = e;
            miss_s[nm] = sl;
            if (slot_expert != nullptr) slot_expert[sl] = -1;   // until its copy is in
          }
          ++nm;
        } else {
          ++hits;
        }
        if (lane == 0) {
          last_use[sl] = t;
          out[i] = sl;
        }
        __syncwarp();
      }
      if (lane == 0) {
        *n_miss = nm;
        hdr[0] = t + 1;
        hdr[1] += k;
        hdr[2] += hits;
        hdr[3] += nm;
      }
      for (int i = lane; i < k; i += 32) slot_ids[i] = out[i];
    }
  }
  __syncthreads();
  if (flag[0]) {   // write the state back
    for (int i = threadIdx.x; i < E; i += blockDim.x) {
      g_count[i] = count[i];
      g_slot_of[i] = slot_of[i];
    }
    for (int i = threadIdx.x; i < S; i += blockDim.x) {
      g_last[i] = last_use[i];
      g_in_slot[i] = in_slot[i];
    }
  }
}

size_t remap_smem(int E, int S) {
  return (size_t)(E + S) * sizeof(long long) + (size_t)(E + S + 2 * kMaxK + 4) * sizeof(int);
}

// Copies of the remap's misses (16 bytes per thread step), then the slot
// table names the new experts.  Kernels later in the stream see all of it.
struct DevFill {
  uint8_t* st;
  int E, S;
  uint8_t* pool_qw;
  const uint8_t* full_qw;
  uint8_t* pool_st;
  const uint8_t* full_st;
  unsigned long long qw_stride, st_stride, qw_units, st_units;
  int32_t* slot_expert;
};

__global__ void __launch_bounds__(256) dev_pool_fill_kernel(const __grid_constant__ DevFill p) {
  pdl_wait();   // the remap's decision
  const Layout l = layout(p.E, p.S);
  const int nm = *reinterpret_cast<const int*>(p.st + l.n_miss);
  const int* miss_e = reinterpret_cast<const int*>(p.st + l.miss_e);
  const int* miss_s = reinterpret_cast<const int*>(p.st + l.miss_s);
  const unsigned long long per = p.qw_units + p.st_units;
  const unsigned long long total = per * (unsigned long long)nm;
  for (unsigned long long u = (unsigned long long)blockIdx.x * blockDim.x + threadIdx.x; u < total;
       u += (unsigned long long)gridDim.x * blockDim.x) {
    const int m = (int)(u / per);
    const unsigned long long r = u - (unsigned long long)m * per;
    const unsigned long long e = (unsigned long long)miss_e[m];
    const unsigned long long sl = (unsigned long long)miss_s[m];
    if (r < p.qw_units) {
      reinterpret_cast<uint4*>(p.pool_qw + sl * p.qw_stride)[r] =
          __ldcs(reinterpret_cast<const uint4*>(p.full_qw + e * p.qw_stride) + r);
    } else {
      const unsigned long long q = r - p.qw_units;
      reinterpret_cast<uint4*>(p.pool_st + sl * p.st_stride)[q] =
          __ldcs(reinterpret_cast<const uint4*>(p.full_st + e * p.st_stride) + q);
    }
  }
  if (p.slot_expert != nullptr && blockIdx.x == 0 && threadIdx.x < nm)
    p.slot_expert[miss_s[threadIdx.x]] = miss_e[threadIdx.x];
}

cudaError_t launch_pdl(const void* fn, dim3 grid, dim3 block, size_t smem, bool pdl,
                       cudaStream_t s, void** args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace
}  // namespace w4

using namespace w4;

extern "C" size_t w4_dev_pool_state_bytes(int num_experts, int num_slots) {
  if (num_experts < 1 || num_slots < 1 || num_slots > kMaxSlots || num_experts > kMaxExperts)
    return 0;
  return layout(num_experts, num_slots).bytes;
}

extern "C" w4_status w4_dev_pool_init(void* state, int num_experts, int num_slots,
                                      w4_stream_t stream) {
  if (state == nullptr || num_experts < 1 || num_slots < 1) return W4_ERR_ARG;
  if (num_slots > kMaxSlots || num_slots > num_experts || num_experts > kMaxExperts)
    return W4_ERR_SHAPE;
  if ((reinterpret_cast<uintptr_t>(state) & 15) != 0) return W4_ERR_ALIGN;
  const int n = num_experts + num_slots + 4;
  dev_pool_init_kernel<<<std::min(1024, (n + 255) / 256), 256, 0,
                         reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<uint8_t*>(state), num_experts, num_slots);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    note_cuda_error(e);
    return W4_ERR_LAUNCH;
  }
  return W4_OK;
}

extern "C" w4_status w4_dev_pool_stage(void* state, int num_experts, int num_slots,
                                       const int32_t* ids, int k, void* pool_qw,
                                       const void* full_qw, size_t qw_stride_bytes,
                                       size_t qw_expert_bytes, void* pool_st,
                                       const void* full_st, size_t st_stride_bytes,
                                       size_t st_expert_bytes, int32_t* slot_ids_dev,
                                       int32_t* slot_expert_dev, int32_t* status_dev,
                                       unsigned flags, w4_stream_t stream) {
  if (state == nullptr || ids == nullptr || pool_qw == nullptr || full_qw == nullptr ||
      pool_st == nullptr || full_st == nullptr || slot_ids_dev == nullptr || k < 1 ||
      num_experts < 1 || num_slots < 1 || (flags & ~W4_FLAG_PDL) != 0)
    return W4_ERR_ARG;
  if (k > kMaxK || num_slots > kMaxSlots || num_slots > num_experts ||
      num_experts > kMaxExperts)
    return W4_ERR_SHAPE;
  if (qw_expert_bytes > qw_stride_bytes || st_expert_bytes > st_stride_bytes ||
      qw_expert_bytes == 0 || st_expert_bytes == 0)
    return W4_ERR_ARG;
  const void* src_qw = device_view(full_qw);
  const void* src_st = device_view(full_st);
  if (src_qw == nullptr || src_st == nullptr) return W4_ERR_ARG;
  const auto a16 = [](const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15) == 0; };
  if (!a16(state) || !a16(pool_qw) || !a16(src_qw) || !a16(pool_st) || !a16(src_st) ||
      qw_stride_bytes % 16 != 0 || st_stride_bytes % 16 != 0 || qw_expert_bytes % 16 != 0 ||
      st_expert_bytes % 16 != 0 || (reinterpret_cast<uintptr_t>(ids) & 3) != 0)
    return W4_ERR_ALIGN;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool pdl = (flags & W4_FLAG_PDL) != 0;
  uint8_t* st = static_cast<uint8_t*>(state);
  int E = num_experts, S = num_slots, kk = k;
  void* rargs[] = {&st, &E, &S, const_cast<int32_t**>(&ids), &kk, &slot_ids_dev,
                   &slot_expert_dev, &status_dev};
  cudaError_t e = launch_pdl(reinterpret_cast<const void*>(dev_pool_remap_kernel), dim3(1),
                             dim3(256), remap_smem(E, S), pdl, s, rargs);
  if (e == cudaSuccess) {
    DevFill fp = {};
    fp.st = st;
    fp.E = E;
    fp.S = S;
    fp.pool_qw = static_cast<uint8_t*>(pool_qw);
    fp.full_qw = static_cast<const uint8_t*>(src_qw);
    fp.pool_st = static_cast<uint8_t*>(pool_st);
    fp.full_st = static_cast<const uint8_t*>(src_st);
    fp.qw_stride = qw_stride_bytes;
    fp.st_stride = st_stride_bytes;
    fp.qw_units = qw_expert_bytes / 16;
    fp.st_units = st_expert_bytes / 16;
    fp.slot_expert = slot_expert_dev;
    // one block per SM, striding over the misses (their number is only
    // known on the device)
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      sms = 152;
    void* fargs[] = {&fp};
    e = launch_pdl(reinterpret_cast<const void*>(dev_pool_fill_kernel), dim3(std::max(1, sms)),
                   dim3(256), 0, true, s, fargs);
  }
  if (e != cudaSuccess) {
    note_cuda_error(e);
    cudaGetLastError();
    return W4_ERR_LAUNCH;
  }
  return W4_OK;
}

extern "C" w4_status w4_dev_pool_stats(const void* state, int num_experts, int num_slots,
                                       long long* requests, long long* hits,
                                       long long* misses) {
  if (state == nullptr || num_experts < 1 || num_slots < 1 || num_slots > kMaxSlots)
    return W4_ERR_ARG;
  long long hdr[4] = {};
  const cudaError_t e = cudaMemcpy(hdr, state, sizeof(hdr), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) {
    note_cuda_error(e);
    cudaGetLastError();
    return W4_ERR_LAUNCH;
  }
  if (requests) *requests = hdr[1];
  if (hits) *hits = hdr[2];
  if (misses) *misses = hdr[3];
  return W4_OK;
}
