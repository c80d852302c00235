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

namespace w4 {
namespace {

constexpr int kMaxK = 64;       // ids per request
constexpr int kMaxSlots = 64;   // slots per pool

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

// One thread: the remap of one request.  On an invalid request (an id out of
// range, more distinct ids than slots) the state is left unchanged, the slot
// ids become -1 (the routed GEMV then leaves those rows unwritten) and the
// error goes to *status.  Slots about to be refilled are marked as holding no
// expert in the slot table until the fill kernel has copied them.
__global__ void dev_pool_remap_kernel(uint8_t* st, int E, int S, const int32_t* ids, int k,
                                      int32_t* slot_ids, int32_t* slot_expert, int32_t* status) {
  pdl_wait();   // the ids come from earlier kernels
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  const Layout l = layout(E, S);
  long long* hdr = reinterpret_cast<long long*>(st);
  long long* count = reinterpret_cast<long long*>(st + l.count);
  long long* last_use = reinterpret_cast<long long*>(st + l.last_use);
  int* slot_of = reinterpret_cast<int*>(st + l.slot_of);
  int* in_slot = reinterpret_cast<int*>(st + l.in_slot);
  int* n_miss = reinterpret_cast<int*>(st + l.n_miss);
  int* miss_e = reinterpret_cast<int*>(st + l.miss_e);
  int* miss_s = reinterpret_cast<int*>(st + l.miss_s);
  int* okp = reinterpret_cast<int*>(st + l.ok);
  int id[kMaxK];
  int distinct = 0, bad = 0;
  for (int i = 0; i < k; ++i) {
    id[i] = ids[i];
    if (id[i] < 0 || id[i] >= E) bad = W4_ERR_INDEX;
  }
  if (!bad) {
    for (int i = 0; i < k; ++i) {
      bool seen = false;
      for (int j = 0; j < i; ++j) seen = seen || id[j] == id[i];
      distinct += seen ? 0 : 1;
    }
    if (distinct > S) bad = W4_ERR_STATE;
  }
  *n_miss = 0;
  *okp = bad ? 0 : 1;
  if (bad) {
    for (int i = 0; i < k; ++i) slot_ids[i] = -1;
    report(status, bad);
    return;
  }
  const long long t = hdr[0];
  for (int i = 0; i < k; ++i) count[id[i]] += 1;
  int out[kMaxK];
  long long hits = 0;
  for (int i = 0; i < k; ++i) {
    const int s = slot_of[id[i]];
    out[i] = s;
    if (s >= 0) {
      last_use[s] = t;
      ++hits;
    }
  }
  int nm = 0;
  for (int i = 0; i < k; ++i) {
    if (out[i] >= 0) continue;
    const int e = id[i];
    int s = slot_of[e];   // loaded earlier in this request
    if (s < 0) {
      for (int j = 0; j < S && s < 0; ++j)
        if (in_slot[j] < 0) s = j;
      if (s < 0) {
        for (int j = 0; j < S; ++j) {
          const int ej = in_slot[j];
          bool needed = false;
          for (int q = 0; q < k; ++q) needed = needed || id[q] == ej;
          if (needed) continue;
          if (s < 0) {
            s = j;
            continue;
          }
          const int es = in_slot[s];
          if (count[ej] < count[es] || (count[ej] == count[es] && last_use[j] < last_use[s]))
            s = j;   // ties on both keep the lower index
        }
        slot_of[in_slot[s]] = -1;
      }
      in_slot[s] = e;
      slot_of[e] = s;
      miss_e[nm] = e;
      miss_s[nm] = s;
      ++nm;
      if (slot_expert != nullptr) slot_expert[s] = -1;   // until its copy is in
    } else {
      ++hits;
    }
    last_use[s] = t;
    out[i] = s;
  }
  *n_miss = nm;
  hdr[0] = t + 1;
  hdr[1] += k;
  hdr[2] += hits;
  hdr[3] += nm;
  for (int i = 0; i < k; ++i) slot_ids[i] = out[i];
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

// Kernel-readable address of `ptr` (device memory of the current device,
// managed memory, page-locked host memory), nullptr otherwise.
const void* kernel_view(const void* ptr) {
  int dev = 0;
  cudaPointerAttributes a = {};
  if (cudaGetDevice(&dev) != cudaSuccess || cudaPointerGetAttributes(&a, ptr) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  switch (a.type) {
    case cudaMemoryTypeDevice: return a.device == dev ? ptr : nullptr;
    case cudaMemoryTypeManaged: return ptr;
    case cudaMemoryTypeHost: return a.devicePointer;
    default: return nullptr;
  }
}

cudaError_t launch_pdl(const void* fn, dim3 grid, dim3 block, bool pdl, cudaStream_t s,
                       void** args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
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
  if (num_experts < 1 || num_slots < 1 || num_slots > kMaxSlots) return 0;
  return layout(num_experts, num_slots).bytes;
}

extern "C" w4_status w4_dev_pool_init(void* state, int num_experts, int num_slots,
                                      w4_stream_t stream) {
  if (state == nullptr || num_experts < 1 || num_slots < 1) return W4_ERR_ARG;
  if (num_slots > kMaxSlots || num_slots > num_experts) return W4_ERR_SHAPE;
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
  if (k > kMaxK || num_slots > kMaxSlots || num_slots > num_experts) return W4_ERR_SHAPE;
  if (qw_expert_bytes > qw_stride_bytes || st_expert_bytes > st_stride_bytes ||
      qw_expert_bytes == 0 || st_expert_bytes == 0)
    return W4_ERR_ARG;
  const void* src_qw = kernel_view(full_qw);
  const void* src_st = kernel_view(full_st);
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
                             dim3(32), pdl, s, rargs);
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
    // enough threads for k misses; blocks past the request's misses exit at once
    const unsigned long long units = (fp.qw_units + fp.st_units) * (unsigned long long)k;
    const int blocks = (int)std::max(1ULL, std::min(1024ULL, (units + 255) / 256));
    void* fargs[] = {&fp};
    e = launch_pdl(reinterpret_cast<const void*>(dev_pool_fill_kernel), dim3(blocks), dim3(256),
                   true, s, fargs);
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
