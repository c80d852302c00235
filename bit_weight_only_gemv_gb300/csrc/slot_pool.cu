// Per-layer expert slot pool (host C++), plus the kernels that load missed
// experts into their slots and publish the slot ids to the device.
//
// Page "Running a 26B MoE on an 8 GB Jetson by streaming experts from SSD",
// section "Streaming without touching a single GPU kernel": every MoE layer
// owns a long-lived set of slots, each the size of one expert, and a short
// tensor of slot numbers.  An LFU policy leaves resident experts where they
// are, copies missing ones into the slots it picks and fills in the slot
// numbers before the expert matmul runs; addressed through those numbers, the
// pool hands the matmul the same bytes as the full expert tensor would.  Here the
// misses are copied from the full expert tensor, held in HBM or in page-locked
// Grace memory that the GPU reads in place over NVLink-C2C (the page reads
// them from an SSD into host memory the Jetson's GPU shares).  An optional
// device slot table names the expert each slot holds, so that consumers of
// the real expert ids can check what a slot id points at.
//
// Policy (the page leaves it open): every requested id counts one use; hits
// stay; misses, in request order, take the lowest free slot, else the slot
// whose expert is not requested now and has the fewest uses, then the least
// recently used, then the lowest index; a repeated id shares one slot.
#include <algorithm>
#include <unordered_set>
#include <vector>

#include "common.cuh"
#include "pointer_view.h"

struct w4_slot_pool {
  int num_experts = 0;
  int num_slots = 0;
  std::vector<long long> count;        // per expert
  std::vector<int> expert_in_slot;     // -1 = free
  std::vector<int> slot_of_expert;     // -1 = not resident
  std::vector<long long> last_use;     // per slot
  long long step = 0;
  long long requests = 0, hits = 0, misses = 0;
};

namespace w4 {

struct IdList {
  int32_t v[64];
};

// Entries of the device slot table: table[slot[i]] = expert[i].
struct SlotEntries {
  int32_t slot[64], expert[64];
  int n;
};

__global__ void write_ids_kernel(int32_t* dst, IdList ids, int k, int32_t* table,
                                 SlotEntries t) {
  const int i = threadIdx.x;
  if (dst != nullptr && i < k) dst[i] = ids.v[i];
  if (table != nullptr && i < t.n) table[t.slot[i]] = t.expert[i];
}

// One launch that loads a request's missed experts into their slots (codes
// and steps, 16 bytes per thread step), writes the request's slot ids and
// names the new experts in the slot table.  Kernels later in the stream see
// all of it at once, so the table needs no ordering inside the launch.
struct FillParams {
  uint8_t* pool_qw;
  const uint8_t* full_qw;
  uint8_t* pool_st;
  const uint8_t* full_st;
  unsigned long long qw_stride, st_stride;   // bytes between experts / slots
  unsigned long long qw_units, st_units;     // 16-byte units per expert
  int32_t* slot_ids_dev;
  int32_t* slot_expert_dev;                  // slot table, or nullptr
  int n_miss, k;
  int32_t miss_expert[64], miss_slot[64];
  int32_t ids[64];
};

__global__ void __launch_bounds__(256) pool_fill_kernel(const __grid_constant__ FillParams p) {
  if (blockIdx.x == 0 && threadIdx.x < p.k) p.slot_ids_dev[threadIdx.x] = p.ids[threadIdx.x];
  if (blockIdx.x == 0 && p.slot_expert_dev != nullptr && threadIdx.x < p.n_miss)
    p.slot_expert_dev[p.miss_slot[threadIdx.x]] = p.miss_expert[threadIdx.x];
  const unsigned long long per = p.qw_units + p.st_units;
  const unsigned long long total = per * (unsigned long long)p.n_miss;
  for (unsigned long long u = (unsigned long long)blockIdx.x * blockDim.x + threadIdx.x; u < total;
       u += (unsigned long long)gridDim.x * blockDim.x) {
    const int m = (int)(u / per);
    const unsigned long long r = u - (unsigned long long)m * per;
    const unsigned long long e = (unsigned long long)p.miss_expert[m];
    const unsigned long long sl = (unsigned long long)p.miss_slot[m];
    if (r < p.qw_units) {
      reinterpret_cast<uint4*>(p.pool_qw + sl * p.qw_stride)[r] =
          __ldcs(reinterpret_cast<const uint4*>(p.full_qw + e * p.qw_stride) + r);
    } else {
      const unsigned long long q = r - p.qw_units;
      reinterpret_cast<uint4*>(p.pool_st + sl * p.st_stride)[q] =
          __ldcs(reinterpret_cast<const uint4*>(p.full_st + e * p.st_stride) + q);
    }
  }
}

const void* device_view(const void* ptr) {
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

namespace {

w4_status remap(w4_slot_pool* p, const int32_t* ids, int k, int32_t* slot_ids,
                std::vector<std::pair<int, int>>* miss_list) {
  std::unordered_set<int> needed;
  for (int i = 0; i < k; ++i) {
    if (ids[i] < 0 || ids[i] >= p->num_experts) return W4_ERR_INDEX;
    needed.insert(ids[i]);
  }
  if ((int)needed.size() > p->num_slots) return W4_ERR_STATE;
  const long long t = p->step;
  for (int i = 0; i < k; ++i) p->count[ids[i]] += 1;
  std::vector<int> out(k, -1);
  for (int i = 0; i < k; ++i) {
    const int s = p->slot_of_expert[ids[i]];
    if (s >= 0) {
      out[i] = s;
      p->last_use[s] = t;
      p->hits += 1;
    }
  }
  for (int i = 0; i < k; ++i) {
    if (out[i] >= 0) continue;
    const int e = ids[i];
    int s = p->slot_of_expert[e];   // loaded earlier in this request
    if (s < 0) {
      for (int j = 0; j < p->num_slots && s < 0; ++j)
        if (p->expert_in_slot[j] < 0) s = j;
      if (s < 0) {
        for (int j = 0; j < p->num_slots; ++j) {
          const int ej = p->expert_in_slot[j];
          if (needed.count(ej)) continue;
          if (s < 0) {
            s = j;
            continue;
          }
          const int es = p->expert_in_slot[s];
          if (p->count[ej] < p->count[es] ||
              (p->count[ej] == p->count[es] && p->last_use[j] < p->last_use[s]))
            s = j;   // ties on both keep the lower index
        }
        p->slot_of_expert[p->expert_in_slot[s]] = -1;
      }
      p->expert_in_slot[s] = e;
      p->slot_of_expert[e] = s;
      miss_list->emplace_back(e, s);
      p->misses += 1;
    } else {
      p->hits += 1;
    }
    p->last_use[s] = t;
    out[i] = s;
  }
  p->requests += k;
  p->step += 1;
  for (int i = 0; i < k; ++i) slot_ids[i] = out[i];
  return W4_OK;
}

}  // namespace
}  // namespace w4

using namespace w4;

extern "C" w4_status w4_slot_pool_create(w4_slot_pool** pool, int num_experts, int num_slots) {
  if (pool == nullptr || num_experts < 1 || num_slots < 1) return W4_ERR_ARG;
  w4_slot_pool* p = new (std::nothrow) w4_slot_pool();
  if (p == nullptr) return W4_ERR_ARG;
  p->num_experts = num_experts;
  p->num_slots = num_slots;
  p->count.assign(num_experts, 0);
  p->slot_of_expert.assign(num_experts, -1);
  p->expert_in_slot.assign(num_slots, -1);
  p->last_use.assign(num_slots, -1);
  *pool = p;
  return W4_OK;
}

extern "C" void w4_slot_pool_destroy(w4_slot_pool* pool) { delete pool; }

extern "C" w4_status w4_slot_pool_remap(w4_slot_pool* pool, const int32_t* expert_ids, int k,
                                        int32_t* slot_ids, int32_t* miss_experts,
                                        int32_t* miss_slots, int* n_miss) {
  if (pool == nullptr || expert_ids == nullptr || slot_ids == nullptr || k < 1) return W4_ERR_ARG;
  std::vector<std::pair<int, int>> misses;
  const w4_status st = remap(pool, expert_ids, k, slot_ids, &misses);
  if (st != W4_OK) return st;
  for (size_t i = 0; i < misses.size(); ++i) {
    if (miss_experts) miss_experts[i] = misses[i].first;
    if (miss_slots) miss_slots[i] = misses[i].second;
  }
  if (n_miss) *n_miss = (int)misses.size();
  return W4_OK;
}

extern "C" w4_status w4_slot_pool_stage(w4_slot_pool* pool, const int32_t* expert_ids, int k,
                                        void* pool_qw, const void* full_qw,
                                        size_t qw_stride_bytes, size_t qw_expert_bytes,
                                        void* pool_st, const void* full_st,
                                        size_t st_stride_bytes, size_t st_expert_bytes,
                                        int32_t* slot_ids_dev, int32_t* slot_expert_dev,
                                        int32_t* slot_ids, int* n_miss, w4_stream_t stream) {
  if (pool == nullptr || expert_ids == nullptr || pool_qw == nullptr || full_qw == nullptr ||
      pool_st == nullptr || full_st == nullptr || slot_ids_dev == nullptr || k < 1)
    return W4_ERR_ARG;
  if (k > 64) return W4_ERR_SHAPE;
  if (qw_expert_bytes > qw_stride_bytes || st_expert_bytes > st_stride_bytes) return W4_ERR_ARG;
  IdList list = {};
  std::vector<std::pair<int, int>> misses;
  const w4_status st = remap(pool, expert_ids, k, list.v, &misses);
  if (st != W4_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  bool failed = false;
  // sources the kernels can read, everything 16-byte aligned: one kernel
  // loads the misses and writes the slot ids
  const auto a16 = [](const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15) == 0; };
  const void* src_qw = misses.empty() ? full_qw : device_view(full_qw);
  const void* src_st = misses.empty() ? full_st : device_view(full_st);
  if (src_qw != nullptr && src_st != nullptr && a16(pool_qw) && a16(src_qw) && a16(pool_st) &&
      a16(src_st) && qw_stride_bytes % 16 == 0 && st_stride_bytes % 16 == 0 &&
      qw_expert_bytes % 16 == 0 && st_expert_bytes % 16 == 0) {
    FillParams fp = {};
    fp.pool_qw = static_cast<uint8_t*>(pool_qw);
    fp.full_qw = static_cast<const uint8_t*>(src_qw);
    fp.pool_st = static_cast<uint8_t*>(pool_st);
    fp.full_st = static_cast<const uint8_t*>(src_st);
    fp.qw_stride = qw_stride_bytes;
    fp.st_stride = st_stride_bytes;
    fp.qw_units = qw_expert_bytes / 16;
    fp.st_units = st_expert_bytes / 16;
    fp.slot_ids_dev = slot_ids_dev;
    fp.slot_expert_dev = slot_expert_dev;
    fp.n_miss = (int)misses.size();
    fp.k = k;
    for (int i = 0; i < fp.n_miss; ++i) {
      fp.miss_expert[i] = misses[i].first;
      fp.miss_slot[i] = misses[i].second;
    }
    std::copy(list.v, list.v + k, fp.ids);
    const unsigned long long total = (fp.qw_units + fp.st_units) * (unsigned long long)fp.n_miss;
    const int blocks = (int)std::max(1ULL, std::min(1024ULL, (total + 255) / 256));
    pool_fill_kernel<<<blocks, 256, 0, s>>>(fp);
    failed = cudaPeekAtLastError() != cudaSuccess;
    if (failed) {
      note_cuda_error(cudaGetLastError());
      for (const auto& m : misses) {
        if (pool->expert_in_slot[m.second] == m.first) {
          pool->expert_in_slot[m.second] = -1;
          pool->slot_of_expert[m.first] = -1;
        }
      }
      return W4_ERR_STATE;
    }
    if (slot_ids) std::copy(list.v, list.v + k, slot_ids);
    if (n_miss) *n_miss = (int)misses.size();
    return W4_OK;
  }
  // Copies one by one: the refilled slots hold no expert until every copy is
  // in (a copy that fails to enqueue leaves them so).
  SlotEntries entries = {};
  entries.n = (int)misses.size();
  for (int i = 0; i < entries.n; ++i) {
    entries.slot[i] = misses[i].second;
    entries.expert[i] = -1;
  }
  if (slot_expert_dev != nullptr && entries.n > 0) {
    write_ids_kernel<<<1, 64, 0, s>>>(nullptr, list, 0, slot_expert_dev, entries);
    failed = cudaPeekAtLastError() != cudaSuccess;
  }
  for (size_t i = 0; i < misses.size() && !failed; ++i) {
    const size_t e = (size_t)misses[i].first, slot = (size_t)misses[i].second;
    if (cudaMemcpyAsync(static_cast<uint8_t*>(pool_qw) + slot * qw_stride_bytes,
                        static_cast<const uint8_t*>(full_qw) + e * qw_stride_bytes,
                        qw_expert_bytes, cudaMemcpyDefault, s) != cudaSuccess ||
        cudaMemcpyAsync(static_cast<uint8_t*>(pool_st) + slot * st_stride_bytes,
                        static_cast<const uint8_t*>(full_st) + e * st_stride_bytes,
                        st_expert_bytes, cudaMemcpyDefault, s) != cudaSuccess)
      failed = true;
  }
  if (!failed) {
    for (int i = 0; i < entries.n; ++i) entries.expert[i] = misses[i].first;
    write_ids_kernel<<<1, 64, 0, s>>>(slot_ids_dev, list, k, slot_expert_dev, entries);
    failed = cudaPeekAtLastError() != cudaSuccess;
  }
  if (failed) {
    note_cuda_error(cudaGetLastError());
    // forget every expert this request was loading: their slots hold nothing valid
    for (const auto& m : misses) {
      if (pool->expert_in_slot[m.second] == m.first) {
        pool->expert_in_slot[m.second] = -1;
        pool->slot_of_expert[m.first] = -1;
      }
    }
    return W4_ERR_STATE;
  }
  if (slot_ids) std::copy(list.v, list.v + k, slot_ids);
  if (n_miss) *n_miss = (int)misses.size();
  return W4_OK;
}

extern "C" void w4_slot_pool_stats(const w4_slot_pool* pool, long long* requests,
                                   long long* hits, long long* misses) {
  if (pool == nullptr) return;
  if (requests) *requests = pool->requests;
  if (hits) *hits = pool->hits;
  if (misses) *misses = pool->misses;
}

extern "C" const char* w4_status_str(int status) {
  switch (status) {
    case W4_OK: return "ok";
    case W4_ERR_ARG: return "invalid argument";
    case W4_ERR_ALIGN: return "misaligned pointer or stride";
    case W4_ERR_SHAPE: return "unsupported shape";
    case W4_ERR_WORKSPACE: return "workspace too small";
    case W4_ERR_LAUNCH: return "kernel launch failed";
    case W4_ERR_INDEX: return "id out of range";
    case W4_ERR_VALUE: return "code out of range";
    case W4_ERR_TIMEOUT: return "device wait timed out";
    case W4_ERR_DEVICE: return "no usable CUDA device";
    case W4_ERR_STATE: return "slot pool request cannot be served";
    case W4_ERR_OWNER: return "slot does not hold the named expert";
    default: return "unknown status";
  }
}

extern "C" int w4_abi_version(void) { return W4_ABI_VERSION; }

namespace w4 {
namespace {
thread_local const char* g_last_cuda_error = "no error";
}
void note_cuda_error(cudaError_t e) { g_last_cuda_error = cudaGetErrorString(e); }
}  // namespace w4

extern "C" const char* w4_last_cuda_error(void) { return w4::g_last_cuda_error; }
