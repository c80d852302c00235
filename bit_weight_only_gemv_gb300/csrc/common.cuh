// Shared device helpers for the W4A16 kernels (sm_103a): status reporting,
// mbarrier + bulk-copy (TMA) wrappers, programmatic-dependent-launch controls.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/w4a16.h"

namespace w4 {

// ---------------------------------------------------------------- status
// Record the first device-side error in the caller's status word (if any).
__device__ __forceinline__ void report(int32_t* status, int code) {
  if (status != nullptr) atomicCAS(reinterpret_cast<int*>(status), 0, code);
}

// ---------------------------------------------------------------- PDL
// With W4_FLAG_PDL the kernel is launched as a programmatic dependent of the
// previous kernel in the stream.  Both instructions are no-ops otherwise.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- L2 prefetch
// Byte ranges to bring into L2 once a launch has requested its own tiles
// (w4a16_gemv_prefetch_l2): normally the next call's weights, so that HBM
// keeps streaming while this launch finishes and the next one starts.
// Addresses are 16-byte aligned; a range's last bytes past a multiple of 16
// are left out (the bulk prefetch moves whole 16-byte units).
constexpr int kMaxL2Ranges = W4_MAX_L2_RANGES;
struct L2Ranges {
  const uint8_t* ptr[kMaxL2Ranges];
  unsigned long long bytes[kMaxL2Ranges];
  int n;
};

// This CTA's share of the ranges, in order: the ranges' bytes are cut into
// `ctas` consecutive shares (16-byte multiples); lane l of the calling warp
// issues the share's chunks l, l + 32, ... of at most kL2Chunk bytes each.
// Fire and forget: nothing waits for the data, and nothing is written.
constexpr unsigned long long kL2Chunk = 16384;
__device__ __forceinline__ void l2_prefetch_share(const L2Ranges& r, int cta, int ctas, int lane) {
  unsigned long long total = 0;
  for (int i = 0; i < r.n; ++i) total += r.bytes[i] & ~15ull;
  if (total == 0) return;
  const unsigned long long share = ((total + ctas - 1) / ctas + 15) & ~15ull;
  unsigned long long lo = share * (unsigned long long)cta;
  const unsigned long long hi = min(total, lo + share);
  unsigned long long base = 0;   // offset of range i within the concatenation
  for (int i = 0; i < r.n && lo < hi; ++i) {
    const unsigned long long len = r.bytes[i] & ~15ull;
    if (lo < base + len) {
      const unsigned long long a = lo - base, b = min(len, hi - base);
      const unsigned long long nchunks = (b - a + kL2Chunk - 1) / kL2Chunk;
      for (unsigned long long c = lane; c < nchunks; c += 32) {
        const unsigned long long o = a + c * kL2Chunk;
        const uint32_t n = (uint32_t)min(kL2Chunk, b - o);
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(r.ptr[i] + o), "r"(n)
                     : "memory");
      }
      lo = base + b;
    }
    base += len;
  }
}

// ---------------------------------------------------------------- smem
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make the initialised barriers visible to the asynchronous (bulk-copy) proxy.
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// One arrival that also announces `bytes` of incoming bulk-copy data.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
               "r"(bytes)
               : "memory");
}

// One plain arrival (release: this thread's earlier accesses happen before).
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with the given parity to complete.  Gives up
// after roughly `limit_cycles` SM clock cycles and returns false; the caller
// records W4_ERR_TIMEOUT and leaves the kernel in an orderly way.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  long long limit_cycles) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (clock64() - t0 > limit_cycles) return false;
  }
}

// ---------------------------------------------------------------- bulk copy
// Order this thread's earlier generic-proxy shared-memory accesses before
// later asynchronous-proxy (bulk copy) writes to the same buffers.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 1-D bulk copy global -> shared, completion counted on `bar` in bytes.
// dst, src 16-byte aligned; bytes a positive multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Same, with an L2 eviction-priority hint (the weights are streamed once).
__device__ __forceinline__ void bulk_g2s_evict_first(uint32_t dst, const void* src,
                                                     uint32_t bytes, uint32_t bar,
                                                     uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], "
      "[%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ---------------------------------------------------------------- misc
__device__ __forceinline__ float bf16_bits_to_float(uint32_t b16) {
  return __uint_as_float(b16 << 16);
}

// Atomic add with acquire-release semantics at GPU scope; returns the old
// value.  Publishes the caller's earlier stores (and those ordered before it
// by a barrier) and makes stores published by earlier releases visible.
__device__ __forceinline__ int atomic_add_acq_rel_gpu(int* p, int v) {
  int old;
  asm volatile("atom.add.acq_rel.gpu.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// (a & b) | c in one LOP3.
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// Host: remember the text of the last CUDA error behind a W4_ERR_LAUNCH /
// W4_ERR_DEVICE return (per thread), for w4_last_cuda_error().
void note_cuda_error(cudaError_t e);

}  // namespace w4
