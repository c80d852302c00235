// Row gather from a 4-bit vocabulary table (embed_tokens / per-layer table).
//
// Page "Gemma 4 on a 4 GB GPU in Plain PyTorch", section "Step 2 — Keep the
// Vocabulary Tables in 4-Bit": the tables stay 4-bit with a 16-bit step per
// group of 32 and are looked up by token id on the GPU; the tied table also
// feeds the output GEMV.  out[t][k] = bf16((code - 8) * step): the product
// is exact in fp32, so the single rounding makes the result bit-exact.
//
// One thread per packed word (8 outputs, one 16-byte store); grid.y = token.
#include "common.cuh"

namespace w4 {

__global__ void __launch_bounds__(256) gather_kernel(__nv_bfloat16* __restrict__ out,
                                                      const uint32_t* __restrict__ qw,
                                                      const uint16_t* __restrict__ st,
                                                      const int32_t* __restrict__ ids, int V,
                                                      int K, int32_t* status) {
  pdl_wait();   // ids and the output may belong to the previous kernel
  const int t = blockIdx.y;
  const int id = __ldg(ids + t);
  if (id < 0 || id >= V) {
    if (threadIdx.x == 0 && blockIdx.x == 0) report(status, W4_ERR_INDEX);
    return;
  }
  const int words = K / 8;
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= words) return;
  const long long row = id;
  const uint32_t wd = __ldg(qw + row * words + j);
  const float s = bf16_bits_to_float(__ldg(st + row * (K / 32) + j / 4));
  uint32_t packed[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float lo = (float)((int)((wd >> (8 * i)) & 0xF) - 8) * s;
    const float hi = (float)((int)((wd >> (8 * i + 4)) & 0xF) - 8) * s;
    const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
    packed[i] = *reinterpret_cast<const uint32_t*>(&b);
  }
  *reinterpret_cast<uint4*>(out + (long long)t * K + 8LL * j) =
      make_uint4(packed[0], packed[1], packed[2], packed[3]);
}

}  // namespace w4

using namespace w4;

extern "C" w4_status w4_embed_gather(void* out, const void* qw, const void* st,
                                     const int32_t* ids, int T, int V, int K, int32_t* status_dev,
                                     unsigned flags, w4_stream_t stream) {
  if (out == nullptr || qw == nullptr || st == nullptr || ids == nullptr) return W4_ERR_ARG;
  if (T < 1 || V < 1 || (flags & ~W4_FLAG_PDL) != 0) return W4_ERR_ARG;
  if (K < 32 || K % 32 != 0 || K > W4_MAX_K) return W4_ERR_SHAPE;
  if ((reinterpret_cast<uintptr_t>(out) | reinterpret_cast<uintptr_t>(qw) |
       reinterpret_cast<uintptr_t>(st)) % 16 != 0 ||
      reinterpret_cast<uintptr_t>(ids) % 4 != 0)
    return W4_ERR_ALIGN;
  if (T > 65535) return W4_ERR_SHAPE;
  const int words = K / 8;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((words + 255) / 256), (unsigned)T);
  cfg.blockDim = dim3(256);
  cfg.stream = reinterpret_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = (flags & W4_FLAG_PDL) ? 1 : 0;
  if (cudaLaunchKernelEx(&cfg, gather_kernel, static_cast<__nv_bfloat16*>(out),
                         static_cast<const uint32_t*>(qw), static_cast<const uint16_t*>(st), ids, V,
                         K, status_dev) != cudaSuccess) {
    note_cuda_error(cudaGetLastError());
    return W4_ERR_LAUNCH;
  }
  return W4_OK;
}
