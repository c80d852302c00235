// Pack and quantise helpers for the W4A16 group-32 layout.
//
// w4_pack: 4-bit codes (one per byte) into uint32 words, low nibble first.
// w4_quantize: page "Gemma 4 on a 4 GB GPU in Plain PyTorch", section "Step 2 —
// Keep the Vocabulary Tables in 4-Bit" recovers each group's step from its
// 4-bit grid; here the plain signed-absmax rule is used, one warp per group:
// m = element of largest |w| (lowest k on ties), step = bf16(m / -8),
// code = 8 if step == 0 else clamp(rint(w / step) + 8, 0, 15) with IEEE fp32
// division (no fast-math) and round-half-even, so it is bit-exact with any
// IEEE implementation of the same steps.
#include "common.cuh"

namespace w4 {

__global__ void __launch_bounds__(256) pack_kernel(uint32_t* __restrict__ qw,
                                                    const uint8_t* __restrict__ codes,
                                                    long long n_words, int32_t* status) {
  const long long j = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= n_words) return;
  const uint2 v = __ldg(reinterpret_cast<const uint2*>(codes) + j);
  const uint32_t b[2] = {v.x, v.y};
  uint32_t word = 0;
  bool bad = false;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t c = (b[i / 4] >> (8 * (i % 4))) & 0xFFu;
    bad |= c > 15;
    word |= (c & 0xFu) << (4 * i);
  }
  if (bad) {
    report(status, W4_ERR_VALUE);
    return;
  }
  qw[j] = word;
}

__global__ void __launch_bounds__(256) quantize_kernel(uint32_t* __restrict__ qw,
                                                        uint16_t* __restrict__ st,
                                                        const float* __restrict__ w,
                                                        long long n_groups, int K) {
  const long long gidx = ((long long)blockIdx.x * blockDim.x + threadIdx.x) / 32;
  const int lane = threadIdx.x & 31;
  if (gidx >= n_groups) return;   // whole warps leave together
  const int Kg = K / 32;
  const long long n = gidx / Kg;
  const int g = (int)(gidx - n * Kg);
  const float v = __ldg(w + n * K + (long long)g * 32 + lane);
  // largest |v|, lowest lane on ties
  float a = fabsf(v);
  int who = lane;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float ao = __shfl_xor_sync(0xffffffffu, a, off);
    const int wo = __shfl_xor_sync(0xffffffffu, who, off);
    if (ao > a || (ao == a && wo < who)) {
      a = ao;
      who = wo;
    }
  }
  const float m = __shfl_sync(0xffffffffu, v, who);
  const __nv_bfloat16 sb = __float2bfloat16_rn(__fdiv_rn(m, -8.0f));
  const float s = __bfloat162float(sb);
  int code = 8;
  if (s != 0.0f) code = min(15, max(0, __float2int_rn(__fdiv_rn(v, s)) + 8));
  uint32_t part = (uint32_t)code << (4 * (lane & 7));
  part |= __shfl_xor_sync(0xffffffffu, part, 1);
  part |= __shfl_xor_sync(0xffffffffu, part, 2);
  part |= __shfl_xor_sync(0xffffffffu, part, 4);
  if ((lane & 7) == 0) qw[n * (K / 8) + (long long)g * 4 + lane / 8] = part;
  if (lane == 0) st[n * Kg + g] = *reinterpret_cast<const uint16_t*>(&sb);
}

}  // namespace w4

using namespace w4;

extern "C" w4_status w4_pack(void* qw, const uint8_t* codes, int N, int K, int32_t* status_dev,
                             w4_stream_t stream) {
  if (qw == nullptr || codes == nullptr || N < 1) return W4_ERR_ARG;
  if (K < 32 || K % 32 != 0 || K > W4_MAX_K) return W4_ERR_SHAPE;
  if (reinterpret_cast<uintptr_t>(qw) % 16 != 0 || reinterpret_cast<uintptr_t>(codes) % 8 != 0)
    return W4_ERR_ALIGN;
  const long long n_words = (long long)N * (K / 8);
  const unsigned blocks = (unsigned)((n_words + 255) / 256);
  pack_kernel<<<blocks, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<uint32_t*>(qw), codes, n_words, status_dev);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    note_cuda_error(e);
    return W4_ERR_LAUNCH;
  }
  return W4_OK;
}

extern "C" w4_status w4_quantize(void* qw, void* st, const float* w, int N, int K,
                                 w4_stream_t stream) {
  if (qw == nullptr || st == nullptr || w == nullptr || N < 1) return W4_ERR_ARG;
  if (K < 32 || K % 32 != 0 || K > W4_MAX_K) return W4_ERR_SHAPE;
  if ((reinterpret_cast<uintptr_t>(qw) | reinterpret_cast<uintptr_t>(st) |
       reinterpret_cast<uintptr_t>(w)) % 16 != 0)
    return W4_ERR_ALIGN;
  const long long n_groups = (long long)N * (K / 32);
  const unsigned blocks = (unsigned)((n_groups * 32 + 255) / 256);
  quantize_kernel<<<blocks, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<uint32_t*>(qw), static_cast<uint16_t*>(st), w, n_groups, K);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    note_cuda_error(e);
    return W4_ERR_LAUNCH;
  }
  return W4_OK;
}
