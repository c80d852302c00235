// Host interface of the tensor-core (tcgen05) small-batch W4A16 path, used by
// the w4a16_gemv entry in gemv.cu.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "common.cuh"

namespace w4 {
namespace tc {

constexpr int kTcMaxM = 32;   // activation rows per launch

struct TcPlan {
  int np = 16;                // MMA N (activation columns, >= M)
  int slices = 0, tiles = 0;  // 256-code K slices, 128-row tiles
  int S = 1, sps = 1, units = 0, ctas = 0;
  int nst = 2, stage_bytes = 0, off_b = 0, smem = 0;
  int bufs = 2, per_sm = 2;   // rounds held in tensor memory; CTAs per SM
  int sk = 0;                 // balanced runs per CTA (tiles cut between CTAs hand
                              // their row sums over through the workspace)
  size_t ws_bytes = 0, ws_part_off = 0;
};

// True when the tensor-core path can run M activation rows with reduction K
// (K a multiple of 256, M <= kTcMaxM, tensor-map encoder available).
bool tc_supported(int M, int K);

// allow_sk: plan balanced runs where they apply (they need ws_bytes of
// workspace; the plain plan computes the same bits without it).
bool tc_plan(int M, int N, int K, int sms, TcPlan* out, bool allow_sk = true);

// l2: byte ranges the copy warps bring into L2 once their own tiles are
// requested (w4a16_gemv_prefetch_l2), or nullptr.
cudaError_t tc_launch(const TcPlan& pl, void* y, const void* qw, const void* st, const void* x,
                      int M, int N, int K, void* workspace, int32_t* status, bool pdl,
                      cudaStream_t stream, int dev, const L2Ranges* l2 = nullptr);

int tc_sms(int dev);

// Prompt chunks (more rows than one small-batch launch takes, up to
// kTpMaxM): one launch of the exact hi/lo-split tcgen05 GEMM.
constexpr int kTpMaxM = 256;

struct TpPlan {
  int xrows = 0, nt = 0;      // activation rows per unit tile, MMA N
  int tiles = 0, units = 0, ctas = 0;
  int xs = 0, x_stage_bytes = 0, smem = 0;
};

bool tp_plan(int M, int N, int K, int sms, TpPlan* out);

cudaError_t tp_launch(const TpPlan& pl, void* y, const void* qw, const void* st, const void* x,
                      int M, int N, int K, int32_t* status, bool pdl, cudaStream_t stream,
                      int dev);

}  // namespace tc
}  // namespace w4
