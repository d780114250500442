// Router of the MoE layer: fp32 logits in one fixed order, then per-token
// top-K with renormalised softmax weights.
//
// "Perplexity Open Sources Lily: A Rust + Metal Inference Engine for
// Qwen3.6-35B-A3B on Apple Silicon", section "Three Workload Shapes": a
// router scores 256 experts and picks eight. The page fixes no precision
// or order; the logit here is defined so that it is bit-reproducible:
// 32 partial sums, partial L taking elements k = 8*(32j+L)+i (j ascending,
// i ascending) with fp32 fma from +0, then combined pairwise at index
// distance 16, 8, 4, 2, 1. One warp lane owns one partial, so the order is
// the natural coalesced warp order: lane L reads 16-byte chunk 32j+L.
#include "common.cuh"
#include "kernels.h"
#include "topk.cuh"

namespace moe {

// One warp computes PT tokens x PE experts; a block holds 4 warps covering
// PT tokens x 4*PE experts. Each lane keeps PT*PE partial sums.
template <int PT, int PE>
__global__ void __launch_bounds__(128) route_logits_kernel(const uint16_t* __restrict__ x,
                                                           const uint16_t* __restrict__ wr,
                                                           const float* __restrict__ bias, int T,
                                                           int H, int E,
                                                           float* __restrict__ logits) {
  pdl_wait();
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * PT;
  const int e0 = (blockIdx.y * 4 + warp) * PE;
  if (e0 >= E) return;
  const int hc = H >> 3;  // 16-byte chunks per row
  float acc[PT][PE];
#pragma unroll
  for (int p = 0; p < PT; ++p)
#pragma unroll
    for (int q = 0; q < PE; ++q) acc[p][q] = 0.0f;

  const uint4* xb = reinterpret_cast<const uint4*>(x);
  const uint4* wb = reinterpret_cast<const uint4*>(wr);
  int xrow[PT], wrow[PE];
#pragma unroll
  for (int p = 0; p < PT; ++p) xrow[p] = min(t0 + p, T - 1) * hc;
#pragma unroll
  for (int q = 0; q < PE; ++q) wrow[q] = min(e0 + q, E - 1) * hc;

  for (int j = 0; j < (H >> 8); ++j) {
    const int c = 32 * j + lane;
    float xf[PT][8];
#pragma unroll
    for (int p = 0; p < PT; ++p) {
      uint4 v = __ldg(xb + xrow[p] + c);
      xf[p][0] = bf_lo(v.x); xf[p][1] = bf_hi(v.x);
      xf[p][2] = bf_lo(v.y); xf[p][3] = bf_hi(v.y);
      xf[p][4] = bf_lo(v.z); xf[p][5] = bf_hi(v.z);
      xf[p][6] = bf_lo(v.w); xf[p][7] = bf_hi(v.w);
    }
#pragma unroll
    for (int q = 0; q < PE; ++q) {
      uint4 v = __ldg(wb + wrow[q] + c);
      float wf[8] = {bf_lo(v.x), bf_hi(v.x), bf_lo(v.y), bf_hi(v.y),
                     bf_lo(v.z), bf_hi(v.z), bf_lo(v.w), bf_hi(v.w)};
#pragma unroll
      for (int p = 0; p < PT; ++p)
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[p][q] = __fmaf_rn(xf[p][i], wf[i], acc[p][q]);
    }
  }
#pragma unroll
  for (int p = 0; p < PT; ++p)
#pragma unroll
    for (int q = 0; q < PE; ++q) {
      float a = acc[p][q];
#pragma unroll
      for (int d = 16; d >= 1; d >>= 1) a = __fadd_rn(a, __shfl_xor_sync(0xFFFFFFFFu, a, d));
      acc[p][q] = a;
    }
  if (lane == 0) {
#pragma unroll
    for (int p = 0; p < PT; ++p)
#pragma unroll
      for (int q = 0; q < PE; ++q) {
        const int t = t0 + p, e = e0 + q;
        if (t < T && e < E) {
          float l = acc[p][q];
          if (bias) l = __fadd_rn(l, bias[e]);
          logits[(size_t)t * E + e] = l;
        }
      }
  }
}

// One warp per token: top-K and renormalised softmax weights (topk.cuh).
constexpr int kTopkWarps = 4;
__global__ void __launch_bounds__(kTopkWarps * 32) route_topk_kernel(const float* __restrict__ logits,
                                                                    int T, int E, int K,
                                                                    int32_t* __restrict__ ids,
                                                                    float* __restrict__ w) {
  pdl_wait();
  pdl_trigger();
  __shared__ TopkWarpSmem<1024> S[kTopkWarps];
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (t >= T) return;
  topk_warp<1024, 32>(logits + (size_t)t * E, E, K, threadIdx.x & 31, S[threadIdx.x >> 5],
            ids + (size_t)t * K, w + (size_t)t * K);
}

cudaError_t launch_route(const uint16_t* x, const uint16_t* wr, const float* bias, int T, int H,
                         int E, int K, float* logits, int32_t* ids, float* w,
                         cudaStream_t stream) {
  cudaError_t err;
  if (T >= 8)
    err = launch_pdl(route_logits_kernel<8, 8>, dim3((T + 7) / 8, (E + 31) / 32), dim3(128), 0,
                     stream, x, wr, bias, T, H, E, logits);
  else
    err = launch_pdl(route_logits_kernel<1, 2>, dim3(T, (E + 7) / 8), dim3(128), 0, stream, x, wr,
                     bias, T, H, E, logits);
  if (err != cudaSuccess) return err;
  return launch_pdl(route_topk_kernel, dim3((T + kTopkWarps - 1) / kTopkWarps),
                    dim3(kTopkWarps * 32), 0, stream, logits, T, E, K, ids, w);
}

}  // namespace moe
