// Weighted combine of the expert outputs back to token order, and the
// debug dequantisation kernel.
//
// y[t] = bf16( sum_{k asc} w[t][k] * y_slots[row_pos[t*K+k]] + y_slots[R+t] )
// in fp32 in that fixed order (the shared expert sees every token with
// weight 1: "Perplexity Open Sources Lily: A Rust + Metal Inference Engine
// for Qwen3.6-35B-A3B on Apple Silicon", section "Three Workload Shapes").
// With x_next, the bf16 y is also normalised to unit RMS,
// y / sqrt(mean(y^2) + 1e-6), as the input of a stacked next layer.
#include "common.cuh"
#include "kernels.h"

namespace moe {

// One block per token; thread c owns the 8 elements [8c, 8c+8).
__global__ void __launch_bounds__(256) combine_kernel(const uint16_t* __restrict__ y_slots,
                                                      const int32_t* __restrict__ row_pos,
                                                      const float* __restrict__ w, int H, int K,
                                                      int R, int n_shared,
                                                      uint16_t* __restrict__ y,
                                                      uint16_t* __restrict__ x_next) {
  const int t = blockIdx.x;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
  const int c = threadIdx.x;  // blockDim.x == H/8: one 16-byte chunk per thread
  for (int k = 0; k < K; ++k) {
    const int r = row_pos[t * K + k];
    const float wk = w[t * K + k];
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(y_slots + (size_t)r * H) + c);
    acc[0] = __fmaf_rn(wk, bf_lo(v.x), acc[0]);
    acc[1] = __fmaf_rn(wk, bf_hi(v.x), acc[1]);
    acc[2] = __fmaf_rn(wk, bf_lo(v.y), acc[2]);
    acc[3] = __fmaf_rn(wk, bf_hi(v.y), acc[3]);
    acc[4] = __fmaf_rn(wk, bf_lo(v.z), acc[4]);
    acc[5] = __fmaf_rn(wk, bf_hi(v.z), acc[5]);
    acc[6] = __fmaf_rn(wk, bf_lo(v.w), acc[6]);
    acc[7] = __fmaf_rn(wk, bf_hi(v.w), acc[7]);
  }
  if (n_shared) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(y_slots + (size_t)(R + t) * H) + c);
    acc[0] += bf_lo(v.x); acc[1] += bf_hi(v.x);
    acc[2] += bf_lo(v.y); acc[3] += bf_hi(v.y);
    acc[4] += bf_lo(v.z); acc[5] += bf_hi(v.z);
    acc[6] += bf_lo(v.w); acc[7] += bf_hi(v.w);
  }
  uint4 o;
  o.x = pack_bf2(acc[0], acc[1]);
  o.y = pack_bf2(acc[2], acc[3]);
  o.z = pack_bf2(acc[4], acc[5]);
  o.w = pack_bf2(acc[6], acc[7]);
  reinterpret_cast<uint4*>(y + (size_t)t * H)[c] = o;
  if (x_next) {
    const float yb[8] = {bf_lo(o.x), bf_hi(o.x), bf_lo(o.y), bf_hi(o.y),
                         bf_lo(o.z), bf_hi(o.z), bf_lo(o.w), bf_hi(o.w)};
    float ss = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) ss = __fmaf_rn(yb[i], yb[i], ss);
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, d);
    __shared__ float wsum[32];
    if ((threadIdx.x & 31) == 0) wsum[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.0f;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) tot += wsum[i];
    const float inv = 1.0f / sqrtf(tot / (float)H + 1e-6f);
    uint4 n;
    n.x = pack_bf2(yb[0] * inv, yb[1] * inv);
    n.y = pack_bf2(yb[2] * inv, yb[3] * inv);
    n.z = pack_bf2(yb[4] * inv, yb[5] * inv);
    n.w = pack_bf2(yb[6] * inv, yb[7] * inv);
    reinterpret_cast<uint4*>(x_next + (size_t)t * H)[c] = n;
  }
}

cudaError_t launch_combine(const uint16_t* y_slots, const int32_t* row_pos, const float* w, int T,
                           int H, int K, int n_shared, uint16_t* y, uint16_t* x_next,
                           cudaStream_t stream) {
  const int threads = H / 8;  // H % 256 == 0 -> a whole number of warps, <= 1024 by validation
  combine_kernel<<<T, threads, 0, stream>>>(y_slots, row_pos, w, H, K, T * K, n_shared, y,
                                            x_next);
  return cudaGetLastError();
}

// Debug: dequantise a packed [N][Kd] matrix with the GEMMs' routine.
__global__ void dequant_kernel(const uint32_t* __restrict__ q, const uint16_t* __restrict__ s,
                               const uint16_t* __restrict__ b, uint16_t* __restrict__ out, int N,
                               int Kd) {
  const size_t words = (size_t)N * (Kd / 8);
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < words;
       i += (size_t)gridDim.x * blockDim.x) {
    const size_t n = i / (Kd / 8), wi = i % (Kd / 8);
    const size_t g = n * (Kd / 64) + wi / 8;
    const uint32_t s2 = s[g] | ((uint32_t)s[g] << 16);
    const uint32_t b2 = b[g] | ((uint32_t)b[g] << 16);
    uint32_t v[4];
    dequant_word(q[i], s2, b2, v);
    reinterpret_cast<uint4*>(out)[i] = make_uint4(v[0], v[1], v[2], v[3]);
  }
}

cudaError_t launch_dequant(const uint32_t* q, const uint16_t* s, const uint16_t* b, uint16_t* out,
                           int N, int Kd, cudaStream_t stream) {
  const size_t words = (size_t)N * (Kd / 8);
  const int grid = (int)((words + 255) / 256 < 4096 ? (words + 255) / 256 : 4096);
  dequant_kernel<<<grid, 256, 0, stream>>>(q, s, b, out, N, Kd);
  return cudaGetLastError();
}

}  // namespace moe
