// Warp-wide top-K of one token's router logits with renormalised softmax
// weights ("Perplexity Open Sources Lily: A Rust + Metal Inference Engine
// for Qwen3.6-35B-A3B on Apple Silicon", section "Three Workload Shapes":
// the router picks the top experts). Experts are ordered by logit
// descending, ties to the lower id (values compare equal for -0 and +0);
// slot k holds the k-th; w_k = exp(l_k - l_0) / sum_j exp(l_j - l_0).
// Logits are finite (a NaN logit has no defined place in the order).
#pragma once
#include "common.cuh"

namespace moe {

// Order-preserving key of a finite logit: a larger key is a larger value,
// and -0 and +0 share one key. Key 0 is below every finite logit's key.
__device__ __forceinline__ uint32_t topk_key(float f) {
  const uint32_t b = __float_as_uint(f == 0.0f ? 0.0f : f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float topk_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Called by all 32 lanes; l = the token's E logits (E <= 1024, K <= 32).
// Lane L holds experts L + 32i. Each pick takes the warp maximum of the
// lanes' best untaken keys, then the lowest id among the lanes holding it;
// only the lane that owned the pick rescans its own keys.
__device__ __forceinline__ void topk_warp(const float* __restrict__ l, int E, int K, int lane,
                                          int32_t* __restrict__ ids, float* __restrict__ w) {
  const int n = (E + 31) >> 5;
  uint32_t key[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const int e = lane + 32 * i;
    key[i] = (i < n && e < E) ? topk_key(__ldcg(l + e)) : 0u;
  }
  uint32_t taken = 0, bk = 0, bi = 0xFFFFFFFFu;
  // the lane's best untaken key; ties go to the lowest i (the lowest id)
  auto rescan = [&]() {
    bk = 0;
    bi = 0xFFFFFFFFu;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      if (i >= n) break;
      if (!((taken >> i) & 1u) && key[i] > bk) {
        bk = key[i];
        bi = (uint32_t)(lane + 32 * i);
      }
    }
  };
  rescan();
  float my_l = 0.0f;
  int my_id = 0;
  for (int k = 0; k < K; ++k) {
    const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, bk);
    const uint32_t win = __reduce_min_sync(0xFFFFFFFFu, bk == m ? bi : 0xFFFFFFFFu);
    if (lane == k) {
      my_l = topk_value(m);
      my_id = (int)win;
    }
    if ((int)(win & 31u) == lane) {
      taken |= 1u << (win >> 5);
      rescan();
    }
  }
  const float l0 = __shfl_sync(0xFFFFFFFFu, my_l, 0);
  const float ex = (lane < K) ? expf(my_l - l0) : 0.0f;
  float z = ex;
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) z += __shfl_xor_sync(0xFFFFFFFFu, z, d);
  if (lane < K) {
    ids[lane] = my_id;
    w[lane] = ex / z;
  }
}

// Block-wide top-K of T tokens at once (T <= 4), for a block of kTopkThreads
// threads. Same order and weights as topk_warp, bit for bit. Stage 1: each
// warp takes 32-expert chunks of a token and counts, for every expert, the
// chunk members that beat it; the chunk's top K (rank < K) become candidates
// (every member of the token's top K is one). Stage 2: a candidate's rank
// among the token's candidates is its slot. Stage 3: the softmax weights, in
// topk_warp's arithmetic.
constexpr int kTopkThreads = 256;
constexpr int kTopkMaxT = 4;
constexpr int kTopkMaxCand = 512;  // per token: ceil(E/32) * K candidates at most

struct TopkSmem {
  unsigned long long cand[kTopkMaxT][kTopkMaxCand];
  int ncand[kTopkMaxT];
  float lsel[kTopkMaxT][32];
  int ids[kTopkMaxT][32];
  float w[kTopkMaxT][32];
};

// composite key: order-preserving logit key, then the lower id first
__device__ __forceinline__ unsigned long long topk_ckey(float v, int e) {
  return ((unsigned long long)topk_key(v) << 32) | (0xFFFFFFFFu - (uint32_t)e);
}

// l: logits [T][E] (read through L2). Results in S.ids / S.w [t][k].
// Requires ceil(E/32) * K <= kTopkMaxCand. Ends with __syncthreads().
__device__ __forceinline__ void topk_block(const float* __restrict__ l, int T, int E, int K,
                                           TopkSmem& S) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = kTopkThreads / 32;
  const int nch = (E + 31) >> 5;
  if (threadIdx.x < kTopkMaxT) S.ncand[threadIdx.x] = 0;
  __syncthreads();
  for (int job = warp; job < T * nch; job += nw) {
    const int t = job / nch, e = (job - t * nch) * 32 + lane;
    const unsigned long long c = e < E ? topk_ckey(__ldcg(l + (size_t)t * E + e), e) : 0ull;
    int r = 0;
#pragma unroll
    for (int j = 0; j < 32; ++j) r += __shfl_sync(0xFFFFFFFFu, c, j) > c;
    if (e < E && r < K) S.cand[t][atomicAdd(&S.ncand[t], 1)] = c;
  }
  __syncthreads();
  // four threads per candidate (consecutive lanes), each comparing it with a
  // quarter of the token's candidates; the quarters' counts are summed by
  // shuffles. Every lane of a warp runs the same iterations.
  for (int t = 0; t < T; ++t) {
    const int n = S.ncand[t], q = (n + 3) >> 2;
    const int work = ((4 * n + kTopkThreads - 1) / kTopkThreads) * kTopkThreads;
    for (int idx = threadIdx.x; idx < work; idx += kTopkThreads) {
      const int i = idx >> 2, part = idx & 3;
      const unsigned long long c = i < n ? S.cand[t][i] : 0ull;
      int r = 0;
      const int j0 = part * q, j1 = min(n, j0 + q);
      if (i < n) {
#pragma unroll 4
        for (int j = j0; j < j1; ++j) r += S.cand[t][j] > c;
      }
      r += __shfl_xor_sync(0xFFFFFFFFu, r, 1);
      r += __shfl_xor_sync(0xFFFFFFFFu, r, 2);
      if (i < n && part == 0 && r < K) {
        S.ids[t][r] = (int)(0xFFFFFFFFu - (uint32_t)c);
        S.lsel[t][r] = topk_value((uint32_t)(c >> 32));
      }
    }
  }
  __syncthreads();
  if (warp < T) {
    const float my_l = lane < K ? S.lsel[warp][lane] : 0.0f;
    const float l0 = __shfl_sync(0xFFFFFFFFu, my_l, 0);
    const float ex = (lane < K) ? expf(my_l - l0) : 0.0f;
    float z = ex;
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) z += __shfl_xor_sync(0xFFFFFFFFu, z, d);
    if (lane < K) S.w[warp][lane] = ex / z;
  }
  __syncthreads();
}

}  // namespace moe
