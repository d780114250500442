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

// Composite key: the logit key, then the lower id first. Unique per expert;
// 0 is below every expert's key.
__device__ __forceinline__ unsigned long long topk_ckey(float v, int e) {
  return ((unsigned long long)topk_key(v) << 32) | (0xFFFFFFFFu - (uint32_t)e);
}

// Slots 0..K-1 of sel hold the selected composite keys in order: writes
// ids[k] and the renormalised softmax weights w[k] = exp(l_k - l_0) / z,
// z summed over the slots by an xor butterfly of the warp's lanes (slot k
// on lane k). Whole warp.
__device__ __forceinline__ void topk_emit(const unsigned long long* sel, int K, int lane,
                                          int32_t* ids, float* w) {
  const unsigned long long mine = lane < K ? sel[lane] : 0ull;
  const float my_l = topk_value((uint32_t)(mine >> 32));
  const float l0 = __shfl_sync(0xFFFFFFFFu, my_l, 0);
  const float ex = (lane < K) ? expf(my_l - l0) : 0.0f;
  float z = ex;
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) z += __shfl_xor_sync(0xFFFFFFFFu, z, d);
  if (lane < K) {
    ids[lane] = (int)(0xFFFFFFFFu - (uint32_t)mine);
    w[lane] = ex / z;
  }
  __syncwarp();
}

// Per-warp scratch of topk_warp in shared memory, for at most CAP
// candidates (CAP >= E).
template <int CAP>
struct TopkWarpSmem {
  unsigned long long cand[CAP];
  unsigned long long sel[32];
};

// Called by all 32 lanes of a warp; l = the token's E logits, read through
// L2 (E <= 32 * NMAX, K <= 32, E <= CAP). Lane L holds experts L + 32i.
// theta = the K-th largest of the lanes' largest logit keys: at least K
// experts have a key >= theta, so every member of the top K does (any
// other would be beaten by K of them). Those candidates are ranked by the
// composite key; a candidate's rank is its slot. With fewer than K lanes
// holding experts, every expert is a candidate. Writes ids[0..K), w[0..K).
// topk_warp_vals takes the logits already in registers: v[i] = the logit
// of expert lane + 32i (ignored for an expert >= E).
template <int CAP, int NMAX>
__device__ __forceinline__ void topk_warp_vals(const float (&v)[NMAX], int E, int K, int lane,
                                               TopkWarpSmem<CAP>& S, int32_t* ids, float* w) {
  const int n = (E + 31) >> 5;
  unsigned long long c[NMAX];
  uint32_t kmax = 0u;
#pragma unroll
  for (int i = 0; i < NMAX; ++i) {
    const int e = lane + 32 * i;
    c[i] = (i < n && e < E) ? topk_ckey(v[i], e) : 0ull;
    kmax = max(kmax, (uint32_t)(c[i] >> 32));
  }
  int r = 0;  // lanes whose largest key is larger than this lane's
#pragma unroll
  for (int j = 0; j < 32; ++j) r += __shfl_sync(0xFFFFFFFFu, kmax, j) > kmax;
  const int holders = __popc(__ballot_sync(0xFFFFFFFFu, kmax != 0u));
  uint32_t theta = __reduce_min_sync(0xFFFFFFFFu, (r < K && kmax != 0u) ? kmax : 0xFFFFFFFFu);
  if (holders < K) theta = 1u;
  int cnt = 0;
#pragma unroll
  for (int i = 0; i < NMAX; ++i) cnt += (uint32_t)(c[i] >> 32) >= theta;
  int pre = cnt;  // inclusive scan of the counts over the lanes
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int v = __shfl_up_sync(0xFFFFFFFFu, pre, d);
    if (lane >= d) pre += v;
  }
  const int total = __shfl_sync(0xFFFFFFFFu, pre, 31);
  int pos = pre - cnt;
#pragma unroll
  for (int i = 0; i < NMAX; ++i)
    if ((uint32_t)(c[i] >> 32) >= theta) S.cand[pos++] = c[i];
  __syncwarp();
  for (int i = lane; i < total; i += 32) {
    const unsigned long long ci = S.cand[i];
    int rk = 0, j = 0;
    for (; j + 8 <= total; j += 8) {
#pragma unroll
      for (int u = 0; u < 8; ++u) rk += S.cand[j + u] > ci;
    }
    for (; j < total; ++j) rk += S.cand[j] > ci;
    if (rk < K) S.sel[rk] = ci;
  }
  __syncwarp();
  topk_emit(S.sel, K, lane, ids, w);
}

template <int CAP, int NMAX>
__device__ __forceinline__ void topk_warp(const float* __restrict__ l, int E, int K, int lane,
                                          TopkWarpSmem<CAP>& S, int32_t* ids, float* w) {
  const int n = (E + 31) >> 5;
  float v[NMAX];
#pragma unroll
  for (int i = 0; i < NMAX; ++i) {
    const int e = lane + 32 * i;
    v[i] = (i < n && e < E) ? __ldcg(l + e) : 0.0f;
  }
  topk_warp_vals<CAP, NMAX>(v, E, K, lane, S, ids, w);
}

}  // namespace moe
