// Router logits screened on the tensor cores, for prefill-sized T.
//
// "Perplexity Open Sources Lily: A Rust + Metal Inference Engine for
// Qwen3.6-35B-A3B on Apple Silicon", section "Three Workload Shapes": a
// router scores 256 experts and picks eight. The logits are a dense T x E x H
// contraction, so a tcgen05 GEMM computes them approximately (bf16 products
// are exact, the fp32 accumulation order is the tensor core's); the selected
// experts must still be those of the fixed-order fp32 logits, so:
//   route_mma_kernel    A[t][e] = sum over one 256-wide K slice (TMA tiles of
//                       128 experts x 128 tokens, fp32 partials per slice) and
//                       the slice's sum of w^2 per expert
//   route_screen_kernel per token: A = the slices' sum + bias; with
//                       d_e = 2^-10 * ||x_t|| * ||w_e|| (at least 20 times any
//                       accumulation error of either order: both are below
//                       2^-14.5 * sum|x w| <= 2^-14.5 * ||x|| ||w||), an expert
//                       can be in the top K only if A_e + d_e reaches the K-th
//                       largest A - d; those candidates get their fixed-order
//                       logit (the arithmetic of route_logits_kernel) and the
//                       top K is taken among them exactly as topk_warp does.
// The selected ids and weights are therefore bit-identical to the CUDA-core
// path; only the work to find them changes.
#include "common.cuh"
#include "kernels.h"
#include "topk.cuh"

namespace moe {

namespace {

constexpr int kRtTile = 128;            // experts (MMA M) and tokens (MMA N) per tile
constexpr int kRtKB = 4;                // 64-element K blocks per CTA (a 256-wide slice)
constexpr int kRtBlock = kRtTile * 128; // bytes of one 128-row x 64-element bf16 tile
constexpr int kRtSmem = 2 * kRtKB * kRtBlock + 1024 + 64;
constexpr int kScreenWarps = 8;
constexpr int kScreenMaxE = 256;        // 8 experts per lane in the screen

__device__ __forceinline__ void mma_bf16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void tmem_ld16r(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]),
        "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr)
      : "memory");
}

}  // namespace

// Grid (token tiles, expert tiles, K slices); 128 threads. P[s][t][e] fp32,
// Wn[s][e] = sum of w^2 over slice s (written by the first token tile).
__global__ void __launch_bounds__(128, 1)
    route_mma_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
                     int T, int E, float* __restrict__ P, float* __restrict__ Wn, Ctrl* ctrl) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (sbase - raw);
  const uint32_t sA = sbase, sB = sbase + kRtKB * kRtBlock;
  const uint32_t bar_tma = sbase + 2 * kRtKB * kRtBlock, bar_mma = bar_tma + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + 2 * kRtKB * kRtBlock + 16);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * kRtTile, e0 = blockIdx.y * kRtTile, s = blockIdx.z;
  const int k0 = s * kRtKB * 64;
  if (threadIdx.x == 0) {
    mbar_init(bar_tma, 1);
    mbar_init(bar_mma, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), kRtTile);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  volatile int never = 0;
  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tm_w);
    tma_prefetch_desc(&tm_x);
    mbar_arrive_expect_tx(bar_tma, 2u * kRtKB * kRtBlock);
    const uint64_t pol = policy_evict_last();
#pragma unroll
    for (int kb = 0; kb < kRtKB; ++kb) {
      tma_load_2d(sA + kb * kRtBlock, &tm_w, k0 + kb * 64, e0, bar_tma, pol);
      tma_load_2d(sB + kb * kRtBlock, &tm_x, k0 + kb * 64, t0, bar_tma, pol);
    }
  }
  // every thread waits for the tiles (the norms below read them); bounded
  bool ok = mbar_wait(bar_tma, 0, &never);
  if (threadIdx.x == 0) {
    if (ok) {
      tc_fence_after();
      const uint32_t idesc = idesc_bf16(kRtTile, kRtTile);
#pragma unroll
      for (int kb = 0; kb < kRtKB; ++kb)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_bf16_ss(tmem, smem_desc_sw128(sA + kb * kRtBlock + kk * 32),
                      smem_desc_sw128(sB + kb * kRtBlock + kk * 32), idesc, (kb | kk) != 0);
      mma_commit(bar_mma);
    } else {
      set_error(ctrl, MOE_ERR_TIMEOUT, KID_ROUTE, 1);
    }
  }
  // slice norms of the experts' rows: row r of a tile is 128 contiguous bytes
  // (the swizzle only permutes its 16-byte chunks)
  if (ok && blockIdx.x == 0 && e0 + (int)threadIdx.x < E) {
    const int r = threadIdx.x;
    float ss = 0.0f;
#pragma unroll
    for (int kb = 0; kb < kRtKB; ++kb) {
      const uint8_t* row = gbase + kb * kRtBlock + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint4 v = *reinterpret_cast<const uint4*>(row + 16 * c);
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          ss = __fmaf_rn(bf_lo(u[i]), bf_lo(u[i]), ss);
          ss = __fmaf_rn(bf_hi(u[i]), bf_hi(u[i]), ss);
        }
      }
    }
    Wn[(size_t)s * E + e0 + r] = ss;
  }
  ok = __syncthreads_and(ok);
  if (ok && mbar_wait(bar_mma, 0, &never)) {
    tc_fence_after();
    const int e = e0 + warp * 32 + lane;
    const uint32_t taddr = tmem + ((uint32_t)(warp * 32) << 16);
    float* out = P + (size_t)s * T * E;
#pragma unroll 1
    for (int c0 = 0; c0 < kRtTile; c0 += 16) {
      uint32_t v[16];
      tmem_ld16r(taddr + c0, v);
      tmem_wait_ld();
      if (e < E) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int t = t0 + c0 + i;
          if (t < T) out[(size_t)t * E + e] = __uint_as_float(v[i]);
        }
      }
    }
  } else if (threadIdx.x == 0) {
    set_error(ctrl, MOE_ERR_TIMEOUT, KID_ROUTE, 2);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kRtTile);
  }
}

// Four warps per token (two tokens per block). Warp 0 of a token's group
// forms the candidate set, the group's four warps compute the candidates'
// fixed-order logits, and warp 0 selects the top K. See the file comment.
constexpr int kScreenGroup = 4;                               // warps per token
constexpr int kScreenTokens = kScreenWarps / kScreenGroup;    // tokens per block

__device__ __forceinline__ void group_sync(int group) {
  asm volatile("bar.sync %0, %1;" ::"r"(1 + group), "r"(kScreenGroup * 32) : "memory");
}

__global__ void __launch_bounds__(kScreenWarps * 32)
    route_screen_kernel(const uint16_t* __restrict__ x, const uint16_t* __restrict__ wr,
                        const float* __restrict__ bias, const float* __restrict__ P,
                        const float* __restrict__ Wn, int T, int H, int E, int K, int S,
                        int32_t* __restrict__ ids, float* __restrict__ w) {
  __shared__ float wn[kScreenMaxE];
  __shared__ float cval[kScreenTokens][kScreenMaxE];
  __shared__ int cid[kScreenTokens][kScreenMaxE];
  __shared__ unsigned long long ckey[kScreenTokens][kScreenMaxE];
  __shared__ unsigned long long csel[kScreenTokens][32];
  __shared__ int ncand[kScreenTokens];
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    float a = 0.0f;
#pragma unroll 8
    for (int s = 0; s < S; ++s) a += __ldcg(Wn + (size_t)s * E + e);
    wn[e] = sqrtf(a);
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = warp / kScreenGroup, gw = warp % kScreenGroup;
  const int t = blockIdx.x * kScreenTokens + g;
  if (t >= T) return;  // the whole group leaves together
  const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)t * H);
  const int nj = H >> 8;
  if (gw == 0) {
    float xx = 0.0f;
#pragma unroll 8
    for (int j = 0; j < nj; ++j) {
      const uint4 v = __ldg(xr + 32 * j + lane);
      const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        xx = __fmaf_rn(bf_lo(u[i]), bf_lo(u[i]), xx);
        xx = __fmaf_rn(bf_hi(u[i]), bf_hi(u[i]), xx);
      }
    }
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) xx += __shfl_xor_sync(0xFFFFFFFFu, xx, d);
    const float xnorm = sqrtf(xx);
    // approximate logits with their bounds, experts lane + 32i
    constexpr int NL = kScreenMaxE / 32;
    float lo[NL], hi[NL], a[NL];
#pragma unroll
    for (int i = 0; i < NL; ++i) a[i] = 0.0f;
    // the loads of one slice for all eight experts are independent
#pragma unroll 4
    for (int s = 0; s < S; ++s) {
      const float* ps = P + ((size_t)s * T + t) * E;
#pragma unroll
      for (int i = 0; i < NL; ++i) {
        const int e = lane + 32 * i;
        if (e < E) a[i] += __ldcg(ps + e);
      }
    }
#pragma unroll
    for (int i = 0; i < NL; ++i) {
      const int e = lane + 32 * i;
      lo[i] = -INFINITY;
      hi[i] = -INFINITY;
      if (e < E) {
        const float v = bias ? a[i] + bias[e] : a[i];
        const float d = 0.0009765625f * xnorm * wn[e] + 1e-30f;
        lo[i] = v - d;
        hi[i] = v + d;
      }
    }
    // theta = the K-th largest lower bound: the K-th largest lane maximum is
    // at most theta, and only values at or above it can be theta
    float lmax = -INFINITY;
#pragma unroll
    for (int i = 0; i < NL; ++i) lmax = fmaxf(lmax, lo[i]);
    int r = 0;
#pragma unroll
    for (int j = 0; j < 32; ++j) r += __shfl_sync(0xFFFFFFFFu, lmax, j) > lmax;
    const uint32_t tkey = __reduce_min_sync(0xFFFFFFFFu, r < K ? topk_key(lmax) : 0xFFFFFFFFu);
    const float theta0 = topk_value(tkey);  // <= theta
    int cnt = 0;
#pragma unroll
    for (int i = 0; i < NL; ++i) cnt += lo[i] >= theta0;
    int pre = cnt;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int v = __shfl_up_sync(0xFFFFFFFFu, pre, d);
      if (lane >= d) pre += v;
    }
    const int n0 = __shfl_sync(0xFFFFFFFFu, pre, 31);
    int pos = pre - cnt;
#pragma unroll
    for (int i = 0; i < NL; ++i)
      if (lo[i] >= theta0) cval[g][pos++] = lo[i];
    __syncwarp();
    // theta = the smallest of these values with fewer than K of them above it
    float th = INFINITY;
    for (int i = lane; i < n0; i += 32) {
      const float v = cval[g][i];
      int above = 0;
      for (int j = 0; j < n0; ++j) above += cval[g][j] > v;
      if (above < K) th = fminf(th, v);
    }
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) th = fminf(th, __shfl_xor_sync(0xFFFFFFFFu, th, d));
    // candidates: upper bound at least theta
    cnt = 0;
#pragma unroll
    for (int i = 0; i < NL; ++i) cnt += hi[i] >= th;
    pre = cnt;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int v = __shfl_up_sync(0xFFFFFFFFu, pre, d);
      if (lane >= d) pre += v;
    }
    pos = pre - cnt;
#pragma unroll
    for (int i = 0; i < NL; ++i)
      if (hi[i] >= th) cid[g][pos++] = lane + 32 * i;
    if (lane == 31) ncand[g] = pre;
  }
  group_sync(g);
  const int nc = ncand[g];
  // fixed-order fp32 logits of the candidates (route_logits_kernel's order):
  // candidate c goes to warp c mod 4 of the group
  for (int c = gw; c < nc; c += kScreenGroup) {
    const int e = cid[g][c];
    const uint4* wq = reinterpret_cast<const uint4*>(wr + (size_t)e * H);
    float acc = 0.0f;
#pragma unroll 8
    for (int j = 0; j < nj; ++j) {
      const uint4 xv = __ldg(xr + 32 * j + lane), wv = __ldg(wq + 32 * j + lane);
      acc = __fmaf_rn(bf_lo(xv.x), bf_lo(wv.x), acc);
      acc = __fmaf_rn(bf_hi(xv.x), bf_hi(wv.x), acc);
      acc = __fmaf_rn(bf_lo(xv.y), bf_lo(wv.y), acc);
      acc = __fmaf_rn(bf_hi(xv.y), bf_hi(wv.y), acc);
      acc = __fmaf_rn(bf_lo(xv.z), bf_lo(wv.z), acc);
      acc = __fmaf_rn(bf_hi(xv.z), bf_hi(wv.z), acc);
      acc = __fmaf_rn(bf_lo(xv.w), bf_lo(wv.w), acc);
      acc = __fmaf_rn(bf_hi(xv.w), bf_hi(wv.w), acc);
    }
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xFFFFFFFFu, acc, d));
    if (lane == 0) ckey[g][c] = topk_ckey(bias ? __fadd_rn(acc, bias[e]) : acc, e);
  }
  group_sync(g);
  if (gw != 0) return;
  for (int i = lane; i < nc; i += 32) {
    const unsigned long long ci = ckey[g][i];
    int rk = 0;
    for (int j = 0; j < nc; ++j) rk += ckey[g][j] > ci;
    if (rk < K) csel[g][rk] = ci;
  }
  __syncwarp();
  const unsigned long long mine = lane < K ? csel[g][lane] : 0ull;
  const float my_l = topk_value((uint32_t)(mine >> 32));
  const float l0 = __shfl_sync(0xFFFFFFFFu, my_l, 0);
  const float ex = (lane < K) ? expf(my_l - l0) : 0.0f;
  float z = ex;
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) z += __shfl_xor_sync(0xFFFFFFFFu, z, d);
  if (lane < K) {
    ids[(size_t)t * K + lane] = (int)(0xFFFFFFFFu - (uint32_t)mine);
    w[(size_t)t * K + lane] = ex / z;
  }
}

bool route_tc_supported(int T, int H, int E, int K) {
  return T >= kRouteTcMinT && E <= kScreenMaxE && K <= 32 && H % (kRtKB * 64) == 0;
}

size_t route_tc_partial_floats(int T, int H, int E) {
  return (size_t)(H / (kRtKB * 64)) * ((size_t)T * E + E);
}

cudaError_t launch_route_tc(const CUtensorMap& tm_w, const CUtensorMap& tm_x, const uint16_t* x,
                            const uint16_t* wr, const float* bias, int T, int H, int E, int K,
                            float* part, int32_t* ids, float* w, Ctrl* ctrl, cudaStream_t stream) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(route_mma_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kRtSmem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int S = H / (kRtKB * 64);
  float* P = part;
  float* Wn = part + (size_t)S * T * E;
  dim3 grid((T + kRtTile - 1) / kRtTile, (E + kRtTile - 1) / kRtTile, S);
  route_mma_kernel<<<grid, 128, kRtSmem, stream>>>(tm_w, tm_x, T, E, P, Wn, ctrl);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  route_screen_kernel<<<(T + kScreenTokens - 1) / kScreenTokens, kScreenWarps * 32, 0, stream>>>(
      x, wr, bias, P, Wn, T, H, E, K, S, ids, w);
  return cudaGetLastError();
}

}  // namespace moe
