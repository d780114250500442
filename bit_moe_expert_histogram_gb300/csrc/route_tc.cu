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
//                       the slice's sum of w^2 per expert (the diagonal of
//                       W W^T, on the tensor cores too: only a bound uses it)
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
// Inside the layer call the screen also counts its selections into the
// plan's per-chunk expert histogram (hist[f / chunk][e] for item f = t*K + k,
// zeroed by route_mma_kernel), which replaces the plan's histogram launch;
// the counts are integers, so the order of the atomic adds does not matter.
#include "common.cuh"
#include "kernels.h"
#include "topk.cuh"

namespace moe {

namespace {

constexpr int kRtTile = 128;            // experts (MMA M) and tokens (MMA N) per tile
constexpr int kRtKB = 4;                // 64-element K blocks per CTA (a 256-wide slice)
constexpr int kRtThreads = 256;
constexpr int kRtBlock = kRtTile * 128; // bytes of one 128-row x 64-element bf16 tile
constexpr int kRtSmem = 2 * kRtKB * kRtBlock + 1024 + 64;
constexpr int kScreenWarps = 4;        // warps per screen block (one or two per token)
constexpr int kScreenMaxE = 256;        // 8 experts per lane in the screen
constexpr int kScreenMaxJ = 8;          // H / 256 at most (the row in registers; K slices)

}  // namespace

// Grid (token tiles, expert tiles, K slices); 256 threads. P[s][t][e] fp32,
// Wn[s][e] = sum of w^2 over slice s (by the first token tile: the diagonal
// of W W^T, 16 more MMAs with the expert tile as both operands, into TMEM
// columns 128..255).
__global__ void __launch_bounds__(kRtThreads, 1)
    route_mma_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
                     int T, int E, float* __restrict__ P, float* __restrict__ Wn, Ctrl* ctrl,
                     int32_t* __restrict__ hist, int hist_n) {
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
  const bool norms = blockIdx.x == 0;
  if (threadIdx.x == 0) {
    mbar_init(bar_tma, 1);
    mbar_init(bar_mma, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), 2 * kRtTile);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();  // everything above reads no global memory
  pdl_trigger();
  if (hist) {  // the plan histogram that the screen fills
    const int nblk = gridDim.x * gridDim.y * gridDim.z;
    const int bid = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
    for (int i = bid * kRtThreads + threadIdx.x; i < hist_n; i += nblk * kRtThreads) hist[i] = 0;
  }
  volatile int never = 0;
  bool ok = true;
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
    ok = mbar_wait(bar_tma, 0, &never);  // bounded
    if (ok) {
      tc_fence_after();
      const uint32_t idesc = idesc_bf16(kRtTile, kRtTile);
#pragma unroll
      for (int kb = 0; kb < kRtKB; ++kb)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_bf16_ss(tmem, smem_desc_sw128(sA + kb * kRtBlock + kk * 32),
                      smem_desc_sw128(sB + kb * kRtBlock + kk * 32), idesc, (kb | kk) != 0);
      if (norms) {
#pragma unroll
        for (int kb = 0; kb < kRtKB; ++kb)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16_ss(tmem + kRtTile, smem_desc_sw128(sA + kb * kRtBlock + kk * 32),
                        smem_desc_sw128(sA + kb * kRtBlock + kk * 32), idesc, (kb | kk) != 0);
      }
      mma_commit(bar_mma);
    } else {
      set_error(ctrl, MOE_ERR_TIMEOUT, KID_ROUTE, 1);
    }
  }
  ok = __syncthreads_and(ok);
  if (ok && mbar_wait(bar_mma, 0, &never)) {
    tc_fence_after();
    // warps q and q + 4 read TMEM lane quarter q (experts), half the columns each
    const int q = warp & 3, half = warp >> 2;
    const int e = e0 + q * 32 + lane;
    const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16);
    float* out = P + (size_t)s * T * E;
    const int c_begin = half * (kRtTile / 2), c_end = c_begin + kRtTile / 2;
#pragma unroll
    for (int c0 = c_begin; c0 < c_end; c0 += 32) {
      uint32_t v[16], u[16];
      tmem_ld16r(taddr + c0, v);
      tmem_ld16r(taddr + c0 + 16, u);
      tmem_wait_ld();
      if (e < E) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int t = t0 + c0 + i;
          if (t < T) out[(size_t)t * E + e] = __uint_as_float(v[i]);
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int t = t0 + c0 + 16 + i;
          if (t < T) out[(size_t)t * E + e] = __uint_as_float(u[i]);
        }
      }
    }
    if (norms && half == 0) {
      // expert e's own column of W W^T: column 32q + lane of TMEM lane 32q + lane
      uint32_t v[16], u[16];
      tmem_ld16r(taddr + kRtTile + q * 32, v);
      tmem_ld16r(taddr + kRtTile + q * 32 + 16, u);
      tmem_wait_ld();
      uint32_t d = 0;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        d = lane == i ? v[i] : d;
        d = lane == 16 + i ? u[i] : d;
      }
      if (e < E) Wn[(size_t)s * E + e] = __uint_as_float(d);
    }
  } else if (threadIdx.x == 0) {
    set_error(ctrl, MOE_ERR_TIMEOUT, KID_ROUTE, 2);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 2 * kRtTile);
  }
}

// SPLIT warps per token, kScreenWarps / SPLIT tokens per block, no barrier
// after the expert norms: each warp of a token forms the token's candidate
// set (the same set in each), computes every SPLIT-th batch of four
// candidates' fixed-order logits (four independent chains per lane), and the
// token's first warp selects the top K among them. Two warps per token halve
// the rounds of candidate loads while every token's warps are resident at
// once; past that, one warp per token. See the file comment.
template <int SPLIT>
__global__ void __launch_bounds__(kScreenWarps * 32)
    route_screen_kernel(const uint16_t* __restrict__ x, const uint16_t* __restrict__ wr,
                        const float* __restrict__ bias, const float* __restrict__ P,
                        const float* __restrict__ Wn, int T, int H, int E, int K, int S,
                        int32_t* __restrict__ ids, float* __restrict__ w,
                        int32_t* __restrict__ hist, int chunk) {
  __shared__ float wn[kScreenMaxE];
  __shared__ float cval[kScreenWarps][kScreenMaxE];
  __shared__ int cid[kScreenWarps][kScreenMaxE];
  __shared__ unsigned long long ckey[kScreenWarps][kScreenMaxE];
  __shared__ unsigned long long csel[kScreenWarps][32];
  const int g = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * (kScreenWarps / SPLIT) + g / SPLIT, sub = g % SPLIT, gk = g - sub;
  const bool active = t < T;
  const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)(active ? t : 0) * H);
  const int nj = H >> 8;  // at most kScreenMaxJ
  constexpr int NL = kScreenMaxE / 32;
  // the token's row stays in registers (lane chunk 32j + lane); it comes
  // from before the router's first kernel, so it is read before the wait
  uint4 xv[kScreenMaxJ];
#pragma unroll
  for (int j = 0; j < kScreenMaxJ; ++j)
    xv[j] = active && j < nj ? __ldg(xr + 32 * j + lane) : make_uint4(0, 0, 0, 0);
  pdl_wait();
  pdl_trigger();
  // the expert norms' slices (whole block) and this token's partial sums
  // (experts lane + 32i): every load in flight at once
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    float v[kScreenMaxJ];
#pragma unroll
    for (int s = 0; s < kScreenMaxJ; ++s) v[s] = s < S ? __ldcg(Wn + (size_t)s * E + e) : 0.0f;
    float a = 0.0f;
#pragma unroll
    for (int s = 0; s < kScreenMaxJ; ++s) a += v[s];
    wn[e] = sqrtf(a);
  }
  float pa[kScreenMaxJ][NL];
#pragma unroll
  for (int s = 0; s < kScreenMaxJ; ++s) {
    const float* ps = P + ((size_t)s * T + (active ? t : 0)) * E;
#pragma unroll
    for (int i = 0; i < NL; ++i) {
      const int e = lane + 32 * i;
      pa[s][i] = (active && s < S && e < E) ? __ldcg(ps + e) : 0.0f;
    }
  }
  __syncthreads();
  if (!active) return;
  float a[NL];
#pragma unroll
  for (int i = 0; i < NL; ++i) {
    a[i] = 0.0f;
#pragma unroll
    for (int s = 0; s < kScreenMaxJ; ++s) a[i] += pa[s][i];
  }
  float xx0 = 0.0f, xx1 = 0.0f;
#pragma unroll
  for (int j = 0; j < kScreenMaxJ; ++j) {
    const uint32_t u[4] = {xv[j].x, xv[j].y, xv[j].z, xv[j].w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      xx0 = __fmaf_rn(bf_lo(u[i]), bf_lo(u[i]), xx0);
      xx1 = __fmaf_rn(bf_hi(u[i]), bf_hi(u[i]), xx1);
    }
  }
  float xx = xx0 + xx1;
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) xx += __shfl_xor_sync(0xFFFFFFFFu, xx, d);
  const float xnorm = sqrtf(xx);
  // approximate logits with their bounds
  float lo[NL], hi[NL];
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
  const int nc = __shfl_sync(0xFFFFFFFFu, pre, 31);
  pos = pre - cnt;
#pragma unroll
  for (int i = 0; i < NL; ++i)
    if (hi[i] >= th) cid[g][pos++] = lane + 32 * i;
  __syncwarp();
  // fixed-order fp32 logits of the candidates (route_logits_kernel's
  // order), four candidates at a time with every chunk of the four rows in
  // flight at once (one round trip per round); a missing fourth repeats the
  // first
  for (int c0 = 4 * sub; c0 < nc; c0 += 4 * SPLIT) {
    int e4[4];
    const uint4* wq[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      e4[m] = cid[g][c0 + m < nc ? c0 + m : c0];
      wq[m] = reinterpret_cast<const uint4*>(wr + (size_t)e4[m] * H);
    }
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    {
      uint4 wv[kScreenMaxJ][4];
#pragma unroll
      for (int jj = 0; jj < kScreenMaxJ; ++jj)
#pragma unroll
        for (int m = 0; m < 4; ++m)
          wv[jj][m] = jj < nj ? __ldg(wq[m] + 32 * jj + lane) : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int jj = 0; jj < kScreenMaxJ; ++jj) {
        if (jj >= nj) break;
        const uint4 xj = xv[jj];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const uint4 wj = wv[jj][m];
          acc[m] = __fmaf_rn(bf_lo(xj.x), bf_lo(wj.x), acc[m]);
          acc[m] = __fmaf_rn(bf_hi(xj.x), bf_hi(wj.x), acc[m]);
          acc[m] = __fmaf_rn(bf_lo(xj.y), bf_lo(wj.y), acc[m]);
          acc[m] = __fmaf_rn(bf_hi(xj.y), bf_hi(wj.y), acc[m]);
          acc[m] = __fmaf_rn(bf_lo(xj.z), bf_lo(wj.z), acc[m]);
          acc[m] = __fmaf_rn(bf_hi(xj.z), bf_hi(wj.z), acc[m]);
          acc[m] = __fmaf_rn(bf_lo(xj.w), bf_lo(wj.w), acc[m]);
          acc[m] = __fmaf_rn(bf_hi(xj.w), bf_hi(wj.w), acc[m]);
        }
      }
    }
#pragma unroll
    for (int m = 0; m < 4; ++m) {
#pragma unroll
      for (int d = 16; d >= 1; d >>= 1)
        acc[m] = __fadd_rn(acc[m], __shfl_xor_sync(0xFFFFFFFFu, acc[m], d));
      if (lane == 0 && c0 + m < nc)
        ckey[gk][c0 + m] = topk_ckey(bias ? __fadd_rn(acc[m], bias[e4[m]]) : acc[m], e4[m]);
    }
  }
  if constexpr (SPLIT == 2) {  // the token's two warps: named barrier 1 + token slot
    asm volatile("bar.sync %0, 64;" ::"r"(1 + g / 2) : "memory");
    if (sub) return;
  } else {
    __syncwarp();
  }
  for (int i = lane; i < nc; i += 32) {
    const unsigned long long ci = ckey[gk][i];
    int rk = 0;
    for (int j = 0; j < nc; ++j) rk += ckey[gk][j] > ci;
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
    const int id = (int)(0xFFFFFFFFu - (uint32_t)mine);
    ids[(size_t)t * K + lane] = id;
    w[(size_t)t * K + lane] = ex / z;
    if (hist) atomicAdd(hist + (size_t)((t * K + lane) / chunk) * E + id, 1);
  }
}

bool route_tc_supported(int T, int H, int E, int K) {
  return T >= kRouteTcMinT && E <= kScreenMaxE && K <= 32 && H % (kRtKB * 64) == 0 &&
         H / (kRtKB * 64) <= kScreenMaxJ;
}

size_t route_tc_partial_floats(int T, int H, int E) {
  return (size_t)(H / (kRtKB * 64)) * ((size_t)T * E + E);
}

cudaError_t launch_route_tc(const CUtensorMap& tm_w, const CUtensorMap& tm_x, const uint16_t* x,
                            const uint16_t* wr, const float* bias, int T, int H, int E, int K,
                            float* part, int32_t* ids, float* w, Ctrl* ctrl, cudaStream_t stream,
                            int32_t* hist, int chunk) {
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
  const int hist_n = hist ? (T * K + chunk - 1) / chunk * E : 0;
  cudaError_t err = launch_pdl(route_mma_kernel, grid, dim3(kRtThreads), kRtSmem, stream, tm_w,
                               tm_x, T, E, P, Wn, ctrl, hist, hist_n);
  if (err != cudaSuccess) return err;
  // two warps per token while every token's warps fit on the device at once
  static int warps_resident = 0;
  if (warps_resident == 0) {
    int dev = 0, nsm = 0, blocks = 0;
    err = cudaGetDevice(&dev);
    if (err == cudaSuccess) err = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    if (err == cudaSuccess)
      err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, route_screen_kernel<2>,
                                                          kScreenWarps * 32, 0);
    if (err != cudaSuccess) return err;
    warps_resident = nsm * blocks * kScreenWarps;
  }
  if (2 * T <= warps_resident)
    return launch_pdl(route_screen_kernel<2>, dim3((T + kScreenWarps / 2 - 1) / (kScreenWarps / 2)),
                      dim3(kScreenWarps * 32), 0, stream, x, wr, bias, (const float*)P,
                      (const float*)Wn, T, H, E, K, S, ids, w, hist, chunk);
  return launch_pdl(route_screen_kernel<1>, dim3((T + kScreenWarps - 1) / kScreenWarps),
                    dim3(kScreenWarps * 32), 0, stream, x, wr, bias, (const float*)P,
                    (const float*)Wn, T, H, E, K, S, ids, w, hist, chunk);
}

}  // namespace moe
