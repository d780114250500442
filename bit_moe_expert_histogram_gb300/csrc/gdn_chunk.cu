// The Gated DeltaNet recurrence in its chunked (parallel) form, for prompts
// ("Perplexity Open Sources Lily: A Rust + Metal Inference Engine for
// Qwen3.6-35B-A3B on Apple Silicon", section "Three Workload Shapes": 30 of
// the 40 layers are Gated DeltaNet, a fixed-size recurrence; section
// "Prefill": the scan is part of every prompt's work).
//
// The rule per value head and token, S <- alpha S (I - beta k k^T) +
// beta v k^T and o = S q, is the one of gdn_scan.cu. Over a chunk of C = 64
// tokens that start from the state S0, with g_t = alpha_1 ... alpha_t, the
// writes u_t = beta_t (v_t - alpha_t S_{t-1} k_t) solve the unit
// lower-triangular system (I + A) U = diag(beta) V - diag(beta g) K S0^T,
// A[t][s] = beta_t (g_t / g_s) (k_t . k_s) for s < t (the WY / UT form of
// the delta rule). So with W1 = (I + A)^-1 diag(beta) V and
// W2 = (I + A)^-1 diag(beta g) K, which do not depend on S0:
//   U  = W1 - W2 S0^T
//   O  = diag(g) Q S0^T + (Mk o Q K^T) U,   Mk[t][s] = g_t / g_s for s <= t
//   S  = g_C S0 + U^T diag(g_C / g) K
// The gate ratios are taken as g_t / g_s = exp(G_t - G_s) with G_t the sum
// of log alpha over the chunk, so a chunk of fast decay never divides two
// products that underflow.
// Two launches:
//   gdn_chunk_prep_kernel     one CTA per (chunk, value head), all chunks at
//                             once: G, K K^T and Q K^T, A and P = Mk o Q K^T,
//                             T = (I + A)^-1 by 16 x 16 blocks, then
//                             W1 = T diag(beta) V and W2 = T diag(beta g) K,
//                             into the workspace
//   gdn_chunk_scan_tc_kernel  one CTA per (value head, 32 state rows): row i
//                             of S only ever meets row i of the state, so the
//                             chunks run in order within the CTA and the rows
//                             of a head in parallel across CTAs; U, O and the
//                             new rows from the chunk's W1, W2, P, Q and K
//   (gdn_chunk_scan_kernel, the same scan on CUDA cores, 16 rows per CTA,
//   serves value heads whose size is not a multiple of 32)
// Sums are fp32. The products run on the tensor cores with mma.sync (bf16
// inputs where both factors are bf16; tf32 where one carries fp32 values,
// that factor split into two tf32 parts so that the product keeps about fp32
// accuracy).
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {
constexpr int kDK = 128;   // key head size
constexpr int kCh = 64;    // tokens per chunk
constexpr int kThr = 256;

// per (chunk, head) block of the workspace, the matrices transposed (token
// index fastest, so the prep's one-row-per-lane stores are coalesced):
// W1^T [dv][C], W2^T [dk][C], P^T [C][C] (P^T[s][t] = P[t][s]), g [C] (g_t),
// gr [C] (g_C / g_t)
__host__ __device__ __forceinline__ size_t blk_floats(int dv) {
  return (size_t)kCh * dv + (size_t)kCh * kDK + (size_t)kCh * kCh + 2 * kCh;
}

__device__ __forceinline__ void bf8_to_f(const uint4& v, float* f) {
  f[0] = bf_lo(v.x); f[1] = bf_hi(v.x); f[2] = bf_lo(v.y); f[3] = bf_hi(v.y);
  f[4] = bf_lo(v.z); f[5] = bf_hi(v.z); f[6] = bf_lo(v.w); f[7] = bf_hi(v.w);
}

// fp32 -> tf32 (round to nearest, ties away) in a 32-bit register
__device__ __forceinline__ uint32_t to_tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}
// x = hi + lo with both parts tf32: three tf32 products (hi*hi + hi*lo +
// lo*hi) then carry an fp32 operand at about fp32 accuracy
__device__ __forceinline__ void split_tf32(float x, uint32_t& hi, uint32_t& lo) {
  hi = to_tf32(x);
  lo = to_tf32(x - __uint_as_float(hi));
}
// D += A * B, m16n8k8, tf32 inputs, fp32 accumulators (fragment layouts of
// the PTX ISA: A row-major a0 (g, c) a1 (g+8, c) a2 (g, c+4) a3 (g+8, c+4);
// B column-major b0 (k = c, n = g) b1 (c+4, g); D d0 (g, 2c) d1 (g, 2c+1)
// d2 (g+8, 2c) d3 (g+8, 2c+1); g = lane / 4, c = lane % 4)
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// acc (+)= sum over nk blocks b of L_b R_b, each a 16 x 16 fp32 block: L_b
// at L + b * lstep (row stride ldL), R_b at R + b * rstep (row stride ldR);
// both factors split into tf32 hi + lo (hi*hi + hi*lo + lo*hi). acc holds
// the warp's D fragments of the two 8-column halves (m16n8k8 layout).
__device__ __forceinline__ void blk16_mm(const float* L, int ldL, int lstep, const float* R,
                                         int ldR, int rstep, int nk, float (&acc)[2][4], int lane) {
  const int gq = lane >> 2, cq = lane & 3;
  for (int b = 0; b < nk; ++b) {
    const float* Lb = L + b * lstep;
    const float* Rb = R + b * rstep;
#pragma unroll
    for (int k0 = 0; k0 < 16; k0 += 8) {
      uint32_t ah[4], al[4];
      split_tf32(Lb[gq * ldL + k0 + cq], ah[0], al[0]);
      split_tf32(Lb[(gq + 8) * ldL + k0 + cq], ah[1], al[1]);
      split_tf32(Lb[gq * ldL + k0 + cq + 4], ah[2], al[2]);
      split_tf32(Lb[(gq + 8) * ldL + k0 + cq + 4], ah[3], al[3]);
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        uint32_t bh0, bl0, bh1, bl1;
        split_tf32(Rb[(k0 + cq) * ldR + 8 * u + gq], bh0, bl0);
        split_tf32(Rb[(k0 + cq + 4) * ldR + 8 * u + gq], bh1, bl1);
        mma_tf32(acc[u], ah, bh0, bh1);
        mma_tf32(acc[u], ah, bl0, bl1);
        mma_tf32(acc[u], al, bh0, bh1);
      }
    }
  }
}

// prep tiles: bf16 rows of 136 halves (68 words) and fp32 rows of 72 / 68
// floats put the fragment loads and stores of the MMAs on 32 distinct banks
constexpr int kLdH = 136;
constexpr int kLdA = 68;  // consecutive rows 4 banks apart: row-per-lane float4 stores conflict-free
constexpr int kLdT = 68;
// tensor-core prep: 128-byte-swizzled bf16 tiles of 128 rows x 64 elements
// (16 KB atoms); region 0 holds the [K; Q] tile (two atoms) and A, later the
// three parts of the step-4 left factor; then the V^T / K^T tile (256 rows)
constexpr int kPrepAtom = 128 * 128;
constexpr int kPrepKQBytes = 2 * kPrepAtom;
constexpr int kPrepR0Bytes = 3 * kPrepAtom > kPrepKQBytes + kCh * kLdA * 4
                                 ? 3 * kPrepAtom
                                 : ((kPrepKQBytes + kCh * kLdA * 4 + 1023) & ~1023);
constexpr int kPrepVKBytes = 256 * 128;
constexpr int kPrepSmemBytes = 1024 + kPrepR0Bytes + kPrepVKBytes +
                               (kCh * kLdT + 3 * 256 + 3 * kCh) * 4 + 2 * 8 + 16;
constexpr uint32_t kPrepTmemCols = 256;
constexpr int kLd = kDK + 1;  // padded row of a [C][dk] tile: rows t and t+1 start in other banks
constexpr int kLdP = kCh + 1;
// tensor-core scan tiles (32 state rows): padded so that every fragment
// load of the MMAs touches 32 distinct banks
constexpr int kTcLdS = 40;    // ST [dk][40]
constexpr int kTcLdT = 72;    // W2^T [dk][72], P^T [C][72] (A operands read transposed)
constexpr int kTcLdW1 = 68;   // W1^T rows r0 .. r0+31 [32][68]
constexpr int kTcLdU = 40;    // U [C][40]
// one stage: W2^T, P^T, W1^T rows, g and g_C / g in fp32, Q and K in bf16
constexpr int kTcStageFloats = kDK * kTcLdT + kCh * kTcLdT + 32 * kTcLdW1 + 2 * kCh + kCh * kLdH;
constexpr int kTcSmemFloats = kDK * kTcLdS + kCh * kTcLdU + 2 * kTcStageFloats;
template <int R>
constexpr int scan_smem_floats() {
  return kDK * (R + 1) + 2 * kCh * kLd + kCh * kDK + kCh * kLdP + 3 * kCh * R + 2 * kCh;
}
}  // namespace

// grid (n_chunks, n_v): one CTA per (chunk, value head), two CTAs per SM.
//  1. K, Q of the chunk into one 128-byte-swizzled K-major bf16 tile
//     ([K; Q], 128 rows), V^T and K^T into another (256 rows over the chunk's
//     64 tokens); G_t = sum of log alpha over the chunk (a warp scan), so
//     every gate ratio g_t / g_s is exp(G_t - G_s) and never a quotient of
//     two products that underflow
//  2. [K; Q] K^T on the tensor cores: one thread issues tcgen05.mma
//     (M = 128, N = 64, bf16, exact products, fp32 sums in TMEM); rows 0..63
//     give A, rows 64..127 give P
//  3. T = (I + A)^-1 by 16 x 16 blocks: the four diagonal blocks by forward
//     substitution (one thread per column), then the blocks below them by
//     distance from the diagonal, T_ij = -T_ii sum_k A_ik T_kj (16 x 16
//     products on mma.sync, tf32 with both factors split)
//  4. [T diag(beta); T diag(beta g)] [V | K] on the tensor cores (M = 128,
//     N = 256): the fp32 left factor is split into three bf16 parts (24
//     significant bits) and the three products summed in TMEM; W1 and W2
//     are the two diagonal blocks of the result
__global__ void __launch_bounds__(kThr, 2)
    gdn_chunk_prep_kernel(const uint16_t* __restrict__ q, const uint16_t* __restrict__ k,
                          const uint16_t* __restrict__ v, const float* __restrict__ alpha,
                          const float* __restrict__ beta, int T, int n_k, int n_v, int dv,
                          float* __restrict__ ws, Ctrl* ctrl) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* gb = smem_raw + (sbase - raw);
  // region 0: the [K; Q] tile (two 16 KB atoms) and A, later the three
  // parts of the left factor of step 4 (16 KB each)
  uint8_t* tKQ = gb;
  float* As = reinterpret_cast<float*>(gb + kPrepKQBytes);  // [C][kLdA]
  uint8_t* tTP = gb;
  uint8_t* tVK = gb + kPrepR0Bytes;                          // 256 rows x 128 B
  float* Ts = reinterpret_cast<float*>(tVK + kPrepVKBytes);  // [C][kLdT]
  float* Xs = Ts + kCh * kLdT;                               // 3 x [16][16]
  float* G = Xs + 3 * 256;                                   // [C] log gates
  float* bt = G + kCh;                                       // [C] beta
  float* bg = bt + kCh;                                      // [C] beta g
  uint64_t* bars = reinterpret_cast<uint64_t*>(bg + kCh);    // two mbarriers
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2);
  const uint32_t bar1 = smem_u32(bars), bar2 = smem_u32(bars + 1);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x, h = blockIdx.y, hk = h / (n_v / n_k);
  const int t0 = c * kCh, n = min(kCh, T - t0);
  if (tid == 0) {
    mbar_init(bar1, 1);
    mbar_init(bar2, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), kPrepTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();
  pdl_trigger();
  volatile int never = 0;
  // 1. tiles. Row r of a K-major tile holds 64 elements in 8 chunks of 16
  // bytes; chunk cc of row r sits at r * 128 + ((cc ^ (r & 7)) << 4) within
  // its 1024-byte-aligned atom. Tokens past the sequence end read as
  // k = q = v = 0, alpha = 1, beta = 0: they change nothing below.
  // Every load of a thread is issued before its stores (one round trip),
  // warp 0's gates too.
  const uint4 z4 = make_uint4(0, 0, 0, 0);
  float alpha_a = 1.0f, alpha_b = 1.0f, beta_a = 0.0f, beta_b = 0.0f;
  if (warp == 0) {
    const int ta = 2 * lane, tb = 2 * lane + 1;
    if (ta < n) {
      alpha_a = __ldg(alpha + (size_t)(t0 + ta) * n_v + h);
      beta_a = __ldg(beta + (size_t)(t0 + ta) * n_v + h);
    }
    if (tb < n) {
      alpha_b = __ldg(alpha + (size_t)(t0 + tb) * n_v + h);
      beta_b = __ldg(beta + (size_t)(t0 + tb) * n_v + h);
    }
  }
  constexpr int kKQItems = 2 * kCh * (kDK / 8) / kThr;   // 8 chunks of [K; Q] per thread
  constexpr int kVKItems = 2 * (kCh / 2) * 16 / kThr;    // 4 (pair, 8 columns) items
  constexpr int kVItems = kVKItems / 2;                  // the V^T half comes from global
  uint4 kq[kKQItems], ra[kVKItems], rb[kVKItems];
#pragma unroll
  for (int m = 0; m < kKQItems; ++m) {
    const int idx = tid + m * kThr, r = idx >> 4, ch = idx & 15;  // r < 64: K; r >= 64: Q
    const int t = r & (kCh - 1);
    kq[m] = z4;
    if (t < n)
      kq[m] = __ldg(reinterpret_cast<const uint4*>((r < kCh ? k : q) +
                                                   ((size_t)(t0 + t) * n_k + hk) * kDK + ch * 8));
  }
  // V^T (rows 0..127, zero past dv) and K^T (rows 128..255): item = (token
  // pair p, 8 columns); two 16-byte row chunks give 8 words of (t = 2p,
  // 2p + 1) pairs. The lanes of a warp take the 32 token pairs, so each of
  // its 4-byte stores fills one 128-byte row without bank conflict. V's
  // chunks come from global memory, K's from the [K; Q] tile once it is in.
#pragma unroll
  for (int m = 0; m < kVItems; ++m) {
    const int idx = tid + m * kThr;
    const int ch = (idx >> 5) & 15, p2 = idx & 31;
    const int ta = 2 * p2, tb = ta + 1;
    ra[m] = z4;
    rb[m] = z4;
    if (ch * 8 < dv) {
      const uint16_t* vb = v + (size_t)h * dv + ch * 8;
      if (ta < n) ra[m] = __ldg(reinterpret_cast<const uint4*>(vb + (size_t)(t0 + ta) * n_v * dv));
      if (tb < n) rb[m] = __ldg(reinterpret_cast<const uint4*>(vb + (size_t)(t0 + tb) * n_v * dv));
    }
  }
#pragma unroll
  for (int m = 0; m < kKQItems; ++m) {
    const int idx = tid + m * kThr, r = idx >> 4, ch = idx & 15;
    const int atom = ch >> 3, cc = ch & 7;
    *reinterpret_cast<uint4*>(tKQ + atom * kPrepAtom + r * 128 + ((cc ^ (r & 7)) << 4)) = kq[m];
  }
  __syncthreads();  // the [K; Q] tile is in: K^T's chunks come from it
#pragma unroll
  for (int m = kVItems; m < kVKItems; ++m) {
    const int idx = tid + m * kThr;
    const int ch = (idx >> 5) & 15, p2 = idx & 31;
    const int ta = 2 * p2, tb = ta + 1, atom = ch >> 3, kc = ch & 7;
    ra[m] = *reinterpret_cast<const uint4*>(tKQ + atom * kPrepAtom + ta * 128 + ((kc ^ (ta & 7)) << 4));
    rb[m] = *reinterpret_cast<const uint4*>(tKQ + atom * kPrepAtom + tb * 128 + ((kc ^ (tb & 7)) << 4));
  }
#pragma unroll
  for (int m = 0; m < kVKItems; ++m) {
    const int idx = tid + m * kThr;
    const int mat = idx >> 9, ch = (idx >> 5) & 15, p2 = idx & 31;
    const int ta = 2 * p2;
    const uint32_t wa[4] = {ra[m].x, ra[m].y, ra[m].z, ra[m].w};
    const uint32_t wb[4] = {rb[m].x, rb[m].y, rb[m].z, rb[m].w};
    const int cc = ta >> 3, within = (ta & 7) * 2;  // bytes of token ta inside its chunk
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int row = mat * 128 + ch * 8 + e;
      const uint32_t lo = (e & 1) ? (wa[e >> 1] >> 16) : (wa[e >> 1] & 0xFFFFu);
      const uint32_t hi = (e & 1) ? (wb[e >> 1] & 0xFFFF0000u) : (wb[e >> 1] << 16);
      *reinterpret_cast<uint32_t*>(tVK + row * 128 + ((cc ^ (row & 7)) << 4) + within) = lo | hi;
    }
  }
  float* blk = ws + ((size_t)c * n_v + h) * blk_floats(dv);
  float* gW1 = blk;
  float* gW2 = gW1 + (size_t)kCh * dv;
  float* gP = gW2 + (size_t)kCh * kDK;
  float* gG = gP + (size_t)kCh * kCh;
  if (warp == 0) {
    // log alpha, bounded below so that a gate of exactly 0 still gives
    // finite differences (exp(-100) is 0 to fp32 precision in every product)
    const int ta = 2 * lane, tb = 2 * lane + 1;
    const float la = ta < n ? fmaxf(logf(alpha_a), -100.0f) : 0.0f;
    const float lb = tb < n ? fmaxf(logf(alpha_b), -100.0f) : 0.0f;
    float incl = la + lb;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const float o = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += o;
    }
    const float Ga = incl - lb, Gb = incl;
    G[ta] = Ga;
    G[tb] = Gb;
    const float GC = __shfl_sync(0xffffffffu, incl, 31);
    const float ba = beta_a, bb = beta_b;
    const float ga = expf(Ga), gbv = expf(Gb);
    bt[ta] = ba;
    bt[tb] = bb;
    bg[ta] = ba * ga;
    bg[tb] = bb * gbv;
    *reinterpret_cast<float2*>(gG + ta) = make_float2(ga, gbv);
    *reinterpret_cast<float2*>(gG + kCh + ta) = make_float2(expf(GC - Ga), expf(GC - Gb));
  }
  fence_proxy_async_smem();  // the tiles are read by the tensor core
  __syncthreads();
  // 2. [K; Q] K^T
  bool ok = true;
  if (tid == 0) {
    tc_fence_after();
    const uint32_t idesc = idesc_bf16(128, kCh);
    const uint32_t a0 = smem_u32(tKQ);
#pragma unroll
    for (int atom = 0; atom < 2; ++atom)
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint64_t d = smem_desc_sw128(a0 + atom * kPrepAtom + kk * 32);
        mma_bf16_ss(tmem, d, d, idesc, (atom | kk) != 0);
      }
    mma_commit(bar1);
  }
  ok = mbar_wait(bar1, 0, &never);
  if (!ok && lane == 0) set_error(ctrl, MOE_ERR_TIMEOUT, KID_GDN, 1);
  tc_fence_after();
  {
    // warps q and q + 4 read TMEM lane quarter q, 32 columns each
    const int qr = warp & 3, half = warp >> 2;
    const int row = 32 * qr + lane, t = row & (kCh - 1);
    const uint32_t taddr = tmem + ((uint32_t)(32 * qr) << 16) + 32 * half;
    uint32_t va[16], vb2[16];
    tmem_ld16r(taddr, va);
    tmem_ld16r(taddr + 16, vb2);
    tmem_wait_ld();
    float out[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int s2 = 32 * half + i;
      const float acc = __uint_as_float(i < 16 ? va[i] : vb2[i - 16]);
      // exp2 of a scaled argument (relative error ~1e-6 for the arguments
      // here, which are <= 0 and above -6400)
      const float ratio = s2 <= t ? __expf(G[t] - G[s2]) : 0.0f;
      out[i] = row < kCh ? (s2 < t ? bt[t] * ratio * acc : 0.0f) : ratio * acc;
    }
    if (row < kCh) {
      float* dst = As + t * kLdA + 32 * half;
#pragma unroll
      for (int i = 0; i < 32; i += 4)
        *reinterpret_cast<float4*>(dst + i) = make_float4(out[i], out[i + 1], out[i + 2], out[i + 3]);
    } else {  // P^T: lanes are consecutive tokens, one 128-byte line per store
#pragma unroll
      for (int i = 0; i < 32; ++i) gP[(size_t)(32 * half + i) * kCh + t] = out[i];
    }
  }
  tc_fence_before();
  __syncthreads();
  // 3. diagonal blocks of T: thread (b, cc) solves column cc of block b;
  // entries above the diagonal come out as 0
  if (tid < 64) {
    const int b = tid >> 4, cc = tid & 15;
    float x[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      const float* ar = As + (16 * b + r) * kLdA + 16 * b;
      float a0 = r == cc ? 1.0f : 0.0f, a1 = 0.0f;
#pragma unroll
      for (int s2 = 0; s2 < r; ++s2) {
        if (s2 & 1)
          a1 = __fmaf_rn(-ar[s2], x[s2], a1);
        else
          a0 = __fmaf_rn(-ar[s2], x[s2], a0);
      }
      x[r] = a0 + a1;
    }
#pragma unroll
    for (int r = 0; r < 16; ++r) Ts[(16 * b + r) * kLdT + 16 * b + cc] = x[r];
  }
  __syncthreads();
  // the blocks below the diagonal by distance d: warp j takes block
  // (i = j + d, j); X_ij = sum_{k=j}^{i-1} A_ik T_kj, then T_ij = -T_ii X_ij,
  // both 16 x 16 products on the tensor cores
  for (int d = 1; d < 4; ++d) {
    const int nb = 4 - d;
    const int gq = lane >> 2, cq = lane & 3;
    if (warp < nb) {
      const int j = warp, i = j + d;
      float acc[2][4] = {{0, 0, 0, 0}, {0, 0, 0, 0}};
      blk16_mm(As + (16 * i) * kLdA + 16 * j, kLdA, 16, Ts + (16 * j) * kLdT + 16 * j, kLdT,
               16 * kLdT, i - j, acc, lane);
      float* X = Xs + (j << 8);
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        *reinterpret_cast<float2*>(X + gq * 16 + 8 * u + 2 * cq) = make_float2(acc[u][0], acc[u][1]);
        *reinterpret_cast<float2*>(X + (gq + 8) * 16 + 8 * u + 2 * cq) =
            make_float2(acc[u][2], acc[u][3]);
      }
      __syncwarp();
      float tacc[2][4] = {{0, 0, 0, 0}, {0, 0, 0, 0}};
      blk16_mm(Ts + (16 * i) * kLdT + 16 * i, kLdT, 0, X, 16, 0, 1, tacc, lane);
      float* To = Ts + (16 * i) * kLdT + 16 * j;
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        *reinterpret_cast<float2*>(To + gq * kLdT + 8 * u + 2 * cq) =
            make_float2(-tacc[u][0], -tacc[u][1]);
        *reinterpret_cast<float2*>(To + (gq + 8) * kLdT + 8 * u + 2 * cq) =
            make_float2(-tacc[u][2], -tacc[u][3]);
      }
    }
    __syncthreads();
  }
  // 4. the left factor [T diag(beta); T diag(beta g)] in three bf16 parts,
  // over the dead [K; Q] tile and A; thread item = (row, 8 columns). T is
  // lower triangular, so the blocks above the diagonal are written as 0.
  for (int idx = tid; idx < 2 * kCh * 8; idx += kThr) {
    const int r = idx >> 3, cc = idx & 7, t = r & (kCh - 1);
    const float* sc = r < kCh ? bt : bg;
    uint32_t pw[3][4];
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
      const int s0 = 8 * cc + e;
      const bool lo_ok = (s0 >> 4) <= (t >> 4), hi_ok = ((s0 + 1) >> 4) <= (t >> 4);
      const float x0 = lo_ok ? Ts[t * kLdT + s0] * sc[s0] : 0.0f;
      const float x1 = hi_ok ? Ts[t * kLdT + s0 + 1] * sc[s0 + 1] : 0.0f;
      const uint32_t h01 = pack_bf2(x0, x1);
      const float r0 = x0 - bf_lo(h01), r1 = x1 - bf_hi(h01);
      const uint32_t m01 = pack_bf2(r0, r1);
      const uint32_t l01 = pack_bf2(r0 - bf_lo(m01), r1 - bf_hi(m01));
      pw[0][e >> 1] = h01;
      pw[1][e >> 1] = m01;
      pw[2][e >> 1] = l01;
    }
#pragma unroll
    for (int part = 0; part < 3; ++part)
      *reinterpret_cast<uint4*>(tTP + part * kPrepAtom + r * 128 + ((cc ^ (r & 7)) << 4)) =
          make_uint4(pw[part][0], pw[part][1], pw[part][2], pw[part][3]);
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  if (tid == 0 && ok) {
    tc_fence_after();
    const uint32_t idesc = idesc_bf16(128, 256);
    const uint32_t a0 = smem_u32(tTP), b0 = smem_u32(tVK);
#pragma unroll
    for (int part = 0; part < 3; ++part)
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        mma_bf16_ss(tmem, smem_desc_sw128(a0 + part * kPrepAtom + kk * 32),
                    smem_desc_sw128(b0 + kk * 32), idesc, (part | kk) != 0);
    mma_commit(bar2);
  }
  if (ok) {
    ok = mbar_wait(bar2, 0, &never);
    if (!ok && lane == 0) set_error(ctrl, MOE_ERR_TIMEOUT, KID_GDN, 2);
  }
  tc_fence_after();
  if (ok) {
    // rows 0..63: T diag(beta) [V | K], columns 0..dv-1 are W1; rows
    // 64..127: T diag(beta g) [V | K], columns 128..255 are W2. Warps q and
    // q + 4 take lane quarter q, 64 columns each.
    const int qr = warp & 3, half = warp >> 2;
    const int row = 32 * qr + lane, t = row & (kCh - 1);
    const bool w1 = row < kCh;
    const int cbase = (w1 ? 0 : 128) + 64 * half;
    const uint32_t taddr = tmem + ((uint32_t)(32 * qr) << 16) + cbase;
#pragma unroll 1
    for (int c0 = 0; c0 < 64; c0 += 16) {
      uint32_t va[16];
      tmem_ld16r(taddr + c0, va);
      tmem_wait_ld();
      const int col = 64 * half + c0;  // column of W1 or W2
      // transposed: lanes are consecutive tokens, one 128-byte line per store
      if (w1) {
        if (col < dv) {
#pragma unroll
          for (int i = 0; i < 16; ++i) gW1[(size_t)(col + i) * kCh + t] = __uint_as_float(va[i]);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) gW2[(size_t)(col + i) * kCh + t] = __uint_as_float(va[i]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kPrepTmemCols);
  }
}

// grid (n_v, dv / R); CTA (h, y) owns state rows r0 = R*y .. R*y + R-1 of
// value head h. s_in and s_out may be the same buffer.
template <int R>
__global__ void __launch_bounds__(kThr, 1)
    gdn_chunk_scan_kernel(const uint16_t* __restrict__ q, const uint16_t* __restrict__ k,
                          const float* __restrict__ ws, const float* s_in, float* s_out,
                          uint16_t* __restrict__ o, int T, int n_k, int n_v, int dv) {
  constexpr int OI = R / 4;        // output rows per thread (4 threads per token)
  constexpr int SJ = kDK * R / kThr;  // state columns per thread in the update
  extern __shared__ float sm[];
  float* ST = sm;                        // [dk][R+1]: ST[j][i] = S[r0 + i][j]
  float* W2 = ST + kDK * (R + 1);        // [C][kLd]
  float* Qs = W2 + kCh * kLd;            // [C][kLd]
  float* Kf = Qs + kCh * kLd;            // [C][dk]
  float* P = Kf + kCh * kDK;             // [C][kLdP]
  float* W1r = P + kCh * kLdP;           // [C][R]
  float* U = W1r + kCh * R;              // [C][R]
  float* Ug = U + kCh * R;               // [C][R]: U[t][i] * g_C / g_t
  float* g = Ug + kCh * R;               // [C] g_t, then [C] g_C / g_t
  const int tid = threadIdx.x;
  const int h = blockIdx.x, hk = h / (n_v / n_k);
  const int r0 = R * blockIdx.y;
  pdl_wait();  // the workspace comes from the prep kernel
  pdl_trigger();
  // this thread's state entries for the update: row si, columns sj..sj+SJ-1
  const int si = tid / (kDK / SJ), sj = (tid % (kDK / SJ)) * SJ;
  float sr[SJ];
  {
    const float* src = s_in + ((size_t)h * dv + r0 + si) * kDK + sj;
#pragma unroll
    for (int e = 0; e < SJ; e += 4) {
      const float4 a = *reinterpret_cast<const float4*>(src + e);
      sr[e] = a.x; sr[e + 1] = a.y; sr[e + 2] = a.z; sr[e + 3] = a.w;
    }
#pragma unroll
    for (int e = 0; e < SJ; ++e) ST[(sj + e) * (R + 1) + si] = sr[e];
  }
  // this thread's outputs: token ot, rows oi..oi+OI-1
  const int ot = tid >> 2, oi = (tid & 3) * OI;
  const int n_chunks = (T + kCh - 1) / kCh;
  for (int c = 0; c < n_chunks; ++c) {
    const int t0 = c * kCh, n = min(kCh, T - t0);
    const float* blk = ws + ((size_t)c * n_v + h) * blk_floats(dv);
    const float* gW1 = blk;
    const float* gW2 = gW1 + (size_t)kCh * dv;
    const float* gP = gW2 + (size_t)kCh * kDK;
    const float* gG = gP + (size_t)kCh * kCh;
    __syncthreads();  // the previous chunk's reads of the tiles are done
    for (int idx = tid; idx < kCh * kDK / 4; idx += kThr) {  // W2^T rows, 16 bytes a thread
      const int j = idx / (kCh / 4), t = (idx % (kCh / 4)) * 4;
      const float4 w = __ldcg(reinterpret_cast<const float4*>(gW2 + (size_t)j * kCh + t));
      W2[(t + 0) * kLd + j] = w.x; W2[(t + 1) * kLd + j] = w.y;
      W2[(t + 2) * kLd + j] = w.z; W2[(t + 3) * kLd + j] = w.w;
    }
    for (int idx = tid; idx < kCh * kCh / 4; idx += kThr) {  // P^T rows
      const int sc = idx / (kCh / 4), t = (idx % (kCh / 4)) * 4;
      const float4 w = __ldcg(reinterpret_cast<const float4*>(gP + (size_t)sc * kCh + t));
      P[(t + 0) * kLdP + sc] = w.x; P[(t + 1) * kLdP + sc] = w.y;
      P[(t + 2) * kLdP + sc] = w.z; P[(t + 3) * kLdP + sc] = w.w;
    }
    for (int idx = tid; idx < kCh * R; idx += kThr) {  // W1^T rows r0 ..
      const int i = idx / kCh, t = idx % kCh;
      W1r[t * R + i] = __ldcg(gW1 + (size_t)(r0 + i) * kCh + t);
    }
    if (tid < 2 * kCh) g[tid] = __ldcg(gG + tid);
    for (int idx = tid; idx < kCh * (kDK / 8); idx += kThr) {
      const int t = idx / (kDK / 8), ch = idx % (kDK / 8);
      float kf[8] = {0, 0, 0, 0, 0, 0, 0, 0}, qf[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      if (t < n) {
        const size_t src = ((size_t)(t0 + t) * n_k + hk) * kDK + ch * 8;
        bf8_to_f(__ldg(reinterpret_cast<const uint4*>(k + src)), kf);
        bf8_to_f(__ldg(reinterpret_cast<const uint4*>(q + src)), qf);
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) Qs[t * kLd + ch * 8 + e] = qf[e];
      float4* kd = reinterpret_cast<float4*>(Kf + t * kDK + ch * 8);
      kd[0] = make_float4(kf[0], kf[1], kf[2], kf[3]);
      kd[1] = make_float4(kf[4], kf[5], kf[6], kf[7]);
    }
    __syncthreads();
    // U[t][i] = W1[t][r0+i] - sum_j W2[t][j] S[r0+i][j];  QS[t][i] = sum_j Q[t][j] S[r0+i][j]
    float u[OI], qs[OI];
#pragma unroll
    for (int e = 0; e < OI; ++e) u[e] = qs[e] = 0.0f;
#pragma unroll 4
    for (int j = 0; j < kDK; ++j) {
      const float w = W2[ot * kLd + j], qv = Qs[ot * kLd + j];
      const float* sp = ST + j * (R + 1) + oi;
#pragma unroll
      for (int e = 0; e < OI; ++e) {
        u[e] = __fmaf_rn(w, sp[e], u[e]);
        qs[e] = __fmaf_rn(qv, sp[e], qs[e]);
      }
    }
    const float gC = g[kCh - 1];
#pragma unroll
    for (int e = 0; e < OI; ++e) {
      const float uu = W1r[ot * R + oi + e] - u[e];
      U[ot * R + oi + e] = uu;
      Ug[ot * R + oi + e] = uu * g[kCh + ot];
    }
    __syncthreads();
    // O[t][i] = g_t QS[t][i] + sum_{s <= t} P[t][s] U[s][i]
    float ov[OI];
#pragma unroll
    for (int e = 0; e < OI; ++e) ov[e] = g[ot] * qs[e];
    for (int s = 0; s <= ot; ++s) {
      const float p = P[ot * kLdP + s];
#pragma unroll
      for (int e = 0; e < OI; ++e) ov[e] = __fmaf_rn(p, U[s * R + oi + e], ov[e]);
    }
    if (ot < n) {
      uint32_t w[OI / 2];
#pragma unroll
      for (int e = 0; e < OI / 2; ++e) w[e] = pack_bf2(ov[2 * e], ov[2 * e + 1]);
      uint16_t* dst = o + ((size_t)(t0 + ot) * n_v + h) * dv + r0 + oi;
      if (OI == 8)
        *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1 % (OI / 2)], w[2 % (OI / 2)], w[3 % (OI / 2)]);
      else
        *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1 % (OI / 2)]);
    }
    // S[r0+si][j] = g_C S[r0+si][j] + sum_t Ug[t][si] K[t][j]
    float acc[SJ];
#pragma unroll
    for (int e = 0; e < SJ; ++e) acc[e] = gC * sr[e];
#pragma unroll 2
    for (int t = 0; t < kCh; ++t) {
      const float ug = Ug[t * R + si];
#pragma unroll
      for (int e = 0; e < SJ; e += 4) {
        const float4 kv = *reinterpret_cast<const float4*>(Kf + t * kDK + sj + e);
        acc[e] = __fmaf_rn(ug, kv.x, acc[e]);
        acc[e + 1] = __fmaf_rn(ug, kv.y, acc[e + 1]);
        acc[e + 2] = __fmaf_rn(ug, kv.z, acc[e + 2]);
        acc[e + 3] = __fmaf_rn(ug, kv.w, acc[e + 3]);
      }
    }
    __syncthreads();  // every read of the old state (U, QS) is done
#pragma unroll
    for (int e = 0; e < SJ; ++e) {
      sr[e] = acc[e];
      ST[(sj + e) * (R + 1) + si] = acc[e];
    }
  }
  float* dst = s_out + ((size_t)h * dv + r0 + si) * kDK + sj;
#pragma unroll
  for (int e = 0; e < SJ; e += 4)
    *reinterpret_cast<float4*>(dst + e) = make_float4(sr[e], sr[e + 1], sr[e + 2], sr[e + 3]);
}

// 16-byte asynchronous copy global -> shared; src_bytes = 0 fills zeros
__device__ __forceinline__ void cp_async16(void* dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// One chunk's tiles for the tensor-core scan, in shared memory
struct ScanStage {
  float* W2;     // [dk][kTcLdT]: W2^T
  float* P;      // [C][kTcLdT]: P^T
  float* W1r;    // [32][kTcLdW1]: W1^T rows r0 .. r0+31
  float* g;      // [C] g_t, then [C] g_C / g_t
  uint16_t* Qb;  // [C][kLdH] bf16
  uint16_t* Kb;  // [C][kLdH] bf16
};
__device__ __forceinline__ ScanStage scan_stage(float* base) {
  ScanStage st;
  st.W2 = base;
  st.P = st.W2 + kDK * kTcLdT;
  st.W1r = st.P + kCh * kTcLdT;
  st.g = st.W1r + 32 * kTcLdW1;
  st.Qb = reinterpret_cast<uint16_t*>(st.g + 2 * kCh);
  st.Kb = st.Qb + kCh * kLdH;
  return st;
}

// every thread issues its share of chunk c's copies (one commit group)
__device__ __forceinline__ void scan_issue(const ScanStage& st, const uint16_t* __restrict__ q,
                                           const uint16_t* __restrict__ k,
                                           const float* __restrict__ ws, int c, int T, int n_k,
                                           int n_v, int dv, int h, int hk, int r0, int tid) {
  const int t0 = c * kCh, n = min(kCh, T - t0);
  const float* blk = ws + ((size_t)c * n_v + h) * blk_floats(dv);
  const float* gW1 = blk;
  const float* gW2 = gW1 + (size_t)kCh * dv;
  const float* gP = gW2 + (size_t)kCh * kDK;
  const float* gG = gP + (size_t)kCh * kCh;
#pragma unroll
  for (int m = 0; m < kCh * kDK / 4 / kThr; ++m) {  // W2^T: 128 rows of 64
    const int idx = tid + m * kThr, j = idx >> 4, t = (idx & 15) * 4;
    cp_async16(st.W2 + j * kTcLdT + t, gW2 + (size_t)j * kCh + t, 16);
  }
#pragma unroll
  for (int m = 0; m < kCh * kCh / 4 / kThr; ++m) {  // P^T: 64 rows of 64
    const int idx = tid + m * kThr, sc = idx >> 4, t = (idx & 15) * 4;
    cp_async16(st.P + sc * kTcLdT + t, gP + (size_t)sc * kCh + t, 16);
  }
#pragma unroll
  for (int m = 0; m < kCh * 32 / 4 / kThr; ++m) {  // W1^T rows r0 .. r0+31
    const int idx = tid + m * kThr, i = idx >> 4, t = (idx & 15) * 4;
    cp_async16(st.W1r + i * kTcLdW1 + t, gW1 + (size_t)(r0 + i) * kCh + t, 16);
  }
  if (tid < 2 * kCh / 4) cp_async16(st.g + 4 * tid, gG + 4 * tid, 16);
#pragma unroll
  for (int m = 0; m < kCh * (kDK / 8) / kThr; ++m) {
    const int idx = tid + m * kThr, t = idx >> 4, ch = idx & 15;
    // tokens past the end read as zeros (from a valid address)
    const size_t src = t < n ? ((size_t)(t0 + t) * n_k + hk) * kDK + ch * 8 : 0;
    const int bytes = t < n ? 16 : 0;
    cp_async16(st.Qb + t * kLdH + ch * 8, q + src, bytes);
    cp_async16(st.Kb + t * kLdH + ch * 8, k + src, bytes);
  }
  cp_async_commit();
}

// The same scan with its four products per chunk on the tensor cores
// (mma.sync m16n8k8, tf32 inputs, fp32 accumulation): U = W1 - W2 S0^T and
// Q S0^T share the state fragments; O = g Q S0^T + P U; S = g_C S0 +
// (diag(g_C / g) U)^T K. Operands that carry fp32 values (W2, S, P, U) are
// split into tf32 hi + lo and multiplied as hi*hi + hi*lo + lo*hi; q and k
// are bf16, exact in tf32. 32 state rows of one value head per CTA, 8 warps;
// the next chunk's tiles are copied in (cp.async, two stages) while the
// current one is computed.
__global__ void __launch_bounds__(kThr, 1)
    gdn_chunk_scan_tc_kernel(const uint16_t* __restrict__ q, const uint16_t* __restrict__ k,
                             const float* __restrict__ ws, const float* s_in, float* s_out,
                             uint16_t* __restrict__ o, int T, int n_k, int n_v, int dv) {
  constexpr int R = 32;
  extern __shared__ float sm[];
  float* ST = sm;                        // [dk][kTcLdS]: ST[j][i] = S[r0 + i][j]
  float* U = ST + kDK * kTcLdS;          // [C][kTcLdU]
  float* const stage0 = U + kCh * kTcLdU;  // two stages of kTcStageFloats
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, cq = lane & 3;
  const int h = blockIdx.x, hk = h / (n_v / n_k);
  const int r0 = R * blockIdx.y;
  const int n_chunks = (T + kCh - 1) / kCh;
  pdl_wait();  // the workspace comes from the prep kernel
  pdl_trigger();
  scan_issue(scan_stage(stage0), q, k, ws, 0, T, n_k, n_v, dv, h, hk, r0, tid);
  for (int idx = tid; idx < R * kDK / 4; idx += kThr) {
    const int i = idx % R, j = (idx / R) * 4;
    const float4 v = *reinterpret_cast<const float4*>(s_in + ((size_t)h * dv + r0 + i) * kDK + j);
    ST[(j + 0) * kTcLdS + i] = v.x;
    ST[(j + 1) * kTcLdS + i] = v.y;
    ST[(j + 2) * kTcLdS + i] = v.z;
    ST[(j + 3) * kTcLdS + i] = v.w;
  }
  // U / QS / O tiles: rows 16*mt.., columns 8*nt0.. and 8*(nt0+1)..
  const int mt = warp & 3, nt0 = 2 * (warp >> 2);
  // state tiles: rows 16*ms.., columns 8*ns0 .. 8*ns0 + 31
  const int ms = warp & 1, ns0 = 4 * (warp >> 1);
  for (int c = 0; c < n_chunks; ++c) {
    const ScanStage sg = scan_stage(stage0 + (c & 1) * kTcStageFloats);
    const int t0 = c * kCh, n = min(kCh, T - t0);
    // the other stage was last read by chunk c-1, before the barrier that
    // ended it (or never): refill it with chunk c+1, then wait for chunk c
    if (c + 1 < n_chunks) {
      scan_issue(scan_stage(stage0 + ((c + 1) & 1) * kTcStageFloats), q, k, ws, c + 1, T, n_k,
                 n_v, dv, h, hk, r0, tid);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();  // chunk c's tiles and the state are in place
    const float* W2 = sg.W2;
    const float* P = sg.P;
    const float* g = sg.g;
    const uint16_t* Qb = sg.Qb;
    const uint16_t* Kb = sg.Kb;
    // (1) W2 S0^T and (2) Q S0^T over j = 0..127
    float au[2][4] = {{0, 0, 0, 0}, {0, 0, 0, 0}}, aq[2][4] = {{0, 0, 0, 0}, {0, 0, 0, 0}};
    const int ra = 16 * mt + gq;
#pragma unroll
    for (int kb = 0; kb < kDK / 8; ++kb) {
      const int j = 8 * kb + cq;
      uint32_t wh[4], wl[4], qa[4];
      split_tf32(W2[j * kTcLdT + ra], wh[0], wl[0]);
      split_tf32(W2[j * kTcLdT + ra + 8], wh[1], wl[1]);
      split_tf32(W2[(j + 4) * kTcLdT + ra], wh[2], wl[2]);
      split_tf32(W2[(j + 4) * kTcLdT + ra + 8], wh[3], wl[3]);
      qa[0] = (uint32_t)Qb[ra * kLdH + j] << 16;
      qa[1] = (uint32_t)Qb[(ra + 8) * kLdH + j] << 16;
      qa[2] = (uint32_t)Qb[ra * kLdH + j + 4] << 16;
      qa[3] = (uint32_t)Qb[(ra + 8) * kLdH + j + 4] << 16;
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int col = 8 * (nt0 + u) + gq;
        uint32_t sh0, sl0, sh1, sl1;
        split_tf32(ST[j * kTcLdS + col], sh0, sl0);
        split_tf32(ST[(j + 4) * kTcLdS + col], sh1, sl1);
        mma_tf32(au[u], wh, sh0, sh1);
        mma_tf32(au[u], wh, sl0, sl1);
        mma_tf32(au[u], wl, sh0, sh1);
        mma_tf32(aq[u], qa, sh0, sh1);
        mma_tf32(aq[u], qa, sl0, sl1);
      }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u)
#pragma unroll
      for (int e = 0; e < 4; e += 2) {
        const int t = ra + 8 * (e >> 1), i = 8 * (nt0 + u) + 2 * cq;
        const float w0 = sg.W1r[i * kTcLdW1 + t], w1 = sg.W1r[(i + 1) * kTcLdW1 + t];
        *reinterpret_cast<float2*>(U + t * kTcLdU + i) = make_float2(w0 - au[u][e], w1 - au[u][e + 1]);
      }
    __syncthreads();
    // (3) O = g Q S0^T + P U; P is zero above the diagonal
    float ao[2][4] = {{0, 0, 0, 0}, {0, 0, 0, 0}};
#pragma unroll
    for (int kb = 0; kb < kCh / 8; ++kb) {
      if (kb > 2 * mt + 1) break;  // P is zero above the diagonal
      const int sc = 8 * kb + cq;
      uint32_t ph[4], pl[4];
      split_tf32(P[sc * kTcLdT + ra], ph[0], pl[0]);
      split_tf32(P[sc * kTcLdT + ra + 8], ph[1], pl[1]);
      split_tf32(P[(sc + 4) * kTcLdT + ra], ph[2], pl[2]);
      split_tf32(P[(sc + 4) * kTcLdT + ra + 8], ph[3], pl[3]);
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int col = 8 * (nt0 + u) + gq;
        uint32_t uh0, ul0, uh1, ul1;
        split_tf32(U[sc * kTcLdU + col], uh0, ul0);
        split_tf32(U[(sc + 4) * kTcLdU + col], uh1, ul1);
        mma_tf32(ao[u], ph, uh0, uh1);
        mma_tf32(ao[u], ph, ul0, ul1);
        mma_tf32(ao[u], pl, uh0, uh1);
      }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u)
#pragma unroll
      for (int e = 0; e < 4; e += 2) {
        const int t = ra + 8 * (e >> 1), i = 8 * (nt0 + u) + 2 * cq;
        if (t < n) {
          const float o0 = g[t] * aq[u][e] + ao[u][e];
          const float o1 = g[t] * aq[u][e + 1] + ao[u][e + 1];
          *reinterpret_cast<uint32_t*>(o + ((size_t)(t0 + t) * n_v + h) * dv + r0 + i) =
              pack_bf2(o0, o1);
        }
      }
    // (4) S = g_C S0 + (diag(g_C / g) U)^T K: rows i (M), columns j (N), over t (K)
    const float gC = g[kCh - 1];
    float as[4][4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = 16 * ms + gq + 8 * (e >> 1), j = 8 * (ns0 + u) + 2 * cq + (e & 1);
        as[u][e] = gC * ST[j * kTcLdS + i];
      }
#pragma unroll
    for (int kb = 0; kb < kCh / 8; ++kb) {
      const int t = 8 * kb + cq;
      const int ia = 16 * ms + gq;
      const float r0g = g[kCh + t], r4g = g[kCh + t + 4];
      uint32_t uh[4], ul[4];
      split_tf32(U[t * kTcLdU + ia] * r0g, uh[0], ul[0]);
      split_tf32(U[t * kTcLdU + ia + 8] * r0g, uh[1], ul[1]);
      split_tf32(U[(t + 4) * kTcLdU + ia] * r4g, uh[2], ul[2]);
      split_tf32(U[(t + 4) * kTcLdU + ia + 8] * r4g, uh[3], ul[3]);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int col = 8 * (ns0 + u) + gq;
        const uint32_t k0 = (uint32_t)Kb[t * kLdH + col] << 16;
        const uint32_t k1 = (uint32_t)Kb[(t + 4) * kLdH + col] << 16;
        mma_tf32(as[u], uh, k0, k1);
        mma_tf32(as[u], ul, k0, k1);
      }
    }
    __syncthreads();  // every read of the old state and of this stage is done
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = 16 * ms + gq + 8 * (e >> 1), j = 8 * (ns0 + u) + 2 * cq + (e & 1);
        ST[j * kTcLdS + i] = as[u][e];
      }
  }
  __syncthreads();
  for (int idx = tid; idx < R * kDK / 4; idx += kThr) {
    const int i = idx % R, j = (idx / R) * 4;
    *reinterpret_cast<float4*>(s_out + ((size_t)h * dv + r0 + i) * kDK + j) =
        make_float4(ST[(j + 0) * kTcLdS + i], ST[(j + 1) * kTcLdS + i], ST[(j + 2) * kTcLdS + i],
                    ST[(j + 3) * kTcLdS + i]);
  }
}

// The workspace: a 256-byte status header (Ctrl, zero-filled once by the
// caller), then the per-(chunk, head) blocks.
size_t gdn_chunk_ws_bytes(const moe_gdn_shape_t* s) {
  const size_t n_chunks = ((size_t)s->T + kCh - 1) / kCh;
  return sizeof(Ctrl) + n_chunks * (size_t)s->n_v * blk_floats(s->dv) * sizeof(float);
}

cudaError_t launch_gdn_chunked(const moe_gdn_shape_t* s, const uint16_t* q, const uint16_t* k,
                               const uint16_t* v, const float* alpha, const float* beta,
                               const float* s_in, float* s_out, uint16_t* o, float* ws,
                               cudaStream_t stream) {
  static bool attr_set = false;
  constexpr int prep_smem = kPrepSmemBytes;
  constexpr int scan16 = scan_smem_floats<16>() * 4, scan_tc = kTcSmemFloats * 4;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(gdn_chunk_prep_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, prep_smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(gdn_chunk_scan_kernel<16>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, scan16);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(gdn_chunk_scan_tc_kernel,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, scan_tc);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int n_chunks = (s->T + kCh - 1) / kCh;
  Ctrl* ctrl = reinterpret_cast<Ctrl*>(ws);
  ws += sizeof(Ctrl) / sizeof(float);
  cudaError_t e = launch_pdl(gdn_chunk_prep_kernel, dim3(n_chunks, s->n_v), dim3(kThr),
                             (size_t)prep_smem, stream, q, k, v, alpha, beta, s->T, s->n_k, s->n_v,
                             s->dv, ws, ctrl);
  if (e != cudaSuccess) return e;
  // the tensor-core scan (32 state rows per CTA) when dv allows, else the
  // CUDA-core one with 16 rows
  if (s->dv % 32 == 0)
    return launch_pdl(gdn_chunk_scan_tc_kernel, dim3(s->n_v, s->dv / 32), dim3(kThr),
                      (size_t)scan_tc, stream, q, k, (const float*)ws, s_in, s_out, o, s->T, s->n_k,
                      s->n_v, s->dv);
  return launch_pdl(gdn_chunk_scan_kernel<16>, dim3(s->n_v, s->dv / 16), dim3(kThr), (size_t)scan16,
                    stream, q, k, (const float*)ws, s_in, s_out, o, s->T, s->n_k, s->n_v, s->dv);
}

}  // namespace moe
