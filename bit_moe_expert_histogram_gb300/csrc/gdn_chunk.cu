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
// Two launches:
//   gdn_chunk_prep_kernel  one CTA per (chunk, value head), all chunks at
//                          once: g, K K^T and Q K^T, A, then W1 and W2 by
//                          forward substitution (each thread owns one
//                          column of [W1 | W2], so the substitution needs no
//                          barrier), and P = Mk o Q K^T, into the workspace
//   gdn_chunk_scan_kernel  one CTA per (value head, 32 or 16 state rows): row i of
//                          S only ever meets row i of the state, so the
//                          chunks run in order within the CTA and the rows
//                          of a head in parallel across CTAs; U, O and the
//                          new rows from the chunk's W1, W2, P, Q and K
// All arithmetic is fp32 (the inputs are bf16, exact in fp32).
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {
constexpr int kDK = 128;   // key head size
constexpr int kCh = 64;    // tokens per chunk
constexpr int kThr = 256;

// per (chunk, head) block of the workspace: W1 [C][dv], W2 [C][dk], P [C][C], g [C]
__host__ __device__ __forceinline__ size_t blk_floats(int dv) {
  return (size_t)kCh * dv + (size_t)kCh * kDK + (size_t)kCh * kCh + kCh;
}

__device__ __forceinline__ void bf8_to_f(const uint4& v, float* f) {
  f[0] = bf_lo(v.x); f[1] = bf_hi(v.x); f[2] = bf_lo(v.y); f[3] = bf_hi(v.y);
  f[4] = bf_lo(v.z); f[5] = bf_hi(v.z); f[6] = bf_lo(v.w); f[7] = bf_hi(v.w);
}

constexpr int kPrepSmemFloats = kDK * kCh * 2 + kCh * kDK + kCh * kCh + kCh * 256 + 2 * kCh;
constexpr int kLd = kDK + 1;  // padded row of a [C][dk] tile: rows t and t+1 start in other banks
constexpr int kLdP = kCh + 1;
template <int R>
constexpr int scan_smem_floats() {
  return kDK * (R + 1) + 2 * kCh * kLd + kCh * kDK + kCh * kLdP + 3 * kCh * R + kCh;
}
}  // namespace

__global__ void __launch_bounds__(kThr, 1)
    gdn_chunk_prep_kernel(const uint16_t* __restrict__ q, const uint16_t* __restrict__ k,
                          const uint16_t* __restrict__ v, const float* __restrict__ alpha,
                          const float* __restrict__ beta, int T, int n_k, int n_v, int dv,
                          float* __restrict__ ws) {
  extern __shared__ float sm[];
  float* KT = sm;                // [dk][C]  K transposed
  float* QT = KT + kDK * kCh;    // [dk][C]  Q transposed
  float* V = QT + kDK * kCh;     // [C][128] (dv columns used)
  float* A = V + kCh * kDK;      // [C][C]
  float* W = A + kCh * kCh;      // [C][256]: columns 0..dv-1 W1, 128..255 W2
  float* g = W + kCh * 256;      // [C]
  float* bt = g + kCh;           // [C]
  const int tid = threadIdx.x;
  const int c = blockIdx.x, h = blockIdx.y, hk = h / (n_v / n_k);
  const int t0 = c * kCh, n = min(kCh, T - t0);
  // tokens past the sequence end read as k = q = v = 0, alpha = 1, beta = 0:
  // they leave every quantity below unchanged
  for (int idx = tid; idx < kCh * (kDK / 8); idx += kThr) {
    const int t = idx % kCh, ch = idx / kCh;
    float kf[8] = {0, 0, 0, 0, 0, 0, 0, 0}, qf[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    if (t < n) {
      const size_t src = ((size_t)(t0 + t) * n_k + hk) * kDK + ch * 8;
      bf8_to_f(__ldg(reinterpret_cast<const uint4*>(k + src)), kf);
      bf8_to_f(__ldg(reinterpret_cast<const uint4*>(q + src)), qf);
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      KT[(ch * 8 + e) * kCh + t] = kf[e];
      QT[(ch * 8 + e) * kCh + t] = qf[e];
    }
  }
  const int vch = dv / 8;
  for (int idx = tid; idx < kCh * vch; idx += kThr) {
    const int t = idx / vch, ch = idx % vch;
    float vf[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    if (t < n)
      bf8_to_f(__ldg(reinterpret_cast<const uint4*>(v + ((size_t)(t0 + t) * n_v + h) * dv + ch * 8)),
               vf);
    float4* dst = reinterpret_cast<float4*>(V + t * kDK + ch * 8);
    dst[0] = make_float4(vf[0], vf[1], vf[2], vf[3]);
    dst[1] = make_float4(vf[4], vf[5], vf[6], vf[7]);
  }
  if (tid < kCh) {
    g[tid] = tid < n ? __ldg(alpha + (size_t)(t0 + tid) * n_v + h) : 1.0f;
    bt[tid] = tid < n ? __ldg(beta + (size_t)(t0 + tid) * n_v + h) : 0.0f;
  }
  __syncthreads();
  if (tid == 0) {  // g_t = alpha_1 ... alpha_t
    float p = 1.0f;
    for (int t = 0; t < kCh; ++t) {
      p *= g[t];
      g[t] = p;
    }
  }
  __syncthreads();
  float* blk = ws + ((size_t)c * n_v + h) * blk_floats(dv);
  float* gW1 = blk;
  float* gW2 = gW1 + (size_t)kCh * dv;
  float* gP = gW2 + (size_t)kCh * kDK;
  float* gG = gP + (size_t)kCh * kCh;
  {
    // K K^T and Q K^T, 4 x 4 tiles: rows t = 4ty.., columns s = 4tx..
    const int ty = tid >> 4, tx = tid & 15;
    float ga[4][4], qa[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) ga[a][b] = qa[a][b] = 0.0f;
#pragma unroll 4
    for (int j = 0; j < kDK; ++j) {
      const float4 kt = *reinterpret_cast<const float4*>(KT + j * kCh + 4 * ty);
      const float4 ks = *reinterpret_cast<const float4*>(KT + j * kCh + 4 * tx);
      const float4 qt = *reinterpret_cast<const float4*>(QT + j * kCh + 4 * ty);
      const float kr[4] = {kt.x, kt.y, kt.z, kt.w}, kc[4] = {ks.x, ks.y, ks.z, ks.w};
      const float qr[4] = {qt.x, qt.y, qt.z, qt.w};
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          ga[a][b] = __fmaf_rn(kr[a], kc[b], ga[a][b]);
          qa[a][b] = __fmaf_rn(qr[a], kc[b], qa[a][b]);
        }
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int t = 4 * ty + a;
      float pr[4];
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int s = 4 * tx + b;
        const float ratio = g[t] / g[s];
        A[t * kCh + s] = s < t ? bt[t] * ratio * ga[a][b] : 0.0f;
        pr[b] = s <= t ? ratio * qa[a][b] : 0.0f;
      }
      *reinterpret_cast<float4*>(gP + (size_t)t * kCh + 4 * tx) = make_float4(pr[0], pr[1], pr[2], pr[3]);
    }
  }
  if (tid < kCh) gG[tid] = g[tid];
  __syncthreads();
  // W1 = (I + A)^-1 diag(beta) V, W2 = (I + A)^-1 diag(beta g) K: thread
  // `col` owns one column and substitutes forward, row after row
  const int col = tid;
  const bool is_w1 = col < dv;
  const bool is_w2 = col >= 128 && col - 128 < kDK;
  if (is_w1 || is_w2) {
    for (int t = 0; t < kCh; ++t) {
      // four interleaved partial sums keep the dependent chain short
      float x0 = is_w1 ? bt[t] * V[t * kDK + col] : bt[t] * g[t] * KT[(col - 128) * kCh + t];
      float x1 = 0.0f, x2 = 0.0f, x3 = 0.0f;
      int s = 0;
      for (; s + 4 <= t; s += 4) {
        x0 = __fmaf_rn(-A[t * kCh + s], W[s * 256 + col], x0);
        x1 = __fmaf_rn(-A[t * kCh + s + 1], W[(s + 1) * 256 + col], x1);
        x2 = __fmaf_rn(-A[t * kCh + s + 2], W[(s + 2) * 256 + col], x2);
        x3 = __fmaf_rn(-A[t * kCh + s + 3], W[(s + 3) * 256 + col], x3);
      }
      for (; s < t; ++s) x0 = __fmaf_rn(-A[t * kCh + s], W[s * 256 + col], x0);
      const float x = (x0 + x1) + (x2 + x3);
      W[t * 256 + col] = x;
      if (is_w1)
        gW1[(size_t)t * dv + col] = x;
      else
        gW2[(size_t)t * kDK + (col - 128)] = x;
    }
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
  float* g = Ug + kCh * R;               // [C]
  const int tid = threadIdx.x;
  const int h = blockIdx.x, hk = h / (n_v / n_k);
  const int r0 = R * blockIdx.y;
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
    for (int idx = tid; idx < kCh * kDK / 4; idx += kThr) {  // coalesced, 16 bytes a thread
      const int t = idx / (kDK / 4), j = (idx % (kDK / 4)) * 4;
      const float4 w = __ldcg(reinterpret_cast<const float4*>(gW2 + (size_t)t * kDK + j));
      float* d = W2 + t * kLd + j;
      d[0] = w.x; d[1] = w.y; d[2] = w.z; d[3] = w.w;
    }
    for (int idx = tid; idx < kCh * kCh / 4; idx += kThr) {
      const int t = idx / (kCh / 4), sc = (idx % (kCh / 4)) * 4;
      const float4 w = __ldcg(reinterpret_cast<const float4*>(gP + (size_t)t * kCh + sc));
      float* d = P + t * kLdP + sc;
      d[0] = w.x; d[1] = w.y; d[2] = w.z; d[3] = w.w;
    }
    for (int idx = tid; idx < kCh * R; idx += kThr) {
      const int t = idx / R, i = idx % R;
      W1r[idx] = __ldcg(gW1 + (size_t)t * dv + r0 + i);
    }
    if (tid < kCh) g[tid] = __ldcg(gG + tid);
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
      Ug[ot * R + oi + e] = uu * (gC / g[ot]);
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

size_t gdn_chunk_ws_bytes(const moe_gdn_shape_t* s) {
  const size_t n_chunks = ((size_t)s->T + kCh - 1) / kCh;
  return n_chunks * (size_t)s->n_v * blk_floats(s->dv) * sizeof(float);
}

cudaError_t launch_gdn_chunked(const moe_gdn_shape_t* s, const uint16_t* q, const uint16_t* k,
                               const uint16_t* v, const float* alpha, const float* beta,
                               const float* s_in, float* s_out, uint16_t* o, float* ws,
                               cudaStream_t stream) {
  static bool attr_set = false;
  constexpr int prep_smem = kPrepSmemFloats * 4;
  constexpr int scan16 = scan_smem_floats<16>() * 4, scan32 = scan_smem_floats<32>() * 4;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(gdn_chunk_prep_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, prep_smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(gdn_chunk_scan_kernel<16>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, scan16);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(gdn_chunk_scan_kernel<32>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, scan32);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int n_chunks = (s->T + kCh - 1) / kCh;
  gdn_chunk_prep_kernel<<<dim3(n_chunks, s->n_v), kThr, prep_smem, stream>>>(
      q, k, v, alpha, beta, s->T, s->n_k, s->n_v, s->dv, ws);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // 32 state rows per CTA when dv allows (fewer CTAs re-reading each chunk's tiles)
  if (s->dv % 32 == 0)
    gdn_chunk_scan_kernel<32><<<dim3(s->n_v, s->dv / 32), kThr, scan32, stream>>>(
        q, k, ws, s_in, s_out, o, s->T, s->n_k, s->n_v, s->dv);
  else
    gdn_chunk_scan_kernel<16><<<dim3(s->n_v, s->dv / 16), kThr, scan16, stream>>>(
        q, k, ws, s_in, s_out, o, s->T, s->n_k, s->n_v, s->dv);
  return cudaGetLastError();
}

}  // namespace moe
