// The fixed-size recurrence of the Gated DeltaNet layers ("Perplexity Open
// Sources Lily: A Rust + Metal Inference Engine for Qwen3.6-35B-A3B on Apple
// Silicon", section "Three Workload Shapes": 30 of the 40 layers are Gated
// DeltaNet; section "Prefill": a register-resident Gated DeltaNet scan) in
// the published gated delta rule: per value head, state S [dv][dk] and
// token t,
//   S <- alpha_t S (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,  o_t = S q_t.
//
// Row i of the update needs only row i of S:
//   S_i <- alpha S_i + (beta v_i - alpha beta (S_i . k)) k^T,
// so each warp keeps two rows of S in registers (lane L holds elements
// 4L..4L+3 of each) through all T tokens: per token two dot products over
// the warp (S_i . k before the update, S_i . q after it), fp32. The state is
// read once and written once per call; a CTA of 8 warps takes 16 rows of
// one head. The tokens' k, q, gates and the CTA's v entries are staged in
// shared memory 64 tokens at a time, so the scan itself reads no global
// memory.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {
constexpr int kGRows = 16;  // state rows per CTA (8 warps x 2)
constexpr int kGThreads = 256;
constexpr int kGChunk = 64;  // tokens staged in shared memory at a time

__device__ __forceinline__ float gdn_warp_sum(float v) {
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, d);
  return v;
}
// 4 bf16 at p (shared memory, 8-byte aligned) as floats
__device__ __forceinline__ void ld_bf4(const uint16_t* p, float (&f)[4]) {
  const uint2 w = *reinterpret_cast<const uint2*>(p);
  f[0] = bf_lo(w.x);
  f[1] = bf_hi(w.x);
  f[2] = bf_lo(w.y);
  f[3] = bf_hi(w.y);
}
}  // namespace

// grid (n_v, dv / 16); state rows r0 = 16 * blockIdx.y + 2 * warp, r0 + 1.
// s_in and s_out may be the same buffer (every CTA reads its rows before it
// writes them, and no other CTA touches them).
__global__ void __launch_bounds__(kGThreads)
    gdn_scan_kernel(const uint16_t* __restrict__ q, const uint16_t* __restrict__ k,
                    const uint16_t* __restrict__ v, const float* __restrict__ alpha,
                    const float* __restrict__ beta, const float* s_in, float* s_out,
                    uint16_t* __restrict__ o, int T, int n_k, int n_v, int dv) {
  constexpr int DK = 128;
  __shared__ __align__(16) uint16_t sk[kGChunk][DK], sq[kGChunk][DK];
  __shared__ float sa[kGChunk], sb[kGChunk];
  __shared__ uint16_t sv[kGChunk][kGRows];
  const int h = blockIdx.x, hk = h / (n_v / n_k);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r0 = kGRows * blockIdx.y + 2 * warp, r1 = r0 + 1;
  const size_t srow0 = ((size_t)h * dv + r0) * DK + 4 * lane;
  const size_t srow1 = srow0 + DK;
  float s0[4], s1[4];
  pdl_wait();  // programmatic dependent launch: global memory only after this
  pdl_trigger();
  {
    const float4 a = *reinterpret_cast<const float4*>(s_in + srow0);
    const float4 b = *reinterpret_cast<const float4*>(s_in + srow1);
    s0[0] = a.x; s0[1] = a.y; s0[2] = a.z; s0[3] = a.w;
    s1[0] = b.x; s1[1] = b.y; s1[2] = b.z; s1[3] = b.w;
  }
  const int rbase = kGRows * blockIdx.y;
  for (int t0 = 0; t0 < T; t0 += kGChunk) {
    const int nt = min(kGChunk, T - t0);
    __syncthreads();  // the previous chunk is consumed
    for (int i = threadIdx.x; i < nt * (DK / 8); i += kGThreads) {
      const int tt = i / (DK / 8), ch = i - tt * (DK / 8);
      const size_t src = ((size_t)(t0 + tt) * n_k + hk) * DK + ch * 8;
      *reinterpret_cast<uint4*>(&sk[tt][ch * 8]) = __ldg(reinterpret_cast<const uint4*>(k + src));
      *reinterpret_cast<uint4*>(&sq[tt][ch * 8]) = __ldg(reinterpret_cast<const uint4*>(q + src));
    }
    for (int i = threadIdx.x; i < nt; i += kGThreads) {
      sa[i] = __ldg(alpha + (size_t)(t0 + i) * n_v + h);
      sb[i] = __ldg(beta + (size_t)(t0 + i) * n_v + h);
    }
    for (int i = threadIdx.x; i < nt * kGRows; i += kGThreads) {
      const int tt = i / kGRows, rr = i - tt * kGRows;
      sv[tt][rr] = __ldg(v + ((size_t)(t0 + tt) * n_v + h) * dv + rbase + rr);
    }
    __syncthreads();
    for (int tt = 0; tt < nt; ++tt) {
      const int t = t0 + tt;
      float kk[4], qq[4];
      ld_bf4(&sk[tt][4 * lane], kk);
      ld_bf4(&sq[tt][4 * lane], qq);
      const float a = sa[tt], b = sb[tt];
      const float v0 = __uint_as_float((uint32_t)sv[tt][r0 - rbase] << 16);
      const float v1 = __uint_as_float((uint32_t)sv[tt][r1 - rbase] << 16);
      float d0 = 0.0f, d1 = 0.0f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        d0 = fmaf(s0[e], kk[e], d0);
        d1 = fmaf(s1[e], kk[e], d1);
      }
      d0 = gdn_warp_sum(d0);
      d1 = gdn_warp_sum(d1);
      const float c0 = b * v0 - a * b * d0, c1 = b * v1 - a * b * d1;
      float o0 = 0.0f, o1 = 0.0f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        s0[e] = fmaf(a, s0[e], c0 * kk[e]);
        s1[e] = fmaf(a, s1[e], c1 * kk[e]);
        o0 = fmaf(s0[e], qq[e], o0);
        o1 = fmaf(s1[e], qq[e], o1);
      }
      o0 = gdn_warp_sum(o0);
      o1 = gdn_warp_sum(o1);
      if (lane == 0) {
        uint16_t* ot = o + ((size_t)t * n_v + h) * dv;
        ot[r0] = (uint16_t)f2bf(o0);
        ot[r1] = (uint16_t)f2bf(o1);
      }
    }
  }
  *reinterpret_cast<float4*>(s_out + srow0) = make_float4(s0[0], s0[1], s0[2], s0[3]);
  *reinterpret_cast<float4*>(s_out + srow1) = make_float4(s1[0], s1[1], s1[2], s1[3]);
}

bool gdn_supported(const moe_gdn_shape_t* s) {
  return s && s->T >= 1 && s->n_k >= 1 && s->n_v >= 1 && s->n_v % s->n_k == 0 && s->dk == 128 &&
         s->dv >= kGRows && s->dv % kGRows == 0 && s->n_v <= 65535 && s->dv / kGRows <= 65535;
}

cudaError_t launch_gdn_scan(const moe_gdn_shape_t* s, const uint16_t* q, const uint16_t* k,
                            const uint16_t* v, const float* alpha, const float* beta,
                            const float* s_in, float* s_out, uint16_t* o, cudaStream_t stream) {
  dim3 grid(s->n_v, s->dv / kGRows);
  return launch_pdl(gdn_scan_kernel, grid, dim3(kGThreads), 0, stream, q, k, v, alpha, beta, s_in,
                    s_out, o, s->T, s->n_k, s->n_v, s->dv);
}

}  // namespace moe
