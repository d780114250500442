// Weighted combine of the expert outputs back to token order, and the
// debug dequantisation kernel.
//
// y[t] = bf16( sum_{k asc} w[t][k] * y_slots[row_pos[t*K+k]] + y_slots[R+t] )
// in fp32 in that fixed order (the shared expert sees every token with
// weight 1: "Perplexity Open Sources Lily: A Rust + Metal Inference Engine
// for Qwen3.6-35B-A3B on Apple Silicon", section "Three Workload Shapes").
// With x_next, the bf16 y is also normalised to unit RMS,
// y / sqrt(mean(y^2) + 1e-6), as the input of a stacked next layer.
// Decoder blocks (h_out set): the residual stream moves on,
// h_out = bf16(h_in + y), and x_next = bf16(gain * (h_out * inv)) with inv
// of h_out; y itself is written only when y is not null.
#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int kCombineBatch = 8;

// One block per token; thread c owns the 8 elements [8c, 8c+8).
__global__ void __launch_bounds__(1024)
    combine_kernel(const uint16_t* __restrict__ y_slots, const int32_t* __restrict__ row_pos,
                   const float* __restrict__ w, int H, int K, int R, int n_shared,
                   uint16_t* __restrict__ y, uint16_t* __restrict__ x_next, const uint16_t* h_in,
                   uint16_t* h_out, const uint16_t* __restrict__ gain) {
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
  const int c = threadIdx.x;  // blockDim.x == H/8: one 16-byte chunk per thread
  // the token's slot rows and weights, then its rows in batches of
  // kCombineBatch with every load of a batch in flight (the sum keeps the
  // ascending k order)
  const uint4* ys = reinterpret_cast<const uint4*>(y_slots);
  const size_t hv = (size_t)H / 8;
  uint4 vsh = make_uint4(0u, 0u, 0u, 0u);
  if (n_shared) vsh = __ldg(ys + (size_t)(R + t) * hv + c);
  for (int k0 = 0; k0 < K; k0 += kCombineBatch) {
    int r[kCombineBatch];
    float wk[kCombineBatch];
#pragma unroll
    for (int j = 0; j < kCombineBatch; ++j) {
      r[j] = k0 + j < K ? __ldg(row_pos + t * K + k0 + j) : 0;
      wk[j] = k0 + j < K ? __ldg(w + t * K + k0 + j) : 0.0f;
    }
    uint4 v[kCombineBatch];
#pragma unroll
    for (int j = 0; j < kCombineBatch; ++j)
      v[j] = k0 + j < K ? __ldg(ys + (size_t)r[j] * hv + c) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int j = 0; j < kCombineBatch; ++j) {
      if (k0 + j >= K) break;
      acc[0] = __fmaf_rn(wk[j], bf_lo(v[j].x), acc[0]);
      acc[1] = __fmaf_rn(wk[j], bf_hi(v[j].x), acc[1]);
      acc[2] = __fmaf_rn(wk[j], bf_lo(v[j].y), acc[2]);
      acc[3] = __fmaf_rn(wk[j], bf_hi(v[j].y), acc[3]);
      acc[4] = __fmaf_rn(wk[j], bf_lo(v[j].z), acc[4]);
      acc[5] = __fmaf_rn(wk[j], bf_hi(v[j].z), acc[5]);
      acc[6] = __fmaf_rn(wk[j], bf_lo(v[j].w), acc[6]);
      acc[7] = __fmaf_rn(wk[j], bf_hi(v[j].w), acc[7]);
    }
  }
  if (n_shared) {
    const uint4 v = vsh;
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
  if (y) reinterpret_cast<uint4*>(y + (size_t)t * H)[c] = o;
  if (h_out) {  // the residual add (h_out may be h_in: each thread its own chunk)
    const uint4 hv = reinterpret_cast<const uint4*>(h_in + (size_t)t * H)[c];
    o.x = pack_bf2(bf_lo(hv.x) + bf_lo(o.x), bf_hi(hv.x) + bf_hi(o.x));
    o.y = pack_bf2(bf_lo(hv.y) + bf_lo(o.y), bf_hi(hv.y) + bf_hi(o.y));
    o.z = pack_bf2(bf_lo(hv.z) + bf_lo(o.z), bf_hi(hv.z) + bf_hi(o.z));
    o.w = pack_bf2(bf_lo(hv.w) + bf_lo(o.w), bf_hi(hv.w) + bf_hi(o.w));
    reinterpret_cast<uint4*>(h_out + (size_t)t * H)[c] = o;
  }
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
    float gv[8] = {1.f, 1.f, 1.f, 1.f, 1.f, 1.f, 1.f, 1.f};
    if (gain) {
      const uint4 g = __ldg(reinterpret_cast<const uint4*>(gain) + c);
      gv[0] = bf_lo(g.x); gv[1] = bf_hi(g.x); gv[2] = bf_lo(g.y); gv[3] = bf_hi(g.y);
      gv[4] = bf_lo(g.z); gv[5] = bf_hi(g.z); gv[6] = bf_lo(g.w); gv[7] = bf_hi(g.w);
    }
    uint4 n;
    if (gain) {
      n.x = pack_bf2(gv[0] * (yb[0] * inv), gv[1] * (yb[1] * inv));
      n.y = pack_bf2(gv[2] * (yb[2] * inv), gv[3] * (yb[3] * inv));
      n.z = pack_bf2(gv[4] * (yb[4] * inv), gv[5] * (yb[5] * inv));
      n.w = pack_bf2(gv[6] * (yb[6] * inv), gv[7] * (yb[7] * inv));
    } else {
      n.x = pack_bf2(yb[0] * inv, yb[1] * inv);
      n.y = pack_bf2(yb[2] * inv, yb[3] * inv);
      n.z = pack_bf2(yb[4] * inv, yb[5] * inv);
      n.w = pack_bf2(yb[6] * inv, yb[7] * inv);
    }
    reinterpret_cast<uint4*>(x_next + (size_t)t * H)[c] = n;
  }
}

// The first decoder block's input: h_0 = the caller's h, or the embedding
// rows of the token ids (copied to h0_out; an id outside [0, vocab) is
// recorded and reads as a zero row), and x = bf16(gain * (h_0 * inv)),
// inv = 1/sqrt(mean(h_0^2) + 1e-6). One block per token, thread c owns the
// 8 elements [8c, 8c+8).
__global__ void __launch_bounds__(1024) block_input_kernel(
    const uint16_t* __restrict__ h_in, const int32_t* __restrict__ tok,
    const uint16_t* __restrict__ embed, int vocab, const uint16_t* __restrict__ gain, int H,
    uint16_t* __restrict__ h0_out, uint16_t* __restrict__ x, Ctrl* ctrl) {
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x, c = threadIdx.x;
  uint4 v = make_uint4(0u, 0u, 0u, 0u);
  if (tok) {
    const int id = __ldg(tok + t);
    if (id >= 0 && id < vocab)
      v = __ldg(reinterpret_cast<const uint4*>(embed + (size_t)id * H) + c);
    else if (c == 0)
      set_error(ctrl, MOE_ERR_BAD_INPUT, KID_DECODE, id);
    reinterpret_cast<uint4*>(h0_out + (size_t)t * H)[c] = v;
  } else {
    v = __ldg(reinterpret_cast<const uint4*>(h_in + (size_t)t * H) + c);
  }
  const float hb[8] = {bf_lo(v.x), bf_hi(v.x), bf_lo(v.y), bf_hi(v.y),
                       bf_lo(v.z), bf_hi(v.z), bf_lo(v.w), bf_hi(v.w)};
  float ss = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) ss = __fmaf_rn(hb[i], hb[i], ss);
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, d);
  __shared__ float wsum[32];
  if ((threadIdx.x & 31) == 0) wsum[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.0f;
  for (int i = 0; i < (int)(blockDim.x >> 5); ++i) tot += wsum[i];
  const float inv = 1.0f / sqrtf(tot / (float)H + 1e-6f);
  const uint4 g = __ldg(reinterpret_cast<const uint4*>(gain) + c);
  uint4 n;
  n.x = pack_bf2(bf_lo(g.x) * (hb[0] * inv), bf_hi(g.x) * (hb[1] * inv));
  n.y = pack_bf2(bf_lo(g.y) * (hb[2] * inv), bf_hi(g.y) * (hb[3] * inv));
  n.z = pack_bf2(bf_lo(g.z) * (hb[4] * inv), bf_hi(g.z) * (hb[5] * inv));
  n.w = pack_bf2(bf_lo(g.w) * (hb[6] * inv), bf_hi(g.w) * (hb[7] * inv));
  reinterpret_cast<uint4*>(x + (size_t)t * H)[c] = n;
}

cudaError_t launch_block_input(const uint16_t* h_in, const int32_t* tok, const uint16_t* embed,
                               int vocab, const uint16_t* gain, int T, int H, uint16_t* h0_out,
                               uint16_t* x, Ctrl* ctrl, cudaStream_t stream) {
  return launch_pdl(block_input_kernel, dim3(T), dim3(H / 8), 0, stream, h_in, tok, embed, vocab,
                    gain, H, h0_out, x, ctrl);
}

cudaError_t launch_combine(const uint16_t* y_slots, const int32_t* row_pos, const float* w, int T,
                           int H, int K, int n_shared, uint16_t* y, uint16_t* x_next,
                           cudaStream_t stream, const uint16_t* h_in, uint16_t* h_out,
                           const uint16_t* gain) {
  const int threads = H / 8;  // H % 256 == 0 -> a whole number of warps, <= 1024 by validation
  return launch_pdl(combine_kernel, dim3(T), dim3(threads), 0, stream, y_slots, row_pos, w, H, K,
                    T * K, n_shared, y, x_next, h_in, h_out, gain);
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

// Debug: the same with the decode kernels' routine (dequant_word_i4), its
// (i, i+4) pairs put back into natural element order.
__global__ void dequant_i4_kernel(const uint32_t* __restrict__ q, const uint16_t* __restrict__ s,
                                  const uint16_t* __restrict__ b, uint16_t* __restrict__ out,
                                  int N, int Kd) {
  const size_t words = (size_t)N * (Kd / 8);
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < words;
       i += (size_t)gridDim.x * blockDim.x) {
    const size_t n = i / (Kd / 8), wi = i % (Kd / 8);
    const size_t g = n * (Kd / 64) + wi / 8;
    const uint32_t s2 = s[g] | ((uint32_t)s[g] << 16);
    const uint32_t b2 = b[g] | ((uint32_t)b[g] << 16);
    uint32_t p[4];
    dequant_word_i4(q[i], s2, b2, p);
    // p[j] = (e_j, e_j+4): natural pairs (e0,e1), (e2,e3) from the low
    // halves, (e4,e5), (e6,e7) from the high halves
    reinterpret_cast<uint4*>(out)[i] =
        make_uint4(__byte_perm(p[0], p[1], 0x5410), __byte_perm(p[2], p[3], 0x5410),
                   __byte_perm(p[0], p[1], 0x7632), __byte_perm(p[2], p[3], 0x7632));
  }
}

cudaError_t launch_dequant(const uint32_t* q, const uint16_t* s, const uint16_t* b, uint16_t* out,
                           int N, int Kd, bool decode_routine, cudaStream_t stream) {
  const size_t words = (size_t)N * (Kd / 8);
  const int grid = (int)((words + 255) / 256 < 4096 ? (words + 255) / 256 : 4096);
  if (decode_routine)
    dequant_i4_kernel<<<grid, 256, 0, stream>>>(q, s, b, out, N, Kd);
  else
    dequant_kernel<<<grid, 256, 0, stream>>>(q, s, b, out, N, Kd);
  return cudaGetLastError();
}

}  // namespace moe
