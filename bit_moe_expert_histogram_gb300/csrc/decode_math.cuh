// Arithmetic shared by the decode kernels: the packed-weight dot products
// on the CUDA cores, warp sums, the unit-RMS normalisation, the activation
// layout in shared memory and the release / acquire accessors.
//
// "Perplexity Open Sources Lily: A Rust + Metal Inference Engine for
// Qwen3.6-35B-A3B on Apple Silicon", sections "Prefill: Keep Weights Packed,
// Keep Routing on the GPU" (groupwise-affine 4-bit weights, 64 per group,
// bf16 scale and bias) and "Decode: Minimize Bytes Moved Per Token" (the
// packed bytes are streamed once and expanded on chip).
#pragma once
#include "common.cuh"

namespace moe {

// acc + lo(p)*half(xa) + hi(p)*half(xb), half = low (HI=0) or high (HI=1):
// fp32 fma with bf16 operands (the product is exact, one rounding per fma,
// the same result as converting both operands to fp32 first).
template <int HI>
__device__ __forceinline__ float fma_pair(uint32_t p, uint32_t xa, uint32_t xb, float acc) {
  if (HI == 0)
    asm("{\n\t.reg .b16 pl, ph, al, ah, bl, bh;\n\t"
        "mov.b32 {pl, ph}, %1;\n\tmov.b32 {al, ah}, %2;\n\tmov.b32 {bl, bh}, %3;\n\t"
        "fma.rn.f32.bf16 %0, pl, al, %0;\n\tfma.rn.f32.bf16 %0, ph, bl, %0;\n\t}"
        : "+f"(acc)
        : "r"(p), "r"(xa), "r"(xb));
  else
    asm("{\n\t.reg .b16 pl, ph, al, ah, bl, bh;\n\t"
        "mov.b32 {pl, ph}, %1;\n\tmov.b32 {al, ah}, %2;\n\tmov.b32 {bl, bh}, %3;\n\t"
        "fma.rn.f32.bf16 %0, pl, ah, %0;\n\tfma.rn.f32.bf16 %0, ph, bh, %0;\n\t}"
        : "+f"(acc)
        : "r"(p), "r"(xa), "r"(xb));
  return acc;
}

// acc + the 8 products of packed word q (group scale s2, bias b2 in both
// halves) with 8 bf16 activations in natural pairs v = (x0x1, x2x3, x4x5,
// x6x7): weight pair i of dequant_word_i4 meets (xi, xi+4).
__device__ __forceinline__ float dot8(uint32_t q, uint32_t s2, uint32_t b2, const uint4& v,
                                     float acc) {
  uint32_t p[4];
  dequant_word_i4(q, s2, b2, p);
  acc = fma_pair<0>(p[0], v.x, v.z, acc);
  acc = fma_pair<1>(p[1], v.x, v.z, acc);
  acc = fma_pair<0>(p[2], v.y, v.w, acc);
  acc = fma_pair<1>(p[3], v.y, v.w, acc);
  return acc;
}

// acc + the 32 products of one 16-byte chunk of packed weights (4 words)
// with the chunk's 32 activations (4 x 8 bf16).
__device__ __forceinline__ float dot32(const uint4& q, uint32_t s2, uint32_t b2, const uint4 xv[4],
                                      float acc) {
  acc = dot8(q.x, s2, b2, xv[0], acc);
  acc = dot8(q.y, s2, b2, xv[1], acc);
  acc = dot8(q.z, s2, b2, xv[2], acc);
  acc = dot8(q.w, s2, b2, xv[3], acc);
  return acc;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, d);
  return v;
}

// 1 / sqrt(mean(y^2) + 1e-6) of one token from its nb block partials of y^2,
// summed in one fixed order: partial i to lane i mod 32 (ascending), then an
// xor butterfly over distances 16..1. Called by a whole warp; every lane
// returns the same value.
__device__ __forceinline__ float rms_inv_warp(const float* part, int nb, int H, int lane) {
  float s = 0.0f;
#pragma unroll 8
  for (int i = lane; i < nb; i += 32) s += __ldcg(part + i);
  s = warp_sum(s);
  return 1.0f / sqrtf(s / (float)H + 1e-6f);
}
// the normalised next-layer input: bf16(y * inv) of 8 packed bf16 y values
__device__ __forceinline__ uint4 norm_chunk(const uint4& v, float inv) {
  uint4 o;
  o.x = pack_bf2(bf_lo(v.x) * inv, bf_hi(v.x) * inv);
  o.y = pack_bf2(bf_lo(v.y) * inv, bf_hi(v.y) * inv);
  o.z = pack_bf2(bf_lo(v.z) * inv, bf_hi(v.z) * inv);
  o.w = pack_bf2(bf_lo(v.w) * inv, bf_hi(v.w) * inv);
  return o;
}

// Activation rows in shared memory, bf16: chunk c (elements 32c..32c+31,
// 64 bytes) keeps its 16-byte piece v at (v + c/2) mod 4. A lane reads the
// four pieces of its own chunk and consecutive lanes take consecutive
// chunks, so each 8-lane phase of a 16-byte load touches 8 distinct bank
// quads.
__device__ __forceinline__ int act_piece_off(int c, int v) { return c * 64 + 16 * ((v + (c >> 1)) & 3); }

__device__ __forceinline__ void act_load_chunk(const uint8_t* row, int c, uint4 xv[4]) {
#pragma unroll
  for (int v = 0; v < 4; ++v) xv[v] = *reinterpret_cast<const uint4*>(row + act_piece_off(c, v));
}

__device__ __forceinline__ uint32_t ld_acquire(const unsigned* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release(unsigned* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t atom_add_acq_rel(unsigned* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

}  // namespace moe
