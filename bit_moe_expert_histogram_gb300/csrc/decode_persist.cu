// Decode through stacked MoE layers in one persistent launch: one block of
// 16 warps per SM, every block resident at once (cooperative launch), the
// layers back to back with no kernel boundary between them.
//
// "Perplexity Open Sources Lily: A Rust + Metal Inference Engine for
// Qwen3.6-35B-A3B on Apple Silicon", section "Decode: Minimize Bytes Moved
// Per Token": at batch 1 a layer reuses almost no weight, so the time is
// the bytes moved plus every wait between dependent steps; the steps of a
// decode token are fused so intermediates stay on chip. Here the waits
// between layers and between the steps of a layer are block-to-block
// handoffs through L2, with no launch, no grid-wide barrier and no host.
//
// Per layer:
//   input    every block forms the layer input x in shared memory: layer 0
//            the caller's x; layer l > 0 bf16(y * inv), y the previous
//            layer's output and inv = 1/sqrt(mean(y^2) + 1e-6) from its
//            y^2 partials. Decoder blocks (BLOCK): every block keeps the
//            residual stream h in shared memory (layer 0: the caller's h or
//            the tokens' embedding rows; later: the previous layer's
//            h + y) and forms x = bf16(gain * (h * inv)) from it
//   router   units (t, e): the fixed-order fp32 logit of the prefill router
//            (so the selected ids are bit-identical with it)
//   top-K    every block selects each token's experts itself
//   gate_up  tiles of 8 gate rows j..j+7 and the 8 up rows I+j..I+j+7 of a
//            routed expert (one token) or of the shared expert (all tokens),
//            split along H over the 4 warps of a warp group; the partial
//            sums meet in shared memory -> SwiGLU -> h. Each warp sends its
//            down rows to L2 behind its first gate_up loads
//   down     items (t, g, pair of slots): output rows 8g..8g+7 of token t
//            for two slots, each times its slot's h, one warp each; the
//            slots are weighted and summed in slot order (shared expert
//            weight 1) -> bf16 y, and each row group's y^2 partial for the
//            next normalisation (BLOCK: y is added to h first, h' =
//            bf16(h + y), and h' and its square partials go on)
//
// The expert GEMVs run on the tensor cores (mma.sync m16n8k16, bf16 in,
// fp32 accumulate) with the weights rebuilt exactly on the CUDA cores:
// bf16(s*q + b), one rounding, as in the grouped GEMM. A 64-element
// segment of a row is 8 packed words; lane (g, c) of a warp (g = lane/4,
// c = lane%4) holds words 2c and 2c+1 of tile rows g and g+8. The
// rebuild pairs elements (i, i+4) of a word in one register, which is the
// A operand's (k, k+1) for the MMA's k-slots 2c.. of that lane; the
// activations are kept in shared memory in the same pairing, so the B
// operand is one 16-byte load. Which of a segment's elements meets which
// k-slot is a permutation of K, the same for A and B, so the products are
// those of the plain dot product.
//
// Block-to-block data (logits, h, y, y^2 partials) travels as 64-bit words
// (epoch << 32 | payload), written and read with single 64-bit accesses at
// GPU scope. The epoch names the layer and the launch; a reader polls its
// words until every tag is the one it expects, so the wait and the data
// take one L2 round trip. A word is never rewritten while a reader of its
// previous value may still come: the grid is capped so that every block
// owns at least one down unit and, for every token, at least one routed
// gate_up tile. A block writing layer l+1's logits or h has read all of
// layer l's y, which every block writes only after its last read of layer
// l's logits and h; a block writing layer l+1's y or partials has read
// h(l+1) of its token, which every block writes only after reading y(l).
// So a reader only ever meets its own epoch or an older one, and one copy
// of each buffer suffices.
//
// Every wait is bounded: a wait that runs out records MOE_ERR_TIMEOUT,
// raises the abort word, and every block then stops waiting and runs to
// the end; the last block out resets the launch's counters.
#include "common.cuh"
#include "decode_math.cuh"
#include "kernels.h"
#include "topk.cuh"

namespace moe {

namespace {

constexpr int kPsWarps = 16;
constexpr int kPsThreads = 32 * kPsWarps;
constexpr int kPsGroup = 8;     // down unit: output rows (one y^2 partial)
constexpr int kGuSlices = 4;    // gate_up tile: warps sharing it along H (a warp group)
constexpr int kSegBatch = 8;    // 64-element segments of a gate_up slice in registers at once
constexpr int kPsMaxT = 4;
constexpr int kPsMaxE = 256;    // logits per lane in the top-K: 8
constexpr int kPsMaxTH = 8192;  // T * H
static_assert(kPsMaxTH / 8 <= 4 * 2 * 4 * 4 * 16, "the input phase's partials fit the reduction buffer");
constexpr uint32_t kPsEpochStride = 64;  // epochs per launch (> kPersistMaxLayers)
// Tagged words are grouped by writer, one 128-byte line (16 words) per
// writer: a line that several SMs write while others poll it is handed
// over about twice as slowly.
constexpr int kLine = 16;
static_assert(kPsEpochStride > kPersistMaxLayers, "one epoch per layer and launch");

// ------------------------------------------------------- tagged words --
__device__ __forceinline__ uint64_t ld_tag(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_tag(uint64_t* p, uint32_t ep, uint32_t v) {
  const uint64_t w = ((uint64_t)ep << 32) | v;
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}
__device__ __forceinline__ uint32_t tag_of(uint64_t w) { return (uint32_t)(w >> 32); }

// Bounds one poll loop: call after every pass that still found a stale
// word; false = stop waiting (the abort word is up, or the limit passed,
// in which case this thread records the timeout and raises the abort).
struct Waiter {
  uint64_t t0 = 0;
  uint32_t n = 0;
  __device__ __forceinline__ bool keep_going(Ctrl* c, int where) {
    if (n++ == 0) t0 = globaltimer_ns();
    if ((n & 31u) == 0) {
      if (*reinterpret_cast<volatile unsigned*>(&c->ps_abort)) return false;
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        set_error(c, MOE_ERR_TIMEOUT, KID_DECODE, where);
        *reinterpret_cast<volatile unsigned*>(&c->ps_abort) = 1u;
        return false;
      }
    }
    return true;
  }
};

// Poll n tagged words at(i), i = threadIdx.x + 512 k, until each carries
// epoch ep, 8 per thread at a time; f(i, payload) receives every word once.
template <typename A, typename F>
__device__ __forceinline__ void poll_block(A at, int n, uint32_t ep, Ctrl* c, int where, F f) {
  for (int k0 = 0; k0 * kPsThreads < n; k0 += 8) {
    uint32_t v[8];
    uint32_t stale = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int i = threadIdx.x + (k0 + k) * kPsThreads;
      v[k] = 0;
      if (i < n) {
        const uint64_t w = ld_tag(at(i));
        v[k] = (uint32_t)w;
        if (tag_of(w) != ep) stale |= 1u << k;
      }
    }
    Waiter wt;
    while (stale) {
      if (!wt.keep_going(c, where)) break;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        if ((stale >> k) & 1u) {
          const uint64_t w = ld_tag(at(threadIdx.x + (k0 + k) * kPsThreads));
          v[k] = (uint32_t)w;
          if (tag_of(w) == ep) stale &= ~(1u << k);
        }
      }
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int i = threadIdx.x + (k0 + k) * kPsThreads;
      if (i < n) f(i, v[k]);
    }
  }
}

// 1/sqrt(mean(y^2) + 1e-6) of a token from its nb tagged partials (epoch
// ep; partial r at part[r * kLine]): lane L adds partials L, L + 32, .. in
// order (polled 8 at a time), then an xor butterfly. Whole warp; every
// lane returns the result.
__device__ __forceinline__ float ps_rms_inv(const uint64_t* part, int nb, int H, uint32_t ep,
                                            int lane, Ctrl* c) {
  float s = 0.0f;
  for (int m0 = 0; 32 * m0 < nb; m0 += 8) {
    float v[8];
    uint32_t stale = 0;
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      v[m] = 0.0f;
      if (32 * (m0 + m) < nb) {
        const uint64_t w = ld_tag(part + (size_t)(lane + 32 * (m0 + m)) * kLine);
        v[m] = __uint_as_float((uint32_t)w);
        if (tag_of(w) != ep) stale |= 1u << m;
      }
    }
    Waiter wt;
    while (__any_sync(0xFFFFFFFFu, stale != 0u)) {
      if (stale && !wt.keep_going(c, 1)) stale = 0;
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        if ((stale >> m) & 1u) {
          const uint64_t w = ld_tag(part + (size_t)(lane + 32 * (m0 + m)) * kLine);
          v[m] = __uint_as_float((uint32_t)w);
          if (tag_of(w) == ep) stale &= ~(1u << m);
        }
      }
    }
#pragma unroll
    for (int m = 0; m < 8; ++m)
      if (32 * (m0 + m) < nb) s += v[m];
  }
  s = warp_sum(s);
  return 1.0f / sqrtf(s / (float)H + 1e-6f);
}

// ---------------------------------------------------------------- MMA --
// d (16x8 fp32, accumulated) += A (16x16 bf16) * B (16x8 bf16): lane (g, c)
// holds A rows g / g+8 at k-slots {2c, 2c+1} (a0 / a1) and {2c+8, 2c+9}
// (a2 / a3), B column g at k-slots {2c, 2c+1} (b0) and {2c+8, 2c+9} (b1),
// and d rows g / g+8, columns 2c, 2c+1.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// One 64-element segment of a 16-row tile: this lane's words 2c, 2c+1 of
// rows g (wg) and g+8 (wh), their group's scale | bias << 16 (sg, sh), and
// the B pairs of the same two words (xa, xb; zero for an unused column).
// Word 2c feeds d0, word 2c+1 feeds d1 (two accumulation chains).
__device__ __forceinline__ void mma_segment(float (&d0)[4], float (&d1)[4], uint2 wg, uint2 wh,
                                            uint32_t sg, uint32_t sh, uint4 xa, uint4 xb) {
  uint32_t pg[4], ph[4];
  dequant_word_i4(wg.x, dup_lo(sg), dup_hi(sg), pg);
  dequant_word_i4(wh.x, dup_lo(sh), dup_hi(sh), ph);
  mma_bf16_16816(d0, pg[0], ph[0], pg[1], ph[1], xa.x, xa.y);
  mma_bf16_16816(d0, pg[2], ph[2], pg[3], ph[3], xa.z, xa.w);
  dequant_word_i4(wg.y, dup_lo(sg), dup_hi(sg), pg);
  dequant_word_i4(wh.y, dup_lo(sh), dup_hi(sh), ph);
  mma_bf16_16816(d1, pg[0], ph[0], pg[1], ph[1], xb.x, xb.y);
  mma_bf16_16816(d1, pg[2], ph[2], pg[3], ph[3], xb.z, xb.w);
}

// A natural 8-element bf16 chunk -> the pair layout (e0,e4), (e1,e5),
// (e2,e6), (e3,e7).
__device__ __forceinline__ uint4 to_pairs(const uint4& v) {
  uint4 o;
  o.x = __byte_perm(v.x, v.z, 0x5410);
  o.y = __byte_perm(v.x, v.z, 0x7632);
  o.z = __byte_perm(v.y, v.w, 0x5410);
  o.w = __byte_perm(v.y, v.w, 0x7632);
  return o;
}

// ------------------------------------------------------------- router --
// The first min(8, H/256) 16-byte pieces of lane `lane` of router row e.
struct RouterRow {
  uint4 q[8];
};
__device__ __forceinline__ void ps_router_load(RouterRow& R, const uint16_t* wrow, int H,
                                               int lane) {
  const uint4* wq = reinterpret_cast<const uint4*>(wrow);
  const int nj = H >> 8;
#pragma unroll
  for (int j = 0; j < 8; ++j)
    if (j < nj) R.q[j] = __ldg(wq + 32 * j + lane);
}

// acc + the 8 products of one chunk: x as pairs (e_i, e_i+4), w natural.
__device__ __forceinline__ float fma8_pairs(const uint4& xp, const uint4& wv, float acc) {
  acc = __fmaf_rn(bf_lo(xp.x), bf_lo(wv.x), acc);
  acc = __fmaf_rn(bf_lo(xp.y), bf_hi(wv.x), acc);
  acc = __fmaf_rn(bf_lo(xp.z), bf_lo(wv.y), acc);
  acc = __fmaf_rn(bf_lo(xp.w), bf_hi(wv.y), acc);
  acc = __fmaf_rn(bf_hi(xp.x), bf_lo(wv.z), acc);
  acc = __fmaf_rn(bf_hi(xp.y), bf_hi(wv.z), acc);
  acc = __fmaf_rn(bf_hi(xp.z), bf_lo(wv.w), acc);
  acc = __fmaf_rn(bf_hi(xp.w), bf_hi(wv.w), acc);
  return acc;
}

// Logit of router row wrow with a token's activations (pairs, 16 bytes per
// 8 elements): partial `lane` over elements 8(32j + lane) + i, j then i
// ascending, then an xor butterfly (the order of the prefill router).
__device__ __forceinline__ float ps_router_compute(const RouterRow& R, const uint16_t* wrow, int H,
                                                   const uint4* xt, int lane) {
  const uint4* wq = reinterpret_cast<const uint4*>(wrow);
  const int nj = H >> 8;
  float acc = 0.0f;
#pragma unroll
  for (int j = 0; j < 8; ++j)
    if (j < nj) acc = fma8_pairs(xt[32 * j + lane], R.q[j], acc);
  for (int j = 8; j < nj; ++j) acc = fma8_pairs(xt[32 * j + lane], __ldg(wq + 32 * j + lane), acc);
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xFFFFFFFFu, acc, d));
  return acc;
}

// ------------------------------------------------------------ gate_up --
// One warp's share of a gate_up tile, one batch of at most kSegBatch
// segments: words 2c, 2c+1 of gate row j0+g (wg) and up row I+j0+g (wh);
// the group scale | bias << 16 of segments 2c and 2c+1 of both rows (sg,
// sh), which the other lanes of the row fetch by shuffle.
struct GuBatch {
  uint2 wg[kSegBatch], wh[kSegBatch];
  uint32_t sg[2], sh[2];
};
static_assert(kSegBatch == 8, "the scale / bias of a batch spread over the 4 lanes of a row");

// Loads segments seg0 .. seg0+n-1 (n <= kSegBatch) of rows rg, rh of one
// expert's gate_up matrix (wpr words, gpr groups per row).
__device__ __forceinline__ void gu_batch_load(GuBatch& B, const uint32_t* q, const uint16_t* s,
                                              const uint16_t* b, size_t rg, size_t rh, int wpr,
                                              int gpr, int seg0, int n, int c) {
#pragma unroll
  for (int i = 0; i < kSegBatch; ++i) {
    if (i < n) {
      B.wg[i] = __ldg(reinterpret_cast<const uint2*>(q + rg * wpr + (seg0 + i) * 8 + 2 * c));
      B.wh[i] = __ldg(reinterpret_cast<const uint2*>(q + rh * wpr + (seg0 + i) * 8 + 2 * c));
    }
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int i = 2 * c + h;
    B.sg[h] = B.sh[h] = 0;
    if (i < n) {
      B.sg[h] = (uint32_t)__ldg(s + rg * gpr + seg0 + i) | ((uint32_t)__ldg(b + rg * gpr + seg0 + i) << 16);
      B.sh[h] = (uint32_t)__ldg(s + rh * gpr + seg0 + i) | ((uint32_t)__ldg(b + rh * gpr + seg0 + i) << 16);
    }
  }
}

// ---------------------------------------------------------------- down --
// One down item: output rows 8g..8g+7 of two slots k1, k2 (k2 may be
// absent): tile row g is slot k1's weight row 8g+g, tile row g+8 slot k2's
// same row, over all of I; B column 0 is h of slot k1, column 1 h of k2.
// Lane c keeps the scale | bias << 16 of segments c, c+4, .. of both rows;
// the other lanes of the row fetch them by shuffle.
template <int I>
struct DownUnit {
  static constexpr int kSeg = I / 64;                   // segments per row
  static constexpr int kOwn = kSeg > 4 ? kSeg / 4 : 1;  // segments whose scales a lane keeps
  uint2 wg[kSeg], wh[kSeg];
  uint32_t sg[kOwn], sh[kOwn];
};

// Row rowg of wtg (slot k1) and, if wth, row rowh of wth (slot k2; else
// zero weights).
template <int I>
__device__ __forceinline__ void down_load(DownUnit<I>& D, const moe_w4_weights_t& wtg, size_t rowg,
                                          const moe_w4_weights_t* wth, size_t rowh, int c) {
  constexpr int kSeg = DownUnit<I>::kSeg, kOwn = DownUnit<I>::kOwn;
  const uint32_t* qg = wtg.q_down_dev + rowg * (I / 8);
#pragma unroll
  for (int i = 0; i < kSeg; ++i) D.wg[i] = __ldg(reinterpret_cast<const uint2*>(qg + i * 8 + 2 * c));
#pragma unroll
  for (int o = 0; o < kOwn; ++o) {
    const int i = c + 4 * o;
    D.sg[o] = i < kSeg ? (uint32_t)__ldg(wtg.s_down_dev + rowg * kSeg + i) |
                             ((uint32_t)__ldg(wtg.b_down_dev + rowg * kSeg + i) << 16)
                       : 0u;
  }
  if (wth) {
    const uint32_t* qh = wth->q_down_dev + rowh * (I / 8);
#pragma unroll
    for (int i = 0; i < kSeg; ++i) D.wh[i] = __ldg(reinterpret_cast<const uint2*>(qh + i * 8 + 2 * c));
#pragma unroll
    for (int o = 0; o < kOwn; ++o) {
      const int i = c + 4 * o;
      D.sh[o] = i < kSeg ? (uint32_t)__ldg(wth->s_down_dev + rowh * kSeg + i) |
                               ((uint32_t)__ldg(wth->b_down_dev + rowh * kSeg + i) << 16)
                         : 0u;
    }
  } else {
#pragma unroll
    for (int i = 0; i < kSeg; ++i) D.wh[i] = make_uint2(0u, 0u);
#pragma unroll
    for (int o = 0; o < kOwn; ++o) D.sh[o] = 0u;
  }
}

struct PsShared {
  TopkWarpSmem<kPsMaxE> ts[kPsMaxT];
  int32_t sid[kPsMaxT][32];
  float swt[kPsMaxT][32];
  float xinv[kPsMaxT];
  // gate_up partial sums [group][round parity][slice][column][row]; also
  // the previous layer's y^2 partials during the input phase
  float red[kGuSlices][2][kGuSlices][kPsMaxT][16];
  uint32_t seq;
};

__device__ __forceinline__ void named_bar(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// BLOCK: decoder blocks (PersistArgs::block); a separate instantiation, so
// the stacked chain keeps its own register allocation
template <int I, bool BLOCK>
__global__ void __launch_bounds__(kPsThreads, 1)
    dec_persist_kernel(const __grid_constant__ PersistArgs a) {
  extern __shared__ __align__(128) uint8_t dyn[];
  __shared__ PsShared S;
  const int T = a.T, H = a.H, E = a.E, K = a.K, ns = a.ns, slots = K + ns;
  const int G = gridDim.x, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, c = lane & 3;         // MMA fragment coordinates
  const int nb = H / kPsGroup;                   // row groups (and partials) per token
  const int nud = (T * nb - (int)blockIdx.x + G - 1) / G;  // this block's row groups
  Ctrl* ctrl = a.ctrl;
  // shared memory: activations and h (pair layout), slot results, y
  uint4* xp = reinterpret_cast<uint4*>(dyn);                 // [T][H/8]
  uint4* hp = xp + (size_t)T * (H / 8);                      // [T][slots][I/8]
  float* dsl = reinterpret_cast<float*>(hp + (size_t)T * slots * (I / 8));  // [nud][slots][8]
  uint16_t* yv = reinterpret_cast<uint16_t*>(dsl + (size_t)nud * slots * kPsGroup);
  // decoder blocks: the residual stream h of this layer, pair layout [T][H/8]
  uint4* rp = reinterpret_cast<uint4*>(
      (reinterpret_cast<uintptr_t>(yv + (size_t)nud * kPsGroup) + 15) & ~(uintptr_t)15);
  // programmatic dependent launch: the blocks may be placed while the
  // previous launch runs; nothing before this wait touches global memory
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x == 0) S.seq = *reinterpret_cast<volatile unsigned*>(&ctrl->ps_seq);
  __syncthreads();
  const uint32_t base = S.seq * kPsEpochStride + 1u;
  const int wpr = H >> 3, gpr = H >> 6;
  const int nR = T * E;                       // router units
  const int tiles_tok = K * (I / 8);          // routed gate_up tiles of a token
  const int nRt = T * tiles_tok;
  const int nTiles = nRt + (ns ? I / 8 : 0);  // then the shared expert's (all tokens)
  const int nseg = H / (64 * kGuSlices);      // segments of a gate_up slice
  const int wg_ = warp / kGuSlices, qs = warp % kGuSlices;  // warp group, slice
  const int u0 = blockIdx.x + G * warp;       // the warp's first router unit
  const int npair = (slots + 1) / 2;          // slot pairs of a row group
  const int nit = nud * npair;                // down items of the block

  for (int l = 0; l < a.n_layers; ++l) {
    const moe_layer_weights_t& Lw = a.layer[l];
    const uint32_t ep = base + (uint32_t)l;
    const bool last = l == a.n_layers - 1;
    const uint16_t* wr = static_cast<const uint16_t*>(Lw.w_router_dev);
    // ---------------------------------------------------------- input --
    RouterRow R;
    float rbias = 0.0f;
    if (u0 < nR) {  // before the wait
      ps_router_load(R, wr + (size_t)(u0 % E) * H, H, lane);
      if (Lw.router_bias_dev) rbias = __ldg(Lw.router_bias_dev + u0 % E);
    }
    if (BLOCK) {
      // decoder block: h_l (pair layout) in rp, then x = bf16(g * (h * inv))
      uint32_t* r32 = reinterpret_cast<uint32_t*>(rp);
      float* part_s = &S.red[0][0][0][0][0];
      const int hv = H / 8;
      if (l == 0) {  // h_0: the caller's h, or the tokens' embedding rows
        for (int i = threadIdx.x; i < T * hv; i += kPsThreads) {
          const int t = i / hv, q = i - t * hv;
          const uint4* src = nullptr;
          if (a.tok) {
            const int id = __ldg(a.tok + t);
            if (id >= 0 && id < a.vocab)
              src = reinterpret_cast<const uint4*>(a.embed + (size_t)id * H) + q;
            else if (q == 0 && blockIdx.x == 0)
              set_error(ctrl, MOE_ERR_BAD_INPUT, KID_DECODE, id);
          } else {
            src = reinterpret_cast<const uint4*>(a.x) + i;
          }
          rp[i] = src ? to_pairs(__ldcg(src)) : make_uint4(0u, 0u, 0u, 0u);
        }
        __syncthreads();
        if (warp < T) {  // sum of squares of token warp's h
          float sq = 0.0f;
          for (int i = lane; i < H / 2; i += 32) {
            const uint32_t v = r32[warp * (H / 2) + i];
            sq += bf_lo(v) * bf_lo(v);
            sq += bf_hi(v) * bf_hi(v);
          }
          sq = warp_sum(sq);
          if (lane == 0) S.xinv[warp] = 1.0f / sqrtf(sq / (float)H + 1e-6f);
        }
      } else {  // h_l and its square partials from the previous layer
        poll_block([&](int i) { return a.y_tag + (size_t)(i / 5) * kLine + (i % 5); },
                   T * H / 8 * 5, ep - 1, ctrl, 2, [&](int i, uint32_t v) {
                     const int line = i / 5, w = i - line * 5;
                     if (w < 4)
                       r32[line * 4 + w] = v;
                     else
                       part_s[line] = __uint_as_float(v);
                   });
        __syncthreads();
        if (warp < T) {
          float sq = 0.0f;
          for (int i = lane; i < nb; i += 32) sq += part_s[warp * nb + i];
          sq = warp_sum(sq);
          if (lane == 0) S.xinv[warp] = 1.0f / sqrtf(sq / (float)H + 1e-6f);
        }
      }
      __syncthreads();
      const uint4* gq = reinterpret_cast<const uint4*>(a.gain[l]);
      for (int i = threadIdx.x; i < T * hv; i += kPsThreads) {
        const int t = i / hv;
        const float inv = S.xinv[t];
        const uint4 gv = to_pairs(__ldg(gq + (i - t * hv)));
        const uint4 hq = rp[i];
        uint4 o;
        o.x = pack_bf2(bf_lo(gv.x) * (bf_lo(hq.x) * inv), bf_hi(gv.x) * (bf_hi(hq.x) * inv));
        o.y = pack_bf2(bf_lo(gv.y) * (bf_lo(hq.y) * inv), bf_hi(gv.y) * (bf_hi(hq.y) * inv));
        o.z = pack_bf2(bf_lo(gv.z) * (bf_lo(hq.z) * inv), bf_hi(gv.z) * (bf_hi(hq.z) * inv));
        o.w = pack_bf2(bf_lo(gv.w) * (bf_lo(hq.w) * inv), bf_hi(gv.w) * (bf_hi(hq.w) * inv));
        xp[i] = o;
      }
    } else if (l == 0) {
      const uint4* xg = reinterpret_cast<const uint4*>(a.x);
      for (int i = threadIdx.x; i < T * H / 8; i += kPsThreads)
        xp[i] = to_pairs(__ldcg(xg + i));  // also the buffer x_next may name (written at the end)
    } else {
      // y of the previous layer and its y^2 partials in one poll: line g of
      // token t holds four tagged pairs of y (the activations' layout) and
      // the partial; y is normalised in place once every token's inv is known
      uint32_t* x32 = reinterpret_cast<uint32_t*>(xp);
      float* part_s = &S.red[0][0][0][0][0];  // T*nb <= 1024 partials (red is free here)
      const int nw = T * H / 2;
      poll_block([&](int i) { return a.y_tag + (size_t)(i / 5) * kLine + (i % 5); }, nw / 4 * 5,
                 ep - 1, ctrl, 2, [&](int i, uint32_t v) {
                   const int line = i / 5, w = i - line * 5;
                   if (w < 4)
                     x32[line * 4 + w] = v;
                   else
                     part_s[line] = __uint_as_float(v);
                 });
      __syncthreads();
      if (warp < T) {  // the partials summed as rms_inv_warp sums them
        float sq = 0.0f;
        for (int i = lane; i < nb; i += 32) sq += part_s[warp * nb + i];
        sq = warp_sum(sq);
        if (lane == 0) S.xinv[warp] = 1.0f / sqrtf(sq / (float)H + 1e-6f);
      }
      __syncthreads();
      for (int i = threadIdx.x; i < nw; i += kPsThreads) {
        const float inv = S.xinv[i / (H / 2)];
        const uint32_t v = x32[i];
        x32[i] = pack_bf2(bf_lo(v) * inv, bf_hi(v) * inv);
      }
    }
    __syncthreads();
    // --------------------------------------------------------- router --
    for (int u = u0; u < nR; u += G * kPsWarps) {
      const int t = u / E, e = u - t * E;
      const uint16_t* wrow = wr + (size_t)e * H;
      if (u != u0) {
        ps_router_load(R, wrow, H, lane);
        if (Lw.router_bias_dev) rbias = __ldg(Lw.router_bias_dev + e);
      }
      float lg = ps_router_compute(R, wrow, H, xp + (size_t)t * (H / 8), lane);
      if (Lw.router_bias_dev) lg = __fadd_rn(lg, rbias);
      if (lane == 0) st_tag(a.logits_tag + (size_t)u * kLine, ep, __float_as_uint(lg));
    }
    // ---------------------------------------------------------- top-K --
    if (warp < T) {
      float v[kPsMaxE / 32];
      uint32_t stale = 0;
      const uint64_t* lt = a.logits_tag + (size_t)warp * E * kLine;
#pragma unroll
      for (int i = 0; i < kPsMaxE / 32; ++i) {
        const int e = lane + 32 * i;
        v[i] = 0.0f;
        if (e < E) {
          const uint64_t w = ld_tag(lt + (size_t)e * kLine);
          v[i] = __uint_as_float((uint32_t)w);
          if (tag_of(w) != ep) stale |= 1u << i;
        }
      }
      Waiter wt;
      while (__any_sync(0xFFFFFFFFu, stale != 0u)) {
        if (stale && !wt.keep_going(ctrl, 3)) stale = 0;
#pragma unroll
        for (int i = 0; i < kPsMaxE / 32; ++i) {
          if ((stale >> i) & 1u) {
            const uint64_t w = ld_tag(lt + (size_t)(lane + 32 * i) * kLine);
            v[i] = __uint_as_float((uint32_t)w);
            if (tag_of(w) == ep) stale &= ~(1u << i);
          }
        }
      }
      topk_warp_vals<kPsMaxE, kPsMaxE / 32>(v, E, K, lane, S.ts[warp], S.sid[warp], S.swt[warp]);
    }
    __syncthreads();
    if (last && blockIdx.x == 0) {
      for (int i = threadIdx.x; i < T * K; i += kPsThreads) {
        a.ids[i] = S.sid[i / K][i % K];
        a.w[i] = S.swt[i / K][i % K];
      }
    }
    // down item it = (row group ud, slot pair p): slots 2p and 2p+1
    auto slot_row = [&](int t, int k, int rgp) -> size_t {  // first weight row, by slot
      int e = k < K ? S.sid[t][k] : 0;
      if (e < 0 || e >= E) {  // not produced by the top-K; recorded, expert 0 read instead
        if (c == 0 && g == 0) set_error(ctrl, MOE_ERR_BAD_INPUT, KID_DECODE, e);
        e = 0;
      }
      return (size_t)e * H + (size_t)rgp * kPsGroup;
    };
    auto item_of = [&](int it, int& ud, int& t, int& rgp, int& k1) {
      ud = it / npair;
      k1 = 2 * (it - ud * npair);
      const int un = blockIdx.x + ud * G;
      t = un / nb;
      rgp = un - t * nb;
    };
    auto load_item = [&](DownUnit<I>& D, int it) {
      int ud, t, rgp, k1;
      item_of(it, ud, t, rgp, k1);
      const int k2 = k1 + 1;
      down_load<I>(D, k1 < K ? Lw.experts : Lw.shared, slot_row(t, k1, rgp) + g,
                   k2 < slots ? (k2 < K ? &Lw.experts : &Lw.shared) : nullptr,
                   k2 < slots ? slot_row(t, k2, rgp) + g : 0, c);
    };
    // ------------------------------------------------------- gate_up --
    // the warp's down rows go to L2 behind its first gate_up loads
    bool pref = false;
    auto prefetch_down = [&]() {
      pref = true;
      if (lane != 0) return;
      for (int it = warp; it < nit; it += kPsWarps) {
        int ud, tt, rgp, k1;
        item_of(it, ud, tt, rgp, k1);
        for (int k = k1; k < k1 + 2 && k < slots; ++k) {
          const moe_w4_weights_t& dw = k < K ? Lw.experts : Lw.shared;
          const size_t row0 = slot_row(tt, k, rgp);
          bulk_prefetch_l2(dw.q_down_dev + row0 * (I / 8), kPsGroup * (I / 2));
          bulk_prefetch_l2(dw.s_down_dev + row0 * (I / 64), kPsGroup * (I / 64) * 2);
          bulk_prefetch_l2(dw.b_down_dev + row0 * (I / 64), kPsGroup * (I / 64) * 2);
        }
      }
    };
    for (int i = wg_, r = 0; ; i += kPsWarps / kGuSlices, ++r) {
      const int tau = (int)blockIdx.x + i * G;
      if (tau >= nTiles) break;
      int t = 0, k = K, j0;
      const moe_w4_weights_t* wt;
      size_t e = 0;
      if (tau < nRt) {
        t = tau / tiles_tok;
        const int rem = tau - t * tiles_tok;
        k = rem / (I / 8);
        j0 = 8 * (rem - k * (I / 8));
        int id = S.sid[t][k];
        e = (id < 0 || id >= E) ? 0 : (size_t)id;
        wt = &Lw.experts;
      } else {
        j0 = 8 * (tau - nRt);
        wt = &Lw.shared;
      }
      const uint32_t* q = wt->q_gate_up_dev + e * (size_t)(2 * I) * wpr;
      const uint16_t* s = wt->s_gate_up_dev + e * (size_t)(2 * I) * gpr;
      const uint16_t* b = wt->b_gate_up_dev + e * (size_t)(2 * I) * gpr;
      // B columns: a routed tile's token in column 0; the shared tile's
      // tokens in columns 0..T-1
      const bool routed = tau < nRt;
      const int ncol = routed ? 1 : T;
      const bool bact = g < ncol;
      const uint4* xb = xp + (size_t)(routed ? t : (bact ? g : 0)) * (H / 8);
      float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
      for (int sg0 = 0; sg0 < nseg; sg0 += kSegBatch) {
        const int n = nseg - sg0 < kSegBatch ? nseg - sg0 : kSegBatch;
        const int seg0 = qs * nseg + sg0;
        GuBatch GB;
        gu_batch_load(GB, q, s, b, (size_t)(j0 + g), (size_t)(I + j0 + g), wpr, gpr, seg0, n, c);
        if (!pref) prefetch_down();
#pragma unroll
        for (int i2 = 0; i2 < kSegBatch; ++i2) {
          if (i2 < n) {
            const int w = (seg0 + i2) * 8 + 2 * c;
            const uint4 xa = bact ? xb[w] : make_uint4(0, 0, 0, 0);
            const uint4 xc = bact ? xb[w + 1] : make_uint4(0, 0, 0, 0);
            const int src = (lane & ~3) | (i2 >> 1);  // the row's lane holding segment i2
            const uint32_t sg = __shfl_sync(0xFFFFFFFFu, GB.sg[i2 & 1], src);
            const uint32_t sh = __shfl_sync(0xFFFFFFFFu, GB.sh[i2 & 1], src);
            mma_segment(d0, d1, GB.wg[i2], GB.wh[i2], sg, sh, xa, xc);
          }
        }
      }
      // partial sums of the slice -> shared memory; the group's first warp
      // adds the slices in order and applies SwiGLU
      float(*red)[kPsMaxT][16] = S.red[wg_][r & 1];
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const int col = 2 * c + h2;
        if (col < ncol) {
          red[qs][col][g] = d0[h2] + d1[h2];
          red[qs][col][8 + g] = d0[2 + h2] + d1[2 + h2];
        }
      }
      named_bar(1 + wg_, 32 * kGuSlices);
      if (qs == 0) {
        const int col = lane >> 3, row = lane & 7;
        uint32_t hb = 0;
        if (col < ncol) {
          const float gt = ((red[0][col][row] + red[1][col][row]) + red[2][col][row]) + red[3][col][row];
          const float ut =
              ((red[0][col][8 + row] + red[1][col][8 + row]) + red[2][col][8 + row]) + red[3][col][8 + row];
          hb = f2bf(gt / (1.0f + expf(-gt)) * ut);
        }
        const uint32_t hi = __shfl_down_sync(0xFFFFFFFFu, hb, 4);
        if (col < ncol && row < 4) {
          st_tag(a.h_tag + (size_t)tau * kLine + col * 4 + row, ep, hb | (hi << 16));
        }
      }
      // the next layer's rows of this shared tile go to L2 now, so that its
      // shared tiles do not share the HBM with the routed rows after its top-K
      if (!routed && l + 1 < a.n_layers && lane == 0) {
        const moe_w4_weights_t& nw = a.layer[l + 1].shared;
        if (qs < 2) {
          bulk_prefetch_l2(nw.q_gate_up_dev + (size_t)(qs * I + j0) * wpr, 8u * wpr * 4u);
        } else {
          const uint16_t* sb = qs == 2 ? nw.s_gate_up_dev : nw.b_gate_up_dev;
          bulk_prefetch_l2(sb + (size_t)j0 * gpr, 8u * gpr * 2u);
          bulk_prefetch_l2(sb + (size_t)(I + j0) * gpr, 8u * gpr * 2u);
        }
      }
    }
    if (!pref) prefetch_down();
    // ------------------------------------------------------------ down --
    // h of every slot -> shared memory (pair layout: the tagged words' order)
    // word i of the pair layout: row (t, k) = i / (I/2), pair word m = i % (I/2)
    // of tile word m / 4; routed tiles hold one token, shared tiles all
    poll_block(
        [&](int i) {
          const int row = i / (I / 2), m = i - row * (I / 2), t = row / slots, k = row - t * slots;
          const int tile = k < K ? t * tiles_tok + k * (I / 8) + (m >> 2) : nRt + (m >> 2);
          return a.h_tag + (size_t)tile * kLine + (k < K ? 0 : 4 * t) + (m & 3);
        },
        T * slots * (I / 2), ep, ctrl, 5, [&](int i, uint32_t v) { reinterpret_cast<uint32_t*>(hp)[i] = v; });
    __syncthreads();
    for (int it = warp; it < nit; it += kPsWarps) {
      int ud, t, rgp, k1;
      item_of(it, ud, t, rgp, k1);
      DownUnit<I> D;  // L2 hits: prefetched during the gate_up work
      load_item(D, it);
      // B: lanes of group 0 h of slot k1, group 1 h of slot k1 + 1
      const bool bact = g == 0 || (g == 1 && k1 + 1 < slots);
      const uint4* hb = hp + ((size_t)t * slots + k1 + (g == 1 ? 1 : 0)) * (I / 8);
      float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int i2 = 0; i2 < DownUnit<I>::kSeg; ++i2) {
        const int w = i2 * 8 + 2 * c;
        const uint4 xa = bact ? hb[w] : make_uint4(0, 0, 0, 0);
        const uint4 xc = bact ? hb[w + 1] : make_uint4(0, 0, 0, 0);
        const int src = (lane & ~3) | (i2 & 3);  // the row's lane holding segment i2
        const uint32_t sg = __shfl_sync(0xFFFFFFFFu, D.sg[i2 >> 2], src);
        const uint32_t sh = __shfl_sync(0xFFFFFFFFu, D.sh[i2 >> 2], src);
        mma_segment(d0, d1, D.wg[i2], D.wh[i2], sg, sh, xa, xc);
      }
      // output row 8 rgp + g: slot k1 in column 0 of tile row g, slot k1+1
      // in column 1 of tile row g+8
      if (c == 0) {
        dsl[((size_t)ud * slots + k1) * kPsGroup + g] = d0[0] + d1[0];
        if (k1 + 1 < slots) dsl[((size_t)ud * slots + k1 + 1) * kPsGroup + g] = d0[3] + d1[3];
      }
    }
    __syncthreads();
    // y = sum_k w_k d_k (slot order) + d_shared; one warp per row group, lane
    // r takes row r; the group's y^2 partial sums lanes 0..7 (the others 0)
    for (int ud = warp; ud < nud; ud += kPsWarps) {
      const int un = blockIdx.x + ud * G, t = un / nb, rgp = un - t * nb;
      float ysq = 0.0f;
      uint32_t yb = 0;
      if (lane < kPsGroup) {
        const float* dr = dsl + (size_t)ud * slots * kPsGroup + lane;
        float acc = 0.0f;
        for (int k = 0; k < K; ++k) acc = __fmaf_rn(S.swt[t][k], dr[k * kPsGroup], acc);
        if (ns) acc += dr[K * kPsGroup];
        yb = f2bf(acc);
        if (BLOCK) {  // the residual add: h_{l+1} = bf16(h_l + y_l)
          const uint32_t hw = reinterpret_cast<const uint32_t*>(
              rp)[(size_t)t * (H / 2) + (size_t)rgp * 4 + (lane & 3)];
          yb = f2bf(((lane >> 2) ? bf_hi(hw) : bf_lo(hw)) + __uint_as_float(yb << 16));
        }
        const float yr = __uint_as_float(yb << 16);
        ysq = yr * yr;
        yv[ud * kPsGroup + lane] = (uint16_t)yb;
      }
      ysq = warp_sum(ysq);
      const uint32_t hi = __shfl_down_sync(0xFFFFFFFFu, yb, 4);
      const size_t y0 = (size_t)t * H + (size_t)rgp * kPsGroup;
      if (last) {
        if (lane < kPsGroup) a.y[y0 + lane] = (uint16_t)yb;
      } else if (lane < 4) {  // pairs (y_r, y_r+4) in the activations' layout
        st_tag(a.y_tag + (size_t)un * kLine + lane, ep, yb | (hi << 16));
      }
      if (lane == 4) st_tag(a.y_tag + (size_t)un * kLine + 4, ep, __float_as_uint(ysq));
    }
    __syncthreads();
  }
  // --------------------------------------- next input of the last layer --
  if (a.x_next) {
    const uint32_t ep = base + (uint32_t)(a.n_layers - 1);
    if (warp < T) {
      const float inv = ps_rms_inv(a.y_tag + (size_t)warp * nb * kLine + 4, nb, H, ep, lane, ctrl);
      if (lane == 0) S.xinv[warp] = inv;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < nud * kPsGroup; i += kPsThreads) {
      const int ud = i / kPsGroup, r = i - ud * kPsGroup;
      const int un = blockIdx.x + ud * G, t = un / nb, rgp = un - t * nb;
      const float y = __uint_as_float((uint32_t)yv[i] << 16);
      a.x_next[(size_t)t * H + (size_t)rgp * kPsGroup + r] = (uint16_t)f2bf(y * S.xinv[t]);
    }
  }
  // ------------------------------------------------------------ exit --
  __syncthreads();
  if (threadIdx.x == 0) {
    if (atom_add_acq_rel(&ctrl->ps_exit, 1u) == (uint32_t)G - 1u) {
      ctrl->ps_exit = 0u;
      ctrl->ps_abort = 0u;
      ctrl->ps_seq = S.seq + 1u;
    }
  }
}

constexpr int kMaxDevices = 64;
int g_sms[kMaxDevices];
bool g_attr[kMaxDevices][4];

template <int I, bool BLOCK>
cudaError_t prepare_one(int dev, int optin) {
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, dec_persist_kernel<I, BLOCK>);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(dec_persist_kernel<I, BLOCK>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              optin - (int)fa.sharedSizeBytes);
}

template <int I>
cudaError_t prepare(int dev) {
  if (g_attr[dev][__builtin_ctz(I / 128)]) return cudaSuccess;
  int optin = 0;
  cudaError_t e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  e = prepare_one<I, false>(dev, optin);
  if (e == cudaSuccess) e = prepare_one<I, true>(dev, optin);
  if (e == cudaSuccess) g_attr[dev][__builtin_ctz(I / 128)] = true;
  return e;
}

template <int I>
bool occupancy_ok(size_t smem, bool block) {
  int occ = 0;
  const cudaError_t e =
      block ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, dec_persist_kernel<I, true>,
                                                            kPsThreads, smem)
            : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, dec_persist_kernel<I, false>,
                                                            kPsThreads, smem);
  return e == cudaSuccess && occ >= 1;
}

size_t dyn_smem(int T, int H, int K, int I, int ns, int grid, bool block) {
  const int slots = K + ns, nud = (T * (H / kPsGroup) + grid - 1) / grid;
  size_t b = (size_t)T * H * 2 + (size_t)T * slots * I * 2;
  b += (size_t)nud * slots * kPsGroup * 4 + (size_t)nud * kPsGroup * 2;
  if (block) b = ((b + 15) & ~(size_t)15) + (size_t)T * H * 2;  // the residual stream
  return (b + 127) & ~(size_t)127;
}

}  // namespace

bool persist_supported(int T, int H, int E, int K, int I, int ns) {
  const bool i_ok = I == 128 || I == 256 || I == 512 || I == 1024;
  return T >= 1 && T <= kPsMaxT && E <= kPsMaxE && K + ns <= 33 && i_ok && H % 256 == 0 &&
         T * H <= kPsMaxTH;
}

PersistTags persist_tags(int T, int H, int E, int K, int I, int ns) {
  PersistTags p;
  p.logits = 0;                                                   // a line per router unit
  p.h = p.logits + (size_t)T * E * kLine;                         // a line per gate_up tile
  p.y = p.h + ((size_t)T * K * (I / 8) + (ns ? I / 8 : 0)) * kLine;  // a line per row group
  p.total = p.y + (size_t)T * (H / kPsGroup) * kLine;
  return p;
}

bool persist_config(int T, int H, int E, int K, int I, int ns, int* grid, size_t* smem,
                    bool block) {
  if (!persist_supported(T, H, E, K, I, ns)) return false;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  if (g_sms[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return false;
    g_sms[dev] = n;
  }
  cudaError_t e = I == 128 ? prepare<128>(dev)
                  : I == 256 ? prepare<256>(dev)
                  : I == 512 ? prepare<512>(dev)
                             : prepare<1024>(dev);
  if (e != cudaSuccess) return false;
  // every block owns a row group and, for every token, a routed gate_up tile
  int G = g_sms[dev];
  G = G < T * (H / kPsGroup) ? G : T * (H / kPsGroup);
  G = G < K * (I / 8) ? G : K * (I / 8);
  const size_t s = dyn_smem(T, H, K, I, ns, G, block);
  const bool ok = I == 128 ? occupancy_ok<128>(s, block)
                  : I == 256 ? occupancy_ok<256>(s, block)
                  : I == 512 ? occupancy_ok<512>(s, block)
                             : occupancy_ok<1024>(s, block);
  if (!ok) return false;
  *grid = G;
  *smem = s;
  return true;
}

cudaError_t launch_decode_persist(const PersistArgs& a, int grid, size_t smem,
                                  cudaStream_t stream) {
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kPsThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (a.block) {
    switch (a.I) {
      case 128: return cudaLaunchKernelEx(&cfg, dec_persist_kernel<128, true>, a);
      case 256: return cudaLaunchKernelEx(&cfg, dec_persist_kernel<256, true>, a);
      case 512: return cudaLaunchKernelEx(&cfg, dec_persist_kernel<512, true>, a);
      default: return cudaLaunchKernelEx(&cfg, dec_persist_kernel<1024, true>, a);
    }
  }
  switch (a.I) {
    case 128: return cudaLaunchKernelEx(&cfg, dec_persist_kernel<128, false>, a);
    case 256: return cudaLaunchKernelEx(&cfg, dec_persist_kernel<256, false>, a);
    case 512: return cudaLaunchKernelEx(&cfg, dec_persist_kernel<512, false>, a);
    default: return cudaLaunchKernelEx(&cfg, dec_persist_kernel<1024, false>, a);
  }
}

}  // namespace moe
