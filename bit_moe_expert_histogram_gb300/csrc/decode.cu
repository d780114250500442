// MoE layer for a few tokens (decode): only the selected experts' packed
// bytes are streamed, with coalesced 16-byte loads, on the CUDA cores.
//
// "Perplexity Open Sources Lily: A Rust + Metal Inference Engine for
// Qwen3.6-35B-A3B on Apple Silicon", section "Decode: Minimize Bytes Moved
// Per Token": batch-1 decode reuses almost no weight, so bytes moved set the
// time; kernel chains are fused so intermediates stay on chip. Three
// launches per layer:
//   dec_route   fixed-order fp32 router logits, one warp per token x expert
//               (the prefill router's order, so the ids are bit-identical)
//   dec_gate_up every block selects the top-K itself from the logits (one
//               warp per token, no serial tail); block 0 publishes ids / w. Warps take 4
//               gate rows and the matching 4 up rows of one slot; SwiGLU -> h
//   dec_down    one block per 8 output columns of a token, one warp per
//               slot: the slot's down rows times its h, then the slots
//               weighted and summed in fp32 in slot order (shared expert
//               weight 1) -> bf16 y; with x_next the last block to finish
//               writes the unit-RMS normalised next-layer input
// A weight is rebuilt to bf16 exactly as in the grouped GEMM (one rounding
// of scale*q + bias); products are exact and sums fp32.
#include "common.cuh"
#include "kernels.h"
#include "topk.cuh"
#include "decode_math.cuh"

namespace moe {

namespace {

constexpr int kGuWarps = 8;                  // gate_up: warps per block
constexpr int kDecCand = 256;                // top-K candidates per token (<= E)
constexpr int kDecMaxE = 256;                // routed experts (8 logits per lane in the top-K)
constexpr int kDownRows = 8;                 // down: output columns per block
constexpr int kDownMaxWarps = 16;            // down: warps per block (slots beyond loop)
constexpr int kGuPairs = 4;  // gate_up: gate rows (and as many up rows) per warp
constexpr int kGuRows = 2 * kGuPairs;
constexpr int kGuPre = 2;    // gate_up: 16-byte chunks per lane and row in one batch of loads

struct SlotW {
  const uint32_t* q;
  const uint16_t* s;
  const uint16_t* b;
  bool ok;
};

// Weights of a slot: routed expert e (k < K; ok = e in [0, E)), else the
// shared expert; rows = weight rows per expert, wpr / gpr = words / groups
// per row.
__device__ __forceinline__ SlotW slot_weights(const DecodeArgs& a, bool gate_up, int k, int e,
                                              int rows, int wpr, int gpr) {
  SlotW r;
  if (k < a.K) {
    r.ok = e >= 0 && e < a.E;
    const size_t ee = r.ok ? (size_t)e : 0;
    r.q = (gate_up ? a.ex.q_gate_up_dev : a.ex.q_down_dev) + ee * rows * wpr;
    r.s = (gate_up ? a.ex.s_gate_up_dev : a.ex.s_down_dev) + ee * rows * gpr;
    r.b = (gate_up ? a.ex.b_gate_up_dev : a.ex.b_down_dev) + ee * rows * gpr;
  } else {
    r.ok = true;
    r.q = gate_up ? a.sh.q_gate_up_dev : a.sh.q_down_dev;
    r.s = gate_up ? a.sh.s_gate_up_dev : a.sh.s_down_dev;
    r.b = gate_up ? a.sh.b_gate_up_dev : a.sh.b_down_dev;
  }
  return r;
}

// One batch of gate_up loads: chunks c = c0 + 32u (u < kGuPre) of the
// warp's kGuRows rows; sb = scale (low half) | bias (high half).
struct GuBatch {
  uint4 q[kGuPre][kGuRows];
  uint32_t sb[kGuPre][kGuRows];
};
__device__ __forceinline__ void gu_load(GuBatch& B, const SlotW& sw, const int* row, int wpr,
                                        int gpr, int c0, int CH) {
#pragma unroll
  for (int u = 0; u < kGuPre; ++u) {
    const int c = c0 + 32 * u;
    if (c < CH) {
#pragma unroll
      for (int r = 0; r < kGuRows; ++r) {
        const size_t rw = (size_t)row[r];
        B.q[u][r] = __ldg(reinterpret_cast<const uint4*>(sw.q + rw * wpr) + c);
        B.sb[u][r] = (uint32_t)__ldg(sw.s + rw * gpr + (c >> 1)) |
                     ((uint32_t)__ldg(sw.b + rw * gpr + (c >> 1)) << 16);
      }
    }
  }
}

// Down loads of one warp: its slot's rows n0 + r, r = s*RPS + lane/CR
// (steps s < kDownRows/RPS, RPS = 32/CR rows per step), chunk c = lane mod
// CR of each row; sb = scale (low half) | bias (high half).
struct DownBatch {
  uint4 q[kDownRows];
  uint32_t sb[kDownRows];
};
__device__ __forceinline__ void down_load(DownBatch& B, const SlotW& sw, int n0, int lane, int CR,
                                          int I) {
  const int wpr = I >> 3, gpr = I >> 6, rps = 32 / CR, c = lane % CR;
#pragma unroll
  for (int st = 0; st < kDownRows; ++st) {
    const int r = st * rps + lane / CR;
    if (st * rps < kDownRows) {
      const size_t rw = (size_t)(n0 + r);
      B.q[st] = __ldg(reinterpret_cast<const uint4*>(sw.q + rw * wpr) + c);
      B.sb[st] = (uint32_t)__ldg(sw.s + rw * gpr + (c >> 1)) |
                 ((uint32_t)__ldg(sw.b + rw * gpr + (c >> 1)) << 16);
    }
  }
}

// L2 prefetch of the down weights of every slot: the packed rows in pieces
// of kPrefetchBytes, spread over the grid's blocks, and the scale / bias
// arrays (one piece each). Called by one thread per block.
constexpr uint32_t kPrefetchBytes = 32768;
__device__ __forceinline__ void prefetch_down_weights(const DecodeArgs& a,
                                                      const int (*sid)[32]) {
  const size_t qbytes = (size_t)a.H * (a.I / 8) * 4, sbytes = (size_t)a.H * (a.I / 64) * 2;
  const int qpieces = (int)((qbytes + kPrefetchBytes - 1) / kPrefetchBytes);
  const int per_region = qpieces + 2;
  const int regions = a.T * a.K + a.ns;  // routed slots of every token, then the shared expert
  for (int p = blockIdx.x; p < regions * per_region; p += gridDim.x) {
    const int rg = p / per_region, piece = p - rg * per_region;
    const moe_w4_weights_t* wt = &a.ex;
    size_t e = 0;
    if (rg < a.T * a.K) {
      const int id = sid[rg / a.K][rg % a.K];
      if (id < 0 || id >= a.E) continue;
      e = (size_t)id;
    } else {
      wt = &a.sh;
    }
    if (piece < qpieces) {
      const size_t off = (size_t)piece * kPrefetchBytes;
      const uint32_t n = (uint32_t)min((size_t)kPrefetchBytes, qbytes - off);
      bulk_prefetch_l2(reinterpret_cast<const uint8_t*>(wt->q_down_dev) + e * qbytes + off, n);
    } else {
      const uint16_t* base = piece == qpieces ? wt->s_down_dev : wt->b_down_dev;
      bulk_prefetch_l2(reinterpret_cast<const uint8_t*>(base) + e * sbytes, (uint32_t)sbytes);
    }
  }
}

}  // namespace

// Dependencies between the three kernels of a layer (all launched with
// programmatic stream serialisation, see pdl_wait / pdl_trigger):
//   dec_route   prefetches its router weights to L2, waits (for the
//               previous layer, or whatever precedes the call), clears the
//               routing-published flag, triggers, writes logits
//   dec_gate_up starts once every router block has passed its wait, so all
//               work before the call is complete: the shared expert's
//               weights load before its wait. After it, each block selects
//               the top-K; block 0 writes ids / w and sets the flag
//               (release); every block then triggers
//   dec_down    starts once every gate_up block has triggered; it acquires
//               the flag, reads ids / w and loads its weights before its
//               wait, and h (from dec_gate_up) after it; it triggers at
//               once (the next router only prefetches before its wait)
// Data written by an earlier kernel of the chain is read through L2
// (ld.global.cg); only the weights use the non-coherent path.

// ---------------------------------------------------------------- router --
// One warp per (token, expert); logit order as in route_logits_kernel.
__global__ void __launch_bounds__(128) dec_route_kernel(DecodeArgs a) {
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  const int T = a.T, E = a.E, H = a.H;
  const bool valid = gw < T * E;
  const int t = valid ? gw / E : 0, e = valid ? gw - t * E : 0;
  if (valid && lane == 0) bulk_prefetch_l2(a.wr + (size_t)e * H, (uint32_t)H * 2);
  pdl_wait();
  if (blockIdx.x == 0 && threadIdx.x == 0) a.ctrl->routed = 0u;
  pdl_trigger();
  if (!valid) return;
  const bool stacked = a.y_prev != nullptr;
  const uint4* xr =
      reinterpret_cast<const uint4*>((stacked ? a.y_prev : a.x) + (size_t)t * H);
  const uint4* wq = reinterpret_cast<const uint4*>(a.wr + (size_t)e * H);
  // the token's input chunks are loaded with the normalisation's partials
  // (one round trip), then normalised
  constexpr int kRouteJ = 8;  // chunks per lane held in registers (H <= 2048)
  const int nj = H >> 8;
  uint4 xin[kRouteJ];
#pragma unroll
  for (int j = 0; j < kRouteJ; ++j)
    if (j < nj) xin[j] = __ldcg(xr + 32 * j + lane);
  const float inv = stacked ? rms_inv_warp(a.part_prev + (size_t)t * a.nb_prev, a.nb_prev, H, lane)
                            : 1.0f;
  float acc = 0.0f;  // partial `lane`: elements 8*(32j+lane)+i, j then i ascending
#pragma unroll
  for (int j = 0; j < kRouteJ + 1; ++j) {
    if (j < kRouteJ && j >= nj) break;
    // j == kRouteJ: the chunks past the registers (H > 2048), in order
    for (int jj = (j < kRouteJ ? j : kRouteJ); jj < (j < kRouteJ ? j + 1 : nj); ++jj) {
      const uint4 xraw = j < kRouteJ ? xin[j] : __ldcg(xr + 32 * jj + lane);
      const uint4 xv = stacked ? norm_chunk(xraw, inv) : xraw;
      const uint4 wv = __ldg(wq + 32 * jj + lane);
      acc = __fmaf_rn(bf_lo(xv.x), bf_lo(wv.x), acc);
      acc = __fmaf_rn(bf_hi(xv.x), bf_hi(wv.x), acc);
      acc = __fmaf_rn(bf_lo(xv.y), bf_lo(wv.y), acc);
      acc = __fmaf_rn(bf_hi(xv.y), bf_hi(wv.y), acc);
      acc = __fmaf_rn(bf_lo(xv.z), bf_lo(wv.z), acc);
      acc = __fmaf_rn(bf_hi(xv.z), bf_hi(wv.z), acc);
      acc = __fmaf_rn(bf_lo(xv.w), bf_lo(wv.w), acc);
      acc = __fmaf_rn(bf_hi(xv.w), bf_hi(wv.w), acc);
    }
  }
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xFFFFFFFFu, acc, d));
  if (lane == 0) a.logits[(size_t)t * E + e] = a.bias ? __fadd_rn(acc, a.bias[e]) : acc;
}

// --------------------------------------------------------------- gate_up --
// Warp gw -> slot (t, k) = gw / (I/kGuPairs), gate rows j..j+kGuPairs-1 and
// the matching up rows I+j.. with j = kGuPairs * (gw mod I/kGuPairs).
// Dynamic smem: the T activation rows.
__global__ void __launch_bounds__(kGuWarps * 32) dec_gate_up_kernel(DecodeArgs a) {
  extern __shared__ __align__(16) uint8_t xs[];
  __shared__ TopkWarpSmem<kDecCand> TS[kDecodeMaxT];
  __shared__ int sid[kDecodeMaxT][32];
  __shared__ float swt[kDecodeMaxT][32];
  __shared__ float xinv[kDecodeMaxT];
  const int T = a.T, H = a.H, I = a.I, K = a.K, slots = K + a.ns;
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * kGuWarps + (threadIdx.x >> 5);
  const int groups = I / kGuPairs;
  const bool valid = gw < T * slots * groups;
  const int sl = valid ? gw / groups : 0, j = valid ? kGuPairs * (gw - sl * groups) : 0;
  const int t = sl / slots, k = sl - t * slots;
  const int wpr = H >> 3, gpr = H >> 6, CH = H >> 5;  // words, groups, chunks per row
  int row[kGuRows];
#pragma unroll
  for (int r = 0; r < kGuPairs; ++r) {
    row[r] = j + r;
    row[kGuPairs + r] = I + j + r;
  }
  GuBatch B;
  SlotW sw = slot_weights(a, true, K, 0, 2 * I, wpr, gpr);  // the shared expert (k == K)
  // the shared expert needs no routing: its weights load before the wait
  if (valid && k == K) gu_load(B, sw, row, wpr, gpr, lane, CH);
  pdl_wait();
  // the activations are fetched now and stored to shared memory after the
  // top-K, so their L2 latency hides behind it
  uint4 xreg[kDecodeMaxT * 2048 / 8 / (kGuWarps * 32)];
  const int xn = T * H / 8;  // 16-byte pieces of all T rows
  const bool stacked = a.y_prev != nullptr;
  const uint16_t* xsrc = stacked ? a.y_prev : a.x;
#pragma unroll
  for (int u = 0; u < (int)(sizeof(xreg) / sizeof(uint4)); ++u) {
    const int i = threadIdx.x + u * kGuWarps * 32;
    if (i < xn) xreg[u] = __ldcg(reinterpret_cast<const uint4*>(xsrc) + i);
  }
  // every block selects the experts itself: warp t takes token t; with a
  // stacked input, warp kGuWarps-1-t forms token t's normalisation meanwhile
  const int warp = threadIdx.x >> 5;
  if (warp < T)
    topk_warp<kDecCand, kDecMaxE / 32>(a.logits + (size_t)warp * a.E, a.E, K, lane, TS[warp],
                                       sid[warp], swt[warp]);
  if (stacked && warp >= kGuWarps - T) {
    const int tt = kGuWarps - 1 - warp;
    const float v = rms_inv_warp(a.part_prev + (size_t)tt * a.nb_prev, a.nb_prev, H, lane);
    if (lane == 0) xinv[tt] = v;
  }
  __syncthreads();
  if (blockIdx.x == 0) {
    for (int i = threadIdx.x; i < T * K; i += blockDim.x) {
      a.ids[i] = sid[i / K][i % K];
      a.w[i] = swt[i / K][i % K];
    }
    __syncthreads();
    if (threadIdx.x == 0) st_release(&a.ctrl->routed, 1u);  // covers the block's writes
  }
  pdl_trigger();
  // the selected experts' down weights go to L2 now, so that dec_down (which
  // cannot share an SM with this kernel) finds them there
  if (threadIdx.x == 0) prefetch_down_weights(a, sid);
  int e = 0;
  if (valid && k < K) {
    e = sid[t][k];
    sw = slot_weights(a, true, k, e, 2 * I, wpr, gpr);
    if (sw.ok) gu_load(B, sw, row, wpr, gpr, lane, CH);
  }
#pragma unroll
  for (int u = 0; u < (int)(sizeof(xreg) / sizeof(uint4)); ++u) {
    const int i = threadIdx.x + u * kGuWarps * 32;
    if (i < xn) {
      const int tt = i / (H / 8), ii = i - tt * (H / 8);
      *reinterpret_cast<uint4*>(xs + (size_t)tt * H * 2 + act_piece_off(ii >> 2, ii & 3)) =
          stacked ? norm_chunk(xreg[u], xinv[tt]) : xreg[u];
    }
  }
  for (int i = threadIdx.x + (int)(sizeof(xreg) / sizeof(uint4)) * kGuWarps * 32; i < xn;
       i += kGuWarps * 32) {  // rows beyond the register budget (T*H > 8192)
    const int tt = i / (H / 8), ii = i - tt * (H / 8);
    const uint4 v = __ldcg(reinterpret_cast<const uint4*>(xsrc) + i);
    *reinterpret_cast<uint4*>(xs + (size_t)tt * H * 2 + act_piece_off(ii >> 2, ii & 3)) =
        stacked ? norm_chunk(v, xinv[tt]) : v;
  }
  __syncthreads();
  if (!valid) return;
  if (!sw.ok) {
    if (lane == 0) {
      set_error(a.ctrl, MOE_ERR_BAD_INPUT, KID_DECODE, e);
      for (int r = 0; r < kGuPairs; ++r) a.h[(size_t)sl * I + j + r] = 0;
    }
    return;
  }
  const uint8_t* xt = xs + (size_t)t * H * 2;
  float acc[kGuRows];
#pragma unroll
  for (int r = 0; r < kGuRows; ++r) acc[r] = 0.0f;
  for (int c0 = lane;;) {
#pragma unroll
    for (int u = 0; u < kGuPre; ++u) {
      const int c = c0 + 32 * u;
      if (c < CH) {
        uint4 xv[4];
        act_load_chunk(xt, c, xv);
#pragma unroll
        for (int r = 0; r < kGuRows; ++r) {
          const uint32_t sb = B.sb[u][r];
          acc[r] = dot32(B.q[u][r], __byte_perm(sb, 0, 0x1010), __byte_perm(sb, 0, 0x3232), xv,
                         acc[r]);
        }
      }
    }
    c0 += 32 * kGuPre;
    if (c0 >= CH) break;
    gu_load(B, sw, row, wpr, gpr, c0, CH);
  }
#pragma unroll
  for (int r = 0; r < kGuRows; ++r) acc[r] = warp_sum(acc[r]);
  if (lane == 0) {
    uint16_t hv[kGuPairs];
#pragma unroll
    for (int r = 0; r < kGuPairs; ++r) {
      const float g = acc[r], u = acc[kGuPairs + r];
      hv[r] = (uint16_t)f2bf(g / (1.0f + expf(-g)) * u);
    }
    uint2 o;
    o.x = (uint32_t)hv[0] | ((uint32_t)hv[1] << 16);
    o.y = (uint32_t)hv[2] | ((uint32_t)hv[3] << 16);
    *reinterpret_cast<uint2*>(a.h + (size_t)sl * I + j) = o;
  }
}

// ------------------------------------------------------ down + combine --
// Block (bx, t): output columns n0 = kDownRows*bx .. n0+kDownRows-1 of token
// t. Warp w takes slots k = w, w + nwarps, ..: lane `lane` holds chunk
// c = lane mod CR (CR = I/32 chunks per row) of the slot's h in registers
// and multiplies it with chunk c of the rows it is given (32/CR rows per
// step); the lanes of a row are summed by shuffles, the slots in order
// through shared memory.
// 96 registers: two blocks of nine warps fit one SM's register file (16
// warps of 110 registers would not).
__global__ void __maxnreg__(96) dec_down_kernel(DecodeArgs a) {
  __shared__ int sid[32];
  __shared__ float swt[32];
  __shared__ float dsl[33][kDownRows];  // slot results of the block's columns
  __shared__ float red[kDownMaxWarps + 1];
  __shared__ int flag_ok, last;
  pdl_trigger();
  const int H = a.H, I = a.I, K = a.K, slots = a.K + a.ns;
  const int t = blockIdx.y, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  const int n0 = blockIdx.x * kDownRows;
  const int CR = I >> 5, rps = 32 / CR, c = lane % CR;
  // routing published by dec_gate_up (release / acquire): the selected
  // down weights stream in before the wait
  if (threadIdx.x == 0) {
    bool ok = ld_acquire(&a.ctrl->routed) == 1u;
    if (!ok) {
      const uint64_t t0 = globaltimer_ns();
      while (!(ok = ld_acquire(&a.ctrl->routed) == 1u) && globaltimer_ns() - t0 < 20000000ull) {
      }
    }
    flag_ok = ok;
  }
  __syncthreads();
  const bool early = flag_ok != 0;
  if (early && threadIdx.x < K) {
    sid[threadIdx.x] = __ldcg(a.ids + t * K + threadIdx.x);
    swt[threadIdx.x] = __ldcg(a.w + t * K + threadIdx.x);
  }
  __syncthreads();
  DownBatch B;
  SlotW sw = slot_weights(a, false, warp, warp < K && early ? sid[warp] : 0, H, I >> 3, I >> 6);
  if (early && warp < slots && sw.ok) down_load(B, sw, n0, lane, CR, I);
  pdl_wait();
  if (!early) {  // the flag did not show within the bound: read after the wait
    if (threadIdx.x < K) {
      sid[threadIdx.x] = __ldcg(a.ids + t * K + threadIdx.x);
      swt[threadIdx.x] = __ldcg(a.w + t * K + threadIdx.x);
    }
    __syncthreads();
    sw = slot_weights(a, false, warp, warp < K ? sid[warp] : 0, H, I >> 3, I >> 6);
    if (warp < slots && sw.ok) down_load(B, sw, n0, lane, CR, I);
  }
  for (int k = warp; k < slots; k += nwarps) {
    if (k != warp) {
      sw = slot_weights(a, false, k, k < K ? sid[k] : 0, H, I >> 3, I >> 6);
      if (sw.ok) down_load(B, sw, n0, lane, CR, I);
    }
    uint4 hv[4];
    const uint4* hr = reinterpret_cast<const uint4*>(a.h + ((size_t)t * slots + k) * I) + 4 * c;
#pragma unroll
    for (int v = 0; v < 4; ++v) hv[v] = __ldcg(hr + v);
    float part[kDownRows];
#pragma unroll
    for (int st = 0; st < kDownRows; ++st) {
      part[st] = 0.0f;
      if (st * rps < kDownRows && sw.ok)
        part[st] = dot32(B.q[st], __byte_perm(B.sb[st], 0, 0x1010),
                         __byte_perm(B.sb[st], 0, 0x3232), hv, 0.0f);
    }
    // sum the CR lanes of each row (lanes of a row are consecutive)
#pragma unroll
    for (int st = 0; st < kDownRows; ++st) {
      if (st * rps < kDownRows) {
        for (int d = CR >> 1; d >= 1; d >>= 1) part[st] += __shfl_xor_sync(0xFFFFFFFFu, part[st], d);
        if (c == 0) dsl[k][st * rps + lane / CR] = part[st];
      }
    }
    if (!sw.ok && lane == 0) set_error(a.ctrl, MOE_ERR_BAD_INPUT, KID_DECODE, sid[k]);
  }
  __syncthreads();
  // y = sum_k w_k d_k (slot order) + d_shared, one thread per column
  float ysq = 0.0f;
  if (threadIdx.x < kDownRows) {
    const int r = threadIdx.x;
    float acc = 0.0f;
    for (int k = 0; k < K; ++k) acc = __fmaf_rn(swt[k], dsl[k][r], acc);
    if (a.ns) acc += dsl[K][r];
    const uint32_t yb = f2bf(acc);
    a.y[(size_t)t * H + n0 + r] = (uint16_t)yb;
    const float yr = __uint_as_float(yb << 16);
    ysq = yr * yr;
  }
  if (!a.x_next && !a.has_next) return;
  // unit-RMS normalisation of the bf16 y: block partials of y^2 (for a
  // stacked next layer, which folds the normalisation into its own
  // kernels), and with x_next the last block writes every token's x_next
  if (warp == 0) {
    ysq = warp_sum(ysq);
    __syncwarp();  // orders lanes 0..kDownRows-1's y stores before lane 0's release
    if (lane == 0) {
      a.part[(size_t)t * gridDim.x + blockIdx.x] = ysq;
      // release: this block's y and partial (lanes 0..kDownRows-1 of this
      // warp wrote them); acquire: every other block's, for the last one
      if (a.x_next) last = atom_add_acq_rel(&a.ctrl->ticket2, 1u) == gridDim.x * gridDim.y - 1;
    }
  }
  if (!a.x_next) return;
  __syncthreads();
  if (!last) return;
  const int nb = gridDim.x, nth = blockDim.x;
  for (int tt = 0; tt < a.T; ++tt) {
    // the token's y loads first, then the normalisation (rms_inv_warp's order)
    const uint32_t* yr = reinterpret_cast<const uint32_t*>(a.y + (size_t)tt * H);
    uint32_t* xr = reinterpret_cast<uint32_t*>(a.x_next + (size_t)tt * H);
    uint32_t yv[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = threadIdx.x + u * nth;
      yv[u] = i < (H >> 1) ? __ldcg(yr + i) : 0u;
    }
    if (warp == 0) {
      const float v = rms_inv_warp(a.part + (size_t)tt * nb, nb, H, lane);
      if (lane == 0) red[kDownMaxWarps] = v;
    }
    __syncthreads();
    const float inv = red[kDownMaxWarps];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = threadIdx.x + u * nth;
      if (i < (H >> 1)) xr[i] = pack_bf2(bf_lo(yv[u]) * inv, bf_hi(yv[u]) * inv);
    }
    for (int i = threadIdx.x + 8 * nth; i < (H >> 1); i += nth) {
      const uint32_t v = __ldcg(yr + i);
      xr[i] = pack_bf2(bf_lo(v) * inv, bf_hi(v) * inv);
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) a.ctrl->ticket2 = 0u;
}

bool decode_supported(int T, int H, int E, int K, int I, int ns) {
  // I/32 chunks per down row must divide the 32 lanes (I = 128..1024, power of two)
  const bool i_ok = I >= 128 && I <= 1024 && (I & (I - 1)) == 0;
  return T >= 1 && T <= kDecodeMaxT && E <= kDecMaxE &&
         (size_t)T * H * 2 + kDecodeMaxT * (sizeof(TopkWarpSmem<kDecCand>) + 256) <= 48 * 1024 &&
         i_ok && K + ns <= 33;
}

size_t decode_part_floats(int T, int H) { return (size_t)T * ((H + kDownRows - 1) / kDownRows); }

cudaError_t launch_decode_layer(const DecodeArgs& a, cudaStream_t stream) {
  const int T = a.T, slots = a.K + a.ns;
  cudaError_t err = launch_pdl(dec_route_kernel, dim3((T * a.E + 3) / 4), dim3(128), 0, stream, a);
  if (err != cudaSuccess) return err;
  const int warps = T * slots * (a.I / kGuPairs);
  err = launch_pdl(dec_gate_up_kernel, dim3((warps + kGuWarps - 1) / kGuWarps),
                   dim3(kGuWarps * 32), (size_t)T * a.H * 2, stream, a);
  if (err != cudaSuccess) return err;
  const int nw = slots < kDownMaxWarps ? slots : kDownMaxWarps;
  return launch_pdl(dec_down_kernel, dim3(a.H / kDownRows, T), dim3(nw * 32), 0, stream, a);
}

}  // namespace moe
