// Grouped-query decode attention over a key/value cache kept in fixed-size
// blocks ("Perplexity Open Sources Lily: A Rust + Metal Inference Engine
// for Qwen3.6-35B-A3B on Apple Silicon", section "Decode: Minimize Bytes
// Moved Per Token": the query heads that share a key/value head are packed
// into one threadgroup so each cache row is loaded once, and a fixed-block
// attention layout serves long contexts; section "Three Workload Shapes":
// 16 query heads, 2 key/value heads).
//
// o[t][h] = softmax_j( q[t][h] . k_j / sqrt(D) ) v_j over the positions
// j <= L - T + t, head h reading key/value head h / (n_q / n_kv).
//
// Split along the sequence: CTA (chunk c, group g) takes cb consecutive
// 64-position blocks of head group g, cb chosen so that the CTAs of all
// groups fill the SMs once. All the group's query rows (its n_q / n_kv
// heads times the T tokens, at most 16) form the M = 16 rows of mma.sync
// m16n8k16 tiles, so every key and value row is read once per group. The
// blocks' keys and values stream into shared memory by TMA through a ring
// of six stages (boxes of 64 rows x 64 elements with the 128-byte
// swizzle, so ldmatrix reads are conflict-free; one mbarrier per stage,
// bounded waits); warp w takes positions 16w..16w+15 of each block
// while the next five blocks are in flight: S = Q K^T (fp32), an online
// softmax per row (exp2 of log2e-scaled
// scores), P = bf16(exp2(S - m)) reused in registers as the A operand of
// O += P V. The four warps' (max, sum, O) meet in shared memory at the end
// of the chunk; with one chunk the output is written directly. Otherwise
// the chunks (at most one CTA per SM over all groups, every CTA resident:
// a cooperative launch) write partials, meet at a grid barrier, and merge
// them: each CTA takes 32 output elements of one query row, its four warps
// a quarter of the chunks each. The launch allows programmatic dependent
// launch, so consecutive calls overlap their launch with the previous
// call's tail.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {
constexpr int kAB = 64;       // positions per cache block
constexpr int kAWarps = 4;    // warps per CTA; warp w: positions 16w..16w+15 of a block
constexpr int kAThreads = 32 * kAWarps;
constexpr int kARows = 16;    // query rows of a group (heads x tokens), the MMA's M
constexpr int kAStages = 6;   // cache blocks in shared memory per CTA (one CTA per SM)

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// byte offset of 16-byte chunk ch (elements 8ch..8ch+7) of row p in a
// [64][D] bf16 tile stored as D/64 TMA boxes of 64 rows x 128 bytes with
// the 128-byte swizzle (chunk c of row p at c ^ (p % 8))
template <int D>
__device__ __forceinline__ uint32_t swz(int p, int ch) {
  return (uint32_t)((ch >> 3) * (kAB * 128) + p * 128 + (((ch & 7) ^ (p & 7)) << 4));
}
}  // namespace

// Partials of chunk c of group g: m (log2 domain) and l per row, then
// O[row][D], fp32, at part + ((g * n_chunks + c) * 16 * (D + 2)).
template <int D>
__global__ void __launch_bounds__(kAThreads)
    attn_split_kernel(const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const uint16_t* __restrict__ q,
                      const int32_t* __restrict__ table,
                      int n_phys, int T, int n_q, int n_kv, int L, int cb, int n_chunks,
                      float* __restrict__ part, uint16_t* __restrict__ o, Ctrl* ctrl) {
  constexpr int kTile = kAB * D * 2;  // bytes of one block's keys (or values)
  constexpr int kKS = D / 16;         // k-steps of Q K^T
  constexpr int kDT = D / 8;          // n-tiles of O
  extern __shared__ __align__(1024) uint8_t sm_raw[];
  __shared__ __align__(8) uint64_t full[kAStages];  // stage landed (TMA bytes)
  __shared__ int s_abort;
  // [kAStages][K | V][kTile], 1024-byte aligned for the swizzle
  const uint32_t sbase = (smem_u32(sm_raw) + 1023u) & ~1023u;
  uint8_t* sm = sm_raw + (sbase - smem_u32(sm_raw));
  const int c = blockIdx.x, g = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, cq = lane & 3;
  const int wq = warp;  // quarter of the block
  const int group = n_q / n_kv, rows = group * T;
  const int nblk = (L + kAB - 1) / kAB;
  const int b0 = c * cb, b1 = min(b0 + cb, nblk);
  // programmatic dependent launch: the next call's CTAs may be placed while
  // this call runs, but nothing before this wait reads or writes global
  // memory (q, the cache and the workspace all come from earlier work)
  pdl_wait();
  pdl_trigger();
  // Q fragments (rows r = t * group + head in group; rows >= rows are zero)
  uint32_t qa[kKS][4];
  {
    const int r0 = gq, r1 = gq + 8;
    const uint16_t* q0 = r0 < rows ? q + ((size_t)(r0 / group) * n_q + g * group + r0 % group) * D : nullptr;
    const uint16_t* q1 = r1 < rows ? q + ((size_t)(r1 / group) * n_q + g * group + r1 % group) * D : nullptr;
#pragma unroll
    for (int ks = 0; ks < kKS; ++ks) {
      const int d = ks * 16 + 2 * cq;
      qa[ks][0] = q0 ? __ldg(reinterpret_cast<const uint32_t*>(q0 + d)) : 0u;
      qa[ks][1] = q1 ? __ldg(reinterpret_cast<const uint32_t*>(q1 + d)) : 0u;
      qa[ks][2] = q0 ? __ldg(reinterpret_cast<const uint32_t*>(q0 + d + 8)) : 0u;
      qa[ks][3] = q1 ? __ldg(reinterpret_cast<const uint32_t*>(q1 + d + 8)) : 0u;
    }
  }
  // the last position each of this lane's two rows may see
  const int lim0 = gq < rows ? L - T + gq / group : -1;
  const int lim1 = gq + 8 < rows ? L - T + (gq + 8) / group : -1;
  const float sl2 = 1.4426950408889634f / sqrtf((float)D);  // log2(e) / sqrt(D)

  const uint32_t fb = smem_u32(&full[0]);
  if (threadIdx.x == 0) {
    for (int i = 0; i < kAStages; ++i) mbar_init(fb + 8u * i, 1);
    s_abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  __syncthreads();
  const uint64_t pol = policy_evict_first();  // the cache is streamed once
  // block b of this group into stage st (thread 0)
  auto issue = [&](int b, int st) {
    int phys = __ldg(table + b);
    if (phys < 0 || phys >= n_phys) {
      set_error(ctrl, MOE_ERR_BAD_INPUT, KID_ATTN, b);
      phys = 0;  // read in bounds; the block's scores are masked below
    }
    const int row0 = (phys * n_kv + g) * kAB;
    const uint32_t sk = sbase + (uint32_t)(st * 2 * kTile), sv = sk + kTile;
    const uint32_t bar = fb + 8u * st;
    mbar_arrive_expect_tx(bar, 2u * kTile);
#pragma unroll
    for (int bx = 0; bx < D / 64; ++bx) {
      tma_load_2d(sk + bx * (kAB * 128), &tm_k, bx * 64, row0, bar, pol);
      tma_load_2d(sv + bx * (kAB * 128), &tm_v, bx * 64, row0, bar, pol);
    }
  };
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.0f, l1 = 0.0f;
  float oacc[kDT][4];
#pragma unroll
  for (int j = 0; j < kDT; ++j) oacc[j][0] = oacc[j][1] = oacc[j][2] = oacc[j][3] = 0.0f;

  // blocks b0 .. b0 + kAStages - 2 first
  if (threadIdx.x == 0)
    for (int i = 0; i < kAStages - 1 && b0 + i < b1; ++i) issue(b0 + i, i);
  int issued = min(kAStages - 1, b1 - b0);  // blocks issued so far (thread 0's count)
  int b = b0;
  for (; b < b1; ++b) {
    // this thread's reads of block b - 1 are ordered before the TMA refill
    // of its stage, which thread 0 issues after the barrier
    fence_proxy_async_smem();
    __syncthreads();
    if (s_abort) break;
    if (b + kAStages - 1 < b1) {
      if (threadIdx.x == 0) issue(b + kAStages - 1, (b - b0 + kAStages - 1) % kAStages);
      ++issued;
    }
    const int st = (b - b0) % kAStages;
    if (!mbar_wait(fb + 8u * st, (uint32_t)((b - b0) / kAStages) & 1u, &s_abort)) {
      // recorded once; every thread leaves at the next barrier
      if (atomicCAS(&s_abort, 0, 1) == 0) set_error(ctrl, MOE_ERR_TIMEOUT, KID_ATTN, b);
      continue;
    }
    const uint32_t sk = sbase + (uint32_t)(st * 2 * kTile), sv = sk + kTile;
    int phys = __ldg(table + b);
    const bool bad = phys < 0 || phys >= n_phys;
    // S = Q K^T for positions 16w .. 16w+15 of block b: n-tiles 0 and 1
    float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    {
      const int mi = lane >> 3, rr = lane & 7;
      const int p = 16 * wq + ((mi & 2) ? 8 : 0) + rr;
#pragma unroll
      for (int ks = 0; ks < kKS; ++ks) {
        uint32_t k0, k1, k2, k3;
        ldsm_x4(sk + swz<D>(p, ks * 2 + (mi & 1)), k0, k1, k2, k3);
        mma16816(s[0], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], k0, k1);
        mma16816(s[1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], k2, k3);
      }
    }
    // scale, mask, online softmax (rows gq and gq + 8 of this lane)
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int pos = b * kAB + 16 * wq + 8 * j + 2 * cq + h;
        s[j][h] = (!bad && pos <= lim0) ? s[j][h] * sl2 : -INFINITY;
        s[j][2 + h] = (!bad && pos <= lim1) ? s[j][2 + h] * sl2 : -INFINITY;
        mx0 = fmaxf(mx0, s[j][h]);
        mx1 = fmaxf(mx1, s[j][2 + h]);
      }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xFFFFFFFFu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xFFFFFFFFu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xFFFFFFFFu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xFFFFFFFFu, mx1, 2));
    const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
    // all masked so far: keep everything at zero (no inf - inf)
    const float u0 = n0 == -INFINITY ? 0.0f : n0, u1 = n1 == -INFINITY ? 0.0f : n1;
    const float f0 = exp2f(m0 - u0), f1 = exp2f(m1 - u1);
    m0 = n0;
    m1 = n1;
    float p[2][4];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      p[j][0] = exp2f(s[j][0] - u0);
      p[j][1] = exp2f(s[j][1] - u0);
      p[j][2] = exp2f(s[j][2] - u1);
      p[j][3] = exp2f(s[j][3] - u1);
    }
    // P as the A operand (k = this warp's 16 positions); the sums take the
    // bf16 values the MMA multiplies
    const uint32_t pa0 = pack_bf2(p[0][0], p[0][1]), pa1 = pack_bf2(p[0][2], p[0][3]);
    const uint32_t pa2 = pack_bf2(p[1][0], p[1][1]), pa3 = pack_bf2(p[1][2], p[1][3]);
    l0 = l0 * f0 + (bf_lo(pa0) + bf_hi(pa0)) + (bf_lo(pa2) + bf_hi(pa2));
    l1 = l1 * f1 + (bf_lo(pa1) + bf_hi(pa1)) + (bf_lo(pa3) + bf_hi(pa3));
    {
      const int mi = lane >> 3, rr = lane & 7;
      const int pv = 16 * wq + ((mi & 1) ? 8 : 0) + rr;
#pragma unroll
      for (int j = 0; j < kDT; j += 2) {
        oacc[j][0] *= f0; oacc[j][1] *= f0; oacc[j][2] *= f1; oacc[j][3] *= f1;
        oacc[j + 1][0] *= f0; oacc[j + 1][1] *= f0; oacc[j + 1][2] *= f1; oacc[j + 1][3] *= f1;
        uint32_t v0, v1, v2, v3;
        ldsm_x4_t(sv + swz<D>(pv, j + (mi >> 1)), v0, v1, v2, v3);
        mma16816(oacc[j], pa0, pa1, pa2, pa3, v0, v1);
        mma16816(oacc[j + 1], pa0, pa1, pa2, pa3, v2, v3);
      }
    }
  }
  __syncthreads();
  if (s_abort) {
    // a wait ran out: wait (again bounded) for the copies that may still be
    // in flight so none lands after the CTA exits, and leave no result
    if (threadIdx.x == 0) {
      volatile int never = 0;
      for (int i = issued > kAStages ? issued - kAStages : 0; i < issued; ++i)
        mbar_wait(fb + 8u * (i % kAStages), (uint32_t)(i / kAStages) & 1u, &never);
    }
    return;
  }
  // row sums over the quad
  l0 += __shfl_xor_sync(0xFFFFFFFFu, l0, 1);
  l0 += __shfl_xor_sync(0xFFFFFFFFu, l0, 2);
  l1 += __shfl_xor_sync(0xFFFFFFFFu, l1, 1);
  l1 += __shfl_xor_sync(0xFFFFFFFFu, l1, 2);
  // the warps' states meet in shared memory (the stages are free now)
  float* wm = reinterpret_cast<float*>(sm);               // [warp][16]
  float* wl = wm + kAWarps * kARows;                      // [warp][16]
  float* wo = wl + kAWarps * kARows;                      // [warp][16][D]
  __syncthreads();
  if (cq == 0) {
    wm[warp * kARows + gq] = m0;
    wm[warp * kARows + gq + 8] = m1;
    wl[warp * kARows + gq] = l0;
    wl[warp * kARows + gq + 8] = l1;
  }
#pragma unroll
  for (int j = 0; j < kDT; ++j) {
    float* r0 = wo + ((size_t)warp * kARows + gq) * D + 8 * j + 2 * cq;
    float* r1 = wo + ((size_t)warp * kARows + gq + 8) * D + 8 * j + 2 * cq;
    r0[0] = oacc[j][0];
    r0[1] = oacc[j][1];
    r1[0] = oacc[j][2];
    r1[1] = oacc[j][3];
  }
  __syncthreads();
  for (int i = threadIdx.x; i < kARows * D; i += kAThreads) {
    const int r = i / D, d = i - r * D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kAWarps; ++w) M = fmaxf(M, wm[w * kARows + r]);
    const float U = M == -INFINITY ? 0.0f : M;
    float Ls = 0.0f, Os = 0.0f;
#pragma unroll
    for (int w = 0; w < kAWarps; ++w) {
      const float f = exp2f(wm[w * kARows + r] - U);
      Ls += wl[w * kARows + r] * f;
      Os += wo[((size_t)w * kARows + r) * D + d] * f;
    }
    if (n_chunks == 1) {
      if (r < rows)
        o[((size_t)(r / group) * n_q + g * group + r % group) * D + d] =
            (uint16_t)f2bf(Ls > 0.0f ? Os / Ls : 0.0f);
    } else {
      float* pc = part + ((size_t)g * n_chunks + c) * kARows * (D + 2);
      if (d == 0) {
        pc[r] = M;
        pc[kARows + r] = Ls;
      }
      pc[2 * kARows + (size_t)r * D + d] = Os;
    }
  }
  if (n_chunks == 1) return;
  // ---- grid barrier: every CTA's partials are written and visible
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    volatile unsigned* gen = &ctrl->attn_gen;
    const unsigned g0 = *gen;
    const unsigned G = gridDim.x * gridDim.y;
    if (atomicAdd(&ctrl->attn_arrive, 1u) == G - 1u) {
      ctrl->attn_arrive = 0u;
      __threadfence();
      atomicAdd(&ctrl->attn_gen, 1u);
    } else {
      const uint64_t t0 = globaltimer_ns();
      while (*gen == g0) {
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
          set_error(ctrl, MOE_ERR_TIMEOUT, KID_ATTN, -1);
          s_abort = 1;
          break;
        }
      }
    }
    __threadfence();
  }
  __syncthreads();
  if (s_abort) return;
  // ---- merge: task = (group, row, 32 elements); warp w takes chunks w, w+4, ..
  // with a running maximum, then warp 0 combines the four in warp order
  float* mm = reinterpret_cast<float*>(sm);  // [warp]: max, sum; then [warp][32] O
  float* ml = mm + kAWarps;
  float* mo = ml + kAWarps;
  const int tasks = n_kv * rows * (D / 32);
  const int cid = blockIdx.y * gridDim.x + blockIdx.x, G = gridDim.x * gridDim.y;
  const size_t stride = (size_t)kARows * (D + 2);
  for (int task = cid; task < tasks; task += G) {
    const int pr = task / (D / 32), dsl = task - pr * (D / 32);
    const int gg = pr / rows, r = pr - gg * rows, d = dsl * 32 + lane;
    const float* pg = part + (size_t)gg * n_chunks * stride;
    float M = -INFINITY, Ls = 0.0f, Os = 0.0f;
#pragma unroll 16  // 16 chunks' loads in flight (8: 2.4% slower at 32K, 24: 26%)
    for (int cc = warp; cc < n_chunks; cc += kAWarps) {
      const float* pc = pg + cc * stride;
      const float mc = __ldcg(pc + r), lc = __ldcg(pc + kARows + r);
      const float oc = __ldcg(pc + 2 * kARows + (size_t)r * D + d);
      const float nM = fmaxf(M, mc);
      const float U = nM == -INFINITY ? 0.0f : nM;
      const float fo = exp2f(M - U), fc = exp2f(mc - U);
      Ls = Ls * fo + lc * fc;
      Os = Os * fo + oc * fc;
      M = nM;
    }
    if (lane == 0) {
      mm[warp] = M;
      ml[warp] = Ls;
    }
    mo[warp * 32 + lane] = Os;
    __syncthreads();
    if (warp == 0) {
      float MM = -INFINITY;
#pragma unroll
      for (int w = 0; w < kAWarps; ++w) MM = fmaxf(MM, mm[w]);
      const float U = MM == -INFINITY ? 0.0f : MM;
      float L = 0.0f, O = 0.0f;
#pragma unroll
      for (int w = 0; w < kAWarps; ++w) {
        const float f = exp2f(mm[w] - U);
        L += ml[w] * f;
        O += mo[w * 32 + lane] * f;
      }
      o[((size_t)(r / group) * n_q + gg * group + r % group) * D + d] =
          (uint16_t)f2bf(L > 0.0f ? O / L : 0.0f);
    }
    __syncthreads();
  }
}

bool attn_supported(const moe_attn_shape_t* s) {
  if (!s) return false;
  if (s->T < 1 || s->T > 2 || s->n_q < 1 || s->n_kv < 1 || s->n_q % s->n_kv) return false;
  if ((s->n_q / s->n_kv) * s->T > kARows) return false;
  if (s->D != 64 && s->D != 128) return false;
  if (s->block != kAB || s->L < s->T || s->L > (1 << 24)) return false;
  return true;
}

size_t attn_smem(int D) {
  const size_t stages = (size_t)kAStages * 2 * kAB * D * 2;
  const size_t merge = (size_t)kAWarps * kARows * (2 + D) * 4;
  return (stages > merge ? stages : merge) + 1024;  // + the alignment of the stages
}

size_t attn_part_floats(const moe_attn_shape_t* s) {
  const size_t nblk = (size_t)(s->L + kAB - 1) / kAB;
  return (size_t)s->n_kv * nblk * kARows * (s->D + 2);
}

cudaError_t launch_attn_decode(const moe_attn_shape_t* s, const CUtensorMap& tm_k,
                               const CUtensorMap& tm_v, const uint16_t* q, const int32_t* table,
                               int n_phys, uint16_t* o, float* part, Ctrl* ctrl, int nsm,
                               cudaStream_t stream) {
  const int nblk = (s->L + kAB - 1) / kAB;
  // chunks of whole blocks, at most one CTA per SM over all groups
  const int per_group = nsm / s->n_kv > 1 ? nsm / s->n_kv : 1;
  const int cb = (nblk + per_group - 1) / per_group;
  const int n_chunks = (nblk + cb - 1) / cb;
  const size_t smem = attn_smem(s->D);
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeCooperative;
  attr[1].val.cooperative = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_chunks, s->n_kv);
  cfg.blockDim = dim3(kAThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = n_chunks > 1 ? 2 : 1;  // the grid barrier needs every CTA resident
  cudaError_t e;
  if (s->D == 64) {
    e = cudaFuncSetAttribute(attn_split_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e == cudaSuccess)
      e = cudaLaunchKernelEx(&cfg, attn_split_kernel<64>, tm_k, tm_v, q, table, n_phys, s->T,
                             s->n_q, s->n_kv, s->L, cb, n_chunks, part, o, ctrl);
  } else {
    e = cudaFuncSetAttribute(attn_split_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e == cudaSuccess)
      e = cudaLaunchKernelEx(&cfg, attn_split_kernel<128>, tm_k, tm_v, q, table, n_phys, s->T,
                             s->n_q, s->n_kv, s->L, cb, n_chunks, part, o, ctrl);
  }
  return e;
}

}  // namespace moe
