// Grouped W4A16 GEMMs of the MoE expert layer on the 5th-generation tensor
// cores (sm_103a): gate_up with a fused SwiGLU epilogue, and down.
//
// "Perplexity Open Sources Lily: A Rust + Metal Inference Engine for
// Qwen3.6-35B-A3B on Apple Silicon", section "Prefill: Keep Weights Packed,
// Keep Routing on the GPU": the tensor units consume bf16, so the 4-bit
// weights are rebuilt one tile at a time inside the grouped GEMM, kept on
// chip and accumulated in FP32; the expanded array never reaches device
// memory. Here the rebuilt tile lives in tensor memory (TMEM) and feeds
// tcgen05.mma as its A operand, so it costs neither shared-memory writes
// nor shared-memory reads.
//
// Swap-AB: the MMA's M (128) runs over weight rows and its N (16..128, a
// multiple of 16) over the tokens of one block-map entry, so an expert with
// 5 rows pads to 16, not to 128.
//
// One persistent CTA per SM walks units u = (block-map entry, 128-row weight
// tile); warp roles:
//   warp 0      TMA producer: packed nibble tiles [128 rows x 64 B] (64-byte
//               swizzle) and the entry's activation rows, one 2 x 128-byte
//               row load each (128-byte swizzle, gathered by row index)
//   warp 1      TMEM allocator and MMA issuer (one thread)
//   warps 2..9  dequantisation into TMEM (tcgen05.st), then the epilogue
//               (tcgen05.ld of the fp32 accumulators -> SwiGLU or plain ->
//               bf16 rows)
// Pipelines: kNS shared-memory stages of kKS reduction elements, kNA TMEM
// stages of the rebuilt A tile. Every wait is bounded; on a timeout the CTA
// records MOE_ERR_TIMEOUT, drains what it started, frees TMEM and returns.
// Before exit the MMA thread waits for the arrival of every commit it issued.
#include <atomic>

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {
constexpr int kTileM = 128;                  // weight rows per tile (MMA M)
constexpr int kTileN = 128;                  // most tokens per tile (MMA N)
constexpr int kKS = 128;                     // reduction elements per stage
constexpr int kNS = 4;                       // shared-memory stages
constexpr int kNA = 2;                       // TMEM stages of the A tile
constexpr int kThreads = 320;
constexpr int kBAtom = kTileN * 128;         // 128 rows x 64 bf16 (128-byte rows)
constexpr int kBStage = 2 * kBAtom;          // kKS = 128 -> two atoms
constexpr int kWMat = kTileM * (kKS / 2);    // 128 rows x 64 B of nibbles

template <bool GATED>
struct Cfg {
  static constexpr int kMats = GATED ? 2 : 1;
  static constexpr int kWStage = kMats * kWMat;
  static constexpr int kAccCols = kMats * kTileN;
  static constexpr int kACols = kMats * (kKS / 2);  // 2 bf16 per 32-bit column
  static constexpr int kTmemCols = GATED ? 512 : 256;
  static constexpr int kSmemW = kNS * kBStage;
  static constexpr int kSmemBar = kSmemW + kNS * kWStage;
  static constexpr int kSmemBytes = kSmemBar + 256 + 1024;
  static_assert(kAccCols + kNA * kACols <= kTmemCols, "TMEM budget");
};

// barrier slots
__host__ __device__ constexpr int b_full(int s) { return s; }
__host__ __device__ constexpr int b_wfree(int s) { return kNS + s; }
__host__ __device__ constexpr int b_bfree(int s) { return 2 * kNS + s; }
__host__ __device__ constexpr int b_afull(int a) { return 3 * kNS + a; }
__host__ __device__ constexpr int b_aempty(int a) { return 3 * kNS + kNA + a; }
constexpr int kBarAccFull = 3 * kNS + 2 * kNA;
constexpr int kBarAccEmpty = kBarAccFull + 1;
constexpr int kNumBars = kBarAccEmpty + 1;
static_assert(kNumBars * 8 + 8 <= 256, "barrier area");

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t ldg_u32(const uint16_t* p) {
  return __ldg(reinterpret_cast<const unsigned int*>(p));
}
}  // namespace

template <bool GATED>
__global__ void __launch_bounds__(kThreads, 1)
    ffn_w4_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_wsh,
                  const __grid_constant__ CUtensorMap tm_b, const FfnArgs a) {
  using C = Cfg<GATED>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (sbase - raw);
  const uint32_t sB = sbase, sW = sbase + C::kSmemW, sBar = sbase + C::kSmemBar;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::kSmemBar + kNumBars * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + C::kSmemBar + kNumBars * 8 + 4);
  auto bar = [&](int i) -> uint32_t { return sBar + 8u * (uint32_t)i; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kNS; ++s) {
      mbar_init(bar(b_full(s)), 1);
      mbar_init(bar(b_wfree(s)), 8);
      mbar_init(bar(b_bfree(s)), 1);
    }
    for (int i = 0; i < kNA; ++i) {
      mbar_init(bar(b_afull(i)), 8);
      mbar_init(bar(b_aempty(i)), 1);
    }
    mbar_init(bar(kBarAccFull), 1);
    mbar_init(bar(kBarAccEmpty), 8);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_w);
    tma_prefetch_desc(&tm_wsh);
    tma_prefetch_desc(&tm_b);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int nblk = *a.num_blocks;
  const int units = min(nblk * a.mtiles, a.max_units);
  bool ok = true;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer --
    const uint64_t pol_w = policy_evict_first();
    const uint64_t pol_b = policy_evict_last();
    uint32_t it = 0;
    for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
      const int blk = u / a.mtiles, mt = u - blk * a.mtiles;
      const int e = a.block_map[3 * blk], row0 = a.block_map[3 * blk + 1];
      const int nrows = a.block_map[3 * blk + 2];
      int src[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int n = lane + 32 * j;
        src[j] = 0;
        if (n < nrows) {
          const int r = row0 + n;
          src[j] = GATED ? (r < a.R ? a.sorted_rows[r] / a.K : r - a.R) : r;
        }
      }
      const CUtensorMap* tw = (e < a.E) ? &tm_w : &tm_wsh;
      const int wrow = (e < a.E ? e : 0) * a.rows_per_expert + mt * kTileM;
      const uint32_t bytes = (uint32_t)C::kWStage + (uint32_t)nrows * (kKS * 2);
      for (int st = 0; st < a.kstages; ++st, ++it) {
        const int s = it % kNS;
        const uint32_t ph = (it / kNS) & 1u;
        bool good = true;
        if (lane == 0)
          good = mbar_wait(bar(b_wfree(s)), ph ^ 1u, abort_flag) &&
                 mbar_wait(bar(b_bfree(s)), ph ^ 1u, abort_flag);
        good = __shfl_sync(0xFFFFFFFFu, good ? 1 : 0, 0) != 0;
        if (!good) {
          ok = false;
          break;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(bar(b_full(s)), bytes);
          tma_load_2d(sW + s * C::kWStage, tw, st * (kKS / 8), wrow, bar(b_full(s)), pol_w);
          if (GATED)
            tma_load_2d(sW + s * C::kWStage + kWMat, tw, st * (kKS / 8), wrow + a.half_rows,
                        bar(b_full(s)), pol_w);
        }
        __syncwarp();
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int n = lane + 32 * j;
          if (n < nrows) {
            const uint32_t dst = sB + s * kBStage + n * 128;
            tma_load_2d(dst, &tm_b, st * kKS, src[j], bar(b_full(s)), pol_b);
            tma_load_2d(dst + kBAtom, &tm_b, st * kKS + 64, src[j], bar(b_full(s)), pol_b);
          }
        }
      }
    }
    if (!ok) {
      if (lane == 0) {
        set_error(a.ctrl, MOE_ERR_TIMEOUT, KID_FFN, 1);
        *abort_flag = 1;
        // drain: the last kNS stages issued may still be in flight
        const uint32_t first = it > (uint32_t)kNS ? it - kNS : 0u;
        for (uint32_t i = first; i < it; ++i) {
          volatile int never = 0;
          mbar_wait(bar(b_full(i % kNS)), (i / kNS) & 1u, &never);
        }
      }
    }
  } else if (warp == 1) {
    // -------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      uint32_t it = 0, ait = 0, uc = 0, nacc = 0;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x, ++uc) {
        const int blk = u / a.mtiles;
        const int nrows = a.block_map[3 * blk + 2];
        const int n_mma = max(16, (nrows + 15) & ~15);
        const uint32_t idesc = idesc_bf16(kTileM, n_mma);
        if (!mbar_wait(bar(kBarAccEmpty), (uc & 1u) ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int st = 0; st < a.kstages; ++st, ++it, ++ait) {
          const int s = it % kNS;
          const uint32_t ph = (it / kNS) & 1u;
          const int ai = ait % kNA;
          const uint32_t aph = (ait / kNA) & 1u;
          if (!mbar_wait(bar(b_full(s)), ph, abort_flag) ||
              !mbar_wait(bar(b_afull(ai)), aph, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t bst = sB + s * kBStage;
#pragma unroll
          for (int kk = 0; kk < kKS / 16; ++kk) {
            const uint64_t bd = smem_desc_sw128(bst + (kk >> 2) * kBAtom + (kk & 3) * 32);
#pragma unroll
            for (int m = 0; m < C::kMats; ++m) {
              const uint32_t acol = C::kAccCols + ai * C::kACols + m * (kKS / 2) + kk * 8;
              mma_bf16_ts(tmem + m * kTileN, tmem + acol, bd, idesc, (st | kk) != 0 ? 1u : 0u);
            }
          }
          mma_commit(bar(b_bfree(s)));
          mma_commit(bar(b_aempty(ai)));
        }
        if (!ok) break;
        mma_commit(bar(kBarAccFull));
        ++nacc;
      }
      if (!ok) {
        set_error(a.ctrl, MOE_ERR_TIMEOUT, KID_FFN, 2);
        *abort_flag = 1;
      }
      // Tail: each tcgen05.commit above arrives on its barrier asynchronously
      // once the MMAs finish. Wait for the latest phase of every barrier a
      // commit targets, so no arrive can land after this CTA has exited (and
      // all MMAs are complete before TMEM is released).
      volatile int never = 0;
      for (uint32_t i = it > (uint32_t)kNS ? it - kNS : 0u; i < it; ++i)
        mbar_wait(bar(b_bfree(i % kNS)), (i / kNS) & 1u, &never);
      for (uint32_t i = ait > (uint32_t)kNA ? ait - kNA : 0u; i < ait; ++i)
        mbar_wait(bar(b_aempty(i % kNA)), (i / kNA) & 1u, &never);
      if (nacc > 0) mbar_wait(bar(kBarAccFull), (nacc - 1) & 1u, &never);
    }
  } else {
    // ------------------------------------------- dequant, then epilogue --
    const int quarter = warp & 3;           // TMEM lanes this warp may touch
    const int half = (warp - 2) >> 2;       // 0: warps 2..5, 1: warps 6..9
    const int r = quarter * 32 + lane;      // tile row == TMEM lane
    const int mat = GATED ? half : 0;
    const int c0 = GATED ? 0 : 2 * half;    // 16-byte chunks of the row's stage slice
    const int c1 = GATED ? 4 : 2 * half + 2;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    uint32_t it = 0, ait = 0, uc = 0;
    for (int u = blockIdx.x; u < units && ok; u += gridDim.x, ++uc) {
      const int blk = u / a.mtiles, mt = u - blk * a.mtiles;
      const int e = a.block_map[3 * blk], row0 = a.block_map[3 * blk + 1];
      const int nrows = a.block_map[3 * blk + 2];
      const int wr = mat * a.half_rows + mt * kTileM + r;
      const size_t goff = (size_t)wr * a.kgroups;
      const uint16_t* sp = (e < a.E ? a.s_exp + (size_t)e * a.rows_per_expert * a.kgroups : a.s_sh) + goff;
      const uint16_t* bp = (e < a.E ? a.b_exp + (size_t)e * a.rows_per_expert * a.kgroups : a.b_sh) + goff;
      uint32_t s_next = ldg_u32(sp), b_next = ldg_u32(bp);
      for (int st = 0; st < a.kstages; ++st, ++it, ++ait) {
        const int s = it % kNS;
        const uint32_t ph = (it / kNS) & 1u;
        const int ai = ait % kNA;
        const uint32_t aph = (ait / kNA) & 1u;
        const uint32_t s_cur = s_next, b_cur = b_next;
        if (st + 1 < a.kstages) {
          s_next = ldg_u32(sp + 2 * (st + 1));
          b_next = ldg_u32(bp + 2 * (st + 1));
        }
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(bar(b_full(s)), ph, abort_flag))) {
          ok = false;
          break;
        }
        uint4 wv[4];
        const uint32_t rowaddr = sW + s * C::kWStage + mat * kWMat + r * (kKS / 2);
#pragma unroll
        for (int c = 0; c < 4; ++c)
          if (c >= c0 && c < c1) wv[c] = lds128(rowaddr + 16u * (uint32_t)(c ^ ((r >> 1) & 3)));
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(b_wfree(s)));
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(bar(b_aempty(ai)), aph ^ 1u, abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t abase = tmem + lane_off + C::kAccCols + ai * C::kACols + mat * (kKS / 2);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          if (c >= c0 && c < c1) {
            const uint32_t sc = (c < 2) ? dup_lo(s_cur) : dup_hi(s_cur);
            const uint32_t bc = (c < 2) ? dup_lo(b_cur) : dup_hi(b_cur);
            uint32_t v[16];
            dequant_word(wv[c].x, sc, bc, &v[0]);
            dequant_word(wv[c].y, sc, bc, &v[4]);
            dequant_word(wv[c].z, sc, bc, &v[8]);
            dequant_word(wv[c].w, sc, bc, &v[12]);
            tmem_st16(abase + c * 16, v);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(b_afull(ai)));
      }
      if (!ok) break;
      // epilogue: fp32 accumulators -> bf16 rows
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(bar(kBarAccFull), uc & 1u, abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int nch = (nrows + 7) >> 3;
      const int col = mt * kTileM + r;
      for (int ci = half; ci < nch; ci += 2) {
        uint32_t g[8];
        tmem_ld8(tmem + lane_off + ci * 8, g);
        if (GATED) {
          uint32_t uu[8];
          tmem_ld8(tmem + lane_off + kTileN + ci * 8, uu);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int n = ci * 8 + i;
            if (n < nrows) {
              const float gf = __uint_as_float(g[i]), uf = __uint_as_float(uu[i]);
              const float hv = gf / (1.0f + expf(-gf)) * uf;
              a.out[(size_t)(row0 + n) * a.out_ld + col] = (uint16_t)f2bf(hv);
            }
          }
        } else {
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int n = ci * 8 + i;
            if (n < nrows)
              a.out[(size_t)(row0 + n) * a.out_ld + col] = (uint16_t)f2bf(__uint_as_float(g[i]));
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarAccEmpty));
    }
    if (!ok && lane == 0) {
      set_error(a.ctrl, MOE_ERR_TIMEOUT, KID_FFN, 3);
      *abort_flag = 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <bool GATED>
static cudaError_t launch_one(const CUtensorMap& tw, const CUtensorMap& twsh, const CUtensorMap& tb,
                              const FfnArgs& a, int grid, cudaStream_t stream) {
  using C = Cfg<GATED>;
  // the dynamic shared-memory opt-in is per device: set it once for each
  static std::atomic<unsigned long long> configured{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(configured.load() & bit)) {
    e = cudaFuncSetAttribute(ffn_w4_kernel<GATED>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::kSmemBytes);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit);
  }
  ffn_w4_kernel<GATED><<<grid, kThreads, C::kSmemBytes, stream>>>(tw, twsh, tb, a);
  return cudaGetLastError();
}

cudaError_t launch_ffn_gate_up(const CUtensorMap& tw, const CUtensorMap& twsh,
                               const CUtensorMap& tx, const FfnArgs& a, int grid,
                               cudaStream_t stream) {
  return launch_one<true>(tw, twsh, tx, a, grid, stream);
}
cudaError_t launch_ffn_down(const CUtensorMap& tw, const CUtensorMap& twsh, const CUtensorMap& th,
                            const FfnArgs& a, int grid, cudaStream_t stream) {
  return launch_one<false>(tw, twsh, th, a, grid, stream);
}

int ffn_tile_m() { return kTileM; }
int ffn_max_tile_n() { return kTileN; }
int ffn_stage_k() { return kKS; }

}  // namespace moe
