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
// tile). Warp roles (16 warps):
//   warp 0       W producer: TMA of packed nibble tiles, 128 rows x 128 B
//                (256 reduction elements) per matrix, 128-byte swizzle
//   warp 1       B producer: the entry's activation rows, 64 elements each,
//                gathered four rows per TMA (tile::gather4, 128-byte swizzle)
//   warp 2       TMEM allocator and MMA issuer (one thread)
//   warps 4..7   epilogue: tcgen05.ld of the fp32 accumulators, released as
//                soon as they are in registers, then SwiGLU (or plain) -> bf16
//   warps 8..15  dequantisation of the nibble tiles into TMEM (tcgen05.st)
// Rings: kNW shared-memory W stages (freed by the dequant warps once read),
// kNB shared-memory B stages and kNA TMEM A sub-stages (freed by the MMAs'
// commits), kNAcc accumulator buffers (freed by the epilogue). Every wait
// is bounded; on a timeout the CTA records MOE_ERR_TIMEOUT, drains what it
// started, frees TMEM and returns. Before exit the MMA thread waits for the
// arrival of every commit it issued.
#include <atomic>

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {
constexpr int kTileM = 128;                // weight rows per tile (MMA M)
constexpr int kTileN = 128;                // most tokens per tile (MMA N)
constexpr int kKW = 256;                   // reduction elements per W stage
constexpr int kKA = 64;                    // reduction elements per A / B sub-stage
constexpr int kSub = kKW / kKA;            // sub-stages per W stage
constexpr int kNW = 4;                     // W stages (shared memory)
constexpr int kNB = 4;                     // B stages (shared memory)
constexpr int kNA = 4;                     // A sub-stages (TMEM)
constexpr int kThreads = 512;
constexpr int kDequantWarps = 8;
constexpr int kEpiWarps = 4;
constexpr int kBStage = kTileN * 128;      // 128 rows x 64 bf16
constexpr int kWMat = kTileM * (kKW / 2);  // 128 rows x 128 B of nibbles

template <bool GATED>
struct Cfg {
  static constexpr int kMats = GATED ? 2 : 1;
  static constexpr int kNAcc = GATED ? 1 : 2;
  static constexpr int kWStage = kMats * kWMat;
  static constexpr int kAccCols = kMats * kTileN;      // one accumulator buffer
  static constexpr int kACols = kMats * (kKA / 2);     // 2 bf16 per 32-bit column
  static constexpr int kABase = kNAcc * kAccCols;
  static constexpr int kTmemCols = 512;
  static constexpr int kSmemW = 0;
  static constexpr int kSmemB = kNW * kWStage;
  static constexpr int kSmemBar = kSmemB + kNB * kBStage;
  static constexpr int kSmemBytes = kSmemBar + 512 + 1024;
  static_assert(kABase + kNA * kACols <= kTmemCols, "TMEM budget");
};

// barrier slots
__host__ __device__ constexpr int b_wfull(int s) { return s; }
__host__ __device__ constexpr int b_wfree(int s) { return kNW + s; }
__host__ __device__ constexpr int b_bfull(int s) { return 2 * kNW + s; }
__host__ __device__ constexpr int b_bfree(int s) { return 2 * kNW + kNB + s; }
__host__ __device__ constexpr int b_afull(int a) { return 2 * kNW + 2 * kNB + a; }
__host__ __device__ constexpr int b_aempty(int a) { return 2 * kNW + 2 * kNB + kNA + a; }
__host__ __device__ constexpr int b_accfull(int i) { return 2 * kNW + 2 * kNB + 2 * kNA + i; }
__host__ __device__ constexpr int b_accempty(int i) { return 2 * kNW + 2 * kNB + 2 * kNA + 2 + i; }
constexpr int kNumBars = 2 * kNW + 2 * kNB + 2 * kNA + 4;
static_assert(kNumBars * 8 + 8 <= 512, "barrier area");

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}
// bf16 scales (or biases) of groups g0..g0+3 of one weight row (the row has
// kgroups groups, an even number); groups past the row end read as 0.
__device__ __forceinline__ uint2 load_groups(const uint16_t* row, int g0, int kgroups) {
  if ((kgroups & 3) == 0) return __ldg(reinterpret_cast<const uint2*>(row + g0));
  uint2 v;
  v.x = __ldg(reinterpret_cast<const unsigned int*>(row + g0));
  v.y = (g0 + 2 < kgroups) ? __ldg(reinterpret_cast<const unsigned int*>(row + g0 + 2)) : 0u;
  return v;
}
__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap* tm, int col, int r0,
                                            int r1, int r2, int r3, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
      "l"(tm), "r"(col), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]),
      "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]),
      "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]),
        "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr)
      : "memory");
}

struct Unit {
  int e, row0, nrows, mt;
};
__device__ __forceinline__ Unit load_unit(const FfnArgs& a, int u) {
  const int blk = u / a.mtiles;
  Unit t;
  t.mt = u - blk * a.mtiles;
  t.e = a.block_map[3 * blk];
  t.row0 = a.block_map[3 * blk + 1];
  t.nrows = a.block_map[3 * blk + 2];
  return t;
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
  const uint32_t sW = sbase + C::kSmemW, sB = sbase + C::kSmemB, sBar = sbase + C::kSmemBar;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::kSmemBar + kNumBars * 8);
  volatile int* abort_flag =
      reinterpret_cast<volatile int*>(gbase + C::kSmemBar + kNumBars * 8 + 4);
  auto bar = [&](int i) -> uint32_t { return sBar + 8u * (uint32_t)i; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kNW; ++s) {
      mbar_init(bar(b_wfull(s)), 1);
      mbar_init(bar(b_wfree(s)), kDequantWarps);
    }
    for (int s = 0; s < kNB; ++s) {
      mbar_init(bar(b_bfull(s)), 1);
      mbar_init(bar(b_bfree(s)), 1);
    }
    for (int i = 0; i < kNA; ++i) {
      mbar_init(bar(b_afull(i)), kDequantWarps);
      mbar_init(bar(b_aempty(i)), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(b_accfull(i)), 1);
      mbar_init(bar(b_accempty(i)), kEpiWarps);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_w);
    tma_prefetch_desc(&tm_wsh);
  }
  if (warp == 1 && lane == 0) tma_prefetch_desc(&tm_b);
  if (warp == 2) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int units = min(*a.num_blocks * a.mtiles, a.max_units);
  const int wstages = (a.kdim + kKW - 1) / kKW;  // W stages per unit (the last may be half)
  const int bstages = a.kdim / kKA;              // B / A sub-stages per unit
  bool ok = true;

  if (warp == 0) {
    // -------------------------------------------------------- W producer --
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      uint32_t it = 0;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
        const Unit t = load_unit(a, u);
        const CUtensorMap* tw = (t.e < a.E) ? &tm_w : &tm_wsh;
        const int wrow = (t.e < a.E ? t.e : 0) * a.rows_per_expert + t.mt * kTileM;
        for (int st = 0; st < wstages; ++st, ++it) {
          const int s = it % kNW;
          if (!mbar_wait(bar(b_wfree(s)), ((it / kNW) & 1u) ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar(b_wfull(s)), (uint32_t)C::kWStage);
          tma_load_2d(sW + s * C::kWStage, tw, st * (kKW / 8), wrow, bar(b_wfull(s)), pol);
          if (GATED)
            tma_load_2d(sW + s * C::kWStage + kWMat, tw, st * (kKW / 8), wrow + a.half_rows,
                        bar(b_wfull(s)), pol);
        }
      }
      if (!ok) {
        set_error(a.ctrl, MOE_ERR_TIMEOUT, KID_FFN, 1);
        *abort_flag = 1;
        volatile int never = 0;
        for (uint32_t i = it > (uint32_t)kNW ? it - kNW : 0u; i < it; ++i)
          mbar_wait(bar(b_wfull(i % kNW)), (i / kNW) & 1u, &never);
      }
    }
  } else if (warp == 1) {
    // -------------------------------------------------------- B producer --
    uint32_t it = 0;
    for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
      const Unit t = load_unit(a, u);
      const int ngroups = (t.nrows + 3) >> 2;  // gather4 groups of rows
      int src[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int n = min(4 * lane + j, t.nrows - 1);  // pad with the last row
        const int r = t.row0 + n;
        src[j] = GATED ? (r < a.R ? a.sorted_rows[r] / a.K : r - a.R) : r;
      }
      const uint32_t bytes = (uint32_t)ngroups * 4 * 128;
      for (int st = 0; st < bstages; ++st, ++it) {
        const int s = it % kNB;
        bool good = true;
        if (lane == 0) good = mbar_wait(bar(b_bfree(s)), ((it / kNB) & 1u) ^ 1u, abort_flag);
        if (!__shfl_sync(0xFFFFFFFFu, good ? 1 : 0, 0)) {
          ok = false;
          break;
        }
        if (lane == 0) mbar_arrive_expect_tx(bar(b_bfull(s)), bytes);
        __syncwarp();
        if (lane < ngroups)
          tma_gather4(sB + s * kBStage + lane * 512, &tm_b, st * kKA, src[0], src[1], src[2],
                      src[3], bar(b_bfull(s)));
      }
    }
    if (!ok && lane == 0) {
      set_error(a.ctrl, MOE_ERR_TIMEOUT, KID_FFN, 2);
      *abort_flag = 1;
      volatile int never = 0;
      for (uint32_t i = it > (uint32_t)kNB ? it - kNB : 0u; i < it; ++i)
        mbar_wait(bar(b_bfull(i % kNB)), (i / kNB) & 1u, &never);
    }
  } else if (warp == 2) {
    // -------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      uint32_t it = 0, uc = 0, committed = 0;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x, ++uc) {
        const Unit t = load_unit(a, u);
        const int n_mma = max(16, (t.nrows + 15) & ~15);
        const uint32_t idesc = idesc_bf16(kTileM, n_mma);
        const int buf = uc % C::kNAcc;
        const uint32_t use = uc / C::kNAcc;
        if (!mbar_wait(bar(b_accempty(buf)), (use & 1u) ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t dcol = buf * C::kAccCols;
        for (int st = 0; st < bstages; ++st, ++it) {
          const int s = it % kNB, ai = it % kNA;
          if (!mbar_wait(bar(b_bfull(s)), (it / kNB) & 1u, abort_flag) ||
              !mbar_wait(bar(b_afull(ai)), (it / kNA) & 1u, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t bst = sB + s * kBStage;
#pragma unroll
          for (int kk = 0; kk < kKA / 16; ++kk) {
            const uint64_t bd = smem_desc_sw128(bst + kk * 32);
#pragma unroll
            for (int m = 0; m < C::kMats; ++m) {
              const uint32_t acol = C::kABase + ai * C::kACols + m * (kKA / 2) + kk * 8;
              mma_bf16_ts(tmem + dcol + m * kTileN, tmem + acol, bd, idesc,
                          (st | kk) != 0 ? 1u : 0u);
            }
          }
          mma_commit(bar(b_bfree(s)));
          mma_commit(bar(b_aempty(ai)));
        }
        if (!ok) break;
        mma_commit(bar(b_accfull(buf)));
        ++committed;
      }
      if (!ok) {
        set_error(a.ctrl, MOE_ERR_TIMEOUT, KID_FFN, 3);
        *abort_flag = 1;
      }
      // Tail: each tcgen05.commit above arrives on its barrier asynchronously
      // once the MMAs finish. Wait for the latest phase of every barrier a
      // commit targets, so no arrive can land after this CTA has exited (and
      // all MMAs are complete before TMEM is released).
      volatile int never = 0;
      for (uint32_t i = it > (uint32_t)kNB ? it - kNB : 0u; i < it; ++i)
        mbar_wait(bar(b_bfree(i % kNB)), (i / kNB) & 1u, &never);
      for (uint32_t i = it > (uint32_t)kNA ? it - kNA : 0u; i < it; ++i)
        mbar_wait(bar(b_aempty(i % kNA)), (i / kNA) & 1u, &never);
      for (uint32_t i = committed > (uint32_t)C::kNAcc ? committed - C::kNAcc : 0u;
           i < committed; ++i)
        mbar_wait(bar(b_accfull(i % C::kNAcc)), (i / C::kNAcc) & 1u, &never);
    }
  } else if (warp >= 4 && warp < 8) {
    // ---------------------------------------------------------- epilogue --
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // accumulator row == TMEM lane
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    uint32_t uc = 0;
    for (int u = blockIdx.x; u < units && ok; u += gridDim.x, ++uc) {
      const Unit t = load_unit(a, u);
      const int buf = uc % C::kNAcc;
      const uint32_t use = uc / C::kNAcc;
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(bar(b_accfull(buf)), use & 1u, abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t dbase = tmem + lane_off + buf * C::kAccCols;
      const int nch = (t.nrows + 15) >> 4;  // >= 1
      uint16_t* out = a.out + (size_t)t.row0 * a.out_ld + t.mt * kTileM + r;
      for (int ci = 0; ci < nch; ++ci) {
        uint32_t g[16], uu[16];
        tmem_ld16(dbase + ci * 16, g);
        if (GATED) tmem_ld16(dbase + kTileN + ci * 16, uu);
        tmem_wait_ld();
        if (ci == nch - 1) {  // accumulator fully read: hand it back to the MMA
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(b_accempty(buf)));
        }
        const int nlim = min(16, t.nrows - ci * 16);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          if (i < nlim) {
            float v = __uint_as_float(g[i]);
            if (GATED) v = v / (1.0f + expf(-v)) * __uint_as_float(uu[i]);
            out[(size_t)(ci * 16 + i) * a.out_ld] = (uint16_t)f2bf(v);
          }
        }
      }
    }
    if (!ok && lane == 0) {
      set_error(a.ctrl, MOE_ERR_TIMEOUT, KID_FFN, 4);
      *abort_flag = 1;
    }
  } else if (warp >= 8) {
    // ------------------------------------------------ dequant into TMEM --
    const int d = warp - 8;
    const int quarter = warp & 3;
    const int part = d >> 2;             // GATED: gate/up; else: half of the row slice
    const int r = quarter * 32 + lane;   // tile row == TMEM lane
    const int mat = GATED ? part : 0;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t sw = (uint32_t)(r & 7);
    uint32_t wit = 0, ait = 0;
    for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
      const Unit t = load_unit(a, u);
      const int wr = mat * a.half_rows + t.mt * kTileM + r;
      const size_t goff = (size_t)wr * a.kgroups;
      const uint16_t* sp =
          (t.e < a.E ? a.s_exp + (size_t)t.e * a.rows_per_expert * a.kgroups : a.s_sh) + goff;
      const uint16_t* bp =
          (t.e < a.E ? a.b_exp + (size_t)t.e * a.rows_per_expert * a.kgroups : a.b_sh) + goff;
      uint2 s_next = load_groups(sp, 0, a.kgroups), b_next = load_groups(bp, 0, a.kgroups);
      for (int st = 0; st < wstages && ok; ++st, ++wit) {
        const int s = wit % kNW;
        const uint2 s_cur = s_next, b_cur = b_next;
        if (st + 1 < wstages) {
          s_next = load_groups(sp, 4 * (st + 1), a.kgroups);
          b_next = load_groups(bp, 4 * (st + 1), a.kgroups);
        }
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(bar(b_wfull(s)), (wit / kNW) & 1u, abort_flag))) {
          ok = false;
          break;
        }
        // this thread's 16-byte chunks of its row (128 B = 4 sub-stages x 2);
        // chunk c of row r sits at chunk c ^ (r % 8) (128-byte swizzle)
        uint4 wv[8];
        const uint32_t rowaddr = sW + s * C::kWStage + mat * kWMat + r * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          if (GATED || (c & 1) == part) wv[c] = lds128(rowaddr + 16u * ((uint32_t)c ^ sw));
        }
        // the stage goes back to the TMA producer: order these generic-proxy
        // reads before its async-proxy refill (write-after-read across proxies)
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(b_wfree(s)));
        const int nsub = min(kSub, bstages - st * kSub);
#pragma unroll
        for (int j = 0; j < kSub; ++j) {
          if (j >= nsub) break;
          const int ai = ait % kNA;
          if (!__all_sync(0xFFFFFFFFu,
                          mbar_wait(bar(b_aempty(ai)), ((ait / kNA) & 1u) ^ 1u, abort_flag))) {
            ok = false;
            break;
          }
          ++ait;
          tc_fence_after();
          // group 4*st + j of this row: scale/bias j of the 4 loaded
          const uint32_t sv = (j & 2) ? s_cur.y : s_cur.x;
          const uint32_t bv = (j & 2) ? b_cur.y : b_cur.x;
          const uint32_t s2 = (j & 1) ? dup_hi(sv) : dup_lo(sv);
          const uint32_t b2 = (j & 1) ? dup_hi(bv) : dup_lo(bv);
          const uint32_t acol = C::kABase + ai * C::kACols + mat * (kKA / 2);
          if (GATED) {
            uint32_t v[32];
            dequant_word(wv[2 * j].x, s2, b2, &v[0]);
            dequant_word(wv[2 * j].y, s2, b2, &v[4]);
            dequant_word(wv[2 * j].z, s2, b2, &v[8]);
            dequant_word(wv[2 * j].w, s2, b2, &v[12]);
            dequant_word(wv[2 * j + 1].x, s2, b2, &v[16]);
            dequant_word(wv[2 * j + 1].y, s2, b2, &v[20]);
            dequant_word(wv[2 * j + 1].z, s2, b2, &v[24]);
            dequant_word(wv[2 * j + 1].w, s2, b2, &v[28]);
            tmem_st32(tmem + lane_off + acol, v);
          } else {
            uint32_t v[16];
            const uint4 q = part ? wv[2 * j + 1] : wv[2 * j];
            dequant_word(q.x, s2, b2, &v[0]);
            dequant_word(q.y, s2, b2, &v[4]);
            dequant_word(q.z, s2, b2, &v[8]);
            dequant_word(q.w, s2, b2, &v[12]);
            tmem_st16(tmem + lane_off + acol + part * 16, v);
          }
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(b_afull(ai)));
        }
      }
    }
    if (!ok && lane == 0) {
      set_error(a.ctrl, MOE_ERR_TIMEOUT, KID_FFN, 5);
      *abort_flag = 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
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
int ffn_stage_k() { return kKW; }

}  // namespace moe
