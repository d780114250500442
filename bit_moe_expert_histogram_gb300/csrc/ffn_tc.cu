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
// A unit is (block-map entry, 128 weight rows) with one accumulator. For
// down these are 128 consecutive rows of the down matrix. For gate_up they
// are 64 gate rows j0..j0+63 and the 64 matching up rows, laid out so that
// each 32-row TMEM lane quarter q holds gate rows j0+16q..j0+16q+15 in its
// lanes 0..15 and the same up rows in lanes 16..31: the SwiGLU epilogue
// pairs lane l with lane l+16 by one warp shuffle. One persistent CTA per SM
// takes units from a device-wide counter, the shared expert's (widest) units
// first; the last CTA to finish resets the counter for the next launch.
// Warp roles (24 warps):
//   warp 0        unit queue and W producer: takes units, decodes their
//                 block-map entry once and publishes it to the CTA through
//                 a small shared-memory queue, prefetches the unit's scales
//                 into L2, and loads the packed nibble tiles by TMA, 128
//                 rows x 128 B (256 reduction elements), 128-byte swizzle
//                 (gate_up: four boxes of 16 gate + 16 up rows)
//   warp 1        B producer: the entry's activation rows, consecutive in
//                 the plan-ordered operand (x gathered by gather_x_kernel,
//                 or h), loaded as TMA tiles of 64 rows x 64 elements
//                 (128-byte swizzle; a short entry loads whole boxes, the
//                 rows past it are never read back)
//   warp 2        TMEM allocator and MMA issuer (one thread)
//   warps 4..7    epilogue: tcgen05.ld of the fp32 accumulator, then SwiGLU
//                 (or plain) -> bf16 stores
//   warps 8..23   dequantisation of the nibble tiles into TMEM (tcgen05.st):
//                 warp 8 + 4g + q rebuilds 64 reduction elements (group g of
//                 every slot) of the 32 rows in lane quarter q. Each
//                 packed word is rebuilt as the pairs (i, i+4), the cheapest
//                 nibble placement, so along the reduction every group of 8
//                 elements sits in the order 0,4,1,5,2,6,3,7; the
//                 activations are stored in the same order (gather_x_kernel
//                 for x, the gate_up epilogue for h), which leaves each dot
//                 product's terms unchanged
// Rings: kNW shared-memory W stages (freed by the dequant warps once read,
// behind a proxy fence); kNS slots of kKS reduction elements, each a
// shared-memory B stage plus a TMEM A stage, filled under one barrier (the
// dequant warps' arrivals and the B tiles' bytes) and freed together by one
// MMA commit, 16 MMAs per handshake (runs of 16 fresh A tiles keep the
// tensor pipe busier than runs of 8); two accumulators, so the MMA moves on to the next unit while
// the epilogue drains the last one. Every wait is bounded; on a timeout the
// CTA records MOE_ERR_TIMEOUT, drains what it started, frees TMEM and
// returns. Before exit the MMA thread waits for the arrival of every commit
// it issued; if that wait itself runs out, the tensor pipe has stopped, and
// the CTA records MOE_ERR_TIMEOUT and leaves its TMEM columns allocated
// rather than free columns MMAs may still write.
#include <atomic>

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {
constexpr int kTileM = 128;                // weight rows per unit (MMA M)
constexpr int kTileN = 128;                // most tokens per tile (MMA N)
constexpr int kKW = 256;                   // reduction elements per W stage
constexpr int kKA = 64;                    // reduction elements per 128-byte swizzle atom
constexpr int kBoxRows = 64;               // activation rows per B tensor-map box
constexpr int kKS = 256;                   // reduction elements per slot (16 MMAs per handshake)
constexpr int kSlotsPerW = kKW / kKS;      // slots per W stage
constexpr int kNW = 4;                     // W stages (shared memory)
constexpr int kNS = 2;                     // slots: B (shared memory) + A (TMEM)
constexpr int kNU = 4;                     // unit queue slots
constexpr int kNAcc = 2;                   // accumulators (TMEM)
constexpr int kGateRows = 16;              // gate (and up) rows per lane quarter, gate_up
constexpr int kDequantWarps = 16;
constexpr int kEpiWarps = 4;
constexpr int kUnitReaders = 2 + kEpiWarps + kDequantWarps;  // B producer, MMA, epilogue, dequant
constexpr int kThreads = (8 + kDequantWarps) * 32;
constexpr int kBAtom = kTileN * 128;       // 128 rows x 64 bf16
constexpr int kBStage = (kKS / kKA) * kBAtom;  // one slot of B: four atoms
constexpr int kWStage = kTileM * (kKW / 2);    // 128 rows x 128 B of nibbles
constexpr int kWBoxGate = 2 * kGateRows * (kKW / 2);  // one gate_up box: 16 gate + 16 up rows
constexpr int kACols = kKS / 2;            // A columns per slot (2 bf16 per column)
constexpr int kABase = kNAcc * kTileN;
constexpr int kTmemCols = 512;
constexpr int kSmemW = 0;
constexpr int kSmemB = kNW * kWStage;
constexpr int kSmemBar = kSmemB + kNS * kBStage;
constexpr int kSmemBytes = kSmemBar + 512 + 1024;
static_assert(kABase + kNS * kACols <= kTmemCols, "TMEM budget");
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(4 * kWBoxGate == kWStage, "gate_up boxes fill a W stage");
static_assert(kSlotsPerW == 1, "one slot per W stage");
static_assert(kTileN % kBoxRows == 0, "B boxes tile a B atom");

// barrier slots
__host__ __device__ constexpr int b_wfull(int s) { return s; }
__host__ __device__ constexpr int b_wfree(int s) { return kNW + s; }
__host__ __device__ constexpr int b_sfull(int s) { return 2 * kNW + s; }
__host__ __device__ constexpr int b_sfree(int s) { return 2 * kNW + kNS + s; }
__host__ __device__ constexpr int b_ufull(int q) { return 2 * kNW + 2 * kNS + q; }
__host__ __device__ constexpr int b_uempty(int q) { return 2 * kNW + 2 * kNS + kNU + q; }
__host__ __device__ constexpr int b_accfull(int b) { return 2 * kNW + 2 * kNS + 2 * kNU + b; }
__host__ __device__ constexpr int b_accempty(int b) { return 2 * kNW + 2 * kNS + 2 * kNU + kNAcc + b; }
constexpr int kNumBars = 2 * kNW + 2 * kNS + 2 * kNU + 2 * kNAcc;
constexpr int kRingOff = kNumBars * 8 + 16;  // unit queue after the barrier words
static_assert(kRingOff + 16 * kNU <= 512, "barrier area");

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
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* tm, int c0, int c1,
                                            int c2, uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"(tm), "r"(c0), "r"(c1), "r"(c2), "r"(bar), "l"(policy)
      : "memory");
}
// silu(g) * u in fp32 (the result is rounded to bf16 by the caller)
__device__ __forceinline__ float swiglu(float g, float u) {
  return g * u * __frcp_rn(1.0f + __expf(-g));
}

// One unit as published in the CTA's queue: its index (-1 = no more units)
// and its block-map entry, decoded once by the W producer so that no other
// role waits on a global load when a unit starts.
struct Unit {
  int u, e, row0, nrows;
};

// Next unit from the CTA's queue (4 ints per slot). Every lane of the
// calling warp waits; one arrival per warp frees the slot.
__device__ __forceinline__ bool next_unit(uint32_t ufull, uint32_t uempty, const volatile int* ring,
                                          uint32_t uc, volatile int* abort, int lane, Unit* t) {
  const int q = uc % kNU;
  if (!__all_sync(0xFFFFFFFFu, mbar_wait(ufull + 8u * q, (uc / kNU) & 1u, abort)))
    return false;
  t->u = ring[4 * q];
  t->e = ring[4 * q + 1];
  t->row0 = ring[4 * q + 2];
  t->nrows = ring[4 * q + 3];
  __syncwarp();
  if (lane == 0) mbar_arrive(uempty + 8u * q);
  return true;
}

// The same for a single thread (the MMA issuer), which spins: its waits are
// short and on the critical path.
__device__ __forceinline__ bool next_unit_1(uint32_t ufull, uint32_t uempty,
                                            const volatile int* ring, uint32_t uc,
                                            volatile int* abort, Unit* t) {
  const int q = uc % kNU;
  if (!mbar_wait(ufull + 8u * q, (uc / kNU) & 1u, abort)) return false;
  t->u = ring[4 * q];
  t->e = ring[4 * q + 1];
  t->row0 = ring[4 * q + 2];
  t->nrows = ring[4 * q + 3];
  mbar_arrive(uempty + 8u * q);
  return true;
}

// Weight row (within its expert) of A-tile row r of unit tile mt.
template <bool GATED>
__device__ __forceinline__ int weight_row(const FfnArgs& a, int mt, int r) {
  if (GATED) {
    const int l = r & 31;
    return (l < kGateRows ? 0 : a.half_rows) + mt * (kTileM / 2) + kGateRows * (r >> 5) +
           (l & (kGateRows - 1));
  }
  return mt * kTileM + r;
}
}  // namespace

// GATED (gate_up): unit tile mt covers h columns mt*64 .. mt*64+63 (gate
// rows and up rows I + ..., a.half_rows = I, a 3-D tensor map over
// (word, row of the half, 2*expert + half)); the epilogue writes
// bf16(silu(g) * u). Otherwise (down): rows mt*128 .., written to columns
// mt*128 + r.
template <bool GATED>
__global__ void __launch_bounds__(kThreads, 1)
    ffn_w4_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_wsh,
                  const __grid_constant__ CUtensorMap tm_b, const FfnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (sbase - raw);
  const uint32_t sW = sbase + kSmemW, sB = sbase + kSmemB, sBar = sbase + kSmemBar;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + kSmemBar + kNumBars * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + kSmemBar + kNumBars * 8 + 4);
  volatile int* tmem_keep = abort_flag + 1;  // set when the MMA drain timed out
  volatile int* ring = reinterpret_cast<volatile int*>(gbase + kSmemBar + kRingOff);
  auto bar = [&](int i) -> uint32_t { return sBar + 8u * (uint32_t)i; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kNW; ++s) {
      mbar_init(bar(b_wfull(s)), 1);
      mbar_init(bar(b_wfree(s)), kDequantWarps);
    }
    for (int s = 0; s < kNS; ++s) {
      // slot full: every dequant warp, plus the B producer's expect_tx arrival
      mbar_init(bar(b_sfull(s)), kDequantWarps + 1);
      mbar_init(bar(b_sfree(s)), 1);
    }
    for (int q = 0; q < kNU; ++q) {
      mbar_init(bar(b_ufull(q)), 1);
      mbar_init(bar(b_uempty(q)), kUnitReaders);
    }
    for (int b = 0; b < kNAcc; ++b) {
      mbar_init(bar(b_accfull(b)), 1);
      mbar_init(bar(b_accempty(b)), kEpiWarps);
    }
    *abort_flag = 0;
    *tmem_keep = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_w);
    tma_prefetch_desc(&tm_wsh);
  }
  if (warp == 1 && lane == 0) tma_prefetch_desc(&tm_b);
  if (warp == 2) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();  // everything above reads no global memory
  pdl_trigger();

  const int units = min(*a.num_blocks * a.mtiles, a.max_units);
  const int wstages = (a.kdim + kKW - 1) / kKW;  // W stages per unit (the last may be half)
  const int bstages = wstages;                   // slots per unit (one per W stage)
  const int ksteps_last = ((a.kdim - (bstages - 1) * kKS) / 16);  // MMAs of the last slot
  const uint32_t ufull0 = bar(b_ufull(0)), uempty0 = bar(b_uempty(0));
  bool ok = true;

  if (warp == 0) {
    // ------------------------------------ unit queue + W producer (lane 0) --
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      // shared-expert units (the last block-map entries, the widest) go first
      const int shared_units = min(a.shared_blocks * a.mtiles, units);
      const int routed_units = units - shared_units;
      uint32_t it = 0, uc = 0;
      for (;; ++uc) {
        const int q = uc % kNU;
        if (!mbar_wait(bar(b_uempty(q)), ((uc / kNU) & 1u) ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        const unsigned v = atomicAdd(&a.ctrl->unit_next, 1u);
        const int u = (v >= (unsigned)units) ? -1
                      : ((int)v < shared_units ? routed_units + (int)v : (int)v - shared_units);
        int e = 0, row0 = 0, nrows = 0, mt = 0;
        if (u >= 0) {
          const int blk = u / a.mtiles;
          mt = u - blk * a.mtiles;
          e = a.block_map[3 * blk];
          row0 = a.block_map[3 * blk + 1];
          nrows = a.block_map[3 * blk + 2];
        }
        ring[4 * q] = u;
        ring[4 * q + 1] = e;
        ring[4 * q + 2] = row0;
        ring[4 * q + 3] = nrows;
        mbar_arrive(bar(b_ufull(q)));
        if (u < 0) break;
        const bool routed = e < a.E;
        const CUtensorMap* tw = routed ? &tm_w : &tm_wsh;
        const int ew = routed ? e : 0;
        {
          // the unit's scales and biases into L2 ahead of the dequant
          // warps' loads: gate_up 64 gate + 64 up rows, down 128 rows
          const size_t ebase = (size_t)ew * a.rows_per_expert * a.kgroups;
          const uint16_t* sx = routed ? a.s_exp : a.s_sh;
          const uint16_t* bx = routed ? a.b_exp : a.b_sh;
          const int runs = GATED ? 2 : 1;
          const int run_rows = kTileM / runs;
          const uint32_t bytes = (uint32_t)(run_rows * a.kgroups * 2);
          for (int h = 0; h < runs; ++h) {
            const size_t off = ebase + (size_t)(h * a.half_rows + mt * run_rows) * a.kgroups;
            bulk_prefetch_l2(sx + off, bytes);
            bulk_prefetch_l2(bx + off, bytes);
          }
        }
        for (int st = 0; st < wstages; ++st, ++it) {
          const int s = it % kNW;
          if (!mbar_wait(bar(b_wfree(s)), ((it / kNW) & 1u) ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar(b_wfull(s)), (uint32_t)kWStage);
          if (GATED) {
#pragma unroll
            for (int qq = 0; qq < 4; ++qq)
              tma_load_3d(sW + s * kWStage + qq * kWBoxGate, tw, st * (kKW / 8),
                          mt * (kTileM / 2) + kGateRows * qq, 2 * ew, bar(b_wfull(s)), pol);
          } else {
            tma_load_2d(sW + s * kWStage, tw, st * (kKW / 8), ew * a.rows_per_expert + mt * kTileM,
                        bar(b_wfull(s)), pol);
          }
        }
        if (!ok) break;
      }
      if (!ok) {
        set_error(a.ctrl, MOE_ERR_TIMEOUT, KID_FFN, 1);
        *abort_flag = 1;
        volatile int never = 0;
        for (uint32_t i = it > (uint32_t)kNW ? it - kNW : 0u; i < it; ++i)
          mbar_wait(bar(b_wfull(i % kNW)), (i / kNW) & 1u, &never);
      }
      // this CTA takes no more units; the last CTA to get here resets the counter
      __threadfence();
      if (atomicAdd(&a.ctrl->unit_done, 1u) == gridDim.x - 1) {
        atomicExch(&a.ctrl->unit_next, 0u);
        atomicExch(&a.ctrl->unit_done, 0u);
      }
    }
  } else if (warp == 1) {
    // -------------------------------------------------------- B producer --
    // the entry's other weight tiles read these rows again, but marking them
    // evict-last crowds the weight tiles that heavy experts' other entries
    // re-read: evict-first measured 0.9% faster at the skewed T=2048 layer
    const uint64_t bpol = policy_evict_first();
    uint32_t it = 0, uc = 0;
    Unit t;
    while (ok) {
      if (!next_unit(ufull0, uempty0, ring, uc++, abort_flag, lane, &t)) {
        ok = false;
        break;
      }
      if (t.u < 0) break;
      // the unit's rows are consecutive rows of the plan-ordered operand:
      // boxes of kBoxRows rows, one per lane and 64-wide atom (rows past the
      // unit's are other units' or zero past the end; their columns are
      // never read back). Fewer, larger copies: 64-row boxes took the
      // skewed layer's FFN call from 242 to 225 us against 16-row ones.
      const int nbox = (t.nrows + kBoxRows - 1) / kBoxRows;
      for (int st = 0; st < bstages; ++st, ++it) {
        const int s = it % kNS;
        const int natoms = min(kKS / kKA, (a.kdim - st * kKS) / kKA);  // 64-wide atoms in this slot
        const uint32_t bytes = (uint32_t)nbox * kBoxRows * 128 * natoms;
        bool good = true;
        if (lane == 0) good = mbar_wait(bar(b_sfree(s)), ((it / kNS) & 1u) ^ 1u, abort_flag);
        if (!__shfl_sync(0xFFFFFFFFu, good ? 1 : 0, 0)) {
          ok = false;
          break;
        }
        if (lane == 0) mbar_arrive_expect_tx(bar(b_sfull(s)), bytes);
        __syncwarp();
        if (lane < nbox * natoms) {
          const int bx = lane / natoms, at = lane % natoms;
          tma_load_2d(sB + s * kBStage + at * kBAtom + bx * kBoxRows * 128, &tm_b,
                      st * kKS + at * kKA, t.row0 + kBoxRows * bx, bar(b_sfull(s)), bpol);
        }
      }
    }
    if (!ok && lane == 0) {
      set_error(a.ctrl, MOE_ERR_TIMEOUT, KID_FFN, 2);
      *abort_flag = 1;
      volatile int never = 0;
      for (uint32_t i = it > (uint32_t)kNS ? it - kNS : 0u; i < it; ++i)
        mbar_wait(bar(b_sfull(i % kNS)), (i / kNS) & 1u, &never);
    }
  } else if (warp == 2) {
    // -------------------------------------------------------- MMA issuer --
    uint32_t it = 0, uc = 0, done_units = 0;
    Unit t;
    // B descriptors: slot s, step kk at +32 B inside an atom, next atom
    // every 4 steps; the descriptor's address field is addr >> 4, so an
    // offset adds (offset >> 4) without carrying out of the field
    const uint64_t bdesc0 = smem_desc_sw128(sB);
    // lane 0 alone runs the loop (the other lanes go straight to the end)
    while (ok && lane == 0) {
      if (!next_unit_1(ufull0, uempty0, ring, uc++, abort_flag, &t)) {
        ok = false;
        break;
      }
      if (t.u < 0) break;
      {
        const int n_mma = max(16, (t.nrows + 15) & ~15);
        const uint32_t idesc = idesc_bf16(kTileM, n_mma);
        const uint32_t ab = done_units % kNAcc;
        const uint32_t dacc = tmem + ab * kTileN;
        if (!mbar_wait(bar(b_accempty(ab)), ((done_units / kNAcc) & 1u) ^ 1u, abort_flag)) ok = false;
        tc_fence_after();
        for (int st = 0; st < bstages && ok; ++st, ++it) {
          const int s = it % kNS;
          const uint32_t ph = (it / kNS) & 1u;
          if (!mbar_wait_spin(bar(b_sfull(s)), ph, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t acol = tmem + kABase + s * kACols;
          const uint64_t bd = bdesc0 + (uint64_t)((s * kBStage) >> 4);
          mma_bf16_ts(dacc, acol, bd, idesc, st != 0 ? 1u : 0u);
          // gate_up's reduction (H) is a multiple of kKS: every slot is full
          if (GATED || st + 1 < bstages || ksteps_last == kKS / 16) {
#pragma unroll
            for (int kk = 1; kk < kKS / 16; ++kk)
              mma_bf16_ts_acc(dacc, acol + kk * 8,
                              bd + (uint64_t)((((kk >> 2) * kBAtom) + (kk & 3) * 32) >> 4), idesc);
          } else {
            for (int kk = 1; kk < ksteps_last; ++kk)
              mma_bf16_ts_acc(dacc, acol + kk * 8,
                              bd + (uint64_t)((((kk >> 2) * kBAtom) + (kk & 3) * 32) >> 4), idesc);
          }
          mma_commit(bar(b_sfree(s)));  // frees this slot's B stage and A stage
        }
        if (ok) {
          mma_commit(bar(b_accfull(ab)));
          ++done_units;
        }
      }
    }
    if (lane == 0) {
      if (!ok) {
        set_error(a.ctrl, MOE_ERR_TIMEOUT, KID_FFN, 3);
        *abort_flag = 1;
      }
      // Tail: each tcgen05.commit above arrives on its barrier asynchronously
      // once the MMAs finish. Wait for the latest phase of every barrier a
      // commit targets, so no arrive can land after this CTA has exited (and
      // all MMAs are complete before TMEM is released).
      volatile int never = 0;
      bool drained = true;
      for (uint32_t i = it > (uint32_t)kNS ? it - kNS : 0u; i < it; ++i)
        drained &= mbar_wait(bar(b_sfree(i % kNS)), (i / kNS) & 1u, &never);
      for (uint32_t i = done_units > (uint32_t)kNAcc ? done_units - kNAcc : 0u; i < done_units; ++i)
        drained &= mbar_wait(bar(b_accfull(i % kNAcc)), (i / kNAcc) & 1u, &never);
      if (!drained) {
        // an MMA commit is still pending after the wait limit: the tensor
        // pipe has stopped. Its MMAs may still write TMEM, so the columns
        // are not released (the context is unusable after this anyway).
        set_error(a.ctrl, MOE_ERR_TIMEOUT, KID_FFN, 6);
        *tmem_keep = 1;
      }
    }
  } else if (warp >= 4 && warp < 8) {
    // ---------------------------------------------------------- epilogue --
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // accumulator row == TMEM lane
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    uint32_t uc = 0, done = 0;
    Unit t;
    while (ok) {
      if (!next_unit(ufull0, uempty0, ring, uc++, abort_flag, lane, &t)) {
        ok = false;
        break;
      }
      if (t.u < 0) break;
      const int mt = t.u % a.mtiles;
      const uint32_t ab = done % kNAcc;
      if (!__all_sync(0xFFFFFFFFu,
                      mbar_wait(bar(b_accfull(ab)), (done / kNAcc) & 1u, abort_flag))) {
        ok = false;
        break;
      }
      ++done;
      tc_fence_after();
      const uint32_t dbase = tmem + lane_off + ab * kTileN;
      const int nch = (t.nrows + 15) >> 4;  // >= 1
      if (GATED) {
        // lane l < 16 holds gate row j, lane l + 16 up row j, j = j0 +
        // 16*quarter + l: the pair exchanges halves of each 16-token chunk
        // and lane l writes tokens 0..7, lane l + 16 tokens 8..15
        const int j = mt * (kTileM / 2) + kGateRows * quarter + (lane & (kGateRows - 1));
        const bool lo = lane < kGateRows;
        uint16_t* out = a.out + (size_t)t.row0 * a.out_ld + i4_pos(j);
        for (int ci = 0; ci < nch; ++ci) {
          uint32_t v[16];
          tmem_ld16(dbase + ci * 16, v);
          tmem_wait_ld();
          const int tok0 = ci * 16 + (lo ? 0 : 8);
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint32_t send = lo ? v[8 + k] : v[k];
            const uint32_t got = __shfl_xor_sync(0xFFFFFFFFu, send, kGateRows);
            const float g = __uint_as_float(lo ? v[k] : got);
            const float u = __uint_as_float(lo ? got : v[8 + k]);
            if (tok0 + k < t.nrows)
              out[(size_t)(tok0 + k) * a.out_ld] = (uint16_t)f2bf(swiglu(g, u));
          }
        }
      } else {
        uint16_t* out = a.out + (size_t)t.row0 * a.out_ld + mt * kTileM + r;
        for (int ci = 0; ci < nch; ++ci) {
          uint32_t v[16];
          tmem_ld16(dbase + ci * 16, v);
          tmem_wait_ld();
          const int nlim = min(16, t.nrows - ci * 16);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if (i < nlim) out[(size_t)(ci * 16 + i) * a.out_ld] = (uint16_t)f2bf(__uint_as_float(v[i]));
        }
      }
      // accumulator fully read: hand it back to the MMA
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(b_accempty(ab)));
    }
    if (!ok && lane == 0) {
      set_error(a.ctrl, MOE_ERR_TIMEOUT, KID_FFN, 4);
      *abort_flag = 1;
    }
  } else if (warp >= 8) {
    // ------------------------------------------------ dequant into TMEM --
    const int d = warp - 8;              // 0..15
    const int quarter = warp & 3;        // TMEM lanes this warp may touch
    const int g4 = d >> 2;               // which 32 elements of every slot
    const int r = quarter * 32 + lane;   // tile row == TMEM lane
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t sw = (uint32_t)(r & 7);
    uint32_t wit = 0, ait = 0, uc = 0;
    // this thread's scale / bias row of a unit
    auto group_rows = [&](const Unit& t, const uint16_t** sp, const uint16_t** bp) {
      const int wr = weight_row<GATED>(a, t.u % a.mtiles, r);
      const size_t goff = (size_t)wr * a.kgroups;
      const size_t ebase = t.e < a.E ? (size_t)t.e * a.rows_per_expert * a.kgroups : 0;
      *sp = (t.e < a.E ? a.s_exp : a.s_sh) + ebase + goff;
      *bp = (t.e < a.E ? a.b_exp : a.b_sh) + ebase + goff;
    };
    Unit t;
    if (!next_unit(ufull0, uempty0, ring, uc++, abort_flag, lane, &t)) ok = false;
    uint2 s_next = make_uint2(0u, 0u), b_next = make_uint2(0u, 0u);
    if (ok && t.u >= 0) {
      const uint16_t *sp, *bp;
      group_rows(t, &sp, &bp);
      s_next = load_groups(sp, 0, a.kgroups);
      b_next = load_groups(bp, 0, a.kgroups);
    }
    while (ok && t.u >= 0) {
      const uint16_t *sp, *bp;
      group_rows(t, &sp, &bp);
      Unit nt;
      nt.u = -1;
      for (int st = 0; st < wstages && ok; ++st, ++wit) {
        const int s = wit % kNW;
        const uint2 s_cur = s_next, b_cur = b_next;
        if (st + 1 < wstages) {
          s_next = load_groups(sp, 4 * (st + 1), a.kgroups);
          b_next = load_groups(bp, 4 * (st + 1), a.kgroups);
        } else {
          // last stage of the unit: take the next unit now and start the
          // loads of its first scales, so they land while this stage runs
          if (!next_unit(ufull0, uempty0, ring, uc++, abort_flag, lane, &nt)) {
            ok = false;
            break;
          }
          if (nt.u >= 0) {
            const uint16_t *sp2, *bp2;
            group_rows(nt, &sp2, &bp2);
            s_next = load_groups(sp2, 0, a.kgroups);
            b_next = load_groups(bp2, 0, a.kgroups);
          }
        }
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(bar(b_wfull(s)), (wit / kNW) & 1u, abort_flag))) {
          ok = false;
          break;
        }
        // this thread's 8 words are 16-byte chunks 2*g4 and 2*g4 + 1 of its
        // row (64-element group 4*st + g4); chunk c of row r sits at chunk
        // c ^ (r % 8) (128-byte swizzle). In a half last stage only groups
        // 0 and 1 exist: the other warps rebuild the zero-filled words, whose
        // columns the MMA never reads.
        const uint32_t rowaddr = sW + s * kWStage + r * 128;
        const uint4 w0 = lds128(rowaddr + 16u * ((uint32_t)(2 * g4) ^ sw));
        const uint4 w1 = lds128(rowaddr + 16u * ((uint32_t)(2 * g4 + 1) ^ sw));
        // the stage goes back to the TMA producer: order these generic-proxy
        // reads before its async-proxy refill (write-after-read across proxies)
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(b_wfree(s)));
        // rebuild into registers first: only the TMEM stores wait for the
        // slot, so a freed slot refills in the time of two stores
        const uint32_t sv = (g4 & 2) ? s_cur.y : s_cur.x;
        const uint32_t bv = (g4 & 2) ? b_cur.y : b_cur.x;
        const uint32_t s2 = (g4 & 1) ? dup_hi(sv) : dup_lo(sv);
        const uint32_t b2 = (g4 & 1) ? dup_hi(bv) : dup_lo(bv);
        uint32_t v0[16], v1[16];
        dequant_word_i4(w0.x, s2, b2, &v0[0]);
        dequant_word_i4(w0.y, s2, b2, &v0[4]);
        dequant_word_i4(w0.z, s2, b2, &v0[8]);
        dequant_word_i4(w0.w, s2, b2, &v0[12]);
        dequant_word_i4(w1.x, s2, b2, &v1[0]);
        dequant_word_i4(w1.y, s2, b2, &v1[4]);
        dequant_word_i4(w1.z, s2, b2, &v1[8]);
        dequant_word_i4(w1.w, s2, b2, &v1[12]);
        const int as = ait % kNS;
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(bar(b_sfree(as)), ((ait / kNS) & 1u) ^ 1u,
                                               abort_flag))) {
          ok = false;
          break;
        }
        ++ait;
        tc_fence_after();
        const uint32_t tcol = tmem + lane_off + kABase + as * kACols + g4 * 32;
        tmem_st16(tcol, v0);
        tmem_st16(tcol + 16, v1);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(b_sfull(as)));
      }
      t = nt;
    }
    if (!ok && lane == 0) {
      set_error(a.ctrl, MOE_ERR_TIMEOUT, KID_FFN, 5);
      *abort_flag = 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2 && !*tmem_keep) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <bool GATED>
static cudaError_t launch_one(const CUtensorMap& tw, const CUtensorMap& twsh, const CUtensorMap& tb,
                              const FfnArgs& a, int grid, cudaStream_t stream) {
  // the dynamic shared-memory opt-in is per device: set it once for each
  static std::atomic<unsigned long long> configured{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(configured.load() & bit)) {
    e = cudaFuncSetAttribute(ffn_w4_kernel<GATED>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemBytes);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit);
  }
  return launch_pdl(ffn_w4_kernel<GATED>, dim3(grid), dim3(kThreads), kSmemBytes, stream, tw, twsh,
                    tb, a);
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

// The grouped GEMM's activations in plan order: xs[p] = x[t(p)] for the
// routed rows p < R (t = sorted_rows[p] / K) and x[p - R] for the shared
// expert's rows, so a unit's rows are consecutive and load as plain TMA
// tiles; each group of 8 elements is stored in the (i, i+4)-paired order of
// the rebuilt weights. A row index outside [0, T) is recorded and copied as
// zeros.
// One warp per plan row p (grid-stride): the row's source token once, then
// every 16-byte chunk of the row in flight at once (lane chunks lane + 32m).
constexpr int kGatherWarps = 8;
constexpr int kGatherChunks = 8;  // chunks per lane in flight (H <= 2048 in one pass)
__global__ void __launch_bounds__(kGatherWarps * 32)
    gather_x_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ sorted_rows, int K,
                    int R, int S, int T, int hv, uint4* __restrict__ xs, Ctrl* ctrl) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  for (int p = blockIdx.x * kGatherWarps + (threadIdx.x >> 5); p < S;
       p += gridDim.x * kGatherWarps) {
    const int src = p < R ? __ldg(sorted_rows + p) / K : p - R;
    const bool ok = src >= 0 && src < T;
    if (!ok && lane == 0) set_error(ctrl, MOE_ERR_BAD_INPUT, KID_FFN, p);
    const uint4* xr = x + (size_t)(ok ? src : 0) * hv;
    uint4* dst = xs + (size_t)p * hv;
    for (int c0 = 0; c0 < hv; c0 += 32 * kGatherChunks) {
      uint4 v[kGatherChunks];
#pragma unroll
      for (int m = 0; m < kGatherChunks; ++m) {
        const int c = c0 + 32 * m + lane;
        v[m] = ok && c < hv ? __ldg(xr + c) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int m = 0; m < kGatherChunks; ++m) {
        const int c = c0 + 32 * m + lane;
        if (c < hv) dst[c] = to_i4_order(v[m]);
      }
    }
  }
}

cudaError_t launch_gather_x(const uint16_t* x, const int32_t* sorted_rows, int K, int R, int S,
                            int T, int H, uint16_t* xs, Ctrl* ctrl, int nsm, cudaStream_t stream) {
  const int want = (S + kGatherWarps - 1) / kGatherWarps;
  const int cap = nsm * 16;
  const int grid = want < cap ? want : cap;
  return launch_pdl(gather_x_kernel, dim3(grid > 0 ? grid : 1), dim3(kGatherWarps * 32), 0, stream,
                    reinterpret_cast<const uint4*>(x), sorted_rows, K, R, S, T, H / 8,
                    reinterpret_cast<uint4*>(xs), ctrl);
}

int ffn_tile_m() { return kTileM; }
int ffn_max_tile_n() { return kTileN; }
int ffn_stage_k() { return kKW; }
int ffn_b_box_rows() { return kBoxRows; }

}  // namespace moe
