// Device-side helpers shared by the kernels of the W4A16 MoE layer:
// status word, bf16 unpacking, the 4-bit dequantisation routine, and thin
// inline-PTX wrappers for mbarrier, TMA and tcgen05 (sm_103a).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_w4.h"

namespace moe {

// ------------------------------------------------------------ workspace --
// The first 256 bytes of every workspace: the device status word and a
// little room for the kernels' own counters.
struct Ctrl {
  int err;           // first device error (moe_status_t), 0 = none
  int err_info[3];   // where it happened (kernel id, block, detail)
  unsigned ticket;   // reserved
  unsigned unit_next;  // grouped GEMM: next unit to hand out (reset by the last CTA)
  unsigned unit_done;  // grouped GEMM: CTAs finished handing out units
  unsigned ticket2;  // last-block counter of the decode down kernel (RMS norm)
  unsigned routed;   // decode: 1 once this layer's ids / w are published
  unsigned ps_seq;   // persistent decode: launches so far (epoch base of the next one)
  unsigned ps_exit;  // persistent decode: blocks finished (reset by the last one)
  unsigned ps_abort; // persistent decode: a wait ran out; every block stops waiting
  unsigned attn_arrive;  // attention: CTAs at the grid barrier (reset by the last)
  unsigned attn_gen;     // attention: grid barriers passed
  int pad[50];
};
static_assert(sizeof(Ctrl) == 256, "Ctrl must be 256 bytes");

enum : int { KID_PLAN = 1, KID_FFN = 2, KID_DECODE = 3, KID_ROUTE = 4, KID_ATTN = 5, KID_GDN = 6 };

__device__ __forceinline__ void set_error(Ctrl* c, int code, int kid, int detail) {
  if (atomicCAS(&c->err, 0, code) == 0) {
    c->err_info[0] = kid;
    c->err_info[1] = blockIdx.x;
    c->err_info[2] = detail;
  }
}

// ------------------------------------------------------------------ bf16 --
__device__ __forceinline__ float bf_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// fp32 pair -> bf16x2 bits (lo in the low half), round to nearest even.
__device__ __forceinline__ uint32_t pack_bf2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint32_t f2bf(float f) { return pack_bf2(f, 0.0f) & 0xFFFFu; }

// ------------------------------------------------------------- dequant --
// Groupwise-affine 4-bit dequantisation ("Perplexity Open Sources Lily: A
// Rust + Metal Inference Engine for Qwen3.6-35B-A3B on Apple Silicon",
// section "Prefill: Keep Weights Packed, Keep Routing on the GPU": 64
// weights per group share a bf16 scale and bias; w = scale*q + bias).
//
// nibble_pair_128: the low nibble of each 16-bit half of x, with the
// exponent pattern of 128.0 set above it -> the bf16 pair (128 + q_lo,
// 128 + q_hi), exact. One lop3: (x & 0x000F000F) | 0x43004300.
__device__ __forceinline__ uint32_t nibble_pair_128(uint32_t x) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(x), "r"(0x000F000Fu), "r"(0x43004300u));
  return d;
}
// affine_pair: m from nibble_pair_128 -> the bf16x2 pair (s*q_lo + b,
// s*q_hi + b), each with one rounding. s2 / b2 hold the group's scale /
// bias in both halves. fma(m, 1, -128) gives q exactly; fma(q, s, b) forms
// the exact product and sum and rounds once to nearest even. The two
// routines below differ only in which two nibbles they place.
__device__ __forceinline__ uint32_t affine_pair(uint32_t m, uint32_t s2, uint32_t b2) {
  uint32_t q, r;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(q) : "r"(m), "r"(0x3F803F80u), "r"(0xC300C300u));
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(q), "r"(s2), "r"(b2));
  return r;
}

// One packed word (element i = bits 4i..4i+3) -> 4 bf16x2 words holding the
// natural pairs (0,1), (2,3), (4,5), (6,7): a byte permute brings nibbles
// 2i and 2i+1 into the low bits of the two halves.
__device__ __forceinline__ void dequant_word(uint32_t w, uint32_t s2, uint32_t b2,
                                             uint32_t out[4]) {
  const uint32_t w4 = w >> 4;
#pragma unroll
  for (int i = 0; i < 4; ++i)
    out[i] = affine_pair(nibble_pair_128(__byte_perm(w, w4, 0x0400u + 0x0101u * i)), s2, b2);
}

// The same word -> 4 bf16x2 words where word i holds elements i (low half)
// and i+4 (high half): a shift by 4i and one lop3 place both nibbles, the
// cheapest placement (7 integer instructions per word). Consumers see the
// elements of each group of 8 in the order 0, 4, 1, 5, 2, 6, 3, 7.
__device__ __forceinline__ void dequant_word_i4(uint32_t w, uint32_t s2, uint32_t b2,
                                                uint32_t out[4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) out[i] = affine_pair(nibble_pair_128(w >> (4 * i)), s2, b2);
}

// Position of reduction element k in the (i, i+4)-paired order of
// dequant_word_i4: element k of its group of 8 sits at 2*(k%4) + (k%8)/4.
__host__ __device__ __forceinline__ int i4_pos(int k) {
  return (k & ~7) | ((k & 3) << 1) | ((k >> 2) & 1);
}
// 8 bf16 in natural order (v.x = (e0,e1), ..., v.w = (e6,e7)) -> the
// (i, i+4)-paired order ((e0,e4), (e1,e5), (e2,e6), (e3,e7)).
__device__ __forceinline__ uint4 to_i4_order(const uint4& v) {
  return make_uint4(__byte_perm(v.x, v.z, 0x5410), __byte_perm(v.x, v.z, 0x7632),
                    __byte_perm(v.y, v.w, 0x5410), __byte_perm(v.y, v.w, 0x7632));
}

__device__ __forceinline__ uint32_t dup_lo(uint32_t v) { return __byte_perm(v, 0, 0x1010); }
__device__ __forceinline__ uint32_t dup_hi(uint32_t v) { return __byte_perm(v, 0, 0x3232); }

// ------------------------------------------------ dependent launches --
// Programmatic dependent launch: a kernel launched with programmatic stream
// serialisation may start before its predecessor in the stream finishes.
// pdl_wait() blocks until the predecessor grid has completed and its writes
// are visible; pdl_trigger() lets the successor launch once every block of
// this grid has triggered or exited. Both are no-ops in a plain launch.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// The MoE layer's kernels (router, plan, gather, grouped GEMMs, combine)
// set up what reads no global memory (barriers, TMEM, tensor-map
// prefetch), call pdl_wait(), then pdl_trigger(): with the trigger after
// the wait, when a kernel starts every kernel two or more launches before it
// on the stream has completed, so only the immediate predecessor's outputs
// need the wait.
// Launches kern on stream with programmatic stream serialisation allowed.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// Asks L2 to fetch [p, p + bytes) (16-byte aligned, bytes % 16 == 0); no
// data reaches the thread, so the copy can never be stale.
__device__ __forceinline__ void bulk_prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// --------------------------------------------------------------- timing --
__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Every spin-wait in this library gives up after this long and reports
// MOE_ERR_TIMEOUT; no correct launch waits anywhere near it.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// -------------------------------------------------------------- mbarrier --
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// Orders this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (TMA) accesses that other threads make after a barrier,
// e.g. before a buffer read with ld.shared is handed back to a TMA refill.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Non-blocking phase test, and a bounded spin on it. Cheaper than try_wait
// for a thread (the MMA issuer) whose waits are usually already satisfied.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_spin(uint32_t bar, uint32_t parity, volatile int* abort) {
  if (mbar_test_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_test_wait(bar, parity)) return true;
    if ((i & 255u) == 0) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
    }
  }
}
// try_wait that may suspend the thread for up to `hint_ns` (woken when the
// phase completes): for roles that wait long, so they do not spin on the
// issue slots the working warps need.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_sleep(uint32_t bar, uint32_t parity, volatile int* abort) {
  if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
    if (*abort) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
  }
}
// Bounded wait for the phase with the given parity to complete. Returns
// false if *abort becomes non-zero or the wait limit passes.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
    }
  }
}

// ------------------------------------------------------------------- TMA --
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* tm) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(tm) : "memory");
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* tm, int c0, int c1,
                                            uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(tm), "r"(c0), "r"(c1), "r"(bar), "l"(policy)
      : "memory");
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// --------------------------------------------------------------- tcgen05 --
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]^T, bf16 inputs, fp32 accumulation.
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Same, always accumulating into D (the predicate is the constant true).
__device__ __forceinline__ void mma_bf16_ts_acc(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                uint32_t idesc) {
  asm volatile("tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, 1;" ::"r"(d_tmem),
               "r"(a_tmem), "l"(b_desc), "r"(idesc)
               : "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, fp32 accumulation.
__device__ __forceinline__ void mma_bf16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// 16 consecutive TMEM columns of this warp's lane quarter, one per register.
__device__ __forceinline__ void tmem_ld16r(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]),
        "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15])
      : "memory");
}
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&v)[8]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7])
      : "r"(taddr)
      : "memory");
}

// Shared-memory matrix descriptor of a K-major bf16 operand stored in
// 128-byte-swizzled atoms (8 rows x 128 bytes, 1024 bytes apart).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)1 << 16;            // leading byte offset (unused for this layout)
  d |= (uint64_t)(1024 >> 4) << 32;  // stride byte offset: next 8-row group
  d |= (uint64_t)1 << 46;            // descriptor version for tcgen05
  d |= (uint64_t)2 << 61;            // 128-byte swizzle
  return d;
}
// Instruction descriptor: kind::f16, A and B bf16 K-major, D fp32, M x N.
__host__ __device__ __forceinline__ uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31u; }

}  // namespace moe
