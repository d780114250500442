// Routing plan on the GPU: expert histogram, exclusive prefix scan, stable
// scatter of (token, slot) rows into expert-contiguous order, and the tile
// block map ("Perplexity Open Sources Lily: A Rust + Metal Inference Engine
// for Qwen3.6-35B-A3B on Apple Silicon", section "Prefill: Keep Weights
// Packed, Keep Routing on the GPU": every step that turns expert ids into
// the grouped GEMM's schedule runs as device kernels, and the host never
// waits on the device between them). Integer work only: results are unique
// and deterministic.
//
// Two launches. plan_hist: block c counts the experts of items
// [c*CH, (c+1)*CH) into hist[c][E] (the layer call has the router's screen
// count them instead and launches plan_scatter alone). plan_scatter: block c derives the
// global offsets and its own starting position per expert from all blocks'
// histograms, then scatters its items in ascending order, 256 per round,
// ranking equal experts inside a warp with match.any and across warps with
// per-warp counts. Block 0 also writes counts, offsets and the block map.
#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int kPlanThreads = 256;
constexpr int kPlanWarps = kPlanThreads / 32;
constexpr int kMaxE = 1024;

__global__ void __launch_bounds__(kPlanThreads) plan_hist_kernel(const int32_t* __restrict__ ids,
                                                                 int R, int E, int chunk,
                                                                 int32_t* __restrict__ hist,
                                                                 Ctrl* ctrl) {
  pdl_wait();
  pdl_trigger();
  __shared__ int h[kMaxE];
  for (int e = threadIdx.x; e < E; e += kPlanThreads) h[e] = 0;
  __syncthreads();
  const int f0 = blockIdx.x * chunk;
  const int f1 = min(f0 + chunk, R);
  for (int f = f0 + threadIdx.x; f < f1; f += kPlanThreads) {
    const int e = ids[f];
    if (e < 0 || e >= E)
      set_error(ctrl, MOE_ERR_BAD_INPUT, KID_PLAN, f);
    else
      atomicAdd(&h[e], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += kPlanThreads) hist[(size_t)blockIdx.x * E + e] = h[e];
}

// Exclusive scan of v over the block (one value per thread); returns the
// thread's exclusive prefix and writes the block total to *total.
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int inc = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int o = __shfl_up_sync(0xFFFFFFFFu, inc, d);
    if (lane >= d) inc += o;
  }
  if (lane == 31) warp_sums[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    int s = (lane < kPlanWarps) ? warp_sums[lane] : 0;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int o = __shfl_up_sync(0xFFFFFFFFu, s, d);
      if (lane >= d) s += o;
    }
    if (lane < kPlanWarps) warp_sums[lane] = s;  // inclusive over warps
  }
  __syncthreads();
  const int before = (warp > 0) ? warp_sums[warp - 1] : 0;
  *total = warp_sums[kPlanWarps - 1];
  __syncthreads();
  return before + inc - v;
}

__global__ void __launch_bounds__(kPlanThreads)
    plan_scatter_kernel(const int32_t* __restrict__ ids, int T, int K, int E, int n_shared,
                        int BM, const int32_t* __restrict__ hist, int nchunks, int chunk,
                        moe_plan_t plan) {
  pdl_wait();
  pdl_trigger();
  __shared__ int base[kMaxE];                 // this block's next position per expert
  __shared__ int wcnt[kPlanWarps][kMaxE];     // per-round, per-warp counts -> prefixes
  __shared__ int warp_sums[32];
  const int R = T * K;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // Each thread owns experts [tid*EPT, tid*EPT + EPT).
  const int EPT = (E + kPlanThreads - 1) / kPlanThreads;  // <= 4
  int tot[4], pre[4];
  int my_sum = 0;
  _Pragma("unroll") for (int i = 0; i < 4; ++i) {
    if (i >= EPT) break;
    const int e = tid * EPT + i;
    int t = 0, p = 0;
    if (e < E) {
#pragma unroll 8
      for (int c = 0; c < nchunks; ++c) {
        const int v = hist[(size_t)c * E + e];
        t += v;
        if (c < (int)blockIdx.x) p += v;
      }
    }
    tot[i] = t;
    pre[i] = p;
    my_sum += t;
  }
  int total;
  int off = block_exclusive_scan(my_sum, warp_sums, &total);
  _Pragma("unroll") for (int i = 0; i < 4; ++i) {
    if (i >= EPT) break;
    const int e = tid * EPT + i;
    if (e < E) {
      base[e] = off + pre[i];
      if (blockIdx.x == 0) {
        plan.counts_dev[e] = tot[i];
        plan.offsets_dev[e] = off;
      }
    }
    off += tot[i];
  }
  if (blockIdx.x == 0 && tid == kPlanThreads - 1) plan.offsets_dev[E] = off;

  // Block map (block 0): routed tiles per expert, then the shared rows.
  if (blockIdx.x == 0) {
    int nb_mine = 0;
    _Pragma("unroll") for (int i = 0; i < 4; ++i) if (i < EPT) nb_mine += (tot[i] + BM - 1) / BM;
    int nb_total;
    int bstart = block_exclusive_scan(nb_mine, warp_sums, &nb_total);
    int rs = off - my_sum;  // first row of my first expert
    _Pragma("unroll") for (int i = 0; i < 4; ++i) {
    if (i >= EPT) break;
      const int e = tid * EPT + i;
      for (int r0 = 0; r0 < tot[i]; r0 += BM) {
        int32_t* b = plan.block_map_dev + 3 * bstart;
        b[0] = e;
        b[1] = rs + r0;
        b[2] = min(BM, tot[i] - r0);
        ++bstart;
      }
      rs += tot[i];
    }
    const int nsb = n_shared ? (T + BM - 1) / BM : 0;
    for (int j = tid; j < nsb; j += kPlanThreads) {
      int32_t* b = plan.block_map_dev + 3 * (nb_total + j);
      b[0] = E;
      b[1] = R + j * BM;
      b[2] = min(BM, T - j * BM);
    }
    if (tid == 0) *plan.num_blocks_dev = nb_total + nsb;
  }

  for (int i = tid; i < kPlanWarps * E; i += kPlanThreads) wcnt[i / E][i % E] = 0;
  __syncthreads();

  const int f0 = blockIdx.x * chunk;
  const int f1 = min(f0 + chunk, R);
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int r0 = f0; r0 < f1; r0 += kPlanThreads) {
    const int f = r0 + tid;
    int e = (f < f1) ? ids[f] : -1;
    if (e < 0 || e >= E) e = -1;  // reported by plan_hist; skipped here
    const unsigned m = __match_any_sync(0xFFFFFFFFu, e);
    const int rank = __popc(m & lt_mask);
    if (e >= 0 && rank == 0) wcnt[warp][e] = __popc(m);
    __syncthreads();
    // per expert: exclusive prefix over warps, in place; remember the total
    int rtot[4];
    _Pragma("unroll") for (int i = 0; i < 4; ++i) {
    if (i >= EPT) break;
      const int ee = tid * EPT + i;
      int s = 0;
      if (ee < E) {
#pragma unroll
        for (int w = 0; w < kPlanWarps; ++w) {
          const int c = wcnt[w][ee];
          wcnt[w][ee] = s;
          s += c;
        }
      }
      rtot[i] = s;
    }
    __syncthreads();
    if (e >= 0) {
      const int pos = base[e] + wcnt[warp][e] + rank;
      plan.sorted_rows_dev[pos] = f;
      plan.row_pos_dev[f] = pos;
    }
    __syncthreads();
    _Pragma("unroll") for (int i = 0; i < 4; ++i) {
    if (i >= EPT) break;
      const int ee = tid * EPT + i;
      if (ee < E) {
        base[ee] += rtot[i];
#pragma unroll
        for (int w = 0; w < kPlanWarps; ++w) wcnt[w][ee] = 0;
      }
    }
    __syncthreads();
  }
}

cudaError_t launch_plan(const int32_t* ids, int T, int K, int E, int n_shared, int BM,
                        const moe_plan_t& plan, int32_t* hist, Ctrl* ctrl, int chunk,
                        cudaStream_t stream, bool hist_ready) {
  const int R = T * K;
  const int nchunks = (R + chunk - 1) / chunk;
  if (!hist_ready) {  // else the router's screen counted the chunks already
    cudaError_t err = launch_pdl(plan_hist_kernel, dim3(nchunks), dim3(kPlanThreads), 0, stream,
                                 ids, R, E, chunk, hist, ctrl);
    if (err != cudaSuccess) return err;
  }
  return launch_pdl(plan_scatter_kernel, dim3(nchunks), dim3(kPlanThreads), 0, stream, ids, T, K,
                    E, n_shared, BM, hist, nchunks, chunk, plan);
}

}  // namespace moe
