// moe_plan_noalloc: the routing plan with its scratch in a fixed, statically
// allocated device array instead of a caller-provided workspace.
//
// Who needs it: code that must not allocate device memory at the point it
// builds a plan, e.g. a caller running inside a memory pool or allocator
// callback (allocating there would re-enter the allocator), an embedding
// runtime that forbids cudaMalloc after start-up, or a caller with no spare
// buffer to hand over. The plan's scratch is small (per-chunk expert
// histograms plus a status word), so it lives in one file-scope
// __device__ array that every device holds from module load until exit.
//
// The array's name in host code is only a host-side handle; its device
// address is looked up once per device with cudaGetSymbolAddress, with that
// device current, on the first call made on that device, and cached for the
// life of the process. A cudaDeviceReset unloads the module, so the array
// may come back at another address: the cached one is then stale, and this
// entry point must not be called on that device again in the process.
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kCtrlInts = (int)(sizeof(Ctrl) / sizeof(int32_t));
// status word + histograms: 256 KiB in total
constexpr size_t kScratchInts = 64 * 1024;
static __device__ __align__(256) int32_t g_plan_scratch[kScratchInts];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int32_t* g_addr[kMaxDevices] = {};

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status_t moe_plan_noalloc(const moe_shape_t* shape, const int32_t* topk_ids_dev,
                                         const moe_plan_t* plan, moe_stream_t stream) {
  if (!shape_supported(shape)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!topk_ids_dev || !plan || !plan->counts_dev || !plan->offsets_dev ||
      !plan->sorted_rows_dev || !plan->row_pos_dev || !plan->block_map_dev ||
      !plan->num_blocks_dev)
    return MOE_ERR_INVALID_ARG;
  const int64_t R = (int64_t)shape->T * shape->K;
  const int64_t nchunks = (R + kPlanChunkNoalloc - 1) / kPlanChunkNoalloc;
  if (kCtrlInts + nchunks * shape->E > (int64_t)kScratchInts) {
    set_last_error("moe_plan_noalloc: ceil(T*K/2048)*E exceeds the 65472-entry static scratch");
    return MOE_ERR_UNSUPPORTED_SHAPE;
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    set_last_cuda_error(e, "cudaGetDevice");
    return MOE_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    set_last_error("moe_plan_noalloc: device index out of range");
    return MOE_ERR_CUDA;
  }
  int32_t* base = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_addr[dev]) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_plan_scratch);
      if (e != cudaSuccess) {
        set_last_cuda_error(e, "cudaGetSymbolAddress");
        return MOE_ERR_CUDA;
      }
      g_addr[dev] = static_cast<int32_t*>(p);
    }
    base = g_addr[dev];
  }
  cudaStream_t st = (cudaStream_t)stream;
  // the status word must start clear; the histograms are fully rewritten
  e = cudaMemsetAsync(base, 0, sizeof(Ctrl), st);
  if (e != cudaSuccess) {
    set_last_cuda_error(e, "moe_plan_noalloc clear");
    return MOE_ERR_CUDA;
  }
  e = launch_plan(topk_ids_dev, shape->T, shape->K, shape->E, shape->n_shared, shape->tile_rows,
                  *plan, base + kCtrlInts, reinterpret_cast<Ctrl*>(base), kPlanChunkNoalloc, st);
  if (e != cudaSuccess) {
    set_last_cuda_error(e, "moe_plan_noalloc launch");
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}
