// C ABI of the W4A16 MoE expert layer (declared in include/moe_w4.h):
// host-side validation, workspace layout, TMA descriptors and launches.
// Nothing here allocates device memory or synchronises a stream, except
// moe_query_device_status, whose job is to synchronise.
#include <atomic>
#include <climits>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <string>

#include "common.cuh"
#include "kernels.h"

using namespace moe;

namespace {

thread_local std::string g_last_error;

moe_status_t cuda_fail(cudaError_t e, const char* where) {
  g_last_error = std::string(where) + ": " + cudaGetErrorString(e);
  return MOE_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool shape_ok(const moe_shape_t* s) {
  if (!s) return false;
  if (s->T < 1 || s->H < 256 || s->H % 256 != 0 || s->H > 8192) return false;
  if (s->I < 128 || s->I % 128 != 0 || s->I > 8192) return false;
  if (s->K < 1 || s->K > 32 || s->E < s->K || s->E > 1024) return false;
  if (s->n_shared != 0 && s->n_shared != 1) return false;
  if (s->tile_rows < 1 || s->tile_rows > ffn_max_tile_n()) return false;
  const int64_t R = (int64_t)s->T * s->K;
  const int64_t S = R + (int64_t)s->T * s->n_shared;
  if (S * s->H >= INT32_MAX || S * s->I >= INT32_MAX) return false;
  if ((int64_t)s->T * s->E >= INT32_MAX) return false;
  if ((int64_t)s->E * 2 * s->I * (s->H / 8) >= INT32_MAX) return false;
  if ((int64_t)s->E * s->H * (s->I / 8) >= INT32_MAX) return false;
  return true;
}

int64_t max_blocks_of(const moe_shape_t* s) {
  const int64_t R = (int64_t)s->T * s->K, BM = s->tile_rows;
  const int64_t shared_blocks = s->n_shared ? (s->T + BM - 1) / BM : 0;
  return (R + BM - 1) / BM + (R < s->E ? R : s->E) + shared_blocks;
}

struct Layout {
  size_t ctrl, hist, logits, h, ids, w, counts, offsets, sorted, rowpos, bmap, nblk, yslots, part,
      rpart, part2, ybuf, tags, xmid, xs, blk, total;
};

Layout layout_of(const moe_shape_t* s) {
  Layout L{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += (bytes + 255) & ~(size_t)255;
    return o;
  };
  const size_t T = s->T, K = s->K, E = s->E, R = T * K, S = R + T * s->n_shared;
  const size_t nchunks = (R + kPlanChunk - 1) / kPlanChunk;
  L.ctrl = take(sizeof(Ctrl));
  L.hist = take(nchunks * E * 4);
  L.logits = take(T * E * 4);
  L.h = take(S * (size_t)s->I * 2);
  L.ids = take(R * 4);
  L.w = take(R * 4);
  L.counts = take(E * 4);
  L.offsets = take((E + 1) * 4);
  L.sorted = take(R * 4);
  L.rowpos = take(R * 4);
  L.bmap = take((size_t)max_blocks_of(s) * 12);
  L.nblk = take(4);
  L.yslots = take(S * (size_t)s->H * 2);
  L.xs = take(S * (size_t)s->H * 2);  // the grouped GEMM's activations in plan order
  L.part = take(decode_part_floats(s->T, s->H) * 4);
  L.rpart = route_tc_supported(s->T, s->H, s->E, s->K)
                ? take(route_tc_partial_floats(s->T, s->H, s->E) * 4)
                : off;
  // stacked decode: a second partial buffer and two y buffers (ping-pong;
  // decoder blocks hand the residual stream between persistent launches
  // through them too)
  const bool dec = decode_supported(s->T, s->H, s->E, s->K, s->I, s->n_shared);
  const bool ps = persist_supported(s->T, s->H, s->E, s->K, s->I, s->n_shared);
  L.part2 = dec ? take(decode_part_floats(s->T, s->H) * 4) : off;
  L.ybuf = (dec || ps) ? take((size_t)2 * T * s->H * 2) : off;
  // persistent decode: the epoch-tagged block-to-block words, and the
  // normalised input handed from one launch of up to kPersistMaxLayers
  // layers to the next
  L.tags = ps ? take(persist_tags(s->T, s->H, s->E, s->K, s->I, s->n_shared).total * 8) : off;
  L.xmid = ps ? take(T * (size_t)s->H * 2) : off;
  // decoder blocks through the four calls: two residual buffers and x
  L.blk = take((size_t)3 * T * s->H * 2);
  L.total = off;
  return L;
}

// ---------------------------------------------------------- device info --
constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];

moe_status_t sm_count(int* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) {
    g_last_error = "device index out of range";
    return MOE_ERR_CUDA;
  }
  int n = g_sm_count[dev].load();
  if (n == 0) {
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    g_sm_count[dev].store(n);
  }
  *out = n;
  return MOE_OK;
}

// ---------------------------------------------------------- tensor maps --
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// Row-major 2-D tensor [outer][inner] of elements of `esize` bytes.
moe_status_t map_2d(CUtensorMap* m, CUtensorMapDataType dt, size_t esize, const void* base,
                    uint64_t inner, uint64_t outer, uint32_t box_inner, uint32_t box_outer,
                    CUtensorMapSwizzle sw) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) {
    g_last_error = "cuTensorMapEncodeTiled unavailable";
    return MOE_ERR_CUDA;
  }
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * esize};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  CUresult r = enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    g_last_error = "cuTensorMapEncodeTiled failed: " + std::to_string((int)r);
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

// 3-D tensor [d2][d1][d0] of elements of `esize` bytes, dense.
moe_status_t map_3d(CUtensorMap* m, CUtensorMapDataType dt, size_t esize, const void* base,
                    uint64_t d0, uint64_t d1, uint64_t d2, uint32_t b0, uint32_t b1, uint32_t b2,
                    CUtensorMapSwizzle sw) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) {
    g_last_error = "cuTensorMapEncodeTiled unavailable";
    return MOE_ERR_CUDA;
  }
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {d0 * esize, d0 * d1 * esize};
  cuuint32_t box[3] = {b0, b1, b2};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(m, dt, 3, const_cast<void*>(base), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    g_last_error = "cuTensorMapEncodeTiled (3-D) failed: " + std::to_string((int)r);
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

bool weights_ok(const moe_w4_weights_t* w) {
  return w && w->q_gate_up_dev && w->s_gate_up_dev && w->b_gate_up_dev && w->q_down_dev &&
         w->s_down_dev && w->b_down_dev && aligned16(w->q_gate_up_dev) &&
         aligned16(w->s_gate_up_dev) && aligned16(w->b_gate_up_dev) &&
         aligned16(w->q_down_dev) && aligned16(w->s_down_dev) && aligned16(w->b_down_dev);
}

bool plan_ok(const moe_plan_t* p) {
  return p && p->counts_dev && p->offsets_dev && p->sorted_rows_dev && p->row_pos_dev &&
         p->block_map_dev && p->num_blocks_dev;
}

moe_status_t check_ws(const moe_shape_t* s, void* ws, size_t ws_bytes) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < layout_of(s).total) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

#define MOE_TRY(x)                     \
  do {                                 \
    moe_status_t st_ = (x);            \
    if (st_ != MOE_OK) return st_;     \
  } while (0)

moe_status_t run_ffn(const moe_shape_t* s, const void* x, const moe_w4_weights_t* ex,
                     const moe_w4_weights_t* sh, const moe_plan_t* plan, void* y_slots,
                     uint8_t* ws, cudaStream_t stream) {
  const Layout L = layout_of(s);
  const int T = s->T, H = s->H, E = s->E, K = s->K, I = s->I;
  const int R = T * K, S = R + T * s->n_shared;
  const int maxb = (int)max_blocks_of(s);
  int nsm = 0;
  MOE_TRY(sm_count(&nsm));
  const moe_w4_weights_t* shw = s->n_shared ? sh : ex;
  uint16_t* h = reinterpret_cast<uint16_t*>(ws + L.h);
  Ctrl* ctrl = reinterpret_cast<Ctrl*>(ws + L.ctrl);

  CUtensorMap tw, twsh, tx, th;
  // packed gate_up weights as (word, row of the half, 2*expert + half):
  // boxes of 32 words (256 reduction elements) x 16 rows x both halves, so
  // one box brings 16 gate rows and the matching 16 up rows
  const uint32_t wbox = (uint32_t)ffn_stage_k() / 8;
  MOE_TRY(map_3d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, ex->q_gate_up_dev, H / 8, I,
                 (uint64_t)E * 2, wbox, 16, 2, CU_TENSOR_MAP_SWIZZLE_128B));
  MOE_TRY(map_3d(&twsh, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, shw->q_gate_up_dev, H / 8, I,
                 (uint64_t)(s->n_shared ? 1 : E) * 2, wbox, 16, 2, CU_TENSOR_MAP_SWIZZLE_128B));
  uint16_t* xs = reinterpret_cast<uint16_t*>(ws + L.xs);
  cudaError_t ge = launch_gather_x(static_cast<const uint16_t*>(x), plan->sorted_rows_dev, K, R, S,
                                   T, H, xs, ctrl, nsm, stream);
  if (ge != cudaSuccess) return cuda_fail(ge, "activation gather launch");
  // operand rows: boxes of ffn_b_box_rows() rows x 64 elements
  const uint32_t bbox = (uint32_t)ffn_b_box_rows();
  MOE_TRY(map_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, xs, H, S, 64, bbox,
                 CU_TENSOR_MAP_SWIZZLE_128B));
  FfnArgs a{};
  a.block_map = plan->block_map_dev;
  a.num_blocks = plan->num_blocks_dev;
  a.sorted_rows = plan->sorted_rows_dev;
  a.K = K;
  a.R = R;
  a.E = E;
  a.rows_per_expert = 2 * I;
  a.half_rows = I;
  a.mtiles = I / (ffn_tile_m() / 2);  // 64 gate + 64 up rows per unit
  a.kdim = H;
  a.kgroups = H / 64;
  a.s_exp = ex->s_gate_up_dev;
  a.b_exp = ex->b_gate_up_dev;
  a.s_sh = shw->s_gate_up_dev;
  a.b_sh = shw->b_gate_up_dev;
  a.out = h;
  a.out_ld = I;
  a.ctrl = ctrl;
  a.max_units = maxb * a.mtiles;
  a.shared_blocks = s->n_shared ? (T + s->tile_rows - 1) / s->tile_rows : 0;
  cudaError_t e = launch_ffn_gate_up(tw, twsh, tx, a, a.max_units < nsm ? a.max_units : nsm, stream);
  if (e != cudaSuccess) return cuda_fail(e, "ffn gate_up launch");

  // packed down weights: boxes of 128 rows x 32 words; a reduction length
  // that is not a multiple of 256 reads zero-filled words past the row end
  // in its last box
  MOE_TRY(map_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, ex->q_down_dev, I / 8, (uint64_t)E * H,
                 wbox, 128, CU_TENSOR_MAP_SWIZZLE_128B));
  MOE_TRY(map_2d(&twsh, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, shw->q_down_dev, I / 8,
                 (uint64_t)(s->n_shared ? 1 : E) * H, wbox, 128, CU_TENSOR_MAP_SWIZZLE_128B));
  MOE_TRY(map_2d(&th, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, h, I, S, 64, bbox,
                 CU_TENSOR_MAP_SWIZZLE_128B));
  a.sorted_rows = nullptr;
  a.rows_per_expert = H;
  a.half_rows = 0;
  a.mtiles = H / ffn_tile_m();            // 128 consecutive rows per unit
  a.kdim = I;
  a.kgroups = I / 64;
  a.s_exp = ex->s_down_dev;
  a.b_exp = ex->b_down_dev;
  a.s_sh = shw->s_down_dev;
  a.b_sh = shw->b_down_dev;
  a.out = reinterpret_cast<uint16_t*>(y_slots);
  a.out_ld = H;
  a.max_units = maxb * a.mtiles;
  e = launch_ffn_down(tw, twsh, th, a, a.max_units < nsm ? a.max_units : nsm, stream);
  if (e != cudaSuccess) return cuda_fail(e, "ffn down launch");
  return MOE_OK;
}

// Arguments of one decode layer with every workspace intermediate; the
// caller sets x / y_prev, ids, w, y, x_next and the stacking fields.
DecodeArgs decode_args(const moe_shape_t* s, const void* w_router, const float* bias,
                       const moe_w4_weights_t* experts, const moe_w4_weights_t* shared,
                       uint8_t* ws, const Layout& L) {
  DecodeArgs d{};
  d.wr = static_cast<const uint16_t*>(w_router);
  d.bias = bias;
  d.T = s->T;
  d.H = s->H;
  d.E = s->E;
  d.K = s->K;
  d.I = s->I;
  d.ns = s->n_shared;
  d.ex = *experts;
  d.sh = s->n_shared ? *shared : *experts;
  d.logits = reinterpret_cast<float*>(ws + L.logits);
  d.ids = reinterpret_cast<int32_t*>(ws + L.ids);
  d.w = reinterpret_cast<float*>(ws + L.w);
  d.h = reinterpret_cast<uint16_t*>(ws + L.h);
  d.part = reinterpret_cast<float*>(ws + L.part);
  d.ctrl = reinterpret_cast<Ctrl*>(ws + L.ctrl);
  return d;
}

// moe_decode_layers on the persistent kernel: launches of up to
// kPersistMaxLayers layers; between two launches the normalised input
// passes through the workspace (the bits the next layer would form itself).
moe_status_t decode_persistent(const moe_shape_t* s, int n_layers,
                               const moe_layer_weights_t* layers, const void* x, void* y,
                               void* x_next, int32_t* ids, float* w, uint8_t* ws,
                               const Layout& L, int grid, size_t smem, cudaStream_t stream) {
  PersistArgs a{};
  a.T = s->T;
  a.H = s->H;
  a.E = s->E;
  a.K = s->K;
  a.I = s->I;
  a.ns = s->n_shared;
  a.y = static_cast<uint16_t*>(y);
  a.ids = ids ? ids : reinterpret_cast<int32_t*>(ws + L.ids);
  a.w = w ? w : reinterpret_cast<float*>(ws + L.w);
  uint64_t* tags = reinterpret_cast<uint64_t*>(ws + L.tags);
  const PersistTags tl = persist_tags(s->T, s->H, s->E, s->K, s->I, s->n_shared);
  a.logits_tag = tags + tl.logits;
  a.h_tag = tags + tl.h;
  a.y_tag = tags + tl.y;
  a.ctrl = reinterpret_cast<Ctrl*>(ws + L.ctrl);
  uint16_t* xmid = reinterpret_cast<uint16_t*>(ws + L.xmid);
  for (int l0 = 0; l0 < n_layers; l0 += kPersistMaxLayers) {
    const int n = n_layers - l0 < kPersistMaxLayers ? n_layers - l0 : kPersistMaxLayers;
    a.n_layers = n;
    a.x = l0 == 0 ? static_cast<const uint16_t*>(x) : xmid;
    a.x_next = l0 + n == n_layers ? static_cast<uint16_t*>(x_next) : xmid;
    for (int i = 0; i < n; ++i) {
      a.layer[i] = layers[l0 + i];
      if (!s->n_shared) a.layer[i].shared = a.layer[i].experts;
    }
    cudaError_t e = launch_decode_persist(a, grid, smem, stream);
    if (e != cudaSuccess) return cuda_fail(e, "persistent decode launch");
  }
  return MOE_OK;
}

// Decoder blocks through the persistent kernel, 48 layers per launch; the
// residual stream passes between launches through the two ybuf halves.
moe_status_t decoder_blocks_persistent(const moe_shape_t* s, int n_layers,
                                     const moe_layer_weights_t* layers,
                                     const void* const* gains, const void* h_in,
                                     const int32_t* tok, const void* embed, int vocab,
                                     void* h_out, uint8_t* ws, const Layout& L, int grid,
                                     size_t smem, cudaStream_t stream) {
  PersistArgs a{};
  a.T = s->T;
  a.H = s->H;
  a.E = s->E;
  a.K = s->K;
  a.I = s->I;
  a.ns = s->n_shared;
  a.ids = reinterpret_cast<int32_t*>(ws + L.ids);
  a.w = reinterpret_cast<float*>(ws + L.w);
  uint64_t* tags = reinterpret_cast<uint64_t*>(ws + L.tags);
  const PersistTags tl = persist_tags(s->T, s->H, s->E, s->K, s->I, s->n_shared);
  a.logits_tag = tags + tl.logits;
  a.h_tag = tags + tl.h;
  a.y_tag = tags + tl.y;
  a.ctrl = reinterpret_cast<Ctrl*>(ws + L.ctrl);
  a.block = 1;
  a.vocab = vocab;
  a.embed = static_cast<const uint16_t*>(embed);
  uint16_t* mid[2] = {reinterpret_cast<uint16_t*>(ws + L.ybuf),
                      reinterpret_cast<uint16_t*>(ws + L.ybuf) + (size_t)s->T * s->H};
  for (int l0 = 0, c = 0; l0 < n_layers; l0 += kPersistMaxLayers, ++c) {
    const int n = n_layers - l0 < kPersistMaxLayers ? n_layers - l0 : kPersistMaxLayers;
    a.n_layers = n;
    a.tok = l0 == 0 ? tok : nullptr;
    a.x = l0 == 0 ? static_cast<const uint16_t*>(h_in) : mid[(c - 1) & 1];
    a.y = l0 + n == n_layers ? static_cast<uint16_t*>(h_out) : mid[c & 1];
    for (int i = 0; i < n; ++i) {
      a.layer[i] = layers[l0 + i];
      if (!s->n_shared) a.layer[i].shared = a.layer[i].experts;
      a.gain[i] = static_cast<const uint16_t*>(gains[l0 + i]);
    }
    cudaError_t e = launch_decode_persist(a, grid, smem, stream);
    if (e != cudaSuccess) return cuda_fail(e, "persistent decode block launch");
  }
  return MOE_OK;
}

}  // namespace

namespace moe {
bool shape_supported(const moe_shape_t* shape) { return shape_ok(shape); }
void set_last_error(const char* text) { g_last_error = text; }
void set_last_cuda_error(cudaError_t e, const char* where) { cuda_fail(e, where); }
}  // namespace moe

extern "C" {

size_t moe_workspace_bytes(const moe_shape_t* shape) {
  return shape_ok(shape) ? layout_of(shape).total : 0;
}

int32_t moe_layer_path(const moe_shape_t* shape) {
  if (!shape_ok(shape)) return -1;
  int grid = 0;
  size_t smem = 0;
  if (persist_config(shape->T, shape->H, shape->E, shape->K, shape->I, shape->n_shared, &grid, &smem))
    return 2;
  return decode_supported(shape->T, shape->H, shape->E, shape->K, shape->I, shape->n_shared) ? 1 : 0;
}

int32_t moe_max_blocks(const moe_shape_t* shape) {
  return shape_ok(shape) ? (int32_t)max_blocks_of(shape) : 0;
}

moe_status_t moe_workspace_init(void* ws_dev, size_t ws_bytes, moe_stream_t stream) {
  if (!ws_dev || ws_bytes < sizeof(Ctrl)) return MOE_ERR_INVALID_ARG;
  cudaError_t e = cudaMemsetAsync(ws_dev, 0, ws_bytes, (cudaStream_t)stream);
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "moe_workspace_init");
}

// The tensor-core router (route_tc_supported shapes); hist != nullptr also
// has its screen count the plan's chunk histogram into hist.
static moe_status_t route_tc(const moe_shape_t* shape, const void* x_dev,
                             const void* w_router_dev, const float* router_bias_dev,
                             int32_t* ids, float* w, uint8_t* ws, const Layout& L,
                             cudaStream_t st, int32_t* hist) {
  CUtensorMap tw, tx;
  MOE_TRY(map_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, w_router_dev, shape->H, shape->E, 64,
                 128, CU_TENSOR_MAP_SWIZZLE_128B));
  MOE_TRY(map_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, x_dev, shape->H, shape->T, 64, 128,
                 CU_TENSOR_MAP_SWIZZLE_128B));
  cudaError_t e = launch_route_tc(
      tw, tx, static_cast<const uint16_t*>(x_dev), static_cast<const uint16_t*>(w_router_dev),
      router_bias_dev, shape->T, shape->H, shape->E, shape->K,
      reinterpret_cast<float*>(ws + L.rpart), ids, w, reinterpret_cast<Ctrl*>(ws + L.ctrl), st,
      hist, kPlanChunk);
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "moe_route launch");
}

moe_status_t moe_route(const moe_shape_t* shape, const void* x_dev, const void* w_router_dev,
                       const float* router_bias_dev, int32_t* topk_ids_dev, float* topk_w_dev,
                       void* ws_dev, size_t ws_bytes, moe_stream_t stream) {
  if (!shape_ok(shape)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!x_dev || !w_router_dev || !topk_ids_dev || !topk_w_dev) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x_dev) || !aligned16(w_router_dev)) return MOE_ERR_INVALID_ARG;
  MOE_TRY(check_ws(shape, ws_dev, ws_bytes));
  uint8_t* ws = static_cast<uint8_t*>(ws_dev);
  const Layout L = layout_of(shape);
  if (route_tc_supported(shape->T, shape->H, shape->E, shape->K))
    return route_tc(shape, x_dev, w_router_dev, router_bias_dev, topk_ids_dev, topk_w_dev, ws, L,
                    (cudaStream_t)stream, nullptr);
  cudaError_t e = launch_route(static_cast<const uint16_t*>(x_dev),
                               static_cast<const uint16_t*>(w_router_dev), router_bias_dev,
                               shape->T, shape->H, shape->E, shape->K,
                               reinterpret_cast<float*>(ws + L.logits), topk_ids_dev, topk_w_dev,
                               (cudaStream_t)stream);
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "moe_route launch");
}

moe_status_t moe_plan(const moe_shape_t* shape, const int32_t* topk_ids_dev,
                      const moe_plan_t* plan, void* ws_dev, size_t ws_bytes,
                      moe_stream_t stream) {
  if (!shape_ok(shape)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!topk_ids_dev || !plan_ok(plan)) return MOE_ERR_INVALID_ARG;
  MOE_TRY(check_ws(shape, ws_dev, ws_bytes));
  uint8_t* ws = static_cast<uint8_t*>(ws_dev);
  const Layout L = layout_of(shape);
  cudaError_t e = launch_plan(topk_ids_dev, shape->T, shape->K, shape->E, shape->n_shared,
                              shape->tile_rows, *plan, reinterpret_cast<int32_t*>(ws + L.hist),
                              reinterpret_cast<Ctrl*>(ws + L.ctrl), kPlanChunk,
                              (cudaStream_t)stream);
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "moe_plan launch");
}

moe_status_t moe_expert_ffn_w4(const moe_shape_t* shape, const void* x_dev,
                               const moe_w4_weights_t* experts, const moe_w4_weights_t* shared,
                               const moe_plan_t* plan, void* y_slots_dev, void* ws_dev,
                               size_t ws_bytes, moe_stream_t stream) {
  if (!shape_ok(shape)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!x_dev || !aligned16(x_dev) || !weights_ok(experts) || !plan_ok(plan) || !y_slots_dev)
    return MOE_ERR_INVALID_ARG;
  if (shape->n_shared && !weights_ok(shared)) return MOE_ERR_INVALID_ARG;
  MOE_TRY(check_ws(shape, ws_dev, ws_bytes));
  return run_ffn(shape, x_dev, experts, shared, plan, y_slots_dev,
                 static_cast<uint8_t*>(ws_dev), (cudaStream_t)stream);
}

moe_status_t moe_combine(const moe_shape_t* shape, const void* y_slots_dev,
                         const int32_t* row_pos_dev, const float* topk_w_dev, void* y_dev,
                         void* x_next_dev, moe_stream_t stream) {
  if (!shape_ok(shape)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!y_slots_dev || !row_pos_dev || !topk_w_dev || !y_dev) return MOE_ERR_INVALID_ARG;
  if (!aligned16(y_slots_dev) || !aligned16(y_dev) || (x_next_dev && !aligned16(x_next_dev)))
    return MOE_ERR_INVALID_ARG;
  cudaError_t e = launch_combine(static_cast<const uint16_t*>(y_slots_dev), row_pos_dev,
                                 topk_w_dev, shape->T, shape->H, shape->K, shape->n_shared,
                                 static_cast<uint16_t*>(y_dev),
                                 static_cast<uint16_t*>(x_next_dev), (cudaStream_t)stream);
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "moe_combine launch");
}

moe_status_t moe_layer_w4(const moe_shape_t* shape, const void* x_dev, const void* w_router_dev,
                          const float* router_bias_dev, const moe_w4_weights_t* experts,
                          const moe_w4_weights_t* shared, void* y_dev, void* x_next_dev,
                          int32_t* topk_ids_dev, float* topk_w_dev, void* ws_dev,
                          size_t ws_bytes, moe_stream_t stream) {
  if (!shape_ok(shape)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!x_dev || !w_router_dev || !y_dev || !aligned16(x_dev) || !aligned16(w_router_dev) ||
      !aligned16(y_dev) || !weights_ok(experts))
    return MOE_ERR_INVALID_ARG;
  if (x_next_dev && !aligned16(x_next_dev)) return MOE_ERR_INVALID_ARG;
  if (shape->n_shared && !weights_ok(shared)) return MOE_ERR_INVALID_ARG;
  MOE_TRY(check_ws(shape, ws_dev, ws_bytes));
  uint8_t* ws = static_cast<uint8_t*>(ws_dev);
  const Layout L = layout_of(shape);
  int32_t* ids = topk_ids_dev ? topk_ids_dev : reinterpret_cast<int32_t*>(ws + L.ids);
  float* w = topk_w_dev ? topk_w_dev : reinterpret_cast<float*>(ws + L.w);
  moe_plan_t plan;
  plan.counts_dev = reinterpret_cast<int32_t*>(ws + L.counts);
  plan.offsets_dev = reinterpret_cast<int32_t*>(ws + L.offsets);
  plan.sorted_rows_dev = reinterpret_cast<int32_t*>(ws + L.sorted);
  plan.row_pos_dev = reinterpret_cast<int32_t*>(ws + L.rowpos);
  plan.block_map_dev = reinterpret_cast<int32_t*>(ws + L.bmap);
  plan.num_blocks_dev = reinterpret_cast<int32_t*>(ws + L.nblk);
  void* y_slots = ws + L.yslots;
  cudaStream_t st = (cudaStream_t)stream;
  int grid = 0;
  size_t smem = 0;
  if (persist_config(shape->T, shape->H, shape->E, shape->K, shape->I, shape->n_shared, &grid,
                     &smem)) {
    moe_layer_weights_t lw;
    lw.w_router_dev = w_router_dev;
    lw.router_bias_dev = router_bias_dev;
    lw.experts = *experts;
    lw.shared = shape->n_shared ? *shared : *experts;
    return decode_persistent(shape, 1, &lw, x_dev, y_dev, x_next_dev, ids, w, ws, L, grid, smem,
                             st);
  }
  if (decode_supported(shape->T, shape->H, shape->E, shape->K, shape->I, shape->n_shared)) {
    DecodeArgs d = decode_args(shape, w_router_dev, router_bias_dev, experts, shared, ws, L);
    d.x = static_cast<const uint16_t*>(x_dev);
    d.ids = ids;
    d.w = w;
    d.y = static_cast<uint16_t*>(y_dev);
    d.x_next = static_cast<uint16_t*>(x_next_dev);
    cudaError_t e = launch_decode_layer(d, st);
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "decode layer launch");
  }
  if (route_tc_supported(shape->T, shape->H, shape->E, shape->K)) {
    // moe_route + moe_plan with the plan's histogram counted by the router's
    // screen: one launch fewer, the same ids, weights and plan
    int32_t* hist = reinterpret_cast<int32_t*>(ws + L.hist);
    MOE_TRY(route_tc(shape, x_dev, w_router_dev, router_bias_dev, ids, w, ws, L, st, hist));
    cudaError_t e = launch_plan(ids, shape->T, shape->K, shape->E, shape->n_shared,
                                shape->tile_rows, plan, hist, reinterpret_cast<Ctrl*>(ws + L.ctrl),
                                kPlanChunk, st, true);
    if (e != cudaSuccess) return cuda_fail(e, "moe_plan launch");
  } else {
    MOE_TRY(moe_route(shape, x_dev, w_router_dev, router_bias_dev, ids, w, ws_dev, ws_bytes,
                      stream));
    MOE_TRY(moe_plan(shape, ids, &plan, ws_dev, ws_bytes, stream));
  }
  MOE_TRY(run_ffn(shape, x_dev, experts, shared, &plan, y_slots, ws, st));
  return moe_combine(shape, y_slots, plan.row_pos_dev, w, y_dev, x_next_dev, stream);
}

moe_status_t moe_decoder_blocks(const moe_shape_t* shape, int32_t n_layers,
                              const moe_layer_weights_t* layers_host,
                              const void* const* gains_host, const void* h_in_dev,
                              const int32_t* token_ids_dev, const void* embed_dev, int32_t vocab,
                              void* h_out_dev, void* ws_dev, size_t ws_bytes,
                              moe_stream_t stream) {
  if (!shape_ok(shape)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (n_layers < 1 || !layers_host || !gains_host || !h_out_dev || !aligned16(h_out_dev))
    return MOE_ERR_INVALID_ARG;
  if (token_ids_dev) {
    if (!embed_dev || !aligned16(embed_dev) || vocab < 1) return MOE_ERR_INVALID_ARG;
  } else if (!h_in_dev || !aligned16(h_in_dev)) {
    return MOE_ERR_INVALID_ARG;
  }
  for (int l = 0; l < n_layers; ++l) {
    const moe_layer_weights_t& lw = layers_host[l];
    if (!lw.w_router_dev || !aligned16(lw.w_router_dev) || !weights_ok(&lw.experts))
      return MOE_ERR_INVALID_ARG;
    if (shape->n_shared && !weights_ok(&lw.shared)) return MOE_ERR_INVALID_ARG;
    if (!gains_host[l] || !aligned16(gains_host[l])) return MOE_ERR_INVALID_ARG;
  }
  MOE_TRY(check_ws(shape, ws_dev, ws_bytes));
  uint8_t* ws = static_cast<uint8_t*>(ws_dev);
  const Layout L = layout_of(shape);
  cudaStream_t st = (cudaStream_t)stream;
  int grid = 0;
  size_t smem = 0;
  if (persist_config(shape->T, shape->H, shape->E, shape->K, shape->I, shape->n_shared, &grid,
                     &smem, true))
    return decoder_blocks_persistent(shape, n_layers, layers_host, gains_host, h_in_dev,
                                     token_ids_dev, embed_dev, vocab, h_out_dev, ws, L, grid,
                                     smem, st);
  // more tokens: per layer the four calls, the pre-norm of the next layer and
  // the residual add fused into the combine
  const size_t TH = (size_t)shape->T * shape->H;
  uint16_t* hb[2] = {reinterpret_cast<uint16_t*>(ws + L.blk),
                     reinterpret_cast<uint16_t*>(ws + L.blk) + TH};
  uint16_t* x = reinterpret_cast<uint16_t*>(ws + L.blk) + 2 * TH;
  Ctrl* ctrl = reinterpret_cast<Ctrl*>(ws + L.ctrl);
  const uint16_t* h = token_ids_dev ? hb[0] : static_cast<const uint16_t*>(h_in_dev);
  cudaError_t e = launch_block_input(
      static_cast<const uint16_t*>(h_in_dev), token_ids_dev,
      static_cast<const uint16_t*>(embed_dev), vocab, static_cast<const uint16_t*>(gains_host[0]),
      shape->T, shape->H, token_ids_dev ? hb[0] : nullptr, x, ctrl, st);
  if (e != cudaSuccess) return cuda_fail(e, "decoder block input launch");
  int32_t* ids = reinterpret_cast<int32_t*>(ws + L.ids);
  float* w = reinterpret_cast<float*>(ws + L.w);
  moe_plan_t plan;
  plan.counts_dev = reinterpret_cast<int32_t*>(ws + L.counts);
  plan.offsets_dev = reinterpret_cast<int32_t*>(ws + L.offsets);
  plan.sorted_rows_dev = reinterpret_cast<int32_t*>(ws + L.sorted);
  plan.row_pos_dev = reinterpret_cast<int32_t*>(ws + L.rowpos);
  plan.block_map_dev = reinterpret_cast<int32_t*>(ws + L.bmap);
  plan.num_blocks_dev = reinterpret_cast<int32_t*>(ws + L.nblk);
  void* y_slots = ws + L.yslots;
  for (int l = 0; l < n_layers; ++l) {
    const moe_layer_weights_t& lw = layers_host[l];
    const bool last = l == n_layers - 1;
    MOE_TRY(moe_route(shape, x, lw.w_router_dev, lw.router_bias_dev, ids, w, ws_dev, ws_bytes,
                      stream));
    MOE_TRY(moe_plan(shape, ids, &plan, ws_dev, ws_bytes, stream));
    MOE_TRY(run_ffn(shape, x, &lw.experts, &lw.shared, &plan, y_slots, ws, st));
    // the next residual buffer: never the one this layer reads
    uint16_t* hn = last ? static_cast<uint16_t*>(h_out_dev) : (h == hb[0] ? hb[1] : hb[0]);
    e = launch_combine(static_cast<const uint16_t*>(y_slots), plan.row_pos_dev, w, shape->T,
                       shape->H, shape->K, shape->n_shared, nullptr, last ? nullptr : x, st, h, hn,
                       last ? nullptr : static_cast<const uint16_t*>(gains_host[l + 1]));
    if (e != cudaSuccess) return cuda_fail(e, "decoder block combine launch");
    h = hn;
  }
  return MOE_OK;
}

moe_status_t moe_gdn_scan(const moe_gdn_shape_t* shape, const void* q_dev, const void* k_dev,
                          const void* v_dev, const float* alpha_dev, const float* beta_dev,
                          const float* state_in_dev, float* state_out_dev, void* o_dev,
                          moe_stream_t stream) {
  if (!gdn_supported(shape)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!q_dev || !k_dev || !v_dev || !alpha_dev || !beta_dev || !state_in_dev || !state_out_dev ||
      !o_dev || !aligned16(q_dev) || !aligned16(k_dev) || !aligned16(v_dev) ||
      !aligned16(state_in_dev) || !aligned16(state_out_dev) || !aligned16(o_dev))
    return MOE_ERR_INVALID_ARG;
  cudaError_t e = launch_gdn_scan(
      shape, static_cast<const uint16_t*>(q_dev), static_cast<const uint16_t*>(k_dev),
      static_cast<const uint16_t*>(v_dev), alpha_dev, beta_dev, state_in_dev, state_out_dev,
      static_cast<uint16_t*>(o_dev), (cudaStream_t)stream);
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "gated delta scan launch");
}

size_t moe_gdn_chunked_workspace_bytes(const moe_gdn_shape_t* shape) {
  if (!gdn_supported(shape) || shape->dv > 128) return 0;
  return gdn_chunk_ws_bytes(shape);
}

moe_status_t moe_gdn_chunked_scan(const moe_gdn_shape_t* shape, const void* q_dev,
                                  const void* k_dev, const void* v_dev, const float* alpha_dev,
                                  const float* beta_dev, const float* state_in_dev,
                                  float* state_out_dev, void* o_dev, void* ws_dev,
                                  size_t ws_bytes, moe_stream_t stream) {
  if (!gdn_supported(shape) || shape->dv > 128) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!q_dev || !k_dev || !v_dev || !alpha_dev || !beta_dev || !state_in_dev || !state_out_dev ||
      !o_dev || !ws_dev || !aligned16(q_dev) || !aligned16(k_dev) || !aligned16(v_dev) ||
      !aligned16(state_in_dev) || !aligned16(state_out_dev) || !aligned16(o_dev) ||
      !aligned16(ws_dev))
    return MOE_ERR_INVALID_ARG;
  if (ws_bytes < gdn_chunk_ws_bytes(shape)) return MOE_ERR_WORKSPACE;
  cudaError_t e = launch_gdn_chunked(
      shape, static_cast<const uint16_t*>(q_dev), static_cast<const uint16_t*>(k_dev),
      static_cast<const uint16_t*>(v_dev), alpha_dev, beta_dev, state_in_dev, state_out_dev,
      static_cast<uint16_t*>(o_dev), static_cast<float*>(ws_dev), (cudaStream_t)stream);
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "chunked gated delta scan launch");
}

size_t moe_attn_workspace_bytes(const moe_attn_shape_t* shape) {
  if (!attn_supported(shape)) return 0;
  return 256 + attn_part_floats(shape) * 4;
}

moe_status_t moe_attn_decode(const moe_attn_shape_t* shape, const void* q_dev,
                             const void* k_cache_dev, const void* v_cache_dev,
                             const int32_t* table_dev, int32_t n_phys, void* o_dev, void* ws_dev,
                             size_t ws_bytes, moe_stream_t stream) {
  if (!attn_supported(shape)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!q_dev || !k_cache_dev || !v_cache_dev || !table_dev || !o_dev || n_phys < 1 ||
      !aligned16(q_dev) || !aligned16(k_cache_dev) || !aligned16(v_cache_dev) ||
      !aligned16(o_dev))
    return MOE_ERR_INVALID_ARG;
  if (!ws_dev || ws_bytes < moe_attn_workspace_bytes(shape)) return MOE_ERR_WORKSPACE;
  if ((int64_t)n_phys * shape->n_kv * shape->block >= INT32_MAX) return MOE_ERR_INVALID_ARG;
  int nsm = 0;
  MOE_TRY(sm_count(&nsm));
  uint8_t* ws = static_cast<uint8_t*>(ws_dev);
  // the caches as [n_phys * n_kv * block rows][D]: boxes of 64 rows x 64 elements
  const uint64_t rows = (uint64_t)n_phys * shape->n_kv * shape->block;
  CUtensorMap tk, tv;
  MOE_TRY(map_2d(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, k_cache_dev, shape->D, rows, 64, 64,
                 CU_TENSOR_MAP_SWIZZLE_128B));
  MOE_TRY(map_2d(&tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, v_cache_dev, shape->D, rows, 64, 64,
                 CU_TENSOR_MAP_SWIZZLE_128B));
  cudaError_t e = launch_attn_decode(
      shape, tk, tv, static_cast<const uint16_t*>(q_dev), table_dev, n_phys,
      static_cast<uint16_t*>(o_dev), reinterpret_cast<float*>(ws + 256),
      reinterpret_cast<Ctrl*>(ws), nsm, (cudaStream_t)stream);
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "attention launch");
}

moe_status_t moe_decode_layers(const moe_shape_t* shape, int32_t n_layers,
                               const moe_layer_weights_t* layers_host, const void* x_dev,
                               void* y_dev, void* x_next_dev, void* ws_dev, size_t ws_bytes,
                               moe_stream_t stream) {
  if (!shape_ok(shape) ||
      !decode_supported(shape->T, shape->H, shape->E, shape->K, shape->I, shape->n_shared))
    return MOE_ERR_UNSUPPORTED_SHAPE;
  if (n_layers < 1 || !layers_host || !x_dev || !y_dev || !aligned16(x_dev) || !aligned16(y_dev) ||
      (x_next_dev && !aligned16(x_next_dev)))
    return MOE_ERR_INVALID_ARG;
  for (int l = 0; l < n_layers; ++l) {
    const moe_layer_weights_t& lw = layers_host[l];
    if (!lw.w_router_dev || !aligned16(lw.w_router_dev) || !weights_ok(&lw.experts))
      return MOE_ERR_INVALID_ARG;
    if (shape->n_shared && !weights_ok(&lw.shared)) return MOE_ERR_INVALID_ARG;
  }
  MOE_TRY(check_ws(shape, ws_dev, ws_bytes));
  uint8_t* ws = static_cast<uint8_t*>(ws_dev);
  const Layout L = layout_of(shape);
  int grid = 0;
  size_t smem = 0;
  if (persist_config(shape->T, shape->H, shape->E, shape->K, shape->I, shape->n_shared, &grid,
                     &smem))
    return decode_persistent(shape, n_layers, layers_host, x_dev, y_dev, x_next_dev, nullptr,
                             nullptr, ws, L, grid, smem, (cudaStream_t)stream);
  float* part[2] = {reinterpret_cast<float*>(ws + L.part), reinterpret_cast<float*>(ws + L.part2)};
  uint16_t* ybuf[2] = {reinterpret_cast<uint16_t*>(ws + L.ybuf),
                       reinterpret_cast<uint16_t*>(ws + L.ybuf) + (size_t)shape->T * shape->H};
  const int nb = (int)(decode_part_floats(shape->T, shape->H) / shape->T);
  for (int l = 0; l < n_layers; ++l) {
    const moe_layer_weights_t& lw = layers_host[l];
    DecodeArgs d = decode_args(shape, lw.w_router_dev, lw.router_bias_dev, &lw.experts,
                               &lw.shared, ws, L);
    if (l == 0) {
      d.x = static_cast<const uint16_t*>(x_dev);
    } else {
      d.y_prev = ybuf[(l - 1) & 1];
      d.part_prev = part[(l - 1) & 1];
      d.nb_prev = nb;
    }
    const bool last = l == n_layers - 1;
    d.y = last ? static_cast<uint16_t*>(y_dev) : ybuf[l & 1];
    d.part = part[l & 1];
    d.x_next = last ? static_cast<uint16_t*>(x_next_dev) : nullptr;
    d.has_next = last ? 0 : 1;
    cudaError_t e = launch_decode_layer(d, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "decode layer launch");
  }
  return MOE_OK;
}

moe_status_t moe_query_device_status(void* ws_dev, size_t ws_bytes, moe_stream_t stream) {
  if (!ws_dev || ws_bytes < sizeof(Ctrl)) return MOE_ERR_INVALID_ARG;
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  int word[4] = {0, 0, 0, 0};
  e = cudaMemcpy(word, ws_dev, sizeof(word), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "status read");
  if (word[0] != 0) {
    g_last_error = "device error " + std::to_string(word[0]) + " in kernel " +
                   std::to_string(word[1]) + " block " + std::to_string(word[2]) + " detail " +
                   std::to_string(word[3]);
    e = cudaMemset(ws_dev, 0, sizeof(word));
    if (e != cudaSuccess) return cuda_fail(e, "status clear");
    return (moe_status_t)word[0];
  }
  return MOE_OK;
}

moe_status_t moe_debug_dequant_w4(const uint32_t* q_dev, const uint16_t* s_dev,
                                  const uint16_t* b_dev, uint16_t* out_dev, int32_t N,
                                  int32_t Kd, moe_stream_t stream) {
  if (!q_dev || !s_dev || !b_dev || !out_dev || N < 1 || Kd < 64 || Kd % 64 != 0)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(out_dev) || (int64_t)N * Kd >= INT32_MAX) return MOE_ERR_INVALID_ARG;
  cudaError_t e = launch_dequant(q_dev, s_dev, b_dev, out_dev, N, Kd, false, (cudaStream_t)stream);
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "moe_debug_dequant_w4 launch");
}

moe_status_t moe_debug_dequant_w4_decode(const uint32_t* q_dev, const uint16_t* s_dev,
                                         const uint16_t* b_dev, uint16_t* out_dev, int32_t N,
                                         int32_t Kd, moe_stream_t stream) {
  if (!q_dev || !s_dev || !b_dev || !out_dev || N < 1 || Kd < 64 || Kd % 64 != 0)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(out_dev) || (int64_t)N * Kd >= INT32_MAX) return MOE_ERR_INVALID_ARG;
  cudaError_t e = launch_dequant(q_dev, s_dev, b_dev, out_dev, N, Kd, true, (cudaStream_t)stream);
  return e == cudaSuccess ? MOE_OK : cuda_fail(e, "moe_debug_dequant_w4_decode launch");
}

const char* moe_status_string(moe_status_t status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case MOE_ERR_WORKSPACE: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_BAD_INPUT: return "bad input on device (expert id out of range)";
    case MOE_ERR_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

const char* moe_last_error(void) { return g_last_error.c_str(); }

}  // extern "C"
