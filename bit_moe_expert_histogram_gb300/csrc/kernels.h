// Internal launch interface between the C ABI (api.cu) and the kernels.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_w4.h"

namespace moe {

struct Ctrl;

constexpr int kPlanChunk = 256;         // routed rows per plan block (workspace path)
constexpr int kPlanChunkNoalloc = 2048; // routed rows per plan block (moe_plan_noalloc)

// Arguments of one grouped W4A16 GEMM launch (gate_up or down).
struct FfnArgs {
  const int32_t* block_map;    // [max_blocks][3] (expert, row_start, nrows)
  const int32_t* num_blocks;   // device count of block-map entries
  const int32_t* sorted_rows;  // unused by the kernel (the operand rows come in plan order)
  int K;                       // experts per token
  int R;                       // routed rows (T*K)
  int E;                       // routed experts; entry expert E = shared
  int rows_per_expert;         // weight rows per expert (2I or H)
  int half_rows;               // gate_up: I (first up row); down: 0
  int mtiles;                  // unit tiles per entry (gate_up: 64 gate + 64 up rows; down: 128 rows)
  int kdim;                    // reduction length (H for gate_up, I for down)
  int kgroups;                 // 64-wide groups per weight row (Kdim / 64)
  const uint16_t* s_exp;       // [E][rows][kgroups] bf16 scales
  const uint16_t* b_exp;       // [E][rows][kgroups] bf16 biases
  const uint16_t* s_sh;        // shared expert [rows][kgroups]
  const uint16_t* b_sh;
  uint16_t* out;               // bf16 [S][out_ld]
  int out_ld;
  Ctrl* ctrl;
  int max_units;               // host bound on units
  int shared_blocks;           // block-map entries of the shared expert (the last ones)
};

// Arguments of the fused decode layer (decode.cu): every pointer device,
// ids / w / logits / h / part in the workspace or the caller's buffers.
constexpr int kDecodeMaxT = 4;  // moe_layer_w4 takes the decode kernels up to this T
struct DecodeArgs {
  const uint16_t* x;    // bf16 [T][H]
  const uint16_t* wr;   // bf16 [E][H]
  const float* bias;    // [E] or null
  int T, H, E, K, I, ns;
  moe_w4_weights_t ex;  // routed experts
  moe_w4_weights_t sh;  // shared expert (used when ns == 1)
  float* logits;        // [T][E]
  int32_t* ids;         // [T][K]
  float* w;             // [T][K]
  uint16_t* h;          // bf16 [T][K+ns][I]
  uint16_t* y;          // bf16 [T][H]
  uint16_t* x_next;     // bf16 [T][H] or null
  float* part;          // [decode_part_floats(T, H)]
  Ctrl* ctrl;
  // stacked layers (moe_decode_layers): with y_prev, the input is
  // bf16(y_prev * inv) with inv from part_prev (the previous layer's block
  // partials, nb_prev per token) instead of x; with has_next, dec_down writes
  // its block partials for the next layer
  const uint16_t* y_prev;
  const float* part_prev;
  int nb_prev;
  int has_next;
};
bool decode_supported(int T, int H, int E, int K, int I, int ns);
size_t decode_part_floats(int T, int H);
cudaError_t launch_decode_layer(const DecodeArgs& a, cudaStream_t stream);

// Persistent decode through stacked layers (decode_persist.cu): one
// cooperative launch runs up to kPersistMaxLayers layers.
constexpr int kPersistMaxLayers = 48;
struct PersistArgs {
  int T, H, E, K, I, ns, n_layers;
  const uint16_t* x;    // bf16 [T][H]: the first layer's input
  uint16_t* y;          // bf16 [T][H]: the last layer's output
  uint16_t* x_next;     // bf16 [T][H] or null: its unit-RMS normalisation
  int32_t* ids;         // [T][K]: routing of the last layer
  float* w;             // [T][K]
  // cross-block words (epoch << 32 | payload), laid out by persist_tags():
  // 16-word lines, each written by one warp
  uint64_t* logits_tag; // line t*E+e: word 0 = fp32 logit
  uint64_t* h_tag;      // line per gate_up tile: words 4 col + r = bf16 pair (h_r, h_r+4)
  uint64_t* y_tag;      // line t*(H/8)+g: words 0..3 = bf16 pairs (y_r, y_r+4), word 4 = y^2 partial
  Ctrl* ctrl;
  // decoder blocks (moe_decoder_blocks) when block != 0: layer l's input is
  // bf16(gain[l] * h_l / rms(h_l)) and its output h_{l+1} = bf16(h_l + y_l)
  // (y is then h, the residual stream; x_next must be null); h_0 is
  // embed[tok[t]] when tok is set (ids outside [0, vocab) are recorded and
  // read as zero rows), else x
  int block;
  const int32_t* tok;
  const uint16_t* embed;
  int vocab;
  const uint16_t* gain[kPersistMaxLayers];
  moe_layer_weights_t layer[kPersistMaxLayers];
};
bool persist_supported(int T, int H, int E, int K, int I, int ns);
// Word offsets of the three tagged buffers in one region, and its size.
struct PersistTags {
  size_t logits, h, y, total;
};
PersistTags persist_tags(int T, int H, int E, int K, int I, int ns);
// Grid and dynamic shared memory of a launch on the current device; false
// when the shape's blocks do not fit on it (the caller takes the per-layer
// kernels then).
// block: room for the residual stream too (decoder blocks)
bool persist_config(int T, int H, int E, int K, int I, int ns, int* grid, size_t* smem,
                    bool block = false);
cudaError_t launch_decode_persist(const PersistArgs& a, int grid, size_t smem,
                                  cudaStream_t stream);

// Tensor-core screened router (route_tc.cu), taken from this many tokens on.
constexpr int kRouteTcMinT = 64;
bool route_tc_supported(int T, int H, int E, int K);
size_t route_tc_partial_floats(int T, int H, int E);
cudaError_t launch_route_tc(const CUtensorMap& tm_w, const CUtensorMap& tm_x, const uint16_t* x,
                            const uint16_t* wr, const float* bias, int T, int H, int E, int K,
                            float* part, int32_t* ids, float* w, Ctrl* ctrl, cudaStream_t stream,
                            int32_t* hist = nullptr, int chunk = 0);

cudaError_t launch_route(const uint16_t* x, const uint16_t* wr, const float* bias, int T, int H,
                         int E, int K, float* logits, int32_t* ids, float* w,
                         cudaStream_t stream);
cudaError_t launch_plan(const int32_t* ids, int T, int K, int E, int n_shared, int BM,
                        const moe_plan_t& plan, int32_t* hist, Ctrl* ctrl, int chunk,
                        cudaStream_t stream, bool hist_ready = false);
cudaError_t launch_ffn_gate_up(const CUtensorMap& tw, const CUtensorMap& twsh,
                               const CUtensorMap& tx, const FfnArgs& a, int grid,
                               cudaStream_t stream);
cudaError_t launch_ffn_down(const CUtensorMap& tw, const CUtensorMap& twsh, const CUtensorMap& th,
                            const FfnArgs& a, int grid, cudaStream_t stream);
// xs[p] = x row of plan row p (routed rows through sorted_rows, then the
// shared expert's rows in token order), S rows of H bf16
cudaError_t launch_gather_x(const uint16_t* x, const int32_t* sorted_rows, int K, int R, int S,
                            int T, int H, uint16_t* xs, Ctrl* ctrl, int nsm, cudaStream_t stream);
// h_out set: decoder blocks (h_out = bf16(h_in + y), x_next of h_out with
// gain); y may then be null
cudaError_t launch_combine(const uint16_t* y_slots, const int32_t* row_pos, const float* w, int T,
                           int H, int K, int n_shared, uint16_t* y, uint16_t* x_next,
                           cudaStream_t stream, const uint16_t* h_in = nullptr,
                           uint16_t* h_out = nullptr, const uint16_t* gain = nullptr);
// The first decoder block's h_0 (h_in, or the embedding rows of tok copied to
// h0_out) and its input x = bf16(gain * h_0 / rms(h_0)).
cudaError_t launch_block_input(const uint16_t* h_in, const int32_t* tok, const uint16_t* embed,
                               int vocab, const uint16_t* gain, int T, int H, uint16_t* h0_out,
                               uint16_t* x, Ctrl* ctrl, cudaStream_t stream);
// decode_routine: the decode kernels' dequant_word_i4 (pairs put back into
// natural order) instead of the grouped GEMMs' dequant_word
cudaError_t launch_dequant(const uint32_t* q, const uint16_t* s, const uint16_t* b, uint16_t* out,
                           int N, int Kd, bool decode_routine, cudaStream_t stream);
// Grouped-query decode attention over a block-paged cache (attn_decode.cu).
bool attn_supported(const moe_attn_shape_t* s);
size_t attn_part_floats(const moe_attn_shape_t* s);
// tm_k / tm_v: the caches as [n_phys * n_kv * 64 rows][D] bf16, boxes of
// 64 rows x 64 elements, 128-byte swizzle
cudaError_t launch_attn_decode(const moe_attn_shape_t* s, const CUtensorMap& tm_k,
                               const CUtensorMap& tm_v, const uint16_t* q, const int32_t* table,
                               int n_phys, uint16_t* o, float* part, Ctrl* ctrl, int nsm,
                               cudaStream_t stream);
// Gated delta rule scan (gdn_scan.cu).
bool gdn_supported(const moe_gdn_shape_t* s);
cudaError_t launch_gdn_scan(const moe_gdn_shape_t* s, const uint16_t* q, const uint16_t* k,
                            const uint16_t* v, const float* alpha, const float* beta,
                            const float* s_in, float* s_out, uint16_t* o, cudaStream_t stream);
// Chunked form of the same rule (gdn_chunk.cu): workspace bytes, launch.
size_t gdn_chunk_ws_bytes(const moe_gdn_shape_t* s);
cudaError_t launch_gdn_chunked(const moe_gdn_shape_t* s, const uint16_t* q, const uint16_t* k,
                               const uint16_t* v, const float* alpha, const float* beta,
                               const float* s_in, float* s_out, uint16_t* o, float* ws,
                               cudaStream_t stream);
// Host helpers shared by the C-ABI translation units (api.cu keeps the state).
bool shape_supported(const moe_shape_t* shape);
void set_last_error(const char* text);
void set_last_cuda_error(cudaError_t e, const char* where);
int ffn_tile_m();
int ffn_max_tile_n();
int ffn_stage_k();
int ffn_b_box_rows();

}  // namespace moe
