/*
 * moe_w4.h - C ABI of the W4A16 Mixture-of-Experts expert layer for GB300
 * (sm_103a): GPU-resident routing and grouped 4-bit-weight GEMMs.
 *
 * The operations follow the announcement "Perplexity Open Sources Lily: A
 * Rust + Metal Inference Engine for Qwen3.6-35B-A3B on Apple Silicon"
 * (abbreviated [Lily] below), sections "Three Workload Shapes" (a router
 * scores 256 experts and picks eight, plus one shared expert that sees every
 * token), "Prefill: Keep Weights Packed, Keep Routing on the GPU" (groupwise
 * affine 4-bit weights, 64 per group with a bf16 scale and bias, rebuilt to
 * bf16 one tile at a time inside the grouped GEMM with FP32 accumulation;
 * routing histogram, prefix scan, scatter and block map kept on the GPU with
 * no CPU synchronisation inside the layer) and "Decode: Minimize Bytes Moved
 * Per Token" (batch-1 decode is bandwidth bound).
 *
 * Conventions for every call:
 *  - Pointers named *_dev are device pointers owned by the caller; the
 *    library never allocates, frees or keeps them. Host pointers are only
 *    read during the call. bf16 tensors are passed as raw 16-bit patterns.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream) and never synchronise it, so they can be captured in a
 *    CUDA graph. The device that is current when a call is made must own all
 *    device pointers of that call.
 *  - Kernels (all but those of the moe_debug_* calls) are launched with
 *    programmatic stream serialisation, the cooperative ones included: a
 *    kernel may be placed on the device while the work before it in the
 *    stream finishes, but it reads no data before the work that wrote it
 *    has completed and writes nothing before the work before it has
 *    completed. To the caller the stream order is unchanged.
 *  - Argument and shape errors are returned before anything is enqueued.
 *    A failed launch returns MOE_ERR_CUDA (text in moe_last_error()).
 *    Errors found on the device (an expert id out of range, a bounded wait
 *    that ran out) are recorded in the workspace's status word and the
 *    kernel returns early; they surface through moe_query_device_status().
 *  - The workspace is caller-owned device memory of at least
 *    moe_workspace_bytes() bytes, 256-byte aligned, zero-filled once before
 *    first use (moe_workspace_init). Calls that share a workspace must be
 *    ordered (same stream, or events); separate workspaces make calls
 *    independent.
 *  - Supported shapes: 1 <= T, H % 256 == 0, I % 128 == 0, 1 <= K <= E <= 1024,
 *    K <= 32, n_shared in {0, 1}, 1 <= tile_rows <= 128, and every row /
 *    element count fits in int32.
 */
#ifndef MOE_W4_H
#define MOE_W4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream_t; /* same type as cudaStream_t */

typedef enum moe_status {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,       /* null pointer, misaligned pointer, bad flag */
  MOE_ERR_UNSUPPORTED_SHAPE = 2, /* shape outside the supported set above */
  MOE_ERR_WORKSPACE = 3,         /* workspace smaller than moe_workspace_bytes() */
  MOE_ERR_CUDA = 4,              /* a CUDA runtime/driver call failed */
  MOE_ERR_BAD_INPUT = 5,         /* device: an expert id outside [0, E) */
  MOE_ERR_TIMEOUT = 6            /* device: a bounded wait ran out */
} moe_status_t;

/* Layer shape. T tokens of hidden size H; E routed experts, K selected per
 * token; expert intermediate size I (routed and shared experts alike);
 * n_shared always-on shared experts (0 or 1); tile_rows = the most rows one
 * block-map entry (one GEMM tile of tokens) may hold. */
typedef struct moe_shape {
  int32_t T, H, E, K, I, n_shared, tile_rows;
} moe_shape_t;

/* Packed 4-bit weights of n experts ([Lily] "Prefill": groupwise affine,
 * 64 weights per group along the reduction dimension, bf16 scale and bias;
 * the dequantised weight is w = bf16(scale * q + bias), q in 0..15).
 *  q_gate_up_dev  uint32 [n][2I][H/8]   rows 0..I-1: gate, rows I..2I-1: up
 *  s_gate_up_dev  bf16   [n][2I][H/64]  scale of group g = k/64
 *  b_gate_up_dev  bf16   [n][2I][H/64]  bias  of group g
 *  q_down_dev     uint32 [n][H][I/8]
 *  s_down_dev     bf16   [n][H][I/64]
 *  b_down_dev     bf16   [n][H][I/64]
 * Word w of a row holds elements k = 8w..8w+7; element 8w+i is the nibble at
 * bits 4i..4i+3 (low nibble first). All six pointers 16-byte aligned. */
typedef struct moe_w4_weights {
  const uint32_t* q_gate_up_dev;
  const uint16_t* s_gate_up_dev;
  const uint16_t* b_gate_up_dev;
  const uint32_t* q_down_dev;
  const uint16_t* s_down_dev;
  const uint16_t* b_down_dev;
} moe_w4_weights_t;

/* Routing plan ([Lily] "Prefill": routing histogram, prefix scan, scatter,
 * block map). All device int32 buffers, caller-owned. R = T*K routed rows
 * f = t*K + k; the shared expert's rows are R..R+T-1 in token order.
 *  counts_dev      [E]      rows routed to each expert
 *  offsets_dev     [E+1]    exclusive prefix sum of counts; offsets[E] = R
 *  sorted_rows_dev [R]      routed rows in expert-contiguous order, ascending
 *                           f within an expert (stable)
 *  row_pos_dev     [R]      inverse: sorted_rows[row_pos[f]] = f
 *  block_map_dev   [moe_max_blocks() * 3]  entries (expert, row_start, nrows):
 *                           for e ascending, tiles of at most tile_rows rows
 *                           over [offsets[e], offsets[e+1]); then, with a
 *                           shared expert, entries (E, R + r0, nrows) over the
 *                           T shared rows. Entries past num_blocks are unused.
 *  num_blocks_dev  [1]      entries written (device-side; never read back) */
typedef struct moe_plan {
  int32_t* counts_dev;
  int32_t* offsets_dev;
  int32_t* sorted_rows_dev;
  int32_t* row_pos_dev;
  int32_t* block_map_dev;
  int32_t* num_blocks_dev;
} moe_plan_t;

/* Bytes of workspace every call below needs for `shape` (all calls of one
 * shape can share one workspace). 0 if the shape is unsupported. */
size_t moe_workspace_bytes(const moe_shape_t* shape);

/* Upper bound on block-map entries: ceil(R/tile_rows) + min(E, R) +
 * ceil(T/tile_rows) with a shared expert. Known on the host, so grids are
 * sized without reading the device count back. 0 if unsupported. */
int32_t moe_max_blocks(const moe_shape_t* shape);

/* Zero-fill the workspace (enqueued on stream): its status word, the
 * kernels' counters and the persistent decode's tagged words. */
moe_status_t moe_workspace_init(void* ws_dev, size_t ws_bytes, moe_stream_t stream);

/* Router: logits, top-K, renormalised softmax ([Lily] "Three Workload
 * Shapes": a router scores the experts and picks the top K).
 *  x_dev           bf16 [T][H] hidden states (16-byte aligned rows)
 *  w_router_dev    bf16 [E][H] router weight
 *  router_bias_dev fp32 [E] added to each logit, or NULL
 *  topk_ids_dev    int32 [T][K] out: experts by logit descending, ties to the
 *                  lower id
 *  topk_w_dev      fp32 [T][K] out: exp(l_k - l_0) / sum_j exp(l_j - l_0)
 * The logit is fp32 in one fixed order: 32 partial sums, partial L
 * accumulating (fma, round to nearest) elements k = 8*(32j+L)+i for
 * j = 0..H/256-1, i = 0..7 from +0; partials then added pairwise at index
 * distance 16, 8, 4, 2, 1; then + bias. Bit-exact and deterministic. */
moe_status_t moe_route(const moe_shape_t* shape, const void* x_dev, const void* w_router_dev,
                       const float* router_bias_dev, int32_t* topk_ids_dev, float* topk_w_dev,
                       void* ws_dev, size_t ws_bytes, moe_stream_t stream);

/* Plan: histogram, exclusive scan, stable scatter and block map of
 * topk_ids_dev [T][K] into `plan` (layouts above). An id outside [0, E)
 * sets MOE_ERR_BAD_INPUT on the device and that item is skipped.
 * Integer work, bit-exact and deterministic. */
moe_status_t moe_plan(const moe_shape_t* shape, const int32_t* topk_ids_dev,
                      const moe_plan_t* plan, void* ws_dev, size_t ws_bytes,
                      moe_stream_t stream);

/* Expert FFNs over the plan's block map ([Lily] "Prefill": grouped GEMM that
 * rebuilds 4-bit weights to bf16 one tile at a time on chip, FP32
 * accumulation; the expanded weights never reach device memory).
 * For every routed row r of expert e (sorted order) with token t =
 * sorted_rows[r]/K, and every shared row R+t:
 *   g = x_t Wg^T, u = x_t Wu^T (fp32 accumulate), h = bf16(silu(g) * u),
 *   y_slots[row] = bf16(h Wd^T)
 *  x_dev        bf16 [T][H]
 *  experts      E routed experts' weights; shared: the shared expert's
 *               weights (n = 1) or NULL when n_shared == 0
 *  y_slots_dev  bf16 [R + T*n_shared][H] out, rows in plan order
 * h lives in the workspace. */
moe_status_t moe_expert_ffn_w4(const moe_shape_t* shape, const void* x_dev,
                               const moe_w4_weights_t* experts, const moe_w4_weights_t* shared,
                               const moe_plan_t* plan, void* y_slots_dev, void* ws_dev,
                               size_t ws_bytes, moe_stream_t stream);

/* Weighted combine back to token order:
 *   y[t] = bf16( sum_{k asc} w[t][k] * y_slots[row_pos[t*K+k]] + y_slots[R+t] )
 * in fp32, in that fixed order (shared term only with a shared expert).
 *  y_dev      bf16 [T][H] out
 *  x_next_dev bf16 [T][H] out or NULL: unit-gain RMS normalisation of the
 *             bf16 y, y / sqrt(mean(y^2) + 1e-6), the input of a stacked
 *             next layer. */
moe_status_t moe_combine(const moe_shape_t* shape, const void* y_slots_dev,
                         const int32_t* row_pos_dev, const float* topk_w_dev, void* y_dev,
                         void* x_next_dev, moe_stream_t stream);

/* The whole layer (route, plan, expert FFNs, combine) with every
 * intermediate in the workspace. Small T takes fused decode kernels that
 * stream only the selected experts' packed bytes ([Lily] "Decode").
 * Results equal the four calls above within the FFN's fp32 tolerance;
 * routing and the plan are bit-identical. Where moe_route takes its
 * tensor-core screen (T >= 64), the screen also counts the plan's per-chunk
 * expert histogram (integer atomic adds), so the plan's histogram launch is
 * skipped. topk_ids_dev / topk_w_dev may be NULL. */
moe_status_t moe_layer_w4(const moe_shape_t* shape, const void* x_dev, const void* w_router_dev,
                          const float* router_bias_dev, const moe_w4_weights_t* experts,
                          const moe_w4_weights_t* shared, void* y_dev, void* x_next_dev,
                          int32_t* topk_ids_dev, float* topk_w_dev, void* ws_dev,
                          size_t ws_bytes, moe_stream_t stream);

/* Which kernels moe_layer_w4 and moe_decode_layers run for `shape` on the
 * current device: 2 = the persistent decode kernel (T <= 4, T*H <= 8192,
 * E <= 256, I one of 128, 256, 512, 1024, K + n_shared <= 33, and one block
 * of 512 threads with the shape's shared memory fits an SM), 1 = the three
 * decode kernels per layer (the same limits but T*H*2 + 10240 <= 49152 in
 * place of T*H <= 8192, when the persistent kernel does not fit), 0 = the
 * four calls above (route, plan, grouped GEMMs, combine), -1 = unsupported
 * shape. Host only; enqueues nothing. The three decode kernels are
 * launched with programmatic stream serialisation: a layer may start while
 * the work before it in the stream finishes, but it reads nothing that
 * work writes before that work has completed. */
int32_t moe_layer_path(const moe_shape_t* shape);

/* One stacked layer's weights for moe_decode_layers. */
typedef struct moe_layer_weights {
  const void* w_router_dev;       /* bf16 [E][H] */
  const float* router_bias_dev;   /* fp32 [E] or NULL */
  moe_w4_weights_t experts;       /* the E routed experts */
  moe_w4_weights_t shared;        /* the shared expert (ignored when n_shared == 0) */
} moe_layer_weights_t;

/* n_layers stacked layers for a few tokens ([Lily] "Decode": the kernel
 * chain of a decode step, with nothing leaving the GPU between layers).
 * Layer 0 takes x_dev; layer l > 0 takes the unit-RMS normalisation of
 * layer l-1's output, bf16(y / sqrt(mean(y^2) + 1e-6)), exactly what
 * moe_layer_w4 writes to x_next, and the results are bit-identical to that
 * chain of moe_layer_w4 calls. Between layers the normalisation is folded
 * into the next layer's kernels: no intermediate x_next is written and no
 * block waits for the last one to normalise. When T <= 4, T*H <= 8192 and
 * E <= 256 and the device holds one block of 512 threads per SM with the
 * shape's shared memory, the layers run in one persistent cooperative
 * launch per 48 layers (all blocks resident; the blocks hand the layer's
 * intermediates to each other through the workspace, with bounded waits
 * that record MOE_ERR_TIMEOUT); otherwise three kernels per layer. The
 * workspace must have been zero-filled by moe_workspace_init.
 *  layers_host  host array of n_layers entries, read during the call
 *  x_dev        bf16 [T][H] input of layer 0
 *  y_dev        bf16 [T][H] output of the last layer
 *  x_next_dev   bf16 [T][H] normalised last output, or NULL
 * Requires moe_layer_path(shape) == 1 (else MOE_ERR_UNSUPPORTED_SHAPE) and
 * n_layers >= 1. Graph-capturable; allocates nothing. */
moe_status_t moe_decode_layers(const moe_shape_t* shape, int32_t n_layers,
                               const moe_layer_weights_t* layers_host, const void* x_dev,
                               void* y_dev, void* x_next_dev, void* ws_dev, size_t ws_bytes,
                               moe_stream_t stream);

/* n_layers decoder blocks around the MoE layers, for a few tokens (the
 * residual stream of a decode step; the pre-norm and residual add are the
 * plainest reading of the block around a layer of the pages' model, which
 * they name but do not spell out; the token feed follows [Lily] "Decode":
 * the sampled token id stays on the device and feeds the next step).
 * For l = 0 .. n_layers-1:
 *   x_l     = bf16(gain_l[n] * h_l[n] / sqrt(mean_n(h_l[n]^2) + 1e-6))
 *   y_l     = layer l on x_l (router, top-K, experts, combine, as
 *             moe_layer_w4 computes them)
 *   h_{l+1} = bf16(h_l + y_l)
 * h_0 = embed_dev[token_ids_dev[t]] when token_ids_dev is not NULL (the
 * tokens' embedding rows, gathered on the device, so a decode loop feeds
 * each step's token ids from device memory with no host round trip; an id
 * outside [0, vocab) is recorded as MOE_ERR_BAD_INPUT and reads as a zero
 * row), else h_in_dev. Writes h_out_dev = h_{n_layers}.
 * A few tokens (the shapes the persistent decode kernel holds) run in one
 * cooperative launch per 48 layers; more tokens run the four calls of each
 * layer, with the residual add and the next layer's pre-norm fused into the
 * combine.
 *  layers_host   n_layers host structs, as for moe_decode_layers
 *  gains_host    n_layers device pointers, each bf16 [H], 16-byte aligned
 *  h_in_dev      bf16 [T][H], or NULL when token_ids_dev is given
 *  token_ids_dev int32 [T] or NULL
 *  embed_dev     bf16 [vocab][H] (used with token_ids_dev)
 *  h_out_dev     bf16 [T][H] out; may be h_in_dev
 * The workspace is the layer's (moe_workspace_bytes), zero-filled by
 * moe_workspace_init; the last layer's ids and weights are left in it. */
moe_status_t moe_decoder_blocks(const moe_shape_t* shape, int32_t n_layers,
                              const moe_layer_weights_t* layers_host,
                              const void* const* gains_host, const void* h_in_dev,
                              const int32_t* token_ids_dev, const void* embed_dev, int32_t vocab,
                              void* h_out_dev, void* ws_dev, size_t ws_bytes,
                              moe_stream_t stream);

/* moe_plan without a workspace: same inputs, same outputs, bit-identical
 * results. The pages have no counterpart; this entry point exists for
 * callers that cannot allocate device memory where they build the plan (code
 * running inside a memory-pool or allocator callback, where allocating would
 * re-enter the allocator, or a runtime that forbids cudaMalloc after
 * start-up) and have no spare buffer to pass. Its scratch (the per-chunk
 * histograms and a status word, 256 KiB) is one static device array that
 * every GPU loading the library holds until the process exits. Limit:
 * ceil(T*K/2048) * E <= 65472, else MOE_ERR_UNSUPPORTED_SHAPE (text in
 * moe_last_error()) before anything is enqueued. The first call on a device
 * looks up that array's device address (cudaGetSymbolAddress, with the
 * device current) and caches it for the life of the process, so make that
 * call before any stream capture, and do not call this entry point on a
 * device after cudaDeviceReset there (the cached address may be stale). It
 * allocates and frees nothing. All calls share the one array: calls that can overlap on
 * the GPU (other streams, other host threads) race and must be ordered by
 * the caller. Expert ids outside [0, E) are skipped, as in moe_plan, but are
 * not reported. */
moe_status_t moe_plan_noalloc(const moe_shape_t* shape, const int32_t* topk_ids_dev,
                              const moe_plan_t* plan, moe_stream_t stream);

/* Synchronise `stream`, read and clear the workspace's device status word.
 * Returns MOE_OK, the recorded device error, or MOE_ERR_CUDA. Test and
 * debug use: it blocks the host. */
moe_status_t moe_query_device_status(void* ws_dev, size_t ws_bytes, moe_stream_t stream);

/* Dequantise a packed matrix [N][Kd] (layout as in moe_w4_weights_t) to
 * bf16 [N][Kd] with the same device routine the GEMMs use. Test use. */
moe_status_t moe_debug_dequant_w4(const uint32_t* q_dev, const uint16_t* s_dev,
                                  const uint16_t* b_dev, uint16_t* out_dev, int32_t N,
                                  int32_t Kd, moe_stream_t stream);

/* The same with the decode kernels' routine, which rebuilds elements i and
 * i+4 of each packed word as one pair; the output is put back into natural
 * element order, so it must equal moe_debug_dequant_w4's bit for bit. Same
 * arguments and errors. Test use. */
moe_status_t moe_debug_dequant_w4_decode(const uint32_t* q_dev, const uint16_t* s_dev,
                                         const uint16_t* b_dev, uint16_t* out_dev, int32_t N,
                                         int32_t Kd, moe_stream_t stream);

/* Static text of a status code; text of the last CUDA error seen by this
 * thread's calls ("" if none). */
const char* moe_status_string(moe_status_t status);
const char* moe_last_error(void);

/* ----------------------------------------------------------------------
 * Grouped-query decode attention ([Lily] "Three Workload Shapes": the
 * model's full-attention layers have 16 query heads sharing 2 key/value
 * heads; [Lily] "Decode": the query heads of a key/value head are packed so
 * each cache row is loaded once, and the cache is kept in fixed-size
 * blocks). For query token t (at position L - T + t) and head h, with
 * g = h / (n_q / n_kv):
 *   o[t][h] = sum_j softmax_j( q[t][h] . k_j / sqrt(D) ) v_j,  j <= L - T + t,
 * fp32 scores and sums, P rounded to bf16 before it multiplies V, o bf16.
 * Position j of group g is row j % block of physical block table[j / block].
 * ---------------------------------------------------------------------- */
typedef struct moe_attn_shape {
  int32_t T;      /* query tokens (1 or 2), the last T positions */
  int32_t n_q;    /* query heads */
  int32_t n_kv;   /* key/value heads; (n_q / n_kv) * T <= 16 */
  int32_t D;      /* head dimension: 64 or 128 */
  int32_t L;      /* sequence length, the T query tokens included (T <= L <= 2^24) */
  int32_t block;  /* positions per cache block: 64 */
} moe_attn_shape_t;

/* Workspace bytes of moe_attn_decode (a status word and the per-chunk
 * partials), 0 for an unsupported shape. Zero-fill it once with
 * moe_workspace_init; moe_query_device_status reads its status. */
size_t moe_attn_workspace_bytes(const moe_attn_shape_t* shape);

/* o = attention of q over the cache (definition above). Device pointers:
 *  q_dev        bf16 [T][n_q][D]
 *  k_cache_dev  bf16 [n_phys][n_kv][block][D]; v_cache_dev likewise
 *  table_dev    int32 [ceil(L / block)]: the physical block of each logical
 *               block; an entry outside [0, n_phys) is recorded as
 *               MOE_ERR_BAD_INPUT and its positions are left out
 *  o_dev        bf16 [T][n_q][D] out
 * All bf16 pointers 16-byte aligned. Errors: MOE_ERR_UNSUPPORTED_SHAPE,
 * MOE_ERR_INVALID_ARG, MOE_ERR_WORKSPACE (too small), MOE_ERR_CUDA. A wait
 * that runs out on the device (MOE_ERR_TIMEOUT from moe_query_device_status)
 * can leave the workspace's grid-barrier counter mid-count: re-initialise
 * the workspace (moe_workspace_init) before the next call. */
moe_status_t moe_attn_decode(const moe_attn_shape_t* shape, const void* q_dev,
                             const void* k_cache_dev, const void* v_cache_dev,
                             const int32_t* table_dev, int32_t n_phys, void* o_dev, void* ws_dev,
                             size_t ws_bytes, moe_stream_t stream);

/* ----------------------------------------------------------------------
 * The Gated DeltaNet recurrence ([Lily] "Three Workload Shapes": 30 of the
 * 40 layers are Gated DeltaNet, a fixed-size recurrence; [Lily] "Prefill":
 * a register-resident scan), in the published gated delta rule: for value
 * head h (key head h / (n_v / n_k)), state S [dv][dk] and t = 0 .. T-1
 *   S <- alpha_t S (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
 *   o_t = S q_t,
 * fp32 state and arithmetic, o bf16. The q/k projections, their
 * normalisation and the gates are the caller's (inputs here).
 * ---------------------------------------------------------------------- */
typedef struct moe_gdn_shape {
  int32_t T;    /* tokens, scanned in order */
  int32_t n_k;  /* key heads */
  int32_t n_v;  /* value heads, a multiple of n_k */
  int32_t dk;   /* key dimension: 128 */
  int32_t dv;   /* value dimension: a multiple of 16 */
} moe_gdn_shape_t;

/* Device pointers:
 *  q_dev, k_dev       bf16 [T][n_k][dk]
 *  v_dev              bf16 [T][n_v][dv]
 *  alpha_dev, beta_dev fp32 [T][n_v]
 *  state_in_dev       fp32 [n_v][dv][dk]; state_out_dev likewise, may be
 *                     state_in_dev (updated in place)
 *  o_dev              bf16 [T][n_v][dv] out
 * All 16-byte aligned. Errors: MOE_ERR_UNSUPPORTED_SHAPE, MOE_ERR_INVALID_ARG,
 * MOE_ERR_CUDA. */
moe_status_t moe_gdn_scan(const moe_gdn_shape_t* shape, const void* q_dev, const void* k_dev,
                          const void* v_dev, const float* alpha_dev, const float* beta_dev,
                          const float* state_in_dev, float* state_out_dev, void* o_dev,
                          moe_stream_t stream);

/* The same rule in its chunked (parallel) form, for prompts: chunks of 64
 * tokens, each solved as a whole from the state before it (the WY / UT form
 * of the delta rule: with g_t the running product of alpha over the chunk,
 * the chunk's writes solve a unit lower-triangular system whose matrix and
 * right-hand sides depend only on the chunk's k, v, alpha and beta), so the
 * work inside a chunk runs in parallel over its tokens and only the chunks
 * follow one another. Same inputs, outputs and supported shapes as
 * moe_gdn_scan (dv <= 128 as well), results within the layer's tolerance
 * of it (fp32 sums; the products run on the tensor cores, bf16 operands
 * exact, fp32 operands split into two tf32 parts; decay ratios taken as
 * exp of differences of summed log alpha). ws_dev: device workspace of at
 * least moe_gdn_chunked_workspace_bytes(shape) bytes, 16-byte aligned,
 * caller owned: a 256-byte status header, zero-filled once before first
 * use (moe_workspace_init), then per chunk and value head the chunk's two
 * solved right-hand sides, its decay-masked q.k matrix and two decay
 * vectors (no initialisation needed). A bounded wait inside the kernels
 * that runs out is recorded in the header and surfaces through
 * moe_query_device_status(ws_dev). Errors: as moe_gdn_scan, plus
 * MOE_ERR_WORKSPACE when ws_bytes is too small. */
size_t moe_gdn_chunked_workspace_bytes(const moe_gdn_shape_t* shape);
moe_status_t moe_gdn_chunked_scan(const moe_gdn_shape_t* shape, const void* q_dev,
                                  const void* k_dev, const void* v_dev, const float* alpha_dev,
                                  const float* beta_dev, const float* state_in_dev,
                                  float* state_out_dev, void* o_dev, void* ws_dev,
                                  size_t ws_bytes, moe_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_W4_H */
