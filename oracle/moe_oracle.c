/*
 * Plain CPU oracle of the W4A16 Mixture-of-Experts expert layer.
 *
 * TEST INFRASTRUCTURE. Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference legs of bench.py load this library. It shares no
 * code, header, table or helper with the CUDA path.
 *
 * Pages followed (all four restate one announcement):
 *   [P3] "Perplexity Open Sources Lily: A Rust + Metal Inference Engine for
 *        Qwen3.6-35B-A3B on Apple Silicon" (insight.aitobox.com), sections
 *        "Three Workload Shapes", "Prefill: Keep Weights Packed, Keep Routing
 *        on the GPU", "Decode: Minimize Bytes Moved Per Token".
 *   [P1] "Perplexity Open Sources Lily : un moteur d'inference Rust + Metal
 *        pour Qwen3.6-35B-A3B sur Apple Silicon" (cmedia.click), paragraphs
 *        on the model, on quantisation and on routing.
 *
 * What the pages fix: a router scores 256 experts and picks eight, plus one
 * shared expert that sees every token [P3 "Three Workload Shapes"]; weights
 * are groupwise-affine 4-bit, 64 weights per group sharing a bf16 scale and
 * bias, rebuilt to bf16 one tile at a time and accumulated in FP32 [P3
 * "Prefill"]; routing keeps a histogram, a prefix scan, a scatter and a
 * block map on the GPU [P3 "Prefill"]. Everything else (fp32 logit order,
 * tie-break, softmax renormalisation over the selected experts, SwiGLU,
 * weight-1 shared expert, gate/up row split, nibble order, block-map
 * format, rounding points) is the layer's workload definition or a stated
 * reading; each function below names the one it follows.
 *
 * Build: gcc -O2 -fno-fast-math -ffp-contract=off -fopenmp -shared -fPIC.
 * -ffp-contract=off matters: the router's adds must not fuse into FMAs.
 *
 * Arithmetic: fp64 everywhere except the router logit, whose fp32 order is
 * itself the definition (see orc_router_logit).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------- bf16 -- */

/* bf16 bits -> value: the bf16 pattern is the high half of an IEEE binary32. */
double orc_bf16_value(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* value -> bf16 bits, one rounding to nearest, ties to even, from the fp64
 * value (not via fp32, which would round twice). bf16 keeps 8 significant
 * bits; below 2^-126 the spacing is fixed at 2^-133 (subnormals). */
uint16_t orc_bf16_rne(double v) {
  if (isnan(v)) return 0x7FC0;
  uint16_t sign = signbit(v) ? 0x8000 : 0;
  double a = fabs(v);
  if (a == 0.0) return sign;
  if (isinf(a)) return sign | 0x7F80;
  int e;
  frexp(a, &e);               /* a = m * 2^e, m in [0.5, 1) */
  int ue = e - 8;             /* spacing of 8-significant-bit values here */
  if (ue < -133) ue = -133;
  double q = nearbyint(ldexp(a, -ue)); /* exact scaling; RNE to an integer */
  double r = ldexp(q, ue);
  if (r >= 0x1p128) return sign | 0x7F80;
  float f = (float)r;         /* exact: r has at most 9 significant bits */
  uint32_t u;
  memcpy(&u, &f, 4);
  return sign | (uint16_t)(u >> 16);
}

static float bf16_f32(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* -------------------------------------------------------------- router -- */

/* Router logit of one token against one expert row, fp32, in a fixed order.
 *
 * The pages say only that a router scores the experts [P3 "Three Workload
 * Shapes"]; they fix no precision or summation order. Reading used: fp32
 * products accumulated with correctly rounded fmaf into 32 partial sums,
 * where partial L takes elements k = 8*(32*j + L) + i for j = 0..H/256-1,
 * i = 0..7 in that order, starting from +0; the 32 partials are then
 * combined pairwise across index distance 16, 8, 4, 2, 1 (partial L
 * becomes a_L + a_{L xor d}), and the logit is partial 0. Requires
 * H % 256 == 0. */
float orc_router_logit(const uint16_t* x, const uint16_t* w, int H) {
  float a[32], b[32];
  for (int L = 0; L < 32; ++L) {
    float acc = 0.0f;
    for (int j = 0; j < H / 256; ++j)
      for (int i = 0; i < 8; ++i) {
        int k = 8 * (32 * j + L) + i;
        acc = fmaf(bf16_f32(x[k]), bf16_f32(w[k]), acc);
      }
    a[L] = acc;
  }
  for (int d = 16; d >= 1; d >>= 1) {
    for (int L = 0; L < 32; ++L) b[L] = a[L] + a[L ^ d];
    memcpy(a, b, sizeof a);
  }
  return a[0];
}

/* logits[t][e] = router logit (+ bias[e] as one fp32 add when bias != NULL). */
void orc_router_logits(const uint16_t* x, const uint16_t* w_r, const float* bias,
                       int T, int H, int E, float* logits) {
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t)
    for (int e = 0; e < E; ++e) {
      float l = orc_router_logit(x + (size_t)t * H, w_r + (size_t)e * H, H);
      if (bias) l = l + bias[e];
      logits[(size_t)t * E + e] = l;
    }
}

/* Top-K selection and renormalised softmax weights, per token.
 *
 * "a router scores 256 experts and picks eight" [P3 "Three Workload
 * Shapes"]; softmax renormalised over the selected experts is the layer's
 * workload definition. Readings: experts are ordered by logit descending,
 * ties to the lower expert id, compared by value (so -0 == +0); slot k
 * holds the k-th expert of that order. Selection is made on the logits
 * (softmax is monotone, so the set is the same in exact arithmetic).
 * w_k = exp(l_k - l_0) / sum_j exp(l_j - l_0), in fp64. */
void orc_topk(const float* logits, int T, int E, int K, int32_t* ids,
              float* w32, double* w64) {
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t) {
    const float* l = logits + (size_t)t * E;
    int sel[1024];
    for (int k = 0; k < K; ++k) {
      int best = -1;
      for (int e = 0; e < E; ++e) {
        int taken = 0;
        for (int j = 0; j < k; ++j) taken |= (sel[j] == e);
        if (taken) continue;
        if (best < 0 || l[e] > l[best]) best = e; /* strict: lower id keeps ties */
      }
      sel[k] = best;
    }
    double z = 0.0, ex[1024];
    for (int k = 0; k < K; ++k) {
      ex[k] = exp((double)l[sel[k]] - (double)l[sel[0]]);
      z += ex[k];
    }
    for (int k = 0; k < K; ++k) {
      ids[(size_t)t * K + k] = sel[k];
      if (w32) w32[(size_t)t * K + k] = (float)(ex[k] / z);
      if (w64) w64[(size_t)t * K + k] = ex[k] / z;
    }
  }
}

/* ---------------------------------------------------------------- plan -- */

/* Histogram, exclusive scan, stable scatter and block map [P3 "Prefill":
 * routing histogram, prefix scan, scatter and block map].
 *
 * Items are f = t*K + k (routed slot rows), R = T*K of them.
 *   counts[e]      = #{f : ids[f] == e}
 *   offsets[e]     = sum_{e' < e} counts[e'],  offsets[E] = R
 *   sorted_rows[p] = f, scattered in ascending f (stable), row_pos[f] = p
 *   block map      = for e ascending, rows [offsets[e] + r0, + min(BM, counts[e]-r0))
 *                    as triples (e, offsets[e] + r0, nrows), r0 = 0, BM, ...;
 *                    then, when n_shared == 1, triples (E, R + r0, nrows) over
 *                    the T shared rows (token order).
 * Returns the number of blocks, or -1 if an id is out of [0, E) or the map
 * would exceed max_blocks. */
int orc_plan(const int32_t* ids, int T, int E, int K, int n_shared, int BM,
             int32_t* counts, int32_t* offsets, int32_t* sorted_rows,
             int32_t* row_pos, int32_t* block_map, int max_blocks) {
  int R = T * K;
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (int f = 0; f < R; ++f) {
    if (ids[f] < 0 || ids[f] >= E) return -1;
    counts[ids[f]]++;
  }
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  int32_t* cur = (int32_t*)malloc(sizeof(int32_t) * (size_t)E);
  for (int e = 0; e < E; ++e) cur[e] = offsets[e];
  for (int f = 0; f < R; ++f) {
    int p = cur[ids[f]]++;
    sorted_rows[p] = f;
    row_pos[f] = p;
  }
  free(cur);
  int nb = 0;
  for (int e = 0; e < E; ++e)
    for (int r0 = 0; r0 < counts[e]; r0 += BM) {
      if (nb >= max_blocks) return -1;
      int n = counts[e] - r0 < BM ? counts[e] - r0 : BM;
      block_map[3 * nb + 0] = e;
      block_map[3 * nb + 1] = offsets[e] + r0;
      block_map[3 * nb + 2] = n;
      nb++;
    }
  if (n_shared)
    for (int r0 = 0; r0 < T; r0 += BM) {
      if (nb >= max_blocks) return -1;
      int n = T - r0 < BM ? T - r0 : BM;
      block_map[3 * nb + 0] = E;
      block_map[3 * nb + 1] = R + r0;
      block_map[3 * nb + 2] = n;
      nb++;
    }
  return nb;
}

/* ------------------------------------------------------------- dequant -- */

/* Groupwise-affine 4-bit dequantisation [P3 "Prefill"; P1 paragraph on
 * quantisation: 64 weights per group share a bf16 scale and bias].
 * Matrix [N][Kd]: q[n][k] is nibble k%8 (bits 4*(k%8)..+3, low nibble first)
 * of word qw[n][k/8]; group g = k/64 has scale s[n][g] and bias b[n][g].
 * w = RNE_bf16(s*q + b). The fp64 sum s*q + b is exact whenever the two
 * terms' exponents differ by less than 40; otherwise the small term is far
 * below half a bf16 step of the large one and cannot move the rounding, so
 * the result equals rounding the exact value once. */
uint16_t orc_dequant_one(const uint32_t* qw, const uint16_t* s, const uint16_t* b,
                         int Kd, int n, int k) {
  uint32_t word = qw[(size_t)n * (Kd / 8) + k / 8];
  int q = (int)((word >> (4 * (k % 8))) & 15u);
  double sv = orc_bf16_value(s[(size_t)n * (Kd / 64) + k / 64]);
  double bv = orc_bf16_value(b[(size_t)n * (Kd / 64) + k / 64]);
  return orc_bf16_rne(sv * (double)q + bv);
}

void orc_dequant(const uint32_t* qw, const uint16_t* s, const uint16_t* b, int N,
                 int Kd, uint16_t* out) {
#pragma omp parallel for schedule(static)
  for (int n = 0; n < N; ++n)
    for (int k = 0; k < Kd; ++k)
      out[(size_t)n * Kd + k] = orc_dequant_one(qw, s, b, Kd, n, k);
}

/* ----------------------------------------------------------------- FFN -- */

/* One expert's SwiGLU FFN on one bf16 input row, fp64 accumulation.
 * Weights are the dequantised bf16 values (as doubles) of
 *   gate_up [2I][H]: rows 0..I-1 gate, rows I..2I-1 up (concatenated),
 *   down    [H][I].
 * g_j = sum_k x_k*Wg[j][k], u_j = sum_k x_k*Wu[j][k] (k ascending),
 * h_j = RNE_bf16(silu(g_j)*u_j), silu(g) = g/(1+exp(-g)),
 * d_n = sum_j h_j*Wd[n][j] (j ascending).
 * FP32-or-better accumulation and bf16 weights/activations into the
 * contraction follow [P3 "Prefill"]; SwiGLU and the gate/up split are the
 * layer's workload definition; h is rounded to bf16 because the second
 * contraction takes bf16 operands, as the first does. */
static void ffn_row(const double* wgu, const double* wd, const double* x, int H,
                    int I, uint16_t* h_out, double* d_out) {
  double* h = (double*)malloc(sizeof(double) * (size_t)I);
  for (int j = 0; j < I; ++j) {
    const double* rg = wgu + (size_t)j * H;
    const double* ru = wgu + (size_t)(I + j) * H;
    double g = 0.0, u = 0.0;
    for (int k = 0; k < H; ++k) {
      g += x[k] * rg[k];
      u += x[k] * ru[k];
    }
    double a = g / (1.0 + exp(-g)) * u;
    uint16_t hb = orc_bf16_rne(a);
    if (h_out) h_out[j] = hb;
    h[j] = orc_bf16_value(hb);
  }
  for (int n = 0; n < H; ++n) {
    const double* r = wd + (size_t)n * I;
    double acc = 0.0;
    for (int j = 0; j < I; ++j) acc += h[j] * r[j];
    d_out[n] = acc;
  }
  free(h);
}

/* Dequantised matrix as doubles. Every weight of group g of row n is one of
 * the 16 values RNE_bf16(s*q + b), q = 0..15, so the group's 16 values are
 * formed once (orc_dequant_one's arithmetic) and selected by the nibble. */
static double* expand(const uint32_t* qw, const uint16_t* s, const uint16_t* b,
                      int N, int Kd) {
  double* w = (double*)malloc(sizeof(double) * (size_t)N * Kd);
  for (int n = 0; n < N; ++n)
    for (int g = 0; g < Kd / 64; ++g) {
      double sv = orc_bf16_value(s[(size_t)n * (Kd / 64) + g]);
      double bv = orc_bf16_value(b[(size_t)n * (Kd / 64) + g]);
      double tab[16];
      for (int q = 0; q < 16; ++q) tab[q] = orc_bf16_value(orc_bf16_rne(sv * (double)q + bv));
      for (int k = 64 * g; k < 64 * g + 64; ++k) {
        uint32_t word = qw[(size_t)n * (Kd / 8) + k / 8];
        w[(size_t)n * Kd + k] = tab[(word >> (4 * (k % 8))) & 15u];
      }
    }
  return w;
}

/* Expert FFN for `nrows` input rows of one expert.
 * x_rows: bf16 [nrows][H]; h_out: bf16 [nrows][I] or NULL; d_out: fp64 [nrows][H]. */
void orc_expert_ffn(const uint32_t* q_gu, const uint16_t* s_gu, const uint16_t* b_gu,
                    const uint32_t* q_d, const uint16_t* s_d, const uint16_t* b_d,
                    int H, int I, const uint16_t* x_rows, int nrows,
                    uint16_t* h_out, double* d_out) {
  double* wgu = expand(q_gu, s_gu, b_gu, 2 * I, H);
  double* wd = expand(q_d, s_d, b_d, H, I);
#pragma omp parallel for schedule(dynamic, 1)
  for (int r = 0; r < nrows; ++r) {
    double* x = (double*)malloc(sizeof(double) * (size_t)H);
    for (int k = 0; k < H; ++k) x[k] = orc_bf16_value(x_rows[(size_t)r * H + k]);
    ffn_row(wgu, wd, x, H, I, h_out ? h_out + (size_t)r * I : NULL,
            d_out + (size_t)r * H);
    free(x);
  }
  free(wgu);
  free(wd);
}

/* --------------------------------------------------------------- layer -- */

/* Whole layer output for a subset of tokens.
 *
 * y[t][n] = RNE_bf16( sum_{k=0..K-1} w[t][k] * FFN_{ids[t][k]}(x_t)[n]
 *                     + FFN_shared(x_t)[n] )
 * summed in fp64 in slot order then the shared term (weight 1, no gate;
 * "one shared expert that sees every token" [P3 "Three Workload Shapes"]).
 * ids/w64 come from orc_topk (w in fp64). Experts with no selected token in
 * the subset are never expanded. Expert e's weights start at
 * q_gu + e*2I*H/8 etc.; the shared expert's arrays are separate (NULL when
 * n_shared == 0).
 * tok: token indices [ntok] into x; y_out: bf16 [ntok][H];
 * d_slots (optional): fp64 [ntok][K+1][H] slot outputs (shared last). */
void orc_layer_tokens(const uint16_t* x, int H, int E, int K, int I,
                      const int32_t* ids, const double* w64,
                      const uint32_t* q_gu, const uint16_t* s_gu, const uint16_t* b_gu,
                      const uint32_t* q_d, const uint16_t* s_d, const uint16_t* b_d,
                      const uint32_t* sq_gu, const uint16_t* ss_gu, const uint16_t* sb_gu,
                      const uint32_t* sq_d, const uint16_t* ss_d, const uint16_t* sb_d,
                      const int32_t* tok, int ntok, uint16_t* y_out, double* d_slots) {
  size_t gu_w = (size_t)2 * I * (H / 8), gu_g = (size_t)2 * I * (H / 64);
  size_t d_w = (size_t)H * (I / 8), d_g = (size_t)H * (I / 64);
  int S = K + 1;
  double* dsl = d_slots ? d_slots : (double*)calloc((size_t)ntok * S * H, sizeof(double));
  int has_shared = sq_gu != NULL;
  /* per expert (shared = E): gather the (token, slot) rows routed to it */
  int* nrow = (int*)calloc((size_t)E + 1, sizeof(int));
  for (int i = 0; i < ntok; ++i)
    for (int k = 0; k < K; ++k) nrow[ids[(size_t)tok[i] * K + k]]++;
  nrow[E] = has_shared ? ntok : 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (int e = 0; e <= E; ++e) {
    if (nrow[e] == 0) continue;
    int* which = (int*)malloc(sizeof(int) * (size_t)nrow[e]); /* i*S + slot */
    int m = 0;
    for (int i = 0; i < ntok; ++i) {
      if (e == E) { which[m++] = i * S + K; continue; }
      for (int k = 0; k < K; ++k)
        if (ids[(size_t)tok[i] * K + k] == e) which[m++] = i * S + k;
    }
    const uint32_t *qg, *qd;
    const uint16_t *sg, *bg, *sd, *bd;
    if (e < E) {
      qg = q_gu + e * gu_w; sg = s_gu + e * gu_g; bg = b_gu + e * gu_g;
      qd = q_d + e * d_w; sd = s_d + e * d_g; bd = b_d + e * d_g;
    } else {
      qg = sq_gu; sg = ss_gu; bg = sb_gu; qd = sq_d; sd = ss_d; bd = sb_d;
    }
    double* wgu = expand(qg, sg, bg, 2 * I, H);
    double* wd = expand(qd, sd, bd, H, I);
    double* xr = (double*)malloc(sizeof(double) * (size_t)H);
    for (int r = 0; r < m; ++r) {
      const uint16_t* xs = x + (size_t)tok[which[r] / S] * H;
      for (int k = 0; k < H; ++k) xr[k] = orc_bf16_value(xs[k]);
      ffn_row(wgu, wd, xr, H, I, NULL, dsl + (size_t)which[r] * H);
    }
    free(xr);
    free(wgu);
    free(wd);
    free(which);
  }
  free(nrow);
#pragma omp parallel for schedule(static)
  for (int i = 0; i < ntok; ++i)
    for (int n = 0; n < H; ++n) {
      double acc = 0.0;
      for (int k = 0; k < K; ++k)
        acc += w64[(size_t)tok[i] * K + k] * dsl[((size_t)i * S + k) * H + n];
      if (has_shared) acc += dsl[((size_t)i * S + K) * H + n];
      y_out[(size_t)i * H + n] = orc_bf16_rne(acc);
    }
  if (!d_slots) free(dsl);
}

/* Unit-gain RMS normalisation between stacked layers:
 * x'[n] = RNE_bf16( y[n] / sqrt(mean_n(y[n]^2) + 1e-6) ), y the bf16 layer
 * output, fp64 arithmetic. The layer's workload stacks layers with each
 * output feeding the next; without a normalisation the activations leave
 * the bf16 range within a few layers, so the plainest normalisation (no
 * learned gain) is the reading used. */
void orc_rmsnorm_rows(const uint16_t* y, int T, int H, uint16_t* out) {
  for (int t = 0; t < T; ++t) {
    double ss = 0.0;
    for (int n = 0; n < H; ++n) {
      double v = orc_bf16_value(y[(size_t)t * H + n]);
      ss += v * v;
    }
    double inv = 1.0 / sqrt(ss / H + 1e-6);
    for (int n = 0; n < H; ++n)
      out[(size_t)t * H + n] = orc_bf16_rne(orc_bf16_value(y[(size_t)t * H + n]) * inv);
  }
}

/* The decoder block around an MoE layer (a reading: the pages name the
 * model, Qwen3.6-35B-A3B, and its decode loop [P3 "Decode"], not the block
 * arithmetic; the plainest pre-norm block is taken): the layer's input is
 * the RMS normalisation of the residual stream h with a learned gain g,
 *   x[n] = RNE_bf16( g[n] * h[n] / sqrt(mean_n(h[n]^2) + 1e-6) ),
 * fp64 arithmetic, g and h bf16; the layer's output y is added back,
 *   h'[n] = RNE_bf16( h[n] + y[n] ),
 * one rounding of the exact sum. */
void orc_rmsnorm_gain_rows(const uint16_t* h, const uint16_t* g, int T, int H, uint16_t* out) {
  for (int t = 0; t < T; ++t) {
    double ss = 0.0;
    for (int n = 0; n < H; ++n) {
      double v = orc_bf16_value(h[(size_t)t * H + n]);
      ss += v * v;
    }
    double inv = 1.0 / sqrt(ss / H + 1e-6);
    for (int n = 0; n < H; ++n)
      out[(size_t)t * H + n] =
          orc_bf16_rne(orc_bf16_value(g[n]) * orc_bf16_value(h[(size_t)t * H + n]) * inv);
  }
}

void orc_residual_add(const uint16_t* h, const uint16_t* y, size_t n, uint16_t* out) {
  for (size_t i = 0; i < n; ++i)
    out[i] = orc_bf16_rne(orc_bf16_value(h[i]) + orc_bf16_value(y[i]));
}

/* Decode attention of a grouped-query layer (the model's full-attention
 * layers: 16 query heads share 2 key/value heads [P3 "Three Workload
 * Shapes"]; at decode the queries of a few new tokens attend to a growing
 * key/value cache kept in fixed-size blocks [P3 "Decode"]). Plain softmax
 * attention, fp64:
 *   query token t sits at position L - T + t and sees positions 0..L-T+t;
 *   head h reads key/value head h / (n_q / n_kv);
 *   s_j = (q . k_j) / sqrt(D),  o = sum_j softmax(s)_j v_j,  RNE to bf16.
 * Position j of head g is row j % B of physical block table[j / B]:
 * k_cache[((table[j / B] * n_kv + g) * B + j % B) * D + d], v likewise.
 * q, o: [T][n_q][D] bf16 bits. Returns -1 for a table entry outside
 * [0, n_phys), else 0. */
int orc_attn_decode(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                    const int32_t* table, int n_phys, int T, int n_q, int n_kv, int D, int L,
                    int B, uint16_t* o) {
  const int nblk = (L + B - 1) / B;
  for (int i = 0; i < nblk; ++i)
    if (table[i] < 0 || table[i] >= n_phys) return -1;
  const int group = n_q / n_kv;
  double* s = (double*)malloc(sizeof(double) * (size_t)L);
  double* acc = (double*)malloc(sizeof(double) * (size_t)D);
  for (int t = 0; t < T; ++t) {
    const int last = L - T + t;  /* the token's own position */
    for (int h = 0; h < n_q; ++h) {
      const int g = h / group;
      const uint16_t* qv = q + ((size_t)t * n_q + h) * D;
      double mx = -INFINITY;
      for (int j = 0; j <= last; ++j) {
        const size_t row = (((size_t)table[j / B] * n_kv + g) * B + j % B) * D;
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += orc_bf16_value(qv[d]) * orc_bf16_value(k_cache[row + d]);
        s[j] = dot / sqrt((double)D);
        if (s[j] > mx) mx = s[j];
      }
      double z = 0.0;
      for (int d = 0; d < D; ++d) acc[d] = 0.0;
      for (int j = 0; j <= last; ++j) {
        const double p = exp(s[j] - mx);
        z += p;
        const size_t row = (((size_t)table[j / B] * n_kv + g) * B + j % B) * D;
        for (int d = 0; d < D; ++d) acc[d] += p * orc_bf16_value(v_cache[row + d]);
      }
      for (int d = 0; d < D; ++d) o[((size_t)t * n_q + h) * D + d] = orc_bf16_rne(acc[d] / z);
    }
  }
  free(s);
  free(acc);
  return 0;
}

/* The fixed-size recurrence of the model's 30 Gated DeltaNet layers [P3
 * "Three Workload Shapes"; the pages name a register-resident scan, P3
 * "Prefill"] in the published gated delta rule (Yang, Kautz, Hatamizadeh,
 * "Gated Delta Networks: Improving Mamba2 with Delta Rule"), fp64: per
 * value head h (key head h / (n_v / n_k)), state S [dv][dk], and token t
 *   S <- alpha_t S (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
 *   o_t = S q_t   (RNE to bf16).
 * q, k [T][n_k][dk] and v [T][n_v][dv] are bf16 bits; alpha, beta [T][n_v]
 * and the states [n_v][dv][dk] are fp32 (s_out may equal s_in). */
static void gdn_scan_core(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                          const float* alpha, const float* beta, const float* s_in, int T,
                          int n_k, int n_v, int dk, int dv, float* s_out, uint16_t* o,
                          double* o64, double* s_out64) {
  const int group = n_v / n_k;
  double* S = (double*)malloc(sizeof(double) * (size_t)dv * dk);
  double* Sk = (double*)malloc(sizeof(double) * (size_t)dv);
  for (int h = 0; h < n_v; ++h) {
    const int hk = h / group;
    for (size_t i = 0; i < (size_t)dv * dk; ++i) S[i] = s_in[(size_t)h * dv * dk + i];
    for (int t = 0; t < T; ++t) {
      const uint16_t* kt = k + ((size_t)t * n_k + hk) * dk;
      const uint16_t* qt = q + ((size_t)t * n_k + hk) * dk;
      const uint16_t* vt = v + ((size_t)t * n_v + h) * dv;
      const double a = alpha[(size_t)t * n_v + h], b = beta[(size_t)t * n_v + h];
      /* S k, then S <- a S - a b (S k) k^T + b v k^T */
      for (int i = 0; i < dv; ++i) {
        double acc = 0.0;
        for (int j = 0; j < dk; ++j) acc += S[(size_t)i * dk + j] * orc_bf16_value(kt[j]);
        Sk[i] = acc;
      }
      for (int i = 0; i < dv; ++i)
        for (int j = 0; j < dk; ++j) {
          const double kj = orc_bf16_value(kt[j]);
          S[(size_t)i * dk + j] =
              a * S[(size_t)i * dk + j] - a * b * Sk[i] * kj + b * orc_bf16_value(vt[i]) * kj;
        }
      for (int i = 0; i < dv; ++i) {
        double acc = 0.0;
        for (int j = 0; j < dk; ++j) acc += S[(size_t)i * dk + j] * orc_bf16_value(qt[j]);
        if (o) o[((size_t)t * n_v + h) * dv + i] = orc_bf16_rne(acc);
        if (o64) o64[((size_t)t * n_v + h) * dv + i] = acc;
      }
    }
    for (size_t i = 0; i < (size_t)dv * dk; ++i) {
      if (s_out) s_out[(size_t)h * dv * dk + i] = (float)S[i];
      if (s_out64) s_out64[(size_t)h * dv * dk + i] = S[i];
    }
  }
  free(S);
  free(Sk);
}

void orc_gdn_scan(const uint16_t* q, const uint16_t* k, const uint16_t* v, const float* alpha,
                  const float* beta, const float* s_in, int T, int n_k, int n_v, int dk, int dv,
                  float* s_out, uint16_t* o) {
  gdn_scan_core(q, k, v, alpha, beta, s_in, T, n_k, n_v, dk, dv, s_out, o, NULL, NULL);
}

/* The same recurrence with its results kept in fp64 (outputs before the
 * bf16 rounding, and the final state): for comparing other forms of the
 * rule with it at full precision. */
void orc_gdn_scan64(const uint16_t* q, const uint16_t* k, const uint16_t* v, const float* alpha,
                    const float* beta, const float* s_in, int T, int n_k, int n_v, int dk,
                    int dv, double* s_out64, double* o64) {
  gdn_scan_core(q, k, v, alpha, beta, s_in, T, n_k, n_v, dk, dv, NULL, NULL, o64, s_out64);
}

/*
 * The same gated delta rule in its chunked (parallel) form: chunks of C
 * tokens, each solved as a whole from the state S0 before it. This is the
 * WY / UT-transform form of the delta rule (Yang et al., "Gated Delta
 * Networks: Improving Mamba2 with Delta Rule", chunkwise algorithm),
 * written out here from the recurrence above. Within a chunk (tokens
 * t = 1..n), with g_t = alpha_1 ... alpha_t (g_0 = 1) and
 * u_t = beta_t (v_t - alpha_t S_{t-1} k_t), the recurrence reads
 * S_t = alpha_t S_{t-1} + u_t k_t^T, so S_t = g_t S0 + sum_{s<=t} (g_t/g_s) u_s k_s^T.
 * Putting that S_{t-1} into u_t gives a unit lower-triangular system:
 *   (1) g_t, t = 1..n
 *   (2) A[t][s] = beta_t (g_t / g_s) (k_t . k_s) for s < t, 0 otherwise
 *   (3) Tm = (I + A)^-1 (forward substitution)
 *   (4) W1 = Tm diag(beta) V  [n x dv],  W2 = Tm diag(beta g) K  [n x dk]
 *   (5) U = W1 - W2 S0^T  [n x dv]  (row t = u_t)
 *   (6) O = diag(g) Q S0^T + (Mk o (Q K^T)) U, Mk[t][s] = g_t / g_s for s <= t, else 0
 *   (7) S = g_n S0 + U^T diag(g_n / g) K
 * o_t = row t of O. All in fp64; o is rounded to bf16 at the end, as in
 * orc_gdn_scan. s_chunks64 (nullable) receives the state after every chunk,
 * [n_chunks][n_v][dv][dk]; o64 (nullable) the unrounded outputs.
 */
void orc_gdn_chunked(const uint16_t* q, const uint16_t* k, const uint16_t* v, const float* alpha,
                     const float* beta, const float* s_in, int T, int n_k, int n_v, int dk,
                     int dv, int C, float* s_out, uint16_t* o, double* o64, double* s_chunks64) {
  const int group = n_v / n_k;
  const int n_chunks = (T + C - 1) / C;
  double* S = (double*)malloc(sizeof(double) * (size_t)dv * dk);
  double* Sn = (double*)malloc(sizeof(double) * (size_t)dv * dk);
  double* g = (double*)malloc(sizeof(double) * (size_t)C);
  double* Kc = (double*)malloc(sizeof(double) * (size_t)C * dk);
  double* Qc = (double*)malloc(sizeof(double) * (size_t)C * dk);
  double* Vc = (double*)malloc(sizeof(double) * (size_t)C * dv);
  double* A = (double*)malloc(sizeof(double) * (size_t)C * C);
  double* Tm = (double*)malloc(sizeof(double) * (size_t)C * C);
  double* W1 = (double*)malloc(sizeof(double) * (size_t)C * dv);
  double* W2 = (double*)malloc(sizeof(double) * (size_t)C * dk);
  double* U = (double*)malloc(sizeof(double) * (size_t)C * dv);
  double* QK = (double*)malloc(sizeof(double) * (size_t)C * C);
  for (int h = 0; h < n_v; ++h) {
    const int hk = h / group;
    for (size_t i = 0; i < (size_t)dv * dk; ++i) S[i] = s_in[(size_t)h * dv * dk + i];
    for (int c = 0; c < n_chunks; ++c) {
      const int t0 = c * C, n = (T - t0 < C) ? T - t0 : C;
      const float* al = alpha + (size_t)t0 * n_v + h;
      const float* be = beta + (size_t)t0 * n_v + h;
      for (int t = 0; t < n; ++t) {
        for (int j = 0; j < dk; ++j) {
          Kc[(size_t)t * dk + j] = orc_bf16_value(k[((size_t)(t0 + t) * n_k + hk) * dk + j]);
          Qc[(size_t)t * dk + j] = orc_bf16_value(q[((size_t)(t0 + t) * n_k + hk) * dk + j]);
        }
        for (int i = 0; i < dv; ++i)
          Vc[(size_t)t * dv + i] = orc_bf16_value(v[((size_t)(t0 + t) * n_v + h) * dv + i]);
      }
      /* (1) */
      for (int t = 0; t < n; ++t) g[t] = (t ? g[t - 1] : 1.0) * (double)al[(size_t)t * n_v];
      /* (2) and Q K^T */
      for (int t = 0; t < n; ++t)
        for (int s2 = 0; s2 < n; ++s2) {
          double kk = 0.0, qk = 0.0;
          for (int j = 0; j < dk; ++j) {
            kk += Kc[(size_t)t * dk + j] * Kc[(size_t)s2 * dk + j];
            qk += Qc[(size_t)t * dk + j] * Kc[(size_t)s2 * dk + j];
          }
          A[(size_t)t * C + s2] = s2 < t ? (double)be[(size_t)t * n_v] * (g[t] / g[s2]) * kk : 0.0;
          QK[(size_t)t * C + s2] = s2 <= t ? (g[t] / g[s2]) * qk : 0.0;
        }
      /* (3) Tm (I + A) = I, row by row: Tm[t] = e_t - sum_{r<t} A[t][r] Tm[r] */
      for (int t = 0; t < n; ++t)
        for (int s2 = 0; s2 < n; ++s2) {
          double x = (s2 == t) ? 1.0 : 0.0;
          for (int r = s2; r < t; ++r) x -= A[(size_t)t * C + r] * Tm[(size_t)r * C + s2];
          Tm[(size_t)t * C + s2] = s2 <= t ? x : 0.0;
        }
      /* (4) */
      for (int t = 0; t < n; ++t) {
        for (int i = 0; i < dv; ++i) {
          double x = 0.0;
          for (int s2 = 0; s2 <= t; ++s2)
            x += Tm[(size_t)t * C + s2] * (double)be[(size_t)s2 * n_v] * Vc[(size_t)s2 * dv + i];
          W1[(size_t)t * dv + i] = x;
        }
        for (int j = 0; j < dk; ++j) {
          double x = 0.0;
          for (int s2 = 0; s2 <= t; ++s2)
            x += Tm[(size_t)t * C + s2] * (double)be[(size_t)s2 * n_v] * g[s2] *
                 Kc[(size_t)s2 * dk + j];
          W2[(size_t)t * dk + j] = x;
        }
      }
      /* (5) */
      for (int t = 0; t < n; ++t)
        for (int i = 0; i < dv; ++i) {
          double x = W1[(size_t)t * dv + i];
          for (int j = 0; j < dk; ++j) x -= W2[(size_t)t * dk + j] * S[(size_t)i * dk + j];
          U[(size_t)t * dv + i] = x;
        }
      /* (6) */
      for (int t = 0; t < n; ++t)
        for (int i = 0; i < dv; ++i) {
          double x = 0.0;
          for (int j = 0; j < dk; ++j) x += Qc[(size_t)t * dk + j] * S[(size_t)i * dk + j];
          x *= g[t];
          for (int s2 = 0; s2 <= t; ++s2) x += QK[(size_t)t * C + s2] * U[(size_t)s2 * dv + i];
          const size_t oi = ((size_t)(t0 + t) * n_v + h) * dv + i;
          if (o) o[oi] = orc_bf16_rne(x);
          if (o64) o64[oi] = x;
        }
      /* (7) */
      for (int i = 0; i < dv; ++i)
        for (int j = 0; j < dk; ++j) {
          double x = g[n - 1] * S[(size_t)i * dk + j];
          for (int t = 0; t < n; ++t)
            x += U[(size_t)t * dv + i] * (g[n - 1] / g[t]) * Kc[(size_t)t * dk + j];
          Sn[(size_t)i * dk + j] = x;
        }
      memcpy(S, Sn, sizeof(double) * (size_t)dv * dk);
      if (s_chunks64)
        memcpy(s_chunks64 + ((size_t)c * n_v + h) * dv * dk, S, sizeof(double) * (size_t)dv * dk);
    }
    for (size_t i = 0; i < (size_t)dv * dk; ++i)
      if (s_out) s_out[(size_t)h * dv * dk + i] = (float)S[i];
  }
  free(S); free(Sn); free(g); free(Kc); free(Qc); free(Vc); free(A); free(Tm); free(W1);
  free(W2); free(U); free(QK);
}

int orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
