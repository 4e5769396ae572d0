/*
 * s2_oracle.c — plain, slow fp32 CPU definition of the S2-Pro Dual-AR frame decode.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product imports, links or runs this
 * file; only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline leg do.
 * It shares no code, header, table or constant with the CUDA path.
 *
 * Sources (cited by page and section):
 *   [ch02] s2.cpp analysis, ch.02 "Overall architecture and Dual-AR data flow"
 *          (blog.chen3feng.top/s2cpp-analysis/02-...)
 *   [ch06] s2.cpp analysis, ch.06 "Fast-AR codebook decoding and the generation main loop"
 *   [ch04] s2.cpp analysis, ch.04 "Model loading and GGUF"
 *   [miz]  Mizuoto docs, "Fish Speech" engine page (mizuoto.netlify.app/docs/engines-fishspeech)
 *
 * Precision: fp32 throughout ([miz] "how it works": fp32 off-GPU; RMSNorm in fp32).
 * Weights are given as fp32 or as bf16 bit patterns widened to fp32 on read.  When
 * the model declares an fp16 KV cache ([ch02] §1: memory_k_/memory_v_ are F16), K and
 * V are rounded to fp16 on store.  Every dot product is a sequential fp32 sum in
 * index order; loops are parallelised only over independent outputs.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- shapes */

typedef struct or_dims {
  int dim, n_layer, n_head, n_kv_head, head_dim, ffn, vocab;
  int sem_begin, sem_end, im_end, n_codebooks, codebook_size;
  float sem_scale, norm_eps, rope_base;
  int qk_norm, rope_table_bf16;
  int fast_dim, fast_n_layer, fast_n_head, fast_n_kv_head, fast_head_dim, fast_ffn, fast_window,
      has_fast_project_in;
  int weight_dtype; /* 0 = fp32, 1 = bf16 */
  int kv_dtype;     /* 0 = fp32, 2 = fp16 */
} or_dims;

typedef struct {
  const void* p;
  int bf16;
  const float* rs; /* non-NULL: p holds e4m3 codes, one scale per row of `cols` codes */
  int cols;
} wref;

static inline float bf16_bits_to_f32(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

static inline float f32_to_bf16_value(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  u += 0x7fffu + ((u >> 16) & 1u); /* round to nearest even on the top 16 bits */
  u &= 0xffff0000u;
  memcpy(&f, &u, 4);
  return f;
}

static inline float f32_to_f16_value(float f) { return (float)(_Float16)f; }

/* ------------------------------------------------------ e4m3 weights
 * Low-precision weight streaming (the K-quantised GGUF tensors of s2.cpp are the pages'
 * precedent, s2.cpp analysis ch.02 §5 and ch.04 §4; the format and the scaling below are the
 * library's choice).  e4m3 as the OCP 8-bit float E4M3 defines it: sign bit, 4 exponent bits with
 * bias 7, 3 mantissa bits, no infinities, S.1111.111 = NaN; exponent field 0 holds the
 * subnormals m * 2^-9.  Largest finite value 1.75 * 2^8 = 448. */

double or_e4m3_value(int code) {
  const int e = (code >> 3) & 15, m = code & 7;
  const double v = e == 0 ? ldexp((double)m, -9) : ldexp((double)(8 + m), e - 10);
  return (code & 0x80) ? -v : v;
}

/* nearest e4m3 value of a finite x, ties to the even mantissa, magnitudes from 448 up -> 448 */
int or_e4m3_encode(float x) {
  const int sign = signbit(x) ? 0x80 : 0;
  const double a = fabs((double)x);
  if (a >= 448.0) return sign | 0x7E;
  if (a < ldexp(1.0, -6)) /* subnormal steps of 2^-9; 8 steps is the smallest normal, code 0x08 */
    return sign | (int)nearbyint(a * 512.0);
  int e2;
  frexp(a, &e2);
  int E = e2 - 1; /* 2^E <= a < 2^(E+1), -6 <= E <= 8 */
  double q = nearbyint(ldexp(a, 3 - E)); /* a / 2^(E-3) in [8, 16): 8 + mantissa */
  if (q == 16.0) {
    q = 8.0;
    E += 1;
  }
  return sign | ((E + 7) << 3) | ((int)q - 8);
}

/* per row: scale = max|w| / 448 (fp32), code = e4m3(w / scale) (fp32 division); all-zero rows get
 * scale 0 and zero codes */
void or_quant_e4m3(const uint16_t* w, long long rows, int cols, uint8_t* codes, float* scales) {
#pragma omp parallel for schedule(static)
  for (long long r = 0; r < rows; ++r) {
    const uint16_t* wr = w + r * cols;
    float amax = 0.f;
    for (int k = 0; k < cols; ++k) {
      const float a = fabsf(bf16_bits_to_f32(wr[k]));
      if (a > amax) amax = a;
    }
    const float scale = amax / 448.0f;
    scales[r] = scale;
    for (int k = 0; k < cols; ++k)
      codes[r * cols + k] = scale > 0.f ? (uint8_t)or_e4m3_encode(bf16_bits_to_f32(wr[k]) / scale) : 0;
  }
}

/* the 256 code values, filled by or_bind_e4m3 before any session reads codes */
static double g_e4m3[256];

static inline float wget(wref w, size_t i) {
  if (w.rs) return (float)(g_e4m3[((const uint8_t*)w.p)[i]] * (double)w.rs[i / (size_t)w.cols]);
  return w.bf16 ? bf16_bits_to_f32(((const uint16_t*)w.p)[i]) : ((const float*)w.p)[i];
}

typedef struct {
  wref an, wqkv, qn, kn, wo, fn, w1, w3, w2;
} or_layer;

typedef struct or_sess {
  or_dims d;
  wref E, CE, norm, P, FE, fnorm, FO;
  or_layer* slow;
  or_layer* fast;
  int slots;
  float* kc; /* [n_layer][n_kv_head][slots][head_dim] */
  float* vc;
  int pos;   /* next free slot == number of positions in the cache */
} or_sess;

/* ------------------------------------------------------------ primitives */

/* RMSNorm in fp32 ([miz] "numerics": Fish's RMSNorm is computed in float32):
 *   out_i = x_i · 1/sqrt(mean_j(x_j²) + eps) · w_i   */
void or_rmsnorm(const float* x, int n, const float* w, float eps, float* out) {
  float ss = 0.f;
  for (int i = 0; i < n; ++i) ss += x[i] * x[i];
  float r = 1.0f / sqrtf(ss / (float)n + eps);
  for (int i = 0; i < n; ++i) out[i] = x[i] * r * (w ? w[i] : 1.0f);
}

static void rmsnorm_w(const float* x, int n, wref w, float eps, float* out) {
  float ss = 0.f;
  for (int i = 0; i < n; ++i) ss += x[i] * x[i];
  float r = 1.0f / sqrtf(ss / (float)n + eps);
  for (int i = 0; i < n; ++i) out[i] = x[i] * r * wget(w, (size_t)i);
}

/* RoPE on one head vector, in place ([ch02] §2: base 1e6; [miz] "numerics": rotation of
 * adjacent element pairs, frequency table rounded to bf16).  Pair i = (x[2i], x[2i+1]) is
 * rotated by angle pos·θ_i with θ_i = base^(-2i/hd); the angle is formed in fp64 and its
 * cos/sin rounded to fp32 (then to bf16 when the table is bf16). */
void or_rope(float* x, int hd, int pos, double base, int table_bf16) {
  for (int i = 0; i < hd / 2; ++i) {
    double theta = pow(base, -2.0 * (double)i / (double)hd);
    double ang = (double)pos * theta;
    float c = (float)cos(ang), s = (float)sin(ang);
    if (table_bf16) {
      c = f32_to_bf16_value(c);
      s = f32_to_bf16_value(s);
    }
    float a = x[2 * i], b = x[2 * i + 1];
    x[2 * i] = a * c - b * s;
    x[2 * i + 1] = a * s + b * c;
  }
}

/* Head map of grouped-query attention built as repeat_interleave of the KV head indices
 * ([miz] "intentional differences": keys and values after repeat_interleave; [ch06] §3:
 * GQA expansion 4x).  map[h] = KV head feeding query head h. */
void or_gqa_head_map(int Hq, int Hkv, int* map) {
  int rep = Hq / Hkv, h = 0;
  for (int g = 0; g < Hkv; ++g)
    for (int r = 0; r < rep; ++r) map[h++] = g;
}

/* Scaled dot-product attention of one query over slots 0..n-1 of one head:
 *   o = Σ_j softmax_j(q·k_j · scale) v_j   (fp32, max-subtracted softmax). */
static void attend_one(const float* q, const float* K, const float* V, int n, int hd, float scale,
                       float* sc, float* o) {
  float m = -INFINITY;
  for (int j = 0; j < n; ++j) {
    float s = 0.f;
    for (int e = 0; e < hd; ++e) s += q[e] * K[(size_t)j * hd + e];
    sc[j] = s * scale;
    if (sc[j] > m) m = sc[j];
  }
  float l = 0.f;
  for (int j = 0; j < n; ++j) {
    sc[j] = expf(sc[j] - m);
    l += sc[j];
  }
  for (int e = 0; e < hd; ++e) o[e] = 0.f;
  for (int j = 0; j < n; ++j) {
    float p = sc[j] / l;
    for (int e = 0; e < hd; ++e) o[e] += p * V[(size_t)j * hd + e];
  }
}

/* Multi-query-head attention of one position: q [Hq][hd]; K,V [Hkv][stride][hd] with the
 * first n slots used; out [Hq][hd].  Query head h reads KV head map[h]. */
void or_attention(const float* q, const float* K, const float* V, int Hq, int Hkv, int hd, int stride,
                  int n, float* out) {
  int* map = (int*)malloc(sizeof(int) * Hq);
  float* sc = (float*)malloc(sizeof(float) * (n > 0 ? n : 1));
  or_gqa_head_map(Hq, Hkv, map);
  float scale = (float)(1.0 / sqrt((double)hd)); /* attn_scale = 1/sqrt(head_dim), [ch02] §3.2 */
  for (int h = 0; h < Hq; ++h) {
    size_t g = (size_t)map[h];
    attend_one(q + (size_t)h * hd, K + g * stride * hd, V + g * stride * hd, n, hd, scale, sc,
               out + (size_t)h * hd);
  }
  free(sc);
  free(map);
}

/* y[t][r] = Σ_k W[r][k]·x[t][k] for t < n, summed in k order (one GEMV per position). */
static void linear(wref W, int M, int K, const float* x, int n, float* y) {
  if (n == 1) {
#pragma omp parallel for schedule(static)
    for (int r = 0; r < M; ++r) {
      float acc = 0.f;
      size_t base = (size_t)r * K;
      for (int k = 0; k < K; ++k) acc += wget(W, base + k) * x[k];
      y[r] = acc;
    }
    return;
  }
  /* several positions: read each weight row once, keep one running sum per position */
  float* xt = (float*)malloc(sizeof(float) * (size_t)K * n); /* x transposed to [k][t] */
  for (int t = 0; t < n; ++t)
    for (int k = 0; k < K; ++k) xt[(size_t)k * n + t] = x[(size_t)t * K + k];
#pragma omp parallel
  {
    float* acc = (float*)malloc(sizeof(float) * n);
#pragma omp for schedule(dynamic, 8)
    for (int r = 0; r < M; ++r) {
      size_t base = (size_t)r * K;
      for (int t = 0; t < n; ++t) acc[t] = 0.f;
      for (int k = 0; k < K; ++k) {
        float w = wget(W, base + k);
        const float* xk = xt + (size_t)k * n;
        for (int t = 0; t < n; ++t) acc[t] += w * xk[t];
      }
      for (int t = 0; t < n; ++t) y[(size_t)t * M + r] = acc[t];
    }
    free(acc);
  }
  free(xt);
}

static inline float silu(float a) { return a / (1.0f + expf(-a)); }

/* --------------------------------------------------------------- a block */

/* One transformer block over n positions (rows of x, at cache slots pos0..pos0+n-1),
 * as described for both Slow-AR and Fast-AR ([ch02] §3.2, [ch06] §3, [miz] "how it works"):
 *   h = RMSNorm(x)·attention_norm;  qkv = wqkv·h  split as [q: Hq·hd | k: Hkv·hd | v: Hkv·hd]
 *   q_h, k_g <- per-head RMSNorm (q_norm / k_norm), then RoPE at their position
 *   k, v stored into the cache slots; position t attends to slots 0..pos0+t (causal)
 *   x += wo·o
 *   h = RMSNorm(x)·ffn_norm;  x += w2·(silu(w1·h) ⊙ w3·h)                                   */
static void block(const or_layer* lw, int D, int Hq, int Hkv, int hd, int F, float eps, int qk_norm,
                  double rope_base, int rope_bf16, int kv_f16, float* x, int n, int pos0, float* kc,
                  float* vc, int slots) {
  const int QKV = (Hq + 2 * Hkv) * hd, O = Hq * hd;
  float* h = (float*)malloc(sizeof(float) * (size_t)n * D);
  float* qkv = (float*)malloc(sizeof(float) * (size_t)n * QKV);
  float* o = (float*)malloc(sizeof(float) * (size_t)n * O);
  float* y = (float*)malloc(sizeof(float) * (size_t)n * (D > F ? D : F));
  float* a = (float*)malloc(sizeof(float) * (size_t)n * F);
  float* b = (float*)malloc(sizeof(float) * (size_t)n * F);
  float* tmp = (float*)malloc(sizeof(float) * hd);

  for (int t = 0; t < n; ++t) rmsnorm_w(x + (size_t)t * D, D, lw->an, eps, h + (size_t)t * D);
  linear(lw->wqkv, QKV, D, h, n, qkv);

  for (int t = 0; t < n; ++t) {
    float* row = qkv + (size_t)t * QKV;
    int pos = pos0 + t;
    for (int hh = 0; hh < Hq + Hkv; ++hh) { /* q heads then k heads */
      float* v = row + (size_t)hh * hd;
      if (qk_norm) {
        wref nw = hh < Hq ? lw->qn : lw->kn;
        rmsnorm_w(v, hd, nw, eps, tmp);
        memcpy(v, tmp, sizeof(float) * hd);
      }
      or_rope(v, hd, pos, rope_base, rope_bf16);
    }
    for (int g = 0; g < Hkv; ++g) {
      const float* kk = row + (size_t)(Hq + g) * hd;
      const float* vv = row + (size_t)(Hq + Hkv + g) * hd;
      float* kd = kc + ((size_t)g * slots + pos) * hd;
      float* vd = vc + ((size_t)g * slots + pos) * hd;
      for (int e = 0; e < hd; ++e) {
        kd[e] = kv_f16 ? f32_to_f16_value(kk[e]) : kk[e];
        vd[e] = kv_f16 ? f32_to_f16_value(vv[e]) : vv[e];
      }
    }
  }
#pragma omp parallel for schedule(dynamic, 1)
  for (int t = 0; t < n; ++t)
    or_attention(qkv + (size_t)t * QKV, kc, vc, Hq, Hkv, hd, slots, pos0 + t + 1, o + (size_t)t * O);

  linear(lw->wo, D, O, o, n, y);
  for (size_t i = 0; i < (size_t)n * D; ++i) x[i] += y[i];

  for (int t = 0; t < n; ++t) rmsnorm_w(x + (size_t)t * D, D, lw->fn, eps, h + (size_t)t * D);
  linear(lw->w1, F, D, h, n, a);
  linear(lw->w3, F, D, h, n, b);
  for (size_t i = 0; i < (size_t)n * F; ++i) a[i] = silu(a[i]) * b[i];
  linear(lw->w2, D, F, a, n, y);
  for (size_t i = 0; i < (size_t)n * D; ++i) x[i] += y[i];

  free(tmp);
  free(b);
  free(a);
  free(y);
  free(o);
  free(qkv);
  free(h);
}

/* ------------------------------------------------------------- sessions */

int or_weight_count(const or_dims* d) { return 3 + 9 * d->n_layer + 4 + 9 * d->fast_n_layer; }

static void bind_layer(or_layer* L, const void* const* w, int bf16) {
  wref* f[9] = {&L->an, &L->wqkv, &L->qn, &L->kn, &L->wo, &L->fn, &L->w1, &L->w3, &L->w2};
  for (int i = 0; i < 9; ++i) {
    f[i]->p = w[i];
    /* norm vectors of a bf16 model are bf16 too */
    f[i]->bf16 = bf16;
  }
}

or_sess* or_new(const or_dims* d, const void* const* w, int n_w, int slots) {
  if (n_w != or_weight_count(d)) return NULL;
  or_sess* s = (or_sess*)calloc(1, sizeof(or_sess));
  s->d = *d;
  int bf = d->weight_dtype == 1;
  int i = 0;
  s->E = (wref){w[i++], bf};
  s->CE = (wref){w[i++], bf};
  s->norm = (wref){w[i++], bf};
  s->slow = (or_layer*)calloc((size_t)(d->n_layer > 0 ? d->n_layer : 1), sizeof(or_layer));
  for (int l = 0; l < d->n_layer; ++l, i += 9) bind_layer(&s->slow[l], w + i, bf);
  s->P = (wref){w[i++], bf};
  s->FE = (wref){w[i++], bf};
  s->fnorm = (wref){w[i++], bf};
  s->FO = (wref){w[i++], bf};
  s->fast = (or_layer*)calloc((size_t)(d->fast_n_layer > 0 ? d->fast_n_layer : 1), sizeof(or_layer));
  for (int l = 0; l < d->fast_n_layer; ++l, i += 9) bind_layer(&s->fast[l], w + i, bf);
  s->slots = slots;
  size_t kvn = (size_t)d->n_layer * d->n_kv_head * (size_t)slots * d->head_dim;
  s->kc = (float*)calloc(kvn ? kvn : 1, sizeof(float));
  s->vc = (float*)calloc(kvn ? kvn : 1, sizeof(float));
  if (!s->kc || !s->vc) {
    free(s->kc);
    free(s->vc);
    free(s->slow);
    free(s->fast);
    free(s);
    return NULL;
  }
  return s;
}

void or_free(or_sess* s) {
  if (!s) return;
  free(s->kc);
  free(s->vc);
  free(s->slow);
  free(s->fast);
  free(s);
}

int or_pos(const or_sess* s) { return s->pos; }

/* Slow-AR input of one position ([ch02] §3.2):
 *   x = sem_scale·embeddings[r0] + m·Σ_{c=0..NCB-1} codebook_embeddings[c·CBS + r_{c+1}]
 * with m = 1 when r0 is a semantic id (sem_begin..sem_end), else 0 (text positions take the
 * semantic/text embedding alone).  Codebook c (matrix row c+1) is offset by c·codebook_size
 * into the shared 10×4096-row table. */
void or_embed(const or_sess* s, const int32_t* vals, float* x) {
  const or_dims* d = &s->d;
  const int D = d->dim;
  int r0 = vals[0];
  float m = (r0 >= d->sem_begin && r0 <= d->sem_end) ? 1.0f : 0.0f;
  for (int e = 0; e < D; ++e) {
    float acc = 0.f;
    for (int c = 0; c < d->n_codebooks; ++c) {
      size_t row = (size_t)c * d->codebook_size + (size_t)vals[1 + c];
      acc += wget(s->CE, row * D + e);
    }
    x[e] = d->sem_scale * wget(s->E, (size_t)r0 * D + e) + m * acc;
  }
}

static int check_vals(const or_dims* d, const int32_t* vals) {
  if (vals[0] < 0 || vals[0] >= d->vocab) return -1;
  for (int c = 0; c < d->n_codebooks; ++c)
    if (vals[1 + c] < 0 || vals[1 + c] >= d->codebook_size) return -1;
  return 0;
}

/* Final norm and tied logits ([ch02] §3.2: logits = hidden · embeddings^T). */
static void head(const or_sess* s, const float* xlast, float* logits, float* hidden) {
  const or_dims* d = &s->d;
  float* h = (float*)malloc(sizeof(float) * d->dim);
  rmsnorm_w(xlast, d->dim, s->norm, d->norm_eps, h);
  if (hidden) memcpy(hidden, h, sizeof(float) * d->dim);
  if (logits) linear(s->E, d->vocab, d->dim, h, 1, logits);
  free(h);
}

/* Slow-AR forward over n positions starting at the session's current slot. */
static int slow_forward(or_sess* s, const int32_t* tokens, int n, float* logits, float* hidden) {
  const or_dims* d = &s->d;
  const int C = d->n_codebooks + 1, D = d->dim;
  if (n <= 0 || s->pos + n > s->slots) return -2;
  for (int t = 0; t < n; ++t)
    if (check_vals(d, tokens + (size_t)t * C)) return -1;
  float* x = (float*)malloc(sizeof(float) * (size_t)n * D);
  for (int t = 0; t < n; ++t) or_embed(s, tokens + (size_t)t * C, x + (size_t)t * D);
  size_t per_layer = (size_t)d->n_kv_head * s->slots * d->head_dim;
  for (int l = 0; l < d->n_layer; ++l)
    block(&s->slow[l], D, d->n_head, d->n_kv_head, d->head_dim, d->ffn, d->norm_eps, d->qk_norm,
          d->rope_base, d->rope_table_bf16, d->kv_dtype == 2, x, n, s->pos, s->kc + l * per_layer,
          s->vc + l * per_layer, s->slots);
  s->pos += n;
  head(s, x + (size_t)(n - 1) * D, logits, hidden);
  free(x);
  return 0;
}

/* Prefill: reset the stream and run the prompt (column-major tokens [t][row], [ch02] §3.1);
 * logits and normalised hidden of the last position come back. */
int or_prefill(or_sess* s, const int32_t* tokens, int T, float* logits, float* hidden) {
  s->pos = 0;
  return slow_forward(s, tokens, T, logits, hidden);
}

/* Further prompt positions after the ones already in the cache: a prompt run in consecutive
 * pieces (causal attention over every earlier slot, [ch02] §3.1) gives what one prefill of the
 * whole prompt gives, with a small working set per piece.  Logits and hidden of the last
 * position come back. */
int or_extend(or_sess* s, const int32_t* tokens, int n, float* logits, float* hidden) {
  return slow_forward(s, tokens, n, logits, hidden);
}

/* One Slow-AR step on the 11 values [main_token, code_0..code_9] ([ch02] §3.4). */
int or_step(or_sess* s, const int32_t* vals, float* logits, float* hidden) {
  return slow_forward(s, vals, 1, logits, hidden);
}

/* Fast-AR call ([ch06] §1-§4): input rows [fast_project_in·hidden ; fast_embeddings[prefix_j]],
 * positions 0..k from zero, causal (mask offset 0), no persistent cache; fast_norm on every
 * row, fast_output on the last row -> codebook_size logits.  `rows` (nullable) receives the
 * fast_norm output of all k+1 rows. */
int or_fast_forward(const or_sess* s, const float* hidden, const int32_t* prefix, int k, float* logits,
                    float* rows) {
  const or_dims* d = &s->d;
  const int Df = d->fast_dim, w = k + 1;
  /* entry checks of [ch06] §1: a fast decoder exists; prefix shorter than the codebook count */
  if (d->fast_n_layer <= 0 || k < 1 || k >= d->n_codebooks || w > d->fast_window) return -1;
  if (!d->has_fast_project_in && Df != d->dim) return -1;
  for (int j = 0; j < k; ++j)
    if (prefix[j] < 0 || prefix[j] >= d->codebook_size) return -1;
  float* x = (float*)malloc(sizeof(float) * (size_t)w * Df);
  if (d->has_fast_project_in)
    linear(s->P, Df, d->dim, hidden, 1, x);
  else
    memcpy(x, hidden, sizeof(float) * Df);
  for (int j = 0; j < k; ++j)
    for (int e = 0; e < Df; ++e) x[(size_t)(1 + j) * Df + e] = wget(s->FE, (size_t)prefix[j] * Df + e);
  const int hkv = d->fast_n_kv_head, hd = d->fast_head_dim;
  float* kc = (float*)calloc((size_t)hkv * w * hd, sizeof(float));
  float* vc = (float*)calloc((size_t)hkv * w * hd, sizeof(float));
  for (int l = 0; l < d->fast_n_layer; ++l)
    block(&s->fast[l], Df, d->fast_n_head, hkv, hd, d->fast_ffn, d->norm_eps, d->qk_norm, d->rope_base,
          d->rope_table_bf16, 0, x, w, 0, kc, vc, w);
  float* y = (float*)malloc(sizeof(float) * (size_t)w * Df);
  for (int t = 0; t < w; ++t) rmsnorm_w(x + (size_t)t * Df, Df, s->fnorm, d->norm_eps, y + (size_t)t * Df);
  if (rows) memcpy(rows, y, sizeof(float) * (size_t)w * Df);
  if (logits) linear(s->FO, d->codebook_size, Df, y + (size_t)(w - 1) * Df, 1, logits);
  free(y);
  free(vc);
  free(kc);
  free(x);
  return 0;
}

/* Cache access for checks at sizes where the oracle cannot prefill by itself: read or
 * overwrite the K/V rows of one layer for slots [s0, s0+n) ([n][Hkv][hd] order). */
int or_kv_io(or_sess* s, int layer, int s0, int n, float* k, float* v, int write) {
  const or_dims* d = &s->d;
  if (layer < 0 || layer >= d->n_layer || s0 < 0 || s0 + n > s->slots) return -1;
  size_t per_layer = (size_t)d->n_kv_head * s->slots * d->head_dim;
  for (int t = 0; t < n; ++t)
    for (int g = 0; g < d->n_kv_head; ++g) {
      float* kc = s->kc + layer * per_layer + ((size_t)g * s->slots + s0 + t) * d->head_dim;
      float* vc = s->vc + layer * per_layer + ((size_t)g * s->slots + s0 + t) * d->head_dim;
      float* ko = k + ((size_t)t * d->n_kv_head + g) * d->head_dim;
      float* vo = v + ((size_t)t * d->n_kv_head + g) * d->head_dim;
      size_t b = sizeof(float) * d->head_dim;
      if (write) {
        memcpy(kc, ko, b);
        memcpy(vc, vo, b);
      } else {
        memcpy(ko, kc, b);
        memcpy(vo, vc, b);
      }
    }
  return 0;
}

/* KV slots [0, n) of one layer from fp16 bit patterns in [kv_head][n][head_dim] order, widened
 * exactly to fp32 (the cache precision of ch.02 §1); the stream's other slots are untouched. */
int or_kv_set_f16(or_sess* s, int layer, int n, const uint16_t* k, const uint16_t* v) {
  const or_dims* d = &s->d;
  if (layer < 0 || layer >= d->n_layer || n < 0 || n > s->slots) return -1;
  size_t per_layer = (size_t)d->n_kv_head * s->slots * d->head_dim;
#pragma omp parallel for schedule(static)
  for (int g = 0; g < d->n_kv_head; ++g)
    for (int t = 0; t < n; ++t) {
      float* kc = s->kc + layer * per_layer + ((size_t)g * s->slots + t) * d->head_dim;
      float* vc = s->vc + layer * per_layer + ((size_t)g * s->slots + t) * d->head_dim;
      const uint16_t* ki = k + ((size_t)g * n + t) * d->head_dim;
      const uint16_t* vi = v + ((size_t)g * n + t) * d->head_dim;
      for (int e = 0; e < d->head_dim; ++e) {
        _Float16 a, b;
        memcpy(&a, ki + e, 2);
        memcpy(&b, vi + e, 2);
        kc[e] = (float)a;
        vc[e] = (float)b;
      }
    }
  return 0;
}

/* The Slow-AR head on a given residual (ch.02 §3.2: final RMSNorm, then logits against the
 * tied embedding table over the whole vocabulary). */
int or_head(const or_sess* s, const float* xlast, float* logits, float* hidden) {
  head(s, xlast, logits, hidden);
  return 0;
}

int or_set_pos(or_sess* s, int pos) {
  if (pos < 0 || pos > s->slots) return -1;
  s->pos = pos;
  return 0;
}

/* --------------------------------------------------------------- sampler */

typedef struct {
  float z;
  int id;
} cand;

static int cand_cmp(const void* a, const void* b) {
  const cand* x = (const cand*)a;
  const cand* y = (const cand*)b;
  if (x->z > y->z) return -1;
  if (x->z < y->z) return 1;
  return (x->id > y->id) - (x->id < y->id);
}

/* One draw ([miz] "parity with upstream": top-k fixed at 30; a draw is argmax(probs / -log u);
 * [ch06] §6 for the repetition-aware settings).  Steps:
 *   z = logits / temperature                      (fp32)
 *   the top_k largest z, descending; equal z -> lower id first
 *   π = softmax of those top_k values             (fp32, max-subtracted)
 *   rank r is kept iff r == 0 or Σ_{s<r} π_s < top_p
 *   return the kept candidate maximising π_r / E_r (E = -log u, given); ties -> lower rank
 * `ids` (nullable) gives the token id of each logit (default: its index).
 * `diag` (nullable, 7 floats) receives, for margin checks: [0] z of rank k-1 minus z of rank k
 * (the top-k cut; +inf if fewer), [1] smallest |Σ_{s<r} π_s - top_p| over ranks 1..k-1,
 * [2] best score, [3] runner-up score (score = log π_r - log E_r), [4] max |logit| over finite
 * entries, [5] rank of the winner, [6] smallest z gap between the winner and its neighbouring
 * ranks (+inf if it has none). */
int or_draw(const float* logits, const int32_t* ids, int n, float temperature, float top_p, int top_k,
            const float* E, float* diag) {
  if (top_k < 1 || top_k > 64 || n <= 0) return -1;
  cand* c = (cand*)malloc(sizeof(cand) * (size_t)n);
  int m = 0;
  float amax = 0.f;
  for (int i = 0; i < n; ++i) {
    if (!isfinite(logits[i])) continue; /* masked entries (−inf) cannot be drawn */
    if (fabsf(logits[i]) > amax) amax = fabsf(logits[i]);
    c[m].z = logits[i] / temperature;
    c[m].id = ids ? ids[i] : i;
    ++m;
  }
  if (m == 0) {
    free(c);
    return -1;
  }
  qsort(c, (size_t)m, sizeof(cand), cand_cmp);
  int k = top_k < m ? top_k : m;
  float pi[64];
  float zmax = c[0].z, sum = 0.f;
  for (int r = 0; r < k; ++r) {
    pi[r] = expf(c[r].z - zmax);
    sum += pi[r];
  }
  for (int r = 0; r < k; ++r) pi[r] = pi[r] / sum;
  float cum = 0.f, pgap = INFINITY;
  int kept = 0;
  for (int r = 0; r < k; ++r) {
    if (r > 0) {
      float g = fabsf(cum - top_p);
      if (g < pgap) pgap = g;
    }
    if (r == 0 || cum < top_p) kept = r + 1;
    else break;
    cum += pi[r];
  }
  int best = 0;
  float bq = pi[0] / E[0];
  for (int r = 1; r < kept; ++r) {
    float q = pi[r] / E[r];
    if (q > bq) {
      best = r;
      bq = q;
    }
  }
  int tok = c[best].id;
  if (diag) {
    float second = -INFINITY;
    for (int r = 0; r < kept; ++r) {
      float sc = logf(pi[r]) - logf(E[r]);
      if (r != best && sc > second) second = sc;
    }
    diag[0] = (k < m) ? c[k - 1].z - c[k].z : INFINITY;
    diag[1] = pgap;
    diag[2] = logf(pi[best]) - logf(E[best]);
    diag[3] = second;
    diag[4] = amax;
    diag[5] = (float)best;
    /* the variates belong to ranks: the winner's token is unambiguous only while its z is apart
     * from the z of the neighbouring ranks */
    float rg = INFINITY;
    if (best > 0) rg = c[best - 1].z - c[best].z;
    if (best + 1 < k && c[best].z - c[best + 1].z < rg) rg = c[best].z - c[best + 1].z;
    diag[6] = rg;
  }
  free(c);
  return tok;
}

/* weight table entry i of a session (the order of or_new's table) */
static wref* table_ref(or_sess* s, int i) {
  const or_dims* d = &s->d;
  if (i < 0 || i >= or_weight_count(d)) return NULL;
  if (i == 0) return &s->E;
  if (i == 1) return &s->CE;
  if (i == 2) return &s->norm;
  i -= 3;
  if (i < 9 * d->n_layer) {
    or_layer* L = &s->slow[i / 9];
    wref* f[9] = {&L->an, &L->wqkv, &L->qn, &L->kn, &L->wo, &L->fn, &L->w1, &L->w3, &L->w2};
    return f[i % 9];
  }
  i -= 9 * d->n_layer;
  if (i == 0) return &s->P;
  if (i == 1) return &s->FE;
  if (i == 2) return &s->fnorm;
  if (i == 3) return &s->FO;
  i -= 4;
  or_layer* L = &s->fast[i / 9];
  wref* f[9] = {&L->an, &L->wqkv, &L->qn, &L->kn, &L->wo, &L->fn, &L->w1, &L->w3, &L->w2};
  return f[i % 9];
}

/* read table entry i from e4m3 codes [rows][cols] and row scales instead */
int or_bind_e4m3(or_sess* s, int i, const uint8_t* codes, const float* scales, int cols) {
  wref* w = table_ref(s, i);
  if (!w || !codes || !scales || cols <= 0) return 1;
  for (int c = 0; c < 256; ++c) g_e4m3[c] = or_e4m3_value(c);
  w->p = codes;
  w->bf16 = 0;
  w->rs = scales;
  w->cols = cols;
  return 0;
}
