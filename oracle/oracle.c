/*
 * oracle.c -- CPU reference for the batch-invariant linear layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  The product path (the
 * CUDA library and its Python binding) never calls it and shares no code with
 * it: no headers, helpers, tables or constants.
 *
 * What it computes, and the passages it follows:
 *   - bf16 storage, fp32 arithmetic.  A bf16 value is the top 16 bits of an
 *     IEEE binary32 value, so decoding is exact.
 *   - GEMM  Y = X . W^T  (the nn.Linear layout) with fp32 accumulation.  Every
 *     output element is one dot product summed sequentially in ascending k:
 *     acc = 0; acc = acc + x_k * w_k.  This is the "a+b+c+d" chain of
 *     CoRun (Padding is Simple and Efficient for Deterministic LLM Inference),
 *     Sec. III-A, Fig. 3, and the non-split reduction of LLM-42, Sec. 2.2,
 *     Fig. 3.  A product of two bf16 values has at most 16 significant bits,
 *     so it is exact in fp32; only the additions round.
 *   - RMSNorm, a per-token reduction over the hidden dimension (LLM-42,
 *     Sec. 2.1).  The pages name the operator but never write its formula; the
 *     reading used here is the usual one:
 *        ss = sum_h x_h^2 (sequential fp32), r = 1 / sqrt(ss / H + eps),
 *        y_h = bf16_rne((x_h * r) * g_h)
 *     with one rounding to bf16 at the end.
 *   - The fused layer RMSNorm -> GEMM is the composition through the bf16
 *     normalised activations.
 *   - Log-softmax of a row of bf16 logits (the lm_head's per-token
 *     log-probabilities), in fp64: x_v - (max + log sum exp(x - max)).
 *   - FP8 (E4M3) with per-token activation scales and per-channel weight
 *     scales: per-row quantisation and the scaled GEMM.
 *   - Decode attention over a paged key/value cache, in fp64: the plain
 *     softmax(scale * q . k) . v of each query head over its request's
 *     positions (grouped-query heads), with no split.
 *   - One decode layer of a Llama-style stack (for the linear-stack
 *     workload): RMSNorm, qkv projection, an attention stand-in for context
 *     length 1 (softmax over one key is exactly 1, so each query head's output
 *     is the value vector of its key/value group), output projection,
 *     residual, RMSNorm, gate/up projection, SiLU(gate) * up, down projection,
 *     residual.
 *
 * Every output row is computed from that row's inputs alone, so the results
 * cannot depend on the number of rows or on the other rows (batch invariance
 * as defined in CoRun, Sec. III-B, Def. 1, and Detent, Sec. 3, Eq. 2, holds by
 * construction).
 *
 * Build with -ffp-contract=off so that no multiply-add is fused: each product
 * and each sum is rounded to fp32 separately, exactly as written; and without
 * gcc's value-range propagation and jump threading, which folded a subnormal
 * quotient to zero in the quantiser (gcc 13, -O2).
 */
#include <float.h>
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* bf16 <-> fp32                                                            */
/* ------------------------------------------------------------------------ */

/* Exact widening: the bf16 bits become the high half of a binary32. */
float oracle_bf16_to_f32(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* Round-to-nearest-even narrowing of a binary32 to bf16.
 * NaN stays NaN (its quiet bit is forced on); everything else adds half an
 * ulp of the 16 dropped bits, plus one more when the kept part is odd (ties go
 * to even), and truncates.  Values past the largest bf16 round to infinity. */
uint16_t oracle_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  if ((u & 0x7fffffffu) > 0x7f800000u) {
    return (uint16_t)((u >> 16) | 0x0040u);
  }
  uint32_t keep_lsb = (u >> 16) & 1u;
  u = u + 0x7fffu + keep_lsb;
  return (uint16_t)(u >> 16);
}

/* ------------------------------------------------------------------------ */
/* A tiny fork/join helper: split [0, total) into nthreads contiguous parts. */
/* Each output element is computed by exactly one thread with the same code */
/* as the single-threaded loop, so the thread count cannot change any bit.  */
/* ------------------------------------------------------------------------ */

typedef void (*range_fn)(void* ctx, int64_t lo, int64_t hi);

typedef struct {
  range_fn fn;
  void* ctx;
  int64_t lo, hi;
} range_job;

static void* range_thread(void* p) {
  range_job* j = (range_job*)p;
  j->fn(j->ctx, j->lo, j->hi);
  return NULL;
}

static void parallel_for(range_fn fn, void* ctx, int64_t total, int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if ((int64_t)nthreads > total) nthreads = (int)(total > 0 ? total : 1);
  if (nthreads == 1) {
    fn(ctx, 0, total);
    return;
  }
  pthread_t tid[256];
  range_job job[256];
  int started[256];
  for (int t = 0; t < nthreads; ++t) {
    job[t].fn = fn;
    job[t].ctx = ctx;
    job[t].lo = total * t / nthreads;
    job[t].hi = total * (t + 1) / nthreads;
    started[t] = pthread_create(&tid[t], NULL, range_thread, &job[t]) == 0;
    if (!started[t]) range_thread(&job[t]); /* no thread: do it inline */
  }
  for (int t = 0; t < nthreads; ++t) {
    if (started[t]) pthread_join(tid[t], NULL);
  }
}

/* ------------------------------------------------------------------------ */
/* RMSNorm                                                                  */
/* ------------------------------------------------------------------------ */

/* One row: ss accumulates x_h * x_h in ascending h; the mean divides by H;
 * r = 1 / sqrt(mean + eps) with the correctly rounded sqrt and division of
 * IEEE binary32; y_h = bf16_rne((x_h * r) * g_h). */
static void rmsnorm_row(const uint16_t* x, const uint16_t* g, uint16_t* y, int64_t H,
                        float eps) {
  float ss = 0.0f;
  for (int64_t h = 0; h < H; ++h) {
    float xh = oracle_bf16_to_f32(x[h]);
    float sq = xh * xh;
    ss = ss + sq;
  }
  float mean = ss / (float)H;
  float r = 1.0f / sqrtf(mean + eps);
  for (int64_t h = 0; h < H; ++h) {
    float xh = oracle_bf16_to_f32(x[h]);
    float scaled = xh * r;
    float v = scaled * oracle_bf16_to_f32(g[h]);
    y[h] = oracle_bf16_rne(v);
  }
}

/* The inverse RMS of one row, as used inside rmsnorm_row. */
float oracle_rmsnorm_inv_rms(const uint16_t* x, int64_t H, float eps) {
  float ss = 0.0f;
  for (int64_t h = 0; h < H; ++h) {
    float xh = oracle_bf16_to_f32(x[h]);
    float sq = xh * xh;
    ss = ss + sq;
  }
  float mean = ss / (float)H;
  return 1.0f / sqrtf(mean + eps);
}

typedef struct {
  const uint16_t *X, *g;
  uint16_t* Y;
  int64_t H;
  float eps;
} rms_ctx;

static void rms_range(void* p, int64_t lo, int64_t hi) {
  rms_ctx* c = (rms_ctx*)p;
  for (int64_t m = lo; m < hi; ++m) rmsnorm_row(c->X + m * c->H, c->g, c->Y + m * c->H, c->H, c->eps);
}

/* X [M,H] bf16, g [H] bf16 -> Y [M,H] bf16. */
void oracle_rmsnorm(const uint16_t* X, const uint16_t* g, uint16_t* Y, int64_t M, int64_t H,
                    float eps, int nthreads) {
  rms_ctx c = {X, g, Y, H, eps};
  parallel_for(rms_range, &c, M, nthreads);
}

/* ------------------------------------------------------------------------ */
/* GEMM  Y = X . W^T                                                        */
/* ------------------------------------------------------------------------ */

/* One output element: the sequential ascending-k fp32 chain. */
static float dot_row(const uint16_t* x, const uint16_t* w, int64_t K) {
  float acc = 0.0f;
  for (int64_t k = 0; k < K; ++k) {
    float p = oracle_bf16_to_f32(x[k]) * oracle_bf16_to_f32(w[k]);
    acc = acc + p;
  }
  return acc;
}

typedef struct {
  const uint16_t *X, *W;
  float* Yf;
  uint16_t* Yb;
  int64_t N, K;
} gemm_ctx;

static void gemm_range(void* p, int64_t lo, int64_t hi) {
  gemm_ctx* c = (gemm_ctx*)p;
  for (int64_t e = lo; e < hi; ++e) {
    int64_t m = e / c->N, n = e % c->N;
    float acc = dot_row(c->X + m * c->K, c->W + n * c->K, c->K);
    if (c->Yf) c->Yf[e] = acc;
    if (c->Yb) c->Yb[e] = oracle_bf16_rne(acc);
  }
}

/* X [M,K] bf16, W [N,K] bf16 -> Yf [M,N] fp32 (may be NULL) and
 * Yb [M,N] bf16 = bf16_rne(Yf) (may be NULL). */
void oracle_gemm(const uint16_t* X, const uint16_t* W, float* Yf, uint16_t* Yb, int64_t M,
                 int64_t N, int64_t K, int nthreads) {
  gemm_ctx c = {X, W, Yf, Yb, N, K};
  parallel_for(gemm_range, &c, M * N, nthreads);
}

typedef struct {
  const uint16_t *X, *W;
  const int64_t *rows, *cols;
  float* out;
  int64_t K;
} sample_ctx;

static void sample_range(void* p, int64_t lo, int64_t hi) {
  sample_ctx* c = (sample_ctx*)p;
  for (int64_t i = lo; i < hi; ++i)
    c->out[i] = dot_row(c->X + c->rows[i] * c->K, c->W + c->cols[i] * c->K, c->K);
}

/* The fp32 result of chosen elements only: out[i] = Y[rows[i], cols[i]].
 * Used to check full-size launches element by element. */
void oracle_gemm_sampled(const uint16_t* X, const uint16_t* W, const int64_t* rows,
                         const int64_t* cols, float* out, int64_t count, int64_t K,
                         int nthreads) {
  sample_ctx c = {X, W, rows, cols, out, K};
  parallel_for(sample_range, &c, count, nthreads);
}

/* Fused layer: Xhat = RMSNorm(X; g, eps) in bf16, then Y = Xhat . W^T.
 * Xhat_out may be NULL; otherwise it receives the bf16 normalised rows. */
void oracle_rmsnorm_gemm(const uint16_t* X, const uint16_t* g, const uint16_t* W, float* Yf,
                         uint16_t* Yb, uint16_t* Xhat_out, int64_t M, int64_t N, int64_t K,
                         float eps, int nthreads) {
  uint16_t* xh = Xhat_out ? Xhat_out : (uint16_t*)malloc((size_t)(M * K) * sizeof(uint16_t));
  if (!xh) return;
  oracle_rmsnorm(X, g, xh, M, K, eps, nthreads);
  oracle_gemm(xh, W, Yf, Yb, M, N, K, nthreads);
  if (!Xhat_out) free(xh);
}

/* ------------------------------------------------------------------------ */
/* Decode-layer glue                                                        */
/* ------------------------------------------------------------------------ */

/* out = bf16_rne(a + b), both operands widened to fp32. */
void oracle_residual_add(const uint16_t* a, const uint16_t* b, uint16_t* out, int64_t count) {
  for (int64_t i = 0; i < count; ++i)
    out[i] = oracle_bf16_rne(oracle_bf16_to_f32(a[i]) + oracle_bf16_to_f32(b[i]));
}

/* SwiGLU activation on a [M, 2*I] gate/up block (gate = columns 0..I-1,
 * up = columns I..2I-1):  out[m,i] = bf16_rne(silu(gate) * up), with
 * silu(v) = v / (1 + exp(-v)) evaluated in fp32. */
void oracle_silu_mul(const uint16_t* gu, uint16_t* out, int64_t M, int64_t I) {
  for (int64_t m = 0; m < M; ++m) {
    for (int64_t i = 0; i < I; ++i) {
      float gate = oracle_bf16_to_f32(gu[m * 2 * I + i]);
      float up = oracle_bf16_to_f32(gu[m * 2 * I + I + i]);
      float e = expf(-gate);
      float den = 1.0f + e;
      float s = gate / den;
      float v = s * up;
      out[m * I + i] = oracle_bf16_rne(v);
    }
  }
}

/* Attention stand-in at context length 1: the qkv row is
 * [q (nq*D) | k (nkv*D) | v (nkv*D)]; query head j reads key/value group
 * j / (nq / nkv), and with one key its softmax weight is exactly 1, so the
 * head's output is that group's v vector copied unchanged. */
void oracle_attention_ctx1(const uint16_t* qkv, uint16_t* out, int64_t M, int64_t nq,
                           int64_t nkv, int64_t D) {
  int64_t width = (nq + 2 * nkv) * D;
  int64_t group = nq / nkv;
  for (int64_t m = 0; m < M; ++m) {
    for (int64_t j = 0; j < nq; ++j) {
      const uint16_t* v = qkv + m * width + (nq + nkv) * D + (j / group) * D;
      for (int64_t d = 0; d < D; ++d) out[m * nq * D + j * D + d] = v[d];
    }
  }
}

/* One decode layer, x_in [M,Hd] -> x_out [M,Hd]:
 *   xn  = RMSNorm(x_in; g_attn)
 *   qkv = xn . Wqkv^T                      Wqkv [(nq+2nkv)*D, Hd]
 *   a   = attention_ctx1(qkv)              [M, nq*D]
 *   o   = a . Wo^T                         Wo [Hd, nq*D]
 *   h   = x_in + o
 *   hn  = RMSNorm(h; g_mlp)
 *   gu  = hn . Wgu^T                       Wgu [2I, Hd]
 *   s   = silu(gate) * up                  [M, I]
 *   d   = s . Wd^T                         Wd [Hd, I]
 *   x_out = h + d
 * Every intermediate is stored as bf16, as a layer of the stack stores it. */
int oracle_decode_layer(const uint16_t* x_in, uint16_t* x_out, const uint16_t* g_attn,
                        const uint16_t* Wqkv, const uint16_t* Wo, const uint16_t* g_mlp,
                        const uint16_t* Wgu, const uint16_t* Wd, int64_t M, int64_t Hd,
                        int64_t nq, int64_t nkv, int64_t D, int64_t I, float eps,
                        int nthreads) {
  int64_t qkv_w = (nq + 2 * nkv) * D;
  uint16_t* xn = (uint16_t*)malloc((size_t)(M * Hd) * 2);
  uint16_t* qkv = (uint16_t*)malloc((size_t)(M * qkv_w) * 2);
  uint16_t* att = (uint16_t*)malloc((size_t)(M * nq * D) * 2);
  uint16_t* o = (uint16_t*)malloc((size_t)(M * Hd) * 2);
  uint16_t* h = (uint16_t*)malloc((size_t)(M * Hd) * 2);
  uint16_t* hn = (uint16_t*)malloc((size_t)(M * Hd) * 2);
  uint16_t* gu = (uint16_t*)malloc((size_t)(M * 2 * I) * 2);
  uint16_t* s = (uint16_t*)malloc((size_t)(M * I) * 2);
  uint16_t* d = (uint16_t*)malloc((size_t)(M * Hd) * 2);
  int ok = xn && qkv && att && o && h && hn && gu && s && d;
  if (ok) {
    oracle_rmsnorm(x_in, g_attn, xn, M, Hd, eps, nthreads);
    oracle_gemm(xn, Wqkv, NULL, qkv, M, qkv_w, Hd, nthreads);
    oracle_attention_ctx1(qkv, att, M, nq, nkv, D);
    oracle_gemm(att, Wo, NULL, o, M, Hd, nq * D, nthreads);
    oracle_residual_add(x_in, o, h, M * Hd);
    oracle_rmsnorm(h, g_mlp, hn, M, Hd, eps, nthreads);
    oracle_gemm(hn, Wgu, NULL, gu, M, 2 * I, Hd, nthreads);
    oracle_silu_mul(gu, s, M, I);
    oracle_gemm(s, Wd, NULL, d, M, Hd, I, nthreads);
    oracle_residual_add(h, d, x_out, M * Hd);
  }
  free(xn); free(qkv); free(att); free(o); free(h); free(hn); free(gu); free(s); free(d);
  return ok ? 0 : -1;
}

/* ------------------------------------------------------------------------ */
/* Log-softmax over a row of logits (the lm_head's per-token log-probabilities)*/
/* ------------------------------------------------------------------------ */

/* One row of V bf16 logits -> V log-probabilities, in fp64:
 *   m = max_v x_v,  s = sum_v exp(x_v - m) (ascending v),  lse = m + log(s),
 *   out_v = x_v - lse.
 * Detent, Sec. 8 (Table 6) and CoRun, Sec. IV compare such per-token
 * log-probabilities bit for bit across batch sizes; the pages give no formula,
 * so the definition above is the textbook one, in fp64.  Rows holding a NaN or
 * a +Inf, and rows that are -Inf everywhere, have no defined distribution:
 * every output is NaN.  Otherwise a -Inf logit has log-probability -Inf.
 * Returns lse (NaN for the undefined rows). */
static double log_softmax_row(const uint16_t* x, int64_t V, double* out) {
  double m = -INFINITY;
  int undefined = 0;
  for (int64_t v = 0; v < V; ++v) {
    const double xv = (double)oracle_bf16_to_f32(x[v]);
    if (isnan(xv) || xv == INFINITY) undefined = 1;
    if (xv > m) m = xv;
  }
  if (m == -INFINITY) undefined = 1;
  double lse = NAN;
  if (!undefined) {
    double sum = 0.0;
    for (int64_t v = 0; v < V; ++v) sum += exp((double)oracle_bf16_to_f32(x[v]) - m);
    lse = m + log(sum);
  }
  if (out) {
    for (int64_t v = 0; v < V; ++v) out[v] = undefined ? NAN : (double)oracle_bf16_to_f32(x[v]) - lse;
  }
  return lse;
}

typedef struct {
  const uint16_t* X;
  const int32_t* ids;
  double* out;
  int64_t V;
} lsm_ctx;

static void lsm_range(void* p, int64_t lo, int64_t hi) {
  lsm_ctx* c = (lsm_ctx*)p;
  for (int64_t r = lo; r < hi; ++r) log_softmax_row(c->X + r * c->V, c->V, c->out + r * c->V);
}

/* X [M,V] bf16 logits -> out [M,V] fp64 log-probabilities. */
void oracle_log_softmax(const uint16_t* X, double* out, int64_t M, int64_t V, int nthreads) {
  lsm_ctx c = {X, NULL, out, V};
  parallel_for(lsm_range, &c, M, nthreads);
}

static void tok_range(void* p, int64_t lo, int64_t hi) {
  lsm_ctx* c = (lsm_ctx*)p;
  for (int64_t r = lo; r < hi; ++r) {
    const int32_t id = c->ids[r];
    const double lse = log_softmax_row(c->X + r * c->V, c->V, NULL);
    c->out[r] = (id < 0 || id >= c->V) ? NAN : (double)oracle_bf16_to_f32(c->X[r * c->V + id]) - lse;
  }
}

/* out[r] = log-probability of token ids[r] in row r of X [M,V]; NaN for an id
 * outside [0, V) (and for the undefined rows). */
void oracle_token_logprobs(const uint16_t* X, const int32_t* ids, double* out, int64_t M, int64_t V,
                           int nthreads) {
  lsm_ctx c = {X, ids, out, V};
  parallel_for(tok_range, &c, M, nthreads);
}

/* ------------------------------------------------------------------------ */
/* FP8 (E4M3) with per-token activation scales and per-channel weight scales  */
/* ------------------------------------------------------------------------ */

/* E4M3, the 8-bit format with 1 sign, 4 exponent (bias 7) and 3 mantissa
 * bits: no infinities; S.1111.111 is NaN; the largest finite value is 448
 * (S.1111.110); exponent field 0 holds the subnormals m/8 * 2^-6.  Decoding is
 * exact in fp32. */
float oracle_e4m3_to_f32(uint8_t c) {
  const int e = (c >> 3) & 15, m = c & 7;
  if (e == 15 && m == 7) return NAN;
  const float v = e == 0 ? ldexpf((float)m, -9) : ldexpf(1.0f + (float)m / 8.0f, e - 7);
  return (c & 0x80) ? -v : v;
}

/* Round to nearest E4M3, ties to the even code (mantissa LSB 0), saturating
 * at +-448; NaN gives 0x7F.  The 127 finite non-negative codes 0x00..0x7E
 * increase with their value, so a binary search finds the two neighbours of
 * |x| and the nearer one wins. */
uint8_t oracle_e4m3_rne_sat(float x) {
  if (isnan(x)) return 0x7F;
  const uint8_t sign = signbit(x) ? 0x80 : 0x00;
  const double a = fabs((double)x);
  if (a >= 448.0) return sign | 0x7E;
  int lo = 0, hi = 0x7E;  /* value(lo) <= a < value(hi) */
  while (hi - lo > 1) {
    const int mid = (lo + hi) / 2;
    if ((double)oracle_e4m3_to_f32((uint8_t)mid) <= a) lo = mid; else hi = mid;
  }
  const double dl = a - (double)oracle_e4m3_to_f32((uint8_t)lo);
  const double dh = (double)oracle_e4m3_to_f32((uint8_t)hi) - a;
  int c;
  if (dl < dh) c = lo;
  else if (dh < dl) c = hi;
  else c = (lo & 1) ? hi : lo;
  return sign | (uint8_t)c;
}

/* Per-row (per-token, or per-channel for weights) quantisation of a bf16 row:
 *   amax = max_k |x_k|;  scale = amax / 448 and inv = 448 / amax (fp32
 *   divisions, once per row);  q_k = e4m3_rne_sat(x_k * inv) (the product
 *   rounded to fp32, then to E4M3).
 * The pages fix no formula; multiplying by the reciprocal scale is the usual
 * form of per-token quantisation.  scale is what dequantises the GEMM's sum.
 * amax == 0 gives scale 1 and inv 1 (zero codes); inv is clamped to the largest
 * finite float when 448 / amax overflows; a NaN or an infinity in the row
 * gives scale NaN and NaN codes.  Detent, Limits: dynamic per-tensor FP8
 * activation scales span the batch; per-token or static scales keep each
 * row's bits its own. */
static void quantize_row(const uint16_t* x, int64_t K, uint8_t* q, float* scale) {
  float amax = 0.0f;
  int bad = 0;
  for (int64_t k = 0; k < K; ++k) {
    const float v = fabsf(oracle_bf16_to_f32(x[k]));
    if (!isfinite(v)) bad = 1;
    else if (v > amax) amax = v;
  }
  if (bad) {
    *scale = NAN;
    for (int64_t k = 0; k < K; ++k) q[k] = 0x7F;
    return;
  }
  const float s = amax == 0.0f ? 1.0f : amax / 448.0f;
  float inv = amax == 0.0f ? 1.0f : 448.0f / amax;
  if (inv > FLT_MAX) inv = FLT_MAX; /* amax below about 1.3e-36: keep the product finite */
  *scale = s;
  for (int64_t k = 0; k < K; ++k) q[k] = oracle_e4m3_rne_sat(oracle_bf16_to_f32(x[k]) * inv);
}

typedef struct {
  const uint16_t* X;
  uint8_t* Q;
  float* S;
  int64_t K;
} quant_ctx;

static void quant_range(void* p, int64_t lo, int64_t hi) {
  quant_ctx* c = (quant_ctx*)p;
  for (int64_t r = lo; r < hi; ++r) quantize_row(c->X + r * c->K, c->K, c->Q + r * c->K, c->S + r);
}

/* X [M,K] bf16 -> Q [M,K] E4M3 codes, scale [M] fp32. */
void oracle_quantize_rows_e4m3(const uint16_t* X, uint8_t* Q, float* scale, int64_t M, int64_t K,
                               int nthreads) {
  quant_ctx c = {X, Q, scale, K};
  parallel_for(quant_range, &c, M, nthreads);
}

typedef struct {
  const uint8_t *Xq, *Wq;
  const float *sx, *sw;
  float* Yf;
  uint16_t* Yb;
  int64_t N, K;
} gemm8_ctx;

/* One output element: acc = sum_k qx_k * qw_k in ascending k (each product of
 * two E4M3 values has at most 8 significant bits, so it is exact in fp32;
 * only the additions round); y = bf16_rne((acc * sx) * sw). */
static void gemm8_range(void* p, int64_t lo, int64_t hi) {
  gemm8_ctx* c = (gemm8_ctx*)p;
  for (int64_t i = lo; i < hi; ++i) {
    const int64_t m = i / c->N, n = i % c->N;
    const uint8_t* x = c->Xq + m * c->K;
    const uint8_t* w = c->Wq + n * c->K;
    float acc = 0.0f;
    for (int64_t k = 0; k < c->K; ++k) {
      const float prod = oracle_e4m3_to_f32(x[k]) * oracle_e4m3_to_f32(w[k]);
      acc = acc + prod;
    }
    if (c->Yf) c->Yf[i] = acc;
    if (c->Yb) c->Yb[i] = oracle_bf16_rne((acc * c->sx[m]) * c->sw[n]);
  }
}

/* Y [M,N] = bf16((Xq . Wq^T) * sx[m] * sw[n]); Yf (may be NULL) gets the
 * unscaled fp32 sums. */
void oracle_gemm_e4m3(const uint8_t* Xq, const float* sx, const uint8_t* Wq, const float* sw, float* Yf,
                      uint16_t* Yb, int64_t M, int64_t N, int64_t K, int nthreads) {
  gemm8_ctx c = {Xq, Wq, sx, sw, Yf, Yb, N, K};
  parallel_for(gemm8_range, &c, M * N, nthreads);
}

/* ------------------------------------------------------------------------ */
/* Decode attention over a paged key/value cache                            */
/* ------------------------------------------------------------------------ */

/* One query token per request (decode).  Request b attends to its first L_b
 * cached positions; query head h reads key/value head h / G, G = Hq / Hkv
 * (grouped-query attention, consecutive query heads share a group).  The plain
 * definition, in fp64:
 *     s_p   = scale * sum_d q_d k_{p,d}                 p = 0 .. L_b - 1
 *     w_p   = exp(s_p - max s) / sum_p' exp(s_p' - max s)
 *     out_d = sum_p w_p v_{p,d}
 * (subtracting the maximum changes no value, only the range of the
 * exponentials).  Position p of request b lives in page block_table[b][p /
 * page_size], row p % page_size; a page holds page_size rows of Hkv heads of D
 * values.  Splitting the positions and combining the partial sums, as
 * FlashDecoding-style kernels do, reaches the same value up to rounding order;
 * Detent (Batch-Invariant LLM Serving and RL Rollouts at Near-Stock Speed),
 * Sec. 7, and LLM-42, Sec. 4.4, fix that split only to make the rounding
 * reproducible.  Here there is no split: the oracle is the definition.
 * L_b = 0 gives zeros (an empty sum).  NaN or +Inf scores give NaN through
 * the IEEE arithmetic of the formula. */
typedef struct {
  const uint16_t *q, *k, *v;
  const int32_t* block_table;
  const int32_t* seq_lens;
  const int64_t* pairs; /* (b, h) pairs to compute, or NULL for all of them */
  double* out;
  int64_t Hq, Hkv, D, page_size, bt_stride;
  double scale;
} attn_ctx;

static void attention_one(const attn_ctx* c, int64_t b, int64_t h, double* out) {
  const int64_t G = c->Hq / c->Hkv, kvh = h / G, L = c->seq_lens[b];
  const uint16_t* q = c->q + (b * c->Hq + h) * c->D;
  for (int64_t d = 0; d < c->D; ++d) out[d] = 0.0;
  if (L <= 0) return;
  double* s = (double*)malloc(sizeof(double) * (size_t)L);
  int64_t* row = (int64_t*)malloc(sizeof(int64_t) * (size_t)L);
  double m = -INFINITY;
  for (int64_t p = 0; p < L; ++p) {
    const int64_t page = c->block_table[b * c->bt_stride + p / c->page_size];
    row[p] = ((page * c->page_size + p % c->page_size) * c->Hkv + kvh) * c->D;
    double dot = 0.0;
    for (int64_t d = 0; d < c->D; ++d)
      dot += (double)oracle_bf16_to_f32(q[d]) * (double)oracle_bf16_to_f32(c->k[row[p] + d]);
    s[p] = c->scale * dot;
    if (s[p] > m) m = s[p];
  }
  double sum = 0.0;
  for (int64_t p = 0; p < L; ++p) {
    s[p] = exp(s[p] - m);
    sum += s[p];
  }
  for (int64_t p = 0; p < L; ++p) {
    const double w = s[p] / sum;
    for (int64_t d = 0; d < c->D; ++d) out[d] += w * (double)oracle_bf16_to_f32(c->v[row[p] + d]);
  }
  free(s);
  free(row);
}

static void attn_range(void* p, int64_t lo, int64_t hi) {
  const attn_ctx* c = (const attn_ctx*)p;
  for (int64_t i = lo; i < hi; ++i) {
    const int64_t b = c->pairs ? c->pairs[2 * i] : i / c->Hq;
    const int64_t h = c->pairs ? c->pairs[2 * i + 1] : i % c->Hq;
    attention_one(c, b, h, c->out + i * c->D);
  }
}

/* q [B,Hq,D] bf16; k_cache, v_cache [num_pages, page_size, Hkv, D] bf16;
 * block_table [B, bt_stride] int32; seq_lens [B] int32.  With pairs == NULL,
 * out [B,Hq,D] fp64 gets every head; otherwise out [n_pairs, D] gets the
 * listed (b, h) pairs. */
void oracle_decode_attention(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                             const int32_t* block_table, int64_t bt_stride, const int32_t* seq_lens,
                             const int64_t* pairs, int64_t n_pairs, double* out, int64_t B, int64_t Hq,
                             int64_t Hkv, int64_t D, int64_t page_size, double scale, int nthreads) {
  attn_ctx c = {q, k_cache, v_cache, block_table, seq_lens, pairs, out, Hq, Hkv, D, page_size,
                bt_stride, scale};
  parallel_for(attn_range, &c, pairs ? n_pairs : B * Hq, nthreads);
}

/* Array forms of the two conversions, for callers that hold whole tensors. */
void oracle_bf16_rne_array(const float* in, uint16_t* out, int64_t count) {
  for (int64_t i = 0; i < count; ++i) out[i] = oracle_bf16_rne(in[i]);
}

void oracle_bf16_to_f32_array(const uint16_t* in, float* out, int64_t count) {
  for (int64_t i = 0; i < count; ++i) out[i] = oracle_bf16_to_f32(in[i]);
}
