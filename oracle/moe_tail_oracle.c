/*
 * moe_tail_oracle.c -- plain, slow, CPU reference of the decode-step MoE layer tail.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or call this file:
 * only the test suite, the smoke check and the benchmark's CPU-baseline leg use it.  It
 * shares no code, header, table or helper with the CUDA library.
 *
 * What it computes (sources are the pages' titles and sections):
 *   - "[AMD] integrate kimi k3 monokernel" (sglang #43481, body of sgl-amd-mono #83, the K2
 *     layer-tail launch), section "Kernel Replacement": the layer tail after attention is
 *     post-attention fused add + RMSNorm -> router GEMV -> top-k gating softmax -> routed
 *     MXFP4 experts (gate/up "g1u1", SiLU, down) -> bf16 shared expert (gate_up, SiLU*mul,
 *     down) -> combine; section "Refusals": norm_topk_prob is required, norm/router/shared
 *     expert are bf16, routed experts are MXFP4; section "Kernel checks": the outputs are
 *     `out` and `res_out` (the updated residual).
 *   - "glm53: Long-context indexer ..." (sgl-amd-mono #86, quoting #85), Modifications table
 *     row 9 (top-8 tie shortcut): only an exact tie of the maximum runs the expert-id
 *     reduction, ties go to the lowest id and the pick order is unchanged; row 10: the
 *     router activations are stored as bf16 before the GEMV.
 *   - OCP MXFP4: 32-element blocks of E2M1 codes that share one E8M0 scale 2^(s-127).
 *   - "Split the Kimi3 AttnRes mix across CTAs for decode rows" (voipmonitor/flare #11):
 *     the second workload, one call of the AttnRes residual mix + RMSNorm
 *     (oracle_attnres_mix at the end of this file, with its own readings).
 *
 * Arithmetic: every sum and product is in double precision.  The only roundings are the
 * bf16 storage points a real layer has (the new residual, the normalised activations, the
 * SiLU*up intermediate of each expert, the output) and the fp32 router logits that rank
 * the experts.  There is no blocking, fusion, deduplication or reordering: every
 * (row, pick) pair runs its expert on its own, in the order the definition states.
 *
 * Readings where the pages are silent (each one is listed in the design notes):
 *   - RMSNorm is the plain form n = r * rstd * gamma (gamma is not offset by one).
 *   - The norm is taken of the bf16-rounded residual r_new, the value written back.
 *   - Experts are ranked by fp32 logit, descending, ties to the lowest id; the weights are
 *     the softmax over all experts renormalised over the picked ones (norm_topk_prob).
 *   - w13 rows [0, I) are the gate projection, rows [I, 2I) the up projection.
 *   - Byte j of a packed MXFP4 row holds element 2j in its low nibble, 2j+1 in its high one.
 *   - SiLU(z) = z / (1 + exp(-z)); mid = bf16(SiLU(gate) * up).
 *   - out = bf16(sum over picks of w * y + shared); the residual becomes r_new.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- number formats ---- */

/* OCP E2M1: sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0; exponent 0 is
 * subnormal (0 or 0.5).  The magnitudes are 0, 0.5, 1, 1.5, 2, 3, 4, 6. */
double oracle_e2m1(int code) {
  static const double mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
  double v = mag[code & 7];
  return (code & 8) ? -v : v;
}

/* OCP E8M0: an exponent alone, value 2^(s-127).  0xFF (NaN) is never produced by the
 * input generator and is not given a meaning here. */
double oracle_e8m0(int s) { return ldexp(1.0, s - 127); }

/* bf16 (1 sign, 8 exponent, 7 mantissa bits) bits -> double. */
double oracle_bf16_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* double -> bf16 bits, round to nearest, ties to even, with subnormals and overflow to
 * infinity.  The value is rounded once, directly from double. */
uint16_t oracle_bf16_round(double d) {
  if (isnan(d)) return 0x7FC0;
  uint16_t sign = signbit(d) ? 0x8000 : 0;
  double a = fabs(d);
  if (a == 0.0) return sign;
  if (isinf(a)) return sign | 0x7F80;
  int ex;
  frexp(a, &ex);            /* a = m * 2^ex, m in [0.5, 1) */
  int e = ex - 1;           /* a in [2^e, 2^(e+1)) */
  if (e < -126) e = -126;   /* subnormal range shares the quantum of the smallest binade */
  double q = ldexp(1.0, e - 7);
  double r = a / q;         /* exact: division by a power of two */
  double fl = floor(r);
  double frac = r - fl;
  if (frac > 0.5 || (frac == 0.5 && fmod(fl, 2.0) != 0.0)) fl += 1.0;
  double v = fl * q;
  if (v >= ldexp(1.0, 128)) return sign | 0x7F80;
  float f = (float)v;       /* exact: v has at most 8 significant bits */
  uint32_t u;
  memcpy(&u, &f, 4);
  return sign | (uint16_t)(u >> 16);
}

/* One MXFP4 element: index k of a packed row (codes: K/2 bytes, scales: K/32 bytes). */
double oracle_mxfp4_elem(const uint8_t* codes, const uint8_t* scales, int64_t k) {
  uint8_t byte = codes[k / 2];
  int code = (k % 2 == 0) ? (byte & 0x0F) : (byte >> 4);
  return oracle_e2m1(code) * oracle_e8m0(scales[k / 32]);
}

/* Decode a whole packed row of K elements into doubles: block b's scale 2^(s_b - 127)
 * times the E2M1 value of each of its 32 elements (same values as oracle_mxfp4_elem). */
void oracle_mxfp4_dequant_row(const uint8_t* codes, const uint8_t* scales, int64_t K,
                              double* out) {
  for (int64_t b = 0; b * 32 < K; ++b) {
    const double sc = oracle_e8m0(scales[b]);
    for (int64_t k = b * 32; k < b * 32 + 32 && k < K; ++k) {
      uint8_t byte = codes[k / 2];
      int code = (k % 2 == 0) ? (byte & 0x0F) : (byte >> 4);
      out[k] = oracle_e2m1(code) * sc;
    }
  }
}

double oracle_silu(double z) { return z / (1.0 + exp(-z)); }

/* ------------------------------------------------- step 1: residual add + RMSNorm ---- */

/* For each row r: s = x + residual; r_new = bf16(s); rstd = 1/sqrt(mean(r_new^2) + eps);
 * n = bf16(r_new * rstd * gamma).  All arrays [R, H] (gamma [H]) as bf16 bits. */
void oracle_add_rmsnorm(int R, int H, const uint16_t* x, const uint16_t* residual,
                        const uint16_t* gamma, double eps, uint16_t* r_new, uint16_t* n,
                        double* rstd_out) {
  for (int r = 0; r < R; ++r) {
    const uint16_t* xr = x + (int64_t)r * H;
    const uint16_t* rr = residual + (int64_t)r * H;
    uint16_t* nr = r_new + (int64_t)r * H;
    double ss = 0.0;
    for (int h = 0; h < H; ++h) {
      double s = oracle_bf16_to_double(xr[h]) + oracle_bf16_to_double(rr[h]);
      nr[h] = oracle_bf16_round(s);
      double v = oracle_bf16_to_double(nr[h]);
      ss += v * v;
    }
    double rstd = 1.0 / sqrt(ss / H + eps);
    if (rstd_out) rstd_out[r] = rstd;
    for (int h = 0; h < H; ++h) {
      double v = oracle_bf16_to_double(nr[h]) * rstd * oracle_bf16_to_double(gamma[h]);
      n[(int64_t)r * H + h] = oracle_bf16_round(v);
    }
  }
}

/* ------------------------------------------------------------ step 2: router ---- */

/* logits[r, e] = sum_h n[r, h] * W_r[e, h], in double.  W_r is [E, H] bf16. */
void oracle_router(int R, int H, int E, const uint16_t* n, const uint16_t* w_r,
                   double* logits) {
  for (int r = 0; r < R; ++r)
    for (int e = 0; e < E; ++e) {
      double acc = 0.0;
      for (int h = 0; h < H; ++h)
        acc += oracle_bf16_to_double(n[(int64_t)r * H + h]) *
               oracle_bf16_to_double(w_r[(int64_t)e * H + h]);
      logits[(int64_t)r * E + e] = acc;
    }
}

/* ------------------------------------------------ step 3: softmax + top-k + renorm ---- */

/* For each row: rank experts by (fp32(logit) descending, id ascending) and take the first
 * k; p = softmax over all E experts of the double logits; the weight of pick i is
 * p_i / sum of the picked p.  ids/wts are [R, k] in pick order. */
void oracle_topk(int R, int E, int k, const double* logits, int32_t* ids, double* wts) {
  char* taken = (char*)malloc((size_t)E);
  double* p = (double*)malloc(sizeof(double) * (size_t)E);
  for (int r = 0; r < R; ++r) {
    const double* l = logits + (int64_t)r * E;
    memset(taken, 0, (size_t)E);
    for (int i = 0; i < k; ++i) {
      int best = -1;
      float bestv = 0.0f;
      for (int e = 0; e < E; ++e) {
        if (taken[e]) continue;
        float v = (float)l[e];
        if (best < 0 || v > bestv) { best = e; bestv = v; }  /* strict: ties keep lowest id */
      }
      taken[best] = 1;
      ids[(int64_t)r * k + i] = best;
    }
    double mx = l[0];
    for (int e = 1; e < E; ++e) if (l[e] > mx) mx = l[e];
    double z = 0.0;
    for (int e = 0; e < E; ++e) { p[e] = exp(l[e] - mx); z += p[e]; }
    double zsel = 0.0;
    for (int i = 0; i < k; ++i) zsel += p[ids[(int64_t)r * k + i]] / z;
    for (int i = 0; i < k; ++i)
      wts[(int64_t)r * k + i] = (p[ids[(int64_t)r * k + i]] / z) / zsel;
  }
  free(taken);
  free(p);
}

/* ---------------------------------------------------- step 4: one routed expert ---- */

/* One row's activation n[H] through expert e: g_j, u_j over dequantised w13 rows j and
 * I + j; mid_j = bf16(SiLU(g_j) * u_j); y_h = sum_j mid_j * deq(w2[e][h, j]).
 * w13_codes [E, 2I, H/2], w13_scales [E, 2I, H/32], w2_codes [E, H, I/2],
 * w2_scales [E, H, I/32].  mid_out (bf16 bits, [I]) may be NULL. */
void oracle_expert(int H, int I, int e, const uint16_t* n, const uint8_t* w13_codes,
                   const uint8_t* w13_scales, const uint8_t* w2_codes,
                   const uint8_t* w2_scales, double* y, uint16_t* mid_out) {
  double* nd = (double*)malloc(sizeof(double) * (size_t)H);
  double* wrow = (double*)malloc(sizeof(double) * (size_t)(H > I ? H : I));
  double* mid = (double*)malloc(sizeof(double) * (size_t)I);
  for (int h = 0; h < H; ++h) nd[h] = oracle_bf16_to_double(n[h]);
  const int64_t c13 = (int64_t)H / 2, s13 = (int64_t)H / 32;
  const uint8_t* e13c = w13_codes + (int64_t)e * 2 * I * c13;
  const uint8_t* e13s = w13_scales + (int64_t)e * 2 * I * s13;
  for (int j = 0; j < I; ++j) {
    double g = 0.0, u = 0.0;
    oracle_mxfp4_dequant_row(e13c + (int64_t)j * c13, e13s + (int64_t)j * s13, H, wrow);
    for (int h = 0; h < H; ++h) g += nd[h] * wrow[h];
    oracle_mxfp4_dequant_row(e13c + (int64_t)(I + j) * c13, e13s + (int64_t)(I + j) * s13, H,
                             wrow);
    for (int h = 0; h < H; ++h) u += nd[h] * wrow[h];
    uint16_t mb = oracle_bf16_round(oracle_silu(g) * u);
    if (mid_out) mid_out[j] = mb;
    mid[j] = oracle_bf16_to_double(mb);
  }
  const int64_t c2 = (int64_t)I / 2, s2 = (int64_t)I / 32;
  const uint8_t* e2c = w2_codes + (int64_t)e * H * c2;
  const uint8_t* e2s = w2_scales + (int64_t)e * H * s2;
  for (int h = 0; h < H; ++h) {
    oracle_mxfp4_dequant_row(e2c + (int64_t)h * c2, e2s + (int64_t)h * s2, I, wrow);
    double acc = 0.0;
    for (int j = 0; j < I; ++j) acc += mid[j] * wrow[j];
    y[h] = acc;
  }
  free(nd);
  free(wrow);
  free(mid);
}

/* ------------------------------------------------------ step 5: shared expert ---- */

/* One row's activation n[H] through the bf16 shared expert: ws13 [2Is, H] (gate rows
 * first), ws2 [H, Is].  ms_j = bf16(SiLU(gs_j) * us_j); ys_h = sum_j ms_j * ws2[h, j]. */
void oracle_shared(int H, int Is, const uint16_t* n, const uint16_t* ws13,
                   const uint16_t* ws2, double* ys, uint16_t* ms_out) {
  double* nd = (double*)malloc(sizeof(double) * (size_t)H);
  double* ms = (double*)malloc(sizeof(double) * (size_t)Is);
  for (int h = 0; h < H; ++h) nd[h] = oracle_bf16_to_double(n[h]);
  for (int j = 0; j < Is; ++j) {
    double g = 0.0, u = 0.0;
    for (int h = 0; h < H; ++h) {
      g += nd[h] * oracle_bf16_to_double(ws13[(int64_t)j * H + h]);
      u += nd[h] * oracle_bf16_to_double(ws13[(int64_t)(Is + j) * H + h]);
    }
    uint16_t mb = oracle_bf16_round(oracle_silu(g) * u);
    if (ms_out) ms_out[j] = mb;
    ms[j] = oracle_bf16_to_double(mb);
  }
  for (int h = 0; h < H; ++h) {
    double acc = 0.0;
    for (int j = 0; j < Is; ++j) acc += ms[j] * oracle_bf16_to_double(ws2[(int64_t)h * Is + j]);
    ys[h] = acc;
  }
  free(nd);
  free(ms);
}

/* ------------------------------------- step 0 (optional): attention out_proj ---- */

/* The attention output projection in front of the tail ("[AMD] integrate kimi k3
 * monokernel" page, Kernel Replacement row 1, a bf16 x bf16 GEMM): attn [R, Ha] bf16,
 * w_o [H, Ha] bf16 -> x [R, H] = bf16(sum_j attn[r, j] * w_o[h, j]), the sum in fp64. */
void oracle_out_proj(int R, int Ha, int H, const uint16_t* attn, const uint16_t* w_o,
                     uint16_t* x_out) {
  double* a = (double*)malloc(sizeof(double) * (size_t)Ha);
  for (int r = 0; r < R; ++r) {
    for (int j = 0; j < Ha; ++j) a[j] = oracle_bf16_to_double(attn[(int64_t)r * Ha + j]);
    for (int h = 0; h < H; ++h) {
      double acc = 0.0;
      for (int j = 0; j < Ha; ++j) acc += a[j] * oracle_bf16_to_double(w_o[(int64_t)h * Ha + j]);
      x_out[(int64_t)r * H + h] = oracle_bf16_round(acc);
    }
  }
  free(a);
}

/* ---------------------------------------------- step 5b: shared-expert gate ---- */

/* The optional sigmoid gate of the shared expert ("[AMD] integrate kimi k3 monokernel" page,
 * Kernel Replacement row "shared expert gate, sigmoid and add"): one weight vector g [H];
 * per row gate = sigmoid(sum_h n_h * g_h) = 1 / (1 + e^-z), in fp64. */
void oracle_shared_gate(int R, int H, const uint16_t* n, const uint16_t* g, double* gate) {
  for (int r = 0; r < R; ++r) {
    double z = 0.0;
    for (int h = 0; h < H; ++h)
      z += oracle_bf16_to_double(n[(int64_t)r * H + h]) * oracle_bf16_to_double(g[h]);
    gate[r] = 1.0 / (1.0 + exp(-z));
  }
}

/* ------------------------------------------------------------ the whole tail ---- */

typedef struct {
  int R, H, E, k, I, Is;
  const uint16_t* n;
  const int32_t* ids;
  const uint8_t *w13c, *w13s, *w2c, *w2s;
  const uint16_t *ws13, *ws2;
  double* y;   /* [R, k, H] */
  double* ys;  /* [R, H] */
  int next_task, n_tasks;
  pthread_mutex_t lock;
} oracle_job_t;

/* Task t < R*k: routed pick (r, i) = (t / k, t % k); t >= R*k: shared expert of row t-R*k.
 * Each task writes its own output row, so the results do not depend on the thread count. */
static void* oracle_worker(void* arg) {
  oracle_job_t* J = (oracle_job_t*)arg;
  for (;;) {
    pthread_mutex_lock(&J->lock);
    int t = J->next_task++;
    pthread_mutex_unlock(&J->lock);
    if (t >= J->n_tasks) break;
    if (t < J->R * J->k) {
      int r = t / J->k;
      oracle_expert(J->H, J->I, J->ids[t], J->n + (int64_t)r * J->H, J->w13c, J->w13s, J->w2c,
                    J->w2s, J->y + (int64_t)t * J->H, NULL);
    } else {
      int r = t - J->R * J->k;
      oracle_shared(J->H, J->Is, J->n + (int64_t)r * J->H, J->ws13, J->ws2,
                    J->ys + (int64_t)r * J->H, NULL);
    }
  }
  return NULL;
}

/* The whole layer tail for R rows.  Inputs are bf16 bits except the MXFP4 arrays (u8).
 * residual_io is read and then overwritten with r_new; out receives the MoE output.
 * ws_gate (bf16 [H]) may be NULL: without it the shared expert's output enters the combine
 * as it is, with it multiplied by the row's gate (oracle_shared_gate).
 * ids_out [R, k], wts_out [R, k], logits_out [R, E] and out_exact [R, H] (the output
 * before its bf16 rounding) may be NULL.
 * nthreads >= 1 splits the independent (row, pick) tasks over threads. */
int oracle_moe_tail_gated(int R, int H, int E, int k, int I, int Is, double eps,
                          const uint16_t* x, uint16_t* residual_io, const uint16_t* gamma,
                          const uint16_t* w_r, const uint8_t* w13_codes,
                          const uint8_t* w13_scales, const uint8_t* w2_codes,
                          const uint8_t* w2_scales, const uint16_t* ws13, const uint16_t* ws2,
                          const uint16_t* ws_gate, uint16_t* out, int32_t* ids_out,
                          double* wts_out, double* logits_out, double* out_exact,
                          int nthreads) {
  if (R < 1 || H < 32 || E < 1 || k < 1 || k > E || I < 32 || Is < 1 || H % 32 || I % 32)
    return -1;
  uint16_t* r_new = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)R * H);
  uint16_t* n = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)R * H);
  double* logits = (double*)malloc(sizeof(double) * (size_t)R * E);
  int32_t* ids = (int32_t*)malloc(sizeof(int32_t) * (size_t)R * k);
  double* wts = (double*)malloc(sizeof(double) * (size_t)R * k);
  double* y = (double*)malloc(sizeof(double) * (size_t)R * k * H);
  double* ys = (double*)malloc(sizeof(double) * (size_t)R * H);
  double* gate = (double*)malloc(sizeof(double) * (size_t)R);

  oracle_add_rmsnorm(R, H, x, residual_io, gamma, eps, r_new, n, NULL);
  for (int r = 0; r < R; ++r) gate[r] = 1.0;
  if (ws_gate) oracle_shared_gate(R, H, n, ws_gate, gate);
  oracle_router(R, H, E, n, w_r, logits);
  oracle_topk(R, E, k, logits, ids, wts);

  oracle_job_t J;
  J.R = R; J.H = H; J.E = E; J.k = k; J.I = I; J.Is = Is;
  J.n = n; J.ids = ids;
  J.w13c = w13_codes; J.w13s = w13_scales; J.w2c = w2_codes; J.w2s = w2_scales;
  J.ws13 = ws13; J.ws2 = ws2; J.y = y; J.ys = ys;
  J.next_task = 0; J.n_tasks = R * k + R;
  pthread_mutex_init(&J.lock, NULL);
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if (nthreads == 1) {
    oracle_worker(&J);
  } else {
    pthread_t th[256];
    int started = 0;
    for (int t = 0; t < nthreads; ++t)
      if (pthread_create(&th[t], NULL, oracle_worker, &J) == 0) ++started;
    if (started == 0) oracle_worker(&J);
    for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
  }
  pthread_mutex_destroy(&J.lock);

  for (int r = 0; r < R; ++r)
    for (int h = 0; h < H; ++h) {
      double acc = 0.0;
      for (int i = 0; i < k; ++i)
        acc += wts[(int64_t)r * k + i] * y[((int64_t)r * k + i) * H + h];
      acc += (ws_gate ? gate[r] * ys[(int64_t)r * H + h] : ys[(int64_t)r * H + h]);
      if (out_exact) out_exact[(int64_t)r * H + h] = acc;
      out[(int64_t)r * H + h] = oracle_bf16_round(acc);
    }
  memcpy(residual_io, r_new, sizeof(uint16_t) * (size_t)R * H);
  if (ids_out) memcpy(ids_out, ids, sizeof(int32_t) * (size_t)R * k);
  if (wts_out) memcpy(wts_out, wts, sizeof(double) * (size_t)R * k);
  if (logits_out) memcpy(logits_out, logits, sizeof(double) * (size_t)R * E);
  free(r_new); free(n); free(logits); free(ids); free(wts); free(y); free(ys); free(gate);
  return 0;
}

/* The tail without a shared-expert gate. */
int oracle_moe_tail(int R, int H, int E, int k, int I, int Is, double eps,
                    const uint16_t* x, uint16_t* residual_io, const uint16_t* gamma,
                    const uint16_t* w_r, const uint8_t* w13_codes, const uint8_t* w13_scales,
                    const uint8_t* w2_codes, const uint8_t* w2_scales, const uint16_t* ws13,
                    const uint16_t* ws2, uint16_t* out, int32_t* ids_out, double* wts_out,
                    double* logits_out, double* out_exact, int nthreads) {
  return oracle_moe_tail_gated(R, H, E, k, I, Is, eps, x, residual_io, gamma, w_r, w13_codes,
                               w13_scales, w2_codes, w2_scales, ws13, ws2, NULL, out, ids_out,
                               wts_out, logits_out, out_exact, nthreads);
}

/* ------------------------------ second workload: AttnRes residual mix + RMSNorm ---- */

/* "Split the Kimi3 AttnRes mix across CTAs for decode rows" (voipmonitor/flare #11),
 * Description and commit message: one call of the mix adds the sublayer output into the
 * current block's running sum (the prefix), commits a finished block, mixes the block
 * sources with softmax weights from per-source dot and square-sum reductions, and applies
 * the RMSNorm to the mixture.  The page gives no formulas; the readings taken here are:
 *   - prefix' = bf16(prefix + sub), one rounding of the exact sum;
 *   - the sources of row r, in this order, are the committed blocks 0 .. n_blocks-1 of the
 *     row and prefix';
 *   - a commit stores prefix' as block n_blocks and leaves the prefix at zero; the mixture
 *     of that call is over the same sources (the block just stored is prefix');
 *   - score_i = (q . v_i) / sqrt(mean(v_i^2) + eps): one learned query vector q [H]
 *     against each source RMS-normalised without a weight; alpha = softmax(score);
 *   - mix = bf16(sum_i alpha_i v_i); y = bf16(mix * rstd(mix) * gamma) with
 *     rstd(mix) = 1 / sqrt(mean(mix^2) + eps) of the bf16 mixture (the layer's input norm).
 * Layouts (bf16 bits): sub, prefix_io, mix, y [R, H]; blocks [n_blocks + 1, R, H], block b
 * of row r at (b * R + r) * H, block n_blocks written only on a commit; q, gamma [H].
 * alpha_out [R, n_blocks + 1] and score_out [R, n_blocks + 1] may be NULL.
 * Returns 0, or -1 for shapes it does not take. */
int oracle_attnres_mix(int R, int H, int n_blocks, int commit, double eps,
                       const uint16_t* sub, uint16_t* prefix_io, uint16_t* blocks,
                       const uint16_t* q, const uint16_t* gamma, uint16_t* mix, uint16_t* y,
                       double* alpha_out, double* score_out) {
  if (R < 1 || H < 1 || n_blocks < 0) return -1;
  const int S = n_blocks + 1;
  uint16_t* pnew = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)H);
  double* score = (double*)malloc(sizeof(double) * (size_t)S);
  double* alpha = (double*)malloc(sizeof(double) * (size_t)S);
  double* acc = (double*)malloc(sizeof(double) * (size_t)H);
  for (int r = 0; r < R; ++r) {
    const uint16_t* o = sub + (int64_t)r * H;
    uint16_t* p = prefix_io + (int64_t)r * H;
    /* residual add */
    for (int h = 0; h < H; ++h)
      pnew[h] = oracle_bf16_round(oracle_bf16_to_double(p[h]) + oracle_bf16_to_double(o[h]));
    /* scores of the sources against q */
    for (int i = 0; i < S; ++i) {
      const uint16_t* v = i < n_blocks ? blocks + ((int64_t)i * R + r) * H : pnew;
      double ss = 0.0, dot = 0.0;
      for (int h = 0; h < H; ++h) {
        const double vh = oracle_bf16_to_double(v[h]);
        ss += vh * vh;
        dot += oracle_bf16_to_double(q[h]) * vh;
      }
      score[i] = dot / sqrt(ss / H + eps);
    }
    /* softmax over the sources */
    double mx = score[0];
    for (int i = 1; i < S; ++i)
      if (score[i] > mx) mx = score[i];
    double den = 0.0;
    for (int i = 0; i < S; ++i) {
      alpha[i] = exp(score[i] - mx);
      den += alpha[i];
    }
    for (int i = 0; i < S; ++i) alpha[i] /= den;
    /* mixture of the sources, then the RMSNorm of the bf16 mixture */
    for (int h = 0; h < H; ++h) acc[h] = 0.0;
    for (int i = 0; i < S; ++i) {
      const uint16_t* v = i < n_blocks ? blocks + ((int64_t)i * R + r) * H : pnew;
      for (int h = 0; h < H; ++h) acc[h] += alpha[i] * oracle_bf16_to_double(v[h]);
    }
    double ssm = 0.0;
    for (int h = 0; h < H; ++h) {
      const uint16_t b = oracle_bf16_round(acc[h]);
      mix[(int64_t)r * H + h] = b;
      const double m = oracle_bf16_to_double(b);
      ssm += m * m;
    }
    const double rstd = 1.0 / sqrt(ssm / H + eps);
    for (int h = 0; h < H; ++h)
      y[(int64_t)r * H + h] = oracle_bf16_round(
          oracle_bf16_to_double(mix[(int64_t)r * H + h]) * rstd * oracle_bf16_to_double(gamma[h]));
    /* commit, or keep the running sum */
    if (commit) {
      memcpy(blocks + ((int64_t)n_blocks * R + r) * H, pnew, sizeof(uint16_t) * (size_t)H);
      memset(p, 0, sizeof(uint16_t) * (size_t)H);
    } else {
      memcpy(p, pnew, sizeof(uint16_t) * (size_t)H);
    }
    for (int i = 0; i < S; ++i) {
      if (alpha_out) alpha_out[(int64_t)r * S + i] = alpha[i];
      if (score_out) score_out[(int64_t)r * S + i] = score[i];
    }
  }
  free(pnew); free(score); free(alpha); free(acc);
  return 0;
}
