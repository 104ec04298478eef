/*
 * moe_oracle.c -- plain, slow fp64 CPU oracle of the W4A16 mixture-of-experts
 * block. TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the
 * benchmark's CPU-baseline leg load it; the product library never does.
 *
 * What it computes follows the description of Qwen3.6-35B-A3B's expert layer
 * in "Perplexity libera Lily, un motor de IA que supera a MLX-LM en Apple
 * Silicon" (diariobitcoin.com):
 *   - section "Qwen3.6 combina tres cargas de trabajo": a router scores all
 *     256 experts and picks 8 per token; one shared expert processes every
 *     token; weights are 4-bit affine in groups of 64 with one bfloat16 scale
 *     and one bfloat16 bias per group;
 *   - section "Las optimizaciones en el prefill": the expert products are
 *     accumulated in FP32 (here: fp64); routing is a histogram, a prefix
 *     scan, a scatter and a block map.
 * Readings taken where the pages are silent (softmax over all experts then
 * renormalised over the selected ones, ties to the lower expert index, SwiGLU
 * experts, shared expert with weight 1, stable token order inside an expert,
 * block map as (expert, first row, rows) triples of BM rows, nibble i of word
 * w holding element 8w+i, w = q*scale + bias with q unsigned) are the plain
 * definitions written out below, one step at a time, with no blocking or
 * reordering.
 *
 * Parity pins: every function is checked against closed forms, brute force,
 * invariants or library routines by the CPU tests; nothing here is shared
 * with the CUDA library.
 *
 * Planted mistakes: building with -DORACLE_PLANT=n (n >= 1) compiles one
 * deliberate bug so the tests can show that some pin catches it.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifndef ORACLE_PLANT
#define ORACLE_PLANT 0
#endif

/* ---------------------------------------------------------------- bf16 --- */

/* exact value of a bfloat16 bit pattern */
double oracle_bf16_to_f64(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* round an fp64 value to bfloat16, nearest-even, in one step */
uint16_t oracle_f64_to_bf16(double v) {
  if (isnan(v)) return 0x7FC0;
  uint16_t sign = signbit(v) ? 0x8000 : 0;
  double a = fabs(v);
  if (a == 0.0) return sign;
  if (isinf(a)) return sign | 0x7F80;
  int e;
  frexp(a, &e);               /* a = m * 2^e, m in [0.5, 1) */
  int ulp_exp = e - 8;        /* 8 significant bits */
  if (ulp_exp < -133) ulp_exp = -133;   /* subnormal spacing 2^-133 */
  double r = nearbyint(ldexp(a, -ulp_exp));   /* default mode: nearest-even */
  double res = ldexp(r, ulp_exp);
  if (res >= 0x1p128) return sign | 0x7F80;
  float f = (float)res;       /* exact: res has <= 8 significant bits */
  uint32_t fu;
  memcpy(&fu, &f, sizeof fu);
  return sign | (uint16_t)((fu >> 16) & 0x7FFF);
}

/* ------------------------------------------------------- 4-bit weights --- */

/* nibble i (0..7) of a packed word: element 8w+i sits in bits 4i..4i+3 */
static unsigned nibble(uint32_t word, int i) {
#if ORACLE_PLANT == 1
  i = 7 - i;                                  /* planted: reversed nibbles */
#endif
  return (word >> (4 * i)) & 15u;
}

/* One dequantised weight W[n][k] of an [N][K] matrix:
 * q[n][k/8] nibble k%8, scale and bias [N][K/G]. */
static double w4_weight(const uint32_t* q, const uint16_t* s, const uint16_t* b,
                        int K, int G, int n, int k) {
  unsigned qv = nibble(q[(size_t)n * (K / 8) + k / 8], k % 8);
#if ORACLE_PLANT == 3
  size_t g = (size_t)n * (K / G) + (k / G) / 2;  /* planted: wrong group */
#else
  size_t g = (size_t)n * (K / G) + k / G;
#endif
  double scale = oracle_bf16_to_f64(s[g]);
  double bias = oracle_bf16_to_f64(b[g]);
#if ORACLE_PLANT == 2
  bias = 0.0;                                 /* planted: bias dropped */
#endif
  return (double)qv * scale + bias;
}

/* W as a dense fp64 [N][K] array */
void oracle_dequant(const uint32_t* q, const uint16_t* s, const uint16_t* b,
                    int N, int K, int G, double* W) {
  for (int n = 0; n < N; ++n)
    for (int k = 0; k < K; ++k)
      W[(size_t)n * K + k] = w4_weight(q, s, b, K, G, n, k);
}

/* ---------------------------------------------------------------- router --- */

/* logits[t][e] = sum_h x[t][h] * Wr[h][e] + bias[e]  (bias may be NULL) */
void oracle_router_logits(const uint16_t* x, int T, int H, const uint16_t* wr,
                          const float* bias, int E, double* logits) {
  for (int t = 0; t < T; ++t)
    for (int e = 0; e < E; ++e) {
      double acc = 0.0;
      for (int h = 0; h < H; ++h)
        acc += oracle_bf16_to_f64(x[(size_t)t * H + h]) *
               oracle_bf16_to_f64(wr[(size_t)h * E + e]);
      if (bias) {
#if ORACLE_PLANT == 9
        acc -= (double)bias[e];               /* planted: bias sign */
#else
        acc += (double)bias[e];
#endif
      }
      logits[(size_t)t * E + e] = acc;
    }
}

/* The value a logit ranks by. The pages say nothing about a NaN score; the
 * reading taken is that a NaN logit counts as -infinity: it ranks below every
 * number (ties among such experts go to the lower index like any other tie)
 * and gets softmax weight zero. -0 and +0 compare equal, so they tie. */
static double rank_value(double l) {
#if ORACLE_PLANT == 13
  return isnan(l) ? INFINITY : l;                /* planted: NaN ranks first */
#else
  return isnan(l) ? -INFINITY : l;
#endif
}

/* is expert a ranked before expert b (higher logit, lower index on ties) */
static int ranks_before(const double* l, int a, int b) {
  double la = rank_value(l[a]), lb = rank_value(l[b]);
#if ORACLE_PLANT == 5
  return la > lb || (la == lb && a > b);         /* planted: ties upward */
#else
  return la > lb || (la == lb && a < b);
#endif
}

/* Top-k of one token's logits by repeated selection; slots in rank order.
 * Weights: softmax over all E experts, then renormalised over the selected
 * ones. gap = logit of rank k minus logit of rank k+1 (INFINITY if k == E). */
void oracle_topk(const double* logits, int T, int E, int k, int32_t* idx,
                 double* w, double* gap) {
  char* taken = (char*)malloc((size_t)E);
  double* p = (double*)malloc(sizeof(double) * (size_t)E);
  for (int t = 0; t < T; ++t) {
    const double* l = logits + (size_t)t * E;
    memset(taken, 0, (size_t)E);
    for (int j = 0; j < k; ++j) {
      int best = -1;
      for (int e = 0; e < E; ++e)
        if (!taken[e] && (best < 0 || ranks_before(l, e, best))) best = e;
      taken[best] = 1;
      idx[(size_t)t * k + j] = best;
    }
    /* runner-up after the k selected */
    int next = -1;
    for (int e = 0; e < E; ++e)
      if (!taken[e] && (next < 0 || ranks_before(l, e, next))) next = e;
    int last = idx[(size_t)t * k + k - 1];
    gap[t] = next < 0 ? INFINITY : rank_value(l[last]) - rank_value(l[next]);
    /* softmax over all experts (a NaN logit as -infinity: weight zero) */
    double mx = rank_value(l[idx[(size_t)t * k]]);
    double z = 0.0;
    for (int e = 0; e < E; ++e) { p[e] = exp(rank_value(l[e]) - mx); z += p[e]; }
    for (int e = 0; e < E; ++e) p[e] /= z;
    /* renormalise over the selected experts */
    double zs = 0.0;
    for (int j = 0; j < k; ++j) zs += p[idx[(size_t)t * k + j]];
    for (int j = 0; j < k; ++j) {
#if ORACLE_PLANT == 6
      w[(size_t)t * k + j] = p[idx[(size_t)t * k + j]];      /* planted */
#else
      w[(size_t)t * k + j] = p[idx[(size_t)t * k + j]] / zs;
#endif
    }
  }
  free(taken);
  free(p);
}

/* --------------------------------------------------------- routing maps --- */

/* Histogram, prefix scan, stable scatter and block map of the routed slots.
 * Slot s = t*k + j. Outputs: cnt[E], off[E+1], tile_off[E+1],
 * perm[T*k] (position -> slot), inv[T*k] (slot -> position),
 * bmap[num_tiles][3] = (expert, first position, rows). Returns num_tiles. */
int oracle_route_maps(const int32_t* idx, int T, int k, int E, int BM,
                      int32_t* cnt, int32_t* off, int32_t* tile_off,
                      int32_t* perm, int32_t* inv, int32_t* bmap) {
  for (int e = 0; e < E; ++e) cnt[e] = 0;
  for (int s = 0; s < T * k; ++s) cnt[idx[s]] += 1;
  off[0] = 0;
  tile_off[0] = 0;
  for (int e = 0; e < E; ++e) {
    off[e + 1] = off[e] + cnt[e];
    tile_off[e + 1] = tile_off[e] + (cnt[e] + BM - 1) / BM;
  }
  int32_t* fill = (int32_t*)malloc(sizeof(int32_t) * (size_t)E);
  for (int e = 0; e < E; ++e) fill[e] = off[e];
#if ORACLE_PLANT == 8
  for (int t = T - 1; t >= 0; --t)            /* planted: unstable order */
#else
  for (int t = 0; t < T; ++t)
#endif
    for (int j = 0; j < k; ++j) {
      int s = t * k + j;
      int pos = fill[idx[s]]++;
      perm[pos] = s;
      inv[s] = pos;
    }
  free(fill);
  for (int e = 0; e < E; ++e)
    for (int i = 0; i < tile_off[e + 1] - tile_off[e]; ++i) {
      int b = tile_off[e] + i;
      int rows = cnt[e] - BM * i;
      bmap[3 * b + 0] = e;
      bmap[3 * b + 1] = off[e] + BM * i;
      bmap[3 * b + 2] = rows < BM ? rows : BM;
    }
  return tile_off[E];
}

/* ------------------------------------------------------------ expert FFN --- */

typedef struct {
  const uint32_t* q;
  const uint16_t* s;
  const uint16_t* b;
} w4ref;

static double silu(double g) {
#if ORACLE_PLANT == 4
  return 1.0 / (1.0 + exp(-g));               /* planted: sigmoid only */
#else
  return g / (1.0 + exp(-g));
#endif
}

/* One SwiGLU expert on one token, fp64:
 *   g[n] = sum_k x[k] Wg[n][k], u[n] = sum_k x[k] Wu[n][k]   (n < I, k < H)
 *   a[n] = silu(g[n]) * u[n]
 *   out[m] = sum_n a[n] Wd[m][n]                            (m < H)
 * gate/up are [I][H] matrices, down is [H][I]. */
static void expert_ffn(const double* x, int H, int I, int G, w4ref gt, w4ref up,
                       w4ref dn, double* a, double* out) {
  for (int n = 0; n < I; ++n) {
    double g = 0.0, u = 0.0;
    for (int k = 0; k < H; ++k) {
      g += x[k] * w4_weight(gt.q, gt.s, gt.b, H, G, n, k);
      u += x[k] * w4_weight(up.q, up.s, up.b, H, G, n, k);
    }
#if ORACLE_PLANT == 7
    a[n] = silu(u) * g;                       /* planted: gate/up swapped */
#else
    a[n] = silu(g) * u;
#endif
  }
  for (int m = 0; m < H; ++m) {
    double d = 0.0;
    for (int n = 0; n < I; ++n) {
#if ORACLE_PLANT == 10
      d += a[n] * w4_weight(dn.q, dn.s, dn.b, H, G, n, m);  /* planted: transposed */
#else
      d += a[n] * w4_weight(dn.q, dn.s, dn.b, I, G, m, n);
#endif
    }
    out[m] = d;
  }
}

/* Expert `e` of a set (arrays [E][N][K/8] etc.) applied to one fp64 token. */
void oracle_expert_ffn(const double* x, int H, int I, int G, int e,
                       const uint32_t* gq, const uint16_t* gs, const uint16_t* gb,
                       const uint32_t* uq, const uint16_t* us, const uint16_t* ub,
                       const uint32_t* dq, const uint16_t* ds, const uint16_t* db,
                       double* out) {
  size_t qa = (size_t)I * H / 8, sa = (size_t)I * H / G;   /* per-expert sizes */
  w4ref gt = {gq + e * qa, gs + e * sa, gb + e * sa};
  w4ref up = {uq + e * qa, us + e * sa, ub + e * sa};
  w4ref dn = {dq + e * qa, ds + e * sa, db + e * sa};
  double* a = (double*)malloc(sizeof(double) * (size_t)I);
  expert_ffn(x, H, I, G, gt, up, dn, a, out);
  free(a);
}

/* -------------------------------------------------------------- MoE layer --- */

typedef struct {
  const uint32_t *gq, *uq, *dq;
  const uint16_t *gs, *gb, *us, *ub, *ds, *db;
} expert_set;

/* y for one token row given its routing: y = shared(x) + sum_j w_j expert_j(x) */
static void layer_token(const double* x, int H, int I, int G, int k,
                        const int32_t* idx, const double* w, const expert_set* routed,
                        const expert_set* shared, double* y, double* d, double* a) {
  size_t qa = (size_t)I * H / 8, sa = (size_t)I * H / G;
  for (int m = 0; m < H; ++m) y[m] = 0.0;
  if (shared) {
    w4ref gt = {shared->gq, shared->gs, shared->gb};
    w4ref up = {shared->uq, shared->us, shared->ub};
    w4ref dn = {shared->dq, shared->ds, shared->db};
    expert_ffn(x, H, I, G, gt, up, dn, a, d);
#if ORACLE_PLANT != 11                          /* planted: shared dropped */
    for (int m = 0; m < H; ++m) y[m] += d[m];
#endif
  }
  for (int j = 0; j < k; ++j) {
    int e = idx[j];
    w4ref gt = {routed->gq + e * qa, routed->gs + e * sa, routed->gb + e * sa};
    w4ref up = {routed->uq + e * qa, routed->us + e * sa, routed->ub + e * sa};
    w4ref dn = {routed->dq + e * qa, routed->ds + e * sa, routed->db + e * sa};
    expert_ffn(x, H, I, G, gt, up, dn, a, d);
    for (int m = 0; m < H; ++m) y[m] += w[j] * d[m];
  }
}

/* Full layer for the token rows listed in `rows` (all rows if rows == NULL,
 * n_rows = T). x is bf16 [T][H]. Per listed row r (output row i):
 *   logits[i][E], idx[i][k], w[i][k], gap[i], y[i][H] (fp64).
 * The shared set may be NULL. nthreads > 1 splits rows across OpenMP threads. */
void oracle_moe_rows(const uint16_t* x, int T, int H, int I, int E, int k, int G,
                     const uint16_t* router_w, const float* router_bias,
                     const uint32_t* gq, const uint16_t* gs, const uint16_t* gb,
                     const uint32_t* uq, const uint16_t* us, const uint16_t* ub,
                     const uint32_t* dq, const uint16_t* ds, const uint16_t* db,
                     const uint32_t* sgq, const uint16_t* sgs, const uint16_t* sgb,
                     const uint32_t* suq, const uint16_t* sus, const uint16_t* sub,
                     const uint32_t* sdq, const uint16_t* sds, const uint16_t* sdb,
                     const int32_t* rows, int n_rows, int nthreads,
                     double* logits, int32_t* idx, double* w, double* gap, double* y) {
  expert_set routed = {gq, uq, dq, gs, gb, us, ub, ds, db};
  expert_set shared = {sgq, suq, sdq, sgs, sgb, sus, sub, sds, sdb};
  const expert_set* sh = sgq ? &shared : NULL;
  (void)T;
  (void)nthreads;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads > 0 ? nthreads : 1)
#endif
  for (int i = 0; i < n_rows; ++i) {
    int r = rows ? rows[i] : i;
    double* xr = (double*)malloc(sizeof(double) * (size_t)H);
    double* d = (double*)malloc(sizeof(double) * (size_t)H);
    double* a = (double*)malloc(sizeof(double) * (size_t)I);
    for (int h = 0; h < H; ++h) xr[h] = oracle_bf16_to_f64(x[(size_t)r * H + h]);
    oracle_router_logits(x + (size_t)r * H, 1, H, router_w, router_bias, E,
                         logits + (size_t)i * E);
    oracle_topk(logits + (size_t)i * E, 1, E, k, idx + (size_t)i * k,
                w + (size_t)i * k, gap + i);
    layer_token(xr, H, I, G, k, idx + (size_t)i * k, w + (size_t)i * k, &routed, sh,
                y + (size_t)i * H, d, a);
    free(xr);
    free(d);
    free(a);
  }
}

/* Residual stack step: x_next = bf16(x + alpha * y) elementwise. */
void oracle_residual(const uint16_t* x, const double* y, int n, double alpha,
                     uint16_t* x_next) {
  for (int i = 0; i < n; ++i)
    x_next[i] = oracle_f64_to_bf16(oracle_bf16_to_f64(x[i]) + alpha * y[i]);
}

/* RMS normalisation of each row (the stacked layers' input):
 *   out[r][h] = bf16(x[r][h] / sqrt(mean_h x[r][h]^2 + eps)), in fp64. */
void oracle_rmsnorm(const uint16_t* x, int rows, int H, double eps, uint16_t* out) {
  for (int r = 0; r < rows; ++r) {
    double ss = 0.0;
    for (int h = 0; h < H; ++h) {
      double v = oracle_bf16_to_f64(x[(size_t)r * H + h]);
      ss += v * v;
    }
#if ORACLE_PLANT == 12
    double den = ss / H + eps;                /* planted: square root dropped */
#else
    double den = sqrt(ss / H + eps);
#endif
    for (int h = 0; h < H; ++h)
      out[(size_t)r * H + h] = oracle_f64_to_bf16(oracle_bf16_to_f64(x[(size_t)r * H + h]) / den);
  }
}

/* Storage accounting of the 4-bit affine format: bits per weight for group
 * size G with one 16-bit scale and one 16-bit bias per group. */
double oracle_w4_bits_per_weight(int G) { return 4.0 + 2.0 * 16.0 / (double)G; }

int oracle_planted(void) { return ORACLE_PLANT; }
