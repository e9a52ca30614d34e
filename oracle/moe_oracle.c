/*
 * moe_oracle.c -- plain fp64 CPU oracle for the NVFP4 MoE expert layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls
 * this file; only the tests, the smoke check and the benchmark's CPU-baseline
 * leg do.  It shares no code, header, table or constant with the CUDA path.
 *
 * What it computes follows "perf: gather tokens per MoE expert, run large NVFP4
 * GEMMs on bf16 tensor cores #91" (gllm pull request page), sections "What
 * changes" (MoE gather; RowSlice / WeightedRowSum; bf16 NVFP4 GEMM), together
 * with the NVFP4 encoding the layer is specified with: e2m1 4-bit codes, one
 * e4m3 (E4M3FN) scale per 16 elements along K, one fp32 global per matrix.
 *
 * The oracle evaluates the plain definition, pair by pair: for every (token t,
 * slot j) with expert e = ids[t,j]
 *     h_i = g_up[e] * sum_c Wup_e[i][c] * x[t][c]                (fp64)
 *     a_i = bf16_rne(max(h_i, 0)^2)                              (rounded once)
 *     y_c = g_dn[e] * sum_i Wdn_e[c][i] * a_i                    (fp64)
 * and then
 *     out[t][c] = bf16_rne(dst[t][c] + sum_{j=0..k-1} w[t,j] * y^{(t,j)}_c)
 * with W[r][c] = e2m1(code) * e4m3(scale[r][c/16]) decoded exactly.
 *
 * The gated variant (the "gate-up" expert kernel of "nvfp4 experts cuda:
 * decode kernels stall on load latency ... #2265", section "What ncu shows",
 * whose warps read "both rows' inputs" per output) replaces the up step by
 *     g_i = g_gate[e] * sum_c Wgate_e[i][c] * x[t][c]           (fp64)
 *     u_i = g_up[e]   * sum_c Wup_e[i][c]   * x[t][c]           (fp64)
 *     a_i = bf16_rne(silu(g_i) * u_i),  silu(g) = g / (1 + exp(-g))
 * (the SwiGLU form of the models that page names; the page does not print the
 * activation, so this is the reading taken).  The
 * gathering into packed rows only reorders this work, so the oracle computes
 * the routing (counts, offsets, stable permutation) separately, and uses it
 * only to report per-row intermediates in packed-row order.
 *
 * Readings of the pages that the oracle fixes (each is a choice where the pages
 * are silent): element 2i of a code byte is its low nibble; weights are
 * [out][in] with K contiguous; rows of one expert are ordered by ascending pair
 * index p = t*k + j; an id outside [0, E) drops its pair (contributes 0).
 *
 * Parity pins: every function here is pinned by tests that do not re-type its
 * formulas (exhaustive format checks against torch's float8_e4m3fn and the OCP
 * e2m1 table, exact-rational bf16 rounding, numpy argsort/bincount for the
 * routing, an independent dense-masked numpy restatement, numpy matvecs, exact
 * dyadic cases, and hand-valued WeightedRowSum fixtures).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define OR_OK 0
#define OR_ERR_ARG (-1)
#define OR_ERR_NAN (-2)
#define OR_ERR_NOMEM (-3)

/* ---------------------------------------------------------------- formats */

/* e2m1: sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0.
 * exponent 0 is subnormal: 0.5 * m.  Otherwise 2^(e-1) * (1 + m/2). */
double or_e2m1(unsigned code) {
  unsigned s = (code >> 3) & 1u, e = (code >> 1) & 3u, m = code & 1u;
  double mag = (e == 0) ? 0.5 * (double)m : ldexp(1.0 + 0.5 * (double)m, (int)e - 1);
  return s ? -mag : mag;
}

/* e4m3 (E4M3FN, bias 7): sign bit 7, exponent bits 6..3, mantissa bits 2..0.
 * exponent 0 is subnormal: (m/8) * 2^-6.  S.1111.111 is NaN; there is no inf.
 * Returns OR_ERR_NAN for the two NaN bytes. */
int or_e4m3(unsigned byte, double *out) {
  unsigned s = (byte >> 7) & 1u, e = (byte >> 3) & 15u, m = byte & 7u;
  if (e == 15u && m == 7u) return OR_ERR_NAN;
  double mag = (e == 0) ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + (double)m / 8.0, (int)e - 7);
  *out = s ? -mag : mag;
  return OR_OK;
}

/* bf16 value of a bit pattern (widening through fp32, which is exact). */
double or_bf16_to_double(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* Round a double straight to bf16, to nearest with ties to even, in one step
 * (no detour through fp32, which could round twice).  bf16 has 8 significant
 * bits, exponents down to -126 for normals and a subnormal quantum of 2^-133. */
uint16_t or_bf16_from_double(double v) {
  if (isnan(v)) return 0x7FC0;
  uint16_t sign = signbit(v) ? 0x8000 : 0;
  double a = fabs(v);
  if (a == 0.0) return sign;
  if (isinf(a)) return (uint16_t)(sign | 0x7F80);
  int e2;
  (void)frexp(a, &e2);          /* a = f * 2^e2, f in [0.5, 1)  =>  a in [2^(e2-1), 2^e2) */
  int binade = e2 - 1;          /* a in [2^binade, 2^(binade+1)) */
  if (binade < -126) binade = -126;
  double q = ldexp(1.0, binade - 7); /* spacing of bf16 values in this binade */
  double n = a / q;             /* exact: division by a power of two */
  double fl = floor(n);
  double frac = n - fl;
  double r;
  if (frac > 0.5) r = fl + 1.0;
  else if (frac < 0.5) r = fl;
  else r = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
  double res = r * q;
  if (res >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80);
  float f = (float)res;         /* exact: res has at most 8 significant bits */
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)(sign | (uint16_t)((u >> 16) & 0x7FFF));
}

/* One decoded NVFP4 weight W[r][c] of a row-major [rows][K] matrix whose
 * codes are [rows][K/2] bytes and block scales [rows][K/16] e4m3 bytes.
 * The per-tensor global is NOT applied here. */
static int weight_at(const uint8_t *codes, const uint8_t *scales, int64_t K, int64_t r, int64_t c,
                     double *w) {
  uint8_t byte = codes[r * (K / 2) + c / 2];
  unsigned code = (c % 2 == 0) ? (byte & 0x0Fu) : (byte >> 4);
  double s;
  if (or_e4m3(scales[r * (K / 16) + c / 16], &s) != OR_OK) return OR_ERR_NAN;
  *w = or_e2m1(code) * s;
  return OR_OK;
}

/* Full fp64 dequantisation of a [rows][K] NVFP4 matrix (tests use it). */
int or_dequant(const uint8_t *codes, const uint8_t *scales, int64_t rows, int64_t K, double *out) {
  if (K % 16 != 0 || rows < 0) return OR_ERR_ARG;
  int bad = 0;
#pragma omp parallel for schedule(static) reduction(| : bad)
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < K; ++c)
      if (weight_at(codes, scales, K, r, c, &out[r * K + c]) != OR_OK) bad = 1;
  return bad ? OR_ERR_NAN : OR_OK;
}

/* ---------------------------------------------------------------- routing */

/* Histogram, exclusive prefix sum and stable scatter of the (token, slot)
 * pairs p = t*k + j into packed rows grouped by expert.  Row r = offsets[e] + (rank of p among the pairs of expert e,
 * by ascending p).  perm_pair[r] = p, inv[p] = r; a pair whose id is outside
 * [0, E) is dropped: inv[p] = -1 and it takes no row.  Returns the number of
 * dropped pairs (>= 0) or an error (< 0).  (Pull request #91, "What changes",
 * MoE gather: every picked (token, expert) pair owns one row of an n*topK-row
 * buffer whose rows are grouped by expert.) */
int64_t or_routing(const int32_t *ids, int64_t n, int k, int E, int32_t *counts, int32_t *offsets,
                   int32_t *perm_pair, int32_t *inv) {
  if (n < 0 || k <= 0 || E <= 0) return OR_ERR_ARG;
  int64_t R = n * (int64_t)k, dropped = 0;
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (int64_t p = 0; p < R; ++p) {
    int32_t e = ids[p];
    if (e >= 0 && e < E) counts[e] += 1;
    else dropped += 1;
  }
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  int32_t *fill = (int32_t *)malloc(sizeof(int32_t) * (size_t)E);
  if (!fill) return OR_ERR_NOMEM;
  for (int e = 0; e < E; ++e) fill[e] = offsets[e];
  for (int64_t p = 0; p < R; ++p) {
    int32_t e = ids[p];
    if (e >= 0 && e < E) {
      int32_t r = fill[e]++;
      perm_pair[r] = (int32_t)p;
      inv[p] = r;
    } else {
      inv[p] = -1;
    }
  }
  free(fill);
  return dropped;
}

/* ------------------------------------------------------ dense NVFP4 matmul */

/* C = g * (A . W^T) for bf16 A [M][K] and NVFP4 W [N][K].  Pull request #91,
 * "What changes", bf16 NVFP4 GEMM: the unpacked weight is code value times
 * block scale (exact), the per-tensor global multiplies the product as the
 * GEMM's alpha, and the activation enters in bf16.  epilogue 0 writes the fp64 result to out_f64
 * [M][N]; epilogue 1 writes bf16_rne(max(C,0)^2) to out_bf16 [M][N]. */
int or_nvfp4_matmul(const uint16_t *A, const uint8_t *codes, const uint8_t *scales, double g, int64_t M,
                    int64_t N, int64_t K, int epilogue, double *out_f64, uint16_t *out_bf16) {
  if (K % 16 != 0 || M < 0 || N < 0) return OR_ERR_ARG;
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (int64_t m = 0; m < M; ++m) {
    for (int64_t j = 0; j < N; ++j) {
      double acc = 0.0, w;
      for (int64_t c = 0; c < K; ++c) {
        if (weight_at(codes, scales, K, j, c, &w) != OR_OK) { bad = 1; w = 0.0; }
        acc += w * or_bf16_to_double(A[m * K + c]);
      }
      double h = g * acc;
      if (epilogue == 0) out_f64[m * N + j] = h;
      else {
        double r = h > 0.0 ? h : 0.0;
        out_bf16[m * N + j] = or_bf16_from_double(r * r);
      }
    }
  }
  return bad ? OR_ERR_NAN : OR_OK;
}

/* ------------------------------------------------------- WeightedRowSum */

/* dst[i][c] = bf16_rne(dst[i][c] + sum_{j=0..k-1} w[i][j] * src[rows[i][j]][c]),
 * the terms added in increasing j (pull request #91, "What changes",
 * WeightedRowSum: each dst row gets its k weighted source rows added in one
 * set order, so the result does not depend on how the work is scheduled).  A row index outside [0, src_rows)
 * contributes nothing and is counted; the count is returned. */
int64_t or_weighted_row_sum(uint16_t *dst, const double *src, const int32_t *rows, const float *w,
                            int64_t n, int k, int64_t cols, int64_t src_rows) {
  int64_t skipped = 0;
  for (int64_t i = 0; i < n; ++i)
    for (int j = 0; j < k; ++j) {
      int32_t r = rows[i * k + j];
      if (r < 0 || r >= src_rows) skipped += 1;
    }
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    for (int64_t c = 0; c < cols; ++c) {
      double acc = or_bf16_to_double(dst[i * cols + c]);
      for (int j = 0; j < k; ++j) {
        int32_t r = rows[i * k + j];
        if (r < 0 || r >= src_rows) continue;
        acc += (double)w[i * k + j] * src[(int64_t)r * cols + c];
      }
      dst[i * cols + c] = or_bf16_from_double(acc);
    }
  }
  return skipped;
}

/* ------------------------------------------------------ the whole layer */

/* Tokens per block of the layer evaluation below: the intermediates of one
 * block's pairs are held in memory at once, and each of the three steps of a
 * block runs its independent output elements in parallel. */
#define OR_TOKEN_BLOCK 32

/* The MoE expert layer on the plain per-pair definition (see file header).
 * act = 0: relu^2 (gate arrays unused, may be NULL); act = 1: the gated form,
 * gate_codes/gate_scales [E][I][H/2], [E][I][H/16] and gate_global [E].
 * dst [n][H] bf16 is updated in place.  Optional outputs (NULL to skip), all
 * indexed by packed row r = inv[p] from or_routing on the same ids:
 *   a_rows     [R][I] bf16  the intermediate (relu^2 or silu*up) of every kept pair
 *   a_rows_f64 [R][I] fp64  the same intermediate before its bf16 rounding
 *   y_rows     [R][H] fp64  the down-projection of every kept pair
 *   out_f64    [n][H] fp64  dst + sum_j w y before the final rounding
 * tok_begin/tok_end restrict the work to a token range (for bounded samples);
 * pass 0 and n for all tokens.  Returns 0, or < 0 on a bad argument / NaN scale.
 *
 * Evaluation order: tokens in blocks of OR_TOKEN_BLOCK; within a block, first
 * every (pair, intermediate feature) value, then every (pair, output column)
 * down value, then every (token, column) weighted sum.  Each value is one
 * plain loop in the order the formulas give (ascending c for the up and gate
 * sums, ascending i for the down sum, j = 0..k-1 onto dst), so running the
 * independent values on several threads changes no result. */
int or_moe_forward_act(int64_t n, int H, int I, int E, int k, const uint16_t *x, const int32_t *ids,
                       const float *topk_w, const uint8_t *up_codes, const uint8_t *up_scales,
                       const uint8_t *dn_codes, const uint8_t *dn_scales, const float *up_global,
                       const float *dn_global, int act, const uint8_t *gate_codes, const uint8_t *gate_scales,
                       const float *gate_global, uint16_t *dst, uint16_t *a_rows, double *a_rows_f64,
                       double *y_rows, double *out_f64, int64_t tok_begin, int64_t tok_end) {
  if (n < 0 || H <= 0 || I <= 0 || E <= 0 || k <= 0 || H % 32 || I % 32) return OR_ERR_ARG;
  if (act != 0 && act != 1) return OR_ERR_ARG;
  if (act == 1 && (!gate_codes || !gate_scales || !gate_global)) return OR_ERR_ARG;
  if (tok_begin < 0 || tok_end > n || tok_begin > tok_end) return OR_ERR_ARG;
  int64_t R = n * (int64_t)k;
  int32_t *inv = NULL;
  if (a_rows || a_rows_f64 || y_rows) {
    int32_t *counts = (int32_t *)malloc(sizeof(int32_t) * (size_t)E);
    int32_t *offsets = (int32_t *)malloc(sizeof(int32_t) * (size_t)(E + 1));
    int32_t *perm = (int32_t *)malloc(sizeof(int32_t) * (size_t)(R > 0 ? R : 1));
    inv = (int32_t *)malloc(sizeof(int32_t) * (size_t)(R > 0 ? R : 1));
    if (!counts || !offsets || !perm || !inv) {
      free(counts); free(offsets); free(perm); free(inv);
      return OR_ERR_NOMEM;
    }
    or_routing(ids, n, k, E, counts, offsets, perm, inv);
    free(counts); free(offsets); free(perm);
  }
  const int64_t up_mat = (int64_t)I * H; /* elements per expert matrix */
  const int64_t bp = (int64_t)OR_TOKEN_BLOCK * k; /* pairs per block, at most */
  double *a = (double *)malloc(sizeof(double) * (size_t)(bp * I)); /* [pair of block][i] */
  double *y = (double *)malloc(sizeof(double) * (size_t)(bp * H)); /* [pair of block][c] */
  if (!a || !y) {
    free(a); free(y); free(inv);
    return OR_ERR_NOMEM;
  }
  int bad = 0;
  for (int64_t t0 = tok_begin; t0 < tok_end; t0 += OR_TOKEN_BLOCK) {
    const int64_t t1 = t0 + OR_TOKEN_BLOCK < tok_end ? t0 + OR_TOKEN_BLOCK : tok_end;
    const int64_t np = (t1 - t0) * k; /* pairs of this block: p = t0*k + q */
    /* up projection and the activation, one bf16 rounding per value */
#pragma omp parallel for schedule(dynamic, 8) reduction(| : bad)
    for (int64_t qi = 0; qi < np * I; ++qi) {
      const int64_t q = qi / I, p = t0 * k + q;
      const int i = (int)(qi % I);
      const int64_t t = p / k;
      int32_t e = ids[p];
      if (e < 0 || e >= E) continue; /* dropped pair */
      const uint8_t *uc = up_codes + (int64_t)e * (up_mat / 2);
      const uint8_t *us = up_scales + (int64_t)e * (up_mat / 16);
      double h = 0.0, w;
      for (int c = 0; c < H; ++c) {
        if (weight_at(uc, us, H, i, c, &w) != OR_OK) { bad = 1; w = 0.0; }
        h += w * or_bf16_to_double(x[t * H + c]);
      }
      h *= (double)up_global[e];
      double av;
      if (act == 0) {
        double r = h > 0.0 ? h : 0.0;
        av = r * r;
      } else {
        const uint8_t *gc = gate_codes + (int64_t)e * (up_mat / 2);
        const uint8_t *gs = gate_scales + (int64_t)e * (up_mat / 16);
        double gv = 0.0;
        for (int c = 0; c < H; ++c) {
          if (weight_at(gc, gs, H, i, c, &w) != OR_OK) { bad = 1; w = 0.0; }
          gv += w * or_bf16_to_double(x[t * H + c]);
        }
        gv *= (double)gate_global[e];
        av = gv / (1.0 + exp(-gv)) * h;
      }
      uint16_t ab = or_bf16_from_double(av);
      a[q * I + i] = or_bf16_to_double(ab);
      if (a_rows) a_rows[(int64_t)inv[p] * I + i] = ab;
      if (a_rows_f64) a_rows_f64[(int64_t)inv[p] * I + i] = av;
    }
    /* down projection of the rounded intermediate */
#pragma omp parallel for schedule(dynamic, 8) reduction(| : bad)
    for (int64_t qc = 0; qc < np * H; ++qc) {
      const int64_t q = qc / H, p = t0 * k + q;
      const int c = (int)(qc % H);
      int32_t e = ids[p];
      if (e < 0 || e >= E) continue; /* dropped pair */
      const uint8_t *dc = dn_codes + (int64_t)e * (up_mat / 2);
      const uint8_t *ds = dn_scales + (int64_t)e * (up_mat / 16);
      double s = 0.0, w;
      for (int i = 0; i < I; ++i) {
        if (weight_at(dc, ds, I, c, i, &w) != OR_OK) { bad = 1; w = 0.0; }
        s += w * a[q * I + i];
      }
      y[q * H + c] = s * (double)dn_global[e];
      if (y_rows) y_rows[(int64_t)inv[p] * H + c] = y[q * H + c];
    }
    /* fixed-order weighted sum onto the pre-filled dst, one rounding */
#pragma omp parallel for schedule(static)
    for (int64_t tc = 0; tc < (t1 - t0) * H; ++tc) {
      const int64_t t = t0 + tc / H;
      const int c = (int)(tc % H);
      double acc = or_bf16_to_double(dst[t * H + c]);
      for (int j = 0; j < k; ++j) {
        int64_t p = t * k + j;
        int32_t e = ids[p];
        if (e < 0 || e >= E) continue; /* dropped pair */
        acc += (double)topk_w[p] * y[(p - t0 * k) * H + c];
      }
      if (out_f64) out_f64[t * H + c] = acc;
      dst[t * H + c] = or_bf16_from_double(acc);
    }
  }
  free(a); free(y); free(inv);
  return bad ? OR_ERR_NAN : OR_OK;
}

/* The relu^2 layer (act = 0 of or_moe_forward_act). */
int or_moe_forward(int64_t n, int H, int I, int E, int k, const uint16_t *x, const int32_t *ids,
                   const float *topk_w, const uint8_t *up_codes, const uint8_t *up_scales,
                   const uint8_t *dn_codes, const uint8_t *dn_scales, const float *up_global,
                   const float *dn_global, uint16_t *dst, uint16_t *a_rows, double *a_rows_f64, double *y_rows,
                   double *out_f64, int64_t tok_begin, int64_t tok_end) {
  return or_moe_forward_act(n, H, I, E, k, x, ids, topk_w, up_codes, up_scales, dn_codes, dn_scales, up_global,
                            dn_global, 0, NULL, NULL, NULL, dst, a_rows, a_rows_f64, y_rows, out_f64, tok_begin,
                            tok_end);
}

/* The router that produces the layer's input (the step before the path; the
 * layer's synthetic workloads are routed this way: fp32 logits, an optional
 * per-expert bias added to them, top-k, softmax renormalised over the k
 * picked).  For each token t:
 *   z[e]   = logits[t][e] + bias[e]          (one fp32 addition, bias may be NULL)
 *   ids[t] = the k experts with the largest z in descending order, equal z
 *            taken lower index first
 *   w[t][j] = exp(z_j - z_0) / sum_i exp(z_i - z_0) over the k picked (fp64,
 *            stored fp32)
 *   counts[e] = number of tokens that picked e (if counts is not NULL)
 * Selection is a plain scan per pick: the next pick is the best z among the
 * experts after the previous pick in the order (z descending, index
 * ascending).  Returns OR_ERR_ARG for k outside [1, E]. */
int or_router_topk(const float *logits, const float *bias, int64_t n, int E, int k, int32_t *ids, float *w,
                   int32_t *counts) {
  if (n < 0 || E <= 0 || k < 1 || k > E) return OR_ERR_ARG;
  if (counts)
    for (int e = 0; e < E; ++e) counts[e] = 0;
  double *zp = (double *)malloc(sizeof(double) * (size_t)k);
  if (!zp) return OR_ERR_NOMEM;
  for (int64_t t = 0; t < n; ++t) {
    const float *row = logits + t * E;
    float prev_z = 0.0f;
    int prev_e = -1;
    for (int j = 0; j < k; ++j) {
      int best = -1;
      float best_z = 0.0f;
      for (int e = 0; e < E; ++e) {
        const float z = bias ? row[e] + bias[e] : row[e];
        /* only experts after the previous pick in the order (z desc, e asc) */
        if (prev_e >= 0 && !(z < prev_z || (z == prev_z && e > prev_e))) continue;
        if (best < 0 || z > best_z) {
          best = e;
          best_z = z;
        }
      }
      if (best < 0) { /* no expert left: k > E, or a broken order rule */
        free(zp);
        return OR_ERR_ARG;
      }
      ids[t * k + j] = best;
      zp[j] = (double)best_z;
      prev_z = best_z;
      prev_e = best;
      if (counts) counts[best] += 1;
    }
    double sum = 0.0;
    for (int j = 0; j < k; ++j) sum += exp(zp[j] - zp[0]);
    for (int j = 0; j < k; ++j) w[t * k + j] = (float)(exp(zp[j] - zp[0]) / sum);
  }
  free(zp);
  return OR_OK;
}

/* Number of OpenMP threads the oracle runs with (1 without OpenMP). */
int or_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
