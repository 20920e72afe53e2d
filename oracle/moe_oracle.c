/*
 * moe_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, fp64 CPU reference of one routed sparse Mixture-of-Experts
 * FFN layer forward pass.  It exists to check the CUDA library against; it is
 * never part of the product path.  Only the test-suite, the smoke check and
 * the benchmark's CPU-baseline leg may load it.  It shares no code, header or
 * table with the CUDA library.
 *
 * What it computes, and where that is stated:
 *
 *  - Router: "Systems engineering playbook: optimizing Qwen 3.5-397B MoE on
 *    Ironwood (TPU7x)", section 1 "Qwen 3.5 architecture overview", subsection
 *    "Sparse Mixture-of-Experts (MoE)": the router gate projects the token
 *    representation, a softmax over the 512 experts is formed and the top 10
 *    routed experts are selected.  The selected probabilities are renormalised
 *    to sum to one (the layer's configuration states this; the page's own
 *    formula survives only as an image caption).
 *  - Shared expert: same subsection: a shared-expert path that always runs and
 *    is added to the routed sum (weight one, no gate).
 *  - Routing metadata blob: same page, section 3 "Sharding strategy and
 *    distributed collectives", "3-to-2 All-Gather optimisation": expert ids
 *    and top-k weights of equal shape are stacked on a new axis, bit-cast and
 *    packed into one dense int32 array.  Layout here: [T][2][k], ids first.
 *  - Dispatch: same page, section 3, "Option B": each device filters the
 *    tokens routed to its experts; here that is the stable grouping of
 *    (token, slot) pairs by expert.
 *  - Expert FFN: SwiGLU (gate, up, SiLU times up, down), the expert form the
 *    layer's configuration names.
 *  - W4A16: "vLLM TPU Inference v0.31.0: hierarchical MoE dispatch and W4A16",
 *    section on 4-bit weight support: symmetric int4 weights in the
 *    pack-quantized layout with per-group scales, activations not quantised.
 *
 * Readings taken where the pages are silent (each is restated in the design
 * notes of the repository):
 *  R1  The logit that decides routing is the fp64 sum, in index order
 *      d = 0..D-1 starting from +0.0, of the products x[t,d]*Wr[e,d] (each
 *      product of two bf16 values is exact in fp64), plus the fp32 bias
 *      widened to fp64, added last.
 *  R2  Top-k order is (logit descending, expert index ascending): an exact tie
 *      goes to the lower expert index.
 *  R3  The k selected ids of a token are stored in ascending expert index
 *      order; each weight sits beside its id.
 *  R4  Weights: p = softmax over all E logits, then w_j = p[id_j] / sum_j p.
 *  R5  Pairs p = t*k + j are grouped by expert, stable in p (equivalently in
 *      token index, since a token's ids are distinct).
 *  R6  W_gate_up of an expert is [2I][D]: rows 0..I-1 gate, I..2I-1 up;
 *      W_down is [D][I].  Both are K-major (rows are output features).
 *  R7  int4 packing: 8 values per int32 along K, in pair order: value 2i of
 *      the 8 in bits [4i, 4i+4) and value 2i+1 in bits [16+4i, 20+4i)
 *      (i = 0..3), two's complement.  Scale: one bf16 per (row, group of
 *      `group` consecutive K); group 0 means channel-wise, one scale per row
 *      (the release note's other supported scale strategy).  Dequantised
 *      weight = q * s, exact in fp64.
 *  R8  Everything after routing is computed in fp64 with no intermediate
 *      rounding.
 *  R21 NaN logits (a NaN in the token row or the router row): a NaN ranks
 *      below every number, NaNs among themselves by index, so a token always
 *      gets k distinct ids.  The weights depend only on the selected logits
 *      (the renormalisation cancels the full denominator): a NaN among the
 *      unselected logits does not reach them; a selected NaN makes them NaN.
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -shared -fPIC (contraction is off
 * so that x86 and Arm hosts give the same bits).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_EINVAL -1
#define ORACLE_ENOMEM -2

/* bf16 bit pattern -> fp64.  bf16 is the upper half of an IEEE binary32. */
static double bf16_to_f64(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Signed value j (0..7) of a packed int32 word (reading R7: value 2i at bit
 * 4i, value 2i+1 at bit 16+4i). */
static int nibble_s4(int32_t word, int j) {
  const int shift = 4 * (j >> 1) + 16 * (j & 1);
  uint32_t n = (((uint32_t)word) >> shift) & 0xFu;
  return n >= 8 ? (int)n - 16 : (int)n;
}

/* A weight matrix of `rows` x `cols`, either bf16 or packed int4 + scales. */
typedef struct {
  int rows, cols, quant, group;
  const uint16_t *bf16;  /* quant == 0: [rows][cols]             */
  const int32_t *q;      /* quant == 1: [rows][cols/8]           */
  const uint16_t *s;     /* quant == 1: [rows][cols/group] bf16 (group 0: [rows]) */
} wview;

/* Scales per row: cols/group, or 1 for channel-wise scales (group 0). */
static int group_len(const wview *w) { return w->group > 0 ? w->group : w->cols; }

/* Row `r` of W as fp64 values (dequantised exactly when quant == 1). */
static void load_row(const wview *w, int r, double *out) {
  if (w->quant == 0) {
    const uint16_t *p = w->bf16 + (size_t)r * w->cols;
    for (int c = 0; c < w->cols; ++c) out[c] = bf16_to_f64(p[c]);
  } else {
    const int g = group_len(w);
    const int32_t *q = w->q + (size_t)r * (w->cols / 8);
    const uint16_t *s = w->s + (size_t)r * (w->cols / g);
    for (int c = 0; c < w->cols; ++c)
      out[c] = (double)nibble_s4(q[c / 8], c % 8) * bf16_to_f64(s[c / g]);
  }
}

/* Index-order fp64 dot product. */
static double dot(const double *a, const double *b, int n) {
  double acc = 0.0;
  for (int i = 0; i < n; ++i) acc += a[i] * b[i];
  return acc;
}

static double silu(double a) { return a / (1.0 + exp(-a)); }

/* ------------------------------------------------------------------ */
/* Router logits (reading R1).  z: [T][E].                             */
/* ------------------------------------------------------------------ */
int oracle_router_logits(int T, int D, int E, const uint16_t *x,
                         const uint16_t *wr, const float *bias, double *z) {
  if (T < 0 || D < 1 || E < 1 || !x || !wr || !z) return ORACLE_EINVAL;
  double *wd = (double *)malloc(sizeof(double) * (size_t)E * D);
  if (!wd) return ORACLE_ENOMEM;
  for (size_t i = 0; i < (size_t)E * D; ++i) wd[i] = bf16_to_f64(wr[i]);
  int err = ORACLE_OK;
#pragma omp parallel
  {
    double *xd = (double *)malloc(sizeof(double) * (size_t)D);
    if (!xd) {
#pragma omp atomic write
      err = ORACLE_ENOMEM;
    } else {
#pragma omp for schedule(static)
      for (int t = 0; t < T; ++t) {
        for (int d = 0; d < D; ++d) xd[d] = bf16_to_f64(x[(size_t)t * D + d]);
        for (int e = 0; e < E; ++e) {
          double s = dot(xd, wd + (size_t)e * D, D);
          if (bias) s += (double)bias[e];
          z[(size_t)t * E + e] = s;
        }
      }
      free(xd);
    }
  }
  free(wd);
  return err;
}

/* ------------------------------------------------------------------ */
/* Top-k selection and weights for one token (readings R2, R3, R4,     */
/* R21).                                                               */
/* ------------------------------------------------------------------ */
/* Does logit a rank above logit b?  Numbers by value; a NaN ranks below every
   number and never above another NaN (reading R21).  Equal ranks keep the
   lower index because experts are visited in ascending order. */
static int ranks_above(double a, double b) {
  if (isnan(a)) return 0;
  return isnan(b) || a > b;
}

static void select_token(int E, int k, const double *z, int32_t *ids,
                         double *w, unsigned char *taken) {
  memset(taken, 0, (size_t)E);
  /* k passes of "largest remaining logit, lowest index on a tie". */
  for (int j = 0; j < k; ++j) {
    int best = -1;
    for (int e = 0; e < E; ++e) {
      if (taken[e]) continue;
      if (best < 0 || ranks_above(z[e], z[best])) best = e;
    }
    taken[best] = 1;
  }
  /* Store the chosen set in ascending expert order. */
  int n = 0;
  for (int e = 0; e < E; ++e)
    if (taken[e]) ids[n++] = e;
  /* Softmax over all E experts ... (a NaN logit has no probability to give
     the denominator; since the renormalisation below cancels the
     denominator, only a NaN among the selected logits reaches the weights) */
  double m = 0.0;
  int have_m = 0;
  for (int e = 0; e < E; ++e)
    if (!isnan(z[e]) && (!have_m || z[e] > m)) {
      m = z[e];
      have_m = 1;
    }
  double denom = 0.0;
  for (int e = 0; e < E; ++e)
    if (!isnan(z[e])) denom += exp(z[e] - m);
  /* ... then renormalise the selected probabilities to sum to one. */
  double sel = 0.0;
  for (int j = 0; j < k; ++j) {
    w[j] = exp(z[ids[j]] - m) / denom;
    sel += w[j];
  }
  for (int j = 0; j < k; ++j) w[j] /= sel;
}

/* Route T tokens.  ids: [T][k] int32, w: [T][k] fp64, z (optional): [T][E]. */
int oracle_route(int T, int D, int E, int k, const uint16_t *x,
                 const uint16_t *wr, const float *bias, int32_t *ids,
                 double *w, double *z_out) {
  if (T < 0 || k < 1 || k > E || !ids || !w) return ORACLE_EINVAL;
  double *z = z_out ? z_out : (double *)malloc(sizeof(double) * (size_t)T * E + 8);
  if (!z) return ORACLE_ENOMEM;
  int err = oracle_router_logits(T, D, E, x, wr, bias, z);
  if (err == ORACLE_OK) {
#pragma omp parallel
    {
      unsigned char *taken = (unsigned char *)malloc((size_t)E);
      if (!taken) {
#pragma omp atomic write
        err = ORACLE_ENOMEM;
      } else {
#pragma omp for schedule(static)
        for (int t = 0; t < T; ++t)
          select_token(E, k, z + (size_t)t * E, ids + (size_t)t * k,
                       w + (size_t)t * k, taken);
        free(taken);
      }
    }
  }
  if (!z_out) free(z);
  return err;
}

/* ------------------------------------------------------------------ */
/* Routing metadata blob: [T][2][k] int32; row t holds the k ids, then */
/* the k weights as fp32 bit patterns.                                  */
/* ------------------------------------------------------------------ */
int oracle_pack_blob(int T, int k, const int32_t *ids, const double *w,
                     int32_t *blob) {
  if (T < 0 || k < 1 || !ids || !w || !blob) return ORACLE_EINVAL;
  for (int t = 0; t < T; ++t)
    for (int j = 0; j < k; ++j) {
      float f = (float)w[(size_t)t * k + j];
      int32_t bits;
      memcpy(&bits, &f, sizeof bits);
      blob[(size_t)t * 2 * k + j] = ids[(size_t)t * k + j];
      blob[(size_t)t * 2 * k + k + j] = bits;
    }
  return ORACLE_OK;
}

int oracle_unpack_blob(int T, int k, const int32_t *blob, int32_t *ids,
                       float *w) {
  if (T < 0 || k < 1 || !ids || !w || !blob) return ORACLE_EINVAL;
  for (int t = 0; t < T; ++t)
    for (int j = 0; j < k; ++j) {
      ids[(size_t)t * k + j] = blob[(size_t)t * 2 * k + j];
      memcpy(&w[(size_t)t * k + j], &blob[(size_t)t * 2 * k + k + j], 4);
    }
  return ORACLE_OK;
}

/* ------------------------------------------------------------------ */
/* Dispatch grouping (reading R5).                                      */
/*   counts[e]   = number of pairs routed to e                          */
/*   offsets[e]  = sum of counts of experts below e; offsets[E] = T*k   */
/*   perm_pair[r]= pair index p = t*k+j held by grouped row r           */
/*   inv_row[p]  = grouped row of pair p                                */
/* ------------------------------------------------------------------ */
int oracle_permute(int T, int E, int k, const int32_t *ids, int32_t *counts,
                   int32_t *offsets, int32_t *perm_pair, int32_t *inv_row) {
  if (T < 0 || E < 1 || k < 1 || !ids || !counts || !offsets) return ORACLE_EINVAL;
  long P = (long)T * k;
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (long p = 0; p < P; ++p) {
    if (ids[p] < 0 || ids[p] >= E) return ORACLE_EINVAL;
    counts[ids[p]] += 1;
  }
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  if (perm_pair) {
    long r = 0;
    for (int e = 0; e < E; ++e)
      for (long p = 0; p < P; ++p)
        if (ids[p] == e) perm_pair[r++] = (int32_t)p;
    if (inv_row)
      for (long q = 0; q < P; ++q) inv_row[perm_pair[q]] = (int32_t)q;
  }
  return ORACLE_OK;
}

/* ------------------------------------------------------------------ */
/* Exact dequantisation of a packed int4 matrix (reading R7).          */
/* ------------------------------------------------------------------ */
int oracle_dequant_w4(int rows, int cols, int group, const int32_t *q,
                      const uint16_t *s, double *out) {
  if (rows < 0 || cols < 8 || cols % 8 || group < 0 || (group > 0 && cols % group) || !q ||
      !s || !out)
    return ORACLE_EINVAL;
  wview v = {rows, cols, 1, group, NULL, q, s};
  for (int r = 0; r < rows; ++r) load_row(&v, r, out + (size_t)r * cols);
  return ORACLE_OK;
}

/* ------------------------------------------------------------------ */
/* One SwiGLU expert on one token, fp64 throughout (reading R6, R8):   */
/*   g_i = <Wgu[i], x>,  u_i = <Wgu[I+i], x>,  h_i = silu(g_i) * u_i,   */
/*   o_c = <Wdn[c], h>.                                                 */
/* ------------------------------------------------------------------ */
static void expert_ffn(const wview *gu, const wview *dn, int D, int Ie,
                       const double *x, double *h, double *row, double *o) {
  for (int i = 0; i < Ie; ++i) {
    load_row(gu, i, row);
    double g = dot(row, x, D);
    load_row(gu, Ie + i, row);
    double u = dot(row, x, D);
    h[i] = silu(g) * u;
  }
  for (int c = 0; c < D; ++c) {
    load_row(dn, c, row);
    o[c] = dot(row, h, Ie);
  }
}

/*
 * Layer output for `nt` tokens given their routing:
 *   y_t = sum_j w[t][j] * FFN_{ids[t][j]}(x_t) + FFN_shared(x_t)
 * The k routed terms are added in slot order j = 0..k-1, then the shared one.
 *
 * Expert weights are passed as arrays of E+1 host addresses (index E = the
 * shared expert); an expert no token uses may have address 0.
 *   quant == 0: w_gu[e] -> bf16 [2Ie][D], w_dn[e] -> bf16 [D][Ie]
 *   quant == 1: w_gu[e] -> int32 [2Ie][D/8], s_gu[e] -> bf16 [2Ie][D/group],
 *               w_dn[e] -> int32 [D][Ie/8], s_dn[e] -> bf16 [D][Ie/group]
 *               (group 0: s_gu[e] -> bf16 [2Ie], s_dn[e] -> bf16 [D])
 * with Ie = I for routed experts and Is for the shared one.
 */
int oracle_forward(int nt, int D, int E, int I, int Is, int k, int quant,
                   int group, const uint16_t *x, const int32_t *ids,
                   const double *w, const uint64_t *w_gu, const uint64_t *s_gu,
                   const uint64_t *w_dn, const uint64_t *s_dn, double *y) {
  if (nt < 0 || D < 1 || E < 1 || I < 1 || Is < 1 || k < 1 || k > E || !x ||
      !ids || !w || !w_gu || !w_dn || !y)
    return ORACLE_EINVAL;
  if (quant == 1 && (!s_gu || !s_dn || group < 0 ||
                     (group > 0 && (D % group || I % group || Is % group)) || D % 8 ||
                     I % 8 || Is % 8))
    return ORACLE_EINVAL;
  for (int t = 0; t < nt; ++t)
    for (int j = 0; j < k; ++j) {
      int e = ids[(size_t)t * k + j];
      if (e < 0 || e >= E || !w_gu[e] || !w_dn[e]) return ORACLE_EINVAL;
      if (quant == 1 && (!s_gu[e] || !s_dn[e])) return ORACLE_EINVAL;
    }
  if (!w_gu[E] || !w_dn[E] || (quant == 1 && (!s_gu[E] || !s_dn[E])))
    return ORACLE_EINVAL;
  int maxI = I > Is ? I : Is;
  int width = D > maxI ? D : maxI;
  int err = ORACLE_OK;
#pragma omp parallel
  {
    double *xd = (double *)malloc(sizeof(double) * (size_t)D);
    double *h = (double *)malloc(sizeof(double) * (size_t)maxI);
    double *row = (double *)malloc(sizeof(double) * (size_t)width);
    double *o = (double *)malloc(sizeof(double) * (size_t)D);
    if (!xd || !h || !row || !o) {
#pragma omp atomic write
      err = ORACLE_ENOMEM;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (int t = 0; t < nt; ++t) {
        double *yt = y + (size_t)t * D;
        for (int d = 0; d < D; ++d) {
          xd[d] = bf16_to_f64(x[(size_t)t * D + d]);
          yt[d] = 0.0;
        }
        for (int j = 0; j <= k; ++j) {
          int e = j < k ? ids[(size_t)t * k + j] : E;
          int Ie = j < k ? I : Is;
          double wt = j < k ? w[(size_t)t * k + j] : 1.0;
          wview gu = {2 * Ie, D, quant, group, NULL, NULL, NULL};
          wview dn = {D, Ie, quant, group, NULL, NULL, NULL};
          if (quant == 0) {
            gu.bf16 = (const uint16_t *)(uintptr_t)w_gu[e];
            dn.bf16 = (const uint16_t *)(uintptr_t)w_dn[e];
          } else {
            gu.q = (const int32_t *)(uintptr_t)w_gu[e];
            gu.s = (const uint16_t *)(uintptr_t)s_gu[e];
            dn.q = (const int32_t *)(uintptr_t)w_dn[e];
            dn.s = (const uint16_t *)(uintptr_t)s_dn[e];
          }
          expert_ffn(&gu, &dn, D, Ie, xd, h, row, o);
          for (int d = 0; d < D; ++d) yt[d] += wt * o[d];
        }
      }
    }
    free(xd);
    free(h);
    free(row);
    free(o);
  }
  return err;
}

/* ------------------------------------------------------------------ */
/* The two halves of one expert, exposed for per-kernel checks:         */
/*   oracle_expert_hidden:  h[n][i] = silu(<Wgu[i], x_n>) * <Wgu[I+i], x_n> */
/*   oracle_expert_down:    o[n][c] = <Wdn[c], h_n>                     */
/* Weight formats as in oracle_forward (quant 0: bf16; 1: int4 + scales). */
/* ------------------------------------------------------------------ */
int oracle_expert_hidden(int n, int D, int Ie, int quant, int group,
                         const uint16_t *x, const void *w_gu, const uint16_t *s_gu,
                         double *h) {
  if (n < 0 || D < 1 || Ie < 1 || !x || !w_gu || !h) return ORACLE_EINVAL;
  if (quant == 1 && (!s_gu || group < 0 || (group > 0 && D % group) || D % 8))
    return ORACLE_EINVAL;
  wview gu = {2 * Ie, D, quant, group, NULL, NULL, NULL};
  if (quant == 0) gu.bf16 = (const uint16_t *)w_gu;
  else { gu.q = (const int32_t *)w_gu; gu.s = s_gu; }
  int err = ORACLE_OK;
#pragma omp parallel
  {
    double *xd = (double *)malloc(sizeof(double) * (size_t)D);
    double *row = (double *)malloc(sizeof(double) * (size_t)D);
    if (!xd || !row) {
#pragma omp atomic write
      err = ORACLE_ENOMEM;
    } else {
#pragma omp for schedule(static)
      for (int r = 0; r < n; ++r) {
        for (int d = 0; d < D; ++d) xd[d] = bf16_to_f64(x[(size_t)r * D + d]);
        for (int i = 0; i < Ie; ++i) {
          load_row(&gu, i, row);
          double g = dot(row, xd, D);
          load_row(&gu, Ie + i, row);
          double u = dot(row, xd, D);
          h[(size_t)r * Ie + i] = silu(g) * u;
        }
      }
    }
    free(xd);
    free(row);
  }
  return err;
}

int oracle_expert_down(int n, int D, int Ie, int quant, int group, const double *h,
                       const void *w_dn, const uint16_t *s_dn, double *o) {
  if (n < 0 || D < 1 || Ie < 1 || !h || !w_dn || !o) return ORACLE_EINVAL;
  if (quant == 1 && (!s_dn || group < 0 || (group > 0 && Ie % group) || Ie % 8))
    return ORACLE_EINVAL;
  wview dn = {D, Ie, quant, group, NULL, NULL, NULL};
  if (quant == 0) dn.bf16 = (const uint16_t *)w_dn;
  else { dn.q = (const int32_t *)w_dn; dn.s = s_dn; }
  int err = ORACLE_OK;
#pragma omp parallel
  {
    double *row = (double *)malloc(sizeof(double) * (size_t)Ie);
    if (!row) {
#pragma omp atomic write
      err = ORACLE_ENOMEM;
    } else {
#pragma omp for schedule(static)
      for (int c = 0; c < D; ++c) {
        load_row(&dn, c, row);
        for (int r = 0; r < n; ++r) o[(size_t)r * D + c] = dot(row, h + (size_t)r * Ie, Ie);
      }
    }
    free(row);
  }
  return err;
}

/* ------------------------------------------------------------------ */
/* Unpermute + combine: y[t][d] = o_shared[t][d] + sum_j o[inv_row[t*k+j]][d] */
/* (o already weighted; o_shared may be NULL).                          */
/* ------------------------------------------------------------------ */
int oracle_combine(int T, int D, int k, const double *o, const double *o_shared,
                   const int32_t *inv_row, double *y) {
  if (T < 0 || D < 1 || k < 1 || !o || !inv_row || !y) return ORACLE_EINVAL;
  for (int t = 0; t < T; ++t)
    for (int d = 0; d < D; ++d) {
      double acc = o_shared ? o_shared[(size_t)t * D + d] : 0.0;
      for (int j = 0; j < k; ++j) acc += o[(size_t)inv_row[(size_t)t * k + j] * D + d];
      y[(size_t)t * D + d] = acc;
    }
  return ORACLE_OK;
}

/* Threads OpenMP will use (reported beside CPU timings). */
int oracle_num_threads(void) {
  int n = 1;
#pragma omp parallel
  {
#pragma omp single
    {
#ifdef _OPENMP
      n = omp_get_num_threads();
#endif
    }
  }
  return n;
}
