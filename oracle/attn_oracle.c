/*
 * Oracle for the fused RoPE + variant attention path — TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, fp64 CPU statement of what the path computes, written from the AttnFuse
 * paper ("AttnFuse: A Composable DSL for Compiling Attentions to Fused GPU Kernels",
 * arXiv 2609.13612). It shares no code, header, table or helper with the CUDA library and
 * must only be used by the tests, by __graft_entry__.smoke() and by bench.py's CPU baseline.
 *
 * The method reaches an exact closed-form result (the paper, §2 "FlashAttention and online
 * softmax": the tiled recurrence is exact; §4.2: the split-KV merge is exact), so this file
 * writes out that definition directly — no tiling, no online rescaling, no splitting:
 *
 *   q'_m = R_m q_m, k'_n = R_n k_n                      (RoPE, §2 and §4.1, NeoX half-split)
 *   s_mn = scale <q'_m, k'_n> (+ slope_h (n - m)) (+ bias[b,h,m,n])     (combinators, §3.1)
 *   s_mn = -inf where the mask forbids (m, n)           (causal / sliding window / block-sparse)
 *   LSE_m = max_n s_mn + ln sum_n exp(s_mn - max)       (§4.4: the saved per-row scalar)
 *   O_m = sum_n exp(s_mn - LSE_m) v_n
 *
 * and the backward by direct differentiation of that definition (§4.4):
 *   D_m = <dO_m, O_m>, dP_mn = <dO_m, v_n>, dS_mn = P_mn (dP_mn - D_m),
 *   dq'_m = scale sum_n dS_mn k'_n, dk'_n = scale sum_m dS_mn q'_m, dv_n = sum_m P_mn dO_m,
 *   dq_m = R_m^T dq'_m, dk_n = R_n^T dk'_n  (gradients w.r.t. the un-rotated inputs),
 *   dk, dv summed over the query heads that share a key/value head (GQA),
 *   dBias_mn = dS_mn (the bias enters s_mn with weight 1, after the scaling, §3.1).
 *
 * Readings where the pages are silent (each is also listed in the design notes):
 *   - theta_i = theta^(-2i/d), i < d/2 (RoFormer, the paper's RoPE reference); pair (i, i+d/2).
 *   - positions are 0-based token indices; decode query sits at q_pos, keys at 0..L-1.
 *   - sliding window W: |m - n| < W, and n <= m when causal.
 *   - ALiBi bias = slope_h * (n - m), slopes supplied by the caller (one per query head).
 *   - GQA: query head h reads key/value head h / (Hq / Hkv).
 *   - a row with no allowed key: O = 0, LSE = -inf.
 *   - relu_attention (§3.1 names this normaliser without defining it): the softmax is replaced
 *     by O_m = (1/N) sum_{allowed n} max(s_mn, 0) v_n, N the number of keys (the sequence
 *     length), as in ReLU attention divided by the sequence length; there is no LSE (NaN is
 *     returned) and no backward.
 * All tensors are contiguous row-major [B, H, N, d] fp64 unless stated.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_MASK_FULL = 0, ORC_MASK_CAUSAL = 1, ORC_MASK_WINDOW = 2, ORC_MASK_BLOCK_SPARSE = 3 };
enum { ORC_BIAS_NONE = 0, ORC_BIAS_ALIBI = 1, ORC_BIAS_ADDITIVE = 2 };
enum { ORC_NORM_SOFTMAX = 0, ORC_NORM_RELU = 1 };

typedef struct {
  int32_t mask;       /* ORC_MASK_* */
  int32_t causal;     /* also forbid n > m (combines with WINDOW / BLOCK_SPARSE / FULL) */
  int32_t window;     /* W for ORC_MASK_WINDOW */
  int32_t bs_block;   /* block edge for ORC_MASK_BLOCK_SPARSE */
  const int32_t* bs_row_ptr; /* CSR over block rows: [ceil(N/bs_block) + 1] */
  const int32_t* bs_col_idx; /* active block columns of each block row */
  int32_t bias;       /* ORC_BIAS_* */
  int32_t norm;       /* ORC_NORM_*: the row normaliser */
  const double* slopes;      /* [Hq] for ORC_BIAS_ALIBI */
  const double* add_bias;    /* additive bias, element (b,h,m,n) at the strides below */
  int64_t add_bias_strides[4];
} orc_variant;

/* ---------------------------------------------------------------------------------------- */
/* RoPE (paper §2 "Rotary Position Embeddings" and §4.1: NeoX convention, half-split pairs)  */
/* ---------------------------------------------------------------------------------------- */

/* Angle of frequency i at position p: p * theta^(-2i/d). */
static double rope_angle(double pos, int i, int d, double theta) {
  return pos * pow(theta, -2.0 * (double)i / (double)d);
}

/* y = R_pos x (inverse != 0: y = R_pos^T x, i.e. rotation by -pos). x and y may not alias. */
static void rope_rotate(const double* x, double* y, int d, double pos, double theta, int inverse) {
  const int h = d / 2;
  for (int i = 0; i < h; ++i) {
    const double a = rope_angle(pos, i, d, theta);
    const double c = cos(a);
    const double s = inverse ? -sin(a) : sin(a);
    y[i] = x[i] * c - x[i + h] * s;
    y[i + h] = x[i + h] * c + x[i] * s;
  }
}

/* Exported for the oracle's own self-tests: rotate `rows` vectors of length d; row r sits at
 * position pos[r]. */
int orc_rope(const double* x, double* y, int64_t rows, int d, const double* pos, double theta,
             int inverse) {
  if (d <= 0 || (d & 1)) return 1;
  for (int64_t r = 0; r < rows; ++r) rope_rotate(x + r * d, y + r * d, d, pos[r], theta, inverse);
  return 0;
}

/* ---------------------------------------------------------------------------------------- */
/* Combinators (paper §3.1: causal, sliding_window, full, block_sparse, alibi, additive_bias) */
/* ---------------------------------------------------------------------------------------- */

static int block_active(const orc_variant* v, int64_t brow, int64_t bcol) {
  for (int32_t e = v->bs_row_ptr[brow]; e < v->bs_row_ptr[brow + 1]; ++e)
    if (v->bs_col_idx[e] == bcol) return 1;
  return 0;
}

/* Is key n visible to query m? */
static int allowed(const orc_variant* v, int64_t m, int64_t n) {
  if ((v->mask == ORC_MASK_CAUSAL || v->causal) && n > m) return 0;
  if (v->mask == ORC_MASK_WINDOW && !(n > m - v->window && n < m + v->window)) return 0;
  if (v->mask == ORC_MASK_BLOCK_SPARSE && !block_active(v, m / v->bs_block, n / v->bs_block))
    return 0;
  return 1;
}

/* Score bias added after scaling. */
static double score_bias(const orc_variant* v, int64_t b, int64_t h, int64_t m, int64_t n) {
  double t = 0.0;
  if (v->bias == ORC_BIAS_ALIBI) t += v->slopes[h] * (double)(n - m);
  if (v->bias == ORC_BIAS_ADDITIVE)
    t += v->add_bias[b * v->add_bias_strides[0] + h * v->add_bias_strides[1] +
                     m * v->add_bias_strides[2] + n * v->add_bias_strides[3]];
  return t;
}

static double dot(const double* a, const double* b, int d) {
  double s = 0.0;
  for (int c = 0; c < d; ++c) s += a[c] * b[c];
  return s;
}

/* One query row of the forward. qr: rotated query; kr: rotated keys of its kv head [N, d];
 * vh: values [N, d]. Writes p[n] (probabilities, 0 where masked), o[d], returns LSE. */
static double row_forward(const orc_variant* var, int64_t b, int64_t h, int64_t m, const double* qr,
                          const double* kr, const double* vh, int64_t N, int d, double scale,
                          double* s, double* p, double* o) {
  double mx = -INFINITY;
  for (int64_t n = 0; n < N; ++n) {
    if (!allowed(var, m, n)) {
      s[n] = -INFINITY;
      continue;
    }
    s[n] = scale * dot(qr, kr + n * d, d) + score_bias(var, b, h, m, n);
    if (s[n] > mx) mx = s[n];
  }
  for (int c = 0; c < d; ++c) o[c] = 0.0;
  if (var->norm == ORC_NORM_RELU) {
    /* relu_attention: weights max(s, 0) / N, no exponent and no row sum */
    for (int64_t n = 0; n < N; ++n) {
      p[n] = (s[n] == -INFINITY || s[n] <= 0.0) ? 0.0 : s[n] / (double)N;
      if (p[n] != 0.0)
        for (int c = 0; c < d; ++c) o[c] += p[n] * vh[n * d + c];
    }
    return NAN;
  }
  if (mx == -INFINITY) {
    for (int64_t n = 0; n < N; ++n) p[n] = 0.0;
    return -INFINITY;
  }
  double sum = 0.0;
  for (int64_t n = 0; n < N; ++n)
    if (s[n] != -INFINITY) sum += exp(s[n] - mx);
  const double lse = mx + log(sum);
  for (int64_t n = 0; n < N; ++n) {
    p[n] = (s[n] == -INFINITY) ? 0.0 : exp(s[n] - lse);
    if (p[n] != 0.0)
      for (int c = 0; c < d; ++c) o[c] += p[n] * vh[n * d + c];
  }
  return lse;
}

/* Rotate (or copy) the N rows of one head: row n at position n. */
static void rotate_head(const double* x, double* y, int64_t N, int d, double theta, int rope) {
  for (int64_t n = 0; n < N; ++n) {
    if (rope)
      rope_rotate(x + n * d, y + n * d, d, (double)n, theta, 0);
    else
      memcpy(y + n * d, x + n * d, sizeof(double) * (size_t)d);
  }
}

static int check_shape(int B, int Hq, int Hkv, int64_t N, int d) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || N <= 0 || d <= 0 || (d & 1)) return 1;
  if (Hq % Hkv) return 1;
  return 0;
}

/* ---------------------------------------------------------------------------------------- */
/* Forward (paper §4.1 fused RoPE + §2 softmax; exact definition)                           */
/* ---------------------------------------------------------------------------------------- */
int orc_fwd(const double* q, const double* k, const double* v, int B, int Hq, int Hkv, int64_t N,
            int d, double scale, double theta, int rope, const orc_variant* var, double* out,
            double* lse) {
  if (check_shape(B, Hq, Hkv, N, d)) return 1;
  const int g = Hq / Hkv;
  int err = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t bh = 0; bh < (int64_t)B * Hq; ++bh) {
    const int64_t b = bh / Hq, h = bh % Hq, kvh = h / g;
    const double* qh = q + bh * N * d;
    const double* kh = k + (b * Hkv + kvh) * N * d;
    const double* vh = v + (b * Hkv + kvh) * N * d;
    double* kr = (double*)malloc(sizeof(double) * (size_t)(N * d));
    double* qr = (double*)malloc(sizeof(double) * (size_t)d);
    double* s = (double*)malloc(sizeof(double) * (size_t)N);
    double* p = (double*)malloc(sizeof(double) * (size_t)N);
    if (!kr || !qr || !s || !p) {
#pragma omp atomic write
      err = 2;
    } else {
      rotate_head(kh, kr, N, d, theta, rope);
      for (int64_t m = 0; m < N; ++m) {
        if (rope)
          rope_rotate(qh + m * d, qr, d, (double)m, theta, 0);
        else
          memcpy(qr, qh + m * d, sizeof(double) * (size_t)d);
        const double l = row_forward(var, b, h, m, qr, kr, vh, N, d, scale, s, p,
                                     out + (bh * N + m) * d);
        if (lse) lse[bh * N + m] = l;
      }
    }
    free(kr); free(qr); free(s); free(p);
  }
  return err;
}

/* Forward for selected rows only: rows[3r..3r+2] = (b, h, m). out: [nrows, d], lse: [nrows].
 * Same definition as orc_fwd, evaluated one row at a time (used at full problem sizes). */
int orc_fwd_rows(const double* q, const double* k, const double* v, int B, int Hq, int Hkv,
                 int64_t N, int d, double scale, double theta, int rope, const orc_variant* var,
                 int64_t nrows, const int64_t* rows, double* out, double* lse) {
  if (check_shape(B, Hq, Hkv, N, d)) return 1;
  const int g = Hq / Hkv;
  int err = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < nrows; ++r) {
    const int64_t b = rows[3 * r], h = rows[3 * r + 1], m = rows[3 * r + 2], kvh = h / g;
    if (b < 0 || b >= B || h < 0 || h >= Hq || m < 0 || m >= N) {
#pragma omp atomic write
      err = 1;
      continue;
    }
    const double* kh = k + (b * Hkv + kvh) * N * d;
    const double* vh = v + (b * Hkv + kvh) * N * d;
    double* kr = (double*)malloc(sizeof(double) * (size_t)(N * d));
    double* qr = (double*)malloc(sizeof(double) * (size_t)d);
    double* s = (double*)malloc(sizeof(double) * (size_t)N);
    double* p = (double*)malloc(sizeof(double) * (size_t)N);
    if (!kr || !qr || !s || !p) {
#pragma omp atomic write
      err = 2;
    } else {
      /* only keys the row can see need rotating */
      for (int64_t n = 0; n < N; ++n) {
        if (!allowed(var, m, n)) continue;
        if (rope)
          rope_rotate(kh + n * d, kr + n * d, d, (double)n, theta, 0);
        else
          memcpy(kr + n * d, kh + n * d, sizeof(double) * (size_t)d);
      }
      const double* qrow = q + ((b * Hq + h) * N + m) * d;
      if (rope)
        rope_rotate(qrow, qr, d, (double)m, theta, 0);
      else
        memcpy(qr, qrow, sizeof(double) * (size_t)d);
      const double l = row_forward(var, b, h, m, qr, kr, vh, N, d, scale, s, p, out + r * d);
      if (lse) lse[r] = l;
    }
    free(kr); free(qr); free(s); free(p);
  }
  return err;
}

/* ---------------------------------------------------------------------------------------- */
/* Backward (paper §4.4), by direct differentiation of the forward definition.              */
/* groups: optional list of (b, kvh) pairs [2*ngroups]; NULL = every group. Only the heads  */
/* of the listed groups are computed; other entries of out/lse/dq/dk/dv are left untouched.  */
/* dbias: optional [B, Hq, N, N] output, the gradient with respect to an additive bias       */
/* element (b, h, m, n): dS_mn, and 0 where (m, n) is masked.                                */
/* ---------------------------------------------------------------------------------------- */
int orc_bwd(const double* q, const double* k, const double* v, const double* dout, int B, int Hq,
            int Hkv, int64_t N, int d, double scale, double theta, int rope,
            const orc_variant* var, int64_t ngroups, const int64_t* groups, double* out,
            double* lse, double* dq, double* dk, double* dv, double* dbias) {
  if (var->norm != ORC_NORM_SOFTMAX) return 1; /* relu_attention has no backward here */
  if (check_shape(B, Hq, Hkv, N, d)) return 1;
  const int g = Hq / Hkv;
  const int64_t G = groups ? ngroups : (int64_t)B * Hkv;
  const size_t hd = (size_t)(N * d);
  /* per (selected group, head-in-group) partial dk', dv */
  double* dkp = (double*)calloc((size_t)G * g * hd, sizeof(double));
  double* dvp = (double*)calloc((size_t)G * g * hd, sizeof(double));
  if (!dkp || !dvp) {
    free(dkp); free(dvp);
    return 2;
  }
  int err = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t gi = 0; gi < G * g; ++gi) {
    const int64_t sel = gi / g, j = gi % g;
    const int64_t b = groups ? groups[2 * sel] : sel / Hkv;
    const int64_t kvh = groups ? groups[2 * sel + 1] : sel % Hkv;
    const int64_t h = kvh * g + j, bh = b * Hq + h;
    if (b < 0 || b >= B || kvh < 0 || kvh >= Hkv) {
#pragma omp atomic write
      err = 1;
      continue;
    }
    const double* kh = k + (b * Hkv + kvh) * N * d;
    const double* vh = v + (b * Hkv + kvh) * N * d;
    double* kr = (double*)malloc(sizeof(double) * hd);
    double* qr = (double*)malloc(sizeof(double) * (size_t)d);
    double* s = (double*)malloc(sizeof(double) * (size_t)N);
    double* p = (double*)malloc(sizeof(double) * (size_t)N);
    double* dqr = (double*)malloc(sizeof(double) * (size_t)d);
    if (!kr || !qr || !s || !p || !dqr) {
#pragma omp atomic write
      err = 2;
    } else {
      double* dk_acc = dkp + (size_t)gi * hd;
      double* dv_acc = dvp + (size_t)gi * hd;
      rotate_head(kh, kr, N, d, theta, rope);
      for (int64_t m = 0; m < N; ++m) {
        const double* qrow = q + (bh * N + m) * d;
        const double* dorow = dout + (bh * N + m) * d;
        double* orow = out + (bh * N + m) * d;
        if (rope)
          rope_rotate(qrow, qr, d, (double)m, theta, 0);
        else
          memcpy(qr, qrow, sizeof(double) * (size_t)d);
        const double l = row_forward(var, b, h, m, qr, kr, vh, N, d, scale, s, p, orow);
        lse[bh * N + m] = l;
        const double Dm = dot(dorow, orow, d);
        double* dbrow = dbias ? dbias + (bh * N + m) * N : NULL;
        if (dbrow)
          for (int64_t n = 0; n < N; ++n) dbrow[n] = 0.0;
        for (int c = 0; c < d; ++c) dqr[c] = 0.0;
        for (int64_t n = 0; n < N; ++n) {
          if (p[n] == 0.0) continue;
          const double dP = dot(dorow, vh + n * d, d);
          const double dS = p[n] * (dP - Dm);
          if (dbrow) dbrow[n] = dS;
          for (int c = 0; c < d; ++c) {
            dqr[c] += scale * dS * kr[n * d + c];
            dk_acc[n * d + c] += scale * dS * qr[c];
            dv_acc[n * d + c] += p[n] * dorow[c];
          }
        }
        if (rope)
          rope_rotate(dqr, dq + (bh * N + m) * d, d, (double)m, theta, 1);
        else
          memcpy(dq + (bh * N + m) * d, dqr, sizeof(double) * (size_t)d);
      }
    }
    free(kr); free(qr); free(s); free(p); free(dqr);
  }
  if (!err) {
    /* sum over the g query heads of each group in head order, then undo the key rotation */
    double* tmp = (double*)malloc(sizeof(double) * (size_t)d);
    for (int64_t sel = 0; sel < G && tmp; ++sel) {
      const int64_t b = groups ? groups[2 * sel] : sel / Hkv;
      const int64_t kvh = groups ? groups[2 * sel + 1] : sel % Hkv;
      double* dkh = dk + (b * Hkv + kvh) * N * d;
      double* dvh = dv + (b * Hkv + kvh) * N * d;
      for (int64_t n = 0; n < N; ++n) {
        for (int c = 0; c < d; ++c) {
          double sk = 0.0, sv = 0.0;
          for (int j = 0; j < g; ++j) {
            sk += dkp[(size_t)(sel * g + j) * hd + n * d + c];
            sv += dvp[(size_t)(sel * g + j) * hd + n * d + c];
          }
          tmp[c] = sk;
          dvh[n * d + c] = sv;
        }
        if (rope)
          rope_rotate(tmp, dkh + n * d, d, (double)n, theta, 1);
        else
          memcpy(dkh + n * d, tmp, sizeof(double) * (size_t)d);
      }
    }
    if (!tmp) err = 2;
    free(tmp);
  }
  free(dkp); free(dvp);
  return err;
}

/* dq for selected rows only (rows as in orc_fwd_rows); dq_rows: [nrows, d]. Needs only the
 * row's own probabilities, so it is cheap at full problem sizes. */
int orc_bwd_dq_rows(const double* q, const double* k, const double* v, const double* dout, int B,
                    int Hq, int Hkv, int64_t N, int d, double scale, double theta, int rope,
                    const orc_variant* var, int64_t nrows, const int64_t* rows, double* dq_rows) {
  if (var->norm != ORC_NORM_SOFTMAX) return 1;
  if (check_shape(B, Hq, Hkv, N, d)) return 1;
  const int g = Hq / Hkv;
  int err = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < nrows; ++r) {
    const int64_t b = rows[3 * r], h = rows[3 * r + 1], m = rows[3 * r + 2], kvh = h / g;
    if (b < 0 || b >= B || h < 0 || h >= Hq || m < 0 || m >= N) {
#pragma omp atomic write
      err = 1;
      continue;
    }
    const int64_t bh = b * Hq + h;
    const double* kh = k + (b * Hkv + kvh) * N * d;
    const double* vh = v + (b * Hkv + kvh) * N * d;
    double* kr = (double*)malloc(sizeof(double) * (size_t)(N * d));
    double* qr = (double*)malloc(sizeof(double) * (size_t)d);
    double* s = (double*)malloc(sizeof(double) * (size_t)N);
    double* p = (double*)malloc(sizeof(double) * (size_t)N);
    double* o = (double*)malloc(sizeof(double) * (size_t)d);
    double* dqr = (double*)malloc(sizeof(double) * (size_t)d);
    if (!kr || !qr || !s || !p || !o || !dqr) {
#pragma omp atomic write
      err = 2;
    } else {
      for (int64_t n = 0; n < N; ++n) {
        if (!allowed(var, m, n)) continue;
        if (rope)
          rope_rotate(kh + n * d, kr + n * d, d, (double)n, theta, 0);
        else
          memcpy(kr + n * d, kh + n * d, sizeof(double) * (size_t)d);
      }
      const double* qrow = q + (bh * N + m) * d;
      const double* dorow = dout + (bh * N + m) * d;
      if (rope)
        rope_rotate(qrow, qr, d, (double)m, theta, 0);
      else
        memcpy(qr, qrow, sizeof(double) * (size_t)d);
      row_forward(var, b, h, m, qr, kr, vh, N, d, scale, s, p, o);
      const double Dm = dot(dorow, o, d);
      for (int c = 0; c < d; ++c) dqr[c] = 0.0;
      for (int64_t n = 0; n < N; ++n) {
        if (p[n] == 0.0) continue;
        const double dS = p[n] * (dot(dorow, vh + n * d, d) - Dm);
        for (int c = 0; c < d; ++c) dqr[c] += scale * dS * kr[n * d + c];
      }
      if (rope)
        rope_rotate(dqr, dq_rows + r * d, d, (double)m, theta, 1);
      else
        memcpy(dq_rows + r * d, dqr, sizeof(double) * (size_t)d);
    }
    free(kr); free(qr); free(s); free(p); free(o); free(dqr);
  }
  return err;
}

/* ---------------------------------------------------------------------------------------- */
/* Decode (paper §4.2): one query row per (b, h) at position q_pos against a cache whose keys */
/* are stored already rotated. The split-KV merge is exact, so the oracle does not split.     */
/* q: [B, Hq, d]; kc, vc: [B, Hkv, L, d]; out: [B, Hq, d]; lse: [B, Hq].                      */
/* ---------------------------------------------------------------------------------------- */
int orc_decode(const double* q, const double* kc, const double* vc, int B, int Hq, int Hkv,
               int64_t L, int d, int64_t q_pos, double scale, double theta, int rope_q,
               double* out, double* lse) {
  if (check_shape(B, Hq, Hkv, L, d)) return 1;
  const int g = Hq / Hkv;
  orc_variant full;
  memset(&full, 0, sizeof(full));
  int err = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t bh = 0; bh < (int64_t)B * Hq; ++bh) {
    const int64_t b = bh / Hq, h = bh % Hq, kvh = h / g;
    double* qr = (double*)malloc(sizeof(double) * (size_t)d);
    double* s = (double*)malloc(sizeof(double) * (size_t)L);
    double* p = (double*)malloc(sizeof(double) * (size_t)L);
    if (!qr || !s || !p) {
#pragma omp atomic write
      err = 2;
    } else {
      if (rope_q)
        rope_rotate(q + bh * d, qr, d, (double)q_pos, theta, 0);
      else
        memcpy(qr, q + bh * d, sizeof(double) * (size_t)d);
      const double l = row_forward(&full, b, h, q_pos, qr, kc + (b * Hkv + kvh) * L * d,
                                   vc + (b * Hkv + kvh) * L * d, L, d, scale, s, p, out + bh * d);
      if (lse) lse[bh] = l;
    }
    free(qr); free(s); free(p);
  }
  return err;
}

/* ---------------------------------------------------------------------------------------- */
/* Tile-visit set (paper §4.3: only blocks with an allowed entry are visited): out[t_q, t_k]  */
/* = 1 iff some (m, n) with m in q-tile t_q (BM rows) and n in kv-tile t_k (BN keys) is     */
/* allowed. out: [ceil(N/BM), ceil(N/BN)] uint8.                                            */
/* ---------------------------------------------------------------------------------------- */
int orc_tile_visits(int64_t N, int BM, int BN, const orc_variant* var, uint8_t* out) {
  if (N <= 0 || BM <= 0 || BN <= 0) return 1;
  const int64_t TQ = (N + BM - 1) / BM, TK = (N + BN - 1) / BN;
  memset(out, 0, (size_t)(TQ * TK));
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t tq = 0; tq < TQ; ++tq)
    for (int64_t m = tq * BM; m < (tq + 1) * BM && m < N; ++m)
      for (int64_t n = 0; n < N; ++n)
        if (!out[tq * TK + n / BN] && allowed(var, m, n)) out[tq * TK + n / BN] = 1;
  return 0;
}

/* Number of allowed (m, n) pairs of one head (the algorithmic work of the forward). */
int64_t orc_allowed_pairs(int64_t N, const orc_variant* var) {
  int64_t cnt = 0;
#pragma omp parallel for reduction(+ : cnt) schedule(dynamic, 16)
  for (int64_t m = 0; m < N; ++m)
    for (int64_t n = 0; n < N; ++n) cnt += allowed(var, m, n);
  return cnt;
}
