/*
 * poetx_oracle.c -- CPU oracle for the POET-X transformed linear layer.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously
 * correct statement of what the GPU library computes.  Only the tests,
 * the smoke check and the benchmark's CPU-baseline leg may build, load or
 * call it.  It shares no code, header, table or helper with the CUDA
 * library, and the CUDA library never calls it.
 *
 * Source of the method: the web page "POET-X: Memory-efficient LLM
 * Training by Scaling Orthogonal Transformation" (gist.science technical
 * summary of arXiv 2603.05500), section 2 "Methodologie", cited below as
 * [POET-X §2.A] .. [POET-X §2.E]:
 *   §2.A input-centric implementation: y = R (W0 (P x)), R.W0.P never formed
 *   §2.B permutations as index maps; merged into W0 ahead of time (4 -> 2)
 *   §2.C block-diagonal orthogonal matrices, each block its own matrix
 *   §2.D Cayley-Neumann parameterisation: skew upper triangle stored,
 *        b(b-1)/2 values per block; Neumann series replaces the inverse
 *   §2.E POET-Xfast / POET-Xmem checkpointing variants
 *
 * Conventions (the pages fix none of them; these are the plain readings):
 *   - all matrices row-major, all arithmetic IEEE double, plain loops;
 *   - a permutation is an int array pi of length d; applying it gathers:
 *     (Pi v)_i = v_{pi(i)}; its transpose scatters: (Pi^T v)_{pi(i)} = v_i;
 *   - P = Pi_P^T B_P Pi_P, R = Pi_R^T B_R Pi_R, B = blockdiag(Q_0..Q_{nb-1});
 *   - skew packing: block parameters theta_p, p = 0..b(b-1)/2-1, fill the
 *     strict upper triangle row by row, (0,1),(0,2),..,(0,b-1),(1,2),..;
 *     K[i][k] = theta_p and K[k][i] = -theta_p for i < k;
 *   - Cayley-Neumann with n terms: Q = (I + K) (I + K + ... + K^n),
 *     the Cayley map (I + K)(I - K)^{-1} with the inverse replaced by its
 *     Neumann series truncated after K^n.
 *
 * Parallelism: OpenMP over independent tokens / blocks / output entries
 * only; every reduction runs in a fixed serial order, so results do not
 * depend on the thread count.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* small dense helpers (b x b or d x d, row-major)                     */
/* ------------------------------------------------------------------ */

static void mat_identity(int b, double *M) {
  memset(M, 0, sizeof(double) * (size_t)b * b);
  for (int i = 0; i < b; ++i) M[(size_t)i * b + i] = 1.0;
}

/* C = A . B, all b x b; C must not alias A or B. */
static void mat_mul(int b, const double *A, const double *B, double *C) {
  for (int i = 0; i < b; ++i) {
    double *c = C + (size_t)i * b;
    for (int j = 0; j < b; ++j) c[j] = 0.0;
    for (int k = 0; k < b; ++k) {
      const double a = A[(size_t)i * b + k];
      const double *brow = B + (size_t)k * b;
      for (int j = 0; j < b; ++j) c[j] += a * brow[j];
    }
  }
}

/* T = M^T, b x b */
static void mat_transpose(int b, const double *M, double *T) {
  for (int i = 0; i < b; ++i)
    for (int j = 0; j < b; ++j) T[(size_t)j * b + i] = M[(size_t)i * b + j];
}

/* ------------------------------------------------------------------ */
/* [POET-X §2.D] packed skew storage: b(b-1)/2 values per block         */
/* ------------------------------------------------------------------ */

long orc_skew_count(int b) { return (long)b * (b - 1) / 2; }

/* theta [b(b-1)/2] -> K [b,b], K = -K^T, zero diagonal. */
void orc_unpack_skew(const double *theta, int b, double *K) {
  memset(K, 0, sizeof(double) * (size_t)b * b);
  long p = 0;
  for (int i = 0; i < b; ++i)
    for (int k = i + 1; k < b; ++k) {
      K[(size_t)i * b + k] = theta[p];
      K[(size_t)k * b + i] = -theta[p];
      ++p;
    }
}

/* Reads the strict upper triangle of M [b,b] in packing order. */
void orc_pack_upper(const double *M, int b, double *theta) {
  long p = 0;
  for (int i = 0; i < b; ++i)
    for (int k = i + 1; k < b; ++k) theta[p++] = M[(size_t)i * b + k];
}

/* ------------------------------------------------------------------ */
/* [POET-X §2.D] Cayley-Neumann parameterisation                        */
/* ------------------------------------------------------------------ */

/* One block: Q = (I + K) . S,  S = sum_{i=0..n} K^i  (n >= 0). */
static void cnp_block(const double *theta, int b, int n, double *Q) {
  const size_t bb = (size_t)b * b;
  double *K = malloc(sizeof(double) * bb);
  double *S = malloc(sizeof(double) * bb);
  double *Pw = malloc(sizeof(double) * bb);
  double *Tmp = malloc(sizeof(double) * bb);
  double *IpK = malloc(sizeof(double) * bb);
  orc_unpack_skew(theta, b, K);
  mat_identity(b, S);
  mat_identity(b, Pw);
  for (int i = 1; i <= n; ++i) {       /* Pw = K^i, S += Pw */
    mat_mul(b, Pw, K, Tmp);
    memcpy(Pw, Tmp, sizeof(double) * bb);
    for (size_t e = 0; e < bb; ++e) S[e] += Pw[e];
  }
  mat_identity(b, IpK);
  for (size_t e = 0; e < bb; ++e) IpK[e] += K[e];
  mat_mul(b, IpK, S, Q);
  free(K); free(S); free(Pw); free(Tmp); free(IpK);
}

/* theta [nb, b(b-1)/2] -> Q [nb, b, b] */
void orc_cnp(const double *theta, int nb, int b, int n, double *Q) {
  const long p = orc_skew_count(b);
#pragma omp parallel for schedule(dynamic)
  for (int j = 0; j < nb; ++j)
    cnp_block(theta + (size_t)j * p, b, n, Q + (size_t)j * b * b);
}

/* Exact Cayley map C = (I + K)(I - K)^{-1}: the inverse by Gauss-Jordan
 * elimination with partial pivoting.  Returns 0, or -1 on a zero pivot
 * (I - K is never singular for real skew K, so -1 means a bug). */
static int cayley_block(const double *theta, int b, double *C) {
  const size_t bb = (size_t)b * b;
  double *K = malloc(sizeof(double) * bb);
  double *A = malloc(sizeof(double) * bb);    /* I - K, reduced to I */
  double *Inv = malloc(sizeof(double) * bb);  /* I, becomes (I - K)^{-1} */
  double *IpK = malloc(sizeof(double) * bb);
  int rc = 0;
  orc_unpack_skew(theta, b, K);
  mat_identity(b, A);
  for (size_t e = 0; e < bb; ++e) A[e] -= K[e];
  mat_identity(b, Inv);
  for (int c = 0; c < b && rc == 0; ++c) {
    int piv = c;
    for (int r = c + 1; r < b; ++r)
      if (fabs(A[(size_t)r * b + c]) > fabs(A[(size_t)piv * b + c])) piv = r;
    if (A[(size_t)piv * b + c] == 0.0) { rc = -1; break; }
    if (piv != c)
      for (int k = 0; k < b; ++k) {
        double t = A[(size_t)c * b + k];
        A[(size_t)c * b + k] = A[(size_t)piv * b + k];
        A[(size_t)piv * b + k] = t;
        t = Inv[(size_t)c * b + k];
        Inv[(size_t)c * b + k] = Inv[(size_t)piv * b + k];
        Inv[(size_t)piv * b + k] = t;
      }
    const double inv_p = 1.0 / A[(size_t)c * b + c];
    for (int k = 0; k < b; ++k) {
      A[(size_t)c * b + k] *= inv_p;
      Inv[(size_t)c * b + k] *= inv_p;
    }
    for (int r = 0; r < b; ++r) {
      if (r == c) continue;
      const double f = A[(size_t)r * b + c];
      if (f == 0.0) continue;
      for (int k = 0; k < b; ++k) {
        A[(size_t)r * b + k] -= f * A[(size_t)c * b + k];
        Inv[(size_t)r * b + k] -= f * Inv[(size_t)c * b + k];
      }
    }
  }
  if (rc == 0) {
    mat_identity(b, IpK);
    for (size_t e = 0; e < bb; ++e) IpK[e] += K[e];
    mat_mul(b, IpK, Inv, C);
  }
  free(K); free(A); free(Inv); free(IpK);
  return rc;
}

int orc_cayley(const double *theta, int nb, int b, double *C) {
  const long p = orc_skew_count(b);
  int bad = 0;
#pragma omp parallel for schedule(dynamic) reduction(| : bad)
  for (int j = 0; j < nb; ++j)
    bad |= (cayley_block(theta + (size_t)j * p, b, C + (size_t)j * b * b) != 0);
  return bad ? -1 : 0;
}

/* Backward of the Cayley-Neumann map, by the chain rule on
 *   Q = sum_{m=0}^{n+1} c_m K^m,  c_0 = 1, c_m = 2 (1 <= m <= n), c_{n+1} = 1
 * (the expansion of (I + K) sum_{i<=n} K^i).  With d(K^m) =
 * sum_{a=0}^{m-1} K^a dK K^{m-1-a} and <G, A dK B> = <A^T G B^T, dK>:
 *   dL/dK = sum_{m=1}^{n+1} c_m sum_{a=0}^{m-1} (K^a)^T G (K^{m-1-a})^T.
 * Each packed parameter enters K twice (+ at (i,k), - at (k,i)), so
 *   dL/dtheta_(i,k) = dL/dK[i][k] - dL/dK[k][i].
 * The backward is not on the pages (they only say "autograd",
 * [POET-X §2.E]); this is the plain derivative of the forward above. */
static void cnp_backward_block(const double *theta, int b, int n, const double *G,
                               double *dtheta) {
  const size_t bb = (size_t)b * b;
  double *pw = malloc(sizeof(double) * bb * (size_t)(n + 1)); /* K^0..K^n */
  double *pwT = malloc(sizeof(double) * bb * (size_t)(n + 1));
  double *dK = calloc(bb, sizeof(double));
  double *T1 = malloc(sizeof(double) * bb);
  double *T2 = malloc(sizeof(double) * bb);
  orc_unpack_skew(theta, b, T1);
  mat_identity(b, pw);
  for (int m = 1; m <= n; ++m) mat_mul(b, pw + (size_t)(m - 1) * bb, T1, pw + (size_t)m * bb);
  for (int m = 0; m <= n; ++m) mat_transpose(b, pw + (size_t)m * bb, pwT + (size_t)m * bb);
  for (int m = 1; m <= n + 1; ++m) {
    const double cm = (m <= n) ? 2.0 : 1.0;
    for (int a = 0; a <= m - 1; ++a) {
      mat_mul(b, pwT + (size_t)a * bb, G, T1);                     /* (K^a)^T G */
      mat_mul(b, T1, pwT + (size_t)(m - 1 - a) * bb, T2);          /* ... (K^{m-1-a})^T */
      for (size_t e = 0; e < bb; ++e) dK[e] += cm * T2[e];
    }
  }
  long p = 0;
  for (int i = 0; i < b; ++i)
    for (int k = i + 1; k < b; ++k)
      dtheta[p++] = dK[(size_t)i * b + k] - dK[(size_t)k * b + i];
  free(pw); free(pwT); free(dK); free(T1); free(T2);
}

void orc_cnp_backward(const double *theta, int nb, int b, int n, const double *dQ,
                      double *dtheta) {
  const long p = orc_skew_count(b);
#pragma omp parallel for schedule(dynamic)
  for (int j = 0; j < nb; ++j)
    cnp_backward_block(theta + (size_t)j * p, b, n, dQ + (size_t)j * b * b,
                       dtheta + (size_t)j * p);
}

/* ------------------------------------------------------------------ */
/* [POET-X §2.B] permutations as index maps                             */
/* ------------------------------------------------------------------ */

/* inv[perm[i]] = i.  Returns 0, or -1 if perm is not a permutation of 0..d-1. */
int orc_invert_perm(const int32_t *perm, int d, int32_t *inv) {
  for (int i = 0; i < d; ++i) inv[i] = -1;
  for (int i = 0; i < d; ++i) {
    const int32_t v = perm[i];
    if (v < 0 || v >= d || inv[v] != -1) return -1;
    inv[v] = i;
  }
  return 0;
}

/* Dense permutation matrix, Pi[i][perm[i]] = 1, so (Pi v)_i = v_{perm(i)}. */
void orc_perm_matrix(const int32_t *perm, int d, double *Pi) {
  memset(Pi, 0, sizeof(double) * (size_t)d * d);
  for (int i = 0; i < d; ++i) Pi[(size_t)i * d + perm[i]] = 1.0;
}

/* Dense blockdiag(Q_0..Q_{nb-1}), d = nb*b. */
void orc_blockdiag(const double *Qs, int nb, int b, double *B) {
  const int d = nb * b;
  memset(B, 0, sizeof(double) * (size_t)d * d);
  for (int j = 0; j < nb; ++j)
    for (int i = 0; i < b; ++i)
      for (int k = 0; k < b; ++k)
        B[(size_t)(j * b + i) * d + (j * b + k)] = Qs[((size_t)j * b + i) * b + k];
}

/* [POET-X §2.B] merged weight: W0m = Pi_R W0 Pi_P^T, i.e.
 * W0m[i][k] = W0[perm_out[i]][perm_in[k]], W0 [d_out, d_in]. */
void orc_merge_w0(const double *W0, int d_out, int d_in, const int32_t *perm_out,
                  const int32_t *perm_in, double *W0m) {
  for (int i = 0; i < d_out; ++i)
    for (int k = 0; k < d_in; ++k)
      W0m[(size_t)i * d_in + k] = W0[(size_t)perm_out[i] * d_in + perm_in[k]];
}

/* ------------------------------------------------------------------ */
/* [POET-X §2.A-§2.C] the transformed linear, input-centric              */
/* ------------------------------------------------------------------ */

/* out_j = Q_j v_j for every block j (v, out of length nb*b). */
static void block_apply(const double *Qs, int nb, int b, const double *v, double *out) {
  for (int j = 0; j < nb; ++j)
    for (int i = 0; i < b; ++i) {
      const double *q = Qs + ((size_t)j * b + i) * b;
      const double *vj = v + (size_t)j * b;
      double s = 0.0;
      for (int k = 0; k < b; ++k) s += q[k] * vj[k];
      out[(size_t)j * b + i] = s;
    }
}

/* out_j = Q_j^T v_j for every block j. */
static void block_apply_t(const double *Qs, int nb, int b, const double *v, double *out) {
  for (int j = 0; j < nb; ++j)
    for (int k = 0; k < b; ++k) {
      double s = 0.0;
      for (int i = 0; i < b; ++i)
        s += Qs[((size_t)j * b + i) * b + k] * v[(size_t)j * b + i];
      out[(size_t)j * b + k] = s;
    }
}

/* Forward, one token at a time, with the UNMERGED W0 and all four
 * permutation applications:
 *   y = Pi_R^T B_R Pi_R . W0 . Pi_P^T B_P Pi_P x.
 * x [T,d_in], W0 [d_out,d_in], QP [d_in/b_in,b_in,b_in], QR [d_out/b_out,..],
 * y [T,d_out].  If zsave is not NULL it receives z = Pi_R W0 Pi_P^T B_P Pi_P x
 * [T,d_out] (the W0 output in R's permuted order).  */
void orc_forward(int T, int d_in, int d_out, const double *x, const double *W0,
                 const double *QP, int b_in, const double *QR, int b_out,
                 const int32_t *perm_in, const int32_t *perm_out, double *y,
                 double *zsave) {
  const int nbi = d_in / b_in, nbo = d_out / b_out;
#pragma omp parallel
  {
    double *v1 = malloc(sizeof(double) * d_in), *v2 = malloc(sizeof(double) * d_in);
    double *v3 = malloc(sizeof(double) * d_in);
    double *v4 = malloc(sizeof(double) * d_out), *v5 = malloc(sizeof(double) * d_out);
    double *v6 = malloc(sizeof(double) * d_out);
#pragma omp for schedule(static)
    for (int t = 0; t < T; ++t) {
      const double *xt = x + (size_t)t * d_in;
      for (int i = 0; i < d_in; ++i) v1[i] = xt[perm_in[i]];        /* Pi_P x */
      block_apply(QP, nbi, b_in, v1, v2);                           /* B_P . */
      for (int i = 0; i < d_in; ++i) v3[perm_in[i]] = v2[i];        /* Pi_P^T . */
      for (int o = 0; o < d_out; ++o) {                             /* W0 . */
        const double *w = W0 + (size_t)o * d_in;
        double s = 0.0;
        for (int k = 0; k < d_in; ++k) s += w[k] * v3[k];
        v4[o] = s;
      }
      for (int i = 0; i < d_out; ++i) v5[i] = v4[perm_out[i]];      /* Pi_R . */
      block_apply(QR, nbo, b_out, v5, v6);                          /* B_R . */
      double *yt = y + (size_t)t * d_out;
      for (int i = 0; i < d_out; ++i) yt[perm_out[i]] = v6[i];      /* Pi_R^T . */
      if (zsave) memcpy(zsave + (size_t)t * d_out, v5, sizeof(double) * d_out);
    }
    free(v1); free(v2); free(v3); free(v4); free(v5); free(v6);
  }
}

/* Dense forward: y_t = R . W0 . P . x_t with R, P given as dense matrices
 * (P [d_in,d_in], R [d_out,d_out]).  Used to pin the index form above. */
void orc_forward_dense(int T, int d_in, int d_out, const double *x, const double *W0,
                       const double *P, const double *R, double *y) {
#pragma omp parallel
  {
    double *a = malloc(sizeof(double) * d_in), *c = malloc(sizeof(double) * d_out);
#pragma omp for schedule(static)
    for (int t = 0; t < T; ++t) {
      const double *xt = x + (size_t)t * d_in;
      for (int i = 0; i < d_in; ++i) {
        double s = 0.0;
        for (int k = 0; k < d_in; ++k) s += P[(size_t)i * d_in + k] * xt[k];
        a[i] = s;
      }
      for (int o = 0; o < d_out; ++o) {
        double s = 0.0;
        for (int k = 0; k < d_in; ++k) s += W0[(size_t)o * d_in + k] * a[k];
        c[o] = s;
      }
      double *yt = y + (size_t)t * d_out;
      for (int o = 0; o < d_out; ++o) {
        double s = 0.0;
        for (int k = 0; k < d_out; ++k) s += R[(size_t)o * d_out + k] * c[k];
        yt[o] = s;
      }
    }
    free(a); free(c);
  }
}

/* dQ[j][i][k] = sum_{t=0}^{T-1} G[t][j*b+i] * V[t][j*b+k], t in serial order. */
static void dq_token_sum(int T, int d, int b, int nb, const double *G, const double *V,
                         double *dQ) {
#pragma omp parallel for schedule(dynamic) collapse(2)
  for (int j = 0; j < nb; ++j)
    for (int i = 0; i < b; ++i) {
      double *row = dQ + ((size_t)j * b + i) * b;
      for (int k = 0; k < b; ++k) row[k] = 0.0;
      for (int t = 0; t < T; ++t) {
        const double g = G[(size_t)t * d + (size_t)j * b + i];
        const double *v = V + (size_t)t * d + (size_t)j * b;
        for (int k = 0; k < b; ++k) row[k] += g * v[k];
      }
    }
}

/* Backward of orc_forward for an upstream gradient dy [T,d_out]
 * (the loss is linear in y with coefficients dy).  Reverse of the chain
 * x -v1-> v2 -v3-> v4 -v5-> v6 -> y:
 *   g6 = Pi_R dy,  dQ_R,j = sum_t g6_j v5_j^T,  g5 = B_R^T g6,
 *   g4 = Pi_R^T g5, g3 = W0^T g4, g2 = Pi_P g3,
 *   dQ_P,j = sum_t g2_j v1_j^T,  g1 = B_P^T g2,  dx = Pi_P^T g1.
 * Outputs dX [T,d_in], dQP [nbi,b_in,b_in], dQR [nbo,b_out,b_out]. */
void orc_backward(int T, int d_in, int d_out, const double *x, const double *dy,
                  const double *W0, const double *QP, int b_in, const double *QR,
                  int b_out, const int32_t *perm_in, const int32_t *perm_out,
                  double *dX, double *dQP, double *dQR) {
  const int nbi = d_in / b_in, nbo = d_out / b_out;
  /* per-token vectors kept for the token sums of dQ */
  double *V1 = malloc(sizeof(double) * (size_t)T * d_in);
  double *G2 = malloc(sizeof(double) * (size_t)T * d_in);
  double *V5 = malloc(sizeof(double) * (size_t)T * d_out);
  double *G6 = malloc(sizeof(double) * (size_t)T * d_out);
#pragma omp parallel
  {
    double *v2 = malloc(sizeof(double) * d_in), *v3 = malloc(sizeof(double) * d_in);
    double *v4 = malloc(sizeof(double) * d_out);
    double *g5 = malloc(sizeof(double) * d_out), *g4 = malloc(sizeof(double) * d_out);
    double *g3 = malloc(sizeof(double) * d_in), *g1 = malloc(sizeof(double) * d_in);
#pragma omp for schedule(static)
    for (int t = 0; t < T; ++t) {
      double *v1 = V1 + (size_t)t * d_in, *g2 = G2 + (size_t)t * d_in;
      double *v5 = V5 + (size_t)t * d_out, *g6 = G6 + (size_t)t * d_out;
      const double *xt = x + (size_t)t * d_in, *dyt = dy + (size_t)t * d_out;
      /* forward values needed by the backward */
      for (int i = 0; i < d_in; ++i) v1[i] = xt[perm_in[i]];
      block_apply(QP, nbi, b_in, v1, v2);
      for (int i = 0; i < d_in; ++i) v3[perm_in[i]] = v2[i];
      for (int o = 0; o < d_out; ++o) {
        const double *w = W0 + (size_t)o * d_in;
        double s = 0.0;
        for (int k = 0; k < d_in; ++k) s += w[k] * v3[k];
        v4[o] = s;
      }
      for (int i = 0; i < d_out; ++i) v5[i] = v4[perm_out[i]];
      /* backward */
      for (int i = 0; i < d_out; ++i) g6[i] = dyt[perm_out[i]];     /* Pi_R dy */
      block_apply_t(QR, nbo, b_out, g6, g5);                        /* B_R^T . */
      for (int i = 0; i < d_out; ++i) g4[perm_out[i]] = g5[i];      /* Pi_R^T . */
      for (int k = 0; k < d_in; ++k) g3[k] = 0.0;                   /* W0^T . */
      for (int o = 0; o < d_out; ++o) {
        const double *w = W0 + (size_t)o * d_in;
        const double go = g4[o];
        for (int k = 0; k < d_in; ++k) g3[k] += w[k] * go;
      }
      for (int i = 0; i < d_in; ++i) g2[i] = g3[perm_in[i]];        /* Pi_P . */
      block_apply_t(QP, nbi, b_in, g2, g1);                         /* B_P^T . */
      double *dxt = dX + (size_t)t * d_in;
      for (int i = 0; i < d_in; ++i) dxt[perm_in[i]] = g1[i];       /* Pi_P^T . */
    }
    free(v2); free(v3); free(v4); free(g5); free(g4); free(g3); free(g1);
  }
  /* dQ blocks: each entry is a token sum in serial order t = 0..T-1;
   * parallel over (block, row), a row of dQ accumulated at once. */
  dq_token_sum(T, d_out, b_out, nbo, G6, V5, dQR);
  dq_token_sum(T, d_in, b_in, nbi, G2, V1, dQP);
  free(V1); free(G2); free(V5); free(G6);
}
