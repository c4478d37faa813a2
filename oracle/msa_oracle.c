/*
 * msa_oracle.c -- plain fp64 CPU oracle for MiniMax Sparse Attention (MSA) training.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or call this file:
 * only the tests, the package's smoke check and the benchmark's CPU-baseline leg use it.
 * It shares no code, header or constant with the CUDA library.
 *
 * What it computes, and where each step comes from:
 *   "Flash-MSA: Accelerating Million-Token Training with Sparse Attention Kernels" (blog),
 *   sections "About MSA", "Forward > Proxy attention", "Forward > Main attention", "Backward",
 *   "KL Divergence Loss" and "Warmup kernels"; and the forum summary "MiniMax Sparse Attention
 *   (MSA): Turning Theoretical Sparse Attention Gains into Real GPU Speedups", sections
 *   "Architecture: two-stage block-sparse attention" and "Training stability".
 *
 *   For batch b, proxy head g (one MSA group), token t, local block m = t / 128:
 *   1. proxy scores   z[t,j] = scale * <Qp[b,t,g], Kp[b,j]>       (one shared proxy key head)
 *   2. block scores   c[n] = max over the 128 keys of block n of z, for every block n < m;
 *                     the local block m is forced to +infinity ("set the local KV block to inf")
 *   3. selection      the first K = min(top_k, m+1) blocks under (c descending, n ascending);
 *                     emitted in ascending block order, padded with -1
 *   4. key set        J = union of the selected blocks, cut causally at t (j <= t)
 *   5. main attention softmax(scale * <Q[b,t,h], K[b,j,h/G]>) over J for every query head h of
 *                     proxy head g (h / Gp == g, Gp = Hq/Hp), O = sum P V, LSE = log sum exp;
 *                     keys and values come from h's own KV head h / G (G = Hq/Hkv)
 *   6. teacher        pbar = mean over the Gp heads of the main probabilities (stop-gradient);
 *      student        p_px = softmax over J of z
 *   7. KL             L_KL = 1/(B*S*Hp) * sum over (b,t,g) of KL(pbar || p_px)
 *   8. main gradients textbook softmax-attention backward of  L = sum(O * dO) + kl_grad * L_KL;
 *                     the teacher is detached, so the KL term adds nothing to dQ, dK, dV
 *   9. proxy grads    dz = kl_grad/(B*S*Hp) * (p_px - pbar)   (the blog's closed form)
 *                     dQp = scale * sum_j dz_j Kp_j ; dKp_j += scale * dz_j Qp
 *  10. warmup         same as 5-9 with J = [0, t] and no selection.
 *
 * Head mapping (blog, "Note about scheduler requiring proxy heads >= KV heads"; package caveat 5):
 * the MSA group is the proxy head.  With Hp == Hkv it is one GQA group; with Hp < Hkv one proxy
 * head selects for Hkv/Hp whole GQA groups (the inverted mapping the blog's kernels do not
 * schedule) and its teacher averages all their Hq/Hp query heads; with Hp > Hkv a GQA group is
 * split among Hp/Hkv proxy heads.  Query heads of proxy head g are g*Gp .. g*Gp + Gp - 1.
 *
 * Plain loops, no blocking and no fusion beyond the steps above.  Every array is contiguous:
 *   q    [B,S,Hq,D]   k, v [B,S,Hkv,D]   qp [B,S,Hp,D]   kp [B,S,D]   dout [B,S,Hq,D]
 *   idx  [B,Hp,S,top_k] int32 (ascending, -1 padded)       o [B,S,Hq,D]   lse [B,Hq,S]
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define MSA_ORACLE_BLOCK 128

static double dot(const double* a, const double* b, int n) {
  double s = 0.0;
  for (int i = 0; i < n; ++i) s += a[i] * b[i];
  return s;
}

/* Index helpers for the contiguous layouts above. */
static size_t at4(int b, int t, int h, int S, int H, int D) {
  return (((size_t)b * S + t) * H + h) * (size_t)D;
}

int msa_oracle_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void msa_oracle_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

/* Does block n come before block n2 in the selection order (score descending, index ascending)? */
static int ranks_before(double c1, int n1, double c2, int n2) {
  if (c1 > c2) return 1;
  if (c1 < c2) return 0;
  return n1 < n2;
}

/*
 * Steps 1-3 for one row (b, g, t).  Writes top_k entries into out (ascending, -1 padded) and
 * returns in *gap the relative gap between the last selected and the first unselected
 * non-local block score (+inf when every visible block is selected).
 * c is scratch of at least S/128 doubles.
 */
static void select_row(int b, int g, int t, int S, int Hp, int D, int top_k, double scale,
                       const double* qp, const double* kp, double* c, char* taken,
                       int32_t* out, double* gap) {
  const int m = t / MSA_ORACLE_BLOCK;
  const double* qrow = qp + at4(b, t, g, S, Hp, D);
  /* steps 1-2: block max of the proxy scores over the fully visible earlier blocks */
  for (int n = 0; n < m; ++n) {
    double best = -INFINITY;
    for (int j = n * MSA_ORACLE_BLOCK; j < (n + 1) * MSA_ORACLE_BLOCK; ++j) {
      double z = scale * dot(qrow, kp + ((size_t)b * S + j) * D, D);
      if (z > best) best = z;
    }
    c[n] = best;
  }
  c[m] = INFINITY; /* forced local block */
  /* step 3: repeated selection of the best remaining block, K times */
  const int K = top_k < m + 1 ? top_k : m + 1;
  for (int n = 0; n <= m; ++n) taken[n] = 0;
  for (int r = 0; r < K; ++r) {
    int best = -1;
    for (int n = 0; n <= m; ++n) {
      if (taken[n]) continue;
      if (best < 0 || ranks_before(c[n], n, c[best], best)) best = n;
    }
    taken[best] = 1;
  }
  int w = 0;
  for (int n = 0; n <= m; ++n)
    if (taken[n]) out[w++] = n;
  for (; w < top_k; ++w) out[w] = -1;
  /* near-tie report: lowest selected non-local score vs highest unselected score */
  double lo_sel = INFINITY, hi_uns = -INFINITY;
  int any_sel = 0, any_uns = 0;
  for (int n = 0; n < m; ++n) {
    if (taken[n]) {
      any_sel = 1;
      if (c[n] < lo_sel) lo_sel = c[n];
    } else {
      any_uns = 1;
      if (c[n] > hi_uns) hi_uns = c[n];
    }
  }
  if (!any_uns) {
    *gap = INFINITY;
  } else if (!any_sel) {
    /* only the local block is selected (top_k == 1): nothing can flip */
    *gap = INFINITY;
  } else {
    double den = fabs(lo_sel) > fabs(hi_uns) ? fabs(lo_sel) : fabs(hi_uns);
    *gap = den > 0.0 ? (lo_sel - hi_uns) / den : 0.0;
  }
}

/*
 * Selection for every row (rows == NULL; idx_out is [B,Hp,S,top_k], gap_out [B,Hp,S]) or for
 * nrows given rows (rows is nrows triples b,g,t; idx_out [nrows,top_k], gap_out [nrows]).
 */
int msa_oracle_select(int B, int S, int Hp, int D, int top_k, double scale, const double* qp,
                      const double* kp, int nrows, const int32_t* rows, int32_t* idx_out,
                      double* gap_out) {
  if (S % MSA_ORACLE_BLOCK != 0 || top_k < 1) return 1;
  const long total = rows ? nrows : (long)B * Hp * S;
  const int nblk = S / MSA_ORACLE_BLOCK;
#pragma omp parallel
  {
    double* c = (double*)malloc(sizeof(double) * (nblk + 1));
    char* taken = (char*)malloc(nblk + 1);
#pragma omp for schedule(dynamic, 16)
    for (long r = 0; r < total; ++r) {
      int b, g, t;
      if (rows) {
        b = rows[3 * r];
        g = rows[3 * r + 1];
        t = rows[3 * r + 2];
      } else {
        b = (int)(r / ((long)Hp * S));
        g = (int)((r / S) % Hp);
        t = (int)(r % S);
      }
      select_row(b, g, t, S, Hp, D, top_k, scale, qp, kp, c, taken, idx_out + r * top_k,
                 gap_out + r);
    }
    free(c);
    free(taken);
  }
  return 0;
}

/*
 * Step 4: the key set of row (b, g, t) as a list of key positions, ascending.
 * idx == NULL means warmup: J = [0, t].  Returns |J|.
 */
static int key_set(int b, int g, int t, int S, int Hp, int top_k, const int32_t* idx,
                   int32_t* J) {
  int nj = 0;
  if (!idx) {
    for (int j = 0; j <= t; ++j) J[nj++] = j;
    return nj;
  }
  const int32_t* sel = idx + (((size_t)b * Hp + g) * S + t) * top_k;
  for (int s = 0; s < top_k; ++s) {
    int n = sel[s];
    if (n < 0) continue;
    for (int j = n * MSA_ORACLE_BLOCK; j < (n + 1) * MSA_ORACLE_BLOCK && j <= t; ++j) J[nj++] = j;
  }
  return nj;
}

/*
 * Step 5 for one (b, t, h): probabilities P over J, output o (D values) and the LSE.
 */
static double attend_row(int b, int t, int h, int S, int Hq, int Hkv, int D, double scale,
                         const double* q, const double* k, const double* v, const int32_t* J,
                         int nj, double* P, double* o) {
  const int G = Hq / Hkv;
  const int g = h / G;
  const double* qrow = q + at4(b, t, h, S, Hq, D);
  double mx = -INFINITY;
  for (int a = 0; a < nj; ++a) {
    P[a] = scale * dot(qrow, k + at4(b, J[a], g, S, Hkv, D), D);
    if (P[a] > mx) mx = P[a];
  }
  double sum = 0.0;
  for (int a = 0; a < nj; ++a) {
    P[a] = exp(P[a] - mx);
    sum += P[a];
  }
  for (int a = 0; a < nj; ++a) P[a] /= sum;
  for (int d = 0; d < D; ++d) o[d] = 0.0;
  for (int a = 0; a < nj; ++a) {
    const double* vrow = v + at4(b, J[a], g, S, Hkv, D);
    for (int d = 0; d < D; ++d) o[d] += P[a] * vrow[d];
  }
  return mx + log(sum);
}

/*
 * Forward for every (b,t,h) (rows == NULL: o_out [B,S,Hq,D], lse_out [B,Hq,S]) or for nrows
 * given triples (b, t, h) (o_out [nrows,D], lse_out [nrows]).  idx == NULL: warmup (dense).
 */
/* Head counts the mapping above accepts. */
static int heads_ok(int Hq, int Hkv, int Hp) {
  if (Hq <= 0 || Hkv <= 0 || Hp <= 0 || Hq % Hkv != 0 || Hq % Hp != 0) return 0;
  return Hp % Hkv == 0 || Hkv % Hp == 0;
}

int msa_oracle_forward(int B, int S, int Hq, int Hkv, int Hp, int D, int top_k, double scale,
                       const double* q, const double* k, const double* v, const int32_t* idx,
                       int nrows, const int32_t* rows, double* o_out, double* lse_out) {
  if (!heads_ok(Hq, Hkv, Hp)) return 1;
  const long total = rows ? nrows : (long)B * S * Hq;
  const int maxJ = idx ? (top_k * MSA_ORACLE_BLOCK < S ? top_k * MSA_ORACLE_BLOCK : S) : S;
#pragma omp parallel
  {
    int32_t* J = (int32_t*)malloc(sizeof(int32_t) * (size_t)maxJ);
    double* P = (double*)malloc(sizeof(double) * (size_t)maxJ);
#pragma omp for schedule(dynamic, 16)
    for (long r = 0; r < total; ++r) {
      int b, t, h;
      if (rows) {
        b = rows[3 * r];
        t = rows[3 * r + 1];
        h = rows[3 * r + 2];
      } else {
        b = (int)(r / ((long)S * Hq));
        t = (int)((r / Hq) % S);
        h = (int)(r % Hq);
      }
      const int g = h / (Hq / Hp); /* the proxy head whose selection h uses */
      int nj = key_set(b, g, t, S, Hp, top_k, idx, J);
      double lse = attend_row(b, t, h, S, Hq, Hkv, D, scale, q, k, v, J, nj, P,
                              o_out + (rows ? (size_t)r * D : at4(b, t, h, S, Hq, D)));
      if (rows)
        lse_out[r] = lse;
      else
        lse_out[((size_t)b * Hq + h) * S + t] = lse;
    }
    free(J);
    free(P);
  }
  return 0;
}

/*
 * Steps 5-10 and the KL value.  Gradients of  L = sum(O * dO) + kl_grad * L_KL.
 *
 * Sampling (for long sequences): dq/dqp are produced only for the tokens flagged in tok_mask
 * ([B,S] bytes, NULL = every token); dk/dv/dkp only for keys in [kj0, kj1) (other entries are
 * left untouched).  With only_masked != 0 the tokens outside tok_mask are skipped entirely, which
 * gives the exact contribution of the flagged tokens to every gradient (used to time a bounded
 * sample of a workload).  Outputs use the full layouts (dq [B,S,Hq,D], dk/dv [B,S,Hkv,D],
 * dqp [B,S,Hp,D], dkp [B,S,D]) and must be zeroed by the caller.  kl_out receives L_KL (summed
 * over every row visited, i.e. the exact KL when nothing is sampled).  idx == NULL: warmup.
 */
int msa_oracle_backward(int B, int S, int Hq, int Hkv, int Hp, int D, int top_k, double scale,
                        double kl_grad, const double* q, const double* k, const double* v,
                        const double* qp, const double* kp, const double* dout,
                        const int32_t* idx, const unsigned char* tok_mask, int only_masked,
                        int kj0, int kj1, double* dq, double* dk, double* dv, double* dqp, double* dkp,
                        double* kl_out) {
  if (!heads_ok(Hq, Hkv, Hp)) return 1;
  const int G = Hq / Hkv;  /* query heads per KV head */
  const int Gp = Hq / Hp;  /* query heads per proxy head (the teacher's average) */
  /* Work unit of one thread: (b, c) with c the coarser of the two groupings, so that every
   * gradient row a unit writes (dq, dk, dv, dqp) belongs to it alone: a proxy head (Hp <= Hkv)
   * with its whole KV heads, or a KV head (Hp > Hkv) with the proxy heads that split it. */
  const int Hu = Hp < Hkv ? Hp : Hkv;
  const int per_unit = Hp / Hu;  /* proxy heads per unit */
  const double cz = kl_grad / ((double)B * S * Hp); /* step 9 factor: mean over (b,t,g) */
  const int npairs = B * Hu;
  const int nwin = kj1 > kj0 ? kj1 - kj0 : 0;
  const int maxJ = idx ? (top_k * MSA_ORACLE_BLOCK < S ? top_k * MSA_ORACLE_BLOCK : S) : S;
  double* dkp_part = (double*)calloc((size_t)npairs * (size_t)nwin * D + 1, sizeof(double));
  double* kl_part = (double*)calloc((size_t)npairs, sizeof(double));
  if (!dkp_part || !kl_part) return 2;
#pragma omp parallel
  {
    int32_t* J = (int32_t*)malloc(sizeof(int32_t) * (size_t)maxJ);
    double* P = (double*)malloc(sizeof(double) * (size_t)maxJ * Gp); /* P[h_local][a]  */
    double* dS = (double*)malloc(sizeof(double) * (size_t)maxJ);    /* one head at a time */
    double* pbar = (double*)malloc(sizeof(double) * (size_t)maxJ);
    double* z = (double*)malloc(sizeof(double) * (size_t)maxJ);
    double* o = (double*)malloc(sizeof(double) * (size_t)D);
#pragma omp for schedule(dynamic, 1)
    for (int pr = 0; pr < npairs; ++pr) {
      const int b = pr / Hu;
      double* my_dkp = dkp_part + (size_t)pr * nwin * D; /* rows kj0 .. kj1-1 */
      double kl_acc = 0.0;
      for (int gi = 0; gi < per_unit; ++gi) {
      const int g = (pr % Hu) * per_unit + gi; /* proxy head */
      for (int t = 0; t < S; ++t) {
        const int want_q = !tok_mask || tok_mask[(size_t)b * S + t];
        if (!want_q && (only_masked || t < kj0)) continue; /* nothing of it is in the sample */
        const int nj = key_set(b, g, t, S, Hp, top_k, idx, J);
        int touches = want_q;
        for (int a = 0; a < nj && !touches; ++a)
          if (J[a] >= kj0 && J[a] < kj1) touches = 1;
        if (!touches) continue;
        /* step 5 + main backward, head by head */
        for (int a = 0; a < nj; ++a) pbar[a] = 0.0;
        for (int hl = 0; hl < Gp; ++hl) {
          const int h = g * Gp + hl;
          const int kvh = h / G; /* the KV head of query head h */
          double* Ph = P + (size_t)hl * maxJ;
          attend_row(b, t, h, S, Hq, Hkv, D, scale, q, k, v, J, nj, Ph, o);
          const double* dorow = dout + at4(b, t, h, S, Hq, D);
          const double Drow = dot(dorow, o, D); /* D = rowsum(dO * O) */
          for (int a = 0; a < nj; ++a) {
            double dP = dot(dorow, v + at4(b, J[a], kvh, S, Hkv, D), D);
            dS[a] = Ph[a] * (dP - Drow);
            pbar[a] += Ph[a] / Gp;
          }
          if (want_q) {
            double* dqrow = dq + at4(b, t, h, S, Hq, D);
            for (int a = 0; a < nj; ++a) {
              const double* krow = k + at4(b, J[a], kvh, S, Hkv, D);
              for (int d = 0; d < D; ++d) dqrow[d] += scale * dS[a] * krow[d];
            }
          }
          const double* qrow = q + at4(b, t, h, S, Hq, D);
          for (int a = 0; a < nj; ++a) {
            const int j = J[a];
            if (j < kj0 || j >= kj1) continue;
            double* dkrow = dk + at4(b, j, kvh, S, Hkv, D);
            double* dvrow = dv + at4(b, j, kvh, S, Hkv, D);
            for (int d = 0; d < D; ++d) {
              dkrow[d] += scale * dS[a] * qrow[d];
              dvrow[d] += Ph[a] * dorow[d];
            }
          }
        }
        /* step 6: student over the same key set */
        const double* qprow = qp + at4(b, t, g, S, Hp, D);
        double zmx = -INFINITY;
        for (int a = 0; a < nj; ++a) {
          z[a] = scale * dot(qprow, kp + ((size_t)b * S + J[a]) * D, D);
          if (z[a] > zmx) zmx = z[a];
        }
        double zsum = 0.0;
        for (int a = 0; a < nj; ++a) zsum += exp(z[a] - zmx);
        const double lse_px = zmx + log(zsum);
        /* step 7 (value) and step 9 (gradient) */
        double* dqprow = dqp + at4(b, t, g, S, Hp, D);
        for (int a = 0; a < nj; ++a) {
          const double logp_px = z[a] - lse_px;
          const double p_px = exp(logp_px);
          if (pbar[a] > 0.0) kl_acc += pbar[a] * (log(pbar[a]) - logp_px);
          const double dz = cz * (p_px - pbar[a]);
          const double* kprow = kp + ((size_t)b * S + J[a]) * D;
          if (want_q)
            for (int d = 0; d < D; ++d) dqprow[d] += scale * dz * kprow[d];
          if (J[a] >= kj0 && J[a] < kj1) {
            double* acc = my_dkp + (size_t)(J[a] - kj0) * D;
            for (int d = 0; d < D; ++d) acc[d] += scale * dz * qprow[d];
          }
        }
      }
      }
      kl_part[pr] = kl_acc;
    }
    free(J);
    free(P);
    free(dS);
    free(pbar);
    free(z);
    free(o);
  }
  /* dKp: the proxy key head is shared by every group, so sum the per-(b,g) parts */
  double kl = 0.0;
  for (int pr = 0; pr < npairs; ++pr) {
    const int b = pr / Hu;
    kl += kl_part[pr];
    for (int j = kj0; j < kj1; ++j)
      for (int d = 0; d < D; ++d)
        dkp[((size_t)b * S + j) * D + d] += dkp_part[((size_t)pr * nwin + (j - kj0)) * D + d];
  }
  if (kl_out) *kl_out = kl / ((double)B * S * Hp);
  free(dkp_part);
  free(kl_part);
  return 0;
}
