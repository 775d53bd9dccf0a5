/*
 * attn_oracle.c — plain, slow fp64 CPU oracle for scaled-dot-product attention
 * (forward producing O and the per-row log-sum-exp, and the backward pass).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark use it.  It shares no code, header, table or helper with the
 * CUDA path.
 *
 * What it follows (page titles as printed; sections as numbered there):
 *   - "ops(8)：self-attention 的 CUDA 实现及优化 (下) - 深度分析",
 *       §2.1 "反向传播数学推导" (matrix-product derivative, softmax derivative,
 *       forward S = QK^T/sqrt(d_k), P = softmax(S), O = PV, and the five-step
 *       backward chain rule dV, dP, dS, dQ, dK);
 *       §2.2 "CPU 参考实现" (loop structure of the explicit softmax-Jacobian
 *       backward, causal visibility t2 <= t, scale applied to dpreatt);
 *       Appendix A.1-A.3 (the same formulas restated).
 *   - "深度学习反向传播优化：2-CTA MMA模式与内存访问优化" does not change the
 *       arithmetic; it is about how a kernel schedules it.
 *
 * Readings taken where the pages are silent (each is listed in the design
 * notes of the repository):
 *   - The scale s multiplies the scores: S = s * Q K^T, with s passed in
 *     (the pages use s = 1/sqrt(d_k)).  dQ = s * dS K and dK = s * dS^T Q.
 *   - The softmax statistic that the forward returns is the natural-log
 *     log-sum-exp of the scaled scores: LSE_i = ln sum_j exp(S_ij).
 *   - Causal visibility is key j visible to query i iff j <= i + (Tk - Tq):
 *     with Tq == Tk that is the §2.2 loop's t2 <= t; with fewer queries than
 *     keys (separate query and key lengths, "ops(8)..." §1.3's seq_len_q /
 *     seq_len_kv) the queries are the last Tq positions of the key sequence
 *     (bottom-right alignment), so every query sees at least one key.  Causal
 *     with Tq > Tk would leave rows with no visible key and is rejected.
 *   - Local (sliding-window) attention, a mask mode of the kind "深度学习反向
 *     传播优化：2-CTA MMA模式与内存访问优化" §5.2 keeps as an independent module
 *     (§5.1: FlexAttention-style variants): with window (wl, wr), wl, wr >= 0,
 *     key j is visible to query i iff
 *     i + off - wl <= j <= i + off + wr (off = Tk - Tq; -1 = no bound on that
 *     side), intersected with the causal bound when causal is set.  The
 *     band's visible keys of a row are one contiguous range.
 *   - Block-sparse attention, the other mask module §5.2 names next to the
 *     causal one ("因果/块稀疏"): the caller marks which pairs of blocks of
 *     `block` consecutive queries and keys take part.  Key j is visible to
 *     query i iff it is in the band above AND mask[i / block][j / block] is
 *     non-zero.  A row can then see no key at all; its output is O_i = 0 with
 *     LSE_i = -inf, and it contributes nothing to any gradient (the limit of
 *     an empty softmax sum, and what a masked score of -inf everywhere gives
 *     once 0 * log 0 is taken as 0).
 *
 * Data layout: a "problem" is one (sequence, head) pair.  All matrices are
 * fp64, row-major, one row per token:
 *   Q, dO, O, dQ : rows qrow0[p] .. qrow0[p]+Tq[p]-1 of [*, dqk] / [*, dv]
 *   K, V, dK, dV : rows krow0[p] .. krow0[p]+Tk[p]-1 of [*, dqk] / [*, dv]
 *   LSE, D       : entries qrow0[p] .. (one per query row)
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

/*
 * ORACLE_PLANT selects a deliberately wrong variant for the mutation tests
 * (which check that the pins catch plausible mistakes).  It is 0 in every
 * build that is used as the oracle.
 *   1: dQ without the scale factor        2: wrong sign of D in dS
 *   3: causal mask off by one (j < i)     4: dV indexed by the key's own row
 *   5: LSE returned in log base 2         6: dK takes dS^T K instead of dS^T Q
 *   7: block mask read transposed ([key block][query block])
 *   8: window's left bound off by one (one key too many)
 *   9: a row that sees no key returns LSE = 0 instead of -inf
 */
#ifndef ORACLE_PLANT
#define ORACLE_PLANT 0
#endif

#define ORACLE_OK 0
#define ORACLE_ERR_ARG (-1)
#define ORACLE_ERR_NOMEM (-2)

/* Keys visible to query row i: lo .. hi (inclusive), one contiguous range:
 * causal: j <= i + off; window (wl, wr >= 0): i + off - wl <= j <= i + off + wr;
 * off = Tk - Tq; -1 leaves that side of the window open. */
static void visible_range(int causal, int wl, int wr, int i, int Tq, int Tk, int *lo,
                          int *hi) {
  const int off = Tk - Tq;
  int l = 0, h = Tk - 1;
  if (causal) h = (ORACLE_PLANT == 3 && i > 0) ? i + off - 1 : i + off;
  if (wr >= 0 && i + off + wr < h) h = i + off + wr;
  if (wl >= 0 && i + off - wl - (ORACLE_PLANT == 8) > l) l = i + off - wl - (ORACLE_PLANT == 8);
  if (h > Tk - 1) h = Tk - 1;
  *lo = l;
  *hi = h;
}

/* Visibility rule of one problem: the band, and an optional block mask
 * (this problem's [nqb][nkb] matrix, row stride bm_nk, blocks of `block`). */
typedef struct {
  int causal, wl, wr;
  const unsigned char *bm;
  int bm_nk, block;
} Vis;

static int block_on(const Vis *vis, int i, int j) {
  if (!vis->bm) return 1;
  const int bi = i / vis->block, bj = j / vis->block;
  return ORACLE_PLANT == 7 ? vis->bm[(long long)bj * vis->bm_nk + bi] != 0
                           : vis->bm[(long long)bi * vis->bm_nk + bj] != 0;
}

static int visible(const Vis *vis, int i, int j, int Tq, int Tk) {
  int lo, hi;
  visible_range(vis->causal, vis->wl, vis->wr, i, Tq, Tk, &lo, &hi);
  return j >= lo && j <= hi && block_on(vis, i, j);
}

/* The keys query row i sees, ascending, into idx; returns how many. */
static int row_keys(const Vis *vis, int i, int Tq, int Tk, int *idx) {
  int lo, hi, n = 0;
  visible_range(vis->causal, vis->wl, vis->wr, i, Tq, Tk, &lo, &hi);
  for (int j = lo; j <= hi; j++)
    if (block_on(vis, i, j)) idx[n++] = j;
  return n;
}

/* A block mask must cover the problem: nqb * block >= Tq, nkb * block >= Tk. */
static int check_mask(const unsigned char *bm, int nqb, int nkb, int block, int Tq, int Tk) {
  if (!bm) return ORACLE_OK;
  if (block <= 0 || nqb <= 0 || nkb <= 0) return ORACLE_ERR_ARG;
  if ((long long)nqb * block < Tq || (long long)nkb * block < Tk) return ORACLE_ERR_ARG;
  return ORACLE_OK;
}

static int check_problem(int causal, int wl, int wr, int Tq, int Tk) {
  if (Tq < 0 || Tk <= 0 || wl < -1 || wr < -1) return ORACLE_ERR_ARG;
  /* with more queries than keys a bound could leave a row with no key */
  if ((causal || wl >= 0 || wr >= 0) && Tq > Tk) return ORACLE_ERR_ARG;
  return ORACLE_OK;
}

/*
 * One query row of the forward, by definition (§2.1 forward, Appendix A.1):
 *   S_ij = s * sum_c Q_ic K_jc            for the visible keys j = idx[0..n)
 *   P_ij = exp(S_ij) / sum_j' exp(S_ij')   (softmax; max subtracted first)
 *   O_i  = sum_j P_ij V_j
 *   LSE_i = ln sum_j exp(S_ij)
 * K and V are the problem's full key rows.  `P` receives the probabilities of
 * the n visible keys (caller's scratch).  With no visible key (n == 0) the
 * sums are empty: O_i = 0 and LSE_i = -inf.
 */
static void forward_row(const double *q, const double *K, const double *V,
                        const int *idx, int n, int dqk, int dv, double scale, double *P,
                        double *o, double *lse) {
  if (o)
    for (int c = 0; c < dv; c++) o[c] = 0.0;
  if (n == 0) {
    if (lse) *lse = (ORACLE_PLANT == 9) ? 0.0 : -INFINITY;
    return;
  }
  double m = -INFINITY;
  for (int t = 0; t < n; t++) {
    double s = 0.0;
    for (int c = 0; c < dqk; c++) s += q[c] * K[(long long)idx[t] * dqk + c];
    s *= scale;
    P[t] = s;
    if (s > m) m = s;
  }
  double sum = 0.0;
  for (int t = 0; t < n; t++) {
    P[t] = exp(P[t] - m);
    sum += P[t];
  }
  for (int t = 0; t < n; t++) P[t] /= sum;
  if (o)
    for (int t = 0; t < n; t++)
      for (int c = 0; c < dv; c++) o[c] += P[t] * V[(long long)idx[t] * dv + c];
  if (lse) *lse = (ORACLE_PLANT == 5) ? (m + log(sum)) / log(2.0) : m + log(sum);
}

/* dP_ij = sum_c dO_ic V_jc for j = idx[0..n)  (§2.1 backward step 2: dP = dO V^T) */
static void dp_row(const double *dout, const double *V, const int *idx, int n, int dv,
                   double *dP) {
  for (int t = 0; t < n; t++) {
    double s = 0.0;
    for (int c = 0; c < dv; c++) s += dout[c] * V[(long long)idx[t] * dv + c];
    dP[t] = s;
  }
}

/*
 * Forward over all problems.  Rows are independent, so the loop runs over
 * every (problem, query row) pair.  When dO and D are given it also returns
 * D_i = sum_j P_ij dP_ij (the row sum that the softmax backward subtracts,
 * §2.1 step 3, written from its definition).
 * bmask: optional block masks, one [bm_nq][bm_nk] uint8 matrix per problem
 * (problem p's at bmask + p * bm_nq * bm_nk), blocks of `block` rows.
 */
int oracle_forward(int nprob, const long long *qrow0, const int *Tq,
                   const long long *krow0, const int *Tk, int dqk, int dv,
                   int causal, int wl, int wr, const unsigned char *bmask, int bm_nq,
                   int bm_nk, int block, double scale, const double *Q,
                   const double *K, const double *V, const double *dO, double *O,
                   double *LSE, double *D) {
  if (nprob < 0 || dqk <= 0 || dv <= 0) return ORACLE_ERR_ARG;
  long long total = 0;
  int maxTk = 1;
  for (int p = 0; p < nprob; p++) {
    if (check_problem(causal, wl, wr, Tq[p], Tk[p])) return ORACLE_ERR_ARG;
    if (check_mask(bmask, bm_nq, bm_nk, block, Tq[p], Tk[p])) return ORACLE_ERR_ARG;
    total += Tq[p];
    if (Tk[p] > maxTk) maxTk = Tk[p];
  }
  /* flattened (problem, row) index */
  long long *start = (long long *)malloc(sizeof(long long) * (nprob + 1));
  if (!start) return ORACLE_ERR_NOMEM;
  start[0] = 0;
  for (int p = 0; p < nprob; p++) start[p + 1] = start[p] + Tq[p];
  int err = ORACLE_OK;
#pragma omp parallel
  {
    double *P = (double *)malloc(sizeof(double) * maxTk);
    double *dP = (double *)malloc(sizeof(double) * maxTk);
    int *idx = (int *)malloc(sizeof(int) * maxTk);
    if (!P || !dP || !idx) {
#pragma omp atomic write
      err = ORACLE_ERR_NOMEM;
    } else {
#pragma omp for schedule(dynamic, 8)
      for (long long r = 0; r < total; r++) {
        int lo = 0, hi = nprob - 1; /* problem holding flattened row r */
        while (lo < hi) {
          int mid = (lo + hi + 1) / 2;
          if (start[mid] <= r) lo = mid; else hi = mid - 1;
        }
        int p = lo;
        int i = (int)(r - start[p]);
        long long qi = qrow0[p] + i;
        Vis vis = {causal, wl, wr,
                   bmask ? bmask + (long long)p * bm_nq * bm_nk : NULL, bm_nk, block};
        const int n = row_keys(&vis, i, Tq[p], Tk[p], idx);
        const double *Kp = K + krow0[p] * dqk;
        const double *Vp = V + krow0[p] * dv;
        double lse;
        forward_row(Q + qi * dqk, Kp, Vp, idx, n, dqk, dv, scale, P,
                    O ? O + qi * dv : NULL, &lse);
        if (LSE) LSE[qi] = lse;
        if (dO && D) {
          dp_row(dO + qi * dv, Vp, idx, n, dv, dP);
          double d = 0.0;
          for (int t = 0; t < n; t++) d += P[t] * dP[t];
          D[qi] = d;
        }
      }
    }
    free(P);
    free(dP);
    free(idx);
  }
  free(start);
  return err;
}

/*
 * Backward of one problem, row by row, for the query rows listed in `rows`
 * (all rows when rows == NULL).  For each row i (§2.1 backward, steps 1-5),
 * over the keys j that row i sees:
 *   P_i  = softmax(S_i)                      (recomputed from Q, K)
 *   dV_j += P_ij dO_i                         (step 1: dV = P^T dO)
 *   dP_ij = dO_i . V_j                        (step 2: dP = dO V^T)
 *   dS_i  = softmax backward of dP_i          (step 3)
 *   dQ_i  = s sum_j dS_ij K_j                 (step 4: dQ = dS K / sqrt(d_k))
 *   dK_j += s dS_ij Q_i                       (step 5: dK = dS^T Q / sqrt(d_k))
 * Step 3 has two forms:
 *   mode 0 (row JVP):  dS_ij = P_ij (dP_ij - sum_k P_ik dP_ik)
 *   mode 1 (explicit Jacobian, as in the §2.2 CPU loop and the softmax
 *           derivative of §2.1 / Appendix A.3):
 *           J_kj = P_ik (delta_kj - P_ij);  dS_ij = sum_k J_kj dP_ik
 * A row that sees no key has empty sums: dQ_i = 0, D_i = 0, and it adds
 * nothing to dK or dV.
 * dK and dV of the problem are zeroed first and receive the contributions of
 * the listed rows only; with all rows they are the full gradients.
 * Optional per-row outputs: O, LSE, D (= sum_j P_ij dP_ij), dQ, and for tiny
 * cases the full Tq x Tk matrices P and dS of the problem (zero where masked).
 */
static int backward_problem(int mode, int Tq, int Tk, int dqk, int dv, const Vis *vis,
                            double scale, const double *Q,
                            const double *K, const double *V, const double *dO,
                            const int *rows, int nrows, double *dQ, double *dK,
                            double *dV, double *O, double *LSE, double *D,
                            double *Pfull, double *dSfull) {
  double *P = (double *)malloc(sizeof(double) * Tk);
  double *dP = (double *)malloc(sizeof(double) * Tk);
  double *dS = (double *)malloc(sizeof(double) * Tk);
  int *idx = (int *)malloc(sizeof(int) * Tk);
  if (!P || !dP || !dS || !idx) {
    free(P); free(dP); free(dS); free(idx);
    return ORACLE_ERR_NOMEM;
  }
  if (dK) memset(dK, 0, sizeof(double) * (size_t)Tk * dqk);
  if (dV) memset(dV, 0, sizeof(double) * (size_t)Tk * dv);
  if (Pfull) memset(Pfull, 0, sizeof(double) * (size_t)Tq * Tk);
  if (dSfull) memset(dSfull, 0, sizeof(double) * (size_t)Tq * Tk);
  int count = rows ? nrows : Tq;
  for (int r = 0; r < count; r++) {
    int i = rows ? rows[r] : r;
    if (i < 0 || i >= Tq) continue;
    const int n = row_keys(vis, i, Tq, Tk, idx);  /* keys idx[0..n) */
    const double *qi = Q + (long long)i * dqk;
    const double *doi = dO + (long long)i * dv;
    double lse;
    forward_row(qi, K, V, idx, n, dqk, dv, scale, P, O ? O + (long long)i * dv : NULL,
                &lse);
    if (LSE) LSE[i] = lse;
    dp_row(doi, V, idx, n, dv, dP);
    double rowdot = 0.0;
    for (int t = 0; t < n; t++) rowdot += P[t] * dP[t];
    if (D) D[i] = rowdot;
    if (mode == 0) {
      for (int t = 0; t < n; t++)
        dS[t] = P[t] * (dP[t] - (ORACLE_PLANT == 2 ? -rowdot : rowdot));
    } else {
      for (int t = 0; t < n; t++) {
        double acc = 0.0;
        for (int u = 0; u < n; u++) {
          double jac = P[u] * ((u == t ? 1.0 : 0.0) - P[t]);
          acc += jac * dP[u];
        }
        dS[t] = acc;
      }
    }
    if (dV)
      for (int t = 0; t < n; t++)
        for (int c = 0; c < dv; c++)
          dV[(long long)idx[t] * dv + c] +=
              P[t] * (ORACLE_PLANT == 4 ? dO[(long long)idx[t] * dv + c] : doi[c]);
    if (dQ) {
      double *dqi = dQ + (long long)i * dqk;
      for (int c = 0; c < dqk; c++) dqi[c] = 0.0;
      for (int t = 0; t < n; t++)
        for (int c = 0; c < dqk; c++)
          dqi[c] += (ORACLE_PLANT == 1 ? 1.0 : scale) * dS[t] *
                    K[(long long)idx[t] * dqk + c];
    }
    if (dK)
      for (int t = 0; t < n; t++)
        for (int c = 0; c < dqk; c++)
          dK[(long long)idx[t] * dqk + c] +=
              scale * dS[t] * (ORACLE_PLANT == 6 ? K[(long long)i * dqk + c] : qi[c]);
    if (Pfull)
      for (int t = 0; t < n; t++) Pfull[(long long)i * Tk + idx[t]] = P[t];
    if (dSfull)
      for (int t = 0; t < n; t++) dSfull[(long long)i * Tk + idx[t]] = dS[t];
  }
  free(P); free(dP); free(dS); free(idx);
  return ORACLE_OK;
}

/*
 * Backward over all problems (parallel over problems; the rows of one problem
 * run in order because dK and dV accumulate over them).
 * rows/nrows: optional per-problem row subsets, concatenated; rows == NULL
 * means every row.  Pfull / dSfull (optional) are concatenated Tq x Tk blocks.
 * bmask / bm_nq / bm_nk / block: optional block masks as in oracle_forward.
 */
int oracle_backward(int mode, int nprob, const long long *qrow0, const int *Tq,
                    const long long *krow0, const int *Tk, int dqk, int dv,
                    int causal, int wl, int wr, const unsigned char *bmask, int bm_nq,
                    int bm_nk, int block, double scale, const double *Q,
                    const double *K, const double *V, const double *dO, const int *rows,
                    const int *nrows, double *dQ, double *dK, double *dV,
                    double *O, double *LSE, double *D, double *Pfull,
                    double *dSfull) {
  if (nprob < 0 || dqk <= 0 || dv <= 0 || (mode != 0 && mode != 1))
    return ORACLE_ERR_ARG;
  for (int p = 0; p < nprob; p++) {
    if (check_problem(causal, wl, wr, Tq[p], Tk[p])) return ORACLE_ERR_ARG;
    if (check_mask(bmask, bm_nq, bm_nk, block, Tq[p], Tk[p])) return ORACLE_ERR_ARG;
  }
  long long *row_start = (long long *)calloc(nprob + 1, sizeof(long long));
  long long *pt_start = (long long *)calloc(nprob + 1, sizeof(long long));
  if (!row_start || !pt_start) {
    free(row_start); free(pt_start);
    return ORACLE_ERR_NOMEM;
  }
  for (int p = 0; p < nprob; p++) {
    row_start[p + 1] = row_start[p] + (rows ? nrows[p] : 0);
    pt_start[p + 1] = pt_start[p] + (long long)Tq[p] * Tk[p];
  }
  int err = ORACLE_OK;
#pragma omp parallel for schedule(dynamic, 1)
  for (int p = 0; p < nprob; p++) {
    long long q0 = qrow0[p], k0 = krow0[p];
    Vis vis = {causal, wl, wr, bmask ? bmask + (long long)p * bm_nq * bm_nk : NULL, bm_nk,
               block};
    int e = backward_problem(
        mode, Tq[p], Tk[p], dqk, dv, &vis, scale, Q + q0 * dqk, K + k0 * dqk,
        V + k0 * dv, dO + q0 * dv, rows ? rows + row_start[p] : NULL,
        rows ? nrows[p] : 0, dQ ? dQ + q0 * dqk : NULL,
        dK ? dK + k0 * dqk : NULL, dV ? dV + k0 * dv : NULL,
        O ? O + q0 * dv : NULL, LSE ? LSE + q0 : NULL, D ? D + q0 : NULL,
        Pfull ? Pfull + pt_start[p] : NULL, dSfull ? dSfull + pt_start[p] : NULL);
    if (e) {
#pragma omp atomic write
      err = e;
    }
  }
  free(row_start);
  free(pt_start);
  return err;
}

/*
 * dK and dV rows for selected keys of one problem, one key at a time, given
 * the forward statistics LSE_i and D_i of every query row (from
 * oracle_forward).  For key j (§2.1 steps 1-3 and 5, column form):
 *   P_ij  = exp(s Q_i.K_j - LSE_i)          for queries i that see key j
 *   dV_j  = sum_i P_ij dO_i
 *   dS_ij = P_ij (dO_i.V_j - D_i)
 *   dK_j  = s sum_i dS_ij Q_i
 * bm: optional [bm_nq][bm_nk] block mask of the problem (blocks of `block`).
 * Parallel over the listed keys.  Outputs are [nkeys][dqk] and [nkeys][dv].
 */
int oracle_kv_rows(int Tq, int Tk, int dqk, int dv, int causal, int wl, int wr,
                   const unsigned char *bm, int bm_nq, int bm_nk, int block, double scale,
                   const double *Q, const double *K, const double *V,
                   const double *dO, const double *LSE, const double *D,
                   const int *keys, int nkeys, double *dK_rows,
                   double *dV_rows) {
  if (check_problem(causal, wl, wr, Tq, Tk) || dqk <= 0 || dv <= 0 ||
      check_mask(bm, bm_nq, bm_nk, block, Tq, Tk))
    return ORACLE_ERR_ARG;
  const Vis vis = {causal, wl, wr, bm, bm_nk, block};
#pragma omp parallel for schedule(dynamic, 1)
  for (int t = 0; t < nkeys; t++) {
    int j = keys[t];
    double *dk = dK_rows + (long long)t * dqk;
    double *dvr = dV_rows + (long long)t * dv;
    for (int c = 0; c < dqk; c++) dk[c] = 0.0;
    for (int c = 0; c < dv; c++) dvr[c] = 0.0;
    if (j < 0 || j >= Tk) continue;
    const double *kj = K + (long long)j * dqk;
    const double *vj = V + (long long)j * dv;
    for (int i = 0; i < Tq; i++) {
      if (!visible(&vis, i, j, Tq, Tk)) continue;
      const double *qi = Q + (long long)i * dqk;
      const double *doi = dO + (long long)i * dv;
      double s = 0.0;
      for (int c = 0; c < dqk; c++) s += qi[c] * kj[c];
      double pij = exp(scale * s - LSE[i]);
      double dpij = 0.0;
      for (int c = 0; c < dv; c++) dpij += doi[c] * vj[c];
      double dsij = pij * (dpij - D[i]);
      for (int c = 0; c < dv; c++) dvr[c] += pij * doi[c];
      for (int c = 0; c < dqk; c++) dk[c] += scale * dsij * qi[c];
    }
  }
  return ORACLE_OK;
}

/* Number of OpenMP threads a parallel region of this library will use. */
int oracle_num_threads(void) {
  int n = 1;
#pragma omp parallel
  {
#pragma omp single
    {
#ifdef _OPENMP
      extern int omp_get_num_threads(void);
      n = omp_get_num_threads();
#endif
    }
  }
  return n;
}
