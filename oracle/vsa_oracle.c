/*
 * vsa_oracle.c -- plain, slow, CPU reference of 64-token block-sparse video attention (VSA):
 * the k2q index inversion, the forward (O and the base-2 "M form" log-sum-exp) and the
 * backward (dQ, dK, dV).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or call this file:
 * only the tests, the smoke check and the benchmark's CPU-baseline leg use it.  It shares no
 * code, header, table or constant generator with the CUDA library.
 *
 * Every function follows the plain definition of the operation, written out loop by loop in
 * double precision, with no blocking, fusion or reordering beyond what the definition states.
 * Sources (web pages; cited by title and section):
 *   [P1] FastVideo, tests/ listing at commit 62f0bc1 -- commit message of the sm_100a VSA
 *        backward ("Semantics" paragraph: kv blocks are the work unit; count 0 gives zero dK/dV
 *        rows; variable_block_sizes masks padded kv rows).
 *   [P2] FastVideo, fastvideo_kernel/block_sparse_attn_bwd_sm100a.py at 88319b7 -- module
 *        docstring (lse in the Triton "M format" max(qk*sm_scale*log2e)+log2(l); dq and dk carry
 *        sm_scale, dv does not).
 *   [P3] FastVideo, compare main...vsa_bwd_fix -- tests/test_block_sparse_bwd_sm100a.py:
 *        reference() (dense attention restricted to the selected blocks, keys past
 *        variable_block_sizes masked to -inf, loss = sum(out * grad_o)),
 *        invert_indices_torch() (k2q rows list their q blocks ascending, padding 0) and
 *        test_invert_indices_torch_matches_q2k() (each pair once, rows sorted);
 *        block_sparse_bwd_launch_sm100a.cuh: BlockSparseVsaBwdArgs (delta is
 *        rowsum(bf16(o) * dout); k2q entries past the count are unread).
 *   [P5] NVIDIA cudnn-frontend PR #926 -- "Summary"/"Why": a slot participates only inside
 *        the bounded active prefix with its index in [0, S_kv); the prefix length is clamped to
 *        [0, width].
 *
 * Readings where the pages are silent (listed with the others in the design notes):
 *   - A q2k row is a SET of kv blocks: duplicates count once.  Ids outside [0, nb) are skipped
 *     and counts are clamped to [0, topk] ([P5]); every such event is counted and returned.
 *   - A query row with no valid key gets O = 0 and lse = -inf, and contributes nothing to any
 *     gradient.
 *   - Query rows are never masked; only kv rows at or past variable_block_sizes[j] are.
 *
 * Layouts: activations [B, H, S, D] row-major doubles, S = blk * nb; lse [B, H, S];
 * q2k_idx [B, H, nb, topk] int32; q2k_num [B, H, nb]; vbs [nb]; k2q_idx [B, H, nb, nb];
 * k2q_num [B, H, nb].
 *
 * Build: gcc -O2 -fopenmp -shared -fPIC (see oracle.py).  OpenMP only splits independent
 * output rows/blocks across threads; each output element is computed by one thread in a fixed
 * order, so results do not depend on the thread count.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define LOG2E 1.4426950408889634

int vsa_oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Number of valid slots of one q2k row: the count clamped to [0, topk] ([P5]).  *bad is
 * incremented when clamping was needed. */
static int active_slots(int32_t num, int topk, long *bad) {
  if (num < 0) {
    ++*bad;
    return 0;
  }
  if (num > topk) {
    ++*bad;
    return topk;
  }
  return num;
}

/* Does q block row `row` (topk slots, `cnt` active) select kv block j?  Set semantics. */
static int selects(const int32_t *row, int cnt, int j) {
  for (int s = 0; s < cnt; ++s)
    if (row[s] == j) return 1;
  return 0;
}

/* Count of invalid entries (negative/too-large counts, ids outside [0, nb)) in q2k. */
static long count_bad(const int32_t *q2k_idx, const int32_t *q2k_num, long rows, int topk,
                      int nb) {
  long bad = 0;
  for (long r = 0; r < rows; ++r) {
    int cnt = active_slots(q2k_num[r], topk, &bad);
    for (int s = 0; s < cnt; ++s) {
      int32_t j = q2k_idx[r * topk + s];
      if (j < 0 || j >= nb) ++bad;
    }
  }
  return bad;
}

/* ---------------------------------------------------------------------------------------- *
 * Inversion q2k -> k2q ([P3] invert_indices_torch / test_invert_indices_torch_matches_q2k):
 * for every (b, h, kv block j) the q blocks i whose active q2k slots contain j, in ascending
 * order of i, each once; entries past the count are 0.  Returns the number of invalid q2k
 * entries.
 * ---------------------------------------------------------------------------------------- */
long vsa_oracle_invert(const int32_t *q2k_idx, const int32_t *q2k_num, int B, int H, int nq,
                       int topk, int nb, int32_t *k2q_idx, int32_t *k2q_num) {
  long bad = count_bad(q2k_idx, q2k_num, (long)B * H * nq, topk, nb);
  for (long bh = 0; bh < (long)B * H; ++bh) {
    for (int j = 0; j < nb; ++j) {
      int32_t *out = k2q_idx + (bh * nb + j) * (long)nq;
      int n = 0;
      for (int i = 0; i < nq; ++i) {
        long r = bh * nq + i;
        long dummy = 0;
        int cnt = active_slots(q2k_num[r], topk, &dummy);
        if (selects(q2k_idx + r * topk, cnt, j)) out[n++] = i;
      }
      for (int t = n; t < nq; ++t) out[t] = 0;
      k2q_num[bh * nb + j] = n;
    }
  }
  return bad;
}

/* Does query block i of head bh select kv block j (set semantics over its active slots)? */
static int block_selected(const int32_t *q2k_idx, const int32_t *q2k_num, int topk, int nq,
                          long bh, int i, int j) {
  long r = bh * nq + i;
  long dummy = 0;
  int cnt = active_slots(q2k_num[r], topk, &dummy);
  return selects(q2k_idx + r * topk, cnt, j);
}

/* Key token t = j*blk + u of kv block j is visible to query block i iff i selects j and
 * u < variable_block_sizes[j] ([P3] reference(): keep[...] = True for kb*BLOCK .. kb*BLOCK+vbs).
 * The loops below walk j = 0 .. nb-1, test block_selected() once per (i, j), then walk
 * u = 0 .. vbs[j]-1. */

/* Valid kv rows of block j: variable_block_sizes[j] clamped to [0, blk] (out-of-range sizes
 * are an input error; clamping is the reading taken for them). */
static int visible_rows(const int32_t *vbs, int j, int blk) {
  int n = vbs[j];
  return n < 0 ? 0 : (n > blk ? blk : n);
}

static double dot(const double *a, const double *b, int d) {
  double s = 0.0;
  for (int x = 0; x < d; ++x) s += a[x] * b[x];
  return s;
}

/* ---------------------------------------------------------------------------------------- *
 * Forward ([P2] docstring, [P3] reference()).  For each query row r of block i:
 *   z_t   = (q_r . k_t) * sm_scale * log2(e)       over the visible keys t
 *   mz    = max_t z_t,   l = sum_t exp2(z_t - mz)
 *   O_r   = sum_t exp2(z_t - mz) * v_t / l
 *   lse_r = mz + log2(l)                            (the "M form")
 * Rows with no visible key: O_r = 0, lse_r = -inf.
 * qblocks: NULL for every query block, else n_qblocks flat ids (bh * nq + i); rows of other
 * blocks are left untouched.  Returns the number of invalid q2k entries.
 * ---------------------------------------------------------------------------------------- */
long vsa_oracle_fwd(const double *q, const double *k, const double *v, const int32_t *q2k_idx,
                    const int32_t *q2k_num, int topk, const int32_t *vbs, double sm_scale, int B,
                    int H, int S, int D, int blk, const int32_t *qblocks, long n_qblocks,
                    double *o, double *lse) {
  const int nb = S / blk, nq = nb;
  long bad = count_bad(q2k_idx, q2k_num, (long)B * H * nq, topk, nb);
  long n_items = qblocks ? n_qblocks : (long)B * H * nq;
#pragma omp parallel for schedule(dynamic)
  for (long it = 0; it < n_items; ++it) {
    long flat = qblocks ? qblocks[it] : it;
    long bh = flat / nq;
    int i = (int)(flat % nq);
    const double *kh = k + bh * S * (long)D, *vh = v + bh * S * (long)D;
    for (int rr = 0; rr < blk; ++rr) {
      long row = bh * S + (long)i * blk + rr;
      const double *qr = q + row * D;
      double *orow = o + row * D;
      double mz = -INFINITY;
      int any = 0;
      for (int j = 0; j < nb; ++j) {
        if (!block_selected(q2k_idx, q2k_num, topk, nq, bh, i, j)) continue;
        for (int u = 0; u < visible_rows(vbs, j, blk); ++u) {
          double z = dot(qr, kh + ((long)j * blk + u) * D, D) * sm_scale * LOG2E;
          if (z > mz) mz = z;
          any = 1;
        }
      }
      for (int x = 0; x < D; ++x) orow[x] = 0.0;
      if (!any) {
        lse[row] = -INFINITY;
        continue;
      }
      double l = 0.0;
      for (int j = 0; j < nb; ++j) {
        if (!block_selected(q2k_idx, q2k_num, topk, nq, bh, i, j)) continue;
        for (int u = 0; u < visible_rows(vbs, j, blk); ++u) {
          long t = (long)j * blk + u;
          double w = exp2(dot(qr, kh + t * D, D) * sm_scale * LOG2E - mz);
          l += w;
          for (int x = 0; x < D; ++x) orow[x] += w * vh[t * D + x];
        }
      }
      for (int x = 0; x < D; ++x) orow[x] /= l;
      lse[row] = mz + log2(l);
    }
  }
  return bad;
}

/* ---------------------------------------------------------------------------------------- *
 * Backward ([P2] docstring for the scaling; [P3] BlockSparseVsaBwdArgs for Delta; the
 * gradient of loss = sum(O * dO) of [P3] reference()).  Given O (as handed to the backward)
 * and lse in M form, for every visible (r, t):
 *   p_rt    = exp2(z_rt - lse_r)
 *   Delta_r = sum_d O_rd * dO_rd
 *   dp_rt   = dO_r . v_t
 *   ds_rt   = p_rt * (dp_rt - Delta_r)
 *   dV_t   += p_rt * dO_r
 *   dK_t   += ds_rt * q_r * sm_scale
 *   dQ_r   += ds_rt * k_t * sm_scale
 * Invisible keys contribute nothing, so unselected kv blocks and padded kv rows come out 0.
 * qblocks: dQ rows are computed (complete) for these flat q blocks (NULL: all); kvblocks: dK
 * and dV rows are computed (complete) for these flat kv blocks (NULL: all).  Rows not listed
 * are left untouched.  Returns the number of invalid q2k entries.
 * ---------------------------------------------------------------------------------------- */
long vsa_oracle_bwd(const double *q, const double *k, const double *v, const double *o,
                    const double *dout, const double *lse, const int32_t *q2k_idx,
                    const int32_t *q2k_num, int topk, const int32_t *vbs, double sm_scale, int B,
                    int H, int S, int D, int blk, const int32_t *qblocks, long n_qblocks,
                    const int32_t *kvblocks, long n_kvblocks, double *dq, double *dk,
                    double *dv) {
  const int nb = S / blk, nq = nb;
  long bad = count_bad(q2k_idx, q2k_num, (long)B * H * nq, topk, nb);

  /* dQ rows: one query block per iteration. */
  long n_q = qblocks ? n_qblocks : (long)B * H * nq;
#pragma omp parallel for schedule(dynamic)
  for (long it = 0; it < n_q; ++it) {
    long flat = qblocks ? qblocks[it] : it;
    long bh = flat / nq;
    int i = (int)(flat % nq);
    const double *kh = k + bh * S * (long)D, *vh = v + bh * S * (long)D;
    for (int rr = 0; rr < blk; ++rr) {
      long row = bh * S + (long)i * blk + rr;
      const double *qr = q + row * D, *dor = dout + row * D;
      double delta = dot(o + row * D, dor, D);
      double *dqr = dq + row * D;
      for (int x = 0; x < D; ++x) dqr[x] = 0.0;
      for (int j = 0; j < nb; ++j) {
        if (!block_selected(q2k_idx, q2k_num, topk, nq, bh, i, j)) continue;
        for (int u = 0; u < visible_rows(vbs, j, blk); ++u) {
          long t = (long)j * blk + u;
          const double *kt = kh + t * D;
          double p = exp2(dot(qr, kt, D) * sm_scale * LOG2E - lse[row]);
          double dp = dot(dor, vh + t * D, D);
          double ds = p * (dp - delta);
          for (int x = 0; x < D; ++x) dqr[x] += ds * kt[x] * sm_scale;
        }
      }
    }
  }

  /* dK, dV rows: one kv block per iteration; every query row of every block that sees it. */
  long n_kv = kvblocks ? n_kvblocks : (long)B * H * nb;
#pragma omp parallel for schedule(dynamic)
  for (long it = 0; it < n_kv; ++it) {
    long flat = kvblocks ? kvblocks[it] : it;
    long bh = flat / nb;
    int j = (int)(flat % nb);
    for (int u = 0; u < blk; ++u) {
      long trow = bh * S + (long)j * blk + u;
      for (int x = 0; x < D; ++x) dk[trow * D + x] = dv[trow * D + x] = 0.0;
    }
    for (int i = 0; i < nq; ++i) {
      if (!block_selected(q2k_idx, q2k_num, topk, nq, bh, i, j)) continue;
      for (int rr = 0; rr < blk; ++rr) {
        long row = bh * S + (long)i * blk + rr;
        const double *qr = q + row * D, *dor = dout + row * D;
        double delta = dot(o + row * D, dor, D);
        for (int u = 0; u < visible_rows(vbs, j, blk); ++u) {
          long trow = bh * S + (long)j * blk + u;
          double p = exp2(dot(qr, k + trow * D, D) * sm_scale * LOG2E - lse[row]);
          double dp = dot(dor, v + trow * D, D);
          double ds = p * (dp - delta);
          for (int x = 0; x < D; ++x) {
            dv[trow * D + x] += p * dor[x];
            dk[trow * D + x] += ds * qr[x] * sm_scale;
          }
        }
      }
    }
  }
  return bad;
}
