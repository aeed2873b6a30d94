/*
 * Plain fp64 CPU oracle for the log-linear Mamba-2 forward and decode step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call this file;
 * it is used by tests/, by __graft_entry__.smoke() and by bench.py's CPU
 * baseline leg.  It shares no code, header, table or constant with the CUDA
 * path in structured_mask_linear_gb300/csrc.
 *
 * Sources (page 1: "对数线性注意力" news write-up of the log-linear attention
 * paper, https://www.yoousoft.com/industry/3746.html; page 3: the article on
 * masked attention and state-space duality, http://biyoush.com/article/202409/463109.htm):
 *
 *   - the masked form O = (A ⊙ M) V with A = Q Kᵀ and M lower triangular
 *     (page 1, section 结构矩阵，一统注意力变体);
 *   - the Mamba-2 scalar-decay mask M^S(t,s) = prod_{r=s+1..t} a_r, the
 *     1-semiseparable mask of the scalar SSD case A_t = a_t I
 *     (page 3, section 狀態空間對偶性; page 1, section 结构矩阵);
 *   - the Fenwick-tree partition: each position summarises a power-of-two
 *     segment ending at itself, so a query sees O(log T) buckets that are finer
 *     near it (page 1, section 特殊结构：树划分, Fig. 2);
 *   - the hierarchical mask M^H(t,s) = lambda_t^{l(t,s)}, one data-dependent
 *     weight per bucket level (page 1, section 特殊结构：树划分, the matrix form);
 *   - the composition M = M^S ⊙ M^H for log-linear Mamba-2 (page 1, section
 *     对Mamba-2和门控的对数线性推广).
 *
 * The stripped mask formula is read as l(t,s) = 0 for s == t and otherwise the
 * bit length of (t xor s) with 0-indexed positions; that is the Fenwick level
 * of the bucket of t that holds s.  The brute-force form below does not use
 * that formula: it builds the buckets by stripping the lowest set bit of the
 * prefix length, the binary-indexed-tree prefix query itself.
 *
 * Layouts (all row-major, fp64):
 *   q, k : (B, T, G, dk)   with G = H / hpg, head h reads group h / hpg
 *   v, o : (B, T, H, dv)
 *   a    : (B, T, H)       decay in (0, 1]
 *   lam  : (B, T, H, L)    lambda_t^l for l = 0 .. L-1
 *
 * Parity pins live in tests/test_oracle_pins.py; every function here is
 * checked there against an independent construction.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Level of key position s in the bucket structure of query position t
 * (0-indexed, s <= t): 0 on the diagonal, else the bit length of t xor s.
 * Page 1, section 特殊结构：树划分 (reading of the stripped mask formula). */
int oracle_level(long t, long s) {
  unsigned long x = (unsigned long)t ^ (unsigned long)s;
  int l = 0;
  while (x) {
    l++;
    x >>= 1;
  }
  return l;
}

/* Binary-indexed-tree prefix decomposition of the positions [0, n): the tree
 * node with 1-indexed label x covers the x&-x positions ending at x, so the
 * prefix of length n is the node n, then node n - lowbit(n), and so on.
 * Writes the start and the length of each segment, nearest first, and
 * returns how many there are (page 1, section 特殊结构：树划分).  */
int oracle_prefix_buckets(long n, long* lo, long* len, int cap) {
  int cnt = 0;
  long x = n;
  while (x > 0 && cnt < cap) {
    long low = x & (-x);
    lo[cnt] = x - low;
    len[cnt] = low;
    cnt++;
    x -= low;
  }
  return cnt;
}

static int ilog2_exact(long p) {
  int l = 0;
  while ((1L << l) < p) l++;
  return l;
}

/* ---------------------------------------------------------------------------
 * Form Q: the quadratic matrix form o_t = sum_{s<=t} lambda_t^{l(t,s)}
 * M^S(t,s) (q_t . k_s) v_s, with M^S(t,s) = exp(G_t - G_s) and G the fp64
 * running sum of log a (page 1, sections 特殊结构：树划分 and
 * 对Mamba-2和门控的对数线性推广; page 3, section 狀態空間對偶性).
 * ------------------------------------------------------------------------- */
static void form_q_head(long T, long dk, long dv, long L, long qs, long vs, long as, long ls,
                        const double* q, const double* k, const double* v, const double* a,
                        const double* lam, double* o, double* G) {
  double acc = 0.0;
  for (long t = 0; t < T; t++) {
    acc += log(a[t * as]);
    G[t] = acc;
  }
  for (long t = 0; t < T; t++) {
    double* ot = o + t * vs;
    for (long j = 0; j < dv; j++) ot[j] = 0.0;
    const double* qt = q + t * qs;
    for (long s = 0; s <= t; s++) {
      const double* ks = k + s * qs;
      double dot = 0.0;
      for (long i = 0; i < dk; i++) dot += qt[i] * ks[i];
      int l = oracle_level(t, s);
      double w = lam[t * ls + l] * exp(G[t] - G[s]) * dot;
      const double* vsv = v + s * vs;
      for (long j = 0; j < dv; j++) ot[j] += w * vsv[j];
    }
  }
  (void)L;
}

void oracle_form_q(long B, long T, long H, long hpg, long dk, long dv, long L,
                   const double* q, const double* k, const double* v, const double* a,
                   const double* lam, double* o) {
  long G = H / hpg;
#pragma omp parallel for collapse(2) schedule(dynamic)
  for (long b = 0; b < B; b++) {
    for (long h = 0; h < H; h++) {
      double* Gbuf = (double*)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
      long g = h / hpg;
      form_q_head(T, dk, dv, L, G * dk, H * dv, H, H * L,
                  q + (b * T * G + g) * dk, k + (b * T * G + g) * dk,
                  v + (b * T * H + h) * dv, a + b * T * H + h,
                  lam + (b * T * H + h) * L, o + (b * T * H + h) * dv, Gbuf);
      free(Gbuf);
    }
  }
}

/* Form Q evaluated at chosen query positions of one head.  q, k: (T, dk),
 * v: (T, dv), a: (T), lam: (n, L) holding lambda of the chosen queries,
 * ts: (n) query positions, o: (n, dv).  Queries run in parallel. */
void oracle_form_q_points(long T, long dk, long dv, long L, const double* q,
                          const double* k, const double* v, const double* a,
                          const double* lam, const long* ts, long n, double* o) {
  double* G = (double*)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
  double acc = 0.0;
  for (long t = 0; t < T; t++) {
    acc += log(a[t]);
    G[t] = acc;
  }
#pragma omp parallel for schedule(dynamic)
  for (long p = 0; p < n; p++) {
    long t = ts[p];
    double* ot = o + p * dv;
    for (long j = 0; j < dv; j++) ot[j] = 0.0;
    const double* qt = q + t * dk;
    for (long s = 0; s <= t; s++) {
      const double* ks = k + s * dk;
      double dot = 0.0;
      for (long i = 0; i < dk; i++) dot += qt[i] * ks[i];
      double w = lam[p * L + oracle_level(t, s)] * exp(G[t] - G[s]) * dot;
      const double* vsv = v + s * dv;
      for (long j = 0; j < dv; j++) ot[j] += w * vsv[j];
    }
  }
  free(G);
}

/* ---------------------------------------------------------------------------
 * Form R: the recurrent form with one d_k x d_v memory per Fenwick bucket,
 * each weighted by its lambda (page 1, section 特殊结构：树划分: per-bucket
 * memories combined with data-dependent scalars; decoding in O(log T) time
 * and memory).  Token by token, with eager decay:
 *   1. every live bucket state is multiplied by a_t (Mamba-2 transition);
 *   2. o_t = lambda_t^0 (q_t . k_t) v_t + sum_l lambda_t^l q_tᵀ S^l;
 *   3. the token and the buckets of levels 1..m, m = number of trailing ones
 *      of t, merge into the level m+1 bucket of position t+1.
 * Bucket level l >= 1 is live at position t when bit l-1 of t is set.
 *
 * One head: q, k (T, dk) with row stride qs; v, o (T, dv) with row stride
 * vs; a with stride as; lam with row stride ls.  Optional capture: for each
 * position cap_pos[c] (ascending, 0..T) the live states at that position,
 * before the decay by a at that position, go to states[c] (Ls, dk, dv);
 * levels that are not live are written as zero.
 * ------------------------------------------------------------------------- */
static void form_r_head(long T, long dk, long dv, long L, long qs, long vs, long as, long ls,
                        const double* q, const double* k, const double* v, const double* a,
                        const double* lam, double* o, long Ls, long ncap, const long* cap_pos,
                        double* states, double* S) {
  long sz = dk * dv;
  memset(S, 0, sizeof(double) * (size_t)(Ls * sz));
  long c = 0;
  for (long t = 0; t <= T; t++) {
    while (c < ncap && cap_pos[c] == t) {
      double* dst = states + c * Ls * sz;
      for (long l = 0; l < Ls; l++) {
        int live = l >= 1 && ((t >> (l - 1)) & 1L);
        for (long e = 0; e < sz; e++) dst[l * sz + e] = live ? S[l * sz + e] : 0.0;
      }
      c++;
    }
    if (t == T) break;
    const double* qt = q + t * qs;
    const double* kt = k + t * qs;
    const double* vt = v + t * vs;
    double at = a[t * as];
    double* ot = o + t * vs;
    /* 1. decay the live buckets */
    for (long l = 1; l < Ls; l++) {
      if ((t >> (l - 1)) & 1L) {
        double* Sl = S + l * sz;
        for (long e = 0; e < sz; e++) Sl[e] *= at;
      }
    }
    /* 2. output */
    double dot = 0.0;
    for (long i = 0; i < dk; i++) dot += qt[i] * kt[i];
    double w0 = lam[t * ls + 0] * dot;
    for (long j = 0; j < dv; j++) ot[j] = w0 * vt[j];
    for (long l = 1; l < Ls; l++) {
      if (!((t >> (l - 1)) & 1L)) continue;
      double wl = lam[t * ls + l];
      const double* Sl = S + l * sz;
      for (long i = 0; i < dk; i++) {
        double qi = wl * qt[i];
        for (long j = 0; j < dv; j++) ot[j] += qi * Sl[i * dv + j];
      }
    }
    /* 3. carry: m trailing ones of t -> level m+1 of t+1 */
    long m = 0;
    while ((t >> m) & 1L) m++;
    double* Sn = S + (m + 1) * sz;
    for (long i = 0; i < dk; i++)
      for (long j = 0; j < dv; j++) Sn[i * dv + j] = kt[i] * vt[j];
    for (long l = 1; l <= m; l++) {
      double* Sl = S + l * sz;
      for (long e = 0; e < sz; e++) {
        Sn[e] += Sl[e];
        Sl[e] = 0.0;
      }
    }
  }
  (void)L;
}

/* Batched Form R.  If states is non-null it receives the bucket states at
 * position T: (B, H, Ls, dk, dv), zero for levels that are not live.  Ls must
 * cover bit_length(T) + 1 levels for the export and bit_length(T) + 1 for the
 * merges, so the caller passes Ls >= bit_length(T) + 1. */
void oracle_form_r(long B, long T, long H, long hpg, long dk, long dv, long L,
                   const double* q, const double* k, const double* v, const double* a,
                   const double* lam, double* o, double* states, long Ls) {
  long G = H / hpg;
#pragma omp parallel for collapse(2) schedule(dynamic)
  for (long b = 0; b < B; b++) {
    for (long h = 0; h < H; h++) {
      double* S = (double*)malloc(sizeof(double) * (size_t)(Ls * dk * dv));
      long g = h / hpg;
      long cap = T;
      form_r_head(T, dk, dv, L, G * dk, H * dv, H, H * L,
                  q + (b * T * G + g) * dk, k + (b * T * G + g) * dk,
                  v + (b * T * H + h) * dv, a + b * T * H + h,
                  lam + (b * T * H + h) * L, o + (b * T * H + h) * dv, Ls,
                  states ? 1 : 0, &cap,
                  states ? states + (b * H + h) * Ls * dk * dv : NULL, S);
      free(S);
    }
  }
}

/* Form R on one head with contiguous inputs, capturing the bucket states at
 * the ascending positions cap_pos (each in 0..T). */
void oracle_form_r_head(long T, long dk, long dv, long L, const double* q, const double* k,
                        const double* v, const double* a, const double* lam, double* o,
                        long Ls, long ncap, const long* cap_pos, double* states) {
  double* S = (double*)malloc(sizeof(double) * (size_t)(Ls * dk * dv));
  form_r_head(T, dk, dv, L, dk, dv, 1, L, q, k, v, a, lam, o, Ls, ncap, cap_pos, states, S);
  free(S);
}

/* ---------------------------------------------------------------------------
 * Sequence segments.  Page 1 (section 特殊结构：树划分) keeps one memory per
 * bucket of the Fenwick partition of the prefix; section 高效训练算法 forms the
 * memories of chunks and combines them level by level.  The same holds for
 * any split of the sequence into segments: the memory of a bucket is the
 * decayed sum of the memories of the pieces it is made of.
 * ------------------------------------------------------------------------- */

/* Form R for the tokens at positions T0 .. T0+T-1 of one head, starting from
 * the bucket memories at position T0 (the live levels of T0, each already
 * decayed to position T0-1, i.e. what form_r_head captures at T0).  The same
 * three steps per token as form_r_head, with the level tests on the absolute
 * position.  q, k (T, dk), v, o (T, dv), a (T), lam (T, L) hold the segment's
 * tokens only; init (Ls, dk, dv); final_states (Ls, dk, dv), if non-null,
 * receives the live memories at T0+T (zero elsewhere).  Ls must be at least
 * bit_length(T0 + T) + 1. */
void oracle_form_r_from(long T0, long T, long dk, long dv, long L, const double* q,
                        const double* k, const double* v, const double* a, const double* lam,
                        long Ls, const double* init, double* o, double* final_states) {
  long sz = dk * dv;
  double* S = (double*)malloc(sizeof(double) * (size_t)(Ls * sz));
  for (long l = 0; l < Ls; l++) {
    int live = l >= 1 && ((T0 >> (l - 1)) & 1L);
    for (long e = 0; e < sz; e++) S[l * sz + e] = live ? init[l * sz + e] : 0.0;
  }
  for (long i = 0; i < T; i++) {
    long t = T0 + i; /* absolute position */
    const double* qt = q + i * dk;
    const double* kt = k + i * dk;
    const double* vt = v + i * dv;
    double* ot = o + i * dv;
    for (long l = 1; l < Ls; l++) /* 1. decay the live buckets */
      if ((t >> (l - 1)) & 1L)
        for (long e = 0; e < sz; e++) S[l * sz + e] *= a[i];
    double dot = 0.0; /* 2. output */
    for (long c = 0; c < dk; c++) dot += qt[c] * kt[c];
    for (long j = 0; j < dv; j++) ot[j] = lam[i * L] * dot * vt[j];
    for (long l = 1; l < Ls; l++) {
      if (!((t >> (l - 1)) & 1L)) continue;
      for (long c = 0; c < dk; c++) {
        double qc = lam[i * L + l] * qt[c];
        for (long j = 0; j < dv; j++) ot[j] += qc * S[l * sz + c * dv + j];
      }
    }
    long m = 0; /* 3. carry into level m+1 of t+1 */
    while ((t >> m) & 1L) m++;
    double* Sn = S + (m + 1) * sz;
    for (long c = 0; c < dk; c++)
      for (long j = 0; j < dv; j++) Sn[c * dv + j] = kt[c] * vt[j];
    for (long l = 1; l <= m; l++)
      for (long e = 0; e < sz; e++) {
        Sn[e] += S[l * sz + e];
        S[l * sz + e] = 0.0;
      }
  }
  if (final_states) {
    long E = T0 + T;
    for (long l = 0; l < Ls; l++) {
      int live = l >= 1 && ((E >> (l - 1)) & 1L);
      for (long e = 0; e < sz; e++) final_states[l * sz + e] = live ? S[l * sz + e] : 0.0;
    }
  }
  free(S);
}

/* The memory of a whole segment of T tokens of one head, by the definition:
 * total = sum over s < T of (a_{s+1} * ... * a_{T-1}) k_s v_sᵀ, the product
 * formed by an explicit loop, and logdecay = sum over r < T of log a_r (the
 * decay the segment applies to everything before it).  k (T, dk), v (T, dv),
 * a (T); total (dk, dv). */
void oracle_segment_total(long T, long dk, long dv, const double* k, const double* v,
                          const double* a, double* total, double* logdecay) {
  memset(total, 0, sizeof(double) * (size_t)(dk * dv));
  for (long s = 0; s < T; s++) {
    double w = 1.0;
    for (long r = s + 1; r < T; r++) w *= a[r];
    for (long c = 0; c < dk; c++)
      for (long j = 0; j < dv; j++) total[c * dv + j] += w * k[s * dk + c] * v[s * dv + j];
  }
  double g = 0.0;
  for (long r = 0; r < T; r++) g += log(a[r]);
  *logdecay = g;
}

/* Bucket memories at position T0 = r * seg_len from the memories of the r
 * segments before it (seg_len a power of two, so every bucket of the prefix
 * [0, T0) is made of whole segments).  The buckets come from the
 * binary-indexed-tree decomposition of the prefix (oracle_prefix_buckets); a
 * bucket of n positions has level log2(n) + 1, and its memory is
 *   sum over its segments sigma of exp(sum of logdecay over the segments
 *   after sigma and before T0) * seg_states[sigma].
 * seg_states (r, dk, dv), seg_logdecay (r); states (Ls, dk, dv), zero for the
 * levels that are not live at T0. */
void oracle_prefix_from_segments(long r, long seg_len, long dk, long dv, const double* seg_states,
                                 const double* seg_logdecay, long Ls, double* states) {
  long sz = dk * dv;
  memset(states, 0, sizeof(double) * (size_t)(Ls * sz));
  long lo[64], len[64];
  int nb = oracle_prefix_buckets(r * seg_len, lo, len, 64);
  for (int b = 0; b < nb; b++) {
    long lvl = ilog2_exact(len[b]) + 1;
    double* dst = states + lvl * sz;
    for (long sg = lo[b] / seg_len; sg < (lo[b] + len[b]) / seg_len; sg++) {
      double g = 0.0;
      for (long later = sg + 1; later < r; later++) g += seg_logdecay[later];
      double w = exp(g);
      for (long e = 0; e < sz; e++) dst[e] += w * seg_states[sg * sz + e];
    }
  }
}

/* ---------------------------------------------------------------------------
 * Brute force for small T: the dense T x T masks built without the level
 * formula, then O = (Q Kᵀ ⊙ M^S ⊙ M^H) V (page 1, section 结构矩阵).
 *   M^S(t,s) = a_{s+1} * ... * a_t by an explicit product loop;
 *   M^H(t,t) = lambda_t^0; for s < t, M^H(t,s) = lambda_t^{log2(n)+1} where
 *   n is the size of the binary-indexed-tree segment of the prefix [0, t)
 *   that holds s.
 * ------------------------------------------------------------------------- */
void oracle_brute(long B, long T, long H, long hpg, long dk, long dv, long L,
                  const double* q, const double* k, const double* v, const double* a,
                  const double* lam, double* o) {
  long G = H / hpg;
  double* MS = (double*)malloc(sizeof(double) * (size_t)(T * T + 1));
  double* MH = (double*)malloc(sizeof(double) * (size_t)(T * T + 1));
  double* A = (double*)malloc(sizeof(double) * (size_t)(T * T + 1));
  long* lo = (long*)malloc(sizeof(long) * 64);
  long* len = (long*)malloc(sizeof(long) * 64);
  for (long b = 0; b < B; b++) {
    for (long h = 0; h < H; h++) {
      long g = h / hpg;
      for (long t = 0; t < T; t++) {
        for (long s = 0; s < T; s++) {
          MS[t * T + s] = 0.0;
          MH[t * T + s] = 0.0;
          A[t * T + s] = 0.0;
        }
      }
      for (long t = 0; t < T; t++) {
        for (long s = 0; s <= t; s++) {
          double p = 1.0;
          for (long r = s + 1; r <= t; r++) p *= a[(b * T + r) * H + h];
          MS[t * T + s] = p;
          double dot = 0.0;
          for (long i = 0; i < dk; i++)
            dot += q[((b * T + t) * G + g) * dk + i] * k[((b * T + s) * G + g) * dk + i];
          A[t * T + s] = dot;
        }
        const double* lt = lam + ((b * T + t) * H + h) * L;
        MH[t * T + t] = lt[0];
        int nb = oracle_prefix_buckets(t, lo, len, 64);
        for (int c = 0; c < nb; c++) {
          int lvl = ilog2_exact(len[c]) + 1;
          for (long s = lo[c]; s < lo[c] + len[c]; s++) MH[t * T + s] = lt[lvl];
        }
      }
      for (long t = 0; t < T; t++) {
        for (long j = 0; j < dv; j++) {
          double acc = 0.0;
          for (long s = 0; s < T; s++)
            acc += A[t * T + s] * MS[t * T + s] * MH[t * T + s] * v[((b * T + s) * H + h) * dv + j];
          o[((b * T + t) * H + h) * dv + j] = acc;
        }
      }
    }
  }
  free(MS);
  free(MH);
  free(A);
  free(lo);
  free(len);
}

/* ---------------------------------------------------------------------------
 * Backward of Form Q for the scalar loss  sum_{t,j} dO[t,j] * o[t,j].
 * The pages give no backward; this is the chain rule applied to the forward
 * definition above (page 1, sections 特殊结构：树划分 and
 * 对Mamba-2和门控的对数线性推广), term by term.  With
 *   e_ts = exp(G_t - G_s),  w_ts = lambda_t^{l(t,s)} e_ts,
 *   A_ts = w_ts (q_t . k_s) (dO_t . v_s)          (s <= t):
 *   dq_t += w_ts (dO_t . v_s) k_s,   dk_s += w_ts (dO_t . v_s) q_t
 *     (q, k are per group: the heads of a group add up),
 *   dv_s += w_ts (q_t . k_s) dO_t,
 *   dlam_t^{l(t,s)} += e_ts (q_t . k_s) (dO_t . v_s),
 *   d(log a_r) = sum over t >= r and s < r of A_ts (log a_r enters e_ts exactly
 *     for s < r <= t), summed here for each t over r = 1..t with a running sum
 *     over s < r.  This gradient with respect to log a is returned (the one with
 *     respect to a is d(log a_r) / a_r).
 * Outputs are overwritten.  One group at a time (its heads share dq, dk).
 * ------------------------------------------------------------------------- */
void oracle_backward(long B, long T, long H, long hpg, long dk, long dv, long L,
                     const double* q, const double* k, const double* v, const double* a,
                     const double* lam, const double* dO, double* dq, double* dkk, double* dvv,
                     double* dloga_out, double* dlam) {
  long G = H / hpg;
  memset(dq, 0, sizeof(double) * (size_t)(B * T * G * dk));
  memset(dkk, 0, sizeof(double) * (size_t)(B * T * G * dk));
  memset(dvv, 0, sizeof(double) * (size_t)(B * T * H * dv));
  memset(dloga_out, 0, sizeof(double) * (size_t)(B * T * H));
  memset(dlam, 0, sizeof(double) * (size_t)(B * T * H * L));
#pragma omp parallel for collapse(2) schedule(dynamic)
  for (long b = 0; b < B; b++) {
    for (long g = 0; g < G; g++) {
      double* Gs = (double*)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
      double* dloga = (double*)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
      for (long h = g * hpg; h < (g + 1) * hpg; h++) {
        double acc = 0.0;
        for (long t = 0; t < T; t++) {
          acc += log(a[(b * T + t) * H + h]);
          Gs[t] = acc;
          dloga[t] = 0.0;
        }
        for (long t = 0; t < T; t++) {
          const double* qt = q + ((b * T + t) * G + g) * dk;
          const double* dot_ = dO + ((b * T + t) * H + h) * dv;
          const double* lt = lam + ((b * T + t) * H + h) * L;
          double* dqt = dq + ((b * T + t) * G + g) * dk;
          double* dlt = dlam + ((b * T + t) * H + h) * L;
          double run = 0.0;  /* sum over s < r of A_ts, for r = s + 1 */
          for (long s = 0; s <= t; s++) {
            const double* ks = k + ((b * T + s) * G + g) * dk;
            const double* vs = v + ((b * T + s) * H + h) * dv;
            double qk = 0.0, dov = 0.0;
            for (long i = 0; i < dk; i++) qk += qt[i] * ks[i];
            for (long j = 0; j < dv; j++) dov += dot_[j] * vs[j];
            int l = oracle_level(t, s);
            double e = exp(Gs[t] - Gs[s]);
            double w = lt[l] * e;
            double* dks = dkk + ((b * T + s) * G + g) * dk;
            double* dvs = dvv + ((b * T + s) * H + h) * dv;
            for (long i = 0; i < dk; i++) {
              dqt[i] += w * dov * ks[i];
              dks[i] += w * dov * qt[i];
            }
            for (long j = 0; j < dv; j++) dvs[j] += w * qk * dot_[j];
            dlt[l] += e * qk * dov;
            /* A_ts counts for every r with s < r <= t */
            if (s + 1 <= t) {
              run += w * qk * dov;
              dloga[s + 1] += run;
            }
          }
        }
        for (long r = 0; r < T; r++) dloga_out[(b * T + r) * H + h] = dloga[r];
      }
      free(Gs);
      free(dloga);
    }
  }
}

/* ---------------------------------------------------------------------------
 * Gated DeltaNet's transformed values.  The write-up extends Gated DeltaNet to
 * log-linear form by keeping the model's own transition and combining its
 * attention mask with the hierarchical one (page 1, section
 * 对Mamba-2和门控的对数线性推广).  The transition is the gated delta rule
 *   S_t = a_t S_{t-1} (I - beta_t k_t k_tᵀ) + beta_t v_t k_tᵀ,
 * which is the same as S_t = a_t S_{t-1} + u_t k_tᵀ with
 *   u_t = beta_t (v_t - a_t S_{t-1} k_t),
 * so S_t = sum_{s<=t} M^S(t,s) u_s k_sᵀ and the output is the masked form
 * with values u (o_t = S_t q_t for lambda = 1; the log-linear model weights the
 * same terms by lambda_t^{l(t,s)}).  This function runs the recurrence token by
 * token with S in fp64 (dv x dk per head) and writes u: (B, T, H, dv).
 * k is per group as elsewhere; v, a, beta are per head.
 * ------------------------------------------------------------------------- */
void oracle_gdn_values(long B, long T, long H, long hpg, long dk, long dv, const double* k,
                       const double* v, const double* a, const double* beta, double* u) {
  long G = H / hpg;
#pragma omp parallel for collapse(2) schedule(dynamic)
  for (long b = 0; b < B; b++) {
    for (long h = 0; h < H; h++) {
      long g = h / hpg;
      double* S = (double*)calloc((size_t)(dv * dk), sizeof(double));
      double* Sk = (double*)malloc(sizeof(double) * (size_t)dv);
      for (long t = 0; t < T; t++) {
        const double* kt = k + ((b * T + t) * G + g) * dk;
        const double* vt = v + ((b * T + t) * H + h) * dv;
        double at = a[(b * T + t) * H + h], bt = beta[(b * T + t) * H + h];
        double* ut = u + ((b * T + t) * H + h) * dv;
        for (long j = 0; j < dv; j++) {
          double acc = 0.0;
          for (long i = 0; i < dk; i++) acc += S[j * dk + i] * kt[i];
          Sk[j] = acc;
        }
        for (long j = 0; j < dv; j++) ut[j] = bt * (vt[j] - at * Sk[j]);
        for (long j = 0; j < dv; j++)
          for (long i = 0; i < dk; i++) S[j * dk + i] = at * S[j * dk + i] + ut[j] * kt[i];
      }
      free(S);
      free(Sk);
    }
  }
}
