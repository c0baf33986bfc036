/*
 * blasst_oracle.c -- plain, slow CPU oracle for skip-softmax (BLASST) attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU-baseline
 * leg of the benchmark may load this library.  The product path (the CUDA
 * library) never calls it and shares no code, header or constant with it.
 *
 * The file is compiled twice: with REAL=float (the fp32 oracle the parity tests
 * compare against) and with REAL=double (used by the oracle's own self-checks).
 * Every function name carries the suffix _f32 or _f64 accordingly.
 *
 * What is computed, and where it is defined:
 *
 *  oracle_dense   softmax(scale * Q K^T) V written out row by row, with the
 *                 log-sum-exp lse = M + ln(sum exp(s - M)).  Definition of
 *                 attention: Hitchhiker's Guide Phase 08, Section 1, "Why
 *                 Standard Attention is IO-Bound"; lse as in its Triton listing's
 *                 "L = m + log(l)".
 *
 *  oracle_prefill_tiled / oracle_decode_tiled
 *                 the streaming pass over key tiles in ascending order, carrying
 *                 per query row the running max m, the running denominator l and
 *                 the running numerator O (Hitchhiker's Guide Phase 08, Section 1,
 *                 "FlashAttention: IO-Optimal Attention" recurrence and
 *                 "FlashAttention Tiling Strategy"; Skip-Softmax design doc,
 *                 "Algorithm"), with the BLASST test inserted between computing a
 *                 tile's scores and accumulating them: with m~ the row's max in
 *                 the tile and m the updated running max, the tile is skipped
 *                 when m~ - m < ln(lambda) for every query row of the tile
 *                 (Skip-Softmax design doc, "Algorithm", log form; BLASST talk
 *                 notes, "BLASST algorithm", Eq. 2).  A skipped tile contributes
 *                 nothing to l and O.
 *
 * Readings where the pages are silent (each is also listed in the design notes):
 *  - the test uses the running max AFTER the tile's own update (m = max(m_prev, m~));
 *  - only query rows that exist (r < Lq; the G heads in decode) vote; a row whose
 *    tile max is -inf votes "skip" when its running max is finite, and a row with
 *    running max -inf votes "compute" (the comparison with NaN/-inf is false);
 *  - causal masking is bottom-right aligned: key c is visible to row r iff
 *    c <= r + (Lkv - Lq); key tiles with no visible key for any row of the query
 *    tile are not visited (map value 2) and are not counted;
 *  - a sliding window of W >= 1 keys (BLASST talk notes, Q&A: the method applies
 *    to windowed attention; the notes give no definition) is the causal mask cut
 *    to the last W keys: with r' = r + (Lkv - Lq), key c is visible iff
 *    r' - W < c <= r'.  W <= 0 means no window.  In decode the query row sits at
 *    r' = Lkv - 1, and the splits cover the visited tiles only: with lo the first
 *    tile holding a visible key, split s covers [lo + floor(s*(nT-lo)/S),
 *    lo + floor((s+1)*(nT-lo)/S));
 *  - the tile's margin is max over voting rows of (m~ - m), +inf when any voting
 *    row has m~ = m = -inf; the tile is skipped iff margin < ln(lambda);
 *  - a row with no visible key at all gets O = 0 and lse = -inf;
 *  - decode split s of S covers key tiles [floor(s*nT/S), floor((s+1)*nT/S)); each
 *    split is an independent pass (m restarts at -inf) and the splits are merged by
 *    lse weighting: lse = ln(sum_s exp(lse_s)), O = sum_s exp(lse_s - lse) O_s.
 *
 *  oracle_mla_decode_tiled
 *                 decode for multi-head latent attention in its absorbed form (the
 *                 pages name MLA as the decode case where the skipped compute
 *                 pays: Skip-Softmax design doc, "Kernel", and BLASST talk notes,
 *                 "Abstract"; the pages give no formula for it).  Reading: every
 *                 cached token holds ONE row of dk values shared by all query heads;
 *                 the score of head h is scale * (q_h . row) over all dk values and
 *                 the value vector is the row's first dv values.  All query heads
 *                 read the same cached rows, so (as with the heads of a GQA group)
 *                 one skip decision covers every head x 128 keys.  A sequence b
 *                 holds seq_lens[b] keys (the whole cache when seq_lens is null);
 *                 its splits cover its own tiles, and a split with no tile gives
 *                 O = 0, lse = -inf.
 *
 * Plain loops, no blocking or fusion beyond the tiling the method itself states;
 * OpenMP only splits independent (batch, head, query-tile) units across cores.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifndef REAL
#define REAL float
#endif
#ifndef SUFFIX
#define SUFFIX _f32
#endif

#define CAT_(a, b) a##b
#define CAT(a, b) CAT_(a, b)
#define FN(name) CAT(name, SUFFIX)

typedef REAL real;

/* exp and log are evaluated in double and rounded to `real` */
#define R_EXP(x) ((real)exp((double)(x)))
#define R_LOG(x) ((real)log((double)(x)))

static const real NEG_INF = -(real)INFINITY;

/* key c visible to query row r? (bottom-right causal alignment; window W > 0
   keeps only the last W keys up to the row's own position) */
static int visible(int causal, long window, long r, long c, long Lq, long Lkv) {
    if (c >= Lkv) return 0;
    if (!causal) return 1;
    const long rr = r + (Lkv - Lq);
    if (c > rr) return 0;
    return window <= 0 || c > rr - window;
}

/* s = scale * (q . k) over d values, accumulated in `real` in index order */
static real score(const real* q, const real* k, int d, real scale) {
    real acc = 0;
    for (int i = 0; i < d; ++i) acc += q[i] * k[i];
    return scale * acc;
}

/* ------------------------------------------------------------------------- */
/* Dense attention: every row on its own, no tiling.                          */
/* ------------------------------------------------------------------------- */
int FN(oracle_dense)(const real* q, const real* k, const real* v, real* o, real* lse,
                     int B, int Hq, int Hkv, int Lq, int Lkv, int d, int causal, double scale_d,
                     int window) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Lq <= 0 || Lkv <= 0 || d <= 0 || Hq % Hkv) return -1;
    const int G = Hq / Hkv;
    const real scale = (real)scale_d;
    long n_rows = (long)B * Hq * Lq;
#pragma omp parallel
    {
        real* s = (real*)malloc(sizeof(real) * (size_t)Lkv);
#pragma omp for schedule(dynamic, 16)
        for (long row = 0; row < n_rows; ++row) {
            long r = row % Lq;
            long bh = row / Lq;
            long h = bh % Hq, b = bh / Hq;
            long hk = h / G;
            const real* qr = q + row * d;
            const real* kb = k + ((b * Hkv + hk) * (long)Lkv) * d;
            const real* vb = v + ((b * Hkv + hk) * (long)Lkv) * d;
            real* orow = o + row * d;
            real M = NEG_INF;
            for (long c = 0; c < Lkv; ++c) {
                if (visible(causal, window, r, c, Lq, Lkv)) {
                    s[c] = score(qr, kb + c * d, d, scale);
                    if (s[c] > M) M = s[c];
                } else {
                    s[c] = NEG_INF;
                }
            }
            for (int i = 0; i < d; ++i) orow[i] = 0;
            if (M == NEG_INF) { /* no visible key */
                lse[row] = NEG_INF;
                continue;
            }
            real sum = 0;
            for (long c = 0; c < Lkv; ++c) {
                if (s[c] == NEG_INF) continue;
                real p = R_EXP(s[c] - M);
                sum += p;
                for (int i = 0; i < d; ++i) orow[i] += p * vb[c * d + i];
            }
            for (int i = 0; i < d; ++i) orow[i] /= sum;
            lse[row] = M + R_LOG(sum);
        }
        free(s);
    }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* One streaming pass of the skip-softmax recurrence over a run of key tiles.  */
/*                                                                           */
/* rows:        n_rows query vectors (pointers), rows_r[i] = the row index used */
/*              for causal masking (ignored when causal == 0)                   */
/* kv:          K/V of the head, Lkv keys                                       */
/* tiles:       key tiles t0 .. t1-1 (tile size Bc), ascending                  */
/* forced:      if non-null, forced[t] (1 = skip) replaces the test             */
/* map/margin:  per-tile outputs indexed by tile number (non-null)              */
/* O, l, m:     per-row state, n_rows x d / n_rows / n_rows (output: O/l, lse)  */
/* ------------------------------------------------------------------------- */
/* kb/vb:       key c is kb + c*kstride (d values), its value vb + c*vstride   */
/*              (dv values; O rows hold dv values)                            */
typedef struct {
    int n_rows;
    const real* const* qrow;
    const long* rpos;
    const real* kb;
    const real* vb;
    long kstride, vstride;
    long Lq, Lkv;
    int d, dv, Bc, causal;
    long window;
    real scale;
    real lnlam;
} pass_args;

static long run_pass(const pass_args* a, int t0, int t1, const uint8_t* forced,
                     uint8_t* map, real* margin, real* O, real* l, real* m,
                     real* S /* n_rows*Bc scratch */, real* mt /* n_rows */, real* mnew /* n_rows */) {
    const int n = a->n_rows, d = a->dv, Bc = a->Bc;
    long skipped = 0;
    for (int i = 0; i < n; ++i) {
        m[i] = NEG_INF;
        l[i] = 0;
        for (int x = 0; x < d; ++x) O[(long)i * d + x] = 0;
    }
    for (int t = t0; t < t1; ++t) {
        long c0 = (long)t * Bc;
        /* visited iff some row sees some key of the tile */
        int vis = 0;
        for (int i = 0; i < n && !vis; ++i)
            for (long c = c0; c < c0 + Bc && !vis; ++c)
                if (visible(a->causal, a->window, a->rpos[i], c, a->Lq, a->Lkv)) vis = 1;
        if (!vis) {
            map[t] = 2;
            margin[t] = (real)NAN;
            continue;
        }
        /* S = scale * Q K_t^T, masked; row max m~ and updated running max */
        for (int i = 0; i < n; ++i) {
            real best = NEG_INF;
            for (int cc = 0; cc < Bc; ++cc) {
                long c = c0 + cc;
                real sv = NEG_INF;
                if (visible(a->causal, a->window, a->rpos[i], c, a->Lq, a->Lkv))
                    sv = score(a->qrow[i], a->kb + c * a->kstride, a->d, a->scale);
                S[(long)i * Bc + cc] = sv;
                if (sv > best) best = sv;
            }
            mt[i] = best;
            mnew[i] = m[i] > best ? m[i] : best;
        }
        /* BLASST test: every row must satisfy m~ - m < ln(lambda) */
        int skip = 1;
        real g = NEG_INF;
        for (int i = 0; i < n; ++i) {
            real diff = mt[i] - mnew[i]; /* NaN when both are -inf */
            int vote = diff < a->lnlam;
            if (!vote) skip = 0;
            real gi = (mt[i] == NEG_INF && mnew[i] == NEG_INF) ? (real)INFINITY : diff;
            if (gi > g) g = gi;
        }
        margin[t] = g;
        if (forced) skip = forced[t] == 1;
        map[t] = (uint8_t)(skip ? 1 : 0);
        if (skip) {
            ++skipped;
            /* no exp/rowsum and no P V; only the running max moves (it cannot
               move for lambda <= 1, but a forced skip may meet any tile) */
            for (int i = 0; i < n; ++i) {
                if (mnew[i] != m[i] && m[i] != NEG_INF) {
                    real alpha = R_EXP(m[i] - mnew[i]);
                    l[i] *= alpha;
                    for (int x = 0; x < d; ++x) O[(long)i * d + x] *= alpha;
                }
                m[i] = mnew[i];
            }
            continue;
        }
        /* online-softmax update of l and O */
        for (int i = 0; i < n; ++i) {
            if (mnew[i] == NEG_INF) continue; /* nothing visible yet in this row */
            real alpha = (m[i] == NEG_INF) ? 0 : R_EXP(m[i] - mnew[i]);
            real rowsum = 0;
            real* Oi = O + (long)i * d;
            for (int x = 0; x < d; ++x) Oi[x] *= alpha;
            for (int cc = 0; cc < Bc; ++cc) {
                real sv = S[(long)i * Bc + cc];
                if (sv == NEG_INF) continue;
                real p = R_EXP(sv - mnew[i]);
                rowsum += p;
                const real* vr = a->vb + (c0 + cc) * a->vstride;
                for (int x = 0; x < d; ++x) Oi[x] += p * vr[x];
            }
            l[i] = alpha * l[i] + rowsum;
            m[i] = mnew[i];
        }
    }
    /* finalise: O <- O / l, lse <- m + ln l (kept in m) */
    for (int i = 0; i < n; ++i) {
        real* Oi = O + (long)i * d;
        if (l[i] > 0) {
            for (int x = 0; x < d; ++x) Oi[x] /= l[i];
            m[i] = m[i] + R_LOG(l[i]);
        } else {
            for (int x = 0; x < d; ++x) Oi[x] = 0;
            m[i] = NEG_INF;
        }
    }
    return skipped;
}

static real ln_lambda(double lambda) {
    if (lambda <= 0) return NEG_INF;
    return (real)log(lambda);
}

/* ------------------------------------------------------------------------- */
/* Prefill: one pass per (b, h, query tile).                                  */
/*                                                                           */
/* units:   nullable list of n_units (b, h, qtile) triples; null = all units   */
/* forced:  nullable [B, Hq, nQ, nK] map (1 = skip) replacing the test         */
/* map:     nullable [B, Hq, nQ, nK] out (0 computed, 1 skipped, 2 not visited)*/
/* margin:  nullable [B, Hq, nQ, nK] out                                       */
/* o/lse:   [B,Hq,Lq,d] / [B,Hq,Lq]; only the rows of processed units written  */
/* returns the number of skipped tiles, or -1 on bad arguments                 */
/* ------------------------------------------------------------------------- */
long long FN(oracle_prefill_tiled)(const real* q, const real* k, const real* v, real* o, real* lse,
                                   int B, int Hq, int Hkv, int Lq, int Lkv, int d, int causal,
                                   double scale, double lambda, int Br, int Bc,
                                   const int32_t* units, int n_units, const uint8_t* forced,
                                   uint8_t* map, real* margin, int window) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Lq <= 0 || Lkv <= 0 || d <= 0 || Hq % Hkv || Br <= 0 ||
        Bc <= 0)
        return -1;
    const int G = Hq / Hkv;
    const int nQ = (Lq + Br - 1) / Br, nK = (Lkv + Bc - 1) / Bc;
    const long total_units = (long)B * Hq * nQ;
    const long nu = units ? n_units : total_units;
    long long skipped_total = 0;
#pragma omp parallel reduction(+ : skipped_total)
    {
        const real** qrow = (const real**)malloc(sizeof(real*) * Br);
        long* rpos = (long*)malloc(sizeof(long) * Br);
        real* O = (real*)malloc(sizeof(real) * (size_t)Br * d);
        real* l = (real*)malloc(sizeof(real) * Br);
        real* m = (real*)malloc(sizeof(real) * Br);
        real* S = (real*)malloc(sizeof(real) * (size_t)Br * Bc);
        real* mt = (real*)malloc(sizeof(real) * Br);
        real* mn = (real*)malloc(sizeof(real) * Br);
        uint8_t* lmap = (uint8_t*)malloc(nK);
        real* lmargin = (real*)malloc(sizeof(real) * nK);
#pragma omp for schedule(dynamic, 1)
        for (long u = 0; u < nu; ++u) {
            long b, h, qt;
            if (units) {
                b = units[3 * u];
                h = units[3 * u + 1];
                qt = units[3 * u + 2];
            } else {
                qt = u % nQ;
                h = (u / nQ) % Hq;
                b = u / ((long)nQ * Hq);
            }
            long r0 = qt * Br;
            int n = (int)((Lq - r0) < Br ? (Lq - r0) : Br);
            long hk = h / G;
            for (int i = 0; i < n; ++i) {
                qrow[i] = q + (((b * Hq + h) * (long)Lq) + r0 + i) * d;
                rpos[i] = r0 + i;
            }
            pass_args a;
            a.n_rows = n;
            a.qrow = qrow;
            a.rpos = rpos;
            a.kb = k + ((b * Hkv + hk) * (long)Lkv) * d;
            a.vb = v + ((b * Hkv + hk) * (long)Lkv) * d;
            a.kstride = a.vstride = d;
            a.Lq = Lq;
            a.Lkv = Lkv;
            a.d = a.dv = d;
            a.Bc = Bc;
            a.causal = causal;
            a.window = window;
            a.scale = (real)scale;
            a.lnlam = ln_lambda(lambda);
            long base = ((b * Hq + h) * (long)nQ + qt) * nK;
            skipped_total += run_pass(&a, 0, nK, forced ? forced + base : NULL, lmap, lmargin, O,
                                      l, m, S, mt, mn);
            for (int i = 0; i < n; ++i) {
                long row = ((b * Hq + h) * (long)Lq) + r0 + i;
                memcpy(o + row * d, O + (long)i * d, sizeof(real) * d);
                lse[row] = m[i];
            }
            if (map) memcpy(map + base, lmap, nK);
            if (margin) memcpy(margin + base, lmargin, sizeof(real) * nK);
        }
        free(qrow); free(rpos); free(O); free(l); free(m); free(S); free(mt); free(mn);
        free(lmap); free(lmargin);
    }
    return skipped_total;
}

/* ------------------------------------------------------------------------- */
/* Decode: one query token per sequence; the G = Hq/Hkv query heads that read  */
/* one KV head form the rows of the tile.  One pass per (b, hkv, split), then  */
/* the lse merge of the splits.                                               */
/*                                                                           */
/* q [B,Hq,d], k/v [B,Hkv,Lkv,d], o [B,Hq,d], lse [B,Hq]                       */
/* units:   nullable list of (b, hkv) pairs; all splits of a pair are run      */
/* forced/map/margin: nullable [B, Hkv, nK]                                    */
/* o_part/lse_part: nullable [S,B,Hq,d] / [S,B,Hq] per-split results           */
/* ------------------------------------------------------------------------- */
long long FN(oracle_decode_tiled)(const real* q, const real* k, const real* v, real* o, real* lse,
                                  int B, int Hq, int Hkv, int Lkv, int d, double scale,
                                  double lambda, int Bc, int num_splits, const int32_t* units,
                                  int n_units, const uint8_t* forced, uint8_t* map, real* margin,
                                  real* o_part, real* lse_part, int window) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Lkv <= 0 || d <= 0 || Hq % Hkv || Bc <= 0) return -1;
    const int G = Hq / Hkv;
    const int nK = (Lkv + Bc - 1) / Bc;
    const int S = num_splits;
    /* first tile holding a visible key: the splits cover tiles lo .. nK-1 */
    const long first_key = window > 0 && Lkv > window ? Lkv - window : 0;
    const int lo = (int)(first_key / Bc);
    if (S < 1 || S > nK - lo) return -1;
    const long nu = units ? n_units : (long)B * Hkv;
    long long skipped_total = 0;
#pragma omp parallel reduction(+ : skipped_total)
    {
        const real** qrow = (const real**)malloc(sizeof(real*) * G);
        long* rpos = (long*)malloc(sizeof(long) * G);
        real* O = (real*)malloc(sizeof(real) * (size_t)G * d);
        real* l = (real*)malloc(sizeof(real) * G);
        real* m = (real*)malloc(sizeof(real) * G);
        real* Sb = (real*)malloc(sizeof(real) * (size_t)G * Bc);
        real* mt = (real*)malloc(sizeof(real) * G);
        real* mn = (real*)malloc(sizeof(real) * G);
        uint8_t* lmap = (uint8_t*)malloc(nK);
        real* lmargin = (real*)malloc(sizeof(real) * nK);
        real* Op = (real*)malloc(sizeof(real) * (size_t)S * G * d);
        real* lp = (real*)malloc(sizeof(real) * (size_t)S * G);
#pragma omp for schedule(dynamic, 1)
        for (long u = 0; u < nu; ++u) {
            long b, hk;
            if (units) {
                b = units[2 * u];
                hk = units[2 * u + 1];
            } else {
                hk = u % Hkv;
                b = u / Hkv;
            }
            for (int i = 0; i < G; ++i) {
                qrow[i] = q + ((b * Hq) + hk * G + i) * (long)d;
                rpos[i] = 0;
            }
            pass_args a;
            a.n_rows = G;
            a.qrow = qrow;
            a.rpos = rpos;
            a.kb = k + ((b * Hkv + hk) * (long)Lkv) * d;
            a.vb = v + ((b * Hkv + hk) * (long)Lkv) * d;
            a.kstride = a.vstride = d;
            a.Lq = 1;
            a.Lkv = Lkv;
            a.d = a.dv = d;
            a.Bc = Bc;
            a.causal = window > 0;  /* the query row sits at Lkv - 1 */
            a.window = window;
            a.scale = (real)scale;
            a.lnlam = ln_lambda(lambda);
            long base = (b * Hkv + hk) * (long)nK;
            for (int t = 0; t < lo; ++t) { /* before the window: not visited */
                lmap[t] = 2;
                lmargin[t] = (real)NAN;
            }
            for (int s = 0; s < S; ++s) {
                int t0 = lo + (int)(((long)s * (nK - lo)) / S), t1 = lo + (int)(((long)(s + 1) * (nK - lo)) / S);
                skipped_total += run_pass(&a, t0, t1, forced ? forced + base : NULL, lmap,
                                          lmargin, O, l, m, Sb, mt, mn);
                memcpy(Op + (long)s * G * d, O, sizeof(real) * (size_t)G * d);
                memcpy(lp + (long)s * G, m, sizeof(real) * G);
            }
            /* merge the splits by their log-sum-exp */
            for (int i = 0; i < G; ++i) {
                long hq = hk * G + i;
                real M = NEG_INF;
                for (int s = 0; s < S; ++s)
                    if (lp[(long)s * G + i] > M) M = lp[(long)s * G + i];
                real* orow = o + (b * Hq + hq) * (long)d;
                for (int x = 0; x < d; ++x) orow[x] = 0;
                if (M == NEG_INF) {
                    lse[b * Hq + hq] = NEG_INF;
                } else {
                    real tot = 0;
                    for (int s = 0; s < S; ++s) tot += R_EXP(lp[(long)s * G + i] - M);
                    real L = M + R_LOG(tot);
                    for (int s = 0; s < S; ++s) {
                        real w = R_EXP(lp[(long)s * G + i] - L);
                        const real* os = Op + ((long)s * G + i) * d;
                        for (int x = 0; x < d; ++x) orow[x] += w * os[x];
                    }
                    lse[b * Hq + hq] = L;
                }
                if (o_part && lse_part) {
                    for (int s = 0; s < S; ++s) {
                        memcpy(o_part + (((long)s * B + b) * Hq + hq) * d, Op + ((long)s * G + i) * d,
                               sizeof(real) * d);
                        lse_part[((long)s * B + b) * Hq + hq] = lp[(long)s * G + i];
                    }
                }
            }
            if (map) memcpy(map + base, lmap, nK);
            if (margin) memcpy(margin + base, lmargin, sizeof(real) * nK);
        }
        free(qrow); free(rpos); free(O); free(l); free(m); free(Sb); free(mt); free(mn);
        free(lmap); free(lmargin); free(Op); free(lp);
    }
    return skipped_total;
}

/* ------------------------------------------------------------------------- */
/* MLA decode (absorbed form): one latent row per cached token, shared by all  */
/* Hq query heads; the Hq heads form the rows of every tile.                  */
/*                                                                           */
/* q [B,Hq,dk], kv [B,Lmax,dk] (value = first dv entries of a row)             */
/* seq_lens: nullable [B], keys of sequence b (clamped to [0, Lmax])           */
/* o [B,Hq,dv], lse [B,Hq]                                                     */
/* units:   nullable list of batch indices; all splits of a sequence are run   */
/* forced/map/margin: nullable [B, nK], nK = ceil(Lmax / Bc); tiles past a     */
/*          sequence's end are not visited (map 2, margin NaN)                 */
/* o_part/lse_part: nullable [S,B,Hq,dv] / [S,B,Hq] per-split results          */
/* returns the number of skipped tiles, or -1 on bad arguments                 */
/* ------------------------------------------------------------------------- */
long long FN(oracle_mla_decode_tiled)(const real* q, const real* kv, const int32_t* seq_lens, real* o,
                                      real* lse, int B, int Hq, int Lmax, int dk, int dv, double scale,
                                      double lambda, int Bc, int num_splits, const int32_t* units,
                                      int n_units, const uint8_t* forced, uint8_t* map, real* margin,
                                      real* o_part, real* lse_part) {
    if (B <= 0 || Hq <= 0 || Lmax <= 0 || dk <= 0 || dv <= 0 || dv > dk || Bc <= 0 || num_splits < 1)
        return -1;
    const int nK = (Lmax + Bc - 1) / Bc;
    const int S = num_splits;
    const long nu = units ? n_units : (long)B;
    long long skipped_total = 0;
#pragma omp parallel reduction(+ : skipped_total)
    {
        const real** qrow = (const real**)malloc(sizeof(real*) * Hq);
        long* rpos = (long*)malloc(sizeof(long) * Hq);
        real* O = (real*)malloc(sizeof(real) * (size_t)Hq * dv);
        real* l = (real*)malloc(sizeof(real) * Hq);
        real* m = (real*)malloc(sizeof(real) * Hq);
        real* Sb = (real*)malloc(sizeof(real) * (size_t)Hq * Bc);
        real* mt = (real*)malloc(sizeof(real) * Hq);
        real* mn = (real*)malloc(sizeof(real) * Hq);
        uint8_t* lmap = (uint8_t*)malloc(nK);
        real* lmargin = (real*)malloc(sizeof(real) * nK);
        real* Op = (real*)malloc(sizeof(real) * (size_t)S * Hq * dv);
        real* lp = (real*)malloc(sizeof(real) * (size_t)S * Hq);
#pragma omp for schedule(dynamic, 1)
        for (long u = 0; u < nu; ++u) {
            const long b = units ? units[u] : u;
            long Lb = Lmax;
            if (seq_lens) {
                Lb = seq_lens[b];
                if (Lb < 0) Lb = 0;
                if (Lb > Lmax) Lb = Lmax;
            }
            const int nT = (int)((Lb + Bc - 1) / Bc);
            for (int i = 0; i < Hq; ++i) {
                qrow[i] = q + (b * Hq + i) * (long)dk;
                rpos[i] = 0;
            }
            pass_args a;
            a.n_rows = Hq;
            a.qrow = qrow;
            a.rpos = rpos;
            a.kb = kv + b * (long)Lmax * dk;
            a.vb = a.kb; /* the value is the leading dv entries of the same row */
            a.kstride = a.vstride = dk;
            a.Lq = 1;
            a.Lkv = Lb;
            a.d = dk;
            a.dv = dv;
            a.Bc = Bc;
            a.causal = 0;
            a.window = 0;
            a.scale = (real)scale;
            a.lnlam = ln_lambda(lambda);
            const long base = b * (long)nK;
            for (int t = 0; t < nK; ++t) { /* past the sequence's end: not visited */
                lmap[t] = 2;
                lmargin[t] = (real)NAN;
            }
            for (int s = 0; s < S; ++s) {
                int t0 = (int)(((long)s * nT) / S), t1 = (int)(((long)(s + 1) * nT) / S);
                skipped_total += run_pass(&a, t0, t1, forced ? forced + base : NULL, lmap, lmargin, O, l,
                                          m, Sb, mt, mn);
                memcpy(Op + (long)s * Hq * dv, O, sizeof(real) * (size_t)Hq * dv);
                memcpy(lp + (long)s * Hq, m, sizeof(real) * Hq);
            }
            for (int i = 0; i < Hq; ++i) {
                real M = NEG_INF;
                for (int s = 0; s < S; ++s)
                    if (lp[(long)s * Hq + i] > M) M = lp[(long)s * Hq + i];
                real* orow = o + (b * Hq + i) * (long)dv;
                for (int x = 0; x < dv; ++x) orow[x] = 0;
                if (M == NEG_INF) {
                    lse[b * Hq + i] = NEG_INF;
                } else {
                    real tot = 0;
                    for (int s = 0; s < S; ++s) tot += R_EXP(lp[(long)s * Hq + i] - M);
                    real L = M + R_LOG(tot);
                    for (int s = 0; s < S; ++s) {
                        real w = R_EXP(lp[(long)s * Hq + i] - L);
                        const real* os = Op + ((long)s * Hq + i) * dv;
                        for (int x = 0; x < dv; ++x) orow[x] += w * os[x];
                    }
                    lse[b * Hq + i] = L;
                }
                if (o_part && lse_part) {
                    for (int s = 0; s < S; ++s) {
                        memcpy(o_part + (((long)s * B + b) * Hq + i) * dv, Op + ((long)s * Hq + i) * dv,
                               sizeof(real) * dv);
                        lse_part[((long)s * B + b) * Hq + i] = lp[(long)s * Hq + i];
                    }
                }
            }
            if (map) memcpy(map + base, lmap, nK);
            if (margin) memcpy(margin + base, lmargin, sizeof(real) * nK);
        }
        free(qrow); free(rpos); free(O); free(l); free(m); free(Sb); free(mt); free(mn);
        free(lmap); free(lmargin); free(Op); free(lp);
    }
    return skipped_total;
}
