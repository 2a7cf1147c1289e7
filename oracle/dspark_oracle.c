/*
 * DSpark per-step hot path: CPU ORACLE.
 *
 * TEST INFRASTRUCTURE ONLY.  This is the plain, slow, obviously-correct CPU
 * statement of what the three hot-path operations compute.  Only the test
 * suite, the smoke check and the benchmark's CPU-baseline leg may load it; the
 * product path never does.  It shares no code, header, table or constant
 * generator with the CUDA library.  Floating point is fp64 unless a step is an
 * explicit rounding to the storage dtype.  Build with -ffp-contract=off so that
 * x86 and Arm hosts give the same results.
 *
 * Sources (page title; section / equation / algorithm):
 *   [DSP]  "DSpark: Confidence-Scheduled Speculative Decoding with
 *          Semi-Autoregressive Generation" (arXiv 2607.05147):
 *          S2.1 acceptance rule; S3.1 semi-autoregressive block distribution
 *          and Markov head B = W1 W2; S3.2.2 Algorithm 1 (hardware-aware prefix
 *          scheduler); Appendix A (non-anticipation counterexample).
 *   [ZTD]  "Speculative decoding, from zero to DSpark": S2 accept rule and
 *          residual norm(max(0, p_t - p_d)); S6 p_k = softmax(U_k + B_k);
 *          S8 objective Theta = tau * SPS(B) and a_k = prod c_i; Appendix A1.
 *   [PRX]  Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as
 *          1, 2, 3" (SC'11), S4 Philox: the Philox4x32 round function, its
 *          multipliers and Weyl key increments, 10 rounds.
 *
 * Parity pins (tests/test_oracle_*.py): every function below is pinned by at
 * least one check that does not restate its own formula (printed worked
 * examples, exact enumeration, closed forms, exhaustive search, published
 * known-answer vectors, statistical laws).  See the per-function notes.
 *
 * Random stream specification (the pages fix none; both implementations
 * reproduce it from this text):
 *   key     = (seed & 0xffffffff, seed >> 32)
 *   counter = (c0, c1 = position, c2 = request id, c3 = tag)
 *   tag     DRAFT = 0 (draft sampling, position k = 1..K_r),
 *           ACCEPT = 1 (accept uniform, position j = 1..ell_r, c0 = 0, word 0),
 *           RESID = 2 (residual at the rejecting position j, or bonus at
 *                      position ell_r + 1),
 *           DRAFT_PICK = 3, RESID_PICK = 4 (the in-block draw of the
 *                      two-level sampler below, same positions)
 *   index i of a stream uses word (i & 3) of the block with c0 = i >> 2
 *   gumbel uniform  u = ((w >> 9) + 0.5) * 2^-23  in (0, 1), exact in fp32
 *   accept uniform  u = (w >> 8) * 2^-24          in [0, 1), exact in fp32
 *   gumbel noise    g = -log(-log(u))
 *
 * Categorical sampling (the pages only say "sample"; this is the reading both
 * implementations follow).  Weights w_v >= 0 over v = 0..n-1 are cut into
 * 32-wide blocks g = v >> 5.  Block g with mass L_g = sum of its weights gets
 * the score log L_g + gumbel(word g of the tag's stream); the block with the
 * largest score wins (ties: smaller g), and inside it the element is the
 * first v whose running weight sum exceeds u' * L_g, u' the accept-style
 * uniform of word g of the PICK stream.  This draws v with probability
 * w_v / sum(w) exactly: the Gumbel-max over blocks picks block g with
 * probability L_g / sum(L) and the inverse-CDF step picks v within it with
 * probability w_v / L_g.  It needs one random word per 32 elements.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---- status codes (oracle's own numbering; tests map them by name) ---- */
enum {
  ORC_OK = 0,
  ORC_ERR_NULL = 1,
  ORC_ERR_DIMS = 2,
  ORC_ERR_DTYPE = 3,
  ORC_ERR_TEMPERATURE = 4,
  ORC_ERR_SPS_TOO_SHORT = 5,
  ORC_ERR_OFFSETS = 6,
  ORC_ERR_TOKEN_RANGE = 7,
  ORC_ERR_LENGTHS = 8,
  ORC_ERR_CONFIDENCE = 9
};

enum { ORC_F32 = 0, ORC_BF16 = 1 };
enum { TAG_DRAFT = 0, TAG_ACCEPT = 1, TAG_RESID = 2, TAG_DRAFT_PICK = 3, TAG_RESID_PICK = 4 };

#define ORC_MAX_K 16
#define ORC_MIN_POS_T 1e-3
#define ORC_SAMPLE_TIE 1e-4 /* sampling near-tie margin (score units) */
#define ORC_ACCEPT_TIE 1e-5 /* |u - min(1, p/q)| near-tie margin        */
#define ORC_PICK_TIE 1e-5   /* |u' - cumulative fraction| near-tie margin */
#define ORC_BLOCK 32        /* block width of the two-level sampler       */
#define ORC_RNN_FEAT_ERR 1e-5 /* bound on the fp32 error of one RNN feature component */

/* ---------------------------------------------------------------------- */
/* Philox4x32-10 [PRX S4].                                                 */
/* One round: the two multipliers act on counter words 0 and 2; the high    */
/* halves are xored with the odd words and the two key words; the low halves */
/* move to the odd positions.  The key is bumped by the Weyl constants       */
/* between rounds.  Pinned by the published known-answer vectors.           */
/* ---------------------------------------------------------------------- */
void dso_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4]) {
  const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
  const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
  uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
  uint32_t k0 = key_in[0], k1 = key_in[1];
  for (int round = 0; round < 10; ++round) {
    uint64_t p0 = (uint64_t)M0 * (uint64_t)c0;
    uint64_t p1 = (uint64_t)M1 * (uint64_t)c2;
    uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    uint32_t n0 = hi1 ^ c1 ^ k0;
    uint32_t n1 = lo1;
    uint32_t n2 = hi0 ^ c3 ^ k1;
    uint32_t n3 = lo0;
    c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    k0 += W0;
    k1 += W1;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* Word for vocabulary element v of the stream (seed, position, request, tag). */
uint32_t dso_stream_word(uint64_t seed, uint64_t v, uint32_t position, uint32_t request, uint32_t tag) {
  uint32_t ctr[4] = {(uint32_t)(v >> 2), position, request, tag};
  uint32_t key[2] = {(uint32_t)(seed & 0xffffffffu), (uint32_t)(seed >> 32)};
  uint32_t out[4];
  dso_philox4x32_10(ctr, key, out);
  return out[v & 3u];
}

double dso_uniform_open(uint32_t w) { return ((double)(w >> 9) + 0.5) * 0x1p-23; }
double dso_uniform_accept(uint32_t w) { return (double)(w >> 8) * 0x1p-24; }
double dso_gumbel(uint32_t w) { return -log(-log(dso_uniform_open(w))); }

/* ---------------------------------------------------------------------- */
/* bf16 <-> fp64.  bf16 is the top half of an IEEE binary32.               */
/* ---------------------------------------------------------------------- */
static double bf16_to_double(uint16_t h) {
  uint32_t bits = (uint32_t)h << 16;
  float f;
  memcpy(&f, &bits, 4);
  return (double)f;
}

/* Quantum (spacing) of bf16 values around finite non-zero x. */
static double bf16_quantum(double x) {
  int e;
  (void)frexp(x, &e);            /* |x| in [2^(e-1), 2^e) */
  if (e - 1 < -126) e = -125;    /* subnormal range: fixed spacing 2^-133 */
  return ldexp(1.0, e - 8);
}

/* Round x to the nearest bf16 value, ties to even; returns the value. */
static double round_bf16(double x) {
  if (x == 0.0 || !isfinite(x)) return x;
  double q = bf16_quantum(x);
  double r = nearbyint(x / q) * q;         /* default mode: to nearest, ties even */
  if (fabs(r) > 0x1.FEp127) r = copysign(INFINITY, x);
  return r;
}

static uint16_t double_to_bf16_bits(double x) {
  float f = (float)round_bf16(x);          /* exact: value is a bf16 value */
  uint32_t bits;
  memcpy(&bits, &f, 4);
  return (uint16_t)(bits >> 16);
}

/* Which bf16 values may an fp32 evaluation of the exact value x store?  The     */
/* evaluation lies within delta of x (delta: an absolute bound on its error, for    */
/* instance the fp32 summation bound of the bias), and never closer to a rounding   */
/* midpoint than 2^-14 of a bf16 step is treated as safe.  With d = max(delta,      */
/* 2^-14 q(x)), rounding is monotone, so every stored value lies in                 */
/* [round(x - d), round(x + d)]; those are returned in *lo / *hi.  Returns 0 when    */
/* the two are equal (the stored value is unambiguous), 1 when they are the two     */
/* neighbours of one midpoint, 2 when the error spans more than one rounding        */
/* interval (a sum that cancels to near zero).                                      */
static int bf16_ambiguity(double x, double delta, double *lo, double *hi) {
  *lo = *hi = round_bf16(x);
  if (!isfinite(x)) return 0;
  double d = (x == 0.0) ? delta : fmax(delta, bf16_quantum(x) * 0x1p-14);
  if (!(d > 0.0)) return 0;
  *lo = round_bf16(x - d);
  *hi = round_bf16(x + d);
  if (*lo == *hi) return 0;
  /* one step apart: the quantum of the lower one, or (across a power of two) of the upper */
  if (*hi - *lo <= fmax(bf16_quantum(*lo), bf16_quantum(*hi))) return 1;
  return 2;
}

/* Largest distance between the value x rounds to and any value an fp32 evaluation */
/* within delta may store (0 when unambiguous); the code in *code when given.       */
static double bf16_spread(double x, double delta, int *code) {
  double lo, hi;
  const int c = bf16_ambiguity(x, delta, &lo, &hi);
  if (code) *code = c;
  if (!c) return 0.0;
  const double r = round_bf16(x);
  return fmax(hi - r, r - lo);
}

static double load_elem(const void *p, int dtype, int64_t i) {
  if (dtype == ORC_F32) return (double)((const float *)p)[i];
  return bf16_to_double(((const uint16_t *)p)[i]);
}

static void store_elem(void *p, int dtype, int64_t i, double x) {
  if (dtype == ORC_F32) ((float *)p)[i] = (float)x;
  else ((uint16_t *)p)[i] = double_to_bf16_bits(x);
}

static int temperature_ok(float t) {
  if (!(t == t) || isinf(t) || t < 0.0f) return 0;
  return t == 0.0f || (double)t >= ORC_MIN_POS_T;
}

static void set_threads(int nthreads) {
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
}

/* ---------------------------------------------------------------------- */
/* Two-level categorical sampler (see the stream specification above).      */
/* lw[v]: log-weights (-INFINITY for zero weight).  le[v] (optional): log of */
/* an absolute uncertainty on w_v (how far an fp32 evaluation may be off);    */
/* -INFINITY or NULL for none.  Reports whether a rounding-sized change could */
/* move the decision: near_block (runner-up block score within               */
/* ORC_SAMPLE_TIE * max(1, |score|)), near_pick (u' within ORC_PICK_TIE of a   */
/* cumulative boundary of the winning block), near_err (the decision moves   */
/* within the uncertainty le).                                              */
/* Pins: Monte-Carlo law against w / sum(w) on ragged block counts, single-  */
/* block and single-element limits, scale invariance.                      */
/* ---------------------------------------------------------------------- */
typedef struct {
  int64_t pick, block;
  double score, margin;
  int near_block, near_pick, near_err;
} race_t;

static race_t block_race(const double *lw, const double *le, int64_t n, uint64_t seed, uint32_t pos,
                         uint32_t rid, uint32_t tag_block, uint32_t tag_pick) {
  race_t o = {-1, -1, -INFINITY, INFINITY, 0, 0, 0};
  const int64_t nb = (n + ORC_BLOCK - 1) / ORC_BLOCK;
  double *t = (double *)malloc(sizeof(double) * (size_t)nb);    /* block score                    */
  double *hi = (double *)malloc(sizeof(double) * (size_t)nb);   /* score with the mass raised by le */
  double *lo = (double *)malloc(sizeof(double) * (size_t)nb);   /* score with the mass lowered     */
  for (int64_t g = 0; g < nb; ++g) {
    const int64_t v0 = g * ORC_BLOCK, v1 = (v0 + ORC_BLOCK < n) ? v0 + ORC_BLOCK : n;
    double ref = -INFINITY;
    for (int64_t v = v0; v < v1; ++v) {
      if (lw[v] > ref) ref = lw[v];
      if (le && le[v] > ref) ref = le[v];
    }
    t[g] = hi[g] = lo[g] = -INFINITY;
    if (ref == -INFINITY) continue;
    double lam = 0.0, er = 0.0;
    for (int64_t v = v0; v < v1; ++v) {
      lam += exp(lw[v] - ref);
      if (le) er += exp(le[v] - ref);
    }
    const double noise = dso_gumbel(dso_stream_word(seed, (uint64_t)g, pos, rid, tag_block));
    if (lam > 0.0) t[g] = ref + log(lam) + noise;
    hi[g] = ref + log(lam + er) + noise;
    if (lam > er) lo[g] = ref + log(lam - er) + noise;
    if (t[g] > o.score) { o.score = t[g]; o.block = g; }
  }
  if (o.block >= 0) {
    const int64_t gs = o.block;
    const double tol = ORC_SAMPLE_TIE * fmax(1.0, fabs(o.score));
    double second = -INFINITY;
    for (int64_t g = 0; g < nb; ++g) {
      if (g == gs) continue;
      if (t[g] > second) second = t[g];
      if (hi[g] >= lo[gs] - tol) o.near_err = 1;
    }
    o.margin = o.score - second;
    o.near_block = o.margin <= tol;
    /* in-block inverse CDF */
    const int64_t v0 = gs * ORC_BLOCK, v1 = (v0 + ORC_BLOCK < n) ? v0 + ORC_BLOCK : n;
    double ref = -INFINITY;
    for (int64_t v = v0; v < v1; ++v) if (lw[v] > ref) ref = lw[v];
    double lam = 0.0, er = 0.0;
    for (int64_t v = v0; v < v1; ++v) {
      lam += exp(lw[v] - ref);
      if (le) er += exp(le[v] - ref);
    }
    const double u = dso_uniform_accept(dso_stream_word(seed, (uint64_t)gs, pos, rid, tag_pick));
    double P = 0.0, dmin = INFINITY;
    int64_t last = -1;
    for (int64_t v = v0; v < v1; ++v) {
      const double w = exp(lw[v] - ref) / lam;
      if (w > 0.0) last = v;
      P += w;
      if (o.pick < 0 && P > u) o.pick = v;
      if (fabs(P - u) < dmin) dmin = fabs(P - u);
    }
    if (o.pick < 0) o.pick = last;   /* only when u sits within rounding of 1 */
    o.near_pick = dmin < ORC_PICK_TIE;
    if (dmin < ORC_PICK_TIE + 2.0 * er / lam) o.near_err = 1;
  }
  o.near_err = o.near_err || o.near_block || o.near_pick;
  free(t);
  free(hi);
  free(lo);
  return o;
}

/* Exposed for the sampler's own pins: returns the pick and the diagnostics. */
int64_t dso_block_race(const double *lw, const double *le, int64_t n, uint64_t seed, uint32_t pos,
                       uint32_t rid, uint32_t tag_block, uint32_t tag_pick, int64_t *block, double *score,
                       double *margin, int32_t *near) {
  race_t o = block_race(lw, le, n, seed, pos, rid, tag_block, tag_pick);
  if (block) *block = o.block;
  if (score) *score = o.score;
  if (margin) *margin = o.margin;
  if (near) { near[0] = o.near_block; near[1] = o.near_pick; near[2] = o.near_err; }
  return o.pick;
}

/* ---------------------------------------------------------------------- */
/* Draft: Markov-head semi-autoregressive sampling.                        */
/* [DSP S3.1], [ZTD S6]:                                                   */
/*   p_k(v | x_0, x_<k) = softmax(U_k(v) + B(x_{k-1}, v)),                  */
/*   B(x_{k-1}, .) = W1[x_{k-1}] . W2   (W1: V x rank lookup, W2: rank x V),  */
/*   x_0 = the anchor (the previous round's bonus/correction token),        */
/*   sampled left to right, k = 1..K_r.                                     */
/* Readings (the pages fix none of these):                                  */
/*   - the biased logits are materialised in the storage dtype (rounded to  */
/*     nearest-even from the exact value) and the draft samples from those  */
/*     stored logits, so verification sees exactly the sampled distribution;*/
/*   - temperature T divides the biased logit; T = 0 means argmax;          */
/*   - sampling is the two-level sampler of the stream specification on the */
/*     weights exp(z / T), streams (seed, k, request, DRAFT / DRAFT_PICK);   */
/*   - T = 0: the largest logit, ties to the smallest vocabulary index.     */
/* Outputs per (request, position): token, log-sum-exp of z/T (the draft    */
/* distribution's normaliser; for T = 0 the largest logit), margin (block   */
/* scores for T > 0, top-2 logits for T = 0), near-tie flags: bit0 block or */
/* greedy margin within tolerance (greedy: fp32 storage only), bit1 a bf16   */
/* rounding ambiguity could change the token, bit2 a bf16 rounding           */
/* ambiguity moves the log-sum-exp by more than 1e-6 relative, bit3 the      */
/* in-block draw sits within 1e-5 of a cumulative boundary.                 */
/* Pins: exact joint law by enumeration vs Monte Carlo; zero bias equals    */
/* independent sampling; one-hot rank-1 transition; hand-computed logits;   */
/* normalisation of the log-sum-exp.                                        */
/* ---------------------------------------------------------------------- */
/* log sum_v exp(z_v / T), fp64 */
static double row_lse_scaled(const double *z, int64_t V, double T) {
  double m = -INFINITY;
  for (int64_t v = 0; v < V; ++v) if (z[v] / T > m) m = z[v] / T;
  double S = 0.0;
  for (int64_t v = 0; v < V; ++v) S += exp(z[v] / T - m);
  return m + log(S);
}

/* One draft position of request rid: z = U row + bias, rounded to the storage dtype     */
/* (stored when draft_logits is given), then the draw (T > 0) or the argmax (T = 0) with   */
/* its normaliser, margin and near-tie flags.  Shared by the Markov and the RNN heads.      */
/* err[v] (bf16 only): an absolute bound on the error of an fp32 evaluation of U + bias    */
/* at element v; an element whose stored value that error could change is ambiguous, and   */
/* spread_out (optional, [V]) receives, per element, the largest distance between the      */
/* stored value and any value such an evaluation may store (0: unambiguous).               */
static int64_t draft_position(const void *U, int dtype, int64_t ubase, const double *bias, const double *err,
                              int64_t V, double T, uint64_t seed, int64_t k, uint32_t rid, void *draft_logits,
                              double *z, double *lw, double *le, double *l_out, double *mg_out, uint8_t *f_out,
                              float *spread_out) {
  for (int64_t v = 0; v < V; ++v) {
    double exact = load_elem(U, dtype, ubase + v) + bias[v];
    z[v] = (dtype == ORC_F32) ? (double)(float)exact : round_bf16(exact);
  }
  if (draft_logits) for (int64_t v = 0; v < V; ++v) store_elem(draft_logits, dtype, ubase + v, z[v]);
  /* spread[v]: how far the stored value may move (0 = unambiguous); kept in le's slot  */
  /* until the weights are formed                                                      */
  double *spread = le;
  int amb_any = 0;
  for (int64_t v = 0; v < V; ++v) {
    spread[v] = 0.0;
    int code = 0;
    if (dtype == ORC_BF16) spread[v] = bf16_spread(load_elem(U, dtype, ubase + v) + bias[v], err[v], &code);
    if (spread_out) spread_out[v] = (float)spread[v];
    if (code) amb_any = 1;
  }
  int64_t best;
  double l, mg;
  uint8_t f = 0;
  if (T > 0.0) {
    l = row_lse_scaled(z, V, T);
    /* lse moves by at most sum_v p_v |dz_v| / T when stored values move by dz_v */
    double lse_shift = 0.0;
    for (int64_t v = 0; v < V; ++v)
      if (spread[v] > 0.0) lse_shift += exp(z[v] / T - l) * spread[v] / T;
    if (lse_shift > 1e-6 * fmax(1.0, fabs(l))) f |= 4;
    /* two-level sampler on the weights exp(z / T); an ambiguous element enters as the  */
    /* uncertainty exp(z / T) (exp(spread / T) - 1) of its weight                        */
    for (int64_t v = 0; v < V; ++v) {
      const double sp = spread[v];
      lw[v] = z[v] / T;
      le[v] = (sp > 0.0) ? lw[v] + log(expm1(sp / T)) : -INFINITY;
    }
    race_t rc = block_race(lw, amb_any ? le : NULL, V, seed, (uint32_t)k, rid, TAG_DRAFT, TAG_DRAFT_PICK);
    best = rc.pick;
    mg = rc.margin;
    if (rc.near_block) f |= 1;
    if (rc.near_pick) f |= 8;
    if (rc.near_err && !(f & 9)) f |= 2;
  } else {
    /* greedy: largest logit, smallest index on ties */
    int64_t second = -1;
    best = 0;
    for (int64_t v = 1; v < V; ++v) {
      if (z[v] > z[best]) { second = best; best = v; }
      else if (second < 0 || z[v] > z[second]) second = v;
    }
    mg = z[best] - z[second];
    l = z[best];
    if (dtype == ORC_F32 && mg < ORC_SAMPLE_TIE) f |= 1;
    if (dtype == ORC_BF16) {
      for (int64_t v = 0; v < V; ++v) {
        if (!(spread[v] > 0.0)) continue;
        double lo, hi;
        bf16_ambiguity(load_elem(U, dtype, ubase + v) + bias[v], err[v], &lo, &hi);
        if (v == best) { if (lo <= z[second] + ORC_SAMPLE_TIE) f |= 2; }
        else if (hi >= z[best] - ORC_SAMPLE_TIE) f |= 2;
      }
    }
  }
  *l_out = l;
  *mg_out = mg;
  *f_out = f;
  return best;
}

int dso_draft_markov_sample(const void *U, const void *E, const void *W, int dtype,
                            const int32_t *anchor, const int32_t *K_r, const float *temperature,
                            const int64_t *req_id, uint64_t seed,
                            int64_t B, int64_t K_max, int64_t V, int64_t rank,
                            int32_t *draft_tok, void *draft_logits, double *lse,
                            double *margin, uint8_t *flags, float *spread, int nthreads) {
  if (!U || !E || !W || !anchor || !K_r || !temperature || !draft_tok) return ORC_ERR_NULL;
  if (dtype != ORC_F32 && dtype != ORC_BF16) return ORC_ERR_DTYPE;
  if (B < 1 || K_max < 1 || K_max > ORC_MAX_K || V < 2 || rank < 1) return ORC_ERR_DIMS;
  for (int64_t b = 0; b < B; ++b) {
    if (K_r[b] < 1 || K_r[b] > K_max) return ORC_ERR_LENGTHS;
    if (anchor[b] < 0 || anchor[b] >= V) return ORC_ERR_TOKEN_RANGE;
    if (!temperature_ok(temperature[b])) return ORC_ERR_TEMPERATURE;
  }
  set_threads(nthreads);
  int64_t b;
#pragma omp parallel for schedule(dynamic, 1)
  for (b = 0; b < B; ++b) {
    double *bias = (double *)malloc(sizeof(double) * (size_t)V);
    double *z = (double *)malloc(sizeof(double) * (size_t)V);
    double *lw = (double *)malloc(sizeof(double) * (size_t)V);
    double *le = (double *)malloc(sizeof(double) * (size_t)V);
    double *err = (double *)malloc(sizeof(double) * (size_t)V);
    uint32_t rid = (uint32_t)(req_id ? req_id[b] : b);
    int32_t x_prev = anchor[b];
    double T = (double)temperature[b];
    for (int64_t k = 1; k <= K_max; ++k) {
      int64_t slot = b * K_max + (k - 1);
      if (k > K_r[b]) { draft_tok[slot] = -1; continue; }
      /* transition bias: one row of the lookup table times the projection; err first */
      /* collects sum_i |E_i W_iv|                                                     */
      for (int64_t v = 0; v < V; ++v) bias[v] = err[v] = 0.0;
      for (int64_t i = 0; i < rank; ++i) {
        double e = load_elem(E, dtype, (int64_t)x_prev * rank + i);
        for (int64_t v = 0; v < V; ++v) {
          const double t = e * load_elem(W, dtype, i * V + v);
          bias[v] += t;
          err[v] += fabs(t);
        }
      }
      const int64_t ubase = slot * V;
      /* fp32 evaluation error of U + bias: the summation bound rank * u * sum |terms| */
      /* (doubled, for an accumulator that may truncate) plus the final rounding, u = 2^-24 */
      for (int64_t v = 0; v < V; ++v)
        err[v] = 0x1p-23 * ((double)rank * err[v] + fabs(load_elem(U, dtype, ubase + v) + bias[v]));
      double l, mg;
      uint8_t f = 0;
      const int64_t best = draft_position(U, dtype, ubase, bias, err, V, T, seed, k, rid, draft_logits, z, lw, le,
                                          &l, &mg, &f, spread ? spread + ubase : NULL);
      draft_tok[slot] = (int32_t)best;
      if (lse) lse[slot] = l;
      if (margin) margin[slot] = mg;
      if (flags) flags[slot] = f;
      x_prev = (int32_t)best;
    }
    free(bias);
    free(z);
    free(lw);
    free(le);
    free(err);
  }
  return ORC_OK;
}

/* ---------------------------------------------------------------------- */
/* Draft with the RNN head [DSP S3.1, RNN head]: a recurrent state s_k of    */
/* size r carries the whole prefix within the block.  Per position, one      */
/* linear projection of z_k = [s_{k-1}; W1[x_{k-1}]; h_k] is split into gate, */
/* candidate and output components (W_g, W_c, W_o, jointly one projection),  */
/* s_0 = 0.  The backbone part W_{.,h} h_k + b has no sequential dependence   */
/* and is an input: cx [B, K_max, 3r]; the sequential part is Wc [3r, 2r]    */
/* (columns 0..r-1 act on s_{k-1}, r..2r-1 on W1[x_{k-1}]; rows 0..r-1 gate,  */
/* r..2r-1 candidate, 2r..3r-1 output).                                      */
/* Readings (the update equation is missing from the paper's page; the text  */
/* names its inputs, its three components and the zero initial state):       */
/*   g = sigmoid(a_g), c = tanh(a_c), o = sigmoid(a_o),                       */
/*   s_k = g * s_{k-1} + (1 - g) * c       (a gated convex update),           */
/*   f_k = o * s_k                          (the output component gates the   */
/*                                           state),                          */
/*   bias_k = f_k . W2                      (the head's feature takes the place*/
/*                                           of the Markov head's W1 row).    */
/* fp64 throughout; the biased logits are rounded and sampled exactly as for  */
/* the Markov head.  feat (optional) returns f_k [B, K_max, r].              */
/* Pins: a closed output gate gives independent drafting; saturated gates    */
/* with an identity candidate block give the Markov head on tanh(W1);        */
/* constant pre-activations give the closed form s_k = c (1 - g^k); the       */
/* feature at position k depends on tokens before k - 1 (memory).            */
/* ---------------------------------------------------------------------- */
static double sigmoid_d(double a) { return 1.0 / (1.0 + exp(-a)); }

int dso_draft_rnn_sample(const void *U, const void *E, const void *W, const void *Wc, int dtype, const float *cx,
                         const int32_t *anchor, const int32_t *K_r, const float *temperature,
                         const int64_t *req_id, uint64_t seed,
                         int64_t B, int64_t K_max, int64_t V, int64_t rank,
                         int32_t *draft_tok, void *draft_logits, double *lse,
                         double *margin, uint8_t *flags, double *feat, float *spread, int nthreads) {
  if (!U || !E || !W || !Wc || !cx || !anchor || !K_r || !temperature || !draft_tok) return ORC_ERR_NULL;
  if (dtype != ORC_F32 && dtype != ORC_BF16) return ORC_ERR_DTYPE;
  if (B < 1 || K_max < 1 || K_max > ORC_MAX_K || V < 2 || rank < 1) return ORC_ERR_DIMS;
  for (int64_t b = 0; b < B; ++b) {
    if (K_r[b] < 1 || K_r[b] > K_max) return ORC_ERR_LENGTHS;
    if (anchor[b] < 0 || anchor[b] >= V) return ORC_ERR_TOKEN_RANGE;
    if (!temperature_ok(temperature[b])) return ORC_ERR_TEMPERATURE;
  }
  set_threads(nthreads);
  int64_t b;
#pragma omp parallel for schedule(dynamic, 1)
  for (b = 0; b < B; ++b) {
    double *bias = (double *)malloc(sizeof(double) * (size_t)V);
    double *z = (double *)malloc(sizeof(double) * (size_t)V);
    double *lw = (double *)malloc(sizeof(double) * (size_t)V);
    double *le = (double *)malloc(sizeof(double) * (size_t)V);
    double *st = (double *)calloc((size_t)rank, sizeof(double));        /* s_0 = 0 */
    double *ft = (double *)malloc(sizeof(double) * (size_t)rank);
    double *pre = (double *)malloc(sizeof(double) * (size_t)(3 * rank));
    double *err = (double *)malloc(sizeof(double) * (size_t)V);
    double *wabs = (double *)calloc((size_t)V, sizeof(double));   /* sum_i |W_iv| */
    for (int64_t i = 0; i < rank; ++i)
      for (int64_t v = 0; v < V; ++v) wabs[v] += fabs(load_elem(W, dtype, i * V + v));
    uint32_t rid = (uint32_t)(req_id ? req_id[b] : b);
    int32_t x_prev = anchor[b];
    double T = (double)temperature[b];
    for (int64_t k = 1; k <= K_max; ++k) {
      int64_t slot = b * K_max + (k - 1);
      if (k > K_r[b]) { draft_tok[slot] = -1; continue; }
      /* the cell: pre-activations of gate, candidate and output */
      for (int64_t j = 0; j < 3 * rank; ++j) {
        double a = (double)cx[slot * 3 * rank + j];
        for (int64_t i = 0; i < rank; ++i) a += load_elem(Wc, dtype, j * 2 * rank + i) * st[i];
        for (int64_t i = 0; i < rank; ++i)
          a += load_elem(Wc, dtype, j * 2 * rank + rank + i) * load_elem(E, dtype, (int64_t)x_prev * rank + i);
        pre[j] = a;
      }
      for (int64_t i = 0; i < rank; ++i) {
        const double g = sigmoid_d(pre[i]), c = tanh(pre[rank + i]), o = sigmoid_d(pre[2 * rank + i]);
        st[i] = g * st[i] + (1.0 - g) * c;
        ft[i] = o * st[i];
        if (feat) feat[slot * rank + i] = ft[i];
      }
      /* transition bias: the head's feature times the projection */
      for (int64_t v = 0; v < V; ++v) bias[v] = err[v] = 0.0;
      for (int64_t i = 0; i < rank; ++i)
        for (int64_t v = 0; v < V; ++v) {
          const double t = ft[i] * load_elem(W, dtype, i * V + v);
          bias[v] += t;
          err[v] += fabs(t);
        }
      /* fp32 evaluation error: the summation and rounding bound of the Markov head plus */
      /* the feature's own fp32 error (sigmoid, tanh and the recurrence), taken as at     */
      /* most ORC_RNN_FEAT_ERR per component                                               */
      for (int64_t v = 0; v < V; ++v)
        err[v] = 0x1p-23 * ((double)rank * err[v] + fabs(load_elem(U, dtype, slot * V + v) + bias[v])) +
                 ORC_RNN_FEAT_ERR * wabs[v];
      double l, mg;
      uint8_t f = 0;
      const int64_t best = draft_position(U, dtype, slot * V, bias, err, V, T, seed, k, rid, draft_logits, z, lw, le,
                                          &l, &mg, &f, spread ? spread + slot * V : NULL);
      draft_tok[slot] = (int32_t)best;
      if (lse) lse[slot] = l;
      if (margin) margin[slot] = mg;
      if (flags) flags[slot] = f;
      x_prev = (int32_t)best;
    }
    free(bias);
    free(z);
    free(lw);
    free(le);
    free(st);
    free(ft);
    free(pre);
    free(err);
    free(wabs);
  }
  return ORC_OK;
}

/* ---------------------------------------------------------------------- */
/* Confidence head, Markov term [DSP S3.2.1], [ZTD S8]: the head is one     */
/* linear projection of [h_k ; W1[x_{k-1}]] followed by a sigmoid, so        */
/*   c_k = sigmoid(w_h . h_k + b + w_e . W1[x_{k-1}]),   x_0 = anchor.      */
/* The backbone term w_h . h_k + b has no sequential dependence and is an    */
/* input (conf_h [B, K_max]); the Markov term needs the token sampled at     */
/* position k-1.  Readings: the display equation is missing from the paper  */
/* page; the tutorial (S8) and the paper's text give its inputs (backbone    */
/* hidden state plus the Markov embedding of the previous token, one linear */
/* projection, sigmoid), and the embedding is the draft's own table W1 (the */
/* "Markov Embedding").  fp64 dot product and sigmoid, rounded once to fp32. */
/* Entries k > K_r are set to 0.                                             */
/* Pins: one-hot embedding rows select one weight; w_e = 0 gives            */
/* sigmoid(conf_h) at every token; sigmoid(0) = 1/2 and the reflection      */
/* c(-s) = 1 - c(s); c_k changes only with x_{k-1}.                          */
/* ---------------------------------------------------------------------- */
int dso_draft_confidence(const void *E, int dtype, int64_t V, int64_t rank, const int32_t *anchor,
                         const int32_t *draft_tok, const int32_t *K_r, const float *conf_h, const float *conf_w,
                         int64_t B, int64_t K_max, float *conf) {
  if (!E || !anchor || !draft_tok || !K_r || !conf_h || !conf_w || !conf) return ORC_ERR_NULL;
  if (dtype != ORC_F32 && dtype != ORC_BF16) return ORC_ERR_DTYPE;
  if (B < 1 || K_max < 1 || K_max > ORC_MAX_K || V < 2 || rank < 1) return ORC_ERR_DIMS;
  for (int64_t r = 0; r < B; ++r) {
    if (K_r[r] < 1 || K_r[r] > K_max) return ORC_ERR_LENGTHS;
    for (int64_t k = 1; k <= K_max; ++k) {
      if (k > K_r[r]) { conf[r * K_max + k - 1] = 0.0f; continue; }
      const int32_t prev = k == 1 ? anchor[r] : draft_tok[r * K_max + k - 2];
      if (prev < 0 || prev >= V) return ORC_ERR_TOKEN_RANGE;
      double s = (double)conf_h[r * K_max + k - 1];
      for (int64_t i = 0; i < rank; ++i) s += load_elem(E, dtype, prev * rank + i) * (double)conf_w[i];
      conf[r * K_max + k - 1] = (float)(1.0 / (1.0 + exp(-s)));
    }
  }
  return ORC_OK;
}

/* ---------------------------------------------------------------------- */
/* Schedule: confidence-scheduled verification lengths.                     */
/* [DSP S3.2.2 Algorithm 1], [ZTD S8]:                                      */
/*   a_{r,j} = prod_{i<=j} c_{r,i};  candidates {(r,j) : a_{r,j} > 0} sorted */
/*   by a descending; B <- R, tau <- R, Theta_best <- R * SPS(R); for each   */
/*   candidate in order: B <- B + 1, tau <- tau + a, Theta <- tau * SPS(B);   */
/*   admit if Theta > Theta_best, else stop.  ell_r = admitted count of r.   */
/* Readings: a is the sequential fp32 product; ties in a go to the smaller  */
/* position j, then the smaller request r (earlier positions must win ties  */
/* for the prefix property); tau is accumulated exactly in 2^-40 fixed point */
/* (each a rounded half-to-even to a multiple of 2^-40), Theta evaluated in  */
/* fp64 as ((double)R + T * 2^-40) * SPS[B]; the SPS table must cover every  */
/* B up to R + #candidates; confidences outside [0, 1] are rejected.        */
/* Pins: Appendix A worked numbers; the two-request worked example; exhaustive */
/* search over admissible length tuples; empty-system limit; marginal test.  */
/* ---------------------------------------------------------------------- */
typedef struct { float a; int32_t j; int32_t r; } cand_t;

static int cand_cmp(const void *pa, const void *pb) {
  const cand_t *x = (const cand_t *)pa, *y = (const cand_t *)pb;
  if (x->a > y->a) return -1;
  if (x->a < y->a) return 1;
  if (x->j != y->j) return x->j < y->j ? -1 : 1;
  if (x->r != y->r) return x->r < y->r ? -1 : 1;
  return 0;
}

int dso_schedule_survival(const float *conf, const int32_t *K_r, const double *sps, int64_t sps_len,
                          int64_t B, int64_t K_max,
                          int32_t *ell, int32_t *tgt_off, double *theta_best, int64_t *B_star,
                          double *tau_star, float *survival, int32_t *order, int64_t *n_cand,
                          int64_t *n_admitted, int64_t *n_theta_ties) {
  if (!conf || !K_r || !sps || !ell || !tgt_off) return ORC_ERR_NULL;
  if (B < 1 || K_max < 1 || K_max > ORC_MAX_K) return ORC_ERR_DIMS;
  for (int64_t r = 0; r < B; ++r)
    if (K_r[r] < 1 || K_r[r] > K_max) return ORC_ERR_LENGTHS;
  for (int64_t r = 0; r < B; ++r)
    for (int64_t j = 0; j < K_r[r]; ++j) {
      float c = conf[r * K_max + j];
      if (!(c >= 0.0f && c <= 1.0f)) return ORC_ERR_CONFIDENCE;
    }
  cand_t *cand = (cand_t *)malloc(sizeof(cand_t) * (size_t)(B * K_max));
  int64_t N = 0;
  for (int64_t r = 0; r < B; ++r) {
    float a = 1.0f;
    for (int64_t j = 1; j <= K_max; ++j) {
      if (j > K_r[r]) { if (survival) survival[r * K_max + j - 1] = 0.0f; continue; }
      a = a * conf[r * K_max + j - 1];
      if (survival) survival[r * K_max + j - 1] = a;
      if (a > 0.0f) { cand[N].a = a; cand[N].j = (int32_t)j; cand[N].r = (int32_t)r; ++N; }
    }
  }
  qsort(cand, (size_t)N, sizeof(cand_t), cand_cmp);
  const int64_t R = B;
  if (sps_len < R + N + 1) { free(cand); return ORC_ERR_SPS_TOO_SHORT; }
  uint64_t T = 0, T_keep = 0;
  double th_best = (double)R * sps[R];
  int64_t admitted = 0, ties = 0;
  for (int64_t i = 1; i <= N; ++i) {
    uint64_t t = (uint64_t)nearbyint((double)cand[i - 1].a * 0x1p40);
    T += t;
    double th = ((double)R + (double)T * 0x1p-40) * sps[R + i];
    if (th == th_best) ++ties;
    if (th > th_best) { th_best = th; admitted = i; T_keep = T; }
    else break;
  }
  for (int64_t r = 0; r < B; ++r) ell[r] = 0;
  for (int64_t i = 0; i < admitted; ++i) ell[cand[i].r] += 1;
  tgt_off[0] = 0;
  for (int64_t r = 0; r < B; ++r) tgt_off[r + 1] = tgt_off[r] + ell[r] + 1;
  if (theta_best) *theta_best = th_best;
  if (B_star) *B_star = R + admitted;
  if (tau_star) *tau_star = (double)R + (double)T_keep * 0x1p-40;
  if (order) for (int64_t i = 0; i < N; ++i) order[i] = (int32_t)((cand[i].j - 1) * B + cand[i].r);
  if (n_cand) *n_cand = N;
  if (n_admitted) *n_admitted = admitted;
  if (n_theta_ties) *n_theta_ties = ties;
  free(cand);
  return ORC_OK;
}

/* ---------------------------------------------------------------------- */
/* Schedule variants of the deployed scheduler and of the static baseline.  */
/*                                                                          */
/* Shared first steps (as in Algorithm 1): validation, survival products    */
/* a_{r,j} (sequential fp32), the candidate pool {(r,j) : a_{r,j} > 0} and   */
/* its ranking by a descending, ties to the smaller j, then the smaller r.  */
/* ---------------------------------------------------------------------- */
static int64_t ranked_candidates(const float *conf, const int32_t *K_r, int64_t B, int64_t K_max,
                                 float *survival, cand_t *cand) {
  int64_t N = 0;
  for (int64_t r = 0; r < B; ++r) {
    float a = 1.0f;
    for (int64_t j = 1; j <= K_max; ++j) {
      if (j > K_r[r]) { if (survival) survival[r * K_max + j - 1] = 0.0f; continue; }
      a = a * conf[r * K_max + j - 1];
      if (survival) survival[r * K_max + j - 1] = a;
      if (a > 0.0f) { cand[N].a = a; cand[N].j = (int32_t)j; cand[N].r = (int32_t)r; ++N; }
    }
  }
  qsort(cand, (size_t)N, sizeof(cand_t), cand_cmp);
  return N;
}

static int check_schedule_inputs(const float *conf, const int32_t *K_r, int64_t B, int64_t K_max) {
  if (B < 1 || K_max < 1 || K_max > ORC_MAX_K) return ORC_ERR_DIMS;
  for (int64_t r = 0; r < B; ++r)
    if (K_r[r] < 1 || K_r[r] > K_max) return ORC_ERR_LENGTHS;
  for (int64_t r = 0; r < B; ++r)
    for (int64_t j = 0; j < K_r[r]; ++j) {
      float c = conf[r * K_max + j];
      if (!(c >= 0.0f && c <= 1.0f)) return ORC_ERR_CONFIDENCE;
    }
  return ORC_OK;
}

static void lengths_from_prefix(const cand_t *cand, int64_t admitted, int64_t B, int32_t *ell, int32_t *tgt_off) {
  for (int64_t r = 0; r < B; ++r) ell[r] = 0;
  for (int64_t i = 0; i < admitted; ++i) ell[cand[i].r] += 1;
  if (tgt_off) {
    tgt_off[0] = 0;
    for (int64_t r = 0; r < B; ++r) tgt_off[r + 1] = tgt_off[r] + ell[r] + 1;
  }
}

/* Capacity of the asynchronous scheduler [DSP S5.2], [ZTD S9]: the early-   */
/* stopping break is removed and the search runs over the whole greedy       */
/* admission path, Theta_i = tau_i * SPS(R + i) for i = 0..N (tau and Theta   */
/* in the same arithmetic as Algorithm 1); the capacity is the i with the    */
/* largest Theta_i.  Fed confidences from two steps earlier it fixes how many */
/* draft tokens the next pass verifies.  Readings: the capacity counts draft- */
/* token slots (the verify batch is R + capacity); ties in Theta go to the    */
/* smaller i (the first maximum, fewer verified tokens for the same value).  */
/* ell gets the lengths of that admission (the retrospective schedule of     */
/* Appendix A when applied to the current confidences).                     */
/* Pins: exhaustive search (Theta at the capacity = the maximum over every   */
/* admissible length tuple); the Appendix A retrospective lengths; crossing */
/* an SPS cliff that stops Algorithm 1.                                      */
int dso_schedule_capacity(const float *conf, const int32_t *K_r, const double *sps, int64_t sps_len,
                          int64_t B, int64_t K_max, int64_t *capacity, double *theta_best,
                          int32_t *ell, int32_t *tgt_off, float *survival) {
  if (!conf || !K_r || !sps || !capacity) return ORC_ERR_NULL;
  int st = check_schedule_inputs(conf, K_r, B, K_max);
  if (st) return st;
  cand_t *cand = (cand_t *)malloc(sizeof(cand_t) * (size_t)(B * K_max));
  const int64_t N = ranked_candidates(conf, K_r, B, K_max, survival, cand);
  const int64_t R = B;
  if (sps_len < R + N + 1) { free(cand); return ORC_ERR_SPS_TOO_SHORT; }
  uint64_t T = 0;
  double th_best = (double)R * sps[R];
  int64_t best = 0;
  for (int64_t i = 1; i <= N; ++i) {
    T += (uint64_t)nearbyint((double)cand[i - 1].a * 0x1p40);
    double th = ((double)R + (double)T * 0x1p-40) * sps[R + i];
    if (th > th_best) { th_best = th; best = i; }
  }
  *capacity = best;
  if (theta_best) *theta_best = th_best;
  if (ell) lengths_from_prefix(cand, best, B, ell, tgt_off);
  free(cand);
  return ORC_OK;
}

/* Dynamic top-K admission of the asynchronous scheduler [DSP S5.2],         */
/* [ZTD S9]: the current step's candidates, ranked by their current survival */
/* (ties to the smaller position, then the smaller request, so that token k  */
/* cannot move its own rank), are admitted in order up to the capacity fixed */
/* two steps earlier: the first min(capacity, N).  ell_r counts the admitted */
/* candidates of r.  Pins: for every capacity the admitted set maximises tau */
/* over all admissible tuples of that size (exhaustive search, the fixed-B   */
/* argument of S3.2.2); exact enumeration of the output law with a Markov    */
/* confidence (non-anticipation: the law equals the target's, where the      */
/* retrospective search reproduces Appendix A's 0.85).                      */
int dso_schedule_topk(const float *conf, const int32_t *K_r, int64_t B, int64_t K_max, int64_t capacity,
                      int32_t *ell, int32_t *tgt_off, int64_t *n_admitted, float *survival, int32_t *order,
                      int64_t *n_cand) {
  if (!conf || !K_r || !ell) return ORC_ERR_NULL;
  int st = check_schedule_inputs(conf, K_r, B, K_max);
  if (st) return st;
  if (capacity < 0) return ORC_ERR_LENGTHS;
  cand_t *cand = (cand_t *)malloc(sizeof(cand_t) * (size_t)(B * K_max));
  const int64_t N = ranked_candidates(conf, K_r, B, K_max, survival, cand);
  const int64_t admitted = capacity < N ? capacity : N;
  lengths_from_prefix(cand, admitted, B, ell, tgt_off);
  if (n_admitted) *n_admitted = admitted;
  if (order) for (int64_t i = 0; i < N; ++i) order[i] = (int32_t)((cand[i].j - 1) * B + cand[i].r);
  if (n_cand) *n_cand = N;
  free(cand);
  return ORC_OK;
}

/* Static-threshold verification length [DSP S3.2.2 (the prior methods it    */
/* contrasts with), S4.3.3 (the threshold sweep of Fig. 5)]: a request       */
/* verifies the longest prefix whose every position passes the threshold.   */
/* mode 0: c_{r,i} >= theta for all i <= j; mode 1: a_{r,i} >= theta (the    */
/* survival products, a prefix by monotonicity).  Readings: the pages do not */
/* say whether the cut is on the raw confidence or on its product, so both   */
/* are offered; a position passes on equality; as in Algorithm 1's candidate */
/* pool a position with a = 0 is never verified.  Pins: theta <= 0 admits    */
/* exactly Algorithm 1's empty-system schedule; theta > 1 admits nothing;    */
/* hand-worked lengths; lengths fall monotonically as theta rises.           */
int dso_schedule_threshold(const float *conf, const int32_t *K_r, int64_t B, int64_t K_max, float theta, int mode,
                           int32_t *ell, int32_t *tgt_off, float *survival) {
  if (!conf || !K_r || !ell) return ORC_ERR_NULL;
  int st = check_schedule_inputs(conf, K_r, B, K_max);
  if (st) return st;
  if (theta != theta || (mode != 0 && mode != 1)) return ORC_ERR_CONFIDENCE;
  for (int64_t r = 0; r < B; ++r) {
    float a = 1.0f;
    int32_t len = 0, open = 1;
    for (int64_t j = 1; j <= K_max; ++j) {
      if (j > K_r[r]) { if (survival) survival[r * K_max + j - 1] = 0.0f; continue; }
      const float c = conf[r * K_max + j - 1];
      a = a * c;
      if (survival) survival[r * K_max + j - 1] = a;
      const float tested = mode == 0 ? c : a;
      if (open && a > 0.0f && tested >= theta) len = (int32_t)j;
      else open = 0;
    }
    ell[r] = len;
  }
  if (tgt_off) {
    tgt_off[0] = 0;
    for (int64_t r = 0; r < B; ++r) tgt_off[r + 1] = tgt_off[r] + ell[r] + 1;
  }
  return ORC_OK;
}

/* ---------------------------------------------------------------------- */
/* Verify: ragged rejection-sampling verification.                          */
/* [DSP S2.1], [ZTD S2, A1]:                                                */
/*   for j = 1..ell_r, left to right: accept x_j iff u < min(1, p_j(x_j) /   */
/*   q_j(x_j)); at the first rejection sample the correction from            */
/*   norm(max(0, p_j - q_j)); if every position is accepted, sample a bonus  */
/*   token from the next target row.                                        */
/* Layout: draft logits [B, K_max, V] (row j-1 is q_j); flattened target    */
/* logits with row tgt_off[r] + j - 1 for p_j and row tgt_off[r] + ell_r for */
/* the bonus; tgt_off[r+1] - tgt_off[r] = ell_r + 1.                         */
/* Readings: q and p both use the request's temperature; T = 0 means greedy */
/* (accept iff x_j is the argmax of p_j, correction/bonus = argmax of p);    */
/* the residual is drawn by the two-level sampler on the weights            */
/* max(0, p_v - q_v), streams (seed, j, request, RESID / RESID_PICK); if no    */
/* element has p_v > q_v in floating point the correction is drawn from p    */
/* instead (rounding guard); the bonus is the two-level sampler on exp(z/T)  */
/* of the next target row, streams (seed, ell+1, request, RESID / RESID_PICK).*/
/* draft_spread (optional, [B, K_max, V], the draft's spreads): a draft logit */
/* may be any value within its spread that an fp32 evaluation of the draft   */
/* could store; the accept tolerance and the residual weights' uncertainties */
/* widen by what those changes can do.                                      */
/* Flags per request: bit0 an accept decision with |u - min(1, p/q)| < 1e-5,  */
/* bit1 the correction/bonus draw is within rounding of another outcome     */
/* (block scores, in-block boundary, or the fp32 error of p - q), bit2 the   */
/* residual mass was below 1e-5 (rounding guard region).  flag_pos is the   */
/* first position whose decision is flagged (ell + 1 for the final sample),  */
/* 0 when unflagged.                                                         */
/* Pins: the two-token worked numbers (output law (0.7, 0.3), acceptance    */
/* 0.8, every rejection yields A, which rules out the 0.64 full-resample     */
/* variant); Monte-Carlo output law against the target rows on enumerated     */
/* tiny cases with Markov-biased drafts; acceptance = sum min(p, q).          */
/* ---------------------------------------------------------------------- */
static void row_scaled(const void *base, int dtype, int64_t row, int64_t V, double T, double *out) {
  for (int64_t v = 0; v < V; ++v) {
    double z = load_elem(base, dtype, row * V + v);
    out[v] = (T > 0.0) ? z / T : z;
  }
}

static double row_lse(const double *s, int64_t V) {
  double m = -INFINITY;
  for (int64_t v = 0; v < V; ++v) if (s[v] > m) m = s[v];
  double S = 0.0;
  for (int64_t v = 0; v < V; ++v) S += exp(s[v] - m);
  return m + log(S);
}

static int64_t row_argmax(const double *s, int64_t V, double *mg) {
  int64_t best = 0, second = -1;
  for (int64_t v = 1; v < V; ++v) {
    if (s[v] > s[best]) { second = best; best = v; }
    else if (second < 0 || s[v] > s[second]) second = v;
  }
  if (mg) *mg = (second >= 0) ? s[best] - s[second] : INFINITY;
  return best;
}

int dso_verify_ragged(const void *draft_logits, const void *tgt_logits, int dtype,
                      const int32_t *tgt_off, const int32_t *ell, const int32_t *draft_tok,
                      const float *temperature, const int64_t *req_id, uint64_t seed,
                      int64_t B, int64_t K_max, int64_t V,
                      const float *draft_spread,
                      int32_t *n_acc, int32_t *out_tok, uint8_t *flags, int32_t *flag_pos,
                      double *sample_margin, int nthreads) {
  if (!draft_logits || !tgt_logits || !tgt_off || !ell || !draft_tok || !temperature || !n_acc || !out_tok)
    return ORC_ERR_NULL;
  if (dtype != ORC_F32 && dtype != ORC_BF16) return ORC_ERR_DTYPE;
  if (B < 1 || K_max < 1 || K_max > ORC_MAX_K || V < 2) return ORC_ERR_DIMS;
  if (tgt_off[0] != 0) return ORC_ERR_OFFSETS;
  for (int64_t r = 0; r < B; ++r) {
    if (ell[r] < 0 || ell[r] > K_max) return ORC_ERR_LENGTHS;
    if (tgt_off[r + 1] - tgt_off[r] != ell[r] + 1) return ORC_ERR_OFFSETS;
    if (!temperature_ok(temperature[r])) return ORC_ERR_TEMPERATURE;
    for (int64_t j = 0; j < ell[r]; ++j)
      if (draft_tok[r * K_max + j] < 0 || draft_tok[r * K_max + j] >= V) return ORC_ERR_TOKEN_RANGE;
  }
  set_threads(nthreads);
  int64_t r;
#pragma omp parallel for schedule(dynamic, 1)
  for (r = 0; r < B; ++r) {
    double *st = (double *)malloc(sizeof(double) * (size_t)V);
    double *sd = (double *)malloc(sizeof(double) * (size_t)V);
    double *lw = (double *)malloc(sizeof(double) * (size_t)V);
    double *le = (double *)malloc(sizeof(double) * (size_t)V);
    uint32_t rid = (uint32_t)(req_id ? req_id[r] : r);
    const double T = (double)temperature[r];
    const int64_t l = ell[r];
    uint8_t f = 0;
    int32_t fpos = 0;
    int64_t n = 0;
    int rejected = 0;
    int32_t token = -1;
    double mg = INFINITY;
    for (int64_t j = 1; j <= l; ++j) {
      int32_t x = draft_tok[r * K_max + j - 1];
      row_scaled(tgt_logits, dtype, (int64_t)tgt_off[r] + j - 1, V, T, st);
      int accept;
      /* draft logits that another fp32 evaluation may store differently move log q_v  */
      /* by at most dz_v / T (dz: their spread); log q(x) moves by at most dlq          */
      const float *am = draft_spread ? draft_spread + (r * K_max + j - 1) * V : NULL;
      double dlse = 0.0, dlq = 0.0;
      if (T > 0.0) {
        row_scaled(draft_logits, dtype, r * K_max + j - 1, V, T, sd);
        double lp = st[x] - row_lse(st, V);
        double lq = sd[x] - row_lse(sd, V);
        if (am) {
          const double ld = row_lse(sd, V);
          for (int64_t v = 0; v < V; ++v)
            if (am[v] > 0.0f) dlse += exp(sd[v] - ld) * (double)am[v] / T;
          dlq = dlse + (double)am[x] / T;
        }
        double rho = exp(lp - lq);
        double thr = rho < 1.0 ? rho : 1.0;
        double u = dso_uniform_accept(dso_stream_word(seed, 0, (uint32_t)j, rid, TAG_ACCEPT));
        if (fabs(u - thr) < ORC_ACCEPT_TIE + thr * expm1(dlq) && !fpos) { f |= 1; fpos = (int32_t)j; }
        accept = u < thr;
      } else {
        double amg;
        int64_t a = row_argmax(st, V, &amg);
        if (dtype == ORC_F32 && amg < ORC_SAMPLE_TIE && !fpos) { f |= 1; fpos = (int32_t)j; }
        accept = (x == a);
      }
      if (!accept) {
        rejected = 1;
        if (T > 0.0) {
          /* residual weights max(0, p - q); each carries the uncertainty of an fp32 */
          /* evaluation of p - q (relative 4e-6 of p + q plus the exponent rounding)  */
          double lt = row_lse(st, V), ld = row_lse(sd, V);
          double mass = 0.0;
          int any = 0;
          for (int64_t v = 0; v < V; ++v) {
            double p = exp(st[v] - lt), q = exp(sd[v] - ld);
            double res = p - q;
            double err = 4e-6 * (p + q) + 6e-8 * (fabs(st[v] - lt) * p + fabs(sd[v] - ld) * q);
            if (am) {      /* q_v moves by at most a factor exp(spread_v / T + dlse) */
              err += q * expm1((double)am[v] / T + dlse);
            }
            lw[v] = res > 0.0 ? log(res) : -INFINITY;
            le[v] = err > 0.0 ? log(err) : -INFINITY;
            if (res > 0.0) { mass += res; any = 1; }
          }
          if (mass < 1e-5 && !fpos) { f |= 4; fpos = (int32_t)j; }
          race_t rc;
          if (any) {
            rc = block_race(lw, le, V, seed, (uint32_t)j, rid, TAG_RESID, TAG_RESID_PICK);
            if (rc.near_err && !fpos) { f |= 2; fpos = (int32_t)j; }
          } else {
            rc = block_race(st, NULL, V, seed, (uint32_t)j, rid, TAG_RESID, TAG_RESID_PICK);
            if (rc.near_err && !fpos) { f |= 2; fpos = (int32_t)j; }
          }
          token = (int32_t)rc.pick;
          mg = rc.margin;
        } else {
          token = (int32_t)row_argmax(st, V, &mg);
          if (dtype == ORC_F32 && mg < ORC_SAMPLE_TIE && !fpos) { f |= 2; fpos = (int32_t)j; }
        }
        break;
      }
      out_tok[r * (K_max + 1) + n] = x;
      ++n;
    }
    if (!rejected) {
      row_scaled(tgt_logits, dtype, (int64_t)tgt_off[r] + l, V, T, st);
      if (T > 0.0) {
        race_t rc = block_race(st, NULL, V, seed, (uint32_t)(l + 1), rid, TAG_RESID, TAG_RESID_PICK);
        token = (int32_t)rc.pick;
        mg = rc.margin;
        if (rc.near_err && !fpos) { f |= 2; fpos = (int32_t)(l + 1); }
      } else {
        token = (int32_t)row_argmax(st, V, &mg);
        if (dtype == ORC_F32 && mg < ORC_SAMPLE_TIE && !fpos) { f |= 2; fpos = (int32_t)(l + 1); }
      }
    }
    out_tok[r * (K_max + 1) + n] = token;
    for (int64_t j = n + 1; j <= K_max; ++j) out_tok[r * (K_max + 1) + j] = -1;
    n_acc[r] = (int32_t)n;
    if (flags) flags[r] = f;
    if (flag_pos) flag_pos[r] = fpos;
    if (sample_margin) sample_margin[r] = mg;
    free(st);
    free(sd);
    free(lw);
    free(le);
  }
  return ORC_OK;
}

/* Log-sum-exp of rows of logits at per-row temperature (fp64); for T = 0 the */
/* row maximum.  Used to hand the CUDA verify a precomputed draft normaliser. */
int dso_row_lse(const void *rows, int dtype, int64_t n_rows, int64_t V, const float *row_temperature,
                double *out) {
  if (!rows || !row_temperature || !out) return ORC_ERR_NULL;
  if (dtype != ORC_F32 && dtype != ORC_BF16) return ORC_ERR_DTYPE;
  double *s = (double *)malloc(sizeof(double) * (size_t)V);
  for (int64_t i = 0; i < n_rows; ++i) {
    double T = (double)row_temperature[i];
    row_scaled(rows, dtype, i, V, T, s);
    if (T > 0.0) out[i] = row_lse(s, V);
    else { double m = s[0]; for (int64_t v = 1; v < V; ++v) if (s[v] > m) m = s[v]; out[i] = m; }
  }
  free(s);
  return ORC_OK;
}

/* bf16 rounding exposed for tests (value in, rounded value out). */
double dso_round_bf16(double x) { return round_bf16(x); }
