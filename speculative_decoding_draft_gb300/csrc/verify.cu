// Ragged rejection-sampling verification ("DSpark", S2.1; "Speculative
// decoding, from zero to DSpark", S2 and Appendix A1).
//
// Three stages:
//  1. verify_plan_count (one CTA) and verify_plan_fill (a thread per request): validate every
//     request, reset its state and list the verified rows (r, j <= ell_r) position-major --
//     every request's position 1, then position 2, ... -- with the draft side of each accept
//     test precomputed (log q(x_j) when the draft normaliser is known).
//  2. verify_scan (persistent): each CTA takes whole listed rows in that order and streams
//     a row's vocabulary slices through a shared-memory ring (bulk copies issued by a
//     staging warp; the target slice, and the draft slice when no draft normaliser is
//     given), folding them into per-thread online-softmax statistics of z/T (the argmax for
//     T = 0).  At the row's last slice the warps reduce in a fixed order and the row is
//     decided there: accept x_j iff u_j < min(1, p(x_j)/q(x_j)) (x_j the target argmax for
//     T = 0); a rejection lowers the request's first-rejection word by atomicMin.  Before
//     staging a row the staging warp reads that word and skips rows past a known
//     rejection, so the rows read are the ones up to each request's deciding row, except
//     where a decision is not known yet.
//  3. verify_jobs (a thread per request): the outcome -- n_acc = (first rejection) - 1 or
//     ell_r, the accepted tokens, then the correction or bonus: the argmax of the rejecting row
//     for T = 0 and the bonus token are the scan's (the bonus row is listed at position
//     ell_r + 1, and the scan draws it -- the two-level draw over z / T, at small batches in
//     up to four parts over slice ranges that merge in a packed (score, index) maximum -- or
//     takes its argmax for T = 0, skipping it once a rejection is known) -- and the list of
//     T > 0 rejections.
//     verify_sample then draws each rejection's residual norm(max(0, p - q)), spread over
//     (rejection x vocabulary chunk) CTAs with the last chunk merging, or takes the
//     tensor-core recompute pass's draw.
#include "dspark_internal.cuh"

namespace dspark {
namespace {

constexpr int kRowThreads = 128;
constexpr int kBatch = 4;          // loads in flight per thread in the accept chain (fp32 / unaligned)
constexpr int kRowPk = 12;          // packed bf16 16-byte loads per thread and row item
constexpr int kRowSlice = kRowThreads * 8 * kRowPk;     // vocabulary slice of one row item
constexpr int kSampleThreads = 256;
constexpr int kSampleUnit = kSampleThreads * kBlockW;   // one 32-wide block per thread

struct Stats {
  float m, S;   // online softmax
  float best;   // greedy max
  int idx;      // greedy argmax
};

__device__ __forceinline__ void stats_init(Stats &s) {
  s.m = -INFINITY;
  s.S = 0.0f;
  s.best = -INFINITY;
  s.idx = -1;
}

__device__ __forceinline__ void stats_merge(Stats &a, const Stats &b) {
  if (b.best > a.best || (b.best == a.best && b.idx >= 0 && (a.idx < 0 || b.idx < a.idx))) {
    a.best = b.best;
    a.idx = b.idx;
  }
  if (b.m > a.m) {
    a.S = (a.m == -INFINITY ? 0.0f : a.S * fast_ex2((a.m - b.m) * kLog2e)) + b.S;
    a.m = b.m;
  } else if (b.m != -INFINITY) {
    a.S += b.S * fast_ex2((b.m - a.m) * kLog2e);
  }
}

// Online softmax of 8 scaled values.
__device__ __forceinline__ void stats_add8(Stats &st, const float (&s)[8]) {
  float cm = s[0];
#pragma unroll
  for (int q = 1; q < 8; ++q) cm = fmaxf(cm, s[q]);
  if (cm == -INFINITY) return;
  if (cm > st.m) {
    st.S = (st.m == -INFINITY) ? 0.0f : st.S * fast_ex2((st.m - cm) * kLog2e);
    st.m = cm;
  }
  const float mL = st.m * kLog2e;
#pragma unroll
  for (int q = 0; q < 8; ++q) st.S += fast_ex2(fmaf(s[q], kLog2e, -mL));
}

__device__ __forceinline__ void argmax_add8(Stats &st, const float (&s)[8], int v0) {
#pragma unroll
  for (int q = 0; q < 8; ++q)
    if (s[q] > st.best) { st.best = s[q]; st.idx = v0 + q; }
}

template <int DT>
__device__ __forceinline__ float load1(const void *base, int64_t i) {
  if (DT == DSPARK_F32) return __ldg((const float *)base + i);
  return bf16_bits_to_float(__ldg((const unsigned short *)base + i));
}

// Load 8 consecutive elements starting at element i (i multiple of 8 and the
// row 16-byte aligned when VEC; scalar with -INF padding otherwise).
template <int DT, bool VEC>
__device__ __forceinline__ void load8(const void *base, int64_t row_off, int v0, int V, float (&x)[8]) {
  if (VEC && v0 + 8 <= V) {
    if (DT == DSPARK_BF16) {
      const uint4 q = __ldcs((const uint4 *)((const unsigned short *)base + row_off + v0));
      const uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        x[2 * i] = __uint_as_float(u[i] << 16);
        x[2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
      }
    } else {
      const float4 *p = (const float4 *)((const float *)base + row_off + v0);
      const float4 a = __ldcs(p), b = __ldcs(p + 1);
      x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
      x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
    }
  } else {
#pragma unroll
    for (int q = 0; q < 8; ++q) x[q] = (v0 + q < V) ? load1<DT>(base, row_off + v0 + q) : -INFINITY;
  }
}

__device__ __forceinline__ float pick8(const float (&x)[8], int q) {
  float v = x[0];
#pragma unroll
  for (int i = 1; i < 8; ++i)
    if (i == q) v = x[i];
  return v;
}

__device__ __forceinline__ __nv_bfloat162 bf162_word(uint32_t w) { return *reinterpret_cast<const __nv_bfloat162 *>(&w); }

// Request checks shared by every CTA of the request (identical results everywhere).
// o0, o1: tgt_off[r], tgt_off[r + 1]; of: tgt_off[0].
__device__ __forceinline__ int request_error(int K, int r, int l, float T, int64_t o0, int64_t o1, int64_t of) {
  if (l < 0 || l > K) return DSPARK_ERR_LENGTHS;
  if (o1 - o0 != l + 1 || (r == 0 && of != 0)) return DSPARK_ERR_OFFSETS;
  if (!temperature_ok(T)) return DSPARK_ERR_TEMPERATURE;
  return 0;
}

// One row item of the statistics pass: vocabulary slice sl of drafted row rowi = r K + j - 1.
struct RowItem {
  int rowi, x, lo, hi;   // the slice is [lo, hi)
  int kind;              // 0 nothing to stream, 1 softmax statistics (T > 0), 2 argmax (T = 0)
  float invT;
  int64_t trow;          // first element of the target row
};

// The item's statistics from its packed loads: the thread's maximum over its 8 kRowPk
// values first (bf16 pairs, exact), then one pass of exponentials against it, two lanes per
// fp32 instruction; slots past the slice hold -inf.
__device__ __forceinline__ void row_consume(const RowItem &it, uint4 (&pk)[kRowPk], int tid, Stats &st,
                                            float *own_t) {
  if (it.hi - it.lo < kRowSlice) {        // the row's last slice: units past the row hold -inf
#pragma unroll
    for (int uu = 0; uu < kRowPk; ++uu)
      if (it.lo + (uu * kRowThreads + tid) * 8 + 8 > it.hi) pk[uu] = make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
  }
  // the 32 pair words of the thread, in element order
#define W_(e) word_of(pk[(e) >> 2], (e) & 3)
  __nv_bfloat162 m2[4] = {bf162_word(W_(0)), bf162_word(W_(1)), bf162_word(W_(2)), bf162_word(W_(3))};
#pragma unroll
  for (int e = 4; e < 4 * kRowPk; ++e) m2[e & 3] = __hmax2(m2[e & 3], bf162_word(W_(e)));
  m2[0] = __hmax2(__hmax2(m2[0], m2[1]), __hmax2(m2[2], m2[3]));
  const float zmax = fmaxf(__low2float(m2[0]), __high2float(m2[0]));
  if (zmax == -INFINITY) return;
  if (it.kind == 2) {                     // argmax: the first element equal to the maximum
    int idx = -1;
#pragma unroll
    for (int e = 4 * kRowPk - 1; e >= 0; --e) {
      const int v = it.lo + ((e >> 2) * kRowThreads + tid) * 8 + 2 * (e & 3);
      if (__uint_as_float(W_(e) & 0xffff0000u) == zmax) idx = v + 1;
      if (__uint_as_float(W_(e) << 16) == zmax) idx = v;
    }
    st.best = zmax;
    st.idx = idx;
    return;
  }
  const float m = zmax * it.invT;         // max(z) / T = max(z / T): scaling by 1/T > 0 is monotone
  const float a2 = it.invT * kLog2e, mL = m * kLog2e;
  const unsigned long long aa = f2_pack(a2, a2), nm = f2_pack(-mL, -mL);
  unsigned long long s0 = f2_pack(0.0f, 0.0f), s1 = s0;
#pragma unroll
  for (int e = 0; e < 4 * kRowPk; ++e) {
    const uint32_t we = W_(e);
    float y0, y1;    // z a2 - m log2(e): one rounding per exponent argument
    f2_unpack(f2_fma(f2_pack(__uint_as_float(we << 16), __uint_as_float(we & 0xffff0000u)), aa, nm), y0, y1);
    const unsigned long long ee = f2_pack(fast_ex2(y0), fast_ex2(y1));
    if (e & 1) s1 = f2_add(s1, ee);
    else s0 = f2_add(s0, ee);
  }
  // the scaled logit at the draft token, taken by the one thread whose loads hold it
  const int xo = it.x - it.lo;
  if (xo >= 0 && it.x < it.hi && ((xo >> 3) & (kRowThreads - 1)) == tid) {
    const int ex = ((xo >> 3) / kRowThreads) * 4 + ((xo & 7) >> 1);
    uint32_t wx = 0;
#pragma unroll
    for (int e = 0; e < 4 * kRowPk; ++e)
      if (e == ex) wx = W_(e);
    *own_t = __uint_as_float((it.x & 1) ? (wx & 0xffff0000u) : (wx << 16)) * it.invT;
  }
  float a0, a1, b0, b1;
  f2_unpack(s0, a0, a1);
  f2_unpack(s1, b0, b1);
  st.m = m;
  st.S = (a0 + a1) + (b0 + b1);
#undef W_
}

// Any dtype / alignment, and the draft row when no draft normaliser is given.
template <int DT, bool VEC>
__device__ __forceinline__ void row_generic(const VerifyArgs &a, const RowItem &it, bool stream_d, int tid, Stats &st,
                                            Stats &sd, float *own_t, float *own_d) {
  const int xv = it.x & ~7;
  const int64_t it_V = a.V;
  for (int base = it.lo + tid * 8; base < it.hi; base += kRowThreads * 8 * kBatch) {
    float x8[kBatch][8];
#pragma unroll
    for (int uu = 0; uu < kBatch; ++uu) load8<DT, VEC>(a.tgt, it.trow, base + uu * kRowThreads * 8, it.hi, x8[uu]);
    if (it.kind == 2) {
#pragma unroll
      for (int uu = 0; uu < kBatch; ++uu) argmax_add8(st, x8[uu], base + uu * kRowThreads * 8);
      continue;
    }
    float y8[kBatch][8];
    if (stream_d) {
#pragma unroll
      for (int uu = 0; uu < kBatch; ++uu) load8<DT, VEC>(a.D, (int64_t)it.rowi * it_V, base + uu * kRowThreads * 8, it.hi, y8[uu]);
    }
#pragma unroll
    for (int uu = 0; uu < kBatch; ++uu) {
      const int v0 = base + uu * kRowThreads * 8;
#pragma unroll
      for (int q = 0; q < 8; ++q) x8[uu][q] *= it.invT;
      if (v0 == xv) *own_t = pick8(x8[uu], it.x & 7);
      stats_add8(st, x8[uu]);
      if (stream_d) {
#pragma unroll
        for (int q = 0; q < 8; ++q) y8[uu][q] *= it.invT;
        if (v0 == xv) *own_d = pick8(y8[uu], it.x & 7);
        stats_add8(sd, y8[uu]);
      }
    }
  }
}

// Warp reduction of one item's statistics, valid in lane 0: the softmax pair (m, S) for
// T > 0 (a branch-free merge), the (maximum, smallest index) pair for T = 0.
__device__ __forceinline__ Stats warp_reduce_row(Stats s, int kind) {
  if (kind == 1) {
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) {
      const float m2 = __shfl_down_sync(0xffffffffu, s.m, d), S2 = __shfl_down_sync(0xffffffffu, s.S, d);
      const float M = fmaxf(s.m, m2);
      if (M != -INFINITY) {
        s.S = s.S * fast_ex2((s.m - M) * kLog2e) + S2 * fast_ex2((m2 - M) * kLog2e);
        s.m = M;
      }
    }
  } else {
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) {
      const float b2 = __shfl_down_sync(0xffffffffu, s.best, d);
      const int i2 = __shfl_down_sync(0xffffffffu, s.idx, d);
      if (i2 >= 0 && (b2 > s.best || (b2 == s.best && (s.idx < 0 || i2 < s.idx)))) {
        s.best = b2;
        s.idx = i2;
      }
    }
  }
  return s;
}

// --------------------------------------------------------------------------
// residual / bonus sampling
// --------------------------------------------------------------------------
template <int DT, bool VEC>
__device__ __forceinline__ void load32(const void *base, int64_t row_off, int v0, int V, float (&x)[kBlockW]) {
#pragma unroll
  for (int h = 0; h < kBlockW / 8; ++h) {
    float t[8];
    load8<DT, VEC>(base, row_off, v0 + 8 * h, V, t);
#pragma unroll
    for (int q = 0; q < 8; ++q) x[8 * h + q] = t[q];
  }
}

// 32 bf16 of a 16-byte aligned row from element v0: four 16-byte loads; 8-element groups
// at or past `hi` hold bf16 -inf (V and hi are multiples of 8 here).
__device__ __forceinline__ void issue_block(const void *base, int64_t row_off, int v0, int hi, uint4 (&u)[4]) {
#pragma unroll
  for (int q = 0; q < 4; ++q)
    u[q] = (v0 + 8 * q + 8 <= hi) ? __ldcs((const uint4 *)((const unsigned short *)base + row_off + v0 + 8 * q))
                                  : make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
}

// One block of residual weights in the two-level draw.
template <class PickWord>
__device__ __forceinline__ void brace_resid_block(BRace &r, float (&t)[kBlockW], const float (&d)[kBlockW],
                                                  float a, float lt2, float ld2, uint32_t wb, int v0, bool &any_pos,
                                                  PickWord pick_word) {
  float s[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
  for (int q = 0; q < kBlockW; ++q) {
    t[q] = resid_weight(t[q], d[q], a, lt2, ld2);   // t now holds the weights
    s[q & 3] += t[q];
  }
  const float L = (s[0] + s[1]) + (s[2] + s[3]);
  if (!(L > 0.0f)) return;
  any_pos = true;
  if (brace_enter(r, fast_lg2(L) * kLn2, wb)) r.idx = v0 + pick_in_block(t, uniform_accept(pick_word()) * L);
}

// The draw of one request over [lo, hi): residual (mode 1), bonus from the
// target row (mode 2, also the rounding guard of mode 1), greedy bonus (mode 3).
template <int DT, bool VEC>
__device__ void sample_range(const VerifyArgs &a, const VerifyJob &job, int r, int lo, int hi, int tid,
                             int nthreads, BRace &rc, bool &any_pos, bool from_p) {
  const int V = (int)a.V;
  const int64_t trow = job.trow * (int64_t)V;
  const int64_t drow = job.drow * (int64_t)V;
  const int mode = from_p ? 2 : job.mode;
  const PhiloxKey key = a.key;   // round keys in registers for the hot loop
  const float a2 = job.invT * kLog2e;
  const float lt2 = job.lse_t * kLog2e, ld2 = job.lse_q * kLog2e;
  if (DT == DSPARK_BF16 && VEC && mode == 1) {
    // residual on packed rows: the next block's target loads are in flight while this block
    // is drawn, and the draft row's loads go out before the block's noise is generated
    uint4 tc[4], dc[4], tn[4];
    int v0 = lo + tid * kBlockW;
    if (v0 < hi) issue_block(a.tgt, trow, v0, hi, tc);
    for (; v0 < hi; v0 += nthreads * kBlockW) {
      const int vn = v0 + nthreads * kBlockW;
      issue_block(a.D, drow, v0, hi, dc);
      if (vn < hi) issue_block(a.tgt, trow, vn, hi, tn);
      // round keys read from the parameter block: registers go to the loads in flight
      const uint32_t g = (uint32_t)v0 >> 5;
      const uint32_t wb = word_of(philox(a.key, g >> 2, (uint32_t)job.pos, (uint32_t)r, kTagResid), (int)(g & 3u));
      brace_resid_packed(rc, tc, dc, a2, lt2, ld2, wb, v0, any_pos, [&] {
        return word_of(philox(a.key, g >> 2, (uint32_t)job.pos, (uint32_t)r, kTagResidPick), (int)(g & 3u));
      });
#pragma unroll
      for (int q = 0; q < 4; ++q) tc[q] = tn[q];
    }
    return;
  }
  for (int v0 = lo + tid * kBlockW; v0 < hi; v0 += nthreads * kBlockW) {
    float t[kBlockW];
    load32<DT, VEC>(a.tgt, trow, v0, hi, t);
    if (mode == 3) {
      brace_argmax_block(rc, t, block_max(t), v0);
      continue;
    }
    const uint32_t g = (uint32_t)v0 >> 5;
    const uint32_t wb = word_of(philox(key, g >> 2, (uint32_t)job.pos, (uint32_t)r, kTagResid), (int)(g & 3u));
    auto pick_word = [&] {
      return word_of(philox(key, g >> 2, (uint32_t)job.pos, (uint32_t)r, kTagResidPick), (int)(g & 3u));
    };
    if (mode == 2) {
      brace_softmax_block(rc, t, block_max(t), a2, wb, v0, pick_word, NoLogit{});
      continue;
    }
    float d[kBlockW];
    load32<DT, VEC>(a.D, drow, v0, hi, d);
    brace_resid_block(rc, t, d, a2, lt2, ld2, wb, v0, any_pos, pick_word);
  }
}

// ---------------------------------------------------------------------------
// 1. plan: validation, per-request reset, the position-major row list
// ---------------------------------------------------------------------------
constexpr int kPlanThreads = 1024;

// Two kernels.  verify_plan_count (one CTA) resets each request's state, counts the rows of
// every position (ell_r + 1 rows of a request whose length is in range; the fill pass checks
// everything else and reports it) and sets each position's first slot.  When the rows and the
// T > 0 bonus draws fit one wave of scan CTAs with room to spare, each bonus draw is listed as
// up to four parts over ranges of its slices (the draw is a maximum over blocks, so the parts
// merge exactly), which keeps a bonus draw from being the one long row of a small batch.  verify_plan_fill (a
// thread per request and position) validates the request and lists its rows j = 1..ell_r and
// its bonus row j = ell_r + 1 at row_start[j] + (a slot taken per warp and position from
// row_fill[j]).
// The order inside a position is whatever the atomics give, and no result depends on it
// (each row is processed by one CTA on its own).  With an invalid request the status word is
// set and every later kernel returns at once.
__global__ void __launch_bounds__(kPlanThreads) verify_plan_count(const __grid_constant__ VerifyArgs a) {
  __shared__ int cnt[kMaxK + 3], cntb[kMaxK + 3];   // rows, T > 0 bonus draws per position
  grid_dep_launch();
  if (read_status(a.dev_status)) return;
  const int K = (int)a.K_max, B = (int)a.B, tid = threadIdx.x, lane = tid & 31;
  if (tid < kMaxK + 3) {
    cnt[tid] = 0;
    cntb[tid] = 0;
  }
  __syncthreads();
  for (int r0 = 0; r0 < B; r0 += kPlanThreads) {   // every thread runs every round: warp-wide ballots
    const int r = r0 + tid;
    int nr = 0;                                    // rows of request r
    if (r < B) {
      a.dead[r] = kNoReject;
      a.bonus_key[r] = 0ull;
      a.counters[r] = 0;
      const int l = a.ell[r];
      nr = (l >= 0 && l <= K) ? l + 1 : 0;
      if (nr > 0 && a.temperature[r] != 0.0f) atomicAdd(&cntb[l + 1], 1);
    }
    for (int j = 1; j <= K + 1; ++j) {
      const uint32_t bal = __ballot_sync(0xffffffffu, j <= nr);
      if (bal == 0u) break;
      if (lane == 0) atomicAdd(&cnt[j], __popc(bal));
    }
  }
  __syncthreads();
  if (tid == 0) {
    int tot = 0, nbt = 0;
    for (int j = 1; j <= K + 1; ++j) {
      tot += cnt[j];
      nbt += cntb[j];
    }
    // parts per bonus draw: all listed rows in one wave of the scan, at most one part per
    // slice, and within the list's capacity B (kMaxK + 1)
    int P = 1;
    if (nbt > 0 && tot + nbt <= a.scan_cap) {
      P = min(4, 1 + (a.scan_cap - tot) / nbt);
      P = min(P, a.row_slices);
      P = min(P, 1 + (int)(((int64_t)B * (kMaxK + 1) - tot) / nbt));
      P = max(P, 1);
    }
    int st = 0;
    for (int j = 1; j <= K + 1; ++j) {
      a.row_start[j] = st;
      a.row_fill[j] = 0;
      st += cnt[j] + (P - 1) * cntb[j];
    }
    a.nrows[0] = st;
    a.nrows[1] = P;
    *a.scan_next = 0;
    a.jobs_nact[0] = B;    // the residual jobs' counts (verify_jobs fills [1])
    a.jobs_nact[1] = 0;
    a.jobs_nact[2] = 0;
    if (a.jobs_gbar) {
      a.jobs_gbar[0] = 0;
      a.jobs_gbar[1] = 0;
    }
  }
}

constexpr int kFillThreads = 256;

// A thread per (request r, position j), j = 1..K_max + 1: the row if j <= ell_r + 1.  The
// thread of j = 1 checks the request's length, offsets and temperature, each row's thread its
// own draft token before using it; a slot is taken per warp and position (the lanes with the
// same j share one atomic).
template <int DT>
__global__ void __launch_bounds__(kFillThreads) verify_plan_fill(const __grid_constant__ VerifyArgs a) {
  grid_dep_wait();
  grid_dep_launch();
  if (read_status(a.dev_status)) return;
  const int K = (int)a.K_max, B = (int)a.B, lane = threadIdx.x & 31;
  const int64_t item = (int64_t)blockIdx.x * kFillThreads + threadIdx.x;
  const int r = (int)(item / (K + 1)), j = (int)(item % (K + 1)) + 1;
  bool row = false;
  VRow w;
  int rs = 0;
  if (r < B) {
    // every value the row may need, loaded together before any of it is used (each index is
    // in range whatever the lengths hold): one round trip to memory instead of a chain
    const int l = a.ell[r];
    const float T = a.temperature[r];
    const int off = a.tgt_off[r];
    const int drow = r * K + min(j, K) - 1;
    const int x = a.draft_tok[drow];
    const float zx_out = a.D_zx ? a.D_zx[drow] : 0.0f;
    const float lse_q = a.D_lse ? a.D_lse[drow] : 0.0f;
    rs = a.row_start[j];
    if (j == 1) {
      const int err = request_error(K, r, l, T, off, a.tgt_off[r + 1], a.tgt_off[0]);
      if (err) set_status(a.dev_status, err);
    }
    if (l >= 0 && l <= K && j <= l + 1) {
      const bool greedy = (T == 0.0f);
      const float invT = greedy ? 1.0f : 1.0f / T;
      row = true;
      w.r = r;
      w.j = j;
      w.invT = invT;
      w.lqx = 0.0f;
      if (j <= l) {
        w.drow = drow;
        w.x = x;
        w.trow = off + j - 1;
        if (w.x < 0 || w.x >= (int)a.V) {
          set_status(a.dev_status, DSPARK_ERR_TOKEN_RANGE);
          row = false;
        } else if (greedy) {
          w.kind = 2;
        } else if (a.D_lse != nullptr) {
          // log q(x_j) from the draft normaliser and the drawn token's logit (its own output,
          // or the stored row's element)
          const float zx = a.D_zx ? zx_out : load1<DT>(a.D, (int64_t)w.drow * a.V + w.x);
          w.lqx = zx * invT - lse_q;
          w.kind = 1;
        } else {
          w.kind = 3;
        }
      } else {
        // the bonus row: drawn (or its argmax taken) by the scan, used when every position is
        // accepted; a draw is listed as nrows[1] parts (x: parts and part, below)
        w.drow = 0;
        w.x = -1;
        w.trow = off + l;
        w.kind = greedy ? 5 : 4;
      }
    }
  }
  // list slots of this thread's row: the parts of a bonus draw, else one; lanes with the same
  // position and the same count share one atomic
  const int np = (row && w.kind == 4) ? a.nrows[1] : 1;
  const uint32_t bal = __ballot_sync(0xffffffffu, row);
  const uint32_t peers = __match_any_sync(0xffffffffu, row ? 2 * j + (np > 1 ? 1 : 0) : 0) & bal;
  if (!row) return;
  const int leader = __ffs(peers) - 1;
  int slot = 0;
  if (lane == leader) slot = atomicAdd(&a.row_fill[j], np * __popc(peers));
  slot = __shfl_sync(peers, slot, leader) + np * __popc(peers & ((1u << lane) - 1u));
  for (int p = 0; p < np; ++p) {
    if (w.kind == 4) w.x = (np << 8) | p;
    a.rows[bchk(rs + slot + p, (int64_t)B * (kMaxK + 1), a.dev_status)] = w;
  }
}

// One block of the bonus draw (the two-level draw over z / T) from its 16 bf16 pair words in
// any order of its four 16-byte units.  The block's maximum and mass do not depend on that
// order beyond the rounding of the sum; only a block that takes the lead needs its elements in
// order, and reload(c) gives them so for the inverse CDF (the weights again by the scalar fma
// that each lane of fma.f32x2 rounds like).  The draw needs no normaliser, so none is kept.
template <class PickWord, class Reload>
__device__ __forceinline__ void bonus_block(BRace &r, const uint32_t (&pk)[16], float a, uint32_t wb, int v0,
                                            PickWord pick_word, Reload reload) {
  __nv_bfloat162 m2[4] = {bf162_word(pk[0]), bf162_word(pk[1]), bf162_word(pk[2]), bf162_word(pk[3])};
#pragma unroll
  for (int e = 4; e < 16; ++e) m2[e & 3] = __hmax2(m2[e & 3], bf162_word(pk[e]));
  m2[0] = __hmax2(__hmax2(m2[0], m2[1]), __hmax2(m2[2], m2[3]));
  const float mz = fmaxf(__low2float(m2[0]), __high2float(m2[0]));
  if (mz == -INFINITY) return;
  const float Mb = mz * a;
  const unsigned long long aa = f2_pack(a, a), mb = f2_pack(-Mb, -Mb);
  unsigned long long s01 = f2_pack(0.0f, 0.0f), s23 = s01;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    float y0, y1;
    f2_unpack(f2_fma(f2_pack(__uint_as_float(pk[j] << 16), __uint_as_float(pk[j] & 0xffff0000u)), aa, mb), y0, y1);
    const unsigned long long ee = f2_pack(fast_ex2(y0), fast_ex2(y1));
    if (j & 1) s23 = f2_add(s23, ee);
    else s01 = f2_add(s01, ee);
  }
  float s0, s1, s2, s3;
  f2_unpack(s01, s0, s1);
  f2_unpack(s23, s2, s3);
  const float Sb = (s0 + s1) + (s2 + s3);
  if (!brace_enter(r, (Mb + fast_lg2(Sb)) * kLn2, wb)) return;
  uint32_t c[16];
  reload(c);
  float w[kBlockW];
#pragma unroll
  for (int q = 0; q < kBlockW; ++q) {
    const uint32_t wq = c[q >> 1];
    w[q] = fast_ex2(fmaf(__uint_as_float((q & 1) ? (wq & 0xffff0000u) : (wq << 16)), a, -Mb));
  }
  r.idx = v0 + pick_in_block(w, uniform_accept(pick_word()) * Sb);
}

// ---------------------------------------------------------------------------
// 2. scan: the rows' statistics, each row decided where it completes
// ---------------------------------------------------------------------------
constexpr int kScanWarps = kRowThreads / 32;        // reducing warps; one more warp stages
constexpr int kScanThreads = kRowThreads + 32;
constexpr int kScanStages = 2;
constexpr int kSliceBytes = kRowSlice * 2;          // one bf16 slice (24 KB)

// One ring slot: a slice of a listed row, a skipped row (kind 0, one slot) or the end (-1).
struct ScanMeta {
  VRow w;
  int ri, sl, kind;
  int last;           // the row's last slice
};

// The accept decision of a completed row from its merged statistics (lane 0 of warp 0):
// stores the row's results and lowers the request's first-rejection word on a rejection.
__device__ __forceinline__ void decide_row(const VerifyArgs &a, const VRow &w, const Stats &ct, const Stats &cd,
                                           float zx_t, float zx_d) {
  const bool greedy = (w.kind == 2), two = (w.kind == 3);
  VRowRes rr;
  rr.amax = ct.idx;
  rr.lse_t = greedy ? ct.best : ct.m + logf(ct.S);
  rr.zx_t = greedy ? 0.0f : zx_t;
  rr.lse_q = two ? cd.m + logf(cd.S) : 0.0f;
  bool reject;
  if (greedy) {
    reject = (w.x != rr.amax);
  } else {
    const float u = uniform_accept(philox(a.key, 0u, (uint32_t)w.j, (uint32_t)w.r, kTagAccept).x);
    const float lqx = two ? zx_d - rr.lse_q : w.lqx;
    reject = !(u < expf((rr.zx_t - rr.lse_t) - lqx));
  }
  a.rres[(int64_t)w.r * (a.K_max + 1) + w.j - 1] = rr;
  if (reject) atomicMin(a.dead + w.r, w.j);
}

__device__ __forceinline__ void named_sync_scan() {
  asm volatile("bar.sync 1, %0;" ::"n"(kRowThreads) : "memory");
}

// Persistent CTAs take whole listed rows in list order (position-major, so every request's
// position j is taken before any position j + 1): CTA c first row c, then the next untaken
// row from a shared counter, so a CTA whose row was cheap (skipped, or statistics only) takes
// the next one sooner than one drawing a bonus row (19 % off the call at B = 2048; the first
// row by CTA index keeps the rows of a small batch on different SMs).  Each CTA streams each row's
// vocabulary slices in order.  BULK (bf16, 16-byte aligned rows): warp kScanWarps stages each
// slice by bulk copy into a kScanStages ring; otherwise the reducing warps load the slice
// themselves (VEC: 16-byte loads) and the staging warp only hands out the slices.  A row
// whose request already has an earlier rejection is skipped before any of it is read.
// Each thread folds its part of every slice into running statistics; at the row's last
// slice the four warps reduce in a fixed order and warp 0 decides the row.
template <int DT, bool VEC, bool BULK>
__global__ void __launch_bounds__(kScanThreads) verify_scan(const __grid_constant__ VerifyArgs a) {
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ uint64_t full[kScanStages], empty[kScanStages];
  __shared__ ScanMeta meta[kScanStages];
  __shared__ Stats s_part[2][2][kScanWarps];   // [row parity][target, draft][warp]
  __shared__ float s_zx[2][2];                  // [row parity][target, draft]: scaled logits at x
  __shared__ Race s_race[2][kScanWarps];        // [row parity][warp]: bonus draws
  __shared__ int abort_flag;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  grid_dep_wait();
  grid_dep_launch();
  if (read_status(a.dev_status)) return;
  const int S = a.row_slices, V = (int)a.V;
  const int nrows = *(volatile const int32_t *)a.nrows;
  if ((int)blockIdx.x >= nrows) return;
  const bool two = (a.D_lse == nullptr);
  const uint32_t stage_bytes = BULK ? (two ? 2u : 1u) * kSliceBytes : 0u;
  const uint32_t bar_full = smem_u32(&full[0]), bar_empty = smem_u32(&empty[0]);
  if (tid == 0) {
    for (int s = 0; s < kScanStages; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, kScanWarps);
    }
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  volatile int *abort = &abort_flag;

  if (warp == kScanWarps) {
    // ---------------- staging warp (lane 0) ----------------
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      uint32_t last_use[kScanStages];
      bool issued[kScanStages];
#pragma unroll
      for (int s = 0; s < kScanStages; ++s) {
        last_use[s] = 0;
        issued[s] = false;
      }
      int t = 0;   // slots handed out
      auto slot = [&](const ScanMeta &m) -> bool {   // the next ring slot gets m (and its copies)
        const int s = t % kScanStages;
        const uint32_t use = (uint32_t)(t / kScanStages);
        if (!mbar_wait(bar_empty + 8 * s, (use & 1u) ^ 1u, abort)) return false;
        meta[s] = m;
        if (!BULK || m.kind <= 0) {
          mbar_arrive(bar_full + 8 * s);
        } else {
          const int lo = m.sl * kRowSlice;
          const uint32_t bytes = (uint32_t)(min(kRowSlice, V - lo) * 2);
          const uint32_t dst = smem_u32(ring) + (uint32_t)s * stage_bytes;
          mbar_arrive_tx(bar_full + 8 * s, bytes * (m.kind == 3 ? 2u : 1u));
          bulk_g2s(dst, (const unsigned short *)a.tgt + ((int64_t)m.w.trow * V + lo), bytes, bar_full + 8 * s, pol);
          if (m.kind == 3)
            bulk_g2s(dst + kSliceBytes, (const unsigned short *)a.D + ((int64_t)m.w.drow * V + lo), bytes,
                     bar_full + 8 * s, pol);
#pragma unroll
          for (int q = 0; q < kScanStages; ++q)
            if (q == s) {
              last_use[q] = use;
              issued[q] = true;
            }
        }
        ++t;
        return true;
      };
      bool ok = true;
      for (int ri = blockIdx.x; ok && ri < nrows; ri = (int)gridDim.x + atomicAdd(a.scan_next, 1)) {
        ScanMeta m;
        m.ri = ri;
        m.w = a.rows[ri];
#ifdef DSPARK_BOUNDS
        m.w.r = (int)bchk(m.w.r, a.B, a.dev_status);
        m.w.j = 1 + (int)bchk(m.w.j - 1, a.K_max + 1, a.dev_status);
        m.w.trow = (int)bchk(m.w.trow, a.tgt_off[a.B], a.dev_status);
        m.w.drow = (int)bchk(m.w.drow, a.B * a.K_max, a.dev_status);
#endif
        // the row's slices (a part of a bonus draw: its range of them)
        int sl0 = 0, sl1 = S;
        if (m.w.kind == 4) {
          const int parts = max(1, m.w.x >> 8), part = m.w.x & 255;
          sl0 = part * S / parts;
          sl1 = min(S, (part + 1) * S / parts);
        }
        // rows past a rejection already found need no statistics
        const bool skip = *(volatile const int32_t *)(a.dead + m.w.r) < m.w.j || sl0 >= sl1;
        if (skip) {
          m.sl = 0;
          m.kind = 0;
          m.last = 1;
          ok = slot(m);
          continue;
        }
        m.kind = m.w.kind;
        for (int sl = sl0; ok && sl < sl1; ++sl) {
          m.sl = sl;
          m.last = (sl == sl1 - 1);
          ok = slot(m);
        }
      }
      if (ok) {
        ScanMeta m;
        m.kind = -1;
        slot(m);
      }
      if (*abort) {   // wait (bounded) until the copies issued into each stage have landed
#pragma unroll
        for (int q = 0; q < kScanStages; ++q) {
          if (!issued[q]) continue;
          const long long t0 = clock64();
          while (!mbar_try(bar_full + 8 * q, last_use[q] & 1u) && clock64() - t0 < kTimeoutCycles / 4) {
          }
        }
        set_status(a.dev_status, DSPARK_ERR_DEVICE_TIMEOUT);
      }
    }
    return;
  }

  // ---------------- reducing warps ----------------
  Stats rt, rd;            // running statistics of the current row (this thread's share)
  stats_init(rt);
  stats_init(rd);
  BRace rb;                // running bonus draw of the current row (kind 4)
  brace_init(rb);
  // parity of the shared partials: it flips at the end of every row that has statistics (all
  // such rows end at the named barrier), never at a skipped row, so a warp can write the
  // partials of a row only after every warp passed the previous row's barrier -- that is,
  // after warp 0 merged the row before that one, which used the same half
  int rows_done = 0;
  for (int t = 0;; ++t) {
    const int s = t % kScanStages;
    const uint32_t use = (uint32_t)(t / kScanStages);
    if (!mbar_wait(bar_full + 8 * s, use & 1u, abort)) break;
    const ScanMeta m = meta[s];
    if (m.kind < 0) break;
    const int par = rows_done & 1;
    if (m.kind == 4) {
      // bonus draw: this thread's 32-wide blocks of the slice (blocks tid, tid + 128, ...), the
      // two-level draw on z / T with the residual / bonus streams at position ell + 1
      const int lo = min(V, m.sl * kRowSlice), hi = min(V, lo + kRowSlice);
      const float a2 = m.w.invT * kLog2e;
      const uint32_t pos = (uint32_t)m.w.j, rq = (uint32_t)m.w.r;
      // noise words: block b = tid + q * kRowThreads of the slice is block (lo / 32 + b) of the
      // row, in Philox group lo / 128 + tid / 4 + q * kRowThreads / 4 as word tid & 3.  The four
      // lanes of a quad share their groups, so lane 4i + c makes the one Philox call of
      // iteration c for its quad and the quad's lanes take their words from it by shuffles
      // (all lanes, before any of them leaves the loop at the row's end)
      static_assert(kRowSlice % 128 == 0 && kRowSlice / 32 / kRowThreads <= 3, "noise groups of a slice");
      const int cw = lane & 3;
      const uint4 pw = philox(a.key, ((uint32_t)lo >> 7) + (uint32_t)(tid >> 2) + (uint32_t)(cw * (kRowThreads / 4)),
                              pos, rq, kTagResid);
      uint32_t wq[3];
#pragma unroll
      for (int q = 0; q < 3; ++q) {
        const int src = (lane & ~3) | q;
        const uint32_t x = __shfl_sync(0xffffffffu, pw.x, src), y = __shfl_sync(0xffffffffu, pw.y, src);
        const uint32_t z = __shfl_sync(0xffffffffu, pw.z, src), w = __shfl_sync(0xffffffffu, pw.w, src);
        wq[q] = cw == 0 ? x : (cw == 1 ? y : (cw == 2 ? z : w));
      }
#pragma unroll 1
      for (int q = 0; q < kRowSlice / 32 / kRowThreads; ++q) {
        const int b = tid + q * kRowThreads;
        const int v0 = lo + 32 * b;
        if (v0 >= hi) break;
        const uint32_t g = (uint32_t)v0 >> 5;
        const uint32_t wb = q == 0 ? wq[0] : (q == 1 ? wq[1] : wq[2]);
        auto pick = [&] { return word_of(philox(a.key, g >> 2, pos, rq, kTagResidPick), (int)(g & 3u)); };
        if (BULK) {
          const uint32_t base = smem_u32(ring) + (uint32_t)s * stage_bytes + 64u * (uint32_t)b;
          // the block's four 16-byte units, loaded in an order rotated by (lane >> 1) & 3 so that
          // the 8 lanes of each quarter warp touch 8 different bank groups; the block's mass is
          // summed in that order, and a block that takes the lead reloads its units in element
          // order for the inverse CDF
          const int rot = (lane >> 1) & 3;
          uint4 u[4];
#pragma unroll
          for (int h = 0; h < 4; ++h) u[h] = ld_shared_u4(base + 16u * (uint32_t)((h + rot) & 3));
          if (v0 + 32 > hi) {                 // the row's ragged end: units past it hold -inf
#pragma unroll
            for (int h = 0; h < 4; ++h)
              if (v0 + 8 * ((h + rot) & 3) + 8 > hi) u[h] = make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
          }
          uint32_t pk[16];
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            pk[4 * h] = u[h].x;
            pk[4 * h + 1] = u[h].y;
            pk[4 * h + 2] = u[h].z;
            pk[4 * h + 3] = u[h].w;
          }
          bonus_block(rb, pk, a2, wb, v0, pick, [&](uint32_t (&c)[16]) {
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              uint4 x = ld_shared_u4(base + 16u * (uint32_t)h);
              if (v0 + 8 * h + 8 > hi) x = make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
              c[4 * h] = x.x;
              c[4 * h + 1] = x.y;
              c[4 * h + 2] = x.z;
              c[4 * h + 3] = x.w;
            }
          });
        } else {
          float t[kBlockW];
          load32<DT, VEC>(a.tgt, (int64_t)m.w.trow * V, v0, hi, t);
          brace_softmax_block(rb, t, block_max(t), a2, wb, v0, pick, NoLogit{});
        }
      }
    } else if (m.kind) {
      RowItem it;
      it.rowi = m.w.drow;
      it.x = m.w.x;
      it.kind = (m.kind == 2 || m.kind == 5) ? 2 : 1;
      it.invT = m.w.invT;
      it.trow = (int64_t)m.w.trow * V;
      it.lo = min(V, m.sl * kRowSlice);
      it.hi = min(V, it.lo + kRowSlice);
      Stats st, sd;
      stats_init(st);
      stats_init(sd);
      if (BULK) {
        const uint32_t base = smem_u32(ring) + (uint32_t)s * stage_bytes;
        uint4 pk[kRowPk];
#pragma unroll
        for (int q = 0; q < kRowPk; ++q) pk[q] = ld_shared_u4(base + 16u * (uint32_t)(q * kRowThreads + tid));
        row_consume(it, pk, tid, st, &s_zx[par][0]);
        if (m.kind == 3) {
#pragma unroll
          for (int q = 0; q < kRowPk; ++q)
            pk[q] = ld_shared_u4(base + kSliceBytes + 16u * (uint32_t)(q * kRowThreads + tid));
          RowItem itd = it;
          itd.kind = 1;
          row_consume(itd, pk, tid, sd, &s_zx[par][1]);
        }
      } else {
        row_generic<DT, VEC>(a, it, m.kind == 3, tid, st, sd, &s_zx[par][0], &s_zx[par][1]);
      }
      stats_merge(rt, st);
      if (m.kind == 3) stats_merge(rd, sd);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_empty + 8 * s);   // the stage is read
    if (!m.last) continue;
    if (m.kind == 4) {
      // the bonus draw of the row (or of its part): warps reduce their races, warp 0 merges
      // the four and folds the winner into the request's packed (score, index) key -- the
      // maximum score, the smallest index on ties, whatever the order the parts arrive in
      Race rc = from_partial(to_partial(rb));
#pragma unroll
      for (int d = 16; d > 0; d >>= 1) race_merge(rc, race_shfl_down(rc, d));
      if (lane == 0) s_race[par][warp] = rc;
      named_sync_scan();
      if (warp == 0 && lane == 0) {
        Race tot = s_race[par][0];
#pragma unroll
        for (int q = 1; q < kScanWarps; ++q) race_merge(tot, s_race[par][q]);
        if (tot.idx >= 0) atomicMax(a.bonus_key + m.w.r, score_key(tot.best, tot.idx));
      }
    } else if (m.kind) {
      // the row is complete: warps reduce their shares, warp 0 merges the four in order
      const int kind = (m.kind == 2 || m.kind == 5) ? 2 : 1;
      Stats wt = warp_reduce_row(rt, kind);
      Stats wd = (m.kind == 3) ? warp_reduce_row(rd, 1) : rd;
      if (lane == 0) {
        s_part[par][0][warp] = wt;
        s_part[par][1][warp] = wd;
      }
      named_sync_scan();
      if (warp == 0 && lane == 0) {
        Stats ct = s_part[par][0][0], cd = s_part[par][1][0];
#pragma unroll
        for (int q = 1; q < kScanWarps; ++q) {
          stats_merge(ct, s_part[par][0][q]);
          if (m.kind == 3) stats_merge(cd, s_part[par][1][q]);
        }
        if (m.kind == 5) {        // greedy bonus: the argmax of the row
          VRowRes rr;
          rr.lse_t = ct.best;
          rr.amax = ct.idx;
          rr.zx_t = 0.0f;
          rr.lse_q = 0.0f;
          a.rres[(int64_t)m.w.r * (a.K_max + 1) + m.w.j - 1] = rr;
        } else {
          decide_row(a, m.w, ct, cd, s_zx[par][0], s_zx[par][1]);
        }
      }
    }
    stats_init(rt);
    stats_init(rd);
    brace_init(rb);
    if (m.kind) ++rows_done;
  }
  if (*abort && tid == 0) set_status(a.dev_status, DSPARK_ERR_DEVICE_TIMEOUT);
}

// ---------------------------------------------------------------------------
// 3. sampling: outcome per request and the residual / bonus draw
// ---------------------------------------------------------------------------
template <int DT, bool VEC>
__global__ void __launch_bounds__(kSampleThreads, 2) verify_sample(const __grid_constant__ VerifyArgs a) {
  __shared__ Race red[kSampleThreads / 32];
  __shared__ int s_any[kSampleThreads / 32];
  __shared__ int s_last, s_tok;
  const int cx = blockIdx.x, tid = threadIdx.x;
  grid_dep_wait();
  if (read_status(a.dev_status)) return;
  const int V = (int)a.V, K = (int)a.K_max;
  const int njobs = *(volatile const int32_t *)(a.jobs_nact + 1);
  for (int ji = blockIdx.y; ji < njobs; ji += gridDim.y) {
    // one T > 0 rejection: its residual token (every other output is verify_jobs')
    const VJob jb = a.jobs[ji];
    const int r = jb.r;
    VerifyJob job;
    job.mode = a.resid_key ? 4 : 1;
    job.pos = jb.j;
    job.trow = jb.trow;
    job.drow = jb.urow;
    job.lse_t = jb.lse_t;
    job.lse_q = jb.lse_q;
    job.invT = jb.invT;
    job.out_slot = r * (K + 1) + jb.j - 1;
    if (job.mode == 4) {
      // the residual was drawn by the tensor-core recompute pass: its token, or (no p > q
      // survived rounding anywhere) the draw from p on the rejecting row; chunk 0 only
      if (cx != 0) continue;
      int tok = -1;
      if (a.resid_any[r]) {
        tok = key_index(a.resid_key[r]);
      } else {
        BRace bp;
        brace_init(bp);
        bool dummy = false;
        sample_range<DT, VEC>(a, job, r, 0, V, tid, kSampleThreads, bp, dummy, true);
        tok = race_block_reduce(from_partial(to_partial(bp)), red).idx;
      }
      if (tid == 0) a.out_tok[job.out_slot] = tok;
      __syncthreads();
      continue;
    }
    const int lo = min(V, cx * a.chunk_len), hi = min(V, lo + a.chunk_len);
    BRace br;
    brace_init(br);
    bool any_pos = false;
    sample_range<DT, VEC>(a, job, r, lo, hi, tid, kSampleThreads, br, any_pos, false);
    const int any = __syncthreads_or(any_pos ? 1 : 0);
    Race rc = race_block_reduce(from_partial(to_partial(br)), red);
    if (tid == 0) {
      Partial p = to_partial(rc);
      p.m = any ? 1.0f : 0.0f;    // the sampling pass needs no softmax: the field carries a flag
      a.partials[(int64_t)r * a.chunks + cx] = p;
      __threadfence();
      const int prev = atomicAdd(&a.counters[r], 1);
      s_last = (prev == a.chunks - 1);
    }
    __syncthreads();
    if (!s_last) continue;
    __threadfence();
    if (tid < 32) {
      Race tot;
      race_init(tot);
      int any_all = 0;
      for (int q = tid; q < a.chunks; q += 32) {
        const Partial p = load_partial(a.partials + ((int64_t)r * a.chunks + q));
        Race x = from_partial(p);
        x.m = -INFINITY;
        x.S = 0.0f;
        race_merge(tot, x);
        any_all |= (p.m != 0.0f);
      }
      for (int d = 16; d > 0; d >>= 1) race_merge(tot, race_shfl_down(tot, d));
      any_all = __any_sync(0xffffffffu, any_all);
      if (tid == 0) {
        s_any[0] = any_all;
        s_tok = tot.idx;
      }
    }
    __syncthreads();
    if (job.mode == 1 && !s_any[0]) {
      // no element with p > q survived rounding: sample the correction from p instead
      BRace bp;
      brace_init(bp);
      bool dummy = false;
      sample_range<DT, VEC>(a, job, r, 0, V, tid, kSampleThreads, bp, dummy, true);
      const Race rp = race_block_reduce(from_partial(to_partial(bp)), red);
      if (tid == 0) s_tok = rp.idx;
    }
    if (tid == 0) a.out_tok[job.out_slot] = s_tok;
    __syncthreads();
  }
}

// Every request's outcome from the scan, and the T > 0 rejections as the jobs of the residual
// draw (a thread per request; job slots from one global atomic per warp, so the order of the
// list is the atomics' and changes no result).  n = (first rejection) - 1, or ell_r when every
// position was accepted; the accepted tokens, the -1 padding and at slot n the greedy
// correction (the rejecting row's argmax) or the bonus token (the scan's draw, or its argmax
// for T = 0) are written here; a T > 0 rejection's token is the residual draw's.  With the
// recompute entry point the residual pass's keys and flags start from zero.
constexpr int kJobThreads = 256;
__global__ void __launch_bounds__(kJobThreads) verify_jobs(const __grid_constant__ VerifyArgs a) {
  grid_dep_wait();
  grid_dep_launch();
  if (read_status(a.dev_status)) return;
  const int K = (int)a.K_max, B = (int)a.B, lane = threadIdx.x & 31;
  const int r = blockIdx.x * kJobThreads + threadIdx.x;
  bool job = false;
  VJob jb;
  if (r < B) {
    if (a.key_out) {
      a.key_out[r] = 0ull;
      a.any_out[r] = 0;
    }
    // the request's values, loaded together before any is used: its length, first rejection,
    // temperature, bonus key, target offset, anchor and draft tokens (the loop is unrolled
    // over kMaxK so that the tokens stay in registers)
    const int l = a.ell[r];
    const int dead = a.dead[r];
    const float T = a.temperature[r];
    const unsigned long long bk = a.bonus_key[r];
    const int off = a.tgt_off[r];
    const int anc = a.anchor ? a.anchor[r] : 0;
    int tok[kMaxK];
#pragma unroll
    for (int i = 0; i < kMaxK; ++i) tok[i] = i < K ? a.draft_tok[(int64_t)r * K + i] : -1;
    const int n = dead <= l ? dead - 1 : l;
    const bool greedy = (T == 0.0f);
    const int64_t rb = (int64_t)r * (K + 1);
    // the deciding row's results (n <= l <= K_max: in range; for a T > 0 bonus not read)
    const VRowRes rr = a.rres[rb + n];
    const float lq = (a.D_lse && n < K) ? a.D_lse[(int64_t)r * K + n] : rr.lse_q;
    int last = -1;    // the token after the accepted ones: the correction, the bonus token
    if (greedy) last = rr.amax;                       // the rejecting row's or the bonus row's argmax
    else if (n == l) last = bk ? key_index(bk) : -1;  // the bonus draw
    int prev = anc;   // x_n, the token before position n + 1
#pragma unroll
    for (int i = 0; i < kMaxK; ++i)
      if (i + 1 == n) prev = tok[i];
#pragma unroll
    for (int i = 0; i <= kMaxK; ++i)
      if (i <= K) a.out_tok[rb + i] = i < n ? tok[i] : (i == n ? last : -1);
    a.n_acc[r] = n;
    job = n < l && !greedy;
    jb.r = r;
    jb.j = n + 1;
    jb.prev = a.anchor ? prev : 0;
    jb.urow = r * K + n;
    jb.trow = off + n;
    jb.lse_t = rr.lse_t;
    jb.lse_q = lq;
    jb.invT = 1.0f / T;
  }
  const uint32_t bal = __ballot_sync(0xffffffffu, job);
  if (bal == 0u) return;
  const int leader = __ffs(bal) - 1;
  int slot = 0;
  if (lane == leader) slot = atomicAdd(&a.jobs_nact[1], __popc(bal));
  slot = __shfl_sync(0xffffffffu, slot, leader) + __popc(bal & ((1u << lane) - 1u));
  if (!job) return;
  a.jobs[bchk(slot, B, a.dev_status)] = jb;
}

// Launch with programmatic stream serialisation: the kernel may become resident while the
// previous kernel in the stream runs, and waits for it in grid_dep_wait().
template <class... P>
cudaError_t launch_dependent(void (*kern)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                             const VerifyArgs &a) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

template <int DT, bool VEC, bool BULK>
cudaError_t launch_typed(VerifyArgs a, cudaStream_t s, int num_sms, const DraftArgs *resid) {
  // sampling chunks: about two CTAs per SM over all requests in one wave, each chunk a
  // multiple of 32 columns (the blocks of the two-level draw) and at most a.chunks of them
  {
    const int64_t want = (2LL * num_sms) / a.B;
    const int c = (int)(want < 1 ? 1 : (want > a.chunks ? a.chunks : want));
    const int64_t per = (a.V + c - 1) / c;
    a.chunk_len = (int)((per + kBlockW - 1) / kBlockW * kBlockW);
    a.chunks = (int)((a.V + a.chunk_len - 1) / a.chunk_len);
  }
  // scan: a wave of persistent CTAs (4 per SM with single-row stages, 2 with two rows; two
  // stages at four CTAs per SM ran 4 % faster than three stages at three)
  const bool two = (a.D_lse == nullptr);
  const int64_t per_sm = (BULK && two) ? 2 : 4;
  a.scan_cap = (int)(per_sm * num_sms);
  verify_plan_count<<<1, kPlanThreads, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = launch_dependent(verify_plan_fill<DT>, dim3((unsigned)((a.B * (a.K_max + 1) + kFillThreads - 1) / kFillThreads)),
                       dim3(kFillThreads), 0, s, a);
  if (e != cudaSuccess) return e;
  const int smem = BULK ? kScanStages * kSliceBytes * (two ? 2 : 1) : 0;
  if (BULK) {
    e = ensure_dynamic_smem((const void *)verify_scan<DT, VEC, BULK>, smem);
    if (e != cudaSuccess) return e;
  }
  const int64_t max_rows = a.B * (a.K_max + 1) + 3 * a.B;     // with bonus draws in four parts
  const int64_t grid = max_rows < a.scan_cap ? max_rows : a.scan_cap;
  e = launch_dependent(verify_scan<DT, VEC, BULK>, dim3((unsigned)grid), dim3(kScanThreads), (size_t)smem, s, a);
  if (e != cudaSuccess) return e;
  e = launch_dependent(verify_jobs, dim3((unsigned)((a.B + kJobThreads - 1) / kJobThreads)), dim3(kJobThreads), 0, s, a);
  if (e != cudaSuccess) return e;
  if (resid) {
    e = launch_resid_tc(*resid, s, num_sms);
    if (e != cudaSuccess) return e;
  }
  return launch_dependent(verify_sample<DT, VEC>, dim3(a.chunks, (unsigned)(a.B < 65535 ? a.B : 65535)),
                          dim3(kSampleThreads), 0, s, a);
}

}  // namespace

int verify_row_slices(int64_t V) { return (int)((V + kRowSlice - 1) / kRowSlice); }

// Workspace layout (every part 256-byte aligned): sampling counters [B], sampling partials
// [B * chunks], the listed rows [B * (kMaxK + 1)], their count, the first-rejection words [B],
// the bonus draws' keys [B], the row results [B * (kMaxK + 1)].  Sized for kMaxK positions, so
// the size depends on B and V only.
size_t verify_ws_bytes(int64_t B, int64_t V, int *chunks) {
  const int c = (int)((V + kSampleUnit - 1) / kSampleUnit);   // the most chunks a call uses
  if (chunks) *chunks = c;
  auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
  const size_t rows = (size_t)B * (size_t)(kMaxK + 1);
  return al(sizeof(int32_t) * (size_t)B) + al(sizeof(Partial) * (size_t)B * (size_t)c) + al(sizeof(VRow) * rows) +
         al(sizeof(int32_t)) + al(sizeof(int32_t) * (size_t)B) + al(sizeof(unsigned long long) * (size_t)B) +
         al(sizeof(VRowRes) * rows) +
         al(sizeof(VJob) * (size_t)B) + al(sizeof(int32_t) * 3);
}

void verify_carve(VerifyArgs &a, void *workspace) {
  auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
  const size_t rows = (size_t)a.B * (size_t)(kMaxK + 1);
  int chunks = 1;
  verify_ws_bytes(a.B, a.V, &chunks);
  a.chunks = chunks;
  a.row_slices = verify_row_slices(a.V);
  char *p = (char *)workspace;
  a.counters = (int32_t *)p;
  p += al(sizeof(int32_t) * (size_t)a.B);
  a.partials = (Partial *)p;
  p += al(sizeof(Partial) * (size_t)a.B * (size_t)chunks);
  a.rows = (VRow *)p;
  p += al(sizeof(VRow) * rows);
  a.nrows = (int32_t *)p;          // one 256-byte block: the count and the bonus parts, the starts, the fill counters
  a.row_start = a.nrows + 4;
  a.row_fill = a.nrows + 32;
  a.scan_next = a.nrows + 60;
  static_assert(32 + kMaxK + 3 <= 60, "plan counters fit one 256-byte block");
  p += al(sizeof(int32_t));
  a.dead = (int32_t *)p;
  p += al(sizeof(int32_t) * (size_t)a.B);
  a.bonus_key = (unsigned long long *)p;
  p += al(sizeof(unsigned long long) * (size_t)a.B);
  a.rres = (VRowRes *)p;
  p += al(sizeof(VRowRes) * rows);
  a.jobs = (VJob *)p;
  p += al(sizeof(VJob) * (size_t)a.B);
  a.jobs_nact = (int32_t *)p;
}

cudaError_t launch_verify(const VerifyArgs &a, cudaStream_t s, int num_sms, const DraftArgs *resid) {
  const int esz = a.dtype == DSPARK_F32 ? 4 : 2;
  const bool vec = ((a.V * esz) % 16 == 0) && ((uintptr_t)a.tgt % 16 == 0) &&
                   (a.D == nullptr || (uintptr_t)a.D % 16 == 0);
  if (a.dtype == DSPARK_F32)
    return vec ? launch_typed<DSPARK_F32, true, false>(a, s, num_sms, resid)
               : launch_typed<DSPARK_F32, false, false>(a, s, num_sms, resid);
  return vec ? launch_typed<DSPARK_BF16, true, true>(a, s, num_sms, resid)
             : launch_typed<DSPARK_BF16, false, false>(a, s, num_sms, resid);
}

}  // namespace dspark
