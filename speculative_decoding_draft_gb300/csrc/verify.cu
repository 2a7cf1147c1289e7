// Ragged rejection-sampling verification ("DSpark", S2.1; "Speculative
// decoding, from zero to DSpark", S2 and Appendix A1).
//
// Two kernels (after a reset of the per-request arrival counters):
//  1. verify_rows: one CTA per (drafted row, vocabulary slice) for every position
//     j = 1..ell_r of every request at once.  Each CTA streams its slice of target
//     row j (and of the draft row when no draft normaliser is given) with 16-byte
//     loads, reduces the online-softmax statistics (max, sum of exponentials) of
//     z/T -- the argmax for T = 0 -- and stores them with the scaled logit at the
//     draft token.  The last CTA of a request merges the slices of each row in a
//     fixed order and walks the positions, one lane per position: the first j with
//     u_j >= min(1, p(x_j)/q(x_j)) (or x_j != argmax for T = 0) ends the walk.  The
//     walk also produces the sampling job of the request: the residual at the
//     rejecting position, the bonus row when every position is accepted, or
//     nothing for greedy rejections (their correction is the argmax already found).
//     Rows past the first rejection are read too: all rows stream in parallel
//     instead of one position after another.
//  2. verify_sample: the residual / bonus two-level draw over the vocabulary,
//     spread over the whole GPU (request x vocabulary chunk, about two CTAs per
//     SM in one wave, each thread a run of 32-wide blocks; for the residual on bf16
//     rows the next block's loads are in flight while a block is drawn), with the
//     last block of each request merging the chunk partials.
#include "dspark_internal.cuh"

namespace dspark {
namespace {

constexpr int kRowThreads = 128;
constexpr int kRowCtasPerSm = 3;
constexpr int kBatch = 4;          // loads in flight per thread in the accept chain (fp32 / unaligned)
constexpr int kRowPk = 12;          // packed bf16 16-byte loads per thread and row item
constexpr int kRowSlice = kRowThreads * 8 * kRowPk;     // vocabulary slice of one row item
constexpr int kRowParts = kRowThreads / 32;              // partial statistics per item: one per warp
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

__device__ __forceinline__ Stats stats_shfl_down(const Stats &s, int d) {
  Stats o;
  o.m = __shfl_down_sync(0xffffffffu, s.m, d);
  o.S = __shfl_down_sync(0xffffffffu, s.S, d);
  o.best = __shfl_down_sync(0xffffffffu, s.best, d);
  o.idx = __shfl_down_sync(0xffffffffu, s.idx, d);
  return o;
}

__device__ __forceinline__ float pick8(const float (&x)[8], int q) {
  float v = x[0];
#pragma unroll
  for (int i = 1; i < 8; ++i)
    if (i == q) v = x[i];
  return v;
}

__device__ __forceinline__ __nv_bfloat162 bf162_word(uint32_t w) { return *reinterpret_cast<const __nv_bfloat162 *>(&w); }

__device__ __forceinline__ Partial stats_to_partial(const Stats &s) {
  Partial p;
  p.best = s.best;
  p.idx = s.idx;
  p.m = s.m;
  p.S = s.S;
  return p;
}
__device__ __forceinline__ Stats partial_to_stats(const Partial &p) {
  Stats s;
  s.best = p.best;
  s.idx = p.idx;
  s.m = p.m;
  s.S = p.S;
  return s;
}

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

// Metadata of item `item` (row-major over rows, then slices), the same in every thread.
// An invalid request raises the status word once (slice 0 of row 1, or of the row with
// the bad token) and streams nothing.
__device__ __forceinline__ RowItem row_item(const VerifyArgs &a, int item, int tid) {
  const int K = (int)a.K_max, V = (int)a.V, S = a.row_slices;
  RowItem it;
  it.rowi = item / S;
  const int sl = item % S;
  const int r = it.rowi / K, j = it.rowi % K + 1;
  it.kind = 0;
  // every value is requested before any is used: one round trip
  const int l = a.ell[r];
  const float T = a.temperature[r];
  const int x = a.draft_tok[it.rowi];
  const int64_t o0 = a.tgt_off[r], o1 = a.tgt_off[r + 1], of = a.tgt_off[0];
  const int err = request_error(K, r, l, T, o0, o1, of);
  if (err) {
    if (sl == 0 && j == 1 && tid == 0) set_status(a.dev_status, err);
    return it;
  }
  if (j > l) return it;
  if (x < 0 || x >= V) {
    if (sl == 0 && tid == 0) set_status(a.dev_status, DSPARK_ERR_TOKEN_RANGE);
    return it;
  }
  it.x = x;
  it.kind = (T == 0.0f) ? 2 : 1;
  it.invT = (T == 0.0f) ? 1.0f : 1.0f / T;
  it.trow = (o0 + j - 1) * (int64_t)V;
  it.lo = min(V, sl * kRowSlice);
  it.hi = min(V, it.lo + kRowSlice);
  return it;
}

// bf16 rows, 16-byte aligned: the item's kRowPk packed loads per thread.
__device__ __forceinline__ void row_issue(const VerifyArgs &a, const RowItem &it, int tid, uint4 (&pk)[kRowPk]) {
#pragma unroll
  for (int uu = 0; uu < kRowPk; ++uu) {
    const int v0 = it.lo + (uu * kRowThreads + tid) * 8;
    pk[uu] = (it.kind && v0 + 8 <= it.hi) ? __ldcs((const uint4 *)((const unsigned short *)a.tgt + it.trow + v0))
                                          : make_uint4(0u, 0u, 0u, 0u);
  }
}

// The item's statistics from its packed loads: the thread's maximum over its 8 kRowPk
// values first (bf16 pairs, exact), then one pass of exponentials against it, two lanes per
// fp32 instruction; slots past the slice hold -inf.
__device__ __forceinline__ void row_consume(const RowItem &it, uint4 (&pk)[kRowPk], int tid, Stats &st,
                                            float *own_t) {
#pragma unroll
  for (int uu = 0; uu < kRowPk; ++uu)
    if (it.lo + (uu * kRowThreads + tid) * 8 + 8 > it.hi) pk[uu] = make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
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

// Merge of the slice statistics of drafted row rowi (one warp, lanes over slices, then a
// fixed shuffle tree: the result does not depend on which CTA streamed which slice).
// Valid in lane 0.
__device__ __forceinline__ RowRes row_merge(const VerifyArgs &a, int64_t rowi, bool greedy, bool stream_d, int lane) {
  const int S = a.row_slices;
  const bool sd_on = !greedy && stream_d;
  Stats ct, cd;
  stats_init(ct);
  stats_init(cd);
  const float zt = greedy ? 0.0f : __ldcg(a.zx_t + rowi);
  const float zd = sd_on ? __ldcg(a.zx_d + rowi) : 0.0f;
  for (int q = lane; q < S * kRowParts; q += 32) {
    stats_merge(ct, partial_to_stats(load_partial(a.row_t + rowi * S * kRowParts + q)));
    if (sd_on) stats_merge(cd, partial_to_stats(load_partial(a.row_d + rowi * S * kRowParts + q)));
  }
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) {
    stats_merge(ct, stats_shfl_down(ct, d));
    if (sd_on) stats_merge(cd, stats_shfl_down(cd, d));
  }
  RowRes rr;
  rr.amax = ct.idx;
  rr.lse_t = greedy ? ct.best : ct.m + logf(ct.S);
  rr.zx_t = zt;
  rr.lse_q = sd_on ? cd.m + logf(cd.S) : 0.0f;
  rr.zx_d = zd;
  return rr;
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

// Statistics pass: persistent CTAs walk the row items (every drafted row of every request,
// cut into vocabulary slices) with the next item's loads in flight while the current one is
// reduced.  Per item: the online-softmax statistics (max, sum of exponentials) of the
// slice of target row j / T -- its argmax for T = 0 -- and of the draft row when no draft
// normaliser is given, and the scaled logits at the draft token in the slice that holds it.
template <int DT, bool VEC>
__global__ void __launch_bounds__(kRowThreads, kRowCtasPerSm) verify_rows(const __grid_constant__ VerifyArgs a) {
  constexpr bool kPacked = (DT == DSPARK_BF16) && VEC;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (read_status(a.dev_status)) return;
  const int S = a.row_slices;
  const int total = (int)(a.B * a.K_max) * S;
  const bool stream_d = (a.D_lse == nullptr);
  int item = blockIdx.x;
  if (item >= total) return;
  RowItem cur = row_item(a, item, tid);
  uint4 pc[kRowPk];
  if (kPacked) row_issue(a, cur, tid, pc);
  for (; item < total; item += gridDim.x) {
    const int nitem = item + gridDim.x;
    RowItem nxt;
    nxt.kind = 0;
    if (nitem < total) nxt = row_item(a, nitem, tid);
    uint4 pn[kRowPk];
    if (kPacked) row_issue(a, nxt, tid, pn);   // in flight while this item is reduced
    if (cur.kind) {
      const bool sd_on = stream_d && cur.kind == 1;
      Stats st, sd;
      stats_init(st);
      stats_init(sd);
      // the thread that holds the draft token writes its scaled logits directly
      if (kPacked && !sd_on) row_consume(cur, pc, tid, st, a.zx_t + cur.rowi);
      else row_generic<DT, VEC>(a, cur, sd_on, tid, st, sd, a.zx_t + cur.rowi, a.zx_d + cur.rowi);
      st = warp_reduce_row(st, cur.kind);
      if (sd_on) sd = warp_reduce_row(sd, 1);
      if (lane == 0) {
        const int64_t at = ((int64_t)cur.rowi * S + cur.lo / kRowSlice) * kRowParts + warp;
        a.row_t[at] = stats_to_partial(st);
        if (sd_on) a.row_d[at] = stats_to_partial(sd);
      }
    }
    cur = nxt;
#pragma unroll
    for (int q = 0; q < kRowPk; ++q) pc[q] = pn[q];
  }
}

// The accept walk of request r from its merged rows (one warp; lane j - 1 tests position
// j, the first rejection ends the walk): the sampling job, and with write_out the
// accepted tokens, the padding and n_acc.  A greedy rejection's correction (the argmax)
// is written here too.
template <int DT>
__device__ void decide_request(const VerifyArgs &a, int r, int lane, bool write_out, const RowRes *rows,
                               VerifyJob *out_job) {
  const int K = (int)a.K_max;
  const int l = a.ell[r];
  const float T = a.temperature[r];
  const bool greedy = (T == 0.0f);
  const float invT = greedy ? 1.0f : 1.0f / T;
  const int64_t off = a.tgt_off[r];
  const int j = lane + 1;
  bool reject = false;
  int amax = -1, x = -1;
  float lt = 0.0f, lq = 0.0f;
  if (j <= l) {
    const int64_t rowi = (int64_t)r * K + j - 1;
    x = a.draft_tok[rowi];
    const RowRes rr = rows[j - 1];
    amax = rr.amax;
    if (greedy) {
      reject = (x != rr.amax);
    } else {
      const float u = uniform_accept(philox(a.key, 0u, (uint32_t)j, (uint32_t)r, kTagAccept).x);
      lt = rr.lse_t;
      float lq_x;
      if (a.D_lse != nullptr) {
        lq = a.D_lse[rowi];
        lq_x = load1<DT>(a.D, rowi * a.V + x) * invT - lq;
      } else {
        lq = rr.lse_q;
        lq_x = rr.zx_d - lq;
      }
      reject = !(u < expf((rr.zx_t - lt) - lq_x));
    }
  }
  const unsigned rej = __ballot_sync(0xffffffffu, reject);
  const int n = rej ? __ffs(rej) - 1 : l;                 // accepted drafts
  const float lt_n = __shfl_sync(0xffffffffu, lt, n & 31);
  const float lq_n = __shfl_sync(0xffffffffu, lq, n & 31);
  const int amax_n = __shfl_sync(0xffffffffu, amax, n & 31);
  if (write_out && lane <= K) {
    int32_t *out = a.out_tok + (int64_t)r * (K + 1);
    if (lane < n) out[lane] = x;
    else if (lane > n) out[lane] = -1;
  }
  if (lane == 0) {
    VerifyJob job;
    job.mode = 0;
    job.pos = 0;
    job.trow = 0;
    job.drow = 0;
    job.lse_t = lt_n;
    job.lse_q = lq_n;
    job.invT = invT;
    job.out_slot = r * (K + 1) + n;
    if (rej) {
      if (greedy) {
        if (write_out) a.out_tok[(int64_t)r * (K + 1) + n] = amax_n;
      } else {
        job.mode = 1;
        job.pos = n + 1;
        job.trow = off + n;
        job.drow = (int64_t)r * K + n;
      }
    } else {
      job.mode = greedy ? 3 : 2;
      job.pos = l + 1;
      job.trow = off + l;
    }
    if (write_out) a.n_acc[r] = n;
    *out_job = job;
  }
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

// Residual weight max(0, p - q) with p = 2^(t a - lt2), q = 2^(d a - ld2).
__device__ __forceinline__ float resid_weight(float t, float d, float a, float lt2, float ld2) {
  return fmaxf(fast_ex2(fmaf(t, a, -lt2)) - fast_ex2(fmaf(d, a, -ld2)), 0.0f);
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

// brace_resid_block on packed bf16 rows: the same weights in the same order, unpacked
// one pair at a time.
template <class PickWord>
__device__ __forceinline__ void brace_resid_packed(BRace &r, const uint4 (&tp)[4], const uint4 (&dp)[4], float a,
                                                   float lt2, float ld2, uint32_t wb, int v0, bool &any_pos,
                                                   PickWord pick_word) {
  float w[kBlockW];
  float s[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
  for (int q = 0; q < kBlockW; ++q) {
    const uint32_t tw = word_of(tp[q >> 3], (q >> 1) & 3), dw = word_of(dp[q >> 3], (q >> 1) & 3);
    const float t = __uint_as_float((q & 1) ? (tw & 0xffff0000u) : (tw << 16));
    const float d = __uint_as_float((q & 1) ? (dw & 0xffff0000u) : (dw << 16));
    w[q] = resid_weight(t, d, a, lt2, ld2);
    s[q & 3] += w[q];
  }
  const float L = (s[0] + s[1]) + (s[2] + s[3]);
  if (!(L > 0.0f)) return;
  any_pos = true;
  if (brace_enter(r, fast_lg2(L) * kLn2, wb)) r.idx = v0 + pick_in_block(w, uniform_accept(pick_word()) * L);
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

template <int DT, bool VEC>
__global__ void __launch_bounds__(kSampleThreads, 2) verify_sample(const __grid_constant__ VerifyArgs a) {
  __shared__ Race red[kSampleThreads / 32];
  __shared__ int s_any[kSampleThreads / 32];
  __shared__ int s_last, s_tok;
  __shared__ VerifyJob s_job;
  __shared__ RowRes s_rows[kMaxK];
  const int cx = blockIdx.x, tid = threadIdx.x;
  if (read_status(a.dev_status)) return;
  const int K = (int)a.K_max;
  for (int r = blockIdx.y; r < (int)a.B; r += gridDim.y) {
    // every chunk merges the request's row statistics (a warp per row) and walks its
    // positions -- the same decision everywhere; chunk 0 writes the accepted tokens
    {
      const bool greedy = a.temperature[r] == 0.0f;
      const bool stream_d = (a.D_lse == nullptr);
      const int l = a.ell[r];
      for (int jw = tid >> 5; jw < l; jw += kSampleThreads / 32) {
        const RowRes rr = row_merge(a, (int64_t)r * K + jw, greedy, stream_d, tid & 31);
        if ((tid & 31) == 0) s_rows[jw] = rr;
      }
    }
    __syncthreads();
    if (tid < 32) decide_request<DT>(a, r, tid, cx == 0, s_rows, &s_job);
    __syncthreads();
    const VerifyJob job = s_job;
    __syncthreads();
    if (job.mode == 0) continue;
    const int V = (int)a.V;
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
    if (tid == 0) {
      a.out_tok[job.out_slot] = s_tok;
      a.counters[r] = 0;
    }
    __syncthreads();
  }
}

template <int DT, bool VEC>
cudaError_t launch_typed(VerifyArgs a, cudaStream_t s, int num_sms) {
  // sampling chunks: about two CTAs per SM over all requests in one wave, each chunk a
  // multiple of 32 columns (the blocks of the two-level draw) and at most a.chunks of them
  {
    const int64_t want = (2LL * num_sms) / a.B;
    const int c = (int)(want < 1 ? 1 : (want > a.chunks ? a.chunks : want));
    const int64_t per = (a.V + c - 1) / c;
    a.chunk_len = (int)((per + kBlockW - 1) / kBlockW * kBlockW);
    a.chunks = (int)((a.V + a.chunk_len - 1) / a.chunk_len);
  }
  const int64_t items = a.B * a.K_max * (int64_t)a.row_slices;
  const int64_t grid = items < (int64_t)kRowCtasPerSm * num_sms ? items : (int64_t)kRowCtasPerSm * num_sms;
  if (grid > 0) {
    verify_rows<DT, VEC><<<(unsigned)grid, kRowThreads, 0, s>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  verify_sample<DT, VEC><<<dim3(a.chunks, (unsigned)(a.B < 65535 ? a.B : 65535)), kSampleThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

int verify_row_slices(int64_t V) { return (int)((V + kRowSlice - 1) / kRowSlice); }

// Workspace layout (every part 256-byte aligned): chunk counters [B] (zeroed at the start
// of every call), sampling partials [B * chunks], slice statistics of the target and draft
// rows [B * kMaxK * slices * warps] each, scaled logits at the draft tokens [B * kMaxK] each.  Rows
// are sized for kMaxK positions so the size depends on B and V only.
size_t verify_ws_bytes(int64_t B, int64_t V, int *chunks) {
  const int c = (int)((V + kSampleUnit - 1) / kSampleUnit);   // the most chunks a call uses
  if (chunks) *chunks = c;
  auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
  const size_t rows = (size_t)B * (size_t)kMaxK;
  return al(sizeof(int32_t) * (size_t)B) + al(sizeof(Partial) * (size_t)B * (size_t)c) +
         2 * al(sizeof(Partial) * rows * verify_row_slices(V) * kRowParts) + 2 * al(sizeof(float) * rows);
}

void verify_carve(VerifyArgs &a, void *workspace) {
  auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
  const size_t rows = (size_t)a.B * (size_t)kMaxK;
  int chunks = 1;
  verify_ws_bytes(a.B, a.V, &chunks);
  a.chunks = chunks;
  a.row_slices = verify_row_slices(a.V);
  char *p = (char *)workspace;
  a.counters = (int32_t *)p;
  p += al(sizeof(int32_t) * (size_t)a.B);
  a.partials = (Partial *)p;
  p += al(sizeof(Partial) * (size_t)a.B * (size_t)chunks);
  a.row_t = (Partial *)p;
  p += al(sizeof(Partial) * rows * a.row_slices * kRowParts);
  a.row_d = (Partial *)p;
  p += al(sizeof(Partial) * rows * a.row_slices * kRowParts);
  a.zx_t = (float *)p;
  p += al(sizeof(float) * rows);
  a.zx_d = (float *)p;
}

cudaError_t launch_verify(const VerifyArgs &a, cudaStream_t s, int num_sms) {
  // arrival counters start from zero on every call (the workspace may be fresh)
  cudaError_t e0 = cudaMemsetAsync(a.counters, 0, sizeof(int32_t) * (size_t)a.B, s);
  if (e0 != cudaSuccess) return e0;
  const int esz = a.dtype == DSPARK_F32 ? 4 : 2;
  const bool vec = ((a.V * esz) % 16 == 0) && ((uintptr_t)a.tgt % 16 == 0) && ((uintptr_t)a.D % 16 == 0);
  if (a.dtype == DSPARK_F32)
    return vec ? launch_typed<DSPARK_F32, true>(a, s, num_sms) : launch_typed<DSPARK_F32, false>(a, s, num_sms);
  return vec ? launch_typed<DSPARK_BF16, true>(a, s, num_sms) : launch_typed<DSPARK_BF16, false>(a, s, num_sms);
}

}  // namespace dspark
