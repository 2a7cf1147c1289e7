// Ragged rejection-sampling verification ("DSpark", S2.1; "Speculative
// decoding, from zero to DSpark", S2 and Appendix A1).
//
// Two kernels:
//  1. verify_chain: one thread-block cluster per request walks positions
//     j = 1..ell_r left to right.  Each CTA of the cluster streams its slice of
//     the target row (and of the draft row when no draft normaliser is given)
//     with 16-byte loads, reduces the online-softmax statistics (max, sum of
//     exponentials) of z/T, and publishes them in shared memory; after a
//     cluster barrier every CTA combines the slices in rank order, so all of
//     them take the same accept decision u < min(1, p(x)/q(x)).  Rows after
//     the deciding position are never read.  The decision also produces the
//     sampling job of the request: the residual at the rejecting position, the
//     bonus row when every position is accepted, or nothing for greedy
//     rejections (their correction is the argmax already found).
//  2. verify_sample: the residual / bonus two-level draw over the vocabulary,
//     spread over the whole GPU (request x vocabulary chunk, one 32-wide block
//     per thread), with the last block of each request merging the chunk
//     partials.
#include "dspark_internal.cuh"

#include <cooperative_groups.h>

namespace cg = cooperative_groups;

namespace dspark {
namespace {

constexpr int kChainThreads = 256;
constexpr int kBatch = 4;          // loads in flight per thread in the accept chain (fp32 / unaligned)
constexpr int kPkBatch = 16;       // packed bf16 16-byte loads in flight per thread
constexpr int kSampleThreads = 256;
constexpr int kSampleChunk = kSampleThreads * kBlockW;   // one 32-wide block per thread

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

// Block reduction; result valid in thread 0.
__device__ __forceinline__ Stats stats_block_reduce(Stats s, Stats *scratch) {
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) stats_merge(s, stats_shfl_down(s, d));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) scratch[warp] = s;
  __syncthreads();
  if (threadIdx.x == 0)
    for (int i = 1; i < (int)(blockDim.x >> 5); ++i) stats_merge(s, scratch[i]);
  __syncthreads();
  return s;
}

struct ChainShared {
  Stats slot_t[2];          // this CTA's target-row statistics (double-buffered by position parity)
  Stats slot_d[2];          // draft-row statistics when no normaliser is given
  float zx_t[2], zx_d[2];   // scaled logit at the draft token, valid in the CTA whose slice holds it
  Stats red[kChainThreads / 32];
  int tok[kMaxK];
  float own_t, own_d;       // written by the thread that streams the draft token's element
  int skip;
  int decision;             // 1 accept, 0 reject
  int amax;
  float lse_t, lse_q;
};

// Slice [lo, hi) of the vocabulary owned by cluster rank `rank` (8-aligned).
__device__ __forceinline__ int slice_per(int V, int ncta) { return ((V + ncta - 1) / ncta + 7) & ~7; }

__device__ __forceinline__ float pick8(const float (&x)[8], int q) {
  float v = x[0];
#pragma unroll
  for (int i = 1; i < 8; ++i)
    if (i == q) v = x[i];
  return v;
}

template <int DT, bool VEC>
__global__ void __launch_bounds__(kChainThreads, 2) verify_chain(const __grid_constant__ VerifyArgs a) {
  __shared__ ChainShared sh;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int ncta = (int)cluster.num_blocks();
  const int r = blockIdx.x / ncta;
  const int tid = threadIdx.x;
  const int V = (int)a.V, K = (int)a.K_max;

  // rank 0 decides for the whole cluster whether an earlier error stops the work
  if (rank == 0 && tid == 0) sh.skip = read_status(a.dev_status);
  cluster.sync();
  const int skip = *cluster.map_shared_rank(&sh.skip, 0);
  if (skip) { cluster.sync(); return; }

  // -- validation (identical in every CTA of the cluster) --------------------
  const int l = a.ell[r];
  const float T = a.temperature[r];
  int err = 0;
  if (l < 0 || l > K) err = DSPARK_ERR_LENGTHS;
  else if (a.tgt_off[r + 1] - a.tgt_off[r] != l + 1 || (r == 0 && a.tgt_off[0] != 0)) err = DSPARK_ERR_OFFSETS;
  else if (!temperature_ok(T)) err = DSPARK_ERR_TEMPERATURE;
  else
    for (int j = 0; j < l; ++j) {
      const int x = a.draft_tok[(int64_t)r * K + j];
      if (x < 0 || x >= V) { err = DSPARK_ERR_TOKEN_RANGE; break; }
    }
  if (err) {
    if (rank == 0 && tid == 0) set_status(a.dev_status, err);
    cluster.sync();
    return;
  }
  if (tid < l) sh.tok[tid] = a.draft_tok[(int64_t)r * K + tid];

  const bool greedy = (T == 0.0f);
  const float invT = greedy ? 1.0f : 1.0f / T;
  const int64_t off = a.tgt_off[r];
  const bool have_lse = (a.D_lse != nullptr);
  const bool stream_d = !greedy && !have_lse;
  const int per = slice_per(V, ncta);
  const int lo = min(V, rank * per), hi = min(V, lo + per);
  __syncthreads();

  int n = 0;
  bool rejected = false;
  int rej_j = 0;
  float lse_t = 0.0f, lse_q = 0.0f;
  int greedy_tok = -1;
  for (int j = 1; j <= l; ++j) {
    const int x = sh.tok[j - 1];
    const int64_t trow = (off + j - 1) * (int64_t)V;
    const int64_t drow = ((int64_t)r * K + j - 1) * (int64_t)V;
    // values only thread 0 needs, requested before the row stream so their latency overlaps it
    float u = 0.0f, dx = 0.0f, lq_given = 0.0f;
    if (tid == 0 && !greedy) {
      u = uniform_accept(philox(a.key, 0u, (uint32_t)j, (uint32_t)r, kTagAccept).x);
      if (have_lse) {
        dx = load1<DT>(a.D, drow + x);
        lq_given = a.D_lse[(int64_t)r * K + j - 1];
      }
    }
    const int xv = x & ~7;   // start of the 8-element group holding x
    Stats st, sd;
    stats_init(st);
    stats_init(sd);
    if (DT == DSPARK_BF16 && VEC) {
      // bf16 rows: keep kPkBatch packed 16-byte loads per thread in flight, unpack when consumed
      const int nb = stream_d ? kPkBatch / 2 : kPkBatch;
      for (int base = lo + tid * 8; base < hi; base += kChainThreads * 8 * nb) {
        uint4 pt[kPkBatch];
#pragma unroll
        for (int uu = 0; uu < kPkBatch; ++uu) {
          const int v0 = base + uu * kChainThreads * 8;
          const bool in = (uu < nb) && (v0 + 8 <= hi);
          pt[uu] = in ? __ldcs((const uint4 *)((const unsigned short *)a.tgt + trow + v0)) : make_uint4(0, 0, 0, 0);
        }
        uint4 pd[kPkBatch / 2];
        if (stream_d) {
#pragma unroll
          for (int uu = 0; uu < kPkBatch / 2; ++uu) {
            const int v0 = base + uu * kChainThreads * 8;
            pd[uu] = (v0 + 8 <= hi) ? __ldcs((const uint4 *)((const unsigned short *)a.D + drow + v0))
                                    : make_uint4(0, 0, 0, 0);
          }
        }
#pragma unroll
        for (int uu = 0; uu < kPkBatch; ++uu) {
          const int v0 = base + uu * kChainThreads * 8;
          if (uu >= nb || v0 + 8 > hi) continue;
          float x8[8];
          const uint32_t w4[4] = {pt[uu].x, pt[uu].y, pt[uu].z, pt[uu].w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            x8[2 * i] = __uint_as_float(w4[i] << 16);
            x8[2 * i + 1] = __uint_as_float(w4[i] & 0xffff0000u);
          }
          if (greedy) {
            argmax_add8(st, x8, v0);
            continue;
          }
#pragma unroll
          for (int q = 0; q < 8; ++q) x8[q] *= invT;
          if (v0 == xv) sh.own_t = pick8(x8, x & 7);
          stats_add8(st, x8);
          if (stream_d && uu < kPkBatch / 2) {
            float y8[8];
            const uint32_t d4[4] = {pd[uu].x, pd[uu].y, pd[uu].z, pd[uu].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              y8[2 * i] = __uint_as_float(d4[i] << 16) * invT;
              y8[2 * i + 1] = __uint_as_float(d4[i] & 0xffff0000u) * invT;
            }
            if (v0 == xv) sh.own_d = pick8(y8, x & 7);
            stats_add8(sd, y8);
          }
        }
      }
    } else {
      // kBatch 16-byte loads per thread are issued before any of them is consumed
      for (int base = lo + tid * 8; base < hi; base += kChainThreads * 8 * kBatch) {
        float x8[kBatch][8];
#pragma unroll
        for (int uu = 0; uu < kBatch; ++uu) load8<DT, VEC>(a.tgt, trow, base + uu * kChainThreads * 8, hi, x8[uu]);
        if (greedy) {
#pragma unroll
          for (int uu = 0; uu < kBatch; ++uu) argmax_add8(st, x8[uu], base + uu * kChainThreads * 8);
          continue;
        }
        float y8[kBatch][8];
        if (stream_d) {
#pragma unroll
          for (int uu = 0; uu < kBatch; ++uu) load8<DT, VEC>(a.D, drow, base + uu * kChainThreads * 8, hi, y8[uu]);
        }
#pragma unroll
        for (int uu = 0; uu < kBatch; ++uu) {
          const int v0 = base + uu * kChainThreads * 8;
#pragma unroll
          for (int q = 0; q < 8; ++q) x8[uu][q] *= invT;
          if (v0 == xv) sh.own_t = pick8(x8[uu], x & 7);
          stats_add8(st, x8[uu]);
          if (stream_d) {
#pragma unroll
            for (int q = 0; q < 8; ++q) y8[uu][q] *= invT;
            if (v0 == xv) sh.own_d = pick8(y8[uu], x & 7);
            stats_add8(sd, y8[uu]);
          }
        }
      }
    }
    st = stats_block_reduce(st, sh.red);
    if (stream_d) sd = stats_block_reduce(sd, sh.red);
    if (tid == 0) {
      sh.slot_t[j & 1] = st;
      sh.slot_d[j & 1] = sd;
      const bool mine = (x >= lo && x < hi);
      sh.zx_t[j & 1] = mine ? sh.own_t : 0.0f;
      sh.zx_d[j & 1] = mine ? sh.own_d : 0.0f;
    }
    cluster.sync();
    if (tid == 0) {
      Stats parts_t[8], parts_d[8];
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (q < ncta) {
          parts_t[q] = *cluster.map_shared_rank(&sh.slot_t[j & 1], q);
          if (stream_d) parts_d[q] = *cluster.map_shared_rank(&sh.slot_d[j & 1], q);
        }
      Stats ct, cd;
      stats_init(ct);
      stats_init(cd);
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (q < ncta) {
          stats_merge(ct, parts_t[q]);
          if (stream_d) stats_merge(cd, parts_d[q]);
        }
      if (greedy) {
        sh.decision = (x == ct.idx);
        sh.amax = ct.idx;
      } else {
        const int owner = x / per;
        const float sx = *cluster.map_shared_rank(&sh.zx_t[j & 1], owner);
        const float lt = ct.m + logf(ct.S);
        float lq_x;
        if (have_lse) {
          lq_x = dx * invT - lq_given;
          sh.lse_q = lq_given;
        } else {
          const float sdx = *cluster.map_shared_rank(&sh.zx_d[j & 1], owner);
          const float ld = cd.m + logf(cd.S);
          lq_x = sdx - ld;
          sh.lse_q = ld;
        }
        sh.decision = u < expf((sx - lt) - lq_x);
        sh.lse_t = lt;
      }
    }
    __syncthreads();
    if (!sh.decision) {
      rejected = true;
      rej_j = j;
      lse_t = sh.lse_t;
      lse_q = sh.lse_q;
      greedy_tok = sh.amax;
      break;
    }
    if (rank == 0 && tid == 0) a.out_tok[(int64_t)r * (K + 1) + n] = x;
    ++n;
  }

  if (rank == 0 && tid == 0) {
    a.n_acc[r] = n;
    for (int q = n + 1; q <= K; ++q) a.out_tok[(int64_t)r * (K + 1) + q] = -1;
    VerifyJob job;
    job.mode = 0;
    job.pos = 0;
    job.trow = 0;
    job.drow = 0;
    job.lse_t = lse_t;
    job.lse_q = lse_q;
    job.invT = invT;
    job.out_slot = r * (K + 1) + n;
    if (rejected) {
      if (greedy) {
        a.out_tok[(int64_t)r * (K + 1) + n] = greedy_tok;
      } else {
        job.mode = 1;
        job.pos = rej_j;
        job.trow = off + rej_j - 1;
        job.drow = (int64_t)r * K + rej_j - 1;
      }
    } else {
      job.mode = greedy ? 3 : 2;
      job.pos = l + 1;
      job.trow = off + l;
    }
    a.jobs[r] = job;
    a.counters[r] = 0;
  }
  cluster.sync();   // peers may still read this CTA's slots
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
      brace_softmax_block(rc, t, block_max(t), a2, wb, v0, pick_word);
      continue;
    }
    float d[kBlockW];
    load32<DT, VEC>(a.D, drow, v0, hi, d);
    brace_resid_block(rc, t, d, a2, lt2, ld2, wb, v0, any_pos, pick_word);
  }
}

template <int DT, bool VEC>
__global__ void __launch_bounds__(kSampleThreads) verify_sample(const __grid_constant__ VerifyArgs a) {
  __shared__ Race red[kSampleThreads / 32];
  __shared__ int s_any[kSampleThreads / 32];
  __shared__ int s_last, s_tok;
  const int cx = blockIdx.x, tid = threadIdx.x;
  if (read_status(a.dev_status)) return;
  for (int r = blockIdx.y; r < (int)a.B; r += gridDim.y) {
    const VerifyJob job = a.jobs[r];
    if (job.mode == 0) continue;
    const int V = (int)a.V;
    const int lo = min(V, cx * kSampleChunk), hi = min(V, lo + kSampleChunk);
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
cudaError_t launch_typed(const VerifyArgs &a, cudaStream_t s, int num_sms) {
  int cl = 1;
  const int64_t target = 2LL * num_sms;
  while (cl < 8 && a.B * cl * 2 <= target) cl *= 2;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(a.B * cl), 1, 1);
  cfg.blockDim = dim3(kChainThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cl;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, verify_chain<DT, VEC>, a);
  if (e != cudaSuccess) return e;
  verify_sample<DT, VEC><<<dim3(a.chunks, (unsigned)(a.B < 65535 ? a.B : 65535)), kSampleThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

size_t verify_ws_bytes(int64_t B, int64_t V, int *chunks) {
  const int c = (int)((V + kSampleChunk - 1) / kSampleChunk);
  if (chunks) *chunks = c;
  auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
  return al(sizeof(VerifyJob) * (size_t)B) + al(sizeof(int32_t) * (size_t)B) +
         al(sizeof(Partial) * (size_t)B * (size_t)c);
}

cudaError_t launch_verify(const VerifyArgs &a, cudaStream_t s, int num_sms) {
  const int esz = a.dtype == DSPARK_F32 ? 4 : 2;
  const bool vec = ((a.V * esz) % 16 == 0) && ((uintptr_t)a.tgt % 16 == 0) && ((uintptr_t)a.D % 16 == 0);
  if (a.dtype == DSPARK_F32)
    return vec ? launch_typed<DSPARK_F32, true>(a, s, num_sms) : launch_typed<DSPARK_F32, false>(a, s, num_sms);
  return vec ? launch_typed<DSPARK_BF16, true>(a, s, num_sms) : launch_typed<DSPARK_BF16, false>(a, s, num_sms);
}

}  // namespace dspark
