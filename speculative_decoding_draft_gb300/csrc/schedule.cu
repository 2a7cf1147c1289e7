// Hardware-aware prefix scheduler ("DSpark", S3.2.2, Algorithm 1;
// "Speculative decoding, from zero to DSpark", S8) in one thread block.
//
// The candidate pool holds at most B * K_max entries (14 336 for the largest
// benchmark configuration) and the walk is inherently sequential, so one
// 1024-thread block does the whole computation: survival products, a stable
// compaction of the candidates in position-major order, a stable LSD radix sort
// by descending survival (which breaks ties by position, then request), an
// exact fixed-point prefix sum of the survivals, the objective
// Theta_i = tau_i * SPS(R + i) in fp64 with explicitly rounded operations, and
// the first decline.  Every step is deterministic, so the lengths agree bit
// for bit with a sequential evaluation of Algorithm 1 in the same arithmetic.
// Pools whose working arrays fit in about 160 KB are kept in shared memory.
//
// The same kernel serves the deployed scheduler of "DSpark" S5.2 (tutorial S9):
// the capacity mode takes the global maximum of Theta along the greedy path
// (no early stop; the first maximum on ties), and the top-K mode admits the first
// min(capacity, N) candidates of the current ranking without any SPS lookup.
// The static-threshold modes (the prior methods of S3.2.2, the sweep of S4.3.3)
// need no ranking: each request's length is the longest prefix whose
// confidences, or survival products, reach the threshold.
#include "schedule.cuh"

namespace dspark {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
// Candidate pools up to this many bytes of working arrays live in shared memory (one
// block, so every phase then exchanges data through shared memory instead of L2 round
// trips); larger pools use the global workspace.
constexpr size_t kSmemPoolMax = 160 * 1024;

struct SchedWs {
  uint32_t *keyA, *keyB, *idxA, *idxB;
  uint64_t *tfix;
  double *theta;
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

__host__ __device__ inline SchedWs carve(void *base, int64_t nc) {
  char *p = (char *)base;
  SchedWs w;
  const size_t u32 = align256((size_t)nc * 4), u64 = align256((size_t)nc * 8);
  w.keyA = (uint32_t *)p; p += u32;
  w.keyB = (uint32_t *)p; p += u32;
  w.idxA = (uint32_t *)p; p += u32;
  w.idxB = (uint32_t *)p; p += u32;
  w.tfix = (uint64_t *)p; p += u64;
  w.theta = (double *)p;
  return w;
}

// Exclusive scan of one value per thread over the block; *total gets the sum.
template <typename T>
__device__ T block_exclusive_scan(T v, T *warp_sums, T *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  T x = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    T y = __shfl_up_sync(0xffffffffu, x, d);
    if (lane >= d) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    T y = warp_sums[lane];
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      T z = __shfl_up_sync(0xffffffffu, y, d);
      if (lane >= d) y += z;
    }
    warp_sums[lane] = y;
  }
  __syncthreads();
  const T prefix = warp > 0 ? warp_sums[warp - 1] : (T)0;
  *total = warp_sums[kWarps - 1];
  __syncthreads();
  return prefix + x - v;
}

// ell -> tgt_off (exclusive scan of ell + 1); returns the number of verified draft tokens.
__device__ int64_t write_offsets(const ScheduleArgs &a, uint32_t *wsum32) {
  const int tid = threadIdx.x;
  const int64_t B = a.B;
  const int64_t per_r = (B + kThreads - 1) / kThreads;
  const int64_t rb = tid * per_r, re = min(B, rb + per_r);
  uint32_t lsum = 0;
  for (int64_t r = rb; r < re; ++r) lsum += (uint32_t)a.ell[r] + 1u;
  uint32_t tot;
  uint32_t o = block_exclusive_scan<uint32_t>(lsum, wsum32, &tot);
  for (int64_t r = rb; r < re; ++r) {
    a.tgt_off[r] = (int32_t)o;
    o += (uint32_t)a.ell[r] + 1u;
  }
  if (tid == 0) a.tgt_off[B] = (int32_t)tot;
  return (int64_t)tot - B;
}

__global__ void __launch_bounds__(kThreads, 1) schedule_kernel(const __grid_constant__ ScheduleArgs a, int in_smem) {
  extern __shared__ __align__(256) uint8_t pool[];
  __shared__ uint32_t hist[kWarps][257];
  __shared__ uint32_t wsum32[kWarps];
  __shared__ unsigned long long wsum64[kWarps];
  __shared__ int s_err, s_stop, s_skip;
  __shared__ double s_wmax[kWarps];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int mode = a.mode;
  const bool by_threshold = mode == kSchedThresholdConf || mode == kSchedThresholdSurv;
  if (tid == 0) {
    s_skip = read_status(a.dev_status);
    s_err = 0;
    s_stop = INT32_MAX;
  }
  __syncthreads();
  if (s_skip) return;
  const int64_t B = a.B, K = a.K_max, NC = B * K;
  SchedWs w = carve(in_smem ? (void *)pool : a.ws, NC);
  float *surv_slot = (float *)w.keyB;   // survival in position-major slot order, reused later

  // -- validation, survival products, zeroed lengths ------------------------
  for (int64_t r = tid; r < B; r += kThreads) {
    const int kr = a.K_r[r];
    if (a.ell) a.ell[r] = 0;
    if (kr < 1 || kr > K) {
      atomicCAS(&s_err, 0, (int)DSPARK_ERR_LENGTHS);
      continue;
    }
    // the row's confidences are requested together, then multiplied in order
    float cr[kMaxK];
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) cr[j] = (j < kr) ? a.conf[r * K + j] : 0.0f;
    float s = 1.0f;
    int len = 0;
    bool open = true;
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
      if (j >= K) break;
      float v = 0.0f;
      if (j < kr) {
        const float c = cr[j];
        if (!(c >= 0.0f && c <= 1.0f)) atomicCAS(&s_err, 0, (int)DSPARK_ERR_CONFIDENCE);
        s = __fmul_rn(s, c);
        v = s;
        // threshold modes: the prefix ends at the first position that fails (or has a = 0)
        const float tested = mode == kSchedThresholdConf ? c : s;
        if (open && s > 0.0f && tested >= a.threshold) len = j + 1;
        else open = false;
      }
      if (!by_threshold) surv_slot[j * B + r] = v;
      if (a.survival) a.survival[r * K + j] = v;
    }
    if (by_threshold) a.ell[r] = len;
  }
  __syncthreads();
  if (s_err) {
    if (tid == 0) set_status(a.dev_status, s_err);
    return;
  }
  if (by_threshold) {
    const int64_t admitted = write_offsets(a, wsum32);
    if (tid == 0 && a.b_star) *a.b_star = B + admitted;
    return;
  }

  // -- stable compaction of candidates (a > 0) in slot order (j-major) -------
  const int64_t per = (NC + kThreads - 1) / kThreads;
  const int64_t beg = tid * per, end = min(NC, beg + per);
  uint32_t cnt = 0;
  for (int64_t i = beg; i < end; ++i) cnt += surv_slot[i] > 0.0f;
  uint32_t N;
  uint32_t pos = block_exclusive_scan<uint32_t>(cnt, wsum32, &N);
  for (int64_t i = beg; i < end; ++i) {
    const float v = surv_slot[i];
    if (v > 0.0f) {
      w.keyA[pos] = ~__float_as_uint(v);    // ascending order of ~bits = descending survival
      w.idxA[pos] = (uint32_t)i;
      ++pos;
    }
  }
  if (mode != kSchedTopK && a.sps_len < B + (int64_t)N + 1) {
    if (tid == 0) set_status(a.dev_status, DSPARK_ERR_SPS_TOO_SHORT);
    return;
  }
  int64_t cap_in = 0;
  if (mode == kSchedTopK) {
    cap_in = *a.capacity_in;
    if (cap_in < 0) {
      if (tid == 0) set_status(a.dev_status, DSPARK_ERR_LENGTHS);
      return;
    }
  }
  __syncthreads();

  uint32_t *sk = w.keyA, *si = w.idxA, *dk = w.keyB, *di = w.idxB;
  // -- stable LSD radix sort, 4 passes of 8 bits -----------------------------
  const uint32_t per_w = (N + kWarps - 1) / kWarps;
  const uint32_t wb = warp * per_w, we = min(N, wb + per_w);
  for (int sh = 0; sh < 32; sh += 8) {
    for (int e = tid; e < kWarps * 257; e += kThreads) (&hist[0][0])[e] = 0;
    __syncthreads();
    for (uint32_t base = wb; base < we; base += 32) {
      const uint32_t i = base + lane;
      const bool valid = i < we;
      const uint32_t d = valid ? (sk[i] >> sh) & 255u : 256u;
      const uint32_t peers = __match_any_sync(0xffffffffu, d);
      if (valid && lane == __ffs(peers) - 1) hist[warp][d] += __popc(peers);
    }
    __syncthreads();
    // exclusive scan over (digit, warp) in digit-major order: 8192 entries, 8 per thread
    {
      uint32_t loc[8], sum = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int e = tid * 8 + q, d = e >> 5, ww = e & 31;
        loc[q] = hist[ww][d];
        sum += loc[q];
      }
      uint32_t tot;
      uint32_t run = block_exclusive_scan<uint32_t>(sum, wsum32, &tot);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int e = tid * 8 + q, d = e >> 5, ww = e & 31;
        hist[ww][d] = run;
        run += loc[q];
      }
    }
    __syncthreads();
    for (uint32_t base = wb; base < we; base += 32) {
      const uint32_t i = base + lane;
      const bool valid = i < we;
      const uint32_t key = valid ? sk[i] : 0u;
      const uint32_t d = valid ? (key >> sh) & 255u : 256u;
      const uint32_t peers = __match_any_sync(0xffffffffu, d);
      const uint32_t rank = __popc(peers & ((1u << lane) - 1u));
      uint32_t dst = 0;
      if (valid) dst = hist[warp][d] + rank;
      __syncwarp();
      if (valid) {
        dk[dst] = key;
        di[dst] = si[i];
        if (lane == __ffs(peers) - 1) hist[warp][d] += __popc(peers);
      }
      __syncwarp();
    }
    __syncthreads();
    uint32_t *t;
    t = sk; sk = dk; dk = t;
    t = si; si = di; di = t;
  }
  // after 4 passes the sorted data is back in keyA / idxA

  int64_t admitted = 0;
  if (mode == kSchedTopK) {
    admitted = min(cap_in, (int64_t)N);
  } else {
    // -- exact fixed-point prefix of survivals and the objective ---------------
    const uint32_t per_t = (N + kThreads - 1) / kThreads;
    const uint32_t tb = tid * per_t, te = min(N, tb + per_t);
    unsigned long long loc = 0;
    for (uint32_t i = tb; i < te; ++i) {
      const float av = __uint_as_float(~sk[i]);
      const unsigned long long t = __double2ull_rn((double)av * 0x1p40);
      w.tfix[i] = t;
      loc += t;
    }
    unsigned long long totT;
    unsigned long long run = block_exclusive_scan<unsigned long long>(loc, wsum64, &totT);
    const double R = (double)B;
    for (uint32_t i = tb; i < te; ++i) {
      run += w.tfix[i];
      const double tau = __dadd_rn(R, __dmul_rn(__ull2double_rn(run), 0x1p-40));
      w.theta[i + 1] = __dmul_rn(tau, a.sps[B + i + 1]);
    }
    if (tid == 0) w.theta[0] = __dmul_rn(R, a.sps[B]);
    __syncthreads();
    if (mode == kSchedAlgorithm1) {
      // first i in 1..N with Theta_i <= Theta_{i-1}
      int my_stop = INT32_MAX;
      for (uint32_t i = tb; i < te; ++i) {
        if (!(w.theta[i + 1] > w.theta[i])) { my_stop = (int)(i + 1); break; }
      }
      if (my_stop != INT32_MAX) atomicMin(&s_stop, my_stop);
      __syncthreads();
      admitted = (s_stop == INT32_MAX) ? (int64_t)N : (int64_t)s_stop - 1;
    } else {
      // capacity: the first i in 0..N with the largest Theta_i (values compared exactly)
      double best = -INFINITY;
      int best_i = INT32_MAX;
      if (tid == 0) { best = w.theta[0]; best_i = 0; }
      for (uint32_t i = tb; i < te; ++i) {
        const double th = w.theta[i + 1];
        if (th > best) { best = th; best_i = (int)(i + 1); }
      }
      double m = best;
#pragma unroll
      for (int d = 16; d > 0; d >>= 1) m = fmax(m, __shfl_xor_sync(0xffffffffu, m, d));
      if (lane == 0) s_wmax[warp] = m;
      __syncthreads();
      m = s_wmax[0];
      for (int q = 1; q < kWarps; ++q) m = fmax(m, s_wmax[q]);
      if (best == m && best_i != INT32_MAX) atomicMin(&s_stop, best_i);
      __syncthreads();
      admitted = s_stop;
    }
  }

  // -- lengths and offsets ----------------------------------------------------
  if (a.ell) {
    for (int64_t i = tid; i < admitted; i += kThreads) atomicAdd(&a.ell[si[i] % (uint32_t)B], 1);
    __syncthreads();
    if (a.tgt_off) write_offsets(a, wsum32);
  }
  if (tid == 0) {
    if (a.theta_best && mode != kSchedTopK) *a.theta_best = w.theta[admitted];
    if (a.b_star) *a.b_star = B + admitted;
    if (a.capacity_out) *a.capacity_out = (int32_t)admitted;
  }
}

}  // namespace

size_t schedule_ws_bytes(int64_t B, int64_t K_max) {
  const int64_t nc = B * K_max;
  return 4 * align256((size_t)nc * 4) + align256((size_t)nc * 8) + align256((size_t)(nc + 1) * 8);
}

cudaError_t launch_schedule(const ScheduleArgs &a, cudaStream_t s) {
  if (a.mode == kSchedThresholdConf || a.mode == kSchedThresholdSurv) {
    schedule_kernel<<<1, kThreads, 0, s>>>(a, 0);   // no ranking, no working arrays
    return cudaGetLastError();
  }
  const size_t pool_bytes = schedule_ws_bytes(a.B, a.K_max);
  const bool in_smem = pool_bytes <= kSmemPoolMax;
  if (in_smem) {
    cudaError_t e = ensure_dynamic_smem((const void *)schedule_kernel, (int)kSmemPoolMax);
    if (e != cudaSuccess) return e;
  }
  schedule_kernel<<<1, kThreads, in_smem ? pool_bytes : 0, s>>>(a, in_smem ? 1 : 0);
  return cudaGetLastError();
}

}  // namespace dspark
