// Markov-head draft sampling ("DSpark", S3.1; "Speculative decoding, from zero
// to DSpark", S6): prologue and the CUDA-core step kernel.
//
// For position k the active requests (K_r >= k) form a prefix of the
// permutation `perm`, which orders requests by K_r descending; the prologue
// builds it together with the active counts nact[k].
//
// CUDA-core step: grid (vocabulary chunk, active row).  Each block loads the
// previous token's embedding row W1[x_{k-1}] into shared memory, forms
// z = U + W1[x_{k-1}] . W2 for its chunk with fp32 FMAs, rounds z to the
// storage dtype, optionally writes it, and runs the Gumbel race (or the greedy
// argmax) with the online softmax.  Block partials go to the workspace; the
// last block of a row merges them and writes the token and the log-sum-exp.
// This path serves fp32 inputs and shapes the tensor-core kernel does not take.
#include "dspark_internal.cuh"

namespace dspark {
namespace {

constexpr int kPrologueThreads = 1024;
constexpr int kSimtThreads = 256;
constexpr int kSimtChunk = 2048;   // vocabulary columns per block

__global__ void __launch_bounds__(kPrologueThreads) draft_prologue(const __grid_constant__ DraftArgs a) {
  __shared__ int s_err, s_skip;
  __shared__ int wsum[kPrologueThreads / 32];
  __shared__ int s_base;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    s_skip = read_status(a.dev_status);
    s_err = 0;
    s_base = 0;
  }
  __syncthreads();
  if (s_skip) return;
  const int B = (int)a.B, K = (int)a.K_max, V = (int)a.V;
  for (int r = tid; r < B; r += kPrologueThreads) {
    const int kr = a.K_r[r];
    if (kr < 1 || kr > K) atomicCAS(&s_err, 0, (int)DSPARK_ERR_LENGTHS);
    const int x0 = a.anchor[r];
    if (x0 < 0 || x0 >= V) atomicCAS(&s_err, 0, (int)DSPARK_ERR_TOKEN_RANGE);
    if (!temperature_ok(a.temperature[r])) atomicCAS(&s_err, 0, (int)DSPARK_ERR_TEMPERATURE);
    a.counters[r] = 0;
    for (int k = 0; k < K; ++k)
      if (k >= kr) a.draft_tok[(int64_t)r * K + k] = -1;
  }
  __syncthreads();
  if (s_err) {
    if (tid == 0) set_status(a.dev_status, s_err);
    return;
  }
  // stable order by K_r descending: one block scan per length value
  const int per = (B + kPrologueThreads - 1) / kPrologueThreads;
  const int rb = tid * per, re = min(B, rb + per);
  for (int val = K; val >= 1; --val) {
    int cnt = 0;
    for (int r = rb; r < re; ++r) cnt += (a.K_r[r] == val);
    int x = cnt;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, d);
      if (lane >= d) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    if (warp == 0) {
      int y = wsum[lane];
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int z = __shfl_up_sync(0xffffffffu, y, d);
        if (lane >= d) y += z;
      }
      wsum[lane] = y;
    }
    __syncthreads();
    int pos = s_base + (warp ? wsum[warp - 1] : 0) + x - cnt;
    for (int r = rb; r < re; ++r)
      if (a.K_r[r] == val) a.perm[pos++] = r;
    __syncthreads();
    if (tid == 0) {
      s_base += wsum[kPrologueThreads / 32 - 1];
      a.nact[val] = s_base;   // requests with K_r >= val
    }
    __syncthreads();
  }
  if (tid == 0) {
    a.nact[0] = B;
    a.nact[K + 1] = 0;
  }
}

template <int DT>
__device__ __forceinline__ float ld(const void *p, int64_t i) {
  if (DT == DSPARK_F32) return __ldg((const float *)p + i);
  return bf16_bits_to_float(__ldg((const unsigned short *)p + i));
}

template <int DT>
__device__ __forceinline__ void st_logit(void *p, int64_t i, float z) {
  if (DT == DSPARK_F32) ((float *)p)[i] = z;
  else ((__nv_bfloat16 *)p)[i] = __float2bfloat16_rn(z);
}

template <int DT>
__global__ void __launch_bounds__(kSimtThreads) draft_simt_step(const __grid_constant__ DraftArgs a, int k,
                                                                 int chunks) {
  extern __shared__ float e_s[];   // [rank]
  __shared__ Race red[kSimtThreads / 32];
  __shared__ int s_last;
  if (read_status(a.dev_status)) return;
  const int i = blockIdx.y;
  if (i >= a.nact[k]) return;
  const int K = (int)a.K_max, V = (int)a.V, rank = (int)a.rank;
  const int r = a.perm[i];
  const int prev = (k == 1) ? a.anchor[r] : a.draft_tok[(int64_t)r * K + k - 2];
  for (int q = threadIdx.x; q < rank; q += kSimtThreads) e_s[q] = ld<DT>(a.E, (int64_t)prev * rank + q);
  __syncthreads();
  const float T = a.temperature[r];
  const bool greedy = (T == 0.0f);
  const float invT = greedy ? 1.0f : 1.0f / T;
  const int64_t urow = ((int64_t)r * K + (k - 1)) * (int64_t)V;
  const int lo = blockIdx.x * kSimtChunk, hi = min(V, lo + kSimtChunk);
  Race st;
  race_init(st);
  for (int v0 = lo + threadIdx.x * 4; v0 < hi; v0 += kSimtThreads * 4) {
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    for (int q = 0; q < rank; ++q) {
      const float e = e_s[q];
      const int64_t wrow = (int64_t)q * V;
#pragma unroll
      for (int c = 0; c < 4; ++c)
        if (v0 + c < hi) acc[c] = fmaf(e, ld<DT>(a.W, wrow + v0 + c), acc[c]);
    }
    float s[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      if (v0 + c < hi) {
        float z = ld<DT>(a.U, urow + v0 + c) + acc[c];
        if (DT == DSPARK_BF16) z = round_to_bf16(z);
        if (a.draft_logits) st_logit<DT>(a.draft_logits, urow + v0 + c, z);
        s[c] = greedy ? z : z * invT;
      } else {
        s[c] = -INFINITY;
      }
    }
    if (greedy) {
      argmax_update<4>(st, s, v0);
    } else {
      const uint4 w4 = philox(a.key, (uint32_t)(v0 >> 2), (uint32_t)k, (uint32_t)r, kTagDraft);
      const uint32_t w[4] = {w4.x, w4.y, w4.z, w4.w};
      race_update<4>(st, s, w, v0);
    }
  }
  st = race_block_reduce(st, red);
  if (threadIdx.x == 0) {
    a.partials[(int64_t)i * chunks + blockIdx.x] = to_partial(st);
    __threadfence();
    s_last = (atomicAdd(&a.counters[i], 1) == chunks - 1);
  }
  __syncthreads();
  if (!s_last || threadIdx.x != 0) return;
  __threadfence();
  Race tot;
  race_init(tot);
  for (int q = 0; q < chunks; ++q)
    race_merge(tot, from_partial(load_partial(a.partials + ((int64_t)i * chunks + q))));
  a.draft_tok[(int64_t)r * K + k - 1] = tot.idx;
  if (a.draft_lse) a.draft_lse[(int64_t)r * K + k - 1] = greedy ? tot.best : tot.m + logf(tot.S);
  a.counters[i] = 0;
}

}  // namespace

cudaError_t launch_draft_prologue(const DraftArgs &a, cudaStream_t s) {
  draft_prologue<<<1, kPrologueThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_draft_simt(const DraftArgs &a, cudaStream_t s) {
  const int chunks = (int)((a.V + kSimtChunk - 1) / kSimtChunk);
  const size_t smem = sizeof(float) * (size_t)a.rank;
  if (smem > 48 * 1024) {
    cudaError_t e = a.dtype == DSPARK_F32
                        ? cudaFuncSetAttribute(draft_simt_step<DSPARK_F32>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)
                        : cudaFuncSetAttribute(draft_simt_step<DSPARK_BF16>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  for (int k = 1; k <= (int)a.K_max; ++k) {
    dim3 grid(chunks, (unsigned)a.B);
    if (a.dtype == DSPARK_F32) draft_simt_step<DSPARK_F32><<<grid, kSimtThreads, smem, s>>>(a, k, chunks);
    else draft_simt_step<DSPARK_BF16><<<grid, kSimtThreads, smem, s>>>(a, k, chunks);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace dspark
