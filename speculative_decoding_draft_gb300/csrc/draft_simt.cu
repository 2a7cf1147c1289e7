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
// storage dtype, optionally writes it, and runs the two-level draw (one 32-wide
// block per thread and iteration; or the greedy argmax) with the online softmax.  Block partials go to the workspace; the
// last block of a row merges them and writes the token and the log-sum-exp.
// This path serves fp32 inputs and shapes the tensor-core kernel does not take.
#include "dspark_internal.cuh"

namespace dspark {
namespace {

constexpr int kPrologueThreads = 1024;
constexpr int kSimtThreads = 256;

__global__ void __launch_bounds__(kPrologueThreads) draft_prologue(const __grid_constant__ DraftArgs a) {
  __shared__ int s_err, s_skip;
  __shared__ int cnt[kMaxK + 2];          // requests per length value
  __shared__ int base[kMaxK + 2];         // next free slot per length value
  __shared__ int wc[kPrologueThreads / 32][kMaxK + 2];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    s_skip = read_status(a.dev_status);
    s_err = 0;
  }
  if (tid < kMaxK + 2) cnt[tid] = 0;
  __syncthreads();
  if (s_skip) return;
  if (tid <= a.K_max) a.gbar[tid] = 0;
  const int B = (int)a.B, K = (int)a.K_max, V = (int)a.V;
  for (int r = tid; r < B; r += kPrologueThreads) {
    const int kr = a.K_r[r];
    if (kr < 1 || kr > K) atomicCAS(&s_err, 0, (int)DSPARK_ERR_LENGTHS);
    else atomicAdd(&cnt[kr], 1);
    const int x0 = a.anchor[r];
    if (x0 < 0 || x0 >= V) atomicCAS(&s_err, 0, (int)DSPARK_ERR_TOKEN_RANGE);
    if (!temperature_ok(a.temperature[r])) atomicCAS(&s_err, 0, (int)DSPARK_ERR_TEMPERATURE);
    a.counters[r] = 0;
    for (int k = 0; k < K; ++k) {
      a.best_key[(int64_t)r * K + k] = 0ull;
      if (k >= kr) {
        a.draft_tok[(int64_t)r * K + k] = -1;
        if (a.conf_out) a.conf_out[(int64_t)r * K + k] = 0.0f;
      }
    }
  }
  __syncthreads();
  if (s_err) {
    if (tid == 0) set_status(a.dev_status, s_err);
    return;
  }
  if (tid == 0) {
    int run = 0;
    for (int val = K; val >= 1; --val) {   // longest drafts first
      base[val] = run;
      run += cnt[val];
      a.nact[val] = run;                   // requests with K_r >= val
    }
    a.nact[0] = B;
    a.nact[K + 1] = 0;
  }
  __syncthreads();
  // stable scatter, 1024 requests per round: rank among equal lengths by warp match + warp prefix
  for (int c0 = 0; c0 < B; c0 += kPrologueThreads) {
    const int r = c0 + tid;
    const int v = r < B ? a.K_r[r] : 0;
    const uint32_t peers = __match_any_sync(0xffffffffu, v);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    for (int e = tid; e < (kPrologueThreads / 32) * (kMaxK + 2); e += kPrologueThreads) (&wc[0][0])[e] = 0;
    __syncthreads();
    if (lane == __ffs(peers) - 1) wc[warp][v] = __popc(peers);
    __syncthreads();
    int before = 0;
    for (int w2 = 0; w2 < warp; ++w2) before += wc[w2][v];
    if (r < B) {
      a.perm[base[v] + before + rank] = r;
      a.iperm[r] = base[v] + before + rank;
    }
    __syncthreads();
    if (tid >= 1 && tid <= K) {
      int tot = 0;
      for (int w2 = 0; w2 < kPrologueThreads / 32; ++w2) tot += wc[w2][tid];
      base[tid] += tot;
    }
    __syncthreads();
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

// RNN head cell ("DSpark" S3.1, RNN head) for position k, one block per active request:
// pre = x_k + W [s_{k-1}; W1[x_{k-1}]] (gate, candidate, output: rows 0..r-1, r..2r-1,
// 2r..3r-1), s_k = g s_{k-1} + (1 - g) tanh(candidate), feature = o s_k, with g and o the
// sigmoids of their pre-activations and s_0 = 0.  One warp per output row, lane-strided
// dot products.
template <int DT>
__global__ void __launch_bounds__(kSimtThreads) rnn_cell(const __grid_constant__ DraftArgs a, int k) {
  extern __shared__ float cell_s[];     // [2 rank] input, then [3 rank] pre-activations
  if (read_status(a.dev_status)) return;
  const int K = (int)a.K_max, rank = (int)a.rank;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = kSimtThreads / 32;
  float *zin = cell_s, *pre = cell_s + 2 * rank;
  const int n_k = a.nact[k];
  for (int i = blockIdx.x; i < n_k; i += gridDim.x) {
    const int r = a.perm[i];
    const int prev = (k == 1) ? a.anchor[r] : a.draft_tok[(int64_t)r * K + k - 2];
    __syncthreads();
    for (int q = threadIdx.x; q < rank; q += kSimtThreads) {
      zin[q] = (k == 1) ? 0.0f : a.rnn_state[(int64_t)r * rank + q];
      zin[rank + q] = ld<DT>(a.E, (int64_t)prev * rank + q);
    }
    __syncthreads();
    const float *xk = a.rnn_x + ((int64_t)r * K + (k - 1)) * 3 * rank;
    for (int j = warp; j < 3 * rank; j += nwarps) {
      float acc = 0.0f;
      for (int q = lane; q < 2 * rank; q += 32) acc = fmaf(ld<DT>(a.rnn_W, (int64_t)j * 2 * rank + q), zin[q], acc);
#pragma unroll
      for (int d = 16; d > 0; d >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, d);
      if (lane == 0) pre[j] = xk[j] + acc;
    }
    __syncthreads();
    for (int q = threadIdx.x; q < rank; q += kSimtThreads) {
      const float g = 1.0f / (1.0f + expf(-pre[q]));
      const float c = tanhf(pre[rank + q]);
      const float o = 1.0f / (1.0f + expf(-pre[2 * rank + q]));
      const float st = g * zin[q] + (1.0f - g) * c;
      a.rnn_state[(int64_t)r * rank + q] = st;
      a.rnn_feat[(int64_t)r * rank + q] = o * st;
    }
  }
}

template <int DT>
__global__ void __launch_bounds__(kSimtThreads) draft_simt_step(const __grid_constant__ DraftArgs a, int k,
                                                                 int chunks) {
  extern __shared__ float e_s[];   // [rank]
  __shared__ Race red[kSimtThreads / 32];
  __shared__ int s_last;
  if (read_status(a.dev_status)) return;
  const int K = (int)a.K_max, V = (int)a.V, rank = (int)a.rank;
  const int n_k = a.nact[k];
  const PhiloxKey key = a.key;   // round keys in registers for the hot loop
  for (int i = blockIdx.y; i < n_k; i += gridDim.y) {
    const int r = a.perm[i];
    const int prev = (k == 1) ? a.anchor[r] : a.draft_tok[(int64_t)r * K + k - 2];
    __syncthreads();
    // the head's feature: the previous token's W1 row (Markov head) or the RNN cell's output
    for (int q = threadIdx.x; q < rank; q += kSimtThreads)
      e_s[q] = a.rnn_feat ? a.rnn_feat[(int64_t)r * rank + q] : ld<DT>(a.E, (int64_t)prev * rank + q);
    __syncthreads();
    const float T = a.temperature[r];
    const bool greedy = (T == 0.0f);
    const float a2 = (greedy ? 1.0f : 1.0f / T) * kLog2e;
    const int64_t urow = ((int64_t)r * K + (k - 1)) * (int64_t)V;
    const int lo = blockIdx.x * kDraftSimtChunk, hi = min(V, lo + kDraftSimtChunk);
    BRace br;
    brace_init(br);
    // one 32-wide block of the two-level draw per thread and iteration
    for (int v0 = lo + threadIdx.x * kBlockW; v0 < hi; v0 += kSimtThreads * kBlockW) {
      float z[kBlockW];
#pragma unroll
      for (int c = 0; c < kBlockW; ++c) z[c] = 0.0f;
      for (int q = 0; q < rank; ++q) {
        const float e = e_s[q];
        const int64_t wrow = (int64_t)q * V;
#pragma unroll
        for (int c = 0; c < kBlockW; ++c)
          if (v0 + c < hi) z[c] = fmaf(e, ld<DT>(a.W, wrow + v0 + c), z[c]);
      }
#pragma unroll
      for (int c = 0; c < kBlockW; ++c) {
        if (v0 + c < hi) {
          float zz = ld<DT>(a.U, urow + v0 + c) + z[c];
          if (DT == DSPARK_BF16) zz = round_to_bf16(zz);
          if (a.draft_logits) st_logit<DT>(a.draft_logits, urow + v0 + c, zz);
          z[c] = zz;
        } else {
          z[c] = -INFINITY;
        }
      }
      const float mz = block_max(z);
      if (greedy) {
        brace_argmax_block(br, z, mz, v0);
      } else {
        const uint32_t g = (uint32_t)(v0 / kBlockW);
        const uint32_t wb = word_of(philox(key, g >> 2, (uint32_t)k, (uint32_t)r, kTagDraft), (int)(g & 3u));
        brace_softmax_block(br, z, mz, a2, wb, v0, [&] {
          return word_of(philox(key, g >> 2, (uint32_t)k, (uint32_t)r, kTagDraftPick), (int)(g & 3u));
        });
      }
    }
    Race st = from_partial(to_partial(br));
    st = race_block_reduce(st, red);
    if (threadIdx.x == 0) {
      a.partials[(int64_t)i * chunks + blockIdx.x] = to_partial(st);
      __threadfence();
      s_last = (atomicAdd(&a.counters[i], 1) == chunks - 1);
    }
    __syncthreads();
    if (s_last && threadIdx.x < 32) {
      __threadfence();
      const Partial *ptr[1] = {a.partials + (int64_t)i * chunks};
      Race tot[1];
      warp_merge_rows<1>(ptr, chunks, tot);
      if (a.conf_out) {   // the previous token's embedding row is this block's e_s
        const float c = warp_confidence([&](int q) { return e_s[q]; }, a.conf_w, rank,
                                        a.conf_h[(int64_t)r * K + k - 1], threadIdx.x);
        if (threadIdx.x == 0) a.conf_out[(int64_t)r * K + k - 1] = c;
      }
      if (threadIdx.x == 0) {
        a.draft_tok[(int64_t)r * K + k - 1] = tot[0].idx;
        if (a.draft_lse) a.draft_lse[(int64_t)r * K + k - 1] = greedy ? tot[0].best : tot[0].m + logf(tot[0].S);
        a.counters[i] = 0;
      }
    }
  }
}

}  // namespace

cudaError_t launch_draft_prologue(const DraftArgs &a, cudaStream_t s) {
  draft_prologue<<<1, kPrologueThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_draft_simt(const DraftArgs &a, cudaStream_t s) {
  const int chunks = (int)((a.V + kDraftSimtChunk - 1) / kDraftSimtChunk);
  const size_t smem = sizeof(float) * (size_t)a.rank;
  if (smem > 48 * 1024) {
    cudaError_t e = a.dtype == DSPARK_F32
                        ? cudaFuncSetAttribute(draft_simt_step<DSPARK_F32>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)
                        : cudaFuncSetAttribute(draft_simt_step<DSPARK_BF16>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  const size_t cell_smem = sizeof(float) * 5 * (size_t)a.rank;
  if (a.rnn_feat && cell_smem > 48 * 1024) {
    cudaError_t e = a.dtype == DSPARK_F32
                        ? cudaFuncSetAttribute(rnn_cell<DSPARK_F32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)cell_smem)
                        : cudaFuncSetAttribute(rnn_cell<DSPARK_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)cell_smem);
    if (e != cudaSuccess) return e;
  }
  for (int k = 1; k <= (int)a.K_max; ++k) {
    if (a.rnn_feat) {
      const unsigned cg = (unsigned)(a.B < 65535 ? a.B : 65535);
      if (a.dtype == DSPARK_F32) rnn_cell<DSPARK_F32><<<cg, kSimtThreads, cell_smem, s>>>(a, k);
      else rnn_cell<DSPARK_BF16><<<cg, kSimtThreads, cell_smem, s>>>(a, k);
      cudaError_t e = cudaGetLastError();
      if (e != cudaSuccess) return e;
    }
    dim3 grid(chunks, (unsigned)(a.B < 65535 ? a.B : 65535));
    if (a.dtype == DSPARK_F32) draft_simt_step<DSPARK_F32><<<grid, kSimtThreads, smem, s>>>(a, k, chunks);
    else draft_simt_step<DSPARK_BF16><<<grid, kSimtThreads, smem, s>>>(a, k, chunks);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace dspark
