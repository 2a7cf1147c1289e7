// Markov-head draft sampling ("DSpark", S3.1; "Speculative decoding, from zero
// to DSpark", S6): prologue and the CUDA-core step kernel.
//
// For position k the active requests (K_r >= k) form a prefix of the
// permutation `perm`, which orders requests by K_r descending; the prologue
// builds it together with the active counts nact[k].
//
// CUDA-core step: grid (vocabulary tile, tile of active rows); each block forms
// z = U + feature . W2 for its rows and columns with fp32 FMAs (the feature is the
// previous token's W1 row, or the RNN head's cell output), rounds z to the storage
// dtype, optionally writes it, and runs the two-level draw (one 32-wide block per
// thread; or the greedy argmax) with the online softmax.  Tile partials go to the
// workspace; the last tile of a row merges them and writes the token and the
// log-sum-exp.  This path serves fp32 inputs, the RNN head and shapes the
// tensor-core kernel does not take.
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
// sigmoids of their pre-activations and s_0 = 0.  Each warp takes four output rows at a
// time; with 16-byte aligned weight rows (VEC) every lane reads eight consecutive weights of
// each row per 16-byte load, all four rows' loads in flight together, otherwise lane-strided
// scalar loads.
template <int DT, bool VEC>
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
    const int n_in = 2 * rank, n_out = 3 * rank;
    for (int j0 = warp * 4; j0 < n_out; j0 += nwarps * 4) {
      float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      if (VEC) {
        constexpr int kPer = 16 / (DT == DSPARK_F32 ? 4 : 2);     // weights per 16-byte load
        for (int q = lane * 8; q < n_in; q += 32 * 8) {            // eight inputs per lane and step
          uint4 w[4][8 / kPer];
#pragma unroll
          for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int h = 0; h < 8 / kPer; ++h)
              w[u][h] = (j0 + u < n_out)
                            ? __ldg((const uint4 *)((const char *)a.rnn_W +
                                                    ((int64_t)(j0 + u) * n_in + q + h * kPer) * (DT == DSPARK_F32 ? 4 : 2)))
                            : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            float wv[8];
#pragma unroll
            for (int h = 0; h < 8 / kPer; ++h) {
              const uint32_t w4[4] = {w[u][h].x, w[u][h].y, w[u][h].z, w[u][h].w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                if (DT == DSPARK_F32) {
                  wv[h * 4 + e] = __uint_as_float(w4[e]);
                } else {
                  wv[2 * e] = __uint_as_float(w4[e] << 16);
                  wv[2 * e + 1] = __uint_as_float(w4[e] & 0xffff0000u);
                }
              }
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[u] = fmaf(wv[e], zin[q + e], acc[u]);
          }
        }
      } else {
        for (int q = lane; q < n_in; q += 32)
#pragma unroll
          for (int u = 0; u < 4; ++u)
            if (j0 + u < n_out) acc[u] = fmaf(ld<DT>(a.rnn_W, (int64_t)(j0 + u) * n_in + q), zin[q], acc[u]);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) acc[u] += __shfl_xor_sync(0xffffffffu, acc[u], d);
        if (lane == 0 && j0 + u < n_out) pre[j0 + u] = xk[j0 + u] + acc[u];
      }
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

// CUDA-core step for position k: one block per tile of kTileRows active rows x kTileCols
// vocabulary columns.  The rows' features (the previous tokens' W1 rows, or the RNN cell's
// output) and W2 are staged through shared memory kRankChunk rank values at a time, and each
// thread accumulates one 32-wide block of one row in registers with fp32 FMAs in ascending
// rank order, so W2 is read once per row tile instead of once per request.  Then, per
// element, U is added, the sum rounded to the storage dtype (and stored), and the two-level
// draw (or the greedy argmax) runs over the block with the online softmax.  The eight blocks
// of a row merge by shuffles into one partial per tile; the last tile of a row merges the
// row's partials and writes the token, the log-sum-exp and, when asked for, the confidence.
constexpr int kTileRows = 32;
constexpr int kTileCols = kSimtThreads / kTileRows * kBlockW;   // 256
constexpr int kRankChunk = 32;
constexpr int kBlocksPerRow = kTileCols / kBlockW;              // 8 threads per row
static_assert(kTileCols == kDraftSimtChunk, "partial slots are sized by kDraftSimtChunk");

// W2 chunk in shared memory: row q of kTileCols floats; inside each 32-column block the
// 16-byte chunk j sits at position j ^ (block & 7), so the eight blocks that the lanes of a
// warp read at one time fall in distinct banks.
__device__ __forceinline__ int wsw(int q, int col) {
  const int b = col >> 5, j = (col >> 2) & 7;
  return q * kTileCols + b * 32 + ((j ^ (b & 7)) << 2) + (col & 3);
}

template <int DT, bool VEC>
__global__ void __launch_bounds__(kSimtThreads) draft_simt_tile(const __grid_constant__ DraftArgs a, int k,
                                                                 int col_tiles) {
  // GEMM layout: thread (ty, tx) accumulates rows 4 ty .. 4 ty + 3 x columns 8 tx .. 8 tx + 7
  // (three 16-byte shared loads per 32 FMAs); the tile then goes through shared memory
  // (swizzled like the W2 chunks) to the epilogue layout, one 32-wide block per thread.
  __shared__ __align__(16) float w_s[kRankChunk * kTileCols];   // W2 chunk, later the bias tile
  __shared__ __align__(16) float f_s[kRankChunk][kTileRows];     // feature chunk, [rank][row]
  __shared__ int s_row_r[kTileRows], s_row_prev[kTileRows];
  static_assert(kRankChunk == kTileRows, "the bias tile reuses the W2 chunk buffer");
  if (read_status(a.dev_status)) return;
  const int K = (int)a.K_max, rank = (int)a.rank;
  const int64_t V = a.V;
  const int n_k = a.nact[k];
  const int i0 = blockIdx.y * kTileRows;
  if (i0 >= n_k) return;
  const int tid = threadIdx.x, lane = tid & 31;
  const int tr = tid / kBlocksPerRow, tb = tid % kBlocksPerRow;   // epilogue layout
  const int ty = tid >> 5, tx = tid & 31;                          // GEMM layout
  const int c0 = blockIdx.x * kTileCols;
  if (tid < kTileRows) {
    const int i = i0 + tid;
    const int r = i < n_k ? a.perm[i] : -1;
    s_row_r[tid] = r;
    s_row_prev[tid] = r < 0 ? 0 : ((k == 1) ? a.anchor[r] : a.draft_tok[(int64_t)r * K + k - 2]);
  }
  __syncthreads();
  const int r = s_row_r[tr];
  const bool valid = r >= 0;
  float acc[4][8];
#pragma unroll
  for (int y = 0; y < 4; ++y)
#pragma unroll
    for (int x = 0; x < 8; ++x) acc[y][x] = 0.0f;
  for (int q0 = 0; q0 < rank; q0 += kRankChunk) {
    const int qn = min(kRankChunk, rank - q0);
    // the rows' features for this rank chunk
    for (int e = tid; e < kTileRows * kRankChunk; e += kSimtThreads) {
      const int row = e / kRankChunk, qq = e % kRankChunk;
      const int rr = s_row_r[row];
      float f = 0.0f;
      if (rr >= 0 && qq < qn)
        f = a.rnn_feat ? a.rnn_feat[(int64_t)rr * rank + q0 + qq] : ld<DT>(a.E, (int64_t)s_row_prev[row] * rank + q0 + qq);
      f_s[qq][row] = f;
    }
    // W2 rows q0 .. q0 + qn - 1, columns c0 .. c0 + kTileCols - 1 (zero past V), row-major
    if (VEC) {
      constexpr int kPer = 16 / (DT == DSPARK_F32 ? 4 : 2);   // elements per 16-byte load
      for (int e = tid; e < kRankChunk * kTileCols / kPer; e += kSimtThreads) {
        const int qq = e / (kTileCols / kPer), col = (e % (kTileCols / kPer)) * kPer;
        float v[kPer];
        if (qq < qn && c0 + col + kPer <= V) {
          const int64_t at = (int64_t)(q0 + qq) * V + c0 + col;
          const uint4 u = __ldg((const uint4 *)((const char *)a.W + at * (DT == DSPARK_F32 ? 4 : 2)));
          if (DT == DSPARK_F32) {
            v[0] = __uint_as_float(u.x); v[1] = __uint_as_float(u.y);
            v[2] = __uint_as_float(u.z); v[3] = __uint_as_float(u.w);
          } else {
            const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              v[2 * h] = __uint_as_float(w4[h] << 16);
              v[2 * h + 1] = __uint_as_float(w4[h] & 0xffff0000u);
            }
          }
        } else {
#pragma unroll
          for (int h = 0; h < kPer; ++h)
            v[h] = (qq < qn && c0 + col + h < V) ? ld<DT>(a.W, (int64_t)(q0 + qq) * V + c0 + col + h) : 0.0f;
        }
#pragma unroll
        for (int h = 0; h < kPer; ++h) w_s[qq * kTileCols + col + h] = v[h];
      }
    } else {
      for (int e = tid; e < kRankChunk * kTileCols; e += kSimtThreads) {
        const int qq = e / kTileCols, col = e % kTileCols;
        w_s[e] = (qq < qn && c0 + col < V) ? ld<DT>(a.W, (int64_t)(q0 + qq) * V + c0 + col) : 0.0f;
      }
    }
    __syncthreads();
    for (int qq = 0; qq < qn; ++qq) {
      const float4 f4 = *reinterpret_cast<const float4 *>(&f_s[qq][4 * ty]);
      const float4 wa = *reinterpret_cast<const float4 *>(&w_s[qq * kTileCols + 8 * tx]);
      const float4 wb = *reinterpret_cast<const float4 *>(&w_s[qq * kTileCols + 8 * tx + 4]);
      const float fy[4] = {f4.x, f4.y, f4.z, f4.w};
      const float wx[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
#pragma unroll
      for (int y = 0; y < 4; ++y)
#pragma unroll
        for (int x = 0; x < 8; ++x) acc[y][x] = fmaf(fy[y], wx[x], acc[y][x]);
    }
    __syncthreads();
  }
  // the bias tile to shared memory (swizzled), then each thread takes its 32-wide block
#pragma unroll
  for (int y = 0; y < 4; ++y)
#pragma unroll
    for (int x = 0; x < 8; ++x) w_s[wsw(4 * ty + y, 8 * tx + x)] = acc[y][x];
  __syncthreads();
  float z[kBlockW];
  {
    const float4 *zrow = reinterpret_cast<const float4 *>(w_s + tr * kTileCols + tb * 32);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float4 w = zrow[j ^ (tb & 7)];
      z[4 * j] = w.x;
      z[4 * j + 1] = w.y;
      z[4 * j + 2] = w.z;
      z[4 * j + 3] = w.w;
    }
  }
  // epilogue: this thread's 32-wide block v0 .. v0 + 31 of row r
  const int v0 = c0 + tb * kBlockW;
  BRace br;
  brace_init(br);
  float T = 1.0f;
  bool greedy = false;
  if (valid) {
    T = a.temperature[r];
    greedy = (T == 0.0f);
    const float a2 = (greedy ? 1.0f : 1.0f / T) * kLog2e;
    const int64_t urow = ((int64_t)r * K + (k - 1)) * V;
    if (v0 < V) {
      if (VEC && v0 + kBlockW <= V) {   // whole block, 16-byte aligned rows: vector loads and stores
        constexpr int kEsz = DT == DSPARK_F32 ? 4 : 2, kUnits = kBlockW * kEsz / 16;
        const uint4 *up = (const uint4 *)((const char *)a.U + (urow + v0) * kEsz);
        uint4 uu[kUnits];
#pragma unroll
        for (int h = 0; h < kUnits; ++h) uu[h] = __ldcs(up + h);
#pragma unroll
        for (int h = 0; h < kUnits; ++h) {
          const uint32_t w4[4] = {uu[h].x, uu[h].y, uu[h].z, uu[h].w};
          if (DT == DSPARK_F32) {
#pragma unroll
            for (int e = 0; e < 4; ++e) z[4 * h + e] = __uint_as_float(w4[e]) + z[4 * h + e];
          } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              z[8 * h + 2 * e] = round_to_bf16(__uint_as_float(w4[e] << 16) + z[8 * h + 2 * e]);
              z[8 * h + 2 * e + 1] = round_to_bf16(__uint_as_float(w4[e] & 0xffff0000u) + z[8 * h + 2 * e + 1]);
            }
          }
        }
        if (a.draft_logits) {
          uint4 *dp = (uint4 *)((char *)a.draft_logits + (urow + v0) * kEsz);
#pragma unroll
          for (int h = 0; h < kUnits; ++h) {
            uint32_t w4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              if (DT == DSPARK_F32) {
                w4[e] = __float_as_uint(z[4 * h + e]);
              } else {   // the rounded values are exact bf16: their high halves
                w4[e] = (__float_as_uint(z[8 * h + 2 * e]) >> 16) | (__float_as_uint(z[8 * h + 2 * e + 1]) & 0xffff0000u);
              }
            }
            dp[h] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
          }
        }
      } else {
#pragma unroll
        for (int c = 0; c < kBlockW; ++c) {
          if (v0 + c < V) {
            float zz = ld<DT>(a.U, urow + v0 + c) + z[c];
            if (DT == DSPARK_BF16) zz = round_to_bf16(zz);
            if (a.draft_logits) st_logit<DT>(a.draft_logits, urow + v0 + c, zz);
            z[c] = zz;
          } else {
            z[c] = -INFINITY;
          }
        }
      }
      const float mz = block_max(z);
      if (greedy) {
        brace_argmax_block(br, z, mz, v0);
      } else {
        const uint32_t g = (uint32_t)(v0 / kBlockW);
        const uint32_t wb = word_of(philox(a.key, g >> 2, (uint32_t)k, (uint32_t)r, kTagDraft), (int)(g & 3u));
        brace_softmax_block(br, z, mz, a2, wb, v0, [&] {
          return word_of(philox(a.key, g >> 2, (uint32_t)k, (uint32_t)r, kTagDraftPick), (int)(g & 3u));
        });
      }
    }
  }
  // the row's eight blocks (lanes 8m .. 8m + 7 of the warp), merged by shuffles
  Race st = from_partial(to_partial(br));
#pragma unroll
  for (int d = kBlocksPerRow / 2; d > 0; d >>= 1) {
    Race o = race_shfl_down(st, d);
    if (tb + d < kBlocksPerRow) race_merge(st, o);
  }
  const int leader = lane & ~(kBlocksPerRow - 1);
  const int i = i0 + tr;
  int last = 0;
  if (valid && tb == 0) {
    a.partials[(int64_t)i * col_tiles + blockIdx.x] = to_partial(st);
    __threadfence();
    last = (atomicAdd(&a.counters[i], 1) == col_tiles - 1);
  }
  last = __shfl_sync(0xffffffffu, last, leader);
  if (!last) return;
  // the last tile of row i: merge its col_tiles partials (the row's eight lanes, strided, then
  // shuffles among those eight lanes only: other rows' lanes may have left)
  const unsigned gmask = 0xFFu << leader;
  __threadfence();
  Race tot;
  race_init(tot);
  for (int j0 = tb; j0 < col_tiles; j0 += kBlocksPerRow * 8) {   // eight loads in flight per lane
    Partial pb[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int j = j0 + u * kBlocksPerRow;
      pb[u] = j < col_tiles ? load_partial(a.partials + (int64_t)i * col_tiles + j) : empty_partial();
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) race_merge(tot, from_partial(pb[u]));
  }
#pragma unroll
  for (int d = kBlocksPerRow / 2; d > 0; d >>= 1) {
    Race o;
    o.best = __shfl_xor_sync(gmask, tot.best, d);
    o.idx = __shfl_xor_sync(gmask, tot.idx, d);
    o.m = __shfl_xor_sync(gmask, tot.m, d);
    o.S = __shfl_xor_sync(gmask, tot.S, d);
    o.c = 0.0f;
    race_merge(tot, o);
  }
  float conf = 0.0f;
  if (a.conf_out) {   // confidence head: the Markov term over the previous token's W1 row
    float acc = 0.0f;
    for (int q = tb; q < rank; q += kBlocksPerRow)
      acc = fmaf(ld<DT>(a.E, (int64_t)s_row_prev[tr] * rank + q), a.conf_w[q], acc);
#pragma unroll
    for (int d = kBlocksPerRow / 2; d > 0; d >>= 1) acc += __shfl_xor_sync(gmask, acc, d);
    const float sc = a.conf_h[(int64_t)r * K + k - 1] + acc;
    if (sc >= 0.0f) {
      conf = 1.0f / (1.0f + expf(-sc));
    } else {
      const float t = expf(sc);
      conf = t / (1.0f + t);
    }
  }
  if (tb == 0) {
    a.draft_tok[(int64_t)r * K + k - 1] = tot.idx;
    if (a.draft_lse) a.draft_lse[(int64_t)r * K + k - 1] = greedy ? tot.best : tot.m + logf(tot.S);
    if (a.conf_out) a.conf_out[(int64_t)r * K + k - 1] = conf;
    a.counters[i] = 0;
  }
}

}  // namespace

cudaError_t launch_draft_prologue(const DraftArgs &a, cudaStream_t s) {
  draft_prologue<<<1, kPrologueThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_draft_simt(const DraftArgs &a, cudaStream_t s) {
  const int col_tiles = (int)((a.V + kTileCols - 1) / kTileCols);
  const int esz = a.dtype == DSPARK_F32 ? 4 : 2;
  const bool vec = ((a.V * esz) % 16 == 0) && (((uintptr_t)a.U | (uintptr_t)a.W) % 16 == 0) &&
                   ((uintptr_t)a.draft_logits % 16 == 0);
  const size_t cell_smem = sizeof(float) * 5 * (size_t)a.rank;
  // 16-byte weight rows: 2 rank elements, a multiple of 8 (the vector step of the cell)
  const bool cell_vec = ((2 * a.rank) % 8 == 0) && ((uintptr_t)a.rnn_W % 16 == 0);
  if (a.rnn_feat && cell_smem > 48 * 1024) {
    void *fns[4] = {(void *)rnn_cell<DSPARK_F32, false>, (void *)rnn_cell<DSPARK_F32, true>,
                    (void *)rnn_cell<DSPARK_BF16, false>, (void *)rnn_cell<DSPARK_BF16, true>};
    for (void *fn : fns) {
      cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)cell_smem);
      if (e != cudaSuccess) return e;
    }
  }
  const int64_t row_tiles = (a.B + kTileRows - 1) / kTileRows;
  const dim3 grid((unsigned)col_tiles, (unsigned)(row_tiles < 65535 ? row_tiles : 65535));
  for (int k = 1; k <= (int)a.K_max; ++k) {
    if (a.rnn_feat) {
      const unsigned cg = (unsigned)(a.B < 65535 ? a.B : 65535);
      if (a.dtype == DSPARK_F32) {
        if (cell_vec) rnn_cell<DSPARK_F32, true><<<cg, kSimtThreads, cell_smem, s>>>(a, k);
        else rnn_cell<DSPARK_F32, false><<<cg, kSimtThreads, cell_smem, s>>>(a, k);
      } else {
        if (cell_vec) rnn_cell<DSPARK_BF16, true><<<cg, kSimtThreads, cell_smem, s>>>(a, k);
        else rnn_cell<DSPARK_BF16, false><<<cg, kSimtThreads, cell_smem, s>>>(a, k);
      }
      cudaError_t e = cudaGetLastError();
      if (e != cudaSuccess) return e;
    }
    if (a.dtype == DSPARK_F32) {
      if (vec) draft_simt_tile<DSPARK_F32, true><<<grid, kSimtThreads, 0, s>>>(a, k, col_tiles);
      else draft_simt_tile<DSPARK_F32, false><<<grid, kSimtThreads, 0, s>>>(a, k, col_tiles);
    } else {
      if (vec) draft_simt_tile<DSPARK_BF16, true><<<grid, kSimtThreads, 0, s>>>(a, k, col_tiles);
      else draft_simt_tile<DSPARK_BF16, false><<<grid, kSimtThreads, 0, s>>>(a, k, col_tiles);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace dspark
