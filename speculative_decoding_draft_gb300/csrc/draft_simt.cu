// Markov-head draft sampling ("DSpark", S3.1; "Speculative decoding, from zero
// to DSpark", S6): prologue, the RNN head's recurrent cell and the CUDA-core step
// kernel.  With the RNN head, the cell of position k runs before that position's
// step kernel and hands it the feature that replaces the W1 row.
//
// For position k the active requests (K_r >= k) form a prefix of the
// permutation `perm`, which orders requests by K_r descending; the CUDA-core path's
// prologue builds it together with the active counts nact[k].  The tensor-core path's
// prologue (one CTA per position) builds the lists act[k - 1] that its tiles take
// instead: the active requests in 32-request groups of one kind (T > 0 or greedy).
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

// Exclusive prefix over the 32 warps of per-warp counts cnt[w][v] for v = 1..K (warp v - 1
// scans value v, a lane per warp), into pre[w][v]; tot[v] gets the sum.  K <= 32.
__device__ __forceinline__ void prologue_warp_prefix(int (*cnt)[kMaxK + 2], int (*pre)[kMaxK + 2], int *tot, int K,
                                                     int warp, int lane) {
  if (warp < K) {
    const int v = warp + 1;
    const int c = cnt[lane][v];
    int incl = c;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += y;
    }
    pre[lane][v] = incl - c;
    if (lane == 31) tot[v] = incl;
  }
}

// Validation and reset of request r (both paths): its length, anchor and temperature; its
// packed maxima cleared, the slots past K_r set to -1.  Returns the error code (0: valid).
__device__ __forceinline__ int prologue_request(const DraftArgs &a, int r) {
  const int K = (int)a.K_max, V = (int)a.V;
  const int kr = a.K_r[r];
  int err = 0;
  if (kr < 1 || kr > K) err = DSPARK_ERR_LENGTHS;
  const int x0 = a.anchor[r];
  if (x0 < 0 || x0 >= V) err = DSPARK_ERR_TOKEN_RANGE;
  if (!temperature_ok(a.temperature[r])) err = DSPARK_ERR_TEMPERATURE;
  a.counters[r] = 0;
  for (int k = 0; k < K; ++k) {
    a.best_key[(int64_t)r * K + k] = 0ull;
    if (k >= kr) {
      a.draft_tok[(int64_t)r * K + k] = -1;
      if (a.conf_out) a.conf_out[(int64_t)r * K + k] = 0.0f;
    }
  }
  return err;
}

// The CUDA-core path's prologue (one CTA): validation and reset, the active counts nact[k],
// and the K_r-descending permutation.
__global__ void __launch_bounds__(kPrologueThreads) draft_prologue(const __grid_constant__ DraftArgs a) {
  __shared__ int s_err, s_skip;
  __shared__ int cnt[kMaxK + 2];          // requests per length value
  __shared__ int base[kMaxK + 2];         // next free slot per length value
  __shared__ int wc[kPrologueThreads / 32][kMaxK + 2];    // per-warp counts of one round
  __shared__ int wp[kPrologueThreads / 32][kMaxK + 2];    // their exclusive prefix over warps
  __shared__ int wt[kMaxK + 2];                           // their sum
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    s_skip = read_status(a.dev_status);
    s_err = 0;
  }
  if (tid < kMaxK + 2) cnt[tid] = 0;
  __syncthreads();
  if (s_skip) return;
  if (tid <= a.K_max) a.gbar[tid] = 0;
  const int B = (int)a.B, K = (int)a.K_max;
  for (int r = tid; r < B; r += kPrologueThreads) {
    const int err = prologue_request(a, r);
    if (err) atomicCAS(&s_err, 0, err);
    else atomicAdd(&cnt[a.K_r[r]], 1);
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
  // stable scatter, 1024 requests per round: rank among equal lengths by warp match, then the
  // prefix of the warps' counts
  for (int c0 = 0; c0 < B; c0 += kPrologueThreads) {
    const int r = c0 + tid;
    const int v = r < B ? a.K_r[r] : 0;
    const uint32_t peers = __match_any_sync(0xffffffffu, v);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    for (int e = tid; e < (kPrologueThreads / 32) * (kMaxK + 2); e += kPrologueThreads) (&wc[0][0])[e] = 0;
    __syncthreads();
    if (lane == __ffs(peers) - 1) wc[warp][v] = __popc(peers);
    __syncthreads();
    prologue_warp_prefix(wc, wp, wt, K, warp, lane);
    __syncthreads();
    if (r < B) {
      const int slot = (int)bchk(base[v] + wp[warp][v] + rank, B, a.dev_status);
      a.perm[slot] = r;
      a.iperm[r] = slot;
    }
    __syncthreads();
    if (tid >= 1 && tid <= K) base[tid] += wt[tid];
    __syncthreads();
  }
}

// Exclusive prefix over the 32 warps of one count per warp (one warp scans), and the sum.
__device__ __forceinline__ void block_warp_prefix(const int *cnt, int *pre, int *tot, int lane) {
  const int c = cnt[lane];
  int incl = c;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += y;
  }
  pre[lane] = incl - c;
  if (lane == 31) *tot = incl;
}

// The tensor-core path's prologue: one CTA per draft position k, since the positions' lists do
// not depend on one another.  CTA k - 1 validates and resets the requests [B (k-1) / K,
// B k / K) and builds act[k - 1]: the requests with K_r >= k as groups of 32 of one kind (T > 0
// or greedy), each group 32 consecutive such requests in request order, the full groups in
// the order they complete (their last member's index), then the partial group of each kind.
// Every warp of a tile then runs one kind of draw (but at most one per position), and a
// tile's rows lie about as close together in U as the active set allows: listing all T > 0
// requests before all greedy ones spread a greedy tile's rows over ~430 requests at 30 %
// greedy and made the draft 7 % slower than with the greedy requests in one run.
//
// A full group of kind c, number g, whose last member has o requests of the other kind before
// it, is the (g + floor(o / 32))-th full group in that order (o / 32 full groups of the other
// kind completed earlier).  Phase 0 records floor(o / 32) per group (a.grp); phase 1 writes the
// list.  (One CTA building every position's list took 29 us at B = 2048.)
__global__ void __launch_bounds__(kPrologueThreads) draft_prologue_tc(const __grid_constant__ DraftArgs a) {
  __shared__ int wc[2][kPrologueThreads / 32], wp[2][kPrologueThreads / 32], wt[2];
  __shared__ int carry[2], n_kind[2];
  if (read_status(a.dev_status)) return;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int B = (int)a.B, K = (int)a.K_max, k = (int)blockIdx.x + 1;
  if (blockIdx.x == 0) {
    if (tid <= K) a.gbar[tid] = 0;
    if (tid == 0) {
      a.nact[0] = B;
      a.nact[K + 1] = 0;
    }
  }
  {
    const int r0 = (int)((int64_t)B * blockIdx.x / K), r1 = (int)((int64_t)B * (blockIdx.x + 1) / K);
    for (int r = r0 + tid; r < r1; r += kPrologueThreads) {
      const int err = prologue_request(a, r);
      if (err) set_status(a.dev_status, err);
    }
  }
  const int G32 = (B + 31) / 32;
  const uint32_t lt = (1u << lane) - 1u;
  for (int phase = 0; phase < 2; ++phase) {
    if (tid < 2) carry[tid] = 0;
    __syncthreads();
    for (int c0 = 0; c0 < B; c0 += kPrologueThreads) {
      const int r = c0 + tid;
      const bool active = r < B && a.K_r[r] >= k;
      const int kind = (r < B && a.temperature[r] == 0.0f) ? 1 : 0;   // 1: greedy
      const uint32_t b0 = __ballot_sync(0xffffffffu, active && kind == 0);
      const uint32_t b1 = __ballot_sync(0xffffffffu, active && kind == 1);
      if (lane == 0) {
        wc[0][warp] = __popc(b0);
        wc[1][warp] = __popc(b1);
      }
      __syncthreads();
      if (warp < 2) block_warp_prefix(wc[warp], wp[warp], &wt[warp], lane);
      __syncthreads();
      if (active) {
        const int before0 = carry[0] + wp[0][warp] + __popc(b0 & lt);   // T > 0 actives before r
        const int before1 = carry[1] + wp[1][warp] + __popc(b1 & lt);   // greedy actives before r
        const int rank = kind ? before1 : before0, other = kind ? before0 : before1;
        const int g = rank >> 5, l = rank & 31;
        int *grp = a.grp + ((int64_t)(k - 1) * 2 + kind) * G32;
        if (phase == 0) {
          if (l == 31) grp[bchk(g, G32, a.dev_status)] = other >> 5;
        } else {
          const int ns = n_kind[0], ng = n_kind[1];
          const int full = (ns >> 5) + (ng >> 5);
          const int pos = (g < ((kind ? ng : ns) >> 5)) ? 32 * (g + grp[bchk(g, G32, a.dev_status)]) + l
                                                        : 32 * full + (kind ? (ns & 31) : 0) + l;
          a.act[(int64_t)(k - 1) * B + bchk(pos, B, a.dev_status)] = r;
        }
      }
      __syncthreads();
      if (tid < 2) carry[tid] += wt[tid];
      __syncthreads();
    }
    if (phase == 0) {
      if (tid < 2) n_kind[tid] = carry[tid];
      __syncthreads();
    }
  }
  if (tid == 0) a.nact[k] = n_kind[0] + n_kind[1];
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

// RNN head cell ("DSpark" S3.1, RNN head) for position k:
// pre = x_k + W [s_{k-1}; W1[x_{k-1}]] (gate, candidate, output: rows 0..r-1, r..2r-1,
// 2r..3r-1), s_k = g s_{k-1} + (1 - g) tanh(candidate), feature = o s_k, with g and o the
// sigmoids of their pre-activations and s_0 = 0.  One block per tile of kCellUnits hidden
// units x kCellReq active requests: lane j of a warp owns request j of the tile, and the
// kCellSplit warps of a unit each take one contiguous part of every staged input chunk,
// accumulating the unit's three pre-activations in ascending input order; the parts' sums
// are added in part order at the end.  The tile's inputs ([input][request], padded) and its
// 3 kCellUnits weight rows are staged kCellChunk inputs at a time, every thread holding one
// input column of all of them, all loads in flight together (the next chunk's while the
// current one is reduced), so every weight row is read once per request tile.  Tiles of
// other units read s_{k-1} of the same requests while this one writes s_k, so the state
// alternates between two buffers by the parity of k.
constexpr int kCellUnits = 4;
constexpr int kCellReq = 32;
constexpr int kCellSplit = 4;
constexpr int kCellThreads = 32 * kCellUnits * kCellSplit;   // 512
constexpr int kCellChunk = kCellThreads;                     // one staged input column per thread
constexpr int kCellPart = kCellChunk / kCellSplit;           // inputs per warp and chunk
constexpr size_t kCellSmem = sizeof(float) * ((size_t)kCellChunk * (kCellReq + 1) + 3 * kCellUnits * kCellChunk);
static_assert(kCellSplit * 3 * kCellUnits * kCellReq <= 3 * kCellUnits * kCellChunk,
              "the partial sums reuse the weight buffer");

template <int DT>
__global__ void __launch_bounds__(kCellThreads) rnn_cell_tile(const __grid_constant__ DraftArgs a, int k) {
  extern __shared__ float cell_s[];
  float(*z_s)[kCellReq + 1] = reinterpret_cast<float(*)[kCellReq + 1]>(cell_s);    // [input][request]
  float *w_s = cell_s + (size_t)kCellChunk * (kCellReq + 1);                         // [gate][unit][input]
  __shared__ int s_row_r[kCellReq], s_row_prev[kCellReq];
  if (read_status(a.dev_status)) return;
  const int K = (int)a.K_max, rank = (int)a.rank;
  const int n_k = a.nact[k];
  const int i0 = blockIdx.y * kCellReq;
  if (i0 >= n_k) return;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int unit = warp % kCellUnits, part = warp / kCellUnits;
  const int q0 = blockIdx.x * kCellUnits;               // first hidden unit of the tile
  const size_t plane = (size_t)a.B * (size_t)rank;
  const float *s_prev = a.rnn_state + (size_t)((k + 1) & 1) * plane;   // s_{k-1}
  float *s_next = a.rnn_state + (size_t)(k & 1) * plane;               // s_k
  if (tid < kCellReq) {
    const int i = i0 + tid;
    const int r = i < n_k ? (int)bchk(a.perm[i], a.B, a.dev_status) : -1;
    s_row_r[tid] = r;
    s_row_prev[tid] =
        r < 0 ? 0 : (int)bchk((k == 1) ? a.anchor[r] : a.draft_tok[(int64_t)r * K + k - 2], a.V, a.dev_status);
  }
  __syncthreads();
  const int n_in = 2 * rank;
  float acc[3] = {0.0f, 0.0f, 0.0f};
  float zr[kCellReq], wr[3 * kCellUnits];
  auto fetch = [&](int c0) {
    const int in = c0 + tid;
    const bool live = in < n_in;
#pragma unroll
    for (int j = 0; j < kCellReq; ++j) {
      const int r = s_row_r[j];
      float z = 0.0f;
      if (r >= 0 && live) {
        if (in < rank) z = (k == 1) ? 0.0f : s_prev[(int64_t)r * rank + in];
        else z = ld<DT>(a.E, (int64_t)s_row_prev[j] * rank + (in - rank));
      }
      zr[j] = z;
    }
#pragma unroll
    for (int gu = 0; gu < 3 * kCellUnits; ++gu) {
      const int g = gu / kCellUnits, q = q0 + gu % kCellUnits;
      wr[gu] = (q < rank && live) ? ld<DT>(a.rnn_W, ((int64_t)g * rank + q) * n_in + in) : 0.0f;
    }
  };
  fetch(0);
  for (int c0 = 0; c0 < n_in; c0 += kCellChunk) {
#pragma unroll
    for (int j = 0; j < kCellReq; ++j) z_s[tid][j] = zr[j];
#pragma unroll
    for (int gu = 0; gu < 3 * kCellUnits; ++gu) w_s[gu * kCellChunk + tid] = wr[gu];
    __syncthreads();
    if (c0 + kCellChunk < n_in) fetch(c0 + kCellChunk);
    const int c_lo = part * kCellPart, c_hi = min(c_lo + kCellPart, n_in - c0);
    const float *wg = w_s + unit * kCellChunk;
#pragma unroll 8
    for (int c = c_lo; c < c_hi; ++c) {
      const float z = z_s[c][lane];
      acc[0] = fmaf(wg[c], z, acc[0]);
      acc[1] = fmaf(wg[kCellUnits * kCellChunk + c], z, acc[1]);
      acc[2] = fmaf(wg[2 * kCellUnits * kCellChunk + c], z, acc[2]);
    }
    __syncthreads();
  }
  // the parts' sums, added in part order by the warps of part 0
  float *red = w_s;   // [part][gate][unit][request]
#pragma unroll
  for (int g = 0; g < 3; ++g) red[((part * 3 + g) * kCellUnits + unit) * kCellReq + lane] = acc[g];
  __syncthreads();
  if (part != 0) return;
  float pre[3];
#pragma unroll
  for (int g = 0; g < 3; ++g) {
    float t = red[(g * kCellUnits + unit) * kCellReq + lane];
#pragma unroll
    for (int p = 1; p < kCellSplit; ++p) t += red[((p * 3 + g) * kCellUnits + unit) * kCellReq + lane];
    pre[g] = t;
  }
  const int r = s_row_r[lane];
  const int q = q0 + unit;
  if (r < 0 || q >= rank) return;
  const float *xk = a.rnn_x + ((int64_t)r * K + (k - 1)) * 3 * rank;
  const float g = 1.0f / (1.0f + expf(-(xk[q] + pre[0])));
  const float c = tanhf(xk[rank + q] + pre[1]);
  const float o = 1.0f / (1.0f + expf(-(xk[2 * rank + q] + pre[2])));
  const float sp = (k == 1) ? 0.0f : s_prev[(int64_t)r * rank + q];
  const float st = g * sp + (1.0f - g) * c;
  s_next[(int64_t)r * rank + q] = st;
  a.rnn_feat[(int64_t)r * rank + q] = o * st;
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
__global__ void __launch_bounds__(kSimtThreads, 3) draft_simt_tile(const __grid_constant__ DraftArgs a, int k,
                                                                 int col_tiles) {
  // GEMM layout: thread (ty, tx) accumulates rows 4 ty .. 4 ty + 3 x columns 4 tx .. 4 tx + 3
  // and 128 + 4 tx .. 128 + 4 tx + 3 (three 16-byte shared loads per 32 FMAs); the tile then
  // goes through shared memory (swizzled) to the epilogue layout, one 32-wide block per thread.
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
    const int r = i < n_k ? (int)bchk(a.perm[i], a.B, a.dev_status) : -1;
    s_row_r[tid] = r;
    s_row_prev[tid] =
        r < 0 ? 0 : (int)bchk((k == 1) ? a.anchor[r] : a.draft_tok[(int64_t)r * K + k - 2], a.V, a.dev_status);
  }
  __syncthreads();
  const int r = s_row_r[tr];
  const bool valid = r >= 0;
  float acc[4][8];
#pragma unroll
  for (int y = 0; y < 4; ++y)
#pragma unroll
    for (int x = 0; x < 8; ++x) acc[y][x] = 0.0f;
  // the rows' feature for rank value q (the previous token's W1 row, or the RNN cell's output)
  auto feature = [&](int row, int q) -> float {
    const int rr = s_row_r[row];
    if (rr < 0) return 0.0f;
    return a.rnn_feat ? a.rnn_feat[(int64_t)rr * rank + q] : ld<DT>(a.E, (int64_t)s_row_prev[row] * rank + q);
  };
  // one staged rank chunk: rows 4 ty .. 4 ty + 3 x columns 4 tx .. 4 tx + 3 and
  // kTileCols / 2 + 4 tx .. + 3, ascending rank (each 16-byte W2 load of a warp covers 512
  // contiguous bytes: four shared-memory wavefronts)
  auto gemm_chunk = [&](int qn) {
#pragma unroll 4
    for (int qq = 0; qq < qn; ++qq) {
      const float4 f4 = *reinterpret_cast<const float4 *>(&f_s[qq][4 * ty]);
      const float4 wa = *reinterpret_cast<const float4 *>(&w_s[qq * kTileCols + 4 * tx]);
      const float4 wb = *reinterpret_cast<const float4 *>(&w_s[qq * kTileCols + kTileCols / 2 + 4 * tx]);
      const float fy[4] = {f4.x, f4.y, f4.z, f4.w};
      const float wx[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
#pragma unroll
      for (int y = 0; y < 4; ++y)
#pragma unroll
        for (int x = 0; x < 8; ++x) acc[y][x] = fmaf(fy[y], wx[x], acc[y][x]);
    }
  };
  if (VEC) {
    // V and the rows are 16-byte aligned: a 16-byte unit of a W2 row is either wholly inside
    // V or wholly past it.  The next chunk's W2 units and features are loaded into registers
    // while the current chunk's FMAs run, then stored to shared memory after the barrier.
    constexpr int kPer = 16 / (DT == DSPARK_F32 ? 4 : 2);                 // elements per unit
    constexpr int kUnitsPerRow = kTileCols / kPer;
    constexpr int kWLoads = kRankChunk * kUnitsPerRow / kSimtThreads;     // units per thread
    constexpr int kFLoads = kTileRows * kRankChunk / kSimtThreads;        // features per thread
    static_assert(kRankChunk * kUnitsPerRow % kSimtThreads == 0 && kTileRows * kRankChunk % kSimtThreads == 0,
                  "staging splits evenly over the block");
    uint4 wreg[kWLoads];
    float freg[kFLoads];
    auto fetch = [&](int q0) {
      const int qn = min(kRankChunk, rank - q0);
#pragma unroll
      for (int u = 0; u < kFLoads; ++u) {
        const int e = tid + u * kSimtThreads;
        const int row = e / kRankChunk, qq = e % kRankChunk;
        freg[u] = qq < qn ? feature(row, q0 + qq) : 0.0f;
      }
#pragma unroll
      for (int h = 0; h < kWLoads; ++h) {
        const int e = tid + h * kSimtThreads;
        const int qq = e / kUnitsPerRow, col = (e % kUnitsPerRow) * kPer;
        wreg[h] = (qq < qn && c0 + col < V)
                      ? __ldg((const uint4 *)((const char *)a.W +
                                              ((int64_t)(q0 + qq) * V + c0 + col) * (DT == DSPARK_F32 ? 4 : 2)))
                      : make_uint4(0u, 0u, 0u, 0u);
      }
    };
    auto stage = [&]() {
#pragma unroll
      for (int u = 0; u < kFLoads; ++u) {
        const int e = tid + u * kSimtThreads;
        f_s[e % kRankChunk][e / kRankChunk] = freg[u];
      }
#pragma unroll
      for (int h = 0; h < kWLoads; ++h) {
        const int e = tid + h * kSimtThreads;
        const int qq = e / kUnitsPerRow, col = (e % kUnitsPerRow) * kPer;
        float4 *dst = reinterpret_cast<float4 *>(&w_s[qq * kTileCols + col]);
        const uint4 w = wreg[h];
        if (DT == DSPARK_F32) {
          dst[0] = make_float4(__uint_as_float(w.x), __uint_as_float(w.y), __uint_as_float(w.z), __uint_as_float(w.w));
        } else {
          dst[0] = make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u),
                               __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u));
          dst[1] = make_float4(__uint_as_float(w.z << 16), __uint_as_float(w.z & 0xffff0000u),
                               __uint_as_float(w.w << 16), __uint_as_float(w.w & 0xffff0000u));
        }
      }
    };
    fetch(0);
    for (int q0 = 0; q0 < rank; q0 += kRankChunk) {
      stage();
      __syncthreads();
      if (q0 + kRankChunk < rank) fetch(q0 + kRankChunk);
      gemm_chunk(min(kRankChunk, rank - q0));
      __syncthreads();
    }
  } else {
    for (int q0 = 0; q0 < rank; q0 += kRankChunk) {
      const int qn = min(kRankChunk, rank - q0);
      for (int e = tid; e < kTileRows * kRankChunk; e += kSimtThreads) {
        const int row = e / kRankChunk, qq = e % kRankChunk;
        f_s[qq][row] = qq < qn ? feature(row, q0 + qq) : 0.0f;
      }
      // W2 rows q0 .. q0 + qn - 1, columns c0 .. c0 + kTileCols - 1 (zero past V), row-major
      for (int e = tid; e < kRankChunk * kTileCols; e += kSimtThreads) {
        const int qq = e / kTileCols, col = e % kTileCols;
        w_s[e] = (qq < qn && c0 + col < V) ? ld<DT>(a.W, (int64_t)(q0 + qq) * V + c0 + col) : 0.0f;
      }
      __syncthreads();
      gemm_chunk(qn);
      __syncthreads();
    }
  }
  // the bias tile to shared memory (swizzled), then each thread takes its 32-wide block
#pragma unroll
  for (int y = 0; y < 4; ++y)
#pragma unroll
    for (int x = 0; x < 8; ++x) w_s[wsw(4 * ty + y, (x < 4 ? 0 : kTileCols / 2 - 4) + 4 * tx + x)] = acc[y][x];
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
        brace_softmax_block(
            br, z, mz, a2, wb, v0,
            [&] { return word_of(philox(a.key, g >> 2, (uint32_t)k, (uint32_t)r, kTagDraftPick), (int)(g & 3u)); },
            [&](int q) {   // the drawn element's logit, recomputed exactly as above from U and the bias tile
              float zz = ld<DT>(a.U, urow + v0 + q) + w_s[tr * kTileCols + tb * 32 + (((q >> 2) ^ (tb & 7)) << 2) + (q & 3)];
              if (DT == DSPARK_BF16) zz = round_to_bf16(zz);
              return zz;
            });
      }
    }
  }
  // the row's eight blocks (lanes 8m .. 8m + 7 of the warp), merged by shuffles
  Race st = from_partial(to_partial(br));
  float zx = br.zx;   // the logit at st.idx
#pragma unroll
  for (int d = kBlocksPerRow / 2; d > 0; d >>= 1) {
    Race o = race_shfl_down(st, d);
    const float ozx = __shfl_down_sync(0xffffffffu, zx, d);
    if (tb + d < kBlocksPerRow) {
      if (race_takes(st, o)) zx = ozx;
      race_merge(st, o);
    }
  }
  const int leader = lane & ~(kBlocksPerRow - 1);
  const int i = i0 + tr;
  int last = 0;
  if (valid && tb == 0) {
    a.partials[(int64_t)i * col_tiles + blockIdx.x] = to_partial(st);
    a.zx_part[(int64_t)i * col_tiles + blockIdx.x] = zx;
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
    // the token's logit: the partial of the column tile that holds the token carries it
    if (a.draft_zx && tot.idx >= 0)
      a.draft_zx[(int64_t)r * K + k - 1] = load_f32_relaxed(a.zx_part + (int64_t)i * col_tiles + tot.idx / kTileCols);
    if (a.conf_out) a.conf_out[(int64_t)r * K + k - 1] = conf;
    a.counters[i] = 0;
  }
}

}  // namespace

cudaError_t launch_draft_prologue(const DraftArgs &a, cudaStream_t s, bool tensor_core) {
  if (tensor_core) draft_prologue_tc<<<(unsigned)a.K_max, kPrologueThreads, 0, s>>>(a);
  else draft_prologue<<<1, kPrologueThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_draft_simt(const DraftArgs &a, cudaStream_t s) {
  const int col_tiles = (int)((a.V + kTileCols - 1) / kTileCols);
  const int esz = a.dtype == DSPARK_F32 ? 4 : 2;
  const bool vec = ((a.V * esz) % 16 == 0) && (((uintptr_t)a.U | (uintptr_t)a.W) % 16 == 0) &&
                   ((uintptr_t)a.draft_logits % 16 == 0);
  const int64_t row_tiles = (a.B + kTileRows - 1) / kTileRows;
  const dim3 grid((unsigned)col_tiles, (unsigned)(row_tiles < 65535 ? row_tiles : 65535));
  for (int k = 1; k <= (int)a.K_max; ++k) {
    if (a.rnn_feat) {
      for (const void *fn : {(const void *)rnn_cell_tile<DSPARK_F32>, (const void *)rnn_cell_tile<DSPARK_BF16>}) {
        cudaError_t e = ensure_dynamic_smem(fn, (int)kCellSmem);
        if (e != cudaSuccess) return e;
      }
      const dim3 cg((unsigned)((a.rank + kCellUnits - 1) / kCellUnits),
                    (unsigned)((a.B + kCellReq - 1) / kCellReq));
      if (a.dtype == DSPARK_F32) rnn_cell_tile<DSPARK_F32><<<cg, kCellThreads, kCellSmem, s>>>(a, k);
      else rnn_cell_tile<DSPARK_BF16><<<cg, kCellThreads, kCellSmem, s>>>(a, k);
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
