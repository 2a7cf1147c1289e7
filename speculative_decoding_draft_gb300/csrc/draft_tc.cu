// Markov-head draft sampling, tensor-core path (sm_103a: tcgen05 + TMA + TMEM).
//
// "DSpark" S3.1 (Markov head B(x_{k-1}, .) = W1[x_{k-1}] . W2, rank r) and
// "Speculative decoding, from zero to DSpark" S6 (p_k = softmax(U_k + B_k)).
//
// One launch per draft position k.  The active requests (K_r >= k) form the
// first n_k entries of `perm`; they are cut into M-tiles of 128 rows.  A
// persistent grid of one CTA per SM gives every M-tile floor(G / M-tiles) CTAs,
// each owning a contiguous range of 64-wide vocabulary tiles, so the gathered
// 128 x r operand is staged once per CTA and reused across its whole range.
//
// Warp roles (320 threads):
//   warp 0     producer: per vocabulary tile, one TMA tile load of W2[:, n:n+64]
//              (128-byte swizzle, r x 64 bf16) and one 1-D bulk copy per active row
//              of U[r, k-1, n:n+64] into a padded row-major slot; both complete on
//              the stage's full barrier.
//   warp 1     allocates TMEM (4 accumulators of 128 x 64 fp32) and one elected
//              lane issues r/16 tcgen05.mma (kind::f16, bf16 in, fp32 accumulate,
//              A K-major from shared memory, B MN-major from shared memory) per tile,
//              committing to the stage's empty barrier and the accumulator's full
//              barrier.
//   warps 2-9  epilogue, two warps per TMEM lane quadrant (one per 32-column half):
//              gather W1[x_{k-1}] rows into the swizzled A operand at the start of a
//              tile range, then per tile tcgen05.ld the 32 fp32 bias values of their
//              row, add U, round to bf16, optionally store the logits, and run the
//              Gumbel race / greedy argmax with the online softmax.  No 128 x V
//              logits tile ever goes back to HBM unless the caller asks for it.
// Block partials per row are merged by the last CTA of each M-tile, which
// writes the token and the log-sum-exp.  Every wait is bounded; on a timeout
// the kernel records DSPARK_ERR_DEVICE_TIMEOUT, drains what it issued, frees
// TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "dspark_internal.cuh"

namespace dspark {
namespace {

constexpr int kTileM = 128;
constexpr int kTileN = 64;
constexpr int kStages = 4;
constexpr int kAccBufs = 4;
constexpr int kEpiWarps = 8;
constexpr int kThreadsTc = 32 * (2 + kEpiWarps);
constexpr int kTmemCols = kAccBufs * kTileN;               // 256
constexpr int kAChunk = kTileM * 128;                      // 16 KB: 128 rows x 64 bf16
constexpr int kASize = 4 * kAChunk;                        // rank <= 256
constexpr int kWSlot = 256 * 128;                          // r rows x 128 B
constexpr int kOffA = 0;
constexpr int kOffW = kOffA + kASize;
constexpr int kOffSh = kOffW + kStages * kWSlot;
constexpr long long kTimeoutCycles = 4000000000LL;

struct TcShared {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t accf[kAccBufs];
  uint64_t acce[kAccBufs];
  uint64_t aready;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int last;
  int skip;
  int row_req[kTileM];
  int row_prev[kTileM];
  float row_invT[kTileM];
  Partial part[2 * kTileM];   // per-row thread partials: [replica group x column half][row]
};

constexpr int kSmemBytes = kOffSh + (int)sizeof(TcShared) + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget");

// ---- PTX wrappers ---------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_tx(uint32_t bar, uint32_t tx) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(tx) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait on a barrier phase.  Returns false (and raises the CTA abort
// flag) when the wait gave up or another role already aborted.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort) {
  const long long t0 = clock64();
  while (!mbar_try(bar, parity)) {
    if (*abort) return false;
    if (clock64() - t0 > kTimeoutCycles) {
      *abort = 1;
      return false;
    }
  }
  return true;
}
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
        "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
        "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"((uint64_t)map), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}

// L2 policies: the projection W2 is re-read at every draft position and should stay in
// L2; the base logits U and the stored draft logits are touched once.
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint4 ld_u4_hint(const void *ptr, uint64_t policy) {
  uint4 v;
  asm volatile("ld.global.nc.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(ptr), "l"(policy));
  return v;
}
__device__ __forceinline__ void st_u4_hint(void *ptr, uint4 v, uint64_t policy) {
  asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(ptr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w), "l"(policy)
               : "memory");
}
__device__ __forceinline__ int ld_acquire(const int32_t *p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Shared-memory matrix descriptor (tcgen05): start, leading and stride byte
// offsets (>> 4), descriptor version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor, kind::f16: fp32 accumulate, bf16 A and B, A K-major,
// B MN-major, N = 64, M = 128.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 16) | ((uint32_t)(kTileN >> 3) << 17) |
                            ((uint32_t)(kTileM >> 4) << 24);

__device__ __forceinline__ void named_sync_epi() {
  asm volatile("bar.sync 1, %0;" ::"n"(kEpiWarps * 32) : "memory");
}

// U row segment of one epilogue thread for one tile: 32 bf16 at column c0 of
// its row (16-byte loads; columns past V are not read).
__device__ __forceinline__ void load_u32(const unsigned short *row, int c0, int V, uint4 (&u)[4], uint64_t pol) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    if (c0 + 8 * q < V) u[q] = ld_u4_hint(row + c0 + 8 * q, pol);
    else u[q] = make_uint4(0u, 0u, 0u, 0u);
  }
}

// Work split of one draft position: M-tiles of 128 active rows, each shared by gm CTAs
// that own contiguous ranges of 64-wide vocabulary tiles.
struct StepPlan {
  int n_k, m_tiles, gm, units;
};
__device__ __forceinline__ StepPlan plan_step(const DraftArgs &a, int k, int G, int n_tiles) {
  StepPlan p;
  p.n_k = a.nact[k];
  p.m_tiles = (p.n_k + kTileM - 1) / kTileM;
  p.gm = p.m_tiles ? max(1, min(G / p.m_tiles, n_tiles)) : 1;
  p.units = p.m_tiles * p.gm;
  return p;
}

// ---------------------------------------------------------------------------
// One persistent CTA per SM walks every draft position k = 1..K_max.  The producer
// and MMA roles run ahead through positions on their own barriers (W2 does not
// depend on the drafted tokens); the epilogue waits on a grid-wide barrier before
// it reads the previous position's tokens, so the next position's W2 tiles and U
// segments are already in flight while the barrier completes.
template <int RCH>   // rank / 64
__global__ void __launch_bounds__(kThreadsTc, 1)
    draft_tc_persistent(const __grid_constant__ DraftArgs a, const __grid_constant__ CUtensorMap tmap_w) {
  constexpr int kRank = RCH * 64;
  constexpr int kKsteps = kRank / 16;
  constexpr int kUpr = kRank / 8;                  // 16-byte units per W1 row
  constexpr uint32_t kWBytes = (uint32_t)(kTileN * kRank * 2);
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;
  uint8_t *gb = smem_raw + (sb - raw);
  TcShared &sh = *reinterpret_cast<TcShared *>(gb + kOffSh);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) sh.skip = read_status(a.dev_status);
  __syncthreads();
  if (sh.skip) return;   // an earlier error: every CTA sees the same word and leaves

  const int K = (int)a.K_max, V = (int)a.V;
  const int G = gridDim.x;
  const int n_tiles = (V + kTileN - 1) / kTileN;

  const uint32_t bar_full = smem_u32(&sh.full[0]);
  const uint32_t bar_empty = smem_u32(&sh.empty[0]);
  const uint32_t bar_accf = smem_u32(&sh.accf[0]);
  const uint32_t bar_acce = smem_u32(&sh.acce[0]);
  const uint32_t bar_aready = smem_u32(&sh.aready);
  const uint32_t bar_drain = smem_u32(&sh.drain);
  volatile int *abort = &sh.abort;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (int b = 0; b < kAccBufs; ++b) {
      mbar_init(bar_accf + 8 * b, 1);
      mbar_init(bar_acce + 8 * b, kEpiWarps);
    }
    mbar_init(bar_aready, kEpiWarps);
    mbar_init(bar_drain, 1);
    sh.abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&sh.tmem_base), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;

  uint32_t last_use[kStages];   // producer: last issued use of each stage (for the abort drain)
  bool issued[kStages];
#pragma unroll
  for (int s = 0; s < kStages; ++s) {
    last_use[s] = 0;
    issued[s] = false;
  }

  if (warp == 0) {
    // ---------------- producer: W2 tiles of every position ----------------
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_last();
      uint32_t it = 0;
      for (int k = 1; k <= K && !*abort; ++k) {
        const StepPlan pl = plan_step(a, k, G, n_tiles);
        if (pl.n_k == 0) break;
        for (int u = blockIdx.x; u < pl.units && !*abort; u += G) {
          const int j = u % pl.gm;
          const int nt0 = (int)((int64_t)j * n_tiles / pl.gm), nt1 = (int)((int64_t)(j + 1) * n_tiles / pl.gm);
          for (int t = nt0; t < nt1; ++t, ++it) {
            const int s = (int)(it % kStages);
            const uint32_t use = it / kStages;
            if (!mbar_wait(bar_empty + 8 * s, (use & 1u) ^ 1u, abort)) break;
            mbar_arrive_tx(bar_full + 8 * s, kWBytes);
            tma_load_2d(sb + kOffW + s * kWSlot, &tmap_w, t * kTileN, 0, bar_full + 8 * s, pol_w);
#pragma unroll
            for (int q = 0; q < kStages; ++q)
              if (q == s) { last_use[q] = use; issued[q] = true; }
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      uint32_t it = 0;
      int unit_no = 0;
      bool ok = true;
      for (int k = 1; k <= K && ok; ++k) {
        const StepPlan pl = plan_step(a, k, G, n_tiles);
        if (pl.n_k == 0) break;
        for (int u = blockIdx.x; u < pl.units && ok; u += G, ++unit_no) {
          const int j = u % pl.gm;
          const int nt0 = (int)((int64_t)j * n_tiles / pl.gm), nt1 = (int)((int64_t)(j + 1) * n_tiles / pl.gm);
          ok = mbar_wait(bar_aready, (uint32_t)(unit_no & 1), abort);
          for (int t = nt0; ok && t < nt1; ++t, ++it) {
            const int s = (int)(it % kStages);
            const uint32_t use = it / kStages;
            const int b = (int)(it % kAccBufs);
            const uint32_t ause = it / kAccBufs;
            if (!(ok = mbar_wait(bar_full + 8 * s, use & 1u, abort))) break;
            if (!(ok = mbar_wait(bar_acce + 8 * b, (ause & 1u) ^ 1u, abort))) break;
            tc_fence_after();
            const uint32_t d = tmem + (uint32_t)(b * kTileN);
#pragma unroll 1
            for (int kk = 0; kk < kKsteps; ++kk) {
              const uint64_t ad = smem_desc(sb + kOffA + (kk >> 2) * kAChunk + (kk & 3) * 32, 16, 1024);
              const uint64_t bd = smem_desc(sb + kOffW + s * kWSlot + kk * 2048, (uint32_t)(kRank * 128), 1024);
              mma_bf16(d, ad, bd, kIdesc, kk > 0 ? 1u : 0u);
            }
            mma_commit(bar_empty + 8 * s);
            mma_commit(bar_accf + 8 * b);
          }
        }
      }
    }
    __syncwarp();
  } else {
    // ---------------- epilogue ----------------
    const int eq = warp - 2;            // 0..7
    const int quad = warp & 3;          // TMEM lanes 32*quad .. +31 are reachable by this warp
    const int half = eq >> 2;           // 32-column half of the 64-wide tile
    const int et = eq * 32 + lane;      // 0..255
    const uint64_t pol_stream = policy_evict_first();
    uint32_t it = 0;
    int unit_no = 0;
    for (int k = 1; k <= K && !*abort; ++k) {
      const StepPlan pl = plan_step(a, k, G, n_tiles);
      if (pl.n_k == 0) break;
      bool waited = (k == 1);
      for (int u = blockIdx.x; u < pl.units && !*abort; u += G, ++unit_no) {
        const int m = u / pl.gm, j = u % pl.gm;
        const int nt0 = (int)((int64_t)j * n_tiles / pl.gm), nt1 = (int)((int64_t)(j + 1) * n_tiles / pl.gm);
        const int row0 = m * kTileM;
        const int nrows = min(kTileM, pl.n_k - row0);
        // replication: with few rows, every TMEM lane quadrant (= SM sub-partition) gets a copy
        // of the rows and takes every F-th vocabulary tile
        const int F = nrows <= 32 ? 4 : (nrows <= 64 ? 2 : 1);
        const int rpg = kTileM / F;
        named_sync_epi();             // readers of the previous unit's row table are done
        if (et < kTileM) {
          const int i = et;
          if (i < nrows) {
            const int r = a.perm[row0 + i];
            sh.row_req[i] = r;
            const float T = a.temperature[r];
            sh.row_invT[i] = (T == 0.0f) ? 0.0f : 1.0f / T;
          } else {
            sh.row_req[i] = -1;
            sh.row_invT[i] = 0.0f;
          }
        }
        named_sync_epi();
        const int arow = quad * 32 + lane;        // TMEM lane = M-row
        const int grp = arow / rpg;               // replica group: takes tiles t with (t - nt0) % F == grp
        const int row = arow % rpg;               // request row of this thread
        const bool valid = row < nrows;
        const int r = valid ? sh.row_req[row] : 0;
        const float invT = sh.row_invT[row];
        const bool greedy = (invT == 0.0f);
        const int64_t urow = ((int64_t)r * K + (k - 1)) * (int64_t)V;
        const unsigned short *uptr = (const unsigned short *)a.U + urow;
        uint4 ucur[4], unext[4];
        int tmine = nt0 + grp;                    // first tile of this thread
        if (valid && tmine < nt1) load_u32(uptr, tmine * kTileN + half * 32, V, ucur, pol_stream);   // before the barrier
        if (!waited) {
          // every CTA has folded its position k-1 maxima into the packed keys
          if (et == 0) {
            const long long t0 = clock64();
            while (ld_acquire(a.gbar + (k - 1)) < G) {
              if (*abort) break;
              if (clock64() - t0 > kTimeoutCycles) { *abort = 1; break; }
            }
          }
          named_sync_epi();
          waited = true;
          if (*abort) break;
        }
        if (et < kTileM && et < nrows) {
          const int rq = sh.row_req[et];
          sh.row_prev[et] = (k == 1) ? a.anchor[rq] : key_index(__ldcg(a.best_key + (int64_t)rq * K + k - 2));
        }
        named_sync_epi();
        // gather the A operand: request row i's 16-byte unit c8 of K-chunk c goes to every replica
        // M-row a = g * rpg + i, chunk c, unit (c8 ^ (a & 7)) -- the 128-byte swizzle.  All loads of a
        // thread are issued before its stores, so the row fetches overlap.
        {
          const int total = nrows * kUpr;
#pragma unroll 1
          for (int q0 = 0; q0 < 16; q0 += 8) {     // two batches of eight 16-byte loads per thread
            uint4 val[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const int e = et + (q0 + q) * kEpiWarps * 32;
              val[q] = make_uint4(0u, 0u, 0u, 0u);
              if (e < total) {
                const int i = e / kUpr, uu = e % kUpr;
                val[q] = __ldg((const uint4 *)((const unsigned short *)a.E + (int64_t)sh.row_prev[i] * kRank) + uu);
              }
            }
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const int e = et + (q0 + q) * kEpiWarps * 32;
              if (e >= total) continue;
              const int i = e / kUpr, uu = e % kUpr;
              const int c = uu >> 3, c8 = uu & 7;
              for (int g = 0; g < F; ++g) {
                const int ar = g * rpg + i;
                const uint32_t dst = sb + kOffA + c * kAChunk + ar * 128 + ((c8 ^ (ar & 7)) << 4);
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(val[q].x), "r"(val[q].y),
                             "r"(val[q].z), "r"(val[q].w)
                             : "memory");
              }
            }
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_aready);

        Race st;
        race_init(st);
        for (int t = nt0; t < nt1; ++t, ++it) {
          const int b = (int)(it % kAccBufs);
          const uint32_t ause = it / kAccBufs;
          if (!mbar_wait(bar_accf + 8 * b, ause & 1u, abort)) break;
          if (t != tmine) {                       // another replica group owns this tile
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_acce + 8 * b);
            continue;
          }
          tc_fence_after();
          uint32_t acc[32];
          tmem_ld32(tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(b * kTileN + half * 32), acc);
          tmem_wait_ld();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_acce + 8 * b);
          tmine += F;
          if (!valid) continue;
          if (tmine < nt1) load_u32(uptr, tmine * kTileN + half * 32, V, unext, pol_stream);   // prefetch
          const int c0 = t * kTileN + half * 32;
          const bool full = (c0 + 32 <= V);
          uint32_t w[32];
          if (!greedy) {
#pragma unroll
            for (int q = 0; q < 8; ++q) {           // eight independent Philox blocks: ILP
              const uint4 wq = philox(a.key, (uint32_t)(c0 >> 2) + (uint32_t)q, (uint32_t)k, (uint32_t)r, kTagDraft);
              w[4 * q] = wq.x;
              w[4 * q + 1] = wq.y;
              w[4 * q + 2] = wq.z;
              w[4 * q + 3] = wq.w;
            }
          }
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            const uint32_t pk[4] = {ucur[g].x, ucur[g].y, ucur[g].z, ucur[g].w};
            float sv[8];
            uint32_t packed[4];
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
              const float z0 = __uint_as_float(pk[e >> 1] << 16) + __uint_as_float(acc[g * 8 + e]);
              const float z1 = __uint_as_float(pk[e >> 1] & 0xffff0000u) + __uint_as_float(acc[g * 8 + e + 1]);
              const __nv_bfloat162 zb = __floats2bfloat162_rn(z0, z1);   // one rounding of each fp32 sum
              packed[e >> 1] = *reinterpret_cast<const uint32_t *>(&zb);
              const float2 zf = __bfloat1622float2(zb);
              sv[e] = greedy ? zf.x : zf.x * invT;
              sv[e + 1] = greedy ? zf.y : zf.y * invT;
            }
            if (!full) {
#pragma unroll
              for (int e = 0; e < 8; ++e)
                if (c0 + g * 8 + e >= V) sv[e] = -INFINITY;
            }
            if (a.draft_logits && (full || c0 + g * 8 + 8 <= V))
              st_u4_hint((unsigned short *)a.draft_logits + urow + c0 + g * 8,
                         make_uint4(packed[0], packed[1], packed[2], packed[3]), pol_stream);
            if (greedy) {
              argmax_update<8>(st, sv, c0 + g * 8);
            } else {
              const uint32_t wg[8] = {w[8 * g], w[8 * g + 1], w[8 * g + 2], w[8 * g + 3],
                                      w[8 * g + 4], w[8 * g + 5], w[8 * g + 6], w[8 * g + 7]};
              race_update<8>(st, sv, wg, c0 + g * 8);
            }
          }
#pragma unroll
          for (int q = 0; q < 4; ++q) ucur[q] = unext[q];
        }
        // merge the 2F thread partials of each row (replica groups x column halves); the row's
        // home thread folds its maximum into the packed (score, index) key of the position with one
        // 64-bit atomicMax -- all the next position needs -- and keeps its softmax partial for the
        // normaliser, which the finalize kernel merges once per call
        sh.part[(grp * 2 + half) * rpg + row] = to_partial(st);
        named_sync_epi();
        if (grp == 0 && half == 0 && valid) {
          for (int q = 1; q < 2 * F; ++q) race_merge(st, from_partial(sh.part[q * rpg + row]));
          if (st.idx >= 0) atomicMax(&a.best_key[(int64_t)r * K + k - 1], score_key(st.best, st.idx));
          a.partials[(int64_t)(k - 1) * kTcPartialsPerStep + ((int64_t)m * kTileM + row) * pl.gm + j] =
              to_partial(st);
        }
      }
      // this CTA is done with position k (every CTA arrives, with or without work)
      __threadfence();
      named_sync_epi();
      if (et == 0) atomicAdd(a.gbar + k, 1);
    }
  }

  // ---- teardown: drain issued MMAs and copies, free TMEM -----------------------
  if (warp == 1) {
    if (lane == 0) {
      mma_commit(bar_drain);
      const long long t0 = clock64();
      while (!mbar_try(bar_drain, 0u) && clock64() - t0 < kTimeoutCycles) {
      }
    }
    __syncwarp();
  }
  if (warp == 0 && lane == 0 && *abort) {
    // wait (bounded) until the last copy issued into each stage has landed
#pragma unroll
    for (int s = 0; s < kStages; ++s) {
      if (!issued[s]) continue;
      const long long t0 = clock64();
      while (!mbar_try(bar_full + 8 * s, last_use[s] & 1u) && clock64() - t0 < kTimeoutCycles / 4) {
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (*abort && threadIdx.x == 0) set_status(a.dev_status, DSPARK_ERR_DEVICE_TIMEOUT);
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
  }
  return fn;
}

// Once per call, after the last position: tokens from the packed maxima and the
// normaliser from the CTA partials of each (request, position), one warp each.
__global__ void __launch_bounds__(256) draft_tc_finalize(const __grid_constant__ DraftArgs a, int G) {
  if (read_status(a.dev_status)) return;
  const int K = (int)a.K_max, B = (int)a.B;
  const int n_tiles = (int)((a.V + kTileN - 1) / kTileN);
  const int lane = threadIdx.x & 31;
  const int64_t nw = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t item = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; item < (int64_t)B * K; item += nw) {
    const int k = (int)(item / B) + 1, i = (int)(item % B);
    const int n_k = a.nact[k];
    if (i >= n_k) continue;
    const int m_tiles = (n_k + kTileM - 1) / kTileM;
    const int gm = max(1, min(G / m_tiles, n_tiles));
    const int r = a.perm[i];
    const Partial *ptr[1] = {a.partials + (int64_t)(k - 1) * kTcPartialsPerStep + (int64_t)i * gm};
    Race tot[1];
    warp_merge_rows<1>(ptr, gm, tot);
    if (lane == 0) {
      const unsigned long long key = a.best_key[(int64_t)r * K + k - 1];
      a.draft_tok[(int64_t)r * K + k - 1] = key_index(key);
      if (a.draft_lse)
        a.draft_lse[(int64_t)r * K + k - 1] = a.temperature[r] == 0.0f ? tot[0].best : tot[0].m + logf(tot[0].S);
    }
  }
}

}  // namespace

bool draft_tc_supported(const DraftArgs &a) {
  if (a.dtype != DSPARK_BF16) return false;
  if (a.rank % 64 != 0 || a.rank > 256) return false;
  if (a.V % 8 != 0 || a.V > (int64_t)INT32_MAX - 64) return false;
  if (((uintptr_t)a.U | (uintptr_t)a.E | (uintptr_t)a.W) & 15u) return false;
  if (a.draft_logits && ((uintptr_t)a.draft_logits & 15u)) return false;
  // partial slots of one position: (M-tiles x 128 rows) x CTAs per M-tile <= 128 x max(grid, M-tiles)
  const int64_t m_tiles = (a.B + kTileM - 1) / kTileM;
  const int64_t units = m_tiles > 1024 ? m_tiles : 1024;
  if (units * kTileM > kTcPartialsPerStep) return false;
  if (a.K_max * kTcPartialsPerStep > a.partial_slots) return false;
  return get_encode() != nullptr;
}

cudaError_t launch_draft_tc(const DraftArgs &a, cudaStream_t s, int num_sms) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = get_encode();
  if (!encode) return cudaErrorNotSupported;
  CUtensorMap tmap;
  const cuuint64_t gdim[2] = {(cuuint64_t)a.V, (cuuint64_t)a.rank};
  const cuuint64_t gstride[1] = {(cuuint64_t)a.V * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kTileN, (cuuint32_t)a.rank};
  const cuuint32_t estride[2] = {1, 1};
  CUresult cr = encode(&tmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(a.W), gdim, gstride, box,
                       estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (cr != CUDA_SUCCESS) return cudaErrorInvalidValue;
  static bool attr_set[5] = {false, false, false, false, false};
  const int rch = (int)(a.rank / 64);
  void *fn = nullptr;
  switch (rch) {
    case 1: fn = (void *)draft_tc_persistent<1>; break;
    case 2: fn = (void *)draft_tc_persistent<2>; break;
    case 3: fn = (void *)draft_tc_persistent<3>; break;
    default: fn = (void *)draft_tc_persistent<4>; break;
  }
  if (!attr_set[rch]) {
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set[rch] = true;
  }
  const int grid = num_sms > 1024 ? 1024 : num_sms;
  // cooperative launch: all CTAs are co-resident, so the bounded grid barrier between
  // positions can always complete
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3(kThreadsTc, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void *args[2] = {(void *)&a, (void *)&tmap};
  cudaError_t e = cudaLaunchKernelExC(&cfg, fn, args);
  if (e != cudaSuccess) return e;
  const int64_t items = a.B * a.K_max;
  const int fblocks = (int)((items + 7) / 8 < 4096 ? (items + 7) / 8 : 4096);
  draft_tc_finalize<<<fblocks, 256, 0, s>>>(a, grid);
  return cudaGetLastError();
}

}  // namespace dspark
