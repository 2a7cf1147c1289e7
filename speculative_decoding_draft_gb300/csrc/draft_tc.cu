// Markov-head draft sampling, tensor-core path (sm_103a: tcgen05 + bulk copies + TMEM).
//
// "DSpark" S3.1 (Markov head B(x_{k-1}, .) = W1[x_{k-1}] . W2, rank r) and
// "Speculative decoding, from zero to DSpark" S6 (p_k = softmax(U_k + B_k)).
//
// One persistent cooperative launch walks every draft position k = 1..K_max.  The
// active requests at position k (K_r >= k), listed in act[k - 1] with the T > 0 requests
// first and the greedy ones after them, each in request order (warps of one kind of draw;
// rows close together in U), are cut into M-tiles of 128 rows, and every M-tile is shared by gm CTAs that
// own contiguous ranges of 64-wide vocabulary blocks.  A CTA stages the gathered
// operand W1[x_{k-1}] (128 x r) once per range and streams W2 through it.
//
// W2 arrives packed (dspark_draft_pack_projection): block (c, t) holds rank rows
// 64c..64c+63 of vocabulary columns 64t..64t+63 as the 128-byte-swizzled image of
// the MN-major tensor-core operand, and the blocks of one rank chunk are
// consecutive, so the up-to-four blocks of one MMA tile and one rank chunk are a
// single contiguous bulk copy.
//
// Warp roles (320 threads):
//   warp 0     producer: per tile (N = 64 m columns, m <= 4) and rank chunk, one
//              bulk copy of m x 8 KB into a 32 KB stage.
//   warp 1     allocates TMEM (two accumulators of 128 x 256 fp32) and one elected
//              lane issues the tcgen05.mma (kind::f16, bf16 in, fp32 accumulate, A
//              K-major, B MN-major, both from shared memory, M = 128, N = 64 m).
//   warps 2-9  epilogue, two warps per TMEM lane quadrant: gather W1[x_{k-1}] into
//              the swizzled A operand, then per 32-column block tcgen05.ld the bias,
//              add U, round to bf16, optionally store the logits, and run the
//              two-level draw (or the greedy argmax) with the online softmax.
// With fewer than 128 rows the rows are replicated F times in the M-tile and the F
// replica groups split each tile's columns.  Per row, the CTA's maximum goes into
// a packed 64-bit (score, index) key by atomicMax; a bounded grid barrier separates
// positions; after the last one the epilogue warps turn keys and partial normalisers
// into tokens and log-sum-exps.  Every wait is bounded; on a timeout the kernel records
// DSPARK_ERR_DEVICE_TIMEOUT, drains what it issued, frees TMEM and returns.
#include "dspark_internal.cuh"

namespace dspark {
namespace {

constexpr int kTileM = 128;
constexpr int kBlkN = 64;                        // vocabulary columns per packed block
constexpr int kMaxBlk = 4;                       // blocks per MMA tile (N <= 256)
constexpr int kAccBufs = 2;
constexpr int kAccCols = kBlkN * kMaxBlk;        // 256
constexpr int kTmemCols = kAccBufs * kAccCols;   // 512
constexpr int kAChunk = kTileM * 128;            // 16 KB: 128 rows x 64 rank values
constexpr int kASize = 4 * kAChunk;              // rank <= 256
constexpr int kPiece = kBlkN * 128;              // 8 KB: one packed block, 64 rank rows
constexpr int kStageBytes = kMaxBlk * kPiece;    // 32 KB
constexpr int kUSlot = 32 * 64;                  // one 32-wide block of a warp's 32 rows (2 KB)
constexpr int kOffA = 0;
constexpr int kOffW = kOffA + kASize;

// Per mode: epilogue warps (three per TMEM lane quadrant for the draft, which fits 128
// registers a thread; two for the residual mode, which needs 168), the U blocks each
// epilogue warp stages ahead, and W2 stages: three in both (the draft's U ring of two blocks
// per warp measured as fast as three and leaves room for the third stage, which took 2 % off
// the draft at B = 64 and changed nothing at large batches).
template <bool RESID>
struct TcCfg {
  static constexpr int kEpiWarps = RESID ? 8 : 12;
  static constexpr int kWpq = kEpiWarps / 4;     // epilogue warps per TMEM lane quadrant
  static constexpr int kThreads = 32 * (2 + kEpiWarps);
  static constexpr int kUDepth = RESID ? 3 : 2;
  static constexpr int kStages = 3;
  static constexpr int kOffUr = kOffW + kStages * kStageBytes;
  static constexpr int kOffSh = kOffUr + kEpiWarps * kUDepth * kUSlot;
};

template <int EPI, int NST>
struct TcShared {
  uint64_t full[NST];
  uint64_t empty[NST];
  uint64_t accf[kAccBufs];
  uint64_t acce[kAccBufs];
  uint64_t aready;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int skip;
  int nact[kMaxK + 2];        // active requests per position (copied once per launch)
  int row_req[kTileM];
  int row_prev[kTileM];
  float row_invT[kTileM];
  Partial part[EPI / 4 * kTileM];   // per-row partials: [column worker][row of the replica group]
  float part_zx[EPI / 4 * kTileM];  // the logit at each partial's index (residual mode: "some p > q")
  int row_urow[kTileM];        // the row of U (of the base logits) each M-tile row reads
  // residual mode: per row the rejecting position, the target row, and the log2-scaled
  // normalisers of p and q
  int row_j[kTileM], row_trow[kTileM];
  float row_lt2[kTileM], row_lq2[kTileM];
};

template <bool RESID>
constexpr int tc_smem_bytes() {
  return TcCfg<RESID>::kOffSh + (int)sizeof(TcShared<TcCfg<RESID>::kEpiWarps, TcCfg<RESID>::kStages>) + 1024;
}
static_assert(tc_smem_bytes<false>() <= 232448 && tc_smem_bytes<true>() <= 232448, "shared memory budget");

// ---- PTX wrappers (the mbarrier and bulk-copy ones are in dspark_internal.cuh) ----
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

__device__ __forceinline__ void st_u4_hint(void *ptr, uint4 v, uint64_t policy) {
  asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(ptr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w), "l"(policy)
               : "memory");
}
// z = bf16 value + fp32 value, rounded once to fp32, for the two halves of a bf16 pair
// word (low half first).
__device__ __forceinline__ void add_bf16x2_f32(uint32_t w, float a0, float a1, float &z0, float &z1) {
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tadd.rn.f32.bf16 %0, l, %3;\n\tadd.rn.f32.bf16 %1, h, %4;\n\t}"
      : "=f"(z0), "=f"(z1)
      : "r"(w), "f"(a0), "f"(a1));
}

// 32-byte (one whole sector) global store, 32-byte aligned address.
__device__ __forceinline__ void st_u8_hint(void *ptr, uint4 lo, uint4 hi, uint64_t policy) {
  asm volatile("st.global.L2::cache_hint.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8}, %9;" ::"l"(ptr), "r"(lo.x),
               "r"(lo.y), "r"(lo.z), "r"(lo.w), "r"(hi.x), "r"(hi.y), "r"(hi.z), "r"(hi.w), "l"(policy)
               : "memory");
}
// 16-byte global -> shared asynchronous copy (L1 bypassed) with an L2 policy; its
// completion is tracked by the thread's commit groups.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint64_t policy) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "l"(policy)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

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
// B MN-major, M = 128; N (a multiple of 64 here) goes into bits 17..22 as N >> 3.
constexpr uint32_t kIdescBase = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 16) | ((uint32_t)(kTileM >> 4) << 24);
__device__ __forceinline__ uint32_t idesc_n(int n) { return kIdescBase | ((uint32_t)(n >> 3) << 17); }

__device__ __forceinline__ __nv_bfloat162 bf162_of(uint32_t w) { return *reinterpret_cast<const __nv_bfloat162 *>(&w); }

template <int EPI>
__device__ __forceinline__ void named_sync_epi() {
  asm volatile("bar.sync 1, %0;" ::"n"(EPI * 32) : "memory");
}

// Work split of one draft position: M-tiles of 128 active rows, each shared by gm CTAs
// that own contiguous ranges of 64-wide vocabulary blocks.  The ranges start at even blocks
// (128 columns), so a range's 32-wide draw blocks fall into the random stream's groups of four
// (one Philox call each) the same way in every range.
struct StepPlan {
  int n_k, m_tiles, gm, units;
};
__device__ __forceinline__ StepPlan plan_step(const int *nact, int k, int G, int nb) {
  StepPlan p;
  p.n_k = nact[k];
  p.m_tiles = (p.n_k + kTileM - 1) / kTileM;
  p.gm = p.m_tiles ? max(1, min(G / p.m_tiles, (nb + 1) / 2)) : 1;
  p.units = p.m_tiles * p.gm;
  return p;
}
__device__ __forceinline__ int range_lo(int j, int nb, int gm) {
  return j >= gm ? nb : 2 * (int)((int64_t)j * ((nb + 1) / 2) / gm);
}

// ---------------------------------------------------------------------------
// RESID: the residual mode of the recompute verification -- one position whose rows are the
// jobs; per row z = U + W1[x_{j-1}] W2 is formed exactly as the draft formed it, and the
// two-level draw runs over max(0, p - q) (streams of the verification's seed, position j, tags
// 2 and 4) instead of softmax(z / T); the winner goes into the request's packed key and a
// positive residual anywhere into its flag.
template <int RCH, bool RESID>   // rank / 64
__global__ void __launch_bounds__(TcCfg<RESID>::kThreads, 1) draft_tc_persistent(const __grid_constant__ DraftArgs a) {
  constexpr int kRank = RCH * 64;
  constexpr int kEpiWarps = TcCfg<RESID>::kEpiWarps;
  constexpr int kWpq = TcCfg<RESID>::kWpq;
  constexpr int kStages = TcCfg<RESID>::kStages;
  constexpr int NS = kStages;
  constexpr int kOffUr = TcCfg<RESID>::kOffUr;
  constexpr int kOffSh = TcCfg<RESID>::kOffSh;
  using Shared = TcShared<kEpiWarps, kStages>;
  constexpr int kUDepth = TcCfg<RESID>::kUDepth;
  constexpr int kLook = kUDepth;
  constexpr int kUpr = kRank / 8;                  // 16-byte units per W1 row
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;
  uint8_t *gb = smem_raw + (sb - raw);
  Shared &sh = *reinterpret_cast<Shared *>(gb + kOffSh);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) sh.skip = read_status(a.dev_status);
  __syncthreads();
  if (sh.skip) return;   // an earlier error: every CTA sees the same word and leaves

  const int K = (int)a.K_max, V = (int)a.V;
  const int G = gridDim.x;
  const int nb = (V + kBlkN - 1) / kBlkN;          // 64-wide vocabulary blocks
  const uint8_t *Wp = (const uint8_t *)a.Wp;

  const uint32_t bar_full = smem_u32(&sh.full[0]);
  const uint32_t bar_empty = smem_u32(&sh.empty[0]);
  const uint32_t bar_accf = smem_u32(&sh.accf[0]);
  const uint32_t bar_acce = smem_u32(&sh.acce[0]);
  const uint32_t bar_aready = smem_u32(&sh.aready);
  const uint32_t bar_drain = smem_u32(&sh.drain);
  volatile int *abort = &sh.abort;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
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
  if (threadIdx.x < kMaxK + 2) sh.nact[threadIdx.x] = threadIdx.x <= K + 1 ? a.nact[threadIdx.x] : 0;
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
    // ---------------- producer: W2 stages of every position ----------------
    // The warp walks the positions in lockstep (abort decided by lane 0 for all lanes);
    // lane 0 issues the copies.
    const uint64_t pol_w = policy_evict_last();
    uint32_t it = 0;
    for (int k = 1; k <= K; ++k) {
      if (__shfl_sync(0xffffffffu, *abort ? 1 : 0, 0)) break;
      const StepPlan pl = plan_step(sh.nact, k, G, nb);
      if (pl.n_k == 0) break;
      if (lane == 0)
      for (int u = blockIdx.x; u < pl.units && !*abort; u += G) {
        const int j = u % pl.gm;
        const int b0 = range_lo(j, nb, pl.gm), b1 = range_lo(j + 1, nb, pl.gm);
        for (int bt = b0; bt < b1 && !*abort; bt += kMaxBlk) {
          const int m = min(kMaxBlk, b1 - bt);
          for (int c = 0; c < RCH; ++c, ++it) {
            const int s = (int)(it % NS);
            const uint32_t use = it / NS;
            if (!mbar_wait(bar_empty + 8 * s, (use & 1u) ^ 1u, abort)) break;
            mbar_arrive_tx(bar_full + 8 * s, (uint32_t)(m * kPiece));
            bulk_g2s(sb + kOffW + s * kStageBytes, Wp + ((int64_t)c * nb + bt) * kPiece, (uint32_t)(m * kPiece),
                     bar_full + 8 * s, pol_w);
#pragma unroll
            for (int q = 0; q < kStages; ++q)
              if (q == s) { last_use[q] = use; issued[q] = true; }
          }
        }
      }
      __syncwarp();
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      uint32_t it = 0, tt = 0;
      int unit_no = 0;
      bool ok = true;
      for (int k = 1; k <= K && ok; ++k) {
        const StepPlan pl = plan_step(sh.nact, k, G, nb);
        if (pl.n_k == 0) break;
        for (int u = blockIdx.x; u < pl.units && ok; u += G, ++unit_no) {
          const int j = u % pl.gm;
          const int b0 = range_lo(j, nb, pl.gm), b1 = range_lo(j + 1, nb, pl.gm);
          ok = mbar_wait(bar_aready, (uint32_t)(unit_no & 1), abort);
          for (int bt = b0; ok && bt < b1; bt += kMaxBlk, ++tt) {
            const int m = min(kMaxBlk, b1 - bt);
            const int b = (int)(tt % kAccBufs);
            const uint32_t ause = tt / kAccBufs;
            if (!(ok = mbar_wait(bar_acce + 8 * b, (ause & 1u) ^ 1u, abort))) break;
            tc_fence_after();
            const uint32_t d = tmem + (uint32_t)(b * kAccCols);
            const uint32_t idesc = idesc_n(m * kBlkN);
            for (int c = 0; ok && c < RCH; ++c, ++it) {
              const int s = (int)(it % NS);
              const uint32_t use = it / NS;
              if (!(ok = mbar_wait(bar_full + 8 * s, use & 1u, abort))) break;
              tc_fence_after();
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                const uint64_t ad = smem_desc(sb + kOffA + c * kAChunk + kk * 32, 16, 1024);
                const uint64_t bd = smem_desc(sb + kOffW + s * kStageBytes + kk * 2048, kPiece, 1024);
                mma_bf16(d, ad, bd, idesc, (c | kk) ? 1u : 0u);
              }
              mma_commit(bar_empty + 8 * s);
            }
            if (ok) mma_commit(bar_accf + 8 * b);
          }
        }
      }
    }
    __syncwarp();
  } else {
    // ---------------- epilogue ----------------
    const int eq = warp - 2;            // 0 .. kEpiWarps - 1
    const int quad = warp & 3;          // TMEM lanes 32*quad .. +31 are reachable by this warp
    const int wq = eq >> 2;             // this warp's rank among the warps of its quadrant
    const int et = eq * 32 + lane;      // 0 .. 32 kEpiWarps - 1
    const uint64_t pol_stream = policy_evict_first();
    // every lane stores to another row, so the logits go out in whole 32-byte sectors where
    // the rows start on 32-byte boundaries (V % 16 == 0 from a 32-byte aligned base)
    const bool wide_s = (V % 16 == 0) && ((uintptr_t)a.draft_logits % 32 == 0);
    uint32_t tt = 0;
    int unit_no = 0;
    int tab_m = -1;                     // (position, M-tile) whose rows sh.row_req / sh.row_invT hold
    int k_last = 0;                     // last position this CTA arrived at
    for (int k = 1; k <= K && !*abort; ++k) {
      const StepPlan pl = plan_step(sh.nact, k, G, nb);
      if (pl.n_k == 0) break;
      bool waited = (k == 1);
      for (int u = blockIdx.x; u < pl.units && !*abort; u += G, ++unit_no) {
        const int m = u / pl.gm, j = u % pl.gm;
        const int b0 = range_lo(j, nb, pl.gm), b1 = range_lo(j + 1, nb, pl.gm);
        const int row0 = m * kTileM;
        const int nrows = min(kTileM, pl.n_k - row0);
        // replication: with few rows, every TMEM lane quadrant (= SM sub-partition) gets a copy
        // of the rows, and the F replica groups split each tile's columns
        const int F = nrows <= 32 ? 4 : (nrows <= 64 ? 2 : 1);
        const int rpg = kTileM / F;
        if (k * 65536 + m != tab_m) {    // the same decision in every epilogue thread
          // rows of M-tile m at position k (a run of the position's active list, in request
          // order) and their 1/T
          named_sync_epi<kEpiWarps>();           // readers of the previous table are done
          if (et < kTileM) {
            const int i = et;
            if (RESID && row0 + i < pl.n_k) {
              const VJob jb = a.jobs[row0 + i];
              sh.row_req[i] = (int)bchk(jb.r, a.B, a.dev_status);
              sh.row_invT[i] = jb.invT;
              sh.row_j[i] = jb.j;
              sh.row_urow[i] = (int)bchk(jb.urow, a.u_rows, a.dev_status);
              sh.row_trow[i] = jb.trow;
              sh.row_lt2[i] = jb.lse_t * kLog2e;
              sh.row_lq2[i] = jb.lse_q * kLog2e;
            } else if (row0 + i < pl.n_k) {
              const int r = (int)bchk(a.act[(int64_t)(k - 1) * a.B + row0 + i], a.B, a.dev_status);
              sh.row_req[i] = r;
              sh.row_urow[i] = r * K + (k - 1);
              const float T = a.temperature[r];
              sh.row_invT[i] = (T == 0.0f) ? 0.0f : 1.0f / T;
            } else {
              sh.row_req[i] = -1;
              sh.row_urow[i] = 0;
              if (RESID) sh.row_trow[i] = 0;
              sh.row_invT[i] = 0.0f;
            }
          }
          named_sync_epi<kEpiWarps>();
          tab_m = k * 65536 + m;
        }
        const int arow = quad * 32 + lane;        // TMEM lane = M-row
        const int grp = arow / rpg;               // replica group (warp-uniform: rpg >= 32)
        const int row = arow % rpg;               // request row of this thread
        const int wk = grp * kWpq + wq;           // column worker of this warp
        const int nwk = kWpq * F;
        const bool valid = row < nrows;
        const int r = valid ? sh.row_req[row] : 0;
        const float invT = sh.row_invT[row];
        const bool greedy = (invT == 0.0f);
        const float a2 = invT * kLog2e;           // scaled logits in log2 units
        const int64_t urow = (int64_t)sh.row_urow[row] * V;   // this thread's row of U and of the logits
        // residual mode: the stream position and the normalisers
        const uint32_t rpos = RESID ? (uint32_t)(valid ? sh.row_j[row] : 0) : (uint32_t)k;
        const float lt2 = RESID ? sh.row_lt2[row] : 0.0f, lq2 = RESID ? sh.row_lq2[row] : 0.0f;
        bool any_pos = false;
        // the unit's 32-wide blocks are numbered 0 .. 2 (b1 - b0) - 1 across its tiles, in groups
        // of 4 / F consecutive blocks (a tile of 8 blocks holds 2F groups); worker wk takes groups
        // wk, wk + nwk, ... across the tiles.  Four consecutive blocks from an even 64-wide block
        // share one Philox call, which a worker then computes once per group.  The worker's i-th block gsb_of(i)'s U (64 bytes of each of the warp's 32
        // rows) is staged into slot i % kUDepth of the warp's ring kUDepth blocks ahead by
        // cp.async.  Four lanes copy one row's 64 contiguous bytes, so each instruction touches 8
        // rows: with one row per lane every instruction touched 32 rows far apart in memory, and
        // the ragged draft (rows of the active requests, scattered) ran 1.5x slower than the same
        // work on consecutive rows.  16-byte unit q of row l sits at l * 64 + ((q ^ ((l >> 1) & 3))
        // << 4), which keeps the quarter-warp reads and writes free of bank conflicts.  Every lane
        // commits one group per block, so wait_group(kUDepth - 1) and a warp barrier mean the
        // oldest staged block has landed for the whole warp.
        const int nsub_u = 2 * (b1 - b0);
        const int gsh = F == 1 ? 2 : (F == 2 ? 1 : 0);      // log2 of the group size
        auto gsb_of = [&](int i) { return (((i >> gsh) * nwk + wk) << gsh) + (i & ((1 << gsh) - 1)); };
        const uint32_t uring0 = sb + kOffUr + (uint32_t)(eq * kUDepth * kUSlot);
        const uint32_t uring = uring0 + (uint32_t)(lane * 64);
        const int usw = (lane >> 1) & 3;
        const int cq = lane & 3;                  // the 16-byte unit this lane copies of each row
        const uint32_t vmask = __ballot_sync(0xffffffffu, valid);
        const int rb = row - lane;                // the warp's first row (rows rb .. rb + 31)
        // the U rows this lane copies: kept in registers for the unit, except in the residual
        // mode, whose extra target registers leave no room (there they come from the row table)
        const unsigned short *uptr_l[4];
        if constexpr (!RESID) {
#pragma unroll
          for (int p = 0; p < 4; ++p)
            uptr_l[p] = (const unsigned short *)a.U + (int64_t)sh.row_urow[rb + p * 8 + (lane >> 2)] * V;
        }
        auto stage_u = [&](int i) {    // U of the worker's i-th block
          const int gsb = gsb_of(i);
          if (gsb < nsub_u) {
            const int c = b0 * kBlkN + gsb * 32 + 8 * cq;
            const uint32_t slot = uring0 + (uint32_t)((i % kUDepth) * kUSlot);
#pragma unroll
            for (int p = 0; p < 4; ++p) {
              const int l = p * 8 + (lane >> 2);
              const unsigned short *src;
              if constexpr (RESID) src = (const unsigned short *)a.U + (int64_t)sh.row_urow[rb + l] * V;
              else src = uptr_l[p];
              if (((vmask >> l) & 1u) && c < V)
                cp_async16(slot + (uint32_t)(l * 64) + (uint32_t)((cq ^ ((l >> 1) & 3)) << 4), src + c, pol_stream);
            }
          }
          cp_async_commit();
        };
#pragma unroll
        for (int i = 0; i < kLook; ++i) stage_u(i);   // before the barrier: U does not depend on the tokens
        int ui = 0;                                    // this worker's blocks consumed in the unit
        if (!waited) {
          // every CTA has folded its position k-1 maxima into the packed keys
          if (et == 0) {
            const long long t0 = clock64();
            while (ld_acquire(a.gbar + (k - 1)) < G + (k == 2 ? a.gbar_extra : 0)) {
              __nanosleep(100);        // back off: many pollers slow the CTAs still working
              if (*abort) break;
              if (clock64() - t0 > kTimeoutCycles) { *abort = 1; break; }
            }
          }
          named_sync_epi<kEpiWarps>();
          waited = true;
          if (*abort) break;
        }
        if (et < kTileM && et < nrows) {
          const int rq = sh.row_req[et];
          sh.row_prev[et] = (int)bchk(RESID ? a.jobs[row0 + et].prev
                                            : ((k == 1) ? a.anchor[rq]
                                                        : key_index(load_key(a.best_key + (int64_t)rq * K + k - 2))),
                                      V, a.dev_status);
        }
        named_sync_epi<kEpiWarps>();
        // gather the A operand with asynchronous 16-byte copies, all in flight at once: request
        // row i's unit c8 of K-chunk c goes to every replica M-row ar = g * rpg + i, chunk c,
        // unit (c8 ^ (ar & 7)) -- the 128-byte swizzle
        {
          const int total = nrows * kUpr;
          for (int e = et; e < total; e += kEpiWarps * 32) {
            const int i = e / kUpr, uu = e % kUpr;
            const int c = uu >> 3, c8 = uu & 7;
            const uint4 *src = (const uint4 *)((const unsigned short *)a.E + (int64_t)sh.row_prev[i] * kRank) + uu;
            for (int g = 0; g < F; ++g) {
              const int ar = g * rpg + i;
              const uint32_t dst = sb + kOffA + c * kAChunk + ar * 128 + ((c8 ^ (ar & 7)) << 4);
              asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
            }
          }
          asm volatile("cp.async.wait_all;" ::: "memory");
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_aready);

        BRace st;
        brace_init(st);
        // residual mode: the target block of this worker's next 32 columns, one block ahead in
        // registers (units past V read as -inf, so their weights are 0).  The first block of the
        // unit is loaded row by row; later blocks are loaded two ahead like U, four lanes per row
        // (traw: unit cq of rows p * 8 + lane / 4), and passed to their rows' lanes through the
        // U slot just consumed, before it is refilled.
        const uint4 kNegInf4 = make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
        uint4 tcur[4], tnext[4], traw[4];
        if (RESID) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int c = b0 * kBlkN + gsb_of(0) * 32 + 8 * q;
            tcur[q] = (valid && gsb_of(0) < nsub_u && c + 8 <= V)
                          ? __ldcs((const uint4 *)((const unsigned short *)a.tgt + ((int64_t)sh.row_trow[row] * V + c)))
                          : kNegInf4;
          }
        }
        auto load_traw = [&](int gsb) {
          const int c = b0 * kBlkN + gsb * 32 + 8 * cq;
#pragma unroll
          for (int p = 0; p < 4; ++p) {
            const int l = p * 8 + (lane >> 2);
            traw[p] = (((vmask >> l) & 1u) && gsb < nsub_u && c + 8 <= V)
                          ? __ldcs((const uint4 *)((const unsigned short *)a.tgt + ((int64_t)sh.row_trow[rb + l] * V + c)))
                          : kNegInf4;
          }
        };
        if (RESID) load_traw(gsb_of(1));
        uint4 pw = make_uint4(0u, 0u, 0u, 0u);   // the last Philox output of this thread's row
        uint32_t pctr = 0xffffffffu;              // ... and its counter (a block group)
        for (int bt = b0; bt < b1; bt += kMaxBlk, ++tt) {
          const int mt = min(kMaxBlk, b1 - bt);
          const int b = (int)(tt % kAccBufs);
          const uint32_t ause = tt / kAccBufs;
          if (!mbar_wait(bar_accf + 8 * b, ause & 1u, abort)) break;
          tc_fence_after();
          const int s0 = 2 * (bt - b0), s1 = s0 + 2 * mt;   // the tile's blocks in unit numbering
          int gs = gsb_of(ui);                               // this worker's first block in the tile
          if (gs >= s1) {                         // nothing for this worker in this tile
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_acce + 8 * b);
            continue;
          }
          for (; gs < s1; gs = gsb_of(++ui)) {
            uint32_t acc[32];
            tmem_ld32(tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(b * kAccCols + (gs - s0) * 32), acc);
            tmem_wait_ld();
            if (gsb_of(ui + 1) >= s1) {           // this warp's last read of the accumulator
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(bar_acce + 8 * b);
            }
            cp_async_wait<kLook - 1>();             // block ui's U has landed (this lane's copies)
            __syncwarp();                           // ... and every lane's
            uint4 ucur[4];
            {
              const uint32_t src = uring + (uint32_t)((ui % kUDepth) * kUSlot);
#pragma unroll
              for (int q = 0; q < 4; ++q) ucur[q] = ld_shared_u4(src + ((q ^ usw) << 4));
            }
            const int c0 = b0 * kBlkN + gs * 32;      // this thread's 32-wide block of the two-level draw
            uint32_t packed[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              float z0, z1;
              add_bf16x2_f32(word_of(ucur[e >> 2], e & 3), __uint_as_float(acc[2 * e]),
                             __uint_as_float(acc[2 * e + 1]), z0, z1);
              const __nv_bfloat162 zb = __floats2bfloat162_rn(z0, z1);   // one rounding of each fp32 sum
              packed[e] = *reinterpret_cast<const uint32_t *>(&zb);
            }
            __syncwarp();                            // every lane has read the slot
            if (RESID) {                             // the next block's target rows, through the slot
              const uint32_t slot = uring0 + (uint32_t)((ui % kUDepth) * kUSlot);
#pragma unroll
              for (int p = 0; p < 4; ++p) {
                const int l = p * 8 + (lane >> 2);
                st_shared_u4(slot + (uint32_t)(l * 64) + (uint32_t)((cq ^ ((l >> 1) & 3)) << 4), traw[p]);
              }
              __syncwarp();
#pragma unroll
              for (int q = 0; q < 4; ++q) tnext[q] = ld_shared_u4(uring + (uint32_t)((ui % kUDepth) * kUSlot) + ((q ^ usw) << 4));
              __syncwarp();
              load_traw(gsb_of(ui + 2));
            }
            stage_u(ui + kLook);                     // the slot is free again: refill it
            if (!valid) continue;
            if (a.draft_logits) {
              unsigned short *drow = (unsigned short *)a.draft_logits + urow;
              if (wide_s) {                           // whole sectors: 32-byte stores
#pragma unroll
                for (int h = 0; h < 2; ++h)
                  if (c0 + 16 * h + 16 <= V)
                    st_u8_hint(drow + c0 + 16 * h,
                               make_uint4(packed[8 * h], packed[8 * h + 1], packed[8 * h + 2], packed[8 * h + 3]),
                               make_uint4(packed[8 * h + 4], packed[8 * h + 5], packed[8 * h + 6], packed[8 * h + 7]),
                               pol_stream);
              } else {
#pragma unroll
                for (int g = 0; g < 4; ++g)
                  if (c0 + g * 8 + 8 <= V)
                    st_u4_hint(drow + c0 + g * 8,
                               make_uint4(packed[4 * g], packed[4 * g + 1], packed[4 * g + 2], packed[4 * g + 3]),
                               pol_stream);
              }
            }
            if (c0 + 32 > V) {                        // ragged tail: whole pairs past V (V is even)
#pragma unroll
              for (int e = 0; e < 16; ++e)
                if (c0 + 2 * e >= V) packed[e] = 0xFF80FF80u;   // two bf16 -inf
            }
            if (RESID) {
              // residual weights max(0, p - q) of the block against the target row
              const uint4 dp[4] = {make_uint4(packed[0], packed[1], packed[2], packed[3]),
                                   make_uint4(packed[4], packed[5], packed[6], packed[7]),
                                   make_uint4(packed[8], packed[9], packed[10], packed[11]),
                                   make_uint4(packed[12], packed[13], packed[14], packed[15])};
              const uint32_t gblk = (uint32_t)c0 >> 5;
              if ((gblk >> 2) != pctr) {
                pctr = gblk >> 2;
                pw = philox(a.key, pctr, rpos, (uint32_t)r, kTagResid);
              }
              const uint32_t wb = word_of(pw, (int)(gblk & 3u));
              brace_resid_packed(st, tcur, dp, a2, lt2, lq2, wb, c0, any_pos, [&] {
                return word_of(philox(a.key, gblk >> 2, rpos, (uint32_t)r, kTagResidPick), (int)(gblk & 3u));
              });
#pragma unroll
              for (int q = 0; q < 4; ++q) tcur[q] = tnext[q];
              continue;
            }
            // block maximum on bf16 pairs (exact), then across the pair
            __nv_bfloat162 m2[4] = {bf162_of(packed[0]), bf162_of(packed[1]), bf162_of(packed[2]), bf162_of(packed[3])};
#pragma unroll
            for (int e = 4; e < 16; ++e) m2[e & 3] = __hmax2(m2[e & 3], bf162_of(packed[e]));
            m2[0] = __hmax2(__hmax2(m2[0], m2[1]), __hmax2(m2[2], m2[3]));
            const float mz = fmaxf(__low2float(m2[0]), __high2float(m2[0]));
            if (greedy) {
              float z[32];
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                z[2 * e] = __uint_as_float(packed[e] << 16);
                z[2 * e + 1] = __uint_as_float(packed[e] & 0xffff0000u);
              }
              brace_argmax_block(st, z, mz, c0);
            } else {
              const uint32_t gblk = (uint32_t)c0 >> 5;
              if ((gblk >> 2) != pctr) {
                pctr = gblk >> 2;
                pw = philox(a.key, pctr, (uint32_t)k, (uint32_t)r, kTagDraft);
              }
              const uint32_t wb = word_of(pw, (int)(gblk & 3u));
              brace_softmax_bf16x32(st, packed, mz, a2, wb, c0, [&] {
                return word_of(philox(a.key, gblk >> 2, (uint32_t)k, (uint32_t)r, kTagDraftPick), (int)(gblk & 3u));
              });
            }
          }
        }
        cp_async_wait<0>();                         // nothing of this unit stays in flight
        // merge the 2F worker partials of each row; the row's home thread folds its maximum
        // into the packed (score, index) key of the position with one 64-bit atomicMax -- all
        // the next position needs -- and keeps its softmax partial for the merge after the last position
        sh.part[wk * rpg + row] = to_partial(st);
        sh.part_zx[wk * rpg + row] = RESID ? (any_pos ? 1.0f : 0.0f) : st.zx;
        named_sync_epi<kEpiWarps>();
        if (RESID && wk == 0 && valid) {
          // the row's residual draw: the CTA's winner into the request's key, its flag
          Race tot = from_partial(sh.part[row]);
          bool any = sh.part_zx[row] != 0.0f;
          for (int q = 1; q < nwk; ++q) {
            race_merge(tot, from_partial(sh.part[q * rpg + row]));
            any = any || sh.part_zx[q * rpg + row] != 0.0f;
          }
          if (tot.idx >= 0) atomicMax(&a.best_key[r], score_key(tot.best, tot.idx));
          if (any) atomicOr(a.resid_any + r, 1);
        } else if (!RESID && wk == 0 && valid) {
          Race tot = from_partial(sh.part[row]);
          float zx = sh.part_zx[row];
          for (int q = 1; q < nwk; ++q) {
            const Race o = from_partial(sh.part[q * rpg + row]);
            if (o.best > tot.best || (o.best == tot.best && o.idx >= 0 && (tot.idx < 0 || o.idx < tot.idx)))
              zx = sh.part_zx[q * rpg + row];      // race_merge takes o's index
            race_merge(tot, o);
          }
          if (tot.idx >= 0) atomicMax(&a.best_key[(int64_t)r * K + k - 1], score_key(tot.best, tot.idx));
          // the CTA's partial for the final merge: the logit at its index (for greedy rows that is
          // the CTA's maximum), the index, the softmax pair
          Partial pp = to_partial(tot);
          pp.best = zx;
          a.partials[bchk((int64_t)(k - 1) * kTcPartialsPerStep + ((int64_t)m * kTileM + row) * pl.gm + j,
                          a.partial_slots, a.dev_status)] = pp;
        }
      }
      // this CTA is done with position k (every CTA arrives, with or without work): the
      // barrier gathers the epilogue's atomics, the arriving thread's fence releases them
      named_sync_epi<kEpiWarps>();
      if (et == 0) {
        __threadfence();
        atomicAdd(a.gbar + k, 1);
      }
      k_last = k;
    }
    // Once every CTA has arrived at the last position: the tokens from the packed maxima,
    // the normalisers from the CTA partials and, when asked for, the confidence head's
    // output (its Markov term needs the previous position's token), one warp per
    // (position, request).
    if (!RESID && k_last > 0 && !*abort) {
      if (et == 0) {
        const long long t0 = clock64();
        while (ld_acquire(a.gbar + k_last) < G) {
          __nanosleep(100);
          if (*abort) break;
          if (clock64() - t0 > kTimeoutCycles) { *abort = 1; break; }
        }
      }
      named_sync_epi<kEpiWarps>();
      if (!*abort) {
        const int B = (int)a.B;
        const int64_t nw = (int64_t)G * kEpiWarps;
        for (int64_t item = (int64_t)blockIdx.x * kEpiWarps + eq; item < (int64_t)B * K; item += nw) {
          const int k = (int)(item / B) + 1, i = (int)(item % B);
          if (k > k_last) break;
          const StepPlan pl = plan_step(sh.nact, k, G, nb);
          if (i >= pl.n_k) continue;
          const int r = (int)bchk(a.act[(int64_t)(k - 1) * B + i], B, a.dev_status);
          const int64_t at = (int64_t)r * K + k - 1;
          const int x = key_index(load_key(a.best_key + at));
          // the gm CTA partials of the row: softmax pair, greedy maximum (the largest logit
          // field) and the logit of the token x, carried by the one partial whose index is x
          const Partial *pr = a.partials + bchk((int64_t)(k - 1) * kTcPartialsPerStep + (int64_t)i * pl.gm,
                                                a.partial_slots - pl.gm + 1, a.dev_status);
          Race tot;
          race_init(tot);
          float zx = 0.0f;
          bool found = false;
          for (int q = lane; q < pl.gm; q += 32) {
            const Partial p = load_partial(pr + q);
            if (p.idx == x) { zx = p.best; found = true; }
            race_merge(tot, from_partial(p));
          }
#pragma unroll
          for (int d = 16; d > 0; d >>= 1) race_merge(tot, race_shfl_down(tot, d));
          const unsigned fb = __ballot_sync(0xffffffffu, found);
          zx = __shfl_sync(0xffffffffu, zx, fb ? __ffs(fb) - 1 : 0);
          if (a.conf_out) {
            const int prev = (int)bchk(k == 1 ? a.anchor[r] : key_index(load_key(a.best_key + at - 1)), V, a.dev_status);
            const __nv_bfloat16 *erow = (const __nv_bfloat16 *)a.E + (int64_t)prev * a.rank;
            const float c = warp_confidence([&](int q) { return __bfloat162float(erow[q]); }, a.conf_w,
                                            (int)a.rank, a.conf_h[(int64_t)r * K + k - 1], lane);
            if (lane == 0) a.conf_out[(int64_t)r * K + k - 1] = c;
          }
          if (lane == 0) {
            a.draft_tok[at] = x;
            if (a.draft_lse) a.draft_lse[at] = a.temperature[r] == 0.0f ? tot.best : tot.m + logf(tot.S);
            if (a.draft_zx) a.draft_zx[at] = zx;
          }
        }
      }
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
  if (warp >= 2) cp_async_wait<0>();   // U copies still in flight after an abort
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (*abort && threadIdx.x == 0) set_status(a.dev_status, DSPARK_ERR_DEVICE_TIMEOUT);
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// W2 [rank, V] -> packed blocks: 16-byte unit e = ((c * nb + t) * 64 + kr) * 8 + u of
// the output holds W2[64c + kr, 64t + 8u' .. 64t + 8u' + 7] with u' = u ^ (kr & 7);
// columns past V are zero.  V is a multiple of 8.
__global__ void __launch_bounds__(256) pack_projection(const uint4 *__restrict__ W, int64_t rank, int64_t V,
                                                       int nb, uint4 *__restrict__ Wp) {
  const int64_t total = (rank / 64) * (int64_t)nb * 64 * 8;
  const int64_t row_units = V / 8;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += (int64_t)gridDim.x * blockDim.x) {
    const int u = (int)(e & 7), kr = (int)((e >> 3) & 63);
    const int64_t ct = e >> 9;
    const int64_t t = ct % nb, c = ct / nb;
    const int64_t cu = t * 8 + (u ^ (kr & 7));     // source 16-byte unit along the W2 row
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (cu < row_units) v = __ldg(W + (c * 64 + kr) * row_units + cu);
    Wp[e] = v;
  }
}

}  // namespace

size_t draft_packed_bytes(int64_t rank, int64_t V) {
  if (rank < 64 || rank % 64 != 0 || V < 1) return 0;
  return (size_t)(rank / 64) * (size_t)((V + kBlkN - 1) / kBlkN) * (size_t)kPiece;
}

bool draft_tc_shape_ok(const DraftArgs &a) {
  if (a.dtype != DSPARK_BF16) return false;
  if (a.rank % 64 != 0 || a.rank > 256) return false;
  if (a.V % 8 != 0 || a.V > (int64_t)INT32_MAX - 64) return false;
  if (((uintptr_t)a.U | (uintptr_t)a.E) & 15u) return false;
  if (a.draft_logits && ((uintptr_t)a.draft_logits & 15u)) return false;
  // partial slots of one position: (M-tiles x 128 rows) x CTAs per M-tile <= 128 x max(grid, M-tiles)
  const int64_t m_tiles = (a.B + kTileM - 1) / kTileM;
  const int64_t units = m_tiles > 1024 ? m_tiles : 1024;
  if (units * kTileM > kTcPartialsPerStep) return false;
  if (a.K_max * kTcPartialsPerStep > a.partial_slots) return false;
  return true;
}

cudaError_t launch_pack_projection(const void *W, int64_t rank, int64_t V, void *Wp, cudaStream_t s) {
  const int nb = (int)((V + kBlkN - 1) / kBlkN);
  const int64_t units = (rank / 64) * (int64_t)nb * 64 * 8;
  const int blocks = (int)((units + 255) / 256 < 65535 ? (units + 255) / 256 : 65535);
  pack_projection<<<blocks, 256, 0, s>>>((const uint4 *)W, rank, V, nb, (uint4 *)Wp);
  return cudaGetLastError();
}

namespace {
template <bool RESID>
cudaError_t launch_tc(const DraftArgs &a, cudaStream_t s, int num_sms) {
  if (!a.Wp || ((uintptr_t)a.Wp & 15u)) return cudaErrorInvalidValue;
  const int rch = (int)(a.rank / 64);
  void *fn = nullptr;
  switch (rch) {
    case 1: fn = (void *)draft_tc_persistent<1, RESID>; break;
    case 2: fn = (void *)draft_tc_persistent<2, RESID>; break;
    case 3: fn = (void *)draft_tc_persistent<3, RESID>; break;
    default: fn = (void *)draft_tc_persistent<4, RESID>; break;
  }
  {
    cudaError_t e = ensure_dynamic_smem(fn, tc_smem_bytes<RESID>());
    if (e != cudaSuccess) return e;
  }
  const int grid = num_sms > 1024 ? 1024 : num_sms;
  // cooperative launch: all CTAs are co-resident, so the bounded grid barrier between
  // positions can always complete
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3(TcCfg<RESID>::kThreads, 1, 1);
  cfg.dynamicSmemBytes = tc_smem_bytes<RESID>();
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void *args[1] = {(void *)&a};
  return cudaLaunchKernelExC(&cfg, fn, args);
}
}  // namespace

cudaError_t launch_draft_tc(const DraftArgs &a, cudaStream_t s, int num_sms) { return launch_tc<false>(a, s, num_sms); }
cudaError_t launch_resid_tc(const DraftArgs &a, cudaStream_t s, int num_sms) { return launch_tc<true>(a, s, num_sms); }

}  // namespace dspark
