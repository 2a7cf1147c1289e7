// Internal device helpers shared by the DSpark kernels (sm_103a).
//
// Random stream: Philox4x32-10 as specified in Salmon, Moraes, Dror, Shaw,
// "Parallel Random Numbers: As Easy as 1, 2, 3" (SC'11), S4.  Round keys are
// precomputed on the host and travel in the kernel parameter block, so the
// rounds read them from the constant bank.
//
// Sampling: a two-level draw over blocks of 32 consecutive indices.  Block g
// (indices 32g .. 32g+31) with mass L_g = sum of its weights enters a Gumbel race
// with score log L_g + g_g, g_g = -log(-log u_g), u_g from word (g & 3) of the
// stream block c0 = g >> 2; the block with the largest score wins, which picks
// block g with probability L_g / sum L.  Inside the winner the index is drawn by
// inverse CDF: the first v whose running weight sum exceeds u' L_g, u' the
// accept-style uniform of word (g & 3) of the PICK stream.  Together this draws
// v with probability w_v / sum w, with one stream word per 32 elements.  The
// race over block scores runs as an exponential race: with E = -log u, a block
// can only beat the running best when (1 - u) < exp(log L_g - best), so the two
// accurate logarithms of the exact score are evaluated only for blocks that
// pass that test, and the inverse-CDF pass only for blocks that take the lead.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "dspark.h"

namespace dspark {

constexpr uint32_t kTagDraft = 0;
constexpr uint32_t kTagAccept = 1;
constexpr uint32_t kTagResid = 2;
constexpr uint32_t kTagDraftPick = 3;
constexpr uint32_t kTagResidPick = 4;
constexpr int kBlockW = 32;   // indices per block of the two-level draw
constexpr int kDraftSimtChunk = 256;   // vocabulary columns per tile of the CUDA-core draft step
constexpr int kMaxK = 16;
constexpr float kMinPositiveT = 1e-3f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kFilterSlack = 1.0f + 1.0f / 1024.0f;   // keeps the race filter conservative
constexpr float kFilterMax = 1.2676506002282294e30f;    // 2^100: "no best yet"

struct PhiloxKey {
  uint32_t k0[10];
  uint32_t k1[10];
};

inline PhiloxKey make_philox_key(uint64_t seed) {
  PhiloxKey k;
  uint32_t a = (uint32_t)(seed & 0xffffffffu), b = (uint32_t)(seed >> 32);
  for (int i = 0; i < 10; ++i) {
    k.k0[i] = a;
    k.k1[i] = b;
    a += 0x9E3779B9u;
    b += 0xBB67AE85u;
  }
  return k;
}

// Ten Philox rounds on counter (c0, c1, c2, c3).
__device__ __forceinline__ uint4 philox(const PhiloxKey &key, uint32_t c0, uint32_t c1, uint32_t c2,
                                        uint32_t c3) {
#pragma unroll
  for (int i = 0; i < 10; ++i) {
    const uint32_t hi0 = __umulhi(0xD2511F53u, c0);
    const uint32_t lo0 = 0xD2511F53u * c0;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c2);
    const uint32_t lo1 = 0xCD9E8D57u * c2;
    const uint32_t n0 = hi1 ^ c1 ^ key.k0[i];
    const uint32_t n2 = hi0 ^ c3 ^ key.k1[i];
    c0 = n0;
    c1 = lo1;
    c2 = n2;
    c3 = lo0;
  }
  return make_uint4(c0, c1, c2, c3);
}

__device__ __forceinline__ uint32_t word_of(const uint4 &w, int i) {
  return i == 0 ? w.x : (i == 1 ? w.y : (i == 2 ? w.z : w.w));
}

// ((w >> 9) + 0.5) * 2^-23: exact, in (0, 1).
__device__ __forceinline__ float uniform_open(uint32_t w) {
  return __uint_as_float((w >> 9) | 0x3F800000u) - 0.99999994039535522f;   // 1 - 2^-24
}

// (w >> 8) * 2^-24: exact, in [0, 1).
__device__ __forceinline__ float uniform_accept(uint32_t w) {
  return __uint2float_rn(w >> 8) * 5.9604644775390625e-08f;
}

// 1 - u for the Gumbel uniform of word w: ((~w >> 9) + 0.5) * 2^-23, exact.
__device__ __forceinline__ float one_minus_uniform_open(uint32_t w) {
  return __uint_as_float((w >> 9) ^ 0x3FFFFFFFu) - 0.99999994039535522f;
}

__device__ __forceinline__ float fast_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float fast_lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t h) {
  return __uint_as_float(((uint32_t)h) << 16);
}

__device__ __forceinline__ float round_to_bf16(float x) {
  return __bfloat162float(__float2bfloat16_rn(x));
}

__device__ __forceinline__ void set_status(int32_t *st, int code) {
  atomicCAS(st, 0, code);
}

__device__ __forceinline__ int read_status(const int32_t *st) {
  return *(volatile const int32_t *)st;
}

// Programmatic dependent launch.  A kernel launched with programmatic stream serialisation
// may become resident while the kernel before it in the stream is still running: it calls
// grid_dep_wait() before its first global memory access, which returns once that kernel has
// completed and its writes are visible.  grid_dep_launch() lets the next such kernel become
// resident early (it changes nothing about what that kernel may read).  Both are no-ops
// when the kernel was launched without the attribute.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ bool temperature_ok(float t) {
  return (t == 0.0f) || (t >= kMinPositiveT && t <= 3.0e38f);
}

// -------------------------------------------------------------------------
// mbarrier, bulk copy and L2-policy wrappers (inline PTX).
// -------------------------------------------------------------------------
constexpr long long kTimeoutCycles = 4000000000LL;   // budget of every bounded wait (about 2 s)

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
// One bounded probe of a barrier phase: the thread sleeps until the phase completes or
// about 20 us pass, so waiting roles do not spin on the issue slots of the epilogue.
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "n"(20000)
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
// Contiguous global -> shared bulk copy completing on an mbarrier (16-byte aligned, size % 16 == 0).
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

// Index check of the bounds-checked build (-DDSPARK_BOUNDS): an index outside [0, n) records
// DSPARK_ERR_BOUNDS in the status word and comes back as 0, so the access stays inside its
// buffer and the caller sees the error.  In the normal build the index passes through.
__device__ __forceinline__ int64_t bchk(int64_t i, int64_t n, int32_t *status) {
#ifdef DSPARK_BOUNDS
  if (i < 0 || i >= n) {
    set_status(status, DSPARK_ERR_BOUNDS);
    return 0;
  }
#else
  (void)n;
  (void)status;
#endif
  return i;
}

// 16-byte shared-memory load and store.
__device__ __forceinline__ uint4 ld_shared_u4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ void st_shared_u4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
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

// -------------------------------------------------------------------------
// Gumbel race state (one per thread; merged across threads and blocks).
// -------------------------------------------------------------------------
struct Race {
  float best;  // best perturbed score s_v + g_v seen
  int idx;     // its index
  float m;     // running max of s_v
  float S;     // sum exp(s_v - m)
  float c;     // filter factor: exp(m - best) * slack (kFilterMax when no best)
};

__device__ __forceinline__ void race_init(Race &r) {
  r.best = -INFINITY;
  r.idx = -1;
  r.m = -INFINITY;
  r.S = 0.0f;
  r.c = kFilterMax;
}

__device__ __forceinline__ float race_filter(float m, float best) {
  if (best == -INFINITY) return kFilterMax;
  const float x = (m - best) * kLog2e;
  return x > 100.0f ? kFilterMax : fast_ex2(x) * kFilterSlack;
}

// Exact perturbed score of a candidate and the update of the running best.
__device__ __forceinline__ void race_exact(Race &r, float s, uint32_t w, int v) {
  const float u = uniform_open(w);
  const float E = -logf(u);
  const float t = s - logf(E);
  if (t > r.best || (t == r.best && v < r.idx)) {
    r.best = t;
    r.idx = v;
    r.c = race_filter(r.m, r.best);
  }
}

// Process N scaled logits s[q] at indices v0 + q (invalid entries hold -INF)
// with their stream words w[q].
template <int N>
__device__ __forceinline__ void race_update(Race &r, const float (&s)[N], const uint32_t (&w)[N], int v0) {
  float cm = s[0];
#pragma unroll
  for (int q = 1; q < N; ++q) cm = fmaxf(cm, s[q]);
  if (cm == -INFINITY) return;
  if (cm > r.m) {
    r.S = (r.m == -INFINITY) ? 0.0f : r.S * fast_ex2((r.m - cm) * kLog2e);
    r.m = cm;
    r.c = race_filter(r.m, r.best);
  }
  const float mL = r.m * kLog2e;
  uint32_t cand = 0;
#pragma unroll
  for (int q = 0; q < N; ++q) {
    const float e = fast_ex2(fmaf(s[q], kLog2e, -mL));
    r.S += e;
    const float d1 = 1.0f - uniform_open(w[q]);
    if (d1 < e * r.c) cand |= 1u << q;
  }
  while (cand) {
    const int q = __ffs(cand) - 1;
    cand &= cand - 1;
    float sq = s[0];
    uint32_t wq = w[0];
#pragma unroll
    for (int i = 1; i < N; ++i)
      if (i == q) { sq = s[i]; wq = w[i]; }
    race_exact(r, sq, wq, v0 + q);
  }
}

// Greedy: running max with smallest index.
template <int N>
__device__ __forceinline__ void argmax_update(Race &r, const float (&s)[N], int v0) {
#pragma unroll
  for (int q = 0; q < N; ++q)
    if (s[q] > r.best) { r.best = s[q]; r.idx = v0 + q; }
}

// Does merging b into a take b's index (score desc, index asc)?
__device__ __forceinline__ bool race_takes(const Race &a, const Race &b) {
  return b.best > a.best || (b.best == a.best && b.idx >= 0 && (a.idx < 0 || b.idx < a.idx));
}

// Merge b into a: best by (score desc, index asc); softmax (m, S).
__device__ __forceinline__ void race_merge(Race &a, const Race &b) {
  if (race_takes(a, b)) {
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

__device__ __forceinline__ Race race_shfl_down(const Race &r, int d) {
  Race o;
  o.best = __shfl_down_sync(0xffffffffu, r.best, d);
  o.idx = __shfl_down_sync(0xffffffffu, r.idx, d);
  o.m = __shfl_down_sync(0xffffffffu, r.m, d);
  o.S = __shfl_down_sync(0xffffffffu, r.S, d);
  o.c = 0.0f;
  return o;
}

// Block-wide merge; the result is valid in thread 0.  `scratch` holds one Race per warp.
__device__ __forceinline__ Race race_block_reduce(Race r, Race *scratch) {
  for (int d = 16; d > 0; d >>= 1) {
    Race o = race_shfl_down(r, d);
    race_merge(r, o);
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nw = (blockDim.x + 31) >> 5;
  __syncthreads();
  if (lane == 0) scratch[warp] = r;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int i = 1; i < nw; ++i) race_merge(r, scratch[i]);
  }
  return r;
}

// Partial result of one block, as stored in the workspace (16 bytes).
struct Partial {
  float best;
  int idx;
  float m;
  float S;
};

__device__ __forceinline__ Partial to_partial(const Race &r) {
  Partial p;
  p.best = r.best;
  p.idx = r.idx;
  p.m = r.m;
  p.S = r.S;
  return p;
}

// Load a partial written by another block: a gpu-scope relaxed load, which (after the
// acquire that observed the writer's release) sees the writer's value.
__device__ __forceinline__ Partial load_partial(const Partial *p) {
  int4 v;
  asm volatile("ld.relaxed.gpu.global.v4.s32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p)
               : "memory");
  Partial o;
  o.best = __int_as_float(v.x);
  o.idx = v.y;
  o.m = __int_as_float(v.z);
  o.S = __int_as_float(v.w);
  return o;
}

__device__ __forceinline__ Race from_partial(const Partial &p) {
  Race r;
  r.best = p.best;
  r.idx = p.idx;
  r.m = p.m;
  r.S = p.S;
  r.c = 0.0f;
  return r;
}

// -------------------------------------------------------------------------
// Two-level draw: per-thread state and block steps.
// -------------------------------------------------------------------------
struct BRace {
  float best;  // best block score seen (natural log units of the scaled weights)
  int idx;     // index drawn inside that block
  float M2;    // running max of the scaled logits, log2 units
  float S;     // sum of 2^(y - M2) over the scaled logits y seen
  float zx;    // the (stored-dtype) logit at idx
};

__device__ __forceinline__ void brace_init(BRace &r) {
  r.best = -INFINITY;
  r.idx = -1;
  r.M2 = -INFINITY;
  r.S = 0.0f;
  r.zx = 0.0f;
}

__device__ __forceinline__ Partial to_partial(const BRace &r) {
  Partial p;
  p.best = r.best;
  p.idx = r.idx;
  p.m = r.M2 == -INFINITY ? -INFINITY : r.M2 * kLn2;
  p.S = r.S;
  return p;
}

// Race entry of a block with log-mass ell and noise word wb; true when the block
// takes the lead (r.best updated), after which the caller draws inside it.
__device__ __forceinline__ bool brace_enter(BRace &r, float ell, uint32_t wb) {
  if (!(one_minus_uniform_open(wb) < fast_ex2((ell - r.best) * kLog2e) * kFilterSlack)) return false;
  const float t = ell - logf(-logf(uniform_open(wb)));
  if (!(t > r.best)) return false;   // equal scores keep the earlier (smaller) block
  r.best = t;
  return true;
}

// Inverse CDF inside a block of non-negative weights: the first q whose running sum
// (left to right, fp32) exceeds target.  The running sums are monotone, so that index
// is the number of running sums <= target.  No crossing happens only when u' is within
// rounding of 1; the draw then takes the last positive weight.
template <int N>
__device__ __forceinline__ int pick_in_block(const float (&w)[N], float target) {
  float P = 0.0f;
  int cnt = 0;
#pragma unroll
  for (int q = 0; q < N; ++q) {
    P += w[q];
    cnt += (P <= target) ? 1 : 0;
  }
  if (cnt < N) return cnt;
  int last = 0;
#pragma unroll
  for (int q = 0; q < N; ++q)
    if (w[q] > 0.0f) last = q;
  return last;
}

// Block of softmax weights 2^(z_q a - Mb) (a = log2(e) / T, Mb = max(z) a): folds
// the block into the running softmax, enters the race and, when the block leads,
// draws the index.  Entries past the vocabulary hold -inf.  z is overwritten with
// the weights, which the in-block draw reuses.  pick_word() returns the PICK
// stream word of the block (evaluated only when needed).
// Returns true when the block took the lead.
// Folds a block with scaled maximum Mb (log2 units) and weights w (sum Sb) into the
// running softmax, enters the race and, when the block leads, draws the index.
// zfn(q) returns the logit of the block's element q; it is evaluated only for a block that
// takes the lead, to record the logit of the drawn index.
template <int N, class PickWord, class ZFn>
__device__ __forceinline__ bool brace_fold_block(BRace &r, const float (&w)[N], float Mb, float Sb, uint32_t wb,
                                                 int v0, PickWord pick_word, ZFn zfn) {
  if (Mb > r.M2) {
    r.S = r.S * fast_ex2(r.M2 - Mb) + Sb;
    r.M2 = Mb;
  } else {
    r.S = fmaf(Sb, fast_ex2(Mb - r.M2), r.S);
  }
  const float ell = (Mb + fast_lg2(Sb)) * kLn2;
  if (!brace_enter(r, ell, wb)) return false;
  const int q = pick_in_block(w, uniform_accept(pick_word()) * Sb);
  r.idx = v0 + q;
  r.zx = zfn(q);
  return true;
}

// The block's weights overwrite z; zfn(q) must recover the logit of element q elsewhere.
template <int N, class PickWord, class ZFn>
__device__ __forceinline__ bool brace_softmax_block(BRace &r, float (&z)[N], float mz, float a, uint32_t wb,
                                                    int v0, PickWord pick_word, ZFn zfn) {
  if (mz == -INFINITY) return false;
  const float Mb = mz * a;
  float s[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
  for (int q = 0; q < N; ++q) {
    z[q] = fast_ex2(fmaf(z[q], a, -Mb));
    s[q & 3] += z[q];
  }
  return brace_fold_block(r, z, Mb, (s[0] + s[1]) + (s[2] + s[3]), wb, v0, pick_word, zfn);
}

// Logits that are not needed after the draw (the bonus draw of verification).
struct NoLogit {
  __device__ __forceinline__ float operator()(int) const { return 0.0f; }
};

// ---- paired fp32 arithmetic: one sm_100 instruction for two independent lanes, each
// rounded exactly like the scalar operation ----
__device__ __forceinline__ unsigned long long f2_pack(float lo, float hi) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(unsigned long long v, float &lo, float &hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ unsigned long long f2_fma(unsigned long long a, unsigned long long b,
                                                     unsigned long long c) {
  unsigned long long r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ unsigned long long f2_mul(unsigned long long a, unsigned long long b) {
  unsigned long long r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ unsigned long long f2_add(unsigned long long a, unsigned long long b) {
  unsigned long long r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// Softmax block of 32 bf16 logits held as 16 pairs (low half first); the same fp32
// operations in the same order as brace_softmax_block on the unpacked values.
template <class PickWord>
__device__ __forceinline__ bool brace_softmax_bf16x32(BRace &r, const uint32_t (&pk)[16], float mz, float a,
                                                      uint32_t wb, int v0, PickWord pick_word) {
  if (mz == -INFINITY) return false;
  const float Mb = mz * a;
  const unsigned long long aa = f2_pack(a, a), mb = f2_pack(-Mb, -Mb);
  unsigned long long s01 = f2_pack(0.0f, 0.0f), s23 = s01;   // (s0, s1), (s2, s3): s[q & 3]
  float w[32];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const unsigned long long zz = f2_pack(__uint_as_float(pk[j] << 16), __uint_as_float(pk[j] & 0xffff0000u));
    float y0, y1;
    f2_unpack(f2_fma(zz, aa, mb), y0, y1);
    w[2 * j] = fast_ex2(y0);
    w[2 * j + 1] = fast_ex2(y1);
    const unsigned long long ee = f2_pack(w[2 * j], w[2 * j + 1]);
    if (j & 1) s23 = f2_add(s23, ee);
    else s01 = f2_add(s01, ee);
  }
  float s0, s1, s2, s3;
  f2_unpack(s01, s0, s1);
  f2_unpack(s23, s2, s3);
  if (!brace_fold_block(r, w, Mb, (s0 + s1) + (s2 + s3), wb, v0, pick_word, NoLogit{})) return false;
  const int q = r.idx - v0;          // the drawn element: its logit from the packed words
  // select word q >> 1 by a tree on its bits (register selects, no indexed access)
  uint32_t t8[8], t4[4], t2[2];
  const uint32_t h = (uint32_t)q >> 1;
#pragma unroll
  for (int j = 0; j < 8; ++j) t8[j] = (h & 1u) ? pk[2 * j + 1] : pk[2 * j];
#pragma unroll
  for (int j = 0; j < 4; ++j) t4[j] = (h & 2u) ? t8[2 * j + 1] : t8[2 * j];
#pragma unroll
  for (int j = 0; j < 2; ++j) t2[j] = (h & 4u) ? t4[2 * j + 1] : t4[2 * j];
  const uint32_t wq = (h & 8u) ? t2[1] : t2[0];
  r.zx = __uint_as_float((q & 1) ? (wq & 0xffff0000u) : (wq << 16));
  return true;
}

// Residual weight max(0, p - q) with p = 2^(t a - lt2), q = 2^(d a - ld2).
__device__ __forceinline__ float resid_weight(float t, float d, float a, float lt2, float ld2) {
  return fmaxf(fast_ex2(fmaf(t, a, -lt2)) - fast_ex2(fmaf(d, a, -ld2)), 0.0f);
}

// One block of residual weights max(0, p - q) on packed bf16 rows (tp: target, dp: draft; pair e
// of the block in word (e & 3) of unit e >> 2), in the two-level draw; any_pos records a positive
// weight.  The verification's stored-row pass and the tensor-core recompute pass share it, so
// both draw the same token.
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

// Greedy block: running maximum, smallest index on ties.
template <int N>
__device__ __forceinline__ void brace_argmax_block(BRace &r, const float (&z)[N], float mz, int v0) {
  if (!(mz > r.best)) return;
  r.best = mz;
  r.zx = mz;
  int q0 = N - 1;
#pragma unroll
  for (int q = N - 1; q >= 0; --q)
    if (z[q] == mz) q0 = q;
  r.idx = v0 + q0;
}

template <int N>
__device__ __forceinline__ float block_max(const float (&z)[N]) {
  float m[4] = {z[0], z[1], z[2], z[3]};
#pragma unroll
  for (int q = 4; q < N; ++q) m[q & 3] = fmaxf(m[q & 3], z[q]);
  return fmaxf(fmaxf(m[0], m[1]), fmaxf(m[2], m[3]));
}

// Warp-cooperative merge of R rows of partials: row i has n consecutive
// partials at p[i] (p[i] == nullptr: skip).  Every lane issues its loads for all
// rows before merging, so many L2 reads are in flight at once.  The merged
// result is valid in lane 0 of the warp.
__device__ __forceinline__ Partial empty_partial() {
  Partial q;
  q.best = -INFINITY;
  q.idx = -1;
  q.m = -INFINITY;
  q.S = 0.0f;
  return q;
}

template <int R>
__device__ __forceinline__ void warp_merge_rows(const Partial *const (&p)[R], int n, Race (&tot)[R]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int i = 0; i < R; ++i) race_init(tot[i]);
  for (int j0 = 0; j0 < n; j0 += 64) {
    Partial q[R][2];
#pragma unroll
    for (int i = 0; i < R; ++i)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int j = j0 + h * 32 + lane;
        q[i][h] = (p[i] != nullptr && j < n) ? load_partial(p[i] + j) : empty_partial();
      }
#pragma unroll
    for (int i = 0; i < R; ++i)
#pragma unroll
      for (int h = 0; h < 2; ++h) race_merge(tot[i], from_partial(q[i][h]));
  }
#pragma unroll
  for (int i = 0; i < R; ++i)
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) race_merge(tot[i], race_shfl_down(tot[i], d));
}

// -------------------------------------------------------------------------
// Host-side launchers (defined in the kernel translation units).
// -------------------------------------------------------------------------
// One residual draw of the recompute verification: request r rejected its draft token at
// position j (T > 0); the draft row (r, j) is recomputed from the base logits and W1[x_{j-1}] W2.
struct VJob {
  int r, j, prev;   // request, rejecting position, x_{j-1} (the anchor for j = 1)
  int urow;         // base-logit row r K_max + j - 1
  int trow;         // flattened target row tgt_off[r] + j - 1
  float lse_t, lse_q, invT;
};

struct DraftArgs {
  const void *U, *E, *W;
  const void *Wp;     // W2 in the packed tensor-core layout (tensor-core path only)
  const int32_t *anchor, *K_r;
  const float *temperature;
  int32_t *draft_tok;
  void *draft_logits;
  float *draft_lse;
  float *draft_zx;    // [B, K_max] the logit of each drawn token (optional)
  int32_t *dev_status;
  int64_t B, K_max, V, rank;
  int dtype;
  PhiloxKey key;
  // workspace carve-out
  int32_t *perm;      // [B] requests ordered by K_r descending
  int32_t *iperm;     // [B] position of each request in perm
  int32_t *act;       // [K_max, B] row k-1: the requests with K_r >= k in groups of 32 of one
                      // kind (T > 0 or greedy), full groups in the order they complete in
                      // request order, then the partial ones (the tensor-core path's M-tiles take
                      // consecutive runs of it: rows close together in U, and warps of one kind
                      // of draw but at most one per position)
  int32_t *grp;       // [K_max, 2, ceil(B / 32)] building act: per full group, the other kind's
                      // full groups completed before it
  int32_t *nact;      // [K_max + 2] active requests per position
  int32_t *counters;  // [B] per-row arrival counters (zero between steps)
  unsigned long long *best_key;  // [B, K_max] packed (score, index) maxima of the tensor-core path
  int32_t *gbar;      // [K_max + 1] grid-barrier arrival counters of the tensor-core path
  Partial *partials;  // [partial_slots]
  float *zx_part;     // [partial_slots] CUDA-core path: the logit at each partial's index
  int64_t partial_slots;
  int64_t u_rows = 0;  // rows of U (B x K_max of the draft; the residual pass runs with K_max = 1)
  // confidence head with the Markov term (optional): conf_out[r, k] =
  // sigmoid(conf_h[r, k] + conf_w . E[x_{k-1}])
  const float *conf_h = nullptr;   // [B, K_max] backbone term w_h . h_k + b
  const float *conf_w = nullptr;   // [rank] weights of the Markov embedding
  float *conf_out = nullptr;       // [B, K_max]
  // failure-path test hook (DSPARK_FLAG_TEST_BARRIER_TIMEOUT): arrivals the barrier before
  // position 2 waits for beyond the grid, which never come, so that bounded wait runs out
  int gbar_extra = 0;
  // RNN head (optional, CUDA-core path): the cell's sequential weights [3 rank, 2 rank] in
  // the call dtype, its backbone term [B, K_max, 3 rank], and in the workspace the state
  // [2, B, rank] (position k writes buffer k & 1) and the feature [B, rank]; the feature
  // replaces the W1 row in the bias
  const void *rnn_W = nullptr;
  const float *rnn_x = nullptr;
  float *rnn_state = nullptr;
  float *rnn_feat = nullptr;
  // residual mode of the tensor-core kernel (the recompute verification): one position whose
  // rows are jobs[0 .. nact[1]); key and flag per request in best_key / resid_any
  const VJob *jobs = nullptr;
  const void *tgt = nullptr;
  int32_t *resid_any = nullptr;
};

// Confidence head ("DSpark" S3.2.1): one linear projection of the backbone state and the
// previous token's Markov embedding, then a sigmoid.  One warp: e(q) returns entry q of
// the embedding row; the rank is summed lane-strided, then across the warp.  The sigmoid
// is evaluated as t / (1 + t), t = exp(s), for s < 0 so that it never overflows.
template <typename EFn>
__device__ __forceinline__ float warp_confidence(EFn e, const float *w, int rank, float h, int lane) {
  float acc = 0.0f;
  for (int q = lane; q < rank; q += 32) acc = fmaf(e(q), w[q], acc);
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, d);
  const float s = h + acc;
  if (s >= 0.0f) return 1.0f / (1.0f + expf(-s));
  const float t = expf(s);
  return t / (1.0f + t);
}

// Total order key of a perturbed score and its index: larger score first, then the
// smaller index, so a 64-bit atomicMax merges (score desc, index asc).
__device__ __forceinline__ unsigned long long score_key(float s, int idx) {
  const uint32_t u = __float_as_uint(s);
  const uint32_t o = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((unsigned long long)o << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)idx);
}
// A float written by another CTA (gpu-scope relaxed load; see load_partial).
__device__ __forceinline__ float load_f32_relaxed(const float *p) {
  float v;
  asm volatile("ld.relaxed.gpu.global.f32 %0, [%1];" : "=f"(v) : "l"(p) : "memory");
  return v;
}

// Packed key written by other CTAs: a gpu-scope relaxed load (after an acquire that
// observed the writers' release it sees their values).
__device__ __forceinline__ unsigned long long load_key(const unsigned long long *p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ int key_index(unsigned long long key) {
  return (int)(0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFull));
}

cudaError_t launch_draft_prologue(const DraftArgs &a, cudaStream_t s, bool tensor_core);
cudaError_t launch_draft_simt(const DraftArgs &a, cudaStream_t s);
cudaError_t launch_draft_tc(const DraftArgs &a, cudaStream_t s, int num_sms);
cudaError_t launch_resid_tc(const DraftArgs &a, cudaStream_t s, int num_sms);   // residual mode
constexpr int64_t kTcPartialsPerStep = 128 * 1024;   // slots per draft position on the tensor-core path
bool draft_tc_shape_ok(const DraftArgs &a);
size_t draft_packed_bytes(int64_t rank, int64_t V);  // 0 when rank is not a positive multiple of 64
cudaError_t launch_pack_projection(const void *W, int64_t rank, int64_t V, void *Wp, cudaStream_t s);


struct VerifyJob {
  int mode;      // 0 none, 1 residual (T > 0), 2 bonus (T > 0), 3 bonus (greedy),
                 // 4 residual drawn by the tensor-core recompute pass (token or rounding guard)
  int pos;       // stream position (j, or ell + 1 for the bonus)
  int64_t trow;  // target row
  int64_t drow;  // draft row (residual only)
  float lse_t, lse_q, invT;
  int out_slot;  // index into out_tok
};

constexpr int kNoReject = 127;   // dead[r] of a request with no rejected position

// One verified drafted row (request r, position j <= ell_r) of the statistics pass; the plan
// kernel lists them position-major (every request's position 1, then position 2, ...).
struct VRow {
  int r, j, x;     // request, position, draft token x_j; for a bonus draw (kind 4) the part:
                   // (parts << 8) | part, the part covering slices [part S / parts, (part + 1) S / parts)
  int trow;        // row of the flattened target logits: tgt_off[r] + j - 1
  float invT;      // 1 / T (1 for greedy)
  float lqx;       // log q_j(x_j), T > 0 with a known draft normaliser
  int kind;        // 1 softmax statistics of the target row, 2 its argmax (T = 0), 3 softmax
                   // statistics of the target and of the draft row (no draft normaliser);
                   // the bonus row j = ell_r + 1: 4 the bonus draw (T > 0), 5 its argmax (T = 0)
  int drow;        // draft row r K_max + j - 1
};

// Statistics of a completed row: log-sum-exp of target / T (the maximum for T = 0), the
// argmax (for a bonus row: the bonus token), the scaled target logit at x_j and (kind 3) the
// draft row's log-sum-exp.  Stored per request and position: r (K_max + 1) + j - 1.
struct VRowRes {
  float lse_t;
  int amax;
  float zx_t;
  float lse_q;
};

struct VerifyArgs {
  const void *D;        // stored draft logits [B, K_max, V]; NULL for the recompute entry point
  const float *D_lse;   // draft normalisers [B, K_max] (optional with stored logits)
  const float *D_zx = nullptr;    // drawn tokens' logits [B, K_max] (recompute entry point)
  const void *tgt;
  const int32_t *tgt_off, *ell, *draft_tok;
  const float *temperature;
  int32_t *n_acc, *out_tok, *dev_status;
  int64_t B, K_max, V;
  int dtype;
  PhiloxKey key;
  // workspace
  VRow *rows;           // [B * (kMaxK + 1)] the verified rows and bonus rows, position-major
  int32_t *nrows;       // [2] how many; [1]: parts per bonus draw row
  int32_t *row_start;   // [kMaxK + 3] first list slot of position j's rows
  int32_t *row_fill;    // [kMaxK + 3] position j's rows listed so far
  int32_t *scan_next;   // [1] the next listed row a scan CTA takes
  int32_t *dead;        // [B] first rejecting position (kNoReject: none)
  unsigned long long *bonus_key;   // [B] packed (score, index) maximum of the bonus draw's parts
  int scan_cap;         // scan CTAs resident at once (the bonus draws are split only within one wave)
  VRowRes *rres;        // [B * (kMaxK + 1)] request-major: r (K_max + 1) + j - 1
  int row_slices;       // vocabulary slices per row of the statistics pass
  int32_t *counters;   // [B] chunk arrivals of the sampling pass (reset by the plan kernel)
  Partial *partials;   // [B * chunks]
  int chunks;          // vocabulary chunks of the sampling pass (at most the workspace's)
  int chunk_len;       // columns per chunk, a multiple of 32
  // recompute entry point: the residual draws of the tensor-core pass
  const unsigned long long *resid_key = nullptr;   // [B] packed (score, index) maximum per request
  const int32_t *resid_any = nullptr;              // [B] non-zero when some p_v > q_v
  // recompute entry point, the job pass: lists the T > 0 rejections for the tensor-core pass
  const int32_t *anchor = nullptr;      // [B] x_0 (the previous token of a rejection at j = 1)
  VJob *jobs = nullptr;                 // [B]
  int32_t *jobs_nact = nullptr;         // [3] active counts of the residual pass: {B, #jobs, 0}
  int32_t *jobs_gbar = nullptr;         // [2] its grid-barrier counters
  unsigned long long *key_out = nullptr;   // = resid_key, reset per call
  int32_t *any_out = nullptr;              // = resid_any, reset per call
};

int verify_row_slices(int64_t V);
size_t verify_ws_bytes(int64_t B, int64_t V, int *chunks);
void verify_carve(VerifyArgs &a, void *workspace);
// resid: the residual pass's arguments for the recompute entry point (nullptr: stored rows)
cudaError_t launch_verify(const VerifyArgs &a, cudaStream_t s, int num_sms, const DraftArgs *resid = nullptr);

// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) applies to the current device: set once per
// (device, kernel), under a lock so that host threads and several devices are safe.
cudaError_t ensure_dynamic_smem(const void *fn, int bytes);

}  // namespace dspark
