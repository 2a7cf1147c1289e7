// Host side of the C ABI declared in include/dspark.h: argument validation,
// workspace carving, kernel-path selection and the status helpers.
#include <cstdio>
#include <cstring>
#include <mutex>
#include <map>
#include <utility>

#include "schedule.cuh"

using namespace dspark;

namespace {

constexpr int64_t kMaxB = 1 << 20;
constexpr int64_t kMaxV = (int64_t)1 << 30;
constexpr int64_t kMaxRank = 8192;
constexpr int64_t kMaxRnnRank = 4096;   // the RNN entry point's documented rank limit

size_t al256(size_t x) { return (x + 255) & ~(size_t)255; }

bool aligned256(const void *p) { return ((uintptr_t)p & 255u) == 0; }

struct DeviceInfo {
  int sms = 0;
  int major = 0, minor = 0;
};

bool device_info(DeviceInfo *out) {
  static DeviceInfo cache[64];
  static bool have[64] = {false};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  std::lock_guard<std::mutex> lock(mu);
  if (!have[dev]) {
    DeviceInfo d;
    if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return false;
    if (cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return false;
    if (cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) return false;
    cache[dev] = d;
    have[dev] = true;
  }
  *out = cache[dev];
  return true;
}

int64_t draft_partial_slots(int64_t B, int64_t K_max, int64_t V) {
  const int64_t simt = B * ((V + kDraftSimtChunk - 1) / kDraftSimtChunk);
  const int64_t tc = K_max * dspark::kTcPartialsPerStep;
  return simt > tc ? simt : tc;
}

dspark_status check_dims(const dspark_dims &d, bool need_rank) {
  if (d.B < 1 || d.B > kMaxB || d.K_max < 1 || d.K_max > kMaxK || d.V < 2 || d.V > kMaxV)
    return DSPARK_ERR_DIMS;
  if (need_rank && (d.rank < 1 || d.rank > kMaxRank)) return DSPARK_ERR_DIMS;
  if (d.dtype != DSPARK_F32 && d.dtype != DSPARK_BF16) return DSPARK_ERR_DTYPE;
  return DSPARK_OK;
}

}  // namespace

namespace dspark {
cudaError_t ensure_dynamic_smem(const void *fn, int bytes) {
  static std::mutex mu;
  static std::map<std::pair<int, const void *>, int> set_to;   // the size each (device, kernel) allows
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  auto it = set_to.find({dev, fn});
  if (it != set_to.end() && it->second >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) set_to[{dev, fn}] = bytes;
  return e;
}
}  // namespace dspark

extern "C" {

int dspark_version(void) { return 200; }

const char *dspark_status_string(dspark_status s) {
  switch (s) {
    case DSPARK_OK: return "DSPARK_OK";
    case DSPARK_ERR_NULL: return "DSPARK_ERR_NULL";
    case DSPARK_ERR_DIMS: return "DSPARK_ERR_DIMS";
    case DSPARK_ERR_DTYPE: return "DSPARK_ERR_DTYPE";
    case DSPARK_ERR_TEMPERATURE: return "DSPARK_ERR_TEMPERATURE";
    case DSPARK_ERR_SPS_TOO_SHORT: return "DSPARK_ERR_SPS_TOO_SHORT";
    case DSPARK_ERR_OFFSETS: return "DSPARK_ERR_OFFSETS";
    case DSPARK_ERR_TOKEN_RANGE: return "DSPARK_ERR_TOKEN_RANGE";
    case DSPARK_ERR_LENGTHS: return "DSPARK_ERR_LENGTHS";
    case DSPARK_ERR_CONFIDENCE: return "DSPARK_ERR_CONFIDENCE";
    case DSPARK_ERR_WORKSPACE: return "DSPARK_ERR_WORKSPACE";
    case DSPARK_ERR_DEVICE_TIMEOUT: return "DSPARK_ERR_DEVICE_TIMEOUT";
    case DSPARK_ERR_CUDA: return "DSPARK_ERR_CUDA";
    case DSPARK_ERR_UNSUPPORTED: return "DSPARK_ERR_UNSUPPORTED";
    case DSPARK_ERR_BOUNDS: return "DSPARK_ERR_BOUNDS";
  }
  return "DSPARK_ERR_UNKNOWN";
}

dspark_status dspark_check(int32_t *dev_status, void *stream) {
  if (!dev_status) return DSPARK_ERR_NULL;
  cudaStream_t s = (cudaStream_t)stream;
  int32_t host = 0;
  if (cudaMemcpyAsync(&host, dev_status, sizeof(int32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return DSPARK_ERR_CUDA;
  if (host != 0) {
    if (cudaMemsetAsync(dev_status, 0, sizeof(int32_t), s) != cudaSuccess) return DSPARK_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return DSPARK_ERR_CUDA;
  }
  return (dspark_status)host;
}

// ---------------------------------------------------------------------------
// draft
// ---------------------------------------------------------------------------
// Does a call with these dims pack W2 into its workspace (tensor-core shape, W not
// pre-packed, CUDA-core path not forced)?
static bool draft_packs_into_workspace(const dspark_dims &d) {
  return d.dtype == DSPARK_BF16 && d.rank >= 64 && d.rank <= 256 && d.rank % 64 == 0 && d.V % 8 == 0 &&
         !(d.flags & (DSPARK_FLAG_FORCE_SIMT | DSPARK_FLAG_W_PACKED));
}

static size_t draft_ws_base(int64_t B, int64_t K_max, int64_t V) {
  return 2 * al256(sizeof(int32_t) * (size_t)B) + al256(sizeof(int32_t) * (size_t)(K_max + 2)) +
         al256(sizeof(int32_t) * (size_t)(B > 4096 ? B : 4096)) + al256(8 * (size_t)(B * K_max)) +
         al256(sizeof(int32_t) * (size_t)(K_max + 1)) + al256(sizeof(int32_t) * (size_t)(B * K_max)) +
         al256(sizeof(int32_t) * (size_t)(2 * K_max * ((B + 31) / 32))) +
         al256(sizeof(Partial) * (size_t)draft_partial_slots(B, K_max, V)) +
         al256(sizeof(float) * (size_t)draft_partial_slots(B, K_max, V));
}

size_t dspark_draft_workspace_bytes(dspark_dims dims) {
  if (check_dims(dims, true) != DSPARK_OK) return 0;
  size_t n = draft_ws_base(dims.B, dims.K_max, dims.V);
  if (draft_packs_into_workspace(dims)) n += al256(draft_packed_bytes(dims.rank, dims.V));
  return n;
}

size_t dspark_draft_packed_projection_bytes(int64_t rank, int64_t V) {
  if (rank < 64 || rank > 256 || rank % 64 != 0 || V < 2 || V > kMaxV || V % 8 != 0) return 0;
  return draft_packed_bytes(rank, V);
}

dspark_status dspark_draft_pack_projection(const void *W, dspark_dims dims, void *W_packed, size_t packed_bytes,
                                           void *stream) {
  if (!W || !W_packed) return DSPARK_ERR_NULL;
  if (dims.rank < 1 || dims.rank > kMaxRank || dims.V < 2 || dims.V > kMaxV) return DSPARK_ERR_DIMS;
  if (dims.dtype != DSPARK_F32 && dims.dtype != DSPARK_BF16) return DSPARK_ERR_DTYPE;
  const size_t need = dspark_draft_packed_projection_bytes(dims.rank, dims.V);
  if (dims.dtype != DSPARK_BF16 || need == 0 || ((uintptr_t)W & 15u)) return DSPARK_ERR_UNSUPPORTED;
  if (!aligned256(W_packed) || packed_bytes < need) return DSPARK_ERR_WORKSPACE;
  return launch_pack_projection(W, dims.rank, dims.V, W_packed, (cudaStream_t)stream) == cudaSuccess
             ? DSPARK_OK
             : DSPARK_ERR_CUDA;
}

namespace {

// The RNN head's part of a draft call (null for the Markov head).
struct RnnHead {
  const void *W;    // [3 rank, 2 rank], call dtype
  const float *x;   // [B, K_max, 3 rank]
};

size_t rnn_state_bytes(const dspark_dims &d) { return al256(sizeof(float) * (size_t)(d.B * d.rank)); }

dspark_status draft_call(const void *U, const void *E, const void *W, const int32_t *anchor, const int32_t *K_r,
                         const float *temperature, uint64_t seed, dspark_dims dims, int32_t *draft_tok,
                         void *draft_logits, float *draft_lse, float *draft_zx, const float *conf_h,
                         const float *conf_w,
                         float *conf, const RnnHead *rnn, void *workspace, size_t workspace_bytes,
                         int32_t *dev_status, void *stream) {
  if (!U || !E || !W || !anchor || !K_r || !temperature || !draft_tok || !dev_status) return DSPARK_ERR_NULL;
  dspark_status st = check_dims(dims, true);
  if (st != DSPARK_OK) return st;
  const size_t need = rnn ? dspark_draft_rnn_workspace_bytes(dims) : dspark_draft_workspace_bytes(dims);
  if (!workspace || !aligned256(workspace) || workspace_bytes < need) return DSPARK_ERR_WORKSPACE;
  DeviceInfo dev;
  if (!device_info(&dev)) return DSPARK_ERR_CUDA;
  const bool packed_in = (dims.flags & DSPARK_FLAG_W_PACKED) != 0;
  DraftArgs a;
  a.U = U;
  a.E = E;
  a.W = W;
  a.Wp = nullptr;
  a.anchor = anchor;
  a.K_r = K_r;
  a.temperature = temperature;
  a.draft_tok = draft_tok;
  a.draft_logits = draft_logits;
  a.draft_lse = draft_lse;
  a.draft_zx = draft_zx;
  a.dev_status = dev_status;
  a.B = dims.B;
  a.K_max = dims.K_max;
  a.u_rows = dims.B * dims.K_max;
  a.V = dims.V;
  a.rank = dims.rank;
  a.dtype = dims.dtype;
  a.key = make_philox_key(seed);
  a.gbar_extra = (dims.flags & DSPARK_FLAG_TEST_BARRIER_TIMEOUT) ? 1 : 0;
  a.conf_h = conf_h;
  a.conf_w = conf_w;
  a.conf_out = conf;
  char *p = (char *)workspace;
  a.perm = (int32_t *)p;
  p += al256(sizeof(int32_t) * (size_t)dims.B);
  a.iperm = (int32_t *)p;
  p += al256(sizeof(int32_t) * (size_t)dims.B);
  a.nact = (int32_t *)p;
  p += al256(sizeof(int32_t) * (size_t)(dims.K_max + 2));
  a.counters = (int32_t *)p;
  p += al256(sizeof(int32_t) * (size_t)(dims.B > 4096 ? dims.B : 4096));
  a.best_key = (unsigned long long *)p;
  p += al256(8 * (size_t)(dims.B * dims.K_max));
  a.gbar = (int32_t *)p;
  p += al256(sizeof(int32_t) * (size_t)(dims.K_max + 1));
  a.act = (int32_t *)p;
  p += al256(sizeof(int32_t) * (size_t)(dims.B * dims.K_max));
  a.grp = (int32_t *)p;
  p += al256(sizeof(int32_t) * (size_t)(2 * dims.K_max * ((dims.B + 31) / 32)));
  a.partials = (Partial *)p;
  a.partial_slots = draft_partial_slots(dims.B, dims.K_max, dims.V);
  p += al256(sizeof(Partial) * (size_t)a.partial_slots);
  a.zx_part = (float *)p;
  p += al256(sizeof(float) * (size_t)a.partial_slots);
  if (rnn) {   // the CUDA-core path only: the workspace holds no packed W2, then two state
               // buffers (the cell alternates between them by position) and the feature
    a.rnn_W = rnn->W;
    a.rnn_x = rnn->x;
    a.rnn_state = (float *)p;
    p += 2 * rnn_state_bytes(dims);
    a.rnn_feat = (float *)p;
    p += rnn_state_bytes(dims);
  }
  const bool use_tc = !(dims.flags & DSPARK_FLAG_FORCE_SIMT) && dev.major == 10 && dev.minor == 3 &&
                      draft_tc_shape_ok(a);
  if (packed_in) {
    // a packed projection only feeds the tensor-core path
    if (!use_tc || ((uintptr_t)W & 15u)) return DSPARK_ERR_UNSUPPORTED;
    a.Wp = W;
  } else if (use_tc) {
    if (((uintptr_t)W & 15u) || !draft_packs_into_workspace(dims)) return DSPARK_ERR_UNSUPPORTED;
    a.Wp = p;   // packed into the workspace by this call
  }
  cudaStream_t s = (cudaStream_t)stream;
  if (launch_draft_prologue(a, s, use_tc) != cudaSuccess) return DSPARK_ERR_CUDA;
  if (use_tc && !packed_in && launch_pack_projection(W, dims.rank, dims.V, (void *)a.Wp, s) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  // with DSPARK_FLAG_SPARE_SM the persistent kernel (one CTA per SM) leaves one SM free
  const int tc_sms = (dims.flags & DSPARK_FLAG_SPARE_SM) && dev.sms > 1 ? dev.sms - 1 : dev.sms;
  cudaError_t e = use_tc ? launch_draft_tc(a, s, tc_sms) : launch_draft_simt(a, s);
  return e == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
}

}  // namespace

dspark_status dspark_draft_markov_sample(const void *U, const void *E, const void *W, const int32_t *anchor,
                                         const int32_t *K_r, const float *temperature, uint64_t seed,
                                         dspark_dims dims, int32_t *draft_tok, void *draft_logits,
                                         float *draft_lse, float *draft_tok_logit, void *workspace,
                                         size_t workspace_bytes, int32_t *dev_status, void *stream) {
  return draft_call(U, E, W, anchor, K_r, temperature, seed, dims, draft_tok, draft_logits, draft_lse,
                    draft_tok_logit, nullptr, nullptr, nullptr, nullptr, workspace, workspace_bytes, dev_status,
                    stream);
}

size_t dspark_draft_rnn_workspace_bytes(dspark_dims dims) {
  if ((dims.flags & DSPARK_FLAG_W_PACKED) || check_dims(dims, true) != DSPARK_OK) return 0;
  dims.flags |= DSPARK_FLAG_FORCE_SIMT;
  return dspark_draft_workspace_bytes(dims) + 3 * rnn_state_bytes(dims);
}

dspark_status dspark_draft_rnn_sample(const void *U, const void *E, const void *W, const void *rnn_W,
                                      const float *rnn_x, const int32_t *anchor, const int32_t *K_r,
                                      const float *temperature, uint64_t seed, dspark_dims dims,
                                      int32_t *draft_tok, void *draft_logits, float *draft_lse,
                                      float *draft_tok_logit, void *workspace, size_t workspace_bytes,
                                      int32_t *dev_status, void *stream) {
  if (!rnn_W || !rnn_x) return DSPARK_ERR_NULL;
  if (dims.flags & DSPARK_FLAG_W_PACKED) return DSPARK_ERR_UNSUPPORTED;
  if (dims.rank > kMaxRnnRank) return DSPARK_ERR_DIMS;
  dims.flags |= DSPARK_FLAG_FORCE_SIMT;   // the cell feeds the CUDA-core bias path
  const RnnHead rnn{rnn_W, rnn_x};
  return draft_call(U, E, W, anchor, K_r, temperature, seed, dims, draft_tok, draft_logits, draft_lse,
                    draft_tok_logit, nullptr, nullptr, nullptr, &rnn, workspace, workspace_bytes, dev_status,
                    stream);
}

dspark_status dspark_draft_markov_sample_confidence(const void *U, const void *E, const void *W,
                                                    const int32_t *anchor, const int32_t *K_r,
                                                    const float *temperature, uint64_t seed, dspark_dims dims,
                                                    const float *conf_h, const float *conf_w,
                                                    int32_t *draft_tok, void *draft_logits, float *draft_lse,
                                                    float *draft_tok_logit, float *conf, void *workspace,
                                                    size_t workspace_bytes, int32_t *dev_status, void *stream) {
  if (!conf_h || !conf_w || !conf) return DSPARK_ERR_NULL;
  return draft_call(U, E, W, anchor, K_r, temperature, seed, dims, draft_tok, draft_logits, draft_lse,
                    draft_tok_logit, conf_h, conf_w, conf, nullptr, workspace, workspace_bytes, dev_status, stream);
}

// ---------------------------------------------------------------------------
// schedule
// ---------------------------------------------------------------------------
size_t dspark_schedule_workspace_bytes(int64_t B, int64_t K_max) {
  if (B < 1 || K_max < 1) return 0;
  return schedule_ws_bytes(B, K_max);
}

dspark_status dspark_schedule_survival(const float *conf, const int32_t *K_r, const double *sps, int64_t sps_len,
                                       int64_t B, int64_t K_max, int32_t *ell, int32_t *tgt_off,
                                       double *theta_best, int64_t *b_star, float *survival, void *workspace,
                                       size_t workspace_bytes, int32_t *dev_status, void *stream) {
  if (!conf || !K_r || !sps || !ell || !tgt_off || !dev_status) return DSPARK_ERR_NULL;
  if (B < 1 || B > kMaxB || K_max < 1 || K_max > kMaxK || sps_len < 1) return DSPARK_ERR_DIMS;
  if (!workspace || !aligned256(workspace) || workspace_bytes < dspark_schedule_workspace_bytes(B, K_max))
    return DSPARK_ERR_WORKSPACE;
  ScheduleArgs a;
  a.conf = conf;
  a.K_r = K_r;
  a.sps = sps;
  a.sps_len = sps_len;
  a.B = B;
  a.K_max = K_max;
  a.ell = ell;
  a.tgt_off = tgt_off;
  a.theta_best = theta_best;
  a.b_star = b_star;
  a.survival = survival;
  a.dev_status = dev_status;
  a.ws = workspace;
  return launch_schedule(a, (cudaStream_t)stream) == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
}

dspark_status dspark_schedule_capacity(const float *conf, const int32_t *K_r, const double *sps, int64_t sps_len,
                                       int64_t B, int64_t K_max, int32_t *capacity, double *theta_best,
                                       int32_t *ell, int32_t *tgt_off, void *workspace, size_t workspace_bytes,
                                       int32_t *dev_status, void *stream) {
  if (!conf || !K_r || !sps || !capacity || !dev_status) return DSPARK_ERR_NULL;
  if ((ell == nullptr) != (tgt_off == nullptr)) return DSPARK_ERR_NULL;
  if (B < 1 || B > kMaxB || K_max < 1 || K_max > kMaxK || sps_len < 1) return DSPARK_ERR_DIMS;
  if (!workspace || !aligned256(workspace) || workspace_bytes < dspark_schedule_workspace_bytes(B, K_max))
    return DSPARK_ERR_WORKSPACE;
  ScheduleArgs a;
  a.conf = conf;
  a.K_r = K_r;
  a.sps = sps;
  a.sps_len = sps_len;
  a.B = B;
  a.K_max = K_max;
  a.ell = ell;
  a.tgt_off = tgt_off;
  a.theta_best = theta_best;
  a.b_star = nullptr;
  a.survival = nullptr;
  a.dev_status = dev_status;
  a.ws = workspace;
  a.mode = kSchedCapacity;
  a.capacity_out = capacity;
  return launch_schedule(a, (cudaStream_t)stream) == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
}

dspark_status dspark_schedule_topk(const float *conf, const int32_t *K_r, const int32_t *capacity, int64_t B,
                                   int64_t K_max, int32_t *ell, int32_t *tgt_off, int64_t *b_star, float *survival,
                                   void *workspace, size_t workspace_bytes, int32_t *dev_status, void *stream) {
  if (!conf || !K_r || !capacity || !ell || !tgt_off || !dev_status) return DSPARK_ERR_NULL;
  if (B < 1 || B > kMaxB || K_max < 1 || K_max > kMaxK) return DSPARK_ERR_DIMS;
  if (!workspace || !aligned256(workspace) || workspace_bytes < dspark_schedule_workspace_bytes(B, K_max))
    return DSPARK_ERR_WORKSPACE;
  ScheduleArgs a;
  a.conf = conf;
  a.K_r = K_r;
  a.sps = nullptr;
  a.sps_len = 0;
  a.B = B;
  a.K_max = K_max;
  a.ell = ell;
  a.tgt_off = tgt_off;
  a.theta_best = nullptr;
  a.b_star = b_star;
  a.survival = survival;
  a.dev_status = dev_status;
  a.ws = workspace;
  a.mode = kSchedTopK;
  a.capacity_in = capacity;
  return launch_schedule(a, (cudaStream_t)stream) == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
}

dspark_status dspark_schedule_threshold(const float *conf, const int32_t *K_r, float threshold, int32_t mode,
                                        int64_t B, int64_t K_max, int32_t *ell, int32_t *tgt_off, int64_t *b_star,
                                        float *survival, int32_t *dev_status, void *stream) {
  if (!conf || !K_r || !ell || !tgt_off || !dev_status) return DSPARK_ERR_NULL;
  if (B < 1 || B > kMaxB || K_max < 1 || K_max > kMaxK) return DSPARK_ERR_DIMS;
  if (mode != DSPARK_THRESHOLD_CONFIDENCE && mode != DSPARK_THRESHOLD_SURVIVAL) return DSPARK_ERR_DIMS;
  if (threshold != threshold) return DSPARK_ERR_CONFIDENCE;
  ScheduleArgs a;
  a.conf = conf;
  a.K_r = K_r;
  a.sps = nullptr;
  a.sps_len = 0;
  a.B = B;
  a.K_max = K_max;
  a.ell = ell;
  a.tgt_off = tgt_off;
  a.theta_best = nullptr;
  a.b_star = b_star;
  a.survival = survival;
  a.dev_status = dev_status;
  a.ws = nullptr;
  a.mode = mode == DSPARK_THRESHOLD_CONFIDENCE ? kSchedThresholdConf : kSchedThresholdSurv;
  a.threshold = threshold;
  return launch_schedule(a, (cudaStream_t)stream) == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// verify
// ---------------------------------------------------------------------------
size_t dspark_verify_workspace_bytes(int64_t B, int64_t V) {
  if (B < 1 || V < 2) return 0;
  return verify_ws_bytes(B, V, nullptr);
}

dspark_status dspark_verify_ragged(const void *draft_logits, const float *draft_lse, const void *tgt_logits,
                                   const int32_t *tgt_off, const int32_t *ell, const int32_t *draft_tok,
                                   const float *temperature, uint64_t seed, dspark_dims dims, int32_t *n_acc,
                                   int32_t *out_tok, void *workspace, size_t workspace_bytes,
                                   int32_t *dev_status, void *stream) {
  if (!draft_logits || !tgt_logits || !tgt_off || !ell || !draft_tok || !temperature || !n_acc || !out_tok ||
      !dev_status)
    return DSPARK_ERR_NULL;
  dspark_status st = check_dims(dims, false);
  if (st != DSPARK_OK) return st;
  if (!workspace || !aligned256(workspace) || workspace_bytes < dspark_verify_workspace_bytes(dims.B, dims.V))
    return DSPARK_ERR_WORKSPACE;
  DeviceInfo dev;
  if (!device_info(&dev)) return DSPARK_ERR_CUDA;
  VerifyArgs a;
  a.D = draft_logits;
  a.D_lse = draft_lse;
  a.tgt = tgt_logits;
  a.tgt_off = tgt_off;
  a.ell = ell;
  a.draft_tok = draft_tok;
  a.temperature = temperature;
  a.n_acc = n_acc;
  a.out_tok = out_tok;
  a.dev_status = dev_status;
  a.B = dims.B;
  a.K_max = dims.K_max;
  a.V = dims.V;
  a.dtype = dims.dtype;
  a.key = make_philox_key(seed);
  verify_carve(a, workspace);
  return launch_verify(a, (cudaStream_t)stream, dev.sms) == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
}

// Recompute entry point: the verify workspace, then the residual pass's jobs [B], keys [B],
// flags [B], active counts [3], barrier counters [2], and the packed W2 when the caller
// passes W as given.
static size_t verify_markov_extra(const dspark_dims &d) {
  size_t n = al256(8 * (size_t)d.B) + al256(sizeof(int32_t) * (size_t)d.B) + al256(sizeof(int32_t) * 2);
  if (!(d.flags & DSPARK_FLAG_W_PACKED)) n += al256(draft_packed_bytes(d.rank, d.V));
  return n;
}

size_t dspark_verify_markov_workspace_bytes(dspark_dims dims) {
  if (check_dims(dims, true) != DSPARK_OK) return 0;
  if (dims.dtype != DSPARK_BF16 || dims.rank % 64 != 0 || dims.rank > 256 || dims.V % 8 != 0) return 0;
  return verify_ws_bytes(dims.B, dims.V, nullptr) + verify_markov_extra(dims);
}

dspark_status dspark_verify_markov(const void *U, const void *E, const void *W, const int32_t *anchor,
                                   const float *draft_lse, const float *draft_tok_logit, const void *tgt_logits,
                                   const int32_t *tgt_off, const int32_t *ell, const int32_t *draft_tok,
                                   const float *temperature, uint64_t seed, dspark_dims dims, int32_t *n_acc,
                                   int32_t *out_tok, void *workspace, size_t workspace_bytes, int32_t *dev_status,
                                   void *stream) {
  if (!U || !E || !W || !anchor || !draft_lse || !draft_tok_logit || !tgt_logits || !tgt_off || !ell ||
      !draft_tok || !temperature || !n_acc || !out_tok || !dev_status)
    return DSPARK_ERR_NULL;
  dspark_status st = check_dims(dims, true);
  if (st != DSPARK_OK) return st;
  const size_t need = dspark_verify_markov_workspace_bytes(dims);
  if (need == 0 || (((uintptr_t)U | (uintptr_t)E | (uintptr_t)W | (uintptr_t)tgt_logits) & 15u))
    return DSPARK_ERR_UNSUPPORTED;   // the recompute runs on the tensor-core path only
  if (!workspace || !aligned256(workspace) || workspace_bytes < need) return DSPARK_ERR_WORKSPACE;
  DeviceInfo dev;
  if (!device_info(&dev)) return DSPARK_ERR_CUDA;
  if (dev.major != 10 || dev.minor != 3) return DSPARK_ERR_UNSUPPORTED;
  VerifyArgs a;
  a.D = nullptr;
  a.D_lse = draft_lse;
  a.D_zx = draft_tok_logit;
  a.tgt = tgt_logits;
  a.tgt_off = tgt_off;
  a.ell = ell;
  a.draft_tok = draft_tok;
  a.temperature = temperature;
  a.n_acc = n_acc;
  a.out_tok = out_tok;
  a.dev_status = dev_status;
  a.B = dims.B;
  a.K_max = dims.K_max;
  a.V = dims.V;
  a.dtype = dims.dtype;
  a.key = make_philox_key(seed);
  verify_carve(a, workspace);
  char *p = (char *)workspace + verify_ws_bytes(dims.B, dims.V, nullptr);
  a.anchor = anchor;
  a.key_out = (unsigned long long *)p;
  a.resid_key = a.key_out;
  p += al256(8 * (size_t)dims.B);
  a.any_out = (int32_t *)p;
  a.resid_any = a.any_out;
  p += al256(sizeof(int32_t) * (size_t)dims.B);
  a.jobs_gbar = (int32_t *)p;
  p += al256(sizeof(int32_t) * 2);
  // the residual pass: the draft kernel's residual mode over the jobs
  DraftArgs r;
  r.U = U;
  r.E = E;
  r.W = W;
  r.Wp = (dims.flags & DSPARK_FLAG_W_PACKED) ? W : (const void *)p;
  r.anchor = anchor;
  r.K_r = nullptr;
  r.temperature = temperature;
  r.draft_tok = nullptr;
  r.draft_logits = nullptr;
  r.draft_lse = nullptr;
  r.draft_zx = nullptr;
  r.dev_status = dev_status;
  r.B = dims.B;
  r.K_max = 1;
  r.u_rows = dims.B * dims.K_max;
  r.V = dims.V;
  r.rank = dims.rank;
  r.dtype = dims.dtype;
  r.key = a.key;
  r.perm = r.iperm = r.counters = r.act = r.grp = nullptr;
  r.nact = a.jobs_nact;
  r.best_key = a.key_out;
  r.gbar = a.jobs_gbar;
  r.partials = nullptr;
  r.zx_part = nullptr;
  r.partial_slots = 0;
  r.jobs = a.jobs;
  r.tgt = tgt_logits;
  r.resid_any = a.any_out;
  cudaStream_t s = (cudaStream_t)stream;
  if (!(dims.flags & DSPARK_FLAG_W_PACKED) && launch_pack_projection(W, dims.rank, dims.V, (void *)r.Wp, s) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  return launch_verify(a, s, dev.sms, &r) == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
}

}  // extern "C"
