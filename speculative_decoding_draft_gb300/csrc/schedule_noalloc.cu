// Allocation-free variant of dspark_schedule_survival.
//
// Some callers cannot allocate device memory at the point where they schedule:
// a serving loop that must not call cudaMalloc between steps (it synchronises
// the whole device and stalls the pipeline), or a plugin loaded into a host
// process whose allocator owns all device memory and hands it no workspace.
// This entry point runs the same scheduler kernel on a scratch area that lives
// in this library's own static device memory instead of a caller workspace.
//
// The scratch array below is part of the library image: every GPU on which the
// library is loaded holds it (DSPARK_NOALLOC_SCRATCH_BYTES, about 1 MiB) until
// the process exits.  Host code cannot use the array's name as a device
// address, so the first call on each device, with that device current, looks
// the address up with cudaGetSymbolAddress and caches it; make that first call
// before any stream capture.  All calls share the one array, so two calls whose
// kernels overlap on the GPU (different streams without ordering) race on it.
// The scheduler writes every scratch entry it later reads, so nothing in the
// array needs to start at zero and no clearing is done.
#include <mutex>

#include "schedule.cuh"

namespace {

constexpr int64_t kMaxCandidates = DSPARK_NOALLOC_MAX_CANDIDATES;

// Same carve-up as the caller workspace of dspark_schedule_survival at the maximum size.
constexpr size_t al256(size_t x) { return (x + 255) & ~(size_t)255; }
constexpr size_t kScratchBytes = 4 * al256((size_t)kMaxCandidates * 4) + al256((size_t)kMaxCandidates * 8) +
                                 al256((size_t)(kMaxCandidates + 1) * 8);
static_assert(kScratchBytes <= DSPARK_NOALLOC_SCRATCH_BYTES, "scratch size");

static __device__ __align__(256) unsigned char g_schedule_scratch[DSPARK_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void *g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array for the current device (looked up once per device).
dspark_status scratch_for_current_device(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DSPARK_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_schedule_scratch) != cudaSuccess || p == nullptr) return DSPARK_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return DSPARK_OK;
}

}  // namespace

extern "C" dspark_status dspark_schedule_survival_noalloc(const float *conf, const int32_t *K_r, const double *sps,
                                                          int64_t sps_len, int64_t B, int64_t K_max, int32_t *ell,
                                                          int32_t *tgt_off, double *theta_best, int64_t *b_star,
                                                          float *survival, int32_t *dev_status, void *stream) {
  if (!conf || !K_r || !sps || !ell || !tgt_off || !dev_status) return DSPARK_ERR_NULL;
  if (B < 1 || K_max < 1 || K_max > dspark::kMaxK || sps_len < 1) return DSPARK_ERR_DIMS;
  if (B * K_max > kMaxCandidates) return DSPARK_ERR_WORKSPACE;   // beyond the static scratch
  void *scratch = nullptr;
  const dspark_status st = scratch_for_current_device(&scratch);
  if (st != DSPARK_OK) return st;
  dspark::ScheduleArgs a;
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
  a.ws = scratch;
  return dspark::launch_schedule(a, (cudaStream_t)stream) == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
}
