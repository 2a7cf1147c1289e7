// Scheduler kernel interface: Algorithm 1 ("DSpark" S3.2.2), the capacity and top-K
// steps of the deployed asynchronous scheduler (S5.2) and the static thresholds.
#pragma once

#include "dspark_internal.cuh"

namespace dspark {

// Scheduler modes: Algorithm 1 with its early stop; the capacity of the asynchronous
// scheduler (global maximum of Theta along the greedy path); dynamic top-K admission of a
// given capacity; static thresholds on the confidences or on the survival products.
enum ScheduleMode : int {
  kSchedAlgorithm1 = 0,
  kSchedCapacity = 1,
  kSchedTopK = 2,
  kSchedThresholdConf = 3,
  kSchedThresholdSurv = 4
};

struct ScheduleArgs {
  const float *conf;
  const int32_t *K_r;
  const double *sps;
  int64_t sps_len, B, K_max;
  int32_t *ell, *tgt_off;
  double *theta_best;
  int64_t *b_star;
  float *survival;
  int32_t *dev_status;
  void *ws;
  int mode = kSchedAlgorithm1;
  const int32_t *capacity_in = nullptr;  // top-K: device [1], admitted candidates
  int32_t *capacity_out = nullptr;       // capacity: device [1], optional
  float threshold = 0.0f;                // threshold modes
};

size_t schedule_ws_bytes(int64_t B, int64_t K_max);
cudaError_t launch_schedule(const ScheduleArgs &a, cudaStream_t s);

}  // namespace dspark
