// Host-side launchers of the library's kernels (internal).
#pragma once

#include <mutex>

#include "chunk_common.cuh"

namespace sala {

// Kernels of the library, for the timing instrumentation (names in api.cu).
enum KernelId {
    kKSegTable = 0,
    kKStatePass,
    kKSegmentScan,
    kKOutputPass,
    kKRecurrentStep,
    kKernelCount
};

// While timing is enabled, brackets one launch with events on `stream` (no-op otherwise).
class LaunchTimer {
  public:
    LaunchTimer(KernelId id, cudaStream_t stream);
    ~LaunchTimer();
    LaunchTimer(const LaunchTimer &) = delete;
    LaunchTimer &operator=(const LaunchTimer &) = delete;

  private:
    KernelId id_;
    cudaStream_t stream_;
    cudaEvent_t start_ = nullptr;
};

// Device address of the library's status word on the current device.
cudaError_t device_status_address(int **out);

cudaError_t launch_recurrent_step(const void *q, const void *k, const void *v, const float *g,
                                  float scale, float *S, void *o, int64_t units,
                                  cudaStream_t stream);

cudaError_t launch_seg_table(const SegTable &t, int64_t T_total, int *status, cudaStream_t st);
cudaError_t launch_segment_scan(const SegTable &t, int H, float *ws_state, const float *ws_decay,
                                const float *h0, float *hT, cudaStream_t st);

// Tensor-core state and output passes (chunk_tc.cu). `status` receives SALA_ERR_TIMEOUT if a
// bounded device-side wait gives up.
cudaError_t setup_tc_kernels();
cudaError_t launch_state_pass(const ChunkArgs &a, const SegTable &t, int64_t T_total,
                              int64_t max_units, int *status, cudaStream_t st);
cudaError_t launch_output_pass(const ChunkArgs &a, const SegTable &t, int64_t T_total,
                               int64_t max_units, int *status, cudaStream_t st);

}  // namespace sala
