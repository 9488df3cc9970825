// Host-side launchers of the library's kernels (internal).
#pragma once

#include <mutex>

#include "chunk_common.cuh"

namespace sala {

// Kernels of the library, for the timing instrumentation (names in api.cu).
enum KernelId {
    kKSegTable = 0,
    kKPrefillFused,
    kKRecurrentStep,
    kKRecurrentStepIndexed,
    kKOutputNormGate,
    kKQkPrologue,
    kKGdnStep,
    kKGdnFwd,
    kKGdnNewv,
    kKPrefillPair,
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

// The q/k prologue in kernel-argument form (qw null: none). inv_freq[i] = float(theta^(-i/64)),
// computed on the host in double precision and rounded once.
struct QkPrologue {
    const uint16_t *qw = nullptr, *kw = nullptr;   // bf16 [128] RMSNorm weights
    const int64_t *pos = nullptr;                  // decode: [N] positions
    float eps = 0.f;
    float inv_freq[64] = {};
};
QkPrologue make_qk_prologue(const sala_qk_prologue *p, const int64_t *positions);

// The same step on states in a pool [P, H, 128, 128] (fp32, or bf16 if `bf16`) addressed by
// idx[N] (negative: padding row, o = 0; >= P: SALA_ERR_BAD_INDEX recorded in `status`), with
// the q/k prologue fused if pro.qw is set.
cudaError_t launch_recurrent_step_indexed(const void *q, const void *k, const void *v,
                                          const float *g, float scale, void *pool, bool bf16,
                                          const int32_t *idx, int64_t P, void *o, int64_t N,
                                          int H, const QkPrologue &pro, int *status,
                                          cudaStream_t stream);

// The q/k prologue in place on a prefill's q and k ([T_total, H, 128] rows; positions from
// the segment table's sequence bounds plus start_pos).
cudaError_t launch_qk_prologue(void *q, void *k, const QkPrologue &pro, const SegTable &t,
                               const int64_t *start_pos, int64_t T_total, int H, int *status,
                               cudaStream_t stream);

// Segment table from cu_seqlens (or B equal rows); also zeroes the work ticket and the
// hand-off flags of the fused prefill, and writes hT (= h0, or zeros) of empty sequences.
cudaError_t launch_seg_table(const SegTable &t, int64_t T_total, uint32_t *ticket,
                             uint32_t *flags, int64_t nflags, int H, const float *h0, float *hT,
                             int *status, cudaStream_t st);

// The fused tensor-core prefill (prefill_fused.cu): one persistent launch of `grid` CTAs
// (the final state of empty sequences is written by the segment-table kernel). `incl` holds [max_units, 128, 128] fp32 hand-off
// states, `flags` [max_units] words, `ticket` one word; `epoch` is nonzero and differs from
// the previous call's. `status` receives SALA_ERR_TIMEOUT if a bounded wait gives up.
cudaError_t setup_fused_kernel();

// The same prefill at two CTAs per SM (prefill_pair.cu): one unit in flight per CTA, half of
// an SM's shared and tensor memory each; `grid` up to twice the SM count. Same arguments.
cudaError_t launch_prefill_pair(const ChunkArgs &a, const SegTable &t, int64_t T_total,
                                int64_t max_units, const float *h0, float *hT, float *incl,
                                uint32_t *flags, uint32_t *ticket, uint32_t epoch, int grid,
                                int *status, cudaStream_t st);
cudaError_t setup_pair_kernel();
cudaError_t launch_prefill_fused(const ChunkArgs &a, const SegTable &t, int64_t T_total,
                                 int64_t max_units, const float *h0, float *hT, float *incl,
                                 uint32_t *flags, uint32_t *ticket, uint32_t epoch, int grid,
                                 int *status, cudaStream_t st);

// out[t] = RMSNorm(o[t]) * w * sigmoid(z[t]) over the H * 128 features of each of T tokens
// (bf16 in and out, fp32 arithmetic); out may be o.
cudaError_t launch_output_norm_gate(const void *o, const void *z, const void *w, float eps,
                                    void *out, int64_t T, int H, cudaStream_t stream);

// One gated-delta-rule step on [units] dense fp32 states (one CTA per (sequence, head)).
cudaError_t launch_gdn_step(const void *q, const void *k, const void *v, const float *g,
                            const float *beta, float scale, float *S, void *o, int64_t units,
                            cudaStream_t stream);

// The gated delta rule over whole sequences (recurrent form), one CTA per (sequence, head);
// sequence bounds from t.cu (or rows of t.T_row tokens); h0 / hT may be null.
cudaError_t launch_gdn_fwd(const void *q, const void *k, const void *v, const float *g,
                           const float *beta, float scale, const float *h0, const SegTable &t,
                           int64_t T_total, void *o, float *hT, int H, cudaStream_t stream);

// Failure-path test settings of the fused prefill (sala_gla_debug_prefill_knobs): the limit
// of the wait for a predecessor's state (0: the default 2 s) and a unit whose flag is withheld
// (-1: none).
void prefill_fault_knobs(uint64_t *wait_ns, int64_t *withhold);

// The gated delta rule's chunked form: new_v = U - W S of every token (bf16 [T_total, H, 128]
// into nv) for sala_gla_gdn_chunk_fwd, one CTA per (sequence, head); sequence bounds from t.cu
// (or rows of t.T_row tokens), kept inside the tensors.
cudaError_t setup_gdn_chunk_kernel();
cudaError_t launch_gdn_newv(const void *k, const void *v, const float *g, const float *beta,
                            const float *h0, const SegTable &t, int64_t T_total, void *nv, int H,
                            int *status, cudaStream_t st);

// Nonzero tag of one prefill call for the hand-off flags (differs from the previous call's).
uint32_t next_prefill_epoch();

// Tokens per segment of the fused prefill for T_total tokens and H heads on sm_count SMs.
int64_t choose_segment_tokens(int64_t T_total, int64_t H, int sm_count);

}  // namespace sala
