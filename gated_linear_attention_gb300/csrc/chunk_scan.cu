// Segment bookkeeping and the segment scan of the chunked prefill.
//
// The state is carried across a long sequence in three steps: a state pass computes, for
// every segment on its own, the state it would leave behind if it started from zero
// (dS_s) and its total log-decay (Bsum_s); this scan then walks the segments of each
// sequence in order,
//     S_in(0) = h0,   S_in(s+1) = exp(Bsum_s) * S_in(s) + dS_s,
// which is the recurrence of "MiniCPM-SALA — Complete Blueprint" ("Simple GLA Recurrence")
// applied a whole segment at a time: its unrolled form (section "Why Linear Attention Loses
// Information", Problem 1, S_n = alpha^n S_0 + sum alpha^(n-i) k_i^T v_i) splits into the
// decayed incoming state plus the segment's own contribution. The output pass then restarts
// every segment from S_in(s).
#include "launch.h"

namespace sala {

// ---------------------------------------------------------------------------------------
// Segment table: seg_off[n] = sum over m < n of ceil(len_m / seg_len); validates cu_seqlens.
// One block; each thread owns a contiguous range of sequences.
constexpr int kPrepThreads = 1024;

__global__ void __launch_bounds__(kPrepThreads)
seg_table_kernel(SegTable t, int64_t T_total, int *status) {
    __shared__ int64_t part[kPrepThreads];
    __shared__ int bad;
    if (threadIdx.x == 0) bad = 0;
    __syncthreads();
    const int64_t per = (t.nseq + kPrepThreads - 1) / kPrepThreads;
    const int64_t n0 = ::min(static_cast<int64_t>(threadIdx.x) * per, t.nseq);
    const int64_t n1 = ::min(n0 + per, t.nseq);
    int64_t local = 0;
    for (int64_t n = n0; n < n1; ++n) {
        const int64_t a = seq_begin(t, n), b = seq_begin(t, n + 1);
        if (b < a) bad = 1;
        else local += (b - a + t.seg_len - 1) / t.seg_len;
    }
    if (threadIdx.x == 0 && t.cu && (t.cu[0] != 0 || t.cu[t.nseq] != T_total)) bad = 1;
    part[threadIdx.x] = local;
    __syncthreads();
    // inclusive scan of the per-thread counts (Hillis-Steele)
    for (int off = 1; off < kPrepThreads; off <<= 1) {
        const int64_t add = threadIdx.x >= off ? part[threadIdx.x - off] : 0;
        __syncthreads();
        part[threadIdx.x] += add;
        __syncthreads();
    }
    int64_t run = threadIdx.x ? part[threadIdx.x - 1] : 0;
    for (int64_t n = n0; n < n1; ++n) {
        t.seg_off[n] = run;
        const int64_t a = seq_begin(t, n), b = seq_begin(t, n + 1);
        if (b >= a) run += (b - a + t.seg_len - 1) / t.seg_len;
    }
    if (threadIdx.x == kPrepThreads - 1) t.seg_off[t.nseq] = part[kPrepThreads - 1];
    __syncthreads();
    if (threadIdx.x == 0) {
        t.seg_off[t.nseq + 1] = bad ? 0 : 1;
        if (bad) record_status(status, SALA_ERR_BAD_SEQLENS);
    }
}

// ---------------------------------------------------------------------------------------
// Segment scan. ws_state[sigma][h] holds dS on entry and S_in on exit; ws_decay[sigma][h]
// holds Bsum. Grid: (nseq * H) x 16 blocks of 256 threads; a thread owns one float4 of the
// 128 x 128 state and walks the sequence's segments with the next segment's dS prefetched.
constexpr int kScanThreads = 256;
constexpr int kScanBlocksPerState = kD * kD / (4 * kScanThreads);  // 16

__global__ void __launch_bounds__(kScanThreads)
segment_scan_kernel(SegTable t, int H, float *__restrict__ ws_state,
                    const float *__restrict__ ws_decay, const float *__restrict__ h0,
                    float *__restrict__ hT) {
    if (t.seg_off[t.nseq + 1] != 1) return;
    const int64_t nh = blockIdx.x / kScanBlocksPerState;
    const int part = blockIdx.x % kScanBlocksPerState;
    const int64_t n = nh / H;
    const int h = static_cast<int>(nh % H);
    const int64_t e = (static_cast<int64_t>(part) * kScanThreads + threadIdx.x) * 4;  // element
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (h0) x = *reinterpret_cast<const float4 *>(h0 + nh * kD * kD + e);
    const int64_t s0 = t.seg_off[n], s1 = t.seg_off[n + 1];
    const size_t stride = static_cast<size_t>(H) * kD * kD;
    float *p = ws_state + (static_cast<size_t>(s0) * H + h) * kD * kD + e;
    float4 d = s0 < s1 ? *reinterpret_cast<const float4 *>(p) : x;
    for (int64_t s = s0; s < s1; ++s, p += stride) {
        const float4 cur = d;
        if (s + 1 < s1) d = *reinterpret_cast<const float4 *>(p + stride);
        const float a = expf(ws_decay[s * H + h]);
        *reinterpret_cast<float4 *>(p) = x;  // state entering segment s
        x.x = fmaf(a, x.x, cur.x);
        x.y = fmaf(a, x.y, cur.y);
        x.z = fmaf(a, x.z, cur.z);
        x.w = fmaf(a, x.w, cur.w);
    }
    if (hT) *reinterpret_cast<float4 *>(hT + nh * kD * kD + e) = x;
}

cudaError_t launch_seg_table(const SegTable &t, int64_t T_total, int *status, cudaStream_t st) {
    LaunchTimer timer(kKSegTable, st);
    seg_table_kernel<<<1, kPrepThreads, 0, st>>>(t, T_total, status);
    return cudaGetLastError();
}

cudaError_t launch_segment_scan(const SegTable &t, int H, float *ws_state, const float *ws_decay,
                                const float *h0, float *hT, cudaStream_t st) {
    const int64_t blocks = t.nseq * H * kScanBlocksPerState;
    if (blocks == 0) return cudaSuccess;
    LaunchTimer timer(kKSegmentScan, st);
    segment_scan_kernel<<<static_cast<unsigned>(blocks), kScanThreads, 0, st>>>(
        t, H, ws_state, ws_decay, h0, hT);
    return cudaGetLastError();
}

}  // namespace sala
