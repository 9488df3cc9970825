// Segment bookkeeping of the chunked prefill: which (sequence, token range) each segment
// covers, from cu_seqlens (validated on the device) or from B equal rows.
#include "launch.h"

namespace sala {

// ---------------------------------------------------------------------------------------
// Segment table: seg_off[n] = sum over m < n of ceil(len_m / seg_len); validates cu_seqlens.
// One block; each thread owns a contiguous range of sequences. Once the table is known to be
// valid, the block also writes hT of every empty sequence (its initial state, or zeros): the
// prefill kernel only visits sequences with tokens.
constexpr int kPrepThreads = 1024;

__global__ void __launch_bounds__(kPrepThreads)
seg_table_kernel(SegTable t, int64_t T_total, uint32_t *ticket, uint32_t *flags, int64_t nflags,
                 int H, const float *__restrict__ h0, float *__restrict__ hT, int *status) {
    __shared__ int64_t part[kPrepThreads];
    // the prefill kernel launched after this one may start its set-up now; it waits for this
    // grid to complete before it reads anything written here
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    for (int64_t i = threadIdx.x; i < nflags; i += kPrepThreads) flags[i] = 0u;
    if (threadIdx.x == 0 && ticket) *ticket = 0u;
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
    if (bad || !hT) return;
    // hT of empty sequences (the block-wide flag `bad` is final after the barrier above): a
    // block of kPrepThreads sequences at a time, each thread testing one, then the block copies
    // the state of every empty one
    constexpr int kVec = kD * kD / 4;   // float4 per (sequence, head)
    __shared__ bool empty[kPrepThreads];
    for (int64_t n0b = 0; n0b < t.nseq; n0b += kPrepThreads) {
        const int64_t nt = n0b + threadIdx.x;
        empty[threadIdx.x] = nt < t.nseq && seq_begin(t, nt + 1) == seq_begin(t, nt);
        __syncthreads();
        const int64_t nb = ::min(static_cast<int64_t>(kPrepThreads), t.nseq - n0b);
        for (int64_t m = 0; m < nb; ++m) {
            if (!empty[m]) continue;
            const int64_t n = n0b + m;
            float4 *dst = reinterpret_cast<float4 *>(hT + n * H * kD * kD);
            const float4 *src = h0 ? reinterpret_cast<const float4 *>(h0 + n * H * kD * kD) : nullptr;
            for (int64_t i = threadIdx.x; i < static_cast<int64_t>(H) * kVec; i += kPrepThreads)
                dst[i] = src ? src[i] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        __syncthreads();   // (the flags are rewritten for the next block of sequences)
    }
}

cudaError_t launch_seg_table(const SegTable &t, int64_t T_total, uint32_t *ticket,
                             uint32_t *flags, int64_t nflags, int H, const float *h0, float *hT,
                             int *status, cudaStream_t st) {
    LaunchTimer timer(kKSegTable, st);
    seg_table_kernel<<<1, kPrepThreads, 0, st>>>(t, T_total, ticket, flags, nflags, H, h0, hT, status);
    return cudaGetLastError();
}

}  // namespace sala
