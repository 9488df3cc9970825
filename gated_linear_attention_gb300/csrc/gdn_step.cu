// One-token recurrent step of the gated delta rule (GDN), state updated in place.
//
// "Formulas and Code for Adapting Inference to GDN/KDA Linear Modules", section 1.1: per
// (sequence, head) with the [128 x 128] state S (row = key dimension): the state decays by
// alpha = exp(g); the memory read at the key, kv = k S (a vector over the value dimension),
// is replaced by the new value through the write strength beta: v_new = beta (v - kv),
// S <- S + k^T v_new; o = scale q S. The decay comes before the read, as in the page's chunked
// form (section 1.2, whose W carries exp(g)).
//
// One CTA of 256 threads per (sequence, head), the dense decode kernel's layout: warp w owns
// rows [16w, 16w + 16), lane l the columns [4l, 4l + 4) (512-byte rows per warp instruction).
// The state is streamed in once; kv needs every row, so the 8 warps' partial sums meet in
// shared memory, then the update is applied, stored, and q S reduced the same way. HBM-bound:
// the state is read and written once.
#include "launch.h"

namespace sala {

constexpr int kGdnThreads = 256;
constexpr int kGdnRows = kD / (kGdnThreads / 32);   // 16 rows per warp

__global__ void __launch_bounds__(kGdnThreads)
gdn_step_kernel(const uint16_t *__restrict__ q, const uint16_t *__restrict__ k,
                const uint16_t *__restrict__ v, const float *__restrict__ g,
                const float *__restrict__ beta, float scale, float *__restrict__ S,
                uint16_t *__restrict__ o) {
    const int unit = blockIdx.x;  // n * H + h
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float *Su = S + static_cast<size_t>(unit) * kD * kD;
    const int row0 = warp * kGdnRows;

    float4 s[kGdnRows];
#pragma unroll
    for (int r = 0; r < kGdnRows; ++r)
        s[r] = __ldcs(reinterpret_cast<const float4 *>(Su + (row0 + r) * kD) + lane);

    __shared__ float q_s[kD], k_s[kD];
    __shared__ float part[kGdnThreads / 32][kD];
    const size_t vec = static_cast<size_t>(unit) * kD;
    if (threadIdx.x < kD) {
        q_s[threadIdx.x] = bf16_bits_to_float(q[vec + threadIdx.x]);
        k_s[threadIdx.x] = bf16_bits_to_float(k[vec + threadIdx.x]);
    }
    const uint2 vw = *reinterpret_cast<const uint2 *>(v + vec + 4 * lane);
    const float2 v01 = bf16x2_to_float2(vw.x), v23 = bf16x2_to_float2(vw.y);
    const float alpha = expf(g[unit]), b = beta[unit];
    __syncthreads();

    // decay, and this warp's part of kv = k S over its rows
    float4 kv = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int r = 0; r < kGdnRows; ++r) {
        const float ki = k_s[row0 + r];
        s[r].x *= alpha;
        s[r].y *= alpha;
        s[r].z *= alpha;
        s[r].w *= alpha;
        kv.x = fmaf(ki, s[r].x, kv.x);
        kv.y = fmaf(ki, s[r].y, kv.y);
        kv.z = fmaf(ki, s[r].z, kv.z);
        kv.w = fmaf(ki, s[r].w, kv.w);
    }
    *reinterpret_cast<float4 *>(&part[warp][4 * lane]) = kv;
    __syncthreads();
    float4 kvs = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < kGdnThreads / 32; ++w) {
        const float4 p = *reinterpret_cast<const float4 *>(&part[w][4 * lane]);
        kvs.x += p.x;
        kvs.y += p.y;
        kvs.z += p.z;
        kvs.w += p.w;
    }
    const float4 vn = make_float4(b * (v01.x - kvs.x), b * (v01.y - kvs.y), b * (v23.x - kvs.z),
                                  b * (v23.y - kvs.w));
    __syncthreads();   // every warp has read its kv before part is reused

    // S <- S + k^T v_new, stored back; q S over this warp's rows
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int r = 0; r < kGdnRows; ++r) {
        const float ki = k_s[row0 + r], qi = q_s[row0 + r];
        float4 x = s[r];
        x.x = fmaf(ki, vn.x, x.x);
        x.y = fmaf(ki, vn.y, x.y);
        x.z = fmaf(ki, vn.z, x.z);
        x.w = fmaf(ki, vn.w, x.w);
        __stcs(reinterpret_cast<float4 *>(Su + (row0 + r) * kD) + lane, x);
        acc.x = fmaf(qi, x.x, acc.x);
        acc.y = fmaf(qi, x.y, acc.y);
        acc.z = fmaf(qi, x.z, acc.z);
        acc.w = fmaf(qi, x.w, acc.w);
    }
    *reinterpret_cast<float4 *>(&part[warp][4 * lane]) = acc;
    __syncthreads();
    if (threadIdx.x < kD / 2) {
        const int j = 2 * threadIdx.x;
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int w = 0; w < kGdnThreads / 32; ++w) {
            a0 += part[w][j];
            a1 += part[w][j + 1];
        }
        reinterpret_cast<uint32_t *>(o + vec)[threadIdx.x] = float2_to_bf16x2(scale * a0, scale * a1);
    }
}

cudaError_t launch_gdn_step(const void *q, const void *k, const void *v, const float *g,
                            const float *beta, float scale, float *S, void *o, int64_t units,
                            cudaStream_t stream) {
    if (units == 0) return cudaSuccess;
    LaunchTimer timer(kKGdnStep, stream);
    gdn_step_kernel<<<static_cast<unsigned>(units), kGdnThreads, 0, stream>>>(
        static_cast<const uint16_t *>(q), static_cast<const uint16_t *>(k),
        static_cast<const uint16_t *>(v), g, beta, scale, S, static_cast<uint16_t *>(o));
    return cudaGetLastError();
}

}  // namespace sala

namespace sala {

// ---------------------------------------------------------------------------------------
// The recurrent form over whole sequences (the page's recurrent prefill, used for short
// sequences): one CTA per (sequence, head) keeps the state in registers for all its tokens
// (the decode kernel's layout: warp w rows [16w, 16w + 16), lane l columns [4l, 4l + 4)), so
// the state is read once (h0) and written once (hT). Per token: the decay and this warp's part
// of kv = k S, an exchange between the warps, the delta-rule update, and this warp's part of
// q S; the token's output is summed after the next exchange. The next token's q, k, v, g, beta
// are loaded while the current one is worked on.
__global__ void __launch_bounds__(kGdnThreads, 2)
gdn_fwd_kernel(const uint16_t *__restrict__ q, const uint16_t *__restrict__ k,
               const uint16_t *__restrict__ v, const float *__restrict__ g,
               const float *__restrict__ beta, float scale, const float *__restrict__ h0,
               SegTable t, int64_t T_total, uint16_t *__restrict__ o, float *__restrict__ hT, int H) {
    const int nh = blockIdx.x;   // n * H + h
    const int n = nh / H, h = nh - n * H;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row0 = warp * kGdnRows;
    // sequence bounds, kept inside the token range whatever cu_seqlens holds
    const int64_t bos = min(max(seq_begin(t, n), int64_t(0)), T_total);
    const int64_t eos = min(max(seq_begin(t, n + 1), bos), T_total);

    float4 s[kGdnRows];
    if (h0) {
        const float *src = h0 + static_cast<size_t>(nh) * kD * kD;
#pragma unroll
        for (int r = 0; r < kGdnRows; ++r) s[r] = *(reinterpret_cast<const float4 *>(src + (row0 + r) * kD) + lane);
    } else {
#pragma unroll
        for (int r = 0; r < kGdnRows; ++r) s[r] = make_float4(0.f, 0.f, 0.f, 0.f);
    }

    __shared__ float qk_s[2][2][kD];                    // [buffer][q, k][i]
    __shared__ float part[kGdnThreads / 32][kD];         // kv partials
    __shared__ float part_o[kGdnThreads / 32][kD];       // q S partials
    // token inputs in registers: q_i, k_i (thread i < 128), v (my 4 columns), g, beta
    float rq = 0.f, rk = 0.f, rg = 0.f, rb = 0.f;
    uint2 rv = make_uint2(0u, 0u);
    auto load_token = [&](int64_t tok) {
        const size_t vec = (static_cast<size_t>(tok) * H + h) * kD;
        if (threadIdx.x < kD) {
            rq = bf16_bits_to_float(q[vec + threadIdx.x]);
            rk = bf16_bits_to_float(k[vec + threadIdx.x]);
        }
        rv = *reinterpret_cast<const uint2 *>(v + vec + 4 * lane);
        rg = g[static_cast<size_t>(tok) * H + h];
        rb = beta[static_cast<size_t>(tok) * H + h];
    };
    if (bos < eos) load_token(bos);
    for (int64_t tok = bos; tok < eos; ++tok) {
        const int b = static_cast<int>(tok - bos) & 1;
        if (threadIdx.x < kD) {
            qk_s[b][0][threadIdx.x] = rq;
            qk_s[b][1][threadIdx.x] = rk;
        }
        const float2 v01 = bf16x2_to_float2(rv.x), v23 = bf16x2_to_float2(rv.y);
        const float alpha = expf(rg), bt = rb;
        if (tok + 1 < eos) load_token(tok + 1);
        __syncthreads();
        // the previous token's output (its partials were written before this barrier)
        if (tok > bos && threadIdx.x < kD / 2) {
            const int j = 2 * threadIdx.x;
            float a0 = 0.f, a1 = 0.f;
#pragma unroll
            for (int w = 0; w < kGdnThreads / 32; ++w) {
                a0 += part_o[w][j];
                a1 += part_o[w][j + 1];
            }
            reinterpret_cast<uint32_t *>(o + (static_cast<size_t>(tok - 1) * H + h) * kD)[threadIdx.x] =
                float2_to_bf16x2(scale * a0, scale * a1);
        }
        // decay and this warp's part of kv = k S
        float4 kv = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int r = 0; r < kGdnRows; ++r) {
            const float ki = qk_s[b][1][row0 + r];
            s[r].x *= alpha;
            s[r].y *= alpha;
            s[r].z *= alpha;
            s[r].w *= alpha;
            kv.x = fmaf(ki, s[r].x, kv.x);
            kv.y = fmaf(ki, s[r].y, kv.y);
            kv.z = fmaf(ki, s[r].z, kv.z);
            kv.w = fmaf(ki, s[r].w, kv.w);
        }
        *reinterpret_cast<float4 *>(&part[warp][4 * lane]) = kv;
        __syncthreads();
        float4 kvs = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < kGdnThreads / 32; ++w) {
            const float4 p = *reinterpret_cast<const float4 *>(&part[w][4 * lane]);
            kvs.x += p.x;
            kvs.y += p.y;
            kvs.z += p.z;
            kvs.w += p.w;
        }
        const float4 vn = make_float4(bt * (v01.x - kvs.x), bt * (v01.y - kvs.y),
                                      bt * (v23.x - kvs.z), bt * (v23.y - kvs.w));
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int r = 0; r < kGdnRows; ++r) {
            const float ki = qk_s[b][1][row0 + r], qi = qk_s[b][0][row0 + r];
            s[r].x = fmaf(ki, vn.x, s[r].x);
            s[r].y = fmaf(ki, vn.y, s[r].y);
            s[r].z = fmaf(ki, vn.z, s[r].z);
            s[r].w = fmaf(ki, vn.w, s[r].w);
            acc.x = fmaf(qi, s[r].x, acc.x);
            acc.y = fmaf(qi, s[r].y, acc.y);
            acc.z = fmaf(qi, s[r].z, acc.z);
            acc.w = fmaf(qi, s[r].w, acc.w);
        }
        *reinterpret_cast<float4 *>(&part_o[warp][4 * lane]) = acc;
    }
    __syncthreads();
    if (eos > bos && threadIdx.x < kD / 2) {
        const int j = 2 * threadIdx.x;
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int w = 0; w < kGdnThreads / 32; ++w) {
            a0 += part_o[w][j];
            a1 += part_o[w][j + 1];
        }
        reinterpret_cast<uint32_t *>(o + (static_cast<size_t>(eos - 1) * H + h) * kD)[threadIdx.x] =
            float2_to_bf16x2(scale * a0, scale * a1);
    }
    if (hT) {
        float *dst = hT + static_cast<size_t>(nh) * kD * kD;
#pragma unroll
        for (int r = 0; r < kGdnRows; ++r) *(reinterpret_cast<float4 *>(dst + (row0 + r) * kD) + lane) = s[r];
    }
}

cudaError_t launch_gdn_fwd(const void *q, const void *k, const void *v, const float *g,
                           const float *beta, float scale, const float *h0, const SegTable &t,
                           int64_t T_total, void *o, float *hT, int H, cudaStream_t stream) {
    if (t.nseq == 0) return cudaSuccess;
    LaunchTimer timer(kKGdnFwd, stream);
    gdn_fwd_kernel<<<static_cast<unsigned>(t.nseq * H), kGdnThreads, 0, stream>>>(
        static_cast<const uint16_t *>(q), static_cast<const uint16_t *>(k),
        static_cast<const uint16_t *>(v), g, beta, scale, h0, t, T_total, static_cast<uint16_t *>(o),
        hT, H);
    return cudaGetLastError();
}

}  // namespace sala
