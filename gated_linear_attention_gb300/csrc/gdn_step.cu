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
    dependent_start();   // (launched by launch_dependent: one decode step after another)
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
    return launch_dependent(gdn_step_kernel, static_cast<unsigned>(units), kGdnThreads, stream,
                            static_cast<const uint16_t *>(q), static_cast<const uint16_t *>(k),
                            static_cast<const uint16_t *>(v), g, beta, scale, S,
                            static_cast<uint16_t *>(o));
}

}  // namespace sala

namespace sala {

// ---------------------------------------------------------------------------------------
// The recurrent form over whole sequences (the page's recurrent prefill, used for short
// sequences). One CTA of 8 warps per (sequence, head); warp w owns the 16 value columns
// [16w, 16w + 16) of the state for all 128 key rows and runs the sequence alone: no barrier
// and nothing shared with the other warps. Lane l = cg + 4 rg keeps rows [16 rg, 16 rg + 16)
// of the columns 16w + 4 cg + [0, 4) in registers. The sums over rows (k S and q S) end in
// three shuffle levels that also spread the four columns over the lanes: afterwards the lane
// whose bits 4 and 3 read m holds column 16w + 4 cg + m. For that to need no selects, slot j
// of a lane's four registers holds column 16w + 4 cg + (j xor m). The state is read once (h0)
// and written once (hT).
//
// The decay is kept out of the stored state: the warp holds S~ with S = c S~, c the product
// of the gates exp(g) since the last renormalisation. Then kv = c (k S~), the update adds
// k^T (v_new / c) to S~, and o = scale c (q S~): three multiply-adds per state entry and
// token instead of a multiply and three. When c leaves [2^-40, 2^40] (a gate of 0 included)
// S~ is multiplied by c and c reset to 1 before the token's read, so S~ stays well inside the
// fp32 range. Each warp copies its next tokens' inputs into shared memory asynchronously,
// four tokens ahead, so the loads' latency stays off the token-to-token chain. The
// multiply-adds are the packed two-wide fp32 kind, over pairs of adjacent rows.
constexpr float kGdnCLo = 0x1p-40f, kGdnCHi = 0x1p40f;
constexpr int kGdnRing = 5;     // token slots per warp
constexpr int kGdnSlot = 576;   // q 256 B, k 256 B, the warp's v 32 B, g, beta (16-byte multiple)

// Asynchronous copy of 16 (or 4) bytes into shared memory, issued only where `on` is set.
__device__ __forceinline__ void gdn_cp_async16(uint32_t dst, const void *src, bool on) {
    asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %2, 0;\n @p cp.async.ca.shared.global [%0], [%1], 16;\n}\n"
                 ::"r"(dst), "l"(src), "r"(static_cast<int>(on)) : "memory");
}
__device__ __forceinline__ void gdn_cp_async4(uint32_t dst, const void *src, bool on) {
    asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %2, 0;\n @p cp.async.ca.shared.global [%0], [%1], 4;\n}\n"
                 ::"r"(dst), "l"(src), "r"(static_cast<int>(on)) : "memory");
}
__device__ __forceinline__ float gdn_ex2(float x) {
    float y;
    asm("ex2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Components reordered so that slot j holds component j xor m (its own inverse).
__device__ __forceinline__ float4 gdn_perm(float4 f, int m) {
    if (m & 2) f = make_float4(f.z, f.w, f.x, f.y);
    if (m & 1) f = make_float4(f.y, f.x, f.w, f.z);
    return f;
}

// Sum a lane's four column partials over the 8 row groups (lane bits 2..4). With slot j
// holding column j xor m, the lane 16 apart holds the same two columns in its slots 2, 3 that
// this lane keeps in slots 0, 1, and the lane 8 apart the kept column in its second place;
// the result is column m (the same in the two lanes that differ in bit 2).
__device__ __forceinline__ float gdn_rows_sum(float4 a) {
    const float p0 = a.x + __shfl_xor_sync(0xffffffffu, a.z, 16);
    const float p1 = a.y + __shfl_xor_sync(0xffffffffu, a.w, 16);
    const float r = p0 + __shfl_xor_sync(0xffffffffu, p1, 8);
    return r + __shfl_xor_sync(0xffffffffu, r, 4);
}

// Eight bf16 -> four pairs of floats (element 2i, element 2i + 1).
__device__ __forceinline__ void gdn_unpack8(uint4 x, float2 *f) {
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) f[i] = make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
}

__global__ void __launch_bounds__(kGdnThreads, 2)
gdn_fwd_kernel(const uint16_t *__restrict__ q, const uint16_t *__restrict__ k,
               const uint16_t *__restrict__ v, const float *__restrict__ g,
               const float *__restrict__ beta, float scale, const float *__restrict__ h0,
               SegTable t, int64_t T_total, uint16_t *__restrict__ o, float *__restrict__ hT, int H) {
    const int nh = blockIdx.x;   // n * H + h
    const int n = nh / H, h = nh - n * H;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cg = lane & 3, row0 = 16 * (lane >> 2), col0 = 16 * warp + 4 * cg;
    const int m = (lane >> 3) & 3;   // this lane's column after gdn_rows_sum: col0 + m
    // sequence bounds, kept inside the token range whatever cu_seqlens holds
    const int64_t bos = min(max(seq_begin(t, n), int64_t(0)), T_total);
    const int64_t eos = min(max(seq_begin(t, n + 1), bos), T_total);

    // s[p][j] = (S~[row0 + 2p][col], S~[row0 + 2p + 1][col]), col the column of slot j: row
    // pairs, so that packed two-wide multiply-adds take the key and query pairs as they unpack
    float2 s[8][4];
#pragma unroll
    for (int p = 0; p < 8; ++p) {
        float4 e = make_float4(0.f, 0.f, 0.f, 0.f), f = e;
        if (h0) {
            const float *src = h0 + static_cast<size_t>(nh) * kD * kD + col0 + (row0 + 2 * p) * kD;
            e = gdn_perm(*reinterpret_cast<const float4 *>(src), m);
            f = gdn_perm(*reinterpret_cast<const float4 *>(src + kD), m);
        }
        s[p][0] = make_float2(e.x, f.x);
        s[p][1] = make_float2(e.y, f.y);
        s[p][2] = make_float2(e.z, f.z);
        s[p][3] = make_float2(e.w, f.w);
    }
    float c = 1.f;

    // Token inputs go through a ring of kGdnRing slots per warp, kGdnRing - 1 tokens ahead:
    // lanes 0-15 copy 16 bytes of k each, lanes 16-31 of q, lanes 0-1 the warp's 16 values of
    // v, lanes 2-3 g and beta.
    __shared__ __align__(16) unsigned char ring_all[kGdnThreads / 32][kGdnRing][kGdnSlot];
    const uint32_t ring = static_cast<uint32_t>(__cvta_generic_to_shared(ring_all[warp]));
    const uint16_t *qk_src = (lane < 16 ? k : q) + 8 * (lane & 15);
    const uint32_t qk_dst = (lane < 16 ? 256u : 0u) + 16u * (lane & 15);
    const uint16_t *v_src = v + 16 * warp + 8 * (lane & 1);
    const float *gb_src = (lane & 1) ? beta : g;
    const uint32_t x_dst = lane < 2 ? 512u + 16u * lane : 544u + 4u * (lane & 1);
    const bool v_lane = lane < 2, gb_lane = lane == 2 || lane == 3;
    size_t gi_fetch = static_cast<size_t>(bos) * H + h;   // token index x H + h of the next copy
    int64_t tok_fetch = bos;
    int ws = 0, rs = 0;
    auto fetch = [&]() {
        const bool in = tok_fetch < eos;
        const uint32_t dst = ring + ws * kGdnSlot;
        gdn_cp_async16(dst + qk_dst, qk_src + gi_fetch * kD, in);
        gdn_cp_async16(dst + x_dst, v_src + gi_fetch * kD, in && v_lane);
        gdn_cp_async4(dst + x_dst, gb_src + gi_fetch, in && gb_lane);
        asm volatile("cp.async.commit_group;\n" ::: "memory");
        ++tok_fetch;
        gi_fetch += H;
        ws = ws + 1 == kGdnRing ? 0 : ws + 1;
    };
#pragma unroll
    for (int i = 0; i < kGdnRing - 1; ++i) fetch();
    const int sl0 = cg + 8 * m, sl1 = cg + 8 * (m ^ 1), sl2 = cg + 8 * (m ^ 2), sl3 = cg + 8 * (m ^ 3);
    const unsigned char *ring_p = ring_all[warp][0];
    uint16_t *o_p = o + (static_cast<size_t>(bos) * H + h) * kD + col0 + m;
    const size_t o_step = static_cast<size_t>(H) * kD;
    for (int64_t tok = bos; tok < eos; ++tok) {
        // this token's copies have landed (each lane waits for its own, the warp then meets)
        asm volatile("cp.async.wait_group %0;\n" ::"n"(kGdnRing - 2) : "memory");
        __syncwarp();
        fetch();
        const unsigned char *cur = ring_p + rs * kGdnSlot;
        rs = rs + 1 == kGdnRing ? 0 : rs + 1;
        const uint4 *cq = reinterpret_cast<const uint4 *>(cur);
        float2 kp[8], qp[8];   // (k, q)[row0 + 2p], (k, q)[row0 + 2p + 1]
        gdn_unpack8(cq[16 + 2 * (lane >> 2)], kp);
        gdn_unpack8(cq[17 + 2 * (lane >> 2)], kp + 4);
        gdn_unpack8(cq[2 * (lane >> 2)], qp);
        gdn_unpack8(cq[1 + 2 * (lane >> 2)], qp + 4);
        const float vj = bf16_bits_to_float(reinterpret_cast<const uint16_t *>(cur + 512)[4 * cg + m]);
        const float bt = *reinterpret_cast<const float *>(cur + 548);
        c *= gdn_ex2(*reinterpret_cast<const float *>(cur + 544) * 1.4426950408889634f);
        if (!(c >= kGdnCLo && c <= kGdnCHi)) {   // fold c into S~ (also a zero or NaN gate)
            const float2 cc = make_float2(c, c);
#pragma unroll
            for (int p = 0; p < 8; ++p)
#pragma unroll
                for (int j = 0; j < 4; ++j) s[p][j] = __fmul2_rn(s[p][j], cc);
            c = 1.f;
        }
        // kv / c = k S~ over this lane's rows, then over all rows
        float2 a[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) a[j] = make_float2(0.f, 0.f);
#pragma unroll
        for (int p = 0; p < 8; ++p)
#pragma unroll
            for (int j = 0; j < 4; ++j) a[j] = __ffma2_rn(kp[p], s[p][j], a[j]);
        const float kvc = gdn_rows_sum(make_float4(a[0].x + a[0].y, a[1].x + a[1].y, a[2].x + a[2].y, a[3].x + a[3].y));
        // v_new / c = beta (v / c - kv / c) at this lane's column, then at its four slots'
        const float u = bt * (__fdividef(vj, c) - kvc);
        const float u0 = __shfl_sync(0xffffffffu, u, sl0), u1 = __shfl_sync(0xffffffffu, u, sl1);
        const float u2 = __shfl_sync(0xffffffffu, u, sl2), u3 = __shfl_sync(0xffffffffu, u, sl3);
        // S~ += k^T (v_new / c); q S~ over this lane's rows
        const float2 uu[4] = {make_float2(u0, u0), make_float2(u1, u1), make_float2(u2, u2), make_float2(u3, u3)};
        float2 b[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) b[j] = make_float2(0.f, 0.f);
#pragma unroll
        for (int p = 0; p < 8; ++p)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                s[p][j] = __ffma2_rn(kp[p], uu[j], s[p][j]);
                b[j] = __ffma2_rn(qp[p], s[p][j], b[j]);
            }
        const float oj = gdn_rows_sum(make_float4(b[0].x + b[0].y, b[1].x + b[1].y, b[2].x + b[2].y, b[3].x + b[3].y)) *
                         (scale * c);
        if (!(lane & 4)) *o_p = __bfloat16_as_ushort(__float2bfloat16_rn(oj));
        o_p += o_step;
    }
    if (hT) {
        float *dst = hT + static_cast<size_t>(nh) * kD * kD + col0;
#pragma unroll
        for (int p = 0; p < 8; ++p) {
            *reinterpret_cast<float4 *>(dst + (row0 + 2 * p) * kD) =
                gdn_perm(make_float4(s[p][0].x * c, s[p][1].x * c, s[p][2].x * c, s[p][3].x * c), m);
            *reinterpret_cast<float4 *>(dst + (row0 + 2 * p + 1) * kD) =
                gdn_perm(make_float4(s[p][0].y * c, s[p][1].y * c, s[p][2].y * c, s[p][3].y * c), m);
        }
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
