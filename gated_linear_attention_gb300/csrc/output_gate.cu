// Output norm and gate of a lightning layer: per token, out = RMSNorm(o) * w * sigmoid(z).
//
// "MiniCPM-SALA — Complete Blueprint", section "B2 lightning-attn (Simple GLA)", block
// "Output Norm + Gate + Projection": the attention output of all 32 heads of a token
// (4096 features) is RMS-normalised with a weight vector (o_norm; RMSNorm as the page's
// input_layernorm block defines it: rms = sqrt(mean(x^2) + 1e-6), x / rms * weight), then
// multiplied element-wise by the gate sigmoid(h W_z^T). The gate logits z = h W_z^T come from
// the caller (the projection needs trained weights).
//
// One CTA of 128 threads per token. The normalisation needs every feature of the token, so
// the pass is: load o (thread t holds 8 consecutive features of each 1024-feature block, so
// each warp instruction moves 512 contiguous bytes), sum of squares reduced over the CTA,
// then z and the weight, and the product is stored. (H = 8, 16, 32, 64 take a variant with
// o and z loaded up front; other widths the general kernel below.) HBM-bound: 3 x 2 bytes per feature
// (o, z read, out written) plus the weight, which stays in L2.
#include "launch.h"

namespace sala {

constexpr int kGateThreads = 128;
constexpr int kGateRegIt = 8;   // features kept in registers: up to 8 x 1024 (H <= 64)

__global__ void __launch_bounds__(kGateThreads)
output_norm_gate_kernel(const uint16_t *__restrict__ o, const uint16_t *__restrict__ z,
                        const uint16_t *__restrict__ w, float eps, uint16_t *out, int F) {
    const size_t tok = static_cast<size_t>(blockIdx.x) * F;
    const int nit = (F + 8 * kGateThreads - 1) / (8 * kGateThreads);
    uint4 ov[kGateRegIt];
    float ss = 0.f;
#pragma unroll
    for (int m = 0; m < kGateRegIt; ++m) {
        const int e = 8 * (threadIdx.x + kGateThreads * m);
        ov[m] = make_uint4(0u, 0u, 0u, 0u);
        if (m < nit && e < F) ov[m] = __ldcs(reinterpret_cast<const uint4 *>(o + tok + e));
    }
    for (int m = kGateRegIt; m < nit; ++m) {   // wider tokens: sum the rest from memory
        const int e = 8 * (threadIdx.x + kGateThreads * m);
        if (e < F) {
            const uint4 x = __ldcg(reinterpret_cast<const uint4 *>(o + tok + e));
            const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 f = bf16x2_to_float2(xs[i]);
                ss = fmaf(f.x, f.x, fmaf(f.y, f.y, ss));
            }
        }
    }
#pragma unroll
    for (int m = 0; m < kGateRegIt; ++m) {
        const uint32_t xs[4] = {ov[m].x, ov[m].y, ov[m].z, ov[m].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = bf16x2_to_float2(xs[i]);
            ss = fmaf(f.x, f.x, fmaf(f.y, f.y, ss));
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    __shared__ float part[kGateThreads / 32];
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int i = 0; i < kGateThreads / 32; ++i) tot += part[i];
    const float rinv = 1.f / sqrtf(tot / static_cast<float>(F) + eps);

    auto emit = [&](const uint4 x, int e) {
        const uint4 zz = __ldcs(reinterpret_cast<const uint4 *>(z + tok + e));
        const uint4 ww = __ldg(reinterpret_cast<const uint4 *>(w + e));
        const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, zs[4] = {zz.x, zz.y, zz.z, zz.w},
                       ws[4] = {ww.x, ww.y, ww.z, ww.w};
        uint32_t r[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 xf = bf16x2_to_float2(xs[i]), zf = bf16x2_to_float2(zs[i]),
                         wf = bf16x2_to_float2(ws[i]);
            const float g0 = __fdividef(1.f, 1.f + __expf(-zf.x)), g1 = __fdividef(1.f, 1.f + __expf(-zf.y));
            r[i] = float2_to_bf16x2(xf.x * rinv * wf.x * g0, xf.y * rinv * wf.y * g1);
        }
        __stcs(reinterpret_cast<uint4 *>(out + tok + e), make_uint4(r[0], r[1], r[2], r[3]));
    };
#pragma unroll
    for (int m = 0; m < kGateRegIt; ++m) {
        const int e = 8 * (threadIdx.x + kGateThreads * m);
        if (m < nit && e < F) emit(ov[m], e);
    }
    for (int m = kGateRegIt; m < nit; ++m) {
        const int e = 8 * (threadIdx.x + kGateThreads * m);
        if (e < F) emit(__ldcg(reinterpret_cast<const uint4 *>(o + tok + e)), e);
    }
}

// The common widths (H = 8, 16, 32, 64: F = 8 kIt kThr features): o and z of the token are
// loaded up front (kIt 16-byte pieces each per thread of kThr), so each CTA has its whole
// token in flight at once, with up to 1536 threads resident per SM; the weight (an L2 hit) is
// read after the reduction, which keeps the registers within that budget. The arithmetic
// runs on packed fp32 pairs (fma.rn.f32x2 / mul.rn.f32x2, rounding like the scalar forms):
// at this rate the SM's instruction issue is close to a limit as well.
template <int kIt, int kThr>
__global__ void __launch_bounds__(kThr, 1536 / kThr)
output_norm_gate_fixed_kernel(const uint16_t *__restrict__ o, const uint16_t *__restrict__ z,
                              const uint16_t *__restrict__ w, float eps, uint16_t *out) {
    constexpr int F = kIt * 8 * kThr;
    const size_t tok = static_cast<size_t>(blockIdx.x) * F;
    dependent_start();   // (launched by launch_dependent)
    uint4 ov[kIt], zv[kIt];
#pragma unroll
    for (int m = 0; m < kIt; ++m) {
        const int e = 8 * (threadIdx.x + kThr * m);
        ov[m] = __ldcs(reinterpret_cast<const uint4 *>(o + tok + e));
        zv[m] = __ldcs(reinterpret_cast<const uint4 *>(z + tok + e));
    }
    float2 s2 = make_float2(0.f, 0.f);
#pragma unroll
    for (int m = 0; m < kIt; ++m) {
        const uint32_t xs[4] = {ov[m].x, ov[m].y, ov[m].z, ov[m].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = bf16x2_to_float2(xs[i]);
            s2 = __ffma2_rn(f, f, s2);
        }
    }
    float ss = s2.x + s2.y;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    __shared__ float part[kThr / 32];
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int i = 0; i < kThr / 32; ++i) tot += part[i];
    const float rinv = 1.f / sqrtf(tot / static_cast<float>(F) + eps);
    const float2 r2 = make_float2(rinv, rinv);
#pragma unroll
    for (int m = 0; m < kIt; ++m) {
        const int e = 8 * (threadIdx.x + kThr * m);
        const uint4 wv = __ldg(reinterpret_cast<const uint4 *>(w + e));
        const uint32_t xs[4] = {ov[m].x, ov[m].y, ov[m].z, ov[m].w},
                       zs[4] = {zv[m].x, zv[m].y, zv[m].z, zv[m].w},
                       ws[4] = {wv.x, wv.y, wv.z, wv.w};
        uint32_t r[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 xf = bf16x2_to_float2(xs[i]), zf = bf16x2_to_float2(zs[i]),
                         wf = bf16x2_to_float2(ws[i]);
            const float2 g = make_float2(__fdividef(1.f, 1.f + __expf(-zf.x)),
                                         __fdividef(1.f, 1.f + __expf(-zf.y)));
            const float2 t = __fmul2_rn(__fmul2_rn(__fmul2_rn(xf, r2), wf), g);
            r[i] = float2_to_bf16x2(t.x, t.y);
        }
        __stcs(reinterpret_cast<uint4 *>(out + tok + e), make_uint4(r[0], r[1], r[2], r[3]));
    }
}

cudaError_t launch_output_norm_gate(const void *o, const void *z, const void *w, float eps,
                                    void *out, int64_t T, int H, cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    LaunchTimer timer(kKOutputNormGate, stream);
    const auto *ob = static_cast<const uint16_t *>(o), *zb = static_cast<const uint16_t *>(z),
               *wb = static_cast<const uint16_t *>(w);
    auto *outb = static_cast<uint16_t *>(out);
    const unsigned grid = static_cast<unsigned>(T);
    // the fixed-width kernels go out as programmatic dependents of the work before them
    switch (H) {
    case 8: return launch_dependent(output_norm_gate_fixed_kernel<1, 128>, grid, 128, stream, ob, zb, wb, eps, outb);
    case 16: return launch_dependent(output_norm_gate_fixed_kernel<1, 256>, grid, 256, stream, ob, zb, wb, eps, outb);
    case 32: return launch_dependent(output_norm_gate_fixed_kernel<2, 256>, grid, 256, stream, ob, zb, wb, eps, outb);
    case 64: return launch_dependent(output_norm_gate_fixed_kernel<2, 512>, grid, 512, stream, ob, zb, wb, eps, outb);
    default:
        output_norm_gate_kernel<<<grid, kGateThreads, 0, stream>>>(ob, zb, wb, eps, outb, H * kD);
    }
    return cudaGetLastError();
}

}  // namespace sala
