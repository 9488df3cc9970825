// The q/k prologue of a lightning layer, in place on a prefill's q and k.
//
// "MiniCPM-SALA — Complete Blueprint", section "B2 lightning-attn (Simple GLA)": per head,
// q = RMSNorm(q, w = [128]) and k = RMSNorm(k, w = [128]) (the page's RMSNorm: x / sqrt(mean(x^2)
// + eps) times the weight), then q, k = RoPE(q.float(), k.float(), pos).bf16() with theta =
// 10000. The pairing is rotate-half: element i < 64 turns with element i + 64 by the angle
// pos * theta^(-i/64).
//
// One CTA per token, one warp per head at a time: lane l holds elements 4l .. 4l + 3 of q and
// of k (8-byte accesses, a whole 256-byte head vector per warp instruction), and the RoPE
// partner of lane l's elements sits in lane l ^ 16. The angles depend only on the token's
// position (its index in its sequence plus the sequence's start position), so their cos/sin
// are computed once per token. HBM-bound: 2 x 256 B read and written per (token, head); at
// that rate the SM's instruction issue is close to a limit too, so the arithmetic is kept
// lean: packed fp32 pairs (fma.rn.f32x2, rounding like the scalar forms), the sums of squares
// of a warp's four heads reduced together, one reciprocal square root per lane.
#include "launch.h"

#include <cmath>

namespace sala {

constexpr int kProThreads = 256;
constexpr int kProWarps = kProThreads / 32;
constexpr int kProHeadsInFlight = 4;   // heads per warp whose loads are issued together (warp_rms4)

// 1 / sqrt(x) for x >= eps > 0 (a mean of squares plus eps, always a normal number, so
// flushing subnormals changes nothing).
__device__ __forceinline__ float rms_rsqrt(float x) {
    float r;
    asm("rsqrt.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// Four sums of squares per lane (heads j = 0..3 of q, or of k) summed over the warp together:
// the xor-16 step keeps two of them (sending the other two to the partner lane) and the xor-8
// step one, so a lane then holds the partial of head 2 b4 + b3 (b4, b3: its lane bits 4 and
// 3), which xor 4, 2 and 1 complete. Each lane turns its total into 1 / rms, and the four
// factors are broadcast back from lanes 0, 8, 16 and 24.
__device__ __forceinline__ void warp_rms4(const float (&v)[4], float eps, float (&rn)[4]) {
    const int lane = threadIdx.x & 31;
    const bool b4 = lane & 16, b3 = lane & 8;
    float w[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const float send = b4 ? v[i] : v[i + 2], keep = b4 ? v[i + 2] : v[i];
        w[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
    }
    float t = (b3 ? w[1] : w[0]) + __shfl_xor_sync(0xffffffffu, b3 ? w[0] : w[1], 8);
    t += __shfl_xor_sync(0xffffffffu, t, 4);
    t += __shfl_xor_sync(0xffffffffu, t, 2);
    t += __shfl_xor_sync(0xffffffffu, t, 1);
    const float r = rms_rsqrt(fmaf(t, 1.f / kD, eps));
#pragma unroll
    for (int j = 0; j < 4; ++j) rn[j] = __shfl_sync(0xffffffffu, r, 16 * (j >> 1) + 8 * (j & 1));
}

// This lane's part of a head vector's sum of squares (its 4 elements).
__device__ __forceinline__ float sumsq4(uint2 xw) {
    const float2 a01 = bf16x2_to_float2(xw.x), a23 = bf16x2_to_float2(xw.y);
    const float2 s2 = __ffma2_rn(a23, a23, __fmul2_rn(a01, a01));
    return s2.x + s2.y;
}

// RMSNorm's output for the lane's 4 elements: x / rms * w, rounded to bf16 two to a word.
__device__ __forceinline__ uint2 scale4(uint2 xw, float r, const float2 (&wv)[2]) {
    const float2 r2 = make_float2(r, r);
    const float2 t0 = __fmul2_rn(__fmul2_rn(bf16x2_to_float2(xw.x), r2), wv[0]);
    const float2 t1 = __fmul2_rn(__fmul2_rn(bf16x2_to_float2(xw.y), r2), wv[1]);
    return make_uint2(float2_to_bf16x2(t0.x, t0.y), float2_to_bf16x2(t1.x, t1.y));
}

// RoPE with the lane's (cos, sin) pairs, bf16. The partners (lane l ^ 16) are exchanged in
// the packed form; ssn is -sin for the first half of the vector (lanes 0-15) and +sin for the
// second.
__device__ __forceinline__ uint2 prologue_rope(uint2 y, const float2 (&cs)[2], const float2 (&ssn)[2]) {
    const uint32_t p01 = __shfl_xor_sync(0xffffffffu, y.x, 16);
    const uint32_t p23 = __shfl_xor_sync(0xffffffffu, y.y, 16);
    const float2 u0 = __ffma2_rn(bf16x2_to_float2(p01), ssn[0], __fmul2_rn(bf16x2_to_float2(y.x), cs[0]));
    const float2 u1 = __ffma2_rn(bf16x2_to_float2(p23), ssn[1], __fmul2_rn(bf16x2_to_float2(y.y), cs[1]));
    return make_uint2(float2_to_bf16x2(u0.x, u0.y), float2_to_bf16x2(u1.x, u1.y));
}

// One CTA per token: the cos / sin of the 64 rotation angles are found once (into shared
// memory; lane l of every warp then holds those of elements 4l .. 4l + 3), and warp w rewrites
// heads w, w + 8, ... of q and k, loading a group of heads before working on it. The first
// group's normalisation runs while the angles are computed; one barrier separates the two.
__global__ void __launch_bounds__(kProThreads, 5)
qk_prologue_kernel(uint16_t *q, uint16_t *k, QkPrologue pro, SegTable t, const int64_t *start_pos,
                   int64_t T_total, int H, int *status) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t tok = blockIdx.x;
    const size_t row = static_cast<size_t>(tok) * H;
    dependent_start();   // (launched by launch_dependent)
    // the first group of heads is loaded before anything else (its latency overlaps the
    // position lookup and the angles)
    uint2 xq[kProHeadsInFlight], xk[kProHeadsInFlight];
#pragma unroll
    for (int j = 0; j < kProHeadsInFlight; ++j) xq[j] = xk[j] = make_uint2(0u, 0u);
    auto load_group = [&](int h0) {
#pragma unroll
        for (int j = 0; j < kProHeadsInFlight; ++j) {
            const int h = h0 + j * kProWarps;
            if (h < H) {
                const size_t off = (row + h) * kD + 4 * lane;
                xq[j] = *reinterpret_cast<const uint2 *>(q + off);
                xk[j] = *reinterpret_cast<const uint2 *>(k + off);
            }
        }
    };
    load_group(warp);
    // the 64 angles' cos / sin of the token's position, once per token: thread i < 64 takes
    // angle i and finds the position itself (the sequence: largest n with begin(n) <= tok), so
    // the angles need no barrier of their own and overlap the first group's normalisation
    __shared__ float cs_s[64], sn_s[64];
    __shared__ bool skip_s;
    if (threadIdx.x < 64) {
        int64_t n = 0;
        if (t.cu) {
            int64_t lo = 0, hi = t.nseq - 1;
            while (lo < hi) {
                const int64_t mid = (lo + hi + 1) >> 1;
                if (t.cu[mid] <= tok) lo = mid; else hi = mid - 1;
            }
            n = lo;
        } else {
            n = tok / t.T_row;
        }
        const float pos = static_cast<float>(tok - seq_begin(t, n) + (start_pos ? start_pos[n] : 0));
        sincosf(pos * pro.inv_freq[threadIdx.x], &sn_s[threadIdx.x], &cs_s[threadIdx.x]);
        // debug build: the token lies in the sequence found (cu_seqlens is not validated here)
        if (threadIdx.x == 0)
            skip_s = !dcheck(seq_begin(t, n) <= tok && tok < seq_begin(t, n + 1), status);
    }
    float2 wq[2], wk[2];
    {
        const uint2 a = *reinterpret_cast<const uint2 *>(pro.qw + 4 * lane);
        const uint2 b = *reinterpret_cast<const uint2 *>(pro.kw + 4 * lane);
        wq[0] = bf16x2_to_float2(a.x); wq[1] = bf16x2_to_float2(a.y);
        wk[0] = bf16x2_to_float2(b.x); wk[1] = bf16x2_to_float2(b.y);
    }
    static_assert(kProHeadsInFlight == 4, "warp_rms4 reduces four heads at a time");
    // (heads past H: zero or stale values, normalised but never stored)
    auto norm_group = [&]() {
#pragma unroll
        for (int side = 0; side < 2; ++side) {
            uint2 (&xs)[kProHeadsInFlight] = side ? xk : xq;
            float v[4], rn[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) v[j] = sumsq4(xs[j]);
            warp_rms4(v, pro.eps, rn);
#pragma unroll
            for (int j = 0; j < 4; ++j) xs[j] = scale4(xs[j], rn[j], side ? wk : wq);
        }
    };
    norm_group();
    __syncthreads();
    if (skip_s) return;   // (only ever set in the debug build)
    float2 cs[2], ssn[2];
    {
        const int a = (4 * lane) & 63;
        const float sg = lane < 16 ? -1.f : 1.f;
        cs[0] = make_float2(cs_s[a], cs_s[a + 1]);
        cs[1] = make_float2(cs_s[a + 2], cs_s[a + 3]);
        ssn[0] = make_float2(sg * sn_s[a], sg * sn_s[a + 1]);
        ssn[1] = make_float2(sg * sn_s[a + 2], sg * sn_s[a + 3]);
    }
    for (int h0 = warp; h0 < H; h0 += kProWarps * kProHeadsInFlight) {
        if (h0 != warp) {
            load_group(h0);
            norm_group();
        }
#pragma unroll
        for (int j = 0; j < kProHeadsInFlight; ++j) {
            const int h = h0 + j * kProWarps;
            if (h < H) {
                const size_t off = (row + h) * kD + 4 * lane;
                *reinterpret_cast<uint2 *>(q + off) = prologue_rope(xq[j], cs, ssn);
                *reinterpret_cast<uint2 *>(k + off) = prologue_rope(xk[j], cs, ssn);
            }
        }
    }
}

QkPrologue make_qk_prologue(const sala_qk_prologue *p, const int64_t *positions) {
    QkPrologue r;
    if (!p) return r;
    r.qw = static_cast<const uint16_t *>(p->q_weight);
    r.kw = static_cast<const uint16_t *>(p->k_weight);
    r.pos = positions;
    r.eps = p->eps;
    for (int i = 0; i < 64; ++i)
        r.inv_freq[i] = static_cast<float>(std::pow(static_cast<double>(p->rope_theta), -i / 64.0));
    return r;
}

cudaError_t launch_qk_prologue(void *q, void *k, const QkPrologue &pro, const SegTable &t,
                               const int64_t *start_pos, int64_t T_total, int H, int *status,
                               cudaStream_t stream) {
    if (T_total == 0) return cudaSuccess;
    LaunchTimer timer(kKQkPrologue, stream);
    return launch_dependent(qk_prologue_kernel, static_cast<unsigned>(T_total), kProThreads, stream,
                            static_cast<uint16_t *>(q), static_cast<uint16_t *>(k), pro, t, start_pos,
                            T_total, H, status);
}

}  // namespace sala
