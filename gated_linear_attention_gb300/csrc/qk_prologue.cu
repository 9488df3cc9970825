// The q/k prologue of a lightning layer, in place on a prefill's q and k.
//
// "MiniCPM-SALA — Complete Blueprint", section "B2 lightning-attn (Simple GLA)": per head,
// q = RMSNorm(q, w = [128]) and k = RMSNorm(k, w = [128]) (the page's RMSNorm: x / sqrt(mean(x^2)
// + eps) times the weight), then q, k = RoPE(q.float(), k.float(), pos).bf16() with theta =
// 10000. The pairing is rotate-half: element i < 64 turns with element i + 64 by the angle
// pos * theta^(-i/64).
//
// One CTA per token, one warp per head at a time: lane l holds elements 4l .. 4l + 3 of q and
// of k (8-byte accesses, a whole 256-byte head vector per warp instruction), the sum of
// squares is a warp reduction, and the RoPE partner of lane l's elements sits in lane l ^ 16.
// The angles depend only on the token's position (its index in its sequence plus the
// sequence's start position), so their cos/sin are computed once per token. HBM-bound:
// 2 x 256 B read and written per (token, head).
#include "launch.h"

#include <cmath>

namespace sala {

constexpr int kProThreads = 256;
constexpr int kProWarps = kProThreads / 32;
constexpr int kProHeadsInFlight = 4;   // heads per warp whose loads are issued together

// One head vector (4 elements per lane), first stage: RMSNorm with weight w, the results
// rounded to bf16 two to a word.
__device__ __forceinline__ uint2 prologue_norm(uint2 xw, const float (&wv)[4], float eps) {
    const float2 a01 = bf16x2_to_float2(xw.x), a23 = bf16x2_to_float2(xw.y);
    float ss = a01.x * a01.x;
    ss = fmaf(a01.y, a01.y, ss);
    ss = fmaf(a23.x, a23.x, ss);
    ss = fmaf(a23.y, a23.y, ss);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float r = rsqrtf(ss * (1.f / kD) + eps);
    return make_uint2(float2_to_bf16x2(a01.x * r * wv[0], a01.y * r * wv[1]),
                      float2_to_bf16x2(a23.x * r * wv[2], a23.y * r * wv[3]));
}

// Second stage: RoPE with the lane's (cos, sin), bf16. The partners (lane l ^ 16) are
// exchanged in the packed form; ssn is -sin for the first half of the vector (lanes 0-15) and
// +sin for the second.
__device__ __forceinline__ uint2 prologue_rope(uint2 y, const float (&cs)[4], const float (&ssn)[4]) {
    const uint32_t p01 = __shfl_xor_sync(0xffffffffu, y.x, 16);
    const uint32_t p23 = __shfl_xor_sync(0xffffffffu, y.y, 16);
    const float2 y0 = bf16x2_to_float2(y.x), y1 = bf16x2_to_float2(y.y);
    const float2 q0 = bf16x2_to_float2(p01), q1 = bf16x2_to_float2(p23);
    return make_uint2(float2_to_bf16x2(fmaf(q0.x, ssn[0], y0.x * cs[0]), fmaf(q0.y, ssn[1], y0.y * cs[1])),
                      float2_to_bf16x2(fmaf(q1.x, ssn[2], y1.x * cs[2]), fmaf(q1.y, ssn[3], y1.y * cs[3])));
}

// One CTA per token: the cos / sin of the 64 rotation angles are found once (into shared
// memory; lane l of every warp then holds those of elements 4l .. 4l + 3), and warp w rewrites
// heads w, w + 8, ... of q and k, loading a group of heads before working on it. The first
// group's normalisation runs while the angles are computed; one barrier separates the two.
__global__ void __launch_bounds__(kProThreads, 5)
qk_prologue_kernel(uint16_t *q, uint16_t *k, QkPrologue pro, SegTable t, const int64_t *start_pos,
                   int64_t T_total, int H) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t tok = blockIdx.x;
    const size_t row = static_cast<size_t>(tok) * H;
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
    }
    float wq[4], wk[4];
    {
        const uint2 a = *reinterpret_cast<const uint2 *>(pro.qw + 4 * lane);
        const uint2 b = *reinterpret_cast<const uint2 *>(pro.kw + 4 * lane);
        const float2 a0 = bf16x2_to_float2(a.x), a1 = bf16x2_to_float2(a.y);
        const float2 b0 = bf16x2_to_float2(b.x), b1 = bf16x2_to_float2(b.y);
        wq[0] = a0.x; wq[1] = a0.y; wq[2] = a1.x; wq[3] = a1.y;
        wk[0] = b0.x; wk[1] = b0.y; wk[2] = b1.x; wk[3] = b1.y;
    }
    auto norm_group = [&]() {
#pragma unroll
        for (int j = 0; j < kProHeadsInFlight; ++j) {
            xq[j] = prologue_norm(xq[j], wq, pro.eps);   // (heads past H: unused lanes' values)
            xk[j] = prologue_norm(xk[j], wk, pro.eps);
        }
    };
    norm_group();
    __syncthreads();
    float cs[4], ssn[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        cs[e] = cs_s[(4 * lane + e) & 63];
        ssn[e] = lane < 16 ? -sn_s[(4 * lane + e) & 63] : sn_s[(4 * lane + e) & 63];
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
                               const int64_t *start_pos, int64_t T_total, int H,
                               cudaStream_t stream) {
    if (T_total == 0) return cudaSuccess;
    LaunchTimer timer(kKQkPrologue, stream);
    qk_prologue_kernel<<<static_cast<unsigned>(T_total), kProThreads, 0, stream>>>(
        static_cast<uint16_t *>(q), static_cast<uint16_t *>(k), pro, t, start_pos, T_total, H);
    return cudaGetLastError();
}

}  // namespace sala
