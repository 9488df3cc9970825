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

__device__ __forceinline__ float round_bf16_f(float x) {
    return __bfloat162float(__float2bfloat16_rn(x));
}

// One head vector (4 elements per lane): RMSNorm with weight w, bf16, RoPE with the lane's
// (cos, sin), bf16. The RoPE partner of lane l's elements is in lane l ^ 16.
__device__ __forceinline__ uint2 prologue_head(uint2 xw, const float (&wv)[4], const float (&cs)[4],
                                               const float (&sn)[4], float eps, bool low) {
    const float2 a01 = bf16x2_to_float2(xw.x), a23 = bf16x2_to_float2(xw.y);
    const float xs[4] = {a01.x, a01.y, a23.x, a23.y};
    float ss = xs[0] * xs[0] + xs[1] * xs[1] + xs[2] * xs[2] + xs[3] * xs[3];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float r = 1.f / sqrtf(ss / kD + eps);
    float out[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float y = round_bf16_f(xs[e] * r * wv[e]);
        const float py = __shfl_xor_sync(0xffffffffu, y, 16);
        out[e] = round_bf16_f(low ? y * cs[e] - py * sn[e] : y * cs[e] + py * sn[e]);
    }
    return make_uint2(float2_to_bf16x2(out[0], out[1]), float2_to_bf16x2(out[2], out[3]));
}

// One CTA per token: the token's position and the cos / sin of the 64 rotation angles are
// found once (into shared memory; lane l of every warp then holds those of elements
// 4l .. 4l + 3), and warp w rewrites heads w, w + 8, ... of q and k, loading a group of heads
// before working on it.
__global__ void __launch_bounds__(kProThreads)
qk_prologue_kernel(uint16_t *q, uint16_t *k, QkPrologue pro, SegTable t, const int64_t *start_pos,
                   int64_t T_total, int H) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t tok = blockIdx.x;
    const size_t row = static_cast<size_t>(tok) * H;
    // the first group of heads is loaded before anything else (its latency overlaps the
    // position lookup and the angles)
    uint2 xq[kProHeadsInFlight], xk[kProHeadsInFlight];
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
    // the token's position and the 64 angles' cos / sin, once per token (thread i < 64 takes
    // angle i; thread 0 finds the sequence: largest n with begin(n) <= tok)
    __shared__ float cs_s[64], sn_s[64];
    __shared__ float pos_s;
    if (threadIdx.x == 0) {
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
        pos_s = static_cast<float>(tok - seq_begin(t, n) + (start_pos ? start_pos[n] : 0));
    }
    __syncthreads();
    if (threadIdx.x < 64) sincosf(pos_s * pro.inv_freq[threadIdx.x], &sn_s[threadIdx.x], &cs_s[threadIdx.x]);
    float wq[4], wk[4];
    {
        const uint2 a = *reinterpret_cast<const uint2 *>(pro.qw + 4 * lane);
        const uint2 b = *reinterpret_cast<const uint2 *>(pro.kw + 4 * lane);
        const float2 a0 = bf16x2_to_float2(a.x), a1 = bf16x2_to_float2(a.y);
        const float2 b0 = bf16x2_to_float2(b.x), b1 = bf16x2_to_float2(b.y);
        wq[0] = a0.x; wq[1] = a0.y; wq[2] = a1.x; wq[3] = a1.y;
        wk[0] = b0.x; wk[1] = b0.y; wk[2] = b1.x; wk[3] = b1.y;
    }
    __syncthreads();
    float cs[4], sn[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        cs[e] = cs_s[(4 * lane + e) & 63];
        sn[e] = sn_s[(4 * lane + e) & 63];
    }
    const bool low = lane < 16;
    for (int h0 = warp; h0 < H; h0 += kProWarps * kProHeadsInFlight) {
        if (h0 != warp) load_group(h0);
#pragma unroll
        for (int j = 0; j < kProHeadsInFlight; ++j) {
            const int h = h0 + j * kProWarps;
            if (h < H) {
                const size_t off = (row + h) * kD + 4 * lane;
                *reinterpret_cast<uint2 *>(q + off) = prologue_head(xq[j], wq, cs, sn, pro.eps, low);
                *reinterpret_cast<uint2 *>(k + off) = prologue_head(xk[j], wk, cs, sn, pro.eps, low);
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
