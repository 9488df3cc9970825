// The q/k prologue of a lightning layer, in place on a prefill's q and k.
//
// "MiniCPM-SALA — Complete Blueprint", section "B2 lightning-attn (Simple GLA)": per head,
// q = RMSNorm(q, w = [128]) and k = RMSNorm(k, w = [128]) (the page's RMSNorm: x / sqrt(mean(x^2)
// + eps) times the weight), then q, k = RoPE(q.float(), k.float(), pos).bf16() with theta =
// 10000. The pairing is rotate-half: element i < 64 turns with element i + 64 by the angle
// pos * theta^(-i/64).
//
// One warp per (token, head): lane l holds elements 4l .. 4l + 3 of q and of k (8-byte
// accesses, a whole 256-byte head vector per warp instruction), the sum of squares is a warp
// reduction, and the RoPE partner of lane l's elements sits in lane l ^ 16. A token's
// position is its index in its sequence plus the sequence's start position. HBM-bound:
// 2 x 256 B read and written per (token, head).
#include "launch.h"

#include <cmath>

namespace sala {

constexpr int kProThreads = 256;

__device__ __forceinline__ float round_bf16_f(float x) {
    return __bfloat162float(__float2bfloat16_rn(x));
}

__global__ void __launch_bounds__(kProThreads)
qk_prologue_kernel(uint16_t *q, uint16_t *k, QkPrologue pro, SegTable t, const int64_t *start_pos,
                   int64_t T_total, int H) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t pair = static_cast<int64_t>(blockIdx.x) * (kProThreads / 32) + warp;
    if (pair >= T_total * H) return;
    const int64_t tok = pair / H;
    // the token's sequence: largest n with begin(n) <= tok
    int64_t n = 0;
    if (lane == 0) {
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
    }
    n = __shfl_sync(0xffffffffu, n, 0);
    const int64_t pos = tok - seq_begin(t, n) + (start_pos ? start_pos[n] : 0);
    const float ang_pos = static_cast<float>(pos);
    const size_t off = static_cast<size_t>(pair) * kD + 4 * lane;
    const uint2 wq = *reinterpret_cast<const uint2 *>(pro.qw + 4 * lane);
    const uint2 wk = *reinterpret_cast<const uint2 *>(pro.kw + 4 * lane);
#pragma unroll
    for (int which = 0; which < 2; ++which) {
        uint16_t *x = which ? k : q;
        const uint2 ww = which ? wk : wq;
        const uint2 xw = *reinterpret_cast<const uint2 *>(x + off);
        const float2 a01 = bf16x2_to_float2(xw.x), a23 = bf16x2_to_float2(xw.y);
        const float w01x = bf16x2_to_float2(ww.x).x, w01y = bf16x2_to_float2(ww.x).y;
        const float w23x = bf16x2_to_float2(ww.y).x, w23y = bf16x2_to_float2(ww.y).y;
        const float xs[4] = {a01.x, a01.y, a23.x, a23.y}, wv[4] = {w01x, w01y, w23x, w23y};
        float ss = xs[0] * xs[0] + xs[1] * xs[1] + xs[2] * xs[2] + xs[3] * xs[3];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        const float r = 1.f / sqrtf(ss / kD + pro.eps);
        float y[4], out[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) y[e] = round_bf16_f(xs[e] * r * wv[e]);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float py = __shfl_xor_sync(0xffffffffu, y[e], 16);
            const int i = 4 * lane + e;
            float sn, cs;
            sincosf(ang_pos * pro.inv_freq[i & 63], &sn, &cs);
            out[e] = round_bf16_f(lane < 16 ? y[e] * cs - py * sn : y[e] * cs + py * sn);
        }
        *reinterpret_cast<uint2 *>(x + off) =
            make_uint2(float2_to_bf16x2(out[0], out[1]), float2_to_bf16x2(out[2], out[3]));
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
    const int64_t pairs = T_total * H;
    const int64_t blocks = (pairs + kProThreads / 32 - 1) / (kProThreads / 32);
    qk_prologue_kernel<<<static_cast<unsigned>(blocks), kProThreads, 0, stream>>>(
        static_cast<uint16_t *>(q), static_cast<uint16_t *>(k), pro, t, start_pos, T_total, H);
    return cudaGetLastError();
}

}  // namespace sala
