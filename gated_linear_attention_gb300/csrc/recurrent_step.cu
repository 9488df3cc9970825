// One-token recurrent decode of Simple GLA, state updated in place.
//
// "MiniCPM-SALA — Complete Blueprint", section "B2 lightning-attn (Simple GLA)", block
// "Simple GLA Recurrence": per head, alpha = exp(g); S = alpha S; S += k^T (outer) v;
// o = q S x scale; the updated state is saved back to where it was loaded from. The page
// notes that the state read and write is the whole cost of this step ("Per-Token Decode
// Bandwidth": GLA recurrence = state R/W), so the kernel is a single streaming pass over
// the fp32 state: every byte of S is loaded once and stored once.
//
// The same kernel serves a state pool addressed through per-sequence slot indices, with the
// states stored in fp32 or bf16 (the Blueprint's "Memory Architecture": per-request temporal
// states in a pool, 1 MB each in bf16 for 32 heads); bf16 storage halves the bytes moved.
//
// Work split: one CTA of 256 threads (8 warps) per (sequence, head) unit. Warp w owns state
// rows [16w, 16w + 16); lane l owns columns [4l, 4l + 4), so each warp instruction moves
// one whole 512-byte row with 128-bit accesses. All 16 row loads of a thread are issued
// before any arithmetic (64 KB in flight per CTA), with the streaming cache hint since the
// state is touched exactly once per step. The q S reduction over rows is split: each thread
// accumulates its 16 rows, then the 8 warp partials are summed through shared memory.
#include "launch.h"

namespace sala {

constexpr int kDecodeThreads = 256;
constexpr int kRowsPerWarp = kD / (kDecodeThreads / 32);  // 16

// Where one unit's state lives and how it is stored: a dense [N, H, 128, 128] fp32 array
// (unit n * H + h at offset unit * 128 * 128), or a pool [P, H, 128, 128] of fp32 or bf16
// addressed through the slot index of the unit's sequence.
struct StateRef {
    void *base;
    const int32_t *idx;   // null: dense
    int64_t P;
    int H;
};

// One CTA per (sequence, head): the state S [128 x 128] is streamed in once, updated and
// streamed back out. fp32 storage: warp w owns rows [16w, 16w + 16) and lane l the 4 columns
// [4l, 4l + 4) of each (one 512-byte row per warp instruction). bf16 storage: the same rows,
// two per warp instruction, lane l holding the 8 columns [8 (l % 16), + 8) of row
// 2i + l / 16 (16-byte accesses, 512 bytes per warp instruction as well).
__device__ __forceinline__ float round_bf16f(float x) {
    return __bfloat162float(__float2bfloat16_rn(x));
}

// The q/k prologue on the token's q and k held in shared memory (element i by thread i < 128):
// per-head RMSNorm with its weight, rounded to bf16, then RoPE (rotate-half pairs (i, i + 64),
// angle float(pos) * inv_freq[i % 64] in fp32), rounded to bf16. Called by the whole CTA.
__device__ __forceinline__ void qk_prologue_smem(float *q_s, float *k_s, const QkPrologue &pro,
                                                 int64_t pos) {
    __shared__ float pss[2][kD / 32];
    const int i = threadIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float xq = 0.f, xk = 0.f;
    if (i < kD) {
        xq = q_s[i];
        xk = k_s[i];
    }
    float sq = xq * xq, sk = xk * xk;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        sq += __shfl_xor_sync(0xffffffffu, sq, off);
        sk += __shfl_xor_sync(0xffffffffu, sk, off);
    }
    if (lane == 0 && warp < kD / 32) {
        pss[0][warp] = sq;
        pss[1][warp] = sk;
    }
    __syncthreads();
    float yq = 0.f, yk = 0.f;
    if (i < kD) {
        const float rq = 1.f / sqrtf((pss[0][0] + pss[0][1] + pss[0][2] + pss[0][3]) / kD + pro.eps);
        const float rk = 1.f / sqrtf((pss[1][0] + pss[1][1] + pss[1][2] + pss[1][3]) / kD + pro.eps);
        yq = round_bf16f(xq * rq * bf16_bits_to_float(pro.qw[i]));
        yk = round_bf16f(xk * rk * bf16_bits_to_float(pro.kw[i]));
        q_s[i] = yq;
        k_s[i] = yk;
    }
    __syncthreads();
    float oq = 0.f, ok = 0.f;
    if (i < kD) {
        const float a = static_cast<float>(pos) * pro.inv_freq[i & 63];
        float sn, cs;
        sincosf(a, &sn, &cs);
        const float pq = q_s[i ^ 64], pk = k_s[i ^ 64];
        oq = round_bf16f(i < 64 ? yq * cs - pq * sn : yq * cs + pq * sn);
        ok = round_bf16f(i < 64 ? yk * cs - pk * sn : yk * cs + pk * sn);
    }
    __syncthreads();
    if (i < kD) {
        q_s[i] = oq;
        k_s[i] = ok;
    }
}

template <bool kBf16>
__global__ void __launch_bounds__(kDecodeThreads)
recurrent_step_kernel(const uint16_t *__restrict__ q, const uint16_t *__restrict__ k,
                      const uint16_t *__restrict__ v, const float *__restrict__ g, float scale,
                      StateRef ref, uint16_t *__restrict__ o, int *status, QkPrologue pro) {
    dependent_start();   // (launched by launch_dependent: one decode step after another)
    const int unit = blockIdx.x;  // n * H + h
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t vec = static_cast<size_t>(unit) * kD;
    size_t slot_unit = unit;
    if (ref.idx) {
        const int n = unit / ref.H, h = unit - n * ref.H;
        const int32_t slot = __ldg(ref.idx + n);
        if (slot < 0 || slot >= ref.P) {
            // padding row (or a slot past the pool, reported): o = 0, no state touched
            if (slot >= ref.P && h == 0 && threadIdx.x == 0) record_status(status, SALA_ERR_BAD_INDEX);
            if (threadIdx.x < kD / 2) reinterpret_cast<uint32_t *>(o + vec)[threadIdx.x] = 0u;
            return;
        }
        slot_unit = static_cast<size_t>(slot) * ref.H + h;
    }
    const int row0 = warp * kRowsPerWarp;
    __shared__ float q_s[kD], k_s[kD];
    __shared__ float part[kDecodeThreads / 32][kD];

    if constexpr (kBf16) {
        uint16_t *Su = static_cast<uint16_t *>(ref.base) + slot_unit * kD * kD;
        const int half = lane >> 4, c0 = 8 * (lane & 15);
        // 1. stream the state rows in (8 x 16 bytes per thread)
        uint4 s[kRowsPerWarp / 2];
#pragma unroll
        for (int i = 0; i < kRowsPerWarp / 2; ++i)
            s[i] = __ldcs(reinterpret_cast<const uint4 *>(Su + (row0 + 2 * i + half) * kD + c0));
        // 2. q, k (rows) and v (my 8 columns)
        if (threadIdx.x < kD) {
            q_s[threadIdx.x] = bf16_bits_to_float(q[vec + threadIdx.x]);
            k_s[threadIdx.x] = bf16_bits_to_float(k[vec + threadIdx.x]);
        }
        const uint4 vw = *reinterpret_cast<const uint4 *>(v + vec + c0);
        float vf[8];
        {
            const uint32_t w4[4] = {vw.x, vw.y, vw.z, vw.w};
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const float2 f = bf16x2_to_float2(w4[m]);
                vf[2 * m] = f.x;
                vf[2 * m + 1] = f.y;
            }
        }
        const float alpha = expf(g[unit]);
        if (pro.qw) qk_prologue_smem(q_s, k_s, pro, pro.pos[unit / ref.H]);
        __syncthreads();
        // 3. decay + rank-1 update, store back rounded to bf16, q S from the unrounded values
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < kRowsPerWarp / 2; ++i) {
            const int r = row0 + 2 * i + half;
            const float ki = k_s[r], qi = q_s[r];
            const uint32_t w4[4] = {s[i].x, s[i].y, s[i].z, s[i].w};
            uint32_t out[4];
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const float2 f = bf16x2_to_float2(w4[m]);
                const float x0 = fmaf(alpha, f.x, ki * vf[2 * m]);
                const float x1 = fmaf(alpha, f.y, ki * vf[2 * m + 1]);
                acc[2 * m] = fmaf(qi, x0, acc[2 * m]);
                acc[2 * m + 1] = fmaf(qi, x1, acc[2 * m + 1]);
                out[m] = float2_to_bf16x2(x0, x1);
            }
            __stcs(reinterpret_cast<uint4 *>(Su + r * kD + c0), make_uint4(out[0], out[1], out[2], out[3]));
        }
        // the two half-warps hold the even and odd rows of the same columns
#pragma unroll
        for (int m = 0; m < 8; ++m) acc[m] += __shfl_xor_sync(0xffffffffu, acc[m], 16);
        if (half == 0) {
            *reinterpret_cast<float4 *>(&part[warp][c0]) = make_float4(acc[0], acc[1], acc[2], acc[3]);
            *reinterpret_cast<float4 *>(&part[warp][c0 + 4]) = make_float4(acc[4], acc[5], acc[6], acc[7]);
        }
    } else {
        float *Su = static_cast<float *>(ref.base) + slot_unit * kD * kD;
        // 1. stream the state rows in (issued first: nothing depends on them yet)
        float4 s[kRowsPerWarp];
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r)
            s[r] = __ldcs(reinterpret_cast<const float4 *>(Su + (row0 + r) * kD) + lane);
        // 2. the token's q, k (for my rows) and v (for my columns)
        if (threadIdx.x < kD) {
            q_s[threadIdx.x] = bf16_bits_to_float(q[vec + threadIdx.x]);
            k_s[threadIdx.x] = bf16_bits_to_float(k[vec + threadIdx.x]);
        }
        const uint2 vw = *reinterpret_cast<const uint2 *>(v + vec + 4 * lane);
        const float2 v01 = bf16x2_to_float2(vw.x), v23 = bf16x2_to_float2(vw.y);
        const float alpha = expf(g[unit]);
        if (pro.qw) qk_prologue_smem(q_s, k_s, pro, pro.pos[unit / ref.H]);
        __syncthreads();
        // 3. decay + rank-1 update, store back, and accumulate q S for my 4 columns
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) {
            const float ki = k_s[row0 + r], qi = q_s[row0 + r];
            float4 x = s[r];
            x.x = fmaf(alpha, x.x, ki * v01.x);
            x.y = fmaf(alpha, x.y, ki * v01.y);
            x.z = fmaf(alpha, x.z, ki * v23.x);
            x.w = fmaf(alpha, x.w, ki * v23.y);
            __stcs(reinterpret_cast<float4 *>(Su + (row0 + r) * kD) + lane, x);
            acc.x = fmaf(qi, x.x, acc.x);
            acc.y = fmaf(qi, x.y, acc.y);
            acc.z = fmaf(qi, x.z, acc.z);
            acc.w = fmaf(qi, x.w, acc.w);
        }
        *reinterpret_cast<float4 *>(&part[warp][4 * lane]) = acc;
    }
    __syncthreads();

    // 4. o_j = scale * sum over the 8 warp partials
    if (threadIdx.x < kD / 2) {
        const int j = 2 * threadIdx.x;
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int w = 0; w < kDecodeThreads / 32; ++w) {
            a0 += part[w][j];
            a1 += part[w][j + 1];
        }
        reinterpret_cast<uint32_t *>(o + vec)[threadIdx.x] = float2_to_bf16x2(scale * a0, scale * a1);
    }
}

cudaError_t launch_recurrent_step(const void *q, const void *k, const void *v, const float *g,
                                  float scale, float *S, void *o, int64_t units,
                                  cudaStream_t stream) {
    if (units == 0) return cudaSuccess;
    LaunchTimer timer(kKRecurrentStep, stream);
    return launch_dependent(recurrent_step_kernel<false>, static_cast<unsigned>(units), kDecodeThreads,
                            stream, static_cast<const uint16_t *>(q), static_cast<const uint16_t *>(k),
                            static_cast<const uint16_t *>(v), g, scale, StateRef{S, nullptr, 0, 1},
                            static_cast<uint16_t *>(o), nullptr, QkPrologue{});
}

cudaError_t launch_recurrent_step_indexed(const void *q, const void *k, const void *v,
                                          const float *g, float scale, void *pool, bool bf16,
                                          const int32_t *idx, int64_t P, void *o, int64_t N,
                                          int H, const QkPrologue &pro, int *status,
                                          cudaStream_t stream) {
    if (N == 0) return cudaSuccess;
    LaunchTimer timer(kKRecurrentStepIndexed, stream);
    const unsigned blocks = static_cast<unsigned>(N * H);
    const StateRef ref{pool, idx, P, H};
    const auto *qb = static_cast<const uint16_t *>(q), *kb = static_cast<const uint16_t *>(k),
               *vb = static_cast<const uint16_t *>(v);
    auto *ob = static_cast<uint16_t *>(o);
    if (bf16)
        return launch_dependent(recurrent_step_kernel<true>, blocks, kDecodeThreads, stream, qb, kb, vb, g,
                                scale, ref, ob, status, pro);
    return launch_dependent(recurrent_step_kernel<false>, blocks, kDecodeThreads, stream, qb, kb, vb, g,
                            scale, ref, ob, status, pro);
}

}  // namespace sala
