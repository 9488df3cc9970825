// State pass and output pass of the chunked prefill on the CUDA cores (fp32 FMA).
//
// Chunked form of the Simple GLA recurrence with chunk size 64 ("Formulas and Code for
// Adapting Inference to GDN/KDA Linear Modules", section 1.2, without the delta rule and
// with beta = 1). Inside a chunk, with b_i the cumulative log-decay of the chunk up to token
// i (inclusive) and S the state entering the chunk:
//     o_i   = scale * ( exp(b_i) q_i S  +  sum_{j<=i} exp(b_i - b_j) (q_i . k_j) v_j )
//     S_out = exp(b_C) S + sum_j exp(b_C - b_j) k_j^T v_j        (b_C: last token's b)
// Only non-positive differences are exponentiated, and the mask is applied before exp.
#include "launch.h"

namespace sala {

constexpr int kSimtThreads = 256;

// Inclusive prefix sum of g over the chunk's n valid tokens into b[0..63] (zeros past n),
// done by warp 0 with two tokens per lane.
__device__ __forceinline__ void chunk_cumsum(const float *__restrict__ g, int64_t t0, int n, int H,
                                             int h, float *b) {
    if (threadIdx.x < 32) {
        const int l = threadIdx.x;
        float a0 = (2 * l < n) ? g[(t0 + 2 * l) * H + h] : 0.f;
        float a1 = (2 * l + 1 < n) ? g[(t0 + 2 * l + 1) * H + h] : 0.f;
        a1 += a0;
        float run = a1;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, run, off);
            if (l >= off) run += y;
        }
        const float excl = run - a1;
        b[2 * l] = excl + a0;
        b[2 * l + 1] = excl + a1;
    }
}

// Load rows [t0, t0 + n) of head h of a [T, H, 128] bf16 tensor into fp32 smem [64][128];
// rows past n are zero.
__device__ __forceinline__ void load_tile(const uint16_t *__restrict__ x, int64_t t0, int n, int H,
                                          int h, float *dst) {
    for (int idx = threadIdx.x; idx < kChunk * kD / 8; idx += blockDim.x) {
        const int r = idx / (kD / 8), c = (idx % (kD / 8)) * 8;
        float4 lo = make_float4(0.f, 0.f, 0.f, 0.f), hi = lo;
        if (r < n) {
            const uint4 w = *reinterpret_cast<const uint4 *>(x + ((t0 + r) * H + h) * kD + c);
            const float2 a = bf16x2_to_float2(w.x), b2 = bf16x2_to_float2(w.y);
            const float2 c2 = bf16x2_to_float2(w.z), d = bf16x2_to_float2(w.w);
            lo = make_float4(a.x, a.y, b2.x, b2.y);
            hi = make_float4(c2.x, c2.y, d.x, d.y);
        }
        *reinterpret_cast<float4 *>(dst + r * kD + c) = lo;
        *reinterpret_cast<float4 *>(dst + r * kD + c + 4) = hi;
    }
}

// ---------------------------------------------------------------------------------------
// State pass: dS = sum over the segment of exp(B_end - B_t) k_t^T v_t, and Bsum = B_end.
// Thread (ty, tx) = (tid / 16, tid % 16) owns rows [8ty, 8ty+8) x cols [8tx, 8tx+8) of dS.
__global__ void __launch_bounds__(kSimtThreads)
state_pass_simt(ChunkArgs a, SegTable t) {
    extern __shared__ float4 smem4[];
    float *k_s = reinterpret_cast<float *>(smem4);
    float *v_s = k_s + kChunk * kD;
    float *b_s = v_s + kChunk * kD;
    float *w_s = b_s + kChunk;
    const int64_t sigma = blockIdx.x / a.H;
    const int h = blockIdx.x % a.H;
    int64_t n, t0, t1;
    if (!locate_segment(t, sigma, n, t0, t1)) return;
    const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
    float Bsum = 0.f;
    for (int64_t c0 = t0; c0 < t1; c0 += kChunk) {
        const int nv = static_cast<int>(::min(static_cast<int64_t>(kChunk), t1 - c0));
        __syncthreads();
        load_tile(a.k, c0, nv, a.H, h, k_s);
        load_tile(a.v, c0, nv, a.H, h, v_s);
        chunk_cumsum(a.g, c0, nv, a.H, h, b_s);
        __syncthreads();
        const float bC = b_s[nv - 1];
        if (threadIdx.x < kChunk)
            w_s[threadIdx.x] = threadIdx.x < nv ? expf(bC - b_s[threadIdx.x]) : 0.f;
        __syncthreads();
        const float dC = expf(bC);
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[i][j] *= dC;
        for (int s = 0; s < nv; ++s) {
            const float w = w_s[s];
            float kv[8], vv[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) kv[i] = w * k_s[s * kD + 8 * ty + i];
#pragma unroll
            for (int j = 0; j < 8; ++j) vv[j] = v_s[s * kD + 8 * tx + j];
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(kv[i], vv[j], acc[i][j]);
        }
        Bsum += bC;
    }
    float *out = a.ws_state + (static_cast<size_t>(sigma) * a.H + h) * kD * kD;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        float4 *row = reinterpret_cast<float4 *>(out + (8 * ty + i) * kD + 8 * tx);
        row[0] = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
        row[1] = make_float4(acc[i][4], acc[i][5], acc[i][6], acc[i][7]);
    }
    if (threadIdx.x == 0) a.ws_decay[sigma * a.H + h] = Bsum;
}

// ---------------------------------------------------------------------------------------
// Output pass: restart the segment from S_in (ws_state) and produce o chunk by chunk.
__global__ void __launch_bounds__(kSimtThreads)
output_pass_simt(ChunkArgs a, SegTable t) {
    extern __shared__ float4 smem4[];
    float *S_s = reinterpret_cast<float *>(smem4);  // [128][128]
    float *q_s = S_s + kD * kD;                      // [64][128]
    float *k_s = q_s + kChunk * kD;
    float *v_s = k_s + kChunk * kD;
    float *P_s = v_s + kChunk * kD;                  // [64][64]
    float *b_s = P_s + kChunk * kChunk;
    float *w_s = b_s + kChunk;
    float *e_s = w_s + kChunk;
    const int64_t sigma = blockIdx.x / a.H;
    const int h = blockIdx.x % a.H;
    int64_t n, t0, t1;
    if (!locate_segment(t, sigma, n, t0, t1)) return;
    const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;

    // my 8 x 8 block of the running state, in registers; a copy lives in S_s
    float st[8][8];
    const float *Sin = a.ws_state + (static_cast<size_t>(sigma) * a.H + h) * kD * kD;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float4 *row = reinterpret_cast<const float4 *>(Sin + (8 * ty + i) * kD + 8 * tx);
        const float4 x0 = row[0], x1 = row[1];
        st[i][0] = x0.x; st[i][1] = x0.y; st[i][2] = x0.z; st[i][3] = x0.w;
        st[i][4] = x1.x; st[i][5] = x1.y; st[i][6] = x1.z; st[i][7] = x1.w;
    }

    for (int64_t c0 = t0; c0 < t1; c0 += kChunk) {
        const int nv = static_cast<int>(::min(static_cast<int64_t>(kChunk), t1 - c0));
        __syncthreads();  // previous chunk finished with every smem buffer
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float4 *row = reinterpret_cast<float4 *>(S_s + (8 * ty + i) * kD + 8 * tx);
            row[0] = make_float4(st[i][0], st[i][1], st[i][2], st[i][3]);
            row[1] = make_float4(st[i][4], st[i][5], st[i][6], st[i][7]);
        }
        load_tile(a.q, c0, nv, a.H, h, q_s);
        load_tile(a.k, c0, nv, a.H, h, k_s);
        load_tile(a.v, c0, nv, a.H, h, v_s);
        chunk_cumsum(a.g, c0, nv, a.H, h, b_s);
        __syncthreads();
        const float bC = b_s[nv - 1];
        if (threadIdx.x < kChunk) {
            const int j = threadIdx.x;
            w_s[j] = j < nv ? expf(bC - b_s[j]) : 0.f;
            e_s[j] = expf(b_s[j]);
        }
        // P = (Q K^T) masked to j <= i and scaled by exp(b_i - b_j); rows 4ty.., cols 4tx..
        {
            float p[4][4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) p[i][j] = 0.f;
            for (int d = 0; d < kD; ++d) {
                float qv[4], kv[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) qv[i] = q_s[(4 * ty + i) * kD + d];
#pragma unroll
                for (int j = 0; j < 4; ++j) kv[j] = k_s[(4 * tx + j) * kD + d];
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) p[i][j] = fmaf(qv[i], kv[j], p[i][j]);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int r = 4 * ty + i, c = 4 * tx + j;
                    P_s[r * kChunk + c] = c <= r ? p[i][j] * expf(b_s[r] - b_s[c]) : 0.f;
                }
        }
        __syncthreads();
        // O rows [4ty, 4ty+4) x cols [8tx, 8tx+8): exp(b_i) q_i S + sum_j P_ij v_j
        {
            float oi[4][8], oa[4][8];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) oi[i][j] = oa[i][j] = 0.f;
            for (int d = 0; d < kD; ++d) {
                float qv[4], sv[8];
#pragma unroll
                for (int i = 0; i < 4; ++i) qv[i] = q_s[(4 * ty + i) * kD + d];
#pragma unroll
                for (int j = 0; j < 8; ++j) sv[j] = S_s[d * kD + 8 * tx + j];
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 8; ++j) oi[i][j] = fmaf(qv[i], sv[j], oi[i][j]);
            }
            for (int s = 0; s < kChunk; ++s) {
                float pv[4], vv[8];
#pragma unroll
                for (int i = 0; i < 4; ++i) pv[i] = P_s[(4 * ty + i) * kChunk + s];
#pragma unroll
                for (int j = 0; j < 8; ++j) vv[j] = v_s[s * kD + 8 * tx + j];
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 8; ++j) oa[i][j] = fmaf(pv[i], vv[j], oa[i][j]);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int r = 4 * ty + i;
                if (r < nv) {
                    const float e = e_s[r];
                    uint4 w;
                    w.x = float2_to_bf16x2(a.scale * fmaf(e, oi[i][0], oa[i][0]),
                                           a.scale * fmaf(e, oi[i][1], oa[i][1]));
                    w.y = float2_to_bf16x2(a.scale * fmaf(e, oi[i][2], oa[i][2]),
                                           a.scale * fmaf(e, oi[i][3], oa[i][3]));
                    w.z = float2_to_bf16x2(a.scale * fmaf(e, oi[i][4], oa[i][4]),
                                           a.scale * fmaf(e, oi[i][5], oa[i][5]));
                    w.w = float2_to_bf16x2(a.scale * fmaf(e, oi[i][6], oa[i][6]),
                                           a.scale * fmaf(e, oi[i][7], oa[i][7]));
                    *reinterpret_cast<uint4 *>(a.o + ((c0 + r) * a.H + h) * kD + 8 * tx) = w;
                }
            }
        }
        // state carry: S = exp(b_C) S + sum_j exp(b_C - b_j) k_j^T v_j
        const float dC = expf(bC);
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) st[i][j] *= dC;
        for (int s = 0; s < nv; ++s) {
            const float w = w_s[s];
            float kv[8], vv[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) kv[i] = w * k_s[s * kD + 8 * ty + i];
#pragma unroll
            for (int j = 0; j < 8; ++j) vv[j] = v_s[s * kD + 8 * tx + j];
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) st[i][j] = fmaf(kv[i], vv[j], st[i][j]);
        }
    }
}

constexpr size_t kStateSimtSmem = (2 * kChunk * kD + 2 * kChunk) * sizeof(float);
constexpr size_t kOutputSimtSmem =
    (kD * kD + 3 * kChunk * kD + kChunk * kChunk + 3 * kChunk) * sizeof(float);

cudaError_t setup_simt_kernels() {
    cudaError_t e = cudaFuncSetAttribute(state_pass_simt,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kStateSimtSmem));
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(output_pass_simt, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(kOutputSimtSmem));
}

cudaError_t launch_state_pass(const ChunkArgs &a, const SegTable &t, int64_t max_units,
                              cudaStream_t st) {
    LaunchTimer timer(kKStatePass, st);
    state_pass_simt<<<static_cast<unsigned>(max_units), kSimtThreads, kStateSimtSmem, st>>>(a, t);
    return cudaGetLastError();
}

cudaError_t launch_output_pass(const ChunkArgs &a, const SegTable &t, int64_t max_units,
                               cudaStream_t st) {
    LaunchTimer timer(kKOutputPass, st);
    output_pass_simt<<<static_cast<unsigned>(max_units), kSimtThreads, kOutputSimtSmem, st>>>(a,
                                                                                              t);
    return cudaGetLastError();
}

}  // namespace sala
