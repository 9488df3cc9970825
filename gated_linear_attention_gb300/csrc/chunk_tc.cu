// State pass and output pass of the chunked prefill on the tcgen05 tensor cores.
//
// Chunked form of the Simple GLA recurrence, chunk size 64 ("Formulas and Code for Adapting
// Inference to GDN/KDA Linear Modules", section 1.2, without the delta rule, beta = 1). For a
// chunk with cumulative in-chunk log-decay b_t (inclusive), last valid token C, incoming
// state S:
//     o_t   = scale * ( exp(b_t) q_t S  +  sum_{s<=t} exp(b_t - b_s) (q_t . k_s) v_s )
//     S_out = exp(b_C) S + sum_s exp(b_C - b_s) k_s^T v_s
// Only non-positive differences are exponentiated; the causal mask is applied before exp.
//
// Tiles: q, k, v chunks [64 tokens x 128] bf16 arrive by TMA (3-D tensor maps over
// [T, H, 128], box 64 x 1 x 64, 128-byte swizzle) into shared memory, two 8 KB regions per
// tile (d in [0,64) and [64,128)). The contractions run as tcgen05.mma kind::f16 (bf16 in,
// fp32 accumulate in tensor memory), issued by one thread:
//   M1  P      = Q K^T          M=64  N=64  K=128   A=Q (K-major)     B=K (K-major)
//   M2  O_x^T  = S^T Q^T        M=128 N=64  K=128   A=S bf16 (MN-major) B=Q (K-major)
//   M3  O_a^T  = V^T P'^T       M=128 N=64  K=64    A=V (MN-major)     B=P' (K-major)
//   M4  dS     = K'^T V         M=128 N=128 K=64    A=K' (MN-major)    B=V (MN-major)
// with P' the masked, decayed scores and K' = K scaled per token by its decay to the chunk
// end (both written to shared memory as bf16 by the epilogue warps). Outputs are kept
// transposed (value dimension on the TMEM lanes) so that every contraction but QK^T uses the
// full 128-row tensor-core shape. The fp32 running state lives in registers of the epilogue
// warps (each of two warpgroups owns 64 value columns); its bf16 copy in shared memory feeds
// M2 of the next chunk.
//
// Every wait is bounded (2 s of %globaltimer); on a timeout the CTA records SALA_ERR_TIMEOUT,
// stops issuing work, drains its own copies and MMAs, frees its tensor memory and returns.
#include <cudaTypedefs.h>

#include "launch.h"
#include "tc.cuh"

namespace sala {
namespace {

constexpr uint64_t kWaitNs = 2000000000ull;
constexpr uint32_t kRegion = 64 * 128;        // bytes of one [64 rows x 64 bf16] SW128 region
constexpr uint32_t kTile = 2 * kRegion;       // [64 tokens x 128] bf16
constexpr uint32_t kSRegion = 128 * 128;      // [128 rows x 64 bf16] SW128 region (16 KB)

__device__ __forceinline__ uint32_t sw(uint32_t row, uint32_t chunk16) {
    return row * 128 + ((chunk16 ^ (row & 7)) << 4);
}

__device__ __forceinline__ void named_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Named-barrier OR-vote: every participating thread contributes `x`, all get the OR.
__device__ __forceinline__ bool named_any(int id, int n, bool x) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(x)), "r"(id), "r"(n)
        : "memory");
    return r != 0;
}

// Bounded wait that also gives up as soon as another role has aborted.
__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity,
                                              volatile int *abort_flag, int *status) {
    if (tc::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = tc::global_timer_ns();
    while (!tc::mbar_try_wait(bar, parity)) {
        if (*abort_flag) return false;
        if (tc::global_timer_ns() - t0 > kWaitNs) {
            *abort_flag = 1;
            record_status(status, SALA_ERR_TIMEOUT);
            return false;
        }
    }
    return true;
}

// Inclusive prefix sum of g over the chunk's n valid tokens (zeros past n); lane l returns
// b[2l] and b[2l+1]. Called by a whole warp.
__device__ __forceinline__ float2 warp_chunk_cumsum(const float *__restrict__ g, int64_t c0, int n,
                                                    int H, int h) {
    const int l = threadIdx.x & 31;
    const float a0 = (2 * l < n) ? g[(c0 + 2 * l) * H + h] : 0.f;
    const float a1 = (2 * l + 1 < n) ? g[(c0 + 2 * l + 1) * H + h] : 0.f;
    const float pair = a0 + a1;
    float run = pair;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, run, off);
        if (l >= off) run += y;
    }
    const float excl = run - pair;
    return make_float2(excl + a0, excl + pair);
}

__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t w, float s) {
    const float2 f = bf16x2_to_float2(w);
    return float2_to_bf16x2(f.x * s, f.y * s);
}

struct TcMaps {
    CUtensorMap q, k, v;
};

}  // namespace

// =======================================================================================
// Output pass
// =======================================================================================

namespace {

constexpr int kOStages = 2;
constexpr int kOThreads = 320;  // warp 0 TMA, warp 1 MMA + TMEM owner, warps 2-5 WG0, 6-9 WG1

// dynamic shared memory layout (offsets from a 1024-aligned base)
constexpr uint32_t kO_Stage = 3 * kTile;                       // Q, K, V of one chunk
constexpr uint32_t kO_Kp = kOStages * kO_Stage;                // K' (MN-major A of M4)
constexpr uint32_t kO_Pp = kO_Kp + kTile;                      // P' (K-major B of M3)
constexpr uint32_t kO_Sb = kO_Pp + kRegion;                    // S bf16 (MN-major A of M2)
constexpr uint32_t kO_Ost = kO_Sb + 2 * kSRegion;              // o staging [64][128] bf16
constexpr uint32_t kO_Vals = kO_Ost + 64 * 256;                // b0[64], w0[64], b1[64], e1[64]
constexpr uint32_t kO_Bytes = kO_Vals + 4 * 64 * 4;
constexpr uint32_t kO_SmemAlloc = kO_Bytes + 1024;

// TMEM columns
constexpr uint32_t kT_P = 0, kT_Ox = 64, kT_Oa = 128, kT_dS = 256, kT_Cols = 512;

constexpr uint32_t kIdescP = tc::idesc_bf16_f32(64, 64, 0, 0);
constexpr uint32_t kIdescO = tc::idesc_bf16_f32(128, 64, 1, 0);
constexpr uint32_t kIdescS = tc::idesc_bf16_f32(128, 128, 1, 1);

}  // namespace

__global__ void __launch_bounds__(kOThreads, 1)
output_pass_tc(const __grid_constant__ TcMaps maps, ChunkArgs a, SegTable t, int *status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
    __shared__ uint64_t full[kOStages], empty[kOStages];
    __shared__ uint64_t p_full, p_ready, k_ready, o_full, o_free, s_full, s_ready, drain;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;

    const int64_t sigma = blockIdx.x / a.H;
    const int h = blockIdx.x % a.H;
    int64_t n_seq, t0, t1;
    if (!locate_segment(t, sigma, n_seq, t0, t1)) return;  // uniform across the CTA
    const int nchunks = static_cast<int>((t1 - t0 + kChunk - 1) / kChunk);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kOStages; ++s) {
            tc::mbar_init(&full[s], 1);
            tc::mbar_init(&empty[s], 2);
        }
        tc::mbar_init(&p_full, 1);
        tc::mbar_init(&p_ready, 1);
        tc::mbar_init(&k_ready, 1);
        tc::mbar_init(&o_full, 1);
        tc::mbar_init(&o_free, 1);
        tc::mbar_init(&s_full, 1);
        tc::mbar_init(&s_ready, 2);
        tc::mbar_init(&drain, 1);
        abort_flag = 0;
        tc::fence_barrier_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(&tmem_slot, kT_Cols);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = tmem_slot;
    volatile int *abort_v = &abort_flag;

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            tc::tma_prefetch_desc(&maps.q);
            tc::tma_prefetch_desc(&maps.k);
            tc::tma_prefetch_desc(&maps.v);
            int issued = 0;
            for (int c = 0; c < nchunks; ++c) {
                const int s = c % kOStages;
                if (c >= kOStages &&
                    !wait_or_abort(&empty[s], ((c / kOStages) - 1) & 1, abort_v, status))
                    break;
                uint8_t *st = sm + s * kO_Stage;
                const int32_t c0 = static_cast<int32_t>(t0 + int64_t(c) * kChunk);
                tc::mbar_arrive_expect_tx(&full[s], 3 * kTile);
                tc::tma_load_3d(st, &maps.q, 0, h, c0, &full[s]);
                tc::tma_load_3d(st + kRegion, &maps.q, 64, h, c0, &full[s]);
                tc::tma_load_3d(st + kTile, &maps.k, 0, h, c0, &full[s]);
                tc::tma_load_3d(st + kTile + kRegion, &maps.k, 64, h, c0, &full[s]);
                tc::tma_load_3d(st + 2 * kTile, &maps.v, 0, h, c0, &full[s]);
                tc::tma_load_3d(st + 2 * kTile + kRegion, &maps.v, 64, h, c0, &full[s]);
                issued = c + 1;
            }
            // drain: the last copies of each stage must land before the CTA may exit
            for (int c = issued - kOStages < 0 ? 0 : issued - kOStages; c < issued; ++c)
                tc::mbar_wait(&full[c % kOStages], (c / kOStages) & 1, kWaitNs);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            const uint32_t sb = tc::smem_u32(sm);
            for (int c = 0; c < nchunks; ++c) {
                const int s = c % kOStages;
                const uint32_t q_s = sb + s * kO_Stage, k_s = q_s + kTile, v_s = q_s + 2 * kTile;
                if (!wait_or_abort(&full[s], (c / kOStages) & 1, abort_v, status)) break;
                if (!wait_or_abort(&s_ready, c & 1, abort_v, status)) break;
                if (c > 0 && !wait_or_abort(&o_free, (c - 1) & 1, abort_v, status)) break;
                tc::tc_fence_after();
                // M1: P = Q K^T
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t off = (ks >> 2) * kRegion + (ks & 3) * 32;
                    tc::umma_bf16(tmem + kT_P, tc::smem_desc_sw128(q_s + off, 16, 1024),
                                  tc::smem_desc_sw128(k_s + off, 16, 1024), kIdescP, ks > 0);
                }
                tc::umma_commit(&p_full);
                // M2: O_x^T = S^T Q^T
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t a_off = ks * 2048, b_off = (ks >> 2) * kRegion + (ks & 3) * 32;
                    tc::umma_bf16(tmem + kT_Ox,
                                  tc::smem_desc_sw128(sb + kO_Sb + a_off, kSRegion, 1024),
                                  tc::smem_desc_sw128(q_s + b_off, 16, 1024), kIdescO, ks > 0);
                }
                if (!wait_or_abort(&k_ready, c & 1, abort_v, status)) break;
                tc::tc_fence_after();
                // M4: dS = K'^T V
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    const uint32_t off = ks * 2048;
                    tc::umma_bf16(tmem + kT_dS, tc::smem_desc_sw128(sb + kO_Kp + off, kRegion, 1024),
                                  tc::smem_desc_sw128(v_s + off, kRegion, 1024), kIdescS, ks > 0);
                }
                tc::umma_commit(&s_full);
                if (!wait_or_abort(&p_ready, c & 1, abort_v, status)) break;
                tc::tc_fence_after();
                // M3: O_a^T = V^T P'^T
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    tc::umma_bf16(tmem + kT_Oa, tc::smem_desc_sw128(v_s + ks * 2048, kRegion, 1024),
                                  tc::smem_desc_sw128(sb + kO_Pp + ks * 32, 16, 1024), kIdescO,
                                  ks > 0);
                }
                tc::umma_commit(&o_full);
                tc::umma_commit(&empty[s]);
            }
            // no MMA may still be running when the tensor memory is freed
            tc::umma_commit(&drain);
            tc::mbar_wait(&drain, 0, kWaitNs);
        }
    } else {
        // ---------------- epilogue warpgroups ----------------
        const int wg = (warp - 2) >> 2;                // 0 or 1
        const int wtid = threadIdx.x - 64 - 128 * wg;  // 0..127 inside the warpgroup
        const int quarter = warp & 3;                  // TMEM lane quarter this warp may access
        const int row = quarter * 32 + lane;           // TMEM lane = state row i / value col j
        const int bar_id = 1 + wg;
        float *vals = reinterpret_cast<float *>(sm + kO_Vals);
        float *bv = vals + 128 * wg;                   // b for this warpgroup's use
        float *wv = bv + 64;                           // WG0: K' weights; WG1: exp(b)
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        const int jc0 = 64 * wg;                       // my 64 state columns

        // the running fp32 state: S[row][jc0 .. jc0 + 64)
        float S[64];
        {
            const float *src = a.ws_state + (static_cast<size_t>(sigma) * a.H + h) * kD * kD +
                               row * kD + jc0;
#pragma unroll
            for (int j = 0; j < 64; j += 4) {
                const float4 x = *reinterpret_cast<const float4 *>(src + j);
                S[j] = x.x; S[j + 1] = x.y; S[j + 2] = x.z; S[j + 3] = x.w;
            }
            uint8_t *dst = sm + kO_Sb + wg * kSRegion;
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8) {
                uint4 w;
                w.x = float2_to_bf16x2(S[8 * c8 + 0], S[8 * c8 + 1]);
                w.y = float2_to_bf16x2(S[8 * c8 + 2], S[8 * c8 + 3]);
                w.z = float2_to_bf16x2(S[8 * c8 + 4], S[8 * c8 + 5]);
                w.w = float2_to_bf16x2(S[8 * c8 + 6], S[8 * c8 + 7]);
                *reinterpret_cast<uint4 *>(dst + sw(row, c8)) = w;
            }
            tc::fence_proxy_async_smem();
            named_sync(bar_id, 128);
            if (wtid == 0) tc::mbar_arrive(&s_ready);
        }

        for (int c = 0; c < nchunks; ++c) {
            const int s = c % kOStages;
            const int64_t c0 = t0 + int64_t(c) * kChunk;
            const int nv = static_cast<int>(min(static_cast<int64_t>(kChunk), t1 - c0));
            // cumulative decay of this chunk (every warp computes it; the first writes it out)
            const float2 bl = warp_chunk_cumsum(a.g, c0, nv, a.H, h);
            const float bC = __shfl_sync(0xffffffffu, (nv - 1) & 1 ? bl.y : bl.x, (nv - 1) >> 1);
            if (wtid < 32) {
                bv[2 * lane] = bl.x;
                bv[2 * lane + 1] = bl.y;
                if (wg == 0) {
                    wv[2 * lane] = 2 * lane < nv ? expf(bC - bl.x) : 0.f;
                    wv[2 * lane + 1] = 2 * lane + 1 < nv ? expf(bC - bl.y) : 0.f;
                } else {
                    wv[2 * lane] = expf(bl.x);
                    wv[2 * lane + 1] = expf(bl.y);
                }
            }
            named_sync(bar_id, 128);
            const float eC = expf(bC);

            if (wg == 0) {
                // (a) K' = K * exp(b_C - b_t) (zero past the valid tokens)
                bool bad = !wait_or_abort(&full[s], (c / kOStages) & 1, abort_v, status);
                if (named_any(bar_id, 128, bad)) break;
                const uint8_t *kt = sm + s * kO_Stage + kTile;
                uint8_t *kp = sm + kO_Kp;
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    const int idx = wtid + 128 * m;          // 1024 chunks of 16 bytes
                    const int r = idx >> 9, tr = (idx >> 3) & 63, ch = idx & 7;
                    const uint32_t off = r * kRegion + sw(tr, ch);
                    const float w = wv[tr];
                    uint4 x = *reinterpret_cast<const uint4 *>(kt + off);
                    x.x = mul_bf16x2(x.x, w);
                    x.y = mul_bf16x2(x.y, w);
                    x.z = mul_bf16x2(x.z, w);
                    x.w = mul_bf16x2(x.w, w);
                    if (tr >= nv) x = make_uint4(0u, 0u, 0u, 0u);
                    *reinterpret_cast<uint4 *>(kp + off) = x;
                }
                tc::fence_proxy_async_smem();
                named_sync(bar_id, 128);
                if (wtid == 0) {
                    tc::mbar_arrive(&k_ready);
                    tc::mbar_arrive(&empty[s]);
                }
                // (b) P' = mask(P) * exp(b_t - b_s) -> shared memory, bf16, K-major rows t
                bad = !wait_or_abort(&p_full, c & 1, abort_v, status);
                if (named_any(bar_id, 128, bad)) break;
                tc::tc_fence_after();
                {
                    uint32_t p0[32], p1[32];
                    tc::tmem_ld_32x32b_x32(tmem + lane_base + kT_P, p0);
                    tc::tmem_ld_32x32b_x32(tmem + lane_base + kT_P + 32, p1);
                    tc::tmem_ld_wait();
                    if (lane < 16) {
                        const int tr = quarter * 16 + lane;   // M=64 accumulator layout
                        const float bt = bv[tr];
                        uint8_t *pp = sm + kO_Pp;
#pragma unroll
                        for (int c8 = 0; c8 < 8; ++c8) {
                            float f[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                const int sc = 8 * c8 + e;
                                const float pv = __uint_as_float(sc < 32 ? p0[sc] : p1[sc - 32]);
                                f[e] = sc <= tr ? pv * expf(bt - bv[sc]) : 0.f;
                            }
                            uint4 w;
                            w.x = float2_to_bf16x2(f[0], f[1]);
                            w.y = float2_to_bf16x2(f[2], f[3]);
                            w.z = float2_to_bf16x2(f[4], f[5]);
                            w.w = float2_to_bf16x2(f[6], f[7]);
                            *reinterpret_cast<uint4 *>(pp + sw(tr, c8)) = w;
                        }
                    }
                }
                tc::fence_proxy_async_smem();
                tc::tc_fence_before();
                named_sync(bar_id, 128);
                if (wtid == 0) tc::mbar_arrive(&p_ready);
            }

            // (c) state carry for my 64 columns: S = exp(b_C) S + dS; bf16 copy for M2
            bool bad = !wait_or_abort(&s_full, c & 1, abort_v, status);
            if (named_any(bar_id, 128, bad)) break;
            tc::tc_fence_after();
            {
                uint32_t d0[32], d1[32];
                tc::tmem_ld_32x32b_x32(tmem + lane_base + kT_dS + jc0, d0);
                tc::tmem_ld_32x32b_x32(tmem + lane_base + kT_dS + jc0 + 32, d1);
                tc::tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    S[j] = fmaf(eC, S[j], __uint_as_float(d0[j]));
                    S[j + 32] = fmaf(eC, S[j + 32], __uint_as_float(d1[j]));
                }
                uint8_t *dst = sm + kO_Sb + wg * kSRegion;
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8) {
                    uint4 w;
                    w.x = float2_to_bf16x2(S[8 * c8 + 0], S[8 * c8 + 1]);
                    w.y = float2_to_bf16x2(S[8 * c8 + 2], S[8 * c8 + 3]);
                    w.z = float2_to_bf16x2(S[8 * c8 + 4], S[8 * c8 + 5]);
                    w.w = float2_to_bf16x2(S[8 * c8 + 6], S[8 * c8 + 7]);
                    *reinterpret_cast<uint4 *>(dst + sw(row, c8)) = w;
                }
            }
            tc::fence_proxy_async_smem();
            tc::tc_fence_before();
            named_sync(bar_id, 128);
            if (wtid == 0) tc::mbar_arrive(&s_ready);

            if (wg == 1) {
                // (d) o_t = scale (exp(b_t) O_x + O_a) for value column j = row; stage, store
                bad = !wait_or_abort(&o_full, c & 1, abort_v, status);
                if (named_any(bar_id, 128, bad)) break;
                tc::tc_fence_after();
                uint16_t *ost = reinterpret_cast<uint16_t *>(sm + kO_Ost);
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t ox[32], oa[32];
                    tc::tmem_ld_32x32b_x32(tmem + lane_base + kT_Ox + 32 * half, ox);
                    tc::tmem_ld_32x32b_x32(tmem + lane_base + kT_Oa + 32 * half, oa);
                    tc::tmem_ld_wait();
#pragma unroll
                    for (int tt = 0; tt < 32; ++tt) {
                        const int tr = 32 * half + tt;
                        const float o = a.scale * fmaf(wv[tr], __uint_as_float(ox[tt]),
                                                       __uint_as_float(oa[tt]));
                        ost[tr * kD + row] = __bfloat16_as_ushort(__float2bfloat16_rn(o));
                    }
                }
                tc::tc_fence_before();
                named_sync(bar_id, 128);
                if (wtid == 0) tc::mbar_arrive(&o_free);
                // coalesced copy of the valid rows to o[c0 + t, h, :]
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    const int idx = wtid + 128 * m;         // 64 rows x 16 chunks of 16 bytes
                    const int tr = idx >> 4, ch = idx & 15;
                    if (tr < nv) {
                        const uint4 x = *reinterpret_cast<const uint4 *>(ost + tr * kD + ch * 8);
                        *reinterpret_cast<uint4 *>(a.o + ((c0 + tr) * a.H + h) * kD + ch * 8) = x;
                    }
                }
                named_sync(bar_id, 128);
            }
        }
    }

    tc::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, kT_Cols);
    }
}

// =======================================================================================
// State pass: dS = sum over the segment of exp(B_end - B_t) k_t^T v_t, and B_end.
// Chunks are visited last to first so that every token's weight (its decay to the segment
// end) is known when its chunk is scaled: w_t = exp((b_C - b_t) + D), D the total decay of
// the chunks after this one. All weights are <= 1 and the MMA simply accumulates.
// =======================================================================================

namespace {

constexpr int kSStages = 3;
constexpr int kSThreads = 192;  // warp 0 TMA, warp 1 MMA + TMEM owner, warps 2-5 scalers
constexpr uint32_t kS_Stage = 2 * kTile;                 // K, V
constexpr uint32_t kS_Kp = kSStages * kS_Stage;          // K' double buffer
constexpr uint32_t kS_Vals = kS_Kp + 2 * kTile;          // w[64]
constexpr uint32_t kS_Bytes = kS_Vals + 64 * 4;
constexpr uint32_t kS_SmemAlloc = kS_Bytes + 1024;
constexpr uint32_t kS_Cols = 128;

}  // namespace

__global__ void __launch_bounds__(kSThreads, 1)
state_pass_tc(const __grid_constant__ TcMaps maps, ChunkArgs a, SegTable t, int *status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
    __shared__ uint64_t full[kSStages], empty[kSStages], kready[2], kfree[2], done;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;

    const int64_t sigma = blockIdx.x / a.H;
    const int h = blockIdx.x % a.H;
    int64_t n_seq, t0, t1;
    if (!locate_segment(t, sigma, n_seq, t0, t1)) return;
    const int nchunks = static_cast<int>((t1 - t0 + kChunk - 1) / kChunk);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kSStages; ++s) {
            tc::mbar_init(&full[s], 1);
            tc::mbar_init(&empty[s], 2);
        }
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(&kready[i], 1);
            tc::mbar_init(&kfree[i], 1);
        }
        tc::mbar_init(&done, 1);
        abort_flag = 0;
        tc::fence_barrier_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(&tmem_slot, kS_Cols);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = tmem_slot;
    volatile int *abort_v = &abort_flag;

    if (warp == 0) {
        if (lane == 0) {
            tc::tma_prefetch_desc(&maps.k);
            tc::tma_prefetch_desc(&maps.v);
            int issued = 0;
            for (int r = 0; r < nchunks; ++r) {
                const int c = nchunks - 1 - r, s = r % kSStages;
                if (r >= kSStages &&
                    !wait_or_abort(&empty[s], ((r / kSStages) - 1) & 1, abort_v, status))
                    break;
                uint8_t *st = sm + s * kS_Stage;
                const int32_t c0 = static_cast<int32_t>(t0 + int64_t(c) * kChunk);
                tc::mbar_arrive_expect_tx(&full[s], 2 * kTile);
                tc::tma_load_3d(st, &maps.k, 0, h, c0, &full[s]);
                tc::tma_load_3d(st + kRegion, &maps.k, 64, h, c0, &full[s]);
                tc::tma_load_3d(st + kTile, &maps.v, 0, h, c0, &full[s]);
                tc::tma_load_3d(st + kTile + kRegion, &maps.v, 64, h, c0, &full[s]);
                issued = r + 1;
            }
            for (int r = issued - kSStages < 0 ? 0 : issued - kSStages; r < issued; ++r)
                tc::mbar_wait(&full[r % kSStages], (r / kSStages) & 1, kWaitNs);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t sb = tc::smem_u32(sm);
            constexpr uint32_t idesc = tc::idesc_bf16_f32(128, 128, 1, 1);
            for (int r = 0; r < nchunks; ++r) {
                const int s = r % kSStages, kb = r & 1;
                if (!wait_or_abort(&full[s], (r / kSStages) & 1, abort_v, status)) break;
                if (!wait_or_abort(&kready[kb], (r >> 1) & 1, abort_v, status)) break;
                tc::tc_fence_after();
                const uint32_t v_s = sb + s * kS_Stage + kTile, kp = sb + kS_Kp + kb * kTile;
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    tc::umma_bf16(tmem, tc::smem_desc_sw128(kp + ks * 2048, kRegion, 1024),
                                  tc::smem_desc_sw128(v_s + ks * 2048, kRegion, 1024), idesc,
                                  (r > 0 || ks > 0) ? 1u : 0u);
                tc::umma_commit(&kfree[kb]);
                tc::umma_commit(&empty[s]);
            }
            tc::umma_commit(&done);
        }
    } else {
        const int wtid = threadIdx.x - 64;
        const int quarter = warp & 3;
        float *wv = reinterpret_cast<float *>(sm + kS_Vals);
        float D = 0.f;  // total log-decay of the chunks already visited (those after this one)
        bool ok = true;
        for (int r = 0; r < nchunks; ++r) {
            const int c = nchunks - 1 - r, s = r % kSStages, kb = r & 1;
            const int64_t c0 = t0 + int64_t(c) * kChunk;
            const int nv = static_cast<int>(min(static_cast<int64_t>(kChunk), t1 - c0));
            const float2 bl = warp_chunk_cumsum(a.g, c0, nv, a.H, h);
            const float bC = __shfl_sync(0xffffffffu, (nv - 1) & 1 ? bl.y : bl.x, (nv - 1) >> 1);
            bool bad = !wait_or_abort(&full[s], (r / kSStages) & 1, abort_v, status);
            if (!bad && r >= 2) bad = !wait_or_abort(&kfree[kb], ((r >> 1) - 1) & 1, abort_v, status);
            if (named_any(1, 128, bad)) {
                ok = false;
                break;
            }
            if (wtid < 32) {
                wv[2 * lane] = 2 * lane < nv ? expf(bC - bl.x + D) : 0.f;
                wv[2 * lane + 1] = 2 * lane + 1 < nv ? expf(bC - bl.y + D) : 0.f;
            }
            named_sync(1, 128);
            const uint8_t *kt = sm + s * kS_Stage;
            uint8_t *kp = sm + kS_Kp + kb * kTile;
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                const int idx = wtid + 128 * m;
                const int rg = idx >> 9, tr = (idx >> 3) & 63, ch = idx & 7;
                const uint32_t off = rg * kRegion + sw(tr, ch);
                const float w = wv[tr];
                uint4 x = *reinterpret_cast<const uint4 *>(kt + off);
                x.x = mul_bf16x2(x.x, w);
                x.y = mul_bf16x2(x.y, w);
                x.z = mul_bf16x2(x.z, w);
                x.w = mul_bf16x2(x.w, w);
                if (tr >= nv) x = make_uint4(0u, 0u, 0u, 0u);
                *reinterpret_cast<uint4 *>(kp + off) = x;
            }
            tc::fence_proxy_async_smem();
            named_sync(1, 128);   // also: every thread has read wv before it is rewritten
            if (wtid == 0) {
                tc::mbar_arrive(&kready[kb]);
                tc::mbar_arrive(&empty[s]);
            }
            D += bC;
        }
        // dS rows (TMEM lane = key row i) -> scratch
        bool bad = !ok || !wait_or_abort(&done, 0, abort_v, status);
        if (!named_any(1, 128, bad)) {
            tc::tc_fence_after();
            const int i = quarter * 32 + lane;
            float *dst = a.ws_state + (static_cast<size_t>(sigma) * a.H + h) * kD * kD + i * kD;
            const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
#pragma unroll
            for (int j0 = 0; j0 < kD; j0 += 32) {
                uint32_t d[32];
                tc::tmem_ld_32x32b_x32(tmem + lane_base + j0, d);
                tc::tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; j += 4)
                    *reinterpret_cast<float4 *>(dst + j0 + j) =
                        make_float4(__uint_as_float(d[j]), __uint_as_float(d[j + 1]),
                                    __uint_as_float(d[j + 2]), __uint_as_float(d[j + 3]));
            }
            if (wtid == 0) a.ws_decay[sigma * a.H + h] = D;
        }
    }

    tc::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        // the MMA thread's final commit covers every MMA it issued
        if (lane == 0) tc::mbar_wait(&done, 0, kWaitNs);
        __syncwarp();
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, kS_Cols);
    }
}

// =======================================================================================
// host side

namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
cudaError_t g_encode_err = cudaSuccess;
std::once_flag g_encode_once;

cudaError_t encode_map(CUtensorMap *map, const void *base, int64_t T_total, int H) {
    std::call_once(g_encode_once, []() {
        cudaDriverEntryPointQueryResult q;
        g_encode_err = cudaGetDriverEntryPointByVersion(
            "cuTensorMapEncodeTiled", reinterpret_cast<void **>(&g_encode), 12000,
            cudaEnableDefault, &q);
        if (g_encode_err == cudaSuccess && q != cudaDriverEntryPointSuccess)
            g_encode_err = cudaErrorNotSupported;
    });
    if (g_encode_err != cudaSuccess) return g_encode_err;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(H),
                          static_cast<cuuint64_t>(T_total)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(kD) * 2, static_cast<cuuint64_t>(H) * kD * 2};
    cuuint32_t box[3] = {64, 1, 64};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_maps(TcMaps *m, const ChunkArgs &a, int64_t T_total) {
    cudaError_t e = encode_map(&m->q, a.q, T_total, a.H);
    if (e == cudaSuccess) e = encode_map(&m->k, a.k, T_total, a.H);
    if (e == cudaSuccess) e = encode_map(&m->v, a.v, T_total, a.H);
    return e;
}

}  // namespace

cudaError_t setup_tc_kernels() {
    cudaError_t e = cudaFuncSetAttribute(output_pass_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kO_SmemAlloc));
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(state_pass_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(kS_SmemAlloc));
}

cudaError_t launch_state_pass(const ChunkArgs &a, const SegTable &t, int64_t T_total,
                              int64_t max_units, int *status, cudaStream_t st) {
    if (T_total == 0 || max_units == 0) return cudaSuccess;
    TcMaps maps;
    cudaError_t e = make_maps(&maps, a, T_total);
    if (e != cudaSuccess) return e;
    LaunchTimer timer(kKStatePass, st);
    state_pass_tc<<<static_cast<unsigned>(max_units), kSThreads, kS_SmemAlloc, st>>>(maps, a, t,
                                                                                    status);
    return cudaGetLastError();
}

cudaError_t launch_output_pass(const ChunkArgs &a, const SegTable &t, int64_t T_total,
                               int64_t max_units, int *status, cudaStream_t st) {
    if (T_total == 0 || max_units == 0) return cudaSuccess;
    TcMaps maps;
    cudaError_t e = make_maps(&maps, a, T_total);
    if (e != cudaSuccess) return e;
    LaunchTimer timer(kKOutputPass, st);
    output_pass_tc<<<static_cast<unsigned>(max_units), kOThreads, kO_SmemAlloc, st>>>(maps, a, t,
                                                                                     status);
    return cudaGetLastError();
}

}  // namespace sala
