// Chunked prefill in one persistent kernel: per-segment state pass, chained hand-off of the
// incoming state between consecutive segments, and the output pass.
//
// The recurrence ("MiniCPM-SALA — Complete Blueprint", "Simple GLA Recurrence") is evaluated
// in its chunked form with chunk size 64 ("Formulas and Code for Adapting Inference to
// GDN/KDA Linear Modules", section 1.2, without the delta rule, beta = 1). A sequence is cut
// into segments of L tokens (a multiple of 64); a work unit is one (segment, head). Units are
// handed out in segment-major order from an atomic ticket, so a unit's predecessor (the
// previous segment of the same sequence and head) always holds a smaller ticket and is
// already running on some CTA. For each unit a CTA runs:
//
//  A. state pass over the segment's chunks, last to first: dS = sum_t exp(B_end - B_t)
//     k_t^T v_t accumulated by tcgen05 in tensor memory (k_t pre-scaled in shared memory by
//     its decay to the segment end, so every weight is <= 1), and the total log-decay B;
//  hand-off: S_in = h0 (first segment) or the state the predecessor published; publish
//     S_out = exp(B) S_in + dS for the successor (hT for the last segment). This is the
//     Blueprint's unrolled form S_n = alpha^n S_0 + sum alpha^(n-i) k_i^T v_i applied a whole
//     segment at a time;
//  C. output pass over the chunks, first to last, from S_in. With b_t the cumulative
//     log-decay of the chunk up to token t and S the state entering the chunk:
//       o_t = scale exp(b_t) [ q_t S + sum_{s<=t} (q_t . k_s) exp(-b_s) v_s ]
//       S  <- exp(b_C) S + sum_s exp(b_C - b_s) k_s^T v_s
//     which keeps both output terms in one accumulator (the weights become per-column
//     factors exp(-b_s) on the scores and per-row factors exp(b_t) on the output). When a
//     chunk's decay range is too wide for those factors (|b_t| > 60), the chunk takes the
//     exact route instead: per-entry factors exp(b_t - b_s) on the scores and q_t scaled by
//     exp(b_t) in place. Contractions (tcgen05.mma kind::f16, bf16 in, fp32 in TMEM):
//       M1  P    = Q K^T       M=64  N=64  K=128   A=Q (K-major)      B=K (K-major)
//       M2  O^T  = S^T Q^T     M=128 N=64  K=128   A=S bf16 (MN-major) B=Q (K-major)
//       M3  O^T += V^T P'^T    M=128 N=64  K=64    A=V (MN-major)      B=P' (K-major)
//       M4  dS   = K'^T V      M=128 N=128 K=64    A=K' (MN-major)     B=V (MN-major)
//
// K and V are read in A and again in C shortly after, while they are still in L2 (the A
// loads ask L2 to keep them, the C loads let them go).
//
// Roles: warp 0 loads (TMA tiles; the lanes load the chunk's 64 log-decays and publish their
// prefix sums), warp 1 issues MMAs and owns the tensor memory, warpgroup 0 (warps 2-5)
// scales K and the scores and owns state columns 0-63, warpgroup 1 (warps 6-9) owns state
// columns 64-127 and writes o, warp 10 publishes hand-off flags. Scores, outputs, dS and the
// bf16 state are double-buffered so that only the fp32 state update is serial per chunk.
// Every wait is bounded (2 s of %globaltimer); a timeout records SALA_ERR_TIMEOUT, stops the
// CTA's work, drains its copies and MMAs, frees its tensor memory and returns.
#include "chunk_tc.cuh"

namespace sala {
namespace {

using namespace tck;

constexpr int kStages = 3;
constexpr int kThreads = 352;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kFastRange = 60.f;   // max |b_t| (natural log) for the factored route

// dynamic shared memory (offsets from a 1024-aligned base)
constexpr uint32_t kStage = 3 * kTile;              // Q | K | V
constexpr uint32_t kKp = kStages * kStage;          // K' [2] (MN-major A of M4)
constexpr uint32_t kPp = kKp + 2 * kTile;           // P' (K-major B of M3)
constexpr uint32_t kSb = kPp + kRegion;             // S bf16 (MN-major A of M2), 32 KB
constexpr uint32_t kMeta = kSb + 2 * kSRegion;      // per stage: chunk metadata (512 B)
constexpr uint32_t kVals = kMeta + kStages * 512;   // per warpgroup: 64 floats
constexpr uint32_t kBytes = kVals + 2 * 64 * 4;
constexpr uint32_t kSmemAlloc = kBytes + 1024;

struct alignas(16) ChunkMeta {
    float b[64];   // inclusive prefix sums of g over the chunk (0 past the valid tokens)
    float bC;      // b at the last valid token
    int fast;      // 1: factored weights are safe (max |b_t| <= kFastRange)
    int nv;        // valid tokens
    int pad_[61];  // one 512-byte slot per stage
};
static_assert(sizeof(ChunkMeta) == 512, "one 512-byte metadata slot per stage");

// TMEM columns: P [2] (M=64 layout), O [2], dS [2]
constexpr uint32_t kTP = 0, kTO = 128, kTdS = 256, kTCols = 512;
constexpr uint32_t kIdescP = tc::idesc_bf16_f32(64, 64, 0, 0);
constexpr uint32_t kIdescO = tc::idesc_bf16_f32(128, 64, 1, 0);
constexpr uint32_t kIdescS = tc::idesc_bf16_f32(128, 128, 1, 1);

struct FusedArgs {
    ChunkArgs c;            // q, k, v, g, scale, o, H
    const float *h0;        // [nseq, H, 128, 128] or null
    float *hT;              // [nseq, H, 128, 128] or null
    float *incl;            // [units, 128, 128]: state after each (segment, head)
    uint32_t *flags;        // [units]: == epoch once incl of that unit is published
    uint32_t *ticket;       // work counter, zeroed by the table kernel
    uint32_t epoch;
};

struct UnitInfo {
    int valid, h, nch, first, last;
    int64_t sigma, n, t0, t1;
};

// Event trace of CTA 0 for latency analysis (compiled only with -DSALA_TRACE): SM clock,
// role, event id and chunk index, kept in shared memory and copied out at exit.
#ifdef SALA_TRACE
constexpr int kTraceN = 512;
__device__ unsigned long long g_trace[4][kTraceN];
__device__ unsigned int g_trace_n[4];
#define TRACE(role, ev, idx)                                                                  \
    do {                                                                                      \
        if (blockIdx.x == 0 && tr_i < kTraceN) {                                              \
            g_trace[role][tr_i] = (static_cast<unsigned long long>(clock64()) & 0xFFFFFFFFFFFFull) | \
                                  (static_cast<unsigned long long>(role) << 60) |             \
                                  (static_cast<unsigned long long>(ev) << 52) |               \
                                  (static_cast<unsigned long long>((idx) & 0xF) << 48);       \
            ++tr_i;                                                                           \
            g_trace_n[role] = tr_i;                                                           \
        }                                                                                     \
    } while (0)
#else
#define TRACE(role, ev, idx) \
    do {                     \
    } while (0)
#endif

// shared-memory matrix descriptors: fixed part | (start address >> 4)
__device__ __forceinline__ uint64_t desc_k(uint32_t addr) {          // K-major, SW128
    return tc::smem_desc_sw128(0, 16, 1024) | ((addr >> 4) & 0x3FFFu);
}
__device__ __forceinline__ uint64_t desc_mn8(uint32_t addr) {        // MN-major, 8 KB atoms
    return tc::smem_desc_sw128(0, kRegion, 1024) | ((addr >> 4) & 0x3FFFu);
}
__device__ __forceinline__ uint64_t desc_mn16(uint32_t addr) {       // MN-major, 16 KB atoms
    return tc::smem_desc_sw128(0, kSRegion, 1024) | ((addr >> 4) & 0x3FFFu);
}

__device__ __forceinline__ void store_bf16_row64(uint8_t *region, int row, const float *S) {
#pragma unroll
    for (int c8 = 0; c8 < 8; ++c8) {
        uint4 w;
        w.x = float2_to_bf16x2(S[8 * c8 + 0], S[8 * c8 + 1]);
        w.y = float2_to_bf16x2(S[8 * c8 + 2], S[8 * c8 + 3]);
        w.z = float2_to_bf16x2(S[8 * c8 + 4], S[8 * c8 + 5]);
        w.w = float2_to_bf16x2(S[8 * c8 + 6], S[8 * c8 + 7]);
        *reinterpret_cast<uint4 *>(region + sw(row, c8)) = w;
    }
}

// Scale 16-byte pieces p0 + stride*m (m < N) of a [64 x 128] bf16 tile (two SW128 regions)
// by a per-row factor 2^(base + sign * b[t] * log2(e)), writing to dst (same layout); rows
// >= nv become zero. All loads are issued before any store (dst may equal src).
template <int N>
__device__ __forceinline__ void scale_rows(const uint8_t *src, uint8_t *dst, int p0, int stride,
                                           int nv, const float *b, float base, float sign) {
    uint4 x[N];
    uint32_t off[N];
    int tr[N];
#pragma unroll
    for (int m = 0; m < N; ++m) {
        const int idx = p0 + stride * m;
        const int rg = idx >> 9, ch = idx & 7;
        tr[m] = (idx >> 3) & 63;
        off[m] = rg * kRegion + sw(tr[m], ch);
        x[m] = *reinterpret_cast<const uint4 *>(src + off[m]);
    }
#pragma unroll
    for (int m = 0; m < N; ++m) {
        if (tr[m] < nv) {
            const float w = tc::ex2(fmaf(sign * kLog2e, b[tr[m]], base));
            x[m].x = mul_bf16x2(x[m].x, w);
            x[m].y = mul_bf16x2(x[m].y, w);
            x[m].z = mul_bf16x2(x[m].z, w);
            x[m].w = mul_bf16x2(x[m].w, w);
        } else {
            x[m] = make_uint4(0u, 0u, 0u, 0u);
        }
    }
#pragma unroll
    for (int m = 0; m < N; ++m) *reinterpret_cast<uint4 *>(dst + off[m]) = x[m];
}

// Bounded wait (if `need`) whose failure only sets the abort flag (see the epilogue loop).
__device__ __forceinline__ void wait_nv(uint64_t *bar, uint32_t par, bool need,
                                        volatile int *abort_v, int *status) {
    if (need) (void)wait_or_abort(bar, par & 1, abort_v, status);
}

// Bounded wait on an mbarrier phase by every thread of a warpgroup (if `need`), then an
// OR-vote so that all 128 threads take the same branch. Returns false if any thread failed.
__device__ __forceinline__ bool wg_wait(uint64_t *bar, uint32_t par, bool need, int bar_id,
                                        volatile int *abort_v, int *status) {
    const bool bad = need ? !wait_or_abort(bar, par & 1, abort_v, status) : false;
    return !named_any(bar_id, 128, bad);
}

}  // namespace

__global__ void __launch_bounds__(kThreads, 1)
prefill_fused_kernel(const __grid_constant__ TcMaps maps, FusedArgs f, SegTable t, int *status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
    __shared__ uint64_t full[kStages], empty[kStages], unit_full[2], unit_empty[2];
    __shared__ uint64_t kp_ready[2], kp_free[2], pub_ready, drain;
    __shared__ uint64_t ds_full[2], ds_free[2], p_full[2], p_free[2], pp_ready, pp_free;
    __shared__ uint64_t o_full[2], o_free[2], sb_ready, sb_free;
    __shared__ UnitInfo units[2];
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;
#ifdef SALA_TRACE
    unsigned tr_i = 0;   // events written by this thread (one tracing thread per role)
#endif

    const ChunkArgs &a = f.c;
    const int H = a.H;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    ChunkMeta *meta = reinterpret_cast<ChunkMeta *>(sm + kMeta);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            tc::mbar_init(&full[s], 33);   // expect_tx arrival + one per producer lane
            tc::mbar_init(&empty[s], 3);   // warpgroup 0, warpgroup 1, MMA commit
        }
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(&unit_full[i], 1);
            tc::mbar_init(&unit_empty[i], 4);
            tc::mbar_init(&ds_full[i], 1);
            tc::mbar_init(&ds_free[i], 2);
            tc::mbar_init(&p_full[i], 1);
            tc::mbar_init(&p_free[i], 1);

            tc::mbar_init(&o_full[i], 1);
            tc::mbar_init(&o_free[i], 1);

        }
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(&kp_ready[i], 1);
            tc::mbar_init(&kp_free[i], 1);
        }
        tc::mbar_init(&pub_ready, 2);
        tc::mbar_init(&pp_ready, 1);
        tc::mbar_init(&pp_free, 1);
        tc::mbar_init(&sb_ready, 2);
        tc::mbar_init(&sb_free, 1);
        tc::mbar_init(&drain, 1);
        abort_flag = 0;
        tc::fence_barrier_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(&tmem_slot, kTCols);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = tmem_slot;
    volatile int *abort_v = &abort_flag;
    const bool table_ok = t.seg_off[t.nseq + 1] == 1;
    const int64_t total_units = table_ok ? t.seg_off[t.nseq] * H : 0;

    if (warp == 0) {
        // =============================== producer ===============================
        const uint64_t keep = tc::policy_evict_last(), drop = tc::policy_evict_first();
        if (lane == 0) {
            tc::tma_prefetch_desc(&maps.q);
            tc::tma_prefetch_desc(&maps.k);
            tc::tma_prefetch_desc(&maps.v);
        }
        uint32_t job = 0, us = 0;
        bool ok = true;
        auto load_job = [&](int64_t c0, int nv, int h, bool with_q) -> bool {
            const uint32_t st = job % kStages;
            bool bad = false;
            if (job >= kStages)
                bad = !wait_or_abort(&empty[st], ((job / kStages) - 1) & 1, abort_v, status);
            if (__any_sync(0xffffffffu, bad)) return false;
            uint8_t *base = sm + st * kStage;
            if (lane == 0) {
                TRACE(0, with_q ? 2 : 1, job);
                const int32_t x0 = static_cast<int32_t>(c0);
                tc::mbar_arrive_expect_tx(&full[st], (with_q ? 3 : 2) * kTile);
                if (with_q) {
                    tc::tma_load_3d_hint(base, &maps.q, 0, h, x0, &full[st], drop);
                    tc::tma_load_3d_hint(base + kRegion, &maps.q, 64, h, x0, &full[st], drop);
                }
                const uint64_t pol = with_q ? drop : keep;
                tc::tma_load_3d_hint(base + kTile, &maps.k, 0, h, x0, &full[st], pol);
                tc::tma_load_3d_hint(base + kTile + kRegion, &maps.k, 64, h, x0, &full[st], pol);
                tc::tma_load_3d_hint(base + 2 * kTile, &maps.v, 0, h, x0, &full[st], pol);
                tc::tma_load_3d_hint(base + 2 * kTile + kRegion, &maps.v, 64, h, x0, &full[st], pol);
            }
            // the chunk's log-decays: inclusive prefix sums, last value, factored-route check
            const int i0 = 2 * lane, i1 = 2 * lane + 1;
            const float g0 = i0 < nv ? a.g[(c0 + i0) * H + h] : 0.f;
            const float g1 = i1 < nv ? a.g[(c0 + i1) * H + h] : 0.f;
            const float pair = g0 + g1;
            float run = pair;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, run, off);
                if (lane >= off) run += y;
            }
            const float b0 = run - pair + g0, b1 = run;
            float mx = fmaxf(fabsf(b0), fabsf(b1));
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
            const float bC = __shfl_sync(0xffffffffu, ((nv - 1) & 1) ? b1 : b0, (nv - 1) >> 1);
            ChunkMeta &md = meta[st];
            *reinterpret_cast<float2 *>(&md.b[i0]) = make_float2(b0, b1);
            if (lane == 0) {
                md.bC = bC;
                md.fast = mx <= kFastRange ? 1 : 0;
                md.nv = nv;
            }
            tc::mbar_arrive(&full[st]);
            ++job;
            return true;
        };
        while (ok) {
            const uint32_t slot = us & 1;
            bool bad = false;
            if (us >= 2) bad = !wait_or_abort(&unit_empty[slot], ((us >> 1) - 1) & 1, abort_v, status);
            if (__any_sync(0xffffffffu, bad)) break;
            uint32_t u = 0;
            if (lane == 0) u = atomicAdd(f.ticket, 1u);
            u = __shfl_sync(0xffffffffu, u, 0);
            UnitInfo info{};
            info.valid = 0;
            if (static_cast<int64_t>(u) < total_units) {
                info.sigma = u / H;
                info.h = static_cast<int>(u % H);
                if (locate_segment(t, info.sigma, info.n, info.t0, info.t1)) {
                    info.valid = 1;
                    info.nch = static_cast<int>((info.t1 - info.t0 + kChunk - 1) / kChunk);
                    info.first = info.t0 == seq_begin(t, info.n);
                    info.last = info.t1 == seq_begin(t, info.n + 1);
                }
            }
            if (lane == 0) {
                units[slot] = info;
                tc::mbar_arrive(&unit_full[slot]);
            }
            __syncwarp();
            if (!info.valid) break;
            for (int r = 0; r < info.nch && ok; ++r) {
                const int64_t c0 = info.t0 + int64_t(info.nch - 1 - r) * kChunk;
                ok = load_job(c0, static_cast<int>(min(int64_t(kChunk), info.t1 - c0)), info.h, false);
            }
            for (int c = 0; c < info.nch && ok; ++c) {
                const int64_t c0 = info.t0 + int64_t(c) * kChunk;
                ok = load_job(c0, static_cast<int>(min(int64_t(kChunk), info.t1 - c0)), info.h, true);
            }
            ++us;
        }
        // drain: the copies of the last stages must land before the CTA may exit
        if (lane == 0)
            for (uint32_t j = job > kStages ? job - kStages : 0; j < job; ++j)
                tc::mbar_wait(&full[j % kStages], (j / kStages) & 1, kWaitNs);
    } else if (warp == 1) {
        // =============================== MMA issuer ===============================
        if (lane == 0) {
            const uint32_t sb = tc::smem_u32(sm);
            uint32_t job = 0, us = 0, kpc = 0, dsc = 0, cc = 0, sbc = 0;
            auto W = [&](uint64_t *bar, uint32_t par) { return wait_or_abort(bar, par & 1, abort_v, status); };
            for (;;) {
                const uint32_t slot = us & 1;
                if (!W(&unit_full[slot], us >> 1)) break;
                const UnitInfo info = units[slot];
                tc::mbar_arrive(&unit_empty[slot]);
                if (!info.valid) break;
                bool ok = true;
                // ---- A: dS = sum over chunks of K'^T V, one accumulator
                const uint32_t dA = dsc & 1;
                if (dsc >= 2) ok = W(&ds_free[dA], (dsc >> 1) - 1);
                for (int r = 0; r < info.nch && ok; ++r) {
                    const uint32_t st = job % kStages;
                    const uint32_t kb = kpc & 1;
                    ok = W(&full[st], job / kStages) && W(&kp_ready[kb], kpc >> 1);
                    if (!ok) break;
                    ++kpc;
                    TRACE(1, 1, r);
                    tc::tc_fence_after();
                    const uint32_t v_s = sb + st * kStage + 2 * kTile;
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        tc::umma_bf16(tmem + kTdS + 128 * dA, desc_mn8(sb + kKp + kb * kTile + ks * 2048),
                                      desc_mn8(v_s + ks * 2048), kIdescS, (r > 0 || ks > 0) ? 1u : 0u);
                    tc::umma_commit(&kp_free[kb]);
                    tc::umma_commit(&empty[st]);
                    ++job;
                }
                if (!ok) break;
                tc::umma_commit(&ds_full[dA]);
                ++dsc;
                // ---- C
                const uint32_t sb_base = sbc;
                for (int c = 0; c < info.nch && ok; ++c) {
                    const uint32_t st = job % kStages;
                    const uint32_t q_s = sb + st * kStage, k_s = q_s + kTile, v_s = q_s + 2 * kTile;
                    const uint32_t pb = cc & 1;
                    if (!W(&full[st], job / kStages)) { ok = false; break; }
                    const bool fast = meta[st].fast != 0;
                    // M1: P = Q K''^T (factored route) or Q K^T (exact route)
                    const uint32_t kb = kpc & 1;
                    if (!W(&kp_ready[kb], kpc >> 1)) { ok = false; break; }
                    ++kpc;
                    if (cc >= 2 && !W(&p_free[pb], (cc >> 1) - 1)) { ok = false; break; }
                    TRACE(1, 2, c);
                    tc::tc_fence_after();
                    const uint32_t kp_s = sb + kKp + kb * kTile;
                    const uint32_t kb_s = fast ? kp_s : k_s;
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const uint32_t off = (ks >> 2) * kRegion + (ks & 3) * 32;
                        tc::umma_bf16(tmem + kTP + 64 * pb, desc_k(q_s + off), desc_k(kb_s + off),
                                      kIdescP, ks > 0);
                    }
                    tc::umma_commit(&p_full[pb]);
                    // M4: dS = K''^T V or K'^T V
                    const uint32_t db = dsc & 1;
                    if (dsc >= 2 && !W(&ds_free[db], (dsc >> 1) - 1)) { ok = false; break; }
                    TRACE(1, 3, c);
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        tc::umma_bf16(tmem + kTdS + 128 * db, desc_mn8(kp_s + ks * 2048),
                                      desc_mn8(v_s + ks * 2048), kIdescS, ks > 0);
                    tc::umma_commit(&ds_full[db]);
                    tc::umma_commit(&kp_free[kb]);
                    ++dsc;
                    // M2: O^T = S^T Q^T (Q scaled in place first on the exact route)
                    const uint32_t sbu = sb_base + c;
                    if (!W(&sb_ready, sbu)) { ok = false; break; }
                    if (cc >= 2 && !W(&o_free[pb], (cc >> 1) - 1)) { ok = false; break; }
                    if (!fast && !W(&pp_ready, cc)) { ok = false; break; }
                    TRACE(1, 4, c);
                    tc::tc_fence_after();
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const uint32_t b_off = (ks >> 2) * kRegion + (ks & 3) * 32;
                        tc::umma_bf16(tmem + kTO + 64 * pb, desc_mn16(sb + kSb + ks * 2048),
                                      desc_k(q_s + b_off), kIdescO, ks > 0);
                    }
                    tc::umma_commit(&sb_free);
                    // M3: O^T += V^T P'^T
                    if (fast && !W(&pp_ready, cc)) { ok = false; break; }
                    TRACE(1, 5, c);
                    tc::tc_fence_after();
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        tc::umma_bf16(tmem + kTO + 64 * pb, desc_mn8(v_s + ks * 2048),
                                      desc_k(sb + kPp + ks * 32), kIdescO, 1u);
                    tc::umma_commit(&o_full[pb]);
                    tc::umma_commit(&pp_free);
                    tc::umma_commit(&empty[st]);
                    ++job;
                    ++cc;
                }
                if (!ok) break;
                sbc += info.nch;
                ++us;
            }
            // no MMA may still run when the tensor memory is freed
            tc::umma_commit(&drain);
            tc::mbar_wait(&drain, 0, kWaitNs);
        }
    } else if (warp == 10) {
        // =============================== publisher ===============================
        if (lane == 0) {
            uint32_t us = 0, pc = 0;
            for (;;) {
                const uint32_t slot = us & 1;
                if (!wait_or_abort(&unit_full[slot], (us >> 1) & 1, abort_v, status)) break;
                const UnitInfo info = units[slot];
                tc::mbar_arrive(&unit_empty[slot]);
                if (!info.valid) break;
                if (!info.last) {
                    if (!wait_or_abort(&pub_ready, (pc++) & 1, abort_v, status)) break;
                    __threadfence();
                    tc::st_release_gpu(f.flags + info.sigma * H + info.h, f.epoch);
                }
                ++us;
            }
        }
    } else {
        // =============================== epilogue warpgroups ===============================
        // Waits inside a chunk do not vote: a thread whose wait gives up has set the abort
        // flag, and every later wait returns at once, so all threads still pass the same
        // barriers; one OR-vote per chunk (and per hand-off) then ends the loop uniformly.
        const int wg = (warp - 2) >> 2;
        const int wtid = threadIdx.x - 64 - 128 * wg;
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;   // state row i / value column j
        const int bar_id = 1 + wg;
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        const int jc0 = 64 * wg;
        float *vals = reinterpret_cast<float *>(sm + kVals) + 64 * wg;
        uint32_t job = 0, us = 0, kpc = 0, dsc = 0, cc = 0, sbc = 0;
        float S[64];

        // K' for one chunk (warpgroup 0): factors exp(base - b_t) into K' buffer kpc & 1
        auto make_kprime = [&](uint32_t st, float base) {
            const uint32_t kb = kpc & 1;
            wait_nv(&kp_free[kb], (kpc >> 1) - 1, kpc >= 2, abort_v, status);
            if (wtid == 0) TRACE(2, 20, kpc);
            const ChunkMeta &m = meta[st];
            scale_rows<8>(sm + st * kStage + kTile, sm + kKp + kb * kTile, wtid, 128, m.nv, m.b,
                          base * kLog2e, -1.f);
            if (wtid == 0) TRACE(2, 21, kpc);
            tc::fence_proxy_async_smem();
            named_sync(bar_id, 128);
            if (wtid == 0) TRACE(2, 22, kpc);
            if (wtid == 0) tc::mbar_arrive(&kp_ready[kb]);
            ++kpc;
        };

        for (;;) {
            const uint32_t slot = us & 1;
            if (!wg_wait(&unit_full[slot], us >> 1, true, bar_id, abort_v, status)) break;
            const UnitInfo info = units[slot];
            named_sync(bar_id, 128);
            if (wtid == 0) tc::mbar_arrive(&unit_empty[slot]);
            if (!info.valid) break;
            const int h = info.h;

            // ---------------- A: K' = K exp(B_end - B_t) (warpgroup 0) ----------------
            float D = 0.f;   // total log-decay of the chunks already visited (the later ones)
            for (int r = 0; r < info.nch; ++r) {
                const uint32_t st = job % kStages;
                wait_nv(&full[st], job / kStages, true, abort_v, status);
                const float bC = meta[st].bC;
                if (wtid == 0) TRACE(2 + wg, 1, r);
                if (wg == 0) {
                    make_kprime(st, bC + D);
                    if (wtid == 0) tc::mbar_arrive(&empty[st]);
                } else {
                    named_sync(bar_id, 128);   // every thread has read this stage's metadata
                    if (wtid == 0) tc::mbar_arrive(&empty[st]);
                }
                D += bC;
                ++job;
            }

            // ---------------- hand-off: S_in, publish S_out, bf16 S_in for M2 ----------------
            {
                const uint32_t db = dsc & 1;
                bool bad = !wait_or_abort(&ds_full[db], (dsc >> 1) & 1, abort_v, status);
                ++dsc;
                if (!bad && !info.first && wtid == 0) {
                    const uint32_t *flag = f.flags + (info.sigma - 1) * H + h;
                    const uint64_t t0ns = tc::global_timer_ns();
                    while (tc::ld_acquire_gpu(flag) != f.epoch) {
                        if (*abort_v) { bad = true; break; }
                        if (tc::global_timer_ns() - t0ns > kWaitNs) {
                            *abort_v = 1;
                            record_status(status, SALA_ERR_TIMEOUT);
                            bad = true;
                            break;
                        }
                    }
                }
                if (named_any(bar_id, 128, bad || *abort_v)) break;
                if (wtid == 0) TRACE(2 + wg, 2, 0);
                tc::tc_fence_after();
                if (info.first) {
                    if (f.h0) {
                        const float *src = f.h0 + ((info.n * H + h) * kD + row) * kD + jc0;
#pragma unroll
                        for (int j = 0; j < 64; j += 4) {
                            const float4 x = *reinterpret_cast<const float4 *>(src + j);
                            S[j] = x.x; S[j + 1] = x.y; S[j + 2] = x.z; S[j + 3] = x.w;
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < 64; ++j) S[j] = 0.f;
                    }
                } else {
                    const float *src = f.incl + (static_cast<size_t>(info.sigma - 1) * H + h) * kD * kD +
                                       row * kD + jc0;
#pragma unroll
                    for (int j = 0; j < 64; j += 4) {
                        const float4 x = __ldcg(reinterpret_cast<const float4 *>(src + j));
                        S[j] = x.x; S[j + 1] = x.y; S[j + 2] = x.z; S[j + 3] = x.w;
                    }
                }
                const float eB = tc::ex2(D * kLog2e);
                float *dst = info.last ? (f.hT ? f.hT + ((info.n * H + h) * kD + row) * kD + jc0 : nullptr)
                                       : f.incl + (static_cast<size_t>(info.sigma) * H + h) * kD * kD +
                                             row * kD + jc0;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t d[32];
                    tc::tmem_ld_32x32b_x32(tmem + lane_base + kTdS + 128 * db + jc0 + 32 * half, d);
                    tc::tmem_ld_wait();
                    if (dst) {
#pragma unroll
                        for (int j = 0; j < 32; j += 4)
                            *reinterpret_cast<float4 *>(dst + 32 * half + j) = make_float4(
                                fmaf(eB, S[32 * half + j], __uint_as_float(d[j])),
                                fmaf(eB, S[32 * half + j + 1], __uint_as_float(d[j + 1])),
                                fmaf(eB, S[32 * half + j + 2], __uint_as_float(d[j + 2])),
                                fmaf(eB, S[32 * half + j + 3], __uint_as_float(d[j + 3])));
                    }
                }
                tc::tc_fence_before();
                named_sync(bar_id, 128);
                if (wtid == 0) {
                    tc::mbar_arrive(&ds_free[db]);
                    if (!info.last) tc::mbar_arrive(&pub_ready);   // publisher fences and flags
                }
                // bf16 S_in for the first chunk's M2
                wait_nv(&sb_free, sbc - 1, sbc >= 1, abort_v, status);
                store_bf16_row64(sm + kSb + wg * kSRegion, row, S);
                tc::fence_proxy_async_smem();
                named_sync(bar_id, 128);
                if (wtid == 0) tc::mbar_arrive(&sb_ready);
                ++sbc;
                if (wtid == 0) TRACE(2 + wg, 3, 0);
            }

            // ---------------- C ----------------
            if (wg == 0) {
                // K'' of chunk 0 (warpgroup 0 stays one chunk ahead)
                const uint32_t st = job % kStages;
                wait_nv(&full[st], job / kStages, true, abort_v, status);
                make_kprime(st, meta[st].fast ? 0.f : meta[st].bC);
            }
            bool ok = true;
            for (int c = 0; c < info.nch; ++c) {
                const uint32_t st = job % kStages;
                const uint32_t pb = cc & 1;
                const int64_t c0 = info.t0 + int64_t(c) * kChunk;
                wait_nv(&full[st], job / kStages, true, abort_v, status);
                const ChunkMeta &md = meta[st];
                const int nv = md.nv;
                const bool fast = md.fast != 0;
                const float eC = tc::ex2(md.bC * kLog2e);
                if (wtid == 0) TRACE(2 + wg, 4, c);

                if (wg == 0) {
                    // (a) K'' of the next chunk: exp(-b_s) (factored) or exp(b_C - b_s) (exact)
                    if (c + 1 < info.nch) {
                        const uint32_t sn = (job + 1) % kStages;
                        wait_nv(&full[sn], (job + 1) / kStages, true, abort_v, status);
                        make_kprime(sn, meta[sn].fast ? 0.f : meta[sn].bC);
                    }
                    // (b) scores -> P' (bf16, K-major rows t)
                    wait_nv(&p_full[pb], cc >> 1, true, abort_v, status);
                    wait_nv(&pp_free, cc - 1, cc >= 1, abort_v, status);
                    if (wtid == 0) TRACE(2, 5, c);
                    tc::tc_fence_after();
                    // M=64 accumulator layout: row t = 16 * quarter + lane in lanes 0-15
                    const int tr = quarter * 16 + (lane & 15);
                    const float bt = md.b[tr] * kLog2e;
                    uint8_t *pp = sm + kPp;
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        uint32_t p[32];
                        tc::tmem_ld_32x32b_x32(tmem + lane_base + kTP + 64 * pb + 32 * half, p);
                        tc::tmem_ld_wait();
                        if (wtid == 0) TRACE(2, 23 + half, c);
                        if (half == 1) {
                            tc::tc_fence_before();
                            named_sync(bar_id, 128);
                            if (wtid == 0) tc::mbar_arrive(&p_free[pb]);
                            if (wtid == 0) TRACE(2, 25, c);
                        }
                        if (lane < 16) {
                            uint32_t w[16];
#pragma unroll
                            for (int e = 0; e < 32; e += 2) {
                                const int sc = 32 * half + e;
                                float f0 = __uint_as_float(p[e]), f1 = __uint_as_float(p[e + 1]);
                                if (!fast) {
                                    f0 *= tc::ex2(bt - md.b[sc] * kLog2e);
                                    f1 *= tc::ex2(bt - md.b[sc + 1] * kLog2e);
                                }
                                w[e >> 1] = float2_to_bf16x2(sc <= tr ? f0 : 0.f, sc + 1 <= tr ? f1 : 0.f);
                            }
#pragma unroll
                            for (int c8 = 0; c8 < 4; ++c8)
                                *reinterpret_cast<uint4 *>(pp + sw(tr, 4 * half + c8)) =
                                    make_uint4(w[4 * c8], w[4 * c8 + 1], w[4 * c8 + 2], w[4 * c8 + 3]);
                        }
                    }
                    if (wtid == 0) TRACE(2, 26, c);
                    if (!fast) {
                        // exact route: q_t <- exp(b_t) q_t in place (M1 has read Q already)
                        uint8_t *qt = sm + st * kStage;
                        scale_rows<8>(qt, qt, wtid, 128, nv, md.b, 0.f, 1.f);
                    }
                    tc::fence_proxy_async_smem();
                    named_sync(bar_id, 128);
                    if (wtid == 0) {
                        tc::mbar_arrive(&pp_ready);
                        tc::mbar_arrive(&empty[st]);
                        TRACE(2, 6, c);
                    }
                } else {
                    // output row factors for (d), then release the stage
                    if (wtid < 64) vals[wtid] = fast ? a.scale * tc::ex2(md.b[wtid] * kLog2e) : a.scale;
                    named_sync(bar_id, 128);
                    if (wtid == 0) tc::mbar_arrive(&empty[st]);
                }

                // (c) state carry for my 64 columns; bf16 copy for the next chunk's M2
                {
                    const uint32_t db = dsc & 1;
                    wait_nv(&ds_full[db], dsc >> 1, true, abort_v, status);
                    ++dsc;
                    if (wtid == 0) TRACE(2 + wg, 7, c);
                    tc::tc_fence_after();
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        uint32_t d[32];
                        tc::tmem_ld_32x32b_x32(tmem + lane_base + kTdS + 128 * db + jc0 + 32 * half, d);
                        tc::tmem_ld_wait();
                        if (fast) {
#pragma unroll
                            for (int j = 0; j < 32; ++j) S[32 * half + j] = eC * (S[32 * half + j] + __uint_as_float(d[j]));
                        } else {
#pragma unroll
                            for (int j = 0; j < 32; ++j) S[32 * half + j] = fmaf(eC, S[32 * half + j], __uint_as_float(d[j]));
                        }
                    }
                    if (wtid == 0 && wg == 0) TRACE(2, 27, c);
                    tc::tc_fence_before();
                    named_sync(bar_id, 128);
                    if (wtid == 0 && wg == 0) TRACE(2, 28, c);
                    if (wtid == 0) tc::mbar_arrive(&ds_free[db]);
                    if (c + 1 < info.nch) {
                        wait_nv(&sb_free, sbc - 1, sbc >= 1, abort_v, status);
                        if (wtid == 0 && wg == 0) TRACE(2, 29, c);
                        store_bf16_row64(sm + kSb + wg * kSRegion, row, S);
                        if (wtid == 0 && wg == 0) TRACE(2, 30, c);
                        tc::fence_proxy_async_smem();
                        named_sync(bar_id, 128);
                        if (wtid == 0) tc::mbar_arrive(&sb_ready);
                        ++sbc;
                    }
                    if (wtid == 0) TRACE(2 + wg, 8, c);
                }

                if (wg == 1) {
                    // (d) o_t = factor_t * O[t] for value column j = row; stage, store
                    wait_nv(&o_full[pb], cc >> 1, true, abort_v, status);
                    if (wtid == 0) TRACE(3, 9, c);
                    tc::tc_fence_after();
                    uint16_t *orow = a.o + (c0 * H + h) * kD + row;   // column j = row of o[c0 + t, h, :]
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        uint32_t o[32];
                        tc::tmem_ld_32x32b_x32(tmem + lane_base + kTO + 64 * pb + 32 * half, o);
                        tc::tmem_ld_wait();
                        if (half == 1) {
                            tc::tc_fence_before();
                            named_sync(bar_id, 128);
                            if (wtid == 0) tc::mbar_arrive(&o_free[pb]);
                        }
#pragma unroll
                        for (int tt = 0; tt < 32; ++tt) {
                            const int t = 32 * half + tt;
                            if (t < nv)
                                orow[static_cast<size_t>(t) * H * kD] =
                                    __bfloat16_as_ushort(__float2bfloat16_rn(vals[t] * __uint_as_float(o[tt])));
                        }
                    }
                    if (wtid == 0) TRACE(3, 10, c);
                }
                ++cc;
                ++job;
                // one uniform decision per chunk (also orders the staging buffer's reuse)
                if (named_any(bar_id, 128, *abort_v != 0)) { ok = false; break; }
            }
            if (!ok) break;
            ++us;
        }
    }

    tc::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, kTCols);
    }
}

// ---------------------------------------------------------------------------------------
// hT of empty sequences: the initial state (or zeros). One block per (sequence, head).
__global__ void __launch_bounds__(256)
empty_seq_state_kernel(SegTable t, int H, const float *__restrict__ h0, float *__restrict__ hT) {
    if (t.seg_off[t.nseq + 1] != 1) return;
    const int64_t nh = blockIdx.x;
    const int64_t n = nh / H;
    if (seq_begin(t, n + 1) != seq_begin(t, n)) return;
    float4 *dst = reinterpret_cast<float4 *>(hT + nh * kD * kD);
    const float4 *src = h0 ? reinterpret_cast<const float4 *>(h0 + nh * kD * kD) : nullptr;
    for (int i = threadIdx.x; i < kD * kD / 4; i += blockDim.x)
        dst[i] = src ? src[i] : make_float4(0.f, 0.f, 0.f, 0.f);
}

// ---------------------------------------------------------------------------------------
// host side

namespace tck {

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
}  // namespace

cudaError_t make_maps(TcMaps *m, const void *q, const void *k, const void *v, int64_t T_total,
                      int H) {
    cudaError_t e = encode_map(&m->q, q, T_total, H);
    if (e == cudaSuccess) e = encode_map(&m->k, k, T_total, H);
    if (e == cudaSuccess) e = encode_map(&m->v, v, T_total, H);
    return e;
}

}  // namespace tck

cudaError_t setup_fused_kernel() {
    return cudaFuncSetAttribute(prefill_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(kSmemAlloc));
}

cudaError_t launch_prefill_fused(const ChunkArgs &a, const SegTable &t, int64_t T_total,
                                 int64_t max_units, const float *h0, float *hT, float *incl,
                                 uint32_t *flags, uint32_t *ticket, uint32_t epoch, int grid,
                                 int *status, cudaStream_t st) {
    if (T_total > 0 && max_units > 0) {
        tck::TcMaps maps;
        cudaError_t e = tck::make_maps(&maps, a.q, a.k, a.v, T_total, a.H);
        if (e != cudaSuccess) return e;
        FusedArgs f;
        f.c = a;
        f.h0 = h0;
        f.hT = hT;
        f.incl = incl;
        f.flags = flags;
        f.ticket = ticket;
        f.epoch = epoch;
        if (grid > max_units) grid = static_cast<int>(max_units);
        LaunchTimer timer(kKPrefillFused, st);
        prefill_fused_kernel<<<grid, kThreads, kSmemAlloc, st>>>(maps, f, t, status);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (hT && t.nseq > 0) {
        const int64_t blocks = t.nseq * a.H;
        LaunchTimer timer(kKEmptySeq, st);
        empty_seq_state_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(t, a.H, h0, hT);
        return cudaGetLastError();
    }
    return cudaSuccess;
}

}  // namespace sala

#ifdef SALA_TRACE
extern "C" int sala_gla_debug_trace(unsigned long long *out, int max) {
    unsigned int n[4];
    if (cudaMemcpyFromSymbol(n, sala::g_trace_n, sizeof(n)) != cudaSuccess) return -1;
    static unsigned long long buf[4][sala::kTraceN];
    if (cudaMemcpyFromSymbol(buf, sala::g_trace, sizeof(buf)) != cudaSuccess) return -1;
    int k = 0;
    for (int r = 0; r < 4; ++r)
        for (unsigned i = 0; i < n[r] && i < static_cast<unsigned>(sala::kTraceN) && k < max; ++i)
            out[k++] = buf[r][i];
    return k;
}
#endif
