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
//     k_t^T v_t accumulated by tcgen05 in tensor memory (k_t scaled by its decay to the
//     segment end, so every weight is <= 1), and the total log-decay B;
//  hand-off: S_in = h0 (first segment) or the state the predecessor published; publish
//     S_out = exp(B) S_in + dS for the successor (hT for the last segment). This is the
//     Blueprint's unrolled form S_n = alpha^n S_0 + sum alpha^(n-i) k_i^T v_i applied a whole
//     segment at a time;
//  C. output pass over the chunks, first to last, from S_in. With b_t the cumulative
//     log-decay of the chunk up to token t and S the state entering the chunk:
//       o_t = scale exp(b_t) [ q_t S + sum_{s<=t} (q_t . k_s) exp(-b_s) v_s ]
//       S  <- exp(b_C) [ S + sum_s exp(-b_s) k_s^T v_s ]
//     which keeps both output terms in one accumulator (the weights become per-column
//     factors exp(-b_s) on the scores and per-row factors exp(b_t) on the output). When a
//     chunk's decay range is too wide for those factors (|b_t| > 60), the chunk takes the
//     exact route instead: per-entry factors exp(b_t - b_s) on the scores, q_t scaled by
//     exp(b_t) in place, and S <- exp(b_C) S + sum_s exp(b_C - b_s) k_s^T v_s.
//
// The state is kept transposed (S^T, value index j in the tensor-memory lane), so that its
// bf16 copy can sit in tensor memory as the A operand of the q.S product. Contractions
// (tcgen05.mma kind::f16, bf16 in, fp32 accumulators in tensor memory):
//   M1  P    = Q K~^T      M=64  N=64  K=128   A=Q smem (K-major)     B=K~ smem (K-major)
//   M2  O^T  = S^T Q^T     M=128 N=64  K=128   A=S^T bf16 in TMEM     B=Q smem (K-major)
//   M3  O^T += V^T P'^T    M=128 N=64  K=64    A=V smem (MN-major)    B=P' smem (K-major)
//   M4  dS^T = V^T K~      M=128 N=128 K=64    A=V smem (MN-major)    B=K~ smem (MN-major)
// K~ is k scaled per token (the factors above). In the state pass the K tile arrives by TMA
// and is scaled in place in shared memory (the tensor core only runs the short M4 there). In
// the output pass, where the tensor core streams operands most of the time, the scaling
// warps make K~ from a global load straight into shared memory instead: ordinary
// shared-memory loads issued while the tensor core reads its operands stall far behind them.
// Q and V tiles arrive by TMA, o leaves by TMA stores.
//
// Roles: warp 0 loads (TMA), warp 1 issues MMAs and owns the tensor memory, warps 4-7 scale K,
// turn scores into P' and (exact route) scale Q, warps 8-11 and 12-15 each own 64 of the
// state's key rows i (all 128 value columns j, one per lane), carry the state, publish the
// hand-off flag and write o for 32 of the chunk's tokens. Every per-token factor is computed
// by the warp that needs it from g (an in-warp prefix sum), never passed through shared
// memory. mbarrier waits compare phase parity only, so every barrier has at most one phase
// in flight per waiter: each waiter consumes every phase of the barriers it waits on, and a
// producer cannot complete a second phase before its consumer has consumed the first.
// Every wait is bounded (2 s of %globaltimer); a timeout records SALA_ERR_TIMEOUT, stops the
// CTA's work, drains its copies and MMAs, frees its tensor memory and returns.
#include "chunk_tc.cuh"

namespace sala {
namespace {

using namespace tck;

constexpr int kStages = 4;
constexpr int kThreads = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kFastRange = 60.f;   // max |b_t| (natural log) for the factored route

// dynamic shared memory (offsets from a 1024-aligned base)
constexpr uint32_t kStage = 2 * kTile;              // Q | V
constexpr uint32_t kKp = kStages * kStage;          // K~ [2] (factored or exact weights)
constexpr uint32_t kKr = kKp + 2 * kTile;           // raw K [2] (exact-route M1)
constexpr uint32_t kPp = kKr + 2 * kTile;           // P' [2] (K-major B of M3)
constexpr uint32_t kOst = kPp + 2 * kRegion;        // o staging [2 state groups][32 t][256 B]
constexpr uint32_t kOstBytes = 32 * 256;
constexpr uint32_t kBytes = kOst + 2 * kOstBytes;
constexpr uint32_t kSmemAlloc = kBytes + 1024;

// TMEM columns: P (M=64 layout), S^T bf16 (A of M2), O^T [2], dS^T [2]
constexpr uint32_t kTP = 0, kTSb = 64, kTO = 128, kTdS = 256, kTCols = 512;
constexpr uint32_t kIdescP = tc::idesc_bf16_f32(64, 64, 0, 0);
constexpr uint32_t kIdescO2 = tc::idesc_bf16_f32(128, 64, 0, 0);
constexpr uint32_t kIdescO3 = tc::idesc_bf16_f32(128, 64, 1, 0);
constexpr uint32_t kIdescS = tc::idesc_bf16_f32(128, 128, 1, 1);

struct FusedArgs {
    ChunkArgs c;            // q, k, v, g, scale, o, H
    const float *h0;        // [nseq, H, 128, 128] or null
    float *hT;              // [nseq, H, 128, 128] or null
    float *incl;            // [units, 128, 128]: S_out of each (segment, head), row-major like hT
    uint32_t *flags;        // [units]: == epoch once incl of that unit is published
    uint32_t *ticket;       // work counter, zeroed by the table kernel
    uint32_t epoch;
};

struct UnitInfo {
    int valid, h, nch, first, last;
    int64_t sigma, n, t0, t1;
};

// Event trace of CTA 0 for latency analysis (compiled only with -DSALA_TRACE): SM clock,
// role, event id and chunk index, written to a global array.
#ifdef SALA_TRACE
constexpr int kTraceN = 512;
__device__ unsigned long long g_trace[5][kTraceN];
__device__ unsigned int g_trace_n[5];
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

// Log-decays of one chunk as seen by one warp: lane l holds the inclusive prefix sums
// b[2l], b[2l+1] of g over the chunk's nv valid tokens (constant past nv).
struct Gate {
    float b0, b1;   // b[2 lane], b[2 lane + 1]
    float bC;       // b at the last valid token
    bool fast;      // max |b| <= kFastRange: factored weights are safe
};

// Raw g of the chunk for lane l (tokens 2l, 2l+1; 0 past nv): loaded early, scanned later.
__device__ __forceinline__ float2 load_gate(const float *__restrict__ g, int64_t c0, int nv, int H,
                                            int h) {
    const int l = threadIdx.x & 31;
    return make_float2(2 * l < nv ? __ldg(g + (c0 + 2 * l) * H + h) : 0.f,
                       2 * l + 1 < nv ? __ldg(g + (c0 + 2 * l + 1) * H + h) : 0.f);
}

__device__ __forceinline__ Gate scan_gate(float2 a, int nv) {
    const int l = threadIdx.x & 31;
    const float pair = a.x + a.y;
    float run = pair;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, run, off);
        if (l >= off) run += y;
    }
    Gate G;
    G.b0 = run - pair + a.x;
    G.b1 = run;
    float mx = fmaxf(fabsf(G.b0), fabsf(G.b1));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    G.bC = __shfl_sync(0xffffffffu, ((nv - 1) & 1) ? G.b1 : G.b0, (nv - 1) >> 1);
    G.fast = mx <= kFastRange;
    return G;
}

// b[t] for a warp-uniform or per-lane t in [0, 64) (all lanes must call).
__device__ __forceinline__ float gate_at(const Gate &G, int t) {
    const float x = __shfl_sync(0xffffffffu, G.b0, t >> 1);
    const float y = __shfl_sync(0xffffffffu, G.b1, t >> 1);
    return (t & 1) ? y : x;
}

// Bounded wait (if `need`) whose failure only sets the abort flag (see the epilogue loops).
__device__ __forceinline__ void wait_nv(uint64_t *bar, uint32_t par, bool need,
                                        volatile int *abort_v, int *status) {
    if (need) (void)wait_or_abort(bar, par & 1, abort_v, status);
}

// Bounded wait on an mbarrier phase by every thread of a group of n threads (if `need`),
// then an OR-vote so that all of them take the same branch. Returns false if any failed.
__device__ __forceinline__ bool wg_wait(uint64_t *bar, uint32_t par, bool need, int bar_id,
                                        volatile int *abort_v, int *status, int n = 128) {
    const bool bad = need ? !wait_or_abort(bar, par & 1, abort_v, status) : false;
    return !named_any(bar_id, n, bad);
}

// 64 bf16 of one row, scaled by f, to a [64 x 128 B] SW128 region row (and, if raw_dst, also
// unscaled to a second tile). kExact: product in fp32, rounded once; otherwise f is rounded to
// bf16 and each pair takes one packed multiply (about 5x fewer instructions, one more
// rounding of the factor: used for the output pass, whose tolerance has more room).
template <bool kExact>
__device__ __forceinline__ void store_row_scaled(uint8_t *dst, uint8_t *raw_dst, int row,
                                                 const uint4 (&x)[8], float f) {
    const __nv_bfloat162 f2 = __float2bfloat162_rn(f);
#pragma unroll
    for (int c8 = 0; c8 < 8; ++c8) {
        uint4 y;
        if constexpr (kExact) {
            y.x = mul_bf16x2(x[c8].x, f);
            y.y = mul_bf16x2(x[c8].y, f);
            y.z = mul_bf16x2(x[c8].z, f);
            y.w = mul_bf16x2(x[c8].w, f);
        } else {
            y.x = mul_bf16x2(x[c8].x, f2);
            y.y = mul_bf16x2(x[c8].y, f2);
            y.z = mul_bf16x2(x[c8].z, f2);
            y.w = mul_bf16x2(x[c8].w, f2);
        }
        *reinterpret_cast<uint4 *>(dst + sw(row, c8)) = y;
        if (raw_dst) *reinterpret_cast<uint4 *>(raw_dst + sw(row, c8)) = x[c8];
    }
}

}  // namespace

__global__ void __launch_bounds__(kThreads, 1)
prefill_fused_kernel(const __grid_constant__ TcMaps maps, FusedArgs f, SegTable t, int *status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
    __shared__ uint64_t full[kStages], empty[kStages], unit_full[2], unit_empty[2];
    __shared__ uint64_t kp_ready[2], kp_free[2], ka_ready[kStages], drain;
    __shared__ uint64_t ds_full[2], ds_free[2], p_full, p_free, pp_ready[2], pp_free[2];
    __shared__ uint64_t o_full[2], o_free[2], sb_ready, sb_free;
    __shared__ uint64_t d_ready, d_free;
    __shared__ UnitInfo units[2];
    __shared__ int kfast[2];
    __shared__ float unit_D;   // total log-decay of the current unit's segment
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;
#ifdef SALA_TRACE
    unsigned tr_i = 0;   // events written by this thread (one tracing thread per role)
#endif

    const ChunkArgs &a = f.c;
    const int H = a.H;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            tc::mbar_init(&full[s], 1);    // expect_tx arrival
            tc::mbar_init(&empty[s], 1);   // MMA commit
        }
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(&unit_full[i], 1);
            tc::mbar_init(&unit_empty[i], 4);   // MMA, scaler, two state groups
            tc::mbar_init(&kp_ready[i], 1);
            tc::mbar_init(&kp_free[i], 1);
            tc::mbar_init(&ds_full[i], 1);
            tc::mbar_init(&ds_free[i], 2);
            tc::mbar_init(&o_full[i], 1);
            tc::mbar_init(&o_free[i], 2);
        }
        tc::mbar_init(&p_full, 1);
        tc::mbar_init(&p_free, 1);
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(&pp_ready[i], 1);
            tc::mbar_init(&pp_free[i], 1);
        }
        tc::mbar_init(&sb_ready, 2);
        tc::mbar_init(&sb_free, 1);
        tc::mbar_init(&drain, 1);
        for (int s = 0; s < kStages; ++s)
            tc::mbar_init(&ka_ready[s], 1);   // the state-pass K' tile of this stage is scaled
                                              // (phases count this stage's state-pass jobs)
        tc::mbar_init(&d_ready, 1);
        tc::mbar_init(&d_free, 2);      // both state groups have read unit_D
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
            tc::tma_prefetch_desc(&maps.o);
        }
        uint32_t job = 0, us = 0;
        bool ok = true;
        // one job: K and V (state pass; K goes to the first tile of the stage) or Q and V
        // (output pass) of the chunk at token c0, with L2 prefetches of the chunk's log-decays
        // (read by other warps a little later)
        auto load_job = [&](int64_t c0, int nv, int h, bool with_q) -> bool {
            const uint32_t st = job % kStages;
            bool bad = false;
            if (job >= kStages)
                bad = !wait_or_abort(&empty[st], ((job / kStages) - 1) & 1, abort_v, status);
            if (__any_sync(0xffffffffu, bad)) return false;
            if (2 * lane < nv) tc::prefetch_l2_keep(a.g + (c0 + 2 * lane) * H + h);
            if (2 * lane + 1 < nv) tc::prefetch_l2_keep(a.g + (c0 + 2 * lane + 1) * H + h);
            if (lane == 0) {
                TRACE(0, with_q ? 2 : 1, job);
                uint8_t *base = sm + st * kStage;
                const int32_t x0 = static_cast<int32_t>(c0);
                tc::mbar_arrive_expect_tx(&full[st], 2 * kTile);
                const CUtensorMap *first = with_q ? &maps.q : &maps.k;
                tc::tma_load_3d_hint(base, first, 0, h, x0, &full[st], with_q ? drop : keep);
                tc::tma_load_3d_hint(base + kRegion, first, 64, h, x0, &full[st], with_q ? drop : keep);
                const uint64_t pol = with_q ? drop : keep;
                tc::tma_load_3d_hint(base + kTile, &maps.v, 0, h, x0, &full[st], pol);
                tc::tma_load_3d_hint(base + kTile + kRegion, &maps.v, 64, h, x0, &full[st], pol);
                // the scaling warps read this chunk's K rows with ordinary loads a little later
                tc::tma_prefetch_l2_3d(&maps.k, 0, h, x0, pol);
                tc::tma_prefetch_l2_3d(&maps.k, 64, h, x0, pol);
            }
            __syncwarp();
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
            uint32_t ka_par = 0;   // bit st: phase parity of ka_ready[st] (state-pass jobs only)
            auto W = [&](uint64_t *bar, uint32_t par) { return wait_or_abort(bar, par & 1, abort_v, status); };
            for (;;) {
                const uint32_t slot = us & 1;
                if (!W(&unit_full[slot], us >> 1)) break;
                const UnitInfo info = units[slot];
                tc::mbar_arrive(&unit_empty[slot]);
                if (!info.valid) break;
                bool ok = true;
                // ---- A: dS^T = sum over chunks of V^T K', one accumulator
                const uint32_t dA = dsc & 1;
                if (dsc >= 2) ok = W(&ds_free[dA], (dsc >> 1) - 1);
                for (int r = 0; r < info.nch && ok; ++r) {
                    const uint32_t st = job % kStages;
                    ok = W(&full[st], job / kStages) && W(&ka_ready[st], (ka_par >> st) & 1);
                    if (!ok) break;
                    ka_par ^= 1u << st;
                    TRACE(1, 1, r);
                    tc::tc_fence_after();
                    const uint32_t k_s = sb + st * kStage, v_s = k_s + kTile;   // K' scaled in place
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        tc::umma_bf16(tmem + kTdS + 128 * dA, desc_mn8(v_s + ks * 2048),
                                      desc_mn8(k_s + ks * 2048), kIdescS, (r > 0 || ks > 0) ? 1u : 0u);
                    tc::umma_commit(&empty[st]);
                    ++job;
                }
                if (!ok) break;
                tc::umma_commit(&ds_full[dA]);
                ++dsc;
                // ---- C, software-pipelined: M1 of chunk c+1 goes out right after M2 of chunk c
                // (before M3 of chunk c), so the scores of c+1 are made while chunk c finishes
                const uint32_t sb_base = sbc;
                auto issue_m1 = [&](uint32_t q_s, uint32_t kb, bool fast) {
                    const uint32_t k1 = sb + (fast ? kKp : kKr) + kb * kTile;
                    tc::tc_fence_after();
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const uint32_t off = (ks >> 2) * kRegion + (ks & 3) * 32;
                        tc::umma_bf16(tmem + kTP, desc_k(q_s + off), desc_k(k1 + off), kIdescP, ks > 0);
                    }
                    tc::umma_commit(&p_full);
                };
                // M1 of chunk 0: P = Q K''^T (factored route) or Q K^T (exact route)
                uint32_t kb = kpc & 1;
                {
                    const uint32_t st = job % kStages;
                    ok = W(&full[st], job / kStages) && W(&kp_ready[kb], kpc >> 1) &&
                         (cc == 0 || W(&p_free, cc - 1));
                    if (ok) {
                        ++kpc;
                        TRACE(1, 2, 0);
                        issue_m1(sb + st * kStage, kb, kfast[kb] != 0);
                    }
                }
                for (int c = 0; c < info.nch && ok; ++c) {
                    const uint32_t st = job % kStages;
                    const uint32_t q_s = sb + st * kStage, v_s = q_s + kTile;
                    const uint32_t ob = cc & 1, pb = cc & 1;
                    const bool fast = kfast[kb] != 0;
                    // M4: dS^T = V^T K~ (not needed after the last chunk)
                    if (c + 1 < info.nch) {
                        const uint32_t db = dsc & 1;
                        if (dsc >= 2 && !W(&ds_free[db], (dsc >> 1) - 1)) { ok = false; break; }
                        TRACE(1, 3, c);
                        tc::tc_fence_after();
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks)
                            tc::umma_bf16(tmem + kTdS + 128 * db, desc_mn8(v_s + ks * 2048),
                                          desc_mn8(sb + kKp + kb * kTile + ks * 2048), kIdescS, ks > 0);
                        tc::umma_commit(&ds_full[db]);
                        ++dsc;
                    }
                    // M2: O^T = S^T Q^T (Q scaled in place first on the exact route)
                    if (!W(&sb_ready, sb_base + c)) { ok = false; break; }
                    if (cc >= 2 && !W(&o_free[ob], (cc >> 1) - 1)) { ok = false; break; }
                    if (!fast && !W(&pp_ready[pb], cc >> 1)) { ok = false; break; }
                    TRACE(1, 4, c);
                    tc::tc_fence_after();
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const uint32_t off = (ks >> 2) * kRegion + (ks & 3) * 32;
                        tc::umma_bf16_ta(tmem + kTO + 64 * ob, tmem + kTSb + 8 * ks, desc_k(q_s + off),
                                         kIdescO2, ks > 0);
                    }
                    tc::umma_commit(&sb_free);
                    tc::umma_commit(&kp_free[kb]);   // M1, M4 and M2 of chunk c have read its set
                    // M1 of chunk c+1, once the scores of chunk c have been read
                    if (c + 1 < info.nch) {
                        const uint32_t st1 = (job + 1) % kStages;
                        kb = kpc & 1;
                        if (!W(&full[st1], (job + 1) / kStages) || !W(&kp_ready[kb], kpc >> 1) ||
                            !W(&p_free, cc)) { ok = false; break; }
                        ++kpc;
                        TRACE(1, 2, c + 1);
                        issue_m1(sb + st1 * kStage, kb, kfast[kb] != 0);
                    }
                    // M3: O^T += V^T P'^T
                    if (fast && !W(&pp_ready[pb], cc >> 1)) { ok = false; break; }
                    TRACE(1, 5, c);
                    tc::tc_fence_after();
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        tc::umma_bf16(tmem + kTO + 64 * ob, desc_mn8(v_s + ks * 2048),
                                      desc_k(sb + kPp + pb * kRegion + ks * 32), kIdescO3, 1u);
                    tc::umma_commit(&o_full[ob]);
                    tc::umma_commit(&pp_free[pb]);
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
    } else if (warp >= 4 && warp < 8) {
        // =============================== scaling warps ===============================
        // Thread wtid makes row s = wtid & 63, columns 64 * (wtid >> 6) .. + 64 of each K~ tile.
        const int wtid = threadIdx.x - 128;
        const int srow = wtid & 63, shalf = wtid >> 6;
        const int quarter = warp & 3;
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        constexpr int kBar = 1;
        const uint64_t keep = tc::policy_evict_last(), drop = tc::policy_evict_first();
        uint32_t us = 0, kpc = 0, cc = 0, job = 0;   // job: stage counter as the producer's

        // K rows and raw g of the output-pass chunk still to scale, loaded one chunk ahead into
        // registers (the scores of the current chunk are done in between); raw g of the
        // state-pass jobs, two jobs ahead
        uint4 kx[8];
        float2 graw = make_float2(0.f, 0.f), gry = make_float2(0.f, 0.f);
        auto prefetch = [&](int64_t c0, int nv, int h, bool state_pass) {
            graw = load_gate(a.g, c0, nv, H, h);
            if (srow < nv) {
                const uint8_t *src = reinterpret_cast<const uint8_t *>(
                    a.k + ((c0 + srow) * H + h) * kD + 64 * shalf);
                const uint64_t pol = state_pass ? keep : drop;
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8) kx[c8] = tc::ldg_nc_hint(src + 16 * c8, pol);
            } else {
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8) kx[c8] = make_uint4(0u, 0u, 0u, 0u);
            }
        };
        // K~ = K exp(base - b_s) into buffer kpc & 1 (and raw K if `raw`); rows >= nv zero.
        auto make_k = [&](const uint4 (&x)[8], const Gate &G, float base, int nv, bool raw,
                          int fast_flag) {
            const uint32_t kb = kpc & 1;
            wait_nv(&kp_free[kb], (kpc >> 1) - 1, kpc >= 2, abort_v, status);
            if (wtid == 0) TRACE(2, 9, kpc);
            const float bs = gate_at(G, srow);
            const float fac = srow < nv ? tc::ex2((base - bs) * kLog2e) : 0.f;
            store_row_scaled<false>(sm + kKp + kb * kTile + shalf * kRegion,
                             raw ? sm + kKr + kb * kTile + shalf * kRegion : nullptr, srow, x, fac);
            if (wtid == 0) TRACE(2, 10, kpc);
            tc::fence_proxy_async_smem();
            named_sync(kBar, 128);
            if (wtid == 0) {
                kfast[kb] = fast_flag;
                tc::mbar_arrive(&kp_ready[kb]);
            }
            ++kpc;
        };

        for (;;) {
            const uint32_t slot = us & 1;
            if (!wg_wait(&unit_full[slot], us >> 1, true, kBar, abort_v, status)) break;
            const UnitInfo info = units[slot];
            named_sync(kBar, 128);
            if (wtid == 0) tc::mbar_arrive(&unit_empty[slot]);
            if (!info.valid) break;
            const int h = info.h, nch = info.nch;
            auto chunk_c0 = [&](int idx) { return info.t0 + int64_t(idx) * kChunk; };
            auto chunk_nv = [&](int idx) {
                return static_cast<int>(min(int64_t(kChunk), info.t1 - chunk_c0(idx)));
            };

            // ---------------- A: K' = K exp(B_end - B_s), chunks last to first ----------------
            // job r is chunk nch - 1 - r; its K tile arrived by TMA in the first tile of the
            // stage and is scaled there in place (ordinary shared-memory loads are cheap here:
            // the tensor core only runs the short state-pass products). The log-decays are
            // loaded two jobs ahead.
            auto job_c0 = [&](int r) { return chunk_c0(nch - 1 - r); };
            auto job_nv = [&](int r) { return chunk_nv(nch - 1 - r); };
            graw = load_gate(a.g, job_c0(0), job_nv(0), H, h);
            if (nch > 1) gry = load_gate(a.g, job_c0(1), job_nv(1), H, h);
            float D = 0.f;   // total log-decay of the chunks already visited (the later ones)
            auto a_job = [&](int r, float2 &gb) {
                const int nv = job_nv(r);
                const uint32_t st = job % kStages;
                if (wtid == 0) TRACE(2, 1, r);
                const Gate G = scan_gate(gb, nv);
                if (r + 2 < nch) gb = load_gate(a.g, job_c0(r + 2), job_nv(r + 2), H, h);
                wait_nv(&full[st], job / kStages, true, abort_v, status);
                if (wtid == 0) TRACE(2, 7, r);
                const float bs = gate_at(G, srow);
                const float fac = srow < nv ? tc::ex2((G.bC + D - bs) * kLog2e) : 0.f;
                uint8_t *kt = sm + st * kStage + shalf * kRegion;
                uint4 x[8];
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8) x[c8] = *reinterpret_cast<const uint4 *>(kt + sw(srow, c8));
                store_row_scaled<true>(kt, nullptr, srow, x, fac);
                tc::fence_proxy_async_smem();
                named_sync(kBar, 128);
                if (wtid == 0) {
                    tc::mbar_arrive(&ka_ready[st]);
                    TRACE(2, 8, r);
                }
                D += G.bC;
                ++job;
            };
            for (int r = 0; r < nch; r += 2) {
                a_job(r, graw);
                if (r + 1 < nch) a_job(r + 1, gry);
            }
            prefetch(chunk_c0(0), chunk_nv(0), h, false);
            wait_nv(&d_free, us - 1, us >= 1, abort_v, status);
            if (wtid == 0) {
                unit_D = D;
                tc::mbar_arrive(&d_ready);
            }

            // ---------------- C ----------------
            // K~ of chunk 0; then per chunk: K~ of the next chunk, P' of this one. The scaling
            // warps wait on every stage phase (mbarrier waits compare parity only, so a waiter
            // must not skip phases), although here they read K with ordinary global loads.
            const uint32_t job_c = job;
            auto wait_stage = [&](int c) {
                wait_nv(&full[(job_c + c) % kStages], (job_c + c) / kStages, true, abort_v, status);
            };
            Gate Gc = scan_gate(graw, chunk_nv(0));
            wait_stage(0);
            make_k(kx, Gc, Gc.fast ? 0.f : Gc.bC, chunk_nv(0), !Gc.fast, Gc.fast);
            if (nch > 1) prefetch(chunk_c0(1), chunk_nv(1), h, false);
            for (int c = 0; c < nch; ++c) {
                const int64_t c0 = chunk_c0(c);
                const int nv = chunk_nv(c);
                const Gate G = Gc;
                if (c + 1 < nch) {
                    const int nv1 = chunk_nv(c + 1);
                    Gc = scan_gate(graw, nv1);
                    wait_stage(c + 1);
                    make_k(kx, Gc, Gc.fast ? 0.f : Gc.bC, nv1, !Gc.fast, Gc.fast);
                    if (c + 2 < nch) prefetch(chunk_c0(c + 2), chunk_nv(c + 2), h, false);
                    if (wtid == 0) TRACE(2, 3, c);
                }
                // scores -> P' (bf16, K-major rows t): mask s <= t < nv; exact route weights
                const uint32_t pb = cc & 1;
                wait_nv(&p_full, cc, true, abort_v, status);
                wait_nv(&pp_free[pb], (cc >> 1) - 1, cc >= 2, abort_v, status);
                if (wtid == 0) TRACE(2, 5, c);
                tc::tc_fence_after();
                // M=64 accumulator layout: row t = 16 * quarter + lane in lanes 0-15
                const int tr = quarter * 16 + (lane & 15);
                const float bt = gate_at(G, tr) * kLog2e;
                uint8_t *pp = sm + kPp + pb * kRegion;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t p[32];
                    tc::tmem_ld_32x32b_x32(tmem + lane_base + kTP + 32 * half, p);
                    tc::tmem_ld_wait();
                    if (half == 1) {
                        tc::tc_fence_before();
                        named_sync(kBar, 128);
                        if (wtid == 0) tc::mbar_arrive(&p_free);
                    }
                    if (!G.fast) {
                        // exact route: P'[t, s] = P[t, s] exp(b_t - b_s)
#pragma unroll
                        for (int s = 0; s < 32; ++s)
                            p[s] = __float_as_uint(__uint_as_float(p[s]) *
                                                   tc::ex2(bt - gate_at(G, 32 * half + s) * kLog2e));
                    }
                    if (lane < 16) {
                        const bool live = tr < nv;
#pragma unroll
                        for (int c4 = 0; c4 < 4; ++c4) {
                            uint32_t w[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int si = 8 * c4 + 2 * e, s = 32 * half + si;
                                const float f0 = (live && s <= tr) ? __uint_as_float(p[si]) : 0.f;
                                const float f1 = (live && s + 1 <= tr) ? __uint_as_float(p[si + 1]) : 0.f;
                                w[e] = float2_to_bf16x2(f0, f1);
                            }
                            *reinterpret_cast<uint4 *>(pp + sw(tr, 4 * half + c4)) =
                                make_uint4(w[0], w[1], w[2], w[3]);
                        }
                    }
                }
                if (!G.fast) {
                    // exact route: q_t <- exp(b_t) q_t in place (M1 has read Q already); the
                    // rows come from global memory, not from the tile
                    uint8_t *qt = sm + ((job_c + c) % kStages) * kStage + shalf * kRegion;
                    uint4 x[8];
                    if (srow < nv) {
                        const uint8_t *src = reinterpret_cast<const uint8_t *>(
                            a.q + ((c0 + srow) * H + h) * kD + 64 * shalf);
#pragma unroll
                        for (int c8 = 0; c8 < 8; ++c8) x[c8] = tc::ldg_nc_hint(src + 16 * c8, drop);
                    } else {
#pragma unroll
                        for (int c8 = 0; c8 < 8; ++c8) x[c8] = make_uint4(0u, 0u, 0u, 0u);
                    }
                    store_row_scaled<false>(qt, nullptr, srow, x, tc::ex2(gate_at(G, srow) * kLog2e));
                }
                tc::fence_proxy_async_smem();
                named_sync(kBar, 128);
                if (wtid == 0) {
                    tc::mbar_arrive(&pp_ready[pb]);
                    TRACE(2, 6, c);
                }
                ++cc;
            }
            // one uniform decision per unit (after an abort every wait returns at once, so all
            // threads still pass the same barriers inside the unit)
            if (named_any(kBar, 128, *abort_v != 0)) break;
            job = job_c + nch;
            ++us;
        }
    } else if (warp >= 8) {
        // =============================== state warps ===============================
        // Waits inside a unit do not vote: a thread whose wait gives up has set the abort
        // flag, and every later wait returns at once, so all threads still pass the same
        // barriers; one OR-vote per hand-off and per unit, taken over both groups together
        // (they also share a barrier in the hand-off), then ends the loop uniformly.
        constexpr int kBarBoth = 4;
        const int wg = (warp - 8) >> 2;
        const int wtid = threadIdx.x - 256 - 128 * wg;
        const int quarter = warp & 3;
        const int j = quarter * 32 + lane;     // value column = TMEM lane
        const int i0 = 64 * wg;                // my key rows i0 .. i0 + 63
        const int bar_id = 2 + wg;
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        uint32_t us = 0, dsc = 0, cc = 0, sbc = 0;
        float S[64];   // S^T[j][i0 + i] = S[i0 + i][j]

        // bf16 copy of S^T for M2: my 64 keys -> 32 packed columns of the A operand
        auto write_sb = [&]() {
            wait_nv(&sb_free, sbc - 1, sbc >= 1, abort_v, status);
            uint32_t w[32];
#pragma unroll
            for (int m = 0; m < 32; ++m) w[m] = float2_to_bf16x2(S[2 * m], S[2 * m + 1]);
            tc::tmem_st_32x32b_x32(tmem + lane_base + kTSb + 32 * wg, w);
            tc::tmem_st_wait();
            tc::tc_fence_before();
            named_sync(bar_id, 128);
            if (wtid == 0) tc::mbar_arrive(&sb_ready);
            ++sbc;
        };

        for (;;) {
            const uint32_t slot = us & 1;
            if (!wg_wait(&unit_full[slot], us >> 1, true, kBarBoth, abort_v, status, 256)) break;
            const UnitInfo info = units[slot];
            named_sync(bar_id, 128);
            if (wtid == 0) tc::mbar_arrive(&unit_empty[slot]);
            if (!info.valid) break;
            const int h = info.h, nch = info.nch;
            if (wtid == 0) TRACE(3 + wg, 1, us);

            // ---------------- hand-off: S_in, bf16 S_in for M2, publish S_out ----------------
            {
                const uint32_t db = dsc & 1;
                bool bad = !wait_or_abort(&ds_full[db], (dsc >> 1) & 1, abort_v, status);
                if (wtid == 0) TRACE(3 + wg, 11, us);
                bad = bad || !wait_or_abort(&d_ready, us & 1, abort_v, status);
                if (wtid == 0) TRACE(3 + wg, 12, us);
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
                if (named_any(kBarBoth, 256, bad || *abort_v)) break;
                if (wtid == 0) TRACE(3 + wg, 2, 0);
                tc::tc_fence_after();
                if (info.first) {
                    if (f.h0) {
                        const float *src = f.h0 + ((info.n * H + h) * kD + i0) * kD + j;
#pragma unroll
                        for (int i = 0; i < 64; ++i) S[i] = __ldg(src + i * kD);
                    } else {
#pragma unroll
                        for (int i = 0; i < 64; ++i) S[i] = 0.f;
                    }
                } else {
                    // the predecessor's S_out, written by another SM: read through L2
                    const float *src = f.incl + ((static_cast<size_t>(info.sigma - 1) * H + h) * kD + i0) * kD + j;
#pragma unroll
                    for (int i = 0; i < 64; ++i) S[i] = __ldcg(src + i * kD);
                }
                if (wtid == 0) TRACE(3 + wg, 13, us);
                const float eB = tc::ex2(unit_D * kLog2e);
                named_sync(bar_id, 128);
                if (wtid == 0) tc::mbar_arrive(&d_free);
                write_sb();   // bf16 S_in for the first chunk's M2 first: the output pass can start
                // S_out = exp(B) S_in + dS: to hT (last segment) or to the successor; each warp
                // store covers one 128-byte row segment (32 consecutive j)
                float *dst = info.last ? (f.hT ? f.hT + (info.n * H + h) * kD * kD : nullptr)
                                       : f.incl + (static_cast<size_t>(info.sigma) * H + h) * kD * kD;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t d[32];
                    tc::tmem_ld_32x32b_x32(tmem + lane_base + kTdS + 128 * db + i0 + 32 * half, d);
                    tc::tmem_ld_wait();
                    if (dst) {
                        float *p = dst + (i0 + 32 * half) * kD + j;
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            p[i * kD] = fmaf(eB, S[32 * half + i], __uint_as_float(d[i]));
                    }
                }
                if (wtid == 0) TRACE(3 + wg, 14, us);
                tc::tc_fence_before();
                named_sync(kBarBoth, 256);   // both state groups have stored S_out and read dS
                if (wtid == 0) tc::mbar_arrive(&ds_free[db]);
                if (wg == 0 && wtid == 0 && !info.last) {
                    // publish for the successor: the barrier orders the groups' stores before
                    // this thread's device-scope fence and release of the flag
                    __threadfence();
                    tc::st_release_gpu(f.flags + info.sigma * H + h, f.epoch);
                }
                if (wtid == 0) TRACE(3 + wg, 3, 0);
            }

            // ---------------- C ----------------
            float2 graw = load_gate(a.g, info.t0, static_cast<int>(min(int64_t(kChunk), info.t1 - info.t0)), H, h);
            for (int c = 0; c < nch; ++c) {
                const int64_t c0 = info.t0 + int64_t(c) * kChunk;
                const int nv = static_cast<int>(min(int64_t(kChunk), info.t1 - c0));
                const Gate G = scan_gate(graw, nv);
                if (c + 1 < nch)
                    graw = load_gate(a.g, c0 + kChunk, static_cast<int>(min(int64_t(kChunk), info.t1 - c0 - kChunk)), H, h);
                if (wtid == 0) TRACE(3 + wg, 4, c);

                // state carry for my 64 keys; bf16 copy for the next chunk's M2
                if (c + 1 < nch) {
                    const uint32_t db = dsc & 1;
                    wait_nv(&ds_full[db], dsc >> 1, true, abort_v, status);
                    ++dsc;
                    if (wtid == 0) TRACE(3 + wg, 7, c);
                    tc::tc_fence_after();
                    const float eC = tc::ex2(G.bC * kLog2e);
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        uint32_t d[32];
                        tc::tmem_ld_32x32b_x32(tmem + lane_base + kTdS + 128 * db + i0 + 32 * half, d);
                        tc::tmem_ld_wait();
                        if (G.fast) {
#pragma unroll
                            for (int i = 0; i < 32; ++i) S[32 * half + i] = eC * (S[32 * half + i] + __uint_as_float(d[i]));
                        } else {
#pragma unroll
                            for (int i = 0; i < 32; ++i) S[32 * half + i] = fmaf(eC, S[32 * half + i], __uint_as_float(d[i]));
                        }
                    }
                    tc::tc_fence_before();
                    named_sync(bar_id, 128);
                    if (wtid == 0) tc::mbar_arrive(&ds_free[db]);
                    write_sb();
                    if (wtid == 0) TRACE(3 + wg, 8, c);
                }

                // o_t = factor_t O^T[j][t] for my 32 tokens t = 32 wg + tt: staged as a
                // [32 t x 128 j] bf16 tile and written by one TMA store (direct stores when the
                // group has rows past the chunk's valid tokens, which belong to another sequence)
                {
                    const uint32_t ob = cc & 1;
                    wait_nv(&o_full[ob], cc >> 1, true, abort_v, status);
                    if (wtid == 0) TRACE(3 + wg, 9, c);
                    tc::tc_fence_after();
                    uint32_t o[32];
                    tc::tmem_ld_32x32b_x32(tmem + lane_base + kTO + 64 * ob + 32 * wg, o);
                    tc::tmem_ld_wait();
                    tc::tc_fence_before();
                    if (wtid == 0) tc::tma_store_wait_read<0>();   // staging buffer free again
                    named_sync(bar_id, 128);
                    if (wtid == 0) tc::mbar_arrive(&o_free[ob]);
                    // lane l's factor for token 32 wg + l, then broadcast
                    const float bl = gate_at(G, 32 * wg + lane);
                    const float fl = G.fast ? a.scale * tc::ex2(bl * kLog2e) : a.scale;
                    if (32 * wg + 32 <= nv) {
                        uint8_t *stg = sm + kOst + wg * kOstBytes + 2 * j;
#pragma unroll
                        for (int tt = 0; tt < 32; ++tt) {
                            const float ft = __shfl_sync(0xffffffffu, fl, tt);
                            *reinterpret_cast<uint16_t *>(stg + tt * 256) =
                                __bfloat16_as_ushort(__float2bfloat16_rn(ft * __uint_as_float(o[tt])));
                        }
                        tc::fence_proxy_async_smem();
                        named_sync(bar_id, 128);
                        if (wtid == 0) {
                            tc::tma_store_3d(&maps.o, 0, h, static_cast<int32_t>(c0 + 32 * wg),
                                             sm + kOst + wg * kOstBytes);
                            tc::tma_store_commit();
                        }
                    } else {
                        uint16_t *orow = a.o + (c0 * H + h) * kD + j;
#pragma unroll
                        for (int tt = 0; tt < 32; ++tt) {
                            const float ft = __shfl_sync(0xffffffffu, fl, tt);
                            const int tk = 32 * wg + tt;
                            if (tk < nv)
                                orow[static_cast<size_t>(tk) * H * kD] =
                                    __bfloat16_as_ushort(__float2bfloat16_rn(ft * __uint_as_float(o[tt])));
                        }
                    }
                    if (wtid == 0) TRACE(3 + wg, 10, c);
                }
                ++cc;
            }
            if (named_any(kBarBoth, 256, *abort_v != 0)) break;
            ++us;
        }
        if (wtid == 0) tc::tma_store_wait_all<0>();
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

cudaError_t encode_map(CUtensorMap *map, const void *base, int64_t T_total, int H, bool store) {
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
    cuuint32_t box_load[3] = {64, 1, 64}, box_store[3] = {128, 1, 32};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims,
                          strides, store ? box_store : box_load, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE,
                          store ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}
}  // namespace

cudaError_t make_maps(TcMaps *m, const void *q, const void *k, const void *v, const void *o,
                      int64_t T_total, int H) {
    cudaError_t e = encode_map(&m->q, q, T_total, H, false);
    if (e == cudaSuccess) e = encode_map(&m->k, k, T_total, H, false);
    if (e == cudaSuccess) e = encode_map(&m->v, v, T_total, H, false);
    if (e == cudaSuccess) e = encode_map(&m->o, o, T_total, H, true);
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
        cudaError_t e = tck::make_maps(&maps, a.q, a.k, a.v, a.o, T_total, a.H);
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
    unsigned int n[5];
    if (cudaMemcpyFromSymbol(n, sala::g_trace_n, sizeof(n)) != cudaSuccess) return -1;
    static unsigned long long buf[5][sala::kTraceN];
    if (cudaMemcpyFromSymbol(buf, sala::g_trace, sizeof(buf)) != cudaSuccess) return -1;
    int k = 0;
    for (int r = 0; r < 5; ++r)
        for (unsigned i = 0; i < n[r] && i < static_cast<unsigned>(sala::kTraceN) && k < max; ++i)
            out[k++] = buf[r][i];
    return k;
}
#endif
