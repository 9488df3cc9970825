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
//  C. output pass over the chunks, first to last, from S_in. The state lives in tensor
//     memory in fp32 and the tensor core adds each chunk to it directly. It is kept relative
//     to a reference point r: with B_t the log-decay from r to token t, the stored state is
//     Z = exp(-B) S, and
//       o_t = scale exp(B_t) [ q_t Z + sum_{s<=t in the chunk} (q_t . k_s) exp(-B_s) v_s ]
//       Z  <- Z + sum_{s in the chunk} exp(-B_s) k_s^T v_s
//     so the weights become per-column factors exp(-B_s) on the keys and per-row factors
//     exp(B_t) on the output, and no per-chunk decay touches the state. Before a chunk whose
//     factors would leave [e^-60, e^60] the reference moves to the chunk start (Z is rescaled
//     once in tensor memory). When the chunk's own decay range is wider than that, the chunk
//     takes the exact route: per-entry weights exp(b_t - b_s) on the scores, q_t scaled by
//     exp(b_t) in place, Z rescaled to the chunk end and k_s weighted by exp(b_C - b_s).
//
// The state is kept transposed (S^T, value index j in the tensor-memory lane), so that its
// bf16 copy can sit in tensor memory as the A operand of the q.S product. Contractions
// (tcgen05.mma kind::f16, bf16 in, fp32 accumulators in tensor memory):
//   M1  P    = Q K~^T      M=64  N=64  K=128   A=Q smem (K-major)     B=K~ smem (K-major)
//   M2  O^T  = Z^T Q^T     M=128 N=64  K=128   A=Z^T bf16 in TMEM     B=Q smem (K-major)
//   M3  O^T += V^T P'^T    M=128 N=64  K=64    A=V smem (MN-major)    B=P' smem (K-major)
//   M4  Z^T += V^T K~      M=128 N=128 K=64    A=V smem (MN-major)    B=K~ smem (MN-major)
// (the state pass runs M4 into its own accumulator dS^T). K~ is k scaled per token. In the
// state pass the K tile arrives by TMA and is scaled in place in shared memory (the tensor
// core only runs the short M4 there). In the output pass, where the tensor core streams
// operands most of the time, the scaling warps make K~ from a global load straight into
// shared memory instead: ordinary shared-memory loads issued while the tensor core reads its
// operands stall far behind them. Q and V tiles arrive by TMA, o leaves by TMA stores.
//
// Roles: warp 0 loads (TMA), warp 1 issues MMAs and owns the tensor memory, warp 2 publishes
// the hand-off flags, warp 3 reads g ahead of everyone and publishes each chunk's prefix sums
// and plan (reference point, rescaling, route) in a small ring of shared-memory records,
// warps 4-7 scale K and turn scores into P' (and, exact route, scale Q), warps 8-11 do the
// hand-off and make the bf16 copy of the state for every chunk (rescaling it when the
// reference moves), warps 12-15 write o (each warp 32 value columns of the chunk's 64
// tokens). The other roles take their per-token factors from the records, so no role waits
// on a load of g or on a prefix sum of its own.
// mbarrier waits compare phase parity only, so every barrier has at most one phase in flight
// per waiter: each waiter consumes every phase of the barriers it waits on, and a producer
// cannot complete a second phase before its consumer has consumed the first. Every wait is
// bounded (2 s of %globaltimer); a timeout records SALA_ERR_TIMEOUT, stops the CTA's work,
// drains its copies and MMAs, frees its tensor memory and returns.
#include "prefill_common.cuh"

namespace sala {
namespace {

using namespace tck;

constexpr int kStages = 4;
constexpr int kThreads = 512;

// dynamic shared memory (offsets from a 1024-aligned base)
constexpr uint32_t kStage = 2 * kTile;              // Q | V
constexpr uint32_t kKp = kStages * kStage;          // K~ [2] (factored or exact weights)
constexpr uint32_t kKr = kKp + 2 * kTile;           // raw K [2] (exact-route M1)
constexpr uint32_t kPp = kKr + 2 * kTile;           // P' (K-major B of M3)
constexpr uint32_t kOst = kPp + kRegion;            // o staging, per output warp [64 t][32 j]
constexpr uint32_t kOstWarp = 64 * 64;
constexpr uint32_t kGate = kOst + 4 * kOstWarp;     // gate records: state pass [kRecA], output pass [kRecC]
constexpr int kRecA = 4, kRecC = 8;
constexpr uint32_t kBytes = kGate + (kRecA + kRecC) * 288;
constexpr uint32_t kSmemAlloc = kBytes + 1024;

// TMEM columns: state-pass dS^T, Z^T (fp32), Z^T bf16 (A of M2), P (M=64 layout), O^T [2].
// The bf16 copy is double-buffered; its second buffer borrows the first 64 columns of dS^T,
// which the output pass does not use: the hand-off has read dS^T before the output pass
// starts, and the next state pass is issued after the output pass's last M2 (tcgen05.mma
// operations of one thread execute in issue order).
constexpr uint32_t kTdS = 0, kTZ = 128, kTZb = 256, kTP = 320, kTO = 384, kTCols = 512;
__device__ __forceinline__ uint32_t zb_col(uint32_t buf) { return buf ? kTdS : kTZb; }
constexpr uint32_t kIdescP = tc::idesc_bf16_f32(64, 64, 0, 0);
constexpr uint32_t kIdescO2 = tc::idesc_bf16_f32(128, 64, 0, 0);
constexpr uint32_t kIdescO3 = tc::idesc_bf16_f32(128, 64, 1, 0);
constexpr uint32_t kIdescS = tc::idesc_bf16_f32(128, 128, 1, 1);

// named barriers (0 is __syncthreads)
constexpr int kBarScale = 1, kBarConv = 2, kBarOut = 3;



// Event trace of CTA 0 for latency analysis (compiled only with -DSALA_TRACE): SM clock,
// role, event id and chunk index, written to a global array.
#ifdef SALA_TRACE
constexpr int kTraceN = 512;
__device__ unsigned long long g_trace[8][kTraceN];
__device__ unsigned int g_trace_n[8];
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
// Per-site wait-cycle totals of CTA 0's MMA thread (slots 0-15) and of scaling thread 0
// (slots 16-31), kept in registers (wacc_) and written once at the end.
__device__ unsigned long long g_wait_acc[32];
#define TIMED(slot, expr)                                        \
    ([&]() {                                                     \
        const long long t0_ = clock64();                         \
        const bool r_ = (expr);                                  \
        wacc_[slot] += clock64() - t0_;                          \
        return r_;                                               \
    }())
#else
#define TRACE(role, ev, idx) \
    do {                     \
    } while (0)
#define TIMED(slot, expr) (expr)
#endif



// 64 bf16 of one row, scaled by f, to a [64 x 128 B] SW128 region row. kExact: product in
// fp32, rounded once; otherwise f is rounded to bf16 and each pair takes one packed multiply
// (about 5x fewer instructions, one more rounding of the factor: used for the output pass,
// whose tolerance has more room).
template <bool kExact>
__device__ __forceinline__ void store_row_scaled(uint8_t *dst, int row, const uint4 (&x)[8], float f) {
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
    }
}


// Exact route, queries: row `row` (columns 64 half .. + 63) of the Q tile at qt becomes
// exp(b_row) q_row, read from global memory (the tile has been consumed by M1).
__device__ __noinline__ void exact_q_scale(uint8_t *qt, const uint16_t *q, int64_t c0, int row, int half,
                                           int nv, int H, int h, float b_row) {
    uint4 x[8];
    if (row < nv) {
        const uint4 *src = reinterpret_cast<const uint4 *>(q + ((c0 + row) * H + h) * kD + 64 * half);
        for (int c8 = 0; c8 < 8; ++c8) x[c8] = src[c8];
    } else {
        for (int c8 = 0; c8 < 8; ++c8) x[c8] = make_uint4(0u, 0u, 0u, 0u);
    }
    store_row_scaled<false>(qt, row, x, tc::ex2(b_row * kLog2e));
}

// State pass: columns 32 q .. + 31 of row `row` of the K tile at kt scaled in place by f (the
// scaling and converting warps share each tile, a quarter of its columns per half-group).
__device__ __forceinline__ void scale_k_quarter(uint8_t *kt, int row, int q, float f) {
    uint8_t *base = kt + (q >> 1) * kRegion;
    uint4 x[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) x[k] = *reinterpret_cast<const uint4 *>(base + sw(row, (q & 1) * 4 + k));
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        uint4 y;
        y.x = mul_bf16x2(x[k].x, f);
        y.y = mul_bf16x2(x[k].y, f);
        y.z = mul_bf16x2(x[k].z, f);
        y.w = mul_bf16x2(x[k].w, f);
        *reinterpret_cast<uint4 *>(base + sw(row, (q & 1) * 4 + k)) = y;
    }
}


}  // namespace

__global__ void __launch_bounds__(kThreads, 1)
prefill_fused_kernel(const __grid_constant__ TcMaps maps, PrefillArgs f, SegTable t, int *status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
    __shared__ uint64_t full[kStages], ka_full[kStages], empty[kStages], ka_ready[kStages];
    __shared__ uint64_t unit_full[2], unit_empty[2], kp_ready[2], kp_free[2];
    __shared__ uint64_t p_full, p_free, pp_ready, pp_free;
    __shared__ uint64_t ga_full[kRecA], ga_empty[kRecA], gc_full[kRecC], gc_empty[kRecC];
    __shared__ uint64_t z_full, z_free, zb_ready[2], zb_free[2], o_full[2], o_free[2];
    __shared__ uint64_t ds_full, ds_free, pub_ready, pub_free, drain;
    __shared__ UnitInfo units[2];
    __shared__ int kfast[2];
    __shared__ uint32_t *pub_flag;   // the flag the publisher releases next
    __shared__ int pub_cmd;          // 0: nothing this unit, 1: release pub_flag, 2: stop
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
            tc::mbar_init(&full[s], 1);       // output-pass job: Q and V landed (expect_tx)
            tc::mbar_init(&ka_full[s], 1);    // state-pass job: K and V landed (expect_tx)
            tc::mbar_init(&empty[s], 1);      // MMA commit
            tc::mbar_init(&ka_ready[s], 8);   // the state-pass K' tile of this stage is scaled
                                              // (scaling and converting warps; phases count
                                              // this stage's state-pass jobs)
        }
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(&unit_full[i], 1);
            tc::mbar_init(&unit_empty[i], 5);   // MMA, gate, scaling, converting, output warps
            tc::mbar_init(&kp_ready[i], 4);     // one arrival per scaling warp
            tc::mbar_init(&kp_free[i], 1);
            tc::mbar_init(&o_full[i], 1);
            tc::mbar_init(&o_free[i], 4);       // one arrival per output warp
        }
        tc::mbar_init(&p_full, 1);
        tc::mbar_init(&p_free, 4);     // one arrival per scaling warp
        tc::mbar_init(&pp_ready, 4);
        tc::mbar_init(&pp_free, 1);
        for (int i = 0; i < kRecA; ++i) {
            tc::mbar_init(&ga_full[i], 1);
            tc::mbar_init(&ga_empty[i], 8);    // scaling and converting warps
        }
        for (int i = 0; i < kRecC; ++i) {
            tc::mbar_init(&gc_full[i], 1);
            tc::mbar_init(&gc_empty[i], 12);   // scaling, converting and output warps
        }
        tc::mbar_init(&z_full, 1);       // MMA commit after M4 into Z
        tc::mbar_init(&z_free, 4);       // converting warps: Z read (and rescaled)
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(&zb_ready[i], 4);   // converting warps: bf16 Z written
            tc::mbar_init(&zb_free[i], 1);    // MMA commit after M2
        }
        tc::mbar_init(&ds_full, 1);
        tc::mbar_init(&ds_free, 4);
        tc::mbar_init(&pub_ready, 4);
        tc::mbar_init(&pub_free, 1);
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
    // launched as a programmatic dependent of the segment-table kernel: the set-up above
    // overlaps it; nothing that kernel writes (table, ticket, flags, hT) is touched before this
    asm volatile("griddepcontrol.wait;" ::: "memory");
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
        uint32_t fpar = 0, kfpar = 0;   // bit st: next phase of full[st] / ka_full[st]
        uint32_t a_mask = 0, lpar = 0;  // bit st: last load of stage st was a state-pass job; its phase
        bool ok = true;
        // one job: K and V (state pass -> ka_full; K goes to the first tile of the stage) or Q
        // and V (output pass -> full) of the chunk at token c0, with L2 prefetches of the
        // chunk's log-decays (read by other warps a little later)
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
                uint64_t *bar = with_q ? &full[st] : &ka_full[st];
                tc::mbar_arrive_expect_tx(bar, 2 * kTile);
                const CUtensorMap *first = with_q ? &maps.q : &maps.k;
                tc::tma_load_3d_hint(base, first, 0, h, x0, bar, with_q ? drop : keep);
                tc::tma_load_3d_hint(base + kRegion, first, 64, h, x0, bar, with_q ? drop : keep);
                const uint64_t pol = with_q ? drop : keep;
                tc::tma_load_3d_hint(base + kTile, &maps.v, 0, h, x0, bar, pol);
                tc::tma_load_3d_hint(base + kTile + kRegion, &maps.v, 64, h, x0, bar, pol);
                // the scaling warps read this chunk's K rows with ordinary loads a little later
                tc::tma_prefetch_l2_3d(&maps.k, 0, h, x0, pol);
                tc::tma_prefetch_l2_3d(&maps.k, 64, h, x0, pol);
            }
            __syncwarp();
            const uint32_t ph = with_q ? (fpar >> st) & 1 : (kfpar >> st) & 1;
            lpar = (lpar & ~(1u << st)) | (ph << st);
            if (with_q) fpar ^= 1u << st; else kfpar ^= 1u << st;
            a_mask = with_q ? (a_mask & ~(1u << st)) : (a_mask | (1u << st));
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
                // (debug build: the segment lies inside its sequence and the tokens)
                if (locate_segment(t, info.sigma, info.n, info.t0, info.t1) &&
                    dcheck(info.n >= 0 && info.n < t.nseq && seq_begin(t, info.n) <= info.t0 &&
                           info.t0 < info.t1 && info.t1 <= seq_begin(t, info.n + 1) &&
                           info.t1 <= seq_begin(t, t.nseq), status)) {
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
            // state pass (K, V; chunks last to first), then output pass (Q, V; first to last)
#pragma unroll 1
            for (int j = 0; j < 2 * info.nch && ok; ++j) {
                const int c = j < info.nch ? info.nch - 1 - j : j - info.nch;
                const int64_t c0 = info.t0 + int64_t(c) * kChunk;
                ok = load_job(c0, static_cast<int>(min(int64_t(kChunk), info.t1 - c0)), info.h, j >= info.nch);
            }
            ++us;
        }
        // drain: the copies of the last stages must land before the CTA may exit
        if (lane == 0)
            for (uint32_t j = job > kStages ? job - kStages : 0; j < job; ++j) {
                const uint32_t st = j % kStages;
                tc::mbar_wait((a_mask >> st) & 1 ? &ka_full[st] : &full[st], (lpar >> st) & 1, kWaitNs);
            }
    } else if (warp == 1) {
        // =============================== MMA issuer ===============================
        // The whole warp follows the schedule (every wait, counter and descriptor is
        // warp-uniform, so it stays in the uniform datapath) and one elected lane issues the
        // MMAs and commits (the same lane every time: a commit tracks its own thread's MMAs).
        const uint32_t sb = tc::smem_u32(sm);
        uint32_t job = 0, us = 0, kpc = 0, cc = 0, zbc = 0, zfc = 0;
        uint32_t ka_par = 0;   // bit st: phase parity of ka_ready[st] (state-pass jobs only)
        uint32_t cpar = 0;     // bit st: phase parity of full[st] (output-pass jobs only)
        auto W = [&](uint64_t *bar, uint32_t par) {
            return __all_sync(0xffffffffu, wait_or_abort(bar, par & 1, abort_v, status));
        };
        // Several phases an MMA group needs: their tests go out together (each mbarrier test
        // takes tens of cycles, and they are usually all complete already); only if one is
        // not does the group wait for them one by one.
        auto W3 = [&](uint64_t *b0, uint32_t p0, bool n0, uint64_t *b1, uint32_t p1, bool n1,
                      uint64_t *b2, uint32_t p2, bool n2) {
            const bool t0 = !n0 || tc::mbar_test_wait(b0, p0 & 1);
            const bool t1 = !n1 || tc::mbar_test_wait(b1, p1 & 1);
            const bool t2 = !n2 || tc::mbar_test_wait(b2, p2 & 1);
            if (__all_sync(0xffffffffu, t0 && t1 && t2)) return true;
            return (!n0 || W(b0, p0)) && (!n1 || W(b1, p1)) && (!n2 || W(b2, p2));
        };
#ifdef SALA_TRACE
        unsigned long long wacc_[16] = {};
#endif
        for (;;) {
            const uint32_t slot = us & 1;
            if (!TIMED(0, W(&unit_full[slot], us >> 1))) break;
            const UnitInfo info = units[slot];
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&unit_empty[slot]);
            if (!info.valid) break;
            bool ok = true;
            // ---- A: dS^T = sum over chunks of V^T K', one accumulator
            if (us >= 1) ok = TIMED(1, W(&ds_free, us - 1));
            for (int r = 0; r < info.nch && ok; ++r) {
                const uint32_t st = job % kStages;
                ok = TIMED(3, W(&ka_ready[st], (ka_par >> st) & 1));
                if (!ok) break;
                ka_par ^= 1u << st;
                TRACE(1, 1, r);
                tc::tc_fence_after();
                const uint32_t k_s = sb + st * kStage, v_s = k_s + kTile;   // K' scaled in place
                const uint64_t da = desc_mn8(v_s), db = desc_mn8(k_s);
                if (tc::elect_one()) {
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        tc::umma_bf16(tmem + kTdS, da + ks * (2048 >> 4), db + ks * (2048 >> 4), kIdescS,
                                      (r > 0 || ks > 0) ? 1u : 0u);
                    tc::umma_commit(&empty[st]);
                }
                __syncwarp();
                ++job;
            }
            if (!ok) break;
            if (tc::elect_one()) tc::umma_commit(&ds_full);
            __syncwarp();
            // ---- C, software-pipelined: M1 of chunk c+1 goes out right after M2 of chunk c
            // (before M3 of chunk c), so the scores of c+1 are made while chunk c finishes
            // per chunk c: M4(c), M2(c), M1(c+1), M3(c); the first pass (c = -1) issues M1(0)
            uint32_t kb = kpc & 1;   // K~ set of the chunk in flight
            for (int c = -1; c < info.nch && ok; ++c) {
                const uint32_t st = job % kStages;
                const uint32_t q_s = sb + st * kStage, v_s = q_s + kTile;
                const uint64_t dv = desc_mn8(v_s);
                const uint32_t ob = cc & 1;
                const bool fast = kfast[kb] != 0;
                if (c >= 0) {
                    // M4: Z^T += V^T K~ (not needed after the last chunk), once the converting
                    // warps have read Z (and rescaled it, if the reference moved)
                    if (c + 1 < info.nch) {
                        if (!TIMED(5, W(&z_free, zfc))) { ok = false; break; }
                        TRACE(1, 3, c);
#ifdef SALA_TRACE
                        const long long ti0 = clock64();
#endif
                        tc::tc_fence_after();
                        const uint64_t dk4 = desc_mn8(sb + kKp + kb * kTile);
                        if (tc::elect_one()) {
#pragma unroll
                            for (int ks = 0; ks < 4; ++ks)
                                tc::umma_bf16(tmem + kTZ, dv + ks * (2048 >> 4), dk4 + ks * (2048 >> 4), kIdescS, 1u);
                            tc::umma_commit(&z_full);
                        }
                        __syncwarp();
#ifdef SALA_TRACE
                        wacc_[13] += clock64() - ti0;
#endif
                        ++zfc;
                    }
                    // M2: O^T = Z^T Q^T (Q scaled in place first on the exact route)
                    const uint32_t zb = zbc & 1;
                    if (!TIMED(6, W3(&zb_ready[zb], zbc >> 1, true, &o_free[ob], (cc >> 1) - 1, cc >= 2,
                                     &pp_ready, cc, !fast))) { ok = false; break; }
                    TRACE(1, 4, c);
#ifdef SALA_TRACE
                    const long long ti1 = clock64();
#endif
                    tc::tc_fence_after();
                    const uint64_t dq = desc_k(q_s);
                    const uint32_t za = tmem + zb_col(zb), od = tmem + kTO + 64 * ob;
                    if (tc::elect_one()) {
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks)
                            tc::umma_bf16_ta(od, za + 8 * ks, dq + (((ks >> 2) * kRegion + (ks & 3) * 32) >> 4),
                                             kIdescO2, ks > 0);
                        tc::umma_commit(&zb_free[zb]);
                        tc::umma_commit(&kp_free[kb]);   // M1, M4 and M2 of chunk c have read its set
                    }
                    __syncwarp();
#ifdef SALA_TRACE
                    wacc_[14] += clock64() - ti1;
#endif
                    ++zbc;
                }
                // M1 of the next chunk (P = Q K~^T, or Q K^T on the exact route), once the
                // scores of the chunk before it have been read
                if (c + 1 < info.nch) {
                    const uint32_t jn = c < 0 ? job : job + 1, gn = c < 0 ? cc : cc + 1;
                    const uint32_t kn = kpc & 1;
                    const uint32_t sn = jn % kStages;
                    if (!TIMED(9, W3(&full[sn], (cpar >> sn) & 1, true, &kp_ready[kn], kpc >> 1, true,
                                     &p_free, gn - 1, gn >= 1))) { ok = false; break; }
                    cpar ^= 1u << sn;
                    ++kpc;
                    TRACE(1, 2, c + 1);
                    const uint64_t dk1 = desc_k(sb + (kfast[kn] != 0 ? kKp : kKr) + kn * kTile);
                    const uint64_t dq1 = desc_k(sb + sn * kStage);
                    tc::tc_fence_after();
                    if (tc::elect_one()) {
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks) {
                            const uint32_t o4 = ((ks >> 2) * kRegion + (ks & 3) * 32) >> 4;
                            tc::umma_bf16(tmem + kTP, dq1 + o4, dk1 + o4, kIdescP, ks > 0);
                        }
                        tc::umma_commit(&p_full);
                    }
                    __syncwarp();
                    if (c < 0) kb = kn;
                }
                if (c < 0) continue;
                // M3: O^T += V^T P'^T
                if (fast && !TIMED(12, W(&pp_ready, cc))) { ok = false; break; }
                TRACE(1, 5, c);
#ifdef SALA_TRACE
                const long long ti2 = clock64();
#endif
                tc::tc_fence_after();
                const uint64_t dp = desc_k(sb + kPp);
                if (tc::elect_one()) {
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        tc::umma_bf16(tmem + kTO + 64 * ob, dv + ks * (2048 >> 4), dp + ks * (32 >> 4), kIdescO3, 1u);
                    tc::umma_commit(&o_full[ob]);
                    tc::umma_commit(&pp_free);
                    tc::umma_commit(&empty[st]);
                }
                __syncwarp();
#ifdef SALA_TRACE
                wacc_[15] += clock64() - ti2;
#endif
                kb = (kpc - 1) & 1;   // the set M1 of the next chunk has taken
                ++job;
                ++cc;
            }
            if (!ok) break;
            ++us;
        }
#ifdef SALA_TRACE
        if (blockIdx.x == 0 && lane == 0)
            for (int i = 0; i < 16; ++i) g_wait_acc[i] = wacc_[i];
#endif
        // no MMA may still run when the tensor memory is freed
        if (tc::elect_one()) {
            tc::umma_commit(&drain);
            tc::mbar_wait(&drain, 0, kWaitNs);
        }
        __syncwarp();
    } else if (warp == 2) {
        // =============================== flag publisher ===============================
        // Releases a unit's hand-off flag once the converting warps have stored its S_out:
        // their mbarrier arrivals order the stores before this thread's device-scope fence, so
        // the fence's latency stays off the converting warps.
        // One command per unit, so that no wait here spans more than one unit.
        if (lane == 0) {
            for (uint32_t n = 0;; ++n) {
                if (!wait_or_abort(&pub_ready, n & 1, abort_v, status)) break;
                const int cmd = pub_cmd;
                if (cmd == 2) break;
                if (cmd == 1 && pub_flag != f.withheld) {
                    __threadfence();
                    tc::st_release_gpu(pub_flag, f.epoch);
                }
                tc::mbar_arrive(&pub_free);
            }
        }
    } else if (warp == 3) {
        // =============================== gate warp ===============================
        // Loads the log-decays g of every chunk (a few chunks ahead), takes their in-warp prefix
        // sums and publishes one record per chunk: for the state pass (chunks last to first)
        // with the total of the later chunks, then for the output pass (chunks first to last)
        // with each chunk's plan. One warp decides every plan, so all roles follow the same one.
        GateRec *recA = reinterpret_cast<GateRec *>(sm + kGate);
        GateRec *recC = recA + kRecA;
        uint32_t us = 0, ja = 0, jc = 0;
        for (;;) {
            const uint32_t slot = us & 1;
            bool bad = !wait_or_abort(&unit_full[slot], (us >> 1) & 1, abort_v, status);
            if (__any_sync(0xffffffffu, bad)) break;
            const UnitInfo info = units[slot];
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&unit_empty[slot]);
            if (!info.valid) break;
            const int h = info.h, nch = info.nch;
            auto c0_of = [&](int c) { return info.t0 + int64_t(c) * kChunk; };
            auto nv_of = [&](int c) { return static_cast<int>(min(int64_t(kChunk), info.t1 - c0_of(c))); };
            // wait until the record slot is free again (its consumers have read the record of
            // kRec chunks before)
            auto claim = [&](uint64_t *empty_b, uint32_t n, int R) {
                const bool b = n >= static_cast<uint32_t>(R) &&
                               !wait_or_abort(&empty_b[n % R], ((n / R) - 1) & 1, abort_v, status);
                return !__any_sync(0xffffffffu, b);
            };
            // jobs 0 .. nch-1: state pass, chunks last to first; jobs nch .. 2 nch-1: output
            // pass, chunks first to last (log-decays loaded two jobs ahead)
            auto chunk_of = [&](int j) { return j < nch ? nch - 1 - j : j - nch; };
            bool ok = true;
            float2 g0 = load_gate(a.g, c0_of(chunk_of(0)), nv_of(chunk_of(0)), H, h);
            float2 g1 = load_gate(a.g, c0_of(chunk_of(1)), nv_of(chunk_of(1)), H, h);
            float D = 0.f, run = 0.f;
#pragma unroll 1
            for (int j = 0; j < 2 * nch; ++j) {
                const int c = chunk_of(j);
                const Gate G = scan_gate(g0, nv_of(c));
                g0 = g1;
                if (j + 2 < 2 * nch) g1 = load_gate(a.g, c0_of(chunk_of(j + 2)), nv_of(chunk_of(j + 2)), H, h);
                const bool state = j < nch;
                uint64_t *empty_b = state ? ga_empty : gc_empty;
                const uint32_t n = state ? ja : jc;
                const int R = state ? kRecA : kRecC;
                if (!(ok = claim(empty_b, n, R))) break;
                GateRec *rec = (state ? recA : recC) + n % R;
                *reinterpret_cast<float2 *>(&rec->b[2 * lane]) = make_float2(G.b0, G.b1);
                if (state) {
                    if (lane == 0) {
                        rec->bC = G.bC;
                        rec->D = D;
                    }
                    D += G.bC;
                } else {
                    const Plan P = plan_chunk(G, run);
                    if (lane == 0) {
                        rec->bC = G.bC;
                        rec->base = P.base;
                        rec->e1 = P.moved ? tc::ex2(P.pre * kLog2e) : 1.f;
                        rec->eC = P.fast ? 1.f : tc::ex2(G.bC * kLog2e);
                        rec->fast = P.fast;
                        rec->moved = P.moved;
                    }
                }
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(state ? &ga_full[n % R] : &gc_full[n % R]);
                if (state) ++ja; else ++jc;
            }
            if (!ok) break;
            ++us;
        }
    } else if (warp >= 4 && warp < 8) {
        // =============================== scaling warps ===============================
        // Thread wtid makes row s = wtid & 63, columns 64 * (wtid >> 6) .. + 64 of each K~ tile.
        const int wtid = threadIdx.x - 128;
        const int srow = wtid & 63, shalf = wtid >> 6;
        const int quarter = warp & 3;
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        constexpr int kBar = kBarScale;
        const uint64_t drop = tc::policy_evict_first();
        const GateRec *recA = reinterpret_cast<const GateRec *>(sm + kGate);
        const GateRec *recC = recA + kRecA;
        uint32_t us = 0, kpc = 0, cc = 0, job = 0;   // job: stage counter as the producer's
        uint32_t kfpar = 0;                          // bit st: phase parity of ka_full[st]
        uint32_t ja = 0, jc = 0;                     // gate records consumed
#ifdef SALA_TRACE
        unsigned long long wacc_[8] = {};
#endif

        // K rows of the output-pass chunk still to scale, loaded one chunk ahead into registers
        // (the scores of the current chunk are done in between). Thread wtid holds 16-byte
        // column kc16 of rows krow + 8 i, so that each load instruction of a warp reads two
        // whole 256-byte rows.
        const int krow = wtid >> 4, kc16 = wtid & 15;
        uint4 kx[8];
        auto prefetch = [&](int64_t c0, int nv, int h) {
            const uint8_t *src = reinterpret_cast<const uint8_t *>(a.k + ((c0 + krow) * H + h) * kD) + 16 * kc16;
            const size_t step = static_cast<size_t>(8) * H * kD * sizeof(uint16_t);   // 8 rows
#pragma unroll
            for (int i = 0; i < 8; ++i)
                kx[i] = krow + 8 * i < nv ? tc::ldg_nc_hint(src + i * step, drop) : make_uint4(0u, 0u, 0u, 0u);
        };
        // K~ of the chunk whose gate record is R into buffer kpc & 1: k exp(-(base + b_s))
        // (factored route) or k exp(b_C - b_s) plus the raw rows (exact route); rows >= nv zero.
        // The factor is rounded to bf16 and each pair takes one packed multiply.
        auto make_k = [&](const uint4 (&x)[8], const GateRec *R, int nv) {
            const uint32_t kb = kpc & 1;
#ifdef SALA_TRACE
            long long tw0 = clock64();
#endif
            wait_nv(&kp_free[kb], (kpc >> 1) - 1, kpc >= 2, abort_v, status);
#ifdef SALA_TRACE
            wacc_[0] += clock64() - tw0;
            tw0 = clock64();
#endif
            if (wtid == 0) TRACE(2, 9, kpc);
            const bool fast = R->fast != 0;
            const float off = fast ? -R->base : R->bC;
            uint8_t *dst = sm + kKp + kb * kTile + (kc16 >> 3) * kRegion;
            uint8_t *raw = sm + kKr + kb * kTile + (kc16 >> 3) * kRegion;
            // the warp's 16 rows (krow parity p, i = 0..7) each get their factor from one lane:
            // lane l computes row 2 (warp % 4) + (l & 1) + 8 ((l & 15) >> 1)
            const int lr = 2 * quarter + (lane & 1) + 8 * ((lane & 15) >> 1);
            const float myfac = lr < nv ? tc::ex2((off - R->b[lr]) * kLog2e) : 0.f;
            const int par = lane >> 4;   // krow = 2 (warp % 4) + par
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int row = krow + 8 * i;
                const float fac = __shfl_sync(0xffffffffu, myfac, 2 * i + par);
                const __nv_bfloat162 f2 = __float2bfloat162_rn(fac);
                uint4 y;
                y.x = mul_bf16x2(x[i].x, f2);
                y.y = mul_bf16x2(x[i].y, f2);
                y.z = mul_bf16x2(x[i].z, f2);
                y.w = mul_bf16x2(x[i].w, f2);
                *reinterpret_cast<uint4 *>(dst + sw(row, kc16 & 7)) = y;
                if (!fast) *reinterpret_cast<uint4 *>(raw + sw(row, kc16 & 7)) = x[i];
            }
            if (wtid == 0) TRACE(2, 10, kpc);
            if (wtid == 0) kfast[kb] = fast;
            tc::fence_proxy_async_smem();
            warp_arrive(&kp_ready[kb]);
#ifdef SALA_TRACE
            wacc_[1] += clock64() - tw0;
#endif
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
            // the tensor core only runs the short state-pass products). These warps take
            // columns 0-63, the converting warps (idle until the hand-off) 64-127.
            for (int r = 0; r < nch; ++r) {
                const int nv = chunk_nv(nch - 1 - r);
                const uint32_t st = job % kStages;
                if (wtid == 0) TRACE(2, 1, r);
                wait_nv(&ga_full[ja % kRecA], ja / kRecA, true, abort_v, status);
                const GateRec *R = recA + ja % kRecA;
                const float e = R->bC + R->D - R->b[srow];
                warp_arrive(&ga_empty[ja % kRecA]);
                ++ja;
                const float fac = srow < nv ? tc::ex2(e * kLog2e) : 0.f;
                wait_nv(&ka_full[st], (kfpar >> st) & 1, true, abort_v, status);
                kfpar ^= 1u << st;
                if (wtid == 0) TRACE(2, 7, r);
                scale_k_quarter(sm + st * kStage, srow, shalf, fac);
                tc::fence_proxy_async_smem();
                warp_arrive(&ka_ready[st]);
                if (wtid == 0) TRACE(2, 8, r);
                ++job;
            }
            prefetch(chunk_c0(0), chunk_nv(0), h);

            // ---------------- C ----------------
            // K~ of chunk 0; then per chunk: K~ of the next chunk, P' of this one. The scaling
            // warps wait on every stage phase (mbarrier waits compare parity only, so a waiter
            // must not skip phases), although here they read K with ordinary global loads.
            // (these warps read K with ordinary global loads and wait on no stage: the scores of
            // a chunk imply that its Q tile has landed)
            const uint32_t job_c = job, jc0 = jc;
            // the gate record of chunk c (held from its K~ until its P' is done)
            auto rec = [&](int c) { return recC + (jc0 + c) % kRecC; };
            auto wait_rec = [&](int c) {
                wait_nv(&gc_full[(jc0 + c) % kRecC], (jc0 + c) / kRecC, true, abort_v, status);
            };
            for (int c = -1; c < nch; ++c) {
                if (c + 1 < nch) {
                    wait_rec(c + 1);
                    make_k(kx, rec(c + 1), chunk_nv(c + 1));
                    if (c + 2 < nch) prefetch(chunk_c0(c + 2), chunk_nv(c + 2), h);
                    if (wtid == 0) TRACE(2, 3, c);
                }
                if (c < 0) continue;
                const int nv = chunk_nv(c);
                const GateRec *R = rec(c);
                // scores -> P' (bf16, K-major rows t): mask s <= t < nv; exact route weights
                const bool fast = R->fast != 0;
#ifdef SALA_TRACE
                long long tw1 = clock64();
#endif
                wait_nv(&p_full, cc, true, abort_v, status);
#ifdef SALA_TRACE
                wacc_[2] += clock64() - tw1;
                tw1 = clock64();
#endif
                wait_nv(&pp_free, cc - 1, cc >= 1, abort_v, status);
#ifdef SALA_TRACE
                wacc_[3] += clock64() - tw1;
                tw1 = clock64();
#endif
                if (wtid == 0) TRACE(2, 5, c);
                tc::tc_fence_after();
                // M=64 accumulator layout: rows t = 16 quarter + (lane & 15) in lanes 0-15 of the
                // quarter; the 16-lane load gives lanes 0-15 columns s = 0-31 of those rows and
                // lanes 16-31 columns 32-63
                const int tr = quarter * 16 + (lane & 15), sh = lane >> 4;
                uint8_t *pp = sm + kPp;
                {
                    uint32_t p[32];
                    tc::tmem_ld_16x32bx2_x32(tmem + lane_base + kTP, p);
                    tc::tmem_ld_wait();
                    if (wtid == 0) TRACE(2, 20, c);
                    tc::tc_fence_before();
                    warp_arrive(&p_free);
                    const bool live = tr < nv;
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) {
                        uint32_t w[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int si = 8 * c4 + 2 * e, s = 32 * sh + si;
                            const float f0 = (live && s <= tr) ? __uint_as_float(p[si]) : 0.f;
                            const float f1 = (live && s + 1 <= tr) ? __uint_as_float(p[si + 1]) : 0.f;
                            w[e] = float2_to_bf16x2(f0, f1);
                        }
                        *reinterpret_cast<uint4 *>(pp + sw(tr, 4 * sh + c4)) = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                    if (wtid == 0) TRACE(2, 23, c);
                }
                if (!fast) {
                    // exact route: P'[t, s] *= exp(b_t - b_s); q_t <- exp(b_t) q_t in place (M1
                    // has read Q already; the rows come from global memory, not from the tile)
                    if (tr < nv) exact_pp_weights(pp, R->b, tr, sh);
                    exact_q_scale(sm + ((job_c + c) % kStages) * kStage + shalf * kRegion,
                                  reinterpret_cast<const uint16_t *>(a.q), chunk_c0(c), srow, shalf,
                                  nv, H, h, R->b[srow]);
                }
                warp_arrive(&gc_empty[(jc0 + c) % kRecC]);   // done with chunk c's record
                tc::fence_proxy_async_smem();
                warp_arrive(&pp_ready);
                if (wtid == 0) TRACE(2, 6, c);
#ifdef SALA_TRACE
                wacc_[4] += clock64() - tw1;
#endif
                ++cc;
            }
            // one uniform decision per unit (after an abort every wait returns at once, so all
            // threads still pass the same barriers inside the unit)
            if (named_any(kBar, 128, *abort_v != 0)) break;
            job = job_c + nch;
            jc = jc0 + nch;
            ++us;
        }
#ifdef SALA_TRACE
        if (blockIdx.x == 0 && wtid == 0)
            for (int i = 0; i < 6; ++i) g_wait_acc[16 + i] = wacc_[i];
#endif
    } else if (warp >= 8 && warp < 12) {
        // =============================== converting warps ===============================
        // Thread j (= TMEM lane) owns row j of Z^T: all 128 keys i, handled 32 at a time.
        // Waits inside a unit do not vote: a thread whose wait gives up has set the abort flag,
        // and every later wait returns at once, so all threads still pass the same barriers;
        // one OR-vote per hand-off and per unit then ends the loop uniformly.
        const int wtid = threadIdx.x - 256;
        const int quarter = warp & 3;
        const int j = quarter * 32 + lane;     // value column = TMEM lane
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        uint32_t us = 0, zfc = 0, zbc = 0, npub = 0, jc = 0;
        uint32_t job = 0, ja = 0, kfpar = 0;   // stage jobs seen, state-pass records, ka_full parity
        const int arow = wtid & 63;           // state-pass row (columns 64 + 32 (wtid >> 6) .. + 31)
        const GateRec *recC = reinterpret_cast<const GateRec *>(sm + kGate) + kRecA;
        const GateRec *recA = reinterpret_cast<const GateRec *>(sm + kGate);
        // the plan of the next chunk from its gate record (released at once)
        struct ConvPlan {
            float e1, eC;
            bool fast, moved;
        };
        auto next_plan = [&]() {
            wait_nv(&gc_full[jc % kRecC], jc / kRecC, true, abort_v, status);
            const GateRec *R = recC + jc % kRecC;
            ConvPlan cp{R->e1, R->eC, R->fast != 0, R->moved != 0};
            warp_arrive(&gc_empty[jc % kRecC]);
            ++jc;
            return cp;
        };

        // bf16 copy of 32 keys (one quarter of the row) into the A operand of M2
        auto store_zb = [&](int k4, const float (&x)[32], float fac) {
            uint32_t w[16];
#pragma unroll
            for (int m = 0; m < 16; ++m) w[m] = float2_to_bf16x2(x[2 * m] * fac, x[2 * m + 1] * fac);
            tc::tmem_st_32x32b_x16(tmem + lane_base + zb_col(zbc & 1) + 16 * k4, w);
        };
        auto store_z = [&](int k4, const float (&x)[32], float fac) {
            uint32_t w[32];
#pragma unroll
            for (int m = 0; m < 32; ++m) w[m] = __float_as_uint(x[m] * fac);
            tc::tmem_st_32x32b_x32(tmem + lane_base + kTZ + 32 * k4, w);
        };

        for (;;) {
            const uint32_t slot = us & 1;
            if (!wg_wait(&unit_full[slot], us >> 1, true, kBarConv, abort_v, status)) break;
            const UnitInfo info = units[slot];
            named_sync(kBarConv, 128);
            if (wtid == 0) tc::mbar_arrive(&unit_empty[slot]);
            if (!info.valid) break;
            const int h = info.h, nch = info.nch;
            if (lane == 0) TRACE(quarter == 0 ? 3 : 4 + quarter, 1, us);
            // a first segment's incoming state is the caller's h0, known from the start: bring
            // its 64 KB into L2 during the state pass (the hand-off reads it 32 rows at a time)
            if (info.first && f.h0) {
                const char *hb = reinterpret_cast<const char *>(f.h0 + (info.n * H + h) * kD * kD);
                for (int i = wtid; i < kD * kD * 4 / 128; i += 128) tc::prefetch_l2_keep(hb + 128 * i);
            }

            // ---------------- state pass: columns 64-127 of every K' tile ----------------
            // (the scaling warps take columns 0-63); and the segment's total log-decay
            float D = 0.f;
#pragma unroll 1
            for (int r = 0; r < nch; ++r) {
                const int64_t c0 = info.t0 + int64_t(nch - 1 - r) * kChunk;
                const uint32_t st = (job + r) % kStages;
                wait_nv(&ga_full[ja % kRecA], ja / kRecA, true, abort_v, status);
                const GateRec *R = recA + ja % kRecA;
                const float e = R->bC + R->D - R->b[arow];
                D += R->bC;
                warp_arrive(&ga_empty[ja % kRecA]);
                ++ja;
                const float fac = c0 + arow < info.t1 ? tc::ex2(e * kLog2e) : 0.f;
                wait_nv(&ka_full[st], (kfpar >> st) & 1, true, abort_v, status);
                kfpar ^= 1u << st;
                scale_k_quarter(sm + st * kStage, arow, 2 + (wtid >> 6), fac);
                tc::fence_proxy_async_smem();
                warp_arrive(&ka_ready[st]);
            }
            job += 2 * nch;

            // ---------------- hand-off: S_in, Z = S_in and its bf16 copy, publish S_out ----------------
            {
                bool bad = !wait_or_abort(&ds_full, us & 1, abort_v, status);
                if (lane == 0) TRACE(quarter == 0 ? 3 : 4 + quarter, 11, us);
                if (!bad && !info.first && wtid == 0) {
                    const uint32_t *flag = f.flags + (info.sigma - 1) * H + h;
                    const uint64_t t0ns = tc::global_timer_ns();
                    while (tc::ld_acquire_gpu(flag) != f.epoch) {
                        if (*abort_v) { bad = true; break; }
                        if (tc::global_timer_ns() - t0ns > f.flag_wait_ns) {
                            *abort_v = 1;
                            record_status(status, SALA_ERR_TIMEOUT);
                            bad = true;
                            break;
                        }
                    }
                }
                if (named_any(kBarConv, 128, bad || *abort_v)) break;
                if (lane == 0) TRACE(quarter == 0 ? 3 : 4 + quarter, 2, 0);
                tc::tc_fence_after();
                // chunk 0 starts at the reference point (pre = 0); the exact route keeps the
                // state scaled to the chunk end
                const float zfac = next_plan().eC;
                const float eB = tc::ex2(D * kLog2e);
                float *dst = info.last ? (f.hT ? f.hT + (info.n * H + h) * kD * kD : nullptr)
                                       : f.incl + (static_cast<size_t>(info.sigma) * H + h) * kD * kD;
                const float *src = info.first
                    ? (f.h0 ? f.h0 + (info.n * H + h) * kD * kD : nullptr)
                    : f.incl + (static_cast<size_t>(info.sigma - 1) * H + h) * kD * kD;
                // (the second bf16 buffer overlays dS^T columns 0-63: quarter k4 writes columns
                // 16 k4 .. + 15, which quarters 0 and 1 have read already)
                wait_nv(&zb_free[zbc & 1], (zbc >> 1) - 1, zbc >= 2, abort_v, status);
#pragma unroll 1
                for (int k4 = 0; k4 < 4; ++k4) {
                    // S_in[i][j] for i = 32 k4 .. + 31: another SM wrote it, so read through L2
                    float s[32];
                    if (src) {
                        const float *p = src + (32 * k4) * kD + j;
#pragma unroll
                        for (int i = 0; i < 32; ++i) s[i] = __ldcg(p + i * kD);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) s[i] = 0.f;
                    }
                    uint32_t d[32];
                    tc::tmem_ld_32x32b_x32(tmem + lane_base + kTdS + 32 * k4, d);
                    tc::tmem_ld_wait();
                    if (dst) {
                        // S_out = exp(B) S_in + dS: each warp store covers one 128-byte row segment
                        float *p = dst + (32 * k4) * kD + j;
#pragma unroll
                        for (int i = 0; i < 32; ++i) p[i * kD] = fmaf(eB, s[i], __uint_as_float(d[i]));
                    }
                    store_z(k4, s, zfac);
                    store_zb(k4, s, 1.f);
                }
                tc::tmem_st_wait();
                tc::tc_fence_before();
                warp_arrive(&ds_free);
                if (nch > 1) warp_arrive(&z_free);
                warp_arrive(&zb_ready[zbc & 1]);
                ++zbc;
                // the publisher releases the flag once all four warps have stored S_out
                wait_nv(&pub_free, npub - 1, npub >= 1, abort_v, status);
                if (wtid == 0) {
                    pub_cmd = info.last ? 0 : 1;
                    pub_flag = f.flags + info.sigma * H + h;
                }
                warp_arrive(&pub_ready);
                ++npub;
                if (wtid == 0) TRACE(3, 3, 0);

                // ---------------- C: the state entering each later chunk ----------------
                for (int c = 1; c < nch; ++c) {
                    const ConvPlan P = next_plan();
                    if (lane == 0) TRACE(quarter == 0 ? 3 : 4 + quarter, 12, c);
                    wait_nv(&z_full, zfc, true, abort_v, status);   // M4 of chunk c - 1 is done
                    ++zfc;
                    if (lane == 0) TRACE(quarter == 0 ? 3 : 4 + quarter, 4, c);
                    tc::tc_fence_after();
                    // stored state -> true state at the chunk start: exp(pre); the stored state
                    // keeps that (moved reference) or goes on to the chunk end (exact route).
                    // Z is read (and rescaled) first and released to the next M4 at once; the
                    // bf16 copy waits for M2 of the previous chunk to have read the old one.
                    const float e1 = P.e1, eC = P.eC;
                    // keys 64 k2 .. + 63 of Z, as the true state at the chunk start
                    // keys 64 k2 .. + 63 of Z: to the true state at the chunk start (times e1),
                    // its bf16 copy into the A operand of M2 (the buffer M2 of two chunks before
                    // has read), and, if the reference moved, the stored state itself (times eC on
                    // the exact route: on to the chunk end). One path for every route.
                    const uint32_t zb_base = tmem + lane_base + zb_col(zbc & 1);
                    wait_nv(&zb_free[zbc & 1], (zbc >> 1) - 1, zbc >= 2, abort_v, status);
                    tc::tc_fence_after();
#pragma unroll 1
                    for (int k2 = 0; k2 < 2; ++k2) {
                        uint32_t d0[32], d1[32];
                        tc::tmem_ld_32x32b_x32(tmem + lane_base + kTZ + 64 * k2, d0);
                        tc::tmem_ld_32x32b_x32(tmem + lane_base + kTZ + 64 * k2 + 32, d1);
                        tc::tmem_ld_wait();
                        uint32_t w[16];
                        if (P.moved) {
#pragma unroll
                            for (int m = 0; m < 16; ++m)
                                w[m] = float2_to_bf16x2(__uint_as_float(d0[2 * m]) * e1, __uint_as_float(d0[2 * m + 1]) * e1);
                            tc::tmem_st_32x32b_x16(zb_base + 32 * k2, w);
#pragma unroll
                            for (int m = 0; m < 16; ++m)
                                w[m] = float2_to_bf16x2(__uint_as_float(d1[2 * m]) * e1, __uint_as_float(d1[2 * m + 1]) * e1);
                            tc::tmem_st_32x32b_x16(zb_base + 32 * k2 + 16, w);
                        } else {
#pragma unroll
                            for (int m = 0; m < 16; ++m)
                                w[m] = float2_to_bf16x2(__uint_as_float(d0[2 * m]), __uint_as_float(d0[2 * m + 1]));
                            tc::tmem_st_32x32b_x16(zb_base + 32 * k2, w);
#pragma unroll
                            for (int m = 0; m < 16; ++m)
                                w[m] = float2_to_bf16x2(__uint_as_float(d1[2 * m]), __uint_as_float(d1[2 * m + 1]));
                            tc::tmem_st_32x32b_x16(zb_base + 32 * k2 + 16, w);
                        }
                        if (P.moved) {
                            const float e2 = e1 * eC;
#pragma unroll
                            for (int i = 0; i < 32; ++i) {
                                d0[i] = __float_as_uint(__uint_as_float(d0[i]) * e2);
                                d1[i] = __float_as_uint(__uint_as_float(d1[i]) * e2);
                            }
                            tc::tmem_st_32x32b_x32(tmem + lane_base + kTZ + 64 * k2, d0);
                            tc::tmem_st_32x32b_x32(tmem + lane_base + kTZ + 64 * k2 + 32, d1);
                        }
                    }
                    tc::tmem_st_wait();
                    tc::tc_fence_before();
                    if (c + 1 < nch) warp_arrive(&z_free);
                    if (lane == 0) TRACE(quarter == 0 ? 3 : 4 + quarter, 5, c);
                    warp_arrive(&zb_ready[zbc & 1]);
                    ++zbc;
                    if (lane == 0) TRACE(quarter == 0 ? 3 : 4 + quarter, 8, c);
                }
            }
            if (named_any(kBarConv, 128, *abort_v != 0)) break;
            ++us;
        }
        // stop the publisher (after an abort it stops by itself)
        if (!named_any(kBarConv, 128, *abort_v != 0)) {
            wait_nv(&pub_free, npub - 1, npub >= 1, abort_v, status);
            if (wtid == 0) pub_cmd = 2;
            warp_arrive(&pub_ready);
        }
    } else if (warp >= 12) {
        // =============================== output warps ===============================
        // Warp quarter q writes value columns j = 32 q .. + 31 of every token: o_t = factor_t
        // O^T[j][t], staged as a [64 t x 32 j] bf16 tile (64-byte swizzle) and written by one
        // TMA store per warp (direct stores when the chunk is ragged: the rows past it belong
        // to another sequence). O^T is read in the 16-lane fragment order, in which each lane
        // holds two neighbouring tokens of one value column, so transposing 8 x 8 matrix
        // stores put the tile in place without any exchange between lanes.
        const int wtid = threadIdx.x - 384;
        const int quarter = warp & 3;
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        uint8_t *stg = sm + kOst + quarter * kOstWarp;
        // this lane's row address for each stmatrix: matrix k = lane / 8 (value columns
        // 8 k .. + 7 of the warp's 32), row p = lane % 8 (token 8 m + p), 16-byte chunk k
        // swizzled by token bits 2..1
        const int p8 = lane & 7, k8 = lane >> 3;
        const uint32_t st_addr = tc::smem_u32(stg) + p8 * 64 + 16 * (k8 ^ ((p8 >> 1) & 3));
        const int tl = 2 * (lane & 3);   // this lane's tokens: 8 m + tl, 8 m + tl + 1
        const GateRec *recC = reinterpret_cast<const GateRec *>(sm + kGate) + kRecA;
        uint32_t us = 0, cc = 0, jc = 0;
        for (;;) {
            const uint32_t slot = us & 1;
            if (!wg_wait(&unit_full[slot], us >> 1, true, kBarOut, abort_v, status)) break;
            const UnitInfo info = units[slot];
            named_sync(kBarOut, 128);
            if (wtid == 0) tc::mbar_arrive(&unit_empty[slot]);
            if (!info.valid) break;
            const int h = info.h, nch = info.nch;
            for (int c = 0; c < nch; ++c) {
                const int64_t c0 = info.t0 + int64_t(c) * kChunk;
                const int nv = static_cast<int>(min(int64_t(kChunk), info.t1 - c0));
                // the factors of this lane's 16 tokens, from the chunk's gate record
                wait_nv(&gc_full[jc % kRecC], jc / kRecC, true, abort_v, status);
                const GateRec *R = recC + jc % kRecC;
                const bool fast = R->fast != 0;
                const float base = R->base;
                float2 ft[8];
#pragma unroll
                for (int m = 0; m < 8; ++m) ft[m] = *reinterpret_cast<const float2 *>(&R->b[8 * m + tl]);
                warp_arrive(&gc_empty[jc % kRecC]);
                ++jc;
#pragma unroll
                for (int m = 0; m < 8; ++m)
                    ft[m] = fast ? make_float2(a.scale * tc::ex2((base + ft[m].x) * kLog2e),
                                               a.scale * tc::ex2((base + ft[m].y) * kLog2e))
                                 : make_float2(a.scale, a.scale);
                const uint32_t ob = cc & 1;
                wait_nv(&o_full[ob], cc >> 1, true, abort_v, status);
                if (wtid == 0) TRACE(4, 9, c);
                tc::tc_fence_after();
                // o0: value columns 0-15 of the warp's 32, o1: 16-31
                uint32_t o0[32], o1[32];
                tc::tmem_ld_16x256b_x8(tmem + lane_base + kTO + 64 * ob, o0);
                tc::tmem_ld_16x256b_x8(tmem + lane_base + (16u << 16) + kTO + 64 * ob, o1);
                tc::tmem_ld_wait();
                tc::tc_fence_before();
                warp_arrive(&o_free[ob]);
                if (lane == 0) tc::tma_store_wait_read<0>();   // staging tile free again
                __syncwarp();
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    const float fa = ft[m].x, fb = ft[m].y;
                    tc::stmatrix_x4_trans(st_addr + 512 * m,
                                          float2_to_bf16x2(__uint_as_float(o0[4 * m]) * fa, __uint_as_float(o0[4 * m + 1]) * fb),
                                          float2_to_bf16x2(__uint_as_float(o0[4 * m + 2]) * fa, __uint_as_float(o0[4 * m + 3]) * fb),
                                          float2_to_bf16x2(__uint_as_float(o1[4 * m]) * fa, __uint_as_float(o1[4 * m + 1]) * fb),
                                          float2_to_bf16x2(__uint_as_float(o1[4 * m + 2]) * fa, __uint_as_float(o1[4 * m + 3]) * fb));
                }
                if (nv == kChunk) {
                    tc::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tc::tma_store_3d(&maps.o, 32 * quarter, h, static_cast<int32_t>(c0), stg);
                        tc::tma_store_commit();
                    }
                } else if (dcheck(nv > 0 && c0 + nv <= info.t1, status)) {
                    // ragged chunk: only its nv rows go out (the rows past it belong to another
                    // sequence), 64 bytes per row
                    __syncwarp();
                    uint16_t *orow = a.o + (c0 * H + h) * kD + 32 * quarter + lane;
#pragma unroll 1
                    for (int tt = 0; tt < nv; ++tt)
                        orow[static_cast<size_t>(tt) * H * kD] = *reinterpret_cast<const uint16_t *>(
                            stg + tt * 64 + 16 * ((lane >> 3) ^ ((tt >> 1) & 3)) + 2 * (lane & 7));
                }
                if (wtid == 0) TRACE(4, 10, c);
                ++cc;
            }
            if (named_any(kBarOut, 128, *abort_v != 0)) break;
            ++us;
        }
        if (lane == 0) tc::tma_store_wait_all<0>();
    }

    tc::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, kTCols);
    }
}
// ---------------------------------------------------------------------------------------
// host side

namespace tck {

namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
cudaError_t g_encode_err = cudaSuccess;
std::once_flag g_encode_once;

cudaError_t encode_map(CUtensorMap *map, const void *base, int64_t T_total, int H, bool store,
                       bool sw64 = false) {
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
    cuuint32_t box_load[3] = {64, 1, 64}, box_store[3] = {32, 1, 64};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims,
                          strides, store ? box_store : box_load, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE,
                          store ? (sw64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_NONE)
                                : CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}
}  // namespace

cudaError_t make_maps(TcMaps *m, const void *q, const void *k, const void *v, const void *o,
                      int64_t T_total, int H, bool o_sw64) {
    cudaError_t e = encode_map(&m->q, q, T_total, H, false);
    if (e == cudaSuccess) e = encode_map(&m->k, k, T_total, H, false);
    if (e == cudaSuccess) e = encode_map(&m->v, v, T_total, H, false);
    if (e == cudaSuccess) e = encode_map(&m->o, o, T_total, H, true, o_sw64);
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
        cudaError_t e = tck::make_maps(&maps, a.q, a.k, a.v, a.o, T_total, a.H, true);
        if (e != cudaSuccess) return e;
        PrefillArgs f;
        f.c = a;
        f.h0 = h0;
        f.hT = hT;
        f.incl = incl;
        f.flags = flags;
        f.ticket = ticket;
        f.epoch = epoch;
        uint64_t wait_ns = 0;
        int64_t withhold = -1;
        prefill_fault_knobs(&wait_ns, &withhold);
        f.flag_wait_ns = wait_ns ? wait_ns : kWaitNs;
        f.withheld = (withhold >= 0 && withhold < max_units) ? flags + withhold : nullptr;
        if (grid > max_units) grid = static_cast<int>(max_units);
        LaunchTimer timer(kKPrefillFused, st);
        // programmatic dependent launch: the kernel's set-up may overlap the segment-table
        // kernel before it on the stream (griddepcontrol.wait orders the rest)
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(grid));
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = kSmemAlloc;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, prefill_fused_kernel, maps, f, t, status);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace sala

#ifdef SALA_TRACE
extern "C" int sala_gla_debug_wait_acc(unsigned long long *out) {
    return cudaMemcpyFromSymbol(out, sala::g_wait_acc, sizeof(sala::g_wait_acc)) == cudaSuccess ? 0 : -1;
}
extern "C" void sala_gla_debug_wait_reset() {
    static unsigned long long z[32] = {};
    cudaMemcpyToSymbol(sala::g_wait_acc, z, sizeof(z));
}
extern "C" int sala_gla_debug_trace(unsigned long long *out, int max) {
    unsigned int n[8];
    if (cudaMemcpyFromSymbol(n, sala::g_trace_n, sizeof(n)) != cudaSuccess) return -1;
    static unsigned long long buf[8][sala::kTraceN];
    if (cudaMemcpyFromSymbol(buf, sala::g_trace, sizeof(buf)) != cudaSuccess) return -1;
    int k = 0;
    for (int r = 0; r < 8; ++r)
        for (unsigned i = 0; i < n[r] && i < static_cast<unsigned>(sala::kTraceN) && k < max; ++i)
            out[k++] = buf[r][i];
    return k;
}
#endif
