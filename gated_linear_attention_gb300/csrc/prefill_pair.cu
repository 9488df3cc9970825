// Chunked prefill at two CTAs per SM.
//
// The algorithm is the one of prefill_fused.cu: the recurrence of "MiniCPM-SALA — Complete
// Blueprint", "Simple GLA Recurrence", in the chunked form of "Formulas and Code for Adapting
// Inference to GDN/KDA Linear Modules", section 1.2 (beta = 1, no delta rule), with a state
// pass per segment, a chained hand-off of the incoming state between consecutive segments and
// an output pass that keeps the state in tensor memory relative to a reference point. What
// differs is the machine layout. Here a CTA holds one unit (segment, head) at a time in half of
// an SM's shared memory (108 KB) and tensor memory (256 columns), so two CTAs share every SM and
// each one's serial chain of products, conversions and waits overlaps the other's.
//
// Tensor memory: Z^T in fp32 (128 columns; the state pass accumulates dS^T there and the
// hand-off replaces it by Z), its bf16 copy (64 columns, the A operand of M2), and 64 columns
// that hold a chunk's scores P until they are read, then its output O^T.
// Shared memory is one 104 KB region used by phase. The state pass streams the K | V tiles of
// its chunks through three 32 KB slots. The output pass holds Q [2], V [2], K~ (on the exact
// route the raw keys until M1 has read them, then the weighted ones), P' and the o staging.
//
// Per output chunk c the products go out as
//   M1  P    = Q K~^T      M=64  N=64  K=128   (once K~(c) is made and O^T(c-1) has been read)
//   M4  Z^T += V^T K~      M=128 N=128 K=64    (not after the last chunk; once Z was copied)
//   M2  O^T  = Z^T Q^T     M=128 N=64  K=128   (A = the bf16 copy of Z^T; once P' is made)
//   M3  O^T += V^T P'^T    M=128 N=64  K=64
// Roles (256 threads): warp 0 loads by TMA, warp 1 issues the products and owns the tensor
// memory, warp 2 reads g ahead and publishes each chunk's prefix sums and plan, warp 3 releases
// the hand-off flags, warps 4-7 (the workers) do the CUDA-core steps in order: the scaled keys
// of the state pass, the hand-off, then per chunk K~, P', the bf16 copy of the next chunk's
// state and the output epilogue. Every wait is bounded (2 s of %globaltimer); a timeout
// records SALA_ERR_TIMEOUT, stops the CTA's work, drains its copies and products, frees its
// tensor memory and returns.
#include "prefill_common.cuh"

namespace sala {
namespace {

using namespace tck;

constexpr int kPThreads = 256;

// dynamic shared memory (offsets from a 1024-aligned base)
constexpr uint32_t kPSlot = 2 * kTile;             // state pass: K | V of one chunk
constexpr int kPSlots = 3;
constexpr uint32_t kPQ = 0;                        // output pass: Q [2]
constexpr uint32_t kPV = 2 * kTile;                // V [2]
constexpr uint32_t kPK = 4 * kTile;                // K~ (raw K first on the exact route)
constexpr uint32_t kPP = 5 * kTile;                // P' (K-major B of M3)
constexpr uint32_t kPO = kPP + kRegion;            // o staging, per worker warp [64 t][32 j]
constexpr uint32_t kPOWarp = 64 * 64;
constexpr uint32_t kPRing = kPO + 4 * kPOWarp;
constexpr uint32_t kPGate = kPRing;                // gate records: state pass, output pass
constexpr int kPRecA = 4, kPRecC = 8;
constexpr uint32_t kPBytes = kPGate + (kPRecA + kPRecC) * 288;
constexpr uint32_t kPSmemAlloc = kPBytes + 1024;
static_assert(kPSlots * kPSlot <= kPRing, "state-pass slots fit the region");
static_assert(2 * (kPSmemAlloc + 1024 + 1024) <= 228 * 1024, "two CTAs per SM");

// tensor-memory columns
constexpr uint32_t kPtZ = 0, kPtZb = 128, kPtPO = 192, kPtCols = 256;
constexpr uint32_t kIdP = tc::idesc_bf16_f32(64, 64, 0, 0);
constexpr uint32_t kIdO2 = tc::idesc_bf16_f32(128, 64, 0, 0);
constexpr uint32_t kIdO3 = tc::idesc_bf16_f32(128, 64, 1, 0);
constexpr uint32_t kIdS = tc::idesc_bf16_f32(128, 128, 1, 1);

constexpr int kBarW = 1;   // named barrier of the four worker warps

// Event trace of CTA 0 for latency analysis (compiled only with -DSALA_TRACE): SM clock, role,
// event id and chunk index, written to a global array.
#ifdef SALA_TRACE
constexpr int kPTraceN = 1024;
__device__ unsigned long long g_ptrace[4][kPTraceN];
__device__ unsigned int g_ptrace_n[4];
#define PTRACE(role, ev, idx)                                                                   \
    do {                                                                                        \
        if (blockIdx.x == 0 && ptr_i < kPTraceN) {                                              \
            g_ptrace[role][ptr_i] = (static_cast<unsigned long long>(clock64()) & 0xFFFFFFFFFFFFull) | \
                                    (static_cast<unsigned long long>(role) << 60) |             \
                                    (static_cast<unsigned long long>(ev) << 52) |               \
                                    (static_cast<unsigned long long>((idx) & 0xF) << 48);       \
            ++ptr_i;                                                                            \
            g_ptrace_n[role] = ptr_i;                                                           \
        }                                                                                       \
    } while (0)
#else
#define PTRACE(role, ev, idx) \
    do {                      \
    } while (0)
#endif





// Two 8 x 8 bf16 matrices stored transposed (lanes 0-15 give the row addresses).
__device__ __forceinline__ void pstmatrix_x2_trans(uint32_t saddr, uint32_t r0, uint32_t r1) {
    asm volatile("stmatrix.sync.aligned.m8n8.x2.trans.shared.b16 [%0], {%1, %2};" ::"r"(saddr), "r"(r0),
                 "r"(r1)
                 : "memory");
}

// Exact route: row `row` (columns 64 half .. + 63) of the tile at dst becomes exp(f_row) x_row
// for the bf16 rows of global memory at src (zero past nv). Used for q_t <- exp(b_t) q_t (M1 has
// read Q) and for the weighted keys k_s exp(b_C - b_s) of M4 (M1 has read the raw ones).
__device__ __noinline__ void pexact_rows(uint8_t *dst, const uint16_t *src, int64_t c0, int row, int half,
                                         int nv, int H, int h, float f_row) {
    uint4 x[8];
    if (row < nv) {
        const uint4 *p = reinterpret_cast<const uint4 *>(src + ((c0 + row) * H + h) * kD + 64 * half);
        for (int c8 = 0; c8 < 8; ++c8) x[c8] = p[c8];
    } else {
        for (int c8 = 0; c8 < 8; ++c8) x[c8] = make_uint4(0u, 0u, 0u, 0u);
    }
    const __nv_bfloat162 f2 = __float2bfloat162_rn(row < nv ? tc::ex2(f_row * kLog2e) : 0.f);
    uint8_t *base = dst + half * kRegion;
    for (int c8 = 0; c8 < 8; ++c8) {
        uint4 y;
        y.x = mul_bf16x2(x[c8].x, f2);
        y.y = mul_bf16x2(x[c8].y, f2);
        y.z = mul_bf16x2(x[c8].z, f2);
        y.w = mul_bf16x2(x[c8].w, f2);
        *reinterpret_cast<uint4 *>(base + sw(row, c8)) = y;
    }
}

}  // namespace

__global__ void __launch_bounds__(kPThreads, 2)
prefill_pair_kernel(const __grid_constant__ TcMaps maps, PrefillArgs f, SegTable t, int *status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
    __shared__ uint64_t unit_full[2], unit_empty[2], unit_free;
    __shared__ uint64_t ka_full[kPSlots], ka_ready[kPSlots], slot_free[kPSlots], ds_full;
    __shared__ uint64_t q_full[2], v_full[2], q_free[2], v_free[2];
    __shared__ uint64_t kp_ready, kp_free, p_full, pp_ready, zb_ready, zb_free, z_full, o_full, po_free;
    __shared__ uint64_t ga_full[kPRecA], ga_empty[kPRecA], gc_full[kPRecC], gc_empty[kPRecC];
    __shared__ uint64_t pub_ready, pub_free, drain;
    __shared__ UnitInfo units[2];
    __shared__ int kfast;
    __shared__ uint32_t *pub_flag;
    __shared__ int pub_cmd;          // 0: nothing this unit, 1: release pub_flag, 2: stop
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;
#ifdef SALA_TRACE
    unsigned ptr_i = 0;
#endif

    const ChunkArgs &a = f.c;
    const int H = a.H;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(&unit_full[i], 1);
            tc::mbar_init(&unit_empty[i], 3);   // MMA, gate and worker warps
            tc::mbar_init(&q_full[i], 1);
            tc::mbar_init(&v_full[i], 1);
            tc::mbar_init(&q_free[i], 1);
            tc::mbar_init(&v_free[i], 1);
        }
        tc::mbar_init(&unit_free, 5);           // MMA commit, four worker warps
        for (int s = 0; s < kPSlots; ++s) {
            tc::mbar_init(&ka_full[s], 1);
            tc::mbar_init(&ka_ready[s], 4);
            tc::mbar_init(&slot_free[s], 1);
        }
        tc::mbar_init(&ds_full, 1);
        tc::mbar_init(&kp_ready, 4);
        tc::mbar_init(&kp_free, 1);
        tc::mbar_init(&p_full, 1);
        tc::mbar_init(&pp_ready, 4);
        tc::mbar_init(&zb_ready, 4);
        tc::mbar_init(&zb_free, 1);
        tc::mbar_init(&z_full, 1);
        tc::mbar_init(&o_full, 1);
        tc::mbar_init(&po_free, 4);
        for (int i = 0; i < kPRecA; ++i) {
            tc::mbar_init(&ga_full[i], 1);
            tc::mbar_init(&ga_empty[i], 4);
        }
        for (int i = 0; i < kPRecC; ++i) {
            tc::mbar_init(&gc_full[i], 1);
            tc::mbar_init(&gc_empty[i], 4);
        }
        tc::mbar_init(&pub_ready, 4);
        tc::mbar_init(&pub_free, 1);
        tc::mbar_init(&drain, 1);
        abort_flag = 0;
        tc::fence_barrier_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(&tmem_slot, kPtCols);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = tmem_slot;
    volatile int *abort_v = &abort_flag;
    // a programmatic dependent of the segment-table kernel: nothing that kernel writes is
    // touched before this
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const bool table_ok = t.seg_off[t.nseq + 1] == 1;
    const int64_t total_units = table_ok ? t.seg_off[t.nseq] * H : 0;
    GateRec *recA = reinterpret_cast<GateRec *>(sm + kPGate);
    GateRec *recC = recA + kPRecA;

    if (warp == 0) {
        // =============================== producer ===============================
        const uint64_t keep = tc::policy_evict_last(), drop = tc::policy_evict_first();
        if (lane == 0) {
            tc::tma_prefetch_desc(&maps.q);
            tc::tma_prefetch_desc(&maps.k);
            tc::tma_prefetch_desc(&maps.v);
            tc::tma_prefetch_desc(&maps.o);
        }
        uint32_t us = 0, jobA = 0, oc = 0;
        auto W = [&](uint64_t *bar, uint32_t par) {
            return __all_sync(0xffffffffu, wait_or_abort(bar, par & 1, abort_v, status));
        };
        for (;;) {
            const uint32_t slot = us & 1;
            if (us >= 2 && !W(&unit_empty[slot], (us >> 1) - 1)) break;
            // the next ticket is taken only once the previous unit has released the region, so
            // that units start in ticket order (a unit's predecessor started before it)
            if (us >= 1 && !W(&unit_free, us - 1)) break;
            uint32_t u = 0;
            if (lane == 0) u = atomicAdd(f.ticket, 1u);
            u = __shfl_sync(0xffffffffu, u, 0);
            UnitInfo info{};
            info.valid = 0;
            if (static_cast<int64_t>(u) < total_units) {
                info.sigma = u / H;
                info.h = static_cast<int>(u % H);
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
            const int h = info.h, nch = info.nch;
            bool ok = true;
            // state pass: K and V of chunks last to first, through three slots
            for (int r = 0; r < nch && ok; ++r) {
                const int c = nch - 1 - r;
                const int64_t c0 = info.t0 + int64_t(c) * kChunk;
                const int nv = static_cast<int>(min(int64_t(kChunk), info.t1 - c0));
                const uint32_t s = jobA % kPSlots;
                if (jobA >= kPSlots && !W(&slot_free[s], (jobA / kPSlots) - 1)) { ok = false; break; }
                if (2 * lane < nv) tc::prefetch_l2_keep(a.g + (c0 + 2 * lane) * H + h);
                if (2 * lane + 1 < nv) tc::prefetch_l2_keep(a.g + (c0 + 2 * lane + 1) * H + h);
                if (lane == 0) {
                    uint8_t *base = sm + s * kPSlot;
                    const int32_t x0 = static_cast<int32_t>(c0);
                    tc::mbar_arrive_expect_tx(&ka_full[s], 2 * kTile);
                    tc::tma_load_3d_hint(base, &maps.k, 0, h, x0, &ka_full[s], keep);
                    tc::tma_load_3d_hint(base + kRegion, &maps.k, 64, h, x0, &ka_full[s], keep);
                    tc::tma_load_3d_hint(base + kTile, &maps.v, 0, h, x0, &ka_full[s], keep);
                    tc::tma_load_3d_hint(base + kTile + kRegion, &maps.v, 64, h, x0, &ka_full[s], keep);
                }
                __syncwarp();
                ++jobA;
            }
            if (!ok) break;
            // output pass, once the state pass has released the slots: Q and V of chunks first
            // to last, each double-buffered
            if (!W(&ds_full, us)) break;
            for (int c = 0; c < nch && ok; ++c) {
                const int64_t c0 = info.t0 + int64_t(c) * kChunk;
                const int nv = static_cast<int>(min(int64_t(kChunk), info.t1 - c0));
                const uint32_t b = oc & 1;
                if (oc >= 2 && !(W(&q_free[b], (oc >> 1) - 1) && W(&v_free[b], (oc >> 1) - 1))) { ok = false; break; }
                if (2 * lane < nv) tc::prefetch_l2_keep(a.g + (c0 + 2 * lane) * H + h);
                if (2 * lane + 1 < nv) tc::prefetch_l2_keep(a.g + (c0 + 2 * lane + 1) * H + h);
                if (lane == 0) {
                    const int32_t x0 = static_cast<int32_t>(c0);
                    uint8_t *qd = sm + kPQ + b * kTile, *vd = sm + kPV + b * kTile;
                    tc::mbar_arrive_expect_tx(&q_full[b], kTile);
                    tc::tma_load_3d_hint(qd, &maps.q, 0, h, x0, &q_full[b], drop);
                    tc::tma_load_3d_hint(qd + kRegion, &maps.q, 64, h, x0, &q_full[b], drop);
                    tc::mbar_arrive_expect_tx(&v_full[b], kTile);
                    tc::tma_load_3d_hint(vd, &maps.v, 0, h, x0, &v_full[b], drop);
                    tc::tma_load_3d_hint(vd + kRegion, &maps.v, 64, h, x0, &v_full[b], drop);
                    // the workers read this chunk's K rows with ordinary loads a little later
                    tc::tma_prefetch_l2_3d(&maps.k, 0, h, x0, drop);
                    tc::tma_prefetch_l2_3d(&maps.k, 64, h, x0, drop);
                }
                __syncwarp();
                ++oc;
            }
            if (!ok) break;
            ++us;
        }
        // drain: the last copies must land before the CTA may exit
        if (lane == 0) {
            for (uint32_t j = jobA > kPSlots ? jobA - kPSlots : 0; j < jobA; ++j)
                tc::mbar_wait(&ka_full[j % kPSlots], (j / kPSlots) & 1, kWaitNs);
            for (uint32_t j = oc > 2 ? oc - 2 : 0; j < oc; ++j) {
                tc::mbar_wait(&q_full[j & 1], (j >> 1) & 1, kWaitNs);
                tc::mbar_wait(&v_full[j & 1], (j >> 1) & 1, kWaitNs);
            }
        }
    } else if (warp == 1) {
        // =============================== MMA issuer ===============================
        // The whole warp follows the schedule (warp-uniform waits and descriptors); one elected
        // lane issues the products and their commits.
        const uint32_t sb = tc::smem_u32(sm);
        uint32_t us = 0, jobA = 0, oc = 0, zbc = 0;
        auto W = [&](uint64_t *bar, uint32_t par) {
            return __all_sync(0xffffffffu, wait_or_abort(bar, par & 1, abort_v, status));
        };
        bool ok = true;
        for (;;) {
            const uint32_t slot = us & 1;
            if (!W(&unit_full[slot], us >> 1)) break;
            const UnitInfo info = units[slot];
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&unit_empty[slot]);
            if (!info.valid) break;
            const int nch = info.nch;
            // ---- state pass: dS^T = sum over chunks of V^T K', in the Z columns
            for (int r = 0; r < nch && ok; ++r) {
                const uint32_t s = jobA % kPSlots;
                if (!(ok = W(&ka_ready[s], jobA / kPSlots))) break;
                if (lane == 0) PTRACE(1, 4, r);
                tc::tc_fence_after();
                const uint32_t k_s = sb + s * kPSlot, v_s = k_s + kTile;
                const uint64_t da = desc_mn8(v_s), db = desc_mn8(k_s);
                if (tc::elect_one()) {
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        tc::umma_bf16(tmem + kPtZ, da + ks * (2048 >> 4), db + ks * (2048 >> 4), kIdS,
                                      (r > 0 || ks > 0) ? 1u : 0u);
                    tc::umma_commit(&slot_free[s]);
                }
                __syncwarp();
                ++jobA;
            }
            if (!ok) break;
            if (tc::elect_one()) tc::umma_commit(&ds_full);
            __syncwarp();
            // ---- output pass
            for (int c = 0; c < nch && ok; ++c) {
                const uint32_t b = oc & 1;
                const uint32_t q_s = sb + kPQ + b * kTile, v_s = sb + kPV + b * kTile;
                const uint64_t dq = desc_k(q_s), dv = desc_mn8(v_s);
                // M1: P = Q K~^T (raw K on the exact route)
                if (!(ok = W(&kp_ready, oc) && W(&q_full[b], oc >> 1) && (oc == 0 || W(&po_free, oc - 1)))) break;
                if (lane == 0) PTRACE(1, 1, c);
                tc::tc_fence_after();
                const bool fast = kfast != 0;
                const uint64_t dk = desc_k(sb + kPK);
                if (tc::elect_one()) {
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const uint32_t o4 = ((ks >> 2) * kRegion + (ks & 3) * 32) >> 4;
                        tc::umma_bf16(tmem + kPtPO, dq + o4, dk + o4, kIdP, ks > 0);
                    }
                    tc::umma_commit(&p_full);
                }
                __syncwarp();
                const bool m4 = c + 1 < nch;
                const uint64_t dk4 = desc_mn8(sb + kPK);
                // the state has been copied (M4 may update it) and V has landed
                if (!(ok = W(&zb_ready, zbc) && W(&v_full[b], oc >> 1))) break;
                if (lane == 0) PTRACE(1, 2, c);
                ++zbc;
                tc::tc_fence_after();
                if (tc::elect_one()) {
                    if (m4 && fast) {
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks)
                            tc::umma_bf16(tmem + kPtZ, dv + ks * (2048 >> 4), dk4 + ks * (2048 >> 4), kIdS, 1u);
                        tc::umma_commit(&z_full);
                    }
                    if (fast || !m4) tc::umma_commit(&kp_free);   // M1 (and M4) have read K~
                }
                __syncwarp();
                // P' is made (the scores are read, so O^T may take their columns); on the exact
                // route Q is scaled and K~ holds the weighted keys
                if (!(ok = W(&pp_ready, oc))) break;
                if (lane == 0) PTRACE(1, 3, c);
                tc::tc_fence_after();
                const uint64_t dp = desc_k(sb + kPP);
                if (tc::elect_one()) {
                    if (m4 && !fast) {
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks)
                            tc::umma_bf16(tmem + kPtZ, dv + ks * (2048 >> 4), dk4 + ks * (2048 >> 4), kIdS, 1u);
                        tc::umma_commit(&z_full);
                        tc::umma_commit(&kp_free);
                    }
                    // M2: O^T = Z^T Q^T (A = the bf16 copy of Z^T), M3: O^T += V^T P'^T
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)
                        tc::umma_bf16_ta(tmem + kPtPO, tmem + kPtZb + 8 * ks,
                                         dq + (((ks >> 2) * kRegion + (ks & 3) * 32) >> 4), kIdO2, ks > 0);
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        tc::umma_bf16(tmem + kPtPO, dv + ks * (2048 >> 4), dp + ks * (32 >> 4), kIdO3, 1u);
                    tc::umma_commit(&o_full);
                    tc::umma_commit(&zb_free);
                    tc::umma_commit(&q_free[b]);
                    tc::umma_commit(&v_free[b]);
                    if (!m4) tc::umma_commit(&unit_free);   // every product of the unit is done
                }
                __syncwarp();
                ++oc;
            }
            if (!ok) break;
            ++us;
        }
        // no product may still run when the tensor memory is freed
        if (tc::elect_one()) {
            tc::umma_commit(&drain);
            tc::mbar_wait(&drain, 0, kWaitNs);
        }
        __syncwarp();
    } else if (warp == 2) {
        // =============================== gate warp ===============================
        // Loads g of every chunk (two jobs ahead), takes the in-warp prefix sums and publishes
        // one record per chunk: for the state pass (chunks last to first) with the total of the
        // later chunks, then for the output pass (chunks first to last) with the chunk's plan.
        uint32_t us = 0, ja = 0, jc = 0;
        for (;;) {
            const uint32_t slot = us & 1;
            const bool bad = !wait_or_abort(&unit_full[slot], (us >> 1) & 1, abort_v, status);
            if (__any_sync(0xffffffffu, bad)) break;
            const UnitInfo info = units[slot];
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&unit_empty[slot]);
            if (!info.valid) break;
            const int h = info.h, nch = info.nch;
            auto c0_of = [&](int c) { return info.t0 + int64_t(c) * kChunk; };
            auto nv_of = [&](int c) { return static_cast<int>(min(int64_t(kChunk), info.t1 - c0_of(c))); };
            auto claim = [&](uint64_t *empty_b, uint32_t n, int R) {
                const bool b = n >= static_cast<uint32_t>(R) &&
                               !wait_or_abort(&empty_b[n % R], ((n / R) - 1) & 1, abort_v, status);
                return !__any_sync(0xffffffffu, b);
            };
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
                const int R = state ? kPRecA : kPRecC;
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
    } else if (warp == 3) {
        // =============================== flag publisher ===============================
        // Releases a unit's hand-off flag once the workers have stored its S_out (their mbarrier
        // arrivals order the stores before this thread's device-scope fence).
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
    } else {
        // =============================== workers ===============================
        // Thread wtid: tensor-memory lane j = wtid of Z^T (value column j); row wtid & 63 and
        // half wtid >> 6 of the key tiles it scales; in the M=64 layouts rows t = 16 quarter +
        // (lane & 15). Waits inside a unit do not vote (a thread whose wait gives up has set the
        // abort flag and every later wait returns at once); one OR-vote per unit ends the loop.
        const int wtid = threadIdx.x - 128;
        const int quarter = warp & 3;
        const int j = wtid;
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        const int srow = wtid & 63, shalf = wtid >> 6;
        const int tr = quarter * 16 + (lane & 15), sh = lane >> 4;   // M=64 layout row, half
        const int krow = wtid >> 4, kc16 = wtid & 15;                // K~ rows krow + 8 i
        const uint64_t drop = tc::policy_evict_first();
        uint32_t us = 0, jobA = 0, oc = 0, ja = 0, jc = 0, zbc = 0, zfc = 0, npub = 0;
        // o staging: the stmatrix addressing of the output tile (64-byte swizzle)
        uint8_t *stg = sm + kPO + quarter * kPOWarp;
        const int p8 = lane & 7;
        const int tl = 2 * (lane & 3);
        for (;;) {
            const uint32_t slot = us & 1;
            if (!wg_wait(&unit_full[slot], us >> 1, true, kBarW, abort_v, status)) break;
            const UnitInfo info = units[slot];
            named_sync(kBarW, 128);
            if (wtid == 0) tc::mbar_arrive(&unit_empty[slot]);
            if (!info.valid) break;
            const int h = info.h, nch = info.nch;
            auto c0_of = [&](int c) { return info.t0 + int64_t(c) * kChunk; };
            auto nv_of = [&](int c) { return static_cast<int>(min(int64_t(kChunk), info.t1 - c0_of(c))); };
            if (info.first && f.h0) {
                const char *hb = reinterpret_cast<const char *>(f.h0 + (info.n * H + h) * kD * kD);
                for (int i = wtid; i < kD * kD * 4 / 128; i += 128) tc::prefetch_l2_keep(hb + 128 * i);
            }

            // ---------------- state pass: K' = K exp(B_end - B_s) in place ----------------
            if (wtid == 0) PTRACE(3, 1, us);
            float D = 0.f;
#pragma unroll 1
            for (int r = 0; r < nch; ++r) {
                const int64_t c0 = c0_of(nch - 1 - r);
                const uint32_t s = (jobA + r) % kPSlots;
                wait_nv(&ga_full[ja % kPRecA], ja / kPRecA, true, abort_v, status);
                const GateRec *R = recA + ja % kPRecA;
                const float e = R->bC + R->D - R->b[srow];
                D += R->bC;
                warp_arrive(&ga_empty[ja % kPRecA]);
                ++ja;
                const float fac = c0 + srow < info.t1 ? tc::ex2(e * kLog2e) : 0.f;
                wait_nv(&ka_full[s], (jobA + r) / kPSlots, true, abort_v, status);
                uint8_t *base = sm + s * kPSlot + shalf * kRegion;
                uint4 x[8];
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8) x[c8] = *reinterpret_cast<const uint4 *>(base + sw(srow, c8));
#pragma unroll
                for (int c8 = 0; c8 < 8; ++c8) {
                    uint4 y;
                    y.x = mul_bf16x2(x[c8].x, fac);
                    y.y = mul_bf16x2(x[c8].y, fac);
                    y.z = mul_bf16x2(x[c8].z, fac);
                    y.w = mul_bf16x2(x[c8].w, fac);
                    *reinterpret_cast<uint4 *>(base + sw(srow, c8)) = y;
                }
                tc::fence_proxy_async_smem();
                warp_arrive(&ka_ready[s]);
            }
            jobA += nch;

            // ---------------- hand-off: S_in, Z = S_in and its bf16 copy, publish S_out ----------------
            {
                bool bad = !wait_or_abort(&ds_full, us & 1, abort_v, status);
                if (wtid == 0) PTRACE(3, 2, us);
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
                if (named_any(kBarW, 128, bad || *abort_v)) break;
                if (wtid == 0) PTRACE(3, 3, us);
                tc::tc_fence_after();
                // chunk 0 starts at the reference point; the exact route keeps the state scaled
                // to the chunk end
                wait_nv(&gc_full[jc % kPRecC], jc / kPRecC, true, abort_v, status);
                const float zfac = recC[jc % kPRecC].eC;
                const float eB = tc::ex2(D * kLog2e);
                float *dst = info.last ? (f.hT ? f.hT + (info.n * H + h) * kD * kD : nullptr)
                                       : f.incl + (static_cast<size_t>(info.sigma) * H + h) * kD * kD;
                const float *src = info.first
                    ? (f.h0 ? f.h0 + (info.n * H + h) * kD * kD : nullptr)
                    : f.incl + (static_cast<size_t>(info.sigma - 1) * H + h) * kD * kD;
                // (the bf16 copy of the previous unit's last chunk has been read: ds_full)
                if (zbc >= 1) wait_nv(&zb_free, zbc - 1, true, abort_v, status);
#pragma unroll 1
                for (int k4 = 0; k4 < 4; ++k4) {
                    float sv[32];
                    if (src) {
                        const float *p = src + (32 * k4) * kD + j;
#pragma unroll
                        for (int i = 0; i < 32; ++i) sv[i] = __ldcg(p + i * kD);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) sv[i] = 0.f;
                    }
                    uint32_t d[32];
                    tc::tmem_ld_32x32b_x32(tmem + lane_base + kPtZ + 32 * k4, d);
                    tc::tmem_ld_wait();
                    if (dst) {
                        float *p = dst + (32 * k4) * kD + j;
#pragma unroll
                        for (int i = 0; i < 32; ++i) p[i * kD] = fmaf(eB, sv[i], __uint_as_float(d[i]));
                    }
                    uint32_t w[16];
#pragma unroll
                    for (int m = 0; m < 16; ++m) w[m] = float2_to_bf16x2(sv[2 * m], sv[2 * m + 1]);
                    tc::tmem_st_32x32b_x16(tmem + lane_base + kPtZb + 16 * k4, w);
#pragma unroll
                    for (int i = 0; i < 32; ++i) d[i] = __float_as_uint(sv[i] * zfac);
                    tc::tmem_st_32x32b_x32(tmem + lane_base + kPtZ + 32 * k4, d);
                }
                tc::tmem_st_wait();
                tc::tc_fence_before();
                warp_arrive(&zb_ready);
                ++zbc;
                // the publisher releases the flag once all four warps have stored S_out
                if (npub >= 1) wait_nv(&pub_free, npub - 1, true, abort_v, status);
                if (wtid == 0) {
                    pub_cmd = info.last ? 0 : 1;
                    pub_flag = f.flags + info.sigma * H + h;
                }
                warp_arrive(&pub_ready);
                ++npub;
                if (wtid == 0) PTRACE(3, 4, us);
            }

            // ---------------- output pass ----------------
            // Per chunk c: P' of c, K~ of c + 1 (its rows loaded while M2 and M3 of c run), the
            // bf16 copy of the state entering c + 1, then the epilogue of c. K~ of chunk 0 goes
            // first.
            uint4 kx[8];
            const uint8_t *kbase = reinterpret_cast<const uint8_t *>(a.k + (krow * H + h) * kD) + 16 * kc16;
            const size_t kstep = static_cast<size_t>(8) * H * kD * sizeof(uint16_t);   // 8 rows
            auto load_rows = [&](int c) {
                const int64_t c0 = c0_of(c);
                const int nv = nv_of(c);
                const uint8_t *src = kbase + static_cast<size_t>(c0) * H * kD * sizeof(uint16_t);
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    kx[i] = krow + 8 * i < nv ? tc::ldg_nc_hint(src + i * kstep, drop) : make_uint4(0u, 0u, 0u, 0u);
            };
            // K~ of chunk c from the rows in kx: k exp(-(base + b_s)), or the raw keys (exact route)
            auto make_k = [&](int c, const GateRec *R) {
                const int nv = nv_of(c);
                const bool fast = R->fast != 0;
                if (oc + c >= 1) wait_nv(&kp_free, oc + c - 1, true, abort_v, status);
                const int lr = 2 * quarter + (lane & 1) + 8 * ((lane & 15) >> 1);
                const float myfac = lr < nv ? (fast ? tc::ex2((-R->base - R->b[lr]) * kLog2e) : 1.f) : 0.f;
                uint8_t *kd = sm + kPK + (kc16 >> 3) * kRegion;
                const int par = lane >> 4;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float fac = __shfl_sync(0xffffffffu, myfac, 2 * i + par);
                    const __nv_bfloat162 f2 = __float2bfloat162_rn(fac);
                    uint4 y;
                    y.x = mul_bf16x2(kx[i].x, f2);
                    y.y = mul_bf16x2(kx[i].y, f2);
                    y.z = mul_bf16x2(kx[i].z, f2);
                    y.w = mul_bf16x2(kx[i].w, f2);
                    *reinterpret_cast<uint4 *>(kd + sw(krow + 8 * i, kc16 & 7)) = y;
                }
                if (wtid == 0) kfast = fast;
                tc::fence_proxy_async_smem();
                warp_arrive(&kp_ready);
            };
            load_rows(0);
            make_k(0, recC + jc % kPRecC);
            // this lane's row addresses for the two halves of the epilogue's transposing stores:
            // value columns 0-15 (matrices 0, 1) and 16-31 (matrices 2, 3) of the warp's 32
            const int k2a = (lane >> 3) & 1;
            const uint32_t st_a = tc::smem_u32(stg) + p8 * 64 + 16 * (k2a ^ ((p8 >> 1) & 3));
            const uint32_t st_b = tc::smem_u32(stg) + p8 * 64 + 16 * ((k2a + 2) ^ ((p8 >> 1) & 3));
            for (int c = 0; c < nch; ++c) {
                const int64_t c0 = c0_of(c);
                const int nv = nv_of(c);
                const uint32_t b = (oc + c) & 1;
                const GateRec *R = recC + (jc + c) % kPRecC;   // (waited for already)
                const bool fast = R->fast != 0;
                // P': the scores, masked (s <= t < nv) and rounded to bf16 (K-major rows t)
                wait_nv(&p_full, oc + c, true, abort_v, status);
                if (wtid == 0) PTRACE(2, 1, c);
                tc::tc_fence_after();
                {
                    uint8_t *pp = sm + kPP;
                    const bool live = tr < nv;
#pragma unroll 1
                    for (int hp = 0; hp < 2; ++hp) {
                        uint32_t p[16];
                        tc::tmem_ld_16x32bx2_x16(tmem + lane_base + kPtPO + 16 * hp, p);
                        tc::tmem_ld_wait();
#pragma unroll
                        for (int c4 = 0; c4 < 2; ++c4) {
                            uint32_t w[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int si = 8 * c4 + 2 * e, s = 32 * sh + 16 * hp + si;
                                const float f0 = (live && s <= tr) ? __uint_as_float(p[si]) : 0.f;
                                const float f1 = (live && s + 1 <= tr) ? __uint_as_float(p[si + 1]) : 0.f;
                                w[e] = float2_to_bf16x2(f0, f1);
                            }
                            *reinterpret_cast<uint4 *>(pp + sw(tr, 4 * sh + 2 * hp + c4)) = make_uint4(w[0], w[1], w[2], w[3]);
                        }
                    }
                    tc::tc_fence_before();
                    if (!fast) {
                        // exact route: P'[t, s] *= exp(b_t - b_s); q_t <- exp(b_t) q_t (M1 has
                        // read Q); the weighted keys k_s exp(b_C - b_s) for M4 (M1 has read the raw)
                        if (tr < nv) exact_pp_weights(pp, R->b, tr, sh);
                        pexact_rows(sm + kPQ + b * kTile, reinterpret_cast<const uint16_t *>(a.q), c0, srow,
                                    shalf, nv, H, h, R->b[srow]);
                        if (c + 1 < nch)
                            pexact_rows(sm + kPK, reinterpret_cast<const uint16_t *>(a.k), c0, srow, shalf, nv,
                                        H, h, R->bC - R->b[srow]);
                    }
                    tc::fence_proxy_async_smem();
                    warp_arrive(&pp_ready);
                    if (wtid == 0) PTRACE(2, 2, c);
                }
                if (c + 1 < nch) {
                    // K~ of the next chunk (once M1 and M4 of this one have read this chunk's)
                    wait_nv(&gc_full[(jc + c + 1) % kPRecC], (jc + c + 1) / kPRecC, true, abort_v, status);
                    const GateRec *Rn = recC + (jc + c + 1) % kPRecC;
                    load_rows(c + 1);
                    if (wtid == 0) PTRACE(2, 3, c);
                    make_k(c + 1, Rn);
                    if (wtid == 0) PTRACE(2, 4, c);
                    // the bf16 copy of the state entering the next chunk (true state at its start:
                    // times e1; if the reference moves, the stored state too, times eC on the
                    // exact route), once M4 of this chunk has updated Z and M2 has read the old copy
                    const float e1 = Rn->e1, eC = Rn->eC;
                    const bool moved = Rn->moved != 0;
                    wait_nv(&z_full, zfc, true, abort_v, status);
                    ++zfc;
                    if (wtid == 0) PTRACE(2, 5, c);
                    wait_nv(&zb_free, zbc - 1, true, abort_v, status);
                    if (wtid == 0) PTRACE(2, 6, c);
                    tc::tc_fence_after();
                    const uint32_t zb_base = tmem + lane_base + kPtZb;
#pragma unroll 1
                    for (int k2 = 0; k2 < 2; ++k2) {
                        uint32_t d0[32], d1[32];
                        tc::tmem_ld_32x32b_x32(tmem + lane_base + kPtZ + 64 * k2, d0);
                        tc::tmem_ld_32x32b_x32(tmem + lane_base + kPtZ + 64 * k2 + 32, d1);
                        tc::tmem_ld_wait();
                        const float m = moved ? e1 : 1.f;
                        uint32_t w[16];
#pragma unroll
                        for (int q = 0; q < 16; ++q)
                            w[q] = float2_to_bf16x2(__uint_as_float(d0[2 * q]) * m, __uint_as_float(d0[2 * q + 1]) * m);
                        tc::tmem_st_32x32b_x16(zb_base + 32 * k2, w);
#pragma unroll
                        for (int q = 0; q < 16; ++q)
                            w[q] = float2_to_bf16x2(__uint_as_float(d1[2 * q]) * m, __uint_as_float(d1[2 * q + 1]) * m);
                        tc::tmem_st_32x32b_x16(zb_base + 32 * k2 + 16, w);
                        if (moved) {
                            const float e2 = e1 * eC;
#pragma unroll
                            for (int i = 0; i < 32; ++i) {
                                d0[i] = __float_as_uint(__uint_as_float(d0[i]) * e2);
                                d1[i] = __float_as_uint(__uint_as_float(d1[i]) * e2);
                            }
                            tc::tmem_st_32x32b_x32(tmem + lane_base + kPtZ + 64 * k2, d0);
                            tc::tmem_st_32x32b_x32(tmem + lane_base + kPtZ + 64 * k2 + 32, d1);
                        }
                    }
                    tc::tmem_st_wait();
                    tc::tc_fence_before();
                    warp_arrive(&zb_ready);
                    if (wtid == 0) PTRACE(2, 7, c);
                    ++zbc;
                }
                // epilogue: o_t = factor_t O^T[j][t] for the warp's 32 value columns, staged as a
                // [64 t x 32 j] tile (64-byte swizzle) in two halves of 16 columns and written by
                // one TMA store per warp (direct stores when the chunk is ragged)
                {
                    const float base = R->base;
                    wait_nv(&o_full, oc + c, true, abort_v, status);
                    if (wtid == 0) PTRACE(2, 8, c);
                    tc::tc_fence_after();
                    uint32_t o0[32], o1[32];
                    tc::tmem_ld_16x256b_x8(tmem + lane_base + kPtPO, o0);
                    tc::tmem_ld_16x256b_x8(tmem + lane_base + (16u << 16) + kPtPO, o1);
                    tc::tmem_ld_wait();
                    tc::tc_fence_before();
                    warp_arrive(&po_free);   // the columns may take the next scores
                    if (lane == 0) tc::tma_store_wait_read<0>();   // staging tile free again
                    __syncwarp();
#pragma unroll
                    for (int m = 0; m < 8; ++m) {
                        const float2 bb = *reinterpret_cast<const float2 *>(&R->b[8 * m + tl]);
                        const float fa = fast ? a.scale * tc::ex2((base + bb.x) * kLog2e) : a.scale;
                        const float fb = fast ? a.scale * tc::ex2((base + bb.y) * kLog2e) : a.scale;
                        pstmatrix_x2_trans(st_a + 512 * m,
                                           float2_to_bf16x2(__uint_as_float(o0[4 * m]) * fa, __uint_as_float(o0[4 * m + 1]) * fb),
                                           float2_to_bf16x2(__uint_as_float(o0[4 * m + 2]) * fa, __uint_as_float(o0[4 * m + 3]) * fb));
                        pstmatrix_x2_trans(st_b + 512 * m,
                                           float2_to_bf16x2(__uint_as_float(o1[4 * m]) * fa, __uint_as_float(o1[4 * m + 1]) * fb),
                                           float2_to_bf16x2(__uint_as_float(o1[4 * m + 2]) * fa, __uint_as_float(o1[4 * m + 3]) * fb));
                    }
                    warp_arrive(&gc_empty[(jc + c) % kPRecC]);   // done with this chunk's record
                    if (nv == kChunk) {
                        tc::fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            tc::tma_store_3d(&maps.o, 32 * quarter, h, static_cast<int32_t>(c0), stg);
                            tc::tma_store_commit();
                        }
                    } else if (dcheck(nv > 0 && c0 + nv <= info.t1, status)) {
                        __syncwarp();
                        uint16_t *orow = a.o + (c0 * H + h) * kD + 32 * quarter + lane;
#pragma unroll 1
                        for (int tt = 0; tt < nv; ++tt)
                            orow[static_cast<size_t>(tt) * H * kD] = *reinterpret_cast<const uint16_t *>(
                                stg + tt * 64 + 16 * ((lane >> 3) ^ ((tt >> 1) & 3)) + 2 * (lane & 7));
                    }
                }
                if (wtid == 0) PTRACE(2, 9, c);
            }
            oc += nch;
            jc += nch;
            // the region may take the next unit's tiles once this unit's stores have read it
            if (lane == 0) tc::tma_store_wait_read<0>();
            warp_arrive(&unit_free);
            if (named_any(kBarW, 128, *abort_v != 0)) break;
            ++us;
        }
        if (lane == 0) tc::tma_store_wait_all<0>();
        // stop the publisher (after an abort it stops by itself)
        if (!named_any(kBarW, 128, *abort_v != 0)) {
            if (npub >= 1) wait_nv(&pub_free, npub - 1, true, abort_v, status);
            if (wtid == 0) pub_cmd = 2;
            warp_arrive(&pub_ready);
        }
    }

    tc::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, kPtCols);
    }
}

cudaError_t setup_pair_kernel() {
    return cudaFuncSetAttribute(prefill_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(kPSmemAlloc));
}

cudaError_t launch_prefill_pair(const ChunkArgs &a, const SegTable &t, int64_t T_total,
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
        LaunchTimer timer(kKPrefillPair, st);
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(grid));
        cfg.blockDim = dim3(kPThreads);
        cfg.dynamicSmemBytes = kPSmemAlloc;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, prefill_pair_kernel, maps, f, t, status);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace sala

#ifdef SALA_TRACE
extern "C" int sala_gla_debug_pair_trace(unsigned long long *out, int max) {
    unsigned int n[4];
    if (cudaMemcpyFromSymbol(n, sala::g_ptrace_n, sizeof(n)) != cudaSuccess) return -1;
    static unsigned long long buf[4][sala::kPTraceN];
    if (cudaMemcpyFromSymbol(buf, sala::g_ptrace, sizeof(buf)) != cudaSuccess) return -1;
    int k = 0;
    for (int r = 0; r < 4; ++r)
        for (unsigned i = 0; i < n[r] && i < static_cast<unsigned>(sala::kPTraceN) && k < max; ++i)
            out[k++] = buf[r][i];
    return k;
}
#endif
