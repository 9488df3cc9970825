// Definitions shared by the two chunked-prefill kernels (prefill_fused.cu: one unit per SM;
// prefill_pair.cu: two CTAs per SM, one unit each): their arguments and unit descriptor, the
// shared-memory matrix descriptors of their tiles, the per-chunk gate records with the plan
// that weights each chunk (reference point, rescaling, factored or exact route), and the
// exact route's per-entry score weights.
#pragma once

#include "chunk_tc.cuh"

namespace sala {
namespace {

using namespace tck;

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kFastRange = 60.f;   // max |log-factor| (natural log) of the factored route

struct PrefillArgs {
    ChunkArgs c;            // q, k, v, g, scale, o, H
    const float *h0;        // [nseq, H, 128, 128] or null
    float *hT;              // [nseq, H, 128, 128] or null
    float *incl;            // [units, 128, 128]: S_out of each (segment, head), row-major like hT
    uint32_t *flags;        // [units]: == epoch once incl of that unit is published
    uint32_t *ticket;       // work counter, zeroed by the table kernel
    uint32_t epoch;
    uint64_t flag_wait_ns;  // limit of the wait for the predecessor's published state
    const uint32_t *withheld;   // failure-path test: this unit's flag is never released (or null)
};

struct UnitInfo {
    int valid, h, nch, first, last;
    int64_t sigma, n, t0, t1;
};

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
    float mx;       // max |b| over the chunk
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
    G.mx = mx;
    return G;
}

// How one chunk of the output pass is weighted, from its gate and `run`, the log-decay from
// the reference point to the chunk start (updated to the next chunk's).
struct Plan {
    float base;   // factored route: log-decay from the reference point to the chunk start
    float pre;    // log-factor the stored state takes before this chunk (0 if it keeps its scale)
    bool fast;    // factored route (else the exact route)
    bool moved;   // the reference moves before this chunk (the stored state is rescaled)
};

__device__ __forceinline__ Plan plan_chunk(const Gate &G, float &run) {
    Plan p;
    if (fabsf(run) + G.mx <= kFastRange) {          // factors stay in range: keep the reference
        p.fast = true;
        p.moved = false;
        p.pre = 0.f;
        p.base = run;
        run = run + G.bC;
    } else if (G.mx <= kFastRange) {                // move the reference to the chunk start
        p.fast = true;
        p.moved = true;
        p.pre = run;
        p.base = 0.f;
        run = G.bC;
    } else {                                        // exact route, reference to the chunk end
        p.fast = false;
        p.moved = true;
        p.pre = run;
        p.base = 0.f;
        run = 0.f;
    }
    return p;
}

// What the gate warp publishes for one chunk: the inclusive prefix sums b of its log-decays
// and, for the state pass, the chunk's total bC and the total D of the later chunks of the
// segment; for the output pass, the plan (reference offset, rescaling factors, route).
struct alignas(16) GateRec {
    float b[64];
    float bC;
    float D;        // state pass: log-decay of the later chunks of the segment
    float base;     // output pass, factored route: log-decay from the reference point
    float e1;       // output pass: exp(pre) if the reference moves before the chunk, else 1
    float eC;       // output pass, exact route: exp(bC), else 1
    uint32_t fast, moved, pad;
};
static_assert(sizeof(GateRec) == 288, "gate record size");

// Exact route, scores: columns 32 half .. + 31 of row t of P' (already masked and rounded to
// bf16 in the SW128 tile at pp) times exp(b_t - b_s) for every causal column s <= t (rare; kept
// out of line so that the hot loops stay short).
__device__ __noinline__ void exact_pp_weights(uint8_t *pp, const float *b, int t, int half) {
    const float bt = b[t] * kLog2e;
#pragma unroll 1
    for (int c8 = 4 * half; c8 < 4 * half + 4; ++c8) {
        uint4 x = *reinterpret_cast<const uint4 *>(pp + sw(t, c8));
        uint32_t *w = reinterpret_cast<uint32_t *>(&x);
        for (int e = 0; e < 4; ++e) {
            // only the causal entries s <= t carry a weight (past t the factor may overflow)
            const int s = 8 * c8 + 2 * e;
            const float2 f = bf16x2_to_float2(w[e]);
            w[e] = float2_to_bf16x2(s <= t ? f.x * tc::ex2(bt - b[s] * kLog2e) : 0.f,
                                    s + 1 <= t ? f.y * tc::ex2(bt - b[s + 1] * kLog2e) : 0.f);
        }
        *reinterpret_cast<uint4 *>(pp + sw(t, c8)) = x;
    }
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

// Per-warp arrival: the warp's lanes have finished their part; lane 0 arrives for the warp.
__device__ __forceinline__ void warp_arrive(uint64_t *bar) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) tc::mbar_arrive(bar);
}

}  // namespace
}  // namespace sala
