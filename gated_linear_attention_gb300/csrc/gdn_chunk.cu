// The gated delta rule (GDN) in its chunked form: the state-dependent value of every token.
//
// "Formulas and Code for Adapting Inference to GDN/KDA Linear Modules", section 1.2 (formulas
// 11-17): per sequence and head, per 64-token chunk with in-chunk log-decay prefix sums b,
// decay matrix Gamma[i][j] = exp(b_i - b_j), keys and values scaled by the write strengths
// (K_beta = diag(beta) K, V_beta = diag(beta) V) and S the state entering the chunk:
//   T     = (I + tril(K_beta K^T * Gamma, -1))^-1          (the UT transform, formula 11)
//   W     = T (K_beta * exp(b)),  U = T V_beta              (formulas 12, 13)
//   new_v = U - W S                                         (formula 15)
//   S    <- exp(b_C) S + (K * exp(b_C - b))^T new_v         (formula 16)
// The output (formula 17) and the state refresh are the Simple GLA chunk products with new_v
// in place of v, so sala_gla_gdn_chunk_fwd runs this kernel for new_v and then the chunked
// Simple GLA prefill on (q, k, new_v, g), which returns o and the final states.
//
// One CTA of 256 threads per (sequence, head) walks the chunks in order, the state in tensor
// memory in fp32 (lane = key row, column = value index); two CTAs share an SM (108 KB of
// shared memory and 256 tensor-memory columns each), so one's serial phases overlap the
// other's. Contractions (tcgen05.mma kind::f16, bf16 operands, fp32 accumulators in tensor
// memory, all but the state in one 128-column region used in turn):
//   X     = K K^T            M=64  N=64  K=128  (scores of the UT transform)
//   W     = T (K_beta e^b)   M=64  N=128 K=64
//   U     = T V_beta         M=64  N=128 K=64   (after W has been read out as -W in bf16)
//   U    += (-W) S           M=64  N=128 K=128  (U becomes new_v)
//   S    += K^T (e^(b_C - b) new_v)   M=128 N=128 K=64   (after S *= exp(b_C) in tensor memory;
//                                     the decay sits on new_v's rows, so K's tile serves as is)
// T itself is inverted on the CUDA cores in fp32 (four diagonal 16 x 16 blocks by forward
// substitution, then the blocks below the diagonal by distance, T_ij = -T_ii sum_k A_ik T_kj). Every factor is at most 1
// (b is non-increasing), so no range handling is needed. K tiles arrive by TMA, double
// buffered (the next chunk's tile loads while this one is processed); the V tile loads once
// the previous chunk's U has read it. Every wait is bounded (2 s); a timeout records
// SALA_ERR_TIMEOUT and the CTA stops after draining its MMAs and copies.
#include "chunk_tc.cuh"

namespace sala {
namespace {

using namespace tck;

constexpr int kGThreads = 256;
constexpr float kLog2eG = 1.4426950408889634f;
constexpr int kAS = 68;   // row stride (floats) of the fp32 A and T matrices in shared memory

// dynamic shared memory (offsets from a 1024-aligned base); two CTAs share an SM, so regions
// are reused across the phases of a chunk:
//   K [2]  TMA tiles, double buffered; a tile is read by X = K K^T, made into K beta e^b, and
//          is the A operand of the state update at the end of its chunk
//   V      TMA tile, scaled in place to V beta (the next chunk's tile loads once U has read it)
//   R      K beta e^b (B of W), then -W bf16 (A of W S), then new_v scaled per row (B of the
//          state update)
//   S      the state entering the chunk in bf16 [k][v] (B of W S), 2 x 16 KB
//   T      T bf16 [t][s] (A of W and U), one 64-column region
// During the inverse the fp32 A, T and the block sums P live in the S and T regions (free
// then; T bf16 is written from the fp32 T, which sits in the S region, after A and P are dead).
constexpr uint32_t kGK = 0;
constexpr uint32_t kGV = kGK + 2 * kTile;
constexpr uint32_t kGR = kGV + kTile;
constexpr uint32_t kGS = kGR + kTile;
constexpr uint32_t kGT = kGS + 2 * kSRegion;
constexpr uint32_t kGTf = kGS;                     // T fp32 [64][kAS]
constexpr uint32_t kGAf = kGTf + 64 * kAS * 4;     // A fp32 [64][kAS]
constexpr uint32_t kGY = kGAf + 64 * kAS * 4;      // P fp32 [32][20], then X fp32 [32][36] (inverse)
constexpr uint32_t kGB = kGT + kRegion;            // b [64], beta [64]
constexpr uint32_t kGBytes = kGB + 2 * 64 * 4;
constexpr uint32_t kGSmem = kGBytes + 1024;
static_assert(kGY + 32 * 36 * 4 <= kGB, "inverse scratch fits the S and T regions");
static_assert(kGTf + 64 * kAS * 4 <= kGT, "fp32 T does not overlap the bf16 T it is copied to");
static_assert(2 * (kGSmem + 1024) <= 228 * 1024, "two CTAs per SM");

// TMEM columns: the fp32 state, and one accumulator region used in turn by X (64 columns), W,
// and U / new_v (128 columns each)
constexpr uint32_t kGtS = 0, kGtAcc = 128, kGtCols = 256;
constexpr uint32_t kIdX = tc::idesc_bf16_f32(64, 64, 0, 0);
constexpr uint32_t kIdWU = tc::idesc_bf16_f32(64, 128, 0, 1);
constexpr uint32_t kIdS = tc::idesc_bf16_f32(128, 128, 1, 1);

__device__ __forceinline__ uint64_t gdesc_k(uint32_t addr) {          // K-major, SW128
    return tc::smem_desc_sw128(0, 16, 1024) | ((addr >> 4) & 0x3FFFu);
}
__device__ __forceinline__ uint64_t gdesc_mn64(uint32_t addr) {       // MN-major, 64-row tiles
    return tc::smem_desc_sw128(0, kRegion, 1024) | ((addr >> 4) & 0x3FFFu);
}
__device__ __forceinline__ uint64_t gdesc_mn128(uint32_t addr) {      // MN-major, 128-row tiles
    return tc::smem_desc_sw128(0, kSRegion, 1024) | ((addr >> 4) & 0x3FFFu);
}

struct GdnChunkArgs {
    const float *g, *beta;    // [T_total, H]
    const float *h0;          // [nseq, H, 128, 128] or null
    uint16_t *nv;             // bf16 [T_total, H, 128], written
    const int64_t *cu;        // [nseq + 1] or null (rows of T_row tokens)
    int64_t T_row, nseq, T_total;
    int H;
};

// bounded wait of every thread of the CTA on phase `par` of `bar`; false on timeout
__device__ __forceinline__ bool gwait(uint64_t *bar, uint32_t par, int *status, volatile int *bad) {
    if (*bad) return false;
    if (tc::mbar_try_wait(bar, par & 1)) return true;
    const uint64_t t0 = tc::global_timer_ns();
    while (!tc::mbar_try_wait(bar, par & 1)) {
        if (*bad) return false;
        if (tc::global_timer_ns() - t0 > kWaitNs) {
            *bad = 1;
            record_status(status, SALA_ERR_TIMEOUT);
            return false;
        }
    }
    return true;
}

}  // namespace

__global__ void __launch_bounds__(kGThreads, 2)
gdn_newv_kernel(const __grid_constant__ TcMaps maps, GdnChunkArgs p, int *status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
    __shared__ uint64_t full_k[2], full_v, bar_x, bar_w, bar_nv, bar_s, drain;
    __shared__ uint32_t tmem_slot;
    __shared__ int bad_flag;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // warps w and w + 4 reach the same quarter of the tensor-memory lanes; they split columns
    const int quarter = warp & 3, wg = warp >> 2;
    const int H = p.H;
    const int unit = blockIdx.x;
    const int64_t n = unit / H;
    const int h = unit % H;
    // sequence bounds, kept inside the tensors whatever cu holds
    int64_t t0 = p.cu ? p.cu[n] : n * p.T_row;
    int64_t t1 = p.cu ? p.cu[n + 1] : (n + 1) * p.T_row;
    t0 = max(int64_t(0), min(t0, p.T_total));
    t1 = max(t0, min(t1, p.T_total));
    const int nch = static_cast<int>((t1 - t0 + kChunk - 1) / kChunk);

    if (tid == 0) {
        tc::mbar_init(&full_k[0], 1);
        tc::mbar_init(&full_k[1], 1);
        tc::mbar_init(&full_v, 1);
        tc::mbar_init(&bar_x, 1);
        tc::mbar_init(&bar_w, 1);
        tc::mbar_init(&bar_nv, 1);
        tc::mbar_init(&bar_s, 1);
        tc::mbar_init(&drain, 1);
        bad_flag = 0;
        tc::fence_barrier_init();
    }
    if (warp == 0) {
        tc::tmem_alloc(&tmem_slot, kGtCols);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = tmem_slot;
    volatile int *bad = &bad_flag;
    const uint32_t sb = tc::smem_u32(sm);
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    float *bsm = reinterpret_cast<float *>(sm + kGB);
    float *betasm = bsm + 64;
    float *Af = reinterpret_cast<float *>(sm + kGAf);
    float *Tf = reinterpret_cast<float *>(sm + kGTf);
    float *Pf = reinterpret_cast<float *>(sm + kGY);   // block products of the inverse
    float *Xf = Pf;                                    // [32][36] (after P is dead)

    auto load_k = [&](int c) {   // thread 0: TMA of chunk c's K tile into buffer c & 1
        const int32_t x0 = static_cast<int32_t>(t0 + int64_t(c) * kChunk);
        uint64_t *bar = &full_k[c & 1];
        tc::mbar_arrive_expect_tx(bar, kTile);
        uint8_t *kd = sm + kGK + (c & 1) * kTile;
        tc::tma_load_3d(kd, &maps.k, 0, h, x0, bar);
        tc::tma_load_3d(kd + kRegion, &maps.k, 64, h, x0, bar);
    };
    auto load_v = [&](int c) {   // thread 0: TMA of chunk c's V tile
        const int32_t x0 = static_cast<int32_t>(t0 + int64_t(c) * kChunk);
        tc::mbar_arrive_expect_tx(&full_v, kTile);
        tc::tma_load_3d(sm + kGV, &maps.v, 0, h, x0, &full_v);
        tc::tma_load_3d(sm + kGV + kRegion, &maps.v, 64, h, x0, &full_v);
    };
    // the first chunk's tiles and gates are requested before the state is read in, so that
    // their latencies overlap
    if (tid == 0 && nch > 0) {
        tc::tma_prefetch_desc(&maps.k);
        tc::tma_prefetch_desc(&maps.v);
        load_k(0);
        load_v(0);
    }
    // g and beta of the next chunk, loaded a chunk ahead (threads 0-63: row tid)
    float g_nx = 0.f, be_nx = 0.f;
    if (tid < 64 && nch > 0 && tid < t1 - t0) {
        g_nx = p.g[(t0 + tid) * H + h];
        be_nx = p.beta[(t0 + tid) * H + h];
    }
    // the state entering the sequence: row k (= TMEM lane) of h0, or zeros; columns 64 wg ..
    {
        const int k = quarter * 32 + lane;
        const float *src = p.h0 ? p.h0 + (static_cast<size_t>(n) * H + h) * kD * kD + k * kD + 64 * wg : nullptr;
#pragma unroll 1
        for (int c4 = 0; c4 < 2; ++c4) {
            uint32_t r[32];
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
                const float4 x = src ? *reinterpret_cast<const float4 *>(src + 32 * c4 + i)
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
                r[i] = __float_as_uint(x.x);
                r[i + 1] = __float_as_uint(x.y);
                r[i + 2] = __float_as_uint(x.z);
                r[i + 3] = __float_as_uint(x.w);
            }
            tc::tmem_st_32x32b_x32(tmem + lane_base + kGtS + 64 * wg + 32 * c4, r);
        }
        tc::tmem_st_wait();
    }

    tc::tc_fence_before();
    __syncthreads();
    uint32_t kpar = 0;      // bit b: next phase of full_k[b]
    int vidx = 0;           // the chunk of the last V load issued
    uint32_t pending = 0;   // bits 0, 1: a K load into that buffer, bit 2: a V load, issued and
                            // not yet waited for
    if (nch > 0) pending = 1u | 4u;
#pragma unroll 1
    for (int c = 0; c < nch; ++c) {
        const int buf = c & 1;
        const int64_t c0 = t0 + int64_t(c) * kChunk;
        const int nv = static_cast<int>(min(int64_t(kChunk), t1 - c0));
        if (c + 1 < nch) {   // its buffer was last read by chunk c - 1's state update
            if (tid == 0) {
                tc::fence_proxy_async_smem();
                load_k(c + 1);
            }
            pending |= 1u << ((c + 1) & 1);
        }
        // log-decays and write strengths of the chunk (zero past nv), prefix sums b
        if (tid < 64) {
            const float gv = g_nx;
            betasm[tid] = be_nx;
            const int64_t cn = c0 + kChunk;
            g_nx = be_nx = 0.f;
            if (c + 1 < nch && cn + tid < t1) {
                g_nx = p.g[(cn + tid) * H + h];
                be_nx = p.beta[(cn + tid) * H + h];
            }
            float run = gv;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, run, off);
                if (lane >= off) run += y;
            }
            bsm[tid] = run;
        }
        __syncthreads();
        if (tid >= 32 && tid < 64) bsm[tid] += bsm[31];
        bool ok_full = gwait(&full_k[buf], (kpar >> buf) & 1, status, bad);
        if (ok_full) {
            kpar ^= 1u << buf;
            pending &= ~(1u << buf);
        }
        ok_full = ok_full && gwait(&full_v, c, status, bad);
        if (ok_full) pending &= ~4u;
        if (__syncthreads_or(!ok_full)) break;
        const float bC = bsm[nv - 1];
        const uint32_t kt = sb + kGK + buf * kTile;

        // X = K K^T (and the previous chunk's new_v stores have read the S region, which the
        // inverse below reuses)
        if (tid == 0) {
            tc::tma_store_wait_read<0>();
            tc::tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint32_t o4 = ((ks >> 2) * kRegion + (ks & 3) * 32) >> 4;
                tc::umma_bf16(tmem + kGtAcc, gdesc_k(kt) + o4, gdesc_k(kt) + o4, kIdX, ks > 0);
            }
            tc::umma_commit(&bar_x);
        }
        // meanwhile: K * beta e^b into R and V * beta in place, from the tiles (row r, 32
        // columns per thread; rows >= nv zero)
        {
            const int r = tid & 63, q4 = tid >> 6;   // row r, columns 32 q4 .. + 31
            const bool live = r < nv;
            const float br = bsm[r], be = betasm[r];
            const float fkb = live ? be * tc::ex2(br * kLog2eG) : 0.f;
            const float fv = live ? be : 0.f;
            const int half = q4 >> 1;
            const uint8_t *ksrc = sm + kGK + buf * kTile + half * kRegion;
            uint8_t *vb = sm + kGV + half * kRegion;
            uint8_t *dkb = sm + kGR + half * kRegion;
#pragma unroll
            for (int c8 = 4 * (q4 & 1); c8 < 4 * (q4 & 1) + 4; ++c8) {
                const uint32_t off = sw(r, c8);
                const uint4 kx = *reinterpret_cast<const uint4 *>(ksrc + off);
                const uint4 vx = *reinterpret_cast<const uint4 *>(vb + off);
                uint4 y;
                y.x = mul_bf16x2(kx.x, fkb); y.y = mul_bf16x2(kx.y, fkb);
                y.z = mul_bf16x2(kx.z, fkb); y.w = mul_bf16x2(kx.w, fkb);
                *reinterpret_cast<uint4 *>(dkb + off) = y;
                y.x = mul_bf16x2(vx.x, fv); y.y = mul_bf16x2(vx.y, fv);
                y.z = mul_bf16x2(vx.z, fv); y.w = mul_bf16x2(vx.w, fv);
                *reinterpret_cast<uint4 *>(vb + off) = y;
            }
        }
        tc::fence_proxy_async_smem();
        if (__syncthreads_or(!gwait(&bar_x, c, status, bad))) break;
        tc::tc_fence_after();
        // A[t][s] = beta_t exp(b_t - b_s) X[t][s] for s < t, else 0 (M=64 accumulator: rows
        // t = 16 warp + (lane & 15) in lanes 0-15 of the quarter; lanes 0-15 get columns 0-31
        // of those rows, lanes 16-31 columns 32-63)
        {
            // (the 16-column form: warps w and w + 4 take columns 16 wg .. + 15 of each half)
            uint32_t x[16];
            tc::tmem_ld_16x32bx2_x16(tmem + lane_base + kGtAcc + 16 * wg, x);
            tc::tmem_ld_wait();
            const int t = quarter * 16 + (lane & 15), s0 = 32 * (lane >> 4) + 16 * wg;
            const float bt = bsm[t] * kLog2eG, be = betasm[t];
            float *arow = Af + t * kAS + s0;
#pragma unroll
            for (int i = 0; i < 16; i += 4) {
                float4 w;
                w.x = (s0 + i < t) ? be * tc::ex2(bt - bsm[s0 + i] * kLog2eG) * __uint_as_float(x[i]) : 0.f;
                w.y = (s0 + i + 1 < t) ? be * tc::ex2(bt - bsm[s0 + i + 1] * kLog2eG) * __uint_as_float(x[i + 1]) : 0.f;
                w.z = (s0 + i + 2 < t) ? be * tc::ex2(bt - bsm[s0 + i + 2] * kLog2eG) * __uint_as_float(x[i + 2]) : 0.f;
                w.w = (s0 + i + 3 < t) ? be * tc::ex2(bt - bsm[s0 + i + 3] * kLog2eG) * __uint_as_float(x[i + 3]) : 0.f;
                *reinterpret_cast<float4 *>(arow + i) = w;
            }
        }
        tc::tc_fence_before();   // X is read: W may overwrite its columns
        __syncthreads();
        // T = (I + A)^-1 by 16 x 16 blocks. Diagonal blocks: thread (blk, j) of the first 64
        // solves column j of block blk by forward substitution, T[i][j] = -sum_{m < i} A[i][m]
        // T[m][j] with T[j][j] = 1 (the column is zero above j)
        if (tid < 64) {
            const int blk = tid >> 4, j = tid & 15, o = 16 * blk;
            float col[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) col[i] = (i == j) ? 1.f : 0.f;
#pragma unroll
            for (int i = 1; i < 16; ++i) {
                const float *ar = Af + (o + i) * kAS + o;
                float acc = 0.f;
#pragma unroll
                for (int m = 0; m < i; ++m) acc = fmaf(ar[m], col[m], acc);
                if (i > j) col[i] = -acc;
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) Tf[(o + i) * kAS + o + j] = col[i];
        }
        __syncthreads();
        // blocks below the diagonal, by the blocked inverse of a lower-triangular matrix
        // [[T_a, 0], [X, T_b]]^-1 = [[T_a^-1, 0], [-T_b^-1 X T_a^-1, T_b^-1]]: first the lower
        // 16 x 16 block of each diagonal 32 x 32 half (T_10 = -T_11 A_10 T_00 and T_32 =
        // -T_33 A_32 T_22), then the lower-left 32 x 32 block, -T_hi (A_[32:64][0:32] T_lo) with
        // T_lo, T_hi the inverses of the two halves. The upper triangles of the blocks on the
        // diagonal are zero (the solve above wrote them) and those above it are never read.
        {
            // Y = A_{i,i-1} T_{i-1,i-1} for i = 1, 3 (into P): thread: half hb, row r, columns
            // c0 .. c0 + 3
            const int hb = tid >> 6, r = (tid >> 2) & 15, c0 = 4 * (tid & 3);
            const int i = 2 * hb + 1, j = 2 * hb;
            if (hb < 2) {
                float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
                const float *ar = Af + (16 * i + r) * kAS + 16 * j;
#pragma unroll
                for (int m = 0; m < 16; ++m) {
                    const float u = ar[m];
                    const float4 tm = *reinterpret_cast<const float4 *>(Tf + (16 * j + m) * kAS + 16 * j + c0);
                    y.x = fmaf(u, tm.x, y.x); y.y = fmaf(u, tm.y, y.y);
                    y.z = fmaf(u, tm.z, y.z); y.w = fmaf(u, tm.w, y.w);
                }
                *reinterpret_cast<float4 *>(Pf + (16 * hb + r) * 20 + c0) = y;
            }
            __syncthreads();
            if (hb < 2) {   // T_{i,i-1} = -T_ii Y
                float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
                const float *tr = Tf + (16 * i + r) * kAS + 16 * i;
#pragma unroll
                for (int m = 0; m < 16; ++m) {
                    const float u = tr[m];
                    const float4 pm = *reinterpret_cast<const float4 *>(Pf + (16 * hb + m) * 20 + c0);
                    y.x = fmaf(u, pm.x, y.x); y.y = fmaf(u, pm.y, y.y);
                    y.z = fmaf(u, pm.z, y.z); y.w = fmaf(u, pm.w, y.w);
                }
                *reinterpret_cast<float4 *>(Tf + (16 * i + r) * kAS + 16 * j + c0) =
                    make_float4(-y.x, -y.y, -y.z, -y.w);
            }
            __syncthreads();
            // Z = A_[32:64][0:32] T_lo (into the scratch X): thread: row rr, columns cc .. cc + 3;
            // T_lo[m][n] = 0 for n > m, so the sum starts at m = cc
            const int rr = tid >> 3, cc = 4 * (tid & 7);
            {
                float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
                const float *ar = Af + (32 + rr) * kAS;
#pragma unroll 4
                for (int m = cc; m < 32; ++m) {
                    const float u = ar[m];
                    const float4 tm = *reinterpret_cast<const float4 *>(Tf + m * kAS + cc);
                    y.x = fmaf(u, tm.x, y.x); y.y = fmaf(u, tm.y, y.y);
                    y.z = fmaf(u, tm.z, y.z); y.w = fmaf(u, tm.w, y.w);
                }
                *reinterpret_cast<float4 *>(Xf + rr * 36 + cc) = y;
            }
            __syncthreads();
            {   // T_[32:64][0:32] = -T_hi Z; T_hi[rr][m] = 0 for m > rr
                float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
                const float *tr = Tf + (32 + rr) * kAS + 32;
#pragma unroll 4
                for (int m = 0; m <= rr; ++m) {
                    const float u = tr[m];
                    const float4 xm = *reinterpret_cast<const float4 *>(Xf + m * 36 + cc);
                    y.x = fmaf(u, xm.x, y.x); y.y = fmaf(u, xm.y, y.y);
                    y.z = fmaf(u, xm.z, y.z); y.w = fmaf(u, xm.w, y.w);
                }
                *reinterpret_cast<float4 *>(Tf + (32 + rr) * kAS + cc) = make_float4(-y.x, -y.y, -y.z, -y.w);
            }
            __syncthreads();
        }
        // T to bf16, K-major [t][s] (one 64-column region): thread: row t, columns 16 q4 .. + 15
        // (block q4; blocks above the diagonal are zero)
        {
            const int t = tid & 63, q4 = tid >> 6;
            const bool upper = q4 > (t >> 4);
            const float *tr = Tf + t * kAS + 16 * q4;
            uint8_t *dst = sm + kGT;
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2) {
                uint4 w = make_uint4(0u, 0u, 0u, 0u);
                if (!upper) {
                    w.x = float2_to_bf16x2(tr[8 * c2], tr[8 * c2 + 1]);
                    w.y = float2_to_bf16x2(tr[8 * c2 + 2], tr[8 * c2 + 3]);
                    w.z = float2_to_bf16x2(tr[8 * c2 + 4], tr[8 * c2 + 5]);
                    w.w = float2_to_bf16x2(tr[8 * c2 + 6], tr[8 * c2 + 7]);
                }
                *reinterpret_cast<uint4 *>(dst + sw(t, 2 * q4 + c2)) = w;
            }
        }
        tc::fence_proxy_async_smem();
        __syncthreads();
        // W = T (K beta e^b)
        if (tid == 0) {
            tc::tc_fence_after();
            const uint64_t dt = gdesc_k(sb + kGT);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                tc::umma_bf16(tmem + kGtAcc, dt + ((ks * 32) >> 4), gdesc_mn64(sb + kGR) + ks * (2048 >> 4), kIdWU, ks > 0);
            tc::umma_commit(&bar_w);
        }
        // meanwhile: the state entering the chunk to bf16 [k][v] (MN-major B of W S), and S
        // taken on by exp(bC) for the update at the end of the chunk (thread = key row k)
        {
            const float eC = tc::ex2(bC * kLog2eG);
            uint8_t *dst = sm + kGS;
            const int krow = quarter * 32 + lane;
#pragma unroll 1
            for (int c4 = 2 * wg; c4 < 2 * wg + 2; ++c4) {
                uint32_t r[32];
                tc::tmem_ld_32x32b_x32(tmem + lane_base + kGtS + 32 * c4, r);
                tc::tmem_ld_wait();
                // columns v = 32 c4 .. + 31: region v / 64, 16-byte chunks 4 (c4 & 1) .. + 3
                uint8_t *reg = dst + (c4 >> 1) * kSRegion;
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    uint4 w;
                    w.x = float2_to_bf16x2(__uint_as_float(r[8 * q4]), __uint_as_float(r[8 * q4 + 1]));
                    w.y = float2_to_bf16x2(__uint_as_float(r[8 * q4 + 2]), __uint_as_float(r[8 * q4 + 3]));
                    w.z = float2_to_bf16x2(__uint_as_float(r[8 * q4 + 4]), __uint_as_float(r[8 * q4 + 5]));
                    w.w = float2_to_bf16x2(__uint_as_float(r[8 * q4 + 6]), __uint_as_float(r[8 * q4 + 7]));
                    *reinterpret_cast<uint4 *>(reg + sw(krow, 4 * (c4 & 1) + q4)) = w;
                }
#pragma unroll
                for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * eC);
                tc::tmem_st_32x32b_x32(tmem + lane_base + kGtS + 32 * c4, r);
            }
            tc::tmem_st_wait();
        }
        tc::fence_proxy_async_smem();
        if (__syncthreads_or(!gwait(&bar_w, c, status, bad))) break;
        tc::tc_fence_after();
        // -W to bf16 [t][k] in R (K-major A of W S; W has read K beta e^b): thread: row t,
        // columns 32 (lane >> 4) .. of the 64-column half wg
        {
            const int t = quarter * 16 + (lane & 15), sh = lane >> 4;
            uint32_t x[32];
            tc::tmem_ld_16x32bx2_x32(tmem + lane_base + kGtAcc + 64 * wg, x);
            tc::tmem_ld_wait();
            uint8_t *dst = sm + kGR + wg * kRegion;
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
                uint4 w;
                w.x = float2_to_bf16x2(-__uint_as_float(x[8 * c4]), -__uint_as_float(x[8 * c4 + 1]));
                w.y = float2_to_bf16x2(-__uint_as_float(x[8 * c4 + 2]), -__uint_as_float(x[8 * c4 + 3]));
                w.z = float2_to_bf16x2(-__uint_as_float(x[8 * c4 + 4]), -__uint_as_float(x[8 * c4 + 5]));
                w.w = float2_to_bf16x2(-__uint_as_float(x[8 * c4 + 6]), -__uint_as_float(x[8 * c4 + 7]));
                *reinterpret_cast<uint4 *>(dst + sw(t, 4 * sh + c4)) = w;
            }
        }
        tc::fence_proxy_async_smem();
        tc::tc_fence_before();   // W is read: U may overwrite its columns
        __syncthreads();
        // U = T (V beta), then new_v = U + (-W) S
        if (tid == 0) {
            tc::tc_fence_after();
            const uint64_t dt = gdesc_k(sb + kGT);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                tc::umma_bf16(tmem + kGtAcc, dt + ((ks * 32) >> 4), gdesc_mn64(sb + kGV) + ks * (2048 >> 4), kIdWU, ks > 0);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint32_t oa = ((ks >> 2) * kRegion + (ks & 3) * 32) >> 4;
                tc::umma_bf16(tmem + kGtAcc, gdesc_k(sb + kGR) + oa, gdesc_mn128(sb + kGS) + ks * (2048 >> 4), kIdWU, 1u);
            }
            tc::umma_commit(&bar_nv);
        }
        if (__syncthreads_or(!gwait(&bar_nv, c, status, bad))) break;
        tc::tc_fence_after();
        if (c + 1 < nch && tid == 0) {   // the V tile is read: the next chunk's may load
            tc::fence_proxy_async_smem();
            load_v(c + 1);
            vidx = c + 1;
            pending |= 4u;
        }
        // new_v out to global memory, and into R scaled by exp(bC - b_t) per row t (zero past
        // nv): the MN-major B of the state update S += K^T (exp(bC - b) new_v)
        {
            const int t = quarter * 16 + (lane & 15), sh = lane >> 4;
            const bool live = t < nv && dcheck(c0 + t < t1 && t1 <= p.T_total, status);
            const float ft = live ? tc::ex2((bC - bsm[t]) * kLog2eG) : 0.f;
            uint16_t *grow = p.nv + ((c0 + t) * H + h) * kD;
            // a whole chunk leaves by TMA stores of four [64 t][32 v] boxes staged in the S region
            // (free until the next chunk's inverse); a ragged one row by row
            uint8_t *stg = sm + kGS + (2 * wg + sh) * 4096 + t * 64;
            uint32_t x[32];
            tc::tmem_ld_16x32bx2_x32(tmem + lane_base + kGtAcc + 64 * wg, x);
            tc::tmem_ld_wait();
            uint8_t *dst = sm + kGR + wg * kRegion;
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
                float f[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) f[i] = __uint_as_float(x[8 * c4 + i]);
                uint4 w;
                w.x = float2_to_bf16x2(f[0], f[1]);
                w.y = float2_to_bf16x2(f[2], f[3]);
                w.z = float2_to_bf16x2(f[4], f[5]);
                w.w = float2_to_bf16x2(f[6], f[7]);
                if (nv == kChunk) *reinterpret_cast<uint4 *>(stg + 16 * c4) = w;
                else if (live) *reinterpret_cast<uint4 *>(grow + 64 * wg + 32 * sh + 8 * c4) = w;
                w.x = float2_to_bf16x2(f[0] * ft, f[1] * ft);
                w.y = float2_to_bf16x2(f[2] * ft, f[3] * ft);
                w.z = float2_to_bf16x2(f[4] * ft, f[5] * ft);
                w.w = float2_to_bf16x2(f[6] * ft, f[7] * ft);
                *reinterpret_cast<uint4 *>(dst + sw(t, 4 * sh + c4)) = w;
            }
        }
        tc::fence_proxy_async_smem();
        tc::tc_fence_before();
        __syncthreads();
        // S += K^T (exp(bC - b) new_v); new_v of a whole chunk out
        if (tid == 0) {
            tc::tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                tc::umma_bf16(tmem + kGtS, gdesc_mn64(kt) + ks * (2048 >> 4),
                              gdesc_mn64(sb + kGR) + ks * (2048 >> 4), kIdS, 1u);
            tc::umma_commit(&bar_s);
            if (nv == kChunk) {
#pragma unroll
                for (int b = 0; b < 4; ++b)
                    tc::tma_store_3d(&maps.o, 32 * b, h, static_cast<int32_t>(c0), sm + kGS + b * 4096);
                tc::tma_store_commit();
            }
        }
        if (__syncthreads_or(!gwait(&bar_s, c, status, bad))) break;
        tc::tc_fence_after();
    }

    // no MMA or copy may be in flight when the CTA ends
    tc::tc_fence_before();
    __syncthreads();
    if (tid == 0) {
        tc::tma_store_wait_all<0>();
        tc::umma_commit(&drain);
        if (!tc::mbar_wait(&drain, 0, kWaitNs)) record_status(status, SALA_ERR_TIMEOUT);
        // tiles still landing if the loop stopped early: every load issued, but not waited for
        for (int b = 0; b < 2; ++b)
            if ((pending >> b) & 1) (void)tc::mbar_wait(&full_k[b], (kpar >> b) & 1, kWaitNs);
        if (pending & 4u) (void)tc::mbar_wait(&full_v, vidx & 1, kWaitNs);
    }
    __syncthreads();
    if (warp == 0) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, kGtCols);
    }
}

cudaError_t setup_gdn_chunk_kernel() {
    return cudaFuncSetAttribute(gdn_newv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(kGSmem));
}

cudaError_t launch_gdn_newv(const void *k, const void *v, const float *g, const float *beta,
                            const float *h0, const SegTable &t, int64_t T_total, void *nv, int H,
                            int *status, cudaStream_t st) {
    if (t.nseq == 0 || T_total == 0) return cudaSuccess;
    tck::TcMaps maps;
    // the q map is not used here (k stands in for it); the o map stores new_v
    cudaError_t e = tck::make_maps(&maps, k, k, v, nv, T_total, H);
    if (e != cudaSuccess) return e;
    GdnChunkArgs p;
    p.g = g;
    p.beta = beta;
    p.h0 = h0;
    p.nv = static_cast<uint16_t *>(nv);
    p.cu = t.cu;
    p.T_row = t.T_row;
    p.nseq = t.nseq;
    p.T_total = T_total;
    p.H = H;
    LaunchTimer timer(kKGdnNewv, st);
    gdn_newv_kernel<<<static_cast<unsigned>(t.nseq * H), kGThreads, kGSmem, st>>>(maps, p, status);
    return cudaGetLastError();
}

}  // namespace sala
