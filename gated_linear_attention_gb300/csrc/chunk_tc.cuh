// Device helpers shared by the tensor-core prefill kernels (internal).
#pragma once

#include <cudaTypedefs.h>

#include "launch.h"
#include "tc.cuh"

namespace sala {
namespace tck {

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

// How the bounded waits poll: SALA_WAIT_POLL_NS > 0 tests the phase without suspending and
// sleeps that long between tests; 0 uses try_wait, which may suspend the thread in hardware.
#ifndef SALA_WAIT_POLL_NS
#define SALA_WAIT_POLL_NS 0
#endif

// Bounded wait that also gives up as soon as another role has aborted. The fast path (phase
// already complete) is inline; the polling loop is a call, which keeps the many wait sites of
// the persistent kernels small (their code shares one instruction cache).
static __device__ __noinline__ bool wait_or_abort_slow(uint64_t *bar, uint32_t parity,
                                                volatile int *abort_flag, int *status) {
    const uint64_t t0 = tc::global_timer_ns();
    while (!(SALA_WAIT_POLL_NS ? tc::mbar_test_wait(bar, parity) : tc::mbar_try_wait(bar, parity))) {
        if (SALA_WAIT_POLL_NS) __nanosleep(SALA_WAIT_POLL_NS);
        if (*abort_flag) return false;
        if (tc::global_timer_ns() - t0 > kWaitNs) {
            *abort_flag = 1;
            record_status(status, SALA_ERR_TIMEOUT);
            return false;
        }
    }
    return true;
}

__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity,
                                              volatile int *abort_flag, int *status) {
    if (tc::mbar_test_wait(bar, parity)) return true;
    return wait_or_abort_slow(bar, parity, abort_flag, status);
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

// Two bf16 times a bf16 factor pair, rounded to nearest (one packed multiply).
__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t w, __nv_bfloat162 f2) {
    __nv_bfloat162 x = *reinterpret_cast<__nv_bfloat162 *>(&w);
    __nv_bfloat162 y = __hmul2(x, f2);
    return *reinterpret_cast<uint32_t *>(&y);
}

struct TcMaps {
    CUtensorMap q, k, v;   // loads: box 64 x 1 x 64, 128-byte swizzle
    CUtensorMap o;         // stores: box 32 x 1 x 64, no swizzle or (o_sw64) 64-byte swizzle
};

// host: 3-D tensor maps over q, k, v and o viewed as [T_total, H, 128] bf16
cudaError_t make_maps(TcMaps *m, const void *q, const void *k, const void *v, const void *o,
                      int64_t T_total, int H, bool o_sw64 = false);

}  // namespace tck
}  // namespace sala
