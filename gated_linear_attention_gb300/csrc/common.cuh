// Shared device helpers of the sala_gla library (not part of the public ABI).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "sala_gla.h"

namespace sala {

constexpr int kD = 128;     // head dimension (d_k = d_v)
constexpr int kChunk = 64;  // chunk length of the chunked prefill

// Record the first device-side error in the status word (later errors keep the first).
__device__ __forceinline__ void record_status(int *status, int code) {
    if (status) atomicCAS(status, 0, code);
}

// Index checks of the debug build (compiled with SALA_GLA_DEBUG): a failed check records
// SALA_ERR_DEBUG_CHECK in the status word and returns false, and the caller skips the access
// it guards. In the release build the check is the constant true and costs nothing.
#ifdef SALA_GLA_DEBUG
__device__ __forceinline__ bool dcheck(bool ok, int *status) {
    if (!ok) record_status(status, SALA_ERR_DEBUG_CHECK);
    return ok;
}
#else
__device__ __forceinline__ constexpr bool dcheck(bool, int *) { return true; }
#endif

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// Two bf16 in one 32-bit word -> two floats (low half is the lower address).
__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// Round two floats to nearest-even bf16 and pack them (x at the lower address).
__device__ __forceinline__ uint32_t float2_to_bf16x2(float x, float y) {
    __nv_bfloat162 p = __floats2bfloat162_rn(x, y);
    return *reinterpret_cast<uint32_t *>(&p);
}

// Start of a kernel launched by launch_dependent: the next kernel on the stream may be
// scheduled once every CTA of this one has passed here, and nothing below runs before the
// previous kernel on the stream has completed and its writes are visible.
__device__ __forceinline__ void dependent_start() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Launch as a programmatic dependent of the work before it on the stream: only the launch
// latency overlaps the previous grid's last wave (the kernel begins with dependent_start).
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kern)(KArgs...), unsigned grid, unsigned block, cudaStream_t st,
                             Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

}  // namespace sala
