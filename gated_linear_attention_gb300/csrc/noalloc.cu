// sala_gla_chunk_fwd_noalloc: the chunked prefill with its scratch in a fixed device array.
//
// For callers that cannot allocate device memory while they run the layer (engines that
// reserve nearly all of HBM up front, plug-in hosts whose execute path forbids allocation,
// latency-critical loops that cannot afford an allocator call). It launches the same
// kernels as sala_gla_chunk_fwd; only the source of the scratch differs.
#include <mutex>

#include "launch.h"

namespace sala {
namespace {

constexpr size_t kScratchBytes = SALA_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;
constexpr size_t kUnitBytes = size_t(kD) * kD * 4 + 4;  // one (segment, head): state + flag

// The scratch itself: one per device that loads the library, held until the process exits.
// In host code this name is only a stand-in; its device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

struct NoAllocDevice {
    std::once_flag once;
    cudaError_t error = cudaSuccess;
    bool supported = false;
    int sm_count = 0;
    unsigned char *scratch = nullptr;  // device address of g_noalloc_scratch
    int *status = nullptr;             // device address of the library's status word
};
NoAllocDevice g_na[kMaxDevices];

// Once per device, with that device current: look up the device addresses and set the
// kernels' shared-memory attributes. Allocates nothing.
NoAllocDevice *noalloc_device(int *err) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        *err = SALA_ERR_CUDA;
        return nullptr;
    }
    NoAllocDevice &d = g_na[dev];
    std::call_once(d.once, [&d, dev]() {
        int major = 0, minor = 0;
        d.error = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        if (d.error == cudaSuccess)
            d.error = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (d.error == cudaSuccess)
            d.error = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
        if (d.error != cudaSuccess) return;
        d.supported = major == 10 && minor == 3;
        if (!d.supported) return;
        d.error = cudaGetSymbolAddress(reinterpret_cast<void **>(&d.scratch), g_noalloc_scratch);
        if (d.error != cudaSuccess) return;
        d.error = device_status_address(&d.status);
        if (d.error != cudaSuccess) return;
        d.error = setup_fused_kernel();
    });
    if (d.error != cudaSuccess) {
        *err = SALA_ERR_CUDA;
        return nullptr;
    }
    if (!d.supported) {
        *err = SALA_ERR_UNSUPPORTED;
        return nullptr;
    }
    return &d;
}

bool al16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlap(const void *a, size_t na, const void *b, size_t nb) {
    if (!a || !b || na == 0 || nb == 0) return false;
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

size_t round256(size_t n) { return (n + 255) & ~size_t(255); }

}  // namespace
}  // namespace sala

using namespace sala;

extern "C" int sala_gla_chunk_fwd_noalloc(const void *q, const void *k, const void *v,
                                          const float *g, float scale, const float *h0,
                                          const int64_t *cu_seqlens, void *o, float *hT,
                                          int64_t B, int64_t T, int32_t H, int64_t num_seqs,
                                          void *stream) {
    // argument checks: the same rules as sala_gla_chunk_fwd
    if (B < 1 || T < 0 || H < 1) return SALA_ERR_INVALID_ARG;
    if (cu_seqlens && (B != 1 || num_seqs < 1)) return SALA_ERR_INVALID_ARG;
    const int64_t nseq = cu_seqlens ? num_seqs : B;
    const int64_t T_total = B * T;
    if (T_total > (int64_t(1) << 40) || nseq > (int64_t(1) << 31)) return SALA_ERR_INVALID_ARG;
    if (T_total > 0 && (!q || !k || !v || !g || !o)) return SALA_ERR_INVALID_ARG;
    const void *al[7] = {q, k, v, g, o, h0, hT};
    for (const void *p : al)
        if (p && !al16(p)) return SALA_ERR_MISALIGNED;
    if (cu_seqlens && (reinterpret_cast<uintptr_t>(cu_seqlens) & 7u)) return SALA_ERR_MISALIGNED;
    const size_t vec = size_t(T_total) * H * kD * 2, gb = size_t(T_total) * H * 4;
    const size_t sb = size_t(nseq) * H * kD * kD * 4;
    const void *ins[6] = {q, k, v, g, h0, cu_seqlens};
    const size_t in_sz[6] = {vec, vec, vec, gb, h0 ? sb : 0, cu_seqlens ? size_t(nseq + 1) * 8 : 0};
    for (int i = 0; i < 6; ++i)
        if (overlap(o, vec, ins[i], in_sz[i]) || overlap(hT, sb, ins[i], in_sz[i]))
            return SALA_ERR_INVALID_ARG;
    if (overlap(o, vec, hT, sb)) return SALA_ERR_INVALID_ARG;
    if (!hT && T_total == 0) return SALA_OK;

    // Segment length: the usual choice unless the fixed scratch needs longer segments. With L
    // tokens per segment there are at most T/L + nseq segments, so floor(T/L) may not exceed
    // r = (segments that fit) - nseq.
    const size_t table = round256(size_t(nseq + 2) * 8) + 256;   // segment table + ticket
    // (this check also keeps the unsigned subtraction below from wrapping)
    if (table + 256 + H * kUnitBytes > kScratchBytes) return SALA_ERR_TOO_LARGE;
    const int64_t units_fit = static_cast<int64_t>((kScratchBytes - table - 256) / kUnitBytes);
    const int64_t r = units_fit / H - nseq;
    if (r < 0) return SALA_ERR_TOO_LARGE;

    int err = SALA_OK;
    NoAllocDevice *d = noalloc_device(&err);
    if (!d) return err;

    int64_t seg_len = choose_segment_tokens(T_total, H, d->sm_count);
    const int64_t need_len = (T_total + 1 + r) / (r + 1);  // floor(T / need_len) <= r
    const int64_t need = ((need_len + kChunk - 1) / kChunk) * kChunk;
    if (seg_len < need) seg_len = need;
    const int64_t max_segs = T_total / seg_len + nseq;
    const int64_t max_units = max_segs * H;
    // the same bound as sala_gla_chunk_fwd (unit indices are 32-bit in the kernels); the
    // scratch size already implies it
    if (max_units >= (int64_t(1) << 31)) return SALA_ERR_TOO_LARGE;
    const size_t flag_bytes = round256(size_t(max_units) * 4);
    if (table + flag_bytes + size_t(max_units) * kD * kD * 4 > kScratchBytes)
        return SALA_ERR_TOO_LARGE;

    unsigned char *ws = d->scratch;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    SegTable tab;
    tab.cu = cu_seqlens;
    tab.T_row = T;
    tab.nseq = nseq;
    tab.seg_len = seg_len;
    tab.seg_off = reinterpret_cast<int64_t *>(ws);
    ChunkArgs a;
    a.q = static_cast<const uint16_t *>(q);
    a.k = static_cast<const uint16_t *>(k);
    a.v = static_cast<const uint16_t *>(v);
    a.g = g;
    a.scale = scale;
    a.o = static_cast<uint16_t *>(o);
    a.H = H;
    uint32_t *ticket = reinterpret_cast<uint32_t *>(ws + table - 256);
    uint32_t *flags = reinterpret_cast<uint32_t *>(ws + table);
    float *incl = reinterpret_cast<float *>(ws + table + flag_bytes);

    if (launch_seg_table(tab, T_total, ticket, flags, max_units, H, h0, hT, d->status, st) != cudaSuccess ||
        launch_prefill_fused(a, tab, T_total, max_units, h0, hT, incl, flags, ticket,
                             next_prefill_epoch(), d->sm_count, d->status, st) != cudaSuccess)
        return SALA_ERR_CUDA;
    return SALA_OK;
}
