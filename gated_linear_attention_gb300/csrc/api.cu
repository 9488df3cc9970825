// C ABI of the sala_gla library: argument validation, per-device set-up, scratch and launch
// order. Declarations and the contract of every entry point are in include/sala_gla.h.
#include <atomic>
#include <cstdlib>
#include <mutex>
#include <string>
#include <vector>

#include "launch.h"

namespace sala {
namespace {

constexpr int kMaxDevices = 64;

// Device-side status word (first error recorded by a kernel since the last query).
__device__ int g_device_status;

struct DeviceState {
    std::once_flag once;
    cudaError_t init_error = cudaSuccess;
    bool supported = false;
    int sm_count = 0;
    int *status = nullptr;         // device address of g_device_status
    cudaMemPool_t pool = nullptr;  // the library's own stream-ordered pool for scratch
};
DeviceState g_dev[kMaxDevices];

DeviceState *device_state(int *err) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        *err = SALA_ERR_CUDA;
        return nullptr;
    }
    DeviceState &d = g_dev[dev];
    std::call_once(d.once, [&d, dev]() {
        cudaDeviceProp prop;
        d.init_error = cudaGetDeviceProperties(&prop, dev);
        if (d.init_error != cudaSuccess) return;
        d.supported = prop.major == 10 && prop.minor == 3;
        d.sm_count = prop.multiProcessorCount;
        if (!d.supported) return;
        d.init_error = cudaGetSymbolAddress(reinterpret_cast<void **>(&d.status), g_device_status);
        if (d.init_error != cudaSuccess) return;
        // Scratch comes from a private pool that keeps its memory between calls (release
        // threshold = unlimited), so steady-state calls do not map or unmap device memory.
        cudaMemPoolProps props = {};
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        d.init_error = cudaMemPoolCreate(&d.pool, &props);
        if (d.init_error != cudaSuccess) return;
        uint64_t keep = ~uint64_t(0);
        d.init_error = cudaMemPoolSetAttribute(d.pool, cudaMemPoolAttrReleaseThreshold, &keep);
        if (d.init_error != cudaSuccess) return;
        d.init_error = setup_fused_kernel();
        if (d.init_error != cudaSuccess) return;
        d.init_error = setup_pair_kernel();
        if (d.init_error != cudaSuccess) return;
        d.init_error = setup_gdn_chunk_kernel();
    });
    if (d.init_error != cudaSuccess) {
        *err = SALA_ERR_CUDA;
        return nullptr;
    }
    if (!d.supported) {
        *err = SALA_ERR_UNSUPPORTED;
        return nullptr;
    }
    return &d;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Half-open byte ranges [a, a + na) and [b, b + nb) intersect (null or empty never does).
bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
    if (!a || !b || na == 0 || nb == 0) return false;
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

std::atomic<uint32_t> g_epoch{0};

// ---- timing instrumentation -------------------------------------------------------------
const char *const kKernelNames[kKernelCount] = {"seg_table", "prefill_fused", "recurrent_step",
                                                "recurrent_step_indexed", "output_norm_gate",
                                                "qk_prologue", "gdn_step", "gdn_fwd",
                                                "gdn_newv", "prefill_pair"};
struct TimingRecord {
    int id;
    cudaEvent_t start, stop;
};
std::atomic<bool> g_timing{false};
std::mutex g_timing_mu;
std::vector<TimingRecord> g_records;

void clear_records_locked() {
    for (auto &r : g_records) {
        cudaEventDestroy(r.start);
        cudaEventDestroy(r.stop);
    }
    g_records.clear();
}

}  // namespace

// Tokens per segment. Each unit pays a fixed cost (its state pass ramp, the hand-off, the
// output pipeline fill) worth several chunks, so long segments win when every SM gets many
// units; when the whole job is only a few waves of units, the last wave's imbalance dominates
// and shorter segments win. Measured on GB300 (H = 32): 8192 tokens (about 1.7K tokens per
// SM) is fastest at 640; 65536 and 131072 tokens (14K and 28K per SM) at 1024, where 512
// costs 25-30 % more. SALA_GLA_SEGMENT_TOKENS overrides the choice (rounded up to a multiple
// of 64).
int64_t choose_segment_tokens(int64_t T_total, int64_t H, int sm_count) {
    static const int64_t forced = []() -> int64_t {
        const char *e = getenv("SALA_GLA_SEGMENT_TOKENS");
        if (!e) return 0;
        const long long v = atoll(e);
        return v > 0 ? ((v + kChunk - 1) / kChunk) * kChunk : 0;
    }();
    if (forced) return forced;
    const int64_t per_sm = T_total * H / (sm_count > 0 ? sm_count : 1);
    int64_t L = per_sm > 8192 ? 1024 : 640;
    if (T_total < L) L = ((T_total + kChunk - 1) / kChunk) * kChunk;
    return L < kChunk ? kChunk : L;
}

uint32_t next_prefill_epoch() {
    uint32_t e = g_epoch.fetch_add(1, std::memory_order_relaxed) + 1;
    if (e == 0) e = g_epoch.fetch_add(1, std::memory_order_relaxed) + 1;
    return e;
}

cudaError_t device_status_address(int **out) {
    return cudaGetSymbolAddress(reinterpret_cast<void **>(out), g_device_status);
}

LaunchTimer::LaunchTimer(KernelId id, cudaStream_t stream) : id_(id), stream_(stream) {
    if (!g_timing.load(std::memory_order_relaxed)) return;
    if (cudaEventCreate(&start_) != cudaSuccess) {
        start_ = nullptr;
        return;
    }
    if (cudaEventRecord(start_, stream_) != cudaSuccess) {
        cudaEventDestroy(start_);
        start_ = nullptr;
    }
}

LaunchTimer::~LaunchTimer() {
    if (!start_) return;
    cudaEvent_t stop = nullptr;
    if (cudaEventCreate(&stop) != cudaSuccess || cudaEventRecord(stop, stream_) != cudaSuccess) {
        cudaEventDestroy(start_);
        if (stop) cudaEventDestroy(stop);
        return;
    }
    std::lock_guard<std::mutex> lock(g_timing_mu);
    g_records.push_back({id_, start_, stop});
}

namespace {
std::atomic<uint64_t> g_fault_wait_ns{0};
std::atomic<int64_t> g_fault_withhold{-1};
}  // namespace

// Prefill kernel choice: -1 until first read from SALA_GLA_PREFILL, then 0 (per call), 1, 2.
std::atomic<int> g_prefill_kernel{-1};

int prefill_kernel_choice() {
    int k = g_prefill_kernel.load();
    if (k < 0) {
        const char *e = getenv("SALA_GLA_PREFILL");
        const int v = !e ? 0 : std::string(e) == "pair" ? 2 : std::string(e) == "fused" ? 1 : 0;
        g_prefill_kernel.compare_exchange_strong(k, v);
        k = g_prefill_kernel.load();
    }
    return k;
}

void prefill_fault_knobs(uint64_t *wait_ns, int64_t *withhold) {
    *wait_ns = g_fault_wait_ns.load();
    *withhold = g_fault_withhold.load();
}

}  // namespace sala

using namespace sala;

extern "C" {

int sala_gla_set_prefill_kernel(int kernel) {
    if (kernel < 0 || kernel > 2) return SALA_ERR_INVALID_ARG;
    g_prefill_kernel.store(kernel);
    return SALA_OK;
}

int sala_gla_debug_prefill_knobs(uint64_t flag_wait_ns, int64_t withhold_unit) {
    if (withhold_unit < -1) return SALA_ERR_INVALID_ARG;
    g_fault_wait_ns.store(flag_wait_ns);
    g_fault_withhold.store(withhold_unit);
    return SALA_OK;
}

const char *sala_gla_version(void) { return "0.1.0"; }

int sala_gla_kernel_count(void) { return kKernelCount; }

const char *sala_gla_kernel_name(int kernel) {
    return (kernel >= 0 && kernel < kKernelCount) ? kKernelNames[kernel] : "unknown";
}

int sala_gla_timing_enable(int enable) {
    std::lock_guard<std::mutex> lock(g_timing_mu);
    if (enable) clear_records_locked();
    g_timing.store(enable != 0);
    return SALA_OK;
}

int sala_gla_timing_read(int kernel, double *total_ms, int64_t *launches) {
    if (kernel < 0 || kernel >= kKernelCount || !total_ms || !launches) return SALA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g_timing_mu);
    double sum = 0.0;
    int64_t count = 0;
    for (const auto &r : g_records) {
        if (r.id != kernel) continue;
        float ms = 0.f;
        if (cudaEventSynchronize(r.stop) != cudaSuccess ||
            cudaEventElapsedTime(&ms, r.start, r.stop) != cudaSuccess)
            return SALA_ERR_CUDA;
        sum += ms;
        ++count;
    }
    *total_ms = sum;
    *launches = count;
    return SALA_OK;
}

const char *sala_gla_status_string(int status) {
    switch (status) {
    case SALA_OK: return "success";
    case SALA_ERR_INVALID_ARG: return "invalid argument";
    case SALA_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case SALA_ERR_UNSUPPORTED: return "unsupported device (needs compute capability 10.3)";
    case SALA_ERR_CUDA: return "CUDA runtime error";
    case SALA_ERR_TIMEOUT: return "device-side wait timed out";
    case SALA_ERR_BAD_SEQLENS: return "cu_seqlens is not monotone from 0 to T";
    case SALA_ERR_TOO_LARGE:
        return "problem needs more scratch than the no-allocation entry point's fixed buffer";
    case SALA_ERR_BAD_INDEX: return "a state index is at or past the pool size";
    case SALA_ERR_DEBUG_CHECK: return "debug build: a device-side index check failed (access skipped)";
    default: return "unknown status";
    }
}

int sala_gla_get_device_status(void *stream) {
    int err = SALA_OK;
    DeviceState *d = device_state(&err);
    if (!d) return err;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return SALA_ERR_CUDA;
    int value = 0, zero = 0;
    if (cudaMemcpy(&value, d->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return SALA_ERR_CUDA;
    if (cudaMemcpy(d->status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
        return SALA_ERR_CUDA;
    return value;
}

int sala_gla_recurrent_step(const void *q, const void *k, const void *v, const float *g,
                            float scale, float *S_inout, void *o, int64_t N, int32_t H,
                            void *stream) {
    if (N < 0 || H < 1) return SALA_ERR_INVALID_ARG;
    if (N == 0) return SALA_OK;
    if (N > (int64_t(1) << 31) / H) return SALA_ERR_INVALID_ARG;
    if (!q || !k || !v || !g || !S_inout || !o) return SALA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(S_inout) ||
        !aligned16(o))
        return SALA_ERR_MISALIGNED;
    const size_t units = static_cast<size_t>(N) * H;
    const size_t vec = units * kD * 2, gb = units * 4, sb = units * kD * kD * 4;
    const void *ins[4] = {q, k, v, g};
    const size_t in_sz[4] = {vec, vec, vec, gb};
    for (int i = 0; i < 4; ++i)
        if (overlaps(S_inout, sb, ins[i], in_sz[i]) || overlaps(o, vec, ins[i], in_sz[i]))
            return SALA_ERR_INVALID_ARG;
    if (overlaps(S_inout, sb, o, vec)) return SALA_ERR_INVALID_ARG;
    int err = SALA_OK;
    if (!device_state(&err)) return err;
    if (launch_recurrent_step(q, k, v, g, scale, S_inout, o, static_cast<int64_t>(units),
                              static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return SALA_ERR_CUDA;
    return SALA_OK;
}

namespace {
// Arguments of a q/k prologue: both weights present and 16-byte aligned, eps >= 0, theta > 0.
int check_prologue(const sala_qk_prologue *p) {
    if (!p) return SALA_OK;
    if (!p->q_weight || !p->k_weight || !(p->eps >= 0.f) || !(p->rope_theta > 0.f))
        return SALA_ERR_INVALID_ARG;
    if (!aligned16(p->q_weight) || !aligned16(p->k_weight)) return SALA_ERR_MISALIGNED;
    return SALA_OK;
}
}  // namespace

int sala_gla_recurrent_step_indexed(const void *q, const void *k, const void *v, const float *g,
                                    float scale, void *state_pool, int32_t state_dtype,
                                    const int32_t *state_indices, int64_t P, void *o, int64_t N,
                                    int32_t H, const sala_qk_prologue *prologue,
                                    const int64_t *positions, void *stream) {
    if (const int e = check_prologue(prologue)) return e;
    if (prologue && !positions) return SALA_ERR_INVALID_ARG;
    if (prologue && (reinterpret_cast<uintptr_t>(positions) & 7u)) return SALA_ERR_MISALIGNED;
    if (N < 0 || H < 1 || P < 1) return SALA_ERR_INVALID_ARG;
    if (state_dtype != SALA_STATE_F32 && state_dtype != SALA_STATE_BF16) return SALA_ERR_INVALID_ARG;
    if (N == 0) return SALA_OK;
    if (N > (int64_t(1) << 31) / H || P > (int64_t(1) << 40) / H) return SALA_ERR_INVALID_ARG;
    if (!q || !k || !v || !g || !state_pool || !state_indices || !o) return SALA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(state_pool) ||
        !aligned16(state_indices) || !aligned16(o))
        return SALA_ERR_MISALIGNED;
    const size_t units = static_cast<size_t>(N) * H;
    const size_t vec = units * kD * 2, gb = units * 4, ib = static_cast<size_t>(N) * 4;
    const size_t pb = static_cast<size_t>(P) * H * kD * kD * (state_dtype == SALA_STATE_BF16 ? 2 : 4);
    const void *ins[5] = {q, k, v, g, state_indices};
    const size_t in_sz[5] = {vec, vec, vec, gb, ib};
    for (int i = 0; i < 5; ++i)
        if (overlaps(state_pool, pb, ins[i], in_sz[i]) || overlaps(o, vec, ins[i], in_sz[i]))
            return SALA_ERR_INVALID_ARG;
    if (overlaps(state_pool, pb, o, vec)) return SALA_ERR_INVALID_ARG;
    int err = SALA_OK;
    DeviceState *d = device_state(&err);
    if (!d) return err;
    if (launch_recurrent_step_indexed(q, k, v, g, scale, state_pool, state_dtype == SALA_STATE_BF16,
                                      state_indices, P, o, N, H, make_qk_prologue(prologue, positions),
                                      d->status, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return SALA_ERR_CUDA;
    return SALA_OK;
}

int sala_gla_qk_prologue(void *q, void *k, const sala_qk_prologue *prologue,
                         const int64_t *cu_seqlens, const int64_t *start_pos, int64_t B,
                         int64_t T, int32_t H, int64_t num_seqs, void *stream) {
    if (!prologue) return SALA_ERR_INVALID_ARG;
    if (const int e = check_prologue(prologue)) return e;
    if (B < 1 || T < 0 || H < 1) return SALA_ERR_INVALID_ARG;
    if (cu_seqlens && (B != 1 || num_seqs < 1)) return SALA_ERR_INVALID_ARG;
    const int64_t nseq = cu_seqlens ? num_seqs : B;
    const int64_t T_total = B * T;
    if (T_total > (int64_t(1) << 31) - 1 || nseq > (int64_t(1) << 31)) return SALA_ERR_INVALID_ARG;
    if (T_total == 0) return SALA_OK;
    if (!q || !k) return SALA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k)) return SALA_ERR_MISALIGNED;
    if ((cu_seqlens && (reinterpret_cast<uintptr_t>(cu_seqlens) & 7u)) ||
        (start_pos && (reinterpret_cast<uintptr_t>(start_pos) & 7u)))
        return SALA_ERR_MISALIGNED;
    const size_t vec = static_cast<size_t>(T_total) * H * kD * 2;
    if (overlaps(q, vec, k, vec)) return SALA_ERR_INVALID_ARG;
    const size_t wb = kD * 2;
    if (overlaps(q, vec, prologue->q_weight, wb) || overlaps(q, vec, prologue->k_weight, wb) ||
        overlaps(k, vec, prologue->q_weight, wb) || overlaps(k, vec, prologue->k_weight, wb))
        return SALA_ERR_INVALID_ARG;
    int err = SALA_OK;
    DeviceState *d = device_state(&err);
    if (!d) return err;
    SegTable tab{};
    tab.cu = cu_seqlens;
    tab.T_row = T;
    tab.nseq = nseq;
    if (launch_qk_prologue(q, k, make_qk_prologue(prologue, nullptr), tab, start_pos, T_total, H,
                           d->status, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return SALA_ERR_CUDA;
    return SALA_OK;
}

int sala_gla_output_norm_gate(const void *o, const void *z, const void *w, float eps, void *out,
                              int64_t T, int32_t H, void *stream) {
    if (T < 0 || H < 1 || !(eps >= 0.f)) return SALA_ERR_INVALID_ARG;
    if (T == 0) return SALA_OK;
    if (T > (int64_t(1) << 31) - 1 || H > 4096) return SALA_ERR_INVALID_ARG;
    if (!o || !z || !w || !out) return SALA_ERR_INVALID_ARG;
    if (!aligned16(o) || !aligned16(z) || !aligned16(w) || !aligned16(out)) return SALA_ERR_MISALIGNED;
    const size_t vec = static_cast<size_t>(T) * H * kD * 2, wb = static_cast<size_t>(H) * kD * 2;
    // out may be o itself (in place), but may not overlap z, w or o partially
    if (out != o && overlaps(out, vec, o, vec)) return SALA_ERR_INVALID_ARG;
    if (overlaps(out, vec, z, vec) || overlaps(out, vec, w, wb)) return SALA_ERR_INVALID_ARG;
    int err = SALA_OK;
    if (!device_state(&err)) return err;
    if (launch_output_norm_gate(o, z, w, eps, out, T, H, static_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
        return SALA_ERR_CUDA;
    return SALA_OK;
}

int sala_gla_gdn_recurrent_step(const void *q, const void *k, const void *v, const float *g,
                                const float *beta, float scale, float *S_inout, void *o,
                                int64_t N, int32_t H, void *stream) {
    if (N < 0 || H < 1) return SALA_ERR_INVALID_ARG;
    if (N == 0) return SALA_OK;
    if (N > (int64_t(1) << 31) / H) return SALA_ERR_INVALID_ARG;
    if (!q || !k || !v || !g || !beta || !S_inout || !o) return SALA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(beta) ||
        !aligned16(S_inout) || !aligned16(o))
        return SALA_ERR_MISALIGNED;
    const size_t units = static_cast<size_t>(N) * H;
    const size_t vec = units * kD * 2, gb = units * 4, sb = units * kD * kD * 4;
    const void *ins[5] = {q, k, v, g, beta};
    const size_t in_sz[5] = {vec, vec, vec, gb, gb};
    for (int i = 0; i < 5; ++i)
        if (overlaps(S_inout, sb, ins[i], in_sz[i]) || overlaps(o, vec, ins[i], in_sz[i]))
            return SALA_ERR_INVALID_ARG;
    if (overlaps(S_inout, sb, o, vec)) return SALA_ERR_INVALID_ARG;
    int err = SALA_OK;
    if (!device_state(&err)) return err;
    if (launch_gdn_step(q, k, v, g, beta, scale, S_inout, o, static_cast<int64_t>(units),
                        static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return SALA_ERR_CUDA;
    return SALA_OK;
}

int sala_gla_gdn_fwd(const void *q, const void *k, const void *v, const float *g,
                     const float *beta, float scale, const float *h0, const int64_t *cu_seqlens,
                     void *o, float *hT, int64_t B, int64_t T, int32_t H, int64_t num_seqs,
                     void *stream) {
    if (B < 1 || T < 0 || H < 1) return SALA_ERR_INVALID_ARG;
    if (cu_seqlens && (B != 1 || num_seqs < 1)) return SALA_ERR_INVALID_ARG;
    const int64_t nseq = cu_seqlens ? num_seqs : B;
    const int64_t T_total = B * T;
    if (T_total > (int64_t(1) << 40) || nseq * H > (int64_t(1) << 31) - 1) return SALA_ERR_INVALID_ARG;
    if (T_total > 0 && (!q || !k || !v || !g || !beta || !o)) return SALA_ERR_INVALID_ARG;
    const void *al[8] = {q, k, v, g, beta, o, h0, hT};
    for (const void *p : al)
        if (p && !aligned16(p)) return SALA_ERR_MISALIGNED;
    if (cu_seqlens && (reinterpret_cast<uintptr_t>(cu_seqlens) & 7u)) return SALA_ERR_MISALIGNED;
    const size_t vec = static_cast<size_t>(T_total) * H * kD * 2, gb = static_cast<size_t>(T_total) * H * 4;
    const size_t sb = static_cast<size_t>(nseq) * H * kD * kD * 4;
    const void *ins[7] = {q, k, v, g, beta, h0, cu_seqlens};
    const size_t in_sz[7] = {vec, vec, vec, gb, gb, h0 ? sb : 0, cu_seqlens ? size_t(nseq + 1) * 8 : 0};
    for (int i = 0; i < 7; ++i)
        if (overlaps(o, vec, ins[i], in_sz[i]) || overlaps(hT, sb, ins[i], in_sz[i]))
            return SALA_ERR_INVALID_ARG;
    if (overlaps(o, vec, hT, sb)) return SALA_ERR_INVALID_ARG;
    if (!hT && T_total == 0) return SALA_OK;
    int err = SALA_OK;
    if (!device_state(&err)) return err;
    SegTable tab{};
    tab.cu = cu_seqlens;
    tab.T_row = T;
    tab.nseq = nseq;
    if (launch_gdn_fwd(q, k, v, g, beta, scale, h0, tab, T_total, o, hT, H,
                       static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return SALA_ERR_CUDA;
    return SALA_OK;
}

int sala_gla_gdn_chunk_fwd(const void *q, const void *k, const void *v, const float *g,
                           const float *beta, float scale, const float *h0,
                           const int64_t *cu_seqlens, void *o, float *hT, int64_t B, int64_t T,
                           int32_t H, int64_t num_seqs, void *stream) {
    if (B < 1 || T < 0 || H < 1) return SALA_ERR_INVALID_ARG;
    if (cu_seqlens && (B != 1 || num_seqs < 1)) return SALA_ERR_INVALID_ARG;
    const int64_t nseq = cu_seqlens ? num_seqs : B;
    const int64_t T_total = B * T;
    // TMA coordinates of the tiles are 32-bit token indices
    if (T_total > (int64_t(1) << 31) - 64 || nseq * H > (int64_t(1) << 31) - 1) return SALA_ERR_INVALID_ARG;
    if (T_total > 0 && (!q || !k || !v || !g || !beta || !o)) return SALA_ERR_INVALID_ARG;
    const void *al[8] = {q, k, v, g, beta, o, h0, hT};
    for (const void *p : al)
        if (p && !aligned16(p)) return SALA_ERR_MISALIGNED;
    if (cu_seqlens && (reinterpret_cast<uintptr_t>(cu_seqlens) & 7u)) return SALA_ERR_MISALIGNED;
    const size_t vec = static_cast<size_t>(T_total) * H * kD * 2, gb = static_cast<size_t>(T_total) * H * 4;
    const size_t sb = static_cast<size_t>(nseq) * H * kD * kD * 4;
    const void *ins[7] = {q, k, v, g, beta, h0, cu_seqlens};
    const size_t in_sz[7] = {vec, vec, vec, gb, gb, h0 ? sb : 0, cu_seqlens ? size_t(nseq + 1) * 8 : 0};
    for (int i = 0; i < 7; ++i)
        if (overlaps(o, vec, ins[i], in_sz[i]) || overlaps(hT, sb, ins[i], in_sz[i]))
            return SALA_ERR_INVALID_ARG;
    if (overlaps(o, vec, hT, sb)) return SALA_ERR_INVALID_ARG;
    if (!hT && T_total == 0) return SALA_OK;
    int err = SALA_OK;
    DeviceState *d = device_state(&err);
    if (!d) return err;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // new_v of every token, then the Simple GLA chunked prefill with it in place of v
    void *nv = nullptr;
    if (T_total > 0 && cudaMallocFromPoolAsync(&nv, vec, d->pool, st) != cudaSuccess)
        return SALA_ERR_CUDA;
    SegTable tab{};
    tab.cu = cu_seqlens;
    tab.T_row = T;
    tab.nseq = nseq;
    int rc = SALA_OK;
    if (T_total > 0 &&
        launch_gdn_newv(k, v, g, beta, h0, tab, T_total, nv, H, d->status, st) != cudaSuccess)
        rc = SALA_ERR_CUDA;
    if (rc == SALA_OK)
        rc = sala_gla_chunk_fwd(q, k, T_total > 0 ? nv : v, g, scale, h0, cu_seqlens, o, hT, B, T,
                                H, num_seqs, stream);
    if (nv && cudaFreeAsync(nv, st) != cudaSuccess && rc == SALA_OK) rc = SALA_ERR_CUDA;
    return rc;
}

int sala_gla_chunk_fwd(const void *q, const void *k, const void *v, const float *g, float scale,
                       const float *h0, const int64_t *cu_seqlens, void *o, float *hT,
                       int64_t B, int64_t T, int32_t H, int64_t num_seqs, void *stream) {
    if (B < 1 || T < 0 || H < 1) return SALA_ERR_INVALID_ARG;
    if (cu_seqlens && (B != 1 || num_seqs < 1)) return SALA_ERR_INVALID_ARG;
    const int64_t nseq = cu_seqlens ? num_seqs : B;
    const int64_t T_total = B * T;
    if (T_total > (int64_t(1) << 40) || nseq > (int64_t(1) << 31)) return SALA_ERR_INVALID_ARG;
    if (T_total > 0 && (!q || !k || !v || !g || !o)) return SALA_ERR_INVALID_ARG;
    const void *al[7] = {q, k, v, g, o, h0, hT};
    for (const void *p : al)
        if (p && !aligned16(p)) return SALA_ERR_MISALIGNED;
    if (cu_seqlens && (reinterpret_cast<uintptr_t>(cu_seqlens) & 7u)) return SALA_ERR_MISALIGNED;
    const size_t vec = static_cast<size_t>(T_total) * H * kD * 2, gb = static_cast<size_t>(T_total) * H * 4;
    const size_t sb = static_cast<size_t>(nseq) * H * kD * kD * 4;
    const void *ins[6] = {q, k, v, g, h0, cu_seqlens};
    const size_t in_sz[6] = {vec, vec, vec, gb, h0 ? sb : 0, cu_seqlens ? size_t(nseq + 1) * 8 : 0};
    for (int i = 0; i < 6; ++i)
        if (overlaps(o, vec, ins[i], in_sz[i]) || overlaps(hT, sb, ins[i], in_sz[i]))
            return SALA_ERR_INVALID_ARG;
    if (overlaps(o, vec, hT, sb)) return SALA_ERR_INVALID_ARG;
    if (!hT && T_total == 0) return SALA_OK;

    int err = SALA_OK;
    DeviceState *d = device_state(&err);
    if (!d) return err;
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    const int64_t seg_len = choose_segment_tokens(T_total, H, d->sm_count);
    const int64_t max_segs = T_total / seg_len + nseq;  // sum of ceil(len/L) <= T/L + nseq
    const int64_t max_units = max_segs * H;
    if (max_units > (int64_t(1) << 31) - 1) return SALA_ERR_INVALID_ARG;

    // scratch: segment table, work ticket, hand-off flags, hand-off states
    const size_t off_bytes = ((static_cast<size_t>(nseq) + 2) * 8 + 255) & ~size_t(255);
    const size_t tick_bytes = 256;
    const size_t flag_bytes = (static_cast<size_t>(max_units) * 4 + 255) & ~size_t(255);
    const size_t st_bytes = static_cast<size_t>(max_units) * kD * kD * 4;
    char *ws = nullptr;
    if (cudaMallocFromPoolAsync(reinterpret_cast<void **>(&ws),
                                off_bytes + tick_bytes + flag_bytes + st_bytes, d->pool,
                                st) != cudaSuccess)
        return SALA_ERR_CUDA;

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
    uint32_t *ticket = reinterpret_cast<uint32_t *>(ws + off_bytes);
    uint32_t *flags = reinterpret_cast<uint32_t *>(ws + off_bytes + tick_bytes);
    float *incl = reinterpret_cast<float *>(ws + off_bytes + tick_bytes + flag_bytes);

    int rc = SALA_OK;
    // many waves of units per SM: two CTAs per SM overlap each other's serial chains; a few
    // waves: one unit per SM (twice as many units in flight would lengthen the chains of
    // hand-offs within a wave)
    const int which = prefill_kernel_choice();
    const bool pair = which == 2 || (which == 0 && T_total * H > int64_t(8192) * d->sm_count);
    if (launch_seg_table(tab, T_total, ticket, flags, max_units, H, h0, hT, d->status, st) != cudaSuccess ||
        (pair ? launch_prefill_pair(a, tab, T_total, max_units, h0, hT, incl, flags, ticket,
                                    next_prefill_epoch(), 2 * d->sm_count, d->status, st)
              : launch_prefill_fused(a, tab, T_total, max_units, h0, hT, incl, flags, ticket,
                                     next_prefill_epoch(), d->sm_count, d->status, st)) != cudaSuccess)
        rc = SALA_ERR_CUDA;
    if (cudaFreeAsync(ws, st) != cudaSuccess) rc = SALA_ERR_CUDA;
    return rc;
}

}  // extern "C"
