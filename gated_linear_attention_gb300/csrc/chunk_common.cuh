// Work decomposition shared by the kernels of the chunked prefill.
//
// A call covers `nseq` sequences packed back to back (token index = position in the packed
// [T_total, H, 128] view). Each sequence is cut into segments of `seg_len` tokens (a
// multiple of the 64-token chunk); the last segment of a sequence may be shorter. A work
// unit is one (segment, head) pair. Segments are numbered globally in sequence order;
// seg_off[n] is the first segment of sequence n and seg_off[nseq] the total. Units are
// numbered segment-major (unit = segment * H + head) so that all heads of one segment run
// side by side and share the cache lines of g, which holds all heads of a token in one line.
#pragma once

#include "common.cuh"

namespace sala {

struct SegTable {
    const int64_t *cu;   // [nseq+1] token offsets (device), or nullptr for B equal rows of T_row
    int64_t T_row;       // row length when cu == nullptr
    int64_t nseq;
    int64_t seg_len;     // tokens per segment, multiple of kChunk
    int64_t *seg_off;    // [nseq+2]: segment offsets, then a validity word at [nseq+1]
};

// Tensors of one prefill call (device pointers) and its scratch.
struct ChunkArgs {
    const uint16_t *q, *k, *v;  // bf16 [T_total, H, 128]
    const float *g;             // [T_total, H]
    float scale;
    uint16_t *o;                // bf16 [T_total, H, 128]
    int H;
};

__device__ __forceinline__ int64_t seq_begin(const SegTable &t, int64_t n) {
    return t.cu ? t.cu[n] : n * t.T_row;
}

// Locate segment `sigma` (0 <= sigma < total): its sequence n and token range [t0, t1).
// Returns false if sigma is past the last segment or the table is invalid.
__device__ __forceinline__ bool locate_segment(const SegTable &t, int64_t sigma, int64_t &n,
                                               int64_t &t0, int64_t &t1) {
    if (t.seg_off[t.nseq + 1] != 1) return false;
    if (sigma >= t.seg_off[t.nseq]) return false;
    int64_t lo = 0, hi = t.nseq - 1;  // largest n with seg_off[n] <= sigma
    while (lo < hi) {
        const int64_t mid = (lo + hi + 1) >> 1;
        if (t.seg_off[mid] <= sigma) lo = mid; else hi = mid - 1;
    }
    n = lo;
    const int64_t bos = seq_begin(t, n), eos = seq_begin(t, n + 1);
    t0 = bos + (sigma - t.seg_off[n]) * t.seg_len;
    t1 = min(t0 + t.seg_len, eos);
    return true;
}

}  // namespace sala
