/*
 * sala_gla.h -- C ABI of the Simple GLA (Lightning attention) hot path on GB300 (sm_103a).
 *
 * The operation. Per sequence n and head h, with a [d_k x d_v] = [128 x 128] fp32 state S
 * (row index = key dimension, column index = value dimension):
 *
 *     S_t = exp(g_t) * S_{t-1} + k_t^T v_t          (decay, then rank-1 update)
 *     o_t = scale * q_t S_t                          (query reads the updated state)
 *
 * Source: "MiniCPM-SALA — Complete Blueprint", section "B2 lightning-attn (Simple GLA)",
 * block "Simple GLA Recurrence" (decay by alpha = exp(g), add k^T (outer) v, read
 * o = q S x 0.08839 = 1/sqrt(128)); the state is the recurrent memory held per request and
 * layer ("Memory Architecture", MambaPool temporal states, written back after each step).
 * The call shape (q, k, v, g, scale, initial state, whether to return the final state,
 * packed sequences through cu_seqlens) follows the chunked/recurrent operator interface
 * shown in "Formulas and Code for Adapting Inference to GDN/KDA Linear Modules", section 2.1.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller; the library keeps none of
 *     them after the call returns. Buffers must stay valid until the work queued on
 *     `stream` has executed.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream). Work is
 *     queued asynchronously; no call synchronises the host except
 *     sala_gla_get_device_status().
 *   - Layouts are row-major with the last index contiguous. bf16 is IEEE bfloat16 stored in
 *     16-bit words. Every pointer must be 16-byte aligned.
 *   - Head dimension is fixed at 128 for q, k and v.
 *   - A call returns a sala_status. Argument errors are detected on the host before anything
 *     is queued. Errors that only the device can see (malformed cu_seqlens contents) are
 *     recorded in a per-device status word, the affected work is skipped, and
 *     sala_gla_get_device_status() reports them.
 *   - Entry points are thread-safe. Per-device one-time set-up (kernel attributes) happens
 *     on the first call on that device.
 */
#ifndef SALA_GLA_H
#define SALA_GLA_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SALA_OK = 0,
    SALA_ERR_INVALID_ARG = 1, /* null pointer where one is required, bad size, aliasing */
    SALA_ERR_MISALIGNED = 2,  /* a pointer is not 16-byte aligned */
    SALA_ERR_UNSUPPORTED = 3, /* device is not sm_103 / compute capability 10.3 */
    SALA_ERR_CUDA = 4,        /* a CUDA runtime call failed (launch, allocation) */
    SALA_ERR_TIMEOUT = 5,     /* a bounded device-side wait gave up */
    SALA_ERR_BAD_SEQLENS = 6, /* device-detected: cu_seqlens not monotone or last != T */
    SALA_ERR_TOO_LARGE = 7,   /* sala_gla_chunk_fwd_noalloc: problem exceeds its fixed scratch */
    SALA_ERR_BAD_INDEX = 8,   /* device-detected: a state index at or past the pool size */
    SALA_ERR_DEBUG_CHECK = 9  /* debug build only (SALA_GLA_DEBUG): a device-side index check
                                 failed; the access it guards was skipped */
} sala_status;

/*
 * The q/k prologue of a lightning layer ("MiniCPM-SALA — Complete Blueprint", section "B2
 * lightning-attn (Simple GLA)": per-head QK RMSNorm with a 128-wide weight, then RoPE with
 * theta = 10000 computed in fp32 and rounded to bf16). For each head vector x of q (or k):
 *     y = bf16( x / sqrt(mean(x^2) + eps) * weight )
 *     for i < 64, with a = float(pos) * inv_freq[i], inv_freq[i] = float(theta^(-i/64)):
 *         out[i]      = bf16( y[i] cos a - y[i + 64] sin a )
 *         out[i + 64] = bf16( y[i + 64] cos a + y[i] sin a )
 * (the rotate-half pairing (i, i + 64); pos is the token's position in its sequence).
 */
typedef struct {
    const void *q_weight; /* bf16 [128] RMSNorm weight of q (shared by all heads) */
    const void *k_weight; /* bf16 [128] RMSNorm weight of k */
    float eps;            /* RMSNorm epsilon, e.g. 1e-6 */
    float rope_theta;     /* RoPE base, e.g. 10000 */
} sala_qk_prologue;

/* Storage type of the states in a state pool (sala_gla_recurrent_step_indexed). The
 * arithmetic is fp32 either way. */
typedef enum {
    SALA_STATE_F32 = 0,  /* fp32 states, 64 KB per (slot, head) */
    SALA_STATE_BF16 = 1  /* bf16 states, 32 KB per (slot, head); rounded to nearest even on store */
} sala_state_dtype;

/*
 * Chunked prefill (chunk size 64).
 *
 * Computes o and, optionally, the final state of every sequence, exactly as the recurrence
 * above run token by token from h0. Internally the sequence is cut into 64-token chunks
 * (intra-chunk causal (Q K^T * decay mask) V plus inter-chunk q S and the state carry;
 * "Formulas and Code for Adapting Inference to GDN/KDA Linear Modules", section 1.2, taken
 * without the delta rule) and the state is carried across chunks by a chunk-parallel state
 * pass followed by an output pass.
 *
 *   q, k, v    bf16 [B, T, H, 128]. With cu_seqlens: B must be 1 and the T tokens hold the
 *              num_seqs sequences packed back to back.
 *   g          fp32 [B, T, H] per-token, per-head log-decay (<= 0 for a decaying state).
 *   scale      output scale, typically 128^-0.5.
 *   h0         fp32 [Nseq, H, 128, 128] initial states, or NULL for zeros. Nseq = B without
 *              cu_seqlens, num_seqs with it.
 *   cu_seqlens int64 [num_seqs + 1] DEVICE array of sequence offsets (0 = cu[0] <= cu[1]
 *              <= ... <= cu[num_seqs] = T), or NULL. A sequence may be empty: its final
 *              state is h0 (or zeros).
 *   o          bf16 [B, T, H, 128] output (written; round to nearest even).
 *   hT         fp32 [Nseq, H, 128, 128] final states, or NULL (not computed). hT may not
 *              alias h0.
 *   B, T, H    sizes; B >= 1, T >= 0, H >= 1. num_seqs >= 1 when cu_seqlens is given,
 *              ignored otherwise.
 *
 * Scratch: the sequences are cut into segments whose states are handed from one segment to
 * the next (64 KB per segment and head, plus a segment table and one flag word per segment
 * and head). This scratch is taken from a stream-ordered memory pool that the library
 * creates once per device (cudaMallocFromPoolAsync on `stream`) and returned to it when the
 * call's work is done (cudaFreeAsync), so the host never waits. The pool keeps its memory
 * for later calls. A device-side wait that gives up (2 s) records SALA_ERR_TIMEOUT in the
 * status word (sala_gla_get_device_status).
 * Errors: SALA_ERR_INVALID_ARG, SALA_ERR_MISALIGNED, SALA_ERR_UNSUPPORTED, SALA_ERR_CUDA.
 */
int sala_gla_chunk_fwd(const void *q, const void *k, const void *v, const float *g, float scale,
                       const float *h0, const int64_t *cu_seqlens, void *o, float *hT,
                       int64_t B, int64_t T, int32_t H, int64_t num_seqs, void *stream);

/*
 * One-token recurrent decode, state updated in place.
 *
 * For each of the N sequences and H heads: S = exp(g) S + k^T v; o = scale q S (the
 * Blueprint page's decode step: load the state, decay, outer-product update, query, save
 * the updated state back).
 *
 *   q, k, v    bf16 [N, H, 128]
 *   g          fp32 [N, H]
 *   S_inout    fp32 [N, H, 128, 128], read and overwritten with the updated states. Must not
 *              overlap q, k, v, g or o.
 *   o          bf16 [N, H, 128] output.
 *   N, H       N >= 0 (0 is a no-op), H >= 1.
 * Errors: SALA_ERR_INVALID_ARG, SALA_ERR_MISALIGNED, SALA_ERR_UNSUPPORTED, SALA_ERR_CUDA.
 */
int sala_gla_recurrent_step(const void *q, const void *k, const void *v, const float *g,
                            float scale, float *S_inout, void *o, int64_t N, int32_t H,
                            void *stream);

/*
 * One-token recurrent decode on states kept in a pool and addressed through an index array.
 *
 * A serving engine keeps each request's recurrent state in a slot of a per-layer pool and
 * hands the layer the slot of every request in the batch ("MiniCPM-SALA — Complete
 * Blueprint", "Memory Architecture": MambaPool temporal states, one per request and layer,
 * 1 MB each in bf16 for 32 heads; the decode step loads the state from the pool, updates it
 * and saves it back in place). For each sequence n of the batch and head h, with
 * i = state_indices[n]:
 *     S = state_pool[i, h];  S = exp(g[n,h]) S + k[n,h]^T v[n,h];  o[n,h] = scale q[n,h] S;
 *     state_pool[i, h] = S
 * A negative index marks a padding row: its o is written as zeros and no state is touched.
 *
 *   q, k, v        bf16 [N, H, 128];  g fp32 [N, H]
 *   state_pool     [P, H, 128, 128] of state_dtype (SALA_STATE_F32: fp32; SALA_STATE_BF16:
 *                  bf16, widened to fp32 for the arithmetic and rounded to nearest even when
 *                  stored). Only the N addressed slots are read and written.
 *   state_indices  int32 [N] DEVICE array of slots (< P), or negative for padding. Two rows
 *                  with the same slot race (the result is one of them); the caller must not
 *                  do that. A slot >= P is recorded as SALA_ERR_BAD_INDEX in the device
 *                  status word and its row is treated as padding.
 *   o              bf16 [N, H, 128] output.
 *   P, N, H        P >= 1, N >= 0 (0 is a no-op), H >= 1.
 *   prologue       NULL: q and k are used as given. Otherwise q and k are the raw
 *                  projections and the step first applies the q/k prologue (RMSNorm, RoPE;
 *                  see sala_qk_prologue) to them, fused into the same kernel; q and k
 *                  themselves are not modified.
 *   positions      int64 [N] DEVICE array, the position of each row's token in its sequence
 *                  (required with a prologue, ignored without).
 * Errors: SALA_ERR_INVALID_ARG (also for an unknown state_dtype or a pool that overlaps
 * another argument), SALA_ERR_MISALIGNED, SALA_ERR_UNSUPPORTED, SALA_ERR_CUDA.
 */
int sala_gla_recurrent_step_indexed(const void *q, const void *k, const void *v, const float *g,
                                    float scale, void *state_pool, int32_t state_dtype,
                                    const int32_t *state_indices, int64_t P, void *o, int64_t N,
                                    int32_t H, const sala_qk_prologue *prologue,
                                    const int64_t *positions, void *stream);

/*
 * The q/k prologue (see sala_qk_prologue) in place on the q and k of a prefill, before
 * sala_gla_chunk_fwd. A separate pass: the chunked prefill loads its q and k tiles straight
 * into shared memory by TMA, and the per-element work of the prologue on its critical path
 * costs more than this pass's read and write of q and k.
 *
 *   q, k         bf16 [B, T, H, 128] (packed [T, H, 128] with cu_seqlens), rewritten in place.
 *   cu_seqlens   int64 [num_seqs + 1] DEVICE array as for sala_gla_chunk_fwd, or NULL (B rows
 *                of T tokens). It must be valid (non-decreasing, from 0 to T); this call does
 *                not check it on the device (the debug build does: SALA_ERR_DEBUG_CHECK, and
 *                tokens it cannot place in a sequence are left as they are).
 *   start_pos    int64 [Nseq] DEVICE array, the position of each sequence's first token here
 *                (a continued sequence), or NULL for 0. A token's position is start_pos[n]
 *                plus its index in sequence n.
 * Errors: SALA_ERR_INVALID_ARG, SALA_ERR_MISALIGNED, SALA_ERR_UNSUPPORTED, SALA_ERR_CUDA.
 */
int sala_gla_qk_prologue(void *q, void *k, const sala_qk_prologue *prologue,
                         const int64_t *cu_seqlens, const int64_t *start_pos, int64_t B,
                         int64_t T, int32_t H, int64_t num_seqs, void *stream);

/*
 * Output norm and gate of a lightning layer, per token:
 *     out[t] = RMSNorm(o[t]) * w * sigmoid(z[t]),   RMSNorm(x) = x / sqrt(mean(x^2) + eps)
 * over the F = H * 128 features of the token (all heads together), fp32 arithmetic.
 * "MiniCPM-SALA — Complete Blueprint", section "B2 lightning-attn (Simple GLA)", block
 * "Output Norm + Gate + Projection" (o_norm with a 4096-wide weight, then the z_proj gate
 * sigmoid(h W_z^T)); RMSNorm as the page's input_layernorm block defines it (eps = 1e-6). The
 * gate logits z = h W_z^T are computed by the caller.
 *
 *   o     bf16 [T, H * 128] attention output (e.g. the o of sala_gla_chunk_fwd, [T, H, 128])
 *   z     bf16 [T, H * 128] gate logits (before the sigmoid)
 *   w     bf16 [H * 128] norm weight
 *   eps   >= 0, typically 1e-6
 *   out   bf16 [T, H * 128] (round to nearest even); may be o itself (in place), must not
 *         overlap z, w or part of o.
 *   T, H  T >= 0 (0 is a no-op), 1 <= H <= 4096.
 * Errors: SALA_ERR_INVALID_ARG, SALA_ERR_MISALIGNED, SALA_ERR_UNSUPPORTED, SALA_ERR_CUDA.
 */
int sala_gla_output_norm_gate(const void *o, const void *z, const void *w, float eps, void *out,
                              int64_t T, int32_t H, void *stream);

/*
 * One-token recurrent step of the gated delta rule (GDN), the second linear-attention
 * workload of "Formulas and Code for Adapting Inference to GDN/KDA Linear Modules", section
 * 1.1. For each of the N sequences and H heads, with the [128 x 128] fp32 state S (row = key
 * dimension):
 *     S = exp(g) S;   v_new = beta (v - k S);   S = S + k^T v_new;   o = scale q S
 * (the decay precedes the memory read, as the page's chunked form computes; k S is the
 * vector over the value dimension read at key k). Normalising q and k (the page's l2norm)
 * and forming g and beta happen before the call.
 *
 *   q, k, v    bf16 [N, H, 128]
 *   g          fp32 [N, H] log-decay;  beta fp32 [N, H] write strength (typically in (0, 1))
 *   S_inout    fp32 [N, H, 128, 128], read and overwritten. Must not overlap the inputs or o.
 *   o          bf16 [N, H, 128] output.
 *   N, H       N >= 0 (0 is a no-op), H >= 1.
 * Errors: SALA_ERR_INVALID_ARG, SALA_ERR_MISALIGNED, SALA_ERR_UNSUPPORTED, SALA_ERR_CUDA.
 */
int sala_gla_gdn_recurrent_step(const void *q, const void *k, const void *v, const float *g,
                                const float *beta, float scale, float *S_inout, void *o,
                                int64_t N, int32_t H, void *stream);

/*
 * The gated delta rule over whole sequences in its recurrent form (the page's prefill for
 * short sequences: "Formulas and Code for Adapting Inference to GDN/KDA Linear Modules",
 * section 1): for each sequence and head, token by token from h0, the update of
 * sala_gla_gdn_recurrent_step. One CTA per (sequence, head) keeps the state in registers, so
 * the work is parallel over sequences and heads only (a long single sequence runs on H SMs).
 *
 *   q, k, v    bf16 [B, T, H, 128] (packed [T, H, 128] with cu_seqlens, B = 1)
 *   g, beta    fp32 [B, T, H]
 *   h0         fp32 [Nseq, H, 128, 128] or NULL (zeros); hT fp32 [Nseq, H, 128, 128] or NULL
 *   cu_seqlens int64 [num_seqs + 1] DEVICE array (0 = cu[0] <= ... <= cu[num_seqs] = T), or NULL
 *   o          bf16 [B, T, H, 128]
 * cu_seqlens is not validated here beyond keeping every sequence inside [0, T) (a malformed
 * one gives meaningless results for the affected sequences, never an access outside the
 * tensors); sala_gla_chunk_fwd reports a malformed one.
 * Errors: SALA_ERR_INVALID_ARG, SALA_ERR_MISALIGNED, SALA_ERR_UNSUPPORTED, SALA_ERR_CUDA.
 */
int sala_gla_gdn_fwd(const void *q, const void *k, const void *v, const float *g,
                     const float *beta, float scale, const float *h0, const int64_t *cu_seqlens,
                     void *o, float *hT, int64_t B, int64_t T, int32_t H, int64_t num_seqs,
                     void *stream);

/*
 * The gated delta rule over whole sequences in its chunked form ("Formulas and Code for
 * Adapting Inference to GDN/KDA Linear Modules", section 1.2, formulas 11-17; chunk size 64):
 * the same results as sala_gla_gdn_fwd (decay first, then the delta-rule write and the read),
 * computed chunk by chunk on the tensor cores. Per chunk the UT transform
 * T = (I + tril(diag(beta) K K^T * Gamma, -1))^-1 gives W = T (diag(beta) K * exp(b)) and
 * U = T diag(beta) V, and the state-dependent values new_v = U - W S; the output and the state
 * refresh are then the Simple GLA chunk products with new_v in place of v, which this call
 * computes with the chunked prefill of sala_gla_chunk_fwd (its segment-parallel state pass and
 * hand-off included). The new_v pass runs one CTA per (sequence, head), so it is parallel over
 * sequences and heads; the prefill that follows is parallel over segments as well.
 *
 * Arguments, layouts and errors as sala_gla_gdn_fwd; in addition T (B * T) must stay below
 * 2^31 - 64 tokens. Scratch: the bf16 new_v [B * T, H, 128] and the prefill's scratch, from the
 * library's stream-ordered pool (as sala_gla_chunk_fwd). A malformed cu_seqlens is reported as
 * by sala_gla_chunk_fwd (SALA_ERR_BAD_SEQLENS; nothing written).
 */
int sala_gla_gdn_chunk_fwd(const void *q, const void *k, const void *v, const float *g,
                           const float *beta, float scale, const float *h0,
                           const int64_t *cu_seqlens, void *o, float *hT, int64_t B, int64_t T,
                           int32_t H, int64_t num_seqs, void *stream);

/*
 * Chunked prefill that allocates nothing: same arguments, layouts, results and errors as
 * sala_gla_chunk_fwd, plus SALA_ERR_TOO_LARGE. The pages have no counterpart to this entry
 * point; it exists for callers that cannot allocate device memory while they run the layer:
 * serving engines that reserve nearly all of HBM for their own pools at start-up (so any
 * further allocation fails), plug-in hosts whose execute path forbids allocation, and
 * latency-critical loops that cannot afford an allocator call, which may synchronise.
 *
 * Its scratch (segment table, per-segment hand-off states and flags) lives in one fixed device
 * array of SALA_NOALLOC_SCRATCH_BYTES (64 MiB) inside the library. Every GPU that loads
 * the library holds that array until the process exits. The call picks segments long
 * enough for the scratch to fit; when even one segment per sequence does not fit (roughly
 * num_seqs * H > 1000) it returns SALA_ERR_TOO_LARGE before queuing any work.
 *
 * The first call on a device looks up the array's device address (and sets kernel
 * attributes) with that device current; make that first call before any stream capture.
 * All calls share the one array and it keeps the last call's contents (every call fully
 * rewrites what it reads, so no clearing is needed between calls). Calls whose work
 * overlaps on the GPU (different streams, or different host threads) race on the array:
 * serialise them on one stream. The call performs no cudaMalloc/cudaFree or other
 * allocation.
 */
#define SALA_NOALLOC_SCRATCH_BYTES (64ull << 20)
int sala_gla_chunk_fwd_noalloc(const void *q, const void *k, const void *v, const float *g,
                               float scale, const float *h0, const int64_t *cu_seqlens, void *o,
                               float *hT, int64_t B, int64_t T, int32_t H, int64_t num_seqs,
                               void *stream);

/*
 * Failure-path test settings of the chunked prefill (process-wide; for tests and diagnosis,
 * not for production use). The prefill hands the state of each (segment, head) unit to the
 * next segment through a flag that the successor waits for, and every such wait is bounded
 * (2 s by default). With these settings a test can make one wait give up on purpose and check
 * that the call still returns, that SALA_ERR_TIMEOUT is recorded in the device status word,
 * and that the next call computes correct results (the aborted kernel released its tensor
 * memory and drained its copies).
 *
 *   flag_wait_ns   limit of the wait for a predecessor's state, in nanoseconds (0: 2 s).
 *   withhold_unit  index of a unit (segment * H + head in the segment table's numbering)
 *                  whose state is computed but whose flag later calls never raise, so that
 *                  the unit after it waits in vain; -1: none. Units past a call's last unit
 *                  are ignored.
 * Affects every later sala_gla_chunk_fwd / sala_gla_chunk_fwd_noalloc call until reset with
 * (0, -1). Errors: SALA_ERR_INVALID_ARG (withhold_unit < -1).
 */
int sala_gla_debug_prefill_knobs(uint64_t flag_wait_ns, int64_t withhold_unit);

/*
 * Which kernel sala_gla_chunk_fwd runs for the chunked prefill; both compute the same result
 * (the recurrence of "MiniCPM-SALA — Complete Blueprint", "Simple GLA Recurrence", in the
 * chunked form of "Formulas and Code for Adapting Inference to GDN/KDA Linear Modules",
 * section 1.2) and differ in how a GB300 runs it:
 *   0  chosen per call (the default): kernel 2 when the call holds more than 8192 token-heads
 *      per SM (many waves of units), else kernel 1;
 *   1  one unit (segment, head) per SM at a time, its steps split over fifteen warps;
 *   2  two CTAs per SM, one unit each, in half of the SM's shared and tensor memory.
 * The environment variable SALA_GLA_PREFILL ("fused" for 1, "pair" for 2) sets the initial
 * choice. Process-wide; affects every later sala_gla_chunk_fwd call (sala_gla_chunk_fwd_noalloc
 * always runs kernel 1). Errors: SALA_ERR_INVALID_ARG (any other value).
 */
int sala_gla_set_prefill_kernel(int kernel);

/* Static English description of a sala_status value (never NULL). */
const char *sala_gla_status_string(int status);

/*
 * Synchronises `stream`, then returns and clears the device-side status word of the current
 * device (SALA_OK if no kernel recorded an error since the last call). Returns SALA_ERR_CUDA
 * if the synchronisation itself fails.
 */
int sala_gla_get_device_status(void *stream);

/* Library version, "major.minor.patch". */
const char *sala_gla_version(void);

/*
 * Kernel timing instrumentation (off by default; process-wide).
 *
 * While enabled, every kernel the library launches is bracketed by a pair of CUDA events
 * recorded on the launching stream, so per-kernel device time is measured in place, inside
 * the caller's own timed region. The kernels are identified by an index in
 * [0, sala_gla_kernel_count()); sala_gla_kernel_name() names them.
 *
 * sala_gla_timing_enable(1) clears earlier records and starts recording; (0) stops.
 * sala_gla_timing_read() waits for the recorded events, then stores the summed device time
 * in milliseconds and the number of launches of kernel `kernel` since the last enable.
 * Returns SALA_ERR_INVALID_ARG for an unknown index or null outputs, SALA_ERR_CUDA if an
 * event query fails.
 */
int sala_gla_timing_enable(int enable);
int sala_gla_timing_read(int kernel, double *total_ms, int64_t *launches);
int sala_gla_kernel_count(void);
const char *sala_gla_kernel_name(int kernel);

#ifdef __cplusplus
}
#endif

#endif /* SALA_GLA_H */
