"""Simple GLA (Lightning attention) hot path for GB300 (sm_103a).

Chunked prefill and one-token recurrent decode of the per-head scalar-decay recurrence
S_t = exp(g_t) S_{t-1} + k_t^T v_t, o_t = scale q_t S_t (head dim 128, fp32 state), as
hand-written CUDA kernels behind a C ABI (``include/sala_gla.h``). This package holds the
build step, the ctypes binding and the seeded synthetic inputs.

The binding is loaded on first use of :mod:`gated_linear_attention_gb300.sala_gla`; it raises
if the compiled library is missing. There is no CPU fallback.
"""

__version__ = "0.1.0"
