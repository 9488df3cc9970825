"""ctypes binding of ``libsala_gla.so`` (argument marshalling only).

Every function here checks shapes and dtypes, allocates outputs with torch when the caller
did not pass them, and calls the C entry point of the same name on the current CUDA stream.
All arithmetic runs in the library's kernels. If the library has not been built, importing
this module raises: there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

_lib = None

SALA_OK = 0
STATUS_NAMES = {
    0: "SALA_OK", 1: "SALA_ERR_INVALID_ARG", 2: "SALA_ERR_MISALIGNED",
    3: "SALA_ERR_UNSUPPORTED", 4: "SALA_ERR_CUDA", 5: "SALA_ERR_TIMEOUT",
    6: "SALA_ERR_BAD_SEQLENS", 7: "SALA_ERR_TOO_LARGE", 8: "SALA_ERR_BAD_INDEX",
    9: "SALA_ERR_DEBUG_CHECK",
}
SALA_STATE_F32, SALA_STATE_BF16 = 0, 1

class QkPrologue(ctypes.Structure):
    """``sala_qk_prologue``: RMSNorm weights of q and k (bf16 [128] device pointers), eps,
    RoPE theta."""
    _fields_ = [("q_weight", ctypes.c_void_p), ("k_weight", ctypes.c_void_p),
                ("eps", ctypes.c_float), ("rope_theta", ctypes.c_float)]


# exported symbols and their ctypes signatures (must match include/sala_gla.h)
_p, _i64, _i32, _f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float
_pro = ctypes.POINTER(QkPrologue)
SIGNATURES = {
    "sala_gla_chunk_fwd": ([_p, _p, _p, _p, _f32, _p, _p, _p, _p, _i64, _i64, _i32, _i64, _p],
                           ctypes.c_int),
    "sala_gla_recurrent_step": ([_p, _p, _p, _p, _f32, _p, _p, _i64, _i32, _p], ctypes.c_int),
    "sala_gla_recurrent_step_indexed": ([_p, _p, _p, _p, _f32, _p, _i32, _p, _i64, _p, _i64, _i32,
                                         _pro, _p, _p], ctypes.c_int),
    "sala_gla_gdn_recurrent_step": ([_p, _p, _p, _p, _p, _f32, _p, _p, _i64, _i32, _p], ctypes.c_int),
    "sala_gla_gdn_fwd": ([_p, _p, _p, _p, _p, _f32, _p, _p, _p, _p, _i64, _i64, _i32, _i64, _p],
                         ctypes.c_int),
    "sala_gla_gdn_chunk_fwd": ([_p, _p, _p, _p, _p, _f32, _p, _p, _p, _p, _i64, _i64, _i32, _i64,
                                _p], ctypes.c_int),
    "sala_gla_qk_prologue": ([_p, _p, _pro, _p, _p, _i64, _i64, _i32, _i64, _p], ctypes.c_int),
    "sala_gla_output_norm_gate": ([_p, _p, _p, _f32, _p, _i64, _i32, _p], ctypes.c_int),
    "sala_gla_chunk_fwd_noalloc": ([_p, _p, _p, _p, _f32, _p, _p, _p, _p, _i64, _i64, _i32,
                                    _i64, _p], ctypes.c_int),
    "sala_gla_status_string": ([ctypes.c_int], ctypes.c_char_p),
    "sala_gla_get_device_status": ([_p], ctypes.c_int),
    "sala_gla_version": ([], ctypes.c_char_p),
    "sala_gla_timing_enable": ([ctypes.c_int], ctypes.c_int),
    "sala_gla_timing_read": ([ctypes.c_int, ctypes.POINTER(ctypes.c_double),
                              ctypes.POINTER(ctypes.c_int64)], ctypes.c_int),
    "sala_gla_kernel_count": ([], ctypes.c_int),
    "sala_gla_kernel_name": ([ctypes.c_int], ctypes.c_char_p),
    "sala_gla_debug_prefill_knobs": ([ctypes.c_uint64, _i64], ctypes.c_int),
    "sala_gla_set_prefill_kernel": ([_i32], ctypes.c_int),
}


class SalaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)} ({status_string(status)})")


def library_path() -> str:
    """The library the binding loads: the debug build when SALA_GLA_DEBUG=1, else the release
    build."""
    return _build.LIB_DEBUG if os.environ.get("SALA_GLA_DEBUG") == "1" else _build.LIB


def load(path: str | None = None):
    """Load the compiled library (raises OSError if it is missing); ``path`` loads another
    build without making it the binding's library."""
    global _lib
    if _lib is None or path is not None:
        p = path or library_path()
        if not os.path.exists(p):
            raise OSError(f"{p} not found: build it with gated_linear_attention_gb300.build.build()"
                          f"{'(debug=True)' if p == _build.LIB_DEBUG else ''}")
        lib = ctypes.CDLL(p)
        for name, (argtypes, restype) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.argtypes = argtypes
            fn.restype = restype
        if path is not None:
            return lib
        _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load().sala_gla_status_string(int(status)).decode()


def version() -> str:
    return load().sala_gla_version().decode()


def _ptr(t):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(rc: int, what: str):
    if rc != SALA_OK:
        raise SalaError(rc, what)


def _need(t, name, dtype, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def chunk_fwd(q, k, v, g, scale, h0=None, cu_seqlens=None, output_final_state=True, o=None,
              hT=None, stream=None, noalloc=False):
    """Chunked prefill, ``sala_gla_chunk_fwd`` (``sala_gla_chunk_fwd_noalloc`` when
    ``noalloc``: scratch from the library's fixed 64 MiB device array instead of a pool).

    q, k, v: bf16 [B, T, H, 128] (or [1, T, H, 128] / [T, H, 128] packed with cu_seqlens);
    g: fp32 [B, T, H] (or [T, H]); h0: fp32 [Nseq, H, 128, 128] or None; cu_seqlens: int64
    CUDA tensor [Nseq + 1] or None. Returns (o, hT); hT is None unless output_final_state.
    """
    packed = q.dim() == 3
    if packed:
        if cu_seqlens is None:
            raise ValueError("packed [T, H, 128] input needs cu_seqlens")
        T, H, D = q.shape
        B = 1
    else:
        B, T, H, D = q.shape
    if D != 128:
        raise ValueError("head dimension must be 128")
    _need(q, "q", torch.bfloat16)
    _need(k, "k", torch.bfloat16, q.shape)
    _need(v, "v", torch.bfloat16, q.shape)
    _need(g, "g", torch.float32, q.shape[:-1])
    nseq = B
    if cu_seqlens is not None:
        _need(cu_seqlens, "cu_seqlens", torch.int64)
        if B != 1:
            raise ValueError("cu_seqlens needs B == 1")
        nseq = cu_seqlens.numel() - 1
        if nseq < 1:
            raise ValueError("cu_seqlens needs at least two entries")
    if h0 is not None:
        _need(h0, "h0", torch.float32, (nseq, H, 128, 128))
    if o is None:
        o = torch.empty_like(q)
    else:
        _need(o, "o", torch.bfloat16, q.shape)
    if output_final_state and hT is None:
        hT = torch.empty((nseq, H, 128, 128), dtype=torch.float32, device=q.device)
    elif hT is not None:
        _need(hT, "hT", torch.float32, (nseq, H, 128, 128))
    lib = load()
    fn = lib.sala_gla_chunk_fwd_noalloc if noalloc else lib.sala_gla_chunk_fwd
    rc = fn(_ptr(q), _ptr(k), _ptr(v), _ptr(g), float(scale), _ptr(h0), _ptr(cu_seqlens), _ptr(o),
            _ptr(hT), B, T, H, nseq if cu_seqlens is not None else 0, _stream(stream))
    _check(rc, "sala_gla_chunk_fwd_noalloc" if noalloc else "sala_gla_chunk_fwd")
    return o, hT


def recurrent_step(q, k, v, g, scale, S, o=None, stream=None):
    """One decode step, ``sala_gla_recurrent_step``; S [N, H, 128, 128] fp32 is updated in
    place. q, k, v: bf16 [N, H, 128]; g: fp32 [N, H]. Returns o (bf16 [N, H, 128])."""
    N, H, D = q.shape
    if D != 128:
        raise ValueError("head dimension must be 128")
    _need(q, "q", torch.bfloat16)
    _need(k, "k", torch.bfloat16, q.shape)
    _need(v, "v", torch.bfloat16, q.shape)
    _need(g, "g", torch.float32, (N, H))
    _need(S, "S", torch.float32, (N, H, 128, 128))
    if o is None:
        o = torch.empty_like(q)
    else:
        _need(o, "o", torch.bfloat16, q.shape)
    rc = load().sala_gla_recurrent_step(_ptr(q), _ptr(k), _ptr(v), _ptr(g), float(scale),
                                        _ptr(S), _ptr(o), N, H, _stream(stream))
    _check(rc, "sala_gla_recurrent_step")
    return o


def _prologue(q_weight, k_weight, eps, rope_theta):
    _need(q_weight, "q_weight", torch.bfloat16, (128,))
    _need(k_weight, "k_weight", torch.bfloat16, (128,))
    return QkPrologue(_ptr(q_weight), _ptr(k_weight), float(eps), float(rope_theta))


def recurrent_step_indexed(q, k, v, g, scale, pool, indices, o=None, stream=None, prologue=None,
                           positions=None):
    """One decode step on pooled states, ``sala_gla_recurrent_step_indexed``: row n uses (and
    updates in place) ``pool[indices[n]]``; a negative index is a padding row (o = 0).
    q, k, v: bf16 [N, H, 128]; g: fp32 [N, H]; pool: fp32 or bf16 [P, H, 128, 128] (its dtype
    is the storage type); indices: int32 [N]. ``prologue=(q_weight, k_weight, eps, theta)``
    applies the q/k RMSNorm and RoPE to the raw q, k in the kernel, with ``positions`` int64
    [N]. Returns o (bf16 [N, H, 128])."""
    N, H, D = q.shape
    if D != 128:
        raise ValueError("head dimension must be 128")
    _need(q, "q", torch.bfloat16)
    _need(k, "k", torch.bfloat16, q.shape)
    _need(v, "v", torch.bfloat16, q.shape)
    _need(g, "g", torch.float32, (N, H))
    if pool.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError(f"pool must be float32 or bfloat16, got {pool.dtype}")
    _need(pool, "pool", pool.dtype)
    if pool.dim() != 4 or tuple(pool.shape[1:]) != (H, 128, 128):
        raise ValueError(f"pool has shape {tuple(pool.shape)}, expected (P, {H}, 128, 128)")
    _need(indices, "indices", torch.int32, (N,))
    if o is None:
        o = torch.empty_like(q)
    else:
        _need(o, "o", torch.bfloat16, q.shape)
    dt = SALA_STATE_BF16 if pool.dtype == torch.bfloat16 else SALA_STATE_F32
    pro = None
    if prologue is not None:
        pro = ctypes.byref(_prologue(*prologue))
        _need(positions, "positions", torch.int64, (N,))
    rc = load().sala_gla_recurrent_step_indexed(_ptr(q), _ptr(k), _ptr(v), _ptr(g), float(scale),
                                                _ptr(pool), dt, _ptr(indices), pool.shape[0],
                                                _ptr(o), N, H, pro,
                                                _ptr(positions) if prologue is not None else None,
                                                _stream(stream))
    _check(rc, "sala_gla_recurrent_step_indexed")
    return o


def qk_prologue(q, k, q_weight, k_weight, eps=1e-6, rope_theta=10000.0, cu_seqlens=None,
                start_pos=None, stream=None):
    """``sala_gla_qk_prologue``: the q/k RMSNorm and RoPE, in place on a prefill's q and k
    (bf16 [B, T, H, 128], or packed [T, H, 128] with ``cu_seqlens``). ``start_pos`` int64
    [Nseq]: position of each sequence's first token (default 0)."""
    if q.dim() == 4:
        Bn, T, H, D = q.shape
        nseq = Bn
    elif q.dim() == 3:
        if cu_seqlens is None:
            raise ValueError("packed q needs cu_seqlens")
        Bn, (T, H, D) = 1, q.shape
        nseq = cu_seqlens.numel() - 1
    else:
        raise ValueError("q must be [B, T, H, 128] or [T, H, 128]")
    if D != 128:
        raise ValueError("head dimension must be 128")
    _need(q, "q", torch.bfloat16)
    _need(k, "k", torch.bfloat16, q.shape)
    if cu_seqlens is not None:
        _need(cu_seqlens, "cu_seqlens", torch.int64, (nseq + 1,))
    if start_pos is not None:
        _need(start_pos, "start_pos", torch.int64, (nseq,))
    pro = _prologue(q_weight, k_weight, eps, rope_theta)
    rc = load().sala_gla_qk_prologue(_ptr(q), _ptr(k), ctypes.byref(pro),
                                     _ptr(cu_seqlens) if cu_seqlens is not None else None,
                                     _ptr(start_pos) if start_pos is not None else None,
                                     Bn, T, H, nseq if cu_seqlens is not None else 0,
                                     _stream(stream))
    _check(rc, "sala_gla_qk_prologue")
    return q, k


def output_norm_gate(o, z, w, eps=1e-6, out=None, stream=None):
    """``sala_gla_output_norm_gate``: out = RMSNorm(o) * w * sigmoid(z) per token over its
    H * 128 features. o, z: bf16 [T, H, 128] or [T, H * 128]; w: bf16 [H * 128]. ``out=o``
    works in place. Returns out (the shape of o)."""
    if o.dim() not in (2, 3) or o.shape[-1] % 128 or (o.dim() == 3 and o.shape[-1] != 128):
        raise ValueError("o must be [T, H, 128] or [T, H * 128]")
    T = o.shape[0]
    F = o.shape[1] * o.shape[2] if o.dim() == 3 else o.shape[1]
    H = F // 128
    _need(o, "o", torch.bfloat16)
    _need(z, "z", torch.bfloat16, o.shape)
    _need(w, "w", torch.bfloat16, (F,))
    if out is None:
        out = torch.empty_like(o)
    else:
        _need(out, "out", torch.bfloat16, o.shape)
    rc = load().sala_gla_output_norm_gate(_ptr(o), _ptr(z), _ptr(w), float(eps), _ptr(out), T, H,
                                          _stream(stream))
    _check(rc, "sala_gla_output_norm_gate")
    return out


def gdn_fwd(q, k, v, g, beta, scale, h0=None, cu_seqlens=None, output_final_state=True,
            o=None, hT=None, stream=None, chunked=False):
    """``sala_gla_gdn_fwd`` (recurrent form) or, with ``chunked=True``,
    ``sala_gla_gdn_chunk_fwd`` (chunked form on the tensor cores): the gated delta rule over
    whole sequences. q, k, v: bf16 [B, T, H, 128] or packed [T, H, 128] with ``cu_seqlens``;
    g, beta: fp32 [B, T, H] / [T, H]. Returns (o, hT or None)."""
    if q.dim() == 4:
        Bn, T, H, D = q.shape
        nseq, packed = Bn, False
    elif q.dim() == 3 and cu_seqlens is not None:
        (T, H, D), Bn = q.shape, 1
        nseq, packed = cu_seqlens.numel() - 1, True
    else:
        raise ValueError("q must be [B, T, H, 128], or [T, H, 128] with cu_seqlens")
    if D != 128:
        raise ValueError("head dimension must be 128")
    _need(q, "q", torch.bfloat16)
    _need(k, "k", torch.bfloat16, q.shape)
    _need(v, "v", torch.bfloat16, q.shape)
    _need(g, "g", torch.float32, q.shape[:-1])
    _need(beta, "beta", torch.float32, q.shape[:-1])
    if h0 is not None:
        _need(h0, "h0", torch.float32, (nseq, H, 128, 128))
    if packed:
        _need(cu_seqlens, "cu_seqlens", torch.int64, (nseq + 1,))
    if o is None:
        o = torch.empty_like(q)
    if output_final_state and hT is None:
        hT = torch.empty((nseq, H, 128, 128), dtype=torch.float32, device=q.device)
    if not output_final_state:
        hT = None
    name = "sala_gla_gdn_chunk_fwd" if chunked else "sala_gla_gdn_fwd"
    rc = getattr(load(), name)(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale),
                               _ptr(h0), _ptr(cu_seqlens) if packed else None, _ptr(o), _ptr(hT),
                               Bn, T, H, nseq if packed else 0, _stream(stream))
    _check(rc, name)
    return o, hT


def gdn_recurrent_step(q, k, v, g, beta, scale, S, o=None, stream=None):
    """One gated-delta-rule step, ``sala_gla_gdn_recurrent_step``; S [N, H, 128, 128] fp32 is
    updated in place. q, k, v: bf16 [N, H, 128]; g, beta: fp32 [N, H]. Returns o."""
    N, H, D = q.shape
    if D != 128:
        raise ValueError("head dimension must be 128")
    _need(q, "q", torch.bfloat16)
    _need(k, "k", torch.bfloat16, q.shape)
    _need(v, "v", torch.bfloat16, q.shape)
    _need(g, "g", torch.float32, (N, H))
    _need(beta, "beta", torch.float32, (N, H))
    _need(S, "S", torch.float32, (N, H, 128, 128))
    if o is None:
        o = torch.empty_like(q)
    else:
        _need(o, "o", torch.bfloat16, q.shape)
    rc = load().sala_gla_gdn_recurrent_step(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                            float(scale), _ptr(S), _ptr(o), N, H, _stream(stream))
    _check(rc, "sala_gla_gdn_recurrent_step")
    return o


def get_device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device-side status word."""
    return int(load().sala_gla_get_device_status(_stream(stream)))


def timing_enable(enable: bool = True) -> None:
    """Start (clearing old records) or stop the per-kernel event timing."""
    _check(load().sala_gla_timing_enable(1 if enable else 0), "sala_gla_timing_enable")


def timing_read() -> dict:
    """{kernel name: (total device ms, launches)} since the last timing_enable(True)."""
    lib = load()
    out = {}
    for i in range(lib.sala_gla_kernel_count()):
        ms, n = ctypes.c_double(), ctypes.c_int64()
        _check(lib.sala_gla_timing_read(i, ctypes.byref(ms), ctypes.byref(n)),
               "sala_gla_timing_read")
        out[lib.sala_gla_kernel_name(i).decode()] = (ms.value, n.value)
    return out


def set_prefill_kernel(kernel: int) -> None:
    """Which chunked-prefill kernel ``chunk_fwd`` runs (``sala_gla_set_prefill_kernel``): 0 chosen
    per call, 1 one unit per SM, 2 two CTAs per SM."""
    _check(load().sala_gla_set_prefill_kernel(int(kernel)), "sala_gla_set_prefill_kernel")


def debug_prefill_knobs(flag_wait_ns: int = 0, withhold_unit: int = -1) -> None:
    """Failure-path test settings of the prefill (``sala_gla_debug_prefill_knobs``): the limit of
    the wait for a predecessor's state (0: the default) and a unit whose hand-off flag is never
    raised (-1: none). ``debug_prefill_knobs()`` restores the defaults."""
    _check(load().sala_gla_debug_prefill_knobs(int(flag_wait_ns), int(withhold_unit)),
           "sala_gla_debug_prefill_knobs")
