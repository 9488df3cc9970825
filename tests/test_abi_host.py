"""Host-side checks of the C ABI (no GPU needed): the library builds, loads, exports every
symbol that include/sala_gla.h declares, and rejects bad arguments before touching CUDA."""
import ctypes
import os
import re

import pytest
import torch

from gated_linear_attention_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))
           if f.endswith(".h")]

no_gpu = pytest.mark.skipif(torch.cuda.is_available(),
                            reason="fake pointers must never reach a real device")


@pytest.fixture(scope="module")
def lib():
    path = B.build()
    from gated_linear_attention_gb300 import sala_gla
    return sala_gla.load()


def declared_functions():
    names = []
    for h in HEADERS:
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(sala_gla_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("sala_gla_chunk_fwd", "sala_gla_recurrent_step", "sala_gla_status_string",
              "sala_gla_get_device_status", "sala_gla_version"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_debug_build_exports_every_declared_symbol():
    # the SALA_GLA_DEBUG build: same ABI, device-side index checks compiled in
    path = B.build(debug=True)
    assert path == B.LIB_DEBUG and path != B.LIB
    from gated_linear_attention_gb300 import sala_gla
    dlib = sala_gla.load(path)
    for name in declared_functions():
        assert hasattr(dlib, name), name
    assert dlib.sala_gla_status_string(9).decode().startswith("debug build")
    assert sala_gla.STATUS_NAMES[9] == "SALA_ERR_DEBUG_CHECK"


def test_debug_library_is_selected_by_environment(monkeypatch):
    from gated_linear_attention_gb300 import sala_gla
    monkeypatch.setenv("SALA_GLA_DEBUG", "1")
    assert sala_gla.library_path() == B.LIB_DEBUG
    monkeypatch.delenv("SALA_GLA_DEBUG")
    assert sala_gla.library_path() == B.LIB


def test_binding_covers_every_declared_symbol():
    from gated_linear_attention_gb300 import sala_gla
    assert sorted(sala_gla.SIGNATURES) == declared_functions()


def test_library_is_sm103a_only_and_links_cudart_statically(lib):
    with open(B.LIB, "rb") as f:
        blob = f.read()
    # a statically linked runtime: no dynamic dependency on libcudart
    import subprocess
    out = subprocess.run(["ldd", B.LIB], capture_output=True, text=True).stdout
    assert "libcudart" not in out
    assert b"sm_103a" in blob or b"sm_103" in blob


def test_status_strings(lib):
    from gated_linear_attention_gb300 import sala_gla
    assert sala_gla.status_string(0) == "success"
    for s in range(1, 9):
        assert sala_gla.status_string(s) not in ("", "unknown status")
    assert sala_gla.status_string(99) == "unknown status"
    assert sala_gla.version().count(".") == 2


P = ctypes.c_void_p


def _chunk(lib, q=0x10000, k=0x20000, v=0x30000, g=0x40000, h0=None, cu=None, o=0x50000,
           hT=0x60000, Bn=1, T=64, H=2, nseq=0):
    return lib.sala_gla_chunk_fwd(P(q), P(k), P(v), P(g), 0.1, P(h0) if h0 else None,
                                  P(cu) if cu else None, P(o), P(hT) if hT else None,
                                  Bn, T, H, nseq, None)


def _step(lib, q=0x10000, k=0x20000, v=0x30000, g=0x40000, S=0x100000, o=0x50000, N=2, H=2):
    return lib.sala_gla_recurrent_step(P(q), P(k), P(v), P(g), 0.1, P(S), P(o), N, H, None)


@no_gpu
def test_chunk_fwd_argument_errors(lib):
    INVALID, MISALIGNED = 1, 2
    # sizes far apart so that only the intended overlap exists: T*H*128*2 = 32 KB per tensor
    assert _chunk(lib, Bn=0) == INVALID
    assert _chunk(lib, T=-1) == INVALID
    assert _chunk(lib, H=0) == INVALID
    assert _chunk(lib, q=0) == INVALID
    assert _chunk(lib, o=0) == INVALID
    assert _chunk(lib, cu=0x70000, nseq=0) == INVALID         # cu_seqlens needs num_seqs >= 1
    assert _chunk(lib, cu=0x70000, nseq=2, Bn=2) == INVALID   # and B == 1
    assert _chunk(lib, q=0x10008) == MISALIGNED
    assert _chunk(lib, hT=0x60004) == MISALIGNED
    assert _chunk(lib, h0=0x80002) == MISALIGNED
    assert _chunk(lib, cu=0x70004, nseq=1) == MISALIGNED
    assert _chunk(lib, o=0x10000 + 16) == INVALID              # o overlaps q
    assert _chunk(lib, hT=0x30000) == INVALID                  # hT overlaps v
    assert _chunk(lib, h0=0x60000) == INVALID                  # hT aliases h0
    # T = 0 and no hT: nothing to do
    assert _chunk(lib, T=0, hT=None) == 0


@no_gpu
def test_recurrent_step_argument_errors(lib):
    INVALID, MISALIGNED = 1, 2
    assert _step(lib, N=-1) == INVALID
    assert _step(lib, H=0) == INVALID
    assert _step(lib, N=0) == 0                                # empty batch is a no-op
    assert _step(lib, S=0) == INVALID
    assert _step(lib, g=0x40001) == MISALIGNED
    assert _step(lib, S=0x100000, o=0x100000 + 1024) == INVALID   # o inside S
    assert _step(lib, S=0x10000) == INVALID                        # S overlaps q


def _istep(lib, q=0x10000, k=0x20000, v=0x30000, g=0x40000, pool=0x100000, dt=0, idx=0x48000,
           Pn=4, o=0x50000, N=2, H=2, pro=None, pos=None):
    return lib.sala_gla_recurrent_step_indexed(P(q), P(k), P(v), P(g), 0.1, P(pool), dt,
                                               P(idx) if idx else None, Pn, P(o), N, H,
                                               ctypes.byref(pro) if pro is not None else None,
                                               P(pos) if pos else None, None)


def _pro(qw=0x60000, kw=0x60100, eps=1e-6, theta=10000.0):
    from gated_linear_attention_gb300 import sala_gla
    return sala_gla.QkPrologue(qw, kw, eps, theta)


def _qkp(lib, q=0x10000, k=0x20000, pro=None, cu=None, sp=None, Bn=1, T=64, H=2, nseq=0):
    pro = pro if pro is not None else _pro()
    return lib.sala_gla_qk_prologue(P(q), P(k), ctypes.byref(pro), P(cu) if cu else None,
                                    P(sp) if sp else None, Bn, T, H, nseq, None)


@no_gpu
def test_qk_prologue_argument_errors(lib):
    INVALID, MISALIGNED = 1, 2
    assert lib.sala_gla_qk_prologue(P(0x10000), P(0x20000), None, None, None, 1, 64, 2, 0, None) == INVALID
    assert _qkp(lib, pro=_pro(qw=0)) == INVALID
    assert _qkp(lib, pro=_pro(eps=-1.0)) == INVALID
    assert _qkp(lib, pro=_pro(theta=0.0)) == INVALID
    assert _qkp(lib, pro=_pro(kw=0x60108)) == MISALIGNED
    assert _qkp(lib, Bn=0) == INVALID
    assert _qkp(lib, cu=0x70000, nseq=0) == INVALID
    assert _qkp(lib, q=0x10008) == MISALIGNED
    assert _qkp(lib, sp=0x70004) == MISALIGNED
    assert _qkp(lib, k=0x10000 + 1024) == INVALID                      # k overlaps q
    assert _qkp(lib, pro=_pro(qw=0x20000 + 256)) == INVALID           # weight inside k
    assert _qkp(lib, T=0) == 0
    assert _qkp(lib) == 4                                              # no GPU here
    # the decode step with a prologue needs positions
    assert _istep(lib, pro=_pro()) == INVALID
    assert _istep(lib, pro=_pro(), pos=0x70004) == MISALIGNED
    assert _istep(lib, pro=_pro(theta=-1.0), pos=0x70000) == INVALID
    assert _istep(lib, pro=_pro(), pos=0x70000) == 4


@no_gpu
def test_recurrent_step_indexed_argument_errors(lib):
    INVALID, MISALIGNED = 1, 2
    assert _istep(lib, N=-1) == INVALID
    assert _istep(lib, H=0) == INVALID
    assert _istep(lib, Pn=0) == INVALID
    assert _istep(lib, dt=2) == INVALID                            # unknown storage type
    assert _istep(lib, N=0) == 0                                   # empty batch is a no-op
    assert _istep(lib, idx=0) == INVALID
    assert _istep(lib, pool=0) == INVALID
    assert _istep(lib, idx=0x48004) == MISALIGNED
    assert _istep(lib, pool=0x100008) == MISALIGNED
    # pool of 4 slots x 2 heads: 512 KB fp32, 256 KB bf16
    assert _istep(lib, o=0x100000 + 300 * 1024) == INVALID           # o inside the fp32 pool
    assert _istep(lib, dt=1, o=0x100000 + 300 * 1024) != INVALID     # past the bf16 pool
    assert _istep(lib, pool=0x40000) == INVALID                      # pool overlaps g
    assert _istep(lib, idx=0x100000 + 4096) == INVALID               # indices inside the pool


def _gate(lib, o=0x10000, z=0x20000, w=0x30000, eps=1e-6, out=0x40000, T=2, H=2):
    return lib.sala_gla_output_norm_gate(P(o), P(z), P(w), eps, P(out) if out else None, T, H, None)


@no_gpu
def test_output_norm_gate_argument_errors(lib):
    INVALID, MISALIGNED = 1, 2
    assert _gate(lib, T=-1) == INVALID
    assert _gate(lib, H=0) == INVALID
    assert _gate(lib, eps=-1.0) == INVALID
    assert _gate(lib, T=0) == 0
    assert _gate(lib, out=0) == INVALID
    assert _gate(lib, z=0x20008) == MISALIGNED
    assert _gate(lib, out=0x20000) == INVALID                 # out overlaps z
    assert _gate(lib, out=0x10000 + 256) == INVALID           # out overlaps part of o
    assert _gate(lib, out=0x10000) == 4                       # in place is allowed (no GPU here)


def _gstep(lib, q=0x10000, k=0x20000, v=0x30000, g=0x40000, b=0x44000, S=0x100000, o=0x50000, N=2, H=2):
    return lib.sala_gla_gdn_recurrent_step(P(q), P(k), P(v), P(g), P(b) if b else None, 0.1, P(S),
                                           P(o), N, H, None)


@no_gpu
def test_gdn_step_argument_errors(lib):
    INVALID, MISALIGNED = 1, 2
    assert _gstep(lib, N=-1) == INVALID
    assert _gstep(lib, H=0) == INVALID
    assert _gstep(lib, N=0) == 0
    assert _gstep(lib, b=0) == INVALID
    assert _gstep(lib, b=0x44004) == MISALIGNED
    assert _gstep(lib, S=0x44000) == INVALID                    # S overlaps beta
    assert _gstep(lib, o=0x100000 + 64) == INVALID              # o inside S
    assert _gstep(lib) == 4                                     # no GPU here


def _gfwd(lib, q=0x10000, k=0x20000, v=0x30000, g=0x40000, b=0x44000, h0=None, cu=None,
          o=0x50000, hT=0x60000, Bn=1, T=64, H=2, nseq=0):
    return lib.sala_gla_gdn_fwd(P(q), P(k), P(v), P(g), P(b) if b else None, 0.1,
                                P(h0) if h0 else None, P(cu) if cu else None, P(o),
                                P(hT) if hT else None, Bn, T, H, nseq, None)


@no_gpu
def test_gdn_fwd_argument_errors(lib):
    INVALID, MISALIGNED = 1, 2
    assert _gfwd(lib, Bn=0) == INVALID
    assert _gfwd(lib, b=0) == INVALID
    assert _gfwd(lib, cu=0x70000, nseq=0) == INVALID
    assert _gfwd(lib, b=0x44004) == MISALIGNED
    assert _gfwd(lib, o=0x10000 + 64) == INVALID                # o overlaps q
    assert _gfwd(lib, hT=0x44000) == INVALID                    # hT overlaps beta
    assert _gfwd(lib, T=0, hT=None) == 0
    assert _gfwd(lib) == 4                                      # no GPU here


@no_gpu
def test_valid_arguments_without_a_gpu_report_cuda_error(lib):
    # validation passes, then the runtime finds no device: nothing is launched
    assert _chunk(lib) == 4
    assert _step(lib) == 4
    assert _istep(lib) == 4
    assert _istep(lib, dt=1) == 4


def test_binding_refuses_cpu_tensors(lib):
    from gated_linear_attention_gb300 import sala_gla
    q = torch.zeros((1, 4, 1, 128), dtype=torch.bfloat16)
    g = torch.zeros((1, 4, 1))
    with pytest.raises(ValueError):
        sala_gla.chunk_fwd(q, q, q, g, 0.1)
    with pytest.raises(ValueError):
        sala_gla.recurrent_step(q[0], q[0], q[0], g[0], 0.1,
                                torch.zeros((4, 1, 128, 128)))


def test_prefill_kernel_choice(lib):
    # host-side setting, no CUDA involved: 0 per call, 1 one unit per SM, 2 two CTAs per SM
    assert lib.sala_gla_set_prefill_kernel(3) == 1     # SALA_ERR_INVALID_ARG
    assert lib.sala_gla_set_prefill_kernel(-1) == 1
    for k in (1, 2, 0):
        assert lib.sala_gla_set_prefill_kernel(k) == 0
