"""The C ABI on the CPU: the library loads, exports every declared symbol, and
rejects bad arguments synchronously (before any CUDA call is made)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__ as g
    g.build()
    from hybrid_linear_attention_chunk_gb300 import _lib
    return _lib.load()


def declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(kda_[a-z0-9_]+)\s*\(", src))
    return sorted(names)


def test_header_declares_the_boundary():
    names = declared_symbols()
    for n in ("kda_chunk_fwd", "kda_decode_step", "kda_status_string"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in declared_symbols():
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"


def test_status_strings(lib):
    for s in range(-8, 1):
        assert lib.kda_status_string(s)
    assert lib.kda_last_cuda_error() is not None


def _desc(**kw):
    from hybrid_linear_attention_chunk_gb300._lib import KdaChunkDesc
    d = KdaChunkDesc()
    vals = dict(B=1, T=128, H=2, dk=64, dv=64, chunk=64, num_seqs=0, qkv_dtype=1, out_dtype=1,
                gate_dtype=0, validate=0, kernel=0, segments=0)
    vals.update(kw)
    for k, v in vals.items():
        setattr(d, k, v)
    return d


FAKE = 1 << 20  # a 16-byte aligned fake device address: never dereferenced


def _call(lib, d, **ptrs):
    p = dict(q=FAKE, k=FAKE * 2, v=FAKE * 3, g=FAKE * 4, b=FAKE * 5, s0=None, cu=None, o=FAKE * 6,
             sT=None)
    p.update(ptrs)
    P = ctypes.c_void_p
    return lib.kda_chunk_fwd(ctypes.byref(d), P(p["q"]), P(p["k"]), P(p["v"]), P(p["g"]), P(p["b"]),
                             P(p["s0"]), P(p["cu"]), P(p["o"]), P(p["sT"]), None)


def test_argument_errors_are_synchronous(lib):
    assert lib.kda_chunk_fwd(None, None, None, None, None, None, None, None, None, None, None) == -1
    assert _call(lib, _desc(), q=None) == -1
    assert _call(lib, _desc(dk=48)) == -2
    assert _call(lib, _desc(chunk=128)) == -2
    assert _call(lib, _desc(H=0)) == -2
    assert _call(lib, _desc(qkv_dtype=7)) == -3
    assert _call(lib, _desc(), k=FAKE * 2 + 4) == -4
    assert _call(lib, _desc(B=2), cu=FAKE * 9) == -2          # varlen needs B == 1
    assert _call(lib, _desc(num_seqs=3)) == -2                # num_seqs without cu_seqlens
    assert _call(lib, _desc(), o=FAKE * 3) == -8              # out aliases v
    assert _call(lib, _desc(segments=-1)) == -2


def test_decode_argument_errors(lib):
    from hybrid_linear_attention_chunk_gb300._lib import KdaDecodeDesc
    d = KdaDecodeDesc()
    d.N, d.H, d.dk, d.dv, d.qkv_dtype, d.out_dtype, d.gate_dtype, d.validate = 4, 2, 128, 128, 1, 1, 0, 0
    P = ctypes.c_void_p
    ok = [P(FAKE * i) for i in range(1, 8)]
    assert lib.kda_decode_step(ctypes.byref(d), *ok[:6], None, None) == -1
    bad = list(ok)
    bad[5] = P(FAKE * 1)  # state aliases q
    assert lib.kda_decode_step(ctypes.byref(d), *bad, None) == -8
    d.dv = 100
    assert lib.kda_decode_step(ctypes.byref(d), *ok, None) == -2


def test_workspace_size_is_host_only(lib):
    n = ctypes.c_size_t(123)
    assert lib.kda_chunk_fwd_workspace_size(ctypes.byref(_desc()), ctypes.byref(n)) == 0


def test_product_package_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "hybrid_linear_attention_chunk_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h", ".c")):
                src = open(os.path.join(dirpath, fn)).read()
                assert "import oracle" not in src and "from oracle" not in src, fn
                assert "kda_oracle" not in src, fn


def test_segment_planner_sizes(lib):
    """The long-sequence planner is host-only: the long-context shape (one
    sequence of 2^20 tokens, 16 heads) gets a workspace, the batch shape
    (4 x 8192 tokens, 32 heads) does not."""
    n = ctypes.c_size_t(0)
    long_ctx = _desc(B=1, T=1 << 20, H=16, dk=128, dv=128)
    assert lib.kda_chunk_fwd_workspace_size(ctypes.byref(long_ctx), ctypes.byref(n)) == 0
    assert n.value > 0 and n.value % (128 * 128 * 4 * 16) == 0
    batch = _desc(B=4, T=8192, H=32, dk=128, dv=128)
    assert lib.kda_chunk_fwd_workspace_size(ctypes.byref(batch), ctypes.byref(n)) == 0
    assert n.value == 0
    forced = _desc(B=1, T=4096, H=2, dk=128, dv=128, segments=4)
    assert lib.kda_chunk_fwd_workspace_size(ctypes.byref(forced), ctypes.byref(n)) == 0
    assert n.value == (3 * 4 - 5) * 2 * 128 * 128 * 4  # P-2 pairs and P-1 entry states per chain
    varlen_split = _desc(B=1, T=4096, H=2, dk=128, dv=128, num_seqs=2, segments=4)
    assert lib.kda_chunk_fwd_workspace_size(ctypes.byref(varlen_split), ctypes.byref(n)) == -7


def test_checkpoint_argument_errors(lib):
    P = ctypes.c_void_p

    def call(d, every, ckpt=FAKE * 7, cu=None, cu_ck=None):
        return lib.kda_chunk_fwd_ckpt(ctypes.byref(d), P(FAKE), P(FAKE * 2), P(FAKE * 3), P(FAKE * 4),
                                      P(FAKE * 5), None, P(cu) if cu else None, P(FAKE * 6), None, every,
                                      P(cu_ck) if cu_ck else None, P(ckpt) if ckpt else None, None, 0, None)

    assert call(_desc(), 64, ckpt=None) == -1                   # no checkpoint buffer
    assert call(_desc(), 96) == -2                              # not a multiple of the chunk
    assert call(_desc(), 0) == -2
    assert call(_desc(num_seqs=2), 64, cu=FAKE * 9) == -1       # packed sequences need cu_ckpt
    assert call(_desc(), 64, ckpt=FAKE * 6) == -8               # checkpoints alias out
    assert call(_desc(), 64, ckpt=FAKE * 7 + 2) == -4           # misaligned


def test_layer_argument_errors(lib):
    """kda_layer_fwd / kda_layer_decode_step check the gates before launching."""
    from hybrid_linear_attention_chunk_gb300._lib import KdaDecodeDesc, KdaLayerGates
    P = ctypes.c_void_p

    def gates(A=FAKE * 10, g_min=-5.0, og=None, w=None, eps=1e-6):
        lg = KdaLayerGates()
        lg.A_log, lg.g_min, lg.out_gate, lg.norm_weight, lg.norm_eps = A, g_min, og, w, eps
        return lg

    def fwd(lg, out=FAKE * 6):
        return lib.kda_layer_fwd(ctypes.byref(_desc()), None if lg is None else ctypes.byref(lg), P(FAKE),
                                 P(FAKE * 2), P(FAKE * 3), P(FAKE * 4), P(FAKE * 5), None, None, P(out), None,
                                 None, 0, None)

    assert fwd(None) == -1                                   # no gates
    assert fwd(gates(A=None)) == -1                          # A_h is required
    assert fwd(gates(g_min=-6.0)) == -5                      # below the Eq. 5 floor the range guard fails
    assert fwd(gates(g_min=0.0)) == -5
    assert fwd(gates(og=FAKE * 11, eps=-1.0)) == -5
    assert fwd(gates(og=FAKE * 11, eps=float("nan"))) == -5
    assert fwd(gates(og=FAKE * 11 + 4)) == -4                # out_gate is tiled with 16-byte copies
    assert fwd(gates(A=FAKE * 10 + 2)) == -4
    assert fwd(gates(og=FAKE * 6)) == -8                     # out_gate aliases out
    assert fwd(gates(w=FAKE * 6 + 64)) == -8                 # norm weight inside out

    d = KdaDecodeDesc()
    d.N, d.H, d.dk, d.dv, d.qkv_dtype, d.out_dtype, d.gate_dtype, d.validate = 4, 2, 64, 64, 1, 1, 0, 0

    def dec(lg):
        return lib.kda_layer_decode_step(ctypes.byref(d), None if lg is None else ctypes.byref(lg), P(FAKE),
                                         P(FAKE * 2), P(FAKE * 3), P(FAKE * 4), P(FAKE * 5), P(FAKE * 7),
                                         P(FAKE * 6), None)

    assert dec(None) == -1
    assert dec(gates(g_min=-5.5)) == -5
    assert dec(gates(og=FAKE * 7)) == -8                     # out_gate aliases the state


def test_backward_argument_errors(lib):
    P = ctypes.c_void_p

    def bwd(d=None, dq=FAKE * 20, dk=FAKE * 21, dv=FAKE * 22, dg=FAKE * 23, db=FAKE * 24, ws=None, ws_bytes=0):
        d = d or _desc()
        return lib.kda_chunk_bwd(ctypes.byref(d), P(FAKE), P(FAKE * 2), P(FAKE * 3), P(FAKE * 4), P(FAKE * 5),
                                 None, None, P(FAKE * 6), None, P(dq) if dq else None, P(dk), P(dv), P(dg), P(db),
                                 None, P(ws) if ws else None, ws_bytes, None)

    assert bwd(d=_desc(kernel=2)) == -7          # no tensor-core backward
    assert bwd(dq=None) == -1
    assert bwd(dq=FAKE) == -8                    # dq aliases q
    assert bwd(dk=FAKE * 20) == -8               # two gradients overlap
    assert bwd(db=FAKE * 24 + 2) == -4
    n = ctypes.c_size_t(0)
    assert lib.kda_chunk_bwd_workspace_size(ctypes.byref(_desc()), ctypes.byref(n)) == 0
    # 8 chunks of 16 tokens x 2 heads x (3*16*64 + 2*256 + 64 + 2*64*64) floats
    assert n.value == 8 * 2 * (3 * 16 * 64 + 2 * 256 + 64 + 2 * 64 * 64) * 4
    assert bwd(ws=FAKE * 40, ws_bytes=n.value - 4) == -2
