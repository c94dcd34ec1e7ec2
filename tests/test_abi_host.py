"""Host-side checks of the C ABI that need no GPU.

The library must load and export every function that include/bw.h declares,
and every argument check must reject bad input on the host, before any CUDA
call, with the documented status.
"""
import ctypes
import os
import re

import pytest

from conftest import ROOT, build_lib

HEADER = os.path.join(ROOT, "include", "bw.h")
OK, INVALID, SHAPE, MISALIGNED = 0, 1, 2, 3


@pytest.fixture(scope="module")
def lib():
    return ctypes.CDLL(build_lib())


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(bw_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


def test_header_declares_the_path():
    names = declared_functions()
    for required in ("bw_quant_act", "bw_repack", "bw_unrepack",
                     "bw_gemv_w2a8", "bw_gemv_w2a8_acc", "bw_repack_bytes",
                     "bw_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_names_match_header(lib):
    import bit_gemv_bitlinear_gb300 as bw
    assert sorted(bw.EXPORTS) == declared_functions()


def test_status_strings_and_version(lib):
    lib.bw_status_string.restype = ctypes.c_char_p
    names = [lib.bw_status_string(i).decode() for i in range(7)]
    assert names == ["BW_OK", "BW_ERR_INVALID_ARG", "BW_ERR_UNSUPPORTED_SHAPE",
                     "BW_ERR_MISALIGNED", "BW_ERR_BAD_CODE", "BW_ERR_CUDA",
                     "BW_ERR_TIMEOUT"]
    assert lib.bw_status_string(99) is not None
    assert lib.bw_version() >= 100


def test_repack_bytes_matches_layout_spec(lib):
    import oracle
    lib.bw_repack_bytes.restype = ctypes.c_size_t
    for N, K in [(1, 4), (8, 64), (5, 68), (2560, 2560), (13824, 2560),
                 (2560, 6912), (55296, 5120), (1000, 300), (3, 65536)]:
        assert lib.bw_repack_bytes(N, K) == oracle.layout_bytes(N, K)
    assert lib.bw_repack_bytes(0, 64) == 0
    assert lib.bw_repack_bytes(8, 0) == 0
    assert lib.bw_repack_bytes(8, 65540) == 0


def test_gemv_needs_no_workspace(lib):
    """No GEMV path reduces across CTAs, so no shape needs scratch."""
    lib.bw_gemv_workspace_bytes.restype = ctypes.c_size_t
    lib.bw_gemv_workspace_bytes.argtypes = [ctypes.c_int] * 3
    for M, N, K in [(1, 2560, 2560), (64, 13824, 2560), (1, 55296, 5120),
                    (5, 17, 65536)]:
        assert lib.bw_gemv_workspace_bytes(M, N, K) == 0


P = ctypes.c_void_p


def gemv(lib, x, w, s, ws, bounds, n_ws, M, N, K, y, fn="bw_gemv_w2a8"):
    f = getattr(lib, fn)
    f.restype = ctypes.c_int
    f.argtypes = [P, P, P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                  ctypes.c_int, P, P]
    b = None if bounds is None else (ctypes.c_int * len(bounds))(*bounds)
    return f(x, w, s, ws, ctypes.cast(b, P) if b is not None else None, n_ws,
             M, N, K, y, None)


# Fake, never-dereferenced device addresses with the alignment required.
A16, A4, A2 = 0x10000, 0x20000, 0x30000


@pytest.mark.parametrize("fn", ["bw_gemv_w2a8", "bw_gemv_w2a8_lut"])
def test_gemv_host_validation(lib, fn):
    good = dict(x=A16, w=A16, s=A4, ws=A2, bounds=[0, 64], n_ws=1, M=1,
                N=64, K=256, y=A2)

    def call(**kw):
        a = dict(good)
        a.update(kw)
        return gemv(lib, a["x"], a["w"], a["s"], a["ws"], a["bounds"],
                    a["n_ws"], a["M"], a["N"], a["K"], a["y"], fn)

    assert call(x=None) == INVALID
    assert call(w=None) == INVALID
    assert call(y=None) == INVALID
    assert call(s=None) == INVALID
    assert call(bounds=None) == INVALID
    assert call(M=0) == INVALID
    assert call(N=0) == INVALID
    assert call(K=0) == INVALID
    assert call(K=258) == SHAPE            # not a multiple of 4
    assert call(K=65540) == SHAPE          # above the maximum
    assert call(M=4097) == SHAPE
    assert call(bounds=[0, 63]) == INVALID           # does not end at N
    assert call(bounds=[1, 64]) == INVALID           # does not start at 0
    assert call(bounds=[0, 32, 32, 64], n_ws=3) == INVALID  # not increasing
    assert call(bounds=list(range(0, 64, 7)) + [64], n_ws=10) == INVALID
    assert call(n_ws=0) == INVALID
    assert call(w=A16 + 4) == MISALIGNED
    assert call(x=A4 + 1) == MISALIGNED
    assert call(s=A4 + 2) == MISALIGNED
    assert call(y=A2 + 1) == MISALIGNED
    assert call(ws=A2 + 1) == MISALIGNED


def test_other_entry_points_host_validation(lib):
    qa = lib.bw_quant_act
    qa.argtypes = [P, ctypes.c_int, ctypes.c_int, P, P, P]
    assert qa(None, 1, 64, A16, A4, None) == INVALID
    assert qa(A4, 0, 64, A16, A4, None) == INVALID
    assert qa(A4, 1, 65537, A16, A4, None) == SHAPE
    assert qa(A4 + 2, 1, 64, A16, A4, None) == MISALIGNED
    rp = lib.bw_repack
    rp.argtypes = [P, ctypes.c_int, ctypes.c_int, P, P]
    assert rp(None, 8, 64, A16, None) == INVALID
    assert rp(A16, 8, 66, A16, None) == SHAPE
    assert rp(A16, 8, 64, A16 + 8, None) == MISALIGNED
    ur = lib.bw_unrepack
    ur.argtypes = [P, ctypes.c_int, ctypes.c_int, P, P]
    assert ur(A16 + 8, 8, 64, A16, None) == MISALIGNED
    assert ur(A16, 0, 64, A16, None) == INVALID
    ga = lib.bw_gemv_w2a8_acc
    ga.argtypes = [P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P]
    assert ga(A16, A16, 1, 64, 256, A4 + 2, None) == MISALIGNED
    assert ga(A16, A16, 1, 64, 6, A4, None) == SHAPE
    la = lib.bw_gemv_w2a8_lut_acc
    la.argtypes = [P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P]
    assert la(A16, A16, 1, 64, 256, A4 + 2, None) == MISALIGNED
    assert la(A16, A16, 1, 64, 6, A4, None) == SHAPE
    assert la(None, A16, 1, 64, 256, A4, None) == INVALID


def test_gemm_workspace_and_host_validation(lib):
    """The prefill product (bw_gemm_w2a8): its workspace size (fp16 tokens
    of 64 C columns plus the token sums, each rounded to 256 bytes), and
    every argument check before any CUDA call."""
    wb = lib.bw_gemm_workspace_bytes
    wb.restype = ctypes.c_size_t
    wb.argtypes = [ctypes.c_int, ctypes.c_int]
    r256 = lambda b: (b + 255) // 256 * 256
    for M, K in [(1, 4), (256, 2560), (1024, 2560), (77, 300), (4096, 16384)]:
        C = (K + 63) // 64
        assert wb(M, K) == r256(M * C * 64 * 2) + r256(M * 4)
    assert wb(0, 2560) == 0 and wb(4097, 2560) == 0
    assert wb(256, 6) == 0 and wb(256, 16388) == 0

    f = lib.bw_gemm_w2a8
    f.restype = ctypes.c_int
    f.argtypes = [P, P, P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                  ctypes.c_int, P, P, ctypes.c_size_t, P]
    W256 = 0x100000  # fake, 256-byte aligned
    good = dict(x=A16, w=A16, s=A4, ws=A2, bounds=[0, 64], n_ws=1, M=300,
                N=64, K=2560, y=A2, work=W256, wbytes=wb(300, 2560))

    def call(**kw):
        a = dict(good)
        a.update(kw)
        b = (None if a["bounds"] is None else
             (ctypes.c_int * len(a["bounds"]))(*a["bounds"]))
        return f(a["x"], a["w"], a["s"], a["ws"],
                 ctypes.cast(b, P) if b is not None else None, a["n_ws"],
                 a["M"], a["N"], a["K"], a["y"], a["work"], a["wbytes"], None)

    assert call(x=None) == INVALID
    assert call(y=None) == INVALID
    assert call(s=None) == INVALID
    assert call(bounds=[0, 63]) == INVALID
    assert call(M=0) == INVALID
    assert call(K=258) == SHAPE
    assert call(K=16388, wbytes=1 << 40) == SHAPE   # above the fp32-exact K
    assert call(M=4097) == SHAPE
    assert call(work=None) == INVALID
    assert call(wbytes=wb(300, 2560) - 1) == INVALID
    assert call(work=W256 + 128) == MISALIGNED
    assert call(x=A4 + 1) == MISALIGNED
    assert call(w=A16 + 4) == MISALIGNED
    fa = lib.bw_gemm_w2a8_acc
    fa.restype = ctypes.c_int
    fa.argtypes = [P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P,
                   ctypes.c_size_t, P]
    assert fa(A16, A16, 300, 64, 2560, A4 + 2, W256, wb(300, 2560),
              None) == MISALIGNED
    assert fa(A16, A16, 300, 64, 2560, A4, W256, 16, None) == INVALID
    assert fa(None, A16, 300, 64, 2560, A4, W256, wb(300, 2560),
              None) == INVALID


def test_product_path_never_touches_the_oracle():
    """The package and its sources must not reference the oracle."""
    pkg = os.path.join(ROOT, "bit_gemv_bitlinear_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in text.lower(), f


class _Desc(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int), ("dim", ctypes.c_int),
                ("ffn", ctypes.c_int), ("n_heads", ctypes.c_int),
                ("n_kv_heads", ctypes.c_int), ("eps", ctypes.c_float),
                ("wqkv", P), ("wo", P), ("w13", P), ("w2", P), ("ws", P),
                ("gammas", P)]


def test_stack_create_host_validation(lib):
    create = lib.bw_stack_create
    create.argtypes = [P, P]
    run = lib.bw_layer_stack
    run.argtypes = [P, P, ctypes.c_int, P, P, P]
    handle = P()
    L = 2
    w16 = (P * L)(A16, A16 + 256)
    ws = (P * L)(A2, A2 + 64)
    gam = (P * L)(A4, A4 + 64)

    def make(**kw):
        base = dict(n_layers=L, dim=256, ffn=512, n_heads=4, n_kv_heads=2,
                    eps=1e-5, wqkv=ctypes.cast(w16, P), wo=ctypes.cast(w16, P),
                    w13=ctypes.cast(w16, P), w2=ctypes.cast(w16, P),
                    ws=ctypes.cast(ws, P), gammas=ctypes.cast(gam, P))
        base.update(kw)
        return create(ctypes.byref(_Desc(**base)), ctypes.byref(handle))

    assert create(None, ctypes.byref(handle)) == INVALID
    assert make(n_layers=0) == INVALID
    assert make(dim=250) == SHAPE           # not a multiple of n_heads
    assert make(n_kv_heads=3) == SHAPE      # does not divide n_heads
    assert make(ffn=8196) == SHAPE          # above the glue limit
    assert make(ffn=1020) == SHAPE          # gate/up pairs need ffn % 8 == 0
    assert make(wo=None) == INVALID
    bad = (P * L)(A16, A16 + 8)             # second layer misaligned
    assert make(w2=ctypes.cast(bad, P)) == MISALIGNED
    gbad = (P * L)(A4, A4 + 4)              # gains read as float4
    assert make(gammas=ctypes.cast(gbad, P)) == MISALIGNED
    assert run(None, A4, 1, A4, None, None) == INVALID


def test_attn_workspace_and_host_validation(lib):
    wsb = lib.bw_attn_workspace_bytes
    wsb.restype = ctypes.c_size_t
    wsb.argtypes = [ctypes.c_int] * 4
    # BitNet-2B: 5 KV heads x 4 query heads; room for the most splits any
    # device uses, one per 64 positions of a 4096 cache: [5][64] partials
    # of 4 x (128 + 4) floats (256-byte rounded), then 5 counters.
    assert wsb(20, 5, 128, 4096) == 5 * 64 * 4 * 132 * 4 + 5 * 4
    assert wsb(20, 5, 128, 65536) == 5 * 1024 * 4 * 132 * 4 + 5 * 4
    assert wsb(20, 5, 128, 10) == (5 * 4 * 132 * 4 + 255) // 256 * 256 + 20
    assert wsb(20, 5, 64, 4096) == 0          # head dim other than 128
    assert wsb(12, 4, 128, 4096) == 0         # 3 query heads per KV head
    assert wsb(20, 5, 128, 65537) == 0
    ad = lib.bw_attn_decode
    ad.restype = ctypes.c_int
    ad.argtypes = [P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                   ctypes.c_int, ctypes.c_float, P, P, P, P, ctypes.c_size_t,
                   P]
    need = wsb(20, 5, 128, 4096)

    def call(qkv=A16, pos=A4, H=20, Hkv=5, D=128, S=4096, theta=5e5,
             kc=A16, vc=A16, out=A4, ws=A16, nb=need):
        return ad(qkv, pos, H, Hkv, D, S, theta, kc, vc, out, ws, nb, None)

    assert call(qkv=None) == INVALID
    assert call(ws=None) == INVALID
    assert call(Hkv=3) == INVALID             # 20 % 3 != 0
    assert call(H=12, Hkv=4) == SHAPE         # G = 3
    assert call(D=64) == SHAPE
    assert call(S=65537) == SHAPE
    assert call(theta=0.0) == INVALID
    assert call(theta=float("nan")) == INVALID
    assert call(nb=need - 1) == INVALID
    assert call(kc=A16 + 8) == MISALIGNED
    assert call(vc=A16 + 2) == MISALIGNED
    assert call(pos=A4 + 2) == MISALIGNED
    assert call(out=A4 + 1) == MISALIGNED
    assert call(ws=A16 + 4) == MISALIGNED
    # The flagged form validates the same way, and refuses unknown flags
    # before any launch.
    ax = lib.bw_attn_decode_ex
    ax.restype = ctypes.c_int
    ax.argtypes = [P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                   ctypes.c_int, ctypes.c_float, P, P, P, P, ctypes.c_size_t,
                   ctypes.c_uint, P]

    def call_ex(flags, qkv=A16, nb=need, D=128):
        return ax(qkv, A4, 20, 5, D, 4096, 5e5, A16, A16, A4, A16, nb, flags,
                  None)

    assert call_ex(2) == INVALID
    assert call_ex(0x80000000) == INVALID
    assert call_ex(1, qkv=None) == INVALID
    assert call_ex(1, nb=need - 1) == INVALID
    assert call_ex(1, D=64) == SHAPE


def test_stack_create_kv_host_validation(lib):
    create = lib.bw_stack_create_kv
    create.argtypes = [P, ctypes.c_int, ctypes.c_float, P]
    handle = P()
    L = 1
    w16 = (P * L)(A16)
    ws = (P * L)(A2)
    gam = (P * L)(A4)

    def make(S=64, theta=5e5, **kw):
        base = dict(n_layers=L, dim=512, ffn=1024, n_heads=4, n_kv_heads=2,
                    eps=1e-5, wqkv=ctypes.cast(w16, P), wo=ctypes.cast(w16, P),
                    w13=ctypes.cast(w16, P), w2=ctypes.cast(w16, P),
                    ws=ctypes.cast(ws, P), gammas=ctypes.cast(gam, P))
        base.update(kw)
        return create(ctypes.byref(_Desc(**base)), S, theta,
                      ctypes.byref(handle))

    assert make(S=0) == INVALID
    assert make(S=-3) == INVALID
    assert make(S=65537) == SHAPE           # beyond BW_ATTN_MAX_S
    assert make(dim=256) == SHAPE           # head dim 64, attention needs 128
    assert make(n_heads=3, dim=384, n_kv_heads=1) == SHAPE   # 3 heads per KV
    assert make(theta=0.0) == INVALID
    assert make(theta=float("inf")) == INVALID
    assert make(wo=None) == INVALID
    reset = lib.bw_stack_reset_kv
    reset.argtypes = [P, P]
    assert reset(None, None) == INVALID
    read = lib.bw_stack_read_kv
    read.argtypes = [P, ctypes.c_int, P, P, P]
    assert read(None, 0, A2, A2, None) == INVALID
