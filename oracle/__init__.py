"""CPU oracle for the W2A8 ternary GEMV path -- TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may
import this package.  The CUDA library never loads it, and it never loads
the CUDA library.  The arithmetic lives in ``oracle.c`` (plain C, one element
at a time); this module only compiles it and marshals numpy arrays.

Sources are cited in ``oracle.c``: the BitNet GPU W2A8 kernel page
("BitNet GPU 推理框架：从零构建 W2A8 的 2-bit 大模型 CUDA GEMV 内核"), §5.2
packing, §5.3 dot product and epilogue, §六 item 3 activation quantisation,
§4.1/§一 the decoder-layer shape.
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

OR_OK, OR_BAD_CODE, OR_OVERFLOW, OR_BAD_ARG = 0, 1, 2, 3


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so with the host gcc (no CUDA)."""
    stamp_path = _LIB + ".stamp"
    stamp = platform.machine()
    same_host = (os.path.exists(stamp_path)
                 and open(stamp_path).read() == stamp)
    if (not force and same_host and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-Wall", "-Wextra", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    with open(stamp_path, "w") as f:
        f.write(stamp)
    return _LIB


_lib = None


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        F = ctypes.c_float
        sig = {
            "or_unpack": (ctypes.c_int, [P, I64, I64, P]),
            "or_pack": (ctypes.c_int, [P, I64, I64, P]),
            "or_gemv_acc": (ctypes.c_int, [P, P, I64, I64, I64, P]),
            "or_bf16_rne": (ctypes.c_uint16, [F]),
            "or_bf16_value": (F, [ctypes.c_uint16]),
            "or_gemv": (ctypes.c_int, [P, P, P, P, P, I64, I64, I64, I64, P]),
            "or_quant_act": (None, [P, I64, I64, P, P]),
            "or_layout_bytes": (I64, [I64, I64]),
            "or_layout": (ctypes.c_int, [P, I64, I64, P]),
            "or_rmsnorm": (None, [P, P, I64, F, P]),
            "or_relu2_gate": (None, [P, I64, P]),
            "or_attn_one_token": (ctypes.c_int, [P, I64, I64, I64, P]),
            "or_layer": (ctypes.c_int, [P, I64, I64, I64, I64, F,
                                        P, P, P, P, P, P, P]),
            "or_quant_weight": (ctypes.c_int, [P, I64, I64, P, I64, P, P]),
            "or_bf16_rne_d": (ctypes.c_uint16, [ctypes.c_double]),
            "or_rope_angle": (F, [I64, I64, I64, F]),
            "or_rope": (ctypes.c_int, [P, I64, I64, F, P]),
            "or_attn_decode": (ctypes.c_int, [P, I64, I64, I64, I64, F, P, P,
                                              I64, P]),
            "or_attn_append": (ctypes.c_int, [P, I64, I64, I64, I64, F, P, P,
                                              I64]),
            "or_attn_over_cache": (ctypes.c_int, [P, I64, I64, I64, I64, F, P,
                                                  P, I64, P]),
            "or_layer_kv": (ctypes.c_int, [P, I64, I64, I64, I64, F,
                                           P, P, P, P, P, P, P, P, P, I64,
                                           I64, F]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, what: str):
    if rc != OR_OK:
        names = {OR_BAD_CODE: "code 3 in canonical bytes",
                 OR_OVERFLOW: "int32 overflow", OR_BAD_ARG: "bad argument"}
        raise OracleError(f"{what}: {names.get(rc, rc)}")


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def unpack(canon: np.ndarray, N: int, K: int) -> np.ndarray:
    """Canonical bytes [N][K/4] -> ternary int8 [N][K]."""
    canon = _c(canon, np.uint8)
    w = np.empty((N, K), np.int8)
    _check(_load().or_unpack(_ptr(canon), N, K, _ptr(w)), "unpack")
    return w


def pack(w: np.ndarray) -> np.ndarray:
    """Ternary int8 [N][K] -> canonical bytes [N][K/4]."""
    w = _c(w, np.int8)
    N, K = w.shape
    canon = np.empty((N, K // 4), np.uint8)
    _check(_load().or_pack(_ptr(w), N, K, _ptr(canon)), "pack")
    return canon


def gemv_acc(q: np.ndarray, canon: np.ndarray, N: int, K: int) -> np.ndarray:
    """Exact int32 acc [M][N] = q [M][K] . W^T."""
    q = _c(q, np.int8).reshape(-1, K)
    canon = _c(canon, np.uint8)
    M = q.shape[0]
    acc = np.empty((M, N), np.int32)
    _check(_load().or_gemv_acc(_ptr(q), _ptr(canon), M, N, K, _ptr(acc)),
           "gemv_acc")
    return acc


def bf16_rne(x: float) -> int:
    return int(_load().or_bf16_rne(float(x)))


def bf16_value(h: int) -> float:
    return float(_load().or_bf16_value(int(h)))


def gemv(q, canon, s, ws_bits, bounds, N: int, K: int) -> np.ndarray:
    """bf16 bit patterns y [M][N] = bf16((acc / s[m]) * ws[seg(n)])."""
    q = _c(q, np.int8).reshape(-1, K)
    canon = _c(canon, np.uint8)
    s = _c(s, np.float32).reshape(-1)
    ws_bits = _c(ws_bits, np.uint16).reshape(-1)
    bounds = _c(bounds, np.int32).reshape(-1)
    M = q.shape[0]
    y = np.empty((M, N), np.uint16)
    _check(_load().or_gemv(_ptr(q), _ptr(canon), _ptr(s), _ptr(ws_bits),
                           _ptr(bounds), len(ws_bits), M, N, K, _ptr(y)),
           "gemv")
    return y


def quant_act(x: np.ndarray):
    """fp32 x [M][K] -> (int8 q [M][K], fp32 s [M])."""
    x = _c(x, np.float32)
    if x.ndim == 1:
        x = x.reshape(1, -1)
    M, K = x.shape
    q = np.empty((M, K), np.int8)
    s = np.empty((M,), np.float32)
    _load().or_quant_act(_ptr(x), M, K, _ptr(q), _ptr(s))
    return q, s


def quant_weight(W: np.ndarray, bounds):
    """Absmean ternarisation: fp32 W [N][K], row segments `bounds` (n_ws + 1
    values from 0 to N) -> (canonical codes uint8 [N][K/4], bf16 bit
    patterns of ws uint16 [n_ws])."""
    W = _c(W, np.float32)
    N, K = W.shape
    b = _c(np.asarray(bounds), np.int32)
    n_ws = len(b) - 1
    canon = np.empty((N, K // 4), np.uint8)
    ws = np.empty((n_ws,), np.uint16)
    _check(_load().or_quant_weight(_ptr(W), N, K, _ptr(b), n_ws, _ptr(canon),
                                   _ptr(ws)), "quant_weight")
    return canon, ws


def layout_bytes(N: int, K: int) -> int:
    return int(_load().or_layout_bytes(N, K))


def layout(canon: np.ndarray, N: int, K: int) -> np.ndarray:
    """Canonical bytes -> the device weight layout, restated element-wise."""
    canon = _c(canon, np.uint8)
    out = np.empty((layout_bytes(N, K),), np.uint8)
    _check(_load().or_layout(_ptr(canon), N, K, _ptr(out)), "layout")
    return out


def rmsnorm(x, gamma, eps: float) -> np.ndarray:
    x = _c(x, np.float32).reshape(-1)
    gamma = _c(gamma, np.float32).reshape(-1)
    out = np.empty_like(x)
    _load().or_rmsnorm(_ptr(x), _ptr(gamma), x.size, eps, _ptr(out))
    return out


def relu2_gate(gu_bits) -> np.ndarray:
    gu_bits = _c(gu_bits, np.uint16).reshape(-1)
    F = gu_bits.size // 2
    out = np.empty((F,), np.float32)
    _load().or_relu2_gate(_ptr(gu_bits), F, _ptr(out))
    return out


def attn_one_token(qkv_bits, n_heads: int, n_kv: int, head_dim: int):
    qkv_bits = _c(qkv_bits, np.uint16).reshape(-1)
    out = np.empty((n_heads * head_dim,), np.float32)
    _check(_load().or_attn_one_token(_ptr(qkv_bits), n_heads, n_kv, head_dim,
                                     _ptr(out)), "attn_one_token")
    return out


def layer(h, dim, ffn, n_heads, n_kv, eps, wqkv, wo, w13, w2, ws_bits,
          gammas) -> np.ndarray:
    """One decoder layer on fp32 h [dim]; returns the updated copy."""
    h = _c(h, np.float32).reshape(-1).copy()
    ws_bits = _c(ws_bits, np.uint16).reshape(-1)
    gammas = _c(gammas, np.float32).reshape(-1)
    mats = [_c(m, np.uint8) for m in (wqkv, wo, w13, w2)]
    scratch = np.zeros((4 * ffn,), np.float32)
    rc = _load().or_layer(_ptr(h), dim, ffn, n_heads, n_kv, eps,
                          *[_ptr(m) for m in mats], _ptr(ws_bits),
                          _ptr(gammas), _ptr(scratch))
    _check(rc, "layer")
    return h


def bf16_rne_d(x: float) -> int:
    """bf16 bit pattern of a double, rounded to nearest even in one step."""
    return int(_load().or_bf16_rne_d(float(x)))


def rope_angle(p: int, i: int, D: int, theta: float) -> float:
    """fp32 angle of pair i at position p: fl(p * fl(theta^(-2i/D)))."""
    return float(_load().or_rope_angle(p, i, D, theta))


def rope(x_bits, p: int, theta: float) -> np.ndarray:
    """RoPE of one head (bf16 bit patterns [D]) at position p, fp64 [D]."""
    x_bits = _c(x_bits, np.uint16).reshape(-1)
    out = np.empty((x_bits.size,), np.float64)
    _check(_load().or_rope(_ptr(x_bits), x_bits.size, p, theta, _ptr(out)),
           "rope")
    return out


def attn_decode(qkv_bits, H: int, Hkv: int, D: int, p: int, theta: float,
                kc_bits, vc_bits):
    """One GQA decode step over a bf16 KV cache [Hkv][S][D].  Returns
    (out fp64 [H][D], the updated key cache, the updated value cache); the
    inputs are not modified."""
    qkv_bits = _c(qkv_bits, np.uint16).reshape(-1)
    kc = _c(kc_bits, np.uint16).copy()
    vc = _c(vc_bits, np.uint16).copy()
    S = kc.size // (Hkv * D)
    out = np.empty((H, D), np.float64)
    _check(_load().or_attn_decode(_ptr(qkv_bits), H, Hkv, D, p, theta,
                                  _ptr(kc), _ptr(vc), S, _ptr(out)),
           "attn_decode")
    return out, kc.reshape(Hkv, S, D), vc.reshape(Hkv, S, D)


def attn_append(qkv_bits, H: int, Hkv: int, D: int, p: int, theta: float,
                kc_bits, vc_bits):
    """The cache append of a decode step alone: returns updated copies of
    the key and value caches [Hkv][S][D]."""
    qkv_bits = _c(qkv_bits, np.uint16).reshape(-1)
    kc = _c(kc_bits, np.uint16).copy()
    vc = _c(vc_bits, np.uint16).copy()
    S = kc.size // (Hkv * D)
    _check(_load().or_attn_append(_ptr(qkv_bits), H, Hkv, D, p, theta,
                                  _ptr(kc), _ptr(vc), S), "attn_append")
    return kc.reshape(Hkv, S, D), vc.reshape(Hkv, S, D)


def attn_over_cache(qkv_bits, H: int, Hkv: int, D: int, p: int,
                    theta: float, kc_bits, vc_bits) -> np.ndarray:
    """The attention of a decode step over the cache as given (rows 0..p
    already hold the new token): fp64 out [H][D]."""
    qkv_bits = _c(qkv_bits, np.uint16).reshape(-1)
    kc = _c(kc_bits, np.uint16)
    vc = _c(vc_bits, np.uint16)
    S = kc.size // (Hkv * D)
    out = np.empty((H, D), np.float64)
    _check(_load().or_attn_over_cache(_ptr(qkv_bits), H, Hkv, D, p, theta,
                                      _ptr(kc), _ptr(vc), S, _ptr(out)),
           "attn_over_cache")
    return out


def layer_kv(h, dim, ffn, n_heads, n_kv, eps, wqkv, wo, w13, w2, ws_bits,
             gammas, kc_bits, vc_bits, p: int, theta: float):
    """One decoder layer with attention over its KV cache at position p:
    returns (h after the layer, the updated key cache, value cache)."""
    h = _c(h, np.float32).reshape(-1).copy()
    ws_bits = _c(ws_bits, np.uint16).reshape(-1)
    gammas = _c(gammas, np.float32).reshape(-1)
    mats = [_c(m, np.uint8) for m in (wqkv, wo, w13, w2)]
    kc = _c(kc_bits, np.uint16).copy()
    vc = _c(vc_bits, np.uint16).copy()
    S = kc.size // (n_kv * (dim // n_heads))
    scratch = np.zeros((4 * ffn,), np.float32)
    rc = _load().or_layer_kv(_ptr(h), dim, ffn, n_heads, n_kv, eps,
                             *[_ptr(m) for m in mats], _ptr(ws_bits),
                             _ptr(gammas), _ptr(scratch), _ptr(kc), _ptr(vc),
                             S, p, theta)
    _check(rc, "layer_kv")
    return h, kc.reshape(kc_bits.shape), vc.reshape(vc_bits.shape)
