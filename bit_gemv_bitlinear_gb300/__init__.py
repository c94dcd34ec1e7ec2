"""Python binding of libbw, the GB300 (sm_103a) W2A8 ternary GEMV library.

Argument marshalling only: every step of the path runs in the library's CUDA
kernels, reached through the C ABI of ``include/bw.h``.  PyTorch provides
device memory and streams.  There is no fallback: if ``libbw.so`` is missing
the import fails (build it with ``python -m bit_gemv_bitlinear_gb300.build``
or ``__graft_entry__.build()``).

Function names follow the C ABI: ``bw_quant_act``, ``bw_repack``,
``bw_unrepack``, ``bw_gemv_w2a8``, ``bw_gemv_w2a8_acc``, ``bw_gemm_w2a8``,
``bw_gemm_w2a8_acc``, ``bw_attn_decode``, ``bw_attn_decode_ex``.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libbw.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build the CUDA library first "
        "(python -m bit_gemv_bitlinear_gb300.build)")

_lib = ctypes.CDLL(LIB_PATH)

BW_OK = 0
STATUS_NAMES = {0: "BW_OK", 1: "BW_ERR_INVALID_ARG",
                2: "BW_ERR_UNSUPPORTED_SHAPE", 3: "BW_ERR_MISALIGNED",
                4: "BW_ERR_BAD_CODE", 5: "BW_ERR_CUDA", 6: "BW_ERR_TIMEOUT"}
MAX_K, MAX_N, MAX_M, MAX_WS = 65536, 1 << 24, 4096, 8
BW_ATTN_PAST_READY = 1

# Every symbol the C ABI declares (checked by the tests without a GPU).
EXPORTS = ("bw_status_string", "bw_last_cuda_error", "bw_version",
           "bw_quant_act", "bw_repack_bytes", "bw_repack", "bw_unrepack",
           "bw_gemv_w2a8", "bw_gemv_w2a8_acc", "bw_repack_noalloc",
           "bw_device_error", "bw_stack_create", "bw_layer_stack",
           "bw_stack_destroy", "bw_selftest_wait_timeout",
           "bw_gemv_workspace_bytes", "bw_quant_weight",
           "bw_attn_workspace_bytes", "bw_attn_decode", "bw_attn_decode_ex",
           "bw_stack_create_kv",
           "bw_stack_read_kv", "bw_stack_reset_kv", "bw_gemv_w2a8_lut",
           "bw_gemv_w2a8_lut_acc", "bw_gemm_workspace_bytes", "bw_gemm_w2a8",
           "bw_gemm_w2a8_acc")

_P = ctypes.c_void_p
_I = ctypes.c_int
_SIGS = {
    "bw_status_string": (ctypes.c_char_p, [_I]),
    "bw_last_cuda_error": (_I, []),
    "bw_version": (_I, []),
    "bw_quant_act": (_I, [_P, _I, _I, _P, _P, _P]),
    "bw_repack_bytes": (ctypes.c_size_t, [_I, _I]),
    "bw_gemv_workspace_bytes": (ctypes.c_size_t, [_I, _I, _I]),
    "bw_repack": (_I, [_P, _I, _I, _P, _P]),
    "bw_unrepack": (_I, [_P, _I, _I, _P, _P]),
    "bw_repack_noalloc": (_I, [_P, _I, _I, _P, _P]),
    "bw_gemv_w2a8": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P]),
    "bw_gemv_w2a8_acc": (_I, [_P, _P, _I, _I, _I, _P, _P]),
    "bw_gemv_w2a8_lut": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P]),
    "bw_gemv_w2a8_lut_acc": (_I, [_P, _P, _I, _I, _I, _P, _P]),
    "bw_gemm_workspace_bytes": (ctypes.c_size_t, [_I, _I]),
    "bw_gemm_w2a8": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P,
                          ctypes.c_size_t, _P]),
    "bw_gemm_w2a8_acc": (_I, [_P, _P, _I, _I, _I, _P, _P, ctypes.c_size_t,
                              _P]),
    "bw_device_error": (_I, [_P, _P]),
    "bw_stack_create": (_I, [_P, _P]),
    "bw_layer_stack": (_I, [_P, _P, _I, _P, _P, _P]),
    "bw_stack_destroy": (None, [_P]),
    "bw_selftest_wait_timeout": (_I, [_P, _P]),
    "bw_quant_weight": (_I, [_P, _I, _I, _P, _I, _P, _P, _P]),
    "bw_attn_workspace_bytes": (ctypes.c_size_t, [_I, _I, _I, _I]),
    "bw_stack_create_kv": (_I, [_P, _I, ctypes.c_float, _P]),
    "bw_stack_read_kv": (_I, [_P, _I, _P, _P, _P]),
    "bw_stack_reset_kv": (_I, [_P, _P]),
    "bw_attn_decode": (_I, [_P, _P, _I, _I, _I, _I, ctypes.c_float, _P, _P,
                            _P, _P, ctypes.c_size_t, _P]),
    "bw_attn_decode_ex": (_I, [_P, _P, _I, _I, _I, _I, ctypes.c_float, _P,
                               _P, _P, _P, ctypes.c_size_t, ctypes.c_uint,
                               _P]),
}
for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args


class BwError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        name = STATUS_NAMES.get(status, str(status))
        extra = ""
        if name == "BW_ERR_CUDA":
            extra = f" (cudaError {_lib.bw_last_cuda_error()})"
        super().__init__(f"{what}: {name}{extra}")


def _check(status: int, what: str):
    if status != BW_OK:
        raise BwError(status, what)


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _dev(t: torch.Tensor, dtype, name: str) -> int:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _need(t: torch.Tensor, count: int, name: str):
    """Rejects a buffer with fewer than `count` elements before any kernel
    can read or write past its end."""
    if t.numel() < count:
        raise ValueError(f"{name} holds {t.numel()} elements, needs {count}")


def version() -> int:
    return _lib.bw_version()


def status_string(status: int) -> str:
    return _lib.bw_status_string(status).decode()


def bw_repack_bytes(N: int, K: int) -> int:
    return int(_lib.bw_repack_bytes(N, K))


def bw_gemv_workspace_bytes(M: int, N: int, K: int) -> int:
    """Device scratch a GEMV of this shape needs from the caller (0)."""
    return int(_lib.bw_gemv_workspace_bytes(M, N, K))


def bw_quant_act(x: torch.Tensor, q: torch.Tensor | None = None,
                 s: torch.Tensor | None = None, stream=None):
    """fp32 x [M][K] -> (int8 q [M][K], fp32 s [M]); s = 127/absmax."""
    x2 = x if x.dim() == 2 else x.reshape(1, -1)
    M, K = x2.shape
    if q is None:
        q = torch.empty((M, K), dtype=torch.int8, device=x.device)
    if s is None:
        s = torch.empty((M,), dtype=torch.float32, device=x.device)
    _need(q, M * K, "q")
    _need(s, M, "s")
    _check(_lib.bw_quant_act(_dev(x2, torch.float32, "x"), M, K,
                             _dev(q, torch.int8, "q"),
                             _dev(s, torch.float32, "s"), _stream(stream)),
           "bw_quant_act")
    return q, s


def _repack_sizes(canon: torch.Tensor, N: int, K: int) -> int:
    """Checks that `canon` holds N * K / 4 bytes; returns the size of the
    device layout."""
    size = bw_repack_bytes(N, K)
    if size == 0 or K % 4:
        raise BwError(2, "bw_repack_bytes")
    _need(canon, N * (K // 4), "canon")
    return size


def bw_repack(canon: torch.Tensor, N: int, K: int,
              packed: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Canonical bytes uint8 [N][K/4] -> device layout (synchronising)."""
    size = _repack_sizes(canon, N, K)
    if packed is None:
        packed = torch.empty((size,), dtype=torch.uint8, device=canon.device)
    _need(packed, size, "packed")
    _check(_lib.bw_repack(_dev(canon, torch.uint8, "canon"), N, K,
                          _dev(packed, torch.uint8, "packed"),
                          _stream(stream)), "bw_repack")
    return packed


def bw_repack_noalloc(canon: torch.Tensor, N: int, K: int,
                      packed: torch.Tensor, stream=None) -> torch.Tensor:
    """bw_repack for callers that may not allocate device memory: the caller
    supplies `packed` (bw_repack_bytes(N, K) bytes) and the library uses a
    fixed internal scratch word instead of allocating one (synchronising;
    overlapping calls race on that word)."""
    _need(packed, _repack_sizes(canon, N, K), "packed")
    _check(_lib.bw_repack_noalloc(_dev(canon, torch.uint8, "canon"), N, K,
                                  _dev(packed, torch.uint8, "packed"),
                                  _stream(stream)), "bw_repack_noalloc")
    return packed


def bw_unrepack(packed: torch.Tensor, N: int, K: int,
                canon: torch.Tensor | None = None, stream=None):
    if canon is None:
        canon = torch.empty((N, K // 4), dtype=torch.uint8,
                            device=packed.device)
    _need(packed, _repack_sizes(canon, N, K), "packed")
    _check(_lib.bw_unrepack(_dev(packed, torch.uint8, "packed"), N, K,
                            _dev(canon, torch.uint8, "canon"),
                            _stream(stream)), "bw_unrepack")
    return canon


def bw_quant_weight(W: torch.Tensor, ws_bounds, canon: torch.Tensor | None = None,
                    ws: torch.Tensor | None = None, stream=None):
    """Absmean ternarisation (synchronising): fp32 W [N][K] (device) and row
    segments `ws_bounds` -> (canonical codes uint8 [N][K/4], bf16 ws
    [n_ws]); the codes are the input of bw_repack."""
    N, K = W.shape
    n_ws = len(ws_bounds) - 1
    if canon is None:
        canon = torch.empty((N, K // 4), dtype=torch.uint8, device=W.device)
    if ws is None:
        ws = torch.empty((n_ws,), dtype=torch.bfloat16, device=W.device)
    _need(canon, N * (K // 4), "canon")
    _need(ws, n_ws, "ws")
    _check(_lib.bw_quant_weight(_dev(W, torch.float32, "W"), N, K,
                                _bounds_array(ws_bounds), n_ws,
                                _dev(canon, torch.uint8, "canon"),
                                _dev(ws, torch.bfloat16, "ws"),
                                _stream(stream)), "bw_quant_weight")
    return canon, ws


def _bounds_array(bounds):
    arr = (ctypes.c_int * len(bounds))(*[int(b) for b in bounds])
    return arr


def bw_gemv_w2a8(x: torch.Tensor, packed: torch.Tensor, s: torch.Tensor,
                 ws: torch.Tensor, ws_bounds, N: int, K: int,
                 y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """bf16 y [M][N] = bf16((acc / s[m]) * ws[seg(n)]); ws is bf16 [n_ws],
    ws_bounds a host sequence of n_ws + 1 ints from 0 to N."""
    x2 = x if x.dim() == 2 else x.reshape(1, -1)
    M = x2.shape[0]
    if x2.shape[1] != K:
        raise ValueError("x has the wrong K")
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _need(packed, bw_repack_bytes(N, K), "packed")
    _need(s, M, "s")
    _need(ws, len(ws_bounds) - 1, "ws")
    _need(y, M * N, "y")
    b = _bounds_array(ws_bounds)
    _check(_lib.bw_gemv_w2a8(
        _dev(x2, torch.int8, "x"), _dev(packed, torch.uint8, "packed"),
        _dev(s, torch.float32, "s"), _dev(ws, torch.bfloat16, "ws"),
        ctypes.cast(b, _P), len(ws_bounds) - 1, M, N, K,
        _dev(y, torch.bfloat16, "y"), _stream(stream)), "bw_gemv_w2a8")
    return y


def bw_gemv_w2a8_lut(x: torch.Tensor, packed: torch.Tensor, s: torch.Tensor,
                     ws: torch.Tensor, ws_bounds, N: int, K: int,
                     y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """bw_gemv_w2a8 computed with pre-summed pair tables (same result)."""
    x2 = x if x.dim() == 2 else x.reshape(1, -1)
    M = x2.shape[0]
    if x2.shape[1] != K:
        raise ValueError("x has the wrong K")
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _need(packed, bw_repack_bytes(N, K), "packed")
    _need(s, M, "s")
    _need(ws, len(ws_bounds) - 1, "ws")
    _need(y, M * N, "y")
    b = _bounds_array(ws_bounds)
    _check(_lib.bw_gemv_w2a8_lut(
        _dev(x2, torch.int8, "x"), _dev(packed, torch.uint8, "packed"),
        _dev(s, torch.float32, "s"), _dev(ws, torch.bfloat16, "ws"),
        ctypes.cast(b, _P), len(ws_bounds) - 1, M, N, K,
        _dev(y, torch.bfloat16, "y"), _stream(stream)), "bw_gemv_w2a8_lut")
    return y


def bw_gemv_w2a8_lut_acc(x: torch.Tensor, packed: torch.Tensor, N: int,
                         K: int, acc: torch.Tensor | None = None,
                         stream=None) -> torch.Tensor:
    """Exact int32 acc [M][N] through the pair-table kernel."""
    x2 = x if x.dim() == 2 else x.reshape(1, -1)
    M = x2.shape[0]
    if x2.shape[1] != K:
        raise ValueError("x has the wrong K")
    if acc is None:
        acc = torch.empty((M, N), dtype=torch.int32, device=x.device)
    _need(packed, bw_repack_bytes(N, K), "packed")
    _need(acc, M * N, "acc")
    _check(_lib.bw_gemv_w2a8_lut_acc(
        _dev(x2, torch.int8, "x"), _dev(packed, torch.uint8, "packed"), M, N,
        K, _dev(acc, torch.int32, "acc"), _stream(stream)),
        "bw_gemv_w2a8_lut_acc")
    return acc


def bw_gemv_w2a8_acc(x: torch.Tensor, packed: torch.Tensor, N: int, K: int,
                     acc: torch.Tensor | None = None,
                     stream=None) -> torch.Tensor:
    """Exact int32 acc [M][N] of the same product, no scales."""
    x2 = x if x.dim() == 2 else x.reshape(1, -1)
    M = x2.shape[0]
    if x2.shape[1] != K:
        raise ValueError("x has the wrong K")
    if acc is None:
        acc = torch.empty((M, N), dtype=torch.int32, device=x.device)
    _need(packed, bw_repack_bytes(N, K), "packed")
    _need(acc, M * N, "acc")
    _check(_lib.bw_gemv_w2a8_acc(
        _dev(x2, torch.int8, "x"), _dev(packed, torch.uint8, "packed"), M, N,
        K, _dev(acc, torch.int32, "acc"), _stream(stream)),
        "bw_gemv_w2a8_acc")
    return acc


def bw_gemm_workspace_bytes(M: int, K: int) -> int:
    """Device scratch a prefill product of M tokens needs (0: unsupported)."""
    return int(_lib.bw_gemm_workspace_bytes(M, K))


def _gemm_workspace(workspace, M: int, K: int, device):
    need = bw_gemm_workspace_bytes(M, K)
    if workspace is None:
        workspace = torch.empty((max(need, 1),), dtype=torch.uint8,
                                device=device)
    _need(workspace, need, "workspace")
    return workspace


def bw_gemm_w2a8(x: torch.Tensor, packed: torch.Tensor, s: torch.Tensor,
                 ws: torch.Tensor, ws_bounds, N: int, K: int,
                 y: torch.Tensor | None = None,
                 workspace: torch.Tensor | None = None,
                 stream=None) -> torch.Tensor:
    """The prefill product: the same bf16 y [M][N] as bw_gemv_w2a8, through
    256-token tensor-core tiles; workspace is a uint8 device tensor of at
    least bw_gemm_workspace_bytes(M, K) bytes (allocated if None)."""
    x2 = x if x.dim() == 2 else x.reshape(1, -1)
    M = x2.shape[0]
    if x2.shape[1] != K:
        raise ValueError("x has the wrong K")
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _need(packed, bw_repack_bytes(N, K), "packed")
    _need(s, M, "s")
    _need(ws, len(ws_bounds) - 1, "ws")
    _need(y, M * N, "y")
    workspace = _gemm_workspace(workspace, M, K, x.device)
    b = _bounds_array(ws_bounds)
    _check(_lib.bw_gemm_w2a8(
        _dev(x2, torch.int8, "x"), _dev(packed, torch.uint8, "packed"),
        _dev(s, torch.float32, "s"), _dev(ws, torch.bfloat16, "ws"),
        ctypes.cast(b, _P), len(ws_bounds) - 1, M, N, K,
        _dev(y, torch.bfloat16, "y"), _dev(workspace, torch.uint8, "workspace"),
        workspace.numel(), _stream(stream)), "bw_gemm_w2a8")
    return y


def bw_gemm_w2a8_acc(x: torch.Tensor, packed: torch.Tensor, N: int, K: int,
                     acc: torch.Tensor | None = None,
                     workspace: torch.Tensor | None = None,
                     stream=None) -> torch.Tensor:
    """Exact int32 acc [M][N] through the prefill tiles."""
    x2 = x if x.dim() == 2 else x.reshape(1, -1)
    M = x2.shape[0]
    if x2.shape[1] != K:
        raise ValueError("x has the wrong K")
    if acc is None:
        acc = torch.empty((M, N), dtype=torch.int32, device=x.device)
    _need(packed, bw_repack_bytes(N, K), "packed")
    _need(acc, M * N, "acc")
    workspace = _gemm_workspace(workspace, M, K, x.device)
    _check(_lib.bw_gemm_w2a8_acc(
        _dev(x2, torch.int8, "x"), _dev(packed, torch.uint8, "packed"), M, N,
        K, _dev(acc, torch.int32, "acc"),
        _dev(workspace, torch.uint8, "workspace"), workspace.numel(),
        _stream(stream)), "bw_gemm_w2a8_acc")
    return acc


def bw_attn_workspace_bytes(H: int, Hkv: int, D: int, S: int) -> int:
    """Device scratch bw_attn_decode needs for this shape (0: unsupported)."""
    return int(_lib.bw_attn_workspace_bytes(H, Hkv, D, S))


def bw_attn_decode(qkv: torch.Tensor, pos: torch.Tensor, H: int, Hkv: int,
                   k_cache: torch.Tensor, v_cache: torch.Tensor,
                   theta: float = 500000.0, out: torch.Tensor | None = None,
                   workspace: torch.Tensor | None = None,
                   stream=None) -> torch.Tensor:
    """One grouped-query decode-attention step at position pos[0] (int32
    device tensor): rotates and appends the new key and value (bf16 qkv
    [(H + 2 Hkv) D]) to the bf16 caches [Hkv][S][D] and returns fp32 out
    [H][D].  `workspace` is a uint8 device tensor of at least
    bw_attn_workspace_bytes bytes, zeroed before its first use; if omitted,
    a zeroed one is made for this call."""
    return bw_attn_decode_ex(qkv, pos, H, Hkv, k_cache, v_cache, theta, out,
                             workspace, 0, stream)


def bw_attn_decode_ex(qkv: torch.Tensor, pos: torch.Tensor, H: int,
                      Hkv: int, k_cache: torch.Tensor, v_cache: torch.Tensor,
                      theta: float = 500000.0,
                      out: torch.Tensor | None = None,
                      workspace: torch.Tensor | None = None, flags: int = 0,
                      stream=None) -> torch.Tensor:
    """bw_attn_decode with flags (BW_ATTN_PAST_READY: pos and the cache
    rows before it are final before the preceding launch on the stream
    starts, so the call reads and copies them before its dependency
    wait)."""
    Hkv_, S, D = k_cache.shape
    if Hkv_ != Hkv or tuple(v_cache.shape) != (Hkv, S, D):
        raise ValueError("k_cache and v_cache must be [Hkv][S][D]")
    if out is None:
        out = torch.empty((H, D), dtype=torch.float32, device=qkv.device)
    if workspace is None:
        workspace = torch.zeros((bw_attn_workspace_bytes(H, Hkv, D, S),),
                                dtype=torch.uint8, device=qkv.device)
    _need(qkv, (H + 2 * Hkv) * D, "qkv")
    _need(pos, 1, "pos")
    _need(out, H * D, "out")
    _check(_lib.bw_attn_decode_ex(
        _dev(qkv, torch.bfloat16, "qkv"), _dev(pos, torch.int32, "pos"),
        H, Hkv, D, S, float(theta), _dev(k_cache, torch.bfloat16, "k_cache"),
        _dev(v_cache, torch.bfloat16, "v_cache"),
        _dev(out, torch.float32, "out"),
        _dev(workspace, torch.uint8, "workspace"), workspace.numel(),
        int(flags), _stream(stream)), "bw_attn_decode_ex")
    return out


def bw_device_error(stream=None) -> int:
    """Read and clear the device error word (synchronises the stream).
    Raises BwError(BW_ERR_TIMEOUT) if a bounded device wait ran out."""
    bits = ctypes.c_uint(0)
    status = _lib.bw_device_error(ctypes.byref(bits), _stream(stream))
    if status == 6:
        raise BwError(status, f"bw_device_error (bits {bits.value:#x})")
    _check(status, "bw_device_error")
    return bits.value


class _StackDesc(ctypes.Structure):
    _fields_ = [("n_layers", _I), ("dim", _I), ("ffn", _I), ("n_heads", _I),
                ("n_kv_heads", _I), ("eps", ctypes.c_float),
                ("wqkv", _P), ("wo", _P), ("w13", _P), ("w2", _P),
                ("ws", _P), ("gammas", _P)]


class _StackTrace(ctypes.Structure):
    _fields_ = [("layer", _I)] + [(n, _P) for n in (
        "h_in", "q_attn", "s_attn", "qkv", "q_o", "s_o", "o", "h_mid",
        "q_ffn", "s_ffn", "gu", "q_down", "s_down", "down", "attn")]


class Stack:
    """A decoder layer stack (bw_stack_create / bw_layer_stack).

    layers: list of dicts with device tensors 'wqkv', 'wo', 'w13', 'w2'
    (uint8 device layouts from bw_repack), 'ws' (bf16 [7]) and 'gammas'
    (fp32 [3 dim + ffn]).  The tensors must outlive the stack.
    max_positions > 0 makes a stack with a KV cache of that many positions
    (bw_stack_create_kv, RoPE base theta): consecutive steps are then
    consecutive tokens of one sequence."""

    def __init__(self, layers, dim, ffn, n_heads, n_kv_heads, eps=1e-5,
                 max_positions=0, theta=500000.0):
        self.dim, self.ffn = dim, ffn
        self.n_heads, self.n_kv_heads = n_heads, n_kv_heads
        self.max_positions = max_positions
        self._keep = layers
        L = len(layers)
        self.head_dim = dim // n_heads
        qkv_n = (n_heads + 2 * n_kv_heads) * self.head_dim
        need = {"wqkv": bw_repack_bytes(qkv_n, dim),
                "wo": bw_repack_bytes(dim, dim),
                "w13": bw_repack_bytes(2 * ffn, dim),
                "w2": bw_repack_bytes(dim, ffn), "ws": 7,
                "gammas": 3 * dim + ffn}
        for i, layer in enumerate(layers):
            for key, count in need.items():
                _need(layer[key], count, f"layers[{i}]['{key}']")
        self._trace_sizes = {
            "h_in": dim, "q_attn": dim, "s_attn": 1, "qkv": qkv_n,
            "q_o": dim, "s_o": 1, "o": dim, "h_mid": dim, "q_ffn": dim,
            "s_ffn": 1, "gu": 2 * ffn, "q_down": ffn, "s_down": 1,
            "down": dim, "attn": dim}
        arr = lambda key, dt: (_P * L)(*[_dev(l[key], dt, key)
                                         for l in layers])
        self._arrays = [arr("wqkv", torch.uint8), arr("wo", torch.uint8),
                        arr("w13", torch.uint8), arr("w2", torch.uint8),
                        arr("ws", torch.bfloat16), arr("gammas", torch.float32)]
        desc = _StackDesc(L, dim, ffn, n_heads, n_kv_heads, eps,
                          *[ctypes.cast(a, _P) for a in self._arrays])
        handle = _P()
        if max_positions > 0:
            _check(_lib.bw_stack_create_kv(ctypes.byref(desc), max_positions,
                                           float(theta),
                                           ctypes.byref(handle)),
                   "bw_stack_create_kv")
        else:
            _check(_lib.bw_stack_create(ctypes.byref(desc),
                                        ctypes.byref(handle)),
                   "bw_stack_create")
        self._h = handle

    def read_kv(self, layer: int, stream=None):
        """(keys, values) of one layer's cache: bf16 [Hkv][S][head_dim]
        copies."""
        shape = (self.n_kv_heads, self.max_positions, self.head_dim)
        k = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
        v = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
        _check(_lib.bw_stack_read_kv(self._h, layer, k.data_ptr(),
                                     v.data_ptr(), _stream(stream)),
               "bw_stack_read_kv")
        return k, v

    def reset_kv(self, stream=None):
        """Start a new sequence at position 0."""
        _check(_lib.bw_stack_reset_kv(self._h, _stream(stream)),
               "bw_stack_reset_kv")

    def run(self, h_in: torch.Tensor, h_out: torch.Tensor | None = None,
            trace: dict | None = None, stream=None) -> torch.Tensor:
        """h_in fp32 [steps][dim] -> h_out fp32 [steps][dim].  trace: a dict
        with 'layer' and device tensors named as bw_stack_trace's fields."""
        h2 = h_in if h_in.dim() == 2 else h_in.reshape(1, -1)
        steps = h2.shape[0]
        if h2.shape[1] != self.dim:
            raise ValueError("h_in has the wrong width")
        if h_out is None:
            h_out = torch.empty_like(h2)
        _need(h_out, steps * self.dim, "h_out")
        tr_ptr = None
        if trace is not None:
            tr = _StackTrace(int(trace["layer"]))
            for name, _ in _StackTrace._fields_[1:]:
                t = trace.get(name)
                if t is not None:
                    if not t.is_cuda or not t.is_contiguous():
                        raise ValueError(f"trace['{name}'] must be a "
                                         "contiguous CUDA tensor")
                    _need(t, self._trace_sizes[name], f"trace['{name}']")
                setattr(tr, name, t.data_ptr() if t is not None else None)
            tr_ptr = ctypes.byref(tr)
        _check(_lib.bw_layer_stack(self._h, _dev(h2, torch.float32, "h_in"),
                                   steps, _dev(h_out, torch.float32, "h_out"),
                                   tr_ptr, _stream(stream)), "bw_layer_stack")
        return h_out

    def close(self):
        if getattr(self, "_h", None):
            _lib.bw_stack_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def bw_selftest_wait_timeout(stream=None) -> tuple[int, int]:
    """Run the bounded-wait self-test; returns (status, device error bits).
    The expected result is (6, 8): BW_ERR_TIMEOUT with bit 8."""
    bits = ctypes.c_uint(0)
    status = _lib.bw_selftest_wait_timeout(ctypes.byref(bits), _stream(stream))
    return status, bits.value
