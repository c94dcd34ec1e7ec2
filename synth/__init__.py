"""Seeded synthetic inputs for the W2A8 ternary GEMV path.

Both sides of every parity check (the CUDA library and the CPU oracle) take
their inputs from here, and nothing else is shared between them.  This module
holds none of the method's arithmetic: it only draws random numbers and lays
them out in the input formats that the boundary header documents (canonical
2-bit weight bytes, int8 activations, fp32 rows, bf16 weight scales).

Random numbers: SplitMix64 (Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014) used as a counter-based
generator -- value i of stream t is the SplitMix64 output function applied to
seed + (t * 2^40 + i + 1) * 0x9E3779B97F4A7C15.  Normal variates use the
Box-Muller transform (Box and Muller, 1958).  The output is identical on
every platform for the integer draws; the normal draws go through the host
libm (log, cos) and are generated on the host that runs both sides.

Workload recipe (the BitNet-2B decode shapes of the W2A8 kernel page, §7.1
and §一):
  * weights i.i.d. ternary, P(-1) = P(+1) = 0.325, P(0) = 0.35, drawn from
    16 random bits per weight (thresholds 21299 and 44237 of 65536);
  * int8 activations uniform on [-127, 127];
  * fp32 activation rows i.i.d. N(0, 1);
  * bf16 weight scales uniform on [0.5, 2), one per fused sub-projection,
    cut to bf16 by dropping the low 16 bits of the fp32 draw.
"""
from __future__ import annotations

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_STREAM_SHIFT = 40
_CHUNK = 1 << 22

# Stream ids: one per kind of quantity, so that changing one size does not
# shift another quantity's numbers.
S_WEIGHTS, S_ACT_I8, S_ACT_F32, S_WS, S_GAMMA, S_STEP = 1, 2, 3, 4, 5, 6
S_ATTN = 7


def base_seed(config: int, sub: int = 0) -> int:
    """Seed of a workload: 0xB17E0000 + 16 * config + sub-case."""
    return 0xB17E0000 + 16 * config + sub


def u64(seed: int, stream: int, n: int, offset: int = 0) -> np.ndarray:
    """n SplitMix64 outputs of (seed, stream), starting at counter offset."""
    ctr = (np.arange(offset + 1, offset + n + 1, dtype=np.uint64)
           + np.uint64(stream << _STREAM_SHIFT))
    z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + ctr * _GOLDEN
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def uniform01(seed: int, stream: int, n: int, offset: int = 0) -> np.ndarray:
    """Doubles in [0, 1) with 53 random bits."""
    return (u64(seed, stream, n, offset) >> np.uint64(11)).astype(np.float64) \
        * (1.0 / 9007199254740992.0)


# --------------------------------------------------------------------------
# Weights
# --------------------------------------------------------------------------
T_NEG = 21299   # 0.325 * 65536, rounded
T_ZERO = 44237  # 0.675 * 65536, rounded


def ternary_codes(seed: int, n: int, offset: int = 0,
                  stream: int = S_WEIGHTS) -> np.ndarray:
    """n codes in {0, 1, 2} (code = weight + 1), four 16-bit draws per u64."""
    words = u64(seed, stream, (n + 3) // 4, offset)
    parts = np.stack([(words >> np.uint64(16 * i)) & np.uint64(0xFFFF)
                      for i in range(4)], axis=1).reshape(-1)[:n]
    codes = np.ones(n, np.uint8)
    codes[parts < T_NEG] = 0
    codes[parts >= T_ZERO] = 2
    return codes


def canonical_weights(seed: int, N: int, K: int,
                      stream: int = S_WEIGHTS) -> np.ndarray:
    """Canonical bytes [N][K/4]: weight 4j+t of a row in byte j, bits 2t.."""
    assert K % 4 == 0
    total = N * K
    out = np.empty(total // 4, np.uint8)
    for start in range(0, total, 4 * _CHUNK):
        stop = min(total, start + 4 * _CHUNK)
        codes = ternary_codes(seed, stop - start, start // 4, stream)
        c = codes.reshape(-1, 4).astype(np.uint8)
        out[start // 4: stop // 4] = (c[:, 0] | (c[:, 1] << 2)
                                      | (c[:, 2] << 4) | (c[:, 3] << 6))
    return out.reshape(N, K // 4)


def canonical_from_codes(codes: np.ndarray) -> np.ndarray:
    """Lay out explicit codes [N][K] in {0,1,2,3} as canonical bytes."""
    c = np.ascontiguousarray(codes, np.uint8)
    N, K = c.shape
    c = c.reshape(N, K // 4, 4)
    return (c[..., 0] | (c[..., 1] << 2) | (c[..., 2] << 4)
            | (c[..., 3] << 6)).astype(np.uint8)


# --------------------------------------------------------------------------
# Activations and scales
# --------------------------------------------------------------------------
def int8_uniform(seed: int, n: int, lo: int = -127, hi: int = 127,
                 stream: int = S_ACT_I8) -> np.ndarray:
    """n int8 values uniform on [lo, hi] (multiply-shift range reduction)."""
    span = np.uint64(hi - lo + 1)
    z = u64(seed, stream, n) >> np.uint64(32)
    offsets = ((z * span) >> np.uint64(32)).astype(np.int64)
    return (offsets + lo).astype(np.int8)


def normal_f32(seed: int, n: int, stream: int = S_ACT_F32,
               offset: int = 0) -> np.ndarray:
    """n fp32 N(0,1) values (Box-Muller, cosine branch)."""
    u = uniform01(seed, stream, 2 * n, 2 * offset).reshape(n, 2)
    u1 = 1.0 - u[:, 0]                       # (0, 1]
    r = np.sqrt(-2.0 * np.log(u1))
    return (r * np.cos(2.0 * np.pi * u[:, 1])).astype(np.float32)


def bf16_uniform(seed: int, n: int, lo: float = 0.5, hi: float = 2.0,
                 stream: int = S_WS) -> np.ndarray:
    """n bf16 bit patterns uniform on [lo, hi): fp32 draw, low 16 bits cut."""
    v = (lo + (hi - lo) * uniform01(seed, stream, n)).astype(np.float32)
    return (v.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, np.uint32) << np.uint32(16)).view(np.float32)


def bf16_normal(seed: int, n: int, stream: int = S_ATTN,
                offset: int = 0) -> np.ndarray:
    """n bf16 bit patterns of N(0,1) draws: fp32 draw, low 16 bits cut."""
    v = normal_f32(seed, n, stream, offset)
    return (v.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


# --------------------------------------------------------------------------
# Workloads
# --------------------------------------------------------------------------
# Fused sub-projection boundaries of the BitNet-2B decoder (dim 2560,
# 20 query heads and 5 KV heads of 128, ffn 6912).
DECODE_SHAPES = {
    "wqkv": (3840, 2560, [0, 2560, 3200, 3840]),
    "wo": (2560, 2560, [0, 2560]),
    "w13": (13824, 2560, [0, 6912, 13824]),
    "w2": (2560, 6912, [0, 2560]),
}


def gemv_case(M: int, N: int, K: int, seed: int, bounds=None,
              uniform_x: bool = True) -> dict:
    """One GEMV workload.

    canon  uint8 [N][K/4]  canonical ternary weights
    q      int8  [M][K]    uniform int8 activations (if uniform_x)
    xf     fp32  [M][K]    N(0,1) rows (their absmax gives the scales s)
    ws     uint16 [n_ws]   bf16 weight scales, one per segment
    bounds int32 [n_ws+1]  segment boundaries over N
    """
    if bounds is None:
        bounds = [0, N]
    bounds = np.asarray(bounds, np.int32)
    case = {
        "M": M, "N": N, "K": K, "seed": seed,
        "canon": canonical_weights(seed, N, K),
        "xf": normal_f32(seed, M * K).reshape(M, K),
        "ws": bf16_uniform(seed, len(bounds) - 1),
        "bounds": bounds,
    }
    if uniform_x:
        case["q"] = int8_uniform(seed, M * K).reshape(M, K)
    return case


def stack_weights(seed: int, n_layers: int, dim: int = 2560,
                  ffn: int = 6912, n_heads: int = 20, n_kv: int = 5,
                  gamma_one: bool = True) -> dict:
    """Random ternary weights of a BitNet-shaped decoder stack.

    Per layer: wqkv [(n_heads+2 n_kv) hd][dim/4], wo [dim][dim/4],
    w13 [2 ffn][dim/4], w2 [dim][ffn/4]; 7 bf16 scales (q, k, v, o, gate,
    up, down); 4 RMSNorm gains (dim, dim, dim, ffn), all ones unless
    gamma_one is False (then uniform on [0.9, 1.1]).
    """
    hd = dim // n_heads
    qkv_n = (n_heads + 2 * n_kv) * hd
    layers = []
    for l in range(n_layers):
        s = seed + 0x1000 * (l + 1)
        g_len = 3 * dim + ffn
        if gamma_one:
            gam = np.ones(g_len, np.float32)
        else:
            gam = (0.9 + 0.2 * uniform01(s, S_GAMMA, g_len)).astype(np.float32)
        layers.append({
            "wqkv": canonical_weights(s, qkv_n, dim, stream=11),
            "wo": canonical_weights(s, dim, dim, stream=12),
            "w13": canonical_weights(s, 2 * ffn, dim, stream=13),
            "w2": canonical_weights(s, dim, ffn, stream=14),
            "ws": bf16_uniform(s, 7),
            "gammas": gam,
        })
    return {"dim": dim, "ffn": ffn, "n_heads": n_heads, "n_kv": n_kv,
            "eps": 1e-5, "layers": layers,
            "bounds": {"wqkv": [0, n_heads * hd, (n_heads + n_kv) * hd, qkv_n],
                       "wo": [0, dim], "w13": [0, ffn, 2 * ffn],
                       "w2": [0, dim]}}


def step_inputs(seed: int, steps: int, dim: int) -> np.ndarray:
    """fp32 N(0,1) decoder inputs [steps][dim], one per decode step."""
    return normal_f32(seed, steps * dim, stream=S_STEP).reshape(steps, dim)


def attn_case(seed: int, H: int, Hkv: int, D: int, S: int, p: int) -> dict:
    """One decode-attention step: the fused q | k | v vector of the token
    (bf16 [(H + 2 Hkv) D]) and a full KV cache (bf16 [Hkv][S][D] each),
    every value an N(0,1) draw cut to bf16.  Rows p.. of the cache hold
    draws too: the step must ignore them and overwrite row p only."""
    nq = (H + 2 * Hkv) * D
    nc = Hkv * S * D
    return {
        "H": H, "Hkv": Hkv, "D": D, "S": S, "p": p, "seed": seed,
        "qkv": bf16_normal(seed, nq),
        "kc": bf16_normal(seed, nc, offset=nq).reshape(Hkv, S, D),
        "vc": bf16_normal(seed, nc, offset=nq + nc).reshape(Hkv, S, D),
    }
