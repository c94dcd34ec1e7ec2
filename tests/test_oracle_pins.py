"""Pins of the CPU oracle to facts fixed by the pages and by mathematics.

Each test checks the oracle against something other than itself: values the
W2A8 kernel page prints (the word interleave of §5.2), hand-worked values of
the formats and formulas (§5.2, §5.3, §六 item 3), closed forms (all-ones,
one-hot, zero weights), brute force over every ternary row of tiny K, exact
rational arithmetic, and invariants (round trips, bijectivity, ties to even).
A plausible slip in the oracle -- a dropped term, a flipped sign, an index
off by one, multiplying by s instead of dividing -- fails at least one.
"""
import itertools
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth
from conftest import read_golden

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def f32(x):
    return float(np.float32(x))


def bits_f32(h):
    return float(synth.bf16_bits_to_f32(np.array([h], np.uint16))[0])


# ---------------------------------------------------------------- packing
def test_canonical_bytes_golden():
    for line in read_golden("canonical_bytes.txt"):
        *w, byte = line.split()
        w = np.array([[int(v) for v in w]], np.int8)
        assert oracle.pack(w)[0, 0] == int(byte, 16), line
        assert (oracle.unpack(np.array([[int(byte, 16)]], np.uint8), 1, 4)
                == w).all(), line


def test_all_valid_bytes_round_trip_and_code3_rejected():
    valid = 0
    for b in range(256):
        codes = [(b >> (2 * t)) & 3 for t in range(4)]
        canon = np.array([[b]], np.uint8)
        if 3 in codes:
            with pytest.raises(oracle.OracleError):
                oracle.unpack(canon, 1, 4)
            continue
        valid += 1
        w = oracle.unpack(canon, 1, 4)
        assert list(w[0]) == [c - 1 for c in codes]
        assert oracle.pack(w)[0, 0] == b
    assert valid == 81


def test_random_round_trip():
    canon = synth.canonical_weights(5, 37, 128)
    w = oracle.unpack(canon, 37, 128)
    assert set(np.unique(w)) <= {-1, 0, 1}
    assert (oracle.pack(w) == canon).all()


# ----------------------------------------------------------- dot product
def _rows_all_ternary(K):
    return np.array(list(itertools.product((-1, 0, 1), repeat=K)), np.int8)


@pytest.mark.parametrize("K", [4, 8])
def test_brute_force_every_ternary_row(K):
    W = _rows_all_ternary(K)              # 3^K rows
    x = synth.int8_uniform(K, K, lo=-128, hi=127).reshape(1, K)
    canon = oracle.pack(W)
    acc = oracle.gemv_acc(x, canon, W.shape[0], K)[0]
    direct = [sum(int(W[n, k]) * int(x[0, k]) for k in range(K))
              for n in range(W.shape[0])]
    assert list(acc) == direct


def test_closed_forms():
    M, N, K = 3, 5, 96
    x = synth.int8_uniform(11, M * K, lo=-128, hi=127).reshape(M, K)
    rowsum = x.astype(np.int64).sum(axis=1)
    plus = oracle.pack(np.ones((N, K), np.int8))
    minus = oracle.pack(-np.ones((N, K), np.int8))
    zero = oracle.pack(np.zeros((N, K), np.int8))
    assert (oracle.gemv_acc(x, plus, N, K) == rowsum[:, None]).all()
    assert (oracle.gemv_acc(x, minus, N, K) == -rowsum[:, None]).all()
    assert (oracle.gemv_acc(x, zero, N, K) == 0).all()
    # one-hot row n picks column j = 7n + 3
    W = np.zeros((N, K), np.int8)
    for n in range(N):
        W[n, 7 * n + 3] = 1
    acc = oracle.gemv_acc(x, oracle.pack(W), N, K)
    for n in range(N):
        assert (acc[:, n] == x[:, 7 * n + 3]).all()
    W[2, 50] = -1
    acc = oracle.gemv_acc(x, oracle.pack(W), N, K)
    assert (acc[:, 2] == x[:, 17].astype(np.int64) - x[:, 50]).all()


def test_linearity_disjoint_supports():
    N, K = 9, 256
    codes = synth.ternary_codes(3, N * K).reshape(N, K)
    W = codes.astype(np.int8) - 1
    mask = (synth.ternary_codes(4, N * K).reshape(N, K) == 0)
    W1 = np.where(mask, W, 0).astype(np.int8)
    W2 = np.where(mask, 0, W).astype(np.int8)
    x = synth.int8_uniform(6, 2 * K).reshape(2, K)
    a = oracle.gemv_acc(x, oracle.pack(W), N, K)
    a1 = oracle.gemv_acc(x, oracle.pack(W1), N, K)
    a2 = oracle.gemv_acc(x, oracle.pack(W2), N, K)
    assert (a == a1 + a2).all()
    # sign: negating W negates acc
    assert (oracle.gemv_acc(x, oracle.pack(-W), N, K) == -a).all()


def test_extremes_no_overflow():
    K = 6912
    plus = oracle.pack(np.ones((1, K), np.int8))
    hi = np.full((1, K), 127, np.int8)
    lo = np.full((1, K), -128, np.int8)
    assert oracle.gemv_acc(hi, plus, 1, K)[0, 0] == 127 * K
    assert oracle.gemv_acc(lo, plus, 1, K)[0, 0] == -128 * K


def test_code3_rejected_by_gemv_and_layout():
    canon = np.full((1, 4), 0x55, np.uint8)
    canon[0, 2] = 0x57        # weight 8 gets code 3
    x = np.ones((1, 16), np.int8)
    with pytest.raises(oracle.OracleError):
        oracle.gemv_acc(x, canon, 1, 16)
    with pytest.raises(oracle.OracleError):
        oracle.layout(canon, 1, 16)


# --------------------------------------------------------------- bf16/epilogue
def test_bf16_rne_matches_torch_cast():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(0)
    v = np.concatenate([
        rng.standard_normal(400_000).astype(np.float32) * 1e3,
        rng.standard_normal(300_000).astype(np.float32) * 1e-30,
        # exact ties: low 16 bits == 0x8000
        ((rng.integers(0, 2**31, 300_000, dtype=np.uint64).astype(np.uint32)
          & np.uint32(0xFFFF0000)) | np.uint32(0x8000)).view(np.float32),
    ])
    v = v[np.isfinite(v)]
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy() \
        .astype(np.uint16)
    lib = oracle._load()
    got = np.array([lib.or_bf16_rne(float(f)) for f in v], np.uint16)
    assert (got == ref).all()


def test_epilogue_golden():
    K = 4
    for line in read_golden("epilogue.txt"):
        acc_s, s_s, ws_s, y_s = line.split()
        acc, s, ws = int(acc_s), float(s_s), float(ws_s)
        ws_bits = oracle.bf16_rne(ws)
        assert bits_f32(ws_bits) == ws
        # realise acc with one weight row against a crafted x
        x = np.zeros((1, K), np.int8)
        W = np.zeros((1, K), np.int8)
        rem, k = acc, 0
        while rem != 0:
            step = max(-127, min(127, rem))
            x[0, k], W[0, k] = abs(step), 1 if step > 0 else -1
            rem -= step
            k += 1
            if k == K:
                x = np.concatenate([x, np.zeros((1, 4), np.int8)], axis=1)
                W = np.concatenate([W, np.zeros((1, 4), np.int8)], axis=1)
                K += 4
        canon = oracle.pack(W)
        assert oracle.gemv_acc(x, canon, 1, x.shape[1])[0, 0] == acc
        y = oracle.gemv(x, canon, [s], [ws_bits], [0, 1], 1, x.shape[1])
        assert y[0, 0] == int(y_s, 16), line
        K = 4


def test_epilogue_exact_rational_bound():
    """y must be the bf16 rounding of a value within fp32 error of the exact
    rational acc/s*ws: |y - exact| <= 1/2 ulp_bf16 + 2^-22 relative."""
    case = synth.gemv_case(1, 512, 256, 21, bounds=[0, 100, 512])
    q, canon = case["q"], case["canon"]
    _, s = oracle.quant_act(case["xf"])
    acc = oracle.gemv_acc(q, canon, 512, 256)[0]
    y = oracle.gemv(q, canon, s, case["ws"], case["bounds"], 512, 256)[0]
    ws = synth.bf16_bits_to_f32(case["ws"])
    for n in range(512):
        wsn = Fraction(float(ws[0 if n < 100 else 1]))
        exact = Fraction(int(acc[n])) / Fraction(float(s[0])) * wsn
        got = Fraction(bits_f32(y[n]))
        if exact == 0:
            assert got == 0
            continue
        e = abs(exact)
        ulp = Fraction(2) ** (int(np.floor(np.log2(float(e)))) - 7)
        assert abs(got - exact) <= ulp / 2 + e * Fraction(1, 2**22), n
        assert (got > 0) == (exact > 0)


def test_epilogue_segments():
    N, K = 12, 64
    W = np.ones((N, K), np.int8)
    x = np.ones((1, K), np.int8)
    ws = [oracle.bf16_rne(v) for v in (1.0, 2.0, 0.5)]
    y = oracle.gemv(x, oracle.pack(W), [1.0], ws, [0, 3, 10, 12], N, K)[0]
    vals = [bits_f32(h) for h in y]
    assert vals == [64.0] * 3 + [128.0] * 7 + [32.0] * 2
    with pytest.raises(oracle.OracleError):
        oracle.gemv(x, oracle.pack(W), [1.0], ws, [0, 3, 3, 12], N, K)
    with pytest.raises(oracle.OracleError):
        oracle.gemv(x, oracle.pack(W), [1.0], ws, [0, 3, 10, 11], N, K)


def test_zero_weights_give_positive_zero():
    K = 64
    canon = oracle.pack(np.zeros((4, K), np.int8))
    x = synth.int8_uniform(1, K).reshape(1, K)
    y = oracle.gemv(x, canon, [3.0], [oracle.bf16_rne(1.5)], [0, 4], 4, K)
    assert (y == 0).all()


# --------------------------------------------------------------- quant_act
def test_quant_act_golden():
    for line in read_golden("quant_act.txt"):
        xs, ss, qs = [p.split() for p in line.split("|")]
        x = np.array([float(v) for v in xs], np.float32)
        q, s = oracle.quant_act(x)
        assert s[0] == np.float32(float(ss[0])), line
        assert list(q[0]) == [int(v) for v in qs], line


def test_quant_act_invariants():
    x = synth.normal_f32(9, 8 * 2560).reshape(8, 2560)
    q, s = oracle.quant_act(x)
    for m in range(8):
        j = int(np.argmax(np.abs(x[m])))
        assert abs(int(q[m, j])) == 127
        assert int(q[m, j]) * x[m, j] > 0
        assert np.abs(q[m].astype(np.int32)).max() == 127
        nz = x[m] != 0
        assert (np.sign(q[m][nz & (q[m] != 0)])
                == np.sign(x[m][nz & (q[m] != 0)])).all()
        assert s[m] == np.float32(127) / np.float32(np.abs(x[m]).max())
    # scaling a row by a power of two leaves q unchanged
    q2, s2 = oracle.quant_act(x * np.float32(4))
    assert (q2 == q).all() and np.allclose(s2 * 4, s, rtol=0, atol=0)


# --------------------------------------------------------------- layout
def test_layout_word_interleave_golden():
    g = {ln.split()[0]: [int(v) for v in ln.split()[1:]]
         for ln in read_golden("word_interleave.txt")}
    pattern, shift = g["pattern"], g["shift"]
    # the pattern and the shift table describe the same map
    for f, e in enumerate(pattern):
        if e < len(shift):
            assert shift[e] == 2 * f
    N, K = 8, 64
    for e in range(16):
        for t in range(4):
            codes = np.ones((N, K), np.uint8)
            codes[0, 16 * t + e] = 2
            dev = oracle.layout(synth.canonical_from_codes(codes), N, K)
            word = int(dev[4 * t: 4 * t + 4].view(np.uint32)[0])
            f = pattern.index(e)
            neutral = 0x55555555
            assert word == (neutral & ~(3 << 2 * f)) | (2 << 2 * f), (e, t)
            if e < len(shift):
                assert word == (neutral & ~(3 << shift[e])) | (2 << shift[e])


def test_layout_is_a_bijection_and_pads_with_zero_weights():
    N, K = 16, 128
    size = oracle.layout_bytes(N, K)
    assert size == N * K // 4
    seen = set()
    for n in range(N):
        for k in range(K):
            codes = np.ones((N, K), np.uint8)
            codes[n, k] = 0
            dev = oracle.layout(synth.canonical_from_codes(codes), N, K)
            fields = np.unpackbits(dev[:, None], axis=1, bitorder="little")
            pairs = fields.reshape(-1, 2)
            where = np.nonzero((pairs[:, 0] == 0) & (pairs[:, 1] == 0))[0]
            assert len(where) == 1
            seen.add(int(where[0]))
            # 128-byte segments hold 8 rows x 64 weights of one chunk
            seg = int(where[0]) * 2 // 8 // 128
            assert seg == (n // 8) * (K // 64) + k // 64
    assert len(seen) == N * K
    # ragged: N=5, K=68 pads to 8 rows and 128 columns with code 1
    canon = synth.canonical_weights(2, 5, 68)
    dev = oracle.layout(canon, 5, 68)
    assert dev.size == oracle.layout_bytes(5, 68) == 8 * 128 // 4
    fields = np.unpackbits(dev[:, None], axis=1, bitorder="little") \
        .reshape(-1, 2)
    codes = fields[:, 0] + 2 * fields[:, 1]
    assert (codes == 1).sum() >= 8 * 128 - 5 * 68
    assert (codes != 3).all()
    w = oracle.unpack(canon, 5, 68)
    assert sorted(codes.tolist()) == sorted(
        (w.reshape(-1) + 1).tolist() + [1] * (8 * 128 - 5 * 68))


# ------------------------------------------------------------ stack glue
def test_rmsnorm_closed_forms():
    x = np.array([3.0, 4.0], np.float32)
    out = oracle.rmsnorm(x, np.ones(2, np.float32), 0.0)
    r = 1.0 / np.sqrt(12.5)
    assert np.allclose(out, [3 * r, 4 * r], rtol=1e-7, atol=0)
    c = np.full(64, -2.5, np.float32)
    out = oracle.rmsnorm(c, np.ones(64, np.float32), 1e-5)
    assert np.allclose(out, -2.5 / np.sqrt(6.25 + 1e-5), rtol=1e-7)
    x = synth.normal_f32(3, 2560)
    g = np.linspace(0.5, 1.5, 2560).astype(np.float32)
    out = oracle.rmsnorm(x, g, 1e-5)
    ms = float(np.mean(x.astype(np.float64) ** 2))
    # mean square of x*r equals ms / (ms + eps); gamma multiplies elementwise
    assert np.isclose(np.mean((out.astype(np.float64) / g) ** 2),
                      ms / (ms + 1e-5), rtol=1e-6)
    assert (oracle.rmsnorm(np.zeros(8, np.float32),
                           np.ones(8, np.float32), 1e-5) == 0).all()


def test_relu2_gate_hand_values():
    gate = [-1.0, 0.0, 2.0, 3.0]
    up = [5.0, 5.0, 0.5, -1.0]
    bits = np.array([oracle.bf16_rne(v) for v in gate + up], np.uint16)
    assert list(oracle.relu2_gate(bits)) == [0.0, 0.0, 2.0, -9.0]


def test_attention_one_token_maps_heads_to_kv_groups():
    n_heads, n_kv, hd = 4, 2, 2
    qkv = [0.0] * (n_heads * hd) + [0.0] * (n_kv * hd) + [1.0, 2.0, 3.0, 4.0]
    bits = np.array([oracle.bf16_rne(v) for v in qkv], np.uint16)
    out = oracle.attn_one_token(bits, n_heads, n_kv, hd)
    assert list(out) == [1.0, 2.0, 1.0, 2.0, 3.0, 4.0, 3.0, 4.0]


def _tiny_stack(zero: bool, seed=8):
    dim, ffn, nh, nkv = 64, 128, 4, 2
    hd = dim // nh
    shapes = {"wqkv": ((nh + 2 * nkv) * hd, dim), "wo": (dim, dim),
              "w13": (2 * ffn, dim), "w2": (dim, ffn)}
    mats = {}
    for i, (name, (n, k)) in enumerate(shapes.items()):
        if zero:
            mats[name] = oracle.pack(np.zeros((n, k), np.int8))
        else:
            mats[name] = synth.canonical_weights(seed + i, n, k)
    ws = synth.bf16_uniform(seed, 7)
    gam = np.ones(3 * dim + ffn, np.float32)
    return dim, ffn, nh, nkv, mats, ws, gam


def test_layer_with_zero_weights_is_identity():
    dim, ffn, nh, nkv, mats, ws, gam = _tiny_stack(zero=True)
    h = synth.normal_f32(4, dim)
    out = oracle.layer(h, dim, ffn, nh, nkv, 1e-5, mats["wqkv"], mats["wo"],
                       mats["w13"], mats["w2"], ws, gam)
    assert (out == h).all()


def test_layer_matches_stagewise_composition():
    """The fused layer equals its stages run one by one (order of the block:
    attn_norm, wqkv, attention, attn_sub_norm, wo, residual, ffn_norm, w13,
    relu^2 gate, ffn_sub_norm, w2, residual)."""
    dim, ffn, nh, nkv, mats, ws, gam = _tiny_stack(zero=False)
    hd = dim // nh
    qkv_n = (nh + 2 * nkv) * hd
    h = synth.normal_f32(5, dim)
    one = np.ones(max(dim, ffn), np.float32)

    def nqg(v, canon, n_out, k, w_bits, bounds):
        normed = oracle.rmsnorm(v, one[:k], 1e-5)
        q, s = oracle.quant_act(normed)
        return oracle.gemv(q, canon, s, w_bits, bounds, n_out, k)[0]

    y = nqg(h, mats["wqkv"], qkv_n, dim, ws[0:3],
            [0, nh * hd, (nh + nkv) * hd, qkv_n])
    att = oracle.attn_one_token(y, nh, nkv, hd)
    o = nqg(att, mats["wo"], dim, dim, ws[3:4], [0, dim])
    h1 = (h + synth.bf16_bits_to_f32(o)).astype(np.float32)
    gu = nqg(h1, mats["w13"], 2 * ffn, dim, ws[4:6], [0, ffn, 2 * ffn])
    g = oracle.relu2_gate(gu)
    d = nqg(g, mats["w2"], dim, ffn, ws[6:7], [0, dim])
    h2 = (h1 + synth.bf16_bits_to_f32(d)).astype(np.float32)
    out = oracle.layer(h, dim, ffn, nh, nkv, 1e-5, mats["wqkv"], mats["wo"],
                       mats["w13"], mats["w2"], ws, gam)
    assert (out == h2).all()
    assert not (out == h).all()


def _tiny_cache(seed, nkv, S, hd):
    c = synth.attn_case(seed, 1, 1, hd, S * nkv, 0)
    return (c["kc"].reshape(nkv, S, hd).copy(),
            c["vc"].reshape(nkv, S, hd).copy())


def test_layer_kv_at_position_zero_is_the_one_token_layer():
    """At p = 0 the attention over the cache returns the value heads
    exactly, so the layer equals the one-token layer bit for bit."""
    dim, ffn, nh, nkv, mats, ws, gam = _tiny_stack(zero=False)
    h = synth.normal_f32(6, dim)
    kc, vc = _tiny_cache(synth.base_seed(23), nkv, 8, dim // nh)
    want = oracle.layer(h, dim, ffn, nh, nkv, 1e-5, mats["wqkv"], mats["wo"],
                        mats["w13"], mats["w2"], ws, gam)
    got, kc2, vc2 = oracle.layer_kv(h, dim, ffn, nh, nkv, 1e-5, mats["wqkv"],
                                    mats["wo"], mats["w13"], mats["w2"], ws,
                                    gam, kc, vc, 0, 10000.0)
    assert (got == want).all()
    assert (kc2[:, 1:] == kc[:, 1:]).all() and (vc2[:, 1:] == vc[:, 1:]).all()


def test_layer_kv_matches_stagewise_composition():
    """The layer with a cache equals its stages run one by one, with the
    decode attention (append + attention over rows 0..p) after wqkv."""
    dim, ffn, nh, nkv, mats, ws, gam = _tiny_stack(zero=False)
    hd = dim // nh
    qkv_n = (nh + 2 * nkv) * hd
    h = synth.normal_f32(7, dim)
    kc, vc = _tiny_cache(synth.base_seed(23, 1), nkv, 8, hd)
    p, theta = 5, 500000.0
    one = np.ones(max(dim, ffn), np.float32)

    def nqg(v, canon, n_out, k, w_bits, bounds):
        normed = oracle.rmsnorm(v, one[:k], 1e-5)
        q, s = oracle.quant_act(normed)
        return oracle.gemv(q, canon, s, w_bits, bounds, n_out, k)[0]

    y = nqg(h, mats["wqkv"], qkv_n, dim, ws[0:3],
            [0, nh * hd, (nh + nkv) * hd, qkv_n])
    att, kc_s, vc_s = oracle.attn_decode(y, nh, nkv, hd, p, theta, kc, vc)
    att = att.reshape(-1).astype(np.float32)
    o = nqg(att, mats["wo"], dim, dim, ws[3:4], [0, dim])
    h1 = (h + synth.bf16_bits_to_f32(o)).astype(np.float32)
    gu = nqg(h1, mats["w13"], 2 * ffn, dim, ws[4:6], [0, ffn, 2 * ffn])
    g = oracle.relu2_gate(gu)
    d = nqg(g, mats["w2"], dim, ffn, ws[6:7], [0, dim])
    h2 = (h1 + synth.bf16_bits_to_f32(d)).astype(np.float32)
    out, kc2, vc2 = oracle.layer_kv(h, dim, ffn, nh, nkv, 1e-5, mats["wqkv"],
                                    mats["wo"], mats["w13"], mats["w2"], ws,
                                    gam, kc, vc, p, theta)
    assert (out == h2).all()
    assert (kc2 == kc_s).all() and (vc2 == vc_s).all()


def test_layer_kv_ignores_rows_past_p():
    dim, ffn, nh, nkv, mats, ws, gam = _tiny_stack(zero=False)
    hd = dim // nh
    h = synth.normal_f32(8, dim)
    kc, vc = _tiny_cache(synth.base_seed(23, 2), nkv, 8, hd)
    args = (dim, ffn, nh, nkv, 1e-5, mats["wqkv"], mats["wo"], mats["w13"],
            mats["w2"], ws, gam)
    base, _, _ = oracle.layer_kv(h, *args, kc, vc, 3, 10000.0)
    kc_late, vc_late = kc.copy(), vc.copy()
    kc_late[:, 4:] ^= 0x1234                 # rows past p: ignored
    vc_late[:, 4:] ^= 0x0101
    late, _, _ = oracle.layer_kv(h, *args, kc_late, vc_late, 3, 10000.0)
    assert (late == base).all()


def _hand_layer():
    """The hand-worked layer of tests/golden/layer_hand.txt as a dict of
    float arrays (matrices as [rows][cols] lists of weights)."""
    out = {}
    for line in read_golden("layer_hand.txt"):
        key, val = (t.strip() for t in line.split("=", 1))
        if "|" in val:
            out[key] = np.array([[float(v) for v in row.split()]
                                 for row in val.split("|")])
        else:
            out[key] = np.array([float(v) for v in val.split()])
    return out


def _exact_bf16(values):
    """bf16 bit patterns of values that bf16 holds exactly (the pattern is
    the high half of the fp32 pattern; checked, no rounding involved)."""
    f = np.asarray(values, np.float32)
    u = f.view(np.uint32)
    assert ((u & 0xFFFF) == 0).all(), values
    return (u >> 16).astype(np.uint16)


def _hand_args(G, case):
    dim, ffn, nh, nkv = (int(v) for v in G[case + ".shape"])
    mats = [oracle.pack(G[case.replace("B", "A") + "." + name]
                        .astype(np.int8))
            for name in ("wqkv", "wo", "w13", "w2")]
    ws = _exact_bf16(G["A.ws"])
    gam = G["A.gammas"].astype(np.float32)
    return dim, ffn, nh, nkv, mats, ws, gam


def test_layer_hand_worked_one_token():
    """h_out of the hand-worked layer (one-token attention), exactly; the
    golden file derives every stage from the block order of the W2A8 page's
    §4.1.  A swapped gain slice, weight-scale offset, query-to-KV head map
    or a dropped residual changes the result."""
    G = _hand_layer()
    dim, ffn, nh, nkv, mats, ws, gam = _hand_args(G, "A")
    h = G["A.h"].astype(np.float32)
    out = oracle.layer(h, dim, ffn, nh, nkv, float(G["A.eps"][0]), *mats, ws,
                       gam)
    assert (out == G["A.h_out"].astype(np.float32)).all(), out


def test_layer_hand_worked_stages():
    """The stage functions reproduce each hand-derived intermediate of the
    golden layer from the previous one (teacher forced)."""
    G = _hand_layer()
    dim, ffn, nh, nkv, mats, ws, gam = _hand_args(G, "A")
    eps = float(G["A.eps"][0])
    hd = dim // nh
    qkv_n = (nh + 2 * nkv) * hd

    def nqg(v, g, canon, n_out, k, w_bits, bounds):
        q, s = oracle.quant_act(oracle.rmsnorm(v, g, eps))
        return oracle.gemv(q, canon, s, w_bits, bounds, n_out, k)[0]

    f = lambda bits: synth.bf16_bits_to_f32(bits)
    qkv = nqg(G["A.h"], gam[:dim], mats[0], qkv_n, dim, ws[0:3],
              [0, nh * hd, (nh + nkv) * hd, qkv_n])
    assert (f(qkv) == [0, 0, 0, 0, 0, 0, -1.5, 1.5]).all(), f(qkv)
    att = oracle.attn_one_token(qkv, nh, nkv, hd)
    assert (att == G["A.attn"]).all()
    o = nqg(G["A.attn"], gam[dim:2 * dim], mats[1], dim, dim, ws[3:4],
            [0, dim])
    assert (f(o) == G["A.o"]).all()
    gu = nqg(G["A.h_mid"], gam[2 * dim:3 * dim], mats[2], 2 * ffn, dim,
             ws[4:6], [0, ffn, 2 * ffn])
    assert (oracle.relu2_gate(gu) == G["A.gated"]).all()
    d = nqg(G["A.gated"], gam[3 * dim:], mats[3], dim, ffn, ws[6:7],
            [0, dim])
    assert (f(d) == G["A.down"]).all()


def test_layer_kv_hand_worked():
    """The hand-worked layer with attention over a KV cache at p = 1: the
    queries are zero, so the softmax over rows 0..1 is uniform; the new
    token's value and (rotated, zero) key are appended at row 1 and rows 2
    and 3, past the context, are neither read nor written."""
    G = _hand_layer()
    dim, ffn, nh, nkv, mats, ws, gam = _hand_args(G, "B")
    hd = dim // nh
    S, p = int(G["B.S"][0]), int(G["B.p"][0])
    kc = _exact_bf16(G["B.k_cache"]).reshape(nkv, S, hd)
    vc = _exact_bf16(G["B.v_cache"]).reshape(nkv, S, hd)
    h = G["B.h"].astype(np.float32)
    out, kc2, vc2 = oracle.layer_kv(h, dim, ffn, nh, nkv,
                                    float(G["B.eps"][0]), *mats, ws, gam,
                                    kc, vc, p, float(G["B.theta"][0]))
    assert (out == G["B.h_out"].astype(np.float32)).all(), out
    assert (synth.bf16_bits_to_f32(kc2[0, p]) == G["B.k_row1"]).all()
    assert (vc2[0, p] == _exact_bf16(G["B.v_row1"])).all()
    rows = [j for j in range(S) if j != p]
    assert (kc2[:, rows] == kc[:, rows]).all()
    assert (vc2[:, rows] == vc[:, rows]).all()
    # the attention stage alone on the appended cache
    qkv = _exact_bf16([0, 0, 0, 0, 0, 0, -1.5, 1.5])
    att = oracle.attn_over_cache(qkv, nh, nkv, hd, p, float(G["B.theta"][0]),
                                 kc2, vc2)
    assert (att.reshape(-1) == G["B.attn"]).all()


# --------------------------------------------- absmean weight ternarisation
# [W2A8] §4.2: s = 1 / max(mean|W|, 1e-5), w = clamp(round(W s), -1, 1),
# ws = bf16(1 / s), one scale per weight-scale segment.

def test_quant_weight_constant_matrices():
    # W = c everywhere: mean = |c|, W s = sign(c), ws = c for a power of 2.
    for c, code, ws_bits in [(0.5, 2, 0x3F00), (-0.25, 0, 0x3E80),
                             (2.0, 2, 0x4000)]:
        W = np.full((3, 8), c, np.float32)
        canon, ws = oracle.quant_weight(W, [0, 3])
        assert (oracle.unpack(canon, 3, 8) == code - 1).all()
        assert ws.tolist() == [ws_bits]


def test_quant_weight_ties_to_even_and_clamp():
    # mean |W| = 1 exactly, so s = 1: round(0.5) = 0, round(1.5) = 2 -> 1,
    # round(-0.5) = -0 -> 0, round(-1.5) = -2 -> -1, round(2.5) = 2 -> 1.
    # sum |W| = 4 + 4 + (2.5 + 0 + 0.5 + 1) = 12 over 12 elements
    W = np.array([[0.5, 1.5, -0.5, -1.5], [0.5, 1.5, -0.5, -1.5],
                  [2.5, 0.0, -0.5, -1.0]], np.float32)
    assert float(np.abs(W).mean()) == 1.0
    canon, ws = oracle.quant_weight(W, [0, 3])
    w = oracle.unpack(canon, 3, 4)
    assert w.tolist() == [[0, 1, 0, -1], [0, 1, 0, -1], [1, 0, 0, -1]]
    assert ws.tolist() == [0x3F80]   # bf16(1.0)


def test_quant_weight_zero_matrix_uses_the_floor():
    canon, ws = oracle.quant_weight(np.zeros((2, 4), np.float32), [0, 2])
    assert (oracle.unpack(canon, 2, 4) == 0).all()
    # ws = 1 / s with s = 1 / 1e-5: 1e-5 within one bf16 step (2^-8 rel.)
    assert abs(bits_f32(int(ws[0])) - 1e-5) <= 1e-5 * 2.0 ** -8


def test_quant_weight_of_a_scaled_ternary_matrix_returns_its_codes():
    # W = alpha * t (t ternary): mean = alpha (1 - p0), so |W s| = 1/(1-p0)
    # lies in (1, 2.5) and rounds-and-clamps back to 1; zeros stay zero.
    N, K, alpha = 40, 256, 0.0371
    t = synth.canonical_weights(synth.base_seed(13), N, K)
    t = oracle.unpack(t, N, K).astype(np.float32)
    W = (alpha * t).astype(np.float32)
    canon, ws = oracle.quant_weight(W, [0, N])
    assert (oracle.unpack(canon, N, K) == t).all()
    mean = float(np.abs(W.astype(np.float64)).mean())
    assert abs(bits_f32(int(ws[0])) - mean) <= mean * 2.0 ** -8


def test_quant_weight_segments_are_independent_and_scale_invariant():
    rng = np.random.default_rng(7)
    W = rng.standard_normal((30, 64)).astype(np.float32)
    W[10:] *= 3.0
    canon, ws = oracle.quant_weight(W, [0, 10, 30])
    c0, w0 = oracle.quant_weight(W[:10], [0, 10])
    c1, w1 = oracle.quant_weight(W[10:], [0, 20])
    assert (canon[:10] == c0).all() and (canon[10:] == c1).all()
    assert ws.tolist() == [int(w0[0]), int(w1[0])]
    # codes of 2^e W equal those of W; the scale moves by 2^e exactly
    c2, w2 = oracle.quant_weight((W * 8.0).astype(np.float32), [0, 10, 30])
    assert (c2 == canon).all()
    assert [bits_f32(int(v)) for v in w2] == \
        [8.0 * bits_f32(int(v)) for v in ws]
    # a sign flip of W flips every weight
    c3, w3 = oracle.quant_weight(-W, [0, 10, 30])
    assert (oracle.unpack(c3, 30, 64) == -oracle.unpack(canon, 30, 64)).all()
    assert (w3 == ws).all()


# --------------------------------------------------------------------------
# Decode attention: RoPE, the KV-cache append and grouped-query softmax
# attention (W2A8 kernel page, §一 head counts, §4.1 adjacent-pair RoPE,
# §六 item 2 the preallocated KV cache).
# --------------------------------------------------------------------------
def _bf16(values):
    return np.array([oracle.bf16_rne(float(v)) for v in values], np.uint16)


def _f(bits):
    return synth.bf16_bits_to_f32(np.asarray(bits, np.uint16)).astype(
        np.float64)


def test_rope_worked_example_golden():
    rows = read_golden("rope.txt")
    assert len(rows) == 2
    for row in rows:
        v = [float(t) for t in row.split()]
        p, theta, q, want = int(v[0]), v[1], v[2:6], np.array(v[6:10])
        got = oracle.rope(_bf16(q), p, theta)
        assert np.abs(got - want).max() < 1e-12, (row, got)


def test_rope_position_zero_is_identity_and_norms_are_kept():
    x = synth.bf16_normal(synth.base_seed(20), 128)
    assert (oracle.rope(x, 0, 10000.0) == _f(x)).all()
    for p in (1, 7, 1000, 65535):
        r = oracle.rope(x, p, 500000.0).reshape(-1, 2)
        n0 = (_f(x).reshape(-1, 2) ** 2).sum(1)
        assert np.allclose((r ** 2).sum(1), n0, rtol=1e-14, atol=0)


def test_rope_scores_depend_on_relative_position():
    """q'(p1) . k'(p2) depends on p1 - p2 only (up to the fp32 angles)."""
    q = synth.bf16_normal(synth.base_seed(20, 1), 128)
    k = synth.bf16_normal(synth.base_seed(20, 2), 128)
    for p1, p2, t in ((5, 3, 11), (40, 0, 17), (9, 9, 50)):
        a = oracle.rope(q, p1, 10000.0) @ oracle.rope(k, p2, 10000.0)
        b = oracle.rope(q, p1 + t, 10000.0) @ oracle.rope(k, p2 + t, 10000.0)
        assert abs(a - b) < 1e-4 * np.linalg.norm(_f(q)) * np.linalg.norm(_f(k))


def test_rope_angles_are_fp32_products():
    f1 = float(np.float32(10000.0 ** -0.5))
    assert oracle.rope_angle(1, 1, 4, 10000.0) == f1
    assert oracle.rope_angle(3, 1, 4, 10000.0) == float(
        np.float32(np.float32(3.0) * np.float32(f1)))
    assert oracle.rope_angle(12345, 0, 128, 500000.0) == 12345.0


def test_bf16_rne_from_double_is_one_rounding():
    for v in (1.0, -2.5, 3.140625, 1e-3, 65504.0, 1e-40):
        assert oracle.bf16_rne_d(v) == oracle.bf16_rne(v)   # exact in fp32
    assert oracle.bf16_rne_d(1.0 + 2.0 ** -8) == 0x3F80     # tie -> even
    assert oracle.bf16_rne_d(1.0 + 3 * 2.0 ** -8) == 0x3F82  # tie -> even
    # just above a tie: an fp32 step first would land on the tie and round
    # down; one rounding goes up
    assert oracle.bf16_rne_d(1.0 + 2.0 ** -8 + 2.0 ** -40) == 0x3F81
    assert oracle.bf16_rne_d(-(1.0 + 2.0 ** -8 + 2.0 ** -40)) == 0xBF81
    assert oracle.bf16_rne_d(3.5e38) == 0x7F80               # overflow
    assert oracle.bf16_rne_d(2.0 ** -133) == 0x0001          # subnormal


def test_attn_first_position_returns_the_new_value():
    """p = 0: a single score, weight 1; the rotation at 0 is the identity,
    so the cached key is the new key itself."""
    c = synth.attn_case(synth.base_seed(21), 8, 2, 16, 4, 0)
    out, kc, vc = oracle.attn_decode(c["qkv"], 8, 2, 16, 0, 10000.0,
                                     c["kc"], c["vc"])
    qkv = c["qkv"].reshape(-1, 16)
    for h in range(8):
        assert (out[h] == _f(qkv[8 + 2 + h // 4])).all()
    assert (kc[:, 0] == qkv[8:10]).all() and (vc[:, 0] == qkv[10:12]).all()


def test_attn_zero_query_averages_the_values_of_its_kv_head():
    """q = 0: every score is 0, so head h returns the mean of the value rows
    0..p of KV head h / (H / Hkv) -- pins the grouped head mapping."""
    H, Hkv, D, S, p = 12, 3, 8, 16, 9
    c = synth.attn_case(synth.base_seed(21, 1), H, Hkv, D, S, p)
    qkv = c["qkv"].copy()
    qkv[:H * D] = 0
    out, _, vc = oracle.attn_decode(qkv, H, Hkv, D, p, 10000.0, c["kc"],
                                    c["vc"])
    for h in range(H):
        mean = _f(vc[h // (H // Hkv), :p + 1]).mean(axis=0)
        assert np.allclose(out[h], mean, rtol=0, atol=1e-14)


def test_attn_scores_are_scaled_by_inverse_sqrt_head_dim():
    """D = 4, p = 1: the cached key is 2 ln 3 along q', the new key is 0, so
    the scores are ln 3 and 0 and the weights 3/4 and 1/4 (up to the bf16
    rounding of the cached key)."""
    H, Hkv, D, S, p = 1, 1, 4, 2, 1
    qkv = _bf16([1, 0, 0, 0, 0, 0, 0, 0, 0.5, -1, 2, 0.25])
    qr = oracle.rope(qkv[:4], p, 10000.0)
    k0 = 2 * np.log(3.0) * qr / (qr @ qr)
    kc = _bf16(k0).reshape(1, 1, 4)
    kc = np.concatenate([kc, np.zeros((1, 1, 4), np.uint16)], axis=1)
    vc = np.concatenate([_bf16([1, 2, -4, 8]).reshape(1, 1, 4),
                         np.zeros((1, 1, 4), np.uint16)], axis=1)
    out, _, _ = oracle.attn_decode(qkv, H, Hkv, D, p, 10000.0, kc, vc)
    want = 0.75 * np.array([1, 2, -4, 8]) + 0.25 * np.array([0.5, -1, 2, 0.25])
    assert np.abs(out[0] - want).max() < 2e-2


def test_attn_is_invariant_to_the_order_of_cached_positions():
    H, Hkv, D, S, p = 4, 2, 16, 32, 20
    c = synth.attn_case(synth.base_seed(21, 2), H, Hkv, D, S, p)
    out, _, _ = oracle.attn_decode(c["qkv"], H, Hkv, D, p, 500000.0, c["kc"],
                                   c["vc"])
    perm = np.concatenate([np.random.default_rng(3).permutation(p),
                           np.arange(p, S)])
    out2, _, _ = oracle.attn_decode(c["qkv"], H, Hkv, D, p, 500000.0,
                                    c["kc"][:, perm], c["vc"][:, perm])
    assert np.allclose(out, out2, rtol=0, atol=1e-13)


def test_attn_dominant_position_returns_its_value():
    """One cached key far along q' (a score 40 above the others) takes all
    of the weight."""
    H, Hkv, D, S, p = 2, 1, 16, 8, 5
    c = synth.attn_case(synth.base_seed(21, 3), H, Hkv, D, S, p)
    qkv = c["qkv"].copy()
    qkv[D:2 * D] = qkv[:D]                   # both query heads alike
    kc = np.zeros_like(c["kc"])
    qkv[H * D:(H + 1) * D] = 0               # the new key: score 0
    qr = oracle.rope(qkv[:D], p, 10000.0)
    kc[0, 3] = _bf16(40 * np.sqrt(D) * qr / (qr @ qr))
    out, _, vc = oracle.attn_decode(qkv, H, Hkv, D, p, 10000.0, kc, c["vc"])
    assert np.allclose(out[0], _f(vc[0, 3]), rtol=0, atol=1e-12 * 8)


def test_attn_appends_only_row_p():
    H, Hkv, D, S, p = 8, 2, 32, 12, 7
    c = synth.attn_case(synth.base_seed(21, 4), H, Hkv, D, S, p)
    _, kc, vc = oracle.attn_decode(c["qkv"], H, Hkv, D, p, 10000.0, c["kc"],
                                   c["vc"])
    rows = [j for j in range(S) if j != p]
    assert (kc[:, rows] == c["kc"][:, rows]).all()
    assert (vc[:, rows] == c["vc"][:, rows]).all()
    qkv = c["qkv"].reshape(-1, D)
    for g in range(Hkv):
        want = [oracle.bf16_rne_d(v)
                for v in oracle.rope(qkv[H + g], p, 10000.0)]
        assert (kc[g, p] == np.array(want, np.uint16)).all()
        assert (vc[g, p] == qkv[H + Hkv + g]).all()


def test_attn_rejects_positions_outside_the_cache():
    c = synth.attn_case(synth.base_seed(21, 5), 4, 2, 8, 4, 0)
    for p in (-1, 4):
        with pytest.raises(oracle.OracleError):
            oracle.attn_decode(c["qkv"], 4, 2, 8, p, 10000.0, c["kc"], c["vc"])
