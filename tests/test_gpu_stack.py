"""GPU parity of the decoder layer stack (bw_stack_create / bw_layer_stack).

The stack chains the W2A8 GEMVs with fp32 glue (RMSNorm, absmax
requantisation, residual adds, the squared-ReLU gate, one-token attention).
End to end it is not bit-reproducible against an independent oracle: a
reduction order that differs in the last fp32 bit can flip an int8 code at a
rounding tie, and the chain amplifies it.  So parity is checked per stage,
teacher-forced from the stack's own trace of one layer:

* each GEMV against the oracle GEMV on the GPU's own int8 input and scale:
  bf16 within one ulp (int32 exact underneath);
* each norm + quantisation against the oracle from the GPU's own fp32 input:
  scale within 1e-5 relative, codes equal except at rounding near-ties
  (|x*s - (k + 1/2)| < 1e-3, and then off by one at most), and few of those;
* residual adds exactly (fp32 adds of the same values).

Closed forms: zero weights make a layer the identity (bit-exact); the
graph-replayed steps equal eagerly launched ones (bit-exact).
"""
import numpy as np
import pytest

import oracle
import synth
from conftest import build_lib

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
DEV = "cuda"


@pytest.fixture(scope="module")
def bw():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build_lib()
    import bit_gemv_bitlinear_gb300 as mod
    return mod


def to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def bf16_dev(bits):
    return to_dev(np.asarray(bits, np.uint16).view(np.int16)).view(
        torch.bfloat16)


def bits_of(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def assert_bf16_within_ulp(got, ref, what):
    g = synth.bf16_bits_to_f32(got).astype(np.float64)
    r = synth.bf16_bits_to_f32(ref).astype(np.float64)
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(r), 1e-38))) - 7)
    bad = np.abs(g - r) > ulp
    assert not bad.any(), f"{what}: {int(bad.sum())} outputs off by > 1 ulp"


def check_norm_quant(x, gamma, eps, q_gpu, s_gpu, what):
    """Oracle norm + quantisation from the GPU's own fp32 input x."""
    normed = oracle.rmsnorm(x, gamma, eps)
    q_ref, s_ref = oracle.quant_act(normed)
    q_ref, s_ref = q_ref[0], float(s_ref[0])
    assert abs(s_gpu - s_ref) <= 1e-5 * abs(s_ref), (what, s_gpu, s_ref)
    diff = np.nonzero(q_gpu.astype(np.int32) != q_ref.astype(np.int32))[0]
    if diff.size:
        prod = normed[diff].astype(np.float64) * s_ref
        frac = np.abs(prod - np.floor(prod) - 0.5)
        assert (frac < 1e-3).all(), (what, diff[:8], prod[:8])
        assert (np.abs(q_gpu[diff].astype(np.int32)
                       - q_ref[diff].astype(np.int32)) <= 1).all(), what
        assert diff.size <= max(2, x.size // 500), (what, diff.size)
    return diff.size


def make_stack(bw, n_layers, dim, ffn, n_heads, n_kv, seed, zero=False,
               gamma_one=True):
    w = synth.stack_weights(seed, n_layers, dim, ffn, n_heads, n_kv,
                            gamma_one=gamma_one)
    dev_layers = []
    for layer in w["layers"]:
        d = {}
        for name in ("wqkv", "wo", "w13", "w2"):
            canon = layer[name]
            if zero:
                canon = np.full_like(canon, 0x55)   # every code 1: weight 0
                layer[name] = canon
            n_rows, kq = canon.shape
            d[name] = bw.bw_repack(to_dev(canon), n_rows, kq * 4)
        d["ws"] = bf16_dev(layer["ws"])
        d["gammas"] = to_dev(layer["gammas"])
        dev_layers.append(d)
    stack = bw.Stack(dev_layers, dim, ffn, n_heads, n_kv, w["eps"])
    return stack, w


def trace_buffers(dim, ffn, qkv_n, layer):
    f = lambda n: torch.empty(n, dtype=torch.float32, device=DEV)
    i8 = lambda n: torch.empty(n, dtype=torch.int8, device=DEV)
    b16 = lambda n: torch.empty(n, dtype=torch.bfloat16, device=DEV)
    return {"layer": layer, "h_in": f(dim), "q_attn": i8(dim), "s_attn": f(1),
            "qkv": b16(qkv_n), "q_o": i8(dim), "s_o": f(1), "o": b16(dim),
            "h_mid": f(dim), "q_ffn": i8(dim), "s_ffn": f(1),
            "gu": b16(2 * ffn), "q_down": i8(ffn), "s_down": f(1),
            "down": b16(dim), "attn": f(dim)}


def test_zero_weights_layer_is_identity(bw):
    dim, ffn, nh, nkv = 256, 512, 4, 2
    stack, _ = make_stack(bw, 2, dim, ffn, nh, nkv, 31, zero=True)
    h = to_dev(synth.step_inputs(5, 3, dim))
    out = stack.run(h)
    assert bw.bw_device_error() == 0
    assert torch.equal(out, h)
    stack.close()


def test_graph_steps_equal_eager_steps(bw):
    dim, ffn, nh, nkv = 512, 1024, 8, 2
    stack, w = make_stack(bw, 3, dim, ffn, nh, nkv, 32)
    qkv_n = (nh + 2 * nkv) * (dim // nh)
    h = to_dev(synth.step_inputs(6, 4, dim))
    out_graph = stack.run(h)                     # graph for every step
    for t in range(4):                           # eager path (trace on)
        tr = trace_buffers(dim, ffn, qkv_n, 1)
        one = stack.run(h[t:t + 1], trace=tr)
        assert torch.equal(one[0], out_graph[t])
    assert bw.bw_device_error() == 0
    stack.close()


@pytest.mark.parametrize("layer,steps", [(0, 2), (1, 2), (1, 256)])
def test_bitnet_stack_per_stage_parity(bw, layer, steps):
    """The trace is of the last step of the call: steps 1 and 255 (the
    bench's runs are 256 steps long)."""
    dim, ffn, nh, nkv = 2560, 6912, 20, 5
    hd = dim // nh
    qkv_n = (nh + 2 * nkv) * hd
    stack, w = make_stack(bw, 2, dim, ffn, nh, nkv, 33, gamma_one=False)
    h0 = synth.step_inputs(7, steps, dim)
    tr = trace_buffers(dim, ffn, qkv_n, layer)
    out = stack.run(to_dev(h0), trace=tr)
    assert bw.bw_device_error() == 0
    T = {k: (v.cpu().numpy() if v.dtype != torch.bfloat16 else bits_of(v))
         for k, v in tr.items() if k != "layer"}
    L = w["layers"][layer]
    g = L["gammas"]
    eps = w["eps"]
    B = w["bounds"]
    p = steps - 1
    if layer == 0:
        assert (T["h_in"] == h0[p]).all()
    flips = 0
    # attention_norm + quant -> wqkv
    flips += check_norm_quant(T["h_in"], g[:dim], eps, T["q_attn"],
                              float(T["s_attn"][0]), "attn_norm")
    ref = oracle.gemv(T["q_attn"], L["wqkv"], T["s_attn"], L["ws"][0:3],
                      B["wqkv"], qkv_n, dim)[0]
    assert_bf16_within_ulp(T["qkv"], ref, "wqkv")
    # one-token attention + attn_sub_norm + quant -> wo
    att = oracle.attn_one_token(T["qkv"], nh, nkv, hd)
    assert (T["attn"] == att).all()          # bf16 values copied exactly
    flips += check_norm_quant(att, g[dim:2 * dim], eps, T["q_o"],
                              float(T["s_o"][0]), "attn_sub_norm")
    ref = oracle.gemv(T["q_o"], L["wo"], T["s_o"], L["ws"][3:4], B["wo"],
                      dim, dim)[0]
    assert_bf16_within_ulp(T["o"], ref, "wo")
    # residual (exact) + ffn_norm + quant -> w13
    h_mid = (T["h_in"] + synth.bf16_bits_to_f32(T["o"])).astype(np.float32)
    assert (T["h_mid"] == h_mid).all()
    flips += check_norm_quant(T["h_mid"], g[2 * dim:3 * dim], eps, T["q_ffn"],
                              float(T["s_ffn"][0]), "ffn_norm")
    ref = oracle.gemv(T["q_ffn"], L["w13"], T["s_ffn"], L["ws"][4:6],
                      B["w13"], 2 * ffn, dim)[0]
    assert_bf16_within_ulp(T["gu"], ref, "w13")
    # relu(gate)^2 * up + ffn_sub_norm + quant -> w2
    gated = oracle.relu2_gate(T["gu"])
    flips += check_norm_quant(gated, g[3 * dim:], eps, T["q_down"],
                              float(T["s_down"][0]), "ffn_sub_norm")
    ref = oracle.gemv(T["q_down"], L["w2"], T["s_down"], L["ws"][6:7],
                      B["w2"], dim, ffn)[0]
    assert_bf16_within_ulp(T["down"], ref, "w2")
    # final residual of the last layer (exact)
    if layer == 1:
        h_out = (T["h_mid"] + synth.bf16_bits_to_f32(T["down"])).astype(
            np.float32)
        assert (out[p].cpu().numpy() == h_out).all()
    stack.close()


def test_tiny_stack_end_to_end_close_to_oracle(bw):
    """Not a bit-exact check (see the module docstring): the fp32 stack
    output stays within 1% (relative L2) of the oracle's after 3 layers."""
    dim, ffn, nh, nkv = 128, 256, 4, 2
    stack, w = make_stack(bw, 3, dim, ffn, nh, nkv, 34)
    h0 = synth.step_inputs(8, 2, dim)
    out = stack.run(to_dev(h0)).cpu().numpy()
    for t in range(2):
        h = h0[t].copy()
        for L in w["layers"]:
            h = oracle.layer(h, dim, ffn, nh, nkv, w["eps"], L["wqkv"],
                             L["wo"], L["w13"], L["w2"], L["ws"],
                             L["gammas"])
        rel = np.linalg.norm(out[t] - h) / np.linalg.norm(h)
        assert rel < 1e-2, rel
    stack.close()


def test_call_replayed_from_a_graph_equals_eager(bw):
    """A stack without a KV cache runs a call as one persistent kernel whose
    exchange epochs live in device memory, so a captured call replays
    correctly: two replays give the eager result bit for bit."""
    dim, ffn, nh, nkv = 512, 1024, 8, 2
    stack, _ = make_stack(bw, 3, dim, ffn, nh, nkv, 35)
    h = to_dev(synth.step_inputs(13, 5, dim))
    want = stack.run(h).clone()
    out = torch.empty_like(h)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        stack.run(h, out, stream=s)
    for _ in range(2):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, want)
    assert bw.bw_device_error() == 0
    stack.close()
