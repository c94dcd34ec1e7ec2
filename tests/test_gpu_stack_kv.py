"""GPU parity of the layer stack with a KV cache (bw_stack_create_kv).

Each layer attends over its cache (RoPE, append at the current position,
softmax over positions 0..p: the W2A8 kernel page's §一 head counts, §4.1
adjacent-pair RoPE and §六 item 2 preallocated cache) instead of the
one-token stand-in; consecutive steps are consecutive tokens.  As for the
plain stack, parity is per stage, teacher-forced from the GPU's own trace
and, for the attention, from the GPU's own cache:
* the appended row of the traced step within one bf16 ulp of the oracle's
  append of the traced q|k|v (values exact), rows past it untouched;
* the traced fp32 attention output against the oracle's attention over the
  GPU's own cache, within 2^-13 of the largest value of the KV head (the
  bound of the attention's own tests), then attn_sub_norm + quantisation
  from that traced output at the plain stack's bar (scale within 1e-5,
  codes equal except within 1e-3 of a rounding tie);
* every GEMV and residual as in the plain stack's test.
End to end over a few tokens it stays within 1 % of the oracle's layers.
"""
import numpy as np
import pytest

import oracle
import synth
from test_gpu_stack import (DEV, assert_bf16_within_ulp, bits_of,
                            check_norm_quant, make_stack, to_dev,
                            trace_buffers)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
THETA = 500000.0


@pytest.fixture(scope="module")
def bw():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from conftest import build_lib
    build_lib()
    import bit_gemv_bitlinear_gb300 as mod
    return mod


def make_kv_stack(bw, n_layers, dim, ffn, nh, nkv, seed, S,
                  gamma_one=True):
    plain, w = make_stack(bw, n_layers, dim, ffn, nh, nkv, seed,
                          gamma_one=gamma_one)
    layers = plain._keep
    plain.close()
    stack = bw.Stack(layers, dim, ffn, nh, nkv, w["eps"], max_positions=S,
                     theta=THETA)
    return stack, w


@pytest.mark.parametrize("layer,steps,S", [(0, 3, 64), (1, 3, 64),
                                           (1, 200, 256), (0, 3, 4096),
                                           (1, 200, 4096)])
def test_kv_stack_per_stage_parity(bw, layer, steps, S):
    """The trace is of the last token of the call: position 2 (a context the
    attention finishes in one CTA per KV head) and position 199 (200
    positions in splits merged across CTAs, the path the bench's 256-token
    runs take past position 127).  With the 4096-position cache the stack
    replays its short-context graphs: position 2 in a launch of one small
    CTA per KV head, position 199 in clusters of 8 small CTAs, after 128
    tokens of the first and 71 of the second."""
    dim, ffn, nh, nkv = 2560, 6912, 20, 5
    hd = dim // nh
    qkv_n = (nh + 2 * nkv) * hd
    stack, w = make_kv_stack(bw, 2, dim, ffn, nh, nkv, 41, S,
                             gamma_one=False)
    h0 = synth.step_inputs(9, steps, dim)
    tr = trace_buffers(dim, ffn, qkv_n, layer)
    out = stack.run(to_dev(h0), trace=tr)        # positions 0 .. steps - 1
    kc_d, vc_d = stack.read_kv(layer)
    torch.cuda.synchronize()
    assert bw.bw_device_error() == 0
    T = {k: (v.cpu().numpy() if v.dtype != torch.bfloat16 else bits_of(v))
         for k, v in tr.items() if k != "layer"}
    kc, vc = bits_of(kc_d), bits_of(vc_d)
    p = steps - 1
    L = w["layers"][layer]
    g, eps, B = L["gammas"], w["eps"], w["bounds"]
    if layer == 0:
        assert (T["h_in"] == h0[p]).all()
    check_norm_quant(T["h_in"], g[:dim], eps, T["q_attn"],
                     float(T["s_attn"][0]), "attn_norm")
    ref = oracle.gemv(T["q_attn"], L["wqkv"], T["s_attn"], L["ws"][0:3],
                      B["wqkv"], qkv_n, dim)[0]
    assert_bf16_within_ulp(T["qkv"], ref, "wqkv")
    # the append of this step: row p from the traced q|k|v; rows past p
    # never written (the cache starts zeroed)
    kref, vref = oracle.attn_append(T["qkv"], nh, nkv, hd, p, THETA, kc, vc)
    assert (vc[:, p] == vref[:, p]).all()
    assert_bf16_within_ulp(kc[:, p].reshape(-1), kref[:, p].reshape(-1),
                           "appended key row")
    assert (kc[:, p + 1:] == 0).all() and (vc[:, p + 1:] == 0).all()
    assert (kc[:, :p] != 0).any() and (vc[:, :p] != 0).any()
    # attention over the GPU's own cache, then attn_sub_norm from the traced
    # attention output -> wo
    att = oracle.attn_over_cache(T["qkv"], nh, nkv, hd, p, THETA, kc, vc)
    G = nh // nkv
    got = T["attn"].reshape(nh, hd).astype(np.float64)
    for h in range(nh):
        vmax = np.abs(synth.bf16_bits_to_f32(vc[h // G, :p + 1])).max()
        err = np.abs(got[h] - att[h]).max()
        assert err <= 2.0 ** -13 * vmax, (h, err, vmax)
    check_norm_quant(T["attn"], g[dim:2 * dim], eps, T["q_o"],
                     float(T["s_o"][0]), "attn_sub_norm")
    ref = oracle.gemv(T["q_o"], L["wo"], T["s_o"], L["ws"][3:4], B["wo"],
                      dim, dim)[0]
    assert_bf16_within_ulp(T["o"], ref, "wo")
    h_mid = (T["h_in"] + synth.bf16_bits_to_f32(T["o"])).astype(np.float32)
    assert (T["h_mid"] == h_mid).all()
    check_norm_quant(T["h_mid"], g[2 * dim:3 * dim], eps, T["q_ffn"],
                     float(T["s_ffn"][0]), "ffn_norm")
    ref = oracle.gemv(T["q_ffn"], L["w13"], T["s_ffn"], L["ws"][4:6],
                      B["w13"], 2 * ffn, dim)[0]
    assert_bf16_within_ulp(T["gu"], ref, "w13")
    gated = oracle.relu2_gate(T["gu"])
    check_norm_quant(gated, g[3 * dim:], eps, T["q_down"],
                     float(T["s_down"][0]), "ffn_sub_norm")
    ref = oracle.gemv(T["q_down"], L["w2"], T["s_down"], L["ws"][6:7],
                      B["w2"], dim, ffn)[0]
    assert_bf16_within_ulp(T["down"], ref, "w2")
    if layer == 1:
        h_out = (T["h_mid"] + synth.bf16_bits_to_f32(T["down"])).astype(
            np.float32)
        assert (out[p].cpu().numpy() == h_out).all()
    stack.close()


def test_kv_stack_short_context_graphs_equal_the_full_cache_launch(bw):
    """Tokens 0..255 through two stacks with the same weights.  With a
    4096-position cache the stack replays its short-context graphs: to
    position 127 one 128-row CTA per KV head, then clusters of 8 CTAs of
    128 rows (the switch between the two inside one call).  With a
    256-position cache it replays its own short graph to position 127, then
    its full-cache graph: clusters of 8 CTAs of the 256-row staging.  Past
    position 127 both split the positions over the same CTAs and merge them
    alike, so the outputs and the caches are bit-identical."""
    dim, ffn, nh, nkv = 2560, 6912, 20, 5
    steps = 256
    h = to_dev(synth.step_inputs(13, steps, dim))
    outs, caches = [], []
    for S in (4096, 256):
        stack, _ = make_kv_stack(bw, 2, dim, ffn, nh, nkv, 45, S,
                                 gamma_one=False)
        outs.append(stack.run(h).clone())
        assert bw.bw_device_error() == 0
        k, v = stack.read_kv(1)
        caches.append((k[:, :steps].clone(), v[:, :steps].clone()))
        stack.close()
    assert torch.equal(outs[0], outs[1])
    assert torch.equal(caches[0][0], caches[1][0])
    assert torch.equal(caches[0][1], caches[1][1])


def test_kv_stack_graph_steps_equal_eager_and_reset_restarts(bw):
    dim, ffn, nh, nkv, S = 512, 1024, 4, 1, 16
    qkv_n = (nh + 2 * nkv) * (dim // nh)
    stack, _ = make_kv_stack(bw, 2, dim, ffn, nh, nkv, 42, S)
    h = to_dev(synth.step_inputs(10, 4, dim))
    out_graph = stack.run(h).clone()               # positions 0..3, graphs
    stack.reset_kv()
    outs = []
    for t in range(4):                             # eager steps (trace on)
        tr = trace_buffers(dim, ffn, qkv_n, 1)
        outs.append(stack.run(h[t:t + 1], trace=tr)[0].clone())
    for t in range(4):
        assert torch.equal(outs[t], out_graph[t]), t
    assert bw.bw_device_error() == 0
    stack.close()


def test_kv_stack_end_to_end_close_to_oracle(bw):
    """Four tokens through 3 layers: within 1 % (relative L2) of the
    oracle's layers run token by token with their own caches."""
    dim, ffn, nh, nkv, S = 256, 512, 2, 1, 8
    hd = dim // nh
    stack, w = make_kv_stack(bw, 3, dim, ffn, nh, nkv, 43, S)
    steps = 4
    h0 = synth.step_inputs(11, steps, dim)
    out = stack.run(to_dev(h0)).cpu().numpy()
    assert bw.bw_device_error() == 0
    caches = [(np.zeros((nkv, S, hd), np.uint16),
               np.zeros((nkv, S, hd), np.uint16)) for _ in w["layers"]]
    for t in range(steps):
        h = h0[t].copy()
        for i, L in enumerate(w["layers"]):
            h, kc, vc = oracle.layer_kv(h, dim, ffn, nh, nkv, w["eps"],
                                        L["wqkv"], L["wo"], L["w13"], L["w2"],
                                        L["ws"], L["gammas"], caches[i][0],
                                        caches[i][1], t, THETA)
            caches[i] = (kc, vc)
        rel = np.linalg.norm(out[t] - h) / np.linalg.norm(h)
        assert rel < 1e-2, (t, rel)
    stack.close()


def test_kv_stack_past_its_capacity_is_reported(bw):
    dim, ffn, nh, nkv, S = 256, 512, 2, 1, 2
    stack, _ = make_kv_stack(bw, 1, dim, ffn, nh, nkv, 44, S)
    h = to_dev(synth.step_inputs(12, 3, dim))
    stack.run(h[:2])                               # positions 0, 1
    assert bw.bw_device_error() == 0
    stack.run(h[2:3])                              # position 2 >= S
    with pytest.raises(bw.BwError) as e:
        bw.bw_device_error()
    assert e.value.status == 1                     # BW_ERR_INVALID_ARG
    stack.reset_kv()
    stack.run(h[:1])
    assert bw.bw_device_error() == 0
    stack.close()
