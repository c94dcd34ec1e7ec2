"""Parity of bw_attn_decode (GB300) with the CPU oracle.

One decode step of grouped-query attention over a bf16 KV cache (the W2A8
kernel page: §一 20 query heads over 5 KV heads of 128 dims, §4.1 RoPE on
adjacent pairs, §六 item 2 the preallocated cache).  Checked per stage, as
the layer stack is:
  * the append: every cache row but p is untouched (bit for bit); the value
    row p is the new value exactly; the key row p is the rotated new key,
    within one bf16 ulp of the oracle's (fp32 against fp64 rotation can land
    on the other side of a bf16 rounding tie), almost always identical;
  * the attention: against the oracle's attention over the GPU's own cache
    after the append, |out - ref| <= 2^-13 max |v| of the KV head's rows
    0..p.  The bound comes from the fp32 arithmetic: scores are 128-term
    fp32 dot products (relative error ~1e-6 of sum |q k| / sqrt(128)),
    expf is within 2 ulp and the weighted sums run over at most 512
    positions per split, all well below 2^-13 of the largest value.
"""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

THETA = 500000.0


@pytest.fixture(scope="module")
def bw():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from conftest import build_lib
    build_lib()
    import bit_gemv_bitlinear_gb300 as bw
    return bw


def _dev_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)) \
        .cuda().view(torch.bfloat16)


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _f(bits):
    return synth.bf16_bits_to_f32(bits).astype(np.float64)


class Step:
    """Device state of one sequence: caches, position, workspace."""

    def __init__(self, bw, case):
        self.bw = bw
        self.c = case
        self.kc = _dev_bf16(case["kc"])
        self.vc = _dev_bf16(case["vc"])
        self.pos = torch.tensor([case["p"]], dtype=torch.int32, device="cuda")
        H, Hkv, D, S = case["H"], case["Hkv"], case["D"], case["S"]
        self.ws = torch.zeros((bw.bw_attn_workspace_bytes(H, Hkv, D, S),),
                              dtype=torch.uint8, device="cuda")
        self.out = torch.empty((H, D), dtype=torch.float32, device="cuda")

    def run(self, qkv_bits, p, flags=0):
        c = self.c
        self.pos.fill_(p)
        qkv = _dev_bf16(qkv_bits)
        if flags & self.bw.BW_ATTN_PAST_READY:
            # the promise: nothing in flight writes the position or the
            # cache when the call is launched
            torch.cuda.synchronize()
        self.bw.bw_attn_decode_ex(qkv, self.pos, c["H"], c["Hkv"], self.kc,
                                  self.vc, theta=THETA, out=self.out,
                                  workspace=self.ws, flags=flags)
        torch.cuda.synchronize()
        return self.out.cpu().numpy().astype(np.float64)


def check_step(case, qkv, p, kc_before, vc_before, out, kc_gpu, vc_gpu):
    """Checks one step; returns the number of key elements of row p that
    differ from the oracle's rounding (each by one ulp)."""
    H, Hkv, D = case["H"], case["Hkv"], case["D"]
    kref, vref = oracle.attn_append(qkv, H, Hkv, D, p, THETA, kc_before,
                                    vc_before)
    rows = [j for j in range(case["S"]) if j != p]
    assert (kc_gpu[:, rows] == kc_before[:, rows]).all(), "cache rows changed"
    assert (vc_gpu[:, rows] == vc_before[:, rows]).all(), "cache rows changed"
    assert (vc_gpu[:, p] == vref[:, p]).all(), "value row p"
    got, want = _f(kc_gpu[:, p]), _f(kref[:, p])
    mag = np.maximum(np.abs(want), np.finfo(np.float32).tiny)
    ulp = np.exp2(np.floor(np.log2(mag)) - 7)
    assert (np.abs(got - want) <= ulp).all(), "key row p beyond one ulp"
    flips = int((kc_gpu[:, p] != kref[:, p]).sum())
    assert flips <= max(2, kc_gpu[:, p].size // 100), flips

    ref = oracle.attn_over_cache(qkv, H, Hkv, D, p, THETA, kc_gpu, vc_gpu)
    G = H // Hkv
    for h in range(H):
        vmax = np.abs(_f(vc_gpu[h // G, :p + 1])).max()
        err = np.abs(out[h] - ref[h]).max()
        assert err <= 2.0 ** -13 * vmax, (h, err, vmax)
    return flips


CASES = [
    # H, Hkv, S, p: BitNet-2B heads (G = 4) over contexts finished by one
    # CTA per head (up to 64 positions), the first split contexts, several
    # splits, a ragged last split and a full cache; G = 1, 2, 8, each on
    # both paths.
    (20, 5, 4096, 0),
    (20, 5, 4096, 1),
    (20, 5, 4096, 63),
    (20, 5, 4096, 64),
    (20, 5, 4096, 127),
    (20, 5, 4096, 128),
    (20, 5, 4096, 1000),
    (20, 5, 4096, 4095),
    (8, 8, 300, 299),
    (8, 8, 300, 50),
    (16, 8, 1000, 517),
    (16, 8, 1000, 128),
    (16, 2, 777, 400),
    (16, 2, 777, 100),
    (4, 1, 65536, 65535),
    # splits of at least 48 positions per CTA take the tensor-core scores
    # and values: G = 2, 8 and 1 on the cluster path and G = 8 alone
    (16, 8, 1000, 999),
    (16, 2, 2048, 2047),
    (16, 2, 777, 60),
    (8, 8, 3000, 2999),
    # caches over 4096 positions: the workspace kernel's splits, G = 1, 2, 8
    (8, 8, 4500, 4499),
    (16, 8, 4200, 3000),
    (16, 2, 5000, 4999),
]


@pytest.mark.parametrize("H,Hkv,S,p", CASES)
def test_attn_decode_matches_oracle(bw, H, Hkv, S, p):
    case = synth.attn_case(synth.base_seed(22, CASES.index((H, Hkv, S, p))),
                           H, Hkv, 128, S, p)
    st = Step(bw, case)
    out = st.run(case["qkv"], p)
    assert bw.bw_device_error() == 0
    check_step(case, case["qkv"], p, case["kc"], case["vc"], out,
               _bits(st.kc), _bits(st.vc))


# BW_ATTN_PAST_READY: the position and the earlier rows are read and copied
# before the dependency wait.  Both kernels; CTA 0 alone, the cluster splits
# and the workspace splits; the first and the last position of a cache.
PAST_READY_CASES = [
    (20, 5, 4096, 0),
    (20, 5, 4096, 127),
    (20, 5, 4096, 128),
    (20, 5, 4096, 1000),
    (20, 5, 4096, 4095),
    (8, 8, 300, 50),
    (16, 8, 1000, 999),
    (16, 2, 777, 60),
    (8, 8, 4500, 4499),
    (16, 8, 4200, 3000),
    (16, 2, 5000, 64),
    (4, 1, 65536, 65535),
]


@pytest.mark.parametrize("H,Hkv,S,p", PAST_READY_CASES)
def test_past_ready_matches_oracle(bw, H, Hkv, S, p):
    case = synth.attn_case(
        synth.base_seed(22, 100 + PAST_READY_CASES.index((H, Hkv, S, p))),
        H, Hkv, 128, S, p)
    st = Step(bw, case)
    out = st.run(case["qkv"], p, flags=bw.BW_ATTN_PAST_READY)
    assert bw.bw_device_error() == 0
    check_step(case, case["qkv"], p, case["kc"], case["vc"], out,
               _bits(st.kc), _bits(st.vc))


def test_past_ready_chain_of_calls_in_a_graph(bw):
    """Flagged calls back to back in one graph, each on its own cache at
    the same position: every call's predecessor is the previous call, which
    writes neither the position nor this call's cache, so each may start
    its copies early.  Every call matches the oracle."""
    H, Hkv, D, S, p = 20, 5, 128, 4096, 700
    n = 4
    cases = [synth.attn_case(synth.base_seed(22, 120 + i), H, Hkv, D, S, p)
             for i in range(n)]
    steps = [Step(bw, c) for c in cases]
    qkvs = [_dev_bf16(c["qkv"]) for c in cases]
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):   # warm-up outside the capture
        bw.bw_attn_decode_ex(qkvs[0], steps[0].pos, H, Hkv, steps[0].kc,
                             steps[0].vc, theta=THETA, out=steps[0].out,
                             workspace=steps[0].ws, stream=stream)
    stream.synchronize()
    steps[0].kc.copy_(_dev_bf16(cases[0]["kc"]))
    steps[0].vc.copy_(_dev_bf16(cases[0]["vc"]))
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(n):
            bw.bw_attn_decode_ex(qkvs[i], steps[i].pos, H, Hkv, steps[i].kc,
                                 steps[i].vc, theta=THETA, out=steps[i].out,
                                 workspace=steps[i].ws,
                                 flags=bw.BW_ATTN_PAST_READY, stream=stream)
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    assert bw.bw_device_error() == 0
    for i in range(n):
        out = steps[i].out.cpu().numpy().astype(np.float64)
        check_step(cases[i], cases[i]["qkv"], p, cases[i]["kc"],
                   cases[i]["vc"], out, _bits(steps[i].kc),
                   _bits(steps[i].vc))


@pytest.mark.parametrize("flags", [0, 1])
def test_consecutive_steps_share_the_workspace_and_see_the_appended_rows(
        bw, flags):
    """Three steps p, p+1, p+2 on one cache and one workspace: every step
    must find the merge counters at zero and read the rows the previous
    steps appended."""
    H, Hkv, D, S, p0 = 20, 5, 128, 512, 190
    case = synth.attn_case(synth.base_seed(22, 50), H, Hkv, D, S, p0)
    st = Step(bw, case)
    kc, vc = case["kc"], case["vc"]
    for t in range(3):
        qkv = synth.bf16_normal(synth.base_seed(22, 51 + t),
                                (H + 2 * Hkv) * D)
        out = st.run(qkv, p0 + t, flags=flags)
        kc_gpu, vc_gpu = _bits(st.kc), _bits(st.vc)
        check_step(case, qkv, p0 + t, kc, vc, out, kc_gpu, vc_gpu)
        kc, vc = kc_gpu, vc_gpu
    assert bw.bw_device_error() == 0


def test_graph_replay_advances_with_the_device_position(bw):
    """A CUDA graph captured once serves every step: the position is read
    on the device."""
    H, Hkv, D, S, p0 = 20, 5, 128, 256, 100
    case = synth.attn_case(synth.base_seed(22, 60), H, Hkv, D, S, p0)
    st = Step(bw, case)
    qkv_d = _dev_bf16(case["qkv"])
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):   # warm-up outside the capture
        bw.bw_attn_decode(qkv_d, st.pos, H, Hkv, st.kc, st.vc, theta=THETA,
                          out=st.out, workspace=st.ws, stream=stream)
    stream.synchronize()
    # restore the cache the warm-up appended to
    st.kc.copy_(_dev_bf16(case["kc"]))
    st.vc.copy_(_dev_bf16(case["vc"]))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        bw.bw_attn_decode(qkv_d, st.pos, H, Hkv, st.kc, st.vc, theta=THETA,
                          out=st.out, workspace=st.ws, stream=stream)
    kc, vc = case["kc"], case["vc"]
    for t in range(3):
        qkv = synth.bf16_normal(synth.base_seed(22, 61 + t),
                                (H + 2 * Hkv) * D)
        qkv_d.copy_(_dev_bf16(qkv))
        st.pos.fill_(p0 + t)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        out = st.out.cpu().numpy().astype(np.float64)
        kc_gpu, vc_gpu = _bits(st.kc), _bits(st.vc)
        check_step(case, qkv, p0 + t, kc, vc, out, kc_gpu, vc_gpu)
        kc, vc = kc_gpu, vc_gpu
    assert bw.bw_device_error() == 0


@pytest.mark.parametrize("flags", [0, 1])
def test_position_outside_the_cache_is_reported(bw, flags):
    H, Hkv, D, S = 20, 5, 128, 128
    case = synth.attn_case(synth.base_seed(22, 70), H, Hkv, D, S, 0)
    st = Step(bw, case)
    st.out.fill_(7.0)
    for p in (S, -1):
        out = st.run(case["qkv"], p, flags=flags)
        assert (out == 0).all()
        assert (_bits(st.kc) == case["kc"]).all()
        assert (_bits(st.vc) == case["vc"]).all()
        with pytest.raises(bw.BwError) as e:
            bw.bw_device_error()
        assert e.value.status == 1                 # BW_ERR_INVALID_ARG
    # the workspace counters are back at zero: a valid step still works
    out = st.run(case["qkv"], 5, flags=flags)
    check_step(case, case["qkv"], 5, case["kc"], case["vc"], out,
               _bits(st.kc), _bits(st.vc))
    assert bw.bw_device_error() == 0
