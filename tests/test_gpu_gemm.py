"""Parity of the prefill product bw_gemm_w2a8 / bw_gemm_w2a8_acc (256-token
tensor-core tiles over fp16 tokens in a workspace) against the oracle.

The W2A8 page ("BitNet GPU 推理框架：从零构建 W2A8 的 2-bit 大模型 CUDA GEMV
内核") runs prefill and decode as separate paths (§一); the prefill product
here has the decode product's definition (§5.3: exact int32 accumulation,
then y = bf16((acc / s) * ws) with the §4.2 segments), so the checks are the
GEMV's: int32 bit-exact against oracle.gemv_acc, bf16 within one ulp of
oracle.gemv, on every output where the oracle finishes in seconds and on
sampled weight rows (all tokens of each) at prompt sizes.
"""
import numpy as np
import pytest

import oracle
import synth
from conftest import build_lib
from test_gpu_gemv import assert_bf16_within_ulp, bf16_dev, bits_of, to_dev

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def bw():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build_lib()
    import bit_gemv_bitlinear_gb300 as mod
    return mod


def check(bw, M, N, K, seed, rows=None, extremes=True):
    bounds = [0, N] if N < 3 else [0, N // 3 + 1, N]
    case = synth.gemv_case(M, N, K, seed, uniform_x=False, bounds=bounds)
    q, s_ref = oracle.quant_act(case["xf"])
    if extremes:                      # both ends of the int8 range
        q[M // 2, ::3] = -128
        q[M // 2, 1::3] = 127
    canon = case["canon"]
    packed = bw.bw_repack(to_dev(canon), N, K)
    x_d = to_dev(q)
    s_d = to_dev(s_ref)
    acc = bw.bw_gemm_w2a8_acc(x_d, packed, N, K)
    y = bw.bw_gemm_w2a8(x_d, packed, s_d, bf16_dev(case["ws"]), bounds, N, K)
    torch.cuda.synchronize()
    assert bw.bw_device_error() == 0      # no bounded wait ran out
    sel = np.arange(N) if rows is None else np.asarray(rows)
    acc_ref = oracle.gemv_acc(q, np.ascontiguousarray(canon[sel]), len(sel), K)
    assert (acc.cpu().numpy()[:, sel] == acc_ref).all()
    seg = np.searchsorted(case["bounds"], sel, side="right") - 1
    if rows is None:
        y_ref = oracle.gemv(q, canon, s_ref, case["ws"], case["bounds"], N, K)
    else:
        y_ref = np.empty((M, len(sel)), np.uint16)
        for i, n in enumerate(sel):
            y_ref[:, i] = oracle.gemv(q, canon[n:n + 1], s_ref,
                                      case["ws"][seg[i]:seg[i] + 1], [0, 1],
                                      1, K)[:, 0]
    assert_bf16_within_ulp(bits_of(y)[:, sel], y_ref)
    return q, packed, acc, y


@pytest.mark.parametrize("M,N,K", [
    (1, 8, 64), (7, 100, 300), (129, 1000, 1028), (256, 2560, 2560),
    (257, 77, 2564), (300, 130, 16384), (511, 513, 640), (64, 2560, 6912),
    (16, 1000, 2560), (100, 777, 1028), (128, 300, 4112)])
def test_gemm_full_parity(bw, M, N, K):
    """Every output: 64-token tiles (M <= 64), 128-token tiles (M <= 128),
    one to three 256-token tiles (ragged last tile), ragged weight-row tiles
    (N not a multiple of 128), K ending in a one-chunk stage (1028, 2564,
    300, 4112) or in a partly valid chunk (300, 2564), the largest K (16384:
    128 stages through the rings)."""
    check(bw, M, N, K, synth.base_seed(15, M % 64 + K % 7))


@pytest.mark.parametrize("M,N,K", [(1024, 13824, 2560), (2048, 2560, 6912),
                                   (768, 3840, 2560), (4096, 1000, 2560)])
def test_gemm_prompt_sizes(bw, M, N, K):
    """Prompt-sized batches at the BitNet-2B shapes and the largest M
    (4096 tokens: 16 token tiles), sampled weight rows (all tokens of each):
    both ends, a row tile boundary and 160 seeded rows."""
    rows = np.unique(np.concatenate([
        np.arange(0, 16), np.arange(120, 136), np.arange(N - 16, N),
        (synth.u64(16, M, 160) % np.uint64(N)).astype(np.int64)]))
    check(bw, M, N, K, synth.base_seed(16, M // 256), rows=rows)


def test_gemm_equals_gemv_and_repeats(bw):
    """The prefill tiles and the GEMV's 128-token tiles compute the same
    exact accumulators and bit-identical bf16 outputs (the GEMV divides by
    s; the prefill epilogue multiplies by 1 / s and corrects the product to
    the IEEE quotient, or divides where s is outside [2^-60, 2^60]: the row
    scaled by 1e25 takes that path; the row scaled by 1e-20 meets the
    quantiser's floor on absmax); repeated calls with one workspace give
    identical results."""
    M, N, K = 384, 1000, 2560
    q, packed, acc, y = check(bw, M, N, K, synth.base_seed(17, 0))
    x_d = to_dev(q)
    xf = synth.normal_f32(synth.base_seed(17, 1), M * K).reshape(M, K)
    xf[3] *= np.float32(1e-20)
    xf[200] *= np.float32(1e25)
    q_d, s_d = bw.bw_quant_act(to_dev(xf))
    ws_d = bf16_dev(synth.bf16_uniform(synth.base_seed(17, 2), 2))
    bounds = [0, 333, N]
    y_gemm = bw.bw_gemm_w2a8(q_d, packed, s_d, ws_d, bounds, N, K)
    y_gemv = bw.bw_gemv_w2a8(q_d, packed, s_d, ws_d, bounds, N, K)
    torch.cuda.synchronize()
    s_h = s_d.cpu().numpy()
    assert s_h[200] < 2.0**-60
    assert torch.equal(y_gemm.view(torch.int16), y_gemv.view(torch.int16))
    acc_gemv = bw.bw_gemv_w2a8_acc(x_d, packed, N, K)
    work = torch.empty((bw.bw_gemm_workspace_bytes(M, K),), dtype=torch.uint8,
                       device="cuda")
    for _ in range(4):
        again = bw.bw_gemm_w2a8_acc(x_d, packed, N, K, workspace=work)
        torch.cuda.synchronize()
        assert bw.bw_device_error() == 0
        assert torch.equal(again, acc)
    assert torch.equal(acc_gemv, acc)


def test_gemm_graph_replay(bw):
    """Captured in a CUDA graph (both launches), replayed on new tokens:
    equal to an eager call on the same tokens."""
    M, N, K = 300, 640, 1024
    case = synth.gemv_case(M, N, K, synth.base_seed(18, 0), uniform_x=True)
    packed = bw.bw_repack(to_dev(case["canon"]), N, K)
    x_d = to_dev(case["q"])
    work = torch.empty((bw.bw_gemm_workspace_bytes(M, K),), dtype=torch.uint8,
                       device="cuda")
    acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        bw.bw_gemm_w2a8_acc(x_d, packed, N, K, acc=acc, workspace=work,
                            stream=s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        bw.bw_gemm_w2a8_acc(x_d, packed, N, K, acc=acc, workspace=work,
                            stream=s)
    q2 = synth.int8_uniform(synth.base_seed(18, 1), M * K).reshape(M, K)
    x_d.copy_(to_dev(q2))
    g.replay()
    torch.cuda.synchronize()
    assert bw.bw_device_error() == 0
    ref = oracle.gemv_acc(q2, case["canon"], N, K)
    assert (acc.cpu().numpy() == ref).all()
