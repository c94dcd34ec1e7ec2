"""GPU parity of the absmean weight ternarisation (bw_quant_weight) against
the CPU oracle, through the C ABI.

Bar: canonical codes bit-exact and the bf16 scales bit-exact.  The fp64 sums
of |W| are added in a different order on the two sides; they decide the fp32
mean, and so everything else, identically unless a sum lies within a few
fp64 rounding steps of an fp32 rounding boundary -- the test checks that the
inputs are not that close (2^-36 relative) before comparing.  Shapes: the BitNet-2B
projections with their scale segments, ragged small shapes, the closed-form
matrices of the oracle pins, and the path into the GEMV.
"""
import numpy as np
import pytest

import oracle
import synth
from conftest import build_lib

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def bw():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build_lib()
    import bit_gemv_bitlinear_gb300 as mod
    return mod


def to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda")


def bits_of(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def weights(N, K, seed, scale=0.02):
    return (scale * synth.normal_f32(seed, N * K)).reshape(N, K) \
        .astype(np.float32)


def assert_means_not_fragile(W, bounds):
    """The fp32 mean of every segment is the same for a sum perturbed by
    2^-36 (relative) either way -- far beyond what the order of an fp64 sum
    of these values changes (typically about 2^-40) -- so the summation
    order cannot change the outcome."""
    for i in range(len(bounds) - 1):
        seg = np.abs(W[bounds[i]:bounds[i + 1]].astype(np.float64))
        total, count = float(seg.sum()), seg.size
        lo = np.float32(total * (1 - 2.0 ** -36) / count)
        hi = np.float32(total * (1 + 2.0 ** -36) / count)
        assert lo == hi, f"segment {i}: mean too close to an fp32 boundary"


def run(bw, W, bounds):
    N, K = W.shape
    canon, ws = bw.bw_quant_weight(to_dev(W), bounds)
    torch.cuda.synchronize()
    ref_canon, ref_ws = oracle.quant_weight(W, bounds)
    assert (canon.cpu().numpy() == ref_canon).all()
    assert (bits_of(ws) == ref_ws).all()
    return canon, ws, ref_canon, ref_ws


@pytest.mark.parametrize("name", list(synth.DECODE_SHAPES))
def test_decode_projections_bit_exact(bw, name):
    N, K, bounds = synth.DECODE_SHAPES[name]
    W = weights(N, K, synth.base_seed(14, len(name)))
    W[bounds[1] - 1:] *= 1.7   # segments with different magnitudes
    assert_means_not_fragile(W, list(bounds))
    run(bw, W, list(bounds))


@pytest.mark.parametrize("N,K,bounds", [
    (1, 4, [0, 1]), (7, 12, [0, 7]), (77, 68, [0, 5, 40, 77]),
    (300, 1028, [0, 1, 299, 300]), (64, 16384, [0, 64])])
def test_ragged_shapes_bit_exact(bw, N, K, bounds):
    W = weights(N, K, synth.base_seed(15, N % 16), scale=1.0)
    assert_means_not_fragile(W, bounds)
    run(bw, W, bounds)


def test_closed_form_matrices(bw):
    # ties to even and the clamp on a matrix of mean exactly 1
    W = np.array([[0.5, 1.5, -0.5, -1.5], [0.5, 1.5, -0.5, -1.5],
                  [2.5, 0.0, -0.5, -1.0]], np.float32)
    canon, ws, _, _ = run(bw, W, [0, 3])
    assert oracle.unpack(canon.cpu().numpy(), 3, 4).tolist() == \
        [[0, 1, 0, -1], [0, 1, 0, -1], [1, 0, 0, -1]]
    assert bits_of(ws).tolist() == [0x3F80]
    # zero matrix: every weight 0, the 1e-5 floor; constant: every weight +1
    run(bw, np.zeros((16, 64), np.float32), [0, 16])
    canon, ws, _, _ = run(bw, np.full((9, 32), 0.5, np.float32), [0, 4, 9])
    assert (oracle.unpack(canon.cpu().numpy(), 9, 32) == 1).all()
    assert bits_of(ws).tolist() == [0x3F00, 0x3F00]


def test_ternarised_weights_drive_the_gemv(bw):
    """quant_weight -> repack -> GEMV equals the oracle GEMV on the oracle's
    own codes and scales."""
    N, K, bounds = synth.DECODE_SHAPES["wqkv"]
    W = weights(N, K, synth.base_seed(16))
    assert_means_not_fragile(W, list(bounds))
    canon, ws, ref_canon, ref_ws = run(bw, W, list(bounds))
    packed = bw.bw_repack(canon, N, K)
    case = synth.gemv_case(1, N, K, synth.base_seed(16, 1))
    q, s = oracle.quant_act(case["xf"])
    y = bw.bw_gemv_w2a8(to_dev(q), packed, to_dev(s), ws, list(bounds), N, K)
    torch.cuda.synchronize()
    y_ref = oracle.gemv(q, ref_canon, s, ref_ws, list(bounds), N, K)
    g = synth.bf16_bits_to_f32(bits_of(y)).astype(np.float64)
    r = synth.bf16_bits_to_f32(y_ref).astype(np.float64)
    mag = np.maximum(np.abs(r), np.finfo(np.float32).tiny)
    assert (np.abs(g - r) <= np.exp2(np.floor(np.log2(mag)) - 7)).all()


def test_invalid_arguments(bw):
    W = to_dev(np.zeros((8, 16), np.float32))
    with pytest.raises(bw.BwError):
        bw.bw_quant_weight(W, [0, 9])           # bounds do not end at N
    with pytest.raises(bw.BwError):
        bw.bw_quant_weight(W, [0, 4, 4, 8])     # empty segment
    unaligned = torch.zeros(8 * 16 + 1, dtype=torch.float32, device="cuda")
    with pytest.raises(bw.BwError):
        bw.bw_quant_weight(unaligned[1:].view(8, 16), [0, 8])  # 4-byte offset
