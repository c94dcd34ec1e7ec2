"""GPU parity of the W2A8 path against the CPU oracle, through the C ABI.

Bars: packed bytes and int8 codes bit-exact; int32 accumulators bit-exact;
activation scales bit-exact (same fp32 operations); bf16 outputs within one
bf16 ulp of the oracle (relative 2^-8); both sides round acc / s and then
its product by ws in fp32 before the one bf16 rounding, so the bar is a
margin.  Shapes cover several tiles with ragged tails, the BitNet-2B decode
shapes at full size, the large shapes, batched M, and the edge cases
(smallest sizes, ragged N and K, unaligned activations, the maximum K,
eight scale segments, zero and all-ones weights, extreme activations).
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


DEV = "cuda"


def to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def bf16_dev(bits):
    return to_dev(np.asarray(bits, np.uint16).view(np.int16)) \
        .view(torch.bfloat16)


def bits_of(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def assert_bf16_within_ulp(got, ref):
    g = synth.bf16_bits_to_f32(got).astype(np.float64)
    r = synth.bf16_bits_to_f32(ref).astype(np.float64)
    mag = np.maximum(np.abs(r), np.finfo(np.float32).tiny)
    ulp = np.exp2(np.floor(np.log2(mag)) - 7)
    bad = np.abs(g - r) > ulp
    assert not bad.any(), (f"{int(bad.sum())} bf16 outputs off by > 1 ulp; "
                           f"first at {np.argwhere(bad)[0]}")
    # sign of zero: a zero accumulator must give +0 on both sides
    zero = r == 0
    assert (got[zero] == ref[zero]).all()


def run_case(bw, case, check_y=True, rows=None):
    """Run repack, quant (for s), GEMV and acc on the GPU; compare."""
    M, N, K = case["M"], case["N"], case["K"]
    canon = case["canon"]
    packed = bw.bw_repack(to_dev(canon), N, K)
    q = case["q"]
    x_d = to_dev(q)
    acc = bw.bw_gemv_w2a8_acc(x_d, packed, N, K)
    _, s_d = bw.bw_quant_act(to_dev(case["xf"]))
    y = bw.bw_gemv_w2a8(x_d, packed, s_d, bf16_dev(case["ws"]),
                        case["bounds"].tolist(), N, K)
    torch.cuda.synchronize()
    assert bw.bw_device_error() == 0      # no bounded wait ran out
    _, s_ref = oracle.quant_act(case["xf"])
    assert (s_d.cpu().numpy() == s_ref).all()
    sel = np.arange(N) if rows is None else np.asarray(rows)
    canon_sel = np.ascontiguousarray(canon[sel])
    acc_ref = oracle.gemv_acc(q, canon_sel, len(sel), K)
    assert (acc.cpu().numpy()[:, sel] == acc_ref).all()
    if check_y and rows is None:
        y_ref = oracle.gemv(q, canon, s_ref, case["ws"], case["bounds"], N, K)
        assert_bf16_within_ulp(bits_of(y), y_ref)
    elif check_y:
        # the oracle epilogue on the selected rows with their segments
        seg = np.searchsorted(case["bounds"], sel, side="right") - 1
        y_ref = np.empty((M, len(sel)), np.uint16)
        for i, n in enumerate(sel):
            y_ref[:, i] = oracle.gemv(q, canon[n:n + 1], s_ref,
                                      case["ws"][seg[i]:seg[i] + 1], [0, 1],
                                      1, K)[:, 0]
        assert_bf16_within_ulp(bits_of(y)[:, sel], y_ref)
    return packed


# ----------------------------------------------------------------- repack
@pytest.mark.parametrize("N,K", [(8, 64), (5, 68), (1000, 300), (64, 1024),
                                 (3840, 2560), (2560, 6912)])
def test_repack_bytes_exact_and_round_trip(bw, N, K):
    canon = synth.canonical_weights(synth.base_seed(9, N % 7), N, K)
    packed = bw.bw_repack(to_dev(canon), N, K)
    assert (packed.cpu().numpy() == oracle.layout(canon, N, K)).all()
    back = bw.bw_unrepack(packed, N, K)
    torch.cuda.synchronize()
    assert (back.cpu().numpy() == canon).all()


def test_repack_rejects_code_3(bw):
    canon = synth.canonical_weights(3, 16, 128)
    canon[7, 5] |= 0x30            # weight 22 of row 7 gets code 3
    with pytest.raises(bw.BwError, match="BW_ERR_BAD_CODE"):
        bw.bw_repack(to_dev(canon), 16, 128)
    # the next call on the same stream still works
    ok = synth.canonical_weights(3, 16, 128)
    bw.bw_repack(to_dev(ok), 16, 128)


# -------------------------------------------------------------- quant_act
@pytest.mark.parametrize("M,K", [(1, 2560), (1, 6912), (4, 2560), (16, 2560),
                                 (64, 2560), (3, 300), (1, 1), (2, 65536)])
def test_quant_act_bit_exact(bw, M, K):
    x = synth.normal_f32(synth.base_seed(8, K % 13), M * K).reshape(M, K)
    if M > 2:
        x[1] = 0.0                 # an all-zero row
        x[2, : min(K, 7)] = np.float32(2.5)   # repeated values, exact ties
    q, s = bw.bw_quant_act(to_dev(x))
    torch.cuda.synchronize()
    q_ref, s_ref = oracle.quant_act(x)
    assert (s.cpu().numpy() == s_ref).all()
    assert (q.cpu().numpy() == q_ref).all()


def test_quant_act_ties_to_even(bw):
    x = np.array([[127.0, 2.5, -2.5, 3.5, -3.5, 0.5, -0.5, 1.5]], np.float32)
    q, s = bw.bw_quant_act(to_dev(x))
    torch.cuda.synchronize()
    assert s.item() == 1.0
    assert q.cpu().numpy().tolist() == [[127, 2, -2, 4, -4, 0, 0, 2]]


# ------------------------------------------------------------------- GEMV
def test_small_case_full_parity(bw):
    """M=1, N=K=2560: the small case, every output."""
    run_case(bw, synth.gemv_case(1, 2560, 2560, synth.base_seed(0)))


@pytest.mark.parametrize("name", list(synth.DECODE_SHAPES))
def test_decode_shapes_full_parity(bw, name):
    N, K, bounds = synth.DECODE_SHAPES[name]
    run_case(bw, synth.gemv_case(1, N, K, synth.base_seed(1, len(name)),
                                 bounds=bounds))


@pytest.mark.parametrize("N,K", [(55296, 5120), (13824, 5120)])
def test_large_shapes(bw, N, K):
    case = synth.gemv_case(1, N, K, synth.base_seed(2, N % 11),
                           bounds=[0, N // 4, N // 2, N])
    rows = np.unique(np.concatenate([
        np.arange(0, 64), np.arange(N - 64, N), N // 4 + np.arange(-8, 8),
        N // 2 + np.arange(-8, 8),
        (synth.u64(7, 9, 2000) % np.uint64(N)).astype(np.int64)]))
    run_case(bw, case, rows=rows)


@pytest.mark.parametrize("M", [2, 3, 4, 5, 7, 16, 64])
def test_batched_m(bw, M):
    N, K = 13824, 2560
    case = synth.gemv_case(M, N, K, synth.base_seed(3, M), uniform_x=False,
                           bounds=[0, 6912, N])
    q, _ = oracle.quant_act(case["xf"])   # int8 rows from absmax quantisation
    case["q"] = q
    rows = np.unique(np.concatenate([
        np.arange(0, 40), np.arange(6900, 6930), np.arange(N - 40, N),
        (synth.u64(5, 9, 600) % np.uint64(N)).astype(np.int64)]))
    run_case(bw, case, rows=rows if M > 4 else None)


@pytest.mark.parametrize("M,N,K", [
    (1, 1, 4), (1, 8, 64), (1, 9, 64), (1, 1000, 300), (3, 1000, 68),
    (1, 257, 4100), (2, 77, 1028), (1, 129, 16384), (1, 17, 65536),
    (5, 40, 65536)])
def test_edge_shapes(bw, M, N, K):
    run_case(bw, synth.gemv_case(M, N, K, synth.base_seed(4, N % 15)))


def test_unaligned_activation_rows(bw):
    """x at a 4-byte (not 16-byte) offset takes the word-load path."""
    M, N, K = 2, 300, 1024
    case = synth.gemv_case(M, N, K, synth.base_seed(5))
    canon = case["canon"]
    packed = bw.bw_repack(to_dev(canon), N, K)
    buf = torch.zeros(M * K + 16, dtype=torch.int8, device=DEV)
    x_view = buf[4:4 + M * K].view(M, K)
    x_view.copy_(to_dev(case["q"]))
    assert x_view.data_ptr() % 16 == 4
    acc = bw.bw_gemv_w2a8_acc(x_view, packed, N, K)
    torch.cuda.synchronize()
    assert (acc.cpu().numpy() == oracle.gemv_acc(case["q"], canon, N, K)).all()


def test_eight_segments(bw):
    N, K = 1000, 512
    bounds = [0, 1, 100, 101, 400, 640, 641, 999, 1000]
    run_case(bw, synth.gemv_case(1, N, K, synth.base_seed(6), bounds=bounds))


def test_closed_forms_on_gpu(bw):
    N, K = 24, 6912
    x = np.full((1, K), 127, np.int8)
    for w_val, expect in [(1, 127 * K), (-1, -127 * K), (0, 0)]:
        canon = oracle.pack(np.full((N, K), w_val, np.int8))
        packed = bw.bw_repack(to_dev(canon), N, K)
        acc = bw.bw_gemv_w2a8_acc(to_dev(x), packed, N, K)
        y = bw.bw_gemv_w2a8(to_dev(x), packed,
                            torch.ones(1, device=DEV),
                            bf16_dev([oracle.bf16_rne(1.0)]), [0, N], N, K)
        torch.cuda.synchronize()
        assert (acc.cpu().numpy() == expect).all()
        if w_val == 0:
            assert (bits_of(y) == 0).all()      # +0, not -0
    xm = np.full((1, K), -128, np.int8)
    canon = oracle.pack(np.ones((N, K), np.int8))
    packed = bw.bw_repack(to_dev(canon), N, K)
    acc = bw.bw_gemv_w2a8_acc(to_dev(xm), packed, N, K)
    torch.cuda.synchronize()
    assert (acc.cpu().numpy() == -128 * K).all()


def test_reproducible_and_stream_ordered(bw):
    """Two launches on a side stream give identical results."""
    N, K = 3840, 2560
    case = synth.gemv_case(1, N, K, synth.base_seed(7),
                           bounds=[0, 2560, 3200, 3840])
    packed = bw.bw_repack(to_dev(case["canon"]), N, K)
    st = torch.cuda.Stream()
    x_d = to_dev(case["q"])
    s_d = torch.full((1,), 40.0, device=DEV)
    ws_d = bf16_dev(case["ws"])
    torch.cuda.synchronize()
    with torch.cuda.stream(st):
        y1 = bw.bw_gemv_w2a8(x_d, packed, s_d, ws_d, [0, 2560, 3200, 3840],
                             N, K, stream=st)
        y2 = bw.bw_gemv_w2a8(x_d, packed, s_d, ws_d, [0, 2560, 3200, 3840],
                             N, K, stream=st)
    st.synchronize()
    assert torch.equal(y1, y2)


@pytest.mark.parametrize("M,N,K", [(16, 77, 8192), (48, 300, 16384),
                                   (128, 77, 8192), (100, 300, 16384)])
def test_batched_long_k_repeated(bw, M, N, K):
    """Long K reuses every ring slot of the tensor-core kernel many times (32
    and 64 stages of 256 k): repeated back-to-back calls must all be exact.
    This caught a refill of a weight slot by a bulk copy that overtook the
    slot's last (generic) loads."""
    case = synth.gemv_case(M, N, K, synth.base_seed(12, M % 16),
                           uniform_x=False, bounds=[0, N])
    q, _ = oracle.quant_act(case["xf"])
    packed = bw.bw_repack(to_dev(case["canon"]), N, K)
    x_d = to_dev(q)
    ref = oracle.gemv_acc(q, case["canon"], N, K)
    for _ in range(6):
        acc = bw.bw_gemv_w2a8_acc(x_d, packed, N, K)
        torch.cuda.synchronize()
        assert bw.bw_device_error() == 0
        assert (acc.cpu().numpy() == ref).all()


@pytest.mark.parametrize("M,N,K", [
    (8, 8, 64), (9, 100, 300), (17, 1000, 1028), (33, 77, 16384),
    (65, 513, 2560), (128, 2560, 2560), (200, 64, 68), (8, 40, 20000),
    (24, 300, 1040), (49, 1000, 6928), (256, 1000, 2560), (96, 2560, 6912),
    (113, 129, 4112)])
def test_batched_tensor_core_tiles(bw, M, N, K):
    """M >= 8 takes the tensor-core path: tcgen05 tiles of up to 64 tokens
    (padded to 16) where rows are 16-byte aligned and K % 16 == 0, else
    mma.sync tiles of 8/16; K > 16384 goes back to CUDA cores.  K = 1040 and
    6928 end in a partly valid chunk and a one-chunk stage.  int32 exact,
    bf16 within 1 ulp."""
    case = synth.gemv_case(M, N, K, synth.base_seed(10, M % 16),
                           uniform_x=False, bounds=[0, N // 3 + 1, N])
    q, _ = oracle.quant_act(case["xf"])
    case["q"] = q
    # extreme activations in one row: +-128/127 saturate the int8 range
    case["q"][M // 2, ::3] = -128
    case["q"][M // 2, 1::3] = 127
    run_case(bw, case)


def test_batched_tensor_core_scale_out_of_range(bw):
    """The tensor-core epilogue multiplies by a stored RN(1 / s) and corrects
    the product to the IEEE quotient. A token whose s is outside
    [2^-60, 2^60] is divided instead: row 5, scaled by 1e25. It shares
    tokens 4..7's group of 4 with three tokens on the corrected path, so
    both forms run in one group. Row 17, scaled by 1e-20, meets the
    quantiser's floor on absmax. Within 1 ulp of the oracle, and bit-equal
    to M = 1 calls on the same rows (the CUDA-core kernel, which divides)."""
    M, N, K = 24, 1000, 2560
    canon = synth.canonical_weights(synth.base_seed(24, 0), N, K)
    packed = bw.bw_repack(to_dev(canon), N, K)
    xf = synth.normal_f32(synth.base_seed(24, 1), M * K).reshape(M, K)
    xf[5] *= np.float32(1e25)
    xf[17] *= np.float32(1e-20)
    ws = synth.bf16_uniform(synth.base_seed(24, 2), 2)
    bounds = [0, 333, N]
    q_d, s_d = bw.bw_quant_act(to_dev(xf))
    y = bw.bw_gemv_w2a8(q_d, packed, s_d, bf16_dev(ws), bounds, N, K)
    torch.cuda.synchronize()
    assert bw.bw_device_error() == 0
    assert s_d.cpu().numpy()[5] < 2.0**-60
    q_ref, s_ref = oracle.quant_act(xf)
    y_ref = oracle.gemv(q_ref, canon, s_ref, ws, bounds, N, K)
    assert_bf16_within_ulp(bits_of(y), y_ref)
    for m in (4, 5, 6, 17):
        y1 = bw.bw_gemv_w2a8(q_d[m:m + 1], packed, s_d[m:m + 1], bf16_dev(ws),
                             bounds, N, K)
        torch.cuda.synchronize()
        assert torch.equal(y1.view(torch.int16), y[m:m + 1].view(torch.int16))


@pytest.mark.parametrize("M", [512, 1024, 2048])
def test_prefill_sizes(bw, M):
    """Prompt-sized batches (the W2A8 page's §一 splits prefill from decode):
    M = 512 .. 2048 tokens of absmax-quantised N(0,1) rows against the w13
    shape, int32 exact and bf16 within one ulp on sampled output rows (all
    M tokens of each), including both ends and the gate/up boundary."""
    N, K = 13824, 2560
    case = synth.gemv_case(M, N, K, synth.base_seed(11, M // 512),
                           uniform_x=False, bounds=[0, 6912, N])
    q, _ = oracle.quant_act(case["xf"])
    case["q"] = q
    rows = np.unique(np.concatenate([
        np.arange(0, 16), np.arange(6904, 6920), np.arange(N - 16, N),
        (synth.u64(13, M, 160) % np.uint64(N)).astype(np.int64)]))
    run_case(bw, case, rows=rows)


# ------------------------------------------------- pair-table (LUT) variant
@pytest.mark.parametrize("M,N,K", [
    (1, 2560, 2560), (1, 3840, 2560), (1, 2560, 6912), (1, 13824, 2560),
    (2, 1000, 300), (3, 77, 1028), (4, 13824, 2560), (5, 129, 68),
    (4, 8, 64), (1, 5, 4)])
def test_lut_variant_parity(bw, M, N, K):
    """bw_gemv_w2a8_lut (the TL pages' lut_ctor / qgemm_lut restated): int32
    exact against the oracle and bit-identical to the dp4a path, bf16
    within one ulp; ragged N and K, 1 to 5 rows (tiles of 4, 2 and 1)."""
    bounds = [0, N] if N < 3 else [0, N // 3 + 1, N]
    case = synth.gemv_case(M, N, K, synth.base_seed(14, M * 7 + K % 5),
                           uniform_x=False, bounds=bounds)
    q, s_ref = oracle.quant_act(case["xf"])
    case["q"] = q
    q[0, ::5] = -128                          # extremes of the int8 range
    q[M - 1, 1::7] = 127
    canon = case["canon"]
    packed = bw.bw_repack(to_dev(canon), N, K)
    x_d = to_dev(q)
    acc = bw.bw_gemv_w2a8_lut_acc(x_d, packed, N, K)
    acc_dp4a = bw.bw_gemv_w2a8_acc(x_d, packed, N, K)
    s_d = to_dev(s_ref)
    ws_d = bf16_dev(case["ws"])
    y = bw.bw_gemv_w2a8_lut(x_d, packed, s_d, ws_d, case["bounds"].tolist(),
                            N, K)
    y_dp4a = bw.bw_gemv_w2a8(x_d, packed, s_d, ws_d, case["bounds"].tolist(),
                             N, K)
    torch.cuda.synchronize()
    assert bw.bw_device_error() == 0
    sel = np.arange(N) if N <= 4000 else np.unique(np.concatenate([
        np.arange(0, 64), np.arange(N - 64, N),
        (synth.u64(14, N, 400) % np.uint64(N)).astype(np.int64)]))
    acc_ref = oracle.gemv_acc(q, np.ascontiguousarray(canon[sel]), len(sel), K)
    assert (acc.cpu().numpy()[:, sel] == acc_ref).all()
    assert torch.equal(acc, acc_dp4a)
    assert torch.equal(y.view(torch.int16), y_dp4a.view(torch.int16))
    if N <= 4000:
        y_ref = oracle.gemv(q, canon, s_ref, case["ws"], case["bounds"], N, K)
        assert_bf16_within_ulp(bits_of(y), y_ref)


def test_lut_variant_rejects_tables_that_do_not_fit(bw):
    """Four rows at K = 6912 need 4 x 6912 x 16 bytes of tables: rejected
    before any launch."""
    N, K = 64, 6912
    x = torch.zeros((4, K), dtype=torch.int8, device=DEV)
    packed = torch.zeros((bw.bw_repack_bytes(N, K),), dtype=torch.uint8,
                         device=DEV)
    with pytest.raises(bw.BwError) as e:
        bw.bw_gemv_w2a8_lut_acc(x, packed, N, K)
    assert e.value.status == 2
