"""bw_repack_noalloc, the repack for callers that may not allocate device
memory, checked through the C ABI against bw_repack.

Some applications own all device memory through their own allocator and may
not call cudaMalloc (or the stream-ordered allocator) behind its back; for
them the library offers a repack whose scratch word lives in a fixed array
inside the library.  Its output must be identical to bw_repack's (packed
bytes are compared exactly, the bar for byte work), on two calls in a row,
since every call reuses the same scratch and must clear it first.  It must
also allocate nothing: the device's default memory pool (which the
stream-ordered allocator behind bw_repack draws from) sees no use, and the
device's free memory does not move, while bw_repack, the control, does draw
from the pool.  This file is collected last and also passes when run alone in
a fresh process.
"""
import ctypes
import os

import numpy as np
import pytest

import synth
from conftest import build_lib

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

P = ctypes.c_void_p
OK, BAD_CODE, SHAPE = 0, 4, 2


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = ctypes.CDLL(build_lib())
    for name in ("bw_repack", "bw_repack_noalloc"):
        f = getattr(lib, name)
        f.restype = ctypes.c_int
        f.argtypes = [P, ctypes.c_int, ctypes.c_int, P, P]
    lib.bw_repack_bytes.restype = ctypes.c_size_t
    lib.bw_repack_bytes.argtypes = [ctypes.c_int, ctypes.c_int]
    return lib


def _repack(lib, fn, canon, N, K):
    canon_d = torch.from_numpy(np.ascontiguousarray(canon)).cuda()
    out = torch.full((lib.bw_repack_bytes(N, K),), 0xEE, dtype=torch.uint8,
                     device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    rc = getattr(lib, fn)(canon_d.data_ptr(), N, K, out.data_ptr(), stream)
    torch.cuda.synchronize()
    return rc, out.cpu().numpy()


def test_noalloc_matches_repack_on_two_calls_in_a_row(lib):
    for i, (N, K) in enumerate([(2560, 6912), (1000, 300)]):
        canon = synth.canonical_weights(synth.base_seed(12, i), N, K)
        rc_ref, ref = _repack(lib, "bw_repack", canon, N, K)
        rc, got = _repack(lib, "bw_repack_noalloc", canon, N, K)
        assert rc_ref == OK and rc == OK
        assert (got == ref).all()


def test_noalloc_flag_is_cleared_between_calls(lib):
    N, K = 64, 256
    canon = synth.canonical_weights(synth.base_seed(12, 5), N, K)
    bad = canon.copy()
    bad[3, 7] |= 0x0C                       # weight 29 of row 3 gets code 3
    rc, _ = _repack(lib, "bw_repack_noalloc", bad, N, K)
    assert rc == BAD_CODE
    rc, got = _repack(lib, "bw_repack_noalloc", canon, N, K)
    assert rc == OK                          # the stale flag was cleared
    rc_ref, ref = _repack(lib, "bw_repack", canon, N, K)
    assert rc_ref == OK and (got == ref).all()


def test_noalloc_rejects_sizes_beyond_the_limits(lib):
    dummy = torch.zeros(16, dtype=torch.uint8, device="cuda")
    f = lib.bw_repack_noalloc
    assert f(dummy.data_ptr(), 8, 65540, dummy.data_ptr(), None) == SHAPE
    assert f(dummy.data_ptr(), (1 << 24) + 1, 64, dummy.data_ptr(),
             None) == SHAPE


# cudaMemPoolAttr values from the CUDA runtime's driver_types.h.
USED_MEM_CURRENT, USED_MEM_HIGH = 0x7, 0x8


def _cudart():
    """The CUDA runtime as a shared library (the library under test links
    its own copy statically; both see the same device memory pool)."""
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    for name in (os.path.join(home, "lib64", "libcudart.so"),
                 os.path.join(home, "lib64", "libcudart.so.13"),
                 "libcudart.so.13", "libcudart.so"):
        try:
            rt = ctypes.CDLL(name)
        except OSError:
            continue
        rt.cudaDeviceGetDefaultMemPool.argtypes = [ctypes.POINTER(P),
                                                   ctypes.c_int]
        rt.cudaMemPoolGetAttribute.argtypes = [P, ctypes.c_int, P]
        rt.cudaMemPoolSetAttribute.argtypes = [P, ctypes.c_int, P]
        return rt
    pytest.skip("no shared CUDA runtime library to query the memory pool")


def test_noalloc_allocates_nothing(lib):
    rt = _cudart()
    pool = P()
    assert rt.cudaDeviceGetDefaultMemPool(
        ctypes.byref(pool), torch.cuda.current_device()) == 0

    def attr(which):
        v = ctypes.c_uint64(0)
        assert rt.cudaMemPoolGetAttribute(pool, which, ctypes.byref(v)) == 0
        return v.value

    def reset_high():
        zero = ctypes.c_uint64(0)
        assert rt.cudaMemPoolSetAttribute(pool, USED_MEM_HIGH,
                                          ctypes.byref(zero)) == 0

    N, K = 2560, 2560
    canon = synth.canonical_weights(synth.base_seed(12, 6), N, K)
    canon_d = torch.from_numpy(canon).cuda()
    out = torch.empty((lib.bw_repack_bytes(N, K),), dtype=torch.uint8,
                      device="cuda")
    stream = torch.cuda.current_stream().cuda_stream

    def call(fn):
        rc = getattr(lib, fn)(canon_d.data_ptr(), N, K, out.data_ptr(),
                              stream)
        torch.cuda.synchronize()
        assert rc == OK

    # A first call may load the library's code onto the device (lazy module
    # loading), which the CUDA driver backs with device memory of its own.
    call("bw_repack_noalloc")
    used = attr(USED_MEM_CURRENT)
    free_before = torch.cuda.mem_get_info()[0]
    reset_high()
    for _ in range(2):
        call("bw_repack_noalloc")
    assert attr(USED_MEM_HIGH) <= used            # nothing drawn from the pool
    assert torch.cuda.mem_get_info()[0] == free_before
    # the control: bw_repack's stream-ordered scratch word shows in the pool
    reset_high()
    call("bw_repack")
    assert attr(USED_MEM_HIGH) > used
