// bw_noalloc.cu -- bw_repack_noalloc: the weight repack for callers that may
// not allocate device memory.
//
// bw_repack needs one 4-byte device word of scratch (the bad-code flag its
// kernel raises) and allocates it on every call with cudaMallocAsync.  Some
// callers cannot do that: applications whose device memory is owned by a
// host framework's own allocator (an inference engine that reserves the
// device up front and treats any stray cudaMalloc as a failure), processes
// running with stream-ordered memory pools disabled, or code that must keep
// a fixed device-memory footprint.  This entry point runs the same repack
// kernel with its scratch taken from a fixed array inside the library
// instead, so it performs no allocation and no free.
#include "bw_internal.cuh"

namespace bw {
namespace {

// The scratch: 64 words (256 bytes) that every GPU which loads the library
// holds until the process exits.  The repack uses word 0 as its bad-code
// flag; the amount does not grow with N or K.
constexpr int kScratchWords = 64;
static __device__ __align__(256) unsigned int g_noalloc_scratch[kScratchWords];

// Device address of the array on the current device.  In host code the
// name g_noalloc_scratch is only a host-side stand-in for the symbol; a
// kernel must be given the address that cudaGetSymbolAddress returns.  It is
// looked up on every call rather than cached: the module can load at another
// address after a cudaDeviceReset or in another context on the same device,
// and a per-call lookup also leaves no shared host state between threads.
// The call is cheap next to the synchronising repack.
cudaError_t scratch_address(unsigned int **out) {
  void *p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess) return e;
  *out = static_cast<unsigned int *>(p);
  return cudaSuccess;
}

bool is_aligned(const void *p, uintptr_t a) {
  return reinterpret_cast<uintptr_t>(p) % a == 0;
}

}  // namespace
}  // namespace bw

using namespace bw;

extern "C" bw_status bw_repack_noalloc(const uint8_t *canon, int N, int K,
                                       uint8_t *packed, bw_stream_t stream) {
  if (!canon || !packed || N < 1 || K < 4) return BW_ERR_INVALID_ARG;
  if (K % 4 != 0 || N > BW_MAX_N || K > BW_MAX_K)
    return BW_ERR_UNSUPPORTED_SHAPE;
  if (!is_aligned(packed, 16)) return BW_ERR_MISALIGNED;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);

  unsigned int *flag = nullptr;
  cudaError_t e = scratch_address(&flag);
  unsigned int bad_host = 0;
  // The array keeps the previous call's contents: clear the flag first.
  if (e == cudaSuccess) e = cudaMemsetAsync(flag, 0, sizeof(unsigned int), cs);
  if (e == cudaSuccess) e = launch_repack(canon, N, K, packed, flag, cs);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(&bad_host, flag, sizeof(unsigned int),
                        cudaMemcpyDeviceToHost, cs);
  if (e == cudaSuccess) e = cudaStreamSynchronize(cs);
  if (e != cudaSuccess) {
    record_cuda_error(int(e));
    return BW_ERR_CUDA;
  }
  return bad_host ? BW_ERR_BAD_CODE : BW_OK;
}
