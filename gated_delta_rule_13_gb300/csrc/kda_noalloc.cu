// kda_chunk_fwd_noalloc: the chunked prefill for callers that cannot hand the
// library device memory of its own.
//
// Some callers own every byte of device memory through their host framework's
// allocator (a serving engine that reserves its whole HBM budget at start-up
// and carves tensors out of it, for instance) and are not allowed to call
// cudaMalloc or to obtain an extra workspace buffer.  This entry point runs the
// same kernels as kda_chunk_fwd, but its scratch (the device status block and
// the device copy of a host cu_seqlens array) lives in a file-scope device
// array of fixed size that every GPU loading the library holds until exit.
// Nothing here allocates: no cudaMalloc, no cudaFree, no allocating library
// routine.
//
// Consequences callers must respect:
//   * Every call shares the one array.  Calls that overlap on the GPU (two
//     streams, or two threads issuing to different streams) race on it; issue
//     them on one stream or serialise them.
//   * The array keeps the last call's contents; each call clears the status
//     block (stream-ordered) before its kernels run.
//   * The first call on each device looks the array's device address up with
//     cudaGetSymbolAddress (once per device, with that device current).  Make
//     that first call before any stream capture begins.
//   * At most kda::kNoAllocMaxSeqs sequences per call; larger calls return
//     KDA_ERR_WORKSPACE without launching anything.
//   * The array has no room for the scratch of the in-device split, the helper
//     ring or the longest-first sequence order, so this entry point always
//     runs the plain schedule (one CTA per sequence and head, in index order).
//     Its results equal kda_chunk_fwd's bitwise where kda_chunk_fwd takes the
//     plain or helper schedule, and within the same tolerance where it splits.
//   * Kernel-recorded errors (a malformed device cu_seqlens, a bounded wait
//     that gave up) land in the array's status block; kda_noalloc_read_status
//     reads them without allocating.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/kda.h"
#include "kda_internal.h"

namespace kda {
namespace {

constexpr int kMaxDevices = 64;
constexpr size_t kNoAllocScratchBytes = kStatusBytes + sizeof(int32_t) * (kNoAllocMaxSeqs + 1);

// The scratch shared by every kda_chunk_fwd_noalloc call on a device.  In host
// code this name is only a stand-in for the symbol; kernels get the device
// address obtained below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::once_flag g_once[kMaxDevices];
void *g_scratch_ptr[kMaxDevices];
cudaError_t g_scratch_err[kMaxDevices];

// Device address of the scratch array for the current device (set-up on first use).
cudaError_t scratch_address(void **ptr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::call_once(g_once[dev], [dev] {
    g_scratch_err[dev] = cudaGetSymbolAddress(&g_scratch_ptr[dev], g_noalloc_scratch);
    if (g_scratch_err[dev] != cudaSuccess) cudaGetLastError();
  });
  if (g_scratch_err[dev] != cudaSuccess) return g_scratch_err[dev];
  *ptr = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace kda

extern "C" int kda_noalloc_read_status(void *stream, int clear, int32_t *device_status) {
  if (!device_status) return KDA_ERR_INVALID_ARG;
  void *scratch = nullptr;
  if (kda::scratch_address(&scratch) != cudaSuccess) return KDA_ERR_CUDA;
  // The status block sits at the start of the scratch, as in a workspace.
  return kda_read_device_status(scratch, stream, clear, device_status);
}

extern "C" int kda_chunk_fwd_noalloc(const void *q, const void *k, const void *v,
                                     const float *log_alpha, const float *beta,
                                     const float *init_state, const int32_t *cu_seqlens,
                                     int32_t n_seqs, int64_t n_tokens, int32_t H, int32_t dk,
                                     int32_t dv, int dtype, void *out, float *final_state,
                                     void *stream) {
  if (n_seqs > kda::kNoAllocMaxSeqs) return KDA_ERR_WORKSPACE;
  if (n_seqs < 0) return KDA_ERR_INVALID_ARG;
  void *scratch = nullptr;
  if (kda::scratch_address(&scratch) != cudaSuccess) return KDA_ERR_CUDA;
  return kda_chunk_fwd(q, k, v, log_alpha, beta, init_state, cu_seqlens, n_seqs, n_tokens, H, dk,
                       dv, dtype, out, final_state, scratch, kda::kNoAllocScratchBytes, stream);
}
