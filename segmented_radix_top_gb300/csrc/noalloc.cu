// Host-buffer segmented top-k that allocates nothing, for callers that
// cannot allocate device memory (see segtopk_batched_topk_host_noalloc in
// include/segtopk.h).
//
// The device staging area is a fixed array in this file's module, which the
// CUDA runtime creates when it loads the library's device code on a GPU. The
// call copies the host inputs into it, runs the ordinary host-buffer path
// on it and copies the results back, so the selection is the same kernel
// and gives the same results as segtopk_batched_topk_host.
#include <mutex>

#include "../../include/segtopk.h"
#include "dispatch.h"

namespace segtopk {
namespace {

static_assert(SEGTOPK_NOALLOC_STAGING_BYTES % 256 == 0, "staging size is a multiple of 256 bytes");

// Shared by every call on a device; it keeps the last call's contents.
static __device__ __align__(256) unsigned char g_noalloc_staging[SEGTOPK_NOALLOC_STAGING_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_staging_mu;
void* g_staging_addr[kMaxDevices]; // device address of g_noalloc_staging, per device (null: not set up)

// The staging array's device address on the current device, looked up once
// per device (with that device current) and kept for the life of the
// process. The array's name in host code is only a handle the runtime maps
// to the device copy; it is never passed to a kernel or a copy itself. A
// device reset destroys the array's device copy, so the address is not
// valid across one (the entry point's documentation says so).
cudaError_t staging_address(void** out)
{
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess)
    return e;
  if (dev < 0 || dev >= kMaxDevices)
    return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_staging_mu);
  if (!g_staging_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_staging);
    if (e != cudaSuccess)
      return e;
    g_staging_addr[dev] = p;
  }
  *out = g_staging_addr[dev];
  return cudaSuccess;
}

} // namespace
} // namespace segtopk

extern "C" int segtopk_batched_topk_host_noalloc(segtopk_dtype key_dtype, const void* keys, const int32_t* values,
                                                 const int64_t* segment_offsets, int64_t num_segments, int32_t k,
                                                 segtopk_direction direction, segtopk_determinism determinism,
                                                 segtopk_tie_break tie_break, segtopk_ordering ordering,
                                                 void* out_keys, int32_t* out_values, int64_t max_segment_len,
                                                 void* stream)
{
  using namespace segtopk;
  // Staging the request needs (the host-buffer path's workspace for these
  // sizes); anything larger is refused before a byte is copied. Offsets are
  // checked first (non-negative), as the host-buffer path checks them.
  if (num_segments > 0 && k > 0 && segment_offsets) {
    int64_t num_keys = 0, max_len = 0;
    const int v = host_offsets_scan(segment_offsets, num_segments, &num_keys, &max_len);
    if (v != SEGTOPK_SUCCESS)
      return v;
    const size_t need = segtopk_host_workspace_bytes(key_dtype, values != nullptr, num_keys, num_segments, k);
    if (need == 0 || need > (size_t)SEGTOPK_NOALLOC_STAGING_BYTES)
      return SEGTOPK_ERROR_NOT_SUPPORTED;
  }
  void* staging = nullptr;
  const cudaError_t e = staging_address(&staging);
  if (e != cudaSuccess)
    return record_cuda_error(e);
  // Every byte the path reads from the staging area is first written by this
  // call (inputs, offsets and the caller's output slots are copied in), so
  // nothing needs clearing between calls.
  return segtopk_batched_topk_host(key_dtype, keys, values, segment_offsets, num_segments, k, direction,
                                   determinism, tie_break, ordering, out_keys, out_values, max_segment_len,
                                   staging, (size_t)SEGTOPK_NOALLOC_STAGING_BYTES, stream);
}
