// noalloc.cu -- dsa_indexer_score_noalloc: the indexer scan for callers that
// cannot hand the library a workspace.
//
// Some callers have no way to allocate device memory at the point of the
// call: code running while a CUDA stream is being captured into a graph
// (cudaMalloc is not allowed during capture), latency-critical decode loops
// that must never enter the allocator (cudaMalloc and cudaFree can
// synchronise the device), and plug-in hosts that hand a kernel library only
// the tensors of the operation and keep all allocation to themselves.  This
// entry point runs the same launch sequence as dsa_indexer_score, with its
// scratch taken from a fixed array that lives in this file.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds it until the process exits, and every call on that GPU shares
// it, so calls that may overlap on the GPU (different streams without an
// ordering between them) race on it.  Its size bounds the rows per call
// (DSA_NOALLOC_MAX_ROWS).  Host code cannot use the array's name as a device
// address: the device address comes from cudaGetSymbolAddress, with the
// calling device current.  Outside a stream capture it is looked up on every
// call (a cheap table lookup once the module is loaded), so a device whose
// context was destroyed and created again (cudaDeviceReset) gets the array's
// new address; during a capture the address cached by the last call made on
// that device outside a capture is used, so make one call before capturing.
#include <mutex>

#include "dsa_common.cuh"

namespace dsa {
namespace {

constexpr size_t kNoallocBytes = 1 << 20;   // 1 MiB: enough for DSA_NOALLOC_MAX_ROWS rows
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoallocBytes];

std::mutex g_addr_mutex;
void* g_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device.
cudaError_t scratch_address(cudaStream_t st, void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  e = cudaStreamIsCapturing(st, &cs);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_addr_mutex);
  if (cs == cudaStreamCaptureStatusNone || !g_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" int dsa_indexer_score_noalloc(const void* q_idx, int q_dtype, const float* q_scale,
                                         const float* w, const uint8_t* key_cache,
                                         int64_t num_pages, const int32_t* block_table, int B,
                                         int max_pages, const int32_t* row_req,
                                         const int32_t* row_len, int R, float* scores,
                                         int64_t ld, uint32_t* dev_status, void* stream) {
  int s = check_score_args(q_idx, q_dtype, q_scale, w, key_cache, num_pages, block_table, B,
                           max_pages, row_req, row_len, R, scores, ld);
  if (s) return s;
  if (R > DSA_NOALLOC_MAX_ROWS) return DSA_ERR_UNSUPPORTED;
  if (kStatusBytes + scan_scratch_bytes(R) > kNoallocBytes) return DSA_ERR_UNSUPPORTED;
  // the kernels raise bits in the status word with 32-bit atomics
  if (dev_status && !is_aligned(dev_status, 4)) return DSA_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  void* base = nullptr;
  if ((s = to_status(scratch_address(st, &base)))) return s;
  // The status word must start at zero; the rest of the scratch is written by
  // the launch sequence before it is read, whatever a previous call left.
  uint32_t* status = dev_status ? dev_status : static_cast<uint32_t*>(base);
  if ((s = to_status(cudaMemsetAsync(status, 0, 4, st)))) return s;
  if (R == 0) return DSA_OK;
  ScanArgs a{q_idx, q_dtype, q_scale, w, key_cache, num_pages, block_table, B, max_pages,
             row_req, row_len, R, scores, ld, static_cast<uint8_t*>(base) + kStatusBytes,
             status};
  return to_status(launch_indexer_scan(a, st));
}
