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
// address, so the device address is looked up once per device with
// cudaGetSymbolAddress, with that device current, on the first call made on
// it; make that first call before capturing a stream.
#include <mutex>

#include "dsa_common.cuh"

namespace dsa {
namespace {

constexpr size_t kNoallocBytes = 1 << 20;   // 1 MiB: enough for DSA_NOALLOC_MAX_ROWS rows
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoallocBytes];

std::mutex g_addr_mutex;
void* g_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_addr_mutex);
  if (!g_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return cudaSuccess;
}

inline bool aligned16(const void* p) { return ((uintptr_t)p % 16) == 0; }

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" int dsa_indexer_score_noalloc(const void* q_idx, int q_dtype, const float* q_scale,
                                         const float* w, const uint8_t* key_cache,
                                         int64_t num_pages, const int32_t* block_table, int B,
                                         int max_pages, const int32_t* row_req,
                                         const int32_t* row_len, int R, float* scores,
                                         int64_t ld, uint32_t* dev_status, void* stream) {
  if (R < 0 || B < 0 || max_pages < 0) return DSA_ERR_INVALID_ARG;
  if (R > DSA_NOALLOC_MAX_ROWS) return DSA_ERR_UNSUPPORTED;
  if (kStatusBytes + scan_scratch_bytes(R) > kNoallocBytes) return DSA_ERR_UNSUPPORTED;
  if (q_dtype != DSA_BF16 && q_dtype != DSA_E4M3) return DSA_ERR_UNSUPPORTED;
  if (R > 0 && (B < 1 || !block_table || !row_req || !row_len || !q_idx || !w || !key_cache ||
                !scores))
    return DSA_ERR_INVALID_ARG;
  if (q_dtype == DSA_E4M3 && R > 0 && !q_scale) return DSA_ERR_INVALID_ARG;
  if (num_pages < 0 || ld < (int64_t)max_pages * kPage || ld % 4 != 0) return DSA_ERR_INVALID_ARG;
  if ((scores && !aligned16(scores)) || (key_cache && !aligned16(key_cache)))
    return DSA_ERR_INVALID_ARG;
  void* base = nullptr;
  if (scratch_address(&base) != cudaSuccess) return DSA_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // The status word must start at zero; the rest of the scratch is written by
  // the launch sequence before it is read, whatever a previous call left.
  uint32_t* status = dev_status ? dev_status : static_cast<uint32_t*>(base);
  if (cudaMemsetAsync(status, 0, 4, st) != cudaSuccess) return DSA_ERR_CUDA;
  if (R == 0) return DSA_OK;
  ScanArgs a{q_idx, q_dtype, q_scale, w, key_cache, num_pages, block_table, B, max_pages,
             row_req, row_len, R, scores, ld, static_cast<uint8_t*>(base) + kStatusBytes,
             status};
  return launch_indexer_scan(a, st) == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}
