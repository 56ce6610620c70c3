// dsa_common.cuh -- shapes, workspace layout and small device helpers shared
// by the kernels of libdsa (sm_103a).  Nothing here is shared with the CPU
// oracle.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/dsa.h"

namespace dsa {

constexpr int kPage = DSA_PAGE_TOKENS;         // tokens per cache page
constexpr int kIdxHeads = DSA_INDEX_HEADS;     // indexer heads
constexpr int kIdxDim = DSA_INDEX_DIM;         // indexer head dim
constexpr int kKeyPageBytes = DSA_KEY_PAGE_BYTES;
constexpr int kKeyScaleOffset = kPage * kIdxDim;   // scales follow the 64 x 128 key bytes
constexpr int kMxKeyPageBytes = DSA_MXFP4_KEY_PAGE_BYTES;   // 64 x 64 E2M1 bytes, 64 x 4 E8M0
static_assert(kMxKeyPageBytes == kPage * (kIdxDim / 2 + 4), "MXFP4 page layout");
constexpr int kLatDim = DSA_LATENT_DIM;
constexpr int kVDim = DSA_V_DIM;
constexpr int kMaxTopk = DSA_MAX_TOPK;
constexpr size_t kAlign = 256;
constexpr size_t kStatusBytes = 256;           // device status word lives here

// ---- top-k partitioning ------------------------------------------------
constexpr int kTopkChunk = 2048;               // scores per collecting CTA
constexpr int kTopkBins1 = 2048;               // first radix digit: key bits 31..21
constexpr int kTopkBins2 = 2048;               // second digit: bits 20..10
constexpr int kTopkBins3 = 1024;               // third digit: bits 9..0

inline size_t align_up(size_t x, size_t a = kAlign) { return (x + a - 1) / a * a; }

// Byte offsets of the top-k scratch inside a workspace region: per row a
// candidate threshold, a candidate count (zeroed by a memset before every
// selection), where each 2048-score chunk put its candidates, and room for
// kTopkCandCap (key, position) candidates.
constexpr int kTopkCandCap = 8192;
struct TopkLayout {
  size_t tau, cnt, runs, items, bytes;
  int nchunks;
  TopkLayout(int R, int64_t max_len) {
    nchunks = (int)((max_len + kTopkChunk - 1) / kTopkChunk);
    if (nchunks < 1) nchunks = 1;
    size_t o = 0;
    tau = o;       o = align_up(o + (size_t)R * 4);
    cnt = o;       o = align_up(o + (size_t)R * 4);
    runs = o;      o = align_up(o + (size_t)R * nchunks * 8);     // per chunk: (offset, count)
    items = o;     o = align_up(o + (size_t)R * kTopkCandCap * 8);
    bytes = o;
  }
};

// Sparse MLA works on tiles of 128 selected slots.  A unit is one query row
// and one group of up to 64 heads; unit u = row * groups + group has
// NT = ceil(k / 128) tiles.  With fewer units than SMs (U < 152), each unit is
// cut into S = min(152 / U, NT) near-equal parts, one CTA each (G = U * S);
// otherwise the U * NT tiles are cut into G = min(152, U * NT) contiguous
// ranges of near-equal length.  The cut is a fixed function of (R, H, k) so
// that results do not depend on the device.  A CTA's range covers whole units
// (written straight to the output) and at most two cut units, whose partials
// it leaves in slots 2c (its first unit) and 2c + 1 (its last) for the
// combine.
constexpr int kMlaTile = 128;
constexpr int kMlaGrid = 152;

__host__ __device__ inline int mla_heads_per_cta(int H) { return H < 64 ? H : 64; }

struct MlaWork {
  int64_t U, NT, T;
  int G;
  int S;   // > 0: each unit is split over S CTAs of its own; 0: one contiguous split of all tiles
  __host__ __device__ MlaWork(int R, int H, int k) {
    U = (int64_t)R * (H / mla_heads_per_cta(H));
    NT = (k + kMlaTile - 1) / kMlaTile;
    T = U * NT;
    if (U > 0 && U < kMlaGrid) {
      // fewer units than SMs: S equal parts per unit, so that no CTA holds the
      // end of one unit and the start of the next (two output epilogues)
      const int64_t sp = kMlaGrid / U;
      S = (int)(sp < NT ? sp : NT);
      G = (int)(U * S);
    } else {
      S = 0;
      G = (int)(T < kMlaGrid ? T : kMlaGrid);
    }
  }
  __host__ __device__ int64_t begin(int64_t c) const {   // first tile of CTA c
    if (S == 0) return c * T / G;
    return (c / S) * NT + (c % S) * NT / S;
  }
  __host__ __device__ int cta_of(int64_t t) const {
    if (S == 0) return (int)(((t + 1) * G - 1) / T);
    const int64_t u = t / NT, lt = t - u * NT;
    return (int)(u * S + ((lt + 1) * S - 1) / NT);
  }
};

struct MlaLayout {
  size_t part_o, part_lse, q8, qc, bytes;
  MlaLayout(int R, int H, int k) {
    const MlaWork w(R, H, k);
    const size_t slots = 2 * (size_t)w.G, hg = (size_t)mla_heads_per_cta(H);
    size_t o = 0;
    part_o = o;   o = align_up(o + slots * hg * kVDim * 4);
    part_lse = o; o = align_up(o + slots * hg * 4);
    q8 = o;       o = align_up(o + (size_t)R * H * 2 * kLatDim);   // E4M3 hi, lo per head
    qc = o;       o = align_up(o + (size_t)R * H * 4);             // per-head logit factor
    bytes = o;
  }
};

// ---- programmatic dependent launch ---------------------------------------
// The kernels of one call run back to back on a stream.  Each but the first
// is launched with programmatic stream serialization: it may be scheduled as
// soon as every CTA of the kernel before it has called pdl_trigger(), so its
// prologue (barrier set-up, tensor-memory allocation, descriptor prefetch)
// overlaps that kernel's tail and the launch gap disappears.  Every CTA of
// every kernel calls pdl_wait() -- which returns once the kernel before it
// has completed and its writes are visible -- before it reads anything an
// earlier kernel wrote, and before it exits, so that the completion of a
// kernel still implies the completion of all kernels before it.  A kernel
// that allocates tensor memory triggers only after its allocation: a
// dependent CTA placed on the same SM then cannot take the columns first and
// wait on a kernel that waits for them.  Launched without the attribute,
// both are no-ops.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Data an earlier kernel of the chain wrote is read with ld_dep(): an
// ordinary (coherent, L1-cached) load through a pointer without __restrict__,
// which the compiler keeps below pdl_wait() (its asm clobbers memory).  Loads
// on the read-only path (__ldg, or plain loads through a const __restrict__
// pointer, which the compiler may turn into them) count as loads of memory
// that never changes during the kernel, so they may be scheduled above
// pdl_wait() and read what was there before the earlier kernel wrote it.
template <typename T>
__device__ __forceinline__ T ld_dep(const T* p) { return *p; }

// Launches `kernel` on `st`; `chained` = may overlap the previous kernel on
// the stream (it must follow the pdl_wait() rule above).
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t st, bool chained, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = chained ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// ---- device helpers ----------------------------------------------------
__device__ __forceinline__ void raise_dev(uint32_t* status, uint32_t bit) {
  if (status) atomicOr(status, bit);
}

// Two E4M3 bytes (low byte first) -> two floats, exact (E4M3 is a subset of f16).
__device__ __forceinline__ float2 e4m3x2_to_float2(uint16_t v) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)v, __NV_E4M3);
  __half2 hh = *reinterpret_cast<__half2*>(&h);
  return __half22float2(hh);
}

__device__ __forceinline__ float e4m3_to_float(uint8_t v) {
  __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)v, __NV_E4M3);
  return __half2float(*reinterpret_cast<__half*>(&h));
}

// Order-preserving map of a finite fp32 to uint32 (larger value -> larger key);
// -0 maps like +0.
__device__ __forceinline__ uint32_t ordered_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

}  // namespace dsa

// ---- launchers (host side, one per kernel family) --------------------------
namespace dsa {

// Query format of the MXFP4 scorer: E2M1 codes [R][32][64] (two per byte) in
// q_idx, E8M0 scales [R][32][4] in q_sf, keys in MXFP4 pages.
constexpr int kQMxfp4 = 2;

struct ScanArgs {
  const void* q_idx; int q_dtype; const float* q_scale; const float* w;
  const uint8_t* key_cache; int64_t num_pages; const int32_t* block_table; int B; int max_pages;
  const int32_t* row_req; const int32_t* row_len; int R; float* scores; int64_t ld;
  uint8_t* scratch;  // scan_scratch_bytes(R) bytes
  uint32_t* status;
  const uint8_t* q_sf = nullptr;   // kQMxfp4 only
  bool clear_status = false;       // the prep kernel zeroes *status (no separate memset)
};
size_t scan_scratch_bytes(int R);
cudaError_t launch_indexer_scan(const ScanArgs& a, cudaStream_t st);

struct TopkArgs {
  const float* scores; int64_t ld; const int32_t* row_len; int R; int64_t max_len; int k;
  int32_t* idx; uint8_t* scratch;  // TopkLayout(R, max_len).bytes bytes
  uint32_t* status;
  bool chained = false;   // the first kernel may overlap the previous one on the stream
};
cudaError_t launch_topk(const TopkArgs& a, cudaStream_t st);

// The Write step (write.cu): T new tokens' index keys (LayerNorm, absmax
// scale, E4M3) and latent rows (E4M3 with the cache's scale) into the caches.
struct WriteArgs {
  const void* k_raw; const float* gamma; const float* beta; float eps;
  const void* latent; float latent_scale; const int32_t* block_table; int B; int max_pages;
  const int32_t* tok_req; const int32_t* tok_pos; int T;
  uint8_t* key_cache; uint8_t* latent_cache; int64_t num_pages;
  uint32_t* status;   // may be NULL: the device checks are then not reported
  bool chained = false;
  bool mx_keys = false;   // MXFP4 index keys (pages of kMxKeyPageBytes)
};
cudaError_t launch_write_kv(const WriteArgs& a, cudaStream_t st);

// Top-k under decode context parallelism, W token shards emulated on one GPU
// (dcp.cu): every row's result equals launch_topk's.
struct DcpArgs {
  const float* scores; int64_t ld; const int32_t* row_len; int R; int64_t max_len; int k; int W;
  int32_t* idx; uint32_t* resend;  // resend [R] or NULL: bit s = shard s's local top-k was read
  uint8_t* scratch;                // dcp_scratch_bytes(R, max_len, k, W) bytes
  uint32_t* status;
  bool chained = false;
};
size_t dcp_scratch_bytes(int R, int64_t max_len, int k, int W);
cudaError_t launch_topk_dcp(const DcpArgs& a, cudaStream_t st);

struct MlaArgs {
  const void* q; int H; float softmax_scale; const uint8_t* latent_cache; int64_t num_pages;
  float latent_scale; const int32_t* block_table; int B; int max_pages; const int32_t* row_req;
  const int32_t* row_len; const int32_t* idx; int k; int R; void* out; float* lse;
  uint8_t* scratch;  // MlaLayout(R, H, k).bytes bytes
  uint32_t* status;
  bool chained = false;   // the first kernel may overlap the previous one on the stream
  bool nvfp4 = false;     // latent_cache holds 352-byte NVFP4 rows instead of 576-byte E4M3
};
cudaError_t launch_sparse_mla(const MlaArgs& a, cudaStream_t st);

// Library self-test: one CTA whose bounded wait on a barrier that nothing
// arrives on runs out after `limit_cycles` SM cycles (workspace layout in
// selftest.cu, selftest_workspace_bytes() bytes).
cudaError_t launch_selftest_wait(void* workspace, long long limit_cycles, cudaStream_t st);
size_t selftest_workspace_bytes();

// ---- host-side argument checks and status codes (dsa_api.cu) ---------------
inline bool is_aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }
inline int64_t score_ld(int max_pages) { return (int64_t)max_pages * kPage; }

// DSA_OK for cudaSuccess; otherwise DSA_ERR_CUDA, after recording the error as
// the calling host thread's dsa_last_cuda_error.
int to_status(cudaError_t e);

// Row and block-table arguments shared by every call that reads the caches.
int check_rows(int B, int max_pages, const int32_t* block_table, const int32_t* row_req,
               const int32_t* row_len, int R);

// Every argument check of the FP8 indexer scan (dsa_indexer_score and its
// workspace-free form), workspace aside.
int check_score_args(const void* q_idx, int q_dtype, const float* q_scale, const float* w,
                     const uint8_t* key_cache, int64_t num_pages, const int32_t* block_table,
                     int B, int max_pages, const int32_t* row_req, const int32_t* row_len, int R,
                     const float* scores, int64_t ld);

// Tiled TMA descriptor over a byte tensor of the given rank: dims[0] is the
// contiguous extent, strides[i] the byte stride of dim i + 1, box the tile
// copied per load; 128-byte swizzle, out-of-range elements read as zero.
// The driver entry point is looked up once per process.
cudaError_t encode_tensor_map_u8(CUtensorMap* map, int rank, const void* base, const uint64_t* dims,
                                 const uint64_t* strides, const uint32_t* box,
                                 int swizzle_bytes = 128);

}  // namespace dsa
