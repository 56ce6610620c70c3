// dsa_api.cu -- the C ABI of libdsa (declared in include/dsa.h): host-side
// argument validation, workspace carving and the launch sequence of each
// entry point.  No allocation, no host synchronisation (except the explicit
// status read), no global mutable state.
#include <cudaTypedefs.h>
#include <string.h>

#include <mutex>

#include "dsa_common.cuh"

namespace dsa {

cudaError_t encode_tensor_map_u8(CUtensorMap* map, int rank, const void* base, const uint64_t* dims,
                                 const uint64_t* strides, const uint32_t* box, int swizzle_bytes) {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  if (!enc) return cudaErrorNotSupported;
  if (rank < 1 || rank > 5) return cudaErrorInvalidValue;
  if (swizzle_bytes != 128 && swizzle_bytes != 64) return cudaErrorInvalidValue;
  cuuint64_t d[5], st[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
    if (i + 1 < rank) st[i] = strides[i];
  }
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, (cuuint32_t)rank, const_cast<void*>(base),
                         d, st, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace dsa

using namespace dsa;

namespace dsa {

namespace {
thread_local cudaError_t t_last_cuda_error = cudaSuccess;
}  // namespace

int to_status(cudaError_t e) {
  if (e == cudaSuccess) return DSA_OK;
  t_last_cuda_error = e;
  return DSA_ERR_CUDA;
}

int check_rows(int B, int max_pages, const int32_t* block_table, const int32_t* row_req,
               const int32_t* row_len, int R) {
  if (R < 0 || B < 0 || max_pages < 0) return DSA_ERR_INVALID_ARG;
  if (R > 0 && (B < 1 || !block_table || !row_req || !row_len)) return DSA_ERR_INVALID_ARG;
  if (R > 65535) return DSA_ERR_UNSUPPORTED;
  return DSA_OK;
}

int check_score_args(const void* q_idx, int q_dtype, const float* q_scale, const float* w,
                     const uint8_t* key_cache, int64_t num_pages, const int32_t* block_table,
                     int B, int max_pages, const int32_t* row_req, const int32_t* row_len, int R,
                     const float* scores, int64_t ld) {
  int s = check_rows(B, max_pages, block_table, row_req, row_len, R);
  if (s) return s;
  if (q_dtype != DSA_BF16 && q_dtype != DSA_E4M3) return DSA_ERR_UNSUPPORTED;
  if (R > 0 && (!q_idx || !w || !key_cache || !scores)) return DSA_ERR_INVALID_ARG;
  if (q_dtype == DSA_E4M3 && R > 0 && !q_scale) return DSA_ERR_INVALID_ARG;
  if (num_pages < 0 || ld < score_ld(max_pages) || ld % 4 != 0) return DSA_ERR_INVALID_ARG;
  if (scores && !is_aligned(scores, 16)) return DSA_ERR_INVALID_ARG;
  if (key_cache && !is_aligned(key_cache, 16)) return DSA_ERR_INVALID_ARG;
  return DSA_OK;
}

}  // namespace dsa

namespace {

constexpr int kVersion = 1 * 10000 + 1 * 100 + 0;

inline bool aligned(const void* p, size_t a) { return is_aligned(p, a); }

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

int check_workspace(void* ws, size_t have, size_t need) {
  if (!ws || have < need || !aligned(ws, kAlign)) return DSA_ERR_WORKSPACE;
  return DSA_OK;
}

int clear_status(void* ws, cudaStream_t st) { return to_status(cudaMemsetAsync(ws, 0, 4, st)); }

bool supported_heads(int H) { return H == 16 || H == 32 || H == 64 || H == 128; }

}  // namespace

extern "C" {

int dsa_version(void) { return kVersion; }

int dsa_last_cuda_error(void) { return (int)t_last_cuda_error; }

const char* dsa_last_cuda_error_string(void) { return cudaGetErrorString(t_last_cuda_error); }

const char* dsa_status_string(int status) {
  switch (status) {
    case DSA_OK: return "ok";
    case DSA_ERR_INVALID_ARG: return "invalid argument";
    case DSA_ERR_UNSUPPORTED: return "unsupported shape or type";
    case DSA_ERR_WORKSPACE: return "workspace missing, too small or not 256-byte aligned";
    case DSA_ERR_CUDA: return "CUDA error";
    case DSA_ERR_DEVICE_CHECK: return "a kernel found an out-of-range value in device memory";
    default: return "unknown status";
  }
}

int dsa_device_info(int* num_sms, int* cc_major, int* cc_minor) {
  int dev = 0;
  int s = to_status(cudaGetDevice(&dev));
  if (s) return s;
  int v = 0;
  if (num_sms) {
    if ((s = to_status(cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev)))) return s;
    *num_sms = v;
  }
  if (cc_major) {
    if ((s = to_status(cudaDeviceGetAttribute(&v, cudaDevAttrComputeCapabilityMajor, dev)))) return s;
    *cc_major = v;
  }
  if (cc_minor) {
    if ((s = to_status(cudaDeviceGetAttribute(&v, cudaDevAttrComputeCapabilityMinor, dev)))) return s;
    *cc_minor = v;
  }
  return DSA_OK;
}

// ---------------------------------------------------------------- Score
size_t dsa_indexer_score_workspace_size(int R) {
  if (R < 0) return 0;
  return kStatusBytes + scan_scratch_bytes(R);
}

int dsa_indexer_score(const void* q_idx, int q_dtype, const float* q_scale, const float* w,
                      const uint8_t* key_cache, int64_t num_pages, const int32_t* block_table,
                      int B, int max_pages, const int32_t* row_req, const int32_t* row_len,
                      int R, float* scores, int64_t ld, void* workspace, size_t ws_bytes,
                      void* stream) {
  int s = check_score_args(q_idx, q_dtype, q_scale, w, key_cache, num_pages, block_table, B,
                           max_pages, row_req, row_len, R, scores, ld);
  if (s) return s;
  s = check_workspace(workspace, ws_bytes, dsa_indexer_score_workspace_size(R));
  if (s) return s;
  cudaStream_t st = as_stream(stream);
  if (R == 0) return clear_status(workspace, st);
  ScanArgs a{q_idx, q_dtype, q_scale, w, key_cache, num_pages, block_table, B, max_pages,
             row_req, row_len, R, scores, ld, static_cast<uint8_t*>(workspace) + kStatusBytes,
             static_cast<uint32_t*>(workspace)};
  a.clear_status = true;                           // the prep kernel clears the word
  return to_status(launch_indexer_scan(a, st));
}

int dsa_indexer_score_mxfp4(const uint8_t* q_codes, const uint8_t* q_scales, const float* w,
                            const uint8_t* key_cache, int64_t num_pages,
                            const int32_t* block_table, int B, int max_pages,
                            const int32_t* row_req, const int32_t* row_len, int R, float* scores,
                            int64_t ld, void* workspace, size_t ws_bytes, void* stream) {
  int s = check_rows(B, max_pages, block_table, row_req, row_len, R);
  if (s) return s;
  if (R > 0 && (!q_codes || !q_scales || !w || !key_cache || !scores)) return DSA_ERR_INVALID_ARG;
  if (num_pages < 0 || ld < score_ld(max_pages) || ld % 4 != 0) return DSA_ERR_INVALID_ARG;
  if ((scores && !aligned(scores, 16)) || (key_cache && !aligned(key_cache, 16)) ||
      (q_codes && !aligned(q_codes, 16)) || (q_scales && !aligned(q_scales, 4)))
    return DSA_ERR_INVALID_ARG;
  s = check_workspace(workspace, ws_bytes, dsa_indexer_score_workspace_size(R));
  if (s) return s;
  cudaStream_t st = as_stream(stream);
  if ((s = clear_status(workspace, st))) return s;
  if (R == 0) return DSA_OK;
  ScanArgs a{q_codes, kQMxfp4, nullptr, w, key_cache, num_pages, block_table, B, max_pages,
             row_req, row_len, R, scores, ld, static_cast<uint8_t*>(workspace) + kStatusBytes,
             static_cast<uint32_t*>(workspace)};
  a.q_sf = q_scales;
  return to_status(launch_indexer_scan(a, st));
}

// ---------------------------------------------------------------- Select
size_t dsa_topk_workspace_size(int R, int64_t max_len, int k) {
  if (R < 0 || max_len < 0 || k < 1) return 0;
  return kStatusBytes + TopkLayout(R, max_len).bytes;
}

int dsa_topk(const float* scores, int64_t ld, const int32_t* row_len, int R, int64_t max_len,
             int k, int32_t* idx, void* workspace, size_t ws_bytes, void* stream) {
  if (R < 0 || max_len < 0 || ld < max_len || ld % 4 != 0) return DSA_ERR_INVALID_ARG;
  if (k < 1) return DSA_ERR_INVALID_ARG;
  if (k > kMaxTopk) return DSA_ERR_UNSUPPORTED;
  if (max_len > ((int64_t)1 << 31) - 1) return DSA_ERR_UNSUPPORTED;
  if (R > 65535) return DSA_ERR_UNSUPPORTED;
  if (R > 0 && (!scores || !row_len || !idx)) return DSA_ERR_INVALID_ARG;
  if (scores && !aligned(scores, 16)) return DSA_ERR_INVALID_ARG;
  int s = check_workspace(workspace, ws_bytes, dsa_topk_workspace_size(R, max_len, k));
  if (s) return s;
  cudaStream_t st = as_stream(stream);
  if ((s = clear_status(workspace, st))) return s;
  if (R == 0) return DSA_OK;
  TopkArgs a{scores, ld, row_len, R, max_len, k, idx,
             static_cast<uint8_t*>(workspace) + kStatusBytes, static_cast<uint32_t*>(workspace)};
  return to_status(launch_topk(a, st));
}

// ---------------------------------------------------------------- Write
namespace {
int write_kv(const void* k_raw, const float* gamma, const float* beta, float eps,
             const void* latent, float latent_scale, const int32_t* block_table, int B,
             int max_pages, const int32_t* tok_req, const int32_t* tok_pos, int T,
             uint8_t* key_cache, uint8_t* latent_cache, int64_t num_pages, uint32_t* dev_status,
             void* stream, bool mx_keys) {
  if (T < 0 || B < 0 || max_pages < 0 || num_pages < 0) return DSA_ERR_INVALID_ARG;
  if (!(latent_scale > 0.f) || !(latent_scale < INFINITY) || !(eps >= 0.f)) return DSA_ERR_INVALID_ARG;
  if (T > 0 && (B < 1 || max_pages < 1 || !k_raw || !gamma || !beta || !latent || !block_table ||
                !tok_req || !tok_pos || !key_cache || !latent_cache))
    return DSA_ERR_INVALID_ARG;
  if ((k_raw && !aligned(k_raw, 8)) || (latent && !aligned(latent, 16)) ||
      (gamma && !aligned(gamma, 16)) || (beta && !aligned(beta, 16)) ||
      (key_cache && !aligned(key_cache, 16)) || (latent_cache && !aligned(latent_cache, 16)))
    return DSA_ERR_INVALID_ARG;
  cudaStream_t st = as_stream(stream);
  if (dev_status && cudaMemsetAsync(dev_status, 0, 4, st) != cudaSuccess) return DSA_ERR_CUDA;
  if (T == 0) return DSA_OK;
  WriteArgs a{k_raw, gamma, beta, eps, latent, latent_scale, block_table, B, max_pages,
              tok_req, tok_pos, T, key_cache, latent_cache, num_pages, dev_status};
  a.mx_keys = mx_keys;
  return to_status(launch_write_kv(a, st));
}
}  // namespace

int dsa_write_kv(const void* k_raw, const float* gamma, const float* beta, float eps,
                 const void* latent, float latent_scale, const int32_t* block_table, int B,
                 int max_pages, const int32_t* tok_req, const int32_t* tok_pos, int T,
                 uint8_t* key_cache, uint8_t* latent_cache, int64_t num_pages,
                 uint32_t* dev_status, void* stream) {
  return write_kv(k_raw, gamma, beta, eps, latent, latent_scale, block_table, B, max_pages,
                  tok_req, tok_pos, T, key_cache, latent_cache, num_pages, dev_status, stream,
                  false);
}

int dsa_write_kv_mxfp4(const void* k_raw, const float* gamma, const float* beta, float eps,
                       const void* latent, float latent_scale, const int32_t* block_table,
                       int B, int max_pages, const int32_t* tok_req, const int32_t* tok_pos,
                       int T, uint8_t* key_cache, uint8_t* latent_cache, int64_t num_pages,
                       uint32_t* dev_status, void* stream) {
  return write_kv(k_raw, gamma, beta, eps, latent, latent_scale, block_table, B, max_pages,
                  tok_req, tok_pos, T, key_cache, latent_cache, num_pages, dev_status, stream,
                  true);
}

// ------------------------------------ Select under decode context parallelism
size_t dsa_topk_dcp_workspace_size(int R, int64_t max_len, int k, int W) {
  if (R < 0 || max_len < 0 || k < 1 || W < 1) return 0;
  return kStatusBytes + dcp_scratch_bytes(R, max_len, k, W);
}

int dsa_topk_dcp(const float* scores, int64_t ld, const int32_t* row_len, int R, int64_t max_len,
                 int k, int W, int32_t* idx, uint32_t* resend, void* workspace, size_t ws_bytes,
                 void* stream) {
  if (R < 0 || max_len < 0 || ld < max_len || ld % 4 != 0) return DSA_ERR_INVALID_ARG;
  if (k < 1 || W < 1) return DSA_ERR_INVALID_ARG;
  if (k > kMaxTopk || W > DSA_MAX_DCP_SHARDS) return DSA_ERR_UNSUPPORTED;
  if (max_len > ((int64_t)1 << 31) - 1) return DSA_ERR_UNSUPPORTED;
  if ((int64_t)R * W > 65535) return DSA_ERR_UNSUPPORTED;
  if (R > 0 && (!scores || !row_len || !idx)) return DSA_ERR_INVALID_ARG;
  if (scores && !aligned(scores, 16)) return DSA_ERR_INVALID_ARG;
  int s = check_workspace(workspace, ws_bytes, dsa_topk_dcp_workspace_size(R, max_len, k, W));
  if (s) return s;
  cudaStream_t st = as_stream(stream);
  if ((s = clear_status(workspace, st))) return s;
  if (R == 0) return DSA_OK;
  DcpArgs a{scores, ld, row_len, R, max_len, k, W, idx, resend,
            static_cast<uint8_t*>(workspace) + kStatusBytes, static_cast<uint32_t*>(workspace)};
  return to_status(launch_topk_dcp(a, st));
}

// ---------------------------------------------------------------- Attend
size_t dsa_sparse_mla_workspace_size(int R, int H, int k) {
  if (R < 0 || H < 1 || k < 1) return 0;
  return kStatusBytes + MlaLayout(R, H, k).bytes;
}

namespace {
int sparse_mla(bool nvfp4, const void* q, int H, float softmax_scale, const uint8_t* latent_cache,
               int64_t num_pages, float latent_scale, const int32_t* block_table, int B,
               int max_pages, const int32_t* row_req, const int32_t* row_len, const int32_t* idx,
               int k, int R, void* out, float* lse, void* workspace, size_t ws_bytes,
               void* stream) {
  int s = check_rows(B, max_pages, block_table, row_req, row_len, R);
  if (s) return s;
  if (!supported_heads(H)) return DSA_ERR_UNSUPPORTED;
  if (k < 1) return DSA_ERR_INVALID_ARG;
  if (k > kMaxTopk) return DSA_ERR_UNSUPPORTED;
  if (num_pages < 0) return DSA_ERR_INVALID_ARG;
  if (R > 0 && (!q || !latent_cache || !idx || !out)) return DSA_ERR_INVALID_ARG;
  if ((q && !aligned(q, 16)) || (latent_cache && !aligned(latent_cache, 16)) ||
      (out && !aligned(out, 16)))
    return DSA_ERR_INVALID_ARG;
  s = check_workspace(workspace, ws_bytes, dsa_sparse_mla_workspace_size(R, H, k));
  if (s) return s;
  cudaStream_t st = as_stream(stream);
  if ((s = clear_status(workspace, st))) return s;
  if (R == 0) return DSA_OK;
  MlaArgs a{q, H, softmax_scale, latent_cache, num_pages, latent_scale, block_table, B,
            max_pages, row_req, row_len, idx, k, R, out, lse,
            static_cast<uint8_t*>(workspace) + kStatusBytes, static_cast<uint32_t*>(workspace)};
  a.nvfp4 = nvfp4;
  return to_status(launch_sparse_mla(a, st));
}
}  // namespace

int dsa_sparse_mla_decode(const void* q, int H, float softmax_scale, const uint8_t* latent_cache,
                          int64_t num_pages, float latent_scale, const int32_t* block_table,
                          int B, int max_pages, const int32_t* row_req, const int32_t* row_len,
                          const int32_t* idx, int k, int R, void* out, float* lse,
                          void* workspace, size_t ws_bytes, void* stream) {
  return sparse_mla(false, q, H, softmax_scale, latent_cache, num_pages, latent_scale,
                    block_table, B, max_pages, row_req, row_len, idx, k, R, out, lse, workspace,
                    ws_bytes, stream);
}

int dsa_sparse_mla_decode_nvfp4(const void* q, int H, float softmax_scale,
                                const uint8_t* latent_cache, int64_t num_pages,
                                float latent_scale, const int32_t* block_table, int B,
                                int max_pages, const int32_t* row_req, const int32_t* row_len,
                                const int32_t* idx, int k, int R, void* out, float* lse,
                                void* workspace, size_t ws_bytes, void* stream) {
  return sparse_mla(true, q, H, softmax_scale, latent_cache, num_pages, latent_scale,
                    block_table, B, max_pages, row_req, row_len, idx, k, R, out, lse, workspace,
                    ws_bytes, stream);
}

// ---------------------------------------------------------------- fused step
namespace {
struct StepLayout {
  size_t scores, idx, topk, mla, scan, bytes;
  StepLayout(int R, int max_pages, int H, int k) {
    size_t o = kStatusBytes;
    scores = o; o = align_up(o + (size_t)R * score_ld(max_pages) * 4);
    idx = o;    o = align_up(o + (size_t)R * k * 4);
    scan = o;   o = align_up(o + scan_scratch_bytes(R));
    topk = o;   o = align_up(o + TopkLayout(R, score_ld(max_pages)).bytes);
    mla = o;    o = align_up(o + MlaLayout(R, H, k).bytes);
    bytes = o;
  }
};
}  // namespace

size_t dsa_decode_step_workspace_size(int B, int R, int max_pages, int H, int k) {
  if (B < 0 || R < 0 || max_pages < 0 || H < 1 || k < 1) return 0;
  return StepLayout(R, max_pages, H, k).bytes;
}

namespace {
// The fused step for both cache formats: q_dtype DSA_BF16 / DSA_E4M3 with FP8
// keys and FP8 latent rows, or kQMxfp4 (q_idx = E2M1 codes, q_sf = E8M0
// scales) with MXFP4 keys and NVFP4 latent rows.
int decode_step(const void* q_idx, int q_dtype, const float* q_scale, const uint8_t* q_sf,
                const float* w, const uint8_t* key_cache, const uint8_t* latent_cache,
                int64_t num_pages, float latent_scale, const int32_t* block_table, int B,
                int max_pages, const int32_t* row_req, const int32_t* row_len, int R,
                const void* q, int H, float softmax_scale, int k, void* out, float* lse,
                int32_t* idx_out, void* workspace, size_t ws_bytes, void* stream) {
  const bool fp4 = q_dtype == kQMxfp4;
  int s = check_rows(B, max_pages, block_table, row_req, row_len, R);
  if (s) return s;
  if (!supported_heads(H)) return DSA_ERR_UNSUPPORTED;
  if (k < 1) return DSA_ERR_INVALID_ARG;
  if (k > kMaxTopk) return DSA_ERR_UNSUPPORTED;
  if (num_pages < 0) return DSA_ERR_INVALID_ARG;
  if (R > 0 && (!q_idx || !w || !key_cache || !latent_cache || !q || !out))
    return DSA_ERR_INVALID_ARG;
  if (q_dtype == DSA_E4M3 && R > 0 && !q_scale) return DSA_ERR_INVALID_ARG;
  if (fp4 && R > 0 && !q_sf) return DSA_ERR_INVALID_ARG;
  if ((key_cache && !aligned(key_cache, 16)) || (latent_cache && !aligned(latent_cache, 16)) ||
      (q && !aligned(q, 16)) || (out && !aligned(out, 16)) ||
      (fp4 && q_idx && !aligned(q_idx, 16)) || (fp4 && q_sf && !aligned(q_sf, 4)))
    return DSA_ERR_INVALID_ARG;
  const StepLayout L(R, max_pages, H, k);
  s = check_workspace(workspace, ws_bytes, L.bytes);
  if (s) return s;
  cudaStream_t st = as_stream(stream);
  if (R == 0) return clear_status(workspace, st);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint32_t* status = reinterpret_cast<uint32_t*>(ws);
  float* scores = reinterpret_cast<float*>(ws + L.scores);
  int32_t* idx = idx_out ? idx_out : reinterpret_cast<int32_t*>(ws + L.idx);
  const int64_t ld = score_ld(max_pages);

  ScanArgs sa{q_idx, q_dtype, q_scale, w, key_cache, num_pages, block_table, B, max_pages,
              row_req, row_len, R, scores, ld, ws + L.scan, status};
  sa.q_sf = q_sf;
  sa.clear_status = true;                          // the step's first kernel clears the word
  cudaError_t e = launch_indexer_scan(sa, st);
  if (e != cudaSuccess) return to_status(e);
  TopkArgs ta{scores, ld, row_len, R, ld, k, idx, ws + L.topk, status, true};
  e = launch_topk(ta, st);
  if (e != cudaSuccess) return to_status(e);
  MlaArgs ma{q, H, softmax_scale, latent_cache, num_pages, latent_scale, block_table, B,
             max_pages, row_req, row_len, idx, k, R, out, lse, ws + L.mla, status, true};
  ma.nvfp4 = fp4;
  return to_status(launch_sparse_mla(ma, st));
}
}  // namespace

int dsa_decode_step(const void* q_idx, int q_dtype, const float* q_scale, const float* w,
                    const uint8_t* key_cache, const uint8_t* latent_cache, int64_t num_pages,
                    float latent_scale, const int32_t* block_table, int B, int max_pages,
                    const int32_t* row_req, const int32_t* row_len, int R, const void* q, int H,
                    float softmax_scale, int k, void* out, float* lse, int32_t* idx_out,
                    void* workspace, size_t ws_bytes, void* stream) {
  if (q_dtype != DSA_BF16 && q_dtype != DSA_E4M3) return DSA_ERR_UNSUPPORTED;
  return decode_step(q_idx, q_dtype, q_scale, nullptr, w, key_cache, latent_cache, num_pages,
                     latent_scale, block_table, B, max_pages, row_req, row_len, R, q, H,
                     softmax_scale, k, out, lse, idx_out, workspace, ws_bytes, stream);
}

int dsa_decode_step_fp4(const uint8_t* q_codes, const uint8_t* q_scales, const float* w,
                        const uint8_t* key_cache, const uint8_t* latent_cache, int64_t num_pages,
                        float latent_scale, const int32_t* block_table, int B, int max_pages,
                        const int32_t* row_req, const int32_t* row_len, int R, const void* q,
                        int H, float softmax_scale, int k, void* out, float* lse,
                        int32_t* idx_out, void* workspace, size_t ws_bytes, void* stream) {
  return decode_step(q_codes, kQMxfp4, nullptr, q_scales, w, key_cache, latent_cache, num_pages,
                     latent_scale, block_table, B, max_pages, row_req, row_len, R, q, H,
                     softmax_scale, k, out, lse, idx_out, workspace, ws_bytes, stream);
}

size_t dsa_selftest_workspace_size(void) { return selftest_workspace_bytes(); }

int dsa_selftest_bounded_wait(int wait_us, void* workspace, size_t ws_bytes, void* stream) {
  if (wait_us < 1 || wait_us > 1000000) return DSA_ERR_INVALID_ARG;
  int s = check_workspace(workspace, ws_bytes, selftest_workspace_bytes());
  if (s) return s;
  int dev = 0, khz = 0;
  if ((s = to_status(cudaGetDevice(&dev)))) return s;
  if ((s = to_status(cudaDeviceGetAttribute(&khz, cudaDevAttrClockRate, dev)))) return s;
  cudaStream_t st = as_stream(stream);
  if ((s = clear_status(workspace, st))) return s;
  const long long cycles = (long long)wait_us * (khz > 0 ? khz : 2000000) / 1000;
  return to_status(launch_selftest_wait(workspace, cycles, st));
}

int dsa_check_device_status(const void* workspace, void* stream, uint32_t* bits) {
  if (!workspace) return DSA_ERR_WORKSPACE;
  uint32_t v = 0;
  int s = to_status(cudaStreamSynchronize(as_stream(stream)));
  if (s) return s;
  if ((s = to_status(cudaMemcpy(&v, workspace, 4, cudaMemcpyDeviceToHost)))) return s;
  if (bits) *bits = v;
  return v ? DSA_ERR_DEVICE_CHECK : DSA_OK;
}

}  // extern "C"
