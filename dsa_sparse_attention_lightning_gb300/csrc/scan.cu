// scan.cu -- lightning-indexer scan (the Score step).
//
// score[r][s] = sum_h w[r][h] * ReLU(q[r][h] . key[s]) * ks[s] for s < row_len[r]
// (TokenSpeed post on Kimi K3.1 Pro, "Integrating sparse attention with the
// K3 stack", step 2; vLLM Day-0 post, "What Kimi K3.1 Pro changes": 32 heads
// x 128 dims, one FP8 key per token).  The key scale is a positive absmax
// scale ("quantizes it to FP8 with a single scale", step 1), so
// ReLU(x * ks) = ks * ReLU(x) and the scale is applied once after the head sum.
//
// This file holds the CUDA-core kernel: one CTA per (64-token page, row),
// 4 threads per token each owning 8 heads.
#include "dsa_common.cuh"

namespace dsa {
namespace {

constexpr int kScanThreads = 256;

template <bool kFp8Q>
__global__ void __launch_bounds__(kScanThreads)
scan_cuda_core_kernel(const void* __restrict__ q_idx, const float* __restrict__ q_scale,
                      const float* __restrict__ w, const uint8_t* __restrict__ key_cache,
                      int64_t num_pages, const int32_t* __restrict__ block_table, int B,
                      int max_pages, const int32_t* __restrict__ row_req,
                      const int32_t* __restrict__ row_len, float* __restrict__ scores, int64_t ld,
                      uint32_t* status) {
  const int r = blockIdx.y;
  const int tile = blockIdx.x;
  const int req = row_req[r];
  const int len = row_len[r];
  if (req < 0 || req >= B || len < 0 || (int64_t)len > (int64_t)max_pages * kPage) {
    if (tile == 0 && threadIdx.x == 0) raise_dev(status, DSA_DEV_BAD_ROW);
    return;
  }
  const int t0 = tile * kPage;
  if (t0 >= len) return;
  const int page = block_table[(int64_t)req * max_pages + tile];
  if (page < 0 || (int64_t)page >= num_pages) {
    if (threadIdx.x == 0) raise_dev(status, DSA_DEV_BAD_PAGE);
    return;
  }

  __shared__ float qs[kIdxHeads][kIdxDim + 1];      // +1: heads land in distinct banks
  __shared__ float ws[kIdxHeads];
  __shared__ __align__(16) uint8_t kb[kPage * kIdxDim];
  __shared__ float ksc[kPage];

  for (int i = threadIdx.x; i < kIdxHeads * kIdxDim; i += kScanThreads) {
    const int h = i / kIdxDim, d = i % kIdxDim;
    float v;
    if (kFp8Q)
      v = e4m3_to_float(static_cast<const uint8_t*>(q_idx)[(size_t)r * kIdxHeads * kIdxDim + i]) *
          q_scale[(size_t)r * kIdxHeads + h];
    else
      v = __bfloat162float(
          static_cast<const __nv_bfloat16*>(q_idx)[(size_t)r * kIdxHeads * kIdxDim + i]);
    qs[h][d] = v;
  }
  if (threadIdx.x < kIdxHeads) ws[threadIdx.x] = w[(size_t)r * kIdxHeads + threadIdx.x];
  const uint8_t* pg = key_cache + (size_t)page * kKeyPageBytes;
  for (int i = threadIdx.x; i < kPage * kIdxDim / 16; i += kScanThreads)
    reinterpret_cast<uint4*>(kb)[i] = __ldg(reinterpret_cast<const uint4*>(pg) + i);
  if (threadIdx.x < kPage)
    ksc[threadIdx.x] = __ldg(reinterpret_cast<const float*>(pg + kKeyScaleOffset) + threadIdx.x);
  __syncthreads();

  const int tok = threadIdx.x >> 2;
  const int hg = threadIdx.x & 3;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
#pragma unroll 2
  for (int d0 = 0; d0 < kIdxDim; d0 += 16) {
    const uint4 raw = *reinterpret_cast<const uint4*>(kb + tok * kIdxDim + d0);
    const uint32_t wds[4] = {raw.x, raw.y, raw.z, raw.w};
    float kf[16];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 lo = e4m3x2_to_float2((uint16_t)(wds[j] & 0xFFFF));
      const float2 hi = e4m3x2_to_float2((uint16_t)(wds[j] >> 16));
      kf[4 * j + 0] = lo.x; kf[4 * j + 1] = lo.y; kf[4 * j + 2] = hi.x; kf[4 * j + 3] = hi.y;
    }
#pragma unroll
    for (int hh = 0; hh < 8; ++hh) {
      const float* qrow = &qs[hg * 8 + hh][d0];
#pragma unroll
      for (int dd = 0; dd < 16; ++dd) acc[hh] = fmaf(qrow[dd], kf[dd], acc[hh]);
    }
  }
  float part = 0.f;
#pragma unroll
  for (int hh = 0; hh < 8; ++hh) part = fmaf(ws[hg * 8 + hh], fmaxf(acc[hh], 0.f), part);
  part += __shfl_xor_sync(0xffffffffu, part, 1);
  part += __shfl_xor_sync(0xffffffffu, part, 2);
  if (hg == 0 && t0 + tok < len) scores[(size_t)r * ld + t0 + tok] = part * ksc[tok];
}

}  // namespace

cudaError_t launch_indexer_scan(const ScanArgs& a, cudaStream_t st) {
  if (a.R == 0 || a.max_pages == 0) return cudaSuccess;
  dim3 grid(a.max_pages, a.R);
  if (a.q_dtype == DSA_E4M3)
    scan_cuda_core_kernel<true><<<grid, kScanThreads, 0, st>>>(
        a.q_idx, a.q_scale, a.w, a.key_cache, a.num_pages, a.block_table, a.B, a.max_pages,
        a.row_req, a.row_len, a.scores, a.ld, a.status);
  else
    scan_cuda_core_kernel<false><<<grid, kScanThreads, 0, st>>>(
        a.q_idx, a.q_scale, a.w, a.key_cache, a.num_pages, a.block_table, a.B, a.max_pages,
        a.row_req, a.row_len, a.scores, a.ld, a.status);
  return cudaGetLastError();
}

}  // namespace dsa
