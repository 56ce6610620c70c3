// smla.cu -- sparse MLA over the selected latent rows (the Attend step) and
// the log-sum-exp combine of its split partials.
//
// For row r, head h and the valid selected tokens j:
//   x_j = softmax_scale * latent_scale * (q[r][h] . dec(L8_j))       (576 dims)
//   o   = sum_j softmax(x)_j * latent_scale * dec(L8_j)[0:512],  lse = ln sum_j e^{x_j}
// (vLLM Day-0 post on Kimi K3.1 Pro, "What Kimi K3.1 Pro changes": MLA runs
// exactly over only the selected tokens; TokenSpeed post, "Sparse attention
// in Kimi K3.1 Pro": all heads attend to the selected tokens; AMD Instinct
// post, overview "MLA": 512 KV + 64 RoPE dims, the 512 part is the value.)
//
// The selected-token dimension is split over CTAs; each split emits a
// normalised partial (o_s, lse_s) and the combine forms
//   lse = ln sum_s e^{lse_s},  o = sum_s e^{lse_s - lse} o_s
// -- the same log-sum-exp merge the pages use to combine per-GPU partial
// outputs under decode context parallelism (vLLM post, "Decode context
// parallelism with a sparse indexer"; TokenSpeed post, "Sharding long
// contexts with decode context parallelism", step 4).
//
// This file holds the CUDA-core version: 256 threads per CTA over a group of
// up to 64 heads, 16 selected rows per batch, online softmax in registers.
#include <math.h>

#include "dsa_common.cuh"

namespace dsa {
namespace {

constexpr int kMlaThreads = 256;
constexpr int kBatch = 16;

template <int HG>  // heads per CTA: 16, 32 or 64
__global__ void __launch_bounds__(kMlaThreads)
smla_cuda_core_kernel(const __nv_bfloat16* __restrict__ q, int H, float softmax_scale,
                      const uint8_t* __restrict__ latent_cache, int64_t num_pages,
                      float latent_scale, const int32_t* __restrict__ block_table, int B,
                      int max_pages, const int32_t* __restrict__ row_req,
                      const int32_t* __restrict__ row_len, const int32_t* __restrict__ idx, int k,
                      int nsplit, float* __restrict__ part_o, float* __restrict__ part_lse,
                      uint32_t* status) {
  constexpr int TPH = kMlaThreads / HG;  // threads per head
  constexpr int DPT = kVDim / TPH;       // output dims per thread
  constexpr int LPT = kLatDim / TPH;     // logit dims per thread
  extern __shared__ __align__(16) uint8_t smem_raw[];
  __nv_bfloat16* qs = reinterpret_cast<__nv_bfloat16*>(smem_raw);                 // [HG][576]
  float* lat = reinterpret_cast<float*>(smem_raw + HG * kLatDim * 2);            // [kBatch][576]
  __shared__ const uint8_t* rows[kBatch];

  const int split = blockIdx.x, r = blockIdx.y, hg0 = blockIdx.z * HG;
  const int tid = threadIdx.x;
  const int hl = tid / TPH;          // head within the group
  const int lane = tid % TPH;        // position within the head's thread group
  const int req = row_req[r];
  const int len = row_len[r];
  const bool row_valid = req >= 0 && req < B && len >= 0 && (int64_t)len <= (int64_t)max_pages * kPage;
  if (!row_valid && split == 0 && blockIdx.z == 0 && tid == 0) raise_dev(status, DSA_DEV_BAD_ROW);

  const int per = (k + nsplit - 1) / nsplit;
  const int j0 = split * per;
  const int j1 = min(k, j0 + per);

  for (int i = tid; i < HG * kLatDim / 8; i += kMlaThreads) {
    const int h = i / (kLatDim / 8), c = i % (kLatDim / 8);
    reinterpret_cast<uint4*>(qs)[i] =
        __ldg(reinterpret_cast<const uint4*>(q + ((size_t)r * H + hg0 + h) * kLatDim) + c);
  }

  float o[DPT];
#pragma unroll
  for (int i = 0; i < DPT; ++i) o[i] = 0.f;
  float m = -INFINITY, l = 0.f;
  const float xscale = softmax_scale * latent_scale;

  for (int jb = j0; jb < j1; jb += kBatch) {
    __syncthreads();  // previous batch fully consumed (and q loaded on the first pass)
    if (tid < kBatch) {
      const uint8_t* p = nullptr;
      const int j = jb + tid;
      if (row_valid && j < j1) {
        const int t = idx[(size_t)r * k + j];
        if (t >= len) {
          raise_dev(status, DSA_DEV_BAD_INDEX);
        } else if (t >= 0) {
          const int page = block_table[(size_t)req * max_pages + t / kPage];
          if (page < 0 || (int64_t)page >= num_pages)
            raise_dev(status, DSA_DEV_BAD_PAGE);
          else
            p = latent_cache + ((size_t)page * kPage + (t % kPage)) * kLatDim;
        }
      }
      rows[tid] = p;
    }
    __syncthreads();
    for (int i = tid; i < kBatch * (kLatDim / 16); i += kMlaThreads) {
      const int j = i / (kLatDim / 16), c = i % (kLatDim / 16);
      float* dst = lat + j * kLatDim + c * 16;
      const uint8_t* src = rows[j];
      if (src) {
        const uint4 raw = __ldg(reinterpret_cast<const uint4*>(src) + c);
        const uint32_t wds[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float2 a = e4m3x2_to_float2((uint16_t)(wds[u] & 0xFFFF));
          const float2 b = e4m3x2_to_float2((uint16_t)(wds[u] >> 16));
          dst[4 * u + 0] = a.x; dst[4 * u + 1] = a.y; dst[4 * u + 2] = b.x; dst[4 * u + 3] = b.y;
        }
      } else {
#pragma unroll
        for (int u = 0; u < 16; ++u) dst[u] = 0.f;
      }
    }
    __syncthreads();

    float x[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) x[j] = 0.f;
    const __nv_bfloat16* qh = qs + hl * kLatDim;
#pragma unroll 4
    for (int i = 0; i < LPT; ++i) {
      const int d = lane + i * TPH;
      const float qv = __bfloat162float(qh[d]);
#pragma unroll
      for (int j = 0; j < kBatch; ++j) x[j] = fmaf(qv, lat[j * kLatDim + d], x[j]);
    }
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
#pragma unroll
      for (int off = TPH / 2; off > 0; off >>= 1) x[j] += __shfl_xor_sync(0xffffffffu, x[j], off);
    }
    float bmax = -INFINITY;
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      x[j] = rows[j] ? x[j] * xscale : -INFINITY;
      bmax = fmaxf(bmax, x[j]);
    }
    if (bmax == -INFINITY) continue;  // nothing valid in this batch (uniform per CTA)
    const float m_new = fmaxf(m, bmax);
    const float corr = __expf(m - m_new);  // m = -inf -> 0
    float p[kBatch];
    float psum = 0.f;
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      p[j] = __expf(x[j] - m_new);
      psum += p[j];
    }
    l = l * corr + psum;
    m = m_new;
#pragma unroll
    for (int i = 0; i < DPT; ++i) {
      const int d = lane + i * TPH;
      float acc = o[i] * corr;
#pragma unroll
      for (int j = 0; j < kBatch; ++j) acc = fmaf(p[j], lat[j * kLatDim + d], acc);
      o[i] = acc;
    }
  }

  const int h = hg0 + hl;
  const size_t pbase = ((size_t)r * nsplit + split) * H + h;
  const float inv = l > 0.f ? latent_scale / l : 0.f;
#pragma unroll
  for (int i = 0; i < DPT; ++i) part_o[pbase * kVDim + lane + i * TPH] = o[i] * inv;
  if (lane == 0) part_lse[pbase] = l > 0.f ? m + logf(l) : -INFINITY;
}

// One CTA per (row, head): merge the splits' partials by log-sum-exp.
__global__ void __launch_bounds__(128)
mla_combine_kernel(const float* __restrict__ part_o, const float* __restrict__ part_lse, int H,
                   int nsplit, __nv_bfloat16* __restrict__ out, float* __restrict__ lse) {
  const int r = blockIdx.x / H, h = blockIdx.x % H;
  float M = -INFINITY;
  for (int s = 0; s < nsplit; ++s) M = fmaxf(M, part_lse[((size_t)r * nsplit + s) * H + h]);
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  float Z = 0.f;
  if (M != -INFINITY) {
    for (int s = 0; s < nsplit; ++s) {
      const size_t pb = ((size_t)r * nsplit + s) * H + h;
      const float ls = part_lse[pb];
      if (ls == -INFINITY) continue;
      const float ws = __expf(ls - M);
      Z += ws;
      const float4 v = __ldg(reinterpret_cast<const float4*>(part_o + pb * kVDim) + threadIdx.x);
      acc[0] = fmaf(ws, v.x, acc[0]);
      acc[1] = fmaf(ws, v.y, acc[1]);
      acc[2] = fmaf(ws, v.z, acc[2]);
      acc[3] = fmaf(ws, v.w, acc[3]);
    }
  }
  const float inv = Z > 0.f ? 1.f / Z : 0.f;
  __nv_bfloat16* dst = out + ((size_t)r * H + h) * kVDim + threadIdx.x * 4;
  dst[0] = __float2bfloat16_rn(acc[0] * inv);
  dst[1] = __float2bfloat16_rn(acc[1] * inv);
  dst[2] = __float2bfloat16_rn(acc[2] * inv);
  dst[3] = __float2bfloat16_rn(acc[3] * inv);
  if (lse && threadIdx.x == 0) lse[(size_t)r * H + h] = Z > 0.f ? M + logf(Z) : -INFINITY;
}

template <int HG>
cudaError_t launch_smla_group(const MlaArgs& a, float* part_o, float* part_lse, int nsplit,
                              cudaStream_t st) {
  const size_t smem = (size_t)HG * kLatDim * 2 + (size_t)kBatch * kLatDim * 4;
  cudaError_t e = cudaFuncSetAttribute(smla_cuda_core_kernel<HG>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(nsplit, a.R, a.H / HG);
  smla_cuda_core_kernel<HG><<<grid, kMlaThreads, smem, st>>>(
      static_cast<const __nv_bfloat16*>(a.q), a.H, a.softmax_scale, a.latent_cache, a.num_pages,
      a.latent_scale, a.block_table, a.B, a.max_pages, a.row_req, a.row_len, a.idx, a.k, nsplit,
      part_o, part_lse, a.status);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_sparse_mla(const MlaArgs& a, cudaStream_t st) {
  if (a.R == 0) return cudaSuccess;
  const MlaLayout L(a.R, a.H, a.k);
  float* part_o = reinterpret_cast<float*>(a.scratch + L.part_o);
  float* part_lse = reinterpret_cast<float*>(a.scratch + L.part_lse);
  cudaError_t e;
  if (a.H == 16) e = launch_smla_group<16>(a, part_o, part_lse, L.nsplit, st);
  else if (a.H == 32) e = launch_smla_group<32>(a, part_o, part_lse, L.nsplit, st);
  else e = launch_smla_group<64>(a, part_o, part_lse, L.nsplit, st);
  if (e != cudaSuccess) return e;
  mla_combine_kernel<<<a.R * a.H, 128, 0, st>>>(part_o, part_lse, a.H, L.nsplit,
                                                static_cast<__nv_bfloat16*>(a.out), a.lse);
  return cudaGetLastError();
}

}  // namespace dsa
