// write.cu -- the Write step: a new token's index key and latent row into the
// paged FP8 caches.
//
// One fused kernel normalizes the new token's index key, quantizes it to FP8
// with a single scale and writes it into the cache, and the latent row is
// written next to it (TokenSpeed post on Kimi K3.1 Pro, "Integrating sparse
// attention with the K3 stack", step 1 "Write", and the kernel table: one
// kernel for the latent row, one for the index key; the only key
// normalization the loader accepts is LayerNorm).  Per new token t:
//   k      = gamma * (x - mean(x)) / sqrt(var(x) + eps) + beta   (x = 128 bf16
//            values, mean and biased variance over the dims)
//   ks     = max_d |k[d]| / 448   (1 when k is all zero)
//   codes  = E4M3(k / ks)         (round to nearest even, saturating)
// into page block_table[req][pos / 64], slot pos % 64: the codes at slot * 128
// of the page's key block and ks (fp32) at 64 * 128 + slot * 4 ("Storing index
// keys in the flat KV cache": 128 FP8 values and one four-byte scale), and
// E4M3(latent / latent_scale) (576 values) at latent_cache[page][slot].
//
// One warp per token: lane l holds key dims 4l .. 4l + 3 (the mean, variance
// and absmax are warp reductions, the codes one 4-byte store per lane) and
// 16-byte chunks l and l + 32 of the 576-byte latent row.  Memory bound
// (256 + 1152 bytes read, 132 + 576 written per token).
//
// MXFP4 index keys (vLLM Day-0 post on Kimi K3.1 Pro, "Hybrid KV cache without
// padding": 68 bytes per key; one E8M0 scale per 32 values): the normalized
// key is quantized per block of 32 dims (OCP Microscaling v1.0 conversion):
//   e      = floor(log2(max |k|)) - 2, clamped to [-127, 127] (-127 for an
//            all-zero block)
//   codes  = E2M1(k / 2^e)   (round to nearest even on the grid 0, 0.5, 1,
//            1.5, 2, 3, 4, 6, beyond 6 clamped to 6)
// into page block_table[req][pos / 64] (4352 bytes): the 64 code bytes at
// slot * 64 (dim 2j in the low nibble of byte j), the four scale bytes
// e + 127 at 64 * 64 + slot * 4.  A block is 8 lanes.
#include "dsa_common.cuh"

namespace dsa {
namespace {

constexpr int kWarps = 8;

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  return (uint32_t)__nv_cvt_float_to_fp8(a, __NV_SATFINITE, __NV_E4M3) |
         ((uint32_t)__nv_cvt_float_to_fp8(b, __NV_SATFINITE, __NV_E4M3) << 8) |
         ((uint32_t)__nv_cvt_float_to_fp8(c, __NV_SATFINITE, __NV_E4M3) << 16) |
         ((uint32_t)__nv_cvt_float_to_fp8(d, __NV_SATFINITE, __NV_E4M3) << 24);
}

// E2M1 code of x (|x| < 8 after the block scaling): the grid's midpoints 0.25,
// 0.75, 1.25, 1.75, 2.5, 3.5 and 5 are counted, a value at a midpoint going to
// the neighbour with an even code.
__device__ __forceinline__ uint32_t e2m1(float x) {
  const float a = fabsf(x);
  const uint32_t m = (a > 0.25f) + (a >= 0.75f) + (a > 1.25f) + (a >= 1.75f) + (a > 2.5f) +
                     (a >= 3.5f) + (a > 5.f);
  return m | (signbit(x) ? 8u : 0u);
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

template <bool kMx>
__global__ void __launch_bounds__(kWarps * 32)
write_kv_kernel(const uint16_t* __restrict__ k_raw, const float* __restrict__ gamma,
                const float* __restrict__ beta, float eps, const uint16_t* __restrict__ latent,
                float latent_scale, const int32_t* __restrict__ block_table, int B, int max_pages,
                const int32_t* __restrict__ tok_req, const int32_t* __restrict__ tok_pos, int T,
                uint8_t* __restrict__ key_cache, uint8_t* __restrict__ latent_cache,
                int64_t num_pages, uint32_t* status) {
  pdl_trigger();
  pdl_wait();
  const int t = blockIdx.x * kWarps + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (t >= T) return;
  const int req = tok_req[t], pos = tok_pos[t];
  if (req < 0 || req >= B || pos < 0 || (int64_t)pos >= (int64_t)max_pages * kPage) {
    if (lane == 0) raise_dev(status, DSA_DEV_BAD_ROW);
    return;
  }
  const int page = block_table[(size_t)req * max_pages + pos / kPage];
  if (page < 0 || (int64_t)page >= num_pages) {
    if (lane == 0) raise_dev(status, DSA_DEV_BAD_PAGE);
    return;
  }
  const int slot = pos % kPage;

  // ---- index key: LayerNorm, absmax scale, E4M3 codes
  const uint2 raw = *reinterpret_cast<const uint2*>(k_raw + (size_t)t * kIdxDim + 4 * lane);
  const float x[4] = {bf16_lo(raw.x), bf16_hi(raw.x), bf16_lo(raw.y), bf16_hi(raw.y)};
  const float mean = warp_sum((x[0] + x[1]) + (x[2] + x[3])) / (float)kIdxDim;
  float sq = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) sq = fmaf(x[i] - mean, x[i] - mean, sq);
  const float var = warp_sum(sq) / (float)kIdxDim;
  const float sd = sqrtf(var + eps);
  const float4 g = *reinterpret_cast<const float4*>(gamma + 4 * lane);
  const float4 bt = *reinterpret_cast<const float4*>(beta + 4 * lane);
  const float k[4] = {g.x * ((x[0] - mean) / sd) + bt.x, g.y * ((x[1] - mean) / sd) + bt.y,
                      g.z * ((x[2] - mean) / sd) + bt.z, g.w * ((x[3] - mean) / sd) + bt.w};
  const float lmax = fmaxf(fmaxf(fabsf(k[0]), fabsf(k[1])), fmaxf(fabsf(k[2]), fabsf(k[3])));
  if constexpr (kMx) {
    float bmax = lmax;                              // the 8 lanes of this lane's block
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) bmax = fmaxf(bmax, __shfl_xor_sync(0xffffffffu, bmax, o));
    // floor(log2(bmax)) is the exponent field of a normal bmax; a subnormal or
    // zero bmax lands below -127 and is clamped
    const int e = min(max((int)(__float_as_uint(bmax) >> 23) - 127 - 2, -127), 127);
    uint32_t c = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) c |= e2m1(ldexpf(k[i], -e)) << (4 * i);
    uint8_t* kp = key_cache + (size_t)page * kMxKeyPageBytes;
    *reinterpret_cast<uint16_t*>(kp + slot * (kIdxDim / 2) + 2 * lane) = (uint16_t)c;
    const uint32_t sc = (uint32_t)(e + 127);        // lanes 0, 8, 16, 24 hold blocks 0-3
    const uint32_t word = __shfl_sync(0xffffffffu, sc, 0) | (__shfl_sync(0xffffffffu, sc, 8) << 8) |
                          (__shfl_sync(0xffffffffu, sc, 16) << 16) |
                          (__shfl_sync(0xffffffffu, sc, 24) << 24);
    if (lane == 0)
      *reinterpret_cast<uint32_t*>(kp + kPage * (kIdxDim / 2) + slot * 4) = word;
  } else {
    const float amax = warp_max(lmax);
    const float ks = amax > 0.f ? amax / 448.f : 1.f;
    uint8_t* kp = key_cache + (size_t)page * kKeyPageBytes;
    *reinterpret_cast<uint32_t*>(kp + slot * kIdxDim + 4 * lane) =
        e4m3x4(k[0] / ks, k[1] / ks, k[2] / ks, k[3] / ks);
    if (lane == 0) *reinterpret_cast<float*>(kp + kKeyScaleOffset + slot * 4) = ks;
  }

  // ---- latent row: 36 chunks of 16 codes (32 bytes of bf16 in each)
  const uint4* src = reinterpret_cast<const uint4*>(latent + (size_t)t * kLatDim);
  uint4* dst = reinterpret_cast<uint4*>(latent_cache + ((size_t)page * kPage + slot) * kLatDim);
  for (int c = lane; c < kLatDim / 16; c += 32) {
    const uint4 a = src[2 * c], b = src[2 * c + 1];
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      o[q] = e4m3x4(bf16_lo(w[2 * q]) / latent_scale, bf16_hi(w[2 * q]) / latent_scale,
                    bf16_lo(w[2 * q + 1]) / latent_scale, bf16_hi(w[2 * q + 1]) / latent_scale);
    dst[c] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

}  // namespace

cudaError_t launch_write_kv(const WriteArgs& a, cudaStream_t st) {
  if (a.T == 0) return cudaSuccess;
  const cudaError_t e =
      launch_kernel(a.mx_keys ? write_kv_kernel<true> : write_kv_kernel<false>, dim3((a.T + kWarps - 1) / kWarps), dim3(kWarps * 32), 0, st,
                    a.chained, static_cast<const uint16_t*>(a.k_raw), a.gamma, a.beta, a.eps,
                    static_cast<const uint16_t*>(a.latent), a.latent_scale, a.block_table, a.B,
                    a.max_pages, a.tok_req, a.tok_pos, a.T, a.key_cache, a.latent_cache,
                    a.num_pages, a.status);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace dsa
