// smla.cu -- sparse MLA over the selected latent rows (the Attend step) on the
// tcgen05 tensor cores, and the log-sum-exp combine of its split partials.
//
// For row r, head h and the valid selected tokens j:
//   x_j = softmax_scale * latent_scale * (q[r][h] . dec(L8_j))       (576 dims)
//   o   = sum_j softmax(x)_j * latent_scale * dec(L8_j)[0:512],  lse = ln sum_j e^{x_j}
// (vLLM Day-0 post on Kimi K3.1 Pro, "What Kimi K3.1 Pro changes": MLA runs
// exactly over only the selected tokens; TokenSpeed post, "Sparse attention
// in Kimi K3.1 Pro": all heads attend to the selected tokens; AMD Instinct
// post, overview "MLA": 512 KV + 64 RoPE dims, the 512 part is the value.)
//
// The selected slots are split over CTAs in tiles of 128; each split emits a
// normalised partial (o_s, lse_s) and the combine forms
//   lse = ln sum_s e^{lse_s},  o = sum_s e^{lse_s - lse} o_s
// -- the log-sum-exp merge the pages use to combine per-GPU partial outputs
// under decode context parallelism (vLLM post, "Decode context parallelism
// with a sparse indexer"; TokenSpeed post, "Sharding long contexts with
// decode context parallelism", step 4).
//
// Per 128-slot tile, one CTA (a query row, a split, up to 64 heads):
//  1. gather the 128 selected 576-byte FP8 latent rows (paged) into shared
//     memory with cp.async, in the K-major 128-byte-swizzle layout (the
//     576 bytes span 4.5 swizzle atoms; the half atom is padded);
//  2. S^T[token, (term, head)] = L8 . Q8^T on tcgen05 kind::f8f6f4, M = 128
//     tokens, N = 2 x heads, K = 576.  The bf16 query is split exactly into
//     two E4M3 terms per (row, head): q * 2^a = hi + lo / 32 (a power of two
//     per head puts its absmax in [128, 256); both terms carry 4 significant
//     bits, a bf16 value has 8);
//  3. softmax across the tile's tokens per head in the log2 domain, with a
//     running maximum that is only moved (and the accumulator rescaled) when
//     a tile's maximum exceeds it by more than 8, so P = 2^(y - m) <= 256
//     fits E4M3; P is written to shared memory as two E4M3 terms, P = P_hi +
//     P_lo (about 8 significant bits), and the running sum takes the fp32 P;
//  4. O^T[dim, head] += V^T . P_hi^T + V^T . P_lo^T, kind::f8f6f4, M = 4 x 128
//     dims, N = heads, K = 128 tokens; V^T is the same shared-memory latent
//     tile read as an MN-major operand, so V is never copied.
// Accumulators (S^T and O^T) live in tensor memory.
#include <math.h>

#include "dsa_common.cuh"
#include "sm100_ptx.cuh"

namespace dsa {
namespace {

using namespace ptx;

constexpr int kThreads = 256;
constexpr int kLatAtoms = 5;                          // 576 B = 4.5 x 128 B, padded
constexpr int kAtom = kMlaTile * 128;                 // 128 token rows x 128 B
constexpr int kLatChunks = kLatDim / 16;              // 36 chunks of 16 B per row
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleT = 8.f;                      // log2 headroom of P before a rescale
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kOCol = 256;                       // O^T columns start here; S^T at 0

template <int HG>
struct MlaSmem {
  static constexpr int lat = 0;
  static constexpr int q = kLatAtoms * kAtom;                        // [5][2HG][128]
  static constexpr int p = q + kLatAtoms * 2 * HG * 128;             // [2][HG][128] hi, lo
  static constexpr int tok = p + 2 * HG * 128;                       // [128] int64
  static constexpr int red = tok + kMlaTile * 8;                     // max, sum: [2][4][32] each
  static constexpr int hs = red + 2 * 8 * 32 * 4;                    // m, l, corr, qc [4][HG]
  static constexpr int flag = hs + 4 * HG * 4;
  static constexpr int bar = (flag + 16 + 7) / 8 * 8;                // s_done, o_done
  static constexpr int tmem = bar + 16;
  static constexpr int bytes = tmem + 16;
  static constexpr int alloc = bytes + 1024;
};

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}

__device__ __forceinline__ void named_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Butterfly reduce-scatter over a warp: on return v[0] holds the reduction
// over all 32 lanes of element (lane % NV).  NV is 8, 16 or 32.
template <int NV, bool kMax>
__device__ __forceinline__ float reduce_scatter(float (&v)[NV], int lane) {
#pragma unroll
  for (int off = 16; off >= NV; off >>= 1) {           // fold lanes that hold the same elements
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const float o = __shfl_xor_sync(0xffffffffu, v[i], off);
      v[i] = kMax ? fmaxf(v[i], o) : v[i] + o;
    }
  }
#pragma unroll
  for (int off = NV / 2; off >= 1; off >>= 1) {
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < off; ++i) {
      const float keep = upper ? v[i + off] : v[i];
      const float send = upper ? v[i] : v[i + off];
      const float o = __shfl_xor_sync(0xffffffffu, send, off);
      v[i] = kMax ? fmaxf(keep, o) : keep + o;
    }
  }
  return v[0];
}

__device__ __forceinline__ float fast_exp2(float x) {   // hardware 2^x, -inf -> 0
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint8_t f32_to_e4m3(float x) {
  return (uint8_t)__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
}

// ---------------------------------------------------------------------------
// Query split: one warp per (row, head).  q * 2^a = hi + lo / 32 with hi, lo
// E4M3, a = 7 - floor(log2 absmax); qc = softmax_scale * latent_scale *
// log2(e) * 2^-a turns (hi.L + lo.L / 32) into the log2-domain logit.
__global__ void __launch_bounds__(256)
mla_qprep_kernel(const __nv_bfloat16* __restrict__ q, int R, int H, float softmax_scale,
                 float latent_scale, uint8_t* __restrict__ q8, float* __restrict__ qc) {
  const int w = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (w >= R * H) return;
  const __nv_bfloat16* src = q + (size_t)w * kLatDim;
  float x[kLatDim / 32];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < kLatDim / 32; ++i) {
    x[i] = __bfloat162float(src[i * 32 + lane]);
    amax = fmaxf(amax, fabsf(x[i]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const int a = amax > 0.f ? 7 - ilogbf(amax) : 0;
  uint8_t* hi = q8 + (size_t)w * 2 * kLatDim;
  uint8_t* lo = hi + kLatDim;
#pragma unroll
  for (int i = 0; i < kLatDim / 32; ++i) {
    const float s = ldexpf(x[i], a);                 // exact: a power of two
    const uint8_t h8 = f32_to_e4m3(s);
    const float r = s - e4m3_to_float(h8);           // exact: both on a common grid
    hi[i * 32 + lane] = h8;
    lo[i * 32 + lane] = f32_to_e4m3(r * 32.f);
  }
  if (lane == 0) qc[w] = softmax_scale * latent_scale * kLog2e * ldexpf(1.f, -a);
}

// ---------------------------------------------------------------------------
template <int HG>  // heads per CTA: 16, 32 or 64
__global__ void __launch_bounds__(kThreads, 1)
smla_tc_kernel(const uint8_t* __restrict__ q8, const float* __restrict__ qc, int H,
               const uint8_t* __restrict__ latent_cache, int64_t num_pages, float latent_scale,
               const int32_t* __restrict__ block_table, int B, int max_pages,
               const int32_t* __restrict__ row_req, const int32_t* __restrict__ row_len,
               const int32_t* __restrict__ idx, int k, int tiles_per_split, int nsplit,
               float* __restrict__ part_o, float* __restrict__ part_lse, uint32_t* status) {
  using L = MlaSmem<HG>;
  constexpr int CW = HG < 32 ? HG : 32;               // heads per softmax chunk
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* lat = smem + L::lat;
  uint8_t* qs = smem + L::q;
  uint8_t* ps = smem + L::p;
  int64_t* tok_off = reinterpret_cast<int64_t*>(smem + L::tok);
  float* red_max = reinterpret_cast<float*>(smem + L::red);          // [half][quarter][32]
  float* red_sum = red_max + 8 * 32;                                  // [half][quarter][32]
  float* m_s = reinterpret_cast<float*>(smem + L::hs);               // running max (log2)
  float* l_s = m_s + HG;                                              // running sum
  float* corr_s = l_s + HG;                                           // this tile's rescale
  float* qc_s = corr_s + HG;
  int* flag_s = reinterpret_cast<int*>(smem + L::flag);
  uint64_t* s_done = reinterpret_cast<uint64_t*>(smem + L::bar);
  uint64_t* o_done = s_done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::tmem);

  const int split = blockIdx.x, r = blockIdx.y, hg0 = blockIdx.z * HG;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int req = row_req[r];
  const int len = row_len[r];
  const bool row_valid =
      req >= 0 && req < B && len >= 0 && (int64_t)len <= (int64_t)max_pages * kPage;
  if (!row_valid && split == 0 && blockIdx.z == 0 && tid == 0) raise_dev(status, DSA_DEV_BAD_ROW);
  const int slot0 = split * tiles_per_split * kMlaTile;
  const int slot1 = min(k, slot0 + tiles_per_split * kMlaTile);
  const int ntiles = (slot1 - slot0 + kMlaTile - 1) / kMlaTile;

  if (tid == 0) {
    mbar_init(s_done, 1);
    mbar_init(o_done, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  // query terms -> shared (K-major, 128B swizzle; row n = term * HG + head)
  for (int id = tid; id < 2 * HG * kLatChunks; id += kThreads) {
    const int n = id / kLatChunks, c = id % kLatChunks;
    const int term = n / HG, h = n % HG;
    const uint4 v = *reinterpret_cast<const uint4*>(
        q8 + (((size_t)r * H + hg0 + h) * 2 + term) * kLatDim + c * 16);
    *reinterpret_cast<uint4*>(qs + (c >> 3) * (2 * HG * 128) + n * 128 +
                              (((c & 7) ^ (n & 7)) << 4)) = v;
  }
  for (int h = tid; h < HG; h += kThreads) {
    m_s[h] = -INFINITY;
    l_s[h] = 0.f;
    qc_s[h] = qc[(size_t)r * H + hg0 + h];
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const uint32_t idesc_s = idesc_e4m3_f32(kMlaTile, 2 * HG, false, false);
  const uint32_t idesc_o = idesc_e4m3_f32(kMlaTile, HG, true, false);
  const bool epi_warp = warp >= 4;        // rescale and final epilogue: warps 4-7
  const int quarter = warp & 3;           // TMEM lane quarter of this warp
  const int half = warp >> 2;             // softmax: heads [half * HG / 2, (half + 1) * HG / 2)
  bool alive = true;

  for (int t = 0; t < ntiles && alive; ++t) {
    // the previous tile's P.V has finished reading the latent tile and P
    if (t > 0 && !mbar_wait(o_done, (uint32_t)(t - 1) & 1, status)) alive = false;
    if (__syncthreads_or(!alive)) break;
    // ---- token row offsets of this tile (-1: masked slot)
    if (tid < kMlaTile) {
      const int j = slot0 + t * kMlaTile + tid;
      int64_t off = -1;
      if (row_valid && j < slot1) {
        const int tok = idx[(size_t)r * k + j];
        if (tok >= len) {
          raise_dev(status, DSA_DEV_BAD_INDEX);
        } else if (tok >= 0) {
          const int page = block_table[(size_t)req * max_pages + tok / kPage];
          if (page < 0 || (int64_t)page >= num_pages)
            raise_dev(status, DSA_DEV_BAD_PAGE);
          else
            off = ((int64_t)page * kPage + (tok % kPage)) * kLatDim;
        }
      }
      tok_off[tid] = off;
    }
    __syncthreads();
    // ---- gather: 128 rows x 36 chunks; masked rows are zero (P = 0 must meet finite V)
    for (int id = tid; id < kMlaTile * kLatChunks; id += kThreads) {
      const int row = id / kLatChunks, c = id % kLatChunks;
      uint8_t* dst = lat + (c >> 3) * kAtom + row * 128 + (((c & 7) ^ (row & 7)) << 4);
      const int64_t off = tok_off[row];
      if (off >= 0)
        cp_async16(dst, latent_cache + off + c * 16);
      else
        *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
    }
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
    fence_proxy_async_smem();
    if (tid == 0) flag_s[0] = 0;
    __syncthreads();
    // ---- S^T = L8 . Q8^T
    if (tid == 0) {
      tc_fence_after();
      const uint32_t a0 = smem_u32(lat), b0 = smem_u32(qs);
#pragma unroll
      for (int j = 0; j < kLatDim / 32; ++j) {
        const uint64_t ad = desc_kmajor_sw128(a0 + (j >> 2) * kAtom + (j & 3) * 32);
        const uint64_t bd = desc_kmajor_sw128(b0 + (j >> 2) * (2 * HG * 128) + (j & 3) * 32);
        mma_e4m3_ss(tmem_base, ad, bd, idesc_s, j > 0 ? 1u : 0u);
      }
      mma_commit(s_done);
    }
    // ---- softmax, all 8 warps: thread = token 32 * quarter + lane, warp half
    // `half` takes half of the heads; warps of one half reduce through smem.
    {
      constexpr int CWH = HG / 2;
      if (!mbar_wait(s_done, (uint32_t)t & 1, status)) alive = false;
      tc_fence_after();
      const int tt = quarter * 32 + lane;
      const bool valid = tok_off[tt] >= 0;
      const int h0 = half * CWH;
      uint32_t dh[32], dl[32];
      const uint32_t ta = tmem_base + ((uint32_t)(quarter * 32) << 16);
      tmem_ld_32x32b_x32(ta + (uint32_t)h0, dh);
      tmem_ld_32x32b_x32(ta + (uint32_t)(HG + h0), dl);
      tmem_wait_ld();
      float y[CWH], v[CWH];
#pragma unroll
      for (int i = 0; i < CWH; ++i) {
        y[i] = valid ? (__uint_as_float(dh[i]) + __uint_as_float(dl[i]) * (1.f / 32.f)) *
                           qc_s[h0 + i]
                     : -INFINITY;
        v[i] = y[i];
      }
      const float wmax = reduce_scatter<CWH, true>(v, lane);
      if (lane < CWH) red_max[(half * 4 + quarter) * 32 + lane] = wmax;
      named_sync(1, kThreads);
      if (quarter == 0 && lane < CWH) {
        const int h = h0 + lane;
        const float* rm = red_max + half * 4 * 32 + lane;
        const float tmax = fmaxf(fmaxf(rm[0], rm[32]), fmaxf(rm[64], rm[96]));
        const float m_old = m_s[h];
        float c = 1.f;
        if (tmax > m_old + kRescaleT) {               // m_old = -inf on the first valid tile
          c = fast_exp2(m_old - tmax);
          m_s[h] = tmax;
          flag_s[0] = 1;
        }
        corr_s[h] = c;
      }
      named_sync(1, kThreads);
      float pf[CWH];
#pragma unroll
      for (int i = 0; i < CWH; ++i) {
        const int h = h0 + i;
        const float m = m_s[h];
        const float p = (valid && m > -INFINITY) ? fast_exp2(y[i] - m) : 0.f;
        const uint8_t p_hi = f32_to_e4m3(p);
        const uint8_t p_lo = f32_to_e4m3(p - e4m3_to_float(p_hi));
        pf[i] = p;
        // P^T is K-major: row = head, byte = token, 16-byte chunks swizzled by row
        const int off = h * 128 + ((((tt >> 4) ^ (h & 7))) << 4) + (tt & 15);
        ps[off] = p_hi;
        ps[HG * 128 + off] = p_lo;
      }
      const float wsum = reduce_scatter<CWH, false>(pf, lane);
      if (lane < CWH) red_sum[(half * 4 + quarter) * 32 + lane] = wsum;
      named_sync(1, kThreads);
      if (quarter == 0 && lane < CWH) {
        const int h = h0 + lane;
        const float* rs = red_sum + half * 4 * 32 + lane;
        l_s[h] = l_s[h] * corr_s[h] + rs[0] + rs[32] + rs[64] + rs[96];
      }
      // rescale the O^T accumulator when a running maximum moved (never on tile 0:
      // the first P.V overwrites the accumulator); warps 4-7 cover all heads
      if (t > 0 && flag_s[0] && epi_warp) {
#pragma unroll
        for (int a = 0; a < kVDim / kMlaTile; ++a) {
#pragma unroll
          for (int c0 = 0; c0 < HG; c0 += CW) {
            uint32_t d[32];
            const uint32_t tb = tmem_base + ((uint32_t)(quarter * 32) << 16) + kOCol +
                                (uint32_t)(a * HG + c0);
            tmem_ld_32x32b_x32(tb, d);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < CW; ++i) d[i] = __float_as_uint(__uint_as_float(d[i]) * corr_s[c0 + i]);
            tmem_st_32x32b_x32(tb, d);
          }
        }
        tmem_wait_st();
      }
      fence_proxy_async_smem();
      tc_fence_before();
    }
    if (__syncthreads_or(!alive)) break;
    // ---- O^T += V^T . P_hi^T + V^T . P_lo^T
    if (tid == 0) {
      tc_fence_after();
      const uint32_t a0 = smem_u32(lat), b0 = smem_u32(ps);
#pragma unroll
      for (int a = 0; a < kVDim / kMlaTile; ++a) {
#pragma unroll
        for (int kk = 0; kk < kMlaTile / 32; ++kk) {
          const uint64_t ad = desc_kmajor_sw128(a0 + a * kAtom + kk * 4096);   // 32 token rows
          const uint32_t d = tmem_base + kOCol + (uint32_t)(a * HG);
          mma_e4m3_ss(d, ad, desc_kmajor_sw128(b0 + kk * 32), idesc_o,
                      (t > 0 || kk > 0) ? 1u : 0u);
          mma_e4m3_ss(d, ad, desc_kmajor_sw128(b0 + HG * 128 + kk * 32), idesc_o, 1u);
        }
      }
      mma_commit(o_done);
    }
  }

  // ---- epilogue: O^T / l -> partial output, lse
  if (alive && ntiles > 0) {
    if (!mbar_wait(o_done, (uint32_t)(ntiles - 1) & 1, status)) alive = false;
  }
  if (epi_warp) {
    tc_fence_after();
    const size_t pbase = ((size_t)r * nsplit + split) * H + hg0;
#pragma unroll
    for (int a = 0; a < kVDim / kMlaTile; ++a) {
#pragma unroll
      for (int h0 = 0; h0 < HG; h0 += CW) {
        uint32_t d[32];
        if (alive && ntiles > 0) {
          tmem_ld_32x32b_x32(tmem_base + ((uint32_t)(quarter * 32) << 16) + kOCol +
                                 (uint32_t)(a * HG + h0),
                             d);
          tmem_wait_ld();
        }
#pragma unroll
        for (int i = 0; i < CW; ++i) {
          const float l = l_s[h0 + i];
          const float o = (alive && ntiles > 0 && l > 0.f) ? __uint_as_float(d[i]) * (latent_scale / l)
                                                            : 0.f;
          part_o[(pbase + h0 + i) * kVDim + a * kMlaTile + quarter * 32 + lane] = o;
        }
      }
    }
    if (quarter == 0) {
      for (int h = lane; h < HG; h += 32) {
        const float l = l_s[h], m = m_s[h];
        part_lse[pbase + h] =
            (alive && l > 0.f && m > -INFINITY) ? (m + log2f(l)) * 0.6931471805599453f : -INFINITY;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
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
cudaError_t launch_smla_group(const MlaArgs& a, const MlaLayout& L, cudaStream_t st) {
  using S = MlaSmem<HG>;
  cudaError_t e = cudaFuncSetAttribute(smla_tc_kernel<HG>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, S::alloc);
  if (e != cudaSuccess) return e;
  dim3 grid(L.nsplit, a.R, a.H / HG);
  smla_tc_kernel<HG><<<grid, kThreads, S::alloc, st>>>(
      a.scratch + L.q8, reinterpret_cast<const float*>(a.scratch + L.qc), a.H, a.latent_cache,
      a.num_pages, a.latent_scale, a.block_table, a.B, a.max_pages, a.row_req, a.row_len, a.idx, a.k,
      mla_tiles_per_split(a.R, a.k), L.nsplit, reinterpret_cast<float*>(a.scratch + L.part_o),
      reinterpret_cast<float*>(a.scratch + L.part_lse), a.status);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_sparse_mla(const MlaArgs& a, cudaStream_t st) {
  if (a.R == 0) return cudaSuccess;
  const MlaLayout L(a.R, a.H, a.k);
  const int warps = a.R * a.H;
  mla_qprep_kernel<<<(warps + 7) / 8, 256, 0, st>>>(
      static_cast<const __nv_bfloat16*>(a.q), a.R, a.H, a.softmax_scale, a.latent_scale,
      a.scratch + L.q8, reinterpret_cast<float*>(a.scratch + L.qc));
  cudaError_t e;
  if (a.H == 16) e = launch_smla_group<16>(a, L, st);
  else if (a.H == 32) e = launch_smla_group<32>(a, L, st);
  else e = launch_smla_group<64>(a, L, st);
  if (e != cudaSuccess) return e;
  mla_combine_kernel<<<a.R * a.H, 128, 0, st>>>(reinterpret_cast<const float*>(a.scratch + L.part_o),
                                                reinterpret_cast<const float*>(a.scratch + L.part_lse),
                                                a.H, L.nsplit, static_cast<__nv_bfloat16*>(a.out),
                                                a.lse);
  return cudaGetLastError();
}

}  // namespace dsa
