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
//  1. six warps gather the 128 selected 576-byte FP8 latent rows (paged) into
//     one of two shared-memory buffers with TMA tile::gather4 (four arbitrary
//     rows x 128 bytes per instruction, one instruction per lane, landing in
//     the K-major 128-byte-swizzle layout for dims 0..511; the RoPE dims
//     512..575 come as 64-byte boxes into a K-major 64-byte-swizzle block),
//     while the previous tile is computed.  Each lane waits only until its own
//     atom of the buffer is free again (the RoPE block after S, atom a after
//     M-block a of P.V), so most of a tile is in flight while P.V still runs.
//     Masked slots use an out-of-range row, which TMA fills with zeros;
//  2. S[(head, term), token] = Q8 . L8^T on tcgen05 kind::f8f6f4, M = 128,
//     N = 128 tokens, K = 576.  The bf16 query is split exactly into two E4M3
//     terms per (row, head): q * 2^a = hi + lo / 32 (a power of two per head
//     puts its absmax in [128, 256); both terms carry 4 significant bits, a
//     bf16 value has 8).  The query sits in tensor memory as the A operand
//     for dims 0..511 (the RoPE dims 512..575 come from shared memory), which
//     leaves shared memory for the second latent buffer;
//  3. softmax per head along the TMEM lane in the log2 domain: the two terms
//     of a head are adjacent lanes of one warp (combined by a shuffle), the
//     maximum over the tile is a per-thread loop plus one exchange between the
//     two warps that hold the tile's token halves.  The running maximum only
//     moves (and the accumulator is rescaled) when a tile's maximum exceeds it
//     by more than 8, so P = 2^(y - m) <= 256 fits E4M3; P goes to shared
//     memory as two E4M3 terms, P = P_hi + P_lo (about 8 significant bits),
//     and the running sum takes the fp32 P;
//  4. O^T[dim, head] += V^T . P_hi^T + V^T . P_lo^T, kind::f8f6f4, M = 4 x 128
//     dims, N = heads, K = 128 tokens; V^T is the same shared-memory latent
//     tile read as an MN-major operand, so V is never copied.
// Accumulators (S and O^T) live in tensor memory; an MMA warp pipelines S of
// tile i + 1 against the softmax and P.V of tile i through mbarriers.
#include <limits.h>
#include <math.h>
#include <string.h>

#include "dsa_common.cuh"
#include "sm100_ptx.cuh"

namespace dsa {
namespace {

using namespace ptx;

constexpr int kLatAtoms = 5;                          // 576 B = 4 x 128 B + 64 B
constexpr int kAtom = kMlaTile * 128;                 // 128 token rows x 128 B (dims 0..511)
constexpr int kRopeAtom = kMlaTile * 64;              // 128 token rows x 64 B (dims 512..575)
constexpr float kLog2e = 1.4426950408889634f;
// P = 2^(x - m + kPOff) with m the running maximum, raised only when a tile's
// maximum passes m + kRescaleT, so P <= 2^(kPOff + kRescaleT) = 256 < 448.
// The offset keeps the tokens near the maximum at P >= 16, where the two E4M3
// terms of P hold 8 significant bits, instead of near 1, where the low term
// reaches E4M3's subnormal step.
constexpr float kRescaleT = 4.f;                      // log2 headroom of P before a rescale
constexpr float kPOff = 4.f;
constexpr uint32_t kTmemCols = 512;

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
  // reads only the caller's query: runs alongside the kernel before it, and
  // completes after it (pdl_wait at the end)
  pdl_trigger();
  const int w = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (w >= R * H) {
    pdl_wait();
    return;
  }
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
  pdl_wait();
}

// ---------------------------------------------------------------------------
// Warp roles (512 threads): warp 0 issues the score MMAs and owns tensor
// memory, warp 1 issues the P.V MMAs (a thread is held at every tcgen05.mma
// until the tensor core takes it, so two issuers keep S of one tile and P.V of
// the previous one both fed); warps 2-7 gather latent rows with TMA
// (double-buffered; 160 gather4 loads per tile spread one per lane, since one
// warp's loads issue one lane at a time); warps 8-15 run the softmax and the
// epilogues: warp w reads TMEM lane quarter (w & 3) and token half (w - 8) / 4
// of S.
constexpr int kThreads = 512;
constexpr int kGatherWarp0 = 2;
constexpr int kGatherLanes = 27;                       // 6 x 27 >= 160 loads per tile
constexpr int kSmWarp0 = 8;                            // first softmax warp
constexpr int kSmThreads = 256;
constexpr int kTileBytes = 4 * kAtom + kRopeAtom;     // one latent buffer
static_assert(kTileBytes % 1024 == 0, "swizzle atoms stay 1024-byte aligned");
constexpr uint32_t kQCol = 0;                          // A operand: Q (dims 0..511), 128 cols
constexpr uint32_t kSCol = 128;                        // S: [(head, term)] x [128 tokens]
constexpr uint32_t kOCol = 256;                        // O^T: 4 blocks x HG cols

// NVFP4 latent rows (352 bytes: 256 bytes of E2M1 codes, dim 2j in the low
// nibble of byte j; 32 unsigned-E4M3 scales, one per 16 dims; 64 E4M3 RoPE
// bytes).  A value c * s (c an E2M1 element, s its block scale) has at most
// six significant bits, so v = c * s / 4 = hi + lo with hi = E4M3(v) and
// lo = v - hi, both exact in E4M3 when v >= 2^-4, i.e. for every s >= 0.5
// (above 448, hi saturates at 448 and lo = v - 448 <= 224 is still exact).
// The 1/4 is folded into the latent scale, so the RoPE bytes r are fed as
// E4M3(r / 4), exact for |r| >= 2^-4.  Below those bounds the terms round to
// E4M3's subnormal step: at most 2^-8 of the latent scale per element.
constexpr int kNvRowBytes = 352;
constexpr int kNvCodes = 256, kNvScales = 32;
constexpr int kNvGatherThreads = (kSmWarp0 - kGatherWarp0) * 32;     // 192

template <int HG, bool kNv>
struct MlaSmem {
  // FP8 rows: two buffers of 4 atoms (dims 0..511) + a RoPE atom, filled by
  // TMA.  NVFP4 rows: one buffer of 4 hi atoms, 4 lo atoms and a RoPE atom,
  // written by the gather warps, then the byte offsets of two tiles' rows.
  static constexpr int lat = 0;
  static constexpr int lat_bytes = kNv ? 8 * kAtom + kRopeAtom : 2 * kTileBytes;
  static constexpr int rowoff = lat + lat_bytes;                     // NVFP4: [2][128] int64
  static constexpr int qrope = rowoff + (kNv ? 2 * kMlaTile * 8 : 0);   // [128 rows][128 B]
  static constexpr int p = qrope + kMlaTile * 128;                   // [2 terms][HG][128]
  static constexpr int corr = p + 2 * HG * 128;                      // [64] f32
  static constexpr int red = corr + 64 * 4;                          // [2 halves][64] f32
  static constexpr int lsum = red + 2 * 64 * 4;                      // [2 halves][64] f32
  static constexpr int flag = lsum + 2 * 64 * 4;                     // [2] int
  static constexpr int bar = (flag + 8 + 7) / 8 * 8;                 // 23 mbarriers
  static constexpr int tmem = bar + 23 * 8;
  static constexpr int bytes = tmem + 16;
  static constexpr int alloc = bytes + 1024;
  static_assert(qrope % 1024 == 0, "the swizzled query operand stays 1024-byte aligned");
};

// TMA gather of four rows (y0..y3) x one box of the 2-D tensor map starting at
// column x; completes on the mbarrier with the box bytes.
__device__ __forceinline__ void tma_gather4(void* dst, const CUtensorMap* tmap, int x, int y0,
                                            int y1, int y2, int y3, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y0), "r"(y1), "r"(y2), "r"(y3),
      "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ bool wwait(uint64_t* bar, uint32_t parity, uint32_t* status) {
  bool ok = true;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, status);
  return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

// Pack four floats into four E4M3 bytes (RNE, saturating).
__device__ __forceinline__ uint32_t pack_e4m3x4(float a, float b, float c, float d) {
  uint16_t lo, hi;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %2, %1;" : "=h"(lo) : "f"(a), "f"(b));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %2, %1;" : "=h"(hi) : "f"(c), "f"(d));
  return (uint32_t)lo | ((uint32_t)hi << 16);
}

// Eight E2M1 values (four code bytes, low nibble first) -> four f16x2 pairs, exact.
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t x, uint32_t (&h)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(x));
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ uint32_t hsub2_u32(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ uint32_t f16x2_to_e4m3x2(uint32_t x) {   // RN, saturating; 16 bits
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(r) : "r"(x));
  return r;
}

__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t x) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"((uint16_t)x));
  return r;
}

// 32 NVFP4 dims (16 code bytes in c, their two block-scale bytes in sc, low
// byte first) -> the E4M3 terms hi and lo of c * s / 4, 16 bytes each per 16
// dims: hi[0], lo[0] for the first 16 dims, hi[1], lo[1] for the next.
__device__ __forceinline__ void nvfp4_split32(const uint4& c, uint32_t sc, uint4 (&hi)[2],
                                              uint4 (&lo)[2]) {
  // the two scales as f16 (unsigned E4M3: the top bit is ignored), times 1/4
  const uint32_t s2 = hmul2_u32(e4m3x2_to_f16x2(sc & 0x7F7Fu), 0x34003400u);   // {s0, s1} / 4
  const uint32_t sa = __byte_perm(s2, 0, 0x1010), sb = __byte_perm(s2, 0, 0x3232);
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
  uint32_t ho[8], lw[8];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t h[4];
    e2m1x8_to_f16x2(w[q], h);
    const uint32_t sq = q < 2 ? sa : sb;
#pragma unroll
    for (int e = 0; e < 4; e += 2) {
      const uint32_t v0 = hmul2_u32(h[e], sq), v1 = hmul2_u32(h[e + 1], sq);
      const uint32_t h0 = f16x2_to_e4m3x2(v0), h1 = f16x2_to_e4m3x2(v1);
      const uint32_t l0 = f16x2_to_e4m3x2(hsub2_u32(v0, e4m3x2_to_f16x2(h0)));
      const uint32_t l1 = f16x2_to_e4m3x2(hsub2_u32(v1, e4m3x2_to_f16x2(h1)));
      ho[2 * q + e / 2] = h0 | (h1 << 16);
      lw[2 * q + e / 2] = l0 | (l1 << 16);
    }
  }
  hi[0] = make_uint4(ho[0], ho[1], ho[2], ho[3]);
  hi[1] = make_uint4(ho[4], ho[5], ho[6], ho[7]);
  lo[0] = make_uint4(lw[0], lw[1], lw[2], lw[3]);
  lo[1] = make_uint4(lw[4], lw[5], lw[6], lw[7]);
}

// Sixteen E4M3 RoPE bytes -> E4M3(r / 4), the scale of the NVFP4 operands.
// Exact for |r| >= 2^-4; below, r / 4 is rounded to E4M3's subnormal step.
__device__ __forceinline__ uint4 e4m3x16_quarter(const uint4& v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t o[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint32_t a = hmul2_u32(e4m3x2_to_f16x2(w[q] & 0xFFFFu), 0x34003400u);
    const uint32_t b = hmul2_u32(e4m3x2_to_f16x2(w[q] >> 16), 0x34003400u);
    o[q] = f16x2_to_e4m3x2(a) | (f16x2_to_e4m3x2(b) << 16);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// Walks a CTA's tiles in order: unit u (row u / groups, head group u % groups)
// and tile lt within the unit; `first` / `last` mark the ends of a segment (a
// run of the CTA's tiles in one unit).
struct TileIt {
  int u, lt, i;
  __device__ __forceinline__ void next(int NT) {
    ++i;
    if (++lt == NT) { lt = 0; ++u; }
  }
  __device__ __forceinline__ int row(int groups) const { return groups == 1 ? u : u >> 1; }
  __device__ __forceinline__ int hg0(int groups, int HG) const {
    return groups == 1 ? 0 : (u & 1) * HG;
  }
  __device__ __forceinline__ bool first() const { return i == 0 || lt == 0; }
  __device__ __forceinline__ bool last(int n, int NT) const { return i == n - 1 || lt == NT - 1; }
};

template <int HG, bool kNv>  // heads per CTA: 16, 32 or 64; NVFP4 latent rows
__global__ void __launch_bounds__(kThreads, 1)
smla_kernel(const __grid_constant__ CUtensorMap lat_map, const __grid_constant__ CUtensorMap rope_map,
            const uint8_t* __restrict__ nv_cache,
            const uint8_t* q8, const float* qc, int H, int64_t num_pages, float latent_scale,
            const int32_t* __restrict__ block_table, int B, int max_pages,
            const int32_t* __restrict__ row_req, const int32_t* __restrict__ row_len,
            const int32_t* idx, int k, int R, float* __restrict__ part_o,
            float* __restrict__ part_lse, __nv_bfloat16* __restrict__ out,
            float* __restrict__ lse_out, uint32_t* status) {
  using L = MlaSmem<HG, kNv>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* lat = smem + L::lat;
  uint8_t* qrope = smem + L::qrope;
  uint8_t* ps = smem + L::p;
  float* corr_s = reinterpret_cast<float*>(smem + L::corr);
  float* red_s = reinterpret_cast<float*>(smem + L::red);
  float* lsum_s = reinterpret_cast<float*>(smem + L::lsum);
  int* flag_s = reinterpret_cast<int*>(smem + L::flag);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::bar);
  uint64_t* lat_full = bars;          // [2] gathered tile landed
  uint64_t* lat_empty = bars + 2;     // [2][5] atom a of the buffer is free again: the RoPE
                                      // atom 4 after S, atom a < 4 after M-block a of P.V
  uint64_t* s_full = bars + 12;       // S of a tile is in TMEM
  uint64_t* s_empty = bars + 13;      // S read (and Q in place) for the next score MMA
  uint64_t* p_full = bars + 14;       // P in shared memory, O rescaled
  uint64_t* p_empty = bars + 15;      // P.V finished (O complete up to this tile)
  uint64_t* mma_done = bars + 16;     // [2] every MMA of an issuer finished
  uint64_t* nv_full = bars + 18;      // NVFP4 [5]: hi/lo atom a (a < 4) or the RoPE atom written
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::tmem);

  const int groups = H / HG;
  const MlaWork w(R, H, k);
  const int c = blockIdx.x;
  const int64_t t0 = w.begin(c);
  const int n = (int)(w.begin(c + 1) - t0);
  const int NT = (int)w.NT;
  const int u_first = (int)(t0 / w.NT);
  const TileIt it0{u_first, (int)(t0 - (int64_t)u_first * w.NT), 0};
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    if constexpr (!kNv) {
      prefetch_tensor_map(&lat_map);
      prefetch_tensor_map(&rope_map);
    }
    // NVFP4: the gather warps each arrive once the tile is written
    for (int b = 0; b < 2; ++b) mbar_init(&lat_full[b], 1);
    for (int a = 0; a < kLatAtoms; ++a) mbar_init(&nv_full[a], kSmWarp0 - kGatherWarp0);
    for (int x = 0; x < 2 * kLatAtoms; ++x) mbar_init(&lat_empty[x], 1);
    mbar_init(s_full, 1);
    mbar_init(s_empty, 8);
    mbar_init(p_full, 8);
    mbar_init(p_empty, 1);
    mbar_init(&mma_done[0], 1);
    mbar_init(&mma_done[1], 1);
    fence_mbar_init();
    flag_s[0] = 0;
    flag_s[1] = 0;
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_trigger();                                    // after the tensor-memory allocation
  pdl_wait();                                       // query terms and selected indices

  const uint32_t idesc_s = idesc_e4m3_f32(kMlaTile, kMlaTile, false, false);
  const uint32_t idesc_o = idesc_e4m3_f32(kMlaTile, HG, true, false);

  if (warp < kGatherWarp0) {
    // ================= MMA issuers: warp 0 issues S(i) once tile i has landed
    // and S(i - 1) has been read; warp 1 issues O(i) once P(i) is in place
    // returns false when a wait ran out (NVFP4 waits for each atom in turn)
    auto issue_s = [&](int i) -> bool {
      const uint32_t lb = smem_u32(lat + (kNv ? 0 : (i & 1) * kTileBytes));
      if constexpr (!kNv) {
#pragma unroll
        for (int j = 0; j < kIdxDim * 4 / 32; ++j)    // dims 0..511 from TMEM
          mma_e4m3_ts(tmem_base + kSCol, tmem_base + kQCol + (uint32_t)(j * 8),
                      desc_kmajor_sw128(lb + (j >> 2) * kAtom + (j & 3) * 32), idesc_s,
                      j > 0 ? 1u : 0u);
      } else {
        // hi and lo terms of atom a as soon as the gather warps have written them
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          if (!mbar_wait(&nv_full[a], (uint32_t)i & 1, status)) return false;
          tc_fence_after();
#pragma unroll
          for (int t = 0; t < 2; ++t)
#pragma unroll
            for (int jj = 0; jj < 4; ++jj)
              mma_e4m3_ts(tmem_base + kSCol, tmem_base + kQCol + (uint32_t)((4 * a + jj) * 8),
                          desc_kmajor_sw128(lb + (4 * t + a) * kAtom + jj * 32), idesc_s,
                          (a | t | jj) ? 1u : 0u);
        }
        if (!mbar_wait(&nv_full[4], (uint32_t)i & 1, status)) return false;
        tc_fence_after();
      }
      const uint32_t rope_atom = lb + (kNv ? 8 : 4) * kAtom;
#pragma unroll
      for (int j = 0; j < 2; ++j)                     // dims 512..575 from shared
        mma_e4m3_ss(tmem_base + kSCol, desc_kmajor_sw128(smem_u32(qrope) + j * 32),
                    desc_kmajor_sw64(rope_atom + j * 32), idesc_s, 1u);
      mma_commit(s_full);
      mma_commit(&lat_empty[(kNv ? 0 : (i & 1)) * kLatAtoms + 4]);   // the RoPE atom is read by S only
      return true;
    };
    auto issue_o = [&](int i, bool first) {
      const uint32_t lb = smem_u32(lat + (kNv ? 0 : (i & 1) * kTileBytes));
      const uint32_t pb = smem_u32(ps);
#pragma unroll
      for (int a = 0; a < kVDim / kMlaTile; ++a) {
#pragma unroll
        for (int kk = 0; kk < kMlaTile / 32; ++kk) {
          const uint64_t ad = desc_kmajor_sw128(lb + a * kAtom + kk * 4096);   // 32 token rows
          const uint32_t d = tmem_base + kOCol + (uint32_t)(a * HG);
          mma_e4m3_ss(d, ad, desc_kmajor_sw128(pb + kk * 32), idesc_o,
                      (!first || kk > 0) ? 1u : 0u);
          mma_e4m3_ss(d, ad, desc_kmajor_sw128(pb + HG * 128 + kk * 32), idesc_o, 1u);
          if constexpr (kNv) {                        // the lo term of V
            const uint64_t al = desc_kmajor_sw128(lb + (4 + a) * kAtom + kk * 4096);
            mma_e4m3_ss(d, al, desc_kmajor_sw128(pb + kk * 32), idesc_o, 1u);
            mma_e4m3_ss(d, al, desc_kmajor_sw128(pb + HG * 128 + kk * 32), idesc_o, 1u);
          }
        }
        // M-block a was the last reader of atom a (NVFP4: hi and lo atoms a)
        mma_commit(&lat_empty[(kNv ? 0 : (i & 1)) * kLatAtoms + a]);
      }
      mma_commit(p_empty);
    };
    if (lane == 0 && n > 0) {
      if (warp == 0) {
        for (int si = 0; si < n; ++si) {
          if (!kNv && !mbar_wait(&lat_full[si & 1], (uint32_t)(si >> 1) & 1, status)) break;
          if (!mbar_wait(s_empty, (uint32_t)si & 1, status)) break;
          tc_fence_after();
          if (!issue_s(si)) break;
        }
      } else {
        TileIt ot = it0;                              // tile of the next O
        for (int oi = 0; oi < n; ++oi) {
          if (!mbar_wait(p_full, (uint32_t)oi & 1, status)) break;
          tc_fence_after();
          issue_o(oi, ot.first());
          ot.next(NT);
        }
      }
      mma_commit(&mma_done[warp]);                    // tensor memory is freed only after this
      mbar_wait(&mma_done[warp], 0, status);
    }
    __syncwarp();
  } else if (warp < kSmWarp0 && kNv) {
    // ================= NVFP4 gather: the six gather warps look up the tile's
    // rows, load their bytes into registers while the buffer is still in use,
    // then write the RoPE atom once S of the previous tile has read it and the
    // hi/lo terms of atom a once M-block a of the previous P.V has finished.
    // Piece (row, p) of an atom is 32 dims (16 code bytes + 2 scale bytes) or,
    // for the RoPE atom, 16 bytes; thread gtid takes pieces gtid + 192 m.
    const int gtid = tid - kGatherWarp0 * 32;
    int64_t* rowoff = reinterpret_cast<int64_t*>(smem + L::rowoff);
    constexpr int kPieces = kMlaTile * 4;                  // per atom
    constexpr int kPer = (kPieces + kNvGatherThreads - 1) / kNvGatherThreads;   // 3
    bool alive = true;
    TileIt gt = it0;
    for (int i = 0; i < n; ++i) {
      int64_t* ro = rowoff + (i & 1) * kMlaTile;
      if (gtid < kMlaTile) {
        const int r = gt.row(groups);
        const int req = row_req[r];
        const int len = row_len[r];
        const bool row_valid =
            req >= 0 && req < B && len >= 0 && (int64_t)len <= (int64_t)max_pages * kPage;
        if (!row_valid && gt.lt == 0 && gt.hg0(groups, HG) == 0 && gtid == 0)
          raise_dev(status, DSA_DEV_BAD_ROW);
        const int j = gt.lt * kMlaTile + gtid;
        int64_t off = -1;                             // masked slot: zero operands
        if (row_valid && j < k) {
          const int tok = ld_dep(idx + (size_t)r * k + j);
          if (tok >= len) {
            raise_dev(status, DSA_DEV_BAD_INDEX);
          } else if (tok >= 0) {
            const int page = block_table[(size_t)req * max_pages + tok / kPage];
            if (page < 0 || (int64_t)page >= num_pages)
              raise_dev(status, DSA_DEV_BAD_PAGE);
            else
              off = ((int64_t)page * kPage + tok % kPage) * kNvRowBytes;
          }
        }
        ro[gtid] = off;
      }
      gt.next(NT);
      // the other half of rowoff was last read before this barrier's previous phase
      named_sync(2, kNvGatherThreads);
      uint4 cv[4][kPer], rv[kPer];
      uint32_t sv[4][kPer];
#pragma unroll
      for (int m = 0; m < kPer; ++m) {
        const int e = gtid + kNvGatherThreads * m;
        const int64_t off = e < kPieces ? ro[e >> 2] : -1;
        const uint8_t* src = nv_cache + (off >= 0 ? off : 0);
        const int p = e & 3;
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          cv[a][m] = off >= 0 ? __ldg(reinterpret_cast<const uint4*>(src + (4 * a + p) * 16))
                              : make_uint4(0, 0, 0, 0);
          sv[a][m] = off >= 0 ? __ldg(reinterpret_cast<const uint16_t*>(src + kNvCodes +
                                                                        (4 * a + p) * 2))
                              : 0u;
        }
        rv[m] = off >= 0 ? __ldg(reinterpret_cast<const uint4*>(src + kNvCodes + kNvScales + p * 16))
                         : make_uint4(0, 0, 0, 0);
      }
      const uint32_t ep = ((uint32_t)i & 1) ^ 1;      // parity of "free again" for tile i
      if (alive && !wwait(&lat_empty[4], ep, status)) alive = false;
      if (alive) {
        uint8_t* ra = lat + 8 * kAtom;                // RoPE atom, 64-byte rows, 64B swizzle
#pragma unroll
        for (int m = 0; m < kPer; ++m) {
          const int e = gtid + kNvGatherThreads * m;
          if (e < kPieces) {
            const int row = e >> 2, p = e & 3;
            *reinterpret_cast<uint4*>(ra + row * 64 + ((p ^ ((row >> 1) & 3)) << 4)) =
                e4m3x16_quarter(rv[m]);
          }
        }
        fence_proxy_async_smem();                     // generic-proxy writes -> tensor core
        __syncwarp();
        if (lane == 0) mbar_arrive(&nv_full[4]);
      }
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        if (alive && !wwait(&lat_empty[a], ep, status)) alive = false;
        if (!alive) continue;
        uint8_t* ha = lat + a * kAtom;                // 128-byte rows, 128B swizzle
        uint8_t* la = lat + (4 + a) * kAtom;
#pragma unroll
        for (int m = 0; m < kPer; ++m) {
          const int e = gtid + kNvGatherThreads * m;
          if (e < kPieces) {
            const int row = e >> 2, p = e & 3;
            uint4 hi[2], lo[2];
            nvfp4_split32(cv[a][m], sv[a][m], hi, lo);
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const int o = row * 128 + (((2 * p + u) ^ (row & 7)) << 4);
              *reinterpret_cast<uint4*>(ha + o) = hi[u];
              *reinterpret_cast<uint4*>(la + o) = lo[u];
            }
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&nv_full[a]);
      }
    }
  } else if (warp < kSmWarp0) {
    // ================= TMA gather: lane op = (group g of 4 tile rows, box a of 5)
    const int op = (warp - kGatherWarp0) * kGatherLanes + lane;
    const bool op_ok = lane < kGatherLanes && op < 32 * kLatAtoms;
    const int g = op & 31, a = op >> 5;
    int y[4] = {-1, -1, -1, -1};
    TileIt gt = it0;                                  // tile of the next lookup
    auto lookup = [&]() {
      const int r = gt.row(groups);
      const int req = row_req[r];
      const int len = row_len[r];
      const bool row_valid =
          req >= 0 && req < B && len >= 0 && (int64_t)len <= (int64_t)max_pages * kPage;
      if (!row_valid && gt.lt == 0 && gt.hg0(groups, HG) == 0 && op == 0)
        raise_dev(status, DSA_DEV_BAD_ROW);
      const int slot0 = gt.lt * kMlaTile;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j = slot0 + 4 * g + u;
        int yy = -1;                                  // out of range: zero-filled by TMA
        if (row_valid && j < k) {
          const int tok = ld_dep(idx + (size_t)r * k + j);
          if (tok >= len) {
            raise_dev(status, DSA_DEV_BAD_INDEX);
          } else if (tok >= 0) {
            const int page = block_table[(size_t)req * max_pages + tok / kPage];
            if (page < 0 || (int64_t)page >= num_pages)
              raise_dev(status, DSA_DEV_BAD_PAGE);
            else
              yy = page * kPage + (tok % kPage);
          }
        }
        y[u] = yy;
      }
      gt.next(NT);
    };
    if (op_ok && n > 0) lookup();
    // Each lane waits for its own atom of the buffer only, so most of a tile is
    // already in flight while the P.V that frees the buffer's last atoms runs.
    for (int i = 0; i < n && op_ok; ++i) {
      const int b = i & 1;
      if (!mbar_wait(&lat_empty[b * kLatAtoms + a], ((uint32_t)(i >> 1) & 1) ^ 1, status)) break;
      // complete_tx of other lanes may land before this arrive: the phase
      // cannot complete until the single arrival has come
      if (warp == kGatherWarp0 && lane == 0) mbar_arrive_expect_tx(&lat_full[b], kTileBytes);
      {
        if (a < 4)
          tma_gather4(lat + b * kTileBytes + a * kAtom + g * 512, &lat_map, a * 128, y[0], y[1],
                      y[2], y[3], &lat_full[b]);
        else                                          // RoPE dims: 4 rows x 64 B
          tma_gather4(lat + b * kTileBytes + 4 * kAtom + g * 256, &rope_map, 512, y[0], y[1],
                      y[2], y[3], &lat_full[b]);
        if (i + 1 < n) lookup();
      }
    }
    // no copy may still be landing in shared memory when the CTA exits
    if (warp == kGatherWarp0 && n > 0) {
      const int last = n - 1;
      wwait(&lat_full[last & 1], (uint32_t)(last >> 1) & 1, status);
      if (n > 1) wwait(&lat_full[(last - 1) & 1], (uint32_t)((last - 1) >> 1) & 1, status);
    }
  } else {
    // ================= softmax + epilogues
    const int sw = warp - kSmWarp0;
    const int quarter = warp & 3;
    const int th = sw >> 2;                            // token half of the tile
    const int hl = 16 * quarter + (lane & 15);          // head within the group
    const bool head_ok = hl < HG;
    const int stid = tid - kSmWarp0 * 32;
    bool alive = true;

    // Q of unit u: rows (head, term) -> TMEM columns [0, 128) (dims 0..511)
    // and the RoPE dims 512..575 -> shared (A operand of the last two K steps)
    auto load_q = [&](int r, int hg0) {
      // token half th loads dims 256 th .. 256 th + 255 and RoPE chunks 2 th, 2 th + 1
      // of its lane quarter's rows, four rounds of four 16-byte loads
      const int term = lane >> 4;
      const uint4* src = reinterpret_cast<const uint4*>(
          q8 + (((size_t)r * H + hg0 + (head_ok ? hl : 0)) * 2 + term) * kLatDim);
      const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll 1
      for (int c8 = 4 * th; c8 < 4 * th + 4; ++c8) {      // 16 columns per round
        uint32_t v[16];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint4 x = head_ok ? ld_dep(src + c8 * 4 + u) : z;
          v[4 * u + 0] = x.x; v[4 * u + 1] = x.y; v[4 * u + 2] = x.z; v[4 * u + 3] = x.w;
        }
        tmem_st_32x32b_x16(tmem_base + ((uint32_t)(quarter * 32) << 16) + kQCol + c8 * 16, v);
      }
      const int m = quarter * 32 + lane;
#pragma unroll
      for (int c4 = 2 * th; c4 < 2 * th + 2; ++c4) {
        const uint4 x = head_ok ? ld_dep(src + 32 + c4) : z;
        *reinterpret_cast<uint4*>(qrope + m * 128 + ((c4 ^ (m & 7)) << 4)) = x;
      }
      tmem_wait_st();
      fence_proxy_async_smem();
    };
    auto load_qc = [&](int r, int hg0) {
      return head_ok ? ld_dep(qc + (size_t)r * H + hg0 + hl) : 0.f;
    };

    float m_run = -INFINITY, l_run = 0.f, qcf = 0.f;
    int seg_lt0 = 0;                                  // first tile (within its unit) of the segment
    // validity of this warp's 64 tokens (tokens th*64 + lane and th*64 + 32 + lane).
    // The ids are loaded a tile ahead from clamped addresses, so that nothing
    // consumes a load before the end of the tile; len_ok is -1 for an invalid row.
    int len_ok = -1;                                  // row length of the prepared tile's unit
    auto unit_len = [&](const TileIt& t) {
      const int r = t.row(groups);
      const int req = row_req[r];
      const int len = row_len[r];
      const bool row_valid =
          req >= 0 && req < B && len >= 0 && (int64_t)len <= (int64_t)max_pages * kPage;
      return row_valid ? len : -1;
    };
    auto load_ids = [&](const TileIt& t, int& ia, int& ib) {
      const int* rowp = idx + (size_t)t.row(groups) * k;
      const int j = t.lt * kMlaTile + th * 64 + lane;
      ia = ld_dep(rowp + min(j, k - 1));
      ib = ld_dep(rowp + min(j + 32, k - 1));
    };
    auto valid_bits = [&](const TileIt& t, int ia, int ib, uint32_t& lo_bits, uint32_t& hi_bits) {
      const int j = t.lt * kMlaTile + th * 64 + lane;
      lo_bits = __ballot_sync(0xffffffffu, j < k && ia >= 0 && ia < len_ok);
      hi_bits = __ballot_sync(0xffffffffu, j + 32 < k && ib >= 0 && ib < len_ok);
    };
    uint32_t vlo = 0, vhi = 0;
    int ida = -1, idb = -1;
    TileIt ta = it0;                                  // current tile
    if (n > 0) {
      load_q(ta.row(groups), ta.hg0(groups, HG));
      qcf = load_qc(ta.row(groups), ta.hg0(groups, HG));
      seg_lt0 = ta.lt;
      len_ok = unit_len(ta);
      load_ids(ta, ida, idb);
      valid_bits(ta, ida, idb, vlo, vhi);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_empty);            // Q in place for S(0)
    }
    for (int i = 0; i < n; ++i, ta.next(NT)) {
      TileIt tn = ta;                                 // the tile after this one
      tn.next(NT);
      const bool seg_last = ta.last(n, NT);
      // ---- S rows -> registers, then S may be overwritten by the next tile's MMA
      if (!wwait(s_full, (uint32_t)i & 1, status)) alive = false;
      tc_fence_after();
      // rows 32q + j hold the hi term of head 16q + j, rows 32q + 16 + j the lo
      // term: thread t gets both for head 16q + (t & 15) and 32 tokens
      // (t < 16: tokens 0..31 of the warp's half, t >= 16: tokens 32..63)
      const uint32_t tq = tmem_base + ((uint32_t)(quarter * 32) << 16);
      const bool hi_lane = lane < 16;
      const uint32_t vb = hi_lane ? vlo : vhi;
      float y[32];
      float tmax = -INFINITY;
#pragma unroll
      for (int h16 = 0; h16 < 2; ++h16) {             // 16 tokens at a time
        uint32_t s_hi[16], s_lo[16];
        if (alive) {
          tmem_ld_16x32bx2_x16<32>(tq + kSCol + th * 64 + h16 * 16, s_hi);
          tmem_ld_16x32bx2_x16<32>(tq + (16u << 16) + kSCol + th * 64 + h16 * 16, s_lo);
          tmem_wait_ld();
        }
        // ---- the two query terms -> log2-domain logits
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float x = __uint_as_float(s_hi[j]) + __uint_as_float(s_lo[j]) * (1.f / 32.f);
          const int jj = h16 * 16 + j;
          y[jj] = ((vb >> jj) & 1u) ? x * qcf : -INFINITY;
          tmax = fmaxf(tmax, y[jj]);
        }
      }
      if (seg_last && i + 1 < n && alive)              // next tile starts a new unit: its Q
        load_q(tn.row(groups), tn.hg0(groups, HG));
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_empty);
      if (i + 1 < n) load_ids(tn, ida, idb);
      tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 16));
      if (hi_lane && head_ok) red_s[th * 64 + hl] = tmax;
      named_sync(1, kSmThreads);
      // every softmax warp is past tile i - 1 here: its flag slot can be reused
      if (stid == 0) flag_s[(i + 1) & 1] = 0;
      if (head_ok) tmax = fmaxf(tmax, red_s[(th ^ 1) * 64 + hl]);
      float corr = 1.f;
      if (tmax > m_run + kRescaleT) {                 // m_run = -inf on a segment's first tile
        corr = fast_exp2(m_run - tmax);
        m_run = tmax;
      }
      if (th == 0 && hi_lane && head_ok) {
        corr_s[hl] = corr;
        if (corr != 1.f) flag_s[i & 1] = 1;
      }
      // ---- P (two E4M3 terms) -> shared, once the previous P.V has finished with it
      if (!wwait(p_empty, ((uint32_t)i & 1) ^ 1, status)) alive = false;
      named_sync(1, kSmThreads);                      // corr_s / flag visible
      float psum = 0.f;
      uint32_t whi[8], wlo[8];
#pragma unroll
      for (int j4 = 0; j4 < 8; ++j4) {
        float p[4], pl[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float v = y[4 * j4 + u];
          p[u] = (m_run > -INFINITY && v > -INFINITY) ? fast_exp2(v - m_run + kPOff) : 0.f;
          psum += p[u];
        }
        whi[j4] = pack_e4m3x4(p[0], p[1], p[2], p[3]);
#pragma unroll
        for (int u = 0; u < 4; ++u)
          pl[u] = p[u] - e4m3_to_float((uint8_t)(whi[j4] >> (8 * u)));
        wlo[j4] = pack_e4m3x4(pl[0], pl[1], pl[2], pl[3]);
      }
      l_run = l_run * corr + psum;
      if (head_ok) {
        // this thread's 32 tokens = two 16-byte chunks of row hl of P^T (K-major, swizzled)
        const int tt = th * 64 + (hi_lane ? 0 : 32);
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
          const int chunk = (tt >> 4) + c2;
          const int off = hl * 128 + ((chunk ^ (hl & 7)) << 4);
          *reinterpret_cast<uint4*>(ps + off) =
              make_uint4(whi[4 * c2], whi[4 * c2 + 1], whi[4 * c2 + 2], whi[4 * c2 + 3]);
          *reinterpret_cast<uint4*>(ps + HG * 128 + off) =
              make_uint4(wlo[4 * c2], wlo[4 * c2 + 1], wlo[4 * c2 + 2], wlo[4 * c2 + 3]);
        }
      }
      // ---- rescale O^T when a running maximum moved (O(i-1) is complete: p_empty)
      if (!ta.first() && flag_s[i & 1] && alive) {
        constexpr int CWO = HG < 32 ? HG : 32;
#pragma unroll 1
        for (int a = 2 * th; a < 2 * th + 2; ++a) {
#pragma unroll 1
          for (int c0 = 0; c0 < HG; c0 += CWO) {
            const uint32_t tb = tq + kOCol + (uint32_t)(a * HG + c0);
            if (CWO == 32) {
              uint32_t d[32];
              tmem_ld_32x32b_x32(tb, d);
              tmem_wait_ld();
#pragma unroll
              for (int u = 0; u < 32; ++u) d[u] = __float_as_uint(__uint_as_float(d[u]) * corr_s[c0 + u]);
              tmem_st_32x32b_x32(tb, d);
            } else {
              uint32_t d[16];
              tmem_ld_32x32b_x16(tb, d);
              tmem_wait_ld();
#pragma unroll
              for (int u = 0; u < 16; ++u) d[u] = __float_as_uint(__uint_as_float(d[u]) * corr_s[c0 + u]);
              tmem_st_32x32b_x16(tb, d);
            }
          }
        }
        tmem_wait_st();
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
      if (i + 1 < n) {
        if (tn.lt == 0) len_ok = unit_len(tn);        // the next tile starts a unit
        valid_bits(tn, ida, idb, vlo, vhi);
      }
      if (!seg_last) continue;

      // ---- end of a segment: O complete -> normalised output (whole unit) or
      // a partial for the combine (unit cut by the CTA range)
      if (!wwait(p_empty, (uint32_t)i & 1, status)) alive = false;
      tc_fence_after();
      const float lpair = l_run + __shfl_xor_sync(0xffffffffu, l_run, 16);
      if (lane < 16 && head_ok) lsum_s[th * 64 + hl] = lpair;
      named_sync(1, kSmThreads);
      if (th == 0 && lane < 16 && head_ok) {          // output factor of head hl
        const float l = lsum_s[hl] + lsum_s[64 + hl];
        corr_s[hl] = (alive && l > 0.f) ? latent_scale / l : 0.f;
      }
      named_sync(1, kSmThreads);
      const bool whole = seg_lt0 == 0 && ta.lt == NT - 1;
      const int slot = 2 * c + (ta.u == u_first ? 0 : 1);
      const int r = ta.row(groups), hg0 = ta.hg0(groups, HG);
      constexpr int CWO = HG < 32 ? HG : 32;
#pragma unroll 1
      for (int a = 2 * th; a < 2 * th + 2; ++a) {
#pragma unroll 1
        for (int c0 = 0; c0 < HG; c0 += CWO) {
          uint32_t d[32];
          const uint32_t tb = tq + kOCol + (uint32_t)(a * HG + c0);
          if (alive) {
            if constexpr (CWO == 32) tmem_ld_32x32b_x32(tb, d);
            else tmem_ld_32x32b_x16(tb, *reinterpret_cast<uint32_t(*)[16]>(d));
            tmem_wait_ld();
          }
          const int dim = a * kMlaTile + quarter * 32 + lane;
#pragma unroll
          for (int u = 0; u < CWO; ++u) {
            const int h = c0 + u;
            const float o = alive ? __uint_as_float(d[u]) * corr_s[h] : 0.f;
            if (whole)
              out[((size_t)r * H + hg0 + h) * kVDim + dim] = __float2bfloat16_rn(o);
            else
              part_o[((size_t)slot * HG + h) * kVDim + dim] = o;
          }
        }
      }
      if (th == 0 && (lane & 16) == 0 && head_ok) {
        const float l = lsum_s[hl] + lsum_s[64 + hl];
        const float ls = (alive && l > 0.f && m_run > -INFINITY)
                             ? (m_run - kPOff + log2f(l)) * 0.6931471805599453f
                             : -INFINITY;
        if (!whole) part_lse[(size_t)slot * HG + hl] = ls;
        else if (lse_out) lse_out[(size_t)r * H + hg0 + hl] = ls;
      }
      tc_fence_before();
      m_run = -INFINITY;
      l_run = 0.f;
      if (i + 1 < n) {
        qcf = load_qc(tn.row(groups), tn.hg0(groups, HG));
        seg_lt0 = tn.lt;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// Merge of the partials of units cut by CTA ranges, by log-sum-exp.  One warp
// per (row, head, 1/W of the 512 dims), kCombHeads heads per CTA and no
// block-wide barrier: a lane takes the partials' lse values of splits lane,
// lane + 32, ...; two warp reductions give the maximum M and
// Z = sum_s e^{lse_s - M}; then every lane accumulates 16 / W dims over the
// splits (16-byte loads, two splits in flight), the split's slot and weight
// broadcast by a shuffle.  W > 1 spreads few rows over more SMs.  Units held
// whole by one CTA were written by the main kernel; with no slots at all
// (k = 0) the outputs are zero and lse = -inf.
constexpr int kCombHeads = 16;

template <int W>
__global__ void __launch_bounds__(32 * kCombHeads)
mla_combine_kernel(const float* part_o, const float* part_lse, int R,
                   int H, int k, __nv_bfloat16* __restrict__ out, float* __restrict__ lse) {
  constexpr int NQ = 4 / W;                         // 16-byte chunks per lane per split
  pdl_trigger();
  pdl_wait();                                       // the partials
  const int hq = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q0 = (int)blockIdx.y * (128 / W);       // first 16-byte chunk of this CTA's dims
  const int h = blockIdx.x % (H / kCombHeads) * kCombHeads + hq;
  const int r = blockIdx.x / (H / kCombHeads);
  const int HG = mla_heads_per_cta(H);
  const int u = r * (H / HG) + h / HG;
  const int hl = h % HG;
  const MlaWork w(R, H, k);
  int c0 = 0, c1 = -1;
  if (w.T > 0) {
    c0 = w.cta_of((int64_t)u * w.NT);
    c1 = w.cta_of((int64_t)(u + 1) * w.NT - 1);
    if (c0 == c1) return;                           // written by the main kernel
  }
  const int ns = c1 - c0 + 1;                       // 0 when there are no slots
  auto slot_of = [&](int sp) {
    const int c = c0 + sp;
    return 2 * c + (w.begin(c) / w.NT == u ? 0 : 1);
  };
  auto lse_of = [&](int sp) { return ld_dep(part_lse + (size_t)slot_of(sp) * HG + hl); };
  float M = -INFINITY;
  for (int sp = lane; sp < ns; sp += 32) M = fmaxf(M, lse_of(sp));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float Z = 0.f;
  for (int sp = lane; sp < ns; sp += 32) {
    const float l = lse_of(sp);
    Z += (M == -INFINITY || l == -INFINITY) ? 0.f : __expf(l - M);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) Z += __shfl_xor_sync(0xffffffffu, Z, o);
  const float inv = Z > 0.f ? 1.f / Z : 0.f;
  float4 acc[NQ];
#pragma unroll
  for (int q = 0; q < NQ; ++q) acc[q] = make_float4(0.f, 0.f, 0.f, 0.f);
  auto add = [&](float ws, const float4& v, float4& a) {
    a.x = fmaf(ws, v.x, a.x);
    a.y = fmaf(ws, v.y, a.y);
    a.z = fmaf(ws, v.z, a.z);
    a.w = fmaf(ws, v.w, a.w);
  };
  for (int sp0 = 0; sp0 < ns; sp0 += 32) {
    int my_slot = 0;
    float my_w = 0.f;
    if (sp0 + lane < ns) {
      my_slot = slot_of(sp0 + lane);
      const float l = ld_dep(part_lse + (size_t)my_slot * HG + hl);
      my_w = (M == -INFINITY || l == -INFINITY) ? 0.f : __expf(l - M) * inv;
    }
    const int cnt = min(32, ns - sp0);
    if constexpr (W == 4) {
      // few heads, many splits (one long row): eight splits in flight, one
      // memory round trip for most of them; missing ones weigh 0
      constexpr int NB = 8;
      for (int j = 0; j < cnt; j += NB) {
        float4 v[NB];
        float wv[NB];
#pragma unroll
        for (int b = 0; b < NB; ++b) {
          const bool has = j + b < cnt;
          const int sl = __shfl_sync(0xffffffffu, my_slot, (j + b) & 31);
          const float wt = __shfl_sync(0xffffffffu, my_w, (j + b) & 31);
          const int s0 = __shfl_sync(0xffffffffu, my_slot, j);
          wv[b] = has ? wt : 0.f;
          const float4* p =
              reinterpret_cast<const float4*>(part_o + ((size_t)(has ? sl : s0) * HG + hl) * kVDim);
          v[b] = ld_dep(p + q0 + lane);
        }
#pragma unroll
        for (int b = 0; b < NB; ++b) add(wv[b], v[b], acc[0]);
      }
      continue;
    }
    for (int j = 0; j < cnt; j += 2) {              // two splits in flight (the second may be empty)
      const int sa = __shfl_sync(0xffffffffu, my_slot, j);
      const float wa = __shfl_sync(0xffffffffu, my_w, j);
      const int sb = __shfl_sync(0xffffffffu, my_slot, (j + 1) & 31);
      const float wb = j + 1 < cnt ? __shfl_sync(0xffffffffu, my_w, (j + 1) & 31) : 0.f;
      const float4* pa = reinterpret_cast<const float4*>(part_o + ((size_t)sa * HG + hl) * kVDim);
      const float4* pb = reinterpret_cast<const float4*>(part_o + ((size_t)(j + 1 < cnt ? sb : sa) * HG + hl) * kVDim);
      float4 va[NQ], vb[NQ];
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        va[q] = ld_dep(pa + q0 + lane + 32 * q);
        vb[q] = ld_dep(pb + q0 + lane + 32 * q);
      }
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        add(wa, va[q], acc[q]);
        add(wb, vb[q], acc[q]);
      }
    }
  }
  __nv_bfloat16* dst = out + ((size_t)r * H + h) * kVDim;
#pragma unroll
  for (int q = 0; q < NQ; ++q) {
    __nv_bfloat162* d2 = reinterpret_cast<__nv_bfloat162*>(dst + (q0 + lane + 32 * q) * 4);
    d2[0] = __floats2bfloat162_rn(acc[q].x, acc[q].y);
    d2[1] = __floats2bfloat162_rn(acc[q].z, acc[q].w);
  }
  if (lse && lane == 0 && blockIdx.y == 0) lse[(size_t)r * H + h] = Z > 0.f ? M + logf(Z) : -INFINITY;
}

// The latent cache as a 2-D tensor of 576-byte rows (one per token slot); a box
// is box_bytes (128 or 64) of one row, stored with the swizzle of that span.
cudaError_t latent_tensor_map(CUtensorMap* map, const uint8_t* cache, int64_t num_pages,
                              uint32_t box_bytes) {
  // Row coordinates are signed 32-bit.  With no pages every lookup is rejected
  // before a coordinate is formed, so a one-page map is never dereferenced.
  if (num_pages * kPage > INT32_MAX) return cudaErrorInvalidValue;
  const int64_t rows = (num_pages > 0 ? num_pages : 1) * kPage;
  const uint64_t dims[2] = {(uint64_t)kLatDim, (uint64_t)rows};
  const uint64_t strides[1] = {(uint64_t)kLatDim};
  const uint32_t box[2] = {box_bytes, 1};
  return encode_tensor_map_u8(map, 2, cache, dims, strides, box, (int)box_bytes);
}

template <int HG, bool kNv>
cudaError_t launch_smla(const MlaArgs& a, const MlaLayout& L, int G, float lat_scale,
                        cudaStream_t st) {
  using S = MlaSmem<HG, kNv>;
  alignas(64) CUtensorMap map, rope;
  memset(&map, 0, sizeof(map));                       // NVFP4 rows are read without TMA
  memset(&rope, 0, sizeof(rope));
  cudaError_t e = cudaSuccess;
  if (!kNv) {
    e = latent_tensor_map(&map, a.latent_cache, a.num_pages, 128);
    if (e != cudaSuccess) return e;
    e = latent_tensor_map(&rope, a.latent_cache, a.num_pages, 64);
    if (e != cudaSuccess) return e;
  }
  e = cudaFuncSetAttribute(smla_kernel<HG, kNv>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           S::alloc);
  if (e != cudaSuccess) return e;
  e = launch_kernel(smla_kernel<HG, kNv>, dim3(G), dim3(kThreads), S::alloc, st, true, map, rope,
                    a.latent_cache, (const uint8_t*)(a.scratch + L.q8),
                    reinterpret_cast<const float*>(a.scratch + L.qc), a.H, a.num_pages,
                    lat_scale, a.block_table, a.B, a.max_pages, a.row_req, a.row_len, a.idx,
                    a.k, a.R, reinterpret_cast<float*>(a.scratch + L.part_o),
                    reinterpret_cast<float*>(a.scratch + L.part_lse),
                    static_cast<__nv_bfloat16*>(a.out), a.lse, a.status);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_sparse_mla(const MlaArgs& a, cudaStream_t st) {
  if (a.R == 0) return cudaSuccess;
  const MlaLayout L(a.R, a.H, a.k);
  const MlaWork w(a.R, a.H, a.k);
  if (w.G > 0) {
    const int warps = a.R * a.H;
    // NVFP4 operands hold c * s / 4 (see nvfp4_split32): the 4 joins the scale
    const float lat_scale = a.nvfp4 ? 4.f * a.latent_scale : a.latent_scale;
    cudaError_t e = launch_kernel(mla_qprep_kernel, dim3((warps + 7) / 8), dim3(256), 0, st,
                                  a.chained, static_cast<const __nv_bfloat16*>(a.q), a.R, a.H,
                                  a.softmax_scale, lat_scale, a.scratch + L.q8,
                                  reinterpret_cast<float*>(a.scratch + L.qc));
    if (e != cudaSuccess) return e;
    if (a.nvfp4) {
      if (a.H == 16) e = launch_smla<16, true>(a, L, w.G, lat_scale, st);
      else if (a.H == 32) e = launch_smla<32, true>(a, L, w.G, lat_scale, st);
      else e = launch_smla<64, true>(a, L, w.G, lat_scale, st);
    } else {
      if (a.H == 16) e = launch_smla<16, false>(a, L, w.G, lat_scale, st);
      else if (a.H == 32) e = launch_smla<32, false>(a, L, w.G, lat_scale, st);
      else e = launch_smla<64, false>(a, L, w.G, lat_scale, st);
    }
    if (e != cudaSuccess) return e;
  }
  // chained after the main kernel, or (no slots at all) after the caller's work
  const int nblk = a.R * a.H / kCombHeads;
  const int W = nblk >= kMlaGrid ? 1 : (2 * nblk >= kMlaGrid ? 2 : 4);
  auto kern = W == 1 ? mla_combine_kernel<1> : (W == 2 ? mla_combine_kernel<2> : mla_combine_kernel<4>);
  cudaError_t e = launch_kernel(kern, dim3(nblk, W), dim3(32 * kCombHeads), 0, st,
                                w.G > 0 || a.chained,
                                reinterpret_cast<const float*>(a.scratch + L.part_o),
                                reinterpret_cast<const float*>(a.scratch + L.part_lse), a.R, a.H,
                                a.k, static_cast<__nv_bfloat16*>(a.out), a.lse);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace dsa
