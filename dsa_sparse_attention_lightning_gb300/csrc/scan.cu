// scan.cu -- lightning-indexer scan (the Score step) on the tcgen05 tensor cores.
//
// score[r][s] = sum_h w[r][h] * ReLU(q[r][h] . key[s]) * ks[s] for s < row_len[r]
// (TokenSpeed post on Kimi K3.1 Pro, "Integrating sparse attention with the
// K3 stack", step 2; vLLM Day-0 post, "What Kimi K3.1 Pro changes": 32 heads
// x 128 dims, one FP8 key per token).  The key scale is a positive absmax
// scale (step 1 quantizes each key "to FP8 with a single scale"), so
// ReLU(x * ks) = ks * ReLU(x) and the scale is applied once after the head sum.
//
// Design (sm_103a):
//  * Rows of one request that are adjacent in the row order form a group of
//    up to 4 rows; the group's keys are read from HBM once for all its rows,
//    as the pages' MI350X scorer does for verification rows ("Reducing
//    indexer overhead on AMD MI350X").
//  * Per 128-token tile the contraction is one GEMM on the FP8 tensor cores,
//      D[token, (row, head)] = [K8 | K8][token, 0:256] . [Qhi | Qlo][(row, head), 0:256]^T,
//    M = 128 tokens, N = 32 x rows, K = 2 x 128, kind::f8f6f4 with f32
//    accumulators in tensor memory: the two query terms are two halves of
//    the contraction against the same key operand, so the tensor core adds
//    them.  The keys are the A operand exactly as they sit in the cache: TMA
//    moves a page's 64 x 128-byte key block straight into the
//    128-byte-swizzled K-major layout, no conversion.
//  * A bf16 query is split into two E4M3 terms per (row, head): s = q * 2^a
//    with a power of two putting the head's absmax in [128, 256), hi =
//    E4M3(s), lo = E4M3(s - hi); 2^-a is folded into the head weight.  The
//    split is exact for every |s| >= 1/4 (all but query elements below about
//    1/500 of the head's absmax, where lo keeps a 2^-9 grid).  An E4M3 query
//    is its own single term (K = 128: the lo half is neither loaded nor
//    multiplied) and its scale is folded into the weight.
//  * Each TMEM lane holds one token's (row, head) logits, so the
//    ReLU-weighted head sum is a per-thread loop: no shuffles.
//  * Persistent CTAs, one per SM, each taking a contiguous run of (group,
//    tile) work items; warp roles: 0-3 MMA issuers (tile i by warp i % 4;
//    warp 0 owns TMEM), 4-7 TMA producers (keys, key scales, group queries;
//    page ids looked up 32 tiles ahead; tile i is loaded by producer i % 4
//    -- the TMA loads one thread issues complete at well under the HBM
//    rate, so each SM runs four streams), 8-23 epilogue in two groups of
//    eight that take alternate tiles (TMEM -> scores; a warp takes TMEM
//    lane quarter w % 4, i.e. 32 tokens, of two of the group's rows).  A key
//    stage is released by the MMA's completion alone; the key scales live in
//    their own ring, held until the epilogue has used them.
//
// MXFP4 keys (scan_kernel<true>; vLLM Day-0 post, "Hybrid KV cache without
// padding" and "Native MXFP4 indexer": 68-byte keys, FP4 products with FP32
// accumulation): 64 bytes of E2M1 codes per token and one E8M0 scale per 32
// dims, the query in the same format.  The contraction is two block-scaled
// MMAs (kind::mxf4, K = 64) per tile with the scale factors in tensor memory,
// so there is no per-token scale in the epilogue:
//   score[r][s] = sum_h w[r][h] * ReLU(sum_b 2^(eq[r][h][b] + ek[s][b]) *
//                 (q4[r][h][b] . k4[s][b]))          (b = 32-dim block)
// The scale factors take tensor-memory columns, so this instance runs three
// accumulators instead of four.
#include <limits.h>
#include <math.h>

#include "dsa_common.cuh"
#include "sm100_ptx.cuh"

namespace dsa {
namespace {

using namespace ptx;

constexpr int kTileTok = 128;
constexpr int kMaxGroupRows = 4;
constexpr int kQAtom = kMaxGroupRows * kIdxHeads * kIdxDim;  // 128 rows x 128 B: one query term
constexpr int kQBytes = 2 * kQAtom;                     // one group's query operand (hi, lo)
constexpr int kQBufs = 1;
constexpr int kStages = 8;                              // key tiles in flight per SM
constexpr int kKeyTileBytes = kTileTok * kIdxDim;       // 2 pages x 64 x 128 B
constexpr int kPageKeyBytes = kPage * kIdxDim;          // 8192
constexpr int kPageBytes = kPage * (kIdxDim + 4);       // 8448: keys, then 64 f32 scales
constexpr int kScRing = 16;                             // key-scale slots (outlive their key stage)
constexpr int kMmaWarps = 4;                            // warps 0-3: lane 0 issues tiles i % 4 == warp
constexpr int kProdWarps = 4;                           // warps 4-7: one TMA stream per warp
constexpr int kEpiWarp0 = kMmaWarps + kProdWarps;       // warps 8-23
constexpr int kEpiGroups = 2;                           // epilogue group g takes tiles i % 2 == g
constexpr int kEpiWarpsPerGroup = 8;
constexpr int kEpiWarps = kEpiGroups * kEpiWarpsPerGroup;
constexpr int kEpiRows = kMaxGroupRows * 4 / kEpiWarpsPerGroup;  // group rows per epilogue warp
static_assert(kStages % kProdWarps == 0, "a stage always belongs to the same producer");
static_assert(kStages % kMmaWarps == 0, "a stage is always released by the same MMA issuer");
static_assert(kScRing % kProdWarps == 0 && kScRing % kEpiGroups == 0, "fixed slot owners");
constexpr int kThreads = (kEpiWarp0 + kEpiWarps) * 32;
constexpr int kDBufs = 4;
static_assert(kDBufs % kEpiGroups == 0, "a TMEM accumulator always belongs to the same group");
static_assert(kDBufs % kMmaWarps == 0 && kMmaWarps % kEpiGroups == 0,
              "an accumulator always belongs to the same MMA issuer and epilogue group");
constexpr int kDCols = kMaxGroupRows * kIdxHeads;       // 128 f32 columns per accumulator
constexpr uint32_t kTmemCols = kDCols * kDBufs;

// shared-memory map (offsets from a 1024-byte aligned base)
constexpr int kOffQ = 0;                                            // [kQBufs] query operands
constexpr int kOffKeys = kOffQ + kQBufs * kQBytes;                  // [kStages] key tiles
constexpr int kOffScale = kOffKeys + kStages * kKeyTileBytes;       // [kScRing][128] f32
constexpr int kOffPv = kOffScale + kScRing * kTileTok * 4;          // [kScRing] page-valid bits
constexpr int kOffW = (kOffPv + kScRing * 4 + 15) / 16 * 16;       // [kEpiWarps][kEpiRows][32] f32
constexpr int kOffBar = (kOffW + kEpiWarps * kEpiRows * kIdxHeads * 4 + 7) / 8 * 8;
static_assert(kOffKeys % 1024 == 0 && kKeyTileBytes % 1024 == 0, "swizzled TMA tiles need 1024-byte alignment");
static_assert(kOffScale % 16 == 0 && kOffW % 16 == 0 && kOffBar % 8 == 0, "vector and mbarrier alignment");
constexpr int kDBars = 12;                               // accumulator barriers (MXFP4: tile mod 12)
constexpr int kNumBars = 2 * kStages + 2 * kScRing + 2 * kDBars + 2 * kQBufs + kMmaWarps;
constexpr int kOffTmem = kOffBar + kNumBars * 8;
constexpr int kSmemBytes = kOffTmem + 16;
constexpr int kSmemAlloc = kSmemBytes + 1024;
static_assert(kSmemAlloc <= 227 * 1024, "shared memory per CTA");

// MXFP4 keys (68 bytes per token: 64 bytes of E2M1 codes, then one E8M0 scale
// per 32 dims).  Page: 64 x 64 code bytes, then 64 x 4 scale bytes.  The same
// shared-memory plan with half-size key stages; the scale-factor rows that the
// tensor core reads sit in the key region's unused second half.
constexpr int kMxKeyBytes = kIdxDim / 2;
constexpr int kMxPageKeyBytes = kPage * kMxKeyBytes;                // 4096
constexpr int kMxKeyTileBytes = kTileTok * kMxKeyBytes;             // 8192
constexpr int kMxQAtom = kMaxGroupRows * kIdxHeads * kMxKeyBytes;   // 128 rows x 64 B
constexpr int kSfRowBytes = 32 * 16;                                // 32 rows x 16 B
constexpr int kOffSfaMx = kOffKeys + kStages * kMxKeyTileBytes;     // [kScRing] key scale rows
constexpr int kMxDBufs = 3;                                         // accumulators (TMEM holds the scales too)
constexpr uint32_t kSfCol0 = kDCols * kMxDBufs;                     // scale columns: 8 per slot
constexpr int kSfSlots = 12;                                        // tile i's scales in slot i % 12
static_assert(kOffSfaMx + kScRing * kSfRowBytes <= kOffScale, "scale rows fit the key region");
static_assert(kMxQAtom + kSfRowBytes <= kQBytes, "query codes and scale rows fit the query buffer");
static_assert(kSfCol0 + 8 * kSfSlots <= kTmemCols, "scale columns fit the allocation");
static_assert(kSfSlots == kDBars, "a scale slot is tracked by the tile's accumulator barrier");
// Three accumulators, tile i in accumulator i % 3, signalled on barrier pair
// i % 12: each barrier is waited on by one epilogue group (i % 2) in tile
// order, and the MMA warp of tile i (i % 4) waits for tile i - 3's release on
// barrier (i - 3) % 12, whose previous phase (tile i - 15) it already waited
// for at tile i - 12, so no parity wait can be satisfied by an older phase.
// Tile i's scale factors go to their own TMEM slot i % 12, which tile i - 12
// last read: the same warp waits for that tile's MMA completion (barrier
// d_full[i % 12], previous phase; tile i - 24's phase completed before the
// warp's own wait at tile i - 12 returned) and copies the scales in before
// its key and accumulator waits, off the path from an epilogue release to the
// next MMA.
static_assert(kDBars % kMxDBufs == 0 && kDBars % kEpiGroups == 0 && kDBars % kMmaWarps == 0 &&
              kDBars >= kDBufs, "accumulator barrier indexing");

// group = {first row, rows, request, max row length}
struct ScanWs {
  uint8_t* q8;     // [2 terms][R][32 heads][128] E4M3 query terms
  float* weff;     // [R][32] head weight times the inverse rescale (and query scale)
  int4* groups;    // [R]
  int* gstart;     // [R + 1] first tile of each group
  int* meta;       // {groups, tiles}
  int4* cta;       // [kMaxScanCtas] {first group, first tile, end tile, groups} of each scan CTA
};

// The prep kernel hands every scan CTA its tile range and first group, so a
// CTA starts with one load instead of a search of the group table; a grid of
// more CTAs searches.
constexpr int kMaxScanCtas = 256;

ScanWs scan_ws(uint8_t* base, int R) {
  ScanWs w;
  size_t o = 0;
  w.q8 = base + o;                              o = align_up(o + (size_t)2 * R * kIdxHeads * kIdxDim);
  w.weff = reinterpret_cast<float*>(base + o); o = align_up(o + (size_t)R * kIdxHeads * 4);
  w.groups = reinterpret_cast<int4*>(base + o); o = align_up(o + (size_t)R * 16);
  w.gstart = reinterpret_cast<int*>(base + o);  o = align_up(o + (size_t)(R + 1) * 4);
  w.meta = reinterpret_cast<int*>(base + o);  o = align_up(o + 16);
  w.cta = reinterpret_cast<int4*>(base + o);
  return w;
}

// ---------------------------------------------------------------------------
// Prep, one launch of R + 1 CTAs of 1024 threads.
//  * CTA r < R: warp h splits head h of row r's query into its two E4M3
//    terms (power-of-two rescale per head, folded into the head weight).
//  * CTA R: groups the rows.  A run is a maximal block of adjacent valid rows
//    of one request; each run is cut into groups of up to 4 rows from its
//    start.  Block-wide scans over chunks of 1024 rows give every row its run
//    start, every group its index and every group its first tile.
//  * MXFP4 query (q_dtype kQMxfp4): the codes are used as they are; CTA r
//    only copies the head weights, and CTA R lays out each group's query
//    scales as the tensor core's scale-factor rows (in the q8 area): row h,
//    32-bit word j = the four E8M0 scales of head h of the group's row j.
constexpr int kPrepThreads = 1024;
constexpr int kPrepGroupCache = 4096;          // group starts kept in shared memory

template <typename T, typename Op>
__device__ __forceinline__ T block_scan_incl(T v, T* warp_buf, Op op, T identity) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const T n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v = op(v, n);
  }
  if (lane == 31) warp_buf[wid] = v;
  __syncthreads();
  if (wid == 0) {
    T x = warp_buf[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const T n = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x = op(x, n);
    }
    warp_buf[lane] = x;
  }
  __syncthreads();
  const T add = wid > 0 ? warp_buf[wid - 1] : identity;
  __syncthreads();
  return op(v, add);
}

struct OpMax { __device__ int operator()(int a, int b) const { return a > b ? a : b; } };
struct OpAdd { __device__ int operator()(int a, int b) const { return a + b; } };

__device__ __forceinline__ bool row_valid(const int32_t* row_req, const int32_t* row_len, int r,
                                          int R, int B, int max_pages) {
  if (r < 0 || r >= R) return false;
  const int req = row_req[r], len = row_len[r];
  return req >= 0 && req < B && len >= 0 && (int64_t)len <= (int64_t)max_pages * kPage;
}

__global__ void __launch_bounds__(kPrepThreads)
scan_prep_kernel(const void* __restrict__ q_idx, int q_dtype, const float* __restrict__ q_scale,
                 const uint8_t* __restrict__ q_sf, const float* __restrict__ w,
                 const int32_t* __restrict__ row_req,
                 const int32_t* __restrict__ row_len, int R, int B, int max_pages, int nctas,
                 ScanWs ws, uint32_t* status, int clear_status) {
  pdl_wait();
  pdl_trigger();
  if (blockIdx.x == (unsigned)R) {
    __shared__ int warp_buf[32];
    __shared__ int s_carry[3];   // run start of the last row, groups so far, tiles so far
    __shared__ int s_gstart[kPrepGroupCache + 1];   // group tile starts, for the CTA-range search
    if (threadIdx.x == 0) {
      s_carry[0] = -1; s_carry[1] = 0; s_carry[2] = 0;
      // the first writer of the step's status word: every raise comes after
      // this (below in this block, or in kernels that wait for this grid)
      if (clear_status) *status = 0u;
    }
    __syncthreads();
    for (int base = 0; base < R; base += kPrepThreads) {
      const int r = base + threadIdx.x;
      const bool v = row_valid(row_req, row_len, r, R, B, max_pages);
      if (r < R && !v) raise_dev(status, DSA_DEV_BAD_ROW);
      const int req = v ? row_req[r] : -1;
      const bool pv = row_valid(row_req, row_len, r - 1, R, B, max_pages);
      const bool run_head = v && (!pv || row_req[r - 1] != req);
      const int carry_run = s_carry[0], carry_groups = s_carry[1], carry_tiles = s_carry[2];
      int run_start = block_scan_incl(run_head ? r : -1, warp_buf, OpMax(), -1);
      if (run_start < 0) run_start = carry_run;         // run continues from the last chunk
      const bool head = v && ((r - run_start) & 3) == 0;
      int nrows = 0, maxlen = 0;
      if (head) {
        for (int j = 0; j < 4; ++j) {
          const int rr = r + j;
          if (j > 0 && (!row_valid(row_req, row_len, rr, R, B, max_pages) || row_req[rr] != req))
            break;
          ++nrows;
          maxlen = max(maxlen, (int)row_len[rr]);
        }
      }
      const int tiles = head ? (maxlen + kTileTok - 1) / kTileTok : 0;
      const int g_incl = block_scan_incl(head ? 1 : 0, warp_buf, OpAdd(), 0);
      const int t_incl = block_scan_incl(tiles, warp_buf, OpAdd(), 0);
      if (head) {
        const int g = carry_groups + g_incl - 1;
        ws.groups[g] = make_int4(r, nrows, req, maxlen);
        ws.gstart[g] = carry_tiles + t_incl - tiles;
        if (g < kPrepGroupCache) s_gstart[g] = carry_tiles + t_incl - tiles;
      }
      __syncthreads();                                    // everyone has read the carries
      if (threadIdx.x == kPrepThreads - 1) {
        s_carry[0] = v ? run_start : -1;
        s_carry[1] = carry_groups + g_incl;
        s_carry[2] = carry_tiles + t_incl;
      }
      __syncthreads();
    }
    if (threadIdx.x == 0) {
      ws.gstart[s_carry[1]] = s_carry[2];
      ws.meta[0] = s_carry[1];
      ws.meta[1] = s_carry[2];
    }
    // each scan CTA's tile range and the group holding its first tile (the
    // last group whose first tile is <= it, as TileCursor::seek finds it)
    const int ngroups = s_carry[1], total = s_carry[2];
    // the search reads the group starts from shared memory when they fit (one
    // dependent global load per step otherwise)
    const int* gs = ngroups <= kPrepGroupCache ? s_gstart : ws.gstart;
    if (nctas <= kMaxScanCtas) {
      for (int c = threadIdx.x; c < nctas; c += kPrepThreads) {
        const int tb = (int)((int64_t)total * c / nctas);
        const int te = (int)((int64_t)total * (c + 1) / nctas);
        int lo = 0, hi = ngroups;
        while (hi - lo > 1) {
          const int mid = (lo + hi) >> 1;
          if (gs[mid] <= tb) lo = mid; else hi = mid;
        }
        ws.cta[c] = make_int4(lo, tb, te, ngroups);
      }
    }
    if (q_dtype == kQMxfp4) {
      __syncthreads();                                    // every group is written
      const uint32_t* qs = reinterpret_cast<const uint32_t*>(q_sf);   // [R][32] words
      uint32_t* rows = reinterpret_cast<uint32_t*>(ws.q8);            // [groups][32][4] words
      for (int e = threadIdx.x; e < ngroups * 128; e += kPrepThreads) {
        const int g = e >> 7, h = (e >> 2) & 31, j = e & 3;
        const int4 G = ws.groups[g];
        rows[e] = j < G.y ? qs[(size_t)(G.x + j) * kIdxHeads + h] : 0x7F7F7F7Fu;
      }
    }
    return;
  }
  if (q_dtype == kQMxfp4) {                         // the head weights as they are
    const int r = blockIdx.x;
    if (threadIdx.x < kIdxHeads)
      ws.weff[(size_t)r * kIdxHeads + threadIdx.x] = w[(size_t)r * kIdxHeads + threadIdx.x];
    return;
  }
  // query split: warp h handles head h of row r, lane l dims [4l, 4l + 4)
  const int r = blockIdx.x;
  const int h = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t off = ((size_t)r * kIdxHeads + h) * kIdxDim + lane * 4;
  uint8_t* hi_dst = ws.q8 + ((size_t)r * kIdxHeads + h) * kIdxDim + lane * 4;
  uint8_t* lo_dst = hi_dst + (size_t)R * kIdxHeads * kIdxDim;
  float wv = w[(size_t)r * kIdxHeads + h];
  if (q_dtype == DSA_E4M3) {                        // already one E4M3 term
    *reinterpret_cast<uint32_t*>(hi_dst) =
        *reinterpret_cast<const uint32_t*>(static_cast<const uint8_t*>(q_idx) + off);
    wv *= q_scale[(size_t)r * kIdxHeads + h];
  } else {
    const uint2 v = *reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(q_idx) + off);
    float x[4];
    x[0] = __uint_as_float(v.x << 16);
    x[1] = __uint_as_float(v.x & 0xFFFF0000u);
    x[2] = __uint_as_float(v.y << 16);
    x[3] = __uint_as_float(v.y & 0xFFFF0000u);
    float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    int a = 0;
    if (amax > 0.f) a = 7 - ilogbf(amax);          // absmax into [128, 256)
    uint32_t hw = 0, lw = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float sx = ldexpf(x[i], a);             // exact: a power of two
      const uint8_t h8 = (uint8_t)__nv_cvt_float_to_fp8(sx, __NV_SATFINITE, __NV_E4M3);
      const float rr = sx - e4m3_to_float(h8);      // exact: both on a common grid
      const uint8_t l8 = (uint8_t)__nv_cvt_float_to_fp8(rr, __NV_SATFINITE, __NV_E4M3);
      hw |= (uint32_t)h8 << (8 * i);
      lw |= (uint32_t)l8 << (8 * i);
    }
    *reinterpret_cast<uint32_t*>(hi_dst) = hw;
    *reinterpret_cast<uint32_t*>(lo_dst) = lw;
    wv = ldexpf(wv, -a);
  }
  if (lane == 0) ws.weff[(size_t)r * kIdxHeads + h] = wv;
}

// ---------------------------------------------------------------------------
// Walks the flattened (group, tile) work list; empty groups are skipped.  The
// current group's tile range and descriptor are cached in registers.
struct TileCursor {
  const int4* groups;
  const int* gstart;
  int ngroups;
  int g, t, gs, ge;
  int4 G;
  __device__ void load() {
    gs = gstart[g];
    ge = gstart[g + 1];
    G = groups[g];
  }
  __device__ void start(int g0, int tile) {   // tile lies in group g0 (non-empty)
    g = g0;
    load();
    t = tile - gs;
  }
  __device__ void seek(int tile) {
    int lo = 0, hi = ngroups;              // last g in [0, ngroups) with gstart[g] <= tile
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (gstart[mid] <= tile) lo = mid; else hi = mid;
    }
    g = lo;
    load();
    t = tile - gs;
  }
  // n tiles forward (crossing group boundaries; at most one load per group crossed)
  __device__ void advance(int n) {
    while (n > 0 && g < ngroups) {
      const int left = (ge - gs) - t - 1;
      if (n <= left) {
        t += n;
        return;
      }
      n -= left + 1;
      ++g;
      t = 0;
      while (g < ngroups && gstart[g] == gstart[g + 1]) ++g;
      if (g < ngroups) load();
    }
  }
  __device__ void next() {
    if (g >= ngroups) return;
    ++t;
    if (gs + t >= ge) {
      ++g;
      t = 0;
      while (g < ngroups && gstart[g] == gstart[g + 1]) ++g;
      if (g < ngroups) load();
    }
  }
};

// Lane 0 waits (bounded); the outcome is the same for the whole warp.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, uint32_t* status) {
  bool ok = true;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, status);
  return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

// Polls without suspending the thread (bounded like mbar_wait).  The
// accumulator barriers are waited on this way: a waiter suspended by
// try_wait resumed measurably later after the phase completed (256K scan:
// MXFP4 147 -> 142 us, FP8 138.9 -> 137.6 us).
__device__ __forceinline__ bool mbar_wait_spin(uint64_t* bar, uint32_t parity, uint32_t* status) {
  if (mbar_test(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_test(bar, parity)) {
    if (clock64() - t0 > kWaitCycles) {
      raise_dev(status, DSA_DEV_TIMEOUT);
      return false;
    }
  }
  return true;
}

// Lane 0 polls (mbar_wait_spin); the outcome is the same for the whole warp.
__device__ __forceinline__ bool warp_wait_spin(uint64_t* bar, uint32_t parity, uint32_t* status) {
  bool ok = true;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait_spin(bar, parity, status);
  return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

// ---- TMA: tensor-map tile loads completing on an mbarrier -------------------
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z,
                                            uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar)),
      "l"(policy)
      : "memory");
}

__device__ __forceinline__ bool page_ok(int p, int64_t num_pages) { return p >= 0 && p < num_pages; }

// Physical pages of a tile's two 64-token halves (-1: past the group's tokens).
// Loads use clamped offsets so that no select waits on them.
struct TilePages {
  int p0, p1;
  bool need0, need1;
};

__device__ __forceinline__ TilePages tile_pages(const TileCursor& c, const int32_t* block_table,
                                                int max_pages) {
  TilePages t;
  const int lp0 = c.t * (kTileTok / kPage);
  const int npg = (c.G.w + kPage - 1) / kPage;
  t.need0 = lp0 < npg;
  t.need1 = lp0 + 1 < npg;
  const size_t base = (size_t)c.G.z * max_pages;
  t.p0 = __ldg(block_table + base + (t.need0 ? lp0 : 0));
  t.p1 = __ldg(block_table + base + (t.need1 ? lp0 + 1 : 0));
  return t;
}

// MXFP4 MMA issuers (warps 0-3, tiles i % 4 == warp): the whole warp turns
// the tile's key scales (landed in token order) into the tensor core's
// scale-factor rows -- row l = the four scale bytes of tokens l, l + 32,
// l + 64, l + 96 -- and lane 0 copies them and the group's query scale rows
// into tensor memory, then issues the two K = 64 block-scaled MMAs (scale
// bytes 0-1, then 2-3).  The MMA takes the scales of operand row m (a token,
// or a (row, head) column) from lane m % 32, column base + m / 32, which is
// where the replicated 32-row copy puts them.
__device__ __forceinline__ void mx_mma_issuer(uint8_t* smem, TileCursor cur, int ntiles,
                                              uint32_t tmem_base, uint64_t* bars,
                                              uint32_t* status) {
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  uint64_t* sc_full = bars + 2 * kStages;
  uint64_t* sc_empty = sc_full + kScRing;
  uint64_t* d_full = sc_empty + kScRing;
  uint64_t* d_empty = d_full + kDBars;
  uint64_t* q_full = d_empty + kDBars;
  uint64_t* q_empty = q_full + kQBufs;
  uint64_t* mma_done = q_empty + kQBufs;
  const int m = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int cur_group = -1, gi = -1, left = 0;
  bool issued_in_group = false;
  uint32_t idesc0 = 0, idesc1 = 0;
  const uint64_t a_desc_base = desc_kmajor_sw64(smem_u32(smem + kOffKeys));
  const uint64_t b_desc = desc_kmajor_sw64(smem_u32(smem + kOffQ));
  const uint64_t sfb_desc = desc_sf_rows16(smem_u32(smem + kOffQ + kMxQAtom));
  int s = 0;
  uint32_t s_phase = 0;
  for (int i = 0; i < ntiles; ++i) {
    if (cur.g != cur_group) {
      cur_group = cur.g;
      ++gi;
      left = (cur.ge - cur.gs) - cur.t;
      issued_in_group = false;
      idesc0 = idesc_mxf4(kTileTok, kIdxHeads * cur.G.y, 0, 0);
      idesc1 = idesc_mxf4(kTileTok, kIdxHeads * cur.G.y, 2, 2);
      if (!warp_wait(&q_full[gi % kQBufs], (uint32_t)(gi / kQBufs) & 1, status)) break;
    }
    if (i % kMmaWarps == m) {
      const int db = i % kMxDBufs, x = i % kScRing, c = i % kDBars;
      // the scale rows are built before the accumulator wait, off the path
      // from the previous epilogue to this tile's MMAs
      if (!warp_wait(&sc_full[x], (uint32_t)(i / kScRing) & 1, status)) break;
      const uint32_t* tok = reinterpret_cast<const uint32_t*>(smem + kOffScale + x * kTileTok * 4);
      uint8_t* sf_rows = smem + kOffSfaMx + x * kSfRowBytes;
      *reinterpret_cast<uint4*>(sf_rows + lane * 16) =
          make_uint4(tok[lane], tok[lane + 32], tok[lane + 64], tok[lane + 96]);
      fence_proxy_async_smem();                       // visible to the tensor core's copy
      __syncwarp();
      // scale slot c was last read by the MMAs of tile i - 12, which completed
      // on barrier c's previous phase; the copies into it go out before the
      // key and accumulator waits
      if (i >= kSfSlots && !warp_wait(&d_full[c], (uint32_t)((i - kSfSlots) / kDBars) & 1, status))
        break;
      const uint32_t sfa = tmem_base + kSfCol0 + (uint32_t)(c * 8), sfb = sfa + 4;
      if (lane == 0) {
        tc_fence_after();
        tmem_cp_32x128b_warpx4(sfa, desc_sf_rows16(smem_u32(sf_rows)));
        tmem_cp_32x128b_warpx4(sfb, sfb_desc);
      }
      if (!warp_wait(&full[s], s_phase, status)) break;
      // the previous user of accumulator db is tile i - 3 (barrier (i - 3) % 12;
      // for i < 3 the wait is on a fresh barrier's preceding phase)
      if (!warp_wait_spin(&d_empty[(i + kDBars - kMxDBufs) % kDBars],
                          ((uint32_t)((i + kDBars - kMxDBufs) / kDBars) & 1) ^ 1, status))
        break;
      if (lane == 0) {
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(db * kDCols);
        const uint64_t a_desc = a_desc_base + (uint64_t)((s * kMxKeyTileBytes) >> 4);
        mma_mxf4_ss(d_tmem, a_desc, b_desc, idesc0, sfa, sfb, 0u);
        mma_mxf4_ss(d_tmem, a_desc + 2, b_desc + 2, idesc1, sfa, sfb, 1u);   // + 32 bytes of K
        mma_commit(&empty[s]);
        mma_commit(&sc_empty[x]);
        mma_commit(&d_full[c]);
      }
      __syncwarp();
      issued_in_group = true;
    }
    --left;
    if ((i + 1 == ntiles || left == 0) && lane == 0) {   // the group's query operand is released
      if (issued_in_group) mma_commit(&q_empty[gi % kQBufs]);
      else mbar_arrive(&q_empty[gi % kQBufs]);
    }
    if (++s == kStages) {
      s = 0;
      s_phase ^= 1u;
    }
    if (left == 0 && i + 1 < ntiles) cur.advance(cur.ge - cur.gs - cur.t);   // next group
  }
  if (lane == 0) {
    mma_commit(&mma_done[m]);                         // tensor memory is freed only after this
    mbar_wait(&mma_done[m], 0, status);
  }
  __syncwarp();
}

template <bool kMx>
__global__ void __launch_bounds__(kThreads, 1)
scan_kernel(const __grid_constant__ CUtensorMap key_map, const __grid_constant__ CUtensorMap q_map,
            const uint8_t* __restrict__ key_cache, int64_t num_pages,
            const int32_t* __restrict__ block_table, int max_pages,
            const int32_t* __restrict__ row_len, float* __restrict__ scores, int64_t ld,
            int n_rows, int q_terms, ScanWs ws, uint32_t* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* full = bars;                            // [kStages] keys landed
  uint64_t* empty = bars + kStages;                 // [kStages] MMA done with a key stage
  uint64_t* sc_full = bars + 2 * kStages;           // [kScRing] scales landed
  uint64_t* sc_empty = sc_full + kScRing;           // [kScRing] epilogue done with them
  uint64_t* d_full = sc_empty + kScRing;            // [kDBars]
  uint64_t* d_empty = d_full + kDBars;              // [kDBars]
  uint64_t* q_full = d_empty + kDBars;              // [kQBufs]
  uint64_t* q_empty = q_full + kQBufs;              // [kQBufs]
  uint64_t* mma_done = q_empty + kQBufs;            // [kMmaWarps] every MMA of an issuer finished
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffTmem);
  const float* scale_s = reinterpret_cast<const float*>(smem + kOffScale);
  uint32_t* pv_s = reinterpret_cast<uint32_t*>(smem + kOffPv);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int x = 0; x < kStages; ++x) {
      mbar_init(&full[x], 1);
      mbar_init(&empty[x], 1);                      // the MMA commit
    }
    for (int x = 0; x < kScRing; ++x) {
      mbar_init(&sc_full[x], 1);
      mbar_init(&sc_empty[x], kEpiWarpsPerGroup + (kMx ? 1 : 0));   // MXFP4: + the MMA commit
    }
    for (int b = 0; b < kDBars; ++b) {
      mbar_init(&d_full[b], 1);
      mbar_init(&d_empty[b], kEpiWarpsPerGroup);
    }
    for (int b = 0; b < kQBufs; ++b) {
      mbar_init(&q_full[b], 1);
      mbar_init(&q_empty[b], kMmaWarps);            // one release per MMA issuer
    }
    for (int m = 0; m < kMmaWarps; ++m) mbar_init(&mma_done[m], 1);
    fence_mbar_init();
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
  pdl_wait();                                       // the prep kernel's groups and query terms

  const bool handed = gridDim.x <= (unsigned)kMaxScanCtas;   // range from the prep kernel
  int ngroups, t_begin, t_end, g_begin = 0;
  if (handed) {
    const int4 cs = ws.cta[blockIdx.x];
    g_begin = cs.x;
    t_begin = cs.y;
    t_end = cs.z;
    ngroups = cs.w;
  } else {
    ngroups = ws.meta[0];
    const int total = ws.meta[1];
    t_begin = (int)((int64_t)total * blockIdx.x / gridDim.x);
    t_end = (int)((int64_t)total * (blockIdx.x + 1) / gridDim.x);
  }
  const int ntiles = t_end - t_begin;
  TileCursor cur;
  cur.groups = ws.groups;
  cur.gstart = ws.gstart;
  cur.ngroups = ngroups;
  if (ntiles > 0) {
    if (handed) cur.start(g_begin, t_begin);
    else cur.seek(t_begin);
  }

  if (ntiles > 0 && warp < kMmaWarps) {
    if constexpr (kMx) {
      mx_mma_issuer(smem, cur, ntiles, tmem_base, bars, status);
    } else {
      // ---------------- MMA issuers: lane 0 of warp m issues the tiles i with
      // i % kMmaWarps == m.  An issuing thread is held at every tcgen05.mma
      // until the tensor core takes it, and its barrier waits and commits cost
      // about as much again per tile; with four issuers the others'
      // bookkeeping overlaps one thread's MMAs (256K scan: 141.5 -> 138.8 us
      // against two issuers).  All walk every tile to follow the group, stage
      // and accumulator sequence.
      if (lane == 0) {
        const int m = warp;
        int cur_group = -1, gi = -1, left = 0;          // tiles left in the current group
        bool issued_in_group = false;
        uint32_t idesc = 0;
        uint64_t b_desc = 0;
        const uint64_t a_desc_base = desc_kmajor_sw128(smem_u32(smem + kOffKeys));
        int s = 0;                                      // key stage of tile i
        uint32_t s_phase = 0;
        for (int i = 0; i < ntiles; ++i) {
          if (cur.g != cur_group) {
            cur_group = cur.g;
            ++gi;
            left = (cur.ge - cur.gs) - cur.t;
            issued_in_group = false;
            idesc = idesc_e4m3_f32(kTileTok, kIdxHeads * cur.G.y, false, false);
            b_desc = desc_kmajor_sw128(smem_u32(smem + kOffQ + (gi % kQBufs) * kQBytes));
            if (!mbar_wait(&q_full[gi % kQBufs], (uint32_t)(gi / kQBufs) & 1, status)) break;
          }
          if (i % kMmaWarps == m) {
            const int db = i % kDBufs;
            if (!mbar_wait(&full[s], s_phase, status)) break;
            if (!mbar_wait_spin(&d_empty[db], ((uint32_t)(i / kDBufs) & 1) ^ 1, status)) break;
            tc_fence_after();
            const uint64_t a_desc = a_desc_base + (uint64_t)((s * kKeyTileBytes) >> 4);
            const uint32_t d_tmem = tmem_base + (uint32_t)(db * kDCols);
  #pragma unroll
            for (int j = 0; j < 2 * kIdxDim / 32; ++j) {  // K = q_terms x 128 bytes in steps of 32
              if (j >= q_terms * (kIdxDim / 32)) break;
              mma_e4m3_ss(d_tmem, a_desc + (uint64_t)((j & 3) * 2),
                          b_desc + (uint64_t)(((j >> 2) * kQAtom + (j & 3) * 32) >> 4), idesc,
                          j > 0 ? 1u : 0u);
            }
            mma_commit(&empty[s]);
            mma_commit(&d_full[db]);
            issued_in_group = true;
          }
          --left;
          if (i + 1 == ntiles || left == 0) {           // the group's query operand is released
            if (issued_in_group) mma_commit(&q_empty[gi % kQBufs]);
            else mbar_arrive(&q_empty[gi % kQBufs]);
          }
          if (++s == kStages) {
            s = 0;
            s_phase ^= 1u;
          }
          if (left == 0 && i + 1 < ntiles) cur.advance(cur.ge - cur.gs - cur.t);   // next group
        }
        mma_commit(&mma_done[m]);                       // tensor memory is freed only after this
        mbar_wait(&mma_done[m], 0, status);
      }
      __syncwarp();
    }
  } else if (ntiles > 0 && warp >= kMmaWarps && warp < kEpiWarp0) {
    // ---------------- TMA producers: warp kMmaWarps + p loads the tiles i with
    // i % kProdWarps == p.  Page ids are looked up a batch of 32 tiles ahead:
    // lane j holds the pages of tile (batch start + j).
    const int pw = warp - kMmaWarps;
    const uint64_t stream_policy = l2_policy_evict_first();
    auto fetch = [&](const TileCursor& b0, int i0) {
      TilePages tp{0, 0, false, false};
      if (i0 + lane < ntiles) {
        TileCursor cj = b0;
        cj.advance(lane);
        tp = tile_pages(cj, block_table, max_pages);
      }
      return tp;
    };
    TileCursor bc = cur;                              // start of the current batch
    TilePages cb = fetch(bc, 0);
    TileCursor bn = bc;
    TilePages nb{0, 0, false, false};
    if (ntiles > 32) {
      bn.advance(32);
      nb = fetch(bn, 32);
    }
    int cur_group = -1, gi = -1;
    bool ok = true;
    for (int i = 0; i < ntiles && ok; ++i) {
      const int j = i & 31;
      if (j == 0 && i > 0) {                          // next batch; fetch the one after it
        cb = nb;
        bc = bn;
        if (i + 32 < ntiles) {
          bn.advance(32);
          nb = fetch(bn, i + 32);
        }
      }
      const int p0 = __shfl_sync(0xffffffffu, cb.p0, j);
      const int p1 = __shfl_sync(0xffffffffu, cb.p1, j);
      const bool need0 = __shfl_sync(0xffffffffu, cb.need0 ? 1 : 0, j) != 0;
      const bool need1 = __shfl_sync(0xffffffffu, cb.need1 ? 1 : 0, j) != 0;
      if (cur.g != cur_group) {                       // the group's query operand
        cur_group = cur.g;
        ++gi;
        if (i % kProdWarps != pw) {                   // loaded by the owner of this tile
          cur.next();
          continue;
        }
        if (!warp_wait(&q_empty[gi % kQBufs], ((uint32_t)(gi / kQBufs) & 1) ^ 1, status)) break;
        if (lane == 0) {
          uint8_t* qd = smem + kOffQ + (gi % kQBufs) * kQBytes;
          if constexpr (kMx) {                        // codes, then the group's scale rows
            mbar_arrive_expect_tx(&q_full[gi % kQBufs], kMxQAtom + kSfRowBytes);
            tma_load_2d(qd, &q_map, 0, cur.G.x * kIdxHeads, &q_full[gi % kQBufs]);
            bulk_g2s(qd + kMxQAtom, ws.q8 + (size_t)cur.g * kSfRowBytes, kSfRowBytes,
                     &q_full[gi % kQBufs]);
          } else {
            mbar_arrive_expect_tx(&q_full[gi % kQBufs], q_terms * kQAtom);
            tma_load_2d(qd, &q_map, 0, cur.G.x * kIdxHeads, &q_full[gi % kQBufs]);
            if (q_terms == 2)
              tma_load_2d(qd + kQAtom, &q_map, 0, (n_rows + cur.G.x) * kIdxHeads,
                          &q_full[gi % kQBufs]);
          }
        }
      }
      if (i % kProdWarps != pw) {
        cur.next();
        continue;
      }
      const int s = i % kStages, x = i % kScRing;
      if (!warp_wait(&empty[s], ((uint32_t)(i / kStages) & 1) ^ 1, status)) break;
      if (!warp_wait(&sc_empty[x], ((uint32_t)(i / kScRing) & 1) ^ 1, status)) break;
      if (lane == 0) {
        const bool v0 = need0 && page_ok(p0, num_pages);
        const bool v1 = need1 && page_ok(p1, num_pages);
        if ((need0 && !v0) || (need1 && !v1)) raise_dev(status, DSA_DEV_BAD_PAGE);
        pv_s[x] = (v0 ? 1u : 0u) | (v1 ? 2u : 0u);
        // key codes of the two pages, and their scales in token order (fp32
        // per token, or the four E8M0 bytes per token of MXFP4 keys)
        constexpr int kStage = kMx ? kMxKeyTileBytes : kKeyTileBytes;
        constexpr int kHalf = kMx ? kMxPageKeyBytes : kPageKeyBytes;
        constexpr int kPg = kMx ? kMxKeyPageBytes : kPageBytes;
        uint8_t* kd = smem + kOffKeys + s * kStage;
        uint8_t* sd = smem + kOffScale + x * kTileTok * 4;
        const uint32_t nv = (v0 ? 1u : 0u) + (v1 ? 1u : 0u);
        mbar_arrive_expect_tx(&full[s], nv * kHalf);
        mbar_arrive_expect_tx(&sc_full[x], nv * kPage * 4);
        // keys are read once: they leave L2 first, so that the scores the
        // epilogue writes stay there for the selection that reads them next
        // (a step at 1M tokens: 101 -> 92 us; an evict-last hint on the score
        // stores as well was slower at 256K)
        if (v0) {
          tma_load_3d(kd, &key_map, 0, 0, p0, &full[s], stream_policy);
          bulk_g2s_hint(sd, key_cache + (size_t)p0 * kPg + kHalf, kPage * 4, &sc_full[x],
                        stream_policy);
        }
        if (v1) {
          tma_load_3d(kd + kHalf, &key_map, 0, 0, p1, &full[s], stream_policy);
          bulk_g2s_hint(sd + kPage * 4, key_cache + (size_t)p1 * kPg + kHalf, kPage * 4,
                        &sc_full[x], stream_policy);
        }
      }
      __syncwarp();
      cur.next();
    }
    // no copy may still be landing in shared memory when the CTA exits
    for (int i = ntiles > kStages ? ntiles - kStages : 0; i < ntiles; ++i)
      if (i % kProdWarps == pw) warp_wait(&full[i % kStages], (uint32_t)(i / kStages) & 1, status);
    for (int i = ntiles > kScRing ? ntiles - kScRing : 0; i < ntiles; ++i)
      if (i % kProdWarps == pw) warp_wait(&sc_full[i % kScRing], (uint32_t)(i / kScRing) & 1, status);
  } else if (ntiles > 0 && warp >= kEpiWarp0) {
    // ---------------- epilogue: group eg takes the tiles i % 2 == eg; in it,
    // warp e takes token (32 x quarter + lane) of the tile and rows
    // kEpiRows * (e / 4) + [0, kEpiRows) of the group
    const int eg = (warp - kEpiWarp0) / kEpiWarpsPerGroup;
    const int e = (warp - kEpiWarp0) % kEpiWarpsPerGroup;
    const int quarter = warp & 3;
    const int r0 = (e >> 2) * kEpiRows;
    const int tok_in = quarter * 32 + lane;
    float* w_s = reinterpret_cast<float*>(smem + kOffW) + (warp - kEpiWarp0) * kEpiRows * kIdxHeads;
    int cur_group = -1;
    int len[kEpiRows];
    if (eg > 0) cur.advance(eg);
    constexpr int kDB = kMx ? kMxDBufs : kDBufs;
    for (int i = eg; i < ntiles; i += kEpiGroups) {
      const int x = i % kScRing, db = i % kDB;
      const int c = kMx ? i % kDBars : db;              // barrier pair of tile i
      const uint32_t par = kMx ? (uint32_t)(i / kDBars) & 1 : (uint32_t)(i / kDB) & 1;
      if (cur.g != cur_group) {                       // this warp's rows of the new group
        cur_group = cur.g;
#pragma unroll
        for (int rr = 0; rr < kEpiRows; ++rr) {
          const bool has = r0 + rr < cur.G.y;
          len[rr] = has ? row_len[cur.G.x + r0 + rr] : 0;
          w_s[rr * kIdxHeads + lane] = has ? ws.weff[(size_t)(cur.G.x + r0 + rr) * kIdxHeads + lane] : 0.f;
        }
        __syncwarp();
      }
      if (!warp_wait_spin(&d_full[c], par, status)) break;
      if (!warp_wait(&sc_full[x], (uint32_t)(i / kScRing) & 1, status)) break;
      tc_fence_after();
      const bool page_valid = (pv_s[x] >> (tok_in >> 6)) & 1u;
      const float ks = kMx ? 1.f : scale_s[x * kTileTok + tok_in];   // MXFP4: scaled in the MMA
      const int tok = cur.t * kTileTok + tok_in;
      // MXFP4: the accumulator and the scale slot are released as soon as
      // this warp's last tensor-memory load of the tile has completed, before
      // the last row's head sum and the score stores (256K: 155 -> 149 us);
      // the FP8 instance releases after its stores (the early release measured
      // 137.6 -> 144.0 us there)
      auto release = [&]() {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&d_empty[c]);
          mbar_arrive(&sc_empty[x]);
        }
      };
      const int nr = min(kEpiRows, cur.G.y - r0);       // this warp's rows in the group (warp-uniform)
      if (nr <= 0 && kMx) release();
#pragma unroll
      for (int rr = 0; rr < kEpiRows; ++rr) {
        const int r = r0 + rr;
        if (rr < nr) {
          uint32_t xv[32];
          const uint32_t ta = tmem_base + ((uint32_t)(quarter * 32) << 16) +
                              (uint32_t)(db * kDCols + r * kIdxHeads);
          tmem_ld_32x32b_x32(ta, xv);
          tmem_wait_ld();
          if (kMx && rr == nr - 1) release();
          const float4* wr = reinterpret_cast<const float4*>(w_s + rr * kIdxHeads);
          float acc[4] = {0.f, 0.f, 0.f, 0.f};          // four independent FMA chains
#pragma unroll
          for (int h4 = 0; h4 < kIdxHeads / 4; ++h4) {
            const float4 wv = wr[h4];
            const float w4[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
            for (int u = 0; u < 4; ++u)
              acc[u] = fmaf(w4[u], fmaxf(__uint_as_float(xv[4 * h4 + u]), 0.f), acc[u]);
          }
          const float sc = (acc[0] + acc[1]) + (acc[2] + acc[3]);
          if (page_valid && tok < len[rr])
            scores[(size_t)(cur.G.x + r) * ld + tok] = sc * ks;
        }
      }
      if (!kMx) release();
      cur.advance(kEpiGroups);
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

}  // namespace

size_t scan_scratch_bytes(int R) {
  return align_up((size_t)2 * R * kIdxHeads * kIdxDim) + align_up((size_t)R * kIdxHeads * 4) +
         align_up((size_t)R * 16) + align_up((size_t)(R + 1) * 4) + align_up(16) +
         align_up((size_t)kMaxScanCtas * 16);
}

cudaError_t launch_indexer_scan(const ScanArgs& a, cudaStream_t st) {
  if (a.R == 0) return cudaSuccess;
  const bool mx = a.q_dtype == kQMxfp4;
  const auto kernel = mx ? scan_kernel<true> : scan_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kSmemAlloc);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  ScanWs ws = scan_ws(a.scratch, a.R);
  // keys: [page][64 tokens][128 B] inside pages of 8448 bytes; a box is one
  // page's key block.  Queries: [2 terms x R x 32 rows][128 B]; a box is 128
  // rows (one term of a group of up to 4 rows; rows past the group are never
  // multiplied).  MXFP4: [page][64 tokens][64 B] inside pages of 4352 bytes
  // and the caller's [R x 32 rows][64 B] query codes, 64-byte swizzle.
  alignas(64) CUtensorMap kmap, qmap;
  const uint64_t row_bytes = mx ? kMxKeyBytes : kIdxDim;
  const uint64_t kdims[3] = {row_bytes, (uint64_t)kPage,
                             (uint64_t)(a.num_pages > 0 ? a.num_pages : 1)};
  const uint64_t kstr[2] = {row_bytes, (uint64_t)(mx ? kMxKeyPageBytes : kPageBytes)};
  const uint32_t kbox[3] = {(uint32_t)row_bytes, (uint32_t)kPage, 1};
  const int swz = mx ? 64 : 128;
  e = encode_tensor_map_u8(&kmap, 3, a.key_cache, kdims, kstr, kbox, swz);
  if (e != cudaSuccess) return e;
  const uint64_t qdims[2] = {row_bytes, (uint64_t)(mx ? 1 : 2) * a.R * kIdxHeads};
  const uint64_t qstr[1] = {row_bytes};
  const uint32_t qbox[2] = {(uint32_t)row_bytes, (uint32_t)(kMaxGroupRows * kIdxHeads)};
  e = encode_tensor_map_u8(&qmap, 2, mx ? a.q_idx : ws.q8, qdims, qstr, qbox, swz);
  if (e != cudaSuccess) return e;
  scan_prep_kernel<<<a.R + 1, kPrepThreads, 0, st>>>(a.q_idx, a.q_dtype, a.q_scale, a.q_sf, a.w,
                                             a.row_req, a.row_len, a.R, a.B, a.max_pages, sms,
                                             ws, a.status, a.clear_status ? 1 : 0);
  e = launch_kernel(kernel, dim3(sms), dim3(kThreads), kSmemAlloc, st, true, kmap, qmap,
                    a.key_cache, a.num_pages, a.block_table, a.max_pages, a.row_len, a.scores,
                    a.ld, a.R, a.q_dtype == DSA_E4M3 ? 1 : 2, ws, a.status);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace dsa
