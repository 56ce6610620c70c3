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
//  * Per 128-token tile the contraction is a real GEMM,
//      D[token, (row, head)] = K8[token, 0:128] . Q[(row, head), 0:128]^T,
//    M = 128 tokens, N = 32 x rows, K = 128: one tcgen05.mma kind::f16 chain
//    with the accumulator in tensor memory.  Keys are widened E4M3 -> f16 in
//    shared memory (exact: E4M3 is a subset of f16); the bf16 query is
//    rescaled per (row, head) by a power of two into f16 range (exact for all
//    but values 2^-22 below the head's absmax) and the inverse power of two is
//    folded into the head weight.  Accumulation is f32.
//  * Each TMEM lane holds one token's (row, head) logits, so the ReLU-weighted
//    head sum is a per-thread loop: no shuffles.
//  * Persistent CTAs, one per SM, each taking a contiguous run of (group, tile)
//    work items; warp roles: 0 MMA issuer and TMEM owner, 1-2 loaders, 3-10
//    converters, 11-14 epilogue (TMEM -> scores).
//  * The loaders stream the keys HBM -> shared staging with 16-byte cp.async
//    copies, kStages tiles ahead (64 KB in flight per SM; many small copies
//    sustain more bandwidth here than page-sized bulk copies issued by one
//    thread); the converters widen them to f16 and store the swizzled
//    tensor-core operand.
#include <limits.h>
#include <math.h>

#include "dsa_common.cuh"
#include "sm100_ptx.cuh"

namespace dsa {
namespace {

using namespace ptx;

constexpr int kTileTok = 128;
constexpr int kAtomBytes = kTileTok * 128;              // 128 rows x 128 B (64 f16 of K)
constexpr int kABytes = 2 * kAtomBytes;                 // K = 128 f16 = two atoms
constexpr int kABufs = 3;                               // f16 key tiles in flight to the MMA
constexpr int kMaxGroupRows = 4;
constexpr int kLoadWarps = 2;                           // warps 1-2
constexpr int kLoadThreads = 32 * kLoadWarps;
constexpr int kConvThreads = 256;                       // warps 3-10
constexpr int kChunks = kTileTok * 8 / kConvThreads;    // 16-byte key chunks per thread per tile
constexpr int kStages = 4;                              // tiles of keys in flight per SM
constexpr int kEpiWarp0 = 1 + kLoadWarps + kConvThreads / 32;   // warps 11-14
constexpr int kThreads = (kEpiWarp0 + 4) * 32;
constexpr int kDBufs = 4;                               // TMEM accumulators of 128 columns
constexpr uint32_t kTmemCols = 128 * kDBufs;

// shared-memory map (offsets from a 1024-byte aligned base)
constexpr int kOffA = 0;                                           // [kABufs] f16 key tiles
constexpr int kOffB = kABufs * kABytes;                            // up to 128 x 128 f16 query
constexpr int kOffW = kOffB + kABytes;                             // [4 warps][4 rows][32] f32
constexpr int kOffLen = kOffW + 4 * kMaxGroupRows * kIdxHeads * 4;  // [4 warps][4 rows]
constexpr int kRing = 8;                                           // scale ring slots
static_assert(kRing >= kABufs + kDBufs, "a scale slot is reused only after its epilogue finished");
constexpr int kOffScale = kOffLen + 4 * kMaxGroupRows * 4;          // [kRing][128] f32
constexpr int kOffValid = kOffScale + kRing * kTileTok * 4;         // [kRing] page-valid bits
constexpr int kOffStage = (kOffValid + kRing * 4 + 1023) / 1024 * 1024;  // [kStages] staging
constexpr int kStageKeyBytes = kTileTok * kIdxDim;                 // E4M3 keys, then 128 f32
constexpr int kStageBytes = kStageKeyBytes + kTileTok * 4 + 16;    // scales, then 2 page ids
constexpr int kOffBar = kOffStage + kStages * kStageBytes;
constexpr int kNumBars = 2 * kABufs + 2 * kDBufs + 2 + kRing + 2 * kStages;
constexpr int kOffTmem = kOffBar + kNumBars * 8;
constexpr int kSmemBytes = kOffTmem + 16;
constexpr int kSmemAlloc = kSmemBytes + 1024;

// group = {first row, rows, request, max row length}
struct ScanWs {
  __half* qh;      // [R][32][128] f16 query, rescaled per (row, head)
  float* weff;     // [R][32] head weight times the inverse rescale
  int4* groups;    // [R]
  int* gstart;     // [R + 1] first tile of each group
  int* meta;       // {groups, tiles}
};

ScanWs scan_ws(uint8_t* base, int R) {
  ScanWs w;
  size_t o = 0;
  w.qh = reinterpret_cast<__half*>(base + o);  o = align_up(o + (size_t)R * kIdxHeads * kIdxDim * 2);
  w.weff = reinterpret_cast<float*>(base + o); o = align_up(o + (size_t)R * kIdxHeads * 4);
  w.groups = reinterpret_cast<int4*>(base + o); o = align_up(o + (size_t)R * 16);
  w.gstart = reinterpret_cast<int*>(base + o);  o = align_up(o + (size_t)(R + 1) * 4);
  w.meta = reinterpret_cast<int*>(base + o);
  return w;
}

// ---------------------------------------------------------------------------
// Prep, one launch of R + 1 CTAs of 1024 threads.
//  * CTA r < R: warp h converts head h of row r's query to f16 (power-of-two
//    rescale per head, folded into the head weight).
//  * CTA R: groups the rows.  A run is a maximal block of adjacent valid rows
//    of one request; each run is cut into groups of up to 4 rows from its
//    start.  Block-wide scans over chunks of 1024 rows give every row its run
//    start, every group its index and every group its first tile.
constexpr int kPrepThreads = 1024;

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
                 const float* __restrict__ w, const int32_t* __restrict__ row_req,
                 const int32_t* __restrict__ row_len, int R, int B, int max_pages, ScanWs ws,
                 uint32_t* status) {
  if (blockIdx.x == (unsigned)R) {
    __shared__ int warp_buf[32];
    __shared__ int s_carry[3];   // run start of the last row, groups so far, tiles so far
    if (threadIdx.x == 0) { s_carry[0] = -1; s_carry[1] = 0; s_carry[2] = 0; }
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
    return;
  }
  // query conversion: warp h handles head h of row r, lane l dims [4l, 4l + 4)
  const int r = blockIdx.x;
  const int h = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t off = ((size_t)r * kIdxHeads + h) * kIdxDim + lane * 4;
  float x[4];
  if (q_dtype == DSA_E4M3) {
    const uint32_t v = *reinterpret_cast<const uint32_t*>(static_cast<const uint8_t*>(q_idx) + off);
    const float2 a = e4m3x2_to_float2((uint16_t)(v & 0xFFFF));
    const float2 b = e4m3x2_to_float2((uint16_t)(v >> 16));
    x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y;       // |x| <= 448: exact in f16
  } else {
    const uint2 v = *reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(q_idx) + off);
    x[0] = __uint_as_float(v.x << 16);
    x[1] = __uint_as_float(v.x & 0xFFFF0000u);
    x[2] = __uint_as_float(v.y << 16);
    x[3] = __uint_as_float(v.y & 0xFFFF0000u);
  }
  float wv = w[(size_t)r * kIdxHeads + h];
  if (q_dtype == DSA_E4M3) {
    wv *= q_scale[(size_t)r * kIdxHeads + h];
  } else {
    float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if (amax > 0.f) {
      const int e = ilogbf(amax);                 // amax in [2^e, 2^(e+1))
#pragma unroll
      for (int i = 0; i < 4; ++i) x[i] = ldexpf(x[i], 7 - e);   // absmax into [128, 256)
      wv = ldexpf(wv, e - 7);
    }
  }
  __half2 h01 = __floats2half2_rn(x[0], x[1]);
  __half2 h23 = __floats2half2_rn(x[2], x[3]);
  uint2 packed;
  packed.x = *reinterpret_cast<uint32_t*>(&h01);
  packed.y = *reinterpret_cast<uint32_t*>(&h23);
  *reinterpret_cast<uint2*>(ws.qh + off) = packed;
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

// ---- cp.async (global -> shared) with mbarrier completion -----------------
// A release-arrive on an mbarrier makes the arriving thread wait for its own
// outstanding copies and loads.  So the threads that fetch keys (loaders) never
// release-arrive: cp.async.mbarrier.arrive.noinc makes the barrier track the
// completion of the loader's copies without the loader waiting, and the
// converters, which release-arrive towards the MMA, have nothing in flight.
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}

__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}

// Arrive on `bar` once all cp.async copies issued so far by this thread landed.
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ bool page_ok(int p, int64_t num_pages) { return p >= 0 && p < num_pages; }

// 15 warps: one scheduler holds 4 of them, so 128 registers per thread is the cap.
__global__ void __launch_bounds__(kThreads, 1)
scan_tc_kernel(const uint8_t* __restrict__ key_cache, int64_t num_pages,
               const int32_t* __restrict__ block_table, int max_pages,
               const int32_t* __restrict__ row_len, float* __restrict__ scores, int64_t ld,
               ScanWs ws, uint32_t* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* a_full = bars;                          // [kABufs]
  uint64_t* a_empty = bars + kABufs;                // [kABufs]
  uint64_t* d_full = bars + 2 * kABufs;             // [kDBufs]
  uint64_t* d_empty = d_full + kDBufs;              // [kDBufs]
  uint64_t* b_full = d_full + 2 * kDBufs;
  uint64_t* b_empty = b_full + 1;
  uint64_t* sc_full = b_full + 2;                   // [kRing]
  uint64_t* st_full = sc_full + kRing;              // [kStages]
  uint64_t* st_empty = st_full + kStages;           // [kStages]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffTmem);
  float* w_s = reinterpret_cast<float*>(smem + kOffW);
  int* len_s = reinterpret_cast<int*>(smem + kOffLen);
  float* sc_ring = reinterpret_cast<float*>(smem + kOffScale);
  uint32_t* valid_ring = reinterpret_cast<uint32_t*>(smem + kOffValid);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int b = 0; b < kABufs; ++b) {
      mbar_init(&a_full[b], kConvThreads / 32);
      mbar_init(&a_empty[b], 1);
    }
    for (int b = 0; b < kDBufs; ++b) {
      mbar_init(&d_full[b], 1);
      mbar_init(&d_empty[b], 4);
    }
    mbar_init(b_full, kConvThreads / 32);
    mbar_init(b_empty, 1);
    for (int x = 0; x < kRing; ++x) mbar_init(&sc_full[x], kConvThreads / 32);
    for (int x = 0; x < kStages; ++x) {
      mbar_init(&st_full[x], kLoadThreads);      // one cp.async-tracked arrival per loader
      mbar_init(&st_empty[x], kConvThreads / 32);
    }
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

  const int ngroups = ws.meta[0];
  const int total = ws.meta[1];
  const int t_begin = (int)((int64_t)total * blockIdx.x / gridDim.x);
  const int t_end = (int)((int64_t)total * (blockIdx.x + 1) / gridDim.x);
  const int ntiles = t_end - t_begin;
  TileCursor cur;
  cur.groups = ws.groups;
  cur.gstart = ws.gstart;
  cur.ngroups = ngroups;
  if (ntiles > 0) cur.seek(t_begin);

  if (ntiles > 0 && warp == 0) {
    // ---------------- MMA issuer (lane 0 issues; the warp walks the same list)
    int cur_group = -1, gi = -1;
    uint32_t idesc = 0;
    int nrows = 1;
    for (int i = 0; i < ntiles; ++i) {
      if (cur.g != cur_group) {
        cur_group = cur.g;
        ++gi;
        nrows = cur.G.y;
        idesc = idesc_f16_f32(kTileTok, 32 * nrows);
        if (!warp_wait(b_full, (uint32_t)gi & 1, status)) break;
      }
      const int ab = i % kABufs;
      const int db = i % kDBufs;
      if (!warp_wait(&a_full[ab], (uint32_t)(i / kABufs) & 1, status)) break;
      if (!warp_wait(&d_empty[db], ((uint32_t)(i / kDBufs) & 1) ^ 1, status)) break;
      tc_fence_after();
      TileCursor nxt = cur;
      if (i + 1 < ntiles) nxt.next();
      if (lane == 0) {
        const uint32_t a_addr = smem_u32(smem + kOffA + ab * kABytes);
        const uint32_t b_addr = smem_u32(smem + kOffB);
        const uint32_t b_atom = (uint32_t)(32 * nrows) * 128;
        const uint32_t d_tmem = tmem_base + (uint32_t)db * 128;
#pragma unroll
        for (int j = 0; j < kIdxDim / 16; ++j) {
          const uint64_t ad = desc_kmajor_sw128(a_addr + (j >> 2) * kAtomBytes + (j & 3) * 32);
          const uint64_t bd = desc_kmajor_sw128(b_addr + (j >> 2) * b_atom + (j & 3) * 32);
          mma_f16_ss(d_tmem, ad, bd, idesc, j > 0 ? 1u : 0u);
        }
        mma_commit(&a_empty[ab]);
        mma_commit(&d_full[db]);
        if (i + 1 == ntiles || nxt.g != cur.g) mma_commit(b_empty);
      }
      __syncwarp();
      cur = nxt;
    }
  } else if (ntiles > 0 && warp >= 1 && warp < 1 + kLoadWarps) {
    // ---------------- loaders: keys, scales and page ids of tile i -> staging slot
    // i % kStages with cp.async.  Lane j looks up the pages of tile i0 + j, so a
    // batch of 32 tiles costs one block-table round trip.
    const int lt = tid - 32;                         // 0 .. kLoadThreads-1
    bool ok = true;
    for (int i0 = 0; i0 < ntiles && ok; i0 += 32) {
      int pg0 = -1, pg1 = -1, two = 0, bt_off = 0;
      if (i0 + lane < ntiles) {
        TileCursor c2 = cur;
        c2.seek(t_begin + i0 + lane);
        const int tok0 = c2.t * kTileTok;
        bt_off = c2.G.z * max_pages + tok0 / kPage;
        two = tok0 + kPage < c2.G.w;
        pg0 = __ldg(block_table + bt_off);
        if (two) pg1 = __ldg(block_table + bt_off + 1);
      }
      const int nb = min(32, ntiles - i0);
      for (int j = 0; j < nb; ++j) {
        const int i = i0 + j;
        const int slot = i % kStages;
        const int q0 = __shfl_sync(0xffffffffu, pg0, j);
        const int q1 = __shfl_sync(0xffffffffu, pg1, j);
        const int qtwo = __shfl_sync(0xffffffffu, two, j);
        const int qoff = __shfl_sync(0xffffffffu, bt_off, j);
        if (!warp_wait(&st_empty[slot], ((uint32_t)(i / kStages) & 1) ^ 1, status)) { ok = false; break; }
        const bool v0 = page_ok(q0, num_pages);
        const bool v1 = qtwo && page_ok(q1, num_pages);
        if (lt == 0 && (!v0 || (qtwo && !v1))) raise_dev(status, DSA_DEV_BAD_PAGE);
        uint8_t* stg = smem + kOffStage + slot * kStageBytes;
#pragma unroll
        for (int it = 0; it < kTileTok * 8 / kLoadThreads; ++it) {
          const int id = it * kLoadThreads + lt;
          const int r = id >> 3, c = id & 7;
          const bool second = r >= kPage;
          const int page = second ? q1 : q0;
          if (second ? v1 : v0)
            cp_async16(stg + r * kIdxDim + c * 16,
                       key_cache + (size_t)page * kKeyPageBytes + (r & 63) * kIdxDim + c * 16);
        }
        float* ssc = reinterpret_cast<float*>(stg + kStageKeyBytes);
#pragma unroll
        for (int x = lt; x < kTileTok; x += kLoadThreads) {
          const bool second = x >= kPage;
          if (second ? v1 : v0)
            cp_async4(ssc + x, key_cache + (size_t)(second ? q1 : q0) * kKeyPageBytes +
                                   kKeyScaleOffset + (x & 63) * 4);
        }
        if (lt == 0) {
          int* spid = reinterpret_cast<int*>(stg + kStageKeyBytes + kTileTok * 4);
          cp_async4(spid, block_table + qoff);
          if (qtwo) cp_async4(spid + 1, block_table + qoff + 1);
        }
        cp_async_arrive(&st_full[slot]);
      }
    }
  } else if (ntiles > 0 && warp >= 1 + kLoadWarps && warp < kEpiWarp0) {
    // ---------------- converters: staging slot -> f16 A tile (K-major, 128B swizzle)
    // + the tile's scales and page-valid bits for the epilogue
    const int ct = tid - 32 * (1 + kLoadWarps);
    int cur_group = -1, gi = -1;
    for (int i = 0; i < ntiles; ++i) {
      if (cur.g != cur_group) {
        cur_group = cur.g;
        ++gi;
        if (gi > 0 && !warp_wait(b_empty, (uint32_t)(gi - 1) & 1, status)) break;
        const int N = 32 * cur.G.y;
        const uint4* src =
            reinterpret_cast<const uint4*>(ws.qh + (size_t)cur.G.x * kIdxHeads * kIdxDim);
        uint8_t* bsm = smem + kOffB;
        for (int id = ct; id < N * 16; id += kConvThreads) {
          const int n = id >> 4, c = id & 15;
          const uint4 v = src[id];
          *reinterpret_cast<uint4*>(bsm + (c >> 3) * (N * 128) + n * 128 + (((c & 7) ^ (n & 7)) << 4)) = v;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(b_full);
      }
      const int slot = i % kStages;
      const int ab = i % kABufs;
      if (!warp_wait(&st_full[slot], (uint32_t)(i / kStages) & 1, status)) break;
      if (!warp_wait(&a_empty[ab], ((uint32_t)(i / kABufs) & 1) ^ 1, status)) break;
      const uint8_t* stg = smem + kOffStage + slot * kStageBytes;
      const int* spid = reinterpret_cast<const int*>(stg + kStageKeyBytes + kTileTok * 4);
      const bool two = cur.t * kTileTok + kPage < cur.G.w;
      const uint32_t vb = (page_ok(spid[0], num_pages) ? 1u : 0u) |
                          ((two && page_ok(spid[1], num_pages)) ? 2u : 0u);
      // scales: ring slot i % kRing is free: the MMA of tile i - kABufs has
      // completed (a_empty above), and it had waited for the epilogue of tile
      // i - kABufs - kDBufs to drain, which is at least kRing tiles back.
      const int rs = i % kRing;
      if (ct < kTileTok)
        sc_ring[rs * kTileTok + ct] =
            ((vb >> (ct >> 6)) & 1u) ? reinterpret_cast<const float*>(stg + kStageKeyBytes)[ct] : 0.f;
      if (ct == 0) valid_ring[rs] = vb;
      __syncwarp();
      if (lane == 0) mbar_arrive(&sc_full[rs]);
      uint8_t* a = smem + kOffA + ab * kABytes;
#pragma unroll
      for (int it = 0; it < kChunks; ++it) {
        const int r = it * (kConvThreads / 8) + (ct >> 3), c = ct & 7;
        const uint4 raw = *reinterpret_cast<const uint4*>(stg + r * kIdxDim + c * 16);
        uint4 lo, hi;
        cvt_e4m3x4_f16x4(raw.x, lo.x, lo.y);
        cvt_e4m3x4_f16x4(raw.y, lo.z, lo.w);
        cvt_e4m3x4_f16x4(raw.z, hi.x, hi.y);
        cvt_e4m3x4_f16x4(raw.w, hi.z, hi.w);
        uint8_t* row = a + (c >> 2) * kAtomBytes + r * 128;
        const int j0 = 2 * (c & 3);
        uint4* plo = reinterpret_cast<uint4*>(row + ((j0 ^ (r & 7)) << 4));
        uint4* phi = reinterpret_cast<uint4*>(row + (((j0 + 1) ^ (r & 7)) << 4));
        if (c < 4) { *plo = lo; *phi = hi; } else { *phi = hi; *plo = lo; }
      }
      fence_proxy_async_smem();
      __syncwarp();                                // the warp's writes are ordered before
      if (lane == 0) {                             // lane 0's release-arrivals
        mbar_arrive(&a_full[ab]);
        mbar_arrive(&st_empty[slot]);
      }
      cur.next();
    }
  } else if (ntiles > 0 && warp >= kEpiWarp0) {
    // ---------------- epilogue: TMEM -> ReLU-weighted head sum -> scores
    const int quarter = warp & 3;                 // TMEM lanes this warp may read
    float* wq = w_s + (warp - kEpiWarp0) * kMaxGroupRows * kIdxHeads;   // this warp's copy
    int* lq = len_s + (warp - kEpiWarp0) * kMaxGroupRows;
    int cur_group = -1;
    for (int i = 0; i < ntiles; ++i) {
      const int4 G = cur.G;
      if (cur.g != cur_group) {
        cur_group = cur.g;
        __syncwarp();
        for (int x = lane; x < G.y * kIdxHeads; x += 32) wq[x] = ws.weff[(size_t)G.x * kIdxHeads + x];
        if (lane < G.y) lq[lane] = row_len[G.x + lane];
        __syncwarp();
      }
      const int b = i % kDBufs;
      const int slot = i % kRing;
      if (!warp_wait(&sc_full[slot], (uint32_t)(i / kRing) & 1, status)) break;
      if (!warp_wait(&d_full[b], (uint32_t)(i / kDBufs) & 1, status)) break;
      tc_fence_after();
      const int tt = quarter * 32 + lane;             // token within the tile
      const int tok = cur.t * kTileTok + tt;
      const float ks = sc_ring[slot * kTileTok + tt];
      const bool valid = tok < G.w && ((valid_ring[slot] >> (tt >> 6)) & 1u);
      const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)b * 128;
#pragma unroll
      for (int p = 0; p < kMaxGroupRows; p += 2) {
        if (p < G.y) {
          uint32_t d[2][32];
          tmem_ld_32x32b_x32(taddr + (uint32_t)p * 32, d[0]);
          if (p + 1 < G.y) tmem_ld_32x32b_x32(taddr + (uint32_t)(p + 1) * 32, d[1]);
          tmem_wait_ld();
          if (p + 2 >= G.y) {                       // accumulator drained into registers
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&d_empty[b]);
          }
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const int nr = p + q;
            if (nr < G.y) {
              const float4* wr = reinterpret_cast<const float4*>(wq + nr * kIdxHeads);
              float acc = 0.f;
#pragma unroll
              for (int h4 = 0; h4 < 8; ++h4) {
                const float4 wv = wr[h4];
                acc = fmaf(wv.x, fmaxf(__uint_as_float(d[q][4 * h4 + 0]), 0.f), acc);
                acc = fmaf(wv.y, fmaxf(__uint_as_float(d[q][4 * h4 + 1]), 0.f), acc);
                acc = fmaf(wv.z, fmaxf(__uint_as_float(d[q][4 * h4 + 2]), 0.f), acc);
                acc = fmaf(wv.w, fmaxf(__uint_as_float(d[q][4 * h4 + 3]), 0.f), acc);
              }
              if (valid && tok < lq[nr]) scores[(size_t)(G.x + nr) * ld + tok] = acc * ks;
            }
          }
        }
      }
      cur.next();
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
  return align_up((size_t)R * kIdxHeads * kIdxDim * 2) + align_up((size_t)R * kIdxHeads * 4) +
         align_up((size_t)R * 16) + align_up((size_t)(R + 1) * 4) + align_up(16);
}

cudaError_t launch_indexer_scan(const ScanArgs& a, cudaStream_t st) {
  if (a.R == 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(scan_tc_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  ScanWs ws = scan_ws(a.scratch, a.R);
  scan_prep_kernel<<<a.R + 1, kPrepThreads, 0, st>>>(a.q_idx, a.q_dtype, a.q_scale, a.w, a.row_req,
                                             a.row_len, a.R, a.B, a.max_pages, ws, a.status);
  scan_tc_kernel<<<sms, kThreads, kSmemAlloc, st>>>(a.key_cache, a.num_pages, a.block_table,
                                                     a.max_pages, a.row_len, a.scores, a.ld, ws,
                                                     a.status);
  return cudaGetLastError();
}

}  // namespace dsa
