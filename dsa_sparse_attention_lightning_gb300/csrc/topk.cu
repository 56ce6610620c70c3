// topk.cu -- exact top-k selection per row (the Select step).
//
// Keeps the min(k, len) highest-scoring positions of each row, ties to the
// lower position (TokenSpeed post on Kimi K3.1 Pro, step 3 "Select": a radix
// top-k keeps the 2,048 highest-scoring positions for each query).  Scores are
// compared as order-preserving uint32 keys.  A row of at most 49,152 scores is
// selected by one CTA (topk_row_kernel, described where it is defined: the
// row in shared memory, the same sample threshold, the exact select over the
// candidates); longer rows take three launches:
//
//   1. sample   (one CTA per row): a fixed sample of the row (every sb-th
//               block of 32 scores, sb >= 16, at most 8192 scores) gives a
//               threshold tau low enough that the row should hold about
//               1.25 k + 16 sb keys >= tau: the key of the sample's rank-rho
//               element, rounded down to its 22-bit prefix (two radix digits
//               over the sample).
//   2. collect  (row x 2048-score chunk CTAs): every key >= tau is appended,
//               with its position, to the row's candidate list (one global
//               reservation per CTA, so each chunk's candidates form one run in
//               position order; the run's place is recorded); the count is
//               kept even past capacity.
//   3. finalize (one CTA per row): if the row holds at least k and at most
//               kTopkCandCap candidates, every one of the k best keys is a
//               candidate (count(key >= tau) >= k means tau <= the k-th key),
//               so an exact radix select over the candidates in shared memory
//               gives the k-th key T and how many keys equal to T to keep (the
//               lowest positions).  The kept candidates are written in
//               position order by ranking them within their chunk's run and
//               the runs in chunk order (scans, no sort).  Otherwise the same
//               exact select runs over the whole row in position order.
// The threshold only decides how much work the exact select does, never its
// result: the result is the exact top-k for any sample.
#include "dsa_common.cuh"

namespace dsa {
namespace {

constexpr int kSampleThreads = 1024;
constexpr int kCollectThreads = 256;
constexpr int kFinalThreads = 1024;
constexpr int kSampleStride = 16;              // one 32-score block in 16

// Inclusive block scan of one uint32 per thread (NT threads).
template <int NT>
__device__ __forceinline__ uint32_t block_inclusive_scan(uint32_t v, uint32_t* warp_sums) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    uint32_t n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) warp_sums[wid] = v;
  __syncthreads();
  if (wid == 0) {
    uint32_t s = lane < NT / 32 ? warp_sums[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      uint32_t n = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += n;
    }
    if (lane < NT / 32) warp_sums[lane] = s;
  }
  __syncthreads();
  const uint32_t add = wid > 0 ? warp_sums[wid - 1] : 0u;
  __syncthreads();  // warp_sums may be reused by the caller's next scan
  return v + add;
}

// Largest digit d with sum_{e >= d} hist[e] >= need, and above = sum_{e > d} hist[e].
// Requires 1 <= need <= sum(hist).  Called by all NT threads.
template <int NBINS, int NT>
__device__ __forceinline__ void find_threshold(const uint32_t* hist, uint32_t need,
                                               uint32_t* warp_sums, int* s_d, uint32_t* s_above) {
  constexpr int PER = NBINS / NT;
  static_assert(NBINS % NT == 0 && PER >= 1, "bins per thread");
  const int g = NT - 1 - (int)threadIdx.x;  // thread 0 owns the highest bins
  if (threadIdx.x == 0) {
    *s_d = 0;
    *s_above = 0;
  }
  uint32_t local = 0;
#pragma unroll
  for (int i = 0; i < PER; ++i) local += hist[g * PER + i];
  const uint32_t incl = block_inclusive_scan<NT>(local, warp_sums);
  const uint32_t excl = incl - local;
  if (excl < need && need <= incl) {
    uint32_t acc = excl;
    for (int b = g * PER + PER - 1; b >= g * PER; --b) {
      if (acc + hist[b] >= need) {
        *s_d = b;
        *s_above = acc;
        break;
      }
      acc += hist[b];
    }
  }
  __syncthreads();
}

__device__ __forceinline__ bool row_ok(int len, int64_t max_len) {
  return len >= 0 && (int64_t)len <= max_len;
}

// Shared-memory histogram add; all 32 lanes of the warp call it.  The keys of
// a row crowd into a few high-order bins, so the lanes that share the first
// valid lane's bin add once through it (two ballots and a shuffle, cheaper
// than a full match), and the others add one each.
__device__ __forceinline__ void hist_add(uint32_t* h, uint32_t bin, bool valid) {
  const unsigned vm = __ballot_sync(0xffffffffu, valid);
  if (vm == 0u) return;
  const int leader = __ffs(vm) - 1;
  const uint32_t lb = __shfl_sync(0xffffffffu, bin, leader);
  const unsigned same = __ballot_sync(0xffffffffu, valid && bin == lb);
  if ((int)(threadIdx.x & 31) == leader) atomicAdd(&h[lb], (uint32_t)__popc(same));
  else if (valid && bin != lb) atomicAdd(&h[bin], 1u);
}

// ---- 1. threshold from a fixed sample ----------------------------------------
// Every sb-th block of 32 scores, sb >= 16 chosen so that the sample holds at
// most kSampleBlocks blocks.
constexpr int kSampleBlocks = 256;

__device__ __forceinline__ int64_t sample_stride(int len) {
  const int64_t blocks = ((int64_t)len + 31) / 32;
  const int64_t sb = (blocks + kSampleBlocks - 1) / kSampleBlocks;
  return sb < kSampleStride ? kSampleStride : sb;
}

// Candidate threshold of a row from its fixed sample: the key of the
// sample's rank-rho element rounded down to its 22-bit prefix (0: take every
// key, when the sample holds fewer than rho keys).  Called by all
// kSampleThreads threads; every thread gets the result.  Thread t holds the
// sample elements e = u * kSampleThreads + t, u < kSamplePer, as key_of(u, pos).
constexpr int kSamplePer = kSampleBlocks * 32 / kSampleThreads;   // sample elements per thread

__device__ __forceinline__ int64_t sample_count(int len, int64_t sb) {
  return ((((int64_t)len + 31) / 32 + sb - 1) / sb) * 32;          // upper bound (ragged end)
}
__device__ __forceinline__ int64_t sample_pos(int64_t e, int64_t sb) {
  return (e / 32) * 32 * sb + (e % 32);
}

template <typename KeyOf>
__device__ uint32_t sample_threshold(KeyOf key_of, int len, int k, uint32_t* h, uint32_t* warp_sums,
                                     int* s_d, uint32_t* s_above, uint32_t* s_n) {
  const int64_t sb = sample_stride(len);
  const int64_t ns = sample_count(len, sb);
  // rank rho in the sample ~ 1.25 k / sb + 16 (about 1.25 k + 16 sb candidates in the row)
  const uint32_t rho = (uint32_t)((5 * (int64_t)k + 4 * sb - 1) / (4 * sb)) + 16;
  for (int i = threadIdx.x; i < kTopkBins1; i += kSampleThreads) h[i] = 0;
  if (threadIdx.x == 0) *s_n = 0;
  __syncthreads();
  uint32_t n_local = 0;
#pragma unroll
  for (int u = 0; u < kSamplePer; ++u) {                          // uniform trip count
    const int64_t e = (int64_t)u * kSampleThreads + threadIdx.x;
    const int64_t pos = sample_pos(e, sb);
    const bool v = e < ns && pos < len;
    const uint32_t key = v ? key_of(u, pos) : 0u;
    n_local += v ? 1u : 0u;
    hist_add(h, key >> 21, v);
  }
  atomicAdd(s_n, n_local);
  __syncthreads();
  if (*s_n < rho) {                            // short sample: take every key
    __syncthreads();                           // every thread has read s_n
    return 0u;
  }
  find_threshold<kTopkBins1, kSampleThreads>(h, rho, warp_sums, s_d, s_above);
  const uint32_t d1 = (uint32_t)*s_d;
  const uint32_t need = rho - *s_above;
  __syncthreads();
  for (int i = threadIdx.x; i < kTopkBins1; i += kSampleThreads) h[i] = 0;
  __syncthreads();
#pragma unroll
  for (int u = 0; u < kSamplePer; ++u) {
    const int64_t e = (int64_t)u * kSampleThreads + threadIdx.x;
    const int64_t pos = sample_pos(e, sb);
    const bool v = e < ns && pos < len;
    const uint32_t key = v ? key_of(u, pos) : 0u;
    hist_add(h, (key >> 10) & 0x7FF, v && (key >> 21) == d1);
  }
  __syncthreads();
  find_threshold<kTopkBins2, kSampleThreads>(h, need, warp_sums, s_d, s_above);
  const uint32_t t = (d1 << 21) | ((uint32_t)*s_d << 10);
  __syncthreads();                             // every thread has read s_d
  return t;
}

__global__ void __launch_bounds__(kSampleThreads)
topk_sample_kernel(const float* scores, int64_t ld, const int32_t* __restrict__ row_len,
                   int64_t max_len, int k, uint32_t* tau, uint32_t* cnt) {
  pdl_trigger();
  pdl_wait();                                  // the scores
  const int r = blockIdx.x;
  if (threadIdx.x == 0) cnt[r] = 0;            // the collect kernel's candidate count
  const int len = row_len[r];
  if (!row_ok(len, max_len) || len <= k) return;
  __shared__ uint32_t h[kTopkBins1];
  __shared__ uint32_t warp_sums[32];
  __shared__ int s_d;
  __shared__ uint32_t s_above, s_n;
  const float* row = scores + (size_t)r * ld;
  // every sample load is issued before the first is used: one memory round trip
  const int64_t sb = sample_stride(len);
  const int64_t ns = sample_count(len, sb);
  uint32_t sk[kSamplePer];
#pragma unroll
  for (int u = 0; u < kSamplePer; ++u) {
    const int64_t e = (int64_t)u * kSampleThreads + threadIdx.x;
    const int64_t pos = sample_pos(e, sb);
    sk[u] = (e < ns && pos < len) ? ordered_key(ld_dep(row + pos)) : 0u;
  }
  const uint32_t t = sample_threshold([&](int u, int64_t) { return sk[u]; }, len, k, h, warp_sums,
                                      &s_d, &s_above, &s_n);
  if (threadIdx.x == 0) tau[r] = t;
}

// ---- 2. candidates: every key >= tau -------------------------------------------
__global__ void __launch_bounds__(kCollectThreads)
topk_collect_kernel(const float* scores, int64_t ld, const int32_t* __restrict__ row_len,
                    int64_t max_len, int k, const uint32_t* tau, uint32_t* cnt, uint2* runs,
                    int nchunks, uint2* items) {
  pdl_trigger();
  pdl_wait();                                  // tau and the zeroed counts
  const int r = blockIdx.y;
  const int c = blockIdx.x;
  const int len = row_len[r];
  const uint32_t t = ld_dep(tau + r);            // issued with the row length: one round trip
  if (!row_ok(len, max_len) || len <= k) return;
  const int64_t s0 = (int64_t)c * kTopkChunk;
  if (s0 >= len) return;
  const int64_t s1 = min((int64_t)len, s0 + kTopkChunk);
  __shared__ uint32_t warp_sums[32];
  __shared__ uint32_t s_base;

  // each thread owns 16 consecutive positions
  constexpr int PER = kTopkChunk / kCollectThreads;
  const float* row = scores + (size_t)r * ld;
  const int64_t base = s0 + (int64_t)threadIdx.x * PER;
  uint32_t keys[PER];
#pragma unroll
  for (int i = 0; i < PER; i += 4) {
    float4 v;
    if (base + i + 4 <= s1) {
      v = ld_dep(reinterpret_cast<const float4*>(row + base + i));
    } else {
      v.x = base + i + 0 < s1 ? row[base + i + 0] : 0.f;
      v.y = base + i + 1 < s1 ? row[base + i + 1] : 0.f;
      v.z = base + i + 2 < s1 ? row[base + i + 2] : 0.f;
      v.w = base + i + 3 < s1 ? row[base + i + 3] : 0.f;
    }
    keys[i + 0] = ordered_key(v.x);
    keys[i + 1] = ordered_key(v.y);
    keys[i + 2] = ordered_key(v.z);
    keys[i + 3] = ordered_key(v.w);
  }
  uint32_t n = 0;
#pragma unroll
  for (int i = 0; i < PER; ++i) n += (base + i < s1 && keys[i] >= t) ? 1u : 0u;
  const uint32_t incl = block_inclusive_scan<kCollectThreads>(n, warp_sums);
  if (threadIdx.x == kCollectThreads - 1) {
    s_base = incl ? atomicAdd(&cnt[r], incl) : 0u;
    runs[(size_t)r * nchunks + c] = make_uint2(s_base, incl);   // this chunk's run in the list
  }
  __syncthreads();
  uint32_t pos = s_base + incl - n;
  uint2* seg = items + (size_t)r * kTopkCandCap;
#pragma unroll
  for (int i = 0; i < PER; ++i)
    if (base + i < s1 && keys[i] >= t) {
      if (pos < (uint32_t)kTopkCandCap) seg[pos] = make_uint2(keys[i], (uint32_t)(base + i));
      ++pos;
    }
}

// ---- 3. exact select ----------------------------------------------------------
struct SelectSmem {
  uint32_t h[kTopkBins1];
  uint32_t warp_sums[32];
  int d;
  uint32_t above, acc[2];
};

// k-th key T of `total` keys key_at(i) and how many keys equal to T to keep:
// three radix digits of 11, 11 and 10 bits.  n_eq = keys equal to T.
template <typename KeyAt>
__device__ void kth_key(KeyAt key_at, uint32_t total, int k, SelectSmem& S, uint32_t& T,
                        uint32_t& need_eq, uint32_t& n_eq) {
  uint32_t need = (uint32_t)k;
  uint32_t prefix = 0;                         // key bits fixed so far
  int shift = 32;
  for (int dgt = 0; dgt < 3; ++dgt) {
    const int w = dgt < 2 ? 11 : 10;
    shift -= w;
    for (int i = threadIdx.x; i < kTopkBins1; i += kFinalThreads) S.h[i] = 0;
    __syncthreads();
    const int pshift = shift + w;              // bits above this digit
    for (uint32_t b = 0; b < total; b += kFinalThreads) {
      const uint32_t i = b + threadIdx.x;
      const uint32_t key = i < total ? key_at(i) : 0u;
      const bool v = i < total && (dgt == 0 || (key >> pshift) == prefix);
      hist_add(S.h, (key >> shift) & ((1u << w) - 1u), v);
    }
    __syncthreads();
    if (w == 11) find_threshold<kTopkBins1, kFinalThreads>(S.h, need, S.warp_sums, &S.d, &S.above);
    else find_threshold<kTopkBins3, kFinalThreads>(S.h, need, S.warp_sums, &S.d, &S.above);
    prefix = (prefix << w) | (uint32_t)S.d;
    need -= S.above;
  }
  T = prefix;
  need_eq = need;
  n_eq = S.h[S.d];
  __syncthreads();
}

// Exclusive scan of PER flags per thread (consecutive elements) into ex[];
// returns the total.  All threads call it.
template <int PER>
__device__ __forceinline__ uint32_t scan_flags(const uint8_t (&f)[PER], uint16_t* ex, uint32_t n,
                                               SelectSmem& S) {
  uint32_t local = 0;
#pragma unroll
  for (int u = 0; u < PER; ++u) local += f[u];
  const uint32_t incl = block_inclusive_scan<kFinalThreads>(local, S.warp_sums);
  uint32_t run = incl - local;
  const uint32_t i0 = threadIdx.x * PER;
#pragma unroll
  for (int u = 0; u < PER; ++u) {
    if (i0 + u <= n) ex[i0 + u] = (uint16_t)run;   // ex[n] = total (run end lookups)
    run += f[u];
  }
  if (threadIdx.x == kFinalThreads - 1) S.acc[0] = incl;
  __syncthreads();
  const uint32_t total = S.acc[0];
  if (threadIdx.x == 0) ex[n] = (uint16_t)total;
  __syncthreads();
  return total;
}

// Exclusive scan over chunks (in chunk order) of the counts cnt_of(c) -> base[c].
template <typename CntOf>
__device__ __forceinline__ void scan_chunks(CntOf cnt_of, int nch, uint32_t* base, SelectSmem& S) {
  uint32_t carry = 0;
  for (int c0 = 0; c0 < nch; c0 += kFinalThreads) {
    const int c = c0 + threadIdx.x;
    const uint32_t v = c < nch ? cnt_of(c) : 0u;
    const uint32_t incl = block_inclusive_scan<kFinalThreads>(v, S.warp_sums);
    if (c < nch) base[c] = carry + incl - v;
    if (threadIdx.x == kFinalThreads - 1) S.acc[1] = incl;
    __syncthreads();
    carry += S.acc[1];
    __syncthreads();
  }
}

constexpr int kCandPer = kTopkCandCap / kFinalThreads;     // candidates per thread
constexpr int kMaxRunChunks = 4096;                       // chunk table held in shared memory

struct CandSmem {
  uint2 cand[kTopkCandCap];
  uint2 run[kMaxRunChunks];                     // each chunk's {start, count} in the list
  uint16_t ex_tie[kTopkCandCap + kFinalThreads];
  uint16_t ex_sel[kTopkCandCap + kFinalThreads];
  uint32_t base_tie[kMaxRunChunks];
  uint32_t base_sel[kMaxRunChunks];
};

__global__ void __launch_bounds__(kFinalThreads, 1)
topk_finalize_kernel(const float* scores, int64_t ld, const int32_t* __restrict__ row_len,
                     int64_t max_len, int k, const uint32_t* cnt, const uint2* runs,
                     int nchunks, const uint2* items, int32_t* __restrict__ idx,
                     uint32_t* status) {
  extern __shared__ __align__(16) uint8_t fin_smem[];
  SelectSmem& S = *reinterpret_cast<SelectSmem*>(fin_smem);
  CandSmem& C = *reinterpret_cast<CandSmem*>(fin_smem + (sizeof(SelectSmem) + 15) / 16 * 16);
  pdl_trigger();
  pdl_wait();                                  // the candidate lists
  const int r = blockIdx.x;
  const int len = row_len[r];
  const uint32_t n = ld_dep(cnt + r);            // issued with the row length: one round trip
  int32_t* out = idx + (size_t)r * k;
  if (!row_ok(len, max_len)) {
    if (threadIdx.x == 0) raise_dev(status, DSA_DEV_BAD_ROW);
    for (int j = threadIdx.x; j < k; j += kFinalThreads) out[j] = -1;
    return;
  }
  if (len <= k) {
    for (int j = threadIdx.x; j < k; j += kFinalThreads) out[j] = j < len ? j : -1;
    return;
  }
  const int nch = (int)((len + kTopkChunk - 1) / kTopkChunk);
  uint32_t T, need_eq, n_eq;
  if (n >= (uint32_t)k && n <= (uint32_t)kTopkCandCap && nch <= kMaxRunChunks) {
    // ---- candidates in shared memory, ranked by position through their runs
    // every candidate load is issued before the first store: one memory round trip
    const uint2* src = items + (size_t)r * kTopkCandCap;
    const uint2* runs_r = runs + (size_t)r * nchunks;
    uint2 cv[kCandPer];
    uint2 rv[kMaxRunChunks / kFinalThreads];
#pragma unroll
    for (int u = 0; u < kCandPer; ++u) {
      const uint32_t i = (uint32_t)u * kFinalThreads + threadIdx.x;
      cv[u] = i < n ? ld_dep(src + i) : make_uint2(0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < kMaxRunChunks / kFinalThreads; ++u) {
      const int ch = u * kFinalThreads + (int)threadIdx.x;
      rv[u] = ch < nch ? ld_dep(runs_r + ch) : make_uint2(0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < kCandPer; ++u) {
      const uint32_t i = (uint32_t)u * kFinalThreads + threadIdx.x;
      if (i < n) C.cand[i] = cv[u];
    }
#pragma unroll
    for (int u = 0; u < kMaxRunChunks / kFinalThreads; ++u) {
      const int ch = u * kFinalThreads + (int)threadIdx.x;
      if (ch < nch) C.run[ch] = rv[u];
    }
    __syncthreads();
    kth_key([&](uint32_t i) { return C.cand[i].x; }, n, k, S, T, need_eq, n_eq);
    const uint2* rr = C.run;
    const uint32_t i0 = threadIdx.x * kCandPer;
    uint8_t f[kCandPer];
    const bool all_ties = need_eq == n_eq;           // every key equal to T is kept
    if (!all_ties) {
      // ties: rank by position = ties in earlier chunks + ties earlier in the run
#pragma unroll
      for (int u = 0; u < kCandPer; ++u) f[u] = (i0 + u < n && C.cand[i0 + u].x == T) ? 1 : 0;
      scan_flags(f, C.ex_tie, n, S);
      scan_chunks([&](int c) { const uint2 q = rr[c]; return (uint32_t)(C.ex_tie[q.x + q.y] - C.ex_tie[q.x]); },
                  nch, C.base_tie, S);
    }
    // kept: key > T, or a tie of rank < need_eq
#pragma unroll
    for (int u = 0; u < kCandPer; ++u) {
      const uint32_t i = i0 + u;
      uint8_t keep = 0;
      if (i < n) {
        const uint2 v = C.cand[i];
        if (v.x > T || (all_ties && v.x == T)) {
          keep = 1;
        } else if (v.x == T) {
          const uint2 q = rr[v.y / kTopkChunk];
          keep = (C.base_tie[v.y / kTopkChunk] + C.ex_tie[i] - C.ex_tie[q.x]) < need_eq ? 1 : 0;
        }
      }
      f[u] = keep;
    }
    scan_flags(f, C.ex_sel, n, S);
    scan_chunks([&](int c) { const uint2 q = rr[c]; return (uint32_t)(C.ex_sel[q.x + q.y] - C.ex_sel[q.x]); },
                nch, C.base_sel, S);
#pragma unroll
    for (int u = 0; u < kCandPer; ++u) {
      if (!f[u]) continue;
      const uint2 v = C.cand[i0 + u];
      const int c = (int)(v.y / kTopkChunk);
      const uint32_t o = C.base_sel[c] + C.ex_sel[i0 + u] - C.ex_sel[rr[c].x];
      if (o < (uint32_t)k) out[o] = (int32_t)v.y;
    }
  } else {
    // ---- the whole row, in position order
    const float* row = scores + (size_t)r * ld;
    kth_key([&](uint32_t i) { return ordered_key(row[i]); }, (uint32_t)len, k, S, T, need_eq, n_eq);
    uint32_t out_count = 0, eq_seen = 0;
    for (uint32_t b = 0; b < (uint32_t)len; b += kFinalThreads) {
      const uint32_t i = b + threadIdx.x;
      const uint32_t key = i < (uint32_t)len ? ordered_key(row[i]) : 0u;
      const uint32_t is_eq = (i < (uint32_t)len && key == T) ? 1u : 0u;
      const uint32_t eq_incl = block_inclusive_scan<kFinalThreads>(is_eq, S.warp_sums);
      const bool take_eq = is_eq && (eq_seen + eq_incl - 1u) < need_eq;
      const uint32_t sel = ((i < (uint32_t)len && key > T) || take_eq) ? 1u : 0u;
      const uint32_t sel_incl = block_inclusive_scan<kFinalThreads>(sel, S.warp_sums);
      const uint32_t pos = out_count + sel_incl - 1u;
      if (sel && pos < (uint32_t)k) out[pos] = (int32_t)i;
      if (threadIdx.x == kFinalThreads - 1) {
        S.acc[0] = sel_incl;
        S.acc[1] = eq_incl;
      }
      __syncthreads();
      out_count += S.acc[0];
      eq_seen += S.acc[1];
      __syncthreads();
    }
  }
}

// ---- one CTA per row: rows that fit in shared memory ---------------------------
// The row's keys are loaded once into shared memory (every load issued before
// the first is used: one memory round trip).  The fixed sample of the
// multi-launch path sets a candidate threshold tau; warp w owns a contiguous
// segment of the row, counts its keys >= tau with ballots, and a 32-entry
// scan places each warp's candidates, so the candidate positions land in
// shared memory in position order.  If there are at least k and at most
// kRowCand of them, the exact select runs over the candidates, else over the
// whole row (the result is the same; only the work differs).  The kept
// positions are then written in position order: over the items in order,
//   slot = #(key > T before it) + min(#(key == T before it), need_eq),
// a tie being kept when #(key == T before it) < need_eq.
constexpr int kRowCap = 49152;                 // scores of a row held in shared memory
constexpr int kRowCand = 6144;                 // candidate positions held in shared memory
static_assert(kRowCap % (4 * kFinalThreads) == 0, "whole vectors per thread");

size_t row_smem_bytes() {
  return (sizeof(SelectSmem) + 15) / 16 * 16 + (size_t)(kRowCap + kRowCand) * 4;
}

// Exclusive count before this warp and total over the block of c (one value
// per warp, in s[32]); all threads call it after s is filled and synced.
__device__ __forceinline__ uint32_t warp_prefix(const uint32_t* s, uint32_t* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const uint32_t x = s[lane];
  uint32_t before = lane < wid ? x : 0u, all = x;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    before += __shfl_xor_sync(0xffffffffu, before, o);
    all += __shfl_xor_sync(0xffffffffu, all, o);
  }
  *total = all;
  return before;
}

// Writes the kept items (key > T, or == T within the first need_eq ties) of
// the n items, in item order, as positions pos_at(i) to out[0, k).
template <typename PosAt>
__device__ __forceinline__ void write_selected(const uint32_t* keys, PosAt pos_at, int n, uint32_t T,
                                               uint32_t need_eq, int k, int32_t* out,
                                               uint32_t* s_gt, uint32_t* s_eq) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int seg = (n + kFinalThreads - 1) / kFinalThreads * 32;    // multiple of 32
  const int i_begin = wid * seg, i_end = min(n, i_begin + seg);
  uint32_t cg = 0, ce = 0;
  for (int i0 = i_begin; i0 < i_end; i0 += 32) {
    const int i = i0 + lane;
    const uint32_t key = i < i_end ? keys[pos_at(i)] : 0u;
    cg += __popc(__ballot_sync(0xffffffffu, i < i_end && key > T));
    ce += __popc(__ballot_sync(0xffffffffu, i < i_end && key == T));
  }
  if (lane == 0) {
    s_gt[wid] = cg;
    s_eq[wid] = ce;
  }
  __syncthreads();
  uint32_t tot;
  uint32_t bg = warp_prefix(s_gt, &tot), be = warp_prefix(s_eq, &tot);
  const uint32_t lt = (1u << lane) - 1u;
  for (int i0 = i_begin; i0 < i_end; i0 += 32) {
    const int i = i0 + lane;
    const int p = i < i_end ? pos_at(i) : 0;
    const uint32_t key = i < i_end ? keys[p] : 0u;
    const bool gt = i < i_end && key > T, eq = i < i_end && key == T;
    const unsigned mg = __ballot_sync(0xffffffffu, gt), me = __ballot_sync(0xffffffffu, eq);
    const uint32_t eq_before = be + __popc(me & lt);
    const uint32_t slot = bg + __popc(mg & lt) + min(eq_before, need_eq);
    if ((gt || (eq && eq_before < need_eq)) && slot < (uint32_t)k) out[slot] = p;
    bg += __popc(mg);
    be += __popc(me);
  }
}

__global__ void __launch_bounds__(kFinalThreads, 1)
topk_row_kernel(const float* scores, int64_t ld, const int32_t* __restrict__ row_len,
                int64_t max_len, int k, int32_t* __restrict__ idx, uint32_t* status) {
  static_assert(kFinalThreads == kSampleThreads, "the sample threshold runs on this block");
  extern __shared__ __align__(16) uint8_t row_smem[];
  SelectSmem& S = *reinterpret_cast<SelectSmem*>(row_smem);
  uint32_t* keys = reinterpret_cast<uint32_t*>(row_smem + (sizeof(SelectSmem) + 15) / 16 * 16);
  uint32_t* cand = keys + kRowCap;
  __shared__ uint32_t s_gt[32], s_eq[32], s_cnt[32];
  pdl_trigger();
  pdl_wait();                                  // the scores
  const int r = blockIdx.x;
  const int len = row_len[r];
  int32_t* out = idx + (size_t)r * k;
  if (!row_ok(len, max_len) || len > kRowCap) {
    if (threadIdx.x == 0) raise_dev(status, DSA_DEV_BAD_ROW);
    for (int j = threadIdx.x; j < k; j += kFinalThreads) out[j] = -1;
    return;
  }
  if (len <= k) {
    for (int j = threadIdx.x; j < k; j += kFinalThreads) out[j] = j < len ? j : -1;
    return;
  }
  // load (16-byte vectors; the row is 16-byte aligned and holds ld >= 4 ceil(len / 4) floats)
  const float* row = scores + (size_t)r * ld;
  const int n4 = (len + 3) >> 2;
  constexpr int kVecPer = kRowCap / 4 / kFinalThreads;
  float4 v[kVecPer];
#pragma unroll
  for (int u = 0; u < kVecPer; ++u) {
    const int g = u * kFinalThreads + (int)threadIdx.x;
    v[u] = g < n4 ? ld_dep(reinterpret_cast<const float4*>(row) + g) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int u = 0; u < kVecPer; ++u) {
    const int g = u * kFinalThreads + (int)threadIdx.x;
    if (g < n4)
      *reinterpret_cast<uint4*>(keys + 4 * g) = make_uint4(
          ordered_key(v[u].x), ordered_key(v[u].y), ordered_key(v[u].z), ordered_key(v[u].w));
  }
  __syncthreads();
  const uint32_t tau = sample_threshold([&](int, int64_t p) { return keys[p]; }, len, k, S.h,
                                        S.warp_sums, &S.d, &S.above, &S.acc[0]);
  // candidates: keys >= tau, counted per warp segment, then placed in position order
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int seg = (len + kFinalThreads - 1) / kFinalThreads * 32;
  const int p_begin = wid * seg, p_end = min(len, p_begin + seg);
  uint32_t c = 0;
  for (int p0 = p_begin; p0 < p_end; p0 += 32) {
    const int p = p0 + lane;
    c += __popc(__ballot_sync(0xffffffffu, p < p_end && keys[p] >= tau));
  }
  if (lane == 0) s_cnt[wid] = c;
  __syncthreads();
  uint32_t n;
  uint32_t base = warp_prefix(s_cnt, &n);
  uint32_t T, need_eq, n_eq;
  if (n >= (uint32_t)k && n <= (uint32_t)kRowCand) {            // uniform
    const uint32_t lt = (1u << lane) - 1u;
    for (int p0 = p_begin; p0 < p_end; p0 += 32) {
      const int p = p0 + lane;
      const bool c1 = p < p_end && keys[p] >= tau;
      const unsigned m = __ballot_sync(0xffffffffu, c1);
      if (c1) cand[base + __popc(m & lt)] = (uint32_t)p;
      base += __popc(m);
    }
    __syncthreads();
    kth_key([&](uint32_t i) { return keys[cand[i]]; }, n, k, S, T, need_eq, n_eq);
    write_selected(keys, [&](int i) { return (int)cand[i]; }, (int)n, T, need_eq, k, out, s_gt,
                   s_eq);
  } else {
    kth_key([&](uint32_t i) { return keys[i]; }, (uint32_t)len, k, S, T, need_eq, n_eq);
    write_selected(keys, [](int i) { return i; }, len, T, need_eq, k, out, s_gt, s_eq);
  }
}

}  // namespace

cudaError_t launch_topk(const TopkArgs& a, cudaStream_t st) {
  if (a.R == 0) return cudaSuccess;
  if (a.max_len <= kRowCap && (reinterpret_cast<uintptr_t>(a.scores) & 15) == 0 && a.ld % 4 == 0) {
    cudaError_t e = cudaFuncSetAttribute(topk_row_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)row_smem_bytes());
    if (e != cudaSuccess) return e;
    e = launch_kernel(topk_row_kernel, dim3(a.R), dim3(kFinalThreads), row_smem_bytes(), st,
                      a.chained, a.scores, a.ld, a.row_len, a.max_len, a.k, a.idx, a.status);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
  }
  const TopkLayout L(a.R, a.max_len);
  uint32_t* tau = reinterpret_cast<uint32_t*>(a.scratch + L.tau);
  uint32_t* cnt = reinterpret_cast<uint32_t*>(a.scratch + L.cnt);
  uint2* runs = reinterpret_cast<uint2*>(a.scratch + L.runs);
  uint2* items = reinterpret_cast<uint2*>(a.scratch + L.items);
  const size_t smem = (sizeof(SelectSmem) + 15) / 16 * 16 + sizeof(CandSmem);
  cudaError_t e = cudaFuncSetAttribute(topk_finalize_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  e = launch_kernel(topk_sample_kernel, dim3(a.R), dim3(kSampleThreads), 0, st, a.chained,
                    a.scores, a.ld, a.row_len, a.max_len, a.k, tau, cnt);
  if (e != cudaSuccess) return e;
  e = launch_kernel(topk_collect_kernel, dim3(L.nchunks, a.R), dim3(kCollectThreads), 0, st, true,
                    a.scores, a.ld, a.row_len, a.max_len, a.k, (const uint32_t*)tau, cnt, runs,
                    L.nchunks, items);
  if (e != cudaSuccess) return e;
  e = launch_kernel(topk_finalize_kernel, dim3(a.R), dim3(kFinalThreads), smem, st, true,
                    a.scores, a.ld, a.row_len, a.max_len, a.k, (const uint32_t*)cnt,
                    (const uint2*)runs, L.nchunks, (const uint2*)items, a.idx, a.status);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace dsa
