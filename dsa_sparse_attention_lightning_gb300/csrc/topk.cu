// topk.cu -- exact top-k selection per row (the Select step).
//
// Keeps the min(k, len) highest-scoring positions of each row, ties to the
// lower position (TokenSpeed post on Kimi K3.1 Pro, step 3 "Select": a radix
// top-k keeps the 2,048 highest-scoring positions for each query).  Like the
// pages' multi-workgroup design ("Reducing indexer overhead on AMD MI350X":
// each row is spread over many workgroups that share a histogram of score
// prefixes), one long row is spread over many CTAs:
//
//   1. hist     (row x 4096-score chunk CTAs): histogram of the top 11 bits of
//               the order-preserving uint32 key of every score.
//   2. collect  (row x chunk CTAs): every CTA finds the threshold digit D1 (the
//               digit holding the k-th best key) from the shared histogram and
//               copies, in position order, the (key, position) pairs whose
//               digit is >= D1 into the chunk's own segment.
//   3. finalize (one CTA per row): two more radix digits over the collected
//               candidates give the exact k-th key T and how many keys equal
//               to T are needed; an ordered pass over the segments emits every
//               key > T and the first `need` keys == T, so ties go to the
//               lower position and idx comes out in ascending order.
#include "dsa_common.cuh"

namespace dsa {
namespace {

constexpr int kHistThreads = 512;
constexpr int kCollectThreads = 256;
constexpr int kFinalThreads = 1024;

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

// ---- 1. histogram of the top digit ---------------------------------------
__global__ void __launch_bounds__(kHistThreads)
topk_hist_kernel(const float* __restrict__ scores, int64_t ld, const int32_t* __restrict__ row_len,
                 int64_t max_len, int k, uint32_t* __restrict__ hist) {
  const int r = blockIdx.y;
  const int len = row_len[r];
  if (!row_ok(len, max_len) || len <= k) return;
  const int64_t s0 = (int64_t)blockIdx.x * kTopkChunk;
  if (s0 >= len) return;
  const int64_t s1 = min((int64_t)len, s0 + kTopkChunk);
  __shared__ uint32_t h[kTopkBins1];
  for (int i = threadIdx.x; i < kTopkBins1; i += kHistThreads) h[i] = 0;
  __syncthreads();
  const float* row = scores + (size_t)r * ld;
  for (int64_t s = s0 + threadIdx.x * 4; s < s1; s += kHistThreads * 4) {
    if (s + 4 <= s1) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(row + s));
      atomicAdd(&h[ordered_key(v.x) >> 21], 1u);
      atomicAdd(&h[ordered_key(v.y) >> 21], 1u);
      atomicAdd(&h[ordered_key(v.z) >> 21], 1u);
      atomicAdd(&h[ordered_key(v.w) >> 21], 1u);
    } else {
      for (int64_t t = s; t < s1; ++t) atomicAdd(&h[ordered_key(row[t]) >> 21], 1u);
    }
  }
  __syncthreads();
  uint32_t* gh = hist + (size_t)r * kTopkBins1;
  for (int i = threadIdx.x; i < kTopkBins1; i += kHistThreads)
    if (h[i]) atomicAdd(&gh[i], h[i]);
}

// ---- 2. ordered collection of digit >= D1 ------------------------------------
__global__ void __launch_bounds__(kCollectThreads)
topk_collect_kernel(const float* __restrict__ scores, int64_t ld,
                    const int32_t* __restrict__ row_len, int64_t max_len, int k,
                    const uint32_t* __restrict__ hist, uint2* __restrict__ thr,
                    uint32_t* __restrict__ seg_count, uint2* __restrict__ items, int nchunks) {
  const int r = blockIdx.y;
  const int c = blockIdx.x;
  const int len = row_len[r];
  if (!row_ok(len, max_len) || len <= k) return;
  const int64_t s0 = (int64_t)c * kTopkChunk;
  if (s0 >= len) return;
  const int64_t s1 = min((int64_t)len, s0 + kTopkChunk);

  __shared__ uint32_t h[kTopkBins1];
  __shared__ uint32_t warp_sums[32];
  __shared__ int s_d;
  __shared__ uint32_t s_above;
  for (int i = threadIdx.x; i < kTopkBins1; i += kCollectThreads)
    h[i] = hist[(size_t)r * kTopkBins1 + i];
  __syncthreads();
  find_threshold<kTopkBins1, kCollectThreads>(h, (uint32_t)k, warp_sums, &s_d, &s_above);
  const uint32_t d1 = (uint32_t)s_d;
  if (c == 0 && threadIdx.x == 0) thr[r] = make_uint2(d1, s_above);

  // each thread owns 16 consecutive positions: keeps the chunk's order
  constexpr int PER = kTopkChunk / kCollectThreads;
  const float* row = scores + (size_t)r * ld;
  const int64_t base = s0 + (int64_t)threadIdx.x * PER;
  uint32_t keys[PER];
  uint32_t cnt = 0;
#pragma unroll
  for (int i = 0; i < PER; i += 4) {
    float4 v;
    if (base + i + 4 <= s1) {
      v = __ldg(reinterpret_cast<const float4*>(row + base + i));
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
#pragma unroll
  for (int i = 0; i < PER; ++i) cnt += (base + i < s1 && (keys[i] >> 21) >= d1) ? 1u : 0u;
  const uint32_t incl = block_inclusive_scan<kCollectThreads>(cnt, warp_sums);
  uint32_t pos = incl - cnt;
  uint2* seg = items + ((size_t)r * nchunks + c) * kTopkChunk;
#pragma unroll
  for (int i = 0; i < PER; ++i)
    if (base + i < s1 && (keys[i] >> 21) >= d1) seg[pos++] = make_uint2(keys[i], (uint32_t)(base + i));
  if (threadIdx.x == kCollectThreads - 1) seg_count[(size_t)r * nchunks + c] = incl;
}

// ---- 3. exact threshold and ordered emission (one CTA per row) -------------
__device__ __forceinline__ uint2 item_at(const uint2* seg_base, const uint32_t* prefix, int nch,
                                         uint32_t i) {
  // chunk c holds flattened items [prefix[c], prefix[c+1])
  int lo = 0, hi = nch;  // find last c with prefix[c] <= i
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid] <= i) lo = mid; else hi = mid;
  }
  return seg_base[(size_t)lo * kTopkChunk + (i - prefix[lo])];
}

__global__ void __launch_bounds__(kFinalThreads)
topk_finalize_kernel(const int32_t* __restrict__ row_len, int64_t max_len, int k,
                     const uint2* __restrict__ thr, const uint32_t* __restrict__ seg_count,
                     const uint2* __restrict__ items, int nchunks, int32_t* __restrict__ idx,
                     uint32_t* status) {
  extern __shared__ uint32_t prefix[];  // nchunks + 1
  __shared__ uint32_t h[kTopkBins2];
  __shared__ uint32_t warp_sums[32];
  __shared__ int s_d;
  __shared__ uint32_t s_above;
  __shared__ uint32_t s_total;
  const int r = blockIdx.x;
  const int len = row_len[r];
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
  const uint2* seg_base = items + (size_t)r * nchunks * kTopkChunk;
  if (threadIdx.x == 0) {
    uint32_t acc = 0;
    for (int c = 0; c < nch; ++c) {
      prefix[c] = acc;
      acc += seg_count[(size_t)r * nchunks + c];
    }
    prefix[nch] = acc;
    s_total = acc;
  }
  __syncthreads();
  const uint32_t total = s_total;
  const uint2 t1 = thr[r];
  const uint32_t d1 = t1.x;
  uint32_t need = (uint32_t)k - t1.y;  // keys with digit == d1 still needed (>= 1)

  // second digit among digit-1 == d1
  for (int i = threadIdx.x; i < kTopkBins2; i += kFinalThreads) h[i] = 0;
  __syncthreads();
  for (uint32_t i = threadIdx.x; i < total; i += kFinalThreads) {
    const uint2 it = item_at(seg_base, prefix, nch, i);
    if ((it.x >> 21) == d1) atomicAdd(&h[(it.x >> 10) & 0x7FF], 1u);
  }
  __syncthreads();
  find_threshold<kTopkBins2, kFinalThreads>(h, need, warp_sums, &s_d, &s_above);
  const uint32_t d2 = (uint32_t)s_d;
  need -= s_above;
  const uint32_t hi22 = (d1 << 11) | d2;

  // third digit among the top 22 bits == (d1, d2)
  for (int i = threadIdx.x; i < kTopkBins2; i += kFinalThreads) h[i] = 0;
  __syncthreads();
  for (uint32_t i = threadIdx.x; i < total; i += kFinalThreads) {
    const uint2 it = item_at(seg_base, prefix, nch, i);
    if ((it.x >> 10) == hi22) atomicAdd(&h[it.x & 0x3FF], 1u);
  }
  __syncthreads();
  find_threshold<kTopkBins3, kFinalThreads>(h, need, warp_sums, &s_d, &s_above);
  const uint32_t T = (hi22 << 10) | (uint32_t)s_d;
  const uint32_t need_eq = need - s_above;  // keys equal to T to take, lowest positions first

  // ordered emission
  uint32_t out_count = 0, eq_seen = 0;
  for (uint32_t b = 0; b < total; b += kFinalThreads) {
    const uint32_t i = b + threadIdx.x;
    uint2 it = make_uint2(0u, 0u);
    if (i < total) it = item_at(seg_base, prefix, nch, i);
    const uint32_t is_eq = (i < total && it.x == T) ? 1u : 0u;
    const uint32_t eq_incl = block_inclusive_scan<kFinalThreads>(is_eq, warp_sums);
    const uint32_t take_eq = is_eq && (eq_seen + eq_incl - 1u) < need_eq;
    const uint32_t sel = (i < total && it.x > T) || take_eq ? 1u : 0u;
    const uint32_t sel_incl = block_inclusive_scan<kFinalThreads>(sel, warp_sums);
    const uint32_t pos = out_count + sel_incl - 1u;
    if (sel && pos < (uint32_t)k) out[pos] = (int32_t)it.y;
    // totals of this batch: the last thread's inclusive values
    __shared__ uint32_t s_batch[2];
    if (threadIdx.x == kFinalThreads - 1) {
      s_batch[0] = sel_incl;
      s_batch[1] = eq_incl;
    }
    __syncthreads();
    out_count += s_batch[0];
    eq_seen += s_batch[1];
    __syncthreads();
  }
  for (int j = (int)out_count + threadIdx.x; j < k; j += kFinalThreads) out[j] = -1;
}

}  // namespace

cudaError_t launch_topk(const TopkArgs& a, cudaStream_t st) {
  if (a.R == 0) return cudaSuccess;
  const TopkLayout L(a.R, a.max_len);
  uint32_t* hist = reinterpret_cast<uint32_t*>(a.scratch + L.hist);
  uint2* thr = reinterpret_cast<uint2*>(a.scratch + L.thr);
  uint32_t* seg_count = reinterpret_cast<uint32_t*>(a.scratch + L.seg_count);
  uint2* items = reinterpret_cast<uint2*>(a.scratch + L.items);
  cudaError_t e = cudaMemsetAsync(hist, 0, (size_t)a.R * kTopkBins1 * 4, st);
  if (e != cudaSuccess) return e;
  dim3 grid(L.nchunks, a.R);
  topk_hist_kernel<<<grid, kHistThreads, 0, st>>>(a.scores, a.ld, a.row_len, a.max_len, a.k, hist);
  topk_collect_kernel<<<grid, kCollectThreads, 0, st>>>(a.scores, a.ld, a.row_len, a.max_len,
                                                        a.k, hist, thr, seg_count, items,
                                                        L.nchunks);
  const size_t smem = (size_t)(L.nchunks + 1) * 4;
  if (smem > 48 * 1024) {
    e = cudaFuncSetAttribute(topk_finalize_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
  }
  topk_finalize_kernel<<<a.R, kFinalThreads, smem, st>>>(a.row_len, a.max_len, a.k, thr,
                                                         seg_count, items, L.nchunks, a.idx,
                                                         a.status);
  return cudaGetLastError();
}

}  // namespace dsa
