// dcp.cu -- the top-k of a row under decode context parallelism, with the W
// token shards emulated on one GPU.
//
// Token p of a request lives on GPU p mod W; each GPU ranks only its own
// tokens, shares its best candidates, takes the k-th best shared score as the
// cutoff, and a GPU whose candidates all beat the cutoff may hide winners, so
// its full local top-k is read and the selection is run again; the result
// matches a single-GPU top-k exactly (SGLang post on Kimi K3.1 Pro, "Decode:
// DSA with decode context parallelism"; vLLM post, "An exact top-k merge with
// about 10x less traffic": 1.5 k / W candidates per GPU, a resend when a GPU
// may hold more winners than it sent).
//
// Every selection below is the library's exact top-k (ties to the lower
// position).  The tokens taking part in a selection are marked in a bitmap
// over the row's positions and compacted in position order (a popcount
// prefix over the bitmap words), so each selection runs on a short row of
// members whose order is the positions' order.  Token sharding by p mod W
// keeps shard sizes within one of each other, so at least min(k, len)
// candidates are always shared.
//   1. shard:     local[s * R + r][j] = scores[r][s + W j], j < n_s(r);
//   2. local top-k and local top-c of every (shard, row), c = ceil(1.5 k / W)
//      (at most 2048);
//   3. members:   the c candidates of every shard;
//   4. their top-k; its worst member (in the order score descending,
//      position ascending) is the cutoff E;
//   5. suspects:  shards that kept tokens back (n_s > c) whose c-th candidate
//      precedes E; their local top-k join the members;
//   6. the top-k of the members is the result.
// A multi-GPU caller runs 1-2 on each GPU over its own shard, exchanges the
// candidates of 2 and the local top-k of the suspects of 5, and runs 3-6 on
// the gathered tokens.
#include "dsa_common.cuh"

namespace dsa {
namespace {

constexpr int kThreads = 256;
constexpr int kCompactThreads = 1024;

__device__ __forceinline__ bool len_ok(int len, int64_t max_len) {
  return len >= 0 && (int64_t)len <= max_len;
}

// number of tokens of shard s among the first len
__device__ __forceinline__ int shard_count(int len, int s, int W) {
  return len > s ? (len - s + W - 1) / W : 0;
}

// key order composite: larger = earlier in the order (score desc, position asc)
typedef unsigned long long u64;
__device__ __forceinline__ u64 rank_key(const float* row, int p) {
  return ((u64)ordered_key(row[p]) << 32) | (u64)(~(uint32_t)p);
}
__device__ __forceinline__ u64 min_u64(u64 a, u64 b) { return a < b ? a : b; }

// ---- 1. shard the rows ---------------------------------------------------------
__global__ void __launch_bounds__(kThreads)
dcp_shard_kernel(const float* __restrict__ scores, int64_t ld, const int32_t* __restrict__ row_len,
                 int R, int64_t max_len, int W, float* __restrict__ local, int64_t ld_s,
                 int32_t* __restrict__ local_len, uint32_t* status) {
  pdl_trigger();
  pdl_wait();
  const int lr = blockIdx.y;                  // s * R + r
  const int s = lr / R, r = lr % R;
  int len = row_len[r];
  if (!len_ok(len, max_len)) {
    if (blockIdx.x == 0 && threadIdx.x == 0 && s == 0) raise_dev(status, DSA_DEV_BAD_ROW);
    len = 0;
  }
  const int n = shard_count(len, s, W);
  if (blockIdx.x == 0 && threadIdx.x == 0) local_len[lr] = n;
  const float* row = scores + (size_t)r * ld;
  float* dst = local + (size_t)lr * ld_s;
  for (int64_t j = (int64_t)blockIdx.x * kThreads + threadIdx.x; j < n;
       j += (int64_t)gridDim.x * kThreads)
    dst[j] = row[s + (int64_t)W * j];
}

// ---- 3. mark the shared candidates in the member bitmap -----------------------
__global__ void __launch_bounds__(kThreads)
dcp_candidates_kernel(const int32_t* __restrict__ row_len, int R, int64_t max_len, int W,
                      const int32_t* lc, int c, uint32_t* bits,
                      int64_t nwords) {
  pdl_trigger();
  pdl_wait();
  const int r = blockIdx.x;
  int len = row_len[r];
  if (!len_ok(len, max_len)) len = 0;
  uint32_t* b = bits + (size_t)r * nwords;
  for (int64_t w = threadIdx.x; w < ((int64_t)len + 31) / 32; w += kThreads) b[w] = 0u;
  __syncthreads();
  for (int e = threadIdx.x; e < W * c; e += kThreads) {
    const int s = e / c, j = lc[((size_t)s * R + r) * c + e % c];
    if (j >= 0) {
      const int p = s + W * j;
      atomicOr(&b[p >> 5], 1u << (p & 31));
    }
  }
}

// ---- members in position order: positions and scores of the set bits ----------
__global__ void __launch_bounds__(kCompactThreads)
dcp_compact_kernel(const float* __restrict__ scores, int64_t ld,
                   const int32_t* __restrict__ row_len, int64_t max_len,
                   const uint32_t* bits, int64_t nwords, int32_t* __restrict__ mpos,
                   float* __restrict__ mscore, int64_t ld_m, int32_t* __restrict__ mlen) {
  __shared__ uint32_t s_warp[kCompactThreads / 32];
  __shared__ uint32_t s_base;
  pdl_trigger();
  pdl_wait();
  const int r = blockIdx.x, lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int len = row_len[r];
  if (!len_ok(len, max_len)) len = 0;
  const uint32_t* b = bits + (size_t)r * nwords;
  const float* row = scores + (size_t)r * ld;
  if (threadIdx.x == 0) s_base = 0u;
  const int64_t nw = ((int64_t)len + 31) / 32;
  for (int64_t w0 = 0; w0 < nw; w0 += kCompactThreads) {          // uniform trip count
    const int64_t w = w0 + threadIdx.x;
    const uint32_t word = w < nw ? b[w] : 0u;
    const uint32_t cnt = __popc(word);
    uint32_t x = cnt;                                             // inclusive warp scan
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[wid] = x;
    __syncthreads();
    uint32_t before = s_base;
    for (int v = 0; v < wid; ++v) before += s_warp[v];
    uint32_t at = before + x - cnt;
    for (uint32_t m = word; m; m &= m - 1) {
      const int p = (int)(w * 32 + __ffs(m) - 1);
      mpos[(size_t)r * ld_m + at] = p;
      mscore[(size_t)r * ld_m + at] = row[p];
      ++at;
    }
    __syncthreads();                                              // every thread read s_base
    if (threadIdx.x == kCompactThreads - 1) s_base = before + x;
    __syncthreads();
  }
  if (threadIdx.x == 0) mlen[r] = (int32_t)s_base;
}

// ---- 5. the cutoff and the suspects; their local top-k join the member row ----
__global__ void __launch_bounds__(kThreads)
dcp_suspects_kernel(const float* __restrict__ scores, int64_t ld,
                    const int32_t* __restrict__ row_len, int R, int64_t max_len, int W, int k,
                    const int32_t* ck, const int32_t* mpos, int64_t ld_m, const int32_t* lc,
                    int c, const int32_t* lk, uint32_t* bits, int64_t nwords,
                    uint32_t* __restrict__ resend) {
  __shared__ u64 s_min[kThreads / 32];
  __shared__ uint32_t s_mask;
  pdl_trigger();
  pdl_wait();
  const int r = blockIdx.x, lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int len = row_len[r];
  if (!len_ok(len, max_len)) len = 0;
  const float* row = scores + (size_t)r * ld;
  // the cutoff E: the worst of the k selected candidates (none when fewer than k)
  u64 m = ~0ull;
  int nsel = 0;
  for (int j = threadIdx.x; j < k; j += kThreads) {
    const int q = ck[(size_t)r * k + j];                      // index among the members
    if (q >= 0) {
      const int p = mpos[(size_t)r * ld_m + q];
      m = min_u64(m, rank_key(row, p));
      ++nsel;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    m = min_u64(m, __shfl_xor_sync(0xffffffffu, m, o));
    nsel += __shfl_xor_sync(0xffffffffu, nsel, o);
  }
  __shared__ int s_nsel[kThreads / 32];
  if (lane == 0) {
    s_min[wid] = m;
    s_nsel[wid] = nsel;
  }
  if (threadIdx.x == 0) s_mask = 0u;
  __syncthreads();
  u64 E = ~0ull;
  int total = 0;
  for (int w = 0; w < kThreads / 32; ++w) {
    E = min_u64(E, s_min[w]);
    total += s_nsel[w];
  }
  const bool has_cut = total >= k;
  // warp w judges shards w, w + 8, ...: the shard's c-th candidate is the
  // worst of its local top-c
  for (int s = wid; s < W; s += kThreads / 32) {
    const int n = shard_count(len, s, W);
    u64 worst = ~0ull;
    for (int j = lane; j < c; j += 32) {
      const int lj = lc[((size_t)s * R + r) * c + j];
      if (lj >= 0) worst = min_u64(worst, rank_key(row, s + W * lj));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) worst = min_u64(worst, __shfl_xor_sync(0xffffffffu, worst, o));
    if (lane == 0 && n > c && (!has_cut || worst > E)) atomicOr(&s_mask, 1u << s);
  }
  __syncthreads();
  const uint32_t mask = s_mask;
  if (threadIdx.x == 0 && resend) resend[r] = mask;
  uint32_t* bm = bits + (size_t)r * nwords;
  for (int e = threadIdx.x; e < W * k; e += kThreads) {
    const int s = e / k;
    if (!((mask >> s) & 1u)) continue;
    const int j = lk[((size_t)s * R + r) * k + e % k];
    if (j >= 0) {
      const int p = s + W * j;
      atomicOr(&bm[p >> 5], 1u << (p & 31));
    }
  }
}

// ---- the selected members' positions (ascending, as the members are) ----------
__global__ void __launch_bounds__(kThreads)
dcp_positions_kernel(const int32_t* sel, const int32_t* mpos,
                     int64_t ld_m, int k, int32_t* __restrict__ idx) {
  pdl_trigger();
  pdl_wait();
  const int r = blockIdx.x;
  for (int j = threadIdx.x; j < k; j += kThreads) {
    const int q = sel[(size_t)r * k + j];
    idx[(size_t)r * k + j] = q >= 0 ? mpos[(size_t)r * ld_m + q] : -1;
  }
}

struct DcpLayout {
  int64_t ld_s, ld_m, nwords;
  int c;
  size_t local, local_len, lk, lc, bits, mpos, mscore, mlen, ck, topk, bytes;
  DcpLayout(int R, int64_t max_len, int k, int W) {
    ld_s = ((max_len + W - 1) / W + 3) / 4 * 4;
    const int64_t cc = (3 * (int64_t)k + 2 * W - 1) / (2 * W);
    c = (int)(cc < kMaxTopk ? cc : kMaxTopk);
    const int64_t most = (int64_t)W * (k > c ? k : c);             // members at most
    ld_m = ((most < max_len ? most : max_len) + 3) / 4 * 4;
    nwords = (max_len + 31) / 32;
    const size_t WR = (size_t)W * R;
    size_t o = 0;
    local = o;     o = align_up(o + WR * (size_t)ld_s * 4);
    local_len = o; o = align_up(o + WR * 4);
    lk = o;        o = align_up(o + WR * (size_t)k * 4);
    lc = o;        o = align_up(o + WR * (size_t)c * 4);
    bits = o;      o = align_up(o + (size_t)R * (size_t)nwords * 4);
    mpos = o;      o = align_up(o + (size_t)R * (size_t)ld_m * 4);
    mscore = o;    o = align_up(o + (size_t)R * (size_t)ld_m * 4);
    mlen = o;      o = align_up(o + (size_t)R * 4);
    ck = o;        o = align_up(o + (size_t)R * (size_t)k * 4);
    topk = o;
    const size_t t1 = TopkLayout((int)WR, ld_s).bytes, t2 = TopkLayout(R, ld_m).bytes;
    o = align_up(o + (t1 > t2 ? t1 : t2));
    bytes = o;
  }
};

}  // namespace

size_t dcp_scratch_bytes(int R, int64_t max_len, int k, int W) {
  return DcpLayout(R, max_len, k, W).bytes;
}

cudaError_t launch_topk_dcp(const DcpArgs& a, cudaStream_t st) {
  if (a.R == 0) return cudaSuccess;
  const DcpLayout L(a.R, a.max_len, a.k, a.W);
  uint8_t* ws = a.scratch;
  float* local = reinterpret_cast<float*>(ws + L.local);
  int32_t* local_len = reinterpret_cast<int32_t*>(ws + L.local_len);
  int32_t* lk = reinterpret_cast<int32_t*>(ws + L.lk);
  int32_t* lc = reinterpret_cast<int32_t*>(ws + L.lc);
  uint32_t* bits = reinterpret_cast<uint32_t*>(ws + L.bits);
  int32_t* mpos = reinterpret_cast<int32_t*>(ws + L.mpos);
  float* mscore = reinterpret_cast<float*>(ws + L.mscore);
  int32_t* mlen = reinterpret_cast<int32_t*>(ws + L.mlen);
  int32_t* ck = reinterpret_cast<int32_t*>(ws + L.ck);
  const int WR = a.W * a.R;
  // 1. shard
  const int gx = (int)((L.ld_s + kThreads - 1) / kThreads);
  cudaError_t e = launch_kernel(dcp_shard_kernel, dim3(gx < 64 ? gx : 64, WR), dim3(kThreads), 0, st,
                                a.chained, a.scores, a.ld, a.row_len, a.R, a.max_len, a.W, local,
                                L.ld_s, local_len, a.status);
  if (e != cudaSuccess) return e;
  // 2. local top-k and local top-c of every (shard, row)
  TopkArgs t{local, L.ld_s, local_len, WR, L.ld_s, a.k, lk, ws + L.topk, a.status, true};
  if ((e = launch_topk(t, st)) != cudaSuccess) return e;
  t.k = L.c;
  t.idx = lc;
  if ((e = launch_topk(t, st)) != cudaSuccess) return e;
  // 3. the shared candidates; 4. their top-k
  e = launch_kernel(dcp_candidates_kernel, dim3(a.R), dim3(kThreads), 0, st, true,
                    a.row_len, a.R, a.max_len, a.W, (const int32_t*)lc, L.c, bits, L.nwords);
  if (e != cudaSuccess) return e;
  auto compact = [&]() {
    return launch_kernel(dcp_compact_kernel, dim3(a.R), dim3(kCompactThreads), 0, st, true,
                         a.scores, a.ld, a.row_len, a.max_len, (const uint32_t*)bits, L.nwords,
                         mpos, mscore, L.ld_m, mlen);
  };
  if ((e = compact()) != cudaSuccess) return e;
  TopkArgs m{mscore, L.ld_m, mlen, a.R, L.ld_m, a.k, ck, ws + L.topk, a.status, true};
  if ((e = launch_topk(m, st)) != cudaSuccess) return e;
  // 5. cutoff and suspects (their local top-k join the members); 6. the final top-k
  e = launch_kernel(dcp_suspects_kernel, dim3(a.R), dim3(kThreads), 0, st, true, a.scores, a.ld,
                    a.row_len, a.R, a.max_len, a.W, a.k, (const int32_t*)ck, (const int32_t*)mpos,
                    L.ld_m, (const int32_t*)lc, L.c, (const int32_t*)lk, bits, L.nwords, a.resend);
  if (e != cudaSuccess) return e;
  if ((e = compact()) != cudaSuccess) return e;
  if ((e = launch_topk(m, st)) != cudaSuccess) return e;
  e = launch_kernel(dcp_positions_kernel, dim3(a.R), dim3(kThreads), 0, st, true,
                    (const int32_t*)ck, (const int32_t*)mpos, L.ld_m, a.k, a.idx);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace dsa
