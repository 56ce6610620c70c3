/*
 * dsa.h -- C ABI of libdsa: one decode step of a DSA (DeepSeek-style sparse
 * attention) layer, as in Kimi K3.1 Pro's Gated Sparse-MLA layers, on one
 * NVIDIA GB300 (sm_103a).
 *
 * The step is the pages' Score -> Select -> Attend (TokenSpeed post on Kimi
 * K3.1 Pro, "Integrating sparse attention with the K3 stack", steps 2-4):
 *   1. the lightning indexer scores every visible token of a query row with
 *      32 heads x 128 dims against one FP8 E4M3 index key per token (vLLM
 *      Day-0 post, "What Kimi K3.1 Pro changes"), in the DeepSeek-V3.2 form
 *        score(r, s) = sum_h w[r,h] * ReLU( (q[r,h] . k[s]) * ks[s] );
 *   2. the k = 2048 best tokens of each row are kept, ties to the lower
 *      token index (SGLang Day-0 post, "What's new in Kimi K3.1 Pro");
 *   3. exact MLA attention, MQA style, runs over only the selected tokens'
 *      576-wide FP8 latent rows, the first 512 dims doubling as the value
 *      (AMD Instinct post, overview table "MLA"; vLLM post, "What Kimi K3.1
 *      Pro changes": attention runs exactly over only those tokens).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every pointer argument is DEVICE memory owned by the caller unless a
 *    comment says otherwise.  The library never allocates, frees or keeps a
 *    pointer after a call returns.  Inputs are only read; outputs never alias
 *    inputs.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream).  Every call only enqueues work on that stream and returns; it
 *    never synchronises, except dsa_check_device_status.
 *  - Scratch memory comes from the caller's `workspace` (device memory, 256-byte
 *    aligned) of at least the size the matching *_workspace_size function
 *    returns.  A workspace must not be shared by calls that may overlap on the
 *    GPU.  Its first 256 bytes hold the device-side status word.
 *  - Every call returns a status (DSA_OK = 0).  Arguments are validated on the
 *    host before anything is launched; an invalid argument launches nothing.
 *    Values that live in device memory (row lengths, request ids, block-table
 *    entries, selected indices) are checked by the kernels: an out-of-range
 *    value is skipped, never dereferenced, and raises a bit in the workspace
 *    status word, read back with dsa_check_device_status.
 *
 * Cache layouts (token s of request b lives in page block_table[b][s / 64],
 * slot s % 64; both caches share one block table, as the TokenSpeed post's
 * "Storing index keys in the flat KV cache" keeps the index-key plane next to
 * the latent rows of the same page):
 *  - key_cache    uint8 [num_pages][8448]: 64 x 128 E4M3 key bytes (token
 *                 major), then 64 fp32 key scales (little endian).  132 B per
 *                 token: 128 FP8 values and one four-byte scale.
 *  - key_cache (MXFP4 index keys, dsa_indexer_score_mxfp4 and
 *                 dsa_write_kv_mxfp4) uint8 [num_pages][4352]: 64 x 64 bytes of
 *                 E2M1 codes (dim 2j in the low nibble of byte j), then 64 x 4
 *                 E8M0 block scales (byte b scales dims 32b .. 32b + 31).
 *                 68 B per token.
 *  - latent_cache uint8 [num_pages][64][576]: E4M3 latent rows; one fp32
 *                 scale `latent_scale` for the whole cache.
 *  - block_table  int32 [B][max_pages], row-major.
 * Query rows: row_req[R] (request of each row) and row_len[R] (tokens row r
 * sees: 0 <= row_len[r] <= max_pages * 64).  Rows of one request that are
 * adjacent in the row order share one read of the request's index keys.
 */
#ifndef DSA_H
#define DSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ---------------------------------------------------- */
#define DSA_OK 0
#define DSA_ERR_INVALID_ARG 1  /* null pointer, negative size, bad stride   */
#define DSA_ERR_UNSUPPORTED 2  /* shape not built (H, k, dtype)              */
#define DSA_ERR_WORKSPACE 3    /* workspace missing, too small or unaligned  */
#define DSA_ERR_CUDA 4         /* a CUDA launch or query failed              */
#define DSA_ERR_DEVICE_CHECK 5 /* a kernel found an out-of-range device value */

/* bits of the device status word (dsa_check_device_status) */
#define DSA_DEV_BAD_ROW 0x1   /* row_req outside [0,B) or row_len outside [0, max_pages*64] */
#define DSA_DEV_BAD_PAGE 0x2  /* block-table entry outside [0, num_pages)   */
#define DSA_DEV_BAD_INDEX 0x4 /* selected index >= row_len                   */
#define DSA_DEV_TIMEOUT 0x8   /* a bounded wait inside a kernel gave up (about 2 s);
                                 the kernel drained and returned, results are invalid */

/* ---- fixed shapes ------------------------------------------------------ */
#define DSA_PAGE_TOKENS 64
#define DSA_INDEX_HEADS 32
#define DSA_INDEX_DIM 128
#define DSA_KEY_PAGE_BYTES 8448
#define DSA_MXFP4_KEY_PAGE_BYTES 4352 /* 64 x 64 E2M1 code bytes, then 64 x 4 E8M0 scales */
#define DSA_LATENT_DIM 576
#define DSA_V_DIM 512
#define DSA_MAX_TOPK 2048

/* indexer query element types */
#define DSA_BF16 0 /* bf16 [R][32][128]                                     */
#define DSA_E4M3 1 /* E4M3 [R][32][128] with one fp32 scale per (row, head) */

/* Library version: major * 10000 + minor * 100 + patch. */
int dsa_version(void);

/* Static, human-readable text for a status code. */
const char* dsa_status_string(int status);

/* The cudaError_t (as int) behind the most recent DSA_ERR_CUDA returned on the
 * calling host thread, and its text; 0 / "no error" if there was none.  Kept
 * per host thread; a call that succeeds does not clear it. */
int dsa_last_cuda_error(void);
const char* dsa_last_cuda_error_string(void);

/* Number of SMs and whether the current device is an sm_103 part; host-only
 * query of the current device.  Returns DSA_OK or DSA_ERR_CUDA. */
int dsa_device_info(int* num_sms, int* cc_major, int* cc_minor);

/* ------------------------------------------------------------------------
 * dsa_indexer_score -- step 1 alone (Score).
 *
 * scores[r][s] = sum_{h<32} w[r][h] * max(0, (q[r][h] . key[s]) * ks[s]) for
 * 0 <= s < row_len[r], fp32, where key[s] is the E4M3 key of token s of
 * request row_req[r] and ks[s] its fp32 scale (TokenSpeed post, step 2
 * "Score"; vLLM post, "What Kimi K3.1 Pro changes": 32 heads x 128 dims).
 *
 *  q_idx    [R][32][128] bf16 (q_dtype DSA_BF16) or E4M3 (DSA_E4M3).
 *  q_scale  fp32 [R][32] for DSA_E4M3 (q = code * q_scale), NULL for bf16.
 *  w        fp32 [R][32] head weights (any sign).
 *  scores   fp32 [R][ld], ld >= max_pages * 64 and a multiple of 4; only
 *           entries s < row_len[r] are written.
 *  workspace >= dsa_indexer_score_workspace_size(R) bytes.
 * Errors: DSA_ERR_INVALID_ARG, DSA_ERR_UNSUPPORTED (unknown q_dtype),
 * DSA_ERR_WORKSPACE, DSA_ERR_CUDA; device-side DSA_DEV_BAD_ROW/BAD_PAGE.
 * ---------------------------------------------------------------------- */
size_t dsa_indexer_score_workspace_size(int R);
int dsa_indexer_score(const void* q_idx, int q_dtype, const float* q_scale, const float* w,
                      const uint8_t* key_cache, int64_t num_pages, const int32_t* block_table,
                      int B, int max_pages, const int32_t* row_req, const int32_t* row_len,
                      int R, float* scores, int64_t ld, void* workspace, size_t ws_bytes,
                      void* stream);

/* ------------------------------------------------------------------------
 * dsa_indexer_score_mxfp4 -- step 1 over MXFP4 index keys and an MXFP4 query
 * (vLLM Day-0 post on Kimi K3.1 Pro, "Hybrid KV cache without padding": index
 * keys at 68 bytes in MXFP4; "Native MXFP4 indexer": FP4 products with FP32
 * accumulation and a weighted reduction over heads).
 *
 * scores[r][s] = sum_{h<32} w[r][h] * max(0, q[r][h] . key[s]), where every
 * value is an E2M1 element times the E8M0 scale of its block of 32 dims
 * (OCP Microscaling v1.0 formats), on the block-scaled FP4 tensor cores.
 *
 *  q_codes  [R][32][64] bytes: E2M1 codes, dim 2j in the low nibble of byte j;
 *           16-byte aligned.
 *  q_scales [R][32][4] E8M0 bytes (byte b scales dims 32b .. 32b + 31).
 *  w        fp32 [R][32] head weights (any sign).
 *  key_cache pages of DSA_MXFP4_KEY_PAGE_BYTES: token slot t's 64 code bytes
 *           at t * 64, its four scale bytes at 64 * 64 + t * 4; 16-byte aligned.
 *  scores, row_req, row_len, block_table, workspace: as dsa_indexer_score
 *  (workspace >= dsa_indexer_score_workspace_size(R)).
 * Errors: as dsa_indexer_score.
 * ---------------------------------------------------------------------- */
int dsa_indexer_score_mxfp4(const uint8_t* q_codes, const uint8_t* q_scales, const float* w,
                            const uint8_t* key_cache, int64_t num_pages,
                            const int32_t* block_table, int B, int max_pages,
                            const int32_t* row_req, const int32_t* row_len, int R, float* scores,
                            int64_t ld, void* workspace, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * dsa_indexer_score_noalloc -- dsa_indexer_score for callers that cannot
 * provide a workspace.  The pages have no counterpart: this entry point
 * exists for callers that may not allocate device memory when they call the
 * scan -- code capturing a stream into a CUDA graph (allocation is not
 * allowed during capture), decode loops that must not enter the allocator
 * (it can synchronise the device), and hosts that hand a library only the
 * operation's tensors.
 *
 * Same arguments and results as dsa_indexer_score, minus the workspace; the
 * scratch is a fixed array inside the library (1 MiB per GPU, held until the
 * process exits), so R <= DSA_NOALLOC_MAX_ROWS (else DSA_ERR_UNSUPPORTED).
 *  dev_status optional device pointer to one uint32 (4-byte aligned, else
 *             DSA_ERR_INVALID_ARG) that receives the DSA_DEV_* bits of this
 *             call (cleared first); NULL to keep them in the array.
 * All calls on one GPU share the array: calls that may overlap on the GPU
 * race and must be ordered by the caller (one stream, or events).  A call
 * made outside a stream capture looks up the array's device address with the
 * calling device current (so a call after cudaDeviceReset finds the array's
 * new address); a call made during a capture reuses the address found by the
 * last call outside one, so make one call on the device before capturing.
 * Nothing is allocated.
 * ---------------------------------------------------------------------- */
#define DSA_NOALLOC_MAX_ROWS 64
int dsa_indexer_score_noalloc(const void* q_idx, int q_dtype, const float* q_scale,
                              const float* w, const uint8_t* key_cache, int64_t num_pages,
                              const int32_t* block_table, int B, int max_pages,
                              const int32_t* row_req, const int32_t* row_len, int R,
                              float* scores, int64_t ld, uint32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------
 * dsa_topk -- step 2 alone (Select).
 *
 * For each row r: the min(k, row_len[r]) positions s in [0, row_len[r]) with
 * the largest scores[r][s], ties broken towards the lower position (a
 * radix top-k keeps the k highest-scoring positions per query: TokenSpeed
 * post, step 3 "Select").  Scores compare as fp32 values; -0 equals +0.
 * idx[r][0..k) receives the selected positions in ASCENDING position order,
 * followed by -1 padding.  The result is unique, so it is deterministic.
 *
 *  scores  fp32 [R][ld] (only [0, row_len[r]) is read); inputs must be finite.
 *  max_len upper bound of row_len (host value), <= ld.
 *  k       1..2048.
 *  idx     int32 [R][k].
 * Errors: DSA_ERR_INVALID_ARG, DSA_ERR_UNSUPPORTED (k > 2048),
 * DSA_ERR_WORKSPACE, DSA_ERR_CUDA; device-side DSA_DEV_BAD_ROW.
 * ---------------------------------------------------------------------- */
size_t dsa_topk_workspace_size(int R, int64_t max_len, int k);
int dsa_topk(const float* scores, int64_t ld, const int32_t* row_len, int R, int64_t max_len,
             int k, int32_t* idx, void* workspace, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * dsa_write_kv -- step 0 (Write): the new tokens' index keys and latent rows
 * into the paged caches.
 *
 * One fused kernel normalizes a new token's index key, quantizes it to FP8
 * with a single scale and writes it into the cache; the latent row is written
 * next to it (TokenSpeed post on Kimi K3.1 Pro, "Integrating sparse attention
 * with the K3 stack", step 1 "Write"; the key normalization is LayerNorm).
 * For new token t of request tok_req[t] at position tok_pos[t]:
 *   k     = gamma * (x - mean(x)) / sqrt(var(x) + eps) + beta
 *           (x = k_raw[t], 128 values; mean and biased variance over them)
 *   ks    = max|k| / 448 (1 when k is all zero); codes = E4M3(k / ks)
 *   latent row codes = E4M3(latent[t] / latent_scale)
 * (E4M3: round to nearest even, saturating at 448), written at page
 * block_table[req][pos / 64], slot pos % 64, in the layouts of
 * dsa_indexer_score (key codes, then the fp32 scale in the page's scale
 * block) and dsa_sparse_mla_decode (576 latent bytes).
 *
 *  k_raw        bf16 [T][128], 8-byte aligned.
 *  gamma, beta  fp32 [128] (LayerNorm weight and bias), 16-byte aligned.
 *  eps          >= 0.
 *  latent       bf16 [T][576], 16-byte aligned.
 *  latent_scale the latent cache's fp32 scale, > 0.
 *  key_cache, latent_cache  the caches (written in place), 16-byte aligned.
 *  dev_status   optional device uint32: cleared, then receives the DSA_DEV_*
 *               bits of tokens skipped for an out-of-range request, position
 *               or page; NULL to skip the report.
 * Tokens of one call must not share a (page, slot).  No workspace.
 * Errors: DSA_ERR_INVALID_ARG, DSA_ERR_CUDA.
 * ---------------------------------------------------------------------- */
int dsa_write_kv(const void* k_raw, const float* gamma, const float* beta, float eps,
                 const void* latent, float latent_scale, const int32_t* block_table, int B,
                 int max_pages, const int32_t* tok_req, const int32_t* tok_pos, int T,
                 uint8_t* key_cache, uint8_t* latent_cache, int64_t num_pages,
                 uint32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------
 * dsa_write_kv_mxfp4 -- the Write step with MXFP4 index keys (68 bytes per
 * key: vLLM Day-0 post on Kimi K3.1 Pro, "Hybrid KV cache without padding";
 * one E8M0 scale per 32 values: AMD Instinct post on Kimi K3.1 Pro,
 * quantization list).  The key is normalized as in dsa_write_kv, then
 * quantized per block of 32 dims by the OCP Microscaling v1.0 conversion:
 * e = floor(log2(max |k|)) - 2 clamped to [-127, 127] (-127 for a zero
 * block), codes = E2M1(k / 2^e) rounded to nearest even and clamped to 6,
 * into key_cache pages of DSA_MXFP4_KEY_PAGE_BYTES (the layout of
 * dsa_indexer_score_mxfp4).  The latent row is written as by dsa_write_kv.
 * Arguments, alignment and errors as dsa_write_kv.
 * ---------------------------------------------------------------------- */
int dsa_write_kv_mxfp4(const void* k_raw, const float* gamma, const float* beta, float eps,
                       const void* latent, float latent_scale, const int32_t* block_table,
                       int B, int max_pages, const int32_t* tok_req, const int32_t* tok_pos,
                       int T, uint8_t* key_cache, uint8_t* latent_cache, int64_t num_pages,
                       uint32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------
 * dsa_topk_dcp -- step 2 as decode context parallelism runs it, the W GPUs
 * emulated on one.
 *
 * Token p of a row belongs to shard p mod W (SGLang post on Kimi K3.1 Pro,
 * "Decode: DSA with decode context parallelism": token p is stored on GPU
 * p mod 8).  Each shard ranks its own tokens; it shares its best
 * c = ceil(1.5 k / W) (vLLM post, "An exact top-k merge with about 10x less
 * traffic"); the k-th best shared token is the cutoff; a shard that kept
 * tokens back and whose c-th candidate still beats the cutoff may hide
 * winners, so its full local top-k joins the shared candidates; the top-k of
 * those is the result.  Order and ties as dsa_topk, so idx equals what
 * dsa_topk returns for the same scores (the exchange is exact).
 *
 *  scores, ld, row_len, max_len, k, idx: as dsa_topk.
 *  W       shards, 1..DSA_MAX_DCP_SHARDS; R * W <= 65535.
 *  resend  uint32 [R] or NULL: bit s set when shard s's full local top-k was
 *          read (the exchange's second round).
 * Errors: DSA_ERR_INVALID_ARG, DSA_ERR_UNSUPPORTED (k > 2048, W > 32,
 * R * W > 65535), DSA_ERR_WORKSPACE, DSA_ERR_CUDA; device-side DSA_DEV_BAD_ROW.
 * ---------------------------------------------------------------------- */
#define DSA_MAX_DCP_SHARDS 32
size_t dsa_topk_dcp_workspace_size(int R, int64_t max_len, int k, int W);
int dsa_topk_dcp(const float* scores, int64_t ld, const int32_t* row_len, int R, int64_t max_len,
                 int k, int W, int32_t* idx, uint32_t* resend, void* workspace, size_t ws_bytes,
                 void* stream);

/* ------------------------------------------------------------------------
 * dsa_sparse_mla_decode -- step 3 alone (Attend).
 *
 * For row r, head h and the valid selected tokens j (0 <= idx[r][j] <
 * row_len[r]; negative entries are padding and are skipped):
 *   L_j = dec(latent_cache row of token idx[r][j]) * latent_scale
 *   x_j = softmax_scale * (q[r][h] . L_j)           (576 dims)
 *   out[r][h][:] = sum_j softmax(x)_j * L_j[0:512]   (bf16, round to nearest)
 *   lse[r][h]    = ln sum_j exp(x_j)                  (fp32, natural log)
 * (vLLM post, "What Kimi K3.1 Pro changes": MLA attention runs exactly over
 * only the selected tokens; TokenSpeed post, "Sparse attention in Kimi K3.1
 * Pro": every attention head attends to the selected tokens.)  A row with no
 * valid token gets out = 0 and lse = -inf.
 *
 *  q       bf16 [R][H][576]; H in {16, 32, 64, 128}.
 *  idx     int32 [R][k], k in 1..2048 (e.g. the output of dsa_topk).
 *  out     bf16 [R][H][512].   lse  fp32 [R][H] or NULL.
 * Errors: DSA_ERR_INVALID_ARG, DSA_ERR_UNSUPPORTED (H or k), DSA_ERR_WORKSPACE,
 * DSA_ERR_CUDA; device-side DSA_DEV_BAD_ROW/BAD_PAGE/BAD_INDEX.
 * ---------------------------------------------------------------------- */
size_t dsa_sparse_mla_workspace_size(int R, int H, int k);
int dsa_sparse_mla_decode(const void* q, int H, float softmax_scale, const uint8_t* latent_cache,
                          int64_t num_pages, float latent_scale, const int32_t* block_table,
                          int B, int max_pages, const int32_t* row_req, const int32_t* row_len,
                          const int32_t* idx, int k, int R, void* out, float* lse,
                          void* workspace, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * dsa_sparse_mla_decode_nvfp4 -- step 3 over an NVFP4 latent cache: 352 bytes
 * per token instead of 576 (vLLM Day-0 post on Kimi K3.1 Pro, "A packed KV
 * cache for three kinds of state": the MLA latent is 576 bytes in FP8 or 352
 * in NVFP4, and FlashInfer's PrimsTS kernels serve an NVFP4 latent).
 *
 * The pages give the row size only.  Row layout read here (the one split of
 * 576 dims that gives 352 bytes): 256 bytes of E2M1 codes for dims 0..511
 * (dim 2j in the low nibble of byte j), then 32 block scales in unsigned
 * E4M3 (byte b scales dims 16b .. 16b + 15; its top bit is ignored), then the
 * 64 RoPE dims as E4M3 bytes; latent_scale is the per-tensor fp32 scale:
 *   L[d] = e2m1(code d) * ue4m3(scale d / 16) * latent_scale   (d < 512)
 *   L[d] = e4m3(rope byte d - 512) * latent_scale              (d >= 512)
 * The attention is then the one of dsa_sparse_mla_decode, with the same
 * arguments, sizes, workspace (dsa_sparse_mla_workspace_size) and errors.
 *
 *  latent_cache  uint8 [num_pages][64][352], 16-byte aligned.
 * Accuracy: the kernel feeds the tensor cores c * s / 4 (c the E2M1 value,
 * s its block scale) as two E4M3 terms and a RoPE byte r as E4M3(r / 4).
 * Both are exact for s >= 0.5 (scale byte >= 0x30) and |r| >= 2^-4; below,
 * an element loses at most 2^-8 * latent_scale.  A scale byte 0x7F (or 0xFF)
 * is NaN, as in E4M3.
 * ---------------------------------------------------------------------- */
#define DSA_NVFP4_LATENT_ROW_BYTES 352
int dsa_sparse_mla_decode_nvfp4(const void* q, int H, float softmax_scale,
                                const uint8_t* latent_cache, int64_t num_pages,
                                float latent_scale, const int32_t* block_table, int B,
                                int max_pages, const int32_t* row_req, const int32_t* row_len,
                                const int32_t* idx, int k, int R, void* out, float* lse,
                                void* workspace, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * dsa_decode_step -- the whole step (Score -> Select -> Attend), fused into
 * one launch sequence on `stream` with no host round trip.  Arguments mean
 * what they mean above; the scores never leave the workspace.
 *  idx_out  optional int32 [R][k]: receives the selection (ascending, -1
 *           padded), e.g. for tests; NULL to skip.
 *  workspace >= dsa_decode_step_workspace_size(B, R, max_pages, H, k).
 * ---------------------------------------------------------------------- */
size_t dsa_decode_step_workspace_size(int B, int R, int max_pages, int H, int k);
int dsa_decode_step(const void* q_idx, int q_dtype, const float* q_scale, const float* w,
                    const uint8_t* key_cache, const uint8_t* latent_cache, int64_t num_pages,
                    float latent_scale, const int32_t* block_table, int B, int max_pages,
                    const int32_t* row_req, const int32_t* row_len, int R, const void* q, int H,
                    float softmax_scale, int k, void* out, float* lse, int32_t* idx_out,
                    void* workspace, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * dsa_decode_step_fp4 -- the whole step over the pages' smaller caches:
 * MXFP4 index keys (68 bytes per token, as dsa_indexer_score_mxfp4) and NVFP4
 * latent rows (352 bytes per token, as dsa_sparse_mla_decode_nvfp4), 10,080
 * bytes per token over 24 layers against 16,992 with both in FP8 (vLLM Day-0
 * post on Kimi K3.1 Pro, "KV cache footprint per token").  Same order of
 * kernels, workspace (dsa_decode_step_workspace_size) and outputs as
 * dsa_decode_step; the query of the indexer is MXFP4 (q_codes [R][32][64],
 * q_scales [R][32][4], as dsa_indexer_score_mxfp4), the MLA query bf16.
 *  key_cache     uint8 [num_pages][4352] (MXFP4 pages), 16-byte aligned.
 *  latent_cache  uint8 [num_pages][64][352] (NVFP4 rows), 16-byte aligned.
 * Errors: as dsa_decode_step; q_codes must be 16-byte aligned, q_scales
 * 4-byte aligned.
 * ---------------------------------------------------------------------- */
int dsa_decode_step_fp4(const uint8_t* q_codes, const uint8_t* q_scales, const float* w,
                        const uint8_t* key_cache, const uint8_t* latent_cache, int64_t num_pages,
                        float latent_scale, const int32_t* block_table, int B, int max_pages,
                        const int32_t* row_req, const int32_t* row_len, int R, const void* q,
                        int H, float softmax_scale, int k, void* out, float* lse,
                        int32_t* idx_out, void* workspace, size_t ws_bytes, void* stream);

/* Synchronises `stream`, then reads the device status word in `workspace`
 * (bits DSA_DEV_*, written by the kernels of the last call that used this
 * workspace) into *bits (may be NULL).  Returns DSA_OK when no bit is set,
 * DSA_ERR_DEVICE_CHECK when one is, DSA_ERR_CUDA when the copy fails. */
int dsa_check_device_status(const void* workspace, void* stream, uint32_t* bits);

/* ------------------------------------------------------------------------
 * dsa_selftest_bounded_wait -- library self-test of failure detection.
 *
 * The pipeline kernels bound every wait on an mbarrier (about 2 s); when one
 * runs out the kernel raises DSA_DEV_TIMEOUT, waits for the copies it issued,
 * frees its tensor memory and returns, leaving the stream and the context
 * usable.  This call takes that path on purpose: it launches one CTA that
 * holds 32 TMEM columns, has a 256-byte bulk copy in flight and waits on an
 * mbarrier that nothing arrives on, with a limit of `wait_us` microseconds
 * (1..1000000, converted with the device's peak SM clock).  Once the stream
 * has run it, dsa_check_device_status reports DSA_DEV_TIMEOUT, and bytes
 * [512,768) of the workspace hold a copy of bytes [256,512) (the bulk copy,
 * drained after the failed wait).
 *  workspace >= dsa_selftest_workspace_size() bytes, 256-byte aligned:
 *             [0,256) status word, [256,512) copy source (any contents,
 *             caller-owned), [512,768) the kernel's copy of it.
 * Returns DSA_OK once enqueued; DSA_ERR_INVALID_ARG (wait_us out of range),
 * DSA_ERR_WORKSPACE, DSA_ERR_CUDA.
 * ------------------------------------------------------------------------ */
size_t dsa_selftest_workspace_size(void);
int dsa_selftest_bounded_wait(int wait_us, void* workspace, size_t ws_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DSA_H */
