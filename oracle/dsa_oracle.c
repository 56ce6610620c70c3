/*
 * dsa_oracle.c -- plain, slow, float64 CPU definition of one DSA decode step.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the oracle that the CUDA library is
 * checked against.  Only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark may load it.  It shares no code, header, table or
 * constant with the CUDA path (dsa_sparse_attention_lightning_gb300/csrc), and
 * neither side includes or links the other.
 *
 * Every function below is the plain definition of what the step computes,
 * written out in float64 with no blocking, fusion or reordering:
 *
 *   - oracle_e4m3_decode       the OCP FP8 E4M3 ("E4M3FN") value of a byte
 *   - oracle_indexer_scores    lightning-indexer score of every visible token
 *   - oracle_topk              top-k positions, ties to the lower token index
 *   - oracle_topk_dcp          the same top-k by the decode-context-parallel
 *                              exchange (W token shards, candidates, cutoff,
 *                              resend of shards that may hide winners)
 *   - oracle_sparse_mla        exact softmax attention over the selected rows
 *   - oracle_e4m3_encode       nearest E4M3 value of a real (ties to even)
 *   - oracle_write_kv          the Write step: LayerNorm of a new token's index
 *                              key, FP8 quantization with one scale, paged
 *                              write; the latent row's FP8 write
 *   - oracle_e2m1_decode, oracle_e2m1_encode, oracle_e8m0_decode,
 *     oracle_mx_quantize, oracle_write_key_mx, oracle_indexer_scores_mx
 *                              MXFP4 index keys (68 bytes per token) and the
 *                              indexer over them
 *   - oracle_nvfp4_latent_decode, oracle_nvfp4_latent_encode,
 *     oracle_sparse_mla_nvfp4  NVFP4 latent rows (352 bytes per token) and
 *                              sparse MLA over them
 *
 * Sources (web pages on Kimi K3.1 Pro's sparse attention):
 *   [TS]   TokenSpeed post on Kimi K3.1 Pro (lightseek.org), sections
 *          "Sparse attention in Kimi K3.1 Pro", "Integrating sparse attention
 *          with the K3 stack" (steps 1-4) and "Storing index keys in the flat
 *          KV cache".
 *   [VLLM] "vLLM Day-0 Support for Kimi K3.1 Pro: Sparse Attention, DCP, and
 *          Zero-Mismatch RL", sections "What Kimi K3.1 Pro changes" (table and
 *          the paragraph after it) and "Sparse attention cuts long-context
 *          decode bandwidth".
 *   [SGL]  "Kimi K3.1 Pro: Day-0 Inference and RL Support with SGLang and
 *          Miles", sections "What's new in Kimi K3.1 Pro" and "Decode: DSA
 *          with decode context parallelism".
 *   [VLLM] also section "An exact top-k merge with about 10x less traffic".
 *   [AMD]  "Kimi K3.1 Pro on AMD Instinct GPUs" (dev48.org, in Russian),
 *          overview table, row "MLA" (KV LoRA rank 512 + 64 RoPE dims), and
 *          the quantization list (MXFP4: one E8M0 scale per 32 values).
 *   [VLLM] also "Hybrid KV cache without padding" (index keys at 68 bytes in
 *          MXFP4) and "Native MXFP4 indexer" (68 bytes including scales;
 *          FP4 products, FP32 accumulation, weighted reduction over heads).
 *
 * The pages do not print the indexer formula; they point to DeepSeek-V3.2 for
 * it.  The form used here is the DeepSeek-V3.2 lightning indexer:
 *   score(r, s) = sum_h w[r,h] * ReLU( (q[r,h] . k[s]) * ks[s] )
 * with the ReLU applied to the scaled dot product, in that literal order.
 *
 * Parity pins: every function is pinned by tests/test_oracle_pins.py against
 * closed forms, library routines and brute force (listed per function).
 * No function here is parity-unpinned.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Index-key page: 64 tokens x 128 E4M3 values, then 64 fp32 scales. */
#define ORA_PAGE 64
#define ORA_IDX_DIM 128
#define ORA_IDX_HEADS 32
#define ORA_KEY_PAGE_BYTES (ORA_PAGE * ORA_IDX_DIM + ORA_PAGE * 4)
/* MXFP4 index-key page: 64 tokens x 64 bytes of packed E2M1 codes, then 64 x 4
 * E8M0 block scales (one per 32 dims); 68 bytes per token. */
#define ORA_MX_BLOCK 32
#define ORA_MX_KEY_BYTES (ORA_IDX_DIM / 2)
#define ORA_MX_SCALES (ORA_IDX_DIM / ORA_MX_BLOCK)
#define ORA_MX_KEY_PAGE_BYTES (ORA_PAGE * ORA_MX_KEY_BYTES + ORA_PAGE * ORA_MX_SCALES)
/* Latent row: 512 compressed-KV dims + 64 RoPE dims ([AMD] overview, "MLA"). */
#define ORA_LAT_DIM 576
#define ORA_V_DIM 512

enum { ORA_OK = 0, ORA_BAD_PAGE = 1, ORA_BAD_INDEX = 2, ORA_BAD_ARG = 3 };

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/*
 * E4M3 ("E4M3FN" in the OCP 8-bit floating point specification): one sign
 * bit, four exponent bits with bias 7, three mantissa bits.  Exponent field 0
 * encodes subnormals 2^-6 * m/8; the all-ones pattern with mantissa 7 is NaN;
 * there are no infinities.  [TS] "Storing index keys in the flat KV cache":
 * each index key is 128 FP8 values plus one four-byte scale.
 * Pinned by: all 256 codes against torch.float8_e4m3fn -> float32.
 */
double oracle_e4m3_decode(uint8_t code) {
    int sign = (code >> 7) & 1;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double mag;
    if (e == 0xF && m == 0x7) return NAN;
    if (e == 0)
        mag = ldexp((double)m / 8.0, -6);
    else
        mag = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -mag : mag;
}

/* bfloat16 is the upper half of an IEEE binary32; its value is exact in double. */
static double bf16_to_double(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double f32_at(const uint8_t* p) {
    float f;
    memcpy(&f, p, sizeof f);
    return (double)f;
}

/*
 * E4M3 encoding of a real value, the inverse of oracle_e4m3_decode on the
 * finite codes: the nearest finite E4M3 value, a tie going to the code whose
 * mantissa is even (round to nearest even), magnitudes of 448 and above
 * saturating to 448 ("satfinite"); the sign is kept (-0 encodes as 0x80).
 * By brute force over the 127 non-negative finite codes.
 * Pinned by: the round trip over every finite code, torch's float8_e4m3fn
 * cast on values in [-448, 448] including every midpoint, golden ties.
 */
uint8_t oracle_e4m3_encode(double x) {
    const int sign = signbit(x) ? 1 : 0;
    const double a = fabs(x);
    if (a >= 448.0) return (uint8_t)((sign << 7) | 0x7E);
    int best = 0;
    double bestd = INFINITY;
    for (int c = 0; c < 0x7F; ++c) {
        const double d = fabs(a - oracle_e4m3_decode((uint8_t)c));
        if (d < bestd || (d == bestd && (c & 1) == 0)) {
            best = c;
            bestd = d;
        }
    }
    return (uint8_t)((sign << 7) | best);
}

/* k = gamma * (x - mean(x)) / sqrt(var(x) + eps) + beta over the 128 dims of one
 * bf16 key, with the biased variance. */
static void layer_norm_key(const uint16_t* k_raw, const double* gamma, const double* beta,
                           double eps, double* k) {
    double x[ORA_IDX_DIM], mean = 0.0, var = 0.0;
    for (int d = 0; d < ORA_IDX_DIM; ++d) {
        x[d] = bf16_to_double(k_raw[d]);
        mean += x[d];
    }
    mean /= ORA_IDX_DIM;
    for (int d = 0; d < ORA_IDX_DIM; ++d) var += (x[d] - mean) * (x[d] - mean);
    var /= ORA_IDX_DIM;
    for (int d = 0; d < ORA_IDX_DIM; ++d)
        k[d] = gamma[d] * (x[d] - mean) / sqrt(var + eps) + beta[d];
}

/*
 * The Write step ([TS] step 1 "Write": one fused kernel normalizes the new
 * token's index key, quantizes it to FP8 with a single scale and writes it
 * into the cache, and one kernel writes the latent row; [TS] "Integrating
 * sparse attention with the K3 stack": the only key normalization accepted
 * is LayerNorm; [TS] "Storing index keys in the flat KV cache": 128 FP8
 * values and one four-byte scale per token).  For new token t of request
 * tok_req[t] at position tok_pos[t]:
 *   x      = k_raw[t] (128 bf16 values)
 *   k      = gamma * (x - mean(x)) / sqrt(var(x) + eps) + beta
 *            (mean and biased variance over the 128 dims)
 *   ks     = max_d |k[d]| / 448   (1 when k is all zero)
 *   codes  = e4m3_encode(k / ks)
 * go to page block_table[req][pos / 64], slot pos % 64 of key_cache: the 128
 * codes at slot * 128, ks as fp32 at 64 * 128 + slot * 4; and the latent row
 * e4m3_encode(latent[t] / latent_scale) (576 bf16 values in) to
 * latent_cache[page][slot][0..576).  The values before rounding (k / ks and
 * latent / latent_scale) are returned in key_pre [T][128] and lat_pre
 * [T][576], and ks in key_scale [T], so that a test can see codes that sit
 * at a rounding midpoint.
 * Pinned by: LayerNorm against torch's float64 layer_norm, the absmax code
 * being exactly 448, a zero key, the latent codes against the generator's
 * torch cast, placement through a shuffled block table.
 */
int oracle_write_kv(const uint16_t* k_raw, const double* gamma, const double* beta, double eps,
                    const uint16_t* latent, double latent_scale, const int32_t* block_table,
                    int B, int max_pages, const int32_t* tok_req, const int32_t* tok_pos, int T,
                    uint8_t* key_cache, uint8_t* latent_cache, int64_t num_pages,
                    double* key_pre, double* lat_pre, double* key_scale) {
    if (T < 0 || !(latent_scale > 0.0) || !(eps >= 0.0)) return ORA_BAD_ARG;
    for (int t = 0; t < T; ++t) {
        const int req = tok_req[t], pos = tok_pos[t];
        if (req < 0 || req >= B || pos < 0 || pos >= max_pages * ORA_PAGE) return ORA_BAD_ARG;
        const int page = block_table[(size_t)req * max_pages + pos / ORA_PAGE];
        if (page < 0 || (int64_t)page >= num_pages) return ORA_BAD_PAGE;
        const int slot = pos % ORA_PAGE;
        /* index key: LayerNorm, absmax scale, E4M3 codes */
        double k[ORA_IDX_DIM], amax = 0.0;
        layer_norm_key(k_raw + (size_t)t * ORA_IDX_DIM, gamma, beta, eps, k);
        for (int d = 0; d < ORA_IDX_DIM; ++d)
            if (fabs(k[d]) > amax) amax = fabs(k[d]);
        const double ks = amax > 0.0 ? amax / 448.0 : 1.0;
        uint8_t* kp = key_cache + (size_t)page * ORA_KEY_PAGE_BYTES;
        for (int d = 0; d < ORA_IDX_DIM; ++d) {
            const double v = k[d] / ks;
            kp[(size_t)slot * ORA_IDX_DIM + d] = oracle_e4m3_encode(v);
            if (key_pre) key_pre[(size_t)t * ORA_IDX_DIM + d] = v;
        }
        const float ksf = (float)ks;
        memcpy(kp + ORA_PAGE * ORA_IDX_DIM + (size_t)slot * 4, &ksf, sizeof ksf);
        if (key_scale) key_scale[t] = ks;
        /* latent row */
        uint8_t* lp = latent_cache + ((size_t)page * ORA_PAGE + slot) * ORA_LAT_DIM;
        for (int d = 0; d < ORA_LAT_DIM; ++d) {
            const double v = bf16_to_double(latent[(size_t)t * ORA_LAT_DIM + d]) / latent_scale;
            lp[d] = oracle_e4m3_encode(v);
            if (lat_pre) lat_pre[(size_t)t * ORA_LAT_DIM + d] = v;
        }
    }
    return ORA_OK;
}

/*
 * Lightning-indexer scores ([SGL] "What's new": the indexer scores every
 * earlier token; [VLLM] "What Kimi K3.1 Pro changes": 32 heads x 128 dims,
 * FP8 keys, one key per token; [TS] step 2 "Score").
 *
 *   score[r][s] = sum_{h<32} w[r][h] * max(0, (sum_{d<128} q[r][h][d] *
 *                 key[s][d]) * ks[s])           for 0 <= s < row_len[r]
 *
 * Token s of request b is in page block_table[b][s / 64], slot s % 64 (the
 * paged cache of [TS] "Storing index keys..."; 64-token pages).  Within a
 * page: 64 x 128 key bytes, then 64 fp32 scales.
 *
 * The query is bf16 (q_bf16 != NULL) or E4M3 with one fp32 scale per (row,
 * head) (q_e4m3 and q_scale != NULL): q[r][h][d] = dec(q8) * q_scale[r][h].
 * Entries s >= row_len[r] of scores are left untouched.
 * Pinned by: dot-product special case vs numpy, q = 0, linearity in w,
 * scale-factoring identity, float64 einsum cross-check.
 */
int oracle_indexer_scores(const uint16_t* q_bf16, const uint8_t* q_e4m3, const float* q_scale,
                          const float* w, const uint8_t* key_cache, int64_t num_pages,
                          const int32_t* block_table, int B, int max_pages,
                          const int32_t* row_req, const int32_t* row_len, int R,
                          double* scores, int64_t ld) {
    int status = ORA_OK;
    if ((q_bf16 == NULL) == (q_e4m3 == NULL)) return ORA_BAD_ARG;
    if (q_e4m3 != NULL && q_scale == NULL) return ORA_BAD_ARG;
    for (int r = 0; r < R; ++r) {
        if (row_req[r] < 0 || row_req[r] >= B) return ORA_BAD_ARG;
        if (row_len[r] < 0 || (int64_t)row_len[r] > ld ||
            (int64_t)row_len[r] > (int64_t)max_pages * ORA_PAGE)
            return ORA_BAD_ARG;
    }
    for (int r = 0; r < R; ++r) {
        const int b = row_req[r];
        const int64_t len = row_len[r];
        /* the query of this row, decoded to double once */
        double q[ORA_IDX_HEADS][ORA_IDX_DIM];
        for (int h = 0; h < ORA_IDX_HEADS; ++h)
            for (int d = 0; d < ORA_IDX_DIM; ++d) {
                size_t off = ((size_t)r * ORA_IDX_HEADS + h) * ORA_IDX_DIM + d;
                if (q_bf16)
                    q[h][d] = bf16_to_double(q_bf16[off]);
                else
                    q[h][d] = oracle_e4m3_decode(q_e4m3[off]) *
                              (double)q_scale[(size_t)r * ORA_IDX_HEADS + h];
            }
        int row_status = ORA_OK;
#pragma omp parallel for schedule(static) reduction(max : row_status)
        for (int64_t s = 0; s < len; ++s) {
            int64_t page = block_table[(size_t)b * max_pages + s / ORA_PAGE];
            if (page < 0 || page >= num_pages) {
                row_status = ORA_BAD_PAGE;
                continue;
            }
            const uint8_t* pg = key_cache + (size_t)page * ORA_KEY_PAGE_BYTES;
            const uint8_t* kb = pg + (s % ORA_PAGE) * ORA_IDX_DIM;
            double ks = f32_at(pg + ORA_PAGE * ORA_IDX_DIM + (s % ORA_PAGE) * 4);
            double key[ORA_IDX_DIM];
            for (int d = 0; d < ORA_IDX_DIM; ++d) key[d] = oracle_e4m3_decode(kb[d]);
            double acc = 0.0;
            for (int h = 0; h < ORA_IDX_HEADS; ++h) {
                double dot = 0.0;
                for (int d = 0; d < ORA_IDX_DIM; ++d) dot += q[h][d] * key[d];
                double x = dot * ks;
                double relu = x > 0.0 ? x : 0.0;
                acc += (double)w[(size_t)r * ORA_IDX_HEADS + h] * relu;
            }
            scores[(size_t)r * ld + s] = acc;
        }
        if (row_status != ORA_OK) status = row_status;
    }
    return status;
}

/*
 * ---- MXFP4 index keys ----
 * [VLLM] "Hybrid KV cache without padding": an index key takes 68 bytes in
 * MXFP4 against 132 in FP8; "Native MXFP4 indexer": the 68 bytes include the
 * scales, the products are FP4 with FP32 accumulation and a weighted
 * reduction over heads; [AMD] quantization list: MXFP4 keeps one E8M0 scale
 * per 32 values.  128 dims = 64 bytes of 4-bit codes + 4 one-byte scales.
 * The element and scale encodings are those of the OCP Microscaling (MX)
 * specification v1.0; the pages name the format and nothing finer.
 */

/*
 * E2M1: one sign bit (bit 3), two exponent bits with bias 1, one mantissa
 * bit.  Exponent field 0 is subnormal (0 or 0.5); no infinities, no NaN.
 * The eight magnitudes are 0, 0.5, 1, 1.5, 2, 3, 4, 6.
 * Pinned by: the 16 codes against their closed form (golden table), the MX
 * cross-format identity with the E4M3 scorer.
 */
double oracle_e2m1_decode(uint8_t nibble) {
    const int sign = (nibble >> 3) & 1;
    const int e = (nibble >> 1) & 0x3;
    const int m = nibble & 0x1;
    const double mag = e == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return sign ? -mag : mag;
}

/*
 * E2M1 encoding: the nearest of the eight magnitudes, a tie going to the code
 * with an even mantissa bit, magnitudes above 6 saturating to 6 (the MX
 * conversion clamps to the element format's largest normal); the sign is
 * kept.  By brute force over the 8 non-negative codes.
 * Pinned by: the round trip over all 16 codes, every midpoint, saturation.
 */
uint8_t oracle_e2m1_encode(double x) {
    const int sign = signbit(x) ? 1 : 0;
    const double a = fabs(x);
    int best = 0;
    double bestd = INFINITY;
    for (int c = 0; c < 8; ++c) {
        const double d = fabs(a - oracle_e2m1_decode((uint8_t)c));
        if (d < bestd || (d == bestd && c % 2 == 0)) {
            best = c;
            bestd = d;
        }
    }
    return (uint8_t)((sign << 3) | best);
}

/*
 * E8M0: an unsigned exponent with bias 127, value 2^(code - 127); code 0xFF
 * is NaN.  Pinned by: every code against torch.float8_e8m0fnu where the
 * installed torch has it, and against ldexp otherwise.
 */
double oracle_e8m0_decode(uint8_t code) {
    if (code == 0xFF) return NAN;
    return ldexp(1.0, (int)code - 127);
}

/*
 * MX quantization of n values (n a multiple of 32), per block of 32:
 *   shared = floor(log2(max |v|)) - 2       (2 = E2M1's largest exponent)
 *   scale  = 2^shared as E8M0, shared clamped to [-127, 127]; an all-zero
 *            block takes shared = -127
 *   code_i = e2m1_encode(v_i / scale)        (saturating at 6)
 * Codes are packed two to a byte, element 2j in the low nibble of byte j.
 * Returns ORA_BAD_ARG if n is not a multiple of 32 or a value is not finite.
 * Pinned by: the scale exponent against frexp on random blocks, exactness on
 * values that are E2M1 times a power of two, the error bound
 * |v - dec(code) * scale| <= scale (and <= scale / 2 below 6 * scale).
 */
int oracle_mx_quantize(const double* v, int n, uint8_t* codes, uint8_t* scales) {
    if (n < 0 || n % ORA_MX_BLOCK != 0) return ORA_BAD_ARG;
    for (int i = 0; i < n; ++i)
        if (!isfinite(v[i])) return ORA_BAD_ARG;
    for (int b = 0; b < n / ORA_MX_BLOCK; ++b) {
        const double* vb = v + (size_t)b * ORA_MX_BLOCK;
        double amax = 0.0;
        for (int i = 0; i < ORA_MX_BLOCK; ++i)
            if (fabs(vb[i]) > amax) amax = fabs(vb[i]);
        int shared = -127;
        if (amax > 0.0) {
            shared = (int)floor(log2(amax)) - 2;
            if (shared < -127) shared = -127;
            if (shared > 127) shared = 127;
        }
        scales[b] = (uint8_t)(shared + 127);
        const double scale = ldexp(1.0, shared);
        for (int i = 0; i < ORA_MX_BLOCK; ++i) {
            const uint8_t c = oracle_e2m1_encode(vb[i] / scale);
            const int j = b * ORA_MX_BLOCK + i;
            if (j % 2 == 0)
                codes[j / 2] = c;
            else
                codes[j / 2] |= (uint8_t)(c << 4);
        }
    }
    return ORA_OK;
}

/* Element d of a packed MX vector, decoded with its block scale. */
static double mx_value(const uint8_t* codes, const uint8_t* scales, int d) {
    const uint8_t nib = (d % 2 == 0) ? (codes[d / 2] & 0xF) : (codes[d / 2] >> 4);
    return oracle_e2m1_decode(nib) * oracle_e8m0_decode(scales[d / ORA_MX_BLOCK]);
}

/*
 * The Write step for MXFP4 index keys: the LayerNorm of oracle_write_kv, then
 * mx_quantize of the 128 normalized values (no per-token scale: the block
 * scales replace it).  Page block_table[req][pos / 64], slot pos % 64 of
 * key_cache (ORA_MX_KEY_PAGE_BYTES per page): the 64 code bytes at slot * 64,
 * the 4 scale bytes at 64 * 64 + slot * 4.  The normalized key is returned in
 * key_pre [T][128] when non-NULL.  The latent row is written as in
 * oracle_write_kv (the two caches are quantized independently: [VLLM] "Hybrid
 * KV cache without padding").
 * Pinned by: the LayerNorm shared with the FP8 Write step (pinned there), the
 * bytes against mx_quantize of that LayerNorm's output, placement through a
 * shuffled block table.
 */
int oracle_write_key_mx(const uint16_t* k_raw, const double* gamma, const double* beta,
                        double eps, const int32_t* block_table, int B, int max_pages,
                        const int32_t* tok_req, const int32_t* tok_pos, int T,
                        uint8_t* key_cache, int64_t num_pages, double* key_pre) {
    if (T < 0 || !(eps >= 0.0)) return ORA_BAD_ARG;
    for (int t = 0; t < T; ++t) {
        const int req = tok_req[t], pos = tok_pos[t];
        if (req < 0 || req >= B || pos < 0 || pos >= max_pages * ORA_PAGE) return ORA_BAD_ARG;
        const int page = block_table[(size_t)req * max_pages + pos / ORA_PAGE];
        if (page < 0 || (int64_t)page >= num_pages) return ORA_BAD_PAGE;
        const int slot = pos % ORA_PAGE;
        double k[ORA_IDX_DIM];
        layer_norm_key(k_raw + (size_t)t * ORA_IDX_DIM, gamma, beta, eps, k);
        uint8_t* pg = key_cache + (size_t)page * ORA_MX_KEY_PAGE_BYTES;
        const int rc = oracle_mx_quantize(k, ORA_IDX_DIM, pg + (size_t)slot * ORA_MX_KEY_BYTES,
                                          pg + ORA_PAGE * ORA_MX_KEY_BYTES +
                                              (size_t)slot * ORA_MX_SCALES);
        if (rc != ORA_OK) return rc;
        if (key_pre) memcpy(key_pre + (size_t)t * ORA_IDX_DIM, k, sizeof k);
    }
    return ORA_OK;
}

/*
 * Lightning-indexer scores over MXFP4 keys with an MXFP4 query ([VLLM]
 * "Native MXFP4 indexer": FP4 products, FP32 accumulation, weighted reduction
 * across heads; the query front quantizes the query to FP8 or MXFP4 with the
 * head weights folded in).
 *
 *   score[r][s] = sum_{h<32} w[r][h] * max(0, sum_{d<128} q[r][h][d] * key[s][d])
 *
 * with q[r][h][d] = e2m1(qc[r][h] element d) * e8m0(qs[r][h][d / 32]) and
 * key[s][d] likewise from its page (codes at slot * 64, scales at 64 * 64 +
 * slot * 4).  The block scales are powers of two, so the FP8 form's per-token
 * scale inside the ReLU has no counterpart here.  qc is [R][32][64] bytes, qs
 * [R][32][4].  Entries s >= row_len[r] are left untouched.
 * Pinned by: the cross-format identity (keys and queries on the MX grid are
 * exactly representable as E4M3 times a power-of-two per-token scale, so the
 * FP8 scorer, pinned separately, must give the same scores), brute force of
 * one score from the golden E2M1 table, linearity in w, q = 0.
 */
int oracle_indexer_scores_mx(const uint8_t* qc, const uint8_t* qs, const float* w,
                             const uint8_t* key_cache, int64_t num_pages,
                             const int32_t* block_table, int B, int max_pages,
                             const int32_t* row_req, const int32_t* row_len, int R,
                             double* scores, int64_t ld) {
    int status = ORA_OK;
    for (int r = 0; r < R; ++r) {
        if (row_req[r] < 0 || row_req[r] >= B) return ORA_BAD_ARG;
        if (row_len[r] < 0 || (int64_t)row_len[r] > ld ||
            (int64_t)row_len[r] > (int64_t)max_pages * ORA_PAGE)
            return ORA_BAD_ARG;
    }
    for (int r = 0; r < R; ++r) {
        const int b = row_req[r];
        const int64_t len = row_len[r];
        double q[ORA_IDX_HEADS][ORA_IDX_DIM];
        for (int h = 0; h < ORA_IDX_HEADS; ++h) {
            const size_t rh = (size_t)r * ORA_IDX_HEADS + h;
            for (int d = 0; d < ORA_IDX_DIM; ++d)
                q[h][d] = mx_value(qc + rh * ORA_MX_KEY_BYTES, qs + rh * ORA_MX_SCALES, d);
        }
        int row_status = ORA_OK;
#pragma omp parallel for schedule(static) reduction(max : row_status)
        for (int64_t s = 0; s < len; ++s) {
            int64_t page = block_table[(size_t)b * max_pages + s / ORA_PAGE];
            if (page < 0 || page >= num_pages) {
                row_status = ORA_BAD_PAGE;
                continue;
            }
            const uint8_t* pg = key_cache + (size_t)page * ORA_MX_KEY_PAGE_BYTES;
            const int slot = (int)(s % ORA_PAGE);
            double key[ORA_IDX_DIM];
            for (int d = 0; d < ORA_IDX_DIM; ++d)
                key[d] = mx_value(pg + (size_t)slot * ORA_MX_KEY_BYTES,
                                  pg + ORA_PAGE * ORA_MX_KEY_BYTES + (size_t)slot * ORA_MX_SCALES,
                                  d);
            double acc = 0.0;
            for (int h = 0; h < ORA_IDX_HEADS; ++h) {
                double qk = 0.0;
                for (int d = 0; d < ORA_IDX_DIM; ++d) qk += q[h][d] * key[d];
                acc += (double)w[(size_t)r * ORA_IDX_HEADS + h] * (qk > 0.0 ? qk : 0.0);
            }
            scores[(size_t)r * ld + s] = acc;
        }
        if (row_status != ORA_OK) status = row_status;
    }
    return status;
}

/* (score descending, token index ascending) */
typedef struct {
    double score;
    int32_t index;
} ora_item;

static int ora_item_cmp(const void* a, const void* b) {
    const ora_item* x = (const ora_item*)a;
    const ora_item* y = (const ora_item*)b;
    if (x->score > y->score) return -1;
    if (x->score < y->score) return 1;
    return (x->index > y->index) - (x->index < y->index);
}

/*
 * Top-k selection ([SGL] "What's new": attention reads only the top 2,048;
 * [TS] step 3 "Select": keep the k highest-scoring positions per query).
 * Per row: order the visible tokens 0..row_len[r]-1 by score descending, ties
 * to the lower token index, take the first min(k, row_len[r]) and pad the
 * rest of idx[r][0..k) with -1.  Output is in that rank order.  -0.0 and
 * +0.0 compare equal (IEEE), so they tie and the lower index wins.
 * Pinned by: numpy.lexsort brute force, k >= len, all-equal scores.
 */
int oracle_topk(const double* scores, int64_t ld, const int32_t* row_len, int R, int k,
                int32_t* idx) {
    if (k < 0) return ORA_BAD_ARG;
    for (int r = 0; r < R; ++r)
        if (row_len[r] < 0 || (int64_t)row_len[r] > ld) return ORA_BAD_ARG;
#pragma omp parallel for schedule(dynamic, 1)
    for (int r = 0; r < R; ++r) {
        const int64_t len = row_len[r];
        ora_item* items = (ora_item*)malloc(sizeof(ora_item) * (size_t)(len > 0 ? len : 1));
        for (int64_t s = 0; s < len; ++s) {
            items[s].score = scores[(size_t)r * ld + s];
            items[s].index = (int32_t)s;
        }
        qsort(items, (size_t)len, sizeof(ora_item), ora_item_cmp);
        for (int j = 0; j < k; ++j)
            idx[(size_t)r * k + j] = (j < len) ? items[j].index : -1;
        free(items);
    }
    return ORA_OK;
}

/*
 * Top-k by the decode-context-parallel exchange ([SGL] "Decode: DSA with
 * decode context parallelism": token p lives on GPU p mod W, each GPU ranks
 * its own tokens, shares its best candidates, takes the k-th best shared
 * score as the cutoff, and a GPU whose candidates all beat the cutoff has its
 * full local top-k read; [VLLM] "An exact top-k merge with about 10x less
 * traffic": 1.5 k / W candidates per GPU, a resend when a GPU may hold more
 * winners than it sent).  The W shards are taken in turn here.  Per row, in
 * the order of oracle_topk (score descending, token index ascending):
 *   1. shard s owns tokens p < row_len with p % W == s (n_s of them) and
 *      orders them; its local top-k is its first min(k, n_s) tokens;
 *   2. it sends its first min(c, n_s) tokens, c = ceil(1.5 k / W);
 *   3. the cutoff E is the k-th of all sent tokens in the order (there is no
 *      cutoff when fewer than k were sent);
 *   4. shard s may hide winners when it kept tokens back (n_s > c) and there
 *      is no cutoff or its c-th token precedes E (a token it kept back comes
 *      after its c-th in the order, so otherwise it comes after E); the full
 *      local top-k of such a shard is gathered;
 *   5. the result is the top-k of the gathered tokens (the sent ones and the
 *      resent local top-ks).
 * idx[r][0..k) receives it in rank order, -1 padded; resend[r] has bit s set
 * when shard s's local top-k was gathered.
 * Pinned by: equality with oracle_topk on random, tied, short and
 * shard-concentrated rows for several W; the resend pattern of rows built so
 * that one shard holds every winner, none does, or all tie.
 */
int oracle_topk_dcp(const double* scores, int64_t ld, const int32_t* row_len, int R, int k,
                    int W, int32_t* idx, uint32_t* resend) {
    if (k < 1 || W < 1 || W > 32) return ORA_BAD_ARG;
    for (int r = 0; r < R; ++r)
        if (row_len[r] < 0 || (int64_t)row_len[r] > ld) return ORA_BAD_ARG;
    const int64_t c = (3 * (int64_t)k + 2 * W - 1) / (2 * W);
#pragma omp parallel for schedule(dynamic, 1)
    for (int r = 0; r < R; ++r) {
        const int64_t len = row_len[r];
        const double* row = scores + (size_t)r * ld;
        ora_item* all = (ora_item*)malloc(sizeof(ora_item) * (size_t)(len > 0 ? len : 1));
        ora_item* sent = (ora_item*)malloc(sizeof(ora_item) * (size_t)(len > 0 ? len : 1));
        ora_item* gathered = (ora_item*)malloc(sizeof(ora_item) * (size_t)(len > 0 ? len : 1));
        int64_t start[33], n[32];
        /* 1. each shard's own tokens, ordered (stored one shard after the other) */
        int64_t off = 0;
        for (int s = 0; s < W; ++s) {
            start[s] = off;
            n[s] = 0;
            for (int64_t p = s; p < len; p += W) {
                all[off + n[s]].score = row[p];
                all[off + n[s]].index = (int32_t)p;
                ++n[s];
            }
            qsort(all + off, (size_t)n[s], sizeof(ora_item), ora_item_cmp);
            off += n[s];
        }
        /* 2. the sent candidates; 3. the cutoff */
        int64_t nsent = 0;
        for (int s = 0; s < W; ++s)
            for (int64_t j = 0; j < n[s] && j < c; ++j) sent[nsent++] = all[start[s] + j];
        qsort(sent, (size_t)nsent, sizeof(ora_item), ora_item_cmp);
        const int has_cut = nsent >= k;
        ora_item cut = {0.0, 0};
        if (has_cut) cut = sent[k - 1];
        /* 4. shards that may hide winners */
        uint32_t mask = 0;
        for (int s = 0; s < W; ++s)
            if (n[s] > c && (!has_cut || ora_item_cmp(&all[start[s] + c - 1], &cut) < 0))
                mask |= 1u << s;
        /* 5. the top-k of everything gathered */
        int64_t ng = 0;
        for (int s = 0; s < W; ++s) {
            const int64_t m = ((mask >> s) & 1u) ? (n[s] < k ? n[s] : k) : (n[s] < c ? n[s] : c);
            for (int64_t j = 0; j < m; ++j) gathered[ng++] = all[start[s] + j];
        }
        qsort(gathered, (size_t)ng, sizeof(ora_item), ora_item_cmp);
        for (int j = 0; j < k; ++j)
            idx[(size_t)r * k + j] = (j < len && j < ng) ? gathered[j].index : -1;
        resend[r] = mask;
        free(all);
        free(sent);
        free(gathered);
    }
    return ORA_OK;
}

/*
 * Sparse MLA over the selected latent rows ([VLLM] "What Kimi K3.1 Pro
 * changes": MLA attention runs exactly over only those tokens; [TS] "Sparse
 * attention in Kimi K3.1 Pro": every attention head attends to the selected
 * tokens; [AMD] overview "MLA": the 576-wide latent is 512 compressed KV +
 * 64 RoPE dims, the 512 part serving as the value).  MQA form: one latent
 * row per token is shared by all H heads.
 *
 * For row r, head h, and the valid selected tokens j (idx[r][j] >= 0):
 *   L[j][:]  = dec(latent8[token_j][:]) * latent_scale
 *   x_j      = softmax_scale * sum_{d<576} q[r][h][d] * L[j][d]
 *   m        = max_j x_j ;  p_j = exp(x_j - m) ;  Z = sum_j p_j
 *   out[r][h][:] = (sum_j p_j * L[j][0:512]) / Z ;  lse[r][h] = m + ln Z
 * With no valid token the output is 0 and lse is -inf.
 * Latent page layout: [page][64 tokens][576 bytes]; token s of request b is
 * in page block_table[b][s / 64], slot s % 64.
 * Pinned by: float64 scaled_dot_product_attention on the dense case, one
 * selected token, q = 0, split/unsplit LSE merge.
 */
int oracle_sparse_mla(const uint16_t* q, int H, double softmax_scale, const uint8_t* latent_cache,
                      int64_t num_pages, double latent_scale, const int32_t* block_table, int B,
                      int max_pages, const int32_t* row_req, const int32_t* row_len,
                      const int32_t* idx, int k, int R, double* out, double* lse) {
    if (H <= 0 || k < 0) return ORA_BAD_ARG;
    for (int r = 0; r < R; ++r) {
        if (row_req[r] < 0 || row_req[r] >= B) return ORA_BAD_ARG;
        if (row_len[r] < 0 || (int64_t)row_len[r] > (int64_t)max_pages * ORA_PAGE)
            return ORA_BAD_ARG;
        for (int j = 0; j < k; ++j) {
            int32_t t = idx[(size_t)r * k + j];
            if (t >= row_len[r]) return ORA_BAD_INDEX;
            if (t >= 0) {
                int64_t page = block_table[(size_t)row_req[r] * max_pages + t / ORA_PAGE];
                if (page < 0 || page >= num_pages) return ORA_BAD_PAGE;
            }
        }
    }
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int r = 0; r < R; ++r) {
        for (int h = 0; h < H; ++h) {
            const int b = row_req[r];
            double qh[ORA_LAT_DIM];
            for (int d = 0; d < ORA_LAT_DIM; ++d)
                qh[d] = bf16_to_double(q[((size_t)r * H + h) * ORA_LAT_DIM + d]);
            double* x = (double*)malloc(sizeof(double) * (size_t)(k > 0 ? k : 1));
            double m = -INFINITY;
            int any = 0;
            for (int j = 0; j < k; ++j) {
                int32_t t = idx[(size_t)r * k + j];
                if (t < 0) continue;
                int64_t page = block_table[(size_t)b * max_pages + t / ORA_PAGE];
                const uint8_t* row =
                    latent_cache + ((size_t)page * ORA_PAGE + (size_t)(t % ORA_PAGE)) * ORA_LAT_DIM;
                double dot = 0.0;
                for (int d = 0; d < ORA_LAT_DIM; ++d)
                    dot += qh[d] * (oracle_e4m3_decode(row[d]) * latent_scale);
                x[j] = softmax_scale * dot;
                if (x[j] > m) m = x[j];
                any = 1;
            }
            double* o = out + ((size_t)r * H + h) * ORA_V_DIM;
            for (int d = 0; d < ORA_V_DIM; ++d) o[d] = 0.0;
            if (!any) {
                if (lse) lse[(size_t)r * H + h] = -INFINITY;
                free(x);
                continue;
            }
            double Z = 0.0;
            for (int j = 0; j < k; ++j) {
                int32_t t = idx[(size_t)r * k + j];
                if (t < 0) continue;
                int64_t page = block_table[(size_t)b * max_pages + t / ORA_PAGE];
                const uint8_t* row =
                    latent_cache + ((size_t)page * ORA_PAGE + (size_t)(t % ORA_PAGE)) * ORA_LAT_DIM;
                double p = exp(x[j] - m);
                Z += p;
                for (int d = 0; d < ORA_V_DIM; ++d)
                    o[d] += p * (oracle_e4m3_decode(row[d]) * latent_scale);
            }
            for (int d = 0; d < ORA_V_DIM; ++d) o[d] /= Z;
            if (lse) lse[(size_t)r * H + h] = m + log(Z);
            free(x);
        }
    }
    return ORA_OK;
}

/*
 * ---- NVFP4 latent ----
 * [VLLM] "Hybrid KV cache without padding": the MLA latent takes 352 bytes
 * per token in NVFP4 against 576 in FP8; "What Kimi K3.1 Pro changes":
 * FlashInfer's kernels serve an NVFP4 latent.  The pages give the size only.
 * NVFP4 (NVIDIA's 4-bit format): E2M1 elements, one unsigned E4M3 scale per
 * 16 elements, and a per-tensor fp32 scale (here the cache's latent_scale).
 * The 352 bytes are read as the 512 compressed-KV dims in NVFP4 (256 code
 * bytes + 32 scale bytes) and the 64 RoPE dims in E4M3 (64 bytes):
 *   row = [codes: 256 B, dim 2j in the low nibble of byte j]
 *         [block scales: 32 B, byte b scales dims 16b .. 16b + 15]
 *         [RoPE: 64 E4M3 bytes, dims 512 .. 575]
 */
#define ORA_NV_BLOCK 16
#define ORA_NV_ROW_BYTES (ORA_V_DIM / 2 + ORA_V_DIM / ORA_NV_BLOCK + (ORA_LAT_DIM - ORA_V_DIM))

/*
 * Decodes one NVFP4 latent row into its 576 real values:
 *   L[d]        = e2m1(code d) * e4m3(scale[d / 16]) * latent_scale   (d < 512)
 *   L[512 + j]  = e4m3(rope[j]) * latent_scale                          (j < 64)
 * The scale byte is an unsigned E4M3 (its top bit is ignored).
 * Pinned by: rows on the shared grid equal the FP8 row's decode exactly (the
 * NVFP4 MLA then equals the pinned FP8 MLA), and the last dims of each part.
 */
void oracle_nvfp4_latent_decode(const uint8_t* row, double latent_scale, double* L) {
    const uint8_t* codes = row;
    const uint8_t* scales = row + ORA_V_DIM / 2;
    const uint8_t* rope = scales + ORA_V_DIM / ORA_NV_BLOCK;
    for (int d = 0; d < ORA_V_DIM; ++d) {
        const uint8_t nib = (d % 2 == 0) ? (codes[d / 2] & 0xF) : (codes[d / 2] >> 4);
        L[d] = oracle_e2m1_decode(nib) * oracle_e4m3_decode(scales[d / ORA_NV_BLOCK] & 0x7F) *
               latent_scale;
    }
    for (int j = 0; j < ORA_LAT_DIM - ORA_V_DIM; ++j)
        L[ORA_V_DIM + j] = oracle_e4m3_decode(rope[j]) * latent_scale;
}

/*
 * NVFP4 quantization of one latent row (576 values already divided by the
 * per-tensor scale): per block of 16 of the first 512 dims
 *   s      = e4m3_encode(max |v| / 6)     (the block maximum onto E2M1's 6)
 *   codes  = e2m1_encode(v / dec(s))       (all zero when dec(s) is 0)
 * and the 64 RoPE dims as e4m3_encode(v).  Writes ORA_NV_ROW_BYTES bytes.
 * Pinned by: exactness on the shared grid, the block error bound.
 */
void oracle_nvfp4_latent_encode(const double* v, uint8_t* row) {
    uint8_t* codes = row;
    uint8_t* scales = row + ORA_V_DIM / 2;
    uint8_t* rope = scales + ORA_V_DIM / ORA_NV_BLOCK;
    memset(codes, 0, ORA_V_DIM / 2);
    for (int b = 0; b < ORA_V_DIM / ORA_NV_BLOCK; ++b) {
        double amax = 0.0;
        for (int i = 0; i < ORA_NV_BLOCK; ++i) {
            const double a = fabs(v[b * ORA_NV_BLOCK + i]);
            if (a > amax) amax = a;
        }
        scales[b] = oracle_e4m3_encode(amax / 6.0);
        const double s = oracle_e4m3_decode(scales[b]);
        for (int i = 0; i < ORA_NV_BLOCK; ++i) {
            const int d = b * ORA_NV_BLOCK + i;
            const uint8_t c = s > 0.0 ? oracle_e2m1_encode(v[d] / s) : 0;
            codes[d / 2] |= (uint8_t)(d % 2 == 0 ? c : c << 4);
        }
    }
    for (int j = 0; j < ORA_LAT_DIM - ORA_V_DIM; ++j) rope[j] = oracle_e4m3_encode(v[ORA_V_DIM + j]);
}

/*
 * Sparse MLA over NVFP4 latent rows: the attention of oracle_sparse_mla with
 * each selected row decoded by oracle_nvfp4_latent_decode.  Latent page
 * layout: [page][64 tokens][352 bytes].
 * Pinned by: equality with oracle_sparse_mla on rows both formats represent
 * exactly, the dense case against float64 scaled_dot_product_attention.
 */
int oracle_sparse_mla_nvfp4(const uint16_t* q, int H, double softmax_scale,
                            const uint8_t* latent_cache, int64_t num_pages, double latent_scale,
                            const int32_t* block_table, int B, int max_pages,
                            const int32_t* row_req, const int32_t* row_len, const int32_t* idx,
                            int k, int R, double* out, double* lse) {
    if (H <= 0 || k < 0) return ORA_BAD_ARG;
    for (int r = 0; r < R; ++r) {
        if (row_req[r] < 0 || row_req[r] >= B) return ORA_BAD_ARG;
        if (row_len[r] < 0 || (int64_t)row_len[r] > (int64_t)max_pages * ORA_PAGE)
            return ORA_BAD_ARG;
        for (int j = 0; j < k; ++j) {
            int32_t t = idx[(size_t)r * k + j];
            if (t >= row_len[r]) return ORA_BAD_INDEX;
            if (t >= 0) {
                int64_t page = block_table[(size_t)row_req[r] * max_pages + t / ORA_PAGE];
                if (page < 0 || page >= num_pages) return ORA_BAD_PAGE;
            }
        }
    }
#pragma omp parallel for schedule(dynamic, 1)
    for (int r = 0; r < R; ++r) {
        const int b = row_req[r];
        /* the selected rows of this query row, decoded once for all heads */
        double* L = (double*)malloc(sizeof(double) * (size_t)(k > 0 ? k : 1) * ORA_LAT_DIM);
        double* x = (double*)malloc(sizeof(double) * (size_t)(k > 0 ? k : 1));
        for (int j = 0; j < k; ++j) {
            int32_t t = idx[(size_t)r * k + j];
            if (t < 0) continue;
            int64_t page = block_table[(size_t)b * max_pages + t / ORA_PAGE];
            oracle_nvfp4_latent_decode(
                latent_cache + ((size_t)page * ORA_PAGE + (size_t)(t % ORA_PAGE)) * ORA_NV_ROW_BYTES,
                latent_scale, L + (size_t)j * ORA_LAT_DIM);
        }
        for (int h = 0; h < H; ++h) {
            double qh[ORA_LAT_DIM];
            for (int d = 0; d < ORA_LAT_DIM; ++d)
                qh[d] = bf16_to_double(q[((size_t)r * H + h) * ORA_LAT_DIM + d]);
            double m = -INFINITY;
            int any = 0;
            for (int j = 0; j < k; ++j) {
                if (idx[(size_t)r * k + j] < 0) continue;
                double s = 0.0;
                for (int d = 0; d < ORA_LAT_DIM; ++d) s += qh[d] * L[(size_t)j * ORA_LAT_DIM + d];
                x[j] = softmax_scale * s;
                if (x[j] > m) m = x[j];
                any = 1;
            }
            double* o = out + ((size_t)r * H + h) * ORA_V_DIM;
            for (int d = 0; d < ORA_V_DIM; ++d) o[d] = 0.0;
            if (!any) {
                if (lse) lse[(size_t)r * H + h] = -INFINITY;
                continue;
            }
            double Z = 0.0;
            for (int j = 0; j < k; ++j) {
                if (idx[(size_t)r * k + j] < 0) continue;
                const double pj = exp(x[j] - m);
                Z += pj;
                for (int d = 0; d < ORA_V_DIM; ++d) o[d] += pj * L[(size_t)j * ORA_LAT_DIM + d];
            }
            for (int d = 0; d < ORA_V_DIM; ++d) o[d] /= Z;
            if (lse) lse[(size_t)r * H + h] = log(Z) + m;
        }
        free(L);
        free(x);
    }
    return ORA_OK;
}
