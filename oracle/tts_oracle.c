/*
 * CPU oracle for the batched codec-LM decode step.  TEST INFRASTRUCTURE ONLY:
 * it is called by the tests, by the smoke check and by the benchmark's CPU
 * baseline, never by the product path, and it shares no code with the CUDA
 * library.
 *
 * Plain loops, one stream at a time, sums in double.  Values the method keeps
 * as fp32 (logits, probabilities, Gumbel keys) are rounded to float before a
 * decision is taken on them, so that an argmax or an accept test is decided in
 * the precision the kernels use.  Inputs are read as stored (fp32, or bf16 bit
 * patterns upcast exactly).
 *
 * Sources (web pages on streaming codec-LM text-to-speech):
 *  [OPT]  "Optimizing Streaming Text-to-Speech Models for Sub-50 Millisecond
 *         Latency": section "Speculative Decoding for Acoustic Tokens"
 *         (verify_draft_tokens) and section "Dynamic Token-Level Batching"
 *         (static pool of 16-token KV blocks).
 *  [TTS]  "TTS (Text-to-Speech) Serving, in depth", section "Token generation
 *         under a frame budget" (one decode step per frame reads the KV cache).
 *  [TON]  "TontaubeV1: Streaming Text-to-Speech with Hierarchical Codec
 *         Modeling and Bounded Context", section 3 (codebooks of 16,384 and
 *         4,096 entries, boundary token, later stages at temperature zero).
 *  [SAL]  Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as
 *         1, 2, 3", SC'11: the Philox4x64-10 bijection.
 *  [NAR]  "How We Made a TTS Model Respond in Sub-50 ms" (the code predictor's
 *         fixed loop and its captured graph).
 *  [MIS]  Misra, "Mish: A Self Regularized Non-Monotonic Activation Function"
 *         (2019): Mish(x) = x tanh(ln(1 + e^x)).
 *
 * Readings where the pages are silent (each is also listed in the design
 * notes): softmax scale 1/sqrt(D); query head h uses KV head h/(Hq/Hkv); the
 * appended token attends to itself; in a q_len-row verify block row j sees the
 * prefix and new tokens 0..j; the boundary token is vocab index V-1; equal
 * keys resolve to the lowest index; the rejection draw samples the clamped
 * residual by Gumbel-max; with every draft accepted no bonus token is drawn
 * unless asked for; the two-layer audio head's intermediate is rounded to
 * bfloat16 once (the precision its second product reads) and its layers'
 * biases are optional; a stage's structural tokens are the last ids of its
 * vocabulary, each allowed per row by one mask bit.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_BLOCK 16

/* ------------------------------------------------------------------ inputs */

static double load_elem(const void *base, size_t i, int is_bf16) {
    if (is_bf16) {
        uint32_t bits = (uint32_t)((const uint16_t *)base)[i] << 16;
        float f;
        memcpy(&f, &bits, sizeof f);
        return (double)f;
    }
    return (double)((const float *)base)[i];
}

/* ------------------------------------------------------------------ Philox */

/* Philox4x64 with 10 rounds [SAL, section 5]: each round multiplies words 0
 * and 2 by fixed 64-bit multipliers, keeps the low halves as the new words 3
 * and 1, and xors the high halves with the other two words and the round key.
 * The key is bumped by the Weyl constants between rounds. */
void orc_philox4x64_10(const uint64_t ctr[4], const uint64_t key[2], uint64_t out[4]) {
    const uint64_t M0 = 0xD2E7470EE14C6C93ULL, M1 = 0xCA5A826395121157ULL;
    const uint64_t W0 = 0x9E3779B97F4A7C15ULL, W1 = 0xBB67AE8584CAA73BULL;
    uint64_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
    uint64_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        unsigned __int128 p0 = (unsigned __int128)M0 * x0;
        unsigned __int128 p1 = (unsigned __int128)M1 * x2;
        uint64_t hi0 = (uint64_t)(p0 >> 64), lo0 = (uint64_t)p0;
        uint64_t hi1 = (uint64_t)(p1 >> 64), lo1 = (uint64_t)p1;
        uint64_t y0 = hi1 ^ x1 ^ k0;
        uint64_t y1 = lo1;
        uint64_t y2 = hi0 ^ x3 ^ k1;
        uint64_t y3 = lo0;
        x0 = y0; x1 = y1; x2 = y2; x3 = y3;
        k0 += W0;
        k1 += W1;
    }
    out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

/* Uniform number idx of the stream named by (seed, step, tag, pos).
 * Key = (seed, step); counter = (idx / 8, tag, pos, 0).  One Philox call gives
 * four 64-bit words = eight 32-bit halves; half (idx % 8) is used, word
 * (idx % 8) / 2, low half first.  Its top 23 bits k map to (2k + 1) / 2^24,
 * which is exact in fp32 and lies strictly inside (0, 1).
 * Tags: 0 head Gumbel noise, 1 verify accept uniforms, 2 verify residual /
 * bonus Gumbel noise. */
float orc_uniform(uint64_t seed, uint64_t step, uint32_t tag, uint32_t pos, uint32_t idx) {
    const uint64_t ctr[4] = {idx / 8u, tag, pos, 0};
    const uint64_t key[2] = {seed, step};
    uint64_t w[4];
    orc_philox4x64_10(ctr, key, w);
    const uint32_t lane = idx % 8u;
    const uint64_t word = w[lane / 2u];
    const uint32_t half = (lane & 1u) ? (uint32_t)(word >> 32) : (uint32_t)word;
    const uint32_t k = half >> 9;
    return (float)(2u * k + 1u) * 0x1.0p-24f;
}

/* Standard Gumbel noise G = -log(-log u), in fp32. */
float orc_gumbel(uint64_t seed, uint64_t step, uint32_t tag, uint32_t pos, uint32_t idx) {
    const float u = orc_uniform(seed, step, tag, pos, idx);
    return -logf(-logf(u));
}

/* ------------------------------------------------------------------ append */

/* [OPT, "Dynamic Token-Level Batching"]: the KV cache is a static pool of
 * 16-token blocks; a stream's logical token s lives in physical block
 * table[b][s / 16], slot s % 16.  Pool layout [num_blocks][Hkv][16][D].
 * New token j of stream b goes to logical slot ctx_before[b] + j.
 * Returns 0, or -1 if a slot falls outside the table or the pool. */
int orc_kv_append(int num_blocks, int Hkv, int D, int elem_bytes, void *k_pool, void *v_pool,
                  const int32_t *block_table, int max_blocks, const int32_t *ctx_before,
                  int B, int q_len, const void *k_new, const void *v_new) {
    const size_t row = (size_t)D * (size_t)elem_bytes;
    for (int b = 0; b < B; ++b) {
        for (int j = 0; j < q_len; ++j) {
            const int s = ctx_before[b] + j;
            if (s < 0 || s / ORC_BLOCK >= max_blocks) return -1;
            const int blk = block_table[(size_t)b * max_blocks + s / ORC_BLOCK];
            if (blk < 0 || blk >= num_blocks) return -1;
            for (int g = 0; g < Hkv; ++g) {
                const size_t dst = (((size_t)blk * Hkv + g) * ORC_BLOCK + s % ORC_BLOCK) * row;
                const size_t src = (((size_t)b * q_len + j) * Hkv + g) * row;
                memcpy((char *)k_pool + dst, (const char *)k_new + src, row);
                memcpy((char *)v_pool + dst, (const char *)v_new + src, row);
            }
        }
    }
    return 0;
}

/* --------------------------------------------------------------- attention */

/* Element d of the cached key (is_v = 0) or value (is_v = 1) row of token slot
 * `slot` of KV head g in physical block blk. */
typedef double (*orc_kv_loader)(const void *ctx, int is_v, int blk, int g, int slot, int d);

typedef struct {
    int Hkv, D, is_bf16;
    const void *k_pool, *v_pool;
} orc_plain_pool;

static double plain_kv(const void *ctx, int is_v, int blk, int g, int slot, int d) {
    const orc_plain_pool *p = (const orc_plain_pool *)ctx;
    const size_t off = (((size_t)blk * p->Hkv + g) * ORC_BLOCK + slot) * p->D + d;
    return load_elem(is_v ? p->v_pool : p->k_pool, off, p->is_bf16);
}

static int attend(int num_blocks, int Hkv, int D, orc_kv_loader kv, const void *ctx,
                  const int32_t *block_table, int max_blocks, const int32_t *ctx_lens,
                  int B, int q_len, int Hq, double scale, int causal,
                  const void *q, int q_is_bf16, double *out) {
    const int group = Hq / Hkv;
    double *s = (double *)malloc(sizeof(double) * (size_t)max_blocks * ORC_BLOCK);
    if (!s) return -1;
    for (int b = 0; b < B; ++b) {
        const int L = ctx_lens[b];
        if (L < q_len || L > max_blocks * ORC_BLOCK) { free(s); return -1; }
        for (int j = 0; j < q_len; ++j) {
            const int limit = causal ? L - q_len + j + 1 : L;
            for (int h = 0; h < Hq; ++h) {
                const int g = h / group;
                const size_t qoff = (((size_t)b * q_len + j) * Hq + h) * D;
                double m = -INFINITY;
                for (int t = 0; t < limit; ++t) {
                    const int blk = block_table[(size_t)b * max_blocks + t / ORC_BLOCK];
                    if (blk < 0 || blk >= num_blocks) { free(s); return -1; }
                    double dot = 0.0;
                    for (int d = 0; d < D; ++d)
                        dot += load_elem(q, qoff + d, q_is_bf16) * kv(ctx, 0, blk, g, t % ORC_BLOCK, d);
                    s[t] = scale * dot;
                    if (s[t] > m) m = s[t];
                }
                double denom = 0.0;
                for (int t = 0; t < limit; ++t) {
                    s[t] = exp(s[t] - m);
                    denom += s[t];
                }
                double *o = out + qoff;
                for (int d = 0; d < D; ++d) o[d] = 0.0;
                for (int t = 0; t < limit; ++t) {
                    const int blk = block_table[(size_t)b * max_blocks + t / ORC_BLOCK];
                    const double p = s[t] / denom;
                    for (int d = 0; d < D; ++d) o[d] += p * kv(ctx, 1, blk, g, t % ORC_BLOCK, d);
                }
            }
        }
    }
    free(s);
    return 0;
}

/* One decode step's attention [TTS, "Token generation under a frame budget"]:
 * every query row of stream b attends over that stream's cached keys/values
 * (gathered through the block table), softmax(scale * q.k) weighted sum of v.
 * ctx_lens[b] counts tokens after the append.  Query row j of a q_len-row
 * block sees tokens t < ctx_lens[b] - q_len + j + 1 when causal, all
 * ctx_lens[b] tokens otherwise.  GQA: query head h reads KV head
 * h / (Hq / Hkv).  Output out[B][q_len][Hq][D] in double.
 * Returns 0, or -1 on an invalid block id or context length. */
int orc_decode_attn(int num_blocks, int Hkv, int D, int is_bf16,
                    const void *k_pool, const void *v_pool,
                    const int32_t *block_table, int max_blocks, const int32_t *ctx_lens,
                    int B, int q_len, int Hq, double scale, int causal,
                    const void *q, double *out) {
    const orc_plain_pool pool = {Hkv, D, is_bf16, k_pool, v_pool};
    return attend(num_blocks, Hkv, D, plain_kv, &pool, block_table, max_blocks, ctx_lens, B, q_len, Hq,
                  scale, causal, q, is_bf16, out);
}

/* ------------------------------------------------------------------- RoPE */

/* Rotary position embedding (Su et al., "RoFormer: Enhanced Transformer with
 * Rotary Position Embedding", 2021, section 3.4, in the rotate-half
 * arrangement that pairs dimension i with i + D/2), fused with the KV cache
 * write on the pages ("Optimizing Streaming Text-to-Speech Models for Sub-50
 * Millisecond Latency", section "Engine-Level Optimizations with
 * TensorRT-LLM").  Row r (D values, bf16 or fp32 input) at position pos[r]:
 * for i < D/2 with angle a = pos * base^(-2i/D),
 *   out[i]       = x[i] cos a - x[i + D/2] sin a
 *   out[i + D/2] = x[i + D/2] cos a + x[i] sin a,
 * in double, rounded to float. */
void orc_rope_rows(const void *x, int is_bf16, int rows, int D, const int32_t *pos, double base, float *out) {
    const int h = D / 2;
    for (int r = 0; r < rows; ++r) {
        for (int i = 0; i < h; ++i) {
            const double a = (double)pos[r] * pow(base, -2.0 * i / D);
            const double c = cos(a), sn = sin(a);
            const double x1 = load_elem(x, (size_t)r * D + i, is_bf16);
            const double x2 = load_elem(x, (size_t)r * D + i + h, is_bf16);
            out[(size_t)r * D + i] = (float)(x1 * c - x2 * sn);
            out[(size_t)r * D + i + h] = (float)(x2 * c + x1 * sn);
        }
    }
}

/* ---------------------------------------------------------------- FP8 cache */

/* FP8 E4M3 ("e4m3fn"): 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits,
 * no infinities; exponent and mantissa all ones (0x7F / 0xFF) is NaN, so the
 * largest finite magnitude is 1.75 * 2^8 = 448; exponent field 0 holds the
 * subnormals m * 2^-9. */
float orc_e4m3_decode(uint8_t c) {
    const int sign = c >> 7, e = (c >> 3) & 15, m = c & 7;
    if (e == 15 && m == 7) return NAN;
    const double mag = e == 0 ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
    return (float)(sign ? -mag : mag);
}

/* Nearest E4M3 value to x, ties to the code with an even mantissa, magnitudes
 * above 448 saturating to +-448 (the largest finite value); NaN -> 0x7F.
 * Written as a search over the 127 non-negative finite codes. */
uint8_t orc_e4m3_encode(float x) {
    if (x != x) return 0x7F;
    const double a = fabs((double)x);
    int best = 0;
    double best_err = INFINITY;
    for (int c = 0; c <= 0x7E; ++c) {
        const double err = fabs((double)orc_e4m3_decode((uint8_t)c) - a);
        if (err < best_err || (err == best_err && (c & 1) == 0)) {
            best = c;
            best_err = err;
        }
    }
    return (uint8_t)((x < 0.0f ? 0x80 : 0) | best);
}

void orc_e4m3_encode_n(const float *x, size_t n, uint8_t *out) {
    for (size_t i = 0; i < n; ++i) out[i] = orc_e4m3_encode(x[i]);
}

void orc_e4m3_decode_n(const uint8_t *c, size_t n, float *out) {
    for (size_t i = 0; i < n; ++i) out[i] = orc_e4m3_decode(c[i]);
}

/* Byte of token slot s within a dimension's 16 value codes: the slot order
 * 0 1 8 9 2 3 10 11 4 5 12 13 6 7 14 15 (a storage-order choice of the cache
 * layout, not part of the arithmetic). */
static int v_pos(int s) { return 4 * ((s % 8) / 2) + (s % 2) + 2 * (s / 8); }

/* Quantises one row of n values: scale = max|x| / 448 (fp32), codes =
 * E4M3(x / scale) computed in fp32; an all-zero row gets scale 0 and codes 0. */
static float quantize_row(const float *x, int n, uint8_t *codes) {
    float amax = 0.0f;
    for (int d = 0; d < n; ++d) {
        const float a = fabsf(x[d]);
        if (a > amax) amax = a;
    }
    const float scale = amax / 448.0f;
    for (int d = 0; d < n; ++d) codes[d] = scale > 0.0f ? orc_e4m3_encode(x[d] / scale) : 0;
    return scale;
}

/* Storage of one (block, KV head) tile of an FP8 cache (D = 128), 4224 bytes:
 * key codes, token slot s and dimension d at byte 128 s + 16 ((d / 16) xor
 * (s % 8)) + d % 16; value codes, dimension d and slot s at byte
 * 2048 + 16 d + v_pos(s); the 16 key scales (fp32) at byte 4096, the 16 value
 * scales at byte 4160.  (A storage-order choice of the cache layout.) */
#define ORC_FP8_TILE 4224
static size_t k_byte(int s, int d) { return (size_t)(128 * s + 16 * ((d / 16) ^ (s % 8)) + d % 16); }
static size_t v_byte(int s, int d) { return (size_t)(2048 + 16 * d + v_pos(s)); }

/* KV append into an FP8 cache (the KV cache in FP8: "Optimizing Streaming
 * Text-to-Speech Models for Sub-50 Millisecond Latency", section
 * "Engine-Level Optimizations with TensorRT-LLM").  Each new key and value row
 * (one token, one KV head: D = 128 values, bf16 or fp32 as rows_are_bf16
 * says) is one quantisation block
 * with its own fp32 scale, stored in the tile layout above; tiles
 * [num_blocks][Hkv][4224 bytes].  Returns 0, or -1 if a slot falls outside
 * the table or the pool, or D != 128. */
int orc_kv_append_fp8(int num_blocks, int Hkv, int D, uint8_t *tiles, const int32_t *block_table,
                      int max_blocks, const int32_t *ctx_before, int B, int q_len, const void *k_new,
                      const void *v_new, int rows_are_bf16) {
    if (D != 128) return -1;
    float row[128];
    uint8_t codes[128];
    for (int b = 0; b < B; ++b) {
        for (int j = 0; j < q_len; ++j) {
            const int s = ctx_before[b] + j;
            const int logical = s / ORC_BLOCK;
            if (s < 0 || logical >= max_blocks) return -1;
            const int blk = block_table[(size_t)b * max_blocks + logical];
            if (blk < 0 || blk >= num_blocks) return -1;
            const int slot = s % ORC_BLOCK;
            for (int g = 0; g < Hkv; ++g) {
                const size_t src = (((size_t)b * q_len + j) * Hkv + g) * D;
                uint8_t *tile = tiles + ((size_t)blk * Hkv + g) * ORC_FP8_TILE;
                for (int d = 0; d < D; ++d) row[d] = (float)load_elem(k_new, src + d, rows_are_bf16);
                const float ks = quantize_row(row, D, codes);
                for (int d = 0; d < D; ++d) tile[k_byte(slot, d)] = codes[d];
                memcpy(tile + 4096 + 4 * slot, &ks, 4);
                for (int d = 0; d < D; ++d) row[d] = (float)load_elem(v_new, src + d, rows_are_bf16);
                const float vs = quantize_row(row, D, codes);
                for (int d = 0; d < D; ++d) tile[v_byte(slot, d)] = codes[d];
                memcpy(tile + 4160 + 4 * slot, &vs, 4);
            }
        }
    }
    return 0;
}

typedef struct {
    int Hkv;
    const uint8_t *tiles;
} orc_fp8_pool;

static double fp8_kv(const void *ctx, int is_v, int blk, int g, int slot, int d) {
    const orc_fp8_pool *p = (const orc_fp8_pool *)ctx;
    const uint8_t *tile = p->tiles + ((size_t)blk * p->Hkv + g) * ORC_FP8_TILE;
    float sc;
    memcpy(&sc, tile + (is_v ? 4160 : 4096) + 4 * slot, 4);
    const uint8_t code = tile[is_v ? v_byte(slot, d) : k_byte(slot, d)];
    return (double)orc_e4m3_decode(code) * (double)sc;
}

/* Attention over an FP8 cache: orc_decode_attn on the dequantised rows
 * (code value times the row's scale); q is bf16; D = 128. */
int orc_decode_attn_fp8(int num_blocks, int Hkv, int D, const uint8_t *tiles, const int32_t *block_table,
                        int max_blocks, const int32_t *ctx_lens, int B, int q_len, int Hq, double scale,
                        int causal, const uint16_t *q, double *out) {
    if (D != 128) return -1;
    const orc_fp8_pool pool = {Hkv, tiles};
    return attend(num_blocks, Hkv, D, fp8_kv, &pool, block_table, max_blocks, ctx_lens, B, q_len, Hq,
                  scale, causal, q, 1, out);
}

/* -------------------------------------------------------------------- head */

/* -------------------------------------------------------------- audio head */

/* Mish [MIS]: x * tanh(softplus(x)), softplus(x) = ln(1 + e^x), in
 * double.  Past x = 40, ln(1 + e^x) equals x to double precision. */
double orc_mish(double x) {
    const double sp = x > 40.0 ? x : log1p(exp(x));
    return x * tanh(sp);
}

/* Round a double to the nearest bfloat16 (8 significant bits; below 2^-126
 * the fixed spacing 2^-133 of its subnormals), ties to the even significand;
 * returns the bit pattern. */
uint16_t orc_bf16_round(double x) {
    float f;
    if (isnan(x) || isinf(x)) {
        f = (float)x;
    } else if (fabs(x) < 0x1p-126) {
        f = (float)ldexp(nearbyint(ldexp(x, 133)), -133);  /* exact: on the float grid */
    } else {
        int e;
        const double m = frexp(x, &e);           /* x = m * 2^e, 0.5 <= |m| < 1 */
        const double q = nearbyint(ldexp(m, 8));  /* 8 significant bits, ties to even */
        f = (float)ldexp(q, e - 8);                /* exact: fits in a float */
    }
    uint32_t bits;
    memcpy(&bits, &f, sizeof bits);
    return (uint16_t)(bits >> 16);
}

/* The first layer of the two-layer audio head ([TON], section 3: the state
 * is expanded to width 4,096 and passed through Mish): for every row r and
 * feature f, pre = sum_k h[r][k] * W1[f][k] + b1[f] (b1 may be NULL), and
 * z[r][f] = bfloat16(Mish(pre)) — the kernel keeps z as the bfloat16 operand
 * of the second layer, so the oracle rounds the exact value once.  h and W1
 * are bf16 bit patterns; mish_out (nullable) receives Mish(pre) unrounded. */
int orc_audio_expand(const uint16_t *h, const uint16_t *W1, const float *b1, int R, int H, int F,
                     uint16_t *z, double *mish_out) {
    if (R < 0 || H <= 0 || F <= 0) return -1;
    for (int r = 0; r < R; ++r) {
        for (int f = 0; f < F; ++f) {
            double acc = b1 ? (double)b1[f] : 0.0;
            for (int k = 0; k < H; ++k)
                acc += load_elem(h, (size_t)r * H + k, 1) * load_elem(W1, (size_t)f * H + k, 1);
            const double m = orc_mish(acc);
            if (mish_out) mish_out[(size_t)r * F + f] = m;
            z[(size_t)r * F + f] = orc_bf16_round(m);
        }
    }
    return 0;
}

/* Head selection with a bias and a vocabulary mask ([TON], section 3: each
 * stage emits its codebook plus the structural tokens it may produce; logits
 * outside the target vocabulary are masked at sampling).  logit[v] =
 * float(sum_k h[r][k] * W[v][k] + b[v]) (b nullable).  The last n_tail ids
 * V - n_tail .. V - 1 are the structural tokens; id V - n_tail + j may be
 * chosen for row r only if bit j of tail_allowed[r] is set (tail_allowed NULL:
 * all may).  Selection as orc_head_select over the allowed ids. */
static int head_select_at(const void *h, const void *W, int is_bf16, const float *b, int R, int H, int V,
                          int mode, float T, const uint64_t *seed, const uint64_t *step, uint32_t pos, int n_tail,
                          const uint32_t *tail_allowed, int32_t *ids, float *best, float *second,
                          float *logits_out) {
    if (R < 0 || H <= 0 || V <= 0 || (mode != 0 && mode != 1) || n_tail < 0 || n_tail > 32 || n_tail > V)
        return -1;
    if (mode == 1 && !(T > 0.0f)) return -1;
    for (int r = 0; r < R; ++r) {
        int arg = -1;
        float top = -INFINITY, next = -INFINITY;
        for (int v = 0; v < V; ++v) {
            double acc = b ? (double)b[v] : 0.0;
            for (int k = 0; k < H; ++k)
                acc += load_elem(h, (size_t)r * H + k, is_bf16) * load_elem(W, (size_t)v * H + k, is_bf16);
            const float logit = (float)acc;
            if (logits_out) logits_out[(size_t)r * V + v] = logit;
            const int j = v - (V - n_tail);
            if (j >= 0 && tail_allowed && !((tail_allowed[r] >> j) & 1u)) continue;
            float key = logit;
            if (mode == 1) key = logit / T + orc_gumbel(seed[r], step[r], 0u, pos, (uint32_t)v);
            if (arg < 0 || key > top) {
                next = top;
                top = key;
                arg = v;
            } else if (key > next) {
                next = key;
            }
        }
        ids[r] = arg;
        if (best) best[r] = top;
        if (second) second[r] = next;
    }
    return 0;
}

/* The selection above with the Gumbel counter's position 0 (one draw per
 * vocabulary entry and step). */
int orc_head_select_masked(const void *h, const void *W, int is_bf16, const float *b, int R, int H, int V,
                           int mode, float T, const uint64_t *seed, const uint64_t *step, int n_tail,
                           const uint32_t *tail_allowed, int32_t *ids, float *best, float *second,
                           float *logits_out) {
    return head_select_at(h, W, is_bf16, b, R, H, V, mode, T, seed, step, 0u, n_tail, tail_allowed, ids, best,
                          second, logits_out);
}

/* Codebook head and token choice [TON, section 3]: logits[r][v] = h[r] . W[v]
 * over the stage vocabulary (V entries, the last one the boundary token).
 * mode 0 (temperature zero): id = argmax_v logits.  mode 1: id =
 * argmax_v (logits / T + G_v) with G_v Gumbel noise (tag 0, pos 0, idx v), a
 * draw from softmax(logits / T).  eos_allowed[r] == 0 removes v = V-1 (the
 * one-id case of the stage vocabulary mask below: a tail of one id whose
 * mask bit is eos_allowed[r]).
 * Equal keys resolve to the lowest index.  best / second receive the top two
 * keys (second = -inf when V == 1); logits_out (nullable) receives the fp32
 * logits [R][V].  Returns 0, or -1 on bad arguments. */
int orc_head_select(const void *h, const void *W, int is_bf16, int R, int H, int V, int mode,
                    float T, const uint64_t *seed, const uint64_t *step,
                    const uint8_t *eos_allowed, int32_t *ids, float *best, float *second,
                    float *logits_out) {
    uint32_t *mask = NULL;
    if (eos_allowed && R > 0) {
        mask = (uint32_t *)malloc((size_t)R * sizeof *mask);
        if (!mask) return -1;
        for (int r = 0; r < R; ++r) mask[r] = eos_allowed[r] ? 1u : 0u;
    }
    const int rc = orc_head_select_masked(h, W, is_bf16, NULL, R, H, V, mode, T, seed, step, eos_allowed ? 1 : 0,
                                          mask, ids, best, second, logits_out);
    free(mask);
    return rc;
}

/* ---------------------------------------------------------- code predictor */

/* The code predictor's frame loop ([NAR], "Exploiting the regular building of
 * the Code Predictor" / "Turn a fixed predictor loop into one GPU program": a
 * fixed number of autoregressive steps per frame, one per remaining codebook,
 * over a short bounded context held in a preallocated KV cache).  The pages
 * give no architecture; the reading is the smallest loop on this path's
 * primitives.  For every stream r, with x = x0[r] (the talker's state for the
 * frame) and an empty cache, for step i = 0 .. n_steps-1:
 *   qkv = bf16(x Wqkv^T)            q [Hq][D], k and v [Hkv][D]
 *   cache position i <- k, v
 *   o_h = bf16(sum_t softmax_t(scale q_h . k_t[g(h)]) v_t[g(h)]), t = 0..i,
 *         g(h) = h / (Hq / Hkv), scale = 1 / sqrt(D)
 *   logit[v] = float(o . W_i[v]), token = argmax of logit (mode 0) or of
 *         logit / T + Gumbel noise (tag 0, pos i + 1, idx v) (mode 1)
 *   x = E_i[token]                  (the embedding of step i's codebook)
 * x0, Wqkv [(Hq + 2 Hkv) D][H], W [n_steps][V][Hq D] and E [n_steps][V][H] are
 * bf16 bit patterns; tokens, best and second are [n_steps][R].  With trace
 * (nullable, doubles): per step and stream the bf16 values of q, k, v and o
 * ([n_steps][R][(Hq + 2 Hkv) D + Hq D]). */
int orc_code_predictor(int R, int H, int Hq, int Hkv, int D, int V, int n_steps, const uint16_t *x0,
                       const uint16_t *Wqkv, const uint16_t *W, const uint16_t *E, int mode, float T,
                       const uint64_t *seed, const uint64_t *step, int32_t *tokens, float *best, float *second,
                       double *trace) {
    if (R < 0 || H <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || D <= 0 || V <= 0 || n_steps <= 0 ||
        n_steps > ORC_BLOCK || (mode != 0 && mode != 1) || (mode == 1 && !(T > 0.0f)))
        return -1;
    const int F = (Hq + 2 * Hkv) * D, HO = Hq * D, group = Hq / Hkv;
    const double scale = 1.0 / sqrt((double)D);
    double *x = malloc(sizeof(double) * (size_t)H);
    double *qkv = malloc(sizeof(double) * (size_t)F);
    double *kc = malloc(sizeof(double) * (size_t)n_steps * Hkv * D);
    double *vc = malloc(sizeof(double) * (size_t)n_steps * Hkv * D);
    double *o = malloc(sizeof(double) * (size_t)HO);
    double *sc = malloc(sizeof(double) * (size_t)n_steps);
    uint16_t *ob = malloc(sizeof(uint16_t) * (size_t)HO);
    if (!x || !qkv || !kc || !vc || !o || !sc || !ob) {
        free(x); free(qkv); free(kc); free(vc); free(o); free(sc); free(ob);
        return -1;
    }
    for (int r = 0; r < R; ++r) {
        for (int k = 0; k < H; ++k) x[k] = load_elem(x0, (size_t)r * H + k, 1);
        for (int i = 0; i < n_steps; ++i) {
            for (int f = 0; f < F; ++f) {
                double acc = 0.0;
                for (int k = 0; k < H; ++k) acc += x[k] * load_elem(Wqkv, (size_t)f * H + k, 1);
                const uint16_t b = orc_bf16_round(acc);
                qkv[f] = load_elem(&b, 0, 1);
            }
            const double *q = qkv, *kn = qkv + HO, *vn = qkv + HO + Hkv * D;
            memcpy(kc + (size_t)i * Hkv * D, kn, sizeof(double) * (size_t)Hkv * D);
            memcpy(vc + (size_t)i * Hkv * D, vn, sizeof(double) * (size_t)Hkv * D);
            for (int h = 0; h < Hq; ++h) {
                const int kvh = h / group;
                double m = -INFINITY;
                for (int t = 0; t <= i; ++t) {
                    double dot = 0.0;
                    for (int d = 0; d < D; ++d) dot += q[h * D + d] * kc[((size_t)t * Hkv + kvh) * D + d];
                    sc[t] = scale * dot;
                    if (sc[t] > m) m = sc[t];
                }
                double denom = 0.0;
                for (int t = 0; t <= i; ++t) {
                    sc[t] = exp(sc[t] - m);
                    denom += sc[t];
                }
                for (int d = 0; d < D; ++d) {
                    double acc = 0.0;
                    for (int t = 0; t <= i; ++t) acc += sc[t] / denom * vc[((size_t)t * Hkv + kvh) * D + d];
                    ob[h * D + d] = orc_bf16_round(acc);
                    o[h * D + d] = load_elem(ob, (size_t)(h * D + d), 1);
                }
            }
            if (trace) {
                double *tr = trace + ((size_t)i * R + r) * (size_t)(F + HO);
                memcpy(tr, qkv, sizeof(double) * (size_t)F);
                memcpy(tr + F, o, sizeof(double) * (size_t)HO);
            }
            const size_t at = (size_t)i * R + r;
            int32_t arg;
            float top, next;
            head_select_at(ob, W + (size_t)i * V * HO, 1, NULL, 1, HO, V, mode, T, seed ? seed + r : NULL,
                           step ? step + r : NULL, (uint32_t)(i + 1), 0, NULL, &arg, &top, &next, NULL);
            tokens[at] = arg;
            if (best) best[at] = top;
            if (second) second[at] = next;
            const uint16_t *Ei = E + (size_t)i * V * H;
            for (int k = 0; k < H; ++k) x[k] = load_elem(Ei, (size_t)arg * H + k, 1);
        }
    }
    free(x); free(qkv); free(kc); free(vc); free(o); free(sc); free(ob);
    return 0;
}

/* ------------------------------------------------------------------ verify */

/* softmax(x / T)[v] for one row, in double, rounded to float. */
static void row_probs(const float *x, int V, float T, float *p) {
    double m = -INFINITY;
    for (int v = 0; v < V; ++v)
        if ((double)x[v] > m) m = (double)x[v];
    double z = 0.0;
    for (int v = 0; v < V; ++v) z += exp(((double)x[v] - m) / (double)T);
    for (int v = 0; v < V; ++v) p[v] = (float)(exp(((double)x[v] - m) / (double)T) / z);
}

/* Speculative verification [OPT, "Speculative Decoding for Acoustic Tokens"],
 * for every stream b (the page's function handles batch row 0 only):
 * target probabilities p_t = softmax(target_logits[b][i] / T); for draft i in
 * order with token d and draft probability p_d = draft_probs[b][i][d]:
 * p_d == 0 rejects; otherwise the draft is accepted when u_i < p_t[d] / p_d
 * (u_i the Philox uniform tag 1, pos 0, idx i).  At the first rejection the
 * replacement token is drawn from the clamped residual max(p_t - p_d, 0),
 * normalised (Gumbel-max over log of the residual, tag 2, pos 0, idx v; if the
 * residual is zero everywhere, from p_t itself) and verification stops.  If
 * every draft is accepted next_token = -1, or with flags & 1 a bonus token is
 * drawn from softmax(target_logits[b][K] / T) (tag 2, pos 0).  A stream draws
 * at most once per call, so the draw's noise is keyed by (stream, step, v)
 * whichever row it draws from.
 * gap_accept[b]: min |p_t/p_d - u| over the tests made (inf if none);
 * gap_resid[b]: gap between the two largest keys of the final draw (inf if
 * none).  Returns 0, or -1 on a draft token outside [0, V). */
int orc_spec_verify(const float *target_logits, const float *draft_probs,
                    const int32_t *draft_tokens, int B, int K, int V, float T,
                    const uint64_t *seed, const uint64_t *step, int flags,
                    int32_t *n_accepted, int32_t *next_token,
                    float *gap_accept, float *gap_resid) {
    float *pt = (float *)malloc(sizeof(float) * (size_t)V);
    if (!pt) return -1;
    for (int b = 0; b < B; ++b) {
        int acc = 0, next = -1;
        float gacc = INFINITY, gres = INFINITY;
        int rejected = 0;
        for (int i = 0; i < K; ++i) {
            const int d = draft_tokens[(size_t)b * K + i];
            if (d < 0 || d >= V) { free(pt); return -1; }
            const float *tl = target_logits + ((size_t)b * (K + 1) + i) * V;
            const float *dp = draft_probs + ((size_t)b * K + i) * V;
            row_probs(tl, V, T, pt);
            int accepted = 0;
            if (dp[d] > 0.0f) {
                const float ratio = pt[d] / dp[d];
                const float u = orc_uniform(seed[b], step[b], 1u, 0u, (uint32_t)i);
                const float gap = fabsf(ratio - u);
                if (gap < gacc) gacc = gap;
                accepted = u < ratio;
            }
            if (accepted) { ++acc; continue; }
            /* rejection: draw from the clamped residual */
            int any = 0;
            for (int v = 0; v < V; ++v)
                if (pt[v] - dp[v] > 0.0f) { any = 1; break; }
            float top = -INFINITY, sec = -INFINITY;
            for (int v = 0; v < V; ++v) {
                const float r = any ? fmaxf(pt[v] - dp[v], 0.0f) : pt[v];
                if (!(r > 0.0f)) continue;
                const float key = logf(r) + orc_gumbel(seed[b], step[b], 2u, 0u, (uint32_t)v);
                if (next < 0 || key > top) { sec = top; top = key; next = v; }
                else if (key > sec) sec = key;
            }
            gres = top - sec;
            rejected = 1;
            break;
        }
        if (!rejected && (flags & 1)) {
            const float *tl = target_logits + ((size_t)b * (K + 1) + K) * V;
            float top = -INFINITY, sec = -INFINITY;
            for (int v = 0; v < V; ++v) {
                const float key = tl[v] / T + orc_gumbel(seed[b], step[b], 2u, 0u, (uint32_t)v);
                if (next < 0 || key > top) { sec = top; top = key; next = v; }
                else if (key > sec) sec = key;
            }
            gres = top - sec;
        }
        n_accepted[b] = acc;
        next_token[b] = next;
        if (gap_accept) gap_accept[b] = gacc;
        if (gap_resid) gap_resid[b] = gres;
    }
    free(pt);
    return 0;
}
