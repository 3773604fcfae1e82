// KV append: scatter this step's key/value rows into the paged pool
// ("Optimizing Streaming Text-to-Speech Models for Sub-50 Millisecond
// Latency", section "Dynamic Token-Level Batching": a static pool of 16-token
// blocks; token s of a stream lives in block table[s / 16], slot s % 16).
//
// One CTA per (stream, new token); its threads copy the token's Hkv rows of K
// and of V as 16-byte vectors.  Pure data movement: bytes per launch =
// 2 (read + write) x 2 (K, V) x B x q_len x Hkv x row bytes.
//
// FP8 cache ("Optimizing Streaming Text-to-Speech Models for Sub-50
// Millisecond Latency", section "Engine-Level Optimizations with
// TensorRT-LLM": the KV cache in FP8): one warp per (K or V, KV head) row of a
// new token; the row is one quantisation block, scale = max|x| / 448 and
// codes = E4M3(x / scale) (IEEE fp32 division, round to nearest even,
// saturating).  Codes and scale go to the (block, head) record of the cache
// layout: keys token-major with 16-byte chunks swizzled, values
// dimension-major in the layout's slot order, then the scales.
#include <cuda_fp8.h>

#include "tts_common.cuh"
#include "tts_internal.h"

namespace tts {
namespace {

__global__ void __launch_bounds__(128)
kv_append_kernel(const int32_t *__restrict__ table, int max_blocks,
                 const int32_t *__restrict__ ctx_before, int q_len, int Hkv, int num_blocks,
                 int row_vecs, const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
                 uint4 *__restrict__ k_pool, uint4 *__restrict__ v_pool, int32_t *err) {
    pdl_wait_prerequisites();
    pdl_allow_dependents();
    const int b = blockIdx.x / q_len;
    const int j = blockIdx.x % q_len;
    const int before = ctx_before[b];
    const int cap = max_blocks * TTS_BLOCK_TOKENS;
    if (before < 0 || before >= cap || j >= cap - before) {
        if (threadIdx.x == 0) flag_error(err, TTS_ERRBIT_CTX_LEN);
        return;
    }
    const int s = before + j;
    const int blk = table[static_cast<size_t>(b) * max_blocks + s / TTS_BLOCK_TOKENS];
    if (blk < 0 || blk >= num_blocks) {
        if (threadIdx.x == 0) flag_error(err, TTS_ERRBIT_BLOCK_ID);
        return;
    }
    const int slot = s % TTS_BLOCK_TOKENS;
    const int per_tensor = Hkv * row_vecs;
    const size_t src0 = static_cast<size_t>(blockIdx.x) * per_tensor;
    for (int i = threadIdx.x; i < 2 * per_tensor; i += blockDim.x) {
        const bool is_v = i >= per_tensor;
        const int e = is_v ? i - per_tensor : i;
        const int g = e / row_vecs;
        const int c = e % row_vecs;
        const size_t dst =
            ((static_cast<size_t>(blk) * Hkv + g) * TTS_BLOCK_TOKENS + slot) * row_vecs + c;
        if (is_v)
            v_pool[dst] = __ldg(v_new + src0 + e);
        else
            k_pool[dst] = __ldg(k_new + src0 + e);
    }
}

// Byte of token slot s within a dimension's 16 value codes (slot order
// 0 1 8 9 2 3 10 11 4 5 12 13 6 7 14 15: lane t of a 16-bit ldmatrix row read
// then holds the slots 2t, 2t+1, 2t+8, 2t+9 its attention fragment needs).
__device__ __forceinline__ int v_code_pos(int s) { return 4 * ((s & 7) >> 1) + (s & 1) + 2 * (s >> 3); }

constexpr int kFp8D = 128;
constexpr int kFp8Tile = 4224;  // bytes of one (block, head) record

__global__ void __launch_bounds__(128)
kv_append_fp8_kernel(const int32_t *__restrict__ table, int max_blocks, const int32_t *__restrict__ ctx_before,
                     int q_len, int Hkv, int num_blocks, const __nv_bfloat16 *__restrict__ k_new,
                     const __nv_bfloat16 *__restrict__ v_new, uint8_t *__restrict__ tiles, int32_t *err) {
    pdl_wait_prerequisites();
    pdl_allow_dependents();
    const int b = blockIdx.x / q_len;
    const int j = blockIdx.x % q_len;
    const int before = ctx_before[b];
    const int cap = max_blocks * TTS_BLOCK_TOKENS;
    if (before < 0 || before >= cap || j >= cap - before) {
        if (threadIdx.x == 0) flag_error(err, TTS_ERRBIT_CTX_LEN);
        return;
    }
    const int s = before + j;
    const int blk = table[static_cast<size_t>(b) * max_blocks + s / TTS_BLOCK_TOKENS];
    if (blk < 0 || blk >= num_blocks) {
        if (threadIdx.x == 0) flag_error(err, TTS_ERRBIT_BLOCK_ID);
        return;
    }
    const int slot = s % TTS_BLOCK_TOKENS;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int row = warp; row < 2 * Hkv; row += blockDim.x >> 5) {
        const bool is_v = row >= Hkv;
        const int g = is_v ? row - Hkv : row;
        const __nv_bfloat16 *src = (is_v ? v_new : k_new) + (static_cast<size_t>(blockIdx.x) * Hkv + g) * kFp8D;
        const uint2 raw = __ldg(reinterpret_cast<const uint2 *>(src) + lane);  // values 4 lane .. 4 lane + 3
        const float x[4] = {bf16_lo(raw.x), bf16_hi(raw.x), bf16_lo(raw.y), bf16_hi(raw.y)};
        float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
        const float scale = amax / 448.0f;
        uint32_t codes = 0;
        if (scale > 0.0f) {
            const __nv_fp8x2_storage_t c01 =
                __nv_cvt_float2_to_fp8x2(make_float2(x[0] / scale, x[1] / scale), __NV_SATFINITE, __NV_E4M3);
            const __nv_fp8x2_storage_t c23 =
                __nv_cvt_float2_to_fp8x2(make_float2(x[2] / scale, x[3] / scale), __NV_SATFINITE, __NV_E4M3);
            codes = static_cast<uint32_t>(c01) | (static_cast<uint32_t>(c23) << 16);
        }
        uint8_t *tile = tiles + (static_cast<size_t>(blk) * Hkv + g) * kFp8Tile;
        if (!is_v) {
            // dims 4 lane .. 4 lane + 3: chunk lane / 4 of the slot's 128-byte row
            *reinterpret_cast<uint32_t *>(tile + 128 * slot + 16 * ((lane >> 2) ^ (slot & 7)) + 4 * (lane & 3)) = codes;
            if (lane == 0) *reinterpret_cast<float *>(tile + 4096 + 4 * slot) = scale;
        } else {
            uint8_t *dst = tile + 2048 + 16 * (4 * lane) + v_code_pos(slot);
#pragma unroll
            for (int i = 0; i < 4; ++i) dst[16 * i] = static_cast<uint8_t>(codes >> (8 * i));
            if (lane == 0) *reinterpret_cast<float *>(tile + 4160 + 4 * slot) = scale;
        }
    }
}

// --------------------------------------------------------------- RoPE append

// Rotary position embedding fused with the cache write (RoFormer's rotation
// in the rotate-half arrangement).  The engine of "Optimizing Streaming
// Text-to-Speech Models for Sub-50 Millisecond Latency", section
// "Engine-Level Optimizations with TensorRT-LLM", folds the KV-cache write and
// the rotary embedding into the same kernel; so does this one.  One CTA per (stream, new
// token) at position s: lane l owns the pairs (i, i + 64) for i = 2l, 2l + 1;
// their angles s * base^(-2i/128) and cosines/sines come from double
// precision, once per token, and rotate every query and key row in fp32.
// Query rows are rewritten in place (bf16); key rows go to the cache rotated
// (bf16, or quantised from the fp32 rotated row for an FP8 cache); value rows
// as tts_kv_append stores them.
template <bool kFp8>
__global__ void __launch_bounds__(128)
kv_append_rope_kernel(const int32_t *__restrict__ table, int max_blocks, const int32_t *__restrict__ ctx_before,
                      int q_len, int Hq, int Hkv, int num_blocks, double base, __nv_bfloat16 *q,
                      const __nv_bfloat16 *__restrict__ k_new, const __nv_bfloat16 *__restrict__ v_new,
                      uint8_t *__restrict__ k_pool, uint8_t *__restrict__ v_pool, int32_t *err) {
    pdl_wait_prerequisites();
    pdl_allow_dependents();
    const int b = blockIdx.x / q_len;
    const int j = blockIdx.x % q_len;
    const int before = ctx_before[b];
    const int cap = max_blocks * TTS_BLOCK_TOKENS;
    if (before < 0 || before >= cap || j >= cap - before) {
        if (threadIdx.x == 0) flag_error(err, TTS_ERRBIT_CTX_LEN);
        return;
    }
    const int s = before + j;
    const int blk = table[static_cast<size_t>(b) * max_blocks + s / TTS_BLOCK_TOKENS];
    if (blk < 0 || blk >= num_blocks) {
        if (threadIdx.x == 0) flag_error(err, TTS_ERRBIT_BLOCK_ID);
        return;
    }
    const int slot = s % TTS_BLOCK_TOKENS;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    float c[2], sn[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const double a = static_cast<double>(s) * pow(base, -2.0 * (2 * lane + e) / kFp8D);
        double sd, cd;
        sincos(a, &sd, &cd);
        c[e] = static_cast<float>(cd);
        sn[e] = static_cast<float>(sd);
    }
    const int rows = Hq + 2 * Hkv;  // query rows, then key rows, then value rows
    for (int row = warp; row < rows; row += blockDim.x >> 5) {
        const bool is_q = row < Hq, is_k = !is_q && row < Hq + Hkv;
        const int g = is_q ? row : (is_k ? row - Hq : row - Hq - Hkv);
        const __nv_bfloat16 *src =
            is_q ? q + (static_cast<size_t>(blockIdx.x) * Hq + g) * kFp8D
                 : (is_k ? k_new : v_new) + (static_cast<size_t>(blockIdx.x) * Hkv + g) * kFp8D;
        const uint32_t w1 = *reinterpret_cast<const uint32_t *>(src + 2 * lane);        // dims 2l, 2l + 1
        const uint32_t w2 = *reinterpret_cast<const uint32_t *>(src + 64 + 2 * lane);   // dims 2l + 64, 2l + 65
        float x[4] = {bf16_lo(w1), bf16_hi(w1), bf16_lo(w2), bf16_hi(w2)};
        if (is_q || is_k) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const float x1 = x[e], x2 = x[2 + e];
                x[e] = fmaf(-x2, sn[e], x1 * c[e]);
                x[2 + e] = fmaf(x1, sn[e], x2 * c[e]);
            }
        }
        if (is_q) {
            uint32_t *dst = reinterpret_cast<uint32_t *>(q + (static_cast<size_t>(blockIdx.x) * Hq + g) * kFp8D);
            const __nv_bfloat162 lo = __floats2bfloat162_rn(x[0], x[1]), hi = __floats2bfloat162_rn(x[2], x[3]);
            dst[lane] = *reinterpret_cast<const uint32_t *>(&lo);
            dst[32 + lane] = *reinterpret_cast<const uint32_t *>(&hi);
            continue;
        }
        const size_t tile = static_cast<size_t>(blk) * Hkv + g;
        if constexpr (!kFp8) {
            __nv_bfloat16 *dst = reinterpret_cast<__nv_bfloat16 *>(is_k ? k_pool : v_pool) +
                                 (tile * TTS_BLOCK_TOKENS + slot) * kFp8D;
            const __nv_bfloat162 lo = __floats2bfloat162_rn(x[0], x[1]), hi = __floats2bfloat162_rn(x[2], x[3]);
            reinterpret_cast<uint32_t *>(dst)[lane] = *reinterpret_cast<const uint32_t *>(&lo);
            reinterpret_cast<uint32_t *>(dst)[32 + lane] = *reinterpret_cast<const uint32_t *>(&hi);
        } else {
            float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
            const float scale = amax / 448.0f;
            uint32_t c01 = 0, c23 = 0;
            if (scale > 0.0f) {
                c01 = __nv_cvt_float2_to_fp8x2(make_float2(x[0] / scale, x[1] / scale), __NV_SATFINITE, __NV_E4M3);
                c23 = __nv_cvt_float2_to_fp8x2(make_float2(x[2] / scale, x[3] / scale), __NV_SATFINITE, __NV_E4M3);
            }
            uint8_t *rec = k_pool + tile * kFp8Tile;
            const int d1 = 2 * lane, d2 = 64 + 2 * lane;
            if (is_k) {
                *reinterpret_cast<uint16_t *>(rec + 128 * slot + 16 * ((d1 >> 4) ^ (slot & 7)) + (d1 & 15)) =
                    static_cast<uint16_t>(c01);
                *reinterpret_cast<uint16_t *>(rec + 128 * slot + 16 * ((d2 >> 4) ^ (slot & 7)) + (d2 & 15)) =
                    static_cast<uint16_t>(c23);
                if (lane == 0) *reinterpret_cast<float *>(rec + 4096 + 4 * slot) = scale;
            } else {
                uint8_t *v = rec + 2048 + v_code_pos(slot);
                v[16 * d1] = static_cast<uint8_t>(c01);
                v[16 * (d1 + 1)] = static_cast<uint8_t>(c01 >> 8);
                v[16 * d2] = static_cast<uint8_t>(c23);
                v[16 * (d2 + 1)] = static_cast<uint8_t>(c23 >> 8);
                if (lane == 0) *reinterpret_cast<float *>(rec + 4160 + 4 * slot) = scale;
            }
        }
    }
}

}  // namespace
}  // namespace tts

extern "C" int tts_kv_append_rope(const tts_kv_cache *cache, const int32_t *d_block_table,
                                  int32_t max_blocks_per_seq, const int32_t *d_ctx_before, int32_t B, int32_t q_len,
                                  int32_t num_q_heads, float rope_base, void *d_q, const void *d_k_new,
                                  const void *d_v_new, int32_t *d_err, void *stream) {
    using namespace tts;
    if (!cache || !d_q || !(rope_base > 1.0f) || rope_base == INFINITY) return TTS_ERR_INVALID;
    if (cache->dtype != TTS_BF16 && cache->dtype != TTS_FP8_E4M3) return TTS_ERR_UNSUPPORTED;
    if (cache->head_dim != kFp8D) return TTS_ERR_UNSUPPORTED;
    if (num_q_heads < 1 || num_q_heads % (cache->num_kv_heads > 0 ? cache->num_kv_heads : 1) != 0)
        return TTS_ERR_INVALID;
    AppendLaunch L;
    const int st = prepare_append(cache, d_block_table, max_blocks_per_seq, d_ctx_before, B, q_len, d_k_new,
                                  d_v_new, d_err, &L);
    if (st != TTS_OK) return st;
    if (!aligned16(d_q)) return TTS_ERR_INVALID;
    if (B == 0) return TTS_OK;
    const unsigned grid = static_cast<unsigned>(static_cast<long>(B) * q_len);
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int nkv = cache->num_kv_heads, nb = cache->num_blocks;
    if (cache->dtype == TTS_FP8_E4M3)
        kv_append_rope_kernel<true><<<grid, 128, 0, s>>>(
            d_block_table, max_blocks_per_seq, d_ctx_before, q_len, num_q_heads, nkv, nb, rope_base,
            static_cast<__nv_bfloat16 *>(d_q), static_cast<const __nv_bfloat16 *>(d_k_new),
            static_cast<const __nv_bfloat16 *>(d_v_new), static_cast<uint8_t *>(cache->k_pool), nullptr, d_err);
    else
        kv_append_rope_kernel<false><<<grid, 128, 0, s>>>(
            d_block_table, max_blocks_per_seq, d_ctx_before, q_len, num_q_heads, nkv, nb, rope_base,
            static_cast<__nv_bfloat16 *>(d_q), static_cast<const __nv_bfloat16 *>(d_k_new),
            static_cast<const __nv_bfloat16 *>(d_v_new), static_cast<uint8_t *>(cache->k_pool),
            static_cast<uint8_t *>(cache->v_pool), d_err);
    return launch_status();
}

namespace tts {

int prepare_append(const tts_kv_cache *cache, const int32_t *d_block_table, int32_t max_blocks_per_seq,
                   const int32_t *d_ctx_before, int32_t B, int32_t q_len, const void *d_k_new,
                   const void *d_v_new, int32_t *d_err, AppendLaunch *out) {
    if (!cache || !d_block_table || !d_ctx_before || !d_k_new || !d_v_new) return TTS_ERR_INVALID;
    if (!cache->k_pool || (!cache->v_pool && cache->dtype != TTS_FP8_E4M3)) return TTS_ERR_INVALID;
    if (B < 0 || q_len < 1 || max_blocks_per_seq < 1 || max_blocks_per_seq > (1 << 20) ||
        cache->num_blocks < 1 || cache->num_kv_heads < 1 || cache->head_dim < 1)
        return TTS_ERR_INVALID;
    if (cache->block_size != TTS_BLOCK_TOKENS) return TTS_ERR_UNSUPPORTED;
    if (cache->dtype == TTS_FP8_E4M3) {
        if (cache->head_dim != kFp8D) return TTS_ERR_UNSUPPORTED;
        if (!aligned16(cache->k_pool) || !aligned16(d_k_new) || !aligned16(d_v_new)) return TTS_ERR_INVALID;
        if (static_cast<long>(B) * q_len > 0x7FFFFFFFL) return TTS_ERR_INVALID;
        *out = AppendLaunch{cache, d_block_table, max_blocks_per_seq, d_ctx_before, B, q_len, d_k_new, d_v_new,
                            d_err};
        return TTS_OK;
    }
    if (cache->dtype != TTS_F32 && cache->dtype != TTS_BF16) return TTS_ERR_UNSUPPORTED;
    const int elem = cache->dtype == TTS_F32 ? 4 : 2;
    const long row_bytes = static_cast<long>(cache->head_dim) * elem;
    if (row_bytes % 16 != 0) return TTS_ERR_UNSUPPORTED;
    if (!aligned16(cache->k_pool) || !aligned16(cache->v_pool) || !aligned16(d_k_new) ||
        !aligned16(d_v_new))
        return TTS_ERR_INVALID;
    if (static_cast<long>(B) * q_len > 0x7FFFFFFFL) return TTS_ERR_INVALID;
    *out = AppendLaunch{cache, d_block_table, max_blocks_per_seq, d_ctx_before, B, q_len, d_k_new, d_v_new, d_err};
    return TTS_OK;
}

int launch_append(const AppendLaunch &L, LaunchOpts o) {
    if (L.B == 0) return TTS_OK;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(static_cast<long>(L.B) * L.q_len), 1, 1);
    cfg.blockDim = dim3(128, 1, 1);
    cfg.stream = o.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = o.pdl ? 1 : 0;
    if (L.cache->dtype == TTS_FP8_E4M3) {
        if (cudaLaunchKernelEx(&cfg, kv_append_fp8_kernel, L.table, L.max_blocks, L.ctx_before, L.q_len,
                               static_cast<int>(L.cache->num_kv_heads), static_cast<int>(L.cache->num_blocks),
                               static_cast<const __nv_bfloat16 *>(L.k_new), static_cast<const __nv_bfloat16 *>(L.v_new),
                               static_cast<uint8_t *>(L.cache->k_pool), L.err) != cudaSuccess) {
            cudaGetLastError();
            return TTS_ERR_CUDA;
        }
        return TTS_OK;
    }
    const int elem = L.cache->dtype == TTS_F32 ? 4 : 2;
    const int row_vecs = L.cache->head_dim * elem / 16;
    if (cudaLaunchKernelEx(&cfg, kv_append_kernel, L.table, L.max_blocks, L.ctx_before, L.q_len,
                           static_cast<int>(L.cache->num_kv_heads), static_cast<int>(L.cache->num_blocks),
                           row_vecs, static_cast<const uint4 *>(L.k_new), static_cast<const uint4 *>(L.v_new),
                           static_cast<uint4 *>(L.cache->k_pool), static_cast<uint4 *>(L.cache->v_pool),
                           L.err) != cudaSuccess) {
        cudaGetLastError();
        return TTS_ERR_CUDA;
    }
    return TTS_OK;
}

}  // namespace tts

extern "C" int tts_kv_append(const tts_kv_cache *cache, const int32_t *d_block_table,
                             int32_t max_blocks_per_seq, const int32_t *d_ctx_before, int32_t B,
                             int32_t q_len, const void *d_k_new, const void *d_v_new,
                             int32_t *d_err, void *stream) {
    tts::AppendLaunch L;
    const int st = tts::prepare_append(cache, d_block_table, max_blocks_per_seq, d_ctx_before, B, q_len,
                                       d_k_new, d_v_new, d_err, &L);
    if (st != TTS_OK) return st;
    return tts::launch_append(L, {static_cast<cudaStream_t>(stream), false});
}
