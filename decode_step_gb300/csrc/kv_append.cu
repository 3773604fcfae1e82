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
// TensorRT-LLM": the KV cache in FP8) and the rotary append: one warp per row
// of a new token (kv_append_rows_kernel).  An FP8 row is one quantisation
// block, scale = max|x| / 448 and codes = E4M3(x / scale) (IEEE fp32
// division, round to nearest even, saturating); codes and scale go to the
// (block, head) record of the cache layout: keys token-major with 16-byte
// chunks swizzled, values dimension-major in the layout's slot order, then
// the scales.  The rotary append rotates the new token's query and key rows
// by its position before these writes.
#include <cuda_fp8.h>

#include <cmath>

#include "tts_common.cuh"
#include "tts_internal.h"

namespace tts {
namespace {

constexpr int kVecsAhead = 4;  // 16-byte words per thread loaded before the position is known

__global__ void __launch_bounds__(128)
kv_append_kernel(const int32_t *__restrict__ table, int max_blocks,
                 const int32_t *__restrict__ ctx_before, int q_len, int Hkv, int num_blocks,
                 int row_vecs, const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
                 uint4 *__restrict__ k_pool, uint4 *__restrict__ v_pool, int32_t *err, int wait_last) {
    // wait_last: the inputs are not written by the kernel before (they come
    // from pinned host memory); the append runs at once and waits for that
    // kernel only before it ends, so the kernels after it still find both done
    if (!wait_last) pdl_wait_prerequisites();
    pdl_allow_dependents();
    const int per_tensor = Hkv * row_vecs;
    const size_t src0 = static_cast<size_t>(blockIdx.x) * per_tensor;
    auto load = [&](int i) { return i < per_tensor ? __ldg(k_new + src0 + i) : __ldg(v_new + src0 + i - per_tensor); };
    // the rows do not depend on the position: their first words are in flight
    // while the position and the block are read
    uint4 ahead[kVecsAhead];
#pragma unroll
    for (int u = 0; u < kVecsAhead; ++u) {
        const int i = threadIdx.x + u * blockDim.x;
        if (i < 2 * per_tensor) ahead[u] = load(i);
    }
    const int b = blockIdx.x / q_len;
    const int j = blockIdx.x % q_len;
    const int before = ctx_before[b];
    const int cap = max_blocks * TTS_BLOCK_TOKENS;
    if (before < 0 || before >= cap || j >= cap - before) {
        if (threadIdx.x == 0) flag_error(err, TTS_ERRBIT_CTX_LEN);
        if (wait_last) pdl_wait_prerequisites();
        return;
    }
    const int s = before + j;
    const int blk = table[static_cast<size_t>(b) * max_blocks + s / TTS_BLOCK_TOKENS];
    if (blk < 0 || blk >= num_blocks) {
        if (threadIdx.x == 0) flag_error(err, TTS_ERRBIT_BLOCK_ID);
        if (wait_last) pdl_wait_prerequisites();
        return;
    }
    const int slot = s % TTS_BLOCK_TOKENS;
    auto store = [&](int i, const uint4 &val) {
        const bool is_v = i >= per_tensor;
        const int e = is_v ? i - per_tensor : i;
        const int g = e / row_vecs;
        const int c = e % row_vecs;
        const size_t dst = ((static_cast<size_t>(blk) * Hkv + g) * TTS_BLOCK_TOKENS + slot) * row_vecs + c;
        (is_v ? v_pool : k_pool)[dst] = val;
    };
#pragma unroll
    for (int u = 0; u < kVecsAhead; ++u) {
        const int i = threadIdx.x + u * blockDim.x;
        if (i < 2 * per_tensor) store(i, ahead[u]);
    }
    for (int i = threadIdx.x + kVecsAhead * blockDim.x; i < 2 * per_tensor; i += blockDim.x) store(i, load(i));
    if (wait_last) pdl_wait_prerequisites();
}

// Byte of token slot s within a dimension's 16 value codes (slot order
// 0 1 8 9 2 3 10 11 4 5 12 13 6 7 14 15: lane t of a 16-bit ldmatrix row read
// then holds the slots 2t, 2t+1, 2t+8, 2t+9 its attention fragment needs).
__device__ __forceinline__ int v_code_pos(int s) { return 4 * ((s & 7) >> 1) + (s & 1) + 2 * (s >> 3); }

constexpr int kFp8D = 128;
constexpr int kFp8Tile = 4224;  // bytes of one (block, head) record

// ------------------------------------------------ bf16 rows, head_dim 128

// Rotary position embedding (RoFormer's rotation in the rotate-half
// arrangement).  The engine of "Optimizing Streaming Text-to-Speech Models for
// Sub-50 Millisecond Latency", section "Engine-Level Optimizations with
// TensorRT-LLM", folds the KV-cache write and the rotary embedding into the
// same kernel; so does this one.  For the token at position s, lane l of a
// warp owns the pairs (i, i + 64) for i = 2l, 2l + 1, whose angles are
// a = s * theta_i.  The angle is formed in double (the same product the
// definition takes) and reduced modulo 2 pi in double (Cody and Waite's
// reduction with 2 pi split into two doubles); the reduced angle r,
// |r| <= pi, is split into floats r_hi + r_lo, and cos/sin come from
// sincosf(r_hi) with the first-order correction for r_lo: an error of a few
// 2^-24 for a handful of double operations per angle (double throughput is
// low on this part).  The rotation itself is fp32.
constexpr double kTwoPiHi = 6.283185307179586;       // 2 pi rounded to double
constexpr double kTwoPiLo = 2.4492935982947064e-16;  // 2 pi - kTwoPiHi
constexpr double kInvTwoPi = 0.15915494309189535;    // 1 / (2 pi)

__device__ __forceinline__ float2 rope_cos_sin(int s, double theta) {
    const double a = static_cast<double>(s) * theta;
    const double k = rint(a * kInvTwoPi);
    const double r = fma(-k, kTwoPiLo, fma(-k, kTwoPiHi, a));
    const float rh = static_cast<float>(r);
    const float rl = static_cast<float>(r - static_cast<double>(rh));
    float sh, ch;
    sincosf(rh, &sh, &ch);
    return make_float2(fmaf(-sh, rl, ch), fmaf(ch, rl, sh));
}

constexpr int kRowThreads = 256;
constexpr int kRowWarps = kRowThreads / 32;
constexpr int kRowsAhead = 4;  // rows per warp loaded before the token's position is known

// One CTA per (stream, new token) of bf16 rows with head_dim 128; one warp per
// row.  Rows: with kRope the Hq query rows first (rotated, written back in
// place as bf16), then the Hkv key rows (rotated with kRope), then the Hkv
// value rows.  Key and value rows go to the cache: bf16 rows, or with kFp8
// one quantisation block per row (scale = max|x| / 448, codes = E4M3(x /
// scale), IEEE fp32 division, round to nearest even, saturating; an all-zero
// row has scale 0 and codes 0) written into the (block, head) record.
//
// Latency: a warp's first kRowsAhead rows are loaded before the position is
// read (they do not depend on it); meanwhile threads 0..63 read the position
// and the block, and with kRope each computes one angle's cos/sin, shared
// through shared memory.
template <bool kFp8, bool kRope>
__global__ void __launch_bounds__(kRowThreads)
kv_append_rows_kernel(const int32_t *__restrict__ table, int max_blocks, const int32_t *__restrict__ ctx_before,
                      int q_len, int Hq, int Hkv, int num_blocks, const RopeFreqs freqs, __nv_bfloat16 *q,
                      const __nv_bfloat16 *__restrict__ k_new, const __nv_bfloat16 *__restrict__ v_new,
                      uint8_t *__restrict__ k_pool, uint8_t *__restrict__ v_pool, int32_t *err) {
    __shared__ float2 cs[kFp8D / 2];
    __shared__ int where[2];  // block (-1: skip the token), slot
    pdl_wait_prerequisites();
    pdl_allow_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nq = kRope ? Hq : 0;
    const int rows = nq + 2 * Hkv;
    auto src_of = [&](int row) -> const __nv_bfloat16 * {
        if (row < nq) return q + (static_cast<size_t>(blockIdx.x) * Hq + row) * kFp8D;
        const int g = row - nq;
        return g < Hkv ? k_new + (static_cast<size_t>(blockIdx.x) * Hkv + g) * kFp8D
                       : v_new + (static_cast<size_t>(blockIdx.x) * Hkv + g - Hkv) * kFp8D;
    };
    // lane's elements: dims 2l, 2l + 1 (word lo) and 2l + 64, 2l + 65 (word hi)
    uint32_t lo[kRowsAhead], hi[kRowsAhead];
#pragma unroll
    for (int u = 0; u < kRowsAhead; ++u) {
        const int row = warp + u * kRowWarps;
        if (row < rows) {
            const uint32_t *src = reinterpret_cast<const uint32_t *>(src_of(row));
            lo[u] = src[lane];
            hi[u] = src[32 + lane];
        }
    }
    if (threadIdx.x < kFp8D / 2) {
        const int b = blockIdx.x / q_len;
        const int j = blockIdx.x % q_len;
        const int before = ctx_before[b];
        const int cap = max_blocks * TTS_BLOCK_TOKENS;
        int blk = -1, s = 0;
        if (before < 0 || before >= cap || j >= cap - before) {
            if (threadIdx.x == 0) flag_error(err, TTS_ERRBIT_CTX_LEN);
        } else {
            s = before + j;
            blk = table[static_cast<size_t>(b) * max_blocks + s / TTS_BLOCK_TOKENS];
            if (blk < 0 || blk >= num_blocks) {
                if (threadIdx.x == 0) flag_error(err, TTS_ERRBIT_BLOCK_ID);
                blk = -1;
            }
        }
        if (threadIdx.x == 0) {
            where[0] = blk;
            where[1] = s % TTS_BLOCK_TOKENS;
        }
        if constexpr (kRope) cs[threadIdx.x] = rope_cos_sin(s, freqs.theta[threadIdx.x]);
    }
    __syncthreads();
    const int blk = where[0], slot = where[1];
    if (blk < 0) return;
    float2 r0 = make_float2(1.0f, 0.0f), r1 = r0;
    if constexpr (kRope) {
        r0 = cs[2 * lane];
        r1 = cs[2 * lane + 1];
    }

    auto emit = [&](int row, uint32_t wlo, uint32_t whi) {
        float x[4] = {bf16_lo(wlo), bf16_hi(wlo), bf16_lo(whi), bf16_hi(whi)};
        const bool is_q = row < nq, is_k = !is_q && row < nq + Hkv;
        if (kRope && (is_q || is_k)) {
            const float2 cse[2] = {r0, r1};
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const float x1 = x[e], x2 = x[2 + e];
                x[e] = fmaf(-x2, cse[e].y, x1 * cse[e].x);
                x[2 + e] = fmaf(x1, cse[e].y, x2 * cse[e].x);
            }
        }
        const __nv_bfloat162 plo = __floats2bfloat162_rn(x[0], x[1]), phi = __floats2bfloat162_rn(x[2], x[3]);
        if (is_q) {
            uint32_t *dst = reinterpret_cast<uint32_t *>(q + (static_cast<size_t>(blockIdx.x) * Hq + row) * kFp8D);
            dst[lane] = *reinterpret_cast<const uint32_t *>(&plo);
            dst[32 + lane] = *reinterpret_cast<const uint32_t *>(&phi);
            return;
        }
        const int g = is_k ? row - nq : row - nq - Hkv;
        const size_t tile = static_cast<size_t>(blk) * Hkv + g;
        if constexpr (!kFp8) {
            uint32_t *dst = reinterpret_cast<uint32_t *>(is_k ? k_pool : v_pool) +
                            (tile * TTS_BLOCK_TOKENS + slot) * (kFp8D / 2);
            dst[lane] = *reinterpret_cast<const uint32_t *>(&plo);
            dst[32 + lane] = *reinterpret_cast<const uint32_t *>(&phi);
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
                // key codes token-major, 16-byte chunk c of slot s at chunk c ^ (s % 8)
                *reinterpret_cast<uint16_t *>(rec + 128 * slot + 16 * ((d1 >> 4) ^ (slot & 7)) + (d1 & 15)) =
                    static_cast<uint16_t>(c01);
                *reinterpret_cast<uint16_t *>(rec + 128 * slot + 16 * ((d2 >> 4) ^ (slot & 7)) + (d2 & 15)) =
                    static_cast<uint16_t>(c23);
                if (lane == 0) *reinterpret_cast<float *>(rec + 4096 + 4 * slot) = scale;
            } else {
                // value codes dimension-major, 16 slots per dimension in the layout's order
                uint8_t *v = rec + 2048 + v_code_pos(slot);
                v[16 * d1] = static_cast<uint8_t>(c01);
                v[16 * (d1 + 1)] = static_cast<uint8_t>(c01 >> 8);
                v[16 * d2] = static_cast<uint8_t>(c23);
                v[16 * (d2 + 1)] = static_cast<uint8_t>(c23 >> 8);
                if (lane == 0) *reinterpret_cast<float *>(rec + 4160 + 4 * slot) = scale;
            }
        }
    };
#pragma unroll
    for (int u = 0; u < kRowsAhead; ++u) {
        const int row = warp + u * kRowWarps;
        if (row < rows) emit(row, lo[u], hi[u]);
    }
    for (int row = warp + kRowsAhead * kRowWarps; row < rows; row += kRowWarps) {
        const uint32_t *src = reinterpret_cast<const uint32_t *>(src_of(row));
        emit(row, src[lane], src[32 + lane]);
    }
}

}  // namespace
}  // namespace tts

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
                            d_err, false, 0, nullptr, {}, false};
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
    *out = AppendLaunch{cache, d_block_table, max_blocks_per_seq, d_ctx_before, B, q_len, d_k_new, d_v_new, d_err,
                        false, 0, nullptr, {}, false};
    return TTS_OK;
}

int prepare_append_rope(const tts_kv_cache *cache, const int32_t *d_block_table, int32_t max_blocks_per_seq,
                        const int32_t *d_ctx_before, int32_t B, int32_t q_len, int32_t num_q_heads,
                        float rope_base, void *d_q, const void *d_k_new, const void *d_v_new, int32_t *d_err,
                        AppendLaunch *out) {
    if (rope_base == 0.0f)
        return prepare_append(cache, d_block_table, max_blocks_per_seq, d_ctx_before, B, q_len, d_k_new, d_v_new,
                              d_err, out);
    if (!cache || !d_q || !(rope_base > 1.0f) || rope_base == INFINITY) return TTS_ERR_INVALID;
    if (cache->dtype != TTS_BF16 && cache->dtype != TTS_FP8_E4M3) return TTS_ERR_UNSUPPORTED;
    if (cache->head_dim != kFp8D) return TTS_ERR_UNSUPPORTED;
    if (cache->num_kv_heads < 1 || num_q_heads < 1 || num_q_heads % cache->num_kv_heads != 0) return TTS_ERR_INVALID;
    const int st = prepare_append(cache, d_block_table, max_blocks_per_seq, d_ctx_before, B, q_len, d_k_new,
                                  d_v_new, d_err, out);
    if (st != TTS_OK) return st;
    if (!aligned16(d_q)) return TTS_ERR_INVALID;
    out->rope = true;
    out->Hq = num_q_heads;
    out->q = d_q;
    for (int i = 0; i < kFp8D / 2; ++i) out->freqs.theta[i] = pow(static_cast<double>(rope_base), -2.0 * i / kFp8D);
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
    if (L.rope || L.cache->dtype == TTS_FP8_E4M3) {
        // bf16 rows of head_dim 128 (checked by the prepare functions)
        cfg.blockDim = dim3(kRowThreads, 1, 1);
        const bool fp8 = L.cache->dtype == TTS_FP8_E4M3;
        auto kernel = L.rope ? (fp8 ? kv_append_rows_kernel<true, true> : kv_append_rows_kernel<false, true>)
                             : kv_append_rows_kernel<true, false>;
        if (cudaLaunchKernelEx(&cfg, kernel, L.table, L.max_blocks, L.ctx_before, L.q_len, L.Hq,
                               static_cast<int>(L.cache->num_kv_heads), static_cast<int>(L.cache->num_blocks), L.freqs,
                               static_cast<__nv_bfloat16 *>(L.q), static_cast<const __nv_bfloat16 *>(L.k_new),
                               static_cast<const __nv_bfloat16 *>(L.v_new), static_cast<uint8_t *>(L.cache->k_pool),
                               fp8 ? nullptr : static_cast<uint8_t *>(L.cache->v_pool), L.err) != cudaSuccess) {
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
                           L.err, L.wait_last ? 1 : 0) != cudaSuccess) {
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
    return tts::launch_append(L, {static_cast<cudaStream_t>(stream), tts::thread_pdl()});
}

extern "C" int tts_kv_append_rope(const tts_kv_cache *cache, const int32_t *d_block_table,
                                  int32_t max_blocks_per_seq, const int32_t *d_ctx_before, int32_t B, int32_t q_len,
                                  int32_t num_q_heads, float rope_base, void *d_q, const void *d_k_new,
                                  const void *d_v_new, int32_t *d_err, void *stream) {
    if (rope_base == 0.0f) return TTS_ERR_INVALID;  // the plain append is tts_kv_append
    tts::AppendLaunch L;
    const int st = tts::prepare_append_rope(cache, d_block_table, max_blocks_per_seq, d_ctx_before, B, q_len,
                                            num_q_heads, rope_base, d_q, d_k_new, d_v_new, d_err, &L);
    if (st != TTS_OK) return st;
    return tts::launch_append(L, {static_cast<cudaStream_t>(stream), tts::thread_pdl()});
}
