// Split-KV flash-decoding GQA attention over the paged KV cache.
//
// What it computes ("TTS Serving, in depth", section "Token generation under
// a frame budget": every decode step reads the stream's KV cache; causal
// q_len-row blocks for speculative verification, "Optimizing Streaming
// Text-to-Speech Models for Sub-50 Millisecond Latency", section "Speculative
// Decoding for Acoustic Tokens"):
//   out[b][j][h] = sum_t softmax_t(scale * q[b][j][h] . k_t) v_t,
// t over the stream's tokens below the row's limit, KV head h / group.
//
// How (HBM-bound: each cached byte is used for 2 flops per query row):
//  - grid (split, KV head, stream); a split is `split_blocks` 16-token blocks.
//    Every query row of the KV head's group (group x q_len rows) is served by
//    one read of each K/V tile.
//  - each warp owns every 4th block of the split and streams its (block, head)
//    K and V tiles (4 KB each, contiguous in the pool) into a private 2-stage
//    shared-memory ring with bulk TMA copies (L2 evict-first), completion on
//    per-stage mbarriers.
//  - lane (p, c) = (lane / 16, lane % 16) reads 16-byte chunk c of the rows of
//    tokens p, p + 2, ..., p + 14 (conflict-free 128-bit shared loads).  Dot
//    products are reduced across the 16 chunk lanes by recursive halving (each
//    shuffle round halves the values a lane carries), leaving every lane the
//    full scores of one token for half of the rows.  Online softmax in the
//    log2 domain with warp-shuffle max reductions; P.V accumulates per lane
//    into its 16-byte slice of the output rows.
//  - warps merge in shared memory; a split writes (m, l, unnormalised o) to
//    the workspace, and the last CTA of a (stream, KV head) — found with an
//    atomic ticket, no waiting — merges the splits (log-sum-exp combine) and
//    writes the output.  A stream with a single split writes its output
//    directly.
#include <mutex>

#include "tts_common.cuh"
#include "tts_internal.h"

namespace tts {
namespace {

constexpr int kWarps = 4;          // warps per CTA
constexpr int kStages = 2;         // pipeline depth per warp
constexpr int kTileBytes = 4096;   // one (block, KV head) tile of K or V: 16 tokens x 256 B
constexpr int kRowBytes = 256;     // one token's key (or value) row
constexpr int kSplitBlocks = 16;   // blocks per split (<= 32 * kWarps)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kNegBig = -1e30f;  // finite "minus infinity" for running maxima
constexpr unsigned kFull = 0xFFFFFFFFu;

struct AttnArgs {
    const uint8_t *k_pool;
    const uint8_t *v_pool;
    int num_blocks;
    int Hkv;
    const int32_t *table;
    int max_blocks;
    const int32_t *ctx_lens;
    int max_ctx;
    int q_len;
    int Hq;
    int group;
    int causal;
    float qscale;  // softmax scale * log2(e)
    const void *q;
    void *out;
    float *o_part;   // [B][Hkv][max_splits][NR][D]
    float2 *ml_part; // [B][Hkv][max_splits][NR]  (running max, sum)
    int32_t *counters;  // [B][Hkv]
    int max_splits;
    int split_blocks;
    int32_t *err;
};

template <int NR, int D>
struct AttnSmem {
    static constexpr size_t stages = size_t(kWarps) * kStages * 2 * kTileBytes;
    static constexpr size_t bars = stages;
    static constexpr size_t pbuf = bars + 8 * kWarps * kStages;
    static constexpr size_t ms = pbuf + 4 * kWarps * 16 * NR;
    static constexpr size_t ls = ms + 4 * kWarps * NR;
    static constexpr size_t os = ls + 4 * kWarps * NR;
    static constexpr size_t flag = os + 4 * size_t(kWarps) * NR * D;
    static constexpr size_t total = flag + 16;
};

template <typename T, int NR>
__global__ void __launch_bounds__(kWarps * 32, NR <= 4 ? 3 : 1)
decode_attn_kernel(const AttnArgs a) {
    using C = Chunk<T>;
    constexpr int EPC = C::N;          // elements per 16-byte chunk
    constexpr int D = 16 * EPC;        // head dim: one 256-byte row per token
    constexpr int HALF = NR / 2;
    using S = AttnSmem<NR, D>;
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + S::bars);
    float *ms = reinterpret_cast<float *>(smem + S::ms);
    float *ls = reinterpret_cast<float *>(smem + S::ls);
    float *os = reinterpret_cast<float *>(smem + S::os);
    int *flag = reinterpret_cast<int *>(smem + S::flag);

    const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_rows = a.group * a.q_len;
    T *out = static_cast<T *>(a.out);
    auto out_ptr = [&](int r) -> T * {
        const int j = r / a.group, hh = r % a.group;
        return out + ((static_cast<size_t>(b) * a.q_len + j) * a.Hq + g * a.group + hh) * D;
    };

    const int L = __ldg(a.ctx_lens + b);
    const int cap = min(a.max_ctx, a.max_blocks * TTS_BLOCK_TOKENS);
    if (L < a.q_len || L > cap) {
        if (split == 0) {
            if (g == 0 && threadIdx.x == 0) flag_error(a.err, TTS_ERRBIT_CTX_LEN);
            for (int i = threadIdx.x; i < n_rows * D; i += blockDim.x)
                store_elem(out_ptr(i / D) + i % D, 0.0f);
        }
        return;
    }
    const int nblk = (L + TTS_BLOCK_TOKENS - 1) / TTS_BLOCK_TOKENS;
    const int n_split = (nblk + a.split_blocks - 1) / a.split_blocks;
    if (split >= n_split) return;
    const int blk0 = split * a.split_blocks;
    const int blk1 = min(nblk, blk0 + a.split_blocks);
    const int my_first = blk0 + warp;
    const int my_n = my_first < blk1 ? (blk1 - my_first + kWarps - 1) / kWarps : 0;

    const uint32_t stage0 = smem_addr(smem) + warp * kStages * 2 * kTileBytes;
    const uint32_t bar0 = smem_addr(bars + warp * kStages);
    float *pbuf = reinterpret_cast<float *>(smem + S::pbuf) + warp * 16 * NR;
    if (lane == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(bar0 + 8 * s, 1);
        fence_mbar_init();
    }
    __syncwarp();

    // Physical block of this warp's i-th tile, held by lane i (-1: invalid).
    int my_id = -1;
    if (lane < my_n) {
        const int id = __ldg(a.table + static_cast<size_t>(b) * a.max_blocks + my_first + lane * kWarps);
        if (id >= 0 && id < a.num_blocks)
            my_id = id;
        else
            flag_error(a.err, TTS_ERRBIT_BLOCK_ID);
    }

    const uint64_t policy = l2_evict_first_policy();
    auto issue = [&](int i) {
        const int id = __shfl_sync(kFull, my_id, i);
        if (lane == 0) {
            const int st = i % kStages;
            const uint32_t bar = bar0 + 8 * st;
            if (id >= 0) {
                const size_t off = (static_cast<size_t>(id) * a.Hkv + g) * kTileBytes;
                mbar_arrive_expect_tx(bar, 2 * kTileBytes);
                bulk_load(stage0 + st * 2 * kTileBytes, a.k_pool + off, kTileBytes, bar, policy);
                bulk_load(stage0 + st * 2 * kTileBytes + kTileBytes, a.v_pool + off, kTileBytes, bar,
                          policy);
            } else {
                mbar_arrive(bar);
            }
        }
    };
    const int n_pre = min(kStages, my_n);
    for (int i = 0; i < n_pre; ++i) issue(i);

    // Query rows at this lane's chunk, pre-scaled into the log2 domain.
    const int p = lane >> 4, c = lane & 15;
    float q[NR][EPC];
#pragma unroll
    for (int r = 0; r < NR; ++r) {
        if (r < n_rows) {
            const int j = r / a.group, hh = r % a.group;
            const T *src = static_cast<const T *>(a.q) +
                           ((static_cast<size_t>(b) * a.q_len + j) * a.Hq + g * a.group + hh) * D +
                           c * EPC;
            C::unpack(__ldg(reinterpret_cast<const uint4 *>(src)), q[r]);
#pragma unroll
            for (int e = 0; e < EPC; ++e) q[r][e] *= a.qscale;
        } else {
#pragma unroll
            for (int e = 0; e < EPC; ++e) q[r][e] = 0.0f;
        }
    }
    // This lane scores token (p + 2 * ((lane >> 1) & 7)) of a tile for rows
    // (lane & 1) * HALF + k; the row's visible-token limit:
    int lim[HALF];
#pragma unroll
    for (int k = 0; k < HALF; ++k) {
        const int r = (lane & 1) * HALF + k;
        lim[k] = r < n_rows ? (a.causal ? L - a.q_len + r / a.group + 1 : L) : 0;
    }
    const int my_tok = p + 2 * ((lane >> 1) & 7);

    float m_run[HALF], l_run[HALF], o[NR][EPC];
#pragma unroll
    for (int k = 0; k < HALF; ++k) { m_run[k] = kNegBig; l_run[k] = 0.0f; }
#pragma unroll
    for (int r = 0; r < NR; ++r)
#pragma unroll
        for (int e = 0; e < EPC; ++e) o[r][e] = 0.0f;

    bool timed_out = false;
    int waited = 0;  // tiles whose copies are known complete
    for (int i = 0; i < my_n; ++i) {
        const int st = i % kStages;
        if (!timed_out) {
            const bool ok = mbar_wait(bar0 + 8 * st, (i / kStages) & 1);
            if (__any_sync(kFull, !ok)) {
                timed_out = true;
                if (lane == 0) flag_error(a.err, TTS_ERRBIT_TIMEOUT);
            } else {
                waited = i + 1;
            }
        }
        const int id = __shfl_sync(kFull, my_id, i);
        if (!timed_out && id >= 0) {
            const uint32_t ks = stage0 + st * 2 * kTileBytes, vs = ks + kTileBytes;
            const int base = (my_first + i * kWarps) * TTS_BLOCK_TOKENS;
            // ---- scores: partial dots over this lane's chunk, 8 tokens x NR rows
            float acc[8 * NR];
#pragma unroll
            for (int jt = 0; jt < 8; ++jt) {
                float kf[EPC];
                C::unpack(lds128(ks + (p + 2 * jt) * kRowBytes + c * 16), kf);
#pragma unroll
                for (int r = 0; r < NR; ++r) {
                    float s = 0.0f;
#pragma unroll
                    for (int e = 0; e < EPC; ++e) s = fmaf(q[r][e], kf[e], s);
                    acc[jt * NR + r] = s;
                }
            }
            // ---- recursive halving across the 16 chunk lanes (masks 8, 4, 2, 1)
#pragma unroll
            for (int step = 0; step < 4; ++step) {
                const int m = 8 >> step;
                const int n = (8 * NR) >> step;
                const bool upper = (lane & m) != 0;
#pragma unroll
                for (int x = 0; x < n / 2; ++x) {
                    const float send = upper ? acc[x] : acc[x + n / 2];
                    const float keep = upper ? acc[x + n / 2] : acc[x];
                    acc[x] = keep + __shfl_xor_sync(kFull, send, m);
                }
            }
            // ---- online softmax (log2 domain)
            const int tpos = base + my_tok;
            float alpha[HALF], other[HALF];
#pragma unroll
            for (int k = 0; k < HALF; ++k) {
                const float s = tpos < lim[k] ? acc[k] : -INFINITY;
                float mx = s;
                mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 2));
                mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 4));
                mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 8));
                mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 16));
                const float m_new = fmaxf(m_run[k], mx);
                alpha[k] = exp2f(m_run[k] - m_new);
                const float pk = exp2f(s - m_new);
                l_run[k] = l_run[k] * alpha[k] + pk;
                m_run[k] = m_new;
                pbuf[my_tok * NR + (lane & 1) * HALF + k] = pk;
                other[k] = __shfl_xor_sync(kFull, alpha[k], 1);
            }
            __syncwarp();
            // ---- rescale and accumulate P.V
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                const bool mine = (r / HALF) == (lane & 1);
                const float f = mine ? alpha[r % HALF] : other[r % HALF];
#pragma unroll
                for (int e = 0; e < EPC; ++e) o[r][e] *= f;
            }
#pragma unroll
            for (int jt = 0; jt < 8; ++jt) {
                const int t = p + 2 * jt;
                uint4 raw = lds128(vs + t * kRowBytes + c * 16);
                if (base + t >= L) raw = make_uint4(0u, 0u, 0u, 0u);  // past the context
                float vf[EPC];
                C::unpack(raw, vf);
                const float *pr = pbuf + t * NR;
#pragma unroll
                for (int r = 0; r < NR; ++r) {
                    const float w = pr[r];
#pragma unroll
                    for (int e = 0; e < EPC; ++e) o[r][e] = fmaf(w, vf[e], o[r][e]);
                }
            }
        }
        __syncwarp();
        if (!timed_out && i + kStages < my_n) issue(i + kStages);
    }
    if (timed_out) {
        // Let copies still in flight land before the CTA's shared memory goes away.
        const int issued = min(my_n, waited + kStages);
        for (int i = waited; i < issued; ++i) mbar_wait(bar0 + 8 * (i % kStages), (i / kStages) & 1);
    }

    // ---- warp totals: sums over the 16 lanes of a row half, outputs over parity
    float l_tot[HALF];
#pragma unroll
    for (int k = 0; k < HALF; ++k) {
        float l = l_run[k];
        l += __shfl_xor_sync(kFull, l, 2);
        l += __shfl_xor_sync(kFull, l, 4);
        l += __shfl_xor_sync(kFull, l, 8);
        l += __shfl_xor_sync(kFull, l, 16);
        l_tot[k] = l;
    }
#pragma unroll
    for (int r = 0; r < NR; ++r)
#pragma unroll
        for (int e = 0; e < EPC; ++e) o[r][e] += __shfl_xor_sync(kFull, o[r][e], 16);
    if (lane < 2) {
#pragma unroll
        for (int k = 0; k < HALF; ++k) {
            ms[warp * NR + lane * HALF + k] = m_run[k];
            ls[warp * NR + lane * HALF + k] = l_tot[k];
        }
    }
    if (lane < 16) {
#pragma unroll
        for (int r = 0; r < NR; ++r)
#pragma unroll
            for (int e = 0; e < EPC; ++e) os[(warp * NR + r) * D + lane * EPC + e] = o[r][e];
    }
    __syncthreads();

    // ---- merge the warps of this split
    const size_t part = (static_cast<size_t>(b) * a.Hkv + g) * a.max_splits;
    for (int idx = threadIdx.x; idx < n_rows * D; idx += blockDim.x) {
        const int r = idx / D, d = idx % D;
        float M = kNegBig;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, ms[w * NR + r]);
        float Ls = 0.0f, O = 0.0f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float f = exp2f(ms[w * NR + r] - M);
            Ls = fmaf(ls[w * NR + r], f, Ls);
            O = fmaf(os[(w * NR + r) * D + d], f, O);
        }
        if (n_split == 1) {
            store_elem(out_ptr(r) + d, Ls > 0.0f ? O / Ls : 0.0f);
        } else {
            a.o_part[((part + split) * NR + r) * D + d] = O;
            if (d == 0) a.ml_part[(part + split) * NR + r] = make_float2(M, Ls);
        }
    }
    if (n_split == 1) return;

    // ---- last split to finish merges all splits (log-sum-exp combine)
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const int ticket = atomicAdd(a.counters + b * a.Hkv + g, 1);
        *flag = ticket == n_split - 1;
    }
    __syncthreads();
    if (!*flag) return;
    __threadfence();
    for (int idx = threadIdx.x; idx < n_rows * D; idx += blockDim.x) {
        const int r = idx / D, d = idx % D;
        float M = kNegBig;
        for (int s = 0; s < n_split; ++s) M = fmaxf(M, __ldcg(&a.ml_part[(part + s) * NR + r].x));
        float Ls = 0.0f, O = 0.0f;
        for (int s = 0; s < n_split; ++s) {
            const float2 ml = __ldcg(&a.ml_part[(part + s) * NR + r]);
            const float f = exp2f(ml.x - M);
            Ls = fmaf(ml.y, f, Ls);
            O = fmaf(__ldcg(&a.o_part[((part + s) * NR + r) * D + d]), f, O);
        }
        store_elem(out_ptr(r) + d, Ls > 0.0f ? O / Ls : 0.0f);
    }
    if (threadIdx.x == 0) a.counters[b * a.Hkv + g] = 0;
}

// Row templates: group * q_len rows are padded up to one of these.
constexpr int kRowTemplates[] = {2, 4, 8, 10, 16};

int padded_rows(int rows) {
    for (int r : kRowTemplates)
        if (rows <= r) return r;
    return 0;
}

template <typename T, int NR>
int launch_nr(const AttnArgs &a, dim3 grid, cudaStream_t stream) {
    constexpr int D = 16 * Chunk<T>::N;
    const size_t smem = AttnSmem<NR, D>::total;
    auto kern = decode_attn_kernel<T, NR>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
        return TTS_ERR_CUDA;
    kern<<<grid, kWarps * 32, smem, stream>>>(a);
    return launch_status();
}

template <typename T>
int launch_typed(const AttnArgs &a, int nr, dim3 grid, cudaStream_t stream) {
    switch (nr) {
        case 2: return launch_nr<T, 2>(a, grid, stream);
        case 4: return launch_nr<T, 4>(a, grid, stream);
        case 8: return launch_nr<T, 8>(a, grid, stream);
        case 10: return launch_nr<T, 10>(a, grid, stream);
        case 16: return launch_nr<T, 16>(a, grid, stream);
        default: return TTS_ERR_UNSUPPORTED;
    }
}

bool supported_head(int dtype, int head_dim) {
    return (dtype == TTS_BF16 && head_dim == 128) || (dtype == TTS_F32 && head_dim == 64);
}

}  // namespace

bool attn_split_policy(int B, int q_len, int num_q_heads, int num_kv_heads, int head_dim,
                       int max_ctx_len, AttnSplit *out) {
    if (B < 1 || q_len < 1 || num_kv_heads < 1 || num_q_heads < num_kv_heads ||
        num_q_heads % num_kv_heads != 0 || head_dim < 1 || max_ctx_len < q_len ||
        max_ctx_len > (1 << 24))
        return false;
    const int rows = padded_rows((num_q_heads / num_kv_heads) * q_len);
    if (rows == 0) return false;
    const int nblk = (max_ctx_len + TTS_BLOCK_TOKENS - 1) / TTS_BLOCK_TOKENS;
    out->blocks = kSplitBlocks;
    out->max_splits = (nblk + kSplitBlocks - 1) / kSplitBlocks;
    out->rows = rows;
    return true;
}

size_t attn_workspace_bytes(int B, int num_kv_heads, int head_dim, const AttnSplit &sp) {
    const size_t units = static_cast<size_t>(B) * num_kv_heads * sp.max_splits * sp.rows;
    return align_up(units * head_dim * sizeof(float), 256) + align_up(units * sizeof(float2), 256) +
           align_up(static_cast<size_t>(B) * num_kv_heads * sizeof(int32_t), 256);
}

}  // namespace tts

extern "C" size_t tts_decode_attn_workspace_size(int32_t B, int32_t q_len, int32_t num_q_heads,
                                                 int32_t num_kv_heads, int32_t head_dim,
                                                 int32_t max_ctx_len) {
    tts::AttnSplit sp;
    if (!tts::attn_split_policy(B, q_len, num_q_heads, num_kv_heads, head_dim, max_ctx_len, &sp))
        return 0;
    return tts::attn_workspace_bytes(B, num_kv_heads, head_dim, sp);
}

extern "C" int tts_decode_attn(const tts_kv_cache *cache, const int32_t *d_block_table,
                               int32_t max_blocks_per_seq, const int32_t *d_ctx_lens,
                               int32_t max_ctx_len, int32_t B, int32_t q_len, int32_t num_q_heads,
                               float scale, int32_t causal, const void *d_q, void *d_out,
                               void *d_ws, size_t ws_bytes, int32_t *d_err, void *stream) {
    using namespace tts;
    if (!cache || !d_block_table || !d_ctx_lens || !d_q || !d_out) return TTS_ERR_INVALID;
    if (!cache->k_pool || !cache->v_pool || cache->num_blocks < 1) return TTS_ERR_INVALID;
    if (B < 0 || B > 65535 || q_len < 1 || max_blocks_per_seq < 1 ||
        max_blocks_per_seq > (1 << 20) || !(scale > 0.0f) || scale != scale)
        return TTS_ERR_INVALID;
    if (cache->block_size != TTS_BLOCK_TOKENS) return TTS_ERR_UNSUPPORTED;
    if (!supported_head(cache->dtype, cache->head_dim)) return TTS_ERR_UNSUPPORTED;
    if (cache->num_kv_heads < 1 || cache->num_kv_heads > 65535) return TTS_ERR_INVALID;
    if (B == 0) return TTS_OK;
    AttnSplit sp;
    if (!attn_split_policy(B, q_len, num_q_heads, cache->num_kv_heads, cache->head_dim,
                           max_ctx_len, &sp)) {
        const int nh = cache->num_kv_heads;
        const bool shape_ok = num_q_heads >= nh && num_q_heads % nh == 0 && max_ctx_len >= q_len &&
                              max_ctx_len <= (1 << 24);
        return shape_ok ? TTS_ERR_UNSUPPORTED : TTS_ERR_INVALID;
    }
    if (!aligned16(cache->k_pool) || !aligned16(cache->v_pool) || !aligned16(d_q))
        return TTS_ERR_INVALID;
    const size_t need = attn_workspace_bytes(B, cache->num_kv_heads, cache->head_dim, sp);
    if (!d_ws || ws_bytes < need || (reinterpret_cast<uintptr_t>(d_ws) & 255u) != 0)
        return TTS_ERR_WORKSPACE;

    const size_t units =
        static_cast<size_t>(B) * cache->num_kv_heads * sp.max_splits * sp.rows;
    uint8_t *ws = static_cast<uint8_t *>(d_ws);
    AttnArgs a;
    a.k_pool = static_cast<const uint8_t *>(cache->k_pool);
    a.v_pool = static_cast<const uint8_t *>(cache->v_pool);
    a.num_blocks = cache->num_blocks;
    a.Hkv = cache->num_kv_heads;
    a.table = d_block_table;
    a.max_blocks = max_blocks_per_seq;
    a.ctx_lens = d_ctx_lens;
    a.max_ctx = max_ctx_len;
    a.q_len = q_len;
    a.Hq = num_q_heads;
    a.group = num_q_heads / cache->num_kv_heads;
    a.causal = causal ? 1 : 0;
    a.qscale = scale * kLog2e;
    a.q = d_q;
    a.out = d_out;
    a.o_part = reinterpret_cast<float *>(ws);
    a.ml_part = reinterpret_cast<float2 *>(ws + align_up(units * cache->head_dim * sizeof(float), 256));
    a.counters = reinterpret_cast<int32_t *>(ws + align_up(units * cache->head_dim * sizeof(float), 256) +
                                             align_up(units * sizeof(float2), 256));
    a.max_splits = sp.max_splits;
    a.split_blocks = sp.blocks;
    a.err = d_err;
    const dim3 grid(sp.max_splits, cache->num_kv_heads, B);
    if (grid.x > 0x7FFFFFFFu) return TTS_ERR_INVALID;
    auto s = static_cast<cudaStream_t>(stream);
    return cache->dtype == TTS_BF16 ? launch_typed<__nv_bfloat16>(a, sp.rows, grid, s)
                                    : launch_typed<float>(a, sp.rows, grid, s);
}

// ---------------------------------------------------------------------------
// Decode attention without a caller workspace.
//
// Some callers cannot allocate device memory where they run a decode step:
// code that runs while a CUDA graph is being captured (an allocation there
// breaks the capture), engines that reserve all free device memory for the KV
// pool at start-up and so leave nothing for cudaMalloc, hosts that hand a
// plugin no allocator, and real-time loops that cannot afford the implicit
// synchronisation and unbounded latency of cudaMalloc / cudaFree inside a
// frame deadline.  For them the split-KV partials live in one file-scope
// device array of fixed size instead of a caller workspace.  Every GPU that
// loads this library holds the array until the process exits.

namespace tts {
namespace {

constexpr size_t kStaticScratchBytes = size_t(16) << 20;  // 16 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_attn_scratch[kStaticScratchBytes];

std::mutex g_scratch_mu;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of g_attn_scratch on the current device.  The symbol's name
// in host code is only a host-side handle, so the address is looked up once
// per device (with that device current) and cached.
int static_scratch_address(void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return TTS_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return TTS_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_attn_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return TTS_ERR_CUDA;
        }
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return TTS_OK;
}

}  // namespace
}  // namespace tts

extern "C" int tts_decode_attn_noalloc(const tts_kv_cache *cache, const int32_t *d_block_table,
                                       int32_t max_blocks_per_seq, const int32_t *d_ctx_lens,
                                       int32_t max_ctx_len, int32_t B, int32_t q_len,
                                       int32_t num_q_heads, float scale, int32_t causal,
                                       const void *d_q, void *d_out, int32_t *d_err, void *stream) {
    using namespace tts;
    if (!cache) return TTS_ERR_INVALID;
    const size_t need = tts_decode_attn_workspace_size(B, q_len, num_q_heads, cache->num_kv_heads,
                                                       cache->head_dim, max_ctx_len);
    if (B == 0 || need == 0)  // nothing to run, or arguments the regular entry point rejects
        return tts_decode_attn(cache, d_block_table, max_blocks_per_seq, d_ctx_lens, max_ctx_len, B,
                               q_len, num_q_heads, scale, causal, d_q, d_out, nullptr, 0, d_err,
                               stream);
    if (need > kStaticScratchBytes) return TTS_ERR_SCRATCH_LIMIT;
    void *scratch = nullptr;
    const int st = static_scratch_address(&scratch);
    if (st != TTS_OK) return st;
    // The split tickets must start at zero; they sit at the end of the
    // workspace layout.  The array keeps whatever the previous call left.
    const size_t tickets = align_up(static_cast<size_t>(B) * cache->num_kv_heads * sizeof(int32_t), 256);
    if (cudaMemsetAsync(static_cast<uint8_t *>(scratch) + need - tickets, 0, tickets,
                        static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return TTS_ERR_CUDA;
    }
    return tts_decode_attn(cache, d_block_table, max_blocks_per_seq, d_ctx_lens, max_ctx_len, B,
                           q_len, num_q_heads, scale, causal, d_q, d_out, scratch, need, d_err,
                           stream);
}
