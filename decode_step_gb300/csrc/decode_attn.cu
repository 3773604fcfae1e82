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
// How (HBM-bound: each cached byte feeds 2 flops per query row):
//  - The work is the flat list of (stream, KV head, 16-token block) tiles,
//    stream-major.  A persistent grid of warps splits that list into equal
//    contiguous ranges (a warp-granular stream-K schedule), so every warp
//    streams the same number of tiles whatever the context-length mix, and a
//    (stream, KV head) "segment" is split across warps only where a range
//    boundary falls inside it.  Each CTA first scans the context lengths into
//    a per-stream tile prefix in shared memory.
//  - Each warp streams its tiles' K and V (4 KB each, contiguous in the pool)
//    through a private 2-stage shared-memory ring with bulk TMA copies (L2
//    evict-first), completion on per-stage mbarriers; the query rows of a new
//    segment ride along in the same stage.  Block ids are fetched 32 tiles at
//    a time, one batch ahead.
//  - Lane (p, c) = (lane / 16, lane % 16) reads 16-byte chunk c of the rows
//    of tokens p, p + 2, ..., p + 14 (conflict-free 128-bit shared loads).
//    Dot products are reduced across the 16 chunk lanes by recursive halving
//    (each shuffle round halves the values a lane carries), leaving every lane
//    the full scores of one token for half of the query rows.  Online softmax
//    in the log2 domain with warp-shuffle max reductions; P.V accumulates per
//    lane into its 16-byte slice of the output rows.  All group x q_len query
//    rows of a KV head share one read of each tile.
//  - A segment wholly inside a warp's range is written out directly.  A split
//    segment's warps write (m, l, unnormalised o) partials; the last of them
//    to finish (an atomic ticket, never a wait) merges the partials with a
//    log-sum-exp combine and writes the output.
#include <mutex>

#include "tts_common.cuh"
#include "tts_internal.h"

namespace tts {
namespace {

constexpr int kWarps = 4;          // warps per CTA
constexpr int kStages = 2;         // pipeline depth per warp
constexpr int kTileBytes = 4096;   // one (block, KV head) tile of K or V: 16 tokens x 256 B
constexpr int kRowBytes = 256;     // one token's key (or value) row
constexpr int kMaxStreams = 4096;  // streams per call (shared-memory prefix table)
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
    int B;
    int q_len;
    int Hq;
    int group;
    int causal;
    float qscale;       // softmax scale * log2(e)
    const uint8_t *q;
    void *out;
    float *part;        // [workers][2][NR * D + 2 * NR]: o, m, l of split segments
    int32_t *counters;  // [B][Hkv] tickets of split segments
    int workers;
    int32_t *err;
};

template <int NR, int D>
struct AttnSmem {
    static constexpr int stage_bytes = 2 * kTileBytes + NR * kRowBytes;  // K, V, query rows
    static constexpr size_t stages = 0;
    static constexpr size_t bars = stages + size_t(kWarps) * kStages * stage_bytes;
    static constexpr size_t pbuf = bars + 8 * kWarps * kStages;
    static constexpr size_t prefix = pbuf + 4 * kWarps * 16 * NR;
    // then: int prefix[B + 1], int ctxs[B], int scan[kWarps]
    static size_t total(int B) { return prefix + 4 * (2 * size_t(B) + 1 + kWarps); }
};

__device__ __forceinline__ int warp_of_tile(long long t, long long T, long long W) {
    return static_cast<int>(((t + 1) * W - 1) / T);
}
__device__ __forceinline__ long long range_start(long long w, long long T, long long W) {
    return w * T / W;
}

template <typename T, int NR>
__global__ void __launch_bounds__(kWarps * 32, NR <= 4 ? 3 : 1)
decode_attn_kernel(const AttnArgs a) {
    using C = Chunk<T>;
    constexpr int EPC = C::N;          // elements per 16-byte chunk
    constexpr int D = 16 * EPC;        // head dim: one 256-byte row per token
    constexpr int HALF = NR / 2;
    constexpr int SF = NR * D + 2 * NR;  // floats per partial slot
    using S = AttnSmem<NR, D>;
    extern __shared__ __align__(1024) uint8_t smem[];
    int *prefix = reinterpret_cast<int *>(smem + S::prefix);  // [B + 1], in tiles
    int *ctxs = prefix + a.B + 1;                              // [B], 0 for an invalid stream
    int *scan = ctxs + a.B;                                    // [kWarps]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_rows = a.group * a.q_len;
    const int cap = min(a.max_ctx, a.max_blocks * TTS_BLOCK_TOKENS);
    T *out = static_cast<T *>(a.out);
    const size_t row_stride = static_cast<size_t>(a.Hq) * D;  // elements between query positions

    // ---- 1. context lengths -> per-stream tile prefix (x Hkv, stream-major)
    {
        const int per = (a.B + blockDim.x - 1) / blockDim.x;
        const int i0 = threadIdx.x * per, i1 = min(a.B, i0 + per);
        int local = 0;
        for (int i = i0; i < i1; ++i) {
            const int L = __ldg(a.ctx_lens + i);
            const bool ok = L >= a.q_len && L <= cap;
            ctxs[i] = ok ? L : 0;
            local += ok ? (L + TTS_BLOCK_TOKENS - 1) / TTS_BLOCK_TOKENS : 0;
            if (!ok && blockIdx.x == 0) {
                flag_error(a.err, TTS_ERRBIT_CTX_LEN);
                T *o = out + static_cast<size_t>(i) * a.q_len * row_stride;
                for (size_t e = 0; e < a.q_len * row_stride; ++e) store_elem(o + e, 0.0f);
            }
        }
        int incl = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += v;
        }
        if (lane == 31) scan[warp] = incl;
        __syncthreads();
        int run = incl - local, total = 0;
        for (int w = 0; w < kWarps; ++w) {
            if (w < warp) run += scan[w];
            total += scan[w];
        }
        for (int i = i0; i < i1; ++i) {
            prefix[i] = run * a.Hkv;
            run += ctxs[i] ? (ctxs[i] + TTS_BLOCK_TOKENS - 1) / TTS_BLOCK_TOKENS : 0;
        }
        if (threadIdx.x == 0) prefix[a.B] = total * a.Hkv;
        __syncthreads();
    }

    // ---- 2. this warp's tile range
    // Every participating warp gets at least one tile (warps beyond the tile
    // count sit out), so a split segment's contributors are consecutive warps.
    const long long Ttot = prefix[a.B];
    const long long Wtot = min(static_cast<long long>(a.workers), Ttot);
    const int wid = blockIdx.x * kWarps + warp;
    if (Ttot == 0 || wid >= Wtot) return;
    const int t0 = static_cast<int>(range_start(wid, Ttot, Wtot));
    const int t1 = static_cast<int>(range_start(wid + 1, Ttot, Wtot));
    const int n = t1 - t0;
    if (n <= 0) return;

    const uint32_t stage0 = smem_addr(smem + S::stages) + warp * kStages * S::stage_bytes;
    const uint32_t bar0 = smem_addr(smem + S::bars) + 8 * warp * kStages;
    float *pbuf = reinterpret_cast<float *>(smem + S::pbuf) + warp * 16 * NR;
    if (lane == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(bar0 + 8 * s, 1);
        fence_mbar_init();
    }
    __syncwarp();

    // Tile metadata, 32 tiles per batch (lane i holds tile 32 k + i of the
    // range): raw block id (validated when used), segment = stream * Hkv + head,
    // block index within the stream.
    auto load_meta = [&](int k, int &id, int &seg, int &blk) {
        const int t = t0 + 32 * k + lane;
        id = -1;
        seg = -1;
        blk = 0;
        if (t < t1) {
            int lo = 0, hi = a.B;  // prefix[lo] <= t < prefix[hi]
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (prefix[mid] <= t) lo = mid; else hi = mid;
            }
            const int nb = (prefix[lo + 1] - prefix[lo]) / a.Hkv;
            const int r = t - prefix[lo];
            const int g = r / nb;
            blk = r - g * nb;
            seg = lo * a.Hkv + g;
            id = __ldg(a.table + static_cast<size_t>(lo) * a.max_blocks + blk);
        }
    };
    int cur_id, cur_seg, cur_blk, nxt_id = -1, nxt_seg = -1, nxt_blk = 0;
    load_meta(0, cur_id, cur_seg, cur_blk);
    if (n > 32) load_meta(1, nxt_id, nxt_seg, nxt_blk);
    int kc = 0;  // batch of the tile being computed

    const uint64_t policy = l2_evict_first_policy();
    const int qbytes_per_pos = a.group * D * static_cast<int>(sizeof(T));
    auto issue = [&](int j) {
        const bool in_cur = (j >> 5) == kc;
        const int src = j & 31;
        int id = __shfl_sync(kFull, in_cur ? cur_id : nxt_id, src);
        const int seg = __shfl_sync(kFull, in_cur ? cur_seg : nxt_seg, src);
        const int blk = __shfl_sync(kFull, in_cur ? cur_blk : nxt_blk, src);
        if (lane == 0) {
            if (id < 0 || id >= a.num_blocks) {
                flag_error(a.err, TTS_ERRBIT_BLOCK_ID);
                id = -1;
            }
            const int st = j % kStages;
            const uint32_t bar = bar0 + 8 * st;
            const uint32_t dst = stage0 + st * S::stage_bytes;
            const bool need_q = j == 0 || blk == 0;
            const uint32_t bytes = (id >= 0 ? 2 * kTileBytes : 0) + (need_q ? a.q_len * qbytes_per_pos : 0);
            if (bytes == 0) {
                mbar_arrive(bar);
            } else {
                mbar_arrive_expect_tx(bar, bytes);
                if (id >= 0) {
                    const size_t off = (static_cast<size_t>(id) * a.Hkv + seg % a.Hkv) * kTileBytes;
                    bulk_load(dst, a.k_pool + off, kTileBytes, bar, policy);
                    bulk_load(dst + kTileBytes, a.v_pool + off, kTileBytes, bar, policy);
                }
                if (need_q) {
                    const int b = seg / a.Hkv, g = seg % a.Hkv;
                    for (int jq = 0; jq < a.q_len; ++jq) {
                        const size_t qoff =
                            ((static_cast<size_t>(b) * a.q_len + jq) * a.Hq + g * a.group) * D * sizeof(T);
                        bulk_load_nohint(dst + 2 * kTileBytes + jq * qbytes_per_pos, a.q + qoff,
                                         qbytes_per_pos, bar);
                    }
                }
            }
        }
    };
    for (int j = 0; j < min(kStages, n); ++j) issue(j);

    const int p = lane >> 4, c = lane & 15;
    const int my_tok = p + 2 * ((lane >> 1) & 7);
    // State of the current segment.
    int seg_id = -1, seg_b = 0, seg_g = 0, seg_L = 0, s0 = 0, s1 = 0;
    int lim[HALF];
    float q[NR][EPC], m_run[HALF], l_run[HALF], o[NR][EPC];

    auto flush = [&]() {
        float l_tot[HALF], l_oth[HALF];
#pragma unroll
        for (int k = 0; k < HALF; ++k) {
            float l = l_run[k];
            l += __shfl_xor_sync(kFull, l, 2);
            l += __shfl_xor_sync(kFull, l, 4);
            l += __shfl_xor_sync(kFull, l, 8);
            l += __shfl_xor_sync(kFull, l, 16);
            l_tot[k] = l;
            l_oth[k] = __shfl_xor_sync(kFull, l, 1);
        }
#pragma unroll
        for (int r = 0; r < NR; ++r)
#pragma unroll
            for (int e = 0; e < EPC; ++e) o[r][e] += __shfl_xor_sync(kFull, o[r][e], 16);
        if (s0 >= t0 && s1 <= t1) {
            // whole segment in this warp: write the output
            if (lane < 16) {
#pragma unroll
                for (int r = 0; r < NR; ++r) {
                    if (r >= n_rows) break;
                    const float l = (r / HALF) == (lane & 1) ? l_tot[r % HALF] : l_oth[r % HALF];
                    const float inv = l > 0.0f ? 1.0f / l : 0.0f;
                    const int j = r / a.group, hh = r % a.group;
                    T *dst = out + (static_cast<size_t>(seg_b) * a.q_len + j) * row_stride +
                             static_cast<size_t>(seg_g * a.group + hh) * D + c * EPC;
#pragma unroll
                    for (int e = 0; e < EPC; ++e) store_elem(dst + e, o[r][e] * inv);
                }
            }
            return;
        }
        // split segment: publish this warp's partial, the last contributor merges
        const int slot = s0 <= t0 ? 0 : 1;
        float *part = a.part + (static_cast<size_t>(wid) * 2 + slot) * SF;
        if (lane < 16) {
#pragma unroll
            for (int r = 0; r < NR; ++r)
#pragma unroll
                for (int e = 0; e < EPC; ++e) part[r * D + c * EPC + e] = o[r][e];
        }
        if (lane < 2) {
#pragma unroll
            for (int k = 0; k < HALF; ++k) {
                part[NR * D + lane * HALF + k] = m_run[k];
                part[NR * D + NR + lane * HALF + k] = l_tot[k];
            }
        }
        __threadfence();
        __syncwarp();
        const int w_first = warp_of_tile(s0, Ttot, Wtot);
        const int w_last = warp_of_tile(s1 - 1, Ttot, Wtot);
        int last = 0;
        if (lane == 0) last = atomicAdd(a.counters + seg_id, 1) == w_last - w_first;
        if (!__shfl_sync(kFull, last, 0)) return;
        __threadfence();
        const bool first_shifted = range_start(w_first, Ttot, Wtot) != s0;
        for (int r = p; r < n_rows; r += 2) {
            float M = kNegBig;
            for (int w2 = w_first; w2 <= w_last; ++w2) {
                const float *pp = a.part + (static_cast<size_t>(w2) * 2 + (w2 == w_first && first_shifted)) * SF;
                M = fmaxf(M, __ldcg(pp + NR * D + r));
            }
            float Ls = 0.0f, O[EPC];
#pragma unroll
            for (int e = 0; e < EPC; ++e) O[e] = 0.0f;
            for (int w2 = w_first; w2 <= w_last; ++w2) {
                const float *pp = a.part + (static_cast<size_t>(w2) * 2 + (w2 == w_first && first_shifted)) * SF;
                const float f = exp2f(__ldcg(pp + NR * D + r) - M);
                Ls = fmaf(__ldcg(pp + NR * D + NR + r), f, Ls);
#pragma unroll
                for (int e = 0; e < EPC; ++e) O[e] = fmaf(__ldcg(pp + r * D + c * EPC + e), f, O[e]);
            }
            const float inv = Ls > 0.0f ? 1.0f / Ls : 0.0f;
            const int j = r / a.group, hh = r % a.group;
            T *dst = out + (static_cast<size_t>(seg_b) * a.q_len + j) * row_stride +
                     static_cast<size_t>(seg_g * a.group + hh) * D + c * EPC;
#pragma unroll
            for (int e = 0; e < EPC; ++e) store_elem(dst + e, O[e] * inv);
        }
        if (lane == 0) a.counters[seg_id] = 0;
    };

    bool timed_out = false;
    int waited = 0;
    for (int i = 0; i < n; ++i) {
        if ((i & 31) == 0 && i > 0) {
            kc = i >> 5;
            cur_id = nxt_id; cur_seg = nxt_seg; cur_blk = nxt_blk;
            if (n > 32 * (kc + 1)) load_meta(kc + 1, nxt_id, nxt_seg, nxt_blk);
        }
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
        const int src = i & 31;
        const int t_id = __shfl_sync(kFull, cur_id, src);
        const int t_seg = __shfl_sync(kFull, cur_seg, src);
        const int t_blk = __shfl_sync(kFull, cur_blk, src);
        const uint32_t ks = stage0 + st * S::stage_bytes, vs = ks + kTileBytes;
        if (i == 0 || t_blk == 0) {
            // ---- a new segment: finish the previous one, set up this one
            if (i > 0) flush();
            seg_id = t_seg;
            seg_b = t_seg / a.Hkv;
            seg_g = t_seg % a.Hkv;
            seg_L = ctxs[seg_b];
            const int nb = (seg_L + TTS_BLOCK_TOKENS - 1) / TTS_BLOCK_TOKENS;
            s0 = prefix[seg_b] + seg_g * nb;
            s1 = s0 + nb;
#pragma unroll
            for (int k = 0; k < HALF; ++k) {
                const int r = (lane & 1) * HALF + k;
                lim[k] = r < n_rows ? (a.causal ? seg_L - a.q_len + r / a.group + 1 : seg_L) : 0;
                m_run[k] = kNegBig;
                l_run[k] = 0.0f;
            }
            const uint32_t qs = ks + 2 * kTileBytes;
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                if (r < n_rows && !timed_out) {
                    C::unpack(lds128(qs + r * kRowBytes + c * 16), q[r]);
#pragma unroll
                    for (int e = 0; e < EPC; ++e) q[r][e] *= a.qscale;
                } else {
#pragma unroll
                    for (int e = 0; e < EPC; ++e) q[r][e] = 0.0f;
                }
#pragma unroll
                for (int e = 0; e < EPC; ++e) o[r][e] = 0.0f;
            }
        }
        if (!timed_out && t_id >= 0 && t_id < a.num_blocks) {
            const int base = t_blk * TTS_BLOCK_TOKENS;
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
                const int nv = (8 * NR) >> step;
                const bool upper = (lane & m) != 0;
#pragma unroll
                for (int x = 0; x < nv / 2; ++x) {
                    const float send = upper ? acc[x] : acc[x + nv / 2];
                    const float keep = upper ? acc[x + nv / 2] : acc[x];
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
                if (base + t >= seg_L) raw = make_uint4(0u, 0u, 0u, 0u);  // past the context
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
        if (!timed_out && i + kStages < n) issue(i + kStages);
    }
    flush();
    if (timed_out) {
        // Let copies still in flight land before the CTA's shared memory goes away.
        const int issued = min(n, waited + kStages);
        for (int i = waited; i < issued; ++i) mbar_wait(bar0 + 8 * (i % kStages), (i / kStages) & 1);
    }
}

// Row templates: group * q_len rows are padded up to one of these.
constexpr int kRowTemplates[] = {2, 4, 8, 10, 16};

int padded_rows(int rows) {
    for (int r : kRowTemplates)
        if (rows <= r) return r;
    return 0;
}

int ctas_per_sm(int nr) { return nr <= 4 ? 3 : 1; }

int device_sms() {
    const int n = sm_count();
    return n > 0 ? n : 160;  // no device visible (size queries on a build host)
}

template <typename T, int NR>
int launch_nr(const AttnArgs &a, int ctas, cudaStream_t stream) {
    constexpr int D = 16 * Chunk<T>::N;
    const size_t smem = AttnSmem<NR, D>::total(a.B);
    auto kern = decode_attn_kernel<T, NR>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
        return TTS_ERR_CUDA;
    kern<<<ctas, kWarps * 32, smem, stream>>>(a);
    return launch_status();
}

template <typename T>
int launch_typed(const AttnArgs &a, int nr, int ctas, cudaStream_t stream) {
    switch (nr) {
        case 2: return launch_nr<T, 2>(a, ctas, stream);
        case 4: return launch_nr<T, 4>(a, ctas, stream);
        case 8: return launch_nr<T, 8>(a, ctas, stream);
        case 10: return launch_nr<T, 10>(a, ctas, stream);
        case 16: return launch_nr<T, 16>(a, ctas, stream);
        default: return TTS_ERR_UNSUPPORTED;
    }
}

bool supported_head(int dtype, int head_dim) {
    return (dtype == TTS_BF16 && head_dim == 128) || (dtype == TTS_F32 && head_dim == 64);
}

}  // namespace

bool attn_plan(int B, int q_len, int num_q_heads, int num_kv_heads, int head_dim,
               int max_ctx_len, AttnPlan *out) {
    if (B < 1 || q_len < 1 || num_kv_heads < 1 || num_q_heads < num_kv_heads ||
        num_q_heads % num_kv_heads != 0 || head_dim < 1 || max_ctx_len < q_len ||
        max_ctx_len > (1 << 24))
        return false;
    const int rows = padded_rows((num_q_heads / num_kv_heads) * q_len);
    if (rows == 0 || B > kMaxStreams) return false;
    const long long nblk = (max_ctx_len + TTS_BLOCK_TOKENS - 1) / TTS_BLOCK_TOKENS;
    if (static_cast<long long>(B) * num_kv_heads * nblk >= (1LL << 31)) return false;
    out->rows = rows;
    out->ctas = device_sms() * ctas_per_sm(rows);
    out->workers = out->ctas * kWarps;
    return true;
}

size_t attn_workspace_bytes(int B, int num_kv_heads, int head_dim, const AttnPlan &pl) {
    const size_t slot = static_cast<size_t>(pl.rows) * head_dim + 2 * pl.rows;
    return align_up(static_cast<size_t>(pl.workers) * 2 * slot * sizeof(float), 256) +
           align_up(static_cast<size_t>(B) * num_kv_heads * sizeof(int32_t), 256);
}

}  // namespace tts

extern "C" size_t tts_decode_attn_workspace_size(int32_t B, int32_t q_len, int32_t num_q_heads,
                                                 int32_t num_kv_heads, int32_t head_dim,
                                                 int32_t max_ctx_len) {
    tts::AttnPlan pl;
    if (!tts::attn_plan(B, q_len, num_q_heads, num_kv_heads, head_dim, max_ctx_len, &pl))
        return 0;
    return tts::attn_workspace_bytes(B, num_kv_heads, head_dim, pl);
}

extern "C" int tts_decode_attn(const tts_kv_cache *cache, const int32_t *d_block_table,
                               int32_t max_blocks_per_seq, const int32_t *d_ctx_lens,
                               int32_t max_ctx_len, int32_t B, int32_t q_len, int32_t num_q_heads,
                               float scale, int32_t causal, const void *d_q, void *d_out,
                               void *d_ws, size_t ws_bytes, int32_t *d_err, void *stream) {
    using namespace tts;
    if (!cache || !d_block_table || !d_ctx_lens || !d_q || !d_out) return TTS_ERR_INVALID;
    if (!cache->k_pool || !cache->v_pool || cache->num_blocks < 1) return TTS_ERR_INVALID;
    if (B < 0 || q_len < 1 || max_blocks_per_seq < 1 || max_blocks_per_seq > (1 << 20) ||
        !(scale > 0.0f) || scale != scale)
        return TTS_ERR_INVALID;
    if (cache->block_size != TTS_BLOCK_TOKENS) return TTS_ERR_UNSUPPORTED;
    if (!supported_head(cache->dtype, cache->head_dim)) return TTS_ERR_UNSUPPORTED;
    if (cache->num_kv_heads < 1) return TTS_ERR_INVALID;
    if (B == 0) return TTS_OK;
    AttnPlan pl;
    if (!attn_plan(B, q_len, num_q_heads, cache->num_kv_heads, cache->head_dim, max_ctx_len, &pl)) {
        const int nh = cache->num_kv_heads;
        const bool shape_ok = num_q_heads >= nh && num_q_heads % nh == 0 && max_ctx_len >= q_len &&
                              max_ctx_len <= (1 << 24);
        return shape_ok ? TTS_ERR_UNSUPPORTED : TTS_ERR_INVALID;
    }
    if (!aligned16(cache->k_pool) || !aligned16(cache->v_pool) || !aligned16(d_q))
        return TTS_ERR_INVALID;
    const size_t need = attn_workspace_bytes(B, cache->num_kv_heads, cache->head_dim, pl);
    if (!d_ws || ws_bytes < need || (reinterpret_cast<uintptr_t>(d_ws) & 255u) != 0)
        return TTS_ERR_WORKSPACE;

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
    a.B = B;
    a.q_len = q_len;
    a.Hq = num_q_heads;
    a.group = num_q_heads / cache->num_kv_heads;
    a.causal = causal ? 1 : 0;
    a.qscale = scale * kLog2e;
    a.q = static_cast<const uint8_t *>(d_q);
    a.out = d_out;
    a.part = reinterpret_cast<float *>(ws);
    a.counters = reinterpret_cast<int32_t *>(
        ws + need - align_up(static_cast<size_t>(B) * cache->num_kv_heads * sizeof(int32_t), 256));
    a.workers = pl.workers;
    a.err = d_err;
    auto s = static_cast<cudaStream_t>(stream);
    return cache->dtype == TTS_BF16 ? launch_typed<__nv_bfloat16>(a, pl.rows, pl.ctas, s)
                                    : launch_typed<float>(a, pl.rows, pl.ctas, s);
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

constexpr size_t kStaticScratchBytes = size_t(8) << 20;  // 8 MiB
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
