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
// Work distribution (shared by both kernels).  The work is the flat list of
// (stream, KV head, 16-token block) tiles, stream-major.  A persistent grid of
// warps splits it into equal contiguous ranges (a warp-granular stream-K
// schedule), so every warp streams the same number of tiles whatever the
// context-length mix; a (stream, KV head) "segment" is split across warps only
// where a range boundary falls inside it.  A segment wholly inside one range
// is written out directly; a split segment's warps publish (m, l, o) partials
// and the last of them (an atomic ticket, never a wait) merges them with a
// log-sum-exp combine.  Each warp streams its tiles through a private 2-stage
// shared-memory ring filled by TMA (L2 evict-first for the cache), completion
// on per-stage mbarriers; a new segment's query rows ride in the same stage.
//
// bf16 (head_dim 128): the per-tile products S = Q K^T and O += P V run as
// mma.sync m16n8k16 (bf16 in, fp32 accumulate) on all group x q_len query rows
// of the KV head at once (padded to 16).  Each KV byte is still read once from
// HBM; the tensor-core instructions only replace the ~8 bf16->fp32 converts
// and FMAs per element that would otherwise make the kernel issue-bound at
// GB300's bandwidth per SM.  K/V tiles arrive through 2-D TMA with a 128-byte
// swizzle, so the ldmatrix fragment loads are bank-conflict free.  Softmax
// (row max, exp2, running sums) is fp32 with warp shuffles among the four
// lanes that share a query row.
//
// fp32 (head_dim 64): CUDA cores.  Lane (p, c) reads 16-byte chunk c of tokens
// p, p + 2, ...; dot products are reduced across the 16 chunk lanes by
// recursive halving, leaving every lane the full scores of one token for half
// of the query rows.
#include <cudaTypedefs.h>

#include <mutex>
#include <new>

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
    float *part;        // [workers][2][nr_slot * D + 2 * nr_slot]: o, m, l of split segments
    int32_t *counters;  // [B][Hkv] tickets of split segments
    int workers;
    int nr_slot;        // query rows per partial slot (group * q_len padded)
    int stages;         // ring depth per warp (tensor-core kernel)
    int32_t *err;
    long long wait_limit;  // SM clock cycles per bounded wait
    int stall;             // test support: first ring stage expects 16 bytes that never come
};

// The work partition: Wtot warps share the flat list of T tiles in order,
// the first rem = T mod Wtot warps taking q + 1 tiles and the others q = T /
// Wtot (32-bit arithmetic: the merges evaluate these at every split segment).
struct Part {
    int q, rem;
};
__device__ __forceinline__ Part make_part(long long T, long long W) {
    Part p;
    p.q = static_cast<int>(T / W);
    p.rem = static_cast<int>(T - static_cast<long long>(p.q) * W);
    return p;
}
__device__ __forceinline__ int range_start(const Part &p, int w) { return w * p.q + min(w, p.rem); }
__device__ __forceinline__ int warp_of_tile(const Part &p, int t) {
    const int big = p.rem * (p.q + 1);
    return t < big ? t / (p.q + 1) : p.rem + (t - big) / p.q;
}

// Context lengths -> per-stream tile prefix (x Hkv, stream-major) in shared
// memory; invalid streams get no tiles, zero outputs (CTA 0) and an error bit.
// Called by every thread of the CTA.
template <typename T, int D, int WARPS>
__device__ void scan_streams(const AttnArgs &a, int *prefix, int *ctxs, int *scan) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cap = min(a.max_ctx, a.max_blocks * TTS_BLOCK_TOKENS);
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
            T *o = static_cast<T *>(a.out) + static_cast<size_t>(i) * a.q_len * a.Hq * D;
            for (int e = 0; e < a.q_len * a.Hq * D; ++e) store_elem(o + e, 0.0f);
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
    for (int w = 0; w < WARPS; ++w) {
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

// Tile t of the flat list -> (raw block id, segment = stream * Hkv + head,
// block index in the stream); t must be < prefix[B].  The block id load is
// left in flight (validated where it is used).
__device__ __forceinline__ void tile_meta(const AttnArgs &a, const int *prefix, int t, int &id,
                                          int &seg, int &blk) {
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

// Output pointer of query row r (= j * group + hh) of segment (b, g).
template <typename T, int D>
__device__ __forceinline__ T *out_row(const AttnArgs &a, int b, int g, int r) {
    const int j = r / a.group, hh = r % a.group;
    return static_cast<T *>(a.out) + ((static_cast<size_t>(b) * a.q_len + j) * a.Hq + g * a.group + hh) * D;
}

// Warps given tiles: at least kMinTilesPerWarp each when the work is small
// (fewer split segments to publish and merge), but never fewer warps than
// segments (B x Hkv): short segments gain nothing from sharing a warp and
// would only run one after another; else every warp of the grid.
constexpr long long kMinTilesPerWarp = 4;
__device__ __forceinline__ long long active_workers(int workers, long long Ttot, long long segments) {
    long long w = (Ttot + kMinTilesPerWarp - 1) / kMinTilesPerWarp;
    w = w > segments ? w : segments;
    return min(static_cast<long long>(workers), w > 0 ? w : 1);
}

// The last contributor of a split segment merges the contributors' partials
// (log-sum-exp combine).  Output unit = 4 dims of one query row; a lane takes
// two units (u and u + 32) per pass and, per batch of 4 contributors, issues
// every load both need (each contributor's row maximum, row sum and 4 output
// dims) before using any, so a merge of up to 4 contributors costs one
// dependent round trip per 64 units (per 2 query rows at head_dim 128)
// instead of one per row for the maxima and another for the outputs.
// Batches fold in with a running maximum.
template <typename T, int D>
__device__ void merge_split_segment(const AttnArgs &a, int b, int g, int n_rows, int w_first,
                                    int w_last, bool first_shifted, int lane) {
    constexpr int UPR = D / 4;  // float4 units per row
    constexpr int CB = 4;       // contributors per batch
    const int NRS = a.nr_slot;
    const size_t SF = static_cast<size_t>(NRS) * D + 2 * NRS;
    const size_t ML = static_cast<size_t>(NRS) * D;  // offset of the maxima; sums follow
    const int nc = w_last - w_first + 1;
    const int units = n_rows * UPR;
    auto slot = [&](int i) -> const float * {
        return a.part + (static_cast<size_t>(w_first + i) * 2 + (i == 0 && first_shifted)) * SF;
    };
    for (int u0 = lane; u0 < units; u0 += 64) {
        int rr[2], cc[2];
        bool has[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int u = u0 + 32 * h;
            has[h] = u < units;
            rr[h] = has[h] ? u / UPR : 0;
            cc[h] = has[h] ? u - rr[h] * UPR : 0;
        }
        float M[2] = {kNegBig, kNegBig}, L[2] = {0.0f, 0.0f};
        float4 O[2] = {make_float4(0.0f, 0.0f, 0.0f, 0.0f), make_float4(0.0f, 0.0f, 0.0f, 0.0f)};
        for (int c0 = 0; c0 < nc; c0 += CB) {
            float mi[2][CB], li[2][CB];
            float4 oi[2][CB];
#pragma unroll
            for (int k = 0; k < CB; ++k) {
                const bool in = c0 + k < nc;
                const float *pk = in ? slot(c0 + k) : nullptr;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    if (in && has[h]) {
                        mi[h][k] = __ldcg(pk + ML + rr[h]);
                        li[h][k] = __ldcg(pk + ML + NRS + rr[h]);
                        oi[h][k] = __ldcg(reinterpret_cast<const float4 *>(pk + static_cast<size_t>(rr[h]) * D) + cc[h]);
                    } else {
                        mi[h][k] = kNegBig;
                        li[h][k] = 0.0f;
                        oi[h][k] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                    }
                }
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                float Mn = M[h];
#pragma unroll
                for (int k = 0; k < CB; ++k) Mn = fmaxf(Mn, mi[h][k]);
                const float sc = exp2f(M[h] - Mn);
                L[h] *= sc;
                O[h].x *= sc; O[h].y *= sc; O[h].z *= sc; O[h].w *= sc;
#pragma unroll
                for (int k = 0; k < CB; ++k) {
                    const float f = exp2f(mi[h][k] - Mn);
                    L[h] = fmaf(li[h][k], f, L[h]);
                    O[h].x = fmaf(oi[h][k].x, f, O[h].x);
                    O[h].y = fmaf(oi[h][k].y, f, O[h].y);
                    O[h].z = fmaf(oi[h][k].z, f, O[h].z);
                    O[h].w = fmaf(oi[h][k].w, f, O[h].w);
                }
                M[h] = Mn;
            }
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            if (!has[h]) continue;
            const float inv = L[h] > 0.0f ? 1.0f / L[h] : 0.0f;
            T *dst = out_row<T, D>(a, b, g, rr[h]) + 4 * cc[h];
            store_elem(dst + 0, O[h].x * inv);
            store_elem(dst + 1, O[h].y * inv);
            store_elem(dst + 2, O[h].z * inv);
            store_elem(dst + 3, O[h].w * inv);
        }
    }
}

// Publishes a warp's partial of a split segment (already written to `part`
// by the caller's lanes) and, if it is the last one, merges.  Whole warp
// calls.  The warp barrier orders every lane's partial stores before lane
// 0's ticket, whose release makes them visible with it (and whose acquire,
// for the last contributor, makes the others' partials visible before the
// warp barrier that precedes the merge's loads).
template <typename T, int D>
__device__ void finish_split_segment(const AttnArgs &a, int seg, int s0, int s1, int n_rows, const Part &pt,
                                     int lane) {
    __syncwarp();
    const int w_first = warp_of_tile(pt, s0);
    const int w_last = warp_of_tile(pt, s1 - 1);
    int last = 0;
    if (lane == 0) {
        int old;
        asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(old) : "l"(a.counters + seg) : "memory");
        last = old == w_last - w_first;
    }
    last = __shfl_sync(kFull, last, 0);
    if (!last) return;
    __syncwarp();
    merge_split_segment<T, D>(a, seg / a.Hkv, seg % a.Hkv, n_rows, w_first, w_last, range_start(pt, w_first) != s0,
                              lane);
    if (lane == 0) a.counters[seg] = 0;
}

// ---------------------------------------------------------------- fp32 kernel

template <int NR>
struct SimtSmem {
    static constexpr int stage_bytes = 2 * kTileBytes + NR * kRowBytes;  // K, V, query rows
    static constexpr size_t stages = 0;
    static constexpr size_t bars = stages + size_t(kWarps) * kStages * stage_bytes;
    static constexpr size_t pbuf = bars + 8 * kWarps * kStages;
    static constexpr size_t prefix = pbuf + 4 * kWarps * 16 * NR;
    static size_t total(int B) { return prefix + 4 * (2 * size_t(B) + 1 + kWarps); }
};

template <int NR>
__global__ void __launch_bounds__(kWarps * 32, NR <= 4 ? 3 : 1)
decode_attn_simt_kernel(const AttnArgs a) {
    using T = float;
    using C = Chunk<T>;
    constexpr int EPC = C::N;          // 4 fp32 per 16-byte chunk
    constexpr int D = 16 * EPC;        // 64: one 256-byte row per token
    constexpr int HALF = NR / 2;
    using S = SimtSmem<NR>;
    extern __shared__ __align__(1024) uint8_t smem[];
    int *prefix = reinterpret_cast<int *>(smem + S::prefix);
    int *ctxs = prefix + a.B + 1;
    int *scan = ctxs + a.B;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_rows = a.group * a.q_len;

    pdl_allow_dependents();
    scan_streams<T, D, kWarps>(a, prefix, ctxs, scan);
    const long long Ttot = prefix[a.B];
    const long long Wtot = active_workers(a.workers, Ttot, static_cast<long long>(a.B) * a.Hkv);
    const int wid = blockIdx.x * kWarps + warp;
    if (Ttot == 0 || wid >= Wtot) return;
    const Part pt = make_part(Ttot, Wtot);
    const int t0 = range_start(pt, wid);
    const int t1 = range_start(pt, wid + 1);
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

    int cur_id, cur_seg, cur_blk, nxt_id = -1, nxt_seg = -1, nxt_blk = 0;
    auto load_meta = [&](int k, int &id, int &seg, int &blk) {
        const int t = t0 + 32 * k + lane;
        id = -1;
        seg = -1;
        blk = 0;
        if (t < t1) tile_meta(a, prefix, t, id, seg, blk);
    };
    load_meta(0, cur_id, cur_seg, cur_blk);
    if (n > 32) load_meta(1, nxt_id, nxt_seg, nxt_blk);
    int kc = 0;

    const uint64_t policy = l2_evict_first_policy();
    const int qbytes_per_pos = a.group * kRowBytes;
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
                            ((static_cast<size_t>(b) * a.q_len + jq) * a.Hq + g * a.group) * kRowBytes;
                        bulk_load_nohint(dst + 2 * kTileBytes + jq * qbytes_per_pos, a.q + qoff,
                                         qbytes_per_pos, bar);
                    }
                }
            }
        }
    };
    pdl_wait_prerequisites();  // the pool may have been written by the kernel before
    for (int j = 0; j < min(kStages, n); ++j) issue(j);

    const int p = lane >> 4, c = lane & 15;
    const int my_tok = p + 2 * ((lane >> 1) & 7);
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
            if (lane < 16) {
#pragma unroll
                for (int r = 0; r < NR; ++r) {
                    if (r >= n_rows) break;
                    const float l = (r / HALF) == (lane & 1) ? l_tot[r % HALF] : l_oth[r % HALF];
                    const float inv = l > 0.0f ? 1.0f / l : 0.0f;
                    T *dst = out_row<T, D>(a, seg_b, seg_g, r) + c * EPC;
#pragma unroll
                    for (int e = 0; e < EPC; ++e) store_elem(dst + e, o[r][e] * inv);
                }
            }
            return;
        }
        const size_t SF = static_cast<size_t>(NR) * D + 2 * NR;
        float *part = a.part + (static_cast<size_t>(wid) * 2 + (s0 <= t0 ? 0 : 1)) * SF;
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
        finish_split_segment<T, D>(a, seg_id, s0, s1, n_rows, pt, lane);
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
            const bool ok = mbar_wait(bar0 + 8 * st, (i / kStages) & 1, a.wait_limit);
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
        const int issued = min(n, waited + kStages);
        for (int i = waited; i < issued; ++i) mbar_wait(bar0 + 8 * (i % kStages), (i / kStages) & 1, a.wait_limit);
    }
}

// ------------------------------------------------------- bf16 tensor-core kernel

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                          uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
// D[16x8] += A[16x16] . B[16x8], bf16 in, fp32 accumulate.
__device__ __forceinline__ void mma_bf16_16816(float *d, const uint32_t *a, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_f16_16816(float *d, const uint32_t *a, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int x, int y, int z,
                                            uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
        : "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Launch shapes of the tensor-core kernel.  Up to 4 query rows per KV head
// (single-token decode): 3 CTAs of 4 warps per SM, two tiles in flight per
// warp (measured best; 2 CTAs with three tiles each were 2-4 % slower at
// workloads 3 and 4).  8 rows and more (the 10 rows of a 5-token verify
// block): 2 CTAs with three tiles in flight per warp, whose larger register
// budget the wider query fragments and merges use (measured 7 % faster at
// workload 5 than 3 CTAs with two).
constexpr int kTcWarps = 4;
constexpr int kTcWideRows = 8;
__host__ __device__ constexpr int tc_ctas_per_sm(int rows) { return rows >= kTcWideRows ? 2 : 3; }
__host__ __device__ constexpr int tc_max_stages(int ctas) { return ctas == 2 ? 3 : 2; }

// One stage of a warp's ring: K and V of one (block, head) tile, each as two
// 16-row x 64-column boxes (128-byte swizzle, 2 KB each), then the query rows
// of a new segment (row-major bf16, n_rows x 256 B).
constexpr int kBoxBytes = 2048;
constexpr int kKVStageBytes = 4 * kBoxBytes;
// FP8 cache: the (block, head) record as stored (K codes: 16 rows x 128 B with
// the 16-byte chunks swizzled; V codes: 128 dimension rows x 16 B; the 16 key
// scales and 16 value scales), one bulk copy, then the query rows.
constexpr int kFp8VOff = 2048;
constexpr int kFp8ScaleOff = 4096;
constexpr int kFp8KVStageBytes = kFp8ScaleOff + 2 * 64;
// Key codes enter S = Q K^T as f16 (the hardware conversion is exact) with the
// queries in f16; value codes enter O += P V as f16 too (exact), against P
// times each token's value scale times 2^8 in f16 (11 bits, where bf16 keeps
// 8), and the softmax sum carries the same 2^8.  The factor keeps products of
// scales above about 2^-14 out of f16's subnormals; value scales must stay
// below 256 (the products below f16's largest value).
constexpr float kFp8PFix = 0x1p8f;

// Address of 16-byte chunk `ch` (0..15) of token row `t` (0..15) in a K or V
// tile stored as two swizzled boxes.
__device__ __forceinline__ uint32_t swz(uint32_t tile, int t, int ch) {
    return tile + (ch >> 3) * kBoxBytes + (t >> 3) * 1024 + (t & 7) * 128 + (((ch & 7) ^ (t & 7)) << 4);
}

struct TcSmem {
    int stage_bytes;  // K/V boxes + query rows, 1 KB multiple
    int stages;       // offset of the rings (from the 1 KB-aligned base)
    int bars;
    int prefix;       // int prefix[B + 1], ctxs[B], scan[kTcWarps]
    int total;        // bytes to request (includes 1 KB of alignment slack)
};
__host__ __device__ inline TcSmem tc_smem(int n_rows, int B, int stages, bool fp8) {
    TcSmem s;
    const int kv = fp8 ? kFp8KVStageBytes : kKVStageBytes;
    s.stage_bytes = ((kv + n_rows * kRowBytes + 1023) / 1024) * 1024;
    s.stages = 0;
    s.bars = s.stages + kTcWarps * stages * s.stage_bytes;
    s.prefix = s.bars + 8 * kTcWarps * stages;
    s.total = s.prefix + 4 * (2 * B + 1 + kTcWarps) + 1024;
    return s;
}

// Deepest ring (up to the shape's maximum) that fits the shape's CTAs per
// SM; 0 if not even one stage fits.  An FP8 tile is half a bf16 tile, so the
// 3-CTA shape keeps a third stage in flight there (measured 2 % faster at
// workload 3's context in an FP8 cache).
__host__ inline int tc_stages(int n_rows, int B, bool fp8) {
    const int ctas = tc_ctas_per_sm(n_rows);
    const int budget = 227 * 1024 / ctas - 1024;
    for (int st = fp8 && ctas == 3 ? 3 : tc_max_stages(ctas); st >= 1; --st)
        if (tc_smem(n_rows, B, st, fp8).total <= budget) return st;
    return 0;
}

// Four E4M3 codes (bytes of w, low first) as two f16 pairs (codes 0, 1 and
// 2, 3, low half first): exact.
__device__ __forceinline__ void e4m3x4_to_f16(uint32_t w, uint32_t &lo, uint32_t &hi) {
    asm("{\n\t.reg .b16 l, h;\n\t"
        "mov.b32 {l, h}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, l;\n\t"
        "cvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
}

// A bf16 pair as an f16 pair (round to nearest; bf16 values outside f16's
// range saturate to infinity, below it become f16 subnormals or zero).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(bf16_hi(w)), "f"(bf16_lo(w)));
    return r;
}

template <bool kFp8, int kRing, int kCtas>
__global__ void __launch_bounds__(kTcWarps * 32, kCtas)
decode_attn_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                      const AttnArgs a) {
    constexpr int D = 128;
    using T = __nv_bfloat16;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (base - raw);
    const int n_rows = a.group * a.q_len;  // <= 16
    constexpr int n_stages = kRing;  // ring depth (a.stages), a compile-time constant
    const TcSmem S = tc_smem(n_rows, a.B, n_stages, kFp8);
    constexpr int kQOff = kFp8 ? kFp8KVStageBytes : kKVStageBytes;  // query rows within a stage
    constexpr int kStageKV = kFp8 ? kFp8KVStageBytes : kKVStageBytes;
    int *prefix = reinterpret_cast<int *>(smem + S.prefix);
    int *ctxs = prefix + a.B + 1;
    int *scan = ctxs + a.B;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    pdl_allow_dependents();
    scan_streams<T, D, kTcWarps>(a, prefix, ctxs, scan);
    const long long Ttot = prefix[a.B];
    const long long Wtot = active_workers(a.workers, Ttot, static_cast<long long>(a.B) * a.Hkv);
    const int wid = blockIdx.x * kTcWarps + warp;
    if (Ttot == 0 || wid >= Wtot) return;
    const Part pt = make_part(Ttot, Wtot);
    const int t0 = range_start(pt, wid);
    const int t1 = range_start(pt, wid + 1);
    const int n = t1 - t0;
    if (n <= 0) return;

    const uint32_t stage0 = base + S.stages + warp * n_stages * S.stage_bytes;
    const uint32_t bar0 = base + S.bars + 8 * warp * n_stages;
    if (lane == 0) {
        for (int s = 0; s < n_stages; ++s) mbar_init(bar0 + 8 * s, 1);
        fence_mbar_init();
    }
    __syncwarp();

    int cur_id, cur_seg, cur_blk, nxt_id = -1, nxt_seg = -1, nxt_blk = 0;
    auto load_meta = [&](int k, int &id, int &seg, int &blk) {
        const int t = t0 + 32 * k + lane;
        id = -1;
        seg = -1;
        blk = 0;
        if (t < t1) tile_meta(a, prefix, t, id, seg, blk);
    };
    load_meta(0, cur_id, cur_seg, cur_blk);
    if (n > 32) load_meta(1, nxt_id, nxt_seg, nxt_blk);
    int kc = 0;

    const uint64_t policy = l2_evict_first_policy();
    const int qbytes_per_pos = a.group * kRowBytes;
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
            const int st = j % n_stages;
            const uint32_t bar = bar0 + 8 * st;
            const uint32_t dst = stage0 + st * S.stage_bytes;
            const bool need_q = j == 0 || blk == 0;
            uint32_t bytes = (id >= 0 ? kStageKV : 0) + (need_q ? a.q_len * qbytes_per_pos : 0);
            if (a.stall && j == 0) bytes += 16;  // test support: this stage never completes
            if (bytes == 0) {
                mbar_arrive(bar);
            } else {
                mbar_arrive_expect_tx(bar, bytes);
                if (id >= 0) {
                    const int tile = id * a.Hkv + seg % a.Hkv;
                    const int row = tile * TTS_BLOCK_TOKENS;
                    if constexpr (kFp8) {
                        bulk_load(dst, a.k_pool + static_cast<size_t>(tile) * kFp8KVStageBytes, kFp8KVStageBytes, bar,
                                  policy);
                    } else {
                        // one 3-D box per tensor: both 64-column halves of the 16 rows
                        tma_load_3d(dst, &kmap, 0, row, 0, bar, policy);
                        tma_load_3d(dst + 2 * kBoxBytes, &vmap, 0, row, 0, bar, policy);
                    }
                }
                if (need_q) {
                    const int b = seg / a.Hkv, g = seg % a.Hkv;
                    for (int jq = 0; jq < a.q_len; ++jq) {
                        const size_t qoff =
                            ((static_cast<size_t>(b) * a.q_len + jq) * a.Hq + g * a.group) * kRowBytes;
                        bulk_load_nohint(dst + kQOff + jq * qbytes_per_pos, a.q + qoff, qbytes_per_pos, bar);
                    }
                }
            }
        }
    };
    pdl_wait_prerequisites();  // the pool may have been written by the kernel before
    for (int j = 0; j < min(n_stages, n); ++j) issue(j);

    // Fragment coordinates: g = lane / 4 (accumulator row, and row g + 8), t = lane % 4.
    const int fg = lane >> 2, ft = lane & 3;
    // ldmatrix row-address roles: matrix mi = lane / 8, row mr = lane % 8.
    const int mi = lane >> 3, mr = lane & 7;

    int seg_id = -1, seg_b = 0, seg_g = 0, seg_L = 0, s0 = 0, s1 = 0;
    int limA = 0, limB = 0;                 // visible-token limits of rows fg and fg + 8
    uint32_t qa[8][4];                      // Q A-fragments, 8 k-steps of 16 dims
    float mA = kNegBig, mB = kNegBig, lA = 0.0f, lB = 0.0f;
    float o[16][4];                         // O accumulators, 16 n-tiles of 8 dims

    auto flush = [&]() {
        float la = lA, lb = lB;
        la += __shfl_xor_sync(kFull, la, 1);
        la += __shfl_xor_sync(kFull, la, 2);
        lb += __shfl_xor_sync(kFull, lb, 1);
        lb += __shfl_xor_sync(kFull, lb, 2);
        if constexpr (kFp8) {  // O carries P's factor 2^8 (kFp8PFix)
            la *= kFp8PFix;
            lb *= kFp8PFix;
        }
        const int rA = fg, rB = fg + 8;
        if (s0 >= t0 && s1 <= t1) {
            // whole segment in this warp: write the output rows
            const float ia = la > 0.0f ? 1.0f / la : 0.0f, ib = lb > 0.0f ? 1.0f / lb : 0.0f;
            if (rA < n_rows) {
                uint32_t *dst = reinterpret_cast<uint32_t *>(out_row<T, D>(a, seg_b, seg_g, rA));
#pragma unroll
                for (int nt = 0; nt < 16; ++nt) dst[nt * 4 + ft] = pack_bf16x2(o[nt][0] * ia, o[nt][1] * ia);
            }
            if (rB < n_rows) {
                uint32_t *dst = reinterpret_cast<uint32_t *>(out_row<T, D>(a, seg_b, seg_g, rB));
#pragma unroll
                for (int nt = 0; nt < 16; ++nt) dst[nt * 4 + ft] = pack_bf16x2(o[nt][2] * ib, o[nt][3] * ib);
            }
            return;
        }
        const int NRS = a.nr_slot;
        const size_t SF = static_cast<size_t>(NRS) * D + 2 * NRS;
        float *part = a.part + (static_cast<size_t>(wid) * 2 + (s0 <= t0 ? 0 : 1)) * SF;
        if (rA < n_rows) {
#pragma unroll
            for (int nt = 0; nt < 16; ++nt)
                *reinterpret_cast<float2 *>(part + rA * D + nt * 8 + 2 * ft) = make_float2(o[nt][0], o[nt][1]);
            if (ft == 0) { part[NRS * D + rA] = mA; part[NRS * D + NRS + rA] = la; }
        }
        if (rB < n_rows) {
#pragma unroll
            for (int nt = 0; nt < 16; ++nt)
                *reinterpret_cast<float2 *>(part + rB * D + nt * 8 + 2 * ft) = make_float2(o[nt][2], o[nt][3]);
            if (ft == 0) { part[NRS * D + rB] = mB; part[NRS * D + NRS + rB] = lb; }
        }
        finish_split_segment<T, D>(a, seg_id, s0, s1, n_rows, pt, lane);
    };

    bool timed_out = false;
    int waited = 0;
    for (int i = 0; i < n; ++i) {
        if ((i & 31) == 0 && i > 0) {
            kc = i >> 5;
            cur_id = nxt_id; cur_seg = nxt_seg; cur_blk = nxt_blk;
            if (n > 32 * (kc + 1)) load_meta(kc + 1, nxt_id, nxt_seg, nxt_blk);
        }
        const int st = i % n_stages;
        if (!timed_out) {
            const bool ok = mbar_wait(bar0 + 8 * st, (i / n_stages) & 1, a.wait_limit);
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
        const uint32_t kt = stage0 + st * S.stage_bytes;                  // K boxes / codes
        const uint32_t vt = kt + (kFp8 ? kFp8VOff : 2 * kBoxBytes);        // V boxes / codes
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
            const int rA = fg, rB = fg + 8;
            limA = rA < n_rows ? (a.causal ? seg_L - a.q_len + rA / a.group + 1 : seg_L) : 0;
            limB = rB < n_rows ? (a.causal ? seg_L - a.q_len + rB / a.group + 1 : seg_L) : 0;
            mA = mB = kNegBig;
            lA = lB = 0.0f;
            const uint32_t qs = kt + kQOff;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                // bf16: dims (2t, 2t+1) and (2t+8, 2t+9) of the k-step; FP8: the
                // k-step's dims permuted to (4t, 4t+1) and (4t+2, 4t+3), the
                // order in which a 16-bit ldmatrix row read hands out the codes
                const int c0 = kFp8 ? (16 * ks + 4 * ft) * 2 : (16 * ks + 2 * ft) * 2;
                const int c1 = kFp8 ? c0 + 4 : c0 + 16;
                const uint8_t *qrA = smem + (qs - base) + rA * kRowBytes;
                const uint8_t *qrB = smem + (qs - base) + rB * kRowBytes;
                qa[ks][0] = (rA < n_rows && !timed_out) ? *reinterpret_cast<const uint32_t *>(qrA + c0) : 0u;
                qa[ks][1] = (rB < n_rows && !timed_out) ? *reinterpret_cast<const uint32_t *>(qrB + c0) : 0u;
                qa[ks][2] = (rA < n_rows && !timed_out) ? *reinterpret_cast<const uint32_t *>(qrA + c1) : 0u;
                qa[ks][3] = (rB < n_rows && !timed_out) ? *reinterpret_cast<const uint32_t *>(qrB + c1) : 0u;
                if constexpr (kFp8) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) qa[ks][e] = bf16x2_to_f16x2(qa[ks][e]);
                }
            }
#pragma unroll
            for (int nt = 0; nt < 16; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) o[nt][e] = 0.0f;
        }
        if (!timed_out && t_id >= 0 && t_id < a.num_blocks) {
            const int base_tok = t_blk * TTS_BLOCK_TOKENS;
            // ---- S = Q K^T: 2 n-tiles of 8 tokens x 8 k-steps of 16 dims
            float s[2][4];
            // FP8: this lane's key and value scales (tokens 2t, 2t+1 | 2t+8, 2t+9)
            float2 ksc[2], vsc[2];
            if constexpr (kFp8) {
                const float *sc = reinterpret_cast<const float *>(smem + (kt - base) + kFp8ScaleOff);
                ksc[0] = *reinterpret_cast<const float2 *>(sc + 2 * ft);
                ksc[1] = *reinterpret_cast<const float2 *>(sc + 8 + 2 * ft);
                vsc[0] = *reinterpret_cast<const float2 *>(sc + 16 + 2 * ft);
                vsc[1] = *reinterpret_cast<const float2 *>(sc + 24 + 2 * ft);
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) s[nt][e] = 0.0f;
#pragma unroll
                    for (int kq = 0; kq < 2; ++kq) {
                        // matrix i = k-step 4 kq + i (16 dims) of tokens 8 nt .. 8 nt + 7
                        const int tok = 8 * nt + (lane & 7);
                        const int ch = 4 * kq + (lane >> 3);
                        uint32_t w[4];
                        ldsm_x4(kt + tok * 128 + ((ch ^ (tok & 7)) << 4), w[0], w[1], w[2], w[3]);
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            uint32_t b0, b1;
                            e4m3x4_to_f16(w[i], b0, b1);
                            mma_f16_16816(s[nt], qa[4 * kq + i], b0, b1);
                        }
                    }
                }
            } else {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
                for (int e = 0; e < 4; ++e) s[nt][e] = 0.0f;
#pragma unroll
                for (int kp = 0; kp < 4; ++kp) {
                    // matrices: (k-step 2kp, low/high 8 dims), (k-step 2kp+1, low/high)
                    const int ch = 2 * (2 * kp + (mi >> 1)) + (mi & 1);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(swz(kt, 8 * nt + mr, ch), b0, b1, b2, b3);
                    mma_bf16_16816(s[nt], qa[2 * kp], b0, b1);
                    mma_bf16_16816(s[nt], qa[2 * kp + 1], b2, b3);
                }
            }
            }
            // ---- online softmax in the log2 domain; rows fg (A) and fg + 8 (B)
            float xa[4], xb[4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int tok = base_tok + 8 * nt + 2 * ft + e;
                    float f = a.qscale;
                    if constexpr (kFp8) f *= (e == 0 ? ksc[nt].x : ksc[nt].y);
                    xa[2 * nt + e] = tok < limA ? s[nt][e] * f : -INFINITY;
                    xb[2 * nt + e] = tok < limB ? s[nt][2 + e] * f : -INFINITY;
                }
            }
            float ma = fmaxf(fmaxf(xa[0], xa[1]), fmaxf(xa[2], xa[3]));
            float mb = fmaxf(fmaxf(xb[0], xb[1]), fmaxf(xb[2], xb[3]));
            ma = fmaxf(ma, __shfl_xor_sync(kFull, ma, 1));
            ma = fmaxf(ma, __shfl_xor_sync(kFull, ma, 2));
            mb = fmaxf(mb, __shfl_xor_sync(kFull, mb, 1));
            mb = fmaxf(mb, __shfl_xor_sync(kFull, mb, 2));
            const float na = fmaxf(mA, ma), nb2 = fmaxf(mB, mb);
            const float aa = exp2f(mA - na), ab = exp2f(mB - nb2);
            mA = na;
            mB = nb2;
            float pa[4], pb[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                pa[e] = exp2f(xa[e] - na);
                pb[e] = exp2f(xb[e] - nb2);
            }
            lA = lA * aa + (pa[0] + pa[1]) + (pa[2] + pa[3]);
            lB = lB * ab + (pb[0] + pb[1]) + (pb[2] + pb[3]);
            if (__any_sync(kFull, aa != 1.0f || ab != 1.0f)) {
#pragma unroll
                for (int nt = 0; nt < 16; ++nt) {
                    o[nt][0] *= aa; o[nt][1] *= aa;
                    o[nt][2] *= ab; o[nt][3] *= ab;
                }
            }
            // P as the A operand (rows fg / fg + 8, tokens 2t, 2t+1, 2t+8, 2t+9)
            uint32_t pf[4];
            if constexpr (kFp8) {
                // times each token's value scale and 2^8, in f16; slots past
                // the context may hold any scale (even NaN), so they give 0
                float qa_[4], qb_[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int tok = base_tok + 8 * (e >> 1) + 2 * ft + (e & 1);
                    const float vs = ((e & 1) ? vsc[e >> 1].y : vsc[e >> 1].x) * kFp8PFix;
                    qa_[e] = tok < limA ? pa[e] * vs : 0.0f;
                    qb_[e] = tok < limB ? pb[e] * vs : 0.0f;
                }
                pf[0] = pack_f16x2(qa_[0], qa_[1]);
                pf[1] = pack_f16x2(qb_[0], qb_[1]);
                pf[2] = pack_f16x2(qa_[2], qa_[3]);
                pf[3] = pack_f16x2(qb_[2], qb_[3]);
            } else {
                pf[0] = pack_bf16x2(pa[0], pa[1]);
                pf[1] = pack_bf16x2(pb[0], pb[1]);
                pf[2] = pack_bf16x2(pa[2], pa[3]);
                pf[3] = pack_bf16x2(pb[2], pb[3]);
            }
            // Tokens past the context may hold anything (even NaN, which the
            // MMA would spread as 0 * NaN): zero their values in the tile.
            if (base_tok + TTS_BLOCK_TOKENS > seg_L) {
                const int first_bad = max(seg_L - base_tok, 0);
                if constexpr (kFp8) {
                    // each dimension's 16 codes: byte 4j + k holds slot 2j + (k & 1) + 8 (k >> 1)
                    uint32_t keep[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        keep[j] = 0u;
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            if (2 * j + (k & 1) + 8 * (k >> 1) < first_bad) keep[j] |= 0xFFu << (8 * k);
                    }
                    uint4 *rows = reinterpret_cast<uint4 *>(smem + (vt - base));
#pragma unroll
                    for (int d = lane; d < D; d += 32) {
                        uint4 v = rows[d];
                        v.x &= keep[0]; v.y &= keep[1]; v.z &= keep[2]; v.w &= keep[3];
                        rows[d] = v;
                    }
                } else {
                    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
                    for (int idx = lane; idx < (TTS_BLOCK_TOKENS - first_bad) * 16; idx += 32) {
                        const int row = first_bad + idx / 16, ch = idx % 16;
                        *reinterpret_cast<uint4 *>(smem + (swz(vt, row, ch) - base)) = z;
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
            }
            // ---- O += P V: 8 pairs of n-tiles (16 dims each), k = 16 tokens
            if constexpr (kFp8) {
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    // matrix i = dims 8 (4 q4 + i) .. + 7, each row the 16 codes of one
                    // dimension in the slot order that gives lane t slots 2t, 2t+1, 2t+8, 2t+9
                    uint32_t w[4];
                    ldsm_x4(vt + (8 * (4 * q4 + (lane >> 3)) + (lane & 7)) * 16, w[0], w[1], w[2], w[3]);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        uint32_t b0, b1;
                        e4m3x4_to_f16(w[i], b0, b1);
                        mma_f16_16816(o[4 * q4 + i], pf, b0, b1);
                    }
                }
            } else {
#pragma unroll
                for (int np = 0; np < 8; ++np) {
                    const int tok = mr + 8 * (mi & 1);
                    const int ch = 2 * np + (mi >> 1);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_t(swz(vt, tok, ch), b0, b1, b2, b3);
                    mma_bf16_16816(o[2 * np], pf, b0, b1);
                    mma_bf16_16816(o[2 * np + 1], pf, b2, b3);
                }
            }
        }
        __syncwarp();
        if (!timed_out && i + n_stages < n) issue(i + n_stages);
    }
    flush();
    if (timed_out) {
        const int issued = min(n, waited + n_stages);
        for (int i = waited; i < issued; ++i) mbar_wait(bar0 + 8 * (i % n_stages), (i / n_stages) & 1, a.wait_limit);
    }
}

// ------------------------------------------------------------------- launch

// Query-row counts per (stream, KV head) are padded up to one of these.
constexpr int kRowTemplates[] = {2, 4, 8, 10, 16};

int padded_rows(int rows) {
    for (int r : kRowTemplates)
        if (rows <= r) return r;
    return 0;
}

int ctas_per_sm(int dtype, int nr) {
    if (dtype == TTS_BF16 || dtype == TTS_FP8_E4M3) return tc_ctas_per_sm(nr);
    return nr <= 4 ? 3 : 1;
}

int device_sms() {
    const int n = sm_count();
    return n > 0 ? n : 160;  // no device visible (size queries on a build host)
}

cudaLaunchAttribute pdl_attr() {
    cudaLaunchAttribute at;
    at.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at.val.programmaticStreamSerializationAllowed = 1;
    return at;
}

template <int NR>
int launch_simt_nr(const AttnArgs &a, int ctas, LaunchOpts o) {
    const size_t smem = SimtSmem<NR>::total(a.B);
    auto kern = decode_attn_simt_kernel<NR>;
    if (!ensure_dynamic_smem(reinterpret_cast<const void *>(kern), static_cast<int>(smem))) return TTS_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ctas, 1, 1);
    cfg.blockDim = dim3(kWarps * 32, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = o.stream;
    cudaLaunchAttribute attr[1] = {pdl_attr()};
    cfg.attrs = attr;
    cfg.numAttrs = o.pdl ? 1 : 0;
    if (cudaLaunchKernelEx(&cfg, kern, a) != cudaSuccess) {
        cudaGetLastError();
        return TTS_ERR_CUDA;
    }
    return TTS_OK;
}

int launch_simt(const AttnArgs &a, int nr, int ctas, LaunchOpts o) {
    switch (nr) {
        case 2: return launch_simt_nr<2>(a, ctas, o);
        case 4: return launch_simt_nr<4>(a, ctas, o);
        case 8: return launch_simt_nr<8>(a, ctas, o);
        case 10: return launch_simt_nr<10>(a, ctas, o);
        case 16: return launch_simt_nr<16>(a, ctas, o);
        default: return TTS_ERR_UNSUPPORTED;
    }
}

template <bool kFp8>
int launch_tc(const AttnArgs &a, const CUtensorMap &kmap, const CUtensorMap &vmap, int ctas, LaunchOpts o) {
    static_assert(tc_max_stages(3) == 2 && tc_max_stages(2) == 3,
                  "instantiated: 3 CTAs x 1-2 stages (1-3 with FP8), 2 x 1-3");
    const int rows = a.group * a.q_len;
    const size_t smem = tc_smem(rows, a.B, a.stages, kFp8).total;
    const auto kern = tc_ctas_per_sm(rows) == 2
                          ? (a.stages == 3   ? decode_attn_tc_kernel<kFp8, 3, 2>
                             : a.stages == 2 ? decode_attn_tc_kernel<kFp8, 2, 2>
                                             : decode_attn_tc_kernel<kFp8, 1, 2>)
                          : (kFp8 && a.stages == 3 ? decode_attn_tc_kernel<kFp8, 3, 3>
                             : a.stages == 2       ? decode_attn_tc_kernel<kFp8, 2, 3>
                                                   : decode_attn_tc_kernel<kFp8, 1, 3>);
    if (!ensure_dynamic_smem(reinterpret_cast<const void *>(kern), static_cast<int>(smem)))
        return TTS_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ctas, 1, 1);
    cfg.blockDim = dim3(kTcWarps * 32, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = o.stream;
    cudaLaunchAttribute attr[1] = {pdl_attr()};
    cfg.attrs = attr;
    cfg.numAttrs = o.pdl ? 1 : 0;
    if (cudaLaunchKernelEx(&cfg, kern, kmap, vmap, a) != cudaSuccess) {
        cudaGetLastError();
        return TTS_ERR_CUDA;
    }
    return TTS_OK;
}

bool supported_head(int dtype, int head_dim) {
    return ((dtype == TTS_BF16 || dtype == TTS_FP8_E4M3) && head_dim == 128) || (dtype == TTS_F32 && head_dim == 64);
}

}  // namespace

bool attn_plan(int dtype, int B, int q_len, int num_q_heads, int num_kv_heads, int head_dim,
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
    out->ctas = device_sms() * ctas_per_sm(dtype, rows);
    out->workers = out->ctas * (dtype == TTS_F32 ? kWarps : kTcWarps);
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
    const int dtype = head_dim == 64 ? TTS_F32 : TTS_BF16;
    if (!tts::attn_plan(dtype, B, q_len, num_q_heads, num_kv_heads, head_dim, max_ctx_len, &pl))
        return 0;
    return tts::attn_workspace_bytes(B, num_kv_heads, head_dim, pl);
}

namespace tts {

struct AttnLaunchState {
    AttnArgs a;
    CUtensorMap kmap, vmap;
    int dtype, rows, ctas;
};
static_assert(sizeof(AttnLaunchState) <= sizeof(AttnLaunch::storage), "AttnLaunch storage too small");

int prepare_attn(const tts_kv_cache *cache, const int32_t *d_block_table, int32_t max_blocks_per_seq,
                 const int32_t *d_ctx_lens, int32_t max_ctx_len, int32_t B, int32_t q_len,
                 int32_t num_q_heads, float scale, int32_t causal, const void *d_q, void *d_out,
                 void *d_ws, size_t ws_bytes, int32_t *d_err, AttnLaunch *out) {
    if (!cache || !d_block_table || !d_ctx_lens || !d_q || !d_out) return TTS_ERR_INVALID;
    if (!cache->k_pool || (!cache->v_pool && cache->dtype != TTS_FP8_E4M3) || cache->num_blocks < 1)
        return TTS_ERR_INVALID;
    if (B < 0 || q_len < 1 || max_blocks_per_seq < 1 || max_blocks_per_seq > (1 << 20) ||
        !(scale > 0.0f) || scale != scale)
        return TTS_ERR_INVALID;
    if (cache->block_size != TTS_BLOCK_TOKENS) return TTS_ERR_UNSUPPORTED;
    if (!supported_head(cache->dtype, cache->head_dim)) return TTS_ERR_UNSUPPORTED;
    if (cache->num_kv_heads < 1) return TTS_ERR_INVALID;
    if (static_cast<long long>(cache->num_blocks) * cache->num_kv_heads * TTS_BLOCK_TOKENS >= (1LL << 31))
        return TTS_ERR_UNSUPPORTED;
    AttnLaunchState *st = new (out->storage) AttnLaunchState();
    st->ctas = 0;
    if (B == 0) return TTS_OK;
    AttnPlan pl;
    if (!attn_plan(cache->dtype, B, q_len, num_q_heads, cache->num_kv_heads, cache->head_dim,
                   max_ctx_len, &pl)) {
        const int nh = cache->num_kv_heads;
        const bool shape_ok = num_q_heads >= nh && num_q_heads % nh == 0 && max_ctx_len >= q_len &&
                              max_ctx_len <= (1 << 24);
        return shape_ok ? TTS_ERR_UNSUPPORTED : TTS_ERR_INVALID;
    }
    const bool fp8 = cache->dtype == TTS_FP8_E4M3;
    if (!aligned16(cache->k_pool) || (!fp8 && !aligned16(cache->v_pool)) || !aligned16(d_q))
        return TTS_ERR_INVALID;
    const size_t need = attn_workspace_bytes(B, cache->num_kv_heads, cache->head_dim, pl);
    if (!d_ws || ws_bytes < need || (reinterpret_cast<uintptr_t>(d_ws) & 255u) != 0)
        return TTS_ERR_WORKSPACE;

    uint8_t *ws = static_cast<uint8_t *>(d_ws);
    AttnArgs &a = st->a;
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
    a.nr_slot = pl.rows;
    a.stages = cache->dtype == TTS_F32 ? kStages : tc_stages(a.group * q_len, B, fp8);

    if (a.stages < 1) return TTS_ERR_UNSUPPORTED;
    a.err = d_err;
    a.wait_limit = thread_opts().wait_limit;
    a.stall = thread_opts().stall == TTS_TEST_STALL_ATTN_RING && cache->dtype != TTS_F32;
    st->dtype = cache->dtype;
    st->rows = pl.rows;
    st->ctas = pl.ctas;
    if (cache->dtype == TTS_BF16) {
        const uint64_t rows = static_cast<uint64_t>(a.num_blocks) * a.Hkv * TTS_BLOCK_TOKENS;
        if (!make_tma_rows_in_halves_bf16(&st->kmap, cache->k_pool, rows, TTS_BLOCK_TOKENS) ||
            !make_tma_rows_in_halves_bf16(&st->vmap, cache->v_pool, rows, TTS_BLOCK_TOKENS))
            return TTS_ERR_CUDA;
    }
    return TTS_OK;
}

int launch_attn(const AttnLaunch &L, LaunchOpts o) {
    const AttnLaunchState *st = reinterpret_cast<const AttnLaunchState *>(L.storage);
    if (st->ctas == 0) return TTS_OK;  // empty batch
    if (st->dtype == TTS_BF16) return launch_tc<false>(st->a, st->kmap, st->vmap, st->ctas, o);
    if (st->dtype == TTS_FP8_E4M3) return launch_tc<true>(st->a, st->kmap, st->vmap, st->ctas, o);
    return launch_simt(st->a, st->rows, st->ctas, o);
}

}  // namespace tts

extern "C" int tts_decode_attn(const tts_kv_cache *cache, const int32_t *d_block_table,
                               int32_t max_blocks_per_seq, const int32_t *d_ctx_lens,
                               int32_t max_ctx_len, int32_t B, int32_t q_len, int32_t num_q_heads,
                               float scale, int32_t causal, const void *d_q, void *d_out,
                               void *d_ws, size_t ws_bytes, int32_t *d_err, void *stream) {
    tts::AttnLaunch L;
    const int st = tts::prepare_attn(cache, d_block_table, max_blocks_per_seq, d_ctx_lens, max_ctx_len, B,
                                     q_len, num_q_heads, scale, causal, d_q, d_out, d_ws, ws_bytes, d_err, &L);
    if (st != TTS_OK) return st;
    return tts::launch_attn(L, {static_cast<cudaStream_t>(stream), tts::thread_pdl()});
}

// ---------------------------------------------------------------------------
// Decode attention without a caller workspace.
//
// Some callers cannot allocate device memory where they run a decode step:
// engines that hand all free device memory to the KV pool at start-up and so
// leave nothing for cudaMalloc, plugin hosts that give a library no
// allocator, and real-time loops that cannot absorb the implicit
// synchronisation and unbounded latency of cudaMalloc / cudaFree inside a
// frame deadline.  For them the split-KV partials live in one file-scope
// device array of fixed size instead of a caller workspace.  Every GPU that
// loads this library holds the array until the process exits.

namespace tts {
namespace {

constexpr size_t kStaticScratchBytes = size_t(16) << 20;  // 16 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_attn_scratch[kStaticScratchBytes];

// The array's device address, cached per device together with the id of the
// CUDA context it was looked up in.  Context ids are never reused within a
// process, so a context replaced after cudaDeviceReset (or a context made
// current through the driver API) triggers a fresh lookup instead of reusing
// an address of a module that is gone.
struct ScratchAddr {
    unsigned long long ctx_id;
    void *addr;
};
std::mutex g_scratch_mu;
ScratchAddr g_scratch_addr[kMaxDevices] = {};

PFN_cuCtxGetCurrent_v4000 g_ctx_get_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_get_id = nullptr;

// Id of the current CUDA context, or 0 if none is current or the driver
// calls are unavailable.
unsigned long long current_context_id() {
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    });
    if (!g_ctx_get_current || !g_ctx_get_id) return 0;
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (g_ctx_get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
    if (g_ctx_get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

// Device address of g_attn_scratch in the current context.  The symbol's
// name in host code is only a host-side handle, so the address is looked up
// with cudaGetSymbolAddress (with the device current) the first time a
// context uses it, and cached for that context.
int static_scratch_address(void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return TTS_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return TTS_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    ScratchAddr &e = g_scratch_addr[dev];
    const unsigned long long id = current_context_id();
    if (!e.addr || id == 0 || id != e.ctx_id) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_attn_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            e.addr = nullptr;
            return TTS_ERR_CUDA;
        }
        e.addr = p;
        // the lookup made the device's primary context current if none was
        e.ctx_id = id != 0 ? id : current_context_id();
    }
    *out = e.addr;
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
    int st = static_scratch_address(&scratch);
    if (st != TTS_OK) return st;
    // Every argument is checked before anything is queued, so a rejected call
    // leaves the shared array untouched.
    AttnLaunch L;
    st = prepare_attn(cache, d_block_table, max_blocks_per_seq, d_ctx_lens, max_ctx_len, B, q_len, num_q_heads,
                      scale, causal, d_q, d_out, scratch, need, d_err, &L);
    if (st != TTS_OK) return st;
    // The split tickets must start at zero; they sit at the end of the
    // workspace layout.  The array keeps whatever the previous call left.
    const size_t tickets = align_up(static_cast<size_t>(B) * cache->num_kv_heads * sizeof(int32_t), 256);
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(static_cast<uint8_t *>(scratch) + need - tickets, 0, tickets, s) != cudaSuccess) {
        cudaGetLastError();
        return TTS_ERR_CUDA;
    }
    return launch_attn(L, {s, false});
}
