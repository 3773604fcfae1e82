// Speculative verification of K draft tokens per stream ("Optimizing
// Streaming Text-to-Speech Models for Sub-50 Millisecond Latency", section
// "Speculative Decoding for Acoustic Tokens"), generalised from the page's
// batch row 0 to every stream, with seeded Philox uniforms in place of an
// unseeded generator and the rejection draw done by Gumbel-max over the log of
// the clamped residual (the same distribution as normalising and sampling it).
//
// One CTA per stream.  Staged kernel (the stream's rows fit in shared
// memory): bulk copies bring the K target rows (K + 1 with the bonus draw)
// and the K draft rows into shared memory while the threads generate the
// draw's Gumbel noise (one Philox block per 8 consecutive vocabulary entries)
// and the accept uniforms; warp groups reduce each target row to its max and
// sum of exp((x - max) / T); lane i of one warp tests draft i and a ballot
// finds the first rejection; the CTA draws the replacement (or bonus) token
// with a block-wide argmax over packed (key, index) pairs.  Streaming kernel
// (rows too large for shared memory): the same steps reading global memory.
#include "tts_common.cuh"
#include "tts_internal.h"

namespace tts {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxK = 16;
constexpr unsigned kFull = 0xFFFFFFFFu;

__device__ __forceinline__ void merge_max_sum(float &m, float &s, float m2, float s2, float T) {
    const float M = fmaxf(m, m2);
    // Terms with a -inf max hold nothing (s == 0).
    const float a = (m == -INFINITY) ? 0.0f : s * expf((m - M) / T);
    const float b = (m2 == -INFINITY) ? 0.0f : s2 * expf((m2 - M) / T);
    m = M;
    s = a + b;
}

__global__ void __launch_bounds__(kThreads)
spec_verify_kernel(const float *__restrict__ tl, const float *__restrict__ dp,
                   const int32_t *__restrict__ dt, int K, int V, float T,
                   const uint64_t *__restrict__ seed, const uint64_t *__restrict__ step, int flags,
                   int32_t *__restrict__ n_accepted, int32_t *__restrict__ next_token,
                   int32_t *err) {
    __shared__ float row_max[kMaxK], row_sum[kMaxK];
    __shared__ int s_reject, s_accepted, s_draw;
    __shared__ unsigned long long s_best;
    pdl_wait_prerequisites();
    pdl_allow_dependents();
    const int b = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float *tl_b = tl + static_cast<size_t>(b) * (K + 1) * V;
    const float *dp_b = dp + static_cast<size_t>(b) * K * V;
    const uint64_t key0 = seed[b], key1 = step[b];

    // Phase 1: softmax statistics of the K target rows, one warp per row.
    for (int i = warp; i < K; i += kThreads / 32) {
        const float *x = tl_b + static_cast<size_t>(i) * V;
        float m = -INFINITY, s = 0.0f;
        for (int v = lane; v < V; v += 32) {
            const float xv = __ldg(x + v);
            if (xv > m) {
                s = (m == -INFINITY ? 0.0f : s * expf((m - xv) / T)) + 1.0f;
                m = xv;
            } else {
                s += expf((xv - m) / T);
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float m2 = __shfl_xor_sync(kFull, m, o);
            const float s2 = __shfl_xor_sync(kFull, s, o);
            merge_max_sum(m, s, m2, s2, T);
        }
        if (lane == 0) { row_max[i] = m; row_sum[i] = s; }
    }
    if (threadIdx.x == 0) s_best = 0ull;
    __syncthreads();

    // Phase 2: accept / reject in order.
    if (threadIdx.x == 0) {
        int accepted = 0, reject = -1, draw = 1;
        for (int i = 0; i < K; ++i) {
            const int d = dt[static_cast<size_t>(b) * K + i];
            if (d < 0 || d >= V) {
                flag_error(err, TTS_ERRBIT_TOKEN);
                reject = i;
                draw = 0;
                break;
            }
            const float pt = expf((tl_b[static_cast<size_t>(i) * V + d] - row_max[i]) / T) / row_sum[i];
            const float pd = dp_b[static_cast<size_t>(i) * V + d];
            bool ok = false;
            if (pd > 0.0f) ok = philox_uniform(key0, key1, 1u, 0u, static_cast<uint32_t>(i)) < pt / pd;
            if (!ok) { reject = i; break; }
            ++accepted;
        }
        if (reject < 0 && !(flags & TTS_VERIFY_BONUS)) draw = 0;
        s_reject = reject;
        s_accepted = accepted;
        s_draw = draw;
    }
    __syncthreads();
    const int reject = s_reject;
    if (!s_draw) {
        if (threadIdx.x == 0) {
            n_accepted[b] = s_accepted;
            next_token[b] = -1;
        }
        return;
    }

    // Phase 3: the replacement draw (rejection at row `reject`) or the bonus
    // draw (row K).  Keys: log(residual) + G, or target / T + G.
    const int row = reject >= 0 ? reject : K;
    const float *x = tl_b + static_cast<size_t>(row) * V;
    const float *pdr = reject >= 0 ? dp_b + static_cast<size_t>(row) * V : nullptr;
    const float m = reject >= 0 ? row_max[row] : 0.0f;
    const float z = reject >= 0 ? row_sum[row] : 1.0f;
    const int groups = (V + 7) / 8;
    // A residual that is zero everywhere falls back to p_t itself.
    bool use_pt = false;
    if (reject >= 0) {
        int any = 0;
        for (int v = threadIdx.x; v < V && !any; v += kThreads)
            any = (expf((__ldg(x + v) - m) / T) / z - __ldg(pdr + v)) > 0.0f;
        use_pt = !__syncthreads_or(any);
    }
    unsigned long long best = 0ull;
    for (int gi = threadIdx.x; gi < groups; gi += kThreads) {
        const Philox4x64 ph(static_cast<uint64_t>(gi), 2u, 0u, 0u, key0, key1);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int v = gi * 8 + e;
            if (v >= V) break;
            const float g = gumbel_from_uniform(bits_to_uniform(ph.half(e)));
            float key;
            if (reject >= 0) {
                const float pt = expf((__ldg(x + v) - m) / T) / z;
                const float r = use_pt ? pt : fmaxf(pt - __ldg(pdr + v), 0.0f);
                if (!(r > 0.0f)) continue;
                key = logf(r) + g;
            } else {
                key = __ldg(x + v) / T + g;
            }
            const unsigned long long pk = pack_argmax(key, v);
            best = pk > best ? pk : best;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long other = __shfl_xor_sync(kFull, best, o);
        best = other > best ? other : best;
    }
    if (lane == 0) atomicMax(&s_best, best);
    __syncthreads();
    if (threadIdx.x == 0) {
        n_accepted[b] = s_accepted;
        next_token[b] = s_best ? unpack_index(s_best) : -1;
    }
}

// ------------------------------------------------------------ staged kernel

constexpr int kStagedThreads = 1024;
constexpr int kStagedWarps = kStagedThreads / 32;
constexpr uint32_t kBulkChunk = 65536;  // bytes per bulk copy

// Bytes of the 16-byte-aligned interior of the `n` floats at `g`.
__device__ __forceinline__ uint32_t interior_bytes(const float *g, size_t n) {
    const uintptr_t s0 = reinterpret_cast<uintptr_t>(g), s1 = s0 + n * 4;
    const uintptr_t a0 = (s0 + 15) & ~uintptr_t(15), a1 = s1 & ~uintptr_t(15);
    return a1 > a0 ? static_cast<uint32_t>(a1 - a0) : 0u;
}

// The 16-byte-aligned interior of the shared-memory image of `n` floats at
// `g` by bulk copies (one thread, completing on `bar`, whose expected bytes
// the caller sets); `dst` is congruent to `g` modulo 16.  The ragged ends
// are the caller's, by plain loads.
__device__ void stage_bulk(float *dst, const float *g, size_t n, uint32_t bar) {
    const uintptr_t s0 = reinterpret_cast<uintptr_t>(g), s1 = s0 + n * 4;
    const uintptr_t a0 = (s0 + 15) & ~uintptr_t(15), a1 = s1 & ~uintptr_t(15);
    if (a1 <= a0) return;
    const size_t head = (a0 - s0) / 4;
    const uint32_t bytes = static_cast<uint32_t>(a1 - a0);
    const uint32_t d = smem_addr(dst + head);
    const uint8_t *src = reinterpret_cast<const uint8_t *>(a0);
    for (uint32_t off = 0; off < bytes; off += kBulkChunk) {
        const uint32_t len = bytes - off < kBulkChunk ? bytes - off : kBulkChunk;
        bulk_load_nohint(d + off, src + off, len, bar);
    }
}
__host__ __device__ inline uint32_t staged_target_rows(int K, int flags) {
    return static_cast<uint32_t>(K) + ((flags & TTS_VERIFY_BONUS) ? 1u : 0u);
}
// Float offsets of the staged kernel's shared-memory areas: the target rows'
// image and the draft rows' image (each placed at the float offset that makes
// it congruent to its global rows modulo 16 bytes, within 4 floats of slack),
// then the draw's Gumbel noise, one float per vocabulary entry.
struct StagedLayout {
    uint32_t draft, noise, bytes;
};
__host__ __device__ inline StagedLayout staged_layout(int K, int V, int flags) {
    const uint32_t nt = staged_target_rows(K, flags) * static_cast<uint32_t>(V);
    const uint32_t nd = static_cast<uint32_t>(K) * static_cast<uint32_t>(V);
    StagedLayout L;
    L.draft = (nt + 4 + 3) & ~3u;
    L.noise = L.draft + ((nd + 4 + 3) & ~3u);
    L.bytes = (L.noise + ((static_cast<uint32_t>(V) + 3) & ~3u)) * 4u;
    return L;
}

// Warp roles of the staged kernel while the rows land.
constexpr int kRaggedWarp = kStagedWarps - 1;    // the rows' unaligned ends by plain loads
constexpr int kAcceptWarp = kStagedWarps - 2;    // the accept test's inputs
constexpr int kDrawWarmWarp = kStagedWarps - 3;  // the draw's warm-up
constexpr int kNoiseThreads = 32 * (kStagedWarps - 3);

// The staged kernel's per-stream scalars in shared memory.
struct VerifyScalars {
    float red_m[kStagedWarps], red_s[kStagedWarps];  // per-warp parts of the row statistics
    float row_max[kMaxK], row_sum[kMaxK];
    float acc_u[kMaxK], acc_pd[kMaxK];  // accept test: uniform, draft probability of the token
    int acc_d[kMaxK];                   // accept test: draft token
    int reject, accepted, draw, ok;
    unsigned long long best, best_p;
    float warm_m, warm_s;  // the warm-up runs' outputs (scratch copy only)
};

// The three phases after the rows land are out-of-line functions: while the
// rows are in flight, three warps each run one of them once on scratch data,
// first thing, so that their instructions are already on the SM when the CTA
// needs them (each runs once per CTA, so every instruction would otherwise be
// fetched cold).

// Elements a thread loads before it uses the first of them in the row
// statistics and the draw: independent shared-memory loads and exponentials
// in flight instead of one load's latency per element.
constexpr int kRowUnroll = 8;
constexpr int kDrawUnroll = 4;

// One warp's part of a row's statistics: the max m of x[v] over
// v = v0 + lane, v0 + lane + stride, ... and the sum of 2^((x[v] - m) k2)
// against it (exp((x - m) / T) with k2 = log2(e) / T); lane 0 stores them.
__device__ __noinline__ void warp_row_part(const float *x, int V, int v0, int stride, float k2, float *m_out,
                                           float *s_out) {
    const int lane = threadIdx.x & 31;
    const int first = v0 + lane, span = kRowUnroll * stride;
    float m = -INFINITY, s = 0.0f;
    int v = first;
    for (; v + (kRowUnroll - 1) * stride < V; v += span) {
        float xv[kRowUnroll];
#pragma unroll
        for (int j = 0; j < kRowUnroll; ++j) xv[j] = x[v + j * stride];
#pragma unroll
        for (int j = 0; j < kRowUnroll; ++j) m = fmaxf(m, xv[j]);
    }
    for (; v < V; v += stride) m = fmaxf(m, x[v]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
    if (m != -INFINITY) {
        v = first;
        for (; v + (kRowUnroll - 1) * stride < V; v += span) {
            float e[kRowUnroll];
#pragma unroll
            for (int j = 0; j < kRowUnroll; ++j) e[j] = hw_ex2((x[v + j * stride] - m) * k2);
#pragma unroll
            for (int w = kRowUnroll / 2; w > 0; w >>= 1)
#pragma unroll
                for (int j = 0; j < w; ++j) e[j] += e[j + w];
            s += e[0];
        }
        for (; v < V; v += stride) s += hw_ex2((x[v] - m) * k2);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(kFull, s, o);
    if (lane == 0) {
        *m_out = m;
        *s_out = s;
    }
}

// The accept walk, one warp: lane i < K merges row i's wpr parts into its max
// M and sum Z and tests draft i, accepted iff p_d > 0 and u_i < p_t / p_d
// (as u_i p_d Z < 2^((x_d - M) k2)); the first failure stops the walk.  An
// out-of-range token stops it with no draw (checked only where the walk
// reaches it).
__device__ __noinline__ void accept_walk(VerifyScalars *S, const float *st, int K, int V, int wpr, float k2,
                                         int flags, int32_t *err) {
    const int lane = threadIdx.x & 31;
    bool ok = true, bad_token = false;
    if (lane < K) {
        float M = -INFINITY, Z = 0.0f;
        for (int w = 0; w < wpr; ++w) M = fmaxf(M, S->red_m[lane * wpr + w]);
        for (int w = 0; w < wpr; ++w) {
            const float mw = S->red_m[lane * wpr + w];
            if (mw != -INFINITY) Z += S->red_s[lane * wpr + w] * hw_ex2((mw - M) * k2);
        }
        S->row_max[lane] = M;
        S->row_sum[lane] = Z;
        const int d = S->acc_d[lane];
        if (d < 0 || d >= V) {
            ok = false;
            bad_token = true;
        } else {
            const float e = hw_ex2((st[static_cast<size_t>(lane) * V + d] - M) * k2);
            const float pd = S->acc_pd[lane];
            ok = pd > 0.0f && S->acc_u[lane] * pd * Z < e;
        }
    }
    const unsigned fails = __ballot_sync(kFull, lane < K && !ok);
    const unsigned bads = __ballot_sync(kFull, bad_token);
    const int reject = fails ? __ffs(fails) - 1 : -1;
    const bool bad_first = reject >= 0 && ((bads >> reject) & 1u);
    if (lane == 0) {
        if (bad_first) flag_error(err, TTS_ERRBIT_TOKEN);
        S->reject = reject;
        S->accepted = reject >= 0 ? reject : K;
        S->draw = !bad_first && (reject >= 0 || (flags & TTS_VERIFY_BONUS)) ? 1 : 0;
    }
}

// One entry of the residual draw: folds its key log(residual) + g into
// `best` when the residual max(2^((x - m) k2) iz - p_d, 0) is positive.
__device__ __forceinline__ void draw_residual(float xv, float pv, float g, int v, float m, float iz, float k2,
                                              unsigned long long &best) {
    constexpr float kLn2 = 0.69314718055994531f;
    const float r = fmaxf(hw_ex2((xv - m) * k2) * iz - pv, 0.0f);
    if (r > 0.0f) {
        const unsigned long long k = pack_argmax(kLn2 * hw_lg2(r) + g, v);
        best = k > best ? k : best;
    }
}
// One thread's part of the draw over row x, entries v = v0, v0 + stride, ...:
// the largest packed (key, index) of log(residual) + G over entries with a
// positive residual when pdr (the rejected row's draft probabilities) is
// given, else of x / T + G (0 if none).
__device__ __noinline__ unsigned long long draw_part(const float *x, const float *pdr, const float *G, int V, int v0,
                                                     int stride, float m, float iz, float inv_t, float k2) {
    unsigned long long best = 0ull;
    const int span = kDrawUnroll * stride;
    int v = v0;
    if (pdr) {
        for (; v + (kDrawUnroll - 1) * stride < V; v += span) {
            float xv[kDrawUnroll], pv[kDrawUnroll], gv[kDrawUnroll];
#pragma unroll
            for (int j = 0; j < kDrawUnroll; ++j) {
                xv[j] = x[v + j * stride];
                pv[j] = pdr[v + j * stride];
                gv[j] = G[v + j * stride];
            }
#pragma unroll
            for (int j = 0; j < kDrawUnroll; ++j) draw_residual(xv[j], pv[j], gv[j], v + j * stride, m, iz, k2, best);
        }
        for (; v < V; v += stride) draw_residual(x[v], pdr[v], G[v], v, m, iz, k2, best);
    } else {
        for (; v + (kDrawUnroll - 1) * stride < V; v += span) {
            float xv[kDrawUnroll], gv[kDrawUnroll];
#pragma unroll
            for (int j = 0; j < kDrawUnroll; ++j) {
                xv[j] = x[v + j * stride];
                gv[j] = G[v + j * stride];
            }
#pragma unroll
            for (int j = 0; j < kDrawUnroll; ++j) {
                const unsigned long long k = pack_argmax(xv[j] * inv_t + gv[j], v + j * stride);
                best = k > best ? k : best;
            }
        }
        for (; v < V; v += stride) {
            const unsigned long long k = pack_argmax(x[v] * inv_t + G[v], v);
            best = k > best ? k : best;
        }
    }
    return best;
}

// The block's largest of each thread's `best` into *dst (a shared word that
// starts at 0); every thread returns after the block barrier.
__device__ __forceinline__ void block_max_key(unsigned long long best, unsigned long long *dst) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long other = __shfl_xor_sync(kFull, best, o);
        best = other > best ? other : best;
    }
    if ((threadIdx.x & 31) == 0 && best) atomicMax(dst, best);
    __syncthreads();
}

// Staged kernel, one CTA per stream.  The stream's rows arrive by bulk copies
// (target rows on one barrier, draft rows on another) while warps compute
// what depends only on the stream's key: the draw's Gumbel noise for every
// vocabulary entry (keyed by (stream, step, entry): a stream draws at most
// once per call, from whichever row) and the accept test's inputs.  Then each
// target row's max and sum of exp((x - max) / T) (per warp: the max of its
// part, then the sum against it; merged across warps with rescaling), the
// accept walk in one warp, and the draw over the chosen row from shared
// memory, spread over every thread.  Every exit waits (bounded) for the
// copies into shared memory.
__global__ void __launch_bounds__(kStagedThreads)
spec_verify_staged_kernel(const float *__restrict__ tl, const float *__restrict__ dp,
                          const int32_t *__restrict__ dt, int K, int V, float T,
                          const uint64_t *__restrict__ seed, const uint64_t *__restrict__ step, int flags,
                          int32_t *__restrict__ n_accepted, int32_t *__restrict__ next_token,
                          int32_t *err) {
    extern __shared__ __align__(16) float sm[];
    __shared__ __align__(8) uint64_t bars[2];  // target rows, draft rows
    __shared__ VerifyScalars S, scratch;       // scratch: the warm-up runs' outputs
    const int b = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t bar_t = smem_addr(&bars[0]), bar_d = smem_addr(&bars[1]);
    const float *tl_b = tl + static_cast<size_t>(b) * (K + 1) * V;
    const float *dp_b = dp + static_cast<size_t>(b) * K * V;
    const uint32_t nt = staged_target_rows(K, flags) * static_cast<uint32_t>(V);
    const uint32_t nd = static_cast<uint32_t>(K) * static_cast<uint32_t>(V);
    const StagedLayout Lo = staged_layout(K, V, flags);
    float *st = sm + ((reinterpret_cast<uintptr_t>(tl_b) & 15) >> 2);
    float *sdr = sm + Lo.draft + ((reinterpret_cast<uintptr_t>(dp_b) & 15) >> 2);
    float *G = sm + Lo.noise;
    pdl_wait_prerequisites();  // the target rows may come from the kernel before
    if (threadIdx.x == 0) {
        mbar_init(bar_t, 1);
        mbar_init(bar_d, 1);
        fence_mbar_init();
        S.best = 0ull;
        S.best_p = 0ull;
        S.ok = 1;
        // target rows first (the statistics need them first)
        mbar_arrive_expect_tx(bar_t, interior_bytes(tl_b, nt));
        stage_bulk(st, tl_b, nt, bar_t);
        mbar_arrive_expect_tx(bar_d, interior_bytes(dp_b, nd));
        stage_bulk(sdr, dp_b, nd, bar_d);
    }
    __syncthreads();  // the barriers are initialised before anyone waits
    pdl_allow_dependents();
    const uint64_t key0 = seed[b], key1 = step[b];
    const int groups = (V + 7) / 8;
    const float inv_t = 1.0f / T, k2 = 1.4426950408889634f / T;
    const int wpr = K >= kStagedWarps ? 1 : kStagedWarps / K;

    // ---- while the rows land.  Three warps each run one of the later
    // phases once on scratch data first (reading scratch or in-flight shared
    // memory, writing only `scratch`), so that the three fetch their
    // instructions in parallel and early; their own global loads are issued
    // before the warm-up and used after it.
    if (warp == kRaggedWarp) {
        // the rows' unaligned ends: at most one head and one tail float per
        // lane and image (all of a row image below 16 bytes: plain copies)
        float *dst_h[2], *dst_t[2];
        float val_h[2], val_t[2];
#pragma unroll
        for (int part = 0; part < 2; ++part) {
            float *dst = part ? sdr : st;
            const float *g = part ? dp_b : tl_b;
            const size_t n = part ? nd : nt;
            const uintptr_t s0 = reinterpret_cast<uintptr_t>(g), s1 = s0 + n * 4;
            const uintptr_t a0 = (s0 + 15) & ~uintptr_t(15), a1 = s1 & ~uintptr_t(15);
            dst_h[part] = dst_t[part] = nullptr;
            val_h[part] = val_t[part] = 0.0f;
            if (a1 <= a0) {
                for (size_t i = lane; i < n; i += 32) dst[i] = __ldg(g + i);
            } else {
                const size_t head = (a0 - s0) / 4, tail_from = (a1 - s0) / 4;
                if (static_cast<size_t>(lane) < head) {
                    dst_h[part] = dst + lane;
                    val_h[part] = __ldg(g + lane);
                }
                if (tail_from + lane < n) {
                    dst_t[part] = dst + tail_from + lane;
                    val_t[part] = __ldg(g + tail_from + lane);
                }
            }
        }
        warp_row_part(G, V < 256 ? V : 256, 0, 32, k2, &scratch.warm_m, &scratch.warm_s);
#pragma unroll
        for (int part = 0; part < 2; ++part) {
            if (dst_h[part]) *dst_h[part] = val_h[part];
            if (dst_t[part]) *dst_t[part] = val_t[part];
        }
    } else if (warp == kAcceptWarp) {
        const int d = lane < K ? dt[static_cast<size_t>(b) * K + lane] : 0;
        if (lane < kMaxK) scratch.acc_d[lane] = 0;
        scratch.red_m[lane] = 0.0f;
        scratch.red_s[lane] = 1.0f;
        __syncwarp();
        // a one-entry "row" per lane inside scratch (V = 1, every token 0)
        accept_walk(&scratch, scratch.red_s, K, 1, wpr, k2, flags, nullptr);
        if (lane < K) {
            S.acc_d[lane] = d;
            S.acc_pd[lane] = (d >= 0 && d < V) ? __ldg(dp_b + static_cast<size_t>(lane) * V + d) : 0.0f;
            S.acc_u[lane] = philox_uniform(key0, key1, 1u, 0u, static_cast<uint32_t>(lane));
        }
    } else if (warp == kDrawWarmWarp) {
        const int vw = V < 256 ? V : 256;  // long enough to run the unrolled loops
        const unsigned long long wr = draw_part(G, G, G, vw, lane, 32, 0.0f, 1.0f, inv_t, k2);
        const unsigned long long wp = draw_part(G, nullptr, G, vw, lane, 32, 0.0f, 1.0f, inv_t, k2);
        if (lane == 0) scratch.best = wr ^ wp;
    } else {
        for (int gi = threadIdx.x; gi < groups; gi += kNoiseThreads) {
            const Philox4x64 ph(static_cast<uint64_t>(gi), 2u, 0u, 0u, key0, key1);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int v = gi * 8 + e;
                if (v < V) G[v] = gumbel_from_uniform(bits_to_uniform(ph.half(e)));
            }
        }
    }
    if (!mbar_wait(bar_t, 0)) S.ok = 0;
    __syncthreads();  // also orders the ragged ends, the noise and the accept inputs
    if (!S.ok) {
        if (threadIdx.x == 0) {
            flag_error(err, TTS_ERRBIT_TIMEOUT);
            n_accepted[b] = 0;
            next_token[b] = -1;
            mbar_wait(bar_t, 0);  // bounded: let the copies land before the CTA exits
            mbar_wait(bar_d, 0);
        }
        return;
    }

    // ---- max and sum of exp((x - M) / T) of the K target rows, wpr warps per row
    const int my_row = warp / wpr, sub = warp - my_row * wpr;
    if (my_row < K)
        warp_row_part(st + static_cast<size_t>(my_row) * V, V, sub * 32, wpr * 32, k2, &S.red_m[warp],
                      &S.red_s[warp]);
    __syncthreads();
    if (warp == 0) accept_walk(&S, st, K, V, wpr, k2, flags, err);
    __syncthreads();
    if (!S.draw) {
        if (threadIdx.x == 0) {
            n_accepted[b] = S.accepted;
            next_token[b] = -1;
            if (!mbar_wait(bar_d, 0)) flag_error(err, TTS_ERRBIT_TIMEOUT);  // the copies land before the exit
        }
        return;
    }
    const int reject = S.reject;
    if (reject >= 0) {  // the residual reads the rejected row's draft probabilities
        if (!mbar_wait(bar_d, 0)) S.ok = 0;
        __syncthreads();
        if (!S.ok) {
            if (threadIdx.x == 0) {
                flag_error(err, TTS_ERRBIT_TIMEOUT);
                n_accepted[b] = 0;
                next_token[b] = -1;
                mbar_wait(bar_d, 0);
            }
            return;
        }
    }

    // ---- the replacement draw (rejection at row `reject`) or the bonus draw
    // (row K).  Rejection: key log(residual) + G over entries with a positive
    // residual; only if there is none (a residual that is zero everywhere) a
    // second pass with x / T + G, the argmax of log p_t + G (p_t is exp(x / T)
    // up to a common factor): the draw falls back to p_t.  Bonus: x / T + G.
    const int row = reject >= 0 ? reject : K;
    const float *x = st + static_cast<size_t>(row) * V;
    if (reject >= 0) {
        block_max_key(draw_part(x, sdr + static_cast<size_t>(row) * V, G, V, threadIdx.x, blockDim.x,
                                S.row_max[row], 1.0f / S.row_sum[row], inv_t, k2),
                      &S.best);
        // a residual that is zero everywhere (p_t = p_d up to rounding): p_t
        if (S.best == 0ull)
            block_max_key(draw_part(x, nullptr, G, V, threadIdx.x, blockDim.x, 0.0f, 1.0f, inv_t, k2), &S.best_p);
    } else {
        block_max_key(draw_part(x, nullptr, G, V, threadIdx.x, blockDim.x, 0.0f, 1.0f, inv_t, k2), &S.best_p);
    }
    if (threadIdx.x == 0) {
        const unsigned long long pick = reject >= 0 && S.best ? S.best : S.best_p;
        n_accepted[b] = S.accepted;
        next_token[b] = pick ? unpack_index(pick) : -1;
        if (reject < 0 && !mbar_wait(bar_d, 0)) flag_error(err, TTS_ERRBIT_TIMEOUT);  // before the exit
    }
}

// Test support: the Gumbel noise of n 32-bit Philox words.
__global__ void gumbel_noise_kernel(const uint32_t *bits, float *out, int n) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) out[i] = gumbel_from_uniform(bits_to_uniform(bits[i]));
}

}  // namespace
}  // namespace tts

extern "C" int tts_spec_verify(const float *d_target_logits, const float *d_draft_probs,
                               const int32_t *d_draft_tokens, int32_t B, int32_t K, int32_t V,
                               float temperature, const uint64_t *d_seed, const uint64_t *d_step,
                               int32_t flags, int32_t *d_n_accepted, int32_t *d_next_token,
                               int32_t *d_err, void *stream) {
    using namespace tts;
    if (!d_target_logits || !d_draft_probs || !d_draft_tokens || !d_seed || !d_step ||
        !d_n_accepted || !d_next_token)
        return TTS_ERR_INVALID;
    if (B < 0 || K < 1 || K > kMaxK || V < 1 || !(temperature > 0.0f) ||
        temperature == INFINITY || (flags & ~TTS_VERIFY_BONUS) != 0)
        return TTS_ERR_INVALID;
    if (B == 0) return TTS_OK;
    const size_t smem = staged_layout(K, V, flags).bytes;
    if (smem <= 200u * 1024u) {
        if (!ensure_dynamic_smem(reinterpret_cast<const void *>(spec_verify_staged_kernel), static_cast<int>(smem)))
            return TTS_ERR_CUDA;
        spec_verify_staged_kernel<<<B, kStagedThreads, smem, static_cast<cudaStream_t>(stream)>>>(
            d_target_logits, d_draft_probs, d_draft_tokens, K, V, temperature, d_seed, d_step, flags,
            d_n_accepted, d_next_token, d_err);
    } else {
        spec_verify_kernel<<<B, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
            d_target_logits, d_draft_probs, d_draft_tokens, K, V, temperature, d_seed, d_step, flags,
            d_n_accepted, d_next_token, d_err);
    }
    return launch_status();
}

extern "C" int tts_test_gumbel_noise(const uint32_t *d_bits, float *d_out, int32_t n, void *stream) {
    using namespace tts;
    if (n < 0 || (n > 0 && (!d_bits || !d_out))) return TTS_ERR_INVALID;
    if (n == 0) return TTS_OK;
    gumbel_noise_kernel<<<(n + 255) / 256, 256, 0, static_cast<cudaStream_t>(stream)>>>(d_bits, d_out, n);
    return launch_status();
}
