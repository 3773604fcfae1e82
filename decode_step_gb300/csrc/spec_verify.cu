// Speculative verification of K draft tokens per stream ("Optimizing
// Streaming Text-to-Speech Models for Sub-50 Millisecond Latency", section
// "Speculative Decoding for Acoustic Tokens"), generalised from the page's
// batch row 0 to every stream, with seeded Philox uniforms in place of an
// unseeded generator and the rejection draw done by Gumbel-max over the log of
// the clamped residual (the same distribution as normalising and sampling it).
//
// One CTA per stream.  Staged kernel (the stream's rows fit in shared
// memory): bulk copies bring the K target rows (K + 1 with the bonus draw)
// and the K draft rows into shared memory at once; warp groups reduce each
// target row to its max and sum of exp((x - max) / T); lane i of one warp
// tests draft i and a ballot finds the first rejection; the CTA draws the
// replacement (or bonus) token with a block-wide argmax over packed
// (key, index) pairs, each thread taking groups of 8 consecutive vocabulary
// entries so one Philox block feeds 8 draws.  Streaming kernel (rows too
// large for shared memory): the same steps reading global memory.
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
        const Philox4x64 ph(static_cast<uint64_t>(gi), 2u, static_cast<uint64_t>(row), 0u, key0, key1);
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

// Shared-memory image of `n` floats at `g`: the 16-byte-aligned interior by
// bulk copies (one thread, completing on `bar`, whose expected bytes are
// already set), the ragged ends by plain loads of the calling threads.
// `dst` is congruent to `g` modulo 16.
__device__ void stage_floats(float *dst, const float *g, size_t n, uint32_t bar) {
    const uintptr_t s0 = reinterpret_cast<uintptr_t>(g), s1 = s0 + n * 4;
    const uintptr_t a0 = (s0 + 15) & ~uintptr_t(15), a1 = s1 & ~uintptr_t(15);
    if (a1 <= a0) {  // no aligned interior
        for (size_t i = threadIdx.x; i < n; i += blockDim.x) dst[i] = __ldg(g + i);
        return;
    }
    const size_t head = (a0 - s0) / 4, tail_from = (a1 - s0) / 4;
    for (size_t i = threadIdx.x; i < head; i += blockDim.x) dst[i] = __ldg(g + i);
    for (size_t i = tail_from + threadIdx.x; i < n; i += blockDim.x) dst[i] = __ldg(g + i);
    const uint32_t bytes = static_cast<uint32_t>(a1 - a0);
    if (threadIdx.x == 0) {
        const uint32_t d = smem_addr(dst + head);
        const uint8_t *src = reinterpret_cast<const uint8_t *>(a0);
        for (uint32_t off = 0; off < bytes; off += kBulkChunk) {
            const uint32_t len = bytes - off < kBulkChunk ? bytes - off : kBulkChunk;
            bulk_load_nohint(d + off, src + off, len, bar);
        }
    }
}

struct StagedLayout {
    uint32_t target, draft, total;  // float offsets of the two images (mod-16 placed), bytes
};
__host__ __device__ inline uint32_t staged_target_rows(int K, int flags) {
    return static_cast<uint32_t>(K) + ((flags & TTS_VERIFY_BONUS) ? 1u : 0u);
}
// Byte offsets of the images are chosen per stream (their alignment follows
// the global rows); this bounds the room they need.
__host__ __device__ inline uint32_t staged_bytes(int K, int V, int flags) {
    return (staged_target_rows(K, flags) + static_cast<uint32_t>(K)) * static_cast<uint32_t>(V) * 4u + 64u;
}

__global__ void __launch_bounds__(kStagedThreads)
spec_verify_staged_kernel(const float *__restrict__ tl, const float *__restrict__ dp,
                          const int32_t *__restrict__ dt, int K, int V, float T,
                          const uint64_t *__restrict__ seed, const uint64_t *__restrict__ step, int flags,
                          int32_t *__restrict__ n_accepted, int32_t *__restrict__ next_token,
                          int32_t *err) {
    extern __shared__ __align__(16) float sm[];
    __shared__ __align__(8) uint64_t bar_storage;
    __shared__ float red_m[kStagedWarps], red_s[kStagedWarps];
    __shared__ float row_max[kMaxK], row_sum[kMaxK];
    __shared__ int s_reject, s_accepted, s_draw, s_ok;
    __shared__ unsigned long long s_best, s_best_p;
    const int b = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t bar = smem_addr(&bar_storage);
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
        s_best = 0ull;
        s_best_p = 0ull;
        s_ok = 1;
    }
    __syncthreads();
    pdl_wait_prerequisites();
    pdl_allow_dependents();

    // ---- stage the rows: each image starts at the float offset that makes it
    // congruent to its global rows modulo 16 bytes
    const float *tl_b = tl + static_cast<size_t>(b) * (K + 1) * V;
    const float *dp_b = dp + static_cast<size_t>(b) * K * V;
    const uint32_t nt = staged_target_rows(K, flags) * static_cast<uint32_t>(V);
    const uint32_t nd = static_cast<uint32_t>(K) * static_cast<uint32_t>(V);
    float *st = sm + ((reinterpret_cast<uintptr_t>(tl_b) & 15) >> 2);
    float *sdr = sm + ((nt + 4 + 3) & ~3u) + ((reinterpret_cast<uintptr_t>(dp_b) & 15) >> 2);
    if (threadIdx.x == 0) mbar_arrive_expect_tx(bar, interior_bytes(tl_b, nt) + interior_bytes(dp_b, nd));
    stage_floats(st, tl_b, nt, bar);
    stage_floats(sdr, dp_b, nd, bar);
    if (!mbar_wait(bar, 0)) {
        if (threadIdx.x == 0) s_ok = 0;
    }
    __syncthreads();  // also orders the ragged ends' plain stores
    if (!s_ok) {
        if (threadIdx.x == 0) {
            flag_error(err, TTS_ERRBIT_TIMEOUT);
            n_accepted[b] = 0;
            next_token[b] = -1;
        }
        mbar_wait(bar, 0);  // bounded: let the copies land before the CTA exits
        return;
    }

    // ---- softmax statistics of the K target rows: wpr warps per row.
    // exp((x - M) / T) as exp2((x - M) * log2(e) / T).
    const float inv_t = 1.0f / T, k2 = 1.4426950408889634f / T;
    const int wpr = K >= kStagedWarps ? 1 : kStagedWarps / K;
    const int my_row = warp / wpr, sub = warp - my_row * wpr;
    const float *x_row = st + static_cast<size_t>(my_row) * V;
    if (my_row < K) {
        float m = -INFINITY;
        for (int v = sub * 32 + lane; v < V; v += wpr * 32) m = fmaxf(m, x_row[v]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
        if (lane == 0) red_m[warp] = m;
    }
    __syncthreads();
    if (my_row < K) {
        float M = -INFINITY;
        for (int w = 0; w < wpr; ++w) M = fmaxf(M, red_m[my_row * wpr + w]);
        float s = 0.0f;
        for (int v = sub * 32 + lane; v < V; v += wpr * 32) s += exp2f((x_row[v] - M) * k2);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(kFull, s, o);
        if (lane == 0) red_s[warp] = s;
        if (sub == 0 && lane == 0) row_max[my_row] = M;
    }
    __syncthreads();
    if (threadIdx.x < K) {
        float s = 0.0f;
        for (int w = 0; w < wpr; ++w) s += red_s[threadIdx.x * wpr + w];
        row_sum[threadIdx.x] = s;
    }
    __syncthreads();

    // ---- accept / reject: lane i tests draft i; the first failure stops
    if (warp == 0) {
        bool ok = true, bad_token = false;
        if (lane < K) {
            const int d = dt[static_cast<size_t>(b) * K + lane];
            if (d < 0 || d >= V) {
                ok = false;
                bad_token = true;
            } else {
                const float pt = exp2f((st[static_cast<size_t>(lane) * V + d] - row_max[lane]) * k2) / row_sum[lane];
                const float pd = sdr[static_cast<size_t>(lane) * V + d];
                ok = pd > 0.0f && philox_uniform(seed[b], step[b], 1u, 0u, static_cast<uint32_t>(lane)) < pt / pd;
            }
        }
        const unsigned fails = __ballot_sync(kFull, lane < K && !ok);
        const unsigned bads = __ballot_sync(kFull, bad_token);
        const int reject = fails ? __ffs(fails) - 1 : -1;
        // an out-of-range token stops the walk with no draw (checked only
        // where the walk reaches it)
        const bool bad_first = reject >= 0 && ((bads >> reject) & 1u);
        if (lane == 0) {
            if (bad_first) flag_error(err, TTS_ERRBIT_TOKEN);
            s_reject = reject;
            s_accepted = reject >= 0 ? reject : K;
            s_draw = !bad_first && (reject >= 0 || (flags & TTS_VERIFY_BONUS)) ? 1 : 0;
        }
    }
    __syncthreads();
    if (!s_draw) {
        if (threadIdx.x == 0) {
            n_accepted[b] = s_accepted;
            next_token[b] = -1;
        }
        return;
    }

    // ---- the replacement draw (rejection at row `reject`) or the bonus draw
    // (row K), in one pass.  Rejection: key log(residual) + G over entries with
    // a positive residual, and alongside it x / T + G (the argmax of
    // log p_t + G, as p_t is exp(x / T) up to a common factor) for the case of
    // a residual that is zero everywhere, where the draw falls back to p_t.
    // Bonus: x / T + G.
    const int reject = s_reject;
    const int row = reject >= 0 ? reject : K;
    const float *x = st + static_cast<size_t>(row) * V;
    const float *pdr = reject >= 0 ? sdr + static_cast<size_t>(row) * V : nullptr;
    const float m = reject >= 0 ? row_max[row] : 0.0f;
    const float iz = reject >= 0 ? 1.0f / row_sum[row] : 1.0f;
    const uint64_t key0 = seed[b], key1 = step[b];
    const int groups = (V + 7) / 8;
    unsigned long long best_r = 0ull, best_p = 0ull;
    for (int gi = threadIdx.x; gi < groups; gi += blockDim.x) {
        const Philox4x64 ph(static_cast<uint64_t>(gi), 2u, static_cast<uint64_t>(row), 0u, key0, key1);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int v = gi * 8 + e;
            if (v >= V) break;
            const float g = gumbel_from_uniform(bits_to_uniform(ph.half(e)));
            const unsigned long long kp = pack_argmax(x[v] * inv_t + g, v);
            best_p = kp > best_p ? kp : best_p;
            if (reject >= 0) {
                const float r = fmaxf(exp2f((x[v] - m) * k2) * iz - pdr[v], 0.0f);
                if (r > 0.0f) {
                    const unsigned long long kr = pack_argmax(logf(r) + g, v);
                    best_r = kr > best_r ? kr : best_r;
                }
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long a = __shfl_xor_sync(kFull, best_r, o);
        const unsigned long long c = __shfl_xor_sync(kFull, best_p, o);
        best_r = a > best_r ? a : best_r;
        best_p = c > best_p ? c : best_p;
    }
    if (lane == 0) {
        if (best_r) atomicMax(&s_best, best_r);
        if (best_p) atomicMax(&s_best_p, best_p);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned long long pick = reject >= 0 && s_best ? s_best : s_best_p;
        n_accepted[b] = s_accepted;
        next_token[b] = pick ? unpack_index(pick) : -1;
    }
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
    const size_t smem = staged_bytes(K, V, flags);
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
