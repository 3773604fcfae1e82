// Speculative verification of K draft tokens per stream ("Optimizing
// Streaming Text-to-Speech Models for Sub-50 Millisecond Latency", section
// "Speculative Decoding for Acoustic Tokens"), generalised from the page's
// batch row 0 to every stream, with seeded Philox uniforms in place of an
// unseeded generator and the rejection draw done by Gumbel-max over the log of
// the clamped residual (the same distribution as normalising and sampling it).
//
// One CTA per stream.  Phase 1: each warp reduces one target row to its max
// and sum of exp((x - max) / T).  Phase 2: one thread walks the drafts in
// order and stops at the first rejection.  Phase 3: the CTA draws the
// replacement (or bonus) token with a block-wide argmax over packed
// (key, index) pairs; each thread handles groups of 8 consecutive vocabulary
// entries so one Philox block feeds 8 draws.
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
    spec_verify_kernel<<<B, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        d_target_logits, d_draft_probs, d_draft_tokens, K, V, temperature, d_seed, d_step, flags,
        d_n_accepted, d_next_token, d_err);
    return launch_status();
}
