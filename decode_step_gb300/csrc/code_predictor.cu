// The code predictor's frame loop ("How We Made a TTS Model Respond in
// Sub-50 ms", sections "Exploiting the regular building of the Code
// Predictor" and "Turn a fixed predictor loop into one GPU program": a fixed
// number of autoregressive steps per frame, one per remaining codebook, over a
// short bounded context in a preallocated KV cache, the whole loop one GPU
// program).
//
// Step i for every stream r (x = the talker's state for the frame at i = 0):
//   projection    q, k, v = bf16(x Wqkv^T)
//   append        k, v at position i of the stream's block
//   attention     o = bf16(attn(q; positions 0..i))
//   selection     token = argmax / Gumbel-max of o W_i^T (counter position i + 1)
//   next input    x = E_i[token]
// Two implementations.  By default one cooperative persistent kernel runs the
// whole frame (below).  Otherwise each stage is its own kernel (the head
// kernel's linear mode, the append, the decode attention, the head, a gather),
// each a programmatic dependent of the one before.  The cache holds one
// 16-token block per stream.
#include <cuda_runtime.h>

#include <algorithm>
#include <new>

#include "tts_common.cuh"
#include "tts_internal.h"

namespace tts {
namespace {

constexpr int kGatherThreads = 128;

// out[r] = table[ids[r]] (H bf16 values; a zero row for an id outside [0, V)).
__global__ void __launch_bounds__(kGatherThreads) gather_rows_kernel(const int32_t *__restrict__ ids,
                                                                     const uint4 *__restrict__ table, int V,
                                                                     int row_vecs, uint4 *__restrict__ out) {
    pdl_wait_prerequisites();
    pdl_allow_dependents();
    const int r = blockIdx.x;
    const int id = ids[r];
    const bool ok = id >= 0 && id < V;
    for (int c = threadIdx.x; c < row_vecs; c += blockDim.x)
        out[static_cast<size_t>(r) * row_vecs + c] =
            ok ? table[static_cast<size_t>(id) * row_vecs + c] : make_uint4(0u, 0u, 0u, 0u);
}

// The loop's constant arrays: block table (stream r owns block r) and, per
// step i, the context before (i) and after (i + 1) the append.
__global__ void predictor_init_kernel(int32_t *table, int32_t *ctx_before, int32_t *ctx_lens, int R, int n_steps) {
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t < R) table[t] = t;
    if (t < R * n_steps) {
        ctx_before[t] = t / R;
        ctx_lens[t] = t / R + 1;
    }
}

// ------------------------------------------------------- persistent kernel
//
// The whole frame in one cooperative launch: one CTA per SM, three phases per
// step separated by grid barriers.
//   A  every CTA stages the R input rows (x0, or step i-1's token embeddings
//      read straight from E) and its 16-feature slices of Wqkv in shared
//      memory and computes those q/k/v features (mma.sync m16n8k16, bf16 in,
//      fp32 accumulate, bf16 out);
//   B  one warp per (stream, query head): the new k, v go to the stream's
//      cache rows; attention over positions 0..i; o as bf16;
//   C  every CTA stages o and its 16-entry slices of W_i, computes the
//      logits and folds each row's best key (argmax or Gumbel-max) into the
//      row's 64-bit key with atomicMax.
// Step i's tokens are read from the keys by phase A of step i + 1 (and after
// the last barrier).  The barrier is a counter that only grows during a
// launch; each wait is bounded (TTS_ERRBIT_TIMEOUT and an abort flag that
// releases every other CTA).
constexpr int kPThreads = 256;
constexpr int kPWarps = kPThreads / 32;
constexpr int kPMaxRows = 64;     // R: four 16-row MMA tiles
constexpr int kPMaxH = 1024;      // shared-memory rows of H bf16 (+ padding)

struct PersistArgs {
    int R, H, Hq, Hkv, V, n_steps, F, mode;
    float temperature, scale;
    const __nv_bfloat16 *x0, *Wqkv, *W, *E;
    const uint64_t *seed, *step;
    int32_t *tokens;
    __nv_bfloat16 *qkv, *kc, *vc, *o;
    unsigned long long *keys;  // [2][R]
    unsigned int *bar;         // [0] barrier count, [1] abort
    int32_t *err;
    long long wait_limit;      // SM clock cycles per bounded wait
    int stall;                 // test support: the first grid barrier waits for one CTA too many
};

__device__ __forceinline__ void p_ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void p_mma(float *d, const uint32_t *a, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ unsigned int ld_acquire_u32(const unsigned int *p) {
    unsigned int v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Grid barrier number `k` (1, 2, ...): false if it timed out or another CTA aborted.
__device__ bool p_grid_sync(const PersistArgs &a, unsigned int k) {
    __shared__ int ok;
    __syncthreads();
    if (threadIdx.x == 0) {
        ok = 1;
        // arrival with release semantics: the CTA's writes (ordered before it
        // by the barrier above) are visible to whoever acquires the count
        asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(a.bar) : "memory");
        const unsigned int target = k * gridDim.x + (a.stall && k == 1 ? 1u : 0u);
        const long long t0 = clock64();
        // poll the count alone (acquire); the abort word and the clock every
        // 16th poll
        for (uint32_t n = 0;; ++n) {
            if (ld_acquire_u32(a.bar) >= target) break;
            if ((n & 15u) == 15u) {
                if (ld_acquire_u32(a.bar + 1) != 0u) {
                    ok = 0;
                    break;
                }
                if (clock64() - t0 > a.wait_limit) {
                    flag_error(a.err, TTS_ERRBIT_TIMEOUT);
                    atomicExch(a.bar + 1, 1u);
                    ok = 0;
                    break;
                }
            }
        }
    }
    __syncthreads();
    return ok != 0;
}

// D[16 x 16] (two n-tiles) += A rows [16 m, 16 m + 16) . B rows [0, 16) over
// k-steps [k0, k1) of 16; A and B in shared memory, rows `stride` bytes apart.
__device__ __forceinline__ void p_tile(uint32_t a_base, uint32_t b_base, uint32_t stride, int k0, int k1, float (&acc)[2][4],
                                       int lane) {
    const int mi = lane >> 3, mr = lane & 7;
    const uint32_t a_row = a_base + static_cast<uint32_t>(((mi & 1) * 8 + mr)) * stride + (mi >> 1) * 16;
    const uint32_t b_row = b_base + static_cast<uint32_t>(((mi >> 1) * 8 + mr)) * stride + (mi & 1) * 16;
    for (int ks = k0; ks < k1; ++ks) {
        uint32_t af[4], b0, b1, b2, b3;
        p_ldsm_x4(a_row + ks * 32, af[0], af[1], af[2], af[3]);
        p_ldsm_x4(b_row + ks * 32, b0, b1, b2, b3);
        p_mma(acc[0], af, b0, b1);
        p_mma(acc[1], af, b2, b3);
    }
}

__global__ void __launch_bounds__(kPThreads, 1) predictor_persistent_kernel(const PersistArgs a) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = (smem_addr(smem_raw) + 127u) & ~127u;
    uint8_t *smem = smem_raw + (base - smem_addr(smem_raw));
    const uint32_t stride = static_cast<uint32_t>(a.H + 8) * 2;  // padded row: conflict-free ldmatrix
    const uint32_t xs = base;                                    // [64][H + 8] bf16: x, then o
    const uint32_t wsm = xs + kPMaxRows * stride;                // [16][H + 8] bf16: weight rows
    const uint32_t bar = wsm + 16 * stride;                      // one mbarrier
    float *part = reinterpret_cast<float *>(smem + (bar - base) + 16);  // [4 warps][32 lanes][8] K-half partials
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int mtiles = (a.R + 15) / 16;
    const int HO = a.Hq * 128, group = a.Hq / a.Hkv;
    const int ksteps = a.H / 16;

    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    // rows R .. 63 of the input tile stay zero
    for (int i = threadIdx.x; i < (kPMaxRows - a.R) * (a.H / 8); i += blockDim.x) {
        const int r = a.R + i / (a.H / 8), c = i % (a.H / 8);
        *reinterpret_cast<uint4 *>(smem + static_cast<size_t>(r) * stride + c * 16) = make_uint4(0u, 0u, 0u, 0u);
    }
    __syncthreads();
    uint32_t phase = 0;
    unsigned int nsync = 0;
    bool alive = true;

    // stage `rows` global rows (row r at src(r)) into the input tile, plus 16
    // weight rows from wrow0; waits for both
    auto stage = [&](bool with_x, auto src_of, const __nv_bfloat16 *wrow0) -> bool {
        const uint32_t rowb = static_cast<uint32_t>(a.H) * 2;
        const int nx = with_x ? a.R : 0;
        if (threadIdx.x == 0) mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nx + 16) * rowb);
        __syncthreads();
        // one row copy per thread, all in flight together; the proxy fence
        // lets the copies see rows other CTAs stored before the last barrier
        for (int j = threadIdx.x; j < nx + 16; j += blockDim.x) {
            asm volatile("fence.proxy.async.global;" ::: "memory");
            if (j < nx)
                bulk_load_nohint(xs + j * stride, src_of(j), rowb, bar);
            else
                bulk_load_nohint(wsm + (j - nx) * stride, wrow0 + static_cast<size_t>(j - nx) * a.H, rowb, bar);
        }
        const bool ok = mbar_wait(bar, phase & 1u, a.wait_limit);
        ++phase;
        if (!ok && lane == 0) flag_error(a.err, TTS_ERRBIT_TIMEOUT);
        return ok;
    };

    // one 16-column chunk of A . W^T: warps (m-tile w % 4, K half w / 4); warps
    // 0-3 receive the other half through shared memory; emit(r, col, v0, v1)
    // for rows < R (cols col, col + 1 of the chunk)
    auto chunk_product = [&](auto emit) {
        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        const int mt = warp & 3, kh = warp >> 2;
        if (mt < mtiles) {
            const int half = ksteps / 2;
            p_tile(xs + static_cast<uint32_t>(mt * 16) * stride, wsm, stride, kh ? half : 0, kh ? ksteps : half, acc, lane);
        }
        if (kh == 1 && mt < mtiles) {
            float *dst = part + (static_cast<size_t>(mt) * 32 + lane) * 8;
#pragma unroll
            for (int n = 0; n < 2; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) dst[n * 4 + e] = acc[n][e];
        }
        __syncthreads();
        if (kh == 0 && mt < mtiles) {
            const float *src = part + (static_cast<size_t>(mt) * 32 + lane) * 8;
#pragma unroll
            for (int n = 0; n < 2; ++n)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[n][e] += src[n * 4 + e];
            const int g = lane >> 2, t = lane & 3;
#pragma unroll
            for (int n = 0; n < 2; ++n) {
                emit(mt * 16 + g, 8 * n + 2 * t, acc[n][0], acc[n][1]);
                emit(mt * 16 + g + 8, 8 * n + 2 * t, acc[n][2], acc[n][3]);
            }
        }
        __syncthreads();  // the weight rows and partials are free again
    };

    for (int i = 0; i < a.n_steps && alive; ++i) {
        // ---- A: the step's input rows and q, k, v
        const unsigned long long *prev = a.keys + static_cast<size_t>((i + 1) & 1) * a.R;  // step i-1's keys
        auto src_x = [&](int r) -> const __nv_bfloat16 * {
            if (i == 0) return a.x0 + static_cast<size_t>(r) * a.H;
            int tok = unpack_index(prev[r]);
            if (tok < 0 || tok >= a.V) tok = 0;
            return a.E + (static_cast<size_t>(i - 1) * a.V + tok) * a.H;
        };
        if (i > 0 && blockIdx.x == 0)
            for (int r = threadIdx.x; r < a.R; r += blockDim.x) {
                const unsigned long long k = prev[r];
                a.tokens[static_cast<size_t>(i - 1) * a.R + r] = k ? unpack_index(k) : -1;
            }
        bool first = true;
        for (int c = blockIdx.x; c < a.F / 16 && alive; c += gridDim.x) {
            if (!stage(first, src_x, a.Wqkv + static_cast<size_t>(c) * 16 * a.H)) {
                alive = false;
                break;
            }
            first = false;
            chunk_product([&](int r, int col, float v0, float v1) {
                if (r >= a.R) return;
                const __nv_bfloat162 p = __floats2bfloat162_rn(v0, v1);
                *reinterpret_cast<__nv_bfloat162 *>(a.qkv + static_cast<size_t>(r) * a.F + c * 16 + col) = p;
            });
        }
        if (!alive || !p_grid_sync(a, ++nsync)) break;

        // ---- B: append and attention, one warp per (stream, query head)
        // step i+1's keys must be zero before its phase C; step i-1's were read in A
        if (blockIdx.x == 0)
            for (int r = threadIdx.x; r < a.R; r += blockDim.x) a.keys[static_cast<size_t>((i + 1) & 1) * a.R + r] = 0ull;
        for (int p = blockIdx.x * kPWarps + warp; p < a.R * a.Hq; p += gridDim.x * kPWarps) {
            const int r = p / a.Hq, h = p % a.Hq, g = h / group;
            const __nv_bfloat16 *row = a.qkv + static_cast<size_t>(r) * a.F;
            const uint2 qw = *reinterpret_cast<const uint2 *>(row + h * 128 + 4 * lane);
            const uint2 kw = *reinterpret_cast<const uint2 *>(row + HO + g * 128 + 4 * lane);
            const uint2 vw = *reinterpret_cast<const uint2 *>(row + HO + a.Hkv * 128 + g * 128 + 4 * lane);
            const size_t cache_row = (static_cast<size_t>(r) * a.Hkv + g) * TTS_BLOCK_TOKENS;
            if (h % group == 0) {
                *reinterpret_cast<uint2 *>(a.kc + (cache_row + i) * 128 + 4 * lane) = kw;
                *reinterpret_cast<uint2 *>(a.vc + (cache_row + i) * 128 + 4 * lane) = vw;
            }
            const float q[4] = {bf16_lo(qw.x), bf16_hi(qw.x), bf16_lo(qw.y), bf16_hi(qw.y)};
            // every cached row's loads first, then the dot products, reduced
            // across the warp for all positions together
            float s[TTS_BLOCK_TOKENS];
            uint2 kk[TTS_BLOCK_TOKENS], vv[TTS_BLOCK_TOKENS];
#pragma unroll
            for (int t = 0; t < TTS_BLOCK_TOKENS; ++t) {
                if (t > i) break;
                kk[t] = t == i ? kw : *reinterpret_cast<const uint2 *>(a.kc + (cache_row + t) * 128 + 4 * lane);
                vv[t] = t == i ? vw : *reinterpret_cast<const uint2 *>(a.vc + (cache_row + t) * 128 + 4 * lane);
            }
#pragma unroll
            for (int t = 0; t < TTS_BLOCK_TOKENS; ++t) {
                if (t > i) break;
                float d = q[0] * bf16_lo(kk[t].x);
                d = fmaf(q[1], bf16_hi(kk[t].x), d);
                d = fmaf(q[2], bf16_lo(kk[t].y), d);
                s[t] = fmaf(q[3], bf16_hi(kk[t].y), d);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
#pragma unroll
                for (int t = 0; t < TTS_BLOCK_TOKENS; ++t)
                    if (t <= i) s[t] += __shfl_xor_sync(0xFFFFFFFFu, s[t], o);
            float m = -INFINITY;
#pragma unroll
            for (int t = 0; t < TTS_BLOCK_TOKENS; ++t) {
                if (t > i) break;
                s[t] *= a.scale;
                m = fmaxf(m, s[t]);
            }
            float l = 0.f, o4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int t = 0; t < TTS_BLOCK_TOKENS; ++t) {
                if (t > i) break;
                const float e = expf(s[t] - m);
                l += e;
                o4[0] = fmaf(e, bf16_lo(vv[t].x), o4[0]);
                o4[1] = fmaf(e, bf16_hi(vv[t].x), o4[1]);
                o4[2] = fmaf(e, bf16_lo(vv[t].y), o4[2]);
                o4[3] = fmaf(e, bf16_hi(vv[t].y), o4[3]);
            }
            const float inv = 1.0f / l;
            const __nv_bfloat162 lo = __floats2bfloat162_rn(o4[0] * inv, o4[1] * inv);
            const __nv_bfloat162 hi = __floats2bfloat162_rn(o4[2] * inv, o4[3] * inv);
            uint2 ow;
            ow.x = *reinterpret_cast<const uint32_t *>(&lo);
            ow.y = *reinterpret_cast<const uint32_t *>(&hi);
            *reinterpret_cast<uint2 *>(a.o + static_cast<size_t>(r) * HO + h * 128 + 4 * lane) = ow;
        }
        if (!p_grid_sync(a, ++nsync)) break;

        // ---- C: logits of this CTA's vocabulary slices and the rows' best keys
        unsigned long long *keys = a.keys + static_cast<size_t>(i & 1) * a.R;
        const __nv_bfloat16 *Wi = a.W + static_cast<size_t>(i) * a.V * a.H;
        auto src_o = [&](int r) -> const __nv_bfloat16 * { return a.o + static_cast<size_t>(r) * HO; };
        first = true;
        for (int c = blockIdx.x; c < a.V / 16 && alive; c += gridDim.x) {
            if (!stage(first, src_o, Wi + static_cast<size_t>(c) * 16 * a.H)) {
                alive = false;
                break;
            }
            first = false;
            chunk_product([&](int r, int col, float v0, float v1) {
                // the four lanes of a quad hold one row's 8 columns of an n-tile
                unsigned long long best = 0ull;
                if (r < a.R) {
                    const int v = c * 16 + col;
                    float k0 = v0, k1 = v1;
                    if (a.mode == TTS_GUMBEL) {
                        const Philox4x64 ph(static_cast<uint64_t>(v >> 3), 0, static_cast<uint64_t>(i + 1), 0,
                                            a.seed[r], a.step[r]);
                        k0 = v0 / a.temperature + gumbel_from_uniform(bits_to_uniform(ph.half(v & 7)));
                        k1 = v1 / a.temperature + gumbel_from_uniform(bits_to_uniform(ph.half((v + 1) & 7)));
                    }
                    const unsigned long long p0 = pack_argmax(k0, v), p1 = pack_argmax(k1, v + 1);
                    best = p0 > p1 ? p0 : p1;
                }
                unsigned long long other = __shfl_xor_sync(0xFFFFFFFFu, best, 1);
                best = other > best ? other : best;
                other = __shfl_xor_sync(0xFFFFFFFFu, best, 2);
                best = other > best ? other : best;
                if ((lane & 3) == 0 && r < a.R && best) atomicMax(keys + r, best);
            });
        }
        if (!alive || !p_grid_sync(a, ++nsync)) break;
    }
    // the last step's tokens
    if (alive && blockIdx.x == 0 && ld_acquire_u32(a.bar + 1) == 0u) {
        const int last = a.n_steps - 1;
        for (int r = threadIdx.x; r < a.R; r += blockDim.x) {
            const unsigned long long k = a.keys[static_cast<size_t>(last & 1) * a.R + r];
            a.tokens[static_cast<size_t>(last) * a.R + r] = k ? unpack_index(k) : -1;
        }
    }
}

size_t persistent_smem(int H) {
    return 128 + static_cast<size_t>(kPMaxRows + 16) * (H + 8) * 2 + 16 + 4 * 32 * 8 * sizeof(float);
}

constexpr size_t kAlign = 256;

struct PredictorLayout {
    size_t x, q, k, v, o, kpool, vpool, table, ctx_before, ctx_lens, attn_ws, attn_ws_bytes, head_ws, head_ws_bytes,
        qkv, keys, bar, total;
};

bool predictor_layout(int R, int H, int Hq, int Hkv, int D, int V, int n_steps, PredictorLayout *L) {
    if (R < 1 || R > 4096 || H < 1 || Hq < 1 || Hkv < 1 || D < 1 || V < 1 || n_steps < 1 ||
        n_steps > TTS_BLOCK_TOKENS)
        return false;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = align_up(off + bytes, kAlign);
        return at;
    };
    const size_t rows = static_cast<size_t>(R);
    L->x = take(rows * H * 2);
    L->q = take(rows * Hq * D * 2);
    L->k = take(rows * Hkv * D * 2);
    L->v = take(rows * Hkv * D * 2);
    L->o = take(rows * Hq * D * 2);
    const size_t pool = rows * Hkv * TTS_BLOCK_TOKENS * D * 2;
    L->kpool = take(pool);
    L->vpool = take(pool);
    L->table = take(rows * 4);
    L->ctx_before = take(rows * n_steps * 4);
    L->ctx_lens = take(rows * n_steps * 4);
    L->attn_ws_bytes = tts_decode_attn_workspace_size(R, 1, Hq, Hkv, D, TTS_BLOCK_TOKENS);
    L->head_ws_bytes = tts_head_workspace_size(R, V);
    if (L->attn_ws_bytes == 0 || L->head_ws_bytes == 0) return false;
    L->attn_ws = take(L->attn_ws_bytes);
    L->head_ws = take(L->head_ws_bytes);
    // the persistent kernel's q|k|v rows, row keys [2][R] and barrier words
    L->qkv = take(rows * (Hq + 2 * Hkv) * D * 2);
    L->keys = take(2 * rows * 8);
    L->bar = take(2 * 4);
    L->total = off;
    return true;
}

// Every launch of one frame, checked and prepared before anything runs.
struct PredictorPlan {
    bool persistent;
    PersistArgs pa;
    unsigned grid;
    size_t smem;
    void *ctrl;            // keys and barrier words, zeroed before each launch
    size_t ctrl_bytes;
    tts_kv_cache cache;
    int R, n_steps;
    int32_t *table, *ctx_before, *ctx_lens;
    HeadLaunch proj[TTS_BLOCK_TOKENS];
    AppendLaunch append[TTS_BLOCK_TOKENS];
    AttnLaunch attn[TTS_BLOCK_TOKENS];
    HeadLaunch select[TTS_BLOCK_TOKENS];
    const int32_t *gather_ids[TTS_BLOCK_TOKENS];
    const uint4 *gather_table[TTS_BLOCK_TOKENS];
    int V, row_vecs;
    uint4 *x;
};

int plan_predictor(const tts_code_predictor_desc *d, PredictorPlan *P) {
    if (!d || !d->d_x0 || !d->d_Wqkv || !d->d_W || !d->d_E || !d->d_tokens || !d->d_ws) return TTS_ERR_INVALID;
    const int R = d->R, H = d->H, Hq = d->num_q_heads, Hkv = d->num_kv_heads, D = d->head_dim, V = d->V;
    const int n = d->n_steps;
    PredictorLayout L;
    if (!predictor_layout(R, H, Hq, Hkv, D, V, n, &L)) return TTS_ERR_INVALID;
    if (Hq % Hkv != 0 || Hq * D != H) return TTS_ERR_UNSUPPORTED;  // the head reads o [R][Hq D] as [R][H]
    if (H % 8 != 0 || (Hq * D) % 8 != 0 || (Hkv * D) % 8 != 0) return TTS_ERR_UNSUPPORTED;
    if (d->ws_bytes < L.total || !aligned16(d->d_ws)) return TTS_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(d->d_ws) % kAlign != 0) return TTS_ERR_WORKSPACE;
    if (!aligned16(d->d_x0) || !aligned16(d->d_E)) return TTS_ERR_INVALID;
    if (d->mode == TTS_GUMBEL && (!d->d_seed || !d->d_step)) return TTS_ERR_INVALID;
    uint8_t *ws = static_cast<uint8_t *>(d->d_ws);
    // one cooperative launch when the shape fits its tiles: at most 64 rows,
    // H up to 1024, 16-wide feature and vocabulary slices
    const int F0 = (Hq + 2 * Hkv) * D;
    const int sms = sm_count();
    const int grid = std::max(F0 / 16, V / 16) < sms ? std::max(F0 / 16, V / 16) : sms;
    P->persistent = !(d->flags & TTS_PREDICTOR_MULTI_KERNEL) && R <= kPMaxRows && H <= kPMaxH && D == 128 &&
                    H % 16 == 0 && F0 % 16 == 0 && V % 16 == 0 && grid >= 1;
    if (P->persistent) {
        P->smem = persistent_smem(H);
        int dev = 0, coop = 0, per_sm = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess || !coop ||
            !ensure_dynamic_smem(reinterpret_cast<const void *>(predictor_persistent_kernel), static_cast<int>(P->smem)) ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, predictor_persistent_kernel, kPThreads, P->smem) !=
                cudaSuccess ||
            per_sm < 1) {
            cudaGetLastError();
            P->persistent = false;
        }
    }
    if (P->persistent) {
        PersistArgs &pa = P->pa;
        pa = PersistArgs{R, H, Hq, Hkv, V, n, F0, d->mode, d->temperature, 1.0f / sqrtf(static_cast<float>(D)),
                         static_cast<const __nv_bfloat16 *>(d->d_x0), static_cast<const __nv_bfloat16 *>(d->d_Wqkv),
                         static_cast<const __nv_bfloat16 *>(d->d_W), static_cast<const __nv_bfloat16 *>(d->d_E),
                         d->d_seed, d->d_step, d->d_tokens, reinterpret_cast<__nv_bfloat16 *>(ws + L.qkv),
                         reinterpret_cast<__nv_bfloat16 *>(ws + L.kpool), reinterpret_cast<__nv_bfloat16 *>(ws + L.vpool),
                         reinterpret_cast<__nv_bfloat16 *>(ws + L.o), reinterpret_cast<unsigned long long *>(ws + L.keys),
                         reinterpret_cast<unsigned int *>(ws + L.bar), d->d_err};
        pa.wait_limit = thread_opts().wait_limit;
        pa.stall = thread_opts().stall == TTS_TEST_STALL_PREDICTOR_GRID;
        P->grid = static_cast<unsigned>(grid);
        P->ctrl = ws + L.keys;
        P->ctrl_bytes = L.bar + 8 - L.keys;
        if (d->mode != TTS_ARGMAX && d->mode != TTS_GUMBEL) return TTS_ERR_INVALID;
        if (d->mode == TTS_GUMBEL && !(d->temperature > 0.0f)) return TTS_ERR_INVALID;
        return TTS_OK;
    }
    P->R = R;
    P->n_steps = n;
    P->V = V;
    P->row_vecs = H * 2 / 16;
    P->x = reinterpret_cast<uint4 *>(ws + L.x);
    P->table = reinterpret_cast<int32_t *>(ws + L.table);
    P->ctx_before = reinterpret_cast<int32_t *>(ws + L.ctx_before);
    P->ctx_lens = reinterpret_cast<int32_t *>(ws + L.ctx_lens);
    P->cache = tts_kv_cache{R, TTS_BLOCK_TOKENS, Hkv, D, TTS_BF16, ws + L.kpool, ws + L.vpool};
    const int F = (Hq + 2 * Hkv) * D;
    const float scale = 1.0f / sqrtf(static_cast<float>(D));
    for (int i = 0; i < n; ++i) {
        HeadExtras xp;
        xp.seg_start[0] = 0;
        xp.seg_start[1] = Hq * D;
        xp.seg_start[2] = (Hq + Hkv) * D;
        xp.seg_start[3] = F;
        xp.seg_out[0] = ws + L.q;
        xp.seg_out[1] = ws + L.k;
        xp.seg_out[2] = ws + L.v;
        const void *h = i == 0 ? d->d_x0 : static_cast<const void *>(ws + L.x);
        int st = prepare_head_ex(h, d->d_Wqkv, TTS_BF16, R, H, F, kHeadModeLinear, 0.0f, nullptr, nullptr, nullptr,
                                 nullptr, nullptr, nullptr, nullptr, 0, xp, &P->proj[i]);
        if (st != TTS_OK) return st;
        st = prepare_append(&P->cache, P->table, 1, P->ctx_before + static_cast<size_t>(i) * R, R, 1, ws + L.k,
                            ws + L.v, d->d_err, &P->append[i]);
        if (st != TTS_OK) return st;
        st = prepare_attn(&P->cache, P->table, 1, P->ctx_lens + static_cast<size_t>(i) * R, TTS_BLOCK_TOKENS, R, 1,
                          Hq, scale, 0, ws + L.q, ws + L.o, ws + L.attn_ws, L.attn_ws_bytes, d->d_err, &P->attn[i]);
        if (st != TTS_OK) return st;
        HeadExtras xs;
        xs.pos = static_cast<uint32_t>(i + 1);
        const __nv_bfloat16 *Wi = static_cast<const __nv_bfloat16 *>(d->d_W) + static_cast<size_t>(i) * V * H;
        st = prepare_head_ex(ws + L.o, Wi, TTS_BF16, R, H, V, d->mode, d->temperature, d->d_seed, d->d_step,
                             nullptr, d->d_tokens + static_cast<size_t>(i) * R, nullptr, nullptr, ws + L.head_ws,
                             L.head_ws_bytes, xs, &P->select[i]);
        if (st != TTS_OK) return st;
        P->gather_ids[i] = d->d_tokens + static_cast<size_t>(i) * R;
        P->gather_table[i] =
            reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(d->d_E) + static_cast<size_t>(i) * V * H);
    }
    return TTS_OK;
}

int launch_predictor(const PredictorPlan &P, cudaStream_t s) {
    if (P.persistent) {
        if (cudaMemsetAsync(P.ctrl, 0, P.ctrl_bytes, s) != cudaSuccess) {
            cudaGetLastError();
            return TTS_ERR_CUDA;
        }
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(P.grid, 1, 1);
        cfg.blockDim = dim3(kPThreads, 1, 1);
        cfg.dynamicSmemBytes = P.smem;
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, predictor_persistent_kernel, P.pa) != cudaSuccess) {
            cudaGetLastError();
            return TTS_ERR_CUDA;
        }
        return TTS_OK;
    }
    const int R = P.R;
    const int init_n = R * P.n_steps;
    predictor_init_kernel<<<(init_n + 255) / 256, 256, 0, s>>>(P.table, P.ctx_before, P.ctx_lens, R, P.n_steps);
    if (cudaGetLastError() != cudaSuccess) return TTS_ERR_CUDA;
    for (int i = 0; i < P.n_steps; ++i) {
        int st = launch_head(P.proj[i], {s, true});
        if (st == TTS_OK) st = launch_append(P.append[i], {s, true});
        if (st == TTS_OK) st = launch_attn(P.attn[i], {s, true});
        if (st == TTS_OK) st = launch_head(P.select[i], {s, true});
        if (st != TTS_OK) return st;
        if (i + 1 == P.n_steps) break;  // the last token's embedding feeds nothing
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(R), 1, 1);
        cfg.blockDim = dim3(kGatherThreads, 1, 1);
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, gather_rows_kernel, P.gather_ids[i], P.gather_table[i], P.V, P.row_vecs, P.x) !=
            cudaSuccess) {
            cudaGetLastError();
            return TTS_ERR_CUDA;
        }
    }
    return TTS_OK;
}

}  // namespace
}  // namespace tts

struct tts_code_predictor_graph {
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
};

extern "C" size_t tts_code_predictor_workspace_size(int32_t R, int32_t H, int32_t num_q_heads, int32_t num_kv_heads,
                                                    int32_t head_dim, int32_t V, int32_t n_steps) {
    tts::PredictorLayout L;
    if (!tts::predictor_layout(R, H, num_q_heads, num_kv_heads, head_dim, V, n_steps, &L)) return 0;
    return L.total;
}

extern "C" int tts_code_predictor_run(const tts_code_predictor_desc *d, void *stream) {
    using namespace tts;
    PredictorPlan *P = new (std::nothrow) PredictorPlan();
    if (!P) return TTS_ERR_CUDA;
    int st = plan_predictor(d, P);
    if (st == TTS_OK) st = launch_predictor(*P, static_cast<cudaStream_t>(stream));
    delete P;
    return st;
}

extern "C" int tts_code_predictor_graph_create(const tts_code_predictor_desc *d, tts_code_predictor_graph **out) {
    using namespace tts;
    if (!out) return TTS_ERR_INVALID;
    *out = nullptr;
    PredictorPlan *P = new (std::nothrow) PredictorPlan();
    if (!P) return TTS_ERR_CUDA;
    int st = plan_predictor(d, P);
    if (st != TTS_OK) {
        delete P;
        return st;
    }
    tts_code_predictor_graph *g = new (std::nothrow) tts_code_predictor_graph();
    cudaStream_t s;
    if (!g || cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) {
        cudaGetLastError();
        delete g;
        delete P;
        return TTS_ERR_CUDA;
    }
    // Relaxed capture: the launch helpers set function attributes, which is
    // not a stream operation.
    bool ok = cudaStreamBeginCapture(s, cudaStreamCaptureModeRelaxed) == cudaSuccess;
    if (ok) {
        ok = launch_predictor(*P, s) == TTS_OK;
        cudaGraph_t graph = nullptr;
        const bool ended = cudaStreamEndCapture(s, &graph) == cudaSuccess;
        ok = ok && ended;
        g->graph = graph;
        if (ok) ok = cudaGraphInstantiate(&g->exec, g->graph, 0) == cudaSuccess;
    }
    cudaStreamDestroy(s);
    delete P;
    if (!ok) {
        cudaGetLastError();
        if (g->exec) cudaGraphExecDestroy(g->exec);
        if (g->graph) cudaGraphDestroy(g->graph);
        delete g;
        return TTS_ERR_CUDA;
    }
    *out = g;
    return TTS_OK;
}

extern "C" int tts_code_predictor_graph_launch(tts_code_predictor_graph *g, void *stream) {
    if (!g || !g->exec) return TTS_ERR_INVALID;
    if (cudaGraphLaunch(g->exec, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return TTS_ERR_CUDA;
    }
    return TTS_OK;
}

extern "C" void tts_code_predictor_graph_destroy(tts_code_predictor_graph *g) {
    if (!g) return;
    if (g->exec) cudaGraphExecDestroy(g->exec);
    if (g->graph) cudaGraphDestroy(g->graph);
    delete g;
}
