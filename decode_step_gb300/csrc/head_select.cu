// Codebook head with fused token selection ("TontaubeV1: Streaming
// Text-to-Speech with Hierarchical Codec Modeling and Bounded Context",
// section 3: each stage scores its codebook (4,096 acoustic or 16,384 semantic
// entries plus a boundary token) and picks a token, at temperature zero for
// the later stages):
//   logits[r][v] = h[r] . W[v];  ids[r] = argmax_v logits[r][v]           (argmax)
//                                ids[r] = argmax_v logits[r][v] / T + G   (Gumbel-max)
//
// bf16: a tcgen05 tensor-core kernel.  The vocabulary is the MMA's M side
// (128 rows of W per tile) and the batch rows are the N side, so a small
// batch still fills the 128-row tensor-core tile.  Per CTA: a TMA producer
// warp streams W and h k-slices (SWIZZLE_128B) through a 4-stage shared-memory
// ring; one thread issues tcgen05.mma into a TMEM accumulator; four epilogue
// warps read the accumulator back with tcgen05.ld.  A cluster of CK CTAs
// splits the hidden dimension of one vocab tile; their partial logits are
// summed through distributed shared memory, so logits never go to global
// memory (unless the caller asks for them).  Selection is fused: each CTA
// reduces its rows to one packed (key, index) per batch row with a 64-bit
// atomicMax, and the last CTA to finish converts the keys to token ids and
// clears the workspace.  No CTA ever waits on another CTA outside its cluster.
//
// fp32: a CUDA-core kernel (tf32 tensor cores would change the rounding of
// fp32 inputs), one warp per vocabulary row.
#include <mutex>
#include <new>

#include "tts_common.cuh"
#include "tts_internal.h"

namespace tts {
namespace {

constexpr unsigned kFull = 0xFFFFFFFFu;
constexpr int kTileM = 128;           // vocab rows per MMA tile
constexpr int kTileK = 64;            // hidden elements per stage (one 128-byte swizzle span)
constexpr int kStagesTC = 4;
// Warps 0-3 read the accumulator, 4 is the TMA producer, 5 the MMA issuer;
// all of them share the token-selection loop, whose Gumbel path (one
// Philox4x64-10 block per 8 vocabulary entries) is bound by the latency of its
// 64-bit multiply chains and wants many warps: the Gumbel build runs 768
// threads (1024 for 256-column chunks, whose items then split evenly over
// the passes), at one CTA per SM (measured at 256 x 2048 x 16385: 41.0 us
// with 384 threads, 35.8 with 768, 34.0 with 1024; at 320 x 2048 x 4097 in
// 160-column chunks: 20.1, 17.7, 19.0).
constexpr int kThreadsTC = 384;
constexpr int kThreadsGumbel = 768;
constexpr int kThreadsGumbelWide = 1024;
__host__ __device__ constexpr int tc_threads(bool gumbel, int N) {
    return !gumbel ? kThreadsTC : (N >= 256 ? kThreadsGumbelWide : kThreadsGumbel);
}
constexpr int kMaxN = 256;            // widest MMA N
constexpr int kATileBytes = kTileM * kTileK * 2;  // 16 KB

// ------------------------------------------------------------ shared parts

struct HeadWs {
    unsigned long long *keys;  // [R] packed (key, index), zero between calls
    unsigned int *ticket;      // CTAs finished, zero between calls
};

HeadWs head_ws(void *ws, int R) {
    HeadWs w;
    w.keys = static_cast<unsigned long long *>(ws);
    w.ticket = reinterpret_cast<unsigned int *>(static_cast<uint8_t *>(ws) +
                                                align_up(static_cast<size_t>(R) * 8, 256));
    return w;
}

// Called by every thread of each of the `publishers` CTAs that publish keys,
// after their atomics.  The last of them converts keys to ids and resets the
// workspace.  No waiting.
// ids_host / count_host (nullable, pinned host memory): the ids again and the
// number of rows whose id is `boundary`, written by the last CTA; then, with
// seq_host, the launch's number (*seq_dev incremented) to seq_host, after a
// system-scope fence, so a host that sees the number sees the ids.
__device__ void finish_selection(const HeadWs &ws, int R, int32_t *ids, float *best, int *flag,
                                 unsigned int publishers, int32_t *ids_host = nullptr, int32_t *count_host = nullptr,
                                 int32_t boundary = -1, int32_t *seq_host = nullptr, uint32_t *seq_dev = nullptr) {
    // The barrier orders every thread's key atomics before thread 0's ticket,
    // whose release (cumulative) publishes them all.
    __syncthreads();
    if (threadIdx.x == 0) {
        // release: the CTA's key atomics (ordered before this by the barrier);
        // acquire, for the last CTA: every other CTA's
        unsigned int old;
        asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(ws.ticket) : "memory");
        *flag = old == publishers - 1u;
    }
    __syncthreads();
    if (!*flag) return;
    // The last CTA alone reads and clears the keys (L2 reads: the atomics live there).
    int hits = 0;
    for (int r = threadIdx.x; r < R; r += blockDim.x) {
        const unsigned long long k = __ldcg(ws.keys + r);
        ws.keys[r] = 0ull;
        const int32_t id = k ? unpack_index(k) : -1;
        ids[r] = id;
        if (ids_host) ids_host[r] = id;
        hits += id == boundary;
        if (best) best[r] = k ? unpack_value(k) : -INFINITY;
    }
    if (threadIdx.x == 0) *ws.ticket = 0u;
    if (count_host) {
        // the flag word is free again: reuse it as the CTA's counter
        __syncthreads();
        if (threadIdx.x == 0) *flag = 0;
        __syncthreads();
        hits = __reduce_add_sync(0xFFFFFFFFu, hits);
        if ((threadIdx.x & 31) == 0 && hits) atomicAdd(flag, hits);
        __syncthreads();
        if (threadIdx.x == 0) *count_host = *flag;
    }
    if (seq_host) {
        __syncthreads();  // every id and the count written before the number
        if (threadIdx.x == 0) {
            const unsigned int seq = atomicAdd(seq_dev, 1u) + 1u;
            __threadfence_system();
            *reinterpret_cast<volatile int32_t *>(seq_host) = static_cast<int32_t>(seq);
        }
    }
}

// Head modes beyond the public TTS_ARGMAX / TTS_GUMBEL: the first layer of
// the two-layer audio head writes Mish(h W^T + b) as bf16 instead of
// selecting; the linear mode writes h W^T as bf16 into up to three outputs
// (consecutive feature ranges, e.g. the q, k and v of a projection).
constexpr int kModeExpand = 2;
constexpr int kModeLinear = 3;

struct HeadArgs {
    int R, H, V, mode;
    float temperature;
    const uint64_t *seed;
    const uint64_t *step;
    const uint8_t *eos;
    float *logits_out;
    int32_t *ids;
    float *best;
    HeadWs ws;
    int32_t *err;
    const float *bias;        // [V] added to the logits (nullable)
    const uint32_t *tail;     // [R] mask bits of the last n_tail ids (nullable: eos, else all allowed)
    int n_tail;
    __nv_bfloat16 *z_out;     // kModeExpand: [R][V] bf16
    uint32_t pos;             // Gumbel noise counter position (tag 0, pos, idx)
    int seg_start[4];         // kModeLinear: feature range j = [seg_start[j], seg_start[j + 1])
    __nv_bfloat16 *seg_out[3];  //   written to seg_out[j] [R][seg_start[j + 1] - seg_start[j]]
    int32_t *ids_host;        // selection: the ids again, in pinned host memory (nullable)
    int32_t *count_host;      //   and the count of rows choosing id V - 1 (nullable)
    int32_t *seq_host;        //   and then the launch's number (nullable; with seq_dev)
    uint32_t *seq_dev;
};

// Mish(x) = x tanh(ln(1 + e^x)) in fp32 (past x = 20, ln(1 + e^x) rounds to x).
__device__ __forceinline__ float mish_f(float x) {
    const float sp = x > 20.0f ? x : log1pf(expf(x));
    return x * tanhf(sp);
}

// Margin (in Gumbel units) kept when skipping entries that cannot win; far
// larger than the rounding of the threshold's exponentials.
constexpr float kGumbelSlack = 0.01f;

// Gumbel-max selection key of logit `x` at the vocab entry drawing half `e`
// of its Philox block `ph` (block = entries 8 * (v / 8) .. 8 * (v / 8) + 7).
__device__ __forceinline__ float gumbel_key(const HeadArgs &a, float x, int e, const Philox4x64 &ph) {
    return x / a.temperature + gumbel_from_uniform(bits_to_uniform(ph.half(e)));
}

// ---------------------------------------------------------------- fp32 SIMT

__global__ void __launch_bounds__(256)
head_simt_f32_kernel(const float *__restrict__ h, const float *__restrict__ W, const HeadArgs a) {
    __shared__ int flag;
    pdl_wait_prerequisites();
    pdl_allow_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int warps_total = gridDim.x * (blockDim.x >> 5);
    for (int v = blockIdx.x * (blockDim.x >> 5) + warp; v < a.V; v += warps_total) {
        const float *w = W + static_cast<size_t>(v) * a.H;
        for (int r = 0; r < a.R; ++r) {
            const float *x = h + static_cast<size_t>(r) * a.H;
            float acc = 0.0f;
            for (int k = lane; k < a.H; k += 32) acc = fmaf(__ldg(w + k), __ldg(x + k), acc);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(kFull, acc, o);
            if (lane == (r & 31)) {
                if (a.logits_out) a.logits_out[static_cast<size_t>(r) * a.V + v] = acc;
                const int vmax = (a.eos && !a.eos[r]) ? a.V - 1 : a.V;
                if (v < vmax) {
                    float key = acc;
                    if (a.mode == TTS_GUMBEL) {
                        const Philox4x64 ph(static_cast<uint64_t>(v >> 3), 0, 0, 0, a.seed[r], a.step[r]);
                        key = gumbel_key(a, acc, v & 7, ph);
                    }
                    atomicMax(a.ws.keys + r, pack_argmax(key, v));
                }
            }
        }
    }
    finish_selection(a.ws, a.R, a.ids, a.best, &flag, gridDim.x * gridDim.y);
}

// --------------------------------------------------------- tcgen05 (bf16)

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
}
__device__ __forceinline__ uint32_t map_cluster(uint32_t addr, uint32_t rank) {
    uint32_t out;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(addr), "r"(rank));
    return out;
}
// Generic pointer to the same shared-memory object in cluster CTA `rank`.
template <typename T>
__device__ __forceinline__ T *map_cluster_ptr(T *p, uint32_t rank) {
    uint64_t out;
    asm volatile("mapa.u64 %0, %1, %2;" : "=l"(out) : "l"(reinterpret_cast<uint64_t>(p)), "r"(rank));
    return reinterpret_cast<T *>(out);
}
__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of
// 128 bytes, 8-row groups 1024 bytes apart (tcgen05 descriptor format:
// start >> 4 in bits 0-13, stride offset >> 4 in bits 32-45, version 1 in
// bits 46-47, swizzle mode 2 (128B) in bits 61-63).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr) {
    return static_cast<uint64_t>((addr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(1) << 16) |
           (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
           (static_cast<uint64_t>(2) << 61);
}

// Instruction descriptor, kind::f16: fp32 accumulator (bits 4-5 = 1), bf16 A
// and B (bits 7-9, 10-12 = 1), both K-major, N >> 3 in bits 17-22, M >> 4 in
// bits 24-28.
__host__ __device__ constexpr uint32_t mma_idesc(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float *v) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32"
        " {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Same, without waiting: the caller issues several and then tmem_wait_ld().
__device__ __forceinline__ void tmem_ld16_nowait(uint32_t taddr, uint32_t *r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32"
        " {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

struct TcLayout {
    uint32_t stage_bytes;   // A tile + B tile
    uint32_t dump_stride;   // floats per accumulator row in shared memory (N + 4)
    uint32_t recv;          // offset of the receive table (after the dump; both reuse the ring)
    uint32_t region;        // ring, or dump + receive table if larger
    uint32_t bars;          // offset of the mbarriers
    uint32_t colbest;       // offset of the per-column best keys ([8][N]: own, then peers' slots)
    uint32_t misc;          // TMEM address, flag
    uint32_t total;
};

// The ring holds the k-slices while the MMAs run; afterwards the same bytes
// hold this CTA's accumulator (the dump, 128 rows) and, with CK > 1, the
// receive table recv[source rank][RS rows] of the rows this CTA owns.
__host__ __device__ inline TcLayout tc_layout(int N, int CK) {
    TcLayout L;
    L.stage_bytes = kATileBytes + N * kTileK * 2;
    const uint32_t ring = kStagesTC * L.stage_bytes;
    L.dump_stride = N + 4;
    const uint32_t dump = kTileM * L.dump_stride * 4;
    L.recv = dump;
    const uint32_t after = CK > 1 ? 2 * dump : dump;  // CK * RS = 128 rows received
    L.region = ring > after ? ring : after;
    L.bars = L.region;
    L.colbest = L.bars + 8 * (2 * kStagesTC + 3);
    L.misc = L.colbest + 8 * 8 * N;
    L.total = L.misc + 16 + 1024;  // + slack to align the dynamic base to 1024
    return L;
}

__device__ __forceinline__ float2 lds_f32x2(uint32_t addr) {
    float2 x;
    asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(x.x), "=f"(x.y) : "r"(addr));
    return x;
}

// Bulk copy shared::cta -> shared::cluster (another CTA of the cluster),
// completing on an mbarrier of the destination CTA.
__device__ __forceinline__ void bulk_copy_to_peer(uint32_t dst_cluster, uint32_t src, uint32_t bytes,
                                                  uint32_t bar_cluster) {
    asm volatile(
        "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            dst_cluster),
        "r"(src), "r"(bytes), "r"(bar_cluster)
        : "memory");
}

// Asynchronous remote store of 8 bytes, completing on the destination CTA's mbarrier.
__device__ __forceinline__ void st_async_u64(uint32_t dst_cluster, unsigned long long v, uint32_t bar_cluster) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b64 [%0], %1, [%2];" ::"r"(dst_cluster),
                 "l"(v), "r"(bar_cluster)
                 : "memory");
}

// kFeatures: the build for the modes that write bf16 features (the audio
// head's first layer, projections); the other builds select tokens.  kWide:
// the argmax build for wide batches (N >= 128), whose scan of each column
// runs long enough to pay for its larger code; the narrow build's epilogue
// runs once per CTA, where every instruction line is fetched cold.  Kept
// apart so each epilogue is compiled without the others' code.
template <bool kFeatures, bool kWide, int kThreads>
__global__ void __launch_bounds__(kThreads, kThreads > kThreadsTC ? 1 : 2)
head_tc_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_h,
               const HeadArgs a, int N, int CK, int alloc_cols) {
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment for the 128-byte swizzle atoms.
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (base - raw);
    const TcLayout Lo = tc_layout(N, CK);
    const uint32_t bar_full = base + Lo.bars;                 // [kStagesTC]
    const uint32_t bar_empty = bar_full + 8 * kStagesTC;      // [kStagesTC]
    const uint32_t bar_acc = bar_empty + 8 * kStagesTC;
    const uint32_t bar_recv = bar_acc + 8;                    // peers' rows have arrived
    const uint32_t bar_fold = bar_recv + 8;                   // peers' column keys have arrived (rank 0)
    unsigned long long *colbest = reinterpret_cast<unsigned long long *>(smem + Lo.colbest);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + Lo.misc);
    int *flag = reinterpret_cast<int *>(smem + Lo.misc + 4);
    int *failed = reinterpret_cast<int *>(smem + Lo.misc + 8);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rank = CK > 1 ? static_cast<int>(cluster_ctarank()) : 0;
    const int vtile = blockIdx.x / CK;
    const int rchunk = blockIdx.y;
    const int v0 = vtile * kTileM;
    const int r0 = rchunk * N;
    const int ktiles = a.H / kTileK / CK;     // k-slices of this CTA
    const int kbase = rank * ktiles * kTileK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStagesTC; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, 1);
        }
        mbar_init(bar_acc, 1);
        mbar_init(bar_recv, 1);
        mbar_init(bar_fold, 1);
        fence_mbar_init();
        *failed = 0;
    }
    pdl_allow_dependents();
    if (warp == 4 && lane == 0) {
        prefetch_tensormap(&map_w);
        prefetch_tensormap(&map_h);
    }
    for (int i = threadIdx.x; i < N; i += blockDim.x) colbest[i] = 0ull;
    __syncthreads();
    // The first stages need no slot to free up: start streaming W and h now,
    // while the TMEM accumulator is being allocated.
    // The weights never depend on the previous kernel, so they are requested
    // before waiting for it; h (its output) only after.
    const int prologue = ktiles < kStagesTC ? ktiles : kStagesTC;
    if (warp == 4 && lane == 0) {
        for (int it = 0; it < prologue; ++it) {
            const uint32_t sa = base + it * Lo.stage_bytes;
            mbar_arrive_expect_tx(bar_full + 8 * it, Lo.stage_bytes);
            tma_load_2d(sa, &map_w, kbase + it * kTileK, v0, bar_full + 8 * it);
        }
        pdl_wait_prerequisites();
        for (int it = 0; it < prologue; ++it)
            tma_load_2d(base + it * Lo.stage_bytes + kATileBytes, &map_h, kbase + it * kTileK, r0,
                        bar_full + 8 * it);
    }
    if (warp == 5) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_addr(tmem_slot)),
                     "r"(alloc_cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 4 && lane == 0) {
        // ---- TMA producer (the first `prologue` stages are already in flight)
        for (int it = prologue; it < ktiles; ++it) {
            const int s = it % kStagesTC;
            if (it >= kStagesTC && !mbar_wait(bar_empty + 8 * s, ((it / kStagesTC) - 1) & 1)) {
                flag_error(a.err, TTS_ERRBIT_TIMEOUT);
                atomicExch(failed, 1);
                break;
            }
            const uint32_t sa = base + s * Lo.stage_bytes;
            mbar_arrive_expect_tx(bar_full + 8 * s, Lo.stage_bytes);
            const int k = kbase + it * kTileK;
            tma_load_2d(sa, &map_w, k, v0, bar_full + 8 * s);
            tma_load_2d(sa + kATileBytes, &map_h, k, r0, bar_full + 8 * s);
        }
    } else if (warp == 5 && lane == 0) {
        // ---- MMA issuer: D[128 x N] += W_tile[128 x 64] . h_tile[N x 64]^T per stage
        const uint32_t idesc = mma_idesc(kTileM, N);
        int it = 0;
        for (; it < ktiles; ++it) {
            const int s = it % kStagesTC;
            if (!mbar_wait(bar_full + 8 * s, (it / kStagesTC) & 1)) {
                flag_error(a.err, TTS_ERRBIT_TIMEOUT);
                atomicExch(failed, 1);
                break;
            }
            tc_fence_after();
            const uint32_t sa = base + s * Lo.stage_bytes;
#pragma unroll
            for (int kk = 0; kk < kTileK / 16; ++kk)
                mma_bf16(tmem, sw128_desc(sa + kk * 32), sw128_desc(sa + kATileBytes + kk * 32), idesc,
                         (it | kk) != 0);
            mma_commit(bar_empty + 8 * s);
        }
        mma_commit(bar_acc);  // fires when every MMA issued above has completed
    }

    // ---- epilogue part 1: the accumulator goes to shared memory (the dump,
    // reusing the ring, so every MMA of this CTA must be done), then each
    // cluster CTA's block of rows (RS rows starting at rank * RS) is moved to
    // it by one bulk copy per warp and owner, completing on the owner's
    // mbarrier; the cluster barrier first makes sure every CTA's ring is free.
    const int RS = kTileM / CK;  // rows owned per CTA
    float *dump = reinterpret_cast<float *>(smem);
    const uint32_t stride_b = Lo.dump_stride * 4;
    bool acc_ready = true;
    if (threadIdx.x == 0 && CK > 1)
        mbar_arrive_expect_tx(bar_recv, static_cast<uint32_t>(CK - 1) * RS * stride_b);
    if (threadIdx.x == 0 && CK > 1 && rank == 0)
        mbar_arrive_expect_tx(bar_fold, static_cast<uint32_t>(CK - 1) * N * 8);
    if (warp < 4 && !mbar_wait(bar_acc, 0)) {
        flag_error(a.err, TTS_ERRBIT_TIMEOUT);
        atomicExch(failed, 1);
        acc_ready = false;
    }
    if (warp < 4 && acc_ready) {
        tc_fence_after();
        const int row = warp * 32 + lane;
        float *dst_row = dump + static_cast<size_t>(row) * Lo.dump_stride;
        for (int c0 = 0; c0 < N; c0 += 32) {
            float v[32];
            const uint32_t t = tmem + (static_cast<uint32_t>(warp * 32) << 16) + c0;
            tmem_ld16(t, v);
            if (c0 + 16 < N) tmem_ld16(t + 16, v + 16);
            float4 *dst = reinterpret_cast<float4 *>(dst_row + c0);
#pragma unroll
            for (int q = 0; q < 8; ++q)
                if (c0 + 4 * q < N) dst[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        }
        // the bulk copies read the dump through the async proxy
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    tc_fence_before();
    if (CK > 1) cluster_sync();  // every CTA's MMAs are done: rings are free to receive
    else __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(alloc_cols)
                     : "memory");
    }
    if (CK > 1 && warp < 4 && lane == 0 && acc_ready) {
        // this warp's 32 rows, split at owner boundaries; own rows stay in the dump
        for (int row = warp * 32; row < warp * 32 + 32;) {
            const int owner = row / RS;
            const int end = min(warp * 32 + 32, (owner + 1) * RS);
            if (owner != rank) {
                const uint32_t dst = base + Lo.recv + (static_cast<uint32_t>(rank) * RS + row % RS) * stride_b;
                bulk_copy_to_peer(map_cluster(dst, owner), base + row * stride_b, (end - row) * stride_b,
                                  map_cluster(bar_recv, owner));
            }
            row = end;
        }
    }
    if (CK > 1 && !mbar_wait(bar_recv, 0)) {
        flag_error(a.err, TTS_ERRBIT_TIMEOUT);
        atomicExch(failed, 1);
    }
    // Every row sent to this CTA has landed, so every copy reading this CTA's
    // dump that targets it is done; the matching wait before exit keeps each
    // CTA's shared memory alive until all copies of the cluster have landed.
    if (CK > 1) asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");

    // ---- epilogue part 2: sum the CK partial copies of this CTA's RS rows and
    // select per batch column.  Work item = (8-row group, column); consecutive
    // threads take consecutive columns.  Source `rank` is this CTA's own dump.
    const float *recv = reinterpret_cast<const float *>(smem + Lo.recv);
    const int items = (RS / 8) * N;
    // Item `item` -> its column, batch row, first vocabulary entry, the end of
    // the entries it may select, and its 8 summed logits (written out too if
    // asked).  False if the item selects nothing.
    auto load_item = [&](int item, int &cn, int &r, int &v, uint32_t &allow, float *lg) -> bool {
        const int gi = item / N;
        cn = item - gi * N;
        r = r0 + cn;
        if (r >= a.R) return false;
#pragma unroll
        for (int e = 0; e < 8; ++e) lg[e] = 0.0f;
        for (int src = 0; src < CK; ++src) {
            const float *col = src == rank
                                   ? dump + (static_cast<size_t>(rank) * RS + gi * 8) * Lo.dump_stride + cn
                                   : recv + (static_cast<size_t>(src) * RS + gi * 8) * Lo.dump_stride + cn;
#pragma unroll
            for (int e = 0; e < 8; ++e) lg[e] += col[e * Lo.dump_stride];
        }
        v = v0 + rank * RS + gi * 8;  // multiple of 8
        if (a.bias) {
#pragma unroll
            for (int e = 0; e < 8; ++e)
                if (v + e < a.V) lg[e] += a.bias[v + e];
        }
        if (a.logits_out) {
#pragma unroll
            for (int e = 0; e < 8; ++e)
                if (v + e < a.V) a.logits_out[static_cast<size_t>(r) * a.V + v + e] = lg[e];
        }
        // ids this row may choose: below the structural tail, or a tail id
        // whose mask bit is set (the boundary token alone with eos_allowed)
        int tail0 = a.V;
        uint32_t tm = 0u;
        if (a.tail) {
            tail0 = a.V - a.n_tail;
            tm = a.tail[r];
        } else if (a.eos && !a.eos[r]) {
            tail0 = a.V - 1;
        }
        if (v + 8 <= tail0) {  // every entry below the structural tail (nearly all items)
            allow = 0xFFu;
            return true;
        }
        allow = 0u;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int id = v + e;
            const bool ok = id < a.V && (id < tail0 || ((tm >> (id - tail0)) & 1u));
            allow |= ok ? 1u << e : 0u;
        }
        return allow != 0u;
    };
    if constexpr (kFeatures) {
        // 8 features of one row per item, one 16-byte store of bf16 values:
        // Mish(x + b) for the audio head's first layer, x for a projection
        const bool mish = a.mode == kModeExpand;
        for (int item = threadIdx.x; item < items; item += blockDim.x) {
            int cn, r, v;
            uint32_t allow;
            float lg[8];
            if (!load_item(item, cn, r, v, allow, lg)) continue;
            uint32_t w[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float x0 = mish ? mish_f(lg[2 * q]) : lg[2 * q];
                const float x1 = mish ? mish_f(lg[2 * q + 1]) : lg[2 * q + 1];
                const __nv_bfloat162 p = __floats2bfloat162_rn(x0, x1);
                w[q] = *reinterpret_cast<const uint32_t *>(&p);
            }
            __nv_bfloat16 *dst;
            if (mish) {
                dst = a.z_out + static_cast<size_t>(r) * a.V + v;
            } else {
                const int j = v < a.seg_start[1] ? 0 : (v < a.seg_start[2] ? 1 : 2);
                const int width = a.seg_start[j + 1] - a.seg_start[j];
                dst = a.seg_out[j] + static_cast<size_t>(r) * width + (v - a.seg_start[j]);
            }
            *reinterpret_cast<uint4 *>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
        }
        if (CK > 1) asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
        return;
    }
    if constexpr (kWide) {
        // Argmax over wide batches: a thread takes 2 adjacent columns (one
        // 8-byte read per vocabulary row) and every PQ-th 8-row group of them,
        // so it runs 2 independent chains.  Logits become 32-bit order keys
        // (larger logit, larger key; 0 = not selectable) reduced by a max tree
        // per group and column; the index is looked up only when a group raises
        // its column's best, and a strict raise keeps the lowest index among
        // equal keys, as the packed key does.  The arguments used per group
        // are read once (a read through the kernel argument in the loop costs
        // a dependent load per group).
        const int aR = a.R, aV = a.V;
        const float *const a_bias = a.bias;
        float *const a_logits = a.logits_out;
        const int groups = RS / 8;
        const int NQ = N / 2;
        const int PQ = max(1, min(groups, static_cast<int>(blockDim.x) / NQ));
        if (static_cast<int>(threadIdx.x) < NQ * PQ) {
            const int q = static_cast<int>(threadIdx.x) % NQ;
            const int part = static_cast<int>(threadIdx.x) / NQ;
            int tail0[2];
            uint32_t tm[2];
            bool live[2];
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const int r = r0 + 2 * q + c;
                live[c] = r < aR;
                // ids this row may choose: below tail0, or a tail id whose bit is set
                tail0[c] = aV;
                tm[c] = 0u;
                if (live[c] && a.tail) {
                    tail0[c] = aV - a.n_tail;
                    tm[c] = a.tail[r];
                } else if (live[c] && a.eos && !a.eos[r]) {
                    tail0[c] = aV - 1;
                }
            }
            uint32_t bk[2] = {0u, 0u};
            int bi[2] = {0, 0};
            for (int gi = part; gi < groups; gi += PQ) {
                const int v = v0 + rank * RS + gi * 8;
                float x[8][2];
#pragma unroll
                for (int e = 0; e < 8; ++e) x[e][0] = x[e][1] = 0.0f;
                for (int src = 0; src < CK; ++src) {
                    const uint32_t row0 = (src == rank ? base : base + Lo.recv) +
                                          static_cast<uint32_t>(src * RS + gi * 8) * stride_b + 8u * q;
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float2 w = lds_f32x2(row0 + e * stride_b);
                        x[e][0] += w.x;
                        x[e][1] += w.y;
                    }
                }
                if (a_bias) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float b = v + e < aV ? a_bias[v + e] : 0.0f;
                        x[e][0] += b;
                        x[e][1] += b;
                    }
                }
                if (a_logits) {
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        if (!live[c]) continue;
                        float *dst = a_logits + static_cast<size_t>(r0 + 2 * q + c) * aV;
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            if (v + e < aV) dst[v + e] = x[e][c];
                    }
                }
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    uint32_t k[8];
                    if (v + 8 <= tail0[c]) {
#pragma unroll
                        for (int e = 0; e < 8; ++e) k[e] = float_order_key(x[e][c]);
                    } else {
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const int id = v + e;
                            const bool ok = id < aV && (id < tail0[c] || ((tm[c] >> (id - tail0[c])) & 1u));
                            k[e] = ok ? float_order_key(x[e][c]) : 0u;
                        }
                    }
                    const uint32_t gk = max(max(max(k[0], k[1]), max(k[2], k[3])),
                                            max(max(k[4], k[5]), max(k[6], k[7])));
                    if (gk > bk[c]) {
                        int ef = 7;
#pragma unroll
                        for (int e = 6; e >= 0; --e)
                            if (k[e] == gk) ef = e;
                        bk[c] = gk;
                        bi[c] = v + ef;
                    }
                }
            }
#pragma unroll
            for (int c = 0; c < 2; ++c)
                if (live[c] && bk[c])
                    atomicMax(colbest + 2 * q + c, (static_cast<unsigned long long>(bk[c]) << 32) |
                                                       static_cast<unsigned long long>(~static_cast<uint32_t>(bi[c])));
        }
    } else if (a.mode == TTS_GUMBEL) {
        // An entry can only beat the column's current best z_cur if its noise
        // exceeds z_cur - logit / T.  With the group's largest logit that gives
        // one uniform threshold for all 8 entries: below it (with a safety
        // margin far above rounding) an entry cannot win, and its logarithms
        // are skipped.  Exact for the entries kept.  Two items per pass, so
        // each thread runs two independent Philox chains.
        auto select = [&](bool live, int cn, int v, uint32_t allow, const float *lg, const Philox4x64 &ph) {
            if (!live) return;
            float lmax = -INFINITY;
#pragma unroll
            for (int e = 0; e < 8; ++e)
                if ((allow >> e) & 1u) lmax = fmaxf(lmax, lg[e]);
            const unsigned long long cur = *reinterpret_cast<volatile unsigned long long *>(colbest + cn);
            float thr = 0.0f;  // uniforms <= thr cannot win
            if (cur) {
                const float g0 = unpack_value(cur) - lmax / a.temperature - kGumbelSlack;
                thr = expf(-expf(-g0));
            }
            unsigned long long best = 0ull;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                if (!((allow >> e) & 1u)) continue;
                const float u = bits_to_uniform(ph.half(e));
                if (!(u > thr)) continue;
                const float key = lg[e] / a.temperature + gumbel_from_uniform(u);
                const unsigned long long k = pack_argmax(key, v + e);
                best = k > best ? k : best;
            }
            if (best) atomicMax(colbest + cn, best);
        };
        for (int i0 = threadIdx.x; i0 < items; i0 += 2 * blockDim.x) {
            const int i1 = i0 + blockDim.x;
            int cn0, r0i, va, cn1 = 0, r1i = 0, vb = 0;
            uint32_t allow0, allow1 = 0u;
            float lg0[8], lg1[8];
            const bool live0 = load_item(i0, cn0, r0i, va, allow0, lg0);
            const bool live1 = i1 < items && load_item(i1, cn1, r1i, vb, allow1, lg1);
            const int ra = live0 ? r0i : r0, rb = live1 ? r1i : r0;
            const Philox4x64 pa(static_cast<uint64_t>(va >> 3), 0, a.pos, 0, a.seed[ra], a.step[ra]);
            const Philox4x64 pb(static_cast<uint64_t>(vb >> 3), 0, a.pos, 0, a.seed[rb], a.step[rb]);
            select(live0, cn0, va, allow0, lg0, pa);
            select(live1, cn1, vb, allow1, lg1, pb);
        }
    } else {
        for (int item = threadIdx.x; item < items; item += blockDim.x) {
            int cn, r, v;
            uint32_t allow;
            float lg[8];
            if (!load_item(item, cn, r, v, allow, lg)) continue;
            unsigned long long best = 0ull;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                if (!((allow >> e) & 1u)) continue;
                const unsigned long long k = pack_argmax(lg[e], v + e);
                best = k > best ? k : best;
            }
            if (best) atomicMax(colbest + cn, best);
        }
    }
    __syncthreads();
    // One global atomic per column and cluster: every other rank sends its
    // column maxima into its own slot of rank 0's table (asynchronous remote
    // stores completing on rank 0's mbarrier), and rank 0 folds them.
    if (CK > 1 && rank != 0) {
        const uint32_t slot = map_cluster(base + Lo.colbest + static_cast<uint32_t>(rank) * N * 8, 0u);
        const uint32_t fold = map_cluster(bar_fold, 0u);
        for (int cn = threadIdx.x; cn < N; cn += blockDim.x) st_async_u64(slot + cn * 8, colbest[cn], fold);
    }
    if (CK > 1) asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
    // Only rank 0 of each cluster publishes keys, so only those CTAs take a
    // ticket: the last ticket then comes after every publication.
    if (rank != 0) return;
    if (CK > 1 && !mbar_wait(bar_fold, 0)) {
        flag_error(a.err, TTS_ERRBIT_TIMEOUT);
        atomicExch(failed, 1);
    }
    for (int cn = threadIdx.x; cn < N; cn += blockDim.x) {
        unsigned long long k = colbest[cn];
        for (int src = 1; src < CK; ++src) {
            const unsigned long long o = colbest[src * N + cn];
            k = o > k ? o : k;
        }
        if (r0 + cn < a.R && k) atomicMax(a.ws.keys + r0 + cn, k);
    }
    finish_selection(a.ws, a.R, a.ids, a.best, flag, (gridDim.x / CK) * gridDim.y, a.ids_host, a.count_host,
                     a.V - 1, a.seq_host, a.seq_dev);
}

// ------------------------------------------- split build (narrow batches)
//
// For batches of up to 64 rows.  A cluster of CK CTAs owns one 128-row vocab
// tile; CTA rank r reduces the hidden range [r H / CK, (r + 1) H / CK).  Every
// W and h k-slice of the CTA is requested at once (no ring reuse: at 64 x
// 2048 x 4097 the CTA's 128 KB of W and 64 KB of h are all in flight), so the
// load time is the HBM burst itself.  The epilogue runs once per CTA with its
// instructions fetched cold, so it is short and has one wait: each warp reads
// its 32 accumulator rows (one vocab row per lane) from TMEM, stages them in
// the idle slice area and sends each owning CTA its rows with one bulk copy
// completing on that CTA's mbarrier; each CTA waits for its own 32 rows from
// all CK sources, sums them, selects per batch row and folds its best keys
// into the global keys; the last CTA converts keys to ids.
constexpr int kSplitThreads = 256;
constexpr int kSplitMaxN = 64;

struct SplitLayout {
    uint32_t hslot;    // bytes of one h k-slice (N rows x 128 B)
    uint32_t h;        // offset of the h slices (after the W slices)
    uint32_t recv;     // offset of recv[CK][RS][NR] fp32 partials (after the slices, or the staging rows if larger)
    uint32_t bars;     // kch full barriers, the accumulator barrier, the receive barrier
    uint32_t colbest;  // [N] packed keys
    uint32_t misc;     // TMEM address, flag
    uint32_t total;
};

// Floats per partial row in recv: N rounded up to a power of two, so the
// chunk swizzle below is a mask.
__host__ __device__ constexpr int split_row(int N) { return N <= 16 ? 16 : (N <= 32 ? 32 : 64); }

__host__ __device__ inline SplitLayout split_layout(int N, int kch, int CK, int RS) {
    SplitLayout L;
    L.hslot = static_cast<uint32_t>(N) * 128u;
    L.h = static_cast<uint32_t>(kch) * kATileBytes;
    // after the MMAs the W and h slices hold the staged accumulator rows
    // (128 rows of NR floats): at least that much room before recv
    const uint32_t slices = L.h + static_cast<uint32_t>(kch) * L.hslot;
    const uint32_t staging = static_cast<uint32_t>(kTileM * split_row(N)) * 4u;
    L.recv = slices > staging ? slices : staging;
    L.bars = L.recv + static_cast<uint32_t>(CK * RS * split_row(N)) * 4u;
    L.colbest = L.bars + 8u * (kch + 2);
    L.misc = L.colbest + 8u * N;
    L.total = L.misc + 16u + 1024u;  // + slack to align the dynamic base to 1024
    return L;
}

constexpr int kSplitMaxCK = 8;  // widest cluster split of the split build

// Position of float n within partial row i of recv (rows of NR floats, NR a
// power of two): the row's 16-byte chunks are permuted by i ^ 2 (i / 8), a
// bijection per row.  Lanes storing the same chunk of 8 consecutive rows
// land in distinct bank groups, and a warp reading 8-row groups g of
// columns n (lane = g + G n) spreads over the banks too, the 2 (i / 8) term
// separating the groups that the low bits of i alone would put on one bank.
template <int NR>
__device__ __forceinline__ int split_pos(int i, int n) {
    return ((((n >> 2) ^ i ^ ((i >> 3) << 1)) & ((NR >> 2) - 1)) << 2) | (n & 3);
}

template <bool kGumbel, int N>
__global__ void __launch_bounds__(kSplitThreads, 1)
head_split_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_h,
                  const HeadArgs a, int CK, int RS, int alloc_cols) {
    constexpr int NR = split_row(N);
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (base - raw);
    const int kch = a.H / kTileK / CK;
    const SplitLayout Lo = split_layout(N, kch, CK, RS);
    const uint32_t bar_full = base + Lo.bars;        // [kch]
    const uint32_t bar_acc = bar_full + 8u * kch;
    const uint32_t bar_recv = bar_acc + 8u;
    unsigned long long *colbest = reinterpret_cast<unsigned long long *>(smem + Lo.colbest);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + Lo.misc);
    int *flag = reinterpret_cast<int *>(smem + Lo.misc + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rank = static_cast<int>(cluster_ctarank());
    const int v0 = (blockIdx.x / CK) * kTileM;  // first vocab row of the cluster's tile
    const int kbase = rank * kch * kTileK;

    if (threadIdx.x == 0) {
        for (int c = 0; c < kch + 2; ++c) mbar_init(bar_full + 8u * c, 1);
        fence_mbar_init();
        // every source's rows of this CTA: CK x RS rows of NR floats
        mbar_arrive_expect_tx(bar_recv, static_cast<uint32_t>(CK * RS * NR) * 4u);
        // Every W slice at once (W never depends on the previous kernel); h,
        // the previous kernel's output, after the programmatic-launch wait.
        prefetch_tensormap(&map_w);
        for (int c = 0; c < kch; ++c) {
            mbar_arrive_expect_tx(bar_full + 8u * c, kATileBytes + Lo.hslot);
            tma_load_2d(base + c * kATileBytes, &map_w, kbase + c * kTileK, v0, bar_full + 8u * c);
        }
    }
    // Peers store into this CTA's shared memory only after the matching wait
    // below, i.e. after this CTA's barriers are initialised.
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
    pdl_allow_dependents();
    for (int i = threadIdx.x; i < N; i += blockDim.x) colbest[i] = 0ull;
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&map_h);
        pdl_wait_prerequisites();
        for (int c = 0; c < kch; ++c)
            tma_load_2d(base + Lo.h + c * Lo.hslot, &map_h, kbase + c * kTileK, 0, bar_full + 8u * c);
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_addr(tmem_slot)),
                     "r"(alloc_cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
    const uint32_t tmem = *tmem_slot;

    if (warp == 1 && lane == 0) {
        // D[128 x N] += W_slice[128 x 64] . h_slice[N x 64]^T per slice, in arrival order
        constexpr uint32_t idesc = mma_idesc(kTileM, N);
        bool ok = true;
        for (int c = 0; c < kch; ++c) {
            if (ok && !mbar_wait(bar_full + 8u * c, 0)) {
                flag_error(a.err, TTS_ERRBIT_TIMEOUT);
                ok = false;
            }
            if (!ok) continue;  // no MMA on a slice that never arrived
            tc_fence_after();
            const uint32_t wa = base + c * kATileBytes, ha = base + Lo.h + c * Lo.hslot;
#pragma unroll
            for (int kk = 0; kk < kTileK / 16; ++kk)
                mma_bf16(tmem, sw128_desc(wa + kk * 32), sw128_desc(ha + kk * 32), idesc, (c | kk) != 0);
        }
        mma_commit(bar_acc);  // fires once every MMA issued above has completed
    }
    __syncwarp();

    // ---- accumulator rows -> their owners.  Warp w holds the tile's rows
    // 32 w .. 32 w + 31 (one per lane, all N columns); it stages them in the
    // now idle slice area in the owner's layout and sends each owner's run of
    // rows with one bulk copy onto the owner's receive barrier (with CK = 4
    // a warp's rows all belong to one owner).
    if (warp < 4) {
        const int vl = warp * 32 + lane;
        const int owner = vl / RS;  // < CK: RS = 128 / CK
        const int i = vl - owner * RS;
        const bool ready = mbar_wait(bar_acc, 0);
        if (!ready) flag_error(a.err, TTS_ERRBIT_TIMEOUT);
        tc_fence_after();
        if (__all_sync(kFull, ready)) {
            uint32_t r[N];
#pragma unroll
            for (int c0 = 0; c0 < N; c0 += 16)
                tmem_ld16_nowait(tmem + (static_cast<uint32_t>(warp * 32) << 16) + c0, r + c0);
            tmem_wait_ld();
            const uint32_t srow = base + static_cast<uint32_t>(vl * NR) * 4u;
#pragma unroll
            for (int q = 0; q < N / 4; ++q)
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(srow + 4u * split_pos<NR>(i, 4 * q)),
                             "r"(r[4 * q]), "r"(r[4 * q + 1]), "r"(r[4 * q + 2]), "r"(r[4 * q + 3])
                             : "memory");
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the copies read through the async proxy
            __syncwarp();
            if (lane == 0) {
                for (int row = warp * 32; row < warp * 32 + 32;) {
                    const int o = row / RS;
                    const int end = min(warp * 32 + 32, (o + 1) * RS);
                    const uint32_t dst = base + Lo.recv + static_cast<uint32_t>((rank * RS + row - o * RS) * NR) * 4u;
                    bulk_copy_to_peer(map_cluster(dst, static_cast<uint32_t>(o)),
                                      base + static_cast<uint32_t>(row * NR) * 4u,
                                      static_cast<uint32_t>((end - row) * NR) * 4u,
                                      map_cluster(bar_recv, static_cast<uint32_t>(o)));
                    row = end;
                }
                asm volatile("cp.async.bulk.commit_group;" ::: "memory");
            }
        }
    }
    tc_fence_before();

    // ---- sum the CK partials of this CTA's rows and select per batch row.
    // Item = (8-row group g, batch row n), G = RS / 8 groups; the G items of
    // one batch row sit in G consecutive lanes and meet in a shuffle max.
    // Warps 4-7 run the same loop once early without committing anything (its
    // reads land on not yet written rows), so its instructions are cached by
    // the time the rows arrive.
    const float *recv = reinterpret_cast<const float *>(smem + Lo.recv);
    const int G = RS / 8;
    const int items = G * N;
    const int aR = a.R, aV = a.V;
    bool got = true;
    for (int pass = warp >= 4 ? 0 : 1; pass < 2; ++pass) {
        const bool commit = pass == 1;
        if (commit) {
            got = mbar_wait(bar_recv, 0);
            if (!got && threadIdx.x == 0) flag_error(a.err, TTS_ERRBIT_TIMEOUT);
        }
        for (int item = threadIdx.x; item < items && got; item += blockDim.x) {
            const int g = item % G, n = item / G;
            const int r = n;
            const int v = v0 + rank * RS + 8 * g;
            const bool live = r < aR && v < aV;
            unsigned long long best = 0ull;
            if (live) {
                // every source's partials first (independent loads, one
                // latency), then the sums in source order
                float part[kSplitMaxCK][8];
#pragma unroll
                for (int sidx = 0; sidx < kSplitMaxCK; ++sidx) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int ii = 8 * g + e;
                        part[sidx][e] = sidx < CK ? recv[(static_cast<size_t>(sidx) * RS + ii) * NR + split_pos<NR>(ii, n)]
                                                  : 0.0f;
                    }
                }
                float lg[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    float x = part[0][e];
#pragma unroll
                    for (int sidx = 1; sidx < kSplitMaxCK; ++sidx)
                        if (sidx < CK) x += part[sidx][e];
                    lg[e] = x;
                }
                if (a.bias) {
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        if (v + e < aV) lg[e] += a.bias[v + e];
                }
                // ids this row may choose: below the structural tail, or a tail
                // id whose mask bit is set (the boundary token alone with eos_allowed)
                int tail0 = aV;
                uint32_t tm = 0u;
                if (a.tail) {
                    tail0 = aV - a.n_tail;
                    tm = a.tail[r];
                } else if (a.eos && !a.eos[r]) {
                    tail0 = aV - 1;
                }
                uint32_t allow = 0xFFu;
                if (v + 8 > tail0) {
                    allow = 0u;
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int id = v + e;
                        const bool ok = id < aV && (id < tail0 || ((tm >> (id - tail0)) & 1u));
                        allow |= ok ? 1u << e : 0u;
                    }
                }
                if constexpr (kGumbel) {
                    const Philox4x64 ph(static_cast<uint64_t>(v >> 3), 0, a.pos, 0, a.seed[r], a.step[r]);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        if (!((allow >> e) & 1u)) continue;
                        const float u = bits_to_uniform(ph.half(e));
                        const unsigned long long k =
                            pack_argmax(lg[e] / a.temperature + gumbel_from_uniform(u), v + e);
                        best = k > best ? k : best;
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        if (!((allow >> e) & 1u)) continue;
                        const unsigned long long k = pack_argmax(lg[e], v + e);
                        best = k > best ? k : best;
                    }
                }
            }
            for (int o = 1; o < G; o <<= 1) {
                const unsigned long long other = __shfl_xor_sync(kFull, best, o);
                best = other > best ? other : best;
            }
            if (commit && g == 0) colbest[n] = best;
        }
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(alloc_cols)
                     : "memory");
    }
    if (static_cast<int>(threadIdx.x) < N) {
        const unsigned long long k = colbest[threadIdx.x];
        if (static_cast<int>(threadIdx.x) < aR && k) atomicMax(a.ws.keys + threadIdx.x, k);
    }
    // this CTA's outgoing copies have finished reading its staging rows
    if (warp < 4 && lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
    finish_selection(a.ws, a.R, a.ids, a.best, flag, gridDim.x, a.ids_host, a.count_host, a.V - 1, a.seq_host,
                     a.seq_dev);
}

// ------------------------------------------------------------- host side

struct TcPlan {
    int N, chunks, CK, alloc_cols;
    uint32_t smem;
};

TcPlan plan_tc(int R, int H, int V, bool gumbel) {
    TcPlan p;
    p.chunks = (R + kMaxN - 1) / kMaxN;
    const int per = (R + p.chunks - 1) / p.chunks;
    p.N = (per + 15) / 16 * 16;
    p.alloc_cols = 32;
    while (p.alloc_cols < p.N) p.alloc_cols <<= 1;
    const int sms = sm_count() > 0 ? sm_count() : 148;
    const int tmem_fit = 512 / p.alloc_cols;
    const int vtiles = (V + kTileM - 1) / kTileM;
    const int ktiles = H / kTileK;
    p.CK = 1;
    p.smem = tc_layout(p.N, 1).total;
    // widest cluster split of the hidden dimension, up to 4, that still runs
    // in one wave (8-CTA clusters start and synchronise more slowly than the
    // extra SMs they bring save: measured 1.5 us slower at 64 x 2048 x 4097);
    // up to 8 for H >= 4096, where a 4-way split leaves 256 KB of W per CTA
    // (measured 4 us faster at 64 x 4096 x 4097)
    const int ck_max = H >= 4096 ? 8 : 4;  // wide reductions: every CTA's W slice stays small
    for (int ck = 2; ck <= ck_max; ck <<= 1) {
        if (ktiles % ck != 0) break;
        const uint32_t smem = tc_layout(p.N, ck).total;
        int per_sm = static_cast<int>((227u * 1024u) / (smem + 1024u));
        per_sm = per_sm < tmem_fit ? per_sm : tmem_fit;
        // registers: the kernel is built for two CTAs per SM, one with more threads
        const int reg_fit = tc_threads(gumbel, p.N) > kThreadsTC ? 1 : 2;
        per_sm = per_sm < reg_fit ? per_sm : reg_fit;
        if (per_sm < 1 || static_cast<long>(vtiles) * p.chunks * ck > static_cast<long>(sms) * per_sm) break;
        p.CK = ck;
        p.smem = smem;
    }
    return p;
}

// The split build, if it takes this shape: batches of up to 64 rows whose
// vocab tiles all run as co-resident clusters (one wave) with every k-slice
// in shared memory at once.  Cluster widths tried in order of measured speed.
struct SplitPlan {
    int N, CK, RS, ncl, alloc_cols;
    uint32_t smem;
};

int max_active_clusters(const void *kernel, int ck, uint32_t smem) {
    struct Entry {
        const void *kernel;
        int device, ck;
        uint32_t smem;
        int n;
    };
    static std::mutex mu;
    static Entry cache[32];
    static int used = 0;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i)
        if (cache[i].kernel == kernel && cache[i].device == dev && cache[i].ck == ck && cache[i].smem == smem)
            return cache[i].n;
    if (!ensure_dynamic_smem(kernel, static_cast<int>(smem))) return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(ck), 1, 1);
    cfg.blockDim = dim3(kSplitThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute at;
    at.id = cudaLaunchAttributeClusterDimension;
    at.val.clusterDim.x = static_cast<unsigned>(ck);
    at.val.clusterDim.y = 1;
    at.val.clusterDim.z = 1;
    cfg.attrs = &at;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) {
        cudaGetLastError();
        n = 0;
    }
    if (used < 32) cache[used++] = {kernel, dev, ck, smem, n};
    return n;
}

// The instance for a padded batch width N (16, 32, 48 or 64).
const void *split_kernel(bool gumbel, int N) {
    using K = void (*)(CUtensorMap, CUtensorMap, HeadArgs, int, int, int);
    static const K table[2][4] = {
        {head_split_kernel<false, 16>, head_split_kernel<false, 32>, head_split_kernel<false, 48>,
         head_split_kernel<false, 64>},
        {head_split_kernel<true, 16>, head_split_kernel<true, 32>, head_split_kernel<true, 48>,
         head_split_kernel<true, 64>}};
    return reinterpret_cast<const void *>(table[gumbel ? 1 : 0][N / 16 - 1]);
}

bool plan_split(int R, int H, int V, bool gumbel, SplitPlan *p) {
    if (R > kSplitMaxN || H % kTileK != 0) return false;
    p->N = (R + 15) / 16 * 16;
    p->alloc_cols = 32;
    while (p->alloc_cols < p->N) p->alloc_cols <<= 1;
    p->ncl = (V + kTileM - 1) / kTileM;
    const void *kernel = split_kernel(gumbel, p->N);
    for (int ck : {4, 8, 2}) {  // each at most kSplitMaxCK
        if (H % (kTileK * ck) != 0) continue;
        const int kch = H / kTileK / ck;
        const int RS = kTileM / ck;
        const uint32_t smem = split_layout(p->N, kch, ck, RS).total;
        if (smem > 227u * 1024u) continue;
        if (p->ncl > max_active_clusters(kernel, ck, smem)) continue;
        p->CK = ck;
        p->RS = RS;
        p->smem = smem;
        return true;
    }
    return false;
}

}  // namespace
}  // namespace tts

extern "C" size_t tts_head_workspace_size(int32_t R, int32_t V) {
    if (R < 1 || R > 4096 || V < 1) return 0;
    return tts::align_up(static_cast<size_t>(R) * 8, 256) + 256;
}

namespace tts {

struct HeadLaunchState {
    HeadArgs a;
    CUtensorMap mw, mh;
    TcPlan p;
    SplitPlan sp;
    bool split;  // the split build (narrow batches) instead of head_tc_kernel
    int dtype;
    int simt_grid;
    const void *h, *W;
};
static_assert(sizeof(HeadLaunchState) <= sizeof(HeadLaunch::storage), "HeadLaunch storage too small");

int prepare_head(const void *d_h, const void *d_W, int32_t dtype, int32_t R, int32_t H, int32_t V,
                 int32_t mode, float temperature, const uint64_t *d_seed, const uint64_t *d_step,
                 const uint8_t *d_eos_allowed, int32_t *d_ids, float *d_best, float *d_logits_out,
                 void *d_ws, size_t ws_bytes, HeadLaunch *out) {
    return prepare_head_ex(d_h, d_W, dtype, R, H, V, mode, temperature, d_seed, d_step, d_eos_allowed, d_ids, d_best,
                           d_logits_out, d_ws, ws_bytes, HeadExtras{}, out);
}

int prepare_head_ex(const void *d_h, const void *d_W, int32_t dtype, int32_t R, int32_t H, int32_t V,
                    int32_t mode, float temperature, const uint64_t *d_seed, const uint64_t *d_step,
                    const uint8_t *d_eos_allowed, int32_t *d_ids, float *d_best, float *d_logits_out,
                    void *d_ws, size_t ws_bytes, const HeadExtras &x, HeadLaunch *out) {
    const bool linear = mode == kModeLinear;
    const bool expand = mode == kModeExpand || linear;  // both write bf16 features instead of selecting
    if (!d_h || !d_W || (!expand && !d_ids)) return TTS_ERR_INVALID;
    if (R < 1 || R > 4096 || H < 1 || V < 1 || V > (1 << 30)) return TTS_ERR_INVALID;
    if (mode != TTS_ARGMAX && mode != TTS_GUMBEL && !expand) return TTS_ERR_INVALID;
    if (mode == TTS_GUMBEL && (!d_seed || !d_step || !(temperature > 0.0f) || temperature == INFINITY))
        return TTS_ERR_INVALID;
    if (x.n_tail < 0 || x.n_tail > 32 || x.n_tail > V) return TTS_ERR_INVALID;
    if (dtype != TTS_F32 && dtype != TTS_BF16) return TTS_ERR_UNSUPPORTED;
    if (dtype == TTS_F32 && (x.bias || x.tail || expand || x.pos || x.ids_host || x.count_host || x.seq_host))
        return TTS_ERR_UNSUPPORTED;
    if ((x.seq_host != nullptr) != (x.seq_dev != nullptr) || (x.seq_host && !x.ids_host)) return TTS_ERR_INVALID;
    if (linear) {
        // up to three outputs over consecutive feature ranges, 8 features per store
        if (x.seg_start[0] != 0 || x.seg_start[3] != V || V % 8 != 0) return TTS_ERR_INVALID;
        for (int j = 0; j < 3; ++j) {
            const int width = x.seg_start[j + 1] - x.seg_start[j];
            if (width < 0 || width % 8 != 0) return TTS_ERR_INVALID;
            if (width > 0 && (!x.seg_out[j] || !aligned16(x.seg_out[j]))) return TTS_ERR_INVALID;
        }
    } else if (expand) {
        // the first audio-head layer: 8 features per 16-byte store of z
        if (!x.z_out || !aligned16(x.z_out) || V % 8 != 0) return TTS_ERR_INVALID;
    } else {
        const size_t need = tts_head_workspace_size(R, V);
        if (!d_ws || ws_bytes < need || (reinterpret_cast<uintptr_t>(d_ws) & 255u) != 0)
            return TTS_ERR_WORKSPACE;
    }
    HeadLaunchState *st = new (out->storage) HeadLaunchState();
    HeadArgs &a = st->a;
    a.R = R; a.H = H; a.V = V; a.mode = mode; a.temperature = temperature;
    a.seed = d_seed; a.step = d_step; a.eos = d_eos_allowed; a.logits_out = d_logits_out;
    a.ids = d_ids; a.best = d_best; a.ws = expand ? HeadWs{nullptr, nullptr} : head_ws(d_ws, R); a.err = nullptr;
    a.bias = x.bias; a.tail = x.tail; a.n_tail = x.n_tail; a.z_out = static_cast<__nv_bfloat16 *>(x.z_out);
    a.pos = x.pos;
    a.ids_host = x.ids_host;
    a.count_host = x.count_host;
    a.seq_host = x.seq_host;
    a.seq_dev = x.seq_dev;
    for (int j = 0; j < 4; ++j) a.seg_start[j] = x.seg_start[j];
    for (int j = 0; j < 3; ++j) a.seg_out[j] = static_cast<__nv_bfloat16 *>(x.seg_out[j]);
    st->dtype = dtype;
    st->h = d_h;
    st->W = d_W;
    if (dtype == TTS_F32) {
        const int sms = sm_count() > 0 ? sm_count() : 148;
        const int grid = (V + 7) / 8;
        st->simt_grid = grid < 4 * sms ? grid : 4 * sms;
        return TTS_OK;
    }
    if (H % kTileK != 0) return TTS_ERR_UNSUPPORTED;
    if (!aligned16(d_h) || !aligned16(d_W)) return TTS_ERR_INVALID;
    st->split = !expand && !d_logits_out && plan_split(R, H, V, mode == TTS_GUMBEL, &st->sp);
    if (st->split) {
        if (!cached_tma_2d_bf16(&st->mw, d_W, static_cast<uint64_t>(V), static_cast<uint64_t>(H), kTileM, kTileK) ||
            !cached_tma_2d_bf16(&st->mh, d_h, static_cast<uint64_t>(R), static_cast<uint64_t>(H),
                                static_cast<uint32_t>(st->sp.N), kTileK))
            return TTS_ERR_CUDA;
        return TTS_OK;
    }
    st->p = plan_tc(R, H, V, mode == TTS_GUMBEL);
    if (!cached_tma_2d_bf16(&st->mw, d_W, static_cast<uint64_t>(V), static_cast<uint64_t>(H), kTileM, kTileK) ||
        !cached_tma_2d_bf16(&st->mh, d_h, static_cast<uint64_t>(R), static_cast<uint64_t>(H),
                            static_cast<uint32_t>(st->p.N), kTileK))
        return TTS_ERR_CUDA;
    return TTS_OK;
}

int launch_head(const HeadLaunch &L, LaunchOpts o) {
    const HeadLaunchState *st = reinterpret_cast<const HeadLaunchState *>(L.storage);
    cudaLaunchConfig_t cfg = {};
    cfg.stream = o.stream;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (o.pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cudaError_t e;
    if (st->dtype == TTS_F32) {
        cfg.gridDim = dim3(st->simt_grid, 1, 1);
        cfg.blockDim = dim3(256, 1, 1);
        cfg.attrs = attr;
        cfg.numAttrs = na;
        e = cudaLaunchKernelEx(&cfg, head_simt_f32_kernel, static_cast<const float *>(st->h),
                               static_cast<const float *>(st->W), st->a);
    } else if (st->split) {
        const SplitPlan &p = st->sp;
        const void *kernel = split_kernel(st->a.mode == TTS_GUMBEL, p.N);
        if (!ensure_dynamic_smem(kernel, static_cast<int>(p.smem))) return TTS_ERR_CUDA;
        cfg.gridDim = dim3(static_cast<unsigned>(p.ncl * p.CK), 1, 1);
        cfg.blockDim = dim3(kSplitThreads, 1, 1);
        cfg.dynamicSmemBytes = p.smem;
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = static_cast<unsigned>(p.CK);
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
        cfg.attrs = attr;
        cfg.numAttrs = na;
        void *args[] = {const_cast<CUtensorMap *>(&st->mw), const_cast<CUtensorMap *>(&st->mh),
                        const_cast<HeadArgs *>(&st->a), const_cast<int *>(&p.CK), const_cast<int *>(&p.RS),
                        const_cast<int *>(&p.alloc_cols)};
        e = cudaLaunchKernelExC(&cfg, kernel, args);
    } else {
        const TcPlan &p = st->p;
        const bool features = st->a.mode == kModeExpand || st->a.mode == kModeLinear;
        const bool wide = !features && st->a.mode == TTS_ARGMAX && p.N >= 128;
        const int threads = tc_threads(!features && st->a.mode == TTS_GUMBEL, p.N);
        const auto kernel = features                          ? head_tc_kernel<true, false, kThreadsTC>
                            : wide                            ? head_tc_kernel<false, true, kThreadsTC>
                            : threads == kThreadsGumbelWide   ? head_tc_kernel<false, false, kThreadsGumbelWide>
                            : threads == kThreadsGumbel       ? head_tc_kernel<false, false, kThreadsGumbel>
                                                              : head_tc_kernel<false, false, kThreadsTC>;
        if (!ensure_dynamic_smem(reinterpret_cast<const void *>(kernel), static_cast<int>(p.smem)))
            return TTS_ERR_CUDA;
        cfg.gridDim = dim3(static_cast<unsigned>(((st->a.V + kTileM - 1) / kTileM) * p.CK),
                           static_cast<unsigned>(p.chunks), 1);
        cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
        cfg.dynamicSmemBytes = p.smem;
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = static_cast<unsigned>(p.CK);
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
        cfg.attrs = attr;
        cfg.numAttrs = na;
        e = cudaLaunchKernelEx(&cfg, kernel, st->mw, st->mh, st->a, p.N, p.CK, p.alloc_cols);
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        return TTS_ERR_CUDA;
    }
    return TTS_OK;
}

}  // namespace tts

extern "C" int tts_codebook_head_select(const void *d_h, const void *d_W, int32_t dtype, int32_t R,
                                        int32_t H, int32_t V, int32_t mode, float temperature,
                                        const uint64_t *d_seed, const uint64_t *d_step,
                                        const uint8_t *d_eos_allowed, int32_t *d_ids, float *d_best,
                                        float *d_logits_out, void *d_ws, size_t ws_bytes,
                                        void *stream) {
    tts::HeadLaunch L;
    const int st = tts::prepare_head(d_h, d_W, dtype, R, H, V, mode, temperature, d_seed, d_step,
                                     d_eos_allowed, d_ids, d_best, d_logits_out, d_ws, ws_bytes, &L);
    if (st != TTS_OK) return st;
    return tts::launch_head(L, {static_cast<cudaStream_t>(stream), tts::thread_pdl()});
}

// The two-layer audio head ("TontaubeV1", section 3): z = Mish(h W1^T + b1)
// as bf16, then the codebook head over z W2^T + b2 with the stage's
// structural tail masked per row.  Two launches of the tcgen05 head; the
// second is a programmatic dependent of the first (its W2 stream starts while
// the first finishes; it reads z only after waiting).
extern "C" int tts_audio_head_select(const void *d_h, const void *d_W1, const float *d_b1, const void *d_W2,
                                     const float *d_b2, int32_t R, int32_t H, int32_t F, int32_t V, int32_t n_tail,
                                     const uint32_t *d_tail_allowed, int32_t mode, float temperature,
                                     const uint64_t *d_seed, const uint64_t *d_step, void *d_z, int32_t *d_ids,
                                     float *d_best, float *d_logits_out, void *d_ws, size_t ws_bytes,
                                     void *stream) {
    using namespace tts;
    if (mode != TTS_ARGMAX && mode != TTS_GUMBEL) return TTS_ERR_INVALID;
    if (F < 8 || F % kTileK != 0) return TTS_ERR_UNSUPPORTED;  // F is the second layer's reduction
    HeadExtras x1;
    x1.bias = d_b1;
    x1.z_out = d_z;
    HeadLaunch L1, L2;
    int st = prepare_head_ex(d_h, d_W1, TTS_BF16, R, H, F, kModeExpand, 0.0f, nullptr, nullptr, nullptr, nullptr,
                             nullptr, nullptr, nullptr, 0, x1, &L1);
    if (st != TTS_OK) return st;
    HeadExtras x2;
    x2.bias = d_b2;
    x2.tail = n_tail > 0 ? d_tail_allowed : nullptr;
    x2.n_tail = n_tail;
    st = prepare_head_ex(d_z, d_W2, TTS_BF16, R, F, V, mode, temperature, d_seed, d_step, nullptr, d_ids, d_best,
                         d_logits_out, d_ws, ws_bytes, x2, &L2);
    if (st != TTS_OK) return st;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    st = launch_head(L1, {s, false});
    if (st != TTS_OK) return st;
    return launch_head(L2, {s, true});
}
