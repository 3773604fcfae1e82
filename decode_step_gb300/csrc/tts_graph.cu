// A decode step captured as one CUDA graph for fixed shapes and addresses
// ("How We Made a TTS Model Respond in Sub-50 ms", section "Additional
// serving optimizations": graphs are captured for a predefined set of batch
// sizes; "Optimizing Streaming Text-to-Speech Models for Sub-50 Millisecond
// Latency", section "Engine-Level Optimizations with TensorRT-LLM": the CPU
// only starts the graph).
//
// One launch: a copy kernel brings the step's packed inputs from pinned host
// memory (read through unified addressing, no copy-engine round trip), the
// fused step runs (append; attention and head as programmatic dependents),
// and the head's last CTA writes the token ids to pinned host memory and
// counts the rows that picked the boundary token, so the host learns that a
// stream ended from one word instead of scanning the ids (an fp32 head leaves
// that to a small kernel).
#include <cuda_runtime.h>

#include <atomic>
#include <chrono>

#include <new>

#include "tts_common.cuh"
#include "tts_internal.h"

namespace tts {
namespace {

constexpr int kCopyThreads = 256;

// dst[i] = src[i] for n 16-byte words; src is pinned host memory.
__global__ void __launch_bounds__(kCopyThreads) copy_from_host_kernel(uint4 *__restrict__ dst,
                                                                      const uint4 *__restrict__ src,
                                                                      size_t n) {
    pdl_allow_dependents();  // the step's append may launch now; it waits for this copy
    const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
    size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    // four loads in flight per thread before the stores
    for (; i + 3 * stride < n; i += 4 * stride) {
        const uint4 a = src[i], b = src[i + stride], c = src[i + 2 * stride], d = src[i + 3 * stride];
        dst[i] = a;
        dst[i + stride] = b;
        dst[i + 2 * stride] = c;
        dst[i + 3 * stride] = d;
    }
    for (; i < n; i += stride) dst[i] = src[i];
}

// Up to kMaxSegs regions of the packed inputs: region i starts at byte
// offset off[i] (a multiple of 16) of both buffers and spans bytes[i] bytes (a
// multiple of 4).  A step for B streams copies the first B rows of each input.
constexpr int kMaxSegs = 16;
struct CopySegs {
    unsigned long long off[kMaxSegs];
    unsigned long long bytes[kMaxSegs];
    int n;
};

__global__ void __launch_bounds__(kCopyThreads) copy_segments_from_host_kernel(uint8_t *__restrict__ dst,
                                                                               const uint8_t *__restrict__ src,
                                                                               const CopySegs segs) {
    pdl_allow_dependents();  // the step's append may launch now; it waits for this copy
    // One index space over every region's 16-byte words, so the reads of all
    // regions are in flight together (each is a round trip to host memory).
    size_t start[kMaxSegs + 1];
    start[0] = 0;
    for (int i = 0; i < segs.n; ++i) start[i + 1] = start[i] + segs.bytes[i] / 16;
    const size_t total = start[segs.n];
    const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
    const size_t t0 = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    for (size_t w = t0; w < total; w += stride) {
        int i = 0;
        while (w >= start[i + 1]) ++i;
        const size_t o = segs.off[i] + (w - start[i]) * 16;
        *reinterpret_cast<uint4 *>(dst + o) = *reinterpret_cast<const uint4 *>(src + o);
    }
    // 4-byte tails of the regions (at most 3 words each)
    if (t0 < static_cast<size_t>(3 * segs.n)) {
        const int i = static_cast<int>(t0 / 3), k = static_cast<int>(t0 % 3);
        const size_t words = segs.bytes[i] / 16, tail = (segs.bytes[i] % 16) / 4;
        if (static_cast<size_t>(k) < tail) {
            const size_t o = segs.off[i] + words * 16 + 4 * k;
            *reinterpret_cast<uint32_t *>(dst + o) = *reinterpret_cast<const uint32_t *>(src + o);
        }
    }
}

// h_ids[r] = d_ids[r]; *h_count = #{r : d_ids[r] == boundary} (if h_count).
__global__ void __launch_bounds__(kCopyThreads) ids_to_host_kernel(const int32_t *__restrict__ d_ids, int R,
                                                                   int32_t boundary, int32_t *h_ids,
                                                                   int32_t *h_count) {
    __shared__ int warp_count[kCopyThreads / 32];
    int count = 0;
    for (int r = threadIdx.x; r < R; r += blockDim.x) {
        const int32_t id = d_ids[r];
        h_ids[r] = id;
        count += id == boundary;
    }
    count = __reduce_add_sync(0xFFFFFFFFu, count);
    if ((threadIdx.x & 31) == 0) warp_count[threadIdx.x >> 5] = count;
    __syncthreads();
    if (threadIdx.x == 0 && h_count) {
        int total = 0;
        for (int w = 0; w < kCopyThreads / 32; ++w) total += warp_count[w];
        *h_count = total;
    }
}

// dst_a[b] = src_a[b], dst_b[b] = src_b[b] for b < n (pinned host destinations).
__global__ void __launch_bounds__(kCopyThreads) pair_to_host_kernel(const int32_t *__restrict__ src_a,
                                                                    const int32_t *__restrict__ src_b, int n,
                                                                    int32_t *dst_a, int32_t *dst_b) {
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        if (dst_a) dst_a[i] = src_a[i];
        if (dst_b) dst_b[i] = src_b[i];
    }
}

bool device_accessible(const void *p) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return at.type == cudaMemoryTypeHost || at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged;
}

bool pinned_host(const void *p) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return at.type == cudaMemoryTypeHost && at.devicePointer == p;
}

}  // namespace
}  // namespace tts

struct tts_step_graph {
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
    // launch numbering for tts_step_graph_run (single graphs whose head
    // writes the ids to host memory): the head's last CTA increments d_seq
    // and writes it to the pinned h_seq after the ids
    int32_t *h_seq = nullptr;
    uint32_t *d_seq = nullptr;
    uint32_t launches = 0;
    bool numbered = false;  // the head writes the number (see capture_step)
};

namespace tts {
namespace {

// Checks every argument of the step described by d (B streams), captures the
// step and instantiates it.  With segs, the input copy moves those regions;
// without, all of input_bytes.
int capture_step(const tts_step_graph_desc *d, const CopySegs *segs, cudaGraph_t *graph_out,
                 cudaGraphExec_t *exec_out, int32_t *h_seq = nullptr, uint32_t *d_seq = nullptr,
                 bool *numbered = nullptr) {
    if (numbered) *numbered = false;
    *graph_out = nullptr;
    *exec_out = nullptr;
    if (!d->cache || d->B < 1) return TTS_ERR_INVALID;
    // host transfers
    if (!d->h_inputs || !d->d_inputs || d->input_bytes == 0 || (d->input_bytes & 15u) != 0 ||
        !aligned16(d->h_inputs) || !aligned16(d->d_inputs) || !d->h_ids || !d->d_ids)
        return TTS_ERR_INVALID;
    if (!pinned_host(d->h_inputs) || !pinned_host(d->h_ids) || (d->h_boundary_count && !pinned_host(d->h_boundary_count)))
        return TTS_ERR_INVALID;
    if (!device_accessible(d->d_inputs)) return TTS_ERR_INVALID;
    const long long R = static_cast<long long>(d->B) * d->q_len;
    if (R < 1 || R > 0x7FFFFFFF) return TTS_ERR_INVALID;

    // every argument of the step is checked here, before any capture
    AppendLaunch ap;
    AttnLaunch at;
    HeadLaunch hd;
    const tts_kv_cache *c = d->cache;
    int st = prepare_append_rope(c, d->d_block_table, d->max_blocks_per_seq, d->d_ctx_before, d->B, d->q_len,
                                 d->num_q_heads, d->rope_base, d->d_q, d->d_k_new, d->d_v_new, d->d_err, &ap);
    if (st != TTS_OK) return st;
    st = prepare_attn(c, d->d_block_table, d->max_blocks_per_seq, d->d_ctx_lens, d->max_ctx_len, d->B, d->q_len,
                      d->num_q_heads, d->scale, d->causal, d->d_q, d->d_attn_out, d->d_attn_ws, d->attn_ws_bytes,
                      d->d_err, &at);
    if (st != TTS_OK) return st;
    // Inputs read straight from the pinned buffer, which nothing writes during
    // a launch: the plain append's table, positions and rows (so it need not
    // wait for the copy kernel, only finish after it), and the attention's
    // table and lengths (read before its programmatic-launch wait).  The query
    // rows, read after the wait, stay on the device copy.
    const auto pinned_alias = [d](const void *p) -> const void * {
        const uint8_t *base = static_cast<const uint8_t *>(d->d_inputs), *q = static_cast<const uint8_t *>(p);
        if (!p || q < base || q >= base + d->input_bytes) return nullptr;
        return static_cast<const uint8_t *>(d->h_inputs) + (q - base);
    };
    const auto *h_table = static_cast<const int32_t *>(pinned_alias(d->d_block_table));
    const auto *h_before = static_cast<const int32_t *>(pinned_alias(d->d_ctx_before));
    const auto *h_lens = static_cast<const int32_t *>(pinned_alias(d->d_ctx_lens));
    const void *h_k = pinned_alias(d->d_k_new), *h_v = pinned_alias(d->d_v_new);
    const bool aliased = (c->dtype == TTS_BF16 || c->dtype == TTS_F32) && d->rope_base == 0.0f && h_table &&
                         h_before && h_lens && h_k && h_v;
    if (aliased) {
        st = prepare_append(c, h_table, d->max_blocks_per_seq, h_before, d->B, d->q_len, h_k, h_v, d->d_err, &ap);
        if (st != TTS_OK) return st;
        ap.wait_last = true;
        st = prepare_attn(c, h_table, d->max_blocks_per_seq, h_lens, d->max_ctx_len, d->B, d->q_len, d->num_q_heads,
                          d->scale, d->causal, d->d_q, d->d_attn_out, d->d_attn_ws, d->attn_ws_bytes, d->d_err, &at);
        if (st != TTS_OK) return st;
    }
    const long long H = static_cast<long long>(d->num_q_heads) * c->head_dim;
    if (H > 0x7FFFFFFF) return TTS_ERR_INVALID;
    // The tensor-core head's last CTA writes the ids and the boundary count to
    // pinned host memory itself; the fp32 head leaves that to a small kernel.
    const bool host_ids = c->dtype != TTS_F32;
    HeadExtras hx;
    if (host_ids) {
        hx.ids_host = d->h_ids;
        hx.count_host = d->h_boundary_count;
        // the launch number marks the ids as complete only when the head is
        // the step's last kernel (no verify stage after it)
        if (!d->d_n_accepted && h_seq && d_seq) {
            hx.seq_host = h_seq;
            hx.seq_dev = d_seq;
            if (numbered) *numbered = true;
        }
    }
    st = prepare_head_ex(d->d_attn_out, d->d_W, c->dtype == TTS_FP8_E4M3 ? TTS_BF16 : c->dtype,
                         static_cast<int32_t>(R), static_cast<int32_t>(H), d->V, d->mode, d->temperature, d->d_seed,
                         d->d_step, d->d_eos_allowed, d->d_ids, d->d_best, d->d_logits_out, d->d_head_ws,
                         d->head_ws_bytes, hx, &hd);
    if (st != TTS_OK) return st;
    // the optional verify stage reads the head's logits for K + 1 rows per stream
    const bool verify = d->d_n_accepted != nullptr;
    if (verify) {
        if (!d->d_logits_out || d->q_len < 2 || !d->d_next_token || !d->d_draft_probs || !d->d_draft_tokens ||
            !d->d_vseed || !d->d_vstep)
            return TTS_ERR_INVALID;
        if ((d->h_n_accepted && !pinned_host(d->h_n_accepted)) || (d->h_next_token && !pinned_host(d->h_next_token)))
            return TTS_ERR_INVALID;
        if (!(d->verify_temperature > 0.0f) || d->verify_temperature == INFINITY || d->q_len - 1 > 16 ||
            (d->verify_flags & ~TTS_VERIFY_BONUS) != 0)
            return TTS_ERR_INVALID;
    }

    cudaStream_t s;
    if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) {
        cudaGetLastError();
        return TTS_ERR_CUDA;
    }
    // With the append's and the attention's inputs read from the pinned
    // buffer, the copy kernel moves only what later kernels read from the
    // device buffer: the query rows, the head's keys and mask, the verify
    // stage's inputs (whichever lie in the buffer).  Regions it cannot move
    // (unaligned, too many) keep the whole copy.
    CopySegs trimmed{};
    const CopySegs *copy_segs = segs;
    if (aliased) {
        const uint8_t *base = static_cast<const uint8_t *>(d->d_inputs);
        const auto off_of = [base](const void *p) { return static_cast<size_t>(static_cast<const uint8_t *>(p) - base); };
        const size_t drop[5] = {off_of(d->d_block_table), off_of(d->d_ctx_before), off_of(d->d_ctx_lens),
                                off_of(d->d_k_new), off_of(d->d_v_new)};
        const auto dropped = [&drop](size_t off) {
            for (size_t x : drop)
                if (x == off) return true;
            return false;
        };
        if (segs) {
            for (int i = 0; i < segs->n; ++i) {
                if (dropped(segs->off[i])) continue;
                trimmed.off[trimmed.n] = segs->off[i];
                trimmed.bytes[trimmed.n] = segs->bytes[i];
                ++trimmed.n;
            }
            copy_segs = &trimmed;
        } else {
            const size_t elem = c->dtype == TTS_F32 ? 4u : 2u;
            const size_t K = d->q_len > 1 ? static_cast<size_t>(d->q_len - 1) : 0u;
            const size_t B = static_cast<size_t>(d->B), Rs = static_cast<size_t>(R);
            const struct { const void *p; size_t bytes; } need[] = {
                {d->d_q, Rs * static_cast<size_t>(d->num_q_heads) * c->head_dim * elem},
                {d->d_seed, Rs * 8}, {d->d_step, Rs * 8}, {d->d_eos_allowed, Rs},
                {d->d_draft_probs, B * K * static_cast<size_t>(d->V) * 4}, {d->d_draft_tokens, B * K * 4},
                {d->d_vseed, B * 8}, {d->d_vstep, B * 8}};
            bool fits = true;
            for (const auto &r : need) {
                if (!r.p) continue;
                const uint8_t *q = static_cast<const uint8_t *>(r.p);
                if (q < base || q >= base + d->input_bytes) continue;  // a device buffer of its own
                const size_t off = static_cast<size_t>(q - base), bytes = (r.bytes + 3) & ~size_t(3);
                if ((off & 15u) != 0 || bytes > d->input_bytes - off || trimmed.n == kMaxSegs) {
                    fits = false;
                    break;
                }
                trimmed.off[trimmed.n] = off;
                trimmed.bytes[trimmed.n] = bytes;
                ++trimmed.n;
            }
            if (fits && trimmed.n > 0) copy_segs = &trimmed;
        }
    }
    const int sms = sm_count() > 0 ? sm_count() : 148;
    size_t words = d->input_bytes / 16;
    if (copy_segs) {
        words = 0;
        for (int i = 0; i < copy_segs->n; ++i) words += (copy_segs->bytes[i] + 15) / 16;
    }
    const size_t want = (words + kCopyThreads - 1) / kCopyThreads;
    const unsigned copy_ctas = static_cast<unsigned>(want < static_cast<size_t>(sms) * 4 ? (want > 0 ? want : 1)
                                                                                         : static_cast<size_t>(sms) * 4);
    // Relaxed capture: the launch helpers set function attributes, which is
    // not a stream operation.
    cudaGraph_t graph = nullptr;
    bool ok = cudaStreamBeginCapture(s, cudaStreamCaptureModeRelaxed) == cudaSuccess;
    if (ok) {
        if (copy_segs)
            copy_segments_from_host_kernel<<<copy_ctas, kCopyThreads, 0, s>>>(
                static_cast<uint8_t *>(d->d_inputs), static_cast<const uint8_t *>(d->h_inputs), *copy_segs);
        else
            copy_from_host_kernel<<<copy_ctas, kCopyThreads, 0, s>>>(static_cast<uint4 *>(d->d_inputs),
                                                                     static_cast<const uint4 *>(d->h_inputs), words);
        ok = cudaGetLastError() == cudaSuccess;
        ok = ok && launch_append(ap, {s, true}) == TTS_OK;
        ok = ok && launch_attn(at, {s, true}) == TTS_OK;
        ok = ok && launch_head(hd, {s, true}) == TTS_OK;
        if (ok && !host_ids) {
            ids_to_host_kernel<<<1, kCopyThreads, 0, s>>>(d->d_ids, static_cast<int>(R), d->V - 1, d->h_ids,
                                                          d->h_boundary_count);
            ok = cudaGetLastError() == cudaSuccess;
        }
        if (ok && verify) {
            ok = tts_spec_verify(d->d_logits_out, d->d_draft_probs, d->d_draft_tokens, d->B, d->q_len - 1, d->V,
                                 d->verify_temperature, d->d_vseed, d->d_vstep, d->verify_flags, d->d_n_accepted,
                                 d->d_next_token, d->d_err, s) == TTS_OK;
            if (ok && (d->h_n_accepted || d->h_next_token)) {
                pair_to_host_kernel<<<1, kCopyThreads, 0, s>>>(d->d_n_accepted, d->d_next_token, d->B,
                                                               d->h_n_accepted, d->h_next_token);
                ok = cudaGetLastError() == cudaSuccess;
            }
        }
        const bool ended = cudaStreamEndCapture(s, &graph) == cudaSuccess;
        ok = ok && ended;
        if (ok) ok = cudaGraphInstantiate(exec_out, graph, 0) == cudaSuccess;
    }
    cudaStreamDestroy(s);
    if (!ok) {
        cudaGetLastError();
        if (*exec_out) cudaGraphExecDestroy(*exec_out);
        if (graph) cudaGraphDestroy(graph);
        *exec_out = nullptr;
        return TTS_ERR_CUDA;
    }
    *graph_out = graph;
    return TTS_OK;
}

}  // namespace
}  // namespace tts

namespace tts {
namespace {

// Launch-number pair of a graph or a graph set: a device counter (zeroed) and
// its pinned host copy, both or neither (an allocation failure leaves the
// caller to synchronise the stream).
void alloc_seq(int32_t **h_seq, uint32_t **d_seq) {
    const uint32_t zero = 0;
    *h_seq = nullptr;
    *d_seq = nullptr;
    if (cudaMalloc(reinterpret_cast<void **>(d_seq), sizeof(uint32_t)) != cudaSuccess ||
        cudaMemcpy(*d_seq, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaHostAlloc(reinterpret_cast<void **>(h_seq), sizeof(int32_t), cudaHostAllocDefault) != cudaSuccess) {
        cudaGetLastError();
        if (*d_seq) cudaFree(*d_seq);
        if (*h_seq) cudaFreeHost(*h_seq);
        cudaGetLastError();
        *h_seq = nullptr;
        *d_seq = nullptr;
        return;
    }
    **h_seq = 0;
}

void free_seq(int32_t *h_seq, uint32_t *d_seq) {
    if (d_seq) cudaFree(d_seq);
    if (h_seq) cudaFreeHost(h_seq);
}

// Waits until launch number `launches` has written its ids: a spin on the
// pinned number (a plain host read; the device's system-scope fence orders
// the ids before it), for at most a second before synchronising the stream
// (a failed launch never writes the number; the stream then reports the
// error).  Without a number (h_seq null, or a step whose head is not its last
// kernel: the number never moves) the stream is synchronised.
int wait_for_launch(const int32_t *h_seq, bool numbered, uint32_t launches, cudaStream_t s) {
    if (h_seq && numbered) {
        const volatile int32_t *w = h_seq;
        const auto t0 = std::chrono::steady_clock::now();
        for (uint32_t n = 0;; ++n) {
            if (static_cast<int32_t>(static_cast<uint32_t>(*w) - launches) >= 0) {
                std::atomic_thread_fence(std::memory_order_acquire);
                return TTS_OK;
            }
            if ((n & 1023u) == 0 && std::chrono::steady_clock::now() - t0 > std::chrono::seconds(1)) break;
        }
    }
    if (cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return TTS_ERR_CUDA;
    }
    return TTS_OK;
}

}  // namespace
}  // namespace tts

extern "C" int tts_step_graph_create(const tts_step_graph_desc *d, tts_step_graph **out) {
    using namespace tts;
    if (!d || !out) return TTS_ERR_INVALID;
    *out = nullptr;
    tts_step_graph *g = new (std::nothrow) tts_step_graph();
    if (!g) return TTS_ERR_CUDA;
    tts::alloc_seq(&g->h_seq, &g->d_seq);
    const int st = capture_step(d, nullptr, &g->graph, &g->exec, g->h_seq, g->d_seq, &g->numbered);
    if (st != TTS_OK) {
        tts_step_graph_destroy(g);
        return st;
    }
    *out = g;
    return TTS_OK;
}

extern "C" int tts_step_graph_launch(tts_step_graph *g, void *stream) {
    if (!g || !g->exec) return TTS_ERR_INVALID;
    if (cudaGraphLaunch(g->exec, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return TTS_ERR_CUDA;
    }
    ++g->launches;
    return TTS_OK;
}

extern "C" int tts_step_graph_run(tts_step_graph *g, void *stream) {
    const int st = tts_step_graph_launch(g, stream);
    if (st != TTS_OK) return st;
    return tts::wait_for_launch(g->h_seq, g->numbered, g->launches, static_cast<cudaStream_t>(stream));
}

extern "C" void tts_step_graph_destroy(tts_step_graph *g) {
    if (!g) return;
    if (g->exec) cudaGraphExecDestroy(g->exec);
    if (g->graph) cudaGraphDestroy(g->graph);
    tts::free_seq(g->h_seq, g->d_seq);
    delete g;
}

// ------------------------------------------------------------ graph sets

struct tts_step_graph_set {
    int n = 0;
    int32_t sizes[TTS_GRAPH_SET_MAX];
    tts_step_graph graphs[TTS_GRAPH_SET_MAX];
    // one launch-number pair shared by every size (launches on one stream)
    int32_t *h_seq = nullptr;
    uint32_t *d_seq = nullptr;
    uint32_t launches = 0;
    bool numbered = false;
};

extern "C" int tts_step_graph_set_create(const tts_step_graph_desc *d, const int32_t *sizes, int32_t n_sizes,
                                         const size_t *seg_offset, const size_t *seg_row_bytes, int32_t n_segs,
                                         tts_step_graph_set **out) {
    using namespace tts;
    if (!d || !out || !sizes || n_sizes < 1 || n_sizes > TTS_GRAPH_SET_MAX) return TTS_ERR_INVALID;
    *out = nullptr;
    if (!seg_offset || !seg_row_bytes || n_segs < 1 || n_segs > kMaxSegs) return TTS_ERR_INVALID;
    for (int i = 0; i < n_sizes; ++i)
        if (sizes[i] < 1 || sizes[i] > d->B || (i > 0 && sizes[i] <= sizes[i - 1])) return TTS_ERR_INVALID;
    if (sizes[n_sizes - 1] != d->B) return TTS_ERR_INVALID;
    // every region of B rows lies inside the packed buffers
    for (int i = 0; i < n_segs; ++i) {
        if ((seg_offset[i] & 15u) != 0 || (seg_row_bytes[i] & 3u) != 0 || seg_row_bytes[i] == 0) return TTS_ERR_INVALID;
        if (seg_offset[i] >= d->input_bytes ||
            seg_row_bytes[i] > (d->input_bytes - seg_offset[i]) / static_cast<size_t>(d->B))
            return TTS_ERR_INVALID;
    }
    tts_step_graph_set *set = new (std::nothrow) tts_step_graph_set();
    if (!set) return TTS_ERR_CUDA;
    alloc_seq(&set->h_seq, &set->d_seq);
    for (int k = 0; k < n_sizes; ++k) {
        tts_step_graph_desc dk = *d;
        dk.B = sizes[k];
        CopySegs segs{};
        segs.n = n_segs;
        for (int i = 0; i < n_segs; ++i) {
            segs.off[i] = seg_offset[i];
            segs.bytes[i] = seg_row_bytes[i] * static_cast<size_t>(sizes[k]);
        }
        const int st = capture_step(&dk, &segs, &set->graphs[k].graph, &set->graphs[k].exec, set->h_seq, set->d_seq,
                                    &set->numbered);
        if (st != TTS_OK) {
            tts_step_graph_set_destroy(set);
            return st;
        }
        set->sizes[k] = sizes[k];
        set->n = k + 1;
    }
    *out = set;
    return TTS_OK;
}

extern "C" int tts_step_graph_set_launch(tts_step_graph_set *set, int32_t n_streams, int32_t *chosen_B,
                                         void *stream) {
    if (!set || n_streams < 1) return TTS_ERR_INVALID;
    int k = 0;
    while (k < set->n && set->sizes[k] < n_streams) ++k;
    if (k == set->n) return TTS_ERR_INVALID;  // more streams than the largest size: split the cohort
    if (chosen_B) *chosen_B = set->sizes[k];
    const int st = tts_step_graph_launch(&set->graphs[k], stream);
    if (st == TTS_OK) ++set->launches;
    return st;
}

extern "C" int tts_step_graph_set_run(tts_step_graph_set *set, int32_t n_streams, int32_t *chosen_B, void *stream) {
    const int st = tts_step_graph_set_launch(set, n_streams, chosen_B, stream);
    if (st != TTS_OK) return st;
    return tts::wait_for_launch(set->h_seq, set->numbered, set->launches, static_cast<cudaStream_t>(stream));
}

extern "C" void tts_step_graph_set_destroy(tts_step_graph_set *set) {
    if (!set) return;
    for (int k = 0; k < set->n; ++k) {
        if (set->graphs[k].exec) cudaGraphExecDestroy(set->graphs[k].exec);
        if (set->graphs[k].graph) cudaGraphDestroy(set->graphs[k].graph);
    }
    tts::free_seq(set->h_seq, set->d_seq);
    delete set;
}
