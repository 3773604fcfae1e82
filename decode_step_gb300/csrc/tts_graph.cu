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
// and a second small kernel writes the token ids to pinned host memory and
// counts the rows that picked the boundary token, so the host learns that a
// stream ended from one word instead of scanning the ids.
#include <cuda_runtime.h>

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
};

extern "C" int tts_step_graph_create(const tts_step_graph_desc *d, tts_step_graph **out) {
    using namespace tts;
    if (!d || !out || !d->cache) return TTS_ERR_INVALID;
    *out = nullptr;
    if (d->B < 1) return TTS_ERR_INVALID;
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
    const long long H = static_cast<long long>(d->num_q_heads) * c->head_dim;
    if (H > 0x7FFFFFFF) return TTS_ERR_INVALID;
    st = prepare_head(d->d_attn_out, d->d_W, c->dtype == TTS_FP8_E4M3 ? TTS_BF16 : c->dtype, static_cast<int32_t>(R), static_cast<int32_t>(H), d->V,
                      d->mode, d->temperature, d->d_seed, d->d_step, d->d_eos_allowed, d->d_ids, d->d_best,
                      d->d_logits_out, d->d_head_ws, d->head_ws_bytes, &hd);
    if (st != TTS_OK) return st;

    tts_step_graph *g = new (std::nothrow) tts_step_graph();
    if (!g) return TTS_ERR_CUDA;
    cudaStream_t s;
    if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) {
        delete g;
        cudaGetLastError();
        return TTS_ERR_CUDA;
    }
    const int sms = sm_count() > 0 ? sm_count() : 148;
    const size_t words = d->input_bytes / 16;
    const size_t want = (words + kCopyThreads - 1) / kCopyThreads;
    const unsigned copy_ctas = static_cast<unsigned>(want < static_cast<size_t>(sms) * 4 ? (want > 0 ? want : 1)
                                                                                         : static_cast<size_t>(sms) * 4);
    // Relaxed capture: the launch helpers set function attributes, which is
    // not a stream operation.
    bool ok = cudaStreamBeginCapture(s, cudaStreamCaptureModeRelaxed) == cudaSuccess;
    if (ok) {
        copy_from_host_kernel<<<copy_ctas, kCopyThreads, 0, s>>>(static_cast<uint4 *>(d->d_inputs),
                                                                 static_cast<const uint4 *>(d->h_inputs), words);
        ok = cudaGetLastError() == cudaSuccess;
        ok = ok && launch_append(ap, {s, false}) == TTS_OK;
        ok = ok && launch_attn(at, {s, true}) == TTS_OK;
        ok = ok && launch_head(hd, {s, true}) == TTS_OK;
        if (ok) {
            ids_to_host_kernel<<<1, kCopyThreads, 0, s>>>(d->d_ids, static_cast<int>(R), d->V - 1, d->h_ids,
                                                          d->h_boundary_count);
            ok = cudaGetLastError() == cudaSuccess;
        }
        cudaGraph_t graph = nullptr;
        const bool ended = cudaStreamEndCapture(s, &graph) == cudaSuccess;
        ok = ok && ended;
        g->graph = graph;
        if (ok) ok = cudaGraphInstantiate(&g->exec, g->graph, 0) == cudaSuccess;
    }
    cudaStreamDestroy(s);
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

extern "C" int tts_step_graph_launch(tts_step_graph *g, void *stream) {
    if (!g || !g->exec) return TTS_ERR_INVALID;
    if (cudaGraphLaunch(g->exec, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return TTS_ERR_CUDA;
    }
    return TTS_OK;
}

extern "C" void tts_step_graph_destroy(tts_step_graph *g) {
    if (!g) return;
    if (g->exec) cudaGraphExecDestroy(g->exec);
    if (g->graph) cudaGraphDestroy(g->graph);
    delete g;
}
