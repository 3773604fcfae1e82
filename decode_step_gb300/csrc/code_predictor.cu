// The code predictor's frame loop ("How We Made a TTS Model Respond in
// Sub-50 ms", sections "Exploiting the regular building of the Code
// Predictor" and "Turn a fixed predictor loop into one GPU program": a fixed
// number of autoregressive steps per frame, one per remaining codebook, over a
// short bounded context in a preallocated KV cache, the whole loop captured as
// one CUDA graph).
//
// Step i for every stream r (x = the talker's state for the frame at i = 0):
//   projection    q, k, v = bf16(x Wqkv^T)              head kernel, linear mode
//   append        k, v at position i of the stream's block   append kernel
//   attention     o = bf16(attn(q; positions 0..i))     decode attention
//   selection     token = argmax / Gumbel-max of o W_i^T   head kernel (pos i + 1)
//   next input    x = E_i[token]                        gather kernel
// Every kernel after the first is a programmatic dependent of the one before
// (its set-up overlaps the predecessor's tail; it waits before reading the
// predecessor's output).  The cache holds one 16-token block per stream.
#include <cuda_runtime.h>

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

constexpr size_t kAlign = 256;

struct PredictorLayout {
    size_t x, q, k, v, o, kpool, vpool, table, ctx_before, ctx_lens, attn_ws, attn_ws_bytes, head_ws, head_ws_bytes,
        total;
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
    L->total = off;
    return true;
}

// Every launch of one frame, checked and prepared before anything runs.
struct PredictorPlan {
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
