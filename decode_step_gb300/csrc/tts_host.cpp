// Host-side parts of the C ABI: the KV block pool, status strings, device
// queries.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>
#include <new>
#include <vector>

#include "tts_decode.h"
#include "tts_internal.h"

// ------------------------------------------------------------- block pool
//
// A static pool of fixed 16-token KV blocks; a request takes free blocks and
// gives them back when it finishes or is aborted ("Optimizing Streaming
// Text-to-Speech Models for Sub-50 Millisecond Latency", section "Dynamic
// Token-Level Batching"; "TTS Serving, in depth", section "Barge-in and
// cancellation").  A LIFO stack of free ids plus an allocation bitmap that
// catches double frees and foreign ids.

struct tts_block_pool {
    std::mutex mu;
    std::vector<int32_t> free_ids;   // stack; back() is handed out next
    std::vector<uint8_t> allocated;  // 1 while a block is out
};

extern "C" int tts_block_pool_create(int32_t num_blocks, tts_block_pool **out) {
    if (!out || num_blocks < 1) return TTS_ERR_INVALID;
    *out = nullptr;
    auto *p = new (std::nothrow) tts_block_pool;
    if (!p) return TTS_ERR_INVALID;
    p->free_ids.resize(num_blocks);
    // Lowest ids on top of the stack, so a fresh pool hands out 0, 1, 2, ...
    for (int32_t i = 0; i < num_blocks; ++i) p->free_ids[i] = num_blocks - 1 - i;
    p->allocated.assign(num_blocks, 0);
    *out = p;
    return TTS_OK;
}

extern "C" int tts_block_pool_alloc(tts_block_pool *pool, int32_t n, int32_t *host_ids_out) {
    if (!pool || n < 0 || (n > 0 && !host_ids_out)) return TTS_ERR_INVALID;
    std::lock_guard<std::mutex> lock(pool->mu);
    if (static_cast<size_t>(n) > pool->free_ids.size()) return TTS_ERR_POOL_EXHAUSTED;
    for (int32_t i = 0; i < n; ++i) {
        const int32_t id = pool->free_ids.back();
        pool->free_ids.pop_back();
        pool->allocated[id] = 1;
        host_ids_out[i] = id;
    }
    return TTS_OK;
}

extern "C" int tts_block_pool_free(tts_block_pool *pool, const int32_t *host_ids, int32_t n) {
    if (!pool || n < 0 || (n > 0 && !host_ids)) return TTS_ERR_INVALID;
    std::lock_guard<std::mutex> lock(pool->mu);
    const int32_t nb = static_cast<int32_t>(pool->allocated.size());
    // Validate everything first (all or nothing), marking with 2 to catch repeats.
    int32_t bad = -1;
    for (int32_t i = 0; i < n; ++i) {
        const int32_t id = host_ids[i];
        if (id < 0 || id >= nb || pool->allocated[id] != 1) { bad = i; break; }
        pool->allocated[id] = 2;
    }
    if (bad >= 0) {
        for (int32_t i = 0; i < bad; ++i) pool->allocated[host_ids[i]] = 1;
        return TTS_ERR_INVALID;
    }
    for (int32_t i = 0; i < n; ++i) {
        pool->allocated[host_ids[i]] = 0;
        pool->free_ids.push_back(host_ids[i]);
    }
    return TTS_OK;
}

extern "C" int32_t tts_block_pool_num_free(const tts_block_pool *pool) {
    if (!pool) return TTS_ERR_INVALID;
    auto *p = const_cast<tts_block_pool *>(pool);
    std::lock_guard<std::mutex> lock(p->mu);
    return static_cast<int32_t>(p->free_ids.size());
}

extern "C" void tts_block_pool_destroy(tts_block_pool *pool) { delete pool; }

// ------------------------------------------------------------------- misc

extern "C" const char *tts_status_string(int status) {
    switch (status) {
        case TTS_OK: return "ok";
        case TTS_ERR_INVALID: return "invalid argument";
        case TTS_ERR_UNSUPPORTED: return "unsupported shape or type";
        case TTS_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        case TTS_ERR_CUDA: return "CUDA error";
        case TTS_ERR_POOL_EXHAUSTED: return "block pool exhausted";
        case TTS_ERR_SCRATCH_LIMIT: return "request exceeds the library's static scratch";
        default: return "unknown status";
    }
}

extern "C" int tts_version(void) { return 100; }

namespace tts {
ThreadOpts &thread_opts() {
    static thread_local ThreadOpts opts;
    return opts;
}
}  // namespace tts

extern "C" int32_t tts_set_launch_flags(int32_t flags) {
    tts::ThreadOpts &o = tts::thread_opts();
    const int32_t prev = o.launch_flags;
    o.launch_flags = flags & TTS_LAUNCH_PROGRAMMATIC;
    return prev;
}

extern "C" int tts_test_set_stall(int32_t what, int64_t wait_limit_cycles) {
    if (what < TTS_TEST_STALL_NONE || what > TTS_TEST_STALL_PREDICTOR_GRID) return TTS_ERR_INVALID;
    if (wait_limit_cycles < 1000 || wait_limit_cycles > 4000000000LL) return TTS_ERR_INVALID;
    tts::ThreadOpts &o = tts::thread_opts();
    o.stall = what;
    o.wait_limit = wait_limit_cycles;
    return TTS_OK;
}

namespace tts {

int sm_count() {
    static std::atomic<int> cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
    if (dev < 64) {
        const int c = cached[dev].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev < 64) cached[dev].store(n, std::memory_order_relaxed);
    return n;
}

namespace {
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}
}  // namespace

bool make_tma_2d(CUtensorMap *map, const void *ptr, uint64_t rows, uint64_t cols, uint32_t box_rows,
                 uint32_t box_cols, int elem_bytes) {
    auto fn = encode_fn();
    if (!fn || (elem_bytes != 1 && elem_bytes != 2)) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * static_cast<cuuint64_t>(elem_bytes)};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
              const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tma_2d_bf16(CUtensorMap *map, const void *ptr, uint64_t rows, uint64_t cols,
                      uint32_t box_rows, uint32_t box_cols) {
    return make_tma_2d(map, ptr, rows, cols, box_rows, box_cols, 2);
}

bool make_tma_rows_in_halves_bf16(CUtensorMap *map, const void *ptr, uint64_t rows, uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {64, rows, 2};
    const cuuint64_t strides[2] = {256, 128};  // next row, next half
    const cuuint32_t box[3] = {64, box_rows, 2};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {
struct MapEntry {
    const void *ptr;
    uint64_t rows, cols;
    uint32_t box_rows, box_cols;
    int elem_bytes;
    int device;
    CUtensorMap map;
};
std::mutex g_map_mu;
MapEntry g_maps[16];
int g_maps_used = 0, g_maps_next = 0;
}  // namespace

bool cached_tma_2d(CUtensorMap *map, const void *ptr, uint64_t rows, uint64_t cols, uint32_t box_rows,
                   uint32_t box_cols, int elem_bytes) {
    int dev = -1;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lock(g_map_mu);
    for (int i = 0; i < g_maps_used; ++i) {
        const MapEntry &e = g_maps[i];
        if (e.ptr == ptr && e.rows == rows && e.cols == cols && e.box_rows == box_rows &&
            e.box_cols == box_cols && e.elem_bytes == elem_bytes && e.device == dev) {
            *map = e.map;
            return true;
        }
    }
    MapEntry e;
    e.ptr = ptr;
    e.rows = rows;
    e.cols = cols;
    e.box_rows = box_rows;
    e.box_cols = box_cols;
    e.elem_bytes = elem_bytes;
    e.device = dev;
    if (!make_tma_2d(&e.map, ptr, rows, cols, box_rows, box_cols, elem_bytes)) return false;
    g_maps[g_maps_next] = e;
    g_maps_next = (g_maps_next + 1) % 16;
    if (g_maps_used < 16) ++g_maps_used;
    *map = e.map;
    return true;
}

bool cached_tma_2d_bf16(CUtensorMap *map, const void *ptr, uint64_t rows, uint64_t cols,
                        uint32_t box_rows, uint32_t box_cols) {
    return cached_tma_2d(map, ptr, rows, cols, box_rows, box_cols, 2);
}

namespace {
struct SmemEntry {
    const void *func;
    int device;
    int bytes;
};
std::mutex g_smem_mu;
std::vector<SmemEntry> g_smem;
}  // namespace

bool ensure_dynamic_smem(const void *func, int bytes) {
    if (bytes <= 48 * 1024) return true;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    std::lock_guard<std::mutex> lock(g_smem_mu);
    for (auto &e : g_smem)
        if (e.func == func && e.device == dev) {
            if (e.bytes >= bytes) return true;
            if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
                return false;
            e.bytes = bytes;
            return true;
        }
    if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
        return false;
    g_smem.push_back({func, dev, bytes});
    return true;
}

}  // namespace tts
