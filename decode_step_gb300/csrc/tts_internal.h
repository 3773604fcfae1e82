// Host-side helpers shared by the C-ABI entry points.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "tts_decode.h"

namespace tts {

// Number of SMs of the current device (cached per device ordinal).
int sm_count();

// Options of the calling thread (tts_set_launch_flags, tts_test_set_stall):
// whether single-kernel calls launch as programmatic dependents, and the
// test-only stall and wait limit handed to the kernels that support them.
struct ThreadOpts {
    int launch_flags = 0;
    int stall = 0;                       // TTS_TEST_STALL_* (0: none)
    long long wait_limit = 2000000000LL; // SM clock cycles per bounded wait
};
ThreadOpts &thread_opts();
inline bool thread_pdl() { return (thread_opts().launch_flags & TTS_LAUNCH_PROGRAMMATIC) != 0; }

// TMA descriptor of a 2-D tensor [rows][cols] (cols contiguous) of 1-byte
// (uint8) or 2-byte (bf16) elements, read in boxes of box_rows x box_cols with
// 128-byte swizzle (box_cols * elem_bytes <= 128); out-of-range box elements
// read as zero.  false if the driver entry point is unavailable or the driver
// rejects the shape.  cached_tma_2d caches descriptors by (address, shape,
// box, element size, device).
bool make_tma_2d(CUtensorMap *map, const void *ptr, uint64_t rows, uint64_t cols, uint32_t box_rows,
                 uint32_t box_cols, int elem_bytes);
bool cached_tma_2d(CUtensorMap *map, const void *ptr, uint64_t rows, uint64_t cols, uint32_t box_rows,
                   uint32_t box_cols, int elem_bytes);
// 3-D descriptor over bf16 rows of 128 elements seen as two 64-element halves:
// dims {64, rows, 2} with strides {256 B, 128 B}, box {64, box_rows, 2}, so one
// copy lands a tile of box_rows rows as [half][row][64] (each half 128-byte
// swizzled), the layout two 2-D boxes of 64 columns would give.
bool make_tma_rows_in_halves_bf16(CUtensorMap *map, const void *ptr, uint64_t rows, uint32_t box_rows);
// bf16 forms of the two.
bool make_tma_2d_bf16(CUtensorMap *map, const void *ptr, uint64_t rows, uint64_t cols,
                      uint32_t box_rows, uint32_t box_cols);

// Maps the last launch error to a status (clears it).
inline int launch_status() {
    return cudaGetLastError() == cudaSuccess ? TTS_OK : TTS_ERR_CUDA;
}

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Same, cached by (address, shape, box): building a descriptor is a driver
// call, and a serving loop passes the same tensors every step.
bool cached_tma_2d_bf16(CUtensorMap *map, const void *ptr, uint64_t rows, uint64_t cols,
                        uint32_t box_rows, uint32_t box_cols);

// Raises a kernel's dynamic shared-memory limit on the current device to at
// least `bytes`, calling the runtime only when the limit has to grow.
bool ensure_dynamic_smem(const void *func, int bytes);

// How a kernel is launched.  `pdl` (programmatic dependent launch) lets it
// start while the previous kernel in the stream is finishing; only set where
// the kernel runs griddepcontrol.wait before touching anything that kernel
// writes.
struct LaunchOpts {
    cudaStream_t stream;
    bool pdl;
};

// Decode-attention launch plan shared by the workspace query and the launch:
// a persistent grid of `ctas` CTAs (`workers` warps) over the flat tile list.
struct AttnPlan {
    int rows;     // query rows per (stream, KV head), padded to the kernel's template
    int ctas;     // CTAs launched
    int workers;  // warps, each owning one contiguous range of tiles
};
bool attn_plan(int dtype, int B, int q_len, int num_q_heads, int num_kv_heads, int head_dim,
               int max_ctx_len, AttnPlan *out);
size_t attn_workspace_bytes(int B, int num_kv_heads, int head_dim, const AttnPlan &pl);

// ---- validated launches, shared by the single-kernel entry points and
// tts_decode_step (which chains them with programmatic dependent launch)

// Inverse frequencies of the rotary embedding for head_dim 128:
// theta[i] = base^(-2i/128), i < 64, in double.
struct RopeFreqs {
    double theta[64];
};

struct AppendLaunch {
    const tts_kv_cache *cache;
    const int32_t *table;
    int max_blocks;
    const int32_t *ctx_before;
    int B, q_len;
    const void *k_new, *v_new;
    int32_t *err;
    // rotary embedding (rope == false: none): q [B][q_len][Hq][128] rotated in place
    bool rope;
    int Hq;
    void *q;
    RopeFreqs freqs;
    // bf16 / fp32 rows without rotation only: the inputs do not come from the
    // kernel before (they are read from pinned host memory), so the append
    // runs at once and waits for that kernel just before it ends
    bool wait_last;
};
int prepare_append(const tts_kv_cache *cache, const int32_t *d_block_table, int32_t max_blocks_per_seq,
                   const int32_t *d_ctx_before, int32_t B, int32_t q_len, const void *d_k_new,
                   const void *d_v_new, int32_t *d_err, AppendLaunch *out);
// prepare_append plus the rotary embedding's checks; rope_base == 0 means none.
int prepare_append_rope(const tts_kv_cache *cache, const int32_t *d_block_table, int32_t max_blocks_per_seq,
                        const int32_t *d_ctx_before, int32_t B, int32_t q_len, int32_t num_q_heads,
                        float rope_base, void *d_q, const void *d_k_new, const void *d_v_new, int32_t *d_err,
                        AppendLaunch *out);
int launch_append(const AppendLaunch &L, LaunchOpts o);

struct AttnLaunchState;  // defined in decode_attn.cu
struct AttnLaunch {
    alignas(64) unsigned char storage[1024];  // AttnLaunchState
};
int prepare_attn(const tts_kv_cache *cache, const int32_t *d_block_table, int32_t max_blocks_per_seq,
                 const int32_t *d_ctx_lens, int32_t max_ctx_len, int32_t B, int32_t q_len,
                 int32_t num_q_heads, float scale, int32_t causal, const void *d_q, void *d_out,
                 void *d_ws, size_t ws_bytes, int32_t *d_err, AttnLaunch *out);
int launch_attn(const AttnLaunch &L, LaunchOpts o);

struct HeadLaunch {
    alignas(64) unsigned char storage[1024];  // HeadLaunchState (tensor maps included)
};
int prepare_head(const void *d_h, const void *d_W, int32_t dtype, int32_t R, int32_t H, int32_t V,
                 int32_t mode, float temperature, const uint64_t *d_seed, const uint64_t *d_step,
                 const uint8_t *d_eos_allowed, int32_t *d_ids, float *d_best, float *d_logits_out,
                 void *d_ws, size_t ws_bytes, HeadLaunch *out);
// The head with a bias, a mask over the last n_tail ids, or (mode 2) the
// first audio-head layer writing Mish(h W^T + bias) as bf16 to z_out [R][V].
constexpr int kHeadModeExpand = 2;
constexpr int kHeadModeLinear = 3;
// Mode 3 (linear): h W^T as bf16, features [seg_start[j], seg_start[j + 1])
// written to seg_out[j] (rows of that width).  pos: the Gumbel noise's
// counter position.
struct HeadExtras {
    const float *bias = nullptr;
    const uint32_t *tail = nullptr;
    int n_tail = 0;
    void *z_out = nullptr;
    uint32_t pos = 0;
    int seg_start[4] = {0, 0, 0, 0};
    void *seg_out[3] = {nullptr, nullptr, nullptr};
    int32_t *ids_host = nullptr;    // the ids again, in pinned host memory
    int32_t *count_host = nullptr;  // rows whose id is the boundary V - 1
    // then the launch's number (*seq_dev incremented) in pinned host memory,
    // written after the ids are visible to the host (both or neither)
    int32_t *seq_host = nullptr;
    uint32_t *seq_dev = nullptr;
};
int prepare_head_ex(const void *d_h, const void *d_W, int32_t dtype, int32_t R, int32_t H, int32_t V,
                    int32_t mode, float temperature, const uint64_t *d_seed, const uint64_t *d_step,
                    const uint8_t *d_eos_allowed, int32_t *d_ids, float *d_best, float *d_logits_out,
                    void *d_ws, size_t ws_bytes, const HeadExtras &x, HeadLaunch *out);
int launch_head(const HeadLaunch &L, LaunchOpts o);

}  // namespace tts
