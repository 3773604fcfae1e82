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

// TMA descriptor of a 2-D bf16 tensor [rows][cols] (cols contiguous) read in
// boxes of box_rows x box_cols with 128-byte swizzle (box_cols * 2 <= 128);
// out-of-range box elements read as zero.  false if the driver entry point is
// unavailable or the driver rejects the shape.
bool make_tma_2d_bf16(CUtensorMap *map, const void *ptr, uint64_t rows, uint64_t cols,
                      uint32_t box_rows, uint32_t box_cols);

// Maps the last launch error to a status (clears it).
inline int launch_status() {
    return cudaGetLastError() == cudaSuccess ? TTS_OK : TTS_ERR_CUDA;
}

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

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

}  // namespace tts
