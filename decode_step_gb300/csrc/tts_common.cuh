// Device helpers shared by the decode-step kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "tts_decode.h"

namespace tts {

// ------------------------------------------------------------------ errors

__device__ __forceinline__ void flag_error(int32_t *err, int bit) {
    if (err) atomicOr(err, bit);
}

// A bounded wait gives up after this many SM clock cycles (about one second).
constexpr long long kWaitLimitCycles = 2000000000LL;

// ------------------------------------------------- programmatic launch

// Lets the next kernel in the stream (if launched as a programmatic
// dependent) start now; its griddepcontrol.wait still waits for this grid.
__device__ __forceinline__ void pdl_allow_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// Waits until the previous kernel in the stream has completed and its writes
// are visible (returns at once when this grid was launched normally).
__device__ __forceinline__ void pdl_wait_prerequisites() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ------------------------------------------------------------ element types

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Eight bf16 or four fp32 values of one 16-byte chunk, as floats.
template <typename T> struct Chunk;
template <> struct Chunk<__nv_bfloat16> {
    static constexpr int N = 8;
    __device__ __forceinline__ static void unpack(const uint4 &c, float *f) {
        f[0] = bf16_lo(c.x); f[1] = bf16_hi(c.x); f[2] = bf16_lo(c.y); f[3] = bf16_hi(c.y);
        f[4] = bf16_lo(c.z); f[5] = bf16_hi(c.z); f[6] = bf16_lo(c.w); f[7] = bf16_hi(c.w);
    }
};
template <> struct Chunk<float> {
    static constexpr int N = 4;
    __device__ __forceinline__ static void unpack(const uint4 &c, float *f) {
        f[0] = __uint_as_float(c.x); f[1] = __uint_as_float(c.y);
        f[2] = __uint_as_float(c.z); f[3] = __uint_as_float(c.w);
    }
};

__device__ __forceinline__ void store_elem(float *p, float v) { *p = v; }
__device__ __forceinline__ void store_elem(__nv_bfloat16 *p, float v) { *p = __float2bfloat16_rn(v); }

// ------------------------------------------------------ shared memory / TMA

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Makes initialised mbarriers visible to the async (TMA / tensor core) proxy.
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.b32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for the phase with the given parity to complete; false after `limit`
// SM clock cycles (default about a second) without completion (the caller
// records TTS_ERRBIT_TIMEOUT).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, long long limit = kWaitLimitCycles) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    for (uint32_t n = 1;; ++n) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((n & 63u) == 0 && clock64() - t0 > limit) return false;
    }
}

// L2 policy for data read exactly once (the KV stream): evict first.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// Bulk (non-tensor) TMA copy global -> shared, completing on `bar` with tx bytes.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar,
                                          uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void bulk_load_nohint(uint32_t dst, const void *src, uint32_t bytes,
                                                 uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

// ------------------------------------------------------------------ Philox

// Philox4x64-10 (Salmon et al., "Parallel Random Numbers: As Easy as 1, 2, 3",
// SC'11): ten rounds of two 64x64->128-bit products with a Weyl-sequence key
// schedule.
struct Philox4x64 {
    uint64_t w[4];
    __device__ __forceinline__ Philox4x64(uint64_t c0, uint64_t c1, uint64_t c2, uint64_t c3,
                                          uint64_t k0, uint64_t k1) {
        constexpr uint64_t M0 = 0xD2E7470EE14C6C93ULL, M1 = 0xCA5A826395121157ULL;
        constexpr uint64_t W0 = 0x9E3779B97F4A7C15ULL, W1 = 0xBB67AE8584CAA73BULL;
#pragma unroll
        for (int r = 0; r < 10; ++r) {
            const uint64_t hi0 = __umul64hi(M0, c0), lo0 = M0 * c0;
            const uint64_t hi1 = __umul64hi(M1, c2), lo1 = M1 * c2;
            c0 = hi1 ^ c1 ^ k0;
            c1 = lo1;
            c2 = hi0 ^ c3 ^ k1;
            c3 = lo0;
            k0 += W0;
            k1 += W1;
        }
        w[0] = c0; w[1] = c1; w[2] = c2; w[3] = c3;
    }
    // 32-bit half `h` (0..7) of the block: word h / 2, low half first.
    __device__ __forceinline__ uint32_t half(int h) const {
        const uint64_t x = w[h >> 1];
        return (h & 1) ? static_cast<uint32_t>(x >> 32) : static_cast<uint32_t>(x);
    }
};

// Top 23 bits k of a 32-bit draw -> (2k + 1) / 2^24, exact, strictly inside (0, 1).
__device__ __forceinline__ float bits_to_uniform(uint32_t x) {
    return static_cast<float>(2u * (x >> 9) + 1u) * 0x1.0p-24f;
}

// Uniform number idx of the stream (seed, step, tag, pos): counter
// (idx / 8, tag, pos, 0), half idx % 8 of the block.
__device__ __forceinline__ float philox_uniform(uint64_t seed, uint64_t step, uint32_t tag,
                                                uint32_t pos, uint32_t idx) {
    const Philox4x64 p(idx >> 3, tag, pos, 0, seed, step);
    return bits_to_uniform(p.half(idx & 7));
}

// Hardware base-2 exponential and logarithm (PTX ex2 / lg2, .approx), for
// selection keys and softmax sums where their error (a few units of 2^-23
// relative for ex2, about 2^-22 absolute for lg2) is far below the 1e-3
// within which two keys or ratios count as near-ties.
__device__ __forceinline__ float hw_ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float hw_lg2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Gumbel noise -ln(-ln u) for u = (2k + 1) 2^-24 in (0, 1) (bits_to_uniform):
// the inner -ln u by the Taylor series of -ln(1 - w) = w + w^2/2 + ... in
// w = 1 - u (exact in fp32) when w < 1/16 (truncated after w^5 / 5: relative
// error below w^5 / 6), else by the hardware log2 (near u = 1 its absolute
// error would swamp -ln u, and those u give the largest draws); the outer log
// by the hardware log2.  Its distance to the exact value is tested over every
// u (tts_test_gumbel_noise).
__device__ __forceinline__ float gumbel_from_uniform(float u) {
    constexpr float kLn2 = 0.69314718055994531f;
    const float w = 1.0f - u;
    const float inner = w < 0.0625f ? w * (1.0f + w * (0.5f + w * (0.33333334f + w * (0.25f + w * 0.2f))))
                                    : -kLn2 * hw_lg2(u);
    return -kLn2 * hw_lg2(inner);
}

// ------------------------------------------------------- argmax key packing

// Order-preserving map float -> uint32 (larger float, larger key).
__device__ __forceinline__ uint32_t float_order_key(float f) {
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float order_key_float(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}
// 64-bit key: value in the high word; ties broken toward the lower index.
// 0 is below every real key, so a zeroed buffer is the identity of atomicMax.
__device__ __forceinline__ unsigned long long pack_argmax(float value, int32_t index) {
    return (static_cast<unsigned long long>(float_order_key(value)) << 32) |
           static_cast<unsigned long long>(~static_cast<uint32_t>(index));
}
__device__ __forceinline__ int32_t unpack_index(unsigned long long key) {
    return static_cast<int32_t>(~static_cast<uint32_t>(key & 0xFFFFFFFFull));
}
__device__ __forceinline__ float unpack_value(unsigned long long key) {
    return order_key_float(static_cast<uint32_t>(key >> 32));
}

}  // namespace tts
