// append_kernel.cuh -- paged KV append: the per-token cache write that precedes a
// decode step (Atlas "CUDA Kernel Engineering", "The kernel inventory": KV append,
// a per-token K/V write into the paged cache).  The new key and value rows of
// sequence b go to logical key position positions[b]: physical page
// block_table[b][pos >> log2 P], slot pos & (P-1) (FlashQuant wiki "CUDA Kernels",
// paged_decode.cu "Page Table Addressing").  K and V are written by the same launch.
//
// One warp per (sequence, kv head): the lanes move the 2*D-byte rows in 16-byte
// vectors, K and V side by side.  A position past the table or a page id outside
// the pool is skipped and recorded in the status word; a negative position means
// "nothing to append" for that sequence.
//
// The fp8 form (kv_append_fp8_kernel) quantises on the way, K and V in one launch
// (OASR "Kernel Layer", "FP8 KV variants": one quantise-and-scatter launch per
// layer): each row of D values gets the scale 2^k, k the smallest integer in
// [-64, 64] with max|x| <= 448 * 2^k (NaN left out of the maximum), and codes
// e4m3(x * 2^-k), rounded to nearest even and saturated at +-448.  The scale goes
// to k_scale/v_scale[page][kv head][slot].
#pragma once

#include <cstdint>

#include "pkv.h"
#include "ptx.cuh"

namespace pkv {

struct AppendParams {
    const uint4 *k_new;      // [B, Hkv, D] bf16, as 16-byte vectors
    const uint4 *v_new;
    const int *block_table;  // [B, max_pages]
    const int *positions;    // [B]
    uint4 *k_cache;          // [num_pages, P, Hkv, D] bf16, as 16-byte vectors
    uint4 *v_cache;
    int *status;             // may be nullptr
    int B, Hkv, D, P, log2P, num_pages, max_pages;
};

constexpr int kAppendWarps = 8;

__global__ void __launch_bounds__(kAppendWarps * 32) kv_append_kernel(const AppendParams p)
{
    griddep_launch_dependents();  // the decode step that follows may start launching
    griddep_wait();               // the new rows may come from the previous kernel
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int unit = blockIdx.x * kAppendWarps + warp;  // (b, kv head)
    if (unit >= p.B * p.Hkv) return;
    const int b = unit / p.Hkv, kvh = unit - b * p.Hkv;
    const int pos = p.positions[b];
    if (pos < 0) return;
    if (pos >= p.max_pages * p.P) {
        if (kvh == 0 && lane == 0 && p.status) atomicCAS(p.status, 0, PKV_ERR_BAD_SEQ_LEN);
        return;
    }
    const int page = p.block_table[(size_t)b * p.max_pages + (pos >> p.log2P)];
    if ((unsigned)page >= (unsigned)p.num_pages) {
        if (kvh == 0 && lane == 0 && p.status) atomicCAS(p.status, 0, PKV_ERR_BAD_PAGE_INDEX);
        return;
    }
    const int vec = p.D / 8;  // 16-byte vectors per row
    const size_t src = (size_t)unit * vec;
    const size_t dst = (((size_t)page * p.P + (pos & (p.P - 1))) * p.Hkv + kvh) * vec;
    for (int i = lane; i < 2 * vec; i += 32) {
        if (i < vec)
            p.k_cache[dst + i] = p.k_new[src + i];
        else
            p.v_cache[dst + i - vec] = p.v_new[src + i - vec];
    }
}

struct Fp8AppendParams {
    const uint16_t *k_new;   // [B, Hkv, D] bf16 bits
    const uint16_t *v_new;
    const int *block_table;  // [B, max_pages]
    const int *positions;    // [B]
    uint8_t *k_cache;        // [num_pages, P, Hkv, D] e4m3 codes
    uint8_t *v_cache;
    float *k_scale;          // [num_pages, Hkv, P]
    float *v_scale;
    int *status;             // may be nullptr
    int B, Hkv, P, log2P, num_pages, max_pages;
};

// Scale exponent of a row from its largest magnitude (f32, exact for bf16 inputs).
__device__ __forceinline__ int fp8_scale_exponent(float amax)
{
    constexpr float kLo = 448.f * 0x1p-64f, kHi = 448.f * 0x1p64f;
    if (!(amax > kLo)) return -64;
    if (amax > kHi) return 64;
    const int e = (int)((__float_as_uint(amax) >> 23) & 0xffu) - 127;  // amax in [2^e, 2^(e+1)), a normal
    const float lim = 448.f * __uint_as_float((uint32_t)(e - 8 + 127) << 23);  // 448 * 2^(e-8) = 1.75 * 2^e
    return amax <= lim ? e - 8 : e - 7;
}

// Quantises the D-value row `src` (bf16 bits) held E values per lane; writes the codes
// to dst and returns the scale.
template <int D>
__device__ __forceinline__ float quantize_row_e4m3(const uint16_t *src, uint8_t *dst, int lane)
{
    constexpr int E = D / 32;  // values per lane: 2, 4 or 8
    float x[E];
    if constexpr (E == 2) {
        const uint32_t w = reinterpret_cast<const uint32_t *>(src)[lane];
        x[0] = __uint_as_float(w << 16);
        x[1] = __uint_as_float(w & 0xffff0000u);
    } else if constexpr (E == 4) {
        const uint2 w = reinterpret_cast<const uint2 *>(src)[lane];
        x[0] = __uint_as_float(w.x << 16);
        x[1] = __uint_as_float(w.x & 0xffff0000u);
        x[2] = __uint_as_float(w.y << 16);
        x[3] = __uint_as_float(w.y & 0xffff0000u);
    } else {
        const uint4 w = reinterpret_cast<const uint4 *>(src)[lane];
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            x[2 * i] = __uint_as_float(ws[i] << 16);
            x[2 * i + 1] = __uint_as_float(ws[i] & 0xffff0000u);
        }
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < E; ++i) amax = fmaxf(amax, fabsf(x[i]));  // fmaxf drops a NaN operand
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const int k = fp8_scale_exponent(amax);
    const float inv = __uint_as_float((uint32_t)(127 - k) << 23);  // 2^-k, exact
    uint32_t packed[E / 2];
#pragma unroll
    for (int i = 0; i < E / 2; ++i) {
        unsigned short c;
        // the first operand lands in the upper byte
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(c) : "f"(x[2 * i + 1] * inv), "f"(x[2 * i] * inv));
        packed[i] = c;
    }
    if constexpr (E == 2) {
        reinterpret_cast<unsigned short *>(dst)[lane] = (unsigned short)packed[0];
    } else if constexpr (E == 4) {
        reinterpret_cast<uint32_t *>(dst)[lane] = packed[0] | (packed[1] << 16);
    } else {
        reinterpret_cast<uint2 *>(dst)[lane] = make_uint2(packed[0] | (packed[1] << 16), packed[2] | (packed[3] << 16));
    }
    return __uint_as_float((uint32_t)(127 + k) << 23);
}

template <int D>
__global__ void __launch_bounds__(kAppendWarps * 32) kv_append_fp8_kernel(const Fp8AppendParams p)
{
    griddep_launch_dependents();
    griddep_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int unit = blockIdx.x * kAppendWarps + warp;  // (b, kv head)
    if (unit >= p.B * p.Hkv) return;
    const int b = unit / p.Hkv, kvh = unit - b * p.Hkv;
    const int pos = p.positions[b];
    if (pos < 0) return;
    if (pos >= p.max_pages * p.P) {
        if (kvh == 0 && lane == 0 && p.status) atomicCAS(p.status, 0, PKV_ERR_BAD_SEQ_LEN);
        return;
    }
    const int page = p.block_table[(size_t)b * p.max_pages + (pos >> p.log2P)];
    if ((unsigned)page >= (unsigned)p.num_pages) {
        if (kvh == 0 && lane == 0 && p.status) atomicCAS(p.status, 0, PKV_ERR_BAD_PAGE_INDEX);
        return;
    }
    const int slot = pos & (p.P - 1);
    const size_t src = (size_t)unit * D;
    const size_t dst = (((size_t)page * p.P + slot) * p.Hkv + kvh) * D;
    const size_t sdst = ((size_t)page * p.Hkv + kvh) * p.P + slot;
    const float ks = quantize_row_e4m3<D>(p.k_new + src, p.k_cache + dst, lane);
    const float vs = quantize_row_e4m3<D>(p.v_new + src, p.v_cache + dst, lane);
    if (lane == 0) {
        p.k_scale[sdst] = ks;
        p.v_scale[sdst] = vs;
    }
}

}  // namespace pkv
