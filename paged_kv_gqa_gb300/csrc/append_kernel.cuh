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

}  // namespace pkv
