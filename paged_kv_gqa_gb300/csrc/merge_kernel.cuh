// merge_kernel.cuh -- log-sum-exp merge of split partials.
//
// FlashQuant wiki "CUDA Kernels", split_k_reduce.cu "Algorithm": find the
// global max over the splits, rescale each split's weight by exp of its
// distance to that max, and take the weighted combination; "Numerical
// Stability": the rescaled weights are at most 1, and an all-empty row is
// guarded instead of dividing by zero.  Here each split carries a normalised
// f32 output and a natural-log LSE, so the weight of split s is
// exp(lse_s - max) and empty splits (lse = -inf) weigh 0.
//
// One warp per (b, query head); lanes cover the head dim with float4 loads.
// Two uses:
//   - after the decode kernel: the number of live splits of sequence b is
//     ceil(L_b / chunk) (splits past L_b never wrote anything), and rows with a
//     single split were already written by the decode kernel;
//   - the public split_kv_merge: exactly S splits for every row.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "ptx.cuh"

namespace pkv {

struct MergeParams {
    const float *part_out;  // [S, B, Hq, D]
    const float *part_lse;  // [S, B, Hq]
    const int *seq_lens;    // nullptr: every row has S splits
    __nv_bfloat16 *out;     // [B, Hq, D]
    float *lse;             // [B, Hq] or nullptr
    int S, B, Hq, chunk_tokens, max_tokens;
};

constexpr int kMergeWarps = 4;

template <int D>
__global__ void __launch_bounds__(kMergeWarps * 32) merge_kernel(const MergeParams p)
{
    griddep_wait();  // the partials may come from the previous kernel (PDL)
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row = blockIdx.x * kMergeWarps + warp;
    const int rows = p.B * p.Hq;
    if (row >= rows) return;

    int n = p.S;
    if (p.seq_lens) {
        int L = p.seq_lens[row / p.Hq];
        if (L < 0 || L > p.max_tokens) L = 0;  // same reading as the decode kernel: empty
        n = (L + p.chunk_tokens - 1) / p.chunk_tokens;
        if (n <= 1) return;  // written directly by the decode kernel
    }
    const size_t split_stride = (size_t)rows;

    float mx = -__int_as_float(0x7f800000);
    for (int s = lane; s < n; s += 32) mx = fmaxf(mx, p.part_lse[s * split_stride + row]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));

    constexpr int V4 = D / 4;  // float4 per row
    __nv_bfloat16 *orow = p.out + (size_t)row * D;
    if (mx == -__int_as_float(0x7f800000)) {
        for (int i = lane; i < V4; i += 32) {
            uint2 z = make_uint2(0u, 0u);
            *reinterpret_cast<uint2 *>(orow + 4 * i) = z;
        }
        if (p.lse && lane == 0) p.lse[row] = mx;
        return;
    }
    const float mx2 = mx * kLog2e;

    float wsum = 0.f;
    for (int s = lane; s < n; s += 32) wsum += ex2(p.part_lse[s * split_stride + row] * kLog2e - mx2);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
    const float inv = 1.f / wsum;

    for (int i = lane; i < V4; i += 32) {
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int s = 0; s < n; ++s) {
            const float w = ex2(p.part_lse[s * split_stride + row] * kLog2e - mx2);
            const float4 v = *reinterpret_cast<const float4 *>(p.part_out + (s * split_stride + row) * D + 4 * i);
            a.x += w * v.x;
            a.y += w * v.y;
            a.z += w * v.z;
            a.w += w * v.w;
        }
        uint2 packed;
        packed.x = pack_bf16x2(a.x * inv, a.y * inv);
        packed.y = pack_bf16x2(a.z * inv, a.w * inv);
        *reinterpret_cast<uint2 *>(orow + 4 * i) = packed;
    }
    if (p.lse && lane == 0) p.lse[row] = mx + __logf(wsum);
}

}  // namespace pkv
