// decode_launch.cuh -- launch of one decode-kernel variant (head dim D, row tiles
// NT, bf16 or fp8 cache, one or several query rows per sequence).  Instantiated by
// decode_{bf16,fp8}.cu and prefill_{bf16,fp8}.cu, one translation unit per family,
// so the families compile in parallel.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "decode_kernel.cuh"
#include "launch_util.h"
#include "plan.h"

namespace pkv {

// Dispatch on (D, NT) for one family; defined in decode_{bf16,fp8}.cu, prefill_{bf16,fp8}.cu.
#define PKV_DECLARE_LAUNCH(NAME)                                                                             \
    pkv_status NAME(int D, int NT, const CUtensorMap &mk, const CUtensorMap &mv, const DecodeParams &p,        \
                    const pkv_plan &plan, int B, int Hkv, int device, cudaStream_t stream);
PKV_DECLARE_LAUNCH(launch_decode_bf16)
PKV_DECLARE_LAUNCH(launch_decode_fp8)
PKV_DECLARE_LAUNCH(launch_decode_adapt_bf16)
PKV_DECLARE_LAUNCH(launch_decode_adapt_fp8)
PKV_DECLARE_LAUNCH(launch_prefill_bf16)
PKV_DECLARE_LAUNCH(launch_prefill_fp8)
#undef PKV_DECLARE_LAUNCH

template <int D, int NT, bool KV8, bool MQ, bool ADAPT>
pkv_status launch_decode_variant(const CUtensorMap &mk, const CUtensorMap &mv, const DecodeParams &p,
                                 const pkv_plan &plan, int B, int Hkv, int device, cudaStream_t stream)
{
    static bool attr_set[64] = {};
    static int8_t cluster_ok[64][kMaxClusterSplits + 1] = {};  // 0 unknown, 1 resident, -1 not
    static std::mutex mu;
    auto kern = decode_split_kernel<D, NT, KV8, MQ, ADAPT>;
    if (device < 0 || device >= 64) return PKV_ERR_UNSUPPORTED;
    dim3 grid(Hkv * plan.q_tiles, plan.num_splits, B);
    dim3 block(plan.warps * 32);
    const unsigned S = (unsigned)plan.num_splits;
    bool cluster = !MQ && p.cluster && S >= 2 && S <= (unsigned)kMaxClusterSplits;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!attr_set[device]) {
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448) != cudaSuccess)
                return PKV_ERR_CUDA;
            attr_set[device] = true;
        }
        // A cluster that cannot be resident falls back to the workspace merge (first call per
        // device and cluster size only: an occupancy query, no launch).
        if (cluster && cluster_ok[device][S] == 0)
            cluster_ok[device][S] = cluster_fits(kern, block, (size_t)plan.smem_bytes, S) ? 1 : -1;
        if (cluster && cluster_ok[device][S] < 0) cluster = false;
    }
    cudaError_t e;
    if (cluster) {
        e = launch_kernel_cluster(kern, grid, block, (size_t)plan.smem_bytes, stream, S, mk, mv, p);
    } else if (p.cluster) {
        DecodeParams q = p;
        q.cluster = 0;
        e = launch_kernel(kern, grid, block, (size_t)plan.smem_bytes, stream, mk, mv, q);
    } else {
        e = launch_kernel(kern, grid, block, (size_t)plan.smem_bytes, stream, mk, mv, p);
    }
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

// (a D = 256 block serves at most 16 rows: no 32-row variant there)
#define PKV_V(DD, NN, KV8, MQ, AD) launch_decode_variant<DD, NN, KV8, MQ, AD>(mk, mv, p, plan, B, Hkv, device, stream)
#define PKV_DECODE_DISPATCH(KV8, MQ, AD)                     \
    switch (D * 8 + NT) {                                    \
        case 64 * 8 + 1: return PKV_V(64, 1, KV8, MQ, AD);       \
        case 64 * 8 + 2: return PKV_V(64, 2, KV8, MQ, AD);       \
        case 64 * 8 + 4: return PKV_V(64, 4, KV8, MQ, AD);       \
        case 128 * 8 + 1: return PKV_V(128, 1, KV8, MQ, AD);     \
        case 128 * 8 + 2: return PKV_V(128, 2, KV8, MQ, AD);     \
        case 128 * 8 + 4: return PKV_V(128, 4, KV8, MQ, AD);     \
        case 256 * 8 + 1: return PKV_V(256, 1, KV8, MQ, AD);     \
        case 256 * 8 + 2: return PKV_V(256, 2, KV8, MQ, AD);     \
        default: return PKV_ERR_UNSUPPORTED;                 \
    }

}  // namespace pkv
