// decode_launch.cuh -- launch of one decode-kernel variant (head dim D, head tiles
// NT, bf16 or fp8 cache).  Instantiated by decode_bf16.cu and decode_fp8.cu, one
// translation unit per cache type, so the two families compile in parallel.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "decode_kernel.cuh"
#include "plan.h"

namespace pkv {

// Dispatch on (D, NT) for one cache type; defined in decode_bf16.cu / decode_fp8.cu.
pkv_status launch_decode_bf16(int D, int NT, const CUtensorMap &mk, const CUtensorMap &mv, const DecodeParams &p,
                              const pkv_plan &plan, int B, int Hkv, int device, cudaStream_t stream);
pkv_status launch_decode_fp8(int D, int NT, const CUtensorMap &mk, const CUtensorMap &mv, const DecodeParams &p,
                             const pkv_plan &plan, int B, int Hkv, int device, cudaStream_t stream);

template <int D, int NT, bool KV8>
pkv_status launch_decode_variant(const CUtensorMap &mk, const CUtensorMap &mv, const DecodeParams &p,
                                 const pkv_plan &plan, int B, int Hkv, int device, cudaStream_t stream)
{
    static bool attr_set[64] = {};
    static std::mutex mu;
    auto kern = decode_split_kernel<D, NT, KV8>;
    if (device < 0 || device >= 64) return PKV_ERR_UNSUPPORTED;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!attr_set[device]) {
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448) != cudaSuccess)
                return PKV_ERR_CUDA;
            attr_set[device] = true;
        }
    }
    dim3 grid(Hkv, plan.num_splits, B);
    dim3 block(plan.warps * 32);
    kern<<<grid, block, plan.smem_bytes, stream>>>(mk, mv, p);
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

#define PKV_DECODE_DISPATCH(KV8)                                                                       \
    switch (D * 8 + NT) {                                                                              \
        case 64 * 8 + 1: return launch_decode_variant<64, 1, KV8>(mk, mv, p, plan, B, Hkv, device, stream);   \
        case 64 * 8 + 2: return launch_decode_variant<64, 2, KV8>(mk, mv, p, plan, B, Hkv, device, stream);   \
        case 64 * 8 + 4: return launch_decode_variant<64, 4, KV8>(mk, mv, p, plan, B, Hkv, device, stream);   \
        case 128 * 8 + 1: return launch_decode_variant<128, 1, KV8>(mk, mv, p, plan, B, Hkv, device, stream); \
        case 128 * 8 + 2: return launch_decode_variant<128, 2, KV8>(mk, mv, p, plan, B, Hkv, device, stream); \
        case 128 * 8 + 4: return launch_decode_variant<128, 4, KV8>(mk, mv, p, plan, B, Hkv, device, stream); \
        case 256 * 8 + 1: return launch_decode_variant<256, 1, KV8>(mk, mv, p, plan, B, Hkv, device, stream); \
        case 256 * 8 + 2: return launch_decode_variant<256, 2, KV8>(mk, mv, p, plan, B, Hkv, device, stream); \
        case 256 * 8 + 4: return launch_decode_variant<256, 4, KV8>(mk, mv, p, plan, B, Hkv, device, stream); \
        default: return PKV_ERR_UNSUPPORTED;                                                           \
    }

}  // namespace pkv
