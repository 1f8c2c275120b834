// prefill_fp8.cu -- the multi-token variants that read an fp8 (e4m3) page pool.
#include "decode_launch.cuh"

namespace pkv {

pkv_status launch_prefill_fp8(int D, int NT, const CUtensorMap &mk, const CUtensorMap &mv, const DecodeParams &p,
                              const pkv_plan &plan, int B, int Hkv, int device, cudaStream_t stream)
{
    PKV_DECODE_DISPATCH(true, true, false)
}

}  // namespace pkv
