// decode_bf16.cu -- the decode kernel variants that read a bf16 page pool.
#include "decode_launch.cuh"

namespace pkv {

pkv_status launch_decode_bf16(int D, int NT, const CUtensorMap &mk, const CUtensorMap &mv, const DecodeParams &p,
                              const pkv_plan &plan, int B, int Hkv, int device, cudaStream_t stream)
{
    PKV_DECODE_DISPATCH(false, false, false)
}

}  // namespace pkv
