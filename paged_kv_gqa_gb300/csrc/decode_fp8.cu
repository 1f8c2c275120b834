// decode_fp8.cu -- the decode kernel variants that read an fp8 (e4m3) page pool
// with per-(token, kv head) scales.
#include "decode_launch.cuh"

namespace pkv {

pkv_status launch_decode_fp8(int D, int NT, const CUtensorMap &mk, const CUtensorMap &mv, const DecodeParams &p,
                             const pkv_plan &plan, int B, int Hkv, int device, cudaStream_t stream)
{
    PKV_DECODE_DISPATCH(true, false, false)
}

}  // namespace pkv
