// prefill_bf16.cu -- the multi-token variants (several query rows per sequence,
// ragged by qo_indptr) that read a bf16 page pool.
#include "decode_launch.cuh"

namespace pkv {

pkv_status launch_prefill_bf16(int D, int NT, const CUtensorMap &mk, const CUtensorMap &mv, const DecodeParams &p,
                               const pkv_plan &plan, int B, int Hkv, int device, cudaStream_t stream)
{
    PKV_DECODE_DISPATCH(false, true, false)
}

}  // namespace pkv
