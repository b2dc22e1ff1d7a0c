// fused_inst_mix.cu -- compiled instances of the one-kernel layer step: 6-bit group-128 q/k/v with 3-bit group-32 o_proj.
#include "fused.cuh"

namespace gattn {

bool fused_ops_part3(const FusedKey &k, FusedOps *ops)
{
    GATTN_FUSED_CASE(6, 128, 3, 32, 1, 1)
    GATTN_FUSED_CASE(6, 128, 3, 32, 1, 4)
    return false;
}

}  // namespace gattn
