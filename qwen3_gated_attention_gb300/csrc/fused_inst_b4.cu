// fused_inst_b4.cu -- compiled instances of the one-kernel layer step: 4-bit group-64 projections.
#include "fused.cuh"

namespace gattn {

bool fused_ops_part2(const FusedKey &k, FusedOps *ops)
{
    GATTN_FUSED_CASE(4, 64, 4, 64, 1, 1)
    GATTN_FUSED_CASE(4, 64, 4, 64, 1, 4)
    GATTN_FUSED_CASE(4, 64, 4, 64, 2, 4)
    GATTN_FUSED_CASE(4, 64, 4, 64, 3, 4)
    return false;
}

}  // namespace gattn
