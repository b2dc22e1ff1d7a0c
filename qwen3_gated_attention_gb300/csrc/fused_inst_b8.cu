// fused_inst_b8.cu -- compiled instances of the one-kernel layer step: 8-bit group-64 projections.
#include "fused.cuh"

namespace gattn {

bool fused_ops_part1(const FusedKey &k, FusedOps *ops)
{
    GATTN_FUSED_CASE(8, 64, 8, 64, 1, 4)
    GATTN_FUSED_CASE(8, 64, 8, 64, 2, 4)
    return false;
}

}  // namespace gattn
