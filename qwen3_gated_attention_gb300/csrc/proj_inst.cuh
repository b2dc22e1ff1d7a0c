// proj_inst.cuh -- per-width entry points of the projection kernel, so the
// widths compile in separate translation units.
#pragma once
#include "proj.cuh"

namespace gattn {

template <int BITS>
cudaError_t occupancy_bits(int NT, int mode, int smem, int *occ)
{
    const int threads = (kWR + 1) * 32;
#define GATTN_OCC(nt, md)                                                                          \
    if (NT == nt && mode == md)                                                                    \
        return cudaOccupancyMaxActiveBlocksPerMultiprocessor(occ, proj_kernel<BITS, nt, md>,       \
                                                             threads, smem);
    GATTN_OCC(1, kModeQKV) GATTN_OCC(2, kModeQKV) GATTN_OCC(4, kModeQKV)
    GATTN_OCC(1, kModeO) GATTN_OCC(2, kModeO) GATTN_OCC(4, kModeO)
#undef GATTN_OCC
    return cudaErrorInvalidValue;
}

}  // namespace gattn

#define GATTN_PROJ_INSTANCE(B)                                                                     \
    namespace gattn {                                                                              \
    cudaError_t launch_proj_b##B(int NT, int mode, const ProjArgs &a, const EpiQKV &eq,            \
                                 const EpiO &eo, int grid, bool pdl, cudaStream_t s)               \
    {                                                                                              \
        return launch_proj_bits<B>(NT, mode, a, eq, eo, grid, pdl, s);                             \
    }                                                                                              \
    cudaError_t set_smem_b##B(int bytes) { return set_smem_bits<B>(bytes); }                       \
    cudaError_t occupancy_b##B(int NT, int mode, int smem, int *occ)                               \
    {                                                                                              \
        return occupancy_bits<B>(NT, mode, smem, occ);                                             \
    }                                                                                              \
    }
