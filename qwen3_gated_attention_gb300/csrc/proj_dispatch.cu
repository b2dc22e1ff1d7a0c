// proj_dispatch.cu -- width dispatch for the projection kernel.
#include "kernels.cuh"

namespace gattn {

#define GATTN_DECL(B)                                                                              \
    cudaError_t launch_proj_b##B(int, int, const ProjArgs &, const EpiQKV &, const EpiO &, int,    \
                                 bool, cudaStream_t);                                              \
    cudaError_t set_smem_b##B(int);                                                                \
    cudaError_t occupancy_b##B(int, int, int, int, int *);                                       \
    cudaError_t clusters_b##B(int, int, int, int, int, int *);
GATTN_DECL(2) GATTN_DECL(3) GATTN_DECL(4) GATTN_DECL(5) GATTN_DECL(6) GATTN_DECL(8)
#undef GATTN_DECL

int proj_smem_bytes(const ProjArgs &a)
{
    // stage ring + barriers/flags + epilogue statics (proj_tail_bytes in kernels.cuh)
    // + the split-K receive area + the converted-x table
    return a.stages * a.stage_bytes + proj_tail_bytes(a.eb_rows) + a.recv_cap * 4 + a.xtab_bytes;
}

cudaError_t launch_proj(int bits, int NT, int mode, const ProjArgs &a, const EpiQKV &eq,
                        const EpiO &eo, int grid, bool pdl, cudaStream_t s)
{
    switch (bits) {
    case 2: return launch_proj_b2(NT, mode, a, eq, eo, grid, pdl, s);
    case 3: return launch_proj_b3(NT, mode, a, eq, eo, grid, pdl, s);
    case 4: return launch_proj_b4(NT, mode, a, eq, eo, grid, pdl, s);
    case 5: return launch_proj_b5(NT, mode, a, eq, eo, grid, pdl, s);
    case 6: return launch_proj_b6(NT, mode, a, eq, eo, grid, pdl, s);
    case 8: return launch_proj_b8(NT, mode, a, eq, eo, grid, pdl, s);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t proj_set_smem_limits(int bits, int NT, int mode, int bytes)
{
    (void)NT;
    (void)mode;
    switch (bits) {
    case 2: return set_smem_b2(bytes);
    case 3: return set_smem_b3(bytes);
    case 4: return set_smem_b4(bytes);
    case 5: return set_smem_b5(bytes);
    case 6: return set_smem_b6(bytes);
    case 8: return set_smem_b8(bytes);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t proj_occupancy(int bits, int NT, int mode, int group, int smem, int *occ)
{
    switch (bits) {
    case 2: return occupancy_b2(NT, mode, group, smem, occ);
    case 3: return occupancy_b3(NT, mode, group, smem, occ);
    case 4: return occupancy_b4(NT, mode, group, smem, occ);
    case 5: return occupancy_b5(NT, mode, group, smem, occ);
    case 6: return occupancy_b6(NT, mode, group, smem, occ);
    case 8: return occupancy_b8(NT, mode, group, smem, occ);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t proj_max_clusters(int bits, int NT, int mode, int group, int smem, int csize, int *n)
{
    switch (bits) {
    case 2: return clusters_b2(NT, mode, group, smem, csize, n);
    case 3: return clusters_b3(NT, mode, group, smem, csize, n);
    case 4: return clusters_b4(NT, mode, group, smem, csize, n);
    case 5: return clusters_b5(NT, mode, group, smem, csize, n);
    case 6: return clusters_b6(NT, mode, group, smem, csize, n);
    case 8: return clusters_b8(NT, mode, group, smem, csize, n);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace gattn
