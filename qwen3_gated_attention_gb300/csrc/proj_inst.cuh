// proj_inst.cuh -- per-width entry points of the projection kernel, so the
// widths compile in separate translation units.
#pragma once
#include "proj.cuh"

#define GATTN_PROJ_INSTANCE(B)                                                                     \
    namespace gattn {                                                                              \
    cudaError_t launch_proj_b##B(int NT, int mode, const ProjArgs &a, const EpiQKV &eq,            \
                                 const EpiO &eo, int grid, bool pdl, cudaStream_t s)               \
    {                                                                                              \
        return with_proj_kernel<B>(NT, mode, a.group, [&](auto kern, auto launch) {                \
            (void)kern;                                                                            \
            return launch(a, eq, eo, grid, pdl, s);                                                \
        });                                                                                        \
    }                                                                                              \
    cudaError_t set_smem_b##B(int bytes)                                                           \
    {                                                                                              \
        cudaError_t e = cudaSuccess;                                                               \
        for (int nt : {1, 2, 4})                                                                   \
            for (int md : {kModeQKV, kModeO})                                                      \
                for (int gr : {32, 64, 128})                                                       \
                    if (e == cudaSuccess)                                                          \
                        e = with_proj_kernel<B>(nt, md, gr, [&](auto kern, auto launch) {          \
                            (void)launch;                                                          \
                            cudaError_t r = cudaFuncSetAttribute(                                  \
                                kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);         \
                            if (r == cudaSuccess)                                                  \
                                r = cudaFuncSetAttribute(                                          \
                                    kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);      \
                            return r;                                                              \
                        });                                                                        \
        return e;                                                                                  \
    }                                                                                              \
    cudaError_t occupancy_b##B(int NT, int mode, int group, int smem, int *occ)                    \
    {                                                                                              \
        return with_proj_kernel<B>(NT, mode, group, [&](auto kern, auto launch) {                  \
            (void)launch;                                                                          \
            return cudaOccupancyMaxActiveBlocksPerMultiprocessor(occ, kern, proj_threads(NT), smem); \
        });                                                                                        \
    }                                                                                              \
    cudaError_t clusters_b##B(int NT, int mode, int group, int smem, int csize, int *n)            \
    {                                                                                              \
        return with_proj_kernel<B>(NT, mode, group, [&](auto kern, auto launch) {                  \
            (void)launch;                                                                          \
            cudaLaunchConfig_t cfg = {};                                                           \
            cfg.gridDim = dim3(csize);                                                             \
            cfg.blockDim = dim3(proj_threads(NT));                                                 \
            cfg.dynamicSmemBytes = smem;                                                           \
            cudaLaunchAttribute at[1];                                                             \
            at[0].id = cudaLaunchAttributeClusterDimension;                                        \
            at[0].val.clusterDim.x = csize;                                                        \
            at[0].val.clusterDim.y = 1;                                                            \
            at[0].val.clusterDim.z = 1;                                                            \
            cfg.attrs = at;                                                                        \
            cfg.numAttrs = 1;                                                                      \
            return cudaOccupancyMaxActiveClusters(n, kern, &cfg);                                  \
        });                                                                                        \
    }                                                                                              \
    }
