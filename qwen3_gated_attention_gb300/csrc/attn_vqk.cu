// attn_vqk.cu -- the attention kernel over a symmetric Turbo4 cache: K and V
// code and scale rows by bulk copies; each warp dequantizes the key rows of
// its own tokens into an fp16 key tile for its q K^T (the q rows rotated once
// per piece, so the keys stay in their rotated basis), each tile's values are
// dequantized as for the Bf16KTurbo4V cache, and the merge rotates the
// output rows back.
#include "attn.cuh"

namespace gattn {

cudaError_t launch_attn_vqk(int MT, int DB, const AttnArgs &a, const CUtensorMap &kmap, int grid,
                            bool pdl, cudaStream_t s)
{
#define GATTN_CASE(mt, db)                                                                         \
    if (MT == mt && DB == db)                                                                      \
        return launch_attn_t<mt, db, 2>(a, kmap, kmap, grid, pdl, s);
    GATTN_ATTN_INSTANCES(GATTN_CASE)
#undef GATTN_CASE
    return cudaErrorInvalidValue;
}

cudaError_t attn_vqk_set_smem_limits()
{
    cudaError_t e = cudaSuccess;
#define GATTN_SET(mt, db)                                                                          \
    if (e == cudaSuccess)                                                                          \
        e = cudaFuncSetAttribute(attn_kernel<mt, db, 2>,                                           \
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,                      \
                                 AttnSmem<mt, db, 2>::kTotal);
    GATTN_ATTN_INSTANCES(GATTN_SET)
#undef GATTN_SET
    return e;
}

}  // namespace gattn
