// attn_vq.cu -- the attention kernel over a Bf16KTurbo4V cache: K bf16 tiles
// by TMA as for a bf16 cache, V code and scale rows by bulk copies, each tile
// dequantized once into an fp16 tile (level pair table x E4M3 scale) and
// multiplied on fp16 mma.sync.  The rotation back to the original basis is
// applied to each output row by the merge.
#include "attn.cuh"

namespace gattn {

cudaError_t launch_attn_vq(int MT, int DB, const AttnArgs &a, const CUtensorMap &kmap, int grid,
                           bool pdl, cudaStream_t s)
{
#define GATTN_CASE(mt, db)                                                                         \
    if (MT == mt && DB == db)                                                                      \
        return launch_attn_t<mt, db, 1>(a, kmap, kmap, grid, pdl, s);
    GATTN_ATTN_INSTANCES(GATTN_CASE)
#undef GATTN_CASE
    return cudaErrorInvalidValue;
}

int attn_vq_smem_bytes(int MT, int DB)
{
#define GATTN_CASE(mt, db)                                                                         \
    if (MT == mt && DB == db)                                                                      \
        return AttnSmem<mt, db, 1>::kTotal;
    GATTN_ATTN_INSTANCES(GATTN_CASE)
#undef GATTN_CASE
    return -1;
}

cudaError_t attn_vq_set_smem_limits()
{
    cudaError_t e = cudaSuccess;
#define GATTN_SET(mt, db)                                                                          \
    if (e == cudaSuccess)                                                                          \
        e = cudaFuncSetAttribute(attn_kernel<mt, db, 1>,                                           \
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,                      \
                                 AttnSmem<mt, db, 1>::kTotal);
    GATTN_ATTN_INSTANCES(GATTN_SET)
#undef GATTN_SET
    return e == cudaSuccess ? attn_vqk_set_smem_limits() : e;
}

}  // namespace gattn
