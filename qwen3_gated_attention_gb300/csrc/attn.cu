// attn.cu -- causal GQA decode / verify attention over a bf16 KV cache (the
// kernel template is in attn.cuh; attn_vq.cu and attn_vqk.cu hold the Turbo4
// instances).
//
// For every (sequence b, KV head kh, row block rb) segment the rows are the
// R new rows of the row block's query heads (at most 16 rows of one KV group,
// or of one chunk of it when the verify head-chunk plan is on), and the keys
// are cache positions [0, cache_pos[b] + R).  Segments are cut into chunks of
// whole 16-token units, of one length for all segments of the step (from the
// unchunked partition, so both head partitions cut every segment alike; at
// most 32 chunks a segment), and the chunks are spread over the grid in
// contiguous ranges balanced by tokens.  One producer warp streams 64-token
// K/V tiles with 4-D TMA tensor copies (128-byte swizzle) into a ring of up to
// four stages; one tile read serves every query row of the segment.  Eight
// consumer warps compute S = q K^T and O += P V with bf16 mma.sync (fp32
// accumulate) and an online softmax in the log2 domain.
//
// A segment of one chunk is finished from the accumulators (bf16 V).
// Otherwise each chunk leaves a partial (m, l, O) and the merge launch that
// follows (attn_merge_kernel, one CTA per segment row) combines them.  Either
// way the output gate attn * sigmoid(gate) is applied and the o_proj operand
// is written in tensor-core fragment order (fp16) with its group sums.
#include "attn.cuh"

namespace gattn {

cudaError_t launch_attn(int MT, int DB, const AttnArgs &a, const CUtensorMap &kmap,
                        const CUtensorMap &vmap, int grid, bool pdl, cudaStream_t s)
{
#define GATTN_CASE(mt, db)                                                                         \
    if (MT == mt && DB == db)                                                                      \
        return launch_attn_t<mt, db, 0>(a, kmap, vmap, grid, pdl, s);
    GATTN_ATTN_INSTANCES(GATTN_CASE)
#undef GATTN_CASE
    return cudaErrorInvalidValue;
}

cudaError_t launch_attn_merge(int DB, int vq, const AttnArgs &a, int segments, bool pdl,
                              cudaStream_t s)
{
    // bf16 V and groups of at most 64 columns: one CTA per 64-column slice,
    // while that makes at most four CTAs per SM (beyond, the per-CTA chunk plan
    // costs more than the slices save: measured on a 32-sequence batch)
    if (vq == 0 && a.group_o <= 64 && (long long)segments * a.merge_rows * DB <= 4LL * a.attn_grid) {
        if (DB == 1)
            return launch_attn_merge_slice_t<1>(a, segments, pdl, s);
        if (DB == 2)
            return launch_attn_merge_slice_t<2>(a, segments, pdl, s);
        if (DB == 4)
            return launch_attn_merge_slice_t<4>(a, segments, pdl, s);
    }
#define GATTN_MERGE(db, v)                                                                         \
    if (DB == db && vq == v)                                                                       \
        return launch_attn_merge_t<db, v>(a, segments, pdl, s);
    GATTN_MERGE(1, 0) GATTN_MERGE(2, 0) GATTN_MERGE(4, 0)
    GATTN_MERGE(1, 1) GATTN_MERGE(2, 1) GATTN_MERGE(4, 1)
    GATTN_MERGE(1, 2) GATTN_MERGE(2, 2) GATTN_MERGE(4, 2)
#undef GATTN_MERGE
    return cudaErrorInvalidValue;
}

int attn_smem_bytes(int MT, int DB)
{
#define GATTN_CASE(mt, db)                                                                         \
    if (MT == mt && DB == db)                                                                      \
        return AttnSmem<mt, db, 0>::kTotal;
    GATTN_ATTN_INSTANCES(GATTN_CASE)
#undef GATTN_CASE
    return -1;
}

cudaError_t attn_set_smem_limits()
{
    cudaError_t e = cudaSuccess;
#define GATTN_SET(mt, db)                                                                          \
    if (e == cudaSuccess)                                                                          \
        e = cudaFuncSetAttribute(attn_kernel<mt, db, 0>,                                           \
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,                      \
                                 AttnSmem<mt, db, 0>::kTotal);
    GATTN_ATTN_INSTANCES(GATTN_SET)
#undef GATTN_SET
    return e == cudaSuccess ? attn_vq_set_smem_limits() : e;
}

}  // namespace gattn
