// The decode attention's instances with the in-launch merges compiled in: the cluster merge
// (pieces of a (session, KV head) merged through distributed shared memory) and the merge by the
// last piece (daScript PR #4293, "The decode attention's split follows the command's rows, not
// the planes' height", merge of the split partials).  They sit in a translation unit of their
// own so that the default instances carry none of that code and both units compile in parallel.
#include "decode_attn_kernel.cuh"

namespace {

template <int D, int EB>
const void *pick_merge_opts(bool mma, int qm)
{
    if (mma) return reinterpret_cast<const void *>(decode_attn_tma_kernel<D, true, 8, EB, true>);
    return qm == 4 ? reinterpret_cast<const void *>(decode_attn_tma_kernel<D, false, 4, EB, true>)
         : qm == 6 ? reinterpret_cast<const void *>(decode_attn_tma_kernel<D, false, 6, EB, true>)
                   : reinterpret_cast<const void *>(decode_attn_tma_kernel<D, false, 8, EB, true>);
}

}  // namespace

namespace dl {

// The instance for a head dimension (64 or 128), mirror element size (1, 2 or 4 bytes), form and
// CUDA-core queries per warp; null for a head dimension without instances.
const void *attn_kernel_merge_opts(int head_dim, int eb, bool mma, int qm)
{
    if (head_dim != 128 && head_dim != 64) return nullptr;
    const bool d128 = head_dim == 128;
    return eb == 4 ? (d128 ? pick_merge_opts<128, 4>(mma, qm) : pick_merge_opts<64, 4>(mma, qm))
         : eb == 1 ? (d128 ? pick_merge_opts<128, 1>(mma, qm) : pick_merge_opts<64, 1>(mma, qm))
                   : (d128 ? pick_merge_opts<128, 2>(mma, qm) : pick_merge_opts<64, 2>(mma, qm));
}

}  // namespace dl
