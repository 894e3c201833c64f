// Instantiations of the tensor-core depth read (bf16, <= 8 sources, <= 4 queries).
#include "depth_read_mma.cuh"
#include "dispatch.h"

namespace attnres {

template <int NQ, int KS>
static KernelRef dm_ref() {
    KernelRef r;
    r.fn = reinterpret_cast<const void *>(&depth_read_mma_kernel<NQ, KS>);
    r.aux_smem = DMLayout::aux_bytes;
    return r;
}

bool lookup_depth_read_mma(int nq, int ks, KernelRef *out) {
#define ATTNRES_DM_CASE(NQ, KS) \
    if (nq == NQ && ks == KS) { *out = dm_ref<NQ, KS>(); return true; }
    ATTNRES_DM_CASE(1, 8) ATTNRES_DM_CASE(1, 16) ATTNRES_DM_CASE(1, 32)
    ATTNRES_DM_CASE(2, 8) ATTNRES_DM_CASE(2, 16) ATTNRES_DM_CASE(2, 32)
    ATTNRES_DM_CASE(4, 8) ATTNRES_DM_CASE(4, 16) ATTNRES_DM_CASE(4, 32)
#undef ATTNRES_DM_CASE
    return false;
}

}  // namespace attnres
