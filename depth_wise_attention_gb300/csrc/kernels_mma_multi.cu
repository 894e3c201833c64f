// Instantiations of the chunked tensor-core depth read (bf16, > 8 sources,
// <= 4 queries, d = 4096: 16 warps x 256 channels).
#include "depth_read_mma.cuh"
#include "dispatch.h"

namespace attnres {

template <int NQ, int KS, int NW>
static KernelRef dmm_ref() {
    KernelRef r;
    r.fn = reinterpret_cast<const void *>(&depth_read_mma_multi_kernel<NQ, KS, NW>);
    r.aux_smem = DMLayout::aux_bytes;
    return r;
}

bool lookup_depth_read_mma_multi(int nq, int ks, int nw, KernelRef *out) {
#define ATTNRES_DMM_CASE(NQ, KS, NW) \
    if (nq == NQ && ks == KS && nw == NW) { *out = dmm_ref<NQ, KS, NW>(); return true; }
    ATTNRES_DMM_CASE(1, 16, 16) ATTNRES_DMM_CASE(2, 16, 16) ATTNRES_DMM_CASE(4, 16, 16)
#undef ATTNRES_DMM_CASE
    return false;
}

}  // namespace attnres
