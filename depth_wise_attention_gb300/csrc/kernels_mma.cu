// Instantiations of the tensor-core depth read (bf16, <= 8 sources, <= 4 queries).
#include "depth_read_mma.cuh"
#include "dispatch.h"

namespace attnres {

template <int NQ, int KS, int NW>
static KernelRef dm_ref() {
    KernelRef r;
    r.fn = reinterpret_cast<const void *>(&depth_read_mma_kernel<NQ, KS, NW>);
    r.aux_smem = DMLayout::aux_bytes;
    return r;
}

template <int NQ, int KS, int NW>
static KernelRef dm2_ref() {
    KernelRef r;
    r.fn = reinterpret_cast<const void *>(&depth_read_mma2_kernel<NQ, KS, NW>);
    r.aux_smem = DMLayout::aux_bytes;
    return r;
}

bool lookup_depth_read_mma2(int nq, int ks, int nw, KernelRef *out) {
#define ATTNRES_DM2_CASE(NQ, KS, NW) \
    if (nq == NQ && ks == KS && nw == NW) { *out = dm2_ref<NQ, KS, NW>(); return true; }
    // d = 1024: 8 warps x 128 channels
    ATTNRES_DM2_CASE(1, 8, 8) ATTNRES_DM2_CASE(2, 8, 8) ATTNRES_DM2_CASE(4, 8, 8)
#undef ATTNRES_DM2_CASE
    return false;
}

bool lookup_depth_read_mma(int nq, int ks, int nw, KernelRef *out) {
#define ATTNRES_DM_CASE(NQ, KS, NW) \
    if (nq == NQ && ks == KS && nw == NW) { *out = dm_ref<NQ, KS, NW>(); return true; }
    // d = 4096: 16 warps x 256 channels, one CTA per SM; d = 2048: 8 warps x 256
    // channels, two CTAs per SM (d = 1024 uses the two-token kernel)
    ATTNRES_DM_CASE(1, 16, 16) ATTNRES_DM_CASE(2, 16, 16) ATTNRES_DM_CASE(4, 16, 16)
    ATTNRES_DM_CASE(1, 16, 8) ATTNRES_DM_CASE(2, 16, 8) ATTNRES_DM_CASE(4, 16, 8)
#undef ATTNRES_DM_CASE
    return false;
}

}  // namespace attnres
