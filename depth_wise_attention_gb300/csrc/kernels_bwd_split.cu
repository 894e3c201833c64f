// Instantiations of the two-kernel read backward: 3 or 4 queries
// (read_bwd_split.cuh; 4 k-steps per warp and half row at d = 2048, 8 at
// 4096), and one query over 17..64 sources (read_bwd_many.cuh).
#include "dispatch.h"
#include "read_bwd_split.cuh"
#include "read_bwd_many.cuh"

namespace attnres {

bool lookup_read_bwd_split(int nq, int d, KernelRef *coef, KernelRef *apply) {
    const int ksh = d / (2 * 16 * RC_NW);
    const void *c = nullptr, *p = nullptr;
    if (nq == 3 && ksh == 4) c = reinterpret_cast<const void *>(&read_bwd_coef_kernel<3, 4>);
    if (nq == 3 && ksh == 8) c = reinterpret_cast<const void *>(&read_bwd_coef_kernel<3, 8>);
    if (nq == 4 && ksh == 4) c = reinterpret_cast<const void *>(&read_bwd_coef_kernel<4, 4>);
    if (nq == 4 && ksh == 8) c = reinterpret_cast<const void *>(&read_bwd_coef_kernel<4, 8>);
    if (nq == 3) p = reinterpret_cast<const void *>(&read_bwd_apply_kernel<3>);
    if (nq == 4) p = reinterpret_cast<const void *>(&read_bwd_apply_kernel<4>);
    if (!c || !p) return false;
    coef->fn = c;
    coef->aux_smem = RC_AUX_BYTES;
    apply->fn = p;
    apply->aux_smem = 0;
    return true;
}

bool lookup_read_bwd_many(int d, KernelRef *coef, KernelRef *apply) {
    const void *c = nullptr;
    if (d == 2048) c = reinterpret_cast<const void *>(&read_bwd_coef_many_kernel<2>);
    if (d == 4096) c = reinterpret_cast<const void *>(&read_bwd_coef_many_kernel<4>);
    if (!c) return false;
    coef->fn = c;
    coef->aux_smem = RM_AUX_BYTES;
    apply->fn = reinterpret_cast<const void *>(&read_bwd_apply_many_kernel<1>);
    apply->aux_smem = 0;
    return true;
}

}  // namespace attnres
