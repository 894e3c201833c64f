// Instantiations of the single-stage depth read for bfloat16 storage.
#include "dr_inst.cuh"

namespace attnres {
bool lookup_depth_read_bf16(int nq, int vpt, bool mh, bool multi, KernelRef *out) {
    if (multi) return lookup_depth_read_bf16_multi(nq, vpt, mh, out);
    ATTNRES_DR_CASE(__nv_bfloat16, 1, 1, false)
    ATTNRES_DR_CASE(__nv_bfloat16, 1, 2, false)
    ATTNRES_DR_CASE(__nv_bfloat16, 1, 4, false)
    ATTNRES_DR_CASE(__nv_bfloat16, 1, 8, false)
    ATTNRES_DR_CASE(__nv_bfloat16, 2, 1, false)
    ATTNRES_DR_CASE(__nv_bfloat16, 2, 2, false)
    ATTNRES_DR_CASE(__nv_bfloat16, 2, 4, false)
    ATTNRES_DR_CASE(__nv_bfloat16, 4, 1, false)
    ATTNRES_DR_CASE(__nv_bfloat16, 4, 2, false)
    ATTNRES_DR_CASE(__nv_bfloat16, 8, 1, false)
    return false;
}
}  // namespace attnres
