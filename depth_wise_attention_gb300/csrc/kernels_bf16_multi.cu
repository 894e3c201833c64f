// Instantiations of the chunked (online-softmax) depth read for bfloat16.
#include "dr_inst.cuh"

namespace attnres {
bool lookup_depth_read_bf16_multi(int nq, int vpt, bool mh, KernelRef *out) {
    ATTNRES_DR_CASE(__nv_bfloat16, 1, 1, true)
    ATTNRES_DR_CASE(__nv_bfloat16, 1, 2, true)
    ATTNRES_DR_CASE(__nv_bfloat16, 1, 4, true)
    ATTNRES_DR_CASE(__nv_bfloat16, 1, 8, true)
    ATTNRES_DR_CASE(__nv_bfloat16, 2, 1, true)
    ATTNRES_DR_CASE(__nv_bfloat16, 2, 2, true)
    ATTNRES_DR_CASE(__nv_bfloat16, 2, 4, true)
    ATTNRES_DR_CASE(__nv_bfloat16, 4, 1, true)
    ATTNRES_DR_CASE(__nv_bfloat16, 4, 2, true)
    ATTNRES_DR_CASE(__nv_bfloat16, 8, 1, true)
    return false;
}
}  // namespace attnres
