// Instantiations of the chunked (online-softmax) depth read for float32.
#include "dr_inst.cuh"

namespace attnres {
bool lookup_depth_read_f32_multi(int nq, int vpt, bool mh, KernelRef *out) {
    ATTNRES_DR_CASE(float, 1, 1, true)
    ATTNRES_DR_CASE(float, 1, 2, true)
    ATTNRES_DR_CASE(float, 1, 4, true)
    ATTNRES_DR_CASE(float, 1, 8, true)
    ATTNRES_DR_CASE(float, 2, 1, true)
    ATTNRES_DR_CASE(float, 2, 2, true)
    ATTNRES_DR_CASE(float, 2, 4, true)
    ATTNRES_DR_CASE(float, 2, 8, true)
    ATTNRES_DR_CASE(float, 4, 1, true)
    ATTNRES_DR_CASE(float, 4, 2, true)
    ATTNRES_DR_CASE(float, 4, 4, true)
    ATTNRES_DR_CASE(float, 8, 1, true)
    ATTNRES_DR_CASE(float, 8, 2, true)
    return false;
}
}  // namespace attnres
