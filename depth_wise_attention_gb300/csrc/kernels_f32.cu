// Instantiations of the single-stage depth read for float32 storage.
#include "dr_inst.cuh"

namespace attnres {
bool lookup_depth_read_f32(int nq, int vpt, bool mh, bool multi, KernelRef *out) {
    if (multi) return lookup_depth_read_f32_multi(nq, vpt, mh, out);
    ATTNRES_DR_CASE(float, 1, 1, false)
    ATTNRES_DR_CASE(float, 1, 2, false)
    ATTNRES_DR_CASE(float, 1, 4, false)
    ATTNRES_DR_CASE(float, 1, 8, false)
    ATTNRES_DR_CASE(float, 2, 1, false)
    ATTNRES_DR_CASE(float, 2, 2, false)
    ATTNRES_DR_CASE(float, 2, 4, false)
    ATTNRES_DR_CASE(float, 2, 8, false)
    ATTNRES_DR_CASE(float, 4, 1, false)
    ATTNRES_DR_CASE(float, 4, 2, false)
    ATTNRES_DR_CASE(float, 4, 4, false)
    ATTNRES_DR_CASE(float, 8, 1, false)
    ATTNRES_DR_CASE(float, 8, 2, false)
    return false;
}
}  // namespace attnres
