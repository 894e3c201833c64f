// Instantiations of the backward of the read with two query groups per launch
// (read_bwd.cuh, QG = 2): up to 4 queries over up to 8 sources in one pass
// over the sources, plain or per head.
#include "dispatch.h"
#include "read_bwd.cuh"

namespace attnres {

template <typename T, int VPT, bool MH, int HG>
static KernelRef rbq_ref() {
    KernelRef r;
    r.fn = reinterpret_cast<const void *>(&read_bwd_kernel<T, 2, 8, VPT, MH, HG, 2>);
    r.aux_smem = RBLayout<2, 8, HG>::aux_bytes;
    return r;
}

#define ATTNRES_RBQ_CASE(T, VPT, MH, HG) \
    if (vpt == VPT && mh == MH && hg == HG) { *out = rbq_ref<T, VPT, MH, HG>(); return true; }

// bf16 with 4 vectors a thread, or with one reduction group per run of a
// warp, keeps one query group per launch (two groups spill registers there)
static bool rbq_lookup_bf16(int vpt, bool mh, int hg, KernelRef *out) {
    ATTNRES_RBQ_CASE(__nv_bfloat16, 1, false, 1) ATTNRES_RBQ_CASE(__nv_bfloat16, 2, false, 1)
    ATTNRES_RBQ_CASE(__nv_bfloat16, 1, true, 1) ATTNRES_RBQ_CASE(__nv_bfloat16, 2, true, 1)
    return false;
}

static bool rbq_lookup_f32(int vpt, bool mh, int hg, KernelRef *out) {
    ATTNRES_RBQ_CASE(float, 1, false, 1) ATTNRES_RBQ_CASE(float, 2, false, 1) ATTNRES_RBQ_CASE(float, 4, false, 1)
    ATTNRES_RBQ_CASE(float, 1, true, 1) ATTNRES_RBQ_CASE(float, 2, true, 1) ATTNRES_RBQ_CASE(float, 2, true, 2)
    ATTNRES_RBQ_CASE(float, 4, true, 1)
    return false;
}
#undef ATTNRES_RBQ_CASE

bool lookup_read_bwd_qg(int dt, int vpt, bool mh, int hg, KernelRef *out) {
    return dt == 1 ? rbq_lookup_bf16(vpt, mh, hg, out) : rbq_lookup_f32(vpt, mh, hg, out);
}

}  // namespace attnres
