// Instantiations of the phase-2 merge kernel (one head; with and without the
// fused partial-sum update).
#include "dispatch.h"
#include "phase2.cuh"

namespace attnres {

template <typename T, int VPT, bool UPD>
static KernelRef p2_ref() {
    KernelRef r;
    r.fn = reinterpret_cast<const void *>(&phase2_merge_kernel<T, VPT, UPD, false>);
    return r;
}

template <typename T, bool UPD>
static bool p2_lookup(int vpt, KernelRef *out) {
    switch (vpt) {
        case 1: *out = p2_ref<T, 1, UPD>(); return true;
        case 2: *out = p2_ref<T, 2, UPD>(); return true;
        case 4: *out = p2_ref<T, 4, UPD>(); return true;
        case 8: *out = p2_ref<T, 8, UPD>(); return true;
    }
    return false;
}

bool lookup_phase2(int dt, int vpt, bool upd, bool mh, KernelRef *out) {
    if (mh) return lookup_phase2_mh(dt, vpt, upd, out);
    if (dt == 1) return upd ? p2_lookup<__nv_bfloat16, true>(vpt, out) : p2_lookup<__nv_bfloat16, false>(vpt, out);
    return upd ? p2_lookup<float, true>(vpt, out) : p2_lookup<float, false>(vpt, out);
}

bool lookup_depth_read(int dt, int nq, int vpt, bool mh, bool multi, KernelRef *out) {
    return dt == 1 ? lookup_depth_read_bf16(nq, vpt, mh, multi, out)
                   : lookup_depth_read_f32(nq, vpt, mh, multi, out);
}

}  // namespace attnres
