// Instantiations of the per-head (MHAR) phase-2 merge kernel, with and
// without the fused partial-sum update.
#include "dispatch.h"
#include "phase2.cuh"

namespace attnres {

template <typename T, int VPT, bool UPD>
static KernelRef p2mh_ref() {
    KernelRef r;
    r.fn = reinterpret_cast<const void *>(&phase2_merge_kernel<T, VPT, UPD, true>);
    return r;
}

template <typename T, bool UPD>
static bool p2mh_lookup(int vpt, KernelRef *out) {
    switch (vpt) {
        case 1: *out = p2mh_ref<T, 1, UPD>(); return true;
        case 2: *out = p2mh_ref<T, 2, UPD>(); return true;
        case 4: *out = p2mh_ref<T, 4, UPD>(); return true;
        case 8: *out = p2mh_ref<T, 8, UPD>(); return true;
    }
    return false;
}

bool lookup_phase2_mh(int dt, int vpt, bool upd, KernelRef *out) {
    if (dt == 1) return upd ? p2mh_lookup<__nv_bfloat16, true>(vpt, out) : p2mh_lookup<__nv_bfloat16, false>(vpt, out);
    return upd ? p2mh_lookup<float, true>(vpt, out) : p2mh_lookup<float, false>(vpt, out);
}

}  // namespace attnres
