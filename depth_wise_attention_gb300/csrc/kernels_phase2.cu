// Instantiations of the phase-2 merge kernel.
#include "dispatch.h"
#include "phase2.cuh"

namespace attnres {

template <typename T, int VPT>
static KernelRef p2_ref() {
    KernelRef r;
    r.fn = reinterpret_cast<const void *>(&phase2_merge_kernel<T, VPT>);
    return r;
}

bool lookup_phase2(int dt, int vpt, KernelRef *out) {
    if (dt == 1) {
        switch (vpt) {
            case 1: *out = p2_ref<__nv_bfloat16, 1>(); return true;
            case 2: *out = p2_ref<__nv_bfloat16, 2>(); return true;
            case 4: *out = p2_ref<__nv_bfloat16, 4>(); return true;
            case 8: *out = p2_ref<__nv_bfloat16, 8>(); return true;
        }
    } else {
        switch (vpt) {
            case 1: *out = p2_ref<float, 1>(); return true;
            case 2: *out = p2_ref<float, 2>(); return true;
            case 4: *out = p2_ref<float, 4>(); return true;
            case 8: *out = p2_ref<float, 8>(); return true;
        }
    }
    return false;
}

bool lookup_depth_read(int dt, int nq, int vpt, bool mh, bool multi, KernelRef *out) {
    return dt == 1 ? lookup_depth_read_bf16(nq, vpt, mh, multi, out)
                   : lookup_depth_read_f32(nq, vpt, mh, multi, out);
}

}  // namespace attnres
