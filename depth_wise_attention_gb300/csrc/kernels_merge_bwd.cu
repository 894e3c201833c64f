// Instantiations of the backward of the Block phase-2 merge (merge_bwd.cuh).
#include "dispatch.h"
#include "merge_bwd.cuh"

namespace attnres {

template <typename T, int VPT>
static KernelRef mb_ref() {
    KernelRef r;
    r.fn = reinterpret_cast<const void *>(&merge_bwd_kernel<T, VPT>);
    r.aux_smem = 0;
    return r;
}

template <typename T>
static bool mb_lookup(int vpt, KernelRef *out) {
    switch (vpt) {
        case 1: *out = mb_ref<T, 1>(); return true;
        case 2: *out = mb_ref<T, 2>(); return true;
        case 4: *out = mb_ref<T, 4>(); return true;
    }
    return false;
}

bool lookup_merge_bwd(int dt, int vpt, KernelRef *out) {
    return dt == 1 ? mb_lookup<__nv_bfloat16>(vpt, out) : mb_lookup<float>(vpt, out);
}

}  // namespace attnres
