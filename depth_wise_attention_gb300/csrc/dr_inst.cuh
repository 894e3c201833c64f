// dr_inst.cuh -- helpers to instantiate depth_read_kernel for one storage type.
#pragma once

#include "depth_read.cuh"
#include "dispatch.h"

namespace attnres {

template <typename Tin, int NQ, int VPT, bool MH, bool MULTI>
inline KernelRef dr_ref() {
    KernelRef r;
    r.fn = reinterpret_cast<const void *>(&depth_read_kernel<Tin, NQ, VPT, MH, MULTI>);
    r.aux_smem = DRLayout<NQ, VPT, MH>::aux_bytes;
    return r;
}

// (NQ, VPT) pairs whose register footprint fits: NQ * VPT * EPV <= 64.
#define ATTNRES_DR_CASE(T, NQ, VPT, MULTI)                                   \
    if (nq == NQ && vpt == VPT) {                                              \
        *out = mh ? dr_ref<T, NQ, VPT, true, MULTI>() : dr_ref<T, NQ, VPT, false, MULTI>(); \
        return true;                                                           \
    }

}  // namespace attnres
