// Instantiations of the per-head backward (the backward of the MHAR read,
// read_bwd.cuh in per-head mode).  HG == 1: a warp's runs lie in one head;
// HG == VPT: each run of 32 vectors is its own group (heads of 32 vectors or
// a multiple of 32 that is not a multiple of 32 * VPT).
#include "dispatch.h"
#include "read_bwd.cuh"

namespace attnres {

template <typename T, int NQ, int NS, int VPT, int HG>
static KernelRef rbh_ref() {
    KernelRef r;
    r.fn = reinterpret_cast<const void *>(&read_bwd_kernel<T, NQ, NS, VPT, true, HG>);
    r.aux_smem = RBLayout<NQ, NS, HG>::aux_bytes;
    return r;
}

template <typename T>
static bool rbh_lookup(int nq, int ns, int vpt, int hg, KernelRef *out) {
#define ATTNRES_RBH_CASE(NQ, NS, VPT, HG) \
    if (nq == NQ && ns == NS && vpt == VPT && hg == HG) { *out = rbh_ref<T, NQ, NS, VPT, HG>(); return true; }
    ATTNRES_RBH_CASE(1, 8, 1, 1) ATTNRES_RBH_CASE(1, 8, 2, 1) ATTNRES_RBH_CASE(1, 8, 2, 2)
    ATTNRES_RBH_CASE(1, 8, 4, 1) ATTNRES_RBH_CASE(1, 8, 4, 4)
    ATTNRES_RBH_CASE(2, 8, 1, 1) ATTNRES_RBH_CASE(2, 8, 2, 1) ATTNRES_RBH_CASE(2, 8, 2, 2)
    ATTNRES_RBH_CASE(2, 8, 4, 1)
    ATTNRES_RBH_CASE(1, 16, 1, 1) ATTNRES_RBH_CASE(1, 16, 2, 1) ATTNRES_RBH_CASE(1, 16, 2, 2)
    ATTNRES_RBH_CASE(1, 16, 4, 1)
#undef ATTNRES_RBH_CASE
    return false;
}

bool lookup_read_bwd_mh(int dt, int nq, int ns, int vpt, int hg, KernelRef *out) {
    return dt == 1 ? rbh_lookup<__nv_bfloat16>(nq, ns, vpt, hg, out) : rbh_lookup<float>(nq, ns, vpt, hg, out);
}

}  // namespace attnres
