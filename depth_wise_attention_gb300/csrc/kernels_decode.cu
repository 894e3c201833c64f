// Instantiations of the few-token depth read (depth_read_decode.cuh): up to
// 16 sources with 1 or 2 queries, 8 with 4 (more sources would not stay in
// registers).
#include "depth_read_decode.cuh"
#include "dispatch.h"

namespace attnres {

template <typename T, int NQ, int NS>
static KernelRef dec_ref() {
    KernelRef r;
    r.fn = reinterpret_cast<const void *>(&depth_read_decode_kernel<T, NQ, NS>);
    return r;
}

template <typename T>
static bool dec_lookup(int nq, int ns, KernelRef *out) {
#define ATTNRES_DEC_CASE(NQ, NS) \
    if (nq == NQ && ns == NS) { *out = dec_ref<T, NQ, NS>(); return true; }
    ATTNRES_DEC_CASE(1, 8) ATTNRES_DEC_CASE(1, 16)
    ATTNRES_DEC_CASE(2, 8) ATTNRES_DEC_CASE(2, 16) ATTNRES_DEC_CASE(4, 8)
#undef ATTNRES_DEC_CASE
    return false;
}

bool lookup_depth_read_decode(int dt, int nq, int ns, KernelRef *out) {
    return dt == 1 ? dec_lookup<__nv_bfloat16>(nq, ns, out) : dec_lookup<float>(nq, ns, out);
}

}  // namespace attnres
