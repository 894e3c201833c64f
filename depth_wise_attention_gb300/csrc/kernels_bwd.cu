// Instantiations of the backward of the depth read (read_bwd.cuh): up to 8
// sources with 1 or 2 queries, up to 16 sources with 1 query.
#include "dispatch.h"
#include "read_bwd.cuh"

namespace attnres {

// 256 threads: 32 channels times 8 groups of partials (group j takes
// partials j, j+8, ...); the groups are then added in order, so the result
// does not depend on scheduling.
__global__ void __launch_bounds__(256) read_bwd_finish_kernel(const ReadBwdFinishArgs a) {
    __shared__ float red[8][32];
    const int lane = threadIdx.x & 31, j = threadIdx.x >> 5;
    const int c = blockIdx.x * 32 + lane;
    const bool ok = c < a.d;
    const float g = ok && a.gain ? __ldg(a.gain + c) : 1.f;
    float dgc = 0.f;
    for (int q = 0; q < a.n_q; ++q) {
        float u = 0.f;
        if (ok)
            for (int p = j; p < a.nparts; p += 8) u += a.ws[((size_t)p * a.n_q + q) * a.d + c];
        red[j][lane] = u;
        __syncthreads();
        if (j == 0 && ok) {
            float s = 0.f;
#pragma unroll
            for (int k = 0; k < 8; ++k) s += red[k][lane];
            a.dq[(size_t)q * a.d + c] = g * s;
            dgc = fmaf(__ldg(a.queries + (size_t)q * a.d + c), s, dgc);
        }
        __syncthreads();
    }
    if (j == 0 && ok && a.dgain) a.dgain[c] = a.accumulate_dgain ? a.dgain[c] + dgc : dgc;
}

template <typename T, int NQ, int NS, int VPT>
static KernelRef rb_ref() {
    KernelRef r;
    r.fn = reinterpret_cast<const void *>(&read_bwd_kernel<T, NQ, NS, VPT>);
    r.aux_smem = RBLayout<NQ, NS>::aux_bytes;
    return r;
}

template <typename T, int NQ, int NS>
static bool rb_vpt(int vpt, KernelRef *out) {
    switch (vpt) {
        case 1: *out = rb_ref<T, NQ, NS, 1>(); return true;
        case 2: *out = rb_ref<T, NQ, NS, 2>(); return true;
        case 4: *out = rb_ref<T, NQ, NS, 4>(); return true;
    }
    return false;
}

template <typename T>
static bool rb_lookup(int nq, int ns, int vpt, KernelRef *out) {
    if (nq == 1 && ns == 8) return rb_vpt<T, 1, 8>(vpt, out);
    if (nq == 2 && ns == 8) return rb_vpt<T, 2, 8>(vpt, out);
    if (nq == 1 && ns == 16) return rb_vpt<T, 1, 16>(vpt, out);
    return false;
}

bool lookup_read_bwd(int dt, int nq, int ns, int vpt, KernelRef *out) {
    return dt == 1 ? rb_lookup<__nv_bfloat16>(nq, ns, vpt, out) : rb_lookup<float>(nq, ns, vpt, out);
}

const void *read_bwd_finish_fn() { return reinterpret_cast<const void *>(&read_bwd_finish_kernel); }

}  // namespace attnres
