// dispatch.h -- host-side lookup of the kernel instantiations compiled in the
// per-type translation units (kernels_*.cu).  Internal to libattnres.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>

namespace attnres {

struct KernelRef {
    const void *fn = nullptr;   // __global__ function
    size_t aux_smem = 0;        // shared memory besides the stages (bytes)
};

// depth_read_kernel<T, nq, vpt, mh, multi>; dt: 0 = f32, 1 = bf16.
// Returns false if that instantiation is not compiled.
bool lookup_depth_read(int dt, int nq, int vpt, bool mh, bool multi, KernelRef *out);
bool lookup_depth_read_f32(int nq, int vpt, bool mh, bool multi, KernelRef *out);
bool lookup_depth_read_bf16(int nq, int vpt, bool mh, bool multi, KernelRef *out);
bool lookup_depth_read_bf16_multi(int nq, int vpt, bool mh, KernelRef *out);
bool lookup_depth_read_f32_multi(int nq, int vpt, bool mh, KernelRef *out);

// depth_read_mma_kernel<nq, ks, nw> (bf16 only; nw warps of 16*ks channels, d = 16*ks*nw)
bool lookup_depth_read_mma(int nq, int ks, int nw, KernelRef *out);
// depth_read_mma2_kernel<nq, ks, nw>: two tokens per item (d = 1024, 2048)
bool lookup_depth_read_mma2(int nq, int ks, int nw, KernelRef *out);
// depth_read_mma_multi_kernel<nq, ks, nw>: > 8 sources in chunks of 8 (online softmax)
bool lookup_depth_read_mma_multi(int nq, int ks, int nw, KernelRef *out);

// depth_read_decode_kernel<T, nq, ns>: one token per cluster of CTAs (few tokens)
bool lookup_depth_read_decode(int dt, int nq, int ns, KernelRef *out);

// read_bwd_kernel<T, nq, ns, vpt> (nq queries, at most ns sources) and the
// workspace reduction kernel that finishes dq and dgain
bool lookup_read_bwd(int dt, int nq, int ns, int vpt, KernelRef *out);
// read_bwd_kernel with two query groups of two (up to 4 queries, <= 8 sources) per launch
bool lookup_read_bwd_qg(int dt, int vpt, bool mh, int hg, KernelRef *out);
// merge_bwd_kernel<T, vpt>: backward of the Block phase-2 merge
bool lookup_merge_bwd(int dt, int vpt, KernelRef *out);
// read_bwd_kernel in per-head mode (MHAR backward), hg reduction groups per warp
bool lookup_read_bwd_mh(int dt, int nq, int ns, int vpt, int hg, KernelRef *out);
const void *read_bwd_finish_fn();
// the two-kernel read backward (read_bwd_split.cuh): read_bwd_coef_kernel and
// read_bwd_apply_kernel for nq = 3 or 4 queries at d = 2048 or 4096
bool lookup_read_bwd_split(int nq, int d, KernelRef *coef, KernelRef *apply);
// its form for one query over 17..64 sources (read_bwd_many.cuh)
bool lookup_read_bwd_many(int d, KernelRef *coef, KernelRef *apply);
// One query over at most 16 bf16 sources in one kernel, d = 2048 or 4096
// (the pipelined kernel up to 8 sources, the one-barrier kernel above).
bool lookup_read_bwd_one(int d, int n_src, KernelRef *kr);

// phase2_merge_kernel<T, vpt, upd, mh>: upd = fused partial-sum update, mh = per-head merge
bool lookup_phase2(int dt, int vpt, bool upd, bool mh, KernelRef *out);
bool lookup_phase2_mh(int dt, int vpt, bool upd, KernelRef *out);

}  // namespace attnres
