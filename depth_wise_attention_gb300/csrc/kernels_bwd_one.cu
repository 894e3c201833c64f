// Instantiations of the one-kernel read backward of one query through a ring
// of half-row stages (read_bwd_one.cuh): up to 8 sources the pipelined kernel
// (2 pairs of k-steps per warp and half row at d = 2048, 4 at d = 4096), 9..16
// sources the one-barrier kernel (4 k-steps at d = 2048, 8 at d = 4096).
#include "dispatch.h"
#include "read_bwd_one.cuh"

namespace attnres {

bool lookup_read_bwd_one(int d, int n_src, KernelRef *kr) {
    const void *f = nullptr;
    if (n_src <= 8) {
        if (d == 2048) f = reinterpret_cast<const void *>(&read_bwd_one_kernel<2>);
        if (d == 4096) f = reinterpret_cast<const void *>(&read_bwd_one_kernel<4>);
    } else {
        if (d == 2048) f = reinterpret_cast<const void *>(&read_bwd_one16_kernel<4>);
        if (d == 4096) f = reinterpret_cast<const void *>(&read_bwd_one16_kernel<8>);
    }
    if (!f) return false;
    kr->fn = f;
    kr->aux_smem = n_src <= 8 ? R1_AUX_BYTES : R16_AUX_BYTES;
    return true;
}

}  // namespace attnres
