// state_merge_bwd.h -- host interface of the merge backward of chunk read
// states (state_merge_bwd.cu), used by the read backward over more than 16
// sources.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace attnres {

struct StateMergeBwdArgs {
    const unsigned char *o;           // [C][n_q][T][d] dtype: the chunks' read outputs
    const float *lse;                 // [C][n_q][T]
    const unsigned char *dh;          // [n_q][T][d] dtype
    const float *dlse;                // [n_q][T] or nullptr
    unsigned char *d_o;               // [C][n_q][T][d] dtype
    float *d_lse;                     // [C][n_q][T]
    int C;                            // chunks, 1..32
    int64_t rows;                     // n_q * T
    int d;                            // a multiple of 8 (bf16) or 4 (f32)
};

// dt: 0 = f32, 1 = bf16
cudaError_t launch_state_merge_bwd(int dt, const StateMergeBwdArgs &a, int sms, void *stream);

}  // namespace attnres
