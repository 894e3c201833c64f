// msar.h -- host interface of the fused MSAR kernel (internal to libattnres).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/attnres.h"
#include "common.cuh"

namespace attnres {

constexpr int MSAR_KMAX = 16;      // largest supported conv kernel
constexpr int MSAR_SMAX = 8;       // most sources per read
constexpr int MSAR_RING = 16;      // token rows kept per source in shared memory
constexpr int MSAR_M = 4;          // streams (identity + 3 convolutions)

struct MsarArgs {
    const unsigned char *src;
    int64_t src_stride_bytes;
    int n_src;
    int64_t T;                 // output tokens
    int64_t t_prev;            // history rows before the first output token: token t is src row t + t_prev
    int d;
    int k[3];                  // conv kernel sizes of streams 1..3
    const float *conv_w;       // packed [d][k_1] [d][k_2] [d][k_3]
    const float *queries;      // [4][d]
    const float *gain;         // [d] or nullptr
    float eps;
    const float *mix_gain;     // [4d] or nullptr
    const float *mix_w;        // [4d][4]
    float mix_eps;
    unsigned char *out;        // [T][d]
    WaitCfg wait;
    // launch shape (filled by launch_msar)
    int cluster;               // CTAs per cluster (channel slices)
    int ch;                    // channels per CTA
    int64_t tokens_per_cluster;
    int nclusters;
};

// Validated arguments in, launch out.  dt: 0 = f32, 1 = bf16.
attnres_status_t launch_msar(int dt, MsarArgs a, int sms, void *stream, char *err, size_t errlen);

}  // namespace attnres
