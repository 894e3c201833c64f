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
    int64_t conv_src_stride;   // floats between sources' packed kernels; 0: all sources share conv_w
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

constexpr int MSAR_P1_MAXL = 4;    // most layers read together by msar_phase1_kernel

// Phase 1 of MSAR in the two-phase Block schedule (msar_phase1.cu).
struct MsarP1Args {
    const unsigned char *src;
    int64_t src_stride_bytes;
    int n_src;
    int64_t T;
    int d;
    int k[3];
    const float *conv_w;
    const float *queries;      // [n_layers][4][d]
    int n_layers;
    const float *gain;
    float eps;
    unsigned char *o;          // [n_layers][4][T][d]
    float *lse;                // [n_layers][4][T]
    WaitCfg wait;
    int cluster;
    int ch;
    int64_t tokens_per_cluster;
};

attnres_status_t launch_msar_phase1(int dt, MsarP1Args a, int sms, void *stream, char *err, size_t errlen);

// Phase 2 of MSAR in the two-phase Block schedule (msar_phase2.cu).
struct MsarP2Args {
    const unsigned char *o;          // [4][T][d] phase-1 state of the layer
    const float *lse;                // [4][T]
    const unsigned char *partial;    // [T][d] or nullptr
    int64_t T;
    int d;
    int k[3];
    const float *conv_w;
    const float *query;              // [4][d]
    const float *gain;
    float eps;
    const float *mix_gain;
    const float *mix_w;
    float mix_eps;
    unsigned char *out;              // [T][d]
    WaitCfg wait;
    int tt;                          // tokens per CTA (set by the launcher)
};

attnres_status_t launch_msar_phase2(int dt, MsarP2Args a, int sms, void *stream, char *err, size_t errlen);

// Two adjacent channels of a row, widened to fp32 / rounded back.
template <typename Tin> struct Pair2;
template <> struct Pair2<__nv_bfloat16> {
    __device__ static __forceinline__ float2 ld(const unsigned char *p) {
        return bf2_to_f2(*reinterpret_cast<const uint32_t *>(p));
    }
    __device__ static __forceinline__ void st(unsigned char *p, float2 v) {
        *reinterpret_cast<uint32_t *>(p) = f2_to_bf2(v.x, v.y);
    }
};
template <> struct Pair2<float> {
    __device__ static __forceinline__ float2 ld(const unsigned char *p) {
        return *reinterpret_cast<const float2 *>(p);
    }
    __device__ static __forceinline__ void st(unsigned char *p, float2 v) {
        *reinterpret_cast<float2 *>(p) = v;
    }
};

__device__ __forceinline__ float dot2(float2 a, float2 b) { return fmaf(a.x, b.x, a.y * b.y); }

// Validated arguments in, launch out.  dt: 0 = f32, 1 = bf16.
attnres_status_t launch_msar(int dt, MsarArgs a, int sms, void *stream, char *err, size_t errlen);

// The tile-batched fused read (msar_tile.cu): bf16 sources, kernel sizes
// 4/8/12 shared by all sources, d a multiple of 256 up to 4096.  Returns
// ATTNRES_ERR_UNSUPPORTED when no cluster of it can be resident.
bool msar_tile_applies(int dt, const MsarArgs &a);
attnres_status_t launch_msar_tile(MsarArgs a, int sms, void *stream, char *err, size_t errlen);

}  // namespace attnres
