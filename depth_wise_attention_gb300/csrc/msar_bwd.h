// msar_bwd.h -- host interface of the kernels of the MSAR backward
// (msar_bwd.cu); the chain of steps is run by msar_expand_bwd in
// attnres_api.cu.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace attnres {

struct MsarBwdArgs {
    const unsigned char *src;       // [n_src] sources, src_stride_bytes apart, [T][d]
    int64_t src_stride_bytes;
    int n_src;
    int64_t T;
    int d;
    int k[3];                       // kernel sizes of streams 1..3
    int ktot;                       // k[0] + k[1] + k[2]
    const float *conv_w;            // packed [d][k_1] [d][k_2] [d][k_3] (per source: conv_src_stride apart)
    int64_t conv_src_stride;        // floats between sources' kernels; 0 = one set shared by all
    int64_t tc;                     // tokens per chunk of the conv backward and of A's partials
    int64_t tc_s;                   // tokens per chunk of the streams kernel
    int64_t tc_m;                   // tokens per CTA of the mixer kernels
    int nsl;                        // channel slices of the mixer (d / 1024)
    unsigned char *u;               // [3][n_src][T][d] the conv streams (source dtype)
    unsigned char *z;               // [4][T][d] the per-stream reads
    unsigned char *dz;              // [4][T][d] their gradients
    const unsigned char *dh;        // [T][d] the output gradient (nullptr in the forward's mixer)
    const float *mix_gain;          // [4d] or nullptr
    const float *mix_w;             // [4d][4]
    float mix_eps;
    float *mix_part;                // [T][nsl][9] the mixer's per-slice sums
    float *mix_e;                   // [T][4] dl_t / nu_t
    float *mix_parts;               // [chunks][4d][4] partial sums of A
    unsigned char *du;              // [4][n_src][T][d] the streams' gradients (source dtype)
    unsigned char *dsrc;            // [n_src] gradients, dsrc_stride_bytes apart
    int64_t dsrc_stride_bytes;
    float *conv_parts;              // [chunks][n_src][ktot][d] partial sums of dconv_w (tap-major)
    float *dmix_w;                  // [4d][4]
    float *dmix_gain;               // [4d] or nullptr
    // Chunked backward: src rows -hist .. -1 (and the matching dsrc rows)
    // exist before row 0; the streams read them, the kernel gradients use
    // them, and the conv transpose adds the chunk's share into their dsrc
    // rows.  acc: the parameter gradients add into their outputs.
    int64_t hist;
    int acc;
};

cudaError_t msar_bwd_streams(int dt, const MsarBwdArgs &a, void *stream);
// the forward's mixer over Z (a.z; a.dh must be nullptr): the per-slice sums
// into a.mix_part, then out[t] = sum_r c_r Z^(r)[t]
cudaError_t msar_fwd_mix(int dt, const MsarBwdArgs &a, void *out, void *stream);
// mixer backward (dz, mix_e) and the per-chunk partials of A; d a multiple
// of 1024 with nsl = d / 1024 (cudaErrorInvalidValue otherwise)
cudaError_t msar_bwd_mix(int dt, const MsarBwdArgs &a, void *stream);
// dmix_w and dmix_gain from A (added into them when a.acc)
cudaError_t msar_bwd_mix_finish(const MsarBwdArgs &a, const float *A, void *stream);
cudaError_t msar_bwd_conv(int dt, const MsarBwdArgs &a, void *stream);
// dconv_w (packed like conv_w) = the nparts conv partials at parts,
// parts + part_stride, ... (floats) summed in order (added into dconv_w when
// a.acc)
cudaError_t msar_bwd_conv_sum(const MsarBwdArgs &a, const float *parts, int64_t nparts, int64_t part_stride,
                              float *dconv_w, void *stream);
// out[e] = (accumulate ? out[e] : 0) + sum_p parts[p][e] in order of p
cudaError_t msar_bwd_sum(const float *parts, int64_t nparts, int64_t n, float *out, int accumulate, void *stream);

}  // namespace attnres
