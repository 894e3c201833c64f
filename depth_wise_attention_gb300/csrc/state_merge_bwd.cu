// state_merge_bwd.cu -- backward of merging the read states of source chunks
// (sm_103a), used by the read backward for more sources than one pass of
// read_bwd_kernel takes.
//
// The sources are read in chunks c = 0..C-1; chunk c's read gives the state
// (o_c, lse_c) with o_c = sum_{i in c} alpha^c_i v_i and lse_c the
// log-sum-exp of its scores.  The whole read is their online-softmax merge:
//     LSE = log sum_c exp(lse_c),  beta_c = exp(lse_c - LSE),
//     h = sum_c beta_c o_c,        lse = LSE.
// For the gradients dh of h and dLSE of LSE (0 when only h is used):
//     d o_c   = beta_c dh
//     d lse_c = beta_c (dh . o_c - dh . h + dLSE),
// and dh . h = sum_c beta_c (dh . o_c).  Each chunk's backward is then the
// read backward with an lse gradient (attnres_block_phase1_bwd).
//
// One CTA per (query, token) row: every thread holds 16-byte vectors of dh,
// forms its partial dh . o_c for every chunk, the CTA sums them, and the
// threads write their vectors of beta_c dh.
#include "common.cuh"
#include "state_merge_bwd.h"

namespace attnres {

constexpr int SMB_THREADS = 256;
constexpr int SMB_MAXC = 32;          // most chunks

template <typename Tin>
__global__ void __launch_bounds__(SMB_THREADS) state_merge_bwd_kernel(const StateMergeBwdArgs a) {
    using E = Elem<Tin>;
    constexpr int EPV = E::EPV;
    constexpr int NP = EPV / 2;                      // float2 pairs per 16-byte vector
    __shared__ float red[SMB_THREADS / 32][SMB_MAXC];
    __shared__ float tot[SMB_MAXC];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nvec = a.d / EPV;
    const int64_t cstride = a.rows * (int64_t)a.d * (int64_t)sizeof(Tin);   // bytes between chunks' tensors
    for (int64_t row = blockIdx.x; row < a.rows; row += gridDim.x) {
        // beta_c from the chunks' log-sum-exps (every thread, same order)
        float mx = -INFINITY;
        for (int c = 0; c < a.C; ++c) mx = fmaxf(mx, a.lse[(int64_t)c * a.rows + row]);
        float den = 0.f;
        for (int c = 0; c < a.C; ++c) den += __expf(a.lse[(int64_t)c * a.rows + row] - mx);
        const float inv = 1.f / den;
        // partial dh . o_c over this thread's vectors
        float dot[SMB_MAXC];
#pragma unroll
        for (int c = 0; c < SMB_MAXC; ++c) dot[c] = 0.f;
        const unsigned char *dhr = a.dh + row * (int64_t)a.d * sizeof(Tin);
        const unsigned char *orow = a.o + row * (int64_t)a.d * sizeof(Tin);
        for (int v = tid; v < nvec; v += SMB_THREADS) {
            float2 g[NP];
            E::unpack(*reinterpret_cast<const uint4 *>(dhr + (int64_t)v * 16), g);
#pragma unroll
            for (int c = 0; c < SMB_MAXC; ++c) {
                if (c >= a.C) break;
                float2 x[NP];
                E::unpack(*reinterpret_cast<const uint4 *>(orow + c * cstride + (int64_t)v * 16), x);
#pragma unroll
                for (int p = 0; p < NP; ++p) dot[c] = fmaf(g[p].x, x[p].x, fmaf(g[p].y, x[p].y, dot[c]));
            }
        }
        // sum over the CTA: warp shuffles, then the warps in order
#pragma unroll
        for (int c = 0; c < SMB_MAXC; ++c) {
            if (c >= a.C) break;
            float s = dot[c];
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
            if (lane == 0) red[warp][c] = s;
        }
        __syncthreads();
        if (tid < a.C) {
            float s = 0.f;
            for (int w = 0; w < SMB_THREADS / 32; ++w) s += red[w][tid];
            tot[tid] = s;
        }
        __syncthreads();
        if (tid < a.C) {
            // dh . h = sum_c beta_c (dh . o_c)
            float dhh = 0.f;
            for (int c = 0; c < a.C; ++c) dhh += __expf(a.lse[(int64_t)c * a.rows + row] - mx) * inv * tot[c];
            const float beta = __expf(a.lse[(int64_t)tid * a.rows + row] - mx) * inv;
            const float extra = a.dlse ? a.dlse[row] : 0.f;
            a.d_lse[(int64_t)tid * a.rows + row] = beta * (tot[tid] - dhh + extra);
        }
        // d o_c = beta_c dh
        unsigned char *dor = a.d_o + row * (int64_t)a.d * sizeof(Tin);
        for (int v = tid; v < nvec; v += SMB_THREADS) {
            float2 g[NP];
            E::unpack(*reinterpret_cast<const uint4 *>(dhr + (int64_t)v * 16), g);
            for (int c = 0; c < a.C; ++c) {
                const float beta = __expf(a.lse[(int64_t)c * a.rows + row] - mx) * inv;
                float2 y[NP];
#pragma unroll
                for (int p = 0; p < NP; ++p) y[p] = make_float2(beta * g[p].x, beta * g[p].y);
                *reinterpret_cast<uint4 *>(dor + c * cstride + (int64_t)v * 16) = E::pack(y);
            }
        }
        __syncthreads();                              // red / tot reused by the next row
    }
}

cudaError_t launch_state_merge_bwd(int dt, const StateMergeBwdArgs &a, int sms, void *stream) {
    if (a.C < 1 || a.C > SMB_MAXC) return cudaErrorInvalidValue;
    if (a.rows == 0) return cudaSuccess;
    int64_t grid = a.rows < (int64_t)sms * 8 ? a.rows : (int64_t)sms * 8;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dt == 1) state_merge_bwd_kernel<__nv_bfloat16><<<(unsigned)grid, SMB_THREADS, 0, s>>>(a);
    else state_merge_bwd_kernel<float><<<(unsigned)grid, SMB_THREADS, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace attnres
