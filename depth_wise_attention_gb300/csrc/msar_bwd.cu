// msar_bwd.cu -- kernels of the backward of the MSAR read.
//
// The backward runs as a chain of steps over tensors in the caller's
// workspace (attnres_api.cu, msar_expand_bwd):
//   1. msar_streams_kernel   the conv streams u_i^(r), r = 1..3, of every source
//   2. the depth read        Z^(r) = read of the sources u_i^(r) with query w_r
//                            (the forward read kernels, one call per stream)
//   3. msar_mix_bwd_kernel   the H^pre mixer's backward: dZ^(r), and per token
//                            e_t[o] = dl_t[o] / nu_t; msar_mix_acc_kernel then
//                            sums A[k][o] = sum_t zf_t[k] e_t[o], from which
//                            dmix_w = mg * A and dmix_gain = sum_o P[:, o] A[:, o]
//   4. the read backward     du_i^(r), dw_r and the gain's share per stream
//                            (read_bwd_kernel, one call per stream)
//   5. msar_conv_bwd_kernel  back through the causal convolutions:
//                            dv_i[t] = du_i^(0)[t] + sum_r sum_j cw_r[j] du_i^(r)[t + j],
//                            and per-CTA partials of dcw_r[j] = sum du_i^(r)[t] v_i[t - j]
//   6. msar_sum_kernel       the partials summed in a fixed order (deterministic)
// The streams and their gradients are stored in the source dtype.
#include <stdio.h>

#include "msar.h"
#include "msar_bwd.h"

namespace attnres {

// ---------------------------------------------------------------- step 1
// One thread per (source, channel pair) walks a chunk of tokens with a
// register window of its source's last KW rows; the three kernels of its two
// channels sit in registers.  Writes U[r-1][i][t][c..c+1] for r = 1..3.
template <typename Tin, int KW>
__global__ void __launch_bounds__(256) msar_streams_kernel(const MsarBwdArgs a) {
    using P2 = Pair2<Tin>;
    constexpr int ES = sizeof(Tin);
    const int c = (blockIdx.x * blockDim.x + threadIdx.x) * 2;
    const int i = blockIdx.y;
    const int64_t t0 = (int64_t)blockIdx.z * a.tc;
    if (c >= a.d) return;
    const int64_t t1 = t0 + a.tc < a.T ? t0 + a.tc : a.T;
    float2 w[3][KW];
    int64_t off = 0;
#pragma unroll
    for (int r = 0; r < 3; ++r) {
#pragma unroll
        for (int j = 0; j < KW; ++j)
            w[r][j] = j < a.k[r] ? make_float2(__ldg(a.conv_w + off + (int64_t)c * a.k[r] + j),
                                               __ldg(a.conv_w + off + (int64_t)(c + 1) * a.k[r] + j))
                                 : make_float2(0.f, 0.f);
        off += (int64_t)a.d * a.k[r];
    }
    const unsigned char *v = a.src + (int64_t)i * a.src_stride_bytes;
    float2 win[KW];                  // win[j] = v[t - j]
#pragma unroll
    for (int j = 0; j < KW; ++j) {
        const int64_t tr = t0 - 1 - j;
        win[j] = (j < KW - 1 && tr >= 0) ? P2::ld(v + (tr * a.d + c) * ES) : make_float2(0.f, 0.f);
    }
    for (int64_t t = t0; t < t1; ++t) {
#pragma unroll
        for (int j = KW - 1; j > 0; --j) win[j] = win[j - 1];
        win[0] = P2::ld(v + (t * a.d + c) * ES);
#pragma unroll
        for (int r = 0; r < 3; ++r) {
            float2 acc = make_float2(0.f, 0.f);
#pragma unroll
            for (int j = 0; j < KW; ++j)
                if (j < a.k[r]) acc = ffma2(w[r][j], win[j], acc);
            P2::st(a.u + ((((int64_t)r * a.n_src + i) * a.T + t) * a.d + c) * ES, acc);
        }
    }
}

// ---------------------------------------------------------------- step 3
// One token per CTA iteration; thread tid of NT owns channels
// [tid*CPT, tid*CPT + CPT) of every stream (d = NT * CPT, CPT a multiple of
// the 16-byte vector).  Two block reductions per token: (sum zf^2, the 4
// projection dots, the 4 dh.Z^(r)), then sum mg dzn zf.  P is read through
// L1/L2 (4d x 4 floats).
template <typename Tin, int NT, int CPT>
__global__ void __launch_bounds__(NT) msar_mix_bwd_kernel(const MsarBwdArgs a) {
    using E = Elem<Tin>;
    constexpr int EPV = E::EPV, NV = CPT / EPV, NP = EPV / 2, NW = NT / 32;
    static_assert(CPT % EPV == 0, "whole vectors per thread");
    __shared__ float red[NW][10];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int d = a.d;
    const int64_t md = 4 * (int64_t)d;
    const int c0 = tid * CPT;
    for (int64_t t = blockIdx.x; t < a.T; t += gridDim.x) {
        float zf[4][CPT], dh[CPT];
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int v = 0; v < NV; ++v) {
                float2 x[NP];
                E::unpack(*reinterpret_cast<const uint4 *>(a.z + (((int64_t)r * a.T + t) * d + c0 + v * EPV) * E::BYTES), x);
#pragma unroll
                for (int p = 0; p < NP; ++p) { zf[r][v * EPV + 2 * p] = x[p].x; zf[r][v * EPV + 2 * p + 1] = x[p].y; }
            }
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            float2 x[NP];
            E::unpack(*reinterpret_cast<const uint4 *>(a.dh + (t * d + c0 + v * EPV) * E::BYTES), x);
#pragma unroll
            for (int p = 0; p < NP; ++p) { dh[v * EPV + 2 * p] = x[p].x; dh[v * EPV + 2 * p + 1] = x[p].y; }
        }
        // round 1: sum zf^2, sum mg zf P[:, o], dh . Z^(r)
        float s[9];
#pragma unroll
        for (int q = 0; q < 9; ++q) s[q] = 0.f;
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int k = 0; k < CPT; ++k) {
                const int64_t kk = (int64_t)r * d + c0 + k;
                const float z = zf[r][k];
                const float g = a.mix_gain ? __ldg(a.mix_gain + kk) : 1.f;
                const float4 pw = __ldg(reinterpret_cast<const float4 *>(a.mix_w + kk * 4));
                s[0] = fmaf(z, z, s[0]);
                const float gz = g * z;
                s[1] = fmaf(gz, pw.x, s[1]);
                s[2] = fmaf(gz, pw.y, s[2]);
                s[3] = fmaf(gz, pw.z, s[3]);
                s[4] = fmaf(gz, pw.w, s[4]);
                s[5 + r] = fmaf(dh[k], z, s[5 + r]);
            }
#pragma unroll
        for (int q = 0; q < 9; ++q) s[q] = seg_sum<32>(s[q]);
        if (lane == 0)
#pragma unroll
            for (int q = 0; q < 9; ++q) red[warp][q] = s[q];
        __syncthreads();
        float tot[9];
#pragma unroll
        for (int q = 0; q < 9; ++q) {
            tot[q] = 0.f;
            for (int w = 0; w < NW; ++w) tot[q] += red[w][q];
        }
        __syncthreads();
        const float ms = fmaf(tot[0], 1.f / (float)md, a.mix_eps);
        const float inv = ms > 0.f ? rsqrtf(ms) : 0.f;              // 1 / nu
        float cr[4], dl[4];
#pragma unroll
        for (int o = 0; o < 4; ++o) {
            cr[o] = 1.f / (1.f + __expf(-tot[1 + o] * inv));
            dl[o] = tot[5 + o] * cr[o] * (1.f - cr[o]);
        }
        // dzn_k = sum_o dl_o P[k][o] (formed again below rather than held);
        // round 2: sum mg dzn zf
        auto dzn_at = [&](int64_t kk) {
            const float4 pw = __ldg(reinterpret_cast<const float4 *>(a.mix_w + kk * 4));
            return dl[0] * pw.x + dl[1] * pw.y + dl[2] * pw.z + dl[3] * pw.w;
        };
        float s2 = 0.f;
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int k = 0; k < CPT; ++k) {
                const int64_t kk = (int64_t)r * d + c0 + k;
                const float g = a.mix_gain ? __ldg(a.mix_gain + kk) : 1.f;
                s2 = fmaf(g * dzn_at(kk), zf[r][k], s2);
            }
        if (tid == 0)
            *reinterpret_cast<float4 *>(a.mix_e + t * 4) = make_float4(dl[0] * inv, dl[1] * inv, dl[2] * inv, dl[3] * inv);
        s2 = seg_sum<32>(s2);
        if (lane == 0) red[warp][9] = s2;
        __syncthreads();
        float ts2 = 0.f;
        for (int w = 0; w < NW; ++w) ts2 += red[w][9];
        __syncthreads();
        const float k3 = ts2 * inv * inv * inv / (float)md;
        // dZ^(r) = c_r dh + mg dzn / nu - zf s / (m d nu^3)
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int v = 0; v < NV; ++v) {
                float2 y[NP];
#pragma unroll
                for (int p = 0; p < NP; ++p) {
                    float yy[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int k = v * EPV + 2 * p + e;
                        const int64_t kk = (int64_t)r * d + c0 + k;
                        const float g = a.mix_gain ? __ldg(a.mix_gain + kk) : 1.f;
                        yy[e] = cr[r] * dh[k] + g * dzn_at(kk) * inv - zf[r][k] * k3;
                    }
                    y[p] = make_float2(yy[0], yy[1]);
                }
                *reinterpret_cast<uint4 *>(a.dz + (((int64_t)r * a.T + t) * d + c0 + v * EPV) * E::BYTES) = E::pack(y);
            }
    }
}

// A[k][o] = sum_t zf_t[k] e_t[o] over a chunk of tokens: one thread per
// element k of the flattened m d vector; per-chunk partials in mix_parts.
template <typename Tin>
__global__ void __launch_bounds__(256) msar_mix_acc_kernel(const MsarBwdArgs a) {
    using P2 = Pair2<Tin>;
    constexpr int ES = sizeof(Tin);
    const int64_t md = 4 * (int64_t)a.d;
    const int64_t k2 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 2;   // elements k2, k2 + 1
    if (k2 >= md) return;
    const int r = (int)(k2 / a.d);
    const int64_t c = k2 - (int64_t)r * a.d;
    const int64_t t0 = (int64_t)blockIdx.y * a.tc;
    const int64_t t1 = t0 + a.tc < a.T ? t0 + a.tc : a.T;
    float4 acc0 = make_float4(0.f, 0.f, 0.f, 0.f), acc1 = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int64_t t = t0; t < t1; ++t) {
        const float2 z = P2::ld(a.z + (((int64_t)r * a.T + t) * a.d + c) * ES);
        const float4 e = __ldg(reinterpret_cast<const float4 *>(a.mix_e + t * 4));
        acc0.x = fmaf(z.x, e.x, acc0.x); acc0.y = fmaf(z.x, e.y, acc0.y);
        acc0.z = fmaf(z.x, e.z, acc0.z); acc0.w = fmaf(z.x, e.w, acc0.w);
        acc1.x = fmaf(z.y, e.x, acc1.x); acc1.y = fmaf(z.y, e.y, acc1.y);
        acc1.z = fmaf(z.y, e.z, acc1.z); acc1.w = fmaf(z.y, e.w, acc1.w);
    }
    float *wp = a.mix_parts + (size_t)blockIdx.y * (size_t)(md * 4);
    *reinterpret_cast<float4 *>(wp + k2 * 4) = acc0;
    *reinterpret_cast<float4 *>(wp + (k2 + 1) * 4) = acc1;
}

// dmix_w[k][o] = mg_k A[k][o];  dmix_gain[k] = sum_o P[k][o] A[k][o]
__global__ void __launch_bounds__(256) msar_mix_finish_kernel(const MsarBwdArgs a, const float *A) {
    const int64_t md = 4 * (int64_t)a.d;
    for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < md; k += (int64_t)gridDim.x * blockDim.x) {
        const float4 ak = *reinterpret_cast<const float4 *>(A + k * 4);
        const float4 pk = __ldg(reinterpret_cast<const float4 *>(a.mix_w + k * 4));
        const float g = a.mix_gain ? __ldg(a.mix_gain + k) : 1.f;
        *reinterpret_cast<float4 *>(a.dmix_w + k * 4) = make_float4(g * ak.x, g * ak.y, g * ak.z, g * ak.w);
        if (a.dmix_gain) a.dmix_gain[k] = pk.x * ak.x + pk.y * ak.y + pk.z * ak.z + pk.w * ak.w;
    }
}

// ---------------------------------------------------------------- step 5
// One thread per (source, channel) walks a chunk of tokens downwards with a
// register window of the three conv streams' gradients ahead
// (dw_r[j] = du^(r)[t + j]) and of the source's rows behind (vw[j] = v[t - j]):
//   dv[t]      = du^(0)[t] + sum_r sum_j cw_r[j] du^(r)[t + j]
//   dcw_r[j]  += du^(r)[t] v[t - j]
// The kernel-gradient partials of the thread's channel go to
// conv_parts[(chunk * n_src + i)][ktot][d], packed like conv_w.  KA, KB, KC > 0
// fix the kernel sizes at compile time; 0 reads them from the arguments
// (windows of MSAR_KMAX rows).
template <typename Tin> __device__ __forceinline__ float ld1(const unsigned char *p);
template <> __device__ __forceinline__ float ld1<float>(const unsigned char *p) {
    return *reinterpret_cast<const float *>(p);
}
template <> __device__ __forceinline__ float ld1<__nv_bfloat16>(const unsigned char *p) {
    return __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(p));
}
template <typename Tin> __device__ __forceinline__ void st1(unsigned char *p, float v);
template <> __device__ __forceinline__ void st1<float>(unsigned char *p, float v) {
    *reinterpret_cast<float *>(p) = v;
}
template <> __device__ __forceinline__ void st1<__nv_bfloat16>(unsigned char *p, float v) {
    *reinterpret_cast<__nv_bfloat16 *>(p) = __float2bfloat16_rn(v);
}

template <typename Tin, int KA, int KB, int KC>
__global__ void __launch_bounds__(256) msar_conv_bwd_kernel(const MsarBwdArgs a) {
    constexpr bool FIXED = KA > 0;
    constexpr int K0 = FIXED ? KA : MSAR_KMAX, K1 = FIXED ? KB : MSAR_KMAX, K2 = FIXED ? KC : MSAR_KMAX;
    constexpr int KT = K0 + K1 + K2;
    constexpr int KM = K0 > K1 ? (K0 > K2 ? K0 : K2) : (K1 > K2 ? K1 : K2);
    constexpr int ES = sizeof(Tin);
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    const int i = blockIdx.y;
    const int64_t t0 = (int64_t)blockIdx.z * a.tc;
    if (c >= a.d) return;
    const int64_t t1 = t0 + a.tc < a.T ? t0 + a.tc : a.T;
    auto has = [&](int r, int j) { return FIXED || j < a.k[r]; };
    float w[KT], g[KT], dw[KT], vw[KM];
    {
        int64_t off = 0;
#pragma unroll
        for (int r = 0; r < 3; ++r) {
#pragma unroll
            for (int j = 0; j < (r == 0 ? K0 : r == 1 ? K1 : K2); ++j) {
                w[(r == 0 ? 0 : r == 1 ? K0 : K0 + K1) + j] = has(r, j) ? __ldg(a.conv_w + off + (int64_t)c * a.k[r] + j) : 0.f;
                g[(r == 0 ? 0 : r == 1 ? K0 : K0 + K1) + j] = 0.f;
            }
            off += (int64_t)a.d * a.k[r];
        }
    }
    const unsigned char *v = a.src + (int64_t)i * a.src_stride_bytes;
    auto du_at = [&](int r, int64_t t) {          // du^(r+1)[t] of source i (zero past the end)
        return t < a.T ? ld1<Tin>(a.du + ((((int64_t)(r + 1) * a.n_src + i) * a.T + t) * a.d + c) * ES) : 0.f;
    };
    // each step first moves the windows down one row; before the first step
    // (t = t1 - 1) they hold dw_r[j] = du^(r)[t1 + j] and vw[j] = v[t1 - j]
#pragma unroll
    for (int r = 0; r < 3; ++r)
#pragma unroll
        for (int j = 0; j < (r == 0 ? K0 : r == 1 ? K1 : K2); ++j) dw[(r == 0 ? 0 : r == 1 ? K0 : K0 + K1) + j] = has(r, j) ? du_at(r, t1 + j) : 0.f;
#pragma unroll
    for (int j = 0; j < KM; ++j) {
        const int64_t tr = t1 - j;
        vw[j] = (j >= 1 && tr >= 0) ? ld1<Tin>(v + (tr * a.d + c) * ES) : 0.f;
    }
    for (int64_t t = t1 - 1; t >= t0; --t) {
        // windows move down one row: dw_r[j] = du^(r)[t + j], vw[j] = v[t - j]
#pragma unroll
        for (int r = 0; r < 3; ++r) {
#pragma unroll
            for (int j = (r == 0 ? K0 : r == 1 ? K1 : K2) - 1; j > 0; --j) dw[(r == 0 ? 0 : r == 1 ? K0 : K0 + K1) + j] = dw[(r == 0 ? 0 : r == 1 ? K0 : K0 + K1) + j - 1];
            dw[(r == 0 ? 0 : r == 1 ? K0 : K0 + K1)] = du_at(r, t);
        }
#pragma unroll
        for (int j = 0; j < KM - 1; ++j) vw[j] = vw[j + 1];
        {
            const int64_t tr = t - (KM - 1);
            vw[KM - 1] = tr >= 0 ? ld1<Tin>(v + (tr * a.d + c) * ES) : 0.f;
        }
        float acc = ld1<Tin>(a.du + (((int64_t)i * a.T + t) * a.d + c) * ES);     // du^(0)[t]
#pragma unroll
        for (int r = 0; r < 3; ++r)
#pragma unroll
            for (int j = 0; j < (r == 0 ? K0 : r == 1 ? K1 : K2); ++j)
                if (has(r, j)) {
                    acc = fmaf(w[(r == 0 ? 0 : r == 1 ? K0 : K0 + K1) + j], dw[(r == 0 ? 0 : r == 1 ? K0 : K0 + K1) + j], acc);
                    g[(r == 0 ? 0 : r == 1 ? K0 : K0 + K1) + j] = fmaf(dw[(r == 0 ? 0 : r == 1 ? K0 : K0 + K1)], vw[j], g[(r == 0 ? 0 : r == 1 ? K0 : K0 + K1) + j]);
                }
        st1<Tin>(a.dsrc + (int64_t)i * a.dsrc_stride_bytes + (t * a.d + c) * ES, acc);
    }
    float *gp = a.conv_parts + ((size_t)blockIdx.z * a.n_src + i) * (size_t)a.ktot * a.d;
    int koff = 0;
#pragma unroll
    for (int r = 0; r < 3; ++r) {
#pragma unroll
        for (int j = 0; j < (r == 0 ? K0 : r == 1 ? K1 : K2); ++j)
            if (has(r, j)) gp[(int64_t)koff * a.d + (int64_t)c * a.k[r] + j] = g[(r == 0 ? 0 : r == 1 ? K0 : K0 + K1) + j];
        koff += a.k[r];
    }
}

// ---------------------------------------------------------------- step 6
// out[e] = (accumulate ? out[e] : 0) + sum_p parts[p * n + e], p in order.
__global__ void __launch_bounds__(256) msar_sum_kernel(const float *parts, int64_t nparts, int64_t n, float *out,
                                                       int accumulate) {
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += (int64_t)gridDim.x * blockDim.x) {
        float s = accumulate ? out[e] : 0.f;
        for (int64_t p = 0; p < nparts; ++p) s += parts[p * n + e];
        out[e] = s;
    }
}

// ---------------------------------------------------------------- launchers
template <typename Tin>
static cudaError_t launch_streams_t(const MsarBwdArgs &a, cudaStream_t s) {
    const dim3 grid((unsigned)((a.d / 2 + 255) / 256), (unsigned)a.n_src, (unsigned)((a.T + a.tc - 1) / a.tc));
    msar_streams_kernel<Tin, MSAR_KMAX><<<grid, 256, 0, s>>>(a);
    return cudaGetLastError();
}

template <typename Tin>
static cudaError_t launch_conv_bwd_t(const MsarBwdArgs &a, cudaStream_t s) {
    const dim3 grid((unsigned)((a.d + 255) / 256), (unsigned)a.n_src, (unsigned)((a.T + a.tc - 1) / a.tc));
    if (a.k[0] == 4 && a.k[1] == 8 && a.k[2] == 12)
        msar_conv_bwd_kernel<Tin, 4, 8, 12><<<grid, 256, 0, s>>>(a);
    else
        msar_conv_bwd_kernel<Tin, 0, 0, 0><<<grid, 256, 0, s>>>(a);
    return cudaGetLastError();
}

template <typename Tin, int NT>
static cudaError_t launch_mix_bwd_nt(const MsarBwdArgs &a, int sms, cudaStream_t s) {
    auto fn = msar_mix_bwd_kernel<Tin, NT, 8>;
    int occ = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, NT, 0);
    if (e != cudaSuccess) return e;
    if (occ < 1) return cudaErrorInvalidConfiguration;
    const int64_t slots = (int64_t)sms * occ;
    fn<<<(unsigned)(a.T < slots ? a.T : slots), NT, 0, s>>>(a);
    return cudaGetLastError();
}

template <typename Tin>
static cudaError_t launch_mix_bwd_t(const MsarBwdArgs &a, int sms, cudaStream_t s) {
    cudaError_t e;
    switch (a.d) {
        case 1024: e = launch_mix_bwd_nt<Tin, 128>(a, sms, s); break;
        case 2048: e = launch_mix_bwd_nt<Tin, 256>(a, sms, s); break;
        case 4096: e = launch_mix_bwd_nt<Tin, 512>(a, sms, s); break;
        default: return cudaErrorInvalidValue;
    }
    if (e != cudaSuccess) return e;
    const dim3 agrid((unsigned)((2 * (int64_t)a.d + 255) / 256), (unsigned)((a.T + a.tc - 1) / a.tc));
    msar_mix_acc_kernel<Tin><<<agrid, 256, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t msar_bwd_streams(int dt, const MsarBwdArgs &a, void *stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return dt == 1 ? launch_streams_t<__nv_bfloat16>(a, s) : launch_streams_t<float>(a, s);
}

cudaError_t msar_bwd_mix(int dt, const MsarBwdArgs &a, int sms, void *stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return dt == 1 ? launch_mix_bwd_t<__nv_bfloat16>(a, sms, s) : launch_mix_bwd_t<float>(a, sms, s);
}

cudaError_t msar_bwd_conv(int dt, const MsarBwdArgs &a, void *stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return dt == 1 ? launch_conv_bwd_t<__nv_bfloat16>(a, s) : launch_conv_bwd_t<float>(a, s);
}

cudaError_t msar_bwd_mix_finish(const MsarBwdArgs &a, const float *A, void *stream) {
    const int64_t n = 4 * (int64_t)a.d;
    msar_mix_finish_kernel<<<(unsigned)((n + 255) / 256), 256, 0, static_cast<cudaStream_t>(stream)>>>(a, A);
    return cudaGetLastError();
}

cudaError_t msar_bwd_sum(const float *parts, int64_t nparts, int64_t n, float *out, int accumulate, void *stream) {
    const int64_t blocks = (n + 255) / 256;
    msar_sum_kernel<<<(unsigned)(blocks < 4096 ? blocks : 4096), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        parts, nparts, n, out, accumulate);
    return cudaGetLastError();
}

}  // namespace attnres
