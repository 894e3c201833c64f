// merge_bwd.cuh -- backward of the Block phase-2 merge for sm_103a.
//
// Forward (phase2.cuh): s_p = (w * g) . p / r_p with r_p = sqrt(mean(p^2) + eps),
// a = e^{lse-M} / (e^{lse-M} + e^{s_p-M}), b = 1 - a, h = a o + b p.  For an
// output gradient dh, per token:
//     d_o       = a dh
//     dlse      = a b (dh . (o - p)),   ds_p = -dlse
//     d_partial = b dh + ds_p ((w * g) / r_p - p ((w * g) . p) / (d r_p^3))
//     U        += ds_p p / r_p          (summed over the tokens)
// and dquery = g * U, dgain = w * U after all tokens (read_bwd_finish_kernel
// with one query).  A streaming kernel like the merge: per token it reads o,
// p and dh once, reduces three sums over the row (sum p^2, (w*g).p and
// dh.(o - p)), and writes d_o, d_partial and dlse once; U stays in registers
// and each CTA row writes its partial to the caller's workspace, reduced in a
// fixed order afterwards.  The next tile's loads are in flight while the
// current one is reduced.
#pragma once

#include "common.cuh"

namespace attnres {

constexpr int MB_THREADS = 256;

struct MergeBwdArgs {
    const unsigned char *o;        // [T][d]
    const float *lse;              // [T]
    const unsigned char *partial;  // [T][d]
    const unsigned char *dh;       // [T][d]
    int64_t T;
    int d;
    int nvec;
    const float *query;            // [d]
    const float *gain;             // [d] or nullptr
    float eps;
    unsigned char *d_o;            // [T][d]
    float *d_lse;                  // [T]
    unsigned char *d_partial;      // [T][d]
    int accumulate;                // 1: d_partial += gradient
    float *ws;                     // [gridDim.x * tt][d] partial U
    int tpr;
    int tt;
    int64_t ntiles;
};

template <typename Tin, int VPT>
__global__ void __launch_bounds__(MB_THREADS, VPT <= 2 ? 2 : 1) merge_bwd_kernel(const MergeBwdArgs a) {
    using E = Elem<Tin>;
    constexpr int EPV = E::EPV;
    constexpr int NP = EPV / 2;
    __shared__ float red[2][MB_THREADS / 32][3];

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int r = tid / a.tpr, tr = tid - r * a.tpr;
    const int nwr = a.tpr >> 5;
    const float inv_d = 1.f / (float)a.d;

    int vid[VPT];
    bool vok[VPT];
    float2 wq[VPT][NP], U[VPT][NP];
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        vid[k] = k * a.tpr + tr;
        vok[k] = vid[k] < a.nvec;
#pragma unroll
        for (int p = 0; p < NP; ++p) {
            float2 w = make_float2(0.f, 0.f);
            if (vok[k]) {
                const int c = vid[k] * EPV + 2 * p;
                w = make_float2(__ldg(a.query + c), __ldg(a.query + c + 1));
                if (a.gain) { w.x *= __ldg(a.gain + c); w.y *= __ldg(a.gain + c + 1); }
            }
            wq[k][p] = w;
            U[k][p] = make_float2(0.f, 0.f);
        }
    }

    uint4 ov[VPT], pv[VPT], hv[VPT];
    float lv;
    auto load_tile = [&](int64_t tile, uint4 (&o_)[VPT], uint4 (&p_)[VPT], uint4 (&h_)[VPT], float &l_) {
        const int64_t t = tile * a.tt + r;
        const bool ok = tile < a.ntiles && t < a.T;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const uint4 z = make_uint4(0, 0, 0, 0);
            if (ok && vok[k]) {
                const int64_t off = (t * a.d + (int64_t)vid[k] * EPV) * E::BYTES;
                o_[k] = ldg128_stream(a.o + off);
                p_[k] = ldg128_stream(a.partial + off);
                h_[k] = ldg128_stream(a.dh + off);
            } else {
                o_[k] = z;
                p_[k] = z;
                h_[k] = z;
            }
        }
        l_ = ok ? __ldg(a.lse + t) : 0.f;
    };
    int64_t tile = blockIdx.x;
    load_tile(tile, ov, pv, hv, lv);
    int buf = 0;
    for (; tile < a.ntiles; tile += gridDim.x, buf ^= 1) {
        const int64_t t = tile * a.tt + r;
        const bool row_ok = t < a.T;
        uint4 on[VPT], pn[VPT], hn[VPT];
        float ln;
        load_tile(tile + gridDim.x, on, pn, hn, ln);

        // the three sums over the row
        float s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            float2 xo[NP], xp[NP], xh[NP];
            E::unpack(ov[k], xo);
            E::unpack(pv[k], xp);
            E::unpack(hv[k], xh);
            float2 ss = make_float2(0.f, 0.f), sw = make_float2(0.f, 0.f), sd = make_float2(0.f, 0.f);
#pragma unroll
            for (int p = 0; p < NP; ++p) {
                ss = ffma2(xp[p], xp[p], ss);
                sw = ffma2(xp[p], wq[k][p], sw);
                sd = ffma2(xh[p], make_float2(xo[p].x - xp[p].x, xo[p].y - xp[p].y), sd);
            }
            s1 += ss.x + ss.y;
            s2 += sw.x + sw.y;
            s3 += sd.x + sd.y;
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            s1 += __shfl_xor_sync(0xffffffffu, s1, o);
            s2 += __shfl_xor_sync(0xffffffffu, s2, o);
            s3 += __shfl_xor_sync(0xffffffffu, s3, o);
        }
        if (lane == 0) { red[buf][warp][0] = s1; red[buf][warp][1] = s2; red[buf][warp][2] = s3; }
        __syncthreads();
        float tss = 0.f, tsw = 0.f, tsd = 0.f;
        for (int w = 0; w < nwr; ++w) {
            tss += red[buf][r * nwr + w][0];
            tsw += red[buf][r * nwr + w][1];
            tsd += red[buf][r * nwr + w][2];
        }
        if (row_ok) {
            const float ms = fmaf(tss, inv_d, a.eps);
            const float rinv = ms > 0.f ? rsqrtf(ms) : 0.f;   // 1 / r_p (0: no score path)
            const float sp = tsw * rinv;
            const float M = fmaxf(lv, sp);
            const float ea = __expf(lv - M), eb = __expf(sp - M);
            const float inv = 1.f / (ea + eb);
            const float ca = ea * inv, cb = eb * inv;
            const float dl = ca * cb * tsd;
            const float k1 = -dl * rinv;                        // ds_p / r_p
            const float k2 = dl * tsw * rinv * rinv * rinv * inv_d;
            if (tr == 0) a.d_lse[t] = dl;
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                if (!vok[k]) continue;
                float2 xp[NP], xh[NP], yo[NP], yp[NP];
                E::unpack(pv[k], xp);
                E::unpack(hv[k], xh);
                const int64_t off = (t * a.d + (int64_t)vid[k] * EPV) * E::BYTES;
#pragma unroll
                for (int p = 0; p < NP; ++p) {
                    yo[p] = fmul2(make_float2(ca, ca), xh[p]);
                    yp[p] = ffma2(make_float2(k2, k2), xp[p],
                                  ffma2(make_float2(k1, k1), wq[k][p], fmul2(make_float2(cb, cb), xh[p])));
                    U[k][p] = ffma2(make_float2(k1, k1), xp[p], U[k][p]);
                }
                if (a.accumulate) {
                    float2 z[NP];
                    E::unpack(*reinterpret_cast<const uint4 *>(a.d_partial + off), z);
#pragma unroll
                    for (int p = 0; p < NP; ++p) yp[p] = make_float2(yp[p].x + z[p].x, yp[p].y + z[p].y);
                }
                stg128_cs(a.d_o + off, E::pack(yo));
                stg128_cs(a.d_partial + off, E::pack(yp));
            }
        }
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            ov[k] = on[k];
            pv[k] = pn[k];
            hv[k] = hn[k];
        }
        lv = ln;
    }

    // this row's U: one partial per (CTA, row) in the workspace
    float *wrow = a.ws + ((size_t)blockIdx.x * a.tt + r) * (size_t)a.d;
#pragma unroll
    for (int k = 0; k < VPT; ++k)
        if (vok[k])
#pragma unroll
            for (int p = 0; p < NP; ++p)
                *reinterpret_cast<float2 *>(wrow + vid[k] * EPV + 2 * p) = U[k][p];
}

}  // namespace attnres
