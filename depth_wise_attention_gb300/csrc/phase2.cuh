// phase2.cuh -- Block AttnRes phase 2 for sm_103a: fold one layer's
// intra-block partial-sum source p into its phase-1 state (o, lse) with the
// online-softmax merge
//     s_p = (w * g) . p / sqrt(mean(p^2) + eps),  M = max(lse, s_p),
//     out = (e^{lse-M} o + e^{s_p-M} p) / (e^{lse-M} + e^{s_p-M}).
// A pure streaming kernel: per token it reads o and p once, writes out once,
// and never touches the cached block representations.  Loads are 128-bit
// and coalesced; many CTAs per SM keep enough bytes in flight.
#pragma once

#include "common.cuh"

namespace attnres {

constexpr int P2_THREADS = 256;

struct MergeArgs {
    const unsigned char *o;        // [T][d]
    const float *lse;              // [T]
    const unsigned char *partial;  // [T][d]
    int64_t T;
    int d;
    int nvec;
    const float *query;            // [d]
    const float *gain;             // [d] or nullptr
    float eps;
    unsigned char *out;            // [T][d], may equal o
    int tpr;                       // threads per token row (32..256)
    int tt;                        // token rows per CTA
    int64_t ntiles;
};

template <typename Tin, int VPT>
__global__ void __launch_bounds__(P2_THREADS) phase2_merge_kernel(const MergeArgs a) {
    using E = Elem<Tin>;
    constexpr int EPV = E::EPV;
    constexpr int NP = EPV / 2;
    __shared__ float red[2][P2_THREADS / 32][2];

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int r = tid / a.tpr, tr = tid - r * a.tpr;
    const int nwr = a.tpr >> 5;
    const float inv_d = 1.f / (float)a.d;

    int vid[VPT];
    bool vok[VPT];
    float2 wq[VPT][NP];
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
        }
    }

    // Software pipeline over this CTA's tiles: the loads of tile n+1 are in
    // flight while tile n is reduced, merged and stored.
    uint4 ov[VPT], pv[VPT];
    float lv = 0.f;
    auto load_tile = [&](int64_t tile, uint4 (&o_)[VPT], uint4 (&p_)[VPT], float &l_) {
        const int64_t t = tile * a.tt + r;
        const bool ok = tile < a.ntiles && t < a.T;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            if (ok && vok[k]) {
                const int64_t off = (t * a.d + (int64_t)vid[k] * EPV) * E::BYTES;
                o_[k] = ldg128_stream(a.o + off);
                p_[k] = ldg128_stream(a.partial + off);
            } else {
                o_[k] = make_uint4(0, 0, 0, 0);
                p_[k] = make_uint4(0, 0, 0, 0);
            }
        }
        l_ = ok ? __ldg(a.lse + t) : 0.f;
    };
    int64_t tile = blockIdx.x;
    load_tile(tile, ov, pv, lv);
    int buf = 0;
    for (; tile < a.ntiles; tile += gridDim.x, buf ^= 1) {
        const int64_t t = tile * a.tt + r;
        const bool row_ok = t < a.T;
        uint4 on[VPT], pn[VPT];
        float ln;
        load_tile(tile + gridDim.x, on, pn, ln);
        float2 ss = make_float2(0.f, 0.f), dt = make_float2(0.f, 0.f);
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            float2 x[NP];
            E::unpack(pv[k], x);
#pragma unroll
            for (int p = 0; p < NP; ++p) {
                ss = ffma2(x[p], x[p], ss);
                dt = ffma2(x[p], wq[k][p], dt);
            }
        }
        float s1 = ss.x + ss.y, s2 = dt.x + dt.y;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            s1 += __shfl_xor_sync(0xffffffffu, s1, o);
            s2 += __shfl_xor_sync(0xffffffffu, s2, o);
        }
        if (lane == 0) { red[buf][warp][0] = s1; red[buf][warp][1] = s2; }
        __syncthreads();
        float tss = 0.f, tdt = 0.f;
        for (int w = 0; w < nwr; ++w) {
            tss += red[buf][r * nwr + w][0];
            tdt += red[buf][r * nwr + w][1];
        }
        if (row_ok) {
            const float sp = key_score(tdt, tss, inv_d, a.eps);
            const float M = fmaxf(lv, sp);
            const float ea = __expf(lv - M), eb = __expf(sp - M);
            const float inv = 1.f / (ea + eb);
            const float2 ca = make_float2(ea * inv, ea * inv), cb = make_float2(eb * inv, eb * inv);
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                if (vok[k]) {
                    float2 xo[NP], xp[NP], y[NP];
                    E::unpack(ov[k], xo);
                    E::unpack(pv[k], xp);
#pragma unroll
                    for (int p = 0; p < NP; ++p) y[p] = ffma2(xp[p], cb, fmul2(xo[p], ca));
                    stg128_cs(a.out + (t * a.d + (int64_t)vid[k] * EPV) * E::BYTES, E::pack(y));
                }
            }
        }
#pragma unroll
        for (int k = 0; k < VPT; ++k) { ov[k] = on[k]; pv[k] = pn[k]; }
        lv = ln;
        // red[buf] is rewritten two tiles later, after the next __syncthreads
    }
}

}  // namespace attnres
