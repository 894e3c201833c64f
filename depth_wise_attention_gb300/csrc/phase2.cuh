// phase2.cuh -- Block AttnRes phase 2 for sm_103a: fold one layer's
// intra-block partial-sum source p into its phase-1 state (o, lse) with the
// online-softmax merge
//     s_p = (w * g) . p / sqrt(mean(p^2) + eps),  M = max(lse, s_p),
//     out = (e^{lse-M} o + e^{s_p-M} p) / (e^{lse-M} + e^{s_p-M}).
// Two options ride on the same streaming pass:
//   UPD  the partial is first updated with the previous layer's output f,
//        p' = p + f (p absent: p' = f): the merge scores and mixes p' in fp32,
//        and p' rounded to the storage type is written back for the following
//        layers and the block's summary -- one read of p and f instead of an
//        update pass plus a merge pass that reads p' again;
//   MH   MHAR heads: the score, the RMSNorm and the merge are taken per head
//        over its d/H channels with its own lse (lse [H][T], query [H][d/H]).
// A pure streaming kernel: per token it reads o, p (and f) once and writes out
// (and p') once, never touching the cached block representations.  Loads are
// 128-bit and coalesced; the next token's loads are in flight while the
// current one is reduced and merged.
#pragma once

#include "common.cuh"

namespace attnres {

constexpr int P2_THREADS = 256;

struct MergeArgs {
    const unsigned char *o;        // [T][d]
    const float *lse;              // [T]; MH: [H][T]
    const unsigned char *partial;  // [T][d]; UPD: may be nullptr (the update starts the sum)
    const unsigned char *f;        // UPD: [T][d], the previous layer's output
    unsigned char *partial_out;    // UPD: [T][d], partial + f (may alias partial or f)
    int64_t T;
    int d;
    int nvec;                      // 16-byte vectors per row
    int seg;                       // MH: vectors per head (a multiple of 32, or a power of 2 below 32)
    const float *query;            // [d] (MH: [H][d/H], the same layout)
    const float *gain;             // [d] or nullptr
    float eps;
    unsigned char *out;            // [T][d], may equal o
    int tpr;                       // threads per token row (32..256)
    int tt;                        // token rows per CTA
    int64_t ntiles;
};

// Residency: three CTAs per SM for the plain merge at <= 2 vectors per thread
// (its loads in flight set the pace), two with the fused update or heads (more
// live registers), one for wider rows.
template <typename Tin, int VPT, bool UPD, bool MH>
__global__ void __launch_bounds__(P2_THREADS, VPT <= 2 ? (UPD || MH ? 2 : 3) : 1)
    phase2_merge_kernel(const MergeArgs a) {
    using E = Elem<Tin>;
    constexpr int EPV = E::EPV;
    constexpr int NP = EPV / 2;
    constexpr int NR = MH ? VPT : 1;   // reductions per thread: one per vector when heads differ
    __shared__ float red[2][P2_THREADS / 32][NR][2];

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int r = tid / a.tpr, tr = tid - r * a.tpr;
    const int nwr = a.tpr >> 5;
    const float inv_n = 1.f / (float)(MH ? a.seg * EPV : a.d);
    // MH: lanes of one head inside a warp (heads narrower than a warp reduce
    // with a segmented shuffle and need no cross-warp step)
    const int segl = MH ? (a.seg < 32 ? a.seg : 32) : 32;

    int vid[VPT], hk[VPT];
    bool vok[VPT];
    float2 wq[VPT][NP];
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        vid[k] = k * a.tpr + tr;
        vok[k] = vid[k] < a.nvec;
        hk[k] = MH ? vid[k] / a.seg : 0;
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

    // MH, heads of whole warps: for each of this thread's heads j and vector
    // slot k2, the warps [wlo, whi) of the row whose slot-k2 vectors lie in
    // head hk[j] (every bound a multiple of 32 vectors, so exact)
    int wlo[NR][NR], whi[NR][NR];
#pragma unroll
    for (int j = 0; j < NR; ++j)
#pragma unroll
        for (int k2 = 0; k2 < NR; ++k2) {
            if (MH) {
                const int lo = (hk[j] * a.seg - k2 * a.tpr) / 32, hi = ((hk[j] + 1) * a.seg - k2 * a.tpr) / 32;
                wlo[j][k2] = lo < 0 ? 0 : (lo > nwr ? nwr : lo);
                whi[j][k2] = hi < 0 ? 0 : (hi > nwr ? nwr : hi);
            } else {
                wlo[j][k2] = 0;
                whi[j][k2] = nwr;
            }
        }

    // Software pipeline over this CTA's tiles: the loads of tile n+1 are in
    // flight while tile n is reduced, merged and stored.
    uint4 ov[VPT], pv[VPT], fv[UPD ? VPT : 1];
    float lv[NR];
    auto load_tile = [&](int64_t tile, uint4 (&o_)[VPT], uint4 (&p_)[VPT], uint4 (&f_)[UPD ? VPT : 1],
                         float (&l_)[NR]) {
        const int64_t t = tile * a.tt + r;
        const bool ok = tile < a.ntiles && t < a.T;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const uint4 z = make_uint4(0, 0, 0, 0);
            if (ok && vok[k]) {
                const int64_t off = (t * a.d + (int64_t)vid[k] * EPV) * E::BYTES;
                o_[k] = ldg128_stream(a.o + off);
                p_[k] = !UPD || a.partial ? ldg128_stream(a.partial + off) : z;
                if constexpr (UPD) f_[k] = ldg128_stream(a.f + off);
            } else {
                o_[k] = z;
                p_[k] = z;
                if constexpr (UPD) f_[k] = z;
            }
        }
#pragma unroll
        for (int j = 0; j < NR; ++j)
            l_[j] = ok && (!MH || vok[j]) ? __ldg(a.lse + (int64_t)hk[j] * a.T + t) : 0.f;
    };
    int64_t tile = blockIdx.x;
    load_tile(tile, ov, pv, fv, lv);
    int buf = 0;
    for (; tile < a.ntiles; tile += gridDim.x, buf ^= 1) {
        const int64_t t = tile * a.tt + r;
        const bool row_ok = t < a.T;
        uint4 on[VPT], pn[VPT], fn[UPD ? VPT : 1];
        float ln[NR];
        load_tile(tile + gridDim.x, on, pn, fn, ln);

        // the partial this layer scores: p, or the updated p + f in fp32; the
        // update is stored rounded to the storage type for the following layers
        // (recomputed from the packed inputs where needed instead of held)
        auto partial_vec = [&](int k, float2 (&x)[NP]) {
            E::unpack(pv[k], x);
            if constexpr (UPD) {
                float2 y[NP];
                E::unpack(fv[k], y);
#pragma unroll
                for (int p = 0; p < NP; ++p) x[p] = make_float2(x[p].x + y[p].x, x[p].y + y[p].y);
            }
        };
        if constexpr (UPD) {
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                float2 x[NP];
                partial_vec(k, x);
                if (row_ok && vok[k])
                    *reinterpret_cast<uint4 *>(a.partial_out + (t * a.d + (int64_t)vid[k] * EPV) * E::BYTES) =
                        E::pack(x);
            }
        }

        // sums of squares and query dots: per row, or per head (MH)
        float s1[NR], s2[NR];
#pragma unroll
        for (int j = 0; j < NR; ++j) { s1[j] = 0.f; s2[j] = 0.f; }
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            float2 x[NP];
            partial_vec(k, x);
            float2 ss = make_float2(0.f, 0.f), dt = make_float2(0.f, 0.f);
#pragma unroll
            for (int p = 0; p < NP; ++p) {
                ss = ffma2(x[p], x[p], ss);
                dt = ffma2(x[p], wq[k][p], dt);
            }
            s1[MH ? k : 0] += ss.x + ss.y;
            s2[MH ? k : 0] += dt.x + dt.y;
        }
#pragma unroll
        for (int j = 0; j < NR; ++j)
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1)
                if (o < segl) {
                    s1[j] += __shfl_xor_sync(0xffffffffu, s1[j], o);
                    s2[j] += __shfl_xor_sync(0xffffffffu, s2[j], o);
                }
        if (lane == 0)
#pragma unroll
            for (int j = 0; j < NR; ++j) { red[buf][warp][j][0] = s1[j]; red[buf][warp][j][1] = s2[j]; }
        __syncthreads();
        float tss[NR], tdt[NR];
        if (!MH || a.seg >= 32) {
#pragma unroll
            for (int j = 0; j < NR; ++j) {
                tss[j] = 0.f;
                tdt[j] = 0.f;
                // every (vector slot, warp) of this row whose head is head j's
#pragma unroll
                for (int k2 = 0; k2 < NR; ++k2)
                    for (int w = wlo[j][k2]; w < whi[j][k2]; ++w) {
                        tss[j] += red[buf][r * nwr + w][k2][0];
                        tdt[j] += red[buf][r * nwr + w][k2][1];
                    }
            }
        } else {
#pragma unroll
            for (int j = 0; j < NR; ++j) { tss[j] = s1[j]; tdt[j] = s2[j]; }
        }
        if (row_ok) {
            float2 ca[NR], cb[NR];
#pragma unroll
            for (int j = 0; j < NR; ++j) {
                const float sp = key_score(tdt[j], tss[j], inv_n, a.eps);
                const float M = fmaxf(lv[j], sp);
                const float ea = __expf(lv[j] - M), eb = __expf(sp - M);
                const float inv = 1.f / (ea + eb);
                ca[j] = make_float2(ea * inv, ea * inv);
                cb[j] = make_float2(eb * inv, eb * inv);
            }
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                if (vok[k]) {
                    float2 xo[NP], xp[NP], y[NP];
                    E::unpack(ov[k], xo);
                    partial_vec(k, xp);
#pragma unroll
                    for (int p = 0; p < NP; ++p)
                        y[p] = ffma2(xp[p], cb[MH ? k : 0], fmul2(xo[p], ca[MH ? k : 0]));
                    stg128_cs(a.out + (t * a.d + (int64_t)vid[k] * EPV) * E::BYTES, E::pack(y));
                }
            }
        }
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            ov[k] = on[k];
            pv[k] = pn[k];
            if constexpr (UPD) fv[k] = fn[k];
        }
#pragma unroll
        for (int j = 0; j < NR; ++j) lv[j] = ln[j];
        // red[buf] is rewritten two tiles later, after the next __syncthreads
    }
}

}  // namespace attnres
