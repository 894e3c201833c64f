// msar_phase2.cu -- phase 2 of MSAR inside the two-phase Block schedule.
//
// For one layer: the layer's partial sum p is expanded into its 4 streams
// (identity and the causal depthwise convolutions), each stream's score
// s_p^(r) = (w^(r) * g) . u_p^(r) / rms(u_p^(r)) is merged into the stream's
// phase-1 state (o^(r), lse^(r)) by the online-softmax merge, and the merged
// streams Z^(r) go through the H^pre mixer:
//     Z^(r) = (e^{lse-M} o^(r) + e^{s_p-M} u_p^(r)) / (e^{lse-M} + e^{s_p-M})
//     h     = sum_r sigmoid(RMSNorm(Flatten(Z)) . P[:, r]) Z^(r).
//
// Structure.  One source leaves little arithmetic per token, so the kernel
// streams rather than synchronising a cluster per token.  A CTA owns a tile
// of tt tokens and walks the row in slices of 512 channels (two per thread,
// the slice's conv kernels in registers), in up to three passes:
//   pass A  the partial's per-stream sum of squares and query dot,
//   pass B  Z and the mixer's sums (sum of Z^2 and the 4 projection dots),
//   pass C  Z again and the output row
// (no partial: passes B and C only, with Z = o).  The (pass, slice, group of
// G tokens) items form one stream: thread 0 bulk-copies each item's state
// rows and partial rows into a ring of shared-memory stages MP2_NST items
// ahead (bounded mbarrier waits).  Each thread keeps the partial's last rows
// of its two channels in registers as it walks the tokens.  Per-token sums
// are reduced by a warp butterfly and added into a per-warp table in shared
// memory (one lane owns each entry); a pass's totals are the sum over the
// warps, taken at the pass boundary.
#include <stdio.h>

#include "msar.h"

namespace attnres {

constexpr int MP2_THREADS = 256;
constexpr int MP2_SW = 2 * MP2_THREADS;       // channels per slice
constexpr int MP2_NA = 8;                     // pass A sums per token: (ss, dot) x 4 streams
constexpr int MP2_NB = 5;                     // pass B sums per token: ss(Z), 4 projection dots
constexpr int MP2_NST = 3;                    // shared-memory stages
constexpr int MP2_TT = 64;                    // tokens per CTA tile (at most)

template <typename Tin> struct MP2Shape {
    static constexpr int G = sizeof(Tin) == 2 ? 8 : 4;          // tokens per item
    static constexpr int ROWS = 5 * G;                          // 4G state rows + G partial rows
    static constexpr size_t STAGE = (size_t)ROWS * MP2_SW * sizeof(Tin);
    // floats after the stages: red_a [8][tt][8], red_b [8][tt][5], coef [tt][8], cmix [tt][4]
    static constexpr size_t TABLE_FLOATS = (size_t)8 * MP2_TT * (MP2_NA + MP2_NB) + (size_t)MP2_TT * 12;
    static constexpr size_t SMEM = MP2_NST * STAGE + TABLE_FLOATS * 4 + MP2_NST * 8 + 16;
};

// KA, KB, KC > 0 fix the kernel sizes at compile time; KW is the register
// window (the largest kernel size the instance handles).
template <typename Tin, int KA, int KB, int KC, int KW>
__global__ void __launch_bounds__(MP2_THREADS, 1) msar_phase2_kernel(const MsarP2Args a) {
    using P2 = Pair2<Tin>;
    using SH = MP2Shape<Tin>;
    constexpr int ES = sizeof(Tin);
    constexpr int G = SH::G;
    constexpr bool FIXED = KA > 0;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int d = a.d, tt = a.tt;
    const int64_t T = a.T;
    const int64_t t0 = (int64_t)blockIdx.x * tt;
    const int ntok = (int)(T - t0 < tt ? T - t0 : tt);
    const int64_t t_end = t0 + ntok;
    const bool has_p = a.partial != nullptr;
    const int kk[3] = {FIXED ? KA : a.k[0], FIXED ? KB : a.k[1], FIXED ? KC : a.k[2]};
    const int hist = max(kk[0], max(kk[1], kk[2])) - 1;
    const int nslices = (d + MP2_SW - 1) / MP2_SW;
    const int ngroups = (ntok + G - 1) / G;
    const int npass = has_p ? 3 : 2;
    const int per_pass = nslices * ngroups;
    const int nitems = npass * per_pass;

    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char *stages = smem;
    float *red_a = reinterpret_cast<float *>(smem + MP2_NST * SH::STAGE);   // [8][tt][8]
    float *red_b = red_a + (size_t)8 * tt * MP2_NA;                          // [8][tt][5]
    float *coef = red_b + (size_t)8 * tt * MP2_NB;                           // [tt][4][2]
    float *cmix = coef + (size_t)tt * 8;                                     // [tt][4]
    uint64_t *bars = reinterpret_cast<uint64_t *>(red_a + SH::TABLE_FLOATS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + MP2_NST);

    for (int e = tid; e < 8 * tt * (MP2_NA + MP2_NB); e += MP2_THREADS) red_a[e] = 0.f;
    for (int e = tid; e < tt * 8; e += MP2_THREADS) coef[e] = (e & 1) ? 0.f : 1.f;   // no partial: Z = o
    if (tid == 0) {
        for (int s = 0; s < MP2_NST; ++s) mbar_init(&bars[s], 1);
        *abort_flag = 0;
        mbar_init_fence();
    }
    __syncthreads();

    // item -> pass (0 = A, 1 = B, 2 = C), slice, group
    auto item_of = [&](int i, int &pass, int &slice, int &group) {
        const int pi = i / per_pass, rem = i - pi * per_pass;
        pass = has_p ? pi : pi + 1;
        slice = rem / ngroups;
        group = rem - slice * ngroups;
    };
    // warp 0 produces: lane 0 arms the stage's mbarrier, then the warp's lanes
    // share the item's row copies (one lane issuing ~40 copies would hold
    // warp 0 back and every warp would wait for it at the next barrier)
    const bool producer = warp == 0 && !a.wait.inject_stall;
    uint64_t pol = 0;
    if (producer) pol = l2_policy_evict_first();
    auto issue = [&](int i) {
        int pass, slice, group;
        item_of(i, pass, slice, group);
        const int c0 = slice * MP2_SW;
        const uint32_t rb = (uint32_t)((d - c0 < MP2_SW ? d - c0 : MP2_SW) * ES);
        const int64_t tb = t0 + (int64_t)group * G;
        const int n = (int)(t_end - tb < G ? t_end - tb : G);
        const int nrows = (pass == 0 ? 0 : 4 * n) + (has_p ? n : 0);
        uint64_t *bar = &bars[i % MP2_NST];
        unsigned char *st = stages + (size_t)(i % MP2_NST) * SH::STAGE;
        if (lane == 0) mbar_arrive_expect_tx(bar, rb * (uint32_t)nrows);
        __syncwarp();
        // copy j < 4n: state row (stream j / n, token j % n); then the partial's rows
        const int nstate = pass == 0 ? 0 : 4 * n;
        for (int j = lane; j < nrows; j += 32) {
            if (j < nstate) {
                const int r = j / n, k = j - r * n;
                bulk_g2s(st + (size_t)(r * G + k) * MP2_SW * ES, a.o + (((int64_t)r * T + tb + k) * d + c0) * ES,
                         rb, bar, pol);
            } else {
                const int k = j - nstate;
                bulk_g2s(st + (size_t)(4 * G + k) * MP2_SW * ES, a.partial + ((tb + k) * d + c0) * ES, rb, bar,
                         pol);
            }
        }
    };
    int issued = 0;
    if (producer)
        for (; issued < nitems && issued < MP2_NST; ++issued) issue(issued);

    const int cl = 2 * tid;
    float2 wc[3][KW];               // this slice's conv kernels on my two channels
    float2 win[KW];                 // the partial's recent rows on my channels: win[j] = p[t - j]
    float2 wq[4], pm[4][4];         // pass A: stream queries; pass B: mixer projection
    int cur_pass = -1, cur_slice = -1;
    for (int i = 0; i < nitems; ++i) {
        int pass, slice, group;
        item_of(i, pass, slice, group);
        const int c0 = slice * MP2_SW, c = c0 + cl;
        const bool valid = c < d;
        if (pass != cur_pass) {
            // pass boundary: the previous pass's totals
            if (cur_pass == 0) {
                for (int e = tid; e < ntok * 4; e += MP2_THREADS) {
                    const int tk = e >> 2, r = e & 3;
                    float ss = 0.f, dt = 0.f;
                    for (int w = 0; w < 8; ++w) {
                        ss += red_a[((size_t)w * tt + tk) * MP2_NA + 2 * r];
                        dt += red_a[((size_t)w * tt + tk) * MP2_NA + 2 * r + 1];
                    }
                    const float s = key_score(dt, ss, 1.f / (float)d, a.eps);
                    const float l = __ldg(a.lse + (int64_t)r * T + t0 + tk);
                    const float M = fmaxf(l, s);
                    const float eo = __expf(l - M), ep = __expf(s - M);
                    const float inv = 1.f / (eo + ep);
                    coef[tk * 8 + 2 * r] = eo * inv;
                    coef[tk * 8 + 2 * r + 1] = ep * inv;
                }
            } else if (cur_pass == 1) {
                for (int e = tid; e < ntok * 4; e += MP2_THREADS) {
                    const int tk = e >> 2, o = e & 3;
                    float ssz = 0.f, dp = 0.f;
                    for (int w = 0; w < 8; ++w) {
                        ssz += red_b[((size_t)w * tt + tk) * MP2_NB];
                        dp += red_b[((size_t)w * tt + tk) * MP2_NB + 1 + o];
                    }
                    const float ms = fmaf(ssz, 1.f / (float)(4 * d), a.mix_eps);
                    const float inv = ms > 0.f ? rsqrtf(ms) : 0.f;
                    cmix[tk * 4 + o] = 1.f / (1.f + __expf(-dp * inv));
                }
            }
            __syncthreads();
            cur_pass = pass;
            cur_slice = -1;
        }
        if (slice != cur_slice) {
            // a new slice: its conv kernels, the pass's per-channel constants
            // and the partial's rows before the tile
            cur_slice = slice;
            if (has_p) {
                int64_t g = 0;
#pragma unroll
                for (int r = 0; r < 3; ++r) {
#pragma unroll
                    for (int j = 0; j < KW; ++j) {
                        wc[r][j] = make_float2(0.f, 0.f);
                        if (j < kk[r] && valid)
                            wc[r][j] = make_float2(__ldg(a.conv_w + g + (int64_t)c * kk[r] + j),
                                                   __ldg(a.conv_w + g + (int64_t)(c + 1) * kk[r] + j));
                    }
                    g += (int64_t)d * kk[r];
                }
                // the walk shifts the window before each token, so it starts
                // with win[j] = p[t0 - 1 - j] (zero before the sequence)
#pragma unroll
                for (int j = 0; j < KW; ++j) {
                    const int64_t tr = t0 - 1 - j;
                    win[j] = (j < hist && tr >= 0 && valid) ? P2::ld(a.partial + (tr * d + c) * ES)
                                                            : make_float2(0.f, 0.f);
                }
            }
            if (pass == 0) {
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    wq[r] = make_float2(0.f, 0.f);
                    if (valid) {
                        wq[r] = make_float2(__ldg(a.query + (size_t)r * d + c), __ldg(a.query + (size_t)r * d + c + 1));
                        if (a.gain) { wq[r].x *= __ldg(a.gain + c); wq[r].y *= __ldg(a.gain + c + 1); }
                    }
                }
            } else if (pass == 1) {
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int64_t k0 = (int64_t)r * d + c;
                    const float g0 = valid && a.mix_gain ? __ldg(a.mix_gain + k0) : 1.f;
                    const float g1 = valid && a.mix_gain ? __ldg(a.mix_gain + k0 + 1) : 1.f;
#pragma unroll
                    for (int o = 0; o < 4; ++o)
                        pm[r][o] = valid ? make_float2(__ldg(a.mix_w + k0 * 4 + o) * g0,
                                                       __ldg(a.mix_w + (k0 + 1) * 4 + o) * g1)
                                         : make_float2(0.f, 0.f);
                }
            }
        }
        mbar_wait_bounded(&bars[i % MP2_NST], (uint32_t)(i / MP2_NST) & 1u, abort_flag, a.wait);
        const unsigned char *st = stages + (size_t)(i % MP2_NST) * SH::STAGE + (size_t)cl * ES;
        const int64_t tb = t0 + (int64_t)group * G;
        const int n = (int)(t_end - tb < G ? t_end - tb : G);
        // The item's G tokens are unrolled so that their convolutions and sums
        // interleave; a pass's per-token sums are collected for all G tokens
        // and reduced by one butterfly per item.  Tokens past the tile's end
        // (k >= n) contribute zeros.
        auto token_streams = [&](int k, float2 *u) {
            if (has_p) {
#pragma unroll
                for (int j = KW - 1; j > 0; --j) win[j] = win[j - 1];
                // channels past d were not copied: threads there carry zeros
                win[0] = (valid && k < n) ? P2::ld(st + (size_t)(4 * G + k) * MP2_SW * ES) : make_float2(0.f, 0.f);
                u[0] = win[0];
#pragma unroll
                for (int r = 0; r < 3; ++r) {
                    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                    for (int j = 0; j < KW; ++j)
                        if (j < kk[r]) acc = ffma2(wc[r][j], win[j], acc);
                    u[r + 1] = acc;
                }
            } else {
#pragma unroll
                for (int r = 0; r < 4; ++r) u[r] = make_float2(0.f, 0.f);
            }
        };
        auto token_merged = [&](int k, const float2 *u, float2 *z) {
            const int tk = group * G + k;
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const float2 ov = (valid && k < n) ? P2::ld(st + (size_t)(r * G + k) * MP2_SW * ES)
                                                   : make_float2(0.f, 0.f);
                const float wo = coef[tk * 8 + 2 * r], wp = coef[tk * 8 + 2 * r + 1];
                z[r] = ffma2(make_float2(wp, wp), u[r], fmul2(make_float2(wo, wo), ov));
            }
        };
        if (pass == 0) {
            float v[G * MP2_NA];
#pragma unroll
            for (int k = 0; k < G; ++k) {
                float2 u[4];
                token_streams(k, u);
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    v[k * MP2_NA + 2 * r] = dot2(u[r], u[r]);
                    v[k * MP2_NA + 2 * r + 1] = dot2(u[r], wq[r]);
                }
            }
            butterfly_reduce<G * MP2_NA>(v, lane);
            constexpr int R = Bfly<G * MP2_NA>::R;
#pragma unroll
            for (int j = 0; j < R; ++j) {
                const int idx = bfly_slot<G * MP2_NA>(lane, j);
                if (idx >= 0) red_a[((size_t)warp * tt + group * G) * MP2_NA + idx] += v[j];
            }
        } else if (pass == 1) {
            float v[G * MP2_NB];
#pragma unroll
            for (int k = 0; k < G; ++k) {
                float2 u[4], z[4];
                token_streams(k, u);
                token_merged(k, u, z);
                float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f, s4 = 0.f;
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    s0 += dot2(z[r], z[r]);
                    s1 += dot2(z[r], pm[r][0]);
                    s2 += dot2(z[r], pm[r][1]);
                    s3 += dot2(z[r], pm[r][2]);
                    s4 += dot2(z[r], pm[r][3]);
                }
                v[k * MP2_NB + 0] = s0;
                v[k * MP2_NB + 1] = s1;
                v[k * MP2_NB + 2] = s2;
                v[k * MP2_NB + 3] = s3;
                v[k * MP2_NB + 4] = s4;
            }
            butterfly_reduce<G * MP2_NB>(v, lane);
            constexpr int R = Bfly<G * MP2_NB>::R;
#pragma unroll
            for (int j = 0; j < R; ++j) {
                const int idx = bfly_slot<G * MP2_NB>(lane, j);
                if (idx >= 0) red_b[((size_t)warp * tt + group * G) * MP2_NB + idx] += v[j];
            }
        } else {
#pragma unroll
            for (int k = 0; k < G; ++k) {
                float2 u[4], z[4];
                token_streams(k, u);
                token_merged(k, u, z);
                const int tk = group * G + k;
                if (valid && k < n && !*abort_flag) {
                    float2 h = make_float2(0.f, 0.f);
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const float cr = cmix[tk * 4 + r];
                        h = ffma2(make_float2(cr, cr), z[r], h);
                    }
                    P2::st(a.out + ((tb + k) * d + c) * ES, h);
                }
            }
        }
        __syncthreads();                         // every thread is done with stage i
        if (producer) {
            // one decision for the whole producer warp
            if (__shfl_sync(0xffffffffu, (issued < nitems && !*abort_flag) ? 1 : 0, 0)) issue(issued++);
        }
    }

    // Drain (only matters after an abort): copies must land before exit.
    if (producer && lane == 0) {
        int never = 0;
        for (int i = issued > MP2_NST ? issued - MP2_NST : 0; i < issued; ++i)
            mbar_wait_bounded(&bars[i % MP2_NST], (uint32_t)(i / MP2_NST) & 1u, &never, a.wait);
    }
}

template <typename Tin>
static const void *mp2_fn(bool k4812) {
    return k4812 ? reinterpret_cast<const void *>(&msar_phase2_kernel<Tin, 4, 8, 12, 12>)
                 : reinterpret_cast<const void *>(&msar_phase2_kernel<Tin, 0, 0, 0, MSAR_KMAX>);
}

attnres_status_t launch_msar_phase2(int dt, MsarP2Args a, int sms, void *stream, char *err, size_t errlen) {
    const bool k4812 = a.k[0] == 4 && a.k[1] == 8 && a.k[2] == 12;
    const void *fn = dt == 1 ? mp2_fn<__nv_bfloat16>(k4812) : mp2_fn<float>(k4812);
    // tiles of up to 64 tokens, smaller (a multiple of the item) when that
    // leaves fewer CTAs than SMs
    const int g = dt == 1 ? MP2Shape<__nv_bfloat16>::G : MP2Shape<float>::G;
    int tt = MP2_TT;
    while (tt > g && (a.T + tt - 1) / tt < (int64_t)sms) tt /= 2;
    a.tt = tt;
    const size_t smem = dt == 1 ? MP2Shape<__nv_bfloat16>::SMEM : MP2Shape<float>::SMEM;
    int dev = 0, optin = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) {
        snprintf(err, errlen, "msar phase 2 device query: %s", cudaGetErrorString(e));
        return ATTNRES_ERR_CUDA;
    }
    if (smem > (size_t)optin) return ATTNRES_ERR_UNSUPPORTED;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) {
        snprintf(err, errlen, "msar phase 2 cudaFuncSetAttribute: %s", cudaGetErrorString(e));
        return ATTNRES_ERR_CUDA;
    }
    const int64_t grid = (a.T + tt - 1) / tt;
    void *args[] = {&a};
    e = cudaLaunchKernel(fn, dim3((unsigned)grid), dim3(MP2_THREADS), args, smem, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        snprintf(err, errlen, "msar phase 2 launch: %s", cudaGetErrorString(e));
        return ATTNRES_ERR_CUDA;
    }
    return ATTNRES_OK;
}

}  // namespace attnres
