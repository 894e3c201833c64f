// read_bwd_one.cuh -- the backward of the depth read for one query over 3 to
// 16 bf16 sources, in one kernel (sm_103a): the per-stream read backward of
// MSAR, a Block layer's read (the block representations and the partial
// sum), the shallow layers of Full AttnRes.
//
// Same operation as read_bwd.cuh with n_q = 1 (per token, alpha recomputed
// from the sources, r_i = sqrt(mean(v_i^2) + eps)):
//     ds_i = alpha_i (dout . v_i - sum_j alpha_j dout . v_j + dlse)
//     dv_i = alpha_i dout + (ds_i / r_i) (w*g) - ds_i ((w*g) . v_i) / (d r_i^3) v_i
//     U   += sum_i (ds_i / r_i) v_i,   dq = g * U,   dgain = w * U.
// With one query the sources only have to be read once: read_bwd_kernel does
// that with whole-token stages, two of which fit, so a token's rows are in
// flight only while the one before is being worked on and the kernel waits
// on memory latency.  Here the rows stream through a ring of half-row stages
// instead (the 8 source rows and the gradient row of one half of the
// channels, 37 KB at d = 4096), so that while a token's two stages are
// worked on, three or four more are in flight:
//   1. per half row, the row sums (w*g).v_i and dout.v_i with one packed
//      mma.sync per 32 channels (A = the sources at two k-steps, B = the
//      query's bf16 hi and lo parts and the gradient row at each), and
//      v_i.v_i as the Gram diagonal (two more MMAs), as in the
//      coefficient kernels of read_bwd_split.cuh / read_bwd_many.cuh;
//   2. the warps' sums go to a double-buffered table (each warp arrives on
//      an mbarrier after its writes); one warp per token, rotating, waits
//      for the table after its gradient pass of the token before, forms the
//      softmax and alpha, ds/r and the v term (lanes i = 0..7) and hands them
//      over through shared memory as ready pairs behind a second mbarrier;
//   3. the gradient pass of a token runs after the row sums of the next one,
//      so no warp waits for the coefficients while there is other work: from
//      the stages, each lane writes dv for 4 (d = 4096) or 2 (d = 2048)
//      channels of each source and keeps U for them; the last warp done with
//      a stage refills it (a shared counter), its lanes issuing one row copy
//      each.  Two tokens' stages are held at a time, so the ring needs at
//      least four stages.
// U leaves as one partial per CTA for read_bwd_finish_kernel, which sums the
// partials in a fixed order.
#pragma once

#include "read_bwd.cuh"
#include "read_bwd_many.cuh"

namespace attnres {

constexpr int R1_NW = 16;             // warps
constexpr int R1_MAX_STAGES = 8;
constexpr int R1_ROWS = 9;            // stage rows: 8 sources and the gradient
constexpr int R1_CF = 8;              // coefficient floats per source: alpha, alpha, b, b, c, c, 0, 0
constexpr size_t R1_AUX_BYTES = 256 + (size_t)2 * RM_NV * RM_RS * 4 + (size_t)2 * 8 * R1_CF * 4;

struct ReadBwdOneArgs {
    const unsigned char *src;         // source 0, token 0 (bf16)
    int64_t src_stride_bytes;
    int n_src;                        // 1..8 (the launcher takes 3..8)
    int64_t T;
    int d;                            // 2048 or 4096
    const float *query;               // [d]
    const float *gain;                // [d] or nullptr
    float eps;
    float inv_d;
    const unsigned char *dout;        // [T][d] bf16
    const float *dlse;                // [T] or nullptr
    unsigned char *dsrc;              // [n_src] x (dsrc_stride_bytes apart) [T][d] bf16
    int64_t dsrc_stride_bytes;
    int accumulate;                   // 1: dsrc += gradient
    float *ws;                        // [gridDim.x][d] partial U
    int nstages;
    uint32_t pitch;                   // bytes between rows of a stage (d + 16: half a row, padded)
    uint32_t stage_bytes;             // 9 rows
    WaitCfg wait;
};

__device__ __forceinline__ void stg32_cs(void *p, uint32_t v) {
    asm volatile("st.global.cs.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint2 ldg64(const void *p) {
    uint2 v;
    asm volatile("ld.global.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}

// A lane's CPL channels (4: one 8-byte piece, 2: one 4-byte piece) of a
// stage row as floats, and back.
template <int CPL>
__device__ __forceinline__ void r1_load(uint32_t addr, float2 (&x)[CPL / 2]) {
    if constexpr (CPL == 4) {
        const uint2 r = lds64(addr);
        x[0] = bf2_to_f2(r.x);
        x[1] = bf2_to_f2(r.y);
    } else {
        x[0] = bf2_to_f2(lds32u(addr));
    }
}

// KS2: pairs of MMA k-steps (32 channels) per warp and half row: d / (2 * 32 * R1_NW).
template <int KS2>
__global__ void __launch_bounds__(R1_NW * 32, 1) read_bwd_one_kernel(const ReadBwdOneArgs a) {
    constexpr int NW = R1_NW;
    constexpr int CWH = KS2 * 32;                 // channels per warp and half row
    constexpr int CPL = CWH / 32;                 // channels per lane in the gradient pass
    constexpr int NP = CPL / 2;
    constexpr int RS = RM_RS;
    static_assert(CPL == 2 || CPL == 4, "d = 2048 or 4096");

    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char *stages = smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)a.nstages * a.stage_bytes);
    uint64_t *tfull = full + R1_MAX_STAGES;      // [2] table of token it&1 written (every warp)
    uint64_t *cfull = tfull + 2;                  // [2] coefficients of token it&1 written
    unsigned *done = reinterpret_cast<unsigned *>(cfull + 2);              // warps done with a stage
    unsigned *imax = done + R1_MAX_STAGES;                                 // halves issued so far
    volatile int *abort_flag = reinterpret_cast<volatile int *>(imax + 1);
    float *red = reinterpret_cast<float *>(smem + (size_t)a.nstages * a.stage_bytes + 256);
    float *cbuf = red + (size_t)2 * RM_NV * RM_RS;  // [2][8 sources][R1_CF]

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int g4 = lane >> 2, t4 = lane & 3;
    const int half_bytes = a.d;                   // d/2 bf16 channels

    if (tid == 0) {
        for (int s = 0; s < a.nstages; ++s) {
            mbar_init(&full[s], 1);
            done[s] = 0;
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], NW);
            mbar_init(&cfull[b], 1);
        }
        *imax = 0;
        *abort_flag = 0;
        mbar_init_fence();
    }
    // rows of absent sources are never loaded (an MMA row only meets its own
    // source's outputs, which are never used): zero them once anyway
    for (int b = tid * 16; b < a.nstages * (int)a.stage_bytes; b += NW * 32 * 16)
        *reinterpret_cast<uint4 *>(stages + b) = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();                     // before the copies that overwrite them
    __syncthreads();

    const int gstride = gridDim.x;
    const int n_items = blockIdx.x < a.T ? (int)((a.T - blockIdx.x + gstride - 1) / gstride) : 0;
    const int n_halves = 2 * n_items;

    // ------------------------------------------------------------ producer
    // half k (token item k/2, channel half k%2) into stage k % nstages, by a
    // whole warp: lane 0 arms the stage's barrier, lane i < n_src copies
    // source row i, lane 8 the gradient row; with accumulate, lanes 16.. bring
    // the half rows of dsrc that the gradient pass will add to into L2.  The
    // first nstages by warp 0, each later one by the warp that finishes the
    // half nstages before it last.
    const bool may_issue = !a.wait.inject_stall;
    const uint64_t pol = l2_policy_evict_first();
    auto issue = [&](int k, int s) {               // s = k % nstages
        const int64_t t = blockIdx.x + (int64_t)(k >> 1) * gstride;
        const int64_t off = (t * a.d + (int64_t)(k & 1) * (a.d / 2)) * 2;
        unsigned char *dst = stages + (size_t)s * a.stage_bytes;
        if (lane == 0) {
            mbar_arrive_expect_tx(&full[s], (uint32_t)half_bytes * (uint32_t)(a.n_src + 1));
            atomicMax(imax, (unsigned)(k + 1));
        }
        __syncwarp();
        if (lane < a.n_src)
            bulk_g2s(dst + (size_t)lane * a.pitch, a.src + (int64_t)lane * a.src_stride_bytes + off,
                     (uint32_t)half_bytes, &full[s], pol);
        else if (lane == 8)
            bulk_g2s(dst + (size_t)8 * a.pitch, a.dout + off, (uint32_t)half_bytes, &full[s], pol);
        else if (a.accumulate && lane >= 16 && lane - 16 < a.n_src)
            bulk_prefetch_l2(a.dsrc + (int64_t)(lane - 16) * a.dsrc_stride_bytes + off, (uint32_t)half_bytes);
    };
    if (warp == 0 && may_issue)
        for (int k = 0; k < n_halves && k < a.nstages; ++k) issue(k, k);

    // ------------------------------------------------------------ constants
    uint32_t bw[2][KS2][2];
    {
        ReadBwdCoefManyArgs m;
        m.query = a.query;
        m.gain = a.gain;
        rm_query_fragments<KS2>(m, warp * CWH, g4, t4, bw[0]);
        rm_query_fragments<KS2>(m, a.d / 2 + warp * CWH, g4, t4, bw[1]);
    }
    // ldmatrix rows: source row lane%8, channel block lane/8 of a 32-channel group
    const uint32_t lrow_x = (uint32_t)(lane & 7) * a.pitch + (uint32_t)(warp * CWH + 8 * (lane >> 3)) * 2;
    // lanes of columns 2 and 6 read the gradient row: channels 2t4.. of the
    // first (g4 = 2) or second (g4 = 6) k-step, and 8 channels on for b1
    const bool dlane = (g4 & 3) == 2;
    const uint32_t drow = (uint32_t)8 * a.pitch + (uint32_t)(warp * CWH + (g4 >> 2) * 16 + 2 * t4) * 2;
    // the gradient pass: this lane's CPL channels of the warp's slice of each half
    const uint32_t bcol = (uint32_t)(warp * CWH + CPL * lane) * 2;
    float2 wg[2][NP], U[2][NP];
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int p = 0; p < NP; ++p) {
            const int c = h * (a.d / 2) + warp * CWH + CPL * lane + 2 * p;
            float2 w = make_float2(__ldg(a.query + c), __ldg(a.query + c + 1));
            if (a.gain) { w.x *= __ldg(a.gain + c); w.y *= __ldg(a.gain + c + 1); }
            wg[h][p] = w;
            U[h][p] = make_float2(0.f, 0.f);
        }
    const uint32_t stage0 = smem_u32(stages);
    const int i8 = lane & 7;                      // the source of this lane's softmax values

    // coefficients of token it (the rotating duty), after this warp's
    // gradient pass of token it-1
    auto coefficients = [&](int it, float dl) {
        const bool ready = mbar_wait_bounded(&tfull[it & 1], (uint32_t)(it >> 1) & 1u, abort_flag, a.wait);
        const float *rb = red + (size_t)(it & 1) * RM_NV * RS;
        const float *pw = rb + i8 * RS, *pd = rb + (8 + i8) * RS, *ps = rb + (16 + i8) * RS;
        float sw = 0.f, sd = 0.f, ss = 0.f;
#pragma unroll
        for (int w = 0; w < NW; w += 4) {
            const float4 x = *reinterpret_cast<const float4 *>(ps + w);
            const float4 y = *reinterpret_cast<const float4 *>(pw + w);
            const float4 z = *reinterpret_cast<const float4 *>(pd + w);
            ss += (x.x + x.y) + (x.z + x.w);
            sw += (y.x + y.y) + (y.z + y.w);
            sd += (z.x + z.y) + (z.z + z.w);
        }
        const bool pv = i8 < a.n_src;
        const float ms = fmaf(ss, a.inv_d, a.eps);
        const float rinv = ms > 0.f ? rsqrtf(ms) : 0.f;          // 1 / r_i (0 for a zero key)
        const float score = pv ? sw * rinv : -INFINITY;
        const float mx = seg_max<8>(score);
        const float e = pv ? __expf(score - mx) : 0.f;
        const float es = seg_sum<8>(e);
        const float alpha = pv ? e / es : 0.f;
        const float mean = seg_sum<8>(pv ? alpha * sd : 0.f);
        const float ds = pv ? alpha * (sd - mean + dl) : 0.f;
        const float b = ds * rinv;
        const float c = pv ? -ds * sw * rinv * rinv * rinv * a.inv_d : 0.f;
        if (lane < 8) {
            float *cf = cbuf + ((size_t)(it & 1) * 8 + lane) * R1_CF;
            *reinterpret_cast<float4 *>(cf) = make_float4(alpha, alpha, b, b);
            *reinterpret_cast<float4 *>(cf + 4) = make_float4(c, c, 0.f, 0.f);
        }
        (void)ready;
        __syncwarp();
        if (lane == 0) mbar_arrive(&cfull[it & 1]);
    };

    float d1[2][4], gr[2][4];
    int s = 0;                                    // stage of the next half, and its phase parity
    uint32_t par = 0;
    int shp[2] = {0, 0};                          // stages of token it-1
    for (int it = 0; it <= n_items; ++it) {
        const bool duty = it < n_items && warp == (it & (NW - 1));
        float dl = 0.f;
        int shc[2] = {0, 0};
        if (it < n_items) {
            const int64_t t = blockIdx.x + (int64_t)it * gstride;
            if (duty && a.dlse != nullptr) dl = __ldg(a.dlse + t);
#pragma unroll
            for (int u = 0; u < 2; ++u)
#pragma unroll
                for (int e = 0; e < 4; ++e) { d1[u][e] = 0.f; gr[u][e] = 0.f; }
            // ---------------- the row sums of token it over both halves
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                mbar_wait_bounded(&full[s], par, abort_flag, a.wait);
                const uint32_t sb = stage0 + (uint32_t)s * a.stage_bytes;
#pragma unroll
                for (int s2 = 0; s2 < KS2; ++s2) {
                    uint32_t x0, x1, x2, x3;
                    ldsm_x4(sb + lrow_x + 64 * s2, x0, x1, x2, x3);
                    uint32_t b0 = bw[h][s2][0], b1 = bw[h][s2][1];
                    if (dlane) {
                        b0 = lds32u(sb + drow + 64 * s2);
                        b1 = lds32u(sb + drow + 64 * s2 + 16);
                    }
                    // rows 0..7: sources at the first k-step, 8..15 at the second
                    mma_full(d1[s2 & 1], x0, x2, x1, x3, b0, b1);
                    mma_rows8(gr[0], x0, x1, x0, x1);
                    mma_rows8(gr[1], x2, x3, x2, x3);
                }
                shc[h] = s;
                if (++s == a.nstages) { s = 0; par ^= 1u; }
            }
            // lane (i, 0): (w*g).v_i = columns 0 + 1 (first k-step) here and 4 + 5
            // (second) in lane (i, 2); lane (i, 1): dout.v_i = column 2 here and 6
            // in lane (i, 3); lane (i, i/2): v_i.v_i on the Gram diagonal.  The
            // table of token it-2 (the same buffer) was read before the
            // coefficients of token it-2 were handed over, which this warp
            // waited for before its gradient pass of token it-2.
            const float e0 = d1[0][0] + d1[1][0], e1 = d1[0][1] + d1[1][1];
            const float e2 = d1[0][2] + d1[1][2], e3 = d1[0][3] + d1[1][3];
            float v = t4 == 0 ? e0 + e1 : t4 == 1 ? e0 : t4 == 2 ? e2 + e3 : e2;
            v += __shfl_xor_sync(0xffffffffu, v, 2);
            const float ssq = (g4 & 1) ? gr[0][1] + gr[1][1] : gr[0][0] + gr[1][0];
            float *rb = red + (size_t)(it & 1) * RM_NV * RS;
            if (t4 < 2) rb[(8 * t4 + g4) * RS + warp] = v;
            if (t4 == (g4 >> 1)) rb[(16 + g4) * RS + warp] = ssq;
            __syncwarp();
            if (lane == 0) mbar_arrive(&tfull[it & 1]);
        }

        // ---------------- dv and U of token it-1 from its stages, half by half
        if (it >= 1) {
            const int ip = it - 1;
            const int64_t tp = blockIdx.x + (int64_t)ip * gstride;
            mbar_wait_bounded(&cfull[ip & 1], (uint32_t)(ip >> 1) & 1u, abort_flag, a.wait);
            const float *cb = cbuf + (size_t)(ip & 1) * 8 * R1_CF;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint32_t sb = stage0 + (uint32_t)shp[h] * a.stage_bytes + bcol;
                const int64_t goff = (tp * a.d + (int64_t)h * (a.d / 2)) * 2 + (int64_t)bcol;
                float2 dg[NP];
                r1_load<CPL>(sb + 8 * a.pitch, dg);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    if (i >= a.n_src) break;
                    const float4 ab = *reinterpret_cast<const float4 *>(cb + i * R1_CF);
                    const float2 cc = *reinterpret_cast<const float2 *>(cb + i * R1_CF + 4);
                    const float2 al = make_float2(ab.x, ab.y), bi = make_float2(ab.z, ab.w);
                    unsigned char *gp = a.dsrc + (int64_t)i * a.dsrc_stride_bytes + goff;
                    uint2 zr = make_uint2(0u, 0u);
                    if (a.accumulate) {
                        if constexpr (CPL == 4) zr = ldg64(gp);
                        else zr.x = *reinterpret_cast<const uint32_t *>(gp);
                    }
                    float2 x[NP], y[NP];
                    r1_load<CPL>(sb + (uint32_t)i * a.pitch, x);
#pragma unroll
                    for (int p = 0; p < NP; ++p) {
                        y[p] = fmul2(cc, x[p]);
                        y[p] = ffma2(al, dg[p], y[p]);
                        y[p] = ffma2(bi, wg[h][p], y[p]);
                        U[h][p] = ffma2(bi, x[p], U[h][p]);
                    }
                    if (a.accumulate) {
                        const float2 z0 = bf2_to_f2(zr.x);
                        y[0] = make_float2(y[0].x + z0.x, y[0].y + z0.y);
                        if constexpr (CPL == 4) {
                            const float2 z1 = bf2_to_f2(zr.y);
                            y[1] = make_float2(y[1].x + z1.x, y[1].y + z1.y);
                        }
                    }
                    if (!*abort_flag) {
                        if constexpr (CPL == 4)
                            stg64_cs(gp, make_uint2(f2_to_bf2(y[0].x, y[0].y), f2_to_bf2(y[1].x, y[1].y)));
                        else
                            stg32_cs(gp, f2_to_bf2(y[0].x, y[0].y));
                    }
                }
                // this warp is done with the stage; the last warp to be refills it
                __syncwarp();
                const int k = 2 * ip + h;
                int refill = 0;
                if (lane == 0) {
                    __threadfence_block();
                    if (atomicAdd(&done[shp[h]], 1u) == NW - 1) {
                        done[shp[h]] = 0;
                        refill = k + a.nstages < n_halves && may_issue && !*abort_flag;
                    }
                }
                if (__shfl_sync(0xffffffffu, refill, 0)) issue(k + a.nstages, shp[h]);
                __syncwarp();
            }
        }
        if (duty) coefficients(it, dl);
        shp[0] = shc[0];
        shp[1] = shc[1];
    }

    // this CTA's U: one partial per CTA
    if (!*abort_flag) {
        float *wrow = a.ws + (size_t)blockIdx.x * a.d;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float *p = wrow + h * (a.d / 2) + warp * CWH + CPL * lane;
            if constexpr (CPL == 4)
                *reinterpret_cast<float4 *>(p) = make_float4(U[h][0].x, U[h][0].y, U[h][1].x, U[h][1].y);
            else
                *reinterpret_cast<float2 *>(p) = U[h][0];
        }
    }
    // copies still in flight (only after an abort) must land before the CTA exits
    __syncthreads();
    if (tid == 0) {
        int never = 0;
        const int issued = (int)*imax;
        for (int k = issued > a.nstages ? issued - a.nstages : 0; k < issued; ++k)
            mbar_wait_bounded(&full[k % a.nstages], (uint32_t)(k / a.nstages) & 1u, &never, a.wait);
    }
}


// 9 to 16 sources (a Block layer's read in training: the N block
// representations and the partial sum): the same per-token work with the
// sources as the 16 rows of one k-step (one MMA per 16 channels for the two
// row dots, two for the Gram diagonal), stages of the n_src source rows and
// the gradient row, and the simpler schedule of one CTA barrier per token
// with every warp forming the coefficients (lanes i = 0..15): holding two
// tokens' stages, as the pipelined schedule above does, would leave too few
// in flight at these row counts.
constexpr int R16_RS = 20;            // table row stride in floats (16 warps + pad, float4-aligned)
constexpr size_t R16_AUX_BYTES = 256 + (size_t)2 * 48 * R16_RS * 4;

// KS: MMA k-steps (16 channels) per warp and half row: d / (2 * 16 * R1_NW).
template <int KS>
__global__ void __launch_bounds__(R1_NW * 32, 1) read_bwd_one16_kernel(const ReadBwdOneArgs a) {
    constexpr int NW = R1_NW;
    constexpr int CWH = KS * 16;                  // channels per warp and half row
    constexpr int CPL = CWH / 32;                 // channels per lane in the gradient pass
    constexpr int NP = CPL / 2;
    constexpr int RS = R16_RS;
    static_assert(CPL == 2 || CPL == 4, "d = 2048 or 4096");

    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char *stages = smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)a.nstages * a.stage_bytes);
    unsigned *done = reinterpret_cast<unsigned *>(full + R1_MAX_STAGES);   // warps done with a stage
    unsigned *imax = done + R1_MAX_STAGES;                                 // halves issued so far
    volatile int *abort_flag = reinterpret_cast<volatile int *>(imax + 1);
    float *red = reinterpret_cast<float *>(smem + (size_t)a.nstages * a.stage_bytes + 256);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int g4 = lane >> 2, t4 = lane & 3;
    const int half_bytes = a.d;                   // d/2 bf16 channels
    const int ns = a.n_src;                       // the gradient row follows the sources

    if (tid == 0) {
        for (int s = 0; s < a.nstages; ++s) {
            mbar_init(&full[s], 1);
            done[s] = 0;
        }
        *imax = 0;
        *abort_flag = 0;
        mbar_init_fence();
    }
    for (int b = tid * 16; b < a.nstages * (int)a.stage_bytes; b += NW * 32 * 16)
        *reinterpret_cast<uint4 *>(stages + b) = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
    __syncthreads();

    const int gstride = gridDim.x;
    const int n_items = blockIdx.x < a.T ? (int)((a.T - blockIdx.x + gstride - 1) / gstride) : 0;
    const int n_halves = 2 * n_items;

    // half k (token item k/2, channel half k%2) into stage k % nstages by a
    // whole warp: lane 0 arms the barrier, lane i < n_src copies source row
    // i, lane n_src the gradient row; with accumulate the half rows of dsrc
    // go to L2 as well.  The first nstages by warp 0, each later one by the
    // warp that finishes the half nstages before it last.
    const bool may_issue = !a.wait.inject_stall;
    const uint64_t pol = l2_policy_evict_first();
    auto issue = [&](int k, int s) {               // s = k % nstages
        const int64_t t = blockIdx.x + (int64_t)(k >> 1) * gstride;
        const int64_t off = (t * a.d + (int64_t)(k & 1) * (a.d / 2)) * 2;
        unsigned char *dst = stages + (size_t)s * a.stage_bytes;
        if (lane == 0) {
            mbar_arrive_expect_tx(&full[s], (uint32_t)half_bytes * (uint32_t)(ns + 1));
            atomicMax(imax, (unsigned)(k + 1));
        }
        __syncwarp();
        if (lane < ns)
            bulk_g2s(dst + (size_t)lane * a.pitch, a.src + (int64_t)lane * a.src_stride_bytes + off,
                     (uint32_t)half_bytes, &full[s], pol);
        else if (lane == ns)
            bulk_g2s(dst + (size_t)ns * a.pitch, a.dout + off, (uint32_t)half_bytes, &full[s], pol);
        if (a.accumulate && lane < ns)
            bulk_prefetch_l2(a.dsrc + (int64_t)lane * a.dsrc_stride_bytes + off, (uint32_t)half_bytes);
    };
    if (warp == 0 && may_issue)
        for (int k = 0; k < n_halves && k < a.nstages; ++k) issue(k, k);

    // ------------------------------------------------------------ constants
    // B fragments: column 0 the query's bf16 hi part, 1 its lo part, 2 the
    // gradient row (read at run time), 3..7 zero
    uint32_t bq[2][KS][2];
    {
        DepthReadMmaArgs m;
        m.queries = a.query;
        m.gain = a.gain;
        m.d = a.d;
        m.n_q = 1;
        dm_query_fragments<KS>(m, warp * CWH, g4, t4, bq[0]);
        dm_query_fragments<KS>(m, a.d / 2 + warp * CWH, g4, t4, bq[1]);
    }
    // ldmatrix rows: lanes 0..7 / 8..15 give rows 0..7 / 8..15 of the first 8
    // channels of a k-step, lanes 16..31 the same rows 8 channels on; rows of
    // absent sources read row 0 (their outputs are never used)
    const int lr = (lane & 7) + 8 * ((lane >> 3) & 1);
    const uint32_t lrow_x = (uint32_t)(lr < ns ? lr : 0) * a.pitch + (uint32_t)(warp * CWH + 8 * (lane >> 4)) * 2;
    const bool dlane = g4 == 2;
    const uint32_t drow = (uint32_t)ns * a.pitch + (uint32_t)(warp * CWH + 2 * t4) * 2;
    const uint32_t bcol = (uint32_t)(warp * CWH + CPL * lane) * 2;
    float2 wg[2][NP], U[2][NP];
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int p = 0; p < NP; ++p) {
            const int c = h * (a.d / 2) + warp * CWH + CPL * lane + 2 * p;
            float2 w = make_float2(__ldg(a.query + c), __ldg(a.query + c + 1));
            if (a.gain) { w.x *= __ldg(a.gain + c); w.y *= __ldg(a.gain + c + 1); }
            wg[h][p] = w;
            U[h][p] = make_float2(0.f, 0.f);
        }
    const uint32_t stage0 = smem_u32(stages);
    const int i16 = lane & 15;                    // the source of this lane's softmax values

    float d1[2][4], g0[4], g1[4];
    int s = 0;                                    // stage of the next half, and its phase parity
    uint32_t par = 0;
    for (int it = 0; it < n_items; ++it) {
        const int64_t t = blockIdx.x + (int64_t)it * gstride;
        const float dl = a.dlse != nullptr ? __ldg(a.dlse + t) : 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) { d1[0][e] = 0.f; d1[1][e] = 0.f; g0[e] = 0.f; g1[e] = 0.f; }
        int sh[2];
        // ---------------- the row sums over both halves
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            mbar_wait_bounded(&full[s], par, abort_flag, a.wait);
            const uint32_t sb = stage0 + (uint32_t)s * a.stage_bytes;
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                uint32_t x0, x1, x2, x3;           // rows 0..7 / 8..15 of channels 0..7, then 8..15
                ldsm_x4(sb + lrow_x + 32 * ks, x0, x1, x2, x3);
                uint32_t b0 = bq[h][ks][0], b1 = bq[h][ks][1];
                if (dlane) {
                    b0 = lds32u(sb + drow + 32 * ks);
                    b1 = lds32u(sb + drow + 32 * ks + 16);
                }
                mma_full(d1[ks & 1], x0, x1, x2, x3, b0, b1);
                mma_full(g0, x0, x1, x2, x3, x0, x2);   // B = sources 0..7: the diagonal of rows 0..7
                mma_full(g1, x0, x1, x2, x3, x1, x3);   // B = sources 8..15: the diagonal of rows 8..15
            }
            sh[h] = s;
            if (++s == a.nstages) { s = 0; par ^= 1u; }
        }
        // lane (i, 0): (w*g).v of sources i and i+8 (columns 0 + 1); lane (i, 1):
        // dout.v of sources i and i+8 (column 2); lane (i, i/2): v.v of source
        // i (rows 0..7 against sources 0..7) and i+8 (rows 8..15 against 8..15)
        {
            float *rb = red + (size_t)(it & 1) * 48 * RS;
            const float e0 = d1[0][0] + d1[1][0], e1 = d1[0][1] + d1[1][1];
            const float e2 = d1[0][2] + d1[1][2], e3 = d1[0][3] + d1[1][3];
            if (t4 == 0) {
                rb[g4 * RS + warp] = e0 + e1;
                rb[(8 + g4) * RS + warp] = e2 + e3;
            } else if (t4 == 1) {
                rb[(16 + g4) * RS + warp] = e0;
                rb[(24 + g4) * RS + warp] = e2;
            }
            if (t4 == (g4 >> 1)) {
                rb[(32 + g4) * RS + warp] = (g4 & 1) ? g0[1] : g0[0];
                rb[(40 + g4) * RS + warp] = (g4 & 1) ? g1[3] : g1[2];
            }
        }
        // the table of token it is complete; the one of token it-1 (the other
        // buffer) was read by every warp before it arrived here
        __syncthreads();

        // ---------------- coefficients (every warp, lanes i = lane % 16)
        float alpha, bco, cco;
        {
            const float *rb = red + (size_t)(it & 1) * 48 * RS;
            const float *pw = rb + i16 * RS, *pd = rb + (16 + i16) * RS, *ps = rb + (32 + i16) * RS;
            float sw = 0.f, sd = 0.f, ss = 0.f;
#pragma unroll
            for (int w = 0; w < NW; w += 4) {
                const float4 x = *reinterpret_cast<const float4 *>(ps + w);
                const float4 y = *reinterpret_cast<const float4 *>(pw + w);
                const float4 z = *reinterpret_cast<const float4 *>(pd + w);
                ss += (x.x + x.y) + (x.z + x.w);
                sw += (y.x + y.y) + (y.z + y.w);
                sd += (z.x + z.y) + (z.z + z.w);
            }
            const bool pv = i16 < ns;
            const float ms = fmaf(ss, a.inv_d, a.eps);
            const float rinv = ms > 0.f ? rsqrtf(ms) : 0.f;      // 1 / r_i (0 for a zero key)
            const float score = pv ? sw * rinv : -INFINITY;
            const float mx = seg_max<16>(score);
            const float e = pv ? __expf(score - mx) : 0.f;
            const float es = seg_sum<16>(e);
            alpha = pv ? e / es : 0.f;
            const float mean = seg_sum<16>(pv ? alpha * sd : 0.f);
            const float ds = pv ? alpha * (sd - mean + dl) : 0.f;
            bco = ds * rinv;
            cco = pv ? -ds * sw * rinv * rinv * rinv * a.inv_d : 0.f;
        }

        // ---------------- dv and U from the same stages, half by half
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint32_t sb = stage0 + (uint32_t)sh[h] * a.stage_bytes + bcol;
            const int64_t goff = (t * a.d + (int64_t)h * (a.d / 2)) * 2 + (int64_t)bcol;
            float2 dg[NP];
            r1_load<CPL>(sb + (uint32_t)ns * a.pitch, dg);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                if (i >= ns) break;
                const float al = __shfl_sync(0xffffffffu, alpha, i);
                const float bi = __shfl_sync(0xffffffffu, bco, i);
                const float ci = __shfl_sync(0xffffffffu, cco, i);
                unsigned char *gp = a.dsrc + (int64_t)i * a.dsrc_stride_bytes + goff;
                uint2 zr = make_uint2(0u, 0u);
                if (a.accumulate) {
                    if constexpr (CPL == 4) zr = ldg64(gp);
                    else zr.x = *reinterpret_cast<const uint32_t *>(gp);
                }
                float2 x[NP], y[NP];
                r1_load<CPL>(sb + (uint32_t)i * a.pitch, x);
#pragma unroll
                for (int p = 0; p < NP; ++p) {
                    y[p] = fmul2(make_float2(ci, ci), x[p]);
                    y[p] = ffma2(make_float2(al, al), dg[p], y[p]);
                    y[p] = ffma2(make_float2(bi, bi), wg[h][p], y[p]);
                    U[h][p] = ffma2(make_float2(bi, bi), x[p], U[h][p]);
                }
                if (a.accumulate) {
                    const float2 z0 = bf2_to_f2(zr.x);
                    y[0] = make_float2(y[0].x + z0.x, y[0].y + z0.y);
                    if constexpr (CPL == 4) {
                        const float2 z1 = bf2_to_f2(zr.y);
                        y[1] = make_float2(y[1].x + z1.x, y[1].y + z1.y);
                    }
                }
                if (!*abort_flag) {
                    if constexpr (CPL == 4)
                        stg64_cs(gp, make_uint2(f2_to_bf2(y[0].x, y[0].y), f2_to_bf2(y[1].x, y[1].y)));
                    else
                        stg32_cs(gp, f2_to_bf2(y[0].x, y[0].y));
                }
            }
            // this warp is done with the stage; the last warp to be refills it
            __syncwarp();
            const int k = 2 * it + h;
            int refill = 0;
            if (lane == 0) {
                __threadfence_block();
                if (atomicAdd(&done[sh[h]], 1u) == NW - 1) {
                    done[sh[h]] = 0;
                    refill = k + a.nstages < n_halves && may_issue && !*abort_flag;
                }
            }
            if (__shfl_sync(0xffffffffu, refill, 0)) issue(k + a.nstages, sh[h]);
            __syncwarp();
        }
    }

    if (!*abort_flag) {
        float *wrow = a.ws + (size_t)blockIdx.x * a.d;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float *p = wrow + h * (a.d / 2) + warp * CWH + CPL * lane;
            if constexpr (CPL == 4)
                *reinterpret_cast<float4 *>(p) = make_float4(U[h][0].x, U[h][0].y, U[h][1].x, U[h][1].y);
            else
                *reinterpret_cast<float2 *>(p) = U[h][0];
        }
    }
    // copies still in flight (only after an abort) must land before the CTA exits
    __syncthreads();
    if (tid == 0) {
        int never = 0;
        const int issued = (int)*imax;
        for (int k = issued > a.nstages ? issued - a.nstages : 0; k < issued; ++k)
            mbar_wait_bounded(&full[k % a.nstages], (uint32_t)(k / a.nstages) & 1u, &never, a.wait);
    }
}

}  // namespace attnres
