// read_bwd_many.cuh -- the backward of the depth read for one query over 17
// to 64 bf16 sources (Full AttnRes past layer 16), in two kernels (sm_103a).
//
// Same operation as read_bwd.cuh with n_q = 1 (per token, alpha recomputed
// from the sources, r_i = sqrt(mean(v_i^2) + eps)):
//     ds_i = alpha_i (dout . v_i - sum_j alpha_j dout . v_j + dlse)
//     dv_i = alpha_i dout + (ds_i / r_i) (w*g) - ds_i ((w*g) . v_i) / (d r_i^3) v_i
//     U   += sum_i (ds_i / r_i) v_i,   dq = g * U,   dgain = w * U.
// The softmax couples every source of a token, so a one-kernel backward
// would have to hold all of them; the split form of read_bwd_split.cuh
// extends to many sources instead:
//
// read_bwd_coef_many_kernel: the sources of a token stream through a ring of
// half-row stages in chunks of 8 (the chunk's 8 source rows and the gradient
// row, which is read again for every chunk and stays in L2).  One packed
// mma.sync per 32 channels takes both row dots of all 8 sources: A = the
// sources at two k-steps (rows 0..7, 8..15), B = (query hi, query lo,
// gradient) at each k-step (columns 0..2 and 4..6).  The sums of squares are
// the Gram diagonal (two more MMAs).  The per-warp sums of each chunk go to a
// double-buffered table; after a token's last chunk one warp (rotating over
// the tokens, one half row later) forms the softmax over all the sources (two
// per lane) and writes coef[t][chunk] = {alpha (8), ds/r (8), the v term (8)}.
//
// read_bwd_apply_many_kernel: a CTA owns 1024 channels (4 per thread) and a
// range of tokens; per (token, chunk) its 8-byte pieces of the chunk's rows
// (and, with the first chunk, of the gradient row) arrive by cp.async two
// units ahead; it writes dv and keeps U in registers, one partial per CTA for
// read_bwd_finish_kernel.
//
// Traffic per token: the sources twice and the source gradients once, about
// 1.5x the essential bytes, where the chunked chain (recomputed chunk states,
// their merge backward, one backward per chunk) moves about 1.75x.
#pragma once

#include "read_bwd_split.cuh"

namespace attnres {

constexpr int RM_MAXC = 8;            // most chunks of 8 sources (64 sources)
constexpr int RM_NV = 24;             // row sums per chunk and column: (w*g).v 8, dout.v 8, v.v 8
constexpr int RM_RS = 20;             // table row stride in floats (16 warps + pad, float4-aligned)
constexpr size_t RM_AUX_BYTES = 256 + (size_t)2 * RM_MAXC * RM_NV * RM_RS * 4;
constexpr int RM_ROWS = 9;            // stage rows: 8 sources and the gradient

struct ReadBwdCoefManyArgs {
    const unsigned char *src;         // source 0, token 0 (bf16)
    int64_t src_stride_bytes;
    int n_src;                        // 17..64
    int C;                            // chunks of 8 sources
    int64_t T;
    int d;                            // 2048 or 4096
    const float *query;               // [d]
    const float *gain;                // [d] or nullptr
    float eps;
    float inv_d;
    const unsigned char *dout;        // [T][d] bf16
    const float *dlse;                // [T] or nullptr
    float *coef;                      // [T][C][24]
    int nstages;
    uint32_t pitch;                   // bytes between rows of a stage (d + 16: half a row, padded)
    uint32_t stage_bytes;             // 9 rows
    WaitCfg wait;
};

// B fragments of the packed dots: column n = g4 of each k-step pair; 0, 1:
// the query's bf16 hi and lo parts on the first k-step (16 channels), 4, 5 on
// the second; 2, 6 take the gradient row at run time; 3, 7 stay zero.
template <int KS2>
__device__ __forceinline__ void rm_query_fragments(const ReadBwdCoefManyArgs &a, int cbase, int g4, int t4,
                                                   uint32_t (&bw)[KS2][2]) {
    const int kb = g4 >> 2, part = g4 & 3;
#pragma unroll
    for (int s2 = 0; s2 < KS2; ++s2)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t v = 0u;
            if (part < 2) {
                const int c = cbase + 32 * s2 + 16 * kb + 8 * h + 2 * t4;
                float v0 = __ldg(a.query + c), v1 = __ldg(a.query + c + 1);
                if (a.gain) { v0 *= __ldg(a.gain + c); v1 *= __ldg(a.gain + c + 1); }
                float h0, l0, h1, l1;
                split_bf16(v0, h0, l0);
                split_bf16(v1, h1, l1);
                v = part == 0 ? pack_bf16(h0, h1) : pack_bf16(l0, l1);
            }
            bw[s2][h] = v;
        }
}

__device__ __forceinline__ uint32_t lds32u(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}

// KS2: pairs of MMA k-steps (32 channels) per warp and half row: d / (2 * 32 * RC_NW).
template <int KS2>
__global__ void __launch_bounds__(RC_NW * 32, 1) read_bwd_coef_many_kernel(const ReadBwdCoefManyArgs a) {
    constexpr int NW = RC_NW;
    constexpr int CWH = KS2 * 32;                 // channels per warp and half row
    constexpr int RS = RM_RS;

    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char *stages = smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)a.nstages * a.stage_bytes);
    unsigned *done = reinterpret_cast<unsigned *>(full + RC_MAX_STAGES);   // warps done with a stage
    unsigned *imax = done + RC_MAX_STAGES;                                 // parts issued so far
    uint64_t *tfull = full + 2 * RC_MAX_STAGES;   // [2] table of token it&1 written
    uint64_t *tfree = tfull + 2;                  // [2] table of token it&1 read
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tfree + 2);
    float *red = reinterpret_cast<float *>(smem + (size_t)a.nstages * a.stage_bytes + 256);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int g4 = lane >> 2, t4 = lane & 3;
    const int half_bytes = a.d;                   // d/2 bf16 channels
    const int C = a.C;

    if (tid == 0) {
        for (int s = 0; s < a.nstages; ++s) {
            mbar_init(&full[s], 1);
            done[s] = 0;
        }
        *imax = 0;
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], NW);
            mbar_init(&tfree[b], 1);
        }
        *abort_flag = 0;
        mbar_init_fence();
    }
    // Rows of a short last chunk keep an earlier chunk's bytes; an MMA row
    // only meets its own source's outputs, which are never used.  Zero them
    // once so that no stale pattern is ever read before the first copy lands.
    for (int b = tid * 16; b < a.nstages * (int)a.stage_bytes; b += NW * 32 * 16)
        *reinterpret_cast<uint4 *>(stages + b) = make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();

    const int gstride = gridDim.x;
    const int n_items = blockIdx.x < a.T ? (int)((a.T - blockIdx.x + gstride - 1) / gstride) : 0;
    const int ppt = 2 * C;                        // parts per token: (chunk, half)
    const int n_parts = ppt * n_items;

    // ------------------------------------------------------------ producer
    // part k (token item k / ppt, chunk (k % ppt) / 2, half k % 2) into stage
    // k % nstages, by a whole warp: lane 0 arms the stage's barrier, then lane
    // i copies row i (one lane issuing every copy was the pace of the ring).
    // The first nstages by warp 0, each later one by the warp that finishes
    // the part nstages before it last.
    const bool may_issue = !a.wait.inject_stall;
    const uint64_t pol_first = l2_policy_evict_first();
    auto issue = [&](int k, int s) {               // s = k % nstages
        const int it = k / ppt, pc = k - it * ppt;
        const int c = pc >> 1, h = pc & 1;
        const int nc = a.n_src - 8 * c < 8 ? a.n_src - 8 * c : 8;
        const int64_t t = blockIdx.x + (int64_t)it * gstride;
        const int64_t off = (t * a.d + (int64_t)h * (a.d / 2)) * 2;
        unsigned char *dst = stages + (size_t)s * a.stage_bytes;
        if (lane == 0) {
            mbar_arrive_expect_tx(&full[s], (uint32_t)half_bytes * (uint32_t)(nc + 1));
            atomicMax(imax, (unsigned)(k + 1));
        }
        __syncwarp();
        if (lane < nc) {
            bulk_g2s(dst + (size_t)lane * a.pitch, a.src + (int64_t)(8 * c + lane) * a.src_stride_bytes + off,
                     (uint32_t)half_bytes, &full[s], pol_first);
        } else if (lane == 8) {
            // the gradient row is read again for every chunk: no evict-first hint
            asm volatile(
                "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                    smem_u32(dst + (size_t)8 * a.pitch)),
                "l"(a.dout + off), "r"((uint32_t)half_bytes), "r"(smem_u32(&full[s]))
                : "memory");
        }
    };
    if (warp == 0 && may_issue)
        for (int k = 0; k < n_parts && k < a.nstages; ++k) issue(k, k);

    // ------------------------------------------------------------ constants
    uint32_t bw[2][KS2][2];
    rm_query_fragments<KS2>(a, warp * CWH, g4, t4, bw[0]);
    rm_query_fragments<KS2>(a, a.d / 2 + warp * CWH, g4, t4, bw[1]);
    // ldmatrix rows: source row lane%8, channel block lane/8 of a 32-channel group
    const uint32_t lrow_x = (uint32_t)(lane & 7) * a.pitch + (uint32_t)(warp * CWH + 8 * (lane >> 3)) * 2;
    // lanes of columns 2 and 6 read the gradient row: channels 2t4.. of the
    // first (g4 = 2) or second (g4 = 6) k-step, and 8 channels on for b1
    const bool dlane = (g4 & 3) == 2;
    const uint32_t drow = (uint32_t)8 * a.pitch + (uint32_t)(warp * CWH + (g4 >> 2) * 16 + 2 * t4) * 2;
    const uint32_t stage0 = smem_u32(stages);
    const size_t tab_floats = (size_t)RM_MAXC * RM_NV * RS;

    // coefficient work taken at the end of a token and done one half row later
    int pend_it = -1;
    int64_t pend_t = 0;
    float pend_dl = 0.f;
    auto coefficients = [&]() {
        const int it = pend_it;
        const bool ready = mbar_wait_bounded(&tfull[it & 1], (uint32_t)(it >> 1) & 1u, abort_flag, a.wait);
        const float *rb = red + (size_t)(it & 1) * tab_floats;
        float ss[2], sw[2], sd[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int i = lane + 32 * j, c = i >> 3, ii = i & 7;
            ss[j] = sw[j] = sd[j] = 0.f;
            if (c < C) {
                const float *ps = rb + (c * RM_NV + 16 + ii) * RS;
                const float *pw = rb + (c * RM_NV + ii) * RS;
                const float *pd = rb + (c * RM_NV + 8 + ii) * RS;
#pragma unroll
                for (int w = 0; w < NW; w += 4) {
                    const float4 x = *reinterpret_cast<const float4 *>(ps + w);
                    const float4 y = *reinterpret_cast<const float4 *>(pw + w);
                    const float4 z = *reinterpret_cast<const float4 *>(pd + w);
                    ss[j] += (x.x + x.y) + (x.z + x.w);
                    sw[j] += (y.x + y.y) + (y.z + y.w);
                    sd[j] += (z.x + z.y) + (z.z + z.w);
                }
            }
        }
        // the warp's reads are done: one arrival per warp (its lanes' reads are
        // ordered before lane 0's release by the warp barrier)
        __syncwarp();
        if (lane == 0) mbar_arrive(&tfree[it & 1]);
        float rinv[2], score[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const bool pv = lane + 32 * j < a.n_src;
            const float ms = fmaf(ss[j], a.inv_d, a.eps);
            rinv[j] = ms > 0.f ? rsqrtf(ms) : 0.f;       // 1 / r_i (0 for a zero key)
            score[j] = pv ? sw[j] * rinv[j] : -INFINITY;
        }
        float mx = fmaxf(score[0], score[1]);
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        float e[2], es = 0.f;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            e[j] = lane + 32 * j < a.n_src ? __expf(score[j] - mx) : 0.f;
            es += e[j];
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) es += __shfl_xor_sync(0xffffffffu, es, o);
        // (sums of absent sources may hold anything, even non-finite values:
        // every use below is guarded, not multiplied by a zero weight)
        float alpha[2], mean = 0.f;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            alpha[j] = e[j] / es;
            if (lane + 32 * j < a.n_src) mean = fmaf(alpha[j], sd[j], mean);
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) mean += __shfl_xor_sync(0xffffffffu, mean, o);
        if (ready && !*abort_flag) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int i = lane + 32 * j, c = i >> 3, ii = i & 7;
                if (c >= C) continue;
                const bool pv = i < a.n_src;
                const float ds = alpha[j] * (sd[j] - mean + pend_dl);
                float *out = a.coef + ((size_t)pend_t * C + c) * RM_NV;
                out[ii] = pv ? alpha[j] : 0.f;
                out[8 + ii] = pv ? ds * rinv[j] : 0.f;
                out[16 + ii] = pv ? -ds * sw[j] * rinv[j] * rinv[j] * rinv[j] * a.inv_d : 0.f;
            }
        }
    };

    float d1[2][4], gr[2][4];
    int s = 0, it = 0, pc = 0;                    // stage of part k and its parity; token item, part in it
    uint32_t par = 0;
    for (int k = 0; k < n_parts; ++k) {
        const int c = pc >> 1, h = pc & 1;
        const int64_t t = blockIdx.x + (int64_t)it * gstride;
        if (h == 0) {
#pragma unroll
            for (int u = 0; u < 2; ++u)
#pragma unroll
                for (int e = 0; e < 4; ++e) { d1[u][e] = 0.f; gr[u][e] = 0.f; }
        }
        mbar_wait_bounded(&full[s], par, abort_flag, a.wait);
        const uint32_t sb = stage0 + (uint32_t)s * a.stage_bytes;
        // (one call per half, so the fragment arrays are indexed statically)
        auto pass = [&](const uint32_t(&b)[KS2][2]) {
#pragma unroll
            for (int s2 = 0; s2 < KS2; ++s2) {
                uint32_t x0, x1, x2, x3;
                ldsm_x4(sb + lrow_x + 64 * s2, x0, x1, x2, x3);
                uint32_t b0 = b[s2][0], b1 = b[s2][1];
                if (dlane) {
                    b0 = lds32u(sb + drow + 64 * s2);
                    b1 = lds32u(sb + drow + 64 * s2 + 16);
                }
                // rows 0..7: sources at the first k-step, 8..15 at the second
                mma_full(d1[s2 & 1], x0, x2, x1, x3, b0, b1);
                mma_rows8(gr[0], x0, x1, x0, x1);
                mma_rows8(gr[1], x2, x3, x2, x3);
            }
        };
        if (h == 0) pass(bw[0]);
        else pass(bw[1]);
        // this warp is done with the stage; the last warp to be refills it
        __syncwarp();
        int refill = 0;
        if (lane == 0) {
            __threadfence_block();
            if (atomicAdd(&done[s], 1u) == NW - 1) {
                done[s] = 0;
                refill = k + a.nstages < n_parts && may_issue && !*abort_flag;
            }
        }
        if (__shfl_sync(0xffffffffu, refill, 0)) issue(k + a.nstages, s);
        __syncwarp();
        if (h == 1) {
            // the chunk's sums: lane (i, 0) (w*g).v_i = columns 0 + 1 (first
            // k-step) here and 4 + 5 (second) in lane (i, 2); lane (i, 1)
            // dout.v_i = column 2 here and 6 in lane (i, 3)
            const float e0 = d1[0][0] + d1[1][0], e1 = d1[0][1] + d1[1][1];
            const float e2 = d1[0][2] + d1[1][2], e3 = d1[0][3] + d1[1][3];
            float v = t4 == 0 ? e0 + e1 : t4 == 1 ? e0 : t4 == 2 ? e2 + e3 : e2;
            v += __shfl_xor_sync(0xffffffffu, v, 2);
            const float ssq = (g4 & 1) ? gr[0][1] + gr[1][1] : gr[0][0] + gr[1][0];   // lane (i, i/2)
            if (c == 0 && it >= 2)           // the table of the token two before has been read
                mbar_wait_bounded(&tfree[it & 1], (uint32_t)((it >> 1) - 1) & 1u, abort_flag, a.wait);
            float *rb = red + (size_t)(it & 1) * tab_floats;
            if (t4 < 2) rb[(c * RM_NV + 8 * t4 + g4) * RS + warp] = v;
            if (t4 == (g4 >> 1)) rb[(c * RM_NV + 16 + g4) * RS + warp] = ssq;
            if (c == C - 1) {
                // the warp's table writes are done: one arrival per warp
                __syncwarp();
                if (lane == 0) mbar_arrive(&tfull[it & 1]);
                // the coefficient duty rotates over the warps; the lse gradient
                // is fetched now, the work done one half row later
                if (warp == (it & (NW - 1))) {
                    pend_it = it;
                    pend_t = t;
                    pend_dl = a.dlse != nullptr ? __ldg(a.dlse + t) : 0.f;
                }
            }
        } else if (pend_it >= 0) {
            coefficients();
            pend_it = -1;
        }
        if (++s == a.nstages) { s = 0; par ^= 1u; }
        if (++pc == ppt) { pc = 0; ++it; }
    }
    if (pend_it >= 0) coefficients();
    // copies still in flight (only after an abort) must land before the CTA exits
    __syncthreads();
    if (tid == 0) {
        int never = 0;
        const int issued = (int)*imax;
        for (int k = issued > a.nstages ? issued - a.nstages : 0; k < issued; ++k)
            mbar_wait_bounded(&full[k % a.nstages], (uint32_t)(k / a.nstages) & 1u, &never, a.wait);
    }
}

// ---------------------------------------------------------------- apply
constexpr int RM_TB = 16;             // tokens per coefficient batch
constexpr size_t RM_RING_BYTES = (size_t)RA_DEPTH * RM_ROWS * RA_THREADS * 8;

struct ReadBwdApplyManyArgs {
    const unsigned char *src;
    int64_t src_stride_bytes;
    int n_src;
    int C;
    int64_t T;
    int d;                            // a multiple of RA_W
    const float *query;
    const float *gain;
    const unsigned char *dout;        // [T][d]
    const float *coef;                // [T][C][24]
    unsigned char *dsrc;
    int64_t dsrc_stride_bytes;
    int accumulate;
    float *ws;                        // [gridDim.y][d] partial U
    int64_t tpc;                      // tokens per CTA
};

template <int NQ>   // 1: the form of one query
__global__ void __launch_bounds__(RA_THREADS, 2) read_bwd_apply_many_kernel(const ReadBwdApplyManyArgs a) {
    static_assert(NQ == 1, "one query");
    // per token of the batch, chunk and source: alpha, ds/r, the v term, pad
    __shared__ __align__(16) float cs[RM_TB][RM_MAXC][8][4];
    extern __shared__ __align__(16) uint2 ring[];
    const int tid = threadIdx.x;
    const int C = a.C;
    const int c = blockIdx.x * RA_W + 4 * tid;             // first of this thread's 4 channels
    const int64_t t0 = (int64_t)blockIdx.y * a.tpc;
    const int64_t t1 = t0 + a.tpc < a.T ? t0 + a.tpc : a.T;
    const int64_t nunits = (t1 > t0 ? t1 - t0 : 0) * C;

    float4 w = *reinterpret_cast<const float4 *>(a.query + c);
    if (a.gain) {
        const float4 g = *reinterpret_cast<const float4 *>(a.gain + c);
        w.x *= g.x; w.y *= g.y; w.z *= g.z; w.w *= g.w;
    }
    const float2 wg[2] = {make_float2(w.x, w.y), make_float2(w.z, w.w)};
    float2 U[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};

    const uint32_t ring0 = smem_u32(ring) + (uint32_t)tid * 8;
    auto slot_addr = [&](int slot, int row) { return ring0 + (uint32_t)((slot * RM_ROWS + row) * RA_THREADS) * 8; };
    // unit u = (token t0 + u / C, chunk u % C): the chunk's rows, and with the
    // first chunk the gradient row, into ring slot `slot` (one commit group
    // per unit, empty past the range).  Units are issued in order; the next
    // one's token and chunk are counted, not divided out.
    int64_t iu = 0, it_tok = t0;
    int it_ch = 0;
    auto issue = [&](int slot) {
        if (iu < nunits) {
            const int64_t tt = it_tok;
            const int ch = it_ch;
            const int nc = a.n_src - 8 * ch < 8 ? a.n_src - 8 * ch : 8;
            const size_t off = ((size_t)tt * a.d + c) * 2;
            for (int i = 0; i < nc; ++i)
                cp_async8(slot_addr(slot, i), a.src + (int64_t)(8 * ch + i) * a.src_stride_bytes + off);
            if (ch == 0) cp_async8(slot_addr(slot, 8), a.dout + off);
        }
        cp_async_commit();
        ++iu;
        if (++it_ch == C) { it_ch = 0; ++it_tok; }
    };
    issue(0);
    issue(1);

    int slot = 0;
    for (int64_t tb = t0; tb < t1; tb += RM_TB) {
        const int nb = t1 - tb < RM_TB ? (int)(t1 - tb) : RM_TB;
        __syncthreads();                                    // the previous batch is consumed
        for (int idx = tid; idx < nb * C * 8; idx += RA_THREADS) {
            const int tok = idx / (C * 8), rem = idx - tok * C * 8;
            const int ch = rem >> 3, i = rem & 7;
            const float *s = a.coef + ((size_t)(tb + tok) * C + ch) * RM_NV;
            *reinterpret_cast<float4 *>(&cs[tok][ch][i][0]) = make_float4(s[i], s[8 + i], s[16 + i], 0.f);
        }
        __syncthreads();
        for (int tok = 0; tok < nb; ++tok) {
            const int64_t t = tb + tok;
            const size_t off = ((size_t)t * a.d + c) * 2;
            float2 dl[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
            for (int ch = 0; ch < C; ++ch) {
                // unit u+2 into the slot unit u-1 used (this thread's reads of it
                // are consumed by the arithmetic below before this issue)
                issue(slot == 0 ? RA_DEPTH - 1 : slot - 1);     // unit u + 2
                cp_async_wait<2>();                         // unit u's rows have landed
                if (ch == 0) {
                    const uint2 r = lds64(slot_addr(slot, 8));
                    dl[0] = bf2_to_f2(r.x);
                    dl[1] = bf2_to_f2(r.y);
                }
                const int nc = a.n_src - 8 * ch < 8 ? a.n_src - 8 * ch : 8;
                for (int i = 0; i < nc; ++i) {
                    const float4 k4 = *reinterpret_cast<const float4 *>(&cs[tok][ch][i][0]);
                    const uint2 xr = lds64(slot_addr(slot, i));
                    const float2 x[2] = {bf2_to_f2(xr.x), bf2_to_f2(xr.y)};
                    unsigned char *gp = a.dsrc + (int64_t)(8 * ch + i) * a.dsrc_stride_bytes + off;
                    uint2 zr = make_uint2(0u, 0u);
                    if (a.accumulate) zr = *reinterpret_cast<const uint2 *>(gp);
                    float2 y[2];
#pragma unroll
                    for (int p = 0; p < 2; ++p) {
                        y[p] = fmul2(make_float2(k4.z, k4.z), x[p]);
                        y[p] = ffma2(make_float2(k4.x, k4.x), dl[p], y[p]);
                        y[p] = ffma2(make_float2(k4.y, k4.y), wg[p], y[p]);
                        U[p] = ffma2(make_float2(k4.y, k4.y), x[p], U[p]);
                    }
                    if (a.accumulate) {
                        const float2 z0 = bf2_to_f2(zr.x), z1 = bf2_to_f2(zr.y);
                        y[0] = make_float2(y[0].x + z0.x, y[0].y + z0.y);
                        y[1] = make_float2(y[1].x + z1.x, y[1].y + z1.y);
                    }
                    stg64_cs(gp, make_uint2(f2_to_bf2(y[0].x, y[0].y), f2_to_bf2(y[1].x, y[1].y)));
                }
                slot = slot == RA_DEPTH - 1 ? 0 : slot + 1;
            }
        }
    }
    cp_async_wait<0>();
    *reinterpret_cast<float4 *>(a.ws + (size_t)blockIdx.y * a.d + c) = make_float4(U[0].x, U[0].y, U[1].x, U[1].y);
}

}  // namespace attnres
