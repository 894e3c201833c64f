// read_bwd_split.cuh -- the backward of the depth read in two kernels
// (sm_103a), for bf16 sources, at most 8 of them, and 3 or 4 queries.
//
// The operation is the one of read_bwd.cuh (per token, alpha recomputed from
// the sources, r_i = sqrt(mean(v_i^2) + eps)):
//     ds_qi = alpha_qi (dout_q . v_i - sum_j alpha_qj dout_q . v_j + dlse_q)
//     b_qi  = ds_qi / r_i,   c_i = - sum_q ds_qi ((w_q*g) . v_i) / (d r_i^3)
//     dv_i  = sum_q alpha_qi dout_q + sum_q b_qi (w_q*g) + c_i v_i
//     U_q  += sum_i b_qi v_i,   dq_q = g * U_q,   dgain = sum_q w_q * U_q.
// A token's coefficients (alpha, b, c) need sums over the whole row, while
// U needs sums over all tokens for every channel.  One kernel that does both
// holds U and w*g for every channel of the row in each SM (with 4 queries at
// d = 4096 that is the whole register file), so here the two directions are
// separate launches:
//
// read_bwd_coef_kernel: per token, the row sums (w_q*g).v_i, dout_q.v_i and
// v_i.v_i on the tensor cores (mma.sync m16n8k16 on ldmatrix fragments, the
// queries split into bf16 hi + lo parts as in the forward read) go to a
// double-buffered table, then per head one warp forms the softmax and the
// coefficients and writes them: coef[t][head] = {alpha[q*8+i] (32),
// b[q*8+i] (32), c[i] (8)}.  The table is handed over by mbarriers, not a
// CTA barrier (each warp arrives on "full" after its writes; the coefficient
// warps wait on it and arrive on "free" after their reads, which the writers
// of the token two later wait on), the coefficient duty
// rotates over the warps from token to token, and a warp does a token's
// coefficients after its first half of the next token (the lse gradient
// fetched when the duty is taken), so neither the softmax nor its loads hold
// up the ring of stages.
// Nothing else is written, so no row has to stay in shared memory after its
// sums: the rows stream through a ring of half-row stages (all 8 source rows
// and the query gradient rows of one half of the channels), which keeps 1.5
// tokens of loads in flight where two whole-row stages would leave one; the
// warp that finishes a half last refills its stage (a shared counter), so no
// warp waits for another to release a stage.
//
// read_bwd_apply_kernel: a CTA owns 1024 channels (4 per thread) and a
// contiguous range of tokens; it reads the tokens' coefficients (staged in
// shared memory in batches), its channels of the source and gradient rows
// (cp.async, two tokens ahead), writes dv and keeps U for its channels in
// registers, then writes U to a per-CTA partial that read_bwd_finish_kernel
// sums in a fixed order.
//
// Traffic: the sources and the gradient rows are read twice (once per
// kernel), about 1.6x the essential bytes at 8 sources and 4 queries, in
// exchange for two kernels that each stream at close to the memory rate.
#pragma once

#include "depth_read_mma.cuh"

namespace attnres {

constexpr int RC_NW = 16;             // warps of the coefficient kernel
constexpr int RC_MAX_STAGES = 8;
constexpr int RC_NV = 72;             // row sums per column: (w*g).v 32, dout.v 32, v.v 8
constexpr int RC_RS = 36;             // table row stride in floats (32 columns, float4-aligned)
constexpr size_t RC_AUX_BYTES = 256 + (size_t)2 * RC_NV * RC_RS * 4;
constexpr bool RC_GRAM = true;        // sums of squares: Gram MMAs (true) or packed FMAs

struct ReadBwdCoefArgs {
    const unsigned char *src;         // source 0, token 0 (bf16)
    int64_t src_stride_bytes;
    int n_src;                        // <= 8
    int64_t T;
    int d;                            // 2048 or 4096
    int n_q;                          // <= NQ
    int H;                            // heads (per-head sums and coefficients)
    const float *queries;             // [n_q][d]
    const float *gain;                // [d] or nullptr
    float eps;
    float inv_dh;                     // 1 / channels per head
    const unsigned char *dout;        // [n_q][T][d] bf16
    const float *dlse;                // [n_q][T] or nullptr (H == 1)
    float *coef;                      // [T][H][72]
    int nstages;
    uint32_t pitch;                   // bytes between rows of a stage (d + 16: half a row, padded)
    uint32_t stage_bytes;             // 12 rows
    WaitCfg wait;
};

__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t &r0, uint32_t &r1) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}

// Fragments of the queries (gain folded in) for the warp's channels of one
// half row, query q = g4/2, bf16 hi part in column 2q, lo part in 2q+1.
template <int KSH>
__device__ __forceinline__ void rc_query_fragments(const ReadBwdCoefArgs &a, int cbase, int g4, int t4,
                                                   uint32_t (&bq)[KSH][2]) {
    DepthReadMmaArgs m;
    m.queries = a.queries;
    m.gain = a.gain;
    m.d = a.d;
    m.n_q = a.n_q;
    dm_query_fragments<KSH>(m, cbase, g4, t4, bq);
}

// KSH: MMA k-steps (16 channels) per warp and half row: d / (2 * 16 * RC_NW).
template <int NQ, int KSH>
__global__ void __launch_bounds__(RC_NW * 32, 1) read_bwd_coef_kernel(const ReadBwdCoefArgs a) {
    static_assert(NQ >= 1 && NQ <= 4, "at most 4 queries");
    static_assert(KSH % 2 == 0, "k-steps in pairs (one ldmatrix.x4 each)");
    constexpr int NW = RC_NW;
    constexpr int CWH = KSH * 16;                 // channels per warp and half row
    constexpr int RS = RC_RS;

    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char *stages = smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)a.nstages * a.stage_bytes);
    // warps done with each stage; the last one to finish a half refills its stage
    unsigned *done = reinterpret_cast<unsigned *>(full + RC_MAX_STAGES);
    unsigned *imax = done + RC_MAX_STAGES;         // halves issued so far
    uint64_t *tfull = full + 2 * RC_MAX_STAGES;   // [2] table of token it&1 written
    uint64_t *tfree = tfull + 2;                  // [2] table of token it&1 read
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tfree + 2);
    float *red = reinterpret_cast<float *>(smem + (size_t)a.nstages * a.stage_bytes + 256);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int g4 = lane >> 2, t4 = lane & 3;
    const int half_bytes = a.d;                   // d/2 bf16 channels

    if (tid == 0) {
        for (int s = 0; s < a.nstages; ++s) {
            mbar_init(&full[s], 1);
            done[s] = 0;
        }
        *imax = 0;
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], NW);
            mbar_init(&tfree[b], a.H);
        }
        *abort_flag = 0;
        mbar_init_fence();
    }
    // rows never loaded (absent sources 8.., absent gradient rows) enter the
    // MMAs times nothing that is used: keep them zero, not stale bits
    for (int s = 0; s < a.nstages; ++s)
        for (int row = 0; row < 12; ++row) {
            if ((row < 8 && row < a.n_src) || (row >= 8 && row - 8 < a.n_q)) continue;
            for (int b = tid * 16; b < half_bytes; b += NW * 32 * 16)
                *reinterpret_cast<uint4 *>(stages + (size_t)s * a.stage_bytes + (size_t)row * a.pitch + b) =
                    make_uint4(0u, 0u, 0u, 0u);
        }
    __syncthreads();

    const int gstride = gridDim.x;
    const int n_items = blockIdx.x < a.T ? (int)((a.T - blockIdx.x + gstride - 1) / gstride) : 0;
    const int n_halves = 2 * n_items;

    // ------------------------------------------------------------ producer
    // half k (token item k/2, channel half k%2) into stage k % nstages, by a
    // whole warp: lane 0 arms the stage's barrier, then lane i copies row i
    // (a single lane issuing every row's bulk copy was the pace of the ring).
    // The first nstages by warp 0, each later one by the warp that finishes
    // the half nstages before it last.
    const bool may_issue = !a.wait.inject_stall;
    const uint64_t pol = l2_policy_evict_first();
    auto issue = [&](int k, int s) {               // s = k % nstages
        const int64_t t = blockIdx.x + (int64_t)(k >> 1) * gstride;
        const int64_t off = (t * a.d + (int64_t)(k & 1) * (a.d / 2)) * 2;
        unsigned char *dst = stages + (size_t)s * a.stage_bytes;
        if (lane == 0) {
            mbar_arrive_expect_tx(&full[s], (uint32_t)half_bytes * (uint32_t)(a.n_src + a.n_q));
            atomicMax(imax, (unsigned)(k + 1));
        }
        __syncwarp();
        if (lane < a.n_src)
            bulk_g2s(dst + (size_t)lane * a.pitch, a.src + (int64_t)lane * a.src_stride_bytes + off,
                     (uint32_t)half_bytes, &full[s], pol);
        else if (lane >= 8 && lane - 8 < a.n_q)
            bulk_g2s(dst + (size_t)lane * a.pitch, a.dout + (int64_t)(lane - 8) * a.T * a.d * 2 + off,
                     (uint32_t)half_bytes, &full[s], pol);
    };
    if (warp == 0 && may_issue)
        for (int k = 0; k < n_halves && k < a.nstages; ++k) issue(k, k);

    // ------------------------------------------------------------ constants
    uint32_t bq[2][KSH][2];
    rc_query_fragments<KSH>(a, warp * CWH, g4, t4, bq[0]);
    rc_query_fragments<KSH>(a, a.d / 2 + warp * CWH, g4, t4, bq[1]);
    // ldmatrix rows of this lane: source row lane%8 / gradient row lane%4 (rows
    // 4..7 of the gradient matrix repeat 0..3 and meet unused columns), channel
    // block lane/8 of a 32-channel group of this warp's slice
    const uint32_t colb = (uint32_t)(warp * CWH + 8 * (lane >> 3)) * 2;
    const uint32_t lrow_x = (uint32_t)(lane & 7) * a.pitch + colb;
    // gradient rows as the B operand of the packed dots (ldmatrix .x2, lanes
    // 0..15): matrix j = (lane/8)&1 holds channels +8j, its rows 0..3 the
    // gradient rows at the first k-step of the 32-channel group, rows 4..7 at
    // the second (+16 channels)
    const uint32_t lrow_d = (uint32_t)(8 + (lane & 3)) * a.pitch +
                            (uint32_t)(warp * CWH + 8 * ((lane >> 3) & 1) + 16 * ((lane >> 2) & 1)) * 2;
    const uint32_t stage0 = smem_u32(stages);
    // table columns: one per warp with one head (both halves summed), else one
    // per (half, warp) ("virtual warp" of CWH channels, in row order)
    const bool per_half = a.H > 1;
    const int ncol = per_half ? 2 * NW / a.H : NW;     // columns of a head

    // coefficient work taken at the end of a token and done one half later
    int pend_it = -1, pend_head = 0;
    int64_t pend_t = 0;
    float pend_dl = 0.f;
    auto coefficients = [&]() {
        const int it = pend_it, chead = pend_head;
        const bool ready = mbar_wait_bounded(&tfull[it & 1], (uint32_t)(it >> 1) & 1u, abort_flag, a.wait);
        // lane (q, i) = q*8 + i: the head's sums, softmax and coefficients
        const float *rb = red + (size_t)(it & 1) * RC_NV * RS;
        const int q = lane >> 3, i = lane & 7;
        const int c0 = chead * ncol;
        float ss = 0.f, sw = 0.f, sd = 0.f;
        const float *ps = rb + (64 + i) * RS + c0;
        const float *pw = rb + (q * 8 + i) * RS + c0;
        const float *pd = rb + (32 + q * 8 + i) * RS + c0;
        if (q < NQ) {
            if (ncol % 4 == 0) {
                for (int c = 0; c < ncol; c += 4) {
                    const float4 x = *reinterpret_cast<const float4 *>(ps + c);
                    const float4 y = *reinterpret_cast<const float4 *>(pw + c);
                    const float4 z = *reinterpret_cast<const float4 *>(pd + c);
                    ss += (x.x + x.y) + (x.z + x.w);
                    sw += (y.x + y.y) + (y.z + y.w);
                    sd += (z.x + z.y) + (z.z + z.w);
                }
            } else {
                for (int c = 0; c < ncol; ++c) { ss += ps[c]; sw += pw[c]; sd += pd[c]; }
            }
        }
        // the warp's reads are done: one arrival per warp (its lanes' reads are
        // ordered before lane 0's release by the warp barrier)
        __syncwarp();
        if (lane == 0) mbar_arrive(&tfree[it & 1]);
        const bool pv = q < a.n_q && i < a.n_src;
        const float ms = fmaf(ss, a.inv_dh, a.eps);
        const float rinv = ms > 0.f ? rsqrtf(ms) : 0.f;  // 1 / r_i (0 for a zero key)
        const float score = pv ? sw * rinv : -INFINITY;
        const float mx = seg_max<8>(score);
        const float e = pv ? __expf(score - mx) : 0.f;
        // every lane takes part in the shuffles
        const float esum = seg_sum<8>(e);
        const float alpha = pv ? e / esum : 0.f;
        const float mean = seg_sum<8>(alpha * sd);
        const float ds = pv ? alpha * (sd - mean + pend_dl) : 0.f;
        const float b = ds * rinv;
        float cp = -ds * sw * rinv * rinv * rinv * a.inv_dh;
        cp += __shfl_xor_sync(0xffffffffu, cp, 8);
        cp += __shfl_xor_sync(0xffffffffu, cp, 16);
        if (ready && !*abort_flag) {
            float *out = a.coef + ((size_t)pend_t * a.H + chead) * RC_NV;
            out[lane] = alpha;
            out[32 + lane] = b;
            if (lane < 8) out[64 + lane] = cp;
        }
    };

    float d1[2][4], dd[2][4], gr[2][4];
    float2 sq = make_float2(0.f, 0.f);
    int s = 0;                                    // stage of half k, and its phase parity
    uint32_t par = 0;
    for (int k = 0; k < n_halves; ++k) {
        const int it = k >> 1, h = k & 1;
        const int64_t t = blockIdx.x + (int64_t)it * gstride;
        if (h == 0 || per_half) {
#pragma unroll
            for (int u = 0; u < 2; ++u)
#pragma unroll
                for (int e = 0; e < 4; ++e) { d1[u][e] = 0.f; dd[u][e] = 0.f; gr[u][e] = 0.f; }
            sq = make_float2(0.f, 0.f);
        }
        mbar_wait_bounded(&full[s], par, abort_flag, a.wait);
        const uint32_t sb = stage0 + (uint32_t)s * a.stage_bytes;
        // (one call per half, so the fragment arrays are indexed statically)
        auto pass = [&](const uint32_t(&b)[KSH][2]) {
#pragma unroll
            for (int s2 = 0; s2 < KSH / 2; ++s2) {
                uint32_t x0, x1, x2, x3, e0, e1;
                ldsm_x4(sb + lrow_x + 64 * s2, x0, x1, x2, x3);
                ldsm_x2(sb + lrow_d + 64 * s2, e0, e1);
                mma_rows8(d1[0], x0, x1, b[2 * s2][0], b[2 * s2][1]);
                mma_rows8(d1[1], x2, x3, b[2 * s2 + 1][0], b[2 * s2 + 1][1]);
                // rows 0..7: sources at the first k-step, 8..15 at the second;
                // columns 0..3 meet the first, 4..7 the second k-step's gradients
                mma_full(dd[s2 & 1], x0, x2, x1, x3, e0, e1);
                if constexpr (RC_GRAM) {
                    mma_rows8(gr[0], x0, x1, x0, x1);
                    mma_rows8(gr[1], x2, x3, x2, x3);
                } else {
                    const float2 f0 = bf2_to_f2(x0), f1 = bf2_to_f2(x1), f2 = bf2_to_f2(x2), f3 = bf2_to_f2(x3);
                    sq = ffma2(f0, f0, sq);
                    sq = ffma2(f1, f1, sq);
                    sq = ffma2(f2, f2, sq);
                    sq = ffma2(f3, f3, sq);
                }
            }
        };
        if (h == 0) pass(bq[0]);
        else pass(bq[1]);
        // this warp is done with the stage; the last warp to be refills it
        __syncwarp();
        int refill = 0;
        if (lane == 0) {
            __threadfence_block();
            if (atomicAdd(&done[s], 1u) == NW - 1) {
                done[s] = 0;
                refill = k + a.nstages < n_halves && may_issue && !*abort_flag;
            }
        }
        if (__shfl_sync(0xffffffffu, refill, 0)) issue(k + a.nstages, s);
        __syncwarp();
        if (per_half || h == 1) {
            // the first write of this token's table waits until the coefficient
            // warps of the token two before have read it
            if ((h == 0 || !per_half) && it >= 2)
                mbar_wait_bounded(&tfree[it & 1], (uint32_t)((it >> 1) - 1) & 1u, abort_flag, a.wait);
            // lane (i = g4, q = t4): (w_q*g).v_i in columns 2q (hi) + 2q+1 (lo);
            // lane (i, t4 < 2): dout.v_i of queries 2t4 and 2t4+1, the first
            // k-steps' part in c0, c1 here, the second's in c2, c3 of lane t4+2
            const float dw = (d1[0][0] + d1[1][0]) + (d1[0][1] + d1[1][1]);
            float dq0 = (t4 < 2) ? dd[0][0] + dd[1][0] : dd[0][2] + dd[1][2];
            float dq1 = (t4 < 2) ? dd[0][1] + dd[1][1] : dd[0][3] + dd[1][3];
            dq0 += __shfl_xor_sync(0xffffffffu, dq0, 2);
            dq1 += __shfl_xor_sync(0xffffffffu, dq1, 2);
            float ss;
            if constexpr (RC_GRAM) {
                // the Gram diagonal: lane (i, i/2), element i&1
                ss = (g4 & 1) ? gr[0][1] + gr[1][1] : gr[0][0] + gr[1][0];
            } else {
                ss = sq.x + sq.y;
                ss += __shfl_xor_sync(0xffffffffu, ss, 1);
                ss += __shfl_xor_sync(0xffffffffu, ss, 2);
            }
            const int col = per_half ? h * NW + warp : warp;
            float *rb = red + (size_t)(it & 1) * RC_NV * RS;
            if (t4 < NQ) rb[(t4 * 8 + g4) * RS + col] = dw;
            if (2 * t4 < NQ) rb[(32 + 2 * t4 * 8 + g4) * RS + col] = dq0;
            if (2 * t4 + 1 < NQ) rb[(32 + (2 * t4 + 1) * 8 + g4) * RS + col] = dq1;
            if (t4 == (RC_GRAM ? g4 >> 1 : 0)) rb[(64 + g4) * RS + col] = ss;
        }
        if (h == 1) {
            // the warp's table writes are done: one arrival per warp
            __syncwarp();
            if (lane == 0) mbar_arrive(&tfull[it & 1]);
            // head whose coefficients this warp forms for this token (the duty
            // rotates: head hd goes to warp (hd + it*H) % NW); the work itself
            // waits until after this warp's first half of the next token, when
            // every warp has long written the table, and the lse gradient it
            // needs is fetched now
            const int hd = (warp - it * a.H) & (NW - 1);
            if (hd < a.H) {
                pend_it = it;
                pend_t = t;
                pend_head = hd;
                const int q = lane >> 3, i = lane & 7;
                pend_dl = (a.dlse != nullptr && q < a.n_q && i < a.n_src) ? __ldg(a.dlse + (int64_t)q * a.T + t) : 0.f;
            }
        } else if (pend_it >= 0) {
            coefficients();
            pend_it = -1;
        }
        if (++s == a.nstages) { s = 0; par ^= 1u; }
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
constexpr int RA_THREADS = 256;
constexpr int RA_W = 4 * RA_THREADS;  // channels per CTA
constexpr int RA_TB = 16;             // tokens per coefficient batch
constexpr int RA_HS = 4;              // most heads in a CTA's channels (heads of >= 256 channels)

struct ReadBwdApplyArgs {
    const unsigned char *src;
    int64_t src_stride_bytes;
    int n_src;
    int64_t T;
    int d;                            // a multiple of RA_W
    int H;
    int dh;                           // channels per head, a multiple of 256
    int n_q;                          // == NQ
    const float *queries;
    const float *gain;
    const unsigned char *dout;        // [n_q][T][d]
    const float *coef;                // [T][H][72]
    unsigned char *dsrc;
    int64_t dsrc_stride_bytes;
    int accumulate;
    float *ws;                        // [gridDim.y][n_q][d] partial U
    int64_t tpc;                      // tokens per CTA
};

__device__ __forceinline__ uint2 ldg64_nc(const void *p) {
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}
__device__ __forceinline__ void stg64_cs(void *p, uint2 v) {
    asm volatile("st.global.cs.v2.u32 [%0], {%1,%2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
}

__device__ __forceinline__ void cp_async8(uint32_t dst_smem, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst_smem), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }
__device__ __forceinline__ uint2 lds64(uint32_t a) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
    return v;
}

// A thread's rows of a token (4 gradient rows, then up to 8 source rows, 8
// bytes each) arrive by cp.async into a thread-private ring of RA_DEPTH
// tokens in dynamic shared memory, laid out [token slot][row][thread] so a
// warp's accesses are consecutive.
constexpr int RA_DEPTH = 3;
constexpr size_t RA_RING_BYTES = (size_t)RA_DEPTH * 12 * RA_THREADS * 8;

template <int NQ>
__global__ void __launch_bounds__(RA_THREADS, 2) read_bwd_apply_kernel(const ReadBwdApplyArgs a) {
    // per token of the batch, head of the slice and source: alpha_q (4), b_q (4), c, pad
    __shared__ __align__(16) float cs[RA_TB][RA_HS][8][12];
    extern __shared__ __align__(16) uint2 ring[];
    const int tid = threadIdx.x;
    const int c = blockIdx.x * RA_W + 4 * tid;             // first of this thread's 4 channels
    const int hs0 = (blockIdx.x * RA_W) / a.dh;            // first head of the slice
    const int hh = c / a.dh - hs0;
    const int nhs = a.dh >= RA_W ? 1 : RA_W / a.dh;
    const int64_t t0 = (int64_t)blockIdx.y * a.tpc;
    const int64_t t1 = t0 + a.tpc < a.T ? t0 + a.tpc : a.T;

    float2 wg[NQ][2], U[NQ][2];
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
        float4 w = *reinterpret_cast<const float4 *>(a.queries + (size_t)q * a.d + c);
        if (a.gain) {
            const float4 g = *reinterpret_cast<const float4 *>(a.gain + c);
            w.x *= g.x; w.y *= g.y; w.z *= g.z; w.w *= g.w;
        }
        wg[q][0] = make_float2(w.x, w.y);
        wg[q][1] = make_float2(w.z, w.w);
        U[q][0] = U[q][1] = make_float2(0.f, 0.f);
    }
    const size_t rowq = (size_t)a.T * a.d * 2;              // bytes between query gradient tensors
    const uint32_t ring0 = smem_u32(ring) + (uint32_t)tid * 8;
    auto slot_addr = [&](int slot, int row) { return ring0 + (uint32_t)((slot * 12 + row) * RA_THREADS) * 8; };
    // the rows of token tt into ring slot `slot` (one commit group per token,
    // empty past the range)
    auto issue = [&](int64_t tt, int slot) {
        if (tt < t1) {
            const size_t off = ((size_t)tt * a.d + c) * 2;
#pragma unroll
            for (int q = 0; q < NQ; ++q) cp_async8(slot_addr(slot, q), a.dout + q * rowq + off);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (i < a.n_src) cp_async8(slot_addr(slot, 4 + i), a.src + i * a.src_stride_bytes + off);
        }
        cp_async_commit();
    };
    issue(t0, 0);
    issue(t0 + 1, 1);

    int slot = 0;
    for (int64_t tb = t0; tb < t1; tb += RA_TB) {
        const int nb = t1 - tb < RA_TB ? (int)(t1 - tb) : RA_TB;
        __syncthreads();                                    // the previous batch is consumed
        for (int idx = tid; idx < nb * nhs * 8; idx += RA_THREADS) {
            const int tok = idx / (nhs * 8), rem = idx - tok * nhs * 8;
            const int h2 = rem >> 3, i = rem & 7;
            const float *s = a.coef + ((size_t)(tb + tok) * a.H + hs0 + h2) * RC_NV;
            float *dst = &cs[tok][h2][i][0];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                dst[q] = s[q * 8 + i];
                dst[4 + q] = s[32 + q * 8 + i];
            }
            dst[8] = s[64 + i];
        }
        __syncthreads();
        for (int tok = 0; tok < nb; ++tok) {
            const int64_t t = tb + tok;
            // token t+2 into the slot token t-1 used (read by this thread only,
            // and consumed by the arithmetic below before this issue)
            issue(t + 2, slot == 0 ? 2 : slot - 1);
            cp_async_wait<2>();                             // token t's rows have landed
            const size_t off = ((size_t)t * a.d + c) * 2;
            float2 dl[NQ][2];
#pragma unroll
            for (int q = 0; q < NQ; ++q) {
                const uint2 r = lds64(slot_addr(slot, q));
                dl[q][0] = bf2_to_f2(r.x);
                dl[q][1] = bf2_to_f2(r.y);
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (i >= a.n_src) break;
                const float4 al = *reinterpret_cast<const float4 *>(&cs[tok][hh][i][0]);
                const float4 bb = *reinterpret_cast<const float4 *>(&cs[tok][hh][i][4]);
                const float ci = cs[tok][hh][i][8];
                const float alq[4] = {al.x, al.y, al.z, al.w}, bq[4] = {bb.x, bb.y, bb.z, bb.w};
                const uint2 xr = lds64(slot_addr(slot, 4 + i));
                const float2 x[2] = {bf2_to_f2(xr.x), bf2_to_f2(xr.y)};
                unsigned char *gp = a.dsrc + i * a.dsrc_stride_bytes + off;
                uint2 zr = make_uint2(0u, 0u);
                if (a.accumulate) zr = *reinterpret_cast<const uint2 *>(gp);
                float2 y[2];
#pragma unroll
                for (int p = 0; p < 2; ++p) {
                    y[p] = fmul2(make_float2(ci, ci), x[p]);
#pragma unroll
                    for (int q = 0; q < NQ; ++q) {
                        y[p] = ffma2(make_float2(alq[q], alq[q]), dl[q][p], y[p]);
                        y[p] = ffma2(make_float2(bq[q], bq[q]), wg[q][p], y[p]);
                        U[q][p] = ffma2(make_float2(bq[q], bq[q]), x[p], U[q][p]);
                    }
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
    cp_async_wait<0>();
    // this CTA's U: one partial per token range
#pragma unroll
    for (int q = 0; q < NQ; ++q)
        *reinterpret_cast<float4 *>(a.ws + ((size_t)blockIdx.y * a.n_q + q) * a.d + c) =
            make_float4(U[q][0].x, U[q][0].y, U[q][1].x, U[q][1].y);
}

}  // namespace attnres
