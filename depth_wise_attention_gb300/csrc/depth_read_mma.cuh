// depth_read_mma.cuh -- tensor-core variant of the fused depth read (sm_103a).
//
// Same operation as depth_read.cuh (Full AttnRes / Block phase 1 / MHAR):
// per token, s_qi = (w_q * g) . v_i / sqrt(mean(v_i^2) + eps), softmax over
// the sources i, o_q = sum_i alpha_qi v_i, lse_q.  Used for bf16 sources
// with at most 8 sources and 4 queries and d a multiple of 128.
//
// The per-token work is two small dense contractions, done with warp-level
// mma.sync.m16n8k16 (bf16 inputs, fp32 accumulation) straight from the
// shared-memory stage (ldmatrix), so no element is unpacked:
//   pass 1:  D1 = X Q over the warp's channel slice, where X = [8 sources x
//            16 channels] (rows 8..15 zero), Q = the queries split into bf16
//            hi + lo parts (columns 2q, 2q+1), so dot_qi = D1[i][2q] +
//            D1[i][2q+1]; sum(v_i^2) is accumulated with packed FMAs on the
//            same ldmatrix fragments;
//   pass 2:  O^T = X'^T A per 16-channel block: X'^T = [16 channels x (8
//            sources | the same 8 sources)] (ldmatrix .trans), A = [(8 sources
//            hi | 8 sources lo) x 4 queries] holding alpha split into bf16 hi
//            and lo parts; movmatrix turns the result back into channel pairs
//            per query, which are staged in the shared-memory rows this warp
//            has finished reading and leave with one bulk store per query.
// The hi/lo split keeps the queries and the weights to about 16 mantissa
// bits; products are exact and sums are fp32.
//
// Work split: one token per item; warp w of NW owns channels [w*cw, (w+1)*cw)
// (cw = d/NW); its partial dots and sums of squares go to a small shared
// table, one CTA barrier publishes them, and each warp computes the softmax
// of its head (all NW warps for H = 1) redundantly.  Stages, producer and
// bounded waits are as in depth_read.cuh; source rows in a stage are padded
// by 16 bytes so ldmatrix row addresses fall in distinct banks.
#pragma once

#include "common.cuh"

namespace attnres {

constexpr int DM_MAX_WARPS = 16;
constexpr int DM_MAX_STAGES = 6;

struct DepthReadMmaArgs {
    const unsigned char *src;
    int64_t src_stride_bytes;
    int n_src;                    // <= 8
    int64_t T;
    int d;
    int n_q;                      // <= NQ
    int H;                        // heads
    int wph;                      // warps per head (NW / H)
    const float *queries;         // [n_q][d]
    const float *gain;            // [d] or nullptr
    float eps;
    unsigned char *out;           // [n_q][T][d] bf16
    int64_t out_q_stride_bytes;
    float *lse;                   // [n_q][H][T] or nullptr
    int nstages;
    uint32_t pitch;               // bytes between source rows in a stage (2d + 16)
    uint32_t stage_bytes;
    WaitCfg wait;
};

struct DMLayout {
    static constexpr size_t bar_bytes = 128;
    // red[2][40 values per token][RS]: for each value (dots q*8+i, then sums
    // of squares 32+i) the partial of every warp; row stride RS = 20 floats
    // keeps the 16-float rows 16-byte aligned and the writes at most 4-way
    // conflicting; two tokens per item use 80 values
    static constexpr int RS = 20;
    static constexpr size_t red_floats = 2 * 80 * RS;
    static constexpr size_t aux_bytes = bar_bytes + 4 * red_floats;
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                          uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
// D += A B, m16n8k16, bf16 x bf16 -> fp32.  a1 = a3 = 0 (rows 8..15 unused).
__device__ __forceinline__ void mma_rows8(float (&c)[4], uint32_t a0, uint32_t a2, uint32_t b0,
                                          uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
}

// Full m16n8k16 with all four A registers given.
__device__ __forceinline__ void mma_full(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// Transpose an 8x8 matrix of 16-bit elements held one row pair per lane.
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}
// Store four 8x8 matrices of 16-bit elements transposed: lane 8j + r gives
// the shared address of stored row r of matrix j (= column r of the fragment).
__device__ __forceinline__ void stsm_x4_t(uint32_t addr, uint32_t r0, uint32_t r1, uint32_t r2,
                                          uint32_t r3) {
    asm volatile("stmatrix.sync.aligned.m8n8.x4.trans.shared.b16 [%0], {%1,%2,%3,%4};" ::"r"(addr),
                 "r"(r0), "r"(r1), "r"(r2), "r"(r3)
                 : "memory");
}
__device__ __forceinline__ void sts32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
// Shared -> global bulk copy (bytes % 16 == 0, both 16-byte aligned).
__device__ __forceinline__ void bulk_s2g(void *gdst, uint32_t ssrc, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst), "r"(ssrc),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// bf16 hi/lo split of x: hi = rn(x), lo = rn(x - hi).
__device__ __forceinline__ void split_bf16(float x, float &hi, float &lo) {
    hi = __bfloat162float(__float2bfloat16_rn(x));
    lo = x - hi;
}
__device__ __forceinline__ uint32_t pack_bf16(float lo_ch, float hi_ch) {
    return f2_to_bf2(lo_ch, hi_ch);
}

// Pass-1 B fragments of a warp's channel slice [cbase, cbase + 16*KS): query
// q = g4/2 with the gain folded in, its bf16 hi part in column 2q and its lo
// part in column 2q+1 (columns of absent queries are zero).
template <int KS>
__device__ __forceinline__ void dm_query_fragments(const DepthReadMmaArgs &a, int cbase, int g4, int t4,
                                                   uint32_t (&bq)[KS][2]) {
    const int q = g4 >> 1, part = g4 & 1;
#pragma unroll
    for (int s = 0; s < KS; ++s)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int c = cbase + 16 * s + 8 * h + 2 * t4;
            float v0 = 0.f, v1 = 0.f;
            if (q < a.n_q) {
                v0 = __ldg(a.queries + (size_t)q * a.d + c);
                v1 = __ldg(a.queries + (size_t)q * a.d + c + 1);
                if (a.gain) { v0 *= __ldg(a.gain + c); v1 *= __ldg(a.gain + c + 1); }
            }
            float h0, l0, h1, l1;
            split_bf16(v0, h0, l0);
            split_bf16(v1, h1, l1);
            bq[s][h] = part == 0 ? pack_bf16(h0, h1) : pack_bf16(l0, l1);
        }
}

// Pass 1 over 8 source rows of a warp's channel slice: D1 = X Q on the tensor
// cores (X = [8 sources x 16 channels], rows 8..15 zero) and sum(v_i^2) with
// packed FMAs on the same ldmatrix fragments.  sa is this lane's ldmatrix row
// address (source lane%8, channel block lane/8 of a 32-channel group).  On
// return lane (i = g4, q = t4) holds dot_qi and lanes 4i.. hold sum(v_i^2).
template <int KS>
__device__ __forceinline__ void dm_pass1_rows8(uint32_t sa, const uint32_t (&bq)[KS][2], float &dot,
                                               float &ssq) {
    float d1[2][4];
#pragma unroll
    for (int u = 0; u < 2; ++u)
#pragma unroll
        for (int e = 0; e < 4; ++e) d1[u][e] = 0.f;
    float2 sq = make_float2(0.f, 0.f);
#pragma unroll
    for (int s2 = 0; s2 < KS / 2; ++s2) {
        uint32_t x0, x1, x2, x3;            // k-step 2*s2: (x0, x1); 2*s2+1: (x2, x3)
        ldsm_x4(sa + 64 * s2, x0, x1, x2, x3);
        mma_rows8(d1[0], x0, x1, bq[2 * s2][0], bq[2 * s2][1]);
        mma_rows8(d1[1], x2, x3, bq[2 * s2 + 1][0], bq[2 * s2 + 1][1]);
        const float2 f0 = bf2_to_f2(x0), f1 = bf2_to_f2(x1), f2 = bf2_to_f2(x2), f3 = bf2_to_f2(x3);
        sq = ffma2(f0, f0, sq);
        sq = ffma2(f1, f1, sq);
        sq = ffma2(f2, f2, sq);
        sq = ffma2(f3, f3, sq);
    }
    dot = (d1[0][0] + d1[1][0]) + (d1[0][1] + d1[1][1]);
    ssq = sq.x + sq.y;
    ssq += __shfl_xor_sync(0xffffffffu, ssq, 1);
    ssq += __shfl_xor_sync(0xffffffffu, ssq, 2);
}

// At most 2 queries: two k-steps per MMA.  A = [8 sources x k-step a; the
// same 8 sources x k-step b] (rows 0..7, 8..15); B column c holds query c/4,
// k-step (c/2)&1 and bf16 part c&1 (hi, lo).  Output rows of k-step a only
// meet its columns in lanes with t4 even (c0 + c1), rows of k-step b in lanes
// with t4 odd (c2 + c3): half the MMAs of dm_pass1_rows8, half the B registers.
template <int KS>
__device__ __forceinline__ void dm_query_fragments_packed(const DepthReadMmaArgs &a, int cbase, int g4, int t4,
                                                          uint32_t (&bq)[KS / 2][2]) {
    const int q = g4 >> 2, kb = (g4 >> 1) & 1, part = g4 & 1;
#pragma unroll
    for (int s2 = 0; s2 < KS / 2; ++s2)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int c = cbase + 32 * s2 + 16 * kb + 8 * h + 2 * t4;
            float v0 = 0.f, v1 = 0.f;
            if (q < a.n_q) {
                v0 = __ldg(a.queries + (size_t)q * a.d + c);
                v1 = __ldg(a.queries + (size_t)q * a.d + c + 1);
                if (a.gain) { v0 *= __ldg(a.gain + c); v1 *= __ldg(a.gain + c + 1); }
            }
            float h0, l0, h1, l1;
            split_bf16(v0, h0, l0);
            split_bf16(v1, h1, l1);
            bq[s2][h] = part == 0 ? pack_bf16(h0, h1) : pack_bf16(l0, l1);
        }
}

// Pass 1 with dm_query_fragments_packed.  The sums of squares come from the
// tensor cores too, as the diagonal of the Gram matrix G = X X^T: the
// ldmatrix fragment of X is already the B fragment of X^T (lane (g4, t4)
// holds X[g4][2t4..2t4+1] and X[g4][8+2t4..]), so one MMA per k-step
// replaces the unpacking and packed FMAs (products exact, sums fp32).  With
// one or two queries the dots take one MMA per two k-steps, and the Gram MMAs
// fill the idle tensor pipe; with more queries (dm_pass1_rows8) they would
// lengthen the per-token chain, measured 1.7% slower there.  On return lanes
// (i = g4, t4 = 2q, 2q+1) hold dot_qi and lane (i, i/2) holds sum(v_i^2).
template <int KS>
__device__ __forceinline__ void dm_pass1_rows8_packed(uint32_t sa, const uint32_t (&bq)[KS / 2][2], int t4,
                                                      float &dot, float &ssq) {
    float d1[2][4], gr[2][4];
#pragma unroll
    for (int u = 0; u < 2; ++u)
#pragma unroll
        for (int e = 0; e < 4; ++e) { d1[u][e] = 0.f; gr[u][e] = 0.f; }
#pragma unroll
    for (int s2 = 0; s2 < KS / 2; ++s2) {
        uint32_t x0, x1, x2, x3;            // k-step a: (x0, x1); k-step b: (x2, x3)
        ldsm_x4(sa + 64 * s2, x0, x1, x2, x3);
        mma_full(d1[s2 & 1], x0, x2, x1, x3, bq[s2][0], bq[s2][1]);
        mma_rows8(gr[0], x0, x1, x0, x1);
        mma_rows8(gr[1], x2, x3, x2, x3);
    }
    const float part = (t4 & 1) ? (d1[0][2] + d1[1][2]) + (d1[0][3] + d1[1][3])
                                : (d1[0][0] + d1[1][0]) + (d1[0][1] + d1[1][1]);
    dot = part + __shfl_xor_sync(0xffffffffu, part, 1);
    ssq = (threadIdx.x & 4) ? gr[0][1] + gr[1][1] : gr[0][0] + gr[1][0];
}

// Sum over the wph warps of a head (starting at gw0) of the partial sum of
// squares of source i and the partial dot of (query q, source i), from the
// value-major table rb[value][warp] (row stride RS).
__device__ __forceinline__ void dm_head_partials(const float *rb, int RS, int gw0, int wph, int q, int i,
                                                 float &ss, float &dt) {
    ss = 0.f;
    dt = 0.f;
    const float *ps = rb + (32 + i) * RS + gw0;
    const float *pd = rb + (q * 8 + i) * RS + gw0;
    if (wph % 4 == 0) {
        for (int w = 0; w < wph; w += 4) {
            const float4 x = *reinterpret_cast<const float4 *>(ps + w);
            const float4 y = *reinterpret_cast<const float4 *>(pd + w);
            ss += (x.x + x.y) + (x.z + x.w);
            dt += (y.x + y.y) + (y.z + y.w);
        }
    } else {
        for (int w = 0; w < wph; ++w) { ss += ps[w]; dt += pd[w]; }
    }
}

// Scale an m16n8 accumulator fragment column-wise: elements 0, 2 belong to
// column 2*t4, elements 1, 3 to column 2*t4+1.
__device__ __forceinline__ void dm_rescale(float (&c)[4], float2 f) {
    const float2 a = fmul2(make_float2(c[0], c[1]), f), b = fmul2(make_float2(c[2], c[3]), f);
    c[0] = a.x; c[1] = a.y; c[2] = b.x; c[3] = b.y;
}

// With 8 warps (d = 2048) two CTAs share an SM (three 32 KB stages each, at
// most 128 registers a thread), so one CTA's per-token chain hides behind the
// other's; with 16 warps (d = 4096) the stages need the whole SM.
template <int NQ, int KS, int NW>
__global__ void __launch_bounds__(NW * 32, NW == 8 ? 2 : 1) depth_read_mma_kernel(const DepthReadMmaArgs a) {
    static_assert(NQ <= 4, "at most 4 queries (8 MMA columns: hi and lo per query)");
    using L = DMLayout;
    constexpr int CW = KS * 16;                 // channels per warp

    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char *stages = smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)a.nstages * a.stage_bytes);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(full + DM_MAX_STAGES);
    float *red = reinterpret_cast<float *>(smem + (size_t)a.nstages * a.stage_bytes + L::bar_bytes);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int g4 = lane >> 2, t4 = lane & 3;    // mma groupID / thread-in-group

    if (tid == 0) {
        for (int s = 0; s < a.nstages; ++s) mbar_init(&full[s], 1);
        *abort_flag = 0;
        mbar_init_fence();
    }
    // Source rows n_src..7 of every stage are never loaded but enter the MMAs
    // (times a zero weight): make them zero, not stale bits that could be NaN.
    for (int s = 0; s < a.nstages; ++s)
        for (int i = a.n_src; i < 8; ++i)
            for (int b = tid * 16; b < a.d * 2; b += NW * 32 * 16)
                *reinterpret_cast<uint4 *>(stages + (size_t)s * a.stage_bytes + (size_t)i * a.pitch + b) =
                    make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();

    const int gstride = gridDim.x;
    const int n_items = blockIdx.x < a.T ? (int)((a.T - blockIdx.x + gstride - 1) / gstride) : 0;

    // ------------------------------------------------------------ producer
    // warp 0 produces (lane 0 arms the stage's mbarrier and issues the copies;
    // measured faster than one copy per lane here)
    const bool producer = (warp == 0) && !a.wait.inject_stall;
    uint64_t pol = 0;
    if (producer) pol = l2_policy_evict_first();
    int p_stage = 0;
    int64_t p_tok = blockIdx.x;
    const uint32_t row_bytes = (uint32_t)a.d * 2;
    auto issue_next = [&]() {
        if (lane == 0) {
            mbar_arrive_expect_tx(&full[p_stage], row_bytes * a.n_src);
            for (int i = 0; i < a.n_src; ++i)
                bulk_g2s(stages + (size_t)p_stage * a.stage_bytes + (size_t)i * a.pitch,
                         a.src + p_tok * row_bytes + (int64_t)i * a.src_stride_bytes, row_bytes, &full[p_stage], pol);
        }
        if (++p_stage == a.nstages) p_stage = 0;
        p_tok += gstride;
    };
    int issued = 0;
    if (producer)
        for (; issued < n_items && issued < a.nstages; ++issued) issue_next();

    // ------------------------------------------------------------ constants
    const int cbase = warp * CW;                // first channel of this warp
    constexpr bool PACK = NQ <= 2;
    uint32_t bq[PACK ? KS / 2 : KS][2];
    if constexpr (PACK) dm_query_fragments_packed<KS>(a, cbase, g4, t4, bq);
    else dm_query_fragments<KS>(a, cbase, g4, t4, bq);
    // head of this warp and the warps that share it
    const int head = warp / a.wph;
    const int gw0 = head * a.wph;
    const float inv_dh = 1.f / (float)(CW * a.wph);
    // ldmatrix row address of this lane inside a stage: source row lane%8,
    // channel block (lane/8) of a 32-channel group
    const uint32_t lrow = (uint32_t)(lane & 7) * a.pitch + (uint32_t)(cbase + 8 * (lane >> 3)) * 2;
    const uint32_t stage0 = smem_u32(stages);

    int s = 0;
    uint32_t par = 0;
    int64_t t = blockIdx.x;
    for (int it = 0; it < n_items; ++it) {
        mbar_wait_bounded(&full[s], par, abort_flag, a.wait);
        const uint32_t sa = stage0 + (uint32_t)s * a.stage_bytes + lrow;

        // ---------------- pass 1: D1 = X Q on the tensor cores, sum(v_i^2) alongside
        float dot, ssq;
        int dq = t4;                         // query of this lane's dot
        if constexpr (PACK) { dm_pass1_rows8_packed<KS>(sa, bq, t4, dot, ssq); dq = t4 >> 1; }
        else dm_pass1_rows8<KS>(sa, bq, dot, ssq);
        constexpr int RS = L::RS;
        float *rb = red + (size_t)(it & 1) * 40 * RS;
        if (!PACK || (t4 & 1) == 0) rb[(dq * 8 + g4) * RS + warp] = dot;
        if (t4 == (g4 >> 1)) rb[(32 + g4) * RS + warp] = ssq;
        // the previous item's output bulk stores must have read their shared rows
        // before the barrier that lets the producer refill that stage
        if (lane < a.n_q && it >= 1) bulk_wait_read0();
        if (a.n_src < a.n_q && it >= 1) {
            // Rows n_src..n_q-1 of the previous stage held outputs but are never
            // reloaded: restore their zeros (this warp's channel slice) once the
            // bulk stores have read them.
            __syncwarp();
            const int sp = s == 0 ? a.nstages - 1 : s - 1;
            for (int row = a.n_src; row < a.n_q; ++row)
                for (int b = lane * 16; b < CW * 2; b += 32 * 16)
                    *reinterpret_cast<uint4 *>(stages + (size_t)sp * a.stage_bytes + (size_t)row * a.pitch +
                                               (size_t)cbase * 2 + b) = make_uint4(0u, 0u, 0u, 0u);
        }
        __syncthreads();
        if (producer && it >= 1 && issued < n_items) {
            // one decision for the whole producer warp (issue_next synchronises it)
            if (__shfl_sync(0xffffffffu, *abort_flag == 0 ? 1 : 0, 0)) { issue_next(); ++issued; }
        }

        // ---------------- softmax over sources: lane p = q*8 + i
        const int q = lane >> 3, i = lane & 7;
        float ss, dt;
        dm_head_partials(rb, RS, gw0, a.wph, q, i, ss, dt);
        const bool pv = i < a.n_src && q < NQ;
        const float score = pv ? key_score(dt, ss, inv_dh, a.eps) : -INFINITY;
        const float cmax = seg_max<8>(score);
        const float e = pv ? __expf(score - cmax) : 0.f;
        const float sum = seg_sum<8>(e);
        const float alpha = pv ? e / sum : 0.f;
        if (i == 0 && q < a.n_q && warp == gw0 && a.lse != nullptr && !*abort_flag)
            a.lse[((int64_t)q * a.H + head) * a.T + t] = cmax + __logf(sum);

        // B fragment of pass 2: k = sources 2*t4, 2*t4+1 (hi) and +8 (lo), column q = g4 (< 4)
        const int srcl = (g4 & 3) * 8 + 2 * t4;
        const float al0 = __shfl_sync(0xffffffffu, alpha, srcl);
        const float al1 = __shfl_sync(0xffffffffu, alpha, srcl + 1);
        uint32_t bb0 = 0u, bb1 = 0u;
        if (g4 < NQ) {
            float h0, l0, h1, l1;
            split_bf16(al0, h0, l0);
            split_bf16(al1, h1, l1);
            bb0 = pack_bf16(h0, h1);
            bb1 = pack_bf16(l0, l1);
        }

        // ---------------- pass 2: O^T = X'^T A per 16-channel block
        // The result tiles are [channels x queries]; stmatrix .trans writes them
        // back as query rows of 8 channels into stage rows 0..7 at the channels
        // this warp has already consumed (queries 4..7 are zero columns, so rows
        // 4..7 only ever receive zeros there).
        const uint32_t orow = stage0 + (uint32_t)s * a.stage_bytes + (uint32_t)(lane & 7) * a.pitch +
                              (uint32_t)(cbase + 8 * (lane >> 3)) * 2;
#pragma unroll 4
        for (int s2 = 0; s2 < KS / 2; ++s2) {
            uint32_t y[4];
            ldsm_x4_t(sa + 64 * s2, y[0], y[1], y[2], y[3]);
            float o0[4] = {0.f, 0.f, 0.f, 0.f}, o1[4] = {0.f, 0.f, 0.f, 0.f};
            mma_full(o0, y[0], y[1], y[0], y[1], bb0, bb1);
            mma_full(o1, y[2], y[3], y[2], y[3], bb0, bb1);
            stsm_x4_t(orow + 64 * s2, f2_to_bf2(o0[0], o0[1]), f2_to_bf2(o0[2], o0[3]),
                      f2_to_bf2(o1[0], o1[1]), f2_to_bf2(o1[2], o1[3]));
        }
        // one bulk store per query row of this warp's channel slice
        fence_proxy_async_smem();
        __syncwarp();
        // (bulk-copy groups belong to the issuing thread: lane q issues, commits
        // and later waits for the store of query q)
        if (lane < a.n_q) {
            if (!*abort_flag)
                bulk_s2g(a.out + (int64_t)lane * a.out_q_stride_bytes + (t * a.d + cbase) * 2,
                         stage0 + (uint32_t)s * a.stage_bytes + (uint32_t)lane * a.pitch + (uint32_t)cbase * 2,
                         (uint32_t)CW * 2);
            bulk_commit();
        }
        if (++s == a.nstages) { s = 0; par ^= 1u; }
        t += gstride;
    }

    // outputs must be written before the CTA exits
    if (lane < a.n_q) bulk_wait0();
    if (producer && lane == 0) {
        int never = 0;
        for (int it = issued > a.nstages ? issued - a.nstages : 0; it < issued; ++it)
            mbar_wait_bounded(&full[it % a.nstages], (uint32_t)(it / a.nstages) & 1, &never, a.wait);
    }
}


// Two tokens per item (d = 1024, where two tokens' 8 source rows fit one
// 33 KB stage).  Pass 1 uses all 16 MMA rows (token 0's sources in rows 0..7,
// token 1's in rows 8..15); the two tokens' softmaxes run as independent
// chains; the per-item barrier, softmax latency and bulk stores are paid
// once per two tokens.  Stage row tok*8 + i holds source i of token tok.
template <int NQ, int KS, int NW>
__global__ void __launch_bounds__(NW * 32, 1) depth_read_mma2_kernel(const DepthReadMmaArgs a) {
    static_assert(NQ <= 4, "at most 4 queries (8 MMA columns: hi and lo per query)");
    using L = DMLayout;
    constexpr int CW = KS * 16;                 // channels per warp
    constexpr int RS = L::RS;

    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char *stages = smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)a.nstages * a.stage_bytes);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(full + DM_MAX_STAGES);
    float *red = reinterpret_cast<float *>(smem + (size_t)a.nstages * a.stage_bytes + L::bar_bytes);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int g4 = lane >> 2, t4 = lane & 3;

    if (tid == 0) {
        for (int s = 0; s < a.nstages; ++s) mbar_init(&full[s], 1);
        *abort_flag = 0;
        mbar_init_fence();
    }
    // rows of absent sources (both tokens) stay zero
    for (int s = 0; s < a.nstages; ++s)
        for (int tk = 0; tk < 2; ++tk)
            for (int i = a.n_src; i < 8; ++i)
                for (int b = tid * 16; b < a.d * 2; b += NW * 32 * 16)
                    *reinterpret_cast<uint4 *>(stages + (size_t)s * a.stage_bytes +
                                               (size_t)(tk * 8 + i) * a.pitch + b) = make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();

    const int64_t npairs = (a.T + 1) / 2;
    const int gstride = gridDim.x;
    const int n_items = blockIdx.x < npairs ? (int)((npairs - blockIdx.x + gstride - 1) / gstride) : 0;

    // ------------------------------------------------------------ producer
    // warp 0 produces: lane 0 arms the mbarrier, lane tk*8 + i copies source i of token tk
    const bool producer = (warp == 0) && !a.wait.inject_stall;
    uint64_t pol = 0;
    if (producer) pol = l2_policy_evict_first();
    int p_stage = 0;
    int64_t p_pair = blockIdx.x;
    const uint32_t row_bytes = (uint32_t)a.d * 2;
    auto issue_next = [&]() {
        const int64_t t0 = 2 * p_pair;
        const int ntok = t0 + 1 < a.T ? 2 : 1;
        if (lane == 0) mbar_arrive_expect_tx(&full[p_stage], row_bytes * a.n_src * ntok);
        __syncwarp();
        const int tk = lane >> 3, i = lane & 7;
        if (lane < 16 && tk < ntok && i < a.n_src) {
            const unsigned char *g = a.src + (t0 + tk) * row_bytes + (int64_t)i * a.src_stride_bytes;
            bulk_g2s(stages + (size_t)p_stage * a.stage_bytes + (size_t)(tk * 8 + i) * a.pitch, g, row_bytes,
                     &full[p_stage], pol);
        }
        if (++p_stage == a.nstages) p_stage = 0;
        p_pair += gstride;
    };
    int issued = 0;
    if (producer)
        for (; issued < n_items && issued < a.nstages; ++issued) issue_next();

    // ------------------------------------------------------------ constants
    const int cbase = warp * CW;
    uint32_t bq[KS][2];
    dm_query_fragments<KS>(a, cbase, g4, t4, bq);
    const int head = warp / a.wph;
    const int gw0 = head * a.wph;
    const float inv_dh = 1.f / (float)(CW * a.wph);
    // ldmatrix (both directions): matrix j = lane/8 is token j&1, channels
    // +8*(j>>1) of the 16-channel step; row = source lane%8
    const uint32_t lrow = (uint32_t)(((lane >> 3) & 1) * 8 + (lane & 7)) * a.pitch +
                          (uint32_t)(cbase + 8 * (lane >> 4)) * 2;
    // stmatrix: matrix j = lane/8 is token j>>1, channels +8*(j&1); row = query lane%8
    const uint32_t orow = (uint32_t)((lane >> 4) * 8 + (lane & 7)) * a.pitch +
                          (uint32_t)(cbase + 8 * ((lane >> 3) & 1)) * 2;
    const uint32_t stage0 = smem_u32(stages);

    int s = 0;
    uint32_t par = 0;
    int64_t pair = blockIdx.x;
    for (int it = 0; it < n_items; ++it) {
        const int64_t t0 = 2 * pair;
        const bool has1 = t0 + 1 < a.T;
        mbar_wait_bounded(&full[s], par, abort_flag, a.wait);
        const uint32_t sbase = stage0 + (uint32_t)s * a.stage_bytes;

        // ---------------- pass 1: D1 = X Q (16 rows) on the tensor cores; sums
        // of squares with packed FMAs on the fragments (lane (g4, t4) holds 4
        // elements of source g4 of each token per k-step)
        float d1[2][4];
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
            for (int e = 0; e < 4; ++e) d1[u][e] = 0.f;
        float2 sq0 = make_float2(0.f, 0.f), sq1 = make_float2(0.f, 0.f);
#pragma unroll
        for (int k = 0; k < KS; ++k) {
            uint32_t x0, x1, x2, x3;       // (tok0, ch 0-7), (tok1, ch 0-7), (tok0, ch 8-15), (tok1, ch 8-15)
            ldsm_x4(sbase + lrow + 32 * k, x0, x1, x2, x3);
            mma_full(d1[k & 1], x0, x1, x2, x3, bq[k][0], bq[k][1]);
            const float2 f0 = bf2_to_f2(x0), f1 = bf2_to_f2(x1), f2 = bf2_to_f2(x2), f3 = bf2_to_f2(x3);
            sq0 = ffma2(f0, f0, sq0);
            sq0 = ffma2(f2, f2, sq0);
            sq1 = ffma2(f1, f1, sq1);
            sq1 = ffma2(f3, f3, sq1);
        }
        // lane (i = g4, q = t4): dots of token 0 in c0+c1, token 1 in c2+c3
        const float dot0 = (d1[0][0] + d1[1][0]) + (d1[0][1] + d1[1][1]);
        const float dot1 = (d1[0][2] + d1[1][2]) + (d1[0][3] + d1[1][3]);
        float s0 = sq0.x + sq0.y, s1 = sq1.x + sq1.y;
        s0 += __shfl_xor_sync(0xffffffffu, s0, 1);
        s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
        s0 += __shfl_xor_sync(0xffffffffu, s0, 2);
        s1 += __shfl_xor_sync(0xffffffffu, s1, 2);
        float *rb = red + (size_t)(it & 1) * 80 * RS;
        rb[(t4 * 8 + g4) * RS + warp] = dot0;
        rb[(40 + t4 * 8 + g4) * RS + warp] = dot1;
        if (t4 == 0) {
            rb[(32 + g4) * RS + warp] = s0;
            rb[(72 + g4) * RS + warp] = s1;
        }
        if (lane < 8 && it >= 1) bulk_wait_read0();
        if (a.n_src < a.n_q && it >= 1) {
            __syncwarp();
            const int sp = s == 0 ? a.nstages - 1 : s - 1;
            for (int tk = 0; tk < 2; ++tk)
                for (int row = a.n_src; row < a.n_q; ++row)
                    for (int b = lane * 16; b < CW * 2; b += 32 * 16)
                        *reinterpret_cast<uint4 *>(stages + (size_t)sp * a.stage_bytes +
                                                   (size_t)(tk * 8 + row) * a.pitch + (size_t)cbase * 2 + b) =
                            make_uint4(0u, 0u, 0u, 0u);
        }
        __syncthreads();
        if (producer && it >= 1 && issued < n_items) {
            // one decision for the whole producer warp (issue_next synchronises it)
            if (__shfl_sync(0xffffffffu, *abort_flag == 0 ? 1 : 0, 0)) { issue_next(); ++issued; }
        }

        // ---------------- softmax over sources for both tokens: lane p = q*8 + i
        const int q = lane >> 3, i = lane & 7;
        float ss0 = 0.f, dt0 = 0.f, ss1 = 0.f, dt1 = 0.f;
        {
            const float *ps0 = rb + (32 + i) * RS + gw0, *pd0 = rb + (q * 8 + i) * RS + gw0;
            const float *ps1 = ps0 + 40 * RS, *pd1 = pd0 + 40 * RS;
            if (a.wph % 4 == 0) {
                for (int w = 0; w < a.wph; w += 4) {
                    const float4 x0 = *reinterpret_cast<const float4 *>(ps0 + w);
                    const float4 y0 = *reinterpret_cast<const float4 *>(pd0 + w);
                    const float4 x1 = *reinterpret_cast<const float4 *>(ps1 + w);
                    const float4 y1 = *reinterpret_cast<const float4 *>(pd1 + w);
                    ss0 += (x0.x + x0.y) + (x0.z + x0.w);
                    dt0 += (y0.x + y0.y) + (y0.z + y0.w);
                    ss1 += (x1.x + x1.y) + (x1.z + x1.w);
                    dt1 += (y1.x + y1.y) + (y1.z + y1.w);
                }
            } else {
                for (int w = 0; w < a.wph; ++w) { ss0 += ps0[w]; dt0 += pd0[w]; ss1 += ps1[w]; dt1 += pd1[w]; }
            }
        }
        const bool pv = i < a.n_src && q < NQ;
        const float sc0 = pv ? key_score(dt0, ss0, inv_dh, a.eps) : -INFINITY;
        const float sc1 = pv ? key_score(dt1, ss1, inv_dh, a.eps) : -INFINITY;
        const float m0 = seg_max<8>(sc0), m1 = seg_max<8>(sc1);
        const float e0 = pv ? __expf(sc0 - m0) : 0.f, e1 = pv ? __expf(sc1 - m1) : 0.f;
        const float l0 = seg_sum<8>(e0), l1 = seg_sum<8>(e1);
        const float al_0 = pv ? e0 / l0 : 0.f, al_1 = pv ? e1 / l1 : 0.f;
        if (i == 0 && q < a.n_q && warp == gw0 && a.lse != nullptr && !*abort_flag) {
            a.lse[((int64_t)q * a.H + head) * a.T + t0] = m0 + __logf(l0);
            if (has1) a.lse[((int64_t)q * a.H + head) * a.T + t0 + 1] = m1 + __logf(l1);
        }
        // pass-2 B fragments of both tokens
        const int srcl = (g4 & 3) * 8 + 2 * t4;
        uint32_t bb[2][2] = {{0u, 0u}, {0u, 0u}};
        {
            const float a00 = __shfl_sync(0xffffffffu, al_0, srcl), a01 = __shfl_sync(0xffffffffu, al_0, srcl + 1);
            const float a10 = __shfl_sync(0xffffffffu, al_1, srcl), a11 = __shfl_sync(0xffffffffu, al_1, srcl + 1);
            if (g4 < NQ) {
                float h0, lo0, h1, lo1;
                split_bf16(a00, h0, lo0);
                split_bf16(a01, h1, lo1);
                bb[0][0] = pack_bf16(h0, h1);
                bb[0][1] = pack_bf16(lo0, lo1);
                split_bf16(a10, h0, lo0);
                split_bf16(a11, h1, lo1);
                bb[1][0] = pack_bf16(h0, h1);
                bb[1][1] = pack_bf16(lo0, lo1);
            }
        }

        // ---------------- pass 2 for both tokens, outputs staged by stmatrix
#pragma unroll 4
        for (int k = 0; k < KS; ++k) {
            uint32_t y0, y1, y2, y3;       // .trans: (tok0, ch 0-7), (tok1, ch 0-7), (tok0, ch 8-15), (tok1, ch 8-15)
            ldsm_x4_t(sbase + lrow + 32 * k, y0, y1, y2, y3);
            float o0[4] = {0.f, 0.f, 0.f, 0.f}, o1[4] = {0.f, 0.f, 0.f, 0.f};
            mma_full(o0, y0, y2, y0, y2, bb[0][0], bb[0][1]);
            mma_full(o1, y1, y3, y1, y3, bb[1][0], bb[1][1]);
            stsm_x4_t(sbase + orow + 32 * k, f2_to_bf2(o0[0], o0[1]), f2_to_bf2(o0[2], o0[3]),
                      f2_to_bf2(o1[0], o1[1]), f2_to_bf2(o1[2], o1[3]));
        }
        fence_proxy_async_smem();
        __syncwarp();
        // lanes 0..3: token 0, query lane; lanes 4..7: token 1, query lane-4
        if (lane < 8) {
            const int tk = lane >> 2, qq = lane & 3;
            if (qq < a.n_q && (tk == 0 || has1) && !*abort_flag)
                bulk_s2g(a.out + (int64_t)qq * a.out_q_stride_bytes + ((t0 + tk) * a.d + cbase) * 2,
                         sbase + (uint32_t)(tk * 8 + qq) * a.pitch + (uint32_t)cbase * 2, (uint32_t)CW * 2);
            bulk_commit();
        }
        if (++s == a.nstages) { s = 0; par ^= 1u; }
        pair += gstride;
    }

    if (lane < 8) bulk_wait0();
    if (producer && lane == 0) {
        int never = 0;
        for (int it = issued > a.nstages ? issued - a.nstages : 0; it < issued; ++it)
            mbar_wait_bounded(&full[it % a.nstages], (uint32_t)(it / a.nstages) & 1, &never, a.wait);
    }
}

// More than 8 sources, one token per item: the token's sources arrive in
// chunks of 8 rows (one stage each) and are folded in by an online softmax.
// Per query the running maximum m and normaliser l live in the softmax lanes
// (lane q*8 + i); the output accumulators O^T stay in the MMA fragments across
// the chunks, each chunk first scaling them by e^{m_old - m_new} and then
// adding X'^T E with E = e^{s - m_new} (at most 1, split into bf16 hi and lo
// like alpha in the one-chunk kernel).  After the token's last chunk the
// fragments are divided by l, staged by stmatrix and stored in bulk as there.
// A partial last chunk (n_src % 8 rows) leaves rows of its stage unfilled:
// the warps that consumed that stage just before zero those rows (their
// channel slice) so that they enter the MMAs as zeros, not as another
// token's values.
template <int NQ, int KS, int NW>
__global__ void __launch_bounds__(NW * 32, 1) depth_read_mma_multi_kernel(const DepthReadMmaArgs a) {
    static_assert(NQ <= 4, "at most 4 queries (8 MMA columns: hi and lo per query)");
    using L = DMLayout;
    constexpr int CW = KS * 16;                 // channels per warp
    constexpr int RS = L::RS;

    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char *stages = smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)a.nstages * a.stage_bytes);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(full + DM_MAX_STAGES);
    float *red = reinterpret_cast<float *>(smem + (size_t)a.nstages * a.stage_bytes + L::bar_bytes);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int g4 = lane >> 2, t4 = lane & 3;

    if (tid == 0) {
        for (int s = 0; s < a.nstages; ++s) mbar_init(&full[s], 1);
        *abort_flag = 0;
        mbar_init_fence();
    }
    // every row of every stage starts zero (the copies overwrite them later:
    // order these generic writes before the async-proxy writes)
    for (int s = 0; s < a.nstages; ++s)
        for (int i = 0; i < 8; ++i)
            for (int b = tid * 16; b < a.d * 2; b += NW * 32 * 16)
                *reinterpret_cast<uint4 *>(stages + (size_t)s * a.stage_bytes + (size_t)i * a.pitch + b) =
                    make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
    __syncthreads();

    const int nch = (a.n_src + 7) >> 3;         // chunks per token
    const int rlast = a.n_src - 8 * (nch - 1);  // rows of the last chunk (1..8)
    const int gstride = gridDim.x;
    const int n_tok = blockIdx.x < a.T ? (int)((a.T - blockIdx.x + gstride - 1) / gstride) : 0;
    const int n_items = n_tok * nch;            // the host keeps this within int

    // ------------------------------------------------------------ producer
    const bool producer = (warp == 0) && !a.wait.inject_stall;
    uint64_t pol = 0;
    if (producer) pol = l2_policy_evict_first();
    int p_stage = 0, p_j = 0;
    int64_t p_tok = blockIdx.x;
    const uint32_t row_bytes = (uint32_t)a.d * 2;
    auto issue_next = [&]() {
        if (lane == 0) {
            const int rows = p_j == nch - 1 ? rlast : 8;
            mbar_arrive_expect_tx(&full[p_stage], row_bytes * rows);
            const unsigned char *g = a.src + p_tok * row_bytes + (int64_t)(8 * p_j) * a.src_stride_bytes;
            for (int i = 0; i < rows; ++i)
                bulk_g2s(stages + (size_t)p_stage * a.stage_bytes + (size_t)i * a.pitch,
                         g + (int64_t)i * a.src_stride_bytes, row_bytes, &full[p_stage], pol);
        }
        if (++p_stage == a.nstages) p_stage = 0;
        if (++p_j == nch) { p_j = 0; p_tok += gstride; }
    };
    int issued = 0;
    if (producer)
        for (; issued < n_items && issued < a.nstages; ++issued) issue_next();

    // ------------------------------------------------------------ constants
    const int cbase = warp * CW;
    constexpr bool PACK = NQ <= 2;
    uint32_t bq[PACK ? KS / 2 : KS][2];
    if constexpr (PACK) dm_query_fragments_packed<KS>(a, cbase, g4, t4, bq);
    else dm_query_fragments<KS>(a, cbase, g4, t4, bq);
    const int head = warp / a.wph;
    const int gw0 = head * a.wph;
    const float inv_dh = 1.f / (float)(CW * a.wph);
    const uint32_t lrow = (uint32_t)(lane & 7) * a.pitch + (uint32_t)(cbase + 8 * (lane >> 3)) * 2;
    const uint32_t stage0 = smem_u32(stages);

    float acc[KS][4];
#pragma unroll
    for (int k = 0; k < KS; ++k)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[k][e] = 0.f;
    // softmax lane p = q*8 + i: running max / normaliser of query q
    const int q = lane >> 3, i = lane & 7;
    float m_run = -INFINITY, l_run = 0.f;

    int s = 0, j = 0;
    uint32_t par = 0;
    int64_t t = blockIdx.x;
    // chunk index of the copy that refills the stage consumed at item it:
    // item it + nstages
    int jn = a.nstages % nch;
    for (int it = 0; it < n_items; ++it) {
        mbar_wait_bounded(&full[s], par, abort_flag, a.wait);
        const uint32_t sa = stage0 + (uint32_t)s * a.stage_bytes + lrow;
        const int rows = j == nch - 1 ? rlast : 8;
        const bool last = j == nch - 1;

        // ---------------- pass 1 (as in the one-chunk kernel)
        float dot, ssq;
        int dq = t4;
        if constexpr (PACK) { dm_pass1_rows8_packed<KS>(sa, bq, t4, dot, ssq); dq = t4 >> 1; }
        else dm_pass1_rows8<KS>(sa, bq, dot, ssq);
        float *rb = red + (size_t)(it & 1) * 40 * RS;
        if (!PACK || (t4 & 1) == 0) rb[(dq * 8 + g4) * RS + warp] = dot;
        if (t4 == (g4 >> 1)) rb[(32 + g4) * RS + warp] = ssq;
        if (it >= 1) {
            // the stage consumed at it-1 is refilled after the barrier below with
            // item it-1+nstages: its output rows (if it held a token's last chunk)
            // must have been read by the bulk stores, and rows that the refill
            // leaves empty must be zero
            if (lane < a.n_q) bulk_wait_read0();
            const int jp = jn == 0 ? nch - 1 : jn - 1;
            if (jp == nch - 1 && rlast < 8 && it - 1 + a.nstages < n_items) {
                __syncwarp();
                const int sp = s == 0 ? a.nstages - 1 : s - 1;
                for (int row = rlast; row < 8; ++row)
                    for (int b = lane * 16; b < CW * 2; b += 32 * 16)
                        *reinterpret_cast<uint4 *>(stages + (size_t)sp * a.stage_bytes + (size_t)row * a.pitch +
                                                   (size_t)cbase * 2 + b) = make_uint4(0u, 0u, 0u, 0u);
                fence_proxy_async_smem();
            }
        }
        __syncthreads();
        if (producer && it >= 1 && issued < n_items) {
            if (__shfl_sync(0xffffffffu, *abort_flag == 0 ? 1 : 0, 0)) { issue_next(); ++issued; }
        }

        // ---------------- online softmax over this chunk's sources
        float ss, dt;
        dm_head_partials(rb, RS, gw0, a.wph, q, i, ss, dt);
        const bool pv = i < rows && q < NQ;
        const float score = pv ? key_score(dt, ss, inv_dh, a.eps) : -INFINITY;
        const float m_new = fmaxf(m_run, seg_max<8>(score));
        const float corr = __expf(m_run - m_new);   // 0 on the token's first chunk
        const float e = pv ? __expf(score - m_new) : 0.f;
        l_run = l_run * corr + seg_sum<8>(e);
        m_run = m_new;
        if (last && i == 0 && q < a.n_q && warp == gw0 && a.lse != nullptr && !*abort_flag)
            a.lse[((int64_t)q * a.H + head) * a.T + t] = m_run + __logf(l_run);

        // pass-2 B fragment (sources 2*t4, 2*t4+1 of column q = g4), and the
        // per-column factors of this lane's accumulators (columns 2*t4, 2*t4+1;
        // columns 4..7 are always zero)
        const int srcl = (g4 & 3) * 8 + 2 * t4;
        const float e0 = __shfl_sync(0xffffffffu, e, srcl);
        const float e1 = __shfl_sync(0xffffffffu, e, srcl + 1);
        uint32_t bb0 = 0u, bb1 = 0u;
        if (g4 < NQ) {
            float h0, l0, h1, l1;
            split_bf16(e0, h0, l0);
            split_bf16(e1, h1, l1);
            bb0 = pack_bf16(h0, h1);
            bb1 = pack_bf16(l0, l1);
        }
        const int cl0 = ((2 * t4) & 3) * 8, cl1 = ((2 * t4 + 1) & 3) * 8;
        const float2 cf = make_float2(__shfl_sync(0xffffffffu, corr, cl0), __shfl_sync(0xffffffffu, corr, cl1));

        // ---------------- pass 2: rescale, accumulate
        if (!last) {
#pragma unroll
            for (int s2 = 0; s2 < KS / 2; ++s2) {
                uint32_t y[4];
                ldsm_x4_t(sa + 64 * s2, y[0], y[1], y[2], y[3]);
                dm_rescale(acc[2 * s2], cf);
                dm_rescale(acc[2 * s2 + 1], cf);
                mma_full(acc[2 * s2], y[0], y[1], y[0], y[1], bb0, bb1);
                mma_full(acc[2 * s2 + 1], y[2], y[3], y[2], y[3], bb0, bb1);
            }
        } else {
            // last chunk: normalise, stage the outputs by stmatrix, clear the
            // accumulators and the running state for the next token
            const float inv_l = 1.f / l_run;
            const float2 fin = make_float2(__shfl_sync(0xffffffffu, inv_l, cl0),
                                           __shfl_sync(0xffffffffu, inv_l, cl1));
            const uint32_t orow = stage0 + (uint32_t)s * a.stage_bytes + (uint32_t)(lane & 7) * a.pitch +
                                  (uint32_t)(cbase + 8 * (lane >> 3)) * 2;
#pragma unroll
            for (int s2 = 0; s2 < KS / 2; ++s2) {
                uint32_t y[4];
                ldsm_x4_t(sa + 64 * s2, y[0], y[1], y[2], y[3]);
                dm_rescale(acc[2 * s2], cf);
                dm_rescale(acc[2 * s2 + 1], cf);
                mma_full(acc[2 * s2], y[0], y[1], y[0], y[1], bb0, bb1);
                mma_full(acc[2 * s2 + 1], y[2], y[3], y[2], y[3], bb0, bb1);
                dm_rescale(acc[2 * s2], fin);
                dm_rescale(acc[2 * s2 + 1], fin);
                stsm_x4_t(orow + 64 * s2, f2_to_bf2(acc[2 * s2][0], acc[2 * s2][1]),
                          f2_to_bf2(acc[2 * s2][2], acc[2 * s2][3]),
                          f2_to_bf2(acc[2 * s2 + 1][0], acc[2 * s2 + 1][1]),
                          f2_to_bf2(acc[2 * s2 + 1][2], acc[2 * s2 + 1][3]));
#pragma unroll
                for (int e2 = 0; e2 < 4; ++e2) { acc[2 * s2][e2] = 0.f; acc[2 * s2 + 1][e2] = 0.f; }
            }
            m_run = -INFINITY;
            l_run = 0.f;
            fence_proxy_async_smem();
            __syncwarp();
            if (lane < a.n_q) {
                if (!*abort_flag)
                    bulk_s2g(a.out + (int64_t)lane * a.out_q_stride_bytes + (t * a.d + cbase) * 2,
                             stage0 + (uint32_t)s * a.stage_bytes + (uint32_t)lane * a.pitch + (uint32_t)cbase * 2,
                             (uint32_t)CW * 2);
                bulk_commit();
            }
        }
        if (++s == a.nstages) { s = 0; par ^= 1u; }
        if (++j == nch) { j = 0; t += gstride; }
        if (++jn == nch) jn = 0;
    }

    if (lane < a.n_q) bulk_wait0();
    if (producer && lane == 0) {
        int never = 0;
        for (int it = issued > a.nstages ? issued - a.nstages : 0; it < issued; ++it)
            mbar_wait_bounded(&full[it % a.nstages], (uint32_t)(it / a.nstages) & 1, &never, a.wait);
    }
}

}  // namespace attnres
