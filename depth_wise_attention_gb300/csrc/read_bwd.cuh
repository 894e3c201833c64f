// read_bwd.cuh -- backward of the depth-wise softmax read for sm_103a.
//
// For n_q queries over n_src sources and output gradients dout_q, per token
// (alpha recomputed from the sources; the chain rule through
// h_q = sum_i alpha_qi v_i, alpha_q = softmax_i(s_q), s_qi = w_q . g*v_i/r_i,
// r_i = sqrt(mean(v_i^2) + eps)):
//     ds_qi = alpha_qi (dout_q . v_i - sum_j alpha_qj dout_q . v_j)
//     b_qi  = ds_qi / r_i
//     c_i   = - sum_q ds_qi ((w_q*g) . v_i) / (d r_i^3)
//     dv_i  = sum_q alpha_qi dout_q + sum_q b_qi (w_q*g) + c_i v_i
//     U_q  += sum_i b_qi v_i           (summed over the tokens)
// and after all tokens dq_q = g * U_q, dgain = sum_q w_q * U_q.  A gradient of
// the read's log-sum-exp (Block phase 1's lse output) adds alpha_qi dlse_q to
// ds_qi, since d lse_q / d s_qi = alpha_qi.
//
// Structure: the forward's streaming layout.  One persistent CTA per SM;
// thread 0 streams each tile's n_src source rows and n_q gradient rows into
// a ring of shared-memory stages with 1-D bulk copies (bounded mbarrier
// waits); a token row is owned by tpr threads, each holding VPT 16-byte
// vectors.  Pass A accumulates per source sum(v^2), (w_q*g).v and dout_q.v
// with packed f32x2 FMAs; a butterfly warp reduction and one CTA barrier give
// the totals; lanes (q, i) of every warp then recompute the softmax and form
// alpha, b and c (kept per warp in shared memory, no second barrier); pass B
// re-reads the stage, writes dv and accumulates U in registers.  Each CTA row
// writes its U to the caller's workspace, and read_bwd_finish_kernel reduces
// the workspace in a fixed order (deterministic) into dq and dgain.
//
// Per-head mode (MH, the backward of the MHAR read): every quantity above is
// taken per head over the head's slice of channels (d becomes d/H in c_i).
// Each warp then owns VPT runs of 32 consecutive vectors, so a run never
// straddles a head when a head is a multiple of 32 vectors: with HG == 1 a
// warp's VPT runs lie in one head and its values are reduced together; with
// HG == VPT each run is its own group.  The coefficient lanes of a group sum
// the table entries of all groups of its head.
//
// Query groups (QG): with QG == 2 one launch takes up to 2 * NQ queries.  The
// stage holds every query's gradient rows; each tile runs passes A and B
// once per group of NQ queries on the same staged sources, so the sources
// are read from memory once, and the second group adds into the dsrc rows
// the first group of the same tile has just written (L2-resident).
#pragma once

#include "common.cuh"

namespace attnres {

// Bulk prefetch of global memory into L2 (no shared memory, no completion).
// src 16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_prefetch_l2(const void *src_gmem, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src_gmem), "r"(bytes) : "memory");
}

constexpr int RB_THREADS = 256;
constexpr int RB_MAX_STAGES = 4;

struct ReadBwdArgs {
    const unsigned char *src;       // source 0, token 0
    int64_t src_stride_bytes;       // between sources
    int n_src;
    int64_t T;
    int d;
    int nvec;                       // 16-byte vectors per row
    int n_q;
    const float *queries;           // [n_q][d]
    const float *gain;              // [d] or nullptr
    float eps;
    const unsigned char *dout;      // [n_q][T][d]
    const float *dlse;              // [n_q][T] gradient of each query's log-sum-exp, or nullptr
    unsigned char *dsrc;            // [n_src] x (dsrc_stride_bytes apart) [T][d]
    int64_t dsrc_stride_bytes;
    int accumulate;                 // 1: dsrc += gradient
    float *ws;                      // [gridDim.x * tt][n_q][d] partial U
    int tpr;
    int tt;                         // token rows per tile
    int nstages;
    uint32_t stage_bytes;
    uint32_t row_pitch;             // bytes of one tensor's tile rows in a stage (tt * d * esize)
    int64_t ntiles;
    int vph;                        // 16-byte vectors per head (nvec for one head)
    int nheads;
    float inv_dh;                   // 1 / channels per head
    WaitCfg wait;
};

template <int NQ, int NS, int HG = 1>
struct RBLayout {
    static constexpr int V = NS * (1 + 2 * NQ);             // values reduced per token row and group
    static constexpr int R = Bfly<HG * V>::R;
    static constexpr size_t bar_bytes = 128;
    // [2][row][value][group in row]
    static constexpr size_t red_floats = 2 * (RB_THREADS / 32) * HG * V;
    // per warp and group: alpha, b, c
    static constexpr size_t coef_floats = (RB_THREADS / 32) * HG * NS * (2 * NQ + 1);
    static constexpr size_t aux_bytes = bar_bytes + 4 * (red_floats + coef_floats);
    // value index: sum of squares of source i, then (w_q*g).v_i, then dout_q.v_i
    __host__ __device__ static constexpr int iss(int i) { return i; }
    __host__ __device__ static constexpr int isw(int q, int i) { return NS + q * NS + i; }
    __host__ __device__ static constexpr int isd(int q, int i) { return NS + NQ * NS + q * NS + i; }
};

template <typename Tin, int NQ, int NS, int VPT, bool MH = false, int HG = 1, int QG = 1>
__global__ void __launch_bounds__(RB_THREADS, 1) read_bwd_kernel(const ReadBwdArgs a) {
    using E = Elem<Tin>;
    using L = RBLayout<NQ, NS, HG>;
    constexpr int EPV = E::EPV;
    constexpr int NP = EPV / 2;
    constexpr int V = L::V, R = L::R;
    static_assert(NQ * NS <= 32, "one lane per (query, source) pair");
    static_assert(HG == 1 || (MH && HG == VPT), "groups per warp: one, or one per run in per-head mode");

    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char *stages = smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)a.nstages * a.stage_bytes);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(full + RB_MAX_STAGES);
    float *red = reinterpret_cast<float *>(smem + (size_t)a.nstages * a.stage_bytes + L::bar_bytes);
    float *coef = red + L::red_floats;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int s = 0; s < a.nstages; ++s) mbar_init(&full[s], 1);
        *abort_flag = 0;
        mbar_init_fence();
    }
    __syncthreads();

    const int gstride = gridDim.x;
    const int n_items = blockIdx.x < a.ntiles ? (int)((a.ntiles - blockIdx.x + gstride - 1) / gstride) : 0;

    // ------------------------------------------------------------ producer
    const bool producer = (tid == 0) && !a.wait.inject_stall;
    uint64_t pol = 0;
    if (producer) pol = l2_policy_evict_first();
    int p_stage = 0;
    int64_t p_tile = blockIdx.x;
    auto issue_next = [&]() {
        const int64_t t0 = p_tile * a.tt;
        const int64_t rem = a.T - t0;
        const int ntok = rem < a.tt ? (int)rem : a.tt;
        const uint32_t bytes = (uint32_t)ntok * (uint32_t)a.d * E::BYTES;
        mbar_arrive_expect_tx(&full[p_stage], bytes * (uint32_t)(a.n_src + a.n_q));
        unsigned char *dst = stages + (size_t)p_stage * a.stage_bytes;
        const int64_t off = t0 * a.d * E::BYTES;
        for (int i = 0; i < a.n_src; ++i)
            bulk_g2s(dst + (size_t)i * a.row_pitch, a.src + (int64_t)i * a.src_stride_bytes + off, bytes,
                     &full[p_stage], pol);
        for (int q = 0; q < a.n_q; ++q)
            bulk_g2s(dst + (size_t)(a.n_src + q) * a.row_pitch, a.dout + (q * a.T * a.d) * E::BYTES + off, bytes,
                     &full[p_stage], pol);
        // a pass that adds into dsrc reads the tile's gradient rows back in
        // pass B: have them in L2 by then
        if (a.accumulate)
            for (int i = 0; i < a.n_src; ++i) bulk_prefetch_l2(a.dsrc + (int64_t)i * a.dsrc_stride_bytes + off, bytes);
        if (++p_stage == a.nstages) p_stage = 0;
        p_tile += gstride;
    };
    int issued = 0;
    if (producer)
        for (; issued < n_items && issued < a.nstages; ++issued) issue_next();

    // ------------------------------------------------------------ constants
    const int r = tid / a.tpr, tr = tid - r * a.tpr;
    const int wr = tr >> 5, nwr = a.tpr >> 5;
    const int ngr = nwr * HG;     // reduction groups per token row
    const float inv_d = a.inv_dh;
    int vid[VPT];
    bool vok[VPT];
    float2 wg[QG][NQ][VPT][NP];   // w_q * g on this thread's channels, per query group
    float2 U[QG][NQ][VPT][NP];    // sum over tokens of sum_i b_qi v_i
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        vid[k] = MH ? (wr * VPT + k) * 32 + lane : k * a.tpr + tr;
        vok[k] = vid[k] < a.nvec;
#pragma unroll
        for (int qg = 0; qg < QG; ++qg)
#pragma unroll
            for (int q = 0; q < NQ; ++q)
#pragma unroll
                for (int p = 0; p < NP; ++p) {
                    const int qq = qg * NQ + q;
                    float2 w = make_float2(0.f, 0.f);
                    if (qq < a.n_q && vok[k]) {
                        const int c = vid[k] * EPV + 2 * p;
                        w = make_float2(__ldg(a.queries + (size_t)qq * a.d + c),
                                        __ldg(a.queries + (size_t)qq * a.d + c + 1));
                        if (a.gain) { w.x *= __ldg(a.gain + c); w.y *= __ldg(a.gain + c + 1); }
                    }
                    wg[qg][q][k][p] = w;
                    U[qg][q][k][p] = make_float2(0.f, 0.f);
                }
    }
    // table offset of each value this lane holds after the butterfly: value
    // jj of local group g goes to [jj][wr * HG + g] of the row's table
    int slot_off[R];
#pragma unroll
    for (int j = 0; j < R; ++j) {
        const int idx = bfly_slot<HG * V>(lane, j);
        const int g = idx / V, jj = idx - g * V;
        slot_off[j] = idx >= 0 ? jj * ngr + wr * HG + g : -1;
    }
    constexpr int CS = 2 * NQ + 1;
    float *cw = coef + (size_t)warp * HG * NS * CS;   // [group][i][alpha_q..., b_q..., c]
    // the table groups that make up the head of each of this warp's groups
    int g_first[HG], g_count;
    {
        const int cv = 32 * VPT / HG;                  // vectors per group
        g_count = MH ? a.vph / cv : nwr;
#pragma unroll
        for (int g = 0; g < HG; ++g) {
            int h = MH ? (wr * HG + g) * cv / a.vph : 0;
            if (h >= a.nheads) h = a.nheads - 1;       // a group past the row: computed, never used
            g_first[g] = h * g_count;
        }
    }

    int s = 0;
    uint32_t par = 0;
    int64_t tile = blockIdx.x;
    for (int it = 0; it < n_items; ++it) {
        const int64_t t = tile * a.tt + r;
        const bool row_ok = t < a.T;
        mbar_wait_bounded(&full[s], par, abort_flag, a.wait);
        const unsigned char *sb = stages + (size_t)s * a.stage_bytes + (size_t)r * a.d * E::BYTES;
#pragma unroll
        for (int qg = 0; qg < QG; ++qg) {
        const int q0 = qg * NQ;             // first query of this group
        // the second group adds into the rows the first one has written
        const bool acc = qg > 0 || a.accumulate;

        // ---------------- pass A: sum(v^2), (w*g).v, dout.v per source
        float2 dl[NQ][VPT][NP];   // this token's output gradients on my channels
#pragma unroll
        for (int q = 0; q < NQ; ++q)
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                if (q0 + q < a.n_q && vok[k]) {
                    E::unpack(*reinterpret_cast<const uint4 *>(sb + (size_t)(a.n_src + q0 + q) * a.row_pitch +
                                                               (size_t)vid[k] * 16),
                              dl[q][k]);
                } else {
#pragma unroll
                    for (int p = 0; p < NP; ++p) dl[q][k][p] = make_float2(0.f, 0.f);
                }
            }
        float v[HG * V];
#pragma unroll
        for (int i = 0; i < NS; ++i) {
            float2 ss[HG], sw[HG][NQ], sd[HG][NQ];
#pragma unroll
            for (int g = 0; g < HG; ++g) {
                ss[g] = make_float2(0.f, 0.f);
#pragma unroll
                for (int q = 0; q < NQ; ++q) { sw[g][q] = make_float2(0.f, 0.f); sd[g][q] = make_float2(0.f, 0.f); }
            }
            if (i < a.n_src) {
#pragma unroll
                for (int k = 0; k < VPT; ++k) {
                    if (!vok[k]) continue;
                    constexpr int one = HG == 1 ? 1 : 0;
                    const int g = one ? 0 : k;
                    float2 x[NP];
                    E::unpack(*reinterpret_cast<const uint4 *>(sb + (size_t)i * a.row_pitch + (size_t)vid[k] * 16), x);
#pragma unroll
                    for (int p = 0; p < NP; ++p) {
                        ss[g] = ffma2(x[p], x[p], ss[g]);
#pragma unroll
                        for (int q = 0; q < NQ; ++q) {
                            sw[g][q] = ffma2(x[p], wg[qg][q][k][p], sw[g][q]);
                            sd[g][q] = ffma2(x[p], dl[q][k][p], sd[g][q]);
                        }
                    }
                }
            }
#pragma unroll
            for (int g = 0; g < HG; ++g) {
                v[g * V + L::iss(i)] = ss[g].x + ss[g].y;
#pragma unroll
                for (int q = 0; q < NQ; ++q) {
                    v[g * V + L::isw(q, i)] = sw[g][q].x + sw[g][q].y;
                    v[g * V + L::isd(q, i)] = sd[g][q].x + sd[g][q].y;
                }
            }
        }
        butterfly_reduce<HG * V>(v, lane);
        float *rrow = red + (size_t)((it * QG + qg) & 1) * (RB_THREADS / 32) * HG * V + (size_t)r * ngr * V;
#pragma unroll
        for (int j = 0; j < R; ++j)
            if (slot_off[j] >= 0) rrow[slot_off[j]] = v[j];
        __syncthreads();
        // every warp has finished item it-1: refill its stage for item it-1+nstages
        if (qg == 0 && producer && it >= 1 && issued < n_items && !*abort_flag) { issue_next(); ++issued; }

        // ---------------- per-token coefficients: lane (q, i) = q*NS + i, for
        // each group of this warp (its head's table groups summed)
#pragma unroll
        for (int g = 0; g < HG; ++g) {
            const int q = lane / NS, i = lane - q * NS;
            const bool pv = q < NQ && q0 + q < a.n_q && i < a.n_src;
            float ss = 0.f, sw = 0.f, sd = 0.f;
            if (q < NQ) {
                for (int w = g_first[g]; w < g_first[g] + g_count; ++w) {
                    ss += rrow[L::iss(i) * ngr + w];
                    sw += rrow[L::isw(q, i) * ngr + w];
                    sd += rrow[L::isd(q, i) * ngr + w];
                }
            }
            const float ms = fmaf(ss, inv_d, a.eps);
            const float rinv = ms > 0.f ? rsqrtf(ms) : 0.f;        // 1 / r_i (0 for a zero key)
            const float score = pv ? sw * rinv : -INFINITY;
            const float mx = seg_max<NS>(score);
            const float e = pv ? __expf(score - mx) : 0.f;
            // every lane takes part in the shuffles (no reduction under a branch)
            const float esum = seg_sum<NS>(e);
            const float alpha = pv ? e / esum : 0.f;
            const float mean = seg_sum<NS>(alpha * sd);
            const float dl = (a.dlse != nullptr && pv && row_ok) ? __ldg(a.dlse + (int64_t)(q0 + q) * a.T + t) : 0.f;
            const float ds = alpha * (sd - mean + dl);
            const float b = ds * rinv;
            float cpart = -ds * sw * rinv * rinv * rinv * inv_d;
            if (NQ == 2) cpart += __shfl_xor_sync(0xffffffffu, cpart, NS);
            if (q < NQ) {
                float *cg = cw + g * NS * CS;
                cg[i * CS + q] = alpha;
                cg[i * CS + NQ + q] = b;
                if (q == 0) cg[i * CS + 2 * NQ] = cpart;
            }
        }
        __syncwarp();

        // ---------------- pass B: dv and the U sums (rows past the end of the
        // sequence hold stale stage bytes and take no part)
#pragma unroll
        for (int i = 0; i < NS; ++i) {
            if (i >= a.n_src || !row_ok) break;
            // the values to add to (accumulate), loaded before the gradient is
            // formed (with 4 vectors a thread, where registers are short, at use)
            constexpr bool EARLY = VPT <= 2;
            uint4 zraw[VPT];
            if (EARLY && acc) {
#pragma unroll
                for (int k = 0; k < VPT; ++k)
                    if (vok[k])
                        zraw[k] = *reinterpret_cast<const uint4 *>(a.dsrc + (int64_t)i * a.dsrc_stride_bytes +
                                                                  (t * a.d + (int64_t)vid[k] * EPV) * E::BYTES);
            }
            float alg[HG][NQ], bqg[HG][NQ], cig[HG];
#pragma unroll
            for (int g = 0; g < HG; ++g) {
                const float *cg = cw + g * NS * CS;
#pragma unroll
                for (int q = 0; q < NQ; ++q) { alg[g][q] = cg[i * CS + q]; bqg[g][q] = cg[i * CS + NQ + q]; }
                cig[g] = cg[i * CS + 2 * NQ];
            }
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                if (!vok[k]) continue;
                constexpr int one = HG == 1 ? 1 : 0;
                const int g = one ? 0 : k;
                const float *al = alg[g], *bq = bqg[g];
                const float2 c2 = make_float2(cig[g], cig[g]);
                float2 x[NP], y[NP];
                E::unpack(*reinterpret_cast<const uint4 *>(sb + (size_t)i * a.row_pitch + (size_t)vid[k] * 16), x);
#pragma unroll
                for (int p = 0; p < NP; ++p) {
                    y[p] = fmul2(c2, x[p]);
#pragma unroll
                    for (int q = 0; q < NQ; ++q) {
                        y[p] = ffma2(make_float2(al[q], al[q]), dl[q][k][p], y[p]);
                        y[p] = ffma2(make_float2(bq[q], bq[q]), wg[qg][q][k][p], y[p]);
                        U[qg][q][k][p] = ffma2(make_float2(bq[q], bq[q]), x[p], U[qg][q][k][p]);
                    }
                }
                if (!*abort_flag) {
                    unsigned char *gp = a.dsrc + (int64_t)i * a.dsrc_stride_bytes +
                                        (t * a.d + (int64_t)vid[k] * EPV) * E::BYTES;
                    if (acc) {
                        float2 z[NP];
                        E::unpack(EARLY ? zraw[k] : *reinterpret_cast<const uint4 *>(gp), z);
#pragma unroll
                        for (int p = 0; p < NP; ++p) y[p] = make_float2(y[p].x + z[p].x, y[p].y + z[p].y);
                    }
                    // the first of two groups keeps its rows in L2 for the second
                    if (QG > 1 && qg == 0) *reinterpret_cast<uint4 *>(gp) = E::pack(y);
                    else stg128_cs(gp, E::pack(y));
                }
            }
        }
        }  // query groups
        if (++s == a.nstages) { s = 0; par ^= 1u; }
        tile += gstride;
    }

    // this row's U: one partial per (CTA, row) in the workspace
    if (!*abort_flag) {
        float *wrow = a.ws + ((size_t)blockIdx.x * a.tt + r) * (size_t)a.n_q * a.d;
#pragma unroll
        for (int qg = 0; qg < QG; ++qg)
#pragma unroll
            for (int q = 0; q < NQ; ++q)
#pragma unroll
                for (int k = 0; k < VPT; ++k)
                    if (qg * NQ + q < a.n_q && vok[k])
#pragma unroll
                        for (int p = 0; p < NP; ++p)
                            *reinterpret_cast<float2 *>(wrow + (size_t)(qg * NQ + q) * a.d + vid[k] * EPV + 2 * p) =
                                U[qg][q][k][p];
    }
    if (producer) {
        int never = 0;
        for (int it = issued > a.nstages ? issued - a.nstages : 0; it < issued; ++it)
            mbar_wait_bounded(&full[it % a.nstages], (uint32_t)(it / a.nstages) & 1, &never, a.wait);
    }
}

// Arguments of read_bwd_finish_kernel (kernels_bwd.cu), which sums the
// workspace's per-row partials in a fixed order: dq_q = g * U_q,
// dgain = sum_q w_q * U_q.
struct ReadBwdFinishArgs {
    const float *ws;
    int nparts;
    int n_q;
    int d;
    const float *queries;
    const float *gain;
    float *dq;                      // [n_q][d]
    float *dgain;                   // [d] or nullptr
    int accumulate_dgain;           // 1: dgain += (a later group of queries)
};

}  // namespace attnres
