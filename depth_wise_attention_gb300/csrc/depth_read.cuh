// depth_read.cuh -- the fused depth-wise softmax read for sm_103a.
//
// One kernel template serves three entry points:
//   * Full AttnRes (one query, any number of sources),
//   * Block AttnRes phase 1 (the S queries of a block against the N cached
//     block representations, one pass over the cache),
//   * MHAR (H per-subspace heads, block-diagonal read).
// For every token it computes, per source i and query q,
//     s_qi = (w_q * g) . v_i / sqrt(mean(v_i^2) + eps)        (per head for MHAR)
// then the softmax over i, and writes o_q = sum_i alpha_qi v_i (raw values) and
// lse_q = max_i s_qi + log sum_i exp(s_qi - max).
//
// Structure (one persistent CTA per SM, 8 warps):
//   thread 0 also acts as the producer: it streams tiles of [chunk sources] x
//     [tt tokens] x [d] from HBM into a ring of shared-memory stages with 1-D
//     bulk copies (cp.async.bulk, completion counted on one mbarrier per
//     stage).  Stage s of item it is refilled (for item it + nstages) right
//     after the CTA barrier of item it + 1, which every warp reaches only
//     after it has finished reading item it, so no "empty" barrier is needed.
//   each token row is owned by tpr threads (one or more whole warps); a
//     thread owns VPT 16-byte vectors of the row, at vector indices
//     k*tpr + (thread in row), so every shared-memory read and global store
//     of a warp is contiguous.
//   Per stage: pass 1 reads the vectors once and accumulates sum(x^2) and the
//   NQ dots per source with packed f32x2 FMAs; a butterfly warp reduction and
//   one CTA barrier combine the partial sums of the row's warps; each warp
//   then computes the scores and the softmax redundantly (no second barrier);
//   pass 2 re-reads the stage and accumulates the weighted raw values.  When
//   the sources do not fit one stage they are processed in chunks with the
//   online-softmax (running max, running sum, rescaled accumulator) update.
// Every wait is bounded (see mbar_wait_bounded); no thread leaves the item
// loop early, so the CTA barrier can never be left half-arrived.
#pragma once

#include "common.cuh"

namespace attnres {

constexpr int DR_CONSUMER_WARPS = 8;
constexpr int DR_THREADS = DR_CONSUMER_WARPS * 32;
constexpr int DR_CMAX = 8;        // sources per stage, at most
constexpr int DR_MAX_STAGES = 4;

// Sources per chunk an instance takes, so that its source loops have a
// compile-time length: the chunked instances with two vectors per thread
// (8 KB per source and stage at d = 1024..4096) get 6, the most that two
// stages fit with two CTAs per SM; the host caps the chunk at this value.
__host__ __device__ constexpr int dr_chunk_cap(int vpt, bool multi) {
    return multi && vpt == 2 ? 6 : DR_CMAX;
}

struct DepthReadArgs {
    const unsigned char *src;     // source 0, row 0
    int64_t src_stride_bytes;     // bytes between consecutive sources
    int n_src;
    int64_t T;
    int d;                        // channels
    int nvec;                     // d / elements-per-16-byte-vector
    int n_q;                      // real number of queries (<= NQ)
    int H;                        // heads (1 unless MHAR)
    int seg;                      // vectors per head (nvec / H)
    const float *queries;         // [n_q][d]
    const float *gain;            // [d] or nullptr
    float eps;
    unsigned char *out;           // [n_q][T][d]
    int64_t out_q_stride_bytes;   // bytes between queries' outputs
    float *lse;                   // [n_q][H][T] or nullptr
    int tpr;                      // threads per token row (32..256)
    int tt;                       // tokens per tile (256 / tpr)
    int chunk;                    // sources per stage
    int nchunks;
    int nstages;
    uint32_t stage_bytes;         // bytes per stage (multiple of 128)
    uint32_t src_pitch;           // bytes between sources inside a stage (tt * d * esz)
    int64_t ntiles;
    WaitCfg wait;
};

// Shared memory needed besides the stages, for one instantiation.
template <int NQ, int VPT, bool MH>
struct DRLayout {
    static constexpr int HS = MH ? VPT : 1;                 // head slots per thread
    static constexpr int V = HS * DR_CMAX * (1 + NQ);       // values reduced per warp
    static constexpr int R = Bfly<V>::R;                    // slots per lane afterwards
    static constexpr int NPAIR = HS * NQ * DR_CMAX;         // (slot, query, source) pairs
    static constexpr int PJ = (NPAIR + 31) / 32;
    static constexpr size_t bar_bytes = 128;                // mbarriers + abort flag (padded)
    // red[2][8 warps][V]: per-warp partial sums, laid out [row][value][warp in row]
    static constexpr size_t red_floats = 2 * DR_CONSUMER_WARPS * V;
    // aw[8 warps][HS][CMAX][NQ]: softmax weights (or unnormalised exps)
    static constexpr size_t aw_floats = DR_CONSUMER_WARPS * NPAIR;
    static constexpr size_t sw_floats = DR_CONSUMER_WARPS * HS * NQ;
    static constexpr size_t aux_bytes = bar_bytes + 4 * (red_floats + aw_floats + 2 * sw_floats);
    // value index of (head slot, 0 = sum of squares / 1+q = dot with query q, source)
    __host__ __device__ static constexpr int vidx(int hs, int slot, int i) {
        return (hs * (1 + NQ) + slot) * DR_CMAX + i;
    }
};

template <typename Tin, int NQ, int VPT, bool MH, bool MULTI>
__global__ void __launch_bounds__(DR_THREADS, 1) depth_read_kernel(const DepthReadArgs a) {
    using E = Elem<Tin>;
    using L = DRLayout<NQ, VPT, MH>;
    constexpr int EPV = E::EPV;
    constexpr int NP = EPV / 2;
    constexpr int HS = L::HS, V = L::V, R = L::R, NPAIR = L::NPAIR, PJ = L::PJ;
    constexpr int CMAX = DR_CMAX;
    constexpr int CK = dr_chunk_cap(VPT, MULTI);            // sources per chunk, at most

    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char *stages = smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)a.nstages * a.stage_bytes);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(full + DR_MAX_STAGES);
    float *red = reinterpret_cast<float *>(smem + (size_t)a.nstages * a.stage_bytes + L::bar_bytes);
    float *aw = red + L::red_floats;
    float *sw = aw + L::aw_floats;
    float *iw = sw + L::sw_floats;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        for (int s = 0; s < a.nstages; ++s) mbar_init(&full[s], 1);
        *abort_flag = 0;
        mbar_init_fence();
    }
    __syncthreads();

    const int gstride = gridDim.x;
    const int first_tile = blockIdx.x;
    const int my_tiles = first_tile < a.ntiles ? (int)((a.ntiles - first_tile + gstride - 1) / gstride) : 0;
    const int n_items = my_tiles * a.nchunks;

    // ------------------------------------------------------------ producer
    // (thread 0 only) fill the stage of the next item with its chunk of sources.
    const bool producer = (tid == 0) && !a.wait.inject_stall;
    uint64_t pol = 0;
    if (producer) pol = l2_policy_evict_first();
    int p_stage = 0, p_chunk = 0, p_tile = first_tile;     // producer's item cursor
    auto issue_next = [&]() {
        const int64_t t0 = (int64_t)p_tile * a.tt;
        const int64_t rem = a.T - t0;
        const int ntok = rem < a.tt ? (int)rem : a.tt;
        const int i0 = p_chunk * a.chunk;
        const int nc = min(a.chunk, a.n_src - i0);
        const uint32_t bytes = (uint32_t)ntok * (uint32_t)a.d * E::BYTES;
        mbar_arrive_expect_tx(&full[p_stage], bytes * nc);
        const unsigned char *g = a.src + (int64_t)i0 * a.src_stride_bytes + t0 * a.d * E::BYTES;
        unsigned char *dst = stages + (size_t)p_stage * a.stage_bytes;
        for (int i = 0; i < nc; ++i)
            bulk_g2s(dst + (size_t)i * a.src_pitch, g + (int64_t)i * a.src_stride_bytes, bytes,
                     &full[p_stage], pol);
        if (++p_stage == a.nstages) p_stage = 0;
        if (++p_chunk == a.nchunks) { p_chunk = 0; p_tile += gstride; }
    };
    int issued = 0;
    if (producer) {
        for (; issued < n_items && issued < a.nstages; ++issued) issue_next();
    }

    // ------------------------------------------------------------ consumers
    const int r = tid / a.tpr;          // token row inside the tile
    const int tr = tid - r * a.tpr;     // thread inside the row
    const int wr = tr >> 5;             // warp inside the row
    const int nwr = a.tpr >> 5;
    const float inv_dh = 1.f / (float)((MH ? a.seg : a.nvec) * EPV);

    int vid[VPT];
    bool vok[VPT];
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        vid[k] = k * a.tpr + tr;
        vok[k] = vid[k] < a.nvec;
    }
    // pseudo-queries with the RMSNorm gain folded in: (w * g) . x / rms(x)
    float2 wq[NQ][VPT][NP];
#pragma unroll
    for (int q = 0; q < NQ; ++q)
#pragma unroll
        for (int k = 0; k < VPT; ++k)
#pragma unroll
            for (int p = 0; p < NP; ++p) {
                float2 w = make_float2(0.f, 0.f);
                if (q < a.n_q && vok[k]) {
                    const int c = vid[k] * EPV + 2 * p;
                    w = make_float2(__ldg(a.queries + (size_t)q * a.d + c), __ldg(a.queries + (size_t)q * a.d + c + 1));
                    if (a.gain) { w.x *= __ldg(a.gain + c); w.y *= __ldg(a.gain + c + 1); }
                }
                wq[q][k][p] = w;
            }
    // where each butterfly slot of this lane lands in the per-row partial-sum table
    int slot_idx[R];
#pragma unroll
    for (int j = 0; j < R; ++j) slot_idx[j] = bfly_slot<V>(lane, j);

    // per-warp shared areas
    float *awp = aw + (size_t)warp * NPAIR;
    float *swp = sw + (size_t)warp * HS * NQ;
    float *iwp = iw + (size_t)warp * HS * NQ;

    float2 acc[NQ][VPT][NP];
    float m_run[PJ], l_run[PJ];
#pragma unroll
    for (int j = 0; j < PJ; ++j) { m_run[j] = -INFINITY; l_run[j] = 0.f; }

    int s = 0, c = 0, tile = first_tile;
    uint32_t par = 0;
    for (int it = 0; it < n_items; ++it) {
        const bool first_chunk = (c == 0), last_chunk = (c == a.nchunks - 1);
        const int64_t t = (int64_t)tile * a.tt + r;
        const bool row_ok = t < a.T;
        const int nc = min(a.chunk, a.n_src - c * a.chunk);
        mbar_wait_bounded(&full[s], par, abort_flag, a.wait);

        // this thread's vectors of source 0 in the stage; source i is i*src_pitch further
        const unsigned char *sb = stages + (size_t)s * a.stage_bytes + (size_t)r * a.d * E::BYTES;
        const uint4 *vp[VPT];
#pragma unroll
        for (int k = 0; k < VPT; ++k) vp[k] = reinterpret_cast<const uint4 *>(sb + (size_t)vid[k] * 16);
        const int pitch4 = (int)(a.src_pitch >> 4);     // in uint4

        // ---------------- pass 1: sum of squares and query dots per source
        float v[V];
#pragma unroll
        for (int i = 0; i < CMAX; ++i) {
            float2 t2[HS][1 + NQ];
            if (i < CK && i < nc) {
#pragma unroll
                for (int k = 0; k < VPT; ++k) {
                    const int h = MH ? k : 0;
                    float2 x[NP];
                    if (vok[k]) {
                        E::unpack(vp[k][i * pitch4], x);
                    } else {
#pragma unroll
                        for (int p = 0; p < NP; ++p) x[p] = make_float2(0.f, 0.f);
                    }
                    const bool init = MH ? true : (k == 0);
#pragma unroll
                    for (int p = 0; p < NP; ++p) {
                        if (init && p == 0) {
                            t2[h][0] = fmul2(x[p], x[p]);
#pragma unroll
                            for (int q = 0; q < NQ; ++q) t2[h][1 + q] = fmul2(x[p], wq[q][k][p]);
                        } else {
                            t2[h][0] = ffma2(x[p], x[p], t2[h][0]);
#pragma unroll
                            for (int q = 0; q < NQ; ++q) t2[h][1 + q] = ffma2(x[p], wq[q][k][p], t2[h][1 + q]);
                        }
                    }
                }
#pragma unroll
                for (int h = 0; h < HS; ++h)
#pragma unroll
                    for (int y = 0; y <= NQ; ++y) v[L::vidx(h, y, i)] = t2[h][y].x + t2[h][y].y;
            } else {
#pragma unroll
                for (int h = 0; h < HS; ++h)
#pragma unroll
                    for (int y = 0; y <= NQ; ++y) v[L::vidx(h, y, i)] = 0.f;
            }
        }
        butterfly_reduce<V>(v, lane);
        // partial-sum table of this item: [row][value][warp in row]
        float *redb = red + (size_t)(it & 1) * DR_CONSUMER_WARPS * V;
        float *rrow = redb + (size_t)r * nwr * V;
#pragma unroll
        for (int j = 0; j < R; ++j)
            if (slot_idx[j] >= 0) rrow[slot_idx[j] * nwr + wr] = v[j];
        __syncthreads();
        // every warp has finished item it-1: refill its stage for item it-1+nstages
        if (producer && it >= 1 && issued < n_items && !*abort_flag) { issue_next(); ++issued; }

        // ---------------- scores and softmax over the sources of this chunk
#pragma unroll
        for (int j = 0; j < PJ; ++j) {
            const int pidx = lane + 32 * j;
            const int h = pidx / (NQ * CMAX);
            const int q = (pidx / CMAX) % NQ;
            const int i = pidx % CMAX;
            const bool pv = pidx < NPAIR && i < nc;
            float score = -INFINITY;
            int head = 0;
            bool lse_writer = false;
            if (pidx < NPAIR) {
                float ss = 0.f, dt = 0.f;
                if (MH) {
                    head = (h * a.tpr + 32 * wr) / a.seg;
                    // slots past the row (masked lanes) map to no head
                    lse_writer = head < a.H && (h * a.tpr + 32 * wr) == head * a.seg;
                    for (int kk = 0; kk < VPT; ++kk)
                        for (int ww = 0; ww < nwr; ++ww)
                            if ((kk * a.tpr + 32 * ww) / a.seg == head) {
                                ss += rrow[(size_t)L::vidx(kk, 0, i) * nwr + ww];
                                dt += rrow[(size_t)L::vidx(kk, 1 + q, i) * nwr + ww];
                            }
                } else {
                    lse_writer = (wr == 0);
                    const float *pss = rrow + (size_t)L::vidx(0, 0, i) * nwr;
                    const float *pdt = rrow + (size_t)L::vidx(0, 1 + q, i) * nwr;
                    if (nwr == 8) {
                        const float4 a0 = reinterpret_cast<const float4 *>(pss)[0];
                        const float4 a1 = reinterpret_cast<const float4 *>(pss)[1];
                        const float4 b0 = reinterpret_cast<const float4 *>(pdt)[0];
                        const float4 b1 = reinterpret_cast<const float4 *>(pdt)[1];
                        ss = ((a0.x + a0.y) + (a0.z + a0.w)) + ((a1.x + a1.y) + (a1.z + a1.w));
                        dt = ((b0.x + b0.y) + (b0.z + b0.w)) + ((b1.x + b1.y) + (b1.z + b1.w));
                    } else {
                        for (int ww = 0; ww < nwr; ++ww) { ss += pss[ww]; dt += pdt[ww]; }
                    }
                }
                if (pv) score = key_score(dt, ss, inv_dh, a.eps);
            }
            const float cmax = seg_max<CMAX>(score);
            const bool write_lse = lse_writer && i == 0 && pidx < NPAIR && q < a.n_q && row_ok &&
                                   a.lse != nullptr && !*abort_flag;
            const int64_t lse_off = ((int64_t)q * a.H + head) * a.T + t;
            // weights stored [head slot][source][query] so pass 2 reads NQ at once
            const int aw_off = (h * CMAX + i) * NQ + q;
            if (!MULTI) {
                const float e = pv ? __expf(score - cmax) : 0.f;
                const float sum = seg_sum<CMAX>(e);
                if (pidx < NPAIR) awp[aw_off] = e / sum;
                if (write_lse) a.lse[lse_off] = cmax + __logf(sum);
            } else {
                if (first_chunk) { m_run[j] = -INFINITY; l_run[j] = 0.f; }
                const float mnew = fmaxf(m_run[j], cmax);
                const float scale = (m_run[j] == -INFINITY) ? 0.f : __expf(m_run[j] - mnew);
                const float e = pv ? __expf(score - mnew) : 0.f;
                const float sum = seg_sum<CMAX>(e);
                l_run[j] = l_run[j] * scale + sum;
                m_run[j] = mnew;
                if (pidx < NPAIR) awp[aw_off] = e;
                if (i == 0 && pidx < NPAIR) {
                    swp[h * NQ + q] = scale;
                    if (last_chunk) iwp[h * NQ + q] = 1.f / l_run[j];
                }
                if (last_chunk && write_lse) a.lse[lse_off] = m_run[j] + __logf(l_run[j]);
            }
        }
        __syncwarp();

        // ---------------- pass 2: weighted sum of the raw source values
        if (MULTI && !first_chunk) {
#pragma unroll
            for (int q = 0; q < NQ; ++q)
#pragma unroll
                for (int k = 0; k < VPT; ++k) {
                    const float sc = swp[(MH ? k : 0) * NQ + q];
                    const float2 sc2 = make_float2(sc, sc);
#pragma unroll
                    for (int p = 0; p < NP; ++p) acc[q][k][p] = fmul2(acc[q][k][p], sc2);
                }
        }
#pragma unroll
        for (int i = 0; i < CMAX; ++i) {
            if (i < CK && i < nc) {
                float al[HS][NQ];
#pragma unroll
                for (int h = 0; h < HS; ++h) {
                    const float *ap = awp + (h * CMAX + i) * NQ;
                    if (NQ % 4 == 0) {
#pragma unroll
                        for (int q4 = 0; q4 < NQ; q4 += 4) {
                            const float4 f = reinterpret_cast<const float4 *>(ap)[q4 / 4];
                            al[h][q4] = f.x; al[h][q4 + 1] = f.y; al[h][q4 + 2] = f.z; al[h][q4 + 3] = f.w;
                        }
                    } else {
#pragma unroll
                        for (int q = 0; q < NQ; ++q) al[h][q] = ap[q];
                    }
                }
                const bool init = (!MULTI || first_chunk) && i == 0;
#pragma unroll
                for (int k = 0; k < VPT; ++k) {
                    float2 x[NP];
                    if (vok[k]) {
                        E::unpack(vp[k][i * pitch4], x);
                    } else {
#pragma unroll
                        for (int p = 0; p < NP; ++p) x[p] = make_float2(0.f, 0.f);
                    }
                    const int h = MH ? k : 0;
#pragma unroll
                    for (int q = 0; q < NQ; ++q) {
                        const float2 al2 = make_float2(al[h][q], al[h][q]);
#pragma unroll
                        for (int p = 0; p < NP; ++p)
                            acc[q][k][p] = init ? fmul2(x[p], al2) : ffma2(x[p], al2, acc[q][k][p]);
                    }
                }
            }
        }

        if ((!MULTI || last_chunk) && row_ok && !*abort_flag) {
            unsigned char *ob = a.out + (t * a.d) * E::BYTES;
#pragma unroll
            for (int q = 0; q < NQ; ++q) {
                if (q < a.n_q) {
#pragma unroll
                    for (int k = 0; k < VPT; ++k) {
                        if (vok[k]) {
                            float2 y[NP];
                            if (MULTI) {
                                const float sc = iwp[(MH ? k : 0) * NQ + q];
                                const float2 sc2 = make_float2(sc, sc);
#pragma unroll
                                for (int p = 0; p < NP; ++p) y[p] = fmul2(acc[q][k][p], sc2);
                            } else {
#pragma unroll
                                for (int p = 0; p < NP; ++p) y[p] = acc[q][k][p];
                            }
                            stg128_cs(ob + (int64_t)vid[k] * 16, E::pack(y));
                        }
                    }
                }
                ob += a.out_q_stride_bytes;
            }
        }
        // advance the item cursor
        if (++s == a.nstages) { s = 0; par ^= 1u; }
        if (++c == a.nchunks) { c = 0; tile += gstride; }
    }

    // Drain: after an abort the consumers stop waiting, so copies may still be
    // in flight; they must land before the CTA exits.
    if (producer) {
        int never = 0;
        for (int it = issued > a.nstages ? issued - a.nstages : 0; it < issued; ++it)
            mbar_wait_bounded(&full[it % a.nstages], (uint32_t)(it / a.nstages) & 1, &never, a.wait);
    }
}

}  // namespace attnres
