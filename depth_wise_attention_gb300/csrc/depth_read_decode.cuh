// depth_read_decode.cuh -- the depth read for few tokens (decode-shaped calls).
//
// Same operation as depth_read.cuh for one head (Full AttnRes, Block phase 1):
// per token s_qi = (w_q * g) . v_i / sqrt(mean(v_i^2) + eps), alpha = softmax_i,
// o_q = sum_i alpha_qi v_i, lse_q.  With few tokens the streaming kernels,
// one CTA per token, pay a whole per-token chain (query fragments, the token's
// sources through shared-memory stages, two passes, bulk stores) on one SM.
// Here a token is spread over a thread-block cluster of cs CTAs instead: CTA
// `rank` holds the 16-byte vectors [rank*vpc, (rank+1)*vpc) of every source,
// one vector per thread, straight in registers (no staging); the per-source
// sums of squares and query dots are reduced by a warp butterfly, a shared
// table and one exchange through distributed shared memory; after the single
// cluster barrier every CTA has the totals, computes the softmax and writes its
// slice of the outputs.
#pragma once

#include <cooperative_groups.h>

#include "common.cuh"

namespace attnres {

constexpr int DEC_MAX_CS = 8;            // CTAs per token (portable cluster size)
constexpr int DEC_MAX_THREADS = 256;

struct DecodeArgs {
    const unsigned char *src;
    int64_t src_stride_bytes;
    int n_src;
    int64_t T;
    int d;
    int n_q;
    const float *queries;                 // [n_q][d]
    const float *gain;                    // [d] or nullptr
    float eps;
    unsigned char *out;                   // [n_q][T][d]
    int64_t out_q_stride_bytes;
    float *lse;                           // [n_q][T] or nullptr
    int cs;                               // CTAs per token (the cluster size)
    int vpc;                              // vectors per CTA = threads per CTA
};

template <int NQ, int NS>
struct DecLayout {
    static constexpr int V = NS * (1 + NQ);                 // per source: sum of squares, NQ dots
    static constexpr int R = Bfly<V>::R;
    static constexpr int NW = DEC_MAX_THREADS / 32;
    // red[NW][V] (per-warp partials), xch[DEC_MAX_CS][V] (the cluster's CTA totals)
    static constexpr size_t smem_floats = (size_t)NW * V + (size_t)DEC_MAX_CS * V;
};

template <typename Tin, int NQ, int NS>
__global__ void __launch_bounds__(DEC_MAX_THREADS) depth_read_decode_kernel(const DecodeArgs a) {
    using E = Elem<Tin>;
    using L = DecLayout<NQ, NS>;
    constexpr int EPV = E::EPV, NP = EPV / 2;
    constexpr int V = L::V, R = L::R;
    static_assert(NQ * NS <= 32, "one lane per (query, source) pair");
    namespace cg = cooperative_groups;
    cg::cluster_group cluster = cg::this_cluster();

    __shared__ float red[L::NW * V];
    __shared__ float xch[DEC_MAX_CS * V];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nw = blockDim.x >> 5;
    const int rank = (int)cluster.block_rank();
    const int64_t t = blockIdx.x / a.cs;
    const int vec = rank * a.vpc + tid;              // this thread's 16-byte vector of the row
    const int c0 = vec * EPV;

    // ---------------- the token's sources (one vector each) and the queries
    uint4 xv[NS];
    const unsigned char *g = a.src + (t * a.d + c0) * E::BYTES;
#pragma unroll
    for (int i = 0; i < NS; ++i)
        xv[i] = i < a.n_src ? ldg128_stream(g + (int64_t)i * a.src_stride_bytes) : make_uint4(0u, 0u, 0u, 0u);
    float2 wq[NQ][NP];
#pragma unroll
    for (int q = 0; q < NQ; ++q)
#pragma unroll
        for (int p = 0; p < NP; ++p) {
            float2 w = make_float2(0.f, 0.f);
            if (q < a.n_q) {
                w = make_float2(__ldg(a.queries + (size_t)q * a.d + c0 + 2 * p),
                                __ldg(a.queries + (size_t)q * a.d + c0 + 2 * p + 1));
                if (a.gain) { w.x *= __ldg(a.gain + c0 + 2 * p); w.y *= __ldg(a.gain + c0 + 2 * p + 1); }
            }
            wq[q][p] = w;
        }

    // ---------------- partial sums: [i] sum of squares, [NS + q*NS + i] dots
    float v[V];
#pragma unroll
    for (int i = 0; i < NS; ++i) {
        float2 x[NP];
        E::unpack(xv[i], x);
        float2 ss = make_float2(0.f, 0.f), dt[NQ];
#pragma unroll
        for (int q = 0; q < NQ; ++q) dt[q] = make_float2(0.f, 0.f);
#pragma unroll
        for (int p = 0; p < NP; ++p) {
            ss = ffma2(x[p], x[p], ss);
#pragma unroll
            for (int q = 0; q < NQ; ++q) dt[q] = ffma2(x[p], wq[q][p], dt[q]);
        }
        v[i] = ss.x + ss.y;
#pragma unroll
        for (int q = 0; q < NQ; ++q) v[NS + q * NS + i] = dt[q].x + dt[q].y;
    }
    butterfly_reduce<V>(v, lane);
#pragma unroll
    for (int j = 0; j < R; ++j) {
        const int idx = bfly_slot<V>(lane, j);
        if (idx >= 0) red[warp * V + idx] = v[j];
    }
    __syncthreads();
    // this CTA's totals, sent to every CTA of the cluster (itself included)
    for (int j = tid; j < V; j += blockDim.x) {
        float s = 0.f;
        for (int w = 0; w < nw; ++w) s += red[w * V + j];
        for (int r = 0; r < a.cs; ++r) {
            float *peer = cluster.map_shared_rank(xch, r);
            peer[rank * V + j] = s;
        }
    }
    cluster.sync();

    // ---------------- softmax per query over the sources: lane q*NS + i
    const int q = lane / NS, i = lane - q * NS;
    const bool pv = q < NQ && q < a.n_q && i < a.n_src;
    float ss = 0.f, dt = 0.f;
    if (q < NQ)
        for (int r = 0; r < a.cs; ++r) {
            ss += xch[r * V + i];
            dt += xch[r * V + NS + q * NS + i];
        }
    const float score = pv ? key_score(dt, ss, 1.f / (float)a.d, a.eps) : -INFINITY;
    const float mx = seg_max<NS>(score);
    const float e = pv ? __expf(score - mx) : 0.f;
    const float sum = seg_sum<NS>(e);
    const float alpha = pv ? e / sum : 0.f;
    if (rank == 0 && warp == 0 && pv && i == 0 && a.lse != nullptr) a.lse[(int64_t)q * a.T + t] = mx + __logf(sum);

    // ---------------- outputs: o_q = sum_i alpha_qi v_i on this thread's vector
#pragma unroll
    for (int qq = 0; qq < NQ; ++qq) {
        float2 y[NP];
#pragma unroll
        for (int p = 0; p < NP; ++p) y[p] = make_float2(0.f, 0.f);
#pragma unroll
        for (int ii = 0; ii < NS; ++ii) {
            const float al = __shfl_sync(0xffffffffu, alpha, qq * NS + ii);
            float2 x[NP];
            E::unpack(xv[ii], x);
#pragma unroll
            for (int p = 0; p < NP; ++p) y[p] = ffma2(make_float2(al, al), x[p], y[p]);
        }
        if (qq < a.n_q) stg128_cs(a.out + (int64_t)qq * a.out_q_stride_bytes + (t * a.d + c0) * E::BYTES, E::pack(y));
    }
}

}  // namespace attnres
