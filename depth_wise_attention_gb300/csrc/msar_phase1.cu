// msar_phase1.cu -- phase 1 of MSAR inside the two-phase Block schedule.
//
// Every cached source v_i is expanded once into its m = 4 streams (identity
// and three causal depthwise convolutions, as in msar.cu) and read by the
// queries of every layer s of the block: for each (s, r)
//     o_s^(r)   = sum_i softmax_i((w_s^(r) * g) . u_i^(r) / rms(u_i^(r))) u_i^(r)
//     lse_s^(r) = log sum_i exp(score)
// which is the state each layer's phase 2 (msar_kernel with a prior) merges
// its partial sum into.  No mixer here: the mixer needs the merged streams.
//
// Work split as msar.cu: a cluster of K CTAs shares a contiguous range of
// tokens, CTA `rank` owns channels [rank*ch, (rank+1)*ch), each thread two
// adjacent channels; source rows arrive through a shared-memory ring filled
// by bulk copies.  Per token the sums over channels -- per (source, stream)
// the sum of squares and one query dot per layer, 32 * (1 + NL) values -- are
// reduced by butterflies of 32 values each, summed over the CTA's warps and
// exchanged through distributed shared memory with one cluster barrier.
#include <cooperative_groups.h>

#include "msar.h"

namespace cg = cooperative_groups;

namespace attnres {

constexpr int MP1_LA = 4;                                // rows prefetched ahead
constexpr int MP1_PAIRS = MSAR_SMAX * MSAR_M;            // (source, stream) pairs: 32

template <int NL> struct MP1Sums {
    static constexpr int NX = MP1_PAIRS * (1 + NL);      // [chunk][source * 4 + stream]
};

// KA, KB, KC > 0 fix the kernel sizes at compile time; NL = most layers.
template <typename Tin, int KA, int KB, int KC, int NL>
__global__ void __launch_bounds__(256, 1) msar_phase1_kernel(const MsarP1Args a, const int ring, const int ktot) {
    using P2 = Pair2<Tin>;
    constexpr int ES = sizeof(Tin);
    constexpr int NX = MP1Sums<NL>::NX;
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank();
    const int K = a.cluster;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nwarps = blockDim.x >> 5;
    const int ch = a.ch;
    const int cl = 2 * tid;
    const int cg0 = rank * ch + cl;
    const int nsrc = a.n_src;
    const int nl = a.n_layers;
    const int d = a.d;
    const size_t row_bytes = (size_t)ch * ES;
    const size_t slot_bytes = row_bytes * MSAR_SMAX;
    constexpr bool FIXED = KA > 0;

    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char *ringbuf = smem;
    float *wconv = reinterpret_cast<float *>(smem + (size_t)ring * slot_bytes);
    float *red = wconv + (size_t)ktot * ch;                       // [nwarps][NX]
    float *cbuf = red + 8 * NX;                                   // [2][K][NX]
    uint64_t *bars = reinterpret_cast<uint64_t *>(cbuf + 2 * 8 * NX);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + 32);

    const int kk[3] = {FIXED ? KA : a.k[0], FIXED ? KB : a.k[1], FIXED ? KC : a.k[2]};
    int koff[3];
    koff[0] = 0;
    koff[1] = kk[0];
    koff[2] = kk[0] + kk[1];
    const int kmax = max(kk[0], max(kk[1], kk[2]));
    const int hist = kmax - 1;
    constexpr int HIST_C = FIXED ? (KA > KB ? (KA > KC ? KA : KC) : (KB > KC ? KB : KC)) - 1 : 0;

    for (size_t b = (size_t)tid * 16; b < (size_t)ring * slot_bytes; b += (size_t)blockDim.x * 16)
        *reinterpret_cast<uint4 *>(ringbuf + b) = make_uint4(0u, 0u, 0u, 0u);
    {
        int64_t goff[3];
        goff[0] = 0;
        goff[1] = (int64_t)d * kk[0];
        goff[2] = (int64_t)d * (kk[0] + kk[1]);
        for (int idx = tid; idx < ktot * ch; idx += blockDim.x) {
            const int jj = idx / ch, c = idx - jj * ch;
            const int r = jj >= koff[2] ? 2 : (jj >= koff[1] ? 1 : 0);
            const int j = jj - koff[r];
            wconv[idx] = __ldg(a.conv_w + goff[r] + (int64_t)(rank * ch + c) * kk[r] + j);
        }
    }
    if (tid == 0) {
        for (int s = 0; s < ring; ++s) mbar_init(&bars[s], 1);
        *abort_flag = 0;
        mbar_init_fence();
    }
    // stream queries of every layer, gain folded in
    float2 wq[NL][MSAR_M];
#pragma unroll
    for (int l = 0; l < NL; ++l)
#pragma unroll
        for (int r = 0; r < MSAR_M; ++r) {
            float2 w = make_float2(0.f, 0.f);
            if (l < nl) {
                const float *qp = a.queries + ((size_t)l * MSAR_M + r) * d + cg0;
                w = make_float2(__ldg(qp), __ldg(qp + 1));
                if (a.gain) { w.x *= __ldg(a.gain + cg0); w.y *= __ldg(a.gain + cg0 + 1); }
            }
            wq[l][r] = w;
        }
    fence_proxy_async_shared();
    cluster.sync();

    const int64_t cid = blockIdx.x / K;
    (void)HIST_C;
    const int64_t tb = cid * a.tokens_per_cluster;
    const int64_t te = min(a.T, tb + a.tokens_per_cluster);
    const int64_t ntok = te > tb ? te - tb : 0;
    const int64_t rho0 = tb - hist > 0 ? tb - hist : 0;

    const bool producer = (tid == 0) && !a.wait.inject_stall;
    uint64_t pol = 0;
    if (producer) pol = l2_policy_evict_first();
    int64_t next_row = rho0;
    int p_slot = 0;
    auto issue_row = [&](int64_t rho) {
        mbar_arrive_expect_tx(&bars[p_slot], (uint32_t)(row_bytes * nsrc));
        const unsigned char *g = a.src + (rho * d + (int64_t)rank * ch) * ES;
        unsigned char *dst = ringbuf + (size_t)p_slot * slot_bytes;
        for (int i = 0; i < nsrc; ++i)
            bulk_g2s(dst + (size_t)i * row_bytes, g + (int64_t)i * a.src_stride_bytes, (uint32_t)row_bytes,
                     &bars[p_slot], pol);
        if (++p_slot == ring) p_slot = 0;
    };
    const int64_t prolog_end = min(te, tb + 1 + MP1_LA);
    if (producer)
        for (; next_row < prolog_end; ++next_row) issue_row(next_row);

    int cur_slot = (int)(tb - rho0);
    uint32_t cur_par = 0;
    for (int64_t n = 0; n < ntok; ++n) {
        const int64_t t = tb + n;
        float2 x[MSAR_SMAX];
        float2 u[MSAR_SMAX][MSAR_M - 1];
        if (n == 0) {
            for (int sl = 0; sl <= cur_slot; ++sl) mbar_wait_bounded(&bars[sl], 0u, abort_flag, a.wait);
        } else {
            mbar_wait_bounded(&bars[cur_slot], cur_par, abort_flag, a.wait);
        }
#pragma unroll
        for (int i = 0; i < MSAR_SMAX; ++i) {
#pragma unroll
            for (int r = 0; r < MSAR_M - 1; ++r) u[i][r] = make_float2(0.f, 0.f);
        }
        // causal depthwise convolutions, each history row read once
        auto conv_row = [&](int j) {
            int sl = cur_slot - j;
            if (sl < 0) sl += ring;
            const unsigned char *row = ringbuf + (size_t)sl * slot_bytes + (size_t)cl * ES;
            float2 xs[MSAR_SMAX];
#pragma unroll
            for (int i = 0; i < MSAR_SMAX; ++i) xs[i] = P2::ld(row + (size_t)i * row_bytes);
            if (j == 0) {
#pragma unroll
                for (int i = 0; i < MSAR_SMAX; ++i) x[i] = xs[i];
            }
#pragma unroll
            for (int r = 0; r < MSAR_M - 1; ++r) {
                if (j < kk[r]) {
                    const float2 w = *reinterpret_cast<const float2 *>(wconv + (size_t)(koff[r] + j) * ch + cl);
#pragma unroll
                    for (int i = 0; i < MSAR_SMAX; ++i) u[i][r] = ffma2(w, xs[i], u[i][r]);
                }
            }
        };
        if (FIXED) {
#pragma unroll
            for (int j = 0; j <= HIST_C; ++j) conv_row(j);
        } else {
            for (int j = 0; j <= hist; ++j) conv_row(j);
        }
        if (++cur_slot == ring) { cur_slot = 0; cur_par ^= 1u; }

        // ---- per-token sums, in chunks of 32 values: chunk 0 the sums of
        // squares, chunk 1 + l the dots with layer l's stream queries
        float *rw = red + (size_t)warp * NX;
#pragma unroll
        for (int c = 0; c < 1 + NL; ++c) {
            if (c > nl) break;
            float v[MP1_PAIRS];
#pragma unroll
            for (int i = 0; i < MSAR_SMAX; ++i)
#pragma unroll
                for (int r = 0; r < MSAR_M; ++r) {
                    const float2 uu = r == 0 ? x[i] : u[i][r - 1];
                    v[i * MSAR_M + r] = c == 0 ? dot2(uu, uu) : dot2(uu, wq[c > 0 ? c - 1 : 0][r]);
                }
            butterfly_reduce<MP1_PAIRS>(v, lane);
            const int idx = bfly_slot<MP1_PAIRS>(lane, 0);
            if (idx >= 0) rw[c * MP1_PAIRS + idx] = v[0];
        }
        __syncthreads();
        // every thread has finished reading row t - hist: reuse its slot
        if (producer && next_row < te && !*abort_flag) issue_row(next_row++);
        const int par = (int)(n & 1);
        const int nval = MP1_PAIRS * (1 + nl);
        for (int j = tid; j < nval; j += blockDim.x) {
            float s = 0.f;
            for (int w = 0; w < nwarps; ++w) s += red[(size_t)w * NX + j];
            for (int q = 0; q < K; ++q) {
                float *peer = cluster.map_shared_rank(cbuf, q);
                peer[((size_t)par * K + rank) * NX + j] = s;
            }
        }
        cluster.sync();
        const float *cb = cbuf + (size_t)par * K * NX;

        // ---- per layer: per-stream softmax over the sources, o and lse
        const int r = lane >> 3, i = lane & 7;           // lane <-> (stream, source)
        float ss = 0.f;
        for (int q = 0; q < K; ++q) ss += cb[(size_t)q * NX + i * MSAR_M + r];
        const float ms = fmaf(ss, 1.f / (float)d, a.eps);
        const float rinv = ms > 0.f ? rsqrtf(ms) : 0.f;
#pragma unroll
        for (int l = 0; l < NL; ++l) {
            if (l >= nl) break;
            float dt = 0.f;
            for (int q = 0; q < K; ++q) dt += cb[(size_t)q * NX + (1 + l) * MP1_PAIRS + i * MSAR_M + r];
            const float score = i < nsrc ? dt * rinv : -INFINITY;
            const float mxs = seg_max<8>(score);
            const float e = i < nsrc ? __expf(score - mxs) : 0.f;
            const float esum = seg_sum<8>(e);
            const float alpha = e / esum;
            if (rank == 0 && i == 0 && !*abort_flag)
                a.lse[((int64_t)l * MSAR_M + r) * a.T + t] = mxs + __logf(esum);
            float2 z[MSAR_M];
#pragma unroll
            for (int rr = 0; rr < MSAR_M; ++rr) z[rr] = make_float2(0.f, 0.f);
#pragma unroll
            for (int ii = 0; ii < MSAR_SMAX; ++ii) {
#pragma unroll
                for (int rr = 0; rr < MSAR_M; ++rr) {
                    const float al = __shfl_sync(0xffffffffu, alpha, rr * 8 + ii);
                    const float2 uu = rr == 0 ? x[ii] : u[ii][rr - 1];
                    z[rr] = ffma2(make_float2(al, al), uu, z[rr]);
                }
            }
            if (!*abort_flag) {
#pragma unroll
                for (int rr = 0; rr < MSAR_M; ++rr)
                    P2::st(a.o + ((((int64_t)l * MSAR_M + rr) * a.T + t) * d + cg0) * ES, z[rr]);
            }
        }
    }

    // Drain (only matters after an abort): copies must land before exit.
    if (producer) {
        int never = 0;
        const int64_t lo = next_row - ring > rho0 ? next_row - ring : rho0;
        for (int64_t rho = lo; rho < next_row; ++rho)
            mbar_wait_bounded(&bars[(rho - rho0) % ring], (uint32_t)((rho - rho0) / ring) & 1u, &never, a.wait);
    }
}

template <typename Tin, int NL>
static const void *mp1_fn(bool k4812) {
    return k4812 ? reinterpret_cast<const void *>(&msar_phase1_kernel<Tin, 4, 8, 12, NL>)
                 : reinterpret_cast<const void *>(&msar_phase1_kernel<Tin, 0, 0, 0, NL>);
}

template <typename Tin>
static const void *mp1_pick(int nl, bool k4812) {
    if (nl <= 1) return mp1_fn<Tin, 1>(k4812);
    if (nl <= 2) return mp1_fn<Tin, 2>(k4812);
    return mp1_fn<Tin, 4>(k4812);
}

attnres_status_t launch_msar_phase1(int dt, MsarP1Args a, int sms, void *stream, char *err, size_t errlen) {
    const int es = dt == 1 ? 2 : 4;
    const int max_ch = dt == 1 ? 512 : 256;
    if (a.n_src < 1 || a.n_src > MSAR_SMAX || a.n_layers < 1 || a.n_layers > MSAR_P1_MAXL)
        return ATTNRES_ERR_UNSUPPORTED;
    int K = 0;
    for (int k = 1; k <= 8; k *= 2) {
        if (a.d % k) continue;
        const int ch = a.d / k;
        if (ch <= max_ch && ch % 64 == 0) { K = k; break; }
    }
    if (K == 0) return ATTNRES_ERR_UNSUPPORTED;
    const int ch = a.d / K;
    const int threads = ch / 2;
    const int kmax = a.k[0] > a.k[1] ? (a.k[0] > a.k[2] ? a.k[0] : a.k[2]) : (a.k[1] > a.k[2] ? a.k[1] : a.k[2]);
    const int ring = kmax + MP1_LA;
    const int ktot = a.k[0] + a.k[1] + a.k[2];
    const int nlc = a.n_layers <= 1 ? 1 : (a.n_layers <= 2 ? 2 : 4);
    const int nx = MP1_PAIRS * (1 + nlc);
    const size_t smem = (size_t)ring * MSAR_SMAX * ch * es + (size_t)ktot * ch * 4 + (size_t)(8 * nx + 2 * 8 * nx) * 4 +
                        32 * 8 + 16;
    const bool k4812 = a.k[0] == 4 && a.k[1] == 8 && a.k[2] == 12;
    const void *fn = dt == 1 ? mp1_pick<__nv_bfloat16>(a.n_layers, k4812) : mp1_pick<float>(a.n_layers, k4812);
    int dev = 0, optin = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) {
        snprintf(err, errlen, "msar phase 1 device query: %s", cudaGetErrorString(e));
        return ATTNRES_ERR_CUDA;
    }
    if (smem > (size_t)optin) return ATTNRES_ERR_UNSUPPORTED;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) {
        snprintf(err, errlen, "msar phase 1 cudaFuncSetAttribute: %s", cudaGetErrorString(e));
        return ATTNRES_ERR_CUDA;
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = K;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cfg.gridDim = dim3(K * (sms / K > 0 ? sms / K : 1));
    int max_clusters = 0;
    e = cudaOccupancyMaxActiveClusters(&max_clusters, fn, &cfg);
    if (e != cudaSuccess) {
        snprintf(err, errlen, "msar phase 1 cudaOccupancyMaxActiveClusters: %s", cudaGetErrorString(e));
        return ATTNRES_ERR_CUDA;
    }
    if (max_clusters < 1) return ATTNRES_ERR_UNSUPPORTED;
    const int64_t min_tokens = 16;
    int64_t nclusters = (a.T + min_tokens - 1) / min_tokens;
    if (nclusters > max_clusters) nclusters = max_clusters;
    a.cluster = K;
    a.ch = ch;
    a.tokens_per_cluster = (a.T + nclusters - 1) / nclusters;
    cfg.gridDim = dim3((unsigned)(nclusters * K));
    e = cudaLaunchKernelEx(&cfg, (void (*)(const MsarP1Args, int, int))fn, a, ring, ktot);
    if (e != cudaSuccess) {
        snprintf(err, errlen, "msar phase 1 launch: %s", cudaGetErrorString(e));
        return ATTNRES_ERR_CUDA;
    }
    return ATTNRES_OK;
}

}  // namespace attnres
