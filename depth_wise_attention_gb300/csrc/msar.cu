// msar.cu -- fused MSAR read for sm_103a: causal depthwise stream expansion,
// per-stream depth softmax and the H^pre mixer in one pass, with no
// intermediate tensor written to memory.
//
// Per token t and source v_i, stream 0 is v_i[t] itself and stream r >= 1 is
//     u_i^(r)[t][c] = sum_{j<k_r} cw_r[c][j] v_i[t-j][c]      (v[<0] = 0).
// Stream r reads the depth history with its own query:
//     Z^(r) = sum_i softmax_i((w_r * g) . u_i^(r) / rms(u_i^(r))) u_i^(r),
// and the mixer gives h = sum_r sigmoid(z . P[:, r]) Z^(r) with
// z = RMSNorm(Flatten(Z)) (stream-major, mixer gain folded into P).
//
// Work split.  A cluster of K CTAs (K <= 8) shares a contiguous range of
// tokens; CTA `rank` owns channels [rank*ch, (rank+1)*ch) and each thread owns
// two adjacent channels, so the conv weights of a CTA fit in shared memory
// and every per-channel quantity (conv outputs, Z) stays in registers.
// Source rows arrive through a ring of R = kmax + 4 token rows per source in
// shared memory, filled by thread 0 with 1-D bulk copies four rows ahead.
// The sums over channels (per stream and source: sum u^2 and the query dot;
// per token: sum Z^2 and the four projection dots) are reduced inside the CTA
// with a butterfly warp reduction, then across the cluster through
// distributed shared memory: each CTA writes its partial sums into every
// peer's buffer and one cluster barrier per token publishes them.  The mixer
// sums of token t travel with the score sums of token t+1, so each token
// costs one cluster barrier.
//
// Per-source kernels (PS): each source has its own conv kernels, packed
// conv_src_stride floats apart.  The 8 sources' kernels of a CTA's slice
// (393 KB at 512 channels) do not fit in shared memory, so each thread reads
// its two channels' taps of every source through L2 (the whole set, 3 MB at
// d = 4096, stays resident) as the convolution needs them.
#include <cooperative_groups.h>

#include "msar.h"

namespace cg = cooperative_groups;

namespace attnres {

constexpr int MSAR_LA = 4;                              // rows prefetched ahead
constexpr int MSAR_NS = MSAR_SMAX * MSAR_M * 2;         // score sums per token (64)
constexpr int MSAR_NX = MSAR_NS + 5;                    // + mixer sums (ssZ, 4 dots)

// KA, KB, KC > 0 fix the three kernel sizes at compile time (fully unrolled,
// branch-free convolution); 0 means they are read from the arguments.
template <typename Tin, int KA, int KB, int KC, bool PS = false>
__global__ void __launch_bounds__(256, 1) msar_kernel(const MsarArgs a, const int ring, const int ktot) {
    using P2 = Pair2<Tin>;
    constexpr int ES = sizeof(Tin);
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank();
    const int K = a.cluster;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nwarps = blockDim.x >> 5;
    const int ch = a.ch;
    const int cl = 2 * tid;                 // my first channel inside the slice
    const int cg0 = rank * ch + cl;         // ... and in the full row
    const int nsrc = a.n_src;
    const int d = a.d;
    const size_t row_bytes = (size_t)ch * ES;            // one source row of the slice
    // one ring slot holds MSAR_SMAX source rows; rows of absent sources (and
    // rows before the start of the sequence) stay zero
    const size_t slot_bytes = row_bytes * MSAR_SMAX;
    constexpr bool FIXED = KA > 0;

    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char *ringbuf = smem;
    float *wconv = reinterpret_cast<float *>(smem + (size_t)ring * slot_bytes);
    float *red = wconv + (size_t)ktot * ch;                       // [nwarps][MSAR_NX]
    float *cbuf = red + 8 * MSAR_NX;                              // [2][K][MSAR_NX]
    uint64_t *bars = reinterpret_cast<uint64_t *>(cbuf + 2 * 8 * MSAR_NX);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + 32);

    const int kk[3] = {FIXED ? KA : a.k[0], FIXED ? KB : a.k[1], FIXED ? KC : a.k[2]};
    int koff[3];
    koff[0] = 0;
    koff[1] = kk[0];
    koff[2] = kk[0] + kk[1];
    const int kmax = max(kk[0], max(kk[1], kk[2]));
    const int hist = kmax - 1;
    constexpr int HIST_C = FIXED ? (KA > KB ? (KA > KC ? KA : KC) : (KB > KC ? KB : KC)) - 1 : 0;

    // zero the whole ring once (absent sources, rows before token 0)
    for (size_t b = (size_t)tid * 16; b < (size_t)ring * slot_bytes; b += (size_t)blockDim.x * 16)
        *reinterpret_cast<uint4 *>(ringbuf + b) = make_uint4(0u, 0u, 0u, 0u);

    // conv weights of this CTA's channel slice, layout [koff_r + j][c]
    // (per-source kernels are read from global memory instead)
    int64_t goff[3];
    goff[0] = 0;
    goff[1] = (int64_t)d * kk[0];
    goff[2] = (int64_t)d * (kk[0] + kk[1]);
    if (!PS) {
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
    // stream queries (gain folded) and the mixer projection (mixer gain folded)
    float2 wq[MSAR_M];
    float2 pm[MSAR_M][4];
#pragma unroll
    for (int r = 0; r < MSAR_M; ++r) {
        wq[r] = make_float2(__ldg(a.queries + (size_t)r * d + cg0), __ldg(a.queries + (size_t)r * d + cg0 + 1));
        if (a.gain) { wq[r].x *= __ldg(a.gain + cg0); wq[r].y *= __ldg(a.gain + cg0 + 1); }
        const int64_t k0 = (int64_t)r * d + cg0;
        const float g0 = a.mix_gain ? __ldg(a.mix_gain + k0) : 1.f;
        const float g1 = a.mix_gain ? __ldg(a.mix_gain + k0 + 1) : 1.f;
#pragma unroll
        for (int o = 0; o < 4; ++o)
            pm[r][o] = make_float2(__ldg(a.mix_w + k0 * 4 + o) * g0, __ldg(a.mix_w + (k0 + 1) * 4 + o) * g1);
    }
    // generic-proxy zero fill must be ordered before the bulk copies into the ring
    fence_proxy_async_shared();
    // every CTA of the cluster is running (and its barriers initialised)
    // before any distributed-shared-memory access
    cluster.sync();

    const int64_t cid = blockIdx.x / K;
    (void)HIST_C;
    const int64_t tb = cid * a.tokens_per_cluster;
    const int64_t te = min(a.T, tb + a.tokens_per_cluster);
    const int64_t ntok = te > tb ? te - tb : 0;
    // source rows of this cluster's first and past-last output tokens (a
    // chunk of a longer sequence starts t_prev history rows into src)
    const int64_t rb = tb + a.t_prev, re = te + a.t_prev;
    const int64_t rho0 = rb - hist > 0 ? rb - hist : 0;   // first row this cluster loads

    const bool producer = (tid == 0) && !a.wait.inject_stall;
    uint64_t pol = 0;
    if (producer) pol = l2_policy_evict_first();
    int64_t next_row = rho0;                              // next row to load
    int p_slot = 0;                                       // its ring slot: (next_row - rho0) % ring
    auto issue_row = [&](int64_t rho) {
        mbar_arrive_expect_tx(&bars[p_slot], (uint32_t)(row_bytes * nsrc));
        const unsigned char *g = a.src + (rho * d + (int64_t)rank * ch) * ES;
        unsigned char *dst = ringbuf + (size_t)p_slot * slot_bytes;
        for (int i = 0; i < nsrc; ++i)
            bulk_g2s(dst + (size_t)i * row_bytes, g + (int64_t)i * a.src_stride_bytes, (uint32_t)row_bytes,
                     &bars[p_slot], pol);
        if (++p_slot == ring) p_slot = 0;
    };
    const int64_t prolog_end = min(re, rb + 1 + MSAR_LA);
    if (producer)
        for (; next_row < prolog_end; ++next_row) issue_row(next_row);

    float2 zprev[MSAR_M];
    float mixp[5];
#pragma unroll
    for (int r = 0; r < MSAR_M; ++r) zprev[r] = make_float2(0.f, 0.f);
#pragma unroll
    for (int o = 0; o < 5; ++o) mixp[o] = 0.f;

    // ring slot and mbarrier phase parity of the current token's row
    int cur_slot = (int)(rb - rho0);
    uint32_t cur_par = 0;
    for (int64_t n = 0; n <= ntok; ++n) {
        const int64_t t = tb + n;
        const bool is_tok = n < ntok;
        float2 x[MSAR_SMAX];
        float2 u[MSAR_SMAX][MSAR_M - 1];
        float v[MSAR_NS];
#pragma unroll
        for (int q = 0; q < MSAR_NS; ++q) v[q] = 0.f;
        if (is_tok) {
            if (n == 0) {
                // rows rho0..t occupy slots 0..t-rho0 for the first time
                for (int sl = 0; sl <= cur_slot; ++sl) mbar_wait_bounded(&bars[sl], 0u, abort_flag, a.wait);
            } else {
                mbar_wait_bounded(&bars[cur_slot], cur_par, abort_flag, a.wait);
            }
#pragma unroll
            for (int i = 0; i < MSAR_SMAX; ++i) {
#pragma unroll
                for (int r = 0; r < MSAR_M - 1; ++r) u[i][r] = make_float2(0.f, 0.f);
            }
            // causal depthwise convolutions: each history row t-j is read once
            // and applied to every stream whose kernel reaches back that far
            // (rows before token 0 and absent sources are zero in the ring)
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
            // Per-source kernels: source by source, the source's three
            // kernels on my two channels are loaded once per token (channels
            // cg0 and cg0 + 1 hold 2 k_r consecutive floats of the [d][k_r]
            // layout: 16-byte loads when k_r is a multiple of 4), then applied
            // to that source's rows of the window.
            auto conv_source = [&](int i) {
                const float *wb = a.conv_w + (int64_t)i * a.conv_src_stride;
                constexpr int KW = FIXED ? HIST_C + 1 : MSAR_KMAX;
                float2 w[MSAR_M - 1][KW];
#pragma unroll
                for (int r = 0; r < MSAR_M - 1; ++r) {
                    const float *wr = wb + goff[r] + (int64_t)cg0 * kk[r];
                    if (FIXED && (kk[r] % 4) == 0) {
#pragma unroll
                        for (int j4 = 0; j4 < KW; j4 += 4) {
                            if (j4 < kk[r]) {
                                const float4 w0 = __ldg(reinterpret_cast<const float4 *>(wr + j4));
                                const float4 w1 = __ldg(reinterpret_cast<const float4 *>(wr + kk[r] + j4));
                                w[r][j4 + 0] = make_float2(w0.x, w1.x);
                                w[r][j4 + 1] = make_float2(w0.y, w1.y);
                                w[r][j4 + 2] = make_float2(w0.z, w1.z);
                                w[r][j4 + 3] = make_float2(w0.w, w1.w);
                            }
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < KW; ++j)
                            w[r][j] = j < kk[r] ? make_float2(__ldg(wr + j), __ldg(wr + kk[r] + j)) : make_float2(0.f, 0.f);
                    }
                }
#pragma unroll
                for (int j = 0; j < KW; ++j) {
                    if (j > hist) break;
                    int sl = cur_slot - j;
                    if (sl < 0) sl += ring;
                    const float2 xs = P2::ld(ringbuf + (size_t)sl * slot_bytes + (size_t)cl * ES + (size_t)i * row_bytes);
                    if (j == 0) x[i] = xs;
#pragma unroll
                    for (int r = 0; r < MSAR_M - 1; ++r)
                        if (j < kk[r]) u[i][r] = ffma2(w[r][j], xs, u[i][r]);
                }
            };
            if (PS) {
#pragma unroll
                for (int i = 0; i < MSAR_SMAX; ++i) {
                    if (i < nsrc) conv_source(i);
                    else x[i] = make_float2(0.f, 0.f);
                }
            } else if (FIXED) {
#pragma unroll
                for (int j = 0; j <= HIST_C; ++j) conv_row(j);
            } else {
                for (int j = 0; j <= hist; ++j) conv_row(j);
            }
            // per (source, stream): sum of squares and the stream-query dot
#pragma unroll
            for (int i = 0; i < MSAR_SMAX; ++i) {
                v[(i * MSAR_M + 0) * 2 + 0] = dot2(x[i], x[i]);
                v[(i * MSAR_M + 0) * 2 + 1] = dot2(x[i], wq[0]);
#pragma unroll
                for (int r = 1; r < MSAR_M; ++r) {
                    v[(i * MSAR_M + r) * 2 + 0] = dot2(u[i][r - 1], u[i][r - 1]);
                    v[(i * MSAR_M + r) * 2 + 1] = dot2(u[i][r - 1], wq[r]);
                }
            }
            if (++cur_slot == ring) { cur_slot = 0; cur_par ^= 1u; }
        }
        // ---- reduce over the CTA: butterfly in each warp, then across warps
        butterfly_reduce<MSAR_NS>(v, lane);
        float mx[5];
#pragma unroll
        for (int o = 0; o < 5; ++o) mx[o] = seg_sum<32>(mixp[o]);
        {
            float *rw = red + (size_t)warp * MSAR_NX;
            rw[2 * lane] = v[0];
            rw[2 * lane + 1] = v[1];
            if (lane < 5) {
                const float mv = lane == 0 ? mx[0] : lane == 1 ? mx[1] : lane == 2 ? mx[2] : lane == 3 ? mx[3] : mx[4];
                rw[MSAR_NS + lane] = mv;
            }
        }
        __syncthreads();
        // every thread has finished reading row t - hist: reuse its slot
        if (producer && next_row < re && !*abort_flag) issue_row(next_row++);
        const int par = (int)(n & 1);
        for (int j = tid; j < MSAR_NX; j += blockDim.x) {
            float s = 0.f;
            for (int w = 0; w < nwarps; ++w) s += red[(size_t)w * MSAR_NX + j];
            for (int q = 0; q < K; ++q) {
                float *peer = cluster.map_shared_rank(cbuf, q);
                peer[((size_t)par * K + rank) * MSAR_NX + j] = s;
            }
        }
        cluster.sync();
        const float *cb = cbuf + (size_t)par * K * MSAR_NX;

        // ---- finish the previous token: mixer weights and output row
        if (n > 0) {
            float tot = 0.f;
            if (lane < 5)
                for (int q = 0; q < K; ++q) tot += cb[(size_t)q * MSAR_NX + MSAR_NS + lane];
            const float ssz = __shfl_sync(0xffffffffu, tot, 0);
            const float ms = fmaf(ssz, 1.f / (float)(MSAR_M * d), a.mix_eps);
            const float inv = ms > 0.f ? rsqrtf(ms) : 0.f;
            float2 h = make_float2(0.f, 0.f);
#pragma unroll
            for (int o = 0; o < MSAR_M; ++o) {
                const float logit = __shfl_sync(0xffffffffu, tot, 1 + o) * inv;
                const float cw = 1.f / (1.f + __expf(-logit));
                h.x = fmaf(cw, zprev[o].x, h.x);
                h.y = fmaf(cw, zprev[o].y, h.y);
            }
            if (!*abort_flag)
                P2::st(a.out + ((t - 1) * d + cg0) * ES, h);
        }
        if (!is_tok) break;

        // ---- this token: scores, per-stream softmax over sources, Z
        {
            const int r = lane >> 3, i = lane & 7;       // lane <-> (stream, source)
            float ss = 0.f, dt = 0.f;
            for (int q = 0; q < K; ++q) {
                ss += cb[(size_t)q * MSAR_NX + (i * MSAR_M + r) * 2 + 0];
                dt += cb[(size_t)q * MSAR_NX + (i * MSAR_M + r) * 2 + 1];
            }
            const float score = i < nsrc ? key_score(dt, ss, 1.f / (float)d, a.eps) : -INFINITY;
            const float mxs = seg_max<8>(score);
            const float e = i < nsrc ? __expf(score - mxs) : 0.f;
            const float alpha = e / seg_sum<8>(e);
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
            float sz = 0.f, dp[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int rr = 0; rr < MSAR_M; ++rr) {
                sz = fmaf(z[rr].x, z[rr].x, fmaf(z[rr].y, z[rr].y, sz));
#pragma unroll
                for (int o = 0; o < 4; ++o) dp[o] += dot2(z[rr], pm[rr][o]);
                zprev[rr] = z[rr];
            }
            mixp[0] = sz;
#pragma unroll
            for (int o = 0; o < 4; ++o) mixp[1 + o] = dp[o];
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

template <typename Tin, bool PS>
static const void *msar_fn(bool k4812) {
    return k4812 ? reinterpret_cast<const void *>(&msar_kernel<Tin, 4, 8, 12, PS>)
                 : reinterpret_cast<const void *>(&msar_kernel<Tin, 0, 0, 0, PS>);
}

attnres_status_t launch_msar(int dt, MsarArgs a, int sms, void *stream, char *err, size_t errlen) {
    const int es = dt == 1 ? 2 : 4;
    const int max_ch = dt == 1 ? 512 : 256;       // ring of 16+ rows x 8 sources fits
    if (a.n_src > MSAR_SMAX) return ATTNRES_ERR_UNSUPPORTED;
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
    const int ring = kmax + MSAR_LA;
    const int ktot = a.k[0] + a.k[1] + a.k[2];
    const bool ps = a.conv_src_stride != 0;
    // per-source kernels stay in global memory: no shared-memory copy
    const int ktot_smem = ps ? 0 : ktot;
    const size_t smem = (size_t)ring * MSAR_SMAX * ch * es + (size_t)ktot_smem * ch * 4 +
                        (size_t)(8 * MSAR_NX + 2 * 8 * MSAR_NX) * 4 + 32 * 8 + 16;
    const bool k4812 = a.k[0] == 4 && a.k[1] == 8 && a.k[2] == 12;
    const void *fn = dt == 1 ? (ps ? msar_fn<__nv_bfloat16, true>(k4812) : msar_fn<__nv_bfloat16, false>(k4812))
                             : (ps ? msar_fn<float, true>(k4812) : msar_fn<float, false>(k4812));
    int dev = 0, optin = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) {
        snprintf(err, errlen, "msar device query: %s", cudaGetErrorString(e));
        return ATTNRES_ERR_CUDA;
    }
    if (smem > (size_t)optin) return ATTNRES_ERR_UNSUPPORTED;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) {
        snprintf(err, errlen, "msar cudaFuncSetAttribute: %s", cudaGetErrorString(e));
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
        snprintf(err, errlen, "msar cudaOccupancyMaxActiveClusters: %s", cudaGetErrorString(e));
        return ATTNRES_ERR_CUDA;
    }
    if (max_clusters < 1) return ATTNRES_ERR_UNSUPPORTED;
    const int64_t min_tokens = 16;
    int64_t nclusters = (a.T + min_tokens - 1) / min_tokens;
    if (nclusters > max_clusters) nclusters = max_clusters;
    a.cluster = K;
    a.ch = ch;
    a.nclusters = (int)nclusters;
    a.tokens_per_cluster = (a.T + nclusters - 1) / nclusters;
    cfg.gridDim = dim3((unsigned)(nclusters * K));
    e = cudaLaunchKernelEx(&cfg, (void (*)(const MsarArgs, int, int))fn, a, ring, ktot_smem);
    if (e != cudaSuccess) {
        snprintf(err, errlen, "msar launch: %s", cudaGetErrorString(e));
        return ATTNRES_ERR_CUDA;
    }
    return ATTNRES_OK;
}

}  // namespace attnres
