// msar_tile.cu -- fused MSAR read for sm_103a, one cluster exchange per tile
// of tokens.  Same computation as msar_kernel (msar.cu): per token, the m = 4
// streams of every source (identity and causal depthwise convolutions of
// sizes 4, 8, 12), one depth softmax per stream, then the H^pre mixer; no
// stream or stream read is written to global memory.
//
// Work split.  A cluster of K = d / 256 CTAs (16 at d = 4096) shares a range
// of tokens; CTA `rank` owns channels [256 rank, 256 rank + 256).  A thread
// owns two adjacent channels of two sources (lane = 8 * source pair + channel
// pair), so the eight lanes of a source pair hold sixteen channels and the
// four source pairs of one channel pair sit in one warp.
//
// Each thread keeps the last 12 rows of its two sources in registers (a
// window indexed by token mod 12, so the code is unrolled per tile phase):
// every source row is read from shared memory and widened to fp32 once, and
// each convolution output costs only its FMAs.  A thread fetches its own two
// 4-byte source pairs per token with cp.async into a thread-private ring of
// shared memory, two tiles ahead (per-thread copies: a 1-D bulk copy per
// source row and CTA issued too slowly for 512-byte rows).
//
// Per tile of TT = 4 tokens:
//   pass A  convolutions; per (source, stream) sum of squares and query dot,
//           reduced over the warp's channels by a butterfly, then over the
//           CTA's warps; the three conv streams are kept in shared memory
//           (thread-private slots) for pass B;
//   exchange  each CTA pushes its tile sums (and the previous tile's mixer
//           sums) into every peer's buffer with st.async, which completes
//           the peer's mbarrier; every CTA then holds all K partial sums and
//           adds them in rank order (the same order everywhere);
//   softmax per (token, stream) over the sources; the previous tile's mixer
//           weights and output rows;
//   pass B  Z^(r) = sum_i alpha_ri u_i^(r) from the kept streams (two sources
//           per thread, then the four source pairs by shuffles), kept in
//           registers until the next exchange brings the mixer sums.
// A split cluster barrier (arrive after reading the buffer, wait before the
// next push) keeps a push from overwriting sums a peer has not read; its
// latency hides behind pass B and the next pass A.
#include <cooperative_groups.h>

#include "msar.h"

namespace cg = cooperative_groups;

namespace attnres {

namespace {

constexpr int TCH = 256;                      // channels per CTA
constexpr int TTHREADS = 512;                 // 128 channel pairs x 4 source pairs
constexpr int TNW = TTHREADS / 32;            // warps
constexpr int TT = 4;                         // tokens per tile (one exchange per tile)
constexpr int TR = 12;                        // ring slots (tokens): the current tile and two ahead
constexpr int TW = 12;                        // window rows (largest kernel)
constexpr int NSC = 64;                       // score sums per token: 8 sources x 4 streams x (ss, dot)
constexpr int NMX = 8;                        // mixer sums per token (ssZ and 4 dots; 3 zero)
constexpr int NV4 = TT * (NSC + NMX) / 4;     // 16-byte values one CTA sends per tile
constexpr int WPITCH = 13 * 16;               // bytes of one channel pair's 12 tap pairs (+ pad)
constexpr int KMAXC = 16;                     // largest cluster

constexpr int OFF_RING = 0;                   // [TR][thread] 8 bytes: my two sources' channel pairs
constexpr int OFF_W = OFF_RING + TR * TTHREADS * 8;
constexpr int OFF_PM = OFF_W + 128 * WPITCH;
constexpr int OFF_U = OFF_PM + 4 * 2 * 128 * 16;
constexpr int OFF_TAB = OFF_U + TT * 3 * TTHREADS * 16;
constexpr int OFF_MTAB = OFF_TAB + TT * TNW * NSC * 4;
constexpr int OFF_RBUF = OFF_MTAB + TT * TNW * NMX * 4;
constexpr int OFF_ALPHA = OFF_RBUF + KMAXC * NV4 * 16;
constexpr int OFF_CMIX = OFF_ALPHA + TT * 32 * 4;
constexpr int OFF_BAR = OFF_CMIX + TT * 4 * 4;
constexpr int OFF_FLAG = OFF_BAR + 8;
constexpr int TSMEM = OFF_FLAG + 16;

template <int N> struct IC { static constexpr int value = N; };

__device__ __forceinline__ uint32_t mapa_u32(uint32_t a, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    return r;
}

// 16 bytes into a peer CTA's shared memory; completes 16 bytes of
// transaction count on the peer's mbarrier.
__device__ __forceinline__ void st_async_v4(uint32_t addr, float4 v, uint32_t bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                     addr),
                 "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(bar)
                 : "memory");
}

// Arrival without release semantics: what it orders is this thread's reads
// of the exchange buffer, whose values are already consumed when it arrives.
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cl(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// mbar_wait_bounded for a barrier completed by other CTAs' st.async.
__device__ __forceinline__ bool mbar_wait_cluster_bounded(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                                          const WaitCfg &cfg) {
    if (mbar_try_wait_cl(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (mbar_try_wait_cl(bar, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > cfg.timeout_ns) {
            atomicOr(cfg.status, DEV_ERR_TIMEOUT);
            *abort_flag = 1;
            return false;
        }
    }
}

// Plain shared-memory accesses at byte offsets of the dynamic shared array
// (no asm: the compiler schedules them around the arithmetic).
template <typename V> __device__ __forceinline__ V sld(const unsigned char *base, uint32_t off) {
    return *reinterpret_cast<const V *>(base + off);
}
template <typename V> __device__ __forceinline__ void sst(unsigned char *base, uint32_t off, V v) {
    *reinterpret_cast<V *>(base + off) = v;
}
// A 16-byte shared load the compiler keeps where it stands (volatile, but
// no memory clobber): used for the conv taps, which are the same for every
// token and would otherwise be hoisted into 48 live registers.
__device__ __forceinline__ float4 lds128_here(uint32_t a) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(a));
    return v;
}
__device__ __forceinline__ float2 f2add(float2 a, float2 b) { return make_float2(a.x + b.x, a.y + b.y); }
__device__ __forceinline__ float2 shfl2(float2 v, int off) {
    return make_float2(__shfl_xor_sync(0xffffffffu, v.x, off), __shfl_xor_sync(0xffffffffu, v.y, off));
}

// 4-byte asynchronous copy global -> shared (this thread's own slot); the
// copies of a tile form one group, waited for with cp.async.wait_group.
__device__ __forceinline__ void cp_async4(uint32_t dst, const void *src, uint64_t pol) {
    asm volatile("cp.async.ca.shared.global.L2::cache_hint [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "l"(pol)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N> __device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// conv stream (0..2) and first tap of tap pair tp (0..11): kernel sizes 4, 8, 12
__host__ __device__ constexpr int tp_stream(int tp) { return tp < 2 ? 0 : (tp < 6 ? 1 : 2); }
__host__ __device__ constexpr int tp_tap(int tp) { return tp < 2 ? 2 * tp : (tp < 6 ? 2 * (tp - 2) : 2 * (tp - 6)); }

}  // namespace

__global__ void __launch_bounds__(TTHREADS, 1) msar_tile_kernel(const MsarArgs a) {
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank();
    const int K = a.cluster;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int sp = lane >> 3;                       // source pair: sources 2sp, 2sp+1
    const int cp = warp * 8 + (lane & 7);           // channel pair inside the slice
    const int c0 = rank * TCH + 2 * cp;             // first of my two channels in the row
    const int d = a.d;
    const int nsrc = a.n_src;

    extern __shared__ __align__(128) unsigned char smem[];
    const uint32_t sbase = smem_u32(smem);
    uint64_t *rbar = reinterpret_cast<uint64_t *>(smem + OFF_BAR);   // the exchange's barrier
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + OFF_FLAG);

    // ---- set-up: conv taps, mixer projection (mixer gain folded), barrier
    {
        // packed kernels [d][4] [d][8] [d][12]: stream r starts at d * (0, 4, 12)
        for (int idx = tid; idx < 128 * 12; idx += TTHREADS) {
            const int p = idx / 12, tp = idx - p * 12;
            const int r = tp_stream(tp), j = tp_tap(tp);
            const int kr = 4 * (r + 1);
            const int64_t goff = r == 0 ? 0 : (r == 1 ? (int64_t)d * 4 : (int64_t)d * 12);
            const float *w0 = a.conv_w + goff + (int64_t)(rank * TCH + 2 * p) * kr;
            const float *w1 = w0 + kr;
            *reinterpret_cast<float4 *>(smem + OFF_W + p * WPITCH + tp * 16) =
                make_float4(__ldg(w0 + j), __ldg(w1 + j), __ldg(w0 + j + 1), __ldg(w1 + j + 1));
        }
        // pm[r][h][p] = (P'[r d + c][2h], P'[r d + c + 1][2h], P'[r d + c][2h+1], P'[r d + c + 1][2h+1])
        for (int idx = tid; idx < 4 * 2 * 128; idx += TTHREADS) {
            const int p = idx & 127, h = (idx >> 7) & 1, r = idx >> 8;
            const int64_t k0 = (int64_t)r * d + rank * TCH + 2 * p;
            const float g0 = a.mix_gain ? __ldg(a.mix_gain + k0) : 1.f;
            const float g1 = a.mix_gain ? __ldg(a.mix_gain + k0 + 1) : 1.f;
            *reinterpret_cast<float4 *>(smem + OFF_PM + idx * 16) =
                make_float4(__ldg(a.mix_w + k0 * 4 + 2 * h) * g0, __ldg(a.mix_w + (k0 + 1) * 4 + 2 * h) * g1,
                            __ldg(a.mix_w + k0 * 4 + 2 * h + 1) * g0, __ldg(a.mix_w + (k0 + 1) * 4 + 2 * h + 1) * g1);
        }
    }
    // stream queries of my channels, gain folded
    float2 wq[MSAR_M];
#pragma unroll
    for (int r = 0; r < MSAR_M; ++r) {
        wq[r] = make_float2(__ldg(a.queries + (size_t)r * d + c0), __ldg(a.queries + (size_t)r * d + c0 + 1));
        if (a.gain) { wq[r].x *= __ldg(a.gain + c0); wq[r].y *= __ldg(a.gain + c0 + 1); }
    }
    const uint32_t xfer = (uint32_t)(K * NV4 * 16);   // bytes every CTA receives per tile
    if (tid == 0) {
        mbar_init(rbar, 1);
        *abort_flag = 0;
        mbar_init_fence();
        mbar_arrive_expect_tx(rbar, xfer);               // tile 0's sums
    }
    fence_proxy_async_shared();
    cluster.sync();

    // ---- this cluster's tokens
    const int64_t cid = blockIdx.x / K;
    const int64_t tb = cid * a.tokens_per_cluster;
    const int64_t te = min(a.T, tb + a.tokens_per_cluster);
    const int ntok = te > tb ? (int)(te - tb) : 0;
    if (ntok == 0) return;                               // the whole cluster (cid is per cluster)
    const int nt = (ntok + TT - 1) / TT;
    const int64_t r0 = tb + a.t_prev;                    // source row of token tb
    const bool have0 = 2 * sp < nsrc, have1 = 2 * sp + 1 < nsrc;   // my two sources exist

    // my two sources' channel pair of source row `row`
    const unsigned char *src0 = a.src + (int64_t)(2 * sp) * a.src_stride_bytes + (int64_t)c0 * 2;
    const unsigned char *src1 = src0 + a.src_stride_bytes;
    const uint64_t pol = l2_policy_evict_first();
    const uint32_t ring_me = sbase + OFF_RING + tid * 8;
    // tile k's tokens into ring slots (token mod TR); one commit group per tile
    auto fetch_tile = [&](int k) {
        if (!a.wait.inject_stall) {
#pragma unroll
            for (int jt = 0; jt < TT; ++jt) {
                const int n = TT * k + jt;
                if (n < ntok) {
                    const int64_t off = (r0 + n) * (int64_t)d * 2;
                    const uint32_t dst = ring_me + (n % TR) * (TTHREADS * 8);
                    if (have0) cp_async4(dst, src0 + off, pol);
                    if (have1) cp_async4(dst + 4, src1 + off, pol);
                }
            }
        }
        cp_async_commit();
    };
    fetch_tile(0);
    fetch_tile(1);

    // ---- window: rows of tokens n - 11 .. n at slot (n mod 12); rows before
    // the sequence and absent sources are zero
    float2 win[2][TW];
#pragma unroll
    for (int j = 0; j < TW; ++j) { win[0][j] = make_float2(0.f, 0.f); win[1][j] = make_float2(0.f, 0.f); }
#pragma unroll
    for (int h = 1; h < TW; ++h) {                       // token n = h - 12, slot h
        const int64_t row = r0 + h - 12;
        if (row >= 0) {
            const int64_t off = row * (int64_t)d * 2;
            if (have0) win[0][h] = bf2_to_f2(__ldg(reinterpret_cast<const unsigned int *>(src0 + off)));
            if (have1) win[1][h] = bf2_to_f2(__ldg(reinterpret_cast<const unsigned int *>(src1 + off)));
        }
    }

    const uint32_t wbase = OFF_W + cp * WPITCH;
    const uint32_t tab_me = OFF_TAB + (warp * NSC + 2 * lane) * 4;
    const uint32_t u_me = OFF_U + tid * 16;
    const int mslot = bfly_slot<8>(lane, 0);             // mixer sum this lane ends with (or -1)
    float2 zk[TT];                                       // this tile's Z (my stream, my channels)
#pragma unroll
    for (int j = 0; j < TT; ++j) zk[j] = make_float2(0.f, 0.f);

    // ---- pass A of tile k: window phase PH = 4k mod 12
    auto pass_a = [&](auto phc, int k) {
        constexpr int PH = decltype(phc)::value;
        cp_async_wait<2>();                               // tile k's copies (k+1, k+2 may be pending)
#pragma unroll
        for (int jt = 0; jt < TT; ++jt) {
            const int n = TT * k + jt;
            const int ws = (PH + jt) % TW;
            win[0][ws] = make_float2(0.f, 0.f);
            win[1][ws] = make_float2(0.f, 0.f);
            if (n < ntok) {
                const uint2 v8 = sld<uint2>(smem, OFF_RING + (n % TR) * (TTHREADS * 8) + tid * 8);
                if (have0) win[0][ws] = bf2_to_f2(v8.x);
                if (have1) win[1][ws] = bf2_to_f2(v8.y);
            }
            // lag-major over the three streams, even and odd taps in separate
            // accumulators: up to twelve independent FMA chains per token
            float2 ue[2][3], uo[2][3];
#pragma unroll
            for (int r = 0; r < 3; ++r) {
                ue[0][r] = ue[1][r] = uo[0][r] = uo[1][r] = make_float2(0.f, 0.f);
            }
            float4 w4[3];
#pragma unroll
            for (int j = 0; j < TW; ++j) {
                const int sj = (ws - j + 2 * TW) % TW;
#pragma unroll
                for (int r = 0; r < 3; ++r) {
                    if (j >= 4 * (r + 1)) continue;                 // kernel sizes 4, 8, 12
                    // tap pair (r, j/2): index 0,1 | 2..5 | 6..11
                    if ((j & 1) == 0) w4[r] = lds128_here(sbase + wbase + ((r == 0 ? 0 : (r == 1 ? 2 : 6)) + j / 2) * 16);
                    const float2 w = (j & 1) ? make_float2(w4[r].z, w4[r].w) : make_float2(w4[r].x, w4[r].y);
                    if (j & 1) {
                        uo[0][r] = ffma2(w, win[0][sj], uo[0][r]);
                        uo[1][r] = ffma2(w, win[1][sj], uo[1][r]);
                    } else {
                        ue[0][r] = ffma2(w, win[0][sj], ue[0][r]);
                        ue[1][r] = ffma2(w, win[1][sj], ue[1][r]);
                    }
                }
            }
            float2 u[2][3];
#pragma unroll
            for (int r = 0; r < 3; ++r) {
                u[0][r] = f2add(ue[0][r], uo[0][r]);
                u[1][r] = f2add(ue[1][r], uo[1][r]);
            }
            float v[16];
#pragma unroll
            for (int ii = 0; ii < 2; ++ii) {
                const float2 xx = win[ii][ws];
                v[(ii * 4 + 0) * 2 + 0] = dot2(xx, xx);
                v[(ii * 4 + 0) * 2 + 1] = dot2(xx, wq[0]);
#pragma unroll
                for (int r = 1; r < 4; ++r) {
                    v[(ii * 4 + r) * 2 + 0] = dot2(u[ii][r - 1], u[ii][r - 1]);
                    v[(ii * 4 + r) * 2 + 1] = dot2(u[ii][r - 1], wq[r]);
                }
            }
            // sum over the eight lanes of my source pair: lane (sp, c) ends
            // with (ss, dot) of source 2 sp + c/4, stream c % 4
            bfly_step<16, 4>(v, lane);
            bfly_step<8, 2>(v, lane);
            bfly_step<4, 1>(v, lane);
            sst<float2>(smem, tab_me + jt * (TNW * NSC * 4), make_float2(v[0], v[1]));
            const uint32_t ua = u_me + jt * (3 * TTHREADS * 16);
            sst<float4>(smem, ua, make_float4(u[0][0].x, u[0][0].y, u[0][1].x, u[0][1].y));
            sst<float4>(smem, ua + TTHREADS * 16, make_float4(u[0][2].x, u[0][2].y, u[1][0].x, u[1][0].y));
            sst<float4>(smem, ua + 2 * TTHREADS * 16, make_float4(u[1][1].x, u[1][1].y, u[1][2].x, u[1][2].y));
        }
    };

    // ---- pass B of tile k: Z^(r) from the kept streams; the identity stream
    // is the window's row of each token (still there: no pass A in between)
    auto pass_b = [&](auto phc, int k) {
        constexpr int PH = decltype(phc)::value;
        const float4 pa = sld<float4>(smem, OFF_PM + ((sp * 2 + 0) * 128 + cp) * 16);
        const float4 pb = sld<float4>(smem, OFF_PM + ((sp * 2 + 1) * 128 + cp) * 16);
        const float2 pw[4] = {make_float2(pa.x, pa.y), make_float2(pa.z, pa.w), make_float2(pb.x, pb.y),
                              make_float2(pb.z, pb.w)};
        const bool hi16 = (lane & 16) != 0, hi8 = (lane & 8) != 0;
#pragma unroll
        for (int jt = 0; jt < TT; ++jt) {
            const int n = TT * k + jt;
            const int ws = (PH + jt) % TW;
            float2 zs = make_float2(0.f, 0.f);
            float mv[8];
#pragma unroll
            for (int o = 0; o < 8; ++o) mv[o] = 0.f;
            if (n < ntok) {
                const float2 x0 = win[0][ws], x1 = win[1][ws];
                const uint32_t ua = u_me + jt * (3 * TTHREADS * 16);
                const float4 u0 = sld<float4>(smem, ua), u1 = sld<float4>(smem, ua + TTHREADS * 16),
                             u2 = sld<float4>(smem, ua + 2 * TTHREADS * 16);
                const float4 a0 = sld<float4>(smem, OFF_ALPHA + (jt * 32 + (2 * sp) * 4) * 4);
                const float4 a1 = sld<float4>(smem, OFF_ALPHA + (jt * 32 + (2 * sp + 1) * 4) * 4);
                // streams of source 2sp: x0, (u0.x,u0.y), (u0.z,u0.w), (u1.x,u1.y)
                // streams of source 2sp+1: x1, (u1.z,u1.w), (u2.x,u2.y), (u2.z,u2.w)
                float2 z[4];
                z[0] = ffma2(make_float2(a1.x, a1.x), x1, fmul2(make_float2(a0.x, a0.x), x0));
                z[1] = ffma2(make_float2(a1.y, a1.y), make_float2(u1.z, u1.w),
                             fmul2(make_float2(a0.y, a0.y), make_float2(u0.x, u0.y)));
                z[2] = ffma2(make_float2(a1.z, a1.z), make_float2(u2.x, u2.y),
                             fmul2(make_float2(a0.z, a0.z), make_float2(u0.z, u0.w)));
                z[3] = ffma2(make_float2(a1.w, a1.w), make_float2(u2.z, u2.w),
                             fmul2(make_float2(a0.w, a0.w), make_float2(u1.x, u1.y)));
                // sum over the four source pairs; lane (sp, c) keeps stream sp
                const float2 y0 = f2add(hi16 ? z[2] : z[0], shfl2(hi16 ? z[0] : z[2], 16));
                const float2 y1 = f2add(hi16 ? z[3] : z[1], shfl2(hi16 ? z[1] : z[3], 16));
                zs = f2add(hi8 ? y1 : y0, shfl2(hi8 ? y0 : y1, 8));
                mv[0] = dot2(zs, zs);
#pragma unroll
                for (int o = 0; o < 4; ++o) mv[1 + o] = dot2(zs, pw[o]);
            }
            zk[jt] = zs;
            butterfly_reduce<8>(mv, lane);
            if (mslot >= 0)
                *reinterpret_cast<float *>(smem + OFF_MTAB + ((jt * TNW + warp) * NMX + mslot) * 4) = mv[0];
        }
    };

    const uint32_t rbuf_local = sbase + OFF_RBUF;
    const uint32_t rbar_local = smem_u32(rbar);
    for (int k = 0; k <= nt; ++k) {
        // tile k+2 into the slots tile k-1 left (this thread read them in its
        // own pass A of tile k-1)
        fetch_tile(k + 2);
        if (k < nt) {
            switch (k % 3) {
                case 0: pass_a(IC<0>{}, k); break;
                case 1: pass_a(IC<4>{}, k); break;
                default: pass_a(IC<8>{}, k); break;
            }
        }
        __syncthreads();                                 // tile sums and last tile's mixer sums complete
        // ---- sums over the CTA's warps (rank order of nothing else: warps 0..15)
        float4 tot = make_float4(0.f, 0.f, 0.f, 0.f);
        if (tid < NV4) {
            uint32_t at;
            int stride;
            bool live;
            if (tid < TT * NSC / 4) {
                const int jt = tid / (NSC / 4);
                at = OFF_TAB + (jt * TNW * NSC + (tid % (NSC / 4)) * 4) * 4;
                stride = NSC * 4;
                live = k < nt;
            } else {
                const int j = tid - TT * NSC / 4;
                const int jt = j / (NMX / 4);
                at = OFF_MTAB + (jt * TNW * NMX + (j % (NMX / 4)) * 4) * 4;
                stride = NMX * 4;
                live = k > 0;
            }
            if (live) {
#pragma unroll
                for (int w = 0; w < TNW; ++w) {
                    const float4 p = sld<float4>(smem, at + w * stride);
                    tot.x += p.x; tot.y += p.y; tot.z += p.z; tot.w += p.w;
                }
            }
        }
        if (k > 0) cluster_wait_acquire();               // every peer has read the previous tile's sums
        if (tid < NV4 && !a.wait.inject_stall) {
            const uint32_t dst = rbuf_local + (rank * NV4 + tid) * 16;
            for (int p = 0; p < K; ++p)
                st_async_v4(mapa_u32(dst, (uint32_t)p), tot, mapa_u32(rbar_local, (uint32_t)p));
        }

        // ---- all CTAs' sums: softmax of tile k, mixer weights of tile k-1
        if (tid < 160) {
            // after a timeout the barrier's phase stays open: a CTA that gave
            // up neither waits on it again (an earlier parity would pass at
            // once) nor re-arms it (its one arrival per phase is spent)
            const bool arrived =
                !*abort_flag && mbar_wait_cluster_bounded(rbar, (uint32_t)(k & 1), abort_flag, a.wait);
            if (tid < 128) {
                const int jt = tid >> 5, r = (tid >> 3) & 3, i = tid & 7;
                float ss = 0.f, dt = 0.f;
                const uint32_t at = OFF_RBUF + (jt * (NSC / 4) + 2 * i + (r >> 1)) * 16 + (r & 1) * 8;
                for (int p = 0; p < K; ++p) {
                    const float2 x = sld<float2>(smem, at + p * NV4 * 16);
                    ss += x.x;
                    dt += x.y;
                }
                const float score = i < nsrc ? key_score(dt, ss, 1.f / (float)d, a.eps) : -INFINITY;
                const float mx = seg_max<8>(score);
                const float e = i < nsrc ? __expf(score - mx) : 0.f;
                const float al = e / seg_sum<8>(e);
                if (k < nt) *reinterpret_cast<float *>(smem + OFF_ALPHA + ((jt * 8 + i) * 4 + r) * 4) = al;
            } else {
                const int l = tid - 128, jt = l >> 3, o = l & 7;
                float t = 0.f;
                if (o < 5) {
                    const uint32_t at = OFF_RBUF + (TT * NSC / 4) * 16 + (jt * NMX + o) * 4;
                    for (int p = 0; p < K; ++p)
                        t += sld<float>(smem, at + p * NV4 * 16);
                }
                const float ssz = __shfl_sync(0xffffffffu, t, lane & ~7);
                const float ms = fmaf(ssz, 1.f / (float)(MSAR_M * d), a.mix_eps);
                const float inv = ms > 0.f ? rsqrtf(ms) : 0.f;
                if (o >= 1 && o <= 4)
                    *reinterpret_cast<float *>(smem + OFF_CMIX + (jt * 4 + o - 1) * 4) =
                        1.f / (1.f + __expf(-t * inv));
            }
            // the next tile's sums
            if (tid == 0 && k < nt && arrived) mbar_arrive_expect_tx(rbar, xfer);
        }
        cluster_arrive_relaxed();                        // done reading this tile's sums
        __syncthreads();                                 // alpha and mixer weights visible

        // ---- output rows of tile k-1
        if (k > 0) {
#pragma unroll
            for (int jt = 0; jt < TT; ++jt) {
                const int n = TT * (k - 1) + jt;
                if (n < ntok) {
                    const float c = *reinterpret_cast<const float *>(smem + OFF_CMIX + (jt * 4 + sp) * 4);
                    float2 h = make_float2(c * zk[jt].x, c * zk[jt].y);
                    h = f2add(h, shfl2(h, 8));
                    h = f2add(h, shfl2(h, 16));
                    if (sp == (jt & 3) && !*abort_flag)
                        *reinterpret_cast<uint32_t *>(a.out + ((tb + n) * d + c0) * 2) = f2_to_bf2(h.x, h.y);
                }
            }
        }
        // ---- pass B of tile k
        if (k < nt) {
            switch (k % 3) {
                case 0: pass_b(IC<0>{}, k); break;
                case 1: pass_b(IC<4>{}, k); break;
                default: pass_b(IC<8>{}, k); break;
            }
        }
    }
    cluster_wait_acquire();                              // last arrive; no peer touches this CTA after

    cp_async_wait<0>();
}

bool msar_tile_applies(int dt, const MsarArgs &a) {
    if (dt != 1 || a.conv_src_stride != 0 || a.n_src < 1 || a.n_src > MSAR_SMAX) return false;
    if (a.k[0] != 4 || a.k[1] != 8 || a.k[2] != 12) return false;
    if (a.d % TCH != 0) return false;
    const int K = a.d / TCH;
    return K == 1 || K == 2 || K == 4 || K == 8 || K == 16;
}

attnres_status_t launch_msar_tile(MsarArgs a, int sms, void *stream, char *err, size_t errlen) {
    (void)sms;
    const int K = a.d / TCH;
    const void *fn = reinterpret_cast<const void *>(&msar_tile_kernel);
    int dev = 0, optin = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) {
        snprintf(err, errlen, "msar tile device query: %s", cudaGetErrorString(e));
        return ATTNRES_ERR_CUDA;
    }
    if (TSMEM > optin) return ATTNRES_ERR_UNSUPPORTED;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, TSMEM);
    if (e == cudaSuccess && K > 8) e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) {
        snprintf(err, errlen, "msar tile cudaFuncSetAttribute: %s", cudaGetErrorString(e));
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
    cfg.blockDim = dim3(TTHREADS);
    cfg.dynamicSmemBytes = TSMEM;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cfg.gridDim = dim3(K);
    int max_clusters = 0;
    e = cudaOccupancyMaxActiveClusters(&max_clusters, fn, &cfg);
    if (e != cudaSuccess) {
        snprintf(err, errlen, "msar tile cudaOccupancyMaxActiveClusters: %s", cudaGetErrorString(e));
        return ATTNRES_ERR_CUDA;
    }
    if (max_clusters < 1) return ATTNRES_ERR_UNSUPPORTED;
    // clusters: as many as are resident, each at least 8 tiles of tokens
    const int64_t min_tokens = 8 * TT;
    int64_t nclusters = (a.T + min_tokens - 1) / min_tokens;
    if (nclusters > max_clusters) nclusters = max_clusters;
    if (nclusters < 1) nclusters = 1;
    int64_t tpc = (a.T + nclusters - 1) / nclusters;
    tpc = (tpc + TT - 1) / TT * TT;
    if (tpc > ((int64_t)1 << 30)) return ATTNRES_ERR_UNSUPPORTED;   // token counts are int inside
    nclusters = (a.T + tpc - 1) / tpc;
    a.cluster = K;
    a.ch = TCH;
    a.tokens_per_cluster = tpc;
    a.nclusters = (int)nclusters;
    cfg.gridDim = dim3((unsigned)(nclusters * K));
    e = cudaLaunchKernelEx(&cfg, msar_tile_kernel, a);
    if (e != cudaSuccess) {
        snprintf(err, errlen, "msar tile launch: %s", cudaGetErrorString(e));
        return ATTNRES_ERR_CUDA;
    }
    return ATTNRES_OK;
}

}  // namespace attnres
