// msar_bwd.cu -- kernels of the backward of the MSAR read (the streams and
// mixer kernels also serve the forward read with a workspace, msar_expand_fwd_ws).
//
// The backward runs as a chain of steps over tensors in the caller's
// workspace (attnres_api.cu, msar_expand_bwd):
//   1. msar_streams_kernel   the conv streams u_i^(r), r = 1..3, of every source
//   2. the depth read        Z^(r) = read of the sources u_i^(r) with query w_r
//                            (the forward read kernels, one call per stream)
//   3. msar_mix_stats_kernel per token and channel slice, the mixer's partial
//                            sums (sum zf^2, the 4 projection dots, the 4
//                            dh . Z^(r));
//      msar_mix_dz_kernel    from their totals the mixer's backward: dZ^(r),
//                            and per token e_t[o] = dl_t[o] / nu_t;
//      msar_mix_acc_kernel   A[k][o] = sum_t zf_t[k] e_t[o] in per-chunk
//                            partials, from which dmix_w = mg * A and
//                            dmix_gain = sum_o P[:, o] A[:, o]
//   4. the read backward     du_i^(r), dw_r and the gain's share per stream
//                            (read_bwd_kernel, one call per stream)
//   5. msar_conv_bwd_kernel  back through the causal convolutions:
//                            dv_i[t] = du_i^(0)[t] + sum_r sum_j cw_r[j] du_i^(r)[t + j],
//                            and per-CTA partials of dcw_r[j] = sum du_i^(r)[t] v_i[t - j]
//   6. msar_sum_kernel       the partials summed in a fixed order (deterministic)
// The streams and their gradients are stored in the source dtype.
//
// The two convolution kernels walk the tokens of a chunk one row at a time
// with register windows of the rows they need again; the rows reach shared
// memory in batches through asynchronous 16-byte copies issued several
// batches ahead, so that each SM keeps tens of KB of loads in flight.
#include <stdio.h>

#include "msar.h"
#include "msar_bwd.h"

namespace attnres {

// ---------------------------------------------------------------- helpers
// 16-byte asynchronous global -> shared copy; valid == false writes zeros and
// reads nothing (src must still be a mapped address).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N> __device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <typename Tin> __device__ __forceinline__ float ld1(const unsigned char *p);
template <> __device__ __forceinline__ float ld1<float>(const unsigned char *p) {
    return *reinterpret_cast<const float *>(p);
}
template <> __device__ __forceinline__ float ld1<__nv_bfloat16>(const unsigned char *p) {
    return __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(p));
}
template <typename Tin> __device__ __forceinline__ void st1(unsigned char *p, float v);
template <> __device__ __forceinline__ void st1<float>(unsigned char *p, float v) {
    *reinterpret_cast<float *>(p) = v;
}
template <> __device__ __forceinline__ void st1<__nv_bfloat16>(unsigned char *p, float v) {
    *reinterpret_cast<__nv_bfloat16 *>(p) = __float2bfloat16_rn(v);
}

// Compile-time kernel sizes: KA, KB, KC > 0 fix them (fully unrolled,
// branch-free taps); 0 reads them from the arguments with windows of
// MSAR_KMAX rows.
template <int KA, int KB, int KC> struct ConvShape {
    static constexpr bool FIXED = KA > 0;
    static constexpr int K0 = FIXED ? KA : MSAR_KMAX, K1 = FIXED ? KB : MSAR_KMAX, K2 = FIXED ? KC : MSAR_KMAX;
    static constexpr int KT = K0 + K1 + K2;
    static constexpr int KM = K0 > K1 ? (K0 > K2 ? K0 : K2) : (K1 > K2 ? K1 : K2);
    __host__ __device__ static constexpr int k(int r) { return r == 0 ? K0 : r == 1 ? K1 : K2; }
    __host__ __device__ static constexpr int off(int r) { return r == 0 ? 0 : r == 1 ? K0 : K0 + K1; }
};

// lcm(rb, km) / rb: stages after which a window of km slots, advanced one
// slot per step, is back at its first slot
__host__ __device__ constexpr int ring_group(int rb, int km) {
    int g = 1;
    while ((g * rb) % km != 0) ++g;
    return g;
}

// ---------------------------------------------------------------- step 1
// CTA = (slice of ST_CB channels, source i, chunk of tc_s tokens); a thread
// owns two adjacent channels with their three kernels in registers and a
// window of the source's last KM rows.  Rows t0 - (KM-1) .. t1-1 arrive in
// batches of ST_RB rows into a ring of ST_NS stages.
constexpr int ST_THREADS = 256;
constexpr int ST_CB = 2 * ST_THREADS;
constexpr int ST_RB = 8;
constexpr int ST_NS = 4;

template <typename Tin, int KA, int KB, int KC>
__global__ void __launch_bounds__(ST_THREADS) msar_streams_kernel(const MsarBwdArgs a) {
    using P2 = Pair2<Tin>;
    using CS = ConvShape<KA, KB, KC>;
    constexpr int ES = sizeof(Tin);
    constexpr int H = CS::KM - 1;
    constexpr int ROWB = ST_CB * ES;
    constexpr int CPR = ROWB / 16;
    constexpr int CPS = ST_RB * CPR;
    extern __shared__ __align__(16) unsigned char smem[];
    const int tid = threadIdx.x;
    const int cb = blockIdx.x * ST_CB;
    const int c = cb + 2 * tid;
    const int i = blockIdx.y;
    const int64_t t0 = (int64_t)blockIdx.z * a.tc_s;
    const int64_t t1 = t0 + a.tc_s < a.T ? t0 + a.tc_s : a.T;
    const int64_t nrows = t1 - t0 + H;
    const int nb = (int)((nrows + ST_RB - 1) / ST_RB);
    const unsigned char *v = a.src + (int64_t)i * a.src_stride_bytes;
    const uint32_t sbase = smem_u32(smem);
    const float *cw = a.conv_w + (int64_t)i * a.conv_src_stride;      // this source's kernels

    float2 w[CS::KT];
    {
        int64_t off = 0;
#pragma unroll
        for (int r = 0; r < 3; ++r) {
#pragma unroll
            for (int j = 0; j < CS::k(r); ++j)
                w[CS::off(r) + j] = (CS::FIXED || j < a.k[r])
                                        ? make_float2(__ldg(cw + off + (int64_t)c * a.k[r] + j),
                                                      __ldg(cw + off + (int64_t)(c + 1) * a.k[r] + j))
                                        : make_float2(0.f, 0.f);
            off += (int64_t)a.d * a.k[r];
        }
    }
    auto issue = [&](int b) {
        if (b < nb) {
            const uint32_t st = sbase + (uint32_t)((b % ST_NS) * ST_RB * ROWB);
            for (int q = tid; q < CPS; q += ST_THREADS) {
                const int rr = q / CPR, cc = q - rr * CPR;
                const int64_t row = t0 - H + (int64_t)b * ST_RB + rr;
                const bool ok = row >= -a.hist && row < t1;
                cp_async16(st + rr * ROWB + cc * 16, v + ((ok ? row : 0) * a.d + cb) * ES + cc * 16, ok);
            }
        }
        cp_async_commit();
    };
#pragma unroll
    for (int b = 0; b < ST_NS - 1; ++b) issue(b);

    // win is a ring: v[row - j] at step q (row = t0 - H + q) sits in slot
    // (q - j) % KM.  Steps are taken in groups of lcm(ST_RB, KM), so every slot
    // index is a compile-time constant (no window shifts).
    constexpr int G = ring_group(ST_RB, CS::KM);
    float2 win[CS::KM];
#pragma unroll
    for (int j = 0; j < CS::KM; ++j) win[j] = make_float2(0.f, 0.f);
    // output pointers of the three streams at token t0, one row apart per step
    const int64_t rowb = (int64_t)a.d * ES;
    unsigned char *up[3];
#pragma unroll
    for (int r = 0; r < 3; ++r) up[r] = a.u + (((int64_t)r * a.n_src + i) * a.T + t0) * rowb + (int64_t)c * ES;
    for (int b0 = 0; b0 < nb; b0 += G) {
#pragma unroll
        for (int gs = 0; gs < G; ++gs) {
            const int b = b0 + gs;
            if (b >= nb) break;
            cp_async_wait<ST_NS - 2>();
            __syncthreads();
            issue(b + ST_NS - 1);
            const unsigned char *stage = smem + (b % ST_NS) * ST_RB * ROWB + 2 * tid * ES;
#pragma unroll
            for (int rr = 0; rr < ST_RB; ++rr) {
                const int64_t row = t0 - H + (int64_t)b * ST_RB + rr;
                const int ph = (gs * ST_RB + rr) % CS::KM;      // q % KM
                win[ph] = P2::ld(stage + rr * ROWB);
                if (row >= t0 && row < t1) {
#pragma unroll
                    for (int r = 0; r < 3; ++r) {
                        // even and odd taps in two independent chains
                        float2 ae = make_float2(0.f, 0.f), ao = make_float2(0.f, 0.f);
#pragma unroll
                        for (int j = 0; j < CS::k(r); ++j)
                            if (CS::FIXED || j < a.k[r]) {
                                const float2 x = win[(ph - j + CS::KM) % CS::KM];
                                if (j & 1) ao = ffma2(w[CS::off(r) + j], x, ao);
                                else ae = ffma2(w[CS::off(r) + j], x, ae);
                            }
                        P2::st(up[r], make_float2(ae.x + ao.x, ae.y + ao.y));
                        up[r] += rowb;
                    }
                }
            }
        }
    }
    cp_async_wait<0>();
}

// ---------------------------------------------------------------- step 3
// Mixer backward, tiled by channel slices of MX_CS channels (of every stream)
// so that a CTA keeps its slice of g * P in shared memory and reuses it over
// a chunk of tokens.  A warp takes one token at a time; a lane owns 8
// adjacent channels per 256-channel step.  gP is stored transposed by the
// channel's position within its 8 ([r][c % 8][c / 8]) so that the lanes'
// reads of one position are consecutive.
constexpr int MX_CS = 1024;
constexpr int MX_THREADS = 256;
constexpr size_t MX_SMEM = (size_t)4 * MX_CS * sizeof(float4);

__device__ __forceinline__ int gp_index(int r, int c) { return r * MX_CS + (c & 7) * (MX_CS / 8) + (c >> 3); }

__device__ __forceinline__ void stage_gp(const MsarBwdArgs &a, float4 *gp, int c0) {
    for (int q = threadIdx.x; q < 4 * MX_CS; q += blockDim.x) {
        const int r = q / MX_CS, cc = q - r * MX_CS;
        const int64_t k = (int64_t)r * a.d + c0 + cc;
        float4 p = __ldg(reinterpret_cast<const float4 *>(a.mix_w) + k);
        const float g = a.mix_gain ? __ldg(a.mix_gain + k) : 1.f;
        p.x *= g; p.y *= g; p.z *= g; p.w *= g;
        gp[gp_index(r, cc)] = p;
    }
    __syncthreads();
}

// 8 channels of one row as floats
template <typename Tin> __device__ __forceinline__ void load8(const unsigned char *p, float (&x)[8]);
template <> __device__ __forceinline__ void load8<__nv_bfloat16>(const unsigned char *p, float (&x)[8]) {
    const uint4 u = *reinterpret_cast<const uint4 *>(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float2 f = bf2_to_f2(w[e]);
        x[2 * e] = f.x;
        x[2 * e + 1] = f.y;
    }
}
template <> __device__ __forceinline__ void load8<float>(const unsigned char *p, float (&x)[8]) {
    const float4 a = *reinterpret_cast<const float4 *>(p), b = *reinterpret_cast<const float4 *>(p + 16);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}
template <typename Tin> __device__ __forceinline__ void store8(unsigned char *p, const float (&x)[8]);
template <> __device__ __forceinline__ void store8<__nv_bfloat16>(unsigned char *p, const float (&x)[8]) {
    *reinterpret_cast<uint4 *>(p) =
        make_uint4(f2_to_bf2(x[0], x[1]), f2_to_bf2(x[2], x[3]), f2_to_bf2(x[4], x[5]), f2_to_bf2(x[6], x[7]));
}
template <> __device__ __forceinline__ void store8<float>(unsigned char *p, const float (&x)[8]) {
    *reinterpret_cast<float4 *>(p) = make_float4(x[0], x[1], x[2], x[3]);
    *reinterpret_cast<float4 *>(p + 16) = make_float4(x[4], x[5], x[6], x[7]);
}

// 8 channels of one row as loaded (one 16-byte load for bf16, two for fp32),
// widened later: lets a step's loads be issued before the step before it is
// computed and stored.
template <typename Tin> struct Raw8;
template <> struct Raw8<__nv_bfloat16> {
    uint4 u;
    __device__ __forceinline__ void load(const unsigned char *p) { u = *reinterpret_cast<const uint4 *>(p); }
    __device__ __forceinline__ void widen(float (&x)[8]) const {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = bf2_to_f2(w[e]);
            x[2 * e] = f.x;
            x[2 * e + 1] = f.y;
        }
    }
};
template <> struct Raw8<float> {
    float4 a, b;
    __device__ __forceinline__ void load(const unsigned char *p) {
        a = *reinterpret_cast<const float4 *>(p);
        b = *reinterpret_cast<const float4 *>(p + 16);
    }
    __device__ __forceinline__ void widen(float (&x)[8]) const {
        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
        x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
    }
};

// Per (token, slice): s[0] = sum zf^2, s[1+o] = sum g zf P[:, o], s[5+r] = dh . Z^(r)
// over the slice's channels -> mix_part[t][slice][9].
template <typename Tin>
__global__ void __launch_bounds__(MX_THREADS) msar_mix_stats_kernel(const MsarBwdArgs a) {
    constexpr int ES = sizeof(Tin);
    extern __shared__ __align__(16) float4 gp[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int sl = blockIdx.x, c0 = sl * MX_CS;
    stage_gp(a, gp, c0);
    const int64_t t0 = (int64_t)blockIdx.y * a.tc_m;
    const int64_t t1 = t0 + a.tc_m < a.T ? t0 + a.tc_m : a.T;
    for (int64_t t = t0 + warp; t < t1; t += MX_THREADS / 32) {
        float s[9];
#pragma unroll
        for (int q = 0; q < 9; ++q) s[q] = 0.f;
        // each 256-channel step's rows are loaded one step ahead (two steps in flight)
        Raw8<Tin> rdh[2], rz[2][4];
        auto fetch = [&](int it, int bf) {
            const int cl = it * 256 + lane * 8;
            if (a.dh) rdh[bf].load(a.dh + (t * a.d + c0 + cl) * ES);
#pragma unroll
            for (int r = 0; r < 4; ++r) rz[bf][r].load(a.z + (((int64_t)r * a.T + t) * a.d + c0 + cl) * ES);
        };
        fetch(0, 0);
#pragma unroll
        for (int it = 0; it < MX_CS / 256; ++it) {
            const int cl = it * 256 + lane * 8;
            if (it + 1 < MX_CS / 256) fetch(it + 1, (it + 1) & 1);
            float dh[8], z[4][8];
            if (a.dh) {
                rdh[it & 1].widen(dh);
            } else {                                    // the forward's mixer: no dh sums
#pragma unroll
                for (int e = 0; e < 8; ++e) dh[e] = 0.f;
            }
#pragma unroll
            for (int r = 0; r < 4; ++r) rz[it & 1][r].widen(z[r]);
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float4 p = gp[gp_index(r, cl + e)];
                    s[0] = fmaf(z[r][e], z[r][e], s[0]);
                    s[1] = fmaf(z[r][e], p.x, s[1]);
                    s[2] = fmaf(z[r][e], p.y, s[2]);
                    s[3] = fmaf(z[r][e], p.z, s[3]);
                    s[4] = fmaf(z[r][e], p.w, s[4]);
                    s[5 + r] = fmaf(dh[e], z[r][e], s[5 + r]);
                }
        }
#pragma unroll
        for (int q = 0; q < 9; ++q) s[q] = seg_sum<32>(s[q]);
        if (lane == 0) {
            float *dst = a.mix_part + (t * a.nsl + sl) * 9;
#pragma unroll
            for (int q = 0; q < 9; ++q) dst[q] = s[q];
        }
    }
}

// The forward's mixer sums, as msar_mix_stats_kernel without dh (s[5..8] = 0).
// A warp takes two tokens at a time: every g*P value read from shared memory
// (16 bytes per channel and stream, the kernel's largest traffic) serves both,
// and their eight rows per 256-channel step are in flight together (measured
// 0.27 ms faster per MSAR two-phase block through the chains; the backward's
// kernels, with dh and dZ, lost more to the extra registers than they gained).
template <typename Tin>
__global__ void __launch_bounds__(MX_THREADS) msar_fwd_mix_stats_kernel(const MsarBwdArgs a) {
    constexpr bool DH = false;
    constexpr int ES = sizeof(Tin);
    constexpr int NSTEP = MX_CS / 256;
    constexpr int TPW = 2;
    extern __shared__ __align__(16) float4 gp[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int sl = blockIdx.x, c0 = sl * MX_CS;
    stage_gp(a, gp, c0);
    const int64_t t0 = (int64_t)blockIdx.y * a.tc_m;
    const int64_t t1 = t0 + a.tc_m < a.T ? t0 + a.tc_m : a.T;
    for (int64_t tb = t0 + (int64_t)warp * TPW; tb < t1; tb += (MX_THREADS / 32) * TPW) {
        const int nt = t1 - tb < TPW ? (int)(t1 - tb) : TPW;
        float s[TPW][9];
#pragma unroll
        for (int u = 0; u < TPW; ++u)
#pragma unroll
            for (int q = 0; q < 9; ++q) s[u][q] = 0.f;
#pragma unroll
        for (int it = 0; it < NSTEP; ++it) {
            // (no later step's loads above this point: hoisting them spills)
            asm volatile("" ::: "memory");
            const int cl = it * 256 + lane * 8;
            Raw8<Tin> rdh[TPW], rz[TPW][4];
#pragma unroll
            for (int u = 0; u < TPW; ++u) {
                const int64_t t = tb + (u < nt ? u : 0);  // a missing second token rereads the first
                if (DH) rdh[u].load(a.dh + (t * a.d + c0 + cl) * ES);
#pragma unroll
                for (int r = 0; r < 4; ++r) rz[u][r].load(a.z + (((int64_t)r * a.T + t) * a.d + c0 + cl) * ES);
            }
            float dh[TPW][8];
            if (DH) {
#pragma unroll
                for (int u = 0; u < TPW; ++u) rdh[u].widen(dh[u]);
            }
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                float z[TPW][8];
#pragma unroll
                for (int u = 0; u < TPW; ++u) rz[u][r].widen(z[u]);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float4 p = gp[gp_index(r, cl + e)];
#pragma unroll
                    for (int u = 0; u < TPW; ++u) {
                        s[u][0] = fmaf(z[u][e], z[u][e], s[u][0]);
                        s[u][1] = fmaf(z[u][e], p.x, s[u][1]);
                        s[u][2] = fmaf(z[u][e], p.y, s[u][2]);
                        s[u][3] = fmaf(z[u][e], p.z, s[u][3]);
                        s[u][4] = fmaf(z[u][e], p.w, s[u][4]);
                        if (DH) s[u][5 + r] = fmaf(dh[u][e], z[u][e], s[u][5 + r]);
                    }
                }
            }
        }
#pragma unroll
        for (int u = 0; u < TPW; ++u)
#pragma unroll
            for (int q = 0; q < (DH ? 9 : 5); ++q) s[u][q] = seg_sum<32>(s[u][q]);
        if (lane == 0) {
#pragma unroll
            for (int u = 0; u < TPW; ++u) {
                if (u >= nt) break;
                float *dst = a.mix_part + ((tb + u) * a.nsl + sl) * 9;
#pragma unroll
                for (int q = 0; q < 9; ++q) dst[q] = s[u][q];
            }
        }
    }
}

// The forward's mixer output from the per-slice sums of token t (added in
// slice order): h = sum_r c_r Z^(r) with c_r = sigmoid(s_r / nu).  A warp per
// token, 8 channels per lane per 256-channel step.
template <typename Tin>
__global__ void __launch_bounds__(256) msar_mix_out_kernel(const MsarBwdArgs a, unsigned char *out) {
    constexpr int ES = sizeof(Tin);
    const int lane = threadIdx.x & 31;
    const int64_t t = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (t >= a.T) return;
    const float inv_md = 1.f / (4.f * (float)a.d);
    float tot[5];
#pragma unroll
    for (int q = 0; q < 5; ++q) tot[q] = 0.f;
    for (int k = 0; k < a.nsl; ++k)
#pragma unroll
        for (int q = 0; q < 5; ++q) tot[q] += __ldg(a.mix_part + (t * a.nsl + k) * 9 + q);
    const float ms = fmaf(tot[0], inv_md, a.mix_eps);
    const float inv = ms > 0.f ? rsqrtf(ms) : 0.f;
    float cr[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) cr[r] = 1.f / (1.f + __expf(-tot[1 + r] * inv));
    for (int c = lane * 8; c < a.d; c += 256) {
        float y[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) y[e] = 0.f;
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            float z[8];
            load8<Tin>(a.z + (((int64_t)r * a.T + t) * a.d + c) * ES, z);
#pragma unroll
            for (int e = 0; e < 8; ++e) y[e] = fmaf(cr[r], z[e], y[e]);
        }
        store8<Tin>(out + (t * a.d + c) * ES, y);
    }
}

// From the per-slice sums of token t (added in slice order): nu, c, dl, and
//   dZ^(r) = c_r dh + (sum_o dl_o gP[:, o]) / nu - zf (sum_o dl_o s_o) / (m d nu^3)
// (sum_k g_k dzn_k zf_k = sum_o dl_o sum_k g_k zf_k P[k][o] = sum_o dl_o s_o).
template <typename Tin>
__global__ void __launch_bounds__(MX_THREADS) msar_mix_dz_kernel(const MsarBwdArgs a) {
    constexpr int ES = sizeof(Tin);
    extern __shared__ __align__(16) float4 gp[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int sl = blockIdx.x, c0 = sl * MX_CS;
    const float inv_md = 1.f / (4.f * (float)a.d);
    stage_gp(a, gp, c0);
    const int64_t t0 = (int64_t)blockIdx.y * a.tc_m;
    const int64_t t1 = t0 + a.tc_m < a.T ? t0 + a.tc_m : a.T;
    for (int64_t t = t0 + warp; t < t1; t += MX_THREADS / 32) {
        float tot[9];
#pragma unroll
        for (int q = 0; q < 9; ++q) tot[q] = 0.f;
        for (int k = 0; k < a.nsl; ++k)
#pragma unroll
            for (int q = 0; q < 9; ++q) tot[q] += __ldg(a.mix_part + (t * a.nsl + k) * 9 + q);
        const float ms = fmaf(tot[0], inv_md, a.mix_eps);
        const float inv = ms > 0.f ? rsqrtf(ms) : 0.f;              // 1 / nu
        float cr[4], dl[4];
        float s2 = 0.f;
#pragma unroll
        for (int o = 0; o < 4; ++o) {
            cr[o] = 1.f / (1.f + __expf(-tot[1 + o] * inv));
            dl[o] = tot[5 + o] * cr[o] * (1.f - cr[o]);
            s2 = fmaf(dl[o], tot[1 + o], s2);
        }
        const float k3 = s2 * inv * inv * inv * inv_md;
        if (sl == 0 && lane == 0)
            *reinterpret_cast<float4 *>(a.mix_e + t * 4) = make_float4(dl[0] * inv, dl[1] * inv, dl[2] * inv, dl[3] * inv);
        // each 256-channel step's rows are loaded one step ahead (two steps in
        // flight; the loads of a step are issued before the stores of the one before)
        Raw8<Tin> rdh[2], rz[2][4];
        auto fetch = [&](int it, int bf) {
            const int cl = it * 256 + lane * 8;
            rdh[bf].load(a.dh + (t * a.d + c0 + cl) * ES);
#pragma unroll
            for (int r = 0; r < 4; ++r) rz[bf][r].load(a.z + (((int64_t)r * a.T + t) * a.d + c0 + cl) * ES);
        };
        fetch(0, 0);
#pragma unroll
        for (int it = 0; it < MX_CS / 256; ++it) {
            const int cl = it * 256 + lane * 8;
            if (it + 1 < MX_CS / 256) fetch(it + 1, (it + 1) & 1);
            float dh[8];
            rdh[it & 1].widen(dh);
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int64_t off = (((int64_t)r * a.T + t) * a.d + c0 + cl) * ES;
                float z[8], y[8];
                rz[it & 1][r].widen(z);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float4 p = gp[gp_index(r, cl + e)];
                    const float gdzn = dl[0] * p.x + dl[1] * p.y + dl[2] * p.z + dl[3] * p.w;
                    y[e] = cr[r] * dh[e] + gdzn * inv - z[e] * k3;
                }
                store8<Tin>(a.dz + off, y);
            }
        }
    }
}

// A[k][o] = sum_t zf_t[k] e_t[o] over a chunk of tokens: one thread per 8
// adjacent elements k of the flattened m d vector (one 16-byte load per
// token), eight tokens' loads at a time; per-chunk partials in mix_parts.
template <typename Tin>
__global__ void __launch_bounds__(256) msar_mix_acc_kernel(const MsarBwdArgs a) {
    constexpr int ES = sizeof(Tin);
    constexpr int U = 8;
    const int64_t md = 4 * (int64_t)a.d;
    const int64_t k8 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 8;   // elements k8 .. k8 + 7
    if (k8 >= md) return;
    const int r = (int)(k8 / a.d);
    const int64_t c = k8 - (int64_t)r * a.d;
    const int64_t t0 = (int64_t)blockIdx.y * a.tc;
    const int64_t t1 = t0 + a.tc < a.T ? t0 + a.tc : a.T;
    const int64_t rowb = (int64_t)a.d * ES;
    const unsigned char *zr = a.z + (int64_t)r * a.T * rowb + c * ES;
    float acc[8][4];
#pragma unroll
    for (int e = 0; e < 8; ++e)
#pragma unroll
        for (int o = 0; o < 4; ++o) acc[e][o] = 0.f;
    for (int64_t t = t0; t < t1; t += U) {
        Raw8<Tin> zraw[U];
        float4 ev[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const bool ok = t + u < t1;
            if (ok) {
                zraw[u].load(zr + (t + u) * rowb);
                ev[u] = __ldg(reinterpret_cast<const float4 *>(a.mix_e) + (t + u));
            } else {
                ev[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            float z[8];
            if (t + u < t1) zraw[u].widen(z);
            else {
#pragma unroll
                for (int e = 0; e < 8; ++e) z[e] = 0.f;
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                acc[e][0] = fmaf(z[e], ev[u].x, acc[e][0]);
                acc[e][1] = fmaf(z[e], ev[u].y, acc[e][1]);
                acc[e][2] = fmaf(z[e], ev[u].z, acc[e][2]);
                acc[e][3] = fmaf(z[e], ev[u].w, acc[e][3]);
            }
        }
    }
    float4 *wp = reinterpret_cast<float4 *>(a.mix_parts + (size_t)blockIdx.y * (size_t)(md * 4)) + k8;
#pragma unroll
    for (int e = 0; e < 8; ++e) wp[e] = make_float4(acc[e][0], acc[e][1], acc[e][2], acc[e][3]);
}

// dmix_w[k][o] = mg_k A[k][o];  dmix_gain[k] = sum_o P[k][o] A[k][o]
__global__ void __launch_bounds__(256) msar_mix_finish_kernel(const MsarBwdArgs a, const float *A) {
    const int64_t md = 4 * (int64_t)a.d;
    for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < md; k += (int64_t)gridDim.x * blockDim.x) {
        const float4 ak = *reinterpret_cast<const float4 *>(A + k * 4);
        const float4 pk = __ldg(reinterpret_cast<const float4 *>(a.mix_w + k * 4));
        const float g = a.mix_gain ? __ldg(a.mix_gain + k) : 1.f;
        float4 dw = make_float4(g * ak.x, g * ak.y, g * ak.z, g * ak.w);
        float dg = pk.x * ak.x + pk.y * ak.y + pk.z * ak.z + pk.w * ak.w;
        if (a.acc) {
            const float4 ow = *reinterpret_cast<const float4 *>(a.dmix_w + k * 4);
            dw = make_float4(ow.x + dw.x, ow.y + dw.y, ow.z + dw.z, ow.w + dw.w);
            if (a.dmix_gain) dg += a.dmix_gain[k];
        }
        *reinterpret_cast<float4 *>(a.dmix_w + k * 4) = dw;
        if (a.dmix_gain) a.dmix_gain[k] = dg;
    }
}

// ---------------------------------------------------------------- step 5
// CTA = (slice of CB_CH channels, source i, chunk [t0, t1) of tc tokens),
// walked downwards one token at a time from t1 - 1 + (KM-1): the first KM-1
// steps (t >= t1) only warm up the windows.  Warp-specialised, two adjacent
// channels per thread:
//   * the first CB_HALF threads scatter each new row of the conv streams'
//     gradients into a window of pending outputs, pend[j] = dv[t - j]:
//         pend[j] += cw_r[j] du^(r)[t]     (r = 1..3, j < k_r)
//     after which dv[t] = pend[0] + du^(0)[t] is complete (every
//     du^(r)[t + j] has arrived) and is written;
//   * the other CB_HALF threads keep a ring of the source's last KM rows
//     (v[t - j] at step s in slot (s + j) % KM) and the sums
//     dcw_r[j] += du^(r)[t] v[t - j] for the chunk's own tokens.
// Each step's five rows (du^(1..3)[t], du^(0)[t], v[t - (KM-1)]) arrive in
// batches of RB steps into a ring of CB_NS stages, copied by all threads.
// The kernel-gradient partials go to conv_parts[(chunk * n_src + i)][ktot][d]
// with tap (r, j) at row koff_r + j and the channels contiguous (coalesced);
// msar_conv_sum_kernel adds them up and packs them like conv_w.
constexpr int CB_CH = 256;
constexpr int CB_HALF = CB_CH / 2;
constexpr int CB_THREADS = 2 * CB_HALF;
constexpr int CB_NS = 4;
constexpr int CB_NROW = 5;
template <typename Tin> struct ConvBwdStage {
    static constexpr int RB = sizeof(Tin) == 2 ? 8 : 4;            // steps per stage
    static constexpr int ROWB = CB_CH * (int)sizeof(Tin);
    static constexpr int BYTES = RB * CB_NROW * ROWB;              // 20 KB either way
};

template <typename Tin, int KA, int KB, int KC>
__global__ void __launch_bounds__(CB_THREADS, KA > 0 ? 2 : 1) msar_conv_bwd_kernel(const MsarBwdArgs a) {
    using P2 = Pair2<Tin>;
    using CS = ConvShape<KA, KB, KC>;
    using SG = ConvBwdStage<Tin>;
    constexpr int ES = sizeof(Tin);
    constexpr int H = CS::KM - 1;
    constexpr int RB = SG::RB, ROWB = SG::ROWB;
    constexpr int CPR = ROWB / 16;
    extern __shared__ __align__(16) unsigned char smem[];
    const int tid = threadIdx.x;
    const int lt = tid & (CB_HALF - 1);
    const int cb = blockIdx.x * CB_CH;
    const int c = cb + 2 * lt;
    const int i = blockIdx.y;
    const int64_t t0 = (int64_t)blockIdx.z * a.tc;
    const int64_t t1 = t0 + a.tc < a.T ? t0 + a.tc : a.T;
    // step s is token t1 - 1 + H - s; the first chunk walks on through the
    // history rows (their dv gets this call's share, added in)
    const int64_t nsteps = t1 - t0 + H + (blockIdx.z == 0 ? a.hist : 0);
    const int nb = (int)((nsteps + RB - 1) / RB);
    const int64_t rowb = (int64_t)a.d * ES;
    const int64_t ttop = t1 - 1 + H;
    const unsigned char *v = a.src + (int64_t)i * a.src_stride_bytes;
    const uint32_t sbase = smem_u32(smem);
    auto has = [&](int r, int j) { return CS::FIXED || j < a.k[r]; };
    // stage layout [RB steps][5 rows][CB_CH channels]; rows outside the
    // sequence (or du^(0) beyond the chunk) are zero-filled.  A stage holds
    // RB x CPR = CB_THREADS (step, 16-byte chunk) pairs: each thread copies
    // the five rows of its pair.
    static_assert(RB * CPR == CB_THREADS, "one (step, chunk) pair per thread");
    const int my_sb = tid / CPR, my_cc = tid - my_sb * CPR;
    const int64_t coff = (int64_t)cb * ES + my_cc * 16;
    const unsigned char *du_i = a.du + (int64_t)i * a.T * rowb + coff;     // du^(0) of source i
    const int64_t sstride = (int64_t)a.n_src * a.T * rowb;                  // du^(r) -> du^(r+1)
    const unsigned char *v_c = v + coff;
    auto issue = [&](int b) {
        const int64_t s = (int64_t)b * RB + my_sb;
        const int64_t t = ttop - s;
        const bool live = b < nb && s < nsteps;
        const int64_t trow = t * rowb;
        const uint32_t dst = sbase + (uint32_t)((b % CB_NS) * SG::BYTES + my_sb * CB_NROW * ROWB + my_cc * 16);
        const bool okr = live && t >= 0 && t < a.T;
#pragma unroll
        for (int r = 0; r < 3; ++r)
            cp_async16(dst + r * ROWB, du_i + (r + 1) * sstride + (okr ? trow : 0), okr);
        const bool ok0 = live && t >= 0 && t < t1;
        cp_async16(dst + 3 * ROWB, du_i + (ok0 ? trow : 0), ok0);
        const bool okv = live && t - H >= -a.hist;
        cp_async16(dst + 4 * ROWB, v_c + (okv ? trow - H * rowb : 0), okv);
        cp_async_commit();
    };
#pragma unroll
    for (int b = 0; b < CB_NS - 1; ++b) issue(b);

    if (tid < CB_HALF) {
        // ---- dv: the kernels and the window of pending outputs
        const float *cw = a.conv_w + (int64_t)i * a.conv_src_stride;  // this source's kernels
        float2 w[CS::KT], pend[CS::KM];
        int64_t off = 0;
#pragma unroll
        for (int r = 0; r < 3; ++r) {
#pragma unroll
            for (int j = 0; j < CS::k(r); ++j)
                w[CS::off(r) + j] = has(r, j) ? make_float2(__ldg(cw + off + (int64_t)c * a.k[r] + j),
                                                            __ldg(cw + off + (int64_t)(c + 1) * a.k[r] + j))
                                              : make_float2(0.f, 0.f);
            off += (int64_t)a.d * a.k[r];
        }
#pragma unroll
        for (int j = 0; j < CS::KM; ++j) pend[j] = make_float2(0.f, 0.f);
        unsigned char *dp = a.dsrc + (int64_t)i * a.dsrc_stride_bytes + (t1 - 1) * rowb + (int64_t)c * ES;
        for (int b = 0; b < nb; ++b) {
            cp_async_wait<CB_NS - 2>();
            named_bar_sync(1, CB_THREADS);
            issue(b + CB_NS - 1);
            const unsigned char *stage = smem + (b % CB_NS) * SG::BYTES + 2 * lt * ES;
#pragma unroll
            for (int sb = 0; sb < RB; ++sb) {
                const int64_t s = (int64_t)b * RB + sb;
                if (s >= nsteps) break;
#pragma unroll
                for (int r = 0; r < 3; ++r) {
                    const float2 dn = P2::ld(stage + (sb * CB_NROW + r) * ROWB);      // du^(r)[t]
#pragma unroll
                    for (int j = 0; j < CS::k(r); ++j)
                        if (has(r, j)) pend[j] = ffma2(w[CS::off(r) + j], dn, pend[j]);
                }
                if (s >= H) {                                   // t < t1: dv[t] is complete
                    const float2 d0 = P2::ld(stage + (sb * CB_NROW + 3) * ROWB);      // du^(0)[t]
                    float2 dv = make_float2(d0.x + pend[0].x, d0.y + pend[0].y);
                    if (s >= nsteps - (blockIdx.z == 0 ? a.hist : 0) && blockIdx.z == 0) {
                        // a history row: add this call's share to what is there
                        const float2 old = P2::ld(dp);
                        dv = make_float2(old.x + dv.x, old.y + dv.y);
                    }
                    P2::st(dp, dv);
                    dp -= rowb;
                }
#pragma unroll
                for (int j = 0; j < CS::KM - 1; ++j) pend[j] = pend[j + 1];
                pend[CS::KM - 1] = make_float2(0.f, 0.f);
            }
        }
    } else {
        // ---- dcw: the window of the source's rows behind and the sums
        float2 g[CS::KT], vw[CS::KM];
#pragma unroll
        for (int j = 0; j < CS::KT; ++j) g[j] = make_float2(0.f, 0.f);
#pragma unroll
        for (int j = 0; j < CS::KM; ++j) vw[j] = make_float2(0.f, 0.f);
        // vw is a ring: v[t - j] at step s sits in slot (s + j) % KM.  Steps
        // are taken in groups of lcm(RB, KM), so every slot index is a
        // compile-time constant (no window shift; measured 0.3 ms faster per
        // MSAR backward at T = 32768 d = 4096, where the same ring for the
        // pending outputs of the other half gained nothing and both together
        // lost time, the larger loop body costing more than the shifts).
        constexpr int CB_G = ring_group(RB, CS::KM);
        for (int b0 = 0; b0 < nb; b0 += CB_G) {
#pragma unroll
            for (int gs = 0; gs < CB_G; ++gs) {
                const int b = b0 + gs;
                if (b >= nb) break;
                cp_async_wait<CB_NS - 2>();
                named_bar_sync(1, CB_THREADS);
                issue(b + CB_NS - 1);
                const unsigned char *stage = smem + (b % CB_NS) * SG::BYTES + 2 * lt * ES;
#pragma unroll
                for (int sb = 0; sb < RB; ++sb) {
                    const int64_t s = (int64_t)b * RB + sb;
                    if (s >= nsteps) break;
                    const int ph = (gs * RB + sb) % CS::KM;     // s % KM
                    // the newest row is v[t - H]
                    vw[(ph + H) % CS::KM] = P2::ld(stage + (sb * CB_NROW + 4) * ROWB);
                    if (s >= H && ttop - s >= 0) {
#pragma unroll
                        for (int r = 0; r < 3; ++r) {
                            const float2 dn = P2::ld(stage + (sb * CB_NROW + r) * ROWB);  // du^(r)[t]
#pragma unroll
                            for (int j = 0; j < CS::k(r); ++j)
                                if (has(r, j)) g[CS::off(r) + j] = ffma2(dn, vw[(ph + j) % CS::KM], g[CS::off(r) + j]);
                        }
                    }
                }
            }
        }
        float *gp = a.conv_parts + ((size_t)blockIdx.z * a.n_src + i) * (size_t)a.ktot * a.d + c;
        int koff = 0;
#pragma unroll
        for (int r = 0; r < 3; ++r) {
#pragma unroll
            for (int j = 0; j < CS::k(r); ++j)
                if (has(r, j)) *reinterpret_cast<float2 *>(gp + (int64_t)(koff + j) * a.d) = g[CS::off(r) + j];
            koff += a.k[r];
        }
    }
    cp_async_wait<0>();
}

// dconv_w from the conv partials (pstride floats apart): element
// e = (koff_r + j) * d + c of every partial, summed over the partials in
// order, lands at koff_r * d + c * k_r + j (conv_w's packing).
__global__ void __launch_bounds__(256) msar_conv_sum_kernel(const float *parts, int64_t nparts, int64_t pstride, int d,
                                                            int k0, int k1, int k2, float *out, int accumulate) {
    const int ktot = k0 + k1 + k2;
    const int64_t n = (int64_t)ktot * d;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += (int64_t)gridDim.x * blockDim.x) {
        float s = 0.f;
        for (int64_t p = 0; p < nparts; ++p) s += parts[p * pstride + e];
        const int jg = (int)(e / d), c = (int)(e - (int64_t)jg * d);
        const int kr = jg < k0 ? k0 : jg < k0 + k1 ? k1 : k2;
        const int koff = jg < k0 ? 0 : jg < k0 + k1 ? k0 : k0 + k1;
        float *o = out + (int64_t)koff * d + (int64_t)c * kr + (jg - koff);
        *o = accumulate ? *o + s : s;
    }
}

// ---------------------------------------------------------------- step 6
// out[e] = (accumulate ? out[e] : 0) + sum_p parts[p * n + e], p in order.
__global__ void __launch_bounds__(256) msar_sum_kernel(const float *parts, int64_t nparts, int64_t n, float *out,
                                                       int accumulate) {
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += (int64_t)gridDim.x * blockDim.x) {
        float s = accumulate ? out[e] : 0.f;
        for (int64_t p = 0; p < nparts; ++p) s += parts[p * n + e];
        out[e] = s;
    }
}

// ---------------------------------------------------------------- launchers
static bool k4812(const MsarBwdArgs &a) { return a.k[0] == 4 && a.k[1] == 8 && a.k[2] == 12; }

template <typename F> static cudaError_t set_smem(F fn, size_t bytes) {
    return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

template <typename Tin, int KA, int KB, int KC>
static cudaError_t launch_streams_k(const MsarBwdArgs &a, cudaStream_t s) {
    auto fn = msar_streams_kernel<Tin, KA, KB, KC>;
    const size_t smem = (size_t)ST_NS * ST_RB * ST_CB * sizeof(Tin);
    cudaError_t e = set_smem(fn, smem);
    if (e != cudaSuccess) return e;
    const dim3 grid((unsigned)(a.d / ST_CB), (unsigned)a.n_src, (unsigned)((a.T + a.tc_s - 1) / a.tc_s));
    fn<<<grid, ST_THREADS, smem, s>>>(a);
    return cudaGetLastError();
}

template <typename Tin, int KA, int KB, int KC>
static cudaError_t launch_conv_bwd_k(const MsarBwdArgs &a, cudaStream_t s) {
    auto fn = msar_conv_bwd_kernel<Tin, KA, KB, KC>;
    const size_t smem = (size_t)CB_NS * ConvBwdStage<Tin>::BYTES;
    cudaError_t e = set_smem(fn, smem);
    if (e != cudaSuccess) return e;
    const dim3 grid((unsigned)(a.d / CB_CH), (unsigned)a.n_src, (unsigned)((a.T + a.tc - 1) / a.tc));
    fn<<<grid, CB_THREADS, smem, s>>>(a);
    return cudaGetLastError();
}

template <typename Tin>
static cudaError_t launch_mix_t(const MsarBwdArgs &a, cudaStream_t s) {
    const dim3 grid((unsigned)a.nsl, (unsigned)((a.T + a.tc_m - 1) / a.tc_m));
    cudaError_t e = set_smem(msar_mix_stats_kernel<Tin>, MX_SMEM);
    if (e == cudaSuccess) e = set_smem(msar_mix_dz_kernel<Tin>, MX_SMEM);
    if (e != cudaSuccess) return e;
    msar_mix_stats_kernel<Tin><<<grid, MX_THREADS, MX_SMEM, s>>>(a);
    msar_mix_dz_kernel<Tin><<<grid, MX_THREADS, MX_SMEM, s>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const dim3 agrid((unsigned)((4 * (int64_t)a.d / 8 + 255) / 256), (unsigned)((a.T + a.tc - 1) / a.tc));
    msar_mix_acc_kernel<Tin><<<agrid, 256, 0, s>>>(a);
    return cudaGetLastError();
}

template <typename Tin>
static cudaError_t launch_fwd_mix_t(const MsarBwdArgs &a, unsigned char *out, cudaStream_t s) {
    const dim3 grid((unsigned)a.nsl, (unsigned)((a.T + a.tc_m - 1) / a.tc_m));
    cudaError_t e = set_smem(msar_fwd_mix_stats_kernel<Tin>, MX_SMEM);
    if (e != cudaSuccess) return e;
    msar_fwd_mix_stats_kernel<Tin><<<grid, MX_THREADS, MX_SMEM, s>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    msar_mix_out_kernel<Tin><<<(unsigned)((a.T + 7) / 8), 256, 0, s>>>(a, out);
    return cudaGetLastError();
}

cudaError_t msar_fwd_mix(int dt, const MsarBwdArgs &a, void *out, void *stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (a.d % MX_CS != 0 || a.nsl != a.d / MX_CS || a.dh != nullptr) return cudaErrorInvalidValue;
    unsigned char *o = static_cast<unsigned char *>(out);
    return dt == 1 ? launch_fwd_mix_t<__nv_bfloat16>(a, o, s) : launch_fwd_mix_t<float>(a, o, s);
}

cudaError_t msar_bwd_streams(int dt, const MsarBwdArgs &a, void *stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (a.d % ST_CB != 0) return cudaErrorInvalidValue;
    if (dt == 1)
        return k4812(a) ? launch_streams_k<__nv_bfloat16, 4, 8, 12>(a, s) : launch_streams_k<__nv_bfloat16, 0, 0, 0>(a, s);
    return k4812(a) ? launch_streams_k<float, 4, 8, 12>(a, s) : launch_streams_k<float, 0, 0, 0>(a, s);
}

cudaError_t msar_bwd_mix(int dt, const MsarBwdArgs &a, void *stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (a.d % MX_CS != 0 || a.nsl != a.d / MX_CS) return cudaErrorInvalidValue;
    return dt == 1 ? launch_mix_t<__nv_bfloat16>(a, s) : launch_mix_t<float>(a, s);
}

cudaError_t msar_bwd_conv(int dt, const MsarBwdArgs &a, void *stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (a.d % CB_CH != 0) return cudaErrorInvalidValue;
    if (dt == 1)
        return k4812(a) ? launch_conv_bwd_k<__nv_bfloat16, 4, 8, 12>(a, s) : launch_conv_bwd_k<__nv_bfloat16, 0, 0, 0>(a, s);
    return k4812(a) ? launch_conv_bwd_k<float, 4, 8, 12>(a, s) : launch_conv_bwd_k<float, 0, 0, 0>(a, s);
}

cudaError_t msar_bwd_conv_sum(const MsarBwdArgs &a, const float *parts, int64_t nparts, int64_t part_stride,
                              float *dconv_w, void *stream) {
    const int64_t n = (int64_t)a.ktot * a.d;
    const int64_t blocks = (n + 255) / 256;
    msar_conv_sum_kernel<<<(unsigned)(blocks < 4096 ? blocks : 4096), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        parts, nparts, part_stride, a.d, a.k[0], a.k[1], a.k[2], dconv_w, a.acc);
    return cudaGetLastError();
}

cudaError_t msar_bwd_mix_finish(const MsarBwdArgs &a, const float *A, void *stream) {
    const int64_t n = 4 * (int64_t)a.d;
    msar_mix_finish_kernel<<<(unsigned)((n + 255) / 256), 256, 0, static_cast<cudaStream_t>(stream)>>>(a, A);
    return cudaGetLastError();
}

cudaError_t msar_bwd_sum(const float *parts, int64_t nparts, int64_t n, float *out, int accumulate, void *stream) {
    const int64_t blocks = (n + 255) / 256;
    msar_sum_kernel<<<(unsigned)(blocks < 4096 ? blocks : 4096), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        parts, nparts, n, out, accumulate);
    return cudaGetLastError();
}

}  // namespace attnres
