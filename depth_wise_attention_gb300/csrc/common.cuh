// common.cuh -- device helpers shared by the libattnres kernels (sm_103a):
// mbarrier / bulk-copy wrappers written as inline PTX, bounded waits,
// bf16 <-> f32 packing and packed f32x2 FMA.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace attnres {

// Bits of the device status word.
enum : int { DEV_ERR_TIMEOUT = 1 };

// Parameters of every bounded device-side wait.
struct WaitCfg {
    int *status;            // device status word (bit DEV_ERR_TIMEOUT)
    uint64_t timeout_ns;    // limit of one wait
    int inject_stall;       // nonzero: producers issue no copies (test hook)
};

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}
// Makes barrier initialisation visible to the async (bulk-copy) proxy and to
// the other threads of the CTA (follow with a CTA barrier).
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for phase `parity` of `bar` to complete.  Gives up when `abort_flag`
// (CTA shared memory) becomes nonzero or after cfg.timeout_ns; on a timeout
// it records DEV_ERR_TIMEOUT in the device status word and raises the CTA's
// abort flag so that every other waiter of the CTA stops waiting too.
// Returns true if the phase completed.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  volatile int *abort_flag, const WaitCfg &cfg) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > cfg.timeout_ns) {
            atomicOr(cfg.status, DEV_ERR_TIMEOUT);
            *abort_flag = 1;
            return false;
        }
    }
}

// ------------------------------------------------------------ bulk copies
// 1-D bulk copy global -> shared (no tensor map); completes `bytes` of
// transaction count on `bar`.  dst, src 16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_g2s(void *dst_smem, const void *src_gmem, uint32_t bytes,
                                         uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst_smem)),
        "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy (bulk copy) accesses of the same memory.
__device__ __forceinline__ void fence_proxy_async_shared() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------ named barrier
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------- packed math
// d = a * b + c on two f32 lanes at once (sm_100+ packed FMA).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;"
        : "=l"(d)
        : "l"(*reinterpret_cast<const uint64_t *>(&a)),
          "l"(*reinterpret_cast<const uint64_t *>(&b)),
          "l"(*reinterpret_cast<const uint64_t *>(&c)));
    return *reinterpret_cast<float2 *>(&d);
}

// d = a * b on two f32 lanes at once.
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;"
        : "=l"(d)
        : "l"(*reinterpret_cast<const uint64_t *>(&a)), "l"(*reinterpret_cast<const uint64_t *>(&b)));
    return *reinterpret_cast<float2 *>(&d);
}

// bf16x2 (one 32-bit word, low half = lower channel) -> two exact floats.
__device__ __forceinline__ float2 bf2_to_f2(uint32_t u) {
    return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
}

// two floats -> bf16x2, round to nearest even.
__device__ __forceinline__ uint32_t f2_to_bf2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

// Storage-type traits: one 16-byte vector = EPV elements = EPV/2 float2 pairs.
template <typename T> struct Elem;
template <> struct Elem<__nv_bfloat16> {
    static constexpr int EPV = 8;
    static constexpr int BYTES = 2;
    // 16-byte vector -> 4 float2 pairs
    __device__ static __forceinline__ void unpack(const uint4 &v, float2 (&x)[4]) {
        x[0] = bf2_to_f2(v.x); x[1] = bf2_to_f2(v.y); x[2] = bf2_to_f2(v.z); x[3] = bf2_to_f2(v.w);
    }
    __device__ static __forceinline__ uint4 pack(const float2 (&x)[4]) {
        return make_uint4(f2_to_bf2(x[0].x, x[0].y), f2_to_bf2(x[1].x, x[1].y),
                          f2_to_bf2(x[2].x, x[2].y), f2_to_bf2(x[3].x, x[3].y));
    }
};
template <> struct Elem<float> {
    static constexpr int EPV = 4;
    static constexpr int BYTES = 4;
    __device__ static __forceinline__ void unpack(const uint4 &v, float2 (&x)[2]) {
        x[0] = make_float2(__uint_as_float(v.x), __uint_as_float(v.y));
        x[1] = make_float2(__uint_as_float(v.z), __uint_as_float(v.w));
    }
    __device__ static __forceinline__ uint4 pack(const float2 (&x)[2]) {
        return make_uint4(__float_as_uint(x[0].x), __float_as_uint(x[0].y),
                          __float_as_uint(x[1].x), __float_as_uint(x[1].y));
    }
};

__device__ __forceinline__ uint4 lds128(const void *p) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(smem_u32(p)));
    return v;
}
// 16-byte shared load from a 32-bit shared-window address.
__device__ __forceinline__ uint4 lds128u(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(a));
    return v;
}
__device__ __forceinline__ float4 lds128f(uint32_t a) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(a));
    return v;
}
__device__ __forceinline__ float lds32f(uint32_t a) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a));
    return v;
}

__device__ __forceinline__ void stg128_cs(void *p, const uint4 &v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ uint4 ldg128_stream(const void *p) {
    uint4 v;
    asm volatile("ld.global.cs.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// ----------------------------------------------------- warp reductions
// Butterfly all-to-some reduction of N values across the 32 lanes of a warp.
// Each of the five steps (partner lane = lane ^ 16, 8, 4, 2, 1) exchanges
// half of the values still held: the lane whose partner bit is set keeps the
// upper half, the other the lower half, so the warp issues about N shuffles
// in total instead of 5 per value.  Sizes shrink as n -> ceil(n/2); an odd
// size pads one zero.  On return lane L holds in v[0..R-1] (R = size after 5
// halvings) warp-wide sums whose value indices bfly_slot() gives.
template <int N>
struct Bfly {
    static constexpr int N1 = (N + 1) / 2, N2 = (N1 + 1) / 2, N3 = (N2 + 1) / 2, N4 = (N3 + 1) / 2,
                         N5 = (N4 + 1) / 2;
    static constexpr int R = N5;
};

template <int N, int OFF>
__device__ __forceinline__ void bfly_step(float *v, int lane) {
    constexpr int H = (N + 1) / 2;
    const bool upper = (lane & OFF) != 0;
#pragma unroll
    for (int i = 0; i < H; ++i) {
        const float lo = v[i];
        const float hi = (i + H < N) ? v[i + H] : 0.f;
        const float send = upper ? lo : hi;
        const float keep = upper ? hi : lo;
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, OFF);
    }
}

template <int N>
__device__ __forceinline__ void butterfly_reduce(float *v, int lane) {
    using B = Bfly<N>;
    bfly_step<N, 16>(v, lane);
    bfly_step<B::N1, 8>(v, lane);
    bfly_step<B::N2, 4>(v, lane);
    bfly_step<B::N3, 2>(v, lane);
    bfly_step<B::N4, 1>(v, lane);
}

// Value index held by slot j of lane `lane` after butterfly_reduce<N>, or -1
// if that slot is padding.
template <int N>
__host__ __device__ inline int bfly_slot(int lane, int j) {
    using B = Bfly<N>;
    const int n[6] = {N, B::N1, B::N2, B::N3, B::N4, B::N5};
    int pos = j;
    if (pos >= n[5]) return -1;
    for (int s = 4; s >= 0; --s) {
        if (lane & (16 >> s)) pos += n[s + 1];
        if (pos >= n[s]) return -1;
    }
    return pos;
}

template <int W>
__device__ __forceinline__ float seg_max(float x) {
#pragma unroll
    for (int o = W / 2; o >= 1; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}
template <int W>
__device__ __forceinline__ float seg_sum(float x) {
#pragma unroll
    for (int o = W / 2; o >= 1; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// score of one key: dot / sqrt(ss / n + eps); a zero key with eps = 0 scores 0.
__device__ __forceinline__ float key_score(float dot, float ss, float inv_n, float eps) {
    const float ms = fmaf(ss, inv_n, eps);
    return ms > 0.f ? dot * rsqrtf(ms) : 0.f;
}

}  // namespace attnres
