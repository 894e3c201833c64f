// attnres_api.cu -- host side of the C ABI declared in include/attnres.h:
// argument validation, launch-shape selection and kernel dispatch.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "../../include/attnres.h"
#include "common.cuh"
#include "depth_read.cuh"
#include "depth_read_decode.cuh"
#include "depth_read_mma.cuh"
#include "dispatch.h"
#include "msar.h"
#include "msar_bwd.h"
#include "phase2.cuh"
#include "merge_bwd.cuh"
#include "read_bwd.cuh"
#include "read_bwd_split.cuh"
#include "read_bwd_one.cuh"
#include "read_bwd_many.cuh"
#include "state_merge_bwd.h"

using namespace attnres;

// Device status word: kernels OR DEV_ERR_* bits into it after a wait ran out.
__device__ int g_attnres_status = 0;

namespace {

thread_local char t_last_err[256] = "";

std::atomic<uint64_t> g_timeout_ns{2000000000ull};
std::atomic<int> g_inject_stall{0};
std::atomic<int> g_kernel_variant{0};   // 0 automatic, 1 general (CUDA-core) depth read only,
                                        // 2 tensor-core depth reads wherever they apply,
                                        // 3 the few-token kernel wherever it applies

constexpr int kMaxDevices = 64;
constexpr size_t kStageMaxBytes = 64 * 1024;        // one ring stage
constexpr size_t kSmemBudget = 227 * 1024;         // stages + aux, per CTA (sm_103a opt-in limit)
constexpr size_t kCtaReserve = 1024;              // shared memory the runtime reserves per CTA

struct DeviceInfo {
    std::once_flag once;
    cudaError_t err = cudaSuccess;
    int sms = 0;
    int smem_optin = 0;
    int *status = nullptr;
};
DeviceInfo g_dev[kMaxDevices];

attnres_status_t cuda_fail(cudaError_t e, const char *what) {
    snprintf(t_last_err, sizeof(t_last_err), "%s: %s (%s)", what, cudaGetErrorName(e),
             cudaGetErrorString(e));
    return ATTNRES_ERR_CUDA;
}

// Per-device constants: SM count, shared-memory limit, status word address.
attnres_status_t device_info(DeviceInfo **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return ATTNRES_ERR_UNSUPPORTED;
    DeviceInfo &d = g_dev[dev];
    std::call_once(d.once, [&] {
        d.err = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
        if (d.err == cudaSuccess)
            d.err = cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (d.err == cudaSuccess)
            d.err = cudaGetSymbolAddress(reinterpret_cast<void **>(&d.status), g_attnres_status);
    });
    if (d.err != cudaSuccess) return cuda_fail(d.err, "device query");
    *out = &d;
    return ATTNRES_OK;
}

WaitCfg wait_cfg(DeviceInfo *d) {
    WaitCfg w;
    w.status = d->status;
    w.timeout_ns = g_timeout_ns.load();
    w.inject_stall = g_inject_stall.load();
    return w;
}

// Kernel attributes are set once per (function, device).
struct FnCache {
    std::mutex mu;
    struct Entry { const void *fn; int dev; size_t smem; int occ; };
    Entry e[512];
    int n = 0;
} g_fn_cache;

attnres_status_t prepare_kernel(const void *fn, size_t smem, int threads, int *occ) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    std::lock_guard<std::mutex> lk(g_fn_cache.mu);
    for (int i = 0; i < g_fn_cache.n; ++i) {
        auto &c = g_fn_cache.e[i];
        if (c.fn == fn && c.dev == dev && c.smem >= smem) { *occ = c.occ; return ATTNRES_OK; }
    }
    if (smem > 48 * 1024) {
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
    }
    int o = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, fn, threads, smem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
    if (o < 1) return ATTNRES_ERR_UNSUPPORTED;
    if (g_fn_cache.n < 512) g_fn_cache.e[g_fn_cache.n++] = {fn, dev, smem, o};
    *occ = o;
    return ATTNRES_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

size_t esize(attnres_dtype_t dt) { return dt == ATTNRES_BF16 ? 2 : 4; }
int epv(attnres_dtype_t dt) { return dt == ATTNRES_BF16 ? 8 : 4; }

// [a, a+na) and [b, b+nb) overlap (bytes)
bool overlap(const void *a, size_t na, const void *b, size_t nb) {
    if (!a || !b || na == 0 || nb == 0) return false;
    auto x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

int pow2ceil(int x) {
    int p = 1;
    while (p < x) p <<= 1;
    return p;
}

// Threads per token row and vectors per thread for a row of nvec vectors.
void row_shape(int nvec, int *tpr, int *vpt) {
    int t = pow2ceil((nvec + 1) / 2);
    if (t < 32) t = 32;
    if (t > 256) t = 256;
    *tpr = t;
    *vpt = pow2ceil((nvec + t - 1) / t);
}

attnres_status_t check_common(const void *src, int64_t n_src, int64_t src_stride, int64_t T,
                              int64_t d, attnres_dtype_t dt, float eps) {
    if (dt != ATTNRES_F32 && dt != ATTNRES_BF16) return ATTNRES_ERR_INVALID_ARG;
    if (n_src < 1 || T < 0 || d < 1 || !(eps >= 0.f) || std::isinf(eps)) return ATTNRES_ERR_INVALID_ARG;
    if (T > 0 && !src) return ATTNRES_ERR_INVALID_ARG;
    if (T > 0 && d > INT64_MAX / T) return ATTNRES_ERR_INVALID_ARG;
    if (src_stride < T * d) return ATTNRES_ERR_INVALID_ARG;
    if (d % 8 != 0) return ATTNRES_ERR_UNSUPPORTED;
    if (!aligned16(src) || (src_stride * (int64_t)esize(dt)) % 16 != 0) return ATTNRES_ERR_UNSUPPORTED;
    if (n_src > (int64_t)1 << 30 || d > (int64_t)1 << 20) return ATTNRES_ERR_UNSUPPORTED;
    return ATTNRES_OK;
}

// Calls with at most this many tokens take the few-token kernel: a token per
// cluster of CTAs beats the streaming kernels' one CTA per token there.
constexpr int64_t kDecodeMaxT = 64;

// Few-token kernel shape: the largest cluster (<= 8 CTAs) whose CTAs each get
// a whole number of warps of 16-byte vectors, one vector per thread.
bool decode_shape(int nvec, int *cs, int *vpc) {
    for (int c = DEC_MAX_CS; c >= 1; c >>= 1) {
        if (nvec % c) continue;
        const int v = nvec / c;
        if (v % 32 == 0 && v <= DEC_MAX_THREADS) { *cs = c; *vpc = v; return true; }
    }
    return false;
}

// Shared launch path of Full / phase 1 / MHAR.
// out_q_stride: elements between the queries' outputs (0: T * d, packed)
attnres_status_t launch_depth_read(const void *src, int64_t n_src, int64_t src_stride, int64_t T,
                                   int64_t d, int64_t H, attnres_dtype_t dt, const float *queries,
                                   int64_t n_q, const float *gain, float eps, void *out, float *lse,
                                   void *stream, int64_t out_q_stride = 0) {
    attnres_status_t st = check_common(src, n_src, src_stride, T, d, dt, eps);
    if (st != ATTNRES_OK) return st;
    if (n_q < 1 || H < 1 || d % H != 0) return ATTNRES_ERR_INVALID_ARG;
    if (T > 0 && (!queries || !out)) return ATTNRES_ERR_INVALID_ARG;
    const int64_t oqs = out_q_stride > 0 ? out_q_stride : T * d;
    if (n_q > 1 && oqs < T * d) return ATTNRES_ERR_INVALID_ARG;
    const size_t es = esize(dt);
    const size_t src_bytes = ((size_t)(n_src - 1) * (size_t)src_stride + (size_t)T * (size_t)d) * es;
    const size_t out_bytes = ((size_t)(n_q - 1) * (size_t)oqs + (size_t)T * (size_t)d) * es;
    if (overlap(out, out_bytes, src, src_bytes)) return ATTNRES_ERR_INVALID_ARG;
    if (lse && overlap(lse, (size_t)n_q * H * T * 4, src, src_bytes)) return ATTNRES_ERR_INVALID_ARG;
    if (lse && overlap(lse, (size_t)n_q * H * T * 4, out, out_bytes)) return ATTNRES_ERR_INVALID_ARG;
    if (n_q > 8) return ATTNRES_ERR_UNSUPPORTED;
    if (!aligned16(out) || !aligned16(queries) || (gain && !aligned16(gain)) || (lse && !aligned4(lse)))
        return ATTNRES_ERR_UNSUPPORTED;
    if (T == 0) return ATTNRES_OK;

    // Few tokens (decode-shaped calls): one token per cluster of CTAs.
    const int kvd = g_kernel_variant.load();
    if (H == 1 && n_q <= 4 && (kvd == 3 || (kvd == 0 && T <= kDecodeMaxT))) {
        int cs = 0, vpc = 0;
        const int ns = n_src <= 8 ? 8 : 16;
        KernelRef kr;
        if (n_src <= 16 && decode_shape((int)(d / epv(dt)), &cs, &vpc) &&
            lookup_depth_read_decode(dt == ATTNRES_BF16 ? 1 : 0, pow2ceil((int)n_q), ns, &kr)) {
            DecodeArgs a;
            a.src = static_cast<const unsigned char *>(src);
            a.src_stride_bytes = src_stride * (int64_t)es;
            a.n_src = (int)n_src;
            a.T = T;
            a.d = (int)d;
            a.n_q = (int)n_q;
            a.queries = queries;
            a.gain = gain;
            a.eps = eps;
            a.out = static_cast<unsigned char *>(out);
            a.out_q_stride_bytes = oqs * (int64_t)es;
            a.lse = lse;
            a.cs = cs;
            a.vpc = vpc;
            cudaLaunchConfig_t cfg = {};
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = cs;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            cfg.gridDim = dim3((unsigned)(T * cs));
            cfg.blockDim = dim3((unsigned)vpc);
            cfg.dynamicSmemBytes = 0;
            cfg.stream = static_cast<cudaStream_t>(stream);
            void *args[] = {&a};
            cudaError_t e = cudaLaunchKernelExC(&cfg, kr.fn, args);
            if (e != cudaSuccess) return cuda_fail(e, "depth_read_decode launch");
            return ATTNRES_OK;
        }
    }

    // Tensor-core path: bf16, <= 4 queries, d = 1024/2048/4096, heads that are
    // whole multiples of the per-warp channel slice.  <= 8 sources: one token
    // per item with 256 channels per warp at d = 4096 (16 warps) and d = 2048
    // (8 warps, two CTAs per SM); d = 1024 two tokens per item (8 warps x 128
    // channels), which fills all 16 MMA rows.
    // > 8 sources: one token per item, its sources in chunks of 8 folded in by
    // an online softmax (only d = 4096 is built: slower than the general
    // kernel at d = 2048).  An item costs about the same whatever its rows
    // and queries.  Measured at d = 4096, T = 16384, 9..64 sources: for one
    // query and one head the general kernel's 6-source chunks (two CTAs per
    // SM) are faster at every count (60.3 ms summed against 70.7 ms); for
    // two to four queries the chunked kernel is faster from 10 sources on
    // (15.2 against 22.9 ms over 9, 14, ..., 64 sources at two queries); for
    // heads (MHAR) it is faster at every count (1.91 against 3.95 ms at 64).
    // One query over at most 4 sources at d = 4096 (the first layers of Full
    // AttnRes at depth): the one-token kernel costs about the same whatever
    // its rows, and the general kernel's tiles of several tokens are faster
    // (measured at T = 16384: 0.12-0.26 ms against 0.28 ms).
    const int kv = g_kernel_variant.load();
    const bool chunked = n_src > 8;
    const bool chunked_wins = H > 1 || (n_q >= 2 && n_src >= 10);
    const bool few_rows = d == 4096 && n_q == 1 && H == 1 && n_src <= 4;
    if (dt == ATTNRES_BF16 && n_q <= 4 && (d == 1024 || d == 2048 || d == 4096) && kv != 1 &&
        (!few_rows || kv == 2) && (!chunked || (d == 4096 && (chunked_wins || kv == 2)))) {
        const bool two = !chunked && d <= 1024;
        const int nw = d <= 2048 ? 8 : 16;
        const int ks = (int)(d / (16 * nw));
        const int rows = two ? 16 : 8;
        const int nq2 = pow2ceil((int)n_q);
        KernelRef kr;
        const bool found = chunked ? lookup_depth_read_mma_multi(nq2, ks, nw, &kr)
                           : two   ? lookup_depth_read_mma2(nq2, ks, nw, &kr)
                                   : lookup_depth_read_mma(nq2, ks, nw, &kr);
        if (nw % H == 0 && found) {
            DeviceInfo *dev = nullptr;
            st = device_info(&dev);
            if (st != ATTNRES_OK) return st;
            const uint32_t pitch = (uint32_t)(2 * d + 16);
            const uint32_t stage_bytes = (rows * pitch + 127) / 128 * 128;
            size_t budget = kSmemBudget;
            if ((size_t)dev->smem_optin < budget) budget = (size_t)dev->smem_optin;
            int nstages = (int)((budget - kr.aux_smem) / stage_bytes);
            if (nstages > DM_MAX_STAGES) nstages = DM_MAX_STAGES;
            // d = 2048: three stages, so that two CTAs share an SM (measured
            // 10-16% faster than one CTA with more stages or two tokens per item)
            if (d == 2048 && !chunked && nstages > 3) nstages = 3;
            if (nstages >= 2) {
                const size_t smem = (size_t)nstages * stage_bytes + kr.aux_smem;
                int occ = 0;
                st = prepare_kernel(kr.fn, smem, nw * 32, &occ);
                if (st != ATTNRES_OK) return st;
                DepthReadMmaArgs m;
                m.src = static_cast<const unsigned char *>(src);
                m.src_stride_bytes = src_stride * 2;
                m.n_src = (int)n_src;
                m.T = T;
                m.d = (int)d;
                m.n_q = (int)n_q;
                m.H = (int)H;
                m.wph = (int)(nw / H);
                m.queries = queries;
                m.gain = gain;
                m.eps = eps;
                m.out = static_cast<unsigned char *>(out);
                m.out_q_stride_bytes = oqs * 2;
                m.lse = lse;
                m.nstages = nstages;
                m.pitch = pitch;
                m.stage_bytes = stage_bytes;
                m.wait = wait_cfg(dev);
                const int64_t items = two ? (T + 1) / 2 : T;
                const int64_t max_grid = (int64_t)dev->sms * occ;
                const int grid = (int)(items < max_grid ? items : max_grid);
                // the chunked kernel counts a CTA's (token, chunk) items in an int
                const int64_t per_cta = (items + grid - 1) / grid * (chunked ? (n_src + 7) / 8 : 1);
                if (per_cta <= (int64_t)INT32_MAX) {
                    void *args[] = {&m};
                    cudaError_t e = cudaLaunchKernel(kr.fn, dim3(grid), dim3(nw * 32), args, smem,
                                                     static_cast<cudaStream_t>(stream));
                    if (e != cudaSuccess) return cuda_fail(e, "depth_read_mma launch");
                    return ATTNRES_OK;
                }
            }
        }
    }

    const int EPV = epv(dt);
    const int nvec = (int)(d / EPV);
    int tpr, vpt;
    row_shape(nvec, &tpr, &vpt);
    const int nq_pad = pow2ceil((int)n_q);
    // more queries need more registers per vector: spread the row over more
    // threads until NQ * VPT * EPV fits the budget of 64 (or no wider row exists)
    while ((int64_t)nq_pad * vpt * EPV > 64 && tpr < 256 && vpt > 1) {
        tpr *= 2;
        vpt = pow2ceil((nvec + tpr - 1) / tpr);
    }
    if (vpt > 8 || (int64_t)nq_pad * vpt * EPV > 64) return ATTNRES_ERR_UNSUPPORTED;
    bool mh = false;
    int seg = nvec;
    if (H > 1) {
        if ((d / H) % EPV != 0) return ATTNRES_ERR_UNSUPPORTED;
        seg = (int)(nvec / H);
        if (seg % 32 != 0) return ATTNRES_ERR_UNSUPPORTED;
        mh = true;
    }
    const int tt = 256 / tpr;
    const size_t row_bytes = (size_t)d * es;
    int chunk = (int)(kStageMaxBytes / ((size_t)tt * row_bytes));
    if (chunk < 1) return ATTNRES_ERR_UNSUPPORTED;
    if (chunk > DR_CMAX) chunk = DR_CMAX;
    if (chunk > n_src) chunk = (int)n_src;
    const bool multi = n_src > chunk;

    KernelRef kr;
    if (!lookup_depth_read(dt == ATTNRES_BF16 ? 1 : 0, nq_pad, vpt, mh, multi, &kr))
        return ATTNRES_ERR_UNSUPPORTED;

    DeviceInfo *dev = nullptr;
    st = device_info(&dev);
    if (st != ATTNRES_OK) return st;

    const uint32_t src_pitch = (uint32_t)(tt * row_bytes);
    size_t budget = kSmemBudget;
    if ((size_t)dev->smem_optin < budget) budget = (size_t)dev->smem_optin;
    if (budget <= kr.aux_smem) return ATTNRES_ERR_UNSUPPORTED;
    int max_stages = DR_MAX_STAGES;
    if (multi) {
        // Chunked (online-softmax) reads: two CTAs per SM, so that they hide
        // each other's per-chunk latency, with two stages each and the
        // largest chunk that fits.  Each chunk costs a CTA-wide reduction
        // whatever its rows, so fewer, larger chunks win over more stages:
        // Full at depth, 9..64 sources at d = 4096 (8 KB per source and
        // stage): 4-source chunks x 3 stages 69.9 ms, 4 x 2 70.0 ms, 6 x 2
        // 60.0 ms; 8 x 2 (one CTA per SM) 86.9 ms.  The same shape at d =
        // 1024 and 2048 gains the same 15%.
        const size_t half = budget / 2;
        const size_t need = kr.aux_smem + kCtaReserve;
        int fit = 0;
        while (fit < chunk && need + 2 * (((size_t)(fit + 1) * src_pitch + 127) / 128 * 128) <= half) ++fit;
        if (fit >= 1) {
            chunk = fit;
            max_stages = 2;
        }
        const int cap = dr_chunk_cap(vpt, true);
        if (chunk > cap) chunk = cap;
    }
    const int nchunks = (int)((n_src + chunk - 1) / chunk);
    const uint32_t stage_bytes = (uint32_t)(((size_t)chunk * src_pitch + 127) / 128 * 128);
    int nstages = (int)((budget - kr.aux_smem) / stage_bytes);
    if (nstages > max_stages) nstages = max_stages;
    if (nstages < 2) return ATTNRES_ERR_UNSUPPORTED;
    size_t smem = (size_t)nstages * stage_bytes + kr.aux_smem;

    int occ = 0;
    st = prepare_kernel(kr.fn, smem, DR_THREADS, &occ);
    if (st != ATTNRES_OK) return st;
    if (max_stages == 2 && occ < 2) {
        // the kernel's registers leave room for one CTA per SM (several
        // queries): it takes the stages the second CTA would have had
        int more = (int)((budget - kr.aux_smem) / stage_bytes);
        if (more > DR_MAX_STAGES) more = DR_MAX_STAGES;
        if (more > nstages) {
            nstages = more;
            smem = (size_t)nstages * stage_bytes + kr.aux_smem;
            st = prepare_kernel(kr.fn, smem, DR_THREADS, &occ);
            if (st != ATTNRES_OK) return st;
        }
    }

    DepthReadArgs a;
    a.src = static_cast<const unsigned char *>(src);
    a.src_stride_bytes = src_stride * (int64_t)es;
    a.n_src = (int)n_src;
    a.T = T;
    a.d = (int)d;
    a.nvec = nvec;
    a.n_q = (int)n_q;
    a.H = (int)H;
    a.seg = seg;
    a.queries = queries;
    a.gain = gain;
    a.eps = eps;
    a.out = static_cast<unsigned char *>(out);
    a.out_q_stride_bytes = oqs * (int64_t)es;
    a.lse = lse;
    a.tpr = tpr;
    a.tt = tt;
    a.chunk = chunk;
    a.nchunks = nchunks;
    a.nstages = nstages;
    a.stage_bytes = stage_bytes;
    a.src_pitch = src_pitch;
    a.ntiles = (T + tt - 1) / tt;
    a.wait = wait_cfg(dev);

    const int64_t max_grid = (int64_t)dev->sms * occ;
    const int grid = (int)(a.ntiles < max_grid ? a.ntiles : max_grid);
    void *args[] = {&a};
    cudaError_t e = cudaLaunchKernel(kr.fn, dim3(grid), dim3(DR_THREADS), args, smem,
                                     static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "depth_read launch");
    return ATTNRES_OK;
}

// Shared launch path of the phase-2 merges (one head or H heads, with or
// without the fused partial-sum update).  upd: partial_out = partial + f, and
// the merge scores it; otherwise the merge scores partial (NULL: out = o).
attnres_status_t launch_phase2(const void *o, const float *lse, const void *partial, const void *f,
                               void *partial_out, bool upd, int64_t T, int64_t d, int64_t H,
                               attnres_dtype_t dt, const float *query, const float *gain, float eps,
                               void *out, void *stream) {
    if (dt != ATTNRES_F32 && dt != ATTNRES_BF16) return ATTNRES_ERR_INVALID_ARG;
    if (T < 0 || d < 1 || H < 1 || d % H != 0 || !(eps >= 0.f) || std::isinf(eps)) return ATTNRES_ERR_INVALID_ARG;
    if (T > 0 && (!o || !out)) return ATTNRES_ERR_INVALID_ARG;
    if (T > 0 && upd && (!f || !partial_out)) return ATTNRES_ERR_INVALID_ARG;
    const bool merges = upd || partial;
    if (T > 0 && merges && (!lse || !query)) return ATTNRES_ERR_INVALID_ARG;
    if (T > 0 && d > INT64_MAX / T) return ATTNRES_ERR_INVALID_ARG;
    const size_t es = esize(dt);
    const size_t nbytes = (size_t)T * (size_t)d * es;
    const size_t lbytes = (size_t)H * (size_t)T * 4;
    // out may be o itself but may overlap no other tensor; the updated partial
    // may be partial or f itself but may overlap nothing else
    if (out != o && overlap(out, nbytes, o, nbytes)) return ATTNRES_ERR_INVALID_ARG;
    if (partial && overlap(out, nbytes, partial, nbytes)) return ATTNRES_ERR_INVALID_ARG;
    if (upd) {
        if (overlap(out, nbytes, f, nbytes) || overlap(out, nbytes, partial_out, nbytes) ||
            overlap(partial_out, nbytes, o, nbytes))
            return ATTNRES_ERR_INVALID_ARG;
        if (partial_out != partial && partial && overlap(partial_out, nbytes, partial, nbytes))
            return ATTNRES_ERR_INVALID_ARG;
        if (partial_out != f && overlap(partial_out, nbytes, f, nbytes)) return ATTNRES_ERR_INVALID_ARG;
    }
    if (merges && lse && (overlap(lse, lbytes, out, nbytes) || (upd && overlap(lse, lbytes, partial_out, nbytes))))
        return ATTNRES_ERR_INVALID_ARG;
    if (d % 8 != 0) return ATTNRES_ERR_UNSUPPORTED;
    if (!aligned16(o) || !aligned16(out) || (partial && !aligned16(partial)) || (f && !aligned16(f)) ||
        (partial_out && !aligned16(partial_out)) || (query && !aligned16(query)) ||
        (gain && !aligned16(gain)) || (lse && !aligned4(lse)))
        return ATTNRES_ERR_UNSUPPORTED;
    const int EPV = epv(dt);
    const int nvec = (int)(d / EPV);
    int seg = nvec;
    if (H > 1) {
        // a head is whole 16-byte vectors, and either whole warps of them or a
        // power-of-two group inside a warp
        if ((d / H) % EPV != 0) return ATTNRES_ERR_UNSUPPORTED;
        seg = (int)(nvec / H);
        if (seg % 32 != 0 && (seg > 32 || (seg & (seg - 1)) != 0)) return ATTNRES_ERR_UNSUPPORTED;
    }
    if (T == 0) return ATTNRES_OK;
    if (!merges) {
        if (out == o) return ATTNRES_OK;
        cudaError_t e = cudaMemcpyAsync(out, o, nbytes, cudaMemcpyDeviceToDevice, static_cast<cudaStream_t>(stream));
        return e == cudaSuccess ? ATTNRES_OK : cuda_fail(e, "cudaMemcpyAsync");
    }
    int tpr, vpt;
    row_shape(nvec, &tpr, &vpt);
    KernelRef kr;
    if (vpt > 8 || !lookup_phase2(dt == ATTNRES_BF16 ? 1 : 0, vpt, upd, H > 1, &kr)) return ATTNRES_ERR_UNSUPPORTED;
    DeviceInfo *dev = nullptr;
    attnres_status_t st = device_info(&dev);
    if (st != ATTNRES_OK) return st;
    int occ = 0;
    st = prepare_kernel(kr.fn, 0, P2_THREADS, &occ);
    if (st != ATTNRES_OK) return st;
    MergeArgs a;
    a.o = static_cast<const unsigned char *>(o);
    a.lse = lse;
    a.partial = static_cast<const unsigned char *>(partial);
    a.f = static_cast<const unsigned char *>(f);
    a.partial_out = static_cast<unsigned char *>(partial_out);
    a.T = T;
    a.d = (int)d;
    a.nvec = nvec;
    a.seg = seg;
    a.query = query;
    a.gain = gain;
    a.eps = eps;
    a.out = static_cast<unsigned char *>(out);
    a.tpr = tpr;
    a.tt = P2_THREADS / tpr;
    a.ntiles = (T + a.tt - 1) / a.tt;
    const int64_t max_grid = (int64_t)dev->sms * occ;
    const int grid = (int)(a.ntiles < max_grid ? a.ntiles : max_grid);
    void *args[] = {&a};
    cudaError_t e = cudaLaunchKernel(kr.fn, dim3(grid), dim3(P2_THREADS), args, 0, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "phase2 launch");
    return ATTNRES_OK;
}

// Backward of the read: tile shape, workspace size and launch.
struct ReadBwdShape {
    int tpr, vpt, tt, ns;
    int nqc;        // queries per kernel pass (more queries take several passes)
    bool mh;        // per-head mode (H > 1)
    int hg;         // reduction groups per warp in per-head mode
    int vph;        // 16-byte vectors per head
};

attnres_status_t read_bwd_shape_for(int64_t n_src, int64_t d, int nqc, int64_t H, attnres_dtype_t dt,
                                    ReadBwdShape *sh) {
    const int nvec = (int)(d / epv(dt));
    sh->nqc = nqc;
    row_shape(nvec, &sh->tpr, &sh->vpt);
    sh->tt = RB_THREADS / sh->tpr;
    // a tile holds n_src + nqc rows of tt tokens and two stages must fit:
    // spread a token over more threads (fewer tokens per tile) until they do
    const size_t rows = (size_t)(n_src + sh->nqc) * (size_t)d * esize(dt);
    while (2 * rows * (size_t)sh->tt + 8 * 1024 > kSmemBudget && sh->tpr < RB_THREADS && sh->vpt > 1) {
        sh->tpr *= 2;
        sh->vpt = pow2ceil((nvec + sh->tpr - 1) / sh->tpr);
        sh->tt = RB_THREADS / sh->tpr;
    }
    if (sh->vpt > 4) return ATTNRES_ERR_UNSUPPORTED;
    sh->mh = H > 1;
    sh->hg = 1;
    sh->vph = nvec;
    if (sh->mh) {
        // heads of whole runs of 32 vectors; one group per warp when a head
        // holds whole warps' worth of vectors, else one group per run
        if ((d / H) % epv(dt) != 0) return ATTNRES_ERR_UNSUPPORTED;
        sh->vph = nvec / (int)H;
        if (sh->vph % (32 * sh->vpt) == 0) sh->hg = 1;
        else if (sh->vph % 32 == 0) sh->hg = sh->vpt;
        else return ATTNRES_ERR_UNSUPPORTED;
    }
    return ATTNRES_OK;
}

// max_nqc: at most this many queries per launch (0: no limit beyond the kernels')
attnres_status_t read_bwd_shape(int64_t n_src, int64_t d, int64_t n_q, int64_t H, attnres_dtype_t dt,
                                ReadBwdShape *sh, int max_nqc = 0) {
    if (n_src > 16) return ATTNRES_ERR_UNSUPPORTED;
    sh->ns = n_src <= 8 ? 8 : 16;
    // queries per launch: up to 4 (two groups of two over the same staged
    // sources) with at most 8 sources where that kernel exists, else 2 (1
    // with more than 8 sources)
    int base = sh->ns == 16 ? 1 : 2;
    if (max_nqc > 0 && base > max_nqc) base = max_nqc;
    if (sh->ns == 8 && n_q > 2 && (max_nqc == 0 || max_nqc > 2)) {
        const int want = n_q < 4 ? (int)n_q : 4;
        KernelRef kr;
        if (read_bwd_shape_for(n_src, d, want, H, dt, sh) == ATTNRES_OK &&
            lookup_read_bwd_qg(dt == ATTNRES_BF16 ? 1 : 0, sh->vpt, sh->mh, sh->hg, &kr))
            return ATTNRES_OK;
    }
    return read_bwd_shape_for(n_src, d, n_q < base ? (int)n_q : base, H, dt, sh);
}

// Per-(CTA, row) partials of U for one pass of queries: one CTA per SM at most.
size_t read_bwd_ws_bytes(int sms, const ReadBwdShape &sh, int64_t d) {
    return (size_t)sms * (size_t)sh.tt * (size_t)sh.nqc * (size_t)d * sizeof(float);
}

// The two-kernel form (read_bwd_split.cuh) takes a pass of 3 or 4 queries
// with bf16 sources, at most 8 of them, d = 2048 or 4096 and heads of at
// least 256 channels (debug kernel variant 1 keeps the one-kernel form).
bool read_bwd_split_applies(attnres_dtype_t dt, int64_t n_src, int64_t nq, int64_t d, int64_t H) {
    if (g_kernel_variant.load() == 1) return false;
    return dt == ATTNRES_BF16 && n_src >= 1 && n_src <= 8 && (nq == 3 || nq == 4) && (d == 2048 || d == 4096) &&
           H >= 1 && H <= RC_NW && d % H == 0 && (d / H) % 256 == 0;
}

struct ReadBwdSplitShape {
    int chunks = 0;          // apply CTAs along the tokens (partials of U)
    int64_t tpc = 0;         // tokens per apply CTA
    int nstages = 0;         // half-row stages of the coefficient kernel
    uint32_t pitch = 0, stage_bytes = 0;
    size_t smem = 0;
    size_t off_coef = 0;     // coefficients after the partials of U
    size_t total = 0;
};

attnres_status_t read_bwd_split_shape(int64_t T, int64_t d, int64_t H, const DeviceInfo *dev,
                                      ReadBwdSplitShape *sh) {
    KernelRef kc, ka;
    if (!lookup_read_bwd_split(4, (int)d, &kc, &ka)) return ATTNRES_ERR_UNSUPPORTED;
    sh->pitch = (uint32_t)d + 16;
    sh->stage_bytes = 12u * sh->pitch;
    size_t budget = kSmemBudget;
    if ((size_t)dev->smem_optin < budget) budget = (size_t)dev->smem_optin;
    if (budget <= RC_AUX_BYTES) return ATTNRES_ERR_UNSUPPORTED;
    int ns = (int)((budget - RC_AUX_BYTES) / sh->stage_bytes);
    if (ns > RC_MAX_STAGES) ns = RC_MAX_STAGES;
    if (ns < 2) return ATTNRES_ERR_UNSUPPORTED;
    sh->nstages = ns;
    sh->smem = (size_t)ns * sh->stage_bytes + RC_AUX_BYTES;
    int occ = 0;
    attnres_status_t st = prepare_kernel(ka.fn, RA_RING_BYTES, RA_THREADS, &occ);
    if (st != ATTNRES_OK) return st;
    // one wave of apply CTAs: d / 1024 channel slices times token ranges
    const int64_t slices = d / RA_W;
    int64_t chunks = ((int64_t)occ * dev->sms + slices - 1) / slices;
    if (chunks > T) chunks = T;
    if (chunks < 1) chunks = 1;
    sh->tpc = (T + chunks - 1) / chunks;
    sh->chunks = (int)(T > 0 ? (T + sh->tpc - 1) / sh->tpc : 0);
    const size_t ws_u = ((size_t)sh->chunks * 4 * (size_t)d * sizeof(float) + 255) / 256 * 256;
    sh->off_coef = ws_u;
    sh->total = ws_u + (size_t)T * (size_t)H * RC_NV * sizeof(float);
    return ATTNRES_OK;
}

// The one-kernel ring form (read_bwd_one.cuh) takes a pass of one query over
// 3 to 16 bf16 sources at d = 2048 or 4096 whose rows can be bulk-copied
// (measured at T = 32768, d = 4096: 0.54 vs 0.55 ms at 3 sources, 0.80 vs
// 1.02 ms at 8; debug kernel variant 1 keeps read_bwd_kernel).  Its
// workspace, one partial of U per CTA, is within read_bwd_ws_bytes.
bool read_bwd_one_applies(attnres_dtype_t dt, int64_t n_src, int64_t nq, int64_t d, int64_t H, const void *src,
                          int64_t src_stride) {
    if (g_kernel_variant.load() == 1) return false;
    return dt == ATTNRES_BF16 && n_src >= 3 && n_src <= 16 && nq == 1 && H == 1 && (d == 2048 || d == 4096) &&
           aligned16(src) && (src_stride * 2) % 16 == 0;
}

// One pass of one query in the one-kernel ring form: one CTA per SM, U as one
// partial per CTA at the start of the workspace (*nparts of them).
attnres_status_t launch_read_bwd_one_pass(const ReadBwdArgs &a, const DeviceInfo *dev, void *stream, int *nparts) {
    KernelRef kr;
    if (!lookup_read_bwd_one(a.d, a.n_src, &kr)) return ATTNRES_ERR_UNSUPPORTED;
    ReadBwdOneArgs o;
    o.pitch = (uint32_t)a.d + 16;
    // up to 8 sources: 8 source rows and the gradient row, two tokens' stages
    // held at a time; more: the n_src source rows and the gradient row, one
    // token's stages held
    const bool pipelined = a.n_src <= 8;
    o.stage_bytes = (uint32_t)(pipelined ? R1_ROWS : a.n_src + 1) * o.pitch;
    size_t budget = kSmemBudget;
    if ((size_t)dev->smem_optin < budget) budget = (size_t)dev->smem_optin;
    if (budget <= kr.aux_smem) return ATTNRES_ERR_UNSUPPORTED;
    int ns = (int)((budget - kr.aux_smem) / o.stage_bytes);
    if (ns > R1_MAX_STAGES) ns = R1_MAX_STAGES;
    if (ns < (pipelined ? 4 : 3)) return ATTNRES_ERR_UNSUPPORTED;
    const size_t smem = (size_t)ns * o.stage_bytes + kr.aux_smem;
    int occ = 0;
    attnres_status_t st = prepare_kernel(kr.fn, smem, R1_NW * 32, &occ);
    if (st != ATTNRES_OK) return st;
    o.src = a.src;
    o.src_stride_bytes = a.src_stride_bytes;
    o.n_src = a.n_src;
    o.T = a.T;
    o.d = a.d;
    o.query = a.queries;
    o.gain = a.gain;
    o.eps = a.eps;
    o.inv_d = a.inv_dh;
    o.dout = a.dout;
    o.dlse = a.dlse;
    o.dsrc = a.dsrc;
    o.dsrc_stride_bytes = a.dsrc_stride_bytes;
    o.accumulate = a.accumulate;
    o.ws = a.ws;
    o.nstages = ns;
    o.wait = a.wait;
    const int grid = (int)(a.T < dev->sms ? a.T : dev->sms);
    void *args[] = {&o};
    cudaError_t e = cudaLaunchKernel(kr.fn, dim3(grid), dim3(R1_NW * 32), args, smem, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "read_bwd one-query launch");
    *nparts = grid;
    return ATTNRES_OK;
}

// Workspace launch_read_bwd needs for these arguments: the larger of the
// kernel forms its query passes take.
attnres_status_t read_bwd_ws_need(int64_t n_src, int64_t T, int64_t d, int64_t H, int64_t n_q,
                                  attnres_dtype_t dt, const DeviceInfo *dev, const ReadBwdShape &sh, size_t *bytes) {
    const int64_t nq_last = n_q - (n_q - 1) / sh.nqc * sh.nqc;
    const int64_t nq_first = n_q < sh.nqc ? n_q : sh.nqc;
    const bool sp0 = read_bwd_split_applies(dt, n_src, nq_first, d, H);
    const bool sp1 = read_bwd_split_applies(dt, n_src, nq_last, d, H);
    size_t need = (!sp0 || !sp1) ? read_bwd_ws_bytes(dev->sms, sh, d) : 0;
    if (sp0 || sp1) {
        ReadBwdSplitShape ss;
        attnres_status_t st = read_bwd_split_shape(T, d, H, dev, &ss);
        if (st != ATTNRES_OK) return st;
        if (ss.total > need) need = ss.total;
    }
    *bytes = need;
    return ATTNRES_OK;
}

// One pass of nq queries in the two-kernel form: the coefficient kernel (one
// CTA per SM) writes every token's coefficients after the partials of U in
// the workspace, the apply kernel writes dv and the partials.
attnres_status_t launch_read_bwd_split_pass(const ReadBwdArgs &a, int nq, int64_t H, const ReadBwdSplitShape &ss,
                                            int sms, void *stream) {
    KernelRef kc, ka;
    if (!lookup_read_bwd_split(nq, a.d, &kc, &ka)) return ATTNRES_ERR_UNSUPPORTED;
    int occ = 0;
    attnres_status_t st = prepare_kernel(kc.fn, ss.smem, RC_NW * 32, &occ);
    if (st == ATTNRES_OK) st = prepare_kernel(ka.fn, RA_RING_BYTES, RA_THREADS, &occ);
    if (st != ATTNRES_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    float *coef = reinterpret_cast<float *>(reinterpret_cast<unsigned char *>(a.ws) + ss.off_coef);
    ReadBwdCoefArgs c;
    c.src = a.src;
    c.src_stride_bytes = a.src_stride_bytes;
    c.n_src = a.n_src;
    c.T = a.T;
    c.d = a.d;
    c.n_q = nq;
    c.H = (int)H;
    c.queries = a.queries;
    c.gain = a.gain;
    c.eps = a.eps;
    c.inv_dh = a.inv_dh;
    c.dout = a.dout;
    c.dlse = a.dlse;
    c.coef = coef;
    c.nstages = ss.nstages;
    c.pitch = ss.pitch;
    c.stage_bytes = ss.stage_bytes;
    c.wait = a.wait;
    const int grid = (int)(a.T < sms ? a.T : sms);
    void *cargs[] = {&c};
    cudaError_t e = cudaLaunchKernel(kc.fn, dim3(grid), dim3(RC_NW * 32), cargs, ss.smem, s);
    if (e != cudaSuccess) return cuda_fail(e, "read_bwd coefficient launch");
    ReadBwdApplyArgs p;
    p.src = a.src;
    p.src_stride_bytes = a.src_stride_bytes;
    p.n_src = a.n_src;
    p.T = a.T;
    p.d = a.d;
    p.H = (int)H;
    p.dh = (int)(a.d / H);
    p.n_q = nq;
    p.queries = a.queries;
    p.gain = a.gain;
    p.dout = a.dout;
    p.coef = coef;
    p.dsrc = a.dsrc;
    p.dsrc_stride_bytes = a.dsrc_stride_bytes;
    p.accumulate = a.accumulate;
    p.ws = a.ws;
    p.tpc = ss.tpc;
    void *pargs[] = {&p};
    e = cudaLaunchKernel(ka.fn, dim3((unsigned)(a.d / RA_W), (unsigned)ss.chunks), dim3(RA_THREADS), pargs,
                         RA_RING_BYTES, s);
    if (e != cudaSuccess) return cuda_fail(e, "read_bwd apply launch");
    return ATTNRES_OK;
}

attnres_status_t launch_read_bwd(const void *src, int64_t n_src, int64_t src_stride, int64_t T, int64_t d,
                                 int64_t H, attnres_dtype_t dt, const float *queries, int64_t n_q,
                                 const float *gain, float eps, const void *dout, const float *dlse, void *dsrc,
                                 int64_t dsrc_stride, int accumulate, float *dq, float *dgain, void *ws,
                                 size_t ws_bytes, void *stream, int max_nqc = 0) {
    attnres_status_t st = check_common(src, n_src, src_stride, T, d, dt, eps);
    if (st != ATTNRES_OK) return st;
    if (n_q < 1 || (accumulate != 0 && accumulate != 1)) return ATTNRES_ERR_INVALID_ARG;
    if (H < 1 || d % H != 0) return ATTNRES_ERR_INVALID_ARG;
    if (T > 0 && (!queries || !dout || !dsrc || !dq || !ws)) return ATTNRES_ERR_INVALID_ARG;
    if (dsrc_stride < T * d) return ATTNRES_ERR_INVALID_ARG;
    const size_t es = esize(dt);
    const size_t src_bytes = ((size_t)(n_src - 1) * (size_t)src_stride + (size_t)T * (size_t)d) * es;
    const size_t dsrc_bytes = ((size_t)(n_src - 1) * (size_t)dsrc_stride + (size_t)T * (size_t)d) * es;
    const size_t dout_bytes = (size_t)n_q * (size_t)T * (size_t)d * es;
    const size_t dq_bytes = (size_t)n_q * (size_t)d * sizeof(float);
    if (overlap(dsrc, dsrc_bytes, src, src_bytes) || overlap(dsrc, dsrc_bytes, dout, dout_bytes) ||
        overlap(ws, ws_bytes, src, src_bytes) || overlap(ws, ws_bytes, dsrc, dsrc_bytes) ||
        overlap(ws, ws_bytes, dout, dout_bytes) || overlap(dq, dq_bytes, ws, ws_bytes) ||
        (dgain && (overlap(dgain, (size_t)d * 4, ws, ws_bytes) || overlap(dgain, (size_t)d * 4, dq, dq_bytes))))
        return ATTNRES_ERR_INVALID_ARG;
    if (dlse && (H != 1 || overlap(dsrc, dsrc_bytes, dlse, (size_t)n_q * (size_t)T * 4)))
        return ATTNRES_ERR_INVALID_ARG;
    ReadBwdShape sh;
    st = read_bwd_shape(n_src, d, n_q, H, dt, &sh, max_nqc);
    if (st != ATTNRES_OK) return st;
    if (!aligned16(dout) || !aligned16(dsrc) || (dsrc_stride * (int64_t)es) % 16 != 0 || !aligned16(queries) ||
        (gain && !aligned16(gain)) || !aligned4(dq) || (dgain && !aligned4(dgain)) || !aligned16(ws) ||
        (dlse && !aligned4(dlse)))
        return ATTNRES_ERR_UNSUPPORTED;
    DeviceInfo *dev = nullptr;
    st = device_info(&dev);
    if (st != ATTNRES_OK) return st;
    if (T == 0) {
        // no tokens: the parameter gradients are zero, the sources have none
        cudaError_t e = dq ? cudaMemsetAsync(dq, 0, dq_bytes, static_cast<cudaStream_t>(stream)) : cudaSuccess;
        if (e == cudaSuccess && dgain) e = cudaMemsetAsync(dgain, 0, (size_t)d * 4, static_cast<cudaStream_t>(stream));
        return e == cudaSuccess ? ATTNRES_OK : cuda_fail(e, "cudaMemsetAsync");
    }
    size_t need = 0;
    st = read_bwd_ws_need(n_src, T, d, H, n_q, dt, dev, sh, &need);
    if (st != ATTNRES_OK) return st;
    if (ws_bytes < need) return ATTNRES_ERR_INVALID_ARG;
    // kernels of every pass (a last pass may take fewer queries): up to 2
    // queries one group, 3 or 4 two groups of two, or the two-kernel form
    KernelRef kr[2];
    bool split[2], one[2], plain[2];
    const int nq_last = (int)(n_q - (n_q - 1) / sh.nqc * sh.nqc);
    for (int v = 0; v < 2; ++v) {
        const int nq = v == 0 ? (int)(n_q < sh.nqc ? n_q : sh.nqc) : nq_last;
        split[v] = read_bwd_split_applies(dt, n_src, nq, d, H);
        one[v] = !split[v] && read_bwd_one_applies(dt, n_src, nq, d, H, src, src_stride);
        plain[v] = !split[v] && !one[v];
        if (!plain[v]) continue;
        const int dti = dt == ATTNRES_BF16 ? 1 : 0;
        const bool ok = nq > 2 ? lookup_read_bwd_qg(dti, sh.vpt, sh.mh, sh.hg, &kr[v])
                        : sh.mh ? lookup_read_bwd_mh(dti, nq, sh.ns, sh.vpt, sh.hg, &kr[v])
                                : lookup_read_bwd(dti, nq, sh.ns, sh.vpt, &kr[v]);
        if (!ok) return ATTNRES_ERR_UNSUPPORTED;
    }
    const uint32_t row_pitch = (uint32_t)((size_t)sh.tt * (size_t)d * es);
    const uint32_t stage_bytes = (uint32_t)(((size_t)(n_src + sh.nqc) * row_pitch + 127) / 128 * 128);
    size_t budget = kSmemBudget;
    if ((size_t)dev->smem_optin < budget) budget = (size_t)dev->smem_optin;
    size_t aux = 0;
    for (int v = 0; v < 2; ++v)
        if (plain[v] && kr[v].aux_smem > aux) aux = kr[v].aux_smem;
    if (budget <= aux) return ATTNRES_ERR_UNSUPPORTED;
    int nstages = (int)((budget - aux) / stage_bytes);
    if (nstages > RB_MAX_STAGES) nstages = RB_MAX_STAGES;
    if (nstages < 2 && (plain[0] || plain[1])) return ATTNRES_ERR_UNSUPPORTED;
    const size_t smem = (size_t)nstages * stage_bytes + aux;
    for (int v = 0; v < 2; ++v) {
        if (!plain[v]) continue;
        int occ = 0;
        st = prepare_kernel(kr[v].fn, smem, RB_THREADS, &occ);
        if (st != ATTNRES_OK) return st;
    }
    ReadBwdSplitShape ss;
    if (split[0] || split[1]) {
        st = read_bwd_split_shape(T, d, H, dev, &ss);
        if (st != ATTNRES_OK) return st;
        if (!aligned16(src) || (src_stride * (int64_t)es) % 16 != 0) return ATTNRES_ERR_UNSUPPORTED;
    }
    ReadBwdArgs a;
    a.src = static_cast<const unsigned char *>(src);
    a.src_stride_bytes = src_stride * (int64_t)es;
    a.n_src = (int)n_src;
    a.T = T;
    a.d = (int)d;
    a.nvec = (int)(d / epv(dt));
    a.gain = gain;
    a.eps = eps;
    a.dsrc = static_cast<unsigned char *>(dsrc);
    a.dsrc_stride_bytes = dsrc_stride * (int64_t)es;
    a.ws = static_cast<float *>(ws);
    a.tpr = sh.tpr;
    a.tt = sh.tt;
    a.nstages = nstages;
    a.stage_bytes = stage_bytes;
    a.row_pitch = row_pitch;
    a.ntiles = (T + sh.tt - 1) / sh.tt;
    a.vph = sh.vph;
    a.nheads = (int)H;
    a.inv_dh = 1.f / (float)(d / H);
    a.wait = wait_cfg(dev);
    const int grid = (int)(a.ntiles < dev->sms ? a.ntiles : dev->sms);
    // queries in passes of nqc: the source gradients and dgain add up over
    // the passes (each query's terms are independent of the others')
    for (int64_t q0 = 0; q0 < n_q; q0 += sh.nqc) {
        const int nq = (int)(n_q - q0 < sh.nqc ? n_q - q0 : sh.nqc);
        a.n_q = nq;
        a.queries = queries + q0 * d;
        a.dout = static_cast<const unsigned char *>(dout) + (size_t)q0 * (size_t)T * (size_t)d * es;
        a.dlse = dlse ? dlse + q0 * T : nullptr;
        a.accumulate = q0 == 0 ? accumulate : 1;
        const int pv = nq == (n_q < sh.nqc ? n_q : sh.nqc) ? 0 : 1;
        int nparts = grid * sh.tt;
        if (split[pv]) {
            st = launch_read_bwd_split_pass(a, nq, H, ss, dev->sms, stream);
            if (st != ATTNRES_OK) return st;
            nparts = ss.chunks;
        } else if (one[pv]) {
            st = launch_read_bwd_one_pass(a, dev, stream, &nparts);
            if (st != ATTNRES_OK) return st;
        } else {
            void *args[] = {&a};
            const void *fn = kr[nq == sh.nqc ? 0 : 1].fn;
            cudaError_t e =
                cudaLaunchKernel(fn, dim3(grid), dim3(RB_THREADS), args, smem, static_cast<cudaStream_t>(stream));
            if (e != cudaSuccess) return cuda_fail(e, "read_bwd launch");
        }
        ReadBwdFinishArgs f;
        f.ws = a.ws;
        f.nparts = nparts;
        f.n_q = nq;
        f.d = (int)d;
        f.queries = a.queries;
        f.gain = gain;
        f.dq = dq + q0 * d;
        f.dgain = dgain;
        f.accumulate_dgain = q0 > 0 ? 1 : 0;
        void *fargs[] = {&f};
        const int fgrid = (int)((d + 31) / 32);          // 32 channels per CTA
        cudaError_t e =
            cudaLaunchKernel(read_bwd_finish_fn(), dim3(fgrid), dim3(256), fargs, 0, static_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) return cuda_fail(e, "read_bwd finish launch");
    }
    return ATTNRES_OK;
}

// Backward of the phase-2 merge: tile shape, workspace and launch.
struct MergeBwdShape {
    int tpr, vpt, tt;
    int grid;
};

attnres_status_t merge_bwd_shape(int64_t T, int64_t d, attnres_dtype_t dt, const DeviceInfo *dev,
                                 MergeBwdShape *sh) {
    row_shape((int)(d / epv(dt)), &sh->tpr, &sh->vpt);
    if (sh->vpt > 4) return ATTNRES_ERR_UNSUPPORTED;
    sh->tt = MB_THREADS / sh->tpr;
    const int64_t ntiles = (T + sh->tt - 1) / sh->tt;
    const int64_t occ = sh->vpt <= 2 ? 2 : 1;
    const int64_t g = (int64_t)dev->sms * occ;
    sh->grid = (int)(ntiles < g ? (ntiles > 0 ? ntiles : 1) : g);
    return ATTNRES_OK;
}

size_t merge_bwd_ws_bytes(const MergeBwdShape &sh, int64_t d) {
    return (size_t)sh.grid * (size_t)sh.tt * (size_t)d * sizeof(float);
}

attnres_status_t launch_merge_bwd(const void *o, const float *lse, const void *partial, int64_t T, int64_t d,
                                  attnres_dtype_t dt, const float *query, const float *gain, float eps,
                                  const void *dh, void *d_o, float *d_lse, void *d_partial, int accumulate,
                                  float *dquery, float *dgain, void *ws, size_t ws_bytes, void *stream) {
    if (dt != ATTNRES_F32 && dt != ATTNRES_BF16) return ATTNRES_ERR_INVALID_ARG;
    if (T < 0 || d < 1 || !(eps >= 0.f) || std::isinf(eps) || (accumulate != 0 && accumulate != 1))
        return ATTNRES_ERR_INVALID_ARG;
    if (T > 0 && d > INT64_MAX / T) return ATTNRES_ERR_INVALID_ARG;
    if (T > 0 && (!o || !lse || !query || !dh || !d_o || !d_lse || !dquery)) return ATTNRES_ERR_INVALID_ARG;
    if (T > 0 && partial && (!d_partial || !ws)) return ATTNRES_ERR_INVALID_ARG;
    const size_t es = esize(dt);
    const size_t rb = (size_t)T * (size_t)d * es;
    const size_t lb = (size_t)T * 4;
    const void *ins[4] = {o, partial, dh, lse};
    const size_t insz[4] = {rb, rb, rb, lb};
    void *outs[3] = {d_o, d_partial, d_lse};
    const size_t outsz[3] = {rb, rb, lb};
    for (int i = 0; i < 3; ++i) {
        if (!outs[i]) continue;
        for (int j = 0; j < 4; ++j)
            if (ins[j] && overlap(outs[i], outsz[i], ins[j], insz[j])) return ATTNRES_ERR_INVALID_ARG;
        for (int j = i + 1; j < 3; ++j)
            if (outs[j] && overlap(outs[i], outsz[i], outs[j], outsz[j])) return ATTNRES_ERR_INVALID_ARG;
        if (ws && overlap(outs[i], outsz[i], ws, ws_bytes)) return ATTNRES_ERR_INVALID_ARG;
    }
    if (dgain && overlap(dgain, (size_t)d * 4, dquery, (size_t)d * 4)) return ATTNRES_ERR_INVALID_ARG;
    if (d % 8 != 0 || d > ((int64_t)1 << 20)) return ATTNRES_ERR_UNSUPPORTED;
    if (!aligned16(o) || (partial && !aligned16(partial)) || !aligned16(dh) || !aligned16(d_o) ||
        (d_partial && !aligned16(d_partial)) || !aligned4(lse) || !aligned4(d_lse) || !aligned16(query) ||
        (gain && !aligned16(gain)) || !aligned4(dquery) || (dgain && !aligned4(dgain)) || (ws && !aligned16(ws)))
        return ATTNRES_ERR_UNSUPPORTED;
    DeviceInfo *dev = nullptr;
    attnres_status_t st = device_info(&dev);
    if (st != ATTNRES_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (T == 0 || !partial) {
        // no tokens, or no partial (out = o): d_o = dh, dlse = 0, no parameter gradient
        cudaError_t e = cudaMemsetAsync(dquery, 0, (size_t)d * 4, s);
        if (e == cudaSuccess && dgain) e = cudaMemsetAsync(dgain, 0, (size_t)d * 4, s);
        if (e == cudaSuccess && T > 0) e = cudaMemcpyAsync(d_o, dh, rb, cudaMemcpyDeviceToDevice, s);
        if (e == cudaSuccess && T > 0) e = cudaMemsetAsync(d_lse, 0, lb, s);
        return e == cudaSuccess ? ATTNRES_OK : cuda_fail(e, "merge backward without a partial");
    }
    MergeBwdShape sh;
    st = merge_bwd_shape(T, d, dt, dev, &sh);
    if (st != ATTNRES_OK) return st;
    if (ws_bytes < merge_bwd_ws_bytes(sh, d)) return ATTNRES_ERR_INVALID_ARG;
    KernelRef kr;
    if (!lookup_merge_bwd(dt == ATTNRES_BF16 ? 1 : 0, sh.vpt, &kr)) return ATTNRES_ERR_UNSUPPORTED;
    MergeBwdArgs a;
    a.o = static_cast<const unsigned char *>(o);
    a.lse = lse;
    a.partial = static_cast<const unsigned char *>(partial);
    a.dh = static_cast<const unsigned char *>(dh);
    a.T = T;
    a.d = (int)d;
    a.nvec = (int)(d / epv(dt));
    a.query = query;
    a.gain = gain;
    a.eps = eps;
    a.d_o = static_cast<unsigned char *>(d_o);
    a.d_lse = d_lse;
    a.d_partial = static_cast<unsigned char *>(d_partial);
    a.accumulate = accumulate;
    a.ws = static_cast<float *>(ws);
    a.tpr = sh.tpr;
    a.tt = sh.tt;
    a.ntiles = (T + sh.tt - 1) / sh.tt;
    void *args[] = {&a};
    cudaError_t e = cudaLaunchKernel(kr.fn, dim3(sh.grid), dim3(MB_THREADS), args, 0, s);
    if (e != cudaSuccess) return cuda_fail(e, "merge backward launch");
    ReadBwdFinishArgs f;
    f.ws = a.ws;
    f.nparts = sh.grid * sh.tt;
    f.n_q = 1;
    f.d = (int)d;
    f.queries = query;
    f.gain = gain;
    f.dq = dquery;
    f.dgain = dgain;
    f.accumulate_dgain = 0;
    void *fargs[] = {&f};
    e = cudaLaunchKernel(read_bwd_finish_fn(), dim3((unsigned)((d + 31) / 32)), dim3(256), fargs, 0, s);
    if (e != cudaSuccess) return cuda_fail(e, "merge backward finish launch");
    return ATTNRES_OK;
}

// ------------------------------------------------ read backward, > 16 sources
// The sources in chunks of 8: each chunk's read state (o_c, lse_c) is
// recomputed with the forward read kernels, the backward of the states'
// online-softmax merge gives each chunk's d o_c and d lse_c
// (state_merge_bwd.cu), and each chunk runs the read backward with its lse
// gradient.  The chunks' query and gain gradients are summed in chunk order.
constexpr int64_t kReadBwdChunk = 8;        // sources per chunk
constexpr int64_t kReadBwdMaxChunks = 32;   // merge kernel limit: 256 sources

struct ReadBwdManyPlan {
    int64_t C;
    size_t rb_bytes, off_o, off_lse, off_do, off_dlse, off_rb, off_dq, off_dg, total;
};

attnres_status_t read_bwd_many_plan(int64_t n_src, int64_t T, int64_t d, int64_t n_q, attnres_dtype_t dt,
                                    const DeviceInfo *dev, ReadBwdManyPlan *p) {
    p->C = (n_src + kReadBwdChunk - 1) / kReadBwdChunk;
    if (p->C > kReadBwdMaxChunks) return ATTNRES_ERR_UNSUPPORTED;
    // the largest workspace over the chunk sizes (a short last chunk may tile wider)
    p->rb_bytes = 0;
    const int64_t sizes[2] = {kReadBwdChunk, n_src - (p->C - 1) * kReadBwdChunk};
    for (int64_t nc : sizes) {
        ReadBwdShape sh;
        attnres_status_t st = read_bwd_shape(nc, d, n_q, 1, dt, &sh);
        if (st != ATTNRES_OK) return st;
        size_t b = 0;
        st = read_bwd_ws_need(nc, T, d, 1, n_q, dt, dev, sh, &b);
        if (st != ATTNRES_OK) return st;
        if (b > p->rb_bytes) p->rb_bytes = b;
    }
    const size_t es = esize(dt);
    const size_t states = (size_t)p->C * (size_t)n_q * (size_t)T;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off += (bytes + 255) / 256 * 256;
        return at;
    };
    p->off_o = take(states * (size_t)d * es);
    p->off_lse = take(states * 4);
    p->off_do = take(states * (size_t)d * es);
    p->off_dlse = take(states * 4);
    p->off_rb = take(p->rb_bytes);
    p->off_dq = take((size_t)n_q * (size_t)d * 4);
    p->off_dg = take((size_t)d * 4);
    p->total = off;
    return ATTNRES_OK;
}

// One query over 17..64 bf16 sources at d = 2048 or 4096 takes the
// two-kernel form (read_bwd_many.cuh) instead of the chunked chain (debug
// kernel variant 1 keeps the chain).
bool read_bwd_many_split_applies(attnres_dtype_t dt, int64_t n_src, int64_t n_q, int64_t d) {
    if (g_kernel_variant.load() == 1) return false;
    return dt == ATTNRES_BF16 && n_q == 1 && n_src > 16 && n_src <= 8 * RM_MAXC && (d == 2048 || d == 4096);
}

struct ReadBwdManySplitShape {
    int C = 0;               // chunks of 8 sources
    int chunks = 0;          // apply CTAs along the tokens (partials of U)
    int64_t tpc = 0;         // tokens per apply CTA
    int nstages = 0;         // half-row stages of the coefficient kernel
    uint32_t pitch = 0, stage_bytes = 0;
    size_t smem = 0;
    size_t off_coef = 0;     // coefficients after the partials of U
    size_t total = 0;
};

attnres_status_t read_bwd_many_split_shape(int64_t n_src, int64_t T, int64_t d, const DeviceInfo *dev,
                                           ReadBwdManySplitShape *sh) {
    KernelRef kc, ka;
    if (!lookup_read_bwd_many((int)d, &kc, &ka)) return ATTNRES_ERR_UNSUPPORTED;
    sh->C = (int)((n_src + 7) / 8);
    sh->pitch = (uint32_t)d + 16;                 // half a row of bf16 (d bytes), padded
    sh->stage_bytes = (uint32_t)RM_ROWS * sh->pitch;
    size_t budget = kSmemBudget;
    if ((size_t)dev->smem_optin < budget) budget = (size_t)dev->smem_optin;
    if (budget <= RM_AUX_BYTES) return ATTNRES_ERR_UNSUPPORTED;
    int ns = (int)((budget - RM_AUX_BYTES) / sh->stage_bytes);
    if (ns > RC_MAX_STAGES) ns = RC_MAX_STAGES;
    if (ns < 2) return ATTNRES_ERR_UNSUPPORTED;
    sh->nstages = ns;
    sh->smem = (size_t)ns * sh->stage_bytes + RM_AUX_BYTES;
    int occ = 0;
    attnres_status_t st = prepare_kernel(ka.fn, RM_RING_BYTES, RA_THREADS, &occ);
    if (st != ATTNRES_OK) return st;
    // one wave of apply CTAs: d / 1024 channel slices times token ranges
    const int64_t slices = d / RA_W;
    int64_t chunks = ((int64_t)occ * dev->sms + slices - 1) / slices;
    if (chunks > T) chunks = T;
    if (chunks < 1) chunks = 1;
    sh->tpc = (T + chunks - 1) / chunks;
    sh->chunks = (int)(T > 0 ? (T + sh->tpc - 1) / sh->tpc : 0);
    const size_t ws_u = ((size_t)sh->chunks * (size_t)d * sizeof(float) + 255) / 256 * 256;
    sh->off_coef = ws_u;
    sh->total = ws_u + (size_t)T * (size_t)sh->C * RM_NV * sizeof(float);
    return ATTNRES_OK;
}

attnres_status_t launch_read_bwd_many(const void *src, int64_t n_src, int64_t src_stride, int64_t T, int64_t d,
                                      attnres_dtype_t dt, const float *queries, int64_t n_q, const float *gain,
                                      float eps, const void *dout, const float *dlse, void *dsrc,
                                      int64_t dsrc_stride, int accumulate, float *dq, float *dgain, void *ws,
                                      size_t ws_bytes, void *stream) {
    attnres_status_t st = check_common(src, n_src, src_stride, T, d, dt, eps);
    if (st != ATTNRES_OK) return st;
    if (n_q < 1 || (accumulate != 0 && accumulate != 1)) return ATTNRES_ERR_INVALID_ARG;
    if (T > 0 && (!queries || !dout || !dsrc || !dq || !ws)) return ATTNRES_ERR_INVALID_ARG;
    if (dsrc_stride < T * d) return ATTNRES_ERR_INVALID_ARG;
    if (n_q > 8 || (n_src + kReadBwdChunk - 1) / kReadBwdChunk > kReadBwdMaxChunks) return ATTNRES_ERR_UNSUPPORTED;
    const size_t es = esize(dt);
    const size_t src_bytes = ((size_t)(n_src - 1) * (size_t)src_stride + (size_t)T * (size_t)d) * es;
    const size_t dsrc_bytes = ((size_t)(n_src - 1) * (size_t)dsrc_stride + (size_t)T * (size_t)d) * es;
    const size_t dout_bytes = (size_t)n_q * (size_t)T * (size_t)d * es;
    const size_t dq_bytes = (size_t)n_q * (size_t)d * sizeof(float);
    if (overlap(dsrc, dsrc_bytes, src, src_bytes) || overlap(dsrc, dsrc_bytes, dout, dout_bytes) ||
        overlap(ws, ws_bytes, src, src_bytes) || overlap(ws, ws_bytes, dsrc, dsrc_bytes) ||
        overlap(ws, ws_bytes, dout, dout_bytes) || overlap(dq, dq_bytes, ws, ws_bytes) ||
        (dgain && (overlap(dgain, (size_t)d * 4, ws, ws_bytes) || overlap(dgain, (size_t)d * 4, dq, dq_bytes))) ||
        (dlse && overlap(dsrc, dsrc_bytes, dlse, (size_t)n_q * (size_t)T * 4)))
        return ATTNRES_ERR_INVALID_ARG;
    DeviceInfo *dev = nullptr;
    st = device_info(&dev);
    if (st != ATTNRES_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (read_bwd_many_split_applies(dt, n_src, n_q, d)) {
        ReadBwdManySplitShape sh;
        st = read_bwd_many_split_shape(n_src, T, d, dev, &sh);
        if (st != ATTNRES_OK) return st;
        if (T == 0) {
            cudaError_t e = cudaMemsetAsync(dq, 0, dq_bytes, s);
            if (e == cudaSuccess && dgain) e = cudaMemsetAsync(dgain, 0, (size_t)d * 4, s);
            return e == cudaSuccess ? ATTNRES_OK : cuda_fail(e, "cudaMemsetAsync");
        }
        if (ws_bytes < sh.total) return ATTNRES_ERR_INVALID_ARG;
        if (!aligned16(src) || (src_stride * (int64_t)es) % 16 != 0 || !aligned16(dout) || !aligned16(dsrc) ||
            (dsrc_stride * (int64_t)es) % 16 != 0 || !aligned16(queries) || (gain && !aligned16(gain)) ||
            !aligned4(dq) || (dgain && !aligned4(dgain)) || !aligned16(ws) || (dlse && !aligned4(dlse)))
            return ATTNRES_ERR_UNSUPPORTED;
        KernelRef kc, ka;
        if (!lookup_read_bwd_many((int)d, &kc, &ka)) return ATTNRES_ERR_UNSUPPORTED;
        int occ = 0;
        st = prepare_kernel(kc.fn, sh.smem, RC_NW * 32, &occ);
        if (st != ATTNRES_OK) return st;
        float *coef = reinterpret_cast<float *>(static_cast<unsigned char *>(ws) + sh.off_coef);
        ReadBwdCoefManyArgs c;
        c.src = static_cast<const unsigned char *>(src);
        c.src_stride_bytes = src_stride * (int64_t)es;
        c.n_src = (int)n_src;
        c.C = sh.C;
        c.T = T;
        c.d = (int)d;
        c.query = queries;
        c.gain = gain;
        c.eps = eps;
        c.inv_d = 1.f / (float)d;
        c.dout = static_cast<const unsigned char *>(dout);
        c.dlse = dlse;
        c.coef = coef;
        c.nstages = sh.nstages;
        c.pitch = sh.pitch;
        c.stage_bytes = sh.stage_bytes;
        c.wait = wait_cfg(dev);
        const int grid = (int)(T < dev->sms ? T : dev->sms);
        void *cargs[] = {&c};
        cudaError_t e = cudaLaunchKernel(kc.fn, dim3(grid), dim3(RC_NW * 32), cargs, sh.smem, s);
        if (e != cudaSuccess) return cuda_fail(e, "read_bwd many-source coefficient launch");
        ReadBwdApplyManyArgs p;
        p.src = c.src;
        p.src_stride_bytes = c.src_stride_bytes;
        p.n_src = (int)n_src;
        p.C = sh.C;
        p.T = T;
        p.d = (int)d;
        p.query = queries;
        p.gain = gain;
        p.dout = c.dout;
        p.coef = coef;
        p.dsrc = static_cast<unsigned char *>(dsrc);
        p.dsrc_stride_bytes = dsrc_stride * (int64_t)es;
        p.accumulate = accumulate;
        p.ws = static_cast<float *>(ws);
        p.tpc = sh.tpc;
        void *pargs[] = {&p};
        e = cudaLaunchKernel(ka.fn, dim3((unsigned)(d / RA_W), (unsigned)sh.chunks), dim3(RA_THREADS), pargs,
                             RM_RING_BYTES, s);
        if (e != cudaSuccess) return cuda_fail(e, "read_bwd many-source apply launch");
        ReadBwdFinishArgs f;
        f.ws = p.ws;
        f.nparts = sh.chunks;
        f.n_q = 1;
        f.d = (int)d;
        f.queries = queries;
        f.gain = gain;
        f.dq = dq;
        f.dgain = dgain;
        f.accumulate_dgain = 0;
        void *fargs[] = {&f};
        e = cudaLaunchKernel(read_bwd_finish_fn(), dim3((unsigned)((d + 31) / 32)), dim3(256), fargs, 0, s);
        if (e != cudaSuccess) return cuda_fail(e, "read_bwd finish launch");
        return ATTNRES_OK;
    }
    ReadBwdManyPlan p;
    st = read_bwd_many_plan(n_src, T, d, n_q, dt, dev, &p);
    if (st != ATTNRES_OK) return st;
    if (T == 0) {
        cudaError_t e = cudaMemsetAsync(dq, 0, dq_bytes, s);
        if (e == cudaSuccess && dgain) e = cudaMemsetAsync(dgain, 0, (size_t)d * 4, s);
        return e == cudaSuccess ? ATTNRES_OK : cuda_fail(e, "cudaMemsetAsync");
    }
    if (ws_bytes < p.total) return ATTNRES_ERR_INVALID_ARG;
    unsigned char *w = static_cast<unsigned char *>(ws);
    const size_t state_bytes = (size_t)n_q * (size_t)T * (size_t)d * es;   // one chunk's o
    const unsigned char *sb = static_cast<const unsigned char *>(src);
    unsigned char *db = static_cast<unsigned char *>(dsrc);
    // each chunk's read state
    for (int64_t c = 0; c < p.C; ++c) {
        const int64_t nc = c + 1 < p.C ? kReadBwdChunk : n_src - c * kReadBwdChunk;
        st = launch_depth_read(sb + (size_t)(c * kReadBwdChunk) * (size_t)src_stride * es, nc, src_stride, T, d, 1,
                               dt, queries, n_q, gain, eps, w + p.off_o + (size_t)c * state_bytes,
                               reinterpret_cast<float *>(w + p.off_lse) + (size_t)c * n_q * T, stream);
        if (st != ATTNRES_OK) return st;
    }
    // the merge's backward: each chunk's d o_c and d lse_c
    StateMergeBwdArgs m;
    m.o = w + p.off_o;
    m.lse = reinterpret_cast<const float *>(w + p.off_lse);
    m.dh = static_cast<const unsigned char *>(dout);
    m.dlse = dlse;
    m.d_o = w + p.off_do;
    m.d_lse = reinterpret_cast<float *>(w + p.off_dlse);
    m.C = (int)p.C;
    m.rows = n_q * T;
    m.d = (int)d;
    cudaError_t e = launch_state_merge_bwd(dt == ATTNRES_BF16 ? 1 : 0, m, dev->sms, stream);
    if (e != cudaSuccess) return cuda_fail(e, "state merge backward launch");
    // each chunk's read backward; its query and gain gradients summed in chunk order
    float *dq_c = reinterpret_cast<float *>(w + p.off_dq);
    float *dg_c = dgain ? reinterpret_cast<float *>(w + p.off_dg) : nullptr;
    for (int64_t c = 0; c < p.C; ++c) {
        const int64_t nc = c + 1 < p.C ? kReadBwdChunk : n_src - c * kReadBwdChunk;
        st = launch_read_bwd(sb + (size_t)(c * kReadBwdChunk) * (size_t)src_stride * es, nc, src_stride, T, d, 1, dt,
                             queries, n_q, gain, eps, w + p.off_do + (size_t)c * state_bytes,
                             reinterpret_cast<const float *>(w + p.off_dlse) + (size_t)c * n_q * T,
                             db + (size_t)(c * kReadBwdChunk) * (size_t)dsrc_stride * es, dsrc_stride, accumulate,
                             dq_c, dg_c, w + p.off_rb, p.rb_bytes, stream);
        if (st != ATTNRES_OK) return st;
        e = msar_bwd_sum(dq_c, 1, n_q * d, dq, c > 0 ? 1 : 0, stream);
        if (e == cudaSuccess && dgain) e = msar_bwd_sum(dg_c, 1, d, dgain, c > 0 ? 1 : 0, stream);
        if (e != cudaSuccess) return cuda_fail(e, "read backward chunk sums launch");
    }
    return ATTNRES_OK;
}

// Scratch of the no-allocation backward: a fixed device array in the
// library's own image (8 MB: every one-query backward and two-query ones up
// to d of about 6.7 K on 152 SMs; one backward at a time per device may use
// it), its address looked up once per device.
constexpr size_t kBwdScratchFloats = (size_t)2 << 20;
static __device__ __align__(256) float g_bwd_scratch[kBwdScratchFloats];

struct ScratchInfo {
    std::once_flag once;
    cudaError_t err = cudaSuccess;
    void *ptr = nullptr;
};
ScratchInfo g_scratch[kMaxDevices];

attnres_status_t bwd_scratch(void **ptr) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return ATTNRES_ERR_UNSUPPORTED;
    ScratchInfo &si = g_scratch[dev];
    std::call_once(si.once, [&] { si.err = cudaGetSymbolAddress(&si.ptr, g_bwd_scratch); });
    if (si.err != cudaSuccess) return cuda_fail(si.err, "cudaGetSymbolAddress");
    *ptr = si.ptr;
    return ATTNRES_OK;
}

// Shared launch path of the MSAR read: src holds t_prev history rows and
// then the T rows whose outputs are written.
attnres_status_t launch_msar_read(const void *src, int64_t n_src, int64_t src_stride, int64_t t_prev, int64_t T,
                                  int64_t d, attnres_dtype_t dt, int64_t m, const int32_t *ksizes,
                                  const float *conv_w, const float *queries, const float *gain, float eps,
                                  const float *mix_gain, const float *mix_w, float mix_eps, void *out,
                                  void *stream, int64_t conv_src_stride = 0) {
    if (T < 0 || t_prev > INT64_MAX - T) return ATTNRES_ERR_INVALID_ARG;
    const int64_t rows = t_prev + T;                      // source rows per source
    attnres_status_t st = check_common(src, n_src, src_stride, rows, d, dt, eps);
    if (st != ATTNRES_OK) return st;
    if (m < 1 || !(mix_eps >= 0.f) || std::isinf(mix_eps)) return ATTNRES_ERR_INVALID_ARG;
    if (T == 0) return ATTNRES_OK;
    if (!ksizes || !conv_w || !queries || !mix_w || !out) return ATTNRES_ERR_INVALID_ARG;
    for (int64_t r = 0; r + 1 < m; ++r)
        if (ksizes[r] < 1) return ATTNRES_ERR_INVALID_ARG;
    if (conv_src_stride != 0) {
        // each source's kernels must not overlap the next source's
        int64_t ktot = 0;
        for (int64_t r = 0; r + 1 < m; ++r) ktot += ksizes[r];
        if (conv_src_stride < 0 || (n_src > 1 && conv_src_stride < d * ktot)) return ATTNRES_ERR_INVALID_ARG;
    }
    const size_t es = esize(dt);
    const size_t src_bytes = ((size_t)(n_src - 1) * (size_t)src_stride + (size_t)rows * (size_t)d) * es;
    if (overlap(out, (size_t)T * (size_t)d * es, src, src_bytes)) return ATTNRES_ERR_INVALID_ARG;
    if (m != 4) return ATTNRES_ERR_UNSUPPORTED;
    for (int r = 0; r < 3; ++r)
        if (ksizes[r] > MSAR_KMAX) return ATTNRES_ERR_UNSUPPORTED;
    // per-source kernels start 16-byte aligned (they are read with 16-byte loads)
    if (conv_src_stride != 0 && n_src > 1 && conv_src_stride % 4 != 0) return ATTNRES_ERR_UNSUPPORTED;
    if (!aligned16(out) || !aligned16(queries) || !aligned16(conv_w) || !aligned16(mix_w) ||
        (gain && !aligned16(gain)) || (mix_gain && !aligned16(mix_gain)))
        return ATTNRES_ERR_UNSUPPORTED;
    DeviceInfo *dev = nullptr;
    st = device_info(&dev);
    if (st != ATTNRES_OK) return st;
    MsarArgs a;
    a.src = static_cast<const unsigned char *>(src);
    a.src_stride_bytes = src_stride * (int64_t)es;
    a.n_src = (int)n_src;
    a.T = T;
    a.t_prev = t_prev;
    a.d = (int)d;
    for (int r = 0; r < 3; ++r) a.k[r] = ksizes[r];
    a.conv_w = conv_w;
    a.conv_src_stride = conv_src_stride;
    a.queries = queries;
    a.gain = gain;
    a.eps = eps;
    a.mix_gain = mix_gain;
    a.mix_w = mix_w;
    a.mix_eps = mix_eps;
    a.out = static_cast<unsigned char *>(out);
    a.wait = wait_cfg(dev);
    const int dti = dt == ATTNRES_BF16 ? 1 : 0;
    // the tile-batched kernel where it applies (variant 1 keeps the per-token one)
    if (g_kernel_variant.load() != 1 && msar_tile_applies(dti, a)) {
        st = launch_msar_tile(a, dev->sms, stream, t_last_err, sizeof(t_last_err));
        if (st != ATTNRES_ERR_UNSUPPORTED) return st;
    }
    return launch_msar(dti, a, dev->sms, stream, t_last_err, sizeof(t_last_err));
}

// MSAR in the two-phase Block schedule.  Kernel sizes as the one-shot read.
attnres_status_t check_msar_kernels(int64_t m, const int32_t *ksizes) {
    if (m < 1) return ATTNRES_ERR_INVALID_ARG;
    if (!ksizes) return ATTNRES_ERR_INVALID_ARG;
    for (int64_t r = 0; r + 1 < m; ++r)
        if (ksizes[r] < 1) return ATTNRES_ERR_INVALID_ARG;
    if (m != 4) return ATTNRES_ERR_UNSUPPORTED;
    for (int r = 0; r < 3; ++r)
        if (ksizes[r] > MSAR_KMAX) return ATTNRES_ERR_UNSUPPORTED;
    return ATTNRES_OK;
}

attnres_status_t launch_msar_phase1_host(const void *src, int64_t n_src, int64_t src_stride, int64_t T, int64_t d,
                                         attnres_dtype_t dt, int64_t m, const int32_t *ksizes,
                                         const float *conv_w, const float *queries, int64_t S, const float *gain,
                                         float eps, void *o, float *lse, void *stream) {
    attnres_status_t st = check_common(src, n_src, src_stride, T, d, dt, eps);
    if (st != ATTNRES_OK) return st;
    if (S < 1) return ATTNRES_ERR_INVALID_ARG;
    if (T == 0) return ATTNRES_OK;
    if (!conv_w || !queries || !o || !lse) return ATTNRES_ERR_INVALID_ARG;
    st = check_msar_kernels(m, ksizes);
    if (st != ATTNRES_OK) return st;
    const size_t es = esize(dt);
    const size_t src_bytes = ((size_t)(n_src - 1) * (size_t)src_stride + (size_t)T * (size_t)d) * es;
    const size_t o_bytes = (size_t)S * 4 * (size_t)T * (size_t)d * es;
    const size_t lse_bytes = (size_t)S * 4 * (size_t)T * sizeof(float);
    if (overlap(o, o_bytes, src, src_bytes) || overlap(lse, lse_bytes, src, src_bytes) ||
        overlap(lse, lse_bytes, o, o_bytes))
        return ATTNRES_ERR_INVALID_ARG;
    if (n_src > MSAR_SMAX) return ATTNRES_ERR_UNSUPPORTED;
    if (!aligned16(o) || !aligned4(lse) || !aligned16(queries) || !aligned16(conv_w) || (gain && !aligned16(gain)))
        return ATTNRES_ERR_UNSUPPORTED;
    DeviceInfo *dev = nullptr;
    st = device_info(&dev);
    if (st != ATTNRES_OK) return st;
    // layers in groups of up to MSAR_P1_MAXL (each group expands the sources again)
    for (int64_t l0 = 0; l0 < S; l0 += MSAR_P1_MAXL) {
        MsarP1Args a;
        a.src = static_cast<const unsigned char *>(src);
        a.src_stride_bytes = src_stride * (int64_t)es;
        a.n_src = (int)n_src;
        a.T = T;
        a.d = (int)d;
        for (int r = 0; r < 3; ++r) a.k[r] = ksizes[r];
        a.conv_w = conv_w;
        a.queries = queries + l0 * 4 * d;
        a.n_layers = (int)(S - l0 < MSAR_P1_MAXL ? S - l0 : MSAR_P1_MAXL);
        a.gain = gain;
        a.eps = eps;
        a.o = static_cast<unsigned char *>(o) + (size_t)l0 * 4 * (size_t)T * (size_t)d * es;
        a.lse = lse + l0 * 4 * T;
        a.wait = wait_cfg(dev);
        st = launch_msar_phase1(dt == ATTNRES_BF16 ? 1 : 0, a, dev->sms, stream, t_last_err, sizeof(t_last_err));
        if (st != ATTNRES_OK) return st;
    }
    return ATTNRES_OK;
}

attnres_status_t launch_msar_phase2_host(const void *o, const float *lse, const void *partial, int64_t T, int64_t d,
                                         attnres_dtype_t dt, int64_t m, const int32_t *ksizes,
                                         const float *conv_w, const float *query, const float *gain, float eps,
                                         const float *mix_gain, const float *mix_w, float mix_eps, void *out,
                                         void *stream) {
    if (dt != ATTNRES_F32 && dt != ATTNRES_BF16) return ATTNRES_ERR_INVALID_ARG;
    if (T < 0 || d < 1 || !(eps >= 0.f) || std::isinf(eps) || !(mix_eps >= 0.f) || std::isinf(mix_eps))
        return ATTNRES_ERR_INVALID_ARG;
    if (T > 0 && d > INT64_MAX / (4 * T)) return ATTNRES_ERR_INVALID_ARG;
    if (T == 0) return ATTNRES_OK;
    if (!o || !lse || !conv_w || !query || !mix_w || !out) return ATTNRES_ERR_INVALID_ARG;
    attnres_status_t st = check_msar_kernels(m, ksizes);
    if (st != ATTNRES_OK) return st;
    const size_t es = esize(dt);
    const size_t row_bytes = (size_t)T * (size_t)d * es;
    if (overlap(out, row_bytes, o, 4 * row_bytes) || overlap(out, row_bytes, lse, (size_t)4 * T * 4) ||
        (partial && overlap(out, row_bytes, partial, row_bytes)))
        return ATTNRES_ERR_INVALID_ARG;
    if (d % 8 != 0 || d > ((int64_t)1 << 20)) return ATTNRES_ERR_UNSUPPORTED;
    if (!aligned16(o) || !aligned4(lse) || (partial && !aligned16(partial)) || !aligned16(out) ||
        !aligned16(query) || !aligned16(conv_w) || !aligned16(mix_w) || (gain && !aligned16(gain)) ||
        (mix_gain && !aligned16(mix_gain)))
        return ATTNRES_ERR_UNSUPPORTED;
    DeviceInfo *dev = nullptr;
    st = device_info(&dev);
    if (st != ATTNRES_OK) return st;
    MsarP2Args a;
    a.o = static_cast<const unsigned char *>(o);
    a.lse = lse;
    a.partial = static_cast<const unsigned char *>(partial);
    a.T = T;
    a.d = (int)d;
    for (int r = 0; r < 3; ++r) a.k[r] = ksizes[r];
    a.conv_w = conv_w;
    a.query = query;
    a.gain = gain;
    a.eps = eps;
    a.mix_gain = mix_gain;
    a.mix_w = mix_w;
    a.mix_eps = mix_eps;
    a.out = static_cast<unsigned char *>(out);
    a.wait = wait_cfg(dev);
    a.tt = 0;
    return launch_msar_phase2(dt == ATTNRES_BF16 ? 1 : 0, a, dev->sms, stream, t_last_err, sizeof(t_last_err));
}

// Tokens per CTA of the MSAR mixer kernels: 128, or more where the token
// chunks would exceed the grid's y limit (65535).
int64_t mix_tokens_per_cta(int64_t T) {
    const int64_t need = (T + 65534) / 65535;
    return need > 128 ? need : 128;
}

// MSAR backward: chunking and workspace layout.  Each region starts on a
// 256-byte boundary of the workspace.
struct MsarBwdPlan {
    int64_t tc, chunks, tc_s, tc_m;
    int nsl;
    ReadBwdShape rb;
    size_t rb_bytes;
    size_t off_u, off_z, off_dz, off_du, off_rb, off_dg, off_dq, off_part, off_e, off_mp, off_a, off_cp, total;
};

attnres_status_t msar_bwd_plan(int64_t n_src, int64_t T, int64_t d, attnres_dtype_t dt, const int32_t *ksizes,
                               const DeviceInfo *dev, MsarBwdPlan *p) {
    if (d != 1024 && d != 2048 && d != 4096) return ATTNRES_ERR_UNSUPPORTED;
    if (n_src > 16) return ATTNRES_ERR_UNSUPPORTED;
    attnres_status_t st = read_bwd_shape(n_src, d, 1, 1, dt, &p->rb);
    if (st != ATTNRES_OK) return st;
    p->rb_bytes = read_bwd_ws_bytes(dev->sms, p->rb, d);
    // token chunks: the conv backward and A's partials in at most 64 chunks
    // of at least 32 tokens; the streams kernel in chunks of T/128 (at least
    // 32); the mixer over d/1024 channel slices, mix_tokens_per_cta(T)
    // tokens per CTA (128, or more so that the token chunks stay within the
    // grid's y limit of 65535)
    p->tc = (T + 63) / 64;
    if (p->tc < 32) p->tc = 32;
    p->chunks = T > 0 ? (T + p->tc - 1) / p->tc : 0;
    p->tc_s = (T + 127) / 128;
    if (p->tc_s < 32) p->tc_s = 32;
    p->tc_m = mix_tokens_per_cta(T);
    p->nsl = (int)(d / 1024);
    const int64_t ktot = (int64_t)ksizes[0] + ksizes[1] + ksizes[2];
    const size_t es = esize(dt);
    const size_t row = (size_t)T * (size_t)d * es;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off += (bytes + 255) / 256 * 256;
        return at;
    };
    p->off_u = take(3 * (size_t)n_src * row);
    p->off_z = take(4 * row);
    p->off_dz = take(4 * row);
    p->off_du = take(4 * (size_t)n_src * row);
    p->off_rb = take(p->rb_bytes);
    p->off_dg = take(4 * (size_t)d * 4);
    p->off_dq = take(4 * (size_t)d * 4);
    p->off_part = take((size_t)T * (size_t)p->nsl * 9 * 4);
    p->off_e = take((size_t)T * 4 * 4);
    p->off_mp = take((size_t)p->chunks * 16 * (size_t)d * 4);
    p->off_a = take(16 * (size_t)d * 4);
    p->off_cp = take((size_t)p->chunks * (size_t)n_src * (size_t)ktot * (size_t)d * 4);
    p->total = off;
    return ATTNRES_OK;
}

// Backward of the MSAR read (msar_expand_fwd), as a chain of steps in the
// caller's workspace: the streams, the per-stream reads Z^(r), the mixer's
// backward, the per-stream read backward, and the causal convolutions'
// transpose.  A chunk of a longer sequence (msar_expand_bwd_chunk): src and
// dsrc start t_prev history rows before the chunk's T rows; the history rows
// feed the chunk's streams and kernel gradients, and get the chunk's share of
// their gradient added into dsrc; with accumulate the parameter gradients are
// added into their outputs.
attnres_status_t launch_msar_bwd(const void *src, int64_t n_src, int64_t src_stride, int64_t T, int64_t d,
                                 attnres_dtype_t dt, int64_t m, const int32_t *ksizes, const float *conv_w,
                                 const float *queries, const float *gain, float eps, const float *mix_gain,
                                 const float *mix_w, float mix_eps, const void *dh, void *dsrc,
                                 int64_t dsrc_stride, float *dconv_w, float *dqueries, float *dgain,
                                 float *dmix_gain, float *dmix_w, void *ws, size_t ws_bytes, void *stream,
                                 int64_t conv_src_stride = 0, int64_t t_prev = 0, int accumulate = 0) {
    if (T < 0 || t_prev < 0 || t_prev > INT64_MAX - T || (accumulate != 0 && accumulate != 1))
        return ATTNRES_ERR_INVALID_ARG;
    const int64_t rows = t_prev + T;                     // source rows per source, history included
    attnres_status_t st = check_common(src, n_src, src_stride, rows, d, dt, eps);
    if (st != ATTNRES_OK) return st;
    if (!(mix_eps >= 0.f) || std::isinf(mix_eps)) return ATTNRES_ERR_INVALID_ARG;
    st = check_msar_kernels(m, ksizes);
    if (st != ATTNRES_OK) return st;
    if (!conv_w || !queries || !mix_w || !dconv_w || !dqueries || !dmix_w) return ATTNRES_ERR_INVALID_ARG;
    if (T > 0 && (!dh || !dsrc || !ws)) return ATTNRES_ERR_INVALID_ARG;
    if (dsrc_stride < rows * d) return ATTNRES_ERR_INVALID_ARG;
    const int64_t ktot = (int64_t)ksizes[0] + ksizes[1] + ksizes[2];
    // per-source kernels: each source's set must not overlap the next one's
    if (conv_src_stride < 0 || (conv_src_stride > 0 && n_src > 1 && conv_src_stride < d * ktot))
        return ATTNRES_ERR_INVALID_ARG;
    const int64_t n_sets = conv_src_stride > 0 ? n_src : 1;              // kernel sets (and gradients)
    const size_t cw_bytes = ((size_t)(n_sets - 1) * (size_t)conv_src_stride + (size_t)ktot * (size_t)d) * 4;
    const size_t es = esize(dt);
    const size_t src_bytes = ((size_t)(n_src - 1) * (size_t)src_stride + (size_t)rows * (size_t)d) * es;
    const size_t dsrc_bytes = ((size_t)(n_src - 1) * (size_t)dsrc_stride + (size_t)rows * (size_t)d) * es;
    const size_t row_bytes = (size_t)T * (size_t)d * es;
    const size_t md = 4 * (size_t)d;
    if (T > 0 && (overlap(dsrc, dsrc_bytes, src, src_bytes) || overlap(dsrc, dsrc_bytes, dh, row_bytes) ||
                  overlap(ws, ws_bytes, src, src_bytes) || overlap(ws, ws_bytes, dsrc, dsrc_bytes) ||
                  overlap(ws, ws_bytes, dh, row_bytes)))
        return ATTNRES_ERR_INVALID_ARG;
    // the parameter gradients: disjoint from one another and from the workspace
    const void *pg[5] = {dconv_w, dqueries, dgain, dmix_gain, dmix_w};
    const size_t pn[5] = {cw_bytes, md * 4, (size_t)d * 4, md * 4, md * 16};
    for (int x = 0; x < 5; ++x) {
        if (!pg[x]) continue;
        if (T > 0 && overlap(pg[x], pn[x], ws, ws_bytes)) return ATTNRES_ERR_INVALID_ARG;
        for (int y = x + 1; y < 5; ++y)
            if (pg[y] && overlap(pg[x], pn[x], pg[y], pn[y])) return ATTNRES_ERR_INVALID_ARG;
    }
    if ((d != 1024 && d != 2048 && d != 4096) || n_src > 16) return ATTNRES_ERR_UNSUPPORTED;
    if (conv_src_stride > 0 && n_src > 1 && conv_src_stride % 4 != 0) return ATTNRES_ERR_UNSUPPORTED;
    if (!aligned16(conv_w) || !aligned16(queries) || !aligned16(mix_w) || (gain && !aligned16(gain)) ||
        (mix_gain && !aligned16(mix_gain)) || !aligned16(dmix_w) || !aligned4(dconv_w) || !aligned4(dqueries) ||
        (dgain && !aligned4(dgain)) || (dmix_gain && !aligned4(dmix_gain)))
        return ATTNRES_ERR_UNSUPPORTED;
    if (T > 0 && (!aligned16(dh) || !aligned16(dsrc) || (dsrc_stride * (int64_t)es) % 16 != 0 || !aligned16(ws)))
        return ATTNRES_ERR_UNSUPPORTED;
    DeviceInfo *dev = nullptr;
    st = device_info(&dev);
    if (st != ATTNRES_OK) return st;
    MsarBwdPlan p;
    st = msar_bwd_plan(n_src, T, d, dt, ksizes, dev, &p);
    if (st != ATTNRES_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (T == 0) {
        // no tokens: every parameter gradient is zero (nothing to add)
        if (accumulate) return ATTNRES_OK;
        cudaError_t e = cudaSuccess;
        for (int x = 1; x < 5 && e == cudaSuccess; ++x)
            if (pg[x]) e = cudaMemsetAsync(const_cast<void *>(pg[x]), 0, pn[x], s);
        for (int64_t k = 0; k < n_sets && e == cudaSuccess; ++k)
            e = cudaMemsetAsync(dconv_w + k * conv_src_stride, 0, (size_t)ktot * (size_t)d * 4, s);
        return e == cudaSuccess ? ATTNRES_OK : cuda_fail(e, "cudaMemsetAsync");
    }
    if (ws_bytes < p.total) return ATTNRES_ERR_INVALID_ARG;
    unsigned char *w = static_cast<unsigned char *>(ws);
    // from here on src and dsrc point at the chunk's first row
    src = static_cast<const unsigned char *>(src) + t_prev * d * (int64_t)es;
    dsrc = static_cast<unsigned char *>(dsrc) + t_prev * d * (int64_t)es;
    MsarBwdArgs a{};
    a.hist = t_prev;
    a.acc = accumulate;
    a.src = static_cast<const unsigned char *>(src);
    a.src_stride_bytes = src_stride * (int64_t)es;
    a.n_src = (int)n_src;
    a.T = T;
    a.d = (int)d;
    for (int r = 0; r < 3; ++r) a.k[r] = ksizes[r];
    a.ktot = (int)ktot;
    a.conv_w = conv_w;
    a.conv_src_stride = conv_src_stride;
    a.tc = p.tc;
    a.tc_s = p.tc_s;
    a.tc_m = p.tc_m;
    a.nsl = p.nsl;
    a.mix_part = reinterpret_cast<float *>(w + p.off_part);
    a.u = w + p.off_u;
    a.z = w + p.off_z;
    a.dz = w + p.off_dz;
    a.dh = static_cast<const unsigned char *>(dh);
    a.mix_gain = mix_gain;
    a.mix_w = mix_w;
    a.mix_eps = mix_eps;
    a.mix_e = reinterpret_cast<float *>(w + p.off_e);
    a.mix_parts = reinterpret_cast<float *>(w + p.off_mp);
    a.du = w + p.off_du;
    a.dsrc = static_cast<unsigned char *>(dsrc);
    a.dsrc_stride_bytes = dsrc_stride * (int64_t)es;
    a.conv_parts = reinterpret_cast<float *>(w + p.off_cp);
    a.dmix_w = dmix_w;
    a.dmix_gain = dmix_gain;
    const int dti = dt == ATTNRES_BF16 ? 1 : 0;
    const int64_t per_stream = n_src * T * d;          // elements of one stream's sources
    cudaError_t e = msar_bwd_streams(dti, a, stream);
    if (e != cudaSuccess) return cuda_fail(e, "msar backward streams launch");
    // Z^(r): stream 0 reads the sources themselves, stream r >= 1 the conv streams
    for (int64_t r = 0; r < 4; ++r) {
        const void *sr = r == 0 ? src : static_cast<const void *>(a.u + (size_t)(r - 1) * per_stream * es);
        st = launch_depth_read(sr, n_src, r == 0 ? src_stride : T * d, T, d, 1, dt, queries + r * d, 1, gain, eps,
                               a.z + (size_t)r * row_bytes, nullptr, stream);
        if (st != ATTNRES_OK) return st;
    }
    e = msar_bwd_mix(dti, a, stream);
    if (e != cudaSuccess) return cuda_fail(e, "msar backward mixer launch");
    float *A = reinterpret_cast<float *>(w + p.off_a);
    e = msar_bwd_sum(a.mix_parts, p.chunks, 16 * (int64_t)d, A, 0, stream);
    if (e == cudaSuccess) e = msar_bwd_mix_finish(a, A, stream);
    if (e != cudaSuccess) return cuda_fail(e, "msar backward mixer sums launch");
    // the per-stream read backward: du^(r), dw_r and stream r's share of dgain
    // (dw_r into a scratch row first when it adds into dqueries)
    float *dg = reinterpret_cast<float *>(w + p.off_dg);
    float *dqw = accumulate ? reinterpret_cast<float *>(w + p.off_dq) : dqueries;
    for (int64_t r = 0; r < 4; ++r) {
        const void *sr = r == 0 ? src : static_cast<const void *>(a.u + (size_t)(r - 1) * per_stream * es);
        st = launch_read_bwd(sr, n_src, r == 0 ? src_stride : T * d, T, d, 1, dt, queries + r * d, 1, gain, eps,
                             a.dz + (size_t)r * row_bytes, nullptr, a.du + (size_t)r * per_stream * es, T * d, 0,
                             dqw + r * d, dg + r * d, w + p.off_rb, p.rb_bytes, stream);
        if (st != ATTNRES_OK) return st;
    }
    if (accumulate) {
        e = msar_bwd_sum(dqw, 1, 4 * d, dqueries, 1, stream);
        if (e != cudaSuccess) return cuda_fail(e, "msar backward query sums launch");
    }
    e = msar_bwd_conv(dti, a, stream);
    if (conv_src_stride == 0) {
        // one kernel set: every (chunk, source) partial adds into it
        if (e == cudaSuccess) e = msar_bwd_conv_sum(a, a.conv_parts, p.chunks * n_src, ktot * d, dconv_w, stream);
    } else {
        // source i's gradient: its partials of every chunk
        for (int64_t i = 0; i < n_src && e == cudaSuccess; ++i)
            e = msar_bwd_conv_sum(a, a.conv_parts + i * ktot * d, p.chunks, n_src * ktot * d,
                                  dconv_w + i * conv_src_stride, stream);
    }
    if (e == cudaSuccess && dgain) e = msar_bwd_sum(dg, 4, d, dgain, accumulate, stream);
    if (e != cudaSuccess) return cuda_fail(e, "msar backward conv launch");
    return ATTNRES_OK;
}

// MSAR forward with a workspace: the conv streams are written once, each
// stream is read by the forward read kernels, and (one-shot read) the mixer
// runs over the per-stream reads.  Workspace regions start on 256-byte
// boundaries.
struct MsarFwdWsPlan {
    int64_t tc_s;
    size_t off_u, off_z, off_part, off_q, off_l, total;
};

MsarFwdWsPlan msar_fwd_ws_plan(int64_t n_src, int64_t T, int64_t d, attnres_dtype_t dt, bool oneshot, int64_t S) {
    MsarFwdWsPlan p{};
    p.tc_s = (T + 127) / 128;
    if (p.tc_s < 32) p.tc_s = 32;
    const size_t row = (size_t)T * (size_t)d * esize(dt);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off += (bytes + 255) / 256 * 256;
        return at;
    };
    p.off_u = take(3 * (size_t)n_src * row);
    if (oneshot) {
        p.off_z = take(4 * row);
        p.off_part = take((size_t)T * (size_t)(d / 1024) * 9 * 4);
    } else {
        p.off_q = take((size_t)4 * (size_t)S * (size_t)d * 4);
        p.off_l = take((size_t)(S < 8 ? S : 8) * (size_t)T * 4);
    }
    p.total = off;
    return p;
}

// the streams of every source into u (shared kernels, or source i's at i * conv_src_stride)
attnres_status_t msar_write_streams(const void *src, int64_t n_src, int64_t src_stride, int64_t T, int64_t d,
                                    attnres_dtype_t dt, const int32_t *ksizes, const float *conv_w,
                                    int64_t conv_src_stride, int64_t tc_s, unsigned char *u, void *stream) {
    MsarBwdArgs a{};
    a.src = static_cast<const unsigned char *>(src);
    a.src_stride_bytes = src_stride * (int64_t)esize(dt);
    a.n_src = (int)n_src;
    a.T = T;
    a.d = (int)d;
    for (int r = 0; r < 3; ++r) a.k[r] = ksizes[r];
    a.ktot = ksizes[0] + ksizes[1] + ksizes[2];
    a.conv_w = conv_w;
    a.conv_src_stride = conv_src_stride;
    a.tc_s = tc_s;
    a.u = u;
    cudaError_t e = msar_bwd_streams(dt == ATTNRES_BF16 ? 1 : 0, a, stream);
    return e == cudaSuccess ? ATTNRES_OK : cuda_fail(e, "msar streams launch");
}

attnres_status_t launch_msar_read_ws(const void *src, int64_t n_src, int64_t src_stride, int64_t T, int64_t d,
                                     attnres_dtype_t dt, int64_t m, const int32_t *ksizes, const float *conv_w,
                                     int64_t conv_src_stride, const float *queries, const float *gain, float eps,
                                     const float *mix_gain, const float *mix_w, float mix_eps, void *out, void *ws,
                                     size_t ws_bytes, void *stream) {
    attnres_status_t st = check_common(src, n_src, src_stride, T, d, dt, eps);
    if (st != ATTNRES_OK) return st;
    if (!(mix_eps >= 0.f) || std::isinf(mix_eps)) return ATTNRES_ERR_INVALID_ARG;
    st = check_msar_kernels(m, ksizes);
    if (st != ATTNRES_OK) return st;
    const int64_t ktot = (int64_t)ksizes[0] + ksizes[1] + ksizes[2];
    if (conv_src_stride < 0 || (conv_src_stride > 0 && n_src > 1 && conv_src_stride < d * ktot))
        return ATTNRES_ERR_INVALID_ARG;
    if (T == 0) return ATTNRES_OK;
    if (!conv_w || !queries || !mix_w || !out || !ws) return ATTNRES_ERR_INVALID_ARG;
    const size_t es = esize(dt);
    const size_t src_bytes = ((size_t)(n_src - 1) * (size_t)src_stride + (size_t)T * (size_t)d) * es;
    const size_t out_bytes = (size_t)T * (size_t)d * es;
    if (overlap(out, out_bytes, src, src_bytes) || overlap(ws, ws_bytes, src, src_bytes) ||
        overlap(ws, ws_bytes, out, out_bytes))
        return ATTNRES_ERR_INVALID_ARG;
    if (d % 1024 != 0 || d > 16384) return ATTNRES_ERR_UNSUPPORTED;
    if (!aligned16(out) || !aligned16(queries) || !aligned4(conv_w) || !aligned16(mix_w) ||
        (gain && !aligned16(gain)) || (mix_gain && !aligned4(mix_gain)) || !aligned16(ws))
        return ATTNRES_ERR_UNSUPPORTED;
    const MsarFwdWsPlan p = msar_fwd_ws_plan(n_src, T, d, dt, true, 0);
    if (ws_bytes < p.total) return ATTNRES_ERR_INVALID_ARG;
    unsigned char *w = static_cast<unsigned char *>(ws);
    st = msar_write_streams(src, n_src, src_stride, T, d, dt, ksizes, conv_w, conv_src_stride, p.tc_s, w + p.off_u,
                            stream);
    if (st != ATTNRES_OK) return st;
    const size_t row = (size_t)T * (size_t)d * es;
    for (int64_t r = 0; r < 4; ++r) {
        const void *sr = r == 0 ? src : static_cast<const void *>(w + p.off_u + (size_t)(r - 1) * (size_t)n_src * row);
        st = launch_depth_read(sr, n_src, r == 0 ? src_stride : T * d, T, d, 1, dt, queries + r * d, 1, gain, eps,
                               w + p.off_z + (size_t)r * row, nullptr, stream);
        if (st != ATTNRES_OK) return st;
    }
    MsarBwdArgs a{};
    a.T = T;
    a.d = (int)d;
    a.z = w + p.off_z;
    a.dh = nullptr;
    a.mix_gain = mix_gain;
    a.mix_w = mix_w;
    a.mix_eps = mix_eps;
    a.mix_part = reinterpret_cast<float *>(w + p.off_part);
    a.nsl = (int)(d / 1024);
    a.tc_m = mix_tokens_per_cta(T);
    cudaError_t e = msar_fwd_mix(dt == ATTNRES_BF16 ? 1 : 0, a, out, stream);
    return e == cudaSuccess ? ATTNRES_OK : cuda_fail(e, "msar mixer launch");
}

attnres_status_t launch_msar_phase1_ws(const void *src, int64_t n_src, int64_t src_stride, int64_t T, int64_t d,
                                       attnres_dtype_t dt, int64_t m, const int32_t *ksizes, const float *conv_w,
                                       const float *queries, int64_t S, const float *gain, float eps, void *o,
                                       float *lse, void *ws, size_t ws_bytes, void *stream) {
    attnres_status_t st = check_common(src, n_src, src_stride, T, d, dt, eps);
    if (st != ATTNRES_OK) return st;
    if (S < 1) return ATTNRES_ERR_INVALID_ARG;
    if (T == 0) return ATTNRES_OK;
    if (!conv_w || !queries || !o || !lse || !ws) return ATTNRES_ERR_INVALID_ARG;
    st = check_msar_kernels(m, ksizes);
    if (st != ATTNRES_OK) return st;
    const size_t es = esize(dt);
    const size_t src_bytes = ((size_t)(n_src - 1) * (size_t)src_stride + (size_t)T * (size_t)d) * es;
    const size_t o_bytes = (size_t)S * 4 * (size_t)T * (size_t)d * es;
    const size_t lse_bytes = (size_t)S * 4 * (size_t)T * sizeof(float);
    if (overlap(o, o_bytes, src, src_bytes) || overlap(lse, lse_bytes, src, src_bytes) ||
        overlap(lse, lse_bytes, o, o_bytes) || overlap(ws, ws_bytes, src, src_bytes) ||
        overlap(ws, ws_bytes, o, o_bytes) || overlap(ws, ws_bytes, lse, lse_bytes))
        return ATTNRES_ERR_INVALID_ARG;
    if (d % 512 != 0 || d > 16384) return ATTNRES_ERR_UNSUPPORTED;
    if (!aligned16(o) || !aligned4(lse) || !aligned16(queries) || !aligned4(conv_w) || (gain && !aligned16(gain)) ||
        !aligned16(ws))
        return ATTNRES_ERR_UNSUPPORTED;
    const MsarFwdWsPlan p = msar_fwd_ws_plan(n_src, T, d, dt, false, S);
    if (ws_bytes < p.total) return ATTNRES_ERR_INVALID_ARG;
    unsigned char *w = static_cast<unsigned char *>(ws);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    st = msar_write_streams(src, n_src, src_stride, T, d, dt, ksizes, conv_w, 0, p.tc_s, w + p.off_u, stream);
    if (st != ATTNRES_OK) return st;
    // stream r's queries of every layer, contiguous: qbuf[r][s] = queries[s][r]
    float *qbuf = reinterpret_cast<float *>(w + p.off_q);
    cudaError_t e = cudaMemcpy2DAsync(qbuf, (size_t)d * 4, queries, (size_t)4 * d * 4, (size_t)d * 4, (size_t)S, cudaMemcpyDeviceToDevice, s);
    for (int64_t r = 1; r < 4 && e == cudaSuccess; ++r)
        e = cudaMemcpy2DAsync(qbuf + r * S * d, (size_t)d * 4, queries + r * d, (size_t)4 * d * 4, (size_t)d * 4,
                              (size_t)S, cudaMemcpyDeviceToDevice, s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy2DAsync");
    float *lbuf = reinterpret_cast<float *>(w + p.off_l);
    const size_t row = (size_t)T * (size_t)d * es;
    for (int64_t r = 0; r < 4; ++r) {
        const void *sr = r == 0 ? src : static_cast<const void *>(w + p.off_u + (size_t)(r - 1) * (size_t)n_src * row);
        // layers in groups of up to 8 queries; o[s][r] is 4 T d elements after o[s-1][r]
        for (int64_t s0 = 0; s0 < S; s0 += 8) {
            const int64_t ns = S - s0 < 8 ? S - s0 : 8;
            st = launch_depth_read(sr, n_src, r == 0 ? src_stride : T * d, T, d, 1, dt, qbuf + (r * S + s0) * d, ns,
                                   gain, eps, static_cast<unsigned char *>(o) + (size_t)(s0 * 4 + r) * row, lbuf,
                                   stream, 4 * T * d);
            if (st != ATTNRES_OK) return st;
            e = cudaMemcpy2DAsync(lse + (s0 * 4 + r) * T, (size_t)4 * T * 4, lbuf, (size_t)T * 4, (size_t)T * 4,
                                  (size_t)ns, cudaMemcpyDeviceToDevice, s);
            if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy2DAsync");
        }
    }
    return ATTNRES_OK;
}

// MSAR phase 2 with a workspace: the partial's three conv streams written
// once, each stream merged into its phase-1 state by the Block merge kernel
// (Z^(r) stored), then the sliced mixer.  No partial: the mixer over o.
attnres_status_t launch_msar_phase2_ws(const void *o, const float *lse, const void *partial, int64_t T, int64_t d,
                                       attnres_dtype_t dt, int64_t m, const int32_t *ksizes, const float *conv_w,
                                       const float *query, const float *gain, float eps, const float *mix_gain,
                                       const float *mix_w, float mix_eps, void *out, void *ws, size_t ws_bytes,
                                       void *stream) {
    if (dt != ATTNRES_F32 && dt != ATTNRES_BF16) return ATTNRES_ERR_INVALID_ARG;
    if (T < 0 || d < 1 || !(eps >= 0.f) || std::isinf(eps) || !(mix_eps >= 0.f) || std::isinf(mix_eps))
        return ATTNRES_ERR_INVALID_ARG;
    if (T > 0 && d > INT64_MAX / (4 * T)) return ATTNRES_ERR_INVALID_ARG;
    if (T == 0) return ATTNRES_OK;
    if (!o || !lse || !conv_w || !query || !mix_w || !out || !ws) return ATTNRES_ERR_INVALID_ARG;
    attnres_status_t st = check_msar_kernels(m, ksizes);
    if (st != ATTNRES_OK) return st;
    const size_t es = esize(dt);
    const size_t row = (size_t)T * (size_t)d * es;
    if (overlap(out, row, o, 4 * row) || overlap(out, row, lse, (size_t)4 * T * 4) ||
        (partial && overlap(out, row, partial, row)) || overlap(ws, ws_bytes, o, 4 * row) ||
        overlap(ws, ws_bytes, lse, (size_t)4 * T * 4) || overlap(ws, ws_bytes, out, row) ||
        (partial && overlap(ws, ws_bytes, partial, row)))
        return ATTNRES_ERR_INVALID_ARG;
    if (d % 1024 != 0 || d > 16384) return ATTNRES_ERR_UNSUPPORTED;
    if (!aligned16(o) || !aligned4(lse) || (partial && !aligned16(partial)) || !aligned16(out) ||
        !aligned16(query) || !aligned4(conv_w) || !aligned16(mix_w) || (gain && !aligned16(gain)) ||
        (mix_gain && !aligned4(mix_gain)) || !aligned16(ws))
        return ATTNRES_ERR_UNSUPPORTED;
    const MsarFwdWsPlan p = msar_fwd_ws_plan(1, T, d, dt, true, 0);
    if (ws_bytes < p.total) return ATTNRES_ERR_INVALID_ARG;
    unsigned char *w = static_cast<unsigned char *>(ws);
    const unsigned char *z = static_cast<const unsigned char *>(o);
    if (partial) {
        st = msar_write_streams(partial, 1, T * d, T, d, dt, ksizes, conv_w, 0, p.tc_s, w + p.off_u, stream);
        if (st != ATTNRES_OK) return st;
        for (int64_t r = 0; r < 4; ++r) {
            const void *pr = r == 0 ? partial : static_cast<const void *>(w + p.off_u + (size_t)(r - 1) * row);
            st = launch_phase2(static_cast<const unsigned char *>(o) + (size_t)r * row, lse + r * T, pr, nullptr,
                               nullptr, false, T, d, 1, dt, query + r * d, gain, eps, w + p.off_z + (size_t)r * row,
                               stream);
            if (st != ATTNRES_OK) return st;
        }
        z = w + p.off_z;
    }
    MsarBwdArgs a{};
    a.T = T;
    a.d = (int)d;
    a.z = const_cast<unsigned char *>(z);          // read only by the mixer
    a.dh = nullptr;
    a.mix_gain = mix_gain;
    a.mix_w = mix_w;
    a.mix_eps = mix_eps;
    a.mix_part = reinterpret_cast<float *>(w + p.off_part);
    a.nsl = (int)(d / 1024);
    a.tc_m = mix_tokens_per_cta(T);
    cudaError_t e = msar_fwd_mix(dt == ATTNRES_BF16 ? 1 : 0, a, out, stream);
    return e == cudaSuccess ? ATTNRES_OK : cuda_fail(e, "msar mixer launch");
}

// Backward of MSAR's two-phase schedule.  Workspace regions start on 256-byte
// boundaries; token chunks of the conv transpose and the mixer sums as the
// one-shot backward's plan.
struct MsarTwoPhaseBwdPlan {
    int64_t tc, chunks, tc_s;
    int nsl;
    MergeBwdShape mb;
    ReadBwdShape rb;
    size_t mb_bytes, rb_bytes;
    size_t off_u, off_z, off_dz, off_du, off_mb, off_rb, off_dg, off_part, off_e, off_mp, off_a, off_cp;
    size_t off_q, off_do, off_dl, off_dq, total;
};

attnres_status_t msar_two_phase_bwd_plan(bool phase2, int64_t n_src, int64_t T, int64_t d, attnres_dtype_t dt,
                                         const int32_t *ksizes, int64_t S, const DeviceInfo *dev,
                                         MsarTwoPhaseBwdPlan *p) {
    *p = MsarTwoPhaseBwdPlan{};
    if (phase2) {
        if (d % 1024 != 0 || d > 4096) return ATTNRES_ERR_UNSUPPORTED;
        attnres_status_t st = merge_bwd_shape(T, d, dt, dev, &p->mb);
        if (st != ATTNRES_OK) return st;
        p->mb_bytes = merge_bwd_ws_bytes(p->mb, d);
    } else {
        if (d % 512 != 0 || d > 4096 || n_src > 16) return ATTNRES_ERR_UNSUPPORTED;
        attnres_status_t st = read_bwd_shape(n_src, d, S, 1, dt, &p->rb);
        if (st != ATTNRES_OK) return st;
        st = read_bwd_ws_need(n_src, T, d, 1, S, dt, dev, p->rb, &p->rb_bytes);
        if (st != ATTNRES_OK) return st;
    }
    p->tc = (T + 63) / 64;
    if (p->tc < 32) p->tc = 32;
    p->chunks = T > 0 ? (T + p->tc - 1) / p->tc : 0;
    p->tc_s = (T + 127) / 128;
    if (p->tc_s < 32) p->tc_s = 32;
    p->nsl = (int)(d / 1024);
    const int64_t ktot = (int64_t)ksizes[0] + ksizes[1] + ksizes[2];
    const size_t es = esize(dt);
    const size_t row = (size_t)T * (size_t)d * es;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off += (bytes + 255) / 256 * 256;
        return at;
    };
    const int64_t ns = phase2 ? 1 : n_src;                  // sources expanded: the partial, or the cached ones
    p->off_u = take(3 * (size_t)ns * row);
    p->off_du = take(4 * (size_t)ns * row);
    p->off_dg = take(4 * (size_t)d * 4);
    p->off_cp = take((size_t)p->chunks * (size_t)ns * (size_t)ktot * (size_t)d * 4);
    if (phase2) {
        p->off_z = take(4 * row);
        p->off_dz = take(4 * row);
        p->off_mb = take(p->mb_bytes);
        p->off_part = take((size_t)T * (size_t)p->nsl * 9 * 4);
        p->off_e = take((size_t)T * 4 * 4);
        p->off_mp = take((size_t)p->chunks * 16 * (size_t)d * 4);
        p->off_a = take(16 * (size_t)d * 4);
    } else {
        p->off_rb = take(p->rb_bytes);
        p->off_q = take((size_t)4 * (size_t)S * (size_t)d * 4);
        p->off_do = take((size_t)S * row);
        p->off_dl = take((size_t)S * (size_t)T * 4);
        p->off_dq = take((size_t)S * (size_t)d * 4);
    }
    p->total = off;
    return ATTNRES_OK;
}

// the conv transpose of ns sources' stream gradients (du [4][ns][T][d]) into
// dsrc and dconv_w (one kernel set), and dgain from the streams' shares
attnres_status_t msar_conv_back(const void *src, int64_t ns, int64_t src_stride, int64_t T, int64_t d,
                                attnres_dtype_t dt, const int32_t *ksizes, const float *conv_w,
                                const MsarTwoPhaseBwdPlan &p, unsigned char *w, void *dsrc, int64_t dsrc_stride,
                                float *dconv_w, float *dgain, void *stream) {
    MsarBwdArgs a{};
    const size_t es = esize(dt);
    a.src = static_cast<const unsigned char *>(src);
    a.src_stride_bytes = src_stride * (int64_t)es;
    a.n_src = (int)ns;
    a.T = T;
    a.d = (int)d;
    for (int r = 0; r < 3; ++r) a.k[r] = ksizes[r];
    a.ktot = ksizes[0] + ksizes[1] + ksizes[2];
    a.conv_w = conv_w;
    a.tc = p.tc;
    a.du = w + p.off_du;
    a.dsrc = static_cast<unsigned char *>(dsrc);
    a.dsrc_stride_bytes = dsrc_stride * (int64_t)es;
    a.conv_parts = reinterpret_cast<float *>(w + p.off_cp);
    const int dti = dt == ATTNRES_BF16 ? 1 : 0;
    cudaError_t e = msar_bwd_conv(dti, a, stream);
    if (e == cudaSuccess) e = msar_bwd_conv_sum(a, a.conv_parts, p.chunks * ns, (int64_t)a.ktot * d, dconv_w, stream);
    if (e == cudaSuccess && dgain)
        e = msar_bwd_sum(reinterpret_cast<const float *>(w + p.off_dg), 4, d, dgain, 0, stream);
    return e == cudaSuccess ? ATTNRES_OK : cuda_fail(e, "msar conv transpose launch");
}

attnres_status_t launch_msar_phase2_bwd(const void *o, const float *lse, const void *partial, int64_t T, int64_t d,
                                        attnres_dtype_t dt, int64_t m, const int32_t *ksizes, const float *conv_w,
                                        const float *query, const float *gain, float eps, const float *mix_gain,
                                        const float *mix_w, float mix_eps, const void *dh, void *d_o, float *d_lse,
                                        void *d_partial, float *dconv_w, float *dquery, float *dgain,
                                        float *dmix_gain, float *dmix_w, void *ws, size_t ws_bytes, void *stream) {
    if (dt != ATTNRES_F32 && dt != ATTNRES_BF16) return ATTNRES_ERR_INVALID_ARG;
    if (T < 0 || d < 1 || !(eps >= 0.f) || std::isinf(eps) || !(mix_eps >= 0.f) || std::isinf(mix_eps))
        return ATTNRES_ERR_INVALID_ARG;
    if (T > 0 && d > INT64_MAX / (4 * T)) return ATTNRES_ERR_INVALID_ARG;
    attnres_status_t st = check_msar_kernels(m, ksizes);
    if (st != ATTNRES_OK) return st;
    if (!conv_w || !query || !mix_w || !dconv_w || !dquery || !dmix_w) return ATTNRES_ERR_INVALID_ARG;
    if (T > 0 && (!o || !lse || !dh || !d_o || !d_lse || !ws || (partial && !d_partial)))
        return ATTNRES_ERR_INVALID_ARG;
    const int64_t ktot = (int64_t)ksizes[0] + ksizes[1] + ksizes[2];
    const size_t es = esize(dt);
    const size_t row = (size_t)T * (size_t)d * es, lrow = (size_t)T * 4;
    const size_t md = 4 * (size_t)d;
    if (T > 0) {
        // outputs against the inputs and one another; the workspace against everything
        const void *in[4] = {o, lse, partial, dh};
        const size_t inb[4] = {4 * row, 4 * lrow, row, row};
        const void *outp[3] = {d_o, d_lse, d_partial};
        const size_t outb[3] = {4 * row, 4 * lrow, row};
        for (int x = 0; x < 3; ++x) {
            if (!outp[x]) continue;
            for (int y = 0; y < 4; ++y)
                if (in[y] && overlap(outp[x], outb[x], in[y], inb[y])) return ATTNRES_ERR_INVALID_ARG;
            for (int y = x + 1; y < 3; ++y)
                if (outp[y] && overlap(outp[x], outb[x], outp[y], outb[y])) return ATTNRES_ERR_INVALID_ARG;
            if (overlap(outp[x], outb[x], ws, ws_bytes)) return ATTNRES_ERR_INVALID_ARG;
        }
        for (int y = 0; y < 4; ++y)
            if (in[y] && overlap(in[y], inb[y], ws, ws_bytes)) return ATTNRES_ERR_INVALID_ARG;
    }
    const void *pg[5] = {dconv_w, dquery, dgain, dmix_gain, dmix_w};
    const size_t pn[5] = {(size_t)ktot * (size_t)d * 4, md * 4, (size_t)d * 4, md * 4, md * 16};
    for (int x = 0; x < 5; ++x) {
        if (!pg[x]) continue;
        if (T > 0 && overlap(pg[x], pn[x], ws, ws_bytes)) return ATTNRES_ERR_INVALID_ARG;
        for (int y = x + 1; y < 5; ++y)
            if (pg[y] && overlap(pg[x], pn[x], pg[y], pn[y])) return ATTNRES_ERR_INVALID_ARG;
    }
    if (d % 1024 != 0 || d > 4096) return ATTNRES_ERR_UNSUPPORTED;
    if (!aligned16(conv_w) || !aligned16(query) || !aligned16(mix_w) || (gain && !aligned16(gain)) ||
        (mix_gain && !aligned16(mix_gain)) || !aligned16(dmix_w) || !aligned4(dconv_w) || !aligned16(dquery) ||
        (dgain && !aligned4(dgain)) || (dmix_gain && !aligned4(dmix_gain)))
        return ATTNRES_ERR_UNSUPPORTED;
    if (T > 0 && (!aligned16(o) || !aligned4(lse) || (partial && !aligned16(partial)) || !aligned16(dh) ||
                  !aligned16(d_o) || !aligned4(d_lse) || (d_partial && !aligned16(d_partial)) || !aligned16(ws)))
        return ATTNRES_ERR_UNSUPPORTED;
    DeviceInfo *dev = nullptr;
    st = device_info(&dev);
    if (st != ATTNRES_OK) return st;
    MsarTwoPhaseBwdPlan p;
    st = msar_two_phase_bwd_plan(true, 1, T, d, dt, ksizes, 0, dev, &p);
    if (st != ATTNRES_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (T == 0) {
        cudaError_t e = cudaSuccess;
        for (int x = 0; x < 5 && e == cudaSuccess; ++x)
            if (pg[x]) e = cudaMemsetAsync(const_cast<void *>(pg[x]), 0, pn[x], s);
        return e == cudaSuccess ? ATTNRES_OK : cuda_fail(e, "cudaMemsetAsync");
    }
    if (ws_bytes < p.total) return ATTNRES_ERR_INVALID_ARG;
    unsigned char *w = static_cast<unsigned char *>(ws);
    const int dti = dt == ATTNRES_BF16 ? 1 : 0;
    // forward again: the partial's streams and the merged states
    const unsigned char *z = static_cast<const unsigned char *>(o);
    if (partial) {
        st = msar_write_streams(partial, 1, T * d, T, d, dt, ksizes, conv_w, 0, p.tc_s, w + p.off_u, stream);
        if (st != ATTNRES_OK) return st;
        for (int64_t r = 0; r < 4; ++r) {
            const void *pr = r == 0 ? partial : static_cast<const void *>(w + p.off_u + (size_t)(r - 1) * row);
            st = launch_phase2(static_cast<const unsigned char *>(o) + (size_t)r * row, lse + r * T, pr, nullptr,
                               nullptr, false, T, d, 1, dt, query + r * d, gain, eps, w + p.off_z + (size_t)r * row,
                               stream);
            if (st != ATTNRES_OK) return st;
        }
        z = w + p.off_z;
    }
    // the mixer's backward: dZ (straight into d_o without a partial) and its parameters
    MsarBwdArgs a{};
    a.T = T;
    a.d = (int)d;
    a.tc = p.tc;
    a.tc_m = mix_tokens_per_cta(T);
    a.nsl = p.nsl;
    a.z = const_cast<unsigned char *>(z);           // read only
    a.dz = partial ? w + p.off_dz : static_cast<unsigned char *>(d_o);
    a.dh = static_cast<const unsigned char *>(dh);
    a.mix_gain = mix_gain;
    a.mix_w = mix_w;
    a.mix_eps = mix_eps;
    a.mix_part = reinterpret_cast<float *>(w + p.off_part);
    a.mix_e = reinterpret_cast<float *>(w + p.off_e);
    a.mix_parts = reinterpret_cast<float *>(w + p.off_mp);
    a.dmix_w = dmix_w;
    a.dmix_gain = dmix_gain;
    cudaError_t e = msar_bwd_mix(dti, a, stream);
    float *A = reinterpret_cast<float *>(w + p.off_a);
    if (e == cudaSuccess) e = msar_bwd_sum(a.mix_parts, p.chunks, 16 * (int64_t)d, A, 0, stream);
    if (e == cudaSuccess) e = msar_bwd_mix_finish(a, A, stream);
    if (e != cudaSuccess) return cuda_fail(e, "msar mixer backward launch");
    if (!partial) {
        // Z = o: the state takes dZ, nothing reaches lse, the queries, the gain or the kernels
        e = cudaMemsetAsync(d_lse, 0, 4 * lrow, s);
        if (e == cudaSuccess) e = cudaMemsetAsync(dquery, 0, md * 4, s);
        if (e == cudaSuccess && dgain) e = cudaMemsetAsync(dgain, 0, (size_t)d * 4, s);
        if (e == cudaSuccess) e = cudaMemsetAsync(dconv_w, 0, (size_t)ktot * (size_t)d * 4, s);
        return e == cudaSuccess ? ATTNRES_OK : cuda_fail(e, "cudaMemsetAsync");
    }
    // each stream's merge backward, then the partial's streams back through the convolutions
    float *dg = reinterpret_cast<float *>(w + p.off_dg);
    for (int64_t r = 0; r < 4; ++r) {
        const void *pr = r == 0 ? partial : static_cast<const void *>(w + p.off_u + (size_t)(r - 1) * row);
        st = launch_merge_bwd(static_cast<const unsigned char *>(o) + (size_t)r * row, lse + r * T, pr, T, d, dt,
                              query + r * d, gain, eps, w + p.off_dz + (size_t)r * row,
                              static_cast<unsigned char *>(d_o) + (size_t)r * row, d_lse + r * T,
                              w + p.off_du + (size_t)r * row, 0, dquery + r * d, dg + r * d, w + p.off_mb, p.mb_bytes,
                              stream);
        if (st != ATTNRES_OK) return st;
    }
    return msar_conv_back(partial, 1, T * d, T, d, dt, ksizes, conv_w, p, w, d_partial, T * d, dconv_w, dgain,
                          stream);
}

attnres_status_t launch_msar_phase1_bwd(const void *src, int64_t n_src, int64_t src_stride, int64_t T, int64_t d,
                                        attnres_dtype_t dt, int64_t m, const int32_t *ksizes, const float *conv_w,
                                        const float *queries, int64_t S, const float *gain, float eps,
                                        const void *d_o, const float *d_lse, void *dsrc, int64_t dsrc_stride,
                                        float *dconv_w, float *dqueries, float *dgain, void *ws, size_t ws_bytes,
                                        void *stream) {
    attnres_status_t st = check_common(src, n_src, src_stride, T, d, dt, eps);
    if (st != ATTNRES_OK) return st;
    if (S < 1) return ATTNRES_ERR_INVALID_ARG;
    st = check_msar_kernels(m, ksizes);
    if (st != ATTNRES_OK) return st;
    if (!conv_w || !queries || !dconv_w || !dqueries) return ATTNRES_ERR_INVALID_ARG;
    if (T > 0 && (!d_o || !d_lse || !dsrc || !ws)) return ATTNRES_ERR_INVALID_ARG;
    if (dsrc_stride < T * d) return ATTNRES_ERR_INVALID_ARG;
    const int64_t ktot = (int64_t)ksizes[0] + ksizes[1] + ksizes[2];
    const size_t es = esize(dt);
    const size_t row = (size_t)T * (size_t)d * es;
    const size_t src_bytes = ((size_t)(n_src - 1) * (size_t)src_stride + (size_t)T * (size_t)d) * es;
    const size_t dsrc_bytes = ((size_t)(n_src - 1) * (size_t)dsrc_stride + (size_t)T * (size_t)d) * es;
    const size_t do_bytes = (size_t)S * 4 * row, dl_bytes = (size_t)S * 4 * (size_t)T * 4;
    if (T > 0 && (overlap(dsrc, dsrc_bytes, src, src_bytes) || overlap(dsrc, dsrc_bytes, d_o, do_bytes) ||
                  overlap(dsrc, dsrc_bytes, d_lse, dl_bytes) || overlap(ws, ws_bytes, src, src_bytes) ||
                  overlap(ws, ws_bytes, dsrc, dsrc_bytes) || overlap(ws, ws_bytes, d_o, do_bytes) ||
                  overlap(ws, ws_bytes, d_lse, dl_bytes)))
        return ATTNRES_ERR_INVALID_ARG;
    const void *pg[3] = {dconv_w, dqueries, dgain};
    const size_t pn[3] = {(size_t)ktot * (size_t)d * 4, (size_t)S * 4 * (size_t)d * 4, (size_t)d * 4};
    for (int x = 0; x < 3; ++x) {
        if (!pg[x]) continue;
        if (T > 0 && overlap(pg[x], pn[x], ws, ws_bytes)) return ATTNRES_ERR_INVALID_ARG;
        for (int y = x + 1; y < 3; ++y)
            if (pg[y] && overlap(pg[x], pn[x], pg[y], pn[y])) return ATTNRES_ERR_INVALID_ARG;
    }
    if (d % 512 != 0 || d > 4096 || n_src > 16) return ATTNRES_ERR_UNSUPPORTED;
    if (!aligned4(conv_w) || !aligned16(queries) || (gain && !aligned16(gain)) || !aligned4(dconv_w) ||
        !aligned4(dqueries) || (dgain && !aligned4(dgain)))
        return ATTNRES_ERR_UNSUPPORTED;
    if (T > 0 && (!aligned16(d_o) || !aligned4(d_lse) || !aligned16(dsrc) || (dsrc_stride * (int64_t)es) % 16 != 0 ||
                  !aligned16(ws)))
        return ATTNRES_ERR_UNSUPPORTED;
    DeviceInfo *dev = nullptr;
    st = device_info(&dev);
    if (st != ATTNRES_OK) return st;
    MsarTwoPhaseBwdPlan p;
    st = msar_two_phase_bwd_plan(false, n_src, T, d, dt, ksizes, S, dev, &p);
    if (st != ATTNRES_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (T == 0) {
        cudaError_t e = cudaSuccess;
        for (int x = 0; x < 3 && e == cudaSuccess; ++x)
            if (pg[x]) e = cudaMemsetAsync(const_cast<void *>(pg[x]), 0, pn[x], s);
        return e == cudaSuccess ? ATTNRES_OK : cuda_fail(e, "cudaMemsetAsync");
    }
    if (ws_bytes < p.total) return ATTNRES_ERR_INVALID_ARG;
    unsigned char *w = static_cast<unsigned char *>(ws);
    st = msar_write_streams(src, n_src, src_stride, T, d, dt, ksizes, conv_w, 0, p.tc_s, w + p.off_u, stream);
    if (st != ATTNRES_OK) return st;
    // stream r's queries of every layer, contiguous: qbuf[r][s] = queries[s][r]
    float *qbuf = reinterpret_cast<float *>(w + p.off_q);
    cudaError_t e = cudaSuccess;
    for (int64_t r = 0; r < 4 && e == cudaSuccess; ++r)
        e = cudaMemcpy2DAsync(qbuf + r * S * d, (size_t)d * 4, queries + r * d, (size_t)4 * d * 4, (size_t)d * 4,
                              (size_t)S, cudaMemcpyDeviceToDevice, s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy2DAsync");
    unsigned char *dobuf = w + p.off_do;
    float *dlbuf = reinterpret_cast<float *>(w + p.off_dl);
    float *dqbuf = reinterpret_cast<float *>(w + p.off_dq);
    float *dg = reinterpret_cast<float *>(w + p.off_dg);
    for (int64_t r = 0; r < 4; ++r) {
        // stream r's gradients of every layer, contiguous, then its read's backward
        e = cudaMemcpy2DAsync(dobuf, row, static_cast<const unsigned char *>(d_o) + (size_t)r * row, 4 * row, row,
                              (size_t)S, cudaMemcpyDeviceToDevice, s);
        if (e == cudaSuccess)
            e = cudaMemcpy2DAsync(dlbuf, (size_t)T * 4, d_lse + r * T, (size_t)4 * T * 4, (size_t)T * 4, (size_t)S,
                                  cudaMemcpyDeviceToDevice, s);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy2DAsync");
        const void *sr = r == 0 ? src : static_cast<const void *>(w + p.off_u + (size_t)(r - 1) * (size_t)n_src * row);
        st = launch_read_bwd(sr, n_src, r == 0 ? src_stride : T * d, T, d, 1, dt, qbuf + r * S * d, S, gain, eps,
                             dobuf, dlbuf, w + p.off_du + (size_t)r * (size_t)n_src * row, T * d, 0, dqbuf,
                             dg + r * d, w + p.off_rb, p.rb_bytes, stream);
        if (st != ATTNRES_OK) return st;
        e = cudaMemcpy2DAsync(dqueries + r * d, (size_t)4 * d * 4, dqbuf, (size_t)d * 4, (size_t)d * 4, (size_t)S,
                              cudaMemcpyDeviceToDevice, s);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy2DAsync");
    }
    return msar_conv_back(src, n_src, src_stride, T, d, dt, ksizes, conv_w, p, w, dsrc, dsrc_stride, dconv_w, dgain,
                          stream);
}

}  // namespace

extern "C" {

attnres_status_t attnres_full_fwd(const void *src, int64_t n_src, int64_t src_stride, int64_t T,
                                  int64_t d, attnres_dtype_t dt, const float *query,
                                  const float *gain, float eps, void *out, void *stream) {
    return launch_depth_read(src, n_src, src_stride, T, d, 1, dt, query, 1, gain, eps, out, nullptr,
                             stream);
}

attnres_status_t attnres_block_phase1(const void *src, int64_t n_src, int64_t src_stride,
                                      int64_t T, int64_t d, attnres_dtype_t dt,
                                      const float *queries, int64_t n_q, const float *gain,
                                      float eps, void *o, float *lse, void *stream) {
    return launch_depth_read(src, n_src, src_stride, T, d, 1, dt, queries, n_q, gain, eps, o, lse,
                             stream);
}

attnres_status_t mhar_fwd(const void *src, int64_t n_src, int64_t src_stride, int64_t T, int64_t d,
                          int64_t H, attnres_dtype_t dt, const float *queries, int64_t n_q,
                          const float *gain, float eps, void *out, float *lse, void *stream) {
    return launch_depth_read(src, n_src, src_stride, T, d, H, dt, queries, n_q, gain, eps, out, lse,
                             stream);
}

attnres_status_t attnres_block_phase2_merge(const void *o, const float *lse, const void *partial,
                                            int64_t T, int64_t d, attnres_dtype_t dt,
                                            const float *query, const float *gain, float eps,
                                            void *out, void *stream) {
    return launch_phase2(o, lse, partial, nullptr, nullptr, false, T, d, 1, dt, query, gain, eps, out, stream);
}

attnres_status_t attnres_block_phase2_update_merge(const void *partial, const void *f, void *partial_out,
                                                   const void *o, const float *lse, int64_t T, int64_t d,
                                                   attnres_dtype_t dt, const float *query, const float *gain,
                                                   float eps, void *out, void *stream) {
    return launch_phase2(o, lse, partial, f, partial_out, true, T, d, 1, dt, query, gain, eps, out, stream);
}

attnres_status_t mhar_phase2_merge(const void *o, const float *lse, const void *partial, const void *f,
                                   void *partial_out, int64_t T, int64_t d, int64_t H, attnres_dtype_t dt,
                                   const float *query, const float *gain, float eps, void *out, void *stream) {
    return launch_phase2(o, lse, partial, f, partial_out, f != nullptr, T, d, H, dt, query, gain, eps, out,
                         stream);
}

static attnres_status_t read_bwd_workspace(int64_t n_src, int64_t T, int64_t d, int64_t H, int64_t n_q,
                                           attnres_dtype_t dt, size_t *bytes) {
    if (!bytes || (dt != ATTNRES_F32 && dt != ATTNRES_BF16) || n_src < 1 || T < 0 || d < 1 || n_q < 1 || H < 1 ||
        d % H != 0)
        return ATTNRES_ERR_INVALID_ARG;
    if (d % 8 != 0) return ATTNRES_ERR_UNSUPPORTED;
    if (n_src > 16 && H == 1) {
        // more sources than one pass takes: chunks of 8 and their states
        if (n_q > 8 || (n_src + kReadBwdChunk - 1) / kReadBwdChunk > kReadBwdMaxChunks)
            return ATTNRES_ERR_UNSUPPORTED;
        DeviceInfo *dev = nullptr;
        attnres_status_t st = device_info(&dev);
        if (st != ATTNRES_OK) return st;
        if (read_bwd_many_split_applies(dt, n_src, n_q, d)) {
            ReadBwdManySplitShape sh;
            st = read_bwd_many_split_shape(n_src, T, d, dev, &sh);
            if (st != ATTNRES_OK) return st;
            *bytes = sh.total;
            return ATTNRES_OK;
        }
        ReadBwdManyPlan p;
        st = read_bwd_many_plan(n_src, T, d, n_q, dt, dev, &p);
        if (st != ATTNRES_OK) return st;
        *bytes = p.total;
        return ATTNRES_OK;
    }
    ReadBwdShape sh;
    attnres_status_t st = read_bwd_shape(n_src, d, n_q, H, dt, &sh);
    if (st != ATTNRES_OK) return st;
    DeviceInfo *dev = nullptr;
    st = device_info(&dev);
    if (st != ATTNRES_OK) return st;
    return read_bwd_ws_need(n_src, T, d, H, n_q, dt, dev, sh, bytes);
}

attnres_status_t attnres_read_bwd_workspace_size(int64_t n_src, int64_t T, int64_t d, int64_t n_q,
                                                attnres_dtype_t dt, size_t *bytes) {
    return read_bwd_workspace(n_src, T, d, 1, n_q, dt, bytes);
}

attnres_status_t attnres_read_bwd(const void *src, int64_t n_src, int64_t src_stride, int64_t T, int64_t d,
                                  attnres_dtype_t dt, const float *queries, int64_t n_q, const float *gain,
                                  float eps, const void *dout, void *dsrc, int64_t dsrc_stride, int accumulate,
                                  float *dqueries, float *dgain, void *workspace, size_t workspace_bytes,
                                  void *stream) {
    if (n_src > 16)
        return launch_read_bwd_many(src, n_src, src_stride, T, d, dt, queries, n_q, gain, eps, dout, nullptr, dsrc,
                                    dsrc_stride, accumulate, dqueries, dgain, workspace, workspace_bytes, stream);
    return launch_read_bwd(src, n_src, src_stride, T, d, 1, dt, queries, n_q, gain, eps, dout, nullptr, dsrc,
                           dsrc_stride,
                           accumulate, dqueries, dgain, workspace, workspace_bytes, stream);
}

attnres_status_t attnres_read_bwd_noalloc(const void *src, int64_t n_src, int64_t src_stride, int64_t T,
                                          int64_t d, attnres_dtype_t dt, const float *queries, int64_t n_q,
                                          const float *gain, float eps, const void *dout, void *dsrc,
                                          int64_t dsrc_stride, int accumulate, float *dqueries, float *dgain,
                                          void *stream) {
    // queries per pass: as many as the kernels take, unless their workspace
    // outgrows the scratch array; then passes of two, then of one
    int max_nqc = 0;
    if (T > 0) {
        size_t need = 0;
        attnres_status_t st = attnres_read_bwd_workspace_size(n_src, T, d, n_q, dt, &need);
        if (st != ATTNRES_OK) return st;
        if (need > kBwdScratchFloats * sizeof(float)) {
            DeviceInfo *dev = nullptr;
            st = device_info(&dev);
            if (st != ATTNRES_OK) return st;
            for (int cap = 2; cap >= 1 && max_nqc == 0; --cap) {
                ReadBwdShape sh;
                st = read_bwd_shape(n_src, d, n_q, 1, dt, &sh, cap);
                if (st != ATTNRES_OK) return st;
                size_t b = 0;
                st = read_bwd_ws_need(n_src, T, d, 1, n_q, dt, dev, sh, &b);
                if (st != ATTNRES_OK) return st;
                if (b <= kBwdScratchFloats * sizeof(float)) max_nqc = cap;
            }
            if (max_nqc == 0) return ATTNRES_ERR_UNSUPPORTED;
        }
    }
    void *ws = nullptr;
    attnres_status_t st = bwd_scratch(&ws);
    if (st != ATTNRES_OK) return st;
    return launch_read_bwd(src, n_src, src_stride, T, d, 1, dt, queries, n_q, gain, eps, dout, nullptr, dsrc,
                           dsrc_stride, accumulate, dqueries, dgain, ws, kBwdScratchFloats * sizeof(float), stream,
                           max_nqc);
}

attnres_status_t attnres_block_phase1_bwd(const void *src, int64_t n_src, int64_t src_stride, int64_t T,
                                          int64_t d, attnres_dtype_t dt, const float *queries, int64_t n_q,
                                          const float *gain, float eps, const void *d_o, const float *d_lse,
                                          void *dsrc, int64_t dsrc_stride, int accumulate, float *dqueries,
                                          float *dgain, void *workspace, size_t workspace_bytes, void *stream) {
    if (n_src > 16)
        return launch_read_bwd_many(src, n_src, src_stride, T, d, dt, queries, n_q, gain, eps, d_o, d_lse, dsrc,
                                    dsrc_stride, accumulate, dqueries, dgain, workspace, workspace_bytes, stream);
    return launch_read_bwd(src, n_src, src_stride, T, d, 1, dt, queries, n_q, gain, eps, d_o, d_lse, dsrc,
                           dsrc_stride, accumulate, dqueries, dgain, workspace, workspace_bytes, stream);
}

attnres_status_t attnres_block_phase2_bwd_workspace_size(int64_t T, int64_t d, attnres_dtype_t dt,
                                                        size_t *bytes) {
    if (!bytes || (dt != ATTNRES_F32 && dt != ATTNRES_BF16) || T < 0 || d < 1) return ATTNRES_ERR_INVALID_ARG;
    if (d % 8 != 0) return ATTNRES_ERR_UNSUPPORTED;
    DeviceInfo *dev = nullptr;
    attnres_status_t st = device_info(&dev);
    if (st != ATTNRES_OK) return st;
    MergeBwdShape sh;
    st = merge_bwd_shape(T, d, dt, dev, &sh);
    if (st != ATTNRES_OK) return st;
    *bytes = merge_bwd_ws_bytes(sh, d);
    return ATTNRES_OK;
}

attnres_status_t attnres_block_phase2_bwd(const void *o, const float *lse, const void *partial, int64_t T,
                                          int64_t d, attnres_dtype_t dt, const float *query, const float *gain,
                                          float eps, const void *dh, void *d_o, float *d_lse, void *d_partial,
                                          int accumulate, float *dquery, float *dgain, void *workspace,
                                          size_t workspace_bytes, void *stream) {
    return launch_merge_bwd(o, lse, partial, T, d, dt, query, gain, eps, dh, d_o, d_lse, d_partial, accumulate,
                            dquery, dgain, workspace, workspace_bytes, stream);
}

attnres_status_t mhar_read_bwd_workspace_size(int64_t n_src, int64_t T, int64_t d, int64_t H, int64_t n_q,
                                             attnres_dtype_t dt, size_t *bytes) {
    return read_bwd_workspace(n_src, T, d, H, n_q, dt, bytes);
}

attnres_status_t mhar_read_bwd(const void *src, int64_t n_src, int64_t src_stride, int64_t T, int64_t d,
                               int64_t H, attnres_dtype_t dt, const float *queries, int64_t n_q,
                               const float *gain, float eps, const void *dout, void *dsrc, int64_t dsrc_stride,
                               int accumulate, float *dqueries, float *dgain, void *workspace,
                               size_t workspace_bytes, void *stream) {
    return launch_read_bwd(src, n_src, src_stride, T, d, H, dt, queries, n_q, gain, eps, dout, nullptr, dsrc,
                           dsrc_stride,
                           accumulate, dqueries, dgain, workspace, workspace_bytes, stream);
}

attnres_status_t msar_expand_fwd(const void *src, int64_t n_src, int64_t src_stride, int64_t T,
                                 int64_t d, attnres_dtype_t dt, int64_t m, const int32_t *ksizes,
                                 const float *conv_w, const float *queries, const float *gain,
                                 float eps, const float *mix_gain, const float *mix_w, float mix_eps,
                                 void *out, void *stream) {
    return launch_msar_read(src, n_src, src_stride, 0, T, d, dt, m, ksizes, conv_w, queries, gain, eps,
                            mix_gain, mix_w, mix_eps, out, stream);
}

attnres_status_t msar_expand_fwd_chunk(const void *src, int64_t n_src, int64_t src_stride, int64_t T_prev,
                                       int64_t T, int64_t d, attnres_dtype_t dt, int64_t m,
                                       const int32_t *ksizes, const float *conv_w, const float *queries,
                                       const float *gain, float eps, const float *mix_gain,
                                       const float *mix_w, float mix_eps, void *out, void *stream) {
    if (T_prev < 0) return ATTNRES_ERR_INVALID_ARG;
    return launch_msar_read(src, n_src, src_stride, T_prev, T, d, dt, m, ksizes, conv_w, queries, gain, eps,
                            mix_gain, mix_w, mix_eps, out, stream);
}

attnres_status_t msar_expand_fwd_ps(const void *src, int64_t n_src, int64_t src_stride, int64_t T, int64_t d,
                                    attnres_dtype_t dt, int64_t m, const int32_t *ksizes, const float *conv_w,
                                    int64_t conv_src_stride, const float *queries, const float *gain, float eps,
                                    const float *mix_gain, const float *mix_w, float mix_eps, void *out,
                                    void *stream) {
    if (conv_src_stride <= 0) return ATTNRES_ERR_INVALID_ARG;
    return launch_msar_read(src, n_src, src_stride, 0, T, d, dt, m, ksizes, conv_w, queries, gain, eps, mix_gain,
                            mix_w, mix_eps, out, stream, conv_src_stride);
}

attnres_status_t msar_block_phase1(const void *src, int64_t n_src, int64_t src_stride, int64_t T, int64_t d,
                                   attnres_dtype_t dt, int64_t m, const int32_t *ksizes, const float *conv_w,
                                   const float *queries, int64_t S, const float *gain, float eps, void *o,
                                   float *lse, void *stream) {
    return launch_msar_phase1_host(src, n_src, src_stride, T, d, dt, m, ksizes, conv_w, queries, S, gain, eps, o,
                                   lse, stream);
}

attnres_status_t msar_block_phase2(const void *o, const float *lse, const void *partial, int64_t T, int64_t d,
                                   attnres_dtype_t dt, int64_t m, const int32_t *ksizes, const float *conv_w,
                                   const float *query, const float *gain, float eps, const float *mix_gain,
                                   const float *mix_w, float mix_eps, void *out, void *stream) {
    return launch_msar_phase2_host(o, lse, partial, T, d, dt, m, ksizes, conv_w, query, gain, eps, mix_gain, mix_w,
                                   mix_eps, out, stream);
}

attnres_status_t msar_expand_bwd_workspace_size(int64_t n_src, int64_t T, int64_t d, attnres_dtype_t dt, int64_t m,
                                               const int32_t *ksizes, size_t *bytes) {
    if (!bytes || (dt != ATTNRES_F32 && dt != ATTNRES_BF16) || n_src < 1 || T < 0 || d < 1)
        return ATTNRES_ERR_INVALID_ARG;
    attnres_status_t st = check_msar_kernels(m, ksizes);
    if (st != ATTNRES_OK) return st;
    if (T > 0 && d > INT64_MAX / T) return ATTNRES_ERR_INVALID_ARG;
    DeviceInfo *dev = nullptr;
    st = device_info(&dev);
    if (st != ATTNRES_OK) return st;
    MsarBwdPlan p;
    st = msar_bwd_plan(n_src, T, d, dt, ksizes, dev, &p);
    if (st != ATTNRES_OK) return st;
    *bytes = p.total;
    return ATTNRES_OK;
}

attnres_status_t msar_expand_bwd_ps(const void *src, int64_t n_src, int64_t src_stride, int64_t T, int64_t d,
                                    attnres_dtype_t dt, int64_t m, const int32_t *ksizes, const float *conv_w,
                                    int64_t conv_src_stride, const float *queries, const float *gain, float eps,
                                    const float *mix_gain, const float *mix_w, float mix_eps, const void *dh,
                                    void *dsrc, int64_t dsrc_stride, float *dconv_w, float *dqueries, float *dgain,
                                    float *dmix_gain, float *dmix_w, void *workspace, size_t workspace_bytes,
                                    void *stream) {
    if (conv_src_stride <= 0) return ATTNRES_ERR_INVALID_ARG;
    return launch_msar_bwd(src, n_src, src_stride, T, d, dt, m, ksizes, conv_w, queries, gain, eps, mix_gain,
                           mix_w, mix_eps, dh, dsrc, dsrc_stride, dconv_w, dqueries, dgain, dmix_gain, dmix_w,
                           workspace, workspace_bytes, stream, conv_src_stride);
}

attnres_status_t msar_expand_bwd(const void *src, int64_t n_src, int64_t src_stride, int64_t T, int64_t d,
                                 attnres_dtype_t dt, int64_t m, const int32_t *ksizes, const float *conv_w,
                                 const float *queries, const float *gain, float eps, const float *mix_gain,
                                 const float *mix_w, float mix_eps, const void *dh, void *dsrc,
                                 int64_t dsrc_stride, float *dconv_w, float *dqueries, float *dgain,
                                 float *dmix_gain, float *dmix_w, void *workspace, size_t workspace_bytes,
                                 void *stream) {
    return launch_msar_bwd(src, n_src, src_stride, T, d, dt, m, ksizes, conv_w, queries, gain, eps, mix_gain,
                           mix_w, mix_eps, dh, dsrc, dsrc_stride, dconv_w, dqueries, dgain, dmix_gain, dmix_w,
                           workspace, workspace_bytes, stream);
}

attnres_status_t msar_expand_bwd_chunk(const void *src, int64_t n_src, int64_t src_stride, int64_t T_prev,
                                       int64_t T, int64_t d, attnres_dtype_t dt, int64_t m, const int32_t *ksizes,
                                       const float *conv_w, const float *queries, const float *gain, float eps,
                                       const float *mix_gain, const float *mix_w, float mix_eps, const void *dh,
                                       void *dsrc, int64_t dsrc_stride, int accumulate, float *dconv_w,
                                       float *dqueries, float *dgain, float *dmix_gain, float *dmix_w,
                                       void *workspace, size_t workspace_bytes, void *stream) {
    return launch_msar_bwd(src, n_src, src_stride, T, d, dt, m, ksizes, conv_w, queries, gain, eps, mix_gain,
                           mix_w, mix_eps, dh, dsrc, dsrc_stride, dconv_w, dqueries, dgain, dmix_gain, dmix_w,
                           workspace, workspace_bytes, stream, 0, T_prev, accumulate);
}

attnres_status_t msar_expand_fwd_ws_workspace_size(int64_t n_src, int64_t T, int64_t d, attnres_dtype_t dt,
                                                  size_t *bytes) {
    if (!bytes || (dt != ATTNRES_F32 && dt != ATTNRES_BF16) || n_src < 1 || T < 0 || d < 1)
        return ATTNRES_ERR_INVALID_ARG;
    if (T > 0 && d > INT64_MAX / T) return ATTNRES_ERR_INVALID_ARG;
    if (d % 1024 != 0) return ATTNRES_ERR_UNSUPPORTED;
    *bytes = msar_fwd_ws_plan(n_src, T, d, dt, true, 0).total;
    return ATTNRES_OK;
}

attnres_status_t msar_expand_fwd_ws(const void *src, int64_t n_src, int64_t src_stride, int64_t T, int64_t d,
                                    attnres_dtype_t dt, int64_t m, const int32_t *ksizes, const float *conv_w,
                                    int64_t conv_src_stride, const float *queries, const float *gain, float eps,
                                    const float *mix_gain, const float *mix_w, float mix_eps, void *out,
                                    void *workspace, size_t workspace_bytes, void *stream) {
    return launch_msar_read_ws(src, n_src, src_stride, T, d, dt, m, ksizes, conv_w, conv_src_stride, queries, gain,
                               eps, mix_gain, mix_w, mix_eps, out, workspace, workspace_bytes, stream);
}

attnres_status_t msar_block_phase1_ws_workspace_size(int64_t n_src, int64_t T, int64_t d, attnres_dtype_t dt,
                                                    int64_t S, size_t *bytes) {
    if (!bytes || (dt != ATTNRES_F32 && dt != ATTNRES_BF16) || n_src < 1 || T < 0 || d < 1 || S < 1)
        return ATTNRES_ERR_INVALID_ARG;
    if (T > 0 && d > INT64_MAX / T) return ATTNRES_ERR_INVALID_ARG;
    if (d % 512 != 0) return ATTNRES_ERR_UNSUPPORTED;
    *bytes = msar_fwd_ws_plan(n_src, T, d, dt, false, S).total;
    return ATTNRES_OK;
}

attnres_status_t msar_block_phase1_ws(const void *src, int64_t n_src, int64_t src_stride, int64_t T, int64_t d,
                                      attnres_dtype_t dt, int64_t m, const int32_t *ksizes, const float *conv_w,
                                      const float *queries, int64_t S, const float *gain, float eps, void *o,
                                      float *lse, void *workspace, size_t workspace_bytes, void *stream) {
    return launch_msar_phase1_ws(src, n_src, src_stride, T, d, dt, m, ksizes, conv_w, queries, S, gain, eps, o, lse,
                                 workspace, workspace_bytes, stream);
}

attnres_status_t msar_block_phase2_ws_workspace_size(int64_t T, int64_t d, attnres_dtype_t dt, size_t *bytes) {
    if (!bytes || (dt != ATTNRES_F32 && dt != ATTNRES_BF16) || T < 0 || d < 1) return ATTNRES_ERR_INVALID_ARG;
    if (T > 0 && d > INT64_MAX / T) return ATTNRES_ERR_INVALID_ARG;
    if (d % 1024 != 0) return ATTNRES_ERR_UNSUPPORTED;
    *bytes = msar_fwd_ws_plan(1, T, d, dt, true, 0).total;
    return ATTNRES_OK;
}

attnres_status_t msar_block_phase2_ws(const void *o, const float *lse, const void *partial, int64_t T, int64_t d,
                                      attnres_dtype_t dt, int64_t m, const int32_t *ksizes, const float *conv_w,
                                      const float *query, const float *gain, float eps, const float *mix_gain,
                                      const float *mix_w, float mix_eps, void *out, void *workspace,
                                      size_t workspace_bytes, void *stream) {
    return launch_msar_phase2_ws(o, lse, partial, T, d, dt, m, ksizes, conv_w, query, gain, eps, mix_gain, mix_w,
                                 mix_eps, out, workspace, workspace_bytes, stream);
}

attnres_status_t msar_block_phase2_bwd_workspace_size(int64_t T, int64_t d, attnres_dtype_t dt, int64_t m,
                                                     const int32_t *ksizes, size_t *bytes) {
    if (!bytes || (dt != ATTNRES_F32 && dt != ATTNRES_BF16) || T < 0 || d < 1) return ATTNRES_ERR_INVALID_ARG;
    attnres_status_t st = check_msar_kernels(m, ksizes);
    if (st != ATTNRES_OK) return st;
    if (T > 0 && d > INT64_MAX / T) return ATTNRES_ERR_INVALID_ARG;
    DeviceInfo *dev = nullptr;
    st = device_info(&dev);
    if (st != ATTNRES_OK) return st;
    MsarTwoPhaseBwdPlan p;
    st = msar_two_phase_bwd_plan(true, 1, T, d, dt, ksizes, 0, dev, &p);
    if (st != ATTNRES_OK) return st;
    *bytes = p.total;
    return ATTNRES_OK;
}

attnres_status_t msar_block_phase2_bwd(const void *o, const float *lse, const void *partial, int64_t T, int64_t d,
                                       attnres_dtype_t dt, int64_t m, const int32_t *ksizes, const float *conv_w,
                                       const float *query, const float *gain, float eps, const float *mix_gain,
                                       const float *mix_w, float mix_eps, const void *dh, void *d_o, float *d_lse,
                                       void *d_partial, float *dconv_w, float *dquery, float *dgain,
                                       float *dmix_gain, float *dmix_w, void *workspace, size_t workspace_bytes,
                                       void *stream) {
    return launch_msar_phase2_bwd(o, lse, partial, T, d, dt, m, ksizes, conv_w, query, gain, eps, mix_gain, mix_w,
                                  mix_eps, dh, d_o, d_lse, d_partial, dconv_w, dquery, dgain, dmix_gain, dmix_w,
                                  workspace, workspace_bytes, stream);
}

attnres_status_t msar_block_phase1_bwd_workspace_size(int64_t n_src, int64_t T, int64_t d, attnres_dtype_t dt,
                                                     int64_t m, const int32_t *ksizes, int64_t S, size_t *bytes) {
    if (!bytes || (dt != ATTNRES_F32 && dt != ATTNRES_BF16) || n_src < 1 || T < 0 || d < 1 || S < 1)
        return ATTNRES_ERR_INVALID_ARG;
    attnres_status_t st = check_msar_kernels(m, ksizes);
    if (st != ATTNRES_OK) return st;
    if (T > 0 && d > INT64_MAX / T) return ATTNRES_ERR_INVALID_ARG;
    DeviceInfo *dev = nullptr;
    st = device_info(&dev);
    if (st != ATTNRES_OK) return st;
    MsarTwoPhaseBwdPlan p;
    st = msar_two_phase_bwd_plan(false, n_src, T, d, dt, ksizes, S, dev, &p);
    if (st != ATTNRES_OK) return st;
    *bytes = p.total;
    return ATTNRES_OK;
}

attnres_status_t msar_block_phase1_bwd(const void *src, int64_t n_src, int64_t src_stride, int64_t T, int64_t d,
                                       attnres_dtype_t dt, int64_t m, const int32_t *ksizes, const float *conv_w,
                                       const float *queries, int64_t S, const float *gain, float eps,
                                       const void *d_o, const float *d_lse, void *dsrc, int64_t dsrc_stride,
                                       float *dconv_w, float *dqueries, float *dgain, void *workspace,
                                       size_t workspace_bytes, void *stream) {
    return launch_msar_phase1_bwd(src, n_src, src_stride, T, d, dt, m, ksizes, conv_w, queries, S, gain, eps, d_o,
                                  d_lse, dsrc, dsrc_stride, dconv_w, dqueries, dgain, workspace, workspace_bytes,
                                  stream);
}

const char *attnres_status_string(attnres_status_t s) {
    switch (s) {
        case ATTNRES_OK: return "ok";
        case ATTNRES_ERR_INVALID_ARG: return "invalid argument";
        case ATTNRES_ERR_UNSUPPORTED: return "unsupported shape, alignment or size";
        case ATTNRES_ERR_CUDA: return "CUDA runtime error";
        case ATTNRES_ERR_TIMEOUT: return "a device-side wait ran out of time";
    }
    return "unknown status";
}

const char *attnres_last_cuda_error(void) { return t_last_err; }

attnres_status_t attnres_sync_status(void *stream) {
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    DeviceInfo *dev = nullptr;
    attnres_status_t st = device_info(&dev);
    if (st != ATTNRES_OK) return st;
    int v = 0;
    e = cudaMemcpy(&v, dev->status, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "read status word");
    if (v != 0) {
        const int zero = 0;
        e = cudaMemcpy(dev->status, &zero, sizeof(int), cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return cuda_fail(e, "clear status word");
        if (v & DEV_ERR_TIMEOUT) return ATTNRES_ERR_TIMEOUT;
    }
    return ATTNRES_OK;
}

void attnres_debug_set_wait_timeout_ns(uint64_t ns) {
    g_timeout_ns.store(ns ? ns : 2000000000ull);
}

void attnres_debug_set_stall_injection(int enable) { g_inject_stall.store(enable ? 1 : 0); }

void attnres_debug_set_kernel_variant(int variant) {
    g_kernel_variant.store(variant >= 1 && variant <= 3 ? variant : 0);
}

const char *attnres_version(void) { return "attnres 0.1.0 sm_103a"; }

}  // extern "C"
