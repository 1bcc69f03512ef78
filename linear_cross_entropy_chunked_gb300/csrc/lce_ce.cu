// Cross-entropy over logits the caller already holds (Z [N, ld], bf16, fp16 or fp32):
// per row the log-sum-exp, the loss lse - z_y, and optionally the gradient
// (softmax - onehot) * scale, written over Z or into a separate dZ. This is the
// row kernel of "Unsloth Kernel Architecture: Custom Triton Backpropagation and
// QLoRA Memory Scaling", section 1 "Fused Cross-Entropy Loss with Logit
// Streaming" (one row at a time, vocabulary blocks, a running max and a running
// sum of exponentials), with the gradient of "Unsloth Architecture: Manual
// Triton Backpropagation, Fused Cross-Entropy, and 80% VRAM Cut", pillar 1.
//
// Two kernels, chosen by the row's size:
//   * cluster kernel (a row fits in the registers of at most 8 CTAs of 512
//     threads: V up to 524288 bf16 / fp16 or 262144 fp32 logits): a cluster of CL CTAs
//     owns one row at a time, each CTA one contiguous segment of it, which a
//     bulk copy brings into shared memory and the threads then hold in
//     registers. Every logit is read from HBM once and written once: the max,
//     the exponentials, their sum and the gradient all come from registers, and
//     the CTAs of the cluster exchange their (max, sum) pairs through
//     distributed shared memory.
//   * streaming kernel (any row): one 1024-thread CTA per row and two passes
//     over global memory, the second mostly served by L2.
// Both use fixed reduction orders, so results are bit-reproducible.
#include <map>
#include <mutex>
#include <type_traits>

#include <cuda_fp16.h>

#include "lce_internal.h"
#include "lce_ptx.cuh"

namespace lce {

__device__ __forceinline__ float ce_warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float ce_warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// ------------------------------------------------------------------ streaming kernel
// Pass 1 streams the row with a running (max, sum of exponentials) per thread;
// pass 2 (gradient) streams it again. A persistent grid of the CTAs that fit
// at once walks the rows, so the few hundred rows in flight mostly stay in L2
// between the passes; each thread keeps CE_UNROLL 16-byte loads in flight.

constexpr int CE_THREADS = 1024;
constexpr int CE_UNROLL = 4;   // independent 16-byte loads in flight per thread

__device__ __forceinline__ void ce_merge(float &m, float &s, float m2, float s2) {
    const float M = fmaxf(m, m2);
    if (M == -INFINITY) return;
    s = s * exp2f((m - M) * LOG2E_F) + s2 * exp2f((m2 - M) * LOG2E_F);
    m = M;
}

template <typename T>
__device__ __forceinline__ int ce_vec_load(const T *row, long long i, float (&x)[8]);
template <>
__device__ __forceinline__ int ce_vec_load<__nv_bfloat16>(const __nv_bfloat16 *row, long long i,
                                                          float (&x)[8]) {
    const uint4 u = *reinterpret_cast<const uint4 *>(row + i);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[q]));
        x[2 * q] = f.x;
        x[2 * q + 1] = f.y;
    }
    return 8;
}
template <>
__device__ __forceinline__ int ce_vec_load<__half>(const __half *row, long long i, float (&x)[8]) {
    const uint4 u = *reinterpret_cast<const uint4 *>(row + i);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&w[q]));
        x[2 * q] = f.x;
        x[2 * q + 1] = f.y;
    }
    return 8;
}
template <>
__device__ __forceinline__ int ce_vec_load<float>(const float *row, long long i, float (&x)[8]) {
    const float4 a = *reinterpret_cast<const float4 *>(row + i);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    return 4;
}
template <typename T> __device__ __forceinline__ T ce_from_float(float v);
template <> __device__ __forceinline__ __nv_bfloat16 ce_from_float<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}
template <> __device__ __forceinline__ __half ce_from_float<__half>(float v) {
    return __float2half_rn(v);
}
template <> __device__ __forceinline__ float ce_from_float<float>(float v) { return v; }

template <typename T>
__global__ void __launch_bounds__(CE_THREADS, 2) lce_ce_logits_kernel(const CELogitsParams p) {
    constexpr int VEC = 16 / sizeof(T);
    constexpr int STEP = CE_THREADS * VEC;          // elements per block-wide sweep
    __shared__ float s_m[CE_THREADS / 32], s_s[CE_THREADS / 32];
    __shared__ float s_lse;
    const int t = threadIdx.x, w = t >> 5, l = t & 31;
    const int nv = p.hdr[HDR_NVALID];
    const long long vmain = (p.V / VEC) * VEC;     // vectorised part of a row
    const long long vunroll = (p.V / (STEP * CE_UNROLL)) * (STEP * CE_UNROLL);
    for (long long r = blockIdx.x; r < p.N; r += gridDim.x) {
        const T *row = static_cast<const T *>(p.Z) + r * p.ld;
        const long long yv = p.y[r];
        const bool y_ok = yv != p.ignore_index && yv >= 0 && yv < p.V;
        // the target logit is read before any thread can overwrite it (dZ == Z)
        const float zy = (t == 0 && y_ok) ? static_cast<float>(row[yv]) : 0.f;
        float m = -INFINITY, s = 0.f;
        // pass 1: running max and sum of exponentials
        for (long long i0 = static_cast<long long>(t) * VEC; i0 < vunroll; i0 += STEP * CE_UNROLL) {
            float x[CE_UNROLL][8];
#pragma unroll
            for (int u = 0; u < CE_UNROLL; ++u) ce_vec_load<T>(row, i0 + u * STEP, x[u]);
#pragma unroll
            for (int u = 0; u < CE_UNROLL; ++u) {
                float mv = x[u][0];
#pragma unroll
                for (int j = 1; j < VEC; ++j) mv = fmaxf(mv, x[u][j]);
                float sv = 0.f;
#pragma unroll
                for (int j = 0; j < VEC; ++j) sv += exp2f((x[u][j] - mv) * LOG2E_F);
                ce_merge(m, s, mv, sv);
            }
        }
        for (long long i = vunroll + static_cast<long long>(t) * VEC; i < vmain; i += STEP) {
            float x[8];
            ce_vec_load<T>(row, i, x);
            float mv = x[0];
#pragma unroll
            for (int j = 1; j < VEC; ++j) mv = fmaxf(mv, x[j]);
            float sv = 0.f;
#pragma unroll
            for (int j = 0; j < VEC; ++j) sv += exp2f((x[j] - mv) * LOG2E_F);
            ce_merge(m, s, mv, sv);
        }
        for (long long i = vmain + t; i < p.V; i += CE_THREADS) {
            const float x = static_cast<float>(row[i]);
            ce_merge(m, s, x, 1.f);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
            const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
            ce_merge(m, s, m2, s2);
        }
        if (l == 0) { s_m[w] = m; s_s[w] = s; }
        __syncthreads();
        if (w == 0) {
            m = (l < CE_THREADS / 32) ? s_m[l] : -INFINITY;
            s = (l < CE_THREADS / 32) ? s_s[l] : 0.f;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
                const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
                ce_merge(m, s, m2, s2);
            }
            if (l == 0) s_lse = m + logf(s);
        }
        __syncthreads();
        const float lse = s_lse;
        if (t == 0) {
            p.lse[r] = lse;
            p.loss_rows[r] = y_ok ? lse - zy : 0.f;
        }
        if (p.dZ) {
            // pass 2: (p - onehot) * scale in the logits' dtype
            const float scale = lce_row_scale(p.dloss, p.dloss_per_row, p.mean, nv, r, y_ok);
            const float lse2 = lse * LOG2E_F;
            T *drow = static_cast<T *>(p.dZ) + r * p.ld;
            for (long long i0 = static_cast<long long>(t) * VEC; i0 < vunroll;
                 i0 += STEP * CE_UNROLL) {
                float x[CE_UNROLL][8];
#pragma unroll
                for (int u = 0; u < CE_UNROLL; ++u) ce_vec_load<T>(row, i0 + u * STEP, x[u]);
#pragma unroll
                for (int u = 0; u < CE_UNROLL; ++u) {
                    const long long i = i0 + u * STEP;
                    T out[VEC];
#pragma unroll
                    for (int j = 0; j < VEC; ++j) {
                        float g = exp2f(fmaf(x[u][j], LOG2E_F, -lse2)) * scale;
                        if (i + j == yv) g -= scale;
                        out[j] = ce_from_float<T>(g);
                    }
                    *reinterpret_cast<uint4 *>(drow + i) = *reinterpret_cast<const uint4 *>(out);
                }
            }
            for (long long i = vunroll + static_cast<long long>(t) * VEC; i < vmain; i += STEP) {
                float x[8];
                ce_vec_load<T>(row, i, x);
                T out[VEC];
#pragma unroll
                for (int j = 0; j < VEC; ++j) {
                    float g = exp2f(fmaf(x[j], LOG2E_F, -lse2)) * scale;
                    if (i + j == yv) g -= scale;
                    out[j] = ce_from_float<T>(g);
                }
                *reinterpret_cast<uint4 *>(drow + i) = *reinterpret_cast<const uint4 *>(out);
            }
            for (long long i = vmain + t; i < p.V; i += CE_THREADS) {
                float g = exp2f(fmaf(static_cast<float>(row[i]), LOG2E_F, -lse2)) * scale;
                if (i == yv) g -= scale;
                drow[i] = ce_from_float<T>(g);
            }
        }
        __syncthreads();   // s_m / s_s / s_lse are reused by the next row
    }
}


// ------------------------------------------------------------------ cluster kernel
// A cluster of CL CTAs (1 to 8) owns one row at a time; rank k owns the
// contiguous segment [k * seg, min(V, (k + 1) * seg)) of it, seg a whole number
// of 16-byte vectors. Per row, in each CTA:
//   * a bulk copy has brought the segment into a shared-memory buffer; each
//     thread moves its vectors (thread t holds vectors t, t + 512, ...) into
//     registers, and as soon as all threads have, the buffer is refilled with
//     the segment of the row nbuf steps ahead, so every logit is read from HBM
//     once and the next copy overlaps this row's arithmetic;
//   * max over the registers (packed bf16 max for bf16 logits), block max;
//     exp(z - max) with packed fp32x2 arithmetic, kept in the same registers
//     (rounded to bf16 for bf16 logits), block sum;
//   * the CTA's (max, sum) pair goes to every CTA of the cluster with st.async,
//     which completes on the receiver's mbarrier without fencing this CTA's
//     earlier global stores;
//   * lse from the CL pairs, merged in rank order; gradient
//     (p - onehot) * scale = exp(z - max) * (exp(max - lse) * scale) - onehot * scale,
//     written with 16-byte stores.
// Elements past the segment's last whole vector (fewer than one vector, at the
// row's end only) are read and written in global memory directly.

constexpr int CEC_THREADS = 512;
constexpr int CEC_WARPS = CEC_THREADS / 32;
constexpr int CEC_MAX_CLUSTER = 8;
constexpr int CEC_MAX_BUF = 3;
constexpr int CEC_MAX_VPT = 16;                     // 16-byte vectors per thread
constexpr uint32_t CEC_COPY_BYTES = 32768;          // bytes per bulk copy instruction
constexpr uint64_t CEC_WAIT_NS = 2000000000ull;     // bound of every wait (2 s)

__device__ __forceinline__ void bulk_load_smem(uint32_t dst, const void *src, uint32_t bytes,
                                               uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}
__device__ __forceinline__ uint32_t cluster_id_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_count_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_size() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
// Stores (a, b) into the shared memory of a CTA of the cluster and completes 8
// bytes of transaction on that CTA's mbarrier `bar`.
__device__ __forceinline__ void st_async_f32x2(uint32_t addr, float a, float b, uint32_t bar) {
    asm volatile(
        "st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];" ::"r"(addr),
        "f"(a), "f"(b), "r"(bar)
        : "memory");
}
__device__ __forceinline__ float ce_ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// A 16-byte vector of logits seen as fp32 pairs.
template <typename T> struct CeVec;
template <> struct CeVec<__nv_bfloat16> {
    static constexpr int ELEMS = 8, PAIRS = 4;
    static constexpr uint32_t NEG_INF = 0xff80ff80u;   // two bf16 -inf
    __device__ static float2 pair(const uint4 &u, int q) {
        const uint32_t w = (&u.x)[q];
        return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
    }
    __device__ static void set_pair(uint4 &u, int q, float2 v) {
        __nv_bfloat162 h = __floats2bfloat162_rn(v.x, v.y);
        (&u.x)[q] = *reinterpret_cast<uint32_t *>(&h);
    }
};
template <> struct CeVec<__half> {
    static constexpr int ELEMS = 8, PAIRS = 4;
    static constexpr uint32_t NEG_INF = 0xfc00fc00u;   // two fp16 -inf
    __device__ static float2 pair(const uint4 &u, int q) {
        const uint32_t w = (&u.x)[q];
        return __half22float2(*reinterpret_cast<const __half2 *>(&w));
    }
    __device__ static void set_pair(uint4 &u, int q, float2 v) {
        __half2 h = __floats2half2_rn(v.x, v.y);
        (&u.x)[q] = *reinterpret_cast<uint32_t *>(&h);
    }
};
template <> struct CeVec<float> {
    static constexpr int ELEMS = 4, PAIRS = 2;
    static constexpr uint32_t NEG_INF = 0xff800000u;
    __device__ static float2 pair(const uint4 &u, int q) {
        return make_float2(__uint_as_float((&u.x)[2 * q]), __uint_as_float((&u.x)[2 * q + 1]));
    }
    __device__ static void set_pair(uint4 &u, int q, float2 v) {
        (&u.x)[2 * q] = __float_as_uint(v.x);
        (&u.x)[2 * q + 1] = __float_as_uint(v.y);
    }
};

template <typename T, int VPT>
__global__ void __launch_bounds__(CEC_THREADS, 1)
    lce_ce_logits_cluster_kernel(const CELogitsParams p, const long long seg, const int nbuf) {
    using CV = CeVec<T>;
    constexpr int EL = CV::ELEMS;
    extern __shared__ __align__(128) uint8_t ce_smem[];
    __shared__ __align__(8) uint64_t lbar[CEC_MAX_BUF];   // a segment copy landed
    __shared__ __align__(8) uint64_t xbar[2];             // all CL (max, sum) pairs landed
    __shared__ __align__(8) float2 xslot[2][CEC_MAX_CLUSTER];
    __shared__ float s_red_m[CEC_WARPS], s_red_s[CEC_WARPS];
    __shared__ int s_abort;

    const int t = threadIdx.x, w = t >> 5, l = t & 31;
    const uint32_t rank = cluster_ctarank(), cl = cluster_size();
    const long long cid = cluster_id_x(), ncl = cluster_count_x();
    const long long s0 = static_cast<long long>(rank) * seg;
    const long long s1 = s0 + seg < p.V ? s0 + seg : p.V;
    const int nvec = s1 > s0 ? static_cast<int>((s1 - s0) / EL) : 0;   // whole vectors
    const long long tail0 = s0 + static_cast<long long>(nvec) * EL;      // [tail0, s1): global
    const uint32_t bulk_bytes = static_cast<uint32_t>(nvec) * 16u;
    const uint32_t buf_bytes = static_cast<uint32_t>(seg * static_cast<long long>(sizeof(T)));
    const int nv = p.hdr[HDR_NVALID];
    const Abort ab{&s_abort, p.hdr, CEC_WAIT_NS};

    if (t == 0) {
        s_abort = 0;
        for (int b = 0; b < nbuf; ++b) mbar_init(&lbar[b], 1);
        mbar_init(&xbar[0], 1);
        mbar_init(&xbar[1], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    cluster_sync_all();   // every CTA's barriers exist before any peer signals them

    // thread 0: start the copies of the segment of the cluster's it-th row into buffer b
    long long issued = 0;
    auto issue = [&](long long it, int b) {
        const long long r = cid + it * ncl;
        if (r >= p.N) return;
        issued = it + 1;
        uint64_t *bar = &lbar[b];
        if (bulk_bytes == 0) {
            mbar_arrive(bar);
            return;
        }
        mbar_arrive_expect_tx(bar, bulk_bytes);
        const uint8_t *src =
            reinterpret_cast<const uint8_t *>(static_cast<const T *>(p.Z) + r * p.ld + s0);
        const uint32_t dst = smem_u32(ce_smem + static_cast<size_t>(b) * buf_bytes);
        for (uint32_t off = 0; off < bulk_bytes; off += CEC_COPY_BYTES) {
            const uint32_t n = bulk_bytes - off < CEC_COPY_BYTES ? bulk_bytes - off : CEC_COPY_BYTES;
            bulk_load_smem(dst + off, src + off, n, smem_u32(bar));
        }
    };
    if (t == 0)
        for (int j = 0; j < nbuf; ++j) issue(j, j);

    const float2 L2 = make_float2(LOG2E_F, LOG2E_F);
    int buf = 0, xs = 0;
    uint32_t lpar = 0, xpar = 0;
    bool bad = false, aborted = false;
    long long it = 0;
    long long y_next = cid < p.N ? p.y[cid] : 0;
    for (; cid + it * ncl < p.N; ++it) {
        const long long r = cid + it * ncl;
        const long long yv = y_next;
        if (r + ncl < p.N) y_next = p.y[r + ncl];
        bad |= !mbar_wait(&lbar[buf], lpar, ab);
        const uint4 *sg4 = reinterpret_cast<const uint4 *>(ce_smem + static_cast<size_t>(buf) * buf_bytes);
        const T *row = static_cast<const T *>(p.Z) + r * p.ld;
        const bool y_ok = yv != p.ignore_index && yv >= 0 && yv < p.V;
        const bool y_mine = y_ok && yv >= s0 && yv < s1;
        const int yl = y_mine ? static_cast<int>(yv - s0) : -1;   // target's index in the segment
        uint4 d[VPT];
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int v = t + k * CEC_THREADS;
            d[k] = v < nvec ? sg4[v] : make_uint4(CV::NEG_INF, CV::NEG_INF, CV::NEG_INF, CV::NEG_INF);
        }
        // the target logit is read before any thread can overwrite it (dZ == Z)
        float zy = 0.f;
        if (t == 0 && y_mine)
            zy = yv < tail0 ? static_cast<float>(reinterpret_cast<const T *>(sg4)[yl])
                            : static_cast<float>(row[yv]);
        if (t == 0) mbar_arrive_expect_tx(&xbar[xs], cl * 8u);

        // max of the segment
        float m = -INFINITY;
        if constexpr (std::is_same<T, __nv_bfloat16>::value) {
            __nv_bfloat162 mx2 = __floats2bfloat162_rn(-INFINITY, -INFINITY);
#pragma unroll
            for (int k = 0; k < VPT; ++k)
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    mx2 = __hmax2(mx2, *reinterpret_cast<const __nv_bfloat162 *>(&(&d[k].x)[q]));
            m = fmaxf(__low2float(mx2), __high2float(mx2));
        } else if constexpr (std::is_same<T, __half>::value) {
            __half2 mx2 = __floats2half2_rn(-INFINITY, -INFINITY);
#pragma unroll
            for (int k = 0; k < VPT; ++k)
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    mx2 = __hmax2(mx2, *reinterpret_cast<const __half2 *>(&(&d[k].x)[q]));
            m = fmaxf(__low2float(mx2), __high2float(mx2));
        } else {
#pragma unroll
            for (int k = 0; k < VPT; ++k)
                m = fmaxf(m, fmaxf(fmaxf(__uint_as_float(d[k].x), __uint_as_float(d[k].y)),
                                   fmaxf(__uint_as_float(d[k].z), __uint_as_float(d[k].w))));
        }
        for (long long i = tail0 + t; i < s1; i += CEC_THREADS) m = fmaxf(m, static_cast<float>(row[i]));
        m = ce_warp_max(m);
        if (l == 0) s_red_m[w] = m;
        // every thread holds its vectors: the buffer may be refilled; also the abort vote
        if (__syncthreads_or(bad)) {
            aborted = true;
            break;
        }
        if (t == 0) {
            fence_proxy_async_smem();
            issue(it + nbuf, buf);
        }
        m = ce_warp_max(l < CEC_WARPS ? s_red_m[l] : -INFINITY);

        // exp(z - max) in registers, and its sum
        const float2 nm2 = make_float2(-m * LOG2E_F, -m * LOG2E_F);
        float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
#pragma unroll
            for (int q = 0; q < CV::PAIRS; ++q) {
                const float2 a = __ffma2_rn(CV::pair(d[k], q), L2, nm2);
                const float2 e = make_float2(ce_ex2(a.x), ce_ex2(a.y));   // 0 for the -inf padding
                if (q & 1) acc1 = __fadd2_rn(acc1, e);
                else acc0 = __fadd2_rn(acc0, e);
                CV::set_pair(d[k], q, e);
            }
        }
        const float2 acc = __fadd2_rn(acc0, acc1);
        float s = acc.x + acc.y;
        for (long long i = tail0 + t; i < s1; i += CEC_THREADS)
            s += ce_ex2(fmaf(static_cast<float>(row[i]), LOG2E_F, nm2.x));
        s = ce_warp_sum(s);
        if (l == 0) s_red_s[w] = s;
        __syncthreads();
        s = ce_warp_sum(l < CEC_WARPS ? s_red_s[l] : 0.f);

        // exchange (max, sum) with the cluster; lane k of warp 0 serves rank k
        if (w == 0 && l < static_cast<int>(cl))
            st_async_f32x2(map_to_rank(&xslot[xs][rank], l), m, s, map_to_rank(&xbar[xs], l));
        const bool xok = mbar_wait_cluster(&xbar[xs], xpar, ab);
        bad |= !xok;
        if (xok) {
            // lane k holds rank k's pair; merged in rank order, then broadcast
            const float2 xv = l < static_cast<int>(cl) ? xslot[xs][l] : make_float2(-INFINITY, 0.f);
            float M = xv.x;
#pragma unroll
            for (int o = 4; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
            float S = xv.x == -INFINITY ? 0.f : xv.y * exp2f((xv.x - M) * LOG2E_F);
#pragma unroll
            for (int o = 4; o > 0; o >>= 1) S += __shfl_xor_sync(0xffffffffu, S, o);
            M = __shfl_sync(0xffffffffu, M, 0);
            S = __shfl_sync(0xffffffffu, S, 0);
            const float lse = M + logf(S);
            if (t == 0) {
                if (rank == 0) {
                    p.lse[r] = lse;
                    if (!y_ok) p.loss_rows[r] = 0.f;
                }
                if (y_mine) p.loss_rows[r] = lse - zy;
            }
            if (p.dZ) {
                const float scale = lce_row_scale(p.dloss, p.dloss_per_row, p.mean, nv, r, y_ok);
                const float f = exp2f((m - lse) * LOG2E_F) * scale;
                const float2 f2 = make_float2(f, f);
                T *drow = static_cast<T *>(p.dZ) + r * p.ld;
                uint4 *dvec = reinterpret_cast<uint4 *>(drow + s0);
                const int vy = yl >= 0 && yl < nvec * EL ? yl / EL : -1, jy = yl & (EL - 1);
#pragma unroll
                for (int k = 0; k < VPT; ++k) {
                    const int v = t + k * CEC_THREADS;
                    if (v < nvec) {
                        uint4 out;
#pragma unroll
                        for (int q = 0; q < CV::PAIRS; ++q) {
                            float2 g = __fmul2_rn(CV::pair(d[k], q), f2);
                            if (v == vy) {
                                if (2 * q == jy) g.x -= scale;
                                if (2 * q + 1 == jy) g.y -= scale;
                            }
                            CV::set_pair(out, q, g);
                        }
                        dvec[v] = out;
                    }
                }
                const float lse2 = lse * LOG2E_F;
                for (long long i = tail0 + t; i < s1; i += CEC_THREADS) {
                    float g = ce_ex2(fmaf(static_cast<float>(row[i]), LOG2E_F, -lse2)) * scale;
                    if (i == yv) g -= scale;
                    drow[i] = ce_from_float<T>(g);
                }
            }
        }
        if (++buf == nbuf) {
            buf = 0;
            lpar ^= 1u;
        }
        xs ^= 1;
        if (xs == 0) xpar ^= 1u;
    }
    aborted = __syncthreads_or(aborted || bad);
    if (aborted && t == 0) {
        // copies started for rows it .. issued - 1 may still be landing here
        for (long long j = it; j < issued; ++j)
            mbar_wait_drain(&lbar[j % nbuf], static_cast<uint32_t>((j / nbuf) & 1), CEC_WAIT_NS);
    }
    __syncthreads();
    cluster_sync_all();   // no CTA leaves while a peer may still write into its slots
}

// ------------------------------------------------------------------ launch

namespace {

using ClusterKernel = void (*)(const CELogitsParams, const long long, const int);

ClusterKernel cluster_kernel(int dtype, int vpt) {
    if (dtype == CE_FP32) {
        if (vpt == 4) return lce_ce_logits_cluster_kernel<float, 4>;
        if (vpt == 8) return lce_ce_logits_cluster_kernel<float, 8>;
        return lce_ce_logits_cluster_kernel<float, 16>;
    }
    if (dtype == CE_FP16) {
        if (vpt == 4) return lce_ce_logits_cluster_kernel<__half, 4>;
        if (vpt == 8) return lce_ce_logits_cluster_kernel<__half, 8>;
        return lce_ce_logits_cluster_kernel<__half, 16>;
    }
    if (vpt == 4) return lce_ce_logits_cluster_kernel<__nv_bfloat16, 4>;
    if (vpt == 8) return lce_ce_logits_cluster_kernel<__nv_bfloat16, 8>;
    return lce_ce_logits_cluster_kernel<__nv_bfloat16, 16>;
}

struct ClusterShape {
    int cl = 0, nbuf = 0, vpt = 0;
    long long seg = 0;
    size_t smem = 0;
};

int g_ce_max_dyn[64];   // per device: dynamic shared memory the cluster kernel may take

// The smallest cluster whose per-CTA segment fits in the registers of 512
// threads (at most 16 vectors each); then the fewest vectors per thread that
// hold it, and as many copy buffers (up to 3) as fit in shared memory.
bool cluster_shape(long long V, int dtype, int max_dyn, ClusterShape *o) {
    const long long elem = dtype == CE_FP32 ? 4 : 2, vec = 16 / elem;
    for (int cl = 1; cl <= CEC_MAX_CLUSTER; ++cl) {
        long long seg = (V + cl - 1) / cl;
        seg = (seg + vec - 1) / vec * vec;
        if (seg > CEC_THREADS * CEC_MAX_VPT * vec) continue;
        int vpt = 4;
        while (CEC_THREADS * vpt * vec < seg) vpt *= 2;
        const size_t bytes = static_cast<size_t>(seg * elem);
        const int nbuf = static_cast<int>(static_cast<size_t>(max_dyn) / bytes);
        if (nbuf < 1) continue;
        o->cl = cl;
        o->vpt = vpt;
        o->nbuf = nbuf < CEC_MAX_BUF ? nbuf : CEC_MAX_BUF;
        o->seg = seg;
        o->smem = o->nbuf * bytes;
        return true;
    }
    return false;
}

std::mutex g_occ_mu;
std::map<long long, int> g_occ;   // (device, kernel, cluster, smem) -> co-resident clusters

cudaError_t launch_cluster_kernel(const CELogitsParams &p, const ClusterShape &sh, int dev,
                                  bool *launched, cudaStream_t s) {
    *launched = false;
    const ClusterKernel fn = cluster_kernel(p.dtype, sh.vpt);
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = sh.cl;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(sh.cl);
    cfg.blockDim = dim3(CEC_THREADS);
    cfg.dynamicSmemBytes = sh.smem;
    cfg.stream = s;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    const long long key =
        (((static_cast<long long>(dev) * 4 + p.dtype) * 32 + sh.vpt) * 16 + sh.cl) *
            (1ll << 24) +
        static_cast<long long>(sh.smem);
    int nclusters = -1;
    {
        std::lock_guard<std::mutex> lock(g_occ_mu);
        auto f = g_occ.find(key);
        if (f != g_occ.end()) nclusters = f->second;
    }
    if (nclusters < 0) {
        if (cudaOccupancyMaxActiveClusters(&nclusters, fn, &cfg) != cudaSuccess) {
            cudaGetLastError();
            nclusters = 0;
        }
        std::lock_guard<std::mutex> lock(g_occ_mu);
        g_occ[key] = nclusters;
    }
    if (nclusters <= 0) return cudaSuccess;   // not launchable here: the caller streams
    const long long g = nclusters < p.N ? nclusters : p.N;
    cfg.gridDim = dim3(static_cast<unsigned>(g * sh.cl));
    *launched = true;
    return cudaLaunchKernelEx(&cfg, fn, p, sh.seg, sh.nbuf);
}

cudaError_t launch_streaming_kernel(const CELogitsParams &p, int sms, cudaStream_t s) {
    // a persistent grid of exactly the CTAs that fit at once (1024 threads each;
    // the rows in flight stay in L2 between the two passes)
    int per_sm = 1;
    cudaError_t e =
        p.dtype == CE_FP32
            ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, lce_ce_logits_kernel<float>,
                                                            CE_THREADS, 0)
        : p.dtype == CE_FP16
            ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, lce_ce_logits_kernel<__half>,
                                                            CE_THREADS, 0)
            : cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                  &per_sm, lce_ce_logits_kernel<__nv_bfloat16>, CE_THREADS, 0);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    long long grid = static_cast<long long>(per_sm) * sms;
    if (grid > p.N) grid = p.N;
    if (p.dtype == CE_FP32) lce_ce_logits_kernel<float><<<static_cast<int>(grid), CE_THREADS, 0, s>>>(p);
    else if (p.dtype == CE_FP16)
        lce_ce_logits_kernel<__half><<<static_cast<int>(grid), CE_THREADS, 0, s>>>(p);
    else lce_ce_logits_kernel<__nv_bfloat16><<<static_cast<int>(grid), CE_THREADS, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t ce_set_attributes() {
    int dev = 0, optin = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return e;
    int static_max = 0;
    for (int dt = 0; dt < 3; ++dt)
        for (int vpt = 4; vpt <= CEC_MAX_VPT; vpt *= 2) {
            cudaFuncAttributes fa{};
            e = cudaFuncGetAttributes(&fa, cluster_kernel(dt, vpt));
            if (e != cudaSuccess) return e;
            if (static_cast<int>(fa.sharedSizeBytes) > static_max) static_max = static_cast<int>(fa.sharedSizeBytes);
        }
    const int max_dyn = optin - static_max - 1024;
    for (int dt = 0; dt < 3; ++dt)
        for (int vpt = 4; vpt <= CEC_MAX_VPT; vpt *= 2) {
            e = cudaFuncSetAttribute(cluster_kernel(dt, vpt),
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, max_dyn);
            if (e != cudaSuccess) return e;
        }
    g_ce_max_dyn[dev] = max_dyn;
    return cudaSuccess;
}

cudaError_t launch_ce_logits(const CELogitsParams &p, int sms, cudaStream_t s) {
    if (p.N <= 0) return cudaSuccess;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    ClusterShape sh;
    if (dev >= 0 && dev < 64 && cluster_shape(p.V, p.dtype, g_ce_max_dyn[dev], &sh)) {
        bool launched = false;
        e = launch_cluster_kernel(p, sh, dev, &launched, s);
        if (e != cudaSuccess || launched) return e;
    }
    return launch_streaming_kernel(p, sms, s);
}

}  // namespace lce
