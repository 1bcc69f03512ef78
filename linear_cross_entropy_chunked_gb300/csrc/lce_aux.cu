// Bandwidth-bound kernels around the tensor-core GEMMs:
//   * label scan: N_valid and the out-of-range check; the valid-row count alone
//     (for sharded batches) and a given total count put in as the normaliser;
//   * slab merge (forward): per row, combine the (max, sumexp) partials of the
//     128-column slabs into lse_i = M + log sum_p s_p exp(m_p - M) and write the
//     row's loss lse_i - z_{i,y_i};
//   * prep (fused path, one launch per chunk): the merge's lse and row loss, then
//     the stored P' = exp(z - m_p) turned into
//     G = (P' exp(m_p - lse_i) - 1[j = y_i]) * dloss / N_valid in place, and the H
//     chunk transposed for the dW contraction
//     ("Unsloth Architecture: Manual Triton Backpropagation, Fused Cross-Entropy,
//     and 80% VRAM Cut", pillar 1: the loss -z_{i,y_i} + log sum_j e^{z_ij} and
//     the gradient p_ij - 1[j = y_i]);
//   * transpose of the H chunk alone (the separate backward);
//   * loss finalisation: fixed-order fp64 sum of the per-row losses / N_valid;
//   * dH combination: the fp32 parts of split dH contractions added in order.
// Every reduction has a fixed order, so results are bit-reproducible.
// Reductions of the loss: mean (sum / N_valid), sum, or none (the per-row losses
// are the output; G's rows are then scaled by a per-row dloss).
#include "lce_internal.h"
#include "lce_ptx.cuh"

namespace lce {

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// ------------------------------------------------------------------ label scan

__global__ void __launch_bounds__(1024) lce_label_scan_kernel(const long long *__restrict__ y,
                                                              long long N, long long V,
                                                              long long ign, int *hdr) {
    __shared__ int s_cnt[32];
    __shared__ int s_bad[32];
    int cnt = 0, bad = 0;
    for (long long i = blockIdx.x * 1024ll + threadIdx.x; i < N; i += 1024ll * gridDim.x) {
        const long long v = y[i];
        if (v != ign) {
            if (v >= 0 && v < V) ++cnt;
            else bad = 1;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
        bad |= __shfl_xor_sync(0xffffffffu, bad, o);
    }
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    if (l == 0) { s_cnt[w] = cnt; s_bad[w] = bad; }
    __syncthreads();
    if (w == 0) {
        cnt = s_cnt[l];
        bad = s_bad[l];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
            bad |= __shfl_xor_sync(0xffffffffu, bad, o);
        }
        if (l == 0) {
            if (cnt) atomicAdd(hdr + HDR_NVALID, cnt);   // integer: order-independent
            if (bad) atomicOr(hdr + HDR_FLAG, FLAG_LABEL);
        }
    }
}

// Count of rows with a label in [0, V) (the same rule as the scan above), written
// as an int64 to *out. One CTA: no atomics, no zeroing, a fixed summation order.
__global__ void __launch_bounds__(1024) lce_count_valid_kernel(const long long *__restrict__ y,
                                                               long long N, long long V,
                                                               long long ign, long long *out) {
    __shared__ long long s_cnt[32];
    long long cnt = 0;
    for (long long i = threadIdx.x; i < N; i += 1024) {
        const long long v = y[i];
        if (v != ign && v >= 0 && v < V) ++cnt;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    if (l == 0) s_cnt[w] = cnt;
    __syncthreads();
    if (w == 0) {
        cnt = s_cnt[l];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
        if (l == 0) *out = cnt;
    }
}

// The normaliser of the mean taken from the caller (the valid rows of every
// shard of a batch) instead of this call's own count; counts beyond the int32
// header word are clamped (the caller's API rejects them before this point).
__global__ void lce_set_nvalid_kernel(const long long *__restrict__ n_total, int *hdr) {
    const long long n = *n_total;
    hdr[HDR_NVALID] = n < 0 ? 0 : (n > 0x7fffffffll ? 0x7fffffff : static_cast<int>(n));
}

// ------------------------------------------------------------------ merge

constexpr int MERGE_THREADS = 256;

// lse of one chunk row from its (max, sumexp) slab partials, by a CTA of
// MERGE_THREADS threads: M = the maximum of the slab maxima, lse = M + log sum_p
// s_p exp(m_p - M). The order of every sum is fixed, so each CTA that computes a
// row's lse gets the same bits. Returns it in every thread.
__device__ __forceinline__ float row_lse(const float2 *parts, int nparts, float *s_red,
                                         float *s_bcast) {
    const int t = threadIdx.x, w = t >> 5, l = t & 31;
    float m = -INFINITY;
    for (int i = t; i < nparts; i += MERGE_THREADS) m = fmaxf(m, parts[i].x);
    m = warp_max(m);
    if (l == 0) s_red[w] = m;
    __syncthreads();
    if (w == 0) {
        m = (l < MERGE_THREADS / 32) ? s_red[l] : -INFINITY;
        m = warp_max(m);
        if (l == 0) *s_bcast = m;
    }
    __syncthreads();
    const float M = *s_bcast;
    const float M2 = M * LOG2E_F;
    float s = 0.f;
    for (int i = t; i < nparts; i += MERGE_THREADS) {
        const float2 q = parts[i];
        s += q.y * exp2f(fmaf(q.x, LOG2E_F, -M2));
    }
    s = warp_sum(s);
    __syncthreads();
    if (l == 0) s_red[w] = s;
    __syncthreads();
    if (w == 0) {
        s = (l < MERGE_THREADS / 32) ? s_red[l] : 0.f;
        s = warp_sum(s);
        if (l == 0) *s_bcast = M + logf(s);
    }
    __syncthreads();
    return *s_bcast;
}

// Forward: one CTA per chunk row, lse_i from the slab partials and the row's loss.
__global__ void __launch_bounds__(MERGE_THREADS) lce_merge_kernel(const MergeParams p) {
    __shared__ float s_red[MERGE_THREADS / 32];
    __shared__ float s_bcast;
    const int r = blockIdx.x;          // row within the chunk
    const int t = threadIdx.x;
    const float2 *parts = p.parts + static_cast<size_t>(r) * p.nparts;
    const float lse = row_lse(parts, p.nparts, s_red, &s_bcast);

    const int grow = p.row0 + r;
    const long long yv = p.y[grow];
    const bool y_ok = yv != p.ignore_index && yv >= 0 && yv < p.V;
    if (t == 0) {
        p.lse[grow] = lse;
        p.loss_rows[grow] = y_ok ? lse - p.zy[r] : 0.f;
    }
}

// ------------------------------------------------------------------ transpose
// 64 x 64 tiles of the H chunk [rows][D] into H^T [D][ld_t] (the K-major B
// operand of the dW contraction).

constexpr int TT = 64;
constexpr int TSTRIDE = 66;   // bf16 elements per staged row: conflict-free row writes, 2-way column reads

__global__ void __launch_bounds__(256) lce_transpose_kernel(const TransposeParams p) {
    __shared__ __align__(16) __nv_bfloat16 tile[TT * TSTRIDE];
    const int c0 = blockIdx.x * TT;      // first column of the tile
    const int r0 = blockIdx.y * TT;      // first chunk row of the tile
    const int tid = threadIdx.x;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int k = tid + 256 * i;
        const int rr = k >> 3, cb = (k & 7) * 8;
        const int r = r0 + rr, c = c0 + cb;
        uint4 u = make_uint4(0u, 0u, 0u, 0u);
        if (r < p.rows && c < p.cols)
            u = *reinterpret_cast<const uint4 *>(p.src + static_cast<size_t>(r) * p.ld_src + c);
        uint32_t *dst = reinterpret_cast<uint32_t *>(tile + rr * TSTRIDE + cb);
        dst[0] = u.x;
        dst[1] = u.y;
        dst[2] = u.z;
        dst[3] = u.w;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int k = tid + 256 * i;
        const int cc = k >> 3, rb = (k & 7) * 8;
        const int c = c0 + cc, r = r0 + rb;
        if (c < p.cols && r < p.rows) {
            uint32_t w[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint32_t lo = reinterpret_cast<const uint16_t &>(tile[(rb + 2 * q) * TSTRIDE + cc]);
                const uint32_t hi =
                    reinterpret_cast<const uint16_t &>(tile[(rb + 2 * q + 1) * TSTRIDE + cc]);
                w[q] = lo | (hi << 16);
            }
            *reinterpret_cast<uint4 *>(p.dst_t + static_cast<size_t>(c) * p.ld_t + r) =
                make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
}

// ------------------------------------------------------------------ prep
// Everything between a chunk's logits GEMM and its gradient GEMMs on the fused
// path in one launch. CTAs [0, rows * segs): row r = b / segs, segment b % segs
// of PREP_VEC_PER_CTA 8-column vectors: the row's lse from its slab partials
// (row_lse, the merge's arithmetic), then P' = exp(z - m_p) -> G = P' * exp(m_p -
// lse) * s - 1[j = y] * s in place, s the stored-G row scale, each slab's factor
// exp(m_p - lse) * s formed once per CTA into shared memory; segment 0 writes lse
// and the row loss. The CTAs after those transpose 64 x 64
// tiles of the H chunk (lce_transpose_kernel's arithmetic) for the dW contraction.
static_assert(PREP_THREADS == MERGE_THREADS, "the prep kernel computes lse as the merge does");
static_assert((PREP_VEC_PER_CTA * 8) % PART_COLS == 0 && PREP_VEC_PER_CTA * 8 / PART_COLS <= PREP_THREADS,
              "a prep segment starts on a slab boundary and each thread forms at most one factor");

__device__ __forceinline__ void bulk_copy_to_smem(uint32_t dst, const void *src, uint32_t bytes,
                                                  uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void transpose_tile(const TransposeParams &p, int c0, int r0,
                                               __nv_bfloat16 *tile) {
    const int tid = threadIdx.x;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int k = tid + 256 * i;
        const int rr = k >> 3, cb = (k & 7) * 8;
        const int r = r0 + rr, c = c0 + cb;
        uint4 u = make_uint4(0u, 0u, 0u, 0u);
        if (r < p.rows && c < p.cols)
            u = *reinterpret_cast<const uint4 *>(p.src + static_cast<size_t>(r) * p.ld_src + c);
        uint32_t *dst = reinterpret_cast<uint32_t *>(tile + rr * TSTRIDE + cb);
        dst[0] = u.x;
        dst[1] = u.y;
        dst[2] = u.z;
        dst[3] = u.w;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int k = tid + 256 * i;
        const int cc = k >> 3, rb = (k & 7) * 8;
        const int c = c0 + cc, r = r0 + rb;
        if (c < p.cols && r < p.rows) {
            uint32_t w[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint32_t lo = reinterpret_cast<const uint16_t &>(tile[(rb + 2 * q) * TSTRIDE + cc]);
                const uint32_t hi =
                    reinterpret_cast<const uint16_t &>(tile[(rb + 2 * q + 1) * TSTRIDE + cc]);
                w[q] = lo | (hi << 16);
            }
            *reinterpret_cast<uint4 *>(p.dst_t + static_cast<size_t>(c) * p.ld_t + r) =
                make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
}

constexpr uint32_t PREP_SEG_BYTES = PREP_VEC_PER_CTA * 16;       // 32 KB of P' per CTA
constexpr unsigned long long PREP_WAIT_NS = 2000000000ull;       // bound of the copy wait

// The segment of P' comes into shared memory by one bulk copy, issued first, so
// it is in flight while the row's lse is formed; shared memory rather than
// registers holds it, which lets 7 CTAs (224 KB of copies) share an SM.
__global__ void __launch_bounds__(MERGE_THREADS) lce_prep_kernel(const PrepParams p) {
    extern __shared__ __align__(128) uint8_t prep_smem[];   // the segment, or a transpose tile
    __shared__ float s_red[MERGE_THREADS / 32];
    __shared__ float s_bcast;
    __shared__ float s_fac[PREP_VEC_PER_CTA * 8 / PART_COLS];   // the segment's slab factors
    __shared__ __align__(8) uint64_t seg_bar;
    __shared__ volatile int s_abort;
    const MergeParams &m = p.m;
    const long long nrow_ctas = static_cast<long long>(m.rows) * p.segs;
    if (blockIdx.x >= nrow_ctas) {
        const int b = static_cast<int>(blockIdx.x - nrow_ctas);
        transpose_tile(p.tp, (b % p.tt_x) * TT, (b / p.tt_x) * TT,
                       reinterpret_cast<__nv_bfloat16 *>(prep_smem));
        return;
    }
    const int r = static_cast<int>(blockIdx.x / p.segs);
    const int seg = static_cast<int>(blockIdx.x % p.segs);
    const int nvec = (m.V + 7) >> 3;
    const int v0 = seg * PREP_VEC_PER_CTA;
    const int nv = min(PREP_VEC_PER_CTA, nvec - v0);      // > 0: segs covers nvec exactly
    uint4 *row = reinterpret_cast<uint4 *>(m.G + static_cast<size_t>(r) * p.ldg);
    if (threadIdx.x == 0) {
        s_abort = 0;
        mbar_init(&seg_bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        mbar_arrive_expect_tx(&seg_bar, static_cast<uint32_t>(nv) * 16u);
        bulk_copy_to_smem(smem_u32(prep_smem), row + v0, static_cast<uint32_t>(nv) * 16u,
                          smem_u32(&seg_bar));
    }
    // (row_lse's block barriers also order the barrier's initialisation before the waits)
    const float2 *parts = m.parts + static_cast<size_t>(r) * m.nparts;
    const float lse = row_lse(parts, m.nparts, s_red, &s_bcast);
    const int grow = m.row0 + r;
    const long long yv = m.y[grow];
    const bool y_ok = yv != m.ignore_index && yv >= 0 && yv < m.V;
    if (seg == 0 && threadIdx.x == 0) {
        m.lse[grow] = lse;
        m.loss_rows[grow] = y_ok ? lse - m.zy[r] : 0.f;
    }
    const float scale = lce_store_scale(m.dloss, m.dloss_per_row, m.mean, m.hdr[HDR_NVALID], grow,
                                        y_ok, m.f16);
    const float lse2 = lse * LOG2E_F;
    const int ycol = y_ok ? static_cast<int>(yv) : -1;
    // the factor exp(m_p - lse) * s of each 128-column slab of the segment, once (a
    // segment starts on a slab boundary: PREP_VEC_PER_CTA * 8 is a multiple of 128)
    const int slab0 = (v0 * 8) / PART_COLS;
    const int nslab = (nv * 8 + PART_COLS - 1) / PART_COLS;
    if (threadIdx.x < nslab)
        s_fac[threadIdx.x] = scale != 0.f
                                 ? exp2f(fmaf(parts[slab0 + threadIdx.x].x, LOG2E_F, -lse2)) * scale
                                 : 0.f;
    __syncthreads();
    const Abort ab{&s_abort, const_cast<int *>(m.hdr), PREP_WAIT_NS};
    if (!mbar_wait(&seg_bar, 0, ab)) {
        // the copy did not complete in time (recorded as a timeout): let it finish
        // (bounded) before the CTA's shared memory is released
        mbar_wait_drain(&seg_bar, 0, PREP_WAIT_NS);
        return;
    }
    const uint4 *sv = reinterpret_cast<const uint4 *>(prep_smem);
#pragma unroll 4
    for (int v = threadIdx.x; v < nv; v += MERGE_THREADS) {
        uint4 u = sv[v];
        const int c = (v0 + v) * 8;
        const float f = s_fac[(v * 8) / PART_COLS];
        uint32_t *wv = reinterpret_cast<uint32_t *>(&u);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            float2 x;
            if (m.f16) x = __half22float2(*reinterpret_cast<__half2 *>(&wv[q]));
            else x = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162 *>(&wv[q]));
            x.x *= f;
            x.y *= f;
            if (c + 2 * q == ycol) x.x -= scale;
            if (c + 2 * q + 1 == ycol) x.y -= scale;
            if (m.f16) {
                __half2 h = __floats2half2_rn(x.x, x.y);
                wv[q] = *reinterpret_cast<uint32_t *>(&h);
            } else {
                __nv_bfloat162 h = __floats2bfloat162_rn(x.x, x.y);
                wv[q] = *reinterpret_cast<uint32_t *>(&h);
            }
        }
        row[v0 + v] = u;
    }
}

// ------------------------------------------------------------------ loss

__global__ void __launch_bounds__(1024) lce_loss_finalize_kernel(const float *__restrict__ loss_rows,
                                                                 long long N, const int *hdr,
                                                                 float *loss, int mean) {
    __shared__ double s_red[32];
    double s = 0.0;
    for (long long i = threadIdx.x; i < N; i += 1024) s += static_cast<double>(loss_rows[i]);
    s = warp_sum_d(s);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    if (l == 0) s_red[w] = s;
    __syncthreads();
    if (w == 0) {
        s = s_red[l];
        s = warp_sum_d(s);
        if (l == 0) {
            const int nv = hdr[HDR_NVALID];
            if (mean) *loss = nv > 0 ? static_cast<float>(s / nv) : 0.f;
            else *loss = static_cast<float>(s);
        }
    }
}

// ------------------------------------------------------------------ dH combination
// dst[rows][D] (bf16, or fp16 when F16) = (ACC ? dst : 0) + the fp32 partial
// sums src[s][rows][D], s = 0 .. splits-1 added in that order, rounded once. The
// fixed order keeps dH bit-reproducible whatever the schedule of the tiles that
// wrote the partials.
template <bool F16, bool ACC>
__global__ void __launch_bounds__(256) lce_combine_dh_kernel(const float *__restrict__ src,
                                                            int splits, long long stride,
                                                            void *__restrict__ dst_, long long nvec) {
    uint4 *dst = static_cast<uint4 *>(dst_);
    for (long long i = blockIdx.x * 256ll + threadIdx.x; i < nvec; i += 256ll * gridDim.x) {
        float4 a = reinterpret_cast<const float4 *>(src)[2 * i];
        float4 b = reinterpret_cast<const float4 *>(src)[2 * i + 1];
        for (int sp = 1; sp < splits; ++sp) {
            const float4 *q = reinterpret_cast<const float4 *>(src + sp * stride);
            const float4 c = q[2 * i], e = q[2 * i + 1];
            a.x += c.x; a.y += c.y; a.z += c.z; a.w += c.w;
            b.x += e.x; b.y += e.y; b.z += e.z; b.w += e.w;
        }
        const float s[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        uint4 d = ACC ? dst[i] : make_uint4(0, 0, 0, 0);
        uint32_t *w = &d.x;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            if constexpr (F16) {
                float2 x = make_float2(0.f, 0.f);
                if constexpr (ACC) x = __half22float2(*reinterpret_cast<__half2 *>(&w[q]));
                __half2 h = __floats2half2_rn(x.x + s[2 * q], x.y + s[2 * q + 1]);
                w[q] = *reinterpret_cast<uint32_t *>(&h);
            } else {
                float lo = s[2 * q], hi = s[2 * q + 1];
                if constexpr (ACC) {
                    lo += __uint_as_float(w[q] << 16);
                    hi += __uint_as_float(w[q] & 0xffff0000u);
                }
                __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
                w[q] = *reinterpret_cast<uint32_t *>(&h);
            }
        }
        dst[i] = d;
    }
}

// ------------------------------------------------------------------ bounded-wait self-test
// One warp waits, with the same bounded wait the pipelines use, on an mbarrier
// that nothing signals; the wait runs out after limit_ns, records FLAG_TIMEOUT in
// the workspace header and the kernel returns. Lets a test check, on the GPU,
// that a stuck pipeline ends as a status instead of a hang.
__global__ void __launch_bounds__(32) lce_wait_selftest_kernel(int *hdr, unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int s_abort;
    if (threadIdx.x == 0) {
        s_abort = 0;
        mbar_init(&bar, 1);   // expects one arrival that never comes
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    const Abort ab{&s_abort, hdr, limit_ns};
    mbar_wait(&bar, 0, ab);
}

// ------------------------------------------------------------------ launchers

cudaError_t launch_label_scan(const long long *y, long long N, long long V, long long ign, int *hdr,
                              cudaStream_t s) {
    long long blocks = (N + 1023) / 1024;
    if (blocks < 1) blocks = 1;
    if (blocks > 64) blocks = 64;
    lce_label_scan_kernel<<<static_cast<int>(blocks), 1024, 0, s>>>(y, N, V, ign, hdr);
    return cudaGetLastError();
}

cudaError_t launch_count_valid(const long long *y, long long N, long long V, long long ign,
                               long long *out, cudaStream_t s) {
    lce_count_valid_kernel<<<1, 1024, 0, s>>>(y, N, V, ign, out);
    return cudaGetLastError();
}

cudaError_t launch_set_nvalid(const long long *n_total, int *hdr, cudaStream_t s) {
    lce_set_nvalid_kernel<<<1, 1, 0, s>>>(n_total, hdr);
    return cudaGetLastError();
}

cudaError_t launch_merge(const MergeParams &p, cudaStream_t s) {
    if (p.rows <= 0) return cudaSuccess;
    lce_merge_kernel<<<p.rows, MERGE_THREADS, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_transpose(const TransposeParams &p, cudaStream_t s) {
    if (p.rows <= 0 || p.cols <= 0) return cudaSuccess;
    const dim3 grid((p.cols + TT - 1) / TT, (p.rows + TT - 1) / TT);
    lce_transpose_kernel<<<grid, 256, 0, s>>>(p);
    return cudaGetLastError();
}


cudaError_t launch_prep(const PrepParams &p, cudaStream_t s) {
    const long long row_ctas = static_cast<long long>(p.m.rows) * p.segs;
    const long long tt = p.tp.rows > 0 ? static_cast<long long>(p.tt_x) * ((p.tp.rows + TT - 1) / TT)
                                       : 0;
    const long long grid = row_ctas + tt;
    if (grid <= 0) return cudaSuccess;
    if (grid > 0x7fffffffll) return cudaErrorInvalidValue;
    lce_prep_kernel<<<static_cast<unsigned>(grid), MERGE_THREADS, PREP_SEG_BYTES, s>>>(p);
    return cudaGetLastError();
}

cudaError_t aux_set_attributes() { return cudaSuccess; }

cudaError_t launch_wait_selftest(int *hdr, unsigned long long limit_ns, cudaStream_t s) {
    lce_wait_selftest_kernel<<<1, 32, 0, s>>>(hdr, limit_ns);
    return cudaGetLastError();
}

cudaError_t launch_combine_dh(const float *src, int splits, long long stride, void *dst,
                              long long n, bool f16, bool accumulate, int sms, cudaStream_t s) {
    const long long nvec = n / 8;
    if (nvec <= 0) return cudaSuccess;
    long long blocks = (nvec + 255) / 256;
    if (blocks > 8ll * sms) blocks = 8ll * sms;
    const int g = static_cast<int>(blocks);
    if (splits < 1) splits = 1;
    if (f16 && accumulate) lce_combine_dh_kernel<true, true><<<g, 256, 0, s>>>(src, splits, stride, dst, nvec);
    else if (f16) lce_combine_dh_kernel<true, false><<<g, 256, 0, s>>>(src, splits, stride, dst, nvec);
    else if (accumulate) lce_combine_dh_kernel<false, true><<<g, 256, 0, s>>>(src, splits, stride, dst, nvec);
    else lce_combine_dh_kernel<false, false><<<g, 256, 0, s>>>(src, splits, stride, dst, nvec);
    return cudaGetLastError();
}

cudaError_t launch_loss_finalize(const float *loss_rows, long long N, const int *hdr, float *loss,
                                 int mean, cudaStream_t s) {
    lce_loss_finalize_kernel<<<1, 1024, 0, s>>>(loss_rows, N, hdr, loss, mean);
    return cudaGetLastError();
}

}  // namespace lce
