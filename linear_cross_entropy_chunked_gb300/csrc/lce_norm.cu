// The final RMSNorm in front of the LM head, forward and backward
// ("Unsloth Architecture: Manual Triton Backpropagation, Fused Cross-Entropy,
// and 80% VRAM Cut", pillar 3 "Fused RMSNorm & SwiGLU Kernels"):
//
//   h  = x * r * gamma,                 r = 1 / sqrt(mean_i x_i^2 + eps)
//   dx = r * (gamma * dh) - x * r^3 * (sum_i gamma_i dh_i x_i) / D
//   dgamma = sum over rows of dh * x * r
//
// The page prints the backward with gamma outside the inner sum; that form is
// exact only when gamma is the same for every channel, so the kernels compute
// the exact derivative above.
//
// Both kernels are HBM-bound row kernels. A persistent grid of 256-thread CTAs
// walks the rows; thread t holds the 16-byte vectors t, t + 256, ... of a row
// in registers, so each input is read once, and the row sums come from one
// block reduction per row (two slots alternate, so one barrier per row). The
// next row's loads are issued before the current row's reduction. The
// backward recomputes r from x inside the same reduction: nothing but X is kept
// from the forward. dgamma: each CTA sums its rows' dh * x * r per column in
// registers and adds that to its own slot of a partials array (a fixed number
// of CTAs, so the same slot receives the same rows on every call); a last
// kernel adds the slots in a fixed order. Results are bit-reproducible.
#include "lce_internal.h"

namespace lce {

namespace {

__device__ __forceinline__ void bf16x8_to_f32(const uint4 &u, float (&x)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        x[2 * q] = __uint_as_float(w[q] << 16);
        x[2 * q + 1] = __uint_as_float(w[q] & 0xffff0000u);
    }
}

__device__ __forceinline__ uint4 f32x8_to_bf16(const float (&x)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        __nv_bfloat162 h = __floats2bfloat162_rn(x[2 * q], x[2 * q + 1]);
        w[q] = *reinterpret_cast<uint32_t *>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ float nrm_warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

constexpr int NRM_WARPS = NRM_THREADS / 32;

// Loads this thread's vectors of row r (zero past D).
template <int VPT>
__device__ __forceinline__ void load_row_bf16(const __nv_bfloat16 *base, long long r, int D, int t,
                                              uint4 (&u)[VPT]) {
    const uint4 *row = reinterpret_cast<const uint4 *>(base + r * D);
    const int nvec = D / 8;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int v = t + k * NRM_THREADS;
        u[k] = v < nvec ? row[v] : make_uint4(0, 0, 0, 0);
    }
}

// fp32 dH: the sum of `splits` partial arrays `stride` elements apart, added in
// order (a split dH contraction leaves its vocabulary parts there)
template <int VPT, bool DH32>
__device__ __forceinline__ void load_row_dh(const void *base, long long r, int D, int t,
                                            float (&dh)[VPT][8], int splits, long long stride) {
    const int nvec = D / 8;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int v = t + k * NRM_THREADS;
        const bool in = v < nvec;
        if constexpr (DH32) {
            const float *row = static_cast<const float *>(base) + r * D;
            float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
            if (in) {
                a = reinterpret_cast<const float4 *>(row)[2 * v];
                b = reinterpret_cast<const float4 *>(row)[2 * v + 1];
                for (int sp = 1; sp < splits; ++sp) {
                    const float4 *q = reinterpret_cast<const float4 *>(row + sp * stride);
                    const float4 c = q[2 * v], e = q[2 * v + 1];
                    a.x += c.x; a.y += c.y; a.z += c.z; a.w += c.w;
                    b.x += e.x; b.y += e.y; b.z += e.z; b.w += e.w;
                }
            }
            dh[k][0] = a.x; dh[k][1] = a.y; dh[k][2] = a.z; dh[k][3] = a.w;
            dh[k][4] = b.x; dh[k][5] = b.y; dh[k][6] = b.z; dh[k][7] = b.w;
        } else {
            const uint4 *dr = reinterpret_cast<const uint4 *>(
                static_cast<const __nv_bfloat16 *>(base) + r * D);
            bf16x8_to_f32(in ? dr[v] : make_uint4(0, 0, 0, 0), dh[k]);
        }
    }
}

// Rows r = blockIdx.x, + gridDim.x, ...; the next row's loads are issued before
// the current row's reduction, so two rows are in flight per CTA.
template <int VPT>
__global__ void __launch_bounds__(NRM_THREADS) lce_rmsnorm_fwd_kernel(const NormParams p) {
    __shared__ float red[2][NRM_WARPS];
    const int t = threadIdx.x, w = t >> 5, l = t & 31;
    const int nvec = p.D / 8;
    float g[VPT][8];
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int v = t + k * NRM_THREADS;
        uint4 u = v < nvec ? reinterpret_cast<const uint4 *>(p.gamma)[v] : make_uint4(0, 0, 0, 0);
        bf16x8_to_f32(u, g[k]);
    }
    int slot = 0;
    long long r = blockIdx.x;
    uint4 cur[VPT];
    if (r < p.rows) load_row_bf16<VPT>(p.X, r, p.D, t, cur);
    for (; r < p.rows; r += gridDim.x) {
        uint4 nxt[VPT];
        if (r + gridDim.x < p.rows) load_row_bf16<VPT>(p.X, r + gridDim.x, p.D, t, nxt);
        float ss = 0.f;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            float x[8];
            bf16x8_to_f32(cur[k], x);
#pragma unroll
            for (int j = 0; j < 8; ++j) ss = fmaf(x[j], x[j], ss);
        }
        ss = nrm_warp_sum(ss);
        if (l == 0) red[slot][w] = ss;
        __syncthreads();
        ss = 0.f;
#pragma unroll
        for (int i = 0; i < NRM_WARPS; ++i) ss += red[slot][i];
        slot ^= 1;
        const float rstd = rsqrtf(ss / static_cast<float>(p.D) + p.eps);
        uint4 *hr = reinterpret_cast<uint4 *>(p.H + r * p.D);
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int v = t + k * NRM_THREADS;
            if (v < nvec) {
                float x[8], h[8];
                bf16x8_to_f32(cur[k], x);
#pragma unroll
                for (int j = 0; j < 8; ++j) h[j] = x[j] * rstd * g[k][j];
                hr[v] = f32x8_to_bf16(h);
            }
        }
        if (p.rstd && t == 0) p.rstd[r] = rstd;
#pragma unroll
        for (int k = 0; k < VPT; ++k) cur[k] = nxt[k];
    }
}

template <int VPT, bool DH32>
__global__ void __launch_bounds__(NRM_THREADS) lce_rmsnorm_bwd_kernel(const NormParams p) {
    __shared__ float2 red[2][NRM_WARPS];
    const int t = threadIdx.x, w = t >> 5, l = t & 31;
    const int nvec = p.D / 8;
    float g[VPT][8], acc[VPT][8];
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int v = t + k * NRM_THREADS;
        uint4 u = v < nvec ? reinterpret_cast<const uint4 *>(p.gamma)[v] : make_uint4(0, 0, 0, 0);
        bf16x8_to_f32(u, g[k]);
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[k][j] = 0.f;
    }
    int slot = 0;
    long long r = blockIdx.x;
    uint4 xc[VPT];
    float dc[VPT][8];
    if (r < p.rows) {
        load_row_bf16<VPT>(p.X, r, p.D, t, xc);
        load_row_dh<VPT, DH32>(p.dH, r, p.D, t, dc, p.dh_splits, p.dh_split_stride);
    }
    for (; r < p.rows; r += gridDim.x) {
        uint4 xn[VPT];
        float dn[VPT][8];
        if (r + gridDim.x < p.rows) {
            load_row_bf16<VPT>(p.X, r + gridDim.x, p.D, t, xn);
            load_row_dh<VPT, DH32>(p.dH, r + gridDim.x, p.D, t, dn, p.dh_splits,
                                        p.dh_split_stride);
        }
        float ss = 0.f, dot = 0.f;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            float x[8];
            bf16x8_to_f32(xc[k], x);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                ss = fmaf(x[j], x[j], ss);
                dot = fmaf(g[k][j] * dc[k][j], x[j], dot);
            }
        }
        ss = nrm_warp_sum(ss);
        dot = nrm_warp_sum(dot);
        if (l == 0) red[slot][w] = make_float2(ss, dot);
        __syncthreads();
        ss = 0.f;
        dot = 0.f;
#pragma unroll
        for (int i = 0; i < NRM_WARPS; ++i) {
            ss += red[slot][i].x;
            dot += red[slot][i].y;
        }
        slot ^= 1;
        const float invd = 1.f / static_cast<float>(p.D);
        const float rstd = rsqrtf(ss * invd + p.eps);
        const float cx = rstd * rstd * rstd * dot * invd;
        uint4 *dxr = reinterpret_cast<uint4 *>(p.dX + r * p.D);
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int v = t + k * NRM_THREADS;
            if (v < nvec) {
                float x[8], dx[8];
                bf16x8_to_f32(xc[k], x);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    dx[j] = fmaf(rstd * g[k][j], dc[k][j], -x[j] * cx);
                    acc[k][j] = fmaf(dc[k][j] * x[j], rstd, acc[k][j]);
                }
                dxr[v] = f32x8_to_bf16(dx);
            }
        }
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            xc[k] = xn[k];
#pragma unroll
            for (int j = 0; j < 8; ++j) dc[k][j] = dn[k][j];
        }
    }
    // this CTA's dgamma partial: its own slot, added to what earlier calls left
    float *slot_row = p.part + static_cast<long long>(blockIdx.x) * p.D;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int v = t + k * NRM_THREADS;
        if (v < nvec) {
            float4 *o = reinterpret_cast<float4 *>(slot_row + 8 * v);
            float4 a = p.first ? make_float4(0.f, 0.f, 0.f, 0.f) : o[0];
            float4 b = p.first ? make_float4(0.f, 0.f, 0.f, 0.f) : o[1];
            a.x += acc[k][0]; a.y += acc[k][1]; a.z += acc[k][2]; a.w += acc[k][3];
            b.x += acc[k][4]; b.y += acc[k][5]; b.z += acc[k][6]; b.w += acc[k][7];
            o[0] = a;
            o[1] = b;
        }
    }
}

// dgamma[j] = sum over the NRM_GRID slots, in slot order.
__global__ void __launch_bounds__(256) lce_dgamma_reduce_kernel(const float *part, int D,
                                                               float *dgamma) {
    const int j = blockIdx.x * 256 + threadIdx.x;
    if (j >= D) return;
    float s = 0.f;
    for (int b = 0; b < NRM_GRID; ++b) s += part[static_cast<long long>(b) * D + j];
    dgamma[j] = s;
}

// The forward keeps no per-CTA state across rows, so it takes one CTA per row
// (up to 2048, then rows are strided): a chunk's rows are all in flight at once.
template <int VPT>
cudaError_t launch_fwd_vpt(const NormParams &p, cudaStream_t s) {
    const int grid = p.rows < 2048 ? static_cast<int>(p.rows) : 2048;
    lce_rmsnorm_fwd_kernel<VPT><<<grid, NRM_THREADS, 0, s>>>(p);
    return cudaGetLastError();
}

template <int VPT>
cudaError_t launch_bwd_vpt(const NormParams &p, cudaStream_t s) {
    if (p.dh_fp32) lce_rmsnorm_bwd_kernel<VPT, true><<<NRM_GRID, NRM_THREADS, 0, s>>>(p);
    else lce_rmsnorm_bwd_kernel<VPT, false><<<NRM_GRID, NRM_THREADS, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_rmsnorm_fwd(const NormParams &p, cudaStream_t s) {
    if (p.rows <= 0) return cudaSuccess;
    const int vpt = (p.D / 8 + NRM_THREADS - 1) / NRM_THREADS;
    if (vpt <= 1) return launch_fwd_vpt<1>(p, s);
    if (vpt <= 2) return launch_fwd_vpt<2>(p, s);
    return launch_fwd_vpt<4>(p, s);
}

cudaError_t launch_rmsnorm_bwd(const NormParams &p, cudaStream_t s) {
    // runs even with no rows: every CTA still initialises / keeps its partial slot
    const int vpt = (p.D / 8 + NRM_THREADS - 1) / NRM_THREADS;
    if (vpt <= 1) return launch_bwd_vpt<1>(p, s);
    if (vpt <= 2) return launch_bwd_vpt<2>(p, s);
    return launch_bwd_vpt<4>(p, s);
}

cudaError_t launch_dgamma_reduce(const float *part, int D, float *dgamma, cudaStream_t s) {
    lce_dgamma_reduce_kernel<<<(D + 255) / 256, 256, 0, s>>>(part, D, dgamma);
    return cudaGetLastError();
}

}  // namespace lce
