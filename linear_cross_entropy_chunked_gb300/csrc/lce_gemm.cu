// tcgen05 / TMEM / TMA GEMM kernels of the fused linear + cross-entropy path
// (sm_103a).
//
// One warp-specialised persistent kernel serves every contraction of the path:
//   * the logits Z_c = H_c W^T of a token chunk, with an epilogue that takes the
//     row max and sum of exponentials of each 128-column slab (the online
//     log-sum-exp of "Unsloth Kernel Architecture ...", section 1 "Fused
//     Cross-Entropy Loss with Logit Streaming", done per tile), picks the target
//     logit, and optionally stores exp(z - slab max) or the final gradient G;
//   * the two gradient contractions dH_c = G_c W and dW += G_c^T H_c of the
//     backward ("Arquitectura interna de Unsloth y optimizacion en Triton",
//     section 3 "Fused Cross Entropy": backpropagation into X and W_vocab),
//     issued as one tile list so that the few long dH tiles and the many short
//     dW tiles share the SMs.
//
// Roles (320 threads): warps 0-7 epilogue (TMEM lane quarter = warp % 4, column
// half = warp / 4), warp 8 TMA producer, warp 9 TMEM owner + MMA issuer.
// Tiles come from a global atomic counter (dynamic persistent schedule); the
// producer publishes each tile index through a small shared-memory ring.
// Every mbarrier wait is bounded: on expiry the CTA records FLAG_TIMEOUT in the
// workspace header, drains its own copies and MMAs (again with a bound), frees
// TMEM and returns.
#include "lce_internal.h"

namespace lce {

// ---------------------------------------------------------------- PTX helpers

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Shared abort word of the CTA: set by whichever thread's wait ran out first.
struct Abort {
    volatile int *flag_smem;
    int *hdr;
    uint64_t limit_ns;
};

// Bounded wait for the phase with the given parity. Returns false (and makes
// every later wait of the CTA return false at once) when the limit runs out.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, const Abort &ab) {
    const uint32_t a = smem_u32(bar);
    if (mbar_try_wait(a, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(a, parity)) return true;
        if (*ab.flag_smem) return false;
        if (global_timer_ns() - t0 > ab.limit_ns) {
            *ab.flag_smem = 1;
            atomicOr(ab.hdr + HDR_FLAG, FLAG_TIMEOUT);
            return false;
        }
    }
}

// Drain wait used on the abort path only: fixed bound, no flag update.
__device__ __forceinline__ void mbar_wait_drain(uint64_t *bar, uint32_t parity, uint64_t limit_ns) {
    const uint32_t a = smem_u32(bar);
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(a, parity)) {
        if (global_timer_ns() - t0 > limit_ns) return;
    }
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
        : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor (tcgen05 format, version 1) for a
// 128-byte-swizzled operand. Byte offsets are encoded >> 4.
//   K-major:  rows of 64 bf16 (128 B), 8-row atoms of 1 KB: SBO = 1024.
//   MN-major: 64 MN-contiguous bf16 per K row, 8 K rows per 1 KB atom; LBO =
//             stride between 64-wide MN blocks, SBO = stride between 8-row K groups.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;  // descriptor version for tcgen05
    d |= static_cast<uint64_t>(2) << 61;  // 128-byte swizzle
    return d;
}

// Instruction descriptor of tcgen05.mma kind::f16: bf16 x bf16 -> fp32.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn_major, bool b_mn_major) {
    return (1u << 4)                                   // D format: f32
           | (1u << 7)                                 // A format: bf16
           | (1u << 10)                                // B format: bf16
           | ((a_mn_major ? 1u : 0u) << 15)            // A major-ness
           | ((b_mn_major ? 1u : 0u) << 16)            // B major-ness
           | (static_cast<uint32_t>(N >> 3) << 17)     // N / 8
           | (static_cast<uint32_t>(M >> 4) << 24);    // M / 16
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void umma_commit(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// 32 lanes x 32 consecutive fp32 columns: thread t gets row (lane base + t).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
}

// 2^x on the SFU (PTX ex2.approx, relative error ~2^-22).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

constexpr float LOG2E = 1.4426950408889634f;

// ---------------------------------------------------------------- tiles

struct Tile {
    int type;   // 0: logits or dH, 1: dW
    int m0, n0; // element offsets of the output tile
    int nk;     // k blocks
};

__device__ __forceinline__ Tile decode_tile(const GemmParams &p, int t) {
    Tile tl;
    const int n0t = p.m_blocks0 * p.n_blocks0;
    if (t < n0t) {
        // m fastest: the chunk's row blocks that share one W slab run together
        tl.type = 0;
        tl.m0 = (t % p.m_blocks0) * BM;
        tl.n0 = (t / p.m_blocks0) * BN;
        tl.nk = p.k_blocks0;
    } else {
        // dW: n (= D) fastest, so the tiles that share one G column slab run together
        t -= n0t;
        tl.type = 1;
        tl.n0 = (t % p.n_blocks1) * BN;
        tl.m0 = (t / p.n_blocks1) * BM;
        tl.nk = p.k_blocks1;
    }
    return tl;
}

// ---------------------------------------------------------------- epilogues
// Each epilogue thread owns one accumulator row (TMEM lane) and 128 columns; a
// warp owns a 32-row x 128-column slab. Outputs leave through a per-warp 4 KB
// staging buffer in shared memory, laid out as a 32 x 128-byte TMA box with the
// 128-byte swizzle (16-byte chunk j of row r at position j ^ (r % 8), so the
// warp's 16-byte shared stores are conflict-free), and one TMA bulk-tensor
// store (or reduce-add) per box. The tensor maps clip rows and columns outside
// the output, so the stores need no masks.

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until the previous bulk store of this thread no longer reads its source.
__device__ __forceinline__ void bulk_wait_read0() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, const void *src, int x, int y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(smem_u32(src)), "r"(x), "r"(y)
                 : "memory");
}
__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap *map, const void *src, int x,
                                                  int y) {
    asm volatile(
        "cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(smem_u32(src)), "r"(x), "r"(y)
        : "memory");
}

// Row `lane` of the staging box receives 8 16-byte chunks (128 bytes).
__device__ __forceinline__ void stage_row(uint8_t *stg, int lane, int j, uint32_t a, uint32_t b,
                                          uint32_t c, uint32_t d) {
    uint4 *dst = reinterpret_cast<uint4 *>(stg + lane * 128 + ((j ^ (lane & 7)) << 4));
    *dst = make_uint4(a, b, c, d);
}

// Hand the staged box to the TMA unit (lane 0 issues), after every lane's
// shared-memory writes are made visible to the async proxy.
__device__ __forceinline__ void flush_box(const CUtensorMap *map, uint8_t *stg, int lane, int x,
                                          int y, bool reduce) {
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        if (reduce) tma_reduce_add_2d(map, stg, x, y);
        else tma_store_2d(map, stg, x, y);
        bulk_commit();
    }
}

// Before writing the staging buffer again: the previous box has been read.
__device__ __forceinline__ void staging_acquire(int lane) {
    if (lane == 0) bulk_wait_read0();
    __syncwarp();
}

template <int MODE>
__device__ __forceinline__ void epilogue_logits(const GemmParams &p, const Tile &tl,
                                                uint32_t taddr, int quarter, int lane, int half,
                                                uint8_t *stg) {
    const int r = tl.m0 + quarter * 32 + lane;  // row within the chunk
    const bool row_ok = r < p.rows;
    const int col0 = tl.n0 + half * 128;        // first vocabulary column of this thread
    const int ncols = min(128, p.V - col0);     // valid columns (may be <= 0)
    long long yv = p.ignore_index;
    if (row_ok) yv = p.y[p.row0 + r];
    const bool y_ok = row_ok && yv != p.ignore_index && yv >= 0 && yv < p.V;
    const int yl = y_ok ? static_cast<int>(yv - col0) : -1;   // local target column
    const int box_y = tl.m0 + quarter * 32;

    if constexpr (MODE == MODE_G) {
        float scale = 0.f, lse2 = 0.f;
        if (row_ok) {
            const int nv = p.hdr[HDR_NVALID];
            const float dl = p.dloss ? *p.dloss : 1.f;
            scale = (y_ok && nv > 0) ? dl / static_cast<float>(nv) : 0.f;
            lse2 = p.lse[p.row0 + r] * LOG2E;
        }
        if (ncols <= 0) return;  // whole half past V: nothing to store (warp-uniform)
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
            float v[32];
            tmem_ld32(taddr + c * 32, v);
            uint32_t w[16];
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
                const int cj = c * 32 + j;
                float g0 = (cj < ncols) ? ex2(fmaf(v[j], LOG2E, -lse2)) * scale : 0.f;
                float g1 = (cj + 1 < ncols) ? ex2(fmaf(v[j + 1], LOG2E, -lse2)) * scale : 0.f;
                if (cj == yl) g0 -= scale;
                if (cj + 1 == yl) g1 -= scale;
                w[j / 2] = pack_bf16x2(g0, g1);
            }
            if ((c & 1) == 0) staging_acquire(lane);
            const int jb = (c & 1) * 4;
#pragma unroll
            for (int q = 0; q < 4; ++q)
                stage_row(stg, lane, jb + q, w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
            if (c & 1) flush_box(&p.tmS0, stg, lane, col0 + (c >> 1) * 64, box_y, false);
        }
    } else {
        // pass 1: slab max (and the target logit when it falls in this slab)
        float m = -INFINITY, zt = 0.f;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
            float v[32];
            tmem_ld32(taddr + c * 32, v);
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const int cj = c * 32 + j;
                if (cj < ncols) m = fmaxf(m, v[j]);
                if (cj == yl) zt = v[j];
            }
        }
        // pass 2: sum of exp(z - m); optionally store P' = exp(z - m) as bf16
        const float m2 = (ncols > 0) ? m * LOG2E : 0.f;
        float s = 0.f;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
            float v[32];
            tmem_ld32(taddr + c * 32, v);
            float e[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const int cj = c * 32 + j;
                e[j] = (cj < ncols) ? ex2(fmaf(v[j], LOG2E, -m2)) : 0.f;
                s += e[j];
            }
            if constexpr (MODE == MODE_LSE_P) {
                if (ncols > 0) {  // warp-uniform
                    if ((c & 1) == 0) staging_acquire(lane);
                    const int jb = (c & 1) * 4;
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        stage_row(stg, lane, jb + q, pack_bf16x2(e[8 * q], e[8 * q + 1]),
                                  pack_bf16x2(e[8 * q + 2], e[8 * q + 3]),
                                  pack_bf16x2(e[8 * q + 4], e[8 * q + 5]),
                                  pack_bf16x2(e[8 * q + 6], e[8 * q + 7]));
                    if (c & 1) flush_box(&p.tmS0, stg, lane, col0 + (c >> 1) * 64, box_y, false);
                }
            }
        }
        if (row_ok && ncols > 0) {
            p.parts[static_cast<size_t>(r) * p.nparts + col0 / PART_COLS] = make_float2(m, s);
            if (yl >= 0 && yl < 128) p.zy[r] = zt;
        }
    }
}

__device__ __forceinline__ void epilogue_dH(const GemmParams &p, const Tile &tl, uint32_t taddr,
                                            int quarter, int lane, int half, uint8_t *stg) {
    const int col0 = tl.n0 + half * 128;
    if (col0 >= p.D) return;  // warp-uniform: this half is past D
    const int box_y = tl.m0 + quarter * 32;
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
        float v[32];
        tmem_ld32(taddr + c * 32, v);
        if ((c & 1) == 0) staging_acquire(lane);
        const int jb = (c & 1) * 4;
#pragma unroll
        for (int q = 0; q < 4; ++q)
            stage_row(stg, lane, jb + q, pack_bf16x2(v[8 * q], v[8 * q + 1]),
                      pack_bf16x2(v[8 * q + 2], v[8 * q + 3]), pack_bf16x2(v[8 * q + 4], v[8 * q + 5]),
                      pack_bf16x2(v[8 * q + 6], v[8 * q + 7]));
        if (c & 1) flush_box(&p.tmS0, stg, lane, col0 + (c >> 1) * 64, box_y, false);
    }
}

__device__ __forceinline__ void epilogue_dW(const GemmParams &p, const Tile &tl, uint32_t taddr,
                                            int quarter, int lane, int half, uint8_t *stg) {
    const int col0 = tl.n0 + half * 128;
    if (col0 >= p.D) return;  // warp-uniform
    const int box_y = tl.m0 + quarter * 32;   // vocabulary row
    const bool reduce = p.dw_accumulate != 0;
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
        float v[32];
        tmem_ld32(taddr + c * 32, v);
        staging_acquire(lane);
#pragma unroll
        for (int q = 0; q < 8; ++q)
            stage_row(stg, lane, q, __float_as_uint(v[4 * q]), __float_as_uint(v[4 * q + 1]),
                      __float_as_uint(v[4 * q + 2]), __float_as_uint(v[4 * q + 3]));
        flush_box(&p.tmS1, stg, lane, col0 + c * 32, box_y, reduce);
    }
}

// ---------------------------------------------------------------- the kernel

template <int MODE>
__global__ void __launch_bounds__(GEMM_THREADS, 1) lce_gemm_kernel(const __grid_constant__ GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[STAGES];
    __shared__ __align__(8) uint64_t empty_bar[STAGES];
    __shared__ __align__(8) uint64_t tfull_bar[2];
    __shared__ __align__(8) uint64_t tempty_bar[2];
    __shared__ __align__(8) uint64_t sfull_bar[SCHED_DEPTH];
    __shared__ __align__(8) uint64_t sempty_bar[SCHED_DEPTH];
    __shared__ __align__(8) uint64_t drain_bar;
    __shared__ int sched_tile[SCHED_DEPTH];
    __shared__ uint32_t tmem_slot;
    __shared__ volatile int abort_flag;

    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull_bar[b], 1);
            mbar_init(&tempty_bar[b], NUM_EPI_WARPS);
        }
        for (int q = 0; q < SCHED_DEPTH; ++q) {
            mbar_init(&sfull_bar[q], 1);
            mbar_init(&sempty_bar[q], 1 + NUM_EPI_WARPS);
        }
        mbar_init(&drain_bar, 1);
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == PRODUCER_WARP && lane == 0) {
        prefetch_tmap(&p.tmA0);
        prefetch_tmap(&p.tmB0);
        if (MODE != MODE_LSE) prefetch_tmap(&p.tmS0);
        if (MODE == MODE_BWD) {
            prefetch_tmap(&p.tmA1);
            prefetch_tmap(&p.tmB1);
            prefetch_tmap(&p.tmS1);
        }
    }
    if (warp == MMA_WARP) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&tmem_slot)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = tmem_slot;

    Abort ab;
    ab.flag_smem = &abort_flag;
    ab.hdr = p.hdr;
    ab.limit_ns = p.timeout_ns;

    if (warp == PRODUCER_WARP) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int sq = 0;
            uint32_t sphase = 0;
            int issued = 0;  // loads issued (for the drain on abort)
            bool ok = true;
            while (ok) {
                // publish the next tile index
                if (!mbar_wait(&sempty_bar[sq], sphase ^ 1, ab)) { ok = false; break; }
                int t = atomicAdd(p.tile_counter, 1);
                if (t >= p.total_tiles) t = -1;
                sched_tile[sq] = t;
                mbar_arrive(&sfull_bar[sq]);
                if (++sq == SCHED_DEPTH) { sq = 0; sphase ^= 1; }
                if (t < 0) break;
                const Tile tl = decode_tile(p, t);
                for (int kb = 0; kb < tl.nk; ++kb) {
                    if (!mbar_wait(&empty_bar[stage], phase ^ 1, ab)) { ok = false; break; }
                    uint8_t *sA = smem + stage * STAGE_BYTES;
                    uint8_t *sB = sA + A_BYTES;
                    uint64_t *fb = &full_bar[stage];
                    mbar_arrive_expect_tx(fb, STAGE_BYTES);
                    const int kx = kb * BK;
                    if (MODE != MODE_BWD) {
                        tma_load_2d(sA, &p.tmA0, fb, kx, p.row0 + tl.m0);
                        tma_load_2d(sB, &p.tmB0, fb, kx, tl.n0);
                    } else if (tl.type == 0) {
                        // dH: A = G rows (K-major), B = W (MN-major, 4 blocks of 64 D-columns)
                        tma_load_2d(sA, &p.tmA0, fb, kx, tl.m0);
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            tma_load_2d(sB + j * 8192, &p.tmB0, fb, tl.n0 + 64 * j, kx);
                    } else {
                        // dW: A = G^T (MN-major, 2 blocks of 64 vocab columns), B = H chunk (MN-major)
#pragma unroll
                        for (int j = 0; j < 2; ++j)
                            tma_load_2d(sA + j * 8192, &p.tmA1, fb, tl.m0 + 64 * j, kx);
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            tma_load_2d(sB + j * 8192, &p.tmB1, fb, tl.n0 + 64 * j, kx);
                    }
                    ++issued;
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
            }
            if (!ok) {
                // drain: wait (bounded) for the copies still in flight into each stage
                const int n = issued < STAGES ? issued : STAGES;
                for (int i = 0; i < n; ++i) {
                    if (--stage < 0) { stage = STAGES - 1; phase ^= 1; }
                    mbar_wait_drain(&full_bar[stage], phase, 50000000ull);
                }
            }
        }
    } else if (warp == MMA_WARP) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int sq = 0;
            uint32_t sphase = 0;
            int acc = 0;
            uint32_t aphase = 0;
            bool ok = true;
            bool any_mma = false;
            while (ok) {
                if (!mbar_wait(&sfull_bar[sq], sphase, ab)) { ok = false; break; }
                const int t = sched_tile[sq];
                mbar_arrive(&sempty_bar[sq]);
                if (++sq == SCHED_DEPTH) { sq = 0; sphase ^= 1; }
                if (t < 0) break;
                const Tile tl = decode_tile(p, t);
                if (!mbar_wait(&tempty_bar[acc], aphase ^ 1, ab)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN;
                // operand layouts of this tile type
                bool a_mn = false, b_mn = false;
                if (MODE == MODE_BWD) {
                    b_mn = true;
                    a_mn = (tl.type == 1);
                }
                const uint32_t idesc = idesc_bf16(BM, BN, a_mn, b_mn);
                const uint32_t a_lbo = a_mn ? 8192u : 16u, b_lbo = b_mn ? 8192u : 16u;
                const uint32_t a_step = a_mn ? (2048u >> 4) : (32u >> 4);
                const uint32_t b_step = b_mn ? (2048u >> 4) : (32u >> 4);
                for (int kb = 0; kb < tl.nk; ++kb) {
                    if (!mbar_wait(&full_bar[stage], phase, ab)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t sA = smem_u32(smem + stage * STAGE_BYTES);
                    const uint32_t sB = sA + A_BYTES;
                    const uint64_t ad = sdesc(sA, a_lbo, 1024u);
                    const uint64_t bd = sdesc(sB, b_lbo, 1024u);
#pragma unroll
                    for (int k = 0; k < BK / UMMA_K; ++k)
                        umma_bf16(d_tmem, ad + static_cast<uint64_t>(k * a_step),
                                  bd + static_cast<uint64_t>(k * b_step), idesc,
                                  (kb | k) != 0 ? 1u : 0u);
                    any_mma = true;
                    umma_commit(&empty_bar[stage]);
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                umma_commit(&tfull_bar[acc]);
                if (++acc == 2) { acc = 0; aphase ^= 1; }
            }
            if (!ok && any_mma) {
                // make sure no MMA is still writing TMEM before it is freed
                umma_commit(&drain_bar);
                mbar_wait_drain(&drain_bar, 0, 50000000ull);
            }
        }
    } else {
        // epilogue warps 0..7
        const int quarter = warp & 3;
        const int half = warp >> 2;
        uint8_t *stg = smem + STAGES * STAGE_BYTES + warp * STAGING_BYTES;
        int sq = 0;
        uint32_t sphase = 0;
        int acc = 0;
        uint32_t aphase = 0;
        while (true) {
            if (!mbar_wait(&sfull_bar[sq], sphase, ab)) break;
            const int t = sched_tile[sq];
            __syncwarp();
            if (lane == 0) mbar_arrive(&sempty_bar[sq]);
            if (++sq == SCHED_DEPTH) { sq = 0; sphase ^= 1; }
            if (t < 0) break;
            const Tile tl = decode_tile(p, t);
            if (!mbar_wait(&tfull_bar[acc], aphase, ab)) break;
            tc_fence_after();
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                   static_cast<uint32_t>(acc * BN + half * 128);
            if (MODE != MODE_BWD) {
                epilogue_logits<MODE>(p, tl, taddr, quarter, lane, half, stg);
            } else if (tl.type == 0) {
                epilogue_dH(p, tl, taddr, quarter, lane, half, stg);
            } else {
                epilogue_dW(p, tl, taddr, quarter, lane, half, stg);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty_bar[acc]);
            if (++acc == 2) { acc = 0; aphase ^= 1; }
        }
        // all bulk stores of this warp complete before the CTA exits
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == MMA_WARP) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                     "r"(TMEM_COLS)
                     : "memory");
    }
}

cudaError_t gemm_set_attributes() {
    cudaError_t e;
    e = cudaFuncSetAttribute(lce_gemm_kernel<MODE_LSE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             GEMM_SMEM_BYTES);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(lce_gemm_kernel<MODE_LSE_P>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, GEMM_SMEM_BYTES);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(lce_gemm_kernel<MODE_G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             GEMM_SMEM_BYTES);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(lce_gemm_kernel<MODE_BWD>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, GEMM_SMEM_BYTES);
}

cudaError_t launch_gemm(int mode, const GemmParams &p, int grid, cudaStream_t s) {
    switch (mode) {
        case MODE_LSE:
            lce_gemm_kernel<MODE_LSE><<<grid, GEMM_THREADS, GEMM_SMEM_BYTES, s>>>(p);
            break;
        case MODE_LSE_P:
            lce_gemm_kernel<MODE_LSE_P><<<grid, GEMM_THREADS, GEMM_SMEM_BYTES, s>>>(p);
            break;
        case MODE_G:
            lce_gemm_kernel<MODE_G><<<grid, GEMM_THREADS, GEMM_SMEM_BYTES, s>>>(p);
            break;
        default:
            lce_gemm_kernel<MODE_BWD><<<grid, GEMM_THREADS, GEMM_SMEM_BYTES, s>>>(p);
            break;
    }
    return cudaGetLastError();
}

}  // namespace lce
