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
//     section 3 "Fused Cross Entropy": backpropagation into X and W_vocab): on
//     CTA pairs the dH tiles (512 columns wide) in one launch and the dW tiles
//     in launches beside and behind it; with one CTA per tile, one tile list in
//     which the few long dH tiles and the many short dW tiles share the SMs.
//
// Roles (320 threads): warps 0-7 epilogue (TMEM lane quarter = warp % 4, column
// half = warp / 4), warp 8 TMA producer, warp 9 TMEM owner + MMA issuer.
// Tiles come from a global atomic counter (dynamic persistent schedule); the
// producer publishes each tile index through a small shared-memory ring.
// Every mbarrier wait is bounded: on expiry the CTA records FLAG_TIMEOUT in the
// workspace header, drains its own copies and MMAs (again with a bound), frees
// TMEM and returns.
#include "lce_internal.h"
#include "lce_ptx.cuh"

namespace lce {

// ---------------------------------------------------------------- PTX helpers
// (generic mbarrier / cluster helpers live in lce_ptx.cuh)

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
        : "memory");
}

// 3-D box (x, y, z): the dW tiles' A operand, two 64-column blocks of G^T per load.
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int x, int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
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

// Instruction descriptor of tcgen05.mma kind::f16: bf16 x bf16 or fp16 x fp16
// (both operands always the same type) -> fp32.
__host__ __device__ constexpr uint32_t idesc_f16kind(int M, int N, bool a_mn_major, bool b_mn_major,
                                                     bool fp16) {
    return (1u << 4)                                   // D format: f32
           | ((fp16 ? 0u : 1u) << 7)                   // A format: f16 (0) / bf16 (1)
           | ((fp16 ? 0u : 1u) << 10)                  // B format: f16 (0) / bf16 (1)
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
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}
// Two 16-bit values in the operand dtype of the call.
__device__ __forceinline__ uint32_t pack_h16x2(float lo, float hi, int f16) {
    return f16 ? pack_f16x2(lo, hi) : pack_bf16x2(lo, hi);
}

constexpr float LOG2E = 1.4426950408889634f;

// ---------------------------------------------------------------- tiles

struct Tile {
    int type;   // TILE_MAIN: logits tile or dH tile; TILE_DW: dW tile
    int m0, n0; // element offsets of the output tile
    int kb0;    // first k block
    int nk;     // k blocks
    int srow;   // row offset of the tile's store (split dH partial sums; else 0)
};
enum : int { TILE_MAIN = 0, TILE_DW = 1 };

// Tiles are scheduled in units of CL vertically adjacent 128-row tiles (CL = 1,
// or 2 for a CTA pair that shares the B operand); `t` indexes those units and
// `crank` picks the CTA's own 128 rows. Logits launches: m fastest, so the
// chunk's row blocks that share one W slab run together. Gradient launches:
// the few long dH tiles first (m fastest, then n, then the vocabulary part
// of a split dH launch), then the many short dW tiles (n fastest, so the tiles
// that share one G^T slab run together); the dynamic schedule lets the SMs
// left over by the dH tiles start on dW at once.
template <int CL>
__device__ __forceinline__ Tile decode_tile(const GemmParams &p, int t, int crank, bool wide) {
    Tile tl;
    const int mp0 = (p.m_blocks0 + CL - 1) / CL;
    const int nH1 = mp0 * p.n_blocks0;
    const int splits = p.k_splits > 1 ? p.k_splits : 1;
    if (t < nH1 * splits) {
        const int sp = t / nH1;
        t -= sp * nH1;
        tl.type = TILE_MAIN;
        tl.m0 = ((t % mp0) * CL + crank) * BM;
        tl.n0 = (t / mp0) * (wide ? BN_WIDE : BN);
        if (splits > 1) {
            tl.kb0 = sp * p.kb_per_split;
            tl.nk = min(p.kb_per_split, p.k_blocks0 - tl.kb0);
            tl.srow = sp * p.split_rows;
        } else {
            tl.kb0 = 0;
            tl.nk = p.k_blocks0;
            tl.srow = 0;
        }
    } else {
        t -= nH1 * splits;
        tl.type = TILE_DW;
        tl.n0 = (t % p.n_blocks1) * BN;
        tl.m0 = ((t / p.n_blocks1) * CL + crank) * BM;
        tl.kb0 = 0;
        tl.nk = p.k_blocks1;
        tl.srow = 0;
    }
    return tl;
}

// ---------------------------------------------------------------- epilogues
// Each epilogue thread owns one accumulator row (TMEM lane) and 128 columns;
// the 4 warps of a column half own a 128-row x 128-column slab. Outputs leave
// through one 16 KB staging box per half in shared memory: 128 rows x 128 bytes
// with the 128-byte swizzle (16-byte chunk j of row r at position j ^ (r % 8),
// which makes the warps' 16-byte shared stores conflict-free). When the box is
// full, one thread of the half issues a single TMA bulk-tensor store (or
// reduce-add) for it. The tensor maps clip rows and columns outside the
// output, so the stores need no masks. The 4 warps of a half meet at a named
// barrier (id 1 + half, 128 threads) before writing the box (it has been read)
// and before issuing it (all rows are in).

__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read0() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ void named_bar_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
// Barrier over `n` threads that also returns the AND of every thread's `ok`.
__device__ __forceinline__ bool named_bar_and(int id, int n, bool ok) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred q, a;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.and.pred a, %2, %3, q;\n\t"
        "selp.u32 %0, 1, 0, a;\n\t}\n"
        : "=r"(r)
        : "r"(ok ? 1u : 0u), "r"(id), "r"(n)
        : "memory");
    return r != 0;
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

enum StoreKind : int { ST_STORE = 0, ST_REDUCE = 1 };

struct HalfStager {
    uint8_t *buf;   // 16 KB, 1 KB aligned
    int bar_id;     // 1 + half
    int row;        // 0..127 = quarter * 32 + lane
    bool leader;    // quarter 0, lane 0: issues the stores

    // The box may be written: its previous store has read it.
    __device__ __forceinline__ void acquire() const {
        if (leader) bulk_wait_read0();
        named_bar_sync(bar_id, 128);
    }
    __device__ __forceinline__ void put(int j, uint32_t a, uint32_t b, uint32_t c,
                                        uint32_t d) const {
        *reinterpret_cast<uint4 *>(buf + row * 128 + ((j ^ (row & 7)) << 4)) = make_uint4(a, b, c, d);
    }
    // 32 fp32 values fill the whole 128-byte row.
    __device__ __forceinline__ void put_f32(const float *v) const {
#pragma unroll
        for (int j = 0; j < 8; ++j)
            put(j, __float_as_uint(v[4 * j]), __float_as_uint(v[4 * j + 1]),
                __float_as_uint(v[4 * j + 2]), __float_as_uint(v[4 * j + 3]));
    }
    // 32 values as 16-bit floats (bf16, or fp16 when f16) fill half of the row:
    // chunks jb .. jb + 3.
    __device__ __forceinline__ void put_h16(int jb, const float *v, int f16) const {
#pragma unroll
        for (int q = 0; q < 4; ++q)
            put(jb + q, pack_h16x2(v[8 * q], v[8 * q + 1], f16),
                pack_h16x2(v[8 * q + 2], v[8 * q + 3], f16), pack_h16x2(v[8 * q + 4], v[8 * q + 5], f16),
                pack_h16x2(v[8 * q + 6], v[8 * q + 7], f16));
    }
    __device__ __forceinline__ void issue(const CUtensorMap *map, int kind, int x, int y) const {
        fence_proxy_async_smem();
        named_bar_sync(bar_id, 128);
        if (leader) {
            if (kind == ST_REDUCE) tma_reduce_add_2d(map, buf, x, y);
            else tma_store_2d(map, buf, x, y);
            bulk_commit();
        }
    }
};

// Logits epilogues stage per warp instead: a 4 KB box of 32 rows x 128 bytes
// per warp (same swizzle), issued by the warp's lane 0 with no cross-warp
// barrier. The logits epilogue does more arithmetic between stores, and the
// per-warp boxes keep the warps independent.
struct WarpStager {
    uint8_t *buf;   // 4 KB, 1 KB aligned
    int lane;
    __device__ __forceinline__ void acquire() const {
        if (lane == 0) bulk_wait_read0();
        __syncwarp();
    }
    __device__ __forceinline__ void put_h16(int jb, const float *v, int f16) const {
#pragma unroll
        for (int q = 0; q < 4; ++q)
            *reinterpret_cast<uint4 *>(buf + lane * 128 + (((jb + q) ^ (lane & 7)) << 4)) =
                make_uint4(pack_h16x2(v[8 * q], v[8 * q + 1], f16),
                           pack_h16x2(v[8 * q + 2], v[8 * q + 3], f16),
                           pack_h16x2(v[8 * q + 4], v[8 * q + 5], f16),
                           pack_h16x2(v[8 * q + 6], v[8 * q + 7], f16));
    }
    __device__ __forceinline__ void issue(const CUtensorMap *map, int x, int y) const {
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            tma_store_2d(map, buf, x, y);
            bulk_commit();
        }
    }
};

template <int MODE>
__device__ __forceinline__ void epilogue_logits(const GemmParams &p, const Tile &tl,
                                                uint32_t taddr, int quarter, int half,
                                                const WarpStager &st) {
    const int r = tl.m0 + quarter * 32 + st.lane;  // row within the chunk
    const int box_y = tl.m0 + quarter * 32;
    const bool box_rows = box_y < p.rows;       // warp-uniform: any row of the box exists
    const bool row_ok = r < p.rows;
    const int col0 = tl.n0 + half * 128;        // first vocabulary column of this half
    const int ncols = min(128, p.V - col0);     // valid columns (may be <= 0); same for the half
    long long yv = p.ignore_index;
    if (row_ok) yv = p.y[p.row0 + r];
    const bool y_ok = row_ok && yv != p.ignore_index && yv >= 0 && yv < p.V;
    const int yl = y_ok ? static_cast<int>(yv - col0) : -1;   // local target column

    if constexpr (MODE == MODE_G) {
        if (ncols <= 0 || !box_rows) return;
        float scale = 0.f, lse2 = 0.f;
        if (row_ok) {
            scale = lce_store_scale(p.dloss, p.dloss_per_row, p.mean, p.hdr[HDR_NVALID],
                                    p.row0 + r, y_ok, p.f16);
            lse2 = p.lse[p.row0 + r] * LOG2E;
        }
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
            const bool box_ok = (c >> 1) * 64 < ncols;
            float v[32];
            tmem_ld32(taddr + c * 32, v);
            if (!box_ok) continue;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const int cj = c * 32 + j;
                float g = (cj < ncols) ? ex2(fmaf(v[j], LOG2E, -lse2)) * scale : 0.f;
                if (cj == yl) g -= scale;
                v[j] = g;
            }
            if ((c & 1) == 0) st.acquire();
            st.put_h16((c & 1) * 4, v, p.f16);
            if (c & 1) st.issue(&p.tmS0, col0 + (c >> 1) * 64, box_y);
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
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const int cj = c * 32 + j;
                v[j] = (cj < ncols) ? ex2(fmaf(v[j], LOG2E, -m2)) : 0.f;
                s += v[j];
            }
            if constexpr (MODE == MODE_LSE_P) {
                if ((c >> 1) * 64 < ncols && box_rows) {
                    if ((c & 1) == 0) st.acquire();
                    st.put_h16((c & 1) * 4, v, p.f16);
                    if (c & 1) st.issue(&p.tmS0, col0 + (c >> 1) * 64, box_y);
                }
            }
        }
        if (row_ok && ncols > 0) {
            p.parts[static_cast<size_t>(r) * p.nparts + col0 / PART_COLS] = make_float2(m, s);
            if (yl >= 0 && yl < 128) p.zy[r] = zt;
        }
    }
}

// Gradient tiles: dH (bf16 / fp16, or fp32 when dh_fp32) or dW (fp32, stored by
// a call's first dW contraction, reduce-added into dW by the later ones). out_scale: the factor
// fp16 calls apply here instead of in G (1 for bf16).
__device__ __forceinline__ void epilogue_grad(const GemmParams &p, const Tile &tl, uint32_t taddr,
                                              int half, const HalfStager &st, float out_scale) {
    const int col0 = tl.n0 + half * 128;
    if (col0 >= p.D) return;  // this half is past D (same for the 4 warps)
    // a tile entirely past the output rows (the second tile of a CTA pair at an
    // odd row-block count) stores nothing
    if (tl.m0 >= (tl.type == TILE_MAIN ? p.rows : p.V)) return;
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
        float v[32];
        tmem_ld32(taddr + c * 32, v);
        if (p.f16) {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] *= out_scale;
        }
        if (tl.type == TILE_MAIN && !p.dh_fp32) {
            if (col0 + (c >> 1) * 64 >= p.D) continue;
            if ((c & 1) == 0) st.acquire();
            st.put_h16((c & 1) * 4, v, p.f16);
            if (c & 1) st.issue(&p.tmS0, ST_STORE, col0 + (c >> 1) * 64, tl.m0);
        } else if (tl.type == TILE_MAIN) {
            if (col0 + c * 32 >= p.D) continue;
            st.acquire();
            st.put_f32(v);
            st.issue(&p.tmS0, ST_STORE, col0 + c * 32, tl.m0 + tl.srow);
        } else {
            if (col0 + c * 32 >= p.D) continue;
            st.acquire();
            st.put_f32(v);
            st.issue(&p.tmS1, p.dw_accumulate ? ST_REDUCE : ST_STORE, col0 + c * 32, tl.m0);
        }
    }
}

// ---------------------------------------------------------------- pair (cta_group::2) helpers

// Pair (cta_group::2) forms. The TMA load writes this CTA's smem and signals the
// mbarrier at the shared::cluster address `bar` (the leader CTA's).
__device__ __forceinline__ void tma_load_2d_pair(void *dst, const CUtensorMap *map, uint32_t bar,
                                                 int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
        : "memory");
}
__device__ __forceinline__ void tma_load_3d_pair(void *dst, const CUtensorMap *map, uint32_t bar,
                                                 int x, int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z)
        : "memory");
}
__device__ __forceinline__ void umma_bf16_pair(uint32_t d_tmem, uint64_t a, uint64_t b,
                                               uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}
// Completion of this CTA's pair MMAs arrives on `bar`'s offset in every CTA of `mask`.
__device__ __forceinline__ void umma_commit_pair(uint64_t *bar, uint16_t mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(smem_u32(bar)),
        "h"(mask)
        : "memory");
}

// ---------------------------------------------------------------- the kernel
// CL = 1: one CTA per 128 x 256 output tile. CL = 2: a CTA pair (cluster of 2)
// per 256 x 256 tile with tcgen05 cta_group::2 MMAs: each CTA loads its own 128
// rows of A and one half (128 columns of N) of B, both TMA loads completing on
// the leader CTA's stage barrier; the leader's single MMA thread issues M = 256
// MMAs that read both CTAs' shared memory and write both CTAs' TMEM (each its
// own 128 rows); its commits arrive on the stage and accumulator barriers of
// both CTAs; both CTAs' epilogues release the leader's accumulator. Per SM this
// halves the B bytes per MMA, so each SM streams 32 KB instead of 48 KB per
// 64-deep k block. The leader also fetches the tiles and writes them into both
// CTAs' schedule rings.

template <int MODE, int CL>
__global__ void __launch_bounds__(GEMM_THREADS, 1) lce_gemm_kernel(const __grid_constant__ GemmParams p) {
    using P = Pipe<CL, MODE == MODE_DH>;
    static_assert(MODE != MODE_DH || CL == 2, "wide dH tiles run on CTA pairs only");
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[MAX_STAGES];
    __shared__ __align__(8) uint64_t empty_bar[MAX_STAGES];
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
    const uint32_t crank = (CL == 2) ? cluster_ctarank() : 0u;
    const bool leader = crank == 0;
    // consumers of one schedule slot: the leader's MMA thread, every epilogue
    // warp of the pair, and the peer's producer
    constexpr int kSchedConsumers = 1 + CL * NUM_EPI_WARPS + (CL - 1);

    if (threadIdx.x == 0) {
        for (int s = 0; s < P::kStages; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull_bar[b], 1);
            mbar_init(&tempty_bar[b], CL * NUM_EPI_WARPS);
        }
        for (int q = 0; q < SCHED_DEPTH; ++q) {
            mbar_init(&sfull_bar[q], 1);
            mbar_init(&sempty_bar[q], kSchedConsumers);
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
        // with CL = 2 both CTAs allocate together: the same columns on both SMs
        if constexpr (CL == 2) {
            asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                             smem_u32(&tmem_slot)),
                         "r"(TMEM_COLS)
                         : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
        } else {
            asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                             smem_u32(&tmem_slot)),
                         "r"(TMEM_COLS)
                         : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
        }
    }
    tc_fence_before();
    __syncthreads();
    if constexpr (CL == 2) cluster_sync_all();   // the peer's barriers exist from here on
    tc_fence_after();
    const uint32_t tmem_base = tmem_slot;

    Abort ab;
    ab.flag_smem = &abort_flag;
    ab.hdr = p.hdr;
    ab.limit_ns = p.timeout_ns;

    // a consumer of schedule slot q (or of accumulator buffer b) releases it on
    // the leader's barrier
    auto release_on_leader = [&](uint64_t *bar) {
        if (CL == 2 && !leader) mbar_arrive_cluster(map_to_rank(bar, 0));
        else mbar_arrive(bar);
    };

    if (warp == PRODUCER_WARP) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int sq = 0;
            uint32_t sphase = 0;
            int issued = 0;  // loads issued (for the drain on abort)
            bool ok = true;
            // The leader fetches tiles from the global counter and publishes them to
            // both CTAs' schedule rings one tile ahead of its own streaming: while it
            // streams tile i, tile i+1 is already in the rings (so the peer's
            // producer and the MMA warp never wait for it at the tile boundary) and
            // the counter fetch for tile i+2 is in flight (its latency is hidden
            // behind tile i's loads).
            auto publish = [&](int v) -> bool {
                if (!mbar_wait_cluster(&sempty_bar[sq], sphase ^ 1, ab)) return false;
                sched_tile[sq] = v;
                if constexpr (CL == 2) {
                    st_cluster_u32(map_to_rank(&sched_tile[sq], 1), v);
                    mbar_arrive_cluster(map_to_rank(&sfull_bar[sq], 1));
                }
                mbar_arrive(&sfull_bar[sq]);
                if (++sq == SCHED_DEPTH) { sq = 0; sphase ^= 1; }
                return true;
            };
            int t_lead = -1;      // leader: the tile it streams next
            int pending_raw = 0;  // leader: counter value fetched for the tile after that
            if (leader) {
                const int f = atomicAdd(p.tile_counter, 1);
                t_lead = f < p.total_tiles ? f : -1;
                ok = publish(t_lead);
                if (ok && t_lead >= 0) pending_raw = atomicAdd(p.tile_counter, 1);
            }
            while (ok) {
                int t;
                if (leader) {
                    if (t_lead < 0) break;
                    // publish the next tile (fetched one tile ago), fetch the one after;
                    // the fetched value is first needed a tile from now
                    const int nxt = pending_raw < p.total_tiles ? pending_raw : -1;
                    if (!publish(nxt)) { ok = false; break; }
                    if (nxt >= 0) pending_raw = atomicAdd(p.tile_counter, 1);
                    t = t_lead;
                    t_lead = nxt;
                } else {
                    if (!mbar_wait_cluster(&sfull_bar[sq], sphase, ab)) { ok = false; break; }
                    t = sched_tile[sq];
                    release_on_leader(&sempty_bar[sq]);
                    if (++sq == SCHED_DEPTH) { sq = 0; sphase ^= 1; }
                    if (t < 0) break;
                }
                const Tile tl = decode_tile<CL>(p, t, static_cast<int>(crank), MODE == MODE_DH);
                for (int kb = 0; kb < tl.nk; ++kb) {
                    if (!mbar_wait(&empty_bar[stage], phase ^ 1, ab)) { ok = false; break; }
                    uint8_t *sA = smem + stage * P::kStageBytes;
                    uint8_t *sB = sA + A_BYTES;
                    uint64_t *fb = &full_bar[stage];
                    const int kx = (tl.kb0 + kb) * BK;
                    const CUtensorMap *ma = (MODE == MODE_BWD && tl.type == TILE_DW) ? &p.tmA1 : &p.tmA0;
                    const int ya = (MODE == MODE_BWD) ? tl.m0 : p.a_row0 + tl.m0;
                    const bool b_mn = (MODE == MODE_BWD) && tl.type != TILE_DW;
                    const CUtensorMap *mb = (MODE == MODE_BWD && !b_mn) ? &p.tmB1 : &p.tmB0;
                    // dW tiles read A = G^T straight from the row-major chunk buffer
                    // (MN-major: two 64-wide vocabulary boxes per 64 chunk rows)
                    const bool a_mn = (MODE == MODE_BWD) && tl.type == TILE_DW;
                    if constexpr (CL == 1) {
                        mbar_arrive_expect_tx(fb, P::kStageBytes);
                        if (a_mn) {
                            // two 64-column blocks of G^T (z = tl.m0 / 64 and the next)
                            tma_load_3d(sA, ma, fb, 0, kx, tl.m0 >> 6);
                        } else {
                            tma_load_2d(sA, ma, fb, kx, ya);
                        }
                        if (b_mn) {
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                tma_load_2d(sB + j * 8192, mb, fb, tl.n0 + 64 * j, kx);
                        } else {
                            tma_load_2d(sB, mb, fb, kx, tl.n0);
                        }
                    } else if constexpr (MODE == MODE_DH) {
                        // A = G rows (K-major); B = W, MN-major, two 256-column halves
                        // of which this CTA loads 128 columns each
                        if (leader) mbar_arrive_expect_tx(fb, 2 * P::kStageBytes);
                        const uint32_t lfb = map_to_rank(fb, 0);
                        tma_load_2d_pair(sA, &p.tmA0, lfb, kx, tl.m0);
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const int nb = tl.n0 + h * BN + static_cast<int>(crank) * (BN / 2);
                            tma_load_2d_pair(sB + h * 16384, &p.tmB0, lfb, nb, kx);
                            tma_load_2d_pair(sB + h * 16384 + 8192, &p.tmB0, lfb, nb + 64, kx);
                        }
                        (void)ma; (void)mb; (void)ya; (void)a_mn; (void)b_mn;
                    } else {
                        // both CTAs' bytes complete on the leader's barrier
                        if (leader) mbar_arrive_expect_tx(fb, 2 * P::kStageBytes);
                        const uint32_t lfb = map_to_rank(fb, 0);
                        const int nb = tl.n0 + static_cast<int>(crank) * (BN / 2);
                        if (a_mn) {
                            // two 64-column blocks of G^T (z = tl.m0 / 64 and the next)
                            tma_load_3d_pair(sA, ma, lfb, 0, kx, tl.m0 >> 6);
                        } else {
                            tma_load_2d_pair(sA, ma, lfb, kx, ya);
                        }
                        if (b_mn) {
                            tma_load_2d_pair(sB, mb, lfb, nb, kx);
                            tma_load_2d_pair(sB + 8192, mb, lfb, nb + 64, kx);
                        } else {
                            tma_load_2d_pair(sB, mb, lfb, kx, nb);
                        }
                    }
                    ++issued;
                    if (++stage == P::kStages) { stage = 0; phase ^= 1; }
                }
            }
            if (!ok) {
                // drain: wait (bounded) for the copies still in flight into each stage
                // (with CL = 2 only the leader's barriers count the bytes)
                const int n = issued < P::kStages ? issued : P::kStages;
                for (int i = 0; i < n; ++i) {
                    if (--stage < 0) { stage = P::kStages - 1; phase ^= 1; }
                    if (leader) mbar_wait_drain(&full_bar[stage], phase, 50000000ull);
                }
                if (!leader) {
                    const uint64_t t0 = global_timer_ns();
                    while (global_timer_ns() - t0 < 50000000ull) {}
                }
            }
        }
    } else if (warp == MMA_WARP) {
        if (lane == 0 && leader) {
            int stage = 0;
            uint32_t phase = 0;
            int sq = 0;
            uint32_t sphase = 0;
            int acc = 0;
            uint32_t aphase = 0;
            bool ok = true;
            bool any_mma = false;
            const uint16_t both = static_cast<uint16_t>((1u << CL) - 1u);
            while (ok) {
                if (!mbar_wait_cluster(&sfull_bar[sq], sphase, ab)) { ok = false; break; }
                const int t = sched_tile[sq];
                release_on_leader(&sempty_bar[sq]);
                if (++sq == SCHED_DEPTH) { sq = 0; sphase ^= 1; }
                if (t < 0) break;
                const Tile tl = decode_tile<CL>(p, t, 0, MODE == MODE_DH);
                if (!mbar_wait_cluster(&tempty_bar[acc], aphase ^ 1, ab)) { ok = false; break; }
                // a wide dH tile accumulates into both buffers (acc is 0 at its start)
                if (MODE == MODE_DH && !mbar_wait_cluster(&tempty_bar[1], aphase ^ 1, ab)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN;
                // MN-major operands: W for the dH tiles (B), the chunk buffer for the
                // dW tiles (A = G^T); everything else is K-major
                const bool b_mn = (MODE == MODE_BWD || MODE == MODE_DH) && tl.type != TILE_DW;
                const bool a_mn = (MODE == MODE_BWD) && tl.type == TILE_DW;
                const uint32_t idesc = idesc_f16kind(CL * BM, BN, a_mn, b_mn, p.f16 != 0);
                const uint32_t a_lbo = a_mn ? 8192u : 16u;
                const uint32_t b_lbo = b_mn ? 8192u : 16u;
                const uint32_t a_step = a_mn ? (2048u >> 4) : (32u >> 4);
                const uint32_t b_step = b_mn ? (2048u >> 4) : (32u >> 4);
                for (int kb = 0; kb < tl.nk; ++kb) {
                    if (!mbar_wait(&full_bar[stage], phase, ab)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t sA = smem_u32(smem + stage * P::kStageBytes);
                    const uint32_t sB = sA + A_BYTES;
                    const uint64_t ad = sdesc(sA, a_lbo, 1024u);
                    const uint64_t bd = sdesc(sB, b_lbo, 1024u);
#pragma unroll
                    for (int k = 0; k < BK / UMMA_K; ++k) {
                        const uint64_t a = ad + static_cast<uint64_t>(k * a_step);
                        const uint64_t b = bd + static_cast<uint64_t>(k * b_step);
                        const uint32_t accumulate = (kb | k) != 0 ? 1u : 0u;
                        if constexpr (CL == 2) umma_bf16_pair(d_tmem, a, b, idesc, accumulate);
                        else umma_bf16(d_tmem, a, b, idesc, accumulate);
                        // the second 256-column half: same A, B 16 KB further on
                        if constexpr (MODE == MODE_DH)
                            umma_bf16_pair(d_tmem + BN, a, b + static_cast<uint64_t>(16384u >> 4), idesc,
                                           accumulate);
                    }
                    any_mma = true;
                    if constexpr (CL == 2) umma_commit_pair(&empty_bar[stage], both);
                    else umma_commit(&empty_bar[stage]);
                    if (++stage == P::kStages) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                if constexpr (MODE == MODE_DH) {
                    umma_commit_pair(&tfull_bar[0], both);
                    umma_commit_pair(&tfull_bar[1], both);
                    aphase ^= 1;
                } else {
                    if constexpr (CL == 2) umma_commit_pair(&tfull_bar[acc], both);
                    else umma_commit(&tfull_bar[acc]);
                    if (++acc == 2) { acc = 0; aphase ^= 1; }
                }
            }
            if (any_mma) {
                // every MMA (and every arrival it sends to the peer) has completed
                // before TMEM is freed and the CTAs leave
                if constexpr (CL == 2) umma_commit_pair(&drain_bar, both);
                else umma_commit(&drain_bar);
                mbar_wait_drain(&drain_bar, 0, 50000000ull);
            }
        }
    } else {
        // epilogue warps 0..7; the 4 warps of a half take every decision together
        // (barrier votes), so an abort never leaves one of them at a named barrier.
        const int quarter = warp & 3;
        const int half = warp >> 2;
        HalfStager st;
        st.buf = smem + PIPE_BYTES + half * STAGING_BYTES;
        st.bar_id = 1 + half;
        st.row = quarter * 32 + lane;
        st.leader = (quarter == 0 && lane == 0);
        WarpStager wst;
        wst.buf = smem + PIPE_BYTES + warp * (2 * STAGING_BYTES / NUM_EPI_WARPS);
        wst.lane = lane;
        const float out_scale = (MODE == MODE_BWD || MODE == MODE_DH)
                                    ? lce_out_scale(p.dloss, p.mean, p.hdr[HDR_NVALID], p.f16)
                                    : 1.f;
        int sq = 0;
        uint32_t sphase = 0;
        int acc = 0;
        uint32_t aphase = 0;
        while (true) {
            bool ok = mbar_wait_cluster(&sfull_bar[sq], sphase, ab);
            if (!named_bar_and(st.bar_id, 128, ok)) break;
            const int t = sched_tile[sq];
            __syncwarp();
            if (lane == 0) release_on_leader(&sempty_bar[sq]);
            if (++sq == SCHED_DEPTH) { sq = 0; sphase ^= 1; }
            if (t < 0) break;
            const Tile tl = decode_tile<CL>(p, t, static_cast<int>(crank), MODE == MODE_DH);
            ok = mbar_wait_cluster(&tfull_bar[acc], aphase, ab);
            if (!named_bar_and(st.bar_id, 128, ok)) break;
            tc_fence_after();
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                   static_cast<uint32_t>(acc * BN + half * 128);
            if constexpr (MODE == MODE_DH) {
                // both accumulators of the wide tile: columns n0 .. n0 + 255, then + 256
                epilogue_grad(p, tl, taddr, half, st, out_scale);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) release_on_leader(&tempty_bar[0]);
                ok = mbar_wait_cluster(&tfull_bar[1], aphase, ab);
                if (!named_bar_and(st.bar_id, 128, ok)) break;
                tc_fence_after();
                Tile tl2 = tl;
                tl2.n0 += BN;
                epilogue_grad(p, tl2, taddr + BN, half, st, out_scale);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) release_on_leader(&tempty_bar[1]);
                aphase ^= 1;
                continue;
            }
            if constexpr (MODE != MODE_BWD && MODE != MODE_DH) {
                epilogue_logits<MODE>(p, tl, taddr, quarter, half, wst);
            } else {
                epilogue_grad(p, tl, taddr, half, st, out_scale);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) release_on_leader(&tempty_bar[acc]);
            if (++acc == 2) { acc = 0; aphase ^= 1; }
        }
        // all bulk stores issued by this warp / half complete before the CTA exits
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    // no CTA of the pair leaves while the other may still write to it
    if constexpr (CL == 2) cluster_sync_all();
    if (warp == MMA_WARP) {
        tc_fence_after();
        if constexpr (CL == 2)
            asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                         "r"(TMEM_COLS)
                         : "memory");
        else
            asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                         "r"(TMEM_COLS)
                         : "memory");
    }
}

template <int MODE, int CL>
static cudaError_t set_attr() {
    return cudaFuncSetAttribute(lce_gemm_kernel<MODE, CL>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, GEMM_SMEM_BYTES);
}

cudaError_t gemm_set_attributes() {
    cudaError_t e;
    if ((e = set_attr<MODE_LSE, 1>()) != cudaSuccess) return e;
    if ((e = set_attr<MODE_LSE_P, 1>()) != cudaSuccess) return e;
    if ((e = set_attr<MODE_G, 1>()) != cudaSuccess) return e;
    if ((e = set_attr<MODE_BWD, 1>()) != cudaSuccess) return e;
    if ((e = set_attr<MODE_LSE, 2>()) != cudaSuccess) return e;
    if ((e = set_attr<MODE_LSE_P, 2>()) != cudaSuccess) return e;
    if ((e = set_attr<MODE_G, 2>()) != cudaSuccess) return e;
    if ((e = set_attr<MODE_BWD, 2>()) != cudaSuccess) return e;
    return set_attr<MODE_DH, 2>();
}

template <int MODE, int CL>
static cudaError_t launch_one(const GemmParams &p, int grid, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(GEMM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = GEMM_SMEM_BYTES;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, lce_gemm_kernel<MODE, CL>, p);
}

cudaError_t launch_gemm(int mode, int cluster, const GemmParams &p, int grid, cudaStream_t s) {
    cudaError_t e;
    if (cluster == 2) {
        switch (mode) {
            case MODE_LSE: e = launch_one<MODE_LSE, 2>(p, grid, s); break;
            case MODE_LSE_P: e = launch_one<MODE_LSE_P, 2>(p, grid, s); break;
            case MODE_G: e = launch_one<MODE_G, 2>(p, grid, s); break;
            case MODE_DH: e = launch_one<MODE_DH, 2>(p, grid, s); break;
            default: e = launch_one<MODE_BWD, 2>(p, grid, s); break;
        }
    } else {
        switch (mode) {
            case MODE_LSE: e = launch_one<MODE_LSE, 1>(p, grid, s); break;
            case MODE_LSE_P: e = launch_one<MODE_LSE_P, 1>(p, grid, s); break;
            case MODE_G: e = launch_one<MODE_G, 1>(p, grid, s); break;
            case MODE_BWD: e = launch_one<MODE_BWD, 1>(p, grid, s); break;
            default: return cudaErrorInvalidValue;   // the wide dH tiles need CTA pairs
        }
    }
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// Largest number of CTA pairs of the gradient kernel that fit on the device at
// once (the persistent grid is sized to it).
cudaError_t gemm_max_pairs(int *pairs) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(GEMM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = GEMM_SMEM_BYTES;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaOccupancyMaxActiveClusters(pairs, lce_gemm_kernel<MODE_BWD, 2>, &cfg);
}

}  // namespace lce
