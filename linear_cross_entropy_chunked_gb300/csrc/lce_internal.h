// Internal declarations shared by the kernels and the C-ABI host code.
// Not part of the public interface (that is include/lce.h).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace lce {

// ---------------------------------------------------------------- GEMM tiling
// One CTA per SM, persistent. A 128 x 256 fp32 accumulator tile lives in TMEM
// (256 columns); two of them (512 columns = all of TMEM) let the epilogue of
// tile t overlap the MMAs of tile t+1.
constexpr int BM = 128;            // UMMA M (TMEM lanes)
constexpr int BN = 256;            // UMMA N (TMEM columns per accumulator)
constexpr int BK = 64;             // one 128-byte swizzle row of bf16
constexpr int UMMA_K = 16;         // K of one tcgen05.mma kind::f16
constexpr int A_BYTES = BM * BK * 2;             // 16 KB
constexpr int B_BYTES = BN * BK * 2;             // 32 KB
// Pipeline per CTA. One CTA per tile: 4 stages of A (16 KB) + B (32 KB). CTA
// pair on one 256 x 256 tile (tcgen05 cta_group::2): each CTA holds its own A
// rows and half of B, 6 stages of 16 + 16 KB.
// Pipeline stages: A (128 rows x 64) plus this CTA's share of B. WIDE: the
// CTA-pair dH tiles 512 columns wide (two N = 256 MMAs share A), whose stage
// carries two B halves.
template <int CL, bool WIDE = false> struct Pipe {
    static constexpr int kBBytes = (WIDE ? 2 : 1) * B_BYTES / CL;
    static constexpr int kStageBytes = A_BYTES + kBBytes;
    static constexpr int kStages = (4 * 48 * 1024) / kStageBytes;
};
constexpr int MAX_STAGES = 6;
constexpr int STAGES = 4;                                  // one-CTA pipeline
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;             // 48 KB
constexpr int STAGING_BYTES = 16384;  // per epilogue column half: one 128-row x 128-byte store box
constexpr int PIPE_BYTES = 4 * 48 * 1024;      // both pipelines use 192 KB
constexpr int GEMM_SMEM_BYTES = PIPE_BYTES + 2 * STAGING_BYTES + 1024;  // + 1 KB alignment
constexpr int NUM_EPI_WARPS = 8;   // warps 0..7: TMEM lane quarter = warp % 4, column half = warp / 4
constexpr int PRODUCER_WARP = 8;
constexpr int MMA_WARP = 9;
constexpr int GEMM_THREADS = 320;
constexpr int SCHED_DEPTH = 4;
constexpr int TMEM_COLS = 512;
constexpr int BN_WIDE = 512;   // MODE_DH tile width: both 256-column TMEM accumulators
// dH tiles (256 rows x 512 columns on a CTA pair) run over the whole vocabulary
// while the dW tiles, whose 256 x 256 shape needs more operand bytes per flop
// and which also stage and reduce-add their fp32 output, run concurrently on the
// other SMs. The phase is shortest when both sets end together: measured on a
// GB300 that is about 32 dH tiles (a dH tile pair runs ~1.3x the flop rate of a
// dW one; 76 pairs). A chunk with fewer dH tiles splits them along the
// vocabulary until there are at least DH_SPLIT_TILES, in at most DH_MAX_SPLITS
// parts, for vocabularies of at least DH_SPLIT_MIN_V; more dH tiles than that
// leave the dW tiles to the end of the phase (measured slower, both with one dW
// contraction per chunk and per pair of chunks).
constexpr int DH_SPLIT_TILES = 28;
constexpr int DH_MAX_SPLITS = 4;
constexpr long long DH_SPLIT_MIN_V = 8192;
constexpr int PART_COLS = 128;     // columns covered by one (max, sum) partial

// Epilogue / tile-set modes of the GEMM kernel.
enum GemmMode : int {
    MODE_LSE = 0,     // logits tiles -> per-(row, 128-col) (max, sumexp) partials + target logit
    MODE_LSE_P = 1,   // ... + store P' = exp(z - max_part) as bf16 into the chunk buffer
    MODE_G = 2,       // logits tiles -> G = (exp(z - lse) - onehot) * scale as bf16 (given lse)
    MODE_BWD = 3,     // dH tiles (G W) followed by dW tiles (G^T H) in one persistent launch
    MODE_DH = 4       // dH tiles only, 256 rows x 512 columns per CTA pair (CTA pairs only)
};

// Scale of row i of G: dloss (a scalar, or row i of a per-row vector) divided
// by N_valid for the mean reduction; 0 for rows that do not count.
__device__ __forceinline__ float lce_row_scale(const float *dloss, int dloss_per_row, int mean,
                                               int n_valid, long long grow, bool y_ok) {
    if (!y_ok) return 0.f;
    const float d = dloss ? dloss[dloss_per_row ? grow : 0] : 1.f;
    if (mean) return n_valid > 0 ? d / static_cast<float>(n_valid) : 0.f;
    return d;
}

// fp16 inputs: G is stored in fp16, where dloss / N_valid (~1e-4 at the
// workloads' sizes) would push it below the format's range. So for fp16 the
// stored G is (p - onehot) * F16_G_SCALE (|G| <= 2^14), and the gradient
// epilogues multiply the dH / dW accumulators by (dloss / N_valid) / F16_G_SCALE
// (reduction mean; dloss / F16_G_SCALE for sum). bf16 keeps the full scale in G.
constexpr float F16_G_SCALE = 16384.f;

// Scale of row i of the stored G.
__device__ __forceinline__ float lce_store_scale(const float *dloss, int dloss_per_row, int mean,
                                                 int n_valid, long long grow, bool y_ok, int f16) {
    if (!f16) return lce_row_scale(dloss, dloss_per_row, mean, n_valid, grow, y_ok);
    return y_ok ? F16_G_SCALE : 0.f;
}

// Factor the gradient epilogues apply to their accumulators (1 for bf16).
__device__ __forceinline__ float lce_out_scale(const float *dloss, int mean, int n_valid, int f16) {
    if (!f16) return 1.f;
    const float d = dloss ? dloss[0] : 1.f;
    if (mean) return n_valid > 0 ? d / (static_cast<float>(n_valid) * F16_G_SCALE) : 0.f;
    return d / F16_G_SCALE;
}

// Workspace header (int32 words).
enum : int {
    HDR_FLAG = 0,       // bit 0: label out of range, bit 1: pipeline wait timed out
    HDR_NVALID = 1,
    HDR_COUNTERS = 16,  // one dynamic tile counter per GEMM launch of a call
};
constexpr int FLAG_LABEL = 1;
constexpr int FLAG_TIMEOUT = 2;

struct GemmParams {
    CUtensorMap tmA0;      // logits A = H (K-major) | dH A = G (K-major)
    CUtensorMap tmB0;      // logits B = W (K-major) | dH B = W (MN-major)
    CUtensorMap tmA1;      // dW A = G^T, read from the chunk buffer G [C][ldg] (MN-major;
                           // 3-D: {64 columns, rows, 64-column blocks})
    CUtensorMap tmB1;      // dW B = H chunk^T [D][C] (K-major)
    CUtensorMap tmS0;      // output store: P' / G chunk buffer (bf16) | dH chunk (bf16)
    CUtensorMap tmS1;      // dW output store / reduce-add (fp32)
    int m_blocks0, n_blocks0, k_blocks0;
    int m_blocks1, n_blocks1, k_blocks1;   // dW tiles (0 in logits launches)
    int total_tiles;       // scheduling units: tiles, or tile pairs for CTA pairs
    int rows;              // rows in this chunk
    int row0;              // first global row of this chunk
    int a_row0;            // logits: row coordinate of the chunk's first row in the H map
    int V, D;
    long long ignore_index;
    const long long *y;    // labels, global [N]
    int *tile_counter;
    int *hdr;
    const float *dloss;    // device scalar, per-row vector, or null (= 1)
    int dloss_per_row;     // 1: dloss[N] (reduction none)
    int mean;              // 1: G scaled by 1 / N_valid (reduction mean)
    // logits epilogue
    float2 *parts;         // [rows][nparts] (max, sumexp)
    int nparts;
    float *zy;             // [rows] target logits
    __nv_bfloat16 *G;      // [rows][ldg] P' or G
    int ldg;
    const float *lse;      // global [N] (MODE_G)
    // backward epilogues
    __nv_bfloat16 *dH;     // global [N][D]
    float *dW;             // [V][D]
    int dw_accumulate;     // 0: store, 1: add to existing dW
    int dh_fp32;           // 1: dH tiles stored as fp32 (tmS0 an fp32 map)
    // dH launches: the vocabulary (K) range of every dH tile split in k_splits
    // parts of kb_per_split k blocks; part s stores fp32 partial sums at row
    // offset s * split_rows of the tmS0 map (k_splits <= 1: one part, no offset)
    int k_splits, kb_per_split, split_rows;
    int f16;               // 1: fp16 operands (H, W, G) and fp16 P' / G / dH stores
    unsigned long long timeout_ns;
};

struct MergeParams {
    const float2 *parts;   // [rows][nparts] (max, sumexp) per 128-column slab
    int nparts;
    const float *zy;
    __nv_bfloat16 *G;
    int ldg;
    int rows, row0, V;
    long long ignore_index;
    const long long *y;
    const int *hdr;
    const float *dloss;
    int dloss_per_row;
    int mean;
    int f16;               // fp16 inputs: slab factors use lce_store_scale
    float *lse;            // global [N]
    float *loss_rows;      // global [N] (the caller's loss vector for reduction none)
};

struct TransposeParams {
    const __nv_bfloat16 *src;   // [rows][ld_src]
    int ld_src;
    __nv_bfloat16 *dst_t;       // [cols][ld_t]
    int ld_t;
    int rows, cols;
};


// The step between a chunk's logits GEMM and its gradient GEMMs on the fused
// path, one launch: for each row, lse from the slab partials, the row's loss,
// and P' -> G in place (each of `segs` CTAs of a row recomputes the row's lse
// from the partials, in the same order, and rescales its own segment of the
// row); then, in the CTAs after those, the H chunk transposed for the dW
// contraction (tp.rows == 0: no transpose).
constexpr int PREP_THREADS = 256;
constexpr int PREP_VPT = 8;                                  // 8-column vectors per thread
constexpr int PREP_VEC_PER_CTA = PREP_THREADS * PREP_VPT;    // 2048 vectors = 16384 columns
struct PrepParams {
    MergeParams m;              // parts, zy, y, hdr, dloss, scales, lse, loss_rows
    int ldg;
    int segs;                   // CTAs per row
    TransposeParams tp;
    int tt_x;                   // transpose tiles along D (64 columns each)
};

// Cross-entropy over precomputed logits Z [N][ld] (bf16 or fp32), one row at a time.
enum : int { CE_BF16 = 0, CE_FP32 = 1, CE_FP16 = 2 };   // logits dtype codes of lce_ce_logits

struct CELogitsParams {
    const void *Z;
    void *dZ;              // null: forward only; may equal Z (gradient written in place)
    long long ld;          // row stride of Z and dZ (elements)
    int dtype;             // CE_BF16, CE_FP32 or CE_FP16
    long long N, V;
    long long ignore_index;
    const long long *y;
    int *hdr;              // workspace header: N_valid in, status flags out
    const float *dloss;
    int dloss_per_row;
    int mean;
    float *lse;            // [N]
    float *loss_rows;      // [N]
};

// final RMSNorm (forward and backward row kernels)
constexpr int NRM_THREADS = 256;
constexpr int NRM_GRID = 256;                        // fixed: one dgamma partial slot per CTA
constexpr long long NRM_MAX_D = NRM_THREADS * 8 * 4; // 4 vectors of 8 bf16 per thread

struct NormParams {
    const __nv_bfloat16 *X;      // [rows][D]
    const __nv_bfloat16 *gamma;  // [D]
    __nv_bfloat16 *H;            // forward output [rows][D]
    float *rstd;                 // forward output [rows] or null
    const void *dH;              // backward input [rows][D], bf16 or fp32
    int dh_fp32;
    int dh_splits;               // fp32 dH: the sum of this many partial arrays,
    long long dh_split_stride;   // this many elements apart (dh_splits <= 1: one)
    __nv_bfloat16 *dX;           // backward output [rows][D]
    float *part;                 // backward: [NRM_GRID][D] dgamma partials
    int first;                   // 1: the partials start from zero
    long long rows;
    int D;
    float eps;
};

// launchers (return cudaError_t of the launch)
// cluster = 1: one CTA per 128 x 256 tile; 2: a CTA pair per 256 x 256 tile
// (tcgen05 cta_group::2, each CTA loading its own A rows and half of B).
// `grid` counts CTAs (a multiple of `cluster`).
cudaError_t launch_gemm(int mode, int cluster, const GemmParams &p, int grid, cudaStream_t s);
cudaError_t gemm_max_pairs(int *pairs);
cudaError_t launch_label_scan(const long long *y, long long N, long long V, long long ign,
                              int *hdr, cudaStream_t s);
// *out (device int64) = number of labels in [0, V) that are not ign
cudaError_t launch_count_valid(const long long *y, long long N, long long V, long long ign,
                               long long *out, cudaStream_t s);
// hdr[HDR_NVALID] = *n_total (device int64), for a mean over several shards' rows
cudaError_t launch_set_nvalid(const long long *n_total, int *hdr, cudaStream_t s);
cudaError_t launch_merge(const MergeParams &p, cudaStream_t s);
cudaError_t launch_transpose(const TransposeParams &p, cudaStream_t s);
cudaError_t launch_prep(const PrepParams &p, cudaStream_t s);
cudaError_t launch_loss_finalize(const float *loss_rows, long long N, const int *hdr,
                                 float *loss, int mean, cudaStream_t s);
cudaError_t launch_ce_logits(const CELogitsParams &p, int sms, cudaStream_t s);
cudaError_t gemm_set_attributes();
cudaError_t aux_set_attributes();
cudaError_t ce_set_attributes();
cudaError_t launch_wait_selftest(int *hdr, unsigned long long limit_ns, cudaStream_t s);
// dst[i] (bf16 / fp16, n elements) = (accumulate ? dst[i] : 0) + the sum over
// s = 0 .. splits-1, in that order, of src[s * stride + i] (fp32)
cudaError_t launch_combine_dh(const float *src, int splits, long long stride, void *dst,
                              long long n, bool f16, bool accumulate, int sms, cudaStream_t s);
cudaError_t launch_rmsnorm_fwd(const NormParams &p, cudaStream_t s);
cudaError_t launch_rmsnorm_bwd(const NormParams &p, cudaStream_t s);
cudaError_t launch_dgamma_reduce(const float *part, int D, float *dgamma, cudaStream_t s);

constexpr float LOG2E_F = 1.4426950408889634f;

// Largest vocabulary: keeps every TMA coordinate and tile index in int32.
constexpr long long MAX_V = 1ll << 30;

}  // namespace lce
