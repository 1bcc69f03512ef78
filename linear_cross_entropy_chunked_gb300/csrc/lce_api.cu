// C ABI of the fused chunked linear + cross-entropy library: argument checks,
// workspace layout, tensor-map encoding and the per-chunk launch sequence.
// Declarations and the contract of every entry point are in include/lce.h.
//
// The token axis is cut into chunks of `chunk` rows ("Arquitectura interna de
// Unsloth y optimizacion en Triton", section 3: token blocks; "Unsloth
// Architecture: Manual Triton Backpropagation, Fused Cross-Entropy, and 80% VRAM
// Cut", pillar 1: chunks of tokens, logits discarded after each chunk). The
// only HBM state beyond the outputs is O(chunk * V): the (max, sumexp) slab
// partials of a chunk and bf16 [chunk, V] buffers that hold exp(z - slab max),
// then G: two by default (chunks go in pairs that share one dW contraction),
// one with LCE_LOW_MEMORY.
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdlib>
#include <mutex>
#include <vector>

#include "../../include/lce.h"
#include "lce_internal.h"

using namespace lce;

namespace {

thread_local int g_launches = 0;

constexpr unsigned long long kDefaultTimeoutNs = 2000000000ull;  // 2 s per pipeline wait

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::mutex g_mu;
constexpr int kMaxDevices = 64;
bool g_dev_ready[kMaxDevices] = {};
int g_dev_sms[kMaxDevices] = {};
int g_dev_pairs[kMaxDevices] = {};   // co-resident CTA pairs of the GEMM kernel (0: no pairs)

// GEMM tiles run on CTA pairs (tcgen05 cta_group::2, 256 x 256 tiles) when the
// device can co-schedule them; LCE_GEMM_CLUSTER=1 selects one CTA per 128 x 256
// tile instead (same work and results; measured ~8 % slower on the Llama-3 head).
int cluster_choice() {
    const char *e = getenv("LCE_GEMM_CLUSTER");
    return (e && e[0] == '1') ? 1 : 2;
}

lce_status init_device(int *sms, int *pairs) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return LCE_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return LCE_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_encode) {
        cudaDriverEntryPointQueryResult q;
        void *fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn)
            return LCE_ERR_CUDA;
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    if (!g_dev_ready[dev]) {
        int major = 0, minor = 0, n = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return LCE_ERR_CUDA;
        if (major != 10 || minor != 3) return LCE_ERR_UNSUPPORTED;
        if (gemm_set_attributes() != cudaSuccess) return LCE_ERR_CUDA;
        if (aux_set_attributes() != cudaSuccess) return LCE_ERR_CUDA;
        if (ce_set_attributes() != cudaSuccess) return LCE_ERR_CUDA;
        int np = 0;
        if (gemm_max_pairs(&np) != cudaSuccess) {
            cudaGetLastError();
            np = 0;
        }
        g_dev_sms[dev] = n;
        g_dev_pairs[dev] = np;
        g_dev_ready[dev] = true;
    }
    *sms = g_dev_sms[dev];
    *pairs = cluster_choice() == 2 ? g_dev_pairs[dev] : 0;
    return LCE_OK;
}

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
inline long long cdiv(long long a, long long b) { return (a + b - 1) / b; }

struct Layout {
    long long C = 0;         // rows per chunk
    long long nchunks = 0;
    int nparts = 0;          // 128-column slabs per row
    int ldg = 0;             // row stride of the chunk buffer (elements)
    int ldt = 0;             // row stride (elements) of H^T: rows of one chunk (or of a
                             // pair of chunks) rounded up to 64
    int nbuf = 1;            // chunk buffers: with two, the dW contraction of a pair of
                             // chunks runs once, over both chunks' G (K = 2 chunks)
    size_t gbuf_bytes = 0;   // bytes of one chunk buffer (the two are contiguous)
    bool frozen_w = false;   // no dW contraction (LCE_FROZEN_W)
    int dh_splits = 1;       // vocabulary parts of a full chunk's dH tiles
    long long ldp = 0;       // rows per fp32 dH partial array: chunk rows rounded up to 128
    size_t off_loss_rows = 0, off_zy = 0, off_parts = 0, off_G = 0, off_HT = 0, off_dHp = 0;
    size_t total = 0;
    size_t fwd_total = 0;    // the forward's share: header, row losses, target logits, partials
    size_t hdr_bytes = 0;
};

// Vocabulary parts of the dH tiles of a chunk of `rows` rows (CTA-pair tiles of
// 256 x 512): enough for DH_SPLIT_TILES tiles, at most DH_MAX_SPLITS and at most
// one per 64-column k block; one below DH_SPLIT_MIN_V. A function of the shapes
// alone, so a result does not depend on the device it ran on.
// With W frozen the dH tiles have the GPU to themselves: they are split into the
// most parts (at most DH_MAX_SPLITS) that keep them within one wave of the
// DH_ALONE_PAIRS CTA pairs a GB300 holds at once (152 SMs).
constexpr int DH_ALONE_PAIRS = 76;

int dh_splits_for(long long rows, long long D, long long V, bool frozen_w = false) {
    if (V < DH_SPLIT_MIN_V || rows <= 0) return 1;
    const long long tiles = cdiv(cdiv(rows, BM), 2) * cdiv(D, BN_WIDE);
    long long sp = frozen_w ? DH_ALONE_PAIRS / tiles : cdiv(DH_SPLIT_TILES, tiles);
    if (sp > DH_MAX_SPLITS) sp = DH_MAX_SPLITS;
    if (sp > cdiv(V, BK)) sp = cdiv(V, BK);
    return sp < 1 ? 1 : static_cast<int>(sp);
}

bool make_layout(long long N, long long D, long long V, long long chunk, Layout &L,
                 bool frozen_w = false, bool low_mem = false) {
    if (N < 0 || D <= 0 || V <= 0 || chunk <= 0) return false;
    if (D % 8 != 0) return false;
    if (N > 0x7fffffffll || D > 0x7fffffffll || V > MAX_V) return false;
    L.C = chunk < (N > 0 ? N : 1) ? chunk : (N > 0 ? N : 1);
    L.nchunks = N > 0 ? cdiv(N, L.C) : 0;
    L.nparts = static_cast<int>(cdiv(V, PART_COLS));
    L.ldg = static_cast<int>(align_up(static_cast<size_t>(V), BN));
    if (static_cast<unsigned long long>(L.C) * L.ldg > (1ull << 40)) return false;
    L.hdr_bytes = align_up(sizeof(int) * (HDR_COUNTERS + 3 * L.nchunks + 2), 1024);
    size_t off = L.hdr_bytes;
    L.off_loss_rows = off;
    off += align_up(sizeof(float) * static_cast<size_t>(N > 0 ? N : 1), 1024);
    L.off_zy = off;
    off += align_up(sizeof(float) * static_cast<size_t>(L.C), 1024);
    L.off_parts = off;
    off += align_up(sizeof(float2) * static_cast<size_t>(L.C) * L.nparts, 1024);
    L.off_G = off;
    L.fwd_total = off;
    // two chunk buffers when there is a dW contraction and more than one chunk:
    // chunks are taken in pairs, the second chunk's G goes into the buffer after the
    // first's, and one dW contraction runs over both (K = the pair's rows), which
    // halves the fp32 read-modify-write of dW (LCE_LOW_MEMORY: one buffer, one dW
    // contraction per chunk). The buffers are contiguous rows of one [2C][ldg]
    // array (2 * C * ldg bytes each, a multiple of 512), and the second chunk's
    // columns of H^T start at column C, which the transpose's 16-byte stores need to
    // be a multiple of 8.
    // With W frozen there is no dW contraction; two buffers then let a chunk's
    // logits GEMM run on the CTA pairs its predecessor's dH GEMM leaves free.
    L.nbuf = (!low_mem && L.nchunks > 1 && (frozen_w || L.C % 8 == 0)) ? 2 : 1;
    L.gbuf_bytes = 2 * static_cast<size_t>(L.C) * L.ldg;
    off += align_up(static_cast<size_t>(L.nbuf) * L.gbuf_bytes, 1024);
    // H chunk^T [D][ldt]: the K-major B operand of the dW contraction (none when W
    // is frozen)
    L.frozen_w = frozen_w;
    L.ldt = static_cast<int>(align_up(static_cast<size_t>(L.nbuf) * L.C, 64));
    L.off_HT = off;
    if (!frozen_w) off += align_up(2 * static_cast<size_t>(D) * L.ldt, 1024);
    // fp32 dH partial sums of a split dH contraction, one [ldp][D] array per part
    // (a single array, past `total`, serves callers that accumulate into dH)
    L.dh_splits = dh_splits_for(L.C, D, V, frozen_w);
    // the first chunk of a pair runs its dH tiles alone (split for all pairs)
    if (L.nbuf == 2 && dh_splits_for(L.C, D, V, true) > L.dh_splits)
        L.dh_splits = dh_splits_for(L.C, D, V, true);
    L.ldp = static_cast<long long>(align_up(static_cast<size_t>(L.C), BM));
    L.off_dHp = off;
    if (L.dh_splits > 1)
        off += align_up(4 * static_cast<size_t>(L.dh_splits) * L.ldp * static_cast<size_t>(D), 1024);
    L.total = off;
    return true;
}

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Workspace of the final-RMSNorm path: the loss path's layout, then the chunk's
// normalised rows H (bf16), the chunk's dH (fp32) and the dgamma partials.
struct NormLayout {
    Layout L;
    size_t off_H = 0, off_dH = 0, off_part = 0, total = 0;
};

// Bytes past the loss path's workspace that accumulating into dH (and the
// RMSNorm path) need: one fp32 dH array for the chunk, added to the caller's dH
// once the chunk is done; none when the layout already holds split partials.
size_t acc_dh_bytes(const Layout &L, long long D) {
    if (L.dh_splits > 1) return 0;
    return align_up(4 * static_cast<size_t>(L.ldp) * static_cast<size_t>(D), 1024);
}

bool make_norm_layout(long long N, long long D, long long V, long long chunk, NormLayout &NL,
                      bool frozen_w = false, bool low_mem = false) {
    // W trained: chunk pairs with one dW contraction each, as on the loss path; W
    // frozen: one chunk buffer
    if (!make_layout(N, D, V, chunk, NL.L, frozen_w, low_mem || frozen_w)) return false;
    if (D > NRM_MAX_D) return false;
    // the chunk's dH (fp32): the layout's partial arrays, or one array past them
    NL.off_dH = NL.L.off_dHp;
    size_t off = NL.L.total + acc_dh_bytes(NL.L, D);
    NL.off_H = off;   // the normalised rows of a chunk (of a pair of chunks with two buffers)
    off += align_up(2 * static_cast<size_t>(NL.L.nbuf) * NL.L.C * D, 1024);
    NL.off_part = off;
    off += align_up(4 * static_cast<size_t>(NRM_GRID) * D, 1024);
    NL.total = off;
    return true;
}

// Element types of the tensor maps.
enum MapType { MAP_BF16, MAP_F16, MAP_F32 };

// Tensor map over a row-major array with the 128-byte swizzle of the MMA
// operand tiles and of the epilogue staging boxes; zero fill out of bounds on
// loads, clipping on stores.
bool encode_map(CUtensorMap *m, const void *base, int rank, const uint64_t *dims,
                const uint64_t *strides_bytes, const uint32_t *box, MapType type) {
    cuuint64_t d[3];
    cuuint64_t st[2];
    cuuint32_t bx[3];
    cuuint32_t es[3] = {1, 1, 1};
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        bx[i] = box[i];
    }
    for (int i = 0; i + 1 < rank; ++i) st[i] = strides_bytes[i];
    const CUtensorMapDataType dt = type == MAP_F32   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : type == MAP_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                     : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    CUresult r = g_encode(m, dt,
                          rank, const_cast<void *>(base), d, st, bx, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// MMA operand tile load map: 2-D, 16-bit elements (bf16 or fp16), box
// {box_inner, box_outer}.
bool encode_2d(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer,
               uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer,
               MapType type = MAP_BF16) {
    const uint64_t dims[2] = {inner, outer};
    const uint64_t st[1] = {row_stride_bytes};
    const uint32_t box[2] = {box_inner, box_outer};
    return encode_map(m, base, 2, dims, st, box, type);
}

// Epilogue store map: 2-D, box = 128 bytes x box_rows rows (128: a column half
// of a gradient tile; 32: one warp's rows of a logits tile).
bool encode_store_2d(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer,
                     uint64_t row_stride_bytes, MapType type, uint32_t box_rows = 128) {
    const uint64_t dims[2] = {inner, outer};
    const uint64_t st[1] = {row_stride_bytes};
    const uint32_t box[2] = {type == MAP_F32 ? 32u : 64u, box_rows};
    return encode_map(m, base, 2, dims, st, box, type);
}

struct Ctx {
    const __nv_bfloat16 *H, *W;
    const long long *y;
    long long N, D, V, ign;
    Layout L;
    uint8_t *ws;
    int *hdr;
    float *loss_rows, *zy;
    float2 *parts;
    __nv_bfloat16 *Gb[2];   // the chunk buffers (Gb[1] == Gb[0] with one)
    __nv_bfloat16 *HT;
    int sms;
    int pairs;   // > 0: GEMMs run as CTA pairs (cluster of 2), at most this many at once
    int reduction;       // LCE_REDUCTION_*
    bool h_chunked;      // H is a buffer of one chunk's rows (of a pair's with two chunk
                         // buffers: chunk k at rows (k mod 2) * C), refilled per chunk
    bool f16;            // H, W, G and dH are fp16 (bf16 otherwise)
    MapType t16;         // the 16-bit map type of this call
    cudaStream_t s;
    CUtensorMap tmH_K, tmW_K, tmW_MN;
};

// Row of H (c.H) where the chunk starting at row0 begins.
inline long long h_row(const Ctx &c, long long row0) {
    return c.h_chunked ? ((row0 / c.L.C) % c.L.nbuf) * c.L.C : row0;
}

// ---- optional per-kernel event timing (lce_profile_*)
struct ProfPair {
    int kind;
    cudaEvent_t a, b;
};
std::mutex g_prof_mu;
std::atomic<bool> g_prof_on{false};   // read without the mutex on every launch
std::vector<ProfPair> g_prof_pending;
std::vector<cudaEvent_t> g_prof_pool;
double g_prof_ms[LCE_KERNEL_KINDS] = {};
int64_t g_prof_n[LCE_KERNEL_KINDS] = {};

cudaEvent_t prof_event() {
    if (!g_prof_pool.empty()) {
        cudaEvent_t e = g_prof_pool.back();
        g_prof_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

// Records the start event of a launch of `kind`; returns the pair index or -1.
int prof_begin(int kind, cudaStream_t s) {
    if (!g_prof_on) return -1;
    std::lock_guard<std::mutex> lock(g_prof_mu);
    ProfPair p{kind, prof_event(), prof_event()};
    if (!p.a || !p.b) return -1;
    cudaEventRecord(p.a, s);
    g_prof_pending.push_back(p);
    return static_cast<int>(g_prof_pending.size()) - 1;
}

void prof_end(int idx, cudaStream_t s) {
    if (idx < 0) return;
    std::lock_guard<std::mutex> lock(g_prof_mu);
    cudaEventRecord(g_prof_pending[idx].b, s);
}

#define LCE_LAUNCH_KIND(kind, stream, expr)                 \
    do {                                                    \
        const int _pi = prof_begin((kind), (stream));       \
        if ((expr) != cudaSuccess) return LCE_ERR_CUDA;     \
        prof_end(_pi, (stream));                            \
        ++g_launches;                                       \
    } while (0)

#define LCE_LAUNCH(expr) LCE_LAUNCH_KIND(LCE_KERNEL_OTHER, c.s, expr)

// A second stream per device for the dW kernel that runs beside the dH kernel
// of a gradient phase (forked from and joined back to the caller's stream
// through two events). The mutex keeps the record / wait / launch sequence of
// one call together when several host threads use the same device.
struct SideStream {
    cudaStream_t s = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
    std::mutex mu;
};
SideStream g_side[64];
std::mutex g_side_mu;

SideStream *side_stream() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(g_side_mu);
    SideStream &ss = g_side[dev];
    if (!ss.s) {
        cudaStream_t st = nullptr;
        if (cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking) != cudaSuccess) return nullptr;
        if (cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming) != cudaSuccess)
            return nullptr;
        ss.s = st;   // last: marks the set as complete
    }
    return &ss;
}

lce_status setup(Ctx &c, const void *H, const void *W, const int64_t *y, int64_t N, int64_t D,
                 int64_t V, int64_t ign, int64_t chunk, void *ws, size_t ws_bytes,
                 lce_stream_t stream, bool h_chunked = false, bool f16 = false,
                 bool frozen_w = false, bool fwd_only = false, bool low_mem = false) {
    g_launches = 0;
    if (!make_layout(N, D, V, chunk, c.L, frozen_w, low_mem)) return LCE_ERR_INVALID_ARG;
    if (!ws) return LCE_ERR_INVALID_ARG;
    if (N > 0 && (!H || !y)) return LCE_ERR_INVALID_ARG;
    if (!W) return LCE_ERR_INVALID_ARG;
    if (!aligned16(ws) || !aligned16(W) || (H && !aligned16(H)) || (y && !aligned16(y)))
        return LCE_ERR_ALIGNMENT;
    if (ws_bytes < (fwd_only ? c.L.fwd_total : c.L.total)) return LCE_ERR_WORKSPACE;
    lce_status st = init_device(&c.sms, &c.pairs);
    if (st != LCE_OK) return st;
    c.H = static_cast<const __nv_bfloat16 *>(H);
    c.W = static_cast<const __nv_bfloat16 *>(W);
    c.y = reinterpret_cast<const long long *>(y);
    c.N = N;
    c.D = D;
    c.V = V;
    c.ign = ign;
    c.ws = static_cast<uint8_t *>(ws);
    c.hdr = reinterpret_cast<int *>(c.ws);
    c.loss_rows = reinterpret_cast<float *>(c.ws + c.L.off_loss_rows);
    c.zy = reinterpret_cast<float *>(c.ws + c.L.off_zy);
    c.parts = reinterpret_cast<float2 *>(c.ws + c.L.off_parts);
    c.Gb[0] = reinterpret_cast<__nv_bfloat16 *>(c.ws + c.L.off_G);
    c.Gb[1] = reinterpret_cast<__nv_bfloat16 *>(c.ws + c.L.off_G +
                                                (c.L.nbuf > 1 ? c.L.gbuf_bytes : 0));
    // (with two buffers Gb[1] is row C of one [2C][ldg] array starting at Gb[0])
    c.HT = reinterpret_cast<__nv_bfloat16 *>(c.ws + c.L.off_HT);
    c.s = reinterpret_cast<cudaStream_t>(stream);
    c.reduction = LCE_REDUCTION_MEAN;
    c.h_chunked = h_chunked;
    c.f16 = f16;
    c.t16 = f16 ? MAP_F16 : MAP_BF16;
    // with CTA pairs each CTA loads its own half (128 rows) of a 256-row W tile; the
    // pair MMA reads both CTAs' halves from their shared memory
    if (!encode_2d(&c.tmW_K, W, D, V, D * 2, BK, c.pairs > 0 ? BN / 2 : BN, c.t16)) return LCE_ERR_CUDA;
    if (!encode_2d(&c.tmW_MN, W, D, V, D * 2, 64, BK, c.t16)) return LCE_ERR_CUDA;
    if (N > 0 && !encode_2d(&c.tmH_K, H, D, h_chunked ? c.L.C * c.L.nbuf : N, D * 2, BK, BM, c.t16))
        return LCE_ERR_CUDA;
    if (cudaMemsetAsync(c.ws, 0, c.L.hdr_bytes, c.s) != cudaSuccess) return LCE_ERR_CUDA;
    LCE_LAUNCH(launch_label_scan(c.y, N, V, ign, c.hdr, c.s));
    return LCE_OK;
}

void base_params(const Ctx &c, GemmParams &p, long long row0, long long rows, int slot) {
    p.rows = static_cast<int>(rows);
    p.row0 = static_cast<int>(row0);
    p.V = static_cast<int>(c.V);
    p.D = static_cast<int>(c.D);
    p.ignore_index = c.ign;
    p.y = c.y;
    p.tile_counter = c.hdr + HDR_COUNTERS + slot;
    p.hdr = c.hdr;
    p.parts = c.parts;
    p.nparts = c.L.nparts;
    p.zy = c.zy;
    p.G = c.Gb[0];
    p.ldg = c.L.ldg;
    p.timeout_ns = kDefaultTimeoutNs;
    p.dloss_per_row = c.reduction == LCE_REDUCTION_NONE ? 1 : 0;
    p.mean = c.reduction == LCE_REDUCTION_MEAN ? 1 : 0;
    p.f16 = c.f16 ? 1 : 0;
}

// The logits launches of the chunk at row0 (MODE_LSE / _LSE_P / _G epilogue, P' or G
// into chunk buffer G).
struct LogitsSpec {
    int mode;
    long long row0, rows;
    int slot;
    const float *lse;       // MODE_G
    const float *dloss;
    __nv_bfloat16 *G;
};

lce_status logits_params(const Ctx &c, const LogitsSpec &l, GemmParams &p) {
    memset(&p, 0, sizeof(p));
    base_params(c, p, l.row0, l.rows, l.slot);
    p.tmA0 = c.tmH_K;
    p.a_row0 = static_cast<int>(h_row(c, l.row0));
    p.tmB0 = c.tmW_K;
    p.m_blocks0 = static_cast<int>(cdiv(l.rows, BM));
    p.n_blocks0 = static_cast<int>(cdiv(c.V, BN));
    p.k_blocks0 = static_cast<int>(cdiv(c.D, BK));
    const int cl = c.pairs > 0 ? 2 : 1;
    p.total_tiles = static_cast<int>(cdiv(p.m_blocks0, cl)) * p.n_blocks0;
    p.lse = l.lse;
    p.dloss = l.dloss;
    p.G = l.G;
    if (l.mode != MODE_LSE &&
        !encode_store_2d(&p.tmS0, l.G, c.V, l.rows, 2ull * c.L.ldg, c.t16, 32))
        return LCE_ERR_CUDA;
    return LCE_OK;
}

lce_status run_logits(const Ctx &c, int mode, long long row0, long long rows, int slot,
                      const float *lse, const float *dloss, __nv_bfloat16 *G) {
    GemmParams p;
    const lce_status st = logits_params(c, LogitsSpec{mode, row0, rows, slot, lse, dloss, G}, p);
    if (st != LCE_OK) return st;
    const int cl = c.pairs > 0 ? 2 : 1;
    const int units = cl == 2 ? c.pairs : c.sms;
    const int grid = cl * (p.total_tiles < units ? p.total_tiles : units);
    LCE_LAUNCH_KIND(LCE_KERNEL_LOGITS, c.s, launch_gemm(mode, cl, p, grid, c.s));
    return LCE_OK;
}

#define LCE_TRY(expr)                         \
    do {                                      \
        lce_status _st = (expr);              \
        if (_st != LCE_OK) return _st;        \
    } while (0)

// Where a gradient phase leaves dH: the caller's rows (bf16 / fp16, stored by the
// dH tiles directly), or fp32 partial sums, `parts` arrays of ldp rows x D (one
// per vocabulary part of the dH tiles), for a combining kernel to add up.
struct DhOut {
    void *ptr;
    bool fp32;
    int parts;
    long long ldp;
};

// Vocabulary parts for a chunk of `rows` rows: one off the CTA-pair path (its
// 256-column dH tiles are many), else the shapes' split, at most the layout's.
// alone: the dH tiles have the GPU to themselves (no dW tiles beside them).
int dh_parts(const Ctx &c, long long rows, bool alone) {
    if (c.pairs <= 0) return 1;
    const int sp = dh_splits_for(rows, c.D, c.V, c.L.frozen_w || alone);
    return sp < c.L.dh_splits ? sp : c.L.dh_splits;
}

// H chunk^T into columns col0 .. col0 + rows - 1 of H^T (the K-major B operand of
// the dW tiles; col0 = C for the second chunk of a pair).
lce_status run_transpose(const Ctx &c, long long row0, long long rows, long long col0) {
    const __nv_bfloat16 *Hc = c.H + h_row(c, row0) * c.D;
    TransposeParams tp;
    tp.src = Hc;
    tp.ld_src = static_cast<int>(c.D);
    tp.dst_t = c.HT + col0;
    tp.ld_t = c.L.ldt;
    tp.rows = static_cast<int>(rows);
    tp.cols = static_cast<int>(c.D);
    LCE_LAUNCH_KIND(LCE_KERNEL_MERGE, c.s, launch_transpose(tp, c.s));
    return LCE_OK;
}

// What one gradient launch set computes. The dH tiles of the chunk at row0 read
// its G (buffer G); the dW tiles, when there are any (dw_rows > 0), contract over
// dw_rows rows of G starting at Gdw (the chunk's own rows, or the rows of a pair of
// chunks) against as many columns of H^T.
struct GradSpec {
    __nv_bfloat16 *G;
    __nv_bfloat16 *Gdw;
    long long dw_rows;      // K of the dW tiles (0: no dW tiles)
    bool transposed;        // H^T is in place (else it is made first, for this chunk)
    bool dh_alone;          // no dW tiles beside the dH tiles: split for all CTA pairs
    bool dw_only;           // the dW tiles alone (the chunk's dH is computed elsewhere)
    const LogitsSpec *beside = nullptr;   // with dh_alone: another chunk's logits tiles on
                                          // the pairs the dH tiles leave free, then on all
};

// *parts_used: the number of non-empty vocabulary parts written (fp32 output).
lce_status run_bwd(const Ctx &c, long long row0, long long rows, int slot, const DhOut &o,
                   float *dW, bool accumulate, const float *dloss, const GradSpec &g,
                   int *parts_used = nullptr) {
    GemmParams p;
    memset(&p, 0, sizeof(p));
    base_params(c, p, row0, rows, slot);
    p.G = g.G;
    void *dHc = o.ptr;
    const bool dh_fp32 = o.fp32;
    const int want_parts = (o.fp32 && o.parts > 1 && c.pairs > 0) ? o.parts : 1;
    // frozen W or the first chunk of a pair: the dH tiles only (no dW maps, dW untouched)
    const bool with_dw = !c.L.frozen_w && g.dw_rows > 0;
    const int cl = c.pairs > 0 ? 2 : 1;
    if (with_dw) {
        // the H chunk^T for the K-major B operand of the dW tiles
        if (!g.transposed) LCE_TRY(run_transpose(c, row0, rows, 0));
        // dW A = G^T read from G itself, MN-major: per k block a CTA's 128 vocabulary
        // columns x 64 rows as two 64-column blocks, fetched by one 3-D box {64
        // columns, 64 rows, 2 blocks} (x: the column within a block, y: the row, z: the
        // 64-column block, 128 bytes apart). The columns of the last block past V read
        // the buffer's padding; they meet only dW rows past V, which the store clips.
        const uint64_t dims[3] = {64, static_cast<uint64_t>(g.dw_rows),
                                  static_cast<uint64_t>(cdiv(c.V, 64))};
        const uint64_t strides[2] = {2ull * c.L.ldg, 128};
        const uint32_t box[3] = {64, BK, 2};
        if (!encode_map(&p.tmA1, g.Gdw, 3, dims, strides, box, c.t16)) return LCE_ERR_CUDA;
        if (!encode_2d(&p.tmB1, c.HT, g.dw_rows, c.D, 2ull * c.L.ldt, BK, BN / cl, c.t16))
            return LCE_ERR_CUDA;
        if (!encode_store_2d(&p.tmS1, dW, c.D, c.V, 4ull * c.D, MAP_F32)) return LCE_ERR_CUDA;
    }
    if (!encode_2d(&p.tmA0, g.G, c.V, rows, 2ull * c.L.ldg, BK, BM, c.t16)) return LCE_ERR_CUDA;
    p.tmB0 = c.tmW_MN;
    const uint64_t s0_rows = want_parts > 1 ? static_cast<uint64_t>(want_parts) * o.ldp : rows;
    if (!encode_store_2d(&p.tmS0, dHc, c.D, s0_rows, (dh_fp32 ? 4ull : 2ull) * c.D,
                         dh_fp32 ? MAP_F32 : c.t16))
        return LCE_ERR_CUDA;
    p.m_blocks0 = static_cast<int>(cdiv(rows, BM));
    p.n_blocks0 = static_cast<int>(cdiv(c.D, BN));
    p.k_blocks0 = static_cast<int>(cdiv(c.V, BK));
    p.m_blocks1 = with_dw ? static_cast<int>(cdiv(c.V, BM)) : 0;
    p.n_blocks1 = with_dw ? static_cast<int>(cdiv(c.D, BN)) : 0;
    p.k_blocks1 = with_dw ? static_cast<int>(cdiv(g.dw_rows, BK)) : 0;
    p.total_tiles = static_cast<int>(cdiv(p.m_blocks0, cl)) * p.n_blocks0 +
                    static_cast<int>(cdiv(p.m_blocks1, cl)) * p.n_blocks1;
    int parts = 1;
    if (want_parts > 1) {
        p.kb_per_split = static_cast<int>(cdiv(p.k_blocks0, want_parts));
        parts = static_cast<int>(cdiv(p.k_blocks0, p.kb_per_split));
        p.k_splits = parts;
        p.split_rows = static_cast<int>(o.ldp);
    }
    if (parts_used) *parts_used = parts;
    p.dH = static_cast<__nv_bfloat16 *>(dHc);
    p.dh_fp32 = dh_fp32 ? 1 : 0;
    p.dloss = dloss;   // fp16: the epilogues apply the uniform part of the scale
    p.dW = dW;
    p.dw_accumulate = accumulate ? 1 : 0;
    const int units = cl == 2 ? c.pairs : c.sms;
    // profiling kind: a pair's second chunk (its dH with both chunks' dW), a pair's
    // first chunk (its dH alone), or a chunk's whole gradient phase
    const int kind = (with_dw && g.dw_rows > rows) ? LCE_KERNEL_PHASE
                     : (!with_dw && (!c.L.frozen_w || g.beside)) ? LCE_KERNEL_DH
                                                                 : LCE_KERNEL_GRAD;
    if (cl == 2) {
        // CTA pairs: the dH tiles run 512 columns wide (two MMAs share each A
        // block: a quarter fewer operand bytes per flop) in one kernel with one
        // pair per tile (at most all pairs); the dW tiles run beside it in a
        // second kernel on the side stream, sized to exactly the pairs the dH
        // kernel leaves free, so the two grids fit on the GPU together whichever
        // the hardware dispatches first (nothing orders two ready grids on
        // separate hardware queues; a dW grid that took every SM would leave the
        // long dH tiles to run after it). A third launch, a dW grid as large as
        // the dH one, queued on the caller's stream behind the dH kernel, takes
        // over the dH kernel's SMs when it ends; both dW grids draw tiles from
        // the same counter.
        GemmParams ph = p;
        ph.n_blocks0 = static_cast<int>(cdiv(c.D, BN_WIDE));
        ph.m_blocks1 = ph.n_blocks1 = ph.k_blocks1 = 0;
        ph.total_tiles = g.dw_only ? 0 : static_cast<int>(cdiv(p.m_blocks0, cl)) * ph.n_blocks0 * parts;
        if (!with_dw && !g.beside) {
            const int gh = cl * (ph.total_tiles < units ? ph.total_tiles : units);
            if (ph.total_tiles > 0)
                LCE_LAUNCH_KIND(kind, c.s, launch_gemm(MODE_DH, cl, ph, gh, c.s));
            return LCE_OK;
        }
        if (!with_dw) {
            // the dH tiles beside another chunk's logits tiles: as with the dW grids
            // below, one logits grid on the side stream sized to the pairs the dH grid
            // leaves free and one behind the dH kernel, drawing from one counter
            GemmParams pl;
            LCE_TRY(logits_params(c, *g.beside, pl));
            SideStream *ss = side_stream();
            if (!ss) return LCE_ERR_CUDA;
            std::lock_guard<std::mutex> lock(ss->mu);
            const int dh_pairs = ph.total_tiles < units ? ph.total_tiles : units;
            const int free_pairs = units - dh_pairs;
            const int l1 = pl.total_tiles < free_pairs ? pl.total_tiles : free_pairs;
            const int l2 = pl.total_tiles < dh_pairs ? pl.total_tiles : dh_pairs;
            const int pi = prof_begin(kind, c.s);
            if (cudaEventRecord(ss->fork, c.s) != cudaSuccess ||
                cudaStreamWaitEvent(ss->s, ss->fork, 0) != cudaSuccess)
                return LCE_ERR_CUDA;
            int launched = 0;
            if (dh_pairs > 0) {
                if (launch_gemm(MODE_DH, cl, ph, cl * dh_pairs, c.s) != cudaSuccess) return LCE_ERR_CUDA;
                ++launched;
            }
            if (l1 > 0) {
                if (launch_gemm(g.beside->mode, cl, pl, cl * l1, ss->s) != cudaSuccess)
                    return LCE_ERR_CUDA;
                ++launched;
            }
            if (l2 > 0 && (dh_pairs > 0 || l1 == 0)) {
                if (launch_gemm(g.beside->mode, cl, pl, cl * l2, c.s) != cudaSuccess)
                    return LCE_ERR_CUDA;
                ++launched;
            }
            if (cudaEventRecord(ss->join, ss->s) != cudaSuccess ||
                cudaStreamWaitEvent(c.s, ss->join, 0) != cudaSuccess)
                return LCE_ERR_CUDA;
            prof_end(pi, c.s);
            g_launches += launched;
            return LCE_OK;
        }
        GemmParams pw = p;
        pw.m_blocks0 = 0;
        pw.k_splits = 0;
        pw.total_tiles = static_cast<int>(cdiv(p.m_blocks1, cl)) * p.n_blocks1;
        pw.tile_counter = c.hdr + HDR_COUNTERS + 2 * c.L.nchunks + 2 + slot / 2;
        SideStream *ss = side_stream();
        if (!ss) return LCE_ERR_CUDA;
        std::lock_guard<std::mutex> lock(ss->mu);
        const int dh_pairs = ph.total_tiles < units ? ph.total_tiles : units;
        const int free_pairs = units - dh_pairs;
        const int w1 = pw.total_tiles < free_pairs ? pw.total_tiles : free_pairs;
        const int w2 = pw.total_tiles < dh_pairs ? pw.total_tiles : dh_pairs;
        const int pi = prof_begin(kind, c.s);
        if (cudaEventRecord(ss->fork, c.s) != cudaSuccess ||
            cudaStreamWaitEvent(ss->s, ss->fork, 0) != cudaSuccess)
            return LCE_ERR_CUDA;
        int launched = 0;
        if (dh_pairs > 0) {
            if (launch_gemm(MODE_DH, cl, ph, cl * dh_pairs, c.s) != cudaSuccess) return LCE_ERR_CUDA;
            ++launched;
        }
        if (w1 > 0) {
            if (launch_gemm(MODE_BWD, cl, pw, cl * w1, ss->s) != cudaSuccess) return LCE_ERR_CUDA;
            ++launched;
        }
        if (w2 > 0 && (dh_pairs > 0 || w1 == 0)) {
            if (launch_gemm(MODE_BWD, cl, pw, cl * w2, c.s) != cudaSuccess) return LCE_ERR_CUDA;
            ++launched;
        }
        if (cudaEventRecord(ss->join, ss->s) != cudaSuccess ||
            cudaStreamWaitEvent(c.s, ss->join, 0) != cudaSuccess)
            return LCE_ERR_CUDA;
        prof_end(pi, c.s);
        g_launches += launched;
        return LCE_OK;
    }
    const int grid = cl * (p.total_tiles < units ? p.total_tiles : units);
    LCE_LAUNCH_KIND(kind, c.s, launch_gemm(MODE_BWD, cl, p, grid, c.s));
    return LCE_OK;
}

// A chunk's gradient launches on the loss path: dH straight into the caller's
// rows when there is one vocabulary part and nothing to accumulate, else through
// the fp32 partial arrays and the combining kernel (which adds into the caller's
// dH when accumulating).
lce_status run_grad(const Ctx &c, long long row0, long long rows, int slot, void *dHc,
                    bool acc_dh, float *dW, bool acc_dw, const float *dloss, const GradSpec &g) {
    if (g.dw_only) return run_bwd(c, row0, rows, slot, DhOut{dHc, false, 1, 0}, dW, acc_dw, dloss, g);
    const int want = dh_parts(c, rows, g.dh_alone);
    if (want <= 1 && !acc_dh)
        return run_bwd(c, row0, rows, slot, DhOut{dHc, false, 1, 0}, dW, acc_dw, dloss, g);
    float *dHp = reinterpret_cast<float *>(c.ws + c.L.off_dHp);
    int parts = 1;
    LCE_TRY(run_bwd(c, row0, rows, slot, DhOut{dHp, true, want, c.L.ldp}, dW, acc_dw, dloss, g,
                    &parts));
    LCE_LAUNCH(launch_combine_dh(dHp, parts, c.L.ldp * c.D, dHc, rows * c.D, c.f16, acc_dh,
                                 c.sms, c.s));
    return LCE_OK;
}

lce_status run_merge(const Ctx &c, long long row0, long long rows, float *lse,
                     const float *dloss, float *loss_rows) {
    MergeParams m;
    m.parts = c.parts;
    m.nparts = c.L.nparts;
    m.zy = c.zy;
    m.G = c.Gb[0];
    m.ldg = c.L.ldg;
    m.rows = static_cast<int>(rows);
    m.row0 = static_cast<int>(row0);
    m.V = static_cast<int>(c.V);
    m.ignore_index = c.ign;
    m.y = c.y;
    m.hdr = c.hdr;
    m.dloss = dloss;
    m.dloss_per_row = c.reduction == LCE_REDUCTION_NONE ? 1 : 0;
    m.mean = c.reduction == LCE_REDUCTION_MEAN ? 1 : 0;
    m.f16 = c.f16 ? 1 : 0;
    m.lse = lse;
    m.loss_rows = loss_rows;
    LCE_LAUNCH_KIND(LCE_KERNEL_MERGE, c.s, launch_merge(m, c.s));
    return LCE_OK;
}

// Fused path, between a chunk's logits GEMM and its gradient GEMMs, one launch:
// lse and the row losses, P' -> G in place in chunk buffer G, and (transpose) the
// H chunk^T the dW tiles read, into columns ht_col0 .. of H^T.
lce_status run_prep(const Ctx &c, long long row0, long long rows, float *lse,
                    const float *dloss, float *loss_rows, __nv_bfloat16 *G, bool transpose,
                    long long ht_col0 = 0) {
    PrepParams pp;
    memset(&pp, 0, sizeof(pp));
    MergeParams &m = pp.m;
    m.parts = c.parts;
    m.nparts = c.L.nparts;
    m.zy = c.zy;
    m.G = G;
    m.ldg = c.L.ldg;
    m.rows = static_cast<int>(rows);
    m.row0 = static_cast<int>(row0);
    m.V = static_cast<int>(c.V);
    m.ignore_index = c.ign;
    m.y = c.y;
    m.hdr = c.hdr;
    m.dloss = dloss;
    m.dloss_per_row = c.reduction == LCE_REDUCTION_NONE ? 1 : 0;
    m.mean = c.reduction == LCE_REDUCTION_MEAN ? 1 : 0;
    m.f16 = c.f16 ? 1 : 0;
    m.lse = lse;
    m.loss_rows = loss_rows;
    pp.ldg = c.L.ldg;
    pp.segs = static_cast<int>(cdiv(cdiv(c.V, 8), PREP_VEC_PER_CTA));
    if (transpose) {
        pp.tp.src = c.H + h_row(c, row0) * c.D;
        pp.tp.ld_src = static_cast<int>(c.D);
        pp.tp.dst_t = c.HT + ht_col0;
        pp.tp.ld_t = c.L.ldt;
        pp.tp.rows = static_cast<int>(rows);
        pp.tp.cols = static_cast<int>(c.D);
        pp.tt_x = static_cast<int>(cdiv(c.D, 64));
    }
    LCE_LAUNCH_KIND(LCE_KERNEL_MERGE, c.s, launch_prep(pp, c.s));
    return LCE_OK;
}

// Rows of chunk k (the last chunk may be shorter).
inline long long chunk_rows(const Ctx &c, long long k) {
    const long long row0 = k * c.L.C;
    return (c.N - row0) < c.L.C ? (c.N - row0) : c.L.C;
}

// Whether chunks are taken in pairs with one dW contraction per pair: CTA pairs,
// a dW contraction, two chunk buffers (so more than one chunk), H in place.
inline bool paired(const Ctx &c, bool h_chunked_ok = false) {
    return c.pairs > 0 && !c.L.frozen_w && c.L.nbuf == 2 && (h_chunked_ok || !c.h_chunked);
}

// W frozen with two chunk buffers: chunk k+1's logits tiles run on the CTA pairs
// chunk k's dH tiles leave free (chunk k in buffer k % 2).
inline bool frozen_overlapped(const Ctx &c) {
    return c.pairs > 0 && c.L.frozen_w && c.L.nbuf == 2 && !c.h_chunked;
}

}  // namespace

extern "C" {

lce_status lce_workspace_size(int64_t N, int64_t D, int64_t V, int64_t chunk, size_t *bytes) {
    if (!bytes) return LCE_ERR_INVALID_ARG;
    Layout L;
    if (!make_layout(N, D, V, chunk, L)) return LCE_ERR_INVALID_ARG;
    *bytes = L.total;
    return LCE_OK;
}

lce_status lce_forward_workspace_size(int64_t N, int64_t D, int64_t V, int64_t chunk,
                                      size_t *bytes) {
    if (!bytes) return LCE_ERR_INVALID_ARG;
    Layout L;
    if (!make_layout(N, D, V, chunk, L)) return LCE_ERR_INVALID_ARG;
    *bytes = L.fwd_total;
    return LCE_OK;
}

lce_status lce_count_valid(const int64_t *y, int64_t N, int64_t V, int64_t ignore_index,
                           int64_t *n_valid, lce_stream_t stream) {
    g_launches = 0;
    if (N < 0 || V <= 0 || !n_valid || (N > 0 && !y)) return LCE_ERR_INVALID_ARG;
    if ((y && !aligned16(y)) || (reinterpret_cast<uintptr_t>(n_valid) & 7u))
        return LCE_ERR_ALIGNMENT;
    int sms = 0, pairs = 0;
    lce_status st = init_device(&sms, &pairs);
    if (st != LCE_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    LCE_LAUNCH_KIND(LCE_KERNEL_OTHER, s,
                    launch_count_valid(reinterpret_cast<const long long *>(y), N, V, ignore_index,
                                       reinterpret_cast<long long *>(n_valid), s));
    return LCE_OK;
}

lce_status lce_workspace_size_opt(int64_t N, int64_t D, int64_t V, int64_t chunk, int flags,
                                  size_t *bytes) {
    if (!bytes || (flags & ~LCE_FLAGS_ALL)) return LCE_ERR_INVALID_ARG;
    Layout L;
    if (!make_layout(N, D, V, chunk, L, (flags & LCE_FROZEN_W) != 0, (flags & LCE_LOW_MEMORY) != 0))
        return LCE_ERR_INVALID_ARG;
    *bytes = L.total + ((flags & LCE_ACCUMULATE_DH) ? acc_dh_bytes(L, D) : 0);
    return LCE_OK;
}

lce_status lce_forward_opt(const void *H, const void *W, const int64_t *y, int64_t N, int64_t D,
                           int64_t V, int64_t ignore_index, int64_t chunk, int reduction, int flags,
                           float *loss, float *lse, void *ws, size_t ws_bytes,
                           lce_stream_t stream) {
    g_launches = 0;
    if (reduction < LCE_REDUCTION_MEAN || reduction > LCE_REDUCTION_NONE) return LCE_ERR_INVALID_ARG;
    // nothing to accumulate here, and no chunk buffer to keep small
    if (flags & ~(LCE_INPUT_FP16 | LCE_LOW_MEMORY)) return LCE_ERR_INVALID_ARG;
    const bool none = reduction == LCE_REDUCTION_NONE;
    if ((!none && !loss) || (N > 0 && (!lse || !loss))) return LCE_ERR_INVALID_ARG;
    if ((loss && !aligned16(loss)) || (lse && !aligned16(lse))) return LCE_ERR_ALIGNMENT;
    Ctx c;
    LCE_TRY(setup(c, H, W, y, N, D, V, ignore_index, chunk, ws, ws_bytes, stream, false,
                  (flags & LCE_INPUT_FP16) != 0, false, true));
    c.reduction = reduction;
    float *rows_out = none ? loss : c.loss_rows;
    for (long long k = 0; k < c.L.nchunks; ++k) {
        const long long row0 = k * c.L.C;
        const long long rows = (c.N - row0) < c.L.C ? (c.N - row0) : c.L.C;
        LCE_TRY(run_logits(c, MODE_LSE, row0, rows, static_cast<int>(k), nullptr, nullptr,
                           c.Gb[0]));
        LCE_TRY(run_merge(c, row0, rows, lse, nullptr, rows_out));
    }
    if (!none)
        LCE_LAUNCH(launch_loss_finalize(c.loss_rows, c.N, c.hdr, loss,
                                        reduction == LCE_REDUCTION_MEAN, c.s));
    return LCE_OK;
}

lce_status lce_forward_ex(const void *H, const void *W, const int64_t *y, int64_t N, int64_t D,
                          int64_t V, int64_t ignore_index, int64_t chunk, int reduction,
                          float *loss, float *lse, void *ws, size_t ws_bytes,
                          lce_stream_t stream) {
    return lce_forward_opt(H, W, y, N, D, V, ignore_index, chunk, reduction, 0, loss, lse, ws,
                           ws_bytes, stream);
}

lce_status lce_forward(const void *H, const void *W, const int64_t *y, int64_t N, int64_t D,
                       int64_t V, int64_t ignore_index, int64_t chunk, float *loss, float *lse,
                       void *ws, size_t ws_bytes, lce_stream_t stream) {
    return lce_forward_ex(H, W, y, N, D, V, ignore_index, chunk, LCE_REDUCTION_MEAN, loss, lse, ws,
                          ws_bytes, stream);
}

lce_status lce_backward_opt(const void *H, const void *W, const int64_t *y, const float *lse,
                            const float *dloss, void *dH, float *dW, int64_t N, int64_t D,
                            int64_t V, int64_t ignore_index, int64_t chunk, int reduction,
                            int flags, void *ws, size_t ws_bytes, lce_stream_t stream) {
    g_launches = 0;
    if (reduction < LCE_REDUCTION_MEAN || reduction > LCE_REDUCTION_NONE) return LCE_ERR_INVALID_ARG;
    if (flags & ~LCE_FLAGS_ALL) return LCE_ERR_INVALID_ARG;
    const bool f16 = (flags & LCE_INPUT_FP16) != 0;
    const bool frozen = (flags & LCE_FROZEN_W) != 0;
    if (frozen && (flags & LCE_ACCUMULATE_DW)) return LCE_ERR_INVALID_ARG;
    if (f16 && reduction == LCE_REDUCTION_NONE) return LCE_ERR_UNSUPPORTED;
    if ((!frozen && !dW) || (N > 0 && (!lse || !dH))) return LCE_ERR_INVALID_ARG;
    if ((dW && !aligned16(dW)) || (dH && !aligned16(dH)) || (lse && !aligned16(lse)))
        return LCE_ERR_ALIGNMENT;
    const bool acc_dh = (flags & LCE_ACCUMULATE_DH) != 0;
    const bool low_mem = (flags & LCE_LOW_MEMORY) != 0;
    Layout L0;
    if (!make_layout(N, D, V, chunk, L0, frozen, low_mem)) return LCE_ERR_INVALID_ARG;
    if (acc_dh && ws_bytes < L0.total + acc_dh_bytes(L0, D)) return LCE_ERR_WORKSPACE;
    Ctx c;
    LCE_TRY(setup(c, H, W, y, N, D, V, ignore_index, chunk, ws, ws_bytes, stream, false, f16,
                  frozen, false, low_mem));
    c.reduction = reduction;
    if (frozen) dW = nullptr;
    if (c.L.nchunks == 0 && dW && !(flags & LCE_ACCUMULATE_DW)) {
        if (cudaMemsetAsync(dW, 0, sizeof(float) * static_cast<size_t>(V) * D, c.s) != cudaSuccess)
            return LCE_ERR_CUDA;
    }
    const bool acc_dw0 = (flags & LCE_ACCUMULATE_DW) != 0;
    __nv_bfloat16 *dHb = static_cast<__nv_bfloat16 *>(dH);
    if (frozen_overlapped(c)) {
        LCE_TRY(run_logits(c, MODE_G, 0, chunk_rows(c, 0), 0, lse, dloss, c.Gb[0]));
        for (long long k = 0; k < c.L.nchunks; ++k) {
            const long long r0 = k * c.L.C, n0 = chunk_rows(c, k);
            GradSpec g{c.Gb[k & 1], c.Gb[k & 1], 0, true, true};
            LogitsSpec next{};
            if (k + 1 < c.L.nchunks) {
                next = LogitsSpec{MODE_G, r0 + c.L.C, chunk_rows(c, k + 1),
                                  static_cast<int>(2 * k + 2), lse, dloss, c.Gb[(k + 1) & 1]};
                g.beside = &next;
            }
            LCE_TRY(run_grad(c, r0, n0, static_cast<int>(2 * k + 1), dHb + r0 * c.D, acc_dh, dW,
                             false, dloss, g));
        }
        return LCE_OK;
    }
    if (paired(c)) {
        // chunks in pairs (a, b): a's G (G epilogue) into buffer 0, its H^T into
        // columns 0..C-1; a's dH tiles, with b's logits (G into buffer 1) on the pairs
        // they leave free; b's H^T into columns C.., then b's dH beside one dW
        // contraction over both chunks (K = C + rows_b). An odd last chunk runs by itself.
        for (long long a = 0; a < c.L.nchunks; a += 2) {
            const long long ra = a * c.L.C, na = chunk_rows(c, a);
            const bool has_b = a + 1 < c.L.nchunks;
            const bool acc = a > 0 || acc_dw0;
            LCE_TRY(run_logits(c, MODE_G, ra, na, static_cast<int>(2 * a), lse, dloss, c.Gb[0]));
            LCE_TRY(run_transpose(c, ra, na, 0));
            if (!has_b) {
                LCE_TRY(run_grad(c, ra, na, static_cast<int>(2 * a + 1), dHb + ra * c.D, acc_dh, dW,
                                 acc, dloss, GradSpec{c.Gb[0], c.Gb[0], na, true, false}));
                break;
            }
            const long long b = a + 1, rb = b * c.L.C, nb = chunk_rows(c, b);
            // a's dH tiles, with b's logits tiles on the pairs they leave free
            const LogitsSpec lb{MODE_G, rb, nb, static_cast<int>(2 * b), lse, dloss, c.Gb[1]};
            GradSpec ga{c.Gb[0], c.Gb[0], 0, true, true};
            ga.beside = &lb;
            LCE_TRY(run_grad(c, ra, na, static_cast<int>(2 * a + 1), dHb + ra * c.D, acc_dh, dW,
                             acc, dloss, ga));
            LCE_TRY(run_transpose(c, rb, nb, c.L.C));
            LCE_TRY(run_grad(c, rb, nb, static_cast<int>(2 * b + 1), dHb + rb * c.D, acc_dh, dW,
                             acc, dloss, GradSpec{c.Gb[1], c.Gb[0], c.L.C + nb, true, false}));
        }
        return LCE_OK;
    }
    for (long long k = 0; k < c.L.nchunks; ++k) {
        const long long row0 = k * c.L.C;
        const long long rows = chunk_rows(c, k);
        LCE_TRY(run_logits(c, MODE_G, row0, rows, static_cast<int>(2 * k), lse, dloss, c.Gb[0]));
        LCE_TRY(run_grad(c, row0, rows, static_cast<int>(2 * k + 1), dHb + row0 * c.D, acc_dh, dW,
                         k > 0 || acc_dw0, dloss, GradSpec{c.Gb[0], c.Gb[0], rows, false, false}));
    }
    return LCE_OK;
}

lce_status lce_backward_ex(const void *H, const void *W, const int64_t *y, const float *lse,
                           const float *dloss, void *dH, float *dW, int64_t N, int64_t D,
                           int64_t V, int64_t ignore_index, int64_t chunk, int reduction,
                           void *ws, size_t ws_bytes, lce_stream_t stream) {
    return lce_backward_opt(H, W, y, lse, dloss, dH, dW, N, D, V, ignore_index, chunk, reduction, 0,
                            ws, ws_bytes, stream);
}

lce_status lce_backward(const void *H, const void *W, const int64_t *y, const float *lse,
                        const float *dloss, void *dH, float *dW, int64_t N, int64_t D, int64_t V,
                        int64_t ignore_index, int64_t chunk, void *ws, size_t ws_bytes,
                        lce_stream_t stream) {
    return lce_backward_ex(H, W, y, lse, dloss, dH, dW, N, D, V, ignore_index, chunk,
                           LCE_REDUCTION_MEAN, ws, ws_bytes, stream);
}

}  // extern "C"

namespace {

// The fused call; n_valid_total (device int64, or null) replaces this call's own
// count of valid rows as the normaliser of the mean.
lce_status fwd_bwd_impl(const void *H, const void *W, const int64_t *y, const float *dloss,
                        int64_t N, int64_t D, int64_t V, int64_t ignore_index, int64_t chunk,
                        int reduction, int flags, float *loss, float *lse, void *dH, float *dW,
                        void *ws, size_t ws_bytes, lce_stream_t stream,
                        const int64_t *n_valid_total) {
    g_launches = 0;
    if (reduction < LCE_REDUCTION_MEAN || reduction > LCE_REDUCTION_NONE) return LCE_ERR_INVALID_ARG;
    if (flags & ~LCE_FLAGS_ALL) return LCE_ERR_INVALID_ARG;
    const bool f16 = (flags & LCE_INPUT_FP16) != 0;
    const bool frozen = (flags & LCE_FROZEN_W) != 0;
    const bool none = reduction == LCE_REDUCTION_NONE;
    if (frozen && (flags & LCE_ACCUMULATE_DW)) return LCE_ERR_INVALID_ARG;
    if (f16 && none) return LCE_ERR_UNSUPPORTED;
    if ((!none && !loss) || (!frozen && !dW) || (N > 0 && (!lse || !dH || !loss)))
        return LCE_ERR_INVALID_ARG;
    if ((loss && !aligned16(loss)) || (dW && !aligned16(dW)) || (dH && !aligned16(dH)) ||
        (lse && !aligned16(lse)))
        return LCE_ERR_ALIGNMENT;
    const bool acc_dh = (flags & LCE_ACCUMULATE_DH) != 0;
    const bool low_mem = (flags & LCE_LOW_MEMORY) != 0;
    Layout L0;
    if (!make_layout(N, D, V, chunk, L0, frozen, low_mem)) return LCE_ERR_INVALID_ARG;
    if (acc_dh && ws_bytes < L0.total + acc_dh_bytes(L0, D)) return LCE_ERR_WORKSPACE;
    Ctx c;
    LCE_TRY(setup(c, H, W, y, N, D, V, ignore_index, chunk, ws, ws_bytes, stream, false, f16,
                  frozen, false, low_mem));
    c.reduction = reduction;
    if (n_valid_total) LCE_LAUNCH(launch_set_nvalid(reinterpret_cast<const long long *>(n_valid_total),
                                                    c.hdr, c.s));
    if (frozen) dW = nullptr;
    float *rows_out = none ? loss : c.loss_rows;
    if (c.L.nchunks == 0 && dW && !(flags & LCE_ACCUMULATE_DW)) {
        if (cudaMemsetAsync(dW, 0, sizeof(float) * static_cast<size_t>(V) * D, c.s) != cudaSuccess)
            return LCE_ERR_CUDA;
    }
    const bool acc_dw0 = (flags & LCE_ACCUMULATE_DW) != 0;
    __nv_bfloat16 *dHb = static_cast<__nv_bfloat16 *>(dH);
    if (frozen_overlapped(c)) {
        // chunk k's dH tiles, with chunk k+1's logits (P' into buffer (k+1) % 2) on
        // the pairs they leave free; then chunk k+1's prep (no H^T: no dW)
        LCE_TRY(run_logits(c, MODE_LSE_P, 0, chunk_rows(c, 0), 0, nullptr, nullptr, c.Gb[0]));
        LCE_TRY(run_prep(c, 0, chunk_rows(c, 0), lse, dloss, rows_out, c.Gb[0], false));
        for (long long k = 0; k < c.L.nchunks; ++k) {
            const long long r0 = k * c.L.C, n0 = chunk_rows(c, k);
            GradSpec g{c.Gb[k & 1], c.Gb[k & 1], 0, true, true};
            LogitsSpec next{};
            if (k + 1 < c.L.nchunks) {
                next = LogitsSpec{MODE_LSE_P, r0 + c.L.C, chunk_rows(c, k + 1),
                                  static_cast<int>(2 * k + 2), nullptr, nullptr, c.Gb[(k + 1) & 1]};
                g.beside = &next;
            }
            LCE_TRY(run_grad(c, r0, n0, static_cast<int>(2 * k + 1), dHb + r0 * c.D, acc_dh, dW,
                             false, dloss, g));
            if (k + 1 < c.L.nchunks)
                LCE_TRY(run_prep(c, r0 + c.L.C, chunk_rows(c, k + 1), lse, dloss, rows_out,
                                 c.Gb[(k + 1) & 1], false));
        }
    } else if (paired(c)) {
        // chunks in pairs (a, b): a's P' into buffer 0, its prep (lse, row losses,
        // P' -> G, H^T into columns 0..C-1); a's dH tiles, with b's logits (P' into
        // buffer 1) on the pairs they leave free; b's prep (H^T into columns C..), then
        // b's dH beside one dW contraction over both chunks (K = C + rows_b). An odd
        // last chunk runs by itself.
        for (long long a = 0; a < c.L.nchunks; a += 2) {
            const long long ra = a * c.L.C, na = chunk_rows(c, a);
            const bool has_b = a + 1 < c.L.nchunks;
            const bool acc = a > 0 || acc_dw0;
            LCE_TRY(run_logits(c, MODE_LSE_P, ra, na, static_cast<int>(2 * a), nullptr, nullptr,
                               c.Gb[0]));
            LCE_TRY(run_prep(c, ra, na, lse, dloss, rows_out, c.Gb[0], true, 0));
            if (!has_b) {
                LCE_TRY(run_grad(c, ra, na, static_cast<int>(2 * a + 1), dHb + ra * c.D, acc_dh, dW,
                                 acc, dloss, GradSpec{c.Gb[0], c.Gb[0], na, true, false}));
                break;
            }
            const long long b = a + 1, rb = b * c.L.C, nb = chunk_rows(c, b);
            // a's dH tiles, with b's logits tiles on the pairs they leave free
            const LogitsSpec lb{MODE_LSE_P, rb, nb, static_cast<int>(2 * b), nullptr, nullptr,
                                c.Gb[1]};
            GradSpec ga{c.Gb[0], c.Gb[0], 0, true, true};
            ga.beside = &lb;
            LCE_TRY(run_grad(c, ra, na, static_cast<int>(2 * a + 1), dHb + ra * c.D, acc_dh, dW,
                             acc, dloss, ga));
            LCE_TRY(run_prep(c, rb, nb, lse, dloss, rows_out, c.Gb[1], true, c.L.C));
            LCE_TRY(run_grad(c, rb, nb, static_cast<int>(2 * b + 1), dHb + rb * c.D, acc_dh, dW,
                             acc, dloss, GradSpec{c.Gb[1], c.Gb[0], c.L.C + nb, true, false}));
        }
    } else {
        for (long long k = 0; k < c.L.nchunks; ++k) {
            const long long row0 = k * c.L.C;
            const long long rows = chunk_rows(c, k);
            LCE_TRY(run_logits(c, MODE_LSE_P, row0, rows, static_cast<int>(2 * k), nullptr, nullptr,
                               c.Gb[0]));
            LCE_TRY(run_prep(c, row0, rows, lse, dloss, rows_out, c.Gb[0], !frozen));
            LCE_TRY(run_grad(c, row0, rows, static_cast<int>(2 * k + 1), dHb + row0 * c.D, acc_dh,
                             dW, k > 0 || acc_dw0, dloss,
                             GradSpec{c.Gb[0], c.Gb[0], frozen ? 0 : rows, true, false}));
        }
    }
    if (!none)
        LCE_LAUNCH(launch_loss_finalize(c.loss_rows, c.N, c.hdr, loss,
                                        reduction == LCE_REDUCTION_MEAN, c.s));
    return LCE_OK;
}

}  // namespace

extern "C" {

lce_status lce_fwd_bwd_opt(const void *H, const void *W, const int64_t *y, const float *dloss,
                           int64_t N, int64_t D, int64_t V, int64_t ignore_index, int64_t chunk,
                           int reduction, int flags, float *loss, float *lse, void *dH, float *dW,
                           void *ws, size_t ws_bytes, lce_stream_t stream) {
    return fwd_bwd_impl(H, W, y, dloss, N, D, V, ignore_index, chunk, reduction, flags, loss, lse,
                        dH, dW, ws, ws_bytes, stream, nullptr);
}

lce_status lce_fwd_bwd_sharded(const void *H, const void *W, const int64_t *y, const float *dloss,
                               const int64_t *n_valid_total, int64_t N, int64_t D, int64_t V,
                               int64_t ignore_index, int64_t chunk, int flags, float *loss,
                               float *lse, void *dH, float *dW, void *ws, size_t ws_bytes,
                               lce_stream_t stream) {
    g_launches = 0;
    if (!n_valid_total) return LCE_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(n_valid_total) & 7u) return LCE_ERR_ALIGNMENT;
    return fwd_bwd_impl(H, W, y, dloss, N, D, V, ignore_index, chunk, LCE_REDUCTION_MEAN, flags,
                        loss, lse, dH, dW, ws, ws_bytes, stream, n_valid_total);
}

lce_status lce_fwd_bwd_ex(const void *H, const void *W, const int64_t *y, const float *dloss,
                          int64_t N, int64_t D, int64_t V, int64_t ignore_index, int64_t chunk,
                          int reduction, float *loss, float *lse, void *dH, float *dW, void *ws,
                          size_t ws_bytes, lce_stream_t stream) {
    return lce_fwd_bwd_opt(H, W, y, dloss, N, D, V, ignore_index, chunk, reduction, 0, loss, lse,
                           dH, dW, ws, ws_bytes, stream);
}

lce_status lce_fwd_bwd(const void *H, const void *W, const int64_t *y, const float *dloss,
                       int64_t N, int64_t D, int64_t V, int64_t ignore_index, int64_t chunk,
                       float *loss, float *lse, void *dH, float *dW, void *ws, size_t ws_bytes,
                       lce_stream_t stream) {
    return lce_fwd_bwd_ex(H, W, y, dloss, N, D, V, ignore_index, chunk, LCE_REDUCTION_MEAN, loss,
                          lse, dH, dW, ws, ws_bytes, stream);
}

lce_status lce_rmsnorm_forward(const void *X, const void *gamma, int64_t N, int64_t D, float eps,
                               void *H, float *rstd, lce_stream_t stream) {
    g_launches = 0;
    if (N < 0 || D <= 0 || D % 8 != 0 || D > NRM_MAX_D || !(eps >= 0.f)) return LCE_ERR_INVALID_ARG;
    if (N > 0 && (!X || !gamma || !H)) return LCE_ERR_INVALID_ARG;
    if ((X && !aligned16(X)) || (gamma && !aligned16(gamma)) || (H && !aligned16(H)))
        return LCE_ERR_ALIGNMENT;
    int sms = 0, pairs = 0;
    lce_status st = init_device(&sms, &pairs);
    if (st != LCE_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    NormParams p;
    memset(&p, 0, sizeof(p));
    p.X = static_cast<const __nv_bfloat16 *>(X);
    p.gamma = static_cast<const __nv_bfloat16 *>(gamma);
    p.H = static_cast<__nv_bfloat16 *>(H);
    p.rstd = rstd;
    p.rows = N;
    p.D = static_cast<int>(D);
    p.eps = eps;
    LCE_LAUNCH_KIND(LCE_KERNEL_NORM, s, launch_rmsnorm_fwd(p, s));
    return LCE_OK;
}

lce_status lce_rmsnorm_backward_workspace_size(int64_t D, size_t *bytes) {
    if (!bytes || D <= 0 || D % 8 != 0 || D > NRM_MAX_D) return LCE_ERR_INVALID_ARG;
    *bytes = align_up(4 * static_cast<size_t>(NRM_GRID) * static_cast<size_t>(D), 1024);
    return LCE_OK;
}

lce_status lce_rmsnorm_backward(const void *X, const void *gamma, const void *dH, int dh_fp32,
                                int64_t N, int64_t D, float eps, void *dX, float *dgamma, void *ws,
                                size_t ws_bytes, lce_stream_t stream) {
    g_launches = 0;
    size_t need = 0;
    if (lce_rmsnorm_backward_workspace_size(D, &need) != LCE_OK || N < 0 || !(eps >= 0.f))
        return LCE_ERR_INVALID_ARG;
    if (!gamma || !dgamma || !ws || (N > 0 && (!X || !dH || !dX))) return LCE_ERR_INVALID_ARG;
    if ((X && !aligned16(X)) || !aligned16(gamma) || (dH && !aligned16(dH)) ||
        (dX && !aligned16(dX)) || !aligned16(ws))
        return LCE_ERR_ALIGNMENT;
    if (ws_bytes < need) return LCE_ERR_WORKSPACE;
    int sms = 0, pairs = 0;
    lce_status st = init_device(&sms, &pairs);
    if (st != LCE_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    NormParams p;
    memset(&p, 0, sizeof(p));
    p.X = static_cast<const __nv_bfloat16 *>(X);
    p.gamma = static_cast<const __nv_bfloat16 *>(gamma);
    p.dH = dH;
    p.dh_fp32 = dh_fp32 ? 1 : 0;
    p.dX = static_cast<__nv_bfloat16 *>(dX);
    p.part = static_cast<float *>(ws);
    p.first = 1;
    p.rows = N;
    p.D = static_cast<int>(D);
    p.eps = eps;
    LCE_LAUNCH_KIND(LCE_KERNEL_NORM, s, launch_rmsnorm_bwd(p, s));
    LCE_LAUNCH_KIND(LCE_KERNEL_NORM, s, launch_dgamma_reduce(p.part, p.D, dgamma, s));
    return LCE_OK;
}

lce_status lce_norm_workspace_size_opt(int64_t N, int64_t D, int64_t V, int64_t chunk, int flags,
                                       size_t *bytes) {
    if (!bytes || (flags & ~(LCE_FROZEN_W | LCE_LOW_MEMORY))) return LCE_ERR_INVALID_ARG;
    NormLayout NL;
    if (!make_norm_layout(N, D, V, chunk, NL, (flags & LCE_FROZEN_W) != 0,
                          (flags & LCE_LOW_MEMORY) != 0))
        return LCE_ERR_INVALID_ARG;
    *bytes = NL.total;
    return LCE_OK;
}

lce_status lce_norm_workspace_size(int64_t N, int64_t D, int64_t V, int64_t chunk, size_t *bytes) {
    return lce_norm_workspace_size_opt(N, D, V, chunk, 0, bytes);
}

lce_status lce_norm_fwd_bwd_opt(const void *X, const void *gamma, float eps, const void *W,
                                const int64_t *y, const float *dloss, int64_t N, int64_t D,
                                int64_t V, int64_t ignore_index, int64_t chunk, int reduction,
                                int flags, float *loss, float *lse, void *dX, float *dgamma,
                                float *dW, void *ws, size_t ws_bytes, lce_stream_t stream) {
    g_launches = 0;
    if (reduction < LCE_REDUCTION_MEAN || reduction > LCE_REDUCTION_NONE) return LCE_ERR_INVALID_ARG;
    if (flags & ~(LCE_FROZEN_W | LCE_LOW_MEMORY)) return LCE_ERR_INVALID_ARG;
    const bool frozen = (flags & LCE_FROZEN_W) != 0;
    const bool low_mem = (flags & LCE_LOW_MEMORY) != 0;
    const bool none = reduction == LCE_REDUCTION_NONE;
    NormLayout NL;
    if (!make_norm_layout(N, D, V, chunk, NL, frozen, low_mem) || !(eps >= 0.f))
        return LCE_ERR_INVALID_ARG;
    if (!gamma || !dgamma || (!frozen && !dW) || (!none && !loss) ||
        (N > 0 && (!X || !lse || !dX || !loss)))
        return LCE_ERR_INVALID_ARG;
    if ((X && !aligned16(X)) || !aligned16(gamma) || (dW && !aligned16(dW)) ||
        (dX && !aligned16(dX)) || (loss && !aligned16(loss)) || (lse && !aligned16(lse)))
        return LCE_ERR_ALIGNMENT;
    if (frozen) dW = nullptr;
    if (!ws) return LCE_ERR_INVALID_ARG;
    if (ws_bytes < NL.total) return LCE_ERR_WORKSPACE;
    uint8_t *w = static_cast<uint8_t *>(ws);
    __nv_bfloat16 *Hbuf = reinterpret_cast<__nv_bfloat16 *>(w + NL.off_H);
    float *dHbuf = reinterpret_cast<float *>(w + NL.off_dH);
    float *part = reinterpret_cast<float *>(w + NL.off_part);
    Ctx c;
    LCE_TRY(setup(c, Hbuf, W, y, N, D, V, ignore_index, chunk, ws, ws_bytes, stream, true, false,
                  frozen, false, low_mem || frozen));
    c.reduction = reduction;
    float *rows_out = none ? loss : c.loss_rows;
    if (c.L.nchunks == 0) {
        if ((dW && cudaMemsetAsync(dW, 0, sizeof(float) * static_cast<size_t>(V) * D, c.s) !=
                       cudaSuccess) ||
            cudaMemsetAsync(dgamma, 0, sizeof(float) * static_cast<size_t>(D), c.s) != cudaSuccess)
            return LCE_ERR_CUDA;
    }
    const __nv_bfloat16 *Xb = static_cast<const __nv_bfloat16 *>(X);
    __nv_bfloat16 *dXb = static_cast<__nv_bfloat16 *>(dX);
    const __nv_bfloat16 *gam = static_cast<const __nv_bfloat16 *>(gamma);
    // RMSNorm forward of rows [row0, row0 + rows) into their place in the H buffer
    auto norm_fwd = [&](long long row0, long long rows) -> lce_status {
        NormParams np;
        memset(&np, 0, sizeof(np));
        np.X = Xb + row0 * c.D;
        np.gamma = gam;
        np.H = Hbuf + h_row(c, row0) * c.D;
        np.rows = rows;
        np.D = static_cast<int>(c.D);
        np.eps = eps;
        LCE_LAUNCH_KIND(LCE_KERNEL_NORM, c.s, launch_rmsnorm_fwd(np, c.s));
        return LCE_OK;
    };
    // RMSNorm backward of a chunk from its fp32 dH (the sum of `parts` arrays)
    auto norm_bwd = [&](long long row0, long long rows, int parts) -> lce_status {
        NormParams np;
        memset(&np, 0, sizeof(np));
        np.X = Xb + row0 * c.D;
        np.gamma = gam;
        np.rows = rows;
        np.D = static_cast<int>(c.D);
        np.eps = eps;
        np.dH = dHbuf;
        np.dh_fp32 = 1;
        np.dh_splits = parts;
        np.dh_split_stride = c.L.ldp * c.D;
        np.dX = dXb + row0 * c.D;
        np.part = part;
        np.first = row0 == 0 ? 1 : 0;
        LCE_LAUNCH_KIND(LCE_KERNEL_NORM, c.s, launch_rmsnorm_bwd(np, c.s));
        return LCE_OK;
    };
    if (paired(c, true)) {
        // chunks in pairs (a, b), as on the loss path: the normalised rows of both
        // in the H buffer; a's logits, prep, a's dH tiles (fp32, in parts) with b's
        // logits beside them, a's RMSNorm backward; b's prep, b's dH beside one dW
        // contraction over both chunks, b's RMSNorm backward
        for (long long a = 0; a < c.L.nchunks; a += 2) {
            const long long ra = a * c.L.C, na = chunk_rows(c, a);
            const bool has_b = a + 1 < c.L.nchunks;
            const long long b = a + 1, rb = b * c.L.C, nb = has_b ? chunk_rows(c, b) : 0;
            LCE_TRY(norm_fwd(ra, na + nb));
            LCE_TRY(run_logits(c, MODE_LSE_P, ra, na, static_cast<int>(2 * a), nullptr, nullptr,
                               c.Gb[0]));
            LCE_TRY(run_prep(c, ra, na, lse, dloss, rows_out, c.Gb[0], true, 0));
            int parts = 1;
            if (!has_b) {
                LCE_TRY(run_bwd(c, ra, na, static_cast<int>(2 * a + 1),
                                DhOut{dHbuf, true, dh_parts(c, na, false), c.L.ldp}, dW, a > 0,
                                dloss, GradSpec{c.Gb[0], c.Gb[0], na, true, false}, &parts));
                LCE_TRY(norm_bwd(ra, na, parts));
                break;
            }
            const LogitsSpec lb{MODE_LSE_P, rb, nb, static_cast<int>(2 * b), nullptr, nullptr,
                                c.Gb[1]};
            GradSpec ga{c.Gb[0], c.Gb[0], 0, true, true};
            ga.beside = &lb;
            LCE_TRY(run_bwd(c, ra, na, static_cast<int>(2 * a + 1),
                            DhOut{dHbuf, true, dh_parts(c, na, true), c.L.ldp}, dW, false, dloss,
                            ga, &parts));
            LCE_TRY(norm_bwd(ra, na, parts));
            LCE_TRY(run_prep(c, rb, nb, lse, dloss, rows_out, c.Gb[1], true, c.L.C));
            LCE_TRY(run_bwd(c, rb, nb, static_cast<int>(2 * b + 1),
                            DhOut{dHbuf, true, dh_parts(c, nb, false), c.L.ldp}, dW, a > 0, dloss,
                            GradSpec{c.Gb[1], c.Gb[0], c.L.C + nb, true, false}, &parts));
            LCE_TRY(norm_bwd(rb, nb, parts));
        }
    } else {
        for (long long k = 0; k < c.L.nchunks; ++k) {
            const long long row0 = k * c.L.C;
            const long long rows = chunk_rows(c, k);
            LCE_TRY(norm_fwd(row0, rows));
            LCE_TRY(run_logits(c, MODE_LSE_P, row0, rows, static_cast<int>(2 * k), nullptr, nullptr,
                               c.Gb[0]));
            LCE_TRY(run_prep(c, row0, rows, lse, dloss, rows_out, c.Gb[0], !frozen));
            int parts = 1;
            LCE_TRY(run_bwd(c, row0, rows, static_cast<int>(2 * k + 1),
                            DhOut{dHbuf, true, dh_parts(c, rows, false), c.L.ldp}, dW, k > 0,
                            dloss, GradSpec{c.Gb[0], c.Gb[0], frozen ? 0 : rows, true, false},
                            &parts));
            LCE_TRY(norm_bwd(row0, rows, parts));
        }
    }
    if (!none)
        LCE_LAUNCH(launch_loss_finalize(c.loss_rows, c.N, c.hdr, loss,
                                        reduction == LCE_REDUCTION_MEAN, c.s));
    if (c.L.nchunks > 0)
        LCE_LAUNCH_KIND(LCE_KERNEL_NORM, c.s, launch_dgamma_reduce(part, static_cast<int>(c.D), dgamma, c.s));
    return LCE_OK;
}

lce_status lce_norm_fwd_bwd(const void *X, const void *gamma, float eps, const void *W,
                            const int64_t *y, const float *dloss, int64_t N, int64_t D, int64_t V,
                            int64_t ignore_index, int64_t chunk, int reduction, float *loss,
                            float *lse, void *dX, float *dgamma, float *dW, void *ws,
                            size_t ws_bytes, lce_stream_t stream) {
    return lce_norm_fwd_bwd_opt(X, gamma, eps, W, y, dloss, N, D, V, ignore_index, chunk, reduction,
                                0, loss, lse, dX, dgamma, dW, ws, ws_bytes, stream);
}

lce_status lce_ce_logits_workspace_size(int64_t N, size_t *bytes) {
    if (!bytes || N < 0) return LCE_ERR_INVALID_ARG;
    *bytes = 1024 + align_up(sizeof(float) * static_cast<size_t>(N > 0 ? N : 1), 1024);
    return LCE_OK;
}

lce_status lce_ce_logits(const void *Z, int z_dtype, int64_t ld, const int64_t *y, int64_t N,
                         int64_t V, int64_t ignore_index, int reduction, const float *dloss,
                         float *loss, float *lse, void *dZ, void *ws, size_t ws_bytes,
                         lce_stream_t stream) {
    g_launches = 0;
    if (reduction < LCE_REDUCTION_MEAN || reduction > LCE_REDUCTION_NONE) return LCE_ERR_INVALID_ARG;
    const bool none = reduction == LCE_REDUCTION_NONE;
    if (N < 0 || V <= 0 || ld < V || !ws) return LCE_ERR_INVALID_ARG;
    if (N > 0 && (!Z || !y || !lse || !loss)) return LCE_ERR_INVALID_ARG;
    if (!none && !loss) return LCE_ERR_INVALID_ARG;
    if (z_dtype < CE_BF16 || z_dtype > CE_FP16) return LCE_ERR_INVALID_ARG;
    const int vec = z_dtype == CE_FP32 ? 4 : 8;
    if (ld % vec != 0) return LCE_ERR_ALIGNMENT;
    if ((Z && !aligned16(Z)) || (dZ && !aligned16(dZ)) || !aligned16(ws) ||
        (loss && !aligned16(loss)) || (lse && !aligned16(lse)) || (y && !aligned16(y)))
        return LCE_ERR_ALIGNMENT;
    size_t need = 0;
    lce_ce_logits_workspace_size(N, &need);
    if (ws_bytes < need) return LCE_ERR_WORKSPACE;
    int sms = 0, pairs = 0;
    lce_status st = init_device(&sms, &pairs);
    if (st != LCE_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint8_t *w = static_cast<uint8_t *>(ws);
    int *hdr = reinterpret_cast<int *>(w);
    float *loss_rows = reinterpret_cast<float *>(w + 1024);
    if (cudaMemsetAsync(hdr, 0, 1024, s) != cudaSuccess) return LCE_ERR_CUDA;
    LCE_LAUNCH_KIND(LCE_KERNEL_OTHER, s,
                    launch_label_scan(reinterpret_cast<const long long *>(y), N, V, ignore_index, hdr, s));
    CELogitsParams p;
    p.Z = Z;
    p.dZ = dZ;
    p.ld = ld;
    p.dtype = z_dtype;
    p.N = N;
    p.V = V;
    p.ignore_index = ignore_index;
    p.y = reinterpret_cast<const long long *>(y);
    p.hdr = hdr;
    p.dloss = dloss;
    p.dloss_per_row = none ? 1 : 0;
    p.mean = reduction == LCE_REDUCTION_MEAN ? 1 : 0;
    p.lse = lse;
    p.loss_rows = none ? loss : loss_rows;
    LCE_LAUNCH_KIND(LCE_KERNEL_MERGE, s, launch_ce_logits(p, sms, s));
    if (!none)
        LCE_LAUNCH_KIND(LCE_KERNEL_OTHER, s,
                        launch_loss_finalize(loss_rows, N, hdr, loss,
                                             reduction == LCE_REDUCTION_MEAN, s));
    return LCE_OK;
}

lce_status lce_selftest_wait_timeout(void *ws, size_t ws_bytes, int64_t limit_us,
                                     lce_stream_t stream) {
    g_launches = 0;
    if (!ws || ws_bytes < 1024) return LCE_ERR_INVALID_ARG;
    if (limit_us < 1 || limit_us > 2000000) return LCE_ERR_INVALID_ARG;
    if (!aligned16(ws)) return LCE_ERR_ALIGNMENT;
    int sms = 0, pairs = 0;
    lce_status st = init_device(&sms, &pairs);
    if (st != LCE_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(ws, 0, 1024, s) != cudaSuccess) return LCE_ERR_CUDA;
    LCE_LAUNCH_KIND(LCE_KERNEL_OTHER, s,
                    launch_wait_selftest(static_cast<int *>(ws),
                                         static_cast<unsigned long long>(limit_us) * 1000ull, s));
    return LCE_OK;
}

lce_status lce_read_status(const void *ws, lce_stream_t stream) {
    if (!ws) return LCE_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return LCE_ERR_CUDA;
    int flag = 0;
    if (cudaMemcpy(&flag, ws, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return LCE_ERR_CUDA;
    if (flag) {
        const int zero = 0;
        if (cudaMemcpy(const_cast<void *>(ws), &zero, sizeof(int), cudaMemcpyHostToDevice) !=
            cudaSuccess)
            return LCE_ERR_CUDA;
    }
    if (flag & FLAG_TIMEOUT) return LCE_ERR_TIMEOUT;
    if (flag & FLAG_LABEL) return LCE_ERR_LABEL_RANGE;
    return LCE_OK;
}

const char *lce_status_string(lce_status s) {
    switch (s) {
        case LCE_OK: return "ok";
        case LCE_ERR_INVALID_ARG: return "invalid argument";
        case LCE_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
        case LCE_ERR_WORKSPACE: return "workspace too small";
        case LCE_ERR_LABEL_RANGE: return "label outside [0, V) and not ignore_index";
        case LCE_ERR_TIMEOUT: return "device pipeline wait timed out";
        case LCE_ERR_CUDA: return "CUDA runtime error";
        case LCE_ERR_UNSUPPORTED: return "device is not sm_103";
    }
    return "unknown status";
}

int lce_version(void) { return 100; }

int lce_last_launch_count(void) { return g_launches; }

lce_status lce_profile_enable(int on) {
    std::lock_guard<std::mutex> lock(g_prof_mu);
    g_prof_on = on != 0;
    return LCE_OK;
}

lce_status lce_profile_read(int kind, double *total_ms, int64_t *launches) {
    if (kind < 0 || kind >= LCE_KERNEL_KINDS || !total_ms || !launches) return LCE_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g_prof_mu);
    for (ProfPair &p : g_prof_pending) {
        if (cudaEventSynchronize(p.b) != cudaSuccess) return LCE_ERR_CUDA;
        float ms = 0.f;
        if (cudaEventElapsedTime(&ms, p.a, p.b) != cudaSuccess) return LCE_ERR_CUDA;
        g_prof_ms[p.kind] += ms;
        g_prof_n[p.kind] += 1;
        g_prof_pool.push_back(p.a);
        g_prof_pool.push_back(p.b);
    }
    g_prof_pending.clear();
    *total_ms = g_prof_ms[kind];
    *launches = g_prof_n[kind];
    return LCE_OK;
}

void lce_profile_reset(void) {
    std::lock_guard<std::mutex> lock(g_prof_mu);
    for (int k = 0; k < LCE_KERNEL_KINDS; ++k) {
        g_prof_ms[k] = 0.0;
        g_prof_n[k] = 0;
    }
}

}  // extern "C"
