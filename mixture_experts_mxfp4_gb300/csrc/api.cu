// Host side of the C ABI (include/moe_mxfp4.h): argument validation, workspace
// planning, TMA descriptor encoding and the launch sequence
//   route -> quant -> stage-1 GEMM -> stage-2 GEMM -> top-k sum
// on the caller's stream.  Nothing here allocates device memory.
#include <cuda.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "../../include/moe_mxfp4.h"
#include "moe_internal.h"

using namespace moe;

namespace {

constexpr int kMaxDevices = 64;
constexpr size_t kAlign = 256;

struct WorkspaceReg {
    void* ptr = nullptr;
    size_t bytes = 0;
};

constexpr int kNumKernels = 4;

struct Timing {
    int mode = 0;
    bool enabled = false;
    bool created = false;
    bool recorded = false;
    unsigned launched = 0;  // bit i: the last call launched something in slot i
    cudaEvent_t ev[kNumKernels + 1];
};

std::mutex g_mu;
WorkspaceReg g_ws[kMaxDevices];

// NVTX ranges (moe_mxfp4_set_nvtx): a call range and one range per launch.
std::atomic<int> g_nvtx{0};

struct LaunchRange {
    bool on;
    explicit LaunchRange(const char* name) : on(g_nvtx.load(std::memory_order_relaxed) != 0) {
        if (on) nvtxRangePushA(name);
    }
    ~LaunchRange() {
        if (on) nvtxRangePop();
    }
};

struct CallRange {
    bool on;
    CallRange(const char* entry, int T, int D, int I, int E, int K, int launches)
        : on(g_nvtx.load(std::memory_order_relaxed) != 0) {
        if (!on) return;
        char msg[160];
        snprintf(msg, sizeof(msg), "moe_mxfp4 forward (%s) T=%d d_model=%d d_inter=%d E=%d topk=%d launches=%d",
                 entry, T, D, I, E, K, launches);
        nvtxRangePushA(msg);
    }
    ~CallRange() {
        if (on) nvtxRangePop();
    }
};
int g_num_sms[kMaxDevices];
// moe_mxfp4_set_single_launch mode per device (0 separate, 1 single, 2 auto); -1 = unset
int g_single_launch[kMaxDevices] = {};
bool g_single_set[kMaxDevices] = {};
Timing g_timing[kMaxDevices];
// Workspace the last forward call on each device used (the registered buffer or
// the no-allocation entry point's static array): moe_mxfp4_last_device_status
// reads its status word.
void* g_last_ws[kMaxDevices];

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Contraction widths the GEMM kernels take as they are: one stage of 128 or 256
// elements, or stages of 512.
bool supported_k(int k) { return k == 128 || k == 256 || (k > 0 && k % 512 == 0); }

// Width the kernels run a width k at: k itself where supported, else the next
// supported width (its extra columns are zero in the activations and read as
// zero from the weights).
int stored_k(int k) {
    if (supported_k(k)) return k;
    if (k < 128) return 128;
    if (k < 256) return 256;
    return (int)round_up((size_t)k, 512);
}

// Weights of widths the kernels do not run at natively (d_model a multiple of
// 128, d_inter of 64, either not a supported width).
bool widened(int D, int I) { return !supported_k(D) || !supported_k(I); }

moe_status_t validate_shape(int T, int D, int I, int E, int K) {
    if (T < 0 || E < 1 || E > 1024 || K < 1 || K > 16) return MOE_ERR_INVALID_ARG;
    if (D <= 0 || I <= 0) return MOE_ERR_INVALID_ARG;
    if (D % 128 != 0 || I % 64 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
    if ((long long)T * K > (1LL << 24)) return MOE_ERR_UNSUPPORTED_SHAPE;
    return MOE_OK;
}

// Tuning override (moe_mxfp4_set_tuning): forced route-tile width and scale-factor
// copy scheme; 0 = the library's choice.  Process-wide.
std::atomic<int> g_force_tile_rows{0};
std::atomic<int> g_force_sf_copies{0};

// Maximum routes per GEMM tile: small tiles when experts see few routes
// (decode), full 128-row tiles when they see many (prefill, dense shards).
int choose_tile_rows(int T, int E, int K) {
    const int forced = g_force_tile_rows.load(std::memory_order_relaxed);
    if (forced) return forced;
    const double per_expert = (double)T * K / (double)E;
    if (per_expert > 48.0) return 128;
    if (per_expert > 24.0) return 64;
    if (per_expert > 8.0) return 32;
    return 16;
}

// bf16_act: layout of the bf16-activation forward (bf16 a1/a2 rows instead of
// the MXFP4 codes and scales).
// D, I: the widths of the weight tensors; the workspace rows use the widths the
// kernels run at (stored_k).
void fill_plan(int T, int Dw, int Iw, int E, int K, moe_mxfp4_plan_t* pl, bool bf16_act = false) {
    memset(pl, 0, sizeof(*pl));
    const int D = stored_k(Dw), I = stored_k(Iw);
    pl->d_model_run = D;
    pl->d_inter_run = I;
    const long long R = (long long)T * K;
    const long long used = R < E ? R : E;
    long long cap = R + used * (kBlockM - 1);
    cap = (cap + kBlockM - 1) / kBlockM * kBlockM;
    pl->block_m = kBlockM;
    pl->tile_rows = choose_tile_rows(T, E, K);
    pl->cap = (int)cap;
    pl->a1s_stride = (int)round_up((size_t)(D / 32), 16);
    pl->a2s_stride = (int)round_up((size_t)(I / 32), 16);
    pl->max_tiles = (int)(cap / kBlockM);
    // No K split of stage 1: the GEMM kernel evens out its CTAs' work with the
    // distribution of stage-2 items instead.
    pl->stage1_splits = 1;
    size_t b[MOE_WS_NUM_REGIONS];
    b[MOE_WS_STATUS] = kStatusWords * sizeof(uint32_t);
    b[MOE_WS_COUNTERS] = (size_t)pl->max_tiles * sizeof(uint32_t);  // finished feature tiles per route tile
    b[MOE_WS_SORTED_IDS] = (size_t)cap * 4;
    b[MOE_WS_SORTED_W] = (size_t)cap * 4;
    b[MOE_WS_BLOCK_EXPERT] = (size_t)(cap / kBlockM) * 4;
    b[MOE_WS_SEG_START] = (size_t)(E + 1) * 4;
    b[MOE_WS_ROUTE_POS] = (size_t)R * 4;
    b[MOE_WS_NUM_VALID] = 4 * 4;
    b[MOE_WS_TILES] = (size_t)pl->max_tiles * 16;
    b[MOE_WS_A1Q] = (size_t)cap * (D / 2);
    b[MOE_WS_A1S] = (size_t)cap * pl->a1s_stride;
    b[MOE_WS_A2Q] = (size_t)cap * (I / 2);
    b[MOE_WS_A2S] = (size_t)cap * pl->a2s_stride;
    b[MOE_WS_P] = (size_t)R * D * 4;
    b[MOE_WS_PARTIAL] = 0;  // (no K split)
    b[MOE_WS_A1B] = 0;
    b[MOE_WS_A2B] = 0;
    // weight scales repacked to rows of D/32 and I/32 bytes (widths run wider)
    b[MOE_WS_WSCALE] = widened(Dw, Iw) ? round_up((size_t)E * 2 * Iw * (D / 32), kAlign) + (size_t)E * Dw * (I / 32)
                                        : 0;
    if (bf16_act) {
        pl->bf16_act = 1;
        b[MOE_WS_A1Q] = b[MOE_WS_A1S] = b[MOE_WS_A2Q] = b[MOE_WS_A2S] = 0;
        b[MOE_WS_A1B] = (size_t)cap * D * 2;
        b[MOE_WS_A2B] = (size_t)cap * I * 2;
    }
    size_t off = 0;
    for (int i = 0; i < MOE_WS_NUM_REGIONS; ++i) {
        pl->offset[i] = off;
        pl->bytes[i] = b[i];
        off = round_up(off + b[i], kAlign);
    }
    pl->workspace_bytes = off;
}

WsPtrs ws_ptrs(void* base, const moe_mxfp4_plan_t& pl) {
    uint8_t* b = static_cast<uint8_t*>(base);
    WsPtrs w;
    w.status = reinterpret_cast<uint32_t*>(b + pl.offset[MOE_WS_STATUS]);
    w.counters = reinterpret_cast<uint32_t*>(b + pl.offset[MOE_WS_COUNTERS]);
    w.sorted_ids = reinterpret_cast<int32_t*>(b + pl.offset[MOE_WS_SORTED_IDS]);
    w.sorted_w = reinterpret_cast<float*>(b + pl.offset[MOE_WS_SORTED_W]);
    w.block_expert = reinterpret_cast<int32_t*>(b + pl.offset[MOE_WS_BLOCK_EXPERT]);
    w.seg_start = reinterpret_cast<int32_t*>(b + pl.offset[MOE_WS_SEG_START]);
    w.route_pos = reinterpret_cast<int32_t*>(b + pl.offset[MOE_WS_ROUTE_POS]);
    w.num_valid = reinterpret_cast<int32_t*>(b + pl.offset[MOE_WS_NUM_VALID]);
    w.tiles = reinterpret_cast<int4*>(b + pl.offset[MOE_WS_TILES]);
    w.a1q = b + pl.offset[MOE_WS_A1Q];
    w.a1s = b + pl.offset[MOE_WS_A1S];
    w.a2q = b + pl.offset[MOE_WS_A2Q];
    w.a2s = b + pl.offset[MOE_WS_A2S];
    w.P = reinterpret_cast<float*>(b + pl.offset[MOE_WS_P]);
    w.tile_done = w.counters;
    w.quant_done = w.status + kFrontQuantWord;
    w.a1b = reinterpret_cast<uint16_t*>(b + pl.offset[MOE_WS_A1B]);
    w.a2b = reinterpret_cast<uint16_t*>(b + pl.offset[MOE_WS_A2B]);
    return w;
}

// ------------------------------------------------------------------ TMA maps

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// Looked up once; guarded by its own mutex because it is called while g_mu is
// held (launch-state construction).
std::mutex g_encode_mu;

EncodeTiledFn get_encode() {
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    std::lock_guard<std::mutex> lk(g_encode_mu);
    if (!tried) {
        tried = true;
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// Tiled u8 tensor map of rank r: dims innermost first, strides (bytes) of dims
// 1..r-1, box extents.  The dimensions may overlap in memory (a K-box dimension
// with a stride smaller than the row stride), which lets one box gather the
// K-tiles of a stage or the gate and up halves of w13.
bool make_map_nd(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
                 const uint64_t* strides, const uint32_t* box, CUtensorMapSwizzle swz) {
    EncodeTiledFn enc = get_encode();
    if (!enc) return false;
    cuuint64_t d[5];
    cuuint64_t st[4];
    cuuint32_t b[5];
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
        if (i + 1 < rank) st[i] = strides[i];
    }
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, (cuuint32_t)rank, const_cast<void*>(base), d,
                     st, b, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 2-D u8 tensor [rows][inner] with row stride `stride` bytes, box {bx, by}.
bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint64_t stride,
              uint32_t bx, uint32_t by, CUtensorMapSwizzle swz) {
    const uint64_t dims[2] = {inner, rows};
    const uint64_t strides[1] = {stride};
    const uint32_t box[2] = {bx, by};
    return make_map_nd(m, base, 2, dims, strides, box, swz);
}

// Packed-e2m1 operand [rows][Kc/2 bytes] seen as {kb bytes, rows, Kc/2/kb K-boxes}
// (optionally with a second row dimension of `halves` at `half_stride` bytes):
// one box brings box_rows rows x nkt K-boxes, laid out [kbox][half][row][kb].
bool make_operand_map(CUtensorMap* m, const void* base, uint64_t rows, int Kc, int kb, int nkt,
                      int box_rows, int halves, uint64_t half_stride) {
    const uint64_t row_bytes = (uint64_t)Kc / 2;
    const CUtensorMapSwizzle swz = kb == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    if (halves > 1) {
        const uint64_t dims[4] = {(uint64_t)kb, rows, (uint64_t)halves, row_bytes / kb};
        const uint64_t strides[3] = {row_bytes, half_stride, (uint64_t)kb};
        const uint32_t box[4] = {(uint32_t)kb, (uint32_t)box_rows, (uint32_t)halves, (uint32_t)nkt};
        return make_map_nd(m, base, 4, dims, strides, box, swz);
    }
    const uint64_t dims[3] = {(uint64_t)kb, rows, row_bytes / kb};
    const uint64_t strides[2] = {row_bytes, (uint64_t)kb};
    const uint32_t box[3] = {(uint32_t)kb, (uint32_t)box_rows, (uint32_t)nkt};
    return make_map_nd(m, base, 3, dims, strides, box, swz);
}

// Weight map for weights narrower than the width the kernels run at: rows of
// Kw/2 bytes, one K box (kb bytes) per copy, the columns past the row read as
// zeros (the copy's out-of-bounds fill).  halves = 2 as for make_operand_map.
bool make_kbox_map(CUtensorMap* m, const void* base, uint64_t rows, int Kw, int kb, int box_rows,
                   int halves, uint64_t half_stride) {
    const uint64_t row_bytes = (uint64_t)Kw / 2;
    const CUtensorMapSwizzle swz = kb == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    if (halves > 1) {
        const uint64_t dims[3] = {row_bytes, rows, (uint64_t)halves};
        const uint64_t strides[2] = {row_bytes, half_stride};
        const uint32_t box[3] = {(uint32_t)kb, (uint32_t)box_rows, (uint32_t)halves};
        return make_map_nd(m, base, 3, dims, strides, box, swz);
    }
    const uint64_t dims[2] = {row_bytes, rows};
    const uint64_t strides[1] = {row_bytes};
    const uint32_t box[2] = {(uint32_t)kb, (uint32_t)box_rows};
    return make_map_nd(m, base, 2, dims, strides, box, swz);
}

// Weight-scale map: [rows][S] e8m0 bytes; S >= 16 read 16 bytes per stage, S < 16
// read through a [rows*S/16][16] view so that one box holds box_rows whole rows.
// With halves = 2 a third dimension adds the rows `half_rows` further (w13 up rows).
bool make_scale_map(CUtensorMap* m, const void* base, uint64_t rows, int S, int box_rows,
                    int halves, uint64_t half_rows) {
    const bool small = S < 16;
    const uint64_t inner = small ? 16 : (uint64_t)S;
    const uint64_t vrows = small ? rows * S / 16 : rows;
    const uint64_t stride = small ? 16 : (uint64_t)S;
    const uint32_t brows = small ? (uint32_t)(box_rows * S / 16) : (uint32_t)box_rows;
    if (halves > 1) {
        const uint64_t dims[3] = {inner, vrows, (uint64_t)halves};
        const uint64_t strides[2] = {stride, half_rows * (uint64_t)S};
        const uint32_t box[3] = {16, brows, (uint32_t)halves};
        return make_map_nd(m, base, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
    }
    return make_map(m, base, inner, vrows, stride, 16, brows, CU_TENSOR_MAP_SWIZZLE_NONE);
}

// Layout of one GEMM stage for contraction length Kc inside a ring slot.
// Returns the bytes one stage of it occupies.
// Stages of up to 512 elements along K.  (Stages of 256 elements with twice as
// many ring slots measured much slower: dense T=512 280 -> 392 us, decode T=16
// 84 -> 155 us; the per-stage hand-offs between the roles set the pace.)
uint32_t stage_geometry(StageGeom& q, int Kc, int tile_rows, int mblocks) {
    q.mblocks = mblocks;
    q.kstage_elems = Kc >= 512 ? 512 : Kc;
    q.kstages = Kc / q.kstage_elems;
    q.kb = q.kstage_elems >= 256 ? 128 : 64;
    q.nkt = (q.kstage_elems / 2) / q.kb;
    q.natoms = q.kstage_elems / 128;
    const int S = Kc / 32;
    q.a_scale_small = S < 16 ? 1 : 0;
    q.sr_a = S < 16 ? S : 16;
    q.b_scale_x = S >= 16 ? 1 : 0;
    const uint32_t a_bytes = 128u * mblocks * (q.kstage_elems / 2);
    const uint32_t b_bytes = (uint32_t)tile_rows * (q.kstage_elems / 2);
    // raw weight scales (128 * mblocks rows of sr_a bytes), rearranged in place
    uint32_t sa_bytes = 128u * mblocks * (uint32_t)q.sr_a;
    if (sa_bytes < 2048u) sa_bytes = 2048u;
    q.off_b = a_bytes;
    q.off_sa = q.off_b + b_bytes;
    q.off_sb = q.off_sa + sa_bytes;
    return (uint32_t)round_up(q.off_sb + 2048, 1024);
}

// Geometry of the fused GEMM kernel.  A kernel that allocates tensor memory runs
// one CTA per SM (the occupancy calculator reports 1 for any kernel containing
// tcgen05.alloc, whatever its threads, registers or shared memory), so each CTA
// owns the SM's 227 KB of shared memory and 512 TMEM columns.  The ring slots
// hold either stage's layout.  Narrow route tiles (decode) use two MMA-issuing
// warps: a single stream of scale-factor copies and narrow MMAs leaves the
// tensor pipe idle between instructions, and a second stream fills it.
// D, I: the widths the kernels run at; Dw, Iw: the weights' (the feature tiles
// cover those: the gate_up GEMM's outputs past Iw, which the down GEMM multiplies
// by zero weight columns, are zeroed before the call instead).
void gemm_geometry(GemmParams& g, int D, int I, int Dw, int Iw, int tile_rows, int mblocks2, int sf_copies) {
    g.tile_rows = tile_rows;
    const uint32_t b1 = stage_geometry(g.g[0], D, tile_rows, 1);
    const uint32_t b2 = stage_geometry(g.g[1], I, tile_rows, mblocks2);
    g.g[0].n_ftiles = Iw / 64;
    g.g[1].n_ftiles = Dw / (128 * mblocks2);
    g.slot_bytes = b1 > b2 ? b1 : b2;
    // epilogue groups: three for 128-route tiles whose stage-2 items are a single
    // stage (the stage-2 epilogue bounds those, see kMaxEpiGroups), else two
    g.epi_groups = (tile_rows == 128 && g.g[1].kstages == 1) ? 3 : 2;
    const uint32_t xchg = (uint32_t)(g.epi_groups * kXchgBytes);  // epilogue exchange buffers
    const uint32_t tcache = (uint32_t)kTileCache * 16u;
    const uint32_t fixed = 1024 /*align slack*/ + 512 /*barriers*/ + xchg + tcache;
    uint32_t budget = 227u * 1024u - fixed;
    // Scale-factor copies (sf_copies, 0 = by shape): 1, each of two MMA warps
    // copies its own stages' (narrow route tiles); 2, the scale-layout warp copies
    // one 128-element chunk per instruction (.32x128b.warpx4) and one MMA warp
    // issues only MMAs (128-route tiles); 3, as 2 but two chunks per instruction
    // (.128x256b, the same cost per instruction) from two staging buffers of
    // (mblocks + 1) * natoms / 2 blocks of 4 KB, where they leave the ring at least
    // 4 slots (else as 2).  Measured (same GB300, alternating processes, trimmed
    // means of 400/300 calls): decode T=16 85.1 / 83.9 / 89.0 us for schemes
    // 1 / 2 / 3, decode T=128 169.5 / 168.9 / 184.6 us; dense T=512 291 us in
    // every scheme (there 3 falls back to 2).  Scheme 2 is the default.  4: the
    // scale-layout warp copies one chunk per instruction and two MMA warps take
    // alternate stages (a single issuing thread serialises its MMAs; where the
    // two warps' accumulators do not fit in TMEM it falls back to 2).
    int mode = sf_copies ? sf_copies : 2;
    auto wide_of = [](const StageGeom& q) {
        return q.natoms % 2 == 0 ? (uint32_t)((q.mblocks + 1) * (q.natoms / 2)) * 4096u : 0u;
    };
    const uint32_t sfw = wide_of(g.g[0]) > wide_of(g.g[1]) ? wide_of(g.g[0]) : wide_of(g.g[1]);
    g.wide_sf = 0;
    g.sfw_bytes = 0;
    if (mode == 3) {
        if (sfw > 0 && (budget - 2 * sfw) / g.slot_bytes >= 4) {
            g.wide_sf = 1;
            g.sfw_bytes = sfw;
            budget -= 2 * sfw;
        } else {
            mode = 2;
        }
    }
    int ns = (int)(budget / g.slot_bytes);
    if (ns > kMaxStages) ns = kMaxStages;
    const int mbmax = mblocks2 > 1 ? mblocks2 : 1;
    int mw = (mode == 1 || mode == 4) ? 2 : 1;
    // TMEM: acc_bufs accumulator buffers of one N-column accumulator per MMA warp
    // and weight block, plus each ring slot's scale factors ((mblocks + 1) atoms
    // of 4 columns per 128-element chunk).
    auto sf_of = [](const StageGeom& q) { return (uint32_t)((q.mblocks + 1) * 4 * q.natoms); };
    const uint32_t sfc = sf_of(g.g[0]) > sf_of(g.g[1]) ? sf_of(g.g[0]) : sf_of(g.g[1]);
    auto cols_for = [&](int b, int m, int n) {
        return (uint32_t)(b * m * mbmax * tile_rows) + (uint32_t)n * sfc;
    };
    // accumulator buffers: as many as fit, up to 4 (128-route tiles: 3, measured
    // dense T=512 290.7 -> 279.8 us and prefill T=4096 814 -> 802.6 us against 2)
    auto pick_nb = [&]() {
        int b = 4;
        if (cols_for(b, mw, ns) > 512u) b = 3;
        if (cols_for(b, mw, ns) > 512u) b = 2;
        return b;
    };
    int nb = pick_nb();
    if (cols_for(nb, mw, ns) > 512u) {  // two MMA warps' accumulators do not fit: one
        mw = 1;
        nb = pick_nb();
    }
    while (ns > 1 && cols_for(nb, mw, ns) > 512u) --ns;
    // An epilogue group's next item uses buffer (item % nb); its wait on that
    // buffer's barrier parity is unambiguous only if the buffer's previous user has
    // completed its MMAs, which the group's own previous item (item - groups)
    // guarantees when nb >= groups (MMAs complete in order).  Fewer buffers than
    // groups (a forced copy scheme whose two MMA warps fell back to one) get fewer
    // groups.
    if (g.epi_groups > nb) g.epi_groups = nb;
    // Two MMA warps take alternate stages and wait for a slot's fill by barrier
    // parity.  That parity is unambiguous only if the warp has seen the slot's
    // previous fill, i.e. if the slot's previous stage (g - ns) was its own: ns
    // even.  (With an odd ns a warp could take the slot's previous fill, still in
    // flight behind a later one, for its own.)  The same holds for the MMA warps'
    // look-ahead test of slot (g + mw) % ns.
    if (mw == 2 && (ns & 1) && ns > 2) --ns;
    if (mw == 2 && ns < 2) mw = 1;  // (one slot: a single MMA warp)
    g.lookahead = (ns % mw == 0 && ns > mw) ? 1 : 0;
    // With one MMA warp (wide route tiles) the scale-layout warp also copies each
    // stage's scale factors to TMEM, so the MMA warp issues MMAs only (measured:
    // dense T512 390 -> 340 us); two MMA warps overlap their copies better themselves.
    g.sf_by_layout_warp = (mode != 1 || mw == 1) ? 1 : 0;
    g.mma_warps = mw;
    g.acc_bufs = nb;
    g.num_stages = ns;
    g.acc_cols = (uint32_t)(mw * mbmax * tile_rows);
    g.sf_cols = sfc;
    g.off_bar = (uint32_t)ns * g.slot_bytes;
    g.off_xchg = g.off_bar + 512;  // barriers, TMEM slot and abort flag fit in 512 bytes
    g.off_tiles = g.off_xchg + xchg;
    g.off_sfw = g.off_tiles + tcache;  // (1024-aligned: every term above is)
    g.smem_bytes = g.off_sfw + 2 * g.sfw_bytes + 1024u;
    const uint32_t cols = cols_for(nb, mw, ns);
    uint32_t alloc = 32;
    while (alloc < cols) alloc <<= 1;
    g.tmem_cols = alloc;
    g.sf_col0 = (uint32_t)nb * g.acc_cols;
}

int num_sms(int dev) {
    if (dev < 0 || dev >= kMaxDevices) return 148;
    if (g_num_sms[dev] == 0) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        g_num_sms[dev] = n > 0 ? n : 148;
    }
    return g_num_sms[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" {

#if MOE_CHECKED
const char* moe_mxfp4_version(void) { return "moe_mxfp4 0.2 (sm_103a, tcgen05 mxf4; bounds-checked build)"; }
#else
const char* moe_mxfp4_version(void) { return "moe_mxfp4 0.2 (sm_103a, tcgen05 mxf4)"; }
#endif

int moe_mxfp4_pointer_kind(const void* ptr) {
    if (!ptr) return -1;
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess) {
        cudaGetLastError();  // clear the error the query may leave
        return -1;
    }
    if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) return 0;
    if (a.type == cudaMemoryTypeHost && a.devicePointer == ptr) return 1;
    return -1;
}

const char* moe_mxfp4_status_string(moe_status_t s) {
    switch (s) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
        case MOE_ERR_MISALIGNED: return "pointer not 16-byte aligned";
        case MOE_ERR_WORKSPACE: return "workspace missing or too small";
        case MOE_ERR_CUDA: return "CUDA error";
        case MOE_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    }
    return "unknown status";
}

moe_status_t moe_mxfp4_get_plan(int T, int d_model, int d_inter, int E, int topk,
                                moe_mxfp4_plan_t* plan) {
    if (!plan) return MOE_ERR_INVALID_ARG;
    moe_status_t st = validate_shape(T, d_model, d_inter, E, topk);
    if (st != MOE_OK) return st;
    fill_plan(T, d_model, d_inter, E, topk, plan);
    return MOE_OK;
}

size_t moe_mxfp4_workspace_size(int T, int d_model, int d_inter, int E, int topk) {
    moe_mxfp4_plan_t pl;
    if (moe_mxfp4_get_plan(T, d_model, d_inter, E, topk, &pl) != MOE_OK) return 0;
    return pl.workspace_bytes;
}

moe_status_t moe_mxfp4_set_workspace(void* dev_ptr, size_t bytes) {
    if (dev_ptr && (reinterpret_cast<uintptr_t>(dev_ptr) % kAlign) != 0) return MOE_ERR_MISALIGNED;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
    if (dev_ptr && bytes < kStatusWords * sizeof(uint32_t)) return MOE_ERR_WORKSPACE;
    std::lock_guard<std::mutex> lk(g_mu);
    g_ws[dev].ptr = dev_ptr;
    g_ws[dev].bytes = dev_ptr ? bytes : 0;
    return MOE_OK;
}

moe_status_t moe_mxfp4_last_device_status(cudaStream_t stream) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
    void* base;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        base = g_last_ws[dev] ? g_last_ws[dev] : g_ws[dev].ptr;
    }
    if (!base) return MOE_ERR_WORKSPACE;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return MOE_ERR_CUDA;
    uint32_t word = 0;
    // status is region 0 at offset 0 of every plan
    if (cudaMemcpy(&word, base, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
        return MOE_ERR_CUDA;
    return word ? MOE_ERR_DEVICE_TIMEOUT : MOE_OK;
}

}  // extern "C"

namespace moe {

moe_status_t validate_forward(const void* hidden, const void* w13, const void* w13_scale,
                              const void* w2, const void* w2_scale, const int32_t* topk_ids,
                              const float* topk_weights, const void* out, int T, int D, int I,
                              int E, int K) {
    moe_status_t st = validate_shape(T, D, I, E, K);
    if (st != MOE_OK) return st;
    if (T == 0) return MOE_OK;
    if (!hidden || !w13 || !w13_scale || !w2 || !w2_scale || !topk_ids || !topk_weights || !out)
        return MOE_ERR_INVALID_ARG;
    if (!aligned16(hidden) || !aligned16(w13) || !aligned16(w13_scale) || !aligned16(w2) ||
        !aligned16(w2_scale) || !aligned16(topk_ids) || !aligned16(topk_weights) || !aligned16(out))
        return MOE_ERR_MISALIGNED;
    return MOE_OK;
}

// Logical sizes of a padded call: multiples of 32 (one scale block), at least
// 32, at most the stored sizes.
moe_status_t validate_padded(int D, int I, int Dl, int Il) {
    if (Dl < 32 || Il < 32 || Dl % 32 != 0 || Il % 32 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (Dl > D || Il > I) return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

// The launch sequence of one forward call on the workspace at `base` (at least
// workspace_bytes of the shape's plan, 256-byte aligned); arguments validated.
}  // namespace moe

namespace {

// Host state of one forward configuration: the plan, both GEMMs' parameters and
// their eight TMA descriptors.  They depend only on the shape, the weight
// pointers and the workspace, so they are built once and reused; this keeps
// the per-call host work to the five launches.
struct LaunchState {
    CUtensorMap maps[8];  // stage-1 A, SA, B, SB, stage-2 A, SA, B, SB
    moe::GemmParams gp;
    moe_mxfp4_plan_t pl;
    void* wscale13;  // repacked weight scales (weights narrower than the run widths)
    void* wscale2;
    const void* key_ptr[5];
    int key_shape[7];  // T, D, I, E, K, forced tile width, forced copy scheme
    bool valid;
};

constexpr int kCacheWays = 4;
LaunchState g_cache[kMaxDevices][kCacheWays];
int g_cache_next[kMaxDevices];

// Plan and GEMM geometry of a shape (no device pointers).
// D, I: the widths of the weight tensors.
void shape_geometry(int T, int D, int I, int E, int K, moe_mxfp4_plan_t* pl, GemmParams* gp) {
    fill_plan(T, D, I, E, K, pl);
    memset(gp, 0, sizeof(*gp));
    gp->D = stored_k(D); gp->I = stored_k(I); gp->E = E; gp->K = K; gp->R = T * K;
    gp->Dw = D; gp->Iw = I;
    gp->kt_boxes = widened(D, I) ? 1 : 0;
    gp->a1s_stride = pl->a1s_stride;
    gp->a2s_stride = pl->a2s_stride;
    // stage 2 on narrow tiles: two 128-row blocks of w2 per item share the route tile
    const int mb2 = (pl->tile_rows <= 64 && D % 256 == 0) ? 2 : 1;
    gemm_geometry(*gp, gp->D, gp->I, D, I, pl->tile_rows, mb2, g_force_sf_copies.load(std::memory_order_relaxed));
}

// Whether a call of this shape routes and quantises inside the GEMM kernel under
// the device's launch mode (0 separate, 1 single where possible, 2 automatic).
// The in-kernel routing scratch must fit in the ring, the route positions in the
// exchange buffer and the route tiles in the tile cache (R / block_m + E <= 512).
bool single_launch_for(int dev, int T, int E, int K, const GemmParams& gp) {
    static_assert(kFrontMaxRoutes * 4 <= kEpiGroups * kXchgBytes, "route positions");
    static_assert(kFrontMaxRoutes / kBlockM + kFrontMaxExperts <= kTileCache, "route tiles");
    static_assert(kFrontTileWord + kTileCache <= kStatusWords, "route-tile counters");
    const size_t scratch = sizeof(int) * ((size_t)(kGemmThreads / 32 + 1) * E + 1 + 2 * (kGemmThreads / 32) + 4);
    const int mode = g_single_set[dev] ? g_single_launch[dev] : 2;
    const long long routes = (long long)T * K;
    return (mode == 1 || (mode == 2 && routes <= kFrontAutoRoutes)) && routes <= kFrontMaxRoutes &&
           E <= kFrontMaxExperts && scratch <= (size_t)gp.num_stages * gp.slot_bytes;
}

bool build_state(LaunchState& st, const void* w13, const void* w13_scale, const void* w2,
                 const void* w2_scale, int T, int D, int I, int E, int K, void* base) {
    using namespace moe;
    moe_mxfp4_plan_t& pl = st.pl;
    GemmParams& gp = st.gp;
    shape_geometry(T, D, I, E, K, &pl, &gp);
    const WsPtrs ws = ws_ptrs(base, pl);
    gp.ws = ws;
    const StageGeom& q1 = gp.g[0];
    const StageGeom& q2 = gp.g[1];

    const int tr = pl.tile_rows;
    CUtensorMap* m = st.maps;
    bool ok = true;
    // D, I: the weights' widths; Dr, Ir: the widths the kernels run at
    const int Dr = gp.D, Ir = gp.I;
    // weight scales the maps read: the caller's, or their copy with rows of Dr/32
    // and Ir/32 bytes (made by the call's first launch)
    const void* s13 = w13_scale;
    const void* s2 = w2_scale;
    st.wscale13 = st.wscale2 = nullptr;
    if (gp.kt_boxes) {
        uint8_t* wsc = static_cast<uint8_t*>(base) + pl.offset[MOE_WS_WSCALE];
        s13 = wsc;
        s2 = wsc + round_up((size_t)E * 2 * I * (Dr / 32), kAlign);
        st.wscale13 = wsc;
        st.wscale2 = const_cast<void*>(s2);
    }
    // stage 1: A = 64 gate rows + the 64 up rows I rows further, both K-boxes of a stage
    if (gp.kt_boxes)
        ok = ok && make_kbox_map(&m[0], w13, (uint64_t)E * 2 * I, D, q1.kb, 64, 2, (uint64_t)I * (D / 2));
    else
        ok = ok && make_operand_map(&m[0], w13, (uint64_t)E * 2 * I, D, q1.kb, q1.nkt, 64, 2,
                                    (uint64_t)I * (D / 2));
    ok = ok && make_scale_map(&m[1], s13, (uint64_t)E * 2 * I, Dr / 32, 64, 2, (uint64_t)I);
    ok = ok && make_operand_map(&m[2], ws.a1q, pl.cap, Dr, q1.kb, q1.nkt, tr, 1, 0);
    ok = ok && make_map(&m[3], ws.a1s, pl.a1s_stride, pl.cap, pl.a1s_stride, 16, tr,
                        CU_TENSOR_MAP_SWIZZLE_NONE);
    // stage 2: A = 128 * mblocks rows of w2
    if (gp.kt_boxes)
        ok = ok && make_kbox_map(&m[4], w2, (uint64_t)E * D, I, q2.kb, 128 * q2.mblocks, 1, 0);
    else
        ok = ok && make_operand_map(&m[4], w2, (uint64_t)E * D, I, q2.kb, q2.nkt, 128 * q2.mblocks, 1, 0);
    ok = ok && make_scale_map(&m[5], s2, (uint64_t)E * D, Ir / 32, 128 * q2.mblocks, 1, 0);
    ok = ok && make_operand_map(&m[6], ws.a2q, pl.cap, Ir, q2.kb, q2.nkt, tr, 1, 0);
    ok = ok && make_map(&m[7], ws.a2s, pl.a2s_stride, pl.cap, pl.a2s_stride, 16, tr,
                        CU_TENSOR_MAP_SWIZZLE_NONE);
    return ok;
}

// Copy of the cached state for this configuration on device `dev` (built on a
// miss) into *out; false when a tensor map cannot be encoded.
bool launch_state(int dev, const void* w13, const void* w13_scale, const void* w2,
                  const void* w2_scale, int T, int D, int I, int E, int K, void* base,
                  LaunchState* out) {
    const void* kp[5] = {w13, w13_scale, w2, w2_scale, base};
    const int ks[7] = {T, D, I, E, K, g_force_tile_rows.load(), g_force_sf_copies.load()};
    std::lock_guard<std::mutex> lk(g_mu);
    for (int w = 0; w < kCacheWays; ++w) {
        const LaunchState& c = g_cache[dev][w];
        if (c.valid && memcmp(c.key_ptr, kp, sizeof(kp)) == 0 &&
            memcmp(c.key_shape, ks, sizeof(ks)) == 0) {
            *out = c;
            return true;
        }
    }
    LaunchState& st = g_cache[dev][g_cache_next[dev]];
    g_cache_next[dev] = (g_cache_next[dev] + 1) % kCacheWays;
    st.valid = false;
    if (!build_state(st, w13, w13_scale, w2, w2_scale, T, D, I, E, K, base)) return false;
    memcpy(st.key_ptr, kp, sizeof(kp));
    memcpy(st.key_shape, ks, sizeof(ks));
    st.valid = true;
    *out = st;
    return true;
}

}  // namespace

namespace moe {

moe_status_t forward_on_workspace(const void* hidden, const void* w13, const void* w13_scale,
                                  const void* w2, const void* w2_scale, const int32_t* topk_ids,
                                  const float* topk_weights, void* out, int T, int D, int I, int E,
                                  int K, int Dl, int Il, void* base, int dev, cudaStream_t stream) {
    LaunchState state;
    if (!launch_state(dev, w13, w13_scale, w2, w2_scale, T, D, I, E, K, base, &state))
        return MOE_ERR_CUDA;
    const LaunchState* st = &state;
    const moe_mxfp4_plan_t& pl = st->pl;
    const GemmParams& gp = st->gp;
    const WsPtrs& ws = gp.ws;

    // ---------------------------------------------------------- launches
    const int sms = num_sms(dev);
    const int n_counters = pl.max_tiles;
    Timing& tm = g_timing[dev];
    const bool timed = tm.enabled && tm.created;
    auto mark = [&](int i) {
        if (timed && (tm.mode == 1 || i == 0 || i == kNumKernels)) cudaEventRecord(tm.ev[i], stream);
    };
    // Single launch: routing and quantisation run inside the GEMM kernel (one
    // launch before the top-k sum); otherwise route -> quant -> GEMM.
    const bool front = single_launch_for(dev, T, E, K, gp);
    GemmParams g = gp;
    g.fused_front = front ? 1 : 0;
    g.topk_ids = topk_ids;
    g.topk_w = topk_weights;
    g.hidden = hidden;
    g.T = T;
    g.cap = pl.cap;
    g.Dl = Dl;
    g.Il = Il;
    if (front) g.ws.tile_done = ws.status + kFrontTileWord;  // zero between calls
    {
        std::lock_guard<std::mutex> lk(g_mu);
        g_last_ws[dev] = base;
    }
    // D, I: the weights' widths; Dr, Ir: the widths the kernels run at
    const int Dr = gp.D, Ir = gp.I;
    const int widen = gp.kt_boxes ? 1 : 0;
    const CallRange call_range(widen ? "run wider" : Dl != D || Il != I ? "padded" : "mxfp4", T, D, I, E, K,
                               widen + (front ? 2 : (T * K >= kRouteMultiMin ? 6 : 4)));
    if (widen) {
        const LaunchRange r("widen");
        if (launch_widen(w13_scale, st->wscale13, (long)E * 2 * I, D / 32, Dr / 32, w2_scale, st->wscale2,
                         (long)E * D, I / 32, Ir / 32, ws, Ir / 2, I / 2, pl.a2s_stride, I / 32, pl.cap,
                         sms * 4, stream) != cudaSuccess)
            return MOE_ERR_CUDA;
    }
    mark(0);
    if (!front) {
        const LaunchRange r("route");
        if (launch_route(topk_ids, topk_weights, T, K, E, pl.tile_rows, pl.cap, n_counters, ws,
                         stream) != cudaSuccess)
            return MOE_ERR_CUDA;
    }
    mark(1);
    if (!front) {
        const LaunchRange r("quant");
        if (launch_quant(hidden, T, K, Dr, Dl, pl.a1s_stride, pl.cap, ws, stream) != cudaSuccess)
            return MOE_ERR_CUDA;
    }
    mark(2);
    {
        const LaunchRange r(front ? "gemm (with routing and quantisation)" : "gemm");
        if (launch_gemm(st->maps, g, sms, stream) != cudaSuccess) return MOE_ERR_CUDA;
    }
    mark(3);
    {
        const LaunchRange r("topk_sum");
        if (launch_reduce(T, K, Dr, Dl, out, ws, stream) != cudaSuccess) return MOE_ERR_CUDA;
    }
    mark(4);
    if (timed) {
        tm.recorded = true;
        tm.launched = front ? 0xcu : 0xfu;
    }
    return MOE_OK;
}

size_t plan_workspace_bytes(int T, int D, int I, int E, int K) {
    moe_mxfp4_plan_t pl;
    fill_plan(T, D, I, E, K, &pl);
    return pl.workspace_bytes;
}

// Geometry of the bf16-activation GEMM kernel (gemm_w4a16.cu): ring slots of a
// raw weight tile and a route tile, two dequantised bf16 weight tiles, one
// epilogue group's exchange buffer, the route-tile cache.
static bool w4_geometry(W4Params& g, int D, int I, int tile_rows) {
    g.tile_rows = tile_rows;
    g.n_ftiles1 = I / 64;
    g.n_ftiles2 = D / 128;
    g.kstages1 = D / kW4Kc;
    g.kstages2 = I / kW4Kc;
    g.slot_bytes = (uint32_t)round_up(kW4RawBytes + (size_t)tile_rows * 256, 1024);
    auto slots_for = [&](int nb) {
        const uint32_t fixed = 1024u + (uint32_t)nb * kW4DeqBytes + 512u + (uint32_t)kXchgBytes +
                               (uint32_t)kTileCache * 16u;
        int n = (int)((uint32_t)kGemmSmemLimit - fixed) / (int)g.slot_bytes;
        return n > kMaxStages ? kMaxStages : n;
    };
    // a third dequantised tile where it leaves the ring at least four slots
    g.deq_bufs = slots_for(kW4MaxDeq) >= 4 ? kW4MaxDeq : 2;
    const int ns = slots_for(g.deq_bufs);
    if (ns < 2) return false;
    g.num_stages = ns;
    g.off_deq = (uint32_t)ns * g.slot_bytes;
    g.off_bar = g.off_deq + (uint32_t)g.deq_bufs * kW4DeqBytes;
    g.off_xchg = g.off_bar + 512u;
    g.off_tiles = g.off_xchg + (uint32_t)kXchgBytes;
    g.smem_bytes = g.off_tiles + (uint32_t)kTileCache * 16u + 1024u;
    g.acc_bufs = 4;
    uint32_t cols = 32;
    while (cols < (uint32_t)(g.acc_bufs * tile_rows)) cols <<= 1;
    g.tmem_cols = cols;
    return cols <= 512u && g.smem_bytes <= (uint32_t)kGemmSmemLimit;
}

moe_status_t forward_w4a16_on_workspace(const void* hidden, const void* w13, const void* w13_scale,
                                        const void* w2, const void* w2_scale,
                                        const int32_t* topk_ids, const float* topk_weights,
                                        void* out, int T, int D, int I, int E, int K, void* base,
                                        int dev, cudaStream_t stream) {
    moe_mxfp4_plan_t pl;
    fill_plan(T, D, I, E, K, &pl, true);
    W4Params g;
    memset(&g, 0, sizeof(g));
    g.ws = ws_ptrs(base, pl);
    g.w13_scale = static_cast<const uint8_t*>(w13_scale);
    g.w2_scale = static_cast<const uint8_t*>(w2_scale);
    g.D = D; g.I = I; g.E = E; g.K = K; g.R = T * K;
    if (!w4_geometry(g, D, I, pl.tile_rows)) return MOE_ERR_UNSUPPORTED_SHAPE;
    const int tr = pl.tile_rows;
    CUtensorMap maps[4];
    bool ok = true;
    // raw e2m1 weights, 64 bytes (128 K elements) x 64 rows (stage 1) / 128 rows (stage 2)
    ok = ok && make_map(&maps[0], w13, (uint64_t)D / 2, (uint64_t)E * 2 * I, (uint64_t)D / 2, 64, 64,
                        CU_TENSOR_MAP_SWIZZLE_NONE);
    ok = ok && make_map(&maps[2], w2, (uint64_t)I / 2, (uint64_t)E * D, (uint64_t)I / 2, 64, 128,
                        CU_TENSOR_MAP_SWIZZLE_NONE);
    // bf16 route tiles seen as {128 bytes, rows, K-boxes}: 2 K-boxes of 64 bf16 per stage
    {
        const uint64_t dims1[3] = {128, (uint64_t)pl.cap, (uint64_t)D * 2 / 128};
        const uint64_t str1[2] = {(uint64_t)D * 2, 128};
        const uint64_t dims2[3] = {128, (uint64_t)pl.cap, (uint64_t)I * 2 / 128};
        const uint64_t str2[2] = {(uint64_t)I * 2, 128};
        const uint32_t box[3] = {128, (uint32_t)tr, 2};
        ok = ok && make_map_nd(&maps[1], g.ws.a1b, 3, dims1, str1, box, CU_TENSOR_MAP_SWIZZLE_128B);
        ok = ok && make_map_nd(&maps[3], g.ws.a2b, 3, dims2, str2, box, CU_TENSOR_MAP_SWIZZLE_128B);
    }
    if (!ok) return MOE_ERR_CUDA;

    const int sms = num_sms(dev);
    Timing& tm = g_timing[dev];
    const bool timed = tm.enabled && tm.created;
    auto mark = [&](int i) {
        if (timed && (tm.mode == 1 || i == 0 || i == kNumKernels)) cudaEventRecord(tm.ev[i], stream);
    };
    const CallRange call_range("w4a16", T, D, I, E, K, T * K >= kRouteMultiMin ? 6 : 4);
    mark(0);
    {
        const LaunchRange r("route");
        if (launch_route(topk_ids, topk_weights, T, K, E, tr, pl.cap, pl.max_tiles, g.ws, stream) != cudaSuccess)
            return MOE_ERR_CUDA;
    }
    mark(1);
    {
        const LaunchRange r("gather_bf16");
        if (launch_gather_bf16(hidden, T, K, D, g.ws, stream) != cudaSuccess) return MOE_ERR_CUDA;
    }
    mark(2);
    {
        const LaunchRange r("gemm_w4a16");
        if (launch_w4a16_gemm(maps, g, sms, stream) != cudaSuccess) return MOE_ERR_CUDA;
    }
    mark(3);
    {
        const LaunchRange r("topk_sum");
        if (launch_reduce(T, K, D, D, out, g.ws, stream) != cudaSuccess) return MOE_ERR_CUDA;
    }
    mark(4);
    if (timed) {
        tm.recorded = true;
        tm.launched = 0xfu;
    }
    {
        std::lock_guard<std::mutex> lk(g_mu);
        g_last_ws[dev] = base;
    }
    return MOE_OK;
}

}  // namespace moe

extern "C" {

moe_status_t moe_mxfp4_forward(const void* hidden, const void* w13, const void* w13_scale,
                               const void* w2, const void* w2_scale, const int32_t* topk_ids,
                               const float* topk_weights, void* out, int T, int d_model,
                               int d_inter, int E, int topk, cudaStream_t stream) {
    return moe_mxfp4_forward_padded(hidden, w13, w13_scale, w2, w2_scale, topk_ids, topk_weights,
                                    out, T, d_model, d_inter, d_model, d_inter, E, topk, stream);
}

moe_status_t moe_mxfp4_forward_padded(const void* hidden, const void* w13, const void* w13_scale,
                                      const void* w2, const void* w2_scale,
                                      const int32_t* topk_ids, const float* topk_weights,
                                      void* out, int T, int d_model, int d_inter,
                                      int d_model_pad, int d_inter_pad, int E, int topk,
                                      cudaStream_t stream) {
    const int D = d_model_pad, I = d_inter_pad, K = topk;
    moe_status_t st = validate_forward(hidden, w13, w13_scale, w2, w2_scale, topk_ids,
                                       topk_weights, out, T, D, I, E, K);
    if (st == MOE_OK) st = validate_padded(D, I, d_model, d_inter);
    // padded storage: widths the kernels run at as they are
    if (st == MOE_OK && (d_model != D || d_inter != I) && widened(D, I)) st = MOE_ERR_UNSUPPORTED_SHAPE;
    if (st != MOE_OK || T == 0) return st;
    const size_t need = plan_workspace_bytes(T, D, I, E, K);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
    void* base;
    size_t ws_bytes;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        base = g_ws[dev].ptr;
        ws_bytes = g_ws[dev].bytes;
    }
    if (!base || ws_bytes < need) return MOE_ERR_WORKSPACE;
    return forward_on_workspace(hidden, w13, w13_scale, w2, w2_scale, topk_ids, topk_weights, out,
                                T, D, I, E, K, d_model, d_inter, base, dev, stream);
}

moe_status_t moe_mxfp4_check_wait_timeout(uint32_t limit_us, cudaStream_t stream) {
    if (limit_us == 0 || limit_us > 1000000u) return MOE_ERR_INVALID_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
    void* base;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        base = g_ws[dev].ptr;
    }
    if (!base) return MOE_ERR_WORKSPACE;
    if (launch_check_wait(static_cast<uint32_t*>(base), (uint64_t)limit_us * 1000u, stream) !=
        cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}

int moe_mxfp4_num_kernels(void) { return kNumKernels; }

int moe_mxfp4_call_launches(int T, int d_model, int d_inter, int E, int topk) {
    if (validate_shape(T, d_model, d_inter, E, topk) != MOE_OK) return -1;
    if (T == 0) return 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    moe_mxfp4_plan_t pl;
    moe::GemmParams gp;
    shape_geometry(T, d_model, d_inter, E, topk, &pl, &gp);
    const int widen = gp.kt_boxes ? 1 : 0;  // the weight-scale copy first
    if (single_launch_for(dev, T, E, topk, gp)) return widen + 2;
    return widen + ((long long)T * topk >= kRouteMultiMin ? 6 : 4);  // routing in three launches
}

moe_status_t moe_mxfp4_get_gemm_config(int T, int d_model, int d_inter, int E, int topk,
                                       moe_mxfp4_gemm_config_t* cfg) {
    if (!cfg) return MOE_ERR_INVALID_ARG;
    const moe_status_t st = validate_shape(T, d_model, d_inter, E, topk);
    if (st != MOE_OK) return st;
    moe_mxfp4_plan_t pl;
    moe::GemmParams gp;
    shape_geometry(T, d_model, d_inter, E, topk, &pl, &gp);
    cfg->tile_rows = gp.tile_rows;
    cfg->stage1_k = gp.g[0].kstage_elems;
    cfg->stage2_k = gp.g[1].kstage_elems;
    cfg->stage2_blocks = gp.g[1].mblocks;
    cfg->num_stages = gp.num_stages;
    cfg->mma_warps = gp.mma_warps;
    cfg->acc_bufs = gp.acc_bufs;
    cfg->epi_groups = gp.epi_groups;
    cfg->sf_by_layout_warp = gp.sf_by_layout_warp;
    cfg->wide_sf = gp.wide_sf;
    cfg->lookahead = gp.lookahead;
    cfg->slot_bytes = gp.slot_bytes;
    cfg->smem_bytes = gp.smem_bytes;
    cfg->smem_limit = (unsigned)kGemmSmemLimit;
    cfg->acc_cols = gp.acc_cols;
    cfg->sf_col0 = gp.sf_col0;
    cfg->sf_cols = gp.sf_cols;
    cfg->tmem_cols = gp.tmem_cols;
    return MOE_OK;
}

moe_status_t moe_mxfp4_get_plan_w4a16(int T, int d_model, int d_inter, int E, int topk,
                                      moe_mxfp4_plan_t* plan) {
    if (!plan) return MOE_ERR_INVALID_ARG;
    moe_status_t st = validate_shape(T, d_model, d_inter, E, topk);
    if (st == MOE_OK && widened(d_model, d_inter)) st = MOE_ERR_UNSUPPORTED_SHAPE;  // native widths only
    if (st != MOE_OK) return st;
    fill_plan(T, d_model, d_inter, E, topk, plan, true);
    return MOE_OK;
}

size_t moe_mxfp4_workspace_size_w4a16(int T, int d_model, int d_inter, int E, int topk) {
    moe_mxfp4_plan_t pl;
    if (moe_mxfp4_get_plan_w4a16(T, d_model, d_inter, E, topk, &pl) != MOE_OK) return 0;
    return pl.workspace_bytes;
}

moe_status_t moe_mxfp4_forward_w4a16(const void* hidden, const void* w13, const void* w13_scale,
                                     const void* w2, const void* w2_scale,
                                     const int32_t* topk_ids, const float* topk_weights,
                                     void* out, int T, int d_model, int d_inter, int E, int topk,
                                     cudaStream_t stream) {
    const int D = d_model, I = d_inter, K = topk;
    moe_status_t st = validate_forward(hidden, w13, w13_scale, w2, w2_scale, topk_ids,
                                       topk_weights, out, T, D, I, E, K);
    if (st == MOE_OK && widened(D, I)) st = MOE_ERR_UNSUPPORTED_SHAPE;  // native widths only
    if (st != MOE_OK || T == 0) return st;
    const size_t need = moe_mxfp4_workspace_size_w4a16(T, D, I, E, K);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
    void* base;
    size_t ws_bytes;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        base = g_ws[dev].ptr;
        ws_bytes = g_ws[dev].bytes;
    }
    if (!base || ws_bytes < need) return MOE_ERR_WORKSPACE;
    return moe::forward_w4a16_on_workspace(hidden, w13, w13_scale, w2, w2_scale, topk_ids,
                                           topk_weights, out, T, D, I, E, K, base, dev, stream);
}

moe_status_t moe_mxfp4_set_single_launch(int mode) {
    if (mode < 0 || mode > 2) return MOE_ERR_INVALID_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
    g_single_launch[dev] = mode;
    g_single_set[dev] = true;
    return MOE_OK;
}

moe_status_t moe_mxfp4_tensor_probe(int n, int iters, int copies_per_mma, int variant,
                                    double* flops, cudaStream_t stream) {
    if (n < 16 || n > 256 || n % 16 != 0 || iters < 1 || iters > 10000000 || copies_per_mma < 0 ||
        copies_per_mma > 8 || variant < 0 || variant > 63 || !flops)
        return MOE_ERR_INVALID_ARG;
    if (n << ((variant >> 2) & 3) > 256) return MOE_ERR_INVALID_ARG;  // accumulators fit in 256 columns
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
    void* base;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        base = g_ws[dev].ptr;
        if (base) g_last_ws[dev] = base;
    }
    if (!base) return MOE_ERR_WORKSPACE;
    const int grid = num_sms(dev);
    if (launch_mxf4_probe(n, iters, copies_per_mma, variant, grid, static_cast<uint32_t*>(base), stream) !=
        cudaSuccess)
        return MOE_ERR_CUDA;
    *flops = 2.0 * 128.0 * (double)n * 64.0 * (double)iters * (double)grid;
    return MOE_OK;
}

moe_status_t moe_mxfp4_set_tuning(int tile_rows, int sf_copies) {
    if (!(tile_rows == 0 || tile_rows == 16 || tile_rows == 32 || tile_rows == 64 || tile_rows == 128))
        return MOE_ERR_INVALID_ARG;
    if (sf_copies < 0 || sf_copies > 4) return MOE_ERR_INVALID_ARG;
    g_force_tile_rows.store(tile_rows);
    g_force_sf_copies.store(sf_copies);
    return MOE_OK;
}

moe_status_t moe_mxfp4_set_nvtx(int on) {
    if (on != 0 && on != 1) return MOE_ERR_INVALID_ARG;
    g_nvtx.store(on, std::memory_order_relaxed);
    return MOE_OK;
}

moe_status_t moe_mxfp4_set_kernel_timing(int mode) {
    if (mode < 0 || mode > 2) return MOE_ERR_INVALID_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    Timing& tm = g_timing[dev];
    if (mode && !tm.created) {
        for (int i = 0; i <= kNumKernels; ++i)
            if (cudaEventCreate(&tm.ev[i]) != cudaSuccess) return MOE_ERR_CUDA;
        tm.created = true;
    }
    tm.mode = mode;
    tm.enabled = mode != 0;
    tm.recorded = false;
    return MOE_OK;
}

float moe_mxfp4_last_call_ms(void) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1.f;
    Timing& tm = g_timing[dev];
    if (!tm.enabled || !tm.recorded) return -1.f;
    if (cudaEventSynchronize(tm.ev[kNumKernels]) != cudaSuccess) return -1.f;
    float t = -1.f;
    if (cudaEventElapsedTime(&t, tm.ev[0], tm.ev[kNumKernels]) != cudaSuccess) return -1.f;
    return t;
}

int moe_mxfp4_kernel_times(float* ms, int n) {
    int dev = 0;
    if (!ms || cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    Timing& tm = g_timing[dev];
    if (!tm.enabled || !tm.recorded || tm.mode != 1) return -1;
    if (cudaEventSynchronize(tm.ev[kNumKernels]) != cudaSuccess) return -1;
    const int m = n < kNumKernels ? n : kNumKernels;
    for (int i = 0; i < m; ++i) {
        float t = 0.f;
        if (!((tm.launched >> i) & 1u)) {
            ms[i] = -1.f;  // nothing ran in this slot
            continue;
        }
        if (cudaEventElapsedTime(&t, tm.ev[i], tm.ev[i + 1]) != cudaSuccess) return -1;
        ms[i] = t;
    }
    return m;
}

}  // extern "C"
