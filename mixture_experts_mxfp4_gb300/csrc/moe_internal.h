// Internal declarations shared by the library's translation units: the
// workspace pointer set, the GEMM launch parameters and the kernel launchers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/moe_mxfp4.h"

namespace moe {

// Device pointers into the caller's workspace (see moe_mxfp4_plan_t).
struct WsPtrs {
    uint32_t* status;      // [kStatusWords]: [0] error bits, [15] single-launch ready word, ...
    uint32_t* counters;    // [max_tiles]: route-tile counters of the multi-kernel path
    int32_t* sorted_ids;   // [cap]
    float* sorted_w;       // [cap]
    int32_t* block_expert; // [cap / block_m]
    int32_t* seg_start;    // [E + 1]
    int32_t* route_pos;    // [R]
    int32_t* num_valid;    // [4]
    int4* tiles;           // [max_tiles]: {expert, first slot, rows, 0}
    uint8_t* a1q;          // [cap][D/2]
    uint8_t* a1s;          // [cap][a1s_stride]
    uint8_t* a2q;          // [cap][I/2]
    uint8_t* a2s;          // [cap][a2s_stride]
    float* P;              // [R][D]: w[route] * stage-2 output of each route, by route id
    uint32_t* tile_done;   // stage-1 feature tiles completed per route tile (counters, or the
                           // status region's block on the single-launch path)
    uint32_t* quant_done;  // CTAs whose share of the hidden states is quantised (single launch)
    uint16_t* a1b;         // bf16-activation path: [cap][D] hidden rows in sorted order
    uint16_t* a2b;         // bf16-activation path: [cap][I] bf16 SwiGLU output in sorted order
};

// Geometry of one grouped block-scaled GEMM stage (stage 1: gate_up, K = D;
// stage 2: down, K = I) inside the fused GEMM kernel.
struct StageGeom {
    int n_ftiles;       // stage 1: I / 64 feature tiles; stage 2: D / (128 * mblocks) output tiles
    int kstages;        // K / kstage_elems
    int kstage_elems;   // K elements per pipeline stage: 128, 256 or 512
    int kb;             // bytes per row of one TMA box along K: 64 or 128
    int nkt;            // TMA boxes along K per stage (kstage_elems / 2 / kb)
    int natoms;         // 128-element scale chunks per stage (kstage_elems / 128)
    int sr_a;           // bytes per raw weight-scale row in shared memory: 4, 8 or 16
    int a_scale_small;  // weight scales read through a [rows*S/16, 16] view
    int b_scale_x;      // 1 when activation scales advance 16 bytes per stage
    int mblocks;        // 128-row weight blocks per item sharing one route tile
    uint32_t off_b, off_sa, off_sb;  // route tile and raw scale tiles within a ring slot (A at 0)
};

// Parameters of the fused GEMM launch: every CTA runs its stage-1 items, then
// its stage-2 items, through one shared-memory ring.
struct GemmParams {
    WsPtrs ws;
    int D, I, E, K, R;  // D, I: widths the kernels run at (native widths, >= Dw, Iw)
    int Dl, Il;         // logical d_model, d_inter (multiples of 32, <= Dw, Iw)
    int Dw, Iw;         // widths of the weight tensors: w13 [E][2 Iw][Dw/2], w2 [E][Dw][Iw/2]
    int kt_boxes;       // weights narrower than D or I: one copy per K box of a stage, the
                        // columns past Dw / Iw zero-filled by the copy (maps of the weights'
                        // own widths; generic instantiations only); weight scales repacked
                        // to D/32, I/32 bytes per row
    int tile_rows;      // maximum MMA N (routes per tile), multiple of 16, <= 128
    StageGeom g[2];     // stage 1, stage 2
    int num_stages;     // shared-memory ring depth
    int mma_warps;      // MMA-issuing warps (1 or 2); warp w takes the CTA's stages g % mma_warps == w
    int acc_bufs;       // TMEM accumulator buffers (items in flight between MMA and epilogue)
    int lookahead;      // MMA warps copy the next stage's scale factors early (needs ns % mma_warps == 0)
    int sf_by_layout_warp;  // the scale-layout warp also copies the scale factors to TMEM (one MMA warp)
    uint32_t slot_bytes;  // bytes per ring slot (the larger stage layout)
    uint32_t acc_cols;    // TMEM columns per accumulator buffer
    uint32_t sf_cols;     // TMEM scale-factor columns per ring slot
    uint32_t tmem_cols;   // TMEM columns allocated
    uint32_t sf_col0;     // first TMEM column of the per-slot scale-factor regions
    uint32_t off_bar, off_xchg, off_tiles;  // barriers, epilogue exchange buffer, tile cache
    uint32_t smem_bytes;                    // dynamic shared memory requested
    // Two-atom scale-factor copies (tcgen05.cp .128x256b) from two staging buffers
    // of sfw_bytes at off_sfw, for the phases whose stages hold an even number of
    // 128-element chunks; otherwise one-atom copies from the ring slot.
    int wide_sf;
    uint32_t off_sfw, sfw_bytes;
    int epi_groups;  // epilogue groups of four warps (2 or 3): 128 + 128 * epi_groups threads
    int a2s_stride;
    int a1s_stride;
    // Routing and quantisation inside the GEMM kernel (fused_front = 1, few
    // routes): the inputs and the sorted-slot capacity.
    int fused_front;
    const int32_t* topk_ids;
    const float* topk_w;
    const void* hidden;
    int T, cap;
};

// Parameters of the bf16-activation (W4A16) GEMM launch: packed e2m1 weights
// with e8m0 scales, bf16 activations, both stages in one persistent launch.
// Stage K chunks of 128 elements; weights dequantised to bf16 in shared memory.
struct W4Params {
    WsPtrs ws;
    const uint8_t* w13_scale;  // [E][2I][D/32]
    const uint8_t* w2_scale;   // [E][D][I/32]
    int D, I, E, K, R;
    int tile_rows;             // routes per tile (MMA N), multiple of 16, <= 128
    int n_ftiles1, n_ftiles2;  // stage 1: I / 64; stage 2: D / 128
    int kstages1, kstages2;    // D / 128, I / 128
    int num_stages;            // TMA ring depth (raw weight tile + route tile per slot)
    int acc_bufs;              // TMEM accumulators
    int deq_bufs;              // dequantised bf16 weight tiles (2 or 3)
    uint32_t slot_bytes;       // raw weights (8 KB) + route tile (tile_rows x 256 B)
    uint32_t off_deq;          // the dequantised tiles (32 KB each, 1024-aligned)
    uint32_t off_bar, off_xchg, off_tiles, smem_bytes;
    uint32_t tmem_cols;
};
constexpr int kW4Kc = 128;                 // K elements per stage
constexpr int kW4Threads = 512;            // 16 warps: producer, MMA, TMEM, -, 4 epilogue, 8 dequantisation
constexpr uint32_t kW4RawBytes = 128 * 64;  // 128 weight rows x 64 bytes of e2m1
constexpr uint32_t kW4DeqBytes = 128 * 256; // 128 rows x 128 bf16
constexpr int kW4MaxDeq = 3;

// Status region (u32 words): [0] error bits, [1..14] spare, [15] ready word of
// the single-launch path, [16] its quantisation count, [17] its count of exited
// CTAs, [512, 1024) its route-tile counters.  Words 15.. are zero between calls:
// the region is zero when the workspace is first used and the last CTA of every
// single-launch GEMM kernel clears them before it exits.
constexpr int kStatusWords = 1024;
constexpr int kFrontQuantWord = 16;
constexpr int kFrontExitWord = 17;
constexpr int kFrontTileWord = 512;

constexpr int kBlockM = 16;          // slots per padded block
// 12 warps: producer, MMA, second MMA / TMEM owner, scale layout, 2 x 4 epilogue
// (the single-launch front end assumes this layout)
constexpr int kGemmThreads = 384;
constexpr int kEpiGroups = 2;
// 128-route tiles whose stage-2 items are one stage long (prefill-like: d_inter
// 256) run a third epilogue group (16 warps): there the stage-2 epilogue bounds
// the kernel (measured prefill T=4096 804 -> 728 us; dense T=512 and decode
// shapes were slower with it, so they keep two).  Not with the single-launch
// front end, which assumes two.
constexpr int kMaxEpiGroups = 3;
constexpr int kXchgBytes = 4352;     // per epilogue group: 4 KB exchange + flag
constexpr int kMaxStages = 8;
constexpr int kGemmSmemLimit = 227 * 1024;  // dynamic shared memory limit set on the GEMMs
constexpr int kMaxAccBufs = 4;
constexpr int kFrontMaxRoutes = 2048;  // single-launch path: routes (position table in the exchange buffer)
constexpr int kFrontMaxExperts = 384;  // single-launch path: one expert per GEMM thread
constexpr int kFrontAutoRoutes = 256;  // automatic mode: single launch up to this many routes
constexpr int kRouteMultiMin = 4096;  // routes from which routing runs in three launches on many CTAs
constexpr int kTileCache = 512;      // route tiles kept in shared memory (the rest read from L2)
// Byte offsets, within the GEMM kernel's 512-byte barrier block, of the
// producer's bitmap of route tiles known to be complete (kTileCache bits) and of
// the two staging-buffer barriers of the scale-factor copies.
constexpr int kReadyBitsOff = 384;
constexpr int kSbufBarOff = kReadyBitsOff + kTileCache / 8;
static_assert(kSbufBarOff + 16 <= 512, "barrier block");

// Host-side pieces of the forward call shared by its entry points (api.cu).
moe_status_t validate_forward(const void* hidden, const void* w13, const void* w13_scale,
                              const void* w2, const void* w2_scale, const int32_t* topk_ids,
                              const float* topk_weights, const void* out, int T, int D, int I,
                              int E, int K);
size_t plan_workspace_bytes(int T, int D, int I, int E, int K);
// D, I: stored (padded) sizes; Dl, Il: logical sizes.
moe_status_t validate_padded(int D, int I, int Dl, int Il);
moe_status_t forward_on_workspace(const void* hidden, const void* w13, const void* w13_scale,
                                  const void* w2, const void* w2_scale, const int32_t* topk_ids,
                                  const float* topk_weights, void* out, int T, int D, int I, int E,
                                  int K, int Dl, int Il, void* base, int dev, cudaStream_t stream);

cudaError_t launch_check_wait(uint32_t* status, uint64_t limit_ns, cudaStream_t stream);
// Weights narrower than the widths the kernels run at: weight-scale rows of S
// bytes copied to rows of Sp bytes (extra bytes 127), and the intermediate's
// columns past the weights' width zeroed (a2q bytes [q_from, q_row), a2s bytes
// [s_from, s_row) of each of the cap slots).
cudaError_t launch_widen(const void* w13_scale, void* d13, long rows13, int S13, int Sp13, const void* w2_scale,
                         void* d2, long rows2, int S2, int Sp2, const WsPtrs& ws, int q_row, int q_from,
                         int s_row, int s_from, long cap, int grid, cudaStream_t stream);
cudaError_t launch_route(const int32_t* topk_ids, const float* topk_w, int T, int K, int E,
                         int tile_rows, int cap, int n_counters, const WsPtrs& ws,
                         cudaStream_t stream);
// hidden rows hold Dl elements; quantised rows D (zero blocks past Dl)
cudaError_t launch_quant(const void* hidden, int T, int K, int D, int Dl, int a1s_stride, int cap,
                         const WsPtrs& ws, cudaStream_t stream);
// Top-k sum: P rows by route id hold D columns, out rows Dl; a route counts where
// route_pos >= 0 (its expert id is in [0, E)).
cudaError_t launch_reduce(int T, int K, int D, int Dl, void* out, const WsPtrs& ws,
                          cudaStream_t stream);
// bf16-activation path: copy each token's hidden row to the sorted slot of
// every valid route (after the routing kernel)
cudaError_t launch_gather_bf16(const void* hidden, int T, int K, int D, const WsPtrs& ws,
                               cudaStream_t stream);
// maps: raw w13 (64 B x 64 rows), a1b route tiles, raw w2 (64 B x 128 rows), a2b route tiles
cudaError_t launch_w4a16_gemm(const CUtensorMap* maps, const W4Params& p, int grid,
                              cudaStream_t stream);
// maps: stage-1 A, SA, B, SB, then stage-2 A, SA, B, SB
cudaError_t launch_gemm(const CUtensorMap* maps, const GemmParams& p, int grid,
                        cudaStream_t stream);
// Tensor-core throughput probe (probe.cu): grid CTAs, each issuing `iters`
// M = 128, N = n, K = 64 mxf4 MMAs and copies_per_mma scale-factor copies per MMA
// (variant bit 0: 128x256b copies; bit 1: copies from a second warp).
cudaError_t launch_mxf4_probe(int n, int iters, int copies_per_mma, int variant, int grid,
                              uint32_t* status, cudaStream_t stream);

}  // namespace moe
