/*
 * moe_mxfp4.h -- C ABI of the fused MXFP4 Mixture-of-Experts forward for
 * NVIDIA GB300 (sm_103a).
 *
 * The operation (sources are the web pages this library restates):
 *   kernelbot-amd-moe-mxfp4-754773, flower_moe.py, custom_kernel: sort routes
 *     by expert -> MXFP4-quantise the hidden states -> stage-1 grouped GEMM with
 *     SiLU(gate)*up -> MXFP4-requantise the bf16 intermediate -> stage-2 grouped
 *     GEMM whose rows are scaled by the top-k weights and summed per token.
 *   kernelbot-amd-moe-mxfp4-723815, solution.py, fused_moe_mxfp4 / _dequant /
 *     kernel_stage1 / kernel_stage2: tensor layouts, e2m1 and e8m0 decoding,
 *     nibble order, gate rows before up rows, weight applied after the down GEMM.
 *
 * Formats: an e2m1 element is 4 bits (sign, 2 exponent bits with bias 1, 1
 * mantissa bit); two elements per byte, element 2j in the low nibble of byte j.
 * An e8m0 scale byte s means 2^(s-127); one scale per 32 consecutive elements
 * along the contraction (K) dimension of a row.
 *
 * Ownership and threading: every pointer argument is owned by the caller and
 * is device memory, except that the per-call buffers of the forward entry
 * points (hidden, topk_ids, topk_weights, out) may instead be pinned host
 * memory mapped into the device's address space (cudaHostAlloc, or
 * cudaHostRegister with cudaHostRegisterMapped, on a system with unified
 * addressing): the kernels then read the inputs and write the output in place
 * (on GB300 over NVLink-C2C) and no staging copy is made.  Weights, scales and
 * the workspace must be device memory (tensor-memory-access copies read them).
 * Pageable host memory is not supported (not checked).
 * Inputs are only read; the library never allocates on the call path.  The scratch it needs is a caller-owned device buffer registered with
 * moe_mxfp4_set_workspace (one per device; calls that share it must be ordered
 * on the GPU, e.g. issued to one stream).  All work is enqueued on `stream`; the
 * call returns after enqueueing.
 *
 * Error behaviour: argument and shape errors are detected on the host before
 * any work is enqueued and returned as a status code (nothing is launched).
 * Launch failures return MOE_ERR_CUDA.  Errors found on the device (a bounded
 * wait that ran out) are recorded in the workspace and reported by
 * moe_mxfp4_last_device_status.
 */
#ifndef MOE_MXFP4_H
#define MOE_MXFP4_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,       /* null pointer, negative size, topk/E out of range   */
    MOE_ERR_UNSUPPORTED_SHAPE = 2, /* d_model / d_inter not a supported multiple        */
    MOE_ERR_MISALIGNED = 3,        /* a pointer is not 16-byte aligned                    */
    MOE_ERR_WORKSPACE = 4,         /* no workspace registered, or too small               */
    MOE_ERR_CUDA = 5,              /* a CUDA runtime/driver call failed                   */
    MOE_ERR_DEVICE_TIMEOUT = 6     /* a bounded device-side wait ran out (see status)     */
} moe_status_t;

/*
 * Supported shapes: T >= 0; 1 <= topk <= 16; 1 <= E <= 1024;
 * d_model a multiple of 128 and d_inter a multiple of 64 (MOE_ERR_UNSUPPORTED_SHAPE
 * otherwise).  The kernels run each width at 128, 256 or a multiple of 512: a
 * width that is none of these runs at the next one.  Such a call adds one launch
 * that copies the weight scales into the workspace (region MOE_WS_WSCALE, rows
 * padded to 16-byte multiples for the tensor-memory-access copies) and zeroes
 * the intermediate's extra columns; the kernels read the weights' missing
 * columns as zeros.  The bf16-activation forward takes only the widths 128, 256
 * and multiples of 512.
 * Every pointer 16-byte aligned.
 */

/* Bytes of workspace one forward call of this shape needs (0 when the shape is
 * not supported).  Depends only on the shape. */
size_t moe_mxfp4_workspace_size(int T, int d_model, int d_inter, int E, int topk);

/*
 * Register the caller-owned device workspace for the current CUDA device.
 * dev_ptr must be 256-byte aligned; bytes its size (at least 4096).  Passing
 * NULL unregisters.  The library keeps the pointer, never frees it, and does
 * no device work here (registering the same buffer again is free).  Not
 * thread-safe with concurrent forward calls on the same device.
 * The first 4096 bytes (region MOE_WS_STATUS) must be zero when a buffer is
 * first used (e.g. allocate it zero-filled or cudaMemset it); the forward
 * calls keep them so.  The rest needs no initialisation.  A kernel that finds
 * a counter there already past its target reports MOE_ERR_DEVICE_TIMEOUT
 * through moe_mxfp4_last_device_status (status bit 8).
 */
moe_status_t moe_mxfp4_set_workspace(void* dev_ptr, size_t bytes);

/*
 * Fused MXFP4 MoE forward.
 *   hidden        bf16 [T, d_model], row-major
 *   w13           u8   [E, 2*d_inter, d_model/2]: packed e2m1, rows [0, d_inter) gate,
 *                      rows [d_inter, 2*d_inter) up (solution.py: W_gate / W_up split)
 *   w13_scale     u8   [E, 2*d_inter, d_model/32]: e8m0
 *   w2            u8   [E, d_model, d_inter/2]: packed e2m1
 *   w2_scale      u8   [E, d_model, d_inter/32]: e8m0
 *   topk_ids      i32  [T, topk]: expert ids; ids outside [0, E) contribute nothing
 *   topk_weights  f32  [T, topk]: multiplies the stage-2 output of that route
 *   out           bf16 [T, d_model]: fully overwritten:
 *                 out[t] = bf16( sum_k w[t,k] * W2[e] . Q( bf16( silu(W13g[e] . Q(x_t))
 *                                                        * (W13u[e] . Q(x_t)) ) ) )
 *                 with Q the MX quantiser (shared exponent floor(log2 amax) - 2,
 *                 round to nearest even, saturate at 6), fp32 accumulation, and the
 *                 sum over k in ascending order (deterministic).
 * hidden, topk_ids, topk_weights and out: device memory or mapped pinned host
 * memory (see Ownership above).
 * Asynchronous on `stream`.  T == 0 returns MOE_OK and enqueues nothing.
 */
moe_status_t moe_mxfp4_forward(const void* hidden, const void* w13, const void* w13_scale,
                               const void* w2, const void* w2_scale, const int32_t* topk_ids,
                               const float* topk_weights, void* out, int T, int d_model,
                               int d_inter, int E, int topk, cudaStream_t stream);

/*
 * Forward with padded weight storage (the d_hidden_pad / d_expert_pad of
 * solution.py's _Cfg and flower_moe.py's custom_kernel: weights stored with
 * padded dimensions, activations and output with the logical ones).
 *   hidden   bf16 [T, d_model];  out bf16 [T, d_model]
 *   w13      u8 [E, 2*d_inter_pad, d_model_pad/2], rows [0, d_inter_pad) gate,
 *            [d_inter_pad, 2*d_inter_pad) up; w13_scale u8 [E, 2*d_inter_pad, d_model_pad/32]
 *   w2       u8 [E, d_model_pad, d_inter_pad/2];  w2_scale u8 [E, d_model_pad, d_inter_pad/32]
 * The result is the forward of the logical problem: the weights' first d_inter
 * gate rows, first d_inter up rows, first d_model columns (w13) and the first
 * d_model rows and d_inter columns (w2).  d_model, d_inter: multiples of 32 (one
 * scale block), at most the padded sizes; the padded sizes 128, 256 or a
 * multiple of 512 (where they differ from d_model, d_inter).  The padding may hold any e2m1 codes but no scale byte 255
 * (NaN): it is multiplied by zeros.  The workspace is that of the padded shape
 * (moe_mxfp4_workspace_size(T, d_model_pad, d_inter_pad, E, topk)).
 * moe_mxfp4_forward(..., d_model, d_inter, ...) is this call with no padding.
 */
moe_status_t moe_mxfp4_forward_padded(const void* hidden, const void* w13, const void* w13_scale,
                                      const void* w2, const void* w2_scale,
                                      const int32_t* topk_ids, const float* topk_weights,
                                      void* out, int T, int d_model, int d_inter,
                                      int d_model_pad, int d_inter_pad, int E, int topk,
                                      cudaStream_t stream);

/*
 * Forward with bf16 activations (W4A16): the weights as for moe_mxfp4_forward,
 * but the hidden states are not quantised and the SwiGLU output stays bf16
 * (b12x moe/fused/w4a16/kernel.py, W4A16GemmKernel; flower_moe.py's
 * bf16-activation path; solution.py, _reference_forward):
 *   out[t] = bf16( sum_k w[t,k] * W2[e] . bf16( silu(W13g[e] . x_t) * (W13u[e] . x_t) ) )
 * with x_t the bf16 hidden row, W = e2m1 * 2^(s-127) and fp32 accumulation.  The
 * weights are expanded to bf16 in shared memory for bf16 tensor-core MMAs.  Same
 * arguments, shapes and errors as moe_mxfp4_forward; the registered workspace
 * must hold moe_mxfp4_workspace_size_w4a16 bytes (its layout:
 * moe_mxfp4_get_plan_w4a16).  Launches: routing (one kernel, or three from 4096
 * routes), row gather, GEMM kernel, top-k sum.
 */
moe_status_t moe_mxfp4_forward_w4a16(const void* hidden, const void* w13, const void* w13_scale,
                                     const void* w2, const void* w2_scale,
                                     const int32_t* topk_ids, const float* topk_weights,
                                     void* out, int T, int d_model, int d_inter, int E, int topk,
                                     cudaStream_t stream);

/*
 * Forward without any device allocation, for callers that cannot allocate.
 * (This entry point has no counterpart in the pages; it is a deployment aid.)
 *
 * Some callers cannot call cudaMalloc when they run this layer: a serving
 * runtime that has handed all free device memory to its own pool (cudaMalloc
 * then fails), a plugin host that forbids plugins to allocate, or a latency-
 * critical loop that must avoid cudaMalloc's implicit synchronisation.  They
 * cannot own the workspace moe_mxfp4_forward needs either.  This call takes the
 * same arguments and computes the same result, but its scratch is a static
 * device array of MOE_MXFP4_STATIC_WORKSPACE_BYTES inside the library, which
 * every GPU that loads the library holds until the process exits.  Nothing is
 * allocated by the call: no cudaMalloc, no allocating library routine.
 *   - Shapes whose workspace (moe_mxfp4_workspace_size) exceeds the array are
 *     rejected with MOE_ERR_WORKSPACE; other errors as for moe_mxfp4_forward.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) for that device.  With CUDA's lazy module loading
 *     that lookup is also when the array's device memory is committed.  A call
 *     with T = 0 (any supported shape; the pointers are not used) does only this
 *     set-up and enqueues nothing: make it once per device at start-up, before
 *     a memory pool takes the free device memory and before any stream capture.
 *   - Every call on a device shares the array and leaves its contents behind;
 *     the parts that must start at zero are cleared by each call.  Calls that
 *     overlap on the GPU (unordered streams) race on the array.
 *   - moe_mxfp4_last_device_status after such a call reads this array's status
 *     word (bounded-wait timeouts of the call are reported there).
 */
#define MOE_MXFP4_STATIC_WORKSPACE_BYTES ((size_t)64 << 20)
moe_status_t moe_mxfp4_forward_noalloc(const void* hidden, const void* w13, const void* w13_scale,
                                       const void* w2, const void* w2_scale,
                                       const int32_t* topk_ids, const float* topk_weights,
                                       void* out, int T, int d_model, int d_inter, int E,
                                       int topk, cudaStream_t stream);

/* Human-readable name of a status code (static string). */
const char* moe_mxfp4_status_string(moe_status_t status);

/*
 * Synchronise `stream`, then read the device status word of the workspace the
 * last forward call on the current device used (the registered workspace, or
 * the static array of moe_mxfp4_forward_noalloc; before any forward call, the
 * registered workspace).  Returns MOE_ERR_DEVICE_TIMEOUT when a kernel of that
 * call gave up on a bounded wait or found a counter in an impossible state,
 * MOE_OK otherwise.  Meant for tests and checked runs (it synchronises).
 */
moe_status_t moe_mxfp4_last_device_status(cudaStream_t stream);

/*
 * Self-check of device-side failure reporting: enqueue one kernel that waits on
 * a barrier nothing arrives on, through the same bounded wait the GEMM kernels
 * use, with a limit of limit_us microseconds (1 .. 1e6).  The wait runs out,
 * the kernel records the timeout in the registered workspace's status word and
 * returns; moe_mxfp4_last_device_status then reports MOE_ERR_DEVICE_TIMEOUT and
 * the next forward call clears the word.  The device stays usable.
 */
moe_status_t moe_mxfp4_check_wait_timeout(uint32_t limit_us, cudaStream_t stream);

/*
 * The forward's last step on its own: the deterministic top-k sum of per-route
 * rows (solution.py, _reference_forward's sum of the weighted expert outputs
 * over a token's top-k routes), for an expert-parallel combine, where the rows
 * come back from the ranks that own the experts.
 *   out[t] = bf16( sum over k = 0 .. topk-1 with route_pos[t*topk+k] >= 0 of
 *                  P[t*topk+k] ), fp32 adds in ascending k from zero, one rounding
 *   P          f32  [T*topk, d_model], rows by route id (w[t,k] * W2[e] . a2 in the
 *              forward; here whatever the caller computed)
 *   route_pos  i32  [T*topk]: >= 0 where the route counts, < 0 where it does not
 *   out        bf16 [T, d_model]; a token with no counted route gets a zero row
 * Device memory (or mapped pinned host memory), 16-byte aligned; d_model a
 * multiple of 128, 1 <= topk <= 16.  The same kernel and order as the forward.
 * Asynchronous on `stream`; T == 0 enqueues nothing.
 */
moe_status_t moe_mxfp4_topk_sum(const float* P, const int32_t* route_pos, void* out, int T,
                                int d_model, int topk, cudaStream_t stream);

/* ------------------------------------------------------------------ inspection */

/* Workspace regions, for tests and tools that inspect intermediate results.
 * Rows of the activation regions use the widths the kernels run at
 * (d_model_run, d_inter_run of the plan: the call's widths where they are 128,
 * 256 or a multiple of 512, else the next such width; the extra columns hold
 * zeros). */
typedef enum {
    MOE_WS_STATUS = 0,      /* u32 [1024]: [0] error bits; [15], [16], [17], [512..1024) the single-launch path's ready word, quantisation count, exit count and route-tile counters (zero between calls) */
    MOE_WS_COUNTERS = 1,    /* u32 [max_tiles]: finished stage-1 feature tiles per route tile (multi-kernel path; zeroed per call) */
    MOE_WS_SORTED_IDS = 2,  /* i32 [cap]: route id t*topk+k per sorted slot, T*topk = padding */
    MOE_WS_SORTED_W = 3,    /* f32 [cap]: topk weight of the slot's route, 0 for padding      */
    MOE_WS_BLOCK_EXPERT = 4,/* i32 [cap/block_m]: expert of each block, -1 unused             */
    MOE_WS_SEG_START = 5,   /* i32 [E+1]: first slot of each expert; [E] = padded length      */
    MOE_WS_ROUTE_POS = 6,   /* i32 [T*topk]: slot of each route, -1 for ids outside [0, E)    */
    MOE_WS_NUM_VALID = 7,   /* i32 [4]: padded length, valid routes, tiles, 0                 */
    MOE_WS_TILES = 8,       /* i32 [cap/block_m][4]: {expert, first slot, rows, 0}            */
    MOE_WS_A1Q = 9,         /* u8 [cap][d_model_run/2]: quantised hidden row of each slot's token */
    MOE_WS_A1S = 10,        /* u8 [cap][a1s_stride]: its e8m0 scales                          */
    MOE_WS_A2Q = 11,        /* u8 [cap][d_inter_run/2]: quantised SwiGLU output of each slot  */
    MOE_WS_A2S = 12,        /* u8 [cap][a2s_stride]: its e8m0 scales                          */
    MOE_WS_P = 13,          /* f32 [T*topk][d_model_run]: w[t,k] * stage-2 output, by route id */
    MOE_WS_PARTIAL = 14,    /* unused (0 bytes): no K split of stage 1                        */
    MOE_WS_A1B = 15,        /* bf16 [cap][d_model]: hidden row of each slot's token (bf16-activation plan only) */
    MOE_WS_A2B = 16,        /* bf16 [cap][d_inter]: bf16 SwiGLU output of each slot (bf16-activation plan only) */
    MOE_WS_WSCALE = 17,     /* u8: the weight scales with rows of d_model_run/32 (w13_scale) and d_inter_run/32 (w2_scale, from the next 256-byte boundary) bytes, the extra bytes 127; only where a width is run wider (else 0 bytes) */
    MOE_WS_NUM_REGIONS = 18
} moe_ws_region_t;

typedef struct {
    int block_m;        /* slots per padded block (segment granularity)                   */
    int tile_rows;      /* maximum routes per GEMM tile (multiple of block_m)             */
    int cap;            /* slots in the sorted arrays                                    */
    int a1s_stride;     /* bytes per row of MOE_WS_A1S                                   */
    int a2s_stride;     /* bytes per row of MOE_WS_A2S                                   */
    int stage1_splits;  /* K splits of the stage-1 GEMM (1)                              */
    int max_tiles;      /* capacity of MOE_WS_TILES                                      */
    int bf16_act;       /* 1: layout of the bf16-activation forward (a1q..a2s empty, a1b/a2b used) */
    int d_model_run;    /* width the kernels run d_model at (see the regions above)        */
    int d_inter_run;    /* width the kernels run d_inter at                                 */
    size_t offset[MOE_WS_NUM_REGIONS]; /* byte offset of each region in the workspace     */
    size_t bytes[MOE_WS_NUM_REGIONS];  /* byte size of each region                        */
    size_t workspace_bytes;            /* total (== moe_mxfp4_workspace_size)              */
} moe_mxfp4_plan_t;

/* Fill *plan with the layout the forward call uses for this shape.  Host-only;
 * touches no device.  Returns a shape/argument status like the forward call. */
moe_status_t moe_mxfp4_get_plan(int T, int d_model, int d_inter, int E, int topk,
                                moe_mxfp4_plan_t* plan);

/* Launch geometry of the fused GEMM kernel for a shape (diagnostics and tests;
 * it follows moe_mxfp4_set_tuning like the forward call).  Host-only; touches
 * no device.  Returns a shape/argument status like the forward call.
 * Properties every configuration keeps (the kernel checks the first three
 * itself and reports a violation in the status word instead of running):
 *   acc_bufs * acc_cols <= sf_col0, sf_col0 + num_stages * sf_cols <= tmem_cols
 *   <= 512 (tensor-memory columns: accumulators, then each slot's scale factors);
 *   acc_bufs >= epi_groups (an epilogue group waits for its item's buffer by
 *   barrier parity, which is unambiguous only if the buffer's previous use has
 *   completed; the group's own previous item, completed, implies that when there
 *   are at least as many buffers as groups, since each MMA warp's operations
 *   complete in issue order);
 *   smem_bytes <= smem_limit;
 *   mma_warps == 2 (alternate stages) implies an even num_stages (a warp waits
 *   for a slot's fill by barrier parity, so it must have seen the slot's
 *   previous fill: that stage must be its own). */
typedef struct {
    int tile_rows;          /* routes per route tile (the MMA's N)                          */
    int stage1_k;           /* K elements per pipeline stage of the gate_up GEMM            */
    int stage2_k;           /* K elements per pipeline stage of the down GEMM                */
    int stage2_blocks;      /* 128-row weight blocks per down-GEMM work item                 */
    int num_stages;         /* shared-memory ring slots                                     */
    int mma_warps;          /* MMA-issuing warps (2: they take alternate stages)            */
    int acc_bufs;           /* tensor-memory accumulator buffers                             */
    int epi_groups;         /* epilogue groups of four warps                                  */
    int sf_by_layout_warp;  /* the scale-layout warp copies the scale factors to TMEM too   */
    int wide_sf;            /* two-chunk scale-factor copies from staging buffers            */
    int lookahead;          /* MMA warps copy the next stage's scale factors early          */
    unsigned slot_bytes;    /* bytes per ring slot                                           */
    unsigned smem_bytes;    /* dynamic shared memory per CTA                                  */
    unsigned smem_limit;    /* the kernel's dynamic shared-memory limit                       */
    unsigned acc_cols;      /* TMEM columns per accumulator buffer                            */
    unsigned sf_col0;       /* first TMEM column of the per-slot scale-factor regions         */
    unsigned sf_cols;       /* TMEM scale-factor columns per ring slot                        */
    unsigned tmem_cols;     /* TMEM columns allocated                                        */
} moe_mxfp4_gemm_config_t;

moe_status_t moe_mxfp4_get_gemm_config(int T, int d_model, int d_inter, int E, int topk,
                                       moe_mxfp4_gemm_config_t* cfg);

/* Workspace bytes and layout of the bf16-activation forward (regions a1b, a2b
 * instead of a1q .. a2s; bf16_act = 1). */
size_t moe_mxfp4_workspace_size_w4a16(int T, int d_model, int d_inter, int E, int topk);
moe_status_t moe_mxfp4_get_plan_w4a16(int T, int d_model, int d_inter, int E, int topk,
                                      moe_mxfp4_plan_t* plan);

/* Version string of the library build. */
const char* moe_mxfp4_version(void);

/* Where a per-call buffer lives, for the host-memory case of the forward entry
 * points: 0 device (or managed) memory; 1 host memory that the current device
 * reads and writes at the same address (pinned and mapped); -1 neither
 * (pageable or unknown memory: not usable as a forward argument).  A host-side
 * query (cudaPointerGetAttributes); no device work. */
int moe_mxfp4_pointer_kind(const void* ptr);

/* ------------------------------------------------------------------ timing */

/* Number of kernel slots of a forward call (route, quant, the GEMM kernel that
 * runs both grouped GEMMs, top-k sum).  In single-launch mode the route and
 * quant slots are empty: routing and quantisation run inside the GEMM kernel. */
int moe_mxfp4_num_kernels(void);

/*
 * Launch mode for the current device (the single launch follows the fused
 * FC1 -> activation -> FC2 persistent launch of b12x moe/fused/w4a16/kernel.py,
 * where one grid runs every step).  In a single launch, shapes with
 * T*topk <= 2048 and E <= 384 route and quantise inside the GEMM kernel: every
 * CTA sorts all routes in shared memory and quantises a share of the hidden
 * states, and the stage-1 route-tile copies wait (bounded) until all CTAs have
 * counted their share; only the GEMM kernel and the top-k sum are launched.
 * Otherwise: routing kernel, quantisation kernel, GEMM kernel, top-k sum.
 *   mode 0: always separate kernels;
 *   mode 1: single launch wherever the shape allows;
 *   mode 2 (default): single launch for decode-sized calls (T*topk <= 256),
 *           where it measured faster; separate kernels above.
 * Results are identical in every mode.  Returns MOE_ERR_INVALID_ARG for other
 * modes.
 */
moe_status_t moe_mxfp4_set_single_launch(int mode);

/* Kernels a forward call of this shape launches on the current device under its
 * launch mode: 4 (route, quant, GEMM, top-k sum), 6 when T*topk >= 4096 (routing
 * then runs on many CTAs in three launches: chunk counts, offsets, scatter),
 * 2 (GEMM with routing and quantisation inside, top-k sum), 0 for T = 0, -1 for
 * an invalid shape or no device. */
int moe_mxfp4_call_launches(int T, int d_model, int d_inter, int E, int topk);

/*
 * Optional instrumentation for benchmarks (events created once per device on
 * first use; no device memory is allocated).
 *   mode 0: off.
 *   mode 1: the forward call records a CUDA event on its stream before each
 *           kernel and after the last one.  Events between kernels serialise
 *           them (the dependent-launch overlap is lost), so use it for the
 *           per-kernel breakdown.
 *   mode 2: events only before the first and after the last kernel.
 * moe_mxfp4_kernel_times (mode 1) waits for the last event and writes each
 * kernel's duration of the most recent call, in ms, to ms[0 .. min(n, num_kernels)-1]
 * (a negative value for a slot in which that call launched nothing) and returns
 * the count, or -1.  moe_mxfp4_last_call_ms (modes 1 and 2) returns
 * the device time of the most recent call in ms, or a negative value.
 */
moe_status_t moe_mxfp4_set_kernel_timing(int mode);

/*
 * NVTX ranges for timeline profilers (process-wide; off by default).  on = 1:
 * every forward call pushes one range named "moe_mxfp4 forward" (with the shape,
 * the entry point and the launch mode) around its enqueue, with nested ranges
 * "route", "quant", "gemm" and "topk_sum" around each kernel launch, so a
 * timeline tool correlates them with the kernels.  The ranges are host-side (the
 * enqueue), cost a few hundred nanoseconds per call without an attached tool
 * and change nothing on the device.  on = 0 turns them off.  MOE_ERR_INVALID_ARG
 * for other values.  The header-only NVTX of the CUDA toolkit is compiled in;
 * nothing is linked.
 */
moe_status_t moe_mxfp4_set_nvtx(int on);

/*
 * Tuning override for measurements (process-wide; results do not change, only
 * speed).  tile_rows: the GEMM route-tile width (maximum MMA N, routes per
 * tile): 16, 32, 64 or 128, or 0 for the library's choice by shape (the
 * per-shape block_m table of flower_moe.py is the pages' counterpart).
 * sf_copies: who copies the block scales to tensor memory: 1 the MMA-issuing
 * warps (two of them), 2 a separate warp, one 128-element chunk per copy, 3 a
 * separate warp, two chunks per copy where shared memory allows (else as 2),
 * 4 a separate warp, one chunk per copy, with two MMA-issuing warps taking
 * alternate pipeline stages where their accumulators fit in tensor memory (else
 * as 2), 0 the library's choice.  Affects
 * calls made after it (their plan, moe_mxfp4_get_plan, follows it); the
 * workspace size does not depend on it.  MOE_ERR_INVALID_ARG for other values.
 */
moe_status_t moe_mxfp4_set_tuning(int tile_rows, int sf_copies);

/*
 * Measurement aid for the roofline's compute term (no counterpart in the pages):
 * enqueue on `stream` one kernel with one CTA per SM, each issuing `iters`
 * block-scaled MXFP4 MMAs (tcgen05.mma .kind::mxf4 .scale_vec::2X, M = 128,
 * N = n, K = 64, operands in shared memory, zero values) into one tensor-memory
 * accumulator, and copies_per_mma scale-factor copies to tensor memory per MMA
 * (the GEMM kernel's per-stage mix).  variant bit 0: the copies are
 * tcgen05.cp .128x256b (else .32x128b.warpx4, the GEMM kernel's); bit 1: a second
 * warp issues the copies (else the MMA thread, before each MMA); bits 2-3: the
 * MMAs rotate over 2^bits independent accumulators (n * 2^bits <= 256); bits
 * 4-5: the MMA thread commits its tensor operations to an mbarrier after every
 * 1, 4 or 8 MMAs (values 1, 2, 3; nothing waits on it).  *flops receives the
 * dense operation count (2*128*n*64 per MMA); time the kernel with events on
 * `stream`.  n: 16..256, multiple of 16; iters: 1..1e7; copies_per_mma: 0..8;
 * variant: 0..63.  Needs a registered workspace (its
 * status word records a timed-out final wait; moe_mxfp4_last_device_status
 * reads it).  Overwrites nothing else.
 */
moe_status_t moe_mxfp4_tensor_probe(int n, int iters, int copies_per_mma, int variant,
                                    double* flops, cudaStream_t stream);
int moe_mxfp4_kernel_times(float* ms, int n);
float moe_mxfp4_last_call_ms(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_MXFP4_H */
