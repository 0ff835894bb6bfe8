// moe_mxfp4_forward_noalloc: the forward call for callers that cannot allocate
// device memory.
//
// Some callers cannot call cudaMalloc (or any allocating routine) at the point
// where they run the MoE layer: a serving runtime that hands all free device
// memory to its own pool at start-up (so a later cudaMalloc fails), a plugin
// host that does not let plugins allocate, or a latency-critical loop that must
// not hit cudaMalloc's implicit device synchronisation.  Such a caller also
// cannot own a workspace for moe_mxfp4_set_workspace.  This entry point instead
// uses a scratch buffer that lives in the library itself: a file-scope
// __device__ array of kStaticWorkspaceBytes, which every GPU that loads the
// library holds until the process exits.  Shapes whose workspace does not fit
// are rejected with MOE_ERR_WORKSPACE.
//
// The array is shared by every call on a device and keeps the previous call's
// contents.  The parts that must start at zero are zero when the library's
// module is loaded (a __device__ array is zero-initialised) and are kept so: the
// routing kernel clears the route-tile counters and status words at the start
// of a multi-kernel call, and the last CTA of a single-launch GEMM kernel clears
// the words that kernel shares across CTAs.  Calls that overlap on the GPU
// (different streams without ordering) race on the array.
//
// The array's device memory is committed when the module that holds it is
// loaded, which with CUDA's lazy module loading is the first address lookup.
// The entry point does that lookup on its first call on a device; a call with
// T = 0 does only that (it enqueues nothing), so a caller makes it at start-up,
// before its own pool takes the free device memory and before any stream
// capture.
#include <cuda_runtime.h>

#include <mutex>

#include "moe_internal.h"

namespace {

constexpr size_t kStaticWorkspaceBytes = MOE_MXFP4_STATIC_WORKSPACE_BYTES;
constexpr int kMaxDev = 64;

static __device__ __align__(256) unsigned char g_static_workspace[kStaticWorkspaceBytes];

std::mutex g_static_mu;
void* g_static_ptr[kMaxDev];

// Device address of g_static_workspace on the current device: looked up once
// per device (the name is only a host-side stand-in for the device array).
void* static_workspace(int dev) {
    std::lock_guard<std::mutex> lk(g_static_mu);
    if (!g_static_ptr[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_static_workspace) != cudaSuccess) return nullptr;
        g_static_ptr[dev] = ptr;
    }
    return g_static_ptr[dev];
}

}  // namespace

extern "C" moe_status_t moe_mxfp4_forward_noalloc(const void* hidden, const void* w13,
                                                  const void* w13_scale, const void* w2,
                                                  const void* w2_scale, const int32_t* topk_ids,
                                                  const float* topk_weights, void* out, int T,
                                                  int d_model, int d_inter, int E, int topk,
                                                  cudaStream_t stream) {
    const moe_status_t st = moe::validate_forward(hidden, w13, w13_scale, w2, w2_scale, topk_ids,
                                                  topk_weights, out, T, d_model, d_inter, E, topk);
    if (st != MOE_OK) return st;
    if (moe::plan_workspace_bytes(T, d_model, d_inter, E, topk) > kStaticWorkspaceBytes)
        return MOE_ERR_WORKSPACE;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return MOE_ERR_CUDA;
    void* base = static_workspace(dev);  // (the set-up; all a T = 0 call does)
    if (!base) return MOE_ERR_CUDA;
    if (T == 0) return MOE_OK;
    return moe::forward_on_workspace(hidden, w13, w13_scale, w2, w2_scale, topk_ids, topk_weights,
                                     out, T, d_model, d_inter, E, topk, d_model, d_inter, base,
                                     dev, stream);
}
