// internal.h -- host-side plan and launcher interface between api.cu (the C
// ABI: validation, dispatch) and the kernel translation units.
#pragma once
#include <cstddef>
#include <utility>
#include <cuda_runtime.h>

#include "../../include/conv.h"
#include "common.cuh"

namespace igc {

struct DevInfo {
    int device = -1;
    int sms = 0;             // streaming multiprocessors
    int smem_optin = 0;      // max dynamic shared memory per block (opt-in)
    int cc_major = 0, cc_minor = 0;
};

// One operation's launch plan.  `algo` uses the conv_algo_t values.
struct Plan {
    int algo = 0;
    int launches = 0;
    int grid = 0, block = 0, smem = 0;
    int splits = 0;
    size_t workspace = 0;
    int variant = 0;         // kernel-family specific selector
};

enum { DT_F32 = 0, DT_BF16 = 1 };
enum { ALGO_AUTO = 0, ALGO_DIRECT = 1, ALGO_FFMA = 2, ALGO_TC = 3 };

// ---- host helpers shared by the C-ABI translation units (api.cu) --------------------
int device_info(DevInfo& out);                      // current device, cached; conv_status_t
int make_params(const conv_desc_t* d, ConvParams& p);  // validation, no CUDA calls
bool aligned16(const void* p);
int cuda_status(cudaError_t e);                     // cudaSuccess -> CONV_OK, else CONV_ERR_CUDA

// Largest thread-block cluster the kernels use (the portable limit).
constexpr int kMaxCluster = 8;

// ---- FFMA and direct families (kernels_ffma.cu) ------------------------------------
bool ffma_fwd_ok(const ConvParams& p, const DevInfo& d);
bool ffma_dgrad_ok(const ConvParams& p, const DevInfo& d);
bool ffma_wgrad_ok(const ConvParams& p, const DevInfo& d);
Plan plan_fwd_ffma(const ConvParams& p, const DevInfo& d);
Plan plan_dgrad_ffma(const ConvParams& p, const DevInfo& d);
Plan plan_wgrad_ffma(const ConvParams& p, const DevInfo& d);
Plan plan_fwd_direct(const ConvParams& p, const DevInfo& d);
Plan plan_dgrad_direct(const ConvParams& p, const DevInfo& d);
Plan plan_wgrad_direct(const ConvParams& p, const DevInfo& d);

// Forward launchers: `bias` (OC values of the dtype) is added to each finished sum before the
// activation; nullptr = no bias.
cudaError_t run_fwd_ffma(const Plan&, const ConvParams&, int dt, const void* x, const void* w,
                         const void* bias, void* y, cudaStream_t s);
cudaError_t run_dgrad_ffma(const Plan&, const ConvParams&, int dt, const void* dy, const void* w,
                           const void* y, void* dx, cudaStream_t s);
cudaError_t run_wgrad_ffma(const Plan&, const ConvParams&, int dt, const void* x, const void* dy,
                           const void* y, void* dw, void* ws, cudaStream_t s);
cudaError_t run_fwd_direct(const Plan&, const ConvParams&, int dt, const void* x, const void* w,
                           const void* bias, void* y, cudaStream_t s);
cudaError_t run_dgrad_direct(const Plan&, const ConvParams&, int dt, const void* dy,
                             const void* w, const void* y, void* dx, cudaStream_t s);
cudaError_t run_wgrad_direct(const Plan&, const ConvParams&, int dt, const void* x,
                             const void* dy, const void* y, void* dw, cudaStream_t s);
// Deterministic split-K sum: dw = sum_{s < splits} ws[s] (fp32 partials, row
// stride kpad), rounded once to the dtype.  splits == 0 writes zeros.  `overlapped`:
// launched to overlap the kernel that writes ws (it waits for that kernel itself).  With db:
// also db[oc] = sum_{q < nbp} bpart[q][oc] (nbp == 0 writes zeros).
cudaError_t run_wgrad_reduce(const ConvParams&, int dt, const float* ws, int splits, int kpad,
                             void* dw, cudaStream_t s, bool overlapped = false, const float* bpart = nullptr,
                             int nbp = 0, void* db = nullptr);
cudaError_t run_l2_flush(void* buf, size_t bytes, cudaStream_t s);

// Dynamic shared memory above 48 KB needs a per-kernel opt-in on every device;
// done once per (kernel, device) and remembered.
template <auto Kern>
cudaError_t ensure_smem(int bytes)
{
    if (bytes <= 48 * 1024) return cudaSuccess;
    static int configured[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64 && configured[dev] >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(Kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && dev >= 0 && dev < 64) configured[dev] = bytes;
    return e;
}

// Launch `Kern` so that it may start while the previous kernel on the stream is still
// running (programmatic dependent launch): the kernel must execute griddepcontrol.wait
// before it reads anything that kernel writes.  Use only for the second kernel of a pair
// whose first kernel was launched in plain stream order.
template <class... KArgs, class... Args>
cudaError_t launch_overlapped(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args&&... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Launch `Kern` with a 1-D thread-block cluster of `cluster` CTAs (1 = none; the grid must be a
// multiple of it), and optionally as a programmatic dependent launch (see launch_overlapped; the
// kernel then executes griddepcontrol.wait before its first global-memory access).
template <class... KArgs, class... Args>
cudaError_t launch_ex(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, int cluster,
                      bool pdl, Args&&... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int n = 0;
    if (pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    if (cluster > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = unsigned(cluster);
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// ---- tcgen05 tensor-core family (kernels_tc.cu) -------------------------------------
// `packed` / `ws`: the workspace path (weights packed once per call into the caller's
// workspace, bulk-copied by the main kernel); else the main kernel formats them itself.
bool tc_fwd_ok(const ConvParams& p, int dt, const DevInfo& d, bool packed);
Plan plan_fwd_tc(const ConvParams& p, int dt, const DevInfo& d, bool packed);
cudaError_t run_fwd_tc(const Plan&, const ConvParams&, int dt, const void* x, const void* w,
                       const void* bias, void* y, void* ws, cudaStream_t s);
bool tc_wgrad_ok(const ConvParams& p, int dt, const DevInfo& d);
Plan plan_wgrad_tc(const ConvParams& p, int dt, const DevInfo& d);
// db != nullptr: also the bias gradient, from the same loads of g (its partial channel sums go
// to the workspace's tail, see plan_wgrad_tc).
cudaError_t run_wgrad_tc(const Plan&, const ConvParams&, int dt, const void* x, const void* dy,
                         const void* y, void* dw, void* ws, void* db, cudaStream_t s);
bool tc_dgrad_ok(const ConvParams& p, int dt, const DevInfo& d, bool packed);
Plan plan_dgrad_tc(const ConvParams& p, int dt, const DevInfo& d, bool packed);
cudaError_t run_dgrad_tc(const Plan&, const ConvParams&, int dt, const void* dy, const void* w,
                         const void* y, void* dx, void* ws, cudaStream_t s);
// Fused backward: d_input and wgrad (and with db the bias gradient) in one launch after packing
// W^T; the split reduction follows.
bool tc_bwd_ok(const ConvParams& p, int dt, const DevInfo& d);
Plan plan_bwd_tc(const ConvParams& p, int dt, const DevInfo& d);
cudaError_t run_bwd_tc(const Plan&, const ConvParams& p, int dt, const DevInfo& d, const void* x, const void* dy,
                       const void* w, const void* y, void* dx, void* dw, void* db, void* ws, cudaStream_t s);
// Two-layer forward chain (layer 2's input = layer 1's output), one kernel after packing both
// weight images into the workspace.
bool tc_chain_ok(const ConvParams& p1, const ConvParams& p2, int dt, const DevInfo& d);
int chain_groups(const ConvParams& p1, const ConvParams& p2);  // groups of whole samples the fused kernel runs
Plan plan_chain_tc(const ConvParams& p1, const ConvParams& p2, int dt, const DevInfo& d);
cudaError_t run_chain_tc(const Plan&, const ConvParams& p1, const ConvParams& p2, int dt, const void* x,
                         const void* w1, const void* b1, const void* w2, const void* b2, void* y1, void* y2, void* ws,
                         cudaStream_t s);
// ---- bias gradient (kernels_bias.cu) ------------------------------------------------
// `direct`: the one-warp-per-channel kernel (any shape); else the column-sum kernel and its
// reduce, when the shape allows.
Plan plan_bgrad(const ConvParams& p, int dt, const DevInfo& d, bool direct);
cudaError_t run_bgrad(const Plan&, const ConvParams&, int dt, const void* dy, const void* y, void* db,
                      cudaStream_t s);

// Error bits the tensor-core kernels set when a bounded wait runs out.
cudaError_t tc_read_status(unsigned* out, bool reset);
// Bounded-wait self-test (kernels_diag.cu): a one-CTA kernel whose wait on a never-completed
// mbarrier runs out and sets CONV_STATUS_WAIT_SELFTEST in its own status word.
cudaError_t run_wait_selftest(unsigned max_sleeps, cudaStream_t s);
cudaError_t diag_read_status(unsigned* out, bool reset);

__host__ __device__ inline int round_up(int a, int b) { return (a + b - 1) / b * b; }
__host__ __device__ inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

}  // namespace igc
