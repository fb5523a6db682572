// noalloc.cu -- conv_bwd_filter_noalloc: the weight gradient for callers that
// cannot allocate device memory.  The split-K partials go to a file-scope
// __device__ array instead of a caller-provided workspace; everything else is
// the FFMA split-K wgrad of kernels_ffma.cu (partials, then the ascending-split
// reduction).
#include <mutex>

#include "internal.h"

using namespace igc;

namespace {

// Scratch for the split-K partials.  Every GPU that loads the library holds it
// until the process exits.  In host code this name is only a host-side handle:
// kernels get the device address from cudaGetSymbolAddress (set up below).
static __device__ __align__(256) unsigned char g_noalloc_scratch[CONV_NOALLOC_SCRATCH_BYTES];

std::mutex g_mu;
void* g_scratch_ptr[64] = {};

// Device address of the scratch on the current device, looked up once per
// device with that device current.
int scratch_address(int dev, void** out)
{
    if (dev < 0 || dev >= 64) return CONV_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_ptr[dev]) {
        void* ptr = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess || !ptr) {
            cudaGetLastError();
            return CONV_ERR_CUDA;
        }
        g_scratch_ptr[dev] = ptr;
    }
    *out = g_scratch_ptr[dev];
    return CONV_OK;
}

}  // namespace

extern "C" int conv_bwd_filter_noalloc(const conv_desc_t* desc, const void* x, const void* dy,
                                       const void* y, void* dw, conv_stream_t stream)
{
    ConvParams p;
    int rc = make_params(desc, p);
    if (rc != CONV_OK) return rc;
    const size_t per_split = size_t(p.OC) * size_t(round_up(p.Kred, 4)) * sizeof(float);
    if (per_split > CONV_NOALLOC_SCRATCH_BYTES) return CONV_ERR_UNSUPPORTED;
    if (!dw) return CONV_ERR_NULL;
    if (p.B > 0 && (!x || !dy || (p.relu && !y))) return CONV_ERR_NULL;
    if (!aligned16(dw) || (p.B > 0 && (!aligned16(x) || !aligned16(dy) || (p.relu && !aligned16(y)))))
        return CONV_ERR_ALIGN;
    DevInfo d;
    if ((rc = device_info(d)) != CONV_OK) return rc;
    void* scratch = nullptr;
    if ((rc = scratch_address(d.device, &scratch)) != CONV_OK) return rc;

    Plan pl = plan_wgrad_ffma(p, d);
    const int max_splits = int(CONV_NOALLOC_SCRATCH_BYTES / per_split);
    if (pl.splits > max_splits) {
        const int tiles = pl.grid / pl.splits;
        pl.splits = max_splits;
        pl.grid = tiles * max_splits;
        pl.workspace = size_t(max_splits) * per_split;
    }
    return cuda_status(run_wgrad_ffma(pl, p, desc->dtype, x, dy, y, dw, scratch,
                                      reinterpret_cast<cudaStream_t>(stream)));
}
