// api.cu -- the C ABI declared in include/conv.h: argument validation (all on
// the host, before anything is enqueued), the per-device facts a plan needs,
// the choice of kernel family, and the launches.
#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/conv.h"
#include "internal.h"

using namespace igc;

namespace igc {

constexpr int64_t kMaxElems = (int64_t(1) << 31) - 1;

struct DevCache {
    std::mutex mu;
    DevInfo info[64];
    bool have[64] = {};
} g_dev;

int device_info(DevInfo& out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return CONV_ERR_CUDA;
    if (dev < 0 || dev >= 64) return CONV_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_dev.mu);
    if (!g_dev.have[dev]) {
        DevInfo d;
        d.device = dev;
        if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
                cudaSuccess ||
            cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
            cudaGetLastError();
            return CONV_ERR_CUDA;
        }
        g_dev.info[dev] = d;
        g_dev.have[dev] = true;
    }
    out = g_dev.info[dev];
    return CONV_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Descriptor checks and the derived parameter block.  Host only, no CUDA calls.
int make_params(const conv_desc_t* d, ConvParams& p)
{
    if (!d) return CONV_ERR_NULL;
    if (d->B < 0 || d->IC < 1 || d->OC < 1 || d->K < 1 || d->S < 1 || d->H < d->K ||
        d->W < d->K || (d->relu != 0 && d->relu != 1) || (d->dtype != CONV_F32 && d->dtype != CONV_BF16))
        return CONV_ERR_DESC;
    const int64_t OH = (int64_t(d->H) - d->K) / d->S + 1, OW = (int64_t(d->W) - d->K) / d->S + 1;
    const int64_t nx = int64_t(d->B) * d->IC * d->H * d->W;
    const int64_t ny = int64_t(d->B) * d->OC * OH * OW;
    const int64_t nw = int64_t(d->OC) * d->IC * d->K * d->K;
    const int64_t per_x = int64_t(d->IC) * d->H * d->W;
    if (nx > kMaxElems || ny > kMaxElems || nw > kMaxElems || per_x > kMaxElems) return CONV_ERR_UNSUPPORTED;
    p.B = d->B; p.IC = d->IC; p.OC = d->OC; p.H = d->H; p.W = d->W; p.K = d->K; p.S = d->S;
    p.OH = int(OH); p.OW = int(OW); p.relu = d->relu;
    p.P = int(OH * OW);
    p.KK = d->K * d->K;
    p.Kred = d->IC * p.KK;
    p.HW = d->H * d->W;
    p.IHW = int(per_x);
    p.OCP = d->OC * p.P;
    p.N = d->B * p.P;
    p.dm_P = FastDivmod(uint32_t(p.P));
    p.dm_OW = FastDivmod(uint32_t(p.OW));
    p.dm_KK = FastDivmod(uint32_t(p.KK));
    p.dm_K = FastDivmod(uint32_t(p.K));
    p.dm_W = FastDivmod(uint32_t(p.W));
    p.dm_HW = FastDivmod(uint32_t(p.HW));
    return CONV_OK;
}

int cuda_status(cudaError_t e)
{
    if (e == cudaSuccess) return CONV_OK;
    cudaGetLastError();
    return CONV_ERR_CUDA;
}

}  // namespace igc

namespace {

std::atomic<int> g_force[4] = {ALGO_AUTO, ALGO_AUTO, ALGO_AUTO, ALGO_AUTO};

// ---- plan selection -------------------------------------------------------------------
// `packed`: the plan of the workspace-taking entry point (conv_fwd_ws / conv_bwd_data_ws).
int choose_fwd(const ConvParams& p, int dt, const DevInfo& d, bool packed, Plan& pl)
{
    const int force = g_force[CONV_OP_FWD].load();
    if (force == ALGO_DIRECT) { pl = plan_fwd_direct(p, d); return CONV_OK; }
    if (force == ALGO_TC || force == ALGO_AUTO) {
        if (tc_fwd_ok(p, dt, d, packed)) { pl = plan_fwd_tc(p, dt, d, packed); return CONV_OK; }
        if (force == ALGO_TC) return CONV_ERR_UNSUPPORTED;
    }
    if (ffma_fwd_ok(p, d)) { pl = plan_fwd_ffma(p, d); return CONV_OK; }
    if (force == ALGO_FFMA) return CONV_ERR_UNSUPPORTED;
    pl = plan_fwd_direct(p, d);
    return CONV_OK;
}

int choose_dgrad(const ConvParams& p, int dt, const DevInfo& d, bool packed, Plan& pl)
{
    const int force = g_force[CONV_OP_BWD_DATA].load();
    if (force == ALGO_DIRECT) { pl = plan_dgrad_direct(p, d); return CONV_OK; }
    if (force == ALGO_TC || force == ALGO_AUTO) {
        if (tc_dgrad_ok(p, dt, d, packed)) { pl = plan_dgrad_tc(p, dt, d, packed); return CONV_OK; }
        if (force == ALGO_TC) return CONV_ERR_UNSUPPORTED;
    }
    if (ffma_dgrad_ok(p, d)) { pl = plan_dgrad_ffma(p, d); return CONV_OK; }
    if (force == ALGO_FFMA) return CONV_ERR_UNSUPPORTED;
    pl = plan_dgrad_direct(p, d);
    return CONV_OK;
}

int choose_wgrad(const ConvParams& p, int dt, const DevInfo& d, Plan& pl)
{
    const int force = g_force[CONV_OP_BWD_FILTER].load();
    if (force == ALGO_DIRECT) { pl = plan_wgrad_direct(p, d); return CONV_OK; }
    if (force == ALGO_TC || force == ALGO_AUTO) {
        if (tc_wgrad_ok(p, dt, d)) { pl = plan_wgrad_tc(p, dt, d); return CONV_OK; }
        if (force == ALGO_TC) return CONV_ERR_UNSUPPORTED;
    }
    if (ffma_wgrad_ok(p, d)) { pl = plan_wgrad_ffma(p, d); return CONV_OK; }
    if (force == ALGO_FFMA) return CONV_ERR_UNSUPPORTED;
    pl = plan_wgrad_direct(p, d);
    return CONV_OK;
}

int choose_bgrad(const ConvParams& p, int dt, const DevInfo& d, Plan& pl)
{
    pl = plan_bgrad(p, dt, d, g_force[CONV_OP_BWD_BIAS].load() == ALGO_DIRECT);
    return CONV_OK;
}

// The fused backward when both operations run on the tensor cores, else d_input (workspace path)
// then wgrad, one after the other, sharing the workspace (laid out one after the other).
int choose_bwd(const ConvParams& p, int dt, const DevInfo& d, Plan& pl)
{
    Plan a, b;
    int rc = choose_dgrad(p, dt, d, true, a);
    if (rc == CONV_OK) rc = choose_wgrad(p, dt, d, b);
    if (rc != CONV_OK) return rc;
    if (a.algo == ALGO_TC && b.algo == ALGO_TC && tc_bwd_ok(p, dt, d)) {
        pl = plan_bwd_tc(p, dt, d);
        return CONV_OK;
    }
    pl = Plan();
    pl.algo = ALGO_AUTO;  // two calls
    pl.launches = a.launches + b.launches;
    pl.grid = std::max(a.grid, b.grid);
    pl.block = std::max(a.block, b.block);
    pl.smem = std::max(a.smem, b.smem);
    pl.splits = b.splits;
    pl.workspace = (a.workspace + 255) / 256 * 256 + b.workspace;
    return CONV_OK;
}

int choose(int op, const ConvParams& p, int dt, const DevInfo& d, Plan& pl)
{
    switch (op) {
    case CONV_OP_FWD: return choose_fwd(p, dt, d, false, pl);
    case CONV_OP_BWD_DATA: return choose_dgrad(p, dt, d, false, pl);
    case CONV_OP_BWD_FILTER: return choose_wgrad(p, dt, d, pl);
    case CONV_OP_BWD_BIAS: return choose_bgrad(p, dt, d, pl);
    case CONV_OP_FWD_WS: return choose_fwd(p, dt, d, true, pl);
    case CONV_OP_BWD_DATA_WS: return choose_dgrad(p, dt, d, true, pl);
    case CONV_OP_BWD: return choose_bwd(p, dt, d, pl);
    default: return CONV_ERR_UNSUPPORTED;
    }
}

// The forward, with (ws != nullptr: the workspace path) or without a workspace.
int fwd_impl(const conv_desc_t* desc, const void* x, const void* w, const void* bias, void* y, void* ws,
             size_t ws_bytes, bool with_ws, conv_stream_t stream)
{
    ConvParams p;
    int rc = make_params(desc, p);
    if (rc != CONV_OK) return rc;
    if (p.B == 0) return CONV_OK;
    if (!x || !w || !y) return CONV_ERR_NULL;
    if (!aligned16(x) || !aligned16(w) || !aligned16(y) || (bias && !aligned16(bias)) || (ws && !aligned16(ws)))
        return CONV_ERR_ALIGN;
    DevInfo d;
    if ((rc = device_info(d)) != CONV_OK) return rc;
    Plan pl;
    if ((rc = choose_fwd(p, desc->dtype, d, with_ws, pl)) != CONV_OK) return rc;
    if (pl.workspace > 0 && (!ws || ws_bytes < pl.workspace)) return CONV_ERR_WORKSPACE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (pl.algo == ALGO_DIRECT) return cuda_status(run_fwd_direct(pl, p, desc->dtype, x, w, bias, y, s));
    if (pl.algo == ALGO_TC)
        return cuda_status(run_fwd_tc(pl, p, desc->dtype, x, w, bias, y, pl.workspace > 0 ? ws : nullptr, s));
    return cuda_status(run_fwd_ffma(pl, p, desc->dtype, x, w, bias, y, s));
}

int dgrad_impl(const conv_desc_t* desc, const void* dy, const void* w, const void* y, void* dx, void* ws,
               size_t ws_bytes, bool with_ws, conv_stream_t stream)
{
    ConvParams p;
    int rc = make_params(desc, p);
    if (rc != CONV_OK) return rc;
    if (p.B == 0) return CONV_OK;
    if (!dy || !w || !dx || (p.relu && !y)) return CONV_ERR_NULL;
    if (!aligned16(dy) || !aligned16(w) || !aligned16(dx) || (p.relu && !aligned16(y)) || (ws && !aligned16(ws)))
        return CONV_ERR_ALIGN;
    DevInfo d;
    if ((rc = device_info(d)) != CONV_OK) return rc;
    Plan pl;
    if ((rc = choose_dgrad(p, desc->dtype, d, with_ws, pl)) != CONV_OK) return rc;
    if (pl.workspace > 0 && (!ws || ws_bytes < pl.workspace)) return CONV_ERR_WORKSPACE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (pl.algo == ALGO_DIRECT) return cuda_status(run_dgrad_direct(pl, p, desc->dtype, dy, w, y, dx, s));
    if (pl.algo == ALGO_TC)
        return cuda_status(run_dgrad_tc(pl, p, desc->dtype, dy, w, y, dx, pl.workspace > 0 ? ws : nullptr, s));
    return cuda_status(run_dgrad_ffma(pl, p, desc->dtype, dy, w, y, dx, s));
}

// Workspace bytes of an operation's plan on the current device (0: none, or invalid).
size_t plan_workspace(int op, const conv_desc_t* desc)
{
    ConvParams p;
    if (make_params(desc, p) != CONV_OK) return 0;
    DevInfo d;
    if (device_info(d) != CONV_OK) return 0;
    Plan pl;
    if (choose(op, p, desc->dtype, d, pl) != CONV_OK) return 0;
    return pl.workspace;
}

}  // namespace

extern "C" {

const char* conv_version(void) { return "0.1.0"; }

const char* conv_status_string(int status)
{
    switch (status) {
    case CONV_OK: return "CONV_OK";
    case CONV_ERR_NULL: return "CONV_ERR_NULL: a required pointer is NULL";
    case CONV_ERR_DESC: return "CONV_ERR_DESC: invalid descriptor";
    case CONV_ERR_UNSUPPORTED: return "CONV_ERR_UNSUPPORTED: outside the library's limits";
    case CONV_ERR_ALIGN: return "CONV_ERR_ALIGN: a pointer is not 16-byte aligned";
    case CONV_ERR_WORKSPACE: return "CONV_ERR_WORKSPACE: workspace missing or too small";
    case CONV_ERR_CUDA: return "CONV_ERR_CUDA: a CUDA call or kernel launch failed";
    default: return "unknown conv status";
    }
}

int conv_out_dims(const conv_desc_t* desc, int32_t* OH, int32_t* OW)
{
    ConvParams p;
    const int rc = make_params(desc, p);
    if (rc != CONV_OK) return rc;
    if (!OH || !OW) return CONV_ERR_NULL;
    *OH = p.OH;
    *OW = p.OW;
    return CONV_OK;
}

int conv_set_algo(int op, int algo)
{
    if (op < 0 || op > 5 || algo < ALGO_AUTO || algo > ALGO_TC) return CONV_ERR_UNSUPPORTED;  // op 6: ops 1, 2
    if (op == CONV_OP_BWD_BIAS && algo != ALGO_AUTO && algo != ALGO_DIRECT) return CONV_ERR_UNSUPPORTED;
    // the workspace-taking entry points share the choice of their operation
    if (op == CONV_OP_FWD_WS) op = CONV_OP_FWD;
    if (op == CONV_OP_BWD_DATA_WS) op = CONV_OP_BWD_DATA;
    g_force[op].store(algo);
    return CONV_OK;
}

static int query_on(int op, const conv_desc_t* desc, const DevInfo& d, conv_plan_info_t* info)
{
    ConvParams p;
    int rc = make_params(desc, p);
    if (rc != CONV_OK) return rc;
    if (!info) return CONV_ERR_NULL;
    if (op < 0 || op > 6) return CONV_ERR_UNSUPPORTED;
    Plan pl;
    if ((rc = choose(op, p, desc->dtype, d, pl)) != CONV_OK) return rc;
    info->algo = pl.algo;
    info->launches = pl.launches;
    info->grid = pl.grid;
    info->block = pl.block;
    info->smem_bytes = pl.smem;
    info->splits = pl.splits;
    info->workspace = pl.workspace;
    return CONV_OK;
}

int conv_query(int op, const conv_desc_t* desc, conv_plan_info_t* info)
{
    ConvParams p;
    int rc = make_params(desc, p);
    if (rc != CONV_OK) return rc;
    if (!info) return CONV_ERR_NULL;
    if (op < 0 || op > 6) return CONV_ERR_UNSUPPORTED;
    DevInfo d;
    if ((rc = device_info(d)) != CONV_OK) return rc;
    return query_on(op, desc, d, info);
}

int conv_query_for_device(int op, const conv_desc_t* desc, int sms, int smem_optin, int cc_major, int cc_minor,
                          conv_plan_info_t* info)
{
    if (sms < 1 || smem_optin < 1 || cc_major < 1 || cc_minor < 0) return CONV_ERR_UNSUPPORTED;
    DevInfo d;
    d.device = -1;
    d.sms = sms;
    d.smem_optin = smem_optin;
    d.cc_major = cc_major;
    d.cc_minor = cc_minor;
    return query_on(op, desc, d, info);
}

int conv_fwd(const conv_desc_t* desc, const void* x, const void* w, void* y, conv_stream_t stream)
{
    return fwd_impl(desc, x, w, nullptr, y, nullptr, 0, false, stream);
}

int conv_fwd_bias(const conv_desc_t* desc, const void* x, const void* w, const void* bias, void* y,
                  conv_stream_t stream)
{
    ConvParams p;
    const int rc = make_params(desc, p);
    if (rc != CONV_OK) return rc;
    if (p.B > 0 && !bias) return CONV_ERR_NULL;
    return fwd_impl(desc, x, w, bias, y, nullptr, 0, false, stream);
}

size_t conv_fwd_workspace_size(const conv_desc_t* desc) { return plan_workspace(CONV_OP_FWD_WS, desc); }

int conv_fwd_ws(const conv_desc_t* desc, const void* x, const void* w, const void* bias, void* y, void* workspace,
                size_t workspace_bytes, conv_stream_t stream)
{
    return fwd_impl(desc, x, w, bias, y, workspace, workspace_bytes, true, stream);
}

size_t conv_bwd_data_workspace_size(const conv_desc_t* desc) { return plan_workspace(CONV_OP_BWD_DATA_WS, desc); }

int conv_bwd_data_ws(const conv_desc_t* desc, const void* dy, const void* w, const void* y, void* dx,
                     void* workspace, size_t workspace_bytes, conv_stream_t stream)
{
    return dgrad_impl(desc, dy, w, y, dx, workspace, workspace_bytes, true, stream);
}

int conv_bwd_bias(const conv_desc_t* desc, const void* dy, const void* y, void* db, conv_stream_t stream)
{
    ConvParams p;
    int rc = make_params(desc, p);
    if (rc != CONV_OK) return rc;
    if (!db) return CONV_ERR_NULL;
    if (p.B > 0 && (!dy || (p.relu && !y))) return CONV_ERR_NULL;
    if (!aligned16(db) || (p.B > 0 && (!aligned16(dy) || (p.relu && !aligned16(y))))) return CONV_ERR_ALIGN;
    DevInfo d;
    if ((rc = device_info(d)) != CONV_OK) return rc;
    Plan pl;
    if ((rc = choose_bgrad(p, desc->dtype, d, pl)) != CONV_OK) return rc;
    return cuda_status(run_bgrad(pl, p, desc->dtype, dy, y, db, reinterpret_cast<cudaStream_t>(stream)));
}

int conv_bwd_data(const conv_desc_t* desc, const void* dy, const void* w, const void* y, void* dx,
                  conv_stream_t stream)
{
    return dgrad_impl(desc, dy, w, y, dx, nullptr, 0, false, stream);
}

size_t conv_bwd_filter_workspace_size(const conv_desc_t* desc)
{
    ConvParams p;
    if (make_params(desc, p) != CONV_OK) return 0;
    DevInfo d;
    if (device_info(d) != CONV_OK) return 0;
    Plan pl;
    if (choose_wgrad(p, desc->dtype, d, pl) != CONV_OK) return 0;
    return pl.workspace;
}

namespace {

// Weight gradient, and with db != nullptr the bias gradient too (fused into the tensor-core
// wgrad: one read of dy and y for both; the other families run the bias-gradient kernel after).
int wgrad_impl(const conv_desc_t* desc, const void* x, const void* dy, const void* y, void* dw, void* db,
               void* workspace, size_t workspace_bytes, conv_stream_t stream)
{
    ConvParams p;
    int rc = make_params(desc, p);
    if (rc != CONV_OK) return rc;
    if (!dw) return CONV_ERR_NULL;
    if (p.B > 0 && (!x || !dy || (p.relu && !y))) return CONV_ERR_NULL;
    if (!aligned16(dw) || (db && !aligned16(db)) ||
        (p.B > 0 && (!aligned16(x) || !aligned16(dy) || (p.relu && !aligned16(y)))))
        return CONV_ERR_ALIGN;
    if (workspace && !aligned16(workspace)) return CONV_ERR_ALIGN;
    DevInfo d;
    if ((rc = device_info(d)) != CONV_OK) return rc;
    Plan pl;
    if ((rc = choose_wgrad(p, desc->dtype, d, pl)) != CONV_OK) return rc;
    if (pl.workspace > 0 && (!workspace || workspace_bytes < pl.workspace)) return CONV_ERR_WORKSPACE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (pl.algo == ALGO_TC)
        return cuda_status(run_wgrad_tc(pl, p, desc->dtype, x, dy, y, dw, workspace, db, s));
    cudaError_t e = pl.algo == ALGO_DIRECT ? run_wgrad_direct(pl, p, desc->dtype, x, dy, y, dw, s)
                                           : run_wgrad_ffma(pl, p, desc->dtype, x, dy, y, dw, workspace, s);
    if (e == cudaSuccess && db) {
        Plan bp;
        if ((rc = choose_bgrad(p, desc->dtype, d, bp)) != CONV_OK) return rc;
        e = run_bgrad(bp, p, desc->dtype, dy, y, db, s);
    }
    return cuda_status(e);
}

}  // namespace

int conv_bwd_filter(const conv_desc_t* desc, const void* x, const void* dy, const void* y, void* dw,
                    void* workspace, size_t workspace_bytes, conv_stream_t stream)
{
    return wgrad_impl(desc, x, dy, y, dw, nullptr, workspace, workspace_bytes, stream);
}

int conv_bwd_filter_bias(const conv_desc_t* desc, const void* x, const void* dy, const void* y, void* dw, void* db,
                         void* workspace, size_t workspace_bytes, conv_stream_t stream)
{
    if (!db && desc) return CONV_ERR_NULL;
    return wgrad_impl(desc, x, dy, y, dw, db, workspace, workspace_bytes, stream);
}

namespace {

// Two descriptors that chain: layer 2's input is layer 1's output.
int chain_params(const conv_desc_t* d1, const conv_desc_t* d2, ConvParams& p1, ConvParams& p2)
{
    int rc = make_params(d1, p1);
    if (rc != CONV_OK) return rc;
    if ((rc = make_params(d2, p2)) != CONV_OK) return rc;
    if (d1->B != d2->B || d1->dtype != d2->dtype || d2->IC != d1->OC || d2->H != p1.OH || d2->W != p1.OW)
        return CONV_ERR_DESC;
    return CONV_OK;
}

// Fused when every CTA gets at most one group of samples (measured on a GB300: with more groups
// per CTA the layer-2 phase, which cannot overlap the next group's layer-1 tile, costs more than
// layer 2's own forward call); otherwise the two forward calls with the workspace path, sharing
// one workspace of the larger size.
int chain_plan(const ConvParams& p1, const ConvParams& p2, int dt, const DevInfo& d, Plan& pl)
{
    // Fused at most one group of samples per CTA, in bf16 (in fp32 the two forward calls were
    // measured faster: 72.9 against 75.7 us at B = 1024) unless the tensor-core family is forced.
    const int f = g_force[CONV_OP_FWD].load();
    if ((f == ALGO_TC || (f == ALGO_AUTO && dt == DT_BF16)) && tc_chain_ok(p1, p2, dt, d)) {
        pl = plan_chain_tc(p1, p2, dt, d);
        if (chain_groups(p1, p2) <= d.sms) return CONV_OK;  // at most one group per CTA
    }
    Plan a, b;
    int rc = choose_fwd(p1, dt, d, true, a);
    if (rc == CONV_OK) rc = choose_fwd(p2, dt, d, true, b);
    if (rc != CONV_OK) return rc;
    pl = Plan();
    pl.algo = ALGO_AUTO;  // not fused: two forward calls
    pl.launches = a.launches + b.launches;
    pl.grid = std::max(a.grid, b.grid);
    pl.block = std::max(a.block, b.block);
    pl.smem = std::max(a.smem, b.smem);
    pl.workspace = std::max(a.workspace, b.workspace);
    return CONV_OK;
}

}  // namespace

size_t conv_fwd_chain2_workspace_size(const conv_desc_t* d1, const conv_desc_t* d2)
{
    ConvParams p1, p2;
    if (chain_params(d1, d2, p1, p2) != CONV_OK) return 0;
    DevInfo d;
    if (device_info(d) != CONV_OK) return 0;
    Plan pl;
    if (chain_plan(p1, p2, d1->dtype, d, pl) != CONV_OK) return 0;
    return pl.workspace;
}

int conv_fwd_chain2(const conv_desc_t* d1, const conv_desc_t* d2, const void* x, const void* w1, const void* bias1,
                    const void* w2, const void* bias2, void* y1, void* y2, void* workspace, size_t workspace_bytes,
                    conv_stream_t stream)
{
    if (!d1 || !d2) return CONV_ERR_NULL;
    ConvParams p1, p2;
    int rc = chain_params(d1, d2, p1, p2);
    if (rc != CONV_OK) return rc;
    if (p1.B == 0) return CONV_OK;
    if (!x || !w1 || !w2 || !y1 || !y2) return CONV_ERR_NULL;
    if (!aligned16(x) || !aligned16(w1) || !aligned16(w2) || !aligned16(y1) || !aligned16(y2) ||
        (bias1 && !aligned16(bias1)) || (bias2 && !aligned16(bias2)) || (workspace && !aligned16(workspace)))
        return CONV_ERR_ALIGN;
    DevInfo d;
    if ((rc = device_info(d)) != CONV_OK) return rc;
    Plan pl;
    if ((rc = chain_plan(p1, p2, d1->dtype, d, pl)) != CONV_OK) return rc;
    if (pl.algo != ALGO_TC) {  // the two layers one after the other, through the workspace path
        if (pl.workspace > 0 && (!workspace || workspace_bytes < pl.workspace)) return CONV_ERR_WORKSPACE;
        if ((rc = fwd_impl(d1, x, w1, bias1, y1, workspace, workspace_bytes, true, stream)) != CONV_OK) return rc;
        return fwd_impl(d2, y1, w2, bias2, y2, workspace, workspace_bytes, true, stream);
    }
    if (!workspace || workspace_bytes < pl.workspace) return CONV_ERR_WORKSPACE;
    return cuda_status(run_chain_tc(pl, p1, p2, d1->dtype, x, w1, bias1, w2, bias2, y1, y2, workspace,
                                    reinterpret_cast<cudaStream_t>(stream)));
}

int conv_query_chain2(const conv_desc_t* d1, const conv_desc_t* d2, conv_plan_info_t* info)
{
    ConvParams p1, p2;
    int rc = chain_params(d1, d2, p1, p2);
    if (rc != CONV_OK) return rc;
    if (!info) return CONV_ERR_NULL;
    DevInfo d;
    if ((rc = device_info(d)) != CONV_OK) return rc;
    Plan pl;
    if ((rc = chain_plan(p1, p2, d1->dtype, d, pl)) != CONV_OK) return rc;
    info->algo = pl.algo;
    info->launches = pl.launches;
    info->grid = pl.grid;
    info->block = pl.block;
    info->smem_bytes = pl.smem;
    info->splits = pl.splits;
    info->workspace = pl.workspace;
    return CONV_OK;
}

size_t conv_bwd_workspace_size(const conv_desc_t* desc) { return plan_workspace(CONV_OP_BWD, desc); }

int conv_bwd(const conv_desc_t* desc, const void* x, const void* dy, const void* w, const void* y, void* dx,
             void* dw, void* db, void* workspace, size_t workspace_bytes, conv_stream_t stream)
{
    ConvParams p;
    int rc = make_params(desc, p);
    if (rc != CONV_OK) return rc;
    if (!dw || !w) return CONV_ERR_NULL;
    if (p.B > 0 && (!x || !dy || !dx || (p.relu && !y))) return CONV_ERR_NULL;
    if (!aligned16(dw) || !aligned16(w) || (db && !aligned16(db)) || (workspace && !aligned16(workspace)) ||
        (p.B > 0 && (!aligned16(x) || !aligned16(dy) || !aligned16(dx) || (p.relu && !aligned16(y)))))
        return CONV_ERR_ALIGN;
    DevInfo d;
    if ((rc = device_info(d)) != CONV_OK) return rc;
    Plan pl;
    if ((rc = choose_bwd(p, desc->dtype, d, pl)) != CONV_OK) return rc;
    if (pl.workspace > 0 && (!workspace || workspace_bytes < pl.workspace)) return CONV_ERR_WORKSPACE;
    if (pl.algo == ALGO_TC)
        return cuda_status(run_bwd_tc(pl, p, desc->dtype, d, x, dy, w, y, dx, dw, db, workspace,
                                      reinterpret_cast<cudaStream_t>(stream)));
    // two calls: d_input's workspace first, wgrad's after it
    Plan a;
    if ((rc = choose_dgrad(p, desc->dtype, d, true, a)) != CONV_OK) return rc;
    const size_t off = (a.workspace + 255) / 256 * 256;
    if ((rc = dgrad_impl(desc, dy, w, y, dx, workspace, a.workspace, true, stream)) != CONV_OK) return rc;
    unsigned char* wws = workspace ? static_cast<unsigned char*>(workspace) + off : nullptr;
    return wgrad_impl(desc, x, dy, y, dw, db, wws, workspace_bytes > off ? workspace_bytes - off : 0, stream);
}

namespace {

// The backward chain's workspace: layer 2's dx (layer 1's dy) first, then the larger of the
// workspaces its calls need (layer 2's conv_bwd, layer 1's conv_bwd or conv_bwd_filter), used
// one call after the other.
size_t bwd_chain_dx2_bytes(const conv_desc_t* d2)
{
    const size_t es = d2->dtype == CONV_BF16 ? 2 : 4;
    return (size_t(d2->B) * d2->IC * d2->H * d2->W * es + 255) / 256 * 256;
}

size_t bwd_chain_call_ws(const conv_desc_t* d1, const conv_desc_t* d2)
{
    return std::max(plan_workspace(CONV_OP_BWD, d2),
                    std::max(plan_workspace(CONV_OP_BWD, d1), plan_workspace(CONV_OP_BWD_FILTER, d1)));
}

}  // namespace

size_t conv_bwd_chain2_workspace_size(const conv_desc_t* d1, const conv_desc_t* d2)
{
    ConvParams p1, p2;
    if (chain_params(d1, d2, p1, p2) != CONV_OK) return 0;
    return bwd_chain_dx2_bytes(d2) + bwd_chain_call_ws(d1, d2);
}

int conv_bwd_chain2(const conv_desc_t* d1, const conv_desc_t* d2, const void* x1, const void* w1, const void* y1,
                    const void* w2, const void* y2, const void* dy2, void* dx1, void* dw1, void* db1, void* dw2,
                    void* db2, void* workspace, size_t workspace_bytes, conv_stream_t stream)
{
    if (!d1 || !d2) return CONV_ERR_NULL;
    ConvParams p1, p2;
    int rc = chain_params(d1, d2, p1, p2);
    if (rc != CONV_OK) return rc;
    if (!w1 || !w2 || !dw1 || !dw2) return CONV_ERR_NULL;
    if (p1.B > 0 && (!x1 || !y1 || !dy2 || (p2.relu && !y2))) return CONV_ERR_NULL;
    if (workspace && !aligned16(workspace)) return CONV_ERR_ALIGN;
    const size_t dx2_bytes = bwd_chain_dx2_bytes(d2), need = dx2_bytes + bwd_chain_call_ws(d1, d2);
    if (need > 0 && (!workspace || workspace_bytes < need)) return CONV_ERR_WORKSPACE;
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    void* dx2 = ws;
    void* rest = ws ? ws + dx2_bytes : nullptr;
    const size_t rest_bytes = ws ? workspace_bytes - dx2_bytes : 0;
    // layer 2: x = y1, the mask source y2
    if ((rc = conv_bwd(d2, y1, dy2, w2, y2, dx2, dw2, db2, rest, rest_bytes, stream)) != CONV_OK) return rc;
    // layer 1 on dy = dx2, masked by y1; its d_input only when dx1 is wanted
    if (dx1) return conv_bwd(d1, x1, dx2, w1, y1, dx1, dw1, db1, rest, rest_bytes, stream);
    return wgrad_impl(d1, x1, dx2, y1, dw1, db1, rest, rest_bytes, stream);
}

uint64_t conv_fastdivmod_check(uint32_t d, uint32_t lo, uint32_t hi)
{
    if (d < 1 || d >= (1u << 31)) return ~uint64_t(0);
    const FastDivmod f(d);
    uint64_t bad = 0;
    if (hi > (1u << 31)) hi = 1u << 31;
    for (uint32_t n = lo; n < hi; ++n) {
        uint32_t q, r;
        f.divmod(n, q, r);
        bad += (q != n / d) | (r != n % d);
    }
    return bad;
}

int conv_device_status(uint32_t* status, int reset)
{
    if (!status) return CONV_ERR_NULL;
    unsigned v = 0, w = 0;
    if (tc_read_status(&v, reset != 0) != cudaSuccess || diag_read_status(&w, reset != 0) != cudaSuccess) {
        cudaGetLastError();
        return CONV_ERR_CUDA;
    }
    *status = v | w;
    return CONV_OK;
}

int conv_wait_selftest(uint32_t max_sleeps, conv_stream_t stream)
{
    if (max_sleeps < 1 || max_sleeps > 1000000u) return CONV_ERR_UNSUPPORTED;
    return cuda_status(run_wait_selftest(max_sleeps, reinterpret_cast<cudaStream_t>(stream)));
}

int conv_l2_flush(void* buf, size_t bytes, conv_stream_t stream)
{
    if (!buf) return CONV_ERR_NULL;
    if (!aligned16(buf) || (bytes & 15u)) return CONV_ERR_ALIGN;
    return cuda_status(run_l2_flush(buf, bytes, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
