// kernels_ffma.cu -- fp32 FFMA register-tiled implicit-GEMM kernels (forward,
// d_input, wgrad split-K partials), the deterministic split-K reduction, and
// the one-thread-per-output "direct" kernels that accept any shape.
//
// The GEMM views (n = (b, oh, ow) a column, k = (ic, kh, kw) a reduction
// index, P = OH*OW, Kred = IC*K*K), per PufferLib PR #522's forward /
// backward d_input / backward wgrad results:
//   forward   y[oc, n]   = act( sum_k w[oc, k] * X[k, n] ),  X[k, n] = x[col_base(n) + k_offset(k)]
//   d_input   D[k, n]    = sum_oc w[oc, k] * g[oc, n],  then dx[col_base(n) + k_offset(k)] += D[k, n]
//   wgrad     dw[oc, k]  = sum_n g[oc, n] * X[k, n]  (split-K over n, summed in a second pass)
// Both dtypes run here: bf16 operands are widened to fp32 on load; results are
// rounded once on store.  Every sum has a fixed order, so results are
// bit-reproducible.
#include <algorithm>

#include "internal.h"

namespace igc {
namespace {

// ======================================================================================
// Forward.  Each warp owns a contiguous range of columns (balanced over all warps of the
// persistent grid) and walks it in sub-tiles of FW_NCOL columns; each lane owns four
// output channels (lane + 32 j), so a thread keeps 4 x 12 accumulators.  The weight chunk
// (128 oc x 32 k) is shared by the CTA; each warp gathers its own patch chunk
// (12 columns x 32 k) through the per-CTA k-offset table.  Both are double-buffered
// through registers.
// ======================================================================================
constexpr int FW_WARPS = 8, FW_THREADS = FW_WARPS * 32;
constexpr int FW_NCOL = 12, FW_OCT = 128, FW_KC = 32, FW_KCP = FW_KC + 4;

__host__ __device__ inline int fw_kred_pad(int kred) { return (kred + FW_KC - 1) / FW_KC * FW_KC; }
inline int fw_smem(const ConvParams& p)
{
    return fw_kred_pad(p.Kred) * 4 + 2 * FW_OCT * FW_KCP * 4 + 2 * FW_WARPS * FW_NCOL * FW_KCP * 4;
}

template <typename T, bool RELU>
__global__ void __launch_bounds__(FW_THREADS, 1)
fwd_ffma_kernel(const ConvParams p, const T* __restrict__ x, const T* __restrict__ w,
                const T* __restrict__ bias, T* __restrict__ y)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int kred_pad = fw_kred_pad(p.Kred);
    int* offk = reinterpret_cast<int*>(smem_raw);
    float* Ws = reinterpret_cast<float*>(offk + kred_pad);
    float* Xs = Ws + 2 * FW_OCT * FW_KCP;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    for (int k = tid; k < kred_pad; k += FW_THREADS) offk[k] = (k < p.Kred) ? k_offset(p, k) : -1;

    const int oc0 = blockIdx.y * FW_OCT;
    const long long Gw = (long long)gridDim.x * FW_WARPS;
    const long long gw = (long long)blockIdx.x * FW_WARPS + warp;
    const int c_lo = int((long long)p.N * gw / Gw);
    const int c_hi = int((long long)p.N * (gw + 1) / Gw);
    const int per_max = int((p.N + Gw - 1) / Gw);
    const int rounds = (per_max + FW_NCOL - 1) / FW_NCOL;
    const int nchunks = kred_pad / FW_KC;
    __syncthreads();

    float wreg[16], xreg[FW_NCOL];
    for (int r = 0; r < rounds; ++r) {
        const int cs = c_lo + r * FW_NCOL;
        const int ncol = max(0, min(FW_NCOL, c_hi - cs));
        const int my_cb = (lane < ncol) ? col_base(p, cs + lane) : -1;

        auto load_chunk = [&](int kc) {
            const int ok = offk[kc * FW_KC + lane];
            const int k = kc * FW_KC + lane;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int oc = oc0 + warp * 16 + i;
                wreg[i] = (ok >= 0 && oc < p.OC) ? Elem<T>::ldg(w + size_t(oc) * p.Kred + k) : 0.f;
            }
#pragma unroll
            for (int c = 0; c < FW_NCOL; ++c) {
                const int cb = __shfl_sync(0xffffffffu, my_cb, c);
                xreg[c] = (ok >= 0 && cb >= 0) ? Elem<T>::ldg(x + cb + ok) : 0.f;
            }
        };
        auto store_chunk = [&](int buf) {
            float* wsm = Ws + buf * FW_OCT * FW_KCP;
#pragma unroll
            for (int i = 0; i < 16; ++i) wsm[(warp * 16 + i) * FW_KCP + lane] = wreg[i];
            float* xsm = Xs + (buf * FW_WARPS + warp) * FW_NCOL * FW_KCP;
#pragma unroll
            for (int c = 0; c < FW_NCOL; ++c) xsm[c * FW_KCP + lane] = xreg[c];
        };

        float acc[4][FW_NCOL];
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int c = 0; c < FW_NCOL; ++c) acc[j][c] = 0.f;

        load_chunk(0);
        store_chunk(0);
        __syncthreads();
        for (int kc = 0; kc < nchunks; ++kc) {
            const bool more = kc + 1 < nchunks;
            if (more) load_chunk(kc + 1);
            const float* wsm = Ws + (kc & 1) * FW_OCT * FW_KCP;
            const float* xsm = Xs + ((kc & 1) * FW_WARPS + warp) * FW_NCOL * FW_KCP;
#pragma unroll 1
            for (int kq = 0; kq < FW_KC / 4; ++kq) {
                float4 wv[4];
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    wv[j] = *reinterpret_cast<const float4*>(wsm + (lane + 32 * j) * FW_KCP + 4 * kq);
#pragma unroll
                for (int c = 0; c < FW_NCOL; ++c) {
                    const float4 xv = *reinterpret_cast<const float4*>(xsm + c * FW_KCP + 4 * kq);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        acc[j][c] = fmaf(wv[j].x, xv.x, acc[j][c]);
                        acc[j][c] = fmaf(wv[j].y, xv.y, acc[j][c]);
                        acc[j][c] = fmaf(wv[j].z, xv.z, acc[j][c]);
                        acc[j][c] = fmaf(wv[j].w, xv.w, acc[j][c]);
                    }
                }
            }
            if (more) store_chunk((kc + 1) & 1);
            __syncthreads();
        }

#pragma unroll
        for (int c = 0; c < FW_NCOL; ++c) {
            if (c < ncol) {
                const int ob = col_out(p, cs + c);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int oc = oc0 + lane + 32 * j;
                    if (oc < p.OC) {
                        float v = acc[j][c];
                        if (bias) v += Elem<T>::ldg(bias + oc);
                        if (RELU) v = v > 0.f ? v : 0.f;
                        Elem<T>::st(y + ob + size_t(oc) * p.P, v);
                    }
                }
            }
        }
    }
}

// ======================================================================================
// d_input.  A unit is (8 sample groups, one channel chunk): the CTA's warps each take a
// sample group (NS whole samples, NS*P <= 12 columns) and share the weight sub-chunks
// (32 oc x 128 k) of the chunk's CIC channels (CIC*K*K <= 128 k).  Each lane owns k =
// lane + 32 i (i < 4) for all 12 columns; after the oc loop the warp writes its 12 x 128
// patch-gradient tile to shared memory and scatters it back (col2im) as a gather: every
// dx element sums its (oh,kh) x (ow,kw) contributions in a fixed order.
// ======================================================================================
constexpr int DG_WARPS = 8, DG_THREADS = DG_WARPS * 32;
constexpr int DG_NCOL = 12, DG_KT = 128, DG_OCC = 32;

struct DgradGeom {
    int NS;      // samples per warp group
    int CIC;     // channels per chunk
    int NKC;     // channel chunks
    int NG;      // sample groups
    int units;   // ceil(NG / 8) * NKC
    int ocpad;   // OC rounded up to DG_OCC
    int rmax;    // max (oh,kh) pairs per input row = ceil(K / S)
};

inline DgradGeom dgrad_geom(const ConvParams& p)
{
    DgradGeom g;
    g.NS = std::max(1, DG_NCOL / std::max(1, p.P));
    g.CIC = std::max(1, DG_KT / p.KK);
    g.NKC = ceil_div(p.IC, g.CIC);
    g.NG = ceil_div(p.B, g.NS);
    g.units = ceil_div(g.NG, DG_WARPS) * g.NKC;
    g.ocpad = round_up(p.OC, DG_OCC);
    g.rmax = (p.K + p.S - 1) / p.S;
    return g;
}

inline int dg_smem(const ConvParams& p, const DgradGeom& g)
{
    return 2 * DG_OCC * DG_KT * 4                   // weight sub-chunks
           + DG_WARPS * g.ocpad * DG_NCOL * 4       // g tiles
           + DG_WARPS * DG_NCOL * DG_KT * 4         // patch-gradient tiles
           + (p.H + p.W) * (1 + g.rmax) * 8;        // col2im row / column tables
}

template <typename T, bool RELU>
__global__ void __launch_bounds__(DG_THREADS, 1)
dgrad_ffma_kernel(const ConvParams p, const T* __restrict__ dy, const T* __restrict__ w,
                  const T* __restrict__ y, T* __restrict__ dx, const DgradGeom geo)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    float* Ws = reinterpret_cast<float*>(smem_raw);
    float* Gs = Ws + 2 * DG_OCC * DG_KT;
    float* Ds = Gs + DG_WARPS * geo.ocpad * DG_NCOL;
    int2* rtab = reinterpret_cast<int2*>(Ds + DG_WARPS * DG_NCOL * DG_KT);  // [H][1 + rmax]
    int2* ctab = rtab + p.H * (1 + geo.rmax);                             // [W][1 + rmax]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int R1 = 1 + geo.rmax;
    // (oh, kh) pairs with oh*S + kh = h, stored as (oh*OW, kh*K); entry 0 holds the count.
    for (int h = tid; h < p.H; h += DG_THREADS) {
        int n = 0;
        for (int oh = 0; oh < p.OH; ++oh) {
            const int kh = h - oh * p.S;
            if (kh >= 0 && kh < p.K) rtab[h * R1 + 1 + n++] = make_int2(oh * p.OW, kh * p.K);
        }
        rtab[h * R1] = make_int2(n, 0);
    }
    for (int c = tid; c < p.W; c += DG_THREADS) {
        int n = 0;
        for (int ow = 0; ow < p.OW; ++ow) {
            const int kw = c - ow * p.S;
            if (kw >= 0 && kw < p.K) ctab[c * R1 + 1 + n++] = make_int2(ow, kw);
        }
        ctab[c * R1] = make_int2(n, 0);
    }

    const int NOC = geo.ocpad / DG_OCC;
    const int u_lo = int((long long)geo.units * blockIdx.x / gridDim.x);
    const int u_hi = int((long long)geo.units * (blockIdx.x + 1) / gridDim.x);
    const int stages = (u_hi - u_lo) * NOC;
    const int kspan = geo.CIC * p.KK;

    float wreg[16];
    auto load_w = [&](int st) {
        const int u = u_lo + st / NOC, oi = st % NOC;
        const int kc = u % geo.NKC;
        const int k0 = kc * kspan;
        const int kend = min(p.Kred, k0 + kspan);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int idx = tid + DG_THREADS * i;
            const int o = idx / DG_KT, kk = idx % DG_KT;
            const int oc = oi * DG_OCC + o, k = k0 + kk;
            wreg[i] = (oc < p.OC && k < kend) ? Elem<T>::ldg(w + size_t(oc) * p.Kred + k) : 0.f;
        }
    };
    auto store_w = [&](int buf) {
        float* wsm = Ws + buf * DG_OCC * DG_KT;
#pragma unroll
        for (int i = 0; i < 16; ++i) wsm[tid + DG_THREADS * i] = wreg[i];
    };

    __syncthreads();
    if (stages > 0) {
        load_w(0);
        store_w(0);
    }
    __syncthreads();

    float acc[4][DG_NCOL];
    int cur_gb = -1;
    float* gsm = Gs + warp * geo.ocpad * DG_NCOL;
    float* dsm = Ds + warp * DG_NCOL * DG_KT;
    for (int st = 0; st < stages; ++st) {
        const int u = u_lo + st / NOC, oi = st % NOC;
        const int gb = u / geo.NKC, kc = u % geo.NKC;
        const int sg = gb * DG_WARPS + warp;  // this warp's sample group
        const int b0 = sg * geo.NS;
        const int nsamp = max(0, min(geo.NS, p.B - b0));
        if (oi == 0) {
            if (gb != cur_gb) {
                // g tile [oc][c], c = s*P + p, from the contiguous dy slab of the group.
                const int ncols = nsamp * p.P;
                for (int t = lane; t < geo.ocpad * DG_NCOL; t += 32) {
                    const int oc = t / DG_NCOL, c = t % DG_NCOL;
                    float v = 0.f;
                    if (oc < p.OC && c < ncols) {
                        const int s = c / p.P, pp = c % p.P;
                        const size_t gi = size_t(b0 + s) * p.OCP + size_t(oc) * p.P + pp;
                        v = Elem<T>::ldg(dy + gi);
                        if (RELU && !(Elem<T>::ldg(y + gi) > 0.f)) v = 0.f;
                    }
                    gsm[t] = v;
                }
                cur_gb = gb;
                __syncwarp();
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int c = 0; c < DG_NCOL; ++c) acc[i][c] = 0.f;
        }
        const bool more = st + 1 < stages;
        if (more) load_w(st + 1);

        const float* wsm = Ws + (st & 1) * DG_OCC * DG_KT;
        const float* g0 = gsm + oi * DG_OCC * DG_NCOL;
#pragma unroll 4
        for (int o = 0; o < DG_OCC; ++o) {
            float wv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) wv[i] = wsm[o * DG_KT + lane + 32 * i];
#pragma unroll
            for (int cq = 0; cq < DG_NCOL / 4; ++cq) {
                const float4 gv = *reinterpret_cast<const float4*>(g0 + o * DG_NCOL + 4 * cq);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    acc[i][4 * cq + 0] = fmaf(wv[i], gv.x, acc[i][4 * cq + 0]);
                    acc[i][4 * cq + 1] = fmaf(wv[i], gv.y, acc[i][4 * cq + 1]);
                    acc[i][4 * cq + 2] = fmaf(wv[i], gv.z, acc[i][4 * cq + 2]);
                    acc[i][4 * cq + 3] = fmaf(wv[i], gv.w, acc[i][4 * cq + 3]);
                }
            }
        }

        if (oi == NOC - 1 && nsamp > 0) {
            // Patch-gradient tile -> shared memory, then gather into dx.
#pragma unroll
            for (int c = 0; c < DG_NCOL; ++c)
#pragma unroll
                for (int i = 0; i < 4; ++i) dsm[c * DG_KT + lane + 32 * i] = acc[i][c];
            __syncwarp();
            const int ic0 = kc * geo.CIC;
            const int nic = min(geo.CIC, p.IC - ic0);
            const int span = nic * p.HW;
            for (int s = 0; s < nsamp; ++s) {
                T* dxs = dx + size_t(b0 + s) * p.IHW + size_t(ic0) * p.HW;
                const float* ds = dsm + s * p.P * DG_KT;
                for (int t = lane; t < span; t += 32) {
                    uint32_t icl, hw, h, ww;
                    p.dm_HW.divmod(uint32_t(t), icl, hw);
                    p.dm_W.divmod(hw, h, ww);
                    const int2* rr = rtab + h * R1;
                    const int2* cc = ctab + ww * R1;
                    const int nr = rr[0].x, ncc = cc[0].x;
                    const int kb = int(icl) * p.KK;
                    float sum = 0.f;
                    for (int a = 1; a <= nr; ++a)
                        for (int bq = 1; bq <= ncc; ++bq)
                            sum += ds[(rr[a].x + cc[bq].x) * DG_KT + kb + rr[a].y + cc[bq].y];
                    Elem<T>::st(dxs + t, sum);
                }
            }
            __syncwarp();
        }

        if (more) store_w((st + 1) & 1);
        __syncthreads();
    }
}

// ======================================================================================
// wgrad partials.  CTA tile 128 oc x 128 k, 16 x 16 threads with 8 x 8 accumulators
// each; the CTA sums the columns n of its split range in ascending order, 16 at a time,
// from shared-memory stages of g (masked dy) and gathered patches, double-buffered
// through registers.  Partials go to ws[split][oc][k] (row stride kpad, fp32).
// ======================================================================================
constexpr int WG_THREADS = 256, WG_TM = 128, WG_TN = 128, WG_NC = 16, WG_LD = 132;

inline int wg_smem() { return WG_TN * 4 + 2 * WG_NC * WG_LD * 4 * 2; }

template <typename T, bool RELU>
__global__ void __launch_bounds__(WG_THREADS, 2)
wgrad_ffma_kernel(const ConvParams p, const T* __restrict__ x, const T* __restrict__ dy,
                  const T* __restrict__ y, float* __restrict__ ws, int splits, int kpad,
                  int tiles_k)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    int* offk = reinterpret_cast<int*>(smem_raw);
    float* Gs = reinterpret_cast<float*>(offk + WG_TN);  // [2][NC][LD] (oc)
    float* Xs = Gs + 2 * WG_NC * WG_LD;                   // [2][NC][LD] (k)

    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int tile = blockIdx.x, split = blockIdx.y;
    const int oc0 = (tile / tiles_k) * WG_TM, k0 = (tile % tiles_k) * WG_TN;
    const int n_lo = int((long long)p.N * split / splits);
    const int n_hi = int((long long)p.N * (split + 1) / splits);
    for (int kk = tid; kk < WG_TN; kk += WG_THREADS)
        offk[kk] = (k0 + kk < p.Kred) ? k_offset(p, k0 + kk) : -1;
    __syncthreads();

    float greg[8], xreg[8];
    auto load = [&](int n0) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int idx = tid + WG_THREADS * i;
            const int c = idx % WG_NC, o = idx / WG_NC;
            const int n = n0 + c, oc = oc0 + o;
            float v = 0.f;
            if (n < n_hi && oc < p.OC) {
                const size_t gi = size_t(col_out(p, n)) + size_t(oc) * p.P;
                v = Elem<T>::ldg(dy + gi);
                if (RELU && !(Elem<T>::ldg(y + gi) > 0.f)) v = 0.f;
            }
            greg[i] = v;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int idx = tid + WG_THREADS * i;
            const int kk = idx % WG_TN, c = idx / WG_TN;
            const int n = n0 + c;
            const int ok = offk[kk];
            xreg[i] = (n < n_hi && ok >= 0) ? Elem<T>::ldg(x + col_base(p, n) + ok) : 0.f;
        }
    };
    auto store = [&](int buf) {
        float* gs = Gs + buf * WG_NC * WG_LD;
        float* xs = Xs + buf * WG_NC * WG_LD;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int idx = tid + WG_THREADS * i;
            gs[(idx % WG_NC) * WG_LD + idx / WG_NC] = greg[i];
            xs[(idx / WG_TN) * WG_LD + idx % WG_TN] = xreg[i];
        }
    };

    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

    const int stages = (n_hi - n_lo + WG_NC - 1) / WG_NC;
    if (stages > 0) {
        load(n_lo);
        store(0);
    }
    __syncthreads();
    for (int st = 0; st < stages; ++st) {
        const bool more = st + 1 < stages;
        if (more) load(n_lo + (st + 1) * WG_NC);
        const float* gs = Gs + (st & 1) * WG_NC * WG_LD;
        const float* xs = Xs + (st & 1) * WG_NC * WG_LD;
#pragma unroll 4
        for (int c = 0; c < WG_NC; ++c) {
            const float4 a0 = *reinterpret_cast<const float4*>(gs + c * WG_LD + ty * 4);
            const float4 a1 = *reinterpret_cast<const float4*>(gs + c * WG_LD + 64 + ty * 4);
            const float4 b0 = *reinterpret_cast<const float4*>(xs + c * WG_LD + tx * 4);
            const float4 b1 = *reinterpret_cast<const float4*>(xs + c * WG_LD + 64 + tx * 4);
            const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
        }
        if (more) store((st + 1) & 1);
        __syncthreads();
    }

#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int oc = oc0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + (i - 4));
        if (oc >= p.OC) continue;
        float* row = ws + (size_t(split) * p.OC + oc) * kpad;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int k = k0 + h * 64 + tx * 4;
            if (k < kpad)
                *reinterpret_cast<float4*>(row + k) =
                    make_float4(acc[i][4 * h], acc[i][4 * h + 1], acc[i][4 * h + 2], acc[i][4 * h + 3]);
        }
    }
}

// Also, when db is given, the bias gradient: db[oc] = sum of the nbp per-(split, lane group)
// partial channel sums bpart[q][oc] in ascending q (the tensor-core wgrad accumulates them
// from the masked g it already loads).
template <typename T>
__global__ void wgrad_reduce_kernel(const float* __restrict__ ws, int splits, int kpad, int OC,
                                    int Kred, FastDivmod dm_kred, T* __restrict__ dw, const float* __restrict__ bpart,
                                    int nbp, T* __restrict__ db)
{
    // When launched to overlap the partials kernel: wait for it (at once otherwise).
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (db) {
        const int oc = blockIdx.x * blockDim.x + threadIdx.x;  // the grid covers OC*Kred >= OC threads
        if (oc < OC) {
            float s = 0.f;
            for (int q = 0; q < nbp; ++q) s += __ldcg(bpart + size_t(q) * OC + oc);
            Elem<T>::st(db + oc, s);
        }
    }
    const int total = OC * Kred;
    const size_t sstride = size_t(OC) * kpad;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
        uint32_t oc, k;
        dm_kred.divmod(uint32_t(i), oc, k);
        const float* src = ws + size_t(oc) * kpad + k;
        // Loads in groups of 8 issued together, added in ascending split order.
        float s = 0.f;
        int sp = 0;
        for (; sp + 8 <= splits; sp += 8) {
            float v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) v[u] = __ldcg(src + size_t(sp + u) * sstride);
#pragma unroll
            for (int u = 0; u < 8; ++u) s += v[u];
        }
        for (; sp < splits; ++sp) s += __ldcg(src + size_t(sp) * sstride);
        Elem<T>::st(dw + i, s);
    }
}

// ======================================================================================
// Direct kernels: one thread per output element, the sum in the definition's order.
// ======================================================================================
template <typename T, bool RELU>
__global__ void fwd_direct_kernel(const ConvParams p, const T* __restrict__ x,
                                  const T* __restrict__ w, const T* __restrict__ bias, T* __restrict__ y)
{
    const int total = p.B * p.OCP;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
        const int b = i / p.OCP, r = i % p.OCP;
        const int oc = r / p.P, pp = r % p.P;
        const int oh = pp / p.OW, ow = pp % p.OW;
        const T* xb = x + size_t(b) * p.IHW + oh * p.S * p.W + ow * p.S;
        const T* wo = w + size_t(oc) * p.Kred;
        float acc = 0.f;
        for (int ic = 0; ic < p.IC; ++ic)
            for (int kh = 0; kh < p.K; ++kh)
                for (int kw = 0; kw < p.K; ++kw)
                    acc = fmaf(Elem<T>::ldg(wo + (ic * p.K + kh) * p.K + kw),
                               Elem<T>::ldg(xb + ic * p.HW + kh * p.W + kw), acc);
        if (bias) acc += Elem<T>::ldg(bias + oc);
        if (RELU) acc = acc > 0.f ? acc : 0.f;
        Elem<T>::st(y + i, acc);
    }
}

template <typename T, bool RELU>
__global__ void dgrad_direct_kernel(const ConvParams p, const T* __restrict__ dy,
                                    const T* __restrict__ w, const T* __restrict__ y,
                                    T* __restrict__ dx)
{
    const int total = p.B * p.IHW;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
        const int b = i / p.IHW, r = i % p.IHW;
        const int ic = r / p.HW, hw = r % p.HW;
        const int h = hw / p.W, ww = hw % p.W;
        float acc = 0.f;
        for (int oc = 0; oc < p.OC; ++oc)
            for (int kh = 0; kh < p.K; ++kh) {
                const int th = h - kh;
                if (th < 0 || th % p.S != 0 || th / p.S >= p.OH) continue;
                for (int kw = 0; kw < p.K; ++kw) {
                    const int tw = ww - kw;
                    if (tw < 0 || tw % p.S != 0 || tw / p.S >= p.OW) continue;
                    const size_t gi = size_t(b) * p.OCP + size_t(oc) * p.P + (th / p.S) * p.OW + tw / p.S;
                    float g = Elem<T>::ldg(dy + gi);
                    if (RELU && !(Elem<T>::ldg(y + gi) > 0.f)) g = 0.f;
                    acc = fmaf(g, Elem<T>::ldg(w + ((size_t(oc) * p.IC + ic) * p.K + kh) * p.K + kw), acc);
                }
            }
        Elem<T>::st(dx + i, acc);
    }
}

template <typename T, bool RELU>
__global__ void wgrad_direct_kernel(const ConvParams p, const T* __restrict__ x,
                                    const T* __restrict__ dy, const T* __restrict__ y,
                                    T* __restrict__ dw)
{
    const int total = p.OC * p.Kred;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
        const int oc = i / p.Kred, k = i % p.Kred;
        const int ic = k / p.KK, r = k % p.KK;
        const int kh = r / p.K, kw = r % p.K;
        float acc = 0.f;
        for (int b = 0; b < p.B; ++b)
            for (int oh = 0; oh < p.OH; ++oh)
                for (int ow = 0; ow < p.OW; ++ow) {
                    const size_t gi = size_t(b) * p.OCP + size_t(oc) * p.P + oh * p.OW + ow;
                    float g = Elem<T>::ldg(dy + gi);
                    if (RELU && !(Elem<T>::ldg(y + gi) > 0.f)) g = 0.f;
                    acc = fmaf(g, Elem<T>::ldg(x + size_t(b) * p.IHW + ic * p.HW +
                                               (oh * p.S + kh) * p.W + ow * p.S + kw), acc);
                }
        Elem<T>::st(dw + i, acc);
    }
}

__global__ void l2_flush_kernel(float4* __restrict__ buf, size_t n, float v)
{
    for (size_t i = blockIdx.x * size_t(blockDim.x) + threadIdx.x; i < n; i += size_t(gridDim.x) * blockDim.x)
        buf[i] = make_float4(v, v, v, v);
}

template <typename T> constexpr int dt_of();
template <> constexpr int dt_of<float>() { return DT_F32; }
template <> constexpr int dt_of<__nv_bfloat16>() { return DT_BF16; }

}  // namespace

// ======================================================================================
// Host side: eligibility, plans, launches.
// ======================================================================================
bool ffma_fwd_ok(const ConvParams& p, const DevInfo& d) { return fw_smem(p) <= d.smem_optin; }

bool ffma_dgrad_ok(const ConvParams& p, const DevInfo& d)
{
    if (p.P > DG_NCOL || p.KK > DG_KT) return false;
    return dg_smem(p, dgrad_geom(p)) <= d.smem_optin;
}

bool ffma_wgrad_ok(const ConvParams&, const DevInfo& d) { return wg_smem() <= d.smem_optin; }

Plan plan_fwd_ffma(const ConvParams& p, const DevInfo& d)
{
    Plan pl;
    pl.algo = ALGO_FFMA;
    pl.launches = p.N > 0 ? 1 : 0;
    pl.grid = std::max(1, std::min(d.sms, ceil_div(std::max(p.N, 1), FW_WARPS * 8))) * ceil_div(p.OC, FW_OCT);
    pl.block = FW_THREADS;
    pl.smem = fw_smem(p);
    return pl;
}

Plan plan_dgrad_ffma(const ConvParams& p, const DevInfo& d)
{
    const DgradGeom g = dgrad_geom(p);
    Plan pl;
    pl.algo = ALGO_FFMA;
    pl.launches = p.B > 0 ? 1 : 0;
    pl.grid = std::max(1, std::min(d.sms, g.units));
    pl.block = DG_THREADS;
    pl.smem = dg_smem(p, g);
    return pl;
}

Plan plan_wgrad_ffma(const ConvParams& p, const DevInfo& d)
{
    Plan pl;
    pl.algo = ALGO_FFMA;
    pl.block = WG_THREADS;
    pl.smem = wg_smem();
    const int tiles = ceil_div(p.OC, WG_TM) * ceil_div(p.Kred, WG_TN);
    pl.grid = tiles;
    if (p.N == 0) {
        pl.splits = 0;
        pl.launches = 1;  // the reduction alone writes zeros
        pl.workspace = 0;
        return pl;
    }
    // Enough split-K ranges to fill two CTAs per SM, each range at least 128 columns.
    int splits = std::max(1, (2 * d.sms) / tiles);
    splits = std::min(splits, std::max(1, ceil_div(p.N, 128)));
    pl.splits = splits;
    pl.grid = tiles * splits;
    pl.launches = 2;
    pl.workspace = size_t(splits) * p.OC * round_up(p.Kred, 4) * sizeof(float);
    return pl;
}

Plan plan_fwd_direct(const ConvParams& p, const DevInfo& d)
{
    Plan pl;
    pl.algo = ALGO_DIRECT;
    pl.launches = p.B > 0 ? 1 : 0;
    pl.block = 256;
    pl.grid = std::max(1, std::min(d.sms * 8, ceil_div(std::max(1, p.B * p.OCP), 256)));
    return pl;
}
Plan plan_dgrad_direct(const ConvParams& p, const DevInfo& d)
{
    Plan pl;
    pl.algo = ALGO_DIRECT;
    pl.launches = p.B > 0 ? 1 : 0;
    pl.block = 256;
    pl.grid = std::max(1, std::min(d.sms * 8, ceil_div(std::max(1, p.B * p.IHW), 256)));
    return pl;
}
Plan plan_wgrad_direct(const ConvParams& p, const DevInfo& d)
{
    Plan pl;
    pl.algo = ALGO_DIRECT;
    pl.launches = 1;
    pl.block = 256;
    pl.grid = std::max(1, std::min(d.sms * 8, ceil_div(p.OC * p.Kred, 256)));
    return pl;
}

#define IG_DISPATCH_RELU(relu, ...)            \
    do {                                       \
        if (relu) {                            \
            constexpr bool R = true;           \
            __VA_ARGS__;                       \
        } else {                               \
            constexpr bool R = false;          \
            __VA_ARGS__;                       \
        }                                      \
    } while (0)

template <typename T>
static cudaError_t fwd_ffma_t(const Plan& pl, const ConvParams& p, const void* x, const void* w,
                              const void* bias, void* y, cudaStream_t s)
{
    const int oct = ceil_div(p.OC, FW_OCT);
    dim3 grid(pl.grid / oct, oct);
    cudaError_t e = cudaSuccess;
    IG_DISPATCH_RELU(p.relu, {
        e = ensure_smem<fwd_ffma_kernel<T, R>>(pl.smem);
        if (e == cudaSuccess)
            fwd_ffma_kernel<T, R><<<grid, pl.block, pl.smem, s>>>(p, (const T*)x, (const T*)w, (const T*)bias,
                                                                  (T*)y);
    });
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t run_fwd_ffma(const Plan& pl, const ConvParams& p, int dt, const void* x, const void* w,
                         const void* bias, void* y, cudaStream_t s)
{
    if (pl.launches == 0) return cudaSuccess;
    return dt == DT_F32 ? fwd_ffma_t<float>(pl, p, x, w, bias, y, s)
                        : fwd_ffma_t<__nv_bfloat16>(pl, p, x, w, bias, y, s);
}

template <typename T>
static cudaError_t dgrad_ffma_t(const Plan& pl, const ConvParams& p, const void* dy, const void* w,
                                const void* y, void* dx, cudaStream_t s)
{
    const DgradGeom g = dgrad_geom(p);
    cudaError_t e = cudaSuccess;
    IG_DISPATCH_RELU(p.relu, {
        e = ensure_smem<dgrad_ffma_kernel<T, R>>(pl.smem);
        if (e == cudaSuccess)
            dgrad_ffma_kernel<T, R><<<pl.grid, pl.block, pl.smem, s>>>(p, (const T*)dy, (const T*)w, (const T*)y, (T*)dx, g);
    });
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t run_dgrad_ffma(const Plan& pl, const ConvParams& p, int dt, const void* dy,
                           const void* w, const void* y, void* dx, cudaStream_t s)
{
    if (pl.launches == 0) return cudaSuccess;
    return dt == DT_F32 ? dgrad_ffma_t<float>(pl, p, dy, w, y, dx, s)
                        : dgrad_ffma_t<__nv_bfloat16>(pl, p, dy, w, y, dx, s);
}

template <typename T>
static cudaError_t wgrad_ffma_t(const Plan& pl, const ConvParams& p, const void* x, const void* dy,
                                const void* y, void* dw, void* ws, cudaStream_t s)
{
    const int kpad = round_up(p.Kred, 4);
    cudaError_t e = cudaSuccess;
    if (pl.splits > 0) {
        const int tiles_k = ceil_div(p.Kred, WG_TN);
        const int tiles = ceil_div(p.OC, WG_TM) * tiles_k;
        IG_DISPATCH_RELU(p.relu, {
            e = ensure_smem<wgrad_ffma_kernel<T, R>>(pl.smem);
            if (e == cudaSuccess)
                wgrad_ffma_kernel<T, R><<<dim3(tiles, pl.splits), pl.block, pl.smem, s>>>(
                    p, (const T*)x, (const T*)dy, (const T*)y, (float*)ws, pl.splits, kpad, tiles_k);
        });
        if (e == cudaSuccess) e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return run_wgrad_reduce(p, dt_of<T>(), (const float*)ws, pl.splits, kpad, dw, s);
}

cudaError_t run_wgrad_ffma(const Plan& pl, const ConvParams& p, int dt, const void* x,
                           const void* dy, const void* y, void* dw, void* ws, cudaStream_t s)
{
    return dt == DT_F32 ? wgrad_ffma_t<float>(pl, p, x, dy, y, dw, ws, s)
                        : wgrad_ffma_t<__nv_bfloat16>(pl, p, x, dy, y, dw, ws, s);
}

cudaError_t run_wgrad_reduce(const ConvParams& p, int dt, const float* ws, int splits, int kpad,
                             void* dw, cudaStream_t s, bool overlapped, const float* bpart, int nbp, void* db)
{
    const int total = p.OC * p.Kred;
    const int grid = std::max(1, std::min(4096, ceil_div(total, 256)));
    const FastDivmod dm(uint32_t(p.Kred));
    if (dt == DT_F32)
        return launch_ex(wgrad_reduce_kernel<float>, dim3(grid), dim3(256), 0, s, 1, overlapped, ws, splits, kpad,
                         p.OC, p.Kred, dm, (float*)dw, bpart, nbp, (float*)db);
    return launch_ex(wgrad_reduce_kernel<__nv_bfloat16>, dim3(grid), dim3(256), 0, s, 1, overlapped, ws, splits,
                     kpad, p.OC, p.Kred, dm, (__nv_bfloat16*)dw, bpart, nbp, (__nv_bfloat16*)db);
}

template <typename T>
static cudaError_t direct_t(int op, const Plan& pl, const ConvParams& p, const void* a,
                            const void* b, const void* c, void* out, cudaStream_t s)
{
    IG_DISPATCH_RELU(p.relu, {
        if (op == 0)  // c: the bias or nullptr
            fwd_direct_kernel<T, R><<<pl.grid, pl.block, 0, s>>>(p, (const T*)a, (const T*)b, (const T*)c,
                                                                 (T*)out);
        else if (op == 1)
            dgrad_direct_kernel<T, R><<<pl.grid, pl.block, 0, s>>>(p, (const T*)a, (const T*)b,
                                                                   (const T*)c, (T*)out);
        else
            wgrad_direct_kernel<T, R><<<pl.grid, pl.block, 0, s>>>(p, (const T*)a, (const T*)b,
                                                                   (const T*)c, (T*)out);
    });
    return cudaGetLastError();
}

cudaError_t run_fwd_direct(const Plan& pl, const ConvParams& p, int dt, const void* x,
                           const void* w, const void* bias, void* y, cudaStream_t s)
{
    if (pl.launches == 0) return cudaSuccess;
    return dt == DT_F32 ? direct_t<float>(0, pl, p, x, w, bias, y, s)
                        : direct_t<__nv_bfloat16>(0, pl, p, x, w, bias, y, s);
}
cudaError_t run_dgrad_direct(const Plan& pl, const ConvParams& p, int dt, const void* dy,
                             const void* w, const void* y, void* dx, cudaStream_t s)
{
    if (pl.launches == 0) return cudaSuccess;
    return dt == DT_F32 ? direct_t<float>(1, pl, p, dy, w, y, dx, s)
                        : direct_t<__nv_bfloat16>(1, pl, p, dy, w, y, dx, s);
}
cudaError_t run_wgrad_direct(const Plan& pl, const ConvParams& p, int dt, const void* x,
                             const void* dy, const void* y, void* dw, cudaStream_t s)
{
    return dt == DT_F32 ? direct_t<float>(2, pl, p, x, dy, y, dw, s)
                        : direct_t<__nv_bfloat16>(2, pl, p, x, dy, y, dw, s);
}

cudaError_t run_l2_flush(void* buf, size_t bytes, cudaStream_t s)
{
    const size_t n = bytes / 16;
    if (n == 0) return cudaSuccess;
    const int grid = int(std::min<size_t>(4096, (n + 255) / 256));
    l2_flush_kernel<<<grid, 256, 0, s>>>(reinterpret_cast<float4*>(buf), n, 1.0f);
    return cudaGetLastError();
}

}  // namespace igc
