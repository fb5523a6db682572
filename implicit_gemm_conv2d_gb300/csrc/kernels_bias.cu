// kernels_bias.cu -- gradient of the per-output-channel conv bias,
//   db[oc] = sum_{b, oh, ow} g[b, oc, oh, ow],   g = dy * [y > 0] when relu, else dy,
// the reduction the "n3_conv_bias_grad" bench blocks of PufferLib PR #522 ("Speedups to
// gemm_conv_forward and gemm_conv_backward kernels") time for both conv layers.
//
// It is a memory-bound reduction: dy is B rows of OC*P contiguous values (P = OH*OW), read
// once (with y beside it under relu) and reduced to OC numbers.
//
// Column-sum kernel: each CTA owns a window of whole channels (all OC unless a row is longer
// than the shared-memory window) and a contiguous range of samples.  Its threads read the
// rows with coalesced 16-byte loads, each thread summing its own columns (oc, oh, ow) down
// its rows in ascending b; a narrow window (few columns) gets several row lanes, thread lane r
// taking rows r, r + R, ...  Then each channel's P columns are added in ascending (oh, ow),
// each over the row lanes in ascending order, into one fp32 partial per (range, channel),
// kept in the per-stream scratch buffer.
// Reduce kernel: 32 warps per 32 channels; warp w adds ranges w, w + 32, ... in ascending
// order, then one warp adds the 32 warp sums in ascending order and rounds once.
// No atomics: the result depends only on the plan (shape and SM count).
#include <algorithm>

#include "internal.h"

namespace igc {

namespace {

constexpr int BG_MAXT = 512;        // threads of a column-sum CTA
constexpr int BG_WIN = 12288;       // fp32 column sums in a CTA's shared-memory window (48 KB)
constexpr int BG_REGS = 64;         // registers per thread the column-sum kernel is built for
constexpr int BG_MINROWS = 4;       // rows per thread of a sample range, at least (when B allows)
constexpr int BG_MAXSPLIT = 1024;   // sample ranges, at most (the reduce adds 32 per warp lane)
constexpr int BG_RED_WARPS = 32;    // warps of a reduce CTA (one CTA per 32 channels)

__device__ __forceinline__ void dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// V consecutive elements widened to fp32: one 16-byte load for V * sizeof(T) == 16.
template <typename T, int V> struct VecLd;
template <typename T> struct VecLd<T, 1> {
    static __device__ __forceinline__ void ld(const T* p, float (&v)[1]) { v[0] = Elem<T>::ldg(p); }
};
template <> struct VecLd<float, 4> {
    static __device__ __forceinline__ void ld(const float* p, float (&v)[4])
    {
        const float4 f = __ldg(reinterpret_cast<const float4*>(p));
        v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
    }
};
template <> struct VecLd<__nv_bfloat16, 8> {
    static __device__ __forceinline__ void ld(const __nv_bfloat16* p, float (&v)[8])
    {
        const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {  // element 2i in the low half of word i
            v[2 * i] = __uint_as_float(w[i] << 16);
            v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    }
};

template <typename T, bool RELU, int V>
__global__ void __launch_bounds__(BG_MAXT, 65536 / (BG_MAXT * BG_REGS))
bias_colsum_kernel(const ConvParams p, const T* __restrict__ dy, const T* __restrict__ y,
                   float* __restrict__ part, int nsplit, int ocw, int lanes_c)
{
    // Thread (r, c) = (threadIdx.x / lanes_c, threadIdx.x % lanes_c): column groups c, c + lanes_c, ...
    // of the window, rows b_lo + r, b_lo + r + R, ... of the range (R = blockDim.x / lanes_c).
    extern __shared__ float colsum[];  // [R][ocw * P] column sums
    const int R = blockDim.x / lanes_c, r = threadIdx.x / lanes_c, c = threadIdx.x % lanes_c;
    const int oc0 = blockIdx.x * ocw;
    const int noc = min(ocw, p.OC - oc0);
    const int wcols = ocw * p.P;
    const int c0 = oc0 * p.P, ncg = noc * p.P / V;  // window columns [c0, c0 + noc*P), V per group
    const int s = blockIdx.y;
    const int b_lo = int(int64_t(p.B) * s / nsplit), b_hi = int(int64_t(p.B) * (s + 1) / nsplit);
    const size_t rstep = size_t(R) * p.OCP;
#pragma unroll 1
    for (int cg = c; cg < ncg; cg += lanes_c) {
        float acc[V];
#pragma unroll
        for (int e = 0; e < V; ++e) acc[e] = 0.f;
        const size_t col = size_t(c0) + size_t(cg) * V;
        int b = b_lo + r;
        // U rows' loads in flight (eight 16-byte loads), added in ascending b.
        constexpr int U = RELU ? 4 : 8;
#pragma unroll 1
        for (; b + (U - 1) * R < b_hi; b += U * R) {
            float v[U][V], m[U][V];
            const size_t off0 = size_t(b) * p.OCP + col;
#pragma unroll
            for (int u = 0; u < U; ++u) {
                VecLd<T, V>::ld(dy + off0 + u * rstep, v[u]);
                if (RELU) VecLd<T, V>::ld(y + off0 + u * rstep, m[u]);
            }
#pragma unroll
            for (int u = 0; u < U; ++u)
#pragma unroll
                for (int e = 0; e < V; ++e) acc[e] += (!RELU || m[u][e] > 0.f) ? v[u][e] : 0.f;
        }
        for (; b < b_hi; b += R) {
            float v[V], m[V];
            const size_t off = size_t(b) * p.OCP + col;
            VecLd<T, V>::ld(dy + off, v);
            if (RELU) VecLd<T, V>::ld(y + off, m);
#pragma unroll
            for (int e = 0; e < V; ++e) acc[e] += (!RELU || m[e] > 0.f) ? v[e] : 0.f;
        }
#pragma unroll
        for (int e = 0; e < V; ++e) colsum[r * wcols + cg * V + e] = acc[e];
    }
    __syncthreads();
    // Channel j of the window: its P columns in ascending (oh, ow), each over the row lanes
    // in ascending r.
    for (int j = threadIdx.x; j < noc; j += blockDim.x) {
        float t = 0.f;
        for (int q = 0; q < p.P; ++q)
            for (int rr = 0; rr < R; ++rr) t += colsum[rr * wcols + j * p.P + q];
        part[size_t(s) * p.OC + oc0 + j] = t;
    }
    dep_launch();
}

// db[oc] = sum of the nsplit partials part[s][oc]; nsplit == 0 writes zeros.
template <typename T>
__global__ void __launch_bounds__(BG_RED_WARPS * 32)
bias_reduce_kernel(const float* __restrict__ part, int nsplit, int OC, T* __restrict__ db)
{
    __shared__ float red[BG_RED_WARPS][33];
    dep_wait();  // the partials come from the kernel launched just before
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int oc = blockIdx.x * 32 + lane;
    float s = 0.f;
    if (oc < OC) {
        // Loads in groups of eight issued together, added in ascending range order.
        int i = warp;
        for (; i + 7 * BG_RED_WARPS < nsplit; i += 8 * BG_RED_WARPS) {
            float v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) v[u] = __ldcg(part + size_t(i + u * BG_RED_WARPS) * OC + oc);
#pragma unroll
            for (int u = 0; u < 8; ++u) s += v[u];
        }
        for (; i < nsplit; i += BG_RED_WARPS) s += __ldcg(part + size_t(i) * OC + oc);
    }
    red[warp][lane] = s;
    __syncthreads();
    if (warp == 0 && oc < OC) {
        float t = 0.f;
#pragma unroll
        for (int w = 0; w < BG_RED_WARPS; ++w) t += red[w][lane];
        Elem<T>::st(db + oc, t);
    }
}

// Any shape: one warp per channel; lane l adds the elements l, l + 32, ... of the channel's
// B*P values (b-major) in ascending order, then a fixed butterfly adds the lanes.
template <typename T, bool RELU>
__global__ void bias_direct_kernel(const ConvParams p, const T* __restrict__ dy, const T* __restrict__ y,
                                   T* __restrict__ db)
{
    const int lane = threadIdx.x & 31;
    const int nwarps = int((size_t(gridDim.x) * blockDim.x) >> 5);
    const int n = p.B * p.P;
    for (int oc = int((size_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5); oc < p.OC; oc += nwarps) {
        float s = 0.f;
        for (int i = lane; i < n; i += 32) {
            uint32_t b, q;
            p.dm_P.divmod(uint32_t(i), b, q);
            const size_t off = size_t(b) * p.OCP + size_t(oc) * p.P + q;
            const float v = Elem<T>::ldg(dy + off);
            if (!RELU || Elem<T>::ldg(y + off) > 0.f) s += v;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
        if (lane == 0) Elem<T>::st(db + oc, s);
    }
}

// Plan fields: grid = column-sum CTAs (windows x ranges), block = its threads (column lanes x row
// lanes), smem = its column sums, splits = sample ranges, variant = (channels per window * 1024 +
// column lanes) * 16 + V.
int vec_width(const ConvParams& p, int dt)
{
    const int v = dt == DT_F32 ? 4 : 8;  // 16 bytes
    // One window holding every channel, rows 16-byte aligned (OC*P a multiple of V).
    return (p.OCP <= BG_WIN && p.OCP % v == 0) ? v : 1;
}

}  // namespace

Plan plan_bgrad(const ConvParams& p, int dt, const DevInfo& d, bool direct)
{
    Plan pl;
    if (direct || p.P > BG_WIN) {
        pl.algo = ALGO_DIRECT;
        pl.launches = 1;
        pl.block = 256;
        pl.grid = std::max(1, std::min(d.sms * 8, ceil_div(p.OC, 8)));
        return pl;
    }
    pl.algo = ALGO_FFMA;
    const int v = vec_width(p, dt);
    const int ocw = v > 1 ? p.OC : std::min(p.OC, BG_WIN / p.P);
    const int wcols = ocw * p.P;
    const int nwin = ceil_div(p.OC, ocw);
    const int lanes_c = std::min(BG_MAXT, round_up(wcols / v, 32));
    // Row lanes: enough for 256 threads when the window is narrow, within the thread and
    // shared-memory limits.
    const int lanes_r = std::max(1, std::min({256 / lanes_c, BG_MAXT / lanes_c, BG_WIN / wcols}));
    pl.block = lanes_c * lanes_r;
    pl.smem = lanes_r * wcols * 4;
    if (p.B == 0) {
        pl.launches = 1;  // the reduce writes zeros
        pl.splits = 0;
        pl.grid = 0;
    } else {
        // One wave of resident CTAs (threads, registers and shared memory per SM).
        const int per_sm = std::max(1, std::min({2048 / pl.block, 65536 / (BG_REGS * pl.block),
                                                 (200 * 1024) / (pl.smem + 1024), 32}));
        int nsplit = std::max(1, d.sms * per_sm / nwin);
        nsplit = std::min(nsplit, std::max(1, p.B / (BG_MINROWS * lanes_r)));
        nsplit = std::min({nsplit, BG_MAXSPLIT, int(kScratchBytes / (sizeof(float) * size_t(p.OC)))});
        pl.splits = std::max(1, nsplit);
        pl.grid = nwin * pl.splits;
        pl.launches = 2;
    }
    pl.variant = (ocw * 1024 + lanes_c) * 16 + v;
    return pl;
}

namespace {

template <typename T>
cudaError_t bgrad_t(const Plan& pl, const ConvParams& p, const void* dy, const void* y, void* db,
                    cudaStream_t s)
{
    cudaError_t e = cudaSuccess;
    if (pl.algo == ALGO_DIRECT) {
        if (p.relu)
            bias_direct_kernel<T, true><<<pl.grid, pl.block, 0, s>>>(p, (const T*)dy, (const T*)y, (T*)db);
        else
            bias_direct_kernel<T, false><<<pl.grid, pl.block, 0, s>>>(p, (const T*)dy, (const T*)y, (T*)db);
        return cudaGetLastError();
    }
    const int ocw = pl.variant / 16 / 1024, lanes_c = pl.variant / 16 % 1024, v = pl.variant % 16;
    if (pl.splits > 0) {
        int dev = 0;
        if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
        float* part = static_cast<float*>(stream_scratch(dev, s));
        if (!part) return cudaErrorMemoryAllocation;
        const dim3 grid(ceil_div(p.OC, ocw), pl.splits);
#define IG_BG_LAUNCH(R, V)                                                                              \
    bias_colsum_kernel<T, R, V><<<grid, pl.block, pl.smem, s>>>(p, (const T*)dy, (const T*)y, part, pl.splits, ocw, \
                                                                 lanes_c)
        constexpr int VW = sizeof(T) == 4 ? 4 : 8;
        if (p.relu) {
            if (v == VW) IG_BG_LAUNCH(true, VW);
            else IG_BG_LAUNCH(true, 1);
        } else {
            if (v == VW) IG_BG_LAUNCH(false, VW);
            else IG_BG_LAUNCH(false, 1);
        }
#undef IG_BG_LAUNCH
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        return launch_overlapped(bias_reduce_kernel<T>, dim3(ceil_div(p.OC, 32)), dim3(BG_RED_WARPS * 32), 0, s,
                                 (const float*)part, pl.splits, p.OC, (T*)db);
    }
    bias_reduce_kernel<T><<<ceil_div(p.OC, 32), BG_RED_WARPS * 32, 0, s>>>(nullptr, 0, p.OC, (T*)db);  // B = 0
    return cudaGetLastError();
}

}  // namespace

cudaError_t run_bgrad(const Plan& pl, const ConvParams& p, int dt, const void* dy, const void* y, void* db,
                      cudaStream_t s)
{
    return dt == DT_F32 ? bgrad_t<float>(pl, p, dy, y, db, s) : bgrad_t<__nv_bfloat16>(pl, p, dy, y, db, s);
}

}  // namespace igc
