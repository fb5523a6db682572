// kernels_bias.cu -- gradient of the per-output-channel conv bias,
//   db[oc] = sum_{b, oh, ow} g[b, oc, oh, ow],   g = dy * [y > 0] when relu, else dy,
// the reduction the "n3_conv_bias_grad" bench blocks of PufferLib PR #522 ("Speedups to
// gemm_conv_forward and gemm_conv_backward kernels") time for both conv layers.
//
// It is a memory-bound reduction: dy is B rows of OC*P contiguous values (P = OH*OW), read
// once (with y beside it under relu) and reduced to OC numbers.
//
// One kernel, no global scratch.  CTA (w, r) owns a window of ocw whole channels -- the
// window's OCW*P values of a sample are contiguous in dy -- and the r-th of R contiguous
// sample ranges; the R CTAs of a window form one thread-block cluster.  Threads read the
// window's rows with coalesced 16-byte loads (8 rows in flight, 4 with the mask), each
// summing its own columns (oc, oh, ow) down its rows in ascending b; a narrow window gets
// several row lanes, thread lane q taking rows q, q + Q, ...  Then each channel's P columns
// are added in ascending (oh, ow), each over the row lanes in ascending order, into one fp32
// sum per channel in shared memory; after a cluster barrier the rank-0 CTA adds the R
// ranges' sums in ascending rank order through distributed shared memory and rounds once.
// No atomics: the result depends only on the plan (shape and SM count).
#include <algorithm>

#include "internal.h"
#include "tc_ptx.cuh"

namespace igc {

namespace {

constexpr int BG_THREADS = 1024;    // threads of a CTA (at most)
constexpr int BG_MIN_THREADS = 256; // threads of a CTA (at least, when the window allows)
constexpr int BG_ROWS_PER_LANE = 8; // rows each row lane gets, about (enough for 8 loads in flight)
constexpr int BG_WIN = 12288;       // fp32 column sums in a CTA's shared-memory window (48 KB)
constexpr int BG_MINROWS = 16;      // rows per sample range, at least (when B allows)
constexpr int BG_MINBYTES = 64;     // bytes of a window's row, at least (when OC allows)

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

// CTA blockIdx.x = window * R + range (cluster of R along x).  Thread (q, c) = (threadIdx.x /
// lanes_c, threadIdx.x % lanes_c): column groups c, c + lanes_c, ... of the window, rows
// b_lo + q, b_lo + q + Q, ... of the range (Q = blockDim.x / lanes_c row lanes).
template <typename T, bool RELU, int V>
__global__ void __launch_bounds__(BG_THREADS)
bias_grad_kernel(const ConvParams p, const T* __restrict__ dy, const T* __restrict__ y, T* __restrict__ db,
                 int ocw, int R, int lanes_c)
{
    extern __shared__ float sm[];  // [Q][ocw * P] column sums, then [ocw] channel sums
    const int Q = blockDim.x / lanes_c, q = threadIdx.x / lanes_c, c = threadIdx.x % lanes_c;
    const int wcols = ocw * p.P;
    float* colsum = sm;
    float* csum = sm + Q * wcols;
    const int win = blockIdx.x / R;
    const int rank = R > 1 ? int(tc::cluster_rank()) : 0;
    const int oc0 = win * ocw;
    const int noc = min(ocw, p.OC - oc0);
    const int ncg = noc * p.P / V;
    const int b_lo = int(int64_t(p.B) * rank / R), b_hi = int(int64_t(p.B) * (rank + 1) / R);
    const size_t rstep = size_t(Q) * p.OCP;
    tc::grid_dep_wait();  // the previous kernel on the stream may still be writing dy / y
#pragma unroll 1
    for (int cg = c; cg < ncg; cg += lanes_c) {
        float acc[V];
#pragma unroll
        for (int e = 0; e < V; ++e) acc[e] = 0.f;
        const size_t col = size_t(oc0) * p.P + size_t(cg) * V;
        int b = b_lo + q;
        // U rows' loads in flight, added in ascending b.
        constexpr int U = RELU ? 4 : 8;
#pragma unroll 1
        for (; b + (U - 1) * Q < b_hi; b += U * Q) {
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
        for (; b < b_hi; b += Q) {
            float v[V], m[V];
            const size_t off = size_t(b) * p.OCP + col;
            VecLd<T, V>::ld(dy + off, v);
            if (RELU) VecLd<T, V>::ld(y + off, m);
#pragma unroll
            for (int e = 0; e < V; ++e) acc[e] += (!RELU || m[e] > 0.f) ? v[e] : 0.f;
        }
#pragma unroll
        for (int e = 0; e < V; ++e) colsum[q * wcols + cg * V + e] = acc[e];
    }
    __syncthreads();
    // Channel j of the window: its P columns in ascending (oh, ow), each over the row lanes
    // in ascending q.
    for (int j = threadIdx.x; j < noc; j += blockDim.x) {
        float t = 0.f;
        for (int pq = 0; pq < p.P; ++pq)
            for (int qq = 0; qq < Q; ++qq) t += colsum[qq * wcols + j * p.P + pq];
        csum[j] = t;
    }
    tc::grid_dep_launch();
    if (R == 1) {
        for (int j = threadIdx.x; j < noc; j += blockDim.x) Elem<T>::st(db + oc0 + j, csum[j]);
        return;
    }
    tc::cluster_sync();  // every range's channel sums are in its CTA's shared memory
    if (rank == 0) {
        const uint32_t cs = tc::smem_u32(csum);
        for (int j = threadIdx.x; j < noc; j += blockDim.x) {
            // All R loads in flight first (R <= kMaxCluster), then the sum in ascending rank order.
            float v[kMaxCluster];
#pragma unroll
            for (int r = 0; r < kMaxCluster; ++r)
                if (r < R) v[r] = tc::ld_dsmem_f32(tc::dsmem_addr(cs + uint32_t(4 * j), uint32_t(r)));
            float t = 0.f;
#pragma unroll
            for (int r = 0; r < kMaxCluster; ++r)
                if (r < R) t += v[r];
            Elem<T>::st(db + oc0 + j, t);
        }
    }
    tc::cluster_sync();  // no CTA leaves while rank 0 still reads its shared memory
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

}  // namespace

// Plan fields: grid = CTAs (windows x ranges), block = threads (column lanes x row lanes),
// smem = column and channel sums, splits = sample ranges R (the cluster size), variant =
// (channels per window * 1024 + column lanes) * 16 + V.
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
    pl.launches = 1;
    const int es = dt == DT_F32 ? 4 : 2;
    const int vw = 16 / es;
    // Sample ranges: the largest power of two up to the cluster limit that leaves every range
    // BG_MINROWS rows.
    int R = 1;
    while (R < kMaxCluster && p.B / (2 * R) >= BG_MINROWS) R *= 2;
    // Channels per window: enough windows for about two CTAs per SM, a row of at least
    // BG_MINBYTES, then rounded up so that windows start on 16-byte boundaries (vector loads).
    const int nwin_target = std::max(1, ceil_div(2 * d.sms, R));
    int ocw = std::max(1, ceil_div(p.OC, nwin_target));
    while (ocw < p.OC && ocw * p.P * es < BG_MINBYTES) ++ocw;
    int v = 1;
    if (p.OCP % vw == 0) {
        int o = ocw;
        while (o <= p.OC && (o * p.P) % vw != 0) ++o;
        if (o <= p.OC && o * p.P <= BG_WIN) {
            ocw = o;
            v = vw;
        }
    }
    ocw = std::min(ocw, std::max(1, BG_WIN / p.P));
    // Column lanes: the window's column groups, rounded up to a power of two below a warp and
    // to whole warps above (the surplus lanes idle), so that blocks are whole warps.
    const int ncg = ocw * p.P / v;
    int lanes_c = 1;
    while (lanes_c < ncg && lanes_c < 32) lanes_c *= 2;
    if (ncg > 32) lanes_c = std::min(BG_THREADS, round_up(ncg, 32));
    // Row lanes: at least 256 threads, more (up to 1024) while every row lane keeps about
    // BG_ROWS_PER_LANE rows, so that a long range has more loads in flight.  Measured on a GB300
    // with 256, 512 and 1024 threads: at B = 32768 1024 threads run 1.8-2.1x faster than 256; at
    // B = 1024 256 threads are fastest.
    const int rows = std::max(1, p.B / R);
    int lanes_r = std::max(1, std::min({BG_THREADS / lanes_c, BG_WIN / (ocw * p.P),
                                        std::max(BG_MIN_THREADS / lanes_c, rows / BG_ROWS_PER_LANE)}));
    while (lanes_r > 1 && (lanes_c * lanes_r) % 32 != 0) --lanes_r;
    pl.block = lanes_c * lanes_r;
    pl.smem = (lanes_r * ocw * p.P + ocw) * 4;
    pl.splits = R;
    pl.grid = ceil_div(p.OC, ocw) * R;
    pl.variant = (ocw * 1024 + lanes_c) * 16 + v;
    return pl;
}

namespace {

template <typename T>
cudaError_t bgrad_t(const Plan& pl, const ConvParams& p, const void* dy, const void* y, void* db,
                    cudaStream_t s)
{
    if (pl.algo == ALGO_DIRECT) {
        if (p.relu)
            bias_direct_kernel<T, true><<<pl.grid, pl.block, 0, s>>>(p, (const T*)dy, (const T*)y, (T*)db);
        else
            bias_direct_kernel<T, false><<<pl.grid, pl.block, 0, s>>>(p, (const T*)dy, (const T*)y, (T*)db);
        return cudaGetLastError();
    }
    const int ocw = pl.variant / 16 / 1024, lanes_c = pl.variant / 16 % 1024, v = pl.variant % 16;
    cudaError_t e = cudaSuccess;
#define IG_BG_LAUNCH(RL, V)                                                                                 \
    do {                                                                                                    \
        e = ensure_smem<bias_grad_kernel<T, RL, V>>(pl.smem);                                               \
        if (e == cudaSuccess)                                                                               \
            e = launch_ex(bias_grad_kernel<T, RL, V>, dim3(pl.grid), dim3(pl.block), pl.smem, s, pl.splits, \
                          true, p, (const T*)dy, (const T*)y, (T*)db, ocw, pl.splits, lanes_c);             \
    } while (0)
    constexpr int VW = sizeof(T) == 4 ? 4 : 8;
    if (p.relu) {
        if (v == VW) IG_BG_LAUNCH(true, VW);
        else IG_BG_LAUNCH(true, 1);
    } else {
        if (v == VW) IG_BG_LAUNCH(false, VW);
        else IG_BG_LAUNCH(false, 1);
    }
#undef IG_BG_LAUNCH
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

cudaError_t run_bgrad(const Plan& pl, const ConvParams& p, int dt, const void* dy, const void* y, void* db,
                      cudaStream_t s)
{
    return dt == DT_F32 ? bgrad_t<float>(pl, p, dy, y, db, s) : bgrad_t<__nv_bfloat16>(pl, p, dy, y, db, s);
}

}  // namespace igc
