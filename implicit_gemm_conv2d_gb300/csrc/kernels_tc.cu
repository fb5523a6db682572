// kernels_tc.cu -- tcgen05 tensor-core implicit-GEMM kernels (5th-generation
// tensor cores, accumulator in tensor memory).
//
// Forward, per CTA tile:  D[oc, n] = sum_k W[oc, k] * X[n, k]   (M = 128 output
// channels, N = NT columns n = (b, oh, ow), K = IC*K*K padded to the chunk size),
// X[n, k] = x[col_base(n) + k_offset(k)] gathered on the fly (implicit im2col).
//   bf16: tcgen05.mma kind::f16, bf16 operands, fp32 accumulation.
//   fp32: three tcgen05.mma kind::tf32 per step (hi*hi + hi*lo + lo*hi with
//         v = hi + lo, hi = tf32(v), lo = tf32(v - hi)), which keeps about 21
//         significant bits per product: fp32-level accuracy on the tensor pipe.
// All 256 threads gather the next K-chunk of both operands into shared memory
// (K-major, 128-byte swizzled core-matrix layout) while one thread issues the
// MMAs of the current chunk; two stages, one mbarrier per stage signalled by
// tcgen05.commit.  The epilogue reads the accumulator with tcgen05.ld, applies
// the ReLU and writes y.  Tiles are scheduled persistently over the grid.
//
// Every mbarrier wait is bounded; a wait that runs out sets a bit in
// g_tc_status, all threads leave their loops together and the CTA frees its
// tensor memory before returning.
#include <algorithm>
#include <cstdlib>

#include "internal.h"
#include "tc_ptx.cuh"

namespace igc {

__device__ unsigned int g_tc_status = 0;

namespace {

using namespace tc;

constexpr int TC_THREADS = 256;
constexpr int TC_STAGES = 2;
constexpr int TC_M = 128;
constexpr int ROWB = 128;  // bytes of one operand row per K-chunk

template <typename T> struct TcTraits;
template <> struct TcTraits<__nv_bfloat16> {
    static constexpr int E = 8;        // elements per 16-byte unit
    static constexpr int KC = 64;      // elements per chunk (one 128-byte row)
    static constexpr bool split = false;
    static constexpr uint32_t fmt = 1; // bf16
};
template <> struct TcTraits<float> {
    static constexpr int E = 4;
    static constexpr int KC = 32;
    static constexpr bool split = true;
    static constexpr uint32_t fmt = 2; // tf32
};

// Byte offset of 16-byte unit (row r, unit column c) of a K-major operand tile
// whose rows are 128 bytes: 8-row groups of 1024 bytes; within a group, with
// the 128-byte swizzle the unit column is XORed with the row index.
template <int SWZ>
__device__ __forceinline__ uint32_t unit_off(int r, int c)
{
    if (SWZ) return uint32_t((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
    return uint32_t((r >> 3) * 1024 + c * 128 + (r & 7) * 16);
}

template <int SWZ>
__device__ __forceinline__ uint64_t op_desc(uint32_t saddr)
{
    if (SWZ) return smem_desc(saddr, 16, 1024) | (uint64_t(2) << 61);  // 128-byte swizzle
    return smem_desc(saddr, 128, 1024);
}
template <int SWZ>
__device__ __forceinline__ uint32_t kstep_off(int j)
{
    return SWZ ? uint32_t(j * 32) : uint32_t(j * 256);  // 32 bytes of K per MMA step
}

__device__ __forceinline__ void st_unit(unsigned char* base, uint32_t off, uint32_t a, uint32_t b, uint32_t c,
                                        uint32_t d)
{
    *reinterpret_cast<uint4*>(base + off) = make_uint4(a, b, c, d);
}

__device__ __forceinline__ void report(int* abort_flag, unsigned code)
{
    *abort_flag = 1;
    atomicOr(&g_tc_status, code);
}

// Write one unit of 4 fp32 values as tf32 hi and lo parts, or of 8 bf16 values.
template <typename T, int SWZ>
__device__ __forceinline__ void put_unit(unsigned char* hi, unsigned char* lo, int r, int c, const float (&v)[8])
{
    const uint32_t off = unit_off<SWZ>(r, c);
    if constexpr (TcTraits<T>::split) {
        float h[4], l[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            h[i] = to_tf32(v[i]);
            l[i] = to_tf32(v[i] - h[i]);
        }
        st_unit(hi, off, __float_as_uint(h[0]), __float_as_uint(h[1]), __float_as_uint(h[2]), __float_as_uint(h[3]));
        st_unit(lo, off, __float_as_uint(l[0]), __float_as_uint(l[1]), __float_as_uint(l[2]), __float_as_uint(l[3]));
    } else {
        uint32_t q[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t a = __bfloat16_as_ushort(__float2bfloat16_rn(v[2 * i]));
            const uint32_t b = __bfloat16_as_ushort(__float2bfloat16_rn(v[2 * i + 1]));
            q[i] = a | (b << 16);
        }
        st_unit(hi, off, q[0], q[1], q[2], q[3]);
    }
}

// Issue the MMAs of one K-chunk (4 steps of 32 bytes of K) from operand tiles at
// the given shared addresses (hi parts; the lo parts of a split fp32 operand
// sit `lo_off` bytes further).
template <typename T, int SWZ>
__device__ __forceinline__ void issue_chunk(uint32_t tmem, uint32_t a_addr, uint32_t b_addr, uint32_t lo_off,
                                            uint32_t idesc, bool first)
{
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint64_t ad = op_desc<SWZ>(a_addr + kstep_off<SWZ>(j));
        const uint64_t bd = op_desc<SWZ>(b_addr + kstep_off<SWZ>(j));
        const uint32_t acc = (first && j == 0) ? 0u : 1u;
        if constexpr (TcTraits<T>::split) {
            const uint64_t al = op_desc<SWZ>(a_addr + lo_off + kstep_off<SWZ>(j));
            const uint64_t bl = op_desc<SWZ>(b_addr + lo_off + kstep_off<SWZ>(j));
            mma_tf32(tmem, ad, bd, idesc, acc);
            mma_tf32(tmem, ad, bl, idesc, 1u);
            mma_tf32(tmem, al, bd, idesc, 1u);
        } else {
            mma_f16(tmem, ad, bd, idesc, acc);
        }
    }
}

// Shared state of one CTA's tensor-core pipeline.  A stage holds the A tile
// (128 rows) then the B tile (NT rows), 128 bytes per row, followed for split
// fp32 operands by the lo parts of both (`half` bytes further).
struct TcPipe {
    unsigned char* smem;   // stage 0 (1024-byte aligned)
    uint32_t smem_base;    // its shared-window address
    uint32_t a_bytes, half, stage_bytes;
    uint64_t* bars;        // one mbarrier per stage, completed by tcgen05.commit
    int* abort_flag;
    uint32_t tmem, idesc;
    uint32_t g;            // K-chunks issued so far; stage = g & 1
};

template <typename T>
__device__ __forceinline__ void pipe_setup(TcPipe& pp, unsigned char* smem, int NT)
{
    using Tr = TcTraits<T>;
    pp.smem = smem;
    pp.smem_base = smem_u32(smem);
    pp.a_bytes = TC_M * ROWB;
    pp.half = pp.a_bytes + NT * ROWB;
    pp.stage_bytes = Tr::split ? 2 * pp.half : pp.half;
    pp.idesc = instr_desc(Tr::fmt, TC_M, NT);
    pp.g = 0;
}

// Tail of the shared-memory carve-up after the stages: barriers, TMEM slot, abort flag.
struct TcTail {
    uint64_t bars[TC_STAGES];
    uint32_t tslot;
    int abort_flag;
};

// Barrier init + TMEM allocation.  Call with all threads; ends with a CTA barrier.
__device__ __forceinline__ void pipe_start(TcPipe& pp, TcTail* tail, int tmem_cols)
{
    const int tid = threadIdx.x;
    if (tid == 0) {
        for (int s = 0; s < TC_STAGES; ++s) mbar_init(smem_u32(&tail->bars[s]), 1);
        fence_mbar_init();
        tail->abort_flag = 0;
    }
    if ((tid >> 5) == 0) tmem_alloc(smem_u32(&tail->tslot), tmem_cols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pp.bars = tail->bars;
    pp.abort_flag = &tail->abort_flag;
    pp.tmem = tail->tslot;
}

__device__ __forceinline__ void pipe_finish(const TcPipe& pp, int tmem_cols)
{
    __syncthreads();
    if ((threadIdx.x >> 5) == 0) {
        tc_fence_after();
        tmem_dealloc(pp.tmem, tmem_cols);
    }
}

// One tile's K loop.  fill(stage_ptr, kc) writes chunk kc of A (at stage_ptr) and B
// (at stage_ptr + a_bytes), plus lo parts at + half, with all threads.  When
// `a_fixed` is nonzero the MMAs read A from that shared address (+ kc * 16 KB
// per chunk) instead of the stage.  Returns false if a wait ran out.
template <typename T, int SWZ, class Fill>
__device__ __forceinline__ bool pipe_tile(TcPipe& pp, int nchunks, Fill&& fill, uint32_t a_fixed = 0,
                                          uint32_t a_fixed_lo_off = 0)
{
    for (int kc = 0; kc < nchunks; ++kc, ++pp.g) {
        const int s = pp.g & 1;
        unsigned char* st = pp.smem + s * pp.stage_bytes;
        if (pp.g >= 2 && !mbar_wait(smem_u32(&pp.bars[s]), ((pp.g >> 1) - 1) & 1)) report(pp.abort_flag, 1u);
        fill(st, kc);
        fence_proxy_async_smem();
        __syncthreads();
        if (*pp.abort_flag) return false;
        if (threadIdx.x == 0) {
            tc_fence_after();
            const uint32_t sa = pp.smem_base + s * pp.stage_bytes;
            if (a_fixed)
                issue_chunk<T, SWZ>(pp.tmem, a_fixed + kc * (TC_M * ROWB), sa + pp.a_bytes, a_fixed_lo_off,
                                    pp.idesc, kc == 0);
            else
                issue_chunk<T, SWZ>(pp.tmem, sa, sa + pp.a_bytes, pp.half, pp.idesc, kc == 0);
            mma_commit(smem_u32(&pp.bars[s]));
        }
    }
    return true;
}

// Wait until the tile's accumulator is complete.  All threads; false if aborted.
__device__ __forceinline__ bool pipe_wait_acc(TcPipe& pp)
{
    const uint32_t last = pp.g - 1;
    if (!mbar_wait(smem_u32(&pp.bars[last & 1]), (last >> 1) & 1)) report(pp.abort_flag, 2u);
    __syncthreads();
    if (*pp.abort_flag) return false;
    tc_fence_after();
    return true;
}

// End of an epilogue that read TMEM: order the reads before the next tile's MMAs.
__device__ __forceinline__ void pipe_release_acc()
{
    tc_fence_before();
    __syncthreads();
}

__device__ __forceinline__ unsigned char* align1024(unsigned char* p)
{
    return reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// ======================================================================================
// Forward: tile = (128 output channels, NT columns); K = IC*K*K in chunks.
// ======================================================================================
struct TcFwdGeom {
    int NT;        // columns per tile (multiple of 16, <= 256)
    int n_tiles;   // ceil(N / NT)
    int oc_tiles;  // ceil(OC / 128)
    int tmem_cols; // power of two >= max(32, NT)
};

template <typename T>
inline int tc_stage_bytes(int NT)
{
    const int half = TC_M * ROWB + NT * ROWB;
    return TcTraits<T>::split ? 2 * half : half;
}

template <typename T>
inline int tc_fwd_smem(const ConvParams& p, int NT)
{
    const int kred_pad = round_up(p.Kred, TcTraits<T>::KC);
    return 1024 + TC_STAGES * tc_stage_bytes<T>(NT) + kred_pad * 4 + NT * 4 + int(sizeof(TcTail));
}

template <typename T, bool RELU, int SWZ>
__global__ void __launch_bounds__(TC_THREADS, 1)
fwd_tc_kernel(const ConvParams p, const T* __restrict__ x, const T* __restrict__ w, T* __restrict__ y,
              const TcFwdGeom geo)
{
    using Tr = TcTraits<T>;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = align1024(smem_raw);
    const int NT = geo.NT;
    const int kred_pad = round_up(p.Kred, Tr::KC);
    const int nchunks = kred_pad / Tr::KC;
    TcPipe pp;
    pipe_setup<T>(pp, smem, NT);
    int* offk = reinterpret_cast<int*>(smem + TC_STAGES * pp.stage_bytes);
    int* colb = offk + kred_pad;
    TcTail* tail = reinterpret_cast<TcTail*>(colb + NT);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    for (int k = tid; k < kred_pad; k += TC_THREADS) offk[k] = (k < p.Kred) ? k_offset(p, k) : -1;
    pipe_start(pp, tail, geo.tmem_cols);

    const int total_tiles = geo.n_tiles * geo.oc_tiles;
    for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
        const int n0 = (tile % geo.n_tiles) * NT;
        const int oc0 = (tile / geo.n_tiles) * TC_M;
        for (int c = tid; c < NT; c += TC_THREADS) colb[c] = (n0 + c < p.N) ? col_base(p, n0 + c) : -1;
        __syncthreads();

        auto fill = [&](unsigned char* st, int kc) {
            const int kbase = kc * Tr::KC;
            // A: weight rows oc0 .. oc0+127, 8 units of 16 bytes per row.
            for (int u = tid; u < TC_M * 8; u += TC_THREADS) {
                const int r = u >> 3, c = u & 7;
                const int oc = oc0 + r, k = kbase + c * Tr::E;
                float v[8];
#pragma unroll
                for (int i = 0; i < Tr::E; ++i)
                    v[i] = (oc < p.OC && k + i < p.Kred) ? Elem<T>::ldg(w + size_t(oc) * p.Kred + k + i) : 0.f;
                put_unit<T, SWZ>(st, st + pp.half, r, c, v);
            }
            // B: gathered patch rows for the tile's columns.
            for (int u = tid; u < NT * 8; u += TC_THREADS) {
                const int r = u >> 3, c = u & 7;
                const int cb = colb[r], k = kbase + c * Tr::E;
                float v[8];
#pragma unroll
                for (int i = 0; i < Tr::E; ++i) {
                    const int off = offk[k + i];
                    v[i] = (cb >= 0 && off >= 0) ? Elem<T>::ldg(x + cb + off) : 0.f;
                }
                put_unit<T, SWZ>(st + pp.a_bytes, st + pp.half + pp.a_bytes, r, c, v);
            }
        };
        if (!pipe_tile<T, SWZ>(pp, nchunks, fill)) break;
        if (!pipe_wait_acc(pp)) break;

        // Epilogue: TMEM -> registers -> y (ReLU, one rounding).
        const int q = warp & 3, hcols = NT >> 1, c0 = (warp >> 2) * hcols;
        const int oc = oc0 + q * 32 + lane;
        for (int cb = 0; cb < hcols; cb += 8) {
            uint32_t r[8];
            tmem_ld8(pp.tmem + (uint32_t(q * 32) << 16) + uint32_t(c0 + cb), r);
            tmem_ld_wait();
            if (oc < p.OC) {
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int n = n0 + c0 + cb + e;
                    if (n < p.N) {
                        float v = __uint_as_float(r[e]);
                        if (RELU) v = v > 0.f ? v : 0.f;
                        Elem<T>::st(y + col_out(p, n) + size_t(oc) * p.P, v);
                    }
                }
            }
        }
        pipe_release_acc();
    }
    pipe_finish(pp, geo.tmem_cols);
}

// ======================================================================================
// wgrad partials: tile = (128 output channels, NT reduction indices k, one split range
// of columns n); the GEMM's K runs over the split's columns in chunks:
//   D[oc, k] = sum_{n in split} g[oc, n] * X[k, n]
// A unit = 16 bytes of g along n for one oc; B unit = 16 bytes of patches along n for
// one k.  The epilogue stores the fp32 tile to ws[split][oc][k] (row stride kpad).
// ======================================================================================
struct TcWgradGeom {
    int NT;        // k per tile (multiple of 16, <= 256)
    int k_tiles;   // ceil(Kred / NT)
    int oc_tiles;  // ceil(OC / 128)
    int splits;
    int kpad;      // workspace row stride (Kred rounded up to 4)
    int tmem_cols;
};

template <typename T>
inline int tc_wgrad_smem(int NT)
{
    return 1024 + TC_STAGES * tc_stage_bytes<T>(NT) + NT * 4 + int(sizeof(TcTail));
}

template <typename T, bool RELU, int SWZ>
__global__ void __launch_bounds__(TC_THREADS, 1)
wgrad_tc_kernel(const ConvParams p, const T* __restrict__ x, const T* __restrict__ dy,
                const T* __restrict__ y, float* __restrict__ ws, const TcWgradGeom geo)
{
    using Tr = TcTraits<T>;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = align1024(smem_raw);
    const int NT = geo.NT;
    TcPipe pp;
    pipe_setup<T>(pp, smem, NT);
    int* offk = reinterpret_cast<int*>(smem + TC_STAGES * pp.stage_bytes);
    TcTail* tail = reinterpret_cast<TcTail*>(offk + NT);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    pipe_start(pp, tail, geo.tmem_cols);

    const int per_split = geo.k_tiles * geo.oc_tiles;
    const int total = per_split * geo.splits;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
        const int split = tile / per_split, rem = tile % per_split;
        const int k0 = (rem % geo.k_tiles) * NT, oc0 = (rem / geo.k_tiles) * TC_M;
        const int n_lo = int((long long)p.N * split / geo.splits);
        const int n_hi = int((long long)p.N * (split + 1) / geo.splits);
        const int nchunks = (n_hi - n_lo + Tr::KC - 1) / Tr::KC;
        __syncthreads();  // previous tile's readers of offk are done
        for (int r = tid; r < NT; r += TC_THREADS) offk[r] = (k0 + r < p.Kred) ? k_offset(p, k0 + r) : -1;
        __syncthreads();

        auto fill = [&](unsigned char* st, int kc) {
            const int nbase = n_lo + kc * Tr::KC;
            for (int u = tid; u < TC_M * 8; u += TC_THREADS) {
                const int r = u >> 3, c = u & 7;
                const int oc = oc0 + r;
                float v[8];
#pragma unroll
                for (int i = 0; i < Tr::E; ++i) {
                    const int n = nbase + c * Tr::E + i;
                    float g = 0.f;
                    if (n < n_hi && oc < p.OC) {
                        const size_t gi = size_t(col_out(p, n)) + size_t(oc) * p.P;
                        g = Elem<T>::ldg(dy + gi);
                        if (RELU && !(Elem<T>::ldg(y + gi) > 0.f)) g = 0.f;
                    }
                    v[i] = g;
                }
                put_unit<T, SWZ>(st, st + pp.half, r, c, v);
            }
            for (int u = tid; u < NT * 8; u += TC_THREADS) {
                const int r = u >> 3, c = u & 7;
                const int off = offk[r];
                float v[8];
#pragma unroll
                for (int i = 0; i < Tr::E; ++i) {
                    const int n = nbase + c * Tr::E + i;
                    v[i] = (n < n_hi && off >= 0) ? Elem<T>::ldg(x + col_base(p, n) + off) : 0.f;
                }
                put_unit<T, SWZ>(st + pp.a_bytes, st + pp.half + pp.a_bytes, r, c, v);
            }
        };
        if (nchunks > 0) {
            if (!pipe_tile<T, SWZ>(pp, nchunks, fill)) break;
            if (!pipe_wait_acc(pp)) break;
        }

        const int q = warp & 3, hcols = NT >> 1, c0 = (warp >> 2) * hcols;
        const int oc = oc0 + q * 32 + lane;
        for (int cb = 0; cb < hcols; cb += 8) {
            uint32_t r[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            if (nchunks > 0) {  // an empty split range contributes zeros
                tmem_ld8(pp.tmem + (uint32_t(q * 32) << 16) + uint32_t(c0 + cb), r);
                tmem_ld_wait();
            }
            const int k = k0 + c0 + cb;
            if (oc < p.OC && k < geo.kpad) {
                float* dst = ws + (size_t(split) * p.OC + oc) * geo.kpad + k;
                *reinterpret_cast<float4*>(dst) = make_float4(__uint_as_float(r[0]), __uint_as_float(r[1]),
                                                              __uint_as_float(r[2]), __uint_as_float(r[3]));
                if (k + 4 < geo.kpad)
                    *reinterpret_cast<float4*>(dst + 4) = make_float4(__uint_as_float(r[4]), __uint_as_float(r[5]),
                                                                      __uint_as_float(r[6]), __uint_as_float(r[7]));
            }
        }
        pipe_release_acc();
    }
    pipe_finish(pp, geo.tmem_cols);
}

template <typename T> constexpr int dt_of_tc();
template <> constexpr int dt_of_tc<float>() { return DT_F32; }
template <> constexpr int dt_of_tc<__nv_bfloat16>() { return DT_BF16; }

int pow2_at_least(int v)
{
    int c = 32;
    while (c < v) c <<= 1;
    return c;
}

// Columns per tile: minimise (rounds of tiles over the grid) x (NT + 128), where 128
// stands for the per-tile cost of streaming the weight chunk (128 rows) next to the
// NT gathered rows.
int choose_nt(const ConvParams& p, int ctas)
{
    int best = 16;
    long best_cost = -1;
    const int oct = ceil_div(p.OC, TC_M);
    for (int nt = 16; nt <= 256; nt += 16) {
        const long tiles = long(ceil_div(p.N, nt)) * oct;
        const long rounds = (tiles + ctas - 1) / ctas;
        const long cost = rounds * (nt + 128);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = nt;
        }
    }
    return best;
}

int tc_swizzle_mode()
{
    static const int mode = [] {
        const char* e = getenv("IGC_TC_SWIZZLE");
        return (e && e[0] == '0') ? 0 : 1;
    }();
    return mode;
}

}  // namespace

bool tc_fwd_ok(const ConvParams& p, int dt, const DevInfo& d)
{
    if (d.cc_major != 10 || p.N <= 0) return false;
    const int nt = choose_nt(p, d.sms);
    return (dt == DT_BF16 ? tc_fwd_smem<__nv_bfloat16>(p, nt) : tc_fwd_smem<float>(p, nt)) <= d.smem_optin;
}

Plan plan_fwd_tc(const ConvParams& p, int dt, const DevInfo& d)
{
    Plan pl;
    pl.algo = ALGO_TC;
    pl.launches = 1;
    pl.block = TC_THREADS;
    const int nt = choose_nt(p, d.sms);
    pl.variant = nt;
    const int tiles = ceil_div(p.N, nt) * ceil_div(p.OC, TC_M);
    pl.grid = std::min(tiles, d.sms);
    pl.smem = dt == DT_BF16 ? tc_fwd_smem<__nv_bfloat16>(p, nt) : tc_fwd_smem<float>(p, nt);
    return pl;
}

template <typename T>
static cudaError_t fwd_tc_t(const Plan& pl, const ConvParams& p, const void* x, const void* w, void* y,
                            cudaStream_t s)
{
    TcFwdGeom g;
    g.NT = pl.variant;
    g.n_tiles = ceil_div(p.N, g.NT);
    g.oc_tiles = ceil_div(p.OC, TC_M);
    g.tmem_cols = pow2_at_least(g.NT);
    cudaError_t e = cudaSuccess;
    const bool swz = tc_swizzle_mode() != 0;
#define IG_LAUNCH_FWD_TC(R, Z)                                                                      \
    do {                                                                                            \
        e = ensure_smem<fwd_tc_kernel<T, R, Z>>(pl.smem);                                           \
        if (e == cudaSuccess)                                                                       \
            fwd_tc_kernel<T, R, Z><<<pl.grid, pl.block, pl.smem, s>>>(p, (const T*)x, (const T*)w, \
                                                                      (T*)y, g);                    \
    } while (0)
    if (p.relu) {
        if (swz) IG_LAUNCH_FWD_TC(true, 1); else IG_LAUNCH_FWD_TC(true, 0);
    } else {
        if (swz) IG_LAUNCH_FWD_TC(false, 1); else IG_LAUNCH_FWD_TC(false, 0);
    }
#undef IG_LAUNCH_FWD_TC
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t run_fwd_tc(const Plan& pl, const ConvParams& p, int dt, const void* x, const void* w, void* y,
                       cudaStream_t s)
{
    return dt == DT_F32 ? fwd_tc_t<float>(pl, p, x, w, y, s) : fwd_tc_t<__nv_bfloat16>(pl, p, x, w, y, s);
}

// ---- wgrad ------------------------------------------------------------------------------
static TcWgradGeom wgrad_geom(const ConvParams& p, int dt, int sms)
{
    TcWgradGeom g;
    g.NT = 128;
    g.k_tiles = ceil_div(p.Kred, g.NT);
    g.oc_tiles = ceil_div(p.OC, TC_M);
    g.kpad = round_up(p.Kred, 4);
    g.tmem_cols = pow2_at_least(g.NT);
    const int kc = dt == DT_BF16 ? TcTraits<__nv_bfloat16>::KC : TcTraits<float>::KC;
    const int tiles = g.k_tiles * g.oc_tiles;
    int splits = std::max(1, sms / tiles);
    splits = std::min(splits, std::max(1, p.N / (4 * kc)));  // >= 4 chunks per split
    g.splits = std::max(1, std::min(splits, std::max(1, p.N)));
    return g;
}

bool tc_wgrad_ok(const ConvParams& p, int dt, const DevInfo& d)
{
    if (d.cc_major != 10) return false;
    const int nt = 128;
    return (dt == DT_BF16 ? tc_wgrad_smem<__nv_bfloat16>(nt) : tc_wgrad_smem<float>(nt)) <= d.smem_optin;
}

Plan plan_wgrad_tc(const ConvParams& p, int dt, const DevInfo& d)
{
    Plan pl;
    pl.algo = ALGO_TC;
    pl.block = TC_THREADS;
    pl.smem = dt == DT_BF16 ? tc_wgrad_smem<__nv_bfloat16>(128) : tc_wgrad_smem<float>(128);
    if (p.N == 0) {
        pl.launches = 1;  // the reduction alone writes zeros
        pl.splits = 0;
        pl.grid = 1;
        return pl;
    }
    const TcWgradGeom g = wgrad_geom(p, dt, d.sms);
    pl.splits = g.splits;
    pl.launches = 2;
    const int tiles = g.k_tiles * g.oc_tiles * g.splits;
    pl.grid = std::min(tiles, d.sms);
    pl.workspace = size_t(g.splits) * p.OC * g.kpad * sizeof(float);
    return pl;
}

template <typename T>
static cudaError_t wgrad_tc_t(const Plan& pl, const ConvParams& p, const void* x, const void* dy,
                              const void* y, void* dw, void* ws, int sms, cudaStream_t s)
{
    cudaError_t e = cudaSuccess;
    const int kpad = round_up(p.Kred, 4);
    if (pl.splits > 0) {
        TcWgradGeom g = wgrad_geom(p, dt_of_tc<T>(), sms);
        g.splits = pl.splits;
        const bool swz = tc_swizzle_mode() != 0;
#define IG_LAUNCH_WG_TC(R, Z)                                                                              \
    do {                                                                                                   \
        e = ensure_smem<wgrad_tc_kernel<T, R, Z>>(pl.smem);                                                \
        if (e == cudaSuccess)                                                                              \
            wgrad_tc_kernel<T, R, Z><<<pl.grid, pl.block, pl.smem, s>>>(p, (const T*)x, (const T*)dy,      \
                                                                        (const T*)y, (float*)ws, g);       \
    } while (0)
        if (p.relu) {
            if (swz) IG_LAUNCH_WG_TC(true, 1); else IG_LAUNCH_WG_TC(true, 0);
        } else {
            if (swz) IG_LAUNCH_WG_TC(false, 1); else IG_LAUNCH_WG_TC(false, 0);
        }
#undef IG_LAUNCH_WG_TC
        if (e == cudaSuccess) e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return run_wgrad_reduce(p, dt_of_tc<T>(), (const float*)ws, pl.splits, kpad, dw, s);
}

cudaError_t run_wgrad_tc(const Plan& pl, const ConvParams& p, int dt, const void* x, const void* dy,
                         const void* y, void* dw, void* ws, int sms, cudaStream_t s)
{
    return dt == DT_F32 ? wgrad_tc_t<float>(pl, p, x, dy, y, dw, ws, sms, s)
                        : wgrad_tc_t<__nv_bfloat16>(pl, p, x, dy, y, dw, ws, sms, s);
}

cudaError_t tc_read_status(unsigned* out, bool reset)
{
    cudaError_t e = cudaMemcpyFromSymbol(out, g_tc_status, sizeof(unsigned));
    if (e == cudaSuccess && reset) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbol(g_tc_status, &zero, sizeof(unsigned));
    }
    return e;
}

}  // namespace igc
