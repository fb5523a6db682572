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

inline int pow2_at_least(int v)
{
    int c = 32;
    while (c < v) c <<= 1;
    return c;
}

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
__device__ __forceinline__ void issue_chunk(uint32_t tmem, uint32_t a_addr, uint32_t b_addr, uint32_t a_lo_off,
                                            uint32_t b_lo_off, uint32_t idesc, bool first)
{
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint64_t ad = op_desc<SWZ>(a_addr + kstep_off<SWZ>(j));
        const uint64_t bd = op_desc<SWZ>(b_addr + kstep_off<SWZ>(j));
        const uint32_t acc = (first && j == 0) ? 0u : 1u;
        if constexpr (TcTraits<T>::split) {
            const uint64_t al = op_desc<SWZ>(a_addr + a_lo_off + kstep_off<SWZ>(j));
            const uint64_t bl = op_desc<SWZ>(b_addr + b_lo_off + kstep_off<SWZ>(j));
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
__device__ __forceinline__ void pipe_setup(TcPipe& pp, unsigned char* smem, int NT, int a_rows = TC_M)
{
    using Tr = TcTraits<T>;
    pp.smem = smem;
    pp.smem_base = smem_u32(smem);
    pp.a_bytes = a_rows * ROWB;
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
// per chunk, lo parts `a_fixed_lo_off` further) instead of the stage.  Returns
// false if a wait ran out.
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
                                    pp.half, pp.idesc, kc == 0);
            else
                issue_chunk<T, SWZ>(pp.tmem, sa, sa + pp.a_bytes, pp.half, pp.half, pp.idesc, kc == 0);
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
// Forward: tile = (128 output channels, NT columns n); K = IC*K*K in chunks of KC.
// Warp roles (352 threads):
//   warps 0-1   copy: per chunk, move the raw slabs the chunk needs into a ring of
//               RAWS shared-memory slots with 16-byte cp.async copies: for each weight
//               row oc, the segment w[oc, k0 : k0+KC]; for each sample b the tile
//               touches, the contiguous channels x[b, ic_lo : ic_hi] that k0 .. k0+KC-1
//               cover.  Sources are rounded down to 16 bytes (the slack is skipped when
//               read) and the last block of a tensor is zero-filled past its end.
//               Each copy thread arrives on the slot's barrier when its copies land.
//   warp 2      MMA: one thread issues the chunk's tcgen05.mma steps into the TMEM
//               accumulator and commits to the stage's "empty" barrier, and after a
//               tile's last chunk to the accumulator barrier.
//   warps 3-10  formatters: build the A (weights) and B (gathered patches) operand
//               tiles of the chunk, 128-byte swizzled K-major, from the raw slot into
//               one of two operand stages; then the tile's epilogue (TMEM -> y).
// ======================================================================================
constexpr int FV_THREADS = 352;
constexpr int FV_COPY = 64;   // copy threads (warps 0-1)
constexpr int FV_MMA_WARP = 2;
constexpr int FV_FMT0 = 96;   // first formatter thread (warp 3)
constexpr int FV_OPS = 2;

struct FwdV2Geom {
    int NT, n_tiles, oc_tiles, tmem_cols;
    int nchunks;      // round_up(Kred, KC) / KC
    int raws;         // raw slots in the ring
    int nsmax;        // samples a tile can span
    int xs;           // bytes per sample in a raw slot
    int rw;           // bytes per weight row in a raw slot (KC * esize + 16)
    int raw_bytes;    // one raw slot: 128 * rw + nsmax * xs (rounded to 128)
    int op_bytes;     // one operand stage: (128 + NT) * 128 bytes, x2 for split fp32
};

struct FwdV2Bars {
    uint64_t raw_full[3], raw_empty[3], op_full[FV_OPS], op_empty[FV_OPS], acc_full;
    uint32_t tslot;
    int abort_flag;
};

template <typename T>
inline FwdV2Geom fwd_v2_geom(const ConvParams& p, int NT, int raws)
{
    using Tr = TcTraits<T>;
    const int es = int(sizeof(T));
    FwdV2Geom g;
    g.NT = NT;
    g.n_tiles = ceil_div(p.N, NT);
    g.oc_tiles = ceil_div(p.OC, TC_M);
    g.tmem_cols = pow2_at_least(NT);
    g.nchunks = round_up(p.Kred, Tr::KC) / Tr::KC;
    g.raws = raws;
    g.nsmax = std::min(p.B, (NT - 1) / p.P + 2);
    const int chmax = std::min(p.IC, (Tr::KC - 1) / p.KK + 2);
    g.xs = round_up(chmax * p.HW * es + 16, 16);
    g.rw = Tr::KC * es + 16;
    g.raw_bytes = round_up(TC_M * g.rw + g.nsmax * g.xs, 128);
    g.op_bytes = (TC_M + NT) * ROWB * (Tr::split ? 2 : 1);
    return g;
}

template <typename T>
inline int fwd_v2_smem(const ConvParams& p, const FwdV2Geom& g)
{
    const int kred_pad = round_up(p.Kred, TcTraits<T>::KC);
    return 1024 + FV_OPS * g.op_bytes + g.raws * g.raw_bytes + kred_pad * 4 + int(sizeof(FwdV2Bars)) + 16;
}

__device__ __forceinline__ int warp_sum(int v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// 16 bytes starting at a 2-byte-aligned shared address, as four 32-bit words.
__device__ __forceinline__ uint4 lds16_unaligned2(const unsigned char* p)
{
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    const uint32_t* w = reinterpret_cast<const uint32_t*>(a & ~uintptr_t(3));
    if ((a & 3) == 0) return make_uint4(w[0], w[1], w[2], w[3]);
    const uint32_t w0 = w[0], w1 = w[1], w2 = w[2], w3 = w[3], w4 = w[4];
    return make_uint4(__funnelshift_r(w0, w1, 16), __funnelshift_r(w1, w2, 16), __funnelshift_r(w2, w3, 16),
                      __funnelshift_r(w3, w4, 16));
}

template <typename T, int SWZ>
__device__ __forceinline__ void put_raw_unit(unsigned char* hi, unsigned char* lo, uint32_t off, uint4 v)
{
    if constexpr (TcTraits<T>::split) {
        float h[4], l[4];
        const float f[4] = {__uint_as_float(v.x), __uint_as_float(v.y), __uint_as_float(v.z), __uint_as_float(v.w)};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            h[i] = to_tf32(f[i]);
            l[i] = to_tf32(f[i] - h[i]);
        }
        st_unit(hi, off, __float_as_uint(h[0]), __float_as_uint(h[1]), __float_as_uint(h[2]), __float_as_uint(h[3]));
        st_unit(lo, off, __float_as_uint(l[0]), __float_as_uint(l[1]), __float_as_uint(l[2]), __float_as_uint(l[3]));
    } else {
        st_unit(hi, off, v.x, v.y, v.z, v.w);
    }
}

template <typename T, bool RELU, int SWZ>
__global__ void __launch_bounds__(FV_THREADS, 1)
fwd_tc_kernel(const ConvParams p, const T* __restrict__ x, const T* __restrict__ w, T* __restrict__ y,
              const FwdV2Geom geo)
{
    using Tr = TcTraits<T>;
    constexpr int ES = int(sizeof(T));
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = align1024(smem_raw);
    const int NT = geo.NT;
    const int kred_pad = round_up(p.Kred, Tr::KC);
    unsigned char* ops = smem;
    unsigned char* raw = ops + FV_OPS * geo.op_bytes;
    int* offk = reinterpret_cast<int*>(raw + geo.raws * geo.raw_bytes);
    FwdV2Bars* bars = reinterpret_cast<FwdV2Bars*>(offk + kred_pad);
    volatile int* abort_flag = &bars->abort_flag;
    const uint32_t a_bytes = TC_M * ROWB;
    const uint32_t half = (TC_M + NT) * ROWB;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    for (int k = tid; k < kred_pad; k += FV_THREADS) offk[k] = (k < p.Kred) ? k_offset(p, k) : -1;
    if (tid == 0) {
        for (int i = 0; i < geo.raws; ++i) {
            mbar_init(smem_u32(&bars->raw_full[i]), FV_COPY);
            mbar_init(smem_u32(&bars->raw_empty[i]), 8);
        }
        for (int i = 0; i < FV_OPS; ++i) {
            mbar_init(smem_u32(&bars->op_full[i]), 8);
            mbar_init(smem_u32(&bars->op_empty[i]), 1);
        }
        mbar_init(smem_u32(&bars->acc_full), 1);
        fence_mbar_init();
        bars->abort_flag = 0;
    }
    if (warp == 0) tmem_alloc(smem_u32(&bars->tslot), geo.tmem_cols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tslot;
    const int total_tiles = geo.n_tiles * geo.oc_tiles;

    if (warp < 2) {
        // ---------------- copy producers ----------------
        // Thread t copies weight rows t and t + 64 (up to rw/16 blocks each) and blocks
        // t, t + 64, ... of every sample's channel range.  Per-tile state is hoisted.
        const unsigned char* wb = reinterpret_cast<const unsigned char*>(w);
        const unsigned char* xb = reinterpret_cast<const unsigned char*>(x);
        const unsigned char* w_end = wb + size_t(p.OC) * p.Kred * ES;
        const unsigned char* x_end = xb + size_t(p.B) * p.IHW * ES;
        uint32_t q = 0;
        for (int tile = blockIdx.x; tile < total_tiles && !*abort_flag; tile += gridDim.x) {
            const int n0 = (tile % geo.n_tiles) * NT, oc0 = (tile / geo.n_tiles) * TC_M;
            const int n_end = min(n0 + NT, p.N);
            const int b_first = n0 / p.P, nsamp = (n_end - 1) / p.P - b_first + 1;
            const int rows = min(TC_M, p.OC - oc0);
            const unsigned char* wrow0 = wb + (size_t(oc0) + tid) * p.Kred * ES;        // row tid
            const unsigned char* wrow1 = wb + (size_t(oc0) + tid + 64) * p.Kred * ES;   // row tid + 64
            const bool has0 = tid < rows, has1 = tid + 64 < rows;
            for (int kc = 0; kc < geo.nchunks; ++kc, ++q) {
                const int s = q % geo.raws;
                const uint32_t use = q / geo.raws;
                if (use >= 1 && !mbar_wait_or_abort(smem_u32(&bars->raw_empty[s]), (use - 1) & 1, abort_flag)) {
                    report(const_cast<int*>(abort_flag), 4u);
                    break;
                }
                const int k0 = kc * Tr::KC;
                const int ic_lo = k0 / p.KK, ic_hi = min(p.IC - 1, (k0 + Tr::KC - 1) / p.KK);
                const int need_w = min(Tr::KC, p.Kred - k0) * ES;
                const uint32_t slot = smem_u32(raw + s * geo.raw_bytes);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    if (h == 0 ? !has0 : !has1) continue;
                    const unsigned char* src = (h == 0 ? wrow0 : wrow1) + k0 * ES;
                    const int d = int(reinterpret_cast<uintptr_t>(src) & 15);
                    src -= d;
                    const int nbk = (d + need_w + 15) >> 4;
                    const uint32_t dst = slot + (tid + 64 * h) * geo.rw;
                    for (int blk = 0; blk < nbk; ++blk) {
                        const long left = long(w_end - src);
                        cp_async16(dst + blk * 16, src, uint32_t(left < 16 ? left : 16));
                        src += 16;
                    }
                }
                const int need_x = (ic_hi - ic_lo + 1) * p.HW * ES;
                const uint32_t xslot = slot + TC_M * geo.rw;
                const unsigned char* xs0 = xb + (size_t(b_first) * p.IHW + size_t(ic_lo) * p.HW) * ES;
                for (int j = 0; j < nsamp; ++j) {
                    const unsigned char* src = xs0 + size_t(j) * p.IHW * ES;
                    const int d = int(reinterpret_cast<uintptr_t>(src) & 15);
                    src -= d;
                    const int nbk = (d + need_x + 15) >> 4;
                    const uint32_t dst = xslot + j * geo.xs;
                    for (int blk = tid; blk < nbk; blk += FV_COPY) {
                        const unsigned char* sb = src + blk * 16;
                        const long left = long(x_end - sb);
                        cp_async16(dst + blk * 16, sb, uint32_t(left < 16 ? left : 16));
                    }
                }
                cp_async_arrive_noinc(smem_u32(&bars->raw_full[s]));
            }
        }
    } else if (warp == FV_MMA_WARP) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            const uint32_t idesc = instr_desc(Tr::fmt, TC_M, NT);
            const uint32_t ops_u32 = smem_u32(ops);
            uint32_t q = 0;
            for (int tile = blockIdx.x; tile < total_tiles && !*abort_flag; tile += gridDim.x) {
                bool ok = true;
                for (int kc = 0; kc < geo.nchunks; ++kc, ++q) {
                    const int st = q % FV_OPS;
                    const uint32_t use = q / FV_OPS;
                    if (!mbar_wait_or_abort(smem_u32(&bars->op_full[st]), use & 1, abort_flag)) {
                        report(const_cast<int*>(abort_flag), 8u);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t base = ops_u32 + st * geo.op_bytes;
                    issue_chunk<T, SWZ>(tmem, base, base + a_bytes, half, half, idesc, kc == 0);
                    mma_commit(smem_u32(&bars->op_empty[st]));
                }
                if (!ok) break;
                mma_commit(smem_u32(&bars->acc_full));
            }
        }
        __syncwarp();
    } else {
        // ---------------- formatters + epilogue ----------------
        // Thread ft owns unit column cfix = ft & 7 of rows (ft >> 3) + 32 i: A rows i < 4,
        // B rows i < NT / 32.  All per-tile addressing is computed once per tile.
        const int ft = tid - FV_FMT0;  // 0 .. 255
        const int fw = warp - 3;       // 0 .. 7
        const int cfix = ft & 7;
        const int rbase = ft >> 3;     // 0 .. 31
        const int nbu = (NT + 31) >> 5;  // B rows per thread (the last may fall past NT)
        constexpr int MAXB = 8;        // NT <= 256
        uint32_t q = 0, t = 0;
        for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x, ++t) {
            const int n0 = (tile % geo.n_tiles) * NT, oc0 = (tile / geo.n_tiles) * TC_M;
            const int b_first = n0 / p.P;
            // A: raw-slot byte offset of each owned unit (the row's 16-byte slack is the same
            // for every chunk because a chunk advances the row by 128 bytes), or -1.
            int aoff[4];
            uint32_t adst[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int r = rbase + 32 * i;
                const int oc = oc0 + r;
                aoff[i] = oc < p.OC ? r * geo.rw + int(((size_t(oc) * p.Kred) * ES) & 15) + cfix * 16 : -1;
                adst[i] = unit_off<SWZ>(r, cfix);
            }
            // B: per owned row (column n): raw-slot byte offset of the sample's slab plus the
            // column's window origin, and the slab start's misalignment before the chunk.
            int boff[MAXB], bmis[MAXB];
            uint32_t bdst[MAXB];
#pragma unroll
            for (int i = 0; i < MAXB; ++i) {
                boff[i] = -1;
                bmis[i] = 0;
                bdst[i] = 0;
                if (i < nbu && rbase + 32 * i < NT) {
                    const int r = rbase + 32 * i;
                    const int n = n0 + r;
                    bdst[i] = unit_off<SWZ>(r, cfix);
                    boff[i] = -2;  // row inside the tile, column past N: zeros
                    if (n < p.N) {
                        uint32_t bq, pq, oh, ow;
                        p.dm_P.divmod(uint32_t(n), bq, pq);
                        p.dm_OW.divmod(pq, oh, ow);
                        boff[i] = TC_M * geo.rw + (int(bq) - b_first) * geo.xs +
                                  (int(oh) * p.S * p.W + int(ow) * p.S) * ES;
                        bmis[i] = int((size_t(bq) * p.IHW * ES) & 15);
                    }
                }
            }
            bool ok = true;
            for (int kc = 0; kc < geo.nchunks; ++kc, ++q) {
                const int s = q % geo.raws;
                const int st = q % FV_OPS;
                const uint32_t ruse = q / geo.raws, ouse = q / FV_OPS;
                if (!mbar_wait_or_abort(smem_u32(&bars->raw_full[s]), ruse & 1, abort_flag) ||
                    (ouse >= 1 && !mbar_wait_or_abort(smem_u32(&bars->op_empty[st]), (ouse - 1) & 1, abort_flag))) {
                    report(const_cast<int*>(abort_flag), 1u);
                    ok = false;
                    break;
                }
                const int k0 = kc * Tr::KC;
                const int ic_lo = k0 / p.KK;
                const unsigned char* slot = raw + s * geo.raw_bytes;
                unsigned char* op = ops + st * geo.op_bytes;
                const int kv = p.Kred - (k0 + cfix * Tr::E);  // valid elements in owned A / B units
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    uint4 v = make_uint4(0, 0, 0, 0);
                    if (aoff[i] >= 0 && kv > 0) {
                        const unsigned char* src = slot + aoff[i];
                        if constexpr (ES == 2) {
                            v = lds16_unaligned2(src);
                        } else {
                            const uint32_t* w4 = reinterpret_cast<const uint32_t*>(src);
                            v = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                        }
                        if (kv < Tr::E) {
                            uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                            for (int e = 0; e < Tr::E; ++e) {
                                if (e >= kv) {
                                    if constexpr (ES == 2) wv[e >> 1] &= (e & 1) ? 0x0000FFFFu : 0xFFFF0000u;
                                    else wv[e] = 0u;
                                }
                            }
                            v = make_uint4(wv[0], wv[1], wv[2], wv[3]);
                        }
                    }
                    put_raw_unit<T, SWZ>(op, op + half, adst[i], v);
                }
                // This thread's E k offsets, in bytes from the chunk's first channel.
                int ko[Tr::E];
#pragma unroll
                for (int e = 0; e < Tr::E; ++e) {
                    const int kk = offk[k0 + cfix * Tr::E + e];
                    ko[e] = kk >= 0 ? (kk - ic_lo * p.HW) * ES : -1;
                }
                const int cmis = (ic_lo * p.HW * ES) & 15;
#pragma unroll
                for (int i = 0; i < MAXB; ++i) {
                    if (i >= nbu) break;
                    if (boff[i] == -1) continue;  // row past NT: not part of the tile
                    uint32_t wv[4] = {0, 0, 0, 0};
                    if (boff[i] >= 0) {
                        const unsigned char* src = slot + boff[i] + ((bmis[i] + cmis) & 15);
#pragma unroll
                        for (int e = 0; e < Tr::E; ++e) {
                            if (ko[e] >= 0) {
                                if constexpr (ES == 2) {
                                    const uint32_t h = *reinterpret_cast<const unsigned short*>(src + ko[e]);
                                    wv[e >> 1] |= (e & 1) ? (h << 16) : h;
                                } else {
                                    wv[e] = *reinterpret_cast<const uint32_t*>(src + ko[e]);
                                }
                            }
                        }
                    }
                    put_raw_unit<T, SWZ>(op + a_bytes, op + half + a_bytes, bdst[i],
                                         make_uint4(wv[0], wv[1], wv[2], wv[3]));
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(smem_u32(&bars->op_full[st]));
                    mbar_arrive(smem_u32(&bars->raw_empty[s]));
                }
            }
            if (!ok) break;
            // Epilogue: TMEM -> y.
            if (!mbar_wait_or_abort(smem_u32(&bars->acc_full), t & 1, abort_flag)) {
                report(const_cast<int*>(abort_flag), 2u);
                break;
            }
            tc_fence_after();
            const int qd = warp & 3, hcols = NT >> 1, c0 = (fw >> 2) * hcols;
            const int oc = oc0 + qd * 32 + lane;
            for (int cb = 0; cb < hcols; cb += 8) {
                uint32_t r[8];
                tmem_ld8(tmem + (uint32_t(qd * 32) << 16) + uint32_t(c0 + cb), r);
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
            tc_fence_before();
        }
    }
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, geo.tmem_cols);
    }
}

// ======================================================================================
// wgrad partials: tile = (128 output channels, NT reduction indices k, one split range of
// samples); the GEMM's K runs over the split's columns n = (b, oh, ow), a chunk being NSC
// whole samples (NSC*P <= KC columns, the rest zero):
//   D[oc, k] = sum_{n in split} g[oc, n] * X[k, n]
// Same warp roles as the forward kernel.  Per chunk the copy warps bring, for each of
// the chunk's samples, the contiguous slabs dy[b, oc0 : oc0+128, :], y[b, oc0 : ..] (ReLU
// mask source) and x[b, ic_lo : ic_hi] (the k-tile's input channels); the formatters
// build A (g = dy * [y > 0] along n per oc) and B (patches along n per k).  The
// epilogue stores the fp32 tile to ws[split][oc][k] (row stride kpad).
// ======================================================================================
struct TcWgradGeom {
    int NT;        // k per tile (multiple of 16, <= 128)
    int k_tiles;   // ceil(Kred / NT)
    int oc_tiles;  // ceil(OC / 128)
    int splits;    // sample ranges
    int kpad;      // workspace row stride (Kred rounded up to 4)
    int tmem_cols;
    int nsc;       // samples per chunk
    int raws;      // raw slots
    int gs;        // bytes per sample of a dy (or y) slab in a raw slot
    int xsb;       // bytes per sample of the x channels in a raw slot
    int raw_bytes;
    int op_bytes;
};

struct WgBars {
    uint64_t raw_full[3], raw_empty[3], op_full[FV_OPS], op_empty[FV_OPS], acc_full;
    uint32_t tslot;
    int abort_flag;
};

template <typename T>
inline TcWgradGeom wgrad_v3_geom(const ConvParams& p, int NT, int raws, int splits)
{
    using Tr = TcTraits<T>;
    const int es = int(sizeof(T));
    TcWgradGeom g;
    g.NT = NT;
    g.k_tiles = ceil_div(p.Kred, NT);
    g.oc_tiles = ceil_div(p.OC, TC_M);
    g.splits = splits;
    g.kpad = round_up(p.Kred, 4);
    g.tmem_cols = pow2_at_least(NT);
    g.nsc = std::max(1, Tr::KC / std::max(1, p.P));
    g.raws = raws;
    g.gs = round_up(std::min(p.OC, TC_M) * p.P * es + 16, 16);
    const int chk = std::min(p.IC, (NT - 1) / p.KK + 2);
    g.xsb = round_up(chk * p.HW * es + 16, 16);
    g.raw_bytes = round_up(g.nsc * (g.gs * (p.relu ? 2 : 1) + g.xsb), 128);
    g.op_bytes = (TC_M + NT) * ROWB * (Tr::split ? 2 : 1);
    return g;
}

template <typename T>
inline int wgrad_v3_smem(const TcWgradGeom& g)
{
    return 1024 + FV_OPS * g.op_bytes + g.raws * g.raw_bytes + g.NT * 4 + int(sizeof(WgBars)) + 16;
}

// Distribute 16-byte cp.async copies of the global byte range [off, off + bytes) of
// `base` (rounded out to 16-byte blocks) over threads t, t + nthr, ...; the first block
// lands at shared address dst.  Blocks are zero-filled past `end`.
__device__ __forceinline__ void copy_range(uint32_t dst, const unsigned char* base, size_t off, int bytes,
                                           const unsigned char* end, int t, int nthr)
{
    const size_t a = off & ~size_t(15);
    const int nb = int((off + size_t(bytes) - a + 15) >> 4);
    for (int i = t; i < nb; i += nthr) {
        const unsigned char* src = base + a + size_t(i) * 16;
        const long left = long(end - src);
        cp_async16(dst + i * 16, src, uint32_t(left < 16 ? left : 16));
    }
}

template <typename T, bool RELU, int SWZ>
__global__ void __launch_bounds__(FV_THREADS, 1)
wgrad_tc_kernel(const ConvParams p, const T* __restrict__ x, const T* __restrict__ dy,
                const T* __restrict__ y, float* __restrict__ ws, const TcWgradGeom geo)
{
    using Tr = TcTraits<T>;
    constexpr int ES = int(sizeof(T));
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = align1024(smem_raw);
    const int NT = geo.NT;
    unsigned char* ops = smem;
    unsigned char* raw = ops + FV_OPS * geo.op_bytes;
    int* offk = reinterpret_cast<int*>(raw + geo.raws * geo.raw_bytes);  // [NT], per tile
    WgBars* bars = reinterpret_cast<WgBars*>(offk + NT);
    volatile int* abort_flag = &bars->abort_flag;
    const uint32_t a_bytes = TC_M * ROWB;
    const uint32_t half = (TC_M + NT) * ROWB;
    const int gsz = geo.gs, nslab = RELU ? 2 : 1;
    const int per_sample = gsz * nslab + geo.xsb;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int i = 0; i < geo.raws; ++i) {
            mbar_init(smem_u32(&bars->raw_full[i]), FV_COPY);
            mbar_init(smem_u32(&bars->raw_empty[i]), 8);
        }
        for (int i = 0; i < FV_OPS; ++i) {
            mbar_init(smem_u32(&bars->op_full[i]), 8);
            mbar_init(smem_u32(&bars->op_empty[i]), 1);
        }
        mbar_init(smem_u32(&bars->acc_full), 1);
        fence_mbar_init();
        bars->abort_flag = 0;
    }
    if (warp == 0) tmem_alloc(smem_u32(&bars->tslot), geo.tmem_cols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tslot;
    const int per_split = geo.k_tiles * geo.oc_tiles;
    const int total = per_split * geo.splits;

    // Tile decode shared by all roles.
    struct TileInfo {
        int split, k0, oc0, rows, s_lo, s_hi, nchunks, ic_lo, ic_hi;
    };
    auto decode = [&](int tile) {
        TileInfo ti;
        ti.split = tile / per_split;
        const int rem = tile % per_split;
        ti.k0 = (rem % geo.k_tiles) * NT;
        ti.oc0 = (rem / geo.k_tiles) * TC_M;
        ti.rows = min(TC_M, p.OC - ti.oc0);
        ti.s_lo = int((long long)p.B * ti.split / geo.splits);
        ti.s_hi = int((long long)p.B * (ti.split + 1) / geo.splits);
        ti.nchunks = (ti.s_hi - ti.s_lo + geo.nsc - 1) / geo.nsc;
        ti.ic_lo = ti.k0 / p.KK;
        ti.ic_hi = min(p.IC - 1, (min(ti.k0 + NT, p.Kred) - 1) / p.KK);
        return ti;
    };

    if (warp < 2) {
        // ---------------- copy producers ----------------
        const unsigned char* xb = reinterpret_cast<const unsigned char*>(x);
        const unsigned char* gb = reinterpret_cast<const unsigned char*>(dy);
        const unsigned char* yb = reinterpret_cast<const unsigned char*>(y);
        const unsigned char* x_end = xb + size_t(p.B) * p.IHW * ES;
        const unsigned char* g_end = gb + size_t(p.B) * p.OCP * ES;
        const unsigned char* y_end = yb + size_t(p.B) * p.OCP * ES;
        uint32_t q = 0;
        for (int tile = blockIdx.x; tile < total && !*abort_flag; tile += gridDim.x) {
            const TileInfo ti = decode(tile);
            const int gbytes = ti.rows * p.P * ES;
            const int xbytes = (ti.ic_hi - ti.ic_lo + 1) * p.HW * ES;
            for (int kc = 0; kc < ti.nchunks; ++kc, ++q) {
                const int s = q % geo.raws;
                const uint32_t use = q / geo.raws;
                if (use >= 1 && !mbar_wait_or_abort(smem_u32(&bars->raw_empty[s]), (use - 1) & 1, abort_flag)) {
                    report(const_cast<int*>(abort_flag), 4u);
                    break;
                }
                const uint32_t slot = smem_u32(raw + s * geo.raw_bytes);
                const int b0 = ti.s_lo + kc * geo.nsc, nb = min(geo.nsc, ti.s_hi - b0);
                for (int j = 0; j < nb; ++j) {
                    const int b = b0 + j;
                    const size_t go = (size_t(b) * p.OCP + size_t(ti.oc0) * p.P) * ES;
                    const uint32_t sj = slot + j * per_sample;
                    copy_range(sj, gb, go, gbytes, g_end, tid, FV_COPY);
                    if (RELU) copy_range(sj + gsz, yb, go, gbytes, y_end, tid, FV_COPY);
                    copy_range(sj + gsz * nslab, xb, (size_t(b) * p.IHW + size_t(ti.ic_lo) * p.HW) * ES, xbytes,
                               x_end, tid, FV_COPY);
                }
                cp_async_arrive_noinc(smem_u32(&bars->raw_full[s]));
            }
        }
    } else if (warp == FV_MMA_WARP) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            const uint32_t idesc = instr_desc(Tr::fmt, TC_M, NT);
            const uint32_t ops_u32 = smem_u32(ops);
            uint32_t q = 0;
            for (int tile = blockIdx.x; tile < total && !*abort_flag; tile += gridDim.x) {
                const TileInfo ti = decode(tile);
                bool ok = true;
                for (int kc = 0; kc < ti.nchunks; ++kc, ++q) {
                    const int st = q % FV_OPS;
                    const uint32_t use = q / FV_OPS;
                    if (!mbar_wait_or_abort(smem_u32(&bars->op_full[st]), use & 1, abort_flag)) {
                        report(const_cast<int*>(abort_flag), 8u);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t base = ops_u32 + st * geo.op_bytes;
                    issue_chunk<T, SWZ>(tmem, base, base + a_bytes, half, half, idesc, kc == 0);
                    mma_commit(smem_u32(&bars->op_empty[st]));
                }
                if (!ok) break;
                mma_commit(smem_u32(&bars->acc_full));
            }
        }
        __syncwarp();
    } else {
        // ---------------- formatters + epilogue ----------------
        const int ft = tid - FV_FMT0;
        const int fw = warp - 3;
        const int cfix = ft & 7;
        // This thread's chunk columns n' = cfix*E + e -> (sample j, position pq) never change.
        int jj[Tr::E], pq[Tr::E], po[Tr::E];
#pragma unroll
        for (int e = 0; e < Tr::E; ++e) {
            const int n = cfix * Tr::E + e;
            uint32_t j, r;
            p.dm_P.divmod(uint32_t(n), j, r);
            jj[e] = int(j);
            pq[e] = int(r);
            uint32_t oh, ow;
            p.dm_OW.divmod(r, oh, ow);
            po[e] = int(oh) * p.S * p.W + int(ow) * p.S;
        }
        uint32_t q = 0, t = 0;
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++t) {
            const TileInfo ti = decode(tile);
            // k-offset table for this tile (relative to ic_lo); formatters only.
            asm volatile("bar.sync 1, 256;" ::: "memory");
            for (int r = ft; r < NT; r += 256) {
                const int k = ti.k0 + r;
                offk[r] = (k < p.Kred) ? k_offset(p, k) - ti.ic_lo * p.HW : -1;
            }
            asm volatile("bar.sync 1, 256;" ::: "memory");
            bool ok = true;
            for (int kc = 0; kc < ti.nchunks; ++kc, ++q) {
                const int s = q % geo.raws;
                const int st = q % FV_OPS;
                const uint32_t ruse = q / geo.raws, ouse = q / FV_OPS;
                if (!mbar_wait_or_abort(smem_u32(&bars->raw_full[s]), ruse & 1, abort_flag) ||
                    (ouse >= 1 && !mbar_wait_or_abort(smem_u32(&bars->op_empty[st]), (ouse - 1) & 1, abort_flag))) {
                    report(const_cast<int*>(abort_flag), 1u);
                    ok = false;
                    break;
                }
                const int b0 = ti.s_lo + kc * geo.nsc;
                const int nb = min(geo.nsc, ti.s_hi - b0);
                const unsigned char* slot = raw + s * geo.raw_bytes;
                unsigned char* op = ops + st * geo.op_bytes;
                // Start of each element's sample slabs in the raw slot, including the
                // 16-byte rounding slack of its copy.
                const unsigned char* gsrc[Tr::E];
                const unsigned char* xsrc[Tr::E];
#pragma unroll
                for (int e = 0; e < Tr::E; ++e) {
                    const size_t b = size_t(b0 + jj[e]);
                    const unsigned char* sj = slot + jj[e] * per_sample;
                    gsrc[e] = sj + int(((b * p.OCP + size_t(ti.oc0) * p.P) * ES) & 15);
                    xsrc[e] = sj + gsz * nslab + int(((b * p.IHW + size_t(ti.ic_lo) * p.HW) * ES) & 15);
                }
                // A: g rows (oc), 16 bytes of columns per unit.
                for (int u = ft; u < TC_M * 8; u += 256) {
                    const int r = u >> 3;
                    uint32_t wv[4] = {0, 0, 0, 0};
                    if (r < ti.rows) {
#pragma unroll
                        for (int e = 0; e < Tr::E; ++e) {
                            if (jj[e] < nb) {
                                const unsigned char* sj = gsrc[e];
                                const int gi = r * p.P + pq[e];
                                if constexpr (ES == 2) {
                                    uint32_t h = *reinterpret_cast<const unsigned short*>(sj + gi * 2);
                                    if (RELU) {
                                        const float yv = __bfloat162float(
                                            *reinterpret_cast<const __nv_bfloat16*>(sj + gsz + gi * 2));
                                        if (!(yv > 0.f)) h = 0;
                                    }
                                    wv[e >> 1] |= (e & 1) ? (h << 16) : h;
                                } else {
                                    uint32_t v = *reinterpret_cast<const uint32_t*>(sj + gi * 4);
                                    if (RELU && !(*reinterpret_cast<const float*>(sj + gsz + gi * 4) > 0.f)) v = 0;
                                    wv[e] = v;
                                }
                            }
                        }
                    }
                    put_raw_unit<T, SWZ>(op, op + half, unit_off<SWZ>(r, cfix), make_uint4(wv[0], wv[1], wv[2], wv[3]));
                }
                // B: patch rows (k), 16 bytes of columns per unit.
                for (int u = ft; u < NT * 8; u += 256) {
                    const int r = u >> 3;
                    const int ko = offk[r];
                    uint32_t wv[4] = {0, 0, 0, 0};
                    if (ko >= 0) {
#pragma unroll
                        for (int e = 0; e < Tr::E; ++e) {
                            if (jj[e] < nb) {
                                const unsigned char* xs = xsrc[e];
                                if constexpr (ES == 2) {
                                    const uint32_t h = *reinterpret_cast<const unsigned short*>(xs + (ko + po[e]) * 2);
                                    wv[e >> 1] |= (e & 1) ? (h << 16) : h;
                                } else {
                                    wv[e] = *reinterpret_cast<const uint32_t*>(xs + (ko + po[e]) * 4);
                                }
                            }
                        }
                    }
                    put_raw_unit<T, SWZ>(op + a_bytes, op + half + a_bytes, unit_off<SWZ>(r, cfix),
                                         make_uint4(wv[0], wv[1], wv[2], wv[3]));
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(smem_u32(&bars->op_full[st]));
                    mbar_arrive(smem_u32(&bars->raw_empty[s]));
                }
            }
            if (!ok) break;
            if (!mbar_wait_or_abort(smem_u32(&bars->acc_full), t & 1, abort_flag)) {
                report(const_cast<int*>(abort_flag), 2u);
                break;
            }
            tc_fence_after();
            const int qd = warp & 3, hcols = NT >> 1, c0 = (fw >> 2) * hcols;
            const int oc = ti.oc0 + qd * 32 + lane;
            for (int cb = 0; cb < hcols; cb += 8) {
                uint32_t r[8];
                tmem_ld8(tmem + (uint32_t(qd * 32) << 16) + uint32_t(c0 + cb), r);
                tmem_ld_wait();
                const int k = ti.k0 + c0 + cb;
                if (oc < p.OC && k < geo.kpad) {
                    float* dst = ws + (size_t(ti.split) * p.OC + oc) * geo.kpad + k;
                    *reinterpret_cast<float4*>(dst) = make_float4(__uint_as_float(r[0]), __uint_as_float(r[1]),
                                                                  __uint_as_float(r[2]), __uint_as_float(r[3]));
                    if (k + 4 < geo.kpad)
                        *reinterpret_cast<float4*>(dst + 4) = make_float4(
                            __uint_as_float(r[4]), __uint_as_float(r[5]), __uint_as_float(r[6]), __uint_as_float(r[7]));
                }
            }
            tc_fence_before();
        }
    }
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, geo.tmem_cols);
    }
}

// ======================================================================================
// d_input: tile = (one chunk of CIC input channels -> M = CIC*K*K <= 128 rows k, NS whole
// samples -> NS*P columns n); the GEMM's K runs over output channels:
//   D[k, n] = sum_oc W[oc, k] * g[oc, n]
// Each CTA keeps its channel chunk's W^T tile (all OC) resident in shared memory and
// streams its range of samples through the stages.  The epilogue stages D in shared
// memory as [n][k] fp32 (over the idle stage buffers) and gathers
//   dx[b, ic, h, w] = sum over (oh, kh) with oh*S + kh = h and (ow, kw) with ow*S + kw = w
//                     of D[(ic, kh, kw), (b, oh, ow)]
// in a fixed order: no atomics, bit-reproducible.
// ======================================================================================
struct TcDgradGeom {
    int NS;         // samples per tile
    int NT;         // columns per tile = round_up(NS * P, 16) <= 128
    int CIC;        // input channels per chunk
    int nkt;        // channel chunks
    int cpk;        // CTAs per channel chunk
    int nch;        // reduction chunks over OC
    int rmax;       // max (oh, kh) pairs per input row = ceil(K / S)
    int tmem_cols;
};

template <typename T>
inline int tc_dgrad_smem(const ConvParams& p, const TcDgradGeom& g)
{
    using Tr = TcTraits<T>;
    const int a = g.nch * TC_M * ROWB * (Tr::split ? 2 : 1);
    const int stages = TC_STAGES * g.NT * ROWB * (Tr::split ? 2 : 1);
    const int region = std::max(stages, g.NT * TC_M * 4);
    return 1024 + a + region + (p.H + p.W) * (1 + g.rmax) * 8 + int(sizeof(TcTail));
}

template <typename T, bool RELU, int SWZ>
__global__ void __launch_bounds__(TC_THREADS, 1)
dgrad_tc_kernel(const ConvParams p, const T* __restrict__ dy, const T* __restrict__ w,
                const T* __restrict__ y, T* __restrict__ dx, const TcDgradGeom geo)
{
    using Tr = TcTraits<T>;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = align1024(smem_raw);
    const int NT = geo.NT;
    const uint32_t a_chunk = TC_M * ROWB;
    const uint32_t a_total = geo.nch * a_chunk;  // hi parts; lo parts follow for fp32
    unsigned char* Ares = smem;
    unsigned char* region = smem + a_total * (Tr::split ? 2 : 1);
    TcPipe pp;
    pipe_setup<T>(pp, region, NT, 0);
    const int rbytes = max(int(TC_STAGES * pp.stage_bytes), NT * TC_M * 4);
    float* Ds = reinterpret_cast<float*>(region);
    const int R1 = 1 + geo.rmax;
    int2* rtab = reinterpret_cast<int2*>(region + rbytes);
    int2* ctab = rtab + p.H * R1;
    TcTail* tail = reinterpret_cast<TcTail*>(ctab + p.W * R1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int kt = blockIdx.x % geo.nkt, j = blockIdx.x / geo.nkt;
    const int ic0 = kt * geo.CIC, nic = min(geo.CIC, p.IC - ic0);
    const int k0 = ic0 * p.KK, mrows = nic * p.KK;

    for (int h = tid; h < p.H; h += TC_THREADS) {
        int n = 0;
        for (int oh = 0; oh < p.OH; ++oh) {
            const int kh = h - oh * p.S;
            if (kh >= 0 && kh < p.K) rtab[h * R1 + 1 + n++] = make_int2(oh * p.OW, kh * p.K);
        }
        rtab[h * R1] = make_int2(n, 0);
    }
    for (int c = tid; c < p.W; c += TC_THREADS) {
        int n = 0;
        for (int ow = 0; ow < p.OW; ++ow) {
            const int kw = c - ow * p.S;
            if (kw >= 0 && kw < p.K) ctab[c * R1 + 1 + n++] = make_int2(ow, kw);
        }
        ctab[c * R1] = make_int2(n, 0);
    }
    // Resident A: row m = k0 + m of W^T, all output channels, chunk by chunk.
    for (int kc = 0; kc < geo.nch; ++kc) {
        for (int u = tid; u < TC_M * 8; u += TC_THREADS) {
            const int r = u >> 3, c = u & 7;
            float v[8];
#pragma unroll
            for (int i = 0; i < Tr::E; ++i) {
                const int oc = kc * Tr::KC + c * Tr::E + i;
                v[i] = (r < mrows && oc < p.OC) ? Elem<T>::ldg(w + size_t(oc) * p.Kred + k0 + r) : 0.f;
            }
            put_unit<T, SWZ>(Ares + kc * a_chunk, Ares + a_total + kc * a_chunk, r, c, v);
        }
    }
    pipe_start(pp, tail, geo.tmem_cols);

    const int b_lo = int((long long)p.B * j / geo.cpk), b_hi = int((long long)p.B * (j + 1) / geo.cpk);
    const int span = nic * p.HW;
    for (int sb = b_lo; sb < b_hi; sb += geo.NS) {
        const int ns = min(geo.NS, b_hi - sb);
        const int ncols = ns * p.P;
        auto fill = [&](unsigned char* st, int kc) {
            for (int u = tid; u < NT * 8; u += TC_THREADS) {
                const int r = u >> 3, c = u & 7;
                float v[8];
                if (r < ncols) {
                    uint32_t si, pq;
                    p.dm_P.divmod(uint32_t(r), si, pq);
                    const size_t base = size_t(sb + int(si)) * p.OCP + pq;
#pragma unroll
                    for (int i = 0; i < Tr::E; ++i) {
                        const int oc = kc * Tr::KC + c * Tr::E + i;
                        float g = 0.f;
                        if (oc < p.OC) {
                            g = Elem<T>::ldg(dy + base + size_t(oc) * p.P);
                            if (RELU && !(Elem<T>::ldg(y + base + size_t(oc) * p.P) > 0.f)) g = 0.f;
                        }
                        v[i] = g;
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i) v[i] = 0.f;
                }
                put_unit<T, SWZ>(st, st + pp.half, r, c, v);
            }
        };
        if (!pipe_tile<T, SWZ>(pp, geo.nch, fill, smem_u32(Ares), a_total)) break;
        if (!pipe_wait_acc(pp)) break;

        // TMEM (lane = k row, column = n) -> Ds[n][k].
        const int q = warp & 3, hcols = NT >> 1, c0 = (warp >> 2) * hcols;
        const int m = q * 32 + lane;
        for (int cb = 0; cb < hcols; cb += 8) {
            uint32_t r[8];
            tmem_ld8(pp.tmem + (uint32_t(q * 32) << 16) + uint32_t(c0 + cb), r);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 8; ++e) Ds[(c0 + cb + e) * TC_M + m] = __uint_as_float(r[e]);
        }
        tc_fence_before();
        __syncthreads();

        for (int s = 0; s < ns; ++s) {
            T* dxs = dx + size_t(sb + s) * p.IHW + size_t(ic0) * p.HW;
            const float* ds = Ds + s * p.P * TC_M;
            for (int t = tid; t < span; t += TC_THREADS) {
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
                        sum += ds[(rr[a].x + cc[bq].x) * TC_M + kb + rr[a].y + cc[bq].y];
                Elem<T>::st(dxs + t, sum);
            }
        }
        __syncthreads();  // Ds (over the stages) consumed before the next tile's fill
    }
    pipe_finish(pp, geo.tmem_cols);
}

template <typename T> constexpr int dt_of_tc();
template <> constexpr int dt_of_tc<float>() { return DT_F32; }
template <> constexpr int dt_of_tc<__nv_bfloat16>() { return DT_BF16; }



int tc_swizzle_mode()
{
    static const int mode = [] {
        const char* e = getenv("IGC_TC_SWIZZLE");
        return (e && e[0] == '0') ? 0 : 1;
    }();
    return mode;
}

}  // namespace

// Tile width NT and raw-ring depth for the forward kernel: the feasible (shared memory)
// choice minimising (rounds of tiles over the grid) x (NT + 128), where 128 stands for
// the per-tile cost of the 128 weight rows next to the NT gathered rows; a 3-slot ring
// is preferred over 2 at equal cost.
template <typename T>
static bool pick_fwd_v2(const ConvParams& p, const DevInfo& d, FwdV2Geom& out)
{
    bool found = false;
    long best = 0;
    const int oct = ceil_div(p.OC, TC_M);
    for (int nt = 16; nt <= 256; nt += 16) {
        for (int raws = 3; raws >= 2; --raws) {
            const FwdV2Geom g = fwd_v2_geom<T>(p, nt, raws);
            if (fwd_v2_smem<T>(p, g) > d.smem_optin) continue;
            const long tiles = long(ceil_div(p.N, nt)) * oct;
            const long cost = ((tiles + d.sms - 1) / d.sms) * (nt + 128) * (raws == 3 ? 20 : 21);
            if (!found || cost < best) {
                best = cost;
                out = g;
                found = true;
            }
            break;  // the deepest feasible ring for this NT
        }
    }
    return found;
}

bool tc_fwd_ok(const ConvParams& p, int dt, const DevInfo& d)
{
    if (d.cc_major != 10 || p.N <= 0) return false;
    FwdV2Geom g;
    return dt == DT_BF16 ? pick_fwd_v2<__nv_bfloat16>(p, d, g) : pick_fwd_v2<float>(p, d, g);
}

Plan plan_fwd_tc(const ConvParams& p, int dt, const DevInfo& d)
{
    FwdV2Geom g;
    if (dt == DT_BF16) pick_fwd_v2<__nv_bfloat16>(p, d, g);
    else pick_fwd_v2<float>(p, d, g);
    Plan pl;
    pl.algo = ALGO_TC;
    pl.launches = 1;
    pl.block = FV_THREADS;
    pl.variant = g.NT * 4 + g.raws;
    pl.grid = std::min(g.n_tiles * g.oc_tiles, d.sms);
    pl.smem = dt == DT_BF16 ? fwd_v2_smem<__nv_bfloat16>(p, g) : fwd_v2_smem<float>(p, g);
    return pl;
}

template <typename T>
static cudaError_t fwd_tc_t(const Plan& pl, const ConvParams& p, const void* x, const void* w, void* y,
                            cudaStream_t s)
{
    const FwdV2Geom g = fwd_v2_geom<T>(p, pl.variant / 4, pl.variant % 4);
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
// Split count: enough tiles to cover the SMs, at least two chunks per split.
template <typename T>
static bool pick_wgrad_v3(const ConvParams& p, const DevInfo& d, TcWgradGeom& out)
{
    if (p.P > TcTraits<T>::KC || p.B <= 0) return false;
    for (int nt : {128, 64, 32}) {
        const int tiles = ceil_div(p.Kred, nt) * ceil_div(p.OC, TC_M);
        const int nsc = std::max(1, TcTraits<T>::KC / p.P);
        int splits = std::max(1, d.sms / tiles);
        splits = std::min(splits, std::max(1, p.B / (2 * nsc)));
        for (int raws = 3; raws >= 2; --raws) {
            const TcWgradGeom g = wgrad_v3_geom<T>(p, nt, raws, splits);
            if (wgrad_v3_smem<T>(g) <= d.smem_optin) {
                out = g;
                return true;
            }
        }
    }
    return false;
}

bool tc_wgrad_ok(const ConvParams& p, int dt, const DevInfo& d)
{
    if (d.cc_major != 10) return false;
    if (p.N == 0) return true;
    TcWgradGeom g;
    return dt == DT_BF16 ? pick_wgrad_v3<__nv_bfloat16>(p, d, g) : pick_wgrad_v3<float>(p, d, g);
}

Plan plan_wgrad_tc(const ConvParams& p, int dt, const DevInfo& d)
{
    Plan pl;
    pl.algo = ALGO_TC;
    pl.block = FV_THREADS;
    if (p.N == 0) {
        pl.launches = 1;  // the reduction alone writes zeros
        pl.splits = 0;
        pl.grid = 1;
        return pl;
    }
    TcWgradGeom g;
    if (dt == DT_BF16) pick_wgrad_v3<__nv_bfloat16>(p, d, g);
    else pick_wgrad_v3<float>(p, d, g);
    pl.smem = dt == DT_BF16 ? wgrad_v3_smem<__nv_bfloat16>(g) : wgrad_v3_smem<float>(g);
    pl.splits = g.splits;
    pl.variant = g.NT * 4 + g.raws;
    pl.launches = 2;
    pl.grid = std::min(g.k_tiles * g.oc_tiles * g.splits, d.sms);
    pl.workspace = size_t(g.splits) * p.OC * g.kpad * sizeof(float);
    return pl;
}

template <typename T>
static cudaError_t wgrad_tc_t(const Plan& pl, const ConvParams& p, const void* x, const void* dy,
                              const void* y, void* dw, void* ws, int, cudaStream_t s)
{
    cudaError_t e = cudaSuccess;
    const int kpad = round_up(p.Kred, 4);
    if (pl.splits > 0) {
        const TcWgradGeom g = wgrad_v3_geom<T>(p, pl.variant / 4, pl.variant % 4, pl.splits);
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

// ---- d_input ------------------------------------------------------------------------
static TcDgradGeom dgrad_geom(const ConvParams& p, int dt, int sms)
{
    TcDgradGeom g;
    g.CIC = std::max(1, TC_M / p.KK);
    g.nkt = ceil_div(p.IC, g.CIC);
    g.cpk = std::max(1, std::min(std::max(1, sms / g.nkt), std::max(1, p.B)));
    g.rmax = (p.K + p.S - 1) / p.S;
    const int kc = dt == DT_BF16 ? TcTraits<__nv_bfloat16>::KC : TcTraits<float>::KC;
    g.nch = ceil_div(p.OC, kc);
    const int spc = std::max(1, ceil_div(p.B, g.cpk));          // samples per CTA
    const int ns_max = std::max(1, TC_M / std::max(1, p.P));
    const int tpc = ceil_div(spc, ns_max);                       // tiles per CTA
    g.NS = ceil_div(spc, tpc);
    g.NT = std::max(16, round_up(g.NS * p.P, 16));
    g.tmem_cols = pow2_at_least(g.NT);
    return g;
}

bool tc_dgrad_ok(const ConvParams& p, int dt, const DevInfo& d)
{
    if (d.cc_major != 10 || p.B <= 0 || p.KK > TC_M || p.P > TC_M) return false;
    const TcDgradGeom g = dgrad_geom(p, dt, d.sms);
    if (g.NT > TC_M) return false;
    return (dt == DT_BF16 ? tc_dgrad_smem<__nv_bfloat16>(p, g) : tc_dgrad_smem<float>(p, g)) <= d.smem_optin;
}

Plan plan_dgrad_tc(const ConvParams& p, int dt, const DevInfo& d)
{
    const TcDgradGeom g = dgrad_geom(p, dt, d.sms);
    Plan pl;
    pl.algo = ALGO_TC;
    pl.launches = 1;
    pl.block = TC_THREADS;
    pl.grid = g.nkt * g.cpk;
    pl.smem = dt == DT_BF16 ? tc_dgrad_smem<__nv_bfloat16>(p, g) : tc_dgrad_smem<float>(p, g);
    return pl;
}

template <typename T>
static cudaError_t dgrad_tc_t(const Plan& pl, const ConvParams& p, const void* dy, const void* w,
                              const void* y, void* dx, int sms, cudaStream_t s)
{
    const TcDgradGeom g = dgrad_geom(p, dt_of_tc<T>(), sms);
    cudaError_t e = cudaSuccess;
    const bool swz = tc_swizzle_mode() != 0;
#define IG_LAUNCH_DG_TC(R, Z)                                                                              \
    do {                                                                                                   \
        e = ensure_smem<dgrad_tc_kernel<T, R, Z>>(pl.smem);                                                \
        if (e == cudaSuccess)                                                                              \
            dgrad_tc_kernel<T, R, Z><<<pl.grid, pl.block, pl.smem, s>>>(p, (const T*)dy, (const T*)w,      \
                                                                        (const T*)y, (T*)dx, g);           \
    } while (0)
    if (p.relu) {
        if (swz) IG_LAUNCH_DG_TC(true, 1); else IG_LAUNCH_DG_TC(true, 0);
    } else {
        if (swz) IG_LAUNCH_DG_TC(false, 1); else IG_LAUNCH_DG_TC(false, 0);
    }
#undef IG_LAUNCH_DG_TC
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t run_dgrad_tc(const Plan& pl, const ConvParams& p, int dt, const void* dy, const void* w,
                         const void* y, void* dx, int sms, cudaStream_t s)
{
    return dt == DT_F32 ? dgrad_tc_t<float>(pl, p, dy, w, y, dx, sms, s)
                        : dgrad_tc_t<__nv_bfloat16>(pl, p, dy, w, y, dx, sms, s);
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
