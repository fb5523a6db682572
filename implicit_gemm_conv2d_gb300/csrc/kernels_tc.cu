// kernels_tc.cu -- tcgen05 tensor-core implicit-GEMM kernels (5th-generation
// tensor cores, accumulator in tensor memory), one per operation:
//
//   forward  Y[n, oc]  = sum_k X[n, k] * W[oc, k]     X[n, k] = x[col_base(n) + k_offset(k)]
//   d_input  dX[n, k]  = sum_oc G[n, oc] * W[oc, k]   then col2im into dx
//   wgrad    dW[oc, k] = sum_n G[n, oc] * X[n, k]     split over n, two-pass reduction
//
// with columns n = (b, oh, ow), k = (ic, kh, kw) and G = dy masked by y > 0 when the
// layer has a fused ReLU (implicit im2col: X and G are gathered on the fly).
//   bf16: tcgen05.mma kind::f16, bf16 operands, fp32 accumulation.
//   fp32: tcgen05.mma kind::tf32 on split operands (v = hi + lo, hi = tf32(v),
//         lo = tf32(v - hi)) summing hi*hi + hi*lo + lo*hi, which keeps about 21
//         significant bits per product: fp32-level accuracy on the tensor pipe.
// Each kernel is warp-specialized: producer warps stage raw input slabs and packed
// weight chunks with bulk asynchronous copies, formatter warps turn the raw slabs into
// MMA operands, one thread issues the MMAs, and mbarriers chain the stages.
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

__device__ __forceinline__ unsigned char* align1024(unsigned char* p)
{
    return reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// ======================================================================================
// Weight packing.  Every call of the tensor-core forward / d_input first rewrites w into
// the exact shared-memory image of the weight operand's K-chunks (rows x 128 bytes,
// 128-byte swizzled, K-major; fp32 as tf32 hi rows followed by lo rows), so that the
// main kernel fetches each chunk with one large bulk copy.
//   forward: tile (ot, kc) holds W[r][kk] = w[ot*OTp + r][kc*KC + kk], OTp rows
//   d_input: tile (kt, ch) holds A[r][kk] = w[ch*KC + kk][k0(kt) + r] (W transposed), rows
//            r < CIC*K*K of input-channel chunk kt
// ======================================================================================
template <typename T>
__global__ void pack_fwd_w_kernel(const ConvParams p, const T* __restrict__ w, unsigned char* __restrict__ out,
                                  int nchunks, int oc_tiles, int OTp)
{
    using Tr = TcTraits<T>;
    const int tile_units = OTp * 8;
    const size_t total = size_t(oc_tiles) * nchunks * tile_units;
    const size_t tb = size_t(OTp) * ROWB * (Tr::split ? 2 : 1);
    for (size_t u = blockIdx.x * size_t(blockDim.x) + threadIdx.x; u < total; u += size_t(gridDim.x) * blockDim.x) {
        const int within = int(u % tile_units);
        const size_t t = u / tile_units;
        const int kc = int(t % nchunks), ot = int(t / nchunks);
        const int r = within >> 3, c = within & 7;
        const int oc = ot * OTp + r, k = kc * Tr::KC + c * Tr::E;
        float v[8];
#pragma unroll
        for (int i = 0; i < Tr::E; ++i)
            v[i] = (oc < p.OC && k + i < p.Kred) ? Elem<T>::ldg(w + size_t(oc) * p.Kred + k + i) : 0.f;
        unsigned char* base = out + t * tb;
        put_unit<T, 1>(base, base + OTp * ROWB, r, c, v);
    }
}

template <typename T>
__global__ void pack_dgrad_w_kernel(const ConvParams p, const T* __restrict__ w, unsigned char* __restrict__ out,
                                    int nkt, int nch, int CIC)
{
    using Tr = TcTraits<T>;
    const int tile_units = TC_M * 8;
    const size_t total = size_t(nkt) * nch * tile_units;
    const size_t tb = size_t(TC_M) * ROWB * (Tr::split ? 2 : 1);
    for (size_t u = blockIdx.x * size_t(blockDim.x) + threadIdx.x; u < total; u += size_t(gridDim.x) * blockDim.x) {
        const int within = int(u % tile_units);
        const size_t t = u / tile_units;
        const int ch = int(t % nch), kt = int(t / nch);
        const int r = within >> 3, c = within & 7;
        const int k0 = kt * CIC * p.KK, mrows = min(CIC, p.IC - kt * CIC) * p.KK;
        float v[8];
#pragma unroll
        for (int i = 0; i < Tr::E; ++i) {
            const int oc = ch * Tr::KC + c * Tr::E + i;
            v[i] = (r < mrows && oc < p.OC) ? Elem<T>::ldg(w + size_t(oc) * p.Kred + k0 + r) : 0.f;
        }
        unsigned char* base = out + t * tb;
        put_unit<T, 1>(base, base + TC_M * ROWB, r, c, v);
    }
}

// ======================================================================================
// Forward: tile = (128 columns n = (b, oh, ow), OTp output channels); K = IC*K*K in
// chunks of KC.  The gathered operand X[n, k] is the MMA's A operand and lives in
// tensor memory (lane m = column n0 + m, K along the TMEM columns); the packed weights
// are the B operand (N = OTp rows; fp32: the tf32 hi rows followed by the lo rows, so
// one N = 2*OTp MMA forms X_hi*W_hi and X_hi*W_lo, and a second N = OTp MMA adds
// X_lo*W_hi into the first half).  Only the weights are read from shared memory by
// the tensor core.
// Warp roles (608 threads):
//   warp 0      x producer: per super-chunk (XG consecutive K-chunks) and per sample the
//               tile touches, one bulk copy of the contiguous channels x[b, ic_lo : ic_hi]
//               the super-chunk covers, into one of two raw slots.  Sources are rounded
//               down to 16 bytes (the slack is skipped when read); bytes of a last
//               16-byte block that lie past the end of x are copied by plain loads.
//   warp 1      w producer: per K-chunk, one bulk copy of the packed weight chunk
//               (OTp rows x 128 bytes; x2 for fp32 hi + lo) into a weight stage.
//   warp 2      MMA: one thread issues the chunk's tcgen05.mma steps, commits to the
//               weight stage's and the TMEM operand stage's "empty" barriers and, after
//               a tile's last chunk, to the accumulator barrier.
//   warps 3-18  formatters: warp w owns TMEM lanes 32*(w%4) .. +31 (one column each) and
//               a quarter of each chunk's K; gathers its column's patch values from the
//               raw slot and writes them with tcgen05.st; then the tile's epilogue
//               (TMEM -> ReLU -> y), each warp a quarter of the output channels.
// ======================================================================================
constexpr int FV_THREADS = 352;
constexpr int FV_MMA_WARP = 2;
constexpr int FV_FMT0 = 96;   // first formatter thread (warp 3)
constexpr int FV_OPS = 2;
constexpr int FV_RAWS = 2;

constexpr int FA_TM = 128;    // columns per forward tile (TMEM lanes)
constexpr int FA_KSPLIT = 4;  // formatter warps per TMEM lane quarter (each a quarter of the chunk's K)
constexpr int FA_FMTW = 4 * FA_KSPLIT;
constexpr int FA_THREADS = FV_FMT0 + 32 * FA_FMTW;
constexpr int FA_MAXW = 6;    // max weight stages
constexpr int FA_MAXA = 8;    // max TMEM operand stages
constexpr int FA_TMEM_COLS = 512;

struct FwdGeom {
    int OTp, oc_tiles;  // output-channel rows per tile (multiple of 16), tiles over OC
    int n_tiles;        // column tiles of FA_TM
    int nchunks;        // K-chunks per tile
    int xg;             // K-chunks per x super-chunk
    int nw, na;         // weight stages (shared memory), operand stages (TMEM)
    int nsmax;          // samples a tile can span
    int xs;             // bytes per sample in a raw slot
    int raw_bytes;      // one raw slot
    int w_bytes;        // one weight stage
    int dcols;          // accumulator columns (2*OTp for split fp32)
    int acol0, acols;   // first TMEM column of the operand stages, columns per stage
};

struct FwdBars {
    uint64_t raw_full[FV_RAWS], raw_empty[FV_RAWS];
    uint64_t w_full[FA_MAXW], w_empty[FA_MAXW];
    uint64_t a_full[FA_MAXA], a_empty[FA_MAXA];
    uint64_t acc_full, acc_empty;
    uint32_t tslot;
    int abort_flag;
};

template <typename T>
inline FwdGeom fwd_geom(const ConvParams& p, int xg, int nw)
{
    using Tr = TcTraits<T>;
    const int es = int(sizeof(T));
    FwdGeom g;
    const int otmax = Tr::split ? 128 : 256;
    g.oc_tiles = ceil_div(p.OC, otmax);
    g.OTp = round_up(ceil_div(p.OC, g.oc_tiles), 16);
    g.n_tiles = ceil_div(p.N, FA_TM);
    g.nchunks = round_up(p.Kred, Tr::KC) / Tr::KC;
    g.xg = xg;
    g.nw = nw;
    g.nsmax = std::min(p.B, (FA_TM - 1) / p.P + 2);
    const int chmax = std::min(p.IC, (xg * Tr::KC - 1) / p.KK + 2);
    g.xs = round_up(chmax * p.HW * es + 16, 16);
    // Sample stride = 12 words mod 32: the columns of consecutive samples fall on
    // different banks when a warp gathers one k for 32 columns.
    while ((g.xs / 4) % 32 != 12) g.xs += 16;
    g.raw_bytes = round_up(g.nsmax * g.xs, 128);
    g.w_bytes = g.OTp * ROWB * (Tr::split ? 2 : 1);
    g.dcols = g.OTp * (Tr::split ? 2 : 1);
    g.acol0 = round_up(g.dcols, 32);
    g.acols = Tr::split ? 2 * Tr::KC : Tr::KC / 2;
    g.na = std::min(FA_MAXA, (FA_TMEM_COLS - g.acol0) / g.acols);
    return g;
}

template <typename T>
inline int fwd_smem(const ConvParams& p, const FwdGeom& g)
{
    const int kred_pad = round_up(p.Kred, TcTraits<T>::KC);
    return 1024 + g.nw * g.w_bytes + FV_RAWS * g.raw_bytes + kred_pad * 4 + int(sizeof(FwdBars)) + 16;
}

template <typename T>
inline size_t fwd_packed_bytes(const FwdGeom& g)
{
    return size_t(g.oc_tiles) * g.nchunks * g.w_bytes;
}

__device__ __forceinline__ int warp_sum(int v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
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

// Bulk-copy the global byte range [src, src + bytes) (src 16-byte aligned, bytes a
// multiple of 16) to shared `dst`, except bytes at or past `end`, which are copied by
// plain loads from the calling thread (a tensor's last partial 16-byte block).  Returns
// the bytes that go through the bulk copy, for the barrier's transaction count.
__device__ __forceinline__ int slab_bytes_bulk(const unsigned char* src, int bytes, const unsigned char* end)
{
    const unsigned char* end16 = reinterpret_cast<const unsigned char*>(reinterpret_cast<uintptr_t>(end) & ~uintptr_t(15));
    if (src + bytes <= end16) return bytes;
    return end16 > src ? int(end16 - src) : 0;
}

// Position in a ring of n stages: slot i, phase parity ph of its current use, and
// whether every slot has been used once (from then on a producer waits for "empty").
struct RingPos {
    int i = 0;
    uint32_t ph = 0;
    bool wrapped = false;
    __device__ __forceinline__ void next(int n)
    {
        if (++i == n) {
            i = 0;
            ph ^= 1u;
            wrapped = true;
        }
    }
};

template <typename T, bool RELU, int SWZ>
__global__ void __launch_bounds__(FA_THREADS, 1)
fwd_tc_kernel(const ConvParams p, const T* __restrict__ x, const unsigned char* __restrict__ wpack,
              T* __restrict__ y, const FwdGeom geo)
{
    using Tr = TcTraits<T>;
    constexpr int ES = int(sizeof(T));
    constexpr int KQ = Tr::KC / FA_KSPLIT;        // K values per formatter warp and chunk
    constexpr int KQC = Tr::split ? KQ : KQ / 2;  // TMEM columns they fill (per part)
    static_assert(KQC == 8, "one tcgen05.st of 8 columns per part");
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = align1024(smem_raw);
    const int kred_pad = round_up(p.Kred, Tr::KC);
    // Layout: weight stages | raw x slots | k offsets | barriers
    unsigned char* wring = smem;
    unsigned char* raw = wring + geo.nw * geo.w_bytes;
    int* offk = reinterpret_cast<int*>(raw + FV_RAWS * geo.raw_bytes);
    FwdBars* bars = reinterpret_cast<FwdBars*>(offk + kred_pad);
    volatile int* abort_flag = &bars->abort_flag;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // offk[k]: byte offset of x[., ic, kh, kw] from channel ic_lo of k's super-chunk (0 past Kred).
    for (int k = tid; k < kred_pad; k += FA_THREADS) {
        const int sc_ic = (k / (geo.xg * Tr::KC)) * geo.xg * Tr::KC / p.KK;
        offk[k] = (k < p.Kred) ? (k_offset(p, k) - sc_ic * p.HW) * ES : 0;
    }
    if (tid == 0) {
        for (int i = 0; i < FV_RAWS; ++i) {
            mbar_init(smem_u32(&bars->raw_full[i]), 1);
            mbar_init(smem_u32(&bars->raw_empty[i]), FA_FMTW);
        }
        for (int i = 0; i < geo.nw; ++i) {
            mbar_init(smem_u32(&bars->w_full[i]), 1);
            mbar_init(smem_u32(&bars->w_empty[i]), 1);
        }
        for (int i = 0; i < geo.na; ++i) {
            mbar_init(smem_u32(&bars->a_full[i]), FA_FMTW);
            mbar_init(smem_u32(&bars->a_empty[i]), 1);
        }
        mbar_init(smem_u32(&bars->acc_full), 1);
        mbar_init(smem_u32(&bars->acc_empty), FA_FMTW);
        fence_mbar_init();
        bars->abort_flag = 0;
    }
    if (warp == 0) tmem_alloc(smem_u32(&bars->tslot), FA_TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tslot;
    const int total_tiles = geo.n_tiles * geo.oc_tiles;
    const int nsuper = (geo.nchunks + geo.xg - 1) / geo.xg;

    if (warp == 0) {
        // ---------------- x producer ----------------
        const unsigned char* xb = reinterpret_cast<const unsigned char*>(x);
        const unsigned char* x_end = xb + size_t(p.B) * p.IHW * ES;
        RingPos rp;
        for (int tile = blockIdx.x; tile < total_tiles && !*abort_flag; tile += gridDim.x) {
            const int n0 = (tile % geo.n_tiles) * FA_TM;
            const int n_end = min(n0 + FA_TM, p.N);
            const int b_first = n0 / p.P, nsamp = (n_end - 1) / p.P - b_first + 1;
            for (int sc = 0; sc < nsuper; ++sc, rp.next(FV_RAWS)) {
                const int s = rp.i;
                if (rp.wrapped && !mbar_wait_or_abort(smem_u32(&bars->raw_empty[s]), rp.ph ^ 1u, abort_flag)) {
                    report(const_cast<int*>(abort_flag), 4u);
                    break;
                }
                const int sk0 = sc * geo.xg * Tr::KC;
                const int ic_lo = sk0 / p.KK;
                const int ic_hi = min(p.IC - 1, (min(sk0 + geo.xg * Tr::KC, p.Kred) - 1) / p.KK);
                const int need = (ic_hi - ic_lo + 1) * p.HW * ES;
                unsigned char* slot = raw + s * geo.raw_bytes;
                // Sample j = lane + 32 i: its source block range and the part that goes by bulk copy.
                auto piece = [&](int j, const unsigned char*& src, int& bulk) {
                    const unsigned char* s0 = xb + (size_t(b_first + j) * p.IHW + size_t(ic_lo) * p.HW) * ES;
                    const int d = int(reinterpret_cast<uintptr_t>(s0) & 15);
                    src = s0 - d;
                    const int bytes = round_up(d + need, 16);
                    bulk = slab_bytes_bulk(src, bytes, x_end);
                    return bytes;
                };
                int tx = 0;
                for (int j = lane; j < nsamp; j += 32) {
                    const unsigned char* src;
                    int bulk;
                    const int bytes = piece(j, src, bulk);
                    // Tail past the last 16-byte boundary of x: plain loads.
                    for (const unsigned char* t = src + bulk; t < src + bytes && t < x_end; ++t)
                        slot[j * geo.xs + int(t - src)] = *t;
                    tx += bulk;
                }
                tx = warp_sum(tx);
                if (lane == 0) mbar_arrive_expect_tx(smem_u32(&bars->raw_full[s]), uint32_t(tx));
                __syncwarp();
                for (int j = lane; j < nsamp; j += 32) {
                    const unsigned char* src;
                    int bulk;
                    piece(j, src, bulk);
                    if (bulk > 0)
                        bulk_g2s(smem_u32(slot + j * geo.xs), src, uint32_t(bulk), smem_u32(&bars->raw_full[s]));
                }
            }
        }
    } else if (warp == 1) {
        // ---------------- w producer ----------------
        if (lane == 0) {
            RingPos wp;
            for (int tile = blockIdx.x; tile < total_tiles && !*abort_flag; tile += gridDim.x) {
                const int ot = tile / geo.n_tiles;
                const unsigned char* src = wpack + size_t(ot) * geo.nchunks * geo.w_bytes;
                for (int kc = 0; kc < geo.nchunks; ++kc, wp.next(geo.nw), src += geo.w_bytes) {
                    if (wp.wrapped && !mbar_wait_or_abort(smem_u32(&bars->w_empty[wp.i]), wp.ph ^ 1u, abort_flag)) {
                        report(const_cast<int*>(abort_flag), 16u);
                        break;
                    }
                    const uint32_t bar = smem_u32(&bars->w_full[wp.i]);
                    mbar_arrive_expect_tx(bar, uint32_t(geo.w_bytes));
                    bulk_g2s(smem_u32(wring + wp.i * geo.w_bytes), src, uint32_t(geo.w_bytes), bar);
                }
            }
        }
        __syncwarp();
    } else if (warp == FV_MMA_WARP) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            // fp32: N = 2*OTp over [W_hi; W_lo], then N = OTp over W_hi; bf16: N = OTp.
            const uint32_t idesc2 = instr_desc(Tr::fmt, FA_TM, geo.dcols);
            const uint32_t idesc1 = instr_desc(Tr::fmt, FA_TM, geo.OTp);
            const uint32_t w_u32 = smem_u32(wring);
            RingPos wp, ap;
            uint32_t t = 0;
            for (int tile = blockIdx.x; tile < total_tiles && !*abort_flag; tile += gridDim.x, ++t) {
                bool ok = true;
                if (t >= 1 && !mbar_wait_or_abort(smem_u32(&bars->acc_empty), (t - 1) & 1, abort_flag)) {
                    report(const_cast<int*>(abort_flag), 8u);
                    break;
                }
                tc_fence_after();
                for (int kc = 0; kc < geo.nchunks; ++kc, wp.next(geo.nw), ap.next(geo.na)) {
                    if (!mbar_wait_or_abort(smem_u32(&bars->w_full[wp.i]), wp.ph, abort_flag) ||
                        !mbar_wait_or_abort(smem_u32(&bars->a_full[ap.i]), ap.ph, abort_flag)) {
                        report(const_cast<int*>(abort_flag), 8u);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t wa = w_u32 + wp.i * geo.w_bytes;
                    const uint32_t aa = tmem + uint32_t(geo.acol0 + ap.i * geo.acols);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const uint64_t bd = op_desc<SWZ>(wa + kstep_off<SWZ>(j));
                        const uint32_t acc = (kc == 0 && j == 0) ? 0u : 1u;
                        if constexpr (Tr::split) {
                            mma_tf32_ta(tmem, aa + 8 * j, bd, idesc2, acc);           // hi * [hi; lo]
                            mma_tf32_ta(tmem, aa + Tr::KC + 8 * j, bd, idesc1, 1u);  // lo * hi
                        } else {
                            mma_f16_ta(tmem, aa + 8 * j, bd, idesc1, acc);
                        }
                    }
                    mma_commit(smem_u32(&bars->w_empty[wp.i]));
                    mma_commit(smem_u32(&bars->a_empty[ap.i]));
                }
                if (!ok) break;
                mma_commit(smem_u32(&bars->acc_full));
            }
        }
        __syncwarp();
    } else {
        // ---------------- formatters + epilogue ----------------
        const int fw = warp - 3;            // 0 .. FA_FMTW - 1
        const int qd = warp & 3;            // TMEM lane quarter this warp may access
        const int sub = fw >> 2;            // which quarter of each chunk's K
        const int m = qd * 32 + lane;       // this thread's column within the tile
        const uint32_t lane_bits = uint32_t(qd * 32) << 16;
        const uint32_t raw_u32 = smem_u32(raw), offk_u32 = smem_u32(offk) + uint32_t(sub * KQ * 4);
        const bool ragged_k = (p.Kred % Tr::KC) != 0;
        RingPos ap, rp;
        uint32_t t = 0;
        for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x, ++t) {
            const int n0 = (tile % geo.n_tiles) * FA_TM, ot = tile / geo.n_tiles;
            const int b_first = n0 / p.P;
            const int n = n0 + m;
            // Columns past N gather column N-1's values: their accumulator rows are
            // computed but never stored (rows of D depend only on rows of A).
            int boff, bmis;
            {
                uint32_t bq, pq, oh, ow;
                p.dm_P.divmod(uint32_t(min(n, p.N - 1)), bq, pq);
                p.dm_OW.divmod(pq, oh, ow);
                boff = (int(bq) - b_first) * geo.xs + (int(oh) * p.S * p.W + int(ow) * p.S) * ES;
                bmis = int((size_t(bq) * p.IHW * ES) & 15);
            }
            bool ok = true;
            uint32_t sbase = 0;
            int xc = 0;  // chunk within the super-chunk
            for (int kc = 0; kc < geo.nchunks; ++kc, ap.next(geo.na)) {
                if (xc == 0) {
                    if (!mbar_wait_or_abort(smem_u32(&bars->raw_full[rp.i]), rp.ph, abort_flag)) {
                        report(const_cast<int*>(abort_flag), 1u);
                        ok = false;
                        break;
                    }
                    const int ic_lo = (kc * Tr::KC) / p.KK;
                    const int cmis = (ic_lo * p.HW * ES) & 15;
                    sbase = raw_u32 + uint32_t(rp.i * geo.raw_bytes + boff + ((bmis + cmis) & 15));
                }
                if (ap.wrapped && !mbar_wait_or_abort(smem_u32(&bars->a_empty[ap.i]), ap.ph ^ 1u, abort_flag)) {
                    report(const_cast<int*>(abort_flag), 1u);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t oaddr = offk_u32 + uint32_t(kc * Tr::KC * 4);
                const uint32_t col = tmem + lane_bits + uint32_t(geo.acol0 + ap.i * geo.acols + sub * KQC);
                // k >= Kred exists only in a ragged last chunk: those values are zeroed.
                const int kvalid = (ragged_k && kc == geo.nchunks - 1) ? p.Kred - (kc * Tr::KC + sub * KQ) : KQ;
                int o[KQ];
#pragma unroll
                for (int i = 0; i < KQ / 4; ++i) {
                    const int4 v4 = lds128(oaddr + 16 * i);
                    o[4 * i] = v4.x;
                    o[4 * i + 1] = v4.y;
                    o[4 * i + 2] = v4.z;
                    o[4 * i + 3] = v4.w;
                }
                uint32_t v[KQ];
#pragma unroll
                for (int e = 0; e < KQ; ++e) v[e] = Tr::split ? lds32(sbase + uint32_t(o[e])) : lds16(sbase + uint32_t(o[e]));
                if (kvalid < KQ) {
#pragma unroll
                    for (int e = 0; e < KQ; ++e)
                        if (e >= kvalid) v[e] = 0;
                }
                if constexpr (Tr::split) {
                    uint32_t hi[8], lo[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        // lo is left unrounded: the MMA reads its tf32 bits (|lo| <= 2^-11 |v|).
                        const float f = __uint_as_float(v[e]);
                        const float h = to_tf32(f);
                        hi[e] = __float_as_uint(h);
                        lo[e] = __float_as_uint(f - h);
                    }
                    tmem_st8(col, hi);
                    tmem_st8(col + Tr::KC, lo);
                } else {
                    uint32_t wv[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) wv[e] = __byte_perm(v[2 * e], v[2 * e + 1], 0x5410);
                    tmem_st8(col, wv);
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                const bool sc_end = (++xc == geo.xg) || kc == geo.nchunks - 1;
                if (lane == 0) {
                    mbar_arrive(smem_u32(&bars->a_full[ap.i]));
                    if (sc_end) mbar_arrive(smem_u32(&bars->raw_empty[rp.i]));
                }
                if (sc_end) {
                    xc = 0;
                    rp.next(FV_RAWS);
                }
            }
            if (!ok) break;
            // Epilogue: TMEM -> y; this warp's lanes, every FA_KSPLIT-th group of 8 channels.
            if (!mbar_wait_or_abort(smem_u32(&bars->acc_full), t & 1, abort_flag)) {
                report(const_cast<int*>(abort_flag), 2u);
                break;
            }
            tc_fence_after();
            T* yc = nullptr;
            if (n < p.N) yc = y + col_out(p, n);
            for (int cb = sub * 8; cb < geo.OTp; cb += 8 * FA_KSPLIT) {
                uint32_t r[8];
                tmem_ld8(tmem + lane_bits + uint32_t(cb), r);
                if constexpr (Tr::split) {
                    uint32_t r2[8];
                    tmem_ld8(tmem + lane_bits + uint32_t(geo.OTp + cb), r2);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 8; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) + __uint_as_float(r2[e]));
                } else {
                    tmem_ld_wait();
                }
                if (yc) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int oc = ot * geo.OTp + cb + e;
                        if (oc < p.OC) {
                            float f = __uint_as_float(r[e]);
                            if (RELU) f = f > 0.f ? f : 0.f;
                            Elem<T>::st(yc + size_t(oc) * p.P, f);
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bars->acc_empty));
        }
    }
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, FA_TMEM_COLS);
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
    // Raw slot: [dy region][y region (ReLU)][x region]; dy / y hold the chunk's samples
    // back to back (one copy when one oc-tile spans all of OC, else one per sample with a
    // 16-byte-rounded stride gs); x holds each sample's k-tile channels at stride xsb.
    g.gs = round_up(std::min(p.OC, TC_M) * p.P * es + 16, 16);
    const int chk = std::min(p.IC, (NT - 1) / p.KK + 2);
    g.xsb = round_up(chk * p.HW * es + 16, 16);
    g.raw_bytes = round_up(g.nsc * (g.gs * (p.relu ? 2 : 1) + g.xsb) + 32, 128);
    g.op_bytes = (TC_M + NT) * ROWB * (Tr::split ? 2 : 1);
    return g;
}

template <typename T>
inline int wgrad_v3_smem(const TcWgradGeom& g)
{
    return 1024 + FV_OPS * g.op_bytes + g.raws * g.raw_bytes + g.NT * 4 + int(sizeof(WgBars)) + 16;
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
    const int gregion = geo.nsc * geo.gs + 16;              // bytes of the dy (and of the y) region
    const int xoff = gregion * (RELU ? 2 : 1);              // start of the x region in a slot
    const bool gcontig = geo.oc_tiles == 1;                 // dy / y of the chunk are one range

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int i = 0; i < geo.raws; ++i) {
            mbar_init(smem_u32(&bars->raw_full[i]), 1);
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

    if (warp == 0) {
        // ---------------- bulk-copy producer ----------------
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
                unsigned char* slot = raw + s * geo.raw_bytes;
                const int b0 = ti.s_lo + kc * geo.nsc, nb = min(geo.nsc, ti.s_hi - b0);
                // Piece i: i < ng -> dy (and y at +gregion), else x of sample i - ng.
                const int ng = gcontig ? 1 : nb;
                const int npieces = ng + nb;
                auto piece = [&](int i, int which, const unsigned char*& src, unsigned char*& dst, int& bytes,
                                 const unsigned char*& end) {
                    if (i < ng) {
                        const int j = i;
                        const size_t off = (size_t(b0 + j) * p.OCP + size_t(ti.oc0) * p.P) * ES;
                        const unsigned char* base = which == 0 ? gb : yb;
                        end = which == 0 ? g_end : y_end;
                        const int d = int(off & 15);
                        src = base + off - d;
                        bytes = round_up(d + (gcontig ? nb * p.OCP * ES : gbytes), 16);
                        dst = slot + (which == 0 ? 0 : gregion) + (gcontig ? 0 : j * geo.gs);
                    } else {
                        const int j = i - ng;
                        const size_t off = (size_t(b0 + j) * p.IHW + size_t(ti.ic_lo) * p.HW) * ES;
                        const int d = int(off & 15);
                        src = xb + off - d;
                        end = x_end;
                        bytes = round_up(d + xbytes, 16);
                        dst = slot + xoff + j * geo.xsb;
                    }
                };
                const int nw = RELU ? 2 : 1;
                int tx = 0;
                for (int i = lane; i < npieces; i += 32) {
                    for (int which = 0; which < (i < ng ? nw : 1); ++which) {
                        const unsigned char* src;
                        unsigned char* dst;
                        int bytes;
                        const unsigned char* end;
                        piece(i, which, src, dst, bytes, end);
                        const int bulk = slab_bytes_bulk(src, bytes, end);
                        for (const unsigned char* t = src + bulk; t < src + bytes && t < end; ++t) dst[int(t - src)] = *t;
                        tx += bulk;
                    }
                }
                tx = warp_sum(tx);
                if (lane == 0) mbar_arrive_expect_tx(smem_u32(&bars->raw_full[s]), uint32_t(tx));
                __syncwarp();
                for (int i = lane; i < npieces; i += 32) {
                    for (int which = 0; which < (i < ng ? nw : 1); ++which) {
                        const unsigned char* src;
                        unsigned char* dst;
                        int bytes;
                        const unsigned char* end;
                        piece(i, which, src, dst, bytes, end);
                        const int bulk = slab_bytes_bulk(src, bytes, end);
                        if (bulk > 0) bulk_g2s(smem_u32(dst), src, uint32_t(bulk), smem_u32(&bars->raw_full[s]));
                    }
                }
            }
        }
    } else if (warp == 1) {
        // idle: the producer of this kernel is warp 0 alone
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
                const int dg0 = int(((size_t(b0) * p.OCP + size_t(ti.oc0) * p.P) * ES) & 15);
#pragma unroll
                for (int e = 0; e < Tr::E; ++e) {
                    const size_t b = size_t(b0 + jj[e]);
                    // Element (j, oc row r, p) of dy is at gsrc[e] + (r * P + p) * ES; y is gregion further.
                    gsrc[e] = gcontig ? slot + dg0 + jj[e] * p.OCP * ES
                                      : slot + jj[e] * geo.gs + int(((b * p.OCP + size_t(ti.oc0) * p.P) * ES) & 15);
                    xsrc[e] = slot + xoff + jj[e] * geo.xsb + int(((b * p.IHW + size_t(ti.ic_lo) * p.HW) * ES) & 15);
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
                                            *reinterpret_cast<const __nv_bfloat16*>(sj + gregion + gi * 2));
                                        if (!(yv > 0.f)) h = 0;
                                    }
                                    wv[e >> 1] |= (e & 1) ? (h << 16) : h;
                                } else {
                                    uint32_t v = *reinterpret_cast<const uint32_t*>(sj + gi * 4);
                                    if (RELU && !(*reinterpret_cast<const float*>(sj + gregion + gi * 4) > 0.f)) v = 0;
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
// d_input:  D[k, n] = sum_oc W[oc, k] * g[oc, n]  for k in one chunk of CIC input channels
// (M = CIC*K*K <= 128 rows, chunk kt) and n the NT columns of NS whole samples, then
//   dx[b, ic, h, w] = sum over (oh, kh) with oh*S + kh = h, (ow, kw) with ow*S + kw = w of D
// in a fixed order (no atomics).  Warp roles (352 threads):
//   warp 0      g producer: per sample tile one bulk copy each of the contiguous dy and y
//               slabs of its NS samples.
//   warp 1      w producer: packed W^T tiles (kt, oc chunk), one bulk copy each, into a ring.
//   warp 2      MMA: per channel chunk kt, the oc-chunk MMAs into one of two TMEM
//               accumulators (alternating), then a commit to that accumulator's barrier.
//   warps 3-10  formatters: per sample tile, transpose and ReLU-mask the dy slab into the
//               B operand [n][oc] (128-byte swizzled, all oc chunks; reused by every
//               channel chunk); per channel chunk, TMEM -> Ds (fp32 [n][k] in shared
//               memory) and the col2im gather into dx.  While they gather chunk kt the
//               MMAs of chunk kt+1 run into the other accumulator.
// ======================================================================================
constexpr int DG_MAXA = 6;

struct TcDgradGeom {
    int NS;          // samples per tile
    int NT;          // columns per tile = round_up(NS * P, 16) <= 128
    int CIC;         // input channels per chunk
    int nkt;         // channel chunks
    int nch;         // K-chunks over OC
    int rmax;        // max (oh, kh) pairs per input row = ceil(K / S)
    int acc_cols;    // TMEM columns per accumulator (power of two >= NT)
    int na;          // weight-tile ring slots
    int a_tile;      // bytes of one packed weight tile (16 KB, 32 KB for split fp32)
    int b_chunk;     // bytes of one B chunk (hi part): NT * 128
    int b_bytes;     // all B chunks, hi (+ lo)
    int slab_bytes;  // bytes of one raw slab region (dy or y): NS samples + 16 slack, rounded
    int ntiles;      // ceil(B / NS)
    int taps;        // max (kh, kw) taps landing on one input pixel
};

struct DgBars {
    uint64_t raw_full, raw_empty, b_full, a_full[DG_MAXA], a_empty[DG_MAXA], acc_full[2], acc_empty[2];
    uint32_t tslot;
    int abort_flag;
};

template <typename T>
inline TcDgradGeom dgrad_geom_ns(const ConvParams& p, int NS, int na)
{
    using Tr = TcTraits<T>;
    const int es = int(sizeof(T));
    TcDgradGeom g;
    g.NS = NS;
    g.NT = std::max(16, round_up(NS * p.P, 16));
    g.CIC = std::max(1, TC_M / p.KK);
    g.nkt = ceil_div(p.IC, g.CIC);
    g.nch = ceil_div(p.OC, Tr::KC);
    g.rmax = (p.K + p.S - 1) / p.S;
    g.acc_cols = pow2_at_least(g.NT);
    g.na = na;
    g.a_tile = TC_M * ROWB * (Tr::split ? 2 : 1);
    g.b_chunk = g.NT * ROWB;
    g.b_bytes = g.nch * g.b_chunk * (Tr::split ? 2 : 1);
    g.slab_bytes = round_up(NS * p.OCP * es + 32, 128);
    g.ntiles = ceil_div(p.B, NS);
    auto axis_max = [](int n, int K, int S, int O) {
        int m = 0;
        for (int h = 0; h < n; ++h) {
            int c = 0;
            for (int o = 0; o < O; ++o) c += (h - o * S >= 0 && h - o * S < K);
            m = std::max(m, c);
        }
        return m;
    };
    g.taps = axis_max(p.H, p.K, p.S, p.OH) * axis_max(p.W, p.K, p.S, p.OW);
    return g;
}

constexpr int DG_DSTR = TC_M + 1;  // Ds row stride (floats): spreads the gather over banks
constexpr int DG_TMAX = 4;         // taps per input pixel handled by the fast gather
constexpr int DG_PROW = 8;         // ints per pixel row of the tap table (32 bytes, int4-aligned)

template <typename T>
inline int dgrad_smem(const ConvParams& p, const TcDgradGeom& g)
{
    return 1024 + g.na * g.a_tile + g.b_bytes + (p.relu ? 2 : 1) * g.slab_bytes + g.NT * DG_DSTR * 4 +
           (p.H + p.W) * (1 + g.rmax) * 8 + 16 + p.HW * DG_PROW * 4 + int(sizeof(DgBars)) + 16;
}

template <typename T>
inline size_t dgrad_packed_bytes(const TcDgradGeom& g)
{
    return size_t(g.nkt) * g.nch * g.a_tile;
}

template <typename T, bool RELU, int SWZ>
__global__ void __launch_bounds__(FV_THREADS, 1)
dgrad_tc_kernel(const ConvParams p, const T* __restrict__ dy, const unsigned char* __restrict__ wpack,
                const T* __restrict__ y, T* __restrict__ dx, const TcDgradGeom geo)
{
    using Tr = TcTraits<T>;
    constexpr int ES = int(sizeof(T));
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = align1024(smem_raw);
    const int NT = geo.NT;
    unsigned char* aring = smem;
    unsigned char* bt = aring + geo.na * geo.a_tile;              // B chunks (hi), then lo
    unsigned char* rdy = bt + geo.b_bytes;                         // raw dy slab
    unsigned char* ry = rdy + geo.slab_bytes;                      // raw y slab (ReLU only)
    float* Ds = reinterpret_cast<float*>(ry + (RELU ? geo.slab_bytes : 0));
    const int R1 = 1 + geo.rmax;
    int2* rtab = reinterpret_cast<int2*>(Ds + NT * DG_DSTR);
    int2* ctab = rtab + p.H * R1;
    // Per input pixel hw: its contributing (p, kh*K + kw) as Ds offsets p*DSTR + kh*K + kw,
    // then the count (only used when every pixel has <= DG_TMAX taps).
    int* ptab = reinterpret_cast<int*>((reinterpret_cast<uintptr_t>(ctab + p.W * R1) + 15) & ~uintptr_t(15));
    DgBars* bars = reinterpret_cast<DgBars*>(ptab + p.HW * DG_PROW);
    volatile int* abort_flag = &bars->abort_flag;
    const uint32_t b_lo = uint32_t(geo.nch * geo.b_chunk);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    for (int h = tid; h < p.H; h += FV_THREADS) {
        int n = 0;
        for (int oh = 0; oh < p.OH; ++oh) {
            const int kh = h - oh * p.S;
            if (kh >= 0 && kh < p.K) rtab[h * R1 + 1 + n++] = make_int2(oh * p.OW, kh * p.K);
        }
        rtab[h * R1] = make_int2(n, 0);
    }
    for (int c = tid; c < p.W; c += FV_THREADS) {
        int n = 0;
        for (int ow = 0; ow < p.OW; ++ow) {
            const int kw = c - ow * p.S;
            if (kw >= 0 && kw < p.K) ctab[c * R1 + 1 + n++] = make_int2(ow, kw);
        }
        ctab[c * R1] = make_int2(n, 0);
    }
    const bool fast_taps = geo.taps <= DG_TMAX;
    __syncthreads();  // rtab / ctab complete
    if (fast_taps) {
        for (int hw = tid; hw < p.HW; hw += FV_THREADS) {
            const int h = hw / p.W, ww = hw % p.W;
            const int2* rr = rtab + h * R1;
            const int2* cc = ctab + ww * R1;
            int n = 0;
            for (int a = 1; a <= rr[0].x; ++a)
                for (int bq = 1; bq <= cc[0].x; ++bq)
                    ptab[hw * DG_PROW + n++] = (rr[a].x + cc[bq].x) * DG_DSTR + rr[a].y + cc[bq].y;
            for (int i = n; i < DG_TMAX; ++i) ptab[hw * DG_PROW + i] = -1;
            ptab[hw * DG_PROW + DG_TMAX] = n;
        }
    }
    if (tid == 0) {
        mbar_init(smem_u32(&bars->raw_full), 1);
        mbar_init(smem_u32(&bars->raw_empty), 8);
        mbar_init(smem_u32(&bars->b_full), 8);
        for (int i = 0; i < geo.na; ++i) {
            mbar_init(smem_u32(&bars->a_full[i]), 1);
            mbar_init(smem_u32(&bars->a_empty[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&bars->acc_full[i]), 1);
            mbar_init(smem_u32(&bars->acc_empty[i]), 8);
        }
        fence_mbar_init();
        bars->abort_flag = 0;
    }
    if (warp == 0) tmem_alloc(smem_u32(&bars->tslot), 2 * geo.acc_cols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tslot;

    if (warp == 0) {
        // ---------------- g producer ----------------
        if (lane == 0) {
            const unsigned char* gb = reinterpret_cast<const unsigned char*>(dy);
            const unsigned char* yb = reinterpret_cast<const unsigned char*>(y);
            const size_t tensor_bytes = size_t(p.B) * p.OCP * ES;
            uint32_t tl = 0;
            for (int tile = blockIdx.x; tile < geo.ntiles && !*abort_flag; tile += gridDim.x, ++tl) {
                if (tl >= 1 && !mbar_wait_or_abort(smem_u32(&bars->raw_empty), (tl - 1) & 1, abort_flag)) {
                    report(const_cast<int*>(abort_flag), 4u);
                    break;
                }
                const int b0 = tile * geo.NS, ns = min(geo.NS, p.B - b0);
                const size_t off = size_t(b0) * p.OCP * ES;
                const int d = int(off & 15);
                const int bytes = round_up(d + ns * p.OCP * ES, 16);
                int tx = 0;
                const int nsl = RELU ? 2 : 1;
                int bulk[2];
                for (int i = 0; i < nsl; ++i) {
                    const unsigned char* base = i == 0 ? gb : yb;
                    unsigned char* dst = i == 0 ? rdy : ry;
                    const unsigned char* src = base + off - d;
                    bulk[i] = slab_bytes_bulk(src, bytes, base + tensor_bytes);
                    for (const unsigned char* t = src + bulk[i]; t < src + bytes && t < base + tensor_bytes; ++t)
                        dst[int(t - src)] = *t;
                    tx += bulk[i];
                }
                mbar_arrive_expect_tx(smem_u32(&bars->raw_full), uint32_t(tx));
                for (int i = 0; i < nsl; ++i)
                    if (bulk[i] > 0)
                        bulk_g2s(smem_u32(i == 0 ? rdy : ry), (i == 0 ? gb : yb) + off - d, uint32_t(bulk[i]),
                                 smem_u32(&bars->raw_full));
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------- w producer ----------------
        if (lane == 0) {
            uint32_t q = 0;
            for (int tile = blockIdx.x; tile < geo.ntiles && !*abort_flag; tile += gridDim.x) {
                bool ok = true;
                for (int kt = 0; kt < geo.nkt && ok; ++kt) {
                    for (int ch = 0; ch < geo.nch; ++ch, ++q) {
                        const int sl = q % geo.na;
                        const uint32_t use = q / geo.na;
                        if (use >= 1 && !mbar_wait_or_abort(smem_u32(&bars->a_empty[sl]), (use - 1) & 1, abort_flag)) {
                            report(const_cast<int*>(abort_flag), 16u);
                            ok = false;
                            break;
                        }
                        const uint32_t bar = smem_u32(&bars->a_full[sl]);
                        mbar_arrive_expect_tx(bar, uint32_t(geo.a_tile));
                        bulk_g2s(smem_u32(aring + sl * geo.a_tile), wpack + (size_t(kt) * geo.nch + ch) * geo.a_tile,
                                 uint32_t(geo.a_tile), bar);
                    }
                }
                if (!ok) break;
            }
        }
        __syncwarp();
    } else if (warp == FV_MMA_WARP) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            const uint32_t idesc = instr_desc(Tr::fmt, TC_M, NT);
            const uint32_t a_u32 = smem_u32(aring), b_u32 = smem_u32(bt);
            uint32_t q = 0, j = 0, tl = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < geo.ntiles && ok && !*abort_flag; tile += gridDim.x, ++tl) {
                if (!mbar_wait_or_abort(smem_u32(&bars->b_full), tl & 1, abort_flag)) {
                    report(const_cast<int*>(abort_flag), 8u);
                    break;
                }
                for (int kt = 0; kt < geo.nkt && ok; ++kt, ++j) {
                    const int buf = j & 1;
                    if ((j >> 1) >= 1 &&
                        !mbar_wait_or_abort(smem_u32(&bars->acc_empty[buf]), ((j >> 1) - 1) & 1, abort_flag)) {
                        report(const_cast<int*>(abort_flag), 8u);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t acc = tmem + uint32_t(buf * geo.acc_cols);
                    for (int ch = 0; ch < geo.nch; ++ch, ++q) {
                        const int sl = q % geo.na;
                        if (!mbar_wait_or_abort(smem_u32(&bars->a_full[sl]), (q / geo.na) & 1, abort_flag)) {
                            report(const_cast<int*>(abort_flag), 8u);
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        issue_chunk<T, SWZ>(acc, a_u32 + sl * geo.a_tile, b_u32 + ch * geo.b_chunk, TC_M * ROWB,
                                            b_lo, idesc, ch == 0);
                        mma_commit(smem_u32(&bars->a_empty[sl]));
                    }
                    if (!ok) break;
                    mma_commit(smem_u32(&bars->acc_full[buf]));
                }
            }
        }
        __syncwarp();
    } else {
        // ---------------- formatters + epilogue ----------------
        const int ft = tid - FV_FMT0;  // 0 .. 255
        const int fw = warp - 3;       // 0 .. 7
        const int units_per_row = geo.nch * (Tr::KC / Tr::E);  // 16-byte units of oc per column
        uint32_t j = 0, tl = 0;
        for (int tile = blockIdx.x; tile < geo.ntiles; tile += gridDim.x, ++tl) {
            const int b0 = tile * geo.NS, ns = min(geo.NS, p.B - b0), ncols = ns * p.P;
            if (!mbar_wait_or_abort(smem_u32(&bars->raw_full), tl & 1, abort_flag)) {
                report(const_cast<int*>(abort_flag), 1u);
                break;
            }
            // B: unit (column n, oc group og) = E consecutive oc of g[., n]; consecutive threads
            // take consecutive columns, so their dy reads are consecutive positions.
            const int d = int((size_t(b0) * p.OCP * ES) & 15);
            const unsigned char* gsl = rdy + d;
            const unsigned char* ysl = ry + d;
            for (int u = ft; u < NT * units_per_row; u += 256) {
                const int n = u % NT, og = u / NT;
                uint32_t wv[4] = {0, 0, 0, 0};
                if (n < ncols) {
                    uint32_t si, pq;
                    p.dm_P.divmod(uint32_t(n), si, pq);
                    const int base = int(si) * p.OCP + int(pq);
#pragma unroll
                    for (int e = 0; e < Tr::E; ++e) {
                        const int oc = og * Tr::E + e;
                        if (oc < p.OC) {
                            const int gi = base + oc * p.P;
                            if constexpr (ES == 2) {
                                uint32_t h = *reinterpret_cast<const unsigned short*>(gsl + gi * 2);
                                if (RELU && !(__bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(ysl + gi * 2)) > 0.f))
                                    h = 0;
                                wv[e >> 1] |= (e & 1) ? (h << 16) : h;
                            } else {
                                uint32_t v = *reinterpret_cast<const uint32_t*>(gsl + gi * 4);
                                if (RELU && !(*reinterpret_cast<const float*>(ysl + gi * 4) > 0.f)) v = 0;
                                wv[e] = v;
                            }
                        }
                    }
                }
                const int ch = (og * Tr::E) / Tr::KC, c = ((og * Tr::E) % Tr::KC) / Tr::E;
                unsigned char* dst = bt + ch * geo.b_chunk;
                put_raw_unit<T, SWZ>(dst, dst + b_lo, unit_off<SWZ>(n, c), make_uint4(wv[0], wv[1], wv[2], wv[3]));
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(smem_u32(&bars->b_full));
                mbar_arrive(smem_u32(&bars->raw_empty));  // the slab is no longer read
            }
            bool ok = true;
            for (int kt = 0; kt < geo.nkt; ++kt, ++j) {
                const int buf = j & 1;
                if (!mbar_wait_or_abort(smem_u32(&bars->acc_full[buf]), (j >> 1) & 1, abort_flag)) {
                    report(const_cast<int*>(abort_flag), 2u);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int qd = warp & 3, hcols = NT >> 1, c0 = (fw >> 2) * hcols;
                const int m = qd * 32 + lane;
                for (int cb = 0; cb < hcols; cb += 8) {
                    uint32_t r[8];
                    tmem_ld8(tmem + uint32_t(buf * geo.acc_cols) + (uint32_t(qd * 32) << 16) + uint32_t(c0 + cb), r);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 8; ++e) Ds[(c0 + cb + e) * DG_DSTR + m] = __uint_as_float(r[e]);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&bars->acc_empty[buf]));
                asm volatile("bar.sync 1, 256;" ::: "memory");
                const int ic0 = kt * geo.CIC, nic = min(geo.CIC, p.IC - ic0);
                if (fast_taps) {
                    // Thread owns pixel hw; its <= 4 tap offsets stay in registers while it
                    // walks every (sample, channel) of the chunk.
                    for (int hw = ft; hw < p.HW; hw += 256) {
                        const int4 o = *reinterpret_cast<const int4*>(ptab + hw * DG_PROW);
                        for (int sI = 0; sI < ns; ++sI) {
                            T* dxs = dx + size_t(b0 + sI) * p.IHW + size_t(ic0) * p.HW + hw;
                            const float* ds = Ds + sI * p.P * DG_DSTR;
                            for (int icl = 0; icl < nic; ++icl) {
                                const float* dk = ds + icl * p.KK;
                                float sum = 0.f;
                                if (o.x >= 0) sum += dk[o.x];
                                if (o.y >= 0) sum += dk[o.y];
                                if (o.z >= 0) sum += dk[o.z];
                                if (o.w >= 0) sum += dk[o.w];
                                Elem<T>::st(dxs + size_t(icl) * p.HW, sum);
                            }
                        }
                    }
                } else {
                    const int span = nic * p.HW;
                    for (int sI = 0; sI < ns; ++sI) {
                        T* dxs = dx + size_t(b0 + sI) * p.IHW + size_t(ic0) * p.HW;
                        const float* ds = Ds + sI * p.P * DG_DSTR;
                        for (int t = ft; t < span; t += 256) {
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
                                    sum += ds[(rr[a].x + cc[bq].x) * DG_DSTR + kb + rr[a].y + cc[bq].y];
                            Elem<T>::st(dxs + t, sum);
                        }
                    }
                }
                asm volatile("bar.sync 1, 256;" ::: "memory");  // Ds consumed
            }
            if (!ok) break;
        }
    }
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 2 * geo.acc_cols);
    }
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

// Tile width NT and x super-chunk length for the forward kernel: the feasible choice
// (shared memory, packed weights within the scratch buffer) minimising (rounds of tiles
// over the grid) x (NT + 64), where 64 stands for the per-tile cost of streaming the
// packed weights next to the NT gathered columns.
template <typename T>
static bool pick_fwd(const ConvParams& p, const DevInfo& d, FwdGeom& out)
{
    // The deepest weight ring, then the longest x super-chunk, that fits.
    static const int cfgs[][2] = {{4, 4}, {4, 2}, {3, 4}, {3, 2}, {2, 2}, {2, 1}};
    for (const auto& c : cfgs) {
        const FwdGeom g = fwd_geom<T>(p, c[1], c[0]);
        if (g.na < 2 || fwd_smem<T>(p, g) > d.smem_optin || fwd_packed_bytes<T>(g) > kScratchBytes) continue;
        out = g;
        return true;
    }
    return false;
}

bool tc_fwd_ok(const ConvParams& p, int dt, const DevInfo& d)
{
    if (d.cc_major != 10 || p.N <= 0) return false;
    FwdGeom g;
    return dt == DT_BF16 ? pick_fwd<__nv_bfloat16>(p, d, g) : pick_fwd<float>(p, d, g);
}

Plan plan_fwd_tc(const ConvParams& p, int dt, const DevInfo& d)
{
    FwdGeom g;
    if (dt == DT_BF16) pick_fwd<__nv_bfloat16>(p, d, g);
    else pick_fwd<float>(p, d, g);
    Plan pl;
    pl.algo = ALGO_TC;
    pl.launches = 2;  // weight packing, then the implicit GEMM
    pl.block = FA_THREADS;
    pl.variant = g.xg * 16 + g.nw;
    pl.grid = std::min(g.n_tiles * g.oc_tiles, d.sms);
    pl.smem = dt == DT_BF16 ? fwd_smem<__nv_bfloat16>(p, g) : fwd_smem<float>(p, g);
    return pl;
}

template <typename T>
static cudaError_t fwd_tc_t(const Plan& pl, const ConvParams& p, const void* x, const void* w, void* y,
                            cudaStream_t s)
{
    const int v = pl.variant;
    const FwdGeom g = fwd_geom<T>(p, v / 16, v % 16);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    unsigned char* wpack = static_cast<unsigned char*>(stream_scratch(dev, s));
    if (!wpack) return cudaErrorMemoryAllocation;
    const size_t units = size_t(g.oc_tiles) * g.nchunks * g.OTp * 8;
    const int pgrid = int(std::min<size_t>((units + 255) / 256, 4096));
    pack_fwd_w_kernel<T><<<pgrid, 256, 0, s>>>(p, (const T*)w, wpack, g.nchunks, g.oc_tiles, g.OTp);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // The weight operand is always in the 128-byte swizzled layout the pack kernel writes.
#define IG_LAUNCH_FWD_TC(R)                                                                         \
    do {                                                                                            \
        e = ensure_smem<fwd_tc_kernel<T, R, 1>>(pl.smem);                                           \
        if (e == cudaSuccess)                                                                       \
            fwd_tc_kernel<T, R, 1><<<pl.grid, pl.block, pl.smem, s>>>(p, (const T*)x, wpack, (T*)y, g); \
    } while (0)
    if (p.relu) IG_LAUNCH_FWD_TC(true);
    else IG_LAUNCH_FWD_TC(false);
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
// Samples per tile: about B / SMs (one tile per CTA at small batches), at most 128 / P;
// then the deepest weight ring that fits in shared memory.
template <typename T>
static bool pick_dgrad(const ConvParams& p, const DevInfo& d, TcDgradGeom& out)
{
    if (p.B <= 0 || p.KK > TC_M || p.P > TC_M) return false;
    const int ns_max = std::max(1, TC_M / p.P);
    for (int ns = std::min(ns_max, ceil_div(p.B, d.sms)); ns >= 1; --ns) {
        for (int na = 4; na >= 2; --na) {
            const TcDgradGeom g = dgrad_geom_ns<T>(p, ns, na);
            if (g.NT > TC_M || 2 * g.acc_cols > 512) continue;
            if (dgrad_smem<T>(p, g) <= d.smem_optin && dgrad_packed_bytes<T>(g) <= kScratchBytes) {
                out = g;
                return true;
            }
        }
    }
    return false;
}

bool tc_dgrad_ok(const ConvParams& p, int dt, const DevInfo& d)
{
    if (d.cc_major != 10) return false;
    TcDgradGeom g;
    return dt == DT_BF16 ? pick_dgrad<__nv_bfloat16>(p, d, g) : pick_dgrad<float>(p, d, g);
}

Plan plan_dgrad_tc(const ConvParams& p, int dt, const DevInfo& d)
{
    TcDgradGeom g;
    if (dt == DT_BF16) pick_dgrad<__nv_bfloat16>(p, d, g);
    else pick_dgrad<float>(p, d, g);
    Plan pl;
    pl.algo = ALGO_TC;
    pl.launches = 2;  // weight packing, then the implicit GEMM + col2im
    pl.block = FV_THREADS;
    pl.variant = g.NS * 8 + g.na;
    pl.grid = std::min(g.ntiles, d.sms);
    pl.smem = dt == DT_BF16 ? dgrad_smem<__nv_bfloat16>(p, g) : dgrad_smem<float>(p, g);
    return pl;
}

template <typename T>
static cudaError_t dgrad_tc_t(const Plan& pl, const ConvParams& p, const void* dy, const void* w,
                              const void* y, void* dx, int, cudaStream_t s)
{
    const TcDgradGeom g = dgrad_geom_ns<T>(p, pl.variant / 8, pl.variant % 8);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    unsigned char* wpack = static_cast<unsigned char*>(stream_scratch(dev, s));
    if (!wpack) return cudaErrorMemoryAllocation;
    const size_t units = size_t(g.nkt) * g.nch * TC_M * 8;
    const int pgrid = int(std::min<size_t>((units + 255) / 256, 4096));
    pack_dgrad_w_kernel<T><<<pgrid, 256, 0, s>>>(p, (const T*)w, wpack, g.nkt, g.nch, g.CIC);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const bool swz = tc_swizzle_mode() != 0;
#define IG_LAUNCH_DG_TC(R, Z)                                                                              \
    do {                                                                                                   \
        e = ensure_smem<dgrad_tc_kernel<T, R, Z>>(pl.smem);                                                \
        if (e == cudaSuccess)                                                                              \
            dgrad_tc_kernel<T, R, Z><<<pl.grid, pl.block, pl.smem, s>>>(p, (const T*)dy, wpack,            \
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
