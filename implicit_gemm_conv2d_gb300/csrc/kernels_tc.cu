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
//         lo = v - hi, of which the MMA reads the leading tf32 bits) summing
//         hi*hi + hi*lo + lo*hi, which keeps about 21 significant bits per product:
//         fp32-level accuracy on the tensor pipe.
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
//   d_input: tile (kt, ch) holds W^T[r][kk] = w[ch*KC + kk][k0(kt) + r] (W transposed),
//            KTp rows, r < CIC*K*K of input-channel chunk kt
// ======================================================================================
template <typename T>
__global__ void pack_fwd_w_kernel(const ConvParams p, const T* __restrict__ w, unsigned char* __restrict__ out,
                                  int nchunks, int oc_tiles, int OTp)
{
    grid_dep_launch();  // the implicit GEMM may start its prologue meanwhile
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
                                    int nkt, int nch, int CIC, int KTp)
{
    grid_dep_launch();  // the implicit GEMM may start its prologue meanwhile
    using Tr = TcTraits<T>;
    const int tile_units = KTp * 8;
    const size_t total = size_t(nkt) * nch * tile_units;
    const size_t tb = size_t(KTp) * ROWB * (Tr::split ? 2 : 1);
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
        put_unit<T, 1>(base, base + KTp * ROWB, r, c, v);
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
constexpr int FV_MMA_WARP = 2;
constexpr int FV_FMT0 = 96;   // first formatter thread (warp 3)
constexpr int FV_MAXRAWS = 4;  // max raw x slots of the forward

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
    int nraw;           // raw x slots (shared memory), one super-chunk each
    int nw, na;         // weight stages (shared memory), operand stages (TMEM)
    int nsmax;          // samples a tile can span
    int xs;             // bytes per sample in a raw slot
    int raw_bytes;      // one raw slot
    int w_bytes;        // one weight stage
    int dcols;          // accumulator columns (2*OTp for split fp32)
    int acol0, acols;   // first TMEM column of the operand stages, columns per stage
    int splits;         // K ranges (split-K when there are too few column tiles)
    int kc_per;         // K-chunks per range (a multiple of xg)
};

struct FwdBars {
    uint64_t raw_full[FV_MAXRAWS], raw_empty[FV_MAXRAWS];
    uint64_t w_full[FA_MAXW], w_empty[FA_MAXW];
    uint64_t a_full[FA_MAXA], a_empty[FA_MAXA];
    uint64_t acc_full, acc_empty;
    uint32_t tslot;
    int abort_flag;
};

template <typename T>
inline FwdGeom fwd_geom(const ConvParams& p, int xg, int nw, int nraw)
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
    g.nraw = nraw;
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
    g.splits = 1;
    g.kc_per = g.nchunks;
    return g;
}

// Estimated forward time in chunk steps of one CTA (about a microsecond each): rounds of
// work items over the SMs x chunks per item, plus, with K ranges, the reduce kernel (a launch
// and one pass over the fp32 partials).
inline double fwd_cost(int tiles, int sms, int splits, int kc, size_t part)
{
    return double(ceil_div(tiles * splits, sms)) * kc +
           (splits > 1 ? 1.5 + double(splits) * double(part) / 8e6 : 0.0);
}

// K ranges, only when the column tiles fill fewer than half the SMs (with more, a range's
// fixed cost -- its own x slabs, pipeline fill and partial sums -- outweighs the gain; layer 1
// at B = 1024, 96 tiles, ran 8 % slower in fp32 and 40 % slower in bf16 with three ranges):
// the split of the nchunks K-chunks (kc_per of them, a multiple of xg, per range) with the
// lowest estimated time, within the scratch buffer's room for partials.  Returns that estimate.
inline double fwd_set_splits(FwdGeom& g, const ConvParams& p, int sms, size_t packed, size_t scratch)
{
    const int tiles = g.n_tiles * g.oc_tiles;
    double best = fwd_cost(tiles, sms, 1, g.nchunks, 0);
    if (2 * tiles >= sms || g.nchunks < 2 * g.xg) return best;
    const size_t part = size_t(p.N) * g.oc_tiles * g.OTp * 4;  // one range's partials
    const size_t room = scratch > packed + 256 ? scratch - round_up(packed, size_t(256)) : 0;
    const int smax = int(std::min<size_t>(std::min<size_t>(room / part, size_t(g.nchunks / g.xg)), 16));
    for (int want = 2; want <= smax; ++want) {
        const int kc = round_up(ceil_div(g.nchunks, want), g.xg);
        const int splits = ceil_div(g.nchunks, kc);
        if (splits < 2) continue;
        const double c = fwd_cost(tiles, sms, splits, kc, part);
        if (c < best) {
            best = c;
            g.kc_per = kc;
            g.splits = splits;
        }
    }
    return best;
}

template <typename T>
inline int fwd_smem(const ConvParams& p, const FwdGeom& g)
{
    const int kred_pad = round_up(p.Kred, TcTraits<T>::KC);
    return 1024 + g.nw * g.w_bytes + g.nraw * g.raw_bytes + kred_pad * 4 + int(sizeof(FwdBars)) + 16;
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
              const T* __restrict__ bias, T* __restrict__ y, float* __restrict__ part, const FwdGeom geo)
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
    int* offk = reinterpret_cast<int*>(raw + geo.nraw * geo.raw_bytes);
    FwdBars* bars = reinterpret_cast<FwdBars*>(offk + kred_pad);
    volatile int* abort_flag = &bars->abort_flag;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // offk[k]: byte offset of x[., ic, kh, kw] from channel ic_lo of k's super-chunk (0 past Kred).
    for (int k = tid; k < kred_pad; k += FA_THREADS) {
        const int sc_ic = (k / (geo.xg * Tr::KC)) * geo.xg * Tr::KC / p.KK;
        offk[k] = (k < p.Kred) ? (k_offset(p, k) - sc_ic * p.HW) * ES : 0;
    }
    if (tid == 0) {
        for (int i = 0; i < geo.nraw; ++i) {
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
    // Tile = (column tile, oc tile, K range); K range sp covers chunks [sp*kc_per, ...).
    const int ctiles = geo.n_tiles * geo.oc_tiles;
    const int total_tiles = ctiles * geo.splits;
    auto krange = [&](int tile, int& lo, int& hi) {
        lo = (tile / ctiles) * geo.kc_per;
        hi = min(geo.nchunks, lo + geo.kc_per);
    };

    if (warp == 0) {
        // ---------------- x producer ----------------
        const unsigned char* xb = reinterpret_cast<const unsigned char*>(x);
        const unsigned char* x_end = xb + size_t(p.B) * p.IHW * ES;
        RingPos rp;
        for (int tile = blockIdx.x; tile < total_tiles && !*abort_flag; tile += gridDim.x) {
            const int n0 = (tile % geo.n_tiles) * FA_TM;
            const int n_end = min(n0 + FA_TM, p.N);
            const int b_first = n0 / p.P, nsamp = (n_end - 1) / p.P - b_first + 1;
            int kc_lo, kc_hi;
            krange(tile, kc_lo, kc_hi);
            for (int sc = kc_lo / geo.xg; sc < (kc_hi + geo.xg - 1) / geo.xg; ++sc, rp.next(geo.nraw)) {
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
            grid_dep_wait();  // the packed weights come from the kernel launched just before
            RingPos wp;
            for (int tile = blockIdx.x; tile < total_tiles && !*abort_flag; tile += gridDim.x) {
                const int ot = (tile / geo.n_tiles) % geo.oc_tiles;
                int kc_lo, kc_hi;
                krange(tile, kc_lo, kc_hi);
                const unsigned char* src = wpack + (size_t(ot) * geo.nchunks + kc_lo) * geo.w_bytes;
                for (int kc = kc_lo; kc < kc_hi; ++kc, wp.next(geo.nw), src += geo.w_bytes) {
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
                int kc_lo, kc_hi;
                krange(tile, kc_lo, kc_hi);
                for (int kc = kc_lo; kc < kc_hi; ++kc, wp.next(geo.nw), ap.next(geo.na)) {
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
                        const uint32_t acc = (kc == kc_lo && j == 0) ? 0u : 1u;
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
            const int n0 = (tile % geo.n_tiles) * FA_TM, ot = (tile / geo.n_tiles) % geo.oc_tiles;
            const int b_first = n0 / p.P;
            const int n = n0 + m;
            int kc_lo, kc_hi;
            krange(tile, kc_lo, kc_hi);
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
            for (int kc = kc_lo; kc < kc_hi; ++kc, ap.next(geo.na)) {
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
                const bool sc_end = (++xc == geo.xg) || kc == kc_hi - 1;
                if (lane == 0) {
                    mbar_arrive(smem_u32(&bars->a_full[ap.i]));
                    if (sc_end) mbar_arrive(smem_u32(&bars->raw_empty[rp.i]));
                }
                if (sc_end) {
                    xc = 0;
                    rp.next(geo.nraw);
                }
            }
            if (!ok) break;
            // Epilogue: TMEM -> y, plus the bias if given, then ReLU (or, with K ranges, -> this
            // range's fp32 partials, the bias and ReLU left to the reduce kernel); this
            // warp's lanes, every FA_KSPLIT-th group of 8 channels.
            if (!mbar_wait_or_abort(smem_u32(&bars->acc_full), t & 1, abort_flag)) {
                report(const_cast<int*>(abort_flag), 2u);
                break;
            }
            tc_fence_after();
            T* yc = nullptr;
            float* pc = nullptr;
            if (n < p.N) {
                if (geo.splits == 1) yc = y + col_out(p, n);
                else pc = part + (size_t(tile / ctiles) * p.N + n) * (geo.oc_tiles * geo.OTp) + ot * geo.OTp;
            }
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
                            if (bias) f += Elem<T>::ldg(bias + oc);
                            if (RELU) f = f > 0.f ? f : 0.f;
                            Elem<T>::st(yc + size_t(oc) * p.P, f);
                        }
                    }
                } else if (pc) {
                    *reinterpret_cast<float4*>(pc + cb) = make_float4(__uint_as_float(r[0]), __uint_as_float(r[1]),
                                                                      __uint_as_float(r[2]), __uint_as_float(r[3]));
                    *reinterpret_cast<float4*>(pc + cb + 4) = make_float4(
                        __uint_as_float(r[4]), __uint_as_float(r[5]), __uint_as_float(r[6]), __uint_as_float(r[7]));
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

// Sum of the forward's K-range partials in ascending range order, then the bias (if any) and
// ReLU, into y.
template <typename T, bool RELU>
__global__ void fwd_reduce_kernel(const ConvParams p, const float* __restrict__ part, int splits, int ocp,
                                  const T* __restrict__ bias, T* __restrict__ y)
{
    grid_dep_wait();  // the partials come from the kernel launched just before
    const size_t total = size_t(p.N) * p.OC;
    const size_t sstride = size_t(p.N) * ocp;
    for (size_t i = blockIdx.x * size_t(blockDim.x) + threadIdx.x; i < total; i += size_t(gridDim.x) * blockDim.x) {
        const int n = int(i / p.OC), oc = int(i % p.OC);
        const float* src = part + size_t(n) * ocp + oc;
        float s = 0.f;
        for (int sp = 0; sp < splits; ++sp) s += __ldcg(src + size_t(sp) * sstride);
        if (bias) s += Elem<T>::ldg(bias + oc);
        if (RELU) s = s > 0.f ? s : 0.f;
        Elem<T>::st(y + col_out(p, n) + size_t(oc) * p.P, s);
    }
}

// ======================================================================================
// wgrad partials: tile = (128 output channels, KTp reduction indices k, one split range of
// samples); the GEMM's K runs over the split's columns n = (b, oh, ow), a chunk being NSC
// whole samples (NSC*P columns, zero-padded to the MMA step):
//   D[oc, k] = sum_{n in split} G[n, oc] * X[n, k]
// G (dy masked by y > 0) is the MMA's A operand in tensor memory (lane = output channel,
// K = n along the columns); X (the patches) is the shared-memory B operand (N = KTp rows
// of k, K-major along n; fp32 as tf32 hi rows then lo rows, so one N = 2*KTp MMA forms
// G_hi*X_hi and G_hi*X_lo and an N = KTp MMA adds G_lo*X_hi).
// Warp roles (608 threads):
//   warps 0, 1  bulk-copy producers (lane 0 each): per chunk, the contiguous slab
//               dy[b0 : b0+nb] (and y, the ReLU mask source) by warp 0, and x[b, ic_lo :
//               ic_hi] (the k-tile's input channels) of each sample by warp 1, into a raw slot.
//   warp 2      MMA.
//   G warps     (the first 8 formatter warps for fp32, 4 for bf16) lane = output channel;
//               the chunk's columns, masked and split, into a TMEM operand stage with
//               tcgen05.st.
//   X warps     (the other formatter warps) 16-byte units (row k, 4 or 8 columns) of the
//               B stage.
//   warps 3-18  epilogue: the fp32 tile to ws[split][oc][k] (row stride kpad).
// ======================================================================================
constexpr int WG_THREADS = FV_FMT0 + 32 * 16;
constexpr int WG_MAXA = 8, WG_MAXB = 4, WG_MAXR = 5;
// Formatter roles: G warps (a multiple of 4, one or more per TMEM lane quarter) and X
// warps; the column groups of 8 words one G thread writes; the B-stage rows one X thread
// builds (its k offsets stay in registers).  fp32 splits the warps evenly (G and X are
// both 128 rows); bf16 gives X three quarters (its KTp is up to 256 rows).
template <typename T> struct WgRoles {
    static constexpr int g_warps = TcTraits<T>::split ? 8 : 4;
    static constexpr int g_groups = TcTraits<T>::split ? 2 : 4;
    static constexpr int x_rows = TcTraits<T>::split ? 4 : 6;
};

struct TcWgradGeom {
    int KTp;       // k rows per tile (multiple of 32): <= 128 (fp32), <= 256 (bf16)
    int k_tiles;   // ceil(Kred / KTp)
    int oc_tiles;  // ceil(OC / 128)
    int splits;    // sample ranges
    int kpad;      // workspace row stride (Kred rounded up to 4)
    int nsc;       // samples per chunk
    int cnp;       // columns per chunk, padded to the MMA K-step
    int raws;      // raw slots
    int gs;        // bytes per sample of a dy (or y) slab in a raw slot
    int xsb;       // bytes per sample of the x channels in a raw slot
    int raw_bytes;
    int b_bytes;   // one B stage: KTp rows x 128 bytes (x2 for split fp32)
    int nbs;       // B stages
    int dcols;     // accumulator columns
    int acols, na; // TMEM columns per A stage, A stages
};

struct WgBars {
    uint64_t raw_full[WG_MAXR], raw_empty[WG_MAXR], a_full[WG_MAXA], a_empty[WG_MAXA];
    uint64_t b_full[WG_MAXB], b_empty[WG_MAXB], acc_full, acc_empty;
    uint32_t tslot;
    int abort_flag;
};

// Samples per chunk: as many whole samples as fit in one 128-byte operand row, reduced
// while that keeps nsc*P a multiple of the MMA K-step (no zero padding), else padded.
inline int wgrad_nsc(int P, int KC, int ks)
{
    const int top = std::max(1, KC / P);
    for (int m = top; m >= 1; --m)
        if ((m * P) % ks == 0) return m;
    return top;
}

template <typename T>
inline TcWgradGeom wgrad_geom(const ConvParams& p, int KTp, int raws, int nbs, int splits)
{
    using Tr = TcTraits<T>;
    const int es = int(sizeof(T));
    const int ks = Tr::KC / 4;  // columns per MMA K-step
    TcWgradGeom g;
    g.KTp = KTp;
    g.k_tiles = ceil_div(p.Kred, KTp);
    g.oc_tiles = ceil_div(p.OC, TC_M);
    g.splits = splits;
    g.kpad = round_up(p.Kred, 4);
    g.nsc = wgrad_nsc(p.P, Tr::KC, ks);
    g.cnp = round_up(g.nsc * p.P, ks);
    g.raws = raws;
    // Raw slot: [dy region][y region (ReLU)][x region]; dy / y hold the chunk's samples
    // back to back (one copy when one oc-tile spans all of OC, else one per sample with a
    // 16-byte-rounded stride gs); x holds each sample's k-tile channels at stride xsb.
    g.gs = round_up(std::min(p.OC, TC_M) * p.P * es + 16, 16);
    const int chk = std::min(p.IC, (KTp - 1) / p.KK + 2);
    g.xsb = round_up(chk * p.HW * es + 16, 16);
    g.raw_bytes = round_up(g.nsc * (g.gs * (p.relu ? 2 : 1) + g.xsb) + 32, 128);
    g.b_bytes = KTp * ROWB * (Tr::split ? 2 : 1);
    g.nbs = nbs;
    g.dcols = KTp * (Tr::split ? 2 : 1);
    g.acols = Tr::split ? 2 * Tr::KC : Tr::KC / 2;
    g.na = std::min(WG_MAXA, (512 - round_up(g.dcols, 32)) / g.acols);
    return g;
}

template <typename T>
inline int wgrad_smem(const TcWgradGeom& g)
{
    return 1024 + g.nbs * g.b_bytes + g.raws * g.raw_bytes + int(sizeof(WgBars)) + 8 * g.cnp + 16;
}

template <typename T, bool RELU>
__global__ void __launch_bounds__(WG_THREADS, 1)
wgrad_tc_kernel(const ConvParams p, const T* __restrict__ x, const T* __restrict__ dy,
                const T* __restrict__ y, float* __restrict__ ws, const TcWgradGeom geo)
{
    using Tr = TcTraits<T>;
    constexpr int ES = int(sizeof(T));
    constexpr int KS = Tr::KC / 4;  // columns per MMA K-step
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = align1024(smem_raw);
    const int KTp = geo.KTp;
    unsigned char* bring = smem;
    unsigned char* raw = bring + geo.nbs * geo.b_bytes;
    WgBars* bars = reinterpret_cast<WgBars*>(raw + geo.raws * geo.raw_bytes);
    // Column table of a chunk: column n -> (sample j, byte offset of (j, pq) in the dy
    // region from channel row 0); padding columns get a sample no chunk has.
    int* gtab = reinterpret_cast<int*>(bars + 1);
    volatile int* abort_flag = &bars->abort_flag;
    const int gregion = geo.nsc * geo.gs + 16;              // bytes of the dy (and of the y) region
    const int xoff = gregion * (RELU ? 2 : 1);              // start of the x region in a slot
    const int acol0 = round_up(geo.dcols, 32);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    for (int n = tid; n < geo.cnp; n += WG_THREADS) {
        const int j = n / p.P, pq = n % p.P;
        gtab[2 * n] = n < geo.nsc * p.P ? j : 1 << 20;
        gtab[2 * n + 1] = (j * p.OCP + pq) * ES;
    }
    if (tid == 0) {
        for (int i = 0; i < geo.raws; ++i) {
            mbar_init(smem_u32(&bars->raw_full[i]), 2);  // the two producers' arrivals
            mbar_init(smem_u32(&bars->raw_empty[i]), 16);
        }
        for (int i = 0; i < geo.na; ++i) {
            mbar_init(smem_u32(&bars->a_full[i]), WgRoles<T>::g_warps);
            mbar_init(smem_u32(&bars->a_empty[i]), 1);
        }
        for (int i = 0; i < geo.nbs; ++i) {
            mbar_init(smem_u32(&bars->b_full[i]), 16 - WgRoles<T>::g_warps);
            mbar_init(smem_u32(&bars->b_empty[i]), 1);
        }
        mbar_init(smem_u32(&bars->acc_full), 1);
        mbar_init(smem_u32(&bars->acc_empty), 16);
        fence_mbar_init();
        bars->abort_flag = 0;
    }
    if (warp == 0) tmem_alloc(smem_u32(&bars->tslot), 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tslot;
    const int per_split = geo.k_tiles * geo.oc_tiles;
    const int total = per_split * geo.splits;

    // Tile decode shared by all roles.
    // The k-tiles of one split read the same dy / y chunks: each starts at a different
    // chunk (a fixed rotation, so the summation order is fixed) so that they do not all
    // request the same lines at once.
    struct TileInfo {
        int split, k0, oc0, rows, s_lo, s_hi, nchunks, ic_lo, ic_hi, rot;
        __device__ int chunk(int kc) const { return kc + rot < nchunks ? kc + rot : kc + rot - nchunks; }
    };
    auto decode = [&](int tile) {
        TileInfo ti;
        ti.split = tile / per_split;
        const int rem = tile % per_split;
        ti.k0 = (rem % geo.k_tiles) * KTp;
        ti.oc0 = (rem / geo.k_tiles) * TC_M;
        ti.rows = min(TC_M, p.OC - ti.oc0);
        ti.s_lo = int((long long)p.B * ti.split / geo.splits);
        ti.s_hi = int((long long)p.B * (ti.split + 1) / geo.splits);
        ti.nchunks = (ti.s_hi - ti.s_lo + geo.nsc - 1) / geo.nsc;
        ti.ic_lo = ti.k0 / p.KK;
        ti.ic_hi = min(p.IC - 1, (min(ti.k0 + KTp, p.Kred) - 1) / p.KK);
        ti.rot = (rem % geo.k_tiles) * ti.nchunks / geo.k_tiles;
        return ti;
    };

    if (warp <= 1) {
        // ---------------- bulk-copy producers ----------------
        // Lane 0 of warp 0 copies dy[b0 : b0+nb] (all channels, contiguous) and y; lane 0
        // of warp 1 copies x[b, ic_lo : ic_hi] of each sample: two threads on two SM
        // sub-partitions, each arriving once (with its transaction bytes) on the slot's
        // barrier.  Sources are rounded down to 16 bytes (the slack is skipped when read);
        // bytes of a last 16-byte block past the end of a tensor are copied by plain loads
        // before the arrival that releases them.
        if (lane == 0) {
            const bool gside = warp == 0;
            const unsigned char* xb = reinterpret_cast<const unsigned char*>(x);
            const unsigned char* gb = reinterpret_cast<const unsigned char*>(dy);
            const unsigned char* yb = reinterpret_cast<const unsigned char*>(y);
            const unsigned char* x_end = xb + size_t(p.B) * p.IHW * ES;
            const unsigned char* g_end = gb + size_t(p.B) * p.OCP * ES;
            const unsigned char* y_end = yb + size_t(p.B) * p.OCP * ES;
            const size_t xstride = size_t(p.IHW) * ES, gstride = size_t(p.OCP) * ES;
            auto tail = [&](unsigned char* dstp, const unsigned char* src, int bytes, const unsigned char* end) -> int {
                const int bulk = slab_bytes_bulk(src, bytes, end);
                for (const unsigned char* t = src + bulk; t < src + bytes && t < end; ++t) dstp[int(t - src)] = *t;
                return bulk;
            };
            RingPos rp;
            for (int tile = blockIdx.x; tile < total && !*abort_flag; tile += gridDim.x) {
                const TileInfo ti = decode(tile);
                const int xbytes = (ti.ic_hi - ti.ic_lo + 1) * p.HW * ES;
                for (int kc = 0; kc < ti.nchunks; ++kc, rp.next(geo.raws)) {
                    const int s = rp.i;
                    if (rp.wrapped && !mbar_wait_or_abort(smem_u32(&bars->raw_empty[s]), rp.ph ^ 1u, abort_flag)) {
                        report(const_cast<int*>(abort_flag), 4u);
                        break;
                    }
                    unsigned char* slot = raw + s * geo.raw_bytes;
                    const uint32_t slot_u32 = smem_u32(slot), bar = smem_u32(&bars->raw_full[s]);
                    const int b0 = ti.s_lo + ti.chunk(kc) * geo.nsc, nb = min(geo.nsc, ti.s_hi - b0);
                    if (gside) {
                        const size_t goff = size_t(b0) * gstride;
                        const int gd = int(goff & 15);
                        const int gbytes = round_up(gd + nb * int(gstride), 16);
                        const bool at_end = b0 + nb == p.B;  // only then can a copy reach dy's end
                        const int gbulk = at_end ? tail(slot, gb + goff - gd, gbytes, g_end) : gbytes;
                        if (RELU && at_end) tail(slot + gregion, yb + goff - gd, gbytes, y_end);
                        mbar_arrive_expect_tx(bar, uint32_t(gbulk * (RELU ? 2 : 1)));
                        if (gbulk > 0) {
                            bulk_g2s(slot_u32, gb + goff - gd, uint32_t(gbulk), bar);
                            if (RELU) bulk_g2s(slot_u32 + gregion, yb + goff - gd, uint32_t(gbulk), bar);
                        }
                    } else {
                        const unsigned char* xs = xb + size_t(b0) * xstride + size_t(ti.ic_lo) * p.HW * ES;
                        const bool at_end = b0 + nb == p.B;  // only then can a copy reach x's end
                        int tx = 0;
                        for (int j = 0; j < nb; ++j) {
                            const int xd = int(reinterpret_cast<uintptr_t>(xs + size_t(j) * xstride) & 15);
                            const int bytes = round_up(xd + xbytes, 16);
                            tx += at_end ? tail(slot + xoff + j * geo.xsb, xs + size_t(j) * xstride - xd, bytes, x_end)
                                         : bytes;
                        }
                        mbar_arrive_expect_tx(bar, uint32_t(tx));
                        for (int j = 0; j < nb; ++j) {
                            const unsigned char* src = xs + size_t(j) * xstride;
                            const int xd = int(reinterpret_cast<uintptr_t>(src) & 15);
                            const int bytes = round_up(xd + xbytes, 16);
                            const int xbulk = at_end ? slab_bytes_bulk(src - xd, bytes, x_end) : bytes;
                            if (xbulk > 0)
                                bulk_g2s(slot_u32 + uint32_t(xoff + j * geo.xsb), src - xd, uint32_t(xbulk), bar);
                        }
                    }
                }
            }
        }
        __syncwarp();
    } else if (warp == FV_MMA_WARP) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            const uint32_t idesc2 = instr_desc(Tr::fmt, TC_M, geo.dcols);
            const uint32_t idesc1 = instr_desc(Tr::fmt, TC_M, KTp);
            const uint32_t b_u32 = smem_u32(bring);
            const int ksteps = geo.cnp / KS;
            RingPos ap, bp;
            uint32_t t = 0;
            for (int tile = blockIdx.x; tile < total && !*abort_flag; tile += gridDim.x, ++t) {
                const TileInfo ti = decode(tile);
                bool ok = true;
                if (t >= 1 && !mbar_wait_or_abort(smem_u32(&bars->acc_empty), (t - 1) & 1, abort_flag)) {
                    report(const_cast<int*>(abort_flag), 8u);
                    break;
                }
                tc_fence_after();
                for (int kc = 0; kc < ti.nchunks; ++kc, ap.next(geo.na), bp.next(geo.nbs)) {
                    if (!mbar_wait_or_abort(smem_u32(&bars->a_full[ap.i]), ap.ph, abort_flag) ||
                        !mbar_wait_or_abort(smem_u32(&bars->b_full[bp.i]), bp.ph, abort_flag)) {
                        report(const_cast<int*>(abort_flag), 8u);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t ba = b_u32 + bp.i * geo.b_bytes;
                    const uint32_t aa = tmem + uint32_t(acol0 + ap.i * geo.acols);
                    for (int j = 0; j < ksteps; ++j) {
                        const uint64_t bd = op_desc<1>(ba + kstep_off<1>(j));
                        const uint32_t acc = (kc == 0 && j == 0) ? 0u : 1u;
                        if constexpr (Tr::split) {
                            mma_tf32_ta(tmem, aa + 8 * j, bd, idesc2, acc);           // hi * [hi; lo]
                            mma_tf32_ta(tmem, aa + Tr::KC + 8 * j, bd, idesc1, 1u);  // lo * hi
                        } else {
                            mma_f16_ta(tmem, aa + 8 * j, bd, idesc1, acc);
                        }
                    }
                    mma_commit(smem_u32(&bars->a_empty[ap.i]));
                    mma_commit(smem_u32(&bars->b_empty[bp.i]));
                }
                if (!ok) break;
                mma_commit(smem_u32(&bars->acc_full));
            }
        }
        __syncwarp();
    } else if (warp >= 3) {
        const int fw = warp - 3;            // 0 .. 15
        const int qd = warp & 3;            // TMEM lane quarter
        const uint32_t lane_bits = uint32_t(qd * 32) << 16;
        constexpr int NGW = WgRoles<T>::g_warps;
        const int m = qd * 32 + lane;       // output channel within the tile (G, epilogue)
        // Epilogue of tile t: D[oc][k] -> ws; this warp's lanes, a quarter of the k columns.
        auto epilogue = [&](const TileInfo& ti, uint32_t t) -> bool {
            if (!mbar_wait_or_abort(smem_u32(&bars->acc_full), t & 1, abort_flag)) {
                report(const_cast<int*>(abort_flag), 2u);
                return false;
            }
            tc_fence_after();
            const int oc = ti.oc0 + m;
            const int kq = KTp / 4, c0 = (fw >> 2) * kq;
            for (int cb = c0; cb < c0 + kq; cb += 8) {
                uint32_t r[8];
                tmem_ld8(tmem + lane_bits + uint32_t(cb), r);
                if constexpr (Tr::split) {
                    uint32_t r2[8];
                    tmem_ld8(tmem + lane_bits + uint32_t(KTp + cb), r2);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 8; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) + __uint_as_float(r2[e]));
                } else {
                    tmem_ld_wait();
                }
                const int k = ti.k0 + cb;
                if (oc < p.OC && m < ti.rows && k < geo.kpad) {
                    float* dst = ws + (size_t(ti.split) * p.OC + oc) * geo.kpad + k;
                    *reinterpret_cast<float4*>(dst) = make_float4(__uint_as_float(r[0]), __uint_as_float(r[1]),
                                                                  __uint_as_float(r[2]), __uint_as_float(r[3]));
                    if (k + 4 < geo.kpad)
                        *reinterpret_cast<float4*>(dst + 4) = make_float4(
                            __uint_as_float(r[4]), __uint_as_float(r[5]), __uint_as_float(r[6]), __uint_as_float(r[7]));
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bars->acc_empty));
            return true;
        };
        if (fw < NGW) {
            // ---------------- G formatters ----------------
            const int gsub = fw >> 2;           // which of the NGW/4 warps of its lane quarter
            constexpr int NG = ES == 4 ? 8 : 16;       // columns per tcgen05.st of 8 words
            constexpr int MAXG = WgRoles<T>::g_groups;  // column groups per thread
            const int ngroups = geo.cnp / NG;
            // Fast path: P a multiple of 4 -> runs of 4 positions of one
            // sample are one vector load; per group of NG columns the byte offsets (from the
            // thread's channel row) and samples of its NG/4 vectors never change.
            const bool gfast = p.P % 4 == 0;
            int goff[MAXG][NG / 4], gsj[MAXG][NG / 4];
#pragma unroll
            for (int gi = 0; gi < MAXG; ++gi)
#pragma unroll
                for (int vi = 0; vi < NG / 4; ++vi) {
                    const int n = (gsub + gi * (NGW / 4)) * NG + vi * 4;
                    uint32_t j, pq;
                    p.dm_P.divmod(uint32_t(n), j, pq);
                    goff[gi][vi] = (int(j) * p.OCP + int(pq)) * ES;
                    gsj[gi][vi] = n < geo.nsc * p.P ? int(j) : 1 << 20;  // padding: never a real sample
                }
            RingPos rp, ap;
            uint32_t t = 0;
            for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++t) {
                const TileInfo ti = decode(tile);
                bool ok = true;
                for (int kc = 0; kc < ti.nchunks; ++kc, rp.next(geo.raws)) {
                    if (!mbar_wait_or_abort(smem_u32(&bars->raw_full[rp.i]), rp.ph, abort_flag)) {
                        report(const_cast<int*>(abort_flag), 1u);
                        ok = false;
                        break;
                    }
                    const int b0 = ti.s_lo + ti.chunk(kc) * geo.nsc;
                    const int nb = min(geo.nsc, ti.s_hi - b0);
                    const uint32_t slot = smem_u32(raw + rp.i * geo.raw_bytes);
                    if (ap.wrapped && !mbar_wait_or_abort(smem_u32(&bars->a_empty[ap.i]), ap.ph ^ 1u, abort_flag)) {
                        report(const_cast<int*>(abort_flag), 1u);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // Element (sample j, channel m, position pq) of the dy region; y is gregion further.
                    const int dg0 = int(((size_t(b0) * p.OCP + size_t(ti.oc0) * p.P) * ES) & 15);
                    const bool live = m < ti.rows;
                    const uint32_t col = tmem + lane_bits + uint32_t(acol0 + ap.i * geo.acols);
                    const uint32_t gbase = slot + uint32_t(dg0 + m * p.P * ES);
                    const uint32_t gtab_u32 = smem_u32(gtab);
#pragma unroll
                    for (int gi = 0; gi < MAXG; ++gi) {
                        const int g = gsub + gi * (NGW / 4);
                        if (g >= ngroups) break;
                        uint32_t v[NG];
                        if (gfast) {
                            uint32_t d[NG], w[NG];
#pragma unroll
                            for (int vi = 0; vi < NG / 4; ++vi) {
                                // Only real rows and samples are read (the rest of the
                                // region may lie past the slot).
                                const uint32_t a = gbase + uint32_t(goff[gi][vi]);
                                d[4 * vi] = d[4 * vi + 1] = d[4 * vi + 2] = d[4 * vi + 3] = 0u;
                                w[4 * vi] = w[4 * vi + 1] = w[4 * vi + 2] = w[4 * vi + 3] = 0u;
                                if (!live || gsj[gi][vi] >= nb) continue;
                                if constexpr (ES == 4) {
                                    const int4 q = lds128(a);
                                    d[4 * vi] = q.x; d[4 * vi + 1] = q.y; d[4 * vi + 2] = q.z; d[4 * vi + 3] = q.w;
                                    if (RELU) {
                                        const int4 r = lds128(a + gregion);
                                        w[4 * vi] = r.x; w[4 * vi + 1] = r.y; w[4 * vi + 2] = r.z; w[4 * vi + 3] = r.w;
                                    }
                                } else {
                                    const uint2 q = lds64(a);
                                    d[4 * vi] = q.x & 0xFFFFu; d[4 * vi + 1] = q.x >> 16;
                                    d[4 * vi + 2] = q.y & 0xFFFFu; d[4 * vi + 3] = q.y >> 16;
                                    if (RELU) {
                                        const uint2 r = lds64(a + gregion);
                                        w[4 * vi] = r.x << 16; w[4 * vi + 1] = r.x & 0xFFFF0000u;
                                        w[4 * vi + 2] = r.y << 16; w[4 * vi + 3] = r.y & 0xFFFF0000u;
                                    }
                                }
                            }
#pragma unroll
                            for (int e = 0; e < NG; ++e) {
                                // mask words are fp32 patterns (bf16 y in the high half)
                                const bool keep = live && gsj[gi][e / 4] < nb && (!RELU || __uint_as_float(w[e]) > 0.f);
                                v[e] = keep ? d[e] : 0u;
                            }
                        } else {
                            // Element by element through the column table (sample, byte offset).
#pragma unroll
                            for (int e = 0; e < NG; ++e) {
                                const int n = g * NG + e;
                                const int j = int(lds32(gtab_u32 + 8 * n)), off = int(lds32(gtab_u32 + 8 * n + 4));
                                uint32_t d = 0u;
                                if (live && j < nb) {
                                    const uint32_t a = gbase + uint32_t(off);
                                    if constexpr (ES == 4) {
                                        d = lds32(a);
                                        if (RELU && !(__uint_as_float(lds32(a + gregion)) > 0.f)) d = 0u;
                                    } else {
                                        d = lds16(a);
                                        if (RELU && !(__uint_as_float(lds16(a + gregion) << 16) > 0.f)) d = 0u;
                                    }
                                }
                                v[e] = d;
                            }
                        }
                        if constexpr (Tr::split) {
                            uint32_t hi[8], lo[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                const float f = __uint_as_float(v[e]);
                                const float h = to_tf32(f);
                                hi[e] = __float_as_uint(h);
                                lo[e] = __float_as_uint(f - h);
                            }
                            tmem_st8(col + uint32_t(g * NG), hi);
                            tmem_st8(col + uint32_t(Tr::KC + g * NG), lo);
                        } else {
                            uint32_t wv[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e) wv[e] = __byte_perm(v[2 * e], v[2 * e + 1], 0x5410);
                            tmem_st8(col + uint32_t(g * NG / 2), wv);
                        }
                    }
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(smem_u32(&bars->a_full[ap.i]));
                        mbar_arrive(smem_u32(&bars->raw_empty[rp.i]));
                    }
                    ap.next(geo.na);
                }
                if (!ok || !epilogue(ti, t)) break;
            }
        } else {
            // ---------------- X formatters ----------------
            // 16-byte unit column c (E columns) of rows rbase + i*rstep.
            const int xthreads = 32 * (16 - NGW);
            const int xt = tid - FV_FMT0 - 32 * NGW;
            const int upr = geo.cnp / Tr::E;     // units per row
            const int cfix = xt % upr;
            const int rbase = xt / upr;
            const int rstep = xthreads / upr;
            const bool xact = xt < rstep * upr;
            constexpr int XMAXR = WgRoles<T>::x_rows;  // rows per thread (checked by the planner)
            int po[Tr::E], jj[Tr::E];            // column offset and sample of this thread's columns
#pragma unroll
            for (int e = 0; e < Tr::E; ++e) {
                const int n = cfix * Tr::E + e;
                uint32_t j, r, oh, ow;
                p.dm_P.divmod(uint32_t(n), j, r);
                p.dm_OW.divmod(r, oh, ow);
                jj[e] = n < geo.nsc * p.P ? int(j) : 1 << 20;  // padding columns: never a real sample
                po[e] = (int(oh) * p.S * p.W + int(ow) * p.S) * ES;
            }
            uint32_t uo[XMAXR];                  // unit offsets of this thread's rows in a B stage
#pragma unroll
            for (int i = 0; i < XMAXR; ++i) uo[i] = unit_off<1>(rbase + i * rstep, cfix);
            RingPos rp, bp;
            uint32_t t = 0;
            for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++t) {
                const TileInfo ti = decode(tile);
                // Byte offsets of this thread's rows k = k0 + rbase + i*rstep (-1: past Kred).
                int ko[XMAXR];
#pragma unroll
                for (int i = 0; i < XMAXR; ++i) {
                    const int r = rbase + i * rstep;
                    const int k = ti.k0 + r;
                    ko[i] = (xact && r < KTp && k < p.Kred) ? (k_offset(p, k) - ti.ic_lo * p.HW) * ES : -1;
                }
                bool ok = true;
                for (int kc = 0; kc < ti.nchunks; ++kc, rp.next(geo.raws)) {
                    if (!mbar_wait_or_abort(smem_u32(&bars->raw_full[rp.i]), rp.ph, abort_flag)) {
                        report(const_cast<int*>(abort_flag), 1u);
                        ok = false;
                        break;
                    }
                    const int b0 = ti.s_lo + ti.chunk(kc) * geo.nsc;
                    const int nb = min(geo.nsc, ti.s_hi - b0);
                    const uint32_t slot = smem_u32(raw + rp.i * geo.raw_bytes);
                    if (bp.wrapped && !mbar_wait_or_abort(smem_u32(&bars->b_empty[bp.i]), bp.ph ^ 1u, abort_flag)) {
                        report(const_cast<int*>(abort_flag), 1u);
                        ok = false;
                        break;
                    }
                    unsigned char* op = bring + bp.i * geo.b_bytes;
                    if (xact) {
                        // Sample bases of this thread's columns in the x region (with the slack
                        // of each sample's 16-byte-rounded copy).
                        uint32_t xs[Tr::E];
#pragma unroll
                        for (int e = 0; e < Tr::E; ++e) {
                            const int j = min(jj[e], geo.nsc - 1);
                            const size_t b = size_t(b0 + j);
                            xs[e] = slot + uint32_t(xoff + j * geo.xsb +
                                                    int(((b * p.IHW + size_t(ti.ic_lo) * p.HW) * ES) & 15) + po[e]);
                        }
#pragma unroll
                        for (int i = 0; i < XMAXR; ++i) {
                            const int r = rbase + i * rstep;
                            if (r >= KTp) break;
                            uint32_t wv[4] = {0, 0, 0, 0};
                            if (ko[i] >= 0) {
#pragma unroll
                                for (int e = 0; e < Tr::E; ++e) {
                                    if (jj[e] < nb) {
                                        if constexpr (ES == 2) {
                                            const uint32_t h = lds16(xs[e] + uint32_t(ko[i]));
                                            wv[e >> 1] |= (e & 1) ? (h << 16) : h;
                                        } else {
                                            wv[e] = lds32(xs[e] + uint32_t(ko[i]));
                                        }
                                    }
                                }
                            }
                            put_raw_unit<T, 1>(op, op + KTp * ROWB, uo[i], make_uint4(wv[0], wv[1], wv[2], wv[3]));
                        }
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(smem_u32(&bars->b_full[bp.i]));
                        mbar_arrive(smem_u32(&bars->raw_empty[rp.i]));
                    }
                    bp.next(geo.nbs);
                                }
                if (!ok || !epilogue(ti, t)) break;
            }
        }
    }
    grid_dep_launch();  // the split reduction may be scheduled now (it waits for this grid)
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ======================================================================================
// d_input:  D[n, k] = sum_oc G[n, oc] * W[oc, k]  for the 128 columns n of NS whole
// samples (TMEM lanes) and k in one k-tile of CIC input channels (KTp >= CIC*K*K rows),
// then  dx[b, ic, h, w] = sum over (oh, kh) with oh*S + kh = h, (ow, kw) with
// ow*S + kw = w of D, in a fixed order (no atomics).  G = dy masked by y > 0 is the
// MMA's A operand in tensor memory (K = output channels along the TMEM columns), built
// once per sample tile; the packed W^T tiles are the shared-memory B operand.
// Warp roles (608 threads):
//   warp 1      w producer: packed W^T tiles (kt, oc chunk), one bulk copy each, into a ring.
//   warp 2      MMA: per k-tile, the oc-chunk MMAs into an accumulator buffer, then a
//               commit to that buffer's barrier (two buffers for bf16: the MMAs of k-tile
//               kt+1 run while k-tile kt is read out).
//   warps 3-18  formatters: per sample tile, load dy (and y) of their lane's column and
//               a quarter of the output channels from global memory, mask, split (fp32)
//               and store G to TMEM; per k-tile, TMEM -> Ds (fp32 [n][k] in shared
//               memory), then the col2im gather into dx with all 512 threads.
//   warp 0      idle after set-up.
// ======================================================================================
constexpr int DG_FMTW = 16;
constexpr int DG_THREADS = FV_FMT0 + 32 * DG_FMTW;
constexpr int DG_NFT = 32 * DG_FMTW;  // formatter threads
constexpr int DG_MAXW = 6;
constexpr int DG_TM = 128;             // columns per sample tile (TMEM lanes)

struct TcDgradGeom {
    int NS;          // samples per tile (NS * P <= 128)
    int CIC;         // input channels per k-tile
    int KTp;         // k rows per k-tile: CIC*K*K rounded up to 32
    int nkt;         // k-tiles
    int nch;         // K-chunks over OC
    int rmax;        // max (oh, kh) pairs per input row = ceil(K / S)
    int taps;        // max (kh, kw) taps landing on one input pixel
    int nw;          // weight ring stages
    int w_tile;      // bytes of one packed tile: KTp rows x 128 (x2 for split fp32)
    int dcols;       // accumulator columns per buffer: KTp (x2 for split fp32)
    int ndb;         // accumulator buffers
    int acol0;       // first TMEM column of the G buffers
    int acols;       // TMEM columns of one G buffer
    int nab;         // G buffers
    int ntiles;      // ceil(B / NS)
    int ktsplit;     // k-tile ranges per sample tile (more work items when the tiles are few)
    int kt_per;      // k-tiles per range
};

struct DgBars {
    uint64_t w_full[DG_MAXW], w_empty[DG_MAXW], a_full[2], a_empty[2], acc_full[2], acc_empty[2];
    uint64_t fbar;  // formatter-warp barrier (Ds written / Ds read)
    uint32_t tslot;
    int abort_flag;
};

template <typename T>
inline TcDgradGeom dgrad_geom(const ConvParams& p, int CIC, int nw)
{
    using Tr = TcTraits<T>;
    TcDgradGeom g;
    g.NS = std::max(1, DG_TM / p.P);
    g.CIC = CIC;
    g.KTp = round_up(CIC * p.KK, 32);
    g.nkt = ceil_div(p.IC, CIC);
    g.nch = ceil_div(p.OC, Tr::KC);
    g.rmax = (p.K + p.S - 1) / p.S;
    g.nw = nw;
    g.w_tile = g.KTp * ROWB * (Tr::split ? 2 : 1);
    g.dcols = g.KTp * (Tr::split ? 2 : 1);
    g.acols = Tr::split ? 2 * g.nch * Tr::KC : g.nch * Tr::KC / 2;
    // Two accumulator and two G buffers when they fit in the 512 TMEM columns.
    g.ndb = 2;
    g.nab = 2;
    if (2 * g.dcols + 2 * g.acols > 512) g.nab = 1;
    if (2 * g.dcols + g.acols > 512) g.ndb = 1;
    g.acol0 = g.ndb * g.dcols;
    g.ntiles = ceil_div(p.B, g.NS);
    g.ktsplit = 1;
    g.kt_per = g.nkt;
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

constexpr int DG_DSTR = DG_TM + 4;  // Ds row stride (floats): 16-byte rows, 4 banks apart
constexpr int DG_TMAX = 4;          // taps per input pixel handled by the fast gather
constexpr int DG_PROW = 8;          // ints per pixel row of the tap table (32 bytes, int4-aligned)

template <typename T>
inline int dgrad_smem(const ConvParams& p, const TcDgradGeom& g)
{
    return 1024 + g.nw * g.w_tile + DG_TM * DG_DSTR * 4 + 16 + (p.H + p.W) * (1 + g.rmax) * 8 + 16 +
           p.HW * DG_PROW * 4 + int(sizeof(DgBars)) + 16;
}

template <typename T>
inline size_t dgrad_packed_bytes(const TcDgradGeom& g)
{
    return size_t(g.nkt) * g.nch * g.w_tile;
}

template <typename T, bool RELU, int SWZ>
__global__ void __launch_bounds__(DG_THREADS, 1)
dgrad_tc_kernel(const ConvParams p, const T* __restrict__ dy, const unsigned char* __restrict__ wpack,
                const T* __restrict__ y, T* __restrict__ dx, const TcDgradGeom geo)
{
    using Tr = TcTraits<T>;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = align1024(smem_raw);
    unsigned char* wring = smem;
    float* Ds = reinterpret_cast<float*>(wring + geo.nw * geo.w_tile);
    const int R1 = 1 + geo.rmax;
    int2* rtab = reinterpret_cast<int2*>(Ds + DG_TM * DG_DSTR + 4);  // 4 floats: the zero word
    int2* ctab = rtab + p.H * R1;
    // Per input pixel hw: its contributing (p, kh*K + kw) as Ds offsets p*DSTR + kh*K + kw,
    // then the count (only used when every pixel has <= DG_TMAX taps).
    int* ptab = reinterpret_cast<int*>((reinterpret_cast<uintptr_t>(ctab + p.W * R1) + 15) & ~uintptr_t(15));
    DgBars* bars = reinterpret_cast<DgBars*>(ptab + p.HW * DG_PROW);
    volatile int* abort_flag = &bars->abort_flag;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid < 4) Ds[DG_TM * DG_DSTR + tid] = 0.f;
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
    const bool fast_taps = geo.taps <= DG_TMAX;
    __syncthreads();  // rtab / ctab complete
    if (fast_taps) {
        for (int hw = tid; hw < p.HW; hw += DG_THREADS) {
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
        for (int i = 0; i < geo.nw; ++i) {
            mbar_init(smem_u32(&bars->w_full[i]), 1);
            mbar_init(smem_u32(&bars->w_empty[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&bars->a_full[i]), DG_FMTW);
            mbar_init(smem_u32(&bars->a_empty[i]), 1);
            mbar_init(smem_u32(&bars->acc_full[i]), 1);
            mbar_init(smem_u32(&bars->acc_empty[i]), DG_FMTW);
        }
        mbar_init(smem_u32(&bars->fbar), DG_FMTW);
        fence_mbar_init();
        bars->abort_flag = 0;
    }
    if (warp == 0) tmem_alloc(smem_u32(&bars->tslot), 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tslot;
    // Work item wi = (sample tile wi % ntiles, k-tile range wi / ntiles).
    const int nwork = geo.ntiles * geo.ktsplit;
    auto ktrange = [&](int wi, int& lo, int& hi) {
        lo = (wi / geo.ntiles) * geo.kt_per;
        hi = min(geo.nkt, lo + geo.kt_per);
    };

    if (warp == 1) {
        // ---------------- w producer ----------------
        if (lane == 0) {
            grid_dep_wait();  // the packed weights come from the kernel launched just before
            RingPos wp;
            bool ok = true;
            for (int wi = blockIdx.x; wi < nwork && ok && !*abort_flag; wi += gridDim.x) {
                int kt_lo, kt_hi;
                ktrange(wi, kt_lo, kt_hi);
                const unsigned char* src = wpack + size_t(kt_lo) * geo.nch * geo.w_tile;
                for (int i = 0; i < (kt_hi - kt_lo) * geo.nch; ++i, wp.next(geo.nw), src += geo.w_tile) {
                    if (wp.wrapped && !mbar_wait_or_abort(smem_u32(&bars->w_empty[wp.i]), wp.ph ^ 1u, abort_flag)) {
                        report(const_cast<int*>(abort_flag), 16u);
                        ok = false;
                        break;
                    }
                    const uint32_t bar = smem_u32(&bars->w_full[wp.i]);
                    mbar_arrive_expect_tx(bar, uint32_t(geo.w_tile));
                    bulk_g2s(smem_u32(wring + wp.i * geo.w_tile), src, uint32_t(geo.w_tile), bar);
                }
            }
        }
        __syncwarp();
    } else if (warp == FV_MMA_WARP) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            const uint32_t idesc2 = instr_desc(Tr::fmt, DG_TM, geo.dcols);
            const uint32_t idesc1 = instr_desc(Tr::fmt, DG_TM, geo.KTp);
            const uint32_t w_u32 = smem_u32(wring);
            RingPos wp, abp, dbp;
            bool ok = true;
            for (int wi = blockIdx.x; wi < nwork && ok && !*abort_flag; wi += gridDim.x, abp.next(geo.nab)) {
                int kt_lo, kt_hi;
                ktrange(wi, kt_lo, kt_hi);
                if (!mbar_wait_or_abort(smem_u32(&bars->a_full[abp.i]), abp.ph, abort_flag)) {
                    report(const_cast<int*>(abort_flag), 8u);
                    break;
                }
                const uint32_t ga = tmem + uint32_t(geo.acol0 + abp.i * geo.acols);
                for (int kt = kt_lo; kt < kt_hi && ok; ++kt, dbp.next(geo.ndb)) {
                    if (dbp.wrapped &&
                        !mbar_wait_or_abort(smem_u32(&bars->acc_empty[dbp.i]), dbp.ph ^ 1u, abort_flag)) {
                        report(const_cast<int*>(abort_flag), 8u);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t acc = tmem + uint32_t(dbp.i * geo.dcols);
                    for (int ch = 0; ch < geo.nch; ++ch, wp.next(geo.nw)) {
                        if (!mbar_wait_or_abort(smem_u32(&bars->w_full[wp.i]), wp.ph, abort_flag)) {
                            report(const_cast<int*>(abort_flag), 8u);
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t wa = w_u32 + wp.i * geo.w_tile;
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const uint64_t bd = op_desc<SWZ>(wa + kstep_off<SWZ>(j));
                            const uint32_t first = (ch == 0 && j == 0) ? 0u : 1u;
                            const uint32_t col = uint32_t(ch * 32 + 8 * j);  // oc columns of this step
                            if constexpr (Tr::split) {
                                mma_tf32_ta(acc, ga + col, bd, idesc2, first);                          // hi*[hi;lo]
                                mma_tf32_ta(acc, ga + uint32_t(geo.nch * Tr::KC) + col, bd, idesc1, 1u);  // lo*hi
                            } else {
                                mma_f16_ta(acc, ga + col, bd, idesc1, first);
                            }
                        }
                        mma_commit(smem_u32(&bars->w_empty[wp.i]));
                    }
                    if (!ok) break;
                    mma_commit(smem_u32(&bars->acc_full[dbp.i]));
                }
                if (!ok) break;
                mma_commit(smem_u32(&bars->a_empty[abp.i]));
            }
        }
        __syncwarp();
    } else if (warp >= 3) {
        // ---------------- formatters + col2im ----------------
        const int ft = tid - FV_FMT0;       // 0 .. 511
        const uint32_t ds_u32 = smem_u32(Ds);
        const int fw = warp - 3;            // 0 .. 15
        const int qd = warp & 3;            // TMEM lane quarter
        const int sub = fw >> 2;            // quarter of the oc range (G) / of the k range (D)
        const int m = qd * 32 + lane;       // column within the tile
        const uint32_t lane_bits = uint32_t(qd * 32) << 16;
        const int ocq = geo.nch * Tr::KC / 4;  // output channels per formatter warp
        // G rows of sample tile `tile` into G buffer `ab`: dy (masked) of column m, channels
        // [sub*ocq, (sub+1)*ocq); zeros past the batch or past OC.
        auto build_g = [&](int tile, const RingPos& ab) -> bool {
            if (ab.wrapped && !mbar_wait_or_abort(smem_u32(&bars->a_empty[ab.i]), ab.ph ^ 1u, abort_flag)) {
                report(const_cast<int*>(abort_flag), 1u);
                return false;
            }
            tc_fence_after();
            const int b0 = tile * geo.NS, ns = min(geo.NS, p.B - b0);
            const bool valid = m < ns * p.P;
            uint32_t si = 0, pq = 0;
            p.dm_P.divmod(uint32_t(valid ? m : 0), si, pq);
            const size_t base = (size_t(b0) + si) * p.OCP + pq;  // si = 0, pq = 0 for invalid lanes
            const uint32_t gcol = tmem + lane_bits + uint32_t(geo.acol0 + ab.i * geo.acols);
            // Batches of 16 channels: every load of a batch is issued before the first use.
            for (int o0 = sub * ocq; o0 < (sub + 1) * ocq; o0 += 16) {
                // Unconditional loads from clamped addresses (invalid lanes and channels
                // past OC read a valid element), zeroed afterwards.
                float v[16], yv[16];
                const T* dyp = dy + base;
                const T* yp = y + base;
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int oc = min(o0 + e, p.OC - 1);
                    v[e] = Elem<T>::ldg(dyp + oc * p.P);
                    if (RELU) yv[e] = Elem<T>::ldg(yp + oc * p.P);
                }
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int oc = o0 + e;
                    bool keep = valid && oc < p.OC && oc < (sub + 1) * ocq;
                    if (RELU) keep = keep && yv[e] > 0.f;
                    if (!keep) v[e] = 0.f;
                }
                const int nb = min(16, (sub + 1) * ocq - o0);  // multiple of 8 (fp32) / 16 (bf16)
                if constexpr (Tr::split) {
#pragma unroll
                    for (int g8 = 0; g8 < 2; ++g8) {
                        if (8 * g8 >= nb) break;
                        uint32_t hi[8], lo[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const float f = v[8 * g8 + e];
                            const float h = to_tf32(f);
                            hi[e] = __float_as_uint(h);
                            lo[e] = __float_as_uint(f - h);
                        }
                        tmem_st8(gcol + uint32_t(o0 + 8 * g8), hi);
                        tmem_st8(gcol + uint32_t(geo.nch * Tr::KC + o0 + 8 * g8), lo);
                    }
                } else {
#pragma unroll
                    for (int g16 = 0; g16 < 1; ++g16) {
                        uint32_t wv[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            wv[e] = uint32_t(__bfloat16_as_ushort(__float2bfloat16_rn(v[16 * g16 + 2 * e]))) |
                                    (uint32_t(__bfloat16_as_ushort(__float2bfloat16_rn(v[16 * g16 + 2 * e + 1]))) << 16);
                        tmem_st8(gcol + uint32_t((o0 + 16 * g16) / 2), wv);
                    }
                }
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bars->a_full[ab.i]));
            return true;
        };
        // Barrier of the 16 formatter warps (bounded wait, unlike bar.sync).
        uint32_t fph = 0;
        auto fmt_sync = [&]() -> bool {
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bars->fbar));
            const bool done = mbar_wait_or_abort(smem_u32(&bars->fbar), fph, abort_flag);
            fph ^= 1u;
            if (!done) report(const_cast<int*>(abort_flag), 2u);
            return done;
        };
        RingPos abp, dbp;
        bool ok = true;
        const int first = blockIdx.x;
        if (first < nwork) ok = build_g(first % geo.ntiles, abp);
        for (int wi = first; wi < nwork && ok; wi += gridDim.x) {
            const int tile = wi % geo.ntiles;
            int kt_lo, kt_hi;
            ktrange(wi, kt_lo, kt_hi);
            RingPos nab = abp;
            nab.next(geo.nab);
            const int next = wi + int(gridDim.x);
            // With two G buffers the next tile's G is written before this tile's k-tiles
            // are read out, so the MMAs move on to it without waiting.
            if (geo.nab == 2 && next < nwork && !(ok = build_g(next % geo.ntiles, nab))) break;
            const int b0 = tile * geo.NS, ns = min(geo.NS, p.B - b0);
            for (int kt = kt_lo; kt < kt_hi; ++kt, dbp.next(geo.ndb)) {
                if (!mbar_wait_or_abort(smem_u32(&bars->acc_full[dbp.i]), dbp.ph, abort_flag)) {
                    report(const_cast<int*>(abort_flag), 2u);
                    ok = false;
                    break;
                }
                tc_fence_after();
                // TMEM -> Ds: this warp's lanes, k columns [sub*KTp/4, (sub+1)*KTp/4) (a
                // multiple of 8), two 8-column loads per wait, then 16-byte shared stores.
                {
                    const uint32_t acc = tmem + lane_bits + uint32_t(dbp.i * geo.dcols);
                    const int kq = geo.KTp / 4, c0 = sub * kq;
                    const uint32_t drow = ds_u32 + uint32_t((m * DG_DSTR + c0) * 4);
                    for (int c = 0; c < kq; c += 16) {
                        const bool two = c + 8 < kq;
                        uint32_t r[2][8], r2[2][8];
                        tmem_ld8(acc + uint32_t(c0 + c), r[0]);
                        if (two) tmem_ld8(acc + uint32_t(c0 + c + 8), r[1]);
                        if constexpr (Tr::split) {
                            tmem_ld8(acc + uint32_t(geo.KTp + c0 + c), r2[0]);
                            if (two) tmem_ld8(acc + uint32_t(geo.KTp + c0 + c + 8), r2[1]);
                        }
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 2; ++i) {
                            if (i == 1 && !two) break;
                            if constexpr (Tr::split) {
#pragma unroll
                                for (int e = 0; e < 8; ++e)
                                    r[i][e] = __float_as_uint(__uint_as_float(r[i][e]) + __uint_as_float(r2[i][e]));
                            }
                            sts128(drow + uint32_t(4 * (c + 8 * i)), r[i][0], r[i][1], r[i][2], r[i][3]);
                            sts128(drow + uint32_t(4 * (c + 8 * i)) + 16, r[i][4], r[i][5], r[i][6], r[i][7]);
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&bars->acc_empty[dbp.i]));
                if (!fmt_sync()) {
                    ok = false;
                    break;
                }
                const int ic0 = kt * geo.CIC, nic = min(geo.CIC, p.IC - ic0);
                if (fast_taps) {
                    // Thread owns (pixel hw, a subset of the samples); its <= 4 tap offsets
                    // stay in registers while it walks the chunk's channels.
                    const int nsplit = max(1, DG_NFT / p.HW);
                    for (int it = ft; it < p.HW * nsplit; it += DG_NFT) {
                        const int hw = it % p.HW, part = it / p.HW;
                        const int4 o = *reinterpret_cast<const int4*>(ptab + hw * DG_PROW);
                        // Absent taps read the zero word kept past the Ds rows and do not move
                        // with the channel; present ones step by one channel's K*K values.
                        const uint32_t zero = ds_u32 + uint32_t(DG_TM * DG_DSTR * 4);
                        const uint32_t kstep = uint32_t(p.KK * 4);
                        const uint32_t d0 = o.x >= 0 ? kstep : 0u, d1 = o.y >= 0 ? kstep : 0u;
                        const uint32_t d2 = o.z >= 0 ? kstep : 0u, d3 = o.w >= 0 ? kstep : 0u;
                        for (int sI = part; sI < ns; sI += nsplit) {
                            T* dxs = dx + size_t(b0 + sI) * p.IHW + size_t(ic0) * p.HW + hw;
                            const uint32_t ds = ds_u32 + uint32_t(sI * p.P * DG_DSTR * 4);
                            uint32_t a0 = o.x >= 0 ? ds + uint32_t(o.x * 4) : zero;
                            uint32_t a1 = o.y >= 0 ? ds + uint32_t(o.y * 4) : zero;
                            uint32_t a2 = o.z >= 0 ? ds + uint32_t(o.z * 4) : zero;
                            uint32_t a3 = o.w >= 0 ? ds + uint32_t(o.w * 4) : zero;
#pragma unroll 4
                            for (int icl = 0; icl < nic; ++icl) {
                                const float v0 = __uint_as_float(lds32(a0)), v1 = __uint_as_float(lds32(a1));
                                const float v2 = __uint_as_float(lds32(a2)), v3 = __uint_as_float(lds32(a3));
                                Elem<T>::st(dxs, ((v0 + v1) + v2) + v3);
                                dxs += p.HW;
                                a0 += d0;
                                a1 += d1;
                                a2 += d2;
                                a3 += d3;
                            }
                        }
                    }
                } else {
                    const int span = nic * p.HW;
                    for (int sI = 0; sI < ns; ++sI) {
                        T* dxs = dx + size_t(b0 + sI) * p.IHW + size_t(ic0) * p.HW;
                        const float* ds = Ds + sI * p.P * DG_DSTR;
                        for (int t = ft; t < span; t += DG_NFT) {
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
                if (!fmt_sync()) {  // Ds consumed
                    ok = false;
                    break;
                }
            }
            if (!ok) break;
            if (geo.nab == 1 && next < nwork && !(ok = build_g(next % geo.ntiles, nab))) break;
            abp = nab;
        }
    }
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <typename T> constexpr int dt_of_tc();
template <> constexpr int dt_of_tc<float>() { return DT_F32; }
template <> constexpr int dt_of_tc<__nv_bfloat16>() { return DT_BF16; }




}  // namespace

// Weight-ring depth, x super-chunk length and K ranges of the forward kernel: feasible
// (shared memory, packed weights and partials within the scratch buffer) and of the lowest
// estimated time (fwd_cost).
template <typename T>
static bool pick_fwd(const ConvParams& p, const DevInfo& d, FwdGeom& out)
{
    // Per list, the first that fits: the deepest weight ring, then the longest x super-chunk
    // (fewer, larger slab copies); or short super-chunks first, so that K splits into more
    // ranges.  Of the two, the lower estimated time (ties: the first list).
    // {weight stages, chunks per x super-chunk, raw x slots}
    static const int cfgs[][3] = {{4, 8, 2}, {4, 6, 2}, {4, 4, 2}, {4, 2, 2}, {3, 4, 2}, {3, 2, 2}, {2, 2, 2},
                                  {2, 1, 2}};
    static const int cfgs_split[][3] = {{4, 2, 2}, {3, 2, 2}, {2, 2, 2}, {4, 1, 2}, {2, 1, 2}};
    bool found = false;
    double best = 0.0;
    for (int pass = 0; pass < 2; ++pass) {
        const int ncfg = pass == 0 ? 8 : 5;
        for (int i = 0; i < ncfg; ++i) {
            const int* c = pass == 0 ? cfgs[i] : cfgs_split[i];
            FwdGeom g = fwd_geom<T>(p, c[1], c[0], c[2]);
            if (g.na < 2 || fwd_smem<T>(p, g) > d.smem_optin || fwd_packed_bytes<T>(g) > kScratchBytes) continue;
            const double t = fwd_set_splits(g, p, d.sms, fwd_packed_bytes<T>(g), kScratchBytes);
            if (!found || t < best) {
                out = g;
                best = t;
                found = true;
            }
            break;
        }
    }
    return found;
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
    // weight packing, the implicit GEMM, and with K ranges the sum of their partials
    pl.launches = g.splits > 1 ? 3 : 2;
    pl.block = FA_THREADS;
    pl.splits = g.splits;
    pl.variant = ((g.kc_per * 16 + g.xg) * 16 + g.nw) * 8 + g.nraw;
    pl.grid = std::min(g.n_tiles * g.oc_tiles * g.splits, d.sms);
    pl.smem = dt == DT_BF16 ? fwd_smem<__nv_bfloat16>(p, g) : fwd_smem<float>(p, g);
    return pl;
}

template <typename T>
static cudaError_t fwd_tc_t(const Plan& pl, const ConvParams& p, const void* x, const void* w,
                            const void* bias, void* y, cudaStream_t s)
{
    const int v = pl.variant;
    FwdGeom g = fwd_geom<T>(p, (v / 128) % 16, (v / 8) % 16, v % 8);
    g.kc_per = v / 2048;
    g.splits = ceil_div(g.nchunks, g.kc_per);
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
    float* part = reinterpret_cast<float*>(wpack + round_up(fwd_packed_bytes<T>(g), size_t(256)));
#define IG_LAUNCH_FWD_TC(R)                                                                         \
    do {                                                                                            \
        e = ensure_smem<fwd_tc_kernel<T, R, 1>>(pl.smem);                                           \
        if (e == cudaSuccess)                                                                       \
            e = launch_overlapped(fwd_tc_kernel<T, R, 1>, dim3(pl.grid), dim3(pl.block), pl.smem, s, p,   \
                                  (const T*)x, (const unsigned char*)wpack, (const T*)bias, (T*)y, part, g); \
        if (e == cudaSuccess && g.splits > 1) {                                                     \
            const size_t total = size_t(p.N) * p.OC;                                                \
            const int rgrid = int(std::min<size_t>((total + 255) / 256, 4096));                     \
            e = launch_overlapped(fwd_reduce_kernel<T, R>, dim3(rgrid), dim3(256), 0, s, p,           \
                                  (const float*)part, g.splits, g.oc_tiles * g.OTp, (const T*)bias,   \
                                  (T*)y);                                                             \
        }                                                                                           \
    } while (0)
    if (p.relu) IG_LAUNCH_FWD_TC(true);
    else IG_LAUNCH_FWD_TC(false);
#undef IG_LAUNCH_FWD_TC
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t run_fwd_tc(const Plan& pl, const ConvParams& p, int dt, const void* x, const void* w,
                       const void* bias, void* y, cudaStream_t s)
{
    return dt == DT_F32 ? fwd_tc_t<float>(pl, p, x, w, bias, y, s)
                        : fwd_tc_t<__nv_bfloat16>(pl, p, x, w, bias, y, s);
}

// ---- wgrad ------------------------------------------------------------------------------
// k rows per tile: the largest the accumulator allows (128 for fp32 hi + lo, 256 for
// bf16), shrunk to K*K*IC rounded up to 32; splits: enough tiles to cover the SMs, at least two
// chunks per split; then the deepest raw / B rings that fit.
template <typename T>
static bool pick_wgrad(const ConvParams& p, const DevInfo& d, TcWgradGeom& out)
{
    using Tr = TcTraits<T>;
    if (p.P > Tr::KC || p.B <= 0 || p.OC > TC_M) return false;  // one dy range of all OC per chunk
    const int ktmax = Tr::split ? 128 : 256;
    const int ktp = std::min(ktmax, round_up(p.Kred, 32));  // epilogue quarters of 8-column loads
    const int cnp = round_up(wgrad_nsc(p.P, Tr::KC, Tr::KC / 4) * p.P, Tr::KC / 4);
    const int upr = cnp / Tr::E;
    if (ceil_div(ktp, 32 * (16 - WgRoles<T>::g_warps) / upr) > WgRoles<T>::x_rows) return false;  // rows per X thread
    const int ng = Tr::split ? 8 : 16;  // G columns per group
    if (ceil_div(cnp / ng, WgRoles<T>::g_warps / 4) > WgRoles<T>::g_groups) return false;
    const int tiles = ceil_div(p.Kred, ktp) * ceil_div(p.OC, TC_M);
    const int nsc = wgrad_nsc(p.P, Tr::KC, Tr::KC / 4);
    int splits = std::max(1, d.sms / tiles);
    splits = std::min(splits, std::max(1, p.B / (2 * nsc)));
    // The raw ring hides the bulk copies' latency (about 1.5k clocks from issue to landing),
    // so it gets the deeper ring; two B stages suffice.
    static const int cfgs[][2] = {{5, 2}, {4, 2}, {3, 3}, {3, 2}, {2, 2}};  // {raws, nbs}
    for (const auto& c : cfgs) {
        const TcWgradGeom g = wgrad_geom<T>(p, ktp, c[0], c[1], splits);
        if (g.na >= 2 && wgrad_smem<T>(g) <= d.smem_optin) {
            out = g;
            return true;
        }
    }
    return false;
}

bool tc_wgrad_ok(const ConvParams& p, int dt, const DevInfo& d)
{
    if (d.cc_major != 10) return false;
    if (p.N == 0) return true;
    TcWgradGeom g;
    return dt == DT_BF16 ? pick_wgrad<__nv_bfloat16>(p, d, g) : pick_wgrad<float>(p, d, g);
}

Plan plan_wgrad_tc(const ConvParams& p, int dt, const DevInfo& d)
{
    Plan pl;
    pl.algo = ALGO_TC;
    pl.block = WG_THREADS;
    if (p.N == 0) {
        pl.launches = 1;  // the reduction alone writes zeros
        pl.splits = 0;
        pl.grid = 1;
        return pl;
    }
    TcWgradGeom g;
    if (dt == DT_BF16) pick_wgrad<__nv_bfloat16>(p, d, g);
    else pick_wgrad<float>(p, d, g);
    pl.smem = dt == DT_BF16 ? wgrad_smem<__nv_bfloat16>(g) : wgrad_smem<float>(g);
    pl.splits = g.splits;
    pl.variant = (g.KTp * 8 + g.raws) * 4 + g.nbs;
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
        const int v = pl.variant;
        const TcWgradGeom g = wgrad_geom<T>(p, v / 32, (v / 4) % 8, v % 4, pl.splits);
#define IG_LAUNCH_WG_TC(R)                                                                                 \
    do {                                                                                                   \
        e = ensure_smem<wgrad_tc_kernel<T, R>>(pl.smem);                                                   \
        if (e == cudaSuccess)                                                                              \
            wgrad_tc_kernel<T, R><<<pl.grid, pl.block, pl.smem, s>>>(p, (const T*)x, (const T*)dy,         \
                                                                     (const T*)y, (float*)ws, g);          \
    } while (0)
        if (p.relu) IG_LAUNCH_WG_TC(true);
        else IG_LAUNCH_WG_TC(false);
#undef IG_LAUNCH_WG_TC
        if (e == cudaSuccess) e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return run_wgrad_reduce(p, dt_of_tc<T>(), (const float*)ws, pl.splits, kpad, dw, s, pl.splits > 0);
}

cudaError_t run_wgrad_tc(const Plan& pl, const ConvParams& p, int dt, const void* x, const void* dy,
                         const void* y, void* dw, void* ws, int sms, cudaStream_t s)
{
    return dt == DT_F32 ? wgrad_tc_t<float>(pl, p, x, dy, y, dw, ws, sms, s)
                        : wgrad_tc_t<__nv_bfloat16>(pl, p, x, dy, y, dw, ws, sms, s);
}

// ---- d_input ------------------------------------------------------------------------
// Channels per k-tile: as many as keep KTp within the accumulator limit (128 rows; the fp32
// accumulator holds hi and lo halves), then the deepest weight ring that fits.
template <typename T>
static bool pick_dgrad(const ConvParams& p, const DevInfo& d, TcDgradGeom& out)
{
    if (p.B <= 0 || p.KK > 128 || p.P > DG_TM) return false;
    for (int cic = std::min(p.IC, 128 / p.KK); cic >= 1; --cic) {
        for (int nw = 4; nw >= 2; --nw) {
            TcDgradGeom g = dgrad_geom<T>(p, cic, nw);
            if (g.dcols * g.ndb + g.acols * g.nab > 512) continue;
            if (dgrad_smem<T>(p, g) <= d.smem_optin && dgrad_packed_bytes<T>(g) <= kScratchBytes) {
                if (2 * g.ntiles < d.sms) {  // few sample tiles: split the k-tiles too
                    const int want = std::min(g.nkt, d.sms / g.ntiles);
                    g.kt_per = ceil_div(g.nkt, want);
                    g.ktsplit = ceil_div(g.nkt, g.kt_per);
                }
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
    pl.block = DG_THREADS;
    pl.variant = (g.kt_per * 128 + g.CIC) * 8 + g.nw;
    pl.grid = std::min(g.ntiles * g.ktsplit, d.sms);
    pl.smem = dt == DT_BF16 ? dgrad_smem<__nv_bfloat16>(p, g) : dgrad_smem<float>(p, g);
    return pl;
}

template <typename T>
static cudaError_t dgrad_tc_t(const Plan& pl, const ConvParams& p, const void* dy, const void* w,
                              const void* y, void* dx, int, cudaStream_t s)
{
    TcDgradGeom g = dgrad_geom<T>(p, (pl.variant / 8) % 128, pl.variant % 8);
    g.kt_per = pl.variant / 1024;
    g.ktsplit = ceil_div(g.nkt, g.kt_per);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    unsigned char* wpack = static_cast<unsigned char*>(stream_scratch(dev, s));
    if (!wpack) return cudaErrorMemoryAllocation;
    const size_t units = size_t(g.nkt) * g.nch * g.KTp * 8;
    const int pgrid = int(std::min<size_t>((units + 255) / 256, 4096));
    pack_dgrad_w_kernel<T><<<pgrid, 256, 0, s>>>(p, (const T*)w, wpack, g.nkt, g.nch, g.CIC, g.KTp);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // The weight operand is always in the 128-byte swizzled layout the pack kernel writes.
#define IG_LAUNCH_DG_TC(R)                                                                                 \
    do {                                                                                                   \
        e = ensure_smem<dgrad_tc_kernel<T, R, 1>>(pl.smem);                                                \
        if (e == cudaSuccess)                                                                              \
            e = launch_overlapped(dgrad_tc_kernel<T, R, 1>, dim3(pl.grid), dim3(pl.block), pl.smem, s, p, \
                                  (const T*)dy, (const unsigned char*)wpack, (const T*)y, (T*)dx, g);      \
    } while (0)
    if (p.relu) IG_LAUNCH_DG_TC(true);
    else IG_LAUNCH_DG_TC(false);
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
