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
#include <climits>
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

__device__ __forceinline__ unsigned char* align1024(unsigned char* p)
{
    return reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Raw bits of one element of w (zero-extended for bf16).
template <typename T>
__device__ __forceinline__ uint32_t ld_bits(const T* p)
{
    if constexpr (sizeof(T) == 4) return __ldg(reinterpret_cast<const unsigned int*>(p));
    else return __ldg(reinterpret_cast<const unsigned short*>(p));
}

// The fp32 split of the 3xTF32 products: hi = tf32(v) (round to nearest), lo = v - hi (exact
// in fp32; the MMA reads its leading tf32 bits).  Every operand of the fp32 path is split so.
__device__ __forceinline__ void split_tf32(uint32_t bits, uint32_t& hi, uint32_t& lo)
{
    const float f = __uint_as_float(bits);
    const float h = to_tf32(f);
    hi = __float_as_uint(h);
    lo = __float_as_uint(f - h);
}

// ======================================================================================
// Weight operand stages, formatted inside the kernels from w as the caller passes it
// (OC x IC*K*K, row-major; 16-byte aligned base): 128-byte rows, 128-byte swizzled, K-major,
// fp32 as tf32 hi rows followed (lo_off bytes further) by lo rows.  Dedicated weight-formatter
// warps do it in two steps per stage, one stage apart:
//   stage_*   each lane issues 16-byte cp.async copies of the aligned blocks that cover the
//             pieces of w the warp itself will format, into a raw slot of the warp's own
//             (no register holds the data in flight; copies past OC or past the end of w
//             are zero-filled); the copies of one stage form one cp.async group;
//   format_*  after cp.async.wait_group and __syncwarp, the warp reads its raw slot
//             (conflict-free 32-lane runs), splits fp32 into tf32 hi / lo, and stores the
//             operand stage; the caller fences the stores for the tensor core and arrives.
// A warp copies exactly what it formats, so no other warp waits on its copies.
// ======================================================================================
constexpr int NWF = 4;      // weight-formatter warps of the forward
constexpr int DG_NWF = 2;   // weight-formatter warps of d_input (608 threads: up to 96 registers each)
constexpr int WRAW = 2;     // raw slots per warp: the next stage's copies fly while one is formatted
constexpr int WRB = 144;    // bytes of a raw row piece: 128 bytes of w plus 16 of alignment slack

// Forward stage: row r = output channel oc0 + r (r < OTp), K = k0 .. k0 + KC - 1 (128 bytes of
// one row of w).  Warp wf owns rows wf, wf + NWF, ...; its raw slot holds them at WRB-byte
// strides, each as the 9 aligned blocks covering [&w[oc][k0], +128).
inline __host__ __device__ int fwd_wraw_warp_bytes(int OTp) { return ((OTp + NWF - 1) / NWF) * WRB; }

template <typename T>
__device__ __forceinline__ void stage_w_fwd(uint32_t slot, const T* __restrict__ w, const ConvParams& p, int oc0,
                                            int k0, int OTp, int wf, int lane)
{
    const char* wb = reinterpret_cast<const char*>(w);
    const char* wend = wb + size_t(p.OC) * p.Kred * sizeof(T);
    const int nrw = (OTp - wf + NWF - 1) / NWF;
    for (int q = lane; q < nrw * 9; q += 32) {
        const int i = q / 9, j = q - 9 * (q / 9);
        const int oc = oc0 + wf + NWF * i;
        const char* a = wb + (size_t(oc) * p.Kred + k0) * sizeof(T);
        const char* s = reinterpret_cast<const char*>(reinterpret_cast<uintptr_t>(a) & ~uintptr_t(15)) + 16 * j;
        const int n = (oc < p.OC && s < wend) ? int(min(ptrdiff_t(16), wend - s)) : 0;
        cp_async16(slot + uint32_t(i * WRB + 16 * j), n > 0 ? s : wb, uint32_t(n));
    }
}

// Lane L stores K value L (+ 32 for bf16) of each of the warp's rows: every read is a
// 32-lane run of one raw row, every store one 128-byte row of the stage (all banks).  The
// warp's rows r = wf + NWF*i have r & 7 = wf + 4 (i & 1) and r >> 3 = i >> 1, and their raw
// pieces start at one of two misalignments (even / odd i), so the loop carries no address
// arithmetic.  Rows past OC were zero-filled by the copies; K values past Kred (the last,
// ragged chunk) are zeroed here.
template <typename T>
__device__ __forceinline__ void format_w_fwd(uint32_t stage, uint32_t lo_off, uint32_t slot, const ConvParams& p,
                                             int oc0, int k0, int OTp, int wf, int lane)
{
    using Tr = TcTraits<T>;
    constexpr int EPL = Tr::KC / 32;  // K values per lane and row
    constexpr int ES = int(sizeof(T));
    const int nrw = OTp / NWF;        // even: OTp is a multiple of 16
    uint32_t src[2], soff[2][EPL];
    bool kval[EPL];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        const int d = int(((size_t(oc0 + wf + NWF * t) * p.Kred + k0) * ES) & 15);
        src[t] = slot + uint32_t(t * WRB + d + lane * ES);
        const int r7 = wf + 4 * t;
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
            const int kk = lane + 32 * e;
            soff[t][e] = stage + uint32_t(r7 * 128 + (((kk / Tr::E) ^ r7) << 4) + (kk % Tr::E) * ES);
        }
    }
#pragma unroll
    for (int e = 0; e < EPL; ++e) kval[e] = k0 + lane + 32 * e < p.Kred;
#pragma unroll 4
    for (int i2 = 0; i2 < nrw / 2; ++i2) {
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            const uint32_t s = src[t] + uint32_t(i2 * 2 * WRB);
#pragma unroll
            for (int e = 0; e < EPL; ++e) {
                uint32_t v = ES == 4 ? lds32(s + uint32_t(64 * e)) : lds16(s + uint32_t(64 * e));
                if (!kval[e]) v = 0u;
                const uint32_t a = soff[t][e] + uint32_t(i2 * 1024);
                if constexpr (Tr::split) {
                    uint32_t hi, lo;
                    split_tf32(v, hi, lo);
                    sts32(a, hi);
                    sts32(a + lo_off, lo);
                } else {
                    sts16(a, v);
                }
            }
        }
    }
}

// d_input stage (W transposed): row r = k0 + r of the reduction index (r < mrows; zero rows
// up to KTp), K = output channels oc0 .. oc0 + KC - 1.  Warp wf owns the 32-row groups
// g = wf, wf + DG_NWF, ...; for each of them and each of the KC channels its raw slot holds the
// aligned blocks covering w[oc][k0 + 32 g .. +32) (9 blocks for fp32, 5 for bf16).
template <typename T> struct DgRaw {
    static constexpr int blocks = sizeof(T) == 4 ? 9 : 5;  // aligned 16-byte blocks per (group, channel)
    static constexpr int rb = 16 * blocks;
};
template <typename T>
inline __host__ __device__ int dgrad_wraw_warp_bytes(int KTp)
{
    return ((KTp / 32 + DG_NWF - 1) / DG_NWF) * TcTraits<T>::KC * DgRaw<T>::rb;
}

template <typename T>
__device__ __forceinline__ void stage_wt_dgrad(uint32_t slot, const T* __restrict__ w, const ConvParams& p, int k0,
                                               int oc0, int KTp, int wf, int lane)
{
    using Tr = TcTraits<T>;
    constexpr int NB = DgRaw<T>::blocks, RB = DgRaw<T>::rb;
    const char* wb = reinterpret_cast<const char*>(w);
    const char* wend = wb + size_t(p.OC) * p.Kred * sizeof(T);
    const int ngw = (KTp / 32 - wf + DG_NWF - 1) / DG_NWF;
    for (int q = lane; q < ngw * Tr::KC * NB; q += 32) {
        const int gi = q / (Tr::KC * NB), rem = q - gi * (Tr::KC * NB);
        const int jj = rem / NB, b = rem - NB * (rem / NB);
        const int oc = oc0 + jj, g = wf + DG_NWF * gi;
        const char* a = wb + (size_t(oc) * p.Kred + k0 + 32 * g) * sizeof(T);
        const char* s = reinterpret_cast<const char*>(reinterpret_cast<uintptr_t>(a) & ~uintptr_t(15)) + 16 * b;
        const int n = (oc < p.OC && s < wend) ? int(min(ptrdiff_t(16), wend - s)) : 0;
        cp_async16(slot + uint32_t((gi * Tr::KC + jj) * RB + 16 * b), n > 0 ? s : wb, uint32_t(n));
    }
}

// Lane L builds row 32 g + L of each of the warp's groups: per 16-byte unit, E channels read
// from E raw runs (32-lane runs, conflict-free) and one 16-byte store (the swizzle spreads the
// warp's 32 rows over all banks).  Channel oc0 + c*E + e starts its run at a misalignment
// that depends on e only, so the loop carries no address arithmetic.  Channels past OC were
// zero-filled by the copies; rows past mrows are zeroed here.
template <typename T>
__device__ __forceinline__ void format_wt_dgrad(uint32_t stage, uint32_t lo_off, uint32_t slot, const ConvParams& p,
                                                int k0, int mrows, int oc0, int KTp, int wf, int lane)
{
    using Tr = TcTraits<T>;
    constexpr int E = Tr::E, ES = int(sizeof(T)), RB = DgRaw<T>::rb;
    const int ngw = (KTp / 32 - wf + DG_NWF - 1) / DG_NWF;
    uint32_t d[E];
#pragma unroll
    for (int e = 0; e < E; ++e) d[e] = uint32_t(((size_t(oc0 + e) * p.Kred + k0) * ES) & 15) + uint32_t(lane * ES);
    const uint32_t rbase = uint32_t((lane >> 3) * 1024 + (lane & 7) * 128);
    for (int gi = 0; gi < ngw; ++gi) {
        const int g = wf + DG_NWF * gi, r = 32 * g + lane;
        const bool rv = r < mrows;
        const uint32_t gslot = slot + uint32_t(gi * Tr::KC * RB);
        const uint32_t gst = stage + uint32_t(4 * g * 1024) + rbase;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            uint32_t v[E];
#pragma unroll
            for (int e = 0; e < E; ++e) {
                v[e] = ES == 4 ? lds32(gslot + uint32_t((c * E + e) * RB) + d[e])
                               : lds16(gslot + uint32_t((c * E + e) * RB) + d[e]);
                if (!rv) v[e] = 0u;
            }
            const uint32_t a = gst + uint32_t((c ^ (lane & 7)) << 4);
            if constexpr (Tr::split) {
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) split_tf32(v[e], hi[e], lo[e]);
                sts128(a, hi[0], hi[1], hi[2], hi[3]);
                sts128(a + lo_off, lo[0], lo[1], lo[2], lo[3]);
            } else {
                sts128(a, v[0] | (v[1] << 16), v[2] | (v[3] << 16), v[4] | (v[5] << 16), v[6] | (v[7] << 16));
            }
        }
    }
}

// Workspace path: the same stages packed once per call into the caller's workspace, so that
// the main kernel fetches each with one bulk copy instead of formatting it in every CTA.
// The images are byte-identical to what in-kernel formatting produces (same split, same
// zeros), so both paths give bit-identical results.  Grid (units / 256, chunks, tiles), one
// 16-byte unit (hi and lo for fp32) per thread: no division.
//   forward: tile (ot, kc) at index ot*nchunks + kc, OTp rows
//   d_input: tile (kt, ch) at index kt*nch + ch, KTp rows (W transposed)
template <typename T>
__device__ __forceinline__ void put_unit(unsigned char* hi, unsigned char* lo, uint32_t off,
                                         const uint32_t (&v)[TcTraits<T>::E])
{
    if constexpr (TcTraits<T>::split) {
        uint32_t h[4], l[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) split_tf32(v[e], h[e], l[e]);
        *reinterpret_cast<uint4*>(hi + off) = make_uint4(h[0], h[1], h[2], h[3]);
        *reinterpret_cast<uint4*>(lo + off) = make_uint4(l[0], l[1], l[2], l[3]);
    } else {
        *reinterpret_cast<uint4*>(hi + off) =
            make_uint4(v[0] | (v[1] << 16), v[2] | (v[3] << 16), v[4] | (v[5] << 16), v[6] | (v[7] << 16));
    }
}

template <typename T>
__global__ void pack_fwd_w_kernel(const ConvParams p, const T* __restrict__ w, unsigned char* __restrict__ out,
                                  int nchunks, int OTp)
{
    grid_dep_launch();  // the implicit GEMM may start its prologue meanwhile
    using Tr = TcTraits<T>;
    const int u = blockIdx.x * blockDim.x + threadIdx.x;
    if (u >= OTp * 8) return;
    const int kc = blockIdx.y, ot = blockIdx.z, r = u >> 3, c = u & 7;
    const int oc = ot * OTp + r, k = kc * Tr::KC + c * Tr::E;
    uint32_t v[Tr::E];
#pragma unroll
    for (int e = 0; e < Tr::E; ++e) v[e] = (oc < p.OC && k + e < p.Kred) ? ld_bits(w + size_t(oc) * p.Kred + k + e) : 0u;
    unsigned char* base = out + (size_t(ot) * nchunks + kc) * (size_t(OTp) * ROWB * (Tr::split ? 2 : 1));
    put_unit<T>(base, base + OTp * ROWB, unit_off<1>(r, c), v);
}

template <typename T>
__global__ void pack_dgrad_w_kernel(const ConvParams p, const T* __restrict__ w, unsigned char* __restrict__ out,
                                    int nch, int CIC, int KTp)
{
    grid_dep_launch();  // the implicit GEMM may start its prologue meanwhile
    using Tr = TcTraits<T>;
    const int u = blockIdx.x * blockDim.x + threadIdx.x;
    if (u >= KTp * 8) return;
    const int ch = blockIdx.y, kt = blockIdx.z, r = u >> 3, c = u & 7;
    const int k0 = kt * CIC * p.KK, mrows = min(CIC, p.IC - kt * CIC) * p.KK;
    uint32_t v[Tr::E];
#pragma unroll
    for (int e = 0; e < Tr::E; ++e) {
        const int oc = ch * Tr::KC + c * Tr::E + e;
        v[e] = (r < mrows && oc < p.OC) ? ld_bits(w + size_t(oc) * p.Kred + k0 + r) : 0u;
    }
    unsigned char* base = out + (size_t(kt) * nch + ch) * (size_t(KTp) * ROWB * (Tr::split ? 2 : 1));
    put_unit<T>(base, base + KTp * ROWB, unit_off<1>(r, c), v);
}

// ======================================================================================
// Forward: tile = (128 columns n = (b, oh, ow), OTp output channels); K = IC*K*K in
// chunks of KC.  The gathered operand X[n, k] is the MMA's A operand and lives in
// tensor memory (lane m = column n0 + m, K along the TMEM columns); the weights are the
// B operand in shared memory (N = OTp rows; fp32: the tf32 hi rows followed by the lo rows,
// so one N = 2*OTp MMA forms X_hi*W_hi and X_hi*W_lo, and a second N = OTp MMA adds
// X_lo*W_hi into the first half).  Only the weights are read from shared memory by the
// tensor core.
// Warp roles (704 threads):
//   warp 0      x producer: per super-chunk (XG consecutive K-chunks) and per sample the
//               tile touches, one bulk copy of the contiguous channels x[b, ic_lo : ic_hi]
//               the super-chunk covers, into one of the raw slots.  Sources are rounded
//               down to 16 bytes (the slack is skipped when read); bytes of a last
//               16-byte block that lie past the end of x are copied by plain loads.
//   warp 1      MMA: one thread issues the chunk's tcgen05.mma steps, commits to the
//               weight stage's and the TMEM operand stage's "empty" barriers and, after
//               a tile's last chunk, to the accumulator barrier.
//   warps 2-5   weight formatters: each K-chunk's weight stage from w (stage_w_fwd, format_w_fwd).
//   warps 6-21  gather formatters: warp w owns TMEM lanes 32*(w%4) .. +31 (one column each)
//               and a quarter of each chunk's K; gathers its column's patch values from the
//               raw slot and writes them with tcgen05.st; then the tile's epilogue
//               (TMEM -> bias -> ReLU -> y), each warp a quarter of the output channels.
// K ranges: with fewer column tiles than half the SMs, the K-chunks of a tile split into
// R ranges computed by the R CTAs of one thread-block cluster.  Each CTA writes its fp32
// partial tile into its own shared memory; after a cluster barrier CTA q sums rows
// [q*128/R, (q+1)*128/R) of the R partials in ascending rank order through distributed
// shared memory, adds the bias, applies the ReLU and writes y.  No global scratch.
// ======================================================================================
constexpr int FV_MAXRAWS = 4;  // max raw x slots of the forward

constexpr int FA_XWARP = 0;    // x producer
constexpr int FA_MMAWARP = 1;  // MMA issuer
constexpr int FA_WF0 = 2;      // first weight-formatter warp
constexpr int FA_FMT0 = 32 * (FA_WF0 + NWF);  // first gather-formatter thread (warp 6)
constexpr int FA_TM = 128;    // columns per forward tile (TMEM lanes)
constexpr int FA_KSPLIT = 4;  // formatter warps per TMEM lane quarter (each a quarter of the chunk's K)
constexpr int FA_FMTW = 4 * FA_KSPLIT;
constexpr int FA_THREADS = FA_FMT0 + 32 * FA_FMTW;
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
    int splits;         // K ranges = cluster size (1: no split)
    int kc_per;         // K-chunks per range (a multiple of xg)
    int packed;         // 1: weight stages bulk-copied from a packed image in the workspace
};

struct FwdBars {
    uint64_t raw_full[FV_MAXRAWS], raw_empty[FV_MAXRAWS];
    uint64_t w_full[FA_MAXW], w_empty[FA_MAXW];
    uint64_t a_full[FA_MAXA], a_empty[FA_MAXA];
    uint64_t acc_full, acc_empty;
    uint32_t tslot;
    int abort_flag;
};

// Row stride (floats) of a CTA's partial tile in the K-range reduction: 16-byte rows whose
// first words fall 4 banks apart.
inline __host__ __device__ int fwd_red_stride(int OTp) { return OTp + 4; }

// Shared-memory wavefronts of one gather load of the forward's formatters: the 32 lanes of a warp
// are 32 consecutive columns n = (b, oh, ow) of a tile, all reading the same k; lane n reads the
// word at (b - b_first) * xs + (its slab's 16-byte misalignment) + its pixel's offset.  A bank
// serves one word per wavefront (equal words broadcast).
inline int fwd_gather_wavefronts(const ConvParams& p, int es, int xs, int n0, int b_first, int cmis)
{
    int word[32], bank_words[32] = {0};
    for (int m = 0; m < 32; ++m) {
        const int n = std::min(n0 + m, p.N - 1);
        const int b = n / p.P, pq = n % p.P, oh = pq / p.OW, ow = pq % p.OW;
        const long long mis = ((long long)b * p.IHW * es + cmis) & 15;
        word[m] = int(((long long)(b - b_first) * xs + mis + (oh * p.S * p.W + ow * p.S) * es) >> 2);
        bool seen = false;
        for (int i = 0; i < m && !seen; ++i) seen = word[i] == word[m];
        if (!seen) ++bank_words[word[m] & 31];
    }
    int w = 0;
    for (int b = 0; b < 32; ++b) w = std::max(w, bank_words[b]);
    return w;
}

// Per-sample stride of the forward's raw x slots (a multiple of 16 bytes, at least xs0): of the
// eight residues modulo 128 bytes, the one whose gather loads need the fewest wavefronts, counted
// over the warps of the first tiles and the misalignments (in steps of the element size, at
// least 4 bytes) a super-chunk's first channel can add.  Each sample's slab sits 0-15 bytes into its slot (its source's misalignment),
// which is why a fixed residue does not serve every shape.  Remembered per shape (per thread).
inline int fwd_sample_stride(const ConvParams& p, int es, int xs0)
{
    struct Entry { int P, OW, S, W, IHW, N, es, xs0, xs; };
    constexpr int NCACHE = 64;
    static thread_local Entry cache[NCACHE];
    static thread_local int next = 0;
    for (const Entry& e : cache)
        if (e.xs0 == xs0 && e.P == p.P && e.OW == p.OW && e.S == p.S && e.W == p.W && e.IHW == p.IHW &&
            e.es == es && e.N == std::min(p.N, 3 * FA_TM))
            return e.xs;
    int best = xs0, best_cost = INT_MAX;
    for (int i = 0; i < 8; ++i) {
        const int xs = xs0 + 16 * i;
        int cost = 0;
        for (int t = 0; t < 3 && t * FA_TM < p.N; ++t)
            for (int q = 0; q < 4; ++q)
                for (int cmis = 0; cmis < 16; cmis += std::min(es, 4))
                    cost += fwd_gather_wavefronts(p, es, xs, t * FA_TM + q * 32, (t * FA_TM) / p.P, cmis);
        if (cost < best_cost) {
            best_cost = cost;
            best = xs;
        }
    }
    cache[next] = Entry{p.P, p.OW, p.S, p.W, p.IHW, std::min(p.N, 3 * FA_TM), es, xs0, best};
    next = (next + 1) % NCACHE;
    return best;
}

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
    g.xs = fwd_sample_stride(p, es, round_up(chmax * p.HW * es + 16, 16));
    g.raw_bytes = round_up(g.nsmax * g.xs, 128);
    g.w_bytes = g.OTp * ROWB * (Tr::split ? 2 : 1);
    g.dcols = g.OTp * (Tr::split ? 2 : 1);
    g.acol0 = round_up(g.dcols, 32);
    g.acols = Tr::split ? 2 * Tr::KC : Tr::KC / 2;
    g.na = std::min(FA_MAXA, (FA_TMEM_COLS - g.acol0) / g.acols);
    g.splits = 1;
    g.kc_per = g.nchunks;
    g.packed = 0;
    return g;
}

// Estimated forward time in chunk steps of one CTA (about a microsecond each): rounds of
// work items over the SMs x chunks per item, plus, with K ranges, the in-cluster reduction
// (a cluster barrier and R distributed-shared-memory reads per output).
inline double fwd_cost(int tiles, int sms, int splits, int kc)
{
    return double(ceil_div(tiles * splits, sms)) * kc + (splits > 1 ? 0.5 + 0.05 * splits : 0.0);
}

// K ranges, only when the column tiles fill fewer than half the SMs (with more, a range's
// fixed cost -- its own x slabs and pipeline fill -- outweighs the gain; layer 1 at B = 1024,
// 96 tiles, ran 8 % slower in fp32 and 40 % slower in bf16 with three ranges): the split of
// the nchunks K-chunks (kc_per of them, a multiple of xg, per range) into R <= kMaxCluster
// ranges, one cluster of R CTAs per tile, with the lowest estimated time.  Returns that
// estimate.
inline double fwd_set_splits(FwdGeom& g, int sms)
{
    const int tiles = g.n_tiles * g.oc_tiles;
    double best = fwd_cost(tiles, sms, 1, g.nchunks);
    if (2 * tiles >= sms || g.nchunks < 2 * g.xg) return best;
    const int smax = std::min(g.nchunks / g.xg, kMaxCluster);
    for (int want = 2; want <= smax; ++want) {
        const int kc = round_up(ceil_div(g.nchunks, want), g.xg);
        const int splits = ceil_div(g.nchunks, kc);
        if (splits < 2 || tiles * splits > sms) continue;  // one work item per CTA
        const double c = fwd_cost(tiles, sms, splits, kc);
        if (c < best) {
            best = c;
            g.kc_per = kc;
            g.splits = splits;
        }
    }
    return best;
}

// Raw w slots of the weight formatters (none on the workspace path).
inline __host__ __device__ int fwd_wraw_bytes(const FwdGeom& g)
{
    return g.packed ? 0 : NWF * WRAW * fwd_wraw_warp_bytes(g.OTp);
}

template <typename T>
inline int fwd_smem(const ConvParams& p, const FwdGeom& g)
{
    const int kred_pad = round_up(p.Kred, TcTraits<T>::KC);
    return 1024 + g.nw * g.w_bytes + g.nraw * g.raw_bytes + fwd_wraw_bytes(g) + kred_pad * 4 + int(sizeof(FwdBars)) +
           16;
}

// With K ranges the partial tile (128 rows x fwd_red_stride(OTp) floats) reuses the weight
// stages and raw slots once the tile's MMAs are done.
inline bool fwd_red_fits(const FwdGeom& g)
{
    return g.splits <= 1 || size_t(FA_TM) * fwd_red_stride(g.OTp) * 4 <= size_t(g.nw) * g.w_bytes +
                                                                           size_t(g.nraw) * g.raw_bytes;
}

__device__ __forceinline__ int warp_sum(int v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Store the 16-byte unit `v` of a B operand stage: as tf32 hi and lo parts (fp32), or as is (bf16).
template <typename T, int SWZ>
__device__ __forceinline__ void put_raw_unit(unsigned char* hi, unsigned char* lo, uint32_t off, uint4 v)
{
    if constexpr (TcTraits<T>::split) {
        uint32_t h[4], l[4];
        split_tf32(v.x, h[0], l[0]);
        split_tf32(v.y, h[1], l[1]);
        split_tf32(v.z, h[2], l[2]);
        split_tf32(v.w, h[3], l[3]);
        st_unit(hi, off, h[0], h[1], h[2], h[3]);
        st_unit(lo, off, l[0], l[1], l[2], l[3]);
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

template <typename T, bool RELU>
__global__ void __launch_bounds__(FA_THREADS, 1)
fwd_tc_kernel(const ConvParams p, const T* __restrict__ x, const T* __restrict__ w,
              const unsigned char* __restrict__ wpack, const T* __restrict__ bias, T* __restrict__ y, const FwdGeom geo)
{
    using Tr = TcTraits<T>;
    constexpr int ES = int(sizeof(T));
    constexpr int KQ = Tr::KC / FA_KSPLIT;        // K values per formatter warp and chunk
    constexpr int KQC = Tr::split ? KQ : KQ / 2;  // TMEM columns they fill (per part)
    static_assert(KQC == 8, "one tcgen05.st of 8 columns per part");
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = align1024(smem_raw);
    const int kred_pad = round_up(p.Kred, Tr::KC);
    // Layout: weight stages | raw x slots | raw w slots (NWF warps x WRAW) | k offsets | barriers
    unsigned char* wring = smem;
    unsigned char* raw = wring + geo.nw * geo.w_bytes;
    unsigned char* wraw = raw + geo.nraw * geo.raw_bytes;
    int* offk = reinterpret_cast<int*>(wraw + fwd_wraw_bytes(geo));
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
            mbar_init(smem_u32(&bars->w_full[i]), geo.packed ? 1 : NWF);
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
    // Nothing above touches global memory: the previous kernel on the stream may still run.
    grid_dep_wait();
    // Work item = (column tile, oc tile, K range).  Without K ranges the CTAs stride over the
    // tiles; with them the grid is one CTA per item and the R CTAs of a cluster share a tile.
    const int R = geo.splits;
    const int ctiles = geo.n_tiles * geo.oc_tiles;
    const int total_items = ctiles * R;
    auto decode = [&](int item, int& ntile, int& ot, int& kc_lo, int& kc_hi) {
        const int ct = item / R, range = item % R;
        ntile = ct % geo.n_tiles;
        ot = ct / geo.n_tiles;
        kc_lo = range * geo.kc_per;
        kc_hi = min(geo.nchunks, kc_lo + geo.kc_per);
    };

    if (warp == FA_XWARP) {
        // ---------------- x producer ----------------
        const unsigned char* xb = reinterpret_cast<const unsigned char*>(x);
        const unsigned char* x_end = xb + size_t(p.B) * p.IHW * ES;
        RingPos rp;
        for (int item = blockIdx.x; item < total_items && !*abort_flag; item += gridDim.x) {
            int ntile, ot, kc_lo, kc_hi;
            decode(item, ntile, ot, kc_lo, kc_hi);
            const int n0 = ntile * FA_TM;
            const int n_end = min(n0 + FA_TM, p.N);
            const int b_first = n0 / p.P, nsamp = (n_end - 1) / p.P - b_first + 1;
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
                __syncwarp();  // every lane's tail stores happen before lane 0's (releasing) arrive
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
    } else if (warp >= FA_WF0 && warp < FA_WF0 + NWF && geo.packed) {
        // ---------------- weight stages from the packed image (workspace path) ----------------
        if (warp == FA_WF0 && lane == 0) {
            RingPos wp;
            for (int item = blockIdx.x; item < total_items && !*abort_flag; item += gridDim.x) {
                int ntile, ot, kc_lo, kc_hi;
                decode(item, ntile, ot, kc_lo, kc_hi);
                const unsigned char* src = wpack + (size_t(ot) * geo.nchunks + kc_lo) * geo.w_bytes;
                bool ok = true;
                for (int kc = kc_lo; kc < kc_hi; ++kc, wp.next(geo.nw), src += geo.w_bytes) {
                    if (wp.wrapped && !mbar_wait_or_abort(smem_u32(&bars->w_empty[wp.i]), wp.ph ^ 1u, abort_flag)) {
                        report(const_cast<int*>(abort_flag), 16u);
                        ok = false;
                        break;
                    }
                    const uint32_t bar = smem_u32(&bars->w_full[wp.i]);
                    mbar_arrive_expect_tx(bar, uint32_t(geo.w_bytes));
                    bulk_g2s(smem_u32(wring + wp.i * geo.w_bytes), src, uint32_t(geo.w_bytes), bar);
                }
                if (!ok) break;
            }
        }
        __syncwarp();
    } else if (warp >= FA_WF0 && warp < FA_WF0 + NWF) {
        // ---------------- weight formatters ----------------
        // The warp's chunk sequence (item, kc) over this CTA's work items; the copies of the
        // next chunk are in flight while the current one is formatted.
        const int wf = warp - FA_WF0;
        const uint32_t w_u32 = smem_u32(wring), lo_off = uint32_t(geo.OTp * ROWB);
        const uint32_t slot0 = smem_u32(wraw) + uint32_t(wf * WRAW * fwd_wraw_warp_bytes(geo.OTp));
        const uint32_t slot_bytes = uint32_t(fwd_wraw_warp_bytes(geo.OTp));
        struct Seq { int item, kc, hi, ot; };
        auto first = [&](Seq& s, int item) -> bool {
            if (item >= total_items) return false;
            int ntile, lo;
            decode(item, ntile, s.ot, lo, s.hi);
            s.item = item;
            s.kc = lo;
            return true;
        };
        auto advance = [&](Seq& s) -> bool { return ++s.kc < s.hi || first(s, s.item + int(gridDim.x)); };
        Seq cur;
        bool have = first(cur, int(blockIdx.x));
        if (have) stage_w_fwd<T>(slot0, w, p, cur.ot * geo.OTp, cur.kc * Tr::KC, geo.OTp, wf, lane);
        cp_async_commit();
        uint32_t slot = 0;
        RingPos wp;
        while (have && !*abort_flag) {
            Seq nxt = cur;
            const bool have_nxt = advance(nxt);
            if (have_nxt)
                stage_w_fwd<T>(slot0 + (slot ^ 1u) * slot_bytes, w, p, nxt.ot * geo.OTp, nxt.kc * Tr::KC, geo.OTp, wf,
                               lane);
            cp_async_commit();
            cp_async_wait<1>();  // this lane's copies of the current chunk have landed
            __syncwarp();        // ... and every lane's are visible to the warp
            if (wp.wrapped && !mbar_wait_or_abort(smem_u32(&bars->w_empty[wp.i]), wp.ph ^ 1u, abort_flag)) {
                report(const_cast<int*>(abort_flag), 16u);
                break;
            }
            format_w_fwd<T>(w_u32 + uint32_t(wp.i * geo.w_bytes), lo_off, slot0 + slot * slot_bytes, p,
                            cur.ot * geo.OTp, cur.kc * Tr::KC, geo.OTp, wf, lane);
            fence_proxy_async_smem();  // the generic-proxy stores, for the tensor core
            __syncwarp();              // also: every lane is done reading this raw slot
            if (lane == 0) mbar_arrive(smem_u32(&bars->w_full[wp.i]));
            wp.next(geo.nw);
            cur = nxt;
            have = have_nxt;
            slot ^= 1u;
        }
        cp_async_wait<0>();  // no copy may land after the CTA's shared memory is reused or released
    } else if (warp == FA_MMAWARP) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            // fp32: N = 2*OTp over [W_hi; W_lo], then N = OTp over W_hi; bf16: N = OTp.
            const uint32_t idesc2 = instr_desc(Tr::fmt, FA_TM, geo.dcols);
            const uint32_t idesc1 = instr_desc(Tr::fmt, FA_TM, geo.OTp);
            const uint32_t w_u32 = smem_u32(wring);
            RingPos wp, ap;
            uint32_t t = 0;
            for (int item = blockIdx.x; item < total_items && !*abort_flag; item += gridDim.x, ++t) {
                int ntile, ot, kc_lo, kc_hi;
                decode(item, ntile, ot, kc_lo, kc_hi);
                bool ok = true;
                if (t >= 1 && !mbar_wait_or_abort(smem_u32(&bars->acc_empty), (t - 1) & 1, abort_flag)) {
                    report(const_cast<int*>(abort_flag), 8u);
                    break;
                }
                tc_fence_after();
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
                        const uint64_t bd = op_desc<1>(wa + kstep_off<1>(j));
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
    } else if (warp >= FA_FMT0 / 32) {
        // ---------------- gather formatters + epilogue ----------------
        const int fw = warp - FA_FMT0 / 32;  // 0 .. FA_FMTW - 1
        const int qd = warp & 3;             // TMEM lane quarter this warp may access
        const int sub = fw >> 2;             // which quarter of each chunk's K
        const int m = qd * 32 + lane;        // this thread's column within the tile
        const uint32_t lane_bits = uint32_t(qd * 32) << 16;
        const uint32_t raw_u32 = smem_u32(raw), offk_u32 = smem_u32(offk) + uint32_t(sub * KQ * 4);
        const bool ragged_k = (p.Kred % Tr::KC) != 0;
        RingPos ap, rp;
        uint32_t t = 0;
        for (int item = blockIdx.x; item < total_items; item += gridDim.x, ++t) {
            int ntile, ot, kc_lo, kc_hi;
            decode(item, ntile, ot, kc_lo, kc_hi);
            const int n0 = ntile * FA_TM;
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
                    for (int e = 0; e < 8; ++e) split_tf32(v[e], hi[e], lo[e]);
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
            // Epilogue: TMEM -> y, plus the bias if given, then ReLU; with K ranges -> this
            // CTA's fp32 partial tile in shared memory (row m, the tile's OTp channels), reduced
            // across the cluster below.  This warp's lanes, every FA_KSPLIT-th group of 8 channels.
            if (!mbar_wait_or_abort(smem_u32(&bars->acc_full), t & 1, abort_flag)) {
                report(const_cast<int*>(abort_flag), 2u);
                break;
            }
            tc_fence_after();
            if (R == 1) grid_dep_launch();  // the last tile: the next kernel may be scheduled now
            T* yc = (R == 1 && n < p.N) ? y + col_out(p, n) : nullptr;
            const uint32_t red_row = smem_u32(smem) + uint32_t(m * fwd_red_stride(geo.OTp) * 4);
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
                } else if (R > 1) {
                    sts128(red_row + uint32_t(cb * 4), r[0], r[1], r[2], r[3]);
                    sts128(red_row + uint32_t(cb * 4 + 16), r[4], r[5], r[6], r[7]);
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
    if (R > 1) {
        // K-range reduction across the cluster (every thread of every CTA passes both cluster
        // barriers exactly once, also after an aborted wait: the status word then already
        // holds the error and the output is unspecified).
        grid_dep_launch();
        cluster_sync();  // every CTA's partial tile is in its shared memory
        const int rank = int(cluster_rank());
        int ntile, ot, kc_lo, kc_hi;
        decode(int(blockIdx.x), ntile, ot, kc_lo, kc_hi);
        const int rows = ceil_div(FA_TM, R);  // tile rows (columns n) this CTA finishes
        const int r0 = rank * rows, r1 = min(FA_TM, r0 + rows);
        const int q4 = geo.OTp / 4;           // 16-byte groups of channels per row
        const int RS = fwd_red_stride(geo.OTp);
        const uint32_t base = smem_u32(smem);
        uint32_t peer[kMaxCluster];
#pragma unroll
        for (int q = 0; q < kMaxCluster; ++q) peer[q] = q < R ? dsmem_addr(base, uint32_t(q)) : 0u;
        for (int it = tid; it < (r1 - r0) * q4; it += FA_THREADS) {
            const int mm = r0 + it % (r1 - r0), g4 = it / (r1 - r0);  // consecutive threads: consecutive columns
            const int n = ntile * FA_TM + mm;
            if (n >= p.N) continue;
            const uint32_t off = uint32_t((mm * RS + g4 * 4) * 4);
            // All R loads in flight first, then the sum in ascending rank order.
            float4 v[kMaxCluster];
#pragma unroll
            for (int q = 0; q < kMaxCluster; ++q)
                if (q < R) v[q] = ld_dsmem_f4(peer[q] + off);
            float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int q = 0; q < kMaxCluster; ++q) {
                if (q >= R) break;
                s.x += v[q].x; s.y += v[q].y; s.z += v[q].z; s.w += v[q].w;
            }
            const float f4[4] = {s.x, s.y, s.z, s.w};
            T* yc = y + col_out(p, n);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int oc = ot * geo.OTp + g4 * 4 + e;
                if (oc < p.OC) {
                    float f = f4[e];
                    if (bias) f += Elem<T>::ldg(bias + oc);
                    if (RELU) f = f > 0.f ? f : 0.f;
                    Elem<T>::st(yc + size_t(oc) * p.P, f);
                }
            }
        }
        cluster_sync();  // no CTA leaves while a peer still reads its shared memory
    }
}

// ======================================================================================
// wgrad partials: tile = (128 output channels, KTp <= 128 reduction indices k, one split
// range of samples); the GEMM's K runs over the split's columns n = (b, oh, ow), a chunk
// being NSC whole samples (NSC*P columns, zero-padded to the MMA step):
//   D[k, oc] = sum_{n in split} X[n, k] * G[n, oc]
// X (the patches) is the MMA's A operand in tensor memory (lane = k row, K = n along the
// columns), written by the X formatters with tcgen05.st: consecutive lanes gather
// consecutive k, mostly consecutive words of the raw x slab.  G (dy masked by y > 0) is the
// shared-memory B operand (N = 128 output-channel rows, K-major along n; fp32 as tf32 hi
// rows then lo rows, so one N = 256 MMA forms X_hi*G_hi and X_hi*G_lo and an N = 128 MMA adds
// X_lo*G_hi), built by the G formatters with conflict-free 16-byte stores.  (With the
// operands the other way round the patch stage's swizzled stores made the kernel
// shared-memory bound: ~1600 wavefronts per 2-sample chunk at layer 1 fp32.)
// Warp roles (608 threads):
//   warps 0, 1  bulk-copy producers (lane 0 each): per chunk, the contiguous slab
//               dy[b0 : b0+nb] (and y, the ReLU mask source) by warp 0, and x[b, ic_lo :
//               ic_hi] (the k-tile's input channels) of each sample by warp 1, into a raw slot.
//   warp 2      MMA.
//   G warps     (the first 8 formatter warps for fp32, 4 for bf16) thread = output channel
//               row; the chunk's columns, masked and split, as 16-byte units of the
//               shared-memory stage.
//   X warps     (the other formatter warps, the same number per TMEM lane quarter) thread =
//               k row; groups of the chunk's columns into the TMEM operand stage.
//   warps 3-18  epilogue: D[k][oc] to ws[split][oc][k] (row stride kpad; lanes store
//               consecutive k).
// ======================================================================================
constexpr int WG_MMA_WARP = 2;
constexpr int WG_FMT0 = 96;  // first formatter thread (warp 3)
constexpr int WG_THREADS = WG_FMT0 + 32 * 16;
constexpr int WG_MAXA = 8, WG_MAXB = 4, WG_MAXR = 5;
// Formatter roles: G warps (a multiple of 4; thread = output channel row of the shared-memory
// stage) and X warps (the rest, a multiple of 4: each TMEM lane quarter gets the same number;
// thread = k row of the tensor-memory stage); the column groups (two 16-byte units, or one
// 8-word tcgen05.st) one thread of each builds.  Both get half the warps: each builds as many
// elements per chunk as the other.
template <typename T> struct WgRoles {
    static constexpr int g_warps = 8;
    static constexpr int g_groups = 2;
    static constexpr int x_groups = 2;
};
// The other layout (wgrad_tc_body_gt): g in tensor memory (lane = output channel) and the
// patches as the shared-memory operand, k-tiles up to 256 rows in bf16.  G warps (thread =
// output channel lane, its column groups of 8 words) and X warps (16-byte units of the
// patch stage, x_rows rows per thread).
template <typename T> struct WgRolesGt {
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
    int layout;    // 0: patches in TMEM (wgrad_tc_body); 1: g in TMEM (wgrad_tc_body_gt)
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
inline TcWgradGeom wgrad_geom(const ConvParams& p, int KTp, int raws, int nbs, int splits, int layout)
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
    // Shared-memory stage: g's TC_M output-channel rows (layout 0) or the KTp patch rows (layout
    // 1), x2 for the tf32 hi and lo rows; accumulator columns: D[k][oc]'s TC_M oc columns or
    // D[oc][k]'s KTp k columns, x2 for the hi and lo products.
    g.layout = layout;
    const int brows = layout ? KTp : TC_M;
    g.b_bytes = brows * ROWB * (Tr::split ? 2 : 1);
    g.nbs = nbs;
    g.dcols = brows * (Tr::split ? 2 : 1);
    g.acols = Tr::split ? 2 * Tr::KC : Tr::KC / 2;
    g.na = std::min(WG_MAXA, (512 - round_up(g.dcols, 32)) / g.acols);
    return g;
}

template <typename T>
inline int wgrad_smem(const TcWgradGeom& g)
{
    return 1024 + g.nbs * g.b_bytes + g.raws * g.raw_bytes + int(sizeof(WgBars)) + 16 * g.cnp + 16;
}

// The wgrad CTA's work: tiles item0, item0 + istride, ... (its own kernel passes the block
// index and the grid size; the fused backward kernel its own numbering of the wgrad CTAs).
template <typename T, bool RELU>
__device__ __forceinline__ void wgrad_tc_body(const ConvParams& p, const T* __restrict__ x, const T* __restrict__ dy,
                                              const T* __restrict__ y, float* __restrict__ ws,
                                              float* __restrict__ bpart, const TcWgradGeom& geo, const int item0,
                                              const int istride)
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
    // Column table of the x gather: column n -> (sample j, byte offset of its pixel from the
    // sample's channel ic_lo in the x region), right after the dy table.
    for (int n = tid; n < geo.cnp; n += WG_THREADS) {
        const int j = n / p.P, pq = n % p.P;
        gtab[2 * n] = n < geo.nsc * p.P ? j : 1 << 20;
        gtab[2 * n + 1] = (j * p.OCP + pq) * ES;
        const int oh = pq / p.OW, ow = pq % p.OW;
        gtab[2 * geo.cnp + 2 * n] = n < geo.nsc * p.P ? j : 1 << 20;
        gtab[2 * geo.cnp + 2 * n + 1] = (oh * p.S * p.W + ow * p.S) * ES;
    }
    if (tid == 0) {
        for (int i = 0; i < geo.raws; ++i) {
            mbar_init(smem_u32(&bars->raw_full[i]), 2);  // the two producers' arrivals
            mbar_init(smem_u32(&bars->raw_empty[i]), 16);
        }
        for (int i = 0; i < geo.na; ++i) {
            mbar_init(smem_u32(&bars->a_full[i]), 16 - WgRoles<T>::g_warps);  // the X warps
            mbar_init(smem_u32(&bars->a_empty[i]), 1);
        }
        for (int i = 0; i < geo.nbs; ++i) {
            mbar_init(smem_u32(&bars->b_full[i]), WgRoles<T>::g_warps);  // the G warps
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
    // Nothing above touches global memory: the previous kernel on the stream may still run.
    grid_dep_wait();
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
            for (int tile = item0; tile < total && !*abort_flag; tile += istride) {
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
    } else if (warp == WG_MMA_WARP) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            // A = the x patches (TMEM, M = TC_M k rows), B = g (shared memory, N = TC_M output
            // channels, fp32: N = 2*TC_M over [g_hi; g_lo], then N = TC_M over g_hi).
            const uint32_t idesc2 = instr_desc(Tr::fmt, TC_M, geo.dcols);
            const uint32_t idesc1 = instr_desc(Tr::fmt, TC_M, TC_M);
            const uint32_t b_u32 = smem_u32(bring);
            const int ksteps = geo.cnp / KS;
            RingPos ap, bp;
            uint32_t t = 0;
            for (int tile = item0; tile < total && !*abort_flag; tile += istride, ++t) {
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
        const int qd = warp & 3;            // TMEM lane quarter (X formatters, epilogue)
        const uint32_t lane_bits = uint32_t(qd * 32) << 16;
        constexpr int NGW = WgRoles<T>::g_warps;
        constexpr int NXS = (16 - NGW) / 4;  // X warps per TMEM lane quarter
        const int2* xtab = reinterpret_cast<const int2*>(gtab + 2 * geo.cnp);
        // Epilogue of tile t: D[k][oc] -> ws[split][oc][k]; lane = k row of this warp's quarter,
        // 32 of the oc columns per warp of the quarter (consecutive lanes store consecutive k).
        auto epilogue = [&](const TileInfo& ti, uint32_t t) -> bool {
            if (!mbar_wait_or_abort(smem_u32(&bars->acc_full), t & 1, abort_flag)) {
                report(const_cast<int*>(abort_flag), 2u);
                return false;
            }
            tc_fence_after();
            const int k = ti.k0 + qd * 32 + lane;
            const bool kin = qd * 32 + lane < KTp && k < p.Kred;
            const int c0 = (fw >> 2) * (TC_M / 4);
            for (int cb = c0; cb < c0 + TC_M / 4; cb += 8) {
                uint32_t r[8];
                tmem_ld8(tmem + lane_bits + uint32_t(cb), r);
                if constexpr (Tr::split) {
                    uint32_t r2[8];
                    tmem_ld8(tmem + lane_bits + uint32_t(TC_M + cb), r2);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 8; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) + __uint_as_float(r2[e]));
                } else {
                    tmem_ld_wait();
                }
                if (kin) {
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        if (cb + e < ti.rows)
                            ws[(size_t(ti.split) * p.OC + ti.oc0 + cb + e) * geo.kpad + k] = __uint_as_float(r[e]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bars->acc_empty));
            return true;
        };
        if (fw < NGW) {
            // ---------------- G formatters: the shared-memory operand ----------------
            // Thread = output channel row m of the B stage (oc0 + m); its column groups of NG
            // columns, each two 16-byte units of the K-major, 128-byte-swizzled row (fp32: the
            // tf32 hi rows, then the lo rows TC_M rows further).
            const int m = qd * 32 + lane;
            const int gsub = fw >> 2;           // which of the NGW/4 warps of its lane quarter
            constexpr int NG = ES == 4 ? 8 : 16;       // columns per group: two 16-byte units
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
            RingPos rp, bp;
            uint32_t t = 0;
            for (int tile = item0; tile < total; tile += istride, ++t) {
                const TileInfo ti = decode(tile);
                // The bias gradient rides on the first k-tile of each split (one per (split, oc
                // tile)): the sum of this thread's masked g values, chunk by chunk in ascending
                // order (k-tile 0 starts at chunk 0), each chunk's values in ascending column.
                const bool bias_tile = bpart != nullptr && ti.k0 == 0;
                float bsum = 0.f;
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
                    // Element (sample j, channel m, position pq) of the dy region; y is gregion further.
                    const int dg0 = int(((size_t(b0) * p.OCP + size_t(ti.oc0) * p.P) * ES) & 15);
                    const bool live = m < ti.rows;
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
                        if (bias_tile) {
#pragma unroll
                            for (int e = 0; e < NG; ++e) bsum += __uint_as_float(ES == 4 ? v[e] : (v[e] << 16));
                        }
                        if constexpr (Tr::split) {
                            put_raw_unit<T, 1>(op, op + TC_M * ROWB, unit_off<1>(m, 2 * g), make_uint4(v[0], v[1], v[2], v[3]));
                            put_raw_unit<T, 1>(op, op + TC_M * ROWB, unit_off<1>(m, 2 * g + 1),
                                               make_uint4(v[4], v[5], v[6], v[7]));
                        } else {
                            uint32_t wv[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e) wv[e] = __byte_perm(v[2 * e], v[2 * e + 1], 0x5410);
                            put_raw_unit<T, 1>(op, op, unit_off<1>(m, 2 * g), make_uint4(wv[0], wv[1], wv[2], wv[3]));
                            put_raw_unit<T, 1>(op, op, unit_off<1>(m, 2 * g + 1), make_uint4(wv[4], wv[5], wv[6], wv[7]));
                        }
                    }
                    fence_proxy_async_smem();  // the generic-proxy stores, for the tensor core
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(smem_u32(&bars->b_full[bp.i]));
                        mbar_arrive(smem_u32(&bars->raw_empty[rp.i]));
                    }
                    bp.next(geo.nbs);
                }
                if (ok && bias_tile && m < ti.rows)
                    bpart[(size_t(ti.split) * (NGW / 4) + gsub) * p.OC + ti.oc0 + m] = bsum;
                if (!ok || !epilogue(ti, t)) break;
            }
        } else {
            // ---------------- X formatters: the tensor-memory operand ----------------
            // Thread = k row of the tile (TMEM lane qd*32 + lane); its column groups of XG
            // columns (one tcgen05.st of 8 words each), the values gathered from the raw x slab:
            // column n = (sample j, position) reads x at the sample's slab + the position's
            // pixel offset + the row's k offset.  Consecutive lanes are consecutive k, i.e.
            // mostly consecutive words of the slab.
            const int xsub = (fw - NGW) >> 2;  // which of the NXS warps of its lane quarter
            constexpr int XG = ES == 4 ? 8 : 16;
            constexpr int XMAXG = WgRoles<T>::x_groups;
            const int xgroups = geo.cnp / XG;
            const int kr = qd * 32 + lane;
            RingPos rp, ap;
            uint32_t t = 0;
            for (int tile = item0; tile < total; tile += istride, ++t) {
                const TileInfo ti = decode(tile);
                const int k = ti.k0 + kr;
                const int ko = (kr < KTp && k < p.Kred) ? (k_offset(p, k) - ti.ic_lo * p.HW) * ES : -1;
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
                    // Sample j's slab sits (m0 + j * mstep) mod 16 bytes into its slot (its source's
                    // 16-byte misalignment).
                    const int m0 = int(((size_t(b0) * p.IHW + size_t(ti.ic_lo) * p.HW) * ES) & 15);
                    const int mstep = int((size_t(p.IHW) * ES) & 15);
                    const uint32_t xbase = slot + uint32_t(xoff + (ko >= 0 ? ko : 0));
                    const uint32_t col = tmem + lane_bits + uint32_t(acol0 + ap.i * geo.acols);
#pragma unroll
                    for (int gi = 0; gi < XMAXG; ++gi) {
                        const int g = xsub + gi * NXS;
                        if (g >= xgroups) break;
                        uint32_t v[XG];
#pragma unroll
                        for (int e = 0; e < XG; ++e) {
                            const int2 c = xtab[g * XG + e];  // (sample, pixel byte offset); the same for the warp
                            v[e] = 0u;
                            if (ko >= 0 && c.x < nb) {
                                const int mj = (m0 + c.x * mstep) & 15;
                                const uint32_t a = xbase + uint32_t(c.x * geo.xsb + mj + c.y);
                                v[e] = ES == 4 ? lds32(a) : lds16(a);
                            }
                        }
                        if constexpr (Tr::split) {
                            uint32_t hi[8], lo[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e) split_tf32(v[e], hi[e], lo[e]);
                            tmem_st8(col + uint32_t(g * 8), hi);
                            tmem_st8(col + uint32_t(Tr::KC + g * 8), lo);
                        } else {
                            uint32_t wv[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e) wv[e] = __byte_perm(v[2 * e], v[2 * e + 1], 0x5410);
                            tmem_st8(col + uint32_t(g * 8), wv);
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
        }
    }
    grid_dep_launch();  // the split reduction may be scheduled now (it waits for this grid)
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <typename T, bool RELU>
__device__ __forceinline__ void wgrad_tc_body_gt(const ConvParams& p, const T* __restrict__ x, const T* __restrict__ dy,
                                              const T* __restrict__ y, float* __restrict__ ws,
                                              float* __restrict__ bpart, const TcWgradGeom& geo, const int item0,
                                              const int istride)
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
            mbar_init(smem_u32(&bars->a_full[i]), WgRolesGt<T>::g_warps);
            mbar_init(smem_u32(&bars->a_empty[i]), 1);
        }
        for (int i = 0; i < geo.nbs; ++i) {
            mbar_init(smem_u32(&bars->b_full[i]), 16 - WgRolesGt<T>::g_warps);
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
    // Nothing above touches global memory: the previous kernel on the stream may still run.
    grid_dep_wait();
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
            for (int tile = item0; tile < total && !*abort_flag; tile += istride) {
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
    } else if (warp == WG_MMA_WARP) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            const uint32_t idesc2 = instr_desc(Tr::fmt, TC_M, geo.dcols);
            const uint32_t idesc1 = instr_desc(Tr::fmt, TC_M, KTp);
            const uint32_t b_u32 = smem_u32(bring);
            const int ksteps = geo.cnp / KS;
            RingPos ap, bp;
            uint32_t t = 0;
            for (int tile = item0; tile < total && !*abort_flag; tile += istride, ++t) {
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
        constexpr int NGW = WgRolesGt<T>::g_warps;
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
            constexpr int MAXG = WgRolesGt<T>::g_groups;  // column groups per thread
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
            for (int tile = item0; tile < total; tile += istride, ++t) {
                const TileInfo ti = decode(tile);
                // The bias gradient rides on the first k-tile of each split (one per (split, oc
                // tile)): the sum of this thread's masked g values, chunk by chunk in ascending
                // order (k-tile 0 starts at chunk 0), each chunk's values in ascending column.
                const bool bias_tile = bpart != nullptr && ti.k0 == 0;
                float bsum = 0.f;
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
                        if (bias_tile) {
#pragma unroll
                            for (int e = 0; e < NG; ++e) bsum += __uint_as_float(ES == 4 ? v[e] : (v[e] << 16));
                        }
                        if constexpr (Tr::split) {
                            uint32_t hi[8], lo[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e) split_tf32(v[e], hi[e], lo[e]);
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
                if (ok && bias_tile && m < ti.rows)
                    bpart[(size_t(ti.split) * (NGW / 4) + gsub) * p.OC + ti.oc0 + m] = bsum;
                if (!ok || !epilogue(ti, t)) break;
            }
        } else {
            // ---------------- X formatters ----------------
            // 16-byte unit column c (E columns) of rows rbase + i*rstep.
            const int xthreads = 32 * (16 - NGW);
            const int xt = tid - WG_FMT0 - 32 * NGW;
            const int upr = geo.cnp / Tr::E;     // units per row
            const int cfix = xt % upr;
            const int rbase = xt / upr;
            const int rstep = xthreads / upr;
            const bool xact = xt < rstep * upr;
            constexpr int XMAXR = WgRolesGt<T>::x_rows;  // rows per thread (checked by the planner)
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
            for (int tile = item0; tile < total; tile += istride, ++t) {
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

// Bias partial channel sums per split: one per G warp of a TMEM lane quarter.
template <typename T>
__host__ __device__ inline int wgrad_bias_parts(const TcWgradGeom& g)
{
    return g.splits * (g.layout ? WgRolesGt<T>::g_warps / 4 : WgRoles<T>::g_warps / 4);
}

// One kernel per operand layout (GT: g in tensor memory), so that each holds one body.
template <typename T, bool RELU, bool GT>
__global__ void __launch_bounds__(WG_THREADS, 1)
wgrad_tc_kernel(const ConvParams p, const T* __restrict__ x, const T* __restrict__ dy,
                const T* __restrict__ y, float* __restrict__ ws, float* __restrict__ bpart, const TcWgradGeom geo)
{
    if constexpr (GT) wgrad_tc_body_gt<T, RELU>(p, x, dy, y, ws, bpart, geo, int(blockIdx.x), int(gridDim.x));
    else wgrad_tc_body<T, RELU>(p, x, dy, y, ws, bpart, geo, int(blockIdx.x), int(gridDim.x));
}

// ======================================================================================
// d_input:  D[n, k] = sum_oc G[n, oc] * W[oc, k]  for the 128 columns n of NS whole
// samples (TMEM lanes) and k in one k-tile of CIC input channels (KTp >= CIC*K*K rows),
// then  dx[b, ic, h, w] = sum over (oh, kh) with oh*S + kh = h, (ow, kw) with
// ow*S + kw = w of D, in a fixed order (no atomics).  G = dy masked by y > 0 is the
// MMA's A operand in tensor memory (K = output channels along the TMEM columns), built
// once per sample tile; the W^T tiles are the shared-memory B operand, formatted in the
// kernel from w.
// Warp roles (608 threads):
//   warp 0      MMA: per k-tile, the oc-chunk MMAs into an accumulator buffer of KTp columns
//               (fp32: hi*hi, hi*lo and lo*hi into the same one), then a commit to that
//               buffer's barrier (two buffers: the MMAs of k-tile kt+1 run while k-tile kt is
//               read out).
//   warps 1-2   weight formatters: the W^T tiles (kt, oc chunk) from w into a ring of
//               stages (stage_wt_dgrad, format_wt_dgrad).
//   warps 3-18  formatters: per sample tile, load dy (and y) of their lane's column and
//               a quarter of the output channels from global memory (with P <= 4 the
//               CTA's first tile from whole sample slabs bulk-copied into the Ds rows), mask,
//               split (fp32) and store G to TMEM; per k-tile, TMEM -> Ds (fp32 [n][k] in
//               shared memory), then the col2im gather into dx with all 512 threads.
// ======================================================================================
constexpr int DG_MMA_WARP = 0;
constexpr int DG_WF0 = 1;                     // first weight-formatter warp
constexpr int DG_FMT0 = 32 * (DG_WF0 + DG_NWF);  // first formatter thread (warp 3)
constexpr int DG_FMTW = 16;
constexpr int DG_THREADS = DG_FMT0 + 32 * DG_FMTW;
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
    int dcols;       // accumulator columns per buffer: KTp
    int dstr;        // Ds row stride in floats (see dgrad_ds_stride)
    int grounds;     // channel blocks of the staged G build (0: not staged; see dgrad_tc_body)
    int gstride;     // bytes per sample block of the staged dy (and y) in the Ds rows
    int ndb;         // accumulator buffers
    int acol0;       // first TMEM column of the G buffers
    int acols;       // TMEM columns of one G buffer
    int nab;         // G buffers
    int ntiles;      // ceil(B / NS)
    int ktsplit;     // k-tile ranges per sample tile (more work items when the tiles are few)
    int kt_per;      // k-tiles per range
    int packed;      // 1: W^T stages bulk-copied from a packed image in the workspace
};

struct DgBars {
    uint64_t w_full[DG_MAXW], w_empty[DG_MAXW], a_full[2], a_empty[2], acc_full[2], acc_empty[2];
    uint64_t fbar;  // formatter-warp barrier (Ds written / Ds read)
    uint64_t gbar;  // staged G build: a channel block's bulk copies landed
    uint32_t tslot;
    int abort_flag;
};

constexpr int DG_TMAX = 4;          // taps per input pixel handled by the fast gather
constexpr int DG_PROW = 8;          // ints per pixel row of the tap table (32 bytes, int4-aligned)

// Shared-memory wavefronts of the fast col2im gather's first pass for Ds row stride `dstr`:
// thread it handles pixel it % HW of sample it / HW (channel 0; later samples and channels
// shift every address of a warp alike), one 4-byte load per tap the pixel has.
inline int dgrad_gather_wavefronts(const ConvParams& p, int NS, int dstr)
{
    const int nsplit = std::max(1, 512 / p.HW);
    const int items = p.HW * std::min(nsplit, NS);
    int total = 0;
    for (int w0 = 0; w0 < items; w0 += 32) {
        for (int t = 0; t < DG_TMAX; ++t) {
            int word[32], n = 0, bank_words[32] = {0};
            for (int it = w0; it < std::min(items, w0 + 32); ++it) {
                const int hw = it % p.HW, sI = it / p.HW, h = hw / p.W, c = hw % p.W;
                int k = 0, found = -1;
                for (int oh = 0; oh < p.OH && found < 0; ++oh) {
                    const int kh = h - oh * p.S;
                    if (kh < 0 || kh >= p.K) continue;
                    for (int ow = 0; ow < p.OW; ++ow) {
                        const int kw = c - ow * p.S;
                        if (kw < 0 || kw >= p.K) continue;
                        if (k++ == t) {
                            found = (sI * p.P + oh * p.OW + ow) * dstr + kh * p.K + kw;
                            break;
                        }
                    }
                }
                if (found < 0) continue;
                bool seen = false;
                for (int i = 0; i < n && !seen; ++i) seen = word[i] == found;
                if (!seen) {
                    word[n++] = found;
                    ++bank_words[found & 31];
                }
            }
            int wf = 0;
            for (int b = 0; b < 32; ++b) wf = std::max(wf, bank_words[b]);
            total += wf;
        }
    }
    return total;
}

// Ds row stride: DG_TM + 4 + 8i floats (i < 4), each an odd number of 16-byte units so that
// the 16-byte stores of eight consecutive rows hit eight different bank groups; of these, the
// one whose gather loads need the fewest wavefronts (layer 1, 11x15 with K=5, S=3: 148 floats,
// about 28 % fewer than at 132).  Remembered per shape (per thread).
inline int dgrad_ds_stride(const ConvParams& p, int NS)
{
    struct Entry { int H, W, K, S, NS, dstr; };
    constexpr int NCACHE = 64;
    static thread_local Entry cache[NCACHE];
    static thread_local int next = 0;
    for (const Entry& e : cache)
        if (e.H == p.H && e.W == p.W && e.K == p.K && e.S == p.S && e.NS == NS && e.dstr > 0) return e.dstr;
    int best = DG_TM + 4, best_cost = INT_MAX;
    for (int i = 0; i < 4; ++i) {
        const int dstr = DG_TM + 4 + 8 * i;
        const int cost = dgrad_gather_wavefronts(p, NS, dstr);
        if (cost < best_cost) {
            best_cost = cost;
            best = dstr;
        }
    }
    cache[next] = Entry{p.H, p.W, p.K, p.S, NS, best};
    next = (next + 1) % NCACHE;
    return best;
}

// Byte stride of the sample blocks of the staged G build (a block: gch channels x P positions
// of one sample, `bytes` long): `bytes` plus 0-28 pad words in steps of 16 bytes, at most
// `max_st`, the one whose reads by the formatter warps (lane = column (sample, position), one
// channel at a time) hit the fewest words per bank; 0 if none fits.
inline int dgrad_stage_stride(int P, int es, int bytes, int max_st)
{
    int best = 0, best_cost = INT_MAX;
    for (int pad = 0; pad < 32; pad += 4) {
        const int st = bytes + 4 * pad;
        if (st > max_st) break;
        int cost = 0;
        for (int w0 = 0; w0 < 128; w0 += 32) {
            int word[32], n = 0, bank_words[32] = {0};
            for (int l = w0; l < w0 + 32; ++l) {
                const int wd = ((l / P) * st + (l % P) * es) / 4;
                bool seen = false;
                for (int i = 0; i < n && !seen; ++i) seen = word[i] == wd;
                if (!seen) {
                    word[n++] = wd;
                    ++bank_words[wd & 31];
                }
            }
            int wf = 0;
            for (int b = 0; b < 32; ++b) wf = std::max(wf, bank_words[b]);
            cost += wf;
        }
        if (cost < best_cost) {
            best_cost = cost;
            best = st;
        }
    }
    return best;
}

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
    g.dcols = g.KTp;
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
    g.packed = 0;
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
    g.dstr = g.taps <= DG_TMAX ? dgrad_ds_stride(p, g.NS) : DG_TM + 4;
    // Staged G build, where a warp's 32 columns span 8 or more samples (P <= 4), so that the
    // strided loads of build_g touch a line per sample for a few bytes each (layer 2 of the
    // PufferLib PR #522 encoder, P = 2, B = 1024: d_input 23.4 -> 21.3 us fp32, 21.1 -> 19.1 us
    // bf16; layer 1, P = 12, gained nothing in fp32 and lost 2 us in bf16): the fewest channel
    // blocks (up to 4) whose dy (and y) slabs for a whole sample tile fit in the Ds rows, each
    // block a whole number of 16-channel groups per formatter quarter, every slab a run of whole
    // 16-byte units.
    g.grounds = 0;
    g.gstride = 0;
    const int es = int(sizeof(T));
    for (int r = 1; r <= 4 && g.grounds == 0 && p.P <= 4 && p.OC == g.nch * Tr::KC; ++r) {
        if (p.OC % (64 * r) != 0) continue;
        const int bytes = p.OC / r * p.P * es;
        if (bytes % 16 != 0 || (p.OCP * es) % 16 != 0) continue;
        const int st = dgrad_stage_stride(p.P, es, bytes, DG_TM * g.dstr * 4 / (g.NS * (p.relu ? 2 : 1)));
        if (st == 0) continue;
        g.grounds = r;
        g.gstride = st;
    }
    return g;
}

// Raw w slots of the weight formatters (none on the workspace path).
template <typename T>
inline __host__ __device__ int dgrad_wraw_bytes(const TcDgradGeom& g)
{
    return g.packed ? 0 : DG_NWF * WRAW * dgrad_wraw_warp_bytes<T>(g.KTp);
}

template <typename T>
inline int dgrad_smem(const ConvParams& p, const TcDgradGeom& g)
{
    return 1024 + g.nw * g.w_tile + dgrad_wraw_bytes<T>(g) + DG_TM * (g.dstr + 1) * 4 + (p.H + p.W) * (1 + g.rmax) * 8 +
           16 + p.HW * DG_PROW * 4 + int(sizeof(DgBars)) + 16;
}

// Compile-time constants of the col2im gather (K*K, H*W, CIC; 0: read from the parameters).
// SH = 1: 11x15 input, K = 5, S = 3, CIC = 5 for 128-row k-tiles -- layer 1 of the PufferLib
// PR #522 encoder, where the gather sets the pace (B = 1024: fp32 51.9 -> 49.9 us, bf16 45.8 ->
// 41.8 us).  Its layer 2 (two k-tiles per sample tile, bound by building G) gains nothing from it.
template <int SH> struct DgShape { static constexpr int KK = 0, HW = 0, CIC = 0; };
template <> struct DgShape<1> { static constexpr int KK = 25, HW = 165, CIC = 5; };

inline int dgrad_shape(const ConvParams& p, const TcDgradGeom& g)
{
    if (g.taps > DG_TMAX) return 0;
    if (p.KK == DgShape<1>::KK && p.HW == DgShape<1>::HW && g.CIC == DgShape<1>::CIC) return 1;
    return 0;
}

// The d_input CTA's work: work items item0, item0 + istride, ... (see wgrad_tc_body).
template <typename T, bool RELU, int SH>
__device__ __forceinline__ void dgrad_tc_body(const ConvParams& p, const T* __restrict__ dy, const T* __restrict__ w,
                                              const unsigned char* __restrict__ wpack, const T* __restrict__ y,
                                              T* __restrict__ dx, const TcDgradGeom& geo, const int item0,
                                              const int istride)
{
    using Tr = TcTraits<T>;
    constexpr int ES = int(sizeof(T));
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = align1024(smem_raw);
    // Layout: weight stages | raw w slots (DG_NWF warps x WRAW) | Ds | row, column, pixel tap tables | barriers
    unsigned char* wring = smem;
    unsigned char* wraw = wring + geo.nw * geo.w_tile;
    float* Ds = reinterpret_cast<float*>(wraw + dgrad_wraw_bytes<T>(geo));
    const int R1 = 1 + geo.rmax;
    const int dstr = geo.dstr;
    int2* rtab = reinterpret_cast<int2*>(Ds + DG_TM * dstr + DG_TM);  // after the zero row
    int2* ctab = rtab + p.H * R1;
    // Per input pixel hw: its contributing (p, kh*K + kw) as Ds offsets p*DSTR + kh*K + kw,
    // then the count (only used when every pixel has <= DG_TMAX taps).
    int* ptab = reinterpret_cast<int*>((reinterpret_cast<uintptr_t>(ctab + p.W * R1) + 15) & ~uintptr_t(15));
    DgBars* bars = reinterpret_cast<DgBars*>(ptab + p.HW * DG_PROW);
    volatile int* abort_flag = &bars->abort_flag;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid < DG_TM) Ds[DG_TM * dstr + tid] = 0.f;
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
                    ptab[hw * DG_PROW + n++] = (rr[a].x + cc[bq].x) * dstr + rr[a].y + cc[bq].y;
            for (int i = n; i < DG_TMAX; ++i) ptab[hw * DG_PROW + i] = -1;
            ptab[hw * DG_PROW + DG_TMAX] = n;
        }
    }
    if (tid == 0) {
        for (int i = 0; i < geo.nw; ++i) {
            mbar_init(smem_u32(&bars->w_full[i]), geo.packed ? 1 : DG_NWF);
            mbar_init(smem_u32(&bars->w_empty[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&bars->a_full[i]), DG_FMTW);
            mbar_init(smem_u32(&bars->a_empty[i]), 1);
            mbar_init(smem_u32(&bars->acc_full[i]), 1);
            mbar_init(smem_u32(&bars->acc_empty[i]), DG_FMTW);
        }
        mbar_init(smem_u32(&bars->fbar), DG_FMTW);
        mbar_init(smem_u32(&bars->gbar), 1);
        fence_mbar_init();
        bars->abort_flag = 0;
    }
    if (warp == 0) tmem_alloc(smem_u32(&bars->tslot), 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tslot;
    // Nothing above touches global memory: the previous kernel on the stream may still run.
    grid_dep_wait();
    // Work item wi = (sample tile wi % ntiles, k-tile range wi / ntiles).
    const int nwork = geo.ntiles * geo.ktsplit;
    auto ktrange = [&](int wi, int& lo, int& hi) {
        lo = (wi / geo.ntiles) * geo.kt_per;
        hi = min(geo.nkt, lo + geo.kt_per);
    };

    if (warp >= DG_WF0 && warp < DG_WF0 + DG_NWF && geo.packed) {
        // ---------------- W^T stages from the packed image (workspace path) ----------------
        if (warp == DG_WF0 && lane == 0) {
            RingPos wp;
            bool ok = true;
            for (int wi = item0; wi < nwork && ok && !*abort_flag; wi += istride) {
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
    } else if (warp >= DG_WF0 && warp < DG_WF0 + DG_NWF) {
        // ---------------- weight formatters ----------------
        // The warp's tile sequence (work item, k-tile, oc chunk); the copies of the next tile
        // are in flight while the current one is formatted.
        const int wf = warp - DG_WF0;
        const uint32_t w_u32 = smem_u32(wring), lo_off = uint32_t(geo.KTp * ROWB);
        const uint32_t slot_bytes = uint32_t(dgrad_wraw_warp_bytes<T>(geo.KTp));
        const uint32_t slot0 = smem_u32(wraw) + uint32_t(wf * WRAW) * slot_bytes;
        struct Seq { int wi, kt, kt_hi, ch; };
        auto first = [&](Seq& s, int wi) -> bool {
            if (wi >= nwork) return false;
            int lo;
            ktrange(wi, lo, s.kt_hi);
            s.wi = wi;
            s.kt = lo;
            s.ch = 0;
            return true;
        };
        auto advance = [&](Seq& s) -> bool {
            if (++s.ch < geo.nch) return true;
            s.ch = 0;
            return ++s.kt < s.kt_hi || first(s, s.wi + istride);
        };
        auto k0_of = [&](const Seq& s) { return s.kt * geo.CIC * p.KK; };
        Seq cur;
        bool have = first(cur, item0);
        if (have) stage_wt_dgrad<T>(slot0, w, p, k0_of(cur), cur.ch * Tr::KC, geo.KTp, wf, lane);
        cp_async_commit();
        uint32_t slot = 0;
        RingPos wp;
        while (have && !*abort_flag) {
            Seq nxt = cur;
            const bool have_nxt = advance(nxt);
            if (have_nxt)
                stage_wt_dgrad<T>(slot0 + (slot ^ 1u) * slot_bytes, w, p, k0_of(nxt), nxt.ch * Tr::KC, geo.KTp, wf,
                                  lane);
            cp_async_commit();
            cp_async_wait<1>();  // this lane's copies of the current tile have landed
            __syncwarp();        // ... and every lane's are visible to the warp
            if (wp.wrapped && !mbar_wait_or_abort(smem_u32(&bars->w_empty[wp.i]), wp.ph ^ 1u, abort_flag)) {
                report(const_cast<int*>(abort_flag), 16u);
                break;
            }
            const int mrows = min(geo.CIC, p.IC - cur.kt * geo.CIC) * p.KK;
            format_wt_dgrad<T>(w_u32 + uint32_t(wp.i * geo.w_tile), lo_off, slot0 + slot * slot_bytes, p, k0_of(cur),
                               mrows, cur.ch * Tr::KC, geo.KTp, wf, lane);
            fence_proxy_async_smem();  // the generic-proxy stores, for the tensor core
            __syncwarp();              // also: every lane is done reading this raw slot
            if (lane == 0) mbar_arrive(smem_u32(&bars->w_full[wp.i]));
            wp.next(geo.nw);
            cur = nxt;
            have = have_nxt;
            slot ^= 1u;
        }
        cp_async_wait<0>();  // no copy may land after the CTA's shared memory is released
    } else if (warp == DG_MMA_WARP) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            const uint32_t idesc1 = instr_desc(Tr::fmt, DG_TM, geo.KTp);
            const uint32_t w_u32 = smem_u32(wring), lo_off = uint32_t(geo.KTp * ROWB);
            RingPos wp, abp, dbp;
            bool ok = true;
            for (int wi = item0; wi < nwork && ok && !*abort_flag; wi += istride, abp.next(geo.nab)) {
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
                            const uint64_t bd = op_desc<1>(wa + kstep_off<1>(j));
                            const uint32_t first = (ch == 0 && j == 0) ? 0u : 1u;
                            const uint32_t col = uint32_t(ch * 32 + 8 * j);  // oc columns of this step
                            if constexpr (Tr::split) {
                                const uint64_t bl = op_desc<1>(wa + lo_off + kstep_off<1>(j));
                                const uint32_t glo = ga + uint32_t(geo.nch * Tr::KC) + col;
                                mma_tf32_ta(acc, ga + col, bd, idesc1, first);  // hi*hi
                                mma_tf32_ta(acc, ga + col, bl, idesc1, 1u);     // hi*lo
                                mma_tf32_ta(acc, glo, bd, idesc1, 1u);          // lo*hi
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
    } else if (warp >= DG_FMT0 / 32) {
        // ---------------- formatters + col2im ----------------
        const int ft = tid - DG_FMT0;       // 0 .. 511
        const uint32_t ds_u32 = smem_u32(Ds);
        const int fw = warp - DG_FMT0 / 32; // 0 .. 15
        const int qd = warp & 3;            // TMEM lane quarter
        const int sub = fw >> 2;            // quarter of the oc range (G) / of the k range (D)
        const int m = qd * 32 + lane;       // column within the tile
        const uint32_t lane_bits = uint32_t(qd * 32) << 16;
        const int ocq = geo.nch * Tr::KC / 4;  // output channels per formatter warp
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
        // G values of channels [o0, o0 + nb) (nb = 8 or 16) of this thread's column into the G
        // buffer at TMEM column gcol: tf32 hi and lo parts (fp32) or bf16 pairs.
        auto store_g16 = [&](uint32_t gcol, int o0, int nb, const float* v) {
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
                uint32_t wv[8];
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    wv[e] = uint32_t(__bfloat16_as_ushort(__float2bfloat16_rn(v[2 * e]))) |
                            (uint32_t(__bfloat16_as_ushort(__float2bfloat16_rn(v[2 * e + 1]))) << 16);
                tmem_st8(gcol + uint32_t(o0 / 2), wv);
            }
        };
        // Staged build of the CTA's first sample tile (the Ds rows are not in use yet): per
        // block of gch = OC / grounds channels, formatter warp 0 bulk-copies each sample's
        // contiguous dy (and y) slab of the block into the Ds rows (sample blocks gstride bytes
        // apart, the y slabs after the dy slabs), and every formatter thread reads its column's
        // gch / 4 channels from there.  The same values as build_g, in whole-tile copies
        // instead of strided 4-byte loads.
        uint32_t gph = 0;
        auto build_g_staged = [&](int tile, const RingPos& ab) -> bool {
            tc_fence_after();
            const int b0 = tile * geo.NS, ns = min(geo.NS, p.B - b0);
            const bool valid = m < ns * p.P;
            uint32_t si = 0, pq = 0;
            p.dm_P.divmod(uint32_t(valid ? m : 0), si, pq);
            const int gch = p.OC / geo.grounds, gq = gch / 4;
            const int bytes = gch * p.P * ES;
            const uint32_t ybase = ds_u32 + uint32_t(ns * geo.gstride);
            const uint32_t mine = uint32_t(int(si) * geo.gstride + int(pq) * ES);
            const uint32_t gcol = tmem + lane_bits + uint32_t(geo.acol0 + ab.i * geo.acols);
            const uint32_t gbar = smem_u32(&bars->gbar);
            for (int r = 0; r < geo.grounds; ++r) {
                if (ft < 32) {
                    if (ft == 0) mbar_arrive_expect_tx(gbar, uint32_t(ns * bytes * (RELU ? 2 : 1)));
                    __syncwarp();
                    for (int sI = ft; sI < ns; sI += 32) {
                        const size_t e0 = size_t(b0 + sI) * p.OCP + size_t(r) * gch * p.P;
                        bulk_g2s(ds_u32 + uint32_t(sI * geo.gstride), dy + e0, uint32_t(bytes), gbar);
                        if (RELU) bulk_g2s(ybase + uint32_t(sI * geo.gstride), y + e0, uint32_t(bytes), gbar);
                    }
                }
                if (!mbar_wait_or_abort(gbar, gph, abort_flag)) {
                    report(const_cast<int*>(abort_flag), 1u);
                    return false;
                }
                gph ^= 1u;
                for (int c0 = sub * gq; c0 < (sub + 1) * gq; c0 += 16) {
                    float v[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const uint32_t a = mine + uint32_t((c0 + e) * p.P * ES);
                        float d = 0.f;
                        if (valid) {
                            d = ES == 4 ? __uint_as_float(lds32(ds_u32 + a)) : __uint_as_float(lds16(ds_u32 + a) << 16);
                            if (RELU) {
                                const float yv = ES == 4 ? __uint_as_float(lds32(ybase + a))
                                                         : __uint_as_float(lds16(ybase + a) << 16);
                                if (!(yv > 0.f)) d = 0.f;
                            }
                        }
                        v[e] = d;
                    }
                    store_g16(gcol, r * gch + c0, 16, v);
                }
                if (!fmt_sync()) return false;  // the block's slabs are consumed
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bars->a_full[ab.i]));
            return true;
        };
        // G rows of sample tile `tile` into G buffer `ab`: dy (masked) of column m, channels
        // [sub*ocq, (sub+1)*ocq); zeros past the batch or past OC.
        auto build_g = [&](int tile, const RingPos& ab) -> bool {
            const int b0 = tile * geo.NS, ns = min(geo.NS, p.B - b0);
            const bool valid = m < ns * p.P;
            uint32_t si = 0, pq = 0;
            p.dm_P.divmod(uint32_t(valid ? m : 0), si, pq);
            const size_t base = (size_t(b0) + si) * p.OCP + pq;  // si = 0, pq = 0 for invalid lanes
            if (ab.wrapped && !mbar_wait_or_abort(smem_u32(&bars->a_empty[ab.i]), ab.ph ^ 1u, abort_flag)) {
                report(const_cast<int*>(abort_flag), 1u);
                return false;
            }
            tc_fence_after();
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
                store_g16(gcol, o0, min(16, (sub + 1) * ocq - o0), v);  // multiple of 8 (fp32) / 16 (bf16)
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bars->a_full[ab.i]));
            return true;
        };
        RingPos abp, dbp;
        bool ok = true;
        const int first = item0;
        // (Staging needs P <= 4: not compiled into the instances for a named shape.)
        const bool staged = SH == 0 && geo.grounds > 0 &&
                            ((reinterpret_cast<uintptr_t>(dy) | (RELU ? reinterpret_cast<uintptr_t>(y) : 0)) & 15) == 0;
        if (first < nwork) {
            if constexpr (SH == 0) ok = staged ? build_g_staged(first % geo.ntiles, abp) : build_g(first % geo.ntiles, abp);
            else ok = build_g(first % geo.ntiles, abp);
        }
        for (int wi = first; wi < nwork && ok; wi += istride) {
            const int tile = wi % geo.ntiles;
            int kt_lo, kt_hi;
            ktrange(wi, kt_lo, kt_hi);
            RingPos nab = abp;
            nab.next(geo.nab);
            const int next = wi + istride;
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
                    const uint32_t drow = ds_u32 + uint32_t((m * dstr + c0) * 4);
                    for (int c = 0; c < kq; c += 16) {
                        const bool two = c + 8 < kq;
                        uint32_t r[2][8];
                        tmem_ld8(acc + uint32_t(c0 + c), r[0]);
                        if (two) tmem_ld8(acc + uint32_t(c0 + c + 8), r[1]);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 2; ++i) {
                            if (i == 1 && !two) break;
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
                    // stay in registers while it walks the k-tile's channels.  Absent taps read
                    // the zero row past the Ds rows (as long as a k-tile's K*K*CIC words), so
                    // every tap moves by one channel's K*K words.  For the shapes DgShape names,
                    // K*K, H*W and CIC are constants: the channel loop unrolls with fixed load
                    // and store offsets.
                    constexpr int KKc = DgShape<SH>::KK, HWc = DgShape<SH>::HW, CICc = DgShape<SH>::CIC;
                    const int KK = KKc ? KKc : p.KK, HW = HWc ? HWc : p.HW;
                    const int nsplit = max(1, DG_NFT / HW);
                    const uint32_t zrow = ds_u32 + uint32_t(DG_TM * dstr * 4);
                    for (int it = ft; it < HW * nsplit; it += DG_NFT) {
                        const int hw = it % HW, part = it / HW;
                        const int4 o = *reinterpret_cast<const int4*>(ptab + hw * DG_PROW);
                        for (int sI = part; sI < ns; sI += nsplit) {
                            T* dxs = dx + size_t(b0 + sI) * p.IHW + size_t(ic0) * HW + hw;
                            const uint32_t ds = ds_u32 + uint32_t(sI * p.P * dstr * 4);
                            uint32_t a0 = o.x >= 0 ? ds + uint32_t(o.x * 4) : zrow;
                            uint32_t a1 = o.y >= 0 ? ds + uint32_t(o.y * 4) : zrow;
                            uint32_t a2 = o.z >= 0 ? ds + uint32_t(o.z * 4) : zrow;
                            uint32_t a3 = o.w >= 0 ? ds + uint32_t(o.w * 4) : zrow;
                            if (CICc > 0 && nic == CICc) {
#pragma unroll
                                for (int icl = 0; icl < (CICc > 0 ? CICc : 1); ++icl) {
                                    const uint32_t off = uint32_t(icl * KK * 4);
                                    const float v0 = __uint_as_float(lds32(a0 + off));
                                    const float v1 = __uint_as_float(lds32(a1 + off));
                                    const float v2 = __uint_as_float(lds32(a2 + off));
                                    const float v3 = __uint_as_float(lds32(a3 + off));
                                    Elem<T>::st(dxs + icl * HW, ((v0 + v1) + v2) + v3);
                                }
                            } else {
                                const uint32_t kstep = uint32_t(KK * 4);
#pragma unroll 4
                                for (int icl = 0; icl < nic; ++icl) {
                                    const float v0 = __uint_as_float(lds32(a0)), v1 = __uint_as_float(lds32(a1));
                                    const float v2 = __uint_as_float(lds32(a2)), v3 = __uint_as_float(lds32(a3));
                                    Elem<T>::st(dxs, ((v0 + v1) + v2) + v3);
                                    dxs += HW;
                                    a0 += kstep;
                                    a1 += kstep;
                                    a2 += kstep;
                                    a3 += kstep;
                                }
                            }
                        }
                    }
                } else {
                    const int span = nic * p.HW;
                    for (int sI = 0; sI < ns; ++sI) {
                        T* dxs = dx + size_t(b0 + sI) * p.IHW + size_t(ic0) * p.HW;
                        const float* ds = Ds + sI * p.P * dstr;
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
                                    sum += ds[(rr[a].x + cc[bq].x) * dstr + kb + rr[a].y + cc[bq].y];
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

template <typename T, bool RELU, int SH>
__global__ void __launch_bounds__(DG_THREADS, 1)
dgrad_tc_kernel(const ConvParams p, const T* __restrict__ dy, const T* __restrict__ w,
                const unsigned char* __restrict__ wpack, const T* __restrict__ y, T* __restrict__ dx,
                const TcDgradGeom geo)
{
    dgrad_tc_body<T, RELU, SH>(p, dy, w, wpack, y, dx, geo, int(blockIdx.x), int(gridDim.x));
}

// ======================================================================================
// Fused backward: d_input and wgrad in one launch, one work item per CTA.  CTAs [0, n_wg) run
// one wgrad tile each (the long items, started first); the CTAs after them run d_input's work
// items, cut into k-tile ranges (disjoint dx channels: no reduction) so that they are short.
// The block scheduler starts the CTAs in index order as SMs free up, so the short d_input items
// fill the SMs the wgrad tiles leave idle and backfill the others as the wgrad tiles finish.
// Both operations compute exactly as in their own kernels.
// ======================================================================================
static_assert(DG_THREADS == WG_THREADS, "one block shape for both operations");

template <typename T, bool RELU, bool GT, int SH>
__global__ void __launch_bounds__(DG_THREADS, 1)
bwd_tc_kernel(const ConvParams p, const T* __restrict__ x, const T* __restrict__ dy, const T* __restrict__ w,
              const unsigned char* __restrict__ wpack, const T* __restrict__ y, T* __restrict__ dx,
              float* __restrict__ ws, float* __restrict__ bpart, const TcDgradGeom dgeo, const TcWgradGeom wgeo,
              const int n_wg)
{
    if (int(blockIdx.x) < n_wg) {
        if constexpr (GT) wgrad_tc_body_gt<T, RELU>(p, x, dy, y, ws, bpart, wgeo, int(blockIdx.x), n_wg);
        else wgrad_tc_body<T, RELU>(p, x, dy, y, ws, bpart, wgeo, int(blockIdx.x), n_wg);
    } else
        dgrad_tc_body<T, RELU, SH>(p, dy, w, wpack, y, dx, dgeo, int(blockIdx.x) - n_wg, int(gridDim.x) - n_wg);
}

// ======================================================================================
// Two-layer forward chain: y1 = act1(conv1(x) + b1), y2 = act2(conv2(y1) + b2), where conv2's
// input is conv1's output (IC2 = OC1, H2 x W2 = OH1 x OW1) -- the encoder of PufferLib PR #522
// (layer 1 -> 3x4 -> layer 2).  A work item is a group of NS whole samples (NS*P1 <= 128
// layer-1 columns).  Phase 1 is layer 1's forward tile for the group, as in fwd_tc_kernel
// (gathered patches in TMEM, weight stages bulk-copied from the packed W1 image); its epilogue
// writes y1 to global memory (the backward needs it) and into a shared-memory slab laid out as
// conv2's NCHW input.  Phase 2 is layer 2's forward for the same samples, with the operands'
// roles swapped because the group has only NS*P2 columns (20 for the encoder): W2 is the TMEM
// operand (M = 128 output channels) -- the weight producer bulk-copies its packed chunks into
// the weight ring, well ahead, and the formatter warps move each landed chunk's rows into TMEM
// -- and the group's layer-2 patches, gathered from the slab into a small ring of patch stages
// (one per TMEM operand stage, released with it), are the shared-memory operand (N = N2p, the
// columns rounded up to 16).  y1 never makes a round trip through memory between the layers,
// layer 2 needs no launch of its own and its MMAs are N2p wide instead of 128.
// Warp roles (608 threads): warp 0 x producer (phase 1), warp 1 weight producer (W1 chunks,
// then W2 chunks), warp 2 MMA, warps 3-18 formatters (phase 1: gather + epilogue; phase 2: W2
// rows into TMEM, patch stages, epilogue).
// ======================================================================================
constexpr int CH_THREADS = 96 + 32 * FA_FMTW;

struct ChainGeom {
    FwdGeom g1;              // layer 1 (tile = NS*P1 columns, OTp1 rows); nw / nraw / xg of the ring
    int ns, ngroups;         // samples per group, groups
    int OTp2, oc_tiles2;     // layer 2 output channels (a single tile: the TMEM lanes)
    int N2p;                 // layer 2 columns of a group, rounded up to 16 (the MMA's N)
    int nchunks2;            // layer 2 K-chunks
    int w_bytes2;            // one layer-2 weight stage
    int stage_bytes;         // weight ring stage = max(w_bytes1, w_bytes2)
    int patch_bytes;         // one patch stage (N2p rows x 128 bytes, x2 for fp32); na of them
    int dcols;               // accumulator columns = max of the two layers'
    int acol0;               // first TMEM column of the operand stages
    int xs2;                 // bytes per sample in the y1 slab
    int slab_bytes;
    size_t wpack2_off;       // byte offset of the packed W2 image in the workspace
    int relu1, relu2;
};

struct ChainBars {
    uint64_t raw_full[FV_MAXRAWS], raw_empty[FV_MAXRAWS];
    uint64_t w_full[FA_MAXW], w_empty[FA_MAXW];
    uint64_t a_full[FA_MAXA], a_empty[FA_MAXA];
    uint64_t acc_full, acc_empty;
    uint64_t slab_full;      // the 16 formatter warps' y1 slab writes of the current group
    uint32_t tslot;
    int abort_flag;
};

template <typename T>
inline int chain_smem(const ConvParams& p1, const ConvParams& p2, const ChainGeom& c)
{
    using Tr = TcTraits<T>;
    return 1024 + c.g1.nw * c.stage_bytes + c.g1.nraw * c.g1.raw_bytes + 1024 + c.g1.na * c.patch_bytes + c.slab_bytes +
           round_up(p1.Kred, Tr::KC) * 4 + round_up(p2.Kred, Tr::KC) * 4 + int(sizeof(ChainBars)) + 16;
}

template <typename T>
__global__ void __launch_bounds__(CH_THREADS, 1)
fwd_chain_kernel(const ConvParams p1, const ConvParams p2, const T* __restrict__ x,
                 const unsigned char* __restrict__ wpack, const T* __restrict__ bias1,
                 const T* __restrict__ bias2, T* __restrict__ y1, T* __restrict__ y2, const ChainGeom cg)
{
    using Tr = TcTraits<T>;
    constexpr int ES = int(sizeof(T));
    constexpr int KQ = Tr::KC / FA_KSPLIT;
    constexpr int KQC = Tr::split ? KQ : KQ / 2;
    static_assert(KQC == 8, "one tcgen05.st of 8 columns per part");
    const FwdGeom& g1 = cg.g1;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = align1024(smem_raw);
    const int kred1 = round_up(p1.Kred, Tr::KC), kred2 = round_up(p2.Kred, Tr::KC);
    // Layout: weight stages | raw x slots | patch stages | y1 slab | k offsets (layer 1, layer 2) | barriers
    unsigned char* wring = smem;
    unsigned char* raw = wring + g1.nw * cg.stage_bytes;
    unsigned char* pring = align1024(raw + g1.nraw * g1.raw_bytes);  // swizzled MMA operand: 1024-aligned
    unsigned char* slab = pring + g1.na * cg.patch_bytes;
    int* offk1 = reinterpret_cast<int*>(slab + cg.slab_bytes);
    int* offk2 = offk1 + kred1;
    ChainBars* bars = reinterpret_cast<ChainBars*>(offk2 + kred2);
    volatile int* abort_flag = &bars->abort_flag;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    for (int k = tid; k < kred1; k += CH_THREADS) {
        const int sc_ic = (k / (g1.xg * Tr::KC)) * g1.xg * Tr::KC / p1.KK;
        offk1[k] = (k < p1.Kred) ? (k_offset(p1, k) - sc_ic * p1.HW) * ES : 0;
    }
    for (int k = tid; k < kred2; k += CH_THREADS) offk2[k] = (k < p2.Kred) ? k_offset(p2, k) * ES : 0;
    if (tid == 0) {
        for (int i = 0; i < g1.nraw; ++i) {
            mbar_init(smem_u32(&bars->raw_full[i]), 1);
            mbar_init(smem_u32(&bars->raw_empty[i]), FA_FMTW);
        }
        for (int i = 0; i < g1.nw; ++i) {
            mbar_init(smem_u32(&bars->w_full[i]), 1);
            mbar_init(smem_u32(&bars->w_empty[i]), 1);
        }
        for (int i = 0; i < g1.na; ++i) {
            mbar_init(smem_u32(&bars->a_full[i]), FA_FMTW);
            mbar_init(smem_u32(&bars->a_empty[i]), 1);
        }
        mbar_init(smem_u32(&bars->acc_full), 1);
        mbar_init(smem_u32(&bars->acc_empty), FA_FMTW);
        mbar_init(smem_u32(&bars->slab_full), FA_FMTW);
        fence_mbar_init();
        bars->abort_flag = 0;
    }
    if (warp == 0) tmem_alloc(smem_u32(&bars->tslot), FA_TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tslot;
    grid_dep_wait();  // the packed weights come from the kernels launched just before

    if (warp == 0) {
        // ---------------- x producer (phase 1) ----------------
        const unsigned char* xb = reinterpret_cast<const unsigned char*>(x);
        const unsigned char* x_end = xb + size_t(p1.B) * p1.IHW * ES;
        RingPos rp;
        for (int grp = blockIdx.x; grp < cg.ngroups && !*abort_flag; grp += gridDim.x) {
            const int b_first = grp * cg.ns, nsamp = min(cg.ns, p1.B - b_first);
            for (int sc = 0; sc < (g1.nchunks + g1.xg - 1) / g1.xg; ++sc, rp.next(g1.nraw)) {
                const int s = rp.i;
                if (rp.wrapped && !mbar_wait_or_abort(smem_u32(&bars->raw_empty[s]), rp.ph ^ 1u, abort_flag)) {
                    report(const_cast<int*>(abort_flag), 4u);
                    break;
                }
                const int sk0 = sc * g1.xg * Tr::KC;
                const int ic_lo = sk0 / p1.KK;
                const int ic_hi = min(p1.IC - 1, (min(sk0 + g1.xg * Tr::KC, p1.Kred) - 1) / p1.KK);
                const int need = (ic_hi - ic_lo + 1) * p1.HW * ES;
                unsigned char* slot = raw + s * g1.raw_bytes;
                auto piece = [&](int j, const unsigned char*& src, int& bulk) {
                    const unsigned char* s0 = xb + (size_t(b_first + j) * p1.IHW + size_t(ic_lo) * p1.HW) * ES;
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
                    for (const unsigned char* t = src + bulk; t < src + bytes && t < x_end; ++t)
                        slot[j * g1.xs + int(t - src)] = *t;
                    tx += bulk;
                }
                tx = warp_sum(tx);
                __syncwarp();
                if (lane == 0) mbar_arrive_expect_tx(smem_u32(&bars->raw_full[s]), uint32_t(tx));
                __syncwarp();
                for (int j = lane; j < nsamp; j += 32) {
                    const unsigned char* src;
                    int bulk;
                    piece(j, src, bulk);
                    if (bulk > 0)
                        bulk_g2s(smem_u32(slot + j * g1.xs), src, uint32_t(bulk), smem_u32(&bars->raw_full[s]));
                }
            }
        }
    } else if (warp == 1) {
        // ---------------- weight producer: W1 chunks, then W2 chunks, per group ----------------
        if (lane == 0) {
            RingPos wp;
            bool ok = true;
            for (int grp = blockIdx.x; grp < cg.ngroups && ok && !*abort_flag; grp += gridDim.x) {
                for (int ph = 0; ph < 2 && ok; ++ph) {  // W1 chunks, then W2 chunks
                    const int n = ph == 0 ? g1.nchunks : cg.nchunks2;
                    const int wb = ph == 0 ? g1.w_bytes : cg.w_bytes2;
                    const unsigned char* src = wpack + (ph == 0 ? size_t(0) : cg.wpack2_off);
                    for (int kc = 0; kc < n; ++kc, wp.next(g1.nw), src += wb) {
                        if (wp.wrapped && !mbar_wait_or_abort(smem_u32(&bars->w_empty[wp.i]), wp.ph ^ 1u, abort_flag)) {
                            report(const_cast<int*>(abort_flag), 16u);
                            ok = false;
                            break;
                        }
                        const uint32_t bar = smem_u32(&bars->w_full[wp.i]);
                        mbar_arrive_expect_tx(bar, uint32_t(wb));
                        bulk_g2s(smem_u32(wring + wp.i * cg.stage_bytes), src, uint32_t(wb), bar);
                    }
                }
            }
        }
        __syncwarp();
    } else if (warp == 2) {
        // ---------------- MMA issuer: phase 1 then phase 2 of each group ----------------
        if (lane == 0) {
            const uint32_t w_u32 = smem_u32(wring);
            RingPos wp, ap;
            uint32_t t = 0;
            bool ok = true;
            for (int grp = blockIdx.x; grp < cg.ngroups && ok && !*abort_flag; grp += gridDim.x) {
                for (int ph = 0; ph < 2 && ok; ++ph, ++t) {
                    const int N = ph == 0 ? g1.OTp : cg.N2p;  // phase 2: the group's columns
                    const uint32_t idesc2 = instr_desc(Tr::fmt, FA_TM, Tr::split ? 2 * N : N);
                    const uint32_t idesc1 = instr_desc(Tr::fmt, FA_TM, N);
                    const int n = ph == 0 ? g1.nchunks : cg.nchunks2;
                    if (t >= 1 && !mbar_wait_or_abort(smem_u32(&bars->acc_empty), (t - 1) & 1, abort_flag)) {
                        report(const_cast<int*>(abort_flag), 8u);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    for (int kc = 0; kc < n; ++kc, wp.next(g1.nw), ap.next(g1.na)) {
                        if (!mbar_wait_or_abort(smem_u32(&bars->w_full[wp.i]), wp.ph, abort_flag) ||
                            !mbar_wait_or_abort(smem_u32(&bars->a_full[ap.i]), ap.ph, abort_flag)) {
                            report(const_cast<int*>(abort_flag), 8u);
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        // phase 1: B = the W1 chunk in the weight ring; phase 2: B = the patch stage
                        // (the W2 chunk in the weight ring was moved into the TMEM operand stage)
                        const uint32_t wa = ph == 0 ? w_u32 + wp.i * cg.stage_bytes
                                                    : smem_u32(pring) + uint32_t(ap.i * cg.patch_bytes);
                        const uint32_t aa = tmem + uint32_t(cg.acol0 + ap.i * g1.acols);
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const uint64_t bd = op_desc<1>(wa + kstep_off<1>(j));
                            const uint32_t acc = (kc == 0 && j == 0) ? 0u : 1u;
                            if constexpr (Tr::split) {
                                mma_tf32_ta(tmem, aa + 8 * j, bd, idesc2, acc);
                                mma_tf32_ta(tmem, aa + Tr::KC + 8 * j, bd, idesc1, 1u);
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
        }
        __syncwarp();
    } else if (warp >= 3) {
        // ---------------- formatters: gather + epilogue, both phases ----------------
        const int fw = warp - 3;
        const int qd = warp & 3;
        const int sub = fw >> 2;
        const int m = qd * 32 + lane;
        const uint32_t lane_bits = uint32_t(qd * 32) << 16;
        const uint32_t raw_u32 = smem_u32(raw), slab_u32 = smem_u32(slab);
        const uint32_t offk1_u32 = smem_u32(offk1) + uint32_t(sub * KQ * 4);
        RingPos ap, rp, wp;
        uint32_t t = 0, sph = 0;
        bool ok = true;
        const int ft = tid - 96;  // formatter thread 0 .. 511
        for (int grp = blockIdx.x; grp < cg.ngroups && ok; grp += gridDim.x) {
            const int b_first = grp * cg.ns, nsamp = min(cg.ns, p1.B - b_first);
            // ================= phase 1: layer 1's tile (gathered patches in TMEM) =================
            {
                const int cols = nsamp * p1.P;
                int boff, bmis;
                {
                    uint32_t bq, pq, oh, ow;
                    p1.dm_P.divmod(uint32_t(min(m, cols - 1)), bq, pq);
                    p1.dm_OW.divmod(pq, oh, ow);
                    boff = int(bq) * g1.xs + (int(oh) * p1.S * p1.W + int(ow) * p1.S) * ES;
                    bmis = int((size_t(b_first + int(bq)) * p1.IHW * ES) & 15);
                }
                const bool ragged_k = (p1.Kred % Tr::KC) != 0;
                uint32_t sbase = 0;
                int xc = 0;
                for (int kc = 0; kc < g1.nchunks; ++kc, ap.next(g1.na), wp.next(g1.nw)) {
                    if (xc == 0) {
                        if (!mbar_wait_or_abort(smem_u32(&bars->raw_full[rp.i]), rp.ph, abort_flag)) {
                            report(const_cast<int*>(abort_flag), 1u);
                            ok = false;
                            break;
                        }
                        const int ic_lo = (kc * Tr::KC) / p1.KK;
                        const int cmis = (ic_lo * p1.HW * ES) & 15;
                        sbase = raw_u32 + uint32_t(rp.i * g1.raw_bytes + boff + ((bmis + cmis) & 15));
                    }
                    if (ap.wrapped && !mbar_wait_or_abort(smem_u32(&bars->a_empty[ap.i]), ap.ph ^ 1u, abort_flag)) {
                        report(const_cast<int*>(abort_flag), 1u);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t oaddr = offk1_u32 + uint32_t(kc * Tr::KC * 4);
                    const uint32_t col = tmem + lane_bits + uint32_t(cg.acol0 + ap.i * g1.acols + sub * KQC);
                    const int kvalid = (ragged_k && kc == g1.nchunks - 1) ? p1.Kred - (kc * Tr::KC + sub * KQ) : KQ;
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
                    for (int e = 0; e < KQ; ++e)
                        v[e] = Tr::split ? lds32(sbase + uint32_t(o[e])) : lds16(sbase + uint32_t(o[e]));
                    if (kvalid < KQ) {
#pragma unroll
                        for (int e = 0; e < KQ; ++e)
                            if (e >= kvalid) v[e] = 0;
                    }
                    if constexpr (Tr::split) {
                        uint32_t hi[8], lo[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) split_tf32(v[e], hi[e], lo[e]);
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
                    const bool sc_end = (++xc == g1.xg) || kc == g1.nchunks - 1;
                    if (lane == 0) {
                        mbar_arrive(smem_u32(&bars->a_full[ap.i]));
                        if (sc_end) mbar_arrive(smem_u32(&bars->raw_empty[rp.i]));
                    }
                    if (sc_end) {
                        xc = 0;
                        rp.next(g1.nraw);
                    }
                }
                if (!ok) break;
                // Epilogue: TMEM -> bias -> activation -> y1 and the y1 slab.
                if (!mbar_wait_or_abort(smem_u32(&bars->acc_full), t & 1, abort_flag)) {
                    report(const_cast<int*>(abort_flag), 2u);
                    ok = false;
                    break;
                }
                tc_fence_after();
                T* yc = nullptr;
                uint32_t srow = 0;
                if (m < cols) {
                    yc = y1 + col_out(p1, b_first * p1.P + m);
                    uint32_t s1, q1;
                    p1.dm_P.divmod(uint32_t(m), s1, q1);
                    srow = slab_u32 + uint32_t(int(s1) * cg.xs2 + int(q1) * ES);  // + oc * P1 * ES
                }
                for (int cb = sub * 8; cb < g1.OTp; cb += 8 * FA_KSPLIT) {
                    uint32_t r[8];
                    tmem_ld8(tmem + lane_bits + uint32_t(cb), r);
                    if constexpr (Tr::split) {
                        uint32_t r2[8];
                        tmem_ld8(tmem + lane_bits + uint32_t(g1.OTp + cb), r2);
                        tmem_ld_wait();
#pragma unroll
                        for (int e = 0; e < 8; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) + __uint_as_float(r2[e]));
                    } else {
                        tmem_ld_wait();
                    }
                    if (yc) {
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const int oc = cb + e;
                            if (oc < p1.OC) {
                                float f = __uint_as_float(r[e]);
                                if (bias1) f += Elem<T>::ldg(bias1 + oc);
                                if (cg.relu1) f = f > 0.f ? f : 0.f;
                                Elem<T>::st(yc + size_t(oc) * p1.P, f);
                                // the slab holds exactly the value y1 holds (rounded to T)
                                const uint32_t a = srow + uint32_t(oc * p1.P * ES);
                                if constexpr (ES == 4) sts32(a, __float_as_uint(f));
                                else sts16(a, __bfloat16_as_ushort(__float2bfloat16_rn(f)));
                            }
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(smem_u32(&bars->acc_empty));
                    mbar_arrive(smem_u32(&bars->slab_full));  // this warp's slab writes are done
                }
                ++t;
            }
            // ================= phase 2: layer 2 (W2 rows in TMEM, patches in a ring slot) =================
            {
                const int cols = nsamp * p2.P;
                // the slab holds this group's y1: wait for every formatter warp's writes
                if (!mbar_wait_or_abort(smem_u32(&bars->slab_full), sph, abort_flag)) {
                    report(const_cast<int*>(abort_flag), 32u);
                    ok = false;
                    break;
                }
                sph ^= 1u;
                // W2 rows: this thread's row m (an output channel) and quarter `sub` of each chunk's K
                // -- two 16-byte units of the chunk in the weight ring (hi, and lo for fp32).
                const bool wrow = m < cg.OTp2;
                // Patch stage: this thread's 16-byte unit (row r = a layer-2 column, unit c) if ft < N2p*8.
                const int prow = ft >> 3, pc = ft & 7;
                const bool punit = ft < cg.N2p * 8;
                const bool pvalid = prow < cols;
                int pboff = 0;
                {
                    uint32_t s2, q2, oh, ow;
                    p2.dm_P.divmod(uint32_t(min(prow, cols - 1)), s2, q2);
                    p2.dm_OW.divmod(q2, oh, ow);
                    pboff = int(s2) * cg.xs2 + (int(oh) * p2.S * p2.W + int(ow) * p2.S) * ES;
                }
                const uint32_t pst = unit_off<1>(prow, pc);
                for (int kc = 0; kc < cg.nchunks2; ++kc, ap.next(g1.na), wp.next(g1.nw)) {
                    if (!mbar_wait_or_abort(smem_u32(&bars->w_full[wp.i]), wp.ph, abort_flag) ||
                        (ap.wrapped && !mbar_wait_or_abort(smem_u32(&bars->a_empty[ap.i]), ap.ph ^ 1u, abort_flag))) {
                        report(const_cast<int*>(abort_flag), 1u);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // (a) W2 rows: weight-ring slot -> TMEM operand stage (the columns phase 1's patches use)
                    const uint32_t col = tmem + lane_bits + uint32_t(cg.acol0 + ap.i * g1.acols + sub * KQC);
                    {
                        const uint32_t wslot = smem_u32(wring) + uint32_t(wp.i * cg.stage_bytes);
                        uint32_t hw[8] = {0, 0, 0, 0, 0, 0, 0, 0}, lw[8] = {0, 0, 0, 0, 0, 0, 0, 0};
                        if (wrow) {
#pragma unroll
                            for (int q = 0; q < 2; ++q) {
                                const int4 h = lds128(wslot + unit_off<1>(m, 2 * sub + q));
                                hw[4 * q] = h.x; hw[4 * q + 1] = h.y; hw[4 * q + 2] = h.z; hw[4 * q + 3] = h.w;
                                if constexpr (Tr::split) {
                                    const int4 l = lds128(wslot + uint32_t(cg.OTp2 * ROWB) + unit_off<1>(m, 2 * sub + q));
                                    lw[4 * q] = l.x; lw[4 * q + 1] = l.y; lw[4 * q + 2] = l.z; lw[4 * q + 3] = l.w;
                                }
                            }
                        }
                        tmem_st8(col, hw);
                        if constexpr (Tr::split) tmem_st8(col + Tr::KC, lw);
                    }
                    // (b) this chunk's patch stage (the one of TMEM operand stage ap.i): rows = the
                    // group's layer-2 columns (zero past `cols`), K-major, 128-byte swizzled; fp32 as
                    // hi rows then lo rows
                    if (punit) {
                        uint32_t pv[Tr::E];
                        const int k0 = kc * Tr::KC + pc * Tr::E;
#pragma unroll
                        for (int e = 0; e < Tr::E; ++e) {
                            const int k = k0 + e;
                            pv[e] = 0u;
                            if (pvalid && k < p2.Kred) {
                                const uint32_t a = slab_u32 + uint32_t(pboff) + uint32_t(lds32(smem_u32(offk2) + 4u * uint32_t(k)));
                                pv[e] = ES == 4 ? lds32(a) : lds16(a);
                            }
                        }
                        unsigned char* stage = pring + ap.i * cg.patch_bytes;
                        put_unit<T>(stage, stage + cg.N2p * ROWB, pst, pv);
                    }
                    fence_proxy_async_smem();  // the patch stage, for the tensor core
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&bars->a_full[ap.i]));  // W2 rows and patches ready
                }
                if (!ok) break;
                // Epilogue: lanes = output channels, columns = the group's layer-2 columns.
                if (!mbar_wait_or_abort(smem_u32(&bars->acc_full), t & 1, abort_flag)) {
                    report(const_cast<int*>(abort_flag), 2u);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int oc = m;
                const float bv = (bias2 && oc < p2.OC) ? Elem<T>::ldg(bias2 + oc) : 0.f;
                for (int cb = sub * 8; cb < cg.N2p; cb += 8 * FA_KSPLIT) {
                    uint32_t r[8];
                    tmem_ld8(tmem + lane_bits + uint32_t(cb), r);
                    if constexpr (Tr::split) {
                        uint32_t r2[8];
                        tmem_ld8(tmem + lane_bits + uint32_t(cg.N2p + cb), r2);
                        tmem_ld_wait();
#pragma unroll
                        for (int e = 0; e < 8; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) + __uint_as_float(r2[e]));
                    } else {
                        tmem_ld_wait();
                    }
                    if (oc < p2.OC) {
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const int n2 = cb + e;
                            if (n2 < cols) {
                                float f = __uint_as_float(r[e]) + bv;
                                if (cg.relu2) f = f > 0.f ? f : 0.f;
                                Elem<T>::st(y2 + col_out(p2, b_first * p2.P + n2) + size_t(oc) * p2.P, f);
                            }
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&bars->acc_empty));
                ++t;
            }
        }
    }
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, FA_TMEM_COLS);
    }
}

template <typename T> constexpr int dt_of_tc();
template <> constexpr int dt_of_tc<float>() { return DT_F32; }
template <> constexpr int dt_of_tc<__nv_bfloat16>() { return DT_BF16; }




}  // namespace

// Weight-ring depth, x super-chunk length and K ranges of the forward kernel: feasible
// (shared memory, including the K-range reduction's partial tile) and of the lowest estimated
// time (fwd_cost).  `packed`: the workspace path (weight stages bulk-copied from the packed
// image, no raw w slots).
template <typename T>
static bool pick_fwd(const ConvParams& p, const DevInfo& d, bool packed, FwdGeom& out)
{
    // Per list, the first that fits: the deepest weight ring, then the longest x super-chunk
    // (fewer, larger slab copies); or short super-chunks first, so that K splits into more
    // ranges.  Of the two, the lower estimated time (ties: the first list).
    // {weight stages, chunks per x super-chunk, raw x slots}
    // Three weight stages with a four-chunk x lookahead before four with two: layer 1 fp32 at
    // B = 1024 measured 43.8 us with {3, 4, 2} against 45.9 with {4, 2, 2} (x slabs from DRAM
    // arrive late with a two-chunk lookahead; two or three weight stages suffice).
    static const int cfgs[][3] = {{4, 8, 2}, {4, 6, 2}, {4, 4, 2}, {3, 4, 2}, {4, 2, 2}, {3, 2, 2}, {2, 2, 2},
                                  {2, 1, 2}};
    static const int cfgs_split[][3] = {{4, 2, 2}, {3, 2, 2}, {2, 2, 2}, {4, 1, 2}, {2, 1, 2}};
    bool found = false;
    double best = 0.0;
    for (int pass = 0; pass < 2; ++pass) {
        const int ncfg = pass == 0 ? 8 : 5;
        for (int i = 0; i < ncfg; ++i) {
            const int* c = pass == 0 ? cfgs[i] : cfgs_split[i];
            FwdGeom g = fwd_geom<T>(p, c[1], c[0], c[2]);
            g.packed = packed ? 1 : 0;
            if (g.na < 2 || fwd_smem<T>(p, g) > d.smem_optin) continue;
            const double t = fwd_set_splits(g, d.sms);
            if (!fwd_red_fits(g)) {
                g.splits = 1;
                g.kc_per = g.nchunks;
            }
            const double tt = g.splits > 1 ? t : fwd_cost(g.n_tiles * g.oc_tiles, d.sms, 1, g.nchunks);
            if (!found || tt < best) {
                out = g;
                best = tt;
                found = true;
            }
            break;
        }
    }
    return found;
}

bool tc_fwd_ok(const ConvParams& p, int dt, const DevInfo& d, bool packed)
{
    if (d.cc_major != 10 || p.N <= 0) return false;
    FwdGeom g;
    return dt == DT_BF16 ? pick_fwd<__nv_bfloat16>(p, d, packed, g) : pick_fwd<float>(p, d, packed, g);
}

Plan plan_fwd_tc(const ConvParams& p, int dt, const DevInfo& d, bool packed)
{
    FwdGeom g;
    if (dt == DT_BF16) pick_fwd<__nv_bfloat16>(p, d, packed, g);
    else pick_fwd<float>(p, d, packed, g);
    Plan pl;
    pl.algo = ALGO_TC;
    // one launch (weights formatted in the kernel, K ranges reduced inside each cluster); the
    // workspace path first packs the weights into the workspace
    pl.launches = packed ? 2 : 1;
    pl.block = FA_THREADS;
    pl.splits = g.splits;
    static_assert(FV_MAXRAWS < 8 && FA_MAXW < 16, "forward plan: ring depths in 3 and 4 bits");
    pl.variant = ((g.kc_per * 16 + g.xg) * 16 + g.nw) * 8 + g.nraw;  // xg <= 8
    pl.grid = g.splits > 1 ? g.n_tiles * g.oc_tiles * g.splits : std::min(g.n_tiles * g.oc_tiles, d.sms);
    pl.smem = dt == DT_BF16 ? fwd_smem<__nv_bfloat16>(p, g) : fwd_smem<float>(p, g);
    if (packed) pl.workspace = size_t(g.oc_tiles) * g.nchunks * g.w_bytes;
    return pl;
}

template <typename T>
static cudaError_t fwd_tc_t(const Plan& pl, const ConvParams& p, const void* x, const void* w,
                            const void* bias, void* y, void* ws, cudaStream_t s)
{
    const int v = pl.variant;
    FwdGeom g = fwd_geom<T>(p, (v / 128) % 16, (v / 8) % 16, v % 8);
    g.kc_per = v / 2048;
    g.splits = ceil_div(g.nchunks, g.kc_per);
    g.packed = ws ? 1 : 0;
    cudaError_t e = cudaSuccess;
    if (ws) {
        const dim3 pgrid(ceil_div(g.OTp * 8, 256), g.nchunks, g.oc_tiles);
        pack_fwd_w_kernel<T><<<pgrid, 256, 0, s>>>(p, (const T*)w, (unsigned char*)ws, g.nchunks, g.OTp);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
#define IG_LAUNCH_FWD_TC(R)                                                                                  \
    do {                                                                                                     \
        e = ensure_smem<fwd_tc_kernel<T, R>>(pl.smem);                                                       \
        if (e == cudaSuccess)                                                                                \
            e = launch_ex(fwd_tc_kernel<T, R>, dim3(pl.grid), dim3(pl.block), pl.smem, s, g.splits, true, p, \
                          (const T*)x, (const T*)w, (const unsigned char*)ws, (const T*)bias, (T*)y, g);     \
    } while (0)
    if (p.relu) IG_LAUNCH_FWD_TC(true);
    else IG_LAUNCH_FWD_TC(false);
#undef IG_LAUNCH_FWD_TC
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t run_fwd_tc(const Plan& pl, const ConvParams& p, int dt, const void* x, const void* w,
                       const void* bias, void* y, void* ws, cudaStream_t s)
{
    return dt == DT_F32 ? fwd_tc_t<float>(pl, p, x, w, bias, y, ws, s)
                        : fwd_tc_t<__nv_bfloat16>(pl, p, x, w, bias, y, ws, s);
}

// ---- wgrad ------------------------------------------------------------------------------
// Layout: the patches in tensor memory (k-tiles of at most 128 rows, the TMEM lanes) except
// for bf16 from WG_GT_MIN_B samples on, which keeps g in tensor memory and the patches in
// shared memory with k-tiles of up to 256 rows: per k row it formats g half as often, which
// decides at large batches (layer 1 bf16 at B = 16384: 305 against 401 us; at B = 1024 both
// 42.7 us; layer 2 bf16 at B = 1024 26.4 against 34.6 us for the patches-in-TMEM layout).
// k rows per tile: the most the layout allows, shrunk to K*K*IC rounded up to 32; splits:
// enough tiles to cover the SMs, at least two chunks per split; then the deepest raw / B rings
// that fit.
constexpr int WG_GT_MIN_B = 2048;

template <typename T>
static bool pick_wgrad(const ConvParams& p, const DevInfo& d, TcWgradGeom& out)
{
    using Tr = TcTraits<T>;
    if (p.P > Tr::KC || p.B <= 0 || p.OC > TC_M) return false;  // one dy range of all OC per chunk
    const int layout = (!Tr::split && p.B >= WG_GT_MIN_B) ? 1 : 0;
    const int ktp = std::min(layout ? 256 : TC_M, round_up(p.Kred, 32));
    const int cnp = round_up(wgrad_nsc(p.P, Tr::KC, Tr::KC / 4) * p.P, Tr::KC / 4);
    const int ng = Tr::split ? 8 : 16;  // columns per G / X group
    if (layout) {
        const int upr = cnp / Tr::E;
        if (ceil_div(ktp, 32 * (16 - WgRolesGt<T>::g_warps) / upr) > WgRolesGt<T>::x_rows) return false;
        if (ceil_div(cnp / ng, WgRolesGt<T>::g_warps / 4) > WgRolesGt<T>::g_groups) return false;
    } else {
        if (ceil_div(cnp / ng, WgRoles<T>::g_warps / 4) > WgRoles<T>::g_groups) return false;
        if (ceil_div(cnp / ng, (16 - WgRoles<T>::g_warps) / 4) > WgRoles<T>::x_groups) return false;
    }
    const int tiles = ceil_div(p.Kred, ktp) * ceil_div(p.OC, TC_M);
    const int nsc = wgrad_nsc(p.P, Tr::KC, Tr::KC / 4);
    int splits = std::max(1, d.sms / tiles);
    splits = std::min(splits, std::max(1, p.B / (2 * nsc)));
    // The raw ring hides the bulk copies' latency (about 1.5k clocks from issue to landing),
    // so it gets the deeper ring; two B stages suffice.
    static const int cfgs[][2] = {{5, 2}, {4, 2}, {3, 3}, {3, 2}, {2, 2}};  // {raws, nbs}
    for (const auto& c : cfgs) {
        const TcWgradGeom g = wgrad_geom<T>(p, ktp, c[0], c[1], splits, layout);
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
    static_assert(WG_MAXR < 8 && WG_MAXB < 8, "wgrad plan: ring depths in 3 bits each");
    pl.variant = ((g.KTp * 8 + g.raws) * 8 + g.nbs) * 2 + g.layout;
    pl.launches = 2;
    pl.grid = std::min(g.k_tiles * g.oc_tiles * g.splits, d.sms);
    // the split-K partials, then room for the bias gradient's partial channel sums (two G lane
    // groups per split at most), so that conv_bwd_filter and conv_bwd_filter_bias share the size
    pl.workspace = size_t(g.splits) * p.OC * g.kpad * sizeof(float) + size_t(g.splits) * 2 * p.OC * sizeof(float);
    return pl;
}

template <typename T>
static cudaError_t wgrad_tc_t(const Plan& pl, const ConvParams& p, const void* x, const void* dy,
                              const void* y, void* dw, void* ws, void* db, cudaStream_t s)
{
    cudaError_t e = cudaSuccess;
    const int kpad = round_up(p.Kred, 4);
    float* bpart = db ? reinterpret_cast<float*>(static_cast<unsigned char*>(ws) +
                                                 size_t(pl.splits) * p.OC * kpad * sizeof(float))
                      : nullptr;
    int nbp = 0;
    if (pl.splits > 0) {
        const int v = pl.variant / 2;
        const TcWgradGeom g = wgrad_geom<T>(p, v / 64, (v / 8) % 8, v % 8, pl.splits, pl.variant % 2);
        nbp = wgrad_bias_parts<T>(g);
#define IG_LAUNCH_WG_TC(R, GT)                                                                             \
    do {                                                                                                   \
        e = ensure_smem<wgrad_tc_kernel<T, R, GT>>(pl.smem);                                               \
        if (e == cudaSuccess)                                                                              \
            e = launch_ex(wgrad_tc_kernel<T, R, GT>, dim3(pl.grid), dim3(pl.block), pl.smem, s, 1, true, p,   \
                          (const T*)x, (const T*)dy, (const T*)y, (float*)ws, bpart, g);                   \
    } while (0)
        if constexpr (!TcTraits<T>::split) {  // the g-in-TMEM layout is a bf16 plan only
            if (g.layout) {
                if (p.relu) IG_LAUNCH_WG_TC(true, true);
                else IG_LAUNCH_WG_TC(false, true);
            }
        }
        if (!g.layout) {
            if (p.relu) IG_LAUNCH_WG_TC(true, false);
            else IG_LAUNCH_WG_TC(false, false);
        }
#undef IG_LAUNCH_WG_TC
        if (e == cudaSuccess) e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return run_wgrad_reduce(p, dt_of_tc<T>(), (const float*)ws, pl.splits, kpad, dw, s, pl.splits > 0, bpart,
                            pl.splits > 0 ? nbp : 0, db);
}

cudaError_t run_wgrad_tc(const Plan& pl, const ConvParams& p, int dt, const void* x, const void* dy,
                         const void* y, void* dw, void* ws, void* db, cudaStream_t s)
{
    return dt == DT_F32 ? wgrad_tc_t<float>(pl, p, x, dy, y, dw, ws, db, s)
                        : wgrad_tc_t<__nv_bfloat16>(pl, p, x, dy, y, dw, ws, db, s);
}

// ---- d_input ------------------------------------------------------------------------
// Channels per k-tile: as many as keep KTp within the accumulator limit (128 rows; the fp32
// accumulator holds hi and lo halves), then the deepest weight ring that fits.  `packed`: the
// workspace path (no raw w slots).
template <typename T>
static bool pick_dgrad(const ConvParams& p, const DevInfo& d, bool packed, TcDgradGeom& out)
{
    if (p.B <= 0 || p.KK > 128 || p.P > DG_TM) return false;
    for (int cic = std::min(p.IC, 128 / p.KK); cic >= 1; --cic) {
        for (int nw = 4; nw >= 2; --nw) {
            TcDgradGeom g = dgrad_geom<T>(p, cic, nw);
            g.packed = packed ? 1 : 0;
            if (g.dcols * g.ndb + g.acols * g.nab > 512) continue;
            if (dgrad_smem<T>(p, g) <= d.smem_optin) {
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

bool tc_dgrad_ok(const ConvParams& p, int dt, const DevInfo& d, bool packed)
{
    if (d.cc_major != 10) return false;
    TcDgradGeom g;
    return dt == DT_BF16 ? pick_dgrad<__nv_bfloat16>(p, d, packed, g) : pick_dgrad<float>(p, d, packed, g);
}

Plan plan_dgrad_tc(const ConvParams& p, int dt, const DevInfo& d, bool packed)
{
    TcDgradGeom g;
    if (dt == DT_BF16) pick_dgrad<__nv_bfloat16>(p, d, packed, g);
    else pick_dgrad<float>(p, d, packed, g);
    Plan pl;
    pl.algo = ALGO_TC;
    // the implicit GEMM + col2im (weights formatted in the kernel); the workspace path first
    // packs W^T into the workspace
    pl.launches = packed ? 2 : 1;
    pl.block = DG_THREADS;
    static_assert(DG_MAXW < 8, "d_input plan: weight stages in 3 bits");
    pl.variant = (g.kt_per * 256 + g.CIC) * 8 + g.nw;  // CIC <= 128 (KTp <= 128 rows)
    pl.grid = std::min(g.ntiles * g.ktsplit, d.sms);
    pl.smem = dt == DT_BF16 ? dgrad_smem<__nv_bfloat16>(p, g) : dgrad_smem<float>(p, g);
    if (packed) pl.workspace = size_t(g.nkt) * g.nch * g.w_tile;
    return pl;
}

template <typename T>
static cudaError_t dgrad_tc_t(const Plan& pl, const ConvParams& p, const void* dy, const void* w,
                              const void* y, void* dx, void* ws, cudaStream_t s)
{
    TcDgradGeom g = dgrad_geom<T>(p, (pl.variant / 8) % 256, pl.variant % 8);
    g.kt_per = pl.variant / 2048;
    g.ktsplit = ceil_div(g.nkt, g.kt_per);
    g.packed = ws ? 1 : 0;
    cudaError_t e = cudaSuccess;
    if (ws) {
        const dim3 pgrid(ceil_div(g.KTp * 8, 256), g.nch, g.nkt);
        pack_dgrad_w_kernel<T><<<pgrid, 256, 0, s>>>(p, (const T*)w, (unsigned char*)ws, g.nch, g.CIC, g.KTp);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
#define IG_LAUNCH_DG_TC(R, SH)                                                                               \
    do {                                                                                                     \
        e = ensure_smem<dgrad_tc_kernel<T, R, SH>>(pl.smem);                                                 \
        if (e == cudaSuccess)                                                                                \
            e = launch_ex(dgrad_tc_kernel<T, R, SH>, dim3(pl.grid), dim3(pl.block), pl.smem, s, 1, true, p,  \
                          (const T*)dy, (const T*)w, (const unsigned char*)ws, (const T*)y, (T*)dx, g);      \
    } while (0)
    switch (dgrad_shape(p, g) * 2 + (p.relu ? 1 : 0)) {
    case 2: IG_LAUNCH_DG_TC(false, 1); break;
    case 3: IG_LAUNCH_DG_TC(true, 1); break;
    case 1: IG_LAUNCH_DG_TC(true, 0); break;
    default: IG_LAUNCH_DG_TC(false, 0); break;
    }
#undef IG_LAUNCH_DG_TC
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t run_dgrad_tc(const Plan& pl, const ConvParams& p, int dt, const void* dy, const void* w,
                         const void* y, void* dx, void* ws, cudaStream_t s)
{
    return dt == DT_F32 ? dgrad_tc_t<float>(pl, p, dy, w, y, dx, ws, s)
                        : dgrad_tc_t<__nv_bfloat16>(pl, p, dy, w, y, dx, ws, s);
}

// ---- fused backward (d_input + wgrad in one launch) -----------------------------------------
// Fused only while d_input's own launch has fewer than two waves of work items: then its last
// wave leaves SMs idle that the wgrad tiles can fill.  With more items the tail is a small part
// of the launch, and one CTA per item (each with its own prologue) loses to the persistent
// standalone kernels.  Fused: wgrad's stages with the split count that gives about two thirds as
// many tiles as SMs (the long items: two thirds of the SMs run them, the rest d_input's items and
// then everything), and d_input's workspace-path geometry with its k-tiles cut into two ranges
// per sample tile, three when the sample tiles fill fewer than a quarter of the SMs (short items
// that backfill).  Measured on a GB300 at both encoder layers and both dtypes (B = 1024: wgrad
// tiles on 35, 50, 65, 80 and 95 % of the SMs, two and three ranges; B = 4096, 16384 for the
// fusion rule).

template <typename T>
static bool pick_bwd(const ConvParams& p, const DevInfo& d, TcDgradGeom& dg, TcWgradGeom& wg)
{
    if (d.cc_major != 10 || p.B <= 0) return false;
    if (!pick_dgrad<T>(p, d, true, dg) || !pick_wgrad<T>(p, d, wg)) return false;
    if (dg.ntiles * dg.ktsplit >= 2 * d.sms) return false;
    const int tiles = wg.k_tiles * wg.oc_tiles;
    const int splits = std::min(std::max(1, (2 * d.sms / 3 + tiles / 2) / tiles), std::max(1, p.B / (2 * wg.nsc)));
    wg = wgrad_geom<T>(p, wg.KTp, wg.raws, wg.nbs, splits, wg.layout);
    const int ranges = 4 * dg.ntiles < d.sms ? 3 : 2;
    dg.kt_per = ceil_div(dg.nkt, std::min(dg.nkt, ranges));
    dg.ktsplit = ceil_div(dg.nkt, dg.kt_per);
    return true;
}

template <typename T>
static size_t bwd_wgrad_offset(const TcDgradGeom& dg)
{
    return round_up(size_t(dg.nkt) * dg.nch * dg.w_tile, size_t(256));
}

bool tc_bwd_ok(const ConvParams& p, int dt, const DevInfo& d)
{
    TcDgradGeom dg;
    TcWgradGeom wg;
    return dt == DT_BF16 ? pick_bwd<__nv_bfloat16>(p, d, dg, wg) : pick_bwd<float>(p, d, dg, wg);
}

Plan plan_bwd_tc(const ConvParams& p, int dt, const DevInfo& d)
{
    TcDgradGeom dg;
    TcWgradGeom wg;
    Plan pl;
    if (dt == DT_BF16) {
        pick_bwd<__nv_bfloat16>(p, d, dg, wg);
        pl.smem = std::max(dgrad_smem<__nv_bfloat16>(p, dg), wgrad_smem<__nv_bfloat16>(wg));
        pl.workspace = bwd_wgrad_offset<__nv_bfloat16>(dg);
    } else {
        pick_bwd<float>(p, d, dg, wg);
        pl.smem = std::max(dgrad_smem<float>(p, dg), wgrad_smem<float>(wg));
        pl.workspace = bwd_wgrad_offset<float>(dg);
    }
    pl.algo = ALGO_TC;
    pl.launches = 3;  // pack W^T, the fused kernel, the split reduction
    pl.block = DG_THREADS;
    pl.splits = wg.splits;
    const int n_wg = wg.k_tiles * wg.oc_tiles * wg.splits;
    pl.grid = n_wg + dg.ntiles * dg.ktsplit;  // one work item per CTA
    pl.variant = n_wg;
    // packed W^T | split-K partials | bias partial channel sums (two G lane groups per split at most)
    pl.workspace += size_t(wg.splits) * p.OC * wg.kpad * sizeof(float) + size_t(wg.splits) * 2 * p.OC * sizeof(float);
    return pl;
}

template <typename T>
static cudaError_t bwd_tc_t(const Plan& pl, const ConvParams& p, const DevInfo& d, const void* x, const void* dy,
                            const void* w, const void* y, void* dx, void* dw, void* db, void* ws, cudaStream_t s)
{
    TcDgradGeom dg;
    TcWgradGeom wg;
    if (!pick_bwd<T>(p, d, dg, wg)) return cudaErrorInvalidValue;
    const int n_wg = pl.variant;
    unsigned char* wsb = static_cast<unsigned char*>(ws);
    float* part = reinterpret_cast<float*>(wsb + bwd_wgrad_offset<T>(dg));
    float* bpart = db ? part + size_t(wg.splits) * p.OC * wg.kpad : nullptr;
    const dim3 pgrid(ceil_div(dg.KTp * 8, 256), dg.nch, dg.nkt);
    pack_dgrad_w_kernel<T><<<pgrid, 256, 0, s>>>(p, (const T*)w, wsb, dg.nch, dg.CIC, dg.KTp);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
#define IG_LAUNCH_BWD_TC(R, GT, SH)                                                                          \
    do {                                                                                                     \
        e = ensure_smem<bwd_tc_kernel<T, R, GT, SH>>(pl.smem);                                               \
        if (e == cudaSuccess)                                                                                \
            e = launch_ex(bwd_tc_kernel<T, R, GT, SH>, dim3(pl.grid), dim3(pl.block), pl.smem, s, 1, true,   \
                          p, (const T*)x, (const T*)dy, (const T*)w, (const unsigned char*)wsb, (const T*)y, \
                          (T*)dx, part, bpart, dg, wg, n_wg);                                                 \
    } while (0)
#define IG_LAUNCH_BWD_SH(R, GT)                 \
    do {                                        \
        if (dgrad_shape(p, dg) == 1)            \
            IG_LAUNCH_BWD_TC(R, GT, 1);         \
        else                                    \
            IG_LAUNCH_BWD_TC(R, GT, 0);         \
    } while (0)
    if constexpr (!TcTraits<T>::split) {
        if (wg.layout) {
            if (p.relu) IG_LAUNCH_BWD_SH(true, true);
            else IG_LAUNCH_BWD_SH(false, true);
        }
    }
    if (!wg.layout) {
        if (p.relu) IG_LAUNCH_BWD_SH(true, false);
        else IG_LAUNCH_BWD_SH(false, false);
    }
#undef IG_LAUNCH_BWD_SH
#undef IG_LAUNCH_BWD_TC
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return run_wgrad_reduce(p, dt_of_tc<T>(), part, wg.splits, wg.kpad, dw, s, true, bpart,
                            wgrad_bias_parts<T>(wg), db);
}

cudaError_t run_bwd_tc(const Plan& pl, const ConvParams& p, int dt, const DevInfo& d, const void* x, const void* dy,
                       const void* w, const void* y, void* dx, void* dw, void* db, void* ws, cudaStream_t s)
{
    return dt == DT_F32 ? bwd_tc_t<float>(pl, p, d, x, dy, w, y, dx, dw, db, ws, s)
                        : bwd_tc_t<__nv_bfloat16>(pl, p, d, x, dy, w, y, dx, dw, db, ws, s);
}

// ---- two-layer forward chain ----------------------------------------------------------
// Samples per group: as many whole samples as fit the 128 TMEM lanes in both layers (layer 1
// usually decides: 10 samples of 3x4); then the deepest weight ring and longest x super-chunk
// that fit, with the y1 slab of the group.
template <typename T>
static ChainGeom chain_geom(const ConvParams& p1, const ConvParams& p2, int xg, int nw, int nraw)
{
    using Tr = TcTraits<T>;
    const int es = int(sizeof(T));
    const int ns = std::min(FA_TM / p1.P, FA_TM / p2.P);
    ChainGeom cg;
    cg.g1 = fwd_geom<T>(p1, xg, nw, nraw);
    cg.g1.packed = 1;
    cg.g1.nsmax = std::min(ns, p1.B);
    cg.g1.raw_bytes = round_up(cg.g1.nsmax * cg.g1.xs, 128);
    cg.ns = ns;
    cg.ngroups = ceil_div(p1.B, ns);
    cg.OTp2 = round_up(p2.OC, 16);
    cg.oc_tiles2 = 1;
    cg.N2p = round_up(ns * p2.P, 16);
    cg.nchunks2 = round_up(p2.Kred, Tr::KC) / Tr::KC;
    cg.w_bytes2 = cg.OTp2 * ROWB * (Tr::split ? 2 : 1);  // one chunk of the packed W2 image
    cg.stage_bytes = std::max(cg.g1.w_bytes, cg.w_bytes2);  // a W1 or a W2 chunk
    cg.patch_bytes = cg.N2p * ROWB * (Tr::split ? 2 : 1);
    cg.dcols = std::max(cg.g1.dcols, cg.N2p * (Tr::split ? 2 : 1));
    cg.acol0 = round_up(cg.dcols, 32);
    cg.g1.na = std::min(FA_MAXA, (FA_TMEM_COLS - cg.acol0) / cg.g1.acols);
    cg.xs2 = round_up(p2.IHW * es, 16) + 16;  // a sample of conv2's input, 16-byte padded
    cg.slab_bytes = round_up(ns * cg.xs2, 128);
    cg.wpack2_off = round_up(size_t(cg.g1.oc_tiles) * cg.g1.nchunks * cg.g1.w_bytes, size_t(256));
    cg.relu1 = p1.relu;
    cg.relu2 = p2.relu;
    return cg;
}

template <typename T>
static bool pick_chain(const ConvParams& p1, const ConvParams& p2, const DevInfo& d, ChainGeom& out)
{
    using Tr = TcTraits<T>;
    const int otmax = Tr::split ? 128 : 256;
    // layer 2's output channels are the TMEM lanes of its accumulator; its columns (a group's
    // samples) the MMA's N, twice over for the fp32 hi / lo pair
    if (d.cc_major != 10 || p1.B <= 0 || p1.P > FA_TM || p2.P > FA_TM || p1.OC > otmax || p2.OC > FA_TM) return false;
    if (round_up(std::min(FA_TM / p1.P, FA_TM / p2.P) * p2.P, 16) * (Tr::split ? 2 : 1) > 256) return false;
    static const int cfgs[][3] = {{4, 8, 2}, {4, 4, 2}, {4, 2, 2}, {3, 4, 2}, {3, 2, 2}, {2, 2, 2}, {2, 1, 2}};
    for (const auto& c : cfgs) {
        const ChainGeom cg = chain_geom<T>(p1, p2, c[1], c[0], c[2]);
        if (cg.g1.na < 2 || chain_smem<T>(p1, p2, cg) > d.smem_optin) continue;
        out = cg;
        return true;
    }
    return false;
}

int chain_groups(const ConvParams& p1, const ConvParams& p2)
{
    return ceil_div(p1.B, std::max(1, std::min(FA_TM / p1.P, FA_TM / p2.P)));
}

bool tc_chain_ok(const ConvParams& p1, const ConvParams& p2, int dt, const DevInfo& d)
{
    ChainGeom cg;
    return dt == DT_BF16 ? pick_chain<__nv_bfloat16>(p1, p2, d, cg) : pick_chain<float>(p1, p2, d, cg);
}

Plan plan_chain_tc(const ConvParams& p1, const ConvParams& p2, int dt, const DevInfo& d)
{
    ChainGeom cg;
    if (dt == DT_BF16) pick_chain<__nv_bfloat16>(p1, p2, d, cg);
    else pick_chain<float>(p1, p2, d, cg);
    Plan pl;
    pl.algo = ALGO_TC;
    pl.launches = 3;  // pack W1, pack W2, the chain
    pl.block = CH_THREADS;
    pl.grid = std::min(cg.ngroups, d.sms);
    pl.smem = dt == DT_BF16 ? chain_smem<__nv_bfloat16>(p1, p2, cg) : chain_smem<float>(p1, p2, cg);
    pl.variant = (cg.g1.xg * 16 + cg.g1.nw) * 8 + cg.g1.nraw;
    pl.workspace = cg.wpack2_off + size_t(cg.nchunks2) * cg.w_bytes2;
    return pl;
}

template <typename T>
static cudaError_t chain_tc_t(const Plan& pl, const ConvParams& p1, const ConvParams& p2, const void* x,
                              const void* w1, const void* b1, const void* w2, const void* b2, void* y1, void* y2,
                              void* ws, cudaStream_t s)
{
    const int v = pl.variant;
    const ChainGeom cg = chain_geom<T>(p1, p2, (v / 128) % 16, (v / 8) % 16, v % 8);
    unsigned char* wsb = static_cast<unsigned char*>(ws);
    const dim3 pg1(ceil_div(cg.g1.OTp * 8, 256), cg.g1.nchunks, cg.g1.oc_tiles);
    pack_fwd_w_kernel<T><<<pg1, 256, 0, s>>>(p1, (const T*)w1, wsb, cg.g1.nchunks, cg.g1.OTp);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const dim3 pg2(ceil_div(cg.OTp2 * 8, 256), cg.nchunks2, 1);
    pack_fwd_w_kernel<T><<<pg2, 256, 0, s>>>(p2, (const T*)w2, wsb + cg.wpack2_off, cg.nchunks2, cg.OTp2);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    e = ensure_smem<fwd_chain_kernel<T>>(pl.smem);
    if (e == cudaSuccess)
        e = launch_ex(fwd_chain_kernel<T>, dim3(pl.grid), dim3(pl.block), pl.smem, s, 1, true, p1, p2, (const T*)x,
                      (const unsigned char*)wsb, (const T*)b1, (const T*)b2, (T*)y1, (T*)y2, cg);
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t run_chain_tc(const Plan& pl, const ConvParams& p1, const ConvParams& p2, int dt, const void* x,
                         const void* w1, const void* b1, const void* w2, const void* b2, void* y1, void* y2, void* ws,
                         cudaStream_t s)
{
    return dt == DT_F32 ? chain_tc_t<float>(pl, p1, p2, x, w1, b1, w2, b2, y1, y2, ws, s)
                        : chain_tc_t<__nv_bfloat16>(pl, p1, p2, x, w1, b1, w2, b2, y1, y2, ws, s);
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
