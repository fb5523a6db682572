// common.cuh -- index math and parameter block shared by every kernel.
//
// Index math follows the fast-divmod idea the PufferLib PR #522 description
// credits for much of its speed-up ("fast divmod operator and caching
// repeatable operations"): every division by a runtime-invariant divisor (P,
// OW, K*K, K) is a multiply-high and a shift, with the magic numbers computed
// once on the host (Granlund & Montgomery, "Division by invariant integers
// using multiplication", PLDI 1994, the round-up method with an N+1-bit
// multiplier).
#pragma once
#include <cstdint>
#include <cuda_bf16.h>

#if defined(__CUDACC__)
#define IG_HD __host__ __device__ __forceinline__
#else
#define IG_HD inline
#endif

// Quotient and remainder of n / d for 0 <= n < 2^31 and 1 <= d < 2^31.
// With l = ceil(log2 d) and m = floor(2^32 (2^l - d) / d) + 1, the quotient
// is floor((mulhi(m, n) + n) / 2^l); the sum stays below 2^32 because
// mulhi(m, n) <= n < 2^31.
struct FastDivmod {
    uint32_t d, m, l;

    FastDivmod() : d(1), m(1), l(0) {}
    explicit FastDivmod(uint32_t div) : d(div)
    {
        l = 0;
        while ((uint64_t(1) << l) < div) ++l;
        m = uint32_t(((uint64_t(1) << 32) * ((uint64_t(1) << l) - div)) / div + 1);
    }

    IG_HD uint32_t mulhi(uint32_t a, uint32_t b) const
    {
#if defined(__CUDA_ARCH__)
        return __umulhi(a, b);
#else
        return uint32_t((uint64_t(a) * uint64_t(b)) >> 32);
#endif
    }
    IG_HD uint32_t div(uint32_t n) const { return (mulhi(m, n) + n) >> l; }
    IG_HD void divmod(uint32_t n, uint32_t& q, uint32_t& r) const
    {
        q = div(n);
        r = n - q * d;
    }
};

// Everything a kernel needs to know about one layer, built on the host.
struct ConvParams {
    int B, IC, OC, H, W, K, S, OH, OW, relu;
    int P;     // OH * OW          output positions per sample
    int KK;    // K * K
    int Kred;  // IC * K * K       GEMM reduction length of fwd / wgrad
    int HW;    // H * W
    int IHW;   // IC * H * W       x / dx elements per sample
    int OCP;   // OC * P           y / dy elements per sample
    int N;     // B * P            GEMM columns (b, oh, ow)
    FastDivmod dm_P, dm_OW, dm_KK, dm_K, dm_W, dm_HW;
};

// Element access: bf16 storage widens to fp32 exactly; stores round once (RNE).
template <typename T> struct Elem;
template <> struct Elem<float> {
    static __device__ __forceinline__ float ld(const float* p) { return *p; }
    static __device__ __forceinline__ float ldg(const float* p) { return __ldg(p); }
    static __device__ __forceinline__ void st(float* p, float v) { *p = v; }
};
template <> struct Elem<__nv_bfloat16> {
    static __device__ __forceinline__ float ld(const __nv_bfloat16* p) { return __bfloat162float(*p); }
    static __device__ __forceinline__ float ldg(const __nv_bfloat16* p) { return __bfloat162float(__ldg(p)); }
    static __device__ __forceinline__ void st(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }
};

// Offset of x[b, ic, oh*S + kh, ow*S + kw] split into a reduction part (ic, kh, kw)
// and a column part (b, oh, ow):  x_index = col_base(n) + k_off(k).
__device__ __forceinline__ int k_offset(const ConvParams& p, int k)
{
    uint32_t ic, r, kh, kw;
    p.dm_KK.divmod(uint32_t(k), ic, r);
    p.dm_K.divmod(r, kh, kw);
    return int(ic) * p.HW + int(kh) * p.W + int(kw);
}
__device__ __forceinline__ int col_base(const ConvParams& p, int n)
{
    uint32_t b, pp, oh, ow;
    p.dm_P.divmod(uint32_t(n), b, pp);
    p.dm_OW.divmod(pp, oh, ow);
    return int(b) * p.IHW + int(oh) * p.S * p.W + int(ow) * p.S;
}
// Offset of y[b, 0, oh, ow] for column n = (b, oh, ow): add oc * P for channel oc.
__device__ __forceinline__ int col_out(const ConvParams& p, int n)
{
    uint32_t b, pp;
    p.dm_P.divmod(uint32_t(n), b, pp);
    return int(b) * p.OCP + int(pp);
}
