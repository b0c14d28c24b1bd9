// tern_mma_common.cuh -- pieces shared by the tensor-core kernels: operand
// encodings, descriptors, bounded waits and tensor-map creation.
//
// The weights enter the MMA as e4m3 bytes of exactly +2, -2 or 0 built from
// the packed 2-bit codes with one shift and one AND per four codes.  Each
// activation enters as e4m3 terms under power-of-two row scales, in one or
// two magnitude bands per row range (see split_word1, split_word2 and
// need_two_bands): band A holds the elements within 2^13 of the row maximum,
// band B the rest under its own scale, and each band carries a value as
// hi + lo/16.  The MMA is tcgen05 kind::f8f6f4 with fp32 accumulation in
// tensor memory.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#ifdef TERN_WAIT_DIAG
#include <cstdio>
#endif

#include "tern_ptx.cuh"

namespace tern {
namespace mma {

constexpr int kStageWords = 32;         // words per row per TMA stage (512 codes, 128 B)
constexpr int kStageBytes = 128 * 128;  // one stage of a 128-row tile
constexpr int kSmemLimit = 227 * 1024;

// B operand, compact layout: per 16-code block (one packed word column) the
// 2 * bands * m rows of the m activation rows, 16 bytes each and contiguous,
// so blocks are 32 * bands * m bytes apart.  With one band, rows 2i and
// 2i + 1 hold hi and lo of activation row i; with two bands rows 4i .. 4i+3
// hold hi_A, lo_A, hi_B, lo_B.  The MMA reads N rows from each block start;
// rows past the live ones read the next blocks' bytes and feed only
// accumulator columns that are never read, so a buffer needs up to 32 * 16
// bytes of readable slack after its last block.
constexpr uint32_t kBPad = 512;
__host__ __device__ constexpr uint32_t b_block_bytes(int m, int bands) { return 32u * (uint32_t)(bands * m); }
// MMA N for m activation rows: 2 * bands * m live B rows, N a multiple of 16.
__host__ __device__ constexpr int mma_n(int m, int bands) { return 2 * bands * m <= 16 ? 16 : 32; }

// Instruction descriptor: kind::f8f6f4, D fp32, A e4m3, B e4m3, both
// K-major, M = 128, N = n.
__host__ __device__ constexpr uint32_t idesc_n(int n)
{
    return (1u << 4) | (0u << 7) | (0u << 10) | (((uint32_t)n >> 3) << 17) | ((128u >> 4) << 24);
}

// Shared-memory descriptor of a K-major, unswizzled B operand made of 8-row
// x 16-byte core matrices: 16-code blocks `lbo` bytes apart along K, and
// within a block rows 8j .. 8j+7 at +128j (SBO 128 bytes along N).
__device__ __forceinline__ uint64_t b_desc_lbo(uint32_t addr, uint32_t lbo)
{
    return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)(128u >> 4) << 32) | (1ull << 46);
}

// Default bound of a Waiter, in SM clock cycles (about one second).
constexpr long long kWaitCycles = 1ll << 31;

// Spin on an mbarrier phase with a time bound (`limit` cycles, normally
// kWaitCycles; the host may pass a shorter one to exercise the time-out
// path).  On time-out the kernel's error word and the CTA's abort flag are
// set; once the abort flag is up every later wait returns false at once.
struct Waiter {
    static constexpr uint32_t kSleepNs = 1000000u;
    volatile uint32_t *abort_flag;  // shared
    unsigned int *err;              // global error word of the kernel
    long long limit;
    // Each try sleeps until the phase completes or `hint` ns pass (kSleepNs,
    // or about half the bound when the bound is shorter, so that a short
    // bound is checked in time); the abort flag and the bound are checked
    // between tries.
    uint32_t hint;
    __device__ Waiter(volatile uint32_t *abort_flag_, unsigned int *err_, long long limit_)
        : abort_flag(abort_flag_), err(err_), limit(limit_),
          hint(limit_ < 2ll * kSleepNs ? (uint32_t)(limit_ / 2 + 1) : kSleepNs)
    {
    }
    __device__ __forceinline__ bool wait(uint32_t bar, uint32_t parity) const
    {
        if (*abort_flag) return false;
        if (ptx::mbar_try_wait(bar, parity)) return true;
        const long long t0 = clock64();
        while (!ptx::mbar_try_wait_sleep(bar, parity, hint)) {
            if (*abort_flag) return false;
            if (clock64() - t0 > limit) {
#ifdef TERN_WAIT_DIAG
                printf("wait ran out: block %d thread %d bar %u parity %u\n", (int)blockIdx.x, (int)threadIdx.x,
                       bar, parity);
#endif
                atomicOr(err, 1u);
                *abort_flag = 1u;
                return false;
            }
        }
        return true;
    }
};

// Bounded wait that ignores the abort flag (used to drain in-flight work).
// Its bound is always kWaitCycles: the copies and MMAs it waits for complete
// on their own, and a CTA must not exit while they are in flight.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, unsigned int *err)
{
    const long long t0 = clock64();
    while (!ptx::mbar_try_wait_sleep(bar, parity, Waiter::kSleepNs)) {
        if (clock64() - t0 > kWaitCycles) {
            atomicOr(err, 1u);
            return;
        }
    }
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + expf(-z)); }

// Knuth's TwoSum (TAOCP vol. 2, 4.2.2; also Moller 1965): s + e == a + b
// exactly, with s = fl(a + b), in round-to-nearest fp32.
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e)
{
    s = __fadd_rn(a, b);
    const float bv = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bv)), __fsub_rn(b, bv));
}

// (hi, lo) += v, keeping hi + lo equal to the running sum up to lo's own
// rounding: band partials of very different magnitude (an outlier channel
// in one band or K range, the bulk in another) then cancel without losing
// the bulk to fp32 rounding at the outliers' scale.
__device__ __forceinline__ void acc_pair(float &hi, float &lo, float v)
{
    float s, e;
    two_sum(hi, v, s, e);
    hi = s;
    lo = __fadd_rn(lo, e);
}

// 2^e as an fp32 (e in [-126, 127]).
__device__ __forceinline__ float exp2i(int e) { return __int_as_float((e + 127) << 23); }

// Per-row scale exponent s for a row whose largest |x| has fp32 bits mb:
// the maximum lands in [128, 256) after multiplying by 2^s.
__device__ __forceinline__ int row_scale_exp(uint32_t mb)
{
    const int e = mb == 0u ? 0 : (int)(mb >> 23) - 127;
    return min(max(7 - e, -120), 120);
}

// Largest bf16 magnitude (bits & 0x7FFF) among 16 values, as the fp32 bits
// of that magnitude (the bf16 bits shifted up by 16).
__device__ __forceinline__ uint32_t max_abs16(const uint4 a, const uint4 b)
{
    const uint32_t v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t mx = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) mx = __vmaxu2(mx, v[q] & 0x7FFF7FFFu);
    return max(mx & 0xFFFFu, mx >> 16) << 16;
}

// Band threshold of a row whose largest |x| has fp32 bits mb, as bf16
// magnitude bits replicated in both halves: 2^(e-13) for 2^e <= max|x| <
// 2^(e+1), the smallest magnitude the row-maximum scale represents exactly
// (see split_pair).  0 (every element in band A) when that is not a normal
// number.
__device__ __forceinline__ uint32_t band_threshold2(uint32_t mb)
{
    const int f = (int)(mb >> 23) - 13;  // biased exponent of 2^(e-13)
    const uint32_t t = f >= 1 ? (uint32_t)f << 7 : 0u;
    return t | (t << 16);
}

// Statistics of the elements below the band threshold tb2 among 16 values,
// added to n (how many are nonzero and below it) and to sabs (the sum of all
// 16 magnitudes, in fp32).
__device__ __forceinline__ void band_stats16(const uint4 a, const uint4 b, uint32_t tb2, uint32_t &n, float &sabs)
{
    const uint32_t v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const uint32_t mag = v[q] & 0x7FFF7FFFu;
        const uint32_t small = __vcmpltu2(mag, tb2) & __vcmpne2(mag, 0u);
        n += (uint32_t)__popc(small) >> 4;
        sabs += __uint_as_float(mag << 16) + __uint_as_float(mag & 0xFFFF0000u);
    }
}

// Whether a row needs band B.  With one band (scale from the row maximum,
// 2^e <= max|x| < 2^(e+1)), each of the n_small nonzero elements below
// 2^(e-13) is off by at most 2^(e-21) (split_pair); one band is kept when
// that bound, n_small * 2^(e-21), is within 2^-24 of sum|x|, i.e. within one
// fp32 rounding unit of the row's own magnitude sum, which fp32 accumulation
// of the same products already allows for.
__device__ __forceinline__ bool need_two_bands(uint32_t mb, uint32_t n_small, float sabs)
{
    const int e = (int)(mb >> 23) - 127;
    return ldexpf((float)n_small, e + 3) > sabs;
}

// Largest bf16 magnitude below the band threshold tb2 among 16 values (the
// maximum of band B), as fp32 bits; 0 if none is below it.
__device__ __forceinline__ uint32_t max_abs16_below(const uint4 a, const uint4 b, uint32_t tb2)
{
    const uint32_t v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t mx = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const uint32_t mag = v[q] & 0x7FFF7FFFu;
        mx = __vmaxu2(mx, mag & __vcmpltu2(mag, tb2));
    }
    return max(mx & 0xFFFFu, mx >> 16) << 16;
}

// Splits a pair of bf16 activations (one 32-bit word, low half = even k)
// scaled by sc = 2^s into e4m3 bytes with x*2^s = hi + lo/16: hi is x*2^s
// rounded to nearest e4m3, lo = (x*2^s - hi)*16 rounded to nearest e4m3 (the
// difference is formed exactly in f16).  For x*2^s >= 2^-6 hi keeps 4
// significant bits and lo the remaining <= 4, so the pair is exact whenever lo
// is an e4m3 normal or zero; below that both round to e4m3 subnormals (steps
// of 2^-9), bounding the error by 2^-14 in units of x*2^s.
// Output: hp/lp = two bytes each, low byte for the even k.
__device__ __forceinline__ void split_pair(uint32_t v, float sc, uint32_t &hp, uint32_t &lp)
{
    const float xa = __uint_as_float(v << 16) * sc;
    const float xb = __uint_as_float(v & 0xFFFF0000u) * sc;
    uint16_t h, l;
    uint32_t xh, hh, d;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(h) : "f"(xb), "f"(xa));
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(hh) : "h"(h));
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(xh) : "f"(xb), "f"(xa));
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(xh), "r"(hh));
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(d), "r"(0x4C004C00u));  // x16
    asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(l) : "r"(d));
    hp = h;
    lp = l;
}

// Eight pairs of split bytes (low byte = even k of each pair, pairs in k
// order) -> one 16-byte B row in the column order the weight decode
// produces: byte b of output word j holds k offset 4b + j (a 4x4 transpose).
__device__ __forceinline__ uint4 transpose_row(const uint32_t (&p)[8])
{
    const uint32_t p02 = p[0] | (p[2] << 16), p46 = p[4] | (p[6] << 16);
    const uint32_t p13 = p[1] | (p[3] << 16), p57 = p[5] | (p[7] << 16);
    return make_uint4(__byte_perm(p02, p46, 0x6420), __byte_perm(p02, p46, 0x7531), __byte_perm(p13, p57, 0x6420),
                      __byte_perm(p13, p57, 0x7531));
}

// Eight pairs of split bytes -> one 16-byte B row in plain k order (the
// int8 head's weights are decoded in k order).
__device__ __forceinline__ uint4 natural_row(const uint32_t (&p)[8])
{
    return make_uint4(p[0] | (p[1] << 16), p[2] | (p[3] << 16), p[4] | (p[5] << 16), p[6] | (p[7] << 16));
}

// RMSNorm prologue (model page spec table: RMSNorm, eps 1e-6, ahead of the
// q/k/v and gate/up projections).  Per activation row the mean square is
// taken in fp64 (every bf16 square is exact there), the row factor
// r = 1 / sqrt(mean + eps) is rounded to fp32, and each element becomes
// bf16_rn(g * fl32(x * r)): the projection then reads bf16 as without the
// norm.  Only the order of the fp64 sum is the kernel's own.

// Sum of the squares of the 16 bf16 activations of one word, in fp64.
__device__ __forceinline__ double sumsq16(const uint4 a, const uint4 b)
{
    const uint32_t v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    double s = 0.0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const double lo = (double)__uint_as_float(v[j] << 16), hi = (double)__uint_as_float(v[j] & 0xFFFF0000u);
        s = fma(lo, lo, s);
        s = fma(hi, hi, s);
    }
    return s;
}

// Sum of the 16 bf16 activations of one word, in fp64.
__device__ __forceinline__ double sum16(const uint4 a, const uint4 b)
{
    const uint32_t v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    double s = 0.0;
#pragma unroll
    for (int j = 0; j < 8; ++j)
        s += (double)__uint_as_float(v[j] << 16) + (double)__uint_as_float(v[j] & 0xFFFF0000u);
    return s;
}

// Row factor from the row's fp64 sum of squares over k channels.
__device__ __forceinline__ float rms_factor(double ss, int k, float eps)
{
    return (float)(1.0 / sqrt(ss / (double)k + (double)eps));
}

// One word of 16 bf16 activations, normalised in place: element j becomes
// bf16_rn(g[j] * fl32(x[j] * r)); g4: its 16 channel weights.
__device__ __forceinline__ void rmsnorm_word(uint4 &a, uint4 &b, const float4 *g4, float r)
{
    const float4 g0 = __ldg(g4), g1 = __ldg(g4 + 1), g2 = __ldg(g4 + 2), g3 = __ldg(g4 + 3);
    const float g[16] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w, g2.x, g2.y, g2.z, g2.w, g3.x, g3.y, g3.z, g3.w};
    uint32_t v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float lo = __fmul_rn(g[2 * j], __fmul_rn(__uint_as_float(v[j] << 16), r));
        const float hi = __fmul_rn(g[2 * j + 1], __fmul_rn(__uint_as_float(v[j] & 0xFFFF0000u), r));
        v[j] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(lo)) |
               ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(hi)) << 16);
    }
    a = make_uint4(v[0], v[1], v[2], v[3]);
    b = make_uint4(v[4], v[5], v[6], v[7]);
}

// One word (16 k) of one activation row -> its two one-band B rows: out[0]
// = hi, out[1] = lo, at scale sc = 2^s (split_pair); in the ternary decode's
// column order, or in k order when nat (the int8 head).
__device__ __forceinline__ void split_word1(const uint4 a, const uint4 b, float sc, uint4 (&out)[2], bool nat = false)
{
    const uint32_t v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t h[8], l[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) split_pair(v[q], sc, h[q], l[q]);
    if (nat) {
        out[0] = natural_row(h);
        out[1] = natural_row(l);
    } else {
        out[0] = transpose_row(h);
        out[1] = transpose_row(l);
    }
}

// One word (16 k) of one activation row -> its four B rows: out[0], out[1]
// = hi and lo of band A (elements with |x| >= the band threshold tb2, at
// scale scA = 2^sA), out[2], out[3] = hi and lo of band B (the others, at
// scB = 2^sB); an element's bytes in the other band are zero.  Each band
// gives x*2^s = hi + lo/16 exactly for every element of magnitude at least
// 2^(e-13) below its band maximum 2^e <= max < 2^(e+1) (split_pair), so band
// A is exact by construction and band B is exact down to 2^-13 of its own
// maximum.
__device__ __forceinline__ void split_word2(const uint4 a, const uint4 b, float scA, float scB, uint32_t tb2,
                                            uint4 (&out)[4], bool nat = false)
{
    const uint32_t v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t ha[8], la[8], hb[8], lb[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const uint32_t in_a = __vcmpgeu2(v[q] & 0x7FFF7FFFu, tb2);  // 0xFFFF per band-A half
        split_pair(v[q] & in_a, scA, ha[q], la[q]);
        split_pair(v[q] & ~in_a, scB, hb[q], lb[q]);
    }
    if (nat) {
        out[0] = natural_row(ha);
        out[1] = natural_row(la);
        out[2] = natural_row(hb);
        out[3] = natural_row(lb);
    } else {
        out[0] = transpose_row(ha);
        out[1] = transpose_row(la);
        out[2] = transpose_row(hb);
        out[3] = transpose_row(lb);
    }
}

// Eight packed words (128 codes of one row) -> 32 registers of e4m3 bytes:
// register 4q+j holds codes 4b+j of word q in byte b, as 0, +2 (0x40) or -2
// (0xC0): b1 lands on the sign bit, b0 on the exponent's top bit.
__device__ __forceinline__ void decode8(const uint4 v0, const uint4 v1, uint32_t (&r)[32])
{
    const uint32_t wv[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        r[4 * q + 0] = (wv[q] << 6) & 0xC0C0C0C0u;
        r[4 * q + 1] = (wv[q] << 4) & 0xC0C0C0C0u;
        r[4 * q + 2] = (wv[q] << 2) & 0xC0C0C0C0u;
        r[4 * q + 3] = wv[q] & 0xC0C0C0C0u;
    }
}

// Host: 2-D tensor map over rows x kw uint32 words, box = 32 words x
// box_rows rows, 128-byte swizzle (rows of 128 B, 16-byte chunk c of row r
// lands at chunk c ^ (r & 7)).
bool make_code_map(CUtensorMap *m, const uint32_t *codes, int rows, int kw, int box_rows);

}  // namespace mma
}  // namespace tern
