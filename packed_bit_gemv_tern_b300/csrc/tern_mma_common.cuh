// tern_mma_common.cuh -- pieces shared by the tensor-core kernels: operand
// encodings, descriptors, bounded waits and tensor-map creation.
//
// The weights enter the MMA as e4m3 bytes of exactly +2, -2 or 0 built from
// the packed 2-bit codes with one shift and one AND per four codes; the
// activations enter as two e4m3 terms per value (see split_pair).  The MMA is
// tcgen05 kind::f8f6f4 with fp32 accumulation in tensor memory.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "tern_ptx.cuh"

namespace tern {
namespace mma {

constexpr int kStageWords = 32;         // words per row per TMA stage (512 codes, 128 B)
constexpr int kStageBytes = 128 * 128;  // one stage of a 128-row tile
constexpr int kBBytesPerWord = 256;     // B operand: 16 rows x 16 e4m3 per word (16 k)
constexpr int kSmemLimit = 227 * 1024;

// Instruction descriptor: kind::f8f6f4, D fp32, A e4m3, B e4m3, both
// K-major, N = 16, M = 128.
constexpr uint32_t kIdesc = (1u << 4) | (0u << 7) | (0u << 10) | ((16u >> 3) << 17) | ((128u >> 4) << 24);

// Shared-memory descriptor of a K-major, unswizzled operand made of 8-row x
// 16-byte core matrices: adjacent core matrices along K are 256 B apart (LBO),
// along N 128 B apart (SBO).
__device__ __forceinline__ uint64_t b_desc(uint32_t addr)
{
    return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)(256u >> 4) << 16) | ((uint64_t)(128u >> 4) << 32) |
           (1ull << 46);
}

// Descriptor of a K-major, unswizzled B operand whose 16-code blocks sit
// `lbo` bytes apart (rows 0-7 of a block at +0, rows 8-15 at +128).
__device__ __forceinline__ uint64_t b_desc_lbo(uint32_t addr, uint32_t lbo)
{
    return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)(128u >> 4) << 32) | (1ull << 46);
}

// Spin on an mbarrier phase with a time bound (~1 s).  On time-out the
// kernel's error word and the CTA's abort flag are set; once the abort flag is
// up every later wait returns false at once.
struct Waiter {
    volatile uint32_t *abort_flag;  // shared
    unsigned int *err;              // global error word of the kernel
    // Each try sleeps until the phase completes or kSleepNs pass; the abort
    // flag and the one-second bound are checked between tries.
    static constexpr uint32_t kSleepNs = 1000000u;
    __device__ __forceinline__ bool wait(uint32_t bar, uint32_t parity) const
    {
        if (*abort_flag) return false;
        if (ptx::mbar_try_wait(bar, parity)) return true;
        const long long t0 = clock64();
        while (!ptx::mbar_try_wait_sleep(bar, parity, kSleepNs)) {
            if (*abort_flag) return false;
            if (clock64() - t0 > (1ll << 31)) {
                atomicOr(err, 1u);
                *abort_flag = 1u;
                return false;
            }
        }
        return true;
    }
};

// Bounded wait that ignores the abort flag (used to drain in-flight work).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, unsigned int *err)
{
    const long long t0 = clock64();
    while (!ptx::mbar_try_wait_sleep(bar, parity, Waiter::kSleepNs)) {
        if (clock64() - t0 > (1ll << 31)) {
            atomicOr(err, 1u);
            return;
        }
    }
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + expf(-z)); }

// 2^e as an fp32 (e in [-126, 127]).
__device__ __forceinline__ float exp2i(int e) { return __int_as_float((e + 127) << 23); }

// Per-row scale exponent s for a row whose largest |x| has fp32 bits mb:
// the maximum lands in [128, 256) after multiplying by 2^s.
__device__ __forceinline__ int row_scale_exp(uint32_t mb)
{
    const int e = mb == 0u ? 0 : (int)(mb >> 23) - 127;
    return min(max(7 - e, -120), 120);
}

// Largest |x| (fp32 bits of the magnitude) among 16 bf16 values.
__device__ __forceinline__ uint32_t max_abs16(const uint4 a, const uint4 b)
{
    const uint32_t v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t mx = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) mx = max(mx, max((v[q] << 16) & 0x7FFF0000u, v[q] & 0x7FFF0000u));
    return mx;
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

// One word (16 k) of one activation row -> the 16-byte hi and lo rows of the
// B operand, in the column order the weight decode produces: byte b of
// output word j holds k offset 4b + j (a 4x4 transpose).
__device__ __forceinline__ void split_word(const uint4 a, const uint4 b, float sc, uint4 &hi4, uint4 &lo4)
{
    const uint32_t v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t hp[8], lp[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) split_pair(v[q], sc, hp[q], lp[q]);
    const uint32_t h02 = hp[0] | (hp[2] << 16), h46 = hp[4] | (hp[6] << 16);
    const uint32_t h13 = hp[1] | (hp[3] << 16), h57 = hp[5] | (hp[7] << 16);
    const uint32_t l02 = lp[0] | (lp[2] << 16), l46 = lp[4] | (lp[6] << 16);
    const uint32_t l13 = lp[1] | (lp[3] << 16), l57 = lp[5] | (lp[7] << 16);
    hi4 = make_uint4(__byte_perm(h02, h46, 0x6420), __byte_perm(h02, h46, 0x7531), __byte_perm(h13, h57, 0x6420),
                     __byte_perm(h13, h57, 0x7531));
    lo4 = make_uint4(__byte_perm(l02, l46, 0x6420), __byte_perm(l02, l46, 0x7531), __byte_perm(l13, l57, 0x6420),
                     __byte_perm(l13, l57, 0x7531));
}

// Byte offset of B row n (0..15) inside one word's 256-byte block.
__device__ __forceinline__ uint32_t b_row_off(int n) { return (uint32_t)((n >> 3) * 128 + (n & 7) * 16); }

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
