// tern_host.cpp -- host-side packer, validator and status strings of the C ABI.
//
// The packed format (16 codes per uint32, code j of a word at bits 2j/2j+1,
// (b1,b0) = 00 -> 0, 01 -> +1, 11 -> -1) is this library's own 2-bit layout;
// the Neutrino-1 8B model page keeps its real coded lane proprietary.  The
// per-row metadata (fp32 scale, int32 row sum) follows the page's
// "Where the bytes live" section.
#include <cstdint>
#include <cstring>

#include "tern.h"

namespace {

// Two's complement makes the low two bits of an int8 in {-1, 0, +1} its code:
// 0 -> 00, +1 -> 01, -1 (0xFF) -> 11.
inline bool is_ternary(int8_t v) { return v >= -1 && v <= 1; }

constexpr uint32_t kLowBits = 0x55555555u;  // b0 of every field

inline int popc32(uint32_t v) { return __builtin_popcount(v); }

}  // namespace

extern "C" tern_status tern_pack(const int8_t *t, int32_t rows, int32_t k,
                                 uint32_t *codes, int32_t *rowsum)
{
    if (rows < 0 || k < 0 || (k % 64) != 0) return TERN_ERR_SHAPE;
    if (rows == 0 || k == 0) {
        if (rowsum != nullptr)
            for (int32_t r = 0; r < rows; ++r) rowsum[r] = 0;
        return TERN_OK;
    }
    if (t == nullptr || codes == nullptr) return TERN_ERR_NULL;
    const int64_t wpr = k / 16;
    for (int64_t r = 0; r < rows; ++r) {
        const int8_t *src = t + r * (int64_t)k;
        uint32_t *dst = codes + r * wpr;
        int64_t sum = 0;
        for (int64_t i = 0; i < wpr; ++i) {
            uint32_t w = 0;
            for (int j = 15; j >= 0; --j) {
                const int8_t v = src[i * 16 + j];
                if (!is_ternary(v)) return TERN_ERR_VALUE;
                w = (w << 2) | ((uint32_t)(uint8_t)v & 3u);
                sum += v;
            }
            dst[i] = w;
        }
        if (rowsum != nullptr) rowsum[r] = (int32_t)sum;
    }
    return TERN_OK;
}

extern "C" tern_status tern5_pack(const int8_t *t, int32_t rows, int32_t k, uint8_t *codes, int32_t *rowsum)
{
    if (rows < 0 || k < 0 || (k % 80) != 0) return TERN_ERR_SHAPE;
    if (rows == 0 || k == 0) {
        if (rowsum != nullptr)
            for (int32_t r = 0; r < rows; ++r) rowsum[r] = 0;
        return TERN_OK;
    }
    if (t == nullptr || codes == nullptr) return TERN_ERR_NULL;
    const int64_t bpr = k / 5;
    for (int64_t r = 0; r < rows; ++r) {
        const int8_t *src = t + r * (int64_t)k;
        int64_t sum = 0;
        for (int64_t j = 0; j < bpr; ++j) {
            // Horner from the most significant digit: b = sum_i (t_i + 1) 3^i
            uint32_t b = 0;
            for (int i = 4; i >= 0; --i) {
                const int8_t v = src[5 * j + i];
                if (!is_ternary(v)) return TERN_ERR_VALUE;
                b = 3u * b + (uint32_t)(v + 1);
                sum += v;
            }
            codes[r * bpr + j] = (uint8_t)b;
        }
        if (rowsum != nullptr) rowsum[r] = (int32_t)sum;
    }
    return TERN_OK;
}

extern "C" tern_status tern_validate(const uint32_t *codes, int32_t rows, int32_t k,
                                     const int32_t *rowsum, int64_t counts_out[3])
{
    if (rows < 0 || k < 0 || (k % 64) != 0) return TERN_ERR_SHAPE;
    int64_t nz_total = 0, minus_total = 0;
    if (counts_out != nullptr) counts_out[0] = counts_out[1] = counts_out[2] = 0;
    if (rows > 0 && k > 0 && codes == nullptr) return TERN_ERR_NULL;
    const int64_t wpr = k / 16;
    tern_status st = TERN_OK;
    for (int64_t r = 0; r < rows && st == TERN_OK; ++r) {
        const uint32_t *row = codes + r * wpr;
        int64_t nz = 0, minus = 0;
        for (int64_t i = 0; i < wpr; ++i) {
            const uint32_t w = row[i];
            // A field is invalid when b1 = 1 and b0 = 0.
            if (((w >> 1) & ~w & kLowBits) != 0u) { st = TERN_ERR_BADCODE; break; }
            nz += popc32(w & kLowBits);
            minus += popc32((w >> 1) & kLowBits);
        }
        nz_total += nz;
        minus_total += minus;
        if (st == TERN_OK && rowsum != nullptr && (int64_t)rowsum[r] != nz - 2 * minus)
            st = TERN_ERR_ROWSUM;
    }
    if (counts_out != nullptr) {
        counts_out[0] = (int64_t)rows * k - nz_total;
        counts_out[1] = nz_total - minus_total;
        counts_out[2] = minus_total;
        if (st == TERN_ERR_BADCODE) counts_out[0] = 0;  // partial scan: zeros unknown
    }
    return st;
}

extern "C" const char *tern_status_str(tern_status s)
{
    switch (s) {
    case TERN_OK: return "ok";
    case TERN_ERR_NULL: return "a required pointer is NULL";
    case TERN_ERR_SHAPE: return "bad shape (negative size, k % 64 != 0, size limit or mismatch)";
    case TERN_ERR_ALIGN: return "misaligned pointer";
    case TERN_ERR_BADCODE: return "packed data holds the invalid 2-bit pattern 10";
    case TERN_ERR_ROWSUM: return "stored row sum disagrees with the codes";
    case TERN_ERR_M_RANGE: return "m outside [1, TERN_MAX_M]";
    case TERN_ERR_CUDA: return "CUDA runtime error";
    case TERN_ERR_TIMEOUT: return "a bounded device-side wait ran out";
    case TERN_ERR_VALUE: return "weight outside {-1, 0, +1}";
    }
    return "unknown status";
}

extern "C" int32_t tern_abi_version(void) { return TERN_ABI_VERSION; }
