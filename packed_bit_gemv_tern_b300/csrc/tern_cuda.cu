// tern_cuda.cu -- device entry points of the C ABI and their CUDA kernels.
//
// What is computed (Neutrino-1 8B model page, intro and "Where the bytes
// live"): y[m][r] = scale[r] * sum_k t[r][k] * x[m][k] with t in {-1,0,+1}
// stored 2 bits per weight and decoded inside the kernel; the gated pair
// h = silu(gate x) * (up x) follows the spec table's SwiGLU feed-forward.
//
// This file holds the CUDA-core kernels: the packed-weight stream is read
// with 128-bit read-only loads, every 2-bit code is decoded with bit
// operations into a sign-selected add of the activation (no multiply by a
// weight), partial sums stay in fp32 registers and warps reduce with shuffles.
#include <cuda_runtime.h>

#include <cstdint>

#include "tern.h"
#include "tern_internal.cuh"

namespace tern {

// ---------------------------------------------------------------------------
// Device helpers
// ---------------------------------------------------------------------------

// Streaming 128-bit load of packed weights: read-only path, no L1 allocation
// (each weight byte is used once per call).
__device__ __forceinline__ uint4 ld_stream_u4(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ float bf16lo(uint32_t pair) { return __uint_as_float(pair << 16); }
__device__ __forceinline__ float bf16hi(uint32_t pair) { return __uint_as_float(pair & 0xFFFF0000u); }

// Sign-select for one 2-bit field c = (b1,b0): b0 keeps x, b1 flips its sign.
// Valid fields: 00 -> +0/-0 contribution of magnitude 0, 01 -> x, 11 -> -x.
// The invalid field 10 contributes 0.  Done entirely with integer bit ops on
// the fp32 pattern of x: mask = -(b0) keeps or clears every bit, and b1 is
// moved onto the sign bit.
__device__ __forceinline__ float sign_select(uint32_t field, float x)
{
    const uint32_t b0 = field & 1u;
    const uint32_t keep = 0u - b0;                 // all ones when b0 = 1
    const uint32_t flip = (field & 2u) << 30;      // b1 onto bit 31
    return __uint_as_float((__float_as_uint(x) & keep) ^ (flip & keep));
}

__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }

template <int M>
__device__ __forceinline__ void warp_reduce(float (&a)[M])
{
#pragma unroll
    for (int m = 0; m < M; ++m) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) a[m] += __shfl_xor_sync(0xFFFFFFFFu, a[m], o);
    }
}

// Accumulate the 64 codes of one 128-bit chunk against M activation rows.
// xs points at column 64*q of activation row 0 in shared memory; rows are
// `ldx` bf16 apart.
template <int M>
__device__ __forceinline__ void accumulate_chunk(const uint4 w4, const uint16_t *xs, int ldx,
                                                 float (&acc)[M])
{
    const uint32_t words[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t w = words[i];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
            for (int m = 0; m < M; ++m) {
                const uint4 xv = *reinterpret_cast<const uint4 *>(xs + (size_t)m * ldx + 16 * i + 8 * h);
                const uint32_t xp[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int code = 8 * h + 2 * j;
                    acc[m] += sign_select(w >> (2 * code), bf16lo(xp[j]));
                    acc[m] += sign_select(w >> (2 * (code + 1)), bf16hi(xp[j]));
                }
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Kernels
// ---------------------------------------------------------------------------

// One thread per packed word: 16 int8 values, sign-extended 2-bit fields
// (00 -> 0, 01 -> 1, 11 -> -1, invalid 10 -> -2).
__global__ void k_unpack(const uint32_t *__restrict__ codes, int8_t *__restrict__ t, int64_t words)
{
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= words) return;
    const uint32_t w = codes[i];
    uint32_t out[4];
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        uint32_t v = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int code = 4 * b + j;
            const int32_t s = ((int32_t)(w << (30 - 2 * code))) >> 30;
            v |= ((uint32_t)s & 0xFFu) << (8 * j);
        }
        out[b] = v;
    }
    reinterpret_cast<uint4 *>(t)[i] = make_uint4(out[0], out[1], out[2], out[3]);
}

// CUDA-core ternary GEMM for M activation rows (M = 1 is the GEMV).
// Activations are staged once per CTA into shared memory as bf16 [M][k].
// One warp per output row at a time; lane l handles 128-bit chunks
// l, l+32, ... of the row.  With SWIGLU the same warp streams the gate row
// and the up row and writes silu(g) * u.
template <int M, bool SWIGLU>
__global__ void __launch_bounds__(kCcThreads)
k_gemm_cc(const uint32_t *__restrict__ cg, const float *__restrict__ sg,
          const uint32_t *__restrict__ cu, const float *__restrict__ su,
          const uint16_t *__restrict__ x, float *__restrict__ y, int rows, int k)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    uint16_t *xs = reinterpret_cast<uint16_t *>(smem_raw);
    const int nvec = (M * k) >> 3;  // 8 bf16 per 16-byte vector
    for (int i = threadIdx.x; i < nvec; i += blockDim.x)
        reinterpret_cast<uint4 *>(xs)[i] = reinterpret_cast<const uint4 *>(x)[i];
    __syncthreads();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int warps = blockDim.x >> 5;
    const int64_t wpr = k >> 4;
    const int chunks = k >> 6;
    for (int r = blockIdx.x * warps + warp; r < rows; r += gridDim.x * warps) {
        float ag[M], au[M];
#pragma unroll
        for (int m = 0; m < M; ++m) { ag[m] = 0.f; au[m] = 0.f; }
        const uint4 *rg = reinterpret_cast<const uint4 *>(cg + (int64_t)r * wpr);
        const uint4 *ru = SWIGLU ? reinterpret_cast<const uint4 *>(cu + (int64_t)r * wpr) : nullptr;
        for (int q = lane; q < chunks; q += 32) {
            const uint4 wg = ld_stream_u4(rg + q);
            accumulate_chunk<M>(wg, xs + 64 * q, k, ag);
            if constexpr (SWIGLU) {
                const uint4 wu = ld_stream_u4(ru + q);
                accumulate_chunk<M>(wu, xs + 64 * q, k, au);
            }
        }
        warp_reduce<M>(ag);
        if constexpr (SWIGLU) warp_reduce<M>(au);
        if (lane == 0) {
#pragma unroll
            for (int m = 0; m < M; ++m) {
                if constexpr (SWIGLU) {
                    const float g = sg[r] * ag[m];
                    const float u = su[r] * au[m];
                    y[(int64_t)m * rows + r] = silu(g) * u;
                } else {
                    y[(int64_t)m * rows + r] = sg[r] * ag[m];
                }
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Launch helpers
// ---------------------------------------------------------------------------

int sm_count()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    static int cached[64] = {0};
    if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    if (dev >= 0 && dev < 64) cached[dev] = n;
    return n;
}

template <typename K>
static cudaError_t allow_smem(K kernel, size_t bytes)
{
    if (bytes <= 48 * 1024) return cudaSuccess;
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

template <int M, bool SWIGLU>
static tern_status launch_cc(const tern_matrix *g, const tern_matrix *u, const uint16_t *x,
                             float *y, cudaStream_t s)
{
    const int rows = g->rows, k = g->k;
    const size_t smem = (size_t)M * k * sizeof(uint16_t);
    auto kern = k_gemm_cc<M, SWIGLU>;
    if (allow_smem(kern, smem) != cudaSuccess) return TERN_ERR_CUDA;
    const int warps = kCcThreads / 32;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kCcThreads, smem) != cudaSuccess || per_sm < 1)
        per_sm = 1;
    int64_t want = ((int64_t)rows + warps - 1) / warps;
    int64_t cap = (int64_t)sm_count() * per_sm;
    const int grid = (int)(want < cap ? want : cap);
    kern<<<grid, kCcThreads, smem, s>>>(g->codes, g->scale, SWIGLU ? u->codes : nullptr,
                                        SWIGLU ? u->scale : nullptr, x, y, rows, k);
    return cudaGetLastError() == cudaSuccess ? TERN_OK : TERN_ERR_CUDA;
}

template <bool SWIGLU>
static tern_status dispatch_cc(int m, const tern_matrix *g, const tern_matrix *u, const uint16_t *x,
                               float *y, cudaStream_t s)
{
    switch (m) {
    case 1: return launch_cc<1, SWIGLU>(g, u, x, y, s);
    case 2: return launch_cc<2, SWIGLU>(g, u, x, y, s);
    case 3: return launch_cc<3, SWIGLU>(g, u, x, y, s);
    case 4: return launch_cc<4, SWIGLU>(g, u, x, y, s);
    case 5: return launch_cc<5, SWIGLU>(g, u, x, y, s);
    case 6: return launch_cc<6, SWIGLU>(g, u, x, y, s);
    case 7: return launch_cc<7, SWIGLU>(g, u, x, y, s);
    case 8: return launch_cc<8, SWIGLU>(g, u, x, y, s);
    }
    return TERN_ERR_M_RANGE;
}

// ---------------------------------------------------------------------------
// Argument checks (host)
// ---------------------------------------------------------------------------

static bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Shape / pointer / alignment rules shared by every device entry point.
tern_status check_matrix(const tern_matrix *w)
{
    if (w == nullptr) return TERN_ERR_NULL;
    if (w->rows < 0 || w->k < 0 || (w->k % 64) != 0) return TERN_ERR_SHAPE;
    if (w->rows == 0) return TERN_OK;
    if (w->scale == nullptr) return TERN_ERR_NULL;
    if (w->k > 0 && w->codes == nullptr) return TERN_ERR_NULL;
    if (!aligned(w->codes, 16) || !aligned(w->scale, 4)) return TERN_ERR_ALIGN;
    return TERN_OK;
}

tern_status check_gemm_args(const tern_matrix *g, const tern_matrix *u, const uint16_t *x, int32_t m,
                            const float *y)
{
    tern_status st = check_matrix(g);
    if (st != TERN_OK) return st;
    if (u != nullptr) {
        if ((st = check_matrix(u)) != TERN_OK) return st;
        if (u->rows != g->rows || u->k != g->k) return TERN_ERR_SHAPE;
    }
    if (m < 1 || m > TERN_MAX_M) return TERN_ERR_M_RANGE;
    if ((int64_t)m * g->k * 2 > TERN_MAX_X_BYTES) return TERN_ERR_SHAPE;
    if (g->rows == 0) return TERN_OK;
    if (y == nullptr) return TERN_ERR_NULL;
    if (g->k > 0 && x == nullptr) return TERN_ERR_NULL;
    if (!aligned(x, 16) || !aligned(y, 4)) return TERN_ERR_ALIGN;
    return TERN_OK;
}

}  // namespace tern

using namespace tern;

// ---------------------------------------------------------------------------
// C ABI
// ---------------------------------------------------------------------------

extern "C" tern_status tern_unpack(const tern_matrix *w, int8_t *t_out, void *stream)
{
    tern_status st = check_matrix(w);
    if (st != TERN_OK) return st;
    if (w->rows == 0 || w->k == 0) return TERN_OK;
    if (t_out == nullptr) return TERN_ERR_NULL;
    if (!aligned(t_out, 16)) return TERN_ERR_ALIGN;
    const int64_t words = (int64_t)w->rows * (w->k / 16);
    const int threads = 256;
    const int64_t blocks = (words + threads - 1) / threads;
    k_unpack<<<(unsigned)blocks, threads, 0, (cudaStream_t)stream>>>(w->codes, t_out, words);
    return cudaGetLastError() == cudaSuccess ? TERN_OK : TERN_ERR_CUDA;
}

extern "C" tern_status tern_gemv(const tern_matrix *w, const uint16_t *x, float *y, void *stream)
{
    tern_status st = check_gemm_args(w, nullptr, x, 1, y);
    if (st != TERN_OK || w->rows == 0) return st;
    return gemv_dispatch(w, x, y, (cudaStream_t)stream);
}

extern "C" tern_status tern_gemv_swiglu(const tern_matrix *gate, const tern_matrix *up,
                                        const uint16_t *x, float *h, void *stream)
{
    if (up == nullptr) return TERN_ERR_NULL;
    tern_status st = check_gemm_args(gate, up, x, 1, h);
    if (st != TERN_OK || gate->rows == 0) return st;
    return swiglu_dispatch(gate, up, x, 1, h, (cudaStream_t)stream);
}

extern "C" tern_status tern_gemm_smallm(const tern_matrix *w, const uint16_t *x, int32_t m,
                                        float *y, void *stream)
{
    tern_status st = check_gemm_args(w, nullptr, x, m, y);
    if (st != TERN_OK || w->rows == 0) return st;
    return smallm_dispatch(w, x, m, y, (cudaStream_t)stream);
}

extern "C" tern_status tern_gemm_smallm_swiglu(const tern_matrix *gate, const tern_matrix *up,
                                               const uint16_t *x, int32_t m, float *h, void *stream)
{
    if (up == nullptr) return TERN_ERR_NULL;
    tern_status st = check_gemm_args(gate, up, x, m, h);
    if (st != TERN_OK || gate->rows == 0) return st;
    return swiglu_dispatch(gate, up, x, m, h, (cudaStream_t)stream);
}

// Checks every item of a batch as the single calls do.
static tern_status check_batch(const tern_batch_item *items, int32_t n)
{
    if (n < 0) return TERN_ERR_SHAPE;
    if (n == 0) return TERN_OK;
    if (items == nullptr) return TERN_ERR_NULL;
    for (int32_t i = 0; i < n; ++i) {
        const tern_batch_item &b = items[i];
        const tern_status st = check_gemm_args(b.w, b.up, b.x, b.m, b.y);
        if (st != TERN_OK) return st;
    }
    return TERN_OK;
}

extern "C" tern_status tern_gemm_batched(const tern_batch_item *items, int32_t n, void *stream)
{
    const tern_status st = check_batch(items, n);
    if (st != TERN_OK || n == 0) return st;
    return batched_dispatch(items, n, (cudaStream_t)stream);
}

extern "C" tern_status tern_gemm_batched_noalloc(const tern_batch_item *items, int32_t n, void *stream)
{
    const tern_status st = check_batch(items, n);
    if (st != TERN_OK || n == 0) return st;
    return gemm_batched_noalloc(items, n, (cudaStream_t)stream);
}

extern "C" int32_t tern_gemm_batched_launches(const tern_batch_item *items, int32_t n)
{
    if (n < 0) return -(int32_t)TERN_ERR_SHAPE;
    if (n == 0) return 0;
    if (items == nullptr) return -(int32_t)TERN_ERR_NULL;
    for (int32_t i = 0; i < n; ++i)
        if (items[i].w == nullptr) return -(int32_t)TERN_ERR_NULL;
    return batched_launches(items, n);
}

extern "C" tern_status tern_last_device_error(void *stream)
{
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return TERN_ERR_CUDA;
    if (cudaGetLastError() != cudaSuccess) return TERN_ERR_CUDA;
    return take_device_error();
}

namespace tern {

tern_status gemm_cc(const tern_matrix *g, const tern_matrix *u, const uint16_t *x, int m, float *y,
                    cudaStream_t s)
{
    return u ? dispatch_cc<true>(m, g, u, x, y, s) : dispatch_cc<false>(m, g, nullptr, x, y, s);
}

}  // namespace tern
