// tern_cuda.cu -- host side of the C ABI's device entry points: argument
// checks, the choice of kernel, the debug unpack kernel and the empty-sum
// kernel.
//
// What is computed (Neutrino-1 8B model page, intro and "Where the bytes
// live"): y[m][r] = scale[r] * sum_k t[r][k] * x[m][k] with t in {-1,0,+1}
// stored 2 bits per weight and decoded inside the kernel; the gated pair
// h = silu(gate x) * (up x) follows the spec table's SwiGLU feed-forward.
// Every product with K > 0 runs on the tensor-core kernels (tern_mma.cu for
// one product per call, tern_batched.cu for batches); K == 0 has no weights
// to stream and is written by k_empty_sum.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "tern.h"
#include "tern_internal.cuh"
#include "tern_mma_common.cuh"

namespace tern {

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

// K == 0: every sum is empty, so y[i][r] = scale[r] * 0 and, for a SwiGLU
// pair, h[i][r] = silu(scale_g[r] * 0) * (scale_u[r] * 0).  No weight is read.
__global__ void k_empty_sum(const float *__restrict__ sg, const float *__restrict__ su, float *__restrict__ y,
                            int rows, int m)
{
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (int64_t)rows * m) return;
    const int r = (int)(i % rows);
    const float g = sg[r] * 0.0f;
    y[i] = su == nullptr ? g : (g / (1.0f + expf(-g))) * (su[r] * 0.0f);
}

// ---------------------------------------------------------------------------
// Launch helpers
// ---------------------------------------------------------------------------

// Driver entry points reached through the runtime (the library does not link
// the driver library itself, so it also loads on a machine without one).
template <typename F>
static F driver_fn(const char *name)
{
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return reinterpret_cast<F>(p);
}

unsigned long long current_context_id()
{
    using GetCurrent = CUresult (*)(CUcontext *);
    using GetId = CUresult (*)(CUcontext, unsigned long long *);
    static const GetCurrent get_current = driver_fn<GetCurrent>("cuCtxGetCurrent");
    static const GetId get_id = driver_fn<GetId>("cuCtxGetId");
    if (get_current == nullptr || get_id == nullptr) return 0;
    CUcontext c = nullptr;
    if (get_current(&c) != CUDA_SUCCESS || c == nullptr) return 0;
    unsigned long long id = 0;
    if (get_id(c, &id) != CUDA_SUCCESS) return 0;
    return id;
}

static std::atomic<long long> g_wait_limit{mma::kWaitCycles};

long long wait_limit() { return g_wait_limit.load(std::memory_order_relaxed); }

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

// One product (a plain projection when u == nullptr, else a SwiGLU pair):
// K == 0 has nothing to stream, everything else runs on the tensor cores.
static tern_status run_product(const tern_matrix *g, const tern_matrix *u, const uint16_t *x, int m, float *y,
                               cudaStream_t s)
{
    if (g->k == 0) return empty_sum(g, u, m, y, s);
    return gemm_mma(g, u, x, m, y, s);
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
    return run_product(w, nullptr, x, 1, y, (cudaStream_t)stream);
}

extern "C" tern_status tern_gemv_swiglu(const tern_matrix *gate, const tern_matrix *up,
                                        const uint16_t *x, float *h, void *stream)
{
    if (up == nullptr) return TERN_ERR_NULL;
    tern_status st = check_gemm_args(gate, up, x, 1, h);
    if (st != TERN_OK || gate->rows == 0) return st;
    return run_product(gate, up, x, 1, h, (cudaStream_t)stream);
}

extern "C" tern_status tern_gemm_smallm(const tern_matrix *w, const uint16_t *x, int32_t m,
                                        float *y, void *stream)
{
    tern_status st = check_gemm_args(w, nullptr, x, m, y);
    if (st != TERN_OK || w->rows == 0) return st;
    return run_product(w, nullptr, x, m, y, (cudaStream_t)stream);
}

extern "C" tern_status tern_gemm_smallm_swiglu(const tern_matrix *gate, const tern_matrix *up,
                                               const uint16_t *x, int32_t m, float *h, void *stream)
{
    if (up == nullptr) return TERN_ERR_NULL;
    tern_status st = check_gemm_args(gate, up, x, m, h);
    if (st != TERN_OK || gate->rows == 0) return st;
    return run_product(gate, up, x, m, h, (cudaStream_t)stream);
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
    return gemm_batched(items, n, (cudaStream_t)stream);
}

extern "C" tern_status tern_gemm_batched_rmsnorm(const tern_batch_item *items, const float *const *norm_w, float eps,
                                                 int32_t n, void *stream)
{
    const tern_status st = check_batch(items, n);
    if (st != TERN_OK || n == 0) return st;
    if (norm_w == nullptr) return TERN_ERR_NULL;
    if (!(eps >= 0.f && eps <= 3.4e38f)) return TERN_ERR_VALUE;  // also rejects NaN and +inf
    for (int32_t i = 0; i < n; ++i)
        if (norm_w[i] != nullptr && (reinterpret_cast<uintptr_t>(norm_w[i]) & 15u) != 0) return TERN_ERR_ALIGN;
    return gemm_batched_rmsnorm(items, norm_w, eps, n, (cudaStream_t)stream);
}

// Checks of a base-3 matrix: shape, pointers, alignment (codes 16 bytes).
static tern_status check5(const tern5_matrix *w)
{
    if (w == nullptr) return TERN_ERR_NULL;
    if (w->rows < 0 || w->k < 0 || w->k % 80 != 0) return TERN_ERR_SHAPE;
    if (w->rows == 0 || w->k == 0) return TERN_OK;
    if (w->codes == nullptr || w->scale == nullptr) return TERN_ERR_NULL;
    if (!aligned(w->codes, 16) || !aligned(w->scale, 4)) return TERN_ERR_ALIGN;
    return TERN_OK;
}

extern "C" tern_status tern5_gemm(const tern5_matrix *w, const uint16_t *x, int32_t m, float *y, void *stream)
{
    tern_status st = check5(w);
    if (st != TERN_OK) return st;
    if (m < 1 || m > TERN_MAX_M) return TERN_ERR_M_RANGE;
    if (w->rows == 0) return TERN_OK;
    if ((int64_t)m * w->k * 2 > TERN_MAX_X_BYTES) return TERN_ERR_SHAPE;
    if (x == nullptr || y == nullptr) return TERN_ERR_NULL;
    if (!aligned(x, 16) || !aligned(y, 4)) return TERN_ERR_ALIGN;
    if (w->k == 0) {  // y = scale * 0
        const tern_matrix z = {w->rows, 0, nullptr, w->scale, nullptr};
        return empty_sum(&z, nullptr, m, y, (cudaStream_t)stream);
    }
    return tern5_gemm_launch(w, x, m, y, (cudaStream_t)stream);
}

extern "C" tern_status tern5_unpack(const tern5_matrix *w, int8_t *t_out, void *stream)
{
    const tern_status st = check5(w);
    if (st != TERN_OK) return st;
    if (w->rows == 0 || w->k == 0) return TERN_OK;
    if (t_out == nullptr) return TERN_ERR_NULL;
    return tern5_unpack_launch(w, t_out, (cudaStream_t)stream);
}

extern "C" tern_status tern_lmhead_argmax(const tern_i8_matrix *w, const uint16_t *x, int32_t m, const float *norm_w,
                                          float eps, float *logits, int32_t *argmax, void *stream)
{
    if (w == nullptr || w->w == nullptr || w->scale == nullptr || x == nullptr || logits == nullptr ||
        argmax == nullptr)
        return TERN_ERR_NULL;
    if (w->rows < 1 || w->k < 64 || w->k % 64 != 0) return TERN_ERR_SHAPE;
    if (m < 1 || m > TERN_MAX_M) return TERN_ERR_M_RANGE;
    if ((int64_t)m * w->k * 2 > TERN_MAX_X_BYTES) return TERN_ERR_SHAPE;
    if (!aligned(w->w, 16) || !aligned(w->scale, 4) || !aligned(x, 16) || !aligned(logits, 4) || !aligned(argmax, 4) ||
        (norm_w != nullptr && !aligned(norm_w, 16)))
        return TERN_ERR_ALIGN;
    if (!(eps >= 0.f && eps <= 3.4e38f)) return TERN_ERR_VALUE;
    return head_argmax(w, x, m, norm_w, eps, logits, argmax, (cudaStream_t)stream);
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

extern "C" void tern_set_wait_limit(int64_t cycles)
{
    g_wait_limit.store(cycles > 0 ? (long long)cycles : mma::kWaitCycles, std::memory_order_relaxed);
}

extern "C" tern_status tern_last_device_error(void *stream)
{
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return TERN_ERR_CUDA;
    if (cudaGetLastError() != cudaSuccess) return TERN_ERR_CUDA;
    return take_device_error();
}

namespace tern {

tern_status empty_sum(const tern_matrix *g, const tern_matrix *u, int m, float *y, cudaStream_t s)
{
    const int64_t n = (int64_t)g->rows * m;
    if (n == 0) return TERN_OK;
    const int threads = 256;
    k_empty_sum<<<(unsigned)((n + threads - 1) / threads), threads, 0, s>>>(g->scale, u ? u->scale : nullptr, y,
                                                                             g->rows, m);
    return cudaGetLastError() == cudaSuccess ? TERN_OK : TERN_ERR_CUDA;
}

tern_status take_device_error()
{
    const tern_status a = take_mma_error();
    const tern_status b = take_batched_error();
    return a != TERN_OK ? a : b;
}

}  // namespace tern
