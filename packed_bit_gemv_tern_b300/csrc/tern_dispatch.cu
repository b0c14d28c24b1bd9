// tern_dispatch.cu -- which kernel serves which entry point.
//
// The tensor-core kernel (tern_mma.cu) serves every entry point.  K == 0 (an
// empty sum, y = 0) goes to the CUDA-core kernel, which needs no weight
// stream.  Setting TERN_KERNEL=cuda_core in the environment before the first
// call routes everything to the CUDA-core kernels (tern_cuda.cu) instead; it
// exists to compare the two designs on the same workloads.
#include <cstdlib>
#include <cstring>

#include "tern_internal.cuh"

namespace tern {

static bool use_cuda_core()
{
    static int v = -1;
    if (v < 0) {
        const char *e = std::getenv("TERN_KERNEL");
        v = (e != nullptr && std::strcmp(e, "cuda_core") == 0) ? 1 : 0;
    }
    return v == 1;
}

static tern_status run(const tern_matrix *g, const tern_matrix *u, const uint16_t *x, int m, float *y,
                       cudaStream_t s)
{
    if (g->k == 0 || use_cuda_core()) return gemm_cc(g, u, x, m, y, s);
    return gemm_mma(g, u, x, m, y, s);
}

tern_status gemv_dispatch(const tern_matrix *w, const uint16_t *x, float *y, cudaStream_t s)
{
    return run(w, nullptr, x, 1, y, s);
}

tern_status swiglu_dispatch(const tern_matrix *g, const tern_matrix *u, const uint16_t *x, int m,
                            float *h, cudaStream_t s)
{
    return run(g, u, x, m, h, s);
}

tern_status smallm_dispatch(const tern_matrix *w, const uint16_t *x, int m, float *y, cudaStream_t s)
{
    return run(w, nullptr, x, m, y, s);
}

tern_status batched_dispatch(const tern_batch_item *items, int n, cudaStream_t s)
{
    if (use_cuda_core()) {
        for (int i = 0; i < n; ++i) {
            const tern_status st = gemm_cc(items[i].w, items[i].up, items[i].x, items[i].m, items[i].y, s);
            if (st != TERN_OK) return st;
        }
        return TERN_OK;
    }
    return gemm_batched(items, n, s);
}

tern_status take_device_error()
{
    const tern_status a = take_mma_error();
    const tern_status b = take_batched_error();
    return a != TERN_OK ? a : b;
}

}  // namespace tern
