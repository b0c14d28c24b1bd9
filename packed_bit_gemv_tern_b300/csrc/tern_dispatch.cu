// tern_dispatch.cu -- which kernel serves which entry point.
#include "tern_internal.cuh"

namespace tern {

tern_status gemv_dispatch(const tern_matrix *w, const uint16_t *x, float *y, cudaStream_t s)
{
    return gemm_cc(w, nullptr, x, 1, y, s);
}

tern_status swiglu_dispatch(const tern_matrix *g, const tern_matrix *u, const uint16_t *x, int m,
                            float *h, cudaStream_t s)
{
    return gemm_cc(g, u, x, m, h, s);
}

tern_status smallm_dispatch(const tern_matrix *w, const uint16_t *x, int m, float *y, cudaStream_t s)
{
    return gemm_cc(w, nullptr, x, m, y, s);
}

tern_status take_device_error() { return TERN_OK; }

}  // namespace tern
