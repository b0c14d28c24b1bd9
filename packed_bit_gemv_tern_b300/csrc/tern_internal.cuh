// tern_internal.cuh -- declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "tern.h"

namespace tern {

constexpr int kCcThreads = 256;  // CUDA-core kernels: 8 warps per CTA

int sm_count();
tern_status check_matrix(const tern_matrix *w);

// CUDA-core kernels (tern_cuda.cu); u == nullptr means a plain projection.
tern_status gemm_cc(const tern_matrix *g, const tern_matrix *u, const uint16_t *x, int m, float *y,
                    cudaStream_t s);

// Tensor-core kernels (tern_mma.cu); same contract as gemm_cc.
tern_status gemm_mma(const tern_matrix *g, const tern_matrix *u, const uint16_t *x, int m, float *y,
                     cudaStream_t s);
tern_status take_mma_error();

// Persistent batched kernel (tern_batched.cu); items already checked.
// Number of kernel launches gemm_batched makes for these items (host only).
int batched_launches(const tern_batch_item *items, int n);
tern_status gemm_batched(const tern_batch_item *items, int n, cudaStream_t s);
// As gemm_batched, with the prepared activations in a fixed module-scope
// scratch of TERN_NOALLOC_WS_BYTES (TERN_ERR_SHAPE, nothing launched, if a
// launch group needs more).
tern_status gemm_batched_noalloc(const tern_batch_item *items, int n, cudaStream_t s);
tern_status take_batched_error();

// Shared argument checks (tern_cuda.cu).
tern_status check_gemm_args(const tern_matrix *g, const tern_matrix *u, const uint16_t *x, int32_t m,
                            const float *y);

// Kernel choice per entry point (tern_dispatch.cu).
tern_status gemv_dispatch(const tern_matrix *w, const uint16_t *x, float *y, cudaStream_t s);
tern_status swiglu_dispatch(const tern_matrix *g, const tern_matrix *u, const uint16_t *x, int m,
                            float *h, cudaStream_t s);
tern_status smallm_dispatch(const tern_matrix *w, const uint16_t *x, int m, float *y, cudaStream_t s);
tern_status batched_dispatch(const tern_batch_item *items, int n, cudaStream_t s);

// Reads and clears every device error word (TERN_OK when all are clear).
tern_status take_device_error();

}  // namespace tern
