// tern_base3.cu -- the base-3 packing: five ternary weights per byte
// (1.6 bits a weight against 2 for the 2-bit codes; the model page's
// "Where the bytes live" budget shows a lane that spends more bits per
// weight than a ternary value needs).  Format: a row of K weights (K a
// multiple of 80) is K/5 bytes; byte j holds weights 5j .. 5j+4 as
// b = sum_i (t_{5j+i} + 1) * 3^i, least significant digit first, so b is in
// [0, 242]; 243..255 are invalid.
//
// The GEMV runs on the CUDA cores: a byte's five digits come out by
// division by 3 done as a multiply and a shift ((b * 171) >> 9 == b / 3 for
// b < 256), which has no short bit-operation form like the 2-bit codes'
// masks, so the decode costs several integer operations per weight; each
// decoded weight is used for all m activation rows.
#include <cuda_runtime.h>

#include <cstdint>

#include "tern.h"
#include "tern_internal.cuh"

namespace tern {

namespace {

constexpr int kB3Threads = 256;  // 8 warps; warp w of a block takes rows w, w + 8 * gridDim.x, ...

// y[i][r] = scale[r] * sum_k t[r][k] x[i][k] for i < M.  x is staged in
// shared memory as bf16 ([M][k]); each lane takes 16-byte pieces of the row
// (80 weights), the warp reduces, lane 0 writes.
template <int M>
__global__ void __launch_bounds__(kB3Threads) k_tern5_gemm(const uint8_t *__restrict__ codes,
                                                           const float *__restrict__ scale,
                                                           const uint16_t *__restrict__ x, float *__restrict__ y,
                                                           int rows, int k)
{
    extern __shared__ uint4 xs4[];
    const uint16_t *xs = reinterpret_cast<const uint16_t *>(xs4);
    const int n16 = M * k / 8;  // uint4 pieces of x
    const uint4 *xg = reinterpret_cast<const uint4 *>(x);
    for (int i = (int)threadIdx.x; i < n16; i += kB3Threads) xs4[i] = xg[i];
    __syncthreads();
    const int warp = (int)threadIdx.x >> 5, lane = (int)threadIdx.x & 31;
    const int bytes = k / 5, pieces = bytes / 16;
    for (int r = (int)blockIdx.x * 8 + warp; r < rows; r += (int)gridDim.x * 8) {
        const uint4 *row = reinterpret_cast<const uint4 *>(codes + (size_t)r * bytes);
        float acc[M];
#pragma unroll
        for (int i = 0; i < M; ++i) acc[i] = 0.f;
        for (int pc = lane; pc < pieces; pc += 32) {
            const uint4 v = __ldg(row + pc);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
            const int k0 = pc * 80;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
#pragma unroll
                for (int bi = 0; bi < 4; ++bi) {
                    uint32_t b = (w[q] >> (8 * bi)) & 0xFFu;
                    const int kb = k0 + 20 * q + 5 * bi;
#pragma unroll
                    for (int d = 0; d < 5; ++d) {
                        const uint32_t qt = (b * 171u) >> 9;  // b / 3
                        const uint32_t dig = b - 3u * qt;     // 0, 1, 2
                        b = qt;
                        // weight dig - 1 as a float: 2^23 + 2^22 + dig, less 2^23 + 2^22 + 1
                        const float wt = __int_as_float(0x4B400000 + (int)dig) - 12582913.0f;
#pragma unroll
                        for (int i = 0; i < M; ++i)
                            acc[i] = fmaf(wt, __uint_as_float((uint32_t)xs[i * k + kb + d] << 16), acc[i]);
                    }
                }
            }
        }
#pragma unroll
        for (int i = 0; i < M; ++i) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) acc[i] += __shfl_xor_sync(0xFFFFFFFFu, acc[i], o);
        }
        if (lane == 0) {
            const float sc = scale[r];
#pragma unroll
            for (int i = 0; i < M; ++i) y[(size_t)i * rows + r] = sc * acc[i];
        }
    }
}

// Codes -> int8 weights (a byte above 242 gives -2 in each of its five).
__global__ void k_tern5_unpack(const uint8_t *__restrict__ codes, int8_t *__restrict__ t, long long nbytes)
{
    for (long long j = (long long)blockIdx.x * blockDim.x + threadIdx.x; j < nbytes;
         j += (long long)gridDim.x * blockDim.x) {
        uint32_t b = codes[j];
        const bool bad = b > 242u;
#pragma unroll
        for (int d = 0; d < 5; ++d) {
            const uint32_t qt = (b * 171u) >> 9;
            t[5 * j + d] = bad ? (int8_t)-2 : (int8_t)((int)(b - 3u * qt) - 1);
            b = qt;
        }
    }
}

template <int M>
cudaError_t launch_m(const tern5_matrix *w, const uint16_t *x, float *y, cudaStream_t s)
{
    const size_t smem = (size_t)M * w->k * 2;
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(k_tern5_gemm<M>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return cudaErrorInvalidValue;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int need = (w->rows + 7) / 8;
    const int grid = need < 2 * sms ? need : 2 * sms;
    k_tern5_gemm<M><<<grid, kB3Threads, smem, s>>>(w->codes, w->scale, x, y, w->rows, w->k);
    return cudaGetLastError();
}

}  // namespace

tern_status tern5_gemm_launch(const tern5_matrix *w, const uint16_t *x, int m, float *y, cudaStream_t s)
{
    cudaError_t e = cudaSuccess;
    switch (m) {
    case 1: e = launch_m<1>(w, x, y, s); break;
    case 2: e = launch_m<2>(w, x, y, s); break;
    case 3: e = launch_m<3>(w, x, y, s); break;
    case 4: e = launch_m<4>(w, x, y, s); break;
    case 5: e = launch_m<5>(w, x, y, s); break;
    case 6: e = launch_m<6>(w, x, y, s); break;
    case 7: e = launch_m<7>(w, x, y, s); break;
    default: e = launch_m<8>(w, x, y, s); break;
    }
    return e == cudaSuccess ? TERN_OK : TERN_ERR_CUDA;
}

tern_status tern5_unpack_launch(const tern5_matrix *w, int8_t *t, cudaStream_t s)
{
    const long long nbytes = (long long)w->rows * (w->k / 5);
    if (nbytes == 0) return TERN_OK;
    long long blocks = (nbytes + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    k_tern5_unpack<<<(unsigned)blocks, 256, 0, s>>>(w->codes, t, nbytes);
    return cudaGetLastError() == cudaSuccess ? TERN_OK : TERN_ERR_CUDA;
}

}  // namespace tern
