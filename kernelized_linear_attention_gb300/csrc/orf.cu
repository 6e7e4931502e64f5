// Orthogonal random features for FAVOR+ ("The Kernel Zoo", §5.1 and §5.3;
// "Performer", §2 Step 4).
//
// One thread block per d x d Gaussian block.  Rows are orthonormalised in
// order: row i loses its components along the finished rows 0..i-1 (all
// coefficients taken from the same row state, repeated once more to undo
// rounding), then is scaled to unit length.  Row g of the stacked result is
// finally scaled to the length of gauss_lengths[g], a chi(d) draw, so each
// row has the length distribution of a Gaussian vector.  fp64 throughout,
// rounded to fp32 on store.
#include "internal.h"

namespace la {

namespace {

constexpr int kOrfThreads = 128;

__device__ double block_sum(double x, double* red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    __syncthreads();
    if (lane == 0) red[warp] = x;
    __syncthreads();
    double t = 0.0;
    for (int w = 0; w < kOrfThreads / 32; ++w) t += red[w];
    return t;
}

__global__ void __launch_bounds__(kOrfThreads) orf_kernel(const double* blocks, const double* lengths,
                                                          int r, int d, float* omega) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    double* Qm = reinterpret_cast<double*>(smem_raw);   // [d][d]
    double* coef = Qm + (size_t)d * d;                  // [d]
    __shared__ double red[kOrfThreads / 32];
    const int b = blockIdx.x;
    const double* src = blocks + (size_t)b * d * d;
    for (int i = threadIdx.x; i < d * d; i += kOrfThreads) Qm[i] = src[i];
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int rows = min(d, r - b * d);
    for (int i = 0; i < rows; ++i) {
        double* row = Qm + (size_t)i * d;
        for (int pass = 0; pass < 2 && i > 0; ++pass) {
            for (int j = warp; j < i; j += kOrfThreads / 32) {
                const double* qj = Qm + (size_t)j * d;
                double acc = 0.0;
                for (int c = lane; c < d; c += 32) acc = fma(qj[c], row[c], acc);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
                if (lane == 0) coef[j] = acc;
            }
            __syncthreads();
            for (int c = threadIdx.x; c < d; c += kOrfThreads) {
                double acc = row[c];
                for (int j = 0; j < i; ++j) acc = fma(-coef[j], Qm[(size_t)j * d + c], acc);
                row[c] = acc;
            }
            __syncthreads();
        }
        double ss = 0.0;
        for (int c = threadIdx.x; c < d; c += kOrfThreads) ss = fma(row[c], row[c], ss);
        const double inv = 1.0 / sqrt(block_sum(ss, red));
        for (int c = threadIdx.x; c < d; c += kOrfThreads) row[c] *= inv;
        __syncthreads();
    }
    for (int i = 0; i < rows; ++i) {
        const size_t g = (size_t)b * d + i;
        double ss = 0.0;
        for (int c = threadIdx.x; c < d; c += kOrfThreads) ss = fma(lengths[g * d + c], lengths[g * d + c], ss);
        const double len = sqrt(block_sum(ss, red));
        for (int c = threadIdx.x; c < d; c += kOrfThreads) omega[g * d + c] = (float)(Qm[(size_t)i * d + c] * len);
    }
}

}  // namespace

cudaError_t orf_build(const double* blocks, const double* lengths, int r, int d, float* omega,
                      cudaStream_t s) {
    const int nb = (int)ceil_div(r, d);
    const size_t bytes = ((size_t)d * d + d) * sizeof(double);
    cudaError_t e = cudaFuncSetAttribute(orf_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return e;
    orf_kernel<<<nb, kOrfThreads, bytes, s>>>(blocks, lengths, r, d, omega);
    return cudaGetLastError();
}

}  // namespace la
