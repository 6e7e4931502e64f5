// Sum normalisation on the tensor-core path ("The Kernel Zoo" §7.2-7.4):
// every query and key feature vector is divided by its component sum and the
// output has no attention denominator, so with sigma = max(sum_f phi_f, eps)
//
//     out_i = sum_{j (<= i)} (phi(q_i) / sigma_q_i) . (phi(k_j) / sigma_k_j) v_j
//           = [ sum_j (phi(q_i) . phi(k_j)) (v_j / sigma_k_j) ] / sigma_q_i .
//
// The bracket is the unnormalised output for the values v_j / sigma_k_j, which
// the tensor-core kernels compute as they are (their output store divides by
// max(sigma_q, eps)); these kernels supply the sums and the scaled values.
// bf16 tensors, fp32 arithmetic.
#include "internal.h"

namespace la {

namespace {

constexpr int kNormThreads = 256;

// One pass for the element-wise maps (identity, ELU+1, DPFP-nu; d = dv = 64,
// one warp per row, two elements per lane): sigma_q of the q row into
// sig_q, sigma_k of the k row, and the v row divided by max(sigma_k, eps) into
// dst (bf16).
__device__ __forceinline__ float phi_sum_row(float2 x, int map, int d, int r, int lane) {
    // the row's 64 inputs are spread two per lane: element 2 lane, 2 lane + 1
    float acc = 0.f;
    if (map == LA_MAP_DPFP) {
        // feature (s-1) 2d + a = x~_a x~_{(a+s) mod 2d}, x~ = relu([x, -x]); gather x~ by shuffles
        const int d2 = 2 * d;
        for (int f = lane; f < r; f += 32) {
            const int s = f / d2 + 1, a = f - (s - 1) * d2, b = (a + s) % d2;
            const int ia = a < d ? a : a - d, ib = b < d ? b : b - d;
            // a shuffle returns the source lane's variable: fetch both halves, choose here
            const float ax = __shfl_sync(0xffffffffu, x.x, ia >> 1), ay = __shfl_sync(0xffffffffu, x.y, ia >> 1);
            const float bx = __shfl_sync(0xffffffffu, x.x, ib >> 1), by = __shfl_sync(0xffffffffu, x.y, ib >> 1);
            const float va = (ia & 1) ? ay : ax, vb = (ib & 1) ? by : bx;
            acc = fmaf(a < d ? fmaxf(va, 0.f) : fmaxf(-va, 0.f), b < d ? fmaxf(vb, 0.f) : fmaxf(-vb, 0.f), acc);
        }
    } else if (map == LA_MAP_ELU1) {
        acc = (x.x > 0.f ? x.x + 1.f : expf(x.x)) + (x.y > 0.f ? x.y + 1.f : expf(x.y));
    } else {
        acc = x.x + x.y;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    return acc;
}

constexpr int kRowsPerWarp = 4;   // rows whose loads a warp issues before it computes

__global__ void __launch_bounds__(kNormThreads) sum_prologue_kernel(const __nv_bfloat16* q, const __nv_bfloat16* k,
                                                                    const __nv_bfloat16* v, int map, int64_t rows,
                                                                    int r, float eps, float* sig_q,
                                                                    __nv_bfloat16* dst) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (kNormThreads / 32);
    const int64_t first = ((int64_t)blockIdx.x * (kNormThreads / 32) + (threadIdx.x >> 5)) * kRowsPerWarp;
    for (int64_t row0 = first; row0 < rows; row0 += warps * kRowsPerWarp) {
        // every load of the warp's rows in flight before the first use
        float2 xq[kRowsPerWarp], xk[kRowsPerWarp], xv[kRowsPerWarp];
#pragma unroll
        for (int i = 0; i < kRowsPerWarp; ++i) {
            const int64_t row = row0 + i < rows ? row0 + i : row0;   // a past-the-end row repeats a valid one
            xq[i] = __bfloat1622float2(reinterpret_cast<const __nv_bfloat162*>(q + row * 64)[lane]);
            xk[i] = __bfloat1622float2(reinterpret_cast<const __nv_bfloat162*>(k + row * 64)[lane]);
            xv[i] = __bfloat1622float2(reinterpret_cast<const __nv_bfloat162*>(v + row * 64)[lane]);
        }
#pragma unroll
        for (int i = 0; i < kRowsPerWarp; ++i) {
            const int64_t row = row0 + i;
            const float sq = phi_sum_row(xq[i], map, 64, r, lane);
            const float sk = fmaxf(phi_sum_row(xk[i], map, 64, r, lane), eps);
            if (row < rows) {
                if (lane == 0) sig_q[row] = sq;
                reinterpret_cast<__nv_bfloat162*>(dst + row * 64)[lane] = __floats2bfloat162_rn(xv[i].x / sk, xv[i].y / sk);
            }
        }
    }
}

// The same for ELU+1 and identity, whose sums need no gather across the row: 16-byte
// loads, eight lanes per row (a warp covers four rows per load) and kGroups such groups
// of four rows in flight per warp; the row sums reduce over the eight lanes.
template <int kGroups>
__global__ void __launch_bounds__(kNormThreads) sum_prologue_vec_kernel(const __nv_bfloat16* q,
                                                                        const __nv_bfloat16* k,
                                                                        const __nv_bfloat16* v, int map,
                                                                        int64_t rows, float eps, float* sig_q,
                                                                        __nv_bfloat16* dst) {
    const int lane = threadIdx.x & 31, sub = lane & 7, rr = lane >> 3;
    const int64_t warps = (int64_t)gridDim.x * (kNormThreads / 32);
    const int64_t first = ((int64_t)blockIdx.x * (kNormThreads / 32) + (threadIdx.x >> 5)) * (4 * kGroups);
    const bool elu = map == LA_MAP_ELU1;
    auto phi_sum8 = [&](const uint4& w) {
        const uint32_t u[4] = {w.x, w.y, w.z, w.w};
        float acc = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u[j]));
            acc += elu ? (x.x > 0.f ? x.x + 1.f : expf(x.x)) : x.x;
            acc += elu ? (x.y > 0.f ? x.y + 1.f : expf(x.y)) : x.y;
        }
        return acc;
    };
    for (int64_t row0 = first; row0 < rows; row0 += warps * (4 * kGroups)) {
        uint4 aq[kGroups], ak[kGroups], av[kGroups];
#pragma unroll
        for (int g = 0; g < kGroups; ++g) {
            int64_t row = row0 + 4 * g + rr;
            row = row < rows ? row : rows - 1;   // a past-the-end row repeats the last one
            aq[g] = reinterpret_cast<const uint4*>(q + row * 64)[sub];
            ak[g] = reinterpret_cast<const uint4*>(k + row * 64)[sub];
            av[g] = reinterpret_cast<const uint4*>(v + row * 64)[sub];
        }
#pragma unroll
        for (int g = 0; g < kGroups; ++g) {
            float sq = phi_sum8(aq[g]), sk = phi_sum8(ak[g]);
#pragma unroll
            for (int o = 1; o < 8; o <<= 1) {
                sq += __shfl_xor_sync(0xffffffffu, sq, o);
                sk += __shfl_xor_sync(0xffffffffu, sk, o);
            }
            sk = fmaxf(sk, eps);
            const int64_t row = row0 + 4 * g + rr;
            if (row < rows) {
                if (sub == 0) sig_q[row] = sq;
                const uint32_t u[4] = {av[g].x, av[g].y, av[g].z, av[g].w};
                uint32_t o4[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u[j]));
                    const __nv_bfloat162 y = __floats2bfloat162_rn(x.x / sk, x.y / sk);
                    o4[j] = *reinterpret_cast<const uint32_t*>(&y);
                }
                reinterpret_cast<uint4*>(dst + row * 64)[sub] = make_uint4(o4[0], o4[1], o4[2], o4[3]);
            }
        }
    }
}

// dst = x / max(sigma_row, eps) element-wise over rows of n values (bf16 in and out).
__global__ void __launch_bounds__(kNormThreads) scale_rows_kernel(const __nv_bfloat16* x, const float* sigma,
                                                                  float eps, int64_t rows, int n,
                                                                  __nv_bfloat16* dst) {
    const int64_t total = rows * n;
    for (int64_t i = (int64_t)blockIdx.x * kNormThreads + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * kNormThreads) {
        const float s = fmaxf(sigma[i / n], eps);
        dst[i] = __float2bfloat16_rn(__bfloat162float(x[i]) / s);
    }
}

unsigned grid_for(int64_t items) {
    const int64_t b = ceil_div(items, kNormThreads);
    return (unsigned)(b < 65535 * 8 ? (b > 0 ? b : 1) : 65535 * 8);
}

}  // namespace

cudaError_t sum_scale_values(const void* v, const float* sigma_k, float eps, int64_t T, int H, int dv, void* dst,
                             cudaStream_t s) {
    const int64_t rows = T * H;
    if (rows == 0) return cudaSuccess;
    scale_rows_kernel<<<grid_for(rows * dv), kNormThreads, 0, s>>>(static_cast<const __nv_bfloat16*>(v), sigma_k, eps,
                                                                   rows, dv, static_cast<__nv_bfloat16*>(dst));
    return cudaGetLastError();
}

cudaError_t sum_prologue_elementwise(const void* q, const void* k, const void* v, int map, int64_t T, int H, int r,
                                     float eps, float* sig_q, void* dst, cudaStream_t s) {
    const int64_t rows = T * H;
    if (rows == 0) return cudaSuccess;
    const bool vec = map != LA_MAP_DPFP && ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                                              reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(dst)) & 15) == 0;
    if (vec) {
        constexpr int kGroups = 4;   // sixteen rows per warp
        const int64_t blocks = ceil_div(rows, (int64_t)(kNormThreads / 32) * 4 * kGroups);
        sum_prologue_vec_kernel<kGroups><<<(unsigned)(blocks < INT32_MAX ? blocks : INT32_MAX), kNormThreads, 0, s>>>(
            static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k),
            static_cast<const __nv_bfloat16*>(v), map, rows, eps, sig_q, static_cast<__nv_bfloat16*>(dst));
        return cudaGetLastError();
    }
    // four rows per warp, every row's loads in flight at once
    const int64_t blocks = ceil_div(rows, (int64_t)(kNormThreads / 32) * kRowsPerWarp);
    sum_prologue_kernel<<<(unsigned)(blocks < INT32_MAX ? blocks : INT32_MAX), kNormThreads, 0, s>>>(
        static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k),
        static_cast<const __nv_bfloat16*>(v), map, rows, r, eps, sig_q, static_cast<__nv_bfloat16*>(dst));
    return cudaGetLastError();
}

}  // namespace la
