// Building blocks of the fp32 CUDA-core kernels (forward and backward): work
// in chunks of CS tokens, rows staged in shared memory as
// fp32.  Internal to liblinattn.so; everything has internal linkage.
#pragma once

#include "internal.h"

namespace la {
namespace {

constexpr int CS = 16;    // tokens per chunk
constexpr int NT = 256;   // threads per block of the forward kernels (the helpers below use blockDim.x)
constexpr int NW = NT / 32;

struct OmegaView {
    const float* p;  // element (c, f) = p[c * s_c + f * s_f]
    int s_c, s_f;
    __device__ __forceinline__ float operator()(int c, int f) const { return p[c * s_c + f * s_f]; }
};

template <typename TIn>
__device__ void load_rows(float* dst, const TIn* src, int64_t row0, int nrows, int H, int h, int d) {
    for (int i = threadIdx.x; i < CS * d; i += blockDim.x) {
        const int rr = i / d, c = i - rr * d;
        dst[i] = (rr < nrows) ? load_elem(src, ((row0 + rr) * H + h) * (int64_t)d + c) : 0.f;
    }
}

// [v | 1] rows; padded rows are all zero (so they add nothing to the state).
template <typename TIn>
__device__ void load_vx(float* dst, const TIn* v, int64_t row0, int nrows, int H, int h, int dv) {
    const int dvx = dv + 1;
    for (int i = threadIdx.x; i < CS * dvx; i += blockDim.x) {
        const int rr = i / dvx, c = i - rr * dvx;
        float x = 0.f;
        if (rr < nrows) x = (c < dv) ? load_elem(v, ((row0 + rr) * H + h) * (int64_t)dv + c) : 1.f;
        dst[i] = x;
    }
}

// phi of CS rows of x ([CS][d] in smem) into phi ([CS][r] in smem); rows >= nrows -> 0.
__device__ void compute_phi(float* phi, const float* x, float* half_sq, const OmegaView om,
                            int nrows, int map, int d, int r) {
    if (map == LA_MAP_FAVOR) {
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        for (int row = warp; row < CS; row += (blockDim.x >> 5)) {
            float s = 0.f;
            for (int c = lane; c < d; c += 32) s = fmaf(x[row * d + c], x[row * d + c], s);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
            if (lane == 0) half_sq[row] = 0.5f * s;   // |x|^2 / 2
        }
        __syncthreads();
        const float inv_sqrt_r = rsqrtf((float)r);
        for (int i = threadIdx.x; i < CS * r; i += blockDim.x) {
            const int row = i / r, f = i - row * r;
            float val = 0.f;
            if (row < nrows) {
                float acc = 0.f;
                for (int c = 0; c < d; ++c) acc = fmaf(x[row * d + c], om(c, f), acc);
                val = expf(acc - half_sq[row]) * inv_sqrt_r;   // exp(omega_f . x - |x|^2/2) / sqrt(r)
            }
            phi[i] = val;
        }
    } else if (map == LA_MAP_DPFP) {
        // x~ = relu([x, -x]); feature (s-1) 2d + i = x~_i x~_{(i+s) mod 2d}, s = 1..r / 2d
        const int d2 = 2 * d;
        for (int i = threadIdx.x; i < CS * r; i += blockDim.x) {
            const int row = i / r, f = i - row * r;
            float val = 0.f;
            if (row < nrows) {
                const int s = f / d2 + 1, a = f - (s - 1) * d2, b = (a + s) % d2;
                const float* xr = x + row * d;
                const float xa = a < d ? fmaxf(xr[a], 0.f) : fmaxf(-xr[a - d], 0.f);
                const float xb = b < d ? fmaxf(xr[b], 0.f) : fmaxf(-xr[b - d], 0.f);
                val = xa * xb;
            }
            phi[i] = val;
        }
    } else {
        for (int i = threadIdx.x; i < CS * r; i += blockDim.x) {
            const int row = i / r;
            const float xv = x[i];   // r == d
            float val = 0.f;
            if (row < nrows) val = (map == LA_MAP_ELU1) ? (xv > 0.f ? xv + 1.f : expf(xv)) : xv;
            phi[i] = val;
        }
    }
}

// Sum normalisation phi'(x) = phi(x) / max(sum_f phi(x)_f, eps) of the first
// nrows rows of phi ([CS][r] in smem), one warp per row ("The Kernel Zoo" §7.2).
__device__ void sum_normalise_rows(float* phi, int nrows, int r, float eps) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int row = warp; row < nrows; row += (blockDim.x >> 5)) {
        float s = 0.f;
        for (int f = lane; f < r; f += 32) s += phi[row * r + f];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        const float inv = 1.0f / fmaxf(s, eps);
        for (int f = lane; f < r; f += 32) phi[row * r + f] *= inv;
    }
}

// FAVOR+ features of nrows (<= CS) rows of x ([CS][d] in shared memory) with
// Omega transposed (omt [d][r], in global or shared memory): one thread per (feature, half
// of the rows), eight rows at a time, so each Omega value (a coalesced load)
// and each 4-wide read of x serve eight and four multiply-adds.  Rows past
// nrows get 0.  Same arithmetic as compute_phi: exp(omega_f . x - |x|^2/2)/sqrt(r).
__device__ void favor_features_tiled(float* phi, const float* x, float* half_sq, const float* omt, int nrows, int d,
                                     int r) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int row = warp; row < CS; row += (blockDim.x >> 5)) {
        float sq = 0.f;
        for (int c = lane; c < d; c += 32) sq = fmaf(x[row * d + c], x[row * d + c], sq);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
        if (lane == 0) half_sq[row] = 0.5f * sq;
    }
    __syncthreads();
    const float inv_sqrt_r = rsqrtf((float)r);
    const bool vec = (d & 3) == 0;
    for (int it = threadIdx.x; it < 2 * r; it += blockDim.x) {
        const int f = it % r, r0 = (it / r) * (CS / 2);
        float acc[CS / 2];
#pragma unroll
        for (int j = 0; j < CS / 2; ++j) acc[j] = 0.f;
        if (vec) {
            for (int c = 0; c < d; c += 4) {
                const float o0 = omt[(int64_t)c * r + f], o1 = omt[(int64_t)(c + 1) * r + f];
                const float o2 = omt[(int64_t)(c + 2) * r + f], o3 = omt[(int64_t)(c + 3) * r + f];
#pragma unroll
                for (int j = 0; j < CS / 2; ++j) {
                    const float4 xv = *reinterpret_cast<const float4*>(x + (r0 + j) * d + c);
                    acc[j] = fmaf(xv.x, o0, fmaf(xv.y, o1, fmaf(xv.z, o2, fmaf(xv.w, o3, acc[j]))));
                }
            }
        } else {
            for (int c = 0; c < d; ++c) {
                const float o = omt[(int64_t)c * r + f];
#pragma unroll
                for (int j = 0; j < CS / 2; ++j) acc[j] = fmaf(x[(r0 + j) * d + c], o, acc[j]);
            }
        }
#pragma unroll
        for (int j = 0; j < CS / 2; ++j) {
            const int row = r0 + j;
            phi[row * r + f] = row < nrows ? expf(acc[j] - half_sq[row]) * inv_sqrt_r : 0.f;
        }
    }
}

// acc[f][c] (+)= sum_i a[i][f] b[i][c] over the CS chunk rows, for the [r][dvx]
// array acc (a: [CS][r], b: [CS][dvx], both in shared memory, r a multiple of
// 4): each thread owns four consecutive features of one column, so a 128-bit
// read of a and one read of b serve four multiply-adds.
__device__ void rank_cs_update(float* acc, const float* a, const float* b, int r, int dvx) {
    const int items = (r / 4) * dvx;
    for (int w = threadIdx.x; w < items; w += blockDim.x) {
        const int f0 = 4 * (w / dvx), c = w - (f0 / 4) * dvx;
        float s0 = acc[(f0 + 0) * dvx + c], s1 = acc[(f0 + 1) * dvx + c];
        float s2 = acc[(f0 + 2) * dvx + c], s3 = acc[(f0 + 3) * dvx + c];
#pragma unroll
        for (int i = 0; i < CS; ++i) {
            const float4 av = *reinterpret_cast<const float4*>(a + i * r + f0);
            const float bv = b[i * dvx + c];
            s0 = fmaf(av.x, bv, s0); s1 = fmaf(av.y, bv, s1); s2 = fmaf(av.z, bv, s2); s3 = fmaf(av.w, bv, s3);
        }
        acc[(f0 + 0) * dvx + c] = s0; acc[(f0 + 1) * dvx + c] = s1;
        acc[(f0 + 2) * dvx + c] = s2; acc[(f0 + 3) * dvx + c] = s3;
    }
}

// Places Omega in shared memory as [d][r] when `om_smem` is set, else reads global [r][d].
__device__ OmegaView stage_omega(float* om_smem, const float* omega, int d, int r) {
    if (om_smem == nullptr) return OmegaView{omega, 1, d};
    for (int j = threadIdx.x; j < d * r; j += blockDim.x) {
        const int c = j / r, f = j - c * r;
        om_smem[j] = omega[f * d + c];
    }
    return OmegaView{om_smem, r, 1};
}

}  // namespace
}  // namespace la
