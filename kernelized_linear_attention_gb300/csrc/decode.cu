// One-token decode step of causal kernelized attention on CUDA cores.
//
// For each of B sequences and H heads, one new token (q, k, v) meets the fp32
// state [S | z] carried from the earlier tokens: the key is added first, then
// the query reads the updated state ("Reassociate a feature-map kernel" ¶4:
// after adding key/value j, the query at j may read it; "The Kernel Zoo" §1.3
// recurrence):
//
//     S += phi(k) v^T,  z += phi(k),  out = phi(q)^T S / max(phi(q)^T z, eps).
//
// The step reads and writes the whole state once, r (d_v + 1) fp32 values per
// (sequence, head), and does two multiply-adds per state element, so it is
// bound by HBM bandwidth.  One block per (sequence, head): warps walk the
// state's rows, lanes its columns (coalesced row reads; the ones column of
// [v | 1] makes the last column z, so the last numerator column is the
// denominator).
#include "internal.h"

namespace la {

namespace {

constexpr int kDecThreads = 256;
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kMaxColsPerLane = (LA_MAX_DV + 1 + 31) / 32;
// state values per lane whose loads are in flight together (kRows(NJ) rows of NJ)
constexpr int kInFlight = 24;

struct DecSmem {
    size_t xq, xk, vx, phq, phk, red, misc, total;
};

__host__ __device__ inline size_t dec_fl(size_t n) { return (n * sizeof(float) + 15) / 16 * 16; }

__host__ __device__ inline DecSmem plan_dec_smem(int dk, int dv, int r) {
    DecSmem s{};
    size_t o = 0;
    const int dvx = dv + 1;
    s.xq = o;   o += dec_fl(dk);
    s.xk = o;   o += dec_fl(dk);
    s.vx = o;   o += dec_fl(dvx);
    s.phq = o;  o += dec_fl(r);
    s.phk = o;  o += dec_fl(r);
    s.red = o;  o += dec_fl((size_t)kDecWarps * dvx);
    s.misc = o; o += dec_fl(2 * kDecWarps + 4);
    s.total = o;
    return s;
}

struct DecodeParams {
    const void* q;
    const void* k;
    const void* v;
    const float* omega;
    float* state;
    void* out;
    int map, norm, H, dk, dv, r;
    float eps;
};

// Block-wide sum of per-thread values; every thread gets the total.
__device__ __forceinline__ float block_sum(float x, float* scratch) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    __syncthreads();
    if (lane == 0) scratch[warp] = x;
    __syncthreads();
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) t += scratch[w];
    return t;
}

// phi of the query and key rows xq, xk [0..d) into phq, phk [0..r) (all
// threads of the block).  FAVOR+: exp(omega_f . x - |x|^2/2) / sqrt(r) with
// one thread per feature f, both rows at once: a thread's loads of Omega row f
// are independent of each other, so they are all in flight together instead
// of one L2 round trip per step of a reduction.  ELU+1, identity and DPFP-nu
// are element-wise in x.
__device__ void decode_phi(float* phq, float* phk, const float* xq, const float* xk, const float* omega,
                           float hq, float hk, int map, int d, int r) {
    if (map == LA_MAP_FAVOR) {
        const float inv_sqrt_r = rsqrtf((float)r);
        for (int f = threadIdx.x; f < r; f += kDecThreads) {
            const float* w = omega + (int64_t)f * d;
            float aq = 0.f, ak = 0.f;
            if ((d & 3) == 0 && (reinterpret_cast<uintptr_t>(w) & 15) == 0) {
#pragma unroll 4
                for (int c = 0; c < d; c += 4) {
                    const float4 o = *reinterpret_cast<const float4*>(w + c);
                    aq = fmaf(o.x, xq[c], aq); aq = fmaf(o.y, xq[c + 1], aq);
                    aq = fmaf(o.z, xq[c + 2], aq); aq = fmaf(o.w, xq[c + 3], aq);
                    ak = fmaf(o.x, xk[c], ak); ak = fmaf(o.y, xk[c + 1], ak);
                    ak = fmaf(o.z, xk[c + 2], ak); ak = fmaf(o.w, xk[c + 3], ak);
                }
            } else {
#pragma unroll 4
                for (int c = 0; c < d; ++c) {
                    const float o = w[c];
                    aq = fmaf(o, xq[c], aq);
                    ak = fmaf(o, xk[c], ak);
                }
            }
            phq[f] = expf(aq - hq) * inv_sqrt_r;
            phk[f] = expf(ak - hk) * inv_sqrt_r;
        }
    } else if (map == LA_MAP_DPFP) {
        // x~ = relu([x, -x]); feature (s-1) 2d + i = x~_i x~_{(i+s) mod 2d}
        const int d2 = 2 * d;
        for (int f = threadIdx.x; f < r; f += kDecThreads) {
            const int s = f / d2 + 1, a = f - (s - 1) * d2, b = (a + s) % d2;
            const float qa = a < d ? fmaxf(xq[a], 0.f) : fmaxf(-xq[a - d], 0.f);
            const float qb = b < d ? fmaxf(xq[b], 0.f) : fmaxf(-xq[b - d], 0.f);
            const float ka = a < d ? fmaxf(xk[a], 0.f) : fmaxf(-xk[a - d], 0.f);
            const float kb = b < d ? fmaxf(xk[b], 0.f) : fmaxf(-xk[b - d], 0.f);
            phq[f] = qa * qb;
            phk[f] = ka * kb;
        }
    } else {
        for (int f = threadIdx.x; f < r; f += kDecThreads) {   // r == d
            const float a = xq[f], b = xk[f];
            phq[f] = (map == LA_MAP_ELU1) ? (a > 0.f ? a + 1.f : expf(a)) : a;
            phk[f] = (map == LA_MAP_ELU1) ? (b > 0.f ? b + 1.f : expf(b)) : b;
        }
    }
}

// The new token's side of a step (every thread of the block): q, k and
// [v | 1] into shared memory, then phi(q) and phi(k) (sum-normalised under
// LA_NORM_SUM, "The Kernel Zoo" §7.2).  Ends with the block synchronised.
template <typename TIn>
__device__ void decode_prologue(const DecodeParams& p, int64_t bh, float* xq, float* xk, float* vx, float* phq,
                                float* phk, float* misc) {
    const int dk = p.dk, dv = p.dv, dvx = dv + 1, r = p.r;
    const TIn* Q = static_cast<const TIn*>(p.q) + bh * dk;
    const TIn* K = static_cast<const TIn*>(p.k) + bh * dk;
    const TIn* V = static_cast<const TIn*>(p.v) + bh * dv;
    for (int c = threadIdx.x; c < dk; c += kDecThreads) {
        xq[c] = load_elem(Q, c);
        xk[c] = load_elem(K, c);
    }
    for (int c = threadIdx.x; c < dvx; c += kDecThreads) vx[c] = c < dv ? load_elem(V, c) : 1.f;
    __syncthreads();

    float hq = 0.f, hk = 0.f;
    if (p.map == LA_MAP_FAVOR) {
        float sq = 0.f, sk = 0.f;
        for (int c = threadIdx.x; c < dk; c += kDecThreads) {
            sq = fmaf(xq[c], xq[c], sq);
            sk = fmaf(xk[c], xk[c], sk);
        }
        hq = 0.5f * block_sum(sq, misc);
        hk = 0.5f * block_sum(sk, misc + kDecWarps);
    }
    decode_phi(phq, phk, xq, xk, p.omega, hq, hk, p.map, dk, r);
    __syncthreads();
    if (p.norm == LA_NORM_SUM) {
        float sq = 0.f, sk = 0.f;
        for (int f = threadIdx.x; f < r; f += kDecThreads) { sq += phq[f]; sk += phk[f]; }
        const float iq = 1.0f / fmaxf(block_sum(sq, misc), p.eps);
        const float ik = 1.0f / fmaxf(block_sum(sk, misc + kDecWarps), p.eps);
        for (int f = threadIdx.x; f < r; f += kDecThreads) { phq[f] *= iq; phk[f] *= ik; }
        __syncthreads();
    }
}

// Per-warp column sums acc -> out = num / max(den, eps) (attention
// normalisation; column d_v of the numerator is the denominator phi(q)^T z)
// or num.
template <typename TIn, int NJ>
__device__ void decode_epilogue(const DecodeParams& p, int64_t bh, const float (&acc)[NJ], float* red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int dv = p.dv, dvx = dv + 1;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
        const int c = lane + 32 * j;
        if (c < dvx) red[warp * dvx + c] = acc[j];
    }
    __syncthreads();
    float den = 0.f;
    if (p.norm == LA_NORM_ATTENTION) {
#pragma unroll
        for (int w = 0; w < kDecWarps; ++w) den += red[w * dvx + dv];
        den = fmaxf(den, p.eps);
    }
    TIn* O = static_cast<TIn*>(p.out) + bh * dv;
    for (int c = threadIdx.x; c < dv; c += kDecThreads) {
        float num = 0.f;
#pragma unroll
        for (int w = 0; w < kDecWarps; ++w) num += red[w * dvx + c];
        store_elem(O, c, p.norm == LA_NORM_ATTENTION ? num / den : num);
    }
}

// NJ = ceil((d_v + 1) / 32) column groups per lane (one instantiation each).
template <typename TIn, int NJ>
__global__ void __launch_bounds__(kDecThreads, 3) decode_kernel(const DecodeParams p) {
    constexpr int kRows = kInFlight / NJ < 8 ? kInFlight / NJ : 8;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const DecSmem sp = plan_dec_smem(p.dk, p.dv, p.r);
    float* sm = reinterpret_cast<float*>(smem_raw);
    float* xq = sm + sp.xq / 4;
    float* xk = sm + sp.xk / 4;
    float* vx = sm + sp.vx / 4;
    float* phq = sm + sp.phq / 4;
    float* phk = sm + sp.phk / 4;
    float* red = sm + sp.red / 4;
    float* misc = sm + sp.misc / 4;
    const int b = blockIdx.x, h = blockIdx.y;
    const int dk = p.dk, dv = p.dv, dvx = dv + 1, r = p.r;
    const int64_t bh = (int64_t)b * p.H + h;
    float* St = p.state + bh * (int64_t)r * dvx;
    {
        // pull this block's state toward L2 while the features are computed
        const int64_t E = (int64_t)r * dvx;
        for (int64_t e = (int64_t)threadIdx.x * 32; e < E; e += kDecThreads * 32)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(St + e));
    }
    decode_prologue<TIn>(p, bh, xq, xk, vx, phq, phk, misc);

    // state update and readout: warp w owns rows f = w, w + 8, ...; lane owns
    // columns lane + 32 j.  A batch of kRows rows is loaded into registers
    // before any of it is stored, so the loads of a batch are in flight
    // together (stores to earlier rows would otherwise hold them back).
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float vl[NJ], acc[NJ];
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
        const int c = lane + 32 * j;
        vl[j] = c < dvx ? vx[c] : 0.f;
        acc[j] = 0.f;
    }
    bool colv[NJ];
#pragma unroll
    for (int j = 0; j < NJ; ++j) colv[j] = lane + 32 * j < dvx;
    const int64_t row_step = (int64_t)kDecWarps * dvx;   // floats between a warp's consecutive rows
    for (int f0 = warp; f0 < r; f0 += kDecWarps * kRows) {
        float* const base = St + (int64_t)f0 * dvx + lane;
        float sv[kRows][NJ];
#pragma unroll
        for (int i = 0; i < kRows; ++i) {
            const float* row = base + i * row_step;
            const bool rv = f0 + i * kDecWarps < r;
#pragma unroll
            for (int j = 0; j < NJ; ++j) sv[i][j] = (rv && colv[j]) ? row[32 * j] : 0.f;
        }
#pragma unroll
        for (int i = 0; i < kRows; ++i) {
            const int f = f0 + i * kDecWarps;
            if (f < r) {
                float* row = base + i * row_step;
                const float pk = phk[f], pq = phq[f];
#pragma unroll
                for (int j = 0; j < NJ; ++j) {
                    if (colv[j]) {
                        const float sn = fmaf(pk, vl[j], sv[i][j]);
                        row[32 * j] = sn;
                        acc[j] = fmaf(pq, sn, acc[j]);
                    }
                }
            }
        }
    }
    decode_epilogue<TIn, NJ>(p, bh, acc, red);
}

template <typename TIn, int NJ>
cudaError_t launch_one(dim3 grid, cudaStream_t s, const DecodeParams& p) {
    decode_kernel<TIn, NJ><<<grid, kDecThreads, plan_dec_smem(p.dk, p.dv, p.r).total, s>>>(p);
    return cudaGetLastError();
}

template <typename TIn>
cudaError_t launch_nj(int nj, dim3 grid, cudaStream_t s, const DecodeParams& p) {
    static_assert(kMaxColsPerLane == 9, "one case per column-group count");
    switch (nj) {
        case 1: return launch_one<TIn, 1>(grid, s, p);
        case 2: return launch_one<TIn, 2>(grid, s, p);
        case 3: return launch_one<TIn, 3>(grid, s, p);
        case 4: return launch_one<TIn, 4>(grid, s, p);
        case 5: return launch_one<TIn, 5>(grid, s, p);
        case 6: return launch_one<TIn, 6>(grid, s, p);
        case 7: return launch_one<TIn, 7>(grid, s, p);
        case 8: return launch_one<TIn, 8>(grid, s, p);
        default: return launch_one<TIn, 9>(grid, s, p);
    }
}

}  // namespace

size_t decode_smem_bytes(int dk, int dv, int r) { return plan_dec_smem(dk, dv, r).total; }

cudaError_t decode_step(const void* q, const void* k, const void* v, const float* omega, int map, int dtype,
                        int norm, int B, int H, int dk, int dv, int r, float eps, float* state, void* out,
                        cudaStream_t s) {
    const DecodeParams p{q, k, v, omega, state, out, map, norm, H, dk, dv, r, eps};
    const dim3 grid((unsigned)B, (unsigned)H);
    const int nj = (dv + 1 + 31) / 32;
    return dtype == LA_F32 ? launch_nj<float>(nj, grid, s, p) : launch_nj<__nv_bfloat16>(nj, grid, s, p);
}

}  // namespace la
