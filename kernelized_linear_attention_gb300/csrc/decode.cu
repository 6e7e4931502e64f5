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
// (sequence, head) pair, and does two multiply-adds per state element, so it
// is bound by HBM bandwidth.  The kernel is persistent: a few blocks per SM,
// each owning a contiguous run of pairs (whose states are contiguous too).
// A block first forms phi(q) and phi(k) of a batch of its pairs at once, so
// each FAVOR+ row of Omega is read once per batch rather than once per pair;
// then it streams the pairs' states one after another, warps over rows and
// lanes over columns (coalesced; the ones column of [v | 1] makes the last
// column z, so the last numerator column is the denominator), with batches of
// rows loaded into registers before any is stored, and the next pair's state
// prefetched into L2 while the current one is processed (two ahead measured
// slower).
#include <algorithm>

#include "internal.h"

namespace la {

namespace {

constexpr int kDecThreads = 256;
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kMaxColsPerLane = (LA_MAX_DV + 1 + 31) / 32;
// state values per lane whose loads are in flight together (kRows(NJ) rows of NJ);
// two 16-row blocks per SM measured faster than three 8-row blocks (120 vs 128 us)
constexpr int kInFlight = 48;
// pairs whose features one pass over Omega forms
constexpr int kBatch = 8;
constexpr int kBlocksPerSm = 2;
// pairs whose states are prefetched into L2 ahead of the one processed
constexpr int kAhead = 1;

struct DecSmem {
    size_t xq, xk, vx, phq, phk, red, misc, total;
};

__host__ __device__ inline size_t dec_fl(size_t n) { return (n * sizeof(float) + 15) / 16 * 16; }
__host__ __device__ inline int pad4(int n) { return (n + 3) & ~3; }

// Rows of kBatch pairs: q, k [kBatch][pad4(dk)] (zero-padded), [v | 1]
// [kBatch][dvx], features [kBatch][r] each, the per-warp column sums, and
// 2 kBatch scalars.
__host__ __device__ inline DecSmem plan_dec_smem(int dk, int dv, int r) {
    DecSmem s{};
    size_t o = 0;
    const int dvx = dv + 1;
    s.xq = o;   o += dec_fl((size_t)kBatch * pad4(dk));
    s.xk = o;   o += dec_fl((size_t)kBatch * pad4(dk));
    s.vx = o;   o += dec_fl((size_t)kBatch * dvx);
    s.phq = o;  o += dec_fl((size_t)kBatch * r);
    s.phk = o;  o += dec_fl((size_t)kBatch * r);
    s.red = o;  o += dec_fl((size_t)kDecWarps * dvx);
    s.misc = o; o += dec_fl(2 * kBatch);
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
    int64_t pairs;   // B * H
    int map, norm, dk, dv, r;
    float eps;
};

// Features of nb (<= kBatch) consecutive pairs starting at pair p0 (every
// thread of the block; ends synchronised): q, k and [v | 1] rows into shared
// memory, then phi(q), phi(k), sum-normalised under LA_NORM_SUM ("The Kernel
// Zoo" §7.2).  FAVOR+: exp(omega_f . x - |x|^2/2) / sqrt(r) with one thread
// per feature f, which reads Omega row f once and forms the 2 nb dot products.
template <typename TIn>
__device__ void batch_features(const DecodeParams& p, int64_t p0, int nb, float* xq, float* xk, float* vx,
                               float* phq, float* phk, float* misc) {
    const int dk = p.dk, dk4 = pad4(dk), dv = p.dv, dvx = dv + 1, r = p.r;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const TIn* Q = static_cast<const TIn*>(p.q) + p0 * dk;
    const TIn* K = static_cast<const TIn*>(p.k) + p0 * dk;
    const TIn* V = static_cast<const TIn*>(p.v) + p0 * dv;
    for (int e = threadIdx.x; e < kBatch * dk4; e += kDecThreads) {
        const int i = e / dk4, c = e - i * dk4;
        const bool in = i < nb && c < dk;
        xq[e] = in ? load_elem(Q, (int64_t)i * dk + c) : 0.f;
        xk[e] = in ? load_elem(K, (int64_t)i * dk + c) : 0.f;
    }
    for (int e = threadIdx.x; e < kBatch * dvx; e += kDecThreads) {
        const int i = e / dvx, c = e - i * dvx;
        vx[e] = i < nb ? (c < dv ? load_elem(V, (int64_t)i * dv + c) : 1.f) : 0.f;
    }
    __syncthreads();
    if (p.map == LA_MAP_FAVOR) {
        float* hq = misc;            // |q|^2 / 2 of each pair
        float* hk = misc + kBatch;   // |k|^2 / 2
        for (int i = warp; i < kBatch; i += kDecWarps) {
            float sq = 0.f, sk = 0.f;
            for (int c = lane; c < dk4; c += 32) {
                sq = fmaf(xq[i * dk4 + c], xq[i * dk4 + c], sq);
                sk = fmaf(xk[i * dk4 + c], xk[i * dk4 + c], sk);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                sq += __shfl_xor_sync(0xffffffffu, sq, o);
                sk += __shfl_xor_sync(0xffffffffu, sk, o);
            }
            if (lane == 0) { hq[i] = 0.5f * sq; hk[i] = 0.5f * sk; }
        }
        __syncthreads();
        const float inv_sqrt_r = rsqrtf((float)r);
        const bool vec = (dk & 3) == 0 && (reinterpret_cast<uintptr_t>(p.omega) & 15) == 0;
        for (int f = threadIdx.x; f < r; f += kDecThreads) {
            const float* w = p.omega + (int64_t)f * dk;
            float aq[kBatch], ak[kBatch];
#pragma unroll
            for (int i = 0; i < kBatch; ++i) { aq[i] = 0.f; ak[i] = 0.f; }
            for (int c = 0; c < dk4; c += 4) {
                float4 o;
                if (vec) {
                    o = *reinterpret_cast<const float4*>(w + c);
                } else {
                    o.x = w[c];
                    o.y = c + 1 < dk ? w[c + 1] : 0.f;
                    o.z = c + 2 < dk ? w[c + 2] : 0.f;
                    o.w = c + 3 < dk ? w[c + 3] : 0.f;
                }
#pragma unroll
                for (int i = 0; i < kBatch; ++i) {
                    const float4 a = *reinterpret_cast<const float4*>(xq + i * dk4 + c);
                    const float4 b = *reinterpret_cast<const float4*>(xk + i * dk4 + c);
                    aq[i] = fmaf(o.x, a.x, fmaf(o.y, a.y, fmaf(o.z, a.z, fmaf(o.w, a.w, aq[i]))));
                    ak[i] = fmaf(o.x, b.x, fmaf(o.y, b.y, fmaf(o.z, b.z, fmaf(o.w, b.w, ak[i]))));
                }
            }
#pragma unroll
            for (int i = 0; i < kBatch; ++i) {
                if (i < nb) {
                    phq[i * r + f] = expf(aq[i] - hq[i]) * inv_sqrt_r;
                    phk[i * r + f] = expf(ak[i] - hk[i]) * inv_sqrt_r;
                }
            }
        }
    } else if (p.map == LA_MAP_DPFP) {
        // x~ = relu([x, -x]); feature (s-1) 2d + a = x~_a x~_{(a+s) mod 2d}
        const int d2 = 2 * dk;
        for (int e = threadIdx.x; e < nb * r; e += kDecThreads) {
            const int i = e / r, f = e - i * r;
            const int s = f / d2 + 1, a = f - (s - 1) * d2, b = (a + s) % d2;
            const float* xqi = xq + i * dk4;
            const float* xki = xk + i * dk4;
            const float qa = a < dk ? fmaxf(xqi[a], 0.f) : fmaxf(-xqi[a - dk], 0.f);
            const float qb = b < dk ? fmaxf(xqi[b], 0.f) : fmaxf(-xqi[b - dk], 0.f);
            const float ka = a < dk ? fmaxf(xki[a], 0.f) : fmaxf(-xki[a - dk], 0.f);
            const float kb = b < dk ? fmaxf(xki[b], 0.f) : fmaxf(-xki[b - dk], 0.f);
            phq[e] = qa * qb;
            phk[e] = ka * kb;
        }
    } else {
        for (int e = threadIdx.x; e < nb * r; e += kDecThreads) {   // r == d
            const int i = e / r, f = e - i * r;
            const float a = xq[i * dk4 + f], b = xk[i * dk4 + f];
            phq[e] = (p.map == LA_MAP_ELU1) ? (a > 0.f ? a + 1.f : expf(a)) : a;
            phk[e] = (p.map == LA_MAP_ELU1) ? (b > 0.f ? b + 1.f : expf(b)) : b;
        }
    }
    __syncthreads();
    if (p.norm == LA_NORM_SUM) {
        // phi' = phi / max(sum_f phi_f, eps), one warp per pair
        for (int i = warp; i < nb; i += kDecWarps) {
            float sq = 0.f, sk = 0.f;
            for (int f = lane; f < r; f += 32) { sq += phq[i * r + f]; sk += phk[i * r + f]; }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                sq += __shfl_xor_sync(0xffffffffu, sq, o);
                sk += __shfl_xor_sync(0xffffffffu, sk, o);
            }
            const float iq = 1.0f / fmaxf(sq, p.eps), ik = 1.0f / fmaxf(sk, p.eps);
            for (int f = lane; f < r; f += 32) { phq[i * r + f] *= iq; phk[i * r + f] *= ik; }
        }
        __syncthreads();
    }
}

// Starts pulling one pair's state (E floats) into L2; every thread issues a share.
__device__ __forceinline__ void prefetch_state(const float* st, int64_t E) {
    for (int64_t e = (int64_t)threadIdx.x * 32; e < E; e += kDecThreads * 32)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(st + e));
}

// Per-warp column sums acc -> out of pair `pr` = num / max(den, eps)
// (attention normalisation; column d_v of the numerator is the denominator
// phi(q)^T z) or num.  Ends synchronised, so `red` can be reused.
template <typename TIn, int NJ>
__device__ void decode_epilogue(const DecodeParams& p, int64_t pr, const float (&acc)[NJ], float* red) {
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
    TIn* O = static_cast<TIn*>(p.out) + pr * dv;
    for (int c = threadIdx.x; c < dv; c += kDecThreads) {
        float num = 0.f;
#pragma unroll
        for (int w = 0; w < kDecWarps; ++w) num += red[w * dvx + c];
        store_elem(O, c, p.norm == LA_NORM_ATTENTION ? num / den : num);
    }
    __syncthreads();
}

// Block b owns pairs [b P / grid, (b + 1) P / grid).  NJ = ceil((d_v + 1) / 32)
// column groups per lane (one instantiation each).
template <typename TIn, int NJ>
__global__ void __launch_bounds__(kDecThreads, kBlocksPerSm) decode_kernel(const DecodeParams p) {
    constexpr int kRows = kInFlight / NJ < 16 ? kInFlight / NJ : 16;
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
    const int dvx = p.dv + 1, r = p.r;
    const int64_t E = (int64_t)r * dvx;
    const int64_t pb = (int64_t)blockIdx.x * p.pairs / gridDim.x;
    const int64_t pe = (int64_t)(blockIdx.x + 1) * p.pairs / gridDim.x;
    if (pb >= pe) return;
    for (int64_t a = pb; a < pe && a < pb + kAhead; ++a) prefetch_state(p.state + a * E, E);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    bool colv[NJ];
#pragma unroll
    for (int j = 0; j < NJ; ++j) colv[j] = lane + 32 * j < dvx;
    const int64_t row_step = (int64_t)kDecWarps * dvx;   // floats between a warp's consecutive rows
    // batches of equal size (at most kBatch), so no batch pays an Omega pass for a few pairs
    const int64_t nbatch = ceil_div(pe - pb, kBatch);
    const int64_t bsz = ceil_div(pe - pb, nbatch);
    for (int64_t b0 = pb; b0 < pe; b0 += bsz) {
        const int nb = (int)min64(bsz, pe - b0);
        batch_features<TIn>(p, b0, nb, xq, xk, vx, phq, phk, misc);
        for (int i = 0; i < nb; ++i) {
            const int64_t pr = b0 + i;
            if (pr + kAhead < pe) prefetch_state(p.state + (pr + kAhead) * E, E);
            float* St = p.state + pr * E;
            const float* fq = phq + i * r;
            const float* fk = phk + i * r;
            float vl[NJ], acc[NJ];
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
                vl[j] = colv[j] ? vx[i * dvx + lane + 32 * j] : 0.f;
                acc[j] = 0.f;
            }
            // state update and readout: warp w owns rows w, w + 8, ...; a batch of
            // kRows rows is loaded into registers before any of it is stored
            for (int f0 = warp; f0 < r; f0 += kDecWarps * kRows) {
                float* const base = St + (int64_t)f0 * dvx + lane;
                float sv[kRows][NJ];
#pragma unroll
                for (int t = 0; t < kRows; ++t) {
                    const float* row = base + t * row_step;
                    const bool rv = f0 + t * kDecWarps < r;
#pragma unroll
                    for (int j = 0; j < NJ; ++j) sv[t][j] = (rv && colv[j]) ? row[32 * j] : 0.f;
                }
#pragma unroll
                for (int t = 0; t < kRows; ++t) {
                    const int f = f0 + t * kDecWarps;
                    if (f < r) {
                        float* row = base + t * row_step;
                        const float pk = fk[f], pq = fq[f];
#pragma unroll
                        for (int j = 0; j < NJ; ++j) {
                            if (colv[j]) {
                                const float sn = fmaf(pk, vl[j], sv[t][j]);
                                row[32 * j] = sn;
                                acc[j] = fmaf(pq, sn, acc[j]);
                            }
                        }
                    }
                }
            }
            decode_epilogue<TIn, NJ>(p, pr, acc, red);
        }
    }
}

template <typename TIn, int NJ>
cudaError_t launch_one(dim3 grid, cudaStream_t s, const DecodeParams& p) {
    const size_t bytes = plan_dec_smem(p.dk, p.dv, p.r).total;
    if (bytes > 48 * 1024) {
        const cudaError_t e = cudaFuncSetAttribute(decode_kernel<TIn, NJ>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
        if (e != cudaSuccess) return e;
    }
    decode_kernel<TIn, NJ><<<grid, kDecThreads, bytes, s>>>(p);
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
    const int64_t pairs = (int64_t)B * H;
    const DecodeParams p{q, k, v, omega, state, out, pairs, map, norm, dk, dv, r, eps};
    int dev = 0, nsm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const int64_t blocks = std::max<int64_t>(1, std::min<int64_t>(pairs, (int64_t)nsm * kBlocksPerSm));
    const dim3 grid((unsigned)blocks);
    const int nj = (dv + 1 + 31) / 32;
    return dtype == LA_F32 ? launch_nj<float>(nj, grid, s, p) : launch_nj<__nv_bfloat16>(nj, grid, s, p);
}

}  // namespace la
