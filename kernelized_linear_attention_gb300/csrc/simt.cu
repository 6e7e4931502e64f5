// fp32 CUDA-core kernels: the exact-arithmetic path for fp32 inputs and the
// general-shape path for any d_k, d_v, r within the size limits.
//
// Chunked evaluation of the causal prefix recurrence ("The Kernel Zoo", §1.3
// and §5.4): a chunk of CS tokens reads the state carried in from earlier
// chunks, adds the in-chunk terms phi(q_i) . phi(k_j) v_j for j <= i, then
// folds its keys into the state.  Bidirectional attention reads the
// whole-sequence state ("Performer", §2 Step 5).  v is extended with a ones
// column, so the last column of the state is z and the last column of the
// numerator is the denominator.
#include "simt_common.cuh"

namespace la {

namespace {

struct SmemPlan {
    size_t om, s, xq, xk, phq, phk, vx, a, num, hsq, hsk, total;
};

__host__ __device__ inline size_t fl(size_t n) { return (n * sizeof(float) + 15) / 16 * 16; }

__host__ __device__ inline SmemPlan plan_smem(int map, int dk, int dv, int r, bool om_in_smem) {
    SmemPlan s{};
    size_t o = 0;
    const int dvx = dv + 1;
    s.om = o;  o += (map == LA_MAP_FAVOR && om_in_smem) ? fl((size_t)dk * r) : 0;
    s.s = o;   o += fl((size_t)r * dvx);
    s.xq = o;  o += fl((size_t)CS * dk);
    s.xk = o;  o += fl((size_t)CS * dk);
    s.phq = o; o += fl((size_t)CS * r);
    s.phk = o; o += fl((size_t)CS * r);
    s.vx = o;  o += fl((size_t)CS * dvx);
    s.a = o;   o += fl((size_t)CS * CS);
    s.num = o; o += fl((size_t)CS * dvx);
    s.hsq = o; o += fl(CS);
    s.hsk = o; o += fl(CS);
    s.total = o;
    return s;
}

constexpr size_t kSmemLimit = 227 * 1024;

// Feature-map kernel: Omega (optional) + x rows + phi rows + |x|^2/2.
__host__ __device__ inline SmemPlan plan_fmap_smem(int map, int d, int r, bool om_in_smem) {
    SmemPlan s{};
    size_t o = 0;
    s.om = o;  o += (map == LA_MAP_FAVOR && om_in_smem) ? fl((size_t)d * r) : 0;
    s.xq = o;  o += fl((size_t)CS * d);
    s.phq = o; o += fl((size_t)CS * r);
    s.hsq = o; o += fl(CS);
    s.total = o;
    return s;
}

inline bool fmap_omega_fits(int map, int d, int r) {
    return map == LA_MAP_FAVOR && plan_fmap_smem(map, d, r, true).total <= kSmemLimit;
}

inline bool omega_fits(int map, int dk, int dv, int r) {
    return map == LA_MAP_FAVOR && plan_smem(map, dk, dv, r, true).total <= kSmemLimit;
}

// ---------------------------------------------------------------------------
template <typename TIn>
__global__ void __launch_bounds__(NT) fmap_kernel(const TIn* x, const float* omega, int map,
                                                  int64_t T, int H, int d, int r, float* out,
                                                  int om_in_smem) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const SmemPlan sp = plan_fmap_smem(map, d, r, om_in_smem);
    float* sm = reinterpret_cast<float*>(smem_raw);
    const OmegaView om = (map == LA_MAP_FAVOR)
        ? stage_omega(om_in_smem ? sm + sp.om / 4 : nullptr, omega, d, r) : OmegaView{nullptr, 0, 0};
    float* xs = sm + sp.xq / 4;
    float* phi = sm + sp.phq / 4;
    float* hs = sm + sp.hsq / 4;
    const int h = blockIdx.y;
    const int64_t row0 = (int64_t)blockIdx.x * CS;
    const int n = (int)min64(CS, T - row0);
    load_rows(xs, x, row0, n, H, h, d);
    __syncthreads();
    compute_phi(phi, xs, hs, om, n, map, d, r);
    __syncthreads();
    for (int i = threadIdx.x; i < n * r; i += NT) {
        const int rr = i / r, f = i - rr * r;
        out[((row0 + rr) * H + h) * (int64_t)r + f] = phi[i];
    }
}

// Per-unit partial state sum_j phi(k_j) [v_j | 1]^T over the unit's tokens.
template <typename TIn>
__global__ void __launch_bounds__(NT) state_kernel(FwdParams p, int om_in_smem) {
    const int u = blockIdx.x, h = blockIdx.y;
    if (u >= p.hdr->n_units) return;
    const Unit un = p.units[u];
    // causal: no later segment adds the last segment of a sequence to its
    // prefix; only a final state needs its sum
    if (p.causal && !p.keep_last && u + 1 == p.seq_first[un.seq + 1]) return;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const SmemPlan sp = plan_smem(p.map, p.dk, p.dv, p.r, om_in_smem);
    float* sm = reinterpret_cast<float*>(smem_raw);
    const OmegaView om = (p.map == LA_MAP_FAVOR)
        ? stage_omega(om_in_smem ? sm + sp.om / 4 : nullptr, p.omega, p.dk, p.r) : OmegaView{nullptr, 0, 0};
    float* S = sm + sp.s / 4;
    float* xk = sm + sp.xk / 4;
    float* phk = sm + sp.phk / 4;
    float* vx = sm + sp.vx / 4;
    float* hs = sm + sp.hsk / 4;
    const int r = p.r, dvx = p.dvx;
    // Omega as [d][r] (staged in shared memory, or the backward's transposed copy): register-tiled features
    const float* omt = (p.map != LA_MAP_FAVOR) ? nullptr : om_in_smem ? om.p : p.omega_t;
    const int E = r * dvx;
    for (int e = threadIdx.x; e < E; e += NT) S[e] = 0.f;
    const TIn* K = static_cast<const TIn*>(p.k);
    const TIn* V = static_cast<const TIn*>(p.v);
    for (int64_t t0 = un.start; t0 < un.end; t0 += CS) {
        const int n = (int)min64(CS, un.end - t0);
        __syncthreads();
        load_rows(xk, K, t0, n, p.H, h, p.dk);
        load_vx(vx, V, t0, n, p.H, h, p.dv);
        __syncthreads();
        if (omt) favor_features_tiled(phk, xk, hs, omt, n, p.dk, r);
        else compute_phi(phk, xk, hs, om, n, p.map, p.dk, r);
        __syncthreads();
        if (p.norm == LA_NORM_SUM) {
            sum_normalise_rows(phk, n, r, p.eps);
            __syncthreads();
        }
        if ((r & 3) == 0) {
            rank_cs_update(S, phk, vx, r, dvx);
        } else {
            for (int e = threadIdx.x; e < E; e += NT) {
                const int f = e / dvx, c = e - f * dvx;
                float acc = S[e];
#pragma unroll
                for (int i = 0; i < CS; ++i) acc = fmaf(phk[i * r + f], vx[i * dvx + c], acc);
                S[e] = acc;
            }
        }
    }
    __syncthreads();
    float* dst = p.partial + ((int64_t)u * p.H + h) * E;
    for (int e = threadIdx.x; e < E; e += NT) dst[e] = S[e];
}

// Outputs of one unit: state in from the scan, then chunk by chunk.
template <typename TIn>
__global__ void __launch_bounds__(NT) out_kernel(FwdParams p, int om_in_smem, int prefix_is_zero) {
    const int u = blockIdx.x, h = blockIdx.y;
    if (u >= p.hdr->n_units) return;
    const Unit un = p.units[u];
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const SmemPlan sp = plan_smem(p.map, p.dk, p.dv, p.r, om_in_smem);
    float* sm = reinterpret_cast<float*>(smem_raw);
    const OmegaView om = (p.map == LA_MAP_FAVOR)
        ? stage_omega(om_in_smem ? sm + sp.om / 4 : nullptr, p.omega, p.dk, p.r) : OmegaView{nullptr, 0, 0};
    float* S = sm + sp.s / 4;
    float* xq = sm + sp.xq / 4;
    float* xk = sm + sp.xk / 4;
    float* phq = sm + sp.phq / 4;
    float* phk = sm + sp.phk / 4;
    float* vx = sm + sp.vx / 4;
    float* A = sm + sp.a / 4;
    float* num = sm + sp.num / 4;
    float* hsq = sm + sp.hsq / 4;
    float* hsk = sm + sp.hsk / 4;
    const int r = p.r, dv = p.dv, dvx = p.dvx;
    const int E = r * dvx;
    const float* omt = (p.map == LA_MAP_FAVOR && om_in_smem) ? om.p : nullptr;   // [d][r]: register-tiled features
    const float* src = p.prefix + ((int64_t)u * p.H + h) * E;
    for (int e = threadIdx.x; e < E; e += NT) S[e] = prefix_is_zero ? 0.f : src[e];
    const TIn* Q = static_cast<const TIn*>(p.q);
    const TIn* K = static_cast<const TIn*>(p.k);
    const TIn* V = static_cast<const TIn*>(p.v);
    TIn* O = static_cast<TIn*>(p.out);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int64_t t0 = un.start; t0 < un.end; t0 += CS) {
        const int n = (int)min64(CS, un.end - t0);
        __syncthreads();
        load_rows(xq, Q, t0, n, p.H, h, p.dk);
        if (p.causal) {
            load_rows(xk, K, t0, n, p.H, h, p.dk);
            load_vx(vx, V, t0, n, p.H, h, dv);
        }
        __syncthreads();
        if (omt) {
            favor_features_tiled(phq, xq, hsq, omt, n, p.dk, r);
            if (p.causal) favor_features_tiled(phk, xk, hsk, omt, n, p.dk, r);
        } else {
            compute_phi(phq, xq, hsq, om, n, p.map, p.dk, r);
            if (p.causal) compute_phi(phk, xk, hsk, om, n, p.map, p.dk, r);
        }
        __syncthreads();
        if (p.norm == LA_NORM_SUM) {
            sum_normalise_rows(phq, n, r, p.eps);
            if (p.causal) sum_normalise_rows(phk, n, r, p.eps);
            __syncthreads();
        }
        if (p.causal) {
            // A[i][j] = phi(q_i) . phi(k_j) for j <= i (diagonal included), one warp per entry
            for (int ij = warp; ij < CS * CS; ij += NW) {
                const int i = ij / CS, j = ij - i * CS;
                float acc = 0.f;
                if (j <= i && i < n) {
                    for (int f = lane; f < r; f += 32) acc = fmaf(phq[i * r + f], phk[j * r + f], acc);
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
                }
                if (lane == 0) A[ij] = acc;
            }
            __syncthreads();
        }
        // num[i][c] = phi(q_i) . S[:, c]  (+ sum_{j<=i} A[i][j] vx[j][c]); column dv is the denominator
        for (int e = threadIdx.x; e < CS * dvx; e += NT) {
            const int i = e / dvx, c = e - i * dvx;
            float acc = 0.f;
            for (int f = 0; f < r; ++f) acc = fmaf(phq[i * r + f], S[f * dvx + c], acc);
            if (p.causal) {
#pragma unroll
                for (int j = 0; j < CS; ++j) acc = fmaf(A[i * CS + j], vx[j * dvx + c], acc);
            }
            num[e] = acc;
        }
        __syncthreads();
        if (p.causal && (r & 3) == 0) {
            rank_cs_update(S, phk, vx, r, dvx);
        } else if (p.causal) {
            for (int e = threadIdx.x; e < E; e += NT) {
                const int f = e / dvx, c = e - f * dvx;
                float acc = S[e];
#pragma unroll
                for (int i = 0; i < CS; ++i) acc = fmaf(phk[i * r + f], vx[i * dvx + c], acc);
                S[e] = acc;
            }
        }
        for (int e = threadIdx.x; e < n * dv; e += NT) {
            const int i = e / dv, c = e - i * dv;
            float o = num[i * dvx + c];
            if (p.norm == LA_NORM_ATTENTION) o /= fmaxf(num[i * dvx + dv], p.eps);   // max(phi(q)^T z, eps)
            store_elem(O, ((t0 + i) * p.H + h) * (int64_t)dv + c, o);
        }
    }
}

}  // namespace

int simt_chunk() { return CS; }

size_t simt_smem_bytes(int map, int dk, int dv, int r) {
    return plan_smem(map, dk, dv, r, omega_fits(map, dk, dv, r)).total;
}

size_t simt_fmap_smem_bytes(int map, int d, int r) {
    return plan_fmap_smem(map, d, r, fmap_omega_fits(map, d, r)).total;
}

template <typename Kern>
static cudaError_t set_smem(Kern k, size_t bytes) {
    return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

cudaError_t simt_feature_map(const void* x, const float* omega, int map, int dtype,
                             int64_t T, int H, int d, int r, float* phi, cudaStream_t s) {
    const int om_smem = fmap_omega_fits(map, d, r) ? 1 : 0;
    const size_t bytes = plan_fmap_smem(map, d, r, om_smem).total;
    if (bytes > kSmemLimit) return cudaErrorInvalidValue;
    dim3 grid((unsigned)ceil_div(T, CS), (unsigned)H);
    cudaError_t e;
    if (dtype == LA_F32) {
        if ((e = set_smem(fmap_kernel<float>, bytes)) != cudaSuccess) return e;
        fmap_kernel<float><<<grid, NT, bytes, s>>>(static_cast<const float*>(x), omega, map, T, H, d, r, phi, om_smem);
    } else {
        if ((e = set_smem(fmap_kernel<__nv_bfloat16>, bytes)) != cudaSuccess) return e;
        fmap_kernel<__nv_bfloat16><<<grid, NT, bytes, s>>>(static_cast<const __nv_bfloat16*>(x), omega, map, T,
                                                          H, d, r, phi, om_smem);
    }
    return cudaGetLastError();
}

cudaError_t simt_state(const FwdParams& p, int dtype, cudaStream_t s) {
    const int om_smem = omega_fits(p.map, p.dk, p.dv, p.r) ? 1 : 0;
    const size_t bytes = plan_smem(p.map, p.dk, p.dv, p.r, om_smem).total;
    dim3 grid((unsigned)p.U, (unsigned)p.H);
    cudaError_t e;
    if (dtype == LA_F32) {
        if ((e = set_smem(state_kernel<float>, bytes)) != cudaSuccess) return e;
        state_kernel<float><<<grid, NT, bytes, s>>>(p, om_smem);
    } else {
        if ((e = set_smem(state_kernel<__nv_bfloat16>, bytes)) != cudaSuccess) return e;
        state_kernel<__nv_bfloat16><<<grid, NT, bytes, s>>>(p, om_smem);
    }
    return cudaGetLastError();
}

cudaError_t simt_out(const FwdParams& p, int dtype, int prefix_is_zero, cudaStream_t s) {
    const int om_smem = omega_fits(p.map, p.dk, p.dv, p.r) ? 1 : 0;
    const size_t bytes = plan_smem(p.map, p.dk, p.dv, p.r, om_smem).total;
    dim3 grid((unsigned)p.U, (unsigned)p.H);
    cudaError_t e;
    if (dtype == LA_F32) {
        if ((e = set_smem(out_kernel<float>, bytes)) != cudaSuccess) return e;
        out_kernel<float><<<grid, NT, bytes, s>>>(p, om_smem, prefix_is_zero);
    } else {
        if ((e = set_smem(out_kernel<__nv_bfloat16>, bytes)) != cudaSuccess) return e;
        out_kernel<__nv_bfloat16><<<grid, NT, bytes, s>>>(p, om_smem, prefix_is_zero);
    }
    return cudaGetLastError();
}

}  // namespace la
