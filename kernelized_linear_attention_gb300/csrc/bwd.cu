// Backward pass of kernelized attention on CUDA cores (fp32 for every dtype):
// gradients of L = sum(dout * out) with respect to q, k and v.
//
// With [v | 1] as the values (so num | den is one product) and g_i the
// gradient of L with respect to num_i | den_i,
//
//     g_i = [dout_i / max(den_i, eps) | -(dout_i . out_i) / den_i]   (attention
//           normalisation; the last entry is 0 where the clamp holds)
//     g_i = [dout_i | 0]                                              (none, sum)
//
// the chain rule through num_i = sum_{j<=i} (phi(q_i) . phi(k_j)) [v_j | 1]
// gives, with S_i = sum_{j<=i} phi(k_j) [v_j | 1]^T (the forward state) and
// R_j = sum_{i>=j} phi(q_i) g_i^T (the same sum run backwards in time):
//
//     dphi(q_i) = S_i g_i,   dphi(k_j) = R_j [v_j | 1],   dv_j = (R_j^T phi(k_j))[:d_v]
//
// (j over the whole sequence, and S, R the whole-sequence sums, for the
// bidirectional form), then dq, dk through the feature map.  Omega is a
// constant.  The causal form runs as a chunked scan in both directions: the
// forward state pass and scan give S at every segment start; bwd_q_kernel
// walks each segment forwards, recomputing num | den to form g (kept in the
// workspace), writing dq and summing phi(q) g^T of the segment; a reverse scan
// gives R at every segment end; bwd_kv_kernel walks each segment backwards and
// writes dk and dv.  ("Reassociate a feature-map kernel" ¶5 asks for errors
// in gradients as well as outputs; the recurrence is that of "The Kernel Zoo"
// §1.3.)
#include "simt_common.cuh"

namespace la {

namespace {

// 16 warps per block: one block per SM fits (its states fill the shared
// memory), so the block itself supplies the warps that hide latency.
constexpr int kBwdThreads = 512;

struct BwdSmem {
    size_t st, racc, xq, xk, phq, phk, dph, vx, gg, num, go, a, gm, hsq, hsk, sgq, sgk, su, total;
};

__host__ __device__ inline size_t bfl(size_t n) { return (n * sizeof(float) + 15) / 16 * 16; }

// `racc`: bwd_q_kernel's running sum of phi(q) g^T (bwd_kv_kernel needs none).
__host__ __device__ inline BwdSmem plan_bwd_smem(int dk, int dv, int r, bool racc) {
    BwdSmem s{};
    size_t o = 0;
    const int dvx = dv + 1;
    s.st = o;   o += bfl((size_t)r * dvx);
    s.racc = o; o += racc ? bfl((size_t)r * dvx) : 0;
    s.xq = o;   o += bfl((size_t)CS * dk);
    s.xk = o;   o += bfl((size_t)CS * dk);
    s.phq = o;  o += bfl((size_t)CS * r);
    s.phk = o;  o += bfl((size_t)CS * r);
    s.dph = o;  o += bfl((size_t)CS * r);
    s.vx = o;   o += bfl((size_t)CS * dvx);
    s.gg = o;   o += bfl((size_t)CS * dvx);
    s.num = o;  o += bfl((size_t)CS * dvx);
    s.go = o;   o += bfl((size_t)CS * dv);
    s.a = o;    o += bfl((size_t)CS * CS);
    s.gm = o;   o += bfl((size_t)CS * CS);
    s.hsq = o;  o += bfl(CS);
    s.hsk = o;  o += bfl(CS);
    s.sgq = o;  o += bfl(CS);
    s.sgk = o;  o += bfl(CS);
    s.su = o;   o += bfl(CS);
    s.total = o;
    return s;
}

// Sum normalisation of the first nrows rows that keeps each row's raw sum
// (the backward pass needs it): phi' = phi / max(sum, eps).
__device__ void sum_normalise_keep(float* phi, float* raw_sum, int nrows, int r, float eps) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int row = warp; row < nrows; row += (blockDim.x >> 5)) {
        float s = 0.f;
        for (int f = lane; f < r; f += 32) s += phi[row * r + f];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (lane == 0) raw_sum[row] = s;
        const float inv = 1.0f / fmaxf(s, eps);
        for (int f = lane; f < r; f += 32) phi[row * r + f] *= inv;
    }
}

// dx of nrows rows from dph = dL/dphi' (overwritten): first through the sum
// normalisation (norm LA_NORM_SUM: dphi = (dphi' - (dphi' . phi') 1) / sigma,
// or dphi' / eps where the sum was clamped; phi is turned back into the raw
// features), then through the map:
//   identity  dx = dphi;  ELU+1  dx = dphi * (x > 0 ? 1 : exp(x));
//   FAVOR+    u = dphi * phi, dx = Omega^T u - x sum_f u_f;
//   DPFP-nu   phi_f = x~_a x~_b (b = (a + s) mod 2d) sends dphi_f x~_b to x~_a
//             and dphi_f x~_a to x~_b; x~ = relu([x, -x]).
// Writes dx rows row0.. of head h to global (dtype of TOut).
template <typename TOut>
__device__ void features_vjp_rows(float* dph, float* phi, const float* x, const float* raw_sum, float* su,
                                  int nrows, const FwdParams& p, const OmegaView om, TOut* dst, int64_t row0,
                                  int h) {
    const int r = p.r, d = p.dk;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (p.norm == LA_NORM_SUM) {
        for (int row = warp; row < nrows; row += (blockDim.x >> 5)) {
            float dot = 0.f;
            for (int f = lane; f < r; f += 32) dot = fmaf(dph[row * r + f], phi[row * r + f], dot);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
            const float raw = raw_sum[row];
            const float sig = fmaxf(raw, p.eps);
            const float sub = raw > p.eps ? dot : 0.f;
            for (int f = lane; f < r; f += 32) {
                dph[row * r + f] = (dph[row * r + f] - sub) / sig;
                phi[row * r + f] *= sig;
            }
        }
        __syncthreads();
    }
    if (p.map == LA_MAP_FAVOR) {
        for (int row = warp; row < nrows; row += (blockDim.x >> 5)) {
            float s = 0.f;
            for (int f = lane; f < r; f += 32) {
                const float u = dph[row * r + f] * phi[row * r + f];
                dph[row * r + f] = u;
                s += u;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
            if (lane == 0) su[row] = s;
        }
        __syncthreads();
        if ((r & 3) == 0) {
            // two rows of one input column per thread: dph read four features at a time (broadcast),
            // each Omega value (a coalesced load) serves two rows
            for (int w = threadIdx.x; w < (CS / 2) * d; w += blockDim.x) {
                const int rp = w / d, c = w - rp * d, ra = 2 * rp;
                if (ra >= nrows) continue;
                float a0 = 0.f, a1 = 0.f;
                for (int f = 0; f < r; f += 4) {
                    const float o0 = om(c, f), o1 = om(c, f + 1), o2 = om(c, f + 2), o3 = om(c, f + 3);
                    const float4 u0 = *reinterpret_cast<const float4*>(dph + ra * r + f);
                    const float4 u1 = *reinterpret_cast<const float4*>(dph + (ra + 1) * r + f);
                    a0 = fmaf(u0.w, o3, fmaf(u0.z, o2, fmaf(u0.y, o1, fmaf(u0.x, o0, a0))));
                    a1 = fmaf(u1.w, o3, fmaf(u1.z, o2, fmaf(u1.y, o1, fmaf(u1.x, o0, a1))));
                }
                store_elem(dst, ((row0 + ra) * p.H + h) * (int64_t)d + c, a0 - x[ra * d + c] * su[ra]);
                if (ra + 1 < nrows)
                    store_elem(dst, ((row0 + ra + 1) * p.H + h) * (int64_t)d + c, a1 - x[(ra + 1) * d + c] * su[ra + 1]);
            }
        } else {
            for (int e = threadIdx.x; e < nrows * d; e += blockDim.x) {
                const int row = e / d, c = e - row * d;
                float acc = 0.f;
                for (int f = 0; f < r; ++f) acc = fmaf(dph[row * r + f], om(c, f), acc);
                store_elem(dst, ((row0 + row) * p.H + h) * (int64_t)d + c, acc - x[row * d + c] * su[row]);
            }
        }
    } else if (p.map == LA_MAP_DPFP) {
        const int d2 = 2 * d, nu = r / d2;
        for (int e = threadIdx.x; e < nrows * d; e += blockDim.x) {
            const int row = e / d, c = e - row * d;
            const float* xr = x + row * d;
            const float* g = dph + row * r;
            auto xt = [&](int i) { return i < d ? fmaxf(xr[i], 0.f) : fmaxf(-xr[i - d], 0.f); };
            float dp = 0.f, dn = 0.f;   // dL/dx~_c and dL/dx~_{c+d}
            for (int s = 1; s <= nu; ++s) {
                const float* gs = g + (s - 1) * d2;
                int i = c;
                dp = fmaf(gs[i], xt((i + s) % d2), dp);
                dp = fmaf(gs[(i - s + d2) % d2], xt((i - s + d2) % d2), dp);
                i = c + d;
                dn = fmaf(gs[i], xt((i + s) % d2), dn);
                dn = fmaf(gs[(i - s + d2) % d2], xt((i - s + d2) % d2), dn);
            }
            const float xv = xr[c];
            store_elem(dst, ((row0 + row) * p.H + h) * (int64_t)d + c, (xv > 0.f ? dp : 0.f) - (xv < 0.f ? dn : 0.f));
        }
    } else {
        for (int e = threadIdx.x; e < nrows * d; e += blockDim.x) {
            const int row = e / d, c = e - row * d;   // r == d
            const float xv = x[row * d + c], gv = dph[row * r + c];
            const float dxv = (p.map == LA_MAP_ELU1) ? gv * (xv > 0.f ? 1.f : expf(xv)) : gv;
            store_elem(dst, ((row0 + row) * p.H + h) * (int64_t)d + c, dxv);
        }
    }
}

// out[i][c] = sum_f a[i][f] M[f][c] (+ sum_s T(i, s) b[s][c] when T is given) for the CS
// chunk rows i and the columns c < ncols; T(i, s) = T[i][s], or T[s][i] when kTT.  a is
// [CS][r] (r a multiple of 4), M [r][dvx], T [CS][CS], b [CS][dvx], out rows ldo apart, all
// in shared memory.  A thread computes rows 4 rb .. 4 rb + 3 of one column: a is read four
// features at a time (a warp broadcast), M once per feature for four multiply-adds.
template <bool kTT>
__device__ void rows_times_state(float* out, int ldo, const float* a, const float* M, const float* T, const float* b,
                                 int r, int dvx, int ncols) {
    for (int w = threadIdx.x; w < 4 * ncols; w += blockDim.x) {
        const int rb = w / ncols, c = w - rb * ncols, i0 = 4 * rb;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        for (int f = 0; f < r; f += 4) {
            const float m0 = M[f * dvx + c], m1 = M[(f + 1) * dvx + c];
            const float m2 = M[(f + 2) * dvx + c], m3 = M[(f + 3) * dvx + c];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float4 av = *reinterpret_cast<const float4*>(a + (i0 + k) * r + f);
                acc[k] = fmaf(av.w, m3, fmaf(av.z, m2, fmaf(av.y, m1, fmaf(av.x, m0, acc[k]))));
            }
        }
        if (T) {
#pragma unroll 4
            for (int s = 0; s < CS; ++s) {
                const float bv = b[s * dvx + c];
#pragma unroll
                for (int k = 0; k < 4; ++k) acc[k] = fmaf(kTT ? T[s * CS + i0 + k] : T[(i0 + k) * CS + s], bv, acc[k]);
            }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) out[(i0 + k) * ldo + c] = acc[k];
    }
}

// out[i][f] = sum_c M[f][c] b[i][c] (+ sum_s G(i, s) P[s][f] when G is given) for the CS
// chunk rows i and the r features f (r even); G(i, s) = G[i][s], or G[s][i] when kGT.  M is
// [r][dvx], b [CS][dvx], G [CS][CS], P [CS][r], out [CS][r], all in shared memory.  A thread
// computes rows 4 rb .. 4 rb + 3 of features f and f + r / 2: the two reads of M are
// 65-float strides across a warp (no bank conflicts), b and G reads are broadcasts.
template <bool kGT>
__device__ void state_times_rows(float* out, const float* M, const float* b, const float* G, const float* P, int r,
                                 int dvx) {
    const int half = r / 2;
    for (int w = threadIdx.x; w < 4 * half; w += blockDim.x) {
        const int rb = w / half, f0 = w - rb * half, f1 = f0 + half, i0 = 4 * rb;
        float a0[4] = {0.f, 0.f, 0.f, 0.f}, a1[4] = {0.f, 0.f, 0.f, 0.f};
        for (int c = 0; c < dvx; ++c) {
            const float m0 = M[f0 * dvx + c], m1 = M[f1 * dvx + c];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float bv = b[(i0 + k) * dvx + c];
                a0[k] = fmaf(m0, bv, a0[k]);
                a1[k] = fmaf(m1, bv, a1[k]);
            }
        }
        if (G) {
#pragma unroll 4
            for (int s = 0; s < CS; ++s) {
                const float p0 = P[s * r + f0], p1 = P[s * r + f1];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float g = kGT ? G[s * CS + i0 + k] : G[(i0 + k) * CS + s];
                    a0[k] = fmaf(g, p0, a0[k]);
                    a1[k] = fmaf(g, p1, a1[k]);
                }
            }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            out[(i0 + k) * r + f0] = a0[k];
            out[(i0 + k) * r + f1] = a1[k];
        }
    }
}

struct BwdView {
    float *st, *racc, *xq, *xk, *phq, *phk, *dph, *vx, *gg, *num, *go, *a, *gm, *hsq, *hsk, *sgq, *sgk, *su;
};

__device__ BwdView bwd_view(unsigned char* raw, const BwdSmem& sp) {
    float* sm = reinterpret_cast<float*>(raw);
    return BwdView{sm + sp.st / 4, sm + sp.racc / 4, sm + sp.xq / 4, sm + sp.xk / 4, sm + sp.phq / 4,
                   sm + sp.phk / 4, sm + sp.dph / 4, sm + sp.vx / 4, sm + sp.gg / 4, sm + sp.num / 4,
                   sm + sp.go / 4, sm + sp.a / 4, sm + sp.gm / 4, sm + sp.hsq / 4, sm + sp.hsk / 4,
                   sm + sp.sgq / 4, sm + sp.sgk / 4, sm + sp.su / 4};
}

// A[i][j] = phi(q_i) . phi(k_j) for j <= i < n (diagonal included), else 0; one warp per entry.
__device__ void causal_scores(float* A, const float* phq, const float* phk, int n, int r) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int ij = warp; ij < CS * CS; ij += (blockDim.x >> 5)) {
        const int i = ij / CS, j = ij - i * CS;
        float acc = 0.f;
        if (j <= i && i < n) {
            for (int f = lane; f < r; f += 32) acc = fmaf(phq[i * r + f], phk[j * r + f], acc);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        }
        if (lane == 0) A[ij] = acc;
    }
}

// Gm[i][j] = g_i . [v_j | 1] for j <= i < n, else 0.
__device__ void causal_gv(float* Gm, const float* gg, const float* vx, int n, int dvx) {
    for (int ij = threadIdx.x; ij < CS * CS; ij += blockDim.x) {
        const int i = ij / CS, j = ij - i * CS;
        float acc = 0.f;
        if (j <= i && i < n)
            for (int c = 0; c < dvx; ++c) acc = fmaf(gg[i * dvx + c], vx[j * dvx + c], acc);
        Gm[ij] = acc;
    }
}

// Forward walk of one segment: g of every row, dq, and the segment's sum of
// phi(q_i) g_i^T (into p.partial).
template <typename TIn>
__global__ void __launch_bounds__(kBwdThreads, 1) bwd_q_kernel(FwdParams p, int prefix_is_zero) {
    const int u = blockIdx.x, h = blockIdx.y;
    if (u >= p.hdr->n_units) return;
    const Unit un = p.units[u];
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const BwdView w = bwd_view(smem_raw, plan_bwd_smem(p.dk, p.dv, p.r, true));
    // features read Omega transposed ([dk][r]: lanes over features, coalesced), the chain
    // rule reads it as given ([r][dk]: lanes over input columns, coalesced)
    const OmegaView om_phi{p.omega_t, p.r, 1};
    const OmegaView om = (p.map == LA_MAP_FAVOR) ? stage_omega(nullptr, p.omega, p.dk, p.r) : OmegaView{nullptr, 0, 0};
    const int r = p.r, dv = p.dv, dvx = p.dvx, dk = p.dk;
    const int E = r * dvx;
    const bool attn = p.norm == LA_NORM_ATTENTION;
    const bool tiled = p.map == LA_MAP_FAVOR;   // FAVOR+ features from the transposed Omega, tiled
    const float* src = p.prefix + ((int64_t)u * p.H + h) * E;
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        w.st[e] = prefix_is_zero ? 0.f : src[e];
        w.racc[e] = 0.f;
    }
    const TIn* Q = static_cast<const TIn*>(p.q);
    const TIn* K = static_cast<const TIn*>(p.k);
    const TIn* V = static_cast<const TIn*>(p.v);
    const TIn* DO = static_cast<const TIn*>(p.dout);
    TIn* DQ = static_cast<TIn*>(p.dq_out);
    for (int64_t t0 = un.start; t0 < un.end; t0 += CS) {
        const int n = (int)min64(CS, un.end - t0);
        __syncthreads();
        load_rows(w.xq, Q, t0, n, p.H, h, dk);
        load_rows(w.go, DO, t0, n, p.H, h, dv);
        if (p.causal) {
            load_rows(w.xk, K, t0, n, p.H, h, dk);
            load_vx(w.vx, V, t0, n, p.H, h, dv);
        }
        __syncthreads();
        if (tiled) {
            favor_features_tiled(w.phq, w.xq, w.hsq, p.omega_t, n, dk, r);
            if (p.causal) favor_features_tiled(w.phk, w.xk, w.hsk, p.omega_t, n, dk, r);
        } else {
            compute_phi(w.phq, w.xq, w.hsq, om_phi, n, p.map, dk, r);
            if (p.causal) compute_phi(w.phk, w.xk, w.hsk, om_phi, n, p.map, dk, r);
        }
        __syncthreads();
        if (p.norm == LA_NORM_SUM) {
            sum_normalise_keep(w.phq, w.sgq, n, r, p.eps);
            if (p.causal) sum_normalise_keep(w.phk, w.sgk, n, r, p.eps);
            __syncthreads();
        }
        if (p.causal) {
            causal_scores(w.a, w.phq, w.phk, n, r);
            __syncthreads();
        }
        // num | den of each row: phi(q_i) S (+ in-chunk terms)
        if ((r & 3) == 0) {
            rows_times_state<false>(w.num, dvx, w.phq, w.st, p.causal ? w.a : nullptr, w.vx, r, dvx, dvx);
        } else {
            for (int e = threadIdx.x; e < n * dvx; e += blockDim.x) {
                const int i = e / dvx, c = e - i * dvx;
                float acc = 0.f;
                for (int f = 0; f < r; ++f) acc = fmaf(w.phq[i * r + f], w.st[f * dvx + c], acc);
                if (p.causal) {
#pragma unroll
                    for (int j = 0; j < CS; ++j) acc = fmaf(w.a[i * CS + j], w.vx[j * dvx + c], acc);
                }
                w.num[e] = acc;
            }
        }
        __syncthreads();
        // g_i = dL/d(num_i | den_i)
        for (int e = threadIdx.x; e < CS * dvx; e += blockDim.x) {
            const int i = e / dvx, c = e - i * dvx;
            float gv = 0.f;
            if (i < n) {
                if (!attn) {
                    gv = c < dv ? w.go[i * dv + c] : 0.f;
                } else {
                    const float den = w.num[i * dvx + dv];
                    const float dc = fmaxf(den, p.eps);
                    if (c < dv) {
                        gv = w.go[i * dv + c] / dc;
                    } else if (den > p.eps) {
                        float dot = 0.f;   // dout_i . out_i
                        for (int c2 = 0; c2 < dv; ++c2) dot = fmaf(w.go[i * dv + c2], w.num[i * dvx + c2] / dc, dot);
                        gv = -dot / den;
                    }
                }
                p.g[((t0 + i) * p.H + h) * (int64_t)dvx + c] = gv;
            }
            w.gg[e] = gv;
        }
        __syncthreads();
        if (p.causal) {
            causal_gv(w.gm, w.gg, w.vx, n, dvx);
            __syncthreads();
        }
        // dphi(q_i) = S g_i (+ sum_{j<=i} (g_i . [v_j|1]) phi(k_j))
        if ((r & 1) == 0) {
            state_times_rows<false>(w.dph, w.st, w.gg, p.causal ? w.gm : nullptr, w.phk, r, dvx);
        } else {
            for (int e = threadIdx.x; e < n * r; e += blockDim.x) {
                const int i = e / r, f = e - i * r;
                float acc = 0.f;
                for (int c = 0; c < dvx; ++c) acc = fmaf(w.st[f * dvx + c], w.gg[i * dvx + c], acc);
                if (p.causal) {
#pragma unroll
                    for (int j = 0; j < CS; ++j) acc = fmaf(w.gm[i * CS + j], w.phk[j * r + f], acc);
                }
                w.dph[e] = acc;
            }
        }
        __syncthreads();   // the state is read above and updated below
        // the segment's sum of phi(q_i) g_i^T, and (causal) the state after the chunk
        if ((r & 3) == 0) {
            rank_cs_update(w.racc, w.phq, w.gg, r, dvx);
            if (p.causal) rank_cs_update(w.st, w.phk, w.vx, r, dvx);
        } else {
            for (int e = threadIdx.x; e < E; e += blockDim.x) {
                const int f = e / dvx, c = e - f * dvx;
                float ra = w.racc[e];
#pragma unroll
                for (int i = 0; i < CS; ++i) ra = fmaf(w.phq[i * r + f], w.gg[i * dvx + c], ra);
                w.racc[e] = ra;
                if (p.causal) {
                    float sa = w.st[e];
#pragma unroll
                    for (int i = 0; i < CS; ++i) sa = fmaf(w.phk[i * r + f], w.vx[i * dvx + c], sa);
                    w.st[e] = sa;
                }
            }
        }
        __syncthreads();
        features_vjp_rows(w.dph, w.phq, w.xq, w.sgq, w.su, n, p, om, DQ, t0, h);
    }
    __syncthreads();
    float* dst = p.partial + ((int64_t)u * p.H + h) * E;
    for (int e = threadIdx.x; e < E; e += blockDim.x) dst[e] = w.racc[e];
}

// Backward walk of one segment: R starts as the sum of phi(q) g^T over the
// later segments (the whole sequence for the bidirectional form); writes dk
// and dv.
template <typename TIn>
__global__ void __launch_bounds__(kBwdThreads, 1) bwd_kv_kernel(FwdParams p) {
    const int u = blockIdx.x, h = blockIdx.y;
    if (u >= p.hdr->n_units) return;
    const Unit un = p.units[u];
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const BwdView w = bwd_view(smem_raw, plan_bwd_smem(p.dk, p.dv, p.r, false));
    const OmegaView om_phi{p.omega_t, p.r, 1};
    const OmegaView om = (p.map == LA_MAP_FAVOR) ? stage_omega(nullptr, p.omega, p.dk, p.r) : OmegaView{nullptr, 0, 0};
    const int r = p.r, dv = p.dv, dvx = p.dvx, dk = p.dk;
    const int E = r * dvx;
    float* R = w.st;
    const float* src = p.suffix + ((int64_t)u * p.H + h) * E;
    for (int e = threadIdx.x; e < E; e += blockDim.x) R[e] = src[e];
    const TIn* Q = static_cast<const TIn*>(p.q);
    const TIn* K = static_cast<const TIn*>(p.k);
    const TIn* V = static_cast<const TIn*>(p.v);
    TIn* DK = static_cast<TIn*>(p.dk_out);
    TIn* DV = static_cast<TIn*>(p.dv_out);
    const int nch = (int)ceil_div(un.end - un.start, CS);
    for (int m = nch - 1; m >= 0; --m) {
        const int64_t t0 = un.start + (int64_t)m * CS;
        const int n = (int)min64(CS, un.end - t0);
        __syncthreads();
        load_rows(w.xk, K, t0, n, p.H, h, dk);
        load_vx(w.vx, V, t0, n, p.H, h, dv);
        if (p.causal) load_rows(w.xq, Q, t0, n, p.H, h, dk);
        for (int e = threadIdx.x; e < CS * dvx; e += blockDim.x) {
            const int i = e / dvx;
            w.gg[e] = i < n ? p.g[((t0 + i) * p.H + h) * (int64_t)dvx + (e - i * dvx)] : 0.f;
        }
        __syncthreads();
        if (p.map == LA_MAP_FAVOR) {
            favor_features_tiled(w.phk, w.xk, w.hsk, p.omega_t, n, dk, r);
            if (p.causal) favor_features_tiled(w.phq, w.xq, w.hsq, p.omega_t, n, dk, r);
        } else {
            compute_phi(w.phk, w.xk, w.hsk, om_phi, n, p.map, dk, r);
            if (p.causal) compute_phi(w.phq, w.xq, w.hsq, om_phi, n, p.map, dk, r);
        }
        __syncthreads();
        if (p.norm == LA_NORM_SUM) {
            sum_normalise_keep(w.phk, w.sgk, n, r, p.eps);
            if (p.causal) sum_normalise_keep(w.phq, w.sgq, n, r, p.eps);
            __syncthreads();
        }
        if (p.causal) {
            causal_scores(w.a, w.phq, w.phk, n, r);   // A[i][j], j <= i
            causal_gv(w.gm, w.gg, w.vx, n, dvx);      // Gm[i][j] = g_i . [v_j | 1], j <= i
            __syncthreads();
        }
        // dphi(k_j) = R [v_j | 1] (+ sum_{i>=j} (g_i . [v_j|1]) phi(q_i))
        if ((r & 1) == 0) {
            state_times_rows<true>(w.dph, R, w.vx, p.causal ? w.gm : nullptr, w.phq, r, dvx);
        } else {
            for (int e = threadIdx.x; e < n * r; e += blockDim.x) {
                const int j = e / r, f = e - j * r;
                float acc = 0.f;
                for (int c = 0; c < dvx; ++c) acc = fmaf(R[f * dvx + c], w.vx[j * dvx + c], acc);
                if (p.causal) {
#pragma unroll
                    for (int i = 0; i < CS; ++i) acc = fmaf(w.gm[i * CS + j], w.phq[i * r + f], acc);
                }
                w.dph[e] = acc;
            }
        }
        // dv_j = R^T phi(k_j) (+ sum_{i>=j} (phi(q_i) . phi(k_j)) g_i), first d_v entries
        if ((r & 3) == 0) {
            rows_times_state<true>(w.num, dvx, w.phk, R, p.causal ? w.a : nullptr, w.gg, r, dvx, dv);
            __syncthreads();
            for (int e = threadIdx.x; e < n * dv; e += blockDim.x) {
                const int j = e / dv, c = e - j * dv;
                store_elem(DV, ((t0 + j) * p.H + h) * (int64_t)dv + c, w.num[j * dvx + c]);
            }
        } else {
            for (int e = threadIdx.x; e < n * dv; e += blockDim.x) {
                const int j = e / dv, c = e - j * dv;
                float acc = 0.f;
                for (int f = 0; f < r; ++f) acc = fmaf(R[f * dvx + c], w.phk[j * r + f], acc);
                if (p.causal) {
#pragma unroll
                    for (int i = 0; i < CS; ++i) acc = fmaf(w.a[i * CS + j], w.gg[i * dvx + c], acc);
                }
                store_elem(DV, ((t0 + j) * p.H + h) * (int64_t)dv + c, acc);
            }
        }
        __syncthreads();   // R is read above and updated below
        if (p.causal) {
            if ((r & 3) == 0) {
                rank_cs_update(R, w.phq, w.gg, r, dvx);
            } else {
                for (int e = threadIdx.x; e < E; e += blockDim.x) {
                    const int f = e / dvx, c = e - f * dvx;
                    float ra = R[e];
#pragma unroll
                    for (int i = 0; i < CS; ++i) ra = fmaf(w.phq[i * r + f], w.gg[i * dvx + c], ra);
                    R[e] = ra;
                }
            }
        }
        __syncthreads();
        features_vjp_rows(w.dph, w.phk, w.xk, w.sgk, w.su, n, p, om, DK, t0, h);
    }
}

__global__ void transpose_omega_kernel(const float* omega, float* omega_t, int r, int d) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;   // index into omega_t [d][r]
    if (i < r * d) {
        const int c = i / r, f = i - c * r;
        omega_t[i] = omega[(int64_t)f * d + c];
    }
}

}  // namespace

cudaError_t bwd_transpose_omega(const FwdParams& p, cudaStream_t s) {
    const int n = p.r * p.dk;
    transpose_omega_kernel<<<(n + 255) / 256, 256, 0, s>>>(p.omega, p.omega_t, p.r, p.dk);
    return cudaGetLastError();
}

size_t bwd_smem_bytes(int dk, int dv, int r) { return plan_bwd_smem(dk, dv, r, true).total; }

template <typename Kern>
static cudaError_t bwd_set_smem(Kern k, size_t bytes) {
    return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

cudaError_t bwd_q(const FwdParams& p, int dtype, int prefix_is_zero, cudaStream_t s) {
    const size_t bytes = plan_bwd_smem(p.dk, p.dv, p.r, true).total;
    const dim3 grid((unsigned)p.U, (unsigned)p.H);
    cudaError_t e;
    if (dtype == LA_F32) {
        if ((e = bwd_set_smem(bwd_q_kernel<float>, bytes)) != cudaSuccess) return e;
        bwd_q_kernel<float><<<grid, kBwdThreads, bytes, s>>>(p, prefix_is_zero);
    } else {
        if ((e = bwd_set_smem(bwd_q_kernel<__nv_bfloat16>, bytes)) != cudaSuccess) return e;
        bwd_q_kernel<__nv_bfloat16><<<grid, kBwdThreads, bytes, s>>>(p, prefix_is_zero);
    }
    return cudaGetLastError();
}

cudaError_t bwd_kv(const FwdParams& p, int dtype, cudaStream_t s) {
    const size_t bytes = plan_bwd_smem(p.dk, p.dv, p.r, false).total;
    const dim3 grid((unsigned)p.U, (unsigned)p.H);
    cudaError_t e;
    if (dtype == LA_F32) {
        if ((e = bwd_set_smem(bwd_kv_kernel<float>, bytes)) != cudaSuccess) return e;
        bwd_kv_kernel<float><<<grid, kBwdThreads, bytes, s>>>(p);
    } else {
        if ((e = bwd_set_smem(bwd_kv_kernel<__nv_bfloat16>, bytes)) != cudaSuccess) return e;
        bwd_kv_kernel<__nv_bfloat16><<<grid, kBwdThreads, bytes, s>>>(p);
    }
    return cudaGetLastError();
}

}  // namespace la
