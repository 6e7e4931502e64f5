// Tensor-core (tcgen05) kernels for bf16 inputs with d_k = d_v = 64.
//
// A chunk is 128 consecutive tokens of one head; one CTA owns one unit (a
// segment of a sequence) of one head and walks its chunks in order:
//
//   FAVOR+ projection   P = X Omega'^T with Omega' = log2(e) Omega held as two
//                       bf16 parts (hi + lo, ~16 significant bits), so the
//                       exponent carries no bf16 rounding of Omega; one more K
//                       step adds each row's offset -c, c = log2(e) |x|^2/2 +
//                       log2(sqrt r) ("The Kernel Zoo" §4.2, "Performer" §2
//                       Step 3); the epilogue writes phi = 2^(P - c) times an
//                       exact power of two as f16, the operand of the products
//   ELU+1 / identity    the same MMA with an identity "projection", phi
//                       element-wise in the epilogue
//   causal scores       A (+)= Phi_Q Phi_K^T                  (TMEM, fp32)
//   cross-chunk readout O_x (+)= Phi_Q [S|z]  (state before this chunk, an f16
//                       copy with z also as its f16 remainder)
//   state update        [S|z] += Phi_K^T [V|1]                (TMEM, fp32, carried)
//   causal in-chunk     O_in = tril(A) [V|1]  (diagonal included, "The Kernel Zoo"
//                       §1.3), A as f16 from tensor memory
//   store               out = num / max(den, eps)  ("Performer" §3 sketch clamp),
//                       num | den = 2^t O_in + 2^g O_x in fp32
//
// Every product is tcgen05.mma kind::f16 with both operands f16 and fp32
// accumulation; each operand carries an exact power-of-two scale (per query row,
// per key chunk or feature, per score row, per state copy) that keeps the values
// that matter normal f16 numbers and is undone in fp32.  The ones column of
// [V|1] makes column 64 of every state z and of every numerator the denominator,
// so numerator and denominator see the same rounded weights.  The causal kernel
// processes the feature dimension in halves of 128 (keys) and quarters of 64
// (queries) so that its operands fit in shared memory; the bidirectional output
// kernel reads the whole-sequence state; the state kernel only projects k and
// updates the state.
//
// Shared-memory operands use the 128-byte-swizzled [rows][64] layout of
// tc_ptx.cuh.  The kernels are warp-specialised (each kernel's roles are listed
// above it): one elected thread issues the TMA loads, one the projection MMAs and
// one the product MMAs; epilogue warps own TMEM lanes 32 (w mod 4) .. + 31.  Waits
// are bounded: a wait that runs out records LA_DEVERR_WAIT_TIMEOUT in the
// workspace, and the CTA drains its outstanding copies and MMAs, frees TMEM and
// returns.
#include "internal.h"
#include "tc_ptx.cuh"

namespace la {

namespace {

using namespace tc;

constexpr int kC = 128;                          // tokens per chunk
constexpr int kThreads = 128;
constexpr uint32_t kTile = kC * 64 * 2;          // [128][64] bf16 = 16 KB
constexpr uint32_t kOmgBytes = 256 * 128;        // Omega' part [256][64] bf16 = 32 KB
constexpr int kNX = 80;                          // d_v + ones column, padded to a multiple of 16
constexpr uint32_t kSbfBlock = kNX * 128;        // [80][64] bf16 = 10 KB

// Tensor-memory columns of the feature-map kernel (512 allocated by every kernel).
constexpr uint32_t kColP = 368;   // projection of up to 128 features [128][128]
constexpr uint32_t kTmemCols = 512;

constexpr float kLog2e = 1.4426950408889634f;
// bound on the exit-time wait for a TMA load the CTA issued (it completes in microseconds)
constexpr uint64_t kDrainLimitNs = 100000000ull;
// Test hook (la_test_force_wait_timeout): nonzero makes the causal output kernel's projection
// epilogue wait on a barrier that nothing arrives at, with kForcedWaitLimitNs.
__device__ int g_force_wait_timeout = 0;
constexpr uint64_t kForcedWaitLimitNs = 1000000ull;

typedef unsigned char Tile[kTile];

struct Bars {
    uint64_t load;       // q (and k) tiles
    uint64_t load_v;     // v tile
    uint64_t mma;        // score / readout / update / in-chunk products
    uint64_t proj[2];    // projection into TMEM buffer 0 / 1
    uint64_t drain;
    uint32_t tmem_base;
    int pad;
};

// Bidirectional output kernel: 208 KB.
struct BidirBars {
    uint64_t q_full[2], q_empty[2];   // TMA -> NE, projection issuer;  (projection commit + 2 NE) -> TMA
    uint64_t cx_full[2];              // NE (2 warps) -> projection issuer: offsets of the stage's queries staged
    uint64_t p_full[2], p_empty[2];   // projection commit -> PE: exponent of a feature half;  PE (8 warps) -> issuer
    uint64_t a_full[2], a_empty[2];   // PE (8 warps) -> readout issuer: phi(q) f16 in TMEM;  readout commit -> PE
    uint64_t o_full, o_empty;         // readout commit -> OE: numerator/denominator;  OE (4 warps) -> readout issuer
    uint64_t rx_full[2];              // PE (8 warps) -> PE: per-row maxima of a chunk posted (two slots)
    uint64_t srow_free[2];            // OE (4 warps) -> PE: the row scales of a chunk read (two slots)
    uint64_t drain[2];
    uint32_t tmem_base;
    int pad;
};

struct __align__(1024) BidirSmem {
    unsigned char omg_hi[kOmgBytes];
    unsigned char omg_lo[kOmgBytes];
    Tile tq[2];                       // two stages
    Tile bias;                        // K-major [query][64]: columns 16 st, 16 st + 1 = -offset (hi, lo)
    Tile ones;                        // K-major [feature][64]: columns 16 i, 16 i + 1 = 1
    unsigned char sf16[4][kSbfBlock]; // whole-sequence [S|z]^T 2^-g as f16: rows 0..63 S, 64 z (hi), 65 z (lo)
    float rowmax[2][2][kC];           // per chunk slot, warpgroup and query row: the maximum it saw
    int srow[2][kC];                  // per chunk slot and query row: the exponent of its phi(q) scale
    int gexp;                         // exponent g of the state copy's scale
    float red[32];                    // per-warp maxima of the set-up
    BidirBars b;
};

// Segment-state kernel: 196 KB.
constexpr int kStateStages = 3;
struct StateBars {
    uint64_t k_full[kStateStages], k_empty[kStateStages];   // TMA -> NE / PE;  (projection commit + NE) / 8 PE warps -> TMA
    uint64_t v_full[kStateStages], v_empty[kStateStages];   // TMA -> NE;  update commit -> TMA
    uint64_t vh_full[kStateStages];   // NE (2 warps) -> update issuer: the stage's V converted to f16
    uint64_t cx_full[kStateStages];   // NE -> projection issuer: exponent offsets of the stage's tokens staged
    uint64_t red_full[2];    // PE (8 warps) -> PE: per-warp maxima of a job posted
    uint64_t p_full[2];      // projection commit -> PE: phi exponent of a feature half in buffer b
    uint64_t a_full[2];      // PE (8 warps) -> update issuer: phi(k)^T of that half in buffer b (bf16)
    uint64_t a_empty[2];     // update commit -> projection issuer: buffer b read
    uint64_t pmx_full[4][2]; // r = 256: the two PE warps of a TMEM lane quarter -> each other: maxima of half h posted
    uint64_t drain[2];
    uint32_t tmem_base;
    int pad;
};

struct __align__(1024) StateSmem {
    unsigned char omg_hi[kOmgBytes];
    unsigned char omg_lo[kOmgBytes];
    Tile tk[kStateStages], tv[kStateStages];
    Tile bias;                    // K-major [token][64]: columns 16 st, 16 st + 1 = -offset (hi, lo) of stage st
    Tile ones;                    // K-major [feature][64]: columns 16 i, 16 i + 1 = 1 (bf16)
    unsigned char ones16[2048];   // f16 ones atom of the update's [V|1]: (row, 0) = 1 (column 64 = z)
    float red[2][8];              // PE maxima per warp (two slots)
    float pmx[2][2][128];         // r = 256: per-feature maxima of half h over tokens 64 wg .. 64 wg + 63
    int kmx[4];                   // per chunk (ring of 4): largest key exponent e over the features
    int rsf[256];                 // each feature's final state scale exponent
    StateBars b;
};
// the [S|z] block of up to 256 features leaves through the k / v stages
static_assert(256 * 65 * sizeof(float) <= 2 * kStateStages * sizeof(Tile), "state staging does not fit");

// Feature-map kernel: 80 KB.
struct __align__(1024) FmapSmem {
    unsigned char omg_hi[kOmgBytes];
    unsigned char omg_lo[kOmgBytes];
    Tile tq;
    Bars b;
};

template <typename S>
constexpr size_t smem_bytes() { return sizeof(S) + 1024; }

template <typename S>
__device__ __forceinline__ S& smem_ref() {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    return *reinterpret_cast<S*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
}

struct TcParams {
    FwdParams p;
    int prefix_is_zero;
};

// ---------------------------------------------------------------------------
// Set-up helpers
// ---------------------------------------------------------------------------
// Omega' = log2(e) * Omega as bf16 hi + lo, [r][64] each, K-major swizzled
// (the B operand of the projection).  lo = bf16(Omega' - hi).
__device__ void stage_omega(unsigned char* hi, unsigned char* lo, const float* __restrict__ omega, int r) {
    constexpr int kBatch = 4;   // 16-byte chunks per thread whose loads are in flight together
    const int n = r * 8;
    for (int i0 = threadIdx.x; i0 < n; i0 += kBatch * blockDim.x) {
        float4 a[kBatch], b[kBatch];
#pragma unroll
        for (int q = 0; q < kBatch; ++q) {
            const int i = i0 + q * blockDim.x;
            a[q] = b[q] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (i < n) {
                const float4* src = reinterpret_cast<const float4*>(omega + (i >> 3) * 64 + (i & 7) * 8);
                a[q] = __ldg(src);
                b[q] = __ldg(src + 1);
            }
        }
#pragma unroll
        for (int q = 0; q < kBatch; ++q) {
            const int i = i0 + q * blockDim.x;
            if (i >= n) break;
            const int row = i >> 3, c = i & 7;
            const float x[8] = {a[q].x * kLog2e, a[q].y * kLog2e, a[q].z * kLog2e, a[q].w * kLog2e,
                                b[q].x * kLog2e, b[q].y * kLog2e, b[q].z * kLog2e, b[q].w * kLog2e};
            uint32_t wh[4], wl[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                wh[j] = pack_bf16x2(x[2 * j], x[2 * j + 1]);
                wl[j] = pack_bf16x2(x[2 * j] - bf16lo(wh[j]), x[2 * j + 1] - bf16hi(wh[j]));
            }
            *reinterpret_cast<uint4*>(hi + sw128_chunk(row, c)) = make_uint4(wh[0], wh[1], wh[2], wh[3]);
            *reinterpret_cast<uint4*>(lo + sw128_chunk(row, c)) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
        }
    }
}

// |x_t|^2 of row t of a staged [128][64] bf16 tile.
__device__ float row_sq_norm(const unsigned char* tile, int t) {
    float s = 0.f;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const uint4 w = *reinterpret_cast<const uint4*>(tile + sw128_chunk(t, c));
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float lo = bf16lo(ws[j]), hi = bf16hi(ws[j]);
            s = fmaf(lo, lo, s);
            s = fmaf(hi, hi, s);
        }
    }
    return s;
}

// |x|^2 of rows t0 and t1 of a tile: four independent partial sums, so that the
// FMA latencies overlap (the sums differ from row_sq_norm's in rounding order only).
__device__ __forceinline__ void row_sq_norm2(const unsigned char* tile, int t0, int t1, float& n0, float& n1) {
    float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const uint4 u = *reinterpret_cast<const uint4*>(tile + sw128_chunk(t0, c));
        const uint4 v = *reinterpret_cast<const uint4*>(tile + sw128_chunk(t1, c));
        const uint32_t wu[4] = {u.x, u.y, u.z, u.w}, wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            a0 = fmaf(bf16lo(wu[j]), bf16lo(wu[j]), a0);
            a1 = fmaf(bf16hi(wu[j]), bf16hi(wu[j]), a1);
            b0 = fmaf(bf16lo(wv[j]), bf16lo(wv[j]), b0);
            b1 = fmaf(bf16hi(wv[j]), bf16hi(wv[j]), b1);
        }
    }
    n0 = a0 + a1;
    n1 = b0 + b1;
}

// Exponent offset of the FAVOR+ epilogue for row t: log2(e) |x|^2 / 2 + log2(sqrt r).
__device__ __forceinline__ float favor_offset(const unsigned char* tile, int t, int r) {
    return row_sq_norm(tile, t) * (0.5f * kLog2e) + 0.5f * __log2f((float)r);
}

// FAVOR+ exponent offsets of row t of the q and k tiles (as favor_offset, two
// independent sums so that their latencies overlap).
__device__ __forceinline__ void favor_offsets2(const unsigned char* tq, const unsigned char* tk, int t, int r,
                                               float& oq, float& ok) {
    float sq = 0.f, sk = 0.f;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const uint4 a = *reinterpret_cast<const uint4*>(tq + sw128_chunk(t, c));
        const uint4 b = *reinterpret_cast<const uint4*>(tk + sw128_chunk(t, c));
        const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            sq = fmaf(bf16lo(wa[j]), bf16lo(wa[j]), sq);
            sq = fmaf(bf16hi(wa[j]), bf16hi(wa[j]), sq);
            sk = fmaf(bf16lo(wb[j]), bf16lo(wb[j]), sk);
            sk = fmaf(bf16hi(wb[j]), bf16hi(wb[j]), sk);
        }
    }
    const float lr = 0.5f * __log2f((float)r);
    oq = sq * (0.5f * kLog2e) + lr;
    ok = sk * (0.5f * kLog2e) + lr;
}

// DPFP-nu features of one row ("The Kernel Zoo" §6.3): x~ = relu([x, -x]) in
// R^128 (d = 64), feature (s-1) 128 + a = x~_a x~_{(a+s) mod 128}.  xw holds
// the row's 64 bf16 inputs in pairs (element j in half j & 1 of xw[j >> 1]);
// hi receives features A0 .. A0 + 31 of shift S as bf16 pairs and lo their
// rounding remainders (a product of two bf16 values has up to 16 significant
// bits).  Every index is a compile-time constant, so the row stays in registers.
template <int S, int A0>
__device__ __forceinline__ void dpfp_features32(const uint32_t (&xw)[32], uint32_t (&hi)[16], uint32_t (&lo)[16]) {
    auto xval = [&](int j) { return (j & 1) ? bf16hi(xw[j >> 1]) : bf16lo(xw[j >> 1]); };
    auto xt = [&](int j) { return j < 64 ? fmaxf(xval(j), 0.f) : fmaxf(-xval(j - 64), 0.f); };
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
        const int a = A0 + i;
        const float f0 = xt(a) * xt((a + S) & 127), f1 = xt(a + 1) * xt((a + 1 + S) & 127);
        const uint32_t h = pack_bf16x2(f0, f1);
        hi[i >> 1] = h;
        lo[i >> 1] = pack_bf16x2(f0 - bf16lo(h), f1 - bf16hi(h));
    }
}

// 32 fp32 values of row t, columns f0..f0+31 -> bf16 into 64-wide blocks blk[f0 / 64].
__device__ __forceinline__ void store_row32_bf16(unsigned char* blk0, int t, int f0, const uint32_t (&w)[16]) {
    unsigned char* blk = blk0 + kTile * (f0 >> 6);
    const int cb = (f0 & 63) >> 3;
#pragma unroll
    for (int q = 0; q < 4; ++q)
        *reinterpret_cast<uint4*>(blk + sw128_chunk(t, cb + q)) =
            make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
}

// fp32 projection epilogue for la_feature_map: phi = 2^(p - c) to global fp32.
__device__ void projection_to_global(uint32_t tbase, int nf, float c, bool valid, float* dst) {
    const int warp = threadIdx.x >> 5;
    for (int f0 = 0; f0 < nf; f0 += 32) {
        uint32_t v[32];
        tmem_ld32(tmem_addr(tbase, warp * 32, kColP + f0), v);
        tmem_ld_wait();
        if (valid) {
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
                const float4 o = make_float4(ex2_approx(__uint_as_float(v[j]) - c),
                                             ex2_approx(__uint_as_float(v[j + 1]) - c),
                                             ex2_approx(__uint_as_float(v[j + 2]) - c),
                                             ex2_approx(__uint_as_float(v[j + 3]) - c));
                *reinterpret_cast<float4*>(dst + f0 + j) = o;
            }
        }
    }
}

// Sum over features nf of phi = 2^(P - c) of this thread's row (TMEM lane), in fp32.
__device__ float projection_rowsum(uint32_t tbase, int nf, float c) {
    const int warp = threadIdx.x >> 5;
    float acc = 0.f;
    for (int f0 = 0; f0 < nf; f0 += 32) {
        uint32_t v[32];
        tmem_ld32(tmem_addr(tbase, warp * 32, kColP + f0), v);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) acc += ex2_approx(__uint_as_float(v[j]) - c);
    }
    return acc;
}

// 64 bf16 (packed in pairs) as row `row` of a 128-byte-swizzled tile.
__device__ __forceinline__ void state_row_bf16(unsigned char* tile, int row, const uint32_t (&w)[32]) {
#pragma unroll
    for (int c = 0; c < 8; ++c)
        *reinterpret_cast<uint4*>(tile + sw128_chunk(row, c)) = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
}

// One output row from registers as bf16 to global: out = O[0..63] * mult.
__device__ __forceinline__ void store_output_row_f(const uint32_t (&a)[32], const uint32_t (&b)[32], float mult,
                                                   __nv_bfloat16* dst_row) {
    uint4* dst = reinterpret_cast<uint4*>(dst_row);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const uint32_t* x = q < 4 ? a + 8 * q : b + 8 * (q - 4);
        dst[q] = make_uint4(pack_bf16x2(__uint_as_float(x[0]) * mult, __uint_as_float(x[1]) * mult),
                            pack_bf16x2(__uint_as_float(x[2]) * mult, __uint_as_float(x[3]) * mult),
                            pack_bf16x2(__uint_as_float(x[4]) * mult, __uint_as_float(x[5]) * mult),
                            pack_bf16x2(__uint_as_float(x[6]) * mult, __uint_as_float(x[7]) * mult));
    }
}

// Factor that turns a row's scaled numerator O (the true one times 2^-e) into the
// output: attention normalisation divides by max(den 2^e, eps) ("Performer" §3
// sketch clamp), none multiplies by 2^e, sum normalisation divides the true
// numerator by max(sigma_q, eps) of the row.
__device__ __forceinline__ float row_multiplier(float den, int e, const FwdParams& p, int64_t orow) {
    if (p.div_rows) return exp2i(e) / fmaxf(p.div_rows[orow], p.eps);
    if (p.norm != LA_NORM_ATTENTION) return exp2i(e);
    return den >= p.eps * exp2i(-e) && den > 0.f ? 1.0f / den : exp2i(e) / p.eps;
}

// The whole-sequence state [r][65] (fp32, true scale) as the f16 B operand of the
// bidirectional readout: K-major blocks [80 rows][64 features], row n < 64 = S[:, n],
// row 64 = z, row 65 = the f16 remainder of z, other rows 0; all times 2^-g with g
// chosen so that the largest entry lies in (2^13, 2^14].  Called by every thread of
// the block during set-up (it synchronises); writes g to *gexp.
__device__ void load_state_f16(unsigned char (*dst)[kSbfBlock], const float* src, int r, int nhalves, float* red,
                               int* gexp) {
    const int t = threadIdx.x, nthreads = blockDim.x;
    // the largest |entry|: 16-byte loads over the contiguous [r][65] block (r * 65 is a
    // multiple of 4 and the block starts 16-byte aligned), every thread of the block
    float m = 0.f;
    const float4* src4 = reinterpret_cast<const float4*>(src);
    for (int i = t; i < r * 65 / 4; i += nthreads) {
        const float4 x = src4[i];
        m = fmaxf(m, fmaxf(fmaxf(fabsf(x.x), fabsf(x.y)), fmaxf(fabsf(x.z), fabsf(x.w))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((t & 31) == 0) red[t >> 5] = m;
    __syncthreads();
    if (t == 0) {
        float mx = 0.f;
        for (int w = 0; w < nthreads / 32; ++w) mx = fmaxf(mx, red[w]);
        *gexp = mx > 0.f && mx < INFINITY ? (int)ceilf(__log2f(mx)) - 14 : 0;
    }
    __syncthreads();
    const float mul = exp2i(-*gexp);
    // rows 66..79 of every block and the blocks of features r.. are zero
    const int nblk = 2 * nhalves;
    for (int i = t; i < nblk * kSbfBlock / 16; i += nthreads) {
        const int blk = i / (kSbfBlock / 16), off = (i - blk * (kSbfBlock / 16)) * 16;
        if (off >= 66 * 128 || 64 * blk >= r)
            *reinterpret_cast<uint4*>(dst[blk] + off) = make_uint4(0u, 0u, 0u, 0u);
    }
    // entry (f, n) of the state, in its own (contiguous) order, to row n (64, 65: z as f16 and
    // its remainder), column f of the K-major operand blocks [80][64]
    for (int e = t; e < r * 65; e += nthreads) {
        const int f = e / 65, n = e - 65 * f;
        const float x = src[e] * mul;
        unsigned char* blk = dst[f >> 6];
        if (n < 64) {
            *reinterpret_cast<__half*>(blk + sw128_off(n, f & 63)) = __float2half_rn(x);
        } else {
            const __half zh = __float2half_rn(x);
            *reinterpret_cast<__half*>(blk + sw128_off(64, f & 63)) = zh;
            *reinterpret_cast<__half*>(blk + sw128_off(65, f & 63)) = __float2half_rn(x - __half2float(zh));
        }
    }
}

// ---------------------------------------------------------------------------
// Synchronisation and MMA helpers
// ---------------------------------------------------------------------------
// Every thread waits for the phase; returns false for all threads if any timed out.
__device__ __forceinline__ bool wait_all(uint64_t* bar, uint32_t parity) {
    const bool ok = mbar_wait(bar, parity);
    return __syncthreads_or(!ok) == 0;
}
// Shared-memory writes and TMEM reads of all threads are done before the MMA issuer proceeds.
__device__ __forceinline__ void handoff_to_mma() {
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
}

// D (+)= A B^T, both K-major in 64-wide blocks: A blocks a0 + a_stride*j, B blocks b0 + b_stride*j.
__device__ __forceinline__ void mma_kk(uint32_t d, const unsigned char* a0, uint32_t a_stride, const unsigned char* b0,
                                       uint32_t b_stride, int ksteps, uint32_t idesc, bool accumulate) {
    for (int k = 0; k < ksteps; ++k) {
        const uint64_t ad = sdesc_sw128(smem_u32(a0) + a_stride * (k >> 2) + 32u * (k & 3), 16, 1024);
        const uint64_t bd = sdesc_sw128(smem_u32(b0) + b_stride * (k >> 2) + 32u * (k & 3), 16, 1024);
        mma_ss(d, ad, bd, idesc, (accumulate || k > 0) ? 1u : 0u);
    }
}

// P = X Omega'^T for `nf` features starting at feature f0 into TMEM address d:
// X tile (K = 64) times the hi part, then the lo part accumulated.
__device__ __forceinline__ void mma_projection(uint32_t d, const unsigned char* x, const unsigned char* omg_hi,
                                               const unsigned char* omg_lo, int f0, int nf) {
    const uint32_t idesc = idesc_bf16(128, nf, false, false);
    mma_kk(d, x, 0, omg_hi + 128u * f0, 0, 4, idesc, false);
    mma_kk(d, x, 0, omg_lo + 128u * f0, 0, 4, idesc, true);
}

__device__ void setup_bars(Bars& b) {
    if (threadIdx.x == 0) {
        mbar_init(&b.load, 1);
        mbar_init(&b.load_v, 1);
        mbar_init(&b.mma, 1);
        mbar_init(&b.proj[0], 1);
        mbar_init(&b.proj[1], 1);
        mbar_init(&b.drain, 1);
        fence_mbar_init();
    }
    if ((threadIdx.x >> 5) == 0) {
        tmem_alloc(&b.tmem_base, kTmemCols);
        tmem_relinquish();
    }
}

// After a timed-out wait: record it, wait (bounded) for this CTA's MMAs to finish.
__device__ void drain_after_timeout(Bars& b, int* err) {
    if (threadIdx.x == 0) {
        if (err) atomicMax(err, LA_DEVERR_WAIT_TIMEOUT);
        mma_commit(&b.drain);
        mbar_wait(&b.drain, 0, 500000000ull);
    }
    __syncthreads();
}

__device__ void teardown(Bars& b) {
    tc_fence_before();
    __syncthreads();
    if ((threadIdx.x >> 5) == 0) tmem_dealloc(b.tmem_base, kTmemCols);
}

// Pending-phase tracker for one mbarrier (all threads keep the same copy).
struct Phase {
    uint32_t bit = 0;
    __device__ __forceinline__ bool wait(uint64_t* bar) {
        const bool ok = wait_all(bar, bit);
        bit ^= 1u;
        return ok;
    }
};

// Descriptor of K step k (16 token rows) of an MN-major [V|1] operand: the start
// advances by 2048 B and the leading-dimension offset (bits 16..29, 16-byte units)
// shrinks by the same amount, so that the second 64-column atom stays on the same
// 16-row ones tile for every step.
__device__ __forceinline__ uint64_t v_ones_desc(uint64_t d0, int k) {
    return d0 + static_cast<uint64_t>(128 * k) - (static_cast<uint64_t>(128 * k) << 16);
}

// The 16-row f16 ones atom of an MN-major [V|1] operand: element (row, 0) = 1.
__device__ void fill_ones_atom_f16(unsigned char* tile, int tid, int nthreads) {
    for (int i = tid; i < 16 * 8; i += nthreads) {
        const int row = i >> 3, c = i & 7;
        *reinterpret_cast<uint4*>(tile + sw128_chunk(row, c)) =
            c == 0 ? make_uint4(0x3C00u, 0u, 0u, 0u) : make_uint4(0u, 0u, 0u, 0u);
    }
}

// Two bf16 values (one word) as two f16 values: exact for |v| in [2^-14, 65504]
// (f16 keeps more significant bits than bf16), rounded in f16's subnormal range,
// |v| > 65504 saturated to 65504 (satfinite).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
    uint32_t r;
    asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;"
        : "=r"(r) : "f"(__uint_as_float(w & 0xFFFF0000u)), "f"(__uint_as_float(w << 16)));
    return r;
}

// Rows row0 .. row0 + nrows - 1 of a [128][64] bf16 tile converted in place to f16
// by `nthreads` cooperating threads (index tid); values beyond the f16 range are
// saturated and, for real tokens (rows < nvalid), reported.  Returns the largest
// |v| among the rows < nvalid this thread converted (for bounds on the state).
__device__ float v_tile_to_f16(unsigned char* tile, int row0, int nrows, int nvalid, WsHeader* hdr, int tid,
                               int nthreads) {
    uint32_t vmax = 0u;
#pragma unroll 4
    for (int i = tid; i < nrows * 8; i += nthreads) {
        const int row = row0 + (i >> 3);
        uint4* p = reinterpret_cast<uint4*>(tile + row * 128 + (i & 7) * 16);
        const uint4 w = *p;
        if (row < nvalid)
            vmax = __vmaxu2(vmax, __vmaxu2(__vmaxu2(w.x & 0x7FFF7FFFu, w.y & 0x7FFF7FFFu),
                                           __vmaxu2(w.z & 0x7FFF7FFFu, w.w & 0x7FFF7FFFu)));
        *p = make_uint4(bf16x2_to_f16x2(w.x), bf16x2_to_f16x2(w.y), bf16x2_to_f16x2(w.z), bf16x2_to_f16x2(w.w));
    }
    // |v| as bf16 bits orders like the value for every non-negative pattern (infinities and NaNs
    // lie above the largest finite): a valid element beyond 65504 shows in the maximum
    const uint32_t m = max(vmax & 0xFFFFu, vmax >> 16);
    if (__any_sync(0xffffffffu, m > 0x477Fu) && (threadIdx.x & 31) == 0) record_range(hdr, kRangeV);
    return __uint_as_float(min(m, 0x4780u) << 16);
}

// ---------------------------------------------------------------------------
// Causal output kernel (warp-specialised)
// ---------------------------------------------------------------------------
// Operands of the feature products are f16 (11 significant bits) with exact
// power-of-two scales, so that every value the products depend on is a normal
// f16 number:
//   phi(k)   2^-e_c for the chunk (e_c from the state kernel: the chunk's largest
//            key feature lands in (2^14, 2^15]); the state [S|z] is held in TMEM
//            times 2^-e_c and rescaled exactly when the chunk's e changes;
//   phi(q)   2^-s_i per query row (s_i from the row's largest exponent over all r
//            features, taken from hi-only projections, so that its largest feature
//            lies just below 2^14); the factor is common to the row's numerator
//            and denominator;
//   scores   A_i. 2^-t_i per row (largest in (2^13, 2^14]), causal mask applied;
//   state    the copy the readout reads is [S|z] 2^-g_c (largest in (2^13, 2^14]),
//            z also as its f16 remainder;
//   V        converted to f16 in place (|v| <= 65504, else clamped).
// The in-chunk numerator O_in = tril(A) [V|1] and the cross-chunk numerator
// O_cross = Phi_Q [S|z] accumulate in separate TMEM blocks (their scales
// differ) and are combined in fp32: num = 2^t_i O_in + 2^g_c O_cross, likewise
// the denominator, all times 2^(s_i + e_c).  Values clamped into the f16 range
// are reported as LA_DEVERR_RANGE.
// Roles (512 threads):
//   warp 0 lane 0      TMA: q, k tiles and the v tile of each chunk
//   warp 1             projection MMAs, one elected lane (warp 1 also owns the TMEM
//                      allocation); runs ahead, throttled by the two projection buffers
//   warp 2             product MMAs (scores, readout, denominator, state update, A V)
//   warp 3             idle (holds no role)
//   warps 4..11 (PE)   projection epilogue in two warpgroups, each converting 32 of
//                      the 64 columns of every job: phi(k), phi(q) of each quarter
//                      of the features into shared memory (token t = TMEM lane t)
//   warps 12..15 (TE)  chunk tail: the chunk's V tile as f16 in place (before its first
//                      state update), FAVOR+: the next chunk's row offsets (once its
//                      tiles land), masked scores as f16 in TMEM, then (while A V
//                      runs) the f16 copy of the state for the next chunk's readout,
//                      then the output rows
// Per chunk the projection warp runs, for each quarter q of the features, the
// projections of k and q (Omega hi + lo) into two TMEM buffers; once the PE has
// written phi, the product warp runs the products of that quarter:
//   A (+)= Phi_Q Phi_K^T,  O_cross (+)= Phi_Q [S|z],  and after the last quarter
//   of each half [S|z] += Phi_K^T [V|1];
// then, once the TE has converted A, O_in = tril(A) [V|1].  All hand-offs are
// mbarriers.  The next chunk's projections overlap this chunk's tail; its
// first products wait only until O has been read out and the TE has written
// the state of the chunks so far.
constexpr int kCausalThreads = 512;

// Tensor-memory columns of the causal kernel (512 allocated).
constexpr uint32_t kColCS = 0;     // state, one 80-column block per feature half (lanes = features)
constexpr uint32_t kColCP = 160;   // two 64-column projection buffers
constexpr uint32_t kColCA = 288;   // scores [128 q][128 k] fp32; then f16 in [288, 352)
constexpr uint32_t kColCI = 352;   // O_in [128][80]: reuses the scores' columns 64.. once converted
constexpr uint32_t kColCX = 432;   // O_cross [128][80]

struct CausalBars {
    uint64_t qk_full, qk_empty;     // TMA -> (MMA, TE or PE);  (MMA commit + 4 TE or 8 PE warps) -> TMA
    uint64_t v_full, v_empty;       // TMA -> TE;         MMA commit -> TMA
    uint64_t vh_full;               // TE (4 warps) -> MMA: V as f16
    uint64_t off_full[2];           // TE (4 warps) -> PE: FAVOR+ offsets of a chunk (slot c & 1)
    uint64_t p_full[2];             // MMA commit -> PE: projection in TMEM buffer b
    uint64_t p_empty[2];            // PE (4 warps) -> MMA: buffer b drained
    uint64_t phik_full[2];          // PE (4 warps) -> MMA: phi(k) of global quarter g in smem (g & 1)
    uint64_t phiq_full[2];          // PE (8 warps) -> MMA: phi(q) of global quarter g in smem (g & 1)
    uint64_t upd_done;              // MMA commit -> PE: a state update has read phi(k) of its half
    uint64_t phq_free[2];           // MMA commit -> PE: products of global quarter g done (g & 1)
    uint64_t a_full;                // MMA commit -> TE: scores, readout, state update of the chunk done
    uint64_t ahl_full;              // TE (4 warps) -> MMA: masked scores as f16 in TMEM
    uint64_t o_full;                // MMA commit -> TE: O_in complete
    uint64_t o_empty;               // TE (4 warps) -> MMA: O_in and O_cross read out of TMEM
    uint64_t sbf_full;              // TE (4 warps) -> MMA, PE: f16 state copy of the previous chunks in smem
    uint64_t rx_full[2];            // PE (8 warps) -> PE: row maxima of phi(q), quarter 0, posted (two slots)
    uint64_t tx_full[2];            // TE (4 warps) -> TE: maxima of the state posted (two slots)
    uint64_t srow_free[2];          // TE (4 warps) -> PE: a chunk's row scales read (two slots)
    uint64_t never;                 // no arrivals: the wait la_test_force_wait_timeout makes run out
    uint64_t drain[2];              // one per MMA-issuing warp
    uint32_t tmem_base;
    int pad;
};

// z of feature f (0..63 within its quarter) as f16 (row 0) and its f16 remainder
// (row 1) of the quarter's 16-row K-major tile: the denominator MMA then yields
// both parts of phi(q) . z in two columns.
__device__ __forceinline__ void store_z_f16(unsigned char* tile, int f, float z) {
    const __half hi = __float2half_rn(z);
    *reinterpret_cast<__half*>(tile + sw128_off(0, f)) = hi;
    *reinterpret_cast<__half*>(tile + sw128_off(1, f)) = __float2half_rn(z - __half2float(hi));
}

struct __align__(1024) CausalSmem {
    unsigned char omg_hi[kOmgBytes];
    unsigned char omg_lo[kOmgBytes];
    Tile tq, tk, tv;
    Tile phq[2];                      // Phi_Q of one quarter (64 features), two buffers
    Tile phk[2];                      // Phi_K of one half (two quarters)
    Tile sbf[2];                      // S 2^-g f16, MN-major [feature][v]: features 128h.. in sbf[h]
    unsigned char zrow[4][2048];      // per quarter: K-major [16][64], rows 0, 1 = z 2^-g as f16 + remainder
    unsigned char ones16[2048];       // f16 ones atom of [V|1]: (row, 0) = 1
    float rowmax[2][2][kC];           // phi(q) row maxima per slot and warpgroup
    int srow[2][kC];                  // per slot and query row: s_i
    float qsum[2][2][kC];             // per slot, warpgroup and query row: sum of |phi(q) 2^-s_i| it wrote
    float tred[2][4];                 // TE maxima per slot and warp
    float vt[2][4];                   // per slot (chunk & 1) and TE warp: largest |v| of its rows
    float offq[2][kC], offk[2][kC];   // per slot: FAVOR+ exponent offsets of the query / key rows
    CausalBars b;
};
static_assert(sizeof(CausalSmem) + 1024 <= 232448, "causal kernel shared memory exceeds 227 KB");

// Power-of-two exponent R of the keys' scale for a chunk whose largest key feature
// exponent bound is e (e = ceil(max) - 15, from the state kernel): the previous R is
// kept while the chunk's largest feature stays within (2^7, 2^15] of the scale, so
// that the state is rescaled only when the keys' magnitude moves; a new R puts the
// largest feature at 2^13.
__device__ __forceinline__ int next_key_scale(int R, int e, bool first) {
    return (first || e > R || e < R - 8) ? e + 2 : R;
}

// Largest of N values as a balanced tree: depth log2 N instead of a chain of N dependent
// maxima, whose latency the few warps of an epilogue cannot hide.
template <int N>
__device__ __forceinline__ float max_tree(const float (&x)[N]) {
    static_assert(N >= 2 && (N & (N - 1)) == 0, "power of two");
    float a[N / 2];
#pragma unroll
    for (int i = 0; i < N / 2; ++i) a[i] = fmaxf(x[2 * i], x[2 * i + 1]);
#pragma unroll
    for (int n = N / 4; n > 0; n >>= 1)
#pragma unroll
        for (int i = 0; i < n; ++i) a[i] = fmaxf(a[i], a[i + n]);
    return a[0];
}
__device__ __forceinline__ float max_tree32(const uint32_t (&v)[32]) {
    float x[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) x[i] = __uint_as_float(v[i]);
    return max_tree(x);
}

// Bounded wait of every lane of a warp; false for the whole warp if any lane timed out.
// Epilogue warps proceed independently and meet only through mbarriers.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity) {
    const bool ok = mbar_wait(bar, parity);
    return !__any_sync(0xffffffffu, !ok);
}
// A warp's threads are done with shared-memory writes / TMEM accesses: lane 0 arrives.
__device__ __forceinline__ void warp_arrive(uint64_t* bar, bool smem_written) {
    if (smem_written) fence_async_smem();
    tc_fence_before();
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

// Element-wise phi (ELU+1 or identity) of row t of a tile as f16 into the same
// position of dst (zero when the row is past the unit's end); |phi| > 65504 is
// clamped.  Adds sum |phi| of the row to `sum`; returns true when it clamped.
__device__ bool elementwise_phi_row_f16(const unsigned char* tile, unsigned char* dst, int t, bool valid, int map,
                                        float& sum) {
    bool big = false;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const uint4 w = *reinterpret_cast<const uint4*>(tile + sw128_chunk(t, c));
        uint4 o = make_uint4(0u, 0u, 0u, 0u);
        if (valid) {
            uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float lo = bf16lo(ws[j]), hi = bf16hi(ws[j]);
                if (map == LA_MAP_ELU1) {   // exponentials unconditional, so that the choices are selects
                    const float el = ex2_approx(lo * kLog2e), eh = ex2_approx(hi * kLog2e);
                    lo = lo > 0.f ? lo + 1.f : el;
                    hi = hi > 0.f ? hi + 1.f : eh;
                }
                big |= !(fabsf(lo) <= 65504.f) || !(fabsf(hi) <= 65504.f);
                lo = fminf(fmaxf(lo, -65504.f), 65504.f);
                hi = fminf(fmaxf(hi, -65504.f), 65504.f);
                sum += fabsf(lo) + fabsf(hi);
                ws[j] = pack_f16x2(lo, hi);
            }
            o = make_uint4(ws[0], ws[1], ws[2], ws[3]);
        }
        *reinterpret_cast<uint4*>(dst + sw128_chunk(t, c)) = o;
    }
    return big;
}

// DPFP-nu features of one row ("The Kernel Zoo" §6.3): x~ = relu([x, -x]) in
// R^128 (d = 64), feature (s-1) 128 + a = x~_a x~_{(a+s) mod 128}, as f16 pairs
// (features A0 .. A0 + 31 of shift S); products beyond 65504 are clamped (big).
template <int S, int A0>
__device__ __forceinline__ void dpfp_features32_f16(const uint32_t (&xw)[32], uint32_t (&out)[16], bool& big,
                                                    float& sum) {
    auto xval = [&](int j) { return (j & 1) ? bf16hi(xw[j >> 1]) : bf16lo(xw[j >> 1]); };
    auto xt = [&](int j) { return j < 64 ? fmaxf(xval(j), 0.f) : fmaxf(-xval(j - 64), 0.f); };
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
        const int a = A0 + i;
        const float f0 = xt(a) * xt((a + S) & 127), f1 = xt(a + 1) * xt((a + 1 + S) & 127);
        big |= !(f0 <= 65504.f) || !(f1 <= 65504.f);
        sum += fminf(f0, 65504.f) + fminf(f1, 65504.f);
        out[i >> 1] = pack_f16x2(fminf(f0, 65504.f), fminf(f1, 65504.f));
    }
}

// Features 64 quarter + 32 half .. + 31 of row t of a [128][64] bf16 input tile,
// as f16 into the same row of dst at columns 32 half .. (zero past the unit's end).
// r = 128 nu: quarters 0, 1 are shift 1, quarters 2, 3 shift 2.  Adds the features'
// sum to `sum`; returns true when a feature was clamped.
__device__ bool dpfp_phi_row32_f16(const unsigned char* tile, unsigned char* dst, int t, bool valid, int quarter,
                                   int half, float& sum) {
    uint32_t xw[32], w[16];
    bool big = false;
    float acc = 0.f;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const uint4 v = *reinterpret_cast<const uint4*>(tile + sw128_chunk(t, c));
        xw[4 * c] = v.x; xw[4 * c + 1] = v.y; xw[4 * c + 2] = v.z; xw[4 * c + 3] = v.w;
    }
    switch (quarter * 2 + half) {
        case 0: dpfp_features32_f16<1, 0>(xw, w, big, acc); break;
        case 1: dpfp_features32_f16<1, 32>(xw, w, big, acc); break;
        case 2: dpfp_features32_f16<1, 64>(xw, w, big, acc); break;
        case 3: dpfp_features32_f16<1, 96>(xw, w, big, acc); break;
        case 4: dpfp_features32_f16<2, 0>(xw, w, big, acc); break;
        case 5: dpfp_features32_f16<2, 32>(xw, w, big, acc); break;
        case 6: dpfp_features32_f16<2, 64>(xw, w, big, acc); break;
        default: dpfp_features32_f16<2, 96>(xw, w, big, acc); break;
    }
    if (!valid) {
#pragma unroll
        for (int j = 0; j < 16; ++j) w[j] = 0u;
        big = false;
        acc = 0.f;
    }
    sum += acc;
#pragma unroll
    for (int q = 0; q < 4; ++q)
        *reinterpret_cast<uint4*>(dst + sw128_chunk(t, 4 * half + q)) = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
    return big;
}

// Maximum over the four TE warps for use j (bounded mbarrier exchange, two slots).
__device__ __forceinline__ bool group_max4(float& m, float (*red)[4], uint64_t* bar, int j, int warp0) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const int slot = j & 1;
    if ((threadIdx.x & 31) == 0) red[slot][(threadIdx.x >> 5) - warp0] = m;
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&bar[slot]);
    if (!warp_wait(&bar[slot], (j >> 1) & 1)) return false;
    m = fmaxf(fmaxf(red[slot][0], red[slot][1]), fmaxf(red[slot][2], red[slot][3]));
    return true;
}

// Exponent g with max * 2^-g in (2^13, 2^14] (0 for max = 0 or not finite).
__device__ __forceinline__ int copy_exponent(float mx) {
    return (mx > 0.f && mx < INFINITY) ? (int)ceilf(__log2f(mx)) - 14 : 0;
}

// FAVOR+ projection schedule of a chunk, in steps of two jobs: one in each TMEM
// projection buffer (kind 0 none, 1 max job, 2 k job, 3 q job; and its quarter).
// The epilogue reads both jobs of a step, frees both buffers, then converts, so
// that the next step's projections run meanwhile.  The q jobs need the rows'
// largest exponents (all max jobs) first; the k jobs do not, and hide the max
// jobs' latency.  Each quarter's k job precedes its q job (the products' order).
struct ProjStep { int kind[2], quarter[2]; };
__device__ __forceinline__ int proj_steps(int nq) { return nq == 4 ? 6 : nq == 2 ? 3 : 2; }
__device__ __forceinline__ ProjStep proj_step(int nq, int i) {
    if (nq == 4) {
        switch (i) {
            case 0: return {{1, 1}, {0, 1}};
            case 1: return {{2, 1}, {0, 2}};
            case 2: return {{2, 1}, {1, 3}};
            case 3: return {{3, 3}, {0, 1}};
            case 4: return {{2, 3}, {2, 2}};
            default: return {{2, 3}, {3, 3}};
        }
    }
    if (nq == 2) {
        switch (i) {
            case 0: return {{1, 1}, {0, 1}};
            case 1: return {{2, 3}, {0, 0}};
            default: return {{2, 3}, {1, 1}};
        }
    }
    return i == 0 ? ProjStep{{1, 0}, {0, 0}} : ProjStep{{2, 3}, {0, 0}};
}

// kFavor: FAVOR+ projections, else element-wise maps of q and k; one instantiation per kind.
template <bool kFavor>
__global__ void __launch_bounds__(kCausalThreads, 1)
tc_causal_out_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                     const __grid_constant__ CUtensorMap map_v, const TcParams tp) {
    const FwdParams& p = tp.p;
    // one block per (unit, head), rank-major: all heads of the longest unit go out first
    const int rank = blockIdx.x / p.H, head = blockIdx.x - rank * p.H;
    if (rank >= p.hdr->n_units) return;
    const int u = p.order[rank];
    const Unit un = p.units[u];
    CausalSmem& s = smem_ref<CausalSmem>();
    CausalBars& B = s.b;
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int r = p.r;
    constexpr bool favor = kFavor;
    const int nq = r / 64;                        // feature quarters (1, 2 or 4)
    const int nhalves = (r + 127) / 128;
    const int nchunks = (un.end - un.start + kC - 1) / kC;
    // exponent of the keys' scale in chunk c (FAVOR+: recorded by the state kernel)
    const int* kscale = favor ? p.kscale + ((int64_t)u * p.H + head) * p.Lc : nullptr;
    auto key_exp = [&](int c) -> int { return favor ? kscale[c] : 0; };
    // V of chunk c into s.tv: FAVOR+ the f16 tile the state kernel wrote (one bulk copy), else the
    // bf16 input tile (the TE converts it in place)
    const unsigned char* v16 = favor ? static_cast<const unsigned char*>(p.v16) + ((int64_t)u * p.H + head) * p.Lc * (int64_t)kTile
                                     : nullptr;
    const float* vmx = favor ? p.vmax + ((int64_t)u * p.H + head) * p.Lc * kVmaxParts : nullptr;
    auto load_v = [&](int c) {
        if (favor) bulk_load(s.tv, v16 + (int64_t)c * kTile, kTile, &B.v_full);
        else tma_load_3d(s.tv, &map_v, 0, head, un.start + c * kC, &B.v_full);
    };
    auto prefetch_v = [&](int c) {
        if (favor) bulk_prefetch_l2(v16 + (int64_t)c * kTile, kTile);
        else tma_prefetch_3d(&map_v, 0, head, un.start + c * kC);
    };

    if (t == 0) {
        prefetch_tensormap(&map_q);
        prefetch_tensormap(&map_k);
        prefetch_tensormap(&map_v);
        mbar_init(&B.qk_full, 1);
        mbar_init(&B.qk_empty, favor ? 5 : 9);   // MMA commit + the 4 TE warps (FAVOR+) or the 8 PE warps
        mbar_init(&B.v_full, 1);
        mbar_init(&B.v_empty, 1);
        mbar_init(&B.vh_full, 4);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&B.p_full[i], 1);
            mbar_init(&B.p_empty[i], 8);
            mbar_init(&B.phik_full[i], 8);
            mbar_init(&B.phiq_full[i], 8);
            mbar_init(&B.phq_free[i], 1);
            mbar_init(&B.rx_full[i], 8);
            mbar_init(&B.off_full[i], 4);
            mbar_init(&B.tx_full[i], 4);
            mbar_init(&B.srow_free[i], 4);
        }
        mbar_init(&B.upd_done, 1);
        mbar_init(&B.a_full, 1);
        mbar_init(&B.ahl_full, 4);
        mbar_init(&B.o_full, 1);
        mbar_init(&B.o_empty, 4);
        mbar_init(&B.sbf_full, 4);
        mbar_init(&B.never, 1);
        mbar_init(&B.drain[0], 1);
        mbar_init(&B.drain[1], 1);
        fence_mbar_init();
        if (nchunks > 0) {   // chunk 0's tiles go out before the set-up below (which does not touch them)
            mbar_arrive_expect_tx(&B.qk_full, 2 * kTile);
            tma_load_3d(s.tq, &map_q, 0, head, un.start, &B.qk_full);
            tma_load_3d(s.tk, &map_k, 0, head, un.start, &B.qk_full);
            mbar_arrive_expect_tx(&B.v_full, kTile);
            load_v(0);
            if (nchunks > 1) prefetch_v(1);
        }
    }
    if (warp == 1) {
        tmem_alloc(&B.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    for (int i = t; i < (favor ? r * 8 : 0); i += kCausalThreads) {
        // Omega' = log2(e) Omega as bf16 hi + lo (one 16-byte chunk per iteration)
        const int row = i >> 3, c = i & 7;
        const float4* src = reinterpret_cast<const float4*>(p.omega + row * 64 + c * 8);
        const float4 a = src[0], b = src[1];
        const float x[8] = {a.x * kLog2e, a.y * kLog2e, a.z * kLog2e, a.w * kLog2e,
                            b.x * kLog2e, b.y * kLog2e, b.z * kLog2e, b.w * kLog2e};
        uint32_t wh[4], wl[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            wh[j] = pack_bf16x2(x[2 * j], x[2 * j + 1]);
            wl[j] = pack_bf16x2(x[2 * j] - bf16lo(wh[j]), x[2 * j + 1] - bf16hi(wh[j]));
        }
        *reinterpret_cast<uint4*>(s.omg_hi + sw128_chunk(row, c)) = make_uint4(wh[0], wh[1], wh[2], wh[3]);
        *reinterpret_cast<uint4*>(s.omg_lo + sw128_chunk(row, c)) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
    }
    for (int i = t; i < 4 * 2048 / 16; i += kCausalThreads)
        reinterpret_cast<uint4*>(s.zrow)[i] = make_uint4(0u, 0u, 0u, 0u);
    fill_ones_atom_f16(s.ones16, t, kCausalThreads);
    for (int i = t; i < kC * 8; i += kCausalThreads) {
        const int row = i >> 3, c = i & 7;
        if (nq == 1)   // feature rows 64..127 of the state update stay zero
            *reinterpret_cast<uint4*>(s.phk[1] + sw128_chunk(row, c)) = make_uint4(0u, 0u, 0u, 0u);
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = B.tmem_base;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA
        if (lane == 0) {
            int nqk = nchunks > 0 ? 1 : 0, nv = nqk;   // chunks whose loads were issued (chunk 0 at set-up)
            for (int c = 1; c < nchunks; ++c) {
                const int t0 = un.start + c * kC;
                if (c > 0 && !mbar_wait(&B.qk_empty, (c - 1) & 1)) { record_error(p.hdr, LA_DEVERR_WAIT_TIMEOUT); break; }
                mbar_arrive_expect_tx(&B.qk_full, 2 * kTile);
                tma_load_3d(s.tq, &map_q, 0, head, t0, &B.qk_full);
                tma_load_3d(s.tk, &map_k, 0, head, t0, &B.qk_full);
                ++nqk;
                if (c + 1 < nchunks) prefetch_v(c + 1);   // into L2 before it is needed
                if (c > 0 && !mbar_wait(&B.v_empty, (c - 1) & 1)) { record_error(p.hdr, LA_DEVERR_WAIT_TIMEOUT); break; }
                mbar_arrive_expect_tx(&B.v_full, kTile);
                load_v(c);
                ++nv;
            }
            // a consumer may have given up on a wait: the CTA must not exit while a load it issued
            // can still write shared memory (bounded; completed loads return at once)
            if (nqk > 0 && !mbar_wait(&B.qk_full, (nqk - 1) & 1, kDrainLimitNs)) record_error(p.hdr, LA_DEVERR_WAIT_TIMEOUT);
            if (nv > 0 && !mbar_wait(&B.v_full, (nv - 1) & 1, kDrainLimitNs)) record_error(p.hdr, LA_DEVERR_WAIT_TIMEOUT);
        }
    }
    else if (warp == 1) {
        // ------------------------------------------------------------ projection MMAs (elected lane issues)
        const uint64_t d_omg_hi = sdesc_sw128(smem_u32(s.omg_hi), 16, 1024);
        const uint64_t d_omg_lo = sdesc_sw128(smem_u32(s.omg_lo), 16, 1024);
        const uint64_t d_tq = sdesc_sw128(smem_u32(s.tq), 16, 1024);
        const uint64_t d_tk = sdesc_sw128(smem_u32(s.tk), 16, 1024);
        const uint32_t id_proj = idesc_bf16(128, 64, false, false);
        uint32_t jobs[2] = {0u, 0u};
        bool ok = true;
        // job of the given kind (1 max: the hi part of Q Omega'^T alone, for the rows' largest
        // exponents; 2 k, 3 q: hi + lo) for features 64 quarter .. into buffer b; waits until the
        // epilogue has read the buffer's previous job
        auto issue = [&](int b, int kind, int quarter) -> bool {
            if (!warp_wait(&B.p_empty[b], jobs[b] & 1u)) return false;
            ++jobs[b];
            tc_fence_after();
            const uint64_t dx = kind == 2 ? d_tk : d_tq;
            const uint32_t d = tb + kColCP + 64 * b, fo = 8192u * quarter;
#pragma unroll
            for (int k = 0; k < 4; ++k) mma_ss_w(d, sdesc_add(dx, 32 * k), sdesc_add(d_omg_hi, fo + 32 * k), id_proj, k > 0);
            if (kind != 1) {
#pragma unroll
                for (int k = 0; k < 4; ++k) mma_ss_w(d, sdesc_add(dx, 32 * k), sdesc_add(d_omg_lo, fo + 32 * k), id_proj, 1u);
            }
            mma_commit_w(&B.p_full[b]);
            return true;
        };
        const int nsteps = proj_steps(nq);
        for (int c = 0; c < nchunks && ok; ++c) {
            if (!(ok = warp_wait(&B.qk_full, c & 1))) break;
            for (int i = 0; favor && i < nsteps && ok; ++i) {
                const ProjStep st = proj_step(nq, i);
                for (int b = 0; b < 2 && ok; ++b)
                    if (st.kind[b] != 0) ok = issue(b, st.kind[b], st.quarter[b]);
            }
            if (ok) mma_commit_w(&B.qk_empty);   // every projection of this chunk issued
        }
        if (!ok && lane == 0) record_error(p.hdr, LA_DEVERR_WAIT_TIMEOUT);
    }
    else if (warp == 2) {
        // ------------------------------------------------------------ product MMAs (elected lane issues)
        const uint64_t d_phq = sdesc_sw128(smem_u32(s.phq[0]), 16, 1024);
        const uint64_t d_phk = sdesc_sw128(smem_u32(s.phk[0]), 16, 1024);
        const uint64_t d_sbf = sdesc_sw128(smem_u32(s.sbf[0]), kTile, 1024);                 // MN-major
        // [V|1]: V MN-major with the f16 ones atom as the second 64-column atom
        const uint64_t d_v1 = sdesc_sw128(smem_u32(s.tv), smem_u32(s.ones16) - smem_u32(s.tv), 1024);
        const uint64_t d_zrow = sdesc_sw128(smem_u32(s.zrow[0]), 16, 1024);
        const uint64_t d_upd_a = sdesc_sw128(smem_u32(s.phk[0]), kTile, 1024);              // MN-major
        const uint32_t id_den = idesc_f16(128, 16, false, false);
        const uint32_t id_scores = idesc_f16(128, 128, false, false);
        const uint32_t id_read = idesc_f16(128, 64, false, true);
        const uint32_t id_upd = idesc_f16(128, kNX, true, true);
        const uint32_t id_av = idesc_f16(128, kNX, false, true);
        bool ok = true;
        for (int c = 0; c < nchunks && ok; ++c) {
            bool v_ready = false;
            for (int q = 0; q < nq; ++q) {
                const int g = c * nq + q;
                if (!(ok = warp_wait(&B.phik_full[g & 1], (g >> 1) & 1))) break;
                if (q == 0) {   // O of chunk c-1 read out; the state of chunks < c copied (and rescaled)
                    if (!(ok = (c == 0 || warp_wait(&B.o_empty, (c - 1) & 1)) && warp_wait(&B.sbf_full, c & 1))) break;
                }
                tc_fence_after();
                if ((q & 1) || q == nq - 1) {   // phi(k) of the half complete: update now, ahead of the scores
                    // V as f16: FAVOR+ loaded so, else converted by the TE
                    if (!v_ready && !(ok = warp_wait(favor ? &B.v_full : &B.vh_full, c & 1))) break;
                    v_ready = true;
                    // [S|z] += phi(k)^T [V|1]: z from the ones column (column 64)
                    const uint32_t ds = tb + kColCS + kNX * (q >> 1);
#pragma unroll
                    for (int k = 0; k < kC / 16; ++k)
                        mma_ss_w(ds, sdesc_add(d_upd_a, 2048 * k), v_ones_desc(d_v1, k), id_upd, 1u);
                    mma_commit_w(&B.upd_done);
                }
                if (!(ok = warp_wait(&B.phiq_full[g & 1], (g >> 1) & 1))) break;
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mma_ss_w(tb + kColCA, sdesc_add(d_phq, kTile * (g & 1) + 32 * k), sdesc_add(d_phk, kTile * (q & 1) + 32 * k), id_scores,
                             (q > 0 || k > 0) ? 1u : 0u);
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mma_ss_w(tb + kColCX, sdesc_add(d_phq, kTile * (g & 1) + 32 * k), sdesc_add(d_sbf, 8192 * q + 2048 * k), id_read,
                             (q > 0 || k > 0) ? 1u : 0u);
                // denominator terms phi(q) . z (f16 and its remainder) into columns 64, 65 of O_cross
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mma_ss_w(tb + kColCX + 64, sdesc_add(d_phq, kTile * (g & 1) + 32 * k), sdesc_add(d_zrow, 2048 * q + 32 * k), id_den,
                             (q > 0 || k > 0) ? 1u : 0u);
                mma_commit_w(&B.phq_free[g & 1]);   // this phi(q) buffer may be rewritten
            }
            if (!ok) break;
            mma_commit_w(&B.a_full);
            if (!(ok = warp_wait(&B.ahl_full, c & 1))) break;
            tc_fence_after();
            // O_in = tril(A) [V|1]: scores as f16 in TMEM, keys 2c, 2c + 1 in column c
#pragma unroll
            for (int k = 0; k < kC / 16; ++k)
                mma_ts_w(tb + kColCI, tb + kColCA + 8 * k, v_ones_desc(d_v1, k), id_av, k > 0 ? 1u : 0u);
            mma_commit_w(&B.o_full);
            mma_commit_w(&B.v_empty);
        }
        if (!ok && lane == 0) record_error(p.hdr, LA_DEVERR_WAIT_TIMEOUT);
    }
    else if (warp == 3) {
    }
    else if (warp >= 4 && warp < 12) {
        // ------------------------------------------------------------ PE: phi(k), phi(q)
        const int tr = (t - 128) & 127;           // token row of the chunk = TMEM lane
        const int wl = (warp & 3) * 32;           // this warp's TMEM lane base
        const int half_cols = (warp - 4) >> 2;    // columns 32 half_cols .. + 31 of every job
        if (favor) {                              // both projection buffers start empty
            warp_arrive(&B.p_empty[0], false);
            warp_arrive(&B.p_empty[1], false);
        }
        bool ok = true;
        bool bigk = false, bigq = false;
        int R = 0;                                        // the keys' scale exponent of the chunk
        uint32_t njob[2] = {0u, 0u};                      // jobs read from each projection buffer
        // Projection job in buffer b (the buffer's next), columns 32 half_cols .. + 31.
        auto fetch = [&](int b, uint32_t (&v)[32]) -> bool {
            if (!warp_wait(&B.p_full[b], njob[b]++ & 1u)) return false;
            tc_fence_after();
            tmem_ld32(tmem_addr(tb, wl, kColCP + 64 * b + 32 * half_cols), v);
            return true;
        };
        // phi of one 32-column block of a job into dst (FAVOR+): 2^(p - cx), cx = inf past the end
        // (values at or beyond the f16 limit saturate to 65504 and are reported: the largest
        // exponent argument of the block decides that, one maximum per element).  Keys skip the
        // check: the chunk's scale R is at least the state kernel's exact e = ceil(max) - 15 over
        // the same projection, so p - R stays below 15 plus the two passes' rounding difference
        // for finite keys; the state kernel reports non-finite ones
        auto favor_phi = [&](const uint32_t (&v)[32], float cx, unsigned char* dst, bool& big,
                             bool check) -> float {
            uint32_t w[16];
            float mx = -INFINITY;
            uint64_t sum2 = f32x2_splat(0.f);             // two partial sums (even, odd columns)
            const uint64_t ncx = f32x2_splat(-cx);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const uint64_t x2 = f32x2_add(f32x2_of(v[2 * j], v[2 * j + 1]), ncx);
                const float xa = f32x2_lo(x2), xb = f32x2_hi(x2);
                if (check) mx = fmaxf(mx, fmaxf(xa, xb));
                const float a = ex2_approx(xa), b = ex2_approx(xb);
                sum2 = f32x2_add(sum2, f32x2_of(__float_as_uint(a), __float_as_uint(b)));
                w[j] = pack_f16x2_sat(a, b);
            }
            const float sum = f32x2_lo(sum2) + f32x2_hi(sum2);
            big |= mx >= 15.9997f;   // 2^15.9997 > 65503
            store_row32_bf16(dst, tr, 32 * half_cols, w);
            return sum;
        };
        // the MMAs that read a phi buffer last must be done before it is rewritten: for phi(q)
        // of global quarter g the products of quarter g - 2 (same buffer); for phi(k) the scores
        // of the previous quarter using that buffer and the state update of its half
        auto phq_writable = [&](int g) -> bool {
            return g < 2 || warp_wait(&B.phq_free[g & 1], ((g >> 1) - 1) & 1);
        };
        auto phk_writable = [&](int g) -> bool {
            const int gw = g - (nq >= 2 ? 2 : 1);
            const int uw = (gw / nq) * nhalves + ((gw % nq) >> 1);   // that update's index
            return gw < 0 || (warp_wait(&B.upd_done, uw & 1) && warp_wait(&B.phq_free[gw & 1], (gw >> 1) & 1));
        };
        if (favor) {
            int e_next = nchunks > 0 ? key_exp(0) : 0;   // the table is read a chunk ahead of its use
            if (g_force_wait_timeout != 0) {
                // test hook: a wait on a barrier that nothing arrives at runs out, as a lost
                // hand-off would; the other roles then give up on their own bounded waits
                const bool got = mbar_wait(&B.never, 0, kForcedWaitLimitNs);
                ok = !__any_sync(0xffffffffu, !got);
            }
            for (int c = 0; c < nchunks && ok; ++c) {
                const int slot = c & 1;
                const bool valid = tr < min(kC, un.end - (un.start + c * kC));
                R = next_key_scale(R, e_next, c == 0);
                e_next = c + 1 < nchunks ? key_exp(c + 1) : 0;
                // the TE has read the row scales and sums of chunk c - 2 (same slot)
                if (c >= 2 && !(ok = warp_wait(&B.srow_free[slot], ((c >> 1) - 1) & 1))) break;
                if (!(ok = warp_wait(&B.off_full[slot], (c >> 1) & 1))) break;
                const float cq = s.offq[slot][tr];
                const float ck = s.offk[slot][tr] + (float)R;
                const float cxk = valid ? ck : __int_as_float(0x7f800000);   // rows past the end: 2^-inf = 0
                // s_i from the row's largest exponent over all r features, taken from Q Omega'_hi^T
                // (the max jobs: the hi part alone, which errs by less than 2^-8 |Omega' x|): the
                // row's largest phi(q) 2^-s_i lies below 2^14 times 2 to that error, inside f16
                float m = -INFINITY;
                float cxq = 0.f;                             // cq + s_i once the maxima are in
                bool have_si = false;
                float qs = 0.f;                              // sum of |phi(q) 2^-s_i| this thread wrote
                const int nsteps = proj_steps(nq);
                for (int i = 0; i < nsteps && ok; ++i) {
                    const ProjStep st = proj_step(nq, i);
                    // both jobs of the step at once: each buffer takes its next job while this warp converts
                    uint32_t v[2][32];
                    if (!(ok = fetch(0, v[0]) && (st.kind[1] == 0 || fetch(1, v[1])))) break;
                    tmem_ld_wait();
                    warp_arrive(&B.p_empty[0], false);
                    if (st.kind[1] != 0) warp_arrive(&B.p_empty[1], false);
#pragma unroll
                    for (int b = 0; b < 2; ++b) {
                        const int kind = st.kind[b], q = st.quarter[b], g = c * nq + q;
                        if (kind == 1) {
#pragma unroll
                            for (int j = 0; j < 32; ++j) m = fmaxf(m, __uint_as_float(v[b][j]));
                        } else if (kind == 2) {
                            if (!(ok = phk_writable(g))) break;
                            favor_phi(v[b], cxk, s.phk[q & 1], bigk, false);
                            warp_arrive(&B.phik_full[g & 1], true);
                        } else if (kind == 3) {
                            if (!have_si) {
                                // the other warpgroup holds the other 32 columns of every job
                                s.rowmax[slot][half_cols][tr] = m;
                                __syncwarp();
                                if (lane == 0) mbar_arrive(&B.rx_full[slot]);
                                if (!(ok = warp_wait(&B.rx_full[slot], (c >> 1) & 1))) break;
                                const float mm = fmaxf(s.rowmax[slot][0][tr], s.rowmax[slot][1][tr]) - cq;
                                const int si = (valid && mm > -1e30f) ? (int)ceilf(mm) - 14 : 0;
                                if (half_cols == 0) s.srow[slot][tr] = si;   // for the TE: the row's factor
                                cxq = valid ? cq + (float)si : __int_as_float(0x7f800000);
                                have_si = true;
                            }
                            if (!(ok = phq_writable(g))) break;
                            qs += favor_phi(v[b], cxq, s.phq[g & 1], bigq, true);
                            // the row's sum of |phi(q)|, for the bound that scales its scores
                            if (q == nq - 1) s.qsum[slot][half_cols][tr] = qs;
                            warp_arrive(&B.phiq_full[g & 1], true);
                        }
                    }
                }
            }
        } else {
            for (int c = 0; c < nchunks && ok; ++c) {
                const int t0 = un.start + c * kC;
                const bool valid = tr < min(kC, un.end - t0);
                if (c >= 2 && !(ok = warp_wait(&B.srow_free[c & 1], ((c >> 1) - 1) & 1))) break;
                if (!(ok = warp_wait(&B.qk_full, c & 1))) break;
                float qs = 0.f;
                for (int q = 0; q < nq && ok; ++q) {
                    const int g = c * nq + q;
                    for (int kind = 0; kind < 2; ++kind) {   // 0: phi(k) of quarter q, 1: phi(q)
                        if (!(ok = kind == 0 ? phk_writable(g) : phq_writable(g))) break;
                        unsigned char* dst = kind == 0 ? s.phk[q & 1] : s.phq[g & 1];
                        float sum = 0.f;
                        if (p.map == LA_MAP_DPFP) {
                            (kind == 0 ? bigk : bigq) |= dpfp_phi_row32_f16(kind == 0 ? s.tk : s.tq, dst, tr, valid, q, half_cols, sum);
                        } else if (half_cols == 0) {
                            (kind == 0 ? bigk : bigq) |= elementwise_phi_row_f16(kind == 0 ? s.tk : s.tq, dst, tr, valid, p.map, sum);
                        }
                        if (kind == 1) qs += sum;
                        if (kind == 1 && q == nq - 1) s.qsum[c & 1][half_cols][tr] = qs;
                        warp_arrive(kind == 0 ? &B.phik_full[g & 1] : &B.phiq_full[g & 1], true);
                    }
                }
                if (ok) warp_arrive(&B.qk_empty, false);
            }
        }
        if (__any_sync(0xffffffffu, bigk) && lane == 0) record_range(p.hdr, kRangeK);
        if (__any_sync(0xffffffffu, bigq) && lane == 0) record_range(p.hdr, kRangeQ);
        if (!ok && lane == 0) record_error(p.hdr, LA_DEVERR_WAIT_TIMEOUT);
    } else if (warp >= 12) {
        // ------------------------------------------------------------ TE: chunk tail
        const int tr = t - 384;                   // query row / state feature = TMEM lane
        const int wl = (warp & 3) * 32;
        const int64_t E = (int64_t)r * 65;
        const float* src = p.prefix + ((int64_t)u * p.H + head) * E;
        const bool zero = tp.prefix_is_zero != 0;
        // the identity map has features of either sign: |S| has no bound from z, so its copy
        // takes the exact largest |entry| (one more pass over the state)
        const bool exact_copy = p.map == LA_MAP_IDENTITY;
        int uses = 0;                             // group_max4 uses (slot alternation)
        bool ok = true;
        // The state the unit starts from (true scale) into TMEM times 2^-R_0, and its f16
        // copy times 2^-(R_0 + g_0) for chunk 0's readout.  min holds the largest |entry|
        // of that entering state in the current TMEM scale (part of the copy's bound).
        int Rcur = favor && nchunks > 0 ? next_key_scale(0, key_exp(0), true) : 0;
        int gcur = 0;
        float min_ = 0.f;
        {
            const float fe = exp2i(-Rcur);
            float m = 0.f;
            for (int half = 0; half < nhalves; ++half) {
                const int feat = 128 * half + tr;
                if (zero || feat >= r) continue;
                for (int n = 0; n < 65; ++n) m = fmaxf(m, fabsf(src[(int64_t)feat * 65 + n] * fe));
            }
            ok = group_max4(m, s.tred, B.tx_full, uses++, 12);
            min_ = m;
            gcur = copy_exponent(m);
            const float fg = exp2i(-gcur);
            for (int half = 0; half < nhalves && ok; ++half) {   // the entering state: TMEM, f16 rows, z
                const int feat = 128 * half + tr;
                const bool have = !zero && feat < r;
                uint32_t w[32];
#pragma unroll
                for (int n0 = 0; n0 < kNX; n0 += 16) {
                    uint32_t x[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        x[j] = __float_as_uint((have && n0 + j < 65) ? src[(int64_t)feat * 65 + n0 + j] * fe : 0.f);
                    tmem_st16(tmem_addr(tb, wl, kColCS + kNX * half + n0), x);
                    if (n0 < 64) {
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            w[n0 / 2 + j] = pack_f16x2(__uint_as_float(x[2 * j]) * fg, __uint_as_float(x[2 * j + 1]) * fg);
                    } else if (feat < r) {
                        store_z_f16(s.zrow[feat >> 6], feat & 63, __uint_as_float(x[0]) * fg);
                    }
                }
                state_row_bf16(s.sbf[half], tr, w);
            }
            tmem_st_wait();
            if (ok) warp_arrive(&B.sbf_full, true);
        }
        // bound on |phi(k) 2^-R| of the chunk's keys: FAVOR+ 2^15 (the state kernel's chunk
        // maximum), element-wise maps the f16 limit
        const float kmax = favor ? 32768.f : 65504.f;
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);
        // FAVOR+: the exponent offsets of chunk c's query and key rows (one row per thread, slot
        // c & 1), computed while the TE waits for the chunk before; the PE starts chunk c on them
        auto post_offsets = [&](int c) -> bool {
            if (!warp_wait(&B.qk_full, c & 1)) return false;
            favor_offsets2(s.tq, s.tk, tr, r, s.offq[c & 1][tr], s.offk[c & 1][tr]);
            warp_arrive(&B.qk_empty, false);      // the tiles are no longer read by this warp
            warp_arrive(&B.off_full[c & 1], false);
            return true;
        };
        if (favor && nchunks > 0 && ok) ok = post_offsets(0);
        float vrun = 0.f;                         // largest |v| of the unit's chunks so far
        for (int c = 0; c < nchunks && ok; ++c) {
            const int t0 = un.start + c * kC;
            const bool valid = tr < min(kC, un.end - t0);
            const int e_next = favor && c + 1 < nchunks ? key_exp(c + 1) : 0;   // read well before its use
            // the state copy's bound takes the chunk's largest |v| (FAVOR+: from the state kernel's table)
            const float vm_c = favor ? fmaxf(fmaxf(vmx[kVmaxParts * c], vmx[kVmaxParts * c + 1]),
                                             fmaxf(vmx[kVmaxParts * c + 2], vmx[kVmaxParts * c + 3]))
                                     : 0.f;
            if (!favor) {
                // the chunk's V tile as f16, in place, rows 32 wq ..: the first state update of
                // the chunk waits for all four warps; each posts its rows' largest |v|
                if (!(ok = warp_wait(&B.v_full, c & 1))) break;
                float vm = v_tile_to_f16(s.tv, 32 * (warp & 3), 32, min(kC, un.end - t0), p.hdr, lane, 32);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) vm = fmaxf(vm, __shfl_xor_sync(0xffffffffu, vm, o));
                if (lane == 0) s.vt[c & 1][warp & 3] = vm;
                warp_arrive(&B.vh_full, true);
            }
            if (favor && c + 1 < nchunks && !(ok = post_offsets(c + 1))) break;
            if (!(ok = warp_wait(&B.a_full, c & 1))) break;
            tc_fence_after();
            // masked scores (key j <= query tr) as f16 times 2^-t_i in TMEM: A_ij <= (sum_f
            // |phi(q)_if|) max |phi(k)| bounds the row, so A 2^-t_i <= 2^14; keys 0..63 go to
            // columns 0..31 (read before written), keys 64..127 to columns 32..63
            const int wq = warp & 3;                  // rows 32 wq .. 32 wq + 31
            const int ti = copy_exponent((s.qsum[c & 1][0][tr] + s.qsum[c & 1][1][tr]) * kmax);
            const int si = favor ? s.srow[c & 1][tr] : 0;
            warp_arrive(&B.srow_free[c & 1], false);   // the PE may rewrite this slot (chunk c + 2)
            const float ft = exp2i(-ti);
            for (int part = 0; part < 2; ++part) {
                const int x0 = 2 * part, x1 = 2 * part + 1;
                uint32_t h0[16], h1[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) h0[j] = h1[j] = 0u;
                if (x0 <= wq) {
                    uint32_t v0[32], v1[32];
                    tmem_ld32(tmem_addr(tb, wl, kColCA + 64 * part), v0);
                    if (x1 <= wq) tmem_ld32(tmem_addr(tb, wl, kColCA + 64 * part + 32), v1);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int k0 = 32 * x0 + 2 * j;
                        const float a = (x0 < wq || k0 <= tr) ? __uint_as_float(v0[2 * j]) * ft : 0.f;
                        const float b = (x0 < wq || k0 + 1 <= tr) ? __uint_as_float(v0[2 * j + 1]) * ft : 0.f;
                        h0[j] = pack_f16x2(a, b);
                    }
                    if (x1 <= wq) {
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const int k0 = 32 * x1 + 2 * j;
                            const float a = (x1 < wq || k0 <= tr) ? __uint_as_float(v1[2 * j]) * ft : 0.f;
                            const float b = (x1 < wq || k0 + 1 <= tr) ? __uint_as_float(v1[2 * j + 1]) * ft : 0.f;
                            h1[j] = pack_f16x2(a, b);
                        }
                    }
                }
                tmem_st16(tmem_addr(tb, wl, kColCA + 32 * part), h0);
                tmem_st16(tmem_addr(tb, wl, kColCA + 32 * part + 16), h1);
            }
            tmem_st_wait();
            warp_arrive(&B.ahl_full, false);
            int gnext = gcur, Rnext = Rcur;
            if (c + 1 < nchunks) {
                // the state after this chunk, while A V runs: rescaled exactly (a power of two)
                // when the next chunk's key scale differs, then its f16 copy times 2^-g, g from
                // |S| <= max|S_in| + z max|v| (non-negative features) or the exact maximum
                Rnext = favor ? next_key_scale(Rcur, e_next, false) : 0;
                const float fe = exp2i(Rcur - Rnext);
                float m = 0.f;
                for (int half = 0; half < nhalves; ++half) {
                    const uint32_t col = kColCS + kNX * half;
                    const bool live = 128 * half + tr < r;
                    if (Rnext != Rcur || exact_copy) {
                        uint32_t a0[32], a1[32], zc;
                        tmem_ld32(tmem_addr(tb, wl, col), a0);
                        tmem_ld32(tmem_addr(tb, wl, col + 32), a1);
                        tmem_ld1(tmem_addr(tb, wl, col + 64), zc);
                        tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            a0[j] = __float_as_uint(__uint_as_float(a0[j]) * fe);
                            a1[j] = __float_as_uint(__uint_as_float(a1[j]) * fe);
                            if (exact_copy && live)
                                m = fmaxf(m, fmaxf(fabsf(__uint_as_float(a0[j])), fabsf(__uint_as_float(a1[j]))));
                        }
                        zc = __float_as_uint(__uint_as_float(zc) * fe);
                        if (live) m = fmaxf(m, fabsf(__uint_as_float(zc)));
                        if (Rnext != Rcur) {
                            tmem_st32(tmem_addr(tb, wl, col), a0);
                            tmem_st32(tmem_addr(tb, wl, col + 32), a1);
                            asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};"
                                         ::"r"(tmem_addr(tb, wl, col + 64)), "r"(zc) : "memory");
                        }
                    } else {
                        uint32_t zc;
                        tmem_ld1(tmem_addr(tb, wl, col + 64), zc);
                        tmem_ld_wait();
                        if (live) m = fmaxf(m, fabsf(__uint_as_float(zc)));
                    }
                }
                if (Rnext != Rcur) tmem_st_wait();
                if (!(ok = group_max4(m, s.tred, B.tx_full, uses++, 12))) break;
                min_ *= fe;
                // every TE warp posted its rows' largest |v| before the exchange above
                vrun = fmaxf(vrun, favor ? vm_c : fmaxf(fmaxf(s.vt[c & 1][0], s.vt[c & 1][1]),
                                                        fmaxf(s.vt[c & 1][2], s.vt[c & 1][3])));
                gnext = copy_exponent(exact_copy ? m : fmaxf(m, min_ + m * vrun));
                const float fg = exp2i(-gnext);
                for (int half = 0; half < nhalves; ++half) {
                    uint32_t a0[32], a1[32], zc;
                    const uint32_t col = kColCS + kNX * half;
                    tmem_ld32(tmem_addr(tb, wl, col), a0);
                    tmem_ld32(tmem_addr(tb, wl, col + 32), a1);
                    tmem_ld1(tmem_addr(tb, wl, col + 64), zc);
                    tmem_ld_wait();
                    uint32_t w[32];
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        w[j] = pack_f16x2(__uint_as_float(a0[2 * j]) * fg, __uint_as_float(a0[2 * j + 1]) * fg);
                        w[16 + j] = pack_f16x2(__uint_as_float(a1[2 * j]) * fg, __uint_as_float(a1[2 * j + 1]) * fg);
                    }
                    state_row_bf16(s.sbf[half], tr, w);
                    const int feat = 128 * half + tr;
                    if (feat < r) store_z_f16(s.zrow[feat >> 6], feat & 63, __uint_as_float(zc) * fg);
                }
                warp_arrive(&B.sbf_full, true);
            }
            if (!(ok = warp_wait(&B.o_full, c & 1))) break;
            tc_fence_after();
            // out = (2^t_i O_in + 2^g O_cross) times the row's multiplier (all in the scale
            // 2^(s_i + R_c)); the denominator first, since it sets the multiplier, then both
            // scales folded into it (exact powers of two), one packed multiply and one packed FMA
            // per pair of columns
            uint32_t di, dh, dl;
            tmem_ld1(tmem_addr(tb, wl, kColCI + 64), di);
            tmem_ld1(tmem_addr(tb, wl, kColCX + 64), dh);
            tmem_ld1(tmem_addr(tb, wl, kColCX + 65), dl);
            tmem_ld_wait();
            const float f2t = exp2i(ti), f2g = exp2i(gcur);
            const float den = fmaf(__uint_as_float(dh) + __uint_as_float(dl), f2g, __uint_as_float(di) * f2t);
            const int64_t orow = (int64_t)(t0 + tr) * p.H + head;
            const float mult = valid ? row_multiplier(den, si + Rcur, p, orow) : 0.f;
            const uint64_t ma = f32x2_splat(f2t * mult), mb = f32x2_splat(f2g * mult);
            uint4* dst = reinterpret_cast<uint4*>(out + orow * 64);
#pragma unroll
            for (int piece = 0; piece < 2; ++piece) {
                uint32_t a[32], x[32];
                tmem_ld32(tmem_addr(tb, wl, kColCI + 32 * piece), a);
                tmem_ld32(tmem_addr(tb, wl, kColCX + 32 * piece), x);
                tmem_ld_wait();
                // the next chunk may overwrite O_in, O_cross and the scores
                if (piece == 1) warp_arrive(&B.o_empty, false);
                if (valid) {
                    uint32_t w[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        w[j] = f32x2_to_bf16x2(f32x2_fma(f32x2_of(x[2 * j], x[2 * j + 1]), mb,
                                                         f32x2_mul(f32x2_of(a[2 * j], a[2 * j + 1]), ma)));
#pragma unroll
                    for (int qq = 0; qq < 4; ++qq)
                        dst[4 * piece + qq] = make_uint4(w[4 * qq], w[4 * qq + 1], w[4 * qq + 2], w[4 * qq + 3]);
                }
            }
            gcur = gnext;
            Rcur = Rnext;
        }
        if (!ok && lane == 0) record_error(p.hdr, LA_DEVERR_WAIT_TIMEOUT);
    }
    // ---------------------------------------------------------------- exit
    tc_fence_before();
    __syncthreads();
    if (warp == 1 || warp == 2) {   // all MMAs of this CTA finished before TMEM is freed (bounded)
        mma_commit_w(&B.drain[warp - 1]);
        if (!warp_wait(&B.drain[warp - 1], 0) && lane == 0) record_error(p.hdr, LA_DEVERR_WAIT_TIMEOUT);
    }
    __syncthreads();
    if (warp == 1) tmem_dealloc(tb, kTmemCols);
}

constexpr int kPrefetchAhead = 4;  // chunks of the streamed tiles requested into L2 ahead of the loads

// phi of one element for the element-wise maps.
__device__ __forceinline__ float phi_elementwise(float x, int map) {
    const float e = ex2_approx(x * kLog2e);   // unconditional, so that the choice is a select
    if (map == LA_MAP_ELU1) return x > 0.f ? x + 1.f : e;
    return x;
}

// ---------------------------------------------------------------------------
// Bidirectional output kernel (warp-specialised): out = phi(q)^T [S|z] / max(phi(q)^T z, eps)
// with [S|z] the whole-sequence state (in shared memory as f16 times 2^-g, z also as its
// f16 remainder)
// ---------------------------------------------------------------------------
// TMEM: two fp32 projection buffers [0, 256) (one 128-feature half each), two f16
// phi(q) buffers [256, 384), O = numerator | denominator [384, 464).
// Roles (544 threads):
//   warp 0 lane 0      TMA: the q tile of each chunk into two stages (and L2 prefetch)
//   warp 1             projection MMAs (elected lane; warp 1 owns the TMEM allocation):
//                      Q Omega'^T (hi, lo) plus one K step adding each query's
//                      exponent offset (FAVOR+), or Q itself (identity, element-wise maps)
//   warp 2             readout MMAs: O (+)= phi(q) [S|z]_f16 (one MMA per K step), A from TMEM
//   warps 3, 12 (NE)   per-query exponent offsets into the bias operand (FAVOR+)
//   warps 4..11 (PE)   phi(q) of each half: warpgroup w converts features 64w.. (lane = query)
//   warps 13..16 (OE)  out rows = O[0..63] / max(O[64], eps), after releasing O
constexpr int kBidirThreads = 544;
constexpr uint32_t kColBP = 0, kColBA = 256, kColBO = 384;

template <bool kFavor>
__global__ void __launch_bounds__(kBidirThreads, 1)
tc_bidir_out_kernel(const __grid_constant__ CUtensorMap map_q, const TcParams tp) {
    const FwdParams& p = tp.p;
    // one block per (unit, head), rank-major: all heads of the longest unit go out first
    const int rank = blockIdx.x / p.H, head = blockIdx.x - rank * p.H;
    if (rank >= p.hdr->n_units) return;
    const int u = p.order[rank];
    const Unit un = p.units[u];
    BidirSmem& s = smem_ref<BidirSmem>();
    BidirBars& B = s.b;
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int r = p.r;
    constexpr bool favor = kFavor;
    const int nhalves = (r + 127) / 128;
    const int nchunks = (un.end - un.start + kC - 1) / kC;

    if (t == 0) {
        prefetch_tensormap(&map_q);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&B.q_full[i], 1);
            mbar_init(&B.q_empty[i], 3);
            mbar_init(&B.cx_full[i], 2);
            mbar_init(&B.p_full[i], 1);
            mbar_init(&B.p_empty[i], 8);
            mbar_init(&B.a_full[i], 8);
            mbar_init(&B.a_empty[i], 1);
            mbar_init(&B.drain[i], 1);
        }
        mbar_init(&B.o_full, 1);
        mbar_init(&B.o_empty, 4);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&B.rx_full[i], 8);
            mbar_init(&B.srow_free[i], 4);
        }
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&B.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    if (favor) {
        stage_omega(s.omg_hi, s.omg_lo, p.omega, r);
        for (int i = t; i < (128 - r) * 8 && r < 128; i += kBidirThreads) {   // features r..127: zero
            const int row = r + (i >> 3), c = i & 7;
            *reinterpret_cast<uint4*>(s.omg_hi + sw128_chunk(row, c)) = make_uint4(0u, 0u, 0u, 0u);
            *reinterpret_cast<uint4*>(s.omg_lo + sw128_chunk(row, c)) = make_uint4(0u, 0u, 0u, 0u);
        }
    } else {
        // element-wise maps (r = d = 64): the projection is the identity, so that q
        // reaches tensor memory by the same exact MMA (features 64..127 zero)
        for (int i = t; i < 128 * 8; i += kBidirThreads) {
            const int row = i >> 3, c = i & 7;
            const bool one = row < r && (row >> 3) == c;
            const uint32_t w = one ? (0x3F80u << (16 * (row & 1))) : 0u;
            const int e = (row & 7) >> 1;
            *reinterpret_cast<uint4*>(s.omg_hi + sw128_chunk(row, c)) =
                make_uint4(e == 0 ? w : 0u, e == 1 ? w : 0u, e == 2 ? w : 0u, e == 3 ? w : 0u);
        }
    }
    for (int i = t; i < kC * 8; i += kBidirThreads) {   // bias columns start at zero; ones at 16 i, 16 i + 1
        const int row = i >> 3, c = i & 7;
        *reinterpret_cast<uint4*>(s.bias + sw128_chunk(row, c)) = make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(s.ones + sw128_chunk(row, c)) =
            make_uint4((c & 1) == 0 ? 0x3F803F80u : 0u, 0u, 0u, 0u);
    }
    // the whole-sequence state as one f16 readout operand, scaled by 2^-g so that its
    // largest entry lies in (2^13, 2^14] (z also as the f16 remainder, row 65)
    load_state_f16(s.sf16, p.prefix + ((int64_t)u * p.H + head) * (int64_t)r * 65, r, nhalves, s.red, &s.gexp);
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = B.tmem_base;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA
        if (lane == 0) {
            int nq = 0;   // chunks whose loads were issued
            for (int c = 0; c < nchunks; ++c) {
                const int st = c & 1, t0 = un.start + c * kC;
                for (int a = (c == 0 ? 0 : kPrefetchAhead); a <= kPrefetchAhead; ++a)
                    if (c + a < nchunks) tma_prefetch_3d(&map_q, 0, head, t0 + a * kC);
                if (c >= 2 && !mbar_wait(&B.q_empty[st], ((c >> 1) - 1) & 1)) {
                    record_error(p.hdr, LA_DEVERR_WAIT_TIMEOUT);
                    break;
                }
                mbar_arrive_expect_tx(&B.q_full[st], kTile);
                tma_load_3d(s.tq[st], &map_q, 0, head, t0, &B.q_full[st]);
                ++nq;
            }
            // no exit while an issued load can still write shared memory (bounded)
            for (int st = 0; st < 2; ++st) {
                const int last = nq - 1 - ((nq - 1 - st) & 1);   // last chunk issued into stage st
                if (last >= 0 && !mbar_wait(&B.q_full[st], (last >> 1) & 1, kDrainLimitNs))
                    record_error(p.hdr, LA_DEVERR_WAIT_TIMEOUT);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ projection MMAs (elected lane issues)
        const uint64_t d_omg_hi = sdesc_sw128(smem_u32(s.omg_hi), 16, 1024);
        const uint64_t d_omg_lo = sdesc_sw128(smem_u32(s.omg_lo), 16, 1024);
        const uint64_t d_bias = sdesc_sw128(smem_u32(s.bias), 16, 1024);
        const uint64_t d_ones = sdesc_sw128(smem_u32(s.ones), 16, 1024);
        const uint32_t id_proj = idesc_bf16(128, min(r, 128), false, false);   // M = queries, N = features
        bool ok = true;
        for (int c = 0; c < nchunks && ok; ++c) {
            const int st = c & 1;
            if (!(ok = warp_wait(&B.cx_full[st], (c >> 1) & 1))) break;   // tile and offsets staged
            const uint64_t d_tq = sdesc_sw128(smem_u32(s.tq[st]), 16, 1024);
            for (int h = 0; h < nhalves && ok; ++h) {
                const int j = c * nhalves + h, b = j & 1;
                if (j >= 2 && !(ok = warp_wait(&B.p_empty[b], ((j >> 1) - 1) & 1))) break;
                tc_fence_after();
                const uint32_t d = tb + kColBP + 128 * b, fo = 16384u * h;
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mma_ss_w(d, sdesc_add(d_tq, 32 * k), sdesc_add(d_omg_hi, fo + 32 * k), id_proj, k > 0);
                if (favor) {
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mma_ss_w(d, sdesc_add(d_tq, 32 * k), sdesc_add(d_omg_lo, fo + 32 * k), id_proj, 1u);
                    mma_ss_w(d, sdesc_add(d_bias, 32 * st), sdesc_add(d_ones, 32 * st), id_proj, 1u);
                }
                mma_commit_w(&B.p_full[b]);
            }
            if (ok) mma_commit_w(&B.q_empty[st]);
        }
        if (!ok && lane == 0) record_error(p.hdr, LA_DEVERR_WAIT_TIMEOUT);
    } else if (warp == 2) {
        // ------------------------------------------------------------ readout MMAs (elected lane issues)
        const uint32_t id_read = idesc_f16(128, kNX, false, false);   // A f16 from TMEM, B f16 K-major
        bool ok = true;
        for (int c = 0; c < nchunks && ok; ++c) {
            for (int h = 0; h < nhalves && ok; ++h) {
                const int j = c * nhalves + h, b = j & 1;
                if (!(ok = warp_wait(&B.a_full[b], (j >> 1) & 1))) break;
                if (h == 0 && c > 0 && !(ok = warp_wait(&B.o_empty, (c - 1) & 1))) break;   // O read out
                tc_fence_after();
                const uint32_t a0 = tb + kColBA + 64 * b;
                const int nk = min(r - 128 * h, 128) / 16;
                for (int k = 0; k < nk; ++k) {
                    const int blk = 2 * h + (k >> 2);
                    mma_ts_w(tb + kColBO, a0 + 8 * k, sdesc_sw128(smem_u32(s.sf16[blk]) + 32u * (k & 3), 16, 1024),
                             id_read, (h > 0 || k > 0) ? 1u : 0u);
                }
                mma_commit_w(&B.a_empty[b]);
            }
            if (ok) mma_commit_w(&B.o_full);
        }
        if (!ok && lane == 0) record_error(p.hdr, LA_DEVERR_WAIT_TIMEOUT);
    } else if (warp >= 4 && warp < 12) {
        // ------------------------------------------------------------ PE: phi(q)
        // per chunk: the exact maximum of each query row over all its features (both
        // halves, both warpgroups), then phi(q) 2^-s_i as f16 (largest in (2^14, 2^15]);
        // the factor 2^-s_i is common to the row's numerator and denominator
        const int wg = (warp - 4) >> 2;           // features 64 wg .. of every half
        const int wl = (warp & 3) * 32;           // TMEM lane base: queries wl ..
        const int row = wl + lane;
        bool ok = true;
        for (int c = 0; c < nchunks && ok; ++c) {
            float m = -INFINITY;
            for (int h = 0; h < nhalves && ok; ++h) {
                const int j = c * nhalves + h, b = j & 1;
                if (!(ok = warp_wait(&B.p_full[b], (j >> 1) & 1))) break;
                tc_fence_after();
                if (128 * h + 64 * wg >= r) continue;   // these 64 features do not exist
#pragma unroll
                for (int piece = 0; piece < 2; ++piece) {
                    uint32_t v[32];
                    tmem_ld32(tmem_addr(tb, wl, kColBP + 128 * b + 64 * wg + 32 * piece), v);
                    tmem_ld_wait();
                    if (favor) {
                        m = fmaxf(m, max_tree32(v));
                    } else {
#pragma unroll
                        for (int e = 0; e < 32; ++e) m = fmaxf(m, fabsf(phi_elementwise(__uint_as_float(v[e]), p.map)));
                    }
                }
            }
            if (!ok) break;
            // the other warpgroup holds the rest of the row
            const int slot = c & 1;
            s.rowmax[slot][wg][row] = m;
            __syncwarp();
            if (lane == 0) mbar_arrive(&B.rx_full[slot]);
            if (!(ok = warp_wait(&B.rx_full[slot], (c >> 1) & 1))) break;
            m = fmaxf(s.rowmax[slot][0][row], s.rowmax[slot][1][row]);
            // FAVOR+: m is the row's largest exponent; element-wise maps: its largest |phi|
            int sx = 0;
            if (favor) sx = m > -1e30f ? (int)ceilf(m) - 15 : 0;
            else sx = m > 0.f ? (int)ceilf(__log2f(m)) - 15 : 0;
            if (wg == 0) {   // for the OE (denominator clamp, unnormalised output)
                if (c >= 2 && !(ok = warp_wait(&B.srow_free[slot], ((c >> 1) - 1) & 1))) break;
                s.srow[slot][row] = sx;
            }
            const float fs = (float)sx, mul = exp2i(-sx);
            for (int h = 0; h < nhalves && ok; ++h) {
                const int j = c * nhalves + h, b = j & 1;
                const bool live = 128 * h + 64 * wg < r;   // these 64 features exist
                uint32_t v0[32], v1[32], w[32];
                tmem_ld32(tmem_addr(tb, wl, kColBP + 128 * b + 64 * wg), v0);
                tmem_ld32(tmem_addr(tb, wl, kColBP + 128 * b + 64 * wg + 32), v1);
                tmem_ld_wait();
                warp_arrive(&B.p_empty[b], false);
                // the readout that read this phi buffer last must be done
                if (j >= 2 && !(ok = warp_wait(&B.a_empty[b], ((j >> 1) - 1) & 1))) break;
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const float a0 = __uint_as_float(v0[2 * e]), a1 = __uint_as_float(v0[2 * e + 1]);
                    w[e] = live ? (favor ? pack_f16x2(ex2_approx(a0 - fs), ex2_approx(a1 - fs))
                                         : pack_f16x2(phi_elementwise(a0, p.map) * mul, phi_elementwise(a1, p.map) * mul))
                                : 0u;
                }
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const float a0 = __uint_as_float(v1[2 * e]), a1 = __uint_as_float(v1[2 * e + 1]);
                    w[16 + e] = live ? (favor ? pack_f16x2(ex2_approx(a0 - fs), ex2_approx(a1 - fs))
                                              : pack_f16x2(phi_elementwise(a0, p.map) * mul, phi_elementwise(a1, p.map) * mul))
                                     : 0u;
                }
                tmem_st32(tmem_addr(tb, wl, kColBA + 64 * b + 32 * wg), w);
                tmem_st_wait();
                warp_arrive(&B.a_full[b], false);
            }
        }
        if (!ok && lane == 0) record_error(p.hdr, LA_DEVERR_WAIT_TIMEOUT);
    } else if (warp == 3 || warp == 12) {
        // ------------------------------------------------------------ NE: exponent offsets (warps 3, 12)
        const int tok0 = warp == 3 ? 0 : 64;
        bool ok = true;
        for (int c = 0; c < nchunks && ok; ++c) {
            const int st = c & 1;
            if (!(ok = warp_wait(&B.q_full[st], (c >> 1) & 1))) break;
            if (favor) {
                float nx[2];
                row_sq_norm2(s.tq[st], tok0 + lane, tok0 + lane + 32, nx[0], nx[1]);
#pragma unroll
                for (int x = 0; x < 2; ++x) {
                    const int tok = tok0 + lane + 32 * x;
                    const float o = -(nx[x] * (0.5f * kLog2e) + 0.5f * __log2f((float)r));
                    const uint32_t hl = pack_bf16x2(o, 0.f);
                    *reinterpret_cast<uint32_t*>(s.bias + sw128_off(tok, 16 * st)) = pack_bf16x2(o, o - bf16lo(hl));
                }
            }
            warp_arrive(&B.cx_full[st], true);
            warp_arrive(&B.q_empty[st], false);   // this warp no longer reads the tile
        }
        if (!ok && lane == 0) record_error(p.hdr, LA_DEVERR_WAIT_TIMEOUT);
    } else {
        // ------------------------------------------------------------ OE: output rows (warps 13..16)
        const int wl = (warp & 3) * 32;
        const int tr = wl + lane;                 // query row = TMEM lane
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);
        const int g = s.gexp;
        bool ok = true;
        for (int c = 0; c < nchunks && ok; ++c) {
            const int t0 = un.start + c * kC;
            if (!(ok = warp_wait(&B.o_full, c & 1))) break;
            tc_fence_after();
            uint32_t o0[32], o1[32], dh, dl;
            tmem_ld32(tmem_addr(tb, wl, kColBO), o0);
            tmem_ld32(tmem_addr(tb, wl, kColBO + 32), o1);
            tmem_ld1(tmem_addr(tb, wl, kColBO + 64), dh);   // phi(q) . z (f16 part)
            tmem_ld1(tmem_addr(tb, wl, kColBO + 65), dl);   // phi(q) . z (f16 remainder)
            tmem_ld_wait();
            const int sx = s.srow[c & 1][tr];
            warp_arrive(&B.o_empty, false);     // the next chunk may overwrite O
            warp_arrive(&B.srow_free[c & 1], false);
            if (tr < min(kC, un.end - t0)) {
                const int64_t orow = (int64_t)(t0 + tr) * p.H + head;
                // O and the denominator are the true values times 2^-(s_i + g)
                const float den = __uint_as_float(dh) + __uint_as_float(dl);
                store_output_row_f(o0, o1, row_multiplier(den, sx + g, p, orow), out + orow * 64);
            }
        }
        if (!ok && lane == 0) record_error(p.hdr, LA_DEVERR_WAIT_TIMEOUT);
    }
    // ---------------------------------------------------------------- exit
    tc_fence_before();
    __syncthreads();
    if (warp == 1 || warp == 2) {   // every MMA of both issuers finished (bounded)
        mma_commit_w(&B.drain[warp - 1]);
        if (!warp_wait(&B.drain[warp - 1], 0) && lane == 0) record_error(p.hdr, LA_DEVERR_WAIT_TIMEOUT);
    }
    __syncthreads();
    if (warp == 1) tmem_dealloc(tb, kTmemCols);
}

// ---------------------------------------------------------------------------
// Segment-state kernel (warp-specialised): [S|z] = sum over the unit of phi(k) [v | 1]^T
// ---------------------------------------------------------------------------
// The projection is computed transposed, P^T = Omega' K^T (TMEM lanes = features,
// columns = tokens); one more K step adds each token's exponent offset -(log2(e)
// |k|^2 / 2 + log2(sqrt r)) as bf16 hi + lo, so that phi = 2^P^T element-wise.
//
// fp16 features with exact power-of-two scales: the PE warps reduce the largest
// exponent, take e = ceil(max) - 15 and write phi(k)^T 2^-R as f16 (11 significant
// bits) back into the buffer it came from, R following e with hysteresis
// (next_key_scale).  For r = 256 the scale is per feature (its own maximum over
// the chunk's 128 tokens, the two warps holding its token halves exchanging
// theirs); for r <= 128 and the element-wise maps one scale per chunk (the
// maximum over all eight warps).  The state is accumulated in TMEM in the latest
// scale: when it changes, the PE rescales the state rows exactly (a power of two)
// before the chunk's update, and the state leaves in true scale.  V is converted to f16 in place by the NE warps (values beyond
// 65504 are clamped and reported as LA_DEVERR_RANGE); [S|z] += phi(k)^T [V|1]
// takes its A operand from TMEM and its B operand from V with an f16 ones tile as
// the second 64-column atom, so z (column 64) comes from the same features as S.
// The chunk's key exponent (the larger of the two halves) is recorded in
// p.kscale for the causal output kernel.
// TMEM: [S|z] [0, 160) (80 columns per 128-feature half), two fp32 projection
// buffers [160, 416).
// Roles (480 threads):
//   warp 0 lane 0     TMA: k and v tiles of each chunk into three stages (and L2 prefetch)
//   warp 1            projection MMAs (one elected lane; warp 1 owns the TMEM
//                     allocation): (c, h) into buffer (c nhalves + h) & 1 once the
//                     update has read that buffer's previous phi(k)^T
//   warp 2            state-update MMAs: (c, h) once the PE has written phi(k)^T
//   warps 3, 12..14   (NE) the exponent offset of every token of a stage (FAVOR+),
//                     into the bias operand of the projection, and the stage's V as
//                     f16 (32 tokens each, on all four SM sub-partitions); with the
//                     causal FAVOR+ output kernel to follow, the f16 rows also go to
//                     the workspace with their largest |v|
//   warps 4..11 (PE)  two warpgroups; warpgroup w converts tokens 64w..64w+63 of
//                     every half (lane = feature)
constexpr int kStateThreads = 480;
// Largest key exponent the chunk scales handle (e = ceil(max) - 15 and the rescales stay far
// inside int and the float exponent); beyond it the state kernel reports LA_DEVERR_RANGE.
constexpr float kKeyExpLimit = 1.0e9f;
constexpr int kStateNE = 4;        // NE warps: 3, 12, 13, 14
constexpr uint32_t kColSS = 0;     // [S|z], 80 columns per half
constexpr uint32_t kColPS = 160;   // two 128-column projection buffers (exponent, then phi(k)^T in place)

// Maximum over the eight warps warp0 .. warp0 + 7 for use j: each warp posts its
// maximum and arrives on bar[j & 1] (count 8), then waits for the others (bounded:
// false if the wait ran out).  Two slots: a warp cannot post use j + 2 before every
// warp has arrived for use j + 1, i.e. finished reading use j.
__device__ __forceinline__ bool group_max8(float& m, float (*red)[8], uint64_t* bar, int j, int warp0) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const int slot = j & 1;
    if ((threadIdx.x & 31) == 0) red[slot][(threadIdx.x >> 5) - warp0] = m;
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&bar[slot]);
    if (!warp_wait(&bar[slot], (j >> 1) & 1)) return false;
    float r = red[slot][0];
#pragma unroll
    for (int i = 1; i < 8; ++i) r = fmaxf(r, red[slot][i]);
    m = r;
    return true;
}

// kFavor: FAVOR+ (projection by Omega' hi + lo and the offset step), else an
// element-wise map of k (identity projection); one instantiation per kind.
template <bool kFavor>
__global__ void __launch_bounds__(kStateThreads, 1)
tc_state_kernel(const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
                const TcParams tp) {
    const FwdParams& p = tp.p;
    // one block per (unit, head), rank-major as in the output kernels: all heads of the
    // longest unit first, so that blocks past the first wave are those of short units
    const int rank = blockIdx.x / p.H, head = blockIdx.x - rank * p.H;
    if (rank >= p.hdr->n_units) return;
    const int u = p.order[rank];
    const Unit un = p.units[u];
    // causal: no later segment adds the last segment of a sequence to its prefix;
    // only a final state or the key exponents of the output kernel need it
    const bool last = p.causal && u + 1 == p.seq_first[un.seq + 1];
    if (last && !p.keep_last && p.kscale == nullptr) return;
    StateSmem& s = smem_ref<StateSmem>();
    StateBars& B = s.b;
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int r = p.r;
    constexpr bool favor = kFavor;
    const int nhalves = (r + 127) / 128;
    const int nchunks = (un.end - un.start + kC - 1) / kC;
    // r = 256 FAVOR+: one warpgroup per feature half, a scale per feature (see the PE)
    const bool per_feature = favor && nhalves == 2;

    if (t == 0) {
        prefetch_tensormap(&map_k);
        prefetch_tensormap(&map_v);
        for (int i = 0; i < 4; ++i) s.kmx[i] = INT_MIN;
        for (int i = 0; i < kStateStages; ++i) {
            mbar_init(&B.k_full[i], 1);
            mbar_init(&B.k_empty[i], 1 + kStateNE);   // projection commit + the NE warps
            mbar_init(&B.v_full[i], 1);
            // update commit, and with the f16 copy of V going out the two NE warps once it has read the stage
            mbar_init(&B.v_empty[i], p.v16 != nullptr ? 1 + kStateNE : 1);
            mbar_init(&B.cx_full[i], kStateNE);
            mbar_init(&B.vh_full[i], kStateNE);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&B.p_full[i], 1);
            mbar_init(&B.a_full[i], 8);
            mbar_init(&B.a_empty[i], 1);
            mbar_init(&B.red_full[i], 8);
        }
        for (int i = 0; i < 4; ++i) {
            mbar_init(&B.pmx_full[i][0], 2);
            mbar_init(&B.pmx_full[i][1], 2);
        }
        mbar_init(&B.drain[0], 1);
        mbar_init(&B.drain[1], 1);
        fence_mbar_init();
        // the first stages' k / v tiles go out before the set-up below (nothing in it
        // touches them), so that their DRAM latency overlaps the staging of Omega
        for (int c = 0; c < nchunks && c < kStateStages; ++c) {
            const int t0 = un.start + c * kC;
            for (int a = (c == 0 ? 0 : kPrefetchAhead); a <= kPrefetchAhead; ++a)
                if (c + a < nchunks) {
                    tma_prefetch_3d(&map_k, 0, head, t0 + a * kC);
                    tma_prefetch_3d(&map_v, 0, head, t0 + a * kC);
                }
            mbar_arrive_expect_tx(&B.k_full[c], kTile);
            tma_load_3d(s.tk[c], &map_k, 0, head, t0, &B.k_full[c]);
            mbar_arrive_expect_tx(&B.v_full[c], kTile);
            tma_load_3d(s.tv[c], &map_v, 0, head, t0, &B.v_full[c]);
        }
    }
    if (warp == 1) {
        tmem_alloc(&B.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    if (favor) {
        stage_omega(s.omg_hi, s.omg_lo, p.omega, r);
        for (int i = t; i < (128 - r) * 8 && r < 128; i += kStateThreads) {   // features r..127 of half 0: zero
            const int row = r + (i >> 3), c = i & 7;
            *reinterpret_cast<uint4*>(s.omg_hi + sw128_chunk(row, c)) = make_uint4(0u, 0u, 0u, 0u);
            *reinterpret_cast<uint4*>(s.omg_lo + sw128_chunk(row, c)) = make_uint4(0u, 0u, 0u, 0u);
        }
    } else {
        // element-wise maps (r = d = 64): the "projection" is the identity, so that
        // k^T reaches tensor memory by the same exact MMA (rows 64..127 zero)
        for (int i = t; i < 128 * 8; i += kStateThreads) {
            const int row = i >> 3, c = i & 7;
            const bool one = row < r && (row >> 3) == c;
            const uint32_t w = one ? (0x3F80u << (16 * (row & 1))) : 0u;
            const int e = (row & 7) >> 1;   // 32-bit word of the chunk holding column row
            *reinterpret_cast<uint4*>(s.omg_hi + sw128_chunk(row, c)) =
                make_uint4(e == 0 ? w : 0u, e == 1 ? w : 0u, e == 2 ? w : 0u, e == 3 ? w : 0u);
        }
    }
    for (int i = t; i < kC * 8; i += kStateThreads) {   // bias columns start at zero; ones at 16 i, 16 i + 1
        const int row = i >> 3, c = i & 7;
        *reinterpret_cast<uint4*>(s.bias + sw128_chunk(row, c)) = make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(s.ones + sw128_chunk(row, c)) =
            make_uint4((c & 1) == 0 ? 0x3F803F80u : 0u, 0u, 0u, 0u);
    }
    fill_ones_atom_f16(s.ones16, t, kStateThreads);
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = B.tmem_base;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA
        if (lane == 0) {
            int nk = min(nchunks, kStateStages), nv = nk;   // chunks whose loads were issued
            for (int c = kStateStages; c < nchunks; ++c) {   // chunks 0 .. kStateStages - 1: issued at set-up
                const int st = c % kStateStages, ph = ((c / kStateStages) - 1) & 1, t0 = un.start + c * kC;
                // into L2 ahead of the stages: the loads below then wait on L2, not DRAM
                for (int a = (c == 0 ? 0 : kPrefetchAhead); a <= kPrefetchAhead; ++a)
                    if (c + a < nchunks) {
                        tma_prefetch_3d(&map_k, 0, head, t0 + a * kC);
                        tma_prefetch_3d(&map_v, 0, head, t0 + a * kC);
                    }
                if (c >= kStateStages && !mbar_wait(&B.k_empty[st], ph)) {
                    record_error(p.hdr, LA_DEVERR_WAIT_TIMEOUT);
                    break;
                }
                mbar_arrive_expect_tx(&B.k_full[st], kTile);
                tma_load_3d(s.tk[st], &map_k, 0, head, t0, &B.k_full[st]);
                ++nk;
                if (c >= kStateStages && !mbar_wait(&B.v_empty[st], ph)) {
                    record_error(p.hdr, LA_DEVERR_WAIT_TIMEOUT);
                    break;
                }
                mbar_arrive_expect_tx(&B.v_full[st], kTile);
                tma_load_3d(s.tv[st], &map_v, 0, head, t0, &B.v_full[st]);
                ++nv;
            }
            // no exit while an issued load can still write shared memory (bounded)
            for (int st = 0; st < kStateStages; ++st) {
                const int lk = nk - 1 - ((nk - 1 - st) % kStateStages + kStateStages) % kStateStages;
                const int lv = nv - 1 - ((nv - 1 - st) % kStateStages + kStateStages) % kStateStages;
                if (lk >= 0 && !mbar_wait(&B.k_full[st], (lk / kStateStages) & 1, kDrainLimitNs))
                    record_error(p.hdr, LA_DEVERR_WAIT_TIMEOUT);
                if (lv >= 0 && !mbar_wait(&B.v_full[st], (lv / kStateStages) & 1, kDrainLimitNs))
                    record_error(p.hdr, LA_DEVERR_WAIT_TIMEOUT);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ projection MMAs (elected lane issues)
        const uint64_t d_omg_hi = sdesc_sw128(smem_u32(s.omg_hi), 16, 1024);
        const uint64_t d_omg_lo = sdesc_sw128(smem_u32(s.omg_lo), 16, 1024);
        const uint64_t d_bias = sdesc_sw128(smem_u32(s.bias), 16, 1024);
        const uint64_t d_ones = sdesc_sw128(smem_u32(s.ones), 16, 1024);
        const uint32_t id_proj = idesc_bf16(128, kC, false, false);   // M = features, N = tokens
        bool ok = true;
        for (int c = 0; c < nchunks && ok; ++c) {
            const int st = c % kStateStages;
            if (!(ok = warp_wait(&B.cx_full[st], (c / kStateStages) & 1))) break;   // tile and offsets staged
            const uint64_t d_tk = sdesc_sw128(smem_u32(s.tk[st]), 16, 1024);
            for (int h = 0; h < nhalves && ok; ++h) {
                // exponent of phi(k)^T, features 128h..: Omega' K^T, then one K step of
                // ones x (-offset hi, -offset lo) per token
                const int j = c * nhalves + h, b = j & 1;
                if (j >= 2 && !(ok = warp_wait(&B.a_empty[b], ((j >> 1) - 1) & 1))) break;
                tc_fence_after();
                const uint32_t d = tb + kColPS + 128 * b, fo = 16384u * h;
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mma_ss_w(d, sdesc_add(d_omg_hi, fo + 32 * k), sdesc_add(d_tk, 32 * k), id_proj, k > 0);
                if (favor) {
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mma_ss_w(d, sdesc_add(d_omg_lo, fo + 32 * k), sdesc_add(d_tk, 32 * k), id_proj, 1u);
                    mma_ss_w(d, sdesc_add(d_ones, 32 * st), sdesc_add(d_bias, 32 * st), id_proj, 1u);
                }
                mma_commit_w(&B.p_full[b]);
            }
            if (ok) mma_commit_w(&B.k_empty[st]);
        }
        if (!ok && lane == 0) record_error(p.hdr, LA_DEVERR_WAIT_TIMEOUT);
    } else if (warp == 2) {
        // ------------------------------------------------------------ state-update MMAs (elected lane issues)
        const uint32_t id_upd = idesc_f16(128, kNX, false, true);    // A f16 from TMEM, B = [V|1] f16 MN-major, N = 80
        bool ok = true;
        for (int c = 0; c < nchunks && ok; ++c) {
            const int st = c % kStateStages;
            if (!(ok = warp_wait(&B.vh_full[st], (c / kStateStages) & 1))) break;   // V as f16
            const uint64_t d_v = sdesc_sw128(smem_u32(s.tv[st]), smem_u32(s.ones16) - smem_u32(s.tv[st]), 1024);
            for (int h = 0; h < nhalves && ok; ++h) {
                const int j = c * nhalves + h, b = j & 1;
                if (!(ok = warp_wait(&B.a_full[b], (j >> 1) & 1))) break;
                tc_fence_after();
                if (per_feature && h == 1 && lane == 0 && p.kscale != nullptr) {
                    // both halves' features have posted their exponents: the chunk's key scale
                    p.kscale[((int64_t)u * p.H + head) * p.Lc + c] = s.kmx[c & 3];
                    s.kmx[c & 3] = INT_MIN;
                }
                // tokens 16k.. of phi(k)^T: columns 64 (k / 4) + 8 (k % 4) of the buffer
                const uint32_t a0 = tb + kColPS + 128 * b;
#pragma unroll
                for (int k = 0; k < kC / 16; ++k)
                    mma_ts_w(tb + kColSS + kNX * h, a0 + 64 * (k >> 2) + 8 * (k & 3), v_ones_desc(d_v, k), id_upd,
                             (c > 0 || k > 0) ? 1u : 0u);
                mma_commit_w(&B.a_empty[b]);
            }
            if (ok) mma_commit_w(&B.v_empty[st]);
        }
        if (!ok && lane == 0) record_error(p.hdr, LA_DEVERR_WAIT_TIMEOUT);
    } else if (warp >= 4 && warp < 12) {
        // ------------------------------------------------------------ PE: phi(k)^T
        const int wg = (warp - 4) >> 2;
        const int wl = (warp & 3) * 32;           // TMEM lane base: features wl .. wl + 31 of a half
        const int f = wl + lane;
        bool ok = true;
        if (per_feature) {
            // r = 256: both warpgroups convert every job (c, h) in turn, warpgroup wg tokens
            // 64 wg .. 64 wg + 63 (lane = feature 128 h + f), so that one half's conversion has
            // all eight warps while the other half's update and next projection run on the
            // tensor pipe.  phi(k)_f 2^-R_f with R_f from the feature's own largest exponent
            // over the chunk's 128 tokens (hysteresis: next_key_scale): the two warps holding a
            // feature's token halves (warps 4 + q and 8 + q) exchange their maxima
            const int q4 = warp & 3;
            int Rh[2] = {0, 0};
            // an exponent beyond the integer scale arithmetic is the one way phi(k) 2^-R can leave
            // the f16 range (the output kernel relies on that and does not check keys): reported
            // once, after the unit
            bool kbig = false;
            for (int c = 0; c < nchunks && ok; ++c) {
                for (int h = 0; h < 2 && ok; ++h) {
                    const int b = h;                      // job 2c + h uses buffer (2c + h) & 1
                    const bool live = 128 * h + f < r;
                    if (!(ok = warp_wait(&B.p_full[b], c & 1))) break;
                    tc_fence_after();
                    const uint32_t col = kColPS + 128 * b + 64 * wg;
                    uint32_t v0[32], v1[32];
                    tmem_ld32(tmem_addr(tb, wl, col), v0);
                    tmem_ld32(tmem_addr(tb, wl, col + 32), v1);
                    tmem_ld_wait();
                    float m = -INFINITY;
#pragma unroll
                    for (int e = 0; e < 32; ++e) m = fmaxf(m, fmaxf(__uint_as_float(v0[e]), __uint_as_float(v1[e])));
                    // slot h: a warp posts the next chunk's maximum of this half only after its
                    // wait for half h ^ 1, i.e. after the partner has read this one
                    s.pmx[h][wg][32 * q4 + lane] = m;
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&B.pmx_full[q4][h]);
                    if (!(ok = warp_wait(&B.pmx_full[q4][h], c & 1))) break;
                    m = fmaxf(m, s.pmx[h][wg ^ 1][32 * q4 + lane]);
                    kbig |= live && !(m <= kKeyExpLimit);
                    const int R = Rh[h];
                    const int e = (live && m > -1e30f) ? (int)ceilf(m) - 15 : R;
                    const int Rn = next_key_scale(R, e, c == 0);
                    if (live) atomicMax(&s.kmx[c & 3], e);
                    // tcgen05.ld / st are warp-collective (.sync.aligned): the whole warp takes the
                    // branch when any of its features changes scale (the others multiply by exactly 1)
                    if (c > 0 && __any_sync(0xffffffffu, Rn != R)) {
                        // the previous update of this half is complete (this job's projection waited
                        // for it): the feature's state row times 2^(R - Rn), exactly; warpgroup 0
                        // takes columns 0..31 and z, warpgroup 1 columns 32..63
                        const float fct = exp2i(R - Rn);
                        const uint32_t sc = kColSS + kNX * h;
                        uint32_t w[32], zc = 0u;
                        tmem_ld32(tmem_addr(tb, wl, sc + 32 * wg), w);
                        if (wg == 0) tmem_ld1(tmem_addr(tb, wl, sc + 64), zc);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i) w[i] = __float_as_uint(__uint_as_float(w[i]) * fct);
                        tmem_st32(tmem_addr(tb, wl, sc + 32 * wg), w);
                        if (wg == 0) {
                            asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};"
                                         ::"r"(tmem_addr(tb, wl, sc + 64)),
                                           "r"(__float_as_uint(__uint_as_float(zc) * fct)) : "memory");
                        }
                        tmem_st_wait();
                    }
                    Rh[h] = Rn;
                    const uint64_t nfe = f32x2_splat(-(float)Rn);
                    uint32_t w[32];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const uint64_t x0 = f32x2_add(f32x2_of(v0[2 * i], v0[2 * i + 1]), nfe);
                        const uint64_t x1 = f32x2_add(f32x2_of(v1[2 * i], v1[2 * i + 1]), nfe);
                        w[i] = live ? pack_f16x2(ex2_approx(f32x2_lo(x0)), ex2_approx(f32x2_hi(x0))) : 0u;
                        w[16 + i] = live ? pack_f16x2(ex2_approx(f32x2_lo(x1)), ex2_approx(f32x2_hi(x1))) : 0u;
                    }
                    tmem_st32(tmem_addr(tb, wl, col), w);   // tokens 64 wg .. packed into columns 64 wg ..
                    tmem_st_wait();
                    warp_arrive(&B.a_full[b], false);
                }
            }
            if (wg == 0) {
                s.rsf[f] = Rh[0];
                s.rsf[128 + f] = Rh[1];
            }
            if (__any_sync(0xffffffffu, kbig) && lane == 0) record_range(p.hdr, kRangeK);
        } else {
            // r <= 128 (one half) and element-wise maps: both warpgroups convert every job, tokens
            // 64 wg .. 64 wg + 63; FAVOR+ takes one scale per chunk from the exact maximum over the
            // eight warps (group_max8), element-wise features keep their own scale
            int R = 0;
            for (int c = 0; c < nchunks && ok; ++c) {
                const int nvalid = min(kC, un.end - (un.start + c * kC));
                const int j = c, b = j & 1;
                const bool live = f < r;
                if (!(ok = warp_wait(&B.p_full[b], (j >> 1) & 1))) break;
                tc_fence_after();
                float x[64];
                {
                    uint32_t v0[32], v1[32];
                    const uint32_t col = kColPS + 128 * b + 64 * wg;   // this warpgroup's 64 tokens
                    tmem_ld32(tmem_addr(tb, wl, col), v0);
                    tmem_ld32(tmem_addr(tb, wl, col + 32), v1);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 32; ++e) { x[e] = __uint_as_float(v0[e]); x[32 + e] = __uint_as_float(v1[e]); }
                }
                // FAVOR+: x is the exponent (log2) of phi; element-wise maps: phi itself, kept in
                // its own scale (|phi| <= 65504 for |k| below that; larger values are clamped)
                float m = -INFINITY;
                const int tbase = 64 * wg;
                bool big = false;
#pragma unroll
                for (int e = 0; e < 64; ++e) {
                    if (!favor) {
                        const float ph = tbase + e < nvalid ? phi_elementwise(x[e], p.map) : 0.f;
                        big |= live && !(fabsf(ph) <= 65504.f);
                        x[e] = fminf(fmaxf(ph, -65504.f), 65504.f);
                    } else if (live) {
                        m = fmaxf(m, x[e]);
                    }
                }
                if (!favor && __any_sync(0xffffffffu, big) && lane == 0) record_range(p.hdr, kRangeElementwise);
                if (favor && !(ok = group_max8(m, s.red, B.red_full, j, 4))) break;
                // as in the per-feature branch (the maximum is the same in every warp)
                if (favor && wg == 0 && warp == 4 && lane == 0 && !(m <= kKeyExpLimit)) record_range(p.hdr, kRangeK);
                const int e = (favor && m > -1e30f) ? (int)ceilf(m) - 15 : 0;
                const int Rn = favor ? next_key_scale(R, e, c == 0) : 0;
                if (c > 0 && Rn != R) {
                    // the previous chunk's update must be complete: rescale exactly
                    if (!(ok = warp_wait(&B.a_empty[b ^ 1], (((j - 1) >> 1)) & 1))) break;
                    const float fct = exp2i(R - Rn);
                    uint32_t w[32];
                    const uint32_t sc = kColSS + 32 * wg;   // columns 0..31 (wg 0), 32..63 (wg 1)
                    tmem_ld32(tmem_addr(tb, wl, sc), w);
                    uint32_t zc = 0u;
                    if (wg == 1) tmem_ld1(tmem_addr(tb, wl, kColSS + 64), zc);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i) w[i] = __float_as_uint(__uint_as_float(w[i]) * fct);
                    tmem_st32(tmem_addr(tb, wl, sc), w);
                    if (wg == 1) {
                        asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};"
                                     ::"r"(tmem_addr(tb, wl, kColSS + 64)),
                                       "r"(__float_as_uint(__uint_as_float(zc) * fct)) : "memory");
                    }
                    tmem_st_wait();
                }
                R = Rn;
                uint32_t w[32];
                if (favor) {
                    const float fe = (float)R;
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        w[i] = live ? pack_f16x2(ex2_approx(x[2 * i] - fe), ex2_approx(x[2 * i + 1] - fe)) : 0u;
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) w[i] = live ? pack_f16x2(x[2 * i], x[2 * i + 1]) : 0u;
                }
                tmem_st32(tmem_addr(tb, wl, kColPS + 128 * b + 64 * wg), w);   // phi(k)^T in place
                tmem_st_wait();
                warp_arrive(&B.a_full[b], false);
                if (favor && p.kscale != nullptr && t == 128) p.kscale[((int64_t)u * p.H + head) * p.Lc + c] = e;
            }
            if (wg == 0) s.rsf[f] = R;
        }
        if (!ok && lane == 0) record_error(p.hdr, LA_DEVERR_WAIT_TIMEOUT);
    } else {
        // ------------------------------------------------------------ NE: exponent offsets, V as f16 (warps 3, 12..14)
        const int ne = warp == 3 ? 0 : warp - 11;
        const int tok0 = 32 * ne;                 // this warp's 32 tokens
        // the f16 V tiles of this (unit, head) for the causal output kernel, and their |v| maxima
        unsigned char* v16 = p.v16 != nullptr
                                 ? static_cast<unsigned char*>(p.v16) + ((int64_t)u * p.H + head) * p.Lc * (int64_t)kTile
                                 : nullptr;
        float* vmx = p.v16 != nullptr ? p.vmax + ((int64_t)u * p.H + head) * p.Lc * kVmaxParts : nullptr;
        int pending = -1;                         // stage whose f16 rows are being copied out
        bool ok = true;
        for (int c = 0; c < nchunks && ok; ++c) {
            const int st = c % kStateStages;
            const int nvalid = min(kC, un.end - (un.start + c * kC));
            if (!(ok = warp_wait(&B.k_full[st], (c / kStateStages) & 1))) break;
            if (favor) {
                // -offset as bf16 hi + lo into the stage's bias columns; past the unit's
                // end a large negative exponent makes phi = 0.  Token tok0 + lane; the partner
                // row is only there to share the loop (its sum is the same token's)
                const int tok = tok0 + lane;
                float n, n_unused;
                row_sq_norm2(s.tk[st], tok, tok, n, n_unused);
                const float o = tok < nvalid ? -(n * (0.5f * kLog2e) + 0.5f * __log2f((float)r)) : -32768.f;
                const uint32_t hl = pack_bf16x2(o, 0.f);
                *reinterpret_cast<uint32_t*>(s.bias + sw128_off(tok, 16 * st)) = pack_bf16x2(o, o - bf16lo(hl));
            }
            warp_arrive(&B.cx_full[st], true);
            warp_arrive(&B.k_empty[st], false);   // this warp no longer reads the tile
            if (!(ok = warp_wait(&B.v_full[st], (c / kStateStages) & 1))) break;
            float vm = v_tile_to_f16(s.tv[st], tok0, 32, nvalid, p.hdr, lane, 32);
            if (v16 != nullptr) {
                // the 32 rows out as they lie in shared memory (4 KB, one bulk copy), and their largest |v|
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) vm = fmaxf(vm, __shfl_xor_sync(0xffffffffu, vm, o));
                fence_async_smem();
                __syncwarp();
                if (lane == 0) {
                    bulk_store(v16 + (int64_t)c * kTile + tok0 * 128, s.tv[st] + tok0 * 128, 32 * 128);
                    bulk_commit();
                    vmx[kVmaxParts * c + ne] = vm;
                }
            }
            warp_arrive(&B.vh_full[st], true);
            if (v16 != nullptr) {
                // the previous chunk's copy has read its stage: the TMA warp may refill it
                if (pending >= 0) {
                    if (lane == 0) bulk_wait_read<1>();
                    __syncwarp();
                    warp_arrive(&B.v_empty[pending], false);
                }
                pending = st;
            }
        }
        if (v16 != nullptr) {   // every copy complete before the block exits (and its stage released)
            if (lane == 0) bulk_wait_all<0>();
            __syncwarp();
            if (pending >= 0) warp_arrive(&B.v_empty[pending], false);
        }
        if (!ok && lane == 0) record_error(p.hdr, LA_DEVERR_WAIT_TIMEOUT);
    }
    // ---------------------------------------------------------------- state out
    tc_fence_before();
    __syncthreads();
    if (warp == 1 || warp == 2) {   // every MMA of both issuers finished (bounded)
        mma_commit_w(&B.drain[warp - 1]);
        if (!warp_wait(&B.drain[warp - 1], 0) && lane == 0) record_error(p.hdr, LA_DEVERR_WAIT_TIMEOUT);
    }
    __syncthreads();
    tc_fence_after();
    if (last && !p.keep_last) {   // only the key exponents were wanted
        if (warp == 1) tmem_dealloc(tb, kTmemCols);
        return;
    }
    // [S|z] as [r][65] fp32 rows in true scale: each thread's feature row into shared
    // memory (the k / v stages, all consumed; a row stride of 65 words keeps the warp's
    // stores on distinct banks), then one coalesced 16-byte copy of the whole block
    float* stage = reinterpret_cast<float*>(s.tk[0]);
    if (warp >= 4 && warp < 8) {
        const int f = t - 128;
        for (int h = 0; h < nhalves; ++h) {
            const int feat = 128 * h + f;
            const float fct = exp2i(feat < r ? s.rsf[feat] : 0);
            for (int n0 = 0; n0 < 65; n0 += 16) {
                uint32_t w[16] = {};
                if (nchunks > 0) {
                    tmem_ld16(tmem_addr(tb, (warp & 3) * 32, kColSS + kNX * h + n0), w);
                    tmem_ld_wait();
                }
                if (feat < r) {
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        if (n0 + e < 65) stage[feat * 65 + n0 + e] = __uint_as_float(w[e]) * fct;
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    {
        float4* dst = reinterpret_cast<float4*>(p.partial + ((int64_t)u * p.H + head) * (int64_t)r * 65);
        const float4* src = reinterpret_cast<const float4*>(stage);
        for (int i = t; i < r * 65 / 4; i += kStateThreads) dst[i] = src[i];
    }
    if (warp == 1) tmem_dealloc(tb, kTmemCols);
}

// ---------------------------------------------------------------------------
// FAVOR+ feature map to global fp32 (la_feature_map for bf16 input)
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads, 1)
tc_fmap_kernel(const __grid_constant__ CUtensorMap map_x, const float* omega, int T, int H, int r, float* phi,
               float* sums, int* err) {
    FmapSmem& s = smem_ref<FmapSmem>();
    const int t = threadIdx.x, head = blockIdx.y;
    const int t0 = blockIdx.x * kC;
    const int fh = r < 128 ? r : 128;
    const int nhalves = (r + 127) / 128;
    if (t == 0) prefetch_tensormap(&map_x);
    setup_bars(s.b);
    stage_omega(s.omg_hi, s.omg_lo, omega, r);
    handoff_to_mma();
    const uint32_t tb = s.b.tmem_base;
    if (t == 0) {
        mbar_arrive_expect_tx(&s.b.load, kTile);
        tma_load_3d(s.tq, &map_x, 0, head, t0, &s.b.load);
    }
    Phase lp, mp;
    bool ok = lp.wait(&s.b.load);
    if (ok) {
        const float c = favor_offset(s.tq, t, r);
        const bool valid = t0 + t < T;
        float rowsum = 0.f;
        for (int half = 0; half < nhalves; ++half) {
            if (t == 0) {
                mma_projection(tb + kColP, s.tq, s.omg_hi, s.omg_lo, 128 * half, fh);
                mma_commit(&s.b.mma);
            }
            if (!(ok = mp.wait(&s.b.mma))) break;
            tc_fence_after();
            if (phi) projection_to_global(tb, fh, c, valid, phi + ((int64_t)(t0 + t) * H + head) * r + 128 * half);
            else rowsum += projection_rowsum(tb, fh, c);
            tc_fence_before();
            __syncthreads();
            tc_fence_after();
        }
        if (ok && !phi && valid) sums[(int64_t)(t0 + t) * H + head] = rowsum;   // sum_f phi_f of the row
    }
    if (!ok) drain_after_timeout(s.b, err);
    teardown(s.b);
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess || q != cudaDriverEntryPointSuccess)
            return static_cast<EncodeTiledFn>(nullptr);
        return reinterpret_cast<EncodeTiledFn>(f);
    }();
    return fn;
}

// [T, H, 64] bf16 -> boxes of 128 tokens x 64 features of one head, 128-byte swizzle.
bool make_row_map(CUtensorMap* m, const void* base, int64_t T, int H) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {64, (cuuint64_t)H, (cuuint64_t)T};
    const cuuint64_t strides[2] = {64 * 2, (cuuint64_t)H * 64 * 2};
    const cuuint32_t box[3] = {64, 1, (cuuint32_t)kC};
    const cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename K>
cudaError_t set_smem(K kernel, size_t bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

}  // namespace

cudaError_t tc_force_wait_timeout(int enable) {
    return cudaMemcpyToSymbol(g_force_wait_timeout, &enable, sizeof(int));
}

bool tc_supported(int map, int dk, int dv, int r, int causal) {
    if (dk != 64 || dv != 64) return false;
    if (map == LA_MAP_FAVOR) return r == 64 || r == 128 || r == 256;
    // DPFP-1 and -2: the causal kernel forms the features from the input tiles
    if (map == LA_MAP_DPFP) return causal && (r == 128 || r == 256);
    return r == 64;
}

cudaError_t tc_state(const FwdParams& p, cudaStream_t s) {
    CUtensorMap mk, mv;
    if (!make_row_map(&mk, p.k, p.T, p.H) || !make_row_map(&mv, p.v, p.T, p.H)) return cudaErrorInvalidValue;
    const size_t bytes = smem_bytes<StateSmem>();
    const bool favor = p.map == LA_MAP_FAVOR;
    cudaError_t e = favor ? set_smem(tc_state_kernel<true>, bytes) : set_smem(tc_state_kernel<false>, bytes);
    if (e != cudaSuccess) return e;
    if ((int64_t)p.U * p.H > INT32_MAX) return cudaErrorInvalidConfiguration;
    const dim3 grid((unsigned)((int64_t)p.U * p.H));
    if (favor) tc_state_kernel<true><<<grid, kStateThreads, bytes, s>>>(mk, mv, TcParams{p, 0});
    else tc_state_kernel<false><<<grid, kStateThreads, bytes, s>>>(mk, mv, TcParams{p, 0});
    return cudaGetLastError();
}

cudaError_t tc_out(const FwdParams& p, int prefix_is_zero, cudaStream_t s) {
    // one-dimensional grid of (unit rank, head) blocks, rank-major (see the kernels)
    if ((int64_t)p.U * p.H > INT32_MAX) return cudaErrorInvalidConfiguration;
    const dim3 grid((unsigned)((int64_t)p.U * p.H));
    const TcParams tp{p, prefix_is_zero};
    CUtensorMap mq;
    if (!make_row_map(&mq, p.q, p.T, p.H)) return cudaErrorInvalidValue;
    cudaError_t e;
    if (p.causal) {
        CUtensorMap mk, mv;
        if (!make_row_map(&mk, p.k, p.T, p.H) || !make_row_map(&mv, p.v, p.T, p.H)) return cudaErrorInvalidValue;
        const size_t bytes = smem_bytes<CausalSmem>();
        if (p.map == LA_MAP_FAVOR) {
            if ((e = set_smem(tc_causal_out_kernel<true>, bytes)) != cudaSuccess) return e;
            tc_causal_out_kernel<true><<<grid, kCausalThreads, bytes, s>>>(mq, mk, mv, tp);
        } else {
            if ((e = set_smem(tc_causal_out_kernel<false>, bytes)) != cudaSuccess) return e;
            tc_causal_out_kernel<false><<<grid, kCausalThreads, bytes, s>>>(mq, mk, mv, tp);
        }
    } else {
        const size_t bytes = smem_bytes<BidirSmem>();
        if (p.map == LA_MAP_FAVOR) {
            if ((e = set_smem(tc_bidir_out_kernel<true>, bytes)) != cudaSuccess) return e;
            tc_bidir_out_kernel<true><<<grid, kBidirThreads, bytes, s>>>(mq, tp);
        } else {
            if ((e = set_smem(tc_bidir_out_kernel<false>, bytes)) != cudaSuccess) return e;
            tc_bidir_out_kernel<false><<<grid, kBidirThreads, bytes, s>>>(mq, tp);
        }
    }
    return cudaGetLastError();
}

static cudaError_t launch_fmap(const void* x, const float* omega, int64_t T, int H, int r, float* phi, float* sums,
                               int* err, cudaStream_t s) {
    CUtensorMap mx;
    if (!make_row_map(&mx, x, T, H)) return cudaErrorInvalidValue;
    const size_t bytes = smem_bytes<FmapSmem>();
    cudaError_t e = set_smem(tc_fmap_kernel, bytes);
    if (e != cudaSuccess) return e;
    tc_fmap_kernel<<<dim3((unsigned)ceil_div(T, kC), (unsigned)H), kThreads, bytes, s>>>(mx, omega, (int)T, H, r,
                                                                                        phi, sums, err);
    return cudaGetLastError();
}

cudaError_t tc_feature_map(const void* x, const float* omega, int64_t T, int H, int r, float* phi, int* err,
                           cudaStream_t s) {
    return launch_fmap(x, omega, T, H, r, phi, nullptr, err, s);
}

cudaError_t tc_feature_sums(const void* x, const float* omega, int64_t T, int H, int r, float* sums, int* err,
                            cudaStream_t s) {
    return launch_fmap(x, omega, T, H, r, nullptr, sums, err, s);
}

}  // namespace la
