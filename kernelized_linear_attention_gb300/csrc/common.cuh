// Shared definitions of the kernelized linear attention library: workspace
// layout, work units, element access helpers.  Internal to liblinattn.so.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <stddef.h>

#include "linattn.h"

namespace la {

// A work unit is one contiguous token range (a segment) of one packed
// sequence; every unit is processed for every head (grid.y).  Segments of one
// sequence are consecutive unit indices, in token order.
struct Unit {
    int seq;     // sequence index
    int start;   // first token (global row)
    int end;     // one past the last token
    int first;   // unit index of the sequence's first segment
};

// First 256 bytes of every workspace.
struct WsHeader {
    int error;     // LA_DEVERR_*; written with atomicMax, never cleared by kernels but the planner
    int n_units;   // units the planner produced
    int range;     // bits of the operands that had a value clamped into the fp16 range
                   // (1 values, 2 key features, 4 query features, 8 element-wise features);
                   // reported as LA_DEVERR_RANGE
    int pad[61];
};

// Byte offsets of the workspace regions for one forward call.
// Parts (32-row quarters) of a chunk whose largest |v| the state kernel records.
constexpr int kVmaxParts = 4;

struct Layout {
    size_t units;      // Unit[U]
    size_t seq_first;  // int[nseq + 1]: first unit of each sequence (+ total)
    size_t order;      // int[U]: units by decreasing token count (packed batches), else 0, 1, ..
    size_t partial;    // float[U][H][r][dvx]: per-unit state sum_j phi(k_j) [v_j | 1]^T
    size_t prefix;     // float[U][H][r][dvx]: state entering the unit (causal) / whole-sequence state (bidir)
    size_t kscale;     // int[U][H][Lc]: power-of-two exponent of the keys' features in each chunk
    size_t v16;        // causal FAVOR+ tensor path: [U][H][Lc] tiles of 128 x 64 f16 V (128B-swizzled rows)
    size_t vmax;       // float[U][H][Lc][kVmaxParts]: largest |v| of each 32-row quarter of a chunk's valid rows
    size_t sig_q;      // float[T][H]: sum_f phi_f(q) (sum normalisation on the tensor-core path)
    size_t sig_k;      // float[T][H]: sum_f phi_f(k)
    size_t suffix;     // backward: float[U][H][r][dvx], sum of phi(q) g^T over later units (or the sequence)
    size_t g;          // backward: float[T][H][dvx], d num | d den of every row
    size_t omega_t;    // backward: float[dk][r], Omega transposed
    size_t total;      // bytes
    int U;             // upper bound on units
    int L;             // segment length in tokens
    int Lc;            // chunks of 128 tokens per segment (tensor-core path)
    int dvx;           // d_v + 1: the ones column carries z
};

constexpr int kAlign = 256;

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
__host__ __device__ inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
__host__ __device__ inline int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }

// Parameters of one forward call, as the kernels see them.
struct FwdParams {
    const void* q;
    const void* k;
    const void* v;
    const float* omega;
    void* out;
    const int32_t* cu_seqlens;  // may be NULL
    int nseq;
    int64_t T;
    int H, dk, dv, r, dvx;
    int map;       // la_map
    int causal;
    int norm;      // la_norm
    float eps;
    const float* state_in;  // [nseq][H][r][dvx] or NULL: state each sequence starts from
    float* state_out;       // [nseq][H][r][dvx] or NULL: state after each sequence's last token
    int keep_last;          // causal: the state pass also sums each sequence's last segment
    // backward pass only
    const void* dout;       // [T][H][dv] upstream gradient
    void* dq_out;           // [T][H][dk] gradients written
    void* dk_out;           // [T][H][dk]
    void* dv_out;           // [T][H][dv]
    float* g;               // [T][H][dvx] workspace: d num | d den of every row
    float* suffix;          // [U][H][r][dvx] workspace: sum of phi(q_i) g_i^T over later units
    int reverse;            // scan: suffix (later units) instead of prefix
    float* omega_t;         // [dk][r] workspace: Omega transposed (coalesced feature loads)
    float* sig_q;           // [T][H] workspace: feature sums of q and k (sum normalisation)
    float* sig_k;
    const float* div_rows;  // [T][H] or NULL: tensor-core outputs are divided by max(div_rows, eps)
    // workspace regions
    WsHeader* hdr;
    Unit* units;
    int* seq_first;
    int* order;             // the tensor-core output kernels take units in this order (longest first)
    float* partial;
    float* prefix;
    // Tensor-core path: for every (unit, head, chunk of 128 tokens) the exponent e such that
    // the chunk's FAVOR+ key features times 2^-e lie below 2^15 (written by the state kernel,
    // read by the causal output kernel).
    int* kscale;
    // Causal FAVOR+ tensor path: every chunk's V tile as f16 in the shared-memory layout of the
    // kernels (rows of 128 bytes, 16-byte pieces swizzled within 1024-byte groups), one 16 KB
    // tile per (unit, head, chunk), and the largest |v| of its valid rows
    // (per 32-row quarter; written by the state kernel, read by the causal output kernel); else NULL.
    void* v16;
    float* vmax;
    int U, L, Lc;
};

// ---------------------------------------------------------------------------
// Element access
// ---------------------------------------------------------------------------
__device__ __forceinline__ float load_elem(const float* p, int64_t i) { return p[i]; }
__device__ __forceinline__ float load_elem(const __nv_bfloat16* p, int64_t i) {
    return __bfloat162float(p[i]);
}
__device__ __forceinline__ void store_elem(float* p, int64_t i, float x) { p[i] = x; }
__device__ __forceinline__ void store_elem(__nv_bfloat16* p, int64_t i, float x) {
    p[i] = __float2bfloat16_rn(x);
}

__device__ __forceinline__ void record_error(WsHeader* hdr, int code) {
    atomicMax(&hdr->error, code);
}
// A value outside the range the fp16 tensor-core operands hold was clamped.
constexpr int kRangeV = 1, kRangeK = 2, kRangeQ = 4, kRangeElementwise = 8;
__device__ __forceinline__ void record_range(WsHeader* hdr, int bits) {
    if ((hdr->range & bits) != bits) atomicOr(&hdr->range, bits);
}

}  // namespace la
