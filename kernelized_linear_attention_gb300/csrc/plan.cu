// Work planning and the segment-state scan.
//
// A forward call splits every packed sequence into segments of at most L
// tokens (one work unit each, processed for every head).  The planner reads
// cu_seqlens on the device, checks the packing rules and writes the unit
// table; the scan turns per-unit partial states into the state each unit
// starts from.  Segments exist only to spread long sequences over the SMs;
// the state still resets exactly at every sequence boundary ("Reassociate a
// feature-map kernel", ¶4: packing must reset the state at the logical
// boundary).
#include "internal.h"

namespace la {

namespace {

constexpr int kPlanThreads = 1024;
constexpr int kSortUnits = 1024;   // packed batches with more units keep the unit order

__device__ __forceinline__ int block_exclusive_scan(int x, int* warp_sums, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int w = (lane < (int)(blockDim.x >> 5)) ? warp_sums[lane] : 0;
        int wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += y;
        }
        warp_sums[lane] = wi - w;  // exclusive prefix of warp totals
        if (lane == 31) *total = wi;
    }
    __syncthreads();
    int r = incl - x + warp_sums[warp];
    __syncthreads();
    return r;
}

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(FwdParams p) {
    __shared__ int bad;
    __shared__ int carry;
    __shared__ int warp_sums[32];
    __shared__ int chunk_total;
    if (threadIdx.x == 0) { bad = 0; carry = 0; }
    __syncthreads();
    const int64_t eq_len = p.cu_seqlens ? 0 : p.T / p.nseq;

    // pass 1: validate
    for (int s = threadIdx.x; s < p.nseq; s += blockDim.x) {
        int64_t a, b;
        if (p.cu_seqlens) { a = p.cu_seqlens[s]; b = p.cu_seqlens[s + 1]; }
        else { a = (int64_t)s * eq_len; b = a + eq_len; }
        bool ok = (b >= a) && (a >= 0) && (b <= p.T);
        if (s == 0 && a != 0) ok = false;
        if (s == p.nseq - 1 && b != p.T) ok = false;
        if (!ok) atomicOr(&bad, 1);
    }
    __syncthreads();
    if (bad) {
        if (threadIdx.x == 0) {
            p.hdr->n_units = 0;
            p.hdr->error = LA_DEVERR_CU_SEQLENS;
            p.hdr->range = 0;
        }
        for (int s = threadIdx.x; s <= p.nseq; s += blockDim.x) p.seq_first[s] = 0;
        return;
    }

    // pass 2: units per sequence, exclusive scan, unit table
    for (int base = 0; base < p.nseq; base += blockDim.x) {
        const int s = base + threadIdx.x;
        int64_t a = 0, b = 0;
        int n = 0;
        if (s < p.nseq) {
            if (p.cu_seqlens) { a = p.cu_seqlens[s]; b = p.cu_seqlens[s + 1]; }
            else { a = (int64_t)s * eq_len; b = a + eq_len; }
            n = (int)ceil_div(b - a, p.L);
        }
        const int off = carry + block_exclusive_scan(n, warp_sums, &chunk_total);
        if (s < p.nseq) {
            p.seq_first[s] = off;
            for (int i = 0; i < n; ++i) {
                const int u = off + i;
                if (u < p.U) {
                    Unit un;
                    un.seq = s;
                    un.start = (int)(a + (int64_t)i * p.L);
                    { const int64_t e_ = a + (int64_t)(i + 1) * p.L; un.end = (int)(e_ < b ? e_ : b); }
                    un.first = off;
                    p.units[u] = un;
                }
            }
        }
        __syncthreads();
        if (threadIdx.x == 0) carry += chunk_total;
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        const int total = carry;
        p.seq_first[p.nseq] = min(total, p.U);
        p.hdr->n_units = min(total, p.U);
        p.hdr->error = (total > p.U) ? LA_DEVERR_CU_SEQLENS : LA_DEVERR_NONE;
        p.hdr->range = 0;
    }

    // pass 3: the order in which the tensor-core kernels take the units.
    // Packed batches mix short and long units, and an equal-length batch's last
    // segments are shorter; launched longest first, the blocks of short units
    // fill in behind the long ones instead of leaving a tail of long units on a
    // few SMs.  Rank = number of units longer, ties by index (a permutation);
    // batches of more than kSortUnits units keep 0, 1, ..
    __shared__ int slen[kSortUnits];
    const int nu = min(carry, p.U);
    const bool sort = nu <= kSortUnits;
    if (sort)
        for (int i = threadIdx.x; i < nu; i += blockDim.x) slen[i] = p.units[i].end - p.units[i].start;
    __syncthreads();
    for (int i = threadIdx.x; i < nu; i += blockDim.x) {
        int rank = i;
        if (sort) {
            const int li = slen[i];
            rank = 0;
            for (int j = 0; j < nu; ++j) {
                const int lj = slen[j];
                rank += (lj > li || (lj == li && j < i)) ? 1 : 0;
            }
        }
        p.order[rank] = i;
    }
}

constexpr int kScanThreads = 256;
constexpr int kScanPerThread = 4;
constexpr int kScanBatch = 8;   // units whose partial sums are in flight before they are added

// grid: (ceil(E / (256*4)), nseq, H).  The result goes to p.prefix (the
// backward pass points it at its suffix buffer and sets p.reverse).  Each
// thread owns elements e of one
// (sequence, head) state and walks the sequence's units in token order, so
// state_in may alias state_out: it is read before the same thread writes it.
// The units are taken kScanBatch at a time, their partial sums loaded before
// any is added, so only the additions form a dependent chain.
__global__ void __launch_bounds__(kScanThreads) scan_kernel(FwdParams p) {
    const int s = blockIdx.y, h = blockIdx.z;
    const int u0 = p.seq_first[s], u1 = p.seq_first[s + 1];
    const int64_t E = (int64_t)p.r * p.dvx;
    const int64_t e0 = (int64_t)blockIdx.x * kScanThreads * kScanPerThread + threadIdx.x;
    const int64_t sbase = ((int64_t)s * p.H + h) * E;
    float acc[kScanPerThread];
#pragma unroll
    for (int j = 0; j < kScanPerThread; ++j) {
        const int64_t e = e0 + j * kScanThreads;
        acc[j] = (p.state_in != nullptr && e < E) ? p.state_in[sbase + e] : 0.f;
    }
    const bool rev = p.causal && p.reverse;
    const int nu = u1 - u0;
    for (int b0 = 0; b0 < nu; b0 += kScanBatch) {
        // position b0 + i of the walk is unit u0 + (b0 + i), or u1 - 1 - (b0 + i) walking backwards
        float part[kScanBatch][kScanPerThread];
#pragma unroll
        for (int i = 0; i < kScanBatch; ++i) {
            const int w = b0 + i, u = rev ? u1 - 1 - w : u0 + w;
            // causal forward: the last unit's sum exists only with keep_last
            const bool add = w < nu && (rev || !p.causal || u + 1 < u1 || p.keep_last);
            const int64_t base = ((int64_t)u * p.H + h) * E;
#pragma unroll
            for (int j = 0; j < kScanPerThread; ++j) {
                const int64_t e = e0 + j * kScanThreads;
                part[i][j] = (add && e < E) ? p.partial[base + e] : 0.f;
            }
        }
#pragma unroll
        for (int i = 0; i < kScanBatch; ++i) {
            const int w = b0 + i, u = rev ? u1 - 1 - w : u0 + w;
            if (w < nu) {
                const int64_t base = ((int64_t)u * p.H + h) * E;
#pragma unroll
                for (int j = 0; j < kScanPerThread; ++j) {
                    const int64_t e = e0 + j * kScanThreads;
                    if (e < E) {
                        if (p.causal) p.prefix[base + e] = acc[j];   // exclusive prefix (or suffix)
                        acc[j] += part[i][j];
                    }
                }
            }
        }
    }
    if (!p.causal) {   // bidirectional: every unit of the sequence reads the whole-sequence sum
        for (int u = u0; u < u1; ++u) {
            const int64_t base = ((int64_t)u * p.H + h) * E;
#pragma unroll
            for (int j = 0; j < kScanPerThread; ++j) {
                const int64_t e = e0 + j * kScanThreads;
                if (e < E) p.prefix[base + e] = acc[j];
            }
        }
    }
    if (p.state_out != nullptr) {
#pragma unroll
        for (int j = 0; j < kScanPerThread; ++j) {
            const int64_t e = e0 + j * kScanThreads;
            if (e < E) p.state_out[sbase + e] = acc[j];
        }
    }
}

}  // namespace

cudaError_t launch_plan(const FwdParams& p, cudaStream_t s) {
    plan_kernel<<<1, kPlanThreads, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_scan(const FwdParams& p, cudaStream_t s) {
    const int64_t E = (int64_t)p.r * p.dvx;
    dim3 grid((unsigned)ceil_div(E, kScanThreads * kScanPerThread), (unsigned)p.nseq, (unsigned)p.H);
    scan_kernel<<<grid, kScanThreads, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace la
