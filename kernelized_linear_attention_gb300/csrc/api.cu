// C ABI of liblinattn.so: argument checks, workspace layout, dispatch.
// The operation each entry point computes is specified in include/linattn.h.
#include <algorithm>
#include <cmath>
#include <functional>
#include <map>
#include <mutex>
#include <tuple>
#include <vector>

#include "internal.h"

namespace la {

namespace {

constexpr int kPathSimt = 0;
constexpr int kPathTensor = 1;

int device_sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

// Shape checks shared by every forward entry point and the size queries.
la_status check_dims(int map, int dtype, int nseq, int64_t T, int H, int dk, int dv, int r,
                     bool has_cu) {
    if (map < LA_MAP_IDENTITY || map > LA_MAP_DPFP) return LA_ERR_INVALID_ARG;
    if (dtype != LA_F32 && dtype != LA_BF16) return LA_ERR_INVALID_ARG;
    if (nseq < 1 || nseq > 65535 || H < 1 || H > 65535) return LA_ERR_INVALID_ARG;
    if (T < 0 || T > (int64_t)INT32_MAX) return LA_ERR_INVALID_ARG;
    if (dk < 1 || dv < 1 || r < 1) return LA_ERR_INVALID_ARG;
    if ((map == LA_MAP_IDENTITY || map == LA_MAP_ELU1) && r != dk) return LA_ERR_INVALID_ARG;
    if (map == LA_MAP_DPFP && (r % (2 * dk) != 0 || r / (2 * dk) > 2 * dk - 1)) return LA_ERR_INVALID_ARG;
    if (!has_cu && (T % nseq) != 0) return LA_ERR_INVALID_ARG;
    if (dk > LA_MAX_DK || dv > LA_MAX_DV || r > LA_MAX_R) return LA_ERR_UNSUPPORTED;
    return LA_OK;
}

// Tensor cores for bf16 shapes the tcgen05 kernels cover; fp32 (exact
// arithmetic) and every other shape on CUDA cores.
int select_path(int causal, int map, int dtype, int dk, int dv, int r, int norm = LA_NORM_ATTENTION) {
    return (dtype == LA_BF16 && norm != LA_NORM_SUM && tc_supported(map, dk, dv, r, causal)) ? kPathTensor
                                                                                              : kPathSimt;
}

// DPFP on tensor cores runs every sequence as one unit: its state pass (CUDA
// cores) then only has work when a final state is wanted.
bool whole_sequences(int path, int map) { return path == kPathTensor && map == LA_MAP_DPFP; }
// The causal FAVOR+ tensor-core route passes V as f16 from the state kernel to the output kernel.
bool vtables(int path, int causal, int map) { return path == kPathTensor && causal && map == LA_MAP_FAVOR; }

// Normalisation variants; sum normalisation needs non-negative features.
la_status check_norm(int norm, int map) {
    if (norm < LA_NORM_ATTENTION || norm > LA_NORM_SUM) return LA_ERR_INVALID_ARG;
    if (norm == LA_NORM_SUM && map == LA_MAP_IDENTITY) return LA_ERR_INVALID_ARG;
    return LA_OK;
}

int path_chunk(int path) { return path == kPathTensor ? 128 : simt_chunk(); }

la_status path_supported(int path, int map, int dk, int dv, int r) {
    if (path == kPathSimt && simt_smem_bytes(map, dk, dv, r) > kSmemLimitBytes) return LA_ERR_UNSUPPORTED;
    return LA_OK;
}

// Finish time, in chunk times, of nbig blocks of big chunks and nsmall of small
// chunks started longest first (the order in which the tensor-core kernels map
// block indices to units) on nsm SMs, each block as its SM frees up and each
// paying one chunk of set-up.
int64_t block_makespan(int64_t nbig, int64_t big, int64_t nsmall, int64_t small, int nsm) {
    std::vector<int64_t> free_at((size_t)std::max(1, nsm), 0);   // min-heap of SM free times
    int64_t end = 0;
    for (int64_t i = 0; i < nbig + nsmall; ++i) {
        std::pop_heap(free_at.begin(), free_at.end(), std::greater<int64_t>());
        free_at.back() += (i < nbig ? big : small) + 1;
        end = std::max(end, free_at.back());
        std::push_heap(free_at.begin(), free_at.end(), std::greater<int64_t>());
    }
    return end;
}

// Tensor-core path, equal-length batches: the segment length in chunks whose blocks
// (pairs (sequence, head) pairs x segments, the last segment of a sequence shorter)
// finish soonest, among those giving between half a wave and two waves of blocks;
// ties go to the longer segment.  B=1 H=16 N=65536 on 152 SMs: 54 chunks (144 blocks
// of 54 and 16 of 26, the second eight of which start where the first eight end)
// instead of 57 in one wave of 144.  Zero: no candidate (the caller keeps its length).
int64_t tensor_segment_chunks(int64_t nchunks, int64_t pairs, int nsm) {
    static std::mutex mu;
    static std::map<std::tuple<int64_t, int64_t, int>, int64_t> memo;
    const auto key = std::make_tuple(nchunks, pairs, nsm);
    {
        std::lock_guard<std::mutex> g(mu);
        auto it = memo.find(key);
        if (it != memo.end()) return it->second;
    }
    const int64_t min_segs = std::max<int64_t>(1, ceil_div((int64_t)nsm, 2 * pairs));
    int64_t best = -1, best_lc = 0;
    for (int64_t lc = nchunks; lc >= 1; --lc) {
        const int64_t segs = ceil_div(nchunks, lc);
        if (segs * pairs > 2 * (int64_t)nsm) break;   // segs only grows as lc falls
        if (segs < min_segs) continue;
        const int64_t t = block_makespan((segs - 1) * pairs, lc, pairs, nchunks - (segs - 1) * lc, nsm);
        if (best < 0 || t < best) { best = t; best_lc = lc; }
    }
    std::lock_guard<std::mutex> g(mu);
    memo[key] = best_lc;
    return best_lc;
}

// Segment length and unit bound.  Equal-length batches split every sequence
// into the same number of segments so that units * heads fills the SMs;
// packed batches (lengths only known on the device) use one length for all.
Layout make_layout(int path, bool has_cu, int nseq, int64_t T, int H, int dv, int r, int nsm, bool bwd = false,
                   bool whole = false, bool vtables = false) {
    Layout lo{};
    const int64_t C = path_chunk(path);
    int64_t L, U;
    if (whole) {
        L = std::max<int64_t>(C, ceil_div(has_cu ? T : T / nseq, C) * C);
        U = has_cu ? nseq + 1 : nseq;
    } else if (!has_cu) {
        const int64_t len = T / nseq, pairs = std::max<int64_t>(1, (int64_t)nseq * H);
        int64_t per = std::max<int64_t>(1, nsm / pairs);   // one wave of CTAs (units x heads)
        if (bwd) {
            // the backward's blocks (one per SM) carry little start-up: take the segment count whose
            // blocks finish soonest, counting whole waves of nsm blocks and one chunk of start-up per
            // wave (B=4 H=8 N=4096: two waves of 36 x 8 blocks instead of one of 16 x 8, 7% faster;
            // the forward's tensor-core state pass lost 19% that way on the 65536-token batch)
            const int64_t nchunks = ceil_div(len, C);
            int64_t best_cost = -1;
            for (int64_t pp = 1; pp <= std::max<int64_t>(1, 2 * nsm / pairs) && pp <= nchunks; ++pp) {
                const int64_t Lp = ceil_div(nchunks, pp) * C, segs = ceil_div(len, Lp);
                const int64_t cost = ceil_div(segs * pairs, (int64_t)std::max(1, nsm)) * (Lp / C + 1);
                if (best_cost < 0 || cost < best_cost) { per = pp; best_cost = cost; }
            }
        }
        L = std::max<int64_t>(C, ceil_div(ceil_div(len, per), C) * C);
        if (path == kPathTensor && !bwd) {
            const int64_t lc = tensor_segment_chunks(ceil_div(len, C), pairs, nsm);
            if (lc > 0) L = lc * C;
        }
        U = (int64_t)nseq * ceil_div(len, L);
    } else {
        L = std::max<int64_t>(C, ceil_div(ceil_div(T * H, std::max(1, nsm)), C) * C);
        U = nseq + ceil_div(T, L);
    }
    U = std::max<int64_t>(U, 1);
    lo.L = (int)std::min<int64_t>(L, INT32_MAX);
    lo.U = (int)U;
    lo.Lc = (int)ceil_div(lo.L, 128);
    lo.dvx = dv + 1;
    size_t o = align_up(sizeof(WsHeader), kAlign);
    lo.units = o;     o = align_up(o + sizeof(Unit) * (size_t)U, kAlign);
    lo.seq_first = o; o = align_up(o + sizeof(int) * (size_t)(nseq + 1), kAlign);
    lo.order = o;     o = align_up(o + sizeof(int) * (size_t)U, kAlign);
    const size_t state_bytes = sizeof(float) * (size_t)U * H * r * lo.dvx;
    lo.partial = o;   o = align_up(o + state_bytes, kAlign);
    lo.prefix = o;    o = align_up(o + state_bytes, kAlign);
    lo.kscale = o;    o = align_up(o + (path == kPathTensor ? sizeof(int) * (size_t)U * H * lo.Lc : 0), kAlign);
    lo.v16 = o;       o = align_up(o + (vtables ? (size_t)16384 * U * H * lo.Lc : 0), kAlign);
    lo.vmax = o;      o = align_up(o + (vtables ? sizeof(float) * kVmaxParts * (size_t)U * H * lo.Lc : 0), kAlign);
    lo.sig_q = o;     o = align_up(o + sizeof(float) * (size_t)T * H, kAlign);
    lo.sig_k = o;     o = align_up(o + sizeof(float) * (size_t)T * H, kAlign);
    if (bwd) {
        lo.suffix = o; o = align_up(o + state_bytes, kAlign);
        lo.g = o;      o = align_up(o + sizeof(float) * (size_t)T * H * lo.dvx, kAlign);
        lo.omega_t = o; o = align_up(o + sizeof(float) * (size_t)r * LA_MAX_DK, kAlign);
    }
    lo.total = o;
    return lo;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

la_status forward(int causal, int phase_lo, int phase_hi, const void* q, const void* k, const void* v,
                  const float* omega, int map, int dtype, const int32_t* cu_seqlens, int nseq, int64_t T,
                  int H, int dk, int dv, int r, float eps, void* out, void* workspace,
                  size_t workspace_bytes, void* stream, int* launched, int norm = LA_NORM_ATTENTION,
                  const float* state_in = nullptr, float* state_out = nullptr) {
    if (launched) *launched = 0;
    const bool has_cu = cu_seqlens != nullptr;
    la_status st = check_dims(map, dtype, nseq, T, H, dk, dv, r, has_cu);
    if (st != LA_OK) return st;
    if ((st = check_norm(norm, map)) != LA_OK) return st;
    if ((state_in && !aligned(state_in, 4)) || (state_out && !aligned(state_out, 4))) return LA_ERR_INVALID_ARG;
    if (!(eps >= 0.f) || !std::isfinite(eps)) return LA_ERR_INVALID_ARG;
    if (map == LA_MAP_FAVOR && omega == nullptr) return LA_ERR_INVALID_ARG;
    if (workspace == nullptr || !aligned(workspace, kAlign)) return LA_ERR_INVALID_ARG;
    if (T > 0 && (!q || !k || !v || !out)) return LA_ERR_INVALID_ARG;
    const size_t esz = dtype == LA_F32 ? 4 : 2;
    if (!aligned(q, esz) || !aligned(k, esz) || !aligned(v, esz) || !aligned(out, esz)) return LA_ERR_INVALID_ARG;
    if (omega && !aligned(omega, 4)) return LA_ERR_INVALID_ARG;
    int path = select_path(causal, map, dtype, dk, dv, r);
    // sum normalisation with a carried state stays on the CUDA-core kernels (their states hold
    // the sum-normalised z; the tensor-core route below scales only the values)
    if (norm == LA_NORM_SUM && (state_in || state_out)) path = kPathSimt;
    // TMA and vector loads need 16-byte aligned operands
    if (path == kPathTensor && !(aligned(q, 16) && aligned(k, 16) && aligned(v, 16) && aligned(out, 16) &&
                                 (omega == nullptr || aligned(omega, 16))))
        path = kPathSimt;
    if ((st = path_supported(path, map, dk, dv, r)) != LA_OK) return st;
    const int nsm = device_sm_count();
    if (nsm <= 0) return LA_ERR_CUDA;
    const Layout lo = make_layout(path, has_cu, nseq, T, H, dv, r, nsm, false, whole_sequences(path, map),
                                  vtables(path, causal, map));
    if (workspace_bytes < lo.total) return LA_ERR_WORKSPACE;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char* ws = static_cast<char*>(workspace);
    FwdParams p{};
    p.q = q; p.k = k; p.v = v; p.omega = omega; p.out = out;
    p.cu_seqlens = cu_seqlens; p.nseq = nseq; p.T = T;
    p.H = H; p.dk = dk; p.dv = dv; p.r = r; p.dvx = lo.dvx;
    p.map = map; p.causal = causal; p.norm = norm; p.eps = eps;
    p.state_in = state_in; p.state_out = state_out;
    // Sum normalisation on tensor cores: the kernels compute the unnormalised output for the
    // values v / sigma_k, which the plan phase writes into `out`; the output phase divides by
    // sigma_q (norm.cu).
    const bool tc_sum = path == kPathTensor && norm == LA_NORM_SUM;
    if (tc_sum) {
        p.v = out;
        p.norm = LA_NORM_NONE;
    }
    p.hdr = reinterpret_cast<WsHeader*>(ws);
    p.units = reinterpret_cast<Unit*>(ws + lo.units);
    p.seq_first = reinterpret_cast<int*>(ws + lo.seq_first);
    p.order = reinterpret_cast<int*>(ws + lo.order);
    p.partial = reinterpret_cast<float*>(ws + lo.partial);
    p.prefix = reinterpret_cast<float*>(ws + lo.prefix);
    p.sig_q = reinterpret_cast<float*>(ws + lo.sig_q);
    p.sig_k = reinterpret_cast<float*>(ws + lo.sig_k);
    if (tc_sum) p.div_rows = p.sig_q;   // the output kernels divide by max(sigma_q, eps)
    p.U = lo.U; p.L = lo.L; p.Lc = lo.Lc;
    // The causal FAVOR+ output kernel scales each chunk's key features by the power of
    // two the state kernel records per chunk: the state pass then covers every unit.
    const bool want_kscale = path == kPathTensor && causal && map == LA_MAP_FAVOR;
    if (want_kscale) {
        p.kscale = reinterpret_cast<int*>(ws + lo.kscale);
        // and hands it each chunk's V as f16 with the chunk's largest |v|
        p.v16 = ws + lo.v16;
        p.vmax = reinterpret_cast<float*>(ws + lo.vmax);
    }

    // A causal call whose sequences are all single segments starts every unit
    // from its sequence's state_in (or zero): unless the final state is
    // wanted, the state pass and the scan are skipped and the output kernel
    // reads state_in in place of the scan's prefix (unit u is sequence u).
    // A final state needs every segment's sum, the last one included.
    const bool single_segments = !has_cu && lo.U == nseq;
    const bool need_state = !causal || !single_segments || state_out != nullptr;
    const bool run_state = need_state || want_kscale;   // the scan only when need_state
    p.keep_last = state_out != nullptr ? 1 : 0;
    int prefix_is_zero = 0;
    if (!need_state) {
        if (state_in) p.prefix = const_cast<float*>(state_in);   // read only by the output kernels
        else prefix_is_zero = 1;
    }
    int n = 0;
    cudaError_t e = cudaSuccess;
    for (int ph = phase_lo; ph <= phase_hi && e == cudaSuccess; ++ph) {
        switch (ph) {
            case LA_PHASE_PLAN:
                e = launch_plan(p, s); ++n;
                if (e == cudaSuccess && tc_sum && T > 0) {
                    if (map == LA_MAP_FAVOR) {
                        e = tc_feature_sums(q, omega, T, H, r, p.sig_q, &p.hdr->error, s);
                        if (e == cudaSuccess) e = tc_feature_sums(k, omega, T, H, r, p.sig_k, &p.hdr->error, s);
                        if (e == cudaSuccess) e = sum_scale_values(v, p.sig_k, eps, T, H, dv, out, s);
                        n += 3;
                    } else {
                        e = sum_prologue_elementwise(q, k, v, map, T, H, r, eps, p.sig_q, out, s);
                        ++n;
                    }
                }
                break;
            case LA_PHASE_STATE:
                if (T > 0 && run_state) {
                    e = (path == kPathTensor && map != LA_MAP_DPFP) ? tc_state(p, s) : simt_state(p, dtype, s);
                    ++n;
                }
                break;
            case LA_PHASE_SCAN:
                // with a final state to write, empty sequences still need the scan
                if ((T > 0 || state_out) && need_state) { e = launch_scan(p, s); ++n; }
                break;
            case LA_PHASE_OUTPUT:
                if (T > 0) {
                    e = path == kPathTensor ? tc_out(p, prefix_is_zero, s)
                                            : simt_out(p, dtype, prefix_is_zero, s);
                    ++n;
                }
                break;
            default:
                return LA_ERR_INVALID_ARG;
        }
    }
    if (launched) *launched = n;
    return e == cudaSuccess ? LA_OK : LA_ERR_CUDA;
}

// The backward pass (always the fp32 CUDA-core kernels): plan, forward state
// pass and scan (the state entering every segment), bwd_q (g, dq, per-segment
// sums of phi(q) g^T), reverse scan (those sums over the later segments),
// bwd_kv (dk, dv).
la_status backward(int causal, int norm, const void* q, const void* k, const void* v, const float* omega, int map,
                   int dtype, const int32_t* cu_seqlens, int nseq, int64_t T, int H, int dk, int dv, int r,
                   float eps, const void* dout, void* dq, void* dkk, void* dvv, void* workspace,
                   size_t workspace_bytes, void* stream) {
    const bool has_cu = cu_seqlens != nullptr;
    la_status st = check_dims(map, dtype, nseq, T, H, dk, dv, r, has_cu);
    if (st != LA_OK) return st;
    if ((st = check_norm(norm, map)) != LA_OK) return st;
    if (!(eps >= 0.f) || !std::isfinite(eps)) return LA_ERR_INVALID_ARG;
    if (map == LA_MAP_FAVOR && omega == nullptr) return LA_ERR_INVALID_ARG;
    if (workspace == nullptr || !aligned(workspace, kAlign)) return LA_ERR_INVALID_ARG;
    if (T > 0 && (!q || !k || !v || !dout || !dq || !dkk || !dvv)) return LA_ERR_INVALID_ARG;
    const size_t esz = dtype == LA_F32 ? 4 : 2;
    for (const void* ptr : {q, k, v, dout, static_cast<const void*>(dq), static_cast<const void*>(dkk),
                            static_cast<const void*>(dvv)})
        if (!aligned(ptr, esz)) return LA_ERR_INVALID_ARG;
    if (omega && !aligned(omega, 4)) return LA_ERR_INVALID_ARG;
    if (bwd_smem_bytes(dk, dv, r) > kSmemLimitBytes || path_supported(kPathSimt, map, dk, dv, r) != LA_OK)
        return LA_ERR_UNSUPPORTED;
    const int nsm = device_sm_count();
    if (nsm <= 0) return LA_ERR_CUDA;
    const Layout lo = make_layout(kPathSimt, has_cu, nseq, T, H, dv, r, nsm, true);
    if (workspace_bytes < lo.total) return LA_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char* ws = static_cast<char*>(workspace);
    FwdParams p{};
    p.q = q; p.k = k; p.v = v; p.omega = omega; p.out = nullptr;
    p.cu_seqlens = cu_seqlens; p.nseq = nseq; p.T = T;
    p.H = H; p.dk = dk; p.dv = dv; p.r = r; p.dvx = lo.dvx;
    p.map = map; p.causal = causal; p.norm = norm; p.eps = eps;
    p.dout = dout; p.dq_out = dq; p.dk_out = dkk; p.dv_out = dvv;
    p.hdr = reinterpret_cast<WsHeader*>(ws);
    p.units = reinterpret_cast<Unit*>(ws + lo.units);
    p.seq_first = reinterpret_cast<int*>(ws + lo.seq_first);
    p.order = reinterpret_cast<int*>(ws + lo.order);
    p.partial = reinterpret_cast<float*>(ws + lo.partial);
    p.prefix = reinterpret_cast<float*>(ws + lo.prefix);
    p.suffix = reinterpret_cast<float*>(ws + lo.suffix);
    p.g = reinterpret_cast<float*>(ws + lo.g);
    p.omega_t = reinterpret_cast<float*>(ws + lo.omega_t);
    p.U = lo.U; p.L = lo.L;
    cudaError_t e = launch_plan(p, s);
    if (e == cudaSuccess && T > 0 && map == LA_MAP_FAVOR) e = bwd_transpose_omega(p, s);
    if (e != cudaSuccess || T == 0) return e == cudaSuccess ? LA_OK : LA_ERR_CUDA;
    const bool single_segments = !has_cu && lo.U == nseq;
    const bool need_state = !causal || !single_segments;
    if (need_state) {
        if ((e = simt_state(p, dtype, s)) != cudaSuccess) return LA_ERR_CUDA;
        if ((e = launch_scan(p, s)) != cudaSuccess) return LA_ERR_CUDA;
    }
    if ((e = bwd_q(p, dtype, need_state ? 0 : 1, s)) != cudaSuccess) return LA_ERR_CUDA;
    FwdParams pr = p;           // suffix sums: scan of the bwd_q partials, written to the suffix buffer
    pr.prefix = p.suffix;
    pr.reverse = 1;
    pr.keep_last = 1;
    if ((e = launch_scan(pr, s)) != cudaSuccess) return LA_ERR_CUDA;
    if ((e = bwd_kv(p, dtype, s)) != cudaSuccess) return LA_ERR_CUDA;
    return LA_OK;
}

size_t backward_workspace_bytes(int causal, int map, int dtype, int has_cu, int nseq, int64_t T, int H, int dk,
                                int dv, int r) {
    (void)causal;
    if (check_dims(map, dtype, nseq, T, H, dk, dv, r, has_cu != 0) != LA_OK) return 0;
    if (bwd_smem_bytes(dk, dv, r) > kSmemLimitBytes) return 0;
    const int nsm = device_sm_count();
    if (nsm <= 0) return 0;
    return make_layout(kPathSimt, has_cu != 0, nseq, T, H, dv, r, nsm, true).total;
}

}  // namespace

la_status forward_entry(int causal, int phase_lo, int phase_hi, const void* q, const void* k, const void* v,
                        const float* omega, int map, int dtype, const int32_t* cu_seqlens, int nseq, int64_t T,
                        int H, int dk, int dv, int r, float eps, void* out, void* workspace,
                        size_t workspace_bytes, void* stream, int* launched) {
    return forward(causal, phase_lo, phase_hi, q, k, v, omega, map, dtype, cu_seqlens, nseq, T, H, dk, dv, r, eps,
                   out, workspace, workspace_bytes, stream, launched, LA_NORM_ATTENTION, nullptr, nullptr);
}

}  // namespace la

using namespace la;

extern "C" {

la_status la_feature_map(const void* x, const float* omega, int map, int dtype, int64_t T, int H, int d,
                         int r, float* phi, void* stream) {
    la_status st = check_dims(map, dtype, 1, T, H, d, 1, r, true);
    if (st != LA_OK) return st;
    if (map == LA_MAP_FAVOR && omega == nullptr) return LA_ERR_INVALID_ARG;
    if (T == 0) return LA_OK;
    if (!x || !phi) return LA_ERR_INVALID_ARG;
    const size_t esz = dtype == LA_F32 ? 4 : 2;
    if (!aligned(x, esz) || !aligned(phi, 4) || (omega && !aligned(omega, 4))) return LA_ERR_INVALID_ARG;
    cudaError_t e;
    if (dtype == LA_BF16 && map == LA_MAP_FAVOR && tc_supported(map, d, d, r, 1) && aligned(x, 16) &&
        aligned(omega, 16) && aligned(phi, 16)) {
        // same projection and exponent as the forward's tensor-core path, before the bf16 rounding
        e = tc_feature_map(x, omega, T, H, r, phi, nullptr, static_cast<cudaStream_t>(stream));
    } else {
        if (simt_fmap_smem_bytes(map, d, r) > kSmemLimitBytes) return LA_ERR_UNSUPPORTED;
        e = simt_feature_map(x, omega, map, dtype, T, H, d, r, phi, static_cast<cudaStream_t>(stream));
    }
    return e == cudaSuccess ? LA_OK : LA_ERR_CUDA;
}

la_status la_forward_bidir(const void* q, const void* k, const void* v, const float* omega, int map, int dtype,
                           const int32_t* cu_seqlens, int nseq, int64_t T, int H, int d_k, int d_v, int r,
                           float eps, void* out, void* workspace, size_t workspace_bytes, void* stream) {
    return forward(0, LA_PHASE_PLAN, LA_PHASE_OUTPUT, q, k, v, omega, map, dtype, cu_seqlens, nseq, T, H, d_k,
                   d_v, r, eps, out, workspace, workspace_bytes, stream, nullptr);
}

la_status la_forward_causal(const void* q, const void* k, const void* v, const float* omega, int map, int dtype,
                            const int32_t* cu_seqlens, int nseq, int64_t T, int H, int d_k, int d_v, int r,
                            float eps, void* out, void* workspace, size_t workspace_bytes, void* stream) {
    return forward(1, LA_PHASE_PLAN, LA_PHASE_OUTPUT, q, k, v, omega, map, dtype, cu_seqlens, nseq, T, H, d_k,
                   d_v, r, eps, out, workspace, workspace_bytes, stream, nullptr);
}

la_status la_forward_phase(int causal, int phase, int norm, const void* q, const void* k, const void* v,
                           const float* omega, int map, int dtype, const int32_t* cu_seqlens, int nseq, int64_t T,
                           int H, int d_k, int d_v, int r, float eps, const float* state_in, float* state_out,
                           void* out, void* workspace, size_t workspace_bytes, void* stream, int* launched) {
    if (phase < LA_PHASE_PLAN || phase > LA_PHASE_OUTPUT) return LA_ERR_INVALID_ARG;
    return forward(causal != 0, phase, phase, q, k, v, omega, map, dtype, cu_seqlens, nseq, T, H, d_k, d_v, r,
                   eps, out, workspace, workspace_bytes, stream, launched, norm, state_in, state_out);
}

la_status la_forward(int causal, int norm, const void* q, const void* k, const void* v, const float* omega,
                     int map, int dtype, const int32_t* cu_seqlens, int nseq, int64_t T, int H, int d_k, int d_v,
                     int r, float eps, const float* state_in, float* state_out, void* out, void* workspace,
                     size_t workspace_bytes, void* stream) {
    return forward(causal != 0, LA_PHASE_PLAN, LA_PHASE_OUTPUT, q, k, v, omega, map, dtype, cu_seqlens, nseq, T,
                   H, d_k, d_v, r, eps, out, workspace, workspace_bytes, stream, nullptr, norm, state_in,
                   state_out);
}

la_status la_decode_step(const void* q, const void* k, const void* v, const float* omega, int map, int dtype,
                         int norm, int B, int H, int d_k, int d_v, int r, float eps, float* state, void* out,
                         void* stream) {
    if (B < 0) return LA_ERR_INVALID_ARG;
    la_status st = check_dims(map, dtype, 1, B, H, d_k, d_v, r, true);
    if (st != LA_OK) return st;
    if ((st = check_norm(norm, map)) != LA_OK) return st;
    if (!(eps >= 0.f) || !std::isfinite(eps)) return LA_ERR_INVALID_ARG;
    if (map == LA_MAP_FAVOR && omega == nullptr) return LA_ERR_INVALID_ARG;
    if (B == 0) return LA_OK;
    if (!q || !k || !v || !out || !state) return LA_ERR_INVALID_ARG;
    const size_t esz = dtype == LA_F32 ? 4 : 2;
    if (!aligned(q, esz) || !aligned(k, esz) || !aligned(v, esz) || !aligned(out, esz) || !aligned(state, 4) ||
        (omega && !aligned(omega, 4)))
        return LA_ERR_INVALID_ARG;
    if (decode_smem_bytes(d_k, d_v, r) > kSmemLimitBytes) return LA_ERR_UNSUPPORTED;
    const cudaError_t e = decode_step(q, k, v, omega, map, dtype, norm, B, H, d_k, d_v, r, eps, state, out,
                                      static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? LA_OK : LA_ERR_CUDA;
}

la_status la_backward(int causal, int norm, const void* q, const void* k, const void* v, const float* omega, int map,
                      int dtype, const int32_t* cu_seqlens, int nseq, int64_t T, int H, int d_k, int d_v, int r,
                      float eps, const void* dout, void* dq, void* dk, void* dv, void* workspace,
                      size_t workspace_bytes, void* stream) {
    return backward(causal != 0, norm, q, k, v, omega, map, dtype, cu_seqlens, nseq, T, H, d_k, d_v, r, eps, dout,
                    dq, dk, dv, workspace, workspace_bytes, stream);
}

size_t la_backward_workspace_bytes(int causal, int map, int dtype, int has_cu_seqlens, int nseq, int64_t T, int H,
                                   int d_k, int d_v, int r) {
    return backward_workspace_bytes(causal, map, dtype, has_cu_seqlens, nseq, T, H, d_k, d_v, r);
}

size_t la_workspace_bytes(int causal, int map, int dtype, int has_cu_seqlens, int nseq, int64_t T, int H,
                          int d_k, int d_v, int r) {
    if (check_dims(map, dtype, nseq, T, H, d_k, d_v, r, has_cu_seqlens != 0) != LA_OK) return 0;
    const int path = select_path(causal, map, dtype, d_k, d_v, r);
    if (path_supported(path, map, d_k, d_v, r) != LA_OK) return 0;
    const int nsm = device_sm_count();
    if (nsm <= 0) return 0;
    size_t bytes = make_layout(path, has_cu_seqlens != 0, nseq, T, H, d_v, r, nsm, false,
                               whole_sequences(path, map), vtables(path, causal, map)).total;
    // sum normalisation and unaligned operands move a tensor-core call to the
    // CUDA-core kernels: the size covers both
    if (path == kPathTensor && path_supported(kPathSimt, map, d_k, d_v, r) == LA_OK)
        bytes = std::max(bytes, make_layout(kPathSimt, has_cu_seqlens != 0, nseq, T, H, d_v, r, nsm).total);
    return bytes;
}

la_status la_check_cu_seqlens(const int32_t* cu_seqlens, int nseq, int64_t T, void* stream) {
    if (cu_seqlens == nullptr || nseq < 1 || T < 0) return LA_ERR_INVALID_ARG;
    std::vector<int32_t> h((size_t)nseq + 1);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(h.data(), cu_seqlens, sizeof(int32_t) * h.size(), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return LA_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return LA_ERR_CUDA;
    if (h[0] != 0 || (int64_t)h[nseq] != T) return LA_ERR_INVALID_ARG;
    for (int i = 0; i < nseq; ++i)
        if (h[i + 1] < h[i]) return LA_ERR_INVALID_ARG;
    return LA_OK;
}

la_status la_workspace_error(const void* workspace, int* code, void* stream) {
    if (workspace == nullptr) return LA_ERR_INVALID_ARG;
    int words[3] = {0, 0, 0};   // WsHeader: error, n_units, range
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(words, workspace, sizeof(words), cudaMemcpyDeviceToHost, s) != cudaSuccess) return LA_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return LA_ERR_CUDA;
    const int err = words[0] != LA_DEVERR_NONE ? words[0] : (words[2] != 0 ? LA_DEVERR_RANGE : LA_DEVERR_NONE);
    if (code) *code = err;
    return err == LA_DEVERR_NONE ? LA_OK : LA_ERR_DEVICE;
}

la_status la_test_force_wait_timeout(int enable) {
    return la::tc_force_wait_timeout(enable ? 1 : 0) == cudaSuccess ? LA_OK : LA_ERR_CUDA;
}

int64_t la_test_segment_plan(int64_t nchunks, int64_t pairs, int nsm, int64_t force_chunks, int64_t* makespan) {
    if (nchunks < 1 || pairs < 1 || nsm < 1) return -1;
    const int64_t lc = force_chunks > 0 ? force_chunks : tensor_segment_chunks(nchunks, pairs, nsm);
    if (makespan) {
        *makespan = 0;
        if (lc > 0) {
            const int64_t segs = ceil_div(nchunks, lc);
            *makespan = block_makespan((segs - 1) * pairs, lc, pairs, nchunks - (segs - 1) * lc, nsm);
        }
    }
    return lc;
}

la_status la_orthogonal_features(const double* gauss_blocks, const double* gauss_lengths, int r, int d,
                                 float* omega, void* stream) {
    if (!gauss_blocks || !gauss_lengths || !omega) return LA_ERR_INVALID_ARG;
    if (r < 1 || d < 1) return LA_ERR_INVALID_ARG;
    if (d > 128 || r > LA_MAX_R) return LA_ERR_UNSUPPORTED;
    cudaError_t e = orf_build(gauss_blocks, gauss_lengths, r, d, omega, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? LA_OK : LA_ERR_CUDA;
}

int la_selected_path(int causal, int map, int dtype, int d_k, int d_v, int r) {
    if (check_dims(map, dtype, 1, 0, 1, d_k, d_v, r, true) != LA_OK) return -1;
    const int path = select_path(causal, map, dtype, d_k, d_v, r);
    if (path_supported(path, map, d_k, d_v, r) != LA_OK) return -1;
    return path;
}

const char* la_status_string(la_status status) {
    switch (status) {
        case LA_OK: return "ok";
        case LA_ERR_INVALID_ARG: return "invalid argument";
        case LA_ERR_UNSUPPORTED: return "unsupported size";
        case LA_ERR_WORKSPACE: return "workspace too small";
        case LA_ERR_CUDA: return "CUDA error";
        case LA_ERR_DEVICE: return "device-side error recorded in the workspace";
    }
    return "unknown status";
}

int la_version(void) { return 200; }

}  // extern "C"
