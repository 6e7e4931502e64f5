// Launchers shared between the translation units of liblinattn.so.
#pragma once

#include "common.cuh"

namespace la {

// Work planning (plan.cu): fills the unit table and sequence index from
// cu_seqlens (or equal lengths), clears the error word.
cudaError_t launch_plan(const FwdParams& p, cudaStream_t s);
// Combines per-unit partial states into the state each unit starts from:
// exclusive prefix over the sequence's units (causal) or the whole-sequence
// sum (bidirectional).  Fixed summation order.
cudaError_t launch_scan(const FwdParams& p, cudaStream_t s);

// fp32 CUDA-core path (simt.cu).
size_t simt_smem_bytes(int map, int dk, int dv, int r);
size_t simt_fmap_smem_bytes(int map, int d, int r);
constexpr size_t kSmemLimitBytes = 227 * 1024;
int simt_chunk();
cudaError_t simt_feature_map(const void* x, const float* omega, int map, int dtype,
                             int64_t T, int H, int d, int r, float* phi, cudaStream_t s);
cudaError_t simt_state(const FwdParams& p, int dtype, cudaStream_t s);
cudaError_t simt_out(const FwdParams& p, int dtype, int prefix_is_zero, cudaStream_t s);

// The forward dispatcher behind the C entry points (api.cu): phases
// phase_lo..phase_hi of a bidirectional (causal = 0) or causal call.
la_status forward_entry(int causal, int phase_lo, int phase_hi, const void* q, const void* k, const void* v,
                        const float* omega, int map, int dtype, const int32_t* cu_seqlens, int nseq, int64_t T,
                        int H, int dk, int dv, int r, float eps, void* out, void* workspace,
                        size_t workspace_bytes, void* stream, int* launched);

// tcgen05 tensor-core path (tc.cu): bf16, d_k = d_v = 64, r in {64, 128, 256}
// (FAVOR+), r = 64 (ELU+1, identity) or, causal only, r in {128, 256}
// (DPFP-1, -2: whole sequences per unit, state pass on CUDA cores); 16-byte
// aligned operands.
bool tc_supported(int map, int dk, int dv, int r, int causal);
// Test hook behind la_test_force_wait_timeout: sets the causal output kernel's flag on the
// current device.
cudaError_t tc_force_wait_timeout(int enable);
cudaError_t tc_state(const FwdParams& p, cudaStream_t s);
cudaError_t tc_out(const FwdParams& p, int prefix_is_zero, cudaStream_t s);
cudaError_t tc_feature_map(const void* x, const float* omega, int64_t T, int H, int r, float* phi, int* err,
                           cudaStream_t s);
// sums[t][h] = sum_f phi_f(x_th) for the FAVOR+ map (same projection and exponent as tc_feature_map)
cudaError_t tc_feature_sums(const void* x, const float* omega, int64_t T, int H, int r, float* sums, int* err,
                            cudaStream_t s);

// Sum normalisation on the tensor-core path (norm.cu): out = phi(q)^T S' / max(sigma_q, eps) with
// S' built from v / max(sigma_k, eps), sigma = sum_f phi_f; the output kernels divide (p.div_rows).
cudaError_t sum_scale_values(const void* v, const float* sigma_k, float eps, int64_t T, int H, int dv, void* dst,
                             cudaStream_t s);
// element-wise maps, d_k = d_v = 64: sigma_q into sig_q and v / max(sigma_k, eps) into dst in one pass
cudaError_t sum_prologue_elementwise(const void* q, const void* k, const void* v, int map, int64_t T, int H, int r,
                                     float eps, float* sig_q, void* dst, cudaStream_t s);

// Backward pass on CUDA cores (bwd.cu): bwd_q writes g, dq and each unit's
// sum of phi(q) g^T (p.partial); bwd_kv writes dk, dv from p.suffix.
size_t bwd_smem_bytes(int dk, int dv, int r);
cudaError_t bwd_q(const FwdParams& p, int dtype, int prefix_is_zero, cudaStream_t s);
cudaError_t bwd_kv(const FwdParams& p, int dtype, cudaStream_t s);
cudaError_t bwd_transpose_omega(const FwdParams& p, cudaStream_t s);   // p.omega [r][dk] -> p.omega_t [dk][r]

// One-token decode step on CUDA cores (decode.cu).
size_t decode_smem_bytes(int dk, int dv, int r);
cudaError_t decode_step(const void* q, const void* k, const void* v, const float* omega, int map, int dtype,
                        int norm, int B, int H, int dk, int dv, int r, float eps, float* state, void* out,
                        cudaStream_t s);

// Orthogonal random features (orf.cu).
cudaError_t orf_build(const double* blocks, const double* lengths, int r, int d, float* omega,
                      cudaStream_t s);

}  // namespace la
