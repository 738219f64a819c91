// Host-side launchers of the device kernels (internal to the library).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "linattn.h"

namespace la {

// The attention launchers take `fm`, the feature map (the la_phi values:
// kPhiElu1 or kPhiIdentity, defined in common.cuh).

// fp32-arithmetic SIMT paths (any 1 <= D, M <= 128, either dtype).
size_t simt_causal_workspace(int64_t BH, int N, int D, int M);
size_t simt_noncausal_workspace(int64_t BH, int N, int D, int M);
int simt_noncausal_splits(int64_t BH, int N);
// S0, z0: initial state [BH, D, M] and [BH, D] (fp32, both or neither; null = zero).
cudaError_t simt_causal(const void* q, const void* k, const void* v, void* o, la_dtype dt,
                        int64_t BH, int N, int D, int M, float eps, int fm, const float* S0,
                        const float* z0, float* S_out, float* z_out, void* scratch,
                        cudaStream_t st);
// Causal or non-causal backward (fp32 arithmetic, D, M <= kBwdMaxDim): dq, dk,
// dv from dout.
constexpr int kBwdMaxDim = 64;
size_t simt_bwd_workspace(int64_t BH, int N, int D, int M);
cudaError_t simt_bwd(const void* q, const void* k, const void* v, const void* dout, void* dq,
                     void* dk, void* dv, la_dtype dt, bool causal, int64_t BH, int N, int D, int M,
                     float eps, int fm, void* scratch, cudaStream_t st);
cudaError_t simt_noncausal(const void* q, const void* k, const void* v, void* o, la_dtype dt,
                           int64_t BH, int N, int D, int M, float eps, int fm, void* scratch,
                           cudaStream_t st);

// Positive random features exp(W x - |x|^2 / 2 - shift) / sqrt(R) (SIMT, fp32
// arithmetic; D <= 128).
cudaError_t simt_random_features(const void* x, const void* W, void* out, la_dtype dt,
                                 int64_t rows, int D, int R, float shift, cudaStream_t st);

// Positive random features on the tensor cores: bf16, D = R = 64.
bool tc_random_features_supported(int D, int R, la_dtype dt);
cudaError_t tc_random_features(const void* x, const void* W, void* out, int64_t rows, float shift,
                               cudaStream_t st);

// Tensor-core (tcgen05) causal path: bf16, Dk = Dv = 64 (one fused launch,
// causal_tc.cu) or 128 (run sums, seed scan, output pass: causal128_tc.cu).
bool tc_causal_supported(int D, int M, la_dtype dt);
size_t tc_causal_workspace(int64_t BH, int N, int D);
int tc_causal_launches(int D, int64_t BH, int N);
cudaError_t tc_causal(const void* q, const void* k, const void* v, void* o, int64_t BH, int N,
                      int D, float eps, int fm, const float* S0, const float* z0, float* S_out,
                      float* z_out, void* ws_header, void* scratch, cudaStream_t st);
// Per-run sums S_run = phi(K)^T V (Dk = Dv = 128, fp32, feature rows) and z_run
// over the persistent chunk partition of (BH, N), one slot of D * D + D floats
// per (CTA, run) at agg + (cta * maxr + run) * (D * D + D); with last_only, only
// each range's last run when its head continues, at agg + cta * (D * D + D)
// (noncausal_tc.cu).
cudaError_t tc_run_sums128(const void* k, const void* v, float* agg, int64_t BH, int N, int fm,
                           bool last_only, void* ws_header, cudaStream_t st);
size_t tc_causal128_workspace(int64_t BH, int N);
int tc_causal128_launches(int64_t BH, int N);
cudaError_t tc_causal128(const void* q, const void* k, const void* v, void* o, int64_t BH, int N,
                         float eps, int fm, const float* S0, const float* z0, float* S_out,
                         float* z_out, void* ws_header, void* scratch, cudaStream_t st);

// Tensor-core (tcgen05) non-causal path: bf16, Dk = Dv = 64 or 128.
bool tc_noncausal_supported(int D, int M, la_dtype dt);
size_t tc_noncausal_workspace(int64_t BH, int N, int D);
cudaError_t tc_noncausal(const void* q, const void* k, const void* v, void* o, int64_t BH, int N,
                         int D, float eps, int fm, void* ws_header, void* scratch, cudaStream_t st);

// Decode step (SIMT, bandwidth bound).
cudaError_t decode_step(const void* q, const void* k, const void* v, void* o, float* S, float* z,
                        la_dtype dt, int64_t BH, int D, int M, float eps, int fm,
                        cudaStream_t st);
// The same step with q, k of head h = b H + j at b ld_qk + j D and v at
// b ld_v + j M (o stays contiguous [BH, M]).
cudaError_t decode_step_strided(const void* q, const void* k, const void* v, void* o, float* S,
                                float* z, la_dtype dt, int64_t BH, int D, int M, float eps, int fm,
                                int H, int64_t ld_qk, int64_t ld_v, cudaStream_t st);

// Scans of the tensor-core backward (csrc/simt.cu), in place over per-chunk
// sums: the reverse exclusive sum (causal) or total (non-causal).
cudaError_t bwd_reverse_sums(float* rstates, bool causal, int64_t BH, int nchunks, int E,
                             cudaStream_t st);
// The exclusive prefix (causal) or total (non-causal) of per-chunk states in place.
cudaError_t bwd_prefix_states(float* states, bool causal, int64_t BH, int nchunks, int D, int M,
                              cudaStream_t st);

// Tensor-core backward (csrc/bwd_tc.cu): bf16, Dk = Dv = 64; same workspace as
// the fp32 backward (simt_bwd_workspace).
bool tc_bwd_supported(int D, int M, la_dtype dt);
cudaError_t tc_bwd(const void* q, const void* k, const void* v, const void* dout, void* dq,
                   void* dk, void* dv, bool causal, int64_t BH, int N, float eps, int fm,
                   void* ws_header, void* scratch, cudaStream_t st);

// Layer decode step (csrc/layer.cu): workspace bytes after the header.
size_t layer_workspace(int B, int H, int D, la_dtype dt);

// Y = X W, row-major X [rows, K], W [K, N], Y [rows, N], fp32 accumulation
// (csrc/gemm.cu): tcgen05 for bf16 with K, N multiples of 8, fp32 FMA otherwise.
// A bounded wait that runs out is recorded in the header at ws_header.
bool gemm_uses_tensor_cores(int K, int N, la_dtype dt);
cudaError_t gemm(const void* X, const void* W, void* Y, int rows, int K, int N, la_dtype dt,
                 void* ws_header, cudaStream_t st);

}  // namespace la
