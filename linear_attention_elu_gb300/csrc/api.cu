// C-ABI entry points (declared in include/linattn.h): argument checks,
// workspace layout, path choice and launches. No entry point allocates
// device memory; every buffer belongs to the caller.
#include <math.h>

#include "common.cuh"
#include "kernels.h"

using la::WsHeader;

namespace {

constexpr size_t kHeaderBytes = sizeof(WsHeader);

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

la_status check_common(int B, int H, int N, int Dk, int Dv, la_dtype dt) {
    if (B < 0 || H < 0 || N < 0) return LA_ERR_INVALID_ARG;
    if (dt != LA_F32 && dt != LA_BF16) return LA_ERR_INVALID_ARG;
    if (Dk <= 0 || Dv <= 0) return LA_ERR_INVALID_ARG;
    if (Dk > la::kMaxDim || Dv > la::kMaxDim) return LA_ERR_UNSUPPORTED;
    if ((int64_t)B * H > 65535) return LA_ERR_UNSUPPORTED;  // heads map to grid.y
    return LA_OK;
}

la_status check_tensor(const void* p, int64_t elems, la_dtype dt) {
    if (elems == 0) return LA_OK;
    if (!p) return LA_ERR_INVALID_ARG;
    if (!aligned(p, 16)) return LA_ERR_INVALID_ARG;
    (void)dt;
    return LA_OK;
}

la_status check_eps(float eps) {
    return (isfinite(eps) && eps >= 0.f) ? LA_OK : LA_ERR_INVALID_ARG;
}

size_t body_bytes(la_op op, int B, int H, int N, int Dk, int Dv, la_dtype dt) {
    const int64_t BH = (int64_t)B * H;
    if (BH == 0 || N == 0) return 0;
    switch (op) {
        case LA_OP_CAUSAL:
            if (la::tc_causal_supported(Dk, Dv, dt)) return la::tc_causal_workspace(BH, N, Dk);
            return la::simt_causal_workspace(BH, N, Dk, Dv);
        case LA_OP_NONCAUSAL:
            if (la::tc_noncausal_supported(Dk, Dv, dt)) return la::tc_noncausal_workspace(BH, N, Dk);
            return la::simt_noncausal_workspace(BH, N, Dk, Dv);
        case LA_OP_CAUSAL_BWD:
        case LA_OP_NONCAUSAL_BWD:
            return la::simt_bwd_workspace(BH, N, Dk, Dv);
        case LA_OP_LAYER_DECODE:
            return la::layer_workspace(B, H, Dk, dt);
        default:
            return 0;
    }
}

la_status check_workspace(void* ws, size_t have, size_t need) {
    if (need == 0) return LA_OK;
    if (!ws || !aligned(ws, 256) || have < need) return LA_ERR_WORKSPACE;
    return LA_OK;
}

la_status from_cuda(cudaError_t e) { return e == cudaSuccess ? LA_OK : LA_ERR_CUDA; }

__global__ void init_header_kernel(WsHeader* h) { la::init_header(h); }

}  // namespace

namespace {

bool overlaps(const void* a, size_t an, const void* b, size_t bn) {
    if (!a || !b || an == 0 || bn == 0) return false;
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + bn && y < x + an;
}

static_assert(LA_PHI_ELU1 == la::kPhiElu1 && LA_PHI_IDENTITY == la::kPhiIdentity,
              "la_phi values are the kernels' feature-map codes");

bool valid_phi(la_phi phi) { return phi == LA_PHI_ELU1 || phi == LA_PHI_IDENTITY; }

la_status causal_fwd(const void* q, const void* k, const void* v, void* o, int B, int H, int N,
                     int Dk, int Dv, la_dtype dt, la_phi phi, float eps, const float* S0,
                     const float* z0, float* S_out, float* z_out, void* workspace,
                     size_t workspace_bytes, la_stream_t stream) {
    la_status s = check_common(B, H, N, Dk, Dv, dt);
    if (s != LA_OK) return s;
    if ((s = check_eps(eps)) != LA_OK) return s;
    if (!valid_phi(phi)) return LA_ERR_INVALID_ARG;
    const int64_t BH = (int64_t)B * H;
    const int64_t rows = BH * N;
    if ((s = check_tensor(q, rows * Dk, dt)) || (s = check_tensor(k, rows * Dk, dt)) ||
        (s = check_tensor(v, rows * Dv, dt)) || (s = check_tensor(o, rows * Dv, dt)))
        return s;
    if ((S_out && !aligned(S_out, 16)) || (z_out && !aligned(z_out, 16)))
        return LA_ERR_INVALID_ARG;
    // The initial state: both parts or neither, aligned, and not overwritten by
    // the final state while other CTAs may still read it.
    const size_t s_bytes = sizeof(float) * (size_t)BH * Dk * Dv, z_bytes = sizeof(float) * (size_t)BH * Dk;
    if ((S0 == nullptr) != (z0 == nullptr)) return LA_ERR_INVALID_ARG;
    if (S0 && BH > 0 && (!aligned(S0, 16) || !aligned(z0, 16) ||
                         overlaps(S0, s_bytes, S_out, s_bytes) || overlaps(S0, s_bytes, z_out, z_bytes) ||
                         overlaps(z0, z_bytes, S_out, s_bytes) || overlaps(z0, z_bytes, z_out, z_bytes)))
        return LA_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    if (BH == 0) return LA_OK;
    if (N == 0) {
        // Empty sequence: the final state is the initial one (zero when absent).
        if (S_out && (S0 ? cudaMemcpyAsync(S_out, S0, s_bytes, cudaMemcpyDeviceToDevice, st)
                         : cudaMemsetAsync(S_out, 0, s_bytes, st)))
            return LA_ERR_CUDA;
        if (z_out && (z0 ? cudaMemcpyAsync(z_out, z0, z_bytes, cudaMemcpyDeviceToDevice, st)
                         : cudaMemsetAsync(z_out, 0, z_bytes, st)))
            return LA_ERR_CUDA;
        return LA_OK;
    }
    const size_t need = kHeaderBytes + body_bytes(LA_OP_CAUSAL, B, H, N, Dk, Dv, dt);
    if ((s = check_workspace(workspace, workspace_bytes, need)) != LA_OK) return s;
    char* body = (char*)workspace + kHeaderBytes;
    if (la::tc_causal_supported(Dk, Dv, dt))
        return from_cuda(
            la::tc_causal(q, k, v, o, BH, N, Dk, eps, phi, S0, z0, S_out, z_out, workspace, body, st));
    return from_cuda(la::simt_causal(q, k, v, o, dt, BH, N, Dk, Dv, eps, phi, S0, z0, S_out, z_out,
                                     body, st));
}

}  // namespace

extern "C" {

const char* la_status_string(la_status s) {
    switch (s) {
        case LA_OK: return "LA_OK";
        case LA_ERR_INVALID_ARG: return "LA_ERR_INVALID_ARG: invalid argument";
        case LA_ERR_UNSUPPORTED: return "LA_ERR_UNSUPPORTED: shape or dtype not supported";
        case LA_ERR_WORKSPACE: return "LA_ERR_WORKSPACE: workspace missing, too small or misaligned";
        case LA_ERR_CUDA: return "LA_ERR_CUDA: CUDA runtime error";
        case LA_ERR_TIMEOUT: return "LA_ERR_TIMEOUT: a bounded device-side wait expired";
    }
    return "unknown la_status";
}

uint32_t la_version(void) { return (0u << 16) | 1u; }

la_status la_workspace_size(la_op op, int B, int H, int N, int Dk, int Dv, la_dtype dt,
                            size_t* bytes) {
    if (!bytes) return LA_ERR_INVALID_ARG;
    if (op != LA_OP_CAUSAL && op != LA_OP_NONCAUSAL && op != LA_OP_DECODE &&
        op != LA_OP_CAUSAL_BWD && op != LA_OP_NONCAUSAL_BWD && op != LA_OP_LAYER_DECODE)
        return LA_ERR_INVALID_ARG;
    const bool one_token = op == LA_OP_DECODE || op == LA_OP_LAYER_DECODE;
    la_status s = check_common(B, H, one_token ? 1 : N, Dk, Dv, dt);
    if (s != LA_OK) return s;
    if (op == LA_OP_LAYER_DECODE) {
        if (Dk != Dv) return LA_ERR_UNSUPPORTED;
        *bytes = kHeaderBytes + round_up(body_bytes(op, B, H, 1, Dk, Dv, dt), 256);
        return LA_OK;
    }
    if (op == LA_OP_DECODE) {
        *bytes = 0;
        return LA_OK;
    }
    if ((op == LA_OP_CAUSAL_BWD || op == LA_OP_NONCAUSAL_BWD) &&
        (Dk > la::kBwdMaxDim || Dv > la::kBwdMaxDim))
        return LA_ERR_UNSUPPORTED;
    *bytes = kHeaderBytes + round_up(body_bytes(op, B, H, N, Dk, Dv, dt), 256);
    return LA_OK;
}

la_status la_launch_count(la_op op, int B, int H, int N, int Dk, int Dv, la_dtype dt,
                          int* launches) {
    if (!launches) return LA_ERR_INVALID_ARG;
    if (op != LA_OP_CAUSAL && op != LA_OP_NONCAUSAL && op != LA_OP_DECODE &&
        op != LA_OP_CAUSAL_BWD && op != LA_OP_NONCAUSAL_BWD && op != LA_OP_LAYER_DECODE)
        return LA_ERR_INVALID_ARG;
    const bool one_token = op == LA_OP_DECODE || op == LA_OP_LAYER_DECODE;
    la_status s = check_common(B, H, one_token ? 1 : N, Dk, Dv, dt);
    if (s != LA_OK) return s;
    const int64_t BH = (int64_t)B * H;
    if (BH == 0 || (!one_token && N == 0)) {
        *launches = 0;
        return LA_OK;
    }
    if (op == LA_OP_LAYER_DECODE)
        *launches = 3;                           // two projections and the decode step
    else if (one_token)
        *launches = 1;
    else if (op == LA_OP_CAUSAL_BWD || op == LA_OP_NONCAUSAL_BWD)
        *launches = 5;
    else if (op == LA_OP_CAUSAL && la::tc_causal_supported(Dk, Dv, dt))
        *launches = la::tc_causal_launches(Dk, (int64_t)B * H, N);
    else if (op == LA_OP_NONCAUSAL && la::tc_noncausal_supported(Dk, Dv, dt))
        *launches = 2;
    else
        *launches = 3;
    return LA_OK;
}

la_status la_workspace_init(void* workspace, size_t workspace_bytes, la_stream_t stream) {
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < kHeaderBytes)
        return LA_ERR_WORKSPACE;
    // The body is cleared too: kernels that publish tagged words across CTAs
    // trust a word only when it carries the current launch's tag.
    cudaError_t e = cudaMemsetAsync(workspace, 0, workspace_bytes, (cudaStream_t)stream);
    if (e != cudaSuccess) return LA_ERR_CUDA;
    init_header_kernel<<<1, 1, 0, (cudaStream_t)stream>>>((WsHeader*)workspace);
    return from_cuda(cudaPeekAtLastError());
}

la_status la_noncausal_fwd(const void* q, const void* k, const void* v, void* o, int B, int H,
                           int N, int Dk, int Dv, la_dtype dt, float eps, void* workspace,
                           size_t workspace_bytes, la_stream_t stream) {
    return la_noncausal_fwd_phi(q, k, v, o, B, H, N, Dk, Dv, dt, LA_PHI_ELU1, eps, workspace,
                                workspace_bytes, stream);
}

la_status la_noncausal_fwd_phi(const void* q, const void* k, const void* v, void* o, int B,
                               int H, int N, int Dk, int Dv, la_dtype dt, la_phi phi, float eps,
                               void* workspace, size_t workspace_bytes, la_stream_t stream) {
    la_status s = check_common(B, H, N, Dk, Dv, dt);
    if (s != LA_OK) return s;
    if ((s = check_eps(eps)) != LA_OK) return s;
    if (!valid_phi(phi)) return LA_ERR_INVALID_ARG;
    const int64_t BH = (int64_t)B * H;
    const int64_t rows = BH * N;
    if ((s = check_tensor(q, rows * Dk, dt)) || (s = check_tensor(k, rows * Dk, dt)) ||
        (s = check_tensor(v, rows * Dv, dt)) || (s = check_tensor(o, rows * Dv, dt)))
        return s;
    if (rows == 0) return LA_OK;
    const size_t need = kHeaderBytes + body_bytes(LA_OP_NONCAUSAL, B, H, N, Dk, Dv, dt);
    if ((s = check_workspace(workspace, workspace_bytes, need)) != LA_OK) return s;
    char* body = (char*)workspace + kHeaderBytes;
    if (la::tc_noncausal_supported(Dk, Dv, dt))
        return from_cuda(la::tc_noncausal(q, k, v, o, BH, N, Dk, eps, phi, workspace, body,
                                          (cudaStream_t)stream));
    return from_cuda(la::simt_noncausal(q, k, v, o, dt, BH, N, Dk, Dv, eps, phi, body,
                                        (cudaStream_t)stream));
}

la_status la_causal_fwd(const void* q, const void* k, const void* v, void* o, int B, int H,
                        int N, int Dk, int Dv, la_dtype dt, float eps, float* S_out,
                        float* z_out, void* workspace, size_t workspace_bytes,
                        la_stream_t stream) {
    return causal_fwd(q, k, v, o, B, H, N, Dk, Dv, dt, LA_PHI_ELU1, eps, nullptr, nullptr, S_out,
                      z_out, workspace, workspace_bytes, stream);
}

la_status la_causal_fwd_state(const void* q, const void* k, const void* v, void* o, int B,
                              int H, int N, int Dk, int Dv, la_dtype dt, float eps,
                              const float* S0, const float* z0, float* S_out, float* z_out,
                              void* workspace, size_t workspace_bytes, la_stream_t stream) {
    return causal_fwd(q, k, v, o, B, H, N, Dk, Dv, dt, LA_PHI_ELU1, eps, S0, z0, S_out, z_out,
                      workspace, workspace_bytes, stream);
}

la_status la_causal_fwd_phi(const void* q, const void* k, const void* v, void* o, int B, int H,
                            int N, int Dk, int Dv, la_dtype dt, la_phi phi, float eps,
                            const float* S0, const float* z0, float* S_out, float* z_out,
                            void* workspace, size_t workspace_bytes, la_stream_t stream) {
    return causal_fwd(q, k, v, o, B, H, N, Dk, Dv, dt, phi, eps, S0, z0, S_out, z_out, workspace,
                      workspace_bytes, stream);
}

}  // extern "C"

namespace {

la_status backward(bool causal, const void* q, const void* k, const void* v, const void* dout,
                   void* dq, void* dk, void* dv, int B, int H, int N, int Dk, int Dv,
                   la_dtype dt, la_phi phi, float eps, void* workspace, size_t workspace_bytes,
                   la_stream_t stream) {
    la_status s = check_common(B, H, N, Dk, Dv, dt);
    if (s != LA_OK) return s;
    if ((s = check_eps(eps)) != LA_OK) return s;
    if (!valid_phi(phi)) return LA_ERR_INVALID_ARG;
    if (Dk > la::kBwdMaxDim || Dv > la::kBwdMaxDim) return LA_ERR_UNSUPPORTED;
    const int64_t BH = (int64_t)B * H;
    const int64_t rows = BH * N;
    if ((s = check_tensor(q, rows * Dk, dt)) || (s = check_tensor(k, rows * Dk, dt)) ||
        (s = check_tensor(v, rows * Dv, dt)) || (s = check_tensor(dout, rows * Dv, dt)) ||
        (s = check_tensor(dq, rows * Dk, dt)) || (s = check_tensor(dk, rows * Dk, dt)) ||
        (s = check_tensor(dv, rows * Dv, dt)))
        return s;
    if (rows == 0) return LA_OK;
    const la_op op = causal ? LA_OP_CAUSAL_BWD : LA_OP_NONCAUSAL_BWD;
    const size_t need = kHeaderBytes + body_bytes(op, B, H, N, Dk, Dv, dt);
    if ((s = check_workspace(workspace, workspace_bytes, need)) != LA_OK) return s;
    char* body = (char*)workspace + kHeaderBytes;
    if (la::tc_bwd_supported(Dk, Dv, dt))
        return from_cuda(la::tc_bwd(q, k, v, dout, dq, dk, dv, causal, BH, N, eps, phi, workspace,
                                    body, (cudaStream_t)stream));
    return from_cuda(la::simt_bwd(q, k, v, dout, dq, dk, dv, dt, causal, BH, N, Dk, Dv, eps, phi,
                                  body, (cudaStream_t)stream));
}

}  // namespace

extern "C" {

la_status la_causal_bwd(const void* q, const void* k, const void* v, const void* dout,
                        void* dq, void* dk, void* dv, int B, int H, int N, int Dk, int Dv,
                        la_dtype dt, float eps, void* workspace, size_t workspace_bytes,
                        la_stream_t stream) {
    return backward(true, q, k, v, dout, dq, dk, dv, B, H, N, Dk, Dv, dt, LA_PHI_ELU1, eps,
                    workspace, workspace_bytes, stream);
}

la_status la_causal_bwd_phi(const void* q, const void* k, const void* v, const void* dout,
                            void* dq, void* dk, void* dv, int B, int H, int N, int Dk, int Dv,
                            la_dtype dt, la_phi phi, float eps, void* workspace,
                            size_t workspace_bytes, la_stream_t stream) {
    return backward(true, q, k, v, dout, dq, dk, dv, B, H, N, Dk, Dv, dt, phi, eps, workspace,
                    workspace_bytes, stream);
}

la_status la_noncausal_bwd(const void* q, const void* k, const void* v, const void* dout,
                           void* dq, void* dk, void* dv, int B, int H, int N, int Dk, int Dv,
                           la_dtype dt, float eps, void* workspace, size_t workspace_bytes,
                           la_stream_t stream) {
    return backward(false, q, k, v, dout, dq, dk, dv, B, H, N, Dk, Dv, dt, LA_PHI_ELU1, eps,
                    workspace, workspace_bytes, stream);
}

la_status la_noncausal_bwd_phi(const void* q, const void* k, const void* v, const void* dout,
                               void* dq, void* dk, void* dv, int B, int H, int N, int Dk, int Dv,
                               la_dtype dt, la_phi phi, float eps, void* workspace,
                               size_t workspace_bytes, la_stream_t stream) {
    return backward(false, q, k, v, dout, dq, dk, dv, B, H, N, Dk, Dv, dt, phi, eps, workspace,
                    workspace_bytes, stream);
}

la_status la_decode_step(const void* q, const void* k, const void* v, void* o, float* S,
                         float* z, int B, int H, int Dk, int Dv, la_dtype dt, float eps,
                         la_stream_t stream) {
    return la_decode_step_phi(q, k, v, o, S, z, B, H, Dk, Dv, dt, LA_PHI_ELU1, eps, stream);
}

la_status la_decode_step_phi(const void* q, const void* k, const void* v, void* o, float* S,
                             float* z, int B, int H, int Dk, int Dv, la_dtype dt, la_phi phi,
                             float eps, la_stream_t stream) {
    la_status s = check_common(B, H, 1, Dk, Dv, dt);
    if (s != LA_OK) return s;
    if ((s = check_eps(eps)) != LA_OK) return s;
    if (!valid_phi(phi)) return LA_ERR_INVALID_ARG;
    const int64_t BH = (int64_t)B * H;
    if (BH == 0) return LA_OK;
    if ((s = check_tensor(q, BH * Dk, dt)) || (s = check_tensor(k, BH * Dk, dt)) ||
        (s = check_tensor(v, BH * Dv, dt)) || (s = check_tensor(o, BH * Dv, dt)))
        return s;
    if (!S || !z || !aligned(S, 16) || !aligned(z, 4)) return LA_ERR_INVALID_ARG;
    return from_cuda(
        la::decode_step(q, k, v, o, S, z, dt, BH, Dk, Dv, eps, phi, (cudaStream_t)stream));
}

la_status la_positive_random_features(const void* x, const void* W, void* out, int64_t rows,
                                      int D, int R, la_dtype dt, float shift,
                                      la_stream_t stream) {
    if (rows < 0 || D < 1 || D > la::kMaxDim || R < 1 || (int64_t)R > 65535LL * la::kChunk ||
        (dt != LA_F32 && dt != LA_BF16) || !isfinite(shift))
        return LA_ERR_INVALID_ARG;
    if (rows == 0) return LA_OK;
    if ((int64_t)((rows + la::kChunk - 1) / la::kChunk) > 2147483647LL) return LA_ERR_UNSUPPORTED;
    la_status s;
    if ((s = check_tensor(x, rows * D, dt)) || (s = check_tensor(W, (int64_t)R * D, dt)) ||
        (s = check_tensor(out, rows * R, dt)))
        return s;
    if (la::tc_random_features_supported(D, R, dt))
        return from_cuda(la::tc_random_features(x, W, out, rows, shift, (cudaStream_t)stream));
    return from_cuda(la::simt_random_features(x, W, out, dt, rows, D, R, shift,
                                              (cudaStream_t)stream));
}

la_status la_query_status(void* workspace, la_stream_t stream) {
    if (!workspace || !aligned(workspace, 256)) return LA_ERR_WORKSPACE;
    cudaStream_t st = (cudaStream_t)stream;
    uint32_t code = 0;
    if (cudaMemcpyAsync(&code, workspace, sizeof(code), cudaMemcpyDeviceToHost, st))
        return LA_ERR_CUDA;
    if (cudaStreamSynchronize(st)) return LA_ERR_CUDA;
    if (code != 0) {
        if (cudaMemsetAsync(workspace, 0, sizeof(uint32_t), st)) return LA_ERR_CUDA;
        if (cudaStreamSynchronize(st)) return LA_ERR_CUDA;
        return (la_status)code;
    }
    return LA_OK;
}

}  // extern "C"
