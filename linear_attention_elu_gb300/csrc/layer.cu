// One decode step of a linear-attention layer for B sequences:
// [q | k | v] = x Wqkv, one recurrent step per head on (S, z), y = o Wo
// ("Why Replace Attention? The Softmax Bottleneck and the Path to Linear
// Time", section 7.2, steps 1-4; "Transformers Are RNNs: Linear Attention",
// the generation loop carrying only (S, z)).
//
// The two projections are plain dense GEMMs and go to cuBLASLt (fp32
// accumulation; bf16 or fp32 storage), with the caller's workspace and no
// device allocation. The attention step is the library's own decode kernel,
// reading q, k, v straight out of the [B, 3 H D] projection through its row
// stride, so nothing is copied between the three launches. All three run on
// the caller's stream and can be captured in one CUDA graph.
#include <cublasLt.h>

#include <math.h>

#include <map>
#include <mutex>
#include <tuple>

#include "common.cuh"
#include "kernels.h"

namespace la {

namespace {

constexpr int kMaxDevices = 128;
constexpr size_t kLtWorkspace = 4u << 20;   // cuBLASLt scratch inside the caller's workspace

size_t elem(la_dtype dt) { return dt == LA_BF16 ? 2 : 4; }
size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// A planned product Y = X W for row-major X [rows, K], W [K, N], Y [rows, N]:
// in cuBLASLt's column-major terms Y^T (N x rows) = W^T (N x K) X^T (K x rows),
// with W^T, X^T and Y^T the row-major arrays as they lie in memory.
struct Plan {
    cublasLtMatmulDesc_t op = nullptr;
    cublasLtMatrixLayout_t w = nullptr, x = nullptr, y = nullptr;
    cublasLtMatmulAlgo_t algo;
};

struct Device {
    std::mutex mu;
    cublasLtHandle_t handle = nullptr;
    std::map<std::tuple<int, int, int, int>, Plan> plans;   // (rows, K, N, dtype)
};
Device g_dev[kMaxDevices];

cublasStatus_t make_plan(cublasLtHandle_t h, int rows, int K, int N, la_dtype dt, Plan* p) {
    const cudaDataType_t ty = dt == LA_BF16 ? CUDA_R_16BF : CUDA_R_32F;
    cublasStatus_t s;
    if ((s = cublasLtMatmulDescCreate(&p->op, CUBLAS_COMPUTE_32F, CUDA_R_32F))) return s;
    if ((s = cublasLtMatrixLayoutCreate(&p->w, ty, N, K, N))) return s;
    if ((s = cublasLtMatrixLayoutCreate(&p->x, ty, K, rows, K))) return s;
    if ((s = cublasLtMatrixLayoutCreate(&p->y, ty, N, rows, N))) return s;
    cublasLtMatmulPreference_t pref = nullptr;
    if ((s = cublasLtMatmulPreferenceCreate(&pref))) return s;
    const size_t ws = kLtWorkspace;
    s = cublasLtMatmulPreferenceSetAttribute(pref, CUBLASLT_MATMUL_PREF_MAX_WORKSPACE_BYTES, &ws,
                                             sizeof(ws));
    // The entry point guarantees 16-byte alignment only (the heuristic's default
    // assumption is 256): exclude algorithms that need more.
    const uint32_t align = 16;
    const cublasLtMatmulPreferenceAttributes_t align_attr[4] = {
        CUBLASLT_MATMUL_PREF_MIN_ALIGNMENT_A_BYTES, CUBLASLT_MATMUL_PREF_MIN_ALIGNMENT_B_BYTES,
        CUBLASLT_MATMUL_PREF_MIN_ALIGNMENT_C_BYTES, CUBLASLT_MATMUL_PREF_MIN_ALIGNMENT_D_BYTES};
    for (int a = 0; a < 4 && s == CUBLAS_STATUS_SUCCESS; ++a)
        s = cublasLtMatmulPreferenceSetAttribute(pref, align_attr[a], &align, sizeof(align));
    cublasLtMatmulHeuristicResult_t res = {};
    int found = 0;
    if (s == CUBLAS_STATUS_SUCCESS)
        s = cublasLtMatmulAlgoGetHeuristic(h, p->op, p->w, p->x, p->y, p->y, pref, 1, &res, &found);
    cublasLtMatmulPreferenceDestroy(pref);
    if (s) return s;
    if (found < 1) return CUBLAS_STATUS_NOT_SUPPORTED;
    p->algo = res.algo;
    return CUBLAS_STATUS_SUCCESS;
}

// Y = X W on `st`; plans are built once per shape and device and kept.
la_status gemm(int dev, int rows, int K, int N, la_dtype dt, const void* X, const void* W, void* Y,
               void* lt_ws, cudaStream_t st) {
    Device& d = g_dev[dev];
    std::lock_guard<std::mutex> lock(d.mu);
    if (!d.handle && cublasLtCreate(&d.handle) != CUBLAS_STATUS_SUCCESS) return LA_ERR_CUDA;
    const auto key = std::make_tuple(rows, K, N, (int)dt);
    auto it = d.plans.find(key);
    if (it == d.plans.end()) {
        Plan p;
        const cublasStatus_t s = make_plan(d.handle, rows, K, N, dt, &p);
        if (s == CUBLAS_STATUS_NOT_SUPPORTED) return LA_ERR_UNSUPPORTED;
        if (s != CUBLAS_STATUS_SUCCESS) return LA_ERR_CUDA;
        it = d.plans.emplace(key, p).first;
    }
    const Plan& p = it->second;
    const float one = 1.f, zero = 0.f;
    const cublasStatus_t s = cublasLtMatmul(d.handle, p.op, &one, W, p.w, X, p.x, &zero, Y, p.y, Y,
                                            p.y, &p.algo, lt_ws, kLtWorkspace, st);
    return s == CUBLAS_STATUS_SUCCESS ? LA_OK : LA_ERR_CUDA;
}

}  // namespace

size_t layer_workspace(int B, int H, int D, la_dtype dt) {
    const size_t dm = (size_t)H * D;
    return align256((size_t)B * 3 * dm * elem(dt)) + align256((size_t)B * dm * elem(dt)) +
           kLtWorkspace;
}

}  // namespace la

extern "C" la_status la_layer_decode_step(const void* x, const void* Wqkv, const void* Wo, void* y,
                                          float* S, float* z, int B, int H, int D, la_dtype dt,
                                          float eps, void* workspace, size_t workspace_bytes,
                                          la_stream_t stream) {
    size_t need = 0;
    la_status s = la_workspace_size(LA_OP_LAYER_DECODE, B, H, 1, D, D, dt, &need);
    if (s != LA_OK) return s;
    if (!isfinite(eps) || eps < 0.f) return LA_ERR_INVALID_ARG;
    const int64_t BH = (int64_t)B * H;
    if (BH == 0) return LA_OK;
    auto bad = [](const void* p) { return !p || (reinterpret_cast<uintptr_t>(p) & 15); };
    if (bad(x) || bad(Wqkv) || bad(Wo) || bad(y) || bad(S) || bad(z)) return LA_ERR_INVALID_ARG;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255) || workspace_bytes < need)
        return LA_ERR_WORKSPACE;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= la::kMaxDevices) return LA_ERR_CUDA;
    cudaStream_t st = (cudaStream_t)stream;
    const size_t eb = la::elem(dt), dm = (size_t)H * D;
    char* body = static_cast<char*>(workspace) + sizeof(la::WsHeader);
    char* qkv = body;
    char* o = qkv + la::align256((size_t)B * 3 * dm * eb);
    char* lt_ws = o + la::align256((size_t)B * dm * eb);
    if ((s = la::gemm(dev, B, (int)dm, (int)(3 * dm), dt, x, Wqkv, qkv, lt_ws, st)) != LA_OK)
        return s;
    // Head j of sequence b: q at b 3 H D + j D, k at + H D, v at + 2 H D.
    if (la::decode_step_strided(qkv, qkv + dm * eb, qkv + 2 * dm * eb, o, S, z, dt, BH, D, D, eps,
                                la::kPhiElu1, H, (int64_t)(3 * dm), (int64_t)(3 * dm), st) !=
        cudaSuccess)
        return LA_ERR_CUDA;
    return la::gemm(dev, B, (int)dm, (int)dm, dt, o, Wo, y, lt_ws, st);
}
