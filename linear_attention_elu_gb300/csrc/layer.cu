// One decode step of a linear-attention layer for B sequences:
// [q | k | v] = x Wqkv, one recurrent step per head on (S, z), y = o Wo
// ("Why Replace Attention? The Softmax Bottleneck and the Path to Linear
// Time", section 7.2, steps 1-4; "Transformers Are RNNs: Linear Attention",
// the generation loop carrying only (S, z)).
//
// The two projections are dense products with fp32 accumulation (csrc/gemm.cu:
// tcgen05 for bf16 storage, fp32 FMA otherwise); the attention step is the
// library's decode kernel, reading q, k, v straight out of the [B, 3 H D]
// projection through its row stride, so nothing is copied between the three
// launches. The projection buffers live in the caller's workspace; all three
// launches run on the caller's stream and can be captured in one CUDA graph.
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace la {

namespace {

size_t elem(la_dtype dt) { return dt == LA_BF16 ? 2 : 4; }
size_t align256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace

size_t layer_workspace(int B, int H, int D, la_dtype dt) {
    const size_t dm = (size_t)H * D;
    return align256((size_t)B * 3 * dm * elem(dt)) + align256((size_t)B * dm * elem(dt));
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
    cudaStream_t st = (cudaStream_t)stream;
    const size_t eb = la::elem(dt), dm = (size_t)H * D;
    char* body = static_cast<char*>(workspace) + sizeof(la::WsHeader);
    char* qkv = body;
    char* o = qkv + la::align256((size_t)B * 3 * dm * eb);
    if (la::gemm(x, Wqkv, qkv, B, (int)dm, (int)(3 * dm), dt, workspace, st) != cudaSuccess)
        return LA_ERR_CUDA;
    // Head j of sequence b: q at b 3 H D + j D, k at + H D, v at + 2 H D.
    if (la::decode_step_strided(qkv, qkv + dm * eb, qkv + 2 * dm * eb, o, S, z, dt, BH, D, D, eps,
                                la::kPhiElu1, H, (int64_t)(3 * dm), (int64_t)(3 * dm), st) !=
        cudaSuccess)
        return LA_ERR_CUDA;
    return la::gemm(o, Wo, y, B, (int)dm, (int)dm, dt, workspace, st) == cudaSuccess ? LA_OK
                                                                                      : LA_ERR_CUDA;
}
