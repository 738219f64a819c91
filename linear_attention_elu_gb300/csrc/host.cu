// Causal forward on HOST buffers with the transfers overlapped.
//
// la_causal_fwd works on device tensors; a caller whose q, k, v live in host
// memory and who wants o back in host memory would otherwise copy everything
// in, run the forward and copy o out, one after the other. Here the heads are
// cut into groups that stream through two device staging buffers: while group
// g is computed, group g + 1 is copied in on one copy engine and group g - 1
// copied out on the other. Heads are independent, so each group is an ordinary
// la_causal_fwd call on its slice (contiguous in the [B, H, N, D] layout).
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace {

constexpr int kMaxDevices = 128;
constexpr int kGroups = 4;           // groups per call (fewer when B*H is smaller)

// Per device: a copy-in and a copy-out stream and their events, created on first
// use and kept for the process lifetime. The mutex also keeps the enqueue
// sequence of concurrent callers from interleaving on the shared events.
struct HostPipe {
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t start = nullptr, done = nullptr;
    cudaEvent_t loaded[2] = {nullptr, nullptr};   // group in buffer b copied in
    cudaEvent_t computed[2] = {nullptr, nullptr}; // group in buffer b computed
    cudaEvent_t drained[2] = {nullptr, nullptr};  // group in buffer b copied out
    bool ready = false;
};
std::mutex g_pipe_mutex[kMaxDevices];
HostPipe g_pipe[kMaxDevices];

cudaError_t make_pipe(HostPipe& p) {
    cudaError_t e;
    if ((e = cudaStreamCreateWithFlags(&p.in, cudaStreamNonBlocking))) return e;
    if ((e = cudaStreamCreateWithFlags(&p.out, cudaStreamNonBlocking))) return e;
    cudaEvent_t* all[] = {&p.start, &p.done, &p.loaded[0], &p.loaded[1], &p.computed[0],
                          &p.computed[1], &p.drained[0], &p.drained[1]};
    for (cudaEvent_t* ev : all)
        if ((e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming))) return e;
    p.ready = true;
    return cudaSuccess;
}

size_t elem_bytes(la_dtype dt) { return dt == LA_BF16 ? 2 : 4; }

// Heads per group: a quarter of B*H, rounded up to a multiple of 4 so that every
// group's slice of S_out and z_out stays 16-byte aligned.
int64_t group_heads(int64_t BH) { return ((BH + kGroups - 1) / kGroups + 3) / 4 * 4; }

// Heads of the group starting at head h0. The last full-size group is cut into
// g - 4 and 4 heads: after the last copy in, only a 4-head forward and its copy
// out remain, instead of a quarter of the batch (group starts stay multiples
// of 4).
int64_t group_size(int64_t BH, int64_t h0) {
    const int64_t g = group_heads(BH), rest = BH - h0;
    if (g >= 8 && rest > 4 && rest <= g) return rest - 4;
    return rest < g ? rest : g;
}

}  // namespace

extern "C" {

la_status la_host_staging_size(int B, int H, int N, int Dk, int Dv, la_dtype dt, size_t* bytes) {
    if (!bytes) return LA_ERR_INVALID_ARG;
    if (B < 0 || H < 0 || N < 0 || Dk <= 0 || Dv <= 0 || (dt != LA_F32 && dt != LA_BF16))
        return LA_ERR_INVALID_ARG;
    const int64_t per_head = (int64_t)N * (2 * Dk + 2 * (int64_t)Dv) * (int64_t)elem_bytes(dt);
    // Two buffers of one group each; every tensor slice starts 256-byte aligned.
    const int64_t g = group_heads((int64_t)B * H);
    *bytes = (size_t)(2 * (g * per_head + 4 * 256));
    return LA_OK;
}

la_status la_causal_fwd_host(const void* q, const void* k, const void* v, void* o, int B, int H,
                             int N, int Dk, int Dv, la_dtype dt, float eps, float* S_out,
                             float* z_out, void* staging, size_t staging_bytes, void* workspace,
                             size_t workspace_bytes, la_stream_t stream) {
    const int64_t BH = (int64_t)B * H;
    size_t need = 0;
    la_status s = la_host_staging_size(B, H, N, Dk, Dv, dt, &need);
    if (s != LA_OK) return s;
    if (BH == 0 || N == 0)  // nothing to copy: the device entry handles the final state
        return la_causal_fwd(nullptr, nullptr, nullptr, nullptr, B, H, N, Dk, Dv, dt, eps, S_out,
                             z_out, workspace, workspace_bytes, stream);
    if (!q || !k || !v || !o) return LA_ERR_INVALID_ARG;
    if (!staging || (reinterpret_cast<uintptr_t>(staging) & 255) || staging_bytes < need)
        return LA_ERR_WORKSPACE;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return LA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_pipe_mutex[dev]);
    HostPipe& p = g_pipe[dev];
    if (!p.ready && make_pipe(p) != cudaSuccess) return LA_ERR_CUDA;

    const size_t eb = elem_bytes(dt);
    const int64_t g_heads = group_heads(BH);
    const int64_t qk_head = (int64_t)N * Dk * eb, vo_head = (int64_t)N * Dv * eb;
    auto align = [](int64_t x) { return (x + 255) / 256 * 256; };
    const int64_t q_off = 0, k_off = align(g_heads * qk_head), v_off = k_off + align(g_heads * qk_head);
    const int64_t o_off = v_off + align(g_heads * vo_head), buf_bytes = o_off + align(g_heads * vo_head);
    cudaStream_t st = (cudaStream_t)stream;
    auto cu = [](cudaError_t e) { return e == cudaSuccess; };
    // Everything is ordered after the work already queued on the caller's stream.
    if (!cu(cudaEventRecord(p.start, st)) || !cu(cudaStreamWaitEvent(p.in, p.start, 0)) ||
        !cu(cudaStreamWaitEvent(p.out, p.start, 0)))
        return LA_ERR_CUDA;
    const char* hq = static_cast<const char*>(q);
    const char* hk = static_cast<const char*>(k);
    const char* hv = static_cast<const char*>(v);
    char* ho = static_cast<char*>(o);
    int g = 0;
    for (int64_t h0 = 0, nh = 0; h0 < BH; h0 += nh, ++g) {
        const int b = g & 1;
        nh = group_size(BH, h0);
        char* buf = static_cast<char*>(staging) + b * buf_bytes;
        // Buffer b is free once the group two before has been copied out (which
        // itself waited for that group's compute).
        if (g >= 2 && !cu(cudaStreamWaitEvent(p.in, p.drained[b], 0))) return LA_ERR_CUDA;
        if (!cu(cudaMemcpyAsync(buf + q_off, hq + h0 * qk_head, nh * qk_head, cudaMemcpyHostToDevice, p.in)) ||
            !cu(cudaMemcpyAsync(buf + k_off, hk + h0 * qk_head, nh * qk_head, cudaMemcpyHostToDevice, p.in)) ||
            !cu(cudaMemcpyAsync(buf + v_off, hv + h0 * vo_head, nh * vo_head, cudaMemcpyHostToDevice, p.in)) ||
            !cu(cudaEventRecord(p.loaded[b], p.in)) || !cu(cudaStreamWaitEvent(st, p.loaded[b], 0)))
            return LA_ERR_CUDA;
        // The group as B = 1, H = nh: heads of the flattened [B*H] axis are independent.
        s = la_causal_fwd(buf + q_off, buf + k_off, buf + v_off, buf + o_off, 1, (int)nh, N, Dk, Dv,
                          dt, eps, S_out ? S_out + h0 * Dk * Dv : nullptr,
                          z_out ? z_out + h0 * Dk : nullptr, workspace, workspace_bytes, stream);
        if (s != LA_OK) return s;
        if (!cu(cudaEventRecord(p.computed[b], st)) || !cu(cudaStreamWaitEvent(p.out, p.computed[b], 0)) ||
            !cu(cudaMemcpyAsync(ho + h0 * vo_head, buf + o_off, nh * vo_head, cudaMemcpyDeviceToHost, p.out)) ||
            !cu(cudaEventRecord(p.drained[b], p.out)))
            return LA_ERR_CUDA;
    }
    // The call completes on the caller's stream once the last output has landed.
    if (!cu(cudaEventRecord(p.done, p.out)) || !cu(cudaStreamWaitEvent(st, p.done, 0)))
        return LA_ERR_CUDA;
    return LA_OK;
}

}  // extern "C"
