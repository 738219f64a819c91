// Causal forward for callers that cannot allocate device memory.
//
// Some callers have no way to obtain a workspace: a plugin host that hands a
// kernel only its input and output buffers, a real-time or safety-certified
// process that forbids device allocation after start-up, or code whose memory
// is owned by another framework's pool that this library cannot call into.
// la_causal_fwd_noalloc serves them: it computes exactly what la_causal_fwd
// computes, but its scratch lives in one fixed array in device memory that is
// part of this library (kNoAllocScratchBytes per GPU, held by every GPU that
// loads the library until the process exits). It calls no allocating routine.
#include <math.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB
constexpr size_t kHeaderBytes = sizeof(la::WsHeader);

// The scratch itself. In host code this name is only a stand-in for the
// device object: the kernels get its device address from cudaGetSymbolAddress.
__device__ __align__(256) unsigned char g_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 128;
std::mutex g_mutex;
void* g_scratch_addr[kMaxDevices];  // device address of g_scratch, per device; null until set up

// Header defaults: no error, default wait limit, test hook off.
__global__ void noalloc_init_header() {
    la::init_header(reinterpret_cast<la::WsHeader*>(g_scratch));
}

// First use on a device: resolve the array's device address (with that device
// current) and initialise the header on the caller's stream.
la_status scratch_for_current_device(cudaStream_t st, void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return LA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_addr[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_scratch) != cudaSuccess || !ptr) return LA_ERR_CUDA;
        noalloc_init_header<<<1, 1, 0, st>>>();
        if (cudaPeekAtLastError() != cudaSuccess) return LA_ERR_CUDA;
        g_scratch_addr[dev] = ptr;
    }
    *out = g_scratch_addr[dev];
    return LA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

extern "C" la_status la_causal_fwd_noalloc(const void* q, const void* k, const void* v, void* o,
                                          int B, int H, int N, int Dk, int Dv, la_dtype dt,
                                          float eps, float* S_out, float* z_out,
                                          la_stream_t stream) {
    if (B < 0 || H < 0 || N < 0 || Dk <= 0 || Dv <= 0) return LA_ERR_INVALID_ARG;
    if (dt != LA_F32 && dt != LA_BF16) return LA_ERR_INVALID_ARG;
    if (!isfinite(eps) || eps < 0.f) return LA_ERR_INVALID_ARG;
    if (Dk > la::kMaxDim || Dv > la::kMaxDim || (int64_t)B * H > 65535) return LA_ERR_UNSUPPORTED;
    const int64_t BH = (int64_t)B * H;
    if (BH == 0 || N == 0) return la_causal_fwd(q, k, v, o, B, H, N, Dk, Dv, dt, eps, S_out,
                                                z_out, nullptr, 0, stream);
    if (!q || !k || !v || !o || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o))
        return LA_ERR_INVALID_ARG;
    if ((S_out && !aligned16(S_out)) || (z_out && !aligned16(z_out))) return LA_ERR_INVALID_ARG;
    const bool tc = la::tc_causal_supported(Dk, Dv, dt);
    const size_t body = tc ? la::tc_causal_workspace(BH, N)
                           : la::simt_causal_workspace(BH, N, Dk, Dv);
    if (kHeaderBytes + body > kNoAllocScratchBytes) return LA_ERR_WORKSPACE;  // beyond capacity
    cudaStream_t st = (cudaStream_t)stream;
    void* ws = nullptr;
    la_status s = scratch_for_current_device(st, &ws);
    if (s != LA_OK) return s;
    char* scratch = static_cast<char*>(ws) + kHeaderBytes;
    cudaError_t err = tc ? la::tc_causal(q, k, v, o, BH, N, eps, LA_PHI_ELU1, nullptr, nullptr, S_out,
                                         z_out, ws, scratch, st)
                         : la::simt_causal(q, k, v, o, dt, BH, N, Dk, Dv, eps, LA_PHI_ELU1, nullptr,
                                           nullptr, S_out, z_out, scratch, st);
    return err == cudaSuccess ? LA_OK : LA_ERR_CUDA;
}
