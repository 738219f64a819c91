// Causal forward for callers that cannot allocate device memory.
//
// Some callers have no way to obtain a workspace: a plugin host that hands a
// kernel only its input and output buffers, a real-time or safety-certified
// process that forbids device allocation after start-up, or code whose memory
// is owned by another framework's pool that this library cannot call into.
// la_causal_fwd_noalloc serves them: it computes what la_causal_fwd computes,
// but its scratch lives in one fixed array in device memory that is part of
// this library (kNoAllocScratchBytes per GPU, held by every GPU that loads the
// library until the process exits). It calls no allocating routine.
// la_noalloc_query_status and la_noalloc_set_wait_limit read and set the
// array's header (status word, wait limit, test hook), as la_query_status and
// the header words of a workspace do for the workspace entry points.
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
// Per device: the body holds per-chunk fp32 states written by the fp32 path.
// The tensor-core path reads 64-bit words of the same body as (value, launch
// tag) pairs, so before its next call the body is cleared (tag 0 never
// matches a launch tag, which is the header's epoch + 1).
bool g_body_untagged[kMaxDevices];

// Header defaults: no error, default wait limit, test hook off.
__global__ void noalloc_init_header() {
    la::init_header(reinterpret_cast<la::WsHeader*>(g_scratch));
}

// Wait limit in microseconds (0: the default) and the load-withholding test hook.
__global__ void noalloc_set_hook(uint32_t max_spin, uint32_t hold) {
    la::WsHeader* h = reinterpret_cast<la::WsHeader*>(g_scratch);
    h->max_spin = max_spin ? max_spin : la::kDefaultMaxSpin;
    h->hold_item = hold;
}

// First use on a device: resolve the array's device address (with that device
// current) and initialise the header on the caller's stream.
la_status scratch_for_device(int dev, cudaStream_t st, void** out) {
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

la_status current_device(int* dev) {
    if (cudaGetDevice(dev) != cudaSuccess || *dev < 0 || *dev >= kMaxDevices) return LA_ERR_CUDA;
    return LA_OK;
}

// The stream (unless it is a default stream) and every given pointer must
// belong to the current device, whose array the call uses.
la_status check_device(int dev, cudaStream_t st, std::initializer_list<const void*> ptrs) {
    if (st != nullptr && st != cudaStreamLegacy && st != cudaStreamPerThread) {
        int sdev = -1;
        if (cudaStreamGetDevice(st, &sdev) != cudaSuccess) return LA_ERR_INVALID_ARG;
        if (sdev != dev) return LA_ERR_INVALID_ARG;
    }
    for (const void* p : ptrs) {
        if (!p) continue;
        cudaPointerAttributes a;
        if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
            cudaGetLastError();
            return LA_ERR_INVALID_ARG;
        }
        if (a.type == cudaMemoryTypeManaged) continue;
        if (a.type != cudaMemoryTypeDevice || a.device != dev) return LA_ERR_INVALID_ARG;
    }
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
    // Tensor-core path when its workspace fits the array, else the fp32 path
    // when its workspace does.
    bool tc = la::tc_causal_supported(Dk, Dv, dt);
    size_t body = tc ? la::tc_causal_workspace(BH, N, Dk) : la::simt_causal_workspace(BH, N, Dk, Dv);
    if (tc && Dk != 64 && kHeaderBytes + body > kNoAllocScratchBytes) {
        tc = false;
        body = la::simt_causal_workspace(BH, N, Dk, Dv);
    }
    if (kHeaderBytes + body > kNoAllocScratchBytes) return LA_ERR_WORKSPACE;  // beyond capacity
    const bool tagged = tc && Dk == 64;   // the only path that reads tagged words
    cudaStream_t st = (cudaStream_t)stream;
    int dev = -1;
    la_status s = current_device(&dev);
    if (s != LA_OK) return s;
    if ((s = check_device(dev, st, {q, k, v, o, S_out, z_out})) != LA_OK) return s;
    void* ws = nullptr;
    if ((s = scratch_for_device(dev, st, &ws)) != LA_OK) return s;
    char* scratch = static_cast<char*>(ws) + kHeaderBytes;
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        if (tagged && g_body_untagged[dev]) {
            if (cudaMemsetAsync(scratch, 0, body, st) != cudaSuccess) return LA_ERR_CUDA;
            g_body_untagged[dev] = false;
        }
        if (!tagged) g_body_untagged[dev] = true;
    }
    cudaError_t err = tc ? la::tc_causal(q, k, v, o, BH, N, Dk, eps, LA_PHI_ELU1, nullptr, nullptr,
                                         S_out, z_out, ws, scratch, st)
                         : la::simt_causal(q, k, v, o, dt, BH, N, Dk, Dv, eps, LA_PHI_ELU1, nullptr,
                                           nullptr, S_out, z_out, scratch, st);
    return err == cudaSuccess ? LA_OK : LA_ERR_CUDA;
}

extern "C" la_status la_noalloc_query_status(la_stream_t stream) {
    int dev = -1;
    la_status s = current_device(&dev);
    if (s != LA_OK) return s;
    void* ws = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        ws = g_scratch_addr[dev];
    }
    if (!ws) return LA_OK;  // no call on this device yet
    return la_query_status(ws, stream);
}

extern "C" la_status la_noalloc_set_wait_limit(unsigned int max_spin_us, int hold_loads,
                                               la_stream_t stream) {
    int dev = -1;
    la_status s = current_device(&dev);
    if (s != LA_OK) return s;
    cudaStream_t st = (cudaStream_t)stream;
    if ((s = check_device(dev, st, {})) != LA_OK) return s;
    void* ws = nullptr;
    if ((s = scratch_for_device(dev, st, &ws)) != LA_OK) return s;
    noalloc_set_hook<<<1, 1, 0, st>>>(max_spin_us, hold_loads ? 1u : 0u);
    return cudaPeekAtLastError() == cudaSuccess ? LA_OK : LA_ERR_CUDA;
}
