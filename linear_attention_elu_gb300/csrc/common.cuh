// Device-side helpers shared by the kernels of the linear-attention library.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "linattn.h"

namespace la {

// Largest head dimension any path accepts (Dk and Dv).
constexpr int kMaxDim = 128;
// Tokens per chunk of the chunked causal evaluation.
constexpr int kChunk = 64;

// phi(x) = elu(x) + 1: x + 1 for x > 0, exp(x) otherwise ("Why Replace
// Attention? The Softmax Bottleneck and the Path to Linear Time", section 5.3).
__device__ __forceinline__ float phi(float x) { return x > 0.f ? x + 1.f : expf(x); }

// Feature maps (the values of la_phi in the C ABI): elu(x) + 1, or the identity
// for features the caller has already computed -- the method leaves phi free
// (same blog, section 4.5). kNoMap marks loads of values, which take no map.
constexpr int kPhiElu1 = 0, kPhiIdentity = 1, kNoMap = -1;
__device__ __forceinline__ float fmap(float x, int kind) {
    return kind == kPhiIdentity ? x : phi(x);
}
// The map's derivative written through its value f = fmap(x): for elu(x) + 1,
// 1 for x > 0 and e^x = f for x <= 0, i.e. min(f, 1); 1 for the identity.
__device__ __forceinline__ float fmap_grad(float f, int kind) {
    return kind == kPhiIdentity ? 1.f : fminf(f, 1.f);
}

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// Workspace header (first 256 bytes of every workspace).
struct WsHeader {
    uint32_t status;     // 0 = ok, else an la_status code set by a kernel
    uint32_t epoch;      // launches of cross-CTA publishing kernels completed so far
    uint32_t ticket;     // reserved
    uint32_t done;       // CTAs finished in the running cross-CTA publishing launch
    uint32_t max_spin;   // limit of every bounded wait, in microseconds
    uint32_t hold_item;  // test hook: when set, input loads are withheld
    uint32_t pad[58];
};
static_assert(sizeof(WsHeader) == 256, "workspace header is 256 bytes");

constexpr uint32_t kDefaultMaxSpin = 2000000;   // 2 s

__device__ __forceinline__ void set_status(WsHeader* h, uint32_t code) {
    atomicCAS(&h->status, 0u, code);
}

// Header defaults: no error, default wait limit, test hook off.
__device__ __forceinline__ void init_header(WsHeader* h) {
    h->status = 0;
    h->epoch = 0;
    h->ticket = 0;
    h->done = 0;
    h->max_spin = kDefaultMaxSpin;
    h->hold_item = 0;
}

}  // namespace la
