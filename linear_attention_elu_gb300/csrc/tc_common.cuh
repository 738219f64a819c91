// Helpers shared by the tensor-core kernels (causal and non-causal paths):
// the persistent-CTA chunk partition, packed bf16 phi, barriers with uniform
// abort decisions, constant operand tiles, programmatic-dependent-launch
// controls and the host-side TMA descriptor encoding.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "common.cuh"
#include "tc_util.cuh"

namespace la {
namespace tcc {

using namespace tc;

constexpr int kC = 128;                        // tokens per chunk (one M = 128 row block)
constexpr uint32_t kTileBytes = kC * 64 * 2;   // one bf16 [128 x 64] tile = 16 KB

// The B*H*ceil(N/128) chunks in head-major order, cut into `grid` contiguous
// ranges (one per persistent CTA). A range holds "runs": its chunks of one head.
struct Partition {
    int64_t T;      // total chunks = BH * nchunks
    int nchunks;    // chunks per head
    int grid;       // CTAs
    int maxr;       // aggregate slots per CTA
    __host__ __device__ int64_t begin(int c) const { return (int64_t)c * T / grid; }
};

inline Partition make_partition(int64_t BH, int N, int grid) {
    Partition p;
    p.nchunks = (N + kC - 1) / kC;
    p.T = BH * p.nchunks;
    p.grid = (int)(grid < p.T ? grid : p.T);
    const int64_t len = (p.T + p.grid - 1) / p.grid;
    p.maxr = (int)((len + p.nchunks - 1) / p.nchunks + 1);
    return p;
}


__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %2, %1;" : "=r"(r) : "f"(a), "f"(b));
    return r;
}

__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }

// One 32-key block of causal scores (r0: keys 0-15, r1: keys 16-31, fp32 bits)
// to 16 words of packed bf16. Blocks below the diagonal keep every key; the
// diagonal block keeps keys 0..last (the row's own position in the block) and
// zeroes the rest. The caller picks the form per block (a warp-uniform choice),
// so the per-key compares run on the diagonal block only.
__device__ __forceinline__ void pack_block32(const uint32_t* r0, const uint32_t* r1, uint32_t* p) {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        p[e] = pack_bf16(__uint_as_float(r0[2 * e]), __uint_as_float(r0[2 * e + 1]));
        p[8 + e] = pack_bf16(__uint_as_float(r1[2 * e]), __uint_as_float(r1[2 * e + 1]));
    }
}

__device__ __forceinline__ void pack_block32_diag(const uint32_t* r0, const uint32_t* r1, int last,
                                                  uint32_t* p) {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        p[e] = pack_bf16(2 * e <= last ? __uint_as_float(r0[2 * e]) : 0.f,
                         2 * e + 1 <= last ? __uint_as_float(r0[2 * e + 1]) : 0.f);
        p[8 + e] = pack_bf16(16 + 2 * e <= last ? __uint_as_float(r1[2 * e]) : 0.f,
                             17 + 2 * e <= last ? __uint_as_float(r1[2 * e + 1]) : 0.f);
    }
}

// phi(x) = max(x, 0) + e^min(x, 0) on two packed bf16 values: x + 1 for
// x > 0 (the exponent is 0, e = 1) and e^x for x <= 0.
// max(x, 0) and max(-x, 0) are packed bf16 fused multiply-adds with relu
// (x * (+-1) + 0, exact), which run on the FMA pipe. Each value of max(-x, 0)
// widens exactly to fp32; t = -max(-x, 0) * fp32(log2 e) = min(x, 0) * log2 e
// is one fp32 product (relative error <= 2^-23; the pair in one packed
// multiply), 2^t is the fp32 hardware ex2 (which flushes results below 2^-126
// to zero), the pair is rounded once to bf16, and the final packed bf16 add
// rounds the exact sum once. Error bound, for every bf16 input x >= -87.3: the
// result is within 2^-8 (+ 1e-5) of phi(x) relative, which is the bf16
// rounding of phi itself; below -87.3 the result is 0 (e^x < 1.2e-38 there).
// A float64 emulation over every bf16 input checks this bound in the CPU
// tests. (t rounded to bf16 before a bf16 ex2 costs fewer instructions, but
// its error grows with |x|: 3 % near x = -5, 13 % below x = -20.)
__device__ __forceinline__ uint32_t phi_bf16x2(uint32_t x) {
    constexpr float kNegLog2e = -1.4426950408889634f;
    constexpr uint32_t kOne = 0x3F803F80u, kMinusOne = 0xBF80BF80u;
    uint32_t n, p;
    asm("fma.rn.relu.bf16x2 %0, %1, %2, %3;" : "=r"(n) : "r"(x), "r"(kMinusOne), "r"(0u));
    asm("fma.rn.relu.bf16x2 %0, %1, %2, %3;" : "=r"(p) : "r"(x), "r"(kOne), "r"(0u));
    const float nlo = __uint_as_float(n << 16), nhi = __uint_as_float(n & 0xFFFF0000u);
    uint64_t xx, cc, tt;
    asm("mov.b64 %0, {%1, %2};" : "=l"(xx) : "f"(nlo), "f"(nhi));
    asm("mov.b64 %0, {%1, %1};" : "=l"(cc) : "f"(kNegLog2e));
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(tt) : "l"(xx), "l"(cc));
    float tlo, thi, elo, ehi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(tlo), "=f"(thi) : "l"(tt));
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(elo) : "f"(tlo));
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(ehi) : "f"(thi));
    uint32_t e, r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(e) : "f"(ehi), "f"(elo));
    asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(p), "r"(e));
    return r;
}

// The feature map on eight packed bf16 values: elu + 1, or (kPhiIdentity) the
// values as they are, for features the caller has already computed.
template <int kPhi = kPhiElu1>
__device__ __forceinline__ uint4 phi8(uint4 u) {
    if constexpr (kPhi == kPhiIdentity) return u;
    else return make_uint4(phi_bf16x2(u.x), phi_bf16x2(u.y), phi_bf16x2(u.z), phi_bf16x2(u.w));
}

__device__ __forceinline__ void named_bar(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Named barrier that also ANDs `pred` over the participating threads, so that
// every thread takes the same abort decision after a bounded wait.
__device__ __forceinline__ bool named_bar_and(int id, int threads, bool pred) {
    uint32_t out;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n"
        " bar.red.and.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}\n"
        : "=r"(out)
        : "r"((uint32_t)pred), "r"(id), "r"(threads)
        : "memory");
    return out != 0;
}

__device__ __forceinline__ void report_timeout(WsHeader* hdr) {
    atomicCAS(&hdr->status, 0u, (uint32_t)LA_ERR_TIMEOUT);
}

// Rows >= zero_from of a 128 x 64 bf16 tile set to 0, for the rows
// (t >> 3) + 32 k, physical chunk (t & 7), that thread t of a 256-thread group
// owns in the phi loops below. Only a sequence's last, ragged chunk needs it;
// the phi loops map every row and the owner then overwrites its own rows past
// the end (program order), so full chunks carry no per-row selects.
__device__ __forceinline__ void zero_rows_256(uint8_t* tile, int t, int zero_from) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int r = (t >> 3) + 32 * k;
        if (r >= zero_from)
            *reinterpret_cast<uint4*>(tile + r * 128 + (t & 7) * 16) = make_uint4(0, 0, 0, 0);
    }
}

// phi in place on the 128 x 64 bf16 tile rows (t >> 3) + 32 k, physical chunk
// (t & 7), for a 256-thread group; rows >= zero_from are set to 0.
template <int kPhi = kPhiElu1>
__device__ __forceinline__ void phi_tile_256(uint8_t* tile, int t, int zero_from) {
    uint4 v[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
        v[k] = *reinterpret_cast<const uint4*>(tile + ((t >> 3) + 32 * k) * 128 + (t & 7) * 16);
#pragma unroll
    for (int k = 0; k < 4; ++k)
        *reinterpret_cast<uint4*>(tile + ((t >> 3) + 32 * k) * 128 + (t & 7) * 16) =
            phi8<kPhi>(v[k]);
    if (zero_from < kC) zero_rows_256(tile, t, zero_from);
}

// phi_tile_256 on two tiles at once, four 16-byte pieces per iteration (all
// four loads issued before any store). The loop is kept rolled on purpose: the
// kernels that call it run many warp roles side by side, and a fully unrolled
// body (eight pieces of ten instructions per value pair) costs more in
// instruction fetch than its extra overlap gains; two pieces per iteration
// were about 1.5 % slower than four.
template <int kPhi = kPhiElu1>
__device__ __forceinline__ void phi_tiles2_256(uint8_t* ta, int zero_a, uint8_t* tb, int zero_b,
                                               int t) {
#pragma unroll 1
    for (int k2 = 0; k2 < 8; k2 += 4) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int k = k2 + u;
            v[u] = *reinterpret_cast<const uint4*>((k < 4 ? ta : tb) +
                                                   ((t >> 3) + 32 * (k & 3)) * 128 + (t & 7) * 16);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int k = k2 + u;
            *reinterpret_cast<uint4*>((k < 4 ? ta : tb) + ((t >> 3) + 32 * (k & 3)) * 128 +
                                      (t & 7) * 16) = phi8<kPhi>(v[u]);
        }
    }
    if (zero_a < kC) zero_rows_256(ta, t, zero_a);
    if (zero_b < kC) zero_rows_256(tb, t, zero_b);
}

// The "ones" operand tile: 128 rows, logical column 0 = 1.0, the rest 0.
__device__ __forceinline__ void init_ones_tile(uint8_t* tile, int t, int nthreads) {
    for (int idx = t; idx < kC * 8; idx += nthreads) {
        const int r = idx >> 3, pc = idx & 7;
        const int logical = pc ^ (r & 7);
        *reinterpret_cast<uint4*>(tile + r * 128 + pc * 16) =
            make_uint4(logical == 0 ? 0x3F80u : 0u, 0, 0, 0);
    }
}

__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }


// ---------------------------------------------------------------- host side

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                 const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                 const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiled get_encoder() {
    static EncodeTiled fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiled>(p);
    }
    return fn;
}

// [BH, N, D] bf16 viewed as 3-D (D, N, BH); box = 64 features x 128 tokens x 1 head.
inline bool encode_bhnd(CUtensorMap* map, const void* ptr, int64_t BH, int N, int D) {
    EncodeTiled enc = get_encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)N, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)N * D * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)kC, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides,
               box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

constexpr int kMaxDevices = 128;

// SM count of the current device (cached per device; host-only).
inline int sm_count() {
    static std::atomic<int> cache[kMaxDevices];
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
    n = cache[dev].load(std::memory_order_relaxed);
    if (n > 0) return n;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        return 148;
    cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

// Opts `kernel` in to `bytes` of dynamic shared memory once per device (the
// setting is per function and device; repeating it costs host time per call).
template <typename Kernel>
inline cudaError_t ensure_smem_optin(Kernel kernel, int bytes, std::atomic<int>* done) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev >= 0 && dev < kMaxDevices && done[dev].load(std::memory_order_acquire)) return cudaSuccess;
    err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (err == cudaSuccess && dev >= 0 && dev < kMaxDevices) done[dev].store(1, std::memory_order_release);
    return err;
}

}  // namespace tcc
}  // namespace la
