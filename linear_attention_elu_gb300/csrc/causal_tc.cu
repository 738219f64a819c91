// Tensor-core (tcgen05) causal forward for bf16 inputs, Dk = Dv = 64.
//
// Method. For chunk c of 128 tokens of one head, with S_{c-1}, z_{c-1} the
// state after the previous chunks ("Why Replace Attention? The Softmax
// Bottleneck and the Path to Linear Time", section 7.1: S_i and z_i are
// prefix sums, so a whole chunk can be added at once):
//   A     = phi(Q_c) phi(K_c)^T, masked to key <= query          (tensor core)
//   O_c   = phi(Q_c) S_{c-1} + A V_c                              (tensor core)
//   den_i = rowsum(A)_i + phi(q_i).z_{c-1} + eps                  (fp32)
//   o_i   = O_c,i / den_i
//   S_c   = S_{c-1} + phi(K_c)^T V_c,  z_c = z_{c-1} + sum phi(k)  (tensor core / fp32)
// This is an exact regrouping of the sums S_i = sum_{j<=i} phi(k_j) v_j^T
// (same blog, section 7.2) into whole chunks plus a masked in-chunk part.
//
// Work split. The B*H*ceil(N/128) chunks form one head-major sequence that is
// cut into gridDim.x contiguous ranges, one per persistent CTA. A range holds
// "runs" (its chunks of one head). Two launches share that partition:
//   state kernel   per run: dS = sum phi(K)^T V, dz = sum phi(K)  -> workspace
//   output kernel  per run: start state = sum of the dS, dz of the same head
//                  from lower-numbered CTAs (only a range's first run can
//                  have one), then the chunk loop above.
// The sum over earlier ranges is the exclusive prefix over segments (the
// parallel scan of the same blog, section 7.7), done in fp32.
//
// Data movement: TMA 3-D tiles (64 features x 128 tokens x 1 head, 128-byte
// swizzle) into shared memory; phi is applied in place in shared memory;
// every contraction is a tcgen05.mma (bf16 operands, fp32 accumulators in
// TMEM); outputs leave through a swizzled staging tile and a TMA store, which
// drops rows past N.
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_util.cuh"

namespace la {

namespace {

using namespace tc;

constexpr int kC = 128;                 // tokens per chunk
constexpr int kD = 64;                  // Dk = Dv
constexpr uint32_t kTileBytes = kC * kD * 2;   // one bf16 [128 x 64] tile = 16 KB
constexpr int kE = kD * kD + kD;        // floats per aggregate (S then z)

struct Partition {
    int64_t T;      // total chunks = BH * nchunks
    int nchunks;    // chunks per head
    int grid;       // CTAs
    int maxr;       // aggregate slots per CTA
    __host__ __device__ int64_t begin(int c) const { return (int64_t)c * T / grid; }
};

__host__ Partition make_partition(int64_t BH, int N, int grid) {
    Partition p;
    p.nchunks = (N + kC - 1) / kC;
    p.T = BH * p.nchunks;
    p.grid = (int)(grid < p.T ? grid : p.T);
    const int64_t len = (p.T + p.grid - 1) / p.grid;
    p.maxr = (int)((len + p.nchunks - 1) / p.nchunks + 1);
    return p;
}

// ---------------------------------------------------------------- helpers

__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %2, %1;" : "=r"(r) : "f"(a), "f"(b));
    return r;
}

__device__ __forceinline__ float phi_fast(float x) { return x > 0.f ? x + 1.f : __expf(x); }

// phi on 8 packed bf16 values in place; returns them (rounded) in f[8].
__device__ __forceinline__ uint4 phi8(uint4 u, float (&f)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float a = phi_fast(bf_lo(w[i])), b = phi_fast(bf_hi(w[i]));
        o[i] = pack_bf16(a, b);
        f[2 * i] = bf_lo(o[i]);
        f[2 * i + 1] = bf_hi(o[i]);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// Sums v over the 4 lanes of a warp that share (lane & 7) ^ (lane >> 3):
// the lanes holding the same logical column group of a swizzled tile.
__device__ __forceinline__ float reduce_colgroup(float v) {
    v += __shfl_xor_sync(0xffffffffu, v, 9);
    v += __shfl_xor_sync(0xffffffffu, v, 18);
    return v;
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
    if (hdr) atomicCAS(&hdr->status, 0u, (uint32_t)LA_ERR_TIMEOUT);
}

// ======================================================== state kernel
// Warps 0-3: phi pass and aggregate read-out. Warp 4: TMA producer. Warp 5: MMA.

constexpr int kStateStages = 4;
constexpr int kStateThreads = 192;
constexpr size_t kStateSmem = 1024 + kStateStages * 2 * kTileBytes + 1024;

__global__ void __launch_bounds__(kStateThreads, 1)
causal_state_kernel(const __grid_constant__ CUtensorMap kmap,
                    const __grid_constant__ CUtensorMap vmap, float* __restrict__ agg,
                    Partition part, int N, WsHeader* hdr) {
    const uint32_t max_spin = hdr->max_spin;
    const bool hold = hdr->hold_item != 0;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    uint8_t* stage_k[kStateStages];
    uint8_t* stage_v[kStateStages];
#pragma unroll
    for (int s = 0; s < kStateStages; ++s) {
        stage_k[s] = base + s * 2 * kTileBytes;
        stage_v[s] = stage_k[s] + kTileBytes;
    }
    __shared__ uint64_t full[kStateStages], empty[kStateStages], phi_ready[kStateStages];
    __shared__ uint64_t run_done, tmem_free, mma_drain;
    __shared__ uint32_t tmem_slot;
    __shared__ float zsum[kD];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cta = blockIdx.x;
    const int64_t u0 = part.begin(cta), u1 = part.begin(cta + 1);
    if (tid == 0) {
        for (int s = 0; s < kStateStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
            mbar_init(&phi_ready[s], 1);
        }
        mbar_init(&run_done, 1);
        mbar_init(&tmem_free, 1);
        mbar_init(&mma_drain, 1);
        fence_mbar_init();
    }
    if (tid < kD) zsum[tid] = 0.f;
    if (warp == 5) {
        tmem_alloc(&tmem_slot, 64);
        tmem_relinquish();
    }
    if (warp == 4 && lane == 0) {
        tma_prefetch_desc(&kmap);
        tma_prefetch_desc(&vmap);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;

    if (warp == 4) {
        if (lane == 0) {
            int i = 0;
            for (int64_t u = u0; u < u1; ++u, ++i) {
                const int s = i % kStateStages;
                if (i >= kStateStages &&
                    !mbar_wait(&empty[s], ((i / kStateStages) - 1) & 1, max_spin)) {
                    report_timeout(hdr);
                    break;
                }
                if (hold) break;  // test hook: a load that is never issued
                const int h = (int)(u / part.nchunks), ch = (int)(u % part.nchunks);
                mbar_arrive_expect_tx(&full[s], 2 * kTileBytes);
                tma_load_3d(stage_k[s], &kmap, &full[s], 0, ch * kC, h);
                tma_load_3d(stage_v[s], &vmap, &full[s], 0, ch * kC, h);
            }
            // Drain: every issued load must land before the CTA may exit.
            const int issued = i;
            for (int j = issued - kStateStages > 0 ? issued - kStateStages : 0; j < issued; ++j)
                mbar_wait(&full[j % kStateStages], (j / kStateStages) & 1, kDefaultMaxSpin);
        }
    } else if (warp == 5) {
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(64, 64, true, true);
            int i = 0, run = 0;
            bool first_in_run = true;
            for (int64_t u = u0; u < u1; ++u, ++i) {
                const int s = i % kStateStages;
                const int h = (int)(u / part.nchunks);
                const bool last_in_run = (u + 1 == u1) || ((u + 1) / part.nchunks != h);
                if (!mbar_wait(&phi_ready[s], (i / kStateStages) & 1, max_spin)) {
                    report_timeout(hdr);
                    break;
                }
                if (first_in_run && run > 0 && !mbar_wait(&tmem_free, (run - 1) & 1, max_spin)) {
                    report_timeout(hdr);
                    break;
                }
                tc_fence_after();
                const uint32_t ka = smem_u32(stage_k[s]), va = smem_u32(stage_v[s]);
#pragma unroll
                for (int k16 = 0; k16 < kC / 16; ++k16) {
                    const uint64_t ad = smem_desc(ka + k16 * 2048, 1024, 1024, kSwizzle128B);
                    const uint64_t bd = smem_desc(va + k16 * 2048, 1024, 1024, kSwizzle128B);
                    mma_bf16(tmem, ad, bd, idesc, (first_in_run && k16 == 0) ? 0u : 1u);
                }
                mma_commit(&empty[s]);
                if (last_in_run) {
                    mma_commit(&run_done);
                    ++run;
                }
                first_in_run = last_in_run;
            }
            // Every issued MMA completes before TMEM is released.
            mma_commit(&mma_drain);
            mbar_wait(&mma_drain, 0, kDefaultMaxSpin);
        }
    } else {
        // Math warps 0-3 (128 threads). Every abort decision is made uniformly.
        const int t = tid;
        const int jgrp = (t & 7) ^ ((t >> 3) & 7);  // logical column group of this thread
        float zp[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) zp[e] = 0.f;
        int i = 0, run = 0;
        for (int64_t u = u0; u < u1; ++u, ++i) {
            const int s = i % kStateStages;
            const int h = (int)(u / part.nchunks), ch = (int)(u % part.nchunks);
            const bool last_in_run = (u + 1 == u1) || ((u + 1) / part.nchunks != h);
            const int valid = min(kC, N - ch * kC);
            bool ok = mbar_wait(&full[s], (i / kStateStages) & 1, max_spin);
            uint8_t* kt = stage_k[s];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int row = (t >> 3) + 16 * k;
                uint4* p = reinterpret_cast<uint4*>(kt + row * 128 + (t & 7) * 16);
                float f[8];
                *p = phi8(*p, f);
                if (row < valid) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) zp[e] += f[e];
                }
            }
            fence_proxy_async_smem();
            ok = named_bar_and(1, 128, ok);
            if (!ok) { if (t == 0) report_timeout(hdr); break; }
            if (t == 0) mbar_arrive(&phi_ready[s]);
            if (last_in_run) {
                // z: reduce the per-thread column-group partials.
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    float v = reduce_colgroup(zp[e]);
                    if ((lane >> 3) == 0) atomicAdd(&zsum[jgrp * 8 + e], v);
                    zp[e] = 0.f;
                }
                float* out = agg + ((int64_t)cta * part.maxr + run) * kE;
                ok = mbar_wait(&run_done, run & 1, max_spin);
                tc_fence_after();
                // dS (M = 64 layout): row 16 * warp + l lives in lane l < 16 of lane quarter `warp`.
                const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
                const int row = 16 * warp + (lane & 15);
#pragma unroll
                for (int cb = 0; cb < kD; cb += 16) {
                    uint32_t r[16];
                    tmem_ld16(tmem + lane_base + cb, r);
                    tmem_ld_wait();
                    if (lane < 16 && ok) {
                        float4* dst = reinterpret_cast<float4*>(out + row * kD + cb);
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            dst[q] = make_float4(__uint_as_float(r[4 * q]),
                                                 __uint_as_float(r[4 * q + 1]),
                                                 __uint_as_float(r[4 * q + 2]),
                                                 __uint_as_float(r[4 * q + 3]));
                    }
                }
                tc_fence_before();
                ok = named_bar_and(1, 128, ok);
                if (!ok) { if (t == 0) report_timeout(hdr); break; }
                if (t < kD) {
                    out[kD * kD + t] = zsum[t];
                    zsum[t] = 0.f;
                }
                named_bar(1, 128);
                if (t == 0) mbar_arrive(&tmem_free);
                ++run;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 64);
    }
}

// ======================================================== output kernel
// Warps 0-7: phi pass and epilogues (two warpgroups; warpgroup g takes half of
// the columns of every TMEM read). Warp 8: TMA producer. Warp 9: MMA issuer.

constexpr int kOutThreads = 320;
constexpr int kMath = 256;
// Shared-memory map (offsets from a 1024-aligned base).
constexpr uint32_t kOffStage = 0;                        // 2 stages x (Q, K, V) tiles
constexpr uint32_t kStageBytes = 3 * kTileBytes;
constexpr uint32_t kOffP = 2 * kStageBytes;              // masked A, bf16, 2 sub-tiles
constexpr uint32_t kOffSnap = kOffP + 2 * kTileBytes;    // 2 x S snapshot (64 x 64 bf16)
constexpr uint32_t kSnapBytes = kD * kD * 2;
constexpr uint32_t kOffO = kOffSnap + 2 * kSnapBytes;    // 2 x output staging tile
constexpr uint32_t kOffMisc = kOffO + 2 * kTileBytes;
constexpr size_t kOutSmem = 1024 + kOffMisc;

struct OutMisc {
    uint64_t full[2], empty[2], phi_ready[2], mma1_done[2], s_ready[2], p_ready[2],
        mma2_done[2], o_free[2], mma_drain;
    uint32_t tmem_slot;
    float zsnap[2][kD];         // z before chunk (index = chunk parity)
    float zpart[8][kD];         // per-warp column sums of phi(K_c)
    float den_part[2][kC];      // per-warpgroup partial denominators
};

__global__ void __launch_bounds__(kOutThreads, 1)
causal_output_kernel(const __grid_constant__ CUtensorMap qmap,
                     const __grid_constant__ CUtensorMap kmap,
                     const __grid_constant__ CUtensorMap vmap,
                     const __grid_constant__ CUtensorMap omap, const float* __restrict__ agg,
                     float* __restrict__ S_out, float* __restrict__ z_out, Partition part, int N,
                     float eps, WsHeader* hdr) {
    const uint32_t max_spin = hdr->max_spin;
    const bool hold = hdr->hold_item != 0;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    __shared__ OutMisc m;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cta = blockIdx.x;
    const int64_t u0 = part.begin(cta), u1 = part.begin(cta + 1);
    const int nch = (int)(u1 - u0);

    if (tid == 0) {
        for (int b = 0; b < 2; ++b) {
            mbar_init(&m.full[b], 1);
            mbar_init(&m.empty[b], 1);
            mbar_init(&m.phi_ready[b], 1);
            mbar_init(&m.mma1_done[b], 1);
            mbar_init(&m.s_ready[b], 1);
            mbar_init(&m.p_ready[b], 1);
            mbar_init(&m.mma2_done[b], 1);
            mbar_init(&m.o_free[b], 1);
        }
        mbar_init(&m.mma_drain, 1);
        fence_mbar_init();
    }
    if (warp == 9) {
        tmem_alloc(&m.tmem_slot, 512);
        tmem_relinquish();
    }
    if (warp == 8 && lane == 0) {
        tma_prefetch_desc(&qmap);
        tma_prefetch_desc(&kmap);
        tma_prefetch_desc(&vmap);
        tma_prefetch_desc(&omap);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = m.tmem_slot;
    // TMEM map per parity b: A at 256b + [0,128), dS at 256b + 128, O at 256b + 192.
    auto tA = [&](int b) { return tmem + 256u * b; };
    auto tS = [&](int b) { return tmem + 256u * b + 128u; };
    auto tO = [&](int b) { return tmem + 256u * b + 192u; };
    auto stage_q = [&](int s) { return base + kOffStage + s * kStageBytes; };
    auto stage_k = [&](int s) { return base + kOffStage + s * kStageBytes + kTileBytes; };
    auto stage_v = [&](int s) { return base + kOffStage + s * kStageBytes + 2 * kTileBytes; };
    uint8_t* sP = base + kOffP;
    auto snap = [&](int b) { return base + kOffSnap + b * kSnapBytes; };
    auto ostage = [&](int b) { return base + kOffO + b * kTileBytes; };

    if (warp == 8) {
        // ---------------------------------------------------------- producer
        if (lane == 0) {
            int i = 0;
            for (; i < nch; ++i) {
                const int s = i & 1;
                if (i >= 2 && !mbar_wait(&m.empty[s], ((i >> 1) - 1) & 1, max_spin)) {
                    report_timeout(hdr);
                    break;
                }
                if (hold) break;  // test hook: a load that is never issued
                const int64_t u = u0 + i;
                const int h = (int)(u / part.nchunks), ch = (int)(u % part.nchunks);
                mbar_arrive_expect_tx(&m.full[s], 3 * kTileBytes);
                tma_load_3d(stage_q(s), &qmap, &m.full[s], 0, ch * kC, h);
                tma_load_3d(stage_k(s), &kmap, &m.full[s], 0, ch * kC, h);
                tma_load_3d(stage_v(s), &vmap, &m.full[s], 0, ch * kC, h);
            }
            for (int j = i - 2 > 0 ? i - 2 : 0; j < i; ++j)
                mbar_wait(&m.full[j & 1], (j >> 1) & 1, kDefaultMaxSpin);
        }
    } else if (warp == 9) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t id_qk = idesc_bf16_f32(128, 128, false, false);
            const uint32_t id_kv = idesc_bf16_f32(64, 64, true, true);
            const uint32_t id_qs = idesc_bf16_f32(128, 64, false, true);
            const uint32_t id_pv = idesc_bf16_f32(128, 64, false, true);
            for (int i = 0; i < nch; ++i) {
                const int b = i & 1;
                const uint32_t par = (i >> 1) & 1;
                if (!mbar_wait(&m.phi_ready[b], par, max_spin)) { report_timeout(hdr); break; }
                tc_fence_after();
                const uint32_t qa = smem_u32(stage_q(b)), ka = smem_u32(stage_k(b)),
                               va = smem_u32(stage_v(b));
                // (1) A = phi(Q) phi(K)^T: M=128 queries, N=128 keys, K=64 features.
#pragma unroll
                for (int k16 = 0; k16 < kD / 16; ++k16)
                    mma_bf16(tA(b), smem_desc(qa + k16 * 32, 16, 1024, kSwizzle128B),
                             smem_desc(ka + k16 * 32, 16, 1024, kSwizzle128B), id_qk, k16 > 0);
                // (2) dS = phi(K)^T V: M=64 features, N=64 values, K=128 tokens.
#pragma unroll
                for (int k16 = 0; k16 < kC / 16; ++k16)
                    mma_bf16(tS(b), smem_desc(ka + k16 * 2048, 1024, 1024, kSwizzle128B),
                             smem_desc(va + k16 * 2048, 1024, 1024, kSwizzle128B), id_kv,
                             k16 > 0);
                mma_commit(&m.mma1_done[b]);
                // (3) O = phi(Q) S_prev: needs the snapshot and a free O accumulator.
                if (i >= 2 && !mbar_wait(&m.o_free[b], par ^ 1, max_spin)) {
                    report_timeout(hdr);
                    break;
                }
                if (!mbar_wait(&m.s_ready[b], par, max_spin)) { report_timeout(hdr); break; }
                tc_fence_after();
                const uint32_t sa = smem_u32(snap(b));
#pragma unroll
                for (int k16 = 0; k16 < kD / 16; ++k16)
                    mma_bf16(tO(b), smem_desc(qa + k16 * 32, 16, 1024, kSwizzle128B),
                             smem_desc(sa + k16 * 2048, 1024, 1024, kSwizzle128B), id_qs,
                             k16 > 0);
                // (4) O += P V: K = 128 keys (P in two 64-key sub-tiles).
                if (!mbar_wait(&m.p_ready[b], par, max_spin)) { report_timeout(hdr); break; }
                tc_fence_after();
                const uint32_t pa = smem_u32(sP);
#pragma unroll
                for (int k16 = 0; k16 < kC / 16; ++k16)
                    mma_bf16(tO(b),
                             smem_desc(pa + (k16 >> 2) * kTileBytes + (k16 & 3) * 32, 16, 1024,
                                       kSwizzle128B),
                             smem_desc(va + k16 * 2048, 1024, 1024, kSwizzle128B), id_pv, 1u);
                mma_commit(&m.mma2_done[b]);
                mma_commit(&m.empty[b]);
            }
            // Every issued MMA completes before TMEM is released.
            mma_commit(&m.mma_drain);
            mbar_wait(&m.mma_drain, 0, kDefaultMaxSpin);
        }
    } else {
        // ---------------------------------------------------------- math warps
        // Order per chunk i: (b)_i, then (a)_{i+1} (overlaps MMAs (3),(4) of i), then (c)_i.
        // Every abort decision is ANDed over the 256 math threads at a barrier.
        const int t = tid;                 // 0..255
        const int g = warp >> 2;           // warpgroup: column half
        const int q4 = warp & 3;           // TMEM lane quarter
        const int row = 32 * q4 + lane;    // query row of this thread (M = 128 layouts)
        const int srow = 16 * q4 + (lane & 15);  // state row (M = 64 layout), lanes < 16
        const bool sowner = lane < 16;
        const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
        const int jgrp = (t & 7) ^ ((t >> 3) & 7);
        float S_run[32];                   // state row srow, columns [32g, 32g + 32)

        // Start state of the first run: sum of the aggregates of this head's
        // chunks held by lower-numbered CTAs.
        auto load_prefix = [&](int64_t u_first) {
            const int h = (int)(u_first / part.nchunks);
            const int64_t head_begin = (int64_t)h * part.nchunks;
#pragma unroll
            for (int e = 0; e < 32; ++e) S_run[e] = 0.f;
            float zacc = 0.f;
            if (u_first > head_begin) {
                for (int c2 = cta - 1; c2 >= 0; --c2) {
                    const int64_t b0 = part.begin(c2), b1 = part.begin(c2 + 1);
                    if (b1 <= head_begin) break;
                    if (b1 <= b0) continue;
                    const int r = (int)(h - b0 / part.nchunks);
                    const float* a = agg + ((int64_t)c2 * part.maxr + r) * kE;
                    if (sowner) {
                        const float4* src =
                            reinterpret_cast<const float4*>(a + srow * kD + 32 * g);
#pragma unroll
                        for (int qd = 0; qd < 8; ++qd) {
                            float4 v = src[qd];
                            S_run[4 * qd] += v.x;
                            S_run[4 * qd + 1] += v.y;
                            S_run[4 * qd + 2] += v.z;
                            S_run[4 * qd + 3] += v.w;
                        }
                    }
                    if (t < kD) zacc += a[kD * kD + t];
                }
            }
            return zacc;
        };
        // Writes bf16(S_run) into snapshot buffer b (MN-major, row = feature, 64 values).
        auto write_snap = [&](int b) {
            if (!sowner) return;
            uint8_t* d = snap(b);
#pragma unroll
            for (int cq = 0; cq < 4; ++cq) {
                const int col = 32 * g + 8 * cq;
                uint4 v = make_uint4(pack_bf16(S_run[8 * cq], S_run[8 * cq + 1]),
                                     pack_bf16(S_run[8 * cq + 2], S_run[8 * cq + 3]),
                                     pack_bf16(S_run[8 * cq + 4], S_run[8 * cq + 5]),
                                     pack_bf16(S_run[8 * cq + 6], S_run[8 * cq + 7]));
                *reinterpret_cast<uint4*>(d + sw128_offset(srow, col)) = v;
            }
        };
        // (a) phi on Q and K of chunk i in place; per-warp column sums of phi(K) (valid rows).
        auto phase_a = [&](int i) -> bool {
            const int b = i & 1;
            const int64_t u = u0 + i;
            const int ch = (int)(u % part.nchunks);
            const int valid = min(kC, N - ch * kC);
            bool ok = mbar_wait(&m.full[b], (i >> 1) & 1, max_spin);
            float zp[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) zp[e] = 0.f;
            uint8_t* qt = stage_q(b);
            uint8_t* kt = stage_k(b);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int r = (t >> 3) + 32 * k;
                uint4* pq = reinterpret_cast<uint4*>(qt + r * 128 + (t & 7) * 16);
                float f[8];
                *pq = phi8(*pq, f);
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int r = (t >> 3) + 32 * k;
                uint4* pk = reinterpret_cast<uint4*>(kt + r * 128 + (t & 7) * 16);
                float f[8];
                *pk = phi8(*pk, f);
                if (r < valid) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) zp[e] += f[e];
                }
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                float v = reduce_colgroup(zp[e]);
                if ((lane >> 3) == 0) m.zpart[warp][jgrp * 8 + e] = v;
            }
            fence_proxy_async_smem();
            ok = named_bar_and(1, kMath, ok);
            if (ok && t == 0) mbar_arrive(&m.phi_ready[b]);
            return ok;
        };

        // Prologue: snapshot for chunk 0, then phi of chunk 0.
        bool ok = true;
        {
            float z0 = load_prefix(u0);
            if (t < kD) m.zsnap[0][t] = z0;
            write_snap(0);
            fence_proxy_async_smem();
            named_bar(1, kMath);
            if (t == 0) mbar_arrive(&m.s_ready[0]);
            if (nch > 0) ok = phase_a(0);
        }
        for (int i = 0; i < nch && ok; ++i) {
            const int b = i & 1;
            const uint32_t par = (i >> 1) & 1;
            const int64_t u = u0 + i;
            const int h = (int)(u / part.nchunks), ch = (int)(u % part.nchunks);
            const bool last_in_run = (u + 1 == u1) || ((u + 1) / part.nchunks != h);

            // (b) masked A -> P (bf16) and row sums; dS -> running state; denominators.
            ok = mbar_wait(&m.mma1_done[b], par, max_spin);
            tc_fence_after();
            float rs = 0.f;
            {
                uint8_t* pt = sP + g * kTileBytes;  // keys [64g, 64g + 64)
                if (g == 1 && q4 < 2) {
                    // Queries 0..63 see no key in 64..127.
#pragma unroll
                    for (int cq = 0; cq < 8; ++cq)
                        *reinterpret_cast<uint4*>(pt + sw128_offset(row, 8 * cq)) =
                            make_uint4(0, 0, 0, 0);
                } else {
#pragma unroll
                    for (int cb = 0; cb < 64; cb += 16) {
                        uint32_t r[16];
                        tmem_ld16(tA(b) + lane_base + 64 * g + cb, r);
                        tmem_ld_wait();
                        float a[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const int key = 64 * g + cb + e;
                            a[e] = key <= row ? __uint_as_float(r[e]) : 0.f;
                            rs += a[e];
                        }
#pragma unroll
                        for (int hq = 0; hq < 2; ++hq) {
                            uint4 v = make_uint4(pack_bf16(a[8 * hq], a[8 * hq + 1]),
                                                 pack_bf16(a[8 * hq + 2], a[8 * hq + 3]),
                                                 pack_bf16(a[8 * hq + 4], a[8 * hq + 5]),
                                                 pack_bf16(a[8 * hq + 6], a[8 * hq + 7]));
                            *reinterpret_cast<uint4*>(pt + sw128_offset(row, cb + 8 * hq)) = v;
                        }
                    }
                }
            }
            // phi(q_row) . z_prev over features [32g, 32g + 32).
            {
                const uint8_t* qt = stage_q(b);
                const float* zs = m.zsnap[b];
#pragma unroll
                for (int cq = 0; cq < 4; ++cq) {
                    const int col = 32 * g + 8 * cq;
                    uint4 v = *reinterpret_cast<const uint4*>(qt + sw128_offset(row, col));
                    const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        rs = fmaf(bf_lo(w4[e]), zs[col + 2 * e], rs);
                        rs = fmaf(bf_hi(w4[e]), zs[col + 2 * e + 1], rs);
                    }
                }
            }
            m.den_part[g][row] = rs;
            // dS read-out and state carry.
#pragma unroll
            for (int cb = 0; cb < 32; cb += 16) {
                uint32_t r[16];
                tmem_ld16(tS(b) + lane_base + 32 * g + cb, r);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 16; ++e) S_run[cb + e] += __uint_as_float(r[e]);
            }
            tc_fence_before();
            ok = named_bar_and(1, kMath, ok);   // zpart, den_part complete
            if (!ok) break;
            const int nb = b ^ 1;
            if (last_in_run) {
                // Final state of the head if its last chunk is here.
                const bool head_end = (ch == part.nchunks - 1);
                if (head_end && S_out && sowner) {
                    float4* dst = reinterpret_cast<float4*>(
                        S_out + ((int64_t)h * kD + srow) * kD + 32 * g);
#pragma unroll
                    for (int qd = 0; qd < 8; ++qd)
                        dst[qd] = make_float4(S_run[4 * qd], S_run[4 * qd + 1],
                                              S_run[4 * qd + 2], S_run[4 * qd + 3]);
                }
                if (t < kD) {
                    float zc = 0.f;
#pragma unroll
                    for (int w = 0; w < 8; ++w) zc += m.zpart[w][t];
                    if (head_end && z_out) z_out[(int64_t)h * kD + t] = m.zsnap[b][t] + zc;
                    m.zsnap[nb][t] = 0.f;  // the next run (if any) starts a new head
                }
#pragma unroll
                for (int e = 0; e < 32; ++e) S_run[e] = 0.f;
            } else if (t < kD) {
                float zc = 0.f;
#pragma unroll
                for (int w = 0; w < 8; ++w) zc += m.zpart[w][t];
                m.zsnap[nb][t] = m.zsnap[b][t] + zc;
            }
            if (i + 1 < nch) write_snap(nb);
            const float den = m.den_part[0][row] + m.den_part[1][row] + eps;
            if (t == 0) tma_store_wait_read<1>();  // staging buffer b is free again
            fence_proxy_async_smem();
            named_bar(1, kMath);
            if (t == 0) {
                mbar_arrive(&m.p_ready[b]);
                if (i + 1 < nch) mbar_arrive(&m.s_ready[nb]);
            }

            // (a) of the next chunk while the tensor core finishes this one.
            if (i + 1 < nch) {
                ok = phase_a(i + 1);
                if (!ok) break;
            }

            // (c) O / den -> bf16 -> staging tile -> TMA store.
            ok = mbar_wait(&m.mma2_done[b], par, max_spin);
            tc_fence_after();
            {
                const float inv = 1.f / den;
                uint8_t* ot = ostage(b);
#pragma unroll
                for (int cb = 0; cb < 32; cb += 16) {
                    uint32_t r[16];
                    tmem_ld16(tO(b) + lane_base + 32 * g + cb, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int hq = 0; hq < 2; ++hq) {
                        const int e0 = 8 * hq;
                        uint4 v = make_uint4(
                            pack_bf16(__uint_as_float(r[e0]) * inv,
                                      __uint_as_float(r[e0 + 1]) * inv),
                            pack_bf16(__uint_as_float(r[e0 + 2]) * inv,
                                      __uint_as_float(r[e0 + 3]) * inv),
                            pack_bf16(__uint_as_float(r[e0 + 4]) * inv,
                                      __uint_as_float(r[e0 + 5]) * inv),
                            pack_bf16(__uint_as_float(r[e0 + 6]) * inv,
                                      __uint_as_float(r[e0 + 7]) * inv));
                        *reinterpret_cast<uint4*>(ot + sw128_offset(row, 32 * g + cb + e0)) = v;
                    }
                }
            }
            tc_fence_before();
            fence_proxy_async_smem();
            ok = named_bar_and(1, kMath, ok);
            if (ok && t == 0) {
                mbar_arrive(&m.o_free[b]);
                tma_store_3d(&omap, ostage(b), 0, ch * kC, h);
                tma_store_commit();
            }
        }
        if (!ok && t == 0) report_timeout(hdr);
        if (t == 0) tma_store_wait_all<0>();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ---------------------------------------------------------------- host side

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                 const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                 const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled get_encoder() {
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
bool encode_bhnd(CUtensorMap* map, const void* ptr, int64_t BH, int N, int D) {
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

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        return 148;
    return n;
}

}  // namespace

bool tc_causal_supported(int D, int M, la_dtype dt) { return dt == LA_BF16 && D == 64 && M == 64; }

size_t tc_causal_workspace(int64_t BH, int N) {
    Partition p = make_partition(BH, N, sm_count());
    return sizeof(float) * (size_t)p.grid * p.maxr * kE;
}

int tc_causal_launches() { return 2; }

cudaError_t tc_causal(const void* q, const void* k, const void* v, void* o, int64_t BH, int N,
                      float eps, float* S_out, float* z_out, void* ws_header, void* scratch,
                      cudaStream_t st) {
    Partition p = make_partition(BH, N, sm_count());
    CUtensorMap qm, km, vm, om;
    if (!encode_bhnd(&qm, q, BH, N, kD) || !encode_bhnd(&km, k, BH, N, kD) ||
        !encode_bhnd(&vm, v, BH, N, kD) || !encode_bhnd(&om, o, BH, N, kD))
        return cudaErrorInvalidValue;
    WsHeader* hdr = reinterpret_cast<WsHeader*>(ws_header);
    float* agg = reinterpret_cast<float*>(scratch);
    cudaError_t err;
    if ((err = cudaFuncSetAttribute(causal_state_kernel,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)kStateSmem)))
        return err;
    if ((err = cudaFuncSetAttribute(causal_output_kernel,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kOutSmem)))
        return err;
    causal_state_kernel<<<p.grid, kStateThreads, kStateSmem, st>>>(km, vm, agg, p, N, hdr);
    causal_output_kernel<<<p.grid, kOutThreads, kOutSmem, st>>>(qm, km, vm, om, agg, S_out,
                                                                 z_out, p, N, eps, hdr);
    return cudaPeekAtLastError();
}

}  // namespace la
