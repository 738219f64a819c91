// Tensor-core (tcgen05) causal forward for bf16 inputs, Dk = Dv = 64.
//
// Method. For chunk c of 128 tokens of one head, with S_{c-1}, z_{c-1} the
// state after the previous chunks ("Why Replace Attention? The Softmax
// Bottleneck and the Path to Linear Time", section 7.1: S_i and z_i are
// prefix sums, so a whole chunk can be added at once):
//   P      = bf16( mask_{key <= query}( phi(Q_c) phi(K_c)^T ) )
//   [num | den] = phi(Q_c) [S_{c-1} | z_{c-1}] + P [V_c | 1]
//   o_i    = num_i / (den_i + eps)
//   [S_c | z_c] = [S_{c-1} | z_{c-1}] + phi(K_c)^T [V_c | 1]
// This is an exact regrouping of S_i = sum_{j<=i} phi(k_j) v_j^T and
// z_i = sum_{j<=i} phi(k_j) (same blog, section 7.2) into whole chunks plus a
// masked in-chunk part. Appending a column of ones to V (and z to S) makes
// every denominator and every z a by-product of the same tensor-core
// contractions as the numerators, so num and den see identical weights.
// z enters the MMA as two bf16 terms (z_hi + z_lo), which keeps it accurate to
// fp32 level; S_{c-1} enters as bf16.
//
// Work split. The B*H*ceil(N/128) chunks form one head-major sequence cut into
// gridDim.x contiguous ranges, one per persistent CTA. A range holds "runs"
// (its chunks of one head). Two launches share that partition:
//   state kernel   per run: [dS | dz] = phi(K)^T [V | 1]  -> workspace (fp32)
//   output kernel  per run: start state = sum of the dS, dz of the same head
//                  from lower-numbered CTAs (only a range's first run can have
//                  one), then the chunk loop above with the state in registers.
// The sum over earlier ranges is the exclusive prefix over segments (the
// parallel scan of the same blog, section 7.7), in fp32. The output kernel is
// launched as a programmatic dependent of the state kernel: everything up to
// the prefix read overlaps the state kernel's tail.
//
// Data movement: TMA 3-D tiles (64 features x 128 tokens x 1 head, 128-byte
// swizzle) into shared memory; phi is applied in place in shared memory with
// packed bf16x2 arithmetic; every contraction is a tcgen05.mma (bf16 operands,
// fp32 accumulators in TMEM); outputs leave through a swizzled staging tile and
// a TMA store, which drops rows past N.
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_util.cuh"

namespace la {

namespace {

using namespace tc;

constexpr int kC = 128;                        // tokens per chunk
constexpr int kD = 64;                         // Dk = Dv
constexpr int kNx = 80;                        // MMA N with the extra ones / z columns
constexpr uint32_t kTileBytes = kC * kD * 2;   // one bf16 [128 x 64] tile = 16 KB
constexpr int kE = kD * kD + kD;               // floats per aggregate (S then z)

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

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %2, %1;" : "=r"(r) : "f"(a), "f"(b));
    return r;
}

__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }

// phi(x) = max(x, 0) + min(2^(x log2 e), 1) on two packed bf16 values: equal
// to x + 1 for x > 0 and e^x for x <= 0 (e^x >= 1 exactly when x >= 0).
// x log2 e is formed as x*c_hi + x*c_lo with c_hi + c_lo = log2 e to about
// 2^-17, rounded once to bf16; the power of two is the hardware ex2.
__device__ __forceinline__ uint32_t phi_bf16x2(uint32_t x) {
    constexpr uint32_t kLog2eHi = 0x3FB93FB9u;  // bf16(log2 e) = 1.4453125, twice
    constexpr uint32_t kLog2eLo = 0xBB2CBB2Cu;  // bf16(log2 e - 1.4453125) = -0.00262451, twice
    constexpr uint32_t kOne = 0x3F803F80u;
    constexpr uint32_t kNegZero = 0x80008000u;
    uint32_t lo, t, e, m, p, r;
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(lo) : "r"(x), "r"(kLog2eLo), "r"(kNegZero));
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(t) : "r"(x), "r"(kLog2eHi), "r"(lo));
    asm("ex2.approx.ftz.bf16x2 %0, %1;" : "=r"(e) : "r"(t));
    asm("min.bf16x2 %0, %1, %2;" : "=r"(m) : "r"(e), "r"(kOne));
    asm("max.bf16x2 %0, %1, %2;" : "=r"(p) : "r"(x), "r"(0u));
    asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(p), "r"(m));
    return r;
}

__device__ __forceinline__ uint4 phi8(uint4 u) {
    return make_uint4(phi_bf16x2(u.x), phi_bf16x2(u.y), phi_bf16x2(u.z), phi_bf16x2(u.w));
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

// phi in place on the 128 x 64 bf16 tile rows (t >> 3) + 32 k, physical chunk
// (t & 7), for a 256-thread group; rows >= zero_from are set to 0.
__device__ __forceinline__ void phi_tile_256(uint8_t* tile, int t, int zero_from) {
    uint4 v[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
        v[k] = *reinterpret_cast<const uint4*>(tile + ((t >> 3) + 32 * k) * 128 + (t & 7) * 16);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int r = (t >> 3) + 32 * k;
        const uint4 o = r < zero_from ? phi8(v[k]) : make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(tile + r * 128 + (t & 7) * 16) = o;
    }
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

// ======================================================== state kernel
// Warps 0-7: phi pass and aggregate read-out. Warp 8: TMA producer. Warp 9: MMA.

constexpr int kStateStages = 4;
constexpr int kStateThreads = 320;
constexpr uint32_t kStateOnes = kStateStages * 2 * kTileBytes;
constexpr size_t kStateSmem = 1024 + kStateOnes + kTileBytes;

__global__ void __launch_bounds__(kStateThreads, 1)
causal_state_kernel(const __grid_constant__ CUtensorMap kmap,
                    const __grid_constant__ CUtensorMap vmap, float* __restrict__ agg,
                    Partition part, int N, WsHeader* hdr) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    __shared__ uint64_t full[kStateStages], empty[kStateStages], phi_ready[kStateStages];
    __shared__ uint64_t run_done, tmem_free, mma_drain;
    __shared__ uint32_t tmem_slot;

    pdl_launch_dependents();
    const uint32_t max_spin = hdr->max_spin;
    const bool hold = hdr->hold_item != 0;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cta = blockIdx.x;
    const int64_t u0 = part.begin(cta), u1 = part.begin(cta + 1);
    auto stage_k = [&](int s) { return base + s * 2 * kTileBytes; };
    auto stage_v = [&](int s) { return base + s * 2 * kTileBytes + kTileBytes; };
    uint8_t* ones = base + kStateOnes;

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
    if (warp < 8) init_ones_tile(ones, tid, 256);
    fence_proxy_async_smem();
    if (warp == 9) {
        tmem_alloc(&tmem_slot, 128);
        tmem_relinquish();
    }
    if (warp == 8 && lane == 0) {
        tma_prefetch_desc(&kmap);
        tma_prefetch_desc(&vmap);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;

    if (warp == 8) {
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
                tma_load_3d(stage_k(s), &kmap, &full[s], 0, ch * kC, h);
                tma_load_3d(stage_v(s), &vmap, &full[s], 0, ch * kC, h);
            }
            // Every issued load lands before the CTA may exit.
            for (int j = i - kStateStages > 0 ? i - kStateStages : 0; j < i; ++j)
                mbar_wait(&full[j % kStateStages], (j / kStateStages) & 1, kDefaultMaxSpin);
        }
    } else if (warp == 9) {
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(64, kNx, true, true);
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
                const uint32_t ka = smem_u32(stage_k(s)), va = smem_u32(stage_v(s));
                const uint32_t lbo = smem_u32(ones) - va;  // [V | 1]: second MN atom
#pragma unroll
                for (int k16 = 0; k16 < kC / 16; ++k16)
                    mma_bf16(tmem, smem_desc(ka + k16 * 2048, 1024, 1024, kSwizzle128B),
                             smem_desc(va + k16 * 2048, lbo, 1024, kSwizzle128B), idesc,
                             (first_in_run && k16 == 0) ? 0u : 1u);
                mma_commit(&empty[s]);
                if (last_in_run) {
                    mma_commit(&run_done);
                    ++run;
                }
                first_in_run = last_in_run;
            }
            mma_commit(&mma_drain);  // every issued MMA completes before TMEM is released
            mbar_wait(&mma_drain, 0, kDefaultMaxSpin);
        }
    } else {
        // Math warps 0-7 (256 threads); abort decisions are uniform.
        const int t = tid;
        const int g = warp >> 2, q4 = warp & 3;
        const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
        const int srow = 16 * q4 + (lane & 15);  // dS row (M = 64 layout), lanes < 16
        int i = 0, run = 0;
        for (int64_t u = u0; u < u1; ++u, ++i) {
            const int s = i % kStateStages;
            const int h = (int)(u / part.nchunks), ch = (int)(u % part.nchunks);
            const bool last_in_run = (u + 1 == u1) || ((u + 1) / part.nchunks != h);
            const int valid = min(kC, N - ch * kC);
            bool ok = mbar_wait(&full[s], (i / kStateStages) & 1, max_spin);
            phi_tile_256(stage_k(s), t, valid);
            fence_proxy_async_smem();
            ok = named_bar_and(1, 256, ok);
            if (!ok) { if (t == 0) report_timeout(hdr); break; }
            if (t == 0) mbar_arrive(&phi_ready[s]);
            if (last_in_run) {
                float* out = agg + ((int64_t)cta * part.maxr + run) * kE;
                ok = mbar_wait(&run_done, run & 1, max_spin);
                tc_fence_after();
                uint32_t r0[16], r1[16], rz[16];
                tmem_ld16(tmem + lane_base + 32 * g, r0);
                tmem_ld16(tmem + lane_base + 32 * g + 16, r1);
                tmem_ld16(tmem + lane_base + 64, rz);
                tmem_ld_wait();
                if (lane < 16 && ok) {
                    float4* dst = reinterpret_cast<float4*>(out + srow * kD + 32 * g);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        dst[q] = make_float4(__uint_as_float(r0[4 * q]), __uint_as_float(r0[4 * q + 1]),
                                             __uint_as_float(r0[4 * q + 2]), __uint_as_float(r0[4 * q + 3]));
                        dst[q + 4] = make_float4(__uint_as_float(r1[4 * q]), __uint_as_float(r1[4 * q + 1]),
                                                 __uint_as_float(r1[4 * q + 2]), __uint_as_float(r1[4 * q + 3]));
                    }
                    if (g == 0) out[kD * kD + srow] = __uint_as_float(rz[0]);
                }
                tc_fence_before();
                ok = named_bar_and(1, 256, ok);
                if (!ok) { if (t == 0) report_timeout(hdr); break; }
                if (t == 0) mbar_arrive(&tmem_free);
                ++run;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 128);
    }
}

// ======================================================== output kernel
// Warp roles (14 warps):
//   warps 0-3   phi:   phi on the Q and K tiles of each landed stage, in place
//   warps 4-7   mask:  A -> causal mask -> bf16 P (shared memory), per chunk
//   warps 8-11  state: [dS | dz] -> running state -> next snapshot; then the
//                      output epilogue num / (den + eps) -> TMA store
//   warp 12     TMA producer       warp 13  MMA issuer (one thread)
// The four warps of a role cover the four TMEM lane quarters.

constexpr int kOutThreads = 448;
constexpr int kStages = 3;
// Shared-memory map (offsets from a 1024-aligned base).
constexpr uint32_t kStageBytes = 3 * kTileBytes;               // Q, K, V tiles
constexpr uint32_t kOffP = kStages * kStageBytes;              // masked A, bf16, 2 sub-tiles
constexpr uint32_t kSnapS = kD * 128;                          // S snapshot: 64 rows x 128 B
constexpr uint32_t kSnapZ = 16 * 128;                          // z tile: 16 rows x 128 B (K-major)
constexpr uint32_t kSnapBytes = kSnapS + kSnapZ;
constexpr uint32_t kOffSnap = kOffP + 2 * kTileBytes;          // 2 x (S | z)
constexpr uint32_t kOffOnes = kOffSnap + 2 * kSnapBytes;       // ones: 16 rows x 128 keys, K-major
constexpr uint32_t kOnesBytes = 2 * 16 * 128;
constexpr uint32_t kOffO = kOffOnes + kOnesBytes;              // output staging tile
constexpr uint32_t kSmemEnd = kOffO + kTileBytes;
constexpr size_t kOutSmem = 1024 + kSmemEnd;
// TMEM columns: A[b] at 128 b; O[b] = [num 64 | den 16] at 256 + 96 b; dS = [dS 64 | dz 16] at 432.
constexpr uint32_t kTmO = 256, kTmOStride = 96, kTmS = 432;

struct OutMisc {
    uint64_t full[kStages], phi_done[kStages], empty[kStages];
    uint64_t a_full[2], a_free[2], o_full[2], o_free[2], snap_full[2];
    uint64_t p_full, p_free, ds_full, ds_free, state_init, mma_drain;
    uint32_t tmem_slot;
};

// K-major "ones" operand: row 0 = 1.0 over 128 keys (two 64-key sub-tiles), rows 1-15 = 0.
__device__ __forceinline__ void init_ones_kmajor(uint8_t* t, int tid, int nthreads) {
    for (int idx = tid; idx < 2 * 16 * 8; idx += nthreads) {
        const int sub = idx / 128, r = (idx / 8) % 16, pc = idx % 8;
        const uint32_t one = r == 0 ? 0x3F803F80u : 0u;
        *reinterpret_cast<uint4*>(t + sub * 2048 + r * 128 + pc * 16) = make_uint4(one, one, one, one);
    }
}

__global__ void __launch_bounds__(kOutThreads, 1)
causal_output_kernel(const __grid_constant__ CUtensorMap qmap,
                     const __grid_constant__ CUtensorMap kmap,
                     const __grid_constant__ CUtensorMap vmap,
                     const __grid_constant__ CUtensorMap omap, const float* __restrict__ agg,
                     float* __restrict__ S_out, float* __restrict__ z_out, Partition part, int N,
                     float eps, WsHeader* hdr) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    __shared__ OutMisc m;
    const uint32_t max_spin = hdr->max_spin;
    const bool hold = hdr->hold_item != 0;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cta = blockIdx.x;
    const int64_t u0 = part.begin(cta), u1 = part.begin(cta + 1);
    const int nch = (int)(u1 - u0);
    auto stage_q = [&](int s) { return base + s * kStageBytes; };
    auto stage_k = [&](int s) { return base + s * kStageBytes + kTileBytes; };
    auto stage_v = [&](int s) { return base + s * kStageBytes + 2 * kTileBytes; };
    uint8_t* sP = base + kOffP;
    auto snap_s = [&](int b) { return base + kOffSnap + b * kSnapBytes; };
    auto snap_z = [&](int b) { return base + kOffSnap + b * kSnapBytes + kSnapS; };
    uint8_t* ones = base + kOffOnes;
    uint8_t* ostage = base + kOffO;

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&m.full[s], 1);
            mbar_init(&m.phi_done[s], 1);
            mbar_init(&m.empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&m.a_full[b], 1);
            mbar_init(&m.a_free[b], 1);
            mbar_init(&m.o_full[b], 1);
            mbar_init(&m.o_free[b], 1);
            mbar_init(&m.snap_full[b], 1);
        }
        mbar_init(&m.p_full, 1);
        mbar_init(&m.p_free, 1);
        mbar_init(&m.ds_full, 1);
        mbar_init(&m.ds_free, 1);
        mbar_init(&m.state_init, 1);
        mbar_init(&m.mma_drain, 1);
        fence_mbar_init();
    }
    if (warp < 12) {
        init_ones_kmajor(ones, tid, 384);
        for (int idx = tid; idx < 2 * (int)kSnapZ / 16; idx += 384) {  // both z tiles
            const int b = idx / (kSnapZ / 16), r = idx % (kSnapZ / 16);
            *reinterpret_cast<uint4*>(snap_z(b) + r * 16) = make_uint4(0, 0, 0, 0);
        }
    }
    fence_proxy_async_smem();
    if (warp == 13) {
        tmem_alloc(&m.tmem_slot, 512);
        tmem_relinquish();
    }
    if (warp == 12 && lane == 0) {
        tma_prefetch_desc(&qmap);
        tma_prefetch_desc(&kmap);
        tma_prefetch_desc(&vmap);
        tma_prefetch_desc(&omap);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = m.tmem_slot;
    const int q4 = warp & 3;                       // TMEM lane quarter of this warp
    const uint32_t lane_base = (uint32_t)(32 * q4) << 16;

    if (warp == 12) {
        // ---------------------------------------------------------- producer
        if (lane == 0) {
            int i = 0;
            for (; i < nch; ++i) {
                const int s = i % kStages;
                if (i >= kStages &&
                    !mbar_wait(&m.empty[s], ((i / kStages) - 1) & 1, max_spin)) {
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
            for (int j = i - kStages > 0 ? i - kStages : 0; j < i; ++j)
                mbar_wait(&m.full[j % kStages], (j / kStages) & 1, kDefaultMaxSpin);
        }
    } else if (warp == 13) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t id_qk = idesc_bf16_f32(128, 128, false, false);
            const uint32_t id_kv = idesc_bf16_f32(64, 64, true, true);
            const uint32_t id_k1 = idesc_bf16_f32(64, 16, true, false);
            const uint32_t id_o = idesc_bf16_f32(128, 64, false, true);
            const uint32_t id_o1 = idesc_bf16_f32(128, 16, false, false);
            const uint32_t onesa = smem_u32(ones), pa = smem_u32(sP);
            const uint32_t tS = tmem + kTmS;
            for (int i = 0; i < nch; ++i) {
                const int s = i % kStages, b = i & 1;
                const uint32_t pb = (i >> 1) & 1, pi = i & 1;
                const uint32_t tA = tmem + 128u * b, tO = tmem + kTmO + kTmOStride * b;
                if (!mbar_wait(&m.phi_done[s], (i / kStages) & 1, max_spin)) { report_timeout(hdr); break; }
                if (i >= 2 && !mbar_wait(&m.a_free[b], pb ^ 1, max_spin)) { report_timeout(hdr); break; }
                tc_fence_after();
                const uint32_t qa = smem_u32(stage_q(s)), ka = smem_u32(stage_k(s)),
                               va = smem_u32(stage_v(s));
                // (1) A = phi(Q) phi(K)^T: M=128 queries, N=128 keys, K=64 features.
#pragma unroll
                for (int k16 = 0; k16 < kD / 16; ++k16)
                    mma_bf16(tA, smem_desc(qa + k16 * 32, 16, 1024, kSwizzle128B),
                             smem_desc(ka + k16 * 32, 16, 1024, kSwizzle128B), id_qk, k16 > 0);
                mma_commit(&m.a_full[b]);
                // (2) S += phi(K)^T V (M=64, N=64) and (2b) z += phi(K)^T 1 (N=16), K=128
                // tokens: the running state [S | z] of the current run lives in TMEM. The
                // first run starts from the state written by the state role; a later run
                // starts a new head from zero.
                const int64_t u = u0 + i;
                const bool run_start = (u % part.nchunks == 0);
                if (i == 0 && !mbar_wait(&m.state_init, 0, max_spin)) { report_timeout(hdr); break; }
                if (i >= 1 && !mbar_wait(&m.ds_free, pi ^ 1, max_spin)) { report_timeout(hdr); break; }
                tc_fence_after();
                const bool fresh = (i > 0 && run_start);
#pragma unroll
                for (int k16 = 0; k16 < kC / 16; ++k16) {
                    const uint64_t kd = smem_desc(ka + k16 * 2048, 1024, 1024, kSwizzle128B);
                    const uint32_t acc = (fresh && k16 == 0) ? 0u : 1u;
                    mma_bf16(tS, kd, smem_desc(va + k16 * 2048, 1024, 1024, kSwizzle128B), id_kv,
                             acc);
                    mma_bf16(tS + 64, kd,
                             smem_desc(onesa + (k16 >> 2) * 2048 + (k16 & 3) * 32, 16, 1024,
                                       kSwizzle128B),
                             id_k1, acc);
                }
                mma_commit(&m.ds_full);
                // (3) num = phi(Q) S_prev and (3b) den = phi(Q) [z_hi; z_lo]: needs the snapshot, free O.
                if (!mbar_wait(&m.snap_full[b], pb, max_spin)) { report_timeout(hdr); break; }
                if (i >= 2 && !mbar_wait(&m.o_free[b], pb ^ 1, max_spin)) { report_timeout(hdr); break; }
                tc_fence_after();
                const uint32_t sa = smem_u32(snap_s(b)), za = smem_u32(snap_z(b));
#pragma unroll
                for (int k16 = 0; k16 < kD / 16; ++k16) {
                    const uint64_t qd = smem_desc(qa + k16 * 32, 16, 1024, kSwizzle128B);
                    mma_bf16(tO, qd, smem_desc(sa + k16 * 2048, 1024, 1024, kSwizzle128B), id_o,
                             k16 > 0);
                    mma_bf16(tO + 64, qd, smem_desc(za + k16 * 32, 16, 1024, kSwizzle128B), id_o1,
                             k16 > 0);
                }
                // (4) num += P V and (4b) den += P 1: K = 128 keys (P in two 64-key sub-tiles).
                if (!mbar_wait(&m.p_full, pi, max_spin)) { report_timeout(hdr); break; }
                tc_fence_after();
#pragma unroll
                for (int k16 = 0; k16 < kC / 16; ++k16) {
                    const uint64_t pd = smem_desc(pa + (k16 >> 2) * kTileBytes + (k16 & 3) * 32, 16,
                                                  1024, kSwizzle128B);
                    mma_bf16(tO, pd, smem_desc(va + k16 * 2048, 1024, 1024, kSwizzle128B), id_o, 1u);
                    mma_bf16(tO + 64, pd,
                             smem_desc(onesa + (k16 >> 2) * 2048 + (k16 & 3) * 32, 16, 1024,
                                       kSwizzle128B),
                             id_o1, 1u);
                }
                mma_commit(&m.o_full[b]);
                mma_commit(&m.p_free);
                mma_commit(&m.empty[s]);
            }
            mma_commit(&m.mma_drain);  // every issued MMA completes before TMEM is released
            mbar_wait(&m.mma_drain, 0, kDefaultMaxSpin);
        }
    } else if (warp < 4) {
        // ---------------------------------------------------------- phi role
        const int t = tid;  // 0..127
        bool ok = true;
        for (int i = 0; i < nch; ++i) {
            const int s = i % kStages;
            const int ch = (int)((u0 + i) % part.nchunks);
            const int valid = min(kC, N - ch * kC);
            ok = mbar_wait(&m.full[s], (i / kStages) & 1, max_spin);
            uint8_t* qt = stage_q(s);
            uint8_t* kt = stage_k(s);
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint4 vq[4], vk[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int r = (t >> 3) + 16 * (4 * half + k);
                    vq[k] = *reinterpret_cast<const uint4*>(qt + r * 128 + (t & 7) * 16);
                    vk[k] = *reinterpret_cast<const uint4*>(kt + r * 128 + (t & 7) * 16);
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int r = (t >> 3) + 16 * (4 * half + k);
                    *reinterpret_cast<uint4*>(qt + r * 128 + (t & 7) * 16) = phi8(vq[k]);
                    *reinterpret_cast<uint4*>(kt + r * 128 + (t & 7) * 16) =
                        r < valid ? phi8(vk[k]) : make_uint4(0, 0, 0, 0);
                }
            }
            fence_proxy_async_smem();
            ok = named_bar_and(1, 128, ok);
            if (!ok) break;
            if (t == 0) mbar_arrive(&m.phi_done[s]);
        }
        if (!ok && t == 0) report_timeout(hdr);
    } else if (warp < 8) {
        // ---------------------------------------------------------- mask role
        const int row = 32 * q4 + lane;  // query row
        const int t = tid - 128;
        bool ok = true;
        for (int i = 0; i < nch; ++i) {
            const int b = i & 1;
            const uint32_t pb = (i >> 1) & 1;
            const uint32_t tA = tmem + 128u * b;
            ok = mbar_wait(&m.a_full[b], pb, max_spin);
            if (i >= 1) ok = mbar_wait(&m.p_free, (i - 1) & 1, max_spin) && ok;
            tc_fence_after();
            // Key block j (32 keys): j < q4 fully visible, j == q4 holds the diagonal, j > q4 masked.
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint8_t* pt = sP + (j >> 1) * kTileBytes;
                const int col0 = 32 * (j & 1);
                if (j > q4) {
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        *reinterpret_cast<uint4*>(pt + sw128_offset(row, col0 + 8 * c)) =
                            make_uint4(0, 0, 0, 0);
                    continue;
                }
                uint32_t r0[16], r1[16];
                tmem_ld16(tA + lane_base + 32 * j, r0);
                tmem_ld16(tA + lane_base + 32 * j + 16, r1);
                tmem_ld_wait();
                float a[32];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    a[e] = __uint_as_float(r0[e]);
                    a[16 + e] = __uint_as_float(r1[e]);
                }
                if (j == q4) {
#pragma unroll
                    for (int e = 0; e < 32; ++e) a[e] = (e <= lane) ? a[e] : 0.f;
                }
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint4 v = make_uint4(pack_bf16(a[8 * c], a[8 * c + 1]),
                                         pack_bf16(a[8 * c + 2], a[8 * c + 3]),
                                         pack_bf16(a[8 * c + 4], a[8 * c + 5]),
                                         pack_bf16(a[8 * c + 6], a[8 * c + 7]));
                    *reinterpret_cast<uint4*>(pt + sw128_offset(row, col0 + 8 * c)) = v;
                }
            }
            tc_fence_before();
            fence_proxy_async_smem();
            ok = named_bar_and(2, 128, ok);
            if (!ok) break;
            if (t == 0) {
                mbar_arrive(&m.a_free[b]);
                mbar_arrive(&m.p_full);
            }
        }
        if (!ok && t == 0) report_timeout(hdr);
    } else {
        // ---------------------------------------------------------- state + output role
        // The running state [S | z] is accumulated in TMEM by the MMAs (2), (2b)
        // (M = 64 layout: state row r in lane 32 (r / 16) + r % 16). This role
        // writes the first run's start state, reads the state after every chunk
        // into the bf16 snapshot used by the next chunk's MMA (3), and writes the
        // outputs.
        const int t = tid - 256;                    // 0..127
        const int row = 32 * q4 + lane;             // query row (M = 128 layout)
        const int srow = 16 * q4 + (lane & 15);     // state row (M = 64 layout), lanes < 16
        const bool sowner = lane < 16;
        const uint32_t tS = tmem + kTmS + lane_base;

        // Start state of the first run: sum of the aggregates of this head's
        // chunks held by lower-numbered CTAs (written by the state kernel), into
        // TMEM and into snapshot 0.
        pdl_wait();  // the state kernel's aggregates are complete and visible
        {
            const int h = (int)(u0 / part.nchunks);
            const int64_t head_begin = (int64_t)h * part.nchunks;
            float S0[kD];
            float z0 = 0.f;
#pragma unroll
            for (int e = 0; e < kD; ++e) S0[e] = 0.f;
            if (u0 > head_begin && sowner) {
                for (int c2 = cta - 1; c2 >= 0; --c2) {
                    const int64_t b0 = part.begin(c2), b1 = part.begin(c2 + 1);
                    if (b1 <= head_begin) break;
                    if (b1 <= b0) continue;
                    const int r = (int)(h - b0 / part.nchunks);
                    const float* a = agg + ((int64_t)c2 * part.maxr + r) * kE;
                    const float4* src = reinterpret_cast<const float4*>(a + srow * kD);
#pragma unroll
                    for (int qd = 0; qd < kD / 4; ++qd) {
                        float4 v = src[qd];
                        S0[4 * qd] += v.x;
                        S0[4 * qd + 1] += v.y;
                        S0[4 * qd + 2] += v.z;
                        S0[4 * qd + 3] += v.w;
                    }
                    z0 += a[kD * kD + srow];
                }
            }
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t w[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) w[e] = __float_as_uint(S0[16 * c + e]);
                tmem_st16(tS + 16 * c, w);
            }
            {
                uint32_t w[16];
                w[0] = __float_as_uint(z0);
#pragma unroll
                for (int e = 1; e < 16; ++e) w[e] = 0u;
                tmem_st16(tS + 64, w);
            }
            tmem_st_wait();
            if (sowner) {
                uint8_t* d = snap_s(0);
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint4 v = make_uint4(pack_bf16(S0[8 * c], S0[8 * c + 1]),
                                         pack_bf16(S0[8 * c + 2], S0[8 * c + 3]),
                                         pack_bf16(S0[8 * c + 4], S0[8 * c + 5]),
                                         pack_bf16(S0[8 * c + 6], S0[8 * c + 7]));
                    *reinterpret_cast<uint4*>(d + sw128_offset(srow, 8 * c)) = v;
                }
                const uint32_t hi = pack_bf16(z0, 0.f);
                const uint32_t lo = pack_bf16(z0 - bf_lo(hi), 0.f);
                *reinterpret_cast<uint16_t*>(snap_z(0) + sw128_offset(0, srow)) = (uint16_t)hi;
                *reinterpret_cast<uint16_t*>(snap_z(0) + sw128_offset(1, srow)) = (uint16_t)lo;
            }
            tc_fence_before();
            fence_proxy_async_smem();
            named_bar(3, 128);
            if (t == 0) {
                mbar_arrive(&m.state_init);
                mbar_arrive(&m.snap_full[0]);
            }
        }
        bool ok = true;
        for (int i = 0; i < nch; ++i) {
            const int b = i & 1;
            const uint32_t pb = (i >> 1) & 1;
            const int64_t u = u0 + i;
            const int h = (int)(u / part.nchunks), ch = (int)(u % part.nchunks);
            const bool last_in_run = (u + 1 == u1) || ((u + 1) / part.nchunks != h);
            const bool head_end = (ch == part.nchunks - 1);

            // State after chunk i -> snapshot for chunk i + 1 (zero when a new head starts).
            ok = mbar_wait(&m.ds_full, i & 1, max_spin);
            tc_fence_after();
            const bool snap_next = (i + 1 < nch);
            uint8_t* dnext = snap_s(b ^ 1);
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2) {
                uint32_t r0[16], r1[16];
                tmem_ld16(tS + 32 * c2, r0);
                tmem_ld16(tS + 32 * c2 + 16, r1);
                tmem_ld_wait();
                if (sowner && last_in_run && head_end && S_out) {
                    float4* dst = reinterpret_cast<float4*>(S_out + ((int64_t)h * kD + srow) * kD + 32 * c2);
#pragma unroll
                    for (int qd = 0; qd < 4; ++qd) {
                        dst[qd] = make_float4(__uint_as_float(r0[4 * qd]), __uint_as_float(r0[4 * qd + 1]),
                                              __uint_as_float(r0[4 * qd + 2]), __uint_as_float(r0[4 * qd + 3]));
                        dst[qd + 4] = make_float4(__uint_as_float(r1[4 * qd]), __uint_as_float(r1[4 * qd + 1]),
                                                  __uint_as_float(r1[4 * qd + 2]), __uint_as_float(r1[4 * qd + 3]));
                    }
                }
                if (sowner && snap_next) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const uint32_t* rr = c < 2 ? r0 : r1;
                        const int e0 = 8 * (c & 1);
                        uint4 v = last_in_run
                                      ? make_uint4(0, 0, 0, 0)
                                      : make_uint4(pack_bf16(__uint_as_float(rr[e0]), __uint_as_float(rr[e0 + 1])),
                                                   pack_bf16(__uint_as_float(rr[e0 + 2]), __uint_as_float(rr[e0 + 3])),
                                                   pack_bf16(__uint_as_float(rr[e0 + 4]), __uint_as_float(rr[e0 + 5])),
                                                   pack_bf16(__uint_as_float(rr[e0 + 6]), __uint_as_float(rr[e0 + 7])));
                        *reinterpret_cast<uint4*>(dnext + sw128_offset(srow, 32 * c2 + 8 * c)) = v;
                    }
                }
            }
            {
                uint32_t rz[16];
                tmem_ld16(tS + 64, rz);
                tmem_ld_wait();
                const float zr = __uint_as_float(rz[0]);
                if (sowner && last_in_run && head_end && z_out) z_out[(int64_t)h * kD + srow] = zr;
                if (sowner && snap_next) {
                    const float zs = last_in_run ? 0.f : zr;
                    const uint32_t hi = pack_bf16(zs, 0.f);
                    const uint32_t lo = pack_bf16(zs - bf_lo(hi), 0.f);
                    *reinterpret_cast<uint16_t*>(snap_z(b ^ 1) + sw128_offset(0, srow)) = (uint16_t)hi;
                    *reinterpret_cast<uint16_t*>(snap_z(b ^ 1) + sw128_offset(1, srow)) = (uint16_t)lo;
                }
            }
            tc_fence_before();
            fence_proxy_async_smem();
            if (t == 0) tma_store_wait_read<0>();  // the output staging tile is free again
            ok = named_bar_and(3, 128, ok);
            if (!ok) break;
            if (t == 0) {
                mbar_arrive(&m.ds_free);
                if (snap_next) mbar_arrive(&m.snap_full[b ^ 1]);
            }

            // Output: num / (den + eps) -> bf16 -> staging tile -> TMA store.
            ok = mbar_wait(&m.o_full[b], pb, max_spin);
            tc_fence_after();
            const uint32_t tO = tmem + kTmO + kTmOStride * b;
            float inv;
            {
                uint32_t rd[16];
                tmem_ld16(tO + lane_base + 64, rd);
                tmem_ld_wait();
                inv = 1.f / (__uint_as_float(rd[0]) + __uint_as_float(rd[1]) + eps);
            }
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2) {
                uint32_t r0[16], r1[16];
                tmem_ld16(tO + lane_base + 32 * c2, r0);
                tmem_ld16(tO + lane_base + 32 * c2 + 16, r1);
                tmem_ld_wait();
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const uint32_t* rr = c < 2 ? r0 : r1;
                    const int e0 = 8 * (c & 1);
                    uint4 v = make_uint4(
                        pack_bf16(__uint_as_float(rr[e0]) * inv, __uint_as_float(rr[e0 + 1]) * inv),
                        pack_bf16(__uint_as_float(rr[e0 + 2]) * inv, __uint_as_float(rr[e0 + 3]) * inv),
                        pack_bf16(__uint_as_float(rr[e0 + 4]) * inv, __uint_as_float(rr[e0 + 5]) * inv),
                        pack_bf16(__uint_as_float(rr[e0 + 6]) * inv, __uint_as_float(rr[e0 + 7]) * inv));
                    *reinterpret_cast<uint4*>(ostage + sw128_offset(row, 32 * c2 + 8 * c)) = v;
                }
            }
            tc_fence_before();
            fence_proxy_async_smem();
            ok = named_bar_and(3, 128, ok);
            if (!ok) break;
            if (t == 0) {
                mbar_arrive(&m.o_free[b]);
                tma_store_3d(&omap, ostage, 0, ch * kC, h);
                tma_store_commit();
            }
        }
        if (!ok && t == 0) report_timeout(hdr);
        if (t == 0) tma_store_wait_all<0>();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 13) {
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

static_assert(kOutSmem <= 232448, "output kernel shared memory exceeds 227 KB");
static_assert(kStateSmem <= 232448, "state kernel shared memory exceeds 227 KB");

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
    if ((err = cudaPeekAtLastError())) return err;
    // The output kernel may start while the state kernel drains; it waits
    // (griddepcontrol.wait) before reading the aggregates.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.grid);
    cfg.blockDim = dim3(kOutThreads);
    cfg.dynamicSmemBytes = kOutSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, causal_output_kernel, qm, km, vm, om,
                              (const float*)agg, S_out, z_out, p, N, eps, hdr);
}

}  // namespace la
