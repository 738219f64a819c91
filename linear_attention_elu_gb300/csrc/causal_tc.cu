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
#include "tc_common.cuh"
#include "tc_util.cuh"

namespace la {

namespace {

using namespace tc;
using namespace tcc;

constexpr int kD = 64;                         // Dk = Dv
constexpr int kNx = 80;                        // MMA N with the extra ones / z columns
constexpr int kE = kD * kD + kD;               // floats per aggregate (S then z)

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
// Warp roles (18 warps):
//   warps 0-7   phi:   phi on the Q and K tiles of each landed stage, in place
//   warps 8-11  mask:  A (fp32, TMEM) -> causal mask -> bf16 P, written back into
//                      the same TMEM columns (A operand of MMA (4))
//   warps 12-15 state: running state (TMEM) -> bf16 snapshot for the next
//                      chunk; then the output epilogue num / (den + eps)
//   warp 16     TMA producer       warp 17  MMA issuer (one thread)
// The four warps of the mask and state roles cover the four TMEM lane quarters.
//
// Per chunk i (stage s = i mod 3, TMEM buffer b = i mod 2), three contraction
// groups, each a few wide tcgen05.mma instructions:
//   (2)   [S^T ; z] += [V | 1]^T phi(K)        M=128 (64 value rows, z row), N=64, K=128 tokens
//   (1+3) [A | num | den] = phi(Q) [phi(K) | S^T | z_hi z_lo]^T      M=128, N=208, K=64
//   (4)   [num | den] += P [V | 1]             M=128, N=80, K=128 keys, P read from TMEM
// (4) of chunk i is issued after (2), (1+3) of chunk i + 1, so that the mask
// role's work on chunk i overlaps the next chunk's contractions.

constexpr int kPhiWarps = 8;
constexpr int kMaskW0 = kPhiWarps, kStateW0 = kPhiWarps + 4;
constexpr int kProdW = kStateW0 + 4, kMmaW = kProdW + 1;
constexpr int kOutThreads = 32 * (kMmaW + 1);
constexpr int kPhiThreads = 32 * kPhiWarps;
constexpr int kStages = 3;
// Shared-memory map (offsets from a 1024-aligned base). A stage holds the Q, K
// and V tiles and, right after K, the snapshot rows S^T (64) and z (16) that
// complete the K-major operand [phi(K) | S^T | z] of MMA (1+3).
constexpr uint32_t kStQ = 0, kStK = kTileBytes, kStS = 2 * kTileBytes;
constexpr uint32_t kStZ = kStS + kD * 128, kStV = kStZ + 16 * 128;
constexpr uint32_t kStageBytes = kStV + kTileBytes;            // 58 KB
constexpr uint32_t kOffOnes = kStages * kStageBytes;           // [V | 1] second atom, MN-major
constexpr uint32_t kOffO = kOffOnes + kTileBytes;              // output staging tile
constexpr uint32_t kSmemEnd = kOffO + kTileBytes;
constexpr size_t kOutSmem = 1024 + kSmemEnd;
// TMEM columns: buffer b = [A / P | num | den] at 224 b (208 columns);
// running state [S^T ; z] at 448 (64 columns, lanes 0-63 = S^T rows, lane 64 = z).
constexpr uint32_t kTmBuf = 224, kTmState = 448;

struct OutMisc {
    uint64_t full[kStages], phi_done[kStages], empty[kStages], snap_full[kStages];
    uint64_t a_full[2], o_full[2], o_free[2];
    uint64_t p_full, ds_full, mma_drain;
    uint32_t tmem_slot;
};

__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
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
    auto stage = [&](int s) { return base + s * kStageBytes; };
    uint8_t* ones = base + kOffOnes;
    uint8_t* ostage = base + kOffO;

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&m.full[s], 1);
            mbar_init(&m.phi_done[s], 1);
            mbar_init(&m.empty[s], 1);
            mbar_init(&m.snap_full[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&m.a_full[b], 1);
            mbar_init(&m.o_full[b], 1);
            mbar_init(&m.o_free[b], 1);
        }
        mbar_init(&m.p_full, 1);
        mbar_init(&m.ds_full, 1);
        mbar_init(&m.mma_drain, 1);
        fence_mbar_init();
    }
    if (warp < kProdW) {
        init_ones_tile(ones, tid, 32 * kProdW);
        for (int idx = tid; idx < kStages * 128; idx += 32 * kProdW) {  // z rows of every stage
            const int s = idx / 128, r = idx % 128;
            *reinterpret_cast<uint4*>(stage(s) + kStZ + r * 16) = make_uint4(0, 0, 0, 0);
        }
    }
    fence_proxy_async_smem();
    if (warp == kMmaW) {
        tmem_alloc(&m.tmem_slot, 512);
        tmem_relinquish();
    }
    if (warp == kProdW && lane == 0) {
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

    if (warp == kProdW) {
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
                tma_load_3d(stage(s) + kStQ, &qmap, &m.full[s], 0, ch * kC, h);
                tma_load_3d(stage(s) + kStK, &kmap, &m.full[s], 0, ch * kC, h);
                tma_load_3d(stage(s) + kStV, &vmap, &m.full[s], 0, ch * kC, h);
            }
            for (int j = i - kStages > 0 ? i - kStages : 0; j < i; ++j)
                mbar_wait(&m.full[j % kStages], (j / kStages) & 1, kDefaultMaxSpin);
        }
    } else if (warp == kMmaW) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t id_s = idesc_bf16_f32(128, 64, true, true);     // (2)
            const uint32_t id_qk = idesc_bf16_f32(128, 208, false, false); // (1+3)
            const uint32_t id_pv = idesc_bf16_f32(128, 80, false, true);   // (4)
            const uint32_t onesa = smem_u32(ones);
            // (4) for chunk j: [num | den] += P_j [V_j | 1].
            auto issue_pv = [&](int j) -> bool {
                if (!mbar_wait(&m.p_full, j & 1, max_spin)) return false;
                tc_fence_after();
                const int sj = j % kStages, bj = j & 1;
                const uint32_t va = smem_u32(stage(sj) + kStV);
                const uint32_t lbo = onesa - va;
                const uint32_t tbuf = tmem + kTmBuf * bj;
#pragma unroll
                for (int k16 = 0; k16 < kC / 16; ++k16)
                    mma_bf16_ts(tbuf + 128, tbuf + 8 * k16,
                                smem_desc(va + k16 * 2048, lbo, 1024, kSwizzle128B), id_pv, 1u);
                mma_commit(&m.o_full[bj]);
                mma_commit(&m.empty[sj]);
                return true;
            };
            bool ok = true;
            for (int i = 0; i < nch && ok; ++i) {
                const int s = i % kStages, b = i & 1;
                const uint32_t ps = (i / kStages) & 1;
                if (!mbar_wait(&m.phi_done[s], ps, max_spin) ||
                    !mbar_wait(&m.snap_full[s], ps, max_spin)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t qa = smem_u32(stage(s) + kStQ), ka = smem_u32(stage(s) + kStK),
                               va = smem_u32(stage(s) + kStV);
                const uint32_t lbo = onesa - va;
                const bool fresh = (i > 0) && ((u0 + i) % part.nchunks == 0);
                // (2) running state [S^T ; z] += [V | 1]^T phi(K)  (A MN-major over 2 atoms).
#pragma unroll
                for (int k16 = 0; k16 < kC / 16; ++k16)
                    mma_bf16(tmem + kTmState,
                             smem_desc(va + k16 * 2048, lbo, 1024, kSwizzle128B),
                             smem_desc(ka + k16 * 2048, 1024, 1024, kSwizzle128B), id_s,
                             (fresh && k16 == 0) ? 0u : 1u);
                mma_commit(&m.ds_full);
                // (1+3) overwrites buffer b: the output epilogue of chunk i - 2 must be done.
                if (i >= 2 && !mbar_wait(&m.o_free[b], ((i >> 1) - 1) & 1, max_spin)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // (1+3) [A | num | den] = phi(Q) [phi(K) | S^T | z]^T (B K-major, 208 rows).
#pragma unroll
                for (int k16 = 0; k16 < kD / 16; ++k16)
                    mma_bf16(tmem + kTmBuf * b,
                             smem_desc(qa + k16 * 32, 16, 1024, kSwizzle128B),
                             smem_desc(ka + k16 * 32, 16, 1024, kSwizzle128B), id_qk, k16 > 0);
                mma_commit(&m.a_full[b]);
                if (i >= 1 && !issue_pv(i - 1)) ok = false;
            }
            if (ok && nch > 0 && !issue_pv(nch - 1)) ok = false;
            if (!ok) report_timeout(hdr);
            mma_commit(&m.mma_drain);  // every issued MMA completes before TMEM is released
            mbar_wait(&m.mma_drain, 0, kDefaultMaxSpin);
        }
    } else if (warp < kMaskW0) {
        // ---------------------------------------------------------- phi role
        const int t = tid;  // 0 .. kPhiThreads - 1
        bool ok = true;
        for (int i = 0; i < nch; ++i) {
            const int s = i % kStages;
            const int ch = (int)((u0 + i) % part.nchunks);
            const int valid = min(kC, N - ch * kC);
            ok = mbar_wait(&m.full[s], (i / kStages) & 1, max_spin);
            phi_tile_256(stage(s) + kStQ, t, kC);
            phi_tile_256(stage(s) + kStK, t, valid);
            fence_proxy_async_smem();
            ok = named_bar_and(1, kPhiThreads, ok);
            if (!ok) break;
            if (t == 0) mbar_arrive(&m.phi_done[s]);
        }
        if (!ok && t == 0) report_timeout(hdr);
    } else if (warp < kStateW0) {
        // ---------------------------------------------------------- mask role
        // A block j (32 keys, columns 32j..32j+31) -> P block j (16 packed columns
        // 16j..16j+15) in the same TMEM buffer; in increasing j every A column is
        // read before the P columns that cover it are written.
        const int t = tid - 32 * kMaskW0;
        bool ok = true;
        for (int i = 0; i < nch; ++i) {
            const int b = i & 1;
            const uint32_t tbuf = tmem + kTmBuf * b + lane_base;
            ok = mbar_wait(&m.a_full[b], (i >> 1) & 1, max_spin);
            tc_fence_after();
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint32_t p[16];
                if (j > q4) {
                    // Queries of this lane quarter see no key of block j.
#pragma unroll
                    for (int e = 0; e < 16; ++e) p[e] = 0u;
                } else {
                    uint32_t r0[16], r1[16];
                    tmem_ld16(tbuf + 32 * j, r0);
                    tmem_ld16(tbuf + 32 * j + 16, r1);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        float a0 = __uint_as_float(r0[2 * e]), a1 = __uint_as_float(r0[2 * e + 1]);
                        float c0 = __uint_as_float(r1[2 * e]), c1 = __uint_as_float(r1[2 * e + 1]);
                        if (j == q4) {  // block holding the diagonal: key 32 q4 + e' <= row 32 q4 + lane
                            a0 = (2 * e <= lane) ? a0 : 0.f;
                            a1 = (2 * e + 1 <= lane) ? a1 : 0.f;
                            c0 = (16 + 2 * e <= lane) ? c0 : 0.f;
                            c1 = (17 + 2 * e <= lane) ? c1 : 0.f;
                        }
                        p[e] = pack_bf16(a0, a1);
                        p[8 + e] = pack_bf16(c0, c1);
                    }
                }
                tmem_st16(tbuf + 16 * j, p);
            }
            tmem_st_wait();
            tc_fence_before();
            ok = named_bar_and(2, 128, ok);
            if (!ok) break;
            if (t == 0) mbar_arrive(&m.p_full);
        }
        if (!ok && t == 0) report_timeout(hdr);
    } else {
        // ---------------------------------------------------------- state + output role
        const int t = tid - 32 * kStateW0;       // 0..127
        const int row = 32 * q4 + lane;          // TMEM lane: S^T row (< 64), z row (64), query row
        const uint32_t tS = tmem + kTmState + lane_base;

        // Output epilogue for chunk j: num / (den + eps) -> bf16 -> staging -> TMA store.
        auto output = [&](int j) -> bool {
            const int bj = j & 1;
            const int64_t u = u0 + j;
            const int h = (int)(u / part.nchunks), ch = (int)(u % part.nchunks);
            bool okj = mbar_wait(&m.o_full[bj], (j >> 1) & 1, max_spin);
            if (t == 0) tma_store_wait_read<0>();  // the staging tile is free again
            named_bar(3, 128);
            tc_fence_after();
            const uint32_t to = tmem + kTmBuf * bj + 128 + lane_base;
            float inv;
            {
                uint32_t rd[16];
                tmem_ld16(to + 64, rd);
                tmem_ld_wait();
                inv = 1.f / (__uint_as_float(rd[0]) + __uint_as_float(rd[1]) + eps);
            }
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2) {
                uint32_t r0[16], r1[16];
                tmem_ld16(to + 32 * c2, r0);
                tmem_ld16(to + 32 * c2 + 16, r1);
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
            okj = named_bar_and(3, 128, okj);
            if (okj && t == 0) {
                mbar_arrive(&m.o_free[bj]);
                tma_store_3d(&omap, ostage, 0, ch * kC, h);
                tma_store_commit();
            }
            return okj;
        };
        // Snapshot rows for chunk j (stage j mod 3): S^T row `row` (rows < 64) and
        // z_hi, z_lo (row 64), from 64 fp32 values v[] of this TMEM lane.
        auto write_snap_half = [&](uint8_t* st, int c2, const uint32_t (&r0)[16],
                                   const uint32_t (&r1)[16], bool zero) {
            if (row < kD) {
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const uint32_t* rr = c < 2 ? r0 : r1;
                    const int e0 = 8 * (c & 1);
                    uint4 v = zero ? make_uint4(0, 0, 0, 0)
                                   : make_uint4(pack_bf16(__uint_as_float(rr[e0]), __uint_as_float(rr[e0 + 1])),
                                                pack_bf16(__uint_as_float(rr[e0 + 2]), __uint_as_float(rr[e0 + 3])),
                                                pack_bf16(__uint_as_float(rr[e0 + 4]), __uint_as_float(rr[e0 + 5])),
                                                pack_bf16(__uint_as_float(rr[e0 + 6]), __uint_as_float(rr[e0 + 7])));
                    *reinterpret_cast<uint4*>(st + kStS + sw128_offset(row, 32 * c2 + 8 * c)) = v;
                }
            } else if (row == kD) {
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const uint32_t* rr = c < 2 ? r0 : r1;
                    const int e0 = 8 * (c & 1);
                    uint32_t hi[4], lo[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float za = zero ? 0.f : __uint_as_float(rr[e0 + 2 * e]);
                        const float zb = zero ? 0.f : __uint_as_float(rr[e0 + 2 * e + 1]);
                        hi[e] = pack_bf16(za, zb);
                        lo[e] = pack_bf16(za - bf_lo(hi[e]), zb - __uint_as_float(hi[e] & 0xFFFF0000u));
                    }
                    *reinterpret_cast<uint4*>(st + kStZ + sw128_offset(0, 32 * c2 + 8 * c)) =
                        make_uint4(hi[0], hi[1], hi[2], hi[3]);
                    *reinterpret_cast<uint4*>(st + kStZ + sw128_offset(1, 32 * c2 + 8 * c)) =
                        make_uint4(lo[0], lo[1], lo[2], lo[3]);
                }
            }
        };

        // Start state of the first run: sum of the aggregates (S row-major
        // [feature][value], then z) of this head's chunks held by lower-numbered
        // CTAs, transposed into TMEM rows (S^T; z) and into the stage-0 snapshot.
        pdl_wait();  // the state kernel's aggregates are complete and visible
        {
            const int h = (int)(u0 / part.nchunks);
            const int64_t head_begin = (int64_t)h * part.nchunks;
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2) {
                uint32_t r0[16], r1[16];
                float acc[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) acc[e] = 0.f;
                if (u0 > head_begin && row <= kD) {
                    for (int cb = cta - 1; cb >= 0; --cb) {
                        const int64_t b0 = part.begin(cb), b1 = part.begin(cb + 1);
                        if (b1 <= head_begin) break;
                        if (b1 <= b0) continue;
                        const float* a = agg + ((int64_t)cb * part.maxr + (h - b0 / part.nchunks)) * kE;
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            const int c = 32 * c2 + e;  // feature index
                            acc[e] += row < kD ? a[c * kD + row] : a[kD * kD + c];
                        }
                    }
                }
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    r0[e] = __float_as_uint(acc[e]);
                    r1[e] = __float_as_uint(acc[16 + e]);
                }
                tmem_st16(tS + 32 * c2, r0);
                tmem_st16(tS + 32 * c2 + 16, r1);
                write_snap_half(stage(0), c2, r0, r1, false);
            }
            tmem_st_wait();
            tc_fence_before();
            fence_proxy_async_smem();
            named_bar(3, 128);
            if (t == 0) mbar_arrive(&m.snap_full[0]);
        }
        bool ok = true;
        for (int i = 0; i < nch; ++i) {
            const int64_t u = u0 + i;
            const int h = (int)(u / part.nchunks), ch = (int)(u % part.nchunks);
            const bool last_in_run = (u + 1 == u1) || ((u + 1) / part.nchunks != h);
            const bool head_end = (ch == part.nchunks - 1);
            const bool snap_next = (i + 1 < nch);
            uint8_t* nst = stage((i + 1) % kStages);

            // State after chunk i -> snapshot for chunk i + 1 (zero when a new head starts).
            ok = mbar_wait(&m.ds_full, i & 1, max_spin);
            tc_fence_after();
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2) {
                uint32_t r0[16], r1[16];
                tmem_ld16(tS + 32 * c2, r0);
                tmem_ld16(tS + 32 * c2 + 16, r1);
                tmem_ld_wait();
                if (last_in_run && head_end) {
                    // Final state of the head: S[c][n] (row n of S^T holds column n of S), z.
                    if (row < kD && S_out) {
                        float* dst = S_out + (int64_t)h * kD * kD + row;
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            dst[(32 * c2 + e) * kD] = __uint_as_float(r0[e]);
                            dst[(32 * c2 + 16 + e) * kD] = __uint_as_float(r1[e]);
                        }
                    } else if (row == kD && z_out) {
                        float* dst = z_out + (int64_t)h * kD + 32 * c2;
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            dst[e] = __uint_as_float(r0[e]);
                            dst[16 + e] = __uint_as_float(r1[e]);
                        }
                    }
                }
                if (snap_next) write_snap_half(nst, c2, r0, r1, last_in_run);
            }
            tc_fence_before();
            fence_proxy_async_smem();
            ok = named_bar_and(3, 128, ok);
            if (!ok) break;
            if (t == 0 && snap_next) mbar_arrive(&m.snap_full[(i + 1) % kStages]);
            // Output of the previous chunk while the tensor core works on this one.
            if (i >= 1 && !(ok = output(i - 1))) break;
        }
        if (ok && nch > 0) ok = output(nch - 1);
        if (!ok && t == 0) report_timeout(hdr);
        if (t == 0) tma_store_wait_all<0>();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaW) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ---------------------------------------------------------------- host side

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
    static std::atomic<int> optin_causal_state_kernel[kMaxDevices];
    if ((err = ensure_smem_optin(causal_state_kernel, (int)kStateSmem, optin_causal_state_kernel))) return err;
    static std::atomic<int> optin_causal_output_kernel[kMaxDevices];
    if ((err = ensure_smem_optin(causal_output_kernel, (int)kOutSmem, optin_causal_output_kernel))) return err;
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
