// Tensor-core (tcgen05) non-causal forward for bf16 inputs, Dk = Dv = 64 or 128.
//
// Method ("Why Replace Attention? The Softmax Bottleneck and the Path to Linear
// Time", section 6.2; "Transformers Are RNNs: Linear Attention", "Reassociate
// the Products"): per head, S = sum_j phi(k_j) v_j^T and z = sum_j phi(k_j),
// then o_i = phi(q_i)^T S / (phi(q_i)^T z + eps) for every query.
//
// Two launches over the persistent-CTA chunk partition (tc_common.cuh):
//   state kernel  per run (a CTA's chunks of one head): S_run = phi(K)^T V on
//                 the tensor core (fp32 in TMEM) and z_run = column sums of
//                 phi(K), both written to the workspace. K and V are read once.
//                 D = 128: M = 128 features, N = 128 values, z summed on the
//                 CUDA cores. D = 64: [S^T ; z] = [V | 1]^T phi(K) (M = 128 rows:
//                 the 64 values, then a column of ones that yields z, then
//                 zeros; N = 64 features), so z comes out of the same MMA.
//   apply kernel  per run: S = sum of the runs of that head (the split-N
//                 reduction), laid out once in shared memory as the K-major
//                 operand [S^T | z_hi | z_lo] (D + 16 rows); per chunk of 128
//                 queries [num | den] = phi(Q) [S^T | z]^T (M = 128, N = D + 16,
//                 K = D), then o = num / (den + eps). phi(Q) is written to
//                 TMEM beside the chunk's accumulator as the MMA's A operand,
//                 so a Q stage is refilled as soon as phi has read it; outputs
//                 leave through two staging buffers. Q is read once, O written
//                 once.
// The apply kernel is a programmatic dependent of the state kernel.
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_common.cuh"
#include "tc_util.cuh"

namespace la {

namespace {

using namespace tc;
using namespace tcc;

// Dk = Dv = kD (64 or 128): features per aggregate row, and the aggregate size
// (S row-major [c][n], then z).
template <int kD> constexpr int kE = kD * kD + kD;
template <int kD> constexpr int kNb = kD + 16;             // B operand rows: S^T, z_hi, z_lo, padding
template <int kD> constexpr int kBoxes = kD / 64;           // 64-feature boxes per tile

// ======================================================== state kernel
// Warps 0-7: phi on K (+ z sums for D = 128) and the read-out of S. Warp 8: TMA.
// Warp 9: MMA.

template <int kD> constexpr int kSStages = kD == 128 ? 3 : 6;
template <int kD> constexpr uint32_t kSStage = 2 * kBoxes<kD> * kTileBytes;   // K boxes, V boxes
// D = 64: the [V | 1] operand's second atom (a column of ones, the rest zero).
template <int kD> constexpr uint32_t kSOnes = kSStages<kD> * kSStage<kD>;
template <int kD> constexpr size_t kSSmem = 1024 + kSOnes<kD> + (kD == 64 ? kTileBytes : 0);
constexpr int kSThreads = 320;

// kLast (causal use): only the last run of each range, and only when its head
// continues into the next range, into slot agg + cta * kE (the run that the
// ranges to the right add up); other chunks are not read.
template <int kD, int kPhi, bool kLast = false>
__global__ void __launch_bounds__(kSThreads, 1)
nc_state_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                float* __restrict__ agg, Partition part, int N, WsHeader* hdr) {
    constexpr int kStg = kSStages<kD>, kB = kBoxes<kD>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    __shared__ uint64_t full[kStg], empty[kStg], phi_done[kStg];
    __shared__ uint64_t run_done, tmem_free, mma_drain;
    __shared__ uint32_t tmem_slot;
    __shared__ float zsum[kD];

    pdl_launch_dependents();
    const uint32_t max_spin = hdr->max_spin;
    const bool hold = hdr->hold_item != 0;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cta = blockIdx.x;
    const int64_t u1 = part.begin(cta + 1);
    const int64_t u0 = !kLast ? part.begin(cta)
                       : (u1 % part.nchunks == 0 ? u1
                                                 : max(part.begin(cta), u1 / part.nchunks * part.nchunks));
    auto stage = [&](int s) { return base + s * kSStage<kD>; };
    uint8_t* ones = base + kSOnes<kD>;

    if (tid == 0) {
        for (int s = 0; s < kStg; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
            mbar_init(&phi_done[s], 1);
        }
        mbar_init(&run_done, 1);
        mbar_init(&tmem_free, 1);
        mbar_init(&mma_drain, 1);
        fence_mbar_init();
    }
    if (tid < kD) zsum[tid] = 0.f;
    if constexpr (kD == 64) {
        if (warp < 8) init_ones_tile(ones, tid, 256);
        fence_proxy_async_smem();
    }
    if (warp == 9) {
        tmem_alloc(&tmem_slot, kD == 128 ? 128 : 64);
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
                const int s = i % kStg;
                if (i >= kStg && !mbar_wait(&empty[s], ((i / kStg) - 1) & 1, max_spin)) {
                    report_timeout(hdr);
                    break;
                }
                if (hold) break;  // test hook: a load that is never issued
                const int h = (int)(u / part.nchunks), ch = (int)(u % part.nchunks);
                mbar_arrive_expect_tx(&full[s], 2 * kB * kTileBytes);
#pragma unroll
                for (int bx = 0; bx < kB; ++bx) {
                    tma_load_3d(stage(s) + bx * kTileBytes, &kmap, &full[s], 64 * bx, ch * kC, h);
                    tma_load_3d(stage(s) + (kB + bx) * kTileBytes, &vmap, &full[s], 64 * bx, ch * kC, h);
                }
            }
            for (int j = i - kStg > 0 ? i - kStg : 0; j < i; ++j)
                mbar_wait(&full[j % kStg], (j / kStg) & 1, kDefaultMaxSpin);
        }
    } else if (warp == 9) {
        if (lane == 0) {
            // D = 128: S += phi(K)^T V, A = phi(K) MN-major (two 64-feature atoms),
            // B = V MN-major. D = 64: [S^T ; z] += [V | 1]^T phi(K), A = [V | 1]
            // MN-major (V, then the ones atom), B = phi(K) MN-major.
            const uint32_t idesc = kD == 128 ? idesc_bf16_f32(128, 128, true, true)
                                             : idesc_bf16_f32(128, 64, true, true);
            const uint32_t onesa = smem_u32(ones);
            int i = 0, run = 0;
            bool first_in_run = true, ok = true;
            for (int64_t u = u0; u < u1; ++u, ++i) {
                const int s = i % kStg;
                const int h = (int)(u / part.nchunks);
                const bool last_in_run = (u + 1 == u1) || ((u + 1) / part.nchunks != h);
                if (!mbar_wait(&phi_done[s], (i / kStg) & 1, max_spin) ||
                    (first_in_run && run > 0 && !mbar_wait(&tmem_free, (run - 1) & 1, max_spin))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t ka = smem_u32(stage(s)), va = smem_u32(stage(s) + kB * kTileBytes);
#pragma unroll
                for (int k16 = 0; k16 < kC / 16; ++k16) {
                    if constexpr (kD == 128)
                        mma_bf16(tmem, smem_desc(ka + k16 * 2048, kTileBytes, 1024, kSwizzle128B),
                                 smem_desc(va + k16 * 2048, kTileBytes, 1024, kSwizzle128B), idesc,
                                 (first_in_run && k16 == 0) ? 0u : 1u);
                    else
                        mma_bf16(tmem, smem_desc(va + k16 * 2048, onesa - va, 1024, kSwizzle128B),
                                 smem_desc(ka + k16 * 2048, 1024, 1024, kSwizzle128B), idesc,
                                 (first_in_run && k16 == 0) ? 0u : 1u);
                }
                mma_commit(&empty[s]);
                if (last_in_run) {
                    mma_commit(&run_done);
                    ++run;
                }
                first_in_run = last_in_run;
            }
            if (!ok) report_timeout(hdr);
            mma_commit(&mma_drain);
            mbar_wait(&mma_drain, 0, kDefaultMaxSpin);
        }
    } else {
        // Math warps 0-7 (256 threads). Thread t handles physical 16-byte chunk
        // (t & 7) of rows (t >> 3) + 32 k of each 64-feature box: logical feature
        // group jgrp = (t & 7) ^ ((t >> 3) & 7), the same for all its rows.
        const int t = tid;
        const int jgrp = (t & 7) ^ ((t >> 3) & 7);
        const int g = warp >> 2, q4 = warp & 3;
        float zp[kB][8];
#pragma unroll
        for (int bx = 0; bx < kB; ++bx)
#pragma unroll
            for (int e = 0; e < 8; ++e) zp[bx][e] = 0.f;
        int i = 0, run = 0;
        bool ok = true;
        for (int64_t u = u0; u < u1; ++u, ++i) {
            const int s = i % kStg;
            const int h = (int)(u / part.nchunks), ch = (int)(u % part.nchunks);
            const bool last_in_run = (u + 1 == u1) || ((u + 1) / part.nchunks != h);
            const int valid = min(kC, N - ch * kC);
            ok = mbar_wait(&full[s], (i / kStg) & 1, max_spin);
#pragma unroll
            for (int bx = 0; bx < kB; ++bx) {
                uint8_t* kt = stage(s) + bx * kTileBytes;
                uint4 v[4];
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    v[k] = *reinterpret_cast<const uint4*>(kt + ((t >> 3) + 32 * k) * 128 + (t & 7) * 16);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int r = (t >> 3) + 32 * k;
                    uint4 o = make_uint4(0, 0, 0, 0);
                    if (r < valid) {
                        o = phi8<kPhi>(v[k]);
                        if constexpr (kD == 128) {
                            const uint32_t w[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                zp[bx][2 * e] += bf_lo(w[e]);
                                zp[bx][2 * e + 1] += __uint_as_float(w[e] & 0xFFFF0000u);
                            }
                        }
                    }
                    *reinterpret_cast<uint4*>(kt + r * 128 + (t & 7) * 16) = o;
                }
            }
            fence_proxy_async_smem();
            ok = named_bar_and(1, 256, ok);
            if (!ok) break;
            if (t == 0) mbar_arrive(&phi_done[s]);
            if (last_in_run) {
                float* out = agg + (kLast ? (int64_t)cta : (int64_t)cta * part.maxr + run) * kE<kD>;
                if constexpr (kD == 128) {
                    // z of the run: reduce the column-group partials.
#pragma unroll
                    for (int bx = 0; bx < kB; ++bx)
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            float vsum = zp[bx][e];
                            vsum += __shfl_xor_sync(0xffffffffu, vsum, 9);
                            vsum += __shfl_xor_sync(0xffffffffu, vsum, 18);
                            if ((lane >> 3) == 0) atomicAdd(&zsum[64 * bx + 8 * jgrp + e], vsum);
                            zp[bx][e] = 0.f;
                        }
                }
                ok = mbar_wait(&run_done, run & 1, max_spin);
                tc_fence_after();
                if constexpr (kD == 128) {
                    // S rows = features: lane 32 q4 + l holds feature row, warpgroup g value
                    // columns [64g, 64g+64).
                    const int row = 32 * q4 + lane;
#pragma unroll
                    for (int c2 = 0; c2 < 2; ++c2) {
                        uint32_t r0[16], r1[16];
                        const uint32_t ta = tmem + ((uint32_t)(32 * q4) << 16) + 64 * g + 32 * c2;
                        tmem_ld16(ta, r0);
                        tmem_ld16(ta + 16, r1);
                        tmem_ld_wait();
                        float4* dst = reinterpret_cast<float4*>(out + row * kD + 64 * g + 32 * c2);
#pragma unroll
                        for (int qd = 0; qd < 4; ++qd) {
                            dst[qd] = make_float4(__uint_as_float(r0[4 * qd]), __uint_as_float(r0[4 * qd + 1]),
                                                  __uint_as_float(r0[4 * qd + 2]), __uint_as_float(r0[4 * qd + 3]));
                            dst[qd + 4] = make_float4(__uint_as_float(r1[4 * qd]), __uint_as_float(r1[4 * qd + 1]),
                                                      __uint_as_float(r1[4 * qd + 2]), __uint_as_float(r1[4 * qd + 3]));
                        }
                    }
                } else {
                    // [S^T ; z] rows = values (lane n < 64) and z (lane 64), columns = features:
                    // warp (q4, g) reads lanes 32 q4 .. + 31 (q4 < 3), features 32 g .. + 31.
                    if (q4 < 3) {
                        const int n = 32 * q4 + lane;
                        uint32_t r0[16], r1[16];
                        const uint32_t ta = tmem + ((uint32_t)(32 * q4) << 16) + 32 * g;
                        tmem_ld16(ta, r0);
                        tmem_ld16(ta + 16, r1);
                        tmem_ld_wait();
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            const float x = __uint_as_float(e < 16 ? r0[e] : r1[e - 16]);
                            const int c = 32 * g + e;
                            if (n < kD) out[c * kD + n] = x;
                            else if (n == kD) out[kD * kD + c] = x;
                        }
                    }
                }
                tc_fence_before();
                ok = named_bar_and(1, 256, ok);   // zsum complete, TMEM read
                if (!ok) break;
                if constexpr (kD == 128) {
                    if (t < kD) {
                        out[kD * kD + t] = zsum[t];
                        zsum[t] = 0.f;
                    }
                    named_bar(1, 256);
                }
                if (t == 0) mbar_arrive(&tmem_free);
                ++run;
            }
        }
        if (!ok && t == 0) report_timeout(hdr);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kD == 128 ? 128 : 64);
    }
}

// ======================================================== apply kernel
// Warps 0-7: phi on Q into TMEM. Warps 8-15: operand build (per run) and output epilogue
// (two warps per TMEM lane quarter, each half the value columns).
// Warp 16: TMA producer. Warp 17: MMA issuer.

template <int kD> constexpr int kAStages = kD == 128 ? 3 : 4;
template <int kD> constexpr uint32_t kAStage = kBoxes<kD> * kTileBytes;       // Q boxes
template <int kD> constexpr uint32_t kBSub = kNb<kD> * 128;   // one 64-feature sub-tile of [S^T | z]
template <int kD> constexpr uint32_t kOffB = kAStages<kD> * kAStage<kD>;
template <int kD> constexpr uint32_t kOffO = kOffB<kD> + ((kBoxes<kD> * kBSub<kD> + 1023) & ~1023u);
template <int kD> constexpr size_t kASmem = 1024 + kOffO<kD> + 2 * kBoxes<kD> * kTileBytes;
constexpr int kAThreads = 576;
// TMEM buffer b at kTmStride b: the accumulator [num | den] (kNb columns), then
// phi(Q) (kD / 2 columns) at kTmQ.
template <int kD> constexpr uint32_t kTmStride = kD == 128 ? 256 : 128;
template <int kD> constexpr uint32_t kTmQ = kNb<kD>;

// phi of row `row` of a 128 x 64 bf16 box (128-byte swizzle), feature halves
// h0 .. h1 - 1 of 32, into 16 TMEM columns each at taddr + 16 h: the kind::f16
// A-operand layout (two features per column).
template <int kPhi>
__device__ __forceinline__ void phi_row_to_tmem(const uint8_t* tile, uint32_t taddr, int row, int h0,
                                                int h1) {
    for (int hlf = h0; hlf < h1; ++hlf) {
        uint32_t w[16];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint4 x = phi8<kPhi>(*reinterpret_cast<const uint4*>(
                tile + row * 128 + (((4 * hlf + c) ^ (row & 7)) << 4)));
            w[4 * c] = x.x;
            w[4 * c + 1] = x.y;
            w[4 * c + 2] = x.z;
            w[4 * c + 3] = x.w;
        }
        tmem_st16(taddr + 16 * hlf, w);
    }
}

template <int kD>
struct ApplyMisc {
    uint64_t full[kAStages<kD>], empty[kAStages<kD>], phi_done[kAStages<kD>];
    uint64_t o_full[2], o_free[2], b_ready, mma_drain;
    uint32_t tmem_slot;
};

template <int kD, int kPhi>
__global__ void __launch_bounds__(kAThreads, 1)
nc_apply_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap omap,
                const float* __restrict__ agg, Partition part, float eps, WsHeader* hdr) {
    constexpr int kStg = kAStages<kD>, kB = kBoxes<kD>, kN = kNb<kD>;
    constexpr uint32_t kStr = kTmStride<kD>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    __shared__ ApplyMisc<kD> m;
    const uint32_t max_spin = hdr->max_spin;
    const bool hold = hdr->hold_item != 0;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cta = blockIdx.x;
    const int64_t u0 = part.begin(cta), u1 = part.begin(cta + 1);
    const int nch = (int)(u1 - u0);
    auto stage = [&](int s) { return base + s * kAStage<kD>; };
    uint8_t* bop = base + kOffB<kD>;
    uint8_t* ostage = base + kOffO<kD>;

    if (tid == 0) {
        for (int s = 0; s < kStg; ++s) {
            mbar_init(&m.full[s], 1);
            mbar_init(&m.empty[s], 1);
            mbar_init(&m.phi_done[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&m.o_full[b], 1);
            mbar_init(&m.o_free[b], 1);
        }
        mbar_init(&m.b_ready, 1);
        mbar_init(&m.mma_drain, 1);
        fence_mbar_init();
    }
    // Zero the whole operand once (its padding rows stay zero).
    for (int idx = tid; idx < (int)(kB * kBSub<kD> / 16); idx += kAThreads)
        reinterpret_cast<uint4*>(bop)[idx] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    if (warp == 17) {
        tmem_alloc(&m.tmem_slot, 512);
        tmem_relinquish();
    }
    if (warp == 16 && lane == 0) {
        tma_prefetch_desc(&qmap);
        tma_prefetch_desc(&omap);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = m.tmem_slot;

    if (warp == 16) {
        // ---------------------------------------------------------- producer
        if (lane == 0) {
            int i = 0;
            for (; i < nch; ++i) {
                const int s = i % kStg;
                if (i >= kStg && !mbar_wait(&m.empty[s], ((i / kStg) - 1) & 1, max_spin)) {
                    report_timeout(hdr);
                    break;
                }
                if (hold) break;  // test hook: a load that is never issued
                const int64_t u = u0 + i;
                const int h = (int)(u / part.nchunks), ch = (int)(u % part.nchunks);
                mbar_arrive_expect_tx(&m.full[s], kB * kTileBytes);
#pragma unroll
                for (int bx = 0; bx < kB; ++bx)
                    tma_load_3d(stage(s) + bx * kTileBytes, &qmap, &m.full[s], 64 * bx, ch * kC, h);
            }
            for (int j = i - kStg > 0 ? i - kStg : 0; j < i; ++j)
                mbar_wait(&m.full[j % kStg], (j / kStg) & 1, kDefaultMaxSpin);
        }
    } else if (warp == 17) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(128, kN, false, false);
            const uint32_t ba = smem_u32(bop);
            int run = 0;
            bool ok = true;
            for (int i = 0; i < nch && ok; ++i) {
                const int s = i % kStg, b = i & 1;
                const int64_t u = u0 + i;
                const bool first_in_run = (i == 0) || (u % part.nchunks == 0);
                if (!mbar_wait(&m.phi_done[s], (i / kStg) & 1, max_spin) ||
                    (first_in_run && !mbar_wait(&m.b_ready, run & 1, max_spin)) ||
                    (i >= 2 && !mbar_wait(&m.o_free[b], ((i >> 1) - 1) & 1, max_spin))) {
                    ok = false;
                    break;
                }
                if (first_in_run) ++run;
                tc_fence_after();
#pragma unroll
                for (int k16 = 0; k16 < kD / 16; ++k16)
                    mma_bf16_ts(tmem + kStr * b, tmem + kStr * b + kTmQ<kD> + 8 * k16,
                           smem_desc(ba + (k16 >> 2) * kBSub<kD> + (k16 & 3) * 32, 16, 1024, kSwizzle128B),
                           idesc, k16 > 0);
                mma_commit(&m.o_full[b]);
            }
            if (!ok) report_timeout(hdr);
            mma_commit(&m.mma_drain);
            mbar_wait(&m.mma_drain, 0, kDefaultMaxSpin);
        }
    } else if (warp < 8) {
        // ---------------------------------------------------------- phi on Q
        const int t = tid;
        bool ok = true;
        // phi(Q) goes to TMEM next to the chunk's accumulator (the MMA's A
        // operand), so the stage is free as soon as it has been read. Warp w
        // takes query rows 32 (w & 3) .. + 31; D = 128: box w >> 2 (both feature
        // halves), D = 64: the one box, feature half w >> 2.
        const uint32_t lb = (uint32_t)(32 * (warp & 3)) << 16;
        const int bx = kB == 2 ? (warp >> 2) : 0;
        const int h0 = kB == 2 ? 0 : (warp >> 2), h1 = kB == 2 ? 2 : h0 + 1;
        for (int i = 0; i < nch; ++i) {
            const int s = i % kStg, b = i & 1;
            ok = mbar_wait(&m.full[s], (i / kStg) & 1, max_spin);
            // The buffer's previous chunk (i - 2) finished its MMA.
            if (ok && i >= 2) ok = mbar_wait(&m.o_full[b], ((i - 2) >> 1) & 1, max_spin);
            ok = __all_sync(0xffffffffu, ok);      // the TMEM stores below are warp-wide
            tc_fence_after();
            if (ok)
                phi_row_to_tmem<kPhi>(stage(s) + bx * kTileBytes,
                                      tmem + kStr * b + kTmQ<kD> + 32 * bx + lb, 32 * (warp & 3) + lane,
                                      h0, h1);
            tmem_st_wait();
            tc_fence_before();
            ok = named_bar_and(1, 256, ok);
            if (!ok) break;
            if (t == 0) {
                mbar_arrive(&m.empty[s]);
                mbar_arrive(&m.phi_done[s]);
            }
        }
        if (!ok && t == 0) report_timeout(hdr);
    } else {
        // ---------------------------------------------------------- operand build + epilogue
        constexpr int kF = kD / 2;              // features (build) or values (epilogue) per g
        const int t = tid - 256;                // 0..255
        const int q4 = warp & 3, g = (warp - 8) >> 2;
        const int row = 32 * q4 + lane;         // query row of the epilogue / operand row n
        const uint32_t lane_base = (uint32_t)(32 * q4) << 16;

        // [S^T | z_hi | z_lo] for head h: S = sum of every run of head h (all CTAs).
        auto build = [&](int h) {
            const int64_t hb = (int64_t)h * part.nchunks, he = hb + part.nchunks;
            // First CTA covering head h: largest c with begin(c) <= hb.
            int c_lo = (int)((hb * part.grid) / part.T);
            while (c_lo > 0 && part.begin(c_lo) > hb) --c_lo;
            while (c_lo + 1 < part.grid && part.begin(c_lo + 1) <= hb) ++c_lo;
            // Thread (row n, half g) sums column n of S over features c in
            // [kF g, kF g + kF) and writes S^T[n][c]; threads with g = 0 also own
            // z[n] (feature n). Rows n >= kD have no operand row.
            if (row < kD) {
                float acc[kF];
#pragma unroll
                for (int e = 0; e < kF; ++e) acc[e] = 0.f;
                float zacc = 0.f;
                for (int c2 = c_lo; c2 < part.grid && part.begin(c2) < he; ++c2) {
                    const int64_t b0 = part.begin(c2);
                    if (part.begin(c2 + 1) <= b0) continue;
                    const float* a = agg + ((int64_t)c2 * part.maxr + (h - b0 / part.nchunks)) * kE<kD>;
#pragma unroll
                    for (int e = 0; e < kF; ++e) acc[e] += a[(kF * g + e) * kD + row];
                    if (g == 0) zacc += a[kD * kD + row];
                }
                uint8_t* sub = bop + ((kF * g) >> 6) * kBSub<kD>;
                const int c0 = (kF * g) & 63;
#pragma unroll
                for (int c = 0; c < kF / 8; ++c) {
                    uint4 v = make_uint4(pack_bf16(acc[8 * c], acc[8 * c + 1]), pack_bf16(acc[8 * c + 2], acc[8 * c + 3]),
                                         pack_bf16(acc[8 * c + 4], acc[8 * c + 5]), pack_bf16(acc[8 * c + 6], acc[8 * c + 7]));
                    *reinterpret_cast<uint4*>(sub + sw128_offset(row, c0 + 8 * c)) = v;
                }
                if (g == 0) {
                    // z as two bf16 terms in rows kD (hi) and kD + 1 (lo), feature = row.
                    const uint32_t hi = pack_bf16(zacc, 0.f);
                    const uint32_t lo = pack_bf16(zacc - bf_lo(hi), 0.f);
                    uint8_t* zsub = bop + (row >> 6) * kBSub<kD>;
                    *reinterpret_cast<uint16_t*>(zsub + sw128_offset(kD, row & 63)) = (uint16_t)hi;
                    *reinterpret_cast<uint16_t*>(zsub + sw128_offset(kD + 1, row & 63)) = (uint16_t)lo;
                }
            }
            fence_proxy_async_smem();
            named_bar(2, 256);
            if (t == 0) mbar_arrive(&m.b_ready);
        };

        pdl_wait();  // the state kernel's aggregates are complete and visible
        bool ok = true;
        for (int i = 0; i < nch; ++i) {
            const int b = i & 1;
            const int64_t u = u0 + i;
            const int h = (int)(u / part.nchunks), ch = (int)(u % part.nchunks);
            // A new run: every MMA of the previous run has completed (its last
            // output was read below), so the operand can be rebuilt.
            if (i == 0 || ch == 0) build(h);
            ok = mbar_wait(&m.o_full[b], (i >> 1) & 1, max_spin);
            if (t == 0) tma_store_wait_read<1>();  // staging buffer b (chunk i - 2) is free again
            named_bar(2, 256);
            tc_fence_after();
            const uint32_t to = tmem + kStr * b + lane_base;
            float inv;
            {
                uint32_t rd[16];
                tmem_ld16(to + kD, rd);
                tmem_ld_wait();
                inv = 1.f / (__uint_as_float(rd[0]) + __uint_as_float(rd[1]) + eps);
            }
            // Value columns [kF g, kF g + kF): box (kF g) / 64, from column (kF g) % 64.
            uint8_t* ot = ostage + (kB * b + ((kF * g) >> 6)) * kTileBytes;
            const int c0 = (kF * g) & 63;
#pragma unroll
            for (int c2 = 0; c2 < kF / 32; ++c2) {
                uint32_t r0[16], r1[16];
                tmem_ld16(to + kF * g + 32 * c2, r0);
                tmem_ld16(to + kF * g + 32 * c2 + 16, r1);
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
                    *reinterpret_cast<uint4*>(ot + sw128_offset(row, c0 + 32 * c2 + 8 * c)) = v;
                }
            }
            tc_fence_before();
            fence_proxy_async_smem();
            ok = named_bar_and(2, 256, ok);
            if (!ok) break;
            if (t == 0) {
                mbar_arrive(&m.o_free[b]);
#pragma unroll
                for (int bx = 0; bx < kB; ++bx)
                    tma_store_3d(&omap, ostage + (kB * b + bx) * kTileBytes, 64 * bx, ch * kC, h);
                tma_store_commit();
            }
        }
        if (!ok && t == 0) report_timeout(hdr);
        if (t == 0) tma_store_wait_all<0>();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 17) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

static_assert(kSSmem<128> <= 232448 && kSSmem<64> <= 232448, "state kernel shared memory exceeds 227 KB");
static_assert(kASmem<128> <= 232448 && kASmem<64> <= 232448, "apply kernel shared memory exceeds 227 KB");

}  // namespace

bool tc_noncausal_supported(int D, int M, la_dtype dt) {
    return dt == LA_BF16 && D == M && (D == 64 || D == 128);
}

size_t tc_noncausal_workspace(int64_t BH, int N, int D) {
    Partition p = make_partition(BH, N, sm_count());
    return sizeof(float) * (size_t)p.grid * p.maxr * (size_t)(D * D + D);
}

namespace {

template <int kD>
cudaError_t launch_noncausal(const CUtensorMap& qm, const CUtensorMap& km, const CUtensorMap& vm,
                             const CUtensorMap& om, const Partition& p, int N, float eps, int fm,
                             WsHeader* hdr, float* agg, cudaStream_t st) {
    cudaError_t err;
    // One instantiation per feature map (elu + 1, identity), each with its own opt-in flag.
    const bool ident = fm == kPhiIdentity;
    auto state_kernel = ident ? nc_state_kernel<kD, kPhiIdentity> : nc_state_kernel<kD, kPhiElu1>;
    auto apply_kernel = ident ? nc_apply_kernel<kD, kPhiIdentity> : nc_apply_kernel<kD, kPhiElu1>;
    static std::atomic<int> optin_state[2][kMaxDevices], optin_apply[2][kMaxDevices];
    if ((err = ensure_smem_optin(state_kernel, (int)kSSmem<kD>, optin_state[ident]))) return err;
    if ((err = ensure_smem_optin(apply_kernel, (int)kASmem<kD>, optin_apply[ident]))) return err;
    state_kernel<<<p.grid, kSThreads, kSSmem<kD>, st>>>(km, vm, agg, p, N, hdr);
    if ((err = cudaPeekAtLastError())) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.grid);
    cfg.blockDim = dim3(kAThreads);
    cfg.dynamicSmemBytes = kASmem<kD>;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, apply_kernel, qm, om, (const float*)agg, p, eps, hdr);
}

}  // namespace

cudaError_t tc_run_sums128(const void* k, const void* v, float* agg, int64_t BH, int N, int fm,
                           bool last_only, void* ws_header, cudaStream_t st) {
    Partition p = make_partition(BH, N, sm_count());
    CUtensorMap kmap, vmap;
    if (!encode_bhnd(&kmap, k, BH, N, 128) || !encode_bhnd(&vmap, v, BH, N, 128))
        return cudaErrorInvalidValue;
    WsHeader* hdr = reinterpret_cast<WsHeader*>(ws_header);
    const bool ident = fm == kPhiIdentity;
    auto state_kernel = last_only ? (ident ? nc_state_kernel<128, kPhiIdentity, true> : nc_state_kernel<128, kPhiElu1, true>)
                                  : (ident ? nc_state_kernel<128, kPhiIdentity> : nc_state_kernel<128, kPhiElu1>);
    static std::atomic<int> optin[2][2][kMaxDevices];
    cudaError_t err = ensure_smem_optin(state_kernel, (int)kSSmem<128>, optin[last_only][ident]);
    if (err) return err;
    state_kernel<<<p.grid, kSThreads, kSSmem<128>, st>>>(kmap, vmap, agg, p, N, hdr);
    return cudaPeekAtLastError();
}

cudaError_t tc_noncausal(const void* q, const void* k, const void* v, void* o, int64_t BH, int N,
                         int D, float eps, int fm, void* ws_header, void* scratch, cudaStream_t st) {
    Partition p = make_partition(BH, N, sm_count());
    CUtensorMap qm, km, vm, om;
    if (!encode_bhnd(&qm, q, BH, N, D) || !encode_bhnd(&km, k, BH, N, D) ||
        !encode_bhnd(&vm, v, BH, N, D) || !encode_bhnd(&om, o, BH, N, D))
        return cudaErrorInvalidValue;
    WsHeader* hdr = reinterpret_cast<WsHeader*>(ws_header);
    float* agg = reinterpret_cast<float*>(scratch);
    return D == 128 ? launch_noncausal<128>(qm, km, vm, om, p, N, eps, fm, hdr, agg, st)
                    : launch_noncausal<64>(qm, km, vm, om, p, N, eps, fm, hdr, agg, st);
}

}  // namespace la
