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
// Work split: one persistent launch. The B*H*ceil(N/128) chunks form one
// head-major sequence cut into gridDim.x contiguous ranges, one per CTA. A
// range holds "runs" (its chunks of one head). Each CTA
//  1. sums [dS | dz] = phi(K)^T [V | 1] over its last run when that run's head
//     continues into the next range, and publishes the sum (fp32) in the
//     workspace as tagged words (value and launch tag in one 64-bit store);
//  2. if its first run continues a head from earlier ranges, looks back over
//     the ranges to its left and adds their published sums (or stops at the
//     first range that already published its inclusive prefix): the exclusive
//     prefix over segments, as in the parallel scan of the same blog, section
//     7.7, in fp32 (decoupled look-back);
//  3. runs the chunk loop above over its whole range with the running state
//     [S | z] in registers (fp32), writing each chunk's S_{c-1}, z_{c-1} as bf16
//     rows behind the Q, K, V tiles of its stage in shared memory.
// The last run's K and V are read twice (steps 1 and 3); the second read is
// expected to hit L2. Tags are the launch epoch from the workspace header plus
// one; the last CTA to finish advances the epoch.
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
constexpr int kE = kD * kD + kD;               // floats per published sum (S row-major, then z)

// Warp roles (24 warps):
//   warps 0-7   phi:   phi on the K (and Q) tiles of each landed slot or stage, in
//                      place; its first thread issues MMA (1) of the chunk when the
//                      chunk's TMEM buffer is already free (see below)
//   warps 8-15  epi:   two warps per TMEM lane quarter. Once per range: publish
//                      the last run's sum, look back, seed the running state.
//                      Then warps 8-11 (mask): A (fp32, TMEM) -> causal mask ->
//                      bf16 P in the same TMEM columns, and their first thread
//                      issues MMA (4) and, once the state rows are written, (3);
//                      warps 12-15 (output): num / (den + eps) to global memory
//   warps 16-18, 20-22 state: running state [S^T ; z] in registers (TMEM lanes
//                      0-95, two warps per lane quarter, 32 columns each): adds
//                      each chunk's [dS ; dz], writes the bf16 state rows of the
//                      next chunk and the final head states
//   warp 19     TMA producer
//   warp 23     MMA (2); allocates and frees TMEM
// MMA (1) of chunk i >= 2 needs phi of chunk i and the output warps' reads of
// chunk i - 2 (same TMEM buffer): both sides count themselves in on a counter
// of chunk i mod 4 and the one that arrives second issues it, so neither waits
// for a wake-up from the other.
// Per chunk i of the range (stage s, TMEM buffer b = i mod 2):
//   (1) A           = phi(Q) phi(K)^T                     M=128, N=128, K=64
//   (4) [num | den] = P [V | 1]                            M=128, N=80,  K=128
//   (3) [num | den] += phi(Q) [S^T | z_hi | z_lo | 0]^T    M=128, N=80,  K=64
//   (2) [dS^T ; dz]  = [V | 1]^T phi(K)                    M=128, N=64,  K=128
// (2) of chunk i fills one of two TMEM buffers; the state role adds it to the
// running state (fp32, registers) and writes the rows S^T, z_hi, z_lo of chunk
// i + 1's stage, which only (3) reads: neither the intra-chunk part
// (1) -> P -> (4) nor the next (2) waits for the state chain.
// Step 1 streams K and V through a deeper ring of 32 KB slots over the same
// shared memory; step 3 loads start once step 1 has released it.
constexpr int kPhiWarps = 8;
constexpr int kEpiW0 = kPhiWarps, kStateW0 = kEpiW0 + 8;       // state: 16-18 and 20-22
constexpr int kProdW = kStateW0 + 3, kStW = kProdW + 4;
constexpr int kThreads = 32 * (kStW + 1);
constexpr int kPhiThreads = 32 * kPhiWarps;
constexpr int kEpiThreads = 256;
constexpr int kStateThreads = 192;
// Named barriers: 1 phi, 2 mask warps, 3 output warps, 6 all epi, 7 state.
constexpr int kBarPhi = 1, kBarPair = 2, kBarEpi = 6, kBarState = 7;
constexpr int kStages = 3;
constexpr int kSlots = 5;                                      // step-1 ring: K, V
// Shared-memory map (offsets from a 1024-aligned base). A stage holds Q, K, the
// state rows (S^T, z_hi, z_lo, zero padding to 16 z rows) and V.
constexpr uint32_t kStQ = 0, kStK = kTileBytes, kStS = 2 * kTileBytes;
constexpr uint32_t kStZ = kStS + kD * 128, kStV = kStZ + 16 * 128;
constexpr uint32_t kStageBytes = kStV + kTileBytes;            // 58 KB
constexpr uint32_t kSlotBytes = 2 * kTileBytes;                // K then V
constexpr uint32_t kOffOnes = kStages * kStageBytes;           // [V | 1] second atom, MN-major
constexpr uint32_t kOffO = kOffOnes + kTileBytes;              // output staging tile
constexpr uint32_t kOffSum = kOffO + kTileBytes;               // look-back sum, fp32 [kE]
constexpr uint32_t kSmemEnd = kOffSum + kE * 4;
constexpr size_t kSmem = 1024 + kSmemEnd;
static_assert(kSlots * kSlotBytes <= kOffOnes, "step-1 ring overlaps the ones tile");
// TMEM columns. Buffer b (144 used): A at +0 (128; P overwrites +0..63 in place),
// [num | den] at +64 (80, written once A has been consumed).
constexpr uint32_t kTmBuf = 160;
constexpr uint32_t kTmNum = 64;
constexpr uint32_t kTmDelta = 320;                             // [dS^T ; dz], two buffers of 64
constexpr uint32_t kTmState = 448;                             // running state: 64 columns

struct Misc {
    uint64_t afull[kSlots], aphi[kSlots], aempty[kSlots];
    uint64_t full[kStages], phi_done[kStages], empty[kStages];
    uint64_t snap_ready[kStages], a_full[2], o_full[2];
    uint64_t a_done, ds_full[2], ds_free[2], drain[4];
    uint32_t tmem_slot;
    int qk_arrive[4];                          // arrivals for MMA (1), per chunk mod 4
    int walk_stop, walk_incl;
};

// Published sums are tagged words: bits of the fp32 value in the low half, the
// launch tag (epoch + 1) in the high half, stored and loaded as single 64-bit
// accesses, so a reader that sees the tag also sees the value: no fence or flag.
__device__ __forceinline__ void st_tagged(uint64_t* p, float v, uint32_t tag) {
    const uint64_t w = ((uint64_t)tag << 32) | __float_as_uint(v);
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}

__device__ __forceinline__ uint64_t ld_tagged(const uint64_t* p) {
    uint64_t w;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(w) : "l"(p) : "memory");
    return w;
}

__device__ __forceinline__ uint32_t tag_of(uint64_t w) { return (uint32_t)(w >> 32); }
__device__ __forceinline__ float value_of(uint64_t w) { return __uint_as_float((uint32_t)w); }

// Writes 16 fp32 values as bf16 into row `row`, columns c0..c0+15 of a swizzled tile.
__device__ __forceinline__ void put_row16(uint8_t* tile, int row, int c0, const float* f) {
#pragma unroll
    for (int h = 0; h < 2; ++h)
        *reinterpret_cast<uint4*>(tile + sw128_offset(row, c0 + 8 * h)) =
            make_uint4(pack_bf16(f[8 * h], f[8 * h + 1]), pack_bf16(f[8 * h + 2], f[8 * h + 3]),
                       pack_bf16(f[8 * h + 4], f[8 * h + 5]), pack_bf16(f[8 * h + 6], f[8 * h + 7]));
}

// z as two bf16 rows: z_hi = bf16(z) in row `row`, z_lo = bf16(z - z_hi) in row + 1.
__device__ __forceinline__ void put_z16(uint8_t* tile, int row, int c0, const float* f) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float a = f[8 * h + 2 * e], b = f[8 * h + 2 * e + 1];
            hi[e] = pack_bf16(a, b);
            lo[e] = pack_bf16(a - bf_lo(hi[e]), b - __uint_as_float(hi[e] & 0xFFFF0000u));
        }
        *reinterpret_cast<uint4*>(tile + sw128_offset(row, c0 + 8 * h)) =
            make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(tile + sw128_offset(row + 1, c0 + 8 * h)) =
            make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
}

// Element (column f, TMEM lane v) of a published sum: S[f][v] for v < 64, z[f] for v = 64.
__device__ __forceinline__ int sum_idx(int v, int f) { return v < kD ? f * kD + v : kD * kD + f; }

// Element idx (sum_idx layout) of the initial state of head h: S0[h][f][v], z0[h][f].
__device__ __forceinline__ float init_elem(const float* S0, const float* z0, int64_t h, int idx) {
    return idx < kD * kD ? S0[h * kD * kD + idx] : z0[h * kD + idx - kD * kD];
}

// kInit: the recurrence starts from (S0, z0) instead of zero. A separate
// instantiation: the extra code costs the zero-start kernel several µs (this
// kernel's timing is sensitive to code added anywhere in it). kPhi: the feature
// map the phi role applies (elu + 1, or the identity for features computed by
// the caller).
template <bool kInit, int kPhi>
__global__ void __launch_bounds__(kThreads, 1)
causal_fused_kernel(const __grid_constant__ CUtensorMap qmap,
                    const __grid_constant__ CUtensorMap kmap,
                    const __grid_constant__ CUtensorMap vmap,
                    const __grid_constant__ CUtensorMap omap, uint64_t* __restrict__ agg,
                    uint64_t* __restrict__ incl, const float* __restrict__ S0,
                    const float* __restrict__ z0, float* __restrict__ S_out,
                    float* __restrict__ z_out, Partition part, int N, float eps, WsHeader* hdr) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    __shared__ Misc m;
    // Launched as a programmatic dependent of the previous kernel in the stream:
    // the set-up below touches no global memory; griddepcontrol.wait then orders
    // everything after it behind that kernel's completion.
    pdl_launch_dependents();
    uint32_t max_spin = 0;
    bool hold = false;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cta = blockIdx.x;
    const int nchunks = part.nchunks;
    const int64_t u0 = part.begin(cta), u1 = part.begin(cta + 1);
    const int nch = (int)(u1 - u0);
    const int h0 = (int)(u0 / nchunks);
    const int64_t hb = (int64_t)h0 * nchunks;
    const int64_t head_end = hb + nchunks;
    const bool use_prefix = u0 != hb;                  // the first run continues a head
    const bool has_A = (u1 % nchunks) != 0;            // the last run's head continues
    const int64_t last_start = has_A ? max(u0, (u1 / nchunks) * (int64_t)nchunks) : u1;
    const int nA = (int)(u1 - last_start);             // chunks of step 1
    const bool publish_P = use_prefix && head_end > u1;
    auto stage = [&](int s) { return base + s * kStageBytes; };
    auto slot = [&](int a) { return base + (a % kSlots) * kSlotBytes; };
    // Stage of range chunk i is free once the chunk three earlier released it
    // (the first uses wait for step 1 to release the memory instead).
    auto wait_stage_free = [&](int i) -> bool {
        if (i < kStages) return nA == 0 || mbar_wait(&m.a_done, 0, max_spin);
        return mbar_wait(&m.empty[i % kStages], ((i / kStages) - 1) & 1, max_spin);
    };
    uint8_t* ones = base + kOffOnes;
    uint8_t* ostage = base + kOffO;

    if (tid == 0) {
        for (int a = 0; a < kSlots; ++a) {
            mbar_init(&m.afull[a], 1);
            mbar_init(&m.aphi[a], 1);
            mbar_init(&m.aempty[a], 1);
        }
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&m.full[s], 1);
            mbar_init(&m.phi_done[s], 1);
            mbar_init(&m.empty[s], 2);             // (2) and (4)+(3) both release it
            mbar_init(&m.snap_ready[s], 1);        // state rows of the stage's chunk written
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&m.a_full[b], 1);
            mbar_init(&m.o_full[b], 1);
            m.qk_arrive[b] = 0;
            m.qk_arrive[b + 2] = 0;
        }
        for (int d = 0; d < 4; ++d) mbar_init(&m.drain[d], 1);
        mbar_init(&m.a_done, 1);
        for (int d = 0; d < 2; ++d) {
            mbar_init(&m.ds_full[d], 1);
            mbar_init(&m.ds_free[d], 1);
        }
        fence_mbar_init();
    }
    if (warp < kProdW) init_ones_tile(ones, tid, 32 * kProdW);
    fence_proxy_async_smem();
    if (warp == kStW) {
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
    pdl_wait();
    max_spin = hdr->max_spin;
    hold = hdr->hold_item != 0;
    const uint32_t tmem = m.tmem_slot;
    const int q4 = warp & 3;                       // TMEM lane quarter of this warp
    const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
    const uint32_t onesa = smem_u32(ones);
    // MMA (1) of range chunk i into TMEM buffer i mod 2, then a_full.
    auto issue_qk = [&](int i) {
        const int s = i % kStages, b = i & 1;
        tc_fence_after();
        const uint32_t qa = smem_u32(stage(s) + kStQ), ka = smem_u32(stage(s) + kStK);
        const uint32_t tbuf = tmem + kTmBuf * b;
        const uint32_t id_qk = idesc_bf16_f32(128, 128, false, false);
#pragma unroll
        for (int k16 = 0; k16 < kD / 16; ++k16)
            mma_bf16(tbuf, smem_desc(qa + k16 * 32, 16, 1024, kSwizzle128B),
                     smem_desc(ka + k16 * 32, 16, 1024, kSwizzle128B), id_qk, k16 > 0);
        mma_commit(&m.a_full[b]);
    };
    // One of the two arrivals (phi of chunk i, output reads of chunk i - 2 from
    // TMEM buffer i mod 2) for MMA (1) of chunk i >= 2, on counter c = i mod 4;
    // true for the second one, whose thread then issues it. Chunks i and i + 4
    // share a counter, but the phi side reaches chunk i + 4 only after (3) of
    // chunk i + 1, hence after the output side counted in for chunk i, and the
    // output side reaches it only after phi of chunk i + 2: a chunk's two
    // arrivals are never mixed with another's, so the counter's old value is
    // odd exactly for the second.
    auto qk_second = [&](int c) -> bool {
        __threadfence_block();
        const int prev = atomicAdd(&m.qk_arrive[c], 1);
        __threadfence_block();
        return (prev & 1) != 0;
    };

    if (warp == kProdW) {
        // ---------------------------------------------------------- producer
        if (lane == 0) {
            bool ok = true;
            int a = 0, i = 0;
            for (; a < nA && ok && !hold; ++a) {   // hold: test hook, loads never issued
                if (a >= kSlots && !mbar_wait(&m.aempty[a % kSlots], ((a / kSlots) - 1) & 1, max_spin)) {
                    ok = false;
                    break;
                }
                const int64_t u = last_start + a;
                const int h = (int)(u / nchunks), ch = (int)(u % nchunks);
                uint64_t* bar = &m.afull[a % kSlots];
                mbar_arrive_expect_tx(bar, 2 * kTileBytes);
                tma_load_3d(slot(a), &kmap, bar, 0, ch * kC, h);
                tma_load_3d(slot(a) + kTileBytes, &vmap, bar, 0, ch * kC, h);
            }
            // Step-3 stages overlap the step-1 slots: start once step 1 is done.
            if (ok && !hold && nA > 0) ok = mbar_wait(&m.a_done, 0, max_spin);
            for (; i < nch && ok && !hold; ++i) {
                const int s = i % kStages;
                if (i >= kStages && !mbar_wait(&m.empty[s], ((i / kStages) - 1) & 1, max_spin)) {
                    ok = false;
                    break;
                }
                const int64_t u = u0 + i;
                const int h = (int)(u / nchunks), ch = (int)(u % nchunks);
                mbar_arrive_expect_tx(&m.full[s], 3 * kTileBytes);
                tma_load_3d(stage(s) + kStQ, &qmap, &m.full[s], 0, ch * kC, h);
                tma_load_3d(stage(s) + kStK, &kmap, &m.full[s], 0, ch * kC, h);
                tma_load_3d(stage(s) + kStV, &vmap, &m.full[s], 0, ch * kC, h);
            }
            if (!ok) report_timeout(hdr);
            // Every issued load lands before the CTA exits.
            for (int j = a - kSlots > 0 ? a - kSlots : 0; j < a; ++j)
                mbar_wait(&m.afull[j % kSlots], (j / kSlots) & 1, kDefaultMaxSpin);
            for (int j = i - kStages > 0 ? i - kStages : 0; j < i; ++j)
                mbar_wait(&m.full[j % kStages], (j / kStages) & 1, kDefaultMaxSpin);
        }
    } else if (warp == kStW) {
        // ---------------------------------------------------------- MMA (2)
        if (lane == 0) {
            const uint32_t id_st = idesc_bf16_f32(128, 64, true, true);
            auto issue_state = [&](uint32_t tst, uint8_t* kt, uint8_t* vt, bool fresh) {
                const uint32_t ka = smem_u32(kt), va = smem_u32(vt);
                const uint32_t lbo = onesa - va;
#pragma unroll
                for (int k16 = 0; k16 < kC / 16; ++k16)
                    mma_bf16(tst, smem_desc(va + k16 * 2048, lbo, 1024, kSwizzle128B),
                             smem_desc(ka + k16 * 2048, 1024, 1024, kSwizzle128B), id_st,
                             (fresh && k16 == 0) ? 0u : 1u);
            };
            bool ok = true;
            for (int a = 0; a < nA && ok; ++a) {
                if (!mbar_wait(&m.aphi[a % kSlots], (a / kSlots) & 1, max_spin)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                issue_state(tmem + kTmState, slot(a), slot(a) + kTileBytes, a == 0);
                mma_commit(&m.aempty[a % kSlots]);
            }
            if (ok && nA > 0) mma_commit(&m.a_done);
            for (int i = 0; i < nch && ok; ++i) {
                const int s = i % kStages;
                const int d = i & 1;
                // (2) of chunk i reuses the buffer of chunk i - 2 once the state role added it
                // (and, for chunk 0 after step 1, once the step-1 sum was read and replaced).
                if (!mbar_wait(&m.phi_done[s], (i / kStages) & 1, max_spin) ||
                    (i >= 2 && !mbar_wait(&m.ds_free[d], ((i >> 1) - 1) & 1, max_spin))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                issue_state(tmem + kTmDelta + 64 * d, stage(s) + kStK, stage(s) + kStV, true);
                mma_commit(&m.ds_full[d]);
                mma_commit(&m.empty[s]);
            }
            if (!ok) report_timeout(hdr);
            mma_commit(&m.drain[2]);  // every issued MMA completes before TMEM is released
            mbar_wait(&m.drain[2], 0, kDefaultMaxSpin);
        }
    } else if (warp < kEpiW0) {
        // ---------------------------------------------------------- phi role
        const int t = tid;
        bool ok = true;
        for (int a = 0; a < nA && ok; ++a) {
            const int ch = (int)((last_start + a) % nchunks);
            ok = mbar_wait(&m.afull[a % kSlots], (a / kSlots) & 1, max_spin);
            phi_tile_256<kPhi>(slot(a), t, min(kC, N - ch * kC));
            fence_proxy_async_smem();
            ok = named_bar_and(kBarPhi, kPhiThreads, ok);
            if (ok && t == 0) mbar_arrive(&m.aphi[a % kSlots]);
        }
        // The first thread's own wait may fail after the barrier; it then carries
        // ok = false into the next barrier, which every phi thread still reaches.
        for (int i = 0; i < nch; ++i) {
            const int s = i % kStages;
            const int ch = (int)((u0 + i) % nchunks);
            if (ok) ok = mbar_wait(&m.full[s], (i / kStages) & 1, max_spin);
            if (ok)
                phi_tiles2_256<kPhi>(stage(s) + kStK, min(kC, N - ch * kC), stage(s) + kStQ, kC, t);
            fence_proxy_async_smem();
            ok = named_bar_and(kBarPhi, kPhiThreads, ok);
            if (!ok) break;
            if (t == 0) {
                mbar_arrive(&m.phi_done[s]);
                // Count in for (1) without waiting: the counters (one per chunk mod 4)
                // keep different chunks' arrivals apart.
                if (ok && (i < 2 || qk_second(i & 3))) issue_qk(i);
            }
        }
        if (t == 0) {
            if (!ok) report_timeout(hdr);
            mma_commit(&m.drain[0]);  // every issued MMA completes before TMEM is released
            mbar_wait(&m.drain[0], 0, kDefaultMaxSpin);
        }
    } else if (warp < kEpiW0 + 8) {
        // ---------------------------------------------------------- epi role
        // Thread (quarter q4, half hh, lane) owns TMEM lane v = 32 q4 + lane and,
        // where 64 columns are split, columns 32 hh .. 32 hh + 31.
        const int t = tid - 32 * kEpiW0;          // 0..255
        const int hh = (warp - kEpiW0) >> 2;      // 0 or 1
        const int v = 32 * q4 + lane;
        const uint32_t tst = tmem + kTmState + lane_base + 32 * hh;
        const uint32_t epoch1 = *reinterpret_cast<volatile uint32_t*>(&hdr->epoch) + 1u;
        uint64_t* my_agg = agg + (int64_t)cta * kE;
        float* sum_s = reinterpret_cast<float*>(base + kOffSum);
        bool ok = true;
        // Step 1: publish the last run's sum (fp32, tagged); keep a copy in shared
        // memory for this range's inclusive prefix.
        if (nA > 0) {
            ok = mbar_wait(&m.a_done, 0, max_spin);
            tc_fence_after();
            uint32_t r[2][16];
            tmem_ld16(tst, r[0]);
            tmem_ld16(tst + 16, r[1]);
            tmem_ld_wait();
            tc_fence_before();
            if (v <= kD) {
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int idx = sum_idx(v, 32 * hh + e);
                    float x = __uint_as_float(r[e >> 4][e & 15]);
                    // A last run that starts its head carries the head's initial state.
                    if constexpr (kInit)
                        if (last_start % nchunks == 0) x += init_elem(S0, z0, last_start / nchunks, idx);
                    st_tagged(my_agg + idx, x, epoch1);
                    sum_s[idx] = x;
                }
            }
        }
        // Step 2: look back over the ranges to the left for the head's earlier
        // part: a range's inclusive prefix ends the walk, else its sum is added and
        // the walk goes on until the range that holds the head's start. The first
        // epi warp polls 32 ranges at once (lane l: range cta - 1 - l - 32 w).
        int stop = cta, stop_incl = 0;
        if (ok && use_prefix && warp == kEpiW0) {
            bool found = false;
            const uint64_t t0 = global_ns();
            int win = cta - 1;                     // range polled by lane 0
            while (!found) {
                const int r2 = win - lane;
                bool isP = false, isA = false, isH = false;
                if (r2 >= 0) {
                    const uint64_t pw = ld_tagged(incl + (int64_t)r2 * kE);
                    const uint64_t aw = ld_tagged(agg + (int64_t)r2 * kE);
                    isP = tag_of(pw) == epoch1;
                    isA = tag_of(aw) == epoch1;
                    isH = part.begin(r2) <= hb;
                }
                const uint32_t endm = __ballot_sync(0xffffffffu, isP || (isA && isH));
                const uint32_t am = __ballot_sync(0xffffffffu, isA);
                const uint32_t pm = __ballot_sync(0xffffffffu, isP);
                if (endm != 0u) {
                    const int e = __ffs(endm) - 1;
                    const uint32_t before = (1u << e) - 1u;     // lanes whose sums are added
                    if ((am & before) == before) {
                        stop = win - e;
                        stop_incl = (pm >> e) & 1u;
                        found = true;
                    }
                } else if (am == 0xffffffffu) {
                    win -= 32;                     // all 32 published, none ends the walk
                }
                // One lane's clock decides, so that the whole warp leaves together.
                const int late = __shfl_sync(0xffffffffu, (int)(global_ns() - t0 > (uint64_t)max_spin * 1000u), 0);
                if (!found && late) break;
            }
            if (lane == 0) {
                m.walk_stop = found ? stop : -1;
                m.walk_incl = stop_incl;
            }
        }
        // Seed: state before the range = prefix (or zero) for chunk 0's rows and
        // the state role; inclusive prefix for ranges to the right.
        if (ok && nA > 0) ok = mbar_wait(&m.a_done, 0, max_spin);   // stage memory is free
        ok = named_bar_and(kBarEpi, kEpiThreads, ok);
        if (ok && use_prefix) {
            stop = m.walk_stop;
            stop_incl = m.walk_incl;
            ok = stop >= 0;
            if (!ok) stop = cta;
        }
        if (ok) {
            // Prefix sum in fp32, element idx = t + 256 k, staged in shared memory.
            // Every word is checked for this launch's tag (re-read until it holds it).
            constexpr int kPer = (kE + kEpiThreads - 1) / kEpiThreads;   // 17
            float acc[kPer];
#pragma unroll
            for (int k = 0; k < kPer; ++k) {
                // A range that starts its head starts from the head's initial state.
                const int idx = t + kEpiThreads * k;
                acc[k] = 0.f;
                if constexpr (kInit)
                    if (!use_prefix && idx < kE) acc[k] = init_elem(S0, z0, h0, idx);
            }
            const uint64_t t0 = global_ns();
            for (int r2 = stop; r2 < cta && ok; ++r2) {
                const uint64_t* src = (r2 == stop && stop_incl ? incl : agg) + (int64_t)r2 * kE;
                uint64_t w[kPer];
#pragma unroll
                for (int k = 0; k < kPer; ++k) {
                    const int idx = t + kEpiThreads * k;
                    w[k] = idx < kE ? ld_tagged(src + idx) : ((uint64_t)epoch1 << 32);
                }
#pragma unroll
                for (int k = 0; k < kPer; ++k) {
                    const int idx = t + kEpiThreads * k;
                    while (tag_of(w[k]) != epoch1) {
                        if (global_ns() - t0 > (uint64_t)max_spin * 1000u) {
                            ok = false;
                            break;
                        }
                        w[k] = ld_tagged(src + idx);
                    }
                    acc[k] += value_of(w[k]);
                }
            }
#pragma unroll
            for (int k = 0; k < kPer; ++k) {
                const int idx = t + kEpiThreads * k;
                if (idx < kE) {
                    if (publish_P) st_tagged(incl + (int64_t)cta * kE + idx, acc[k] + sum_s[idx], epoch1);
                    sum_s[idx] = acc[k];
                }
            }
            // z padding rows 2-15 of every stage (the (3) operand's last 14 rows).
            for (int idx = t; idx < kStages * 112; idx += kEpiThreads) {
                const int s = idx / 112, r = idx % 112;
                *reinterpret_cast<uint4*>(stage(s) + kStZ + 256 + r * 16) = make_uint4(0, 0, 0, 0);
            }
            ok = named_bar_and(kBarEpi, kEpiThreads, ok);
            // This thread's TMEM lane v, columns 32 hh .. 32 hh + 31.
            uint8_t* st0 = stage(0) + kStS;
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2) {
                float f[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) f[e] = v <= kD ? sum_s[sum_idx(v, 32 * hh + 16 * c2 + e)] : 0.f;
                if (v < kD) put_row16(st0, v, 32 * hh + 16 * c2, f);
                else if (v == kD) put_z16(st0, kD, 32 * hh + 16 * c2, f);
            }
            fence_proxy_async_smem();
            named_bar(kBarEpi, kEpiThreads);
            if (ok && t == 0) mbar_arrive(&m.snap_ready[0]);
        }
        if (hh == 0) {
            // ------------------------------------------------------ mask (warps 8-11)
            // A block j (32 keys, columns 32j..32j+31) -> P block j (16 packed
            // columns 16j..16j+15) in the same TMEM buffer; in increasing j every A
            // column is read before the P columns that cover it are written. Blocks
            // past the diagonal block q4 are zero for this lane quarter. The first
            // thread then issues (4) [num | den] = P [V | 1] and, once the state
            // rows of the chunk are written, (3) += phi(Q) [S^T | z]. Its waits may
            // fail after the barrier: it then carries ok = false into the next
            // barrier, which every mask thread still reaches.
            const int tm = t;                             // 0..127
            const uint32_t id_pv = idesc_bf16_f32(128, 80, false, true);
            const uint32_t id_qs = idesc_bf16_f32(128, 80, false, false);
            for (int i = 0; i < nch; ++i) {
                const int b = i & 1, s = i % kStages;
                const uint32_t tbuf = tmem + kTmBuf * b + lane_base;
                if (ok) ok = mbar_wait(&m.a_full[b], (i >> 1) & 1, max_spin);
                tc_fence_after();
                for (int j = 0; ok && j <= q4; ++j) {
                    uint32_t r0[16], r1[16];
                    tmem_ld16(tbuf + 32 * j, r0);
                    tmem_ld16(tbuf + 32 * j + 16, r1);
                    tmem_ld_wait();
                    // Diagonal block: key 32 q4 + e <= row 32 q4 + lane.
                    uint32_t p[16];
                    if (j < q4) pack_block32(r0, r1, p);
                    else pack_block32_diag(r0, r1, lane, p);
                    tmem_st16(tbuf + 16 * j, p);
                }
                for (int j = q4 + 1; ok && j < 4; ++j) {
                    uint32_t p[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) p[e] = 0u;
                    tmem_st16(tbuf + 16 * j, p);
                }
                tmem_st_wait();
                tc_fence_before();
                ok = named_bar_and(kBarPair, 128, ok);
                if (!ok) break;
                if (tm == 0) {
                    tc_fence_after();
                    const uint32_t va = smem_u32(stage(s) + kStV);
                    const uint32_t lbo = onesa - va;
                    const uint32_t tb = tmem + kTmBuf * b;
#pragma unroll
                    for (int k16 = 0; k16 < kC / 16; ++k16)
                        mma_bf16_ts(tb + kTmNum, tb + 8 * k16,
                                    smem_desc(va + k16 * 2048, lbo, 1024, kSwizzle128B), id_pv,
                                    k16 > 0);
                    ok = mbar_wait(&m.snap_ready[s], (i / kStages) & 1, max_spin);
                    if (ok) {
                        tc_fence_after();
                        const uint32_t qa = smem_u32(stage(s) + kStQ), sa = smem_u32(stage(s) + kStS);
#pragma unroll
                        for (int k16 = 0; k16 < kD / 16; ++k16)
                            mma_bf16(tb + kTmNum, smem_desc(qa + k16 * 32, 16, 1024, kSwizzle128B),
                                     smem_desc(sa + k16 * 32, 16, 1024, kSwizzle128B), id_qs, 1u);
                        mma_commit(&m.o_full[b]);
                        mma_commit(&m.empty[s]);  // (1) of the chunk completed before P existed
                    }
                }
            }
            if (tm == 0) {
                if (!ok) report_timeout(hdr);
                mma_commit(&m.drain[1]);
                mbar_wait(&m.drain[1], 0, kDefaultMaxSpin);
            }
        } else {
            // ------------------------------------------------------ output (warps 12-15)
            // Thread = query row v of its lane quarter. The TMEM buffer is released
            // as soon as num and den are in registers (scaled and packed to bf16):
            // the first thread counts in for MMA (1) of chunk j + 2.
            const int to_t = t - 128;                     // 0..127
            for (int j = 0; j < nch && ok; ++j) {
                const int bj = j & 1;
                const int64_t u = u0 + j;
                const int h = (int)(u / nchunks), ch = (int)(u % nchunks);
                ok = mbar_wait(&m.o_full[bj], (j >> 1) & 1, max_spin);
                tc_fence_after();
                const uint32_t to = tmem + kTmBuf * bj + kTmNum + lane_base;
                // Two TMEM round trips: den (two columns) with num 0..31, then num 32..63.
                uint32_t o[32];
                {
                    uint32_t rd[2], r[2][16];
                    tmem_ld2(to + 64, rd);
                    tmem_ld16(to, r[0]);
                    tmem_ld16(to + 16, r[1]);
                    tmem_ld_wait();
                    const float inv = 1.f / (__uint_as_float(rd[0]) + __uint_as_float(rd[1]) + eps);
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        o[e] = pack_bf16(__uint_as_float(r[e >> 3][2 * (e & 7)]) * inv,
                                         __uint_as_float(r[e >> 3][2 * (e & 7) + 1]) * inv);
                    tmem_ld16(to + 32, r[0]);
                    tmem_ld16(to + 48, r[1]);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        o[16 + e] = pack_bf16(__uint_as_float(r[e >> 3][2 * (e & 7)]) * inv,
                                              __uint_as_float(r[e >> 3][2 * (e & 7) + 1]) * inv);
                }
                tc_fence_before();
                ok = named_bar_and(kBarPair + 1, 128, ok);
                if (!ok) break;
                if (to_t == 0) {
                    if (j + 2 < nch && qk_second((j + 2) & 3)) issue_qk(j + 2);
                    tma_store_wait_read<0>();             // the staging tile is free again
                }
                named_bar(kBarPair + 1, 128);
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    *reinterpret_cast<uint4*>(ostage + sw128_offset(v, 8 * c)) =
                        make_uint4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
                fence_proxy_async_smem();
                named_bar(kBarPair + 1, 128);
                if (to_t == 0) {
                    tma_store_3d(&omap, ostage, 0, ch * kC, h);
                    tma_store_commit();
                }
            }
            if (to_t == 0) {
                if (!ok) report_timeout(hdr);
                tma_store_wait_all<0>();
                mma_commit(&m.drain[3]);
                mbar_wait(&m.drain[3], 0, kDefaultMaxSpin);
            }
        }
    } else {
        // ---------------------------------------------------------- state role
        // Thread (half hh, lane v) owns row v of [S^T ; z] (v < 64: value v over
        // the features; v = 64: z), columns 32 hh .. 32 hh + 31, in registers.
        // Threads with v > 64 only take part in the warp-wide TMEM loads.
        const int hh = warp >= kProdW + 1 ? 1 : 0;
        const int t = (warp - (hh ? kProdW + 1 : kStateW0)) * 32 + lane;   // TMEM lane 0..95
        const int ts = hh * 96 + t;
        const uint32_t tds0 = tmem + kTmDelta + lane_base + 32 * hh;
        // The epi role seeded the prefix (or zero) into the shared sum buffer.
        bool ok = mbar_wait(&m.snap_ready[0], 0, max_spin);
        ok = named_bar_and(kBarState, kStateThreads, ok);
        float srun[32];
        {
            const float* sum_s = reinterpret_cast<const float*>(base + kOffSum);
#pragma unroll
            for (int e = 0; e < 32; ++e) srun[e] = t <= kD ? sum_s[sum_idx(t, 32 * hh + e)] : 0.f;
        }
        // Chunk i: state after it = state before + [dS ; dz] of chunk i. That is the
        // final head state at a head's last chunk (and the state restarts at zero),
        // else the rows of chunk i + 1.
        for (int i = 0; i < nch && ok; ++i) {
            const int d = i & 1;
            const int64_t u = u0 + i;
            const int h = (int)(u / nchunks);
            const bool head_last = (u % nchunks) == nchunks - 1;
            const bool next = i + 1 < nch;
            ok = mbar_wait(&m.ds_full[d], (i >> 1) & 1, max_spin);
            if (ok && next) ok = wait_stage_free(i + 1);
            tc_fence_after();
            {
                uint32_t r[2][16];
                tmem_ld16(tds0 + 64 * d, r[0]);
                tmem_ld16(tds0 + 64 * d + 16, r[1]);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 32; ++e) srun[e] += __uint_as_float(r[e >> 4][e & 15]);
            }
            tc_fence_before();
            if (head_last) {
                // Final head state: through the (now unused) look-back sum buffer in
                // shared memory, then copied out row-major by all state threads
                // (direct per-element global stores cost registers in this loop).
                float* sum_w = reinterpret_cast<float*>(base + kOffSum);
                if (t <= kD) {
#pragma unroll
                    for (int e = 0; e < 32; ++e) sum_w[sum_idx(t, 32 * hh + e)] = srun[e];
                }
                named_bar(kBarState, kStateThreads);
                for (int idx = ts; idx < kE; idx += kStateThreads) {
                    if (idx < kD * kD) {
                        if (S_out) S_out[(int64_t)h * kD * kD + idx] = sum_w[idx];
                    } else if (z_out) {
                        z_out[(int64_t)h * kD + idx - kD * kD] = sum_w[idx];
                    }
                }
                // The next head (if this range holds its start) begins at its initial state.
#pragma unroll
                for (int e = 0; e < 32; ++e) srun[e] = 0.f;
                if constexpr (kInit) {
                    if (next && t <= kD) {
#pragma unroll
                        for (int e = 0; e < 32; ++e) srun[e] = init_elem(S0, z0, h + 1, sum_idx(t, 32 * hh + e));
                    }
                }
            }
            if (next) {
                uint8_t* stn = stage((i + 1) % kStages) + kStS;
                if (t < kD) {
                    put_row16(stn, t, 32 * hh, srun);
                    put_row16(stn, t, 32 * hh + 16, srun + 16);
                } else if (t == kD) {
                    put_z16(stn, kD, 32 * hh, srun);
                    put_z16(stn, kD, 32 * hh + 16, srun + 16);
                }
                fence_proxy_async_smem();
            }
            ok = named_bar_and(kBarState, kStateThreads, ok);
            if (!ok) break;
            if (ts == 0) {
                mbar_arrive(&m.ds_free[d]);      // (2) of chunk i + 2 may refill this buffer
                if (next) mbar_arrive(&m.snap_ready[(i + 1) % kStages]);
            }
        }
        if (!ok && ts == 0) report_timeout(hdr);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kStW) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
    if (tid == 0) {
        // The last CTA to finish advances the epoch for the next launch.
        __threadfence();
        if (atomicAdd(&hdr->done, 1u) == (uint32_t)gridDim.x - 1u) {
            hdr->done = 0;
            __threadfence();
            atomicAdd(&hdr->epoch, 1u);
        }
    }
}

static_assert(kSmem <= 232448, "shared memory exceeds 227 KB");

int grid_cap() { return sm_count(); }

}  // namespace

bool tc_causal_supported(int D, int M, la_dtype dt) {
    return dt == LA_BF16 && D == M && (D == 64 || D == 128);
}

// Workspace after the header. D = 64: per CTA one published sum and one
// inclusive prefix (tagged 64-bit words). D = 128: the run sums and seeds.
size_t tc_causal_workspace(int64_t BH, int N, int D) {
    if (D == 128) return tc_causal128_workspace(BH, N);
    Partition p = make_partition(BH, N, grid_cap());
    return 2 * sizeof(uint64_t) * (size_t)p.grid * kE;
}

int tc_causal_launches(int D, int64_t BH, int N) { return D == 128 ? tc_causal128_launches(BH, N) : 1; }

cudaError_t tc_causal(const void* q, const void* k, const void* v, void* o, int64_t BH, int N,
                      int D, float eps, int fm, const float* S0, const float* z0, float* S_out,
                      float* z_out, void* ws_header, void* scratch, cudaStream_t st) {
    if (D == 128)
        return tc_causal128(q, k, v, o, BH, N, eps, fm, S0, z0, S_out, z_out, ws_header, scratch, st);
    Partition p = make_partition(BH, N, grid_cap());
    WsHeader* hdr = reinterpret_cast<WsHeader*>(ws_header);
    uint64_t* agg = reinterpret_cast<uint64_t*>(scratch);
    uint64_t* incl = agg + (size_t)p.grid * kE;
    CUtensorMap qm, km, vm, om;
    if (!encode_bhnd(&qm, q, BH, N, kD) || !encode_bhnd(&km, k, BH, N, kD) ||
        !encode_bhnd(&vm, v, BH, N, kD) || !encode_bhnd(&om, o, BH, N, kD))
        return cudaErrorInvalidValue;
    cudaError_t err;
    // One instantiation per (initial state, feature map), each with its own opt-in flag.
    using Kernel = decltype(&causal_fused_kernel<false, kPhiElu1>);
    static std::atomic<int> optin[4][kMaxDevices];
    const Kernel kernels[4] = {causal_fused_kernel<false, kPhiElu1>,
                               causal_fused_kernel<true, kPhiElu1>,
                               causal_fused_kernel<false, kPhiIdentity>,
                               causal_fused_kernel<true, kPhiIdentity>};
    const int variant = (S0 ? 1 : 0) + (fm == kPhiIdentity ? 2 : 0);
    if ((err = ensure_smem_optin(kernels[variant], (int)kSmem, optin[variant]))) return err;
    // Programmatic stream serialization: the next call's CTAs may be scheduled on
    // SMs as this launch's CTAs finish and run their set-up; the kernel waits
    // (griddepcontrol.wait) before its first global-memory access.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernels[variant], qm, km, vm, om, agg, incl, S0, z0, S_out,
                              z_out, p, N, eps, hdr);
}

}  // namespace la
