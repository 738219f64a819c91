// Tensor-core (tcgen05) causal forward for bf16 inputs, Dk = Dv = 128.
//
// Method. For chunk c of 128 tokens of one head, with [S | z] the state after
// the chunks before it ("Why Replace Attention? The Softmax Bottleneck and the
// Path to Linear Time", sections 7.1-7.2: S_i and z_i are prefix sums, so a
// chunk can be added at once and the rest regrouped exactly):
//   P           = bf16( mask_{key <= query}( phi(Q_c) phi(K_c)^T ) )
//   [num | den] = P [V_c | 1] + phi(Q_c) [S | z_hi | z_lo]
//   o_i         = num_i / (den_i + eps)
//   [S | z]    += phi(K_c)^T [V_c | 1]
// S is kept Dk x Dv (feature rows), so the state update is one MMA with the
// features as M, and z falls out of the ones column of [V | 1].
//
// At 128 features a chunk's tiles and accumulators are twice those of the
// 64-wide fused kernel, so the work is two or three launches over the
// persistent chunk partition (each CTA one contiguous range of the head-major
// chunk sequence):
//   1. run sums (nc_state_kernel<128, *, true>, noncausal_tc.cu): S_run =
//      phi(K)^T V and z_run (fp32) of each range's last run when its head
//      continues into the next range, the only runs a seed adds up (a range to
//      the left of range c that holds part of c's first head has it as its
//      last run); other chunks are not read;
//   2. c128_seed_kernel: per CTA the state before its first chunk, the head's
//      initial state plus the sums of that head's runs in the ranges to the
//      left (an exclusive prefix over segments, same blog, section 7.7, as a
//      segmented scan over the ranges), fp32. Where every head spans at most
//      kWalkMax + 1 ranges, the output kernel sums its own seed instead and this
//      launch is skipped;
//   3. c128_out_kernel: each CTA walks its range chunk by chunk. The running
//      state lives in TMEM as fp32 and is advanced by the state MMA itself
//      (accumulate); after each chunk a bf16 copy (z as hi + lo) is written to
//      shared memory as the B operand of the next chunk's phi(Q) [S | z].
// Launches 2 and 3 are programmatic dependents of the launch before them. The
// workspace holds one last-run sum and one seed per CTA.
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_common.cuh"
#include "tc_util.cuh"

namespace la {

namespace {

using namespace tc;
using namespace tcc;

constexpr int kD = 128;
constexpr int kE = kD * kD + kD;               // floats per state: S [f][v] row-major, then z [f]

// ======================================================== seed kernel
// seed(c) = init(h0) when range c starts its head h0, else carry(c - 1), where
// carry(c) = (its last head is h0 ? seed(c) : init(last head)) + last run sum(c)
// is what range c passes to the next one. This is a segmented scan over the
// ranges, done per block for 32 state elements (lane = element): each of the 16
// warps scans one segment of the ranges with an unknown carry-in, the segments'
// carries are chained, and each warp writes its segment's seeds.
constexpr int kSeedMaxGrid = 1024;
constexpr int kSeedWarps = 16;
// Where no range's first head reaches back over more than this many ranges, the
// output kernel sums its seed from the run sums itself and the scan is skipped.
constexpr int kWalkMax = 4;

// Ranges to the left of range c that hold part of its first head (0 when the
// range starts its head), counted up to kWalkMax + 1.
__host__ __device__ inline int left_walk(const Partition& p, int c) {
    const int64_t u0 = p.begin(c), hb = u0 / p.nchunks * p.nchunks;
    if (u0 == hb) return 0;
    int w = 0;
    for (int c2 = c - 1; c2 >= 0 && w <= kWalkMax; --c2) {
        ++w;
        if (p.begin(c2) <= hb) break;
    }
    return w;
}

struct RangeInfo {
    int flags;        // 1: starts its first head; 2: its last head continues
    int h0, hl;       // first and last head
};

__global__ void __launch_bounds__(32 * kSeedWarps)
c128_seed_kernel(const float* __restrict__ agg, float* __restrict__ seeds, Partition p,
                 const float* __restrict__ S0, const float* __restrict__ z0) {
    __shared__ RangeInfo info[kSeedMaxGrid];
    __shared__ float seg_val[kSeedWarps][32];
    __shared__ int seg_reset[kSeedWarps][32];
    __shared__ float seg_in[kSeedWarps][32];
    pdl_launch_dependents();
    const int G = p.grid, nch = p.nchunks;
    for (int c = threadIdx.x; c < G; c += blockDim.x) {
        const int64_t u0 = p.begin(c), u1 = p.begin(c + 1);
        RangeInfo r;
        r.h0 = (int)(u0 / nch);
        r.hl = (int)((u1 - 1) / nch);
        r.flags = (u0 % nch == 0 ? 1 : 0) | (u1 % nch != 0 ? 2 : 0);
        info[c] = r;
    }
    __syncthreads();
    pdl_wait();
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int idx = blockIdx.x * 32 + lane;
    const bool live = idx < kE;
    auto init = [&](int h) -> float {
        if (!S0 || !live) return 0.f;
        return idx < kD * kD ? S0[(int64_t)h * kD * kD + idx] : z0[(int64_t)h * kD + idx - kD * kD];
    };
    auto last_sum = [&](int c) -> float { return live ? agg[(int64_t)c * kE + idx] : 0.f; };
    const int L = (G + kSeedWarps - 1) / kSeedWarps;
    const int c0 = min(G, w * L), c1 = min(G, c0 + L);
    // The last-run sums of 8 ranges are loaded before they are used, so that a
    // warp has 8 loads in flight instead of one.
    auto load8 = [&](int cb, float (&a)[8]) {
#pragma unroll
        for (int j = 0; j < 8; ++j)
            a[j] = (cb + j < c1 && (info[cb + j].flags & 2)) ? last_sum(cb + j) : 0.f;
    };
    // Pass 1: the segment's carry-out as (reset, v): v if a reset happened in the
    // segment, else carry-in + v.
    bool reset = false;
    float val = 0.f;
    for (int cb = c0; cb < c1; cb += 8) {
        float a[8];
        load8(cb, a);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int c = cb + j;
            if (c >= c1) break;
            const RangeInfo r = info[c];
            if (r.flags & 1) {
                reset = true;
                val = init(r.h0);
            }
            // val is now seed(c) (relative to the carry-in when no reset yet).
            if (r.flags & 2) {
                if (r.hl != r.h0) {
                    reset = true;
                    val = init(r.hl);
                }
                val += a[j];
            } else {
                reset = true;   // the next range starts a head: nothing is carried
                val = 0.f;
            }
        }
    }
    seg_val[w][lane] = val;
    seg_reset[w][lane] = reset;
    __syncthreads();
    if (w == 0) {
        float carry = 0.f;
        for (int sg = 0; sg < kSeedWarps; ++sg) {
            seg_in[sg][lane] = carry;
            carry = seg_reset[sg][lane] ? seg_val[sg][lane] : carry + seg_val[sg][lane];
        }
    }
    __syncthreads();
    // Pass 2: the seeds, from the segment's carry-in.
    float carry = seg_in[w][lane];
    for (int cb = c0; cb < c1; cb += 8) {
        float a[8];
        load8(cb, a);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int c = cb + j;
            if (c >= c1) break;
            const RangeInfo r = info[c];
            const float seed = (r.flags & 1) ? init(r.h0) : carry;
            if (live) seeds[(int64_t)c * kE + idx] = seed;
            carry = (r.flags & 2) ? (r.hl == r.h0 ? seed : init(r.hl)) + a[j] : 0.f;
        }
    }
}

// ======================================================== output kernel
// Warp roles (22 warps):
//   warps 0-3    mask:   A (fp32, TMEM) -> causal mask -> bf16 P in place
//   warps 4-7    output: [num | den] (TMEM) -> o = num / (den + eps) -> bf16,
//                        staged in the chunk's Q buffer, TMA store
//   warps 8-11   state:  seed, the bf16 [S | z_hi | z_lo] operand after each
//                        chunk, resets and final states at head boundaries
//   warps 12-19  phi:    phi on the chunk's Q and K tiles in place
//   warp 20      TMA producer
//   warp 21      MMA issuer; allocates and frees TMEM
// Warps w and w + 4 k share TMEM lane quarter w mod 4 (rows or features
// 32 (w mod 4) .. + 31).
// Per chunk i (Q, K buffer b = i mod 2; one V buffer):
//   (1) A           = phi(Q) phi(K)^T                 M=128, N=128, K=128 (features)
//   (4) [num | den] = P [V | 1]                        M=128, N=144, K=128 (keys)
//   (3) [num | den] += phi(Q) [S | z_hi | z_lo]        M=128, N=144, K=128 (features)
//   (2) [S | z]    += phi(K)^T [V | 1]                 M=128, N=144, K=128 (tokens)
// issued in that order; (2) after (3), so the operand (3) reads is rewritten
// only once (2) has completed.
constexpr int kMaskW0 = 0, kOutW0 = 4, kStateW0 = 8, kPhiW0 = 12, kProdW = 20, kMmaW = 21;
constexpr int kThreads = 32 * (kMmaW + 1);
constexpr int kBarPhi = 1, kBarMask = 2, kBarOut = 3, kBarState = 4;
constexpr uint32_t kBuf = 2 * kTileBytes;                 // one 128 x 128 bf16 tile (two boxes)
// Shared memory (offsets from a 1024-aligned base): Q buffers, K buffers, V,
// the ones atom right after V (so [V | 1] is three atoms 16 KB apart), then the
// state operand: three 16 KB planes [128 feature rows x 64 values] (values
// 0-63, 64-127, then z_hi, z_lo and zeros), MN-major with the same stride.
constexpr uint32_t kOffQ = 0, kOffK = 2 * kBuf, kOffV = 4 * kBuf;
constexpr uint32_t kOffOnes = kOffV + kBuf, kOffS = kOffOnes + kTileBytes;
constexpr uint32_t kSmemEnd = kOffS + 3 * kTileBytes;
constexpr size_t kSmem = 1024 + kSmemEnd;
// TMEM columns: A at 0 (P over its first 64 columns), [num | den] at 128
// (num 0-127, den parts at 128 and 129), the running state at 288 (S 0-127,
// z at 128).
constexpr uint32_t kTmA = 0, kTmND = 128, kTmS = 288;
constexpr uint32_t kNb = 144;                             // N of (2), (3), (4)

struct Bars {
    uint64_t qk_full[2], k_free[2], q_free[2], phi_done[2];
    uint64_t v_full, v_free, a_full, p_ready, pv_done, o_done, out_read, st_full, snap, drain;
    uint32_t tmem_slot;
};

// 32 consecutive fp32 values -> 16 packed bf16 pairs.
__device__ __forceinline__ void pack32(const float (&f)[32], uint32_t (&p)[16]) {
#pragma unroll
    for (int e = 0; e < 16; ++e) p[e] = pack_bf16(f[2 * e], f[2 * e + 1]);
}

// Row r (a feature) of one 64-column plane of an MN-major operand: 16-byte
// chunks c0 .. c0 + 3 from p.
__device__ __forceinline__ void put_plane_row(uint8_t* plane, int r, int c0, const uint32_t (&p)[16]) {
#pragma unroll
    for (int c = 0; c < 4; ++c)
        *reinterpret_cast<uint4*>(plane + r * 128 + (((c0 + c) ^ (r & 7)) << 4)) =
            make_uint4(p[4 * c], p[4 * c + 1], p[4 * c + 2], p[4 * c + 3]);
}

template <bool kInit, int kPhi>
__global__ void __launch_bounds__(kThreads, 1)
c128_out_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                const __grid_constant__ CUtensorMap vmap, const __grid_constant__ CUtensorMap omap,
                const float* __restrict__ agg, const float* __restrict__ seeds,
                const float* __restrict__ S0,
                const float* __restrict__ z0, float* __restrict__ S_out, float* __restrict__ z_out,
                Partition part, int N, float eps, WsHeader* hdr) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    __shared__ Bars m;
    pdl_launch_dependents();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cta = blockIdx.x;
    const int nchunks = part.nchunks;
    const int64_t u0 = part.begin(cta), u1 = part.begin(cta + 1);
    const int nch = (int)(u1 - u0);
    auto qbuf = [&](int b) { return base + kOffQ + b * kBuf; };
    auto kbuf = [&](int b) { return base + kOffK + b * kBuf; };
    uint8_t* vb = base + kOffV;
    uint8_t* sop = base + kOffS;

    if (tid == 0) {
        for (int b = 0; b < 2; ++b) {
            mbar_init(&m.qk_full[b], 1);
            mbar_init(&m.k_free[b], 1);
            mbar_init(&m.q_free[b], 1);
            mbar_init(&m.phi_done[b], 1);
        }
        mbar_init(&m.v_full, 1);
        mbar_init(&m.v_free, 1);
        mbar_init(&m.a_full, 1);
        mbar_init(&m.p_ready, 1);
        mbar_init(&m.pv_done, 1);
        mbar_init(&m.o_done, 1);
        mbar_init(&m.out_read, 1);
        mbar_init(&m.st_full, 1);
        mbar_init(&m.snap, 1);
        mbar_init(&m.drain, 1);
        fence_mbar_init();
    }
    if (warp >= kPhiW0 && warp < kProdW) init_ones_tile(base + kOffOnes, tid - 32 * kPhiW0, 256);
    // z plane: chunk 1 of every row (values 8-15 of the z atom) stays zero.
    if (warp >= kMaskW0 && warp < kStateW0) {
        const int r = tid - 32 * kMaskW0;    // 0..255 -> rows 0..127, twice
        if (r < 128)
            *reinterpret_cast<uint4*>(sop + 2 * kTileBytes + r * 128 + ((1 ^ (r & 7)) << 4)) =
                make_uint4(0, 0, 0, 0);
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
    const uint32_t max_spin = hdr->max_spin;
    const bool hold = hdr->hold_item != 0;
    const uint32_t tmem = m.tmem_slot;
    const int q4 = warp & 3;
    const uint32_t lane_base = (uint32_t)(32 * q4) << 16;

    if (warp == kProdW) {
        // ---------------------------------------------------------- producer
        // Q, K of chunk i into buffer i mod 2 once (2) of chunk i - 2 released K
        // and the output of chunk i - 2 left the Q buffer (its staging); V once
        // (2) of chunk i - 1 completed. The inputs depend on no earlier launch.
        if (lane == 0) {
            bool ok = true;
            int i = 0, nv = 0;
            for (; i < nch && ok && !hold; ++i) {   // hold: test hook, loads never issued
                const int b = i & 1;
                const int64_t u = u0 + i;
                const int h = (int)(u / nchunks), ch = (int)(u % nchunks);
                if (i >= 2 && (!mbar_wait(&m.k_free[b], ((i >> 1) - 1) & 1, max_spin) ||
                               !mbar_wait(&m.q_free[b], ((i >> 1) - 1) & 1, max_spin))) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&m.qk_full[b], 2 * kBuf);
                for (int bx = 0; bx < 2; ++bx) {
                    tma_load_3d(qbuf(b) + bx * kTileBytes, &qmap, &m.qk_full[b], 64 * bx, ch * kC, h);
                    tma_load_3d(kbuf(b) + bx * kTileBytes, &kmap, &m.qk_full[b], 64 * bx, ch * kC, h);
                }
                if (i >= 1 && !mbar_wait(&m.v_free, (i - 1) & 1, max_spin)) {
                    ok = false;
                    ++i;
                    break;
                }
                mbar_arrive_expect_tx(&m.v_full, kBuf);
                for (int bx = 0; bx < 2; ++bx)
                    tma_load_3d(vb + bx * kTileBytes, &vmap, &m.v_full, 64 * bx, ch * kC, h);
                nv = i + 1;
            }
            if (!ok) report_timeout(hdr);
            // Every issued load lands before the CTA exits.
            for (int j = i - 2 > 0 ? i - 2 : 0; j < i; ++j)
                mbar_wait(&m.qk_full[j & 1], (j >> 1) & 1, kDefaultMaxSpin);
            if (nv > 0) mbar_wait(&m.v_full, (nv - 1) & 1, kDefaultMaxSpin);
        }
    } else if (warp == kMmaW) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t id_qk = idesc_bf16_f32(128, 128, false, false);
            const uint32_t id_pv = idesc_bf16_f32(128, kNb, false, true);
            const uint32_t id_qs = idesc_bf16_f32(128, kNb, false, true);
            const uint32_t id_st = idesc_bf16_f32(128, kNb, true, true);
            const uint32_t va = smem_u32(vb), sa = smem_u32(sop);
            bool ok = true;
            for (int i = 0; i < nch && ok; ++i) {
                const int b = i & 1;
                const uint32_t qa = smem_u32(qbuf(b)), ka = smem_u32(kbuf(b));
                // (1) overwrites the columns (4) of chunk i - 1 read P from.
                if (!mbar_wait(&m.phi_done[b], (i >> 1) & 1, max_spin) ||
                    (i >= 1 && !mbar_wait(&m.pv_done, (i - 1) & 1, max_spin))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int k16 = 0; k16 < 8; ++k16) {
                    const uint32_t off = (k16 >> 2) * kTileBytes + (k16 & 3) * 32;
                    mma_bf16(tmem + kTmA, smem_desc(qa + off, 16, 1024, kSwizzle128B),
                             smem_desc(ka + off, 16, 1024, kSwizzle128B), id_qk, k16 > 0);
                }
                mma_commit(&m.a_full);
                // (4) once P is written, V has landed and the output warps have read
                // [num | den] of chunk i - 1.
                if (!mbar_wait(&m.p_ready, i & 1, max_spin) || !mbar_wait(&m.v_full, i & 1, max_spin) ||
                    (i >= 1 && !mbar_wait(&m.out_read, (i - 1) & 1, max_spin))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int k16 = 0; k16 < 8; ++k16)
                    mma_bf16_ts(tmem + kTmND, tmem + kTmA + 8 * k16,
                                smem_desc(va + k16 * 2048, kTileBytes, 1024, kSwizzle128B), id_pv,
                                k16 > 0);
                mma_commit(&m.pv_done);
                // (3) and (2) once the state operand (and the TMEM state) of chunk i is ready.
                if (!mbar_wait(&m.snap, i & 1, max_spin)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int k16 = 0; k16 < 8; ++k16) {
                    const uint32_t off = (k16 >> 2) * kTileBytes + (k16 & 3) * 32;
                    mma_bf16(tmem + kTmND, smem_desc(qa + off, 16, 1024, kSwizzle128B),
                             smem_desc(sa + k16 * 2048, kTileBytes, 1024, kSwizzle128B), id_qs, 1u);
                }
                mma_commit(&m.o_done);
#pragma unroll
                for (int k16 = 0; k16 < 8; ++k16)
                    mma_bf16(tmem + kTmS, smem_desc(ka + k16 * 2048, kTileBytes, 1024, kSwizzle128B),
                             smem_desc(va + k16 * 2048, kTileBytes, 1024, kSwizzle128B), id_st, 1u);
                mma_commit(&m.st_full);
                mma_commit(&m.k_free[b]);
                mma_commit(&m.v_free);
            }
            if (!ok) report_timeout(hdr);
            mma_commit(&m.drain);  // every issued MMA completes before TMEM is released
            mbar_wait(&m.drain, 0, kDefaultMaxSpin);
        }
    } else if (warp >= kPhiW0) {
        // ---------------------------------------------------------- phi
        const int t = tid - 32 * kPhiW0;     // 0..255
        bool ok = true;
        for (int i = 0; i < nch; ++i) {
            const int b = i & 1;
            const int ch = (int)((u0 + i) % nchunks);
            const int valid = min(kC, N - ch * kC);
            if (ok) ok = mbar_wait(&m.qk_full[b], (i >> 1) & 1, max_spin);
            if (ok) {
                phi_tiles2_256<kPhi>(kbuf(b), valid, qbuf(b), kC, t);
                phi_tiles2_256<kPhi>(kbuf(b) + kTileBytes, valid, qbuf(b) + kTileBytes, kC, t);
            }
            fence_proxy_async_smem();
            ok = named_bar_and(kBarPhi, 256, ok);
            if (!ok) break;
            if (t == 0) mbar_arrive(&m.phi_done[b]);
        }
        if (!ok && t == 0) report_timeout(hdr);
    } else if (warp < kOutW0) {
        // ---------------------------------------------------------- mask
        // Block j (keys 32 j .. 32 j + 31) of A -> 16 packed P columns at 16 j; in
        // increasing j every A column is read before the P columns over it are
        // written. Blocks past the diagonal block q4 are zero for this quarter.
        const int t = tid - 32 * kMaskW0;
        const uint32_t ta = tmem + kTmA + lane_base;
        bool ok = true;
        for (int i = 0; i < nch; ++i) {
            if (ok) ok = mbar_wait(&m.a_full, i & 1, max_spin);
            tc_fence_after();
            for (int j = 0; ok && j <= q4; ++j) {
                uint32_t r0[16], r1[16];
                tmem_ld16(ta + 32 * j, r0);
                tmem_ld16(ta + 32 * j + 16, r1);
                tmem_ld_wait();
                // Diagonal block: key 32 q4 + e <= row 32 q4 + lane.
                uint32_t p[16];
                if (j < q4) pack_block32(r0, r1, p);
                else pack_block32_diag(r0, r1, lane, p);
                tmem_st16(ta + 16 * j, p);
            }
            for (int j = q4 + 1; ok && j < 4; ++j) {
                uint32_t p[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) p[e] = 0u;
                tmem_st16(ta + 16 * j, p);
            }
            tmem_st_wait();
            tc_fence_before();
            ok = named_bar_and(kBarMask, 128, ok);
            if (!ok) break;
            if (t == 0) mbar_arrive(&m.p_ready);
        }
        if (!ok && t == 0) report_timeout(hdr);
    } else if (warp < kStateW0) {
        // ---------------------------------------------------------- output
        // Thread = query row v of its lane quarter; o goes to the chunk's Q buffer
        // (free once (3) completed) in the TMA tile layout, then one store per box.
        const int t = tid - 32 * kOutW0;
        const int v = 32 * q4 + lane;
        const uint32_t tn = tmem + kTmND + lane_base;
        bool ok = true;
        for (int i = 0; i < nch; ++i) {
            const int b = i & 1;
            const int64_t u = u0 + i;
            const int h = (int)(u / nchunks), ch = (int)(u % nchunks);
            if (ok) ok = mbar_wait(&m.o_done, i & 1, max_spin);
            tc_fence_after();
            if (ok) {
                uint32_t rd[2];
                tmem_ld2(tn + 128, rd);
                tmem_ld_wait();
                const float inv = 1.f / (__uint_as_float(rd[0]) + __uint_as_float(rd[1]) + eps);
                uint8_t* ob = qbuf(b);
#pragma unroll 1
                for (int pc = 0; pc < 4; ++pc) {          // 32 values per piece
                    uint32_t r0[16], r1[16];
                    tmem_ld16(tn + 32 * pc, r0);
                    tmem_ld16(tn + 32 * pc + 16, r1);
                    tmem_ld_wait();
                    uint32_t p[16];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        p[e] = pack_bf16(__uint_as_float(r0[2 * e]) * inv, __uint_as_float(r0[2 * e + 1]) * inv);
                        p[8 + e] = pack_bf16(__uint_as_float(r1[2 * e]) * inv, __uint_as_float(r1[2 * e + 1]) * inv);
                    }
                    put_plane_row(ob + (pc >> 1) * kTileBytes, v, 4 * (pc & 1), p);
                }
            }
            tc_fence_before();
            fence_proxy_async_smem();
            ok = named_bar_and(kBarOut, 128, ok);
            if (!ok) break;
            if (t == 0) {
                mbar_arrive(&m.out_read);               // (4) of chunk i + 1 may overwrite
                tma_store_3d(&omap, qbuf(b), 0, ch * kC, h);
                tma_store_3d(&omap, qbuf(b) + kTileBytes, 64, ch * kC, h);
                tma_store_commit();
                tma_store_wait_read<0>();
                mbar_arrive(&m.q_free[b]);              // Q of chunk i + 2 may load
            }
        }
        if (t == 0) {
            if (!ok) report_timeout(hdr);
            tma_store_wait_all<0>();
        }
    } else {
        // ---------------------------------------------------------- state
        // Thread = feature row f of its lane quarter: TMEM lane f of the running
        // state, row f of the shared-memory operand.
        const int t = tid - 32 * kStateW0;
        const int f = 32 * q4 + lane;
        const uint32_t ts = tmem + kTmS + lane_base;
        // Writes state row f to TMEM and the operand: values row[0..127] (zero when
        // row is null) plus adds[w][0..127] for w < nadd, and z. Rows are read as
        // 16-byte pieces, eight in flight per 32 values.
        auto write_row = [&](const float* row, const float* const* adds, int nadd, float z) {
#pragma unroll 1
            for (int pc = 0; pc < 4; ++pc) {
                float x[32];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const float4 a = row ? reinterpret_cast<const float4*>(row + 32 * pc)[q]
                                         : make_float4(0.f, 0.f, 0.f, 0.f);
                    x[4 * q] = a.x; x[4 * q + 1] = a.y; x[4 * q + 2] = a.z; x[4 * q + 3] = a.w;
                }
                for (int w = 0; w < nadd; ++w) {
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const float4 a = reinterpret_cast<const float4*>(adds[w] + 32 * pc)[q];
                        x[4 * q] += a.x; x[4 * q + 1] += a.y; x[4 * q + 2] += a.z; x[4 * q + 3] += a.w;
                    }
                }
                uint32_t w[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) w[e] = __float_as_uint(x[e]);
                tmem_st16(ts + 32 * pc, w);
#pragma unroll
                for (int e = 0; e < 16; ++e) w[e] = __float_as_uint(x[16 + e]);
                tmem_st16(ts + 32 * pc + 16, w);
                uint32_t p[16];
                pack32(x, p);
                put_plane_row(sop + (pc >> 1) * kTileBytes, f, 4 * (pc & 1), p);
            }
            uint32_t w[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) w[e] = 0u;
            w[0] = __float_as_uint(z);
            tmem_st16(ts + 128, w);
            const float zh = __bfloat162float(__float2bfloat16_rn(z));
            *reinterpret_cast<uint4*>(sop + 2 * kTileBytes + f * 128 + ((0 ^ (f & 7)) << 4)) =
                make_uint4(pack_bf16(zh, z - zh), 0, 0, 0);
        };
        // The seed comes from the scan launch, or (seeds == nullptr) from the run
        // sums of the at most kWalkMax ranges to the left that hold this range's
        // first head, added to that head's initial state.
        pdl_wait();
        bool ok = true;
        if (seeds) {
            const float* sd = seeds + (int64_t)cta * kE;
            write_row(sd + f * kD, nullptr, 0, sd[kD * kD + f]);
        } else {
            const int64_t h0 = u0 / nchunks, hb = h0 * nchunks;
            const float* wp[kWalkMax];
            int nw = 0;
            if (u0 != hb) {
                for (int c2 = cta - 1; c2 >= 0 && nw < kWalkMax; --c2) {
                    const int64_t a0 = part.begin(c2);
                    wp[nw++] = agg + (int64_t)c2 * kE;   // its last run: this range's first head
                    if (a0 <= hb) break;
                }
            }
            float z = kInit ? z0[h0 * kD + f] : 0.f;
            for (int w = 0; w < nw; ++w) z += wp[w][kD * kD + f];
            const float* rows[kWalkMax];
            for (int w = 0; w < nw; ++w) rows[w] = wp[w] + f * kD;
            write_row(kInit ? S0 + h0 * kD * kD + (int64_t)f * kD : nullptr, rows, nw, z);
        }
        tmem_st_wait();
        fence_proxy_async_smem();
        tc_fence_before();
        ok = named_bar_and(kBarState, 128, ok);
        if (ok && t == 0) mbar_arrive(&m.snap);
        for (int i = 0; i < nch && ok; ++i) {
            const int64_t u = u0 + i;
            const int64_t h = u / nchunks;
            const bool head_last = (u % nchunks) == nchunks - 1;
            const bool next = i + 1 < nch;
            ok = mbar_wait(&m.st_full, i & 1, max_spin);
            tc_fence_after();
            if (ok && (head_last || next)) {
                if (head_last) {
                    // Final head state (fp32), then the next head's initial state.
#pragma unroll 1
                    for (int pc = 0; pc < 5; ++pc) {
                        uint32_t r0[16], r1[16];
                        tmem_ld16(ts + 32 * pc, r0);
                        tmem_ld16(ts + 32 * pc + 16, r1);
                        tmem_ld_wait();
                        if (pc < 4) {
                            if (S_out) {
                                float4* dst = reinterpret_cast<float4*>(S_out + (h * kD + f) * kD + 32 * pc);
#pragma unroll
                                for (int qd = 0; qd < 4; ++qd) {
                                    dst[qd] = make_float4(__uint_as_float(r0[4 * qd]), __uint_as_float(r0[4 * qd + 1]),
                                                          __uint_as_float(r0[4 * qd + 2]), __uint_as_float(r0[4 * qd + 3]));
                                    dst[4 + qd] = make_float4(__uint_as_float(r1[4 * qd]), __uint_as_float(r1[4 * qd + 1]),
                                                              __uint_as_float(r1[4 * qd + 2]), __uint_as_float(r1[4 * qd + 3]));
                                }
                            }
                        } else if (z_out) {
                            z_out[h * kD + f] = __uint_as_float(r0[0]);
                        }
                    }
                    if (next) {
                        if constexpr (kInit)
                            write_row(S0 + (h + 1) * kD * kD + (int64_t)f * kD, nullptr, 0, z0[(h + 1) * kD + f]);
                        else
                            write_row(nullptr, nullptr, 0, 0.f);
                        tmem_st_wait();
                    }
                } else {
                    // The TMEM state stays; its bf16 copy becomes the next operand.
#pragma unroll 1
                    for (int pc = 0; pc < 4; ++pc) {
                        uint32_t r0[16], r1[16];
                        tmem_ld16(ts + 32 * pc, r0);
                        tmem_ld16(ts + 32 * pc + 16, r1);
                        tmem_ld_wait();
                        uint32_t p[16];
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            p[e] = pack_bf16(__uint_as_float(r0[2 * e]), __uint_as_float(r0[2 * e + 1]));
                            p[8 + e] = pack_bf16(__uint_as_float(r1[2 * e]), __uint_as_float(r1[2 * e + 1]));
                        }
                        put_plane_row(sop + (pc >> 1) * kTileBytes, f, 4 * (pc & 1), p);
                    }
                    uint32_t rz[2];
                    tmem_ld2(ts + 128, rz);
                    tmem_ld_wait();
                    const float z = __uint_as_float(rz[0]);
                    const float zh = __bfloat162float(__float2bfloat16_rn(z));
                    *reinterpret_cast<uint4*>(sop + 2 * kTileBytes + f * 128 + ((0 ^ (f & 7)) << 4)) =
                        make_uint4(pack_bf16(zh, z - zh), 0, 0, 0);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            ok = named_bar_and(kBarState, 128, ok);
            if (ok && next && t == 0) mbar_arrive(&m.snap);
        }
        if (!ok && t == 0) report_timeout(hdr);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaW) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

static_assert(kSmem <= 232448, "shared memory exceeds 227 KB");

}  // namespace

int tc_causal128_launches(int64_t BH, int N) {
    Partition p = make_partition(BH, N, sm_count());
    int walk = 0;
    for (int c = 0; c < p.grid && walk <= kWalkMax; ++c) walk = max(walk, left_walk(p, c));
    return walk <= kWalkMax ? 2 : 3;
}

// Workspace after the header: one last-run sum and one seed per CTA.
size_t tc_causal128_workspace(int64_t BH, int N) {
    Partition p = make_partition(BH, N, sm_count());
    return sizeof(float) * (size_t)p.grid * 2 * (size_t)kE;
}

cudaError_t tc_causal128(const void* q, const void* k, const void* v, void* o, int64_t BH, int N,
                         float eps, int fm, const float* S0, const float* z0, float* S_out,
                         float* z_out, void* ws_header, void* scratch, cudaStream_t st) {
    Partition p = make_partition(BH, N, sm_count());
    if (p.grid > kSeedMaxGrid) return cudaErrorInvalidConfiguration;
    WsHeader* hdr = reinterpret_cast<WsHeader*>(ws_header);
    float* agg = reinterpret_cast<float*>(scratch);
    float* seeds = agg + (size_t)p.grid * kE;
    int walk = 0;
    for (int c = 0; c < p.grid && walk <= kWalkMax; ++c) walk = max(walk, left_walk(p, c));
    if (walk <= kWalkMax) seeds = nullptr;     // each range sums its own seed
    CUtensorMap qm, km, vm, om;
    if (!encode_bhnd(&qm, q, BH, N, kD) || !encode_bhnd(&km, k, BH, N, kD) ||
        !encode_bhnd(&vm, v, BH, N, kD) || !encode_bhnd(&om, o, BH, N, kD))
        return cudaErrorInvalidValue;
    cudaError_t err;
    if ((err = tc_run_sums128(k, v, agg, BH, N, fm, true, ws_header, st))) return err;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((kE + 31) / 32);
    cfg.blockDim = dim3(32 * kSeedWarps);
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (seeds && (err = cudaLaunchKernelEx(&cfg, c128_seed_kernel, (const float*)agg, seeds, p, S0, z0)))
        return err;
    using Kernel = decltype(&c128_out_kernel<false, kPhiElu1>);
    static std::atomic<int> optin[4][kMaxDevices];
    const Kernel kernels[4] = {c128_out_kernel<false, kPhiElu1>, c128_out_kernel<true, kPhiElu1>,
                               c128_out_kernel<false, kPhiIdentity>, c128_out_kernel<true, kPhiIdentity>};
    const int variant = (S0 ? 1 : 0) + (fm == kPhiIdentity ? 2 : 0);
    if ((err = ensure_smem_optin(kernels[variant], (int)kSmem, optin[variant]))) return err;
    cfg.gridDim = dim3(p.grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmem;
    return cudaLaunchKernelEx(&cfg, kernels[variant], qm, km, vm, om, (const float*)agg,
                              (const float*)seeds, S0, z0, S_out, z_out, p, N, eps, hdr);
}

}  // namespace la
