// Tensor-core (tcgen05) backward for bf16 inputs, Dk = Dv = 64: dq, dk, dv of
// o_i = phi(q_i)^T S_i / (phi(q_i)^T z_i + eps) from dout, without storing any
// S_i ("Transformers Are RNNs: Linear Attention", "Turn Causal Attention into a
// Recurrence": the gradients are again prefix sums, forward for dq and reverse
// for dk, dv, so training stays linear in N).
//
// Per row i (g = dout_i): num_i = phi(q_i)^T S_i, den_i = phi(q_i)^T z_i + eps,
// dnum_i = g / den_i, dd_i = -(g . o_i) / den_i. Then, per chunk of 128 tokens,
// with (S_prev, z_prev) the forward state before the chunk and (R_next, r_next)
// the reverse sums of phi(q) [dnum | dd]^T over the chunks after it:
//   dphi(q_i) = S_prev dnum_i + dd_i z_prev + sum_{j<=i in chunk} G_ij phi(k_j)
//   dphi(k_j) = R_next v_j + r_next + sum_{i>=j in chunk} G_ij phi(q_i)
//   dv_j      = R_next^T phi(k_j) + sum_{i>=j in chunk} W_ij dnum_i
// with G_ij = v_j . dnum_i + dd_i and W_ij = phi(q_i) . phi(k_j) (j <= i), and
// dq = dphi(q) phi'(q), dk = dphi(k) phi'(k). Non-causal: the whole sequence's
// (S, z) and (R, r), no in-chunk terms.
//
// Launches: bwd_state_tc_kernel, one CTA per 128-token chunk, computes the
// chunk's forward state [S^T ; z] = [V | 1]^T phi(K) on the tensor core;
// simt.cu's scan turns the chunk states into exclusive prefixes (causal) or the
// total (non-causal); bwd_rows_tc_kernel, one CTA per chunk, does
//   (1) A = phi(Q) phi(K)^T -> causal mask -> bf16 P (TMEM),
//   (2) [num | den] = P [V | 1] + phi(Q) [S_prev^T | z_hi | z_lo]^T,
//   epilogue: dnum, dd (to shared memory and global),
//   (3) [dR^T ; dr] = [dnum | dd]^T phi(Q)  (the chunk's reverse-sum term);
// simt.cu's reverse scan sums (3) over later chunks; bwd_grad_tc_kernel, one
// CTA per chunk and two CTAs per SM, forms W and then G (bf16, one shared
// buffer) and the three gradients as tcgen05 products with fp32 accumulators
// in TMEM (256 columns). Operands are 128 x 64 bf16
// tiles with the 128-byte swizzle; a tile of rows r and columns c serves as a
// K-major operand (K = c) or an MN-major one (K = r), so no transposes are
// written.
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_common.cuh"
#include "tc_util.cuh"

namespace la {

namespace {

using namespace tc;
using namespace tcc;

constexpr int kD = 64;
constexpr int kE = kD * kD + kD;
constexpr int kBThreads = 256;
constexpr uint32_t kSRows = kD * 128 + 16 * 128;            // [S^T | z_hi | z_lo | 0]: 80 rows

// ------------------------------------------------------------ state kernel
// [S^T ; z] = [V | 1]^T phi(K) of one chunk (M = 128: values, a ones row that
// yields z, zeros; N = 64 features; K = the chunk's rows), written as fp32
// S [d][m] and z [d] into the chunk's slot.
constexpr uint32_t kSK = 0, kSV = kTileBytes, kSOnesOff = 2 * kTileBytes;
constexpr size_t kStateSmem = 1024 + 3 * kTileBytes;

template <int kPhi>
__global__ void __launch_bounds__(kBThreads)
bwd_state_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                    float* __restrict__ states, int N, WsHeader* hdr) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    __shared__ uint64_t ld, mma;
    __shared__ uint32_t tmem_slot;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = blockIdx.x, nch = gridDim.x;
    const int64_t bh = blockIdx.y;
    const int t0 = c * kC;
    const int valid = min(kC, N - t0);
    uint8_t *tK = base + kSK, *tV = base + kSV, *tOnes = base + kSOnesOff;
    if (tid == 0) {
        mbar_init(&ld, 1);
        mbar_init(&mma, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&tmem_slot, 64);
        tmem_relinquish();
    }
    init_ones_tile(tOnes, tid, kBThreads);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    const uint32_t max_spin = hdr->max_spin;
    const bool hold = hdr->hold_item != 0;
    if (tid == 0 && !hold) {
        mbar_arrive_expect_tx(&ld, 2 * kTileBytes);
        tma_load_3d(tK, &kmap, &ld, 0, t0, (int)bh);
        tma_load_3d(tV, &vmap, &ld, 0, t0, (int)bh);
    }
    bool ok = hold ? false : mbar_wait(&ld, 0, max_spin);
    if (ok) phi_tile_256<kPhi>(tK, tid, valid);
    fence_proxy_async_smem();
    tc_fence_before();
    ok = __syncthreads_and(ok);
    tc_fence_after();
    if (tid == 0 && ok) {
        const uint32_t ka = smem_u32(tK), va = smem_u32(tV);
        const uint32_t id = idesc_bf16_f32(128, 64, true, true);
#pragma unroll
        for (int k16 = 0; k16 < kC / 16; ++k16)
            mma_bf16(tmem, smem_desc(va + k16 * 2048, smem_u32(tOnes) - va, 1024, kSwizzle128B),
                     smem_desc(ka + k16 * 2048, 1024, 1024, kSwizzle128B), id, k16 > 0);
        mma_commit(&mma);
    }
    if (ok) ok = mbar_wait(&mma, 0, max_spin);
    ok = __syncthreads_and(ok);
    tc_fence_after();
    const int q4 = warp & 3, hh = warp >> 2;
    if (q4 < 3) {
        // Lane v < 64: S^T row (value v); lane 64: z. Columns: features 32 hh ...
        uint32_t r[2][16];
        const uint32_t ta = tmem + ((uint32_t)(32 * q4) << 16) + 32 * hh;
        tmem_ld16(ta, r[0]);
        tmem_ld16(ta + 16, r[1]);
        tmem_ld_wait();
        float* out = states + ((int64_t)bh * nch + c) * kE;
        const int v = 32 * q4 + lane;
#pragma unroll
        for (int e = 0; e < 32; ++e) {
            const int d = 32 * hh + e;
            const float x = __uint_as_float(r[e >> 4][e & 15]);
            if (v < kD) out[d * kD + v] = x;
            else if (v == kD) out[kD * kD + d] = x;
        }
    }
    if (!ok && tid == 0) report_timeout(hdr);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 64);
    }
}

// ------------------------------------------------------------ rows kernel
// Shared memory: Q, K (later dnum), V (later the dd tile), ones, dout, S rows.
constexpr uint32_t kRQ = 0, kRK = kTileBytes, kRV = 2 * kTileBytes, kROnes = 3 * kTileBytes;
constexpr uint32_t kRG = 4 * kTileBytes, kRS = 5 * kTileBytes;
constexpr size_t kRowsSmem = 1024 + kRS + kSRows;
constexpr uint32_t kTmNumR = 64;                            // [num | den] at columns 64..143

struct BwdMisc {
    uint64_t ld, mma;
    uint32_t tmem_slot;
    float red[2][kC];
};

// Rows r of the state block src ([kD][kD] fp32, row-major) as bf16 rows of a
// swizzled tile: dst row r, columns 16 p .. 16 p + 15 from src[r][16 p + e]
// (transposed: from src[16 p + e][r]). 256 threads cover 64 rows x 4 pieces.
__device__ __forceinline__ void state_rows_to_tile(uint8_t* dst, const float* src, bool transposed,
                                                   int t) {
    const int r = t & 63, p = t >> 6;
    float f[16];
    if (transposed) {
#pragma unroll
        for (int e = 0; e < 16; ++e) f[e] = src[(16 * p + e) * kD + r];
    } else {
        // 16 consecutive floats: four 16-byte loads (the block is 16-byte aligned).
#pragma unroll
        for (int e4 = 0; e4 < 4; ++e4) {
            const float4 x = reinterpret_cast<const float4*>(src + r * kD + 16 * p)[e4];
            f[4 * e4] = x.x;
            f[4 * e4 + 1] = x.y;
            f[4 * e4 + 2] = x.z;
            f[4 * e4 + 3] = x.w;
        }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h)
        *reinterpret_cast<uint4*>(dst + sw128_offset(r, 16 * p + 8 * h)) =
            make_uint4(pack_bf16(f[8 * h], f[8 * h + 1]), pack_bf16(f[8 * h + 2], f[8 * h + 3]),
                       pack_bf16(f[8 * h + 4], f[8 * h + 5]), pack_bf16(f[8 * h + 6], f[8 * h + 7]));
}

template <bool kCausal, int kPhi>
__global__ void __launch_bounds__(kBThreads, 2)
bwd_rows_tc_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap, const __grid_constant__ CUtensorMap gmap,
                   const float* __restrict__ states, float* __restrict__ rstates,
                   __nv_bfloat16* __restrict__ dnum_out, float* __restrict__ dd_out, int N,
                   float eps, WsHeader* hdr) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    __shared__ BwdMisc m;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = blockIdx.x, nch = gridDim.x;
    const int64_t bh = blockIdx.y;
    const int t0 = c * kC;
    const int valid = min(kC, N - t0);
    uint8_t *tQ = base + kRQ, *tK = base + kRK, *tV = base + kRV, *tOnes = base + kROnes;
    uint8_t *tG = base + kRG, *tS = base + kRS;
    uint8_t* tDn = tK;                            // dnum, once (1) has read phi(K)
    uint8_t* tDd = tV;                            // [dd | 0], once (2) has read V

    if (tid == 0) {
        mbar_init(&m.ld, 1);
        mbar_init(&m.mma, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&m.tmem_slot, 256);
        tmem_relinquish();
    }
    if (kCausal) init_ones_tile(tOnes, tid, kBThreads);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = m.tmem_slot;
    const uint32_t max_spin = hdr->max_spin;
    const bool hold = hdr->hold_item != 0;
    if (tid == 0 && !hold) {
        mbar_arrive_expect_tx(&m.ld, (kCausal ? 4 : 2) * kTileBytes);
        tma_load_3d(tQ, &qmap, &m.ld, 0, t0, (int)bh);
        tma_load_3d(tG, &gmap, &m.ld, 0, t0, (int)bh);
        if (kCausal) {
            tma_load_3d(tK, &kmap, &m.ld, 0, t0, (int)bh);
            tma_load_3d(tV, &vmap, &m.ld, 0, t0, (int)bh);
        }
    }
    // [S_prev^T | z_hi | z_lo | 0]: row n = value index (S^T), K = feature.
    const float* sp = states + ((int64_t)bh * nch + (kCausal ? c : 0)) * kE;
    state_rows_to_tile(tS, sp, true, tid);
    if (tid < 8) {
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float a = sp[kD * kD + 8 * tid + 2 * e], b = sp[kD * kD + 8 * tid + 2 * e + 1];
            hi[e] = pack_bf16(a, b);
            lo[e] = pack_bf16(a - bf_lo(hi[e]), b - __uint_as_float(hi[e] & 0xFFFF0000u));
        }
        *reinterpret_cast<uint4*>(tS + sw128_offset(kD, 8 * tid)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(tS + sw128_offset(kD + 1, 8 * tid)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
    for (int idx = tid; idx < 112; idx += kBThreads)
        *reinterpret_cast<uint4*>(tS + kD * 128 + 256 + idx * 16) = make_uint4(0, 0, 0, 0);
    bool ok = hold ? false : mbar_wait(&m.ld, 0, max_spin);
    if (ok) {
        phi_tile_256<kPhi>(tQ, tid, valid);
        if (kCausal) phi_tile_256<kPhi>(tK, tid, valid);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    ok = __syncthreads_and(ok);
    tc_fence_after();
    const int q4 = warp & 3, hh = warp >> 2;
    const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
    uint32_t ph = 0;
    if (kCausal) {
        if (tid == 0 && ok) {
            const uint32_t id = idesc_bf16_f32(128, 128, false, false);
            const uint32_t qa = smem_u32(tQ), ka = smem_u32(tK);
#pragma unroll
            for (int k16 = 0; k16 < kD / 16; ++k16)
                mma_bf16(tmem, smem_desc(qa + k16 * 32, 16, 1024, kSwizzle128B),
                         smem_desc(ka + k16 * 32, 16, 1024, kSwizzle128B), id, k16 > 0);
            mma_commit(&m.mma);
        }
        if (ok) ok = mbar_wait(&m.mma, ph, max_spin);
        ok = __syncthreads_and(ok);
        ph ^= 1;
        tc_fence_after();
        // Causal mask: A block jb (32 keys) -> P block jb (16 packed columns), warps 0-3.
        if (hh == 0 && ok) {
            const uint32_t tb = tmem + lane_base;
            for (int jb = 0; jb <= q4; ++jb) {
                uint32_t r0[16], r1[16];
                tmem_ld16(tb + 32 * jb, r0);
                tmem_ld16(tb + 32 * jb + 16, r1);
                tmem_ld_wait();
                uint32_t p[16];
                if (jb < q4) pack_block32(r0, r1, p);
                else pack_block32_diag(r0, r1, lane, p);
                tmem_st16(tb + 16 * jb, p);
            }
            for (int jb = q4 + 1; jb < 4; ++jb) {
                uint32_t p[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) p[e] = 0u;
                tmem_st16(tb + 16 * jb, p);
            }
            tmem_st_wait();
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }
    // (2): [num | den] = P [V | 1] (causal) + phi(Q) [S_prev^T | z_hi | z_lo]^T.
    if (tid == 0 && ok) {
        if (kCausal) {
            const uint32_t va = smem_u32(tV);
            const uint32_t id = idesc_bf16_f32(128, 80, false, true);
#pragma unroll
            for (int k16 = 0; k16 < kC / 16; ++k16)
                mma_bf16_ts(tmem + kTmNumR, tmem + 8 * k16,
                            smem_desc(va + k16 * 2048, smem_u32(tOnes) - va, 1024, kSwizzle128B), id,
                            k16 > 0);
        }
        const uint32_t qa = smem_u32(tQ), sa = smem_u32(tS);
        const uint32_t id = idesc_bf16_f32(128, 80, false, false);
#pragma unroll
        for (int k16 = 0; k16 < kD / 16; ++k16)
            mma_bf16(tmem + kTmNumR, smem_desc(qa + k16 * 32, 16, 1024, kSwizzle128B),
                     smem_desc(sa + k16 * 32, 16, 1024, kSwizzle128B), id,
                     (kCausal || k16 > 0) ? 1u : 0u);
        mma_commit(&m.mma);
    }
    if (ok) ok = mbar_wait(&m.mma, ph, max_spin);
    ok = __syncthreads_and(ok);
    ph ^= 1;
    tc_fence_after();
    // Epilogue: row i, value columns 32 hh .. 32 hh + 31. o = num / den, dnum =
    // g / den, dot = g . o (both halves), dd = -dot / den.
    const int i = 32 * q4 + lane;
    const bool live = i < valid;
    float dn[32], inv;
    {
        uint32_t rd[2], r[2][16];
        const uint32_t ta = tmem + lane_base + kTmNumR;
        tmem_ld2(ta + 64, rd);
        tmem_ld16(ta + 32 * hh, r[0]);
        tmem_ld16(ta + 32 * hh + 16, r[1]);
        tmem_ld_wait();
        inv = 1.f / (__uint_as_float(rd[0]) + __uint_as_float(rd[1]) + eps);
        float part = 0.f;
#pragma unroll
        for (int c8 = 0; c8 < 4; ++c8) {
            const uint4 gw = *reinterpret_cast<const uint4*>(tG + sw128_offset(i, 32 * hh + 8 * c8));
            const uint32_t gv[4] = {gw.x, gw.y, gw.z, gw.w};
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float g = (e & 1) ? __uint_as_float(gv[e >> 1] & 0xFFFF0000u) : bf_lo(gv[e >> 1]);
                const int col = 8 * c8 + e;
                const float o = __uint_as_float(r[col >> 4][col & 15]) * inv;
                part = fmaf(g, o, part);
                dn[col] = live ? g * inv : 0.f;
            }
        }
        m.red[hh][i] = part;
    }
    tc_fence_before();
    __syncthreads();
    const float dd = live ? -(m.red[0][i] + m.red[1][i]) * inv : 0.f;
    // dnum (bf16) into the K tile's place and to global; [dd | 0] into V's place.
    __nv_bfloat16* dng = dnum_out + ((int64_t)bh * N + t0 + i) * kD + 32 * hh;
#pragma unroll
    for (int c8 = 0; c8 < 4; ++c8) {
        const uint4 w = make_uint4(pack_bf16(dn[8 * c8], dn[8 * c8 + 1]), pack_bf16(dn[8 * c8 + 2], dn[8 * c8 + 3]),
                                   pack_bf16(dn[8 * c8 + 4], dn[8 * c8 + 5]), pack_bf16(dn[8 * c8 + 6], dn[8 * c8 + 7]));
        *reinterpret_cast<uint4*>(tDn + sw128_offset(i, 32 * hh + 8 * c8)) = w;
        if (live) reinterpret_cast<uint4*>(dng)[c8] = w;
        *reinterpret_cast<uint4*>(tDd + sw128_offset(i, 32 * hh + 8 * c8)) =
            make_uint4((hh == 0 && c8 == 0) ? pack_bf16(dd, 0.f) : 0u, 0, 0, 0);
    }
    if (hh == 0 && live) dd_out[(int64_t)bh * N + t0 + i] = dd;
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // (3): [dR^T ; dr] = [dnum | dd]^T phi(Q): A MN-major (dnum, then the dd tile),
    // B = phi(Q) MN-major; M = 128 (values, dd, zeros), N = 64 features, K = rows.
    if (tid == 0 && ok) {
        const uint32_t da = smem_u32(tDn), qa = smem_u32(tQ);
        const uint32_t id = idesc_bf16_f32(128, 64, true, true);
#pragma unroll
        for (int k16 = 0; k16 < kC / 16; ++k16)
            mma_bf16(tmem, smem_desc(da + k16 * 2048, smem_u32(tDd) - da, 1024, kSwizzle128B),
                     smem_desc(qa + k16 * 2048, 1024, 1024, kSwizzle128B), id, k16 > 0);
        mma_commit(&m.mma);
    }
    if (ok) ok = mbar_wait(&m.mma, ph, max_spin);
    ok = __syncthreads_and(ok);
    tc_fence_after();
    // Lanes 0..63: dR^T rows (value m); lane 64: dr. Columns: features 32 hh ...
    if (q4 < 3) {
        uint32_t r[2][16];
        const uint32_t ta = tmem + lane_base + 32 * hh;
        tmem_ld16(ta, r[0]);
        tmem_ld16(ta + 16, r[1]);
        tmem_ld_wait();
        float* out = rstates + ((int64_t)bh * nch + c) * kE;
        const int v = 32 * q4 + lane;
#pragma unroll
        for (int e = 0; e < 32; ++e) {
            const int d = 32 * hh + e;
            const float x = __uint_as_float(r[e >> 4][e & 15]);
            if (v < kD) out[d * kD + v] = x;
            else if (v == kD) out[kD * kD + d] = x;
        }
    }
    if (!ok && tid == 0) report_timeout(hdr);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 256);
    }
}

// ------------------------------------------------------------ gradient kernel
// Shared memory (dynamic only, so that its base is 1024-aligned without slack):
// Q, K, V, dnum, S_prev [d][m] and R_next [d][m] (64-row tiles); for the causal
// kernel one G/W buffer (two tiles: keys 0..63, 64..127) that holds W, then G;
// then the barriers, the TMEM address and z_prev, r_next.
constexpr uint32_t kGQ = 0, kGK = kTileBytes, kGV = 2 * kTileBytes, kGDn = 3 * kTileBytes;
constexpr uint32_t kGS = 4 * kTileBytes, kGR = kGS + kD * 128, kGB = kGR + kD * 128;
template <bool kCausal> constexpr uint32_t kGMisc = kCausal ? kGB + 2 * kTileBytes : kGB;

struct GradMisc {
    uint64_t ld, mma;
    uint32_t tmem_slot, pad;
    float zp[kD], rn[kD];
};
template <bool kCausal> constexpr size_t kGradSmem = kGMisc<kCausal> + sizeof(GradMisc);

// TMEM columns, 256 allocated in both forms (two CTAs per SM). Causal, in three
// product phases: (a) W at 0..127, dv at 128, dphi(q) at 192; (b) dv += W^T dnum,
// G at 0..127 (W already read out); (c) dphi(k) at 0 (G already read out),
// dphi(q) += G phi(K). Non-causal: dphi(q) 0, dphi(k) 64, dv 128.
template <bool kCausal> constexpr uint32_t kTmDqG = kCausal ? 192 : 0;
template <bool kCausal> constexpr uint32_t kTmDkG = kCausal ? 0 : 64;
constexpr uint32_t kTmDvG = 128, kTmAllocG = 256;

template <bool kCausal, int kPhi>
__global__ void __launch_bounds__(kBThreads, 2)
bwd_grad_tc_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap, const __grid_constant__ CUtensorMap dnmap,
                   const float* __restrict__ states, const float* __restrict__ rstates,
                   const float* __restrict__ dd_in, __nv_bfloat16* __restrict__ dq,
                   __nv_bfloat16* __restrict__ dk, __nv_bfloat16* __restrict__ dv, int N,
                   WsHeader* hdr) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // With no static shared memory the dynamic base is 1024-aligned, which the
    // 128-byte swizzle needs; if it ever is not, report it and touch nothing.
    if (smem_u32(smem_raw) & 1023u) {
        if (threadIdx.x == 0) atomicCAS(&hdr->status, 0u, (uint32_t)LA_ERR_CUDA);
        return;
    }
    uint8_t* base = smem_raw;
    GradMisc& m = *reinterpret_cast<GradMisc*>(base + kGMisc<kCausal>);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = blockIdx.x, nch = gridDim.x;
    const int64_t bh = blockIdx.y;
    const int t0 = c * kC;
    const int valid = min(kC, N - t0);
    uint8_t *tQ = base + kGQ, *tK = base + kGK, *tV = base + kGV, *tDn = base + kGDn;
    uint8_t *tB = base + kGB, *tS = base + kGS, *tR = base + kGR;

    if (tid == 0) {
        mbar_init(&m.ld, 1);
        mbar_init(&m.mma, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&m.tmem_slot, kTmAllocG);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = m.tmem_slot;
    constexpr uint32_t kTmDq = kTmDqG<kCausal>, kTmDk = kTmDkG<kCausal>, kTmDv = kTmDvG;
    const uint32_t max_spin = hdr->max_spin;
    const bool hold = hdr->hold_item != 0;
    if (tid == 0 && !hold) {
        mbar_arrive_expect_tx(&m.ld, 4 * kTileBytes);
        tma_load_3d(tQ, &qmap, &m.ld, 0, t0, (int)bh);
        tma_load_3d(tK, &kmap, &m.ld, 0, t0, (int)bh);
        tma_load_3d(tV, &vmap, &m.ld, 0, t0, (int)bh);
        tma_load_3d(tDn, &dnmap, &m.ld, 0, t0, (int)bh);
    }
    // S_prev and R_next as stored ([d][m]: rows d, columns m), z_prev, r_next.
    const float* sp = states + ((int64_t)bh * nch + (kCausal ? c : 0)) * kE;
    const float* rp = rstates + ((int64_t)bh * nch + (kCausal ? c : 0)) * kE;
    state_rows_to_tile(tS, sp, false, tid);
    state_rows_to_tile(tR, rp, false, tid);
    if (tid < kD) {
        m.zp[tid] = sp[kD * kD + tid];
        m.rn[tid] = rp[kD * kD + tid];
    }
    const int q4 = warp & 3, hh = warp >> 2;
    const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
    const int i = 32 * q4 + lane;                 // this thread's row (query i or key j)
    const bool live_row = i < valid;
    const float ddi = live_row ? dd_in[(int64_t)bh * N + t0 + i] : 0.f;
    bool ok = hold ? false : mbar_wait(&m.ld, 0, max_spin);
    if (ok) {
        phi_tile_256<kPhi>(tQ, tid, valid);
        phi_tile_256<kPhi>(tK, tid, valid);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    ok = __syncthreads_and(ok);
    tc_fence_after();
    uint32_t ph = 0;
    const uint32_t id_kk = idesc_bf16_f32(128, 64, false, false);
    const uint32_t id_km = idesc_bf16_f32(128, 64, false, true);
    const uint32_t id_mm = idesc_bf16_f32(128, 64, true, true);
    const uint32_t qa = smem_u32(tQ), ka = smem_u32(tK), va = smem_u32(tV), dna = smem_u32(tDn);
    const uint32_t sa = smem_u32(tS), ra = smem_u32(tR), ba = smem_u32(tB);
    // dphi(q) = dnum S_prev^T (+ G phi(K)): B = S [d][m] K-major (N = d, K = m).
    auto issue_dq_base = [&]() {
#pragma unroll
        for (int k16 = 0; k16 < kD / 16; ++k16)
            mma_bf16(tmem + kTmDq, smem_desc(dna + k16 * 32, 16, 1024, kSwizzle128B),
                     smem_desc(sa + k16 * 32, 16, 1024, kSwizzle128B), id_kk, k16 > 0);
    };
    // dphi(k) = V R_next^T (+ G^T phi(Q)): B = R [d][m] K-major.
    auto issue_dk_base = [&]() {
#pragma unroll
        for (int k16 = 0; k16 < kD / 16; ++k16)
            mma_bf16(tmem + kTmDk, smem_desc(va + k16 * 32, 16, 1024, kSwizzle128B),
                     smem_desc(ra + k16 * 32, 16, 1024, kSwizzle128B), id_kk, k16 > 0);
    };
    // dv = phi(K) R_next (+ W^T dnum): B = R [d][m] MN-major (K = d rows, N = m).
    auto issue_dv_base = [&]() {
#pragma unroll
        for (int k16 = 0; k16 < kD / 16; ++k16)
            mma_bf16(tmem + kTmDv, smem_desc(ka + k16 * 32, 16, 1024, kSwizzle128B),
                     smem_desc(ra + k16 * 2048, 1024, 1024, kSwizzle128B), id_km, k16 > 0);
    };
    // The MMAs issued so far complete; every thread then sees their results.
    auto wait_mma = [&]() {
        if (ok) ok = mbar_wait(&m.mma, ph, max_spin);
        ok = __syncthreads_and(ok);
        ph ^= 1;
        tc_fence_after();
    };
    if constexpr (kCausal) {
        // Row i, keys 64 hh .. 64 hh + 63 of the 128 x 128 product at TMEM column
        // 0 (+ add for G), kept for j <= i and zero otherwise, bf16 into tile hh of
        // the G/W buffer. Key block kb = 2 hh + h2 against the warp's rows
        // 32 q4 .. 32 q4 + 31 is below the diagonal (kb < q4: every key kept), the
        // diagonal block (kb == q4: key 32 kb + col kept for col <= lane) or above
        // it (zeros, no TMEM read), the same for the whole warp. Rows past a
        // ragged end (i >= valid) are 0.
        auto masked_to_buffer = [&](float add) {
            uint8_t* dst = tB + hh * kTileBytes;
            const uint32_t ta = tmem + lane_base + 64 * hh;
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                const int kb = 2 * hh + h2;
                uint32_t w[16];
                if (kb > q4) {
#pragma unroll
                    for (int e = 0; e < 16; ++e) w[e] = 0u;
                } else {
                    uint32_t r[2][16];
                    tmem_ld16(ta + 32 * h2, r[0]);
                    tmem_ld16(ta + 32 * h2 + 16, r[1]);
                    tmem_ld_wait();
                    if (kb < q4) {
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            w[e] = pack_bf16(__uint_as_float(r[e >> 3][2 * (e & 7)]) + add,
                                             __uint_as_float(r[e >> 3][2 * (e & 7) + 1]) + add);
                    } else {
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            w[e] = pack_bf16(
                                2 * e <= lane ? __uint_as_float(r[e >> 3][2 * (e & 7)]) + add : 0.f,
                                2 * e + 1 <= lane ? __uint_as_float(r[e >> 3][2 * (e & 7) + 1]) + add
                                                  : 0.f);
                    }
                    if (!live_row) {
#pragma unroll
                        for (int e = 0; e < 16; ++e) w[e] = 0u;
                    }
                }
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8)
                    *reinterpret_cast<uint4*>(dst + sw128_offset(i, 32 * h2 + 8 * c8)) =
                        make_uint4(w[4 * c8], w[4 * c8 + 1], w[4 * c8 + 2], w[4 * c8 + 3]);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncthreads();
            tc_fence_after();
        };
        const uint32_t id_sq = idesc_bf16_f32(128, 128, false, false);
        // (a) W = phi(Q) phi(K)^T (128 x 128, K = 64), with the base terms of dv
        // and dphi(q), whose columns are free.
        if (tid == 0 && ok) {
#pragma unroll
            for (int k16 = 0; k16 < kD / 16; ++k16)
                mma_bf16(tmem, smem_desc(qa + k16 * 32, 16, 1024, kSwizzle128B),
                         smem_desc(ka + k16 * 32, 16, 1024, kSwizzle128B), id_sq, k16 > 0);
            issue_dv_base();
            issue_dq_base();
            mma_commit(&m.mma);
        }
        wait_mma();
        if (ok) masked_to_buffer(0.f);
        // (b) dv += W^T dnum (A = W MN-major, B = dnum MN-major), and
        // G = dnum V^T into W's columns.
        if (tid == 0 && ok) {
#pragma unroll
            for (int k16 = 0; k16 < kC / 16; ++k16)
                mma_bf16(tmem + kTmDv, smem_desc(ba + k16 * 2048, kTileBytes, 1024, kSwizzle128B),
                         smem_desc(dna + k16 * 2048, 1024, 1024, kSwizzle128B), id_mm, 1u);
#pragma unroll
            for (int k16 = 0; k16 < kD / 16; ++k16)
                mma_bf16(tmem, smem_desc(dna + k16 * 32, 16, 1024, kSwizzle128B),
                         smem_desc(va + k16 * 32, 16, 1024, kSwizzle128B), id_sq, k16 > 0);
            mma_commit(&m.mma);
        }
        wait_mma();                                   // also: W^T dnum has read the buffer
        if (ok) masked_to_buffer(ddi);
        // (c) dphi(k) = V R_next^T into G's first columns, then + G^T phi(Q);
        // dphi(q) += G phi(K).
        if (tid == 0 && ok) {
            issue_dk_base();
#pragma unroll
            for (int k16 = 0; k16 < kC / 16; ++k16) {
                // + G phi(K): A = G K-major (keys in two tiles), B = phi(K) MN-major.
                mma_bf16(tmem + kTmDq,
                         smem_desc(ba + (k16 >> 2) * kTileBytes + (k16 & 3) * 32, 16, 1024, kSwizzle128B),
                         smem_desc(ka + k16 * 2048, 1024, 1024, kSwizzle128B), id_km, 1u);
                // + G^T phi(Q): A = G MN-major (M = keys, two atoms), B = phi(Q) MN-major.
                mma_bf16(tmem + kTmDk, smem_desc(ba + k16 * 2048, kTileBytes, 1024, kSwizzle128B),
                         smem_desc(qa + k16 * 2048, 1024, 1024, kSwizzle128B), id_mm, 1u);
            }
            mma_commit(&m.mma);
        }
        wait_mma();
    } else {
        if (tid == 0 && ok) {
            issue_dq_base();
            issue_dk_base();
            issue_dv_base();
            mma_commit(&m.mma);
        }
        wait_mma();
    }
    // Epilogue: row i, columns 32 hh .. 32 hh + 31 of each gradient.
    {
        const bool live = live_row && ok;
        const int64_t row = (int64_t)bh * N + t0 + i;
#pragma unroll 1
        for (int which = 0; which < 3; ++which) {
            uint32_t r[2][16];
            const uint32_t ta = tmem + lane_base + (which == 0 ? kTmDq : which == 1 ? kTmDk : kTmDv) + 32 * hh;
            tmem_ld16(ta, r[0]);
            tmem_ld16(ta + 16, r[1]);
            tmem_ld_wait();
            const uint8_t* ft = which == 0 ? tQ : tK;    // phi values for phi'
            __nv_bfloat16* out = (which == 0 ? dq : which == 1 ? dk : dv) + row * kD + 32 * hh;
#pragma unroll
            for (int c8 = 0; c8 < 4; ++c8) {
                uint32_t fw[4] = {0, 0, 0, 0};
                if (which < 2 && kPhi != kPhiIdentity) {
                    const uint4 f4 = *reinterpret_cast<const uint4*>(ft + sw128_offset(i, 32 * hh + 8 * c8));
                    fw[0] = f4.x; fw[1] = f4.y; fw[2] = f4.z; fw[3] = f4.w;
                }
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float x2[2];
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int col = 8 * c8 + 2 * e + u;
                        const int d = 32 * hh + col;
                        float x = __uint_as_float(r[col >> 4][col & 15]);
                        if (which == 0) x = fmaf(ddi, m.zp[d], x);
                        else if (which == 1) x += m.rn[d];
                        if (which < 2 && kPhi != kPhiIdentity) {
                            // phi'(x) = 1 for x > 0, e^x = phi(x) otherwise: min(phi, 1).
                            const float f = u ? __uint_as_float(fw[e] & 0xFFFF0000u) : bf_lo(fw[e]);
                            x *= fminf(f, 1.f);
                        }
                        x2[u] = x;
                    }
                    w[e] = pack_bf16(x2[0], x2[1]);
                }
                if (live) reinterpret_cast<uint4*>(out)[c8] = make_uint4(w[0], w[1], w[2], w[3]);
            }
        }
    }
    if (!ok && tid == 0) report_timeout(hdr);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmAllocG);
    }
}

static_assert(kRowsSmem <= 232448 / 2 - 1024, "two rows CTAs per SM");
// Two gradient CTAs per SM: each takes its dynamic shared memory plus the 1 KB
// the system reserves per CTA, out of the SM's 228 KB.
static_assert(2 * (kGradSmem<true> + 1024) <= 233472, "two causal gradient CTAs per SM");
static_assert(2 * (kGradSmem<false> + 1024) <= 233472, "two non-causal gradient CTAs per SM");

template <bool kCausal, int kPhi>
cudaError_t launch(const CUtensorMap& qm, const CUtensorMap& km, const CUtensorMap& vm,
                   const CUtensorMap& gm, const CUtensorMap& dnm, float* states, float* rstates,
                   __nv_bfloat16* dnum, float* dd, void* dq, void* dk, void* dv, int64_t BH, int N,
                   float eps, WsHeader* hdr, cudaStream_t st) {
    const int nch = (N + kC - 1) / kC;
    static std::atomic<int> optin_s[kMaxDevices], optin_r[kMaxDevices], optin_g[kMaxDevices];
    cudaError_t err;
    if ((err = ensure_smem_optin(bwd_state_tc_kernel<kPhi>, (int)kStateSmem, optin_s)) ||
        (err = ensure_smem_optin(bwd_rows_tc_kernel<kCausal, kPhi>, (int)kRowsSmem, optin_r)) ||
        (err = ensure_smem_optin(bwd_grad_tc_kernel<kCausal, kPhi>, (int)kGradSmem<kCausal>, optin_g)))
        return err;
    const dim3 grid(nch, (unsigned)BH);
    bwd_state_tc_kernel<kPhi><<<grid, kBThreads, kStateSmem, st>>>(km, vm, states, N, hdr);
    if ((err = cudaPeekAtLastError())) return err;
    if ((err = bwd_prefix_states(states, kCausal, BH, nch, kD, kD, st))) return err;
    bwd_rows_tc_kernel<kCausal, kPhi><<<grid, kBThreads, kRowsSmem, st>>>(
        qm, km, vm, gm, states, rstates, dnum, dd, N, eps, hdr);
    if ((err = cudaPeekAtLastError())) return err;
    if ((err = bwd_reverse_sums(rstates, kCausal, BH, nch, kE, st))) return err;
    bwd_grad_tc_kernel<kCausal, kPhi><<<grid, kBThreads, kGradSmem<kCausal>, st>>>(
        qm, km, vm, dnm, states, rstates, dd, (__nv_bfloat16*)dq, (__nv_bfloat16*)dk,
        (__nv_bfloat16*)dv, N, hdr);
    return cudaPeekAtLastError();
}

}  // namespace

bool tc_bwd_supported(int D, int M, la_dtype dt) { return dt == LA_BF16 && D == kD && M == kD; }

cudaError_t tc_bwd(const void* q, const void* k, const void* v, const void* dout, void* dq,
                   void* dk, void* dv, bool causal, int64_t BH, int N, float eps, int fm,
                   void* ws_header, void* scratch, cudaStream_t st) {
    const int nch64 = (N + kChunk - 1) / kChunk;
    // Within the fp32 backward's workspace (sized for 64-token chunks): forward
    // states and reverse sums per 128-token chunk, then dnum (bf16) and dd in
    // place of its row gradients.
    float* states = static_cast<float*>(scratch);
    float* rstates = states + (size_t)BH * nch64 * kE;
    __nv_bfloat16* dnum = reinterpret_cast<__nv_bfloat16*>(rstates + (size_t)BH * nch64 * kE);
    float* dd = reinterpret_cast<float*>(dnum + (size_t)BH * N * kD);
    CUtensorMap qm, km, vm, gm, dnm;
    if (!encode_bhnd(&qm, q, BH, N, kD) || !encode_bhnd(&km, k, BH, N, kD) ||
        !encode_bhnd(&vm, v, BH, N, kD) || !encode_bhnd(&gm, dout, BH, N, kD) ||
        !encode_bhnd(&dnm, dnum, BH, N, kD))
        return cudaErrorInvalidValue;
    WsHeader* hdr = reinterpret_cast<WsHeader*>(ws_header);
    const bool ident = fm == kPhiIdentity;
    if (causal)
        return ident ? launch<true, kPhiIdentity>(qm, km, vm, gm, dnm, states, rstates, dnum, dd, dq,
                                                  dk, dv, BH, N, eps, hdr, st)
                     : launch<true, kPhiElu1>(qm, km, vm, gm, dnm, states, rstates, dnum, dd, dq, dk,
                                              dv, BH, N, eps, hdr, st);
    return ident ? launch<false, kPhiIdentity>(qm, km, vm, gm, dnm, states, rstates, dnum, dd, dq,
                                               dk, dv, BH, N, eps, hdr, st)
                 : launch<false, kPhiElu1>(qm, km, vm, gm, dnm, states, rstates, dnum, dd, dq, dk,
                                           dv, BH, N, eps, hdr, st);
}

}  // namespace la
