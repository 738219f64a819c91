// Positive random features on the tensor cores: out = exp(X W^T - |x|^2 / 2 -
// shift) / sqrt(R) for bf16 X [rows, 64] and W [64, 64] (R = D = 64), the
// random-feature map the research-hub "Linear Attention" page names ("Key math /
// How it works": positive random features for an unbiased softmax-kernel
// estimate). The projection X W^T is a dense contraction: one tcgen05 MMA group
// (M = 128 rows, N = 64 features, K = 64) per 128-row tile, fp32 accumulators
// in TMEM.
//
// One persistent CTA per SM walks the row tiles. Warp 0 streams X tiles in
// through 4 TMA stages (128-byte swizzle); warp 1 owns TMEM (two 64-column
// accumulators) and issues the MMAs against W, loaded once; two epilogue
// warpgroups (warps 2-5 and 6-9) take alternate tiles, each with its own
// accumulator: one tile row per thread, they read the row's |x|^2 from the
// stage and the projections from TMEM, apply the exponential and store bf16
// rows through two swizzled staging tiles of their own with TMA. The exponential is CUDA's fast __expf: its error
// (a few ulp of fp32 at these arguments) is far below the bf16 rounding of the
// output. Every wait is bounded (kDefaultMaxSpin); a wait that expires makes the
// CTA drain its copies, free TMEM and return.
#include <atomic>

#include "common.cuh"
#include "kernels.h"
#include "tc_util.cuh"
#include "tc_common.cuh"

namespace la {
namespace tcc {
namespace {

using namespace la::tc;

constexpr int kRfStages = 4;
constexpr int kRfThreads = 320;                   // producer, MMA, 2 x 4 epilogue warps
constexpr uint32_t kXTile = 128 * 128;            // 128 rows x 64 bf16
constexpr uint32_t kWTile = 64 * 128;             // 64 rows x 64 bf16
constexpr uint32_t kOffW = kRfStages * kXTile;
constexpr uint32_t kOffOut = kOffW + kWTile;      // 2 x 2 output staging tiles
constexpr size_t kRfSmem = 1024 + kOffOut + 4 * kXTile;
constexpr uint32_t kRfCols = 128;                 // two 64-column fp32 accumulators

struct RfMisc {
    uint64_t full[kRfStages], empty[kRfStages];
    uint64_t acc_full[2], tmem_free[2], w_full;
    uint32_t tmem_slot;
};

__global__ void __launch_bounds__(kRfThreads, 1)
rf_tc_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap wmap,
             const __grid_constant__ CUtensorMap omap, int ntiles, float shift, float scale) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    __shared__ RfMisc m;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nlocal = (ntiles - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;
    const uint32_t spin = kDefaultMaxSpin;
    auto xstage = [&](int s) { return base + s * kXTile; };
    uint8_t* wtile = base + kOffW;
    auto ostage = [&](int b) { return base + kOffOut + b * kXTile; };

    if (threadIdx.x == 0) {
        for (int s = 0; s < kRfStages; ++s) {
            mbar_init(&m.full[s], 1);
            mbar_init(&m.empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&m.acc_full[b], 1);
            mbar_init(&m.tmem_free[b], 1);
        }
        mbar_init(&m.w_full, 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&m.tmem_slot, kRfCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = m.tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------ producer
        if (lane == 0) {
            mbar_arrive_expect_tx(&m.w_full, kWTile);
            tma_load_3d(wtile, &wmap, &m.w_full, 0, 0, 0);
            int i = 0;
            for (; i < nlocal; ++i) {
                const int s = i % kRfStages;
                if (i >= kRfStages && !mbar_wait(&m.empty[s], ((i / kRfStages) - 1) & 1, spin))
                    break;
                const int tile = (int)blockIdx.x + i * (int)gridDim.x;
                mbar_arrive_expect_tx(&m.full[s], kXTile);
                tma_load_3d(xstage(s), &xmap, &m.full[s], 0, tile * 128, 0);
            }
            // Every issued load lands before the CTA exits.
            mbar_wait(&m.w_full, 0, spin);
            for (int j = i - kRfStages > 0 ? i - kRfStages : 0; j < i; ++j)
                mbar_wait(&m.full[j % kRfStages], (j / kRfStages) & 1, spin);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issue
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(128, 64, false, false);
            bool ok = mbar_wait(&m.w_full, 0, spin);
            const uint32_t wa = smem_u32(wtile);
            for (int i = 0; i < nlocal && ok; ++i) {
                const int s = i % kRfStages, b = i & 1;
                if (!mbar_wait(&m.full[s], (i / kRfStages) & 1, spin)) break;
                if (i >= 2 && !mbar_wait(&m.tmem_free[b], ((i - 2) >> 1) & 1, spin)) break;
                tc_fence_after();
                const uint32_t xa = smem_u32(xstage(s));
#pragma unroll
                for (int k16 = 0; k16 < 4; ++k16)
                    mma_bf16(tmem + 64 * b, smem_desc(xa + k16 * 32, 16, 1024, kSwizzle128B),
                             smem_desc(wa + k16 * 32, 16, 1024, kSwizzle128B), idesc, k16 > 0);
                mma_commit(&m.acc_full[b]);
            }
        }
    } else {
        // ------------------------------------------------------ epilogue
        // Group eg takes the tiles i = eg (mod 2), which use accumulator eg.
        // Thread = tile row `row` = TMEM lane; warp w reads lane quarter w % 4.
        const int eg = (warp - 2) >> 2;
        const int et = threadIdx.x - 64 - 128 * eg;       // 0..127
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        const int bar_id = 1 + eg;
        bool ok = true;
        for (int i = eg; i < nlocal; i += 2) {
            const int s = i % kRfStages, b = i & 1;
            const int tile = (int)blockIdx.x + i * (int)gridDim.x;
            ok = ok && mbar_wait(&m.acc_full[b], (i >> 1) & 1, spin);
            tc_fence_after();
            // |x|^2 over the row. The sum takes the row's eight 16-byte pieces in
            // any order; reading piece c ^ (row & 7) spreads a warp's 32 rows over
            // all banks instead of stacking them on four.
            float ss = 0.f;
            const uint8_t* xr = xstage(s) + row * 128;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const uint4 u = *reinterpret_cast<const uint4*>(xr + ((c ^ (row & 7)) << 4));
                const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float lo = bf_lo(w[e]), hi = __uint_as_float(w[e] & 0xFFFF0000u);
                    ss = fmaf(lo, lo, ss);
                    ss = fmaf(hi, hi, ss);
                }
            }
            const float off = 0.5f * ss + shift;
            uint32_t o[32];
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t r[2][16];
                tmem_ld16(tmem + lane_base + 64 * b + 32 * half, r[0]);
                tmem_ld16(tmem + lane_base + 64 * b + 32 * half + 16, r[1]);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    o[16 * half + e] =
                        pack_bf16(__expf(__uint_as_float(r[e >> 3][2 * (e & 7)]) - off) * scale,
                                  __expf(__uint_as_float(r[e >> 3][2 * (e & 7) + 1]) - off) * scale);
            }
            tc_fence_before();
            ok = named_bar_and(bar_id, 128, ok);
            if (!ok) break;
            if (et == 0) {
                mbar_arrive(&m.empty[s]);          // stage read (MMA done, rows read)
                mbar_arrive(&m.tmem_free[b]);      // accumulator read
                tma_store_wait_read<1>();          // this group's tile before last is stored
            }
            named_bar(bar_id, 128);
            uint8_t* os = ostage(2 * eg + ((i >> 1) & 1));
#pragma unroll
            for (int c = 0; c < 8; ++c)
                *reinterpret_cast<uint4*>(os + sw128_offset(row, 8 * c)) =
                    make_uint4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
            fence_proxy_async_smem();
            named_bar(bar_id, 128);
            if (et == 0) {
                tma_store_3d(&omap, os, 0, tile * 128, 0);
                tma_store_commit();
            }
        }
        if (et == 0) tma_store_wait_all<0>();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kRfCols);
}

// [rows, 64] bf16 as 3-D (64, rows, 1); box 64 x box_rows x 1, 128-byte swizzle.
bool encode_rows64(CUtensorMap* map, const void* ptr, int64_t rows, int box_rows) {
    EncodeTiled enc = get_encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {64, (cuuint64_t)rows, 1};
    cuuint64_t strides[2] = {128, (cuuint64_t)rows * 128};
    cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides,
               box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace
}  // namespace tcc

bool tc_random_features_supported(int D, int R, la_dtype dt) {
    return dt == LA_BF16 && D == 64 && R == 64;
}

cudaError_t tc_random_features(const void* x, const void* W, void* out, int64_t rows, float shift,
                               cudaStream_t st) {
    using namespace tcc;
    const int64_t ntiles = (rows + 127) / 128;
    if (ntiles > (1LL << 24)) return cudaErrorInvalidValue;   // row coordinates stay in int
    CUtensorMap xm, wm, om;
    if (!encode_rows64(&xm, x, rows, 128) || !encode_rows64(&wm, W, 64, 64) ||
        !encode_rows64(&om, out, rows, 128))
        return cudaErrorInvalidValue;
    static std::atomic<int> optin[kMaxDevices];
    cudaError_t err = ensure_smem_optin(rf_tc_kernel, (int)kRfSmem, optin);
    if (err != cudaSuccess) return err;
    const int grid = (int)(ntiles < sm_count() ? ntiles : sm_count());
    rf_tc_kernel<<<grid, kRfThreads, kRfSmem, st>>>(xm, wm, om, (int)ntiles, shift,
                                                    0.125f /* 1 / sqrt(64) */);
    return cudaPeekAtLastError();
}

}  // namespace la
