// Dense products Y = X W of the layer decode step (row-major X [rows, K],
// W [K, N], Y [rows, N], fp32 accumulation): the QKV projection and the output
// projection around the recurrent step ("Why Replace Attention? The Softmax
// Bottleneck and the Path to Linear Time", section 7.2, step 1: q, k, v are
// linear maps of the token's hidden state; the head outputs are mixed by W_o).
//
// bf16 storage with K and N multiples of 8 (16-byte row strides for TMA):
// gemm_tc_kernel, one CTA per 128 x 64 tile of Y. X tiles (128 rows x 64 k,
// K-major) and W tiles (64 k x 64 n, N-major) stream through a 4-stage TMA ring;
// one thread issues tcgen05.mma (M = 128, N = 64, K = 16) into a 64-column fp32
// accumulator in TMEM; four warps read it back (one TMEM lane quarter each),
// round to bf16 into a swizzled staging tile and a TMA store writes Y (rows and
// columns past the matrix are dropped; loads past it read zeros).
// Every other case (fp32 storage, unaligned widths): gemm_simt_kernel, 64 x 64
// tiles of Y, each of 256 threads accumulating a 4 x 4 block in fp32 registers
// over 16-deep slices of X and W staged in shared memory.
#include <cuda.h>
#include <cuda_bf16.h>

#include <atomic>

#include "common.cuh"
#include "kernels.h"
#include "tc_common.cuh"
#include "tc_util.cuh"

namespace la {

namespace {

using namespace tc;
using namespace tcc;

constexpr int kBM = 128, kBN = 64, kBK = 64, kGStages = 4;
constexpr uint32_t kATile = kBM * kBK * 2;                  // 16 KB
constexpr uint32_t kBTile = kBK * kBN * 2;                  // 8 KB
constexpr uint32_t kGStage = kATile + kBTile;
constexpr uint32_t kOffY = kGStages * kGStage;              // output staging [128 x 64] bf16
constexpr size_t kGSmem = 1024 + kOffY + kBM * kBN * 2;
constexpr int kGThreads = 128;

struct GemmMisc {
    uint64_t full[kGStages], empty[kGStages], done;
    uint32_t tmem_slot;
};

// Warp 0 lane 0: TMA producer. Warp 1: TMEM allocation, lane 0 issues the MMAs.
// All four warps: the epilogue (warp w reads TMEM lanes 32 w .. 32 w + 31 = rows).
__global__ void __launch_bounds__(kGThreads, 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap wmap,
               const __grid_constant__ CUtensorMap ymap, int K, WsHeader* hdr) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    __shared__ GemmMisc m;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n0 = blockIdx.x * kBN, r0 = blockIdx.y * kBM;
    const int nk = (K + kBK - 1) / kBK;
    auto a_tile = [&](int s) { return base + s * kGStage; };
    auto b_tile = [&](int s) { return base + s * kGStage + kATile; };
    uint8_t* ystage = base + kOffY;

    if (tid == 0) {
        for (int s = 0; s < kGStages; ++s) {
            mbar_init(&m.full[s], 1);
            mbar_init(&m.empty[s], 1);
        }
        mbar_init(&m.done, 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&m.tmem_slot, 64);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&xmap);
        tma_prefetch_desc(&wmap);
        tma_prefetch_desc(&ymap);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // Launched as a programmatic dependent of the previous kernel in the stream:
    // the set-up above touches no global memory; everything below waits for that
    // kernel's completion.
    pdl_launch_dependents();
    pdl_wait();
    const uint32_t tmem = m.tmem_slot;
    const uint32_t max_spin = hdr->max_spin;
    bool ok = true;

    if (warp == 0 && lane == 0) {
        int kk = 0;
        for (; kk < nk; ++kk) {
            const int s = kk % kGStages;
            if (kk >= kGStages && !mbar_wait(&m.empty[s], ((kk / kGStages) - 1) & 1, max_spin)) {
                ok = false;
                break;
            }
            mbar_arrive_expect_tx(&m.full[s], kGStage);
            tma_load_3d(a_tile(s), &xmap, &m.full[s], kk * kBK, r0, 0);
            tma_load_3d(b_tile(s), &wmap, &m.full[s], n0, kk * kBK, 0);
        }
        // Every issued load lands before the CTA exits.
        for (int j = kk - kGStages > 0 ? kk - kGStages : 0; j < kk; ++j)
            mbar_wait(&m.full[j % kGStages], (j / kGStages) & 1, kDefaultMaxSpin);
    } else if (warp == 1 && lane == 0) {
        // A: X tile, K-major (rows of 64 k). B: W tile, N-major (rows of 64 n, one atom).
        const uint32_t idesc = idesc_bf16_f32(kBM, kBN, false, true);
        for (int kk = 0; kk < nk; ++kk) {
            const int s = kk % kGStages;
            if (!mbar_wait(&m.full[s], (kk / kGStages) & 1, max_spin)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t aa = smem_u32(a_tile(s)), ba = smem_u32(b_tile(s));
#pragma unroll
            for (int k16 = 0; k16 < kBK / 16; ++k16)
                mma_bf16(tmem, smem_desc(aa + k16 * 32, 16, 1024, kSwizzle128B),
                         smem_desc(ba + k16 * 2048, 1024, 1024, kSwizzle128B), idesc,
                         (kk > 0 || k16 > 0) ? 1u : 0u);
            mma_commit(&m.empty[s]);
        }
        mma_commit(&m.done);
    }
    // Epilogue: row 32 warp + lane, 64 fp32 columns -> bf16 staging -> TMA store.
    __syncwarp();
    const bool done = mbar_wait(&m.done, 0, max_spin);
    tc_fence_after();
    const int row = 32 * warp + lane;
    const uint32_t ta = tmem + ((uint32_t)(32 * warp) << 16);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint32_t r[2][16];
        tmem_ld16(ta + 32 * h, r[0]);
        tmem_ld16(ta + 32 * h + 16, r[1]);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint32_t* rr = r[c >> 1];
            const int e0 = 8 * (c & 1);
            const uint4 v = make_uint4(pack_bf16(__uint_as_float(rr[e0]), __uint_as_float(rr[e0 + 1])),
                                       pack_bf16(__uint_as_float(rr[e0 + 2]), __uint_as_float(rr[e0 + 3])),
                                       pack_bf16(__uint_as_float(rr[e0 + 4]), __uint_as_float(rr[e0 + 5])),
                                       pack_bf16(__uint_as_float(rr[e0 + 6]), __uint_as_float(rr[e0 + 7])));
            *reinterpret_cast<uint4*>(ystage + sw128_offset(row, 32 * h + 8 * c)) = v;
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    const bool all_ok = __syncthreads_and(ok && done);
    if (tid == 0) {
        if (all_ok) {
            tma_store_3d(&ymap, ystage, n0, r0, 0);
            tma_store_commit();
            tma_store_wait_read<0>();   // the staging tile has been read; the writes land by kernel end
        } else {
            report_timeout(hdr);
        }
    }
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, 64);
    }
}

// fp32-FMA product for the remaining cases: 64 x 64 tiles of Y, 256 threads,
// thread (ty, tx) owns rows 4 ty .. 4 ty + 3 and columns 4 tx .. 4 tx + 3.
template <typename T>
__global__ void __launch_bounds__(256) gemm_simt_kernel(const T* __restrict__ X, const T* __restrict__ W,
                                                       T* __restrict__ Y, int rows, int K, int N) {
    __shared__ float xs[16][64 + 4];   // xs[k][r]
    __shared__ float ws[16][64 + 4];   // ws[k][n]
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int r0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < K; k0 += 16) {
        for (int idx = tid; idx < 16 * 64; idx += 256) {
            const int kk = idx & 15, r = idx >> 4;           // X: 16 consecutive k per row
            const int gr = r0 + r, gk = k0 + kk;
            xs[kk][r] = (gr < rows && gk < K) ? to_f(X[(int64_t)gr * K + gk]) : 0.f;
            const int n = idx & 63, kw = idx >> 6;           // W: 64 consecutive n per k
            const int gn = n0 + n, gkw = k0 + kw;
            ws[kw][n] = (gkw < K && gn < N) ? to_f(W[(int64_t)gkw * N + gn]) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = xs[kk][4 * ty + i];
#pragma unroll
            for (int j = 0; j < 4; ++j) b[j] = ws[kk][4 * tx + j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int gr = r0 + 4 * ty + i;
        if (gr >= rows) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int gn = n0 + 4 * tx + j;
            if (gn < N) Y[(int64_t)gr * N + gn] = from_f<T>(acc[i][j]);
        }
    }
}

// Row-major [outer, inner] bf16 matrix as a 3-D tensor map (inner, outer, 1),
// 128-byte swizzled boxes of box_inner x box_outer.
bool encode_rowmajor(CUtensorMap* map, const void* ptr, int inner, int outer, int box_inner,
                     int box_outer) {
    EncodeTiled enc = get_encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)outer, 1};
    cuuint64_t strides[2] = {(cuuint64_t)inner * 2, (cuuint64_t)inner * 2 * outer};
    cuuint32_t box[3] = {(cuuint32_t)box_inner, (cuuint32_t)box_outer, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides,
               box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool gemm_uses_tensor_cores(int K, int N, la_dtype dt) {
    return dt == LA_BF16 && K % 8 == 0 && N % 8 == 0;
}

cudaError_t gemm(const void* X, const void* W, void* Y, int rows, int K, int N, la_dtype dt,
                 void* ws_header, cudaStream_t st) {
    if (rows <= 0 || N <= 0) return cudaSuccess;
    if (gemm_uses_tensor_cores(K, N, dt)) {
        CUtensorMap xm, wm, ym;
        if (!encode_rowmajor(&xm, X, K, rows, kBK, kBM) || !encode_rowmajor(&wm, W, N, K, kBN, kBK) ||
            !encode_rowmajor(&ym, Y, N, rows, kBN, kBM))
            return cudaErrorInvalidValue;
        static std::atomic<int> optin[kMaxDevices];
        cudaError_t err = ensure_smem_optin(gemm_tc_kernel, (int)kGSmem, optin);
        if (err) return err;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((N + kBN - 1) / kBN, (rows + kBM - 1) / kBM);
        cfg.blockDim = dim3(kGThreads);
        cfg.dynamicSmemBytes = kGSmem;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, gemm_tc_kernel, xm, wm, ym, K,
                                  reinterpret_cast<WsHeader*>(ws_header));
    }
    const dim3 grid((N + 63) / 64, (rows + 63) / 64);
    if (dt == LA_BF16)
        gemm_simt_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(
            static_cast<const __nv_bfloat16*>(X), static_cast<const __nv_bfloat16*>(W),
            static_cast<__nv_bfloat16*>(Y), rows, K, N);
    else
        gemm_simt_kernel<float><<<grid, 256, 0, st>>>(static_cast<const float*>(X),
                                                     static_cast<const float*>(W),
                                                     static_cast<float*>(Y), rows, K, N);
    return cudaPeekAtLastError();
}

}  // namespace la
