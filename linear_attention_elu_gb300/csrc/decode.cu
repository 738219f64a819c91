// Recurrent decode step: S <- S + phi(k) v^T, z <- z + phi(k),
// o = phi(q)^T S / (phi(q)^T z + eps), in place on caller-owned fp32 state
// ("Why Replace Attention? The Softmax Bottleneck and the Path to Linear
// Time", section 7.2, steps 1-4; "Transformers Are RNNs: Linear Attention",
// "Turn Causal Attention into a Recurrence").
//
// The step is bound by streaming S (Dk*Dv fp32) in and out once per head.
// For Dk = Dv = 64 one warp owns one head: lanes 0-15 and 16-31 take the
// even and odd rows of S, each lane a 16-byte column group, so every row
// pass is one coalesced 128-bit load and store per lane; the new S row is
// contracted with phi(q) while it is still in registers.
#include "common.cuh"
#include "kernels.h"

namespace la {

namespace {

// Head h = b H + j of the flattened [B*H] axis reads its q and k at
// b ld_qk + j Dk and its v at b ld_v + j Dv: contiguous [B, H, D] inputs are
// passed as H = 1 (one row per head); the layer step reads them out of one
// [B, 3 H D] projection. B*H < 2^16 (the entry points check it), so the split
// is a 32-bit division, skipped for H = 1: it sits before the first load.
struct HeadRow {
    int64_t b;
    int j;
};
__device__ __forceinline__ HeadRow head_row(int64_t h, int H) {
    if (H == 1) return {h, 0};
    const int b = (int)h / H;
    return {b, (int)h - b * H};
}

// One warp per head, Dk = Dv = 64. blockDim = 256 (8 heads per block). The
// feature map is a template parameter: selected at run time it cost the step
// about 6 %.
template <typename T, int kFm>
__global__ void __launch_bounds__(256, 4) decode64_kernel(const T* __restrict__ q,
                                                       const T* __restrict__ k,
                                                       const T* __restrict__ v,
                                                       T* __restrict__ o, float* __restrict__ S,
                                                       float* __restrict__ z, int64_t BH,
                                                       float eps, int H, int64_t ld_qk,
                                                       int64_t ld_v) {
    constexpr int fm = kFm;
    // When launched as a programmatic dependent (the layer step), the inputs
    // come from the kernel before: wait for it (a no-op otherwise).
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int lane = threadIdx.x & 31;
    const int64_t h = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (h >= BH) return;
    const HeadRow hr = head_row(h, H);
    const T* qh = q + hr.b * ld_qk + hr.j * 64;
    const T* kh = k + hr.b * ld_qk + hr.j * 64;
    const T* vh = v + hr.b * ld_v + hr.j * 64;
    // Lane l holds phi(k), phi(q) and z for features l and l + 32.
    const float fk0 = fmap(to_f(kh[lane]), fm), fk1 = fmap(to_f(kh[lane + 32]), fm);
    const float fq0 = fmap(to_f(qh[lane]), fm), fq1 = fmap(to_f(qh[lane + 32]), fm);
    float* zh = z + h * 64;
    const float z0 = zh[lane] + fk0, z1 = zh[lane + 32] + fk1;
    zh[lane] = z0;
    zh[lane + 32] = z1;
    float den = fq0 * z0 + fq1 * z1;
    // Column group g = lane & 15 covers value columns 4g..4g+3; row parity = lane >> 4.
    const int g = lane & 15, par = lane >> 4;
    const float4 vv = make_float4(to_f(vh[4 * g]), to_f(vh[4 * g + 1]), to_f(vh[4 * g + 2]),
                                  to_f(vh[4 * g + 3]));
    float4* Sh = reinterpret_cast<float4*>(S + h * 64 * 64);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    // Rows in batches of 8: the batch's loads are all issued before any of its
    // stores, so each lane keeps 8 state loads in flight.
#pragma unroll
    for (int r0 = 0; r0 < 32; r0 += 8) {
        float4 sv[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) sv[u] = Sh[(2 * (r0 + u) + par) * 16 + g];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int row = 2 * (r0 + u) + par;
            // Feature `row` lives in lane row & 31, register (row >> 5).
            const float fkr = __shfl_sync(0xffffffffu, row < 32 ? fk0 : fk1, row & 31);
            const float fqr = __shfl_sync(0xffffffffu, row < 32 ? fq0 : fq1, row & 31);
            float4 s = sv[u];
            s.x = fmaf(fkr, vv.x, s.x);
            s.y = fmaf(fkr, vv.y, s.y);
            s.z = fmaf(fkr, vv.z, s.z);
            s.w = fmaf(fkr, vv.w, s.w);
            Sh[row * 16 + g] = s;
            acc.x = fmaf(fqr, s.x, acc.x);
            acc.y = fmaf(fqr, s.y, acc.y);
            acc.z = fmaf(fqr, s.z, acc.z);
            acc.w = fmaf(fqr, s.w, acc.w);
        }
    }
    // Rows were split by parity across the two half-warps: add the halves.
    acc.x += __shfl_xor_sync(0xffffffffu, acc.x, 16);
    acc.y += __shfl_xor_sync(0xffffffffu, acc.y, 16);
    acc.z += __shfl_xor_sync(0xffffffffu, acc.z, 16);
    acc.w += __shfl_xor_sync(0xffffffffu, acc.w, 16);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
    const float inv = 1.f / (den + eps);
    if (par == 0) {
        T* oh = o + h * 64 + 4 * g;
        oh[0] = from_f<T>(acc.x * inv);
        oh[1] = from_f<T>(acc.y * inv);
        oh[2] = from_f<T>(acc.z * inv);
        oh[3] = from_f<T>(acc.w * inv);
    }
}

// Any Dk, Dv <= 128: one block of 128 threads per head, thread m owns column m.
template <typename T, int kFm>
__global__ void __launch_bounds__(128) decode_generic_kernel(
    const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
    T* __restrict__ o, float* __restrict__ S, float* __restrict__ z, int D, int M, float eps,
    int H, int64_t ld_qk, int64_t ld_v) {
    constexpr int fm = kFm;
    __shared__ float fk[kMaxDim], fq[kMaxDim], red[4];
    const int64_t h = blockIdx.x;
    const int t = threadIdx.x;
    float dpart = 0.f;
    const HeadRow hr = head_row(h, H);
    if (t < D) {
        fk[t] = fmap(to_f(k[hr.b * ld_qk + hr.j * D + t]), fm);
        fq[t] = fmap(to_f(q[hr.b * ld_qk + hr.j * D + t]), fm);
        float zn = z[h * D + t] + fk[t];
        z[h * D + t] = zn;
        dpart = fq[t] * zn;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) dpart += __shfl_xor_sync(0xffffffffu, dpart, off);
    if ((t & 31) == 0) red[t >> 5] = dpart;
    __syncthreads();
    const float den = red[0] + red[1] + red[2] + red[3];
    if (t < M) {
        const float vm = to_f(v[hr.b * ld_v + hr.j * M + t]);
        float* Sh = S + h * (int64_t)D * M;
        float acc = 0.f;
        for (int c = 0; c < D; ++c) {
            float s = fmaf(fk[c], vm, Sh[c * M + t]);
            Sh[c * M + t] = s;
            acc = fmaf(fq[c], s, acc);
        }
        o[h * M + t] = from_f<T>(acc / (den + eps));
    }
}

template <typename T, int kFm>
cudaError_t decode_launch(const void* q, const void* k, const void* v, void* o, float* S, float* z,
                          int64_t BH, int D, int M, float eps, int H, int64_t ld_qk, int64_t ld_v,
                          cudaStream_t st) {
    if (D == 64 && M == 64) {
        const int heads_per_block = 8;
        const int64_t blocks = (BH + heads_per_block - 1) / heads_per_block;
        if (H > 1) {
            // The layer step: a programmatic dependent of the projection before it.
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3((unsigned)blocks);
            cfg.blockDim = dim3(256);
            cfg.stream = st;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[0].val.programmaticStreamSerializationAllowed = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            return cudaLaunchKernelEx(&cfg, decode64_kernel<T, kFm>, (const T*)q, (const T*)k,
                                      (const T*)v, (T*)o, S, z, BH, eps, H, ld_qk, ld_v);
        }
        decode64_kernel<T, kFm><<<(unsigned)blocks, 256, 0, st>>>(
            (const T*)q, (const T*)k, (const T*)v, (T*)o, S, z, BH, eps, H, ld_qk, ld_v);
    } else {
        decode_generic_kernel<T, kFm><<<(unsigned)BH, 128, 0, st>>>(
            (const T*)q, (const T*)k, (const T*)v, (T*)o, S, z, D, M, eps, H, ld_qk, ld_v);
    }
    return cudaPeekAtLastError();
}

template <typename T>
cudaError_t decode_impl(const void* q, const void* k, const void* v, void* o, float* S, float* z,
                        int64_t BH, int D, int M, float eps, int fm, int H, int64_t ld_qk,
                        int64_t ld_v, cudaStream_t st) {
    if (fm == kPhiIdentity)
        return decode_launch<T, kPhiIdentity>(q, k, v, o, S, z, BH, D, M, eps, H, ld_qk, ld_v, st);
    return decode_launch<T, kPhiElu1>(q, k, v, o, S, z, BH, D, M, eps, H, ld_qk, ld_v, st);
}

}  // namespace

cudaError_t decode_step(const void* q, const void* k, const void* v, void* o, float* S, float* z,
                        la_dtype dt, int64_t BH, int D, int M, float eps, int fm,
                        cudaStream_t st) {
    // Contiguous [B*H, D] inputs: one "batch row" per head.
    return decode_step_strided(q, k, v, o, S, z, dt, BH, D, M, eps, fm, 1, D, M, st);
}

cudaError_t decode_step_strided(const void* q, const void* k, const void* v, void* o, float* S,
                                float* z, la_dtype dt, int64_t BH, int D, int M, float eps, int fm,
                                int H, int64_t ld_qk, int64_t ld_v, cudaStream_t st) {
    if (dt == LA_F32)
        return decode_impl<float>(q, k, v, o, S, z, BH, D, M, eps, fm, H, ld_qk, ld_v, st);
    return decode_impl<__nv_bfloat16>(q, k, v, o, S, z, BH, D, M, eps, fm, H, ld_qk, ld_v, st);
}

}  // namespace la
