// SIMT (fp32 FMA) kernels for the causal and non-causal forward passes.
//
// These take any 1 <= Dk, Dv <= 128 and either input dtype, and compute in
// fp32 throughout, so float32 inputs are never rounded to a tensor-core
// operand type. Causal evaluation is the chunked two-pass form:
//   pass 1  per chunk c of 64 tokens: dS_c = sum_{j in c} phi(k_j) v_j^T,
//           dz_c = sum_{j in c} phi(k_j)                       (chunk_state)
//   scan    P_c = sum_{c' < c} dS_c' (exclusive prefix over chunks)   (scan)
//   pass 2  o_i = [phi(q_i)^T P_c + sum_{j in c, j <= i} w_ij v_j]
//               / [phi(q_i)^T zP_c + sum_{j in c, j <= i} w_ij + eps],
//           w_ij = phi(q_i).phi(k_j)                         (chunk_output)
// This is an exact regrouping of the prefix sums S_i, z_i of "Why Replace
// Attention? The Softmax Bottleneck and the Path to Linear Time", section 7.1,
// into whole chunks plus a masked in-chunk part; the prefix over chunks is
// the parallel scan the same blog names in section 7.7.
// Non-causal evaluation splits the sequence, reduces the partial S, z
// (section 6.2's boxed S and z) and applies them to every query.
#include "common.cuh"
#include "kernels.h"

namespace la {

namespace {

constexpr int kThreads = 256;

template <typename T>
__device__ __forceinline__ void load_rows_phi(float* dst, int ld, const T* src, int rows,
                                              int valid, int D) {
    // dst[r * ld + c] = phi(src[r * D + c]) for r < valid, 0 for padded rows.
    for (int idx = threadIdx.x; idx < rows * D; idx += blockDim.x) {
        int r = idx / D, c = idx - r * D;
        dst[r * ld + c] = r < valid ? phi(to_f(src[(int64_t)r * D + c])) : 0.f;
    }
}

template <typename T>
__device__ __forceinline__ void load_rows(float* dst, int ld, const T* src, int rows, int valid,
                                          int M) {
    for (int idx = threadIdx.x; idx < rows * M; idx += blockDim.x) {
        int r = idx / M, c = idx - r * M;
        dst[r * ld + c] = r < valid ? to_f(src[(int64_t)r * M + c]) : 0.f;
    }
}

// grid (nchunks, BH). states: [BH, nchunks, D*M + D] fp32.
template <typename T>
__global__ void __launch_bounds__(kThreads) chunk_state_kernel(const T* __restrict__ k,
                                                               const T* __restrict__ v,
                                                               float* __restrict__ states,
                                                               int N, int D, int M) {
    extern __shared__ float sm[];
    float* fK = sm;                 // [64][D]
    float* sV = sm + kChunk * D;    // [64][M]
    const int c = blockIdx.x, nchunks = gridDim.x;
    const int64_t bh = blockIdx.y;
    const int t0 = c * kChunk;
    const int valid = min(kChunk, N - t0);
    load_rows_phi(fK, D, k + (bh * N + t0) * D, kChunk, valid, D);
    load_rows(sV, M, v + (bh * N + t0) * M, kChunk, valid, M);
    __syncthreads();
    const int E = D * M + D;
    float* out = states + (bh * nchunks + c) * (int64_t)E;
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        float s = 0.f;
        if (e < D * M) {
            int cc = e / M, m = e - cc * M;
            for (int j = 0; j < valid; ++j) s = fmaf(fK[j * D + cc], sV[j * M + m], s);
        } else {
            int cc = e - D * M;
            for (int j = 0; j < valid; ++j) s += fK[j * D + cc];
        }
        out[e] = s;
    }
}

// Exclusive prefix over chunks, in place, starting from the initial state
// (S0, z0; zero when null); the total goes to S_out / z_out.
// One thread per (bh, element).
__global__ void chunk_scan_kernel(float* __restrict__ states, const float* __restrict__ S0,
                                  const float* __restrict__ z0, float* __restrict__ S_out,
                                  float* __restrict__ z_out, int64_t BH, int nchunks, int D,
                                  int M) {
    const int E = D * M + D;
    int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (gid >= BH * E) return;
    int64_t bh = gid / E;
    int e = (int)(gid - bh * E);
    float* p = states + bh * nchunks * (int64_t)E + e;
    float run = !S0 ? 0.f : e < D * M ? S0[bh * D * M + e] : z0[bh * D + (e - D * M)];
    for (int c = 0; c < nchunks; ++c) {
        float t = p[(int64_t)c * E];
        p[(int64_t)c * E] = run;
        run += t;
    }
    if (e < D * M) {
        if (S_out) S_out[bh * D * M + e] = run;
    } else if (z_out) {
        z_out[bh * D + (e - D * M)] = run;
    }
}

// grid (nchunks, BH). Reads the exclusive prefix state of its chunk.
template <typename T>
__global__ void __launch_bounds__(kThreads) chunk_output_kernel(
    const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
    const float* __restrict__ states, T* __restrict__ o, int N, int D, int M, float eps) {
    extern __shared__ float sm[];
    const int ldk = D + 1;
    float* fQ = sm;                       // [64][D+1]
    float* fK = fQ + kChunk * ldk;        // [64][D+1]
    float* sV = fK + kChunk * ldk;        // [64][M]
    float* P = sV + kChunk * M;           // [D][M] then zP [D]
    float* A = P + D * M + D;             // [64][65]
    float* den = A + kChunk * (kChunk + 1);  // [64]
    const int c = blockIdx.x, nchunks = gridDim.x;
    const int64_t bh = blockIdx.y;
    const int t0 = c * kChunk;
    const int valid = min(kChunk, N - t0);
    const int E = D * M + D;
    load_rows_phi(fQ, ldk, q + (bh * N + t0) * D, kChunk, valid, D);
    load_rows_phi(fK, ldk, k + (bh * N + t0) * D, kChunk, valid, D);
    load_rows(sV, M, v + (bh * N + t0) * M, kChunk, valid, M);
    const float* st = states + (bh * nchunks + c) * (int64_t)E;
    for (int e = threadIdx.x; e < E; e += blockDim.x) P[e] = st[e];
    __syncthreads();
    const float* zP = P + D * M;
    // Masked in-chunk similarities A_ij = phi(q_i).phi(k_j) for j <= i.
    for (int idx = threadIdx.x; idx < kChunk * kChunk; idx += blockDim.x) {
        int i = idx >> 6, j = idx & 63;
        float s = 0.f;
        if (j <= i && i < valid) {
            for (int cc = 0; cc < D; ++cc) s = fmaf(fQ[i * ldk + cc], fK[j * ldk + cc], s);
        }
        A[i * (kChunk + 1) + j] = s;
    }
    __syncthreads();
    // Denominators: in-chunk row sum + phi(q_i).zP, one warp per row.
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = warp; i < kChunk; i += kThreads / 32) {
        float s = A[i * (kChunk + 1) + lane] + A[i * (kChunk + 1) + lane + 32];
        for (int cc = lane; cc < D; cc += 32) s = fmaf(fQ[i * ldk + cc], zP[cc], s);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
        if (lane == 0) den[i] = s + eps;
    }
    __syncthreads();
    T* oc = o + (bh * N + t0) * M;
    for (int idx = threadIdx.x; idx < kChunk * M; idx += blockDim.x) {
        int i = idx / M, m = idx - i * M;
        if (i >= valid) continue;
        float s = 0.f;
        for (int j = 0; j <= i; ++j) s = fmaf(A[i * (kChunk + 1) + j], sV[j * M + m], s);
        for (int cc = 0; cc < D; ++cc) s = fmaf(fQ[i * ldk + cc], P[cc * M + m], s);
        oc[(int64_t)i * M + m] = from_f<T>(s / den[i]);
    }
}

// grid (nsplit, BH): partial S, z over a contiguous token range.
template <typename T>
__global__ void __launch_bounds__(kThreads) nc_partial_kernel(const T* __restrict__ k,
                                                              const T* __restrict__ v,
                                                              float* __restrict__ partials,
                                                              int N, int D, int M,
                                                              int tokens_per_split) {
    extern __shared__ float sm[];
    float* fK = sm;               // [64][D]
    float* sV = sm + kChunk * D;  // [64][M]
    const int s = blockIdx.x, nsplit = gridDim.x;
    const int64_t bh = blockIdx.y;
    const int E = D * M + D;
    constexpr int kPer = (kMaxDim * kMaxDim + kMaxDim + kThreads - 1) / kThreads;
    float acc[kPer];
#pragma unroll
    for (int r = 0; r < kPer; ++r) acc[r] = 0.f;
    const int begin = s * tokens_per_split;
    const int end = min(N, begin + tokens_per_split);
    for (int t0 = begin; t0 < end; t0 += kChunk) {
        const int valid = min(kChunk, end - t0);
        __syncthreads();
        load_rows_phi(fK, D, k + (bh * N + t0) * D, kChunk, valid, D);
        load_rows(sV, M, v + (bh * N + t0) * M, kChunk, valid, M);
        __syncthreads();
#pragma unroll
        for (int r = 0; r < kPer; ++r) {
            int e = threadIdx.x + r * kThreads;
            if (e < D * M) {
                int cc = e / M, m = e - cc * M;
                float a = acc[r];
                for (int j = 0; j < valid; ++j) a = fmaf(fK[j * D + cc], sV[j * M + m], a);
                acc[r] = a;
            } else if (e < E) {
                int cc = e - D * M;
                float a = acc[r];
                for (int j = 0; j < valid; ++j) a += fK[j * D + cc];
                acc[r] = a;
            }
        }
    }
    float* out = partials + (bh * nsplit + s) * (int64_t)E;
#pragma unroll
    for (int r = 0; r < kPer; ++r) {
        int e = threadIdx.x + r * kThreads;
        if (e < E) out[e] = acc[r];
    }
}

// Sums the partials of every split into total [BH, E]; one thread per (bh, element).
__global__ void nc_reduce_kernel(const float* __restrict__ partials, float* __restrict__ total,
                                 int64_t BH, int nsplit, int E) {
    int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (gid >= BH * E) return;
    int64_t bh = gid / E;
    int e = (int)(gid - bh * E);
    const float* p = partials + bh * nsplit * (int64_t)E + e;
    float s = 0.f;
    for (int i = 0; i < nsplit; ++i) s += p[(int64_t)i * E];
    total[gid] = s;
}

// grid (ceil(N/64), BH): o_i = phi(q_i)^T S / (phi(q_i)^T z + eps).
template <typename T>
__global__ void __launch_bounds__(kThreads) nc_apply_kernel(const T* __restrict__ q,
                                                            const float* __restrict__ total,
                                                            T* __restrict__ o, int N, int D,
                                                            int M, float eps) {
    extern __shared__ float sm[];
    const int ldk = D + 1;
    float* fQ = sm;                    // [64][D+1]
    float* S = fQ + kChunk * ldk;      // [D][M] then z [D]
    float* den = S + D * M + D;        // [64]
    const int64_t bh = blockIdx.y;
    const int t0 = blockIdx.x * kChunk;
    const int valid = min(kChunk, N - t0);
    const int E = D * M + D;
    load_rows_phi(fQ, ldk, q + (bh * N + t0) * D, kChunk, valid, D);
    const float* st = total + bh * E;
    for (int e = threadIdx.x; e < E; e += blockDim.x) S[e] = st[e];
    __syncthreads();
    const float* z = S + D * M;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = warp; i < kChunk; i += kThreads / 32) {
        float s = 0.f;
        for (int cc = lane; cc < D; cc += 32) s = fmaf(fQ[i * ldk + cc], z[cc], s);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
        if (lane == 0) den[i] = s + eps;
    }
    __syncthreads();
    T* oc = o + (bh * N + t0) * M;
    for (int idx = threadIdx.x; idx < kChunk * M; idx += blockDim.x) {
        int i = idx / M, m = idx - i * M;
        if (i >= valid) continue;
        float s = 0.f;
        for (int cc = 0; cc < D; ++cc) s = fmaf(fQ[i * ldk + cc], S[cc * M + m], s);
        oc[(int64_t)i * M + m] = from_f<T>(s / den[i]);
    }
}

template <typename T>
cudaError_t simt_causal_impl(const void* q, const void* k, const void* v, void* o, int64_t BH,
                             int N, int D, int M, float eps, const float* S0, const float* z0,
                             float* S_out, float* z_out, float* states, cudaStream_t st) {
    const int nchunks = (N + kChunk - 1) / kChunk;
    dim3 grid(nchunks, (unsigned)BH);
    size_t sm1 = sizeof(float) * (size_t)kChunk * (D + M);
    size_t sm3 = sizeof(float) * ((size_t)kChunk * (2 * (D + 1) + M) + (size_t)D * M + D +
                                  kChunk * (kChunk + 1) + kChunk);
    cudaError_t err;
    if ((err = cudaFuncSetAttribute(chunk_state_kernel<T>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm1)))
        return err;
    if ((err = cudaFuncSetAttribute(chunk_output_kernel<T>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm3)))
        return err;
    chunk_state_kernel<T><<<grid, kThreads, sm1, st>>>((const T*)k, (const T*)v, states, N, D, M);
    const int64_t total = BH * (int64_t)(D * M + D);
    chunk_scan_kernel<<<(unsigned)((total + 255) / 256), 256, 0, st>>>(states, S0, z0, S_out,
                                                                        z_out, BH, nchunks, D, M);
    chunk_output_kernel<T><<<grid, kThreads, sm3, st>>>((const T*)q, (const T*)k, (const T*)v,
                                                        states, (T*)o, N, D, M, eps);
    return cudaPeekAtLastError();
}

template <typename T>
cudaError_t simt_noncausal_impl(const void* q, const void* k, const void* v, void* o,
                                int64_t BH, int N, int D, int M, float eps, int nsplit,
                                float* partials, float* total, cudaStream_t st) {
    const int nchunks = (N + kChunk - 1) / kChunk;
    const int per_split = ((nchunks + nsplit - 1) / nsplit) * kChunk;
    size_t sm1 = sizeof(float) * (size_t)kChunk * (D + M);
    size_t sm3 = sizeof(float) * ((size_t)kChunk * (D + 1) + (size_t)D * M + D + kChunk);
    cudaError_t err;
    if ((err = cudaFuncSetAttribute(nc_partial_kernel<T>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm1)))
        return err;
    if ((err = cudaFuncSetAttribute(nc_apply_kernel<T>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm3)))
        return err;
    nc_partial_kernel<T><<<dim3(nsplit, (unsigned)BH), kThreads, sm1, st>>>(
        (const T*)k, (const T*)v, partials, N, D, M, per_split);
    const int E = D * M + D;
    const int64_t tot = BH * (int64_t)E;
    nc_reduce_kernel<<<(unsigned)((tot + 255) / 256), 256, 0, st>>>(partials, total, BH, nsplit,
                                                                     E);
    nc_apply_kernel<T><<<dim3(nchunks, (unsigned)BH), kThreads, sm3, st>>>(
        (const T*)q, total, (T*)o, N, D, M, eps);
    return cudaPeekAtLastError();
}

// ------------------------------------------------------------ causal backward
//
// Gradients of L through o for o_i = num_i / den_i, num_i = phi(q_i)^T S_i,
// den_i = phi(q_i)^T z_i + eps (S_i, z_i the inclusive prefix sums). With
// g_i = dL/do_i, dnum_i = g_i / den_i and dden_i = -(g_i . o_i) / den_i:
//   dphi(q_i) = S_i dnum_i + z_i dden_i
//   dphi(k_j) = R_j v_j + r_j,   dv_j = R_j^T phi(k_j),
// with the reverse (suffix) sums R_j = sum_{i>=j} phi(q_i) dnum_i^T and
// r_j = sum_{i>=j} phi(q_i) dden_i: a forward and a reverse cumulative sum, so
// no S_i is stored ("Transformers Are RNNs: Linear Attention", "Turn Causal
// Attention into a Recurrence"). Per chunk of 64 tokens both sums split into
// the chunk's carried-in state and a masked in-chunk part, as in the forward.
// dq = dphi(q) * phi'(q) with phi'(x) = 1 (x > 0), e^x (x <= 0) = min(phi(x), 1).

// grid (nchunks, BH): per row dnum (M) and dden into rowg [BH, N, M + 1]; per
// chunk [dR ; dr] = sum_i phi(q_i) [dnum_i ; dden_i]^T into rstates.
template <typename T>
__global__ void __launch_bounds__(kThreads) bwd_rows_kernel(
    const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
    const T* __restrict__ dout, const float* __restrict__ states, float* __restrict__ rowg,
    float* __restrict__ rstates, int N, int D, int M, float eps) {
    extern __shared__ float sm[];
    const int ldk = D + 1;
    float* fQ = sm;                       // [64][D+1]
    float* fK = fQ + kChunk * ldk;        // [64][D+1]
    float* sV = fK + kChunk * ldk;        // [64][M]
    float* sG = sV + kChunk * M;          // [64][M]   g, then dnum
    float* P = sG + kChunk * M;           // [D][M] then zP [D]
    float* A = P + D * M + D;             // [64][65]
    float* den = A + kChunk * (kChunk + 1);   // [64]
    float* dd = den + kChunk;                 // [64] dden
    const int c = blockIdx.x, nchunks = gridDim.x;
    const int64_t bh = blockIdx.y;
    const int t0 = c * kChunk;
    const int valid = min(kChunk, N - t0);
    const int E = D * M + D;
    load_rows_phi(fQ, ldk, q + (bh * N + t0) * D, kChunk, valid, D);
    load_rows_phi(fK, ldk, k + (bh * N + t0) * D, kChunk, valid, D);
    load_rows(sV, M, v + (bh * N + t0) * M, kChunk, valid, M);
    load_rows(sG, M, dout + (bh * N + t0) * M, kChunk, valid, M);
    const float* st = states + (bh * nchunks + c) * (int64_t)E;
    for (int e = threadIdx.x; e < E; e += blockDim.x) P[e] = st[e];
    __syncthreads();
    const float* zP = P + D * M;
    for (int idx = threadIdx.x; idx < kChunk * kChunk; idx += blockDim.x) {
        int i = idx >> 6, j = idx & 63;
        float s = 0.f;
        if (j <= i && i < valid)
            for (int cc = 0; cc < D; ++cc) s = fmaf(fQ[i * ldk + cc], fK[j * ldk + cc], s);
        A[i * (kChunk + 1) + j] = s;
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = warp; i < kChunk; i += kThreads / 32) {
        float s = A[i * (kChunk + 1) + lane] + A[i * (kChunk + 1) + lane + 32];
        for (int cc = lane; cc < D; cc += 32) s = fmaf(fQ[i * ldk + cc], zP[cc], s);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
        if (lane == 0) den[i] = s + eps;
    }
    __syncthreads();
    // o_i (recomputed) -> dnum_i = g_i / den_i and the row dot g_i . o_i, one warp per row.
    float* rg = rowg + (bh * N + t0) * (int64_t)(M + 1);
    for (int i = warp; i < kChunk; i += kThreads / 32) {
        float dot = 0.f;
        for (int m = lane; m < M; m += 32) {
            float s = 0.f;
            for (int j = 0; j <= i; ++j) s = fmaf(A[i * (kChunk + 1) + j], sV[j * M + m], s);
            for (int cc = 0; cc < D; ++cc) s = fmaf(fQ[i * ldk + cc], P[cc * M + m], s);
            const float o = s / den[i];
            const float g = sG[i * M + m];
            dot = fmaf(g, o, dot);
            sG[i * M + m] = g / den[i];                   // dnum (a row is owned by one warp)
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
        const float ddn = -dot / den[i];
        if (lane == 0) dd[i] = i < valid ? ddn : 0.f;
        if (i < valid) {
            for (int m = lane; m < M; m += 32) rg[(int64_t)i * (M + 1) + m] = sG[i * M + m];
            if (lane == 0) rg[(int64_t)i * (M + 1) + M] = ddn;
        }
    }
    __syncthreads();
    float* out = rstates + (bh * nchunks + c) * (int64_t)E;
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        float s = 0.f;
        if (e < D * M) {
            int cc = e / M, m = e - cc * M;
            for (int i = 0; i < valid; ++i) s = fmaf(fQ[i * ldk + cc], sG[i * M + m], s);
        } else {
            int cc = e - D * M;
            for (int i = 0; i < valid; ++i) s = fmaf(fQ[i * ldk + cc], dd[i], s);
        }
        out[e] = s;
    }
}

// Reverse exclusive sum over chunks, in place: chunk c gets the sum of chunks > c.
__global__ void chunk_rscan_kernel(float* __restrict__ rstates, int64_t BH, int nchunks, int E) {
    int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (gid >= BH * E) return;
    int64_t bh = gid / E;
    int e = (int)(gid - bh * E);
    float* p = rstates + bh * nchunks * (int64_t)E + e;
    float run = 0.f;
    for (int c = nchunks - 1; c >= 0; --c) {
        float t = p[(int64_t)c * E];
        p[(int64_t)c * E] = run;
        run += t;
    }
}

// grid (nchunks, BH): dq, dk, dv of the chunk from its carried-in forward state
// (S_prev, z_prev), the carried-in reverse sums (R_next, r_next) and the rows'
// dnum, dden.
template <typename T>
__global__ void __launch_bounds__(kThreads) bwd_grad_kernel(
    const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
    const float* __restrict__ states, const float* __restrict__ rstates,
    const float* __restrict__ rowg, T* __restrict__ dq, T* __restrict__ dk, T* __restrict__ dv,
    int N, int D, int M) {
    extern __shared__ float sm[];
    const int ldk = D + 1;
    float* fQ = sm;                       // [64][D+1]
    float* fK = fQ + kChunk * ldk;        // [64][D+1]
    float* sV = fK + kChunk * ldk;        // [64][M]
    float* DN = sV + kChunk * M;          // [64][M] dnum
    float* dd = DN + kChunk * M;          // [64] dden
    float* P = dd + kChunk;               // [D][M] S_prev, then z_prev [D]
    float* R = P + D * M + D;             // [D][M] R_next, then r_next [D]
    float* W = R + D * M + D;             // [64][65] phi(q_i).phi(k_j), j <= i
    float* G = W + kChunk * (kChunk + 1); // [64][65] v_j.dnum_i + dden_i, j <= i
    const int c = blockIdx.x, nchunks = gridDim.x;
    const int64_t bh = blockIdx.y;
    const int t0 = c * kChunk;
    const int valid = min(kChunk, N - t0);
    const int E = D * M + D;
    load_rows_phi(fQ, ldk, q + (bh * N + t0) * D, kChunk, valid, D);
    load_rows_phi(fK, ldk, k + (bh * N + t0) * D, kChunk, valid, D);
    load_rows(sV, M, v + (bh * N + t0) * M, kChunk, valid, M);
    const float* rg = rowg + (bh * N + t0) * (int64_t)(M + 1);
    for (int idx = threadIdx.x; idx < kChunk * (M + 1); idx += blockDim.x) {
        int i = idx / (M + 1), m = idx - i * (M + 1);
        float x = i < valid ? rg[idx] : 0.f;
        if (m < M) DN[i * M + m] = x;
        else dd[i] = x;
    }
    const float* st = states + (bh * nchunks + c) * (int64_t)E;
    const float* rs = rstates + (bh * nchunks + c) * (int64_t)E;
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        P[e] = st[e];
        R[e] = rs[e];
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < kChunk * kChunk; idx += blockDim.x) {
        int i = idx >> 6, j = idx & 63;
        float w = 0.f, g = 0.f;
        if (j <= i && i < valid) {
            for (int cc = 0; cc < D; ++cc) w = fmaf(fQ[i * ldk + cc], fK[j * ldk + cc], w);
            for (int m = 0; m < M; ++m) g = fmaf(sV[j * M + m], DN[i * M + m], g);
            g += dd[i];
        }
        W[i * (kChunk + 1) + j] = w;
        G[i * (kChunk + 1) + j] = g;
    }
    __syncthreads();
    // dq: dphi(q_i) = S_prev dnum_i + z_prev dden_i + sum_{j<=i} G_ij phi(k_j).
    T* dqc = dq + (bh * N + t0) * D;
    for (int idx = threadIdx.x; idx < kChunk * D; idx += blockDim.x) {
        int i = idx / D, d = idx - i * D;
        if (i >= valid) continue;
        float s = P[D * M + d] * dd[i];
        for (int m = 0; m < M; ++m) s = fmaf(P[d * M + m], DN[i * M + m], s);
        for (int j = 0; j <= i; ++j) s = fmaf(G[i * (kChunk + 1) + j], fK[j * ldk + d], s);
        const float f = fQ[i * ldk + d];
        dqc[(int64_t)i * D + d] = from_f<T>(s * fminf(f, 1.f));
    }
    // dk: dphi(k_j) = R_next v_j + r_next + sum_{i>=j} G_ij phi(q_i).
    T* dkc = dk + (bh * N + t0) * D;
    for (int idx = threadIdx.x; idx < kChunk * D; idx += blockDim.x) {
        int j = idx / D, d = idx - j * D;
        if (j >= valid) continue;
        float s = R[D * M + d];
        for (int m = 0; m < M; ++m) s = fmaf(R[d * M + m], sV[j * M + m], s);
        for (int i = j; i < valid; ++i) s = fmaf(G[i * (kChunk + 1) + j], fQ[i * ldk + d], s);
        const float f = fK[j * ldk + d];
        dkc[(int64_t)j * D + d] = from_f<T>(s * fminf(f, 1.f));
    }
    // dv: dv_j = R_next^T phi(k_j) + sum_{i>=j} W_ij dnum_i.
    T* dvc = dv + (bh * N + t0) * M;
    for (int idx = threadIdx.x; idx < kChunk * M; idx += blockDim.x) {
        int j = idx / M, m = idx - j * M;
        if (j >= valid) continue;
        float s = 0.f;
        for (int d = 0; d < D; ++d) s = fmaf(R[d * M + m], fK[j * ldk + d], s);
        for (int i = j; i < valid; ++i) s = fmaf(W[i * (kChunk + 1) + j], DN[i * M + m], s);
        dvc[(int64_t)j * M + m] = from_f<T>(s);
    }
}

template <typename T>
cudaError_t simt_causal_bwd_impl(const void* q, const void* k, const void* v, const void* dout,
                                 void* dq, void* dk, void* dv, int64_t BH, int N, int D, int M,
                                 float eps, float* states, float* rstates, float* rowg,
                                 cudaStream_t st) {
    const int nchunks = (N + kChunk - 1) / kChunk;
    dim3 grid(nchunks, (unsigned)BH);
    const size_t sm1 = sizeof(float) * (size_t)kChunk * (D + M);
    const size_t sm2 = sizeof(float) * ((size_t)kChunk * (2 * (D + 1) + 2 * M) + (size_t)D * M + D +
                                        kChunk * (kChunk + 1) + 2 * kChunk);
    const size_t sm3 = sizeof(float) * ((size_t)kChunk * (2 * (D + 1) + 2 * M) + kChunk +
                                        2 * ((size_t)D * M + D) + 2 * kChunk * (kChunk + 1));
    cudaError_t err;
    if ((err = cudaFuncSetAttribute(chunk_state_kernel<T>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm1)) ||
        (err = cudaFuncSetAttribute(bwd_rows_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)sm2)) ||
        (err = cudaFuncSetAttribute(bwd_grad_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)sm3)))
        return err;
    const int E = D * M + D;
    const int64_t total = BH * (int64_t)E;
    chunk_state_kernel<T><<<grid, kThreads, sm1, st>>>((const T*)k, (const T*)v, states, N, D, M);
    chunk_scan_kernel<<<(unsigned)((total + 255) / 256), 256, 0, st>>>(states, nullptr, nullptr,
                                                                        nullptr, nullptr, BH,
                                                                        nchunks, D, M);
    bwd_rows_kernel<T><<<grid, kThreads, sm2, st>>>((const T*)q, (const T*)k, (const T*)v,
                                                    (const T*)dout, states, rowg, rstates, N, D,
                                                    M, eps);
    chunk_rscan_kernel<<<(unsigned)((total + 255) / 256), 256, 0, st>>>(rstates, BH, nchunks, E);
    bwd_grad_kernel<T><<<grid, kThreads, sm3, st>>>((const T*)q, (const T*)k, (const T*)v, states,
                                                    rstates, rowg, (T*)dq, (T*)dk, (T*)dv, N, D, M);
    return cudaPeekAtLastError();
}

}  // namespace

size_t simt_causal_workspace(int64_t BH, int N, int D, int M) {
    const int nchunks = (N + kChunk - 1) / kChunk;
    return sizeof(float) * (size_t)BH * nchunks * (size_t)(D * M + D);
}

int simt_noncausal_splits(int64_t BH, int N) {
    const int nchunks = (N + kChunk - 1) / kChunk;
    int64_t want = (2 * 152 + BH - 1) / BH;
    if (want < 1) want = 1;
    if (want > nchunks) want = nchunks;
    if (want > 1024) want = 1024;
    return (int)want;
}

size_t simt_noncausal_workspace(int64_t BH, int N, int D, int M) {
    const int nsplit = simt_noncausal_splits(BH, N);
    return sizeof(float) * (size_t)BH * (size_t)(nsplit + 1) * (size_t)(D * M + D);
}

cudaError_t simt_causal(const void* q, const void* k, const void* v, void* o, la_dtype dt,
                        int64_t BH, int N, int D, int M, float eps, const float* S0,
                        const float* z0, float* S_out, float* z_out, void* scratch,
                        cudaStream_t st) {
    float* states = (float*)scratch;
    if (dt == LA_F32)
        return simt_causal_impl<float>(q, k, v, o, BH, N, D, M, eps, S0, z0, S_out, z_out,
                                       states, st);
    return simt_causal_impl<__nv_bfloat16>(q, k, v, o, BH, N, D, M, eps, S0, z0, S_out, z_out,
                                           states, st);
}

cudaError_t simt_noncausal(const void* q, const void* k, const void* v, void* o, la_dtype dt,
                           int64_t BH, int N, int D, int M, float eps, void* scratch,
                           cudaStream_t st) {
    const int nsplit = simt_noncausal_splits(BH, N);
    float* partials = (float*)scratch;
    float* total = partials + (size_t)BH * nsplit * (size_t)(D * M + D);
    if (dt == LA_F32)
        return simt_noncausal_impl<float>(q, k, v, o, BH, N, D, M, eps, nsplit, partials, total,
                                          st);
    return simt_noncausal_impl<__nv_bfloat16>(q, k, v, o, BH, N, D, M, eps, nsplit, partials,
                                              total, st);
}

size_t simt_causal_bwd_workspace(int64_t BH, int N, int D, int M) {
    const int nchunks = (N + kChunk - 1) / kChunk;
    return sizeof(float) * ((size_t)2 * BH * nchunks * (size_t)(D * M + D) +
                            (size_t)BH * N * (size_t)(M + 1));
}

cudaError_t simt_causal_bwd(const void* q, const void* k, const void* v, const void* dout,
                            void* dq, void* dk, void* dv, la_dtype dt, int64_t BH, int N, int D,
                            int M, float eps, void* scratch, cudaStream_t st) {
    const int nchunks = (N + kChunk - 1) / kChunk;
    float* states = (float*)scratch;
    float* rstates = states + (size_t)BH * nchunks * (size_t)(D * M + D);
    float* rowg = rstates + (size_t)BH * nchunks * (size_t)(D * M + D);
    if (dt == LA_F32)
        return simt_causal_bwd_impl<float>(q, k, v, dout, dq, dk, dv, BH, N, D, M, eps, states,
                                           rstates, rowg, st);
    return simt_causal_bwd_impl<__nv_bfloat16>(q, k, v, dout, dq, dk, dv, BH, N, D, M, eps, states,
                                               rstates, rowg, st);
}

}  // namespace la
