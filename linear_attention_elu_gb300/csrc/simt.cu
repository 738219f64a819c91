// SIMT (fp32 FMA) kernels: the causal and non-causal forward passes, the
// causal and non-causal backward, and the positive random features for the
// shapes the tensor-core kernel does not take.
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
// (section 6.2's boxed S and z) and applies them to every query. For
// Dk, Dv <= 64 the chunk products run in the register-tiled kernels further
// down (the same sums in the same order); the general kernels take the rest.
#include "common.cuh"
#include "kernels.h"

namespace la {

namespace {

constexpr int kThreads = 256;
constexpr int kScanBatch = 16;  // chunks per batch of loads in the chunk scans

template <typename T>
__device__ __forceinline__ void load_rows_phi(float* dst, int ld, const T* src, int rows,
                                              int valid, int D, int fm) {
    // dst[r * ld + c] = phi(src[r * D + c]) for r < valid, 0 for padded rows.
    for (int idx = threadIdx.x; idx < rows * D; idx += blockDim.x) {
        int r = idx / D, c = idx - r * D;
        dst[r * ld + c] = r < valid ? fmap(to_f(src[(int64_t)r * D + c]), fm) : 0.f;
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
                                                               int N, int D, int M, int fm) {
    extern __shared__ float sm[];
    float* fK = sm;                 // [64][D]
    float* sV = sm + kChunk * D;    // [64][M]
    const int c = blockIdx.x, nchunks = gridDim.x;
    const int64_t bh = blockIdx.y;
    const int t0 = c * kChunk;
    const int valid = min(kChunk, N - t0);
    load_rows_phi(fK, D, k + (bh * N + t0) * D, kChunk, valid, D, fm);
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
    // Batches of kScanBatch chunks: all loads of a batch are in flight before
    // its stores, instead of one DRAM round trip per chunk.
    for (int c0 = 0; c0 < nchunks; c0 += kScanBatch) {
        float t[kScanBatch];
#pragma unroll
        for (int u = 0; u < kScanBatch; ++u)
            t[u] = c0 + u < nchunks ? p[(int64_t)(c0 + u) * E] : 0.f;
#pragma unroll
        for (int u = 0; u < kScanBatch; ++u)
            if (c0 + u < nchunks) {
                p[(int64_t)(c0 + u) * E] = run;
                run += t[u];
            }
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
    const float* __restrict__ states, T* __restrict__ o, int N, int D, int M, float eps, int fm) {
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
    load_rows_phi(fQ, ldk, q + (bh * N + t0) * D, kChunk, valid, D, fm);
    load_rows_phi(fK, ldk, k + (bh * N + t0) * D, kChunk, valid, D, fm);
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
                                                              int tokens_per_split, int fm) {
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
        load_rows_phi(fK, D, k + (bh * N + t0) * D, kChunk, valid, D, fm);
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
                                                            int M, float eps, int fm) {
    extern __shared__ float sm[];
    const int ldk = D + 1;
    float* fQ = sm;                    // [64][D+1]
    float* S = fQ + kChunk * ldk;      // [D][M] then z [D]
    float* den = S + D * M + D;        // [64]
    const int64_t bh = blockIdx.y;
    const int t0 = blockIdx.x * kChunk;
    const int valid = min(kChunk, N - t0);
    const int E = D * M + D;
    load_rows_phi(fQ, ldk, q + (bh * N + t0) * D, kChunk, valid, D, fm);
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

// Register-tiled products on 64 x 64 fp32 tiles in shared memory, rows of kLd
// floats. Thread t of 256 owns output rows 4 tr .. 4 tr + 3 (tr = t / 16) and
// four columns: 4 tc .. 4 tc + 3 when the B operand is stored k-major, tc,
// tc + 16, tc + 32, tc + 48 when it is stored column-major (tc = t % 16). Every
// operand load is a float4 over four consecutive k (or four consecutive rows,
// or columns); with rows of 68 floats none of them is bank-conflicted beyond
// the two wavefronts a 16-lane float4 load needs. The 32 lanes of warp w own
// rows 8 w .. 8 w + 7, which bounds the triangular sums warp-uniformly.
constexpr int kLd = 68;

__device__ __forceinline__ int col_of(bool b_kmajor, int tc, int y) {
    return b_kmajor ? 4 * tc + y : tc + 16 * y;
}

// acc[x][y] += sum_{k0 <= k < k1} Aop(4 tr + x, k) Bop(k, col_of(y)), k0 and k1
// multiples of 4. Aop(r, k) is A[r kLdA + k] (row-major) or A[k kLdA + r]
// (k-major); Bop(k, c) is B[k kLdB + c] (k-major) or B[c kLdB + k] (column-major).
// Row lengths other than 68 keep the bank pattern when they are 4 mod 32.
template <bool kAKmaj, bool kBKmaj, int kLdA = kLd, int kLdB = kLd>
__device__ __forceinline__ void mm4(float (&acc)[4][4], const float* A, const float* B, int k0,
                                    int k1, int tr, int tc) {
#pragma unroll 2
    for (int kk = k0; kk < k1; kk += 4) {
        float a[4][4], b[4][4];  // a[x][u] = Aop(r_x, kk + u), b[u][y] = Bop(kk + u, c_y)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if (kAKmaj) {
                const float4 f = *reinterpret_cast<const float4*>(A + (kk + i) * kLdA + 4 * tr);
                a[0][i] = f.x, a[1][i] = f.y, a[2][i] = f.z, a[3][i] = f.w;
            } else {
                const float4 f = *reinterpret_cast<const float4*>(A + (4 * tr + i) * kLdA + kk);
                a[i][0] = f.x, a[i][1] = f.y, a[i][2] = f.z, a[i][3] = f.w;
            }
            if (kBKmaj) {
                const float4 f = *reinterpret_cast<const float4*>(B + (kk + i) * kLdB + 4 * tc);
                b[i][0] = f.x, b[i][1] = f.y, b[i][2] = f.z, b[i][3] = f.w;
            } else {
                const float4 f = *reinterpret_cast<const float4*>(B + (tc + 16 * i) * kLdB + kk);
                b[0][i] = f.x, b[1][i] = f.y, b[2][i] = f.z, b[3][i] = f.w;
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int x = 0; x < 4; ++x)
#pragma unroll
                for (int y = 0; y < 4; ++y) acc[x][y] = fmaf(a[x][u], b[u][y], acc[x][y]);
    }
}

__device__ __forceinline__ void zero4x4(float (&acc)[4][4]) {
#pragma unroll
    for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y) acc[x][y] = 0.f;
}

// A [64][width] global tile into shared rows of kLd floats (feature map `fm`
// applied unless kNoMap); rows >= valid and columns >= width are zero. The trip count is
// fixed so that each thread's 16 loads are in flight together.
constexpr int kPerThread = kChunk * kChunk / kThreads;
template <typename T>
__device__ __forceinline__ void load_tile(float* dst, const T* src, int valid, int width,
                                          int fm) {
    float x[kPerThread];
#pragma unroll
    for (int u = 0; u < kPerThread; ++u) {
        const int idx = threadIdx.x + u * kThreads, r = idx >> 6, c = idx & 63;
        x[u] = (r < valid && c < width) ? to_f(src[(int64_t)r * width + c]) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kPerThread; ++u) {
        const int idx = threadIdx.x + u * kThreads, r = idx >> 6, c = idx & 63;
        dst[r * kLd + c] = (fm != kNoMap && r < valid && c < width) ? fmap(x[u], fm) : x[u];
    }
}

// A [D][M] state block into shared memory, as stored (dst[d kLd + m]) or
// transposed (dst[m kLd + d]); entries beyond D or M are zero.
__device__ __forceinline__ void load_state(float* dst, const float* src, int D, int M,
                                           bool transposed) {
    float x[kPerThread];
#pragma unroll
    for (int u = 0; u < kPerThread; ++u) {
        const int idx = threadIdx.x + u * kThreads, d = idx >> 6, m = idx & 63;
        x[u] = (d < D && m < M) ? src[d * M + m] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kPerThread; ++u) {
        const int idx = threadIdx.x + u * kThreads, d = idx >> 6, m = idx & 63;
        dst[transposed ? m * kLd + d : d * kLd + m] = x[u];
    }
}

// The chunk's dnum rows of rowg ([64][M + 1] from row 0) into shared rows.
__device__ __forceinline__ void load_dnum(float* dst, const float* rg, int valid, int M) {
    float x[kPerThread];
#pragma unroll
    for (int u = 0; u < kPerThread; ++u) {
        const int idx = threadIdx.x + u * kThreads, r = idx >> 6, c = idx & 63;
        x[u] = (r < valid && c < M) ? rg[(int64_t)r * (M + 1) + c] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kPerThread; ++u) {
        const int idx = threadIdx.x + u * kThreads;
        dst[(idx >> 6) * kLd + (idx & 63)] = x[u];
    }
}

// grid (nchunks, BH): per row dnum (M) and dden into rowg [BH, N, M + 1]; per
// chunk [dR ; dr] = sum_i phi(q_i) [dnum_i ; dden_i]^T into rstates. Causal:
// the chunk's slot of `states` holds its carried-in state and the rows add the
// masked in-chunk part; non-causal: chunk 0's slot holds the whole sequence's
// (S, z), which every row sees.
template <typename T, bool kCausal, int kFm>
__global__ void __launch_bounds__(kThreads, 2) bwd_rows_kernel(
    const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
    const T* __restrict__ dout, const float* __restrict__ states, float* __restrict__ rowg,
    float* __restrict__ rstates, int N, int D, int M, float eps) {
    constexpr int fm = kFm;
    extern __shared__ __align__(16) float sm[];
    float* fQ = sm;                       // [64][kLd] each
    float* fK = fQ + kChunk * kLd;
    float* sV = fK + kChunk * kLd;
    float* sG = sV + kChunk * kLd;        // g, then dnum
    float* P = sG + kChunk * kLd;         // S_prev [d][m]
    float* A = P + kChunk * kLd;          // phi(q_i).phi(k_j), j <= i
    float* zP = A + kChunk * kLd;         // [64]
    float* den = zP + kChunk;             // [64]
    float* dot = den + kChunk;            // [64]
    float* dd = dot + kChunk;             // [64]
    const int c = blockIdx.x, nchunks = gridDim.x;
    const int64_t bh = blockIdx.y;
    const int t0 = c * kChunk;
    const int valid = min(kChunk, N - t0);
    const int E = D * M + D;
    const int t = threadIdx.x, tr = t >> 4, tc = t & 15, warp = t >> 5, lane = t & 31;
    load_tile(fQ, q + (bh * N + t0) * D, valid, D, fm);
    if (kCausal) {
        load_tile(fK, k + (bh * N + t0) * D, valid, D, fm);
        load_tile(sV, v + (bh * N + t0) * M, valid, M, kNoMap);
    }
    load_tile(sG, dout + (bh * N + t0) * M, valid, M, kNoMap);
    const float* st = states + (bh * nchunks + (kCausal ? c : 0)) * (int64_t)E;
    load_state(P, st, D, M, false);
    for (int idx = t; idx < kChunk; idx += blockDim.x) zP[idx] = idx < D ? st[D * M + idx] : 0.f;
    __syncthreads();
    float acc[4][4];
    if (kCausal) {
        // A = phi(Q) phi(K)^T, masked to j <= i.
        zero4x4(acc);
        mm4<false, false>(acc, fQ, fK, 0, kChunk, tr, tc);
#pragma unroll
        for (int x = 0; x < 4; ++x)
#pragma unroll
            for (int y = 0; y < 4; ++y) {
                const int i = 4 * tr + x, j = col_of(false, tc, y);
                A[i * kLd + j] = j <= i ? acc[x][y] : 0.f;
            }
        __syncthreads();
    }
    for (int i = warp; i < kChunk; i += kThreads / 32) {
        float s2 = kCausal ? A[i * kLd + lane] + A[i * kLd + lane + 32] : 0.f;
        for (int cc = lane; cc < D; cc += 32) s2 = fmaf(fQ[i * kLd + cc], zP[cc], s2);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) s2 += __shfl_xor_sync(0xffffffffu, s2, off);
        if (lane == 0) den[i] = s2 + eps;
    }
    __syncthreads();
    // num = A V + phi(Q) S_prev; o = num / den; dnum = g / den; row dots g . o.
    // A(i, j) is zero for j > i: the sum over j stops after the warp's last row.
    zero4x4(acc);
    if (kCausal) mm4<false, true>(acc, A, sV, 0, 8 * warp + 8, tr, tc);
    mm4<false, true>(acc, fQ, P, 0, kChunk, tr, tc);
#pragma unroll
    for (int x = 0; x < 4; ++x) {
        const int i = 4 * tr + x;
        float part = 0.f;
#pragma unroll
        for (int y = 0; y < 4; ++y) {
            const int m = col_of(true, tc, y);
            const float g = sG[i * kLd + m];
            part = fmaf(g, acc[x][y] / den[i], part);
            sG[i * kLd + m] = (i < valid && m < M) ? g / den[i] : 0.f;
        }
        // The 16 lanes with the same tr share row i.
#pragma unroll
        for (int off = 8; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
        if (tc == 0) dot[i] = part;
    }
    __syncthreads();
    for (int i = t; i < kChunk; i += blockDim.x) dd[i] = i < valid ? -dot[i] / den[i] : 0.f;
    __syncthreads();
    float* rg = rowg + (bh * N + t0) * (int64_t)(M + 1);
    for (int idx = t; idx < valid * (M + 1); idx += blockDim.x) {
        const int i = idx / (M + 1), m = idx - i * (M + 1);
        rg[idx] = m < M ? sG[i * kLd + m] : dd[i];
    }
    // dR = phi(Q)^T dnum (rows d, columns m); dr = phi(Q)^T dden.
    float* out = rstates + (bh * nchunks + c) * (int64_t)E;
    zero4x4(acc);
    mm4<true, true>(acc, fQ, sG, 0, kChunk, tr, tc);
#pragma unroll
    for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y) {
            const int d = 4 * tr + x, m = col_of(true, tc, y);
            if (d < D && m < M) out[d * M + m] = acc[x][y];
        }
    for (int d = t; d < D; d += blockDim.x) {
        float s2 = 0.f;
        for (int i = 0; i < valid; ++i) s2 = fmaf(fQ[i * kLd + d], dd[i], s2);
        out[D * M + d] = s2;
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
    for (int c0 = nchunks - 1; c0 >= 0; c0 -= kScanBatch) {
        float t[kScanBatch];
#pragma unroll
        for (int u = 0; u < kScanBatch; ++u) t[u] = c0 - u >= 0 ? p[(int64_t)(c0 - u) * E] : 0.f;
#pragma unroll
        for (int u = 0; u < kScanBatch; ++u)
            if (c0 - u >= 0) {
                p[(int64_t)(c0 - u) * E] = run;
                run += t[u];
            }
    }
}

// Sum over chunks, in place: chunk 0 of each (bh) gets the sum of all chunks.
__global__ void chunk_total_kernel(float* __restrict__ parts, int64_t BH, int nchunks, int E) {
    int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (gid >= BH * E) return;
    int64_t bh = gid / E;
    int e = (int)(gid - bh * E);
    float* p = parts + bh * nchunks * (int64_t)E + e;
    float run = 0.f;
    for (int c0 = 0; c0 < nchunks; c0 += kScanBatch) {
        float t[kScanBatch];
#pragma unroll
        for (int u = 0; u < kScanBatch; ++u) t[u] = c0 + u < nchunks ? p[(int64_t)(c0 + u) * E] : 0.f;
#pragma unroll
        for (int u = 0; u < kScanBatch; ++u)
            if (c0 + u < nchunks) run += t[u];
    }
    p[0] = run;
}

// grid (nchunks, BH), D, M <= 64: the chunk's [S ; z] = phi(K)^T [V | 1] into
// states [BH, nchunks, D*M + D].
template <typename T>
__global__ void __launch_bounds__(kThreads) chunk_state_tiled_kernel(const T* __restrict__ k,
                                                             const T* __restrict__ v,
                                                             float* __restrict__ states, int N,
                                                             int D, int M, int fm) {
    extern __shared__ __align__(16) float sm[];
    float* fK = sm;                       // [64][kLd]
    float* sV = fK + kChunk * kLd;
    const int c = blockIdx.x, nchunks = gridDim.x;
    const int64_t bh = blockIdx.y;
    const int t0 = c * kChunk;
    const int valid = min(kChunk, N - t0);
    const int t = threadIdx.x, tr = t >> 4, tc = t & 15;
    load_tile(fK, k + (bh * N + t0) * D, valid, D, fm);
    load_tile(sV, v + (bh * N + t0) * M, valid, M, kNoMap);
    __syncthreads();
    float* out = states + (bh * nchunks + c) * (int64_t)(D * M + D);
    float acc[4][4];
    zero4x4(acc);
    mm4<true, true>(acc, fK, sV, 0, kChunk, tr, tc);
#pragma unroll
    for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y) {
            const int d = 4 * tr + x, m = col_of(true, tc, y);
            if (d < D && m < M) out[d * M + m] = acc[x][y];
        }
    if (t < D) {
        float s2 = 0.f;
        for (int j = 0; j < kChunk; ++j) s2 += fK[j * kLd + t];
        out[D * M + t] = s2;
    }
}

// grid (nchunks, BH): dq, dk, dv of the chunk from its carried-in forward state
// (S_prev, z_prev), the carried-in reverse sums (R_next, r_next) and the rows'
// dnum, dden. Non-causal: chunk 0's slots hold the whole sequence's (S, z) and
// (R, r), and there are no in-chunk terms.
template <typename T, bool kCausal, int kFm>
__global__ void __launch_bounds__(kThreads) bwd_grad_kernel(
    const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
    const float* __restrict__ states, const float* __restrict__ rstates,
    const float* __restrict__ rowg, T* __restrict__ dq, T* __restrict__ dk, T* __restrict__ dv,
    int N, int D, int M) {
    constexpr int fm = kFm;
    extern __shared__ __align__(16) float sm[];
    float* fQ = sm;                       // [64][kLd] each
    float* fK = fQ + kChunk * kLd;
    float* sV = fK + kChunk * kLd;
    float* DN = sV + kChunk * kLd;        // dnum [i][m]
    float* G = DN + kChunk * kLd;         // v_j.dnum_i + dden_i, j <= i
    float* PW = G + kChunk * kLd;         // S_prev^T [m][d], then W = phi(q_i).phi(k_j), j <= i
    float* R = PW + kChunk * kLd;         // R_next [d][m]
    float* Rt = R + kChunk * kLd;         // R_next^T [m][d]
    float* dd = Rt + kChunk * kLd;        // [64]
    float* zP = dd + kChunk;              // [64]
    float* rr = zP + kChunk;              // [64]
    const int c = blockIdx.x, nchunks = gridDim.x;
    const int64_t bh = blockIdx.y;
    const int t0 = c * kChunk;
    const int valid = min(kChunk, N - t0);
    const int E = D * M + D;
    const int t = threadIdx.x, tr = t >> 4, tc = t & 15, warp = t >> 5;
    load_tile(fQ, q + (bh * N + t0) * D, valid, D, fm);
    load_tile(fK, k + (bh * N + t0) * D, valid, D, fm);
    load_tile(sV, v + (bh * N + t0) * M, valid, M, kNoMap);
    const float* rg = rowg + (bh * N + t0) * (int64_t)(M + 1);
    const float* st = states + (bh * nchunks + (kCausal ? c : 0)) * (int64_t)E;
    const float* rs = rstates + (bh * nchunks + (kCausal ? c : 0)) * (int64_t)E;
    load_dnum(DN, rg, valid, M);
    load_state(PW, st, D, M, true);
    load_state(R, rs, D, M, false);
    load_state(Rt, rs, D, M, true);
    for (int idx = t; idx < kChunk; idx += blockDim.x) {
        dd[idx] = idx < valid ? rg[(int64_t)idx * (M + 1) + M] : 0.f;
        zP[idx] = idx < D ? st[D * M + idx] : 0.f;
        rr[idx] = idx < D ? rs[D * M + idx] : 0.f;
    }
    __syncthreads();
    float acc[4][4];
    if (kCausal) {
        // G = dnum V^T + dden 1^T, masked to j <= i.
        zero4x4(acc);
        mm4<false, false>(acc, DN, sV, 0, kChunk, tr, tc);
#pragma unroll
        for (int x = 0; x < 4; ++x)
#pragma unroll
            for (int y = 0; y < 4; ++y) {
                const int i = 4 * tr + x, j = col_of(false, tc, y);
                G[i * kLd + j] = (j <= i && i < valid) ? acc[x][y] + dd[i] : 0.f;
            }
    }
    __syncthreads();
    // dphi(q) = dnum S_prev^T + dden z_prev^T + G phi(K); rows i, columns d.
    zero4x4(acc);
    mm4<false, true>(acc, DN, PW, 0, kChunk, tr, tc);
    if (kCausal) mm4<false, true>(acc, G, fK, 0, 8 * warp + 8, tr, tc);
    T* dqc = dq + (bh * N + t0) * D;
#pragma unroll
    for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y) {
            const int i = 4 * tr + x, d = col_of(true, tc, y);
            if (i < valid && d < D) {
                const float s2 = fmaf(zP[d], dd[i], acc[x][y]);
                dqc[(int64_t)i * D + d] = from_f<T>(s2 * fmap_grad(fQ[i * kLd + d], fm));
            }
        }
    if (kCausal) {
        __syncthreads();  // S_prev^T is dead: its tile takes W
        zero4x4(acc);
        mm4<false, false>(acc, fQ, fK, 0, kChunk, tr, tc);
#pragma unroll
        for (int x = 0; x < 4; ++x)
#pragma unroll
            for (int y = 0; y < 4; ++y) {
                const int i = 4 * tr + x, j = col_of(false, tc, y);
                PW[i * kLd + j] = j <= i ? acc[x][y] : 0.f;
            }
    }
    // dphi(k) = V R_next^T + r_next^T + G^T phi(Q); rows j, columns d. G(i, j) is
    // zero for i < j: the sum over i starts at the warp's first row.
    zero4x4(acc);
    mm4<false, true>(acc, sV, Rt, 0, kChunk, tr, tc);
    if (kCausal) mm4<true, true>(acc, G, fQ, 8 * warp, kChunk, tr, tc);
    T* dkc = dk + (bh * N + t0) * D;
#pragma unroll
    for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y) {
            const int j = 4 * tr + x, d = col_of(true, tc, y);
            if (j < valid && d < D)
                dkc[(int64_t)j * D + d] =
                    from_f<T>((acc[x][y] + rr[d]) * fmap_grad(fK[j * kLd + d], fm));
        }
    if (kCausal) __syncthreads();
    // dv = phi(K) R_next + W^T dnum; rows j, columns m.
    zero4x4(acc);
    mm4<false, true>(acc, fK, R, 0, kChunk, tr, tc);
    if (kCausal) mm4<true, true>(acc, PW, DN, 8 * warp, kChunk, tr, tc);
    T* dvc = dv + (bh * N + t0) * M;
#pragma unroll
    for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y) {
            const int j = 4 * tr + x, m = col_of(true, tc, y);
            if (j < valid && m < M) dvc[(int64_t)j * M + m] = from_f<T>(acc[x][y]);
        }
}

// grid (nchunks, BH), D, M <= 64: the chunk's rows of the causal output from
// its exclusive prefix state (S_prev, z_prev) and the masked in-chunk terms,
// o_i = (sum_{j <= i} A_ij v_j + phi(q_i)^T S_prev) / (sum_{j <= i} A_ij +
// phi(q_i)^T z_prev + eps) with A_ij = phi(q_i).phi(k_j). Register-tiled; the
// same sums in the same order as chunk_output_kernel.
template <typename T>
__global__ void __launch_bounds__(kThreads, 2) chunk_output_tiled_kernel(
    const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
    const float* __restrict__ states, T* __restrict__ o, int N, int D, int M, float eps, int fm) {
    extern __shared__ __align__(16) float sm[];
    float* fQ = sm;                       // [64][kLd] each
    float* fK = fQ + kChunk * kLd;
    float* sV = fK + kChunk * kLd;
    float* P = sV + kChunk * kLd;         // S_prev [d][m]
    float* A = P + kChunk * kLd;          // phi(q_i).phi(k_j), j <= i
    float* zP = A + kChunk * kLd;         // [64]
    float* den = zP + kChunk;             // [64]
    const int c = blockIdx.x, nchunks = gridDim.x;
    const int64_t bh = blockIdx.y;
    const int t0 = c * kChunk;
    const int valid = min(kChunk, N - t0);
    const int E = D * M + D;
    const int t = threadIdx.x, tr = t >> 4, tc = t & 15, warp = t >> 5, lane = t & 31;
    load_tile(fQ, q + (bh * N + t0) * D, valid, D, fm);
    load_tile(fK, k + (bh * N + t0) * D, valid, D, fm);
    load_tile(sV, v + (bh * N + t0) * M, valid, M, kNoMap);
    const float* st = states + (bh * nchunks + c) * (int64_t)E;
    load_state(P, st, D, M, false);
    for (int idx = t; idx < kChunk; idx += blockDim.x) zP[idx] = idx < D ? st[D * M + idx] : 0.f;
    __syncthreads();
    float acc[4][4];
    zero4x4(acc);
    mm4<false, false>(acc, fQ, fK, 0, kChunk, tr, tc);
#pragma unroll
    for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y) {
            const int i = 4 * tr + x, j = col_of(false, tc, y);
            A[i * kLd + j] = (j <= i && i < valid) ? acc[x][y] : 0.f;
        }
    __syncthreads();
    for (int i = warp; i < kChunk; i += kThreads / 32) {
        float s2 = A[i * kLd + lane] + A[i * kLd + lane + 32];
        for (int cc = lane; cc < D; cc += 32) s2 = fmaf(fQ[i * kLd + cc], zP[cc], s2);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) s2 += __shfl_xor_sync(0xffffffffu, s2, off);
        if (lane == 0) den[i] = s2 + eps;
    }
    __syncthreads();
    zero4x4(acc);
    mm4<false, true>(acc, A, sV, 0, 8 * warp + 8, tr, tc);
    mm4<false, true>(acc, fQ, P, 0, kChunk, tr, tc);
    T* oc = o + (bh * N + t0) * M;
#pragma unroll
    for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y) {
            const int i = 4 * tr + x, m = col_of(true, tc, y);
            if (i < valid && m < M) oc[(int64_t)i * M + m] = from_f<T>(acc[x][y] / den[i]);
        }
}

template <typename T>
cudaError_t simt_causal_impl(const void* q, const void* k, const void* v, void* o, int64_t BH,
                             int N, int D, int M, float eps, int fm, const float* S0,
                             const float* z0, float* S_out, float* z_out, float* states,
                             cudaStream_t st) {
    const int nchunks = (N + kChunk - 1) / kChunk;
    dim3 grid(nchunks, (unsigned)BH);
    const bool tiled = D <= kChunk && M <= kChunk;
    const size_t sm1 = tiled ? sizeof(float) * (2 * (size_t)kChunk * kLd)
                             : sizeof(float) * (size_t)kChunk * (D + M);
    const size_t sm3 = tiled ? sizeof(float) * (5 * (size_t)kChunk * kLd + 2 * kChunk)
                             : sizeof(float) * ((size_t)kChunk * (2 * (D + 1) + M) +
                                                (size_t)D * M + D + kChunk * (kChunk + 1) + kChunk);
    cudaError_t err;
    if (tiled) {
        if ((err = cudaFuncSetAttribute(chunk_state_tiled_kernel<T>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm1)) ||
            (err = cudaFuncSetAttribute(chunk_output_tiled_kernel<T>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm3)))
            return err;
        chunk_state_tiled_kernel<T><<<grid, kThreads, sm1, st>>>((const T*)k, (const T*)v, states,
                                                                 N, D, M, fm);
    } else {
        if ((err = cudaFuncSetAttribute(chunk_state_kernel<T>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm1)) ||
            (err = cudaFuncSetAttribute(chunk_output_kernel<T>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm3)))
            return err;
        chunk_state_kernel<T><<<grid, kThreads, sm1, st>>>((const T*)k, (const T*)v, states, N, D,
                                                           M, fm);
    }
    const int64_t total = BH * (int64_t)(D * M + D);
    chunk_scan_kernel<<<(unsigned)((total + 255) / 256), 256, 0, st>>>(states, S0, z0, S_out,
                                                                        z_out, BH, nchunks, D, M);
    if (tiled)
        chunk_output_tiled_kernel<T><<<grid, kThreads, sm3, st>>>(
            (const T*)q, (const T*)k, (const T*)v, states, (T*)o, N, D, M, eps, fm);
    else
        chunk_output_kernel<T><<<grid, kThreads, sm3, st>>>((const T*)q, (const T*)k, (const T*)v,
                                                            states, (T*)o, N, D, M, eps, fm);
    return cudaPeekAtLastError();
}

// grid (nsplit, BH), D, M <= 64: partial [S ; z] over a contiguous token range,
// register-tiled; the same sums in the same order as nc_partial_kernel.
template <typename T>
__global__ void __launch_bounds__(kThreads) nc_partial_tiled_kernel(const T* __restrict__ k,
                                                                    const T* __restrict__ v,
                                                                    float* __restrict__ partials,
                                                                    int N, int D, int M,
                                                                    int tokens_per_split, int fm) {
    extern __shared__ __align__(16) float sm[];
    float* fK = sm;                       // [64][kLd]
    float* sV = fK + kChunk * kLd;
    const int s = blockIdx.x, nsplit = gridDim.x;
    const int64_t bh = blockIdx.y;
    const int E = D * M + D;
    const int t = threadIdx.x, tr = t >> 4, tc = t & 15;
    float acc[4][4];
    zero4x4(acc);
    float zacc = 0.f;
    const int begin = s * tokens_per_split;
    const int end = min(N, begin + tokens_per_split);
    for (int t0 = begin; t0 < end; t0 += kChunk) {
        const int valid = min(kChunk, end - t0);
        __syncthreads();
        load_tile(fK, k + (bh * N + t0) * D, valid, D, fm);
        load_tile(sV, v + (bh * N + t0) * M, valid, M, kNoMap);
        __syncthreads();
        mm4<true, true>(acc, fK, sV, 0, kChunk, tr, tc);
        if (t < D)
            for (int j = 0; j < kChunk; ++j) zacc += fK[j * kLd + t];
    }
    float* out = partials + (bh * nsplit + s) * (int64_t)E;
#pragma unroll
    for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y) {
            const int d = 4 * tr + x, m = col_of(true, tc, y);
            if (d < D && m < M) out[d * M + m] = acc[x][y];
        }
    if (t < D) out[D * M + t] = zacc;
}

// grid (ceil(N/64), BH), D, M <= 64: o_i = phi(q_i)^T S / (phi(q_i)^T z + eps),
// register-tiled; the same sums in the same order as nc_apply_kernel.
template <typename T>
__global__ void __launch_bounds__(kThreads) nc_apply_tiled_kernel(const T* __restrict__ q,
                                                                  const float* __restrict__ total,
                                                                  T* __restrict__ o, int N, int D,
                                                                  int M, float eps, int fm) {
    extern __shared__ __align__(16) float sm[];
    float* fQ = sm;                       // [64][kLd]
    float* S = fQ + kChunk * kLd;         // [d][m]
    float* z = S + kChunk * kLd;          // [64]
    float* den = z + kChunk;              // [64]
    const int64_t bh = blockIdx.y;
    const int t0 = blockIdx.x * kChunk;
    const int valid = min(kChunk, N - t0);
    const int E = D * M + D;
    const int t = threadIdx.x, tr = t >> 4, tc = t & 15, warp = t >> 5, lane = t & 31;
    load_tile(fQ, q + (bh * N + t0) * D, valid, D, fm);
    const float* st = total + bh * E;
    load_state(S, st, D, M, false);
    for (int idx = t; idx < kChunk; idx += blockDim.x) z[idx] = idx < D ? st[D * M + idx] : 0.f;
    __syncthreads();
    for (int i = warp; i < kChunk; i += kThreads / 32) {
        float s2 = 0.f;
        for (int cc = lane; cc < D; cc += 32) s2 = fmaf(fQ[i * kLd + cc], z[cc], s2);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) s2 += __shfl_xor_sync(0xffffffffu, s2, off);
        if (lane == 0) den[i] = s2 + eps;
    }
    __syncthreads();
    float acc[4][4];
    zero4x4(acc);
    mm4<false, true>(acc, fQ, S, 0, kChunk, tr, tc);
    T* oc = o + (bh * N + t0) * M;
#pragma unroll
    for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y) {
            const int i = 4 * tr + x, m = col_of(true, tc, y);
            if (i < valid && m < M) oc[(int64_t)i * M + m] = from_f<T>(acc[x][y] / den[i]);
        }
}

template <typename T>
cudaError_t simt_noncausal_impl(const void* q, const void* k, const void* v, void* o,
                                int64_t BH, int N, int D, int M, float eps, int fm, int nsplit,
                                float* partials, float* total, cudaStream_t st) {
    const int nchunks = (N + kChunk - 1) / kChunk;
    const int per_split = ((nchunks + nsplit - 1) / nsplit) * kChunk;
    const bool tiled = D <= kChunk && M <= kChunk;
    const size_t sm1 = tiled ? sizeof(float) * (2 * (size_t)kChunk * kLd)
                             : sizeof(float) * (size_t)kChunk * (D + M);
    const size_t sm3 = tiled ? sizeof(float) * (2 * (size_t)kChunk * kLd + 2 * kChunk)
                             : sizeof(float) * ((size_t)kChunk * (D + 1) + (size_t)D * M + D +
                                                kChunk);
    cudaError_t err;
    if (tiled) {
        if ((err = cudaFuncSetAttribute(nc_partial_tiled_kernel<T>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm1)) ||
            (err = cudaFuncSetAttribute(nc_apply_tiled_kernel<T>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm3)))
            return err;
        nc_partial_tiled_kernel<T><<<dim3(nsplit, (unsigned)BH), kThreads, sm1, st>>>(
            (const T*)k, (const T*)v, partials, N, D, M, per_split, fm);
    } else {
        if ((err = cudaFuncSetAttribute(nc_partial_kernel<T>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm1)) ||
            (err = cudaFuncSetAttribute(nc_apply_kernel<T>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm3)))
            return err;
        nc_partial_kernel<T><<<dim3(nsplit, (unsigned)BH), kThreads, sm1, st>>>(
            (const T*)k, (const T*)v, partials, N, D, M, per_split, fm);
    }
    const int E = D * M + D;
    const int64_t tot = BH * (int64_t)E;
    nc_reduce_kernel<<<(unsigned)((tot + 255) / 256), 256, 0, st>>>(partials, total, BH, nsplit,
                                                                     E);
    if (tiled)
        nc_apply_tiled_kernel<T><<<dim3(nchunks, (unsigned)BH), kThreads, sm3, st>>>(
            (const T*)q, total, (T*)o, N, D, M, eps, fm);
    else
        nc_apply_kernel<T><<<dim3(nchunks, (unsigned)BH), kThreads, sm3, st>>>(
            (const T*)q, total, (T*)o, N, D, M, eps, fm);
    return cudaPeekAtLastError();
}

// grid (ceil(rows / 64), ceil(R / 64)): positive random features of 64 rows x
// 64 features, out[i, r] = exp(w_r . x_i - |x_i|^2 / 2 - shift) * scale with
// scale = 1 / sqrt(R); the projections register-tiled, D <= kLdX - 4.
template <typename T, int kLdX>
__global__ void __launch_bounds__(kThreads) random_features_kernel(
    const T* __restrict__ x, const T* __restrict__ W, T* __restrict__ out, int64_t rows, int D,
    int R, float shift, float scale) {
    extern __shared__ __align__(16) float sm[];
    float* X = sm;                        // [64][kLdX]: the block's rows of x
    float* Wt = X + kChunk * kLdX;        // [64][kLdX]: the block's rows of W
    float* hsq = Wt + kChunk * kLdX;      // [64]: |x_i|^2 / 2
    const int64_t r0 = (int64_t)blockIdx.x * kChunk;
    const int f0 = blockIdx.y * kChunk;
    const int vrows = (int)min((int64_t)kChunk, rows - r0);
    const int vfeat = min(kChunk, R - f0);
    const int Dp = (D + 3) & ~3;          // the sums run to a multiple of 4 over zeros
    const int t = threadIdx.x, tr = t >> 4, tc = t & 15, warp = t >> 5, lane = t & 31;
#pragma unroll 4
    for (int idx = t; idx < kChunk * Dp; idx += kThreads) {
        const int r = idx / Dp, d = idx - r * Dp;
        X[r * kLdX + d] = (r < vrows && d < D) ? to_f(x[(r0 + r) * D + d]) : 0.f;
        Wt[r * kLdX + d] = (r < vfeat && d < D) ? to_f(W[(int64_t)(f0 + r) * D + d]) : 0.f;
    }
    __syncthreads();
    for (int i = warp; i < kChunk; i += kThreads / 32) {
        float s2 = 0.f;
        for (int d = lane; d < Dp; d += 32) s2 = fmaf(X[i * kLdX + d], X[i * kLdX + d], s2);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) s2 += __shfl_xor_sync(0xffffffffu, s2, off);
        if (lane == 0) hsq[i] = 0.5f * s2;
    }
    __syncthreads();
    float acc[4][4];
    zero4x4(acc);
    mm4<false, false, kLdX, kLdX>(acc, X, Wt, 0, Dp, tr, tc);
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int y = 0; y < 4; ++y) {
            const int i = 4 * tr + a, c = col_of(false, tc, y);
            if (i < vrows && c < vfeat)
                out[(r0 + i) * R + f0 + c] = from_f<T>(expf(acc[a][y] - hsq[i] - shift) * scale);
        }
}

template <typename T, int kLdX>
cudaError_t random_features_impl(const void* x, const void* W, void* out, int64_t rows, int D,
                                 int R, float shift, cudaStream_t st) {
    const size_t smem = sizeof(float) * (2 * (size_t)kChunk * kLdX + kChunk);
    cudaError_t err;
    if ((err = cudaFuncSetAttribute(random_features_kernel<T, kLdX>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)))
        return err;
    const dim3 grid((unsigned)((rows + kChunk - 1) / kChunk), (unsigned)((R + kChunk - 1) / kChunk));
    random_features_kernel<T, kLdX><<<grid, kThreads, smem, st>>>(
        (const T*)x, (const T*)W, (T*)out, rows, D, R, shift, 1.f / sqrtf((float)R));
    return cudaPeekAtLastError();
}

template <typename T, bool kCausal, int kFm>
cudaError_t simt_bwd_launch(const void* q, const void* k, const void* v, const void* dout,
                            void* dq, void* dk, void* dv, int64_t BH, int N, int D, int M,
                            float eps, float* states, float* rstates, float* rowg,
                            cudaStream_t st) {
    const int nchunks = (N + kChunk - 1) / kChunk;
    dim3 grid(nchunks, (unsigned)BH);
    const size_t sm1 = sizeof(float) * (2 * (size_t)kChunk * kLd);
    const size_t sm2 = sizeof(float) * (6 * (size_t)kChunk * kLd + 4 * kChunk);
    const size_t sm3 = sizeof(float) * (8 * (size_t)kChunk * kLd + 3 * kChunk);
    cudaError_t err;
    if ((err = cudaFuncSetAttribute(chunk_state_tiled_kernel<T>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm1)) ||
        (err = cudaFuncSetAttribute(bwd_rows_kernel<T, kCausal, kFm>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm2)) ||
        (err = cudaFuncSetAttribute(bwd_grad_kernel<T, kCausal, kFm>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm3)))
        return err;
    const int E = D * M + D;
    const int64_t total = BH * (int64_t)E;
    const unsigned sgrid = (unsigned)((total + 255) / 256);
    chunk_state_tiled_kernel<T><<<grid, kThreads, sm1, st>>>((const T*)k, (const T*)v, states, N, D,
                                                             M, kFm);
    if (kCausal)
        chunk_scan_kernel<<<sgrid, 256, 0, st>>>(states, nullptr, nullptr, nullptr, nullptr, BH,
                                                 nchunks, D, M);
    else
        chunk_total_kernel<<<sgrid, 256, 0, st>>>(states, BH, nchunks, E);
    bwd_rows_kernel<T, kCausal, kFm><<<grid, kThreads, sm2, st>>>(
        (const T*)q, (const T*)k, (const T*)v, (const T*)dout, states, rowg, rstates, N, D, M, eps);
    if (kCausal)
        chunk_rscan_kernel<<<sgrid, 256, 0, st>>>(rstates, BH, nchunks, E);
    else
        chunk_total_kernel<<<sgrid, 256, 0, st>>>(rstates, BH, nchunks, E);
    bwd_grad_kernel<T, kCausal, kFm><<<grid, kThreads, sm3, st>>>(
        (const T*)q, (const T*)k, (const T*)v, states, rstates, rowg, (T*)dq, (T*)dk, (T*)dv, N, D,
        M);
    return cudaPeekAtLastError();
}

// The feature map is a compile-time parameter of the backward kernels: taken at
// run time it cost the gradient pass about 20 %.
template <typename T, bool kCausal>
cudaError_t simt_bwd_impl(const void* q, const void* k, const void* v, const void* dout, void* dq,
                          void* dk, void* dv, int64_t BH, int N, int D, int M, float eps, int fm,
                          float* states, float* rstates, float* rowg, cudaStream_t st) {
    if (fm == kPhiIdentity)
        return simt_bwd_launch<T, kCausal, kPhiIdentity>(q, k, v, dout, dq, dk, dv, BH, N, D, M,
                                                         eps, states, rstates, rowg, st);
    return simt_bwd_launch<T, kCausal, kPhiElu1>(q, k, v, dout, dq, dk, dv, BH, N, D, M, eps,
                                                 states, rstates, rowg, st);
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
                        int64_t BH, int N, int D, int M, float eps, int fm, const float* S0,
                        const float* z0, float* S_out, float* z_out, void* scratch,
                        cudaStream_t st) {
    float* states = (float*)scratch;
    if (dt == LA_F32)
        return simt_causal_impl<float>(q, k, v, o, BH, N, D, M, eps, fm, S0, z0, S_out, z_out,
                                       states, st);
    return simt_causal_impl<__nv_bfloat16>(q, k, v, o, BH, N, D, M, eps, fm, S0, z0, S_out, z_out,
                                           states, st);
}

cudaError_t simt_noncausal(const void* q, const void* k, const void* v, void* o, la_dtype dt,
                           int64_t BH, int N, int D, int M, float eps, int fm, void* scratch,
                           cudaStream_t st) {
    const int nsplit = simt_noncausal_splits(BH, N);
    float* partials = (float*)scratch;
    float* total = partials + (size_t)BH * nsplit * (size_t)(D * M + D);
    if (dt == LA_F32)
        return simt_noncausal_impl<float>(q, k, v, o, BH, N, D, M, eps, fm, nsplit, partials,
                                          total, st);
    return simt_noncausal_impl<__nv_bfloat16>(q, k, v, o, BH, N, D, M, eps, fm, nsplit, partials,
                                              total, st);
}

cudaError_t bwd_prefix_states(float* states, bool causal, int64_t BH, int nchunks, int D, int M,
                              cudaStream_t st) {
    const int E = D * M + D;
    const unsigned sgrid = (unsigned)((BH * (int64_t)E + 255) / 256);
    if (causal)
        chunk_scan_kernel<<<sgrid, 256, 0, st>>>(states, nullptr, nullptr, nullptr, nullptr, BH,
                                                 nchunks, D, M);
    else
        chunk_total_kernel<<<sgrid, 256, 0, st>>>(states, BH, nchunks, E);
    return cudaPeekAtLastError();
}

cudaError_t bwd_reverse_sums(float* rstates, bool causal, int64_t BH, int nchunks, int E,
                             cudaStream_t st) {
    const unsigned sgrid = (unsigned)((BH * (int64_t)E + 255) / 256);
    if (causal)
        chunk_rscan_kernel<<<sgrid, 256, 0, st>>>(rstates, BH, nchunks, E);
    else
        chunk_total_kernel<<<sgrid, 256, 0, st>>>(rstates, BH, nchunks, E);
    return cudaPeekAtLastError();
}

size_t simt_bwd_workspace(int64_t BH, int N, int D, int M) {
    const int nchunks = (N + kChunk - 1) / kChunk;
    return sizeof(float) * ((size_t)2 * BH * nchunks * (size_t)(D * M + D) +
                            (size_t)BH * N * (size_t)(M + 1));
}

cudaError_t simt_bwd(const void* q, const void* k, const void* v, const void* dout, void* dq,
                     void* dk, void* dv, la_dtype dt, bool causal, int64_t BH, int N, int D, int M,
                     float eps, int fm, void* scratch, cudaStream_t st) {
    const int nchunks = (N + kChunk - 1) / kChunk;
    float* states = (float*)scratch;
    float* rstates = states + (size_t)BH * nchunks * (size_t)(D * M + D);
    float* rowg = rstates + (size_t)BH * nchunks * (size_t)(D * M + D);
    if (dt == LA_F32)
        return causal ? simt_bwd_impl<float, true>(q, k, v, dout, dq, dk, dv, BH, N, D, M, eps, fm,
                                                   states, rstates, rowg, st)
                      : simt_bwd_impl<float, false>(q, k, v, dout, dq, dk, dv, BH, N, D, M, eps, fm,
                                                    states, rstates, rowg, st);
    return causal ? simt_bwd_impl<__nv_bfloat16, true>(q, k, v, dout, dq, dk, dv, BH, N, D, M, eps,
                                                       fm, states, rstates, rowg, st)
                  : simt_bwd_impl<__nv_bfloat16, false>(q, k, v, dout, dq, dk, dv, BH, N, D, M,
                                                        eps, fm, states, rstates, rowg, st);
}

cudaError_t simt_random_features(const void* x, const void* W, void* out, la_dtype dt,
                                 int64_t rows, int D, int R, float shift, cudaStream_t st) {
    if (dt == LA_F32)
        return D <= 64 ? random_features_impl<float, 68>(x, W, out, rows, D, R, shift, st)
                       : random_features_impl<float, 132>(x, W, out, rows, D, R, shift, st);
    return D <= 64 ? random_features_impl<__nv_bfloat16, 68>(x, W, out, rows, D, R, shift, st)
                   : random_features_impl<__nv_bfloat16, 132>(x, W, out, rows, D, R, shift, st);
}

}  // namespace la
