/*
 * linattn.h — C ABI of the GB300 (sm_103a) kernels for kernelized linear
 * attention with the feature map phi(x) = elu(x) + 1.
 *
 * Definitions this library computes (all per (b, h) head, rows i = 1..N):
 *
 *   phi(x)  = x + 1 for x > 0, exp(x) for x <= 0, element-wise
 *             ("Why Replace Attention? The Softmax Bottleneck and the Path to
 *              Linear Time", section 5.3; "Transformers Are RNNs: Linear
 *              Attention", "Factor the Similarity Kernel").
 *   non-causal:  S = sum_j phi(k_j) v_j^T,  z = sum_j phi(k_j),
 *                o_i = phi(q_i)^T S / (phi(q_i)^T z + eps)
 *             ("Transformers Are RNNs: Linear Attention", "Reassociate the
 *              Products"; "Why Replace Attention? ...", section 6.2;
 *              "Linear Attention" research-hub note, the matrix form
 *              O = (phi(Q)(phi(K)^T V)) / (phi(Q)(phi(K)^T 1))).
 *   causal:      S_i = sum_{j<=i} phi(k_j) v_j^T,  z_i = sum_{j<=i} phi(k_j),
 *                o_i = phi(q_i)^T S_i / (phi(q_i)^T z_i + eps)
 *             ("Why Replace Attention? ...", sections 7.1-7.2;
 *              "[Paper Review] Transformers are RNNs ...", section 3.4).
 *   decode step: S <- S + phi(k) v^T, z <- z + phi(k), then
 *                o = phi(q)^T S / (phi(q)^T z + eps)   (update, then read)
 *             ("Transformers Are RNNs: Linear Attention", "Turn Causal
 *              Attention into a Recurrence"; "Why Replace Attention? ...",
 *              section 7.2, steps 1-4).
 *
 * eps is added once to the scalar denominator (the pages ask for an epsilon
 * without fixing its value or place; 1e-6 is the customary value).
 *
 * Conventions shared by every entry point:
 *  - Tensors are contiguous, row-major [B, H, N, D] with D innermost
 *    (decode: [B, H, D]). q and k have Dk columns, v and o have Dv columns.
 *    o has the input dtype. S is [B, H, Dk, Dv] float32 (row = feature index,
 *    column = value index) and z is [B, H, Dk] float32.
 *  - All pointers except the host-side `bytes` out-parameter are DEVICE
 *    pointers owned by the caller. The library allocates no memory and keeps
 *    no global state; per-call scratch lives in the caller's workspace.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; 0 = legacy default
 *    stream). Argument errors are reported synchronously by the return
 *    value and nothing is launched. A launch failure returns LA_ERR_CUDA.
 *    A bounded device-side wait that expires sets the workspace status word;
 *    la_query_status() reports it as LA_ERR_TIMEOUT.
 *  - No C++ exception crosses this boundary.
 */
#ifndef LINATTN_H
#define LINATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / CUstream. */
typedef struct CUstream_st* la_stream_t;

typedef enum { LA_F32 = 0, LA_BF16 = 1 } la_dtype;

typedef enum {
    LA_OK = 0,
    LA_ERR_INVALID_ARG = 1,  /* null pointer, non-positive size, bad dtype/op     */
    LA_ERR_UNSUPPORTED = 2,  /* valid but not implemented (e.g. Dk > 128)         */
    LA_ERR_WORKSPACE = 3,    /* workspace missing, too small or misaligned        */
    LA_ERR_CUDA = 4,         /* a CUDA runtime call or kernel launch failed       */
    LA_ERR_TIMEOUT = 5       /* a bounded device-side wait expired (see status)   */
} la_status;

typedef enum {
    LA_OP_NONCAUSAL = 0,
    LA_OP_CAUSAL = 1,
    LA_OP_DECODE = 2,
    LA_OP_CAUSAL_BWD = 3,
    LA_OP_NONCAUSAL_BWD = 4,
    LA_OP_LAYER_DECODE = 5
} la_op;

/*
 * The feature map phi the kernels apply to q and k. The method leaves phi free
 * ("Why Replace Attention? The Softmax Bottleneck and the Path to Linear Time",
 * section 4.5: any map into a feature space of its own width). LA_PHI_ELU1 is
 * elu(x) + 1, the map of every entry without a `phi` argument; LA_PHI_IDENTITY
 * applies none, for features the caller has already computed (for example with
 * la_positive_random_features), whose width is then Dk. Features should be
 * non-negative so that the denominators stay positive; nothing checks it.
 */
typedef enum { LA_PHI_ELU1 = 0, LA_PHI_IDENTITY = 1 } la_phi;

/* Human-readable name of a status code (static string, never NULL). */
const char* la_status_string(la_status s);

/* Library ABI version, (major << 16) | minor. */
uint32_t la_version(void);

/*
 * Workspace bytes needed by `op` for this shape and dtype (0 for
 * LA_OP_DECODE, which needs none). `bytes` is a HOST pointer. The workspace
 * must be 256-byte aligned and, before its first use, prepared once with
 * la_workspace_init(); afterwards the library keeps it consistent across
 * calls. A workspace may be reused by any later call on the same stream;
 * calls that overlap in time must use distinct workspaces.
 */
la_status la_workspace_size(la_op op, int B, int H, int N, int Dk, int Dv, la_dtype dt,
                            size_t* bytes);

/*
 * Number of kernel launches one call of `op` makes for this shape and dtype
 * (host-only query; `launches` is a HOST pointer). Useful for stream and
 * graph planning and for counting launches in a timed region.
 */
la_status la_launch_count(la_op op, int B, int H, int N, int Dk, int Dv, la_dtype dt,
                          int* launches);

/*
 * Prepares a workspace (async on stream): zero-fills all `workspace_bytes`
 * bytes, then sets the header (its first 256 bytes) to no error, launch
 * counters at zero and the default wait limit. Needed once per workspace, and
 * again after a call was abandoned mid-flight (a killed process, a reset
 * device). Calls then keep the workspace consistent: the causal tensor-core
 * path publishes per-CTA sums in the body as words tagged with a launch
 * counter kept in the header, so the body must not be written by anything
 * else between init and the calls that use it.
 */
la_status la_workspace_init(void* workspace, size_t workspace_bytes, la_stream_t stream);

/*
 * Non-causal forward: o_i = phi(q_i)^T S / (phi(q_i)^T z + eps) with
 * S = sum_j phi(k_j) v_j^T and z = sum_j phi(k_j) over all j of the head.
 * q, k: [B,H,N,Dk]; v, o: [B,H,N,Dv]; dtype dt for all four.
 * Supported: LA_F32 with 1 <= Dk, Dv <= 128; LA_BF16 with the same range
 * (Dk = Dv in {64, 128} use the tensor-core path).
 */
la_status la_noncausal_fwd(const void* q, const void* k, const void* v, void* o,
                           int B, int H, int N, int Dk, int Dv, la_dtype dt, float eps,
                           void* workspace, size_t workspace_bytes, la_stream_t stream);

/*
 * Causal forward: o_i = phi(q_i)^T S_i / (phi(q_i)^T z_i + eps) with the
 * inclusive prefix sums S_i, z_i. Shapes and dtypes as la_noncausal_fwd.
 * S_out [B,H,Dk,Dv] and z_out [B,H,Dk] (float32, nullable) receive the final
 * state S_N, z_N, so that la_decode_step can continue the sequence.
 * bf16 with Dk = Dv = 64 runs one fused tensor-core launch; bf16 with
 * Dk = Dv = 128 three (run sums, a seed scan over them, the output pass);
 * other shapes and fp32 run fp32 arithmetic on the CUDA cores.
 */
la_status la_causal_fwd(const void* q, const void* k, const void* v, void* o,
                        int B, int H, int N, int Dk, int Dv, la_dtype dt, float eps,
                        float* S_out, float* z_out,
                        void* workspace, size_t workspace_bytes, la_stream_t stream);

/*
 * Causal backward: given dout = dL/do for the causal forward o of (q, k, v),
 * writes dq = dL/dq, dk = dL/dk, dv = dL/dv (same layouts and dtype as q, k, v).
 * With dnum_i = dout_i / den_i and dden_i = -(dout_i . o_i) / den_i, the
 * gradients are dphi(q_i) = S_i dnum_i + z_i dden_i (a forward prefix sum) and
 * dphi(k_j) = R_j v_j + r_j, dv_j = R_j^T phi(k_j) with R_j = sum_{i>=j}
 * phi(q_i) dnum_i^T, r_j = sum_{i>=j} phi(q_i) dden_i (a reverse one), so no
 * S_i is stored ("Transformers Are RNNs: Linear Attention", "Turn Causal
 * Attention into a Recurrence", on cumulative-sum gradients); then
 * dq = dphi(q) phi'(q) with phi'(x) = 1 for x > 0, e^x for x <= 0.
 *  - bf16 with Dk = Dv = 64: tensor-core products (bf16 operands, fp32
 *    accumulation); otherwise fp32 arithmetic. Dk, Dv <= 64 (larger:
 *    LA_ERR_UNSUPPORTED).
 *  - workspace: la_workspace_size(LA_OP_CAUSAL_BWD, ...) bytes, initialised once
 *    with la_workspace_init.
 */
la_status la_causal_bwd(const void* q, const void* k, const void* v, const void* dout,
                        void* dq, void* dk, void* dv, int B, int H, int N, int Dk, int Dv,
                        la_dtype dt, float eps, void* workspace, size_t workspace_bytes,
                        la_stream_t stream);

/*
 * Non-causal backward: the same gradients for the non-causal forward
 * o_i = phi(q_i)^T S / (phi(q_i)^T z + eps), where S, z and the reverse sums
 * R = sum_i phi(q_i) dnum_i^T, r = sum_i phi(q_i) dden_i run over the whole
 * sequence: dphi(q_i) = S dnum_i + z dden_i, dphi(k_j) = R v_j + r,
 * dv_j = R^T phi(k_j) ("Transformers Are RNNs: Linear Attention", the
 * associativity rewrite that shares S and z among all queries).
 *  - bf16 with Dk = Dv = 64: tensor-core products (bf16 operands, fp32
 *    accumulation); otherwise fp32 arithmetic. Dk, Dv <= 64 (larger:
 *    LA_ERR_UNSUPPORTED).
 *  - workspace: la_workspace_size(LA_OP_NONCAUSAL_BWD, ...) bytes, initialised
 *    once with la_workspace_init.
 */
la_status la_noncausal_bwd(const void* q, const void* k, const void* v, const void* dout,
                           void* dq, void* dk, void* dv, int B, int H, int N, int Dk, int Dv,
                           la_dtype dt, float eps, void* workspace, size_t workspace_bytes,
                           la_stream_t stream);

/*
 * Causal forward that continues from a given state: the recurrence starts at
 * S_0 = S0, z_0 = z0 instead of zero, so that o_i = phi(q_i)^T S_i /
 * (phi(q_i)^T z_i + eps) with S_i = S0 + sum_{j<=i} phi(k_j) v_j^T and
 * z_i = z0 + sum_{j<=i} phi(k_j). A long sequence processed in pieces (the
 * prefill of a prompt in parts, or a prompt extended after decode steps) gives
 * the result of one call on the whole sequence, up to fp32 rounding, when each
 * piece starts from the previous piece's S_out, z_out ("Transformers Are RNNs:
 * Linear Attention", "Turn Causal Attention into a Recurrence": the running
 * state is all that is carried forward).
 *  - S0 [B,H,Dk,Dv] and z0 [B,H,Dk]: float32 device pointers, 16-byte aligned,
 *    both given or both null (null: start from zero, as la_causal_fwd). They
 *    must not overlap S_out or z_out (LA_ERR_INVALID_ARG): other CTAs may still
 *    read the initial state while the final state is written.
 *  - Everything else as la_causal_fwd (same workspace size).
 */
la_status la_causal_fwd_state(const void* q, const void* k, const void* v, void* o,
                              int B, int H, int N, int Dk, int Dv, la_dtype dt, float eps,
                              const float* S0, const float* z0, float* S_out, float* z_out,
                              void* workspace, size_t workspace_bytes, la_stream_t stream);

/*
 * Causal forward for callers that cannot allocate device memory: a plugin
 * host that passes only input and output buffers, a real-time process that
 * forbids device allocation once it runs, or code whose memory belongs to
 * another framework's allocator. The paper has no counterpart; this is a
 * property of the library. It computes exactly what la_causal_fwd computes
 * (same arguments, minus the workspace) and allocates nothing: its scratch is
 * one fixed 16 MiB array in device memory that belongs to this library, held
 * by every GPU that loads it until the process exits.
 *  - The first call on a device looks up that array's device address and
 *    initialises its header on `stream`; make that first call before any
 *    stream capture.
 *  - Shapes whose scratch would exceed 16 MiB return LA_ERR_WORKSPACE and
 *    launch nothing. bf16 with Dk = Dv = 64 needs two tagged state sums per
 *    CTA (about 10 MB on a 152-SM GPU) whatever the shape, so it always fits.
 *    bf16 with Dk = Dv = 128 keeps two 66 KB states per CTA range, which fit
 *    up to 127 chunks of 128 tokens in all (B*H*ceil(N/128) <= 127). The fp32
 *    path keeps one fp32 state per 64-token chunk: at Dk = Dv = 64 it fits
 *    B*H*ceil(N/64) <= 1008.
 *  - All calls share the one array, which keeps the last call's contents:
 *    calls that overlap on the GPU (different streams, or concurrent host
 *    threads without ordering) race on it and must be serialised by the caller.
 *    A bf16 call that follows an fp32 call on the same device first clears the
 *    part of the array it reads (cudaMemsetAsync on `stream`), so the fp32
 *    path's per-chunk states are never taken for the bf16 path's tagged sums.
 *  - The array used is the current device's: `stream` (unless it is a default
 *    stream) and every pointer must belong to that device, else
 *    LA_ERR_INVALID_ARG (checked with cudaStreamGetDevice and
 *    cudaPointerGetAttributes before any launch).
 *  - Device-side wait timeouts are recorded in the array's header:
 *    la_noalloc_query_status reads and clears that status.
 */
la_status la_causal_fwd_noalloc(const void* q, const void* k, const void* v, void* o,
                                int B, int H, int N, int Dk, int Dv, la_dtype dt, float eps,
                                float* S_out, float* z_out, la_stream_t stream);

/*
 * Status of the la_causal_fwd_noalloc calls on the current device, as
 * la_query_status gives it for a workspace: synchronises `stream`, returns the
 * first device-side error recorded since the last query (LA_ERR_TIMEOUT when
 * a bounded wait ran out and the output is incomplete) and clears it; LA_OK
 * when none was recorded or no call has run on this device yet. No
 * counterpart in the paper: it reports on the library's own array.
 */
la_status la_noalloc_query_status(la_stream_t stream);

/*
 * Wait limit of the la_causal_fwd_noalloc calls on the current device, in
 * microseconds (0 restores the default of 2 s), and a test hook: hold_loads
 * != 0 makes the tensor-core path withhold its input loads so that its waits
 * run out (used to test failure detection without a GPU fault; 0 in normal
 * use). Written into the array's header by a one-thread kernel on `stream`,
 * so it applies to the calls queued after it. No counterpart in the paper.
 */
la_status la_noalloc_set_wait_limit(unsigned int max_spin_us, int hold_loads, la_stream_t stream);

/*
 * Causal forward on HOST buffers: q, k, v, o are host pointers in the layout of
 * la_causal_fwd ([B,H,N,D], dtype dt), S_out / z_out device pointers (nullable),
 * as in la_causal_fwd. The heads are processed in groups (a quarter of them
 * each, the last quarter split into all but four heads and four, so that
 * little work is left after the last copy in) that
 * stream through two device staging buffers, so that copying a group in,
 * computing the previous one and copying the one before out overlap (separate
 * copy engines for the two directions). Each group is an la_causal_fwd call on
 * its slice of heads (heads are independent; the result equals la_causal_fwd's
 * up to the order of fp32 additions across CTAs). Host buffers should be
 * page-locked (cudaHostAlloc / cudaHostRegister): with pageable memory the
 * copies are still correct but do not overlap.
 *  - staging: device memory of at least la_host_staging_size() bytes, 256-byte
 *    aligned, owned by the caller; workspace as for la_causal_fwd at (B, H, N).
 *  - The call is asynchronous on `stream`: it starts after the work already
 *    queued there and `stream` waits for the last output copy. On first use on
 *    a device it creates two streams and eight events for that device (no device
 *    memory), kept until the process exits; concurrent calls on one device are
 *    serialised while they enqueue.
 *  - Returns LA_ERR_WORKSPACE if the staging buffer is missing, misaligned or
 *    too small, and otherwise what la_causal_fwd returns for a group.
 */
la_status la_host_staging_size(int B, int H, int N, int Dk, int Dv, la_dtype dt, size_t* bytes);

la_status la_causal_fwd_host(const void* q, const void* k, const void* v, void* o,
                             int B, int H, int N, int Dk, int Dv, la_dtype dt, float eps,
                             float* S_out, float* z_out, void* staging, size_t staging_bytes,
                             void* workspace, size_t workspace_bytes, la_stream_t stream);

/*
 * One recurrent decode step for B*H independent heads, in place:
 * S <- S + phi(k) v^T, z <- z + phi(k), o = phi(q)^T S / (phi(q)^T z + eps).
 * q, k: [B,H,Dk]; v, o: [B,H,Dv] in dtype dt; S: [B,H,Dk,Dv] and z: [B,H,Dk]
 * float32, read and written. A fresh sequence starts from S = 0, z = 0
 * (caller zero-fills). Needs no workspace. S must be 16-byte aligned.
 */
la_status la_decode_step(const void* q, const void* k, const void* v, void* o,
                         float* S, float* z, int B, int H, int Dk, int Dv, la_dtype dt,
                         float eps, la_stream_t stream);

/*
 * The entries above with the feature map as an argument (LA_ERR_INVALID_ARG for
 * any other value). Same shapes, dtypes, workspaces, paths and errors as the
 * entry of the same name without `_phi`; la_causal_fwd_phi also takes the
 * optional initial state of la_causal_fwd_state. The backward entries multiply
 * by the map's derivative: min(phi(x), 1) for elu + 1, 1 for the identity.
 */
la_status la_noncausal_fwd_phi(const void* q, const void* k, const void* v, void* o,
                               int B, int H, int N, int Dk, int Dv, la_dtype dt, la_phi phi,
                               float eps, void* workspace, size_t workspace_bytes,
                               la_stream_t stream);
la_status la_causal_fwd_phi(const void* q, const void* k, const void* v, void* o,
                            int B, int H, int N, int Dk, int Dv, la_dtype dt, la_phi phi,
                            float eps, const float* S0, const float* z0, float* S_out,
                            float* z_out, void* workspace, size_t workspace_bytes,
                            la_stream_t stream);
la_status la_decode_step_phi(const void* q, const void* k, const void* v, void* o,
                             float* S, float* z, int B, int H, int Dk, int Dv, la_dtype dt,
                             la_phi phi, float eps, la_stream_t stream);
la_status la_causal_bwd_phi(const void* q, const void* k, const void* v, const void* dout,
                            void* dq, void* dk, void* dv, int B, int H, int N, int Dk, int Dv,
                            la_dtype dt, la_phi phi, float eps, void* workspace,
                            size_t workspace_bytes, la_stream_t stream);
la_status la_noncausal_bwd_phi(const void* q, const void* k, const void* v, const void* dout,
                               void* dq, void* dk, void* dv, int B, int H, int N, int Dk, int Dv,
                               la_dtype dt, la_phi phi, float eps, void* workspace,
                               size_t workspace_bytes, la_stream_t stream);

/*
 * Positive random features: out[i, r] = exp(w_r . x_i - |x_i|^2 / 2 - shift)
 * / sqrt(R) for the rows w_r of W. With the entries of W drawn from N(0, 1)
 * (by the caller), E[phi(x) . phi(y)] = exp(x . y): an unbiased estimate of
 * the exponential (softmax) kernel, the positive random features the
 * research-hub "Linear Attention" page names ("Key math / How it works").
 * `shift` is subtracted in every exponent against overflow; one shift for all
 * keys of a head, or any per query row, cancels in the attention output.
 *  - x: [rows, D], W: [R, D], out: [rows, R], all dtype dt, device pointers,
 *    16-byte aligned; fp32 arithmetic. 1 <= D <= 128, 1 <= R <= 65535 * 64.
 *  - The result feeds the *_phi entries with LA_PHI_IDENTITY and Dk = R.
 *  - Needs no workspace; asynchronous on `stream`.
 */
la_status la_positive_random_features(const void* x, const void* W, void* out, int64_t rows,
                                      int D, int R, la_dtype dt, float shift,
                                      la_stream_t stream);

/*
 * One decode step of a linear-attention layer for B sequences (d_model = H D):
 * [q | k | v] = x Wqkv; per head h the recurrent step S <- S + phi(k_h) v_h^T,
 * z <- z + phi(k_h), o_h = phi(q_h)^T S / (phi(q_h)^T z + eps) (elu + 1);
 * y = [o_1 | ... | o_H] Wo ("Why Replace Attention? The Softmax Bottleneck and
 * the Path to Linear Time", section 7.2, steps 1-4: k and v computed from the
 * token's hidden state, then the update and the read).
 *  - x: [B, d_model]; Wqkv: [d_model, 3 H D] (columns h D .. h D + D - 1 are
 *    head h of q, then of k, then of v); Wo: [H D, d_model]; y: [B, d_model];
 *    all row-major, dtype dt, device pointers, 16-byte aligned.
 *  - S: [B, H, D, D], z: [B, H, D] float32, read and written in place.
 *  - workspace: la_workspace_size(LA_OP_LAYER_DECODE, B, H, 1, D, D, dt, ...)
 *    bytes (a header and the projection buffers), 256-byte aligned, zeroed
 *    once by la_workspace_init; la_query_status reports a projection whose
 *    bounded waits ran out.
 *  - The projections are this library's products with fp32 accumulation
 *    (tcgen05 tensor cores for bf16 when d_model is a multiple of 8, fp32 FMA
 *    otherwise); the step between them is its decode kernel, reading q, k, v
 *    in place in the projection. The three launches go to `stream`;
 *    la_launch_count gives 3.
 */
la_status la_layer_decode_step(const void* x, const void* Wqkv, const void* Wo, void* y,
                               float* S, float* z, int B, int H, int D, la_dtype dt, float eps,
                               void* workspace, size_t workspace_bytes, la_stream_t stream);

/*
 * Synchronises `stream`, then reads and clears the workspace status word.
 * Returns LA_OK, LA_ERR_TIMEOUT (a bounded wait expired in an earlier call
 * that used this workspace) or LA_ERR_CUDA.
 */
la_status la_query_status(void* workspace, la_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* LINATTN_H */
