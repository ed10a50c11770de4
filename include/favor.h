/*
 * favor.h -- C ABI of the FAVOR+ forward-attention library for one GB300 (sm_103a).
 *
 * FAVOR+ (Rethinking Attention with Performers, §2.2-2.4 and App. B Alg. 1)
 * replaces the L x L softmax attention matrix by random features:
 *
 *   positive features (Lemma 1, Eq. 7):  phi_r(x) = m^-1/2 exp(omega_r . x - ||x||^2 / 2)
 *   ReLU features (§4.4, App. A.4):      phi_r(x) = m^-1/2 max(omega_r . x, 0)
 *
 * with x = s*q for queries and y = s*k for keys (s = data_scale; §2.3 after
 * Eq. 6 moves the sqrt(d) temperature into the inputs, s = d^-1/4 reproduces
 * exp(q.k / sqrt(d))).  Attention is then the reordered product of Eq. 4:
 *
 *   bidirectional:  S = Phi_K^T V, z = Phi_K^T 1,  out_i = phi(q_i)^T S / phi(q_i)^T z
 *   causal (App. B.1, Eq. 11): the same with S_i, z_i summed over keys j <= i.
 *
 * All tensors are contiguous row-major device buffers of the handle's dtype:
 *   q, k, x: [B, H, L, d]    v, out: [B, H, L, dv]    phi: [B, H, L, m]
 * The caller owns them.  Every call only enqueues work on `stream` (a
 * cudaStream_t passed as void*, NULL = legacy default stream) and returns;
 * launch errors are returned, execution errors appear at the caller's next
 * synchronisation, as usual in CUDA.  All argument checks happen on the host
 * before anything is launched; nothing traps on the device.
 *
 * A handle owns device copies of omega, per-head constants and a workspace
 * sized at creation for max_B and max_L.  Calls on one handle must not overlap
 * in time on the device (they share the workspace); use one handle per
 * concurrent stream.  A handle belongs to the device that was current at
 * favor_create; call it with that device current.
 */
#ifndef FAVOR_H
#define FAVOR_H

#if defined(__GNUC__)
#define FAVOR_API __attribute__((visibility("default")))
#else
#define FAVOR_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FAVOR_OK = 0,
    FAVOR_ERR_INVALID_ARG = 1,   /* null pointer, non-positive size, size above the handle's maximum */
    FAVOR_ERR_UNSUPPORTED = 2,   /* shape or enum value this library does not implement */
    FAVOR_ERR_NOMEM = 3,         /* device or host allocation failed in favor_create */
    FAVOR_ERR_CUDA = 4           /* a CUDA runtime call or kernel launch failed */
} favor_status;

/* Feature map f in Eq. 5 of Rethinking Attention with Performers.  The last
 * two have l = 2 functions per projection row: omega has m/2 rows and the map
 * has m features. */
typedef enum {
    FAVOR_KERNEL_SOFTMAX_POS = 0,  /* positive random features for the softmax kernel (Lemma 1) */
    FAVOR_KERNEL_RELU = 1,         /* generalized attention with f = ReLU (§4.4, App. A.4) */
    FAVOR_KERNEL_SOFTMAX_HYP = 2,  /* hyperbolic positive features SM^hyp+ (Lemma 1, second form):
                                      (2M)^-1/2 exp(-||x||^2/2) (exp(omega x), exp(-omega x)), M = m/2 */
    FAVOR_KERNEL_SOFTMAX_TRIG = 3  /* trigonometric features SM^trig (§2.3): M^-1/2 exp(||x||^2/2)
                                      (sin(omega x), cos(omega x)), M = m/2; features of either sign */
} favor_kernel;

/* Storage type of q, k, v, out, x and phi.  Arithmetic: F32 computes in fp32
 * throughout; BF16 rounds the features to bf16 for the tensor-core
 * contractions and accumulates in fp32. */
typedef enum {
    FAVOR_DTYPE_F32 = 0,
    FAVOR_DTYPE_BF16 = 1
} favor_dtype;

typedef struct favor_handle_s* favor_handle;

/*
 * favor_create -- build a handle for H heads with m features of width d and
 * values of width dv.
 *
 *   omega_host  host float array [H, m, d], row r of head h is omega_r
 *               (Eq. 5; drawn by the caller, e.g. orthogonal blocks as in §2.4
 *               and App. B.2 (1), or rows of length sqrt(d) for the
 *               regularized kernel SMREG of §2.3).  [H, m/2, d] for the
 *               hyperbolic and trigonometric kinds (m features from m/2
 *               rows).  Copied synchronously; the caller may free it on
 *               return.  The BF16 dtype rounds omega to bf16 (nearest even)
 *               for the tensor-core projection.
 *   data_scale  s > 0: features are taken of s*q and s*k.
 *   max_B, max_L  upper bounds for later calls; they size the workspace.
 *
 * Supported: d, dv in {16, 32, 64, 128}; m a multiple of 16 in [16, 256];
 * H >= 1.  The hyperbolic kind runs every call the positive kind runs (on the
 * rows [omega; -omega]).  The trigonometric kind runs on the rows
 * [omega; omega] (sin on the first m/2 features, cos on the others): its
 * forward calls take the tensor-core kernels for bf16 with d = dv = 64 and
 * m = 256 (features rounded to bf16 there, so a row's rounding error grows
 * with its cancellation) and the CUDA cores otherwise; the plain feature map
 * stays on the CUDA cores.  Its key features carry exp(||s k||^2/2) unshifted, so keys with
 * ||s k||^2 above about 170 overflow fp32; its denominators can be zero or
 * negative (the instability §2.3 describes), and a zero one gives a zero row
 * as for ReLU.  It has no backward and no handle-free call
 * (FAVOR_ERR_UNSUPPORTED).  Anything else gives FAVOR_ERR_UNSUPPORTED (enum values out of
 * range: FAVOR_ERR_INVALID_ARG).  Fails with FAVOR_ERR_NOMEM if device memory
 * runs out, FAVOR_ERR_CUDA if no device is usable.  *out is set to NULL on
 * any failure.
 */
FAVOR_API favor_status favor_create(favor_handle* out, int H, int m, int d, int dv,
                          favor_kernel kind, favor_dtype dtype,
                          const float* omega_host, float data_scale,
                          int max_B, int max_L);

/*
 * favor_feature_map -- phi = feature map of s*x, exactly as defined above
 * (Lemma 1 with the m^-1/2 factor and the -||x||^2/2 term, or the ReLU form),
 * with no stabilising shift.  x [B,H,L,d] -> phi [B,H,L,m], both of the
 * handle's dtype; phi is only written.  1 <= B <= max_B, 1 <= L <= max_L.
 * (Positive features overflow to inf only when omega_r . x - ||x||^2/2 > 88,
 * which needs ||omega_r||^2 > 176.)
 */
FAVOR_API favor_status favor_feature_map(favor_handle h, const void* x, void* phi,
                               int B, int L, void* stream);

/*
 * favor_attn_bidir -- bidirectional FAVOR+ attention (Eq. 4; Alg. 1 with
 * isBidirectional): out_i = phi(q_i)^T S / phi(q_i)^T z over all L keys of
 * the same (b, h).  q, k [B,H,L,d], v [B,H,L,dv] are read; out [B,H,L,dv] is
 * only written.  A row whose denominator is exactly 0 (possible only with
 * ReLU features) is written as zeros.  Shifts that cancel between numerator
 * and denominator are applied for range safety (a per-query-row shift and a
 * per-head key shift); they do not change the result beyond rounding.
 */
FAVOR_API favor_status favor_attn_bidir(favor_handle h, const void* q, const void* k,
                              const void* v, void* out, int B, int L, void* stream);

/*
 * favor_attn_causal -- unidirectional FAVOR+ attention (App. B.1, Eq. 11):
 * out_i = phi(q_i)^T S_i / phi(q_i)^T z_i with S_i, z_i summed over keys
 * j <= i (the diagonal included, as tril in Eq. 2).  Same layouts, ownership
 * and zero-denominator rule as favor_attn_bidir.  No L x L matrix and no
 * per-token prefix tensor is built.
 */
FAVOR_API favor_status favor_attn_causal(favor_handle h, const void* q, const void* k,
                               const void* v, void* out, int B, int L, void* stream);

/*
 * Stateful calls: the key/value summary carried across calls for decoding,
 * chunked prefill and cross attention (the RNN form of causal linear
 * attention: App. B.1 Eq. 11 of Rethinking Attention with Performers with the
 * prefix sum started at a given state; the recurrence of Exploring Linear
 * Attention, "Autoregressive Generation"; causal Random Feature Attention).
 *
 * A state is a caller-owned DEVICE float array [B, H, m, dv+1], row-major,
 * 16-byte aligned (else FAVOR_ERR_INVALID_ARG):
 * row r of head (b, h) is (S_r0 .. S_r,dv-1, z_r) with
 *     S = e^-kappa_h * sum_j phi(k_j) v_j^T,   z = e^-kappa_h * sum_j phi(k_j)
 * over the keys it summarises (phi the plain feature map above, m^-1/2
 * included; kappa_h = max(0, max_r ||omega_r||^2/2 - 60) is the handle's
 * per-head key shift, 0 unless some ||omega_r||^2 > 120, which keeps every
 * term finite).  A zero-filled array is the empty state.  Calls on one
 * handle must not overlap; a state may be shared by calls on one stream.
 */

/*
 * favor_kv_state -- state += the summary of keys k [B,H,L,d] and values v
 * [B,H,L,dv] (App. B Alg. 1, Buf1 = K'^T [V 1]).  Accumulates, so a long
 * sequence may be summarised chunk by chunk; fixed-order sums (bitwise
 * repeatable).  1 <= B <= max_B, 1 <= L <= max_L.
 */
FAVOR_API favor_status favor_kv_state(favor_handle h, const void* k, const void* v, float* state,
                                      int B, int L, void* stream);

/*
 * favor_attn_from_state -- out_i = phi(q_i)^T S / phi(q_i)^T z for queries q
 * [B,H,L,d] against a given state (Eq. 4 with the key side given): with
 * favor_kv_state of another sequence this is cross attention (query and key
 * lengths differ).  out [B,H,L,dv] is only written; zero-denominator rows are
 * 0.  1 <= B <= max_B, 1 <= L <= max_L.
 */
FAVOR_API favor_status favor_attn_from_state(favor_handle h, const void* q, const float* state, void* out,
                                             int B, int L, void* stream);

/*
 * favor_attn_causal_step -- causal attention over T new tokens q, k [B,H,T,d],
 * v [B,H,T,dv] that follow the keys summarised by state:
 *     out_t = phi(q_t)^T (S + sum_{j<=t} phi(k_j) v_j^T) / phi(q_t)^T (z + sum_{j<=t} phi(k_j)),
 * then state += the new tokens' summary.  Starting from a zero state and
 * calling it block after block gives favor_attn_causal of the whole sequence
 * (up to rounding).  Runs one CTA per (b, h) on the CUDA cores, tokens in
 * order: meant for decoding (T = 1) and short blocks; a long prefix is better
 * served by favor_attn_causal for its outputs and favor_kv_state for its
 * state.  1 <= B <= max_B, 1 <= T <= max_L.
 */
FAVOR_API favor_status favor_attn_causal_step(favor_handle h, const void* q, const void* k, const void* v,
                                              void* out, float* state, int B, int T, void* stream);

/*
 * favor_attn_causal_gated -- causal attention with a gated, decaying state
 * (RFA-Gate, Random Feature Attention §3.2).  The page describes the gate in
 * words: scalar gates g_t in [0, 1], computed by the model from the timestep's
 * input, decay the history of both the value state and the normalisation
 * state.  The reading implemented (the gate interpolates between history and
 * the current token):
 *     S_t = g_t S_{t-1} + (1 - g_t) phi(k_t) v_t^T,   z_t = g_t z_{t-1} + (1 - g_t) phi(k_t),
 *     out_t = phi(q_t)^T S_t / phi(q_t)^T z_t                (0 where the denominator is 0)
 *   gate   DEVICE float array [B,H,L] (fp32 whatever the dtype), caller-owned,
 *          read only; values outside [0, 1] are not checked.
 * Other arguments as favor_attn_causal.  Chunked: the ranges' states are
 * combined with the products of their gates.  Positive and ReLU features of
 * the bf16 d = dv = 64, m = 256 shape run on the tensor cores (each chunk's
 * gates scanned in log2, clamped below at 2^-126, the within-chunk decay
 * applied per element of the masked product); every other case on the CUDA
 * cores.  The gate pointer must stay valid until the call's work on the stream
 * is done.  Not combined with favor_set_relpos (FAVOR_ERR_UNSUPPORTED while it is set).
 *
 * favor_attn_causal_step_gated -- favor_attn_causal_step with the same gated
 * update; gate [B,H,T].
 */
FAVOR_API favor_status favor_attn_causal_gated(favor_handle h, const void* q, const void* k, const void* v,
                                               const float* gate, void* out, int B, int L, void* stream);
FAVOR_API favor_status favor_attn_causal_step_gated(favor_handle h, const void* q, const void* k, const void* v,
                                                    const float* gate, void* out, float* state, int B, int T,
                                                    void* stream);

/*
 * favor_set_relpos -- PermuteFormer relative position encoding (PermuteFormer:
 * Efficient Relative Position Encoding for Long Sequences, §PermuteFormer).
 * Query and key features at position i are transformed by r^i P_pi^i and
 * r^-i P_pi^i, P_pi the permutation matrix of pi ((P_pi phi)_a = phi_pi(a)),
 * so the similarity of query i and key j is r^(i-j) phi(q_i)^T P_pi^(j-i) phi(k_j):
 * it depends on i - j only.  Positions count from 0 within each call.
 *   perm  HOST int array [H, m]: row h is a permutation of 0..m-1 (NULL: the
 *         identity).  Stored as each permutation's cycles (O(H m) device
 *         memory); pi^i(a) is looked up from a's cycle, not precomputed per
 *         position.
 *   r     HOST float array [H], 0 < r <= 1 (NULL: 1).  Applies to causal calls
 *         (a state decayed by r per token); bidirectional calls use r = 1, as
 *         the page prescribes for bidirectional models.
 * Both NULL clears the setting.  While set, favor_attn_bidir and
 * favor_attn_causal apply it (on the CUDA cores); favor_feature_map still
 * returns the plain phi; the gated, state, step and backward calls fail with
 * FAVOR_ERR_UNSUPPORTED.  Synchronises the handle's device and allocates, like
 * favor_create; call it with no call of the handle in flight.
 * INVALID_ARG for a row that is not a permutation or an r outside (0, 1].
 */
FAVOR_API favor_status favor_set_relpos(favor_handle h, const int* perm, const float* r);

/*
 * favor_attn_bidir_backward / favor_attn_causal_backward -- gradients of
 * favor_attn_bidir / favor_attn_causal with respect to q, k and v.
 *
 * Rethinking Attention with Performers times the backward pass (§4.1, Fig. 3)
 * without printing its formulas; these calls return the exact derivative of
 * the forward (App. B Alg. 1 and App. B.1 Eq. 11), up to rounding: for a loss
 * with upstream gradient dO = dloss/dout,
 *     D_i = [dO_i / den_i, -(dO_i . out_i) / den_i]       (0 where den_i == 0)
 *     dphi(q_i) = G_i D_i,  G_i = sum over the keys row i sees of phi(k_j) [v_j 1]^T
 *     dphi(k_j) = H_j [v_j 1],  dv_j = H_j^T phi(k_j),
 *                 H_j = sum over the queries that see key j of phi(q_i) D_i^T
 * then through the feature map (x = s*q): positive features
 *     dq = s * ((dphi . phi) Omega - x sum_r (dphi . phi)_r),
 * ReLU features dq = s * m^-1/2 (dphi . [Omega x > 0]) Omega (the derivative of
 * max(u, 0) at u = 0 is taken as 0); likewise dk.
 *
 *   q, k, v    the forward's inputs, as passed to the forward call.
 *   dout       dO [B,H,L,dv].
 * The forward's output is not an argument: dO_i . out_i is computed inside,
 * in fp32, as phi(q_i) . (G_i applied to dO_i) / den_i, so a rounded copy of
 * out (e.g. bf16) cannot perturb the gradients.
 *   dq, dk     [B,H,L,d], dv [B,H,L,dv]: written, never read; must not alias
 *              any input.
 * All tensors are contiguous device arrays of the handle's dtype.  For bf16
 * with d = dv = 64 and m = 256 (positive, hyperbolic and ReLU features) and
 * 16-byte-aligned pointers both calls run on the tensor cores: bf16 operands
 * with fp32 accumulation, the key/value and query states and G entering as
 * bf16 pairs hi + lo; the causal call works in 128-token chunks (states of
 * the earlier and later chunks, masked products inside the chunk).  Otherwise
 * the arithmetic is fp32 on the CUDA cores.  Both use the forward's
 * cancelling shifts.  Same argument checks, asynchrony and one-call-per-handle
 * rule as the forward calls; the handle's workspace (allocated by
 * favor_create) is reused, nothing is allocated.
 */
FAVOR_API favor_status favor_attn_bidir_backward(favor_handle h, const void* q, const void* k, const void* v,
                                                 const void* dout, void* dq, void* dk, void* dv,
                                                 int B, int L, void* stream);
FAVOR_API favor_status favor_attn_causal_backward(favor_handle h, const void* q, const void* k, const void* v,
                                                  const void* dout, void* dq, void* dk, void* dv,
                                                  int B, int L, void* stream);

/*
 * favor_attn_bidir_noalloc -- favor_attn_bidir without a handle and without
 * any allocation.  The paper has no counterpart: this is an interface
 * convenience.  It serves callers that may not allocate device memory through
 * this library, e.g. a host framework whose caching allocator owns the device
 * memory, or a serving process that reserves the device memory up front.
 * favor_create allocates its workspace with cudaMalloc, so these callers
 * cannot make a handle.
 *
 *   omega       DEVICE float array [H, m, d] (caller-owned, read only), used
 *               as given (favor_create's bf16 rounding of omega is not
 *               applied); entries must be finite.  It must be 16-byte aligned
 *               memory of the current device (device or managed); anything
 *               else fails with FAVOR_ERR_INVALID_ARG before any launch.
 *   H, m, d, dv, kind, dtype, data_scale   as in favor_create, same limits.
 *   q, k, v, out, B, L, stream             as in favor_attn_bidir.
 *
 * Computes what favor_attn_bidir computes, on the CUDA-core kernels (fp32
 * arithmetic for both dtypes), with the same zero-denominator rule and
 * the same cancelling shifts (the per-head key shift is derived on the device
 * from omega).  Scratch is one fixed 16 MiB device array inside the library
 * (4,194,304 floats): calls need H (rounded up to 64) + 2*B*H*m*(dv+1) floats at
 * least, and larger sizes fail with FAVOR_ERR_UNSUPPORTED before anything is
 * launched; the work split is narrowed to fit.  No part of the array needs to
 * start at zero.  Every device has its own copy.  Its address is looked up
 * the first time the call runs on a device (cudaGetSymbolAddress, which may
 * load the library's device code there), and again the first time after the
 * device's context was made anew (e.g. after cudaDeviceReset); make that first
 * call before any stream capture begins.  Calls on one device share the array: two calls
 * that overlap in time on the device race and give wrong results, so order
 * them (one stream, or events).
 */
FAVOR_API favor_status favor_attn_bidir_noalloc(const float* omega, int H, int m, int d, int dv,
                                                favor_kernel kind, favor_dtype dtype, float data_scale,
                                                const void* q, const void* k, const void* v, void* out,
                                                int B, int L, void* stream);

/* favor_destroy -- free everything the handle owns (after synchronising its
 * device).  Accepts NULL. */
FAVOR_API favor_status favor_destroy(favor_handle h);

/* Name of a status code (static string). */
FAVOR_API const char* favor_status_str(favor_status s);

/* Text of the most recent failure in the calling thread (static buffer,
 * empty if none). */
FAVOR_API const char* favor_last_error(void);

/* Number of kernels this library has launched in this process (all handles,
 * all threads); a counter for measurement. */
FAVOR_API unsigned long long favor_launch_count(void);

/*
 * favor_device_error -- synchronise with the handle's device (a blocking copy)
 * and report its device-side error word in *code: 0 if every bounded wait in
 * the kernels completed, otherwise the code of the first wait that gave up
 * (the kernel then skipped the rest of its work and returned).  No
 * counterpart on the pages; it exists so that a stalled pipeline surfaces as
 * an error instead of a hang.
 */
FAVOR_API favor_status favor_device_error(favor_handle h, int* code);

/*
 * favor_check_bounded_wait -- exercise the failure path of the kernels'
 * bounded waits without faulting anything (no counterpart on the pages).
 * Enqueues on `stream` one single-thread kernel that waits on an mbarrier
 * phase nothing completes, with a limit of limit_cycles SM clock cycles
 * (1000 <= limit_cycles <= 2^24, else FAVOR_ERR_INVALID_ARG).  The wait gives
 * up, the kernel writes FAVOR_WAIT_CHECK_CODE to the handle's device error
 * word (unless an earlier failure already left its code there) and returns; the
 * context stays usable.  favor_device_error then reports the code.  The
 * handle's error word is not cleared afterwards: use a handle made for the
 * check.
 */
#define FAVOR_WAIT_CHECK_CODE 901
FAVOR_API favor_status favor_check_bounded_wait(favor_handle h, int limit_cycles, void* stream);

/*
 * Per-kernel timing for measurement (no counterpart on the pages).
 *
 * favor_profile_enable(h, 1) makes every later kernel launch through h record
 * a pair of CUDA events on the launching stream around the kernel;
 * favor_profile_read(h, slot, &ms, &n) synchronises those events and returns
 * the summed device time in milliseconds and the number of launches recorded
 * for one kernel slot since the last reset; favor_profile_enable(h, 0) stops
 * recording and favor_profile_reset(h) clears the totals.  Slots are numbered
 * 0 .. favor_profile_slots()-1 and named by favor_profile_name(slot).  Recording
 * allocates events lazily on the host thread that launches; errors come back
 * as FAVOR_ERR_CUDA.
 */
FAVOR_API favor_status favor_profile_enable(favor_handle h, int enable);
FAVOR_API favor_status favor_profile_reset(favor_handle h);
FAVOR_API favor_status favor_profile_read(favor_handle h, int slot, double* ms_total,
                                          unsigned long long* launches);
FAVOR_API int favor_profile_slots(void);
FAVOR_API const char* favor_profile_name(int slot);

#ifdef __cplusplus
}
#endif

#endif /* FAVOR_H */
