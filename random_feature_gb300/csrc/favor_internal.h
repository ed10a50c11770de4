// Internal declarations shared by the host API and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cstddef>
#include <cstdint>
#include <vector>

#include "../../include/favor.h"

namespace favor {

// Kernel slots for the optional per-kernel event timing.
enum ProfSlot {
    PROF_FEATURE_MAP = 0,
    PROF_STATE,         // per-segment key/value state (bidirectional partials, causal totals)
    PROF_COMBINE,       // fixed-order reduce / exclusive scan of segment states
    PROF_READOUT,       // bidirectional query readout
    PROF_CAUSAL,        // causal chunked attention
    PROF_BWD_QUERY,     // backward: query-side pass (dq, per-segment phi_q D^T sums)
    PROF_BWD_KEY,       // backward: key-side pass (dk, dv)
    PROF_NSLOTS
};

struct ProfEvent {
    int slot;
    cudaEvent_t a, b;
};

struct Profile {
    bool on = false;
    std::vector<ProfEvent> pending;   // recorded, not yet read
    std::vector<cudaEvent_t> spare;   // reusable events
    double ms[PROF_NSLOTS] = {};
    unsigned long long n[PROF_NSLOTS] = {};
};

// Everything a handle owns.  Device pointers unless noted.
struct Handle {
    int H, m, d, dv;
    favor_kernel kind;        // computation kind: SOFTMAX_POS, RELU or SOFTMAX_TRIG (HYP runs as POS)
    favor_kernel features;    // the kind the handle was created with
    favor_dtype dtype;
    float s;                  // data scale: x = s*q, y = s*k
    int max_B, max_L;
    int device;
    int num_sms;
    int cc_major;             // compute capability of the device
    int* dev_err;             // device error word: 0, or the code of the first bounded wait that gave up

    float* omega_f32;         // [H, m, d] (bf16-rounded values for the BF16 dtype)
    __nv_bfloat16* omega_bf16;// [H, m, d] (BF16 dtype only)
    float* kshift;            // [H] per-head key shift kappa_h (natural-log units)
    float* omega_wmax;        // [H] per head, a bound W_h >= max_r ||omega_r|| (query shift of the causal kernel)
    float* omega_sqnorm_half_host; // host [H]: max_r ||omega_r||^2 / 2

    float* ws_partial;        // [rows][m * (dv+1)] per-segment states (bidir partials / causal prefixes):
                              // row-major [m][dv+1] on the CUDA-core path, column-major [dv+1][m]
                              // on the tensor-core path (coalesced by feature)
    float* ws_state;          // [max_B*H][m][dv+1] reduced bidirectional states
    float* ws_partial2;       // like ws_partial (row-major): backward per-segment sums of phi~_q D^T
    float* ws_dstate;         // [max_B*H][m][dv+1] backward: reduced sum of phi~_q D^T (bidirectional)
    float* ws_rowstat;        // [max_B*H*max_L][4] backward (causal): per query (den~, row shift, dO . out, 0)
    size_t ws_partial_rows;   // capacity of ws_partial in (head, segment) rows
    float* ws_segdecay;       // [rows] per-segment products of a decaying causal state's factors
    // PermuteFormer relative positions (favor_set_relpos); null when unset.
    int* perm_cyc;            // [H*m] each head's permutation written cycle by cycle
    int4* perm_meta;          // [H*m] per feature: (cycle start, cycle length, place in the cycle, 0)
    float* relpos_r;          // [H] decay r of causal calls (null: 1)
    double* ws64;             // FP32 dtype: [rows][m][dv+1] float64 per-segment states
    double* ws64_state;       // FP32 dtype: [max_B*H][m][dv+1] float64 reduced bidirectional states
    void* ws_tc;              // tensor-core path scratch (bf16 operand copies), may be null
    void* ws_bimg;            // tensor-core backward: per head S (or dS) hi / lo images + z, may be null
    size_t ws_tc_bytes;
    Profile* prof;            // per-kernel timing (host object)
};

// Bracket one kernel launch with timing events when the handle's profiling is on.
struct ProfScope {
    const Handle& h;
    int slot;
    cudaStream_t st;
    cudaEvent_t b = nullptr;
    ProfScope(const Handle& hh, int sl, cudaStream_t s);
    ~ProfScope();
};

// Work split of a (B*H, L) call into per-head segments of whole 128-token tiles.
struct SegPlan {
    int tiles;        // ceil(L / 128)
    int seg_tiles;    // tiles per segment
    int n_seg;        // segments per head
    int cap;          // upper bound of n_seg for this BH and any L' <= L (sizes the workspace)
};

SegPlan plan_segments(int BH, int L, int num_sms);

// Bookkeeping shared by every launcher.
void count_launch(int n = 1);
// 16-byte alignment of a device pointer (asynchronous 16-byte copies need it).
inline bool is_aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
favor_status set_error(favor_status st, const char* fmt, ...);
favor_status check_launch(const char* what);

// The key-side shift is kappa_h = max(0, max_r ||omega_r||^2/2 - KSHIFT_HEADROOM): it
// bounds every key feature by exp(KSHIFT_HEADROOM) whatever the input, since
// omega.y - ||y||^2/2 = (||omega||^2 - ||y - omega||^2)/2 <= ||omega||^2/2.
constexpr float KSHIFT_HEADROOM = 60.0f;

// ---- generic SIMT kernels (any supported shape, fp32 or bf16 storage) ----
favor_status simt_feature_map(const Handle& h, const void* x, void* phi, int B, int L, cudaStream_t st);
favor_status simt_bidir(const Handle& h, const void* q, const void* k, const void* v, void* out,
                        int B, int L, cudaStream_t st);
favor_status simt_causal(const Handle& h, const void* q, const void* k, const void* v, void* out,
                         int B, int L, cudaStream_t st, const float* gate = nullptr);

// Optional position-dependent inputs of the CUDA-core segment kernels.
struct RelposArgs {
    const int* cyc = nullptr;      // PermuteFormer permutation cycles (null: identity)
    const int4* meta = nullptr;
    const float* gate = nullptr;   // RFA-Gate gates [B*H*L] (null: none)
    const float* rdec = nullptr;   // per-head decay r (null: 1)
    float* segdecay = nullptr;     // out: per-segment decay products (decaying causal calls)
};

// Per-segment key/value states of the CUDA-core path into h.ws_partial (row-major).
favor_status simt_state_partials(const Handle& h, const void* k, const void* v, int BH, int L, const SegPlan& p,
                                 cudaStream_t st);

// ---- backward (gradients of the bidirectional / causal call), CUDA cores ----
favor_status simt_bidir_backward(const Handle& h, const void* q, const void* k, const void* v, const void* dout,
                                 void* dq, void* dk, void* dv, int B, int L, cudaStream_t st);
favor_status simt_causal_backward(const Handle& h, const void* q, const void* k, const void* v, const void* dout,
                                  void* dq, void* dk, void* dv, int B, int L, cudaStream_t st);

// ---- stateful calls: public state [B*H][m][dv+1] fp32 (S | z), see favor.h ----
favor_status simt_kv_state(const Handle& h, const void* k, const void* v, float* state, int B, int L,
                           cudaStream_t st);
favor_status simt_attn_from_state(const Handle& h, const void* q, const float* state, void* out, int B, int L,
                                  cudaStream_t st);
favor_status simt_causal_step(const Handle& h, const void* q, const void* k, const void* v, void* out, float* state,
                              int B, int Tn, cudaStream_t st, const float* gate = nullptr);
favor_status tc_kv_state(const Handle& h, const void* k, const void* v, float* state, int B, int L, cudaStream_t st);
favor_status tc_attn_from_state(const Handle& h, const void* q, const float* state, void* out, int B, int L,
                                cudaStream_t st);

// ---- fp32 storage with float64 arithmetic (bidirectional and causal, positive / ReLU) ----
size_t f64_workspace_rows(int max_BH, int num_sms);
bool f64_supported(const Handle& h);
favor_status f64_bidir(const Handle& h, const void* q, const void* k, const void* v, void* out, int B, int L,
                       cudaStream_t st);
favor_status f64_causal(const Handle& h, const void* q, const void* k, const void* v, void* out, int B, int L,
                        cudaStream_t st);

// ---- bidirectional call on a fixed, statically sized device scratch array ----
// 16 MiB: enough for B*H*m*(dv+1)*(1 + n_seg) + H floats with n_seg >= 1 up to
// B*H = 63 at m = 256, dv = 128 (more heads at smaller m, dv).
constexpr size_t kFixedScratchFloats = (size_t)4 << 20;
size_t fixed_scratch_floats(int H, int BH, int m, int dv, int n_seg);
// proto: H, m, d, dv, kind, dtype, s, device, num_sms and omega_f32 (the
// caller's device omega) filled in; nothing else is read.
favor_status simt_bidir_fixed_scratch(const Handle& proto, const void* q, const void* k, const void* v,
                                      void* out, int B, int L, cudaStream_t st);

// ---- tensor-core (tcgen05) kernels: bf16, d = dv = 64, m = 256 ----
// One-thread kernel whose mbarrier wait has no arriver: it gives up after
// `limit` cycles and writes `code` to the handle's error word.
favor_status launch_wait_expiry(const Handle& h, long long limit, int code, cudaStream_t st);
bool tc_supported(const Handle& h);
favor_status tc_feature_map(const Handle& h, const void* x, void* phi, int B, int L, cudaStream_t st);
favor_status tc_bidir(const Handle& h, const void* q, const void* k, const void* v, void* out,
                      int B, int L, cudaStream_t st);
favor_status tc_causal(const Handle& h, const void* q, const void* k, const void* v, void* out,
                       int B, int L, cudaStream_t st);
// RFA-Gate causal call on the tensor cores (positive and ReLU kinds; gate [B*H, L] fp32).
favor_status tc_causal_gated(const Handle& h, const void* q, const void* k, const void* v, const float* gate,
                             void* out, int B, int L, cudaStream_t st);
// Tensor-core bidirectional backward (falls back to the CUDA-core one for unaligned pointers).
favor_status tc_bidir_backward(const Handle& h, const void* q, const void* k, const void* v, const void* dout,
                               void* dq, void* dk, void* dv, int B, int L, cudaStream_t st);
// Tensor-core causal backward, chunked (falls back to the CUDA-core one for unaligned pointers).
favor_status tc_causal_backward(const Handle& h, const void* q, const void* k, const void* v, const void* dout,
                                void* dq, void* dk, void* dv, int B, int L, cudaStream_t st);
size_t tc_bwd_image_bytes(size_t BH);

// ---- fixed-order combines of per-segment states (shared by both paths) ----
favor_status launch_reduce_segments(const Handle& h, int BH, int n_seg, cudaStream_t st);
favor_status launch_scan_segments(const Handle& h, int BH, int n_seg, cudaStream_t st);

}  // namespace favor
