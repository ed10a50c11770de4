// Host side of the C ABI: argument checks, handle lifetime, workspace, dispatch.
//
// Every check runs before anything is enqueued; a failing call launches nothing.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include "favor_internal.h"

namespace favor {

static std::atomic<unsigned long long> g_launches{0};
static thread_local char g_err[512] = "";

void count_launch(int n) { g_launches.fetch_add((unsigned long long)n, std::memory_order_relaxed); }

favor_status set_error(favor_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return st;
}

favor_status check_launch(const char* what) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return set_error(FAVOR_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
    return FAVOR_OK;
}

SegPlan plan_segments(int BH, int L, int num_sms) {
    SegPlan p;
    p.tiles = (L + 127) / 128;
    // Aim for about two independent segments per SM across all heads, but keep
    // segments at least 4 tiles long so the per-segment state write stays small
    // next to the segment's own traffic.
    long target = 2L * num_sms;
    int want = (int)((target + BH - 1) / BH);
    int max_seg = (p.tiles + 3) / 4;
    if (want > max_seg) want = max_seg;
    if (want < 1) want = 1;
    p.cap = want;   // n_seg <= want, and want does not decrease with L
    p.seg_tiles = (p.tiles + want - 1) / want;
    p.n_seg = (p.tiles + p.seg_tiles - 1) / p.seg_tiles;
    return p;
}

static cudaEvent_t take_event(Profile* p) {
    if (!p->spare.empty()) {
        cudaEvent_t e = p->spare.back();
        p->spare.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) { cudaGetLastError(); return nullptr; }
    return e;
}

ProfScope::ProfScope(const Handle& hh, int sl, cudaStream_t s) : h(hh), slot(sl), st(s) {
    if (!h.prof || !h.prof->on) return;
    cudaEvent_t a = take_event(h.prof);
    b = take_event(h.prof);
    if (!a || !b) { b = nullptr; return; }
    cudaEventRecord(a, st);
    h.prof->pending.push_back({slot, a, b});
}

ProfScope::~ProfScope() {
    if (b) cudaEventRecord(b, st);
}

static bool shape_ok(int x) { return x == 16 || x == 32 || x == 64 || x == 128; }

}  // namespace favor

using namespace favor;

extern "C" {

const char* favor_status_str(favor_status s) {
    switch (s) {
        case FAVOR_OK: return "FAVOR_OK";
        case FAVOR_ERR_INVALID_ARG: return "FAVOR_ERR_INVALID_ARG";
        case FAVOR_ERR_UNSUPPORTED: return "FAVOR_ERR_UNSUPPORTED";
        case FAVOR_ERR_NOMEM: return "FAVOR_ERR_NOMEM";
        case FAVOR_ERR_CUDA: return "FAVOR_ERR_CUDA";
    }
    return "FAVOR_ERR_UNKNOWN";
}

const char* favor_last_error(void) { return g_err; }

unsigned long long favor_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

static void free_handle(Handle* h) {
    if (!h) return;
    cudaFree(h->omega_f32);
    cudaFree(h->omega_bf16);
    cudaFree(h->kshift);
    cudaFree(h->omega_wmax);
    cudaFree(h->dev_err);
    cudaFree(h->ws_partial);
    cudaFree(h->ws_state);
    cudaFree(h->ws_partial2);
    cudaFree(h->ws_dstate);
    cudaFree(h->ws_rowstat);
    cudaFree(h->ws_segdecay);
    cudaFree(h->perm_cyc);
    cudaFree(h->perm_meta);
    cudaFree(h->relpos_r);
    cudaFree(h->ws64);
    cudaFree(h->ws64_state);
    cudaFree(h->ws_tc);
    cudaFree(h->ws_bimg);
    free(h->omega_sqnorm_half_host);
    if (h->prof) {
        for (auto& pe : h->prof->pending) { cudaEventDestroy(pe.a); cudaEventDestroy(pe.b); }
        for (auto e : h->prof->spare) cudaEventDestroy(e);
        delete h->prof;
    }
    delete h;
}

favor_status favor_create(favor_handle* out, int H, int m, int d, int dv, favor_kernel kind,
                          favor_dtype dtype, const float* omega_host, float data_scale,
                          int max_B, int max_L) {
    g_err[0] = 0;
    if (!out) return set_error(FAVOR_ERR_INVALID_ARG, "favor_create: out is NULL");
    *out = nullptr;
    if (!omega_host) return set_error(FAVOR_ERR_INVALID_ARG, "favor_create: omega_host is NULL");
    if (H < 1 || m < 1 || d < 1 || dv < 1 || max_B < 1 || max_L < 1)
        return set_error(FAVOR_ERR_INVALID_ARG, "favor_create: sizes must be >= 1 (H=%d m=%d d=%d dv=%d max_B=%d max_L=%d)",
                         H, m, d, dv, max_B, max_L);
    if (kind != FAVOR_KERNEL_SOFTMAX_POS && kind != FAVOR_KERNEL_RELU && kind != FAVOR_KERNEL_SOFTMAX_HYP &&
        kind != FAVOR_KERNEL_SOFTMAX_TRIG)
        return set_error(FAVOR_ERR_INVALID_ARG, "favor_create: unknown kernel kind %d", (int)kind);
    if (dtype != FAVOR_DTYPE_F32 && dtype != FAVOR_DTYPE_BF16)
        return set_error(FAVOR_ERR_INVALID_ARG, "favor_create: unknown dtype %d", (int)dtype);
    if (!(data_scale > 0.0f) || !std::isfinite(data_scale))
        return set_error(FAVOR_ERR_INVALID_ARG, "favor_create: data_scale must be finite and > 0");
    if (!shape_ok(d) || !shape_ok(dv))
        return set_error(FAVOR_ERR_UNSUPPORTED, "favor_create: d=%d dv=%d (supported: 16, 32, 64, 128)", d, dv);
    if (m % 16 != 0 || m < 16 || m > 256)
        return set_error(FAVOR_ERR_UNSUPPORTED, "favor_create: m=%d (supported: multiples of 16 in [16, 256])", m);
    if ((long long)max_B * H * (long long)max_L * (d > dv ? d : dv) > (1LL << 40))
        return set_error(FAVOR_ERR_UNSUPPORTED, "favor_create: max_B*H*max_L too large");

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return set_error(FAVOR_ERR_CUDA, "favor_create: no usable CUDA device");
    }
    Handle* h = new (std::nothrow) Handle();
    if (!h) return set_error(FAVOR_ERR_NOMEM, "favor_create: host allocation failed");
    std::memset(h, 0, sizeof(*h));
    h->prof = new (std::nothrow) Profile();
    if (!h->prof) { delete h; return set_error(FAVOR_ERR_NOMEM, "favor_create: host allocation failed"); }
    const bool two_fn = kind == FAVOR_KERNEL_SOFTMAX_HYP || kind == FAVOR_KERNEL_SOFTMAX_TRIG;
    h->H = H; h->m = m; h->d = d; h->dv = dv; h->dtype = dtype; h->features = kind;
    h->kind = kind == FAVOR_KERNEL_SOFTMAX_HYP ? FAVOR_KERNEL_SOFTMAX_POS : kind;
    h->s = data_scale; h->max_B = max_B; h->max_L = max_L; h->device = dev;
    cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (h->num_sms < 1) h->num_sms = 1;
    cudaDeviceGetAttribute(&h->cc_major, cudaDevAttrComputeCapabilityMajor, dev);

    const size_t n_om = (size_t)H * m * d;
    // The two-function kinds get m/2 rows per head and run on [omega; -omega]
    // (hyperbolic: exp(-omega.x) = exp((-omega).x)) or [omega; omega]
    // (trigonometric: sin on the first half, cos on the second).
    const size_t n_in = two_fn ? n_om / 2 : n_om;
    for (size_t i = 0; i < n_in; ++i) {
        if (!std::isfinite(omega_host[i])) {
            free_handle(h);
            return set_error(FAVOR_ERR_INVALID_ARG, "favor_create: omega has a non-finite entry at %zu", i);
        }
    }
    std::vector<float> om(n_om);
    if (!two_fn) {
        std::copy(omega_host, omega_host + n_om, om.begin());
    } else {
        const int M = m / 2;
        const float sign = kind == FAVOR_KERNEL_SOFTMAX_HYP ? -1.f : 1.f;
        for (int hh = 0; hh < H; ++hh)
            for (int r = 0; r < M; ++r)
                for (int c = 0; c < d; ++c) {
                    const float w = omega_host[((size_t)hh * M + r) * d + c];
                    om[((size_t)hh * m + r) * d + c] = w;
                    om[((size_t)hh * m + M + r) * d + c] = sign * w;
                }
    }
    std::vector<__nv_bfloat16> om_bf;
    if (dtype == FAVOR_DTYPE_BF16) {
        om_bf.resize(n_om);
        for (size_t i = 0; i < n_om; ++i) {
            om_bf[i] = __float2bfloat16_rn(om[i]);
            om[i] = __bfloat162float(om_bf[i]);   // the fp32 copy holds exactly what the MMA sees
        }
    }
    // Per-head key shift: kappa_h = max(0, max_r ||omega_r||^2/2 - headroom).
    std::vector<float> ks(H), wmax(H);
    h->omega_sqnorm_half_host = (float*)malloc(sizeof(float) * H);
    if (!h->omega_sqnorm_half_host) { free_handle(h); return set_error(FAVOR_ERR_NOMEM, "favor_create: host allocation failed"); }
    for (int hh = 0; hh < H; ++hh) {
        double mx = 0.0;
        for (int r = 0; r < m; ++r) {
            double acc = 0.0;
            for (int c = 0; c < d; ++c) {
                double w = om[((size_t)hh * m + r) * d + c];
                acc += w * w;
            }
            if (acc > mx) mx = acc;
        }
        h->omega_sqnorm_half_host[hh] = (float)(0.5 * mx);
        // largest row length, rounded up (its only use is an upper bound)
        wmax[hh] = (float)(std::sqrt(mx) * (1.0 + 1e-6));
        double k = 0.5 * mx - (double)KSHIFT_HEADROOM;
        ks[hh] = (float)(k > 0.0 && kind != FAVOR_KERNEL_SOFTMAX_TRIG ? k : 0.0);
    }

    // Workspace: per-(head, segment) states.  Both work splits stay within
    // 2*SMs + 2*B*H rows: the CUDA-core segments use at most
    // B*H*ceil(2*SMs/(B*H)) rows, the tensor-core ranges B*H*(ceil(SMs/(B*H))+1).
    size_t rows = 2 * (size_t)h->num_sms + 2 * (size_t)max_B * H;
    h->ws_partial_rows = rows;
    const size_t st_elems = (size_t)m * (dv + 1);

    cudaError_t e = cudaSuccess;
    if (e == cudaSuccess) e = cudaMalloc(&h->omega_f32, n_om * sizeof(float));
    if (e == cudaSuccess && dtype == FAVOR_DTYPE_BF16) e = cudaMalloc(&h->omega_bf16, n_om * sizeof(__nv_bfloat16));
    if (e == cudaSuccess) e = cudaMalloc(&h->kshift, H * sizeof(float));
    if (e == cudaSuccess) e = cudaMalloc(&h->omega_wmax, H * sizeof(float));
    if (e == cudaSuccess) e = cudaMalloc(&h->dev_err, sizeof(int));
    if (e == cudaSuccess) e = cudaMemset(h->dev_err, 0, sizeof(int));
    if (e == cudaSuccess) e = cudaMalloc(&h->ws_partial, rows * st_elems * sizeof(float));
    if (e == cudaSuccess) e = cudaMalloc(&h->ws_state, (size_t)max_B * H * st_elems * sizeof(float));
    // Backward: a second set of per-segment states, the reduced sum of
    // phi~_q D^T, and four floats per (head, query) for the causal key pass.
    if (e == cudaSuccess) e = cudaMalloc(&h->ws_partial2, rows * st_elems * sizeof(float));
    if (e == cudaSuccess) e = cudaMalloc(&h->ws_dstate, (size_t)max_B * H * st_elems * sizeof(float));
    if (e == cudaSuccess) e = cudaMalloc(&h->ws_rowstat, (size_t)max_B * H * (size_t)max_L * 4 * sizeof(float));
    if (e == cudaSuccess) e = cudaMalloc(&h->ws_segdecay, rows * sizeof(float));
    // fp32 storage: float64 per-segment and reduced states of the bidirectional and causal calls
    if (e == cudaSuccess && dtype == FAVOR_DTYPE_F32 && kind != FAVOR_KERNEL_SOFTMAX_TRIG) {
        e = cudaMalloc(&h->ws64, f64_workspace_rows(max_B * H, h->num_sms) * st_elems * sizeof(double));
        if (e == cudaSuccess) e = cudaMalloc(&h->ws64_state, (size_t)max_B * H * st_elems * sizeof(double));
    }
    if (e != cudaSuccess) {
        favor_status st = (e == cudaErrorMemoryAllocation) ? FAVOR_ERR_NOMEM : FAVOR_ERR_CUDA;
        set_error(st, "favor_create: cudaMalloc: %s", cudaGetErrorString(e));
        cudaGetLastError();
        free_handle(h);
        return st;
    }
    if (tc_supported(*h)) {
        // bf16 copies of the reduced states in the tensor-core operand layout.
        // bf16 readout operand images, two [m][64] blocks per (batch, head); the
        // second block holds z~ in column 0 and zeros elsewhere, so it starts zeroed.
        h->ws_tc_bytes = (size_t)max_B * H * 128 * m * sizeof(__nv_bfloat16);
        e = cudaMalloc(&h->ws_tc, h->ws_tc_bytes);
        if (e == cudaSuccess) e = cudaMemset(h->ws_tc, 0, h->ws_tc_bytes);
        // backward: per head S~ (then dS~) as bf16 hi / lo operand images + the fp32 z column
        if (e == cudaSuccess) e = cudaMalloc(&h->ws_bimg, tc_bwd_image_bytes((size_t)max_B * H));
        if (e != cudaSuccess) {
            favor_status st = (e == cudaErrorMemoryAllocation) ? FAVOR_ERR_NOMEM : FAVOR_ERR_CUDA;
            set_error(st, "favor_create: cudaMalloc: %s", cudaGetErrorString(e));
            cudaGetLastError();
            free_handle(h);
            return st;
        }
    }
    e = cudaMemcpy(h->omega_f32, om.data(), n_om * sizeof(float), cudaMemcpyHostToDevice);
    if (e == cudaSuccess && dtype == FAVOR_DTYPE_BF16)
        e = cudaMemcpy(h->omega_bf16, om_bf.data(), n_om * sizeof(__nv_bfloat16), cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemcpy(h->kshift, ks.data(), H * sizeof(float), cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemcpy(h->omega_wmax, wmax.data(), H * sizeof(float), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) {
        set_error(FAVOR_ERR_CUDA, "favor_create: cudaMemcpy: %s", cudaGetErrorString(e));
        cudaGetLastError();
        free_handle(h);
        return FAVOR_ERR_CUDA;
    }
    *out = reinterpret_cast<favor_handle>(h);
    return FAVOR_OK;
}

favor_status favor_destroy(favor_handle hd) {
    if (!hd) return FAVOR_OK;
    Handle* h = reinterpret_cast<Handle*>(hd);
    const int dev = h->device;
    int cur = 0;
    cudaGetDevice(&cur);
    if (cur != dev) cudaSetDevice(dev);
    cudaDeviceSynchronize();
    free_handle(h);
    if (cur != dev) cudaSetDevice(cur);
    cudaGetLastError();
    return FAVOR_OK;
}

static bool relpos_on(const Handle& h) { return h.perm_cyc != nullptr || h.relpos_r != nullptr; }

static favor_status check_call(const char* fn, favor_handle hd, int B, int L) {
    g_err[0] = 0;
    if (!hd) return set_error(FAVOR_ERR_INVALID_ARG, "%s: handle is NULL", fn);
    const Handle* h = reinterpret_cast<const Handle*>(hd);
    if (B < 1 || L < 1) return set_error(FAVOR_ERR_INVALID_ARG, "%s: B=%d L=%d must be >= 1", fn, B, L);
    if (B > h->max_B || L > h->max_L)
        return set_error(FAVOR_ERR_INVALID_ARG, "%s: B=%d L=%d exceed the handle's max_B=%d max_L=%d",
                         fn, B, L, h->max_B, h->max_L);
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess || cur != h->device) {
        cudaGetLastError();
        return set_error(FAVOR_ERR_INVALID_ARG, "%s: current device %d is not the handle's device %d",
                         fn, cur, h->device);
    }
    return FAVOR_OK;
}

favor_status favor_feature_map(favor_handle hd, const void* x, void* phi, int B, int L, void* stream) {
    favor_status st = check_call("favor_feature_map", hd, B, L);
    if (st != FAVOR_OK) return st;
    if (!x || !phi) return set_error(FAVOR_ERR_INVALID_ARG, "favor_feature_map: null tensor pointer");
    const Handle& h = *reinterpret_cast<const Handle*>(hd);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (tc_supported(h)) return tc_feature_map(h, x, phi, B, L, s);
    return simt_feature_map(h, x, phi, B, L, s);
}

favor_status favor_attn_bidir(favor_handle hd, const void* q, const void* k, const void* v, void* out,
                              int B, int L, void* stream) {
    favor_status st = check_call("favor_attn_bidir", hd, B, L);
    if (st != FAVOR_OK) return st;
    if (!q || !k || !v || !out) return set_error(FAVOR_ERR_INVALID_ARG, "favor_attn_bidir: null tensor pointer");
    const Handle& h = *reinterpret_cast<const Handle*>(hd);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (tc_supported(h) && !relpos_on(h)) return tc_bidir(h, q, k, v, out, B, L, s);
    if (f64_supported(h) && !relpos_on(h)) return f64_bidir(h, q, k, v, out, B, L, s);
    return simt_bidir(h, q, k, v, out, B, L, s);
}

favor_status favor_attn_causal(favor_handle hd, const void* q, const void* k, const void* v, void* out,
                               int B, int L, void* stream) {
    favor_status st = check_call("favor_attn_causal", hd, B, L);
    if (st != FAVOR_OK) return st;
    if (!q || !k || !v || !out) return set_error(FAVOR_ERR_INVALID_ARG, "favor_attn_causal: null tensor pointer");
    const Handle& h = *reinterpret_cast<const Handle*>(hd);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (tc_supported(h) && !relpos_on(h)) return tc_causal(h, q, k, v, out, B, L, s);
    if (f64_supported(h) && !relpos_on(h)) return f64_causal(h, q, k, v, out, B, L, s);
    return simt_causal(h, q, k, v, out, B, L, s);
}

favor_status favor_attn_causal_gated(favor_handle hd, const void* q, const void* k, const void* v, const float* gate,
                                     void* out, int B, int L, void* stream) {
    favor_status st = check_call("favor_attn_causal_gated", hd, B, L);
    if (st != FAVOR_OK) return st;
    if (!q || !k || !v || !gate || !out)
        return set_error(FAVOR_ERR_INVALID_ARG, "favor_attn_causal_gated: null pointer");
    const Handle& h = *reinterpret_cast<const Handle*>(hd);
    if (relpos_on(h)) return set_error(FAVOR_ERR_UNSUPPORTED, "favor_attn_causal_gated: relative positions are set");
    if (tc_supported(h) && (h.kind == FAVOR_KERNEL_SOFTMAX_POS || h.kind == FAVOR_KERNEL_RELU))
        return tc_causal_gated(h, q, k, v, gate, out, B, L, reinterpret_cast<cudaStream_t>(stream));
    return simt_causal(h, q, k, v, out, B, L, reinterpret_cast<cudaStream_t>(stream), gate);
}

favor_status favor_set_relpos(favor_handle hd, const int* perm, const float* r) {
    g_err[0] = 0;
    if (!hd) return set_error(FAVOR_ERR_INVALID_ARG, "favor_set_relpos: handle is NULL");
    Handle* h = reinterpret_cast<Handle*>(hd);
    const int H = h->H, m = h->m;
    if (r) {
        for (int i = 0; i < H; ++i)
            if (!(r[i] > 0.f && r[i] <= 1.f))
                return set_error(FAVOR_ERR_INVALID_ARG, "favor_set_relpos: r[%d] = %g is not in (0, 1]", i, (double)r[i]);
    }
    // cycle tables: per head, the permutation written cycle by cycle, and per
    // feature (start of its cycle, cycle length, its place in the cycle)
    std::vector<int> cyc, meta;
    if (perm) {
        cyc.resize((size_t)H * m);
        meta.resize((size_t)H * m * 4);
        std::vector<char> seen(m);
        for (int hh = 0; hh < H; ++hh) {
            const int* p = perm + (size_t)hh * m;
            std::fill(seen.begin(), seen.end(), 0);
            for (int a = 0; a < m; ++a) {
                if (p[a] < 0 || p[a] >= m || seen[p[a]])
                    return set_error(FAVOR_ERR_INVALID_ARG, "favor_set_relpos: row %d is not a permutation of 0..%d",
                                     hh, m - 1);
                seen[p[a]] = 1;
            }
            std::fill(seen.begin(), seen.end(), 0);
            int fill = 0;
            for (int a0 = 0; a0 < m; ++a0) {
                if (seen[a0]) continue;
                const int start = fill;
                int a = a0;
                do {
                    seen[a] = 1;
                    cyc[(size_t)hh * m + fill++] = a;
                    a = p[a];
                } while (a != a0);
                const int len = fill - start;
                for (int t = 0; t < len; ++t) {
                    int* mt = &meta[((size_t)hh * m + cyc[(size_t)hh * m + start + t]) * 4];
                    mt[0] = start; mt[1] = len; mt[2] = t; mt[3] = 0;
                }
            }
        }
    }
    int cur = -1;
    cudaGetDevice(&cur);
    if (cur != h->device) cudaSetDevice(h->device);
    cudaDeviceSynchronize();   // no call of this handle may still read the old tables
    cudaFree(h->perm_cyc);
    cudaFree(h->perm_meta);
    cudaFree(h->relpos_r);
    h->perm_cyc = nullptr;
    h->perm_meta = nullptr;
    h->relpos_r = nullptr;
    cudaError_t e = cudaSuccess;
    if (perm) {
        e = cudaMalloc(&h->perm_cyc, cyc.size() * sizeof(int));
        if (e == cudaSuccess) e = cudaMalloc(&h->perm_meta, meta.size() * sizeof(int));
        if (e == cudaSuccess) e = cudaMemcpy(h->perm_cyc, cyc.data(), cyc.size() * sizeof(int), cudaMemcpyHostToDevice);
        if (e == cudaSuccess)
            e = cudaMemcpy(h->perm_meta, meta.data(), meta.size() * sizeof(int), cudaMemcpyHostToDevice);
    }
    if (e == cudaSuccess && r) {
        e = cudaMalloc(&h->relpos_r, H * sizeof(float));
        if (e == cudaSuccess) e = cudaMemcpy(h->relpos_r, r, H * sizeof(float), cudaMemcpyHostToDevice);
    }
    if (cur != h->device) cudaSetDevice(cur);
    if (e != cudaSuccess) {
        cudaGetLastError();
        cudaFree(h->perm_cyc); cudaFree(h->perm_meta); cudaFree(h->relpos_r);
        h->perm_cyc = nullptr; h->perm_meta = nullptr; h->relpos_r = nullptr;
        return set_error(e == cudaErrorMemoryAllocation ? FAVOR_ERR_NOMEM : FAVOR_ERR_CUDA, "favor_set_relpos: %s",
                         cudaGetErrorString(e));
    }
    return FAVOR_OK;
}

favor_status favor_attn_bidir_noalloc(const float* omega, int H, int m, int d, int dv, favor_kernel kind,
                                      favor_dtype dtype, float data_scale, const void* q, const void* k,
                                      const void* v, void* out, int B, int L, void* stream) {
    const char* fn = "favor_attn_bidir_noalloc";
    g_err[0] = 0;
    if (!omega || !q || !k || !v || !out) return set_error(FAVOR_ERR_INVALID_ARG, "%s: null pointer", fn);
    if (H < 1 || m < 1 || d < 1 || dv < 1 || B < 1 || L < 1)
        return set_error(FAVOR_ERR_INVALID_ARG, "%s: sizes must be >= 1 (H=%d m=%d d=%d dv=%d B=%d L=%d)", fn, H, m,
                         d, dv, B, L);
    if (kind == FAVOR_KERNEL_SOFTMAX_HYP || kind == FAVOR_KERNEL_SOFTMAX_TRIG)
        return set_error(FAVOR_ERR_UNSUPPORTED, "%s: kind %d needs a handle (favor_create)", fn, (int)kind);
    if (kind != FAVOR_KERNEL_SOFTMAX_POS && kind != FAVOR_KERNEL_RELU)
        return set_error(FAVOR_ERR_INVALID_ARG, "%s: unknown kernel kind %d", fn, (int)kind);
    if (dtype != FAVOR_DTYPE_F32 && dtype != FAVOR_DTYPE_BF16)
        return set_error(FAVOR_ERR_INVALID_ARG, "%s: unknown dtype %d", fn, (int)dtype);
    if (!(data_scale > 0.0f) || !std::isfinite(data_scale))
        return set_error(FAVOR_ERR_INVALID_ARG, "%s: data_scale must be finite and > 0", fn);
    if (!shape_ok(d) || !shape_ok(dv))
        return set_error(FAVOR_ERR_UNSUPPORTED, "%s: d=%d dv=%d (supported: 16, 32, 64, 128)", fn, d, dv);
    if (m % 16 != 0 || m < 16 || m > 256)
        return set_error(FAVOR_ERR_UNSUPPORTED, "%s: m=%d (supported: multiples of 16 in [16, 256])", fn, m);
    if ((long long)B * H * (long long)L * (d > dv ? d : dv) > (1LL << 40))
        return set_error(FAVOR_ERR_UNSUPPORTED, "%s: B*H*L too large", fn);
    const long long BH = (long long)B * H;
    if (BH > (1 << 20) || fixed_scratch_floats(H, (int)BH, m, dv, 1) > kFixedScratchFloats)
        return set_error(FAVOR_ERR_UNSUPPORTED,
                         "%s: B*H*m*(dv+1) = %lld needs more than the fixed scratch of %zu floats (at most %zu "
                         "per state copy, two copies)", fn, BH * m * (dv + 1), kFixedScratchFloats,
                         (kFixedScratchFloats - ((size_t)H + 63) / 64 * 64) / 2);
    // omega is read as float4 rows by the kernels: it must be 16-byte aligned
    // memory of the current device (a host or misaligned address would fault
    // on the device instead of failing here)
    if (reinterpret_cast<uintptr_t>(omega) % 16 != 0)
        return set_error(FAVOR_ERR_INVALID_ARG, "%s: omega must be 16-byte aligned", fn);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return set_error(FAVOR_ERR_INVALID_ARG, "%s: no usable CUDA device, so omega cannot be device memory", fn);
    }
    {
        cudaPointerAttributes pa;
        std::memset(&pa, 0, sizeof(pa));
        const cudaError_t e = cudaPointerGetAttributes(&pa, omega);
        cudaGetLastError();
        if (e != cudaSuccess || (pa.type != cudaMemoryTypeDevice && pa.type != cudaMemoryTypeManaged) ||
            pa.device != dev)
            return set_error(FAVOR_ERR_INVALID_ARG, "%s: omega is not device (or managed) memory of device %d", fn,
                             dev);
    }
    Handle h;
    std::memset(&h, 0, sizeof(h));
    h.H = H; h.m = m; h.d = d; h.dv = dv; h.kind = kind; h.features = kind; h.dtype = dtype; h.s = data_scale;
    h.max_B = B; h.max_L = L; h.device = dev;
    cudaDeviceGetAttribute(&h.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (h.num_sms < 1) h.num_sms = 1;
    cudaDeviceGetAttribute(&h.cc_major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaGetLastError();
    h.omega_f32 = const_cast<float*>(omega);
    return simt_bidir_fixed_scratch(h, q, k, v, out, B, L, reinterpret_cast<cudaStream_t>(stream));
}

favor_status favor_kv_state(favor_handle hd, const void* k, const void* v, float* state, int B, int L,
                            void* stream) {
    favor_status st = check_call("favor_kv_state", hd, B, L);
    if (st != FAVOR_OK) return st;
    if (!k || !v || !state) return set_error(FAVOR_ERR_INVALID_ARG, "favor_kv_state: null pointer");
    if (reinterpret_cast<uintptr_t>(state) % 16)
        return set_error(FAVOR_ERR_INVALID_ARG, "favor_kv_state: state must be 16-byte aligned");
    const Handle& h = *reinterpret_cast<const Handle*>(hd);
    if (relpos_on(h)) return set_error(FAVOR_ERR_UNSUPPORTED, "favor_kv_state: relative positions are set");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (tc_supported(h)) return tc_kv_state(h, k, v, state, B, L, s);
    return simt_kv_state(h, k, v, state, B, L, s);
}

favor_status favor_attn_from_state(favor_handle hd, const void* q, const float* state, void* out, int B, int L,
                                   void* stream) {
    favor_status st = check_call("favor_attn_from_state", hd, B, L);
    if (st != FAVOR_OK) return st;
    if (!q || !state || !out) return set_error(FAVOR_ERR_INVALID_ARG, "favor_attn_from_state: null pointer");
    if (reinterpret_cast<uintptr_t>(state) % 16)
        return set_error(FAVOR_ERR_INVALID_ARG, "favor_attn_from_state: state must be 16-byte aligned");
    const Handle& h = *reinterpret_cast<const Handle*>(hd);
    if (relpos_on(h)) return set_error(FAVOR_ERR_UNSUPPORTED, "favor_attn_from_state: relative positions are set");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (tc_supported(h)) return tc_attn_from_state(h, q, state, out, B, L, s);
    return simt_attn_from_state(h, q, state, out, B, L, s);
}

static favor_status causal_step_call(const char* fn, favor_handle hd, const void* q, const void* k, const void* v,
                                     const float* gate, bool gated, void* out, float* state, int B, int T,
                                     void* stream) {
    favor_status st = check_call(fn, hd, B, T);
    if (st != FAVOR_OK) return st;
    if (!q || !k || !v || !out || !state || (gated && !gate)) return set_error(FAVOR_ERR_INVALID_ARG, "%s: null pointer", fn);
    if (reinterpret_cast<uintptr_t>(state) % 16)
        return set_error(FAVOR_ERR_INVALID_ARG, "%s: state must be 16-byte aligned", fn);
    const Handle& h = *reinterpret_cast<const Handle*>(hd);
    if (relpos_on(h)) return set_error(FAVOR_ERR_UNSUPPORTED, "%s: relative positions are set", fn);
    return simt_causal_step(h, q, k, v, out, state, B, T, reinterpret_cast<cudaStream_t>(stream), gate);
}

favor_status favor_attn_causal_step(favor_handle hd, const void* q, const void* k, const void* v, void* out,
                                    float* state, int B, int T, void* stream) {
    return causal_step_call("favor_attn_causal_step", hd, q, k, v, nullptr, false, out, state, B, T, stream);
}

favor_status favor_attn_causal_step_gated(favor_handle hd, const void* q, const void* k, const void* v,
                                          const float* gate, void* out, float* state, int B, int T, void* stream) {
    return causal_step_call("favor_attn_causal_step_gated", hd, q, k, v, gate, true, out, state, B, T, stream);
}

static favor_status backward_call(const char* fn, bool causal, favor_handle hd, const void* q, const void* k,
                                  const void* v, const void* dout, void* dq, void* dk, void* dv, int B, int L,
                                  void* stream) {
    favor_status st = check_call(fn, hd, B, L);
    if (st != FAVOR_OK) return st;
    if (!q || !k || !v || !dout || !dq || !dk || !dv)
        return set_error(FAVOR_ERR_INVALID_ARG, "%s: null tensor pointer", fn);
    const Handle& h = *reinterpret_cast<const Handle*>(hd);
    if (h.kind == FAVOR_KERNEL_SOFTMAX_TRIG)
        return set_error(FAVOR_ERR_UNSUPPORTED, "%s: no backward for trigonometric features", fn);
    if (relpos_on(h)) return set_error(FAVOR_ERR_UNSUPPORTED, "%s: relative positions are set", fn);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (causal) {
        if (tc_supported(h)) return tc_causal_backward(h, q, k, v, dout, dq, dk, dv, B, L, s);
        return simt_causal_backward(h, q, k, v, dout, dq, dk, dv, B, L, s);
    }
    if (tc_supported(h)) return tc_bidir_backward(h, q, k, v, dout, dq, dk, dv, B, L, s);
    return simt_bidir_backward(h, q, k, v, dout, dq, dk, dv, B, L, s);
}

favor_status favor_attn_bidir_backward(favor_handle hd, const void* q, const void* k, const void* v,
                                       const void* dout, void* dq, void* dk, void* dv, int B, int L, void* stream) {
    return backward_call("favor_attn_bidir_backward", false, hd, q, k, v, dout, dq, dk, dv, B, L, stream);
}

favor_status favor_attn_causal_backward(favor_handle hd, const void* q, const void* k, const void* v,
                                        const void* dout, void* dq, void* dk, void* dv, int B, int L, void* stream) {
    return backward_call("favor_attn_causal_backward", true, hd, q, k, v, dout, dq, dk, dv, B, L, stream);
}

favor_status favor_device_error(favor_handle hd, int* code) {
    if (!hd || !code) return set_error(FAVOR_ERR_INVALID_ARG, "favor_device_error: null argument");
    const Handle* h = reinterpret_cast<const Handle*>(hd);
    cudaError_t e = cudaMemcpy(code, h->dev_err, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return set_error(FAVOR_ERR_CUDA, "favor_device_error: %s", cudaGetErrorString(e));
    }
    return FAVOR_OK;
}

favor_status favor_check_bounded_wait(favor_handle hd, int limit_cycles, void* stream) {
    g_err[0] = 0;
    if (!hd) return set_error(FAVOR_ERR_INVALID_ARG, "favor_check_bounded_wait: handle is NULL");
    if (limit_cycles < 1000 || limit_cycles > (1 << 24))
        return set_error(FAVOR_ERR_INVALID_ARG, "favor_check_bounded_wait: limit_cycles=%d outside [1000, 2^24]",
                         limit_cycles);
    const Handle& h = *reinterpret_cast<const Handle*>(hd);
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess || cur != h.device) {
        cudaGetLastError();
        return set_error(FAVOR_ERR_INVALID_ARG, "favor_check_bounded_wait: current device %d is not the handle's", cur);
    }
    return launch_wait_expiry(h, limit_cycles, FAVOR_WAIT_CHECK_CODE, reinterpret_cast<cudaStream_t>(stream));
}

static const char* kSlotNames[PROF_NSLOTS] = {"feature_map", "segment_state", "segment_combine",
                                               "bidir_readout", "causal_chunks", "backward_query",
                                               "backward_key"};

int favor_profile_slots(void) { return PROF_NSLOTS; }

const char* favor_profile_name(int slot) {
    return (slot >= 0 && slot < PROF_NSLOTS) ? kSlotNames[slot] : "";
}

favor_status favor_profile_enable(favor_handle hd, int enable) {
    if (!hd) return set_error(FAVOR_ERR_INVALID_ARG, "favor_profile_enable: handle is NULL");
    reinterpret_cast<Handle*>(hd)->prof->on = enable != 0;
    return FAVOR_OK;
}

favor_status favor_profile_reset(favor_handle hd) {
    if (!hd) return set_error(FAVOR_ERR_INVALID_ARG, "favor_profile_reset: handle is NULL");
    Profile* p = reinterpret_cast<Handle*>(hd)->prof;
    for (auto& pe : p->pending) { p->spare.push_back(pe.a); p->spare.push_back(pe.b); }
    p->pending.clear();
    for (int i = 0; i < PROF_NSLOTS; ++i) { p->ms[i] = 0.0; p->n[i] = 0; }
    return FAVOR_OK;
}

favor_status favor_profile_read(favor_handle hd, int slot, double* ms_total, unsigned long long* launches) {
    if (!hd || !ms_total || !launches)
        return set_error(FAVOR_ERR_INVALID_ARG, "favor_profile_read: null argument");
    if (slot < 0 || slot >= PROF_NSLOTS) return set_error(FAVOR_ERR_INVALID_ARG, "favor_profile_read: bad slot %d", slot);
    Profile* p = reinterpret_cast<Handle*>(hd)->prof;
    for (auto& pe : p->pending) {
        if (cudaEventSynchronize(pe.b) != cudaSuccess) {
            cudaGetLastError();
            return set_error(FAVOR_ERR_CUDA, "favor_profile_read: event synchronize failed");
        }
        float ms = 0.f;
        if (cudaEventElapsedTime(&ms, pe.a, pe.b) != cudaSuccess) {
            cudaGetLastError();
            return set_error(FAVOR_ERR_CUDA, "favor_profile_read: elapsed time failed");
        }
        p->ms[pe.slot] += ms;
        p->n[pe.slot] += 1;
        p->spare.push_back(pe.a);
        p->spare.push_back(pe.b);
    }
    p->pending.clear();
    *ms_total = p->ms[slot];
    *launches = p->n[slot];
    return FAVOR_OK;
}

}  // extern "C"
