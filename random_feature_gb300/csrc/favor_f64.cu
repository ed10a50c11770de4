// FAVOR+ forward for fp32 storage with float64 arithmetic (CUDA cores).
//
// Bidirectional (Alg. 1 of Rethinking Attention with Performers) and causal
// (App. B.1 Eq. 11) attention for handles of the FP32 dtype with positive,
// hyperbolic or ReLU features.  Inputs are fp32; every projection, exponential,
// state sum and output sum runs in double precision, and only the output of
// the final division is rounded to fp32.
//
// Why double: the outputs are weighted averages of V rows whose entries cancel,
// so an element-wise error measure amplifies rounding in the feature arguments.
// A 1-ulp fp32 error in a key's exponent changes that key's weight in every
// output row, and on the approximation-error workload (L = 4096, d = 16,
// m up to 256) fp32 feature arithmetic lands at about 1e-4 element-wise with
// every later step exact.  In double the same steps stay many orders below.
//
// Work split: per head, the sequence is cut into segments of whole 32-token
// tiles (about two segments per SM over all heads).
//   k64_state   per (segment, head, block of 32 features): the segment's
//               S | z = sum_j phi(k_j) [v_j 1]^T for those features
//   k64_combine fixed-order sum (bidirectional) or exclusive prefix (causal)
//               of the segment states
//   k64_readout per (tile, head): Phi_Q [S | z], then num / den
//   k64_causal  per (segment, head): tile by tile, the output from the running
//               state plus the within-tile masked products, then the state
//               update by the tile's keys
// Shifts that cancel between num and den: each query row by its largest
// projection, keys by the per-head kappa_h (see favor_internal.h); m^-1/2 and
// the query norm term are row constants and are left out.
#include <cmath>

#include "favor_internal.h"

namespace favor {
namespace {

constexpr int kT64 = 32;       // tokens per tile
constexpr int kThr64 = 256;    // threads per block
constexpr int kMaxW64 = 129;   // dv + 1 for dv <= 128
constexpr int kAcc64 = (kMaxW64 + 7) / 8;   // state entries per thread in k64_state

struct Plan64 {
    int tiles;       // ceil(L / 32)
    int seg_tiles;   // tiles per segment
    int n_seg;       // segments per head
};

// About two segments per SM over all heads; BH * n_seg <= 2 * SMs + BH.
Plan64 plan64(int BH, int L, int num_sms) {
    Plan64 p;
    p.tiles = (L + kT64 - 1) / kT64;
    long want = (2L * num_sms + BH - 1) / BH;
    if (want > p.tiles) want = p.tiles;
    if (want < 1) want = 1;
    p.seg_tiles = (int)((p.tiles + want - 1) / want);
    p.n_seg = (p.tiles + p.seg_tiles - 1) / p.seg_tiles;
    return p;
}

// rows [t0, t0 + 32) of one head's [L, w] fp32 tensor, times `scale`, as
// doubles into dst[32][w]; rows at or past `lim` are zero.
__device__ void stage64(const float* __restrict__ src, double* dst, int t0, int lim, int w, double scale) {
    for (int i = threadIdx.x; i < kT64 * w; i += blockDim.x) {
        const int j = i / w;
        dst[i] = (t0 + j < lim) ? scale * (double)src[(size_t)(t0 + j) * w + (i - j * w)] : 0.0;
    }
}

// [v_j 1] rows of a tile into vv[32][dv+1]; rows at or past `lim` are zero.
__device__ void stage_vv64(const float* __restrict__ v, double* vv, int t0, int lim, int dv) {
    const int W = dv + 1;
    for (int i = threadIdx.x; i < kT64 * W; i += blockDim.x) {
        const int j = i / W, e = i - j * W;
        double x = 0.0;
        if (t0 + j < lim) x = e < dv ? (double)v[(size_t)(t0 + j) * dv + e] : 1.0;
        vv[i] = x;
    }
}

// Squared norms of the tile's rows (one warp per row).
__device__ void norms64(const double* xs, double* nrm, int d) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    for (int j = warp; j < kT64; j += nw) {
        double a = 0.0;
        for (int c = lane; c < d; c += 32) a = fma(xs[j * d + c], xs[j * d + c], a);
        for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
        if (lane == 0) nrm[j] = a;
    }
}

// ph[j * ld + r] = omega_r . x_j for every feature r of the head and every row
// j of the tile (xs [32][d]); one thread per feature, 32 rows in registers.
__device__ void project64(const float* __restrict__ om, const double* xs, double* ph, int ld, int m, int d) {
    for (int r = threadIdx.x; r < m; r += blockDim.x) {
        double acc[kT64];
#pragma unroll
        for (int j = 0; j < kT64; ++j) acc[j] = 0.0;
        const float* w = om + (size_t)r * d;
#pragma unroll 1
        for (int c = 0; c < d; ++c) {
            const double wc = (double)__ldg(w + c);
#pragma unroll
            for (int j = 0; j < kT64; ++j) acc[j] = fma(wc, xs[j * d + c], acc[j]);
        }
#pragma unroll
        for (int j = 0; j < kT64; ++j) ph[j * ld + r] = acc[j];
    }
}

// Query features in place: exp(p - max_r p) (positive) or max(p, 0) (ReLU).
template <int KIND>
__device__ void query_features64(double* ph, int ld, int m, double* mx) {
    if (KIND == FAVOR_KERNEL_SOFTMAX_POS) {
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
        for (int j = warp; j < kT64; j += nw) {
            double a = -INFINITY;
            for (int r = lane; r < m; r += 32) a = fmax(a, ph[j * ld + r]);
            for (int o = 16; o > 0; o >>= 1) a = fmax(a, __shfl_xor_sync(0xffffffffu, a, o));
            if (lane == 0) mx[j] = a;
        }
        __syncthreads();
    }
    for (int i = threadIdx.x; i < kT64 * m; i += blockDim.x) {
        const int j = i / m, r = i - j * m;
        double& p = ph[j * ld + r];
        p = KIND == FAVOR_KERNEL_SOFTMAX_POS ? exp(p - mx[j]) : fmax(p, 0.0);
    }
}

// Key feature from its projection p = omega_r . y, ||y||^2 and kappa_h.
template <int KIND>
__device__ __forceinline__ double key_feature64(double p, double nrm, double kap) {
    return KIND == FAVOR_KERNEL_SOFTMAX_POS ? exp(p - 0.5 * nrm - kap) : fmax(p, 0.0);
}

// ------------------------------------------------------------------ kernels
// grid (n_seg, B*H, ceil(m/32)), 256 threads.  Thread (rr = tid % 32, eg =
// tid / 32) owns feature r0 + rr and state columns eg, eg + 8, ...; the
// segment's sums go to part[(bh * n_seg + seg)][m][dv+1].
template <int KIND>
__global__ void __launch_bounds__(kThr64) k64_state(const float* __restrict__ k, const float* __restrict__ v,
                                                    const float* __restrict__ omega, const float* __restrict__ kshift,
                                                    double* __restrict__ part, int H, int L, int m, int d, int dv,
                                                    double s, int seg_len, int n_seg) {
    extern __shared__ double sm64[];
    const int seg = blockIdx.x, bh = blockIdx.y, r0 = blockIdx.z * 32, h = bh % H;
    const int W = dv + 1, tid = threadIdx.x;
    double* om_s = sm64;                  // [32][d+1] omega rows r0.. (padded against bank conflicts)
    double* ys = om_s + 32 * (d + 1);     // [32][d] key rows times s
    double* vv = ys + kT64 * d;           // [32][dv+1]
    double* ph = vv + kT64 * W;           // [32 tokens][32 features]
    double* nrm = ph + kT64 * 32;         // [32]
    for (int i = tid; i < 32 * d; i += blockDim.x) {
        const int rr = i / d, c = i - rr * d;
        om_s[rr * (d + 1) + c] = r0 + rr < m ? (double)omega[((size_t)h * m + r0 + rr) * d + c] : 0.0;
    }
    const double kap = (double)kshift[h];
    const int rr = tid & 31, eg = tid >> 5;
    double acc[kAcc64];
#pragma unroll
    for (int u = 0; u < kAcc64; ++u) acc[u] = 0.0;
    const int tb = seg * seg_len, te = min(L, tb + seg_len);
    const float* kb = k + (size_t)bh * L * d;
    const float* vb = v + (size_t)bh * L * dv;
    for (int t0 = tb; t0 < te; t0 += kT64) {
        __syncthreads();   // the previous tile's features and values are read
        stage64(kb, ys, t0, te, d, s);
        stage_vv64(vb, vv, t0, te, dv);
        __syncthreads();
        if (KIND == FAVOR_KERNEL_SOFTMAX_POS) {
            norms64(ys, nrm, d);
            __syncthreads();
        }
#pragma unroll 1
        for (int u = 0; u < kT64 / 8; ++u) {
            const int j = eg + 8 * u;
            double p = 0.0;
            for (int c = 0; c < d; ++c) p = fma(om_s[rr * (d + 1) + c], ys[j * d + c], p);
            ph[j * 32 + rr] = key_feature64<KIND>(p, KIND == FAVOR_KERNEL_SOFTMAX_POS ? nrm[j] : 0.0, kap);
        }
        __syncthreads();
#pragma unroll 1
        for (int j = 0; j < kT64; ++j) {
            const double a = ph[j * 32 + rr];
#pragma unroll
            for (int u = 0; u < kAcc64; ++u) {
                const int e = eg + 8 * u;
                if (e < W) acc[u] = fma(a, vv[j * W + e], acc[u]);
            }
        }
    }
    if (r0 + rr < m) {
        double* o = part + ((size_t)bh * n_seg + seg) * (size_t)m * W + (size_t)(r0 + rr) * W;
#pragma unroll
        for (int u = 0; u < kAcc64; ++u) {
            const int e = eg + 8 * u;
            if (e < W) o[e] = acc[u];
        }
    }
}

// grid (ceil(m*(dv+1)/256), B*H).  scan = 0: state[bh] = sum of the head's
// segment states in order; scan = 1: each segment state <- the sum of the
// segments before it (in place).
__global__ void k64_combine(double* __restrict__ part, double* __restrict__ state, int n_seg, int n, int scan) {
    const int bh = blockIdx.y;
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    double* p = part + (size_t)bh * n_seg * n + i;
    double run = 0.0;
    for (int sg = 0; sg < n_seg; ++sg) {
        const double x = p[(size_t)sg * n];
        if (scan) p[(size_t)sg * n] = run;
        run += x;
    }
    if (!scan) state[(size_t)bh * n + i] = run;
}

// out rows of a tile from its query features (pq [32][m+1]), a state S [m][dv+1]
// in global memory, and (causal) the masked within-tile products A [32][33]
// against vv [32][dv+1].  Warp w owns rows w, w+8, w+16, w+24; lane the
// columns lane, lane+32, ...  Rows at or past `lim` are not written.  S is
// not marked restrict: the causal kernel writes it between tiles, so its loads
// must stay on the coherent path.
template <bool INTRA>
__device__ void outputs64(const double* pq, int ld, const double* S, const double* A,
                          const double* vv, float* __restrict__ ob, int t0, int lim, int m, int dv) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int W = dv + 1;
    double num[4][4], den[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        den[i] = 0.0;
#pragma unroll
        for (int u = 0; u < 4; ++u) num[i][u] = 0.0;
    }
#pragma unroll 1
    for (int r = 0; r < m; ++r) {
        const double zr = S[(size_t)r * W + dv];
        double sv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int e = lane + 32 * u;
            sv[u] = e < dv ? S[(size_t)r * W + e] : 0.0;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const double f = pq[(warp + 8 * i) * ld + r];
            den[i] = fma(f, zr, den[i]);
#pragma unroll
            for (int u = 0; u < 4; ++u) num[i][u] = fma(f, sv[u], num[i][u]);
        }
    }
    if (INTRA) {
#pragma unroll 1
        for (int j = 0; j < kT64; ++j) {
            const double zr = vv[j * W + dv];
            double sv[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int e = lane + 32 * u;
                sv[u] = e < dv ? vv[j * W + e] : 0.0;
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const double a = A[(warp + 8 * i) * (kT64 + 1) + j];
                den[i] = fma(a, zr, den[i]);
#pragma unroll
                for (int u = 0; u < 4; ++u) num[i][u] = fma(a, sv[u], num[i][u]);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int tok = t0 + warp + 8 * i;
        if (tok >= lim) continue;
        const double inv = den[i] != 0.0 ? 1.0 / den[i] : 0.0;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int e = lane + 32 * u;
            if (e < dv) ob[(size_t)tok * dv + e] = (float)(num[i][u] * inv);
        }
    }
}

// grid (ceil(L/32), B*H), 256 threads: bidirectional readout of one tile.
template <int KIND>
__global__ void __launch_bounds__(kThr64) k64_readout(const float* __restrict__ q, const double* __restrict__ state,
                                                      const float* __restrict__ omega, float* __restrict__ out, int H,
                                                      int L, int m, int d, int dv, double s) {
    extern __shared__ double sm64[];
    const int t0 = blockIdx.x * kT64, bh = blockIdx.y, h = bh % H;
    const int ld = m + 1;
    double* xs = sm64;             // [32][d]
    double* pq = xs + kT64 * d;    // [32][m+1]
    double* mx = pq + kT64 * ld;   // [32]
    stage64(q + (size_t)bh * L * d, xs, t0, L, d, s);
    __syncthreads();
    project64(omega + (size_t)h * m * d, xs, pq, ld, m, d);
    __syncthreads();
    query_features64<KIND>(pq, ld, m, mx);
    __syncthreads();
    outputs64<false>(pq, ld, state + (size_t)bh * m * (dv + 1), nullptr, nullptr, out + (size_t)bh * L * dv, t0, L,
                     m, dv);
}

// grid (n_seg, B*H), 256 threads: causal attention over one segment, tile by
// tile.  part holds, per (head, segment), the exclusive prefix of the earlier
// segments; it is the running state here and is advanced in place.
template <int KIND>
__global__ void __launch_bounds__(kThr64) k64_causal(const float* __restrict__ q, const float* __restrict__ k,
                                                     const float* __restrict__ v, const float* __restrict__ omega,
                                                     const float* __restrict__ kshift, double* __restrict__ part,
                                                     float* __restrict__ out, int H, int L, int m, int d, int dv,
                                                     double s, int seg_len, int n_seg) {
    extern __shared__ double sm64[];
    const int seg = blockIdx.x, bh = blockIdx.y, h = bh % H;
    const int W = dv + 1, ld = m + 1, tid = threadIdx.x;
    double* xs = sm64;               // [32][d]  query rows, then key rows (times s)
    double* pq = xs + kT64 * d;      // [32][m+1] query features
    double* pk = pq + kT64 * ld;     // [32][m+1] key features
    double* vv = pk + kT64 * ld;     // [32][dv+1]
    double* A = vv + kT64 * W;       // [32][33] masked phi_q . phi_k
    double* mx = A + kT64 * (kT64 + 1);
    double* nrm = mx + kT64;
    double* S = part + ((size_t)bh * n_seg + seg) * (size_t)m * W;
    const float* om = omega + (size_t)h * m * d;
    const double kap = (double)kshift[h];
    const size_t hb = (size_t)bh * L;
    const int tb = seg * seg_len, te = min(L, tb + seg_len);
    for (int t0 = tb; t0 < te; t0 += kT64) {
        __syncthreads();   // the previous tile's reads of xs, pk, vv and S are done
        stage64(q + hb * d, xs, t0, te, d, s);
        __syncthreads();
        project64(om, xs, pq, ld, m, d);
        __syncthreads();
        query_features64<KIND>(pq, ld, m, mx);
        stage64(k + hb * d, xs, t0, te, d, s);   // pq no longer needs xs
        stage_vv64(v + hb * dv, vv, t0, te, dv);
        __syncthreads();
        if (KIND == FAVOR_KERNEL_SOFTMAX_POS) norms64(xs, nrm, d);
        project64(om, xs, pk, ld, m, d);
        __syncthreads();
        for (int i = tid; i < kT64 * m; i += blockDim.x) {
            const int j = i / m, r = i - j * m;
            pk[j * ld + r] = key_feature64<KIND>(pk[j * ld + r], KIND == FAVOR_KERNEL_SOFTMAX_POS ? nrm[j] : 0.0, kap);
        }
        __syncthreads();
        // within-tile products, key j <= query i (the diagonal included)
        for (int p = tid; p < kT64 * kT64; p += blockDim.x) {
            const int i = p / kT64, j = p - i * kT64;
            double a = 0.0;
            if (j <= i)
                for (int r = 0; r < m; ++r) a = fma(pq[i * ld + r], pk[j * ld + r], a);
            A[i * (kT64 + 1) + j] = a;
        }
        __syncthreads();
        outputs64<true>(pq, ld, S, A, vv, out + hb * dv, t0, te, m, dv);
        __syncthreads();   // every read of S for this tile precedes the update
        for (int i = tid; i < m * W; i += blockDim.x) {
            const int r = i / W, e = i - r * W;
            double a = S[i];
            for (int j = 0; j < kT64; ++j) a = fma(pk[j * ld + r], vv[j * W + e], a);
            S[i] = a;
        }
    }
}

template <typename K>
void smem_attr(K kern, size_t bytes) {
    if (bytes > 48 * 1024) cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

size_t state_smem(int d, int dv) {
    return (size_t)(32 * (d + 1) + kT64 * d + kT64 * (dv + 1) + kT64 * 32 + kT64) * sizeof(double);
}
size_t readout_smem(int m, int d) { return (size_t)(kT64 * d + kT64 * (m + 1) + kT64) * sizeof(double); }
size_t causal_smem(int m, int d, int dv) {
    return (size_t)(kT64 * d + 2 * kT64 * (m + 1) + kT64 * (dv + 1) + kT64 * (kT64 + 1) + 2 * kT64) * sizeof(double);
}

template <int KIND>
favor_status state64(const Handle& h, const float* k, const float* v, int BH, int L, const Plan64& p,
                     cudaStream_t st) {
    const size_t smem = state_smem(h.d, h.dv);
    smem_attr(k64_state<KIND>, smem);
    dim3 grid(p.n_seg, BH, (h.m + 31) / 32);
    ProfScope ps(h, PROF_STATE, st);
    k64_state<KIND><<<grid, kThr64, smem, st>>>(k, v, h.omega_f32, h.kshift, h.ws64, h.H, L, h.m, h.d, h.dv,
                                                (double)h.s, p.seg_tiles * kT64, p.n_seg);
    count_launch();
    return check_launch("float64 segment state kernel");
}

favor_status combine64(const Handle& h, int BH, const Plan64& p, bool scan, cudaStream_t st) {
    const int n = h.m * (h.dv + 1);
    dim3 grid((n + 255) / 256, BH);
    ProfScope ps(h, PROF_COMBINE, st);
    k64_combine<<<grid, 256, 0, st>>>(h.ws64, h.ws64_state, p.n_seg, n, scan ? 1 : 0);
    count_launch();
    return check_launch("float64 segment combine kernel");
}

template <int KIND>
favor_status bidir64(const Handle& h, const float* q, const float* k, const float* v, float* out, int B, int L,
                     cudaStream_t st) {
    const int BH = B * h.H;
    const Plan64 p = plan64(BH, L, h.num_sms);
    favor_status s = state64<KIND>(h, k, v, BH, L, p, st);
    if (s != FAVOR_OK) return s;
    s = combine64(h, BH, p, false, st);
    if (s != FAVOR_OK) return s;
    const size_t smem = readout_smem(h.m, h.d);
    smem_attr(k64_readout<KIND>, smem);
    dim3 grid(p.tiles, BH);
    ProfScope ps(h, PROF_READOUT, st);
    k64_readout<KIND><<<grid, kThr64, smem, st>>>(q, h.ws64_state, h.omega_f32, out, h.H, L, h.m, h.d, h.dv,
                                                  (double)h.s);
    count_launch();
    return check_launch("float64 readout kernel");
}

template <int KIND>
favor_status causal64(const Handle& h, const float* q, const float* k, const float* v, float* out, int B, int L,
                      cudaStream_t st) {
    const int BH = B * h.H;
    const Plan64 p = plan64(BH, L, h.num_sms);
    favor_status s = FAVOR_OK;
    if (p.n_seg > 1) {
        s = state64<KIND>(h, k, v, BH, L, p, st);
        if (s == FAVOR_OK) s = combine64(h, BH, p, true, st);
    } else if (cudaMemsetAsync(h.ws64, 0, (size_t)BH * h.m * (h.dv + 1) * sizeof(double), st) != cudaSuccess) {
        cudaGetLastError();
        s = set_error(FAVOR_ERR_CUDA, "cudaMemsetAsync failed");
    }
    if (s != FAVOR_OK) return s;
    const size_t smem = causal_smem(h.m, h.d, h.dv);
    smem_attr(k64_causal<KIND>, smem);
    dim3 grid(p.n_seg, BH);
    ProfScope ps(h, PROF_CAUSAL, st);
    k64_causal<KIND><<<grid, kThr64, smem, st>>>(q, k, v, h.omega_f32, h.kshift, h.ws64, out, h.H, L, h.m, h.d,
                                                 h.dv, (double)h.s, p.seg_tiles * kT64, p.n_seg);
    count_launch();
    return check_launch("float64 causal kernel");
}

}  // namespace

size_t f64_workspace_rows(int max_BH, int num_sms) { return 2 * (size_t)num_sms + (size_t)max_BH; }

bool f64_supported(const Handle& h) {
    return h.dtype == FAVOR_DTYPE_F32 && (h.kind == FAVOR_KERNEL_SOFTMAX_POS || h.kind == FAVOR_KERNEL_RELU) &&
           h.ws64 != nullptr && causal_smem(h.m, h.d, h.dv) <= 227 * 1024;
}

favor_status f64_bidir(const Handle& h, const void* q, const void* k, const void* v, void* out, int B, int L,
                       cudaStream_t st) {
    const float *qq = (const float*)q, *kk = (const float*)k, *vv = (const float*)v;
    if (h.kind == FAVOR_KERNEL_RELU) return bidir64<FAVOR_KERNEL_RELU>(h, qq, kk, vv, (float*)out, B, L, st);
    return bidir64<FAVOR_KERNEL_SOFTMAX_POS>(h, qq, kk, vv, (float*)out, B, L, st);
}

favor_status f64_causal(const Handle& h, const void* q, const void* k, const void* v, void* out, int B, int L,
                        cudaStream_t st) {
    const float *qq = (const float*)q, *kk = (const float*)k, *vv = (const float*)v;
    if (h.kind == FAVOR_KERNEL_RELU) return causal64<FAVOR_KERNEL_RELU>(h, qq, kk, vv, (float*)out, B, L, st);
    return causal64<FAVOR_KERNEL_SOFTMAX_POS>(h, qq, kk, vv, (float*)out, B, L, st);
}

}  // namespace favor
