// Generic FAVOR+ kernels on the CUDA cores (FFMA), for every supported shape
// and for fp32 storage.  fp32 storage computes everything in fp32 with the
// accurate expf; bf16 storage reads bf16 and computes in fp32 too.
//
// Feature conventions inside attention (all shifts cancel between numerator
// and denominator, so the output equals Eq. 4 / Eq. 11 of Rethinking Attention
// with Performers up to rounding):
//   key   features  exp(s*p - s^2||k||^2/2 - kappa_h)   (positive)  | max(s*p, 0) (ReLU)
//   query features  exp(s*(p - max_r p_r))               (positive)  | max(s*p, 0) (ReLU)
// where p = omega_r . k (or q).  The query shift drops the -||x||^2/2 term and
// the m^-1/2 factor, both common to a query row; the key shift kappa_h is
// common to a head.  favor_feature_map returns the unshifted definition.
#include <cmath>
#include <mutex>

#include "favor_internal.h"

namespace favor {
namespace {

template <typename T> __device__ __forceinline__ float ldf(const T* p);
template <> __device__ __forceinline__ float ldf<float>(const float* p) { return *p; }
template <> __device__ __forceinline__ float ldf<__nv_bfloat16>(const __nv_bfloat16* p) { return __bfloat162float(*p); }

template <typename T> __device__ __forceinline__ void stf(T* p, float x);
template <> __device__ __forceinline__ void stf<float>(float* p, float x) { *p = x; }
template <> __device__ __forceinline__ void stf<__nv_bfloat16>(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

constexpr int kTokTile = 32;  // tokens staged per shared-memory tile in the state/causal kernels

// Feature values by computation kind, from the unscaled projection p = omega_r . x
// (r the feature index of m).  The hyperbolic map runs as the positive kind on
// the mirrored rows [omega; -omega].  The trigonometric kind holds the rows
// [omega; omega]: features r < m/2 take sin, the others cos, of the same
// projection, and its key features carry h(y) = exp(||y||^2/2) with no shift.
template <int KIND>
__device__ __forceinline__ float key_feat(float p, float nrm, float s, float kap, int r, int m) {
    if (KIND == FAVOR_KERNEL_SOFTMAX_POS) return expf(s * p - 0.5f * s * s * nrm - kap);
    if (KIND == FAVOR_KERNEL_RELU) return fmaxf(s * p, 0.f);
    const float a = s * p;
    return (r < (m >> 1) ? sinf(a) : cosf(a)) * expf(0.5f * s * s * nrm);
}

// Query features up to a factor common to the row (the shift mx, m^-1/2, and
// for the trigonometric kind h(x)): they cancel in num / den.
template <int KIND>
__device__ __forceinline__ float query_feat(float sp, float mx, int r, int m) {
    if (KIND == FAVOR_KERNEL_SOFTMAX_POS) return expf(sp - mx);
    if (KIND == FAVOR_KERNEL_RELU) return fmaxf(sp, 0.f);
    return r < (m >> 1) ? sinf(sp) : cosf(sp);
}

// The plain definition (favor_feature_map).
template <int KIND>
__device__ __forceinline__ float plain_feat(float p, float nrm, float s, int r, int m) {
    if (KIND == FAVOR_KERNEL_SOFTMAX_POS) return expf(s * p - 0.5f * s * s * nrm) * rsqrtf((float)m);
    if (KIND == FAVOR_KERNEL_RELU) return fmaxf(s * p, 0.f) * rsqrtf((float)m);
    const float a = s * p;
    return (r < (m >> 1) ? sinf(a) : cosf(a)) * expf(0.5f * s * s * nrm) * rsqrtf((float)(m >> 1));
}

// Position-dependent feature order of PermuteFormer: at position j the slot r
// holds feature pi^j(r).  Per head, the permutation's cycles are listed in
// cyc[h*m + ...]; meta[h*m + r] = (start of r's cycle, its length, r's place in
// it, 0), so pi^j(r) = cyc[h*m + start + (place + j) mod length].
struct PermCursor {
    const int* cyc;   // null: identity
    int base, len, idx;
    __device__ __forceinline__ void init(const int* c, const int4* meta, int h, int m, int r, long long j) {
        cyc = c;
        base = 0; len = 1; idx = 0;
        if (c) {
            const int4 mt = meta[(size_t)h * m + r];
            base = h * m + mt.x;
            len = mt.y;
            idx = (int)((mt.z + j) % mt.y);
        }
    }
    __device__ __forceinline__ int row(int r) const { return cyc ? cyc[base + idx] : r; }
    __device__ __forceinline__ void next() {
        if (cyc && ++idx == len) idx = 0;
    }
};

// Per-token decay of a causal state: S_j = a_j S_{j-1} + b_j phi(k_j) [v_j 1]^T
// with a_j = r_h g_j and b_j = 1 - g_j (RFA-Gate gates g, PermuteFormer r).
__device__ __forceinline__ void token_decay(const float* gate, size_t gidx, float rd, float* a, float* b) {
    const float g = gate ? gate[gidx] : 0.f;
    *a = rd * (gate ? g : 1.f);
    *b = gate ? 1.f - g : 1.f;
}

// ---------------------------------------------------------------- feature map
// grid (ceil(L/16), B*H), 256 threads.  Output phi[bh, i, r] = plain definition.
template <typename T, int KIND>
__global__ void __launch_bounds__(256) k_feature_map(const T* __restrict__ x, T* __restrict__ phi,
                                                     const float* __restrict__ omega, int H, int L,
                                                     int m, int d, float s) {
    constexpr int TQ = 16;
    extern __shared__ float sm[];
    float* xs = sm;                 // [TQ][d]
    float* nrm = xs + TQ * d;       // [TQ]
    const int bh = blockIdx.y, h = bh % H;
    const int i0 = blockIdx.x * TQ;
    const int nq = min(TQ, L - i0);
    const T* xb = x + ((size_t)bh * L + i0) * d;
    for (int idx = threadIdx.x; idx < nq * d; idx += blockDim.x) xs[idx] = ldf(xb + idx);
    __syncthreads();
    if (threadIdx.x < nq) {
        float a = 0.f;
        for (int c = 0; c < d; ++c) a = fmaf(xs[threadIdx.x * d + c], xs[threadIdx.x * d + c], a);
        nrm[threadIdx.x] = a;
    }
    __syncthreads();
    const float* om = omega + (size_t)h * m * d;
    T* out = phi + ((size_t)bh * L + i0) * m;
    for (int idx = threadIdx.x; idx < nq * m; idx += blockDim.x) {
        const int i = idx / m, r = idx - i * m;
        float p = 0.f;
        for (int c = 0; c < d; ++c) p = fmaf(__ldg(om + r * d + c), xs[i * d + c], p);
        stf(out + idx, plain_feat<KIND>(p, nrm[i], s, r, m));
    }
}

// ------------------------------------------------------- per-segment key state
// grid (n_seg, B*H), m threads.  Thread r accumulates S[r, 0:dv] and z[r] over
// its segment's keys and writes them to part[(bh*n_seg + seg)][r][0:dv+1].
template <typename T, int KIND, int DV>
__global__ void __launch_bounds__(256) k_segment_state(const T* __restrict__ k, const T* __restrict__ v,
                                                       const float* __restrict__ omega,
                                                       const float* __restrict__ kshift, float* __restrict__ part,
                                                       int H, int L, int m, int d, float s, int seg_len, int n_seg,
                                                       const int* __restrict__ pcyc, const int4* __restrict__ pmeta,
                                                       const float* __restrict__ gate, const float* __restrict__ rdec,
                                                       float* __restrict__ segdecay) {
    extern __shared__ float sm[];
    const int dp = d + 1;
    float* oms = sm;                       // [m][d+1]
    float* ks = oms + m * dp;              // [kTokTile][d]
    float* vs = ks + kTokTile * d;         // [kTokTile][DV]
    float* nrm = vs + kTokTile * DV;       // [kTokTile]
    const int seg = blockIdx.x, bh = blockIdx.y, h = bh % H;
    const int r = threadIdx.x;
    for (int idx = threadIdx.x; idx < m * d; idx += blockDim.x)
        oms[(idx / d) * dp + idx % d] = omega[(size_t)h * m * d + idx];
    const float kap = kshift[h];
    float S[DV];
#pragma unroll
    for (int e = 0; e < DV; ++e) S[e] = 0.f;
    float z = 0.f;
    const int j0 = seg * seg_len, j1 = min(L, j0 + seg_len);
    PermCursor pc;
    pc.init(pcyc, pmeta, h, m, r, j0);
    const bool decay = gate || rdec;
    const float rd = rdec ? rdec[h] : 1.f;
    float A = 1.f;   // product of the segment's a_j
    for (int t0 = j0; t0 < j1; t0 += kTokTile) {
        const int nt = min(kTokTile, j1 - t0);
        __syncthreads();
        for (int idx = threadIdx.x; idx < nt * d; idx += blockDim.x)
            ks[idx] = ldf(k + ((size_t)bh * L + t0) * d + idx);
        for (int idx = threadIdx.x; idx < nt * DV; idx += blockDim.x)
            vs[idx] = ldf(v + ((size_t)bh * L + t0) * DV + idx);
        __syncthreads();
        for (int j = threadIdx.x; j < nt; j += blockDim.x) {   // blockDim may be below kTokTile
            float a = 0.f;
            for (int c = 0; c < d; ++c) a = fmaf(ks[j * d + c], ks[j * d + c], a);
            nrm[j] = a;
        }
        __syncthreads();
        for (int j = 0; j < nt; ++j) {
            const int row = pc.row(r);
            float p = 0.f;
            for (int c = 0; c < d; ++c) p = fmaf(oms[row * dp + c], ks[j * d + c], p);
            const float f = key_feat<KIND>(p, nrm[j], s, kap, row, m);
            if (decay) {
                float a, b;
                token_decay(gate, (size_t)bh * L + t0 + j, rd, &a, &b);
                const float fb = f * b;
#pragma unroll
                for (int e = 0; e < DV; ++e) S[e] = fmaf(a, S[e], fb * vs[j * DV + e]);
                z = fmaf(a, z, fb);
                A *= a;
            } else {
#pragma unroll
                for (int e = 0; e < DV; ++e) S[e] = fmaf(f, vs[j * DV + e], S[e]);
                z += f;
            }
            pc.next();
        }
    }
    float* o = part + ((size_t)bh * n_seg + seg) * m * (DV + 1) + (size_t)r * (DV + 1);
#pragma unroll
    for (int e = 0; e < DV; ++e) o[e] = S[e];
    o[DV] = z;
    if (segdecay && r == 0) segdecay[(size_t)bh * n_seg + seg] = A;
}

// ------------------------------------------------- fixed-order segment combines
// Bidirectional: state[bh] = sum over seg (in order) of part[bh, seg].
__global__ void k_reduce_segments(const float* __restrict__ part, float* __restrict__ state, int n_seg, int n) {
    const int bh = blockIdx.y;
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const float* p = part + (size_t)bh * n_seg * n + i;
    float a = 0.f;
    for (int sg = 0; sg < n_seg; ++sg) a += p[(size_t)sg * n];
    state[(size_t)bh * n + i] = a;
}

// Causal: part[bh, seg] <- sum of part[bh, 0..seg-1] (exclusive prefix, in order).
__global__ void k_scan_segments(float* __restrict__ part, int n_seg, int n) {
    const int bh = blockIdx.y;
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    float* p = part + (size_t)bh * n_seg * n + i;
    float run = 0.f;
    for (int sg = 0; sg < n_seg; ++sg) {
        const float t = p[(size_t)sg * n];
        p[(size_t)sg * n] = run;
        run += t;
    }
}

// Causal with a decaying state: prefix[seg+1] = A_seg prefix[seg] + total[seg],
// A_seg the product of the segment's per-token decays.
__global__ void k_scan_segments_decay(float* __restrict__ part, const float* __restrict__ segdecay, int n_seg,
                                      int n) {
    const int bh = blockIdx.y;
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    float* p = part + (size_t)bh * n_seg * n + i;
    const float* a = segdecay + (size_t)bh * n_seg;
    float run = 0.f;
    for (int sg = 0; sg < n_seg; ++sg) {
        const float t = p[(size_t)sg * n];
        p[(size_t)sg * n] = run;
        run = fmaf(a[sg], run, t);
    }
}

// ------------------------------------------------------- bidirectional readout
// grid (ceil(L/16), B*H), 256 threads.  out_i = phi(q_i)^T S / phi(q_i)^T z.
template <typename T, int KIND>
__global__ void __launch_bounds__(256) k_readout(const T* __restrict__ q, const float* __restrict__ state,
                                                 const float* __restrict__ omega, T* __restrict__ out,
                                                 int H, int L, int m, int d, int dv, float s,
                                                 const int* __restrict__ pcyc, const int4* __restrict__ pmeta) {
    constexpr int TQ = 16;
    extern __shared__ float sm[];
    const int sw = dv + 1;
    float* sts = sm;                 // [m][dv+1]
    float* fq = sts + m * sw;        // [TQ][m]
    float* xs = fq + TQ * m;         // [TQ][d]
    float* num = xs + TQ * d;        // [TQ][dv+1]
    float* rmax = num + TQ * sw;     // [TQ]
    const int bh = blockIdx.y, h = bh % H;
    const int i0 = blockIdx.x * TQ;
    const int nq = min(TQ, L - i0);
    const float* stg = state + (size_t)bh * m * sw;
    for (int idx = threadIdx.x; idx < m * sw; idx += blockDim.x) sts[idx] = stg[idx];
    for (int idx = threadIdx.x; idx < nq * d; idx += blockDim.x) xs[idx] = ldf(q + ((size_t)bh * L + i0) * d + idx);
    __syncthreads();
    const float* om = omega + (size_t)h * m * d;
    for (int idx = threadIdx.x; idx < nq * m; idx += blockDim.x) {
        const int i = idx / m, r = idx - i * m;
        PermCursor pc;
        pc.init(pcyc, pmeta, h, m, r, i0 + i);
        const int row = pc.row(r);
        float p = 0.f;
        for (int c = 0; c < d; ++c) p = fmaf(__ldg(om + row * d + c), xs[i * d + c], p);
        fq[idx] = s * p;
    }
    __syncthreads();
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (KIND == FAVOR_KERNEL_SOFTMAX_POS) {
        for (int i = warp; i < nq; i += blockDim.x / 32) {
            float mx = -INFINITY;
            for (int r = lane; r < m; r += 32) mx = fmaxf(mx, fq[i * m + r]);
            for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            if (lane == 0) rmax[i] = mx;
        }
        __syncthreads();
        for (int idx = threadIdx.x; idx < nq * m; idx += blockDim.x) fq[idx] = expf(fq[idx] - rmax[idx / m]);
    } else {
        for (int idx = threadIdx.x; idx < nq * m; idx += blockDim.x) {
            const int i = idx / m, r = idx - i * m;
            PermCursor pc;
            pc.init(pcyc, pmeta, h, m, r, i0 + i);
            fq[idx] = query_feat<KIND>(fq[idx], 0.f, pc.row(r), m);
        }
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < nq * sw; idx += blockDim.x) {
        const int i = idx / sw, e = idx - i * sw;
        float a = 0.f;
        for (int r = 0; r < m; ++r) a = fmaf(fq[i * m + r], sts[r * sw + e], a);
        num[idx] = a;
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < nq * dv; idx += blockDim.x) {
        const int i = idx / dv, e = idx - i * dv;
        const float den = num[i * sw + dv];
        stf(out + ((size_t)bh * L + i0) * dv + idx, den != 0.f ? num[i * sw + e] / den : 0.f);
    }
}

// --------------------------------------------------------- causal, per segment
// grid (n_seg, B*H), m threads.  Thread r holds S[r, :], z[r] starting from the
// segment's exclusive prefix state and walks the segment token by token:
// S += phi(k_i) v_i^T, z += phi(k_i) (inclusive of i), then
// out_i = phi(q_i)^T S / phi(q_i)^T z, the sum over r done across the block.
template <typename T, int KIND, int DV>
__global__ void __launch_bounds__(256) k_causal_segment(const T* __restrict__ q, const T* __restrict__ k,
                                                        const T* __restrict__ v, const float* __restrict__ omega,
                                                        const float* __restrict__ kshift,
                                                        const float* __restrict__ prefix, T* __restrict__ out,
                                                        int H, int L, int m, int d, float s, int seg_len, int n_seg,
                                                        const int* __restrict__ pcyc, const int4* __restrict__ pmeta,
                                                        const float* __restrict__ gate,
                                                        const float* __restrict__ rdec) {
    extern __shared__ float sm[];
    const int dp = d + 1;
    const int nwarps = (m + 31) / 32;
    float* oms = sm;                        // [m][d+1]
    float* qs = oms + m * dp;               // [kTokTile][d]
    float* ks = qs + kTokTile * d;          // [kTokTile][d]
    float* vs = ks + kTokTile * d;          // [kTokTile][DV]
    float* nrm = vs + kTokTile * DV;        // [kTokTile]
    float* red = nrm + kTokTile;            // [nwarps][DV+1]
    float* wmax = red + nwarps * (DV + 1);  // [nwarps]
    const int seg = blockIdx.x, bh = blockIdx.y, h = bh % H;
    const int r = threadIdx.x, warp = r / 32, lane = r % 32;
    for (int idx = threadIdx.x; idx < m * d; idx += blockDim.x)
        oms[(idx / d) * dp + idx % d] = omega[(size_t)h * m * d + idx];
    const float kap = kshift[h];
    float S[DV];
    const float* pre = prefix + ((size_t)bh * n_seg + seg) * m * (DV + 1) + (size_t)r * (DV + 1);
#pragma unroll
    for (int e = 0; e < DV; ++e) S[e] = pre[e];
    float z = pre[DV];
    // m is a multiple of 16, so only a last warp of 16 lanes can be partial.
    const int width = (m % 32 != 0 && warp == nwarps - 1) ? 16 : 32;
    const unsigned full = width == 32 ? 0xffffffffu : 0x0000ffffu;
    const int j0 = seg * seg_len, j1 = min(L, j0 + seg_len);
    PermCursor pc;
    pc.init(pcyc, pmeta, h, m, r, j0);
    const bool decay = gate || rdec;
    const float rd = rdec ? rdec[h] : 1.f;
    for (int t0 = j0; t0 < j1; t0 += kTokTile) {
        const int nt = min(kTokTile, j1 - t0);
        __syncthreads();
        for (int idx = threadIdx.x; idx < nt * d; idx += blockDim.x) {
            qs[idx] = ldf(q + ((size_t)bh * L + t0) * d + idx);
            ks[idx] = ldf(k + ((size_t)bh * L + t0) * d + idx);
        }
        for (int idx = threadIdx.x; idx < nt * DV; idx += blockDim.x)
            vs[idx] = ldf(v + ((size_t)bh * L + t0) * DV + idx);
        __syncthreads();
        for (int j = threadIdx.x; j < nt; j += blockDim.x) {   // blockDim may be below kTokTile
            float a = 0.f;
            for (int c = 0; c < d; ++c) a = fmaf(ks[j * d + c], ks[j * d + c], a);
            nrm[j] = a;
        }
        __syncthreads();
        for (int j = 0; j < nt; ++j) {
            const int row = pc.row(r);   // query and key at one position share pi^j
            float pk = 0.f, pq = 0.f;
            for (int c = 0; c < d; ++c) {
                pk = fmaf(oms[row * dp + c], ks[j * d + c], pk);
                pq = fmaf(oms[row * dp + c], qs[j * d + c], pq);
            }
            const float fk = key_feat<KIND>(pk, nrm[j], s, kap, row, m);
            if (decay) {
                float a, b;
                token_decay(gate, (size_t)bh * L + t0 + j, rd, &a, &b);
                const float fb = fk * b;
#pragma unroll
                for (int e = 0; e < DV; ++e) S[e] = fmaf(a, S[e], fb * vs[j * DV + e]);
                z = fmaf(a, z, fb);
            } else {
#pragma unroll
                for (int e = 0; e < DV; ++e) S[e] = fmaf(fk, vs[j * DV + e], S[e]);
                z += fk;
            }
            pc.next();
            float fq;
            if (KIND == FAVOR_KERNEL_SOFTMAX_POS) {
                float mx = s * pq;
                for (int o = width / 2; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(full, mx, o));
                if (lane == 0) wmax[warp] = mx;
                __syncthreads();
                mx = wmax[0];
                for (int w = 1; w < nwarps; ++w) mx = fmaxf(mx, wmax[w]);
                fq = expf(s * pq - mx);
            } else {
                fq = query_feat<KIND>(s * pq, 0.f, row, m);
            }
            // sum over r of fq * [S | z]: warp shuffles, then across warps in smem.
#pragma unroll
            for (int e = 0; e <= DV; ++e) {
                float a = fq * (e < DV ? S[e] : z);
                for (int o = width / 2; o > 0; o >>= 1) a += __shfl_xor_sync(full, a, o);
                if (lane == 0) red[warp * (DV + 1) + e] = a;
            }
            __syncthreads();
            for (int e = threadIdx.x; e < DV; e += blockDim.x) {   // blockDim = m may be below DV
                float a = 0.f, den = 0.f;
                for (int w = 0; w < nwarps; ++w) {
                    a += red[w * (DV + 1) + e];
                    den += red[w * (DV + 1) + DV];
                }
                stf(out + ((size_t)bh * L + t0 + j) * DV + e, den != 0.f ? a / den : 0.f);
            }
            __syncthreads();
        }
    }
}

template <typename K>
static void set_smem(K kern, size_t bytes) {
    if (bytes > 48 * 1024) cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

template <typename T, int KIND>
favor_status feature_map_t(const Handle& h, const void* x, void* phi, int B, int L, cudaStream_t st) {
    const size_t smem = (16 * h.d + 16) * sizeof(float);
    dim3 grid((L + 15) / 16, B * h.H);
    ProfScope ps(h, PROF_FEATURE_MAP, st);
    k_feature_map<T, KIND><<<grid, 256, smem, st>>>((const T*)x, (T*)phi, h.omega_f32, h.H, L, h.m, h.d, h.s);
    count_launch();
    return check_launch("feature map kernel");
}

template <typename T, int KIND, int DV>
favor_status state_t(const Handle& h, const void* k, const void* v, int BH, int L, const SegPlan& p,
                     const RelposArgs& rp, cudaStream_t st) {
    const size_t smem = (size_t)(h.m * (h.d + 1) + kTokTile * h.d + kTokTile * DV + kTokTile) * sizeof(float);
    auto kern = k_segment_state<T, KIND, DV>;
    set_smem(kern, smem);
    dim3 grid(p.n_seg, BH);
    ProfScope ps(h, PROF_STATE, st);
    kern<<<grid, h.m, smem, st>>>((const T*)k, (const T*)v, h.omega_f32, h.kshift, h.ws_partial, h.H, L, h.m,
                                  h.d, h.s, p.seg_tiles * 128, p.n_seg, rp.cyc, rp.meta, rp.gate, rp.rdec,
                                  rp.segdecay);
    count_launch();
    return check_launch("segment state kernel");
}

template <typename T, int KIND>
favor_status readout_t(const Handle& h, const void* q, void* out, int BH, int L, cudaStream_t st,
                       const RelposArgs& rp = RelposArgs()) {
    const int sw = h.dv + 1;
    const size_t smem = (size_t)(h.m * sw + 16 * h.m + 16 * h.d + 16 * sw + 16) * sizeof(float);
    auto kern = k_readout<T, KIND>;
    set_smem(kern, smem);
    dim3 grid((L + 15) / 16, BH);
    ProfScope ps(h, PROF_READOUT, st);
    kern<<<grid, 256, smem, st>>>((const T*)q, h.ws_state, h.omega_f32, (T*)out, h.H, L, h.m, h.d, h.dv, h.s,
                                  rp.cyc, rp.meta);
    count_launch();
    return check_launch("readout kernel");
}

template <typename T, int KIND, int DV>
favor_status causal_t(const Handle& h, const void* q, const void* k, const void* v, void* out, int BH, int L,
                      const SegPlan& p, const RelposArgs& rp, cudaStream_t st) {
    const int nwarps = (h.m + 31) / 32;
    const size_t smem = (size_t)(h.m * (h.d + 1) + 2 * kTokTile * h.d + kTokTile * DV + kTokTile +
                                 nwarps * (DV + 1) + nwarps) * sizeof(float);
    auto kern = k_causal_segment<T, KIND, DV>;
    set_smem(kern, smem);
    dim3 grid(p.n_seg, BH);
    ProfScope ps(h, PROF_CAUSAL, st);
    kern<<<grid, h.m, smem, st>>>((const T*)q, (const T*)k, (const T*)v, h.omega_f32, h.kshift, h.ws_partial,
                                  (T*)out, h.H, L, h.m, h.d, h.s, p.seg_tiles * 128, p.n_seg, rp.cyc, rp.meta,
                                  rp.gate, rp.rdec);
    count_launch();
    return check_launch("causal segment kernel");
}

// Runtime (dtype, kind, dv) -> template instantiation.
template <template <typename, int, int> class F, typename... A>
favor_status dispatch3(const Handle& h, A... a) {
#define FAVOR_DV_CASES(T, KIND)                                   \
    switch (h.dv) {                                               \
        case 16: return F<T, KIND, 16>::run(h, a...);             \
        case 32: return F<T, KIND, 32>::run(h, a...);             \
        case 64: return F<T, KIND, 64>::run(h, a...);             \
        case 128: return F<T, KIND, 128>::run(h, a...);           \
    }
    if (h.dtype == FAVOR_DTYPE_F32) {
        if (h.kind == FAVOR_KERNEL_SOFTMAX_POS) { FAVOR_DV_CASES(float, FAVOR_KERNEL_SOFTMAX_POS) }
        else if (h.kind == FAVOR_KERNEL_RELU) { FAVOR_DV_CASES(float, FAVOR_KERNEL_RELU) }
        else { FAVOR_DV_CASES(float, FAVOR_KERNEL_SOFTMAX_TRIG) }
    } else {
        if (h.kind == FAVOR_KERNEL_SOFTMAX_POS) { FAVOR_DV_CASES(__nv_bfloat16, FAVOR_KERNEL_SOFTMAX_POS) }
        else if (h.kind == FAVOR_KERNEL_RELU) { FAVOR_DV_CASES(__nv_bfloat16, FAVOR_KERNEL_RELU) }
        else { FAVOR_DV_CASES(__nv_bfloat16, FAVOR_KERNEL_SOFTMAX_TRIG) }
    }
#undef FAVOR_DV_CASES
    return set_error(FAVOR_ERR_UNSUPPORTED, "unsupported dv=%d", h.dv);
}

// (dtype, kind) -> FN<T, KIND>(args...), for launchers templated on both.
#define FAVOR_KIND_DISPATCH(hh, FN, ...)                                                             \
    do {                                                                                            \
        if ((hh).dtype == FAVOR_DTYPE_F32) {                                                        \
            if ((hh).kind == FAVOR_KERNEL_SOFTMAX_POS) return FN<float, FAVOR_KERNEL_SOFTMAX_POS>(__VA_ARGS__); \
            if ((hh).kind == FAVOR_KERNEL_RELU) return FN<float, FAVOR_KERNEL_RELU>(__VA_ARGS__);    \
            return FN<float, FAVOR_KERNEL_SOFTMAX_TRIG>(__VA_ARGS__);                               \
        }                                                                                           \
        if ((hh).kind == FAVOR_KERNEL_SOFTMAX_POS) return FN<__nv_bfloat16, FAVOR_KERNEL_SOFTMAX_POS>(__VA_ARGS__); \
        if ((hh).kind == FAVOR_KERNEL_RELU) return FN<__nv_bfloat16, FAVOR_KERNEL_RELU>(__VA_ARGS__); \
        return FN<__nv_bfloat16, FAVOR_KERNEL_SOFTMAX_TRIG>(__VA_ARGS__);                           \
    } while (0)

template <typename T, int KIND, int DV>
struct StateF {
    static favor_status run(const Handle& h, const void* k, const void* v, int BH, int L, const SegPlan* p,
                            const RelposArgs* rp, cudaStream_t st) {
        return state_t<T, KIND, DV>(h, k, v, BH, L, *p, *rp, st);
    }
};

template <typename T, int KIND, int DV>
struct CausalF {
    static favor_status run(const Handle& h, const void* q, const void* k, const void* v, void* out, int BH,
                            int L, const SegPlan* p, const RelposArgs* rp, cudaStream_t st) {
        return causal_t<T, KIND, DV>(h, q, k, v, out, BH, L, *p, *rp, st);
    }
};

}  // namespace

favor_status launch_reduce_segments(const Handle& h, int BH, int n_seg, cudaStream_t st) {
    const int n = h.m * (h.dv + 1);
    dim3 grid((n + 255) / 256, BH);
    ProfScope ps(h, PROF_COMBINE, st);
    k_reduce_segments<<<grid, 256, 0, st>>>(h.ws_partial, h.ws_state, n_seg, n);
    count_launch();
    return check_launch("segment reduce kernel");
}

favor_status launch_scan_segments(const Handle& h, int BH, int n_seg, cudaStream_t st) {
    const int n = h.m * (h.dv + 1);
    dim3 grid((n + 255) / 256, BH);
    ProfScope ps(h, PROF_COMBINE, st);
    k_scan_segments<<<grid, 256, 0, st>>>(h.ws_partial, n_seg, n);
    count_launch();
    return check_launch("segment scan kernel");
}

favor_status simt_feature_map(const Handle& h, const void* x, void* phi, int B, int L, cudaStream_t st) {
    FAVOR_KIND_DISPATCH(h, feature_map_t, h, x, phi, B, L, st);
}

favor_status simt_bidir(const Handle& h, const void* q, const void* k, const void* v, void* out, int B, int L,
                        cudaStream_t st) {
    const int BH = B * h.H;
    SegPlan p = plan_segments(BH, L, h.num_sms);
    RelposArgs rp;   // bidirectional: the permutation only (r = 1)
    rp.cyc = h.perm_cyc;
    rp.meta = h.perm_meta;
    favor_status s = dispatch3<StateF>(h, k, v, BH, L, (const SegPlan*)&p, (const RelposArgs*)&rp, st);
    if (s != FAVOR_OK) return s;
    s = launch_reduce_segments(h, BH, p.n_seg, st);
    if (s != FAVOR_OK) return s;
    FAVOR_KIND_DISPATCH(h, readout_t, h, q, out, BH, L, st, rp);
}

favor_status simt_causal(const Handle& h, const void* q, const void* k, const void* v, void* out, int B, int L,
                         cudaStream_t st, const float* gate) {
    const int BH = B * h.H;
    SegPlan p = plan_segments(BH, L, h.num_sms);
    RelposArgs rp;
    rp.cyc = h.perm_cyc;
    rp.meta = h.perm_meta;
    rp.gate = gate;
    rp.rdec = h.relpos_r;
    const bool decay = gate || h.relpos_r;
    rp.segdecay = decay ? h.ws_segdecay : nullptr;
    favor_status s = FAVOR_OK;
    if (p.n_seg > 1) {
        s = dispatch3<StateF>(h, k, v, BH, L, (const SegPlan*)&p, (const RelposArgs*)&rp, st);
        if (s != FAVOR_OK) return s;
        if (decay) {
            const int n = h.m * (h.dv + 1);
            dim3 grid((n + 255) / 256, BH);
            ProfScope ps(h, PROF_COMBINE, st);
            k_scan_segments_decay<<<grid, 256, 0, st>>>(h.ws_partial, h.ws_segdecay, p.n_seg, n);
            count_launch();
            s = check_launch("segment scan kernel");
        } else {
            s = launch_scan_segments(h, BH, p.n_seg, st);
        }
    } else {
        s = cudaMemsetAsync(h.ws_partial, 0, (size_t)BH * h.m * (h.dv + 1) * sizeof(float), st) == cudaSuccess
                ? FAVOR_OK
                : set_error(FAVOR_ERR_CUDA, "cudaMemsetAsync failed");
    }
    if (s != FAVOR_OK) return s;
    return dispatch3<CausalF>(h, q, k, v, out, BH, L, (const SegPlan*)&p, (const RelposArgs*)&rp, st);
}

// ------------------------------------------------------- stateful calls
// Public state convention: state[b,h] is [m][dv+1] fp32, row r = (S_r, z_r) with
// S = e^-kappa_h sum_j phi(k_j) v_j^T and z = e^-kappa_h sum_j phi(k_j), phi the
// plain feature map (m^-1/2 included), kappa_h the handle's per-head key shift.
// The segment kernels above leave out m^-1/2, so their sums are scaled here.

namespace {

// state[bh][i] += scale * sum over segments (in order) of part[bh, seg][i].
__global__ void k_accum_rows(const float* __restrict__ part, float* __restrict__ state, int n_seg, int n, float scale) {
    const int bh = blockIdx.y;
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const float* p = part + (size_t)bh * n_seg * n + i;
    float a = 0.f;
    for (int sg = 0; sg < n_seg; ++sg) a += p[(size_t)sg * n];
    state[(size_t)bh * n + i] += scale * a;
}

__device__ __forceinline__ float block_max(float x, float* red) {
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = x;
    __syncthreads();
    if (threadIdx.x < 32) {
        float y = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : -INFINITY;
        for (int o = 16; o > 0; o >>= 1) y = fmaxf(y, __shfl_xor_sync(0xffffffffu, y, o));
        if (threadIdx.x == 0) red[0] = y;
    }
    __syncthreads();
    return red[0];
}

// Causal attention over Tn new tokens continuing from state[bh] (App. B.1 Eq. 11
// with the prefix started at the given state; the token recurrence
// S_t = S_{t-1} + phi(k_t) v_t^T, z_t = z_{t-1} + phi(k_t), out_t = phi(q_t)^T S_t /
// phi(q_t)^T z_t).  One CTA per (b, h), thread r owns feature r; the state lives
// in shared memory for the whole call.  Meant for short blocks (decoding).
template <typename T, int KIND>
__global__ void __launch_bounds__(256) k_causal_step(const T* __restrict__ q, const T* __restrict__ k,
                                                     const T* __restrict__ v, T* __restrict__ out,
                                                     float* __restrict__ state, const float* __restrict__ omega,
                                                     const float* __restrict__ kshift, int H, int Tn, int m, int d,
                                                     int dv, float s, int omega_in_smem,
                                                     const float* __restrict__ gate) {
    extern __shared__ float sm[];
    const int dp = dv + 1, wp = d + 1;
    float* S = sm;             // [m][dv+1]
    float* xq = S + m * dp;    // [d]
    float* xk = xq + d;        // [d]
    float* xv = xk + d;        // [dv]
    float* fq = xv + dv;       // [m]
    float* rs = fq + m;        // [dv+1] readout sums
    float* red = rs + dp;      // [32]
    float* ws = red + 32;      // [m][d+1] omega rows (when they fit)
    const int bh = blockIdx.x, h = bh % H, tid = threadIdx.x, nt = blockDim.x;
    // state in: m*(dv+1) is a multiple of 4 (m is a multiple of 16), and so is every head's offset
    const int n4 = m * dp / 4;
    const float4* st4 = reinterpret_cast<const float4*>(state + (size_t)bh * m * dp);
    for (int i = tid; i < n4; i += nt) {
        const float4 x = st4[i];
        S[4 * i] = x.x; S[4 * i + 1] = x.y; S[4 * i + 2] = x.z; S[4 * i + 3] = x.w;
    }
    const float* wg = omega + (size_t)h * m * d;
    if (omega_in_smem) {
        const float4* w4 = reinterpret_cast<const float4*>(wg);   // m*d is a multiple of 4
        for (int i = tid; i < m * d / 4; i += nt) {
            const float4 x = w4[i];
            const int e = 4 * i, r = e / d, c = e - r * d;      // d is a multiple of 4: one row per float4
            float* o = ws + r * wp + c;
            o[0] = x.x; o[1] = x.y; o[2] = x.z; o[3] = x.w;
        }
    }
    const float inv_sqrt_m = 1.f / sqrtf((float)(KIND == FAVOR_KERNEL_SOFTMAX_TRIG ? m / 2 : m));
    const float kap = kshift[h];
    const int rr = tid < m ? tid : 0;
    for (int t = 0; t < Tn; ++t) {
        const size_t row = (size_t)bh * Tn + t;
        __syncthreads();   // the previous token's readout is done with fq, rs and S (and the staging is done)
        for (int i = tid; i < d; i += nt) {
            xq[i] = ldf(q + row * d + i);
            xk[i] = ldf(k + row * d + i);
        }
        for (int i = tid; i < dv; i += nt) xv[i] = ldf(v + row * dv + i);
        __syncthreads();
        float pq = 0.f, pk = 0.f, nk = 0.f;
        if (tid < m) {
            if (omega_in_smem) {
                const float* w = ws + rr * wp;
                for (int c = 0; c < d; ++c) {
                    pq = fmaf(w[c], xq[c], pq);
                    pk = fmaf(w[c], xk[c], pk);
                    nk = fmaf(xk[c], xk[c], nk);
                }
            } else {
                const float* w = wg + (size_t)rr * d;
                for (int c = 0; c < d; ++c) {
                    const float wc = __ldg(w + c);
                    pq = fmaf(wc, xq[c], pq);
                    pk = fmaf(wc, xk[c], pk);
                    nk = fmaf(xk[c], xk[c], nk);
                }
            }
        }
        const float qx = s * pq;
        const float mx = KIND == FAVOR_KERNEL_SOFTMAX_POS ? block_max(tid < m ? qx : -INFINITY, red) : 0.f;
        if (tid < m) {
            // the state holds the plain features (m^-1/2, or (m/2)^-1/2 for the
            // trigonometric map); the query side drops row-common factors.
            const float fk = inv_sqrt_m * key_feat<KIND>(pk, nk, s, kap, tid, m);
            const float f = query_feat<KIND>(qx, mx, tid, m);   // mx: a per-query shift, cancels
            float* Sr = S + tid * dp;
            if (gate) {   // RFA-Gate: S = g S + (1 - g) phi(k) [v 1]^T
                const float g = gate[row], fb = (1.f - g) * fk;
                for (int e = 0; e < dv; ++e) Sr[e] = fmaf(g, Sr[e], fb * xv[e]);
                Sr[dv] = fmaf(g, Sr[dv], fb);
            } else {
                for (int e = 0; e < dv; ++e) Sr[e] = fmaf(fk, xv[e], Sr[e]);
                Sr[dv] += fk;
            }
            fq[tid] = f;
        }
        __syncthreads();
        if (tid <= dv) {
            float acc = 0.f;
            for (int r = 0; r < m; ++r) acc = fmaf(fq[r], S[r * dp + tid], acc);
            rs[tid] = acc;
        }
        __syncthreads();
        if (tid < dv) {
            const float den = rs[dv];
            stf(out + row * dv + tid, den != 0.f ? rs[tid] / den : 0.f);
        }
    }
    __syncthreads();
    float4* so4 = reinterpret_cast<float4*>(state + (size_t)bh * m * dp);
    for (int i = tid; i < n4; i += nt) so4[i] = make_float4(S[4 * i], S[4 * i + 1], S[4 * i + 2], S[4 * i + 3]);
}

template <typename T, int KIND>
favor_status causal_step_t(const Handle& h, const void* q, const void* k, const void* v, void* out, float* state,
                           int BH, int Tn, cudaStream_t st, const float* gate) {
    const size_t base = (size_t)(h.m * (h.dv + 1) + 2 * h.d + h.dv + h.m + (h.dv + 1) + 32) * sizeof(float);
    const size_t wbytes = (size_t)h.m * (h.d + 1) * sizeof(float);
    const int in_smem = base + wbytes <= 200 * 1024 ? 1 : 0;
    const size_t smem = base + (in_smem ? wbytes : 0);
    auto kern = k_causal_step<T, KIND>;
    set_smem(kern, smem);
    ProfScope ps(h, PROF_CAUSAL, st);
    kern<<<BH, 256, smem, st>>>((const T*)q, (const T*)k, (const T*)v, (T*)out, state, h.omega_f32, h.kshift, h.H,
                                Tn, h.m, h.d, h.dv, h.s, in_smem, gate);
    count_launch();
    return check_launch("causal step kernel");
}

}  // namespace

favor_status simt_state_partials(const Handle& h, const void* k, const void* v, int BH, int L, const SegPlan& p,
                                 cudaStream_t st) {
    const RelposArgs rp;
    return dispatch3<StateF>(h, k, v, BH, L, &p, &rp, st);
}

favor_status simt_kv_state(const Handle& h, const void* k, const void* v, float* state, int B, int L,
                           cudaStream_t st) {
    const int BH = B * h.H;
    SegPlan p = plan_segments(BH, L, h.num_sms);
    const RelposArgs rp;
    favor_status s = dispatch3<StateF>(h, k, v, BH, L, (const SegPlan*)&p, &rp, st);
    if (s != FAVOR_OK) return s;
    const int n = h.m * (h.dv + 1);
    dim3 grid((n + 255) / 256, BH);
    ProfScope ps(h, PROF_COMBINE, st);
    const int m_norm = h.kind == FAVOR_KERNEL_SOFTMAX_TRIG ? h.m / 2 : h.m;   // the plain map's 1/sqrt
    k_accum_rows<<<grid, 256, 0, st>>>(h.ws_partial, state, p.n_seg, n, 1.f / sqrtf((float)m_norm));
    count_launch();
    return check_launch("state accumulate kernel");
}

favor_status simt_attn_from_state(const Handle& proto, const void* q, const float* state, void* out, int B, int L,
                                  cudaStream_t st) {
    Handle h = proto;
    h.ws_state = const_cast<float*>(state);   // the readout only reads it
    const int BH = B * h.H;
    FAVOR_KIND_DISPATCH(h, readout_t, h, q, out, BH, L, st);
}

favor_status simt_causal_step(const Handle& h, const void* q, const void* k, const void* v, void* out, float* state,
                              int B, int Tn, cudaStream_t st, const float* gate) {
    const int BH = B * h.H;
    FAVOR_KIND_DISPATCH(h, causal_step_t, h, q, k, v, out, state, BH, Tn, st, gate);
}

// ------------------------------------------------ bidirectional call, fixed scratch
// favor_attn_bidir_noalloc runs the CUDA-core bidirectional path above with no
// handle and no allocation: its scratch (per-head key shifts, per-segment
// partial states, reduced states) is one statically sized device array that
// is part of this library's device image.  Each device has its own copy; the
// address is looked up once per device with that device current.  No word of
// the array needs to start at zero: every word a call reads was written
// earlier in the same call.  Overlapping calls on one device share the array
// and race; order them on one stream.

static __device__ __align__(256) float g_fixed_scratch[kFixedScratchFloats];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_fixed_mu;
float* g_fixed_ptr[kMaxDevices] = {};

favor_status fixed_scratch_ptr(int dev, float** out) {
    if (dev < 0 || dev >= kMaxDevices)
        return set_error(FAVOR_ERR_UNSUPPORTED, "favor_attn_bidir_noalloc: device ordinal %d above %d", dev,
                         kMaxDevices - 1);
    std::lock_guard<std::mutex> lk(g_fixed_mu);
    if (!g_fixed_ptr[dev]) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_fixed_scratch);
        if (e != cudaSuccess || !p) {
            cudaGetLastError();
            return set_error(FAVOR_ERR_CUDA, "favor_attn_bidir_noalloc: cudaGetSymbolAddress: %s",
                             cudaGetErrorString(e));
        }
        g_fixed_ptr[dev] = static_cast<float*>(p);
    }
    *out = g_fixed_ptr[dev];
    return FAVOR_OK;
}

// kappa_h = max(0, max_r ||omega_r||^2/2 - KSHIFT_HEADROOM), one block per head.
__global__ void __launch_bounds__(256) k_key_shift(const float* __restrict__ omega, float* __restrict__ kshift,
                                                   int m, int d) {
    __shared__ float red[8];
    const int h = blockIdx.x;
    float mx = 0.f;
    for (int r = threadIdx.x; r < m; r += blockDim.x) {
        const float* w = omega + ((size_t)h * m + r) * d;
        float a = 0.f;
        for (int c = 0; c < d; ++c) a = fmaf(w[c], w[c], a);
        mx = fmaxf(mx, a);
    }
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = red[0];
        for (int w = 1; w < (int)(blockDim.x >> 5); ++w) t = fmaxf(t, red[w]);
        kshift[h] = fmaxf(0.f, 0.5f * t - KSHIFT_HEADROOM);
    }
}

}  // namespace

size_t fixed_scratch_floats(int H, int BH, int m, int dv, int n_seg) {
    const size_t hpad = ((size_t)H + 63) / 64 * 64;
    return hpad + (size_t)BH * m * (dv + 1) * (size_t)(1 + n_seg);
}

favor_status simt_bidir_fixed_scratch(const Handle& proto, const void* q, const void* k, const void* v,
                                      void* out, int B, int L, cudaStream_t st) {
    float* base = nullptr;
    favor_status s = fixed_scratch_ptr(proto.device, &base);
    if (s != FAVOR_OK) return s;
    const int BH = B * proto.H;
    SegPlan p = plan_segments(BH, L, proto.num_sms);
    const size_t per_seg = (size_t)BH * proto.m * (proto.dv + 1);
    const size_t hpad = fixed_scratch_floats(proto.H, BH, proto.m, proto.dv, 0) - per_seg;
    if (kFixedScratchFloats < hpad + 2 * per_seg)
        return set_error(FAVOR_ERR_UNSUPPORTED, "favor_attn_bidir_noalloc: B*H*m*(dv+1) too large for the fixed scratch");
    const int max_seg = (int)((kFixedScratchFloats - hpad) / per_seg - 1);
    if (p.n_seg > max_seg) {
        p.seg_tiles = (p.tiles + max_seg - 1) / max_seg;
        p.n_seg = (p.tiles + p.seg_tiles - 1) / p.seg_tiles;
    }
    Handle h = proto;
    h.kshift = base;
    h.ws_state = base + hpad;
    h.ws_partial = h.ws_state + per_seg;
    h.ws_partial_rows = (size_t)BH * p.n_seg;
    h.prof = nullptr;
    k_key_shift<<<h.H, 256, 0, st>>>(h.omega_f32, h.kshift, h.m, h.d);
    count_launch();
    s = check_launch("key shift kernel");
    if (s != FAVOR_OK) return s;
    const RelposArgs rp;
    s = dispatch3<StateF>(h, k, v, BH, L, (const SegPlan*)&p, &rp, st);
    if (s != FAVOR_OK) return s;
    s = launch_reduce_segments(h, BH, p.n_seg, st);
    if (s != FAVOR_OK) return s;
    FAVOR_KIND_DISPATCH(h, readout_t, h, q, out, BH, L, st);
}

}  // namespace favor
