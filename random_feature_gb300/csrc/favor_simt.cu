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
#include "simt_common.cuh"

namespace favor {
namespace {

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

// Tiled shape of the CUDA-core segment kernels: tokens per tile and padded
// [v 1] / state row widths (16-byte rows for float4 access).
template <int DV>
struct FwdShape {
    static constexpr int TT = DV >= 128 ? 16 : 32;
    static constexpr int DVP = DV + 4;
    static constexpr int W = DV + 1;
};

__host__ __device__ inline int al4f(int n) { return (n + 3) & ~3; }

// ------------------------------------------------------- per-segment key state
// grid (n_seg, B*H), 256 threads.  Per tile of TT keys, thread `row` projects
// its omega row on every key (float4 row against broadcast key rows), takes
// the key feature and places it in slot pi^-j(row) (PermuteFormer; the
// identity otherwise); thread r then folds slot r's features into its state
// row in token order: S = a_j S + b_j f_j [v_j 1] (a = b = 1 without decay),
// and writes it to part[(bh*n_seg + seg)][r][0:dv+1].  With decay the product
// of the segment's a_j goes to segdecay[bh*n_seg + seg].
template <typename T, int KIND, int DV>
__global__ void __launch_bounds__(256) k_segment_state(const T* __restrict__ k, const T* __restrict__ v,
                                                       const float* __restrict__ omega,
                                                       const float* __restrict__ kshift, float* __restrict__ part,
                                                       int H, int L, int m, int d, float s, int seg_len, int n_seg,
                                                       const int* __restrict__ pcyc, const int4* __restrict__ pmeta,
                                                       const float* __restrict__ gate, const float* __restrict__ rdec,
                                                       float* __restrict__ segdecay, int async_stage) {
    using F = FwdShape<DV>;
    constexpr int TT = F::TT, DVP = F::DVP, W = F::W;
    extern __shared__ __align__(16) float sm[];
    const int MP = m + 1;
    float* ys = sm;                          // [TT][d]
    float* cs = ys + TT * d;                 // [TT][DVP]: v, 1, 0...
    float* fk = cs + TT * DVP;               // [TT][m+1] key features by slot
    float* kn = fk + al4f(TT * MP);          // [TT]
    float* ga = kn + TT;                     // [TT] a_j
    float* gb = ga + TT;                     // [TT] b_j
    uint8_t* rk = reinterpret_cast<uint8_t*>(gb + TT);   // raw k | v rows of the next tile (async staging)
    uint8_t* rv = rk + raw_rows_bytes<T>(TT, d);
    const int seg = blockIdx.x, bh = blockIdx.y, h = bh % H;
    const int r = threadIdx.x;
    const bool own = r < m;
    const float* om = omega + (size_t)h * m * d;
    const float kap = kshift[h];
    const size_t row0 = (size_t)bh * L;
    const bool decay = gate || rdec;
    const float rd = rdec ? rdec[h] : 1.f;
    float st[W];
#pragma unroll
    for (int e = 0; e < W; ++e) st[e] = 0.f;
    float A = 1.f;
    const int j0 = seg * seg_len, j1 = min(L, j0 + seg_len);
    PermCursor pc;
    pc.init_inv(pcyc, pmeta, h, m, own ? r : 0, j0);
    auto prefetch = [&](int t) {
        const int n = min(TT, j1 - t);
        prefetch_rows(k + row0 * d, rk, t, n, TT, d);
        prefetch_rows(v + row0 * DV, rv, t, n, TT, DV);
        cp_async_commit();
    };
    if (async_stage && j0 < j1) prefetch(j0);
    for (int t0 = j0; t0 < j1; t0 += TT) {
        const int nt = min(TT, j1 - t0);
        __syncthreads();
        if (async_stage) {
            cp_async_wait_all();
            __syncthreads();   // every thread's copies of this tile have landed
            unpack_rows<T>(rk, ys, TT, d, d, -1.f, nt);
            unpack_rows<T>(rv, cs, TT, DV, DVP, 1.f, nt);
        } else {
            stage_rows(k + row0 * d, ys, t0, nt, TT, d, d, -1.f);
            stage_rows(v + row0 * DV, cs, t0, nt, TT, DV, DVP, 1.f);
        }
        if (decay)
            for (int j = threadIdx.x; j < TT; j += blockDim.x) {
                float a = 1.f, b = 0.f;
                if (j < nt) token_decay(gate, row0 + t0 + j, rd, &a, &b);
                ga[j] = a;
                gb[j] = b;
            }
        __syncthreads();
        if (async_stage && t0 + TT < j1) prefetch(t0 + TT);   // lands while this tile computes
        key_norms(ys, kn, TT, d);
        __syncthreads();
        if (own) {
            float p[TT];
            project_regs<TT>(om, ys, r, d, p);
#pragma unroll
            for (int j = 0; j < TT; ++j) {
                fk[j * MP + pc.row(r)] = j < nt ? key_feat<KIND>(p[j], kn[j], s, kap, r, m) : 0.f;
                pc.prev();
            }
        }
        __syncthreads();
        if (own) {
#pragma unroll 1
            for (int j = 0; j < TT; ++j) {
                const float f = fk[j * MP + r];
                const float4* cj = reinterpret_cast<const float4*>(cs + j * DVP);
                float a = 1.f, fb = f;
                if (decay) {
                    a = ga[j];
                    fb = f * gb[j];
                    A *= a;
                }
#pragma unroll
                for (int e4 = 0; e4 < DV / 4; ++e4) {
                    const float4 c = cj[e4];
                    st[4 * e4 + 0] = fmaf(a, st[4 * e4 + 0], fb * c.x);
                    st[4 * e4 + 1] = fmaf(a, st[4 * e4 + 1], fb * c.y);
                    st[4 * e4 + 2] = fmaf(a, st[4 * e4 + 2], fb * c.z);
                    st[4 * e4 + 3] = fmaf(a, st[4 * e4 + 3], fb * c.w);
                }
                st[DV] = fmaf(a, st[DV], fb);
            }
        }
    }
    if (own) {
        float* o = part + ((size_t)bh * n_seg + seg) * m * W + (size_t)r * W;
#pragma unroll
        for (int e = 0; e < W; ++e) o[e] = st[e];
        if (segdecay && r == 0) segdecay[(size_t)bh * n_seg + seg] = A;
    }
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
// grid (n_seg, B*H), 512 threads.  The state [m][dv+1] (row-major, fp32) is
// staged once per CTA; per tile of TT queries: projections (thread (r, half)
// takes feature row r for its half of the tile's queries), row shift,
// features placed by slot, den by one warp per query, and out_j[e..e+3] for
// two queries per thread as sums over the features.
template <typename T, int KIND, int DV>
__global__ void __launch_bounds__(512) k_readout(const T* __restrict__ q, const float* __restrict__ state,
                                                 const float* __restrict__ omega, T* __restrict__ out,
                                                 int H, int L, int m, int d, float s, int seg_len, int n_seg,
                                                 const int* __restrict__ pcyc, const int4* __restrict__ pmeta,
                                                 int async_stage) {
    using F = FwdShape<DV>;
    constexpr int TT = F::TT, DVP = F::DVP, W = F::W;
    extern __shared__ __align__(16) float sm[];
    const int MP = m + 1;
    float* ss = sm;                          // [m][DVP] state rows
    float* xs = ss + m * DVP;                // [TT][d]
    float* raw = xs + TT * d;                // [TT][m+1] s * projections
    float* fq = raw + al4f(TT * MP);         // [TT][m+1] features by slot
    float* cq = fq + al4f(TT * MP);          // [TT]
    float* den = cq + TT;                    // [TT]
    uint8_t* rq = reinterpret_cast<uint8_t*>(den + TT);   // raw q rows of the next tile (async staging)
    constexpr int TH = TT / 2;               // queries of a tile per half
    const int seg = blockIdx.x, bh = blockIdx.y, h = bh % H;
    const int r = threadIdx.x & 255, hf = threadIdx.x >> 8;
    const bool own = r < m;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    const float* om = omega + (size_t)h * m * d;
    const size_t row0 = (size_t)bh * L;
    {
        const float* sg = state + (size_t)bh * m * W;
        for (int idx = threadIdx.x; idx < m * DVP; idx += blockDim.x) {
            const int rr = idx / DVP, e = idx - rr * DVP;
            ss[idx] = e < W ? sg[rr * W + e] : 0.f;
        }
    }
    const int j0 = seg * seg_len, j1 = min(L, j0 + seg_len);
    PermCursor pc;
    pc.init_inv(pcyc, pmeta, h, m, own ? r : 0, j0);
    auto prefetch = [&](int t) {
        prefetch_rows(q + row0 * d, rq, t, min(TT, j1 - t), TT, d);
        cp_async_commit();
    };
    if (async_stage && j0 < j1) prefetch(j0);
    for (int t0 = j0; t0 < j1; t0 += TT) {
        const int nt = min(TT, j1 - t0);
        __syncthreads();
        if (async_stage) {
            cp_async_wait_all();
            __syncthreads();   // every thread's copies of this tile have landed
            unpack_rows<T>(rq, xs, TT, d, d, -1.f, nt);
        } else {
            stage_rows(q + row0 * d, xs, t0, nt, TT, d, d, -1.f);
        }
        __syncthreads();
        if (async_stage && t0 + TT < j1) prefetch(t0 + TT);   // lands while this tile computes
        float p[TH];
        const int jb = hf * TH;   // this half's first query of the tile
        if (own) {
            project_regs<TH>(om, xs + jb * d, r, d, p);
#pragma unroll
            for (int j = 0; j < TH; ++j) raw[(jb + j) * MP + r] = s * p[j];
        }
        __syncthreads();
        if (KIND == FAVOR_KERNEL_SOFTMAX_POS) {
            row_shift(raw, cq, TT, nt, m);
            __syncthreads();
        }
        if (own) {
            // the cursor walks every query of the tile: half 1 passes half 0's first
            if (hf)
                for (int j = 0; j < TH; ++j) pc.prev();
#pragma unroll
            for (int jj = 0; jj < TH; ++jj) {
                const int j = jb + jj;
                const float mx = KIND == FAVOR_KERNEL_SOFTMAX_POS ? cq[j] : 0.f;
                fq[j * MP + pc.row(r)] = j < nt ? query_feat<KIND>(s * p[jj], mx, r, m) : 0.f;
                pc.prev();
            }
            if (!hf)
                for (int j = 0; j < TH; ++j) pc.prev();
        }
        __syncthreads();
        for (int j = warp; j < TT; j += nw) {
            float a = 0.f;
            for (int rr = lane; rr < m; rr += 32) a = fmaf(fq[j * MP + rr], ss[rr * DVP + DV], a);
            a = warp_sum(a);
            if (lane == 0) den[j] = a;
        }
        __syncthreads();
        for (int idx = threadIdx.x; idx < (TT / 2) * (DV / 4); idx += blockDim.x) {
            const int jp = idx / (DV / 4), e4 = idx - jp * (DV / 4);
            const int ja = 2 * jp, jb = ja + 1;
            float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0;
#pragma unroll 4
            for (int rr = 0; rr < m; ++rr) {
                const float4 sv = *reinterpret_cast<const float4*>(ss + rr * DVP + 4 * e4);
                const float f0 = fq[ja * MP + rr], f1 = fq[jb * MP + rr];
                a0.x = fmaf(f0, sv.x, a0.x); a0.y = fmaf(f0, sv.y, a0.y);
                a0.z = fmaf(f0, sv.z, a0.z); a0.w = fmaf(f0, sv.w, a0.w);
                a1.x = fmaf(f1, sv.x, a1.x); a1.y = fmaf(f1, sv.y, a1.y);
                a1.z = fmaf(f1, sv.z, a1.z); a1.w = fmaf(f1, sv.w, a1.w);
            }
            if (ja < nt) {
                const float dn = den[ja];
                T* o = out + (row0 + t0 + ja) * DV + 4 * e4;
                stf(o + 0, dn != 0.f ? a0.x / dn : 0.f); stf(o + 1, dn != 0.f ? a0.y / dn : 0.f);
                stf(o + 2, dn != 0.f ? a0.z / dn : 0.f); stf(o + 3, dn != 0.f ? a0.w / dn : 0.f);
            }
            if (jb < nt) {
                const float dn = den[jb];
                T* o = out + (row0 + t0 + jb) * DV + 4 * e4;
                stf(o + 0, dn != 0.f ? a1.x / dn : 0.f); stf(o + 1, dn != 0.f ? a1.y / dn : 0.f);
                stf(o + 2, dn != 0.f ? a1.z / dn : 0.f); stf(o + 3, dn != 0.f ? a1.w / dn : 0.f);
            }
        }
    }
}

// --------------------------------------------------------- causal, per segment
// grid (n_seg, B*H), 512 threads: thread (r, half) owns feature row r for the
// tokens of its half of each tile (projections, features) and half of the
// state row's columns (update).  The state at the tile start (the segment's
// exclusive prefix, then carried) lives in shared memory; per tile of TT
// tokens (the chunked form of App. B.1 Eq. 11):
//   num_j = P_j phi~_q(j) S + sum_{i<=j} D_ji (phi~_q(j) . phi~_k(i)) [v_i 1],
//   S <- P_tile S + sum_i w_i phi~_k(i) [v_i 1]^T,
// with the decay weights P_j = prod_{l<=j} a_l, D_ji = b_i prod_{i<l<=j} a_l,
// w_i = D_{last,i} and P_tile = prod_l a_l (all 1 without decay), out_j =
// num_j / den_j (den the last column).  No per-token block reductions.
template <typename T, int KIND, int DV>
__global__ void __launch_bounds__(512) k_causal_segment(const T* __restrict__ q, const T* __restrict__ k,
                                                        const T* __restrict__ v, const float* __restrict__ omega,
                                                        const float* __restrict__ kshift,
                                                        const float* __restrict__ prefix, T* __restrict__ out,
                                                        int H, int L, int m, int d, float s, int seg_len, int n_seg,
                                                        const int* __restrict__ pcyc, const int4* __restrict__ pmeta,
                                                        const float* __restrict__ gate,
                                                        const float* __restrict__ rdec, int async_stage) {
    using F = FwdShape<DV>;
    constexpr int TT = F::TT, DVP = F::DVP, W = F::W;
    extern __shared__ __align__(16) float sm[];
    const int MP = m + 1;
    float* ss = sm;                          // [m][DVP] state at the tile start
    float* xs = ss + m * DVP;                // [TT][d] queries
    float* ys = xs + TT * d;                 // [TT][d] keys
    float* cs = ys + TT * d;                 // [TT][DVP] v, 1, 0...
    float* raw = cs + TT * DVP;              // [TT][m+1] s * query projections
    float* fq = raw + al4f(TT * MP);         // [TT][m+1] query features by slot
    float* fk = fq + al4f(TT * MP);          // [TT][m+1] key features by slot
    float* aa = fk + al4f(TT * MP);          // [TT][TT+1] D_ji phi_q(j).phi_k(i), i <= j
    float* cq = aa + al4f(TT * (TT + 1));    // [TT]
    float* den = cq + TT;                    // [TT]
    float* kn = den + TT;                    // [TT]
    float* ga = kn + TT;                     // [TT] a_j
    float* gb = ga + TT;                     // [TT] b_j
    float* pj = gb + TT;                     // [TT] P_j
    float* wi = pj + TT;                     // [TT] w_i
    float* pt = wi + TT;                     // [4] P_tile
    uint8_t* rq = reinterpret_cast<uint8_t*>(pt + 4);   // raw q | k | v rows of the next tile (async staging)
    uint8_t* rk = rq + raw_rows_bytes<T>(TT, d);
    uint8_t* rv = rk + raw_rows_bytes<T>(TT, d);
    constexpr int TH = TT / 2;               // tokens of a tile per half
    const int seg = blockIdx.x, bh = blockIdx.y, h = bh % H;
    const int r = threadIdx.x & 255, hf = threadIdx.x >> 8;
    const bool own = r < m;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    const float* om = omega + (size_t)h * m * d;
    const float kap = kshift[h];
    const size_t row0 = (size_t)bh * L;
    const bool decay = gate || rdec;
    const float rd = rdec ? rdec[h] : 1.f;
    {
        const float* pre = prefix + ((size_t)bh * n_seg + seg) * m * W;
        for (int idx = threadIdx.x; idx < m * DVP; idx += blockDim.x) {
            const int rr = idx / DVP, e = idx - rr * DVP;
            ss[idx] = e < W ? pre[rr * W + e] : 0.f;
        }
    }
    const int j0 = seg * seg_len, j1 = min(L, j0 + seg_len);
    PermCursor pc;
    pc.init_inv(pcyc, pmeta, h, m, own ? r : 0, j0);
    auto prefetch = [&](int t) {
        const int n = min(TT, j1 - t);
        prefetch_rows(q + row0 * d, rq, t, n, TT, d);
        prefetch_rows(k + row0 * d, rk, t, n, TT, d);
        prefetch_rows(v + row0 * DV, rv, t, n, TT, DV);
        cp_async_commit();
    };
    if (async_stage && j0 < j1) prefetch(j0);
    for (int t0 = j0; t0 < j1; t0 += TT) {
        const int nt = min(TT, j1 - t0);
        __syncthreads();   // the previous tile's state update is done
        if (async_stage) {
            cp_async_wait_all();
            __syncthreads();   // every thread's copies of this tile have landed
            unpack_rows<T>(rq, xs, TT, d, d, -1.f, nt);
            unpack_rows<T>(rk, ys, TT, d, d, -1.f, nt);
            unpack_rows<T>(rv, cs, TT, DV, DVP, 1.f, nt);
        } else {
            stage_rows(q + row0 * d, xs, t0, nt, TT, d, d, -1.f);
            stage_rows(k + row0 * d, ys, t0, nt, TT, d, d, -1.f);
            stage_rows(v + row0 * DV, cs, t0, nt, TT, DV, DVP, 1.f);
        }
        for (int j = threadIdx.x; j < TT; j += blockDim.x) {
            float a = 1.f, b = j < nt ? 1.f : 0.f;
            if (decay && j < nt) token_decay(gate, row0 + t0 + j, rd, &a, &b);
            ga[j] = a;
            gb[j] = b;
        }
        __syncthreads();
        if (async_stage && t0 + TT < j1) prefetch(t0 + TT);   // lands while this tile computes
        key_norms(ys, kn, TT, d);
        if (threadIdx.x == 32 * (nw - 1)) {   // decay weights, one thread (TT <= 32 steps)
            float P = 1.f;
            for (int j = 0; j < TT; ++j) {
                P *= ga[j];
                pj[j] = P;
            }
            pt[0] = P;
            float tail = 1.f;
            for (int i = TT - 1; i >= 0; --i) {
                wi[i] = gb[i] * tail;
                tail *= ga[i];
            }
        }
        float pq[TH], pk[TH];
        const int jb = hf * TH;   // this half's first token of the tile
        if (own) {
            project_regs<TH>(om, xs + jb * d, r, d, pq);
            project_regs<TH>(om, ys + jb * d, r, d, pk);
#pragma unroll
            for (int j = 0; j < TH; ++j) raw[(jb + j) * MP + r] = s * pq[j];
        }
        __syncthreads();
        if (KIND == FAVOR_KERNEL_SOFTMAX_POS) {
            row_shift(raw, cq, TT, nt, m);
            __syncthreads();
        }
        if (own) {
            // the cursor walks every token of the tile: half 1 passes half 0's first
            if (hf)
                for (int j = 0; j < TH; ++j) pc.prev();
#pragma unroll
            for (int jj = 0; jj < TH; ++jj) {
                const int j = jb + jj;
                const int slot = pc.row(r);   // query and key at one position share pi^j
                const float mx = KIND == FAVOR_KERNEL_SOFTMAX_POS ? cq[j] : 0.f;
                fq[j * MP + slot] = j < nt ? query_feat<KIND>(s * pq[jj], mx, r, m) : 0.f;
                fk[j * MP + slot] = j < nt ? key_feat<KIND>(pk[jj], kn[j], s, kap, r, m) : 0.f;
                pc.prev();
            }
            if (!hf)
                for (int j = 0; j < TH; ++j) pc.prev();
        }
        __syncthreads();
        for (int idx = threadIdx.x; idx < TT * (TT + 1) / 2; idx += blockDim.x) {   // pairs i <= j only
            int j, i;
            tri_pair(idx, j, i);
            float a = 0.f;
            for (int rr = 0; rr < m; ++rr) a = fmaf(fq[j * MP + rr], fk[i * MP + rr], a);
            float wgt = gb[i];
            for (int l = i + 1; l <= j; ++l) wgt *= ga[l];
            aa[j * (TT + 1) + i] = a * wgt;
        }
        __syncthreads();
        for (int j = warp; j < TT; j += nw) {
            float a = 0.f;
            for (int rr = lane; rr < m; rr += 32) a = fmaf(fq[j * MP + rr], ss[rr * DVP + DV], a);
            a *= pj[j];
            if (lane <= j && lane < TT) a += aa[j * (TT + 1) + lane];
            a = warp_sum(a);
            if (lane == 0) den[j] = a;
        }
        __syncthreads();
        for (int idx = threadIdx.x; idx < (TT / 2) * (DV / 4); idx += blockDim.x) {
            const int jp = idx / (DV / 4), e4 = idx - jp * (DV / 4);
            const int ja = 2 * jp, jb = ja + 1;
            float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0;
#pragma unroll 4
            for (int rr = 0; rr < m; ++rr) {
                const float4 sv = *reinterpret_cast<const float4*>(ss + rr * DVP + 4 * e4);
                const float f0 = fq[ja * MP + rr], f1 = fq[jb * MP + rr];
                a0.x = fmaf(f0, sv.x, a0.x); a0.y = fmaf(f0, sv.y, a0.y);
                a0.z = fmaf(f0, sv.z, a0.z); a0.w = fmaf(f0, sv.w, a0.w);
                a1.x = fmaf(f1, sv.x, a1.x); a1.y = fmaf(f1, sv.y, a1.y);
                a1.z = fmaf(f1, sv.z, a1.z); a1.w = fmaf(f1, sv.w, a1.w);
            }
            const float p0 = pj[ja], p1 = pj[jb];
            a0.x *= p0; a0.y *= p0; a0.z *= p0; a0.w *= p0;
            a1.x *= p1; a1.y *= p1; a1.z *= p1; a1.w *= p1;
            for (int i = 0; i <= jb; ++i) {
                const float4 c = *reinterpret_cast<const float4*>(cs + i * DVP + 4 * e4);
                const float w0 = i <= ja ? aa[ja * (TT + 1) + i] : 0.f, w1 = aa[jb * (TT + 1) + i];
                a0.x = fmaf(w0, c.x, a0.x); a0.y = fmaf(w0, c.y, a0.y);
                a0.z = fmaf(w0, c.z, a0.z); a0.w = fmaf(w0, c.w, a0.w);
                a1.x = fmaf(w1, c.x, a1.x); a1.y = fmaf(w1, c.y, a1.y);
                a1.z = fmaf(w1, c.z, a1.z); a1.w = fmaf(w1, c.w, a1.w);
            }
            if (ja < nt) {
                const float dn = den[ja];
                T* o = out + (row0 + t0 + ja) * DV + 4 * e4;
                stf(o + 0, dn != 0.f ? a0.x / dn : 0.f); stf(o + 1, dn != 0.f ? a0.y / dn : 0.f);
                stf(o + 2, dn != 0.f ? a0.z / dn : 0.f); stf(o + 3, dn != 0.f ? a0.w / dn : 0.f);
            }
            if (jb < nt) {
                const float dn = den[jb];
                T* o = out + (row0 + t0 + jb) * DV + 4 * e4;
                stf(o + 0, dn != 0.f ? a1.x / dn : 0.f); stf(o + 1, dn != 0.f ? a1.y / dn : 0.f);
                stf(o + 2, dn != 0.f ? a1.z / dn : 0.f); stf(o + 3, dn != 0.f ? a1.w / dn : 0.f);
            }
        }
        __syncthreads();   // every output read the state at the tile start
        if (own) {
            float wf[TT];
#pragma unroll
            for (int i = 0; i < TT; ++i) wf[i] = wi[i] * fk[i * MP + r];
            const float P = pt[0];
            float4* srow = reinterpret_cast<float4*>(ss + r * DVP);
            constexpr int G4 = DVP / 4, G0 = G4 / 2;   // float4 groups of the row: [0, G0) half 0, [G0, G4) half 1
#pragma unroll 1
            for (int e4 = hf ? G0 : 0; e4 < (hf ? G4 : G0); ++e4) {
                float4 a = srow[e4];
                a.x *= P; a.y *= P; a.z *= P; a.w *= P;
#pragma unroll
                for (int i = 0; i < TT; ++i) {
                    const float4 c = *reinterpret_cast<const float4*>(cs + i * DVP + 4 * e4);
                    a.x = fmaf(wf[i], c.x, a.x); a.y = fmaf(wf[i], c.y, a.y);
                    a.z = fmaf(wf[i], c.z, a.z); a.w = fmaf(wf[i], c.w, a.w);
                }
                srow[e4] = a;
            }
        }
    }
}

template <typename K>
static void set_smem(K kern, size_t bytes) {
    if (bytes > 48 * 1024) cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

// Asynchronous staging of a segment kernel's input tiles: on when every input
// is 16-byte aligned and the raw area (raw_bytes) still fits next to the
// kernel's buffers (base bytes); the returned size includes it when on.
static size_t with_raw(size_t base, size_t raw_bytes, bool aligned, int* async_stage) {
    *async_stage = aligned && base + raw_bytes <= 227 * 1024 ? 1 : 0;
    return *async_stage ? base + raw_bytes : base;
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
    using F = FwdShape<DV>;
    int as = 0;
    const size_t smem = with_raw(
        (size_t)(F::TT * h.d + F::TT * F::DVP + al4f(F::TT * (h.m + 1)) + 3 * F::TT) * sizeof(float),
        raw_rows_bytes<T>(F::TT, h.d) + raw_rows_bytes<T>(F::TT, DV), is_aligned16(k) && is_aligned16(v), &as);
    auto kern = k_segment_state<T, KIND, DV>;
    set_smem(kern, smem);
    dim3 grid(p.n_seg, BH);
    ProfScope ps(h, PROF_STATE, st);
    kern<<<grid, 256, smem, st>>>((const T*)k, (const T*)v, h.omega_f32, h.kshift, h.ws_partial, h.H, L, h.m,
                                  h.d, h.s, p.seg_tiles * 128, p.n_seg, rp.cyc, rp.meta, rp.gate, rp.rdec,
                                  rp.segdecay, as);
    count_launch();
    return check_launch("segment state kernel");
}

template <typename T, int KIND, int DV>
favor_status readout_dv(const Handle& h, const void* q, void* out, int BH, int L, cudaStream_t st,
                        const RelposArgs& rp) {
    using F = FwdShape<DV>;
    const SegPlan p = plan_segments(BH, L, h.num_sms);
    int as = 0;
    const size_t smem =
        with_raw((size_t)(h.m * F::DVP + F::TT * h.d + 2 * al4f(F::TT * (h.m + 1)) + 2 * F::TT) * sizeof(float),
                 raw_rows_bytes<T>(F::TT, h.d), is_aligned16(q), &as);
    auto kern = k_readout<T, KIND, DV>;
    set_smem(kern, smem);
    dim3 grid(p.n_seg, BH);
    ProfScope ps(h, PROF_READOUT, st);
    kern<<<grid, 512, smem, st>>>((const T*)q, h.ws_state, h.omega_f32, (T*)out, h.H, L, h.m, h.d, h.s,
                                  p.seg_tiles * 128, p.n_seg, rp.cyc, rp.meta, as);
    count_launch();
    return check_launch("readout kernel");
}

template <typename T, int KIND>
favor_status readout_t(const Handle& h, const void* q, void* out, int BH, int L, cudaStream_t st,
                       const RelposArgs& rp = RelposArgs()) {
    switch (h.dv) {
        case 16: return readout_dv<T, KIND, 16>(h, q, out, BH, L, st, rp);
        case 32: return readout_dv<T, KIND, 32>(h, q, out, BH, L, st, rp);
        case 64: return readout_dv<T, KIND, 64>(h, q, out, BH, L, st, rp);
        case 128: return readout_dv<T, KIND, 128>(h, q, out, BH, L, st, rp);
    }
    return set_error(FAVOR_ERR_UNSUPPORTED, "readout: unsupported dv=%d", h.dv);
}

template <typename T, int KIND, int DV>
favor_status causal_t(const Handle& h, const void* q, const void* k, const void* v, void* out, int BH, int L,
                      const SegPlan& p, const RelposArgs& rp, cudaStream_t st) {
    using F = FwdShape<DV>;
    const int TT = F::TT;
    const size_t base = (size_t)(h.m * F::DVP + 2 * TT * h.d + TT * F::DVP + 3 * al4f(TT * (h.m + 1)) +
                                 al4f(TT * (TT + 1)) + 8 * TT + 4) * sizeof(float);
    if (base > 227 * 1024)
        return set_error(FAVOR_ERR_UNSUPPORTED, "causal: %zu bytes of shared memory", base);
    int as = 0;
    const size_t smem = with_raw(base, 2 * raw_rows_bytes<T>(TT, h.d) + raw_rows_bytes<T>(TT, DV),
                                 is_aligned16(q) && is_aligned16(k) && is_aligned16(v), &as);
    auto kern = k_causal_segment<T, KIND, DV>;
    set_smem(kern, smem);
    dim3 grid(p.n_seg, BH);
    ProfScope ps(h, PROF_CAUSAL, st);
    kern<<<grid, 512, smem, st>>>((const T*)q, (const T*)k, (const T*)v, h.omega_f32, h.kshift, h.ws_partial,
                                  (T*)out, h.H, L, h.m, h.d, h.s, p.seg_tiles * 128, p.n_seg, rp.cyc, rp.meta,
                                  rp.gate, rp.rdec, as);
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
                const float4* w4 = reinterpret_cast<const float4*>(wg + (size_t)rr * d);   // d is a multiple of 16
                for (int c4 = 0; c4 < d / 4; ++c4) {
                    const float4 w = __ldg(w4 + c4);
                    const int c = 4 * c4;
                    pq = fmaf(w.x, xq[c], fmaf(w.y, xq[c + 1], fmaf(w.z, xq[c + 2], fmaf(w.w, xq[c + 3], pq))));
                    pk = fmaf(w.x, xk[c], fmaf(w.y, xk[c + 1], fmaf(w.z, xk[c + 2], fmaf(w.w, xk[c + 3], pk))));
                    nk = fmaf(xk[c], xk[c], fmaf(xk[c + 1], xk[c + 1], fmaf(xk[c + 2], xk[c + 2], fmaf(xk[c + 3], xk[c + 3], nk))));
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
        // readout sums rs[e] = sum_r fq[r] S[r][e]: one warp per column, lanes over features
        {
            const int warp = tid >> 5, lane = tid & 31, nw = nt >> 5;
            for (int e = warp; e <= dv; e += nw) {
                float acc = 0.f;
                for (int r = lane; r < m; r += 32) acc = fmaf(fq[r], S[r * dp + e], acc);
                acc = warp_sum(acc);
                if (lane == 0) rs[e] = acc;
            }
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

// The device address of g_fixed_scratch, looked up (cudaGetSymbolAddress) once
// per device and CUDA context: a context torn down and made again (for
// instance after cudaDeviceReset) loads the module anew, possibly elsewhere,
// so the cached address is only reused while the current context is the one
// it was taken in.
struct FixedScratchSlot {
    void* ctx;
    float* ptr;
};
FixedScratchSlot g_fixed[kMaxDevices] = {};

using CtxGetCurrentFn = int (*)(void**);
CtxGetCurrentFn ctx_get_current_fn() {
    static CtxGetCurrentFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(p);
        cudaGetLastError();
    });
    return fn;
}

favor_status fixed_scratch_ptr(int dev, float** out) {
    if (dev < 0 || dev >= kMaxDevices)
        return set_error(FAVOR_ERR_UNSUPPORTED, "favor_attn_bidir_noalloc: device ordinal %d above %d", dev,
                         kMaxDevices - 1);
    CtxGetCurrentFn get = ctx_get_current_fn();
    if (!get) return set_error(FAVOR_ERR_CUDA, "favor_attn_bidir_noalloc: cuCtxGetCurrent is not available");
    void* ctx = nullptr;
    if (get(&ctx) != 0) ctx = nullptr;   // null: no context is current yet
    std::lock_guard<std::mutex> lk(g_fixed_mu);
    if (ctx && g_fixed[dev].ptr && g_fixed[dev].ctx == ctx) {
        *out = g_fixed[dev].ptr;
        return FAVOR_OK;
    }
    // set-up: the lookup makes the device's primary context current if it was not
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_fixed_scratch);
    if (e != cudaSuccess || !p) {
        cudaGetLastError();
        return set_error(FAVOR_ERR_CUDA, "favor_attn_bidir_noalloc: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
    }
    if (get(&ctx) != 0 || !ctx) return set_error(FAVOR_ERR_CUDA, "favor_attn_bidir_noalloc: no current CUDA context");
    g_fixed[dev].ctx = ctx;
    g_fixed[dev].ptr = static_cast<float*>(p);
    *out = g_fixed[dev].ptr;
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
