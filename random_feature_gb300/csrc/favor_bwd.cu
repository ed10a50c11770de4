// Backward of FAVOR+ attention on the CUDA cores (FFMA): dq, dk, dv of the
// bidirectional and causal calls, for every supported shape, fp32 arithmetic.
//
// The gradients are the exact derivative of the forward of Rethinking Attention
// with Performers, App. B Alg. 1 (bidirectional) and App. B.1 Eq. 11 (causal).
// With C = [V 1], Buf2 = Q' (K'^T C) = [num den] and out = num / den:
//   D_i   = [dO_i / den_i,  -(dO_i . out_i) / den_i]      (0 where den_i == 0)
//   dQ'_i = G^PS_i D_i    with G^PS_i = sum_{j<=i} K'_j C_j^T (all j if bidirectional)
//   dK'_j = H_j C_j       with H_j    = sum_{i>=j} Q'_i D_i^T (all i if bidirectional)
//   dC_j  = H_j^T K'_j    (dv = its first dv columns)
// and through the feature maps (x = s*q):
//   positive  dq = s * (G Omega - x sum_r G_r),  G = dQ' * Q'   (elementwise)
//   ReLU      dq = s * (dQ'~ * [Omega x > 0]) Omega
// dO_i . out_i is not taken from the caller: with u_i = G^PS_i^T-applied dO_i,
// i.e. u_i[r] = sum_e G^PS_i[r][e] dO_i[e], it is sum_r phi_q(i)[r] u_i[r] / den_i,
// computed here in fp32 from the same features (the identity that makes
// sum_r G_r vanish then holds to fp32 rounding).
// The kernels use the same shifted features as the forward (a per-head key
// shift kappa_h, a per-query row shift, no m^-1/2); every product above pairs a
// feature with a quantity divided by the matching denominator, so the shifts
// cancel exactly, as they do in the forward output.
//
// Work split: every (batch, head) row of tokens is cut into the forward's
// segments; a segment is walked in tiles of TT tokens.  The query pass needs
// G^PS at each query (the forward's per-segment prefix states, plus the
// tile's own keys), the key pass needs H at each key (per-segment suffix sums
// of phi~_q D^T, plus the tile's own queries): the chunked form of Eq. 11, in
// which the within-tile terms are a masked TT x TT product and the rest is one
// state per tile.  Bidirectional calls are the same passes with a single full
// state and no within-tile terms.
#include <cmath>

#include "favor_internal.h"
#include "simt_common.cuh"

namespace favor {
namespace {

template <int DV>
struct BwdShape {
    static constexpr int TT = DV >= 128 ? 16 : 32;   // tokens per tile
    static constexpr int DVP = DV + 4;               // padded [V 1] / D row (16-byte rows)
    static constexpr int W = DV + 1;                 // state row width
};

// Shared-memory plan (floats) of one pass; every buffer starts 16-byte aligned.
struct BwdSmem {
    int xs, ys, cs, dd, fq, fk, ub, aa, mm, rs, zs, cq, den, go, kn, raw, total;
};

__host__ __device__ inline int al4(int n) { return (n + 3) & ~3; }

// raw_bytes: the asynchronous staging area of one tile's input rows (0: staged synchronously).
__host__ __device__ inline BwdSmem bwd_smem(int TT, int DVP, int W, int m, int d, bool causal, bool key_pass,
                                           int raw_bytes) {
    BwdSmem p;
    int o = 0;
    const int MP = m + 1;
    p.xs = o; o += al4(TT * d);                                   // query tile (raw)
    p.ys = o; o += al4(TT * d);                                   // key tile (raw)
    p.cs = o; o += al4(TT * DVP);                                 // [v 1 0 0 0] rows
    p.dd = o; o += al4(TT * DVP);                                 // dO, then D = [dnum dden]
    p.fq = o; o += al4(TT * MP);                                  // query features (then G on the query pass)
    p.fk = o; o += al4(TT * MP);                                  // key features (then G on the key pass)
    p.ub = o; o += key_pass ? 0 : al4(TT * MP);                   // u = G^PS dO (query pass)
    p.aa = o; o += causal ? al4(TT * (TT + 1)) : 0;               // masked phi_q . phi_k
    p.mm = o; o += causal ? al4(TT * (TT + 1)) : 0;               // masked dO . v (query) / D . C (key)
    p.rs = o; o += key_pass ? al4(m * DVP) : 0;                   // H at the tile end, value columns (key pass)
    p.zs = o; o += al4(m);                                        // z column of the query pass state
    p.cq = o; o += al4(TT);
    p.den = o; o += al4(TT);
    p.go = o; o += al4(TT);
    p.kn = o; o += al4(TT);
    p.raw = o; o += al4(raw_bytes / 4);
    p.total = o;
    return p;
}

// Raw staging bytes of one tile: the query pass reads q, dO (and k, v when
// causal), the key pass k, v (and q, dO and the per-query row statistics when
// causal).
template <typename T>
__host__ __device__ inline int bwd_raw_bytes(int TT, int d, int DV, bool causal, bool key_pass) {
    int b = raw_rows_bytes<T>(TT, d) + raw_rows_bytes<T>(TT, DV);
    if (causal) b *= 2;
    if (causal && key_pass) b += TT * 16;
    return b;
}

// D rows from dO (in place in dd), den and go: D = [dO/den, -go/den, 0...].
__device__ __forceinline__ void make_d(float* dd, const float* den, const float* go, int TT, int DV, int DVP) {
    for (int idx = threadIdx.x; idx < TT * DVP; idx += blockDim.x) {
        const int j = idx / DVP, e = idx - j * DVP;
        const float dn = den[j];
        float x = 0.f;
        if (dn != 0.f) {
            if (e < DV) x = dd[idx] / dn;
            else if (e == DV) x = -go[j] / dn;
        }
        dd[idx] = x;
    }
}

// dx rows from G (row stride m+1) for a tile: dx_j = s*(G_j Omega - s*x_j sum_r G_jr)
// (positive) or s*G_j Omega (ReLU), written as rows [t0, t0+nt) of dst; two
// tokens x four columns per thread (one float4 omega load feeds 8 FMAs; eight
// omega rows are in flight before the first use, m being a multiple of 16).
template <typename T, int KIND>
__device__ __forceinline__ void grad_inputs(const float* g, const float* xs, const float* __restrict__ om,
                                            T* __restrict__ dst, int t0, int nt, int TT, int m, int d, float s) {
    const int d4 = d >> 2;
    const float4* w4 = reinterpret_cast<const float4*>(om);
    for (int idx = threadIdx.x; idx < (TT / 2) * d4; idx += blockDim.x) {
        const int jp = idx / d4, c4 = idx - jp * d4;
        const int ja = 2 * jp, jb = ja + 1;
        if (ja >= nt) continue;
        float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0;
        float gs0 = 0.f, gs1 = 0.f;
        const float* g0 = g + ja * (m + 1);
        const float* g1 = g + jb * (m + 1);
#pragma unroll 1
        for (int r0 = 0; r0 < m; r0 += 8) {
            float4 w[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) w[u] = __ldg(w4 + (r0 + u) * d4 + c4);
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const float x0 = g0[r0 + u], x1 = g1[r0 + u];
                a0.x = fmaf(x0, w[u].x, a0.x); a0.y = fmaf(x0, w[u].y, a0.y);
                a0.z = fmaf(x0, w[u].z, a0.z); a0.w = fmaf(x0, w[u].w, a0.w);
                a1.x = fmaf(x1, w[u].x, a1.x); a1.y = fmaf(x1, w[u].y, a1.y);
                a1.z = fmaf(x1, w[u].z, a1.z); a1.w = fmaf(x1, w[u].w, a1.w);
                gs0 += x0;
                gs1 += x1;
            }
        }
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            const int j = ja + t;
            if (j >= nt) break;
            const float4 a = t == 0 ? a0 : a1;
            const float* xj = xs + j * d + 4 * c4;
            T* o = dst + (size_t)(t0 + j) * d + 4 * c4;
            if (KIND == FAVOR_KERNEL_SOFTMAX_POS) {
                const float u = s * (t == 0 ? gs0 : gs1);
                stf(o + 0, s * fmaf(-u, xj[0], a.x));
                stf(o + 1, s * fmaf(-u, xj[1], a.y));
                stf(o + 2, s * fmaf(-u, xj[2], a.z));
                stf(o + 3, s * fmaf(-u, xj[3], a.w));
            } else {
                stf(o + 0, s * a.x);
                stf(o + 1, s * a.y);
                stf(o + 2, s * a.z);
                stf(o + 3, s * a.w);
            }
        }
    }
}

// ------------------------------------------------------------ query pass
// grid (n_seg, B*H), blockDim = m rounded up to 32.  Thread r < m owns feature
// r: the state row (G^PS at the tile start, or the full S~ | z~) and the
// segment's running sum of phi~_q D^T.  Writes dq, the per-segment sums into
// part, and (causal) the per-query (den~, shift, dO . out) for the key pass.
template <typename T, int KIND, int DV, bool CAUSAL>
__global__ void __launch_bounds__(256) k_bwd_query(const T* __restrict__ q, const T* __restrict__ k,
                                                   const T* __restrict__ v, const T* __restrict__ dout,
                                                   T* __restrict__ dq, const float* __restrict__ omega,
                                                   const float* __restrict__ kshift, const float* __restrict__ state0,
                                                   float* __restrict__ part, float4* __restrict__ rowstat, int H,
                                                   int L, int m, int d, float s, int seg_len, int n_seg,
                                                   int async_stage) {
    using S = BwdShape<DV>;
    constexpr int TT = S::TT, DVP = S::DVP, W = S::W;
    extern __shared__ __align__(16) float sm[];
    const BwdSmem P =
        bwd_smem(TT, DVP, W, m, d, CAUSAL, false, async_stage ? bwd_raw_bytes<T>(TT, d, DV, CAUSAL, false) : 0);
    float *xs = sm + P.xs, *ys = sm + P.ys, *cs = sm + P.cs, *dd = sm + P.dd, *fq = sm + P.fq, *fk = sm + P.fk;
    float *ub = sm + P.ub, *aa = sm + P.aa, *mm = sm + P.mm, *zs = sm + P.zs, *cq = sm + P.cq, *den = sm + P.den,
          *go = sm + P.go, *kn = sm + P.kn;
    const int MP = m + 1;
    const int seg = blockIdx.x, bh = blockIdx.y, h = bh % H;
    const int r = threadIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    const bool own = r < m;
    const float* om = omega + (size_t)h * m * d;
    const float kap = kshift[h];
    const size_t row0 = (size_t)bh * L;

    float st[W], acc[W];
    {
        const float* s0 = state0 + (CAUSAL ? ((size_t)bh * n_seg + seg) : (size_t)bh) * m * W + (size_t)r * W;
#pragma unroll
        for (int e = 0; e < W; ++e) {
            st[e] = own ? s0[e] : 0.f;
            acc[e] = 0.f;
        }
    }
    const int j0 = seg * seg_len, j1 = min(L, j0 + seg_len);
    // asynchronous staging: raw q | dO | k | v rows of the next tile
    uint8_t* rq = reinterpret_cast<uint8_t*>(sm + P.raw);
    uint8_t* rdo = rq + raw_rows_bytes<T>(TT, d);
    uint8_t* rk = rdo + raw_rows_bytes<T>(TT, DV);
    uint8_t* rv = rk + raw_rows_bytes<T>(TT, d);
    auto prefetch = [&](int t) {
        const int n = min(TT, j1 - t);
        prefetch_rows(q + row0 * d, rq, t, n, TT, d);
        prefetch_rows(dout + row0 * DV, rdo, t, n, TT, DV);
        if (CAUSAL) {
            prefetch_rows(k + row0 * d, rk, t, n, TT, d);
            prefetch_rows(v + row0 * DV, rv, t, n, TT, DV);
        }
        cp_async_commit();
    };
    if (async_stage && j0 < j1) prefetch(j0);
    for (int t0 = j0; t0 < j1; t0 += TT) {
        const int nt = min(TT, j1 - t0);
        __syncthreads();   // the previous tile is done with every buffer
        if (async_stage) {
            cp_async_wait_all();
            __syncthreads();   // every thread's copies of this tile have landed
            unpack_rows<T>(rq, xs, TT, d, d, -1.f, nt);
            unpack_rows<T>(rdo, dd, TT, DV, DVP, -1.f, nt);
            if (CAUSAL) {
                unpack_rows<T>(rk, ys, TT, d, d, -1.f, nt);
                unpack_rows<T>(rv, cs, TT, DV, DVP, 1.f, nt);
            }
        } else {
            stage_rows(q + row0 * d, xs, t0, nt, TT, d, d, -1.f);
            stage_rows(dout + row0 * DV, dd, t0, nt, TT, DV, DVP, -1.f);
            if (CAUSAL) {
                stage_rows(k + row0 * d, ys, t0, nt, TT, d, d, -1.f);
                stage_rows(v + row0 * DV, cs, t0, nt, TT, DV, DVP, 1.f);
            }
        }
        __syncthreads();
        if (async_stage && t0 + TT < j1) prefetch(t0 + TT);   // lands while this tile computes
        if (CAUSAL) key_norms(ys, kn, TT, d);
        if (own) {
            project_tile<TT>(om, xs, fq, r, m, d, s);
            if (CAUSAL) project_tile<TT>(om, ys, fk, r, m, d, s);
            zs[r] = st[DV];
        }
        __syncthreads();
        if (KIND == FAVOR_KERNEL_SOFTMAX_POS) {
            row_shift(fq, cq, TT, nt, m);
            __syncthreads();
        }
        if (own) {
#pragma unroll 4
            for (int j = 0; j < TT; ++j) {
                const float pq = fq[j * MP + r];
                float f = 0.f;
                if (j < nt) f = KIND == FAVOR_KERNEL_SOFTMAX_POS ? expf(pq - cq[j]) : fmaxf(pq, 0.f);
                fq[j * MP + r] = f;
                if (CAUSAL) {
                    const float pk = fk[j * MP + r];
                    float g = 0.f;
                    if (j < nt)
                        g = KIND == FAVOR_KERNEL_SOFTMAX_POS ? expf(pk - 0.5f * s * s * kn[j] - kap) : fmaxf(pk, 0.f);
                    fk[j * MP + r] = g;
                }
            }
        }
        __syncthreads();
        if (CAUSAL) {   // aa[j][i] = phi~_q(j) . phi~_k(i), mm[j][i] = dO_j . v_i, for i <= j
            for (int idx = threadIdx.x; idx < TT * (TT + 1) / 2; idx += blockDim.x) {   // pairs i <= j only
                int j, i;
                tri_pair(idx, j, i);
                float a = 0.f, b = 0.f;
                {
                    for (int rr = 0; rr < m; ++rr) a = fmaf(fq[j * MP + rr], fk[i * MP + rr], a);
                    const float4* gj = reinterpret_cast<const float4*>(dd + j * DVP);
                    const float4* ci = reinterpret_cast<const float4*>(cs + i * DVP);
#pragma unroll 4
                    for (int e4 = 0; e4 < DVP / 4; ++e4) b += dot4(gj[e4], ci[e4]);
                }
                aa[j * (TT + 1) + i] = a;
                mm[j * (TT + 1) + i] = b;
            }
            __syncthreads();
        }
        // den~_j = phi~_q(j) . z(tile start) + sum_{i<=j} aa[j][i]
        for (int j = warp; j < TT; j += nw) {
            float a = 0.f;
            for (int rr = lane; rr < m; rr += 32) a = fmaf(fq[j * MP + rr], zs[rr], a);
            if (CAUSAL && lane <= j && lane < TT) a += aa[j * (TT + 1) + lane];
            a = warp_sum(a);
            if (lane == 0) den[j] = j < nt ? a : 0.f;
        }
        // u_j[r] = sum_e G^PS_j[r][e] dO_j[e] (value columns only)
        if (own) {
#pragma unroll 1
            for (int j = 0; j < TT; ++j) {
                const float4* gj = reinterpret_cast<const float4*>(dd + j * DVP);
                float u0 = 0.f, u1 = 0.f, u2 = 0.f, u3 = 0.f;   // independent partial sums
#pragma unroll
                for (int e4 = 0; e4 < DV / 4; ++e4) {
                    const float4 x = gj[e4];
                    u0 = fmaf(st[4 * e4 + 0], x.x, u0);
                    u1 = fmaf(st[4 * e4 + 1], x.y, u1);
                    u2 = fmaf(st[4 * e4 + 2], x.z, u2);
                    u3 = fmaf(st[4 * e4 + 3], x.w, u3);
                }
                if (CAUSAL) {
                    const float* mj = mm + j * (TT + 1);
                    int i = 0;
                    for (; i + 1 <= j; i += 2) {
                        u0 = fmaf(fk[i * MP + r], mj[i], u0);
                        u1 = fmaf(fk[(i + 1) * MP + r], mj[i + 1], u1);
                    }
                    if (i <= j) u2 = fmaf(fk[i * MP + r], mj[i], u2);
                }
                ub[j * MP + r] = (u0 + u1) + (u2 + u3);
            }
        }
        __syncthreads();
        // go_j = dO_j . out_j = phi~_q(j) . u_j / den~_j
        for (int j = warp; j < TT; j += nw) {
            float a = 0.f;
            for (int rr = lane; rr < m; rr += 32) a = fmaf(fq[j * MP + rr], ub[j * MP + rr], a);
            a = warp_sum(a);
            if (lane == 0) {
                const float dn = den[j];
                const float g = dn != 0.f ? a / dn : 0.f;
                go[j] = g;
                if (CAUSAL && j < nt)
                    rowstat[row0 + t0 + j] =
                        make_float4(dn, KIND == FAVOR_KERNEL_SOFTMAX_POS ? cq[j] : 0.f, g, 0.f);
            }
        }
        __syncthreads();
        make_d(dd, den, go, TT, DV, DVP);
        __syncthreads();
        if (own) {
            float zr = st[DV];   // z at query j: tile start plus the tile's keys i <= j
#pragma unroll 1
            for (int j = 0; j < TT; ++j) {
                const float f = fq[j * MP + r];
                if (CAUSAL) zr += fk[j * MP + r];
                const float4* dj = reinterpret_cast<const float4*>(dd + j * DVP);
#pragma unroll
                for (int e4 = 0; e4 < DV / 4; ++e4) {
                    const float4 x = dj[e4];
                    acc[4 * e4 + 0] = fmaf(f, x.x, acc[4 * e4 + 0]);
                    acc[4 * e4 + 1] = fmaf(f, x.y, acc[4 * e4 + 1]);
                    acc[4 * e4 + 2] = fmaf(f, x.z, acc[4 * e4 + 2]);
                    acc[4 * e4 + 3] = fmaf(f, x.w, acc[4 * e4 + 3]);
                }
                const float dz = dd[j * DVP + DV];   // -go_j / den_j
                acc[DV] = fmaf(f, dz, acc[DV]);
                const float dn = den[j];
                const float dphi = dn != 0.f ? fmaf(zr, dz, ub[j * MP + r] / dn) : 0.f;
                fq[j * MP + r] = KIND == FAVOR_KERNEL_SOFTMAX_POS ? dphi * f : (f > 0.f ? dphi : 0.f);
            }
            if (CAUSAL) {   // G^PS at the next tile start
#pragma unroll 1
                for (int i = 0; i < TT; ++i) {
                    const float g = fk[i * MP + r];
                    const float4* ci = reinterpret_cast<const float4*>(cs + i * DVP);
#pragma unroll
                    for (int e4 = 0; e4 < DV / 4; ++e4) {
                        const float4 x = ci[e4];
                        st[4 * e4 + 0] = fmaf(g, x.x, st[4 * e4 + 0]);
                        st[4 * e4 + 1] = fmaf(g, x.y, st[4 * e4 + 1]);
                        st[4 * e4 + 2] = fmaf(g, x.z, st[4 * e4 + 2]);
                        st[4 * e4 + 3] = fmaf(g, x.w, st[4 * e4 + 3]);
                    }
                    st[DV] += g;
                }
            }
        }
        __syncthreads();
        grad_inputs<T, KIND>(fq, xs, om, dq + row0 * d, t0, nt, TT, m, d, s);
    }
    if (own) {
        float* o = part + ((size_t)bh * n_seg + seg) * m * W + (size_t)r * W;
#pragma unroll
        for (int e = 0; e < W; ++e) o[e] = acc[e];
    }
}

// -------------------------------------------------------------- key pass
// grid (n_seg, B*H), blockDim = m rounded up to 32.  Thread r < m owns row r of
// H (the sum of phi~_q D^T over the queries after the current tile, or the
// full sum when bidirectional).  Causal segments are walked backwards.
template <typename T, int KIND, int DV, bool CAUSAL>
__global__ void __launch_bounds__(256) k_bwd_key(const T* __restrict__ q, const T* __restrict__ k,
                                                 const T* __restrict__ v, const T* __restrict__ dout,
                                                 T* __restrict__ dk, T* __restrict__ dvv,
                                                 const float* __restrict__ omega, const float* __restrict__ kshift,
                                                 const float* __restrict__ hstate, const float4* __restrict__ rowstat,
                                                 int H, int L, int m, int d, float s, int seg_len, int n_seg,
                                                 int async_stage) {
    using S = BwdShape<DV>;
    constexpr int TT = S::TT, DVP = S::DVP, W = S::W;
    extern __shared__ __align__(16) float sm[];
    const BwdSmem P =
        bwd_smem(TT, DVP, W, m, d, CAUSAL, true, async_stage ? bwd_raw_bytes<T>(TT, d, DV, CAUSAL, true) : 0);
    float *xs = sm + P.xs, *ys = sm + P.ys, *cs = sm + P.cs, *dd = sm + P.dd, *fq = sm + P.fq, *fk = sm + P.fk;
    float *aa = sm + P.aa, *mm = sm + P.mm, *rs = sm + P.rs, *cq = sm + P.cq, *den = sm + P.den, *go = sm + P.go,
          *kn = sm + P.kn;
    const int MP = m + 1;
    const int seg = blockIdx.x, bh = blockIdx.y, h = bh % H;
    const int r = threadIdx.x;
    const bool own = r < m;
    const float* om = omega + (size_t)h * m * d;
    const float kap = kshift[h];
    const size_t row0 = (size_t)bh * L;

    float hr[W];
    {
        const float* h0 = hstate + (CAUSAL ? ((size_t)bh * n_seg + seg) : (size_t)bh) * m * W + (size_t)r * W;
#pragma unroll
        for (int e = 0; e < W; ++e) hr[e] = own ? h0[e] : 0.f;
    }
    const int j0 = seg * seg_len, j1 = min(L, j0 + seg_len);
    if (j0 >= j1) return;
    const int last = j0 + ((j1 - j0 - 1) / TT) * TT;
    // asynchronous staging: raw k | v | q | dO rows and row statistics of the next tile
    uint8_t* rk = reinterpret_cast<uint8_t*>(sm + P.raw);
    uint8_t* rv = rk + raw_rows_bytes<T>(TT, d);
    uint8_t* rq = rv + raw_rows_bytes<T>(TT, DV);
    uint8_t* rdo = rq + raw_rows_bytes<T>(TT, d);
    uint8_t* rst = rdo + raw_rows_bytes<T>(TT, DV);
    auto prefetch = [&](int t) {
        const int n = min(TT, j1 - t);
        prefetch_rows(k + row0 * d, rk, t, n, TT, d);
        prefetch_rows(v + row0 * DV, rv, t, n, TT, DV);
        if (CAUSAL) {
            prefetch_rows(q + row0 * d, rq, t, n, TT, d);
            prefetch_rows(dout + row0 * DV, rdo, t, n, TT, DV);
            for (int j = threadIdx.x; j < TT; j += blockDim.x)
                cp_async16(rst + 16 * j, rowstat + row0 + t + (j < n ? j : 0), j < n ? 16 : 0);
        }
        cp_async_commit();
    };
    if (async_stage) prefetch(CAUSAL ? last : j0);
    for (int t0 = CAUSAL ? last : j0; CAUSAL ? t0 >= j0 : t0 < j1; t0 += CAUSAL ? -TT : TT) {
        const int nt = min(TT, j1 - t0);
        __syncthreads();
        if (async_stage) {
            cp_async_wait_all();
            __syncthreads();   // every thread's copies of this tile have landed
            unpack_rows<T>(rk, ys, TT, d, d, -1.f, nt);
            unpack_rows<T>(rv, cs, TT, DV, DVP, 1.f, nt);
            if (CAUSAL) {
                unpack_rows<T>(rq, xs, TT, d, d, -1.f, nt);
                unpack_rows<T>(rdo, dd, TT, DV, DVP, -1.f, nt);
                for (int j = threadIdx.x; j < TT; j += blockDim.x) {
                    const float4 rsj = reinterpret_cast<const float4*>(rst)[j];   // zeros past nt
                    den[j] = rsj.x;
                    cq[j] = rsj.y;
                    go[j] = rsj.z;
                }
            }
        } else {
            stage_rows(k + row0 * d, ys, t0, nt, TT, d, d, -1.f);
            stage_rows(v + row0 * DV, cs, t0, nt, TT, DV, DVP, 1.f);
            if (CAUSAL) {
                stage_rows(q + row0 * d, xs, t0, nt, TT, d, d, -1.f);
                stage_rows(dout + row0 * DV, dd, t0, nt, TT, DV, DVP, -1.f);
                for (int j = threadIdx.x; j < TT; j += blockDim.x) {
                    const float4 rsj = j < nt ? rowstat[row0 + t0 + j] : make_float4(0.f, 0.f, 0.f, 0.f);
                    den[j] = rsj.x;
                    cq[j] = rsj.y;
                    go[j] = rsj.z;
                }
            }
        }
        if (own && (CAUSAL || t0 == j0)) {
#pragma unroll
            for (int e = 0; e < DVP; ++e) rs[r * DVP + e] = e < DV ? hr[e < W ? e : 0] : 0.f;
        }
        __syncthreads();
        if (async_stage) {   // the next tile lands while this one computes
            const int nx = CAUSAL ? t0 - TT : t0 + TT;
            if (CAUSAL ? nx >= j0 : nx < j1) prefetch(nx);
        }
        key_norms(ys, kn, TT, d);
        if (own) {
            project_tile<TT>(om, ys, fk, r, m, d, s);
            if (CAUSAL) project_tile<TT>(om, xs, fq, r, m, d, s);
        }
        __syncthreads();
        if (own) {
#pragma unroll 4
            for (int j = 0; j < TT; ++j) {
                const float pk = fk[j * MP + r];
                float g = 0.f;
                if (j < nt)
                    g = KIND == FAVOR_KERNEL_SOFTMAX_POS ? expf(pk - 0.5f * s * s * kn[j] - kap) : fmaxf(pk, 0.f);
                fk[j * MP + r] = g;
                if (CAUSAL) {
                    const float pq = fq[j * MP + r];
                    float f = 0.f;
                    if (j < nt) f = KIND == FAVOR_KERNEL_SOFTMAX_POS ? expf(pq - cq[j]) : fmaxf(pq, 0.f);
                    fq[j * MP + r] = f;
                }
            }
        }
        if (CAUSAL) make_d(dd, den, go, TT, DV, DVP);
        __syncthreads();
        if (CAUSAL) {   // aa[j][i] = phi~_q(i) . phi~_k(j), mm[j][i] = D_i . C_j, for i >= j
            for (int idx = threadIdx.x; idx < TT * (TT + 1) / 2; idx += blockDim.x) {   // pairs i >= j only
                int i, j;
                tri_pair(idx, i, j);
                float a = 0.f, b = 0.f;
                {
                    for (int rr = 0; rr < m; ++rr) a = fmaf(fq[i * MP + rr], fk[j * MP + rr], a);
                    const float4* di = reinterpret_cast<const float4*>(dd + i * DVP);
                    const float4* cj = reinterpret_cast<const float4*>(cs + j * DVP);
#pragma unroll 4
                    for (int e4 = 0; e4 < DVP / 4; ++e4) b += dot4(di[e4], cj[e4]);
                }
                aa[j * (TT + 1) + i] = a;
                mm[j * (TT + 1) + i] = b;
            }
            __syncthreads();
        }
        // dv_j = H(tile end)^T phi~_k(j) + sum_{i>=j} aa[j][i] D_i, two keys x four columns per thread
        for (int idx = threadIdx.x; idx < (TT / 2) * (DV / 4); idx += blockDim.x) {
            const int jp = idx / (DV / 4), e4 = idx - jp * (DV / 4);
            const int ja = 2 * jp, jb = ja + 1;
            float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0;
#pragma unroll 4
            for (int rr = 0; rr < m; ++rr) {
                const float4 hv = *reinterpret_cast<const float4*>(rs + rr * DVP + 4 * e4);
                const float f0 = fk[ja * MP + rr], f1 = fk[jb * MP + rr];
                a0.x = fmaf(f0, hv.x, a0.x); a0.y = fmaf(f0, hv.y, a0.y);
                a0.z = fmaf(f0, hv.z, a0.z); a0.w = fmaf(f0, hv.w, a0.w);
                a1.x = fmaf(f1, hv.x, a1.x); a1.y = fmaf(f1, hv.y, a1.y);
                a1.z = fmaf(f1, hv.z, a1.z); a1.w = fmaf(f1, hv.w, a1.w);
            }
            if (CAUSAL)
                for (int i = ja; i < TT; ++i) {
                    const float4 dvec = *reinterpret_cast<const float4*>(dd + i * DVP + 4 * e4);
                    const float w0 = aa[ja * (TT + 1) + i], w1 = i >= jb ? aa[jb * (TT + 1) + i] : 0.f;
                    a0.x = fmaf(w0, dvec.x, a0.x); a0.y = fmaf(w0, dvec.y, a0.y);
                    a0.z = fmaf(w0, dvec.z, a0.z); a0.w = fmaf(w0, dvec.w, a0.w);
                    a1.x = fmaf(w1, dvec.x, a1.x); a1.y = fmaf(w1, dvec.y, a1.y);
                    a1.z = fmaf(w1, dvec.z, a1.z); a1.w = fmaf(w1, dvec.w, a1.w);
                }
            if (ja < nt) {
                T* o = dvv + (row0 + t0 + ja) * DV + 4 * e4;
                stf(o + 0, a0.x); stf(o + 1, a0.y); stf(o + 2, a0.z); stf(o + 3, a0.w);
            }
            if (jb < nt) {
                T* o = dvv + (row0 + t0 + jb) * DV + 4 * e4;
                stf(o + 0, a1.x); stf(o + 1, a1.y); stf(o + 2, a1.z); stf(o + 3, a1.w);
            }
        }
        __syncthreads();
        if (own) {
#pragma unroll 1
            for (int j = 0; j < TT; ++j) {
                const float g = fk[j * MP + r];
                const float4* cj = reinterpret_cast<const float4*>(cs + j * DVP);
                float p0 = 0.f, p1 = 0.f, p2 = 0.f, p3 = 0.f;   // independent partial sums
#pragma unroll
                for (int e4 = 0; e4 < DV / 4; ++e4) {
                    const float4 x = cj[e4];
                    p0 = fmaf(hr[4 * e4 + 0], x.x, p0);
                    p1 = fmaf(hr[4 * e4 + 1], x.y, p1);
                    p2 = fmaf(hr[4 * e4 + 2], x.z, p2);
                    p3 = fmaf(hr[4 * e4 + 3], x.w, p3);
                }
                p3 += j < nt ? hr[DV] : 0.f;
                if (CAUSAL) {
                    const float* mj = mm + j * (TT + 1);
                    int i = j;
                    for (; i + 1 < TT; i += 2) {
                        p0 = fmaf(fq[i * MP + r], mj[i], p0);
                        p1 = fmaf(fq[(i + 1) * MP + r], mj[i + 1], p1);
                    }
                    if (i < TT) p2 = fmaf(fq[i * MP + r], mj[i], p2);
                }
                const float dphi = (p0 + p1) + (p2 + p3);
                fk[j * MP + r] = KIND == FAVOR_KERNEL_SOFTMAX_POS ? dphi * g : (g > 0.f ? dphi : 0.f);
            }
            if (CAUSAL) {   // H at the previous tile's end
#pragma unroll 1
                for (int i = 0; i < TT; ++i) {
                    const float f = fq[i * MP + r];
                    const float4* di = reinterpret_cast<const float4*>(dd + i * DVP);
#pragma unroll
                    for (int e4 = 0; e4 < DV / 4; ++e4) {
                        const float4 x = di[e4];
                        hr[4 * e4 + 0] = fmaf(f, x.x, hr[4 * e4 + 0]);
                        hr[4 * e4 + 1] = fmaf(f, x.y, hr[4 * e4 + 1]);
                        hr[4 * e4 + 2] = fmaf(f, x.z, hr[4 * e4 + 2]);
                        hr[4 * e4 + 3] = fmaf(f, x.w, hr[4 * e4 + 3]);
                    }
                    hr[DV] = fmaf(f, dd[i * DVP + DV], hr[DV]);
                }
            }
        }
        __syncthreads();
        grad_inputs<T, KIND>(fk, ys, om, dk + row0 * d, t0, nt, TT, m, d, s);
    }
}

// ------------------------------------------------------- segment combines
// out[bh] = sum over segments (in order) of part[bh, seg].
__global__ void k_bwd_reduce(const float* __restrict__ part, float* __restrict__ out, int n_seg, int n) {
    const int bh = blockIdx.y;
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const float* p = part + (size_t)bh * n_seg * n + i;
    float a = 0.f;
    for (int sg = 0; sg < n_seg; ++sg) a += p[(size_t)sg * n];
    out[(size_t)bh * n + i] = a;
}

// part[bh, seg] <- sum of part[bh, seg+1 .. n_seg-1] (exclusive suffix, from the last segment back).
__global__ void k_bwd_rscan(float* __restrict__ part, int n_seg, int n) {
    const int bh = blockIdx.y;
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    float* p = part + (size_t)bh * n_seg * n + i;
    float run = 0.f;
    for (int sg = n_seg - 1; sg >= 0; --sg) {
        const float t = p[(size_t)sg * n];
        p[(size_t)sg * n] = run;
        run += t;
    }
}

template <typename K>
favor_status set_smem_bytes(K kern, size_t bytes) {
    if (bytes > 227 * 1024) return set_error(FAVOR_ERR_UNSUPPORTED, "backward: %zu bytes of shared memory", bytes);
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) != cudaSuccess) {
        cudaGetLastError();
        return set_error(FAVOR_ERR_CUDA, "backward: cannot set %zu bytes of shared memory", bytes);
    }
    return FAVOR_OK;
}

struct BwdCall {
    const void *q, *k, *v, *dout;
    void *dq, *dk, *dv;
};

// Shared-memory plan of one pass.  Tiles are staged asynchronously when every
// input is 16-byte aligned and the raw area still fits; otherwise synchronously.
template <typename T, int DV, bool CAUSAL>
BwdSmem pass_plan(const Handle& h, const BwdCall& c, bool key_pass, int* async_stage) {
    using S = BwdShape<DV>;
    const bool aligned = is_aligned16(c.q) && is_aligned16(c.k) && is_aligned16(c.v) && is_aligned16(c.dout);
    const int raw = bwd_raw_bytes<T>(S::TT, h.d, DV, CAUSAL, key_pass);
    BwdSmem P = bwd_smem(S::TT, S::DVP, S::W, h.m, h.d, CAUSAL, key_pass, raw);
    *async_stage = aligned && P.total * sizeof(float) <= 227 * 1024 ? 1 : 0;
    if (!*async_stage) P = bwd_smem(S::TT, S::DVP, S::W, h.m, h.d, CAUSAL, key_pass, 0);
    return P;
}

template <typename T, int KIND, int DV, bool CAUSAL>
favor_status bwd_passes(const Handle& h, const BwdCall& c, int BH, int L, const SegPlan& p, cudaStream_t st) {
    using S = BwdShape<DV>;
    const int threads = (h.m + 31) / 32 * 32;
    const int n = h.m * (DV + 1);
    const dim3 grid(p.n_seg, BH), cgrid((n + 255) / 256, BH);
    const int seg_len = p.seg_tiles * 128;
    float* qsum = CAUSAL ? h.ws_partial2 : h.ws_partial;     // per-segment sums of phi~_q D^T
    float4* rowstat = reinterpret_cast<float4*>(h.ws_rowstat);
    {
        int as = 0;
        const BwdSmem P = pass_plan<T, DV, CAUSAL>(h, c, false, &as);
        auto kern = k_bwd_query<T, KIND, DV, CAUSAL>;
        favor_status e = set_smem_bytes(kern, P.total * sizeof(float));
        if (e != FAVOR_OK) return e;
        ProfScope ps(h, PROF_BWD_QUERY, st);
        kern<<<grid, threads, P.total * sizeof(float), st>>>(
            (const T*)c.q, (const T*)c.k, (const T*)c.v, (const T*)c.dout, (T*)c.dq, h.omega_f32,
            h.kshift, CAUSAL ? h.ws_partial : h.ws_state, qsum, rowstat, h.H, L, h.m, h.d, h.s, seg_len, p.n_seg, as);
        count_launch();
        e = check_launch("backward query kernel");
        if (e != FAVOR_OK) return e;
    }
    {
        ProfScope ps(h, PROF_COMBINE, st);
        if (CAUSAL) k_bwd_rscan<<<cgrid, 256, 0, st>>>(qsum, p.n_seg, n);
        else k_bwd_reduce<<<cgrid, 256, 0, st>>>(qsum, h.ws_dstate, p.n_seg, n);
        count_launch();
        favor_status e = check_launch("backward combine kernel");
        if (e != FAVOR_OK) return e;
    }
    int as = 0;
    const BwdSmem P = pass_plan<T, DV, CAUSAL>(h, c, true, &as);
    auto kern = k_bwd_key<T, KIND, DV, CAUSAL>;
    favor_status e = set_smem_bytes(kern, P.total * sizeof(float));
    if (e != FAVOR_OK) return e;
    ProfScope ps(h, PROF_BWD_KEY, st);
    kern<<<grid, threads, P.total * sizeof(float), st>>>(
        (const T*)c.q, (const T*)c.k, (const T*)c.v, (const T*)c.dout, (T*)c.dk, (T*)c.dv,
        h.omega_f32, h.kshift, CAUSAL ? h.ws_partial2 : h.ws_dstate, rowstat, h.H, L, h.m, h.d, h.s, seg_len,
        p.n_seg, as);
    count_launch();
    return check_launch("backward key kernel");
}

template <bool CAUSAL>
favor_status bwd_dispatch(const Handle& h, const BwdCall& c, int BH, int L, const SegPlan& p, cudaStream_t st) {
#define FAVOR_BWD_DV(T, KIND)                                                  \
    switch (h.dv) {                                                            \
        case 16: return bwd_passes<T, KIND, 16, CAUSAL>(h, c, BH, L, p, st);   \
        case 32: return bwd_passes<T, KIND, 32, CAUSAL>(h, c, BH, L, p, st);   \
        case 64: return bwd_passes<T, KIND, 64, CAUSAL>(h, c, BH, L, p, st);   \
        case 128: return bwd_passes<T, KIND, 128, CAUSAL>(h, c, BH, L, p, st); \
    }
    if (h.dtype == FAVOR_DTYPE_F32) {
        if (h.kind == FAVOR_KERNEL_SOFTMAX_POS) { FAVOR_BWD_DV(float, FAVOR_KERNEL_SOFTMAX_POS) }
        else { FAVOR_BWD_DV(float, FAVOR_KERNEL_RELU) }
    } else {
        if (h.kind == FAVOR_KERNEL_SOFTMAX_POS) { FAVOR_BWD_DV(__nv_bfloat16, FAVOR_KERNEL_SOFTMAX_POS) }
        else { FAVOR_BWD_DV(__nv_bfloat16, FAVOR_KERNEL_RELU) }
    }
#undef FAVOR_BWD_DV
    return set_error(FAVOR_ERR_UNSUPPORTED, "backward: unsupported dv=%d", h.dv);
}

}  // namespace

favor_status simt_bidir_backward(const Handle& h, const void* q, const void* k, const void* v,
                                 const void* dout, void* dq, void* dk, void* dv, int B, int L, cudaStream_t st) {
    const int BH = B * h.H;
    const SegPlan p = plan_segments(BH, L, h.num_sms);
    favor_status s = simt_state_partials(h, k, v, BH, L, p, st);   // S~ | z~ per segment
    if (s != FAVOR_OK) return s;
    s = launch_reduce_segments(h, BH, p.n_seg, st);                // -> h.ws_state
    if (s != FAVOR_OK) return s;
    const BwdCall c{q, k, v, dout, dq, dk, dv};
    return bwd_dispatch<false>(h, c, BH, L, p, st);
}

favor_status simt_causal_backward(const Handle& h, const void* q, const void* k, const void* v,
                                  const void* dout, void* dq, void* dk, void* dv, int B, int L, cudaStream_t st) {
    const int BH = B * h.H;
    const SegPlan p = plan_segments(BH, L, h.num_sms);
    favor_status s = FAVOR_OK;
    if (p.n_seg > 1) {   // exclusive prefix states of the segments
        s = simt_state_partials(h, k, v, BH, L, p, st);
        if (s != FAVOR_OK) return s;
        s = launch_scan_segments(h, BH, p.n_seg, st);
    } else if (cudaMemsetAsync(h.ws_partial, 0, (size_t)BH * h.m * (h.dv + 1) * sizeof(float), st) != cudaSuccess) {
        cudaGetLastError();
        s = set_error(FAVOR_ERR_CUDA, "backward: cudaMemsetAsync failed");
    }
    if (s != FAVOR_OK) return s;
    const BwdCall c{q, k, v, dout, dq, dk, dv};
    return bwd_dispatch<true>(h, c, BH, L, p, st);
}

}  // namespace favor
