// Device helpers shared by the CUDA-core kernels (favor_simt.cu, favor_bwd.cu):
// element loads/stores of the storage type, warp reductions, feature values by
// kind, PermuteFormer's permutation cursor, per-token decay, and the tile
// staging / projection loops.
#pragma once

#include <cmath>

#include "favor_internal.h"

namespace favor {
namespace {

template <typename T> __device__ __forceinline__ float ldf(const T* p);
template <> __device__ __forceinline__ float ldf<float>(const float* p) { return *p; }
template <> __device__ __forceinline__ float ldf<__nv_bfloat16>(const __nv_bfloat16* p) { return __bfloat162float(*p); }

template <typename T> __device__ __forceinline__ void stf(T* p, float x);
template <> __device__ __forceinline__ void stf<float>(float* p, float x) { *p = x; }
template <> __device__ __forceinline__ void stf<__nv_bfloat16>(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

__device__ __forceinline__ float warp_sum(float a) {
    for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
    return a;
}
__device__ __forceinline__ float warp_max(float a) {
    for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    return a;
}
__device__ __forceinline__ float dot4(float4 a, float4 b) {
    return fmaf(a.x, b.x, fmaf(a.y, b.y, fmaf(a.z, b.z, a.w * b.w)));
}

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
    // Inverse direction: slot_j = pi^-j(r), the slot that holds feature r at position j.
    __device__ __forceinline__ void init_inv(const int* c, const int4* meta, int h, int m, int r, long long j) {
        cyc = c;
        base = 0; len = 1; idx = 0;
        if (c) {
            const int4 mt = meta[(size_t)h * m + r];
            base = h * m + mt.x;
            len = mt.y;
            long long t = ((long long)mt.z - j) % mt.y;
            idx = (int)(t < 0 ? t + mt.y : t);
        }
    }
    __device__ __forceinline__ int row(int r) const { return cyc ? cyc[base + idx] : r; }
    __device__ __forceinline__ void next() {
        if (cyc && ++idx == len) idx = 0;
    }
    __device__ __forceinline__ void prev() {
        if (cyc && --idx < 0) idx = len - 1;
    }
};

// Per-token decay of a causal state: S_j = a_j S_{j-1} + b_j phi(k_j) [v_j 1]^T
// with a_j = r_h g_j and b_j = 1 - g_j (RFA-Gate gates g, PermuteFormer r).
__device__ __forceinline__ void token_decay(const float* gate, size_t gidx, float rd, float* a, float* b) {
    const float g = gate ? gate[gidx] : 0.f;
    *a = rd * (gate ? g : 1.f);
    *b = gate ? 1.f - g : 1.f;
}

// Pair number idx of the lower triangle (diagonal included), row by row:
// (0,0), (1,0), (1,1), (2,0), ... -> (hi, lo) with lo <= hi.
__device__ __forceinline__ void tri_pair(int idx, int& hi, int& lo) {
    int a = (int)((sqrtf(8.f * (float)idx + 1.f) - 1.f) * 0.5f);
    while ((a + 1) * (a + 2) / 2 <= idx) ++a;   // float rounding guards
    while (a * (a + 1) / 2 > idx) --a;
    hi = a;
    lo = idx - a * (a + 1) / 2;
}

// Unscaled projections p[j] = omega_r . x_j, j < TT, of a staged token tile
// (float4 omega row against broadcast token rows).
template <int TT>
__device__ __forceinline__ void project_regs(const float* __restrict__ om, const float* xs, int r, int d, float* p) {
#pragma unroll
    for (int j = 0; j < TT; ++j) p[j] = 0.f;
    const float4* w4 = reinterpret_cast<const float4*>(om + (size_t)r * d);
    const float4* x4 = reinterpret_cast<const float4*>(xs);
    const int d4 = d >> 2;
#pragma unroll 1
    for (int c4 = 0; c4 < d4; ++c4) {
        const float4 w = __ldg(w4 + c4);
#pragma unroll
        for (int j = 0; j < TT; ++j) p[j] += dot4(w, x4[j * d4 + c4]);
    }
}

// Row max of raw query projections (row stride m+1), one warp per token; 0 for rows >= nt.
__device__ __forceinline__ void row_shift(const float* fq, float* cq, int TT, int nt, int m) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    for (int j = warp; j < TT; j += nw) {
        float mx = -INFINITY;
        for (int r = lane; r < m; r += 32) mx = fmaxf(mx, fq[j * (m + 1) + r]);
        mx = warp_max(mx);
        if (lane == 0) cq[j] = j < nt ? mx : 0.f;
    }
}

// Projections s*(omega_r . x_j) for j < TT into buf[j][r] (row stride m+1).
template <int TT>
__device__ __forceinline__ void project_tile(const float* __restrict__ om, const float* xs, float* buf, int r, int m,
                                             int d, float s) {
    float p[TT];
    project_regs<TT>(om, xs, r, d, p);
#pragma unroll
    for (int j = 0; j < TT; ++j) buf[j * (m + 1) + r] = s * p[j];
}

// Stage rows [t0, t0+nt) of a [BH, L, w] tensor into dst[TT][stride] as fp32;
// rows past nt and columns [w, stride) are zero, column w is `one_col` if >= 0.
template <typename T>
__device__ __forceinline__ void stage_rows(const T* __restrict__ src, float* dst, int t0, int nt, int TT, int w,
                                           int stride, float one_col) {
    for (int idx = threadIdx.x; idx < TT * stride; idx += blockDim.x) {
        const int j = idx / stride, c = idx - j * stride;
        float x = 0.f;
        if (j < nt) {
            if (c < w) x = ldf(src + (size_t)(t0 + j) * w + c);
            else if (c == w && one_col >= 0.f) x = one_col;
        }
        dst[idx] = x;
    }
}

// Asynchronous tile staging: the rows of the next tile are copied into a raw
// shared-memory area while the current tile computes, then unpacked to fp32.
// 16-byte copies; a copy with src_bytes = 0 reads nothing and writes zeros.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, int src_bytes) {
    const uint32_t a = (uint32_t)__cvta_generic_to_shared(dst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(a), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;\n" ::: "memory"); }

// Bytes of a raw tile of TT rows of w elements.
template <typename T>
__host__ __device__ __forceinline__ int raw_rows_bytes(int TT, int w) { return TT * w * (int)sizeof(T); }

// Start copying rows [t0, t0+nt) of a [BH, L, w] tensor (16-byte aligned base,
// w * sizeof(T) a multiple of 16) into raw[TT][w]; rows past nt become zeros.
template <typename T>
__device__ __forceinline__ void prefetch_rows(const T* __restrict__ src, uint8_t* raw, int t0, int nt, int TT, int w) {
    const int cpr = w * (int)sizeof(T) / 16;
    for (int idx = threadIdx.x; idx < TT * cpr; idx += blockDim.x) {
        const int j = idx / cpr, c = idx - j * cpr;
        const bool live = j < nt;
        const uint8_t* g = reinterpret_cast<const uint8_t*>(src + (size_t)(t0 + (live ? j : 0)) * w) + 16 * c;
        cp_async16(raw + (size_t)idx * 16, g, live ? 16 : 0);
    }
}

// raw[TT][w] -> dst[TT][stride] as fp32; columns [w, stride) are zero, column w
// is one_col (if >= 0) on rows below nt.  Equals stage_rows of the same rows.
template <typename T>
__device__ __forceinline__ void unpack_rows(const uint8_t* raw, float* dst, int TT, int w, int stride, float one_col,
                                            int nt) {
    const int s4 = stride >> 2;
    for (int idx = threadIdx.x; idx < TT * s4; idx += blockDim.x) {
        const int j = idx / s4, c = 4 * (idx - j * s4);
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (c < w) {
            const uint8_t* e = raw + ((size_t)j * w + c) * sizeof(T);
            if (sizeof(T) == 4) {
                x = *reinterpret_cast<const float4*>(e);
            } else {
                const uint2 b = *reinterpret_cast<const uint2*>(e);
                x = make_float4(__uint_as_float(b.x << 16), __uint_as_float(b.x & 0xffff0000u),
                                __uint_as_float(b.y << 16), __uint_as_float(b.y & 0xffff0000u));
            }
        } else if (c == w && one_col >= 0.f && j < nt) {
            x.x = one_col;
        }
        *reinterpret_cast<float4*>(dst + (size_t)j * stride + c) = x;
    }
}

// Squared key norms kn_j of a staged key tile, one warp per token.
__device__ __forceinline__ void key_norms(const float* ys, float* kn, int TT, int d) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    for (int j = warp; j < TT; j += nw) {
        float a = 0.f;
        for (int c = lane; c < d; c += 32) a = fmaf(ys[j * d + c], ys[j * d + c], a);
        a = warp_sum(a);
        if (lane == 0) kn[j] = a;
    }
}

}  // namespace
}  // namespace favor
