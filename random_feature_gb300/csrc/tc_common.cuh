// Shared pieces of the tensor-core kernels (favor_tc.cu: forward and stateful
// calls; favor_tc_bwd.cu: bidirectional backward): tile geometry for bf16,
// d = dv = 64, m = 256, the 128-byte swizzle, the projection MMA, the
// persistent (head, tile) ranges, and the host-side tensor maps.
#pragma once

#include <cstddef>
#include <cstdint>
#include <mutex>

#include <cudaTypedefs.h>

#include "favor_internal.h"
#include "tc_ptx.cuh"

namespace favor {
namespace {

using namespace tc;

constexpr int kTile = 128;         // tokens per tile / chunk
constexpr int kD = 64;             // head dim of q, k
constexpr int kDV = 64;            // head dim of v
constexpr int kM = 256;            // features
constexpr uint32_t kTileBytes = kTile * kD * 2;   // 16 KB
constexpr uint32_t kOmegaBytes = kM * kD * 2;     // 32 KB
constexpr uint32_t kPhiBlock = kTile * 128;       // one 64-column image of a 128-row tile
constexpr uint32_t kSBytes = kM * 128;            // S~ image [256 rows][64] = 32 KB
constexpr float kLog2e = 1.4426950408889634f;

// sin(x) (cosine = false) or cos(x) for the trigonometric features: x is first
// reduced to [-pi, pi] by Cody and Waite's method (x - n 2pi with 2pi split in
// two parts, the leading one 201/32, so that n times it is exact for |n| < 2^15),
// then the hardware approximation, accurate on that interval, is taken.
__device__ __forceinline__ float sincos_reduced(float x, bool cosine) {
    constexpr float kInvTwoPi = 0.15915494309189535f;
    constexpr float kTwoPiHi = 6.28125f;
    constexpr float kTwoPiLo = 1.9353071795864769e-3f;   // 2pi - kTwoPiHi
    const float n = rintf(x * kInvTwoPi);
    const float r = fmaf(-n, kTwoPiLo, fmaf(-n, kTwoPiHi, x));
    return cosine ? __cosf(r) : __sinf(r);
}

// sin(x) and cos(x) from one reduction (as sincos_reduced).
__device__ __forceinline__ void sincos_pair(float x, float& sn, float& cs) {
    constexpr float kInvTwoPi = 0.15915494309189535f;
    constexpr float kTwoPiHi = 6.28125f;
    constexpr float kTwoPiLo = 1.9353071795864769e-3f;
    const float n = rintf(x * kInvTwoPi);
    const float r = fmaf(-n, kTwoPiLo, fmaf(-n, kTwoPiHi, x));
    sn = __sinf(r);
    cs = __cosf(r);
}

// byte offset of chunk `c` (16 B) of row `r` inside an SW128 image
__device__ __forceinline__ uint32_t sw128(uint32_t r, uint32_t c) { return r * 128u + ((c ^ (r & 7u)) << 4); }

__device__ __forceinline__ uint8_t* align1k(uint8_t* p) {
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Squared norms of rows r0 and r1 of a bf16 SW128 tile: all sixteen 16-byte
// loads first, then sixteen independent accumulation chains of depth 8.
__device__ __forceinline__ void row_sqnorm2(uint32_t tile, uint32_t r0, uint32_t r1, float& n0, float& n1) {
    uint4 v[16];
#pragma unroll
    for (uint32_t c = 0; c < 8; ++c) {
        v[c] = ld_shared_v4(tile + sw128(r0, c));
        v[8 + c] = ld_shared_v4(tile + sw128(r1, c));
    }
    float acc[16];
#pragma unroll
    for (int c = 0; c < 16; ++c) {
        const uint32_t w[4] = {v[c].x, v[c].y, v[c].z, v[c].w};
        float t = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float lo = bf16lo(w[i]), hi = bf16hi(w[i]);
            t = fmaf(lo, lo, t);
            t = fmaf(hi, hi, t);
        }
        acc[c] = t;
    }
    n0 = ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
    n1 = ((acc[8] + acc[9]) + (acc[10] + acc[11])) + ((acc[12] + acc[13]) + (acc[14] + acc[15]));
}

// Squared norm of row `r` of a bf16 SW128 tile (loads first, eight chains).
__device__ __forceinline__ float row_sqnorm(uint32_t tile, uint32_t r) {
    uint4 v[8];
#pragma unroll
    for (uint32_t c = 0; c < 8; ++c) v[c] = ld_shared_v4(tile + sw128(r, c));
    float acc[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const uint32_t w[4] = {v[c].x, v[c].y, v[c].z, v[c].w};
        float t = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float lo = bf16lo(w[i]), hi = bf16hi(w[i]);
            t = fmaf(lo, lo, t);
            t = fmaf(hi, hi, t);
        }
        acc[c] = t;
    }
    return ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
}

// Issue `n` projection MMAs (K = 64 in 4 steps) of a 128-row tile against
// `nrows` rows of omega starting at omega_row: D[tmem_d] = X * omega^T.
__device__ __forceinline__ void issue_projection(uint32_t tmem_d, uint32_t x_tile, uint32_t omega, int N) {
    const uint32_t idesc = make_idesc(128, N, 0, 0);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
        const uint64_t a = make_desc(x_tile + kk * 32, 16, 1024, SW_128B);
        const uint64_t b = make_desc(omega + kk * 32, 16, 1024, SW_128B);
        mma_ss(tmem_d, a, b, idesc, kk > 0);
    }
}

// ======================================================== persistent ranges
// The flattened (head, tile) space of a call is cut into G contiguous ranges
// of `per` tiles, one per CTA.  A head's tiles are covered by CTAs
// first_cta(bh) .. last_cta(bh); CTA c writes the state of its part of head bh
// to piece c - first_cta(bh) of that head (pstride pieces per head).
struct Ranges {
    int tph;      // tiles per head
    int T;        // total tiles
    int per;      // tiles per CTA
    int G;        // CTAs
    int pstride;  // piece slots per head
};

__host__ __device__ __forceinline__ int first_cta(const Ranges& r, int bh) { return (bh * r.tph) / r.per; }
__host__ __device__ __forceinline__ int last_cta(const Ranges& r, int bh) { return ((bh + 1) * r.tph - 1) / r.per; }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        cudaGetLastError();
    });
    return fn;
}

// [BH, L, 64] bf16, box [1, 128, 64], 128-byte swizzle; rows past L read as zeros.
bool map_tokens(CUtensorMap* m, const void* base, int BH, int L) {
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)L, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)kD * 2 * (cuuint64_t)L};
    cuuint32_t box[3] = {(cuuint32_t)kD, (cuuint32_t)kTile, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// omega [H*256, 64] bf16, box [256, 64], 128-byte swizzle.
bool map_omega(CUtensorMap* m, const void* base, int H) {
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)H * kM};
    cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
    cuuint32_t box[2] = {(cuuint32_t)kD, (cuuint32_t)kM};
    cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename K>
void allow_smem(K kern, size_t bytes) {
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

Ranges plan_ranges(int BH, int L, int num_sms) {
    Ranges r;
    r.tph = (L + kTile - 1) / kTile;
    r.T = BH * r.tph;
    int G = num_sms < r.T ? num_sms : r.T;
    r.per = (r.T + G - 1) / G;
    r.G = (r.T + r.per - 1) / r.per;
    int mx = 1;
    for (int bh = 0; bh < BH; ++bh) {
        const int np = last_cta(r, bh) - first_cta(r, bh) + 1;
        if (np > mx) mx = np;
    }
    r.pstride = mx;
    return r;
}

}  // namespace
}  // namespace favor
