// Tensor-core FAVOR+ path for sm_103a: bf16 storage, d = dv = 64, m = 256.
//
// Every contraction runs on tcgen05.mma (bf16 operands, fp32 accumulators in
// tensor memory); tiles arrive by TMA with 128-byte swizzle; the exp / ReLU
// feature epilogues run on the CUDA cores between contractions, so Phi_Q and
// Phi_K never reach HBM.
//
// Shared-memory tiles are "SW128" images: rows of 64 bf16 (128 B), 8-row
// groups of 1 KB, and the 16-byte chunk c of row r stored at chunk c ^ (r & 7).
// A [rows x 256] feature tile is four such images of 64 columns, 16 KB apart.
//
// Tensor-memory use (512 columns, lane = tile row):
//   state kernel : [0,256) projection | [256,384) S halves (2 x 64) | [384,416) z halves (2 x 16)
//   readout      : [0,256) projection, then Phi_Q as packed bf16 in [0,128) | [128,208) output num|den
//   causal       : [0,128) Phi_Q bf16 (from a 256-column projection) | [128,256) key projection
//                  half, then Phi_Q Phi_K^T, then its masked bf16 copy | [256,336) output |
//                  [336,368) z halves | [384,512) S halves
#include <cmath>
#include <cstring>
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
constexpr uint32_t kZBytes = kM * 32;             // z~ image [256 rows][16] = 8 KB
constexpr uint32_t kImageBytes = kSBytes + kZBytes;
constexpr float kLog2e = 1.4426950408889634f;

// byte offset of chunk `c` (16 B) of row `r` inside an SW128 image
__device__ __forceinline__ uint32_t sw128(uint32_t r, uint32_t c) { return r * 128u + ((c ^ (r & 7u)) << 4); }

struct Bars {
    uint64_t tma;
    uint64_t mma;
    uint32_t tmem_base;
    uint32_t pad;
};

__device__ __forceinline__ uint8_t* align1k(uint8_t* p) {
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Squared norm of row `r` of a bf16 SW128 tile.
__device__ __forceinline__ float row_sqnorm(uint32_t tile, uint32_t r) {
    float a = 0.f;
#pragma unroll
    for (uint32_t c = 0; c < 8; ++c) {
        uint4 v = ld_shared_v4(tile + sw128(r, c));
        uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float lo = bf16lo(w[i]), hi = bf16hi(w[i]);
            a = fmaf(lo, lo, a);
            a = fmaf(hi, hi, a);
        }
    }
    return a;
}

// Common prologue: barriers, tensor memory, optional all-ones operand.
__device__ __forceinline__ void setup(Bars* bars, uint32_t ncols) {
    if (threadIdx.x == 0) {
        mbar_init(&bars->tma, 1);
        mbar_init(&bars->mma, 1);
        fence_mbar_init();
    }
    if (threadIdx.x / 32 == 0) {
        tmem_alloc(&bars->tmem_base, ncols);
        tmem_relinquish();
    }
}

__device__ __forceinline__ void teardown(Bars* bars, uint32_t tmem, uint32_t ncols) {
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x / 32 == 0) tmem_dealloc(tmem, ncols);
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

// Key features of one row for 32 consecutive projection columns -> 16 packed bf16 words.
template <int KIND>
__device__ __forceinline__ void key_features32(const uint32_t (&p)[32], float a, float c, bool live,
                                               uint32_t (&w)[16]) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        float f0, f1;
        if (KIND == FAVOR_KERNEL_SOFTMAX_POS) {
            f0 = ex2(fmaf(__uint_as_float(p[2 * i]), a, c));
            f1 = ex2(fmaf(__uint_as_float(p[2 * i + 1]), a, c));
        } else {
            f0 = fmaxf(__uint_as_float(p[2 * i]), 0.f);
            f1 = fmaxf(__uint_as_float(p[2 * i + 1]), 0.f);
        }
        w[i] = live ? pack_bf16(f0, f1) : 0u;
    }
}

// Write 16 packed words (32 features starting at feature f0) into row r of a
// [128 x 256] feature tile made of four SW128 images.
__device__ __forceinline__ void store_feat32(uint32_t phi, uint32_t r, int f0, const uint32_t (&w)[16]) {
    const uint32_t blk = phi + (uint32_t)(f0 / 64) * kPhiBlock;
    const uint32_t c0 = (uint32_t)(f0 % 64) / 8;
#pragma unroll
    for (int q = 0; q < 4; ++q)
        st_shared_v4(blk + sw128(r, c0 + q), w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
}

// Query features of one row into packed bf16 in tensor memory, in place:
// columns [col0, col0+256) hold the fp32 projection; afterwards
// [col0, col0+128) hold the 256 features as bf16 pairs.
template <int KIND>
__device__ __forceinline__ void query_features_to_tmem(uint32_t tl, float a) {
    float mx = 0.f;
    if (KIND == FAVOR_KERNEL_SOFTMAX_POS) {
        mx = -INFINITY;
        for (int c = 0; c < 8; ++c) {
            uint32_t p[32];
            tmem_ld32(tl + 32 * c, p);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) mx = fmaxf(mx, __uint_as_float(p[i]));
        }
    }
    const float cm = -mx * a;
    for (int c = 0; c < 8; ++c) {
        uint32_t p[32];
        tmem_ld32(tl + 32 * c, p);
        tmem_ld_wait();
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            float f0, f1;
            if (KIND == FAVOR_KERNEL_SOFTMAX_POS) {
                f0 = ex2(fmaf(__uint_as_float(p[2 * i]), a, cm));
                f1 = ex2(fmaf(__uint_as_float(p[2 * i + 1]), a, cm));
            } else {
                f0 = fmaxf(__uint_as_float(p[2 * i]), 0.f);
                f1 = fmaxf(__uint_as_float(p[2 * i + 1]), 0.f);
            }
            w[i] = pack_bf16(f0, f1);
        }
        tmem_st16(tl + 16 * c, w);
    }
    tmem_st_wait();
}

// out row = num / den from tensor-memory columns [col, col+64) and col+64.
__device__ __forceinline__ void store_output_row(uint32_t tl, __nv_bfloat16* dst, bool live) {
    uint32_t n0[32], n1[32], z[16];
    tmem_ld32(tl, n0);
    tmem_ld32(tl + 32, n1);
    tmem_ld16(tl + 64, z);
    tmem_ld_wait();
    if (!live) return;
    const float den = __uint_as_float(z[0]);
    const float inv = den != 0.f ? 1.f / den : 0.f;
    uint4* o = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint4 v;
        v.x = pack_bf16(__uint_as_float(n0[8 * q + 0]) * inv, __uint_as_float(n0[8 * q + 1]) * inv);
        v.y = pack_bf16(__uint_as_float(n0[8 * q + 2]) * inv, __uint_as_float(n0[8 * q + 3]) * inv);
        v.z = pack_bf16(__uint_as_float(n0[8 * q + 4]) * inv, __uint_as_float(n0[8 * q + 5]) * inv);
        v.w = pack_bf16(__uint_as_float(n0[8 * q + 6]) * inv, __uint_as_float(n0[8 * q + 7]) * inv);
        o[q] = v;
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint4 v;
        v.x = pack_bf16(__uint_as_float(n1[8 * q + 0]) * inv, __uint_as_float(n1[8 * q + 1]) * inv);
        v.y = pack_bf16(__uint_as_float(n1[8 * q + 2]) * inv, __uint_as_float(n1[8 * q + 3]) * inv);
        v.z = pack_bf16(__uint_as_float(n1[8 * q + 4]) * inv, __uint_as_float(n1[8 * q + 5]) * inv);
        v.w = pack_bf16(__uint_as_float(n1[8 * q + 6]) * inv, __uint_as_float(n1[8 * q + 7]) * inv);
        o[4 + q] = v;
    }
}

// Row r of the S~ / z~ operand images from 64 fp32 S values and z.
__device__ __forceinline__ void store_state_row(uint32_t simg, uint32_t zimg, uint32_t r, const float* sv,
                                                float z) {
#pragma unroll
    for (uint32_t c = 0; c < 8; ++c)
        st_shared_v4(simg + sw128(r, c), pack_bf16(sv[8 * c], sv[8 * c + 1]), pack_bf16(sv[8 * c + 2], sv[8 * c + 3]),
                     pack_bf16(sv[8 * c + 4], sv[8 * c + 5]), pack_bf16(sv[8 * c + 6], sv[8 * c + 7]));
    const uint32_t zz = pack_bf16(z, z);
    st_shared_v4(zimg + r * 32, zz, zz, zz, zz);
    st_shared_v4(zimg + r * 32 + 16, zz, zz, zz, zz);
}

// ====================================================================== state
// grid (n_seg, B*H), 128 threads.  Partial S (as [r][0:64]) and z ([r][64]) of
// one segment's keys, fp32, to part[(bh*n_seg + seg)][256][65].
template <int KIND>
__global__ void __launch_bounds__(128, 1)
k_tc_state(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
           const __grid_constant__ CUtensorMap tm_w, const float* __restrict__ kshift, float* __restrict__ part,
           int H, int L, float s, int seg_tiles, int n_seg, int* err) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1k(smem_raw);
    const uint32_t s_w = smem_u32(sm);
    const uint32_t s_k = s_w + kOmegaBytes;
    const uint32_t s_v = s_k + kTileBytes;
    const uint32_t s_phi = s_v + kTileBytes;
    const uint32_t s_one = s_phi + 4 * kPhiBlock;
    Bars* bars = reinterpret_cast<Bars*>(sm + (s_one - s_w) + 1024);
    const int seg = blockIdx.x, bh = blockIdx.y, h = bh % H;
    const int tid = threadIdx.x, warp = tid / 32;
    const uint32_t row = tid;   // tile row = tensor-memory lane

    setup(bars, 512);
    for (int i = tid; i < 256; i += 128)
        reinterpret_cast<uint32_t*>(sm + (s_one - s_w))[i] = 0x3F803F80u;   // bf16 1.0 pairs
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    const uint32_t tl = tmem + ((uint32_t)(warp * 32) << 16);

    uint32_t tma_ph = 0, mma_ph = 0;
    bool ok = true;
    if (tid == 0) {
        mbar_expect_tx(&bars->tma, kOmegaBytes);
        tma_load_2d(sm, &tm_w, &bars->tma, 0, h * kM);
    }
    ok = __syncthreads_and(mbar_wait(&bars->tma, tma_ph, err, 1));
    tma_ph ^= 1;

    const float a = s * kLog2e;
    const float kap = kshift[h];
    int done = 0;
    for (int t = 0; t < seg_tiles && ok; ++t) {
        const int tok0 = (seg * seg_tiles + t) * kTile;
        if (tok0 >= L) break;
        if (tid == 0) {
            mbar_expect_tx(&bars->tma, 2 * kTileBytes);
            tma_load_3d(sm + (s_k - s_w), &tm_k, &bars->tma, 0, tok0, bh);
            tma_load_3d(sm + (s_v - s_w), &tm_v, &bars->tma, 0, tok0, bh);
        }
        ok = __syncthreads_and(mbar_wait(&bars->tma, tma_ph, err, 2));
        tma_ph ^= 1;
        if (!ok) break;
        const float c = -(0.5f * s * s * row_sqnorm(s_k, row) + kap) * kLog2e;
        const bool live = tok0 + (int)row < L;
        if (tid == 0) {
            tc_fence_after();
            issue_projection(tmem, s_k, s_w, 256);
            mma_commit(&bars->mma);
        }
        ok = __syncthreads_and(mbar_wait(&bars->mma, mma_ph, err, 3));
        mma_ph ^= 1;
        tc_fence_after();
        if (!ok) break;
        for (int cc = 0; cc < 8; ++cc) {
            uint32_t p[32], w[16];
            tmem_ld32(tl + 32 * cc, p);
            tmem_ld_wait();
            key_features32<KIND>(p, a, c, live, w);
            store_feat32(s_phi, row, 32 * cc, w);
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            const uint32_t id_s = make_idesc(128, 64, 1, 1);
            const uint32_t id_z = make_idesc(128, 16, 1, 0);
            const uint64_t b1 = make_desc(s_one, 128, 256, SW_NONE);
            for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint64_t av = make_desc(s_phi + 2 * hh * kPhiBlock + kk * 2048, kPhiBlock, 1024, SW_128B);
                    const uint64_t bv = make_desc(s_v + kk * 2048, kPhiBlock, 1024, SW_128B);
                    const uint32_t acc = (t > 0 || kk > 0) ? 1u : 0u;
                    mma_ss(tmem + 256 + 64 * hh, av, bv, id_s, acc);
                    mma_ss(tmem + 384 + 16 * hh, av, b1, id_z, acc);
                }
            }
            mma_commit(&bars->mma);
        }
        ok = __syncthreads_and(mbar_wait(&bars->mma, mma_ph, err, 4));
        mma_ph ^= 1;
        tc_fence_after();
        ++done;
    }
    if (ok && done > 0) {
        for (int hh = 0; hh < 2; ++hh) {
            uint32_t s0[32], s1[32], z[16];
            tmem_ld32(tl + 256 + 64 * hh, s0);
            tmem_ld32(tl + 256 + 64 * hh + 32, s1);
            tmem_ld16(tl + 384 + 16 * hh, z);
            tmem_ld_wait();
            float* o = part + ((size_t)bh * n_seg + seg) * (kM * (kDV + 1)) + (size_t)(128 * hh + row) * (kDV + 1);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __uint_as_float(s0[e]);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[32 + e] = __uint_as_float(s1[e]);
            o[64] = __uint_as_float(z[0]);
        }
    }
    teardown(bars, tmem, 512);
}

// ================================================ reduce + pack (bidirectional)
// grid (ceil(256*65/256), B*H).  Sum the segment partials in order and write
// the bf16 operand image: S~ ([256][64] SW128) then z~ ([256][16], z repeated).
__global__ void k_reduce_pack(const float* __restrict__ part, uint8_t* __restrict__ image, int n_seg) {
    const int bh = blockIdx.y;
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    constexpr int n = kM * (kDV + 1);
    if (i >= n) return;
    const float* p = part + (size_t)bh * n_seg * n + i;
    float acc = 0.f;
    for (int sg = 0; sg < n_seg; ++sg) acc += p[(size_t)sg * n];
    const int r = i / (kDV + 1), e = i - r * (kDV + 1);
    uint8_t* img = image + (size_t)bh * kImageBytes;
    const __nv_bfloat16 b = __float2bfloat16_rn(acc);
    if (e < kDV) {
        const uint32_t off = (uint32_t)r * 128u + ((((uint32_t)e >> 3) ^ ((uint32_t)r & 7u)) << 4) + ((uint32_t)e & 7u) * 2u;
        *reinterpret_cast<__nv_bfloat16*>(img + off) = b;
    } else {
        __nv_bfloat16* z = reinterpret_cast<__nv_bfloat16*>(img + kSBytes + (size_t)r * 32);
#pragma unroll
        for (int q = 0; q < 16; ++q) z[q] = b;
    }
}

// ==================================================================== readout
// grid (tiles, B*H), 128 threads: one 128-query tile per CTA.
template <int KIND>
__global__ void __launch_bounds__(128, 1)
k_tc_readout(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_w,
             const uint8_t* __restrict__ image, __nv_bfloat16* __restrict__ out, int H, int L, float s, int* err) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1k(smem_raw);
    const uint32_t s_w = smem_u32(sm);
    const uint32_t s_q = s_w + kOmegaBytes;
    const uint32_t s_s = s_q + kTileBytes;
    const uint32_t s_z = s_s + kSBytes;
    Bars* bars = reinterpret_cast<Bars*>(sm + (s_z - s_w) + kZBytes);
    const int tile = blockIdx.x, bh = blockIdx.y, h = bh % H;
    const int tid = threadIdx.x, warp = tid / 32;
    const uint32_t row = tid;
    const int tok0 = tile * kTile;

    setup(bars, 256);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    const uint32_t tl = tmem + ((uint32_t)(warp * 32) << 16);

    if (tid == 0) {
        mbar_expect_tx(&bars->tma, kOmegaBytes + kTileBytes + kImageBytes);
        tma_load_2d(sm, &tm_w, &bars->tma, 0, h * kM);
        tma_load_3d(sm + (s_q - s_w), &tm_q, &bars->tma, 0, tok0, bh);
        bulk_load(sm + (s_s - s_w), image + (size_t)bh * kImageBytes, kImageBytes, &bars->tma);
    }
    bool ok = __syncthreads_and(mbar_wait(&bars->tma, 0, err, 11));
    if (ok && tid == 0) {
        tc_fence_after();
        issue_projection(tmem, s_q, s_w, 256);
        mma_commit(&bars->mma);
    }
    ok = __syncthreads_and(ok && mbar_wait(&bars->mma, 0, err, 12));
    tc_fence_after();
    if (ok) query_features_to_tmem<KIND>(tl, s * kLog2e);
    tc_fence_before();
    __syncthreads();
    if (ok && tid == 0) {
        tc_fence_after();
        const uint32_t id_s = make_idesc(128, 64, 0, 1);
        const uint32_t id_z = make_idesc(128, 16, 0, 1);
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
            const uint64_t bs = make_desc(s_s + kk * 2048, 8192, 1024, SW_128B);
            const uint64_t bz = make_desc(s_z + kk * 512, 8192, 256, SW_32B);
            mma_ts(tmem + 128, tmem + 8 * kk, bs, id_s, kk > 0);
            mma_ts(tmem + 192, tmem + 8 * kk, bz, id_z, kk > 0);
        }
        mma_commit(&bars->mma);
    }
    ok = __syncthreads_and(ok && mbar_wait(&bars->mma, 1, err, 13));
    tc_fence_after();
    if (ok) {
        const int tok = tok0 + (int)row;
        store_output_row(tl + 128, out + ((size_t)bh * L + tok) * kDV, tok < L);
    }
    teardown(bars, tmem, 256);
}

// ===================================================================== causal
// grid (n_seg, B*H), 128 threads.  Walks one segment chunk by chunk starting
// from the segment's exclusive prefix state prefix[(bh*n_seg + seg)][256][65].
template <int KIND>
__global__ void __launch_bounds__(128, 1)
k_tc_causal(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
            const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_w,
            const float* __restrict__ kshift, const float* __restrict__ prefix, __nv_bfloat16* __restrict__ out,
            int H, int L, float s, int seg_tiles, int n_seg, int* err) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1k(smem_raw);
    const uint32_t s_w = smem_u32(sm);
    const uint32_t s_q = s_w + kOmegaBytes;
    const uint32_t s_k = s_q + kTileBytes;
    const uint32_t s_v = s_k + kTileBytes;
    const uint32_t s_phi = s_v + kTileBytes;
    const uint32_t s_s = s_phi + 4 * kPhiBlock;
    const uint32_t s_z = s_s + kSBytes;
    const uint32_t s_one = s_z + kZBytes;
    Bars* bars = reinterpret_cast<Bars*>(sm + (s_one - s_w) + 1024);
    const int seg = blockIdx.x, bh = blockIdx.y, h = bh % H;
    const int tid = threadIdx.x, warp = tid / 32;
    const uint32_t row = tid;

    setup(bars, 512);
    for (int i = tid; i < 256; i += 128)
        reinterpret_cast<uint32_t*>(sm + (s_one - s_w))[i] = 0x3F803F80u;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    const uint32_t tl = tmem + ((uint32_t)(warp * 32) << 16);

    uint32_t tma_ph = 0, mma_ph = 0;
    if (tid == 0) {
        mbar_expect_tx(&bars->tma, kOmegaBytes);
        tma_load_2d(sm, &tm_w, &bars->tma, 0, h * kM);
    }
    // Initial state from the exclusive prefix: tensor memory (fp32 master) and
    // the bf16 operand images.
    const float* pre = prefix + ((size_t)bh * n_seg + seg) * (kM * (kDV + 1));
    for (int hh = 0; hh < 2; ++hh) {
        const uint32_t r = 128 * hh + row;
        float sv[64];
#pragma unroll
        for (int e = 0; e < 64; ++e) sv[e] = pre[(size_t)r * (kDV + 1) + e];
        const float z = pre[(size_t)r * (kDV + 1) + 64];
        uint32_t w[16];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
#pragma unroll
            for (int i = 0; i < 16; ++i) w[i] = __float_as_uint(sv[16 * q + i]);
            tmem_st16(tl + 384 + 64 * hh + 16 * q, w);
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) w[i] = __float_as_uint(z);
        tmem_st16(tl + 336 + 16 * hh, w);
        store_state_row(s_s, s_z, r, sv, z);
    }
    tmem_st_wait();
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    bool ok = __syncthreads_and(mbar_wait(&bars->tma, tma_ph, err, 21));
    tma_ph ^= 1;

    const float a = s * kLog2e;
    const float kap = kshift[h];
    for (int t = 0; t < seg_tiles && ok; ++t) {
        const int tok0 = (seg * seg_tiles + t) * kTile;
        if (tok0 >= L) break;
        if (tid == 0) {
            mbar_expect_tx(&bars->tma, 3 * kTileBytes);
            tma_load_3d(sm + (s_q - s_w), &tm_q, &bars->tma, 0, tok0, bh);
            tma_load_3d(sm + (s_k - s_w), &tm_k, &bars->tma, 0, tok0, bh);
            tma_load_3d(sm + (s_v - s_w), &tm_v, &bars->tma, 0, tok0, bh);
        }
        ok = __syncthreads_and(mbar_wait(&bars->tma, tma_ph, err, 22));
        tma_ph ^= 1;
        if (!ok) break;
        const float c = -(0.5f * s * s * row_sqnorm(s_k, row) + kap) * kLog2e;
        const bool live = tok0 + (int)row < L;
        // query projection and features (bf16 pairs into [0,128))
        if (tid == 0) {
            tc_fence_after();
            issue_projection(tmem, s_q, s_w, 256);
            mma_commit(&bars->mma);
        }
        ok = __syncthreads_and(mbar_wait(&bars->mma, mma_ph, err, 23));
        mma_ph ^= 1;
        tc_fence_after();
        if (!ok) break;
        query_features_to_tmem<KIND>(tl, a);
        tc_fence_before();
        __syncthreads();
        // key projection in two halves of 128 features -> Phi_K in shared memory
        for (int hk = 0; hk < 2 && ok; ++hk) {
            if (tid == 0) {
                tc_fence_after();
                issue_projection(tmem + 128, s_k, s_w + hk * 128 * 128, 128);
                mma_commit(&bars->mma);
            }
            ok = __syncthreads_and(mbar_wait(&bars->mma, mma_ph, err, 24));
            mma_ph ^= 1;
            tc_fence_after();
            if (!ok) break;
            for (int cc = 0; cc < 4; ++cc) {
                uint32_t p[32], w[16];
                tmem_ld32(tl + 128 + 32 * cc, p);
                tmem_ld_wait();
                key_features32<KIND>(p, a, c, live, w);
                store_feat32(s_phi, row, 128 * hk + 32 * cc, w);
            }
            fence_async_smem();
            tc_fence_before();
            __syncthreads();
        }
        if (!ok) break;
        // A = Phi_Q Phi_K^T (N = 128 keys) and the inter-chunk term Phi_Q [S~ | z~]
        if (tid == 0) {
            tc_fence_after();
            const uint32_t id_a = make_idesc(128, 128, 0, 0);
            const uint32_t id_s = make_idesc(128, 64, 0, 1);
            const uint32_t id_z = make_idesc(128, 16, 0, 1);
#pragma unroll
            for (int kk = 0; kk < 16; ++kk) {
                const uint64_t bk = make_desc(s_phi + (kk / 4) * kPhiBlock + (kk % 4) * 32, 16, 1024, SW_128B);
                mma_ts(tmem + 128, tmem + 8 * kk, bk, id_a, kk > 0);
                const uint64_t bs = make_desc(s_s + kk * 2048, 8192, 1024, SW_128B);
                const uint64_t bz = make_desc(s_z + kk * 512, 8192, 256, SW_32B);
                mma_ts(tmem + 256, tmem + 8 * kk, bs, id_s, kk > 0);
                mma_ts(tmem + 320, tmem + 8 * kk, bz, id_z, kk > 0);
            }
            mma_commit(&bars->mma);
        }
        ok = __syncthreads_and(mbar_wait(&bars->mma, mma_ph, err, 25));
        mma_ph ^= 1;
        tc_fence_after();
        if (!ok) break;
        // causal mask (keep key j <= query i) and bf16 pairs in place into [128,192)
        for (int cc = 0; cc < 4; ++cc) {
            uint32_t p[32], w[16];
            tmem_ld32(tl + 128 + 32 * cc, p);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int j0 = 32 * cc + 2 * i;
                const float f0 = (j0 <= (int)row) ? __uint_as_float(p[2 * i]) : 0.f;
                const float f1 = (j0 + 1 <= (int)row) ? __uint_as_float(p[2 * i + 1]) : 0.f;
                w[i] = pack_bf16(f0, f1);
            }
            tmem_st16(tl + 128 + 16 * cc, w);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncthreads();
        // intra-chunk term tril(A) [V | 1] and the state update [S | z] += Phi_K^T [V | 1]
        if (tid == 0) {
            tc_fence_after();
            const uint32_t id_v = make_idesc(128, 64, 0, 1);
            const uint32_t id_1 = make_idesc(128, 16, 0, 0);
            const uint32_t id_sv = make_idesc(128, 64, 1, 1);
            const uint32_t id_s1 = make_idesc(128, 16, 1, 0);
            const uint64_t b1 = make_desc(s_one, 128, 256, SW_NONE);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint64_t bv = make_desc(s_v + kk * 2048, 8192, 1024, SW_128B);
                mma_ts(tmem + 256, tmem + 128 + 8 * kk, bv, id_v, 1);
                mma_ts(tmem + 320, tmem + 128 + 8 * kk, b1, id_1, 1);
            }
            for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint64_t av = make_desc(s_phi + 2 * hh * kPhiBlock + kk * 2048, kPhiBlock, 1024, SW_128B);
                    const uint64_t bv = make_desc(s_v + kk * 2048, 8192, 1024, SW_128B);
                    mma_ss(tmem + 384 + 64 * hh, av, bv, id_sv, 1);
                    mma_ss(tmem + 336 + 16 * hh, av, b1, id_s1, 1);
                }
            }
            mma_commit(&bars->mma);
        }
        ok = __syncthreads_and(mbar_wait(&bars->mma, mma_ph, err, 26));
        mma_ph ^= 1;
        tc_fence_after();
        if (!ok) break;
        {
            const int tok = tok0 + (int)row;
            store_output_row(tl + 256, out + ((size_t)bh * L + tok) * kDV, tok < L);
        }
        // refresh the bf16 state images for the next chunk
        for (int hh = 0; hh < 2; ++hh) {
            uint32_t s0[32], s1[32], z[16];
            tmem_ld32(tl + 384 + 64 * hh, s0);
            tmem_ld32(tl + 384 + 64 * hh + 32, s1);
            tmem_ld16(tl + 336 + 16 * hh, z);
            tmem_ld_wait();
            float sv[64];
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                sv[e] = __uint_as_float(s0[e]);
                sv[32 + e] = __uint_as_float(s1[e]);
            }
            store_state_row(s_s, s_z, 128 * hh + row, sv, __uint_as_float(z[0]));
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }
    teardown(bars, tmem, 512);
}

// ================================================================ feature map
// grid (tiles, B*H), 128 threads.  phi = the plain definition, bf16.
template <int KIND>
__global__ void __launch_bounds__(128, 1)
k_tc_feature_map(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                 __nv_bfloat16* __restrict__ phi, int H, int L, float s, int* err) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1k(smem_raw);
    const uint32_t s_w = smem_u32(sm);
    const uint32_t s_x = s_w + kOmegaBytes;
    Bars* bars = reinterpret_cast<Bars*>(sm + kOmegaBytes + kTileBytes);
    const int tile = blockIdx.x, bh = blockIdx.y, h = bh % H;
    const int tid = threadIdx.x, warp = tid / 32;
    const uint32_t row = tid;
    const int tok0 = tile * kTile;

    setup(bars, 256);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    const uint32_t tl = tmem + ((uint32_t)(warp * 32) << 16);
    if (tid == 0) {
        mbar_expect_tx(&bars->tma, kOmegaBytes + kTileBytes);
        tma_load_2d(sm, &tm_w, &bars->tma, 0, h * kM);
        tma_load_3d(sm + kOmegaBytes, &tm_x, &bars->tma, 0, tok0, bh);
    }
    bool ok = __syncthreads_and(mbar_wait(&bars->tma, 0, err, 31));
    if (ok && tid == 0) {
        tc_fence_after();
        issue_projection(tmem, s_x, s_w, 256);
        mma_commit(&bars->mma);
    }
    ok = __syncthreads_and(ok && mbar_wait(&bars->mma, 0, err, 32));
    tc_fence_after();
    const int tok = tok0 + (int)row;
    if (ok) {
        const float a = s * kLog2e;
        const float c = -(0.5f * s * s * row_sqnorm(s_x, row)) * kLog2e - 4.0f;   // m^-1/2 = 2^-4 for m = 256
        uint4* dst = reinterpret_cast<uint4*>(phi + ((size_t)bh * L + tok) * kM);
        for (int cc = 0; cc < 8; ++cc) {
            uint32_t p[32], w[16];
            tmem_ld32(tl + 32 * cc, p);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                float f0, f1;
                if (KIND == FAVOR_KERNEL_SOFTMAX_POS) {
                    f0 = ex2(fmaf(__uint_as_float(p[2 * i]), a, c));
                    f1 = ex2(fmaf(__uint_as_float(p[2 * i + 1]), a, c));
                } else {
                    f0 = fmaxf(__uint_as_float(p[2 * i]) * s, 0.f) * 0.0625f;
                    f1 = fmaxf(__uint_as_float(p[2 * i + 1]) * s, 0.f) * 0.0625f;
                }
                w[i] = pack_bf16(f0, f1);
            }
            if (tok < L) {
#pragma unroll
                for (int q = 0; q < 4; ++q) dst[4 * cc + q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
            }
        }
    }
    teardown(bars, tmem, 256);
}

// ================================================================ host side
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

constexpr size_t kSmemState = 1024 + kOmegaBytes + 2 * kTileBytes + 4 * kPhiBlock + 1024 + 64;
constexpr size_t kSmemReadout = 1024 + kOmegaBytes + kTileBytes + kImageBytes + 64;
constexpr size_t kSmemCausal = 1024 + kOmegaBytes + 3 * kTileBytes + 4 * kPhiBlock + kImageBytes + 1024 + 64;
constexpr size_t kSmemFmap = 1024 + kOmegaBytes + kTileBytes + 64;

template <typename K>
void allow_smem(K kern, size_t bytes) {
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

void allow_all_once() {
    static std::once_flag once;
    std::call_once(once, [] {
        allow_smem(k_tc_state<FAVOR_KERNEL_SOFTMAX_POS>, kSmemState);
        allow_smem(k_tc_state<FAVOR_KERNEL_RELU>, kSmemState);
        allow_smem(k_tc_readout<FAVOR_KERNEL_SOFTMAX_POS>, kSmemReadout);
        allow_smem(k_tc_readout<FAVOR_KERNEL_RELU>, kSmemReadout);
        allow_smem(k_tc_causal<FAVOR_KERNEL_SOFTMAX_POS>, kSmemCausal);
        allow_smem(k_tc_causal<FAVOR_KERNEL_RELU>, kSmemCausal);
        allow_smem(k_tc_feature_map<FAVOR_KERNEL_SOFTMAX_POS>, kSmemFmap);
        allow_smem(k_tc_feature_map<FAVOR_KERNEL_RELU>, kSmemFmap);
        cudaGetLastError();
    });
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

favor_status launch_state(const Handle& h, const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mw,
                          int BH, int L, const SegPlan& p, cudaStream_t st) {
    dim3 grid(p.n_seg, BH);
    ProfScope ps(h, PROF_STATE, st);
    if (h.kind == FAVOR_KERNEL_SOFTMAX_POS)
        k_tc_state<FAVOR_KERNEL_SOFTMAX_POS><<<grid, 128, kSmemState, st>>>(mk, mv, mw, h.kshift, h.ws_partial, h.H, L,
                                                                              h.s, p.seg_tiles, p.n_seg, h.dev_err);
    else
        k_tc_state<FAVOR_KERNEL_RELU><<<grid, 128, kSmemState, st>>>(mk, mv, mw, h.kshift, h.ws_partial, h.H, L, h.s,
                                                                       p.seg_tiles, p.n_seg, h.dev_err);
    count_launch();
    return check_launch("tensor-core state kernel");
}

}  // namespace

bool tc_supported(const Handle& h) {
    return h.dtype == FAVOR_DTYPE_BF16 && h.d == kD && h.dv == kDV && h.m == kM && h.cc_major >= 10 &&
           encode_fn() != nullptr;
}

favor_status tc_feature_map(const Handle& h, const void* x, void* phi, int B, int L, cudaStream_t st) {
    if (!aligned16(x) || !aligned16(phi)) return simt_feature_map(h, x, phi, B, L, st);
    allow_all_once();
    const int BH = B * h.H;
    CUtensorMap mx, mw;
    if (!map_tokens(&mx, x, BH, L) || !map_omega(&mw, h.omega_bf16, h.H))
        return set_error(FAVOR_ERR_CUDA, "cuTensorMapEncodeTiled failed");
    dim3 grid((L + kTile - 1) / kTile, BH);
    ProfScope ps(h, PROF_FEATURE_MAP, st);
    if (h.kind == FAVOR_KERNEL_SOFTMAX_POS)
        k_tc_feature_map<FAVOR_KERNEL_SOFTMAX_POS><<<grid, 128, kSmemFmap, st>>>(mx, mw, (__nv_bfloat16*)phi, h.H, L,
                                                                                   h.s, h.dev_err);
    else
        k_tc_feature_map<FAVOR_KERNEL_RELU><<<grid, 128, kSmemFmap, st>>>(mx, mw, (__nv_bfloat16*)phi, h.H, L, h.s,
                                                                            h.dev_err);
    count_launch();
    return check_launch("tensor-core feature map kernel");
}

favor_status tc_bidir(const Handle& h, const void* q, const void* k, const void* v, void* out, int B, int L,
                      cudaStream_t st) {
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
        return simt_bidir(h, q, k, v, out, B, L, st);
    allow_all_once();
    const int BH = B * h.H;
    SegPlan p = plan_segments(BH, L, h.num_sms);
    CUtensorMap mq, mk, mv, mw;
    if (!map_tokens(&mq, q, BH, L) || !map_tokens(&mk, k, BH, L) || !map_tokens(&mv, v, BH, L) ||
        !map_omega(&mw, h.omega_bf16, h.H))
        return set_error(FAVOR_ERR_CUDA, "cuTensorMapEncodeTiled failed");
    favor_status s = launch_state(h, mk, mv, mw, BH, L, p, st);
    if (s != FAVOR_OK) return s;
    {
        dim3 grid((kM * (kDV + 1) + 255) / 256, BH);
        ProfScope ps(h, PROF_COMBINE, st);
        k_reduce_pack<<<grid, 256, 0, st>>>(h.ws_partial, (uint8_t*)h.ws_tc, p.n_seg);
        count_launch();
        s = check_launch("reduce/pack kernel");
        if (s != FAVOR_OK) return s;
    }
    dim3 grid(p.tiles, BH);
    ProfScope ps(h, PROF_READOUT, st);
    if (h.kind == FAVOR_KERNEL_SOFTMAX_POS)
        k_tc_readout<FAVOR_KERNEL_SOFTMAX_POS><<<grid, 128, kSmemReadout, st>>>(
            mq, mw, (const uint8_t*)h.ws_tc, (__nv_bfloat16*)out, h.H, L, h.s, h.dev_err);
    else
        k_tc_readout<FAVOR_KERNEL_RELU><<<grid, 128, kSmemReadout, st>>>(mq, mw, (const uint8_t*)h.ws_tc,
                                                                           (__nv_bfloat16*)out, h.H, L, h.s, h.dev_err);
    count_launch();
    return check_launch("tensor-core readout kernel");
}

favor_status tc_causal(const Handle& h, const void* q, const void* k, const void* v, void* out, int B, int L,
                       cudaStream_t st) {
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
        return simt_causal(h, q, k, v, out, B, L, st);
    allow_all_once();
    const int BH = B * h.H;
    SegPlan p = plan_segments(BH, L, h.num_sms);
    CUtensorMap mq, mk, mv, mw;
    if (!map_tokens(&mq, q, BH, L) || !map_tokens(&mk, k, BH, L) || !map_tokens(&mv, v, BH, L) ||
        !map_omega(&mw, h.omega_bf16, h.H))
        return set_error(FAVOR_ERR_CUDA, "cuTensorMapEncodeTiled failed");
    favor_status s;
    if (p.n_seg > 1) {
        s = launch_state(h, mk, mv, mw, BH, L, p, st);
        if (s != FAVOR_OK) return s;
        s = launch_scan_segments(h, BH, p.n_seg, st);
    } else {
        s = cudaMemsetAsync(h.ws_partial, 0, (size_t)BH * kM * (kDV + 1) * sizeof(float), st) == cudaSuccess
                ? FAVOR_OK
                : set_error(FAVOR_ERR_CUDA, "cudaMemsetAsync failed");
    }
    if (s != FAVOR_OK) return s;
    dim3 grid(p.n_seg, BH);
    ProfScope ps(h, PROF_CAUSAL, st);
    if (h.kind == FAVOR_KERNEL_SOFTMAX_POS)
        k_tc_causal<FAVOR_KERNEL_SOFTMAX_POS><<<grid, 128, kSmemCausal, st>>>(
            mq, mk, mv, mw, h.kshift, h.ws_partial, (__nv_bfloat16*)out, h.H, L, h.s, p.seg_tiles, p.n_seg, h.dev_err);
    else
        k_tc_causal<FAVOR_KERNEL_RELU><<<grid, 128, kSmemCausal, st>>>(mq, mk, mv, mw, h.kshift, h.ws_partial,
                                                                         (__nv_bfloat16*)out, h.H, L, h.s, p.seg_tiles,
                                                                         p.n_seg, h.dev_err);
    count_launch();
    return check_launch("tensor-core causal kernel");
}

}  // namespace favor
