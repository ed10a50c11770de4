// Tensor-core bidirectional backward for sm_103a: bf16, d = dv = 64, m = 256.
// The formulas are those of favor_bwd.cu (the derivative of App. B Alg. 1 of
// Rethinking Attention with Performers); here every contraction runs on
// tcgen05.mma with operands staged by TMA, as in favor_tc.cu.
#include <cmath>
#include <cstddef>
#include <cstring>
#include <mutex>

#include "favor_internal.h"
#include "tc_common.cuh"
#include "tc_ptx.cuh"

namespace favor {
namespace {

using namespace tc;

// ============================================================ backward (bidirectional)
// The gradients of Alg. 1 (see favor_bwd.cu for the formulas) on the tensor
// cores.  Two steps subtract nearly equal terms (u - z (dO . out) on the query
// side, dS~ [v 1] on the key side), so their operands enter the contractions as
// bf16 pairs hi + lo (hi = bf16(x), lo = bf16(x - hi)): S~, dS~, the features
// that build them, G and D.  Column sums (z, dz) accumulate in fp32 registers.
//
//   k_tc_bstate<MODE 0>  K, V            -> pieces of [S~ | z~]   (features from fp32, hi + lo)
//   k_tc_bstate<MODE 1>  Q, dO, rowstat  -> pieces of [dS~ | dz~] (D = [dO/den, -go/den], hi + lo)
//   k_bwd_reduce_pack    pieces          -> per head: S hi, S lo images (SW128 [256][64]) + z fp32
//   k_tc_bwd_q           Q, dO, image    -> dq, rowstat (den~, row shift, dO . out)
//   k_tc_bwd_k           K, V, image     -> dk, dv
constexpr uint32_t kBImg = 2 * kSBytes + kM * 4;   // S hi | S lo | z (fp32)
constexpr int kBStateThreads = 256;

struct BwBars {
    uint64_t head;      // per-head operands (omega, images)
    uint64_t tile[2];   // double-buffered token tiles
    uint64_t mma;
    uint32_t tmem_base;
    uint32_t pad;
};

// Persistent loop bookkeeping of the backward kernels: the flattened (head,
// tile) range of this CTA; token tiles are double-buffered (tile g+1 loads
// while tile g computes), per-head operands reload only when the head changes.
__device__ __forceinline__ void bw_init_bars(BwBars* bars) {
    if (threadIdx.x == 0) {
        mbar_init(&bars->head, 1);
        mbar_init(&bars->tile[0], 1);
        mbar_init(&bars->tile[1], 1);
        mbar_init(&bars->mma, 1);
        fence_mbar_init();
    }
    if (threadIdx.x / 32 == 0) {
        tmem_alloc(&bars->tmem_base, 512);
        tmem_relinquish();
    }
}

// Loads issued and not yet waited for, tracked by the issuing thread so that a
// kernel whose bounded wait gave up still waits (bounded) for its own copies
// before it exits: parity of the pending phase per barrier, -1 when none.
struct BwPending {
    int head = -1, tile[2] = {-1, -1};
    __device__ __forceinline__ void drain(BwBars* bars, int* err, int code) {
        if (head >= 0) mbar_wait(&bars->head, (uint32_t)head, err, code);
        for (int b = 0; b < 2; ++b)
            if (tile[b] >= 0) mbar_wait(&bars->tile[b], (uint32_t)tile[b], err, code);
    }
};

// Two token tiles (x, y) of flattened tile g into buffer `dst` (x at dst, y at dst + 16 KB).
__device__ __forceinline__ void bw_load_tiles(const CUtensorMap* mx, const CUtensorMap* my, uint8_t* dst,
                                              uint64_t* bar, int g, int tph) {
    const int bh = g / tph, tile = g - bh * tph;
    mbar_expect_tx(bar, 2 * kTileBytes);
    tma_load_3d(dst, mx, bar, 0, tile * kTile, bh);
    tma_load_3d(dst + kTileBytes, my, bar, 0, tile * kTile, bh);
}

// Split x into bf16 hi + lo and pack pairs: (x0, x1) -> hi word, lo word.
__device__ __forceinline__ void split_pack(float x0, float x1, uint32_t& hi, uint32_t& lo) {
    hi = pack_bf16(x0, x1);
    lo = pack_bf16(x0 - bf16lo(hi), x1 - bf16hi(hi));
}

// Transposed projection + features + state contraction.  grid R.G, 256 threads;
// warp w owns features 128*(w/4) + 32*(w%4) + lane (tensor-memory lane = feature).
// Tensor memory: half h: P^T_h [128h, 128h+128) (fp32, column = token), then the
// packed features hi [128h, 128h+64) and lo [128h+64, 128h+128); accumulators
// [256 + 64h, 256 + 64h + 64).
template <int KIND, int MODE>
__global__ void __launch_bounds__(kBStateThreads, 1)
k_tc_bstate(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_y,
            const __grid_constant__ CUtensorMap tm_w, const float* __restrict__ kshift,
            const float4* __restrict__ rowstat, float* __restrict__ part, int H, int L, float s, Ranges R, int* err) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1k(smem_raw);
    const uint32_t s_w = smem_u32(sm);
    uint8_t* buf = sm + kOmegaBytes;                              // 2 x [x tile | y tile]
    const uint32_t s_dlo = s_w + kOmegaBytes + 4 * kTileBytes;
    float* s_c = reinterpret_cast<float*>(sm + kOmegaBytes + 5 * kTileBytes);   // [128] exponent offsets
    float* s_wz = s_c + kTile;                                                  // [128] z-column weights
    BwBars* bars = reinterpret_cast<BwBars*>(s_wz + kTile);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int half = warp >> 2, quad = warp & 3;
    const int cta = blockIdx.x;
    const int g0 = cta * R.per, g1 = min(R.T, g0 + R.per);

    bw_init_bars(bars);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    const uint32_t t_lane = (uint32_t)(32 * quad) << 16;
    const uint32_t t_ph = tmem + t_lane + 128 * half;           // this warp's P^T / feature columns
    const uint32_t t_acc = tmem + t_lane + 256 + 64 * half;     // this warp's accumulator columns
    const int r_feat = 128 * half + 32 * quad + lane;
    const float a = s * kLog2e;
    BwPending pend;
    if (tid == 0 && g0 < g1) {
        mbar_expect_tx(&bars->head, kOmegaBytes);
        tma_load_2d(sm, &tm_w, &bars->head, 0, ((g0 / R.tph) % H) * kM);
        pend.head = 0;
        bw_load_tiles(&tm_x, &tm_y, buf, &bars->tile[0], g0, R.tph);
        pend.tile[0] = 0;
    }

    bool ok = true;
    float zacc = 0.f;
    bool first = true;
    int loaded_h = -1;
    uint32_t nhead = 0;
    for (int g = g0, it = 0; g < g1; ++g, ++it) {
        const int b = it & 1;
        const int bh = g / R.tph, tile = g - bh * R.tph, h = bh % H;
        const int tok0 = tile * kTile;
        const uint32_t s_x = s_w + kOmegaBytes + b * 2 * kTileBytes, s_y = s_x + kTileBytes;
        __syncthreads();   // the previous tile is done with its buffers and tensor memory
        const bool new_head = h != loaded_h;
        if (tid == 0) {
            if (new_head && it > 0) {
                mbar_expect_tx(&bars->head, kOmegaBytes);
                tma_load_2d(sm, &tm_w, &bars->head, 0, h * kM);
                pend.head = (int)(nhead & 1);
            }
            if (g + 1 < g1) {
                bw_load_tiles(&tm_x, &tm_y, buf + (b ^ 1) * 2 * kTileBytes, &bars->tile[b ^ 1], g + 1, R.tph);
                pend.tile[b ^ 1] = ((it + 1) >> 1) & 1;
            }
        }
        if (new_head) {
            ok = __syncthreads_and(mbar_wait(&bars->head, nhead & 1, err, 40));
            ++nhead;
            loaded_h = h;
            if (!ok) break;
            pend.head = -1;
        }
        ok = __syncthreads_and(mbar_wait(&bars->tile[b], (it >> 1) & 1, err, 41));
        if (!ok) break;
        pend.tile[b] = -1;
        if (tid < kTile) {
            const int t = tid, tok = tok0 + t;
            const bool live = tok < L;
            float c = -INFINITY, wz = 0.f;
            if (MODE == 0) {
                if (live) {
                    c = -(0.5f * s * s * row_sqnorm(s_x, t) + kshift[h]) * kLog2e;
                    wz = 1.f;
                }
            } else {
                float inv = 0.f;
                if (live) {
                    const float4 rs = rowstat[(size_t)bh * L + tok];
                    c = -rs.y * kLog2e;
                    inv = rs.x != 0.f ? 1.f / rs.x : 0.f;
                    wz = -rs.z * inv;
                }
                // D row t = dO_t / den_t as hi (in place) + lo
#pragma unroll
                for (uint32_t ch = 0; ch < 8; ++ch) {
                    const uint32_t off = sw128(t, ch);
                    const uint4 x = ld_shared_v4(s_y + off);
                    const uint32_t xin[4] = {x.x, x.y, x.z, x.w};
                    uint32_t hi[4], lo[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) split_pack(bf16lo(xin[i]) * inv, bf16hi(xin[i]) * inv, hi[i], lo[i]);
                    st_shared_v4(s_y + off, hi[0], hi[1], hi[2], hi[3]);
                    st_shared_v4(s_dlo + off, lo[0], lo[1], lo[2], lo[3]);
                }
                fence_async_smem();
            }
            s_c[t] = c;
            s_wz[t] = wz;
        }
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            const uint32_t id_p = make_idesc(128, 128, 0, 0);
#pragma unroll
            for (int hp = 0; hp < 2; ++hp) {
                const uint64_t a0 = make_desc(s_w + hp * 128 * 128, 16, 1024, SW_128B);
                const uint64_t b0 = make_desc(s_x, 16, 1024, SW_128B);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) mma_ss(tmem + 128 * hp, a0 + 2 * kk, b0 + 2 * kk, id_p, kk > 0 ? 1u : 0u);
            }
            mma_commit(&bars->mma);
        }
        ok = __syncthreads_and(mbar_wait(&bars->mma, 0, err, 42));
        if (!ok) break;
        tc_fence_after();
        {
            float f[128];
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                uint32_t pw[32];
                tmem_ld32(t_ph + 32 * cc, pw);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int t = 32 * cc + i;
                    const float pv = __uint_as_float(pw[i]);
                    float x;
                    if (KIND == FAVOR_KERNEL_SOFTMAX_POS) x = ex2(fmaf(pv, a, s_c[t]));   // 0 for dead tokens (c = -inf)
                    else x = s_wz[t] != 0.f || MODE == 1 ? fmaxf(s * pv, 0.f) : 0.f;
                    f[t] = x;
                    zacc = fmaf(x, s_wz[t], zacc);
                }
            }
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                uint32_t hw[16], lw[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) split_pack(f[32 * cc + 2 * i], f[32 * cc + 2 * i + 1], hw[i], lw[i]);
                tmem_st16(t_ph + 16 * cc, hw);
                tmem_st16(t_ph + 64 + 16 * cc, lw);
            }
            tmem_st_wait();
        }
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            const uint32_t id_s = make_idesc(128, 64, 0, 1);
            const uint64_t by = make_desc(s_y, 8192, 1024, SW_128B);
            const uint64_t bl = make_desc(s_dlo, 8192, 1024, SW_128B);
#pragma unroll
            for (int hp = 0; hp < 2; ++hp) {
                const uint32_t d = tmem + 256 + 64 * hp;
                const uint32_t ahi = tmem + 128 * hp, alo = tmem + 128 * hp + 64;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) mma_ts(d, ahi + 8 * kk, by + 128 * kk, id_s, (first && kk == 0) ? 0u : 1u);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) mma_ts(d, alo + 8 * kk, by + 128 * kk, id_s, 1u);
                if (MODE == 1) {
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) mma_ts(d, ahi + 8 * kk, bl + 128 * kk, id_s, 1u);
                }
            }
            mma_commit(&bars->mma);
        }
        ok = __syncthreads_and(mbar_wait(&bars->mma, 1, err, 43));
        if (!ok) break;
        tc_fence_after();
        first = false;
        const bool piece_end = (g + 1 == g1) || ((g + 1) / R.tph != bh);
        if (piece_end) {
            uint32_t v0[32], v1[32];
            tmem_ld32(t_acc, v0);
            tmem_ld32(t_acc + 32, v1);
            tmem_ld_wait();
            const int piece = cta - first_cta(R, bh);
            float* o = part + ((size_t)bh * R.pstride + piece) * (kM * (kDV + 1)) + (size_t)r_feat * (kDV + 1);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                o[i] = __uint_as_float(v0[i]);
                o[32 + i] = __uint_as_float(v1[i]);
            }
            o[kDV] = zacc;
            zacc = 0.f;
            first = true;
            tc_fence_before();   // the next piece's first MMA overwrites the accumulator after the loop-top barrier
        }
    }
    if (!ok && tid == 0) pend.drain(bars, err, 40);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

// Fixed-order sum of a head's pieces (row-major [m][dv+1]) -> hi / lo SW128
// images of the value columns and the z column in fp32.  grid (m*(dv+1)/256 up, B*H).
__global__ void k_bwd_reduce_pack(const float* __restrict__ part, uint8_t* __restrict__ img, Ranges R) {
    const int bh = blockIdx.y;
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= kM * (kDV + 1)) return;
    const int np = last_cta(R, bh) - first_cta(R, bh) + 1;
    const float* p = part + (size_t)bh * R.pstride * (kM * (kDV + 1)) + i;
    float acc = 0.f;
    for (int k = 0; k < np; ++k) acc += p[(size_t)k * (kM * (kDV + 1))];
    const int r = i / (kDV + 1), c = i - r * (kDV + 1);
    uint8_t* base = img + (size_t)bh * kBImg;
    if (c == kDV) {
        reinterpret_cast<float*>(base + 2 * kSBytes)[r] = acc;
    } else {
        const __nv_bfloat16 hi = __float2bfloat16_rn(acc);
        const __nv_bfloat16 lo = __float2bfloat16_rn(acc - __bfloat162float(hi));
        const uint32_t off = sw128((uint32_t)r, (uint32_t)c >> 3) + 2 * (c & 7);
        *reinterpret_cast<__nv_bfloat16*>(base + off) = hi;
        *reinterpret_cast<__nv_bfloat16*>(base + kSBytes + off) = lo;
    }
}

constexpr int kBwdThreads = 256;   // two threads per row: features [0,128) and [128,256)

// Per-head operands of the backward passes: omega (TMA) and the state image (bulk copy).
__device__ __forceinline__ void bw_load_head(const CUtensorMap* mw, const uint8_t* img, uint8_t* sm, BwBars* bars,
                                             int bh, int h) {
    mbar_expect_tx(&bars->head, kOmegaBytes + kBImg);
    tma_load_2d(sm, mw, &bars->head, 0, h * kM);
    bulk_load(sm + kOmegaBytes, img + (size_t)bh * kBImg, kBImg, &bars->head);
}

// Query pass, persistent over the call's tile ranges (grid R.G, 256 threads: thread t
// takes query row t % 128 and features 128*(t/128) .. +127 of it).  Tensor memory per
// tile: P [0,256), U = dO (S hi + S lo)^T [256,512); each thread then writes the packed
// G of its features as lo over its P columns (from 128 ch) and hi over its U columns
// (from 256 + 128 ch), 64 columns each, at or behind the columns it has read; the dq
// accumulator takes the freed [64,128).
template <int KIND>
__global__ void __launch_bounds__(kBwdThreads, 1)
k_tc_bwd_q(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
           const __grid_constant__ CUtensorMap tm_w, const uint8_t* __restrict__ img, __nv_bfloat16* __restrict__ dq,
           float4* __restrict__ rowstat, int H, int L, float s, Ranges R, int* err) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1k(smem_raw);
    const uint32_t s_w = smem_u32(sm);
    const uint32_t s_img = s_w + kOmegaBytes;
    uint8_t* buf = sm + kOmegaBytes + kBImg;                      // 2 x [q tile | dO tile]
    const float* z = reinterpret_cast<const float*>(sm + kOmegaBytes + 2 * kSBytes);
    float* red = reinterpret_cast<float*>(sm + kOmegaBytes + kBImg + 4 * kTileBytes);   // [3][2][128] row partials
    BwBars* bars = reinterpret_cast<BwBars*>(red + 3 * 2 * kTile);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int row = tid & (kTile - 1), ch = tid >> 7;
    const int g0 = blockIdx.x * R.per, g1 = min(R.T, g0 + R.per);

    bw_init_bars(bars);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    const uint32_t tl = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    const uint32_t tp = tl + 128 * ch, tu = tl + 256 + 128 * ch;   // this thread's P and U columns
    const float a = s * kLog2e;
    BwPending pend;
    if (tid == 0 && g0 < g1) {
        bw_load_head(&tm_w, img, sm, bars, g0 / R.tph, (g0 / R.tph) % H);
        pend.head = 0;
        bw_load_tiles(&tm_q, &tm_do, buf, &bars->tile[0], g0, R.tph);
        pend.tile[0] = 0;
    }
    bool ok = true;
    int loaded_bh = -1;
    uint32_t nhead = 0;
    for (int g = g0, it = 0; g < g1; ++g, ++it) {
        const int b = it & 1;
        const int bh = g / R.tph, tile = g - bh * R.tph, h = bh % H;
        const int tok = tile * kTile + row;
        const bool live = tok < L;
        const uint32_t s_q = s_img + kBImg + b * 2 * kTileBytes, s_do = s_q + kTileBytes;
        __syncthreads();   // the previous tile is done with its buffers and tensor memory
        const bool new_head = bh != loaded_bh;
        if (tid == 0) {
            if (new_head && it > 0) {
                bw_load_head(&tm_w, img, sm, bars, bh, h);
                pend.head = (int)(nhead & 1);
            }
            if (g + 1 < g1) {
                bw_load_tiles(&tm_q, &tm_do, buf + (b ^ 1) * 2 * kTileBytes, &bars->tile[b ^ 1], g + 1, R.tph);
                pend.tile[b ^ 1] = ((it + 1) >> 1) & 1;
            }
        }
        if (new_head) {
            ok = __syncthreads_and(mbar_wait(&bars->head, nhead & 1, err, 44));
            ++nhead;
            loaded_bh = bh;
            if (!ok) break;
            pend.head = -1;
        }
        ok = __syncthreads_and(mbar_wait(&bars->tile[b], (it >> 1) & 1, err, 50));
        if (!ok) break;
        pend.tile[b] = -1;
        if (tid == 0) {
            tc_fence_after();
            issue_projection(tmem, s_q, s_w, 256);
            const uint32_t id_u = make_idesc(128, 256, 0, 0);
            const uint64_t a0 = make_desc(s_do, 16, 1024, SW_128B);
            const uint64_t bh0 = make_desc(s_img, 16, 1024, SW_128B);
            const uint64_t bl0 = make_desc(s_img + kSBytes, 16, 1024, SW_128B);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) mma_ss(tmem + 256, a0 + 2 * kk, bh0 + 2 * kk, id_u, kk > 0 ? 1u : 0u);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) mma_ss(tmem + 256, a0 + 2 * kk, bl0 + 2 * kk, id_u, 1u);
            mma_commit(&bars->mma);
        }
        ok = __syncthreads_and(mbar_wait(&bars->mma, 0, err, 45));
        if (!ok) break;
        tc_fence_after();
        float gsum = 0.f;
        {
            float mx = 0.f;
            if (KIND == FAVOR_KERNEL_SOFTMAX_POS) {
                mx = -INFINITY;
                for (int cc = 0; cc < 4; ++cc) {
                    uint32_t pw[32];
                    tmem_ld32(tp + 32 * cc, pw);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i) mx = fmaxf(mx, __uint_as_float(pw[i]));
                }
                red[ch * kTile + row] = mx;
                __syncthreads();
                mx = fmaxf(red[row], red[kTile + row]);
            }
            const float c = -mx * a;
            float den = 0.f, fu = 0.f;
            for (int cc = 0; cc < 4; ++cc) {
                uint32_t pw[32], uw[32];
                tmem_ld32(tp + 32 * cc, pw);
                tmem_ld32(tu + 32 * cc, uw);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const float pv = __uint_as_float(pw[i]);
                    const float f = KIND == FAVOR_KERNEL_SOFTMAX_POS ? ex2(fmaf(pv, a, c)) : fmaxf(s * pv, 0.f);
                    den = fmaf(f, z[128 * ch + 32 * cc + i], den);
                    fu = fmaf(f, __uint_as_float(uw[i]), fu);
                }
            }
            red[2 * kTile + ch * kTile + row] = den;
            red[4 * kTile + ch * kTile + row] = fu;
            __syncthreads();
            den = red[2 * kTile + row] + red[3 * kTile + row];
            fu = red[4 * kTile + row] + red[5 * kTile + row];
            const float inv = den != 0.f ? 1.f / den : 0.f;
            const float go = fu * inv;
            for (int cc = 0; cc < 4; ++cc) {
                uint32_t pw[32], uw[32];
                tmem_ld32(tp + 32 * cc, pw);
                tmem_ld32(tu + 32 * cc, uw);
                tmem_ld_wait();
                uint32_t hw[16], lw[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    float gg[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int k = 2 * i + e;
                        const float pv = __uint_as_float(pw[k]);
                        const float dphi = (__uint_as_float(uw[k]) - z[128 * ch + 32 * cc + k] * go) * inv;
                        float gv;
                        if (KIND == FAVOR_KERNEL_SOFTMAX_POS) gv = dphi * ex2(fmaf(pv, a, c));
                        else gv = pv > 0.f ? dphi : 0.f;
                        gg[e] = gv;
                        gsum += gv;
                    }
                    split_pack(gg[0], gg[1], hw[i], lw[i]);
                }
                tmem_st16(tu + 16 * cc, hw);
                tmem_st16(tp + 16 * cc, lw);
            }
            tmem_st_wait();
            if (live && ch == 0)
                rowstat[(size_t)bh * L + tok] = make_float4(den, KIND == FAVOR_KERNEL_SOFTMAX_POS ? s * mx : 0.f, go, 0.f);
            __syncthreads();   // the den / fu partials are read; reuse red for gsum
            red[ch * kTile + row] = gsum;
        }
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            const uint32_t id_q = make_idesc(128, 64, 0, 1);
            const uint64_t bw = make_desc(s_w, 8192, 1024, SW_128B);
#pragma unroll
            for (int kk = 0; kk < 16; ++kk)   // G hi: features 16 kk .. +15 at 256 + 128 (kk / 8) + 8 (kk % 8)
                mma_ts(tmem + 64, tmem + 256 + 128 * (kk >> 3) + 8 * (kk & 7), bw + 128 * kk, id_q, kk > 0 ? 1u : 0u);
#pragma unroll
            for (int kk = 0; kk < 16; ++kk)   // G lo at 128 (kk / 8) + 8 (kk % 8)
                mma_ts(tmem + 64, tmem + 128 * (kk >> 3) + 8 * (kk & 7), bw + 128 * kk, id_q, 1u);
            mma_commit(&bars->mma);
        }
        ok = __syncthreads_and(mbar_wait(&bars->mma, 1, err, 46));
        if (!ok) break;
        tc_fence_after();
        gsum = red[row] + red[kTile + row];
        {
            // thread half ch writes columns 32 ch .. 32 ch + 31 of its row's dq
            uint32_t v0[32];
            tmem_ld32(tl + 64 + 32 * ch, v0);
            tmem_ld_wait();
            if (live) {
                uint4* dst = reinterpret_cast<uint4*>(dq + ((size_t)bh * L + tok) * kD);
#pragma unroll
                for (uint32_t c4 = 0; c4 < 4; ++c4) {
                    const uint32_t chk = 4 * ch + c4;
                    const uint4 x = ld_shared_v4(s_q + sw128((uint32_t)row, chk));
                    const uint32_t xin[4] = {x.x, x.y, x.z, x.w};
                    uint32_t w[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int c0 = 8 * c4 + 2 * i;
                        const float acc0 = __uint_as_float(v0[c0]), acc1 = __uint_as_float(v0[c0 + 1]);
                        float d0 = s * acc0, d1 = s * acc1;
                        if (KIND == FAVOR_KERNEL_SOFTMAX_POS) {
                            d0 = s * fmaf(-s * gsum, bf16lo(xin[i]), acc0);
                            d1 = s * fmaf(-s * gsum, bf16hi(xin[i]), acc1);
                        }
                        w[i] = pack_bf16(d0, d1);
                    }
                    dst[chk] = make_uint4(w[0], w[1], w[2], w[3]);
                }
            }
        }
        tc_fence_before();
    }
    if (!ok && tid == 0) pend.drain(bars, err, 44);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

// Key pass, persistent over the call's tile ranges (grid R.G, 256 threads: thread t takes
// key row t % 128 and features 128*(t/128) .. +127 of it).  Tensor memory per tile:
// P [0,256), dphi = V (dS hi + dS lo)^T [256,512); G packed as in the query pass (lo
// over the thread's P columns, hi over its dphi columns), dk [64,128), dv [192,256).
template <int KIND>
__global__ void __launch_bounds__(kBwdThreads, 1)
k_tc_bwd_k(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
           const __grid_constant__ CUtensorMap tm_w, const uint8_t* __restrict__ img,
           const float* __restrict__ kshift, __nv_bfloat16* __restrict__ dk, __nv_bfloat16* __restrict__ dvv, int H,
           int L, float s, Ranges R, int* err) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1k(smem_raw);
    const uint32_t s_w = smem_u32(sm);
    const uint32_t s_img = s_w + kOmegaBytes;
    uint8_t* buf = sm + kOmegaBytes + kBImg;                      // 2 x [k tile | v tile]
    const uint32_t s_phi = s_img + kBImg + 4 * kTileBytes;       // [128 keys][256 features] bf16, four SW128 blocks
    const float* dz = reinterpret_cast<const float*>(sm + kOmegaBytes + 2 * kSBytes);
    BwBars* bars = reinterpret_cast<BwBars*>(sm + kOmegaBytes + kBImg + 4 * kTileBytes + 4 * kPhiBlock);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int row = tid & (kTile - 1), ch = tid >> 7;
    const int g0 = blockIdx.x * R.per, g1 = min(R.T, g0 + R.per);

    bw_init_bars(bars);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    const uint32_t tl = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    const uint32_t tp = tl + 128 * ch, tu = tl + 256 + 128 * ch;   // this thread's P and dphi columns
    const float a = s * kLog2e;
    BwPending pend;
    if (tid == 0 && g0 < g1) {
        bw_load_head(&tm_w, img, sm, bars, g0 / R.tph, (g0 / R.tph) % H);
        pend.head = 0;
        bw_load_tiles(&tm_k, &tm_v, buf, &bars->tile[0], g0, R.tph);
        pend.tile[0] = 0;
    }
    bool ok = true;
    int loaded_bh = -1;
    uint32_t nhead = 0;
    for (int g = g0, it = 0; g < g1; ++g, ++it) {
        const int b = it & 1;
        const int bh = g / R.tph, tile = g - bh * R.tph, h = bh % H;
        const int tok = tile * kTile + row;
        const bool live = tok < L;
        const uint32_t s_k = s_img + kBImg + b * 2 * kTileBytes, s_v = s_k + kTileBytes;
        // row partials [2][128]: in this tile's v buffer, which nothing reads after the dphi MMA
        float* red = reinterpret_cast<float*>(buf + b * 2 * kTileBytes + kTileBytes);
        __syncthreads();   // the previous tile is done with its buffers, features and tensor memory
        const bool new_head = bh != loaded_bh;
        if (tid == 0) {
            if (new_head && it > 0) {
                bw_load_head(&tm_w, img, sm, bars, bh, h);
                pend.head = (int)(nhead & 1);
            }
            if (g + 1 < g1) {
                bw_load_tiles(&tm_k, &tm_v, buf + (b ^ 1) * 2 * kTileBytes, &bars->tile[b ^ 1], g + 1, R.tph);
                pend.tile[b ^ 1] = ((it + 1) >> 1) & 1;
            }
        }
        if (new_head) {
            ok = __syncthreads_and(mbar_wait(&bars->head, nhead & 1, err, 47));
            ++nhead;
            loaded_bh = bh;
            if (!ok) break;
            pend.head = -1;
        }
        ok = __syncthreads_and(mbar_wait(&bars->tile[b], (it >> 1) & 1, err, 51));
        if (!ok) break;
        pend.tile[b] = -1;
        if (tid == 0) {
            tc_fence_after();
            issue_projection(tmem, s_k, s_w, 256);
            const uint32_t id_u = make_idesc(128, 256, 0, 0);
            const uint64_t a0 = make_desc(s_v, 16, 1024, SW_128B);
            const uint64_t bh0 = make_desc(s_img, 16, 1024, SW_128B);
            const uint64_t bl0 = make_desc(s_img + kSBytes, 16, 1024, SW_128B);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) mma_ss(tmem + 256, a0 + 2 * kk, bh0 + 2 * kk, id_u, kk > 0 ? 1u : 0u);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) mma_ss(tmem + 256, a0 + 2 * kk, bl0 + 2 * kk, id_u, 1u);
            mma_commit(&bars->mma);
        }
        ok = __syncthreads_and(mbar_wait(&bars->mma, 0, err, 48));
        if (!ok) break;
        tc_fence_after();
        float gsum = 0.f;
        {
            const float c = live ? -(0.5f * s * s * row_sqnorm(s_k, (uint32_t)row) + kshift[h]) * kLog2e : -INFINITY;
            for (int cc = 0; cc < 4; ++cc) {
                uint32_t pw[32], uw[32];
                tmem_ld32(tp + 32 * cc, pw);
                tmem_ld32(tu + 32 * cc, uw);
                tmem_ld_wait();
                uint32_t hw[16], lw[16], fw[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    float gg[2], ff[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int k = 2 * i + e;
                        const float pv = __uint_as_float(pw[k]);
                        const float dphi = __uint_as_float(uw[k]) + dz[128 * ch + 32 * cc + k];
                        float f, gv;
                        if (KIND == FAVOR_KERNEL_SOFTMAX_POS) {
                            f = ex2(fmaf(pv, a, c));
                            gv = dphi * f;
                        } else {
                            f = live ? fmaxf(s * pv, 0.f) : 0.f;
                            gv = live && pv > 0.f ? dphi : 0.f;
                        }
                        ff[e] = f;
                        gg[e] = gv;
                        gsum += gv;
                    }
                    split_pack(gg[0], gg[1], hw[i], lw[i]);
                    fw[i] = pack_bf16(ff[0], ff[1]);
                }
                tmem_st16(tu + 16 * cc, hw);
                tmem_st16(tp + 16 * cc, lw);
                // features of this row: global 32-column chunk gc = 4 ch + cc = chunks 4 (gc % 2) .. +3 of block gc / 2
                const int gc = 4 * ch + cc;
                const uint32_t blk = s_phi + (uint32_t)(gc >> 1) * kPhiBlock;
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    st_shared_v4(blk + sw128((uint32_t)row, (uint32_t)(4 * (gc & 1) + q)), fw[4 * q], fw[4 * q + 1],
                                 fw[4 * q + 2], fw[4 * q + 3]);
            }
            tmem_st_wait();
            red[ch * kTile + row] = gsum;
            fence_async_smem();   // generic writes (features, partials) before later async-proxy use
        }
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            const uint32_t id_q = make_idesc(128, 64, 0, 1);
            const uint64_t bw = make_desc(s_w, 8192, 1024, SW_128B);
#pragma unroll
            for (int kk = 0; kk < 16; ++kk)
                mma_ts(tmem + 64, tmem + 256 + 128 * (kk >> 3) + 8 * (kk & 7), bw + 128 * kk, id_q, kk > 0 ? 1u : 0u);
#pragma unroll
            for (int kk = 0; kk < 16; ++kk)
                mma_ts(tmem + 64, tmem + 128 * (kk >> 3) + 8 * (kk & 7), bw + 128 * kk, id_q, 1u);
            const uint64_t bs = make_desc(s_img, 8192, 1024, SW_128B);
#pragma unroll
            for (int kk = 0; kk < 16; ++kk) {
                const uint64_t af = make_desc(s_phi + (uint32_t)(kk >> 2) * kPhiBlock + (uint32_t)(kk & 3) * 32, 16,
                                              1024, SW_128B);
                mma_ss(tmem + 192, af, bs + 128 * kk, id_q, kk > 0 ? 1u : 0u);
            }
            mma_commit(&bars->mma);
        }
        ok = __syncthreads_and(mbar_wait(&bars->mma, 1, err, 49));
        if (!ok) break;
        tc_fence_after();
        gsum = red[row] + red[kTile + row];
        {
            // thread half ch writes columns 32 ch .. 32 ch + 31 of its row's dk and dv
            uint32_t v0[32], w0[32];
            tmem_ld32(tl + 64 + 32 * ch, v0);
            tmem_ld32(tl + 192 + 32 * ch, w0);
            tmem_ld_wait();
            if (live) {
                uint4* dstk = reinterpret_cast<uint4*>(dk + ((size_t)bh * L + tok) * kD);
                uint4* dstv = reinterpret_cast<uint4*>(dvv + ((size_t)bh * L + tok) * kDV);
#pragma unroll
                for (uint32_t c4 = 0; c4 < 4; ++c4) {
                    const uint32_t chk = 4 * ch + c4;
                    const uint4 x = ld_shared_v4(s_k + sw128((uint32_t)row, chk));
                    const uint32_t xin[4] = {x.x, x.y, x.z, x.w};
                    uint32_t wk[4], wv[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int c0 = 8 * c4 + 2 * i;
                        const float k0 = __uint_as_float(v0[c0]), k1 = __uint_as_float(v0[c0 + 1]);
                        float d0 = s * k0, d1 = s * k1;
                        if (KIND == FAVOR_KERNEL_SOFTMAX_POS) {
                            d0 = s * fmaf(-s * gsum, bf16lo(xin[i]), k0);
                            d1 = s * fmaf(-s * gsum, bf16hi(xin[i]), k1);
                        }
                        wk[i] = pack_bf16(d0, d1);
                        wv[i] = pack_bf16(__uint_as_float(w0[c0]), __uint_as_float(w0[c0 + 1]));
                    }
                    dstk[chk] = make_uint4(wk[0], wk[1], wk[2], wk[3]);
                    dstv[chk] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
                }
            }
        }
        tc_fence_before();
    }
    if (!ok && tid == 0) pend.drain(bars, err, 47);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

// ================================================================ host side
// the state kernel asks for more than half an SM's shared memory so that two
// CTAs (each allocating all 512 tensor-memory columns) never share an SM
constexpr size_t kSmemBState = 120 * 1024;
static_assert(1024 + kOmegaBytes + 5 * kTileBytes + 2 * kTile * 4 + sizeof(BwBars) <= kSmemBState, "bstate smem");
constexpr size_t kSmemBwdQ = 1024 + kOmegaBytes + kBImg + 4 * kTileBytes + 3 * 2 * kTile * 4 + sizeof(BwBars);
constexpr size_t kSmemBwdK = 1024 + kOmegaBytes + kBImg + 4 * kTileBytes + 4 * kPhiBlock + sizeof(BwBars);
static_assert(kSmemBwdK <= 232448, "backward key pass shared memory");

void allow_bwd_once() {
    static std::once_flag once;
    std::call_once(once, [] {
        allow_smem(k_tc_bstate<FAVOR_KERNEL_SOFTMAX_POS, 0>, kSmemBState);
        allow_smem(k_tc_bstate<FAVOR_KERNEL_SOFTMAX_POS, 1>, kSmemBState);
        allow_smem(k_tc_bstate<FAVOR_KERNEL_RELU, 0>, kSmemBState);
        allow_smem(k_tc_bstate<FAVOR_KERNEL_RELU, 1>, kSmemBState);
        allow_smem(k_tc_bwd_q<FAVOR_KERNEL_SOFTMAX_POS>, kSmemBwdQ);
        allow_smem(k_tc_bwd_q<FAVOR_KERNEL_RELU>, kSmemBwdQ);
        allow_smem(k_tc_bwd_k<FAVOR_KERNEL_SOFTMAX_POS>, kSmemBwdK);
        allow_smem(k_tc_bwd_k<FAVOR_KERNEL_RELU>, kSmemBwdK);
        cudaGetLastError();
    });
}

template <int KIND>
favor_status tc_bidir_backward_t(const Handle& h, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                                 const CUtensorMap& mdo, const CUtensorMap& mw, void* dq, void* dk, void* dv, int BH,
                                 int L, const Ranges& R, cudaStream_t st) {
    float4* rowstat = reinterpret_cast<float4*>(h.ws_rowstat);
    uint8_t* img = reinterpret_cast<uint8_t*>(h.ws_bimg);
    const dim3 cgrid((kM * (kDV + 1) + 255) / 256, BH);
    favor_status e;
    {
        ProfScope ps(h, PROF_STATE, st);
        k_tc_bstate<KIND, 0><<<R.G, kBStateThreads, kSmemBState, st>>>(mk, mv, mw, h.kshift, nullptr, h.ws_partial,
                                                                         h.H, L, h.s, R, h.dev_err);
        count_launch();
        if ((e = check_launch("backward state kernel")) != FAVOR_OK) return e;
    }
    {
        ProfScope ps(h, PROF_COMBINE, st);
        k_bwd_reduce_pack<<<cgrid, 256, 0, st>>>(h.ws_partial, img, R);
        count_launch();
        if ((e = check_launch("backward reduce/pack kernel")) != FAVOR_OK) return e;
    }
    {
        ProfScope ps(h, PROF_BWD_QUERY, st);
        k_tc_bwd_q<KIND><<<R.G, kBwdThreads, kSmemBwdQ, st>>>(mq, mdo, mw, img, (__nv_bfloat16*)dq, rowstat, h.H,
                                                                L, h.s, R, h.dev_err);
        count_launch();
        if ((e = check_launch("backward query kernel")) != FAVOR_OK) return e;
        k_tc_bstate<KIND, 1><<<R.G, kBStateThreads, kSmemBState, st>>>(mq, mdo, mw, h.kshift, rowstat, h.ws_partial,
                                                                         h.H, L, h.s, R, h.dev_err);
        count_launch();
        if ((e = check_launch("backward query-state kernel")) != FAVOR_OK) return e;
    }
    {
        ProfScope ps(h, PROF_COMBINE, st);
        k_bwd_reduce_pack<<<cgrid, 256, 0, st>>>(h.ws_partial, img, R);
        count_launch();
        if ((e = check_launch("backward reduce/pack kernel")) != FAVOR_OK) return e;
    }
    ProfScope ps(h, PROF_BWD_KEY, st);
    k_tc_bwd_k<KIND><<<R.G, kBwdThreads, kSmemBwdK, st>>>(mk, mv, mw, img, h.kshift, (__nv_bfloat16*)dk,
                                                            (__nv_bfloat16*)dv, h.H, L, h.s, R, h.dev_err);
    count_launch();
    return check_launch("backward key kernel");
}

}  // namespace

size_t tc_bwd_image_bytes(size_t BH) { return BH * kBImg; }

favor_status tc_bidir_backward(const Handle& h, const void* q, const void* k, const void* v, const void* dout,
                               void* dq, void* dk, void* dv, int B, int L, cudaStream_t st) {
    if (!h.ws_bimg || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dout) || !aligned16(dq) ||
        !aligned16(dk) || !aligned16(dv))
        return simt_bidir_backward(h, q, k, v, dout, dq, dk, dv, B, L, st);
    allow_bwd_once();
    const int BH = B * h.H;
    const Ranges R = plan_ranges(BH, L, h.num_sms);
    if ((size_t)BH * R.pstride > h.ws_partial_rows)
        return set_error(FAVOR_ERR_INVALID_ARG, "backward workspace too small (%d x %d rows)", BH, R.pstride);
    CUtensorMap mq, mk, mv, mdo, mw;
    if (!map_tokens(&mq, q, BH, L) || !map_tokens(&mk, k, BH, L) || !map_tokens(&mv, v, BH, L) ||
        !map_tokens(&mdo, dout, BH, L) || !map_omega(&mw, h.omega_bf16, h.H))
        return set_error(FAVOR_ERR_CUDA, "cuTensorMapEncodeTiled failed");
    if (h.kind == FAVOR_KERNEL_SOFTMAX_POS)
        return tc_bidir_backward_t<FAVOR_KERNEL_SOFTMAX_POS>(h, mq, mk, mv, mdo, mw, dq, dk, dv, BH, L, R, st);
    return tc_bidir_backward_t<FAVOR_KERNEL_RELU>(h, mq, mk, mv, mdo, mw, dq, dk, dv, BH, L, R, st);
}

}  // namespace favor
