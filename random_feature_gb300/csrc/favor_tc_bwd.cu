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

// ============================================================ backward (causal)
// The causal gradients of favor_bwd.cu, chunk by chunk (128 tokens) on the
// tensor cores.  With A = Phi_Q Phi_K^T and C = dO V^T inside a chunk, the
// exclusive prefix S, z of the keys before it (S = sum phi_k v^T, z = sum
// phi_k) and the exclusive suffix T, t of the queries after it (T = sum
// phi~_q dO^T, t = -sum phi~_q go, phi~_q = phi_q / den):
//   den_i = phi_q,i . z + sum_{j<=i} A_ij
//   go_i  = (phi_q,i . (S dO_i) + sum_{j<=i} A_ij C_ij) / den_i          (= dO_i . out_i)
//   dphi_q,i = (S dO_i - z go_i + sum_{j<=i} (C_ij - go_i) phi_k,j) / den_i
//   dphi_k,j = T v_j + t + sum_{i>=j} (C_ij - go_i) phi~_q,i
//   dv_j     = T^T phi_k,j + sum_{i>=j} (phi_k,j . phi~_q,i) dO_i
// The states of each CTA's piece of a head come from k_tc_bstate (MODE 0: S,
// z; MODE 1: T, t) and a fixed-order scan over the pieces; inside the piece
// the query pass carries S, z forward and the key pass carries T, t backward,
// thread f holding feature row f in fp32 registers and writing the next
// chunk's hi + lo image.  The subtractions S dO_i - z go_i and T v_j + t, as
// in the bidirectional passes, need the states near fp32, so each chunk's
// increment takes its features as hi + lo pairs (kept in tensor memory where
// the transposed projection left them).  In the query pass the in-chunk
// products take the key features and B as bf16 pairs too (dq cancels the
// most); the key pass's in-chunk term of dk takes f16 operands under
// power-of-two scales; dv, which subtracts nothing, takes bf16.
//
//   k_tc_bstate<MODE 0>, k_piece_scan<false>   K, V            -> prefix S, z per piece
//   k_tc_cbwd_q                                Q, K, V, dO     -> dq, rowstat (den, row shift, go, ReLU f16 scale)
//   k_tc_bstate<MODE 1>, k_piece_scan<true>    Q, dO, rowstat  -> suffix T, t per piece
//   k_tc_cbwd_k                                Q, K, V, dO     -> dk
//   k_tc_cbwd_v                                Q, K, dO        -> dv
//
// Shared memory of both passes (from a 1 KB boundary): omega 32 KB | state
// image hi, lo 64 KB | Q, K, V, dO tiles 64 KB | features [2 token blocks][256]
// [64] bf16 64 KB | z or t fp32 [256] | [128] fp32 column terms | barriers.
// Each tile buffer is reloaded with the next chunk's tile as soon as the chunk
// is done with it; the K tile (query pass) and the Q tile (key pass) also hold
// row partials or the queries' statistics between their last read and that load.
constexpr uint32_t kCbImgOff = kOmegaBytes;
constexpr uint32_t kCbTiles = kCbImgOff + 2 * kSBytes;
constexpr uint32_t kCbPhi = kCbTiles + 4 * kTileBytes;
constexpr uint32_t kCbVec = kCbPhi + 4 * kPhiBlock;
constexpr uint32_t kCbBars = kCbVec + kM * 4 + kTile * 4;
enum { CB_Q = 0, CB_K = 1, CB_V = 2, CB_O = 3 };

struct CbBars {
    uint64_t w;         // omega
    uint64_t tile[4];   // Q, K, V, dO buffers (one load per chunk each)
    uint64_t mma;
    uint32_t tmem_base;
    uint32_t pad;
};

// Loads issued and not yet waited for (parity, -1 when none), drained
// (bounded) by the issuing thread before a CTA whose wait gave up exits.
struct CbPending {
    int w = -1, tile[4] = {-1, -1, -1, -1};
    __device__ __forceinline__ void drain(CbBars* bars, int* err, int code) {
        if (w >= 0) mbar_wait(&bars->w, (uint32_t)w, err, code);
        for (int b = 0; b < 4; ++b)
            if (tile[b] >= 0) mbar_wait(&bars->tile[b], (uint32_t)tile[b], err, code);
    }
};

__device__ __forceinline__ void cb_init(CbBars* bars) {
    if (threadIdx.x == 0) {
        mbar_init(&bars->w, 1);
        for (int b = 0; b < 4; ++b) mbar_init(&bars->tile[b], 1);
        mbar_init(&bars->mma, 1);
        fence_mbar_init();
    }
    if (threadIdx.x / 32 == 0) {
        tmem_alloc(&bars->tmem_base, 512);
        tmem_relinquish();
    }
}

__device__ __forceinline__ void cb_load_tile(const CUtensorMap* m, uint8_t* sm, int buf, CbBars* bars, int g,
                                             int tph) {
    const int bh = g / tph, tile = g - bh * tph;
    mbar_expect_tx(&bars->tile[buf], kTileBytes);
    tma_load_3d(sm + kCbTiles + buf * kTileBytes, m, &bars->tile[buf], 0, tile * kTile, bh);
}

__device__ __forceinline__ void cb_load_omega(const CUtensorMap* m, uint8_t* sm, CbBars* bars, int h) {
    mbar_expect_tx(&bars->w, kOmegaBytes);
    tma_load_2d(sm, m, &bars->w, 0, h * kM);
}

// Two floats -> packed f16x2 (round to nearest even); `lo` in the low half.
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Instruction descriptor of kind::f16 with f16 A and B (format 0), fp32 accumulator.
__host__ __device__ constexpr uint32_t make_idesc_h(int M, int N, int a_mn, int b_mn) {
    return (1u << 4) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

// 2^e, e in [-126, 127] (exact); floor(log2 x) of a finite normal x > 0.
__device__ __forceinline__ float exp2i(int e) { return __int_as_float((e + 127) << 23); }
__device__ __forceinline__ int ilog2f(float x) { return (int)((__float_as_uint(x) >> 23) & 0xFFu) - 127; }

// Power-of-two exponent e with m 2^-e in [2^13, 2^14) for m > 0 (0 for m = 0), clamped to +-100:
// values up to m scaled by 2^-e stay inside f16's normal range with 11 significant bits.
__device__ __forceinline__ int f16_scale_exp(float m) {
    if (!(m > 0.f)) return 0;
    return max(-100, min(100, ilog2f(m) - 13));
}

// D[128 x N] = A tile [128 rows][64] . B rows [N][64]^T (both K-major SW128), N = 64 or 128.
__device__ __forceinline__ void cb_project(uint32_t d, uint32_t a_tile, uint32_t b_rows, int N) {
    const uint32_t id = make_idesc(128, N, 0, 0);
    const uint64_t a0 = make_desc(a_tile, 16, 1024, SW_128B);
    const uint64_t b0 = make_desc(b_rows, 16, 1024, SW_128B);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) mma_ss(d, a0 + 2 * kk, b0 + 2 * kk, id, kk > 0 ? 1u : 0u);
}

// D[128 tokens][256 features] = X tile . (state hi + state lo)^T, the state image [256][64] K-major.
__device__ __forceinline__ void cb_state_mult(uint32_t d, uint32_t x_tile, uint32_t img) {
    const uint32_t id_u = make_idesc(128, 256, 0, 0);
    const uint64_t a0 = make_desc(x_tile, 16, 1024, SW_128B);
    const uint64_t bh0 = make_desc(img, 16, 1024, SW_128B);
    const uint64_t bl0 = make_desc(img + kSBytes, 16, 1024, SW_128B);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) mma_ss(d, a0 + 2 * kk, bh0 + 2 * kk, id_u, kk > 0 ? 1u : 0u);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) mma_ss(d, a0 + 2 * kk, bl0 + 2 * kk, id_u, 1u);
}

// The chunk's state increment, half h of the features into d_h (128 lanes = features, 64
// columns): D_h = F^T_h Y with the features F^T_h in tensor memory as hi + lo pairs (at x_h:
// token block u at + 64 u, hi then lo, 8 columns per 16 tokens) and Y a token tile [128
// tokens][64] (MN-major).
__device__ __forceinline__ void cb_state_inc(uint32_t d0, uint32_t d1, uint32_t x0, uint32_t x1, uint32_t y_tile) {
    const uint32_t id_o = make_idesc(128, 64, 0, 1);
    const uint64_t by = make_desc(y_tile, 8192, 1024, SW_128B);
#pragma unroll
    for (int hp = 0; hp < 2; ++hp) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const uint32_t hi = (hp ? x1 : x0) + 64 * (kk >> 2) + 8 * (kk & 3);
            mma_ts(hp ? d1 : d0, hi, by + 128 * kk, id_o, kk > 0 ? 1u : 0u);
            mma_ts(hp ? d1 : d0, hi + 32, by + 128 * kk, id_o, 1u);
        }
    }
}

// D[128 rows][128 tokens] = X . F where X is packed f16 (F16) or bf16 in tensor memory (features 0..127 at
// x0, 128..255 at x1, 8 columns per 16 features) and F the features [feature][token] in shared
// memory (MN-major, N = token in two 64-token blocks).
template <bool F16>
__device__ __forceinline__ void cb_scores(uint32_t d, uint32_t x0, uint32_t x1, uint32_t feat) {
    const uint32_t id_a = F16 ? make_idesc_h(128, 128, 0, 1) : make_idesc(128, 128, 0, 1);
    const uint64_t bf = make_desc(feat, 2 * kPhiBlock, 1024, SW_128B);
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) mma_ts(d, kk < 8 ? x0 + 8 * kk : x1 + 8 * (kk - 8), bf + 128 * kk, id_a, kk > 0 ? 1u : 0u);
}

// D[128 rows][256 features] += W . F^T where W is packed f16 in tensor memory (tokens 0..63 at
// w0, 64..127 at w1) and F the features [feature][token] in shared memory (K-major over tokens).
__device__ __forceinline__ void cb_weighted_features(uint32_t d, uint32_t w0, uint32_t w1, uint32_t feat) {
    const uint32_t id_b = make_idesc_h(128, 256, 0, 0);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
        mma_ts(d, (kk < 4 ? w0 : w1) + 8 * (kk & 3),
               make_desc(feat + (uint32_t)(kk >> 2) * 2 * kPhiBlock + (uint32_t)(kk & 3) * 32, 16, 1024, SW_128B),
               id_b, 1u);
}

// D[128 rows][64] = G . omega (G hi then lo, packed in tensor memory: features 16 kk .. +15 at
// hi0/lo0 + 8 kk for kk < 8, hi1/lo1 + 8 (kk - 8) after).
__device__ __forceinline__ void cb_grad_omega(uint32_t d, uint32_t hi0, uint32_t hi1, uint32_t lo0, uint32_t lo1,
                                              uint32_t s_w) {
    const uint32_t id_q = make_idesc(128, 64, 0, 1);
    const uint64_t bw = make_desc(s_w, 8192, 1024, SW_128B);
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) mma_ts(d, kk < 8 ? hi0 + 8 * kk : hi1 + 8 * (kk - 8), bw + 128 * kk, id_q, kk > 0 ? 1u : 0u);
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) mma_ts(d, kk < 8 ? lo0 + 8 * kk : lo1 + 8 * (kk - 8), bw + 128 * kk, id_q, 1u);
}

// Row r of the hi + lo state image from a fp32 state row times sc (a power of two).
__device__ __forceinline__ void cb_write_image(uint32_t img, uint32_t r, const float (&x)[64], float sc) {
#pragma unroll
    for (uint32_t c = 0; c < 8; ++c) {
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) split_pack(x[8 * c + 2 * i] * sc, x[8 * c + 2 * i + 1] * sc, hi[i], lo[i]);
        st_shared_v4(img + sw128(r, c), hi[0], hi[1], hi[2], hi[3]);
        st_shared_v4(img + kSBytes + sw128(r, c), lo[0], lo[1], lo[2], lo[3]);
    }
}

// Feature row f of 64 tokens (fp32 projections: 64 columns at taddr).  x_t = exp2(a p + off_t)
// (positive) or max(p off_t, 0) (ReLU: off_t = the token's scale, 0 past L) goes to row f of the
// features block `feat` ([feature][token], shared memory) as f16 (f16 true) or bf16; the value
// e_t = x_t mt_t ms (mt may be null) goes over the row's own columns as a bf16 pair hi + lo (hi at
// taddr, lo at taddr + 32, 8 columns per 16 tokens).  Returns sum_t e_t wt_t (wt null: weights 1).
template <int KIND, bool F16>
__device__ __forceinline__ float cb_feature_row(uint32_t taddr, uint32_t feat, uint32_t f, float a,
                                                const float* off, const float* mt, float ms, const float* wt) {
    uint32_t p0[32], p1[32];
    tmem_ld32(taddr, p0);
    tmem_ld32(taddr + 32, p1);
    tmem_ld_wait();
    float acc = 0.f;
    uint32_t x0[16], x1[16], h0[16], h1[16], l0[16], l1[16];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        float x[2], e[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int t = 2 * i + u;
            const float pv = __uint_as_float(t < 32 ? p0[t] : p1[t - 32]);
            x[u] = KIND == FAVOR_KERNEL_SOFTMAX_POS ? ex2(fmaf(pv, a, off[t])) : fmaxf(pv * off[t], 0.f);
            e[u] = (mt ? x[u] * mt[t] : x[u]) * ms;
            acc = wt ? fmaf(e[u], wt[t], acc) : acc + e[u];
        }
        const uint32_t xp = F16 ? pack_f16(x[0], x[1]) : pack_bf16(x[0], x[1]);
        if (i < 16) {
            x0[i] = xp;
            split_pack(e[0], e[1], h0[i], l0[i]);
        } else {
            x1[i - 16] = xp;
            split_pack(e[0], e[1], h1[i - 16], l1[i - 16]);
        }
    }
#pragma unroll
    for (uint32_t c = 0; c < 4; ++c) {
        st_shared_v4(feat + sw128(f, c), x0[4 * c], x0[4 * c + 1], x0[4 * c + 2], x0[4 * c + 3]);
        st_shared_v4(feat + sw128(f, 4 + c), x1[4 * c], x1[4 * c + 1], x1[4 * c + 2], x1[4 * c + 3]);
    }
    tmem_st16(taddr, h0);
    tmem_st16(taddr + 16, h1);
    tmem_st16(taddr + 32, l0);
    tmem_st16(taddr + 48, l1);
    return acc;
}

// dx row epilogue: columns 32 ch .. +31 of d = s (acc - s gsum x) (positive) or s acc (ReLU), bf16,
// stored when dst_row is not null (the tensor-memory load is warp-wide).
template <int KIND>
__device__ __forceinline__ void cb_store_grad(__nv_bfloat16* dst_row, uint32_t taddr, int ch, float s, float gsum,
                                              const uint4 (&xrow)[4]) {
    uint32_t v0[32];
    tmem_ld32(taddr, v0);
    tmem_ld_wait();
    if (!dst_row) return;
    uint4* dst = reinterpret_cast<uint4*>(dst_row);
#pragma unroll
    for (uint32_t c4 = 0; c4 < 4; ++c4) {
        const uint32_t xin[4] = {xrow[c4].x, xrow[c4].y, xrow[c4].z, xrow[c4].w};
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
        dst[4 * ch + c4] = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// Key features of feature row f for 64 keys (fp32 projections: 64 columns at taddr): x_t =
// exp2(a p + off_t) (positive) or max(p off_t, 0) (ReLU: off_t = s for a live key, 0 past L).
// SMEM: the pair hi + lo of x into row f of the [256 features][64 keys] blocks hi_blk, lo_blk;
// TMEM: the pair over the row's own columns (hi at taddr, lo at taddr + 32, 8 columns per 16
// keys).  Returns sum_t x_t.
template <int KIND, bool SMEM, bool TMEM>
__device__ __forceinline__ float cb_key_row_hl(uint32_t taddr, uint32_t hi_blk, uint32_t lo_blk, uint32_t f,
                                               float a, const float* off) {
    uint32_t p0[32], p1[32];
    tmem_ld32(taddr, p0);
    tmem_ld32(taddr + 32, p1);
    tmem_ld_wait();
    float acc = 0.f;
    uint32_t h0[16], h1[16], l0[16], l1[16];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        float x[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int t = 2 * i + u;
            const float pv = __uint_as_float(t < 32 ? p0[t] : p1[t - 32]);
            x[u] = KIND == FAVOR_KERNEL_SOFTMAX_POS ? ex2(fmaf(pv, a, off[t])) : fmaxf(pv * off[t], 0.f);
            acc += x[u];
        }
        if (i < 16) split_pack(x[0], x[1], h0[i], l0[i]);
        else split_pack(x[0], x[1], h1[i - 16], l1[i - 16]);
    }
    if (SMEM) {
#pragma unroll
        for (uint32_t c = 0; c < 4; ++c) {
            st_shared_v4(hi_blk + sw128(f, c), h0[4 * c], h0[4 * c + 1], h0[4 * c + 2], h0[4 * c + 3]);
            st_shared_v4(hi_blk + sw128(f, 4 + c), h1[4 * c], h1[4 * c + 1], h1[4 * c + 2], h1[4 * c + 3]);
            st_shared_v4(lo_blk + sw128(f, c), l0[4 * c], l0[4 * c + 1], l0[4 * c + 2], l0[4 * c + 3]);
            st_shared_v4(lo_blk + sw128(f, 4 + c), l1[4 * c], l1[4 * c + 1], l1[4 * c + 2], l1[4 * c + 3]);
        }
    }
    if (TMEM) {
        tmem_st16(taddr, h0);
        tmem_st16(taddr + 16, h1);
        tmem_st16(taddr + 32, l0);
        tmem_st16(taddr + 48, l1);
    }
    return acc;
}

// D[128 rows][64 keys] = X . (K_hi + K_lo) where X is packed bf16 in tensor memory (features
// 0..127 at x0, 128..255 at x1, 8 columns per 16 features) and K_hi, K_lo the key features
// [256 features][64 keys] in shared memory (MN-major, N = key).
__device__ __forceinline__ void cb_scores_half(uint32_t d, uint32_t x0, uint32_t x1, uint32_t khi, uint32_t klo) {
    const uint32_t id = make_idesc(128, 64, 0, 1);
    const uint64_t bh0 = make_desc(khi, 8192, 1024, SW_128B), bl0 = make_desc(klo, 8192, 1024, SW_128B);
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) mma_ts(d, kk < 8 ? x0 + 8 * kk : x1 + 8 * (kk - 8), bh0 + 128 * kk, id, kk > 0 ? 1u : 0u);
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) mma_ts(d, kk < 8 ? x0 + 8 * kk : x1 + 8 * (kk - 8), bl0 + 128 * kk, id, 1u);
}

// D[128 rows][256 features] += W . F for 64 keys, W = W_hi + W_lo packed bf16 in tensor memory
// (8 columns per 16 keys at whi, wlo) and F = F_hi + F_lo the keys' features [256 features][64
// keys] in shared memory (K-major over keys): W_hi F_hi + W_lo F_hi + W_hi F_lo.
__device__ __forceinline__ void cb_weighted_half(uint32_t d, uint32_t whi, uint32_t wlo, uint32_t fhi, uint32_t flo) {
    const uint32_t id = make_idesc(128, 256, 0, 0);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
        const uint64_t bh = make_desc(fhi + (uint32_t)kk * 32, 16, 1024, SW_128B);
        const uint64_t bl = make_desc(flo + (uint32_t)kk * 32, 16, 1024, SW_128B);
        mma_ts(d, whi + 8 * kk, bh, id, 1u);
        mma_ts(d, wlo + 8 * kk, bh, id, 1u);
        mma_ts(d, whi + 8 * kk, bl, id, 1u);
    }
}

// The masked sums of 32 keys j0 .. j0+31 of row `row`: den += sum_{j<=row} A_j, fu += sum_{j<=row} A_j C_j
// (A at ta, C at tc, 32 fp32 columns each).
__device__ __forceinline__ void cb_masked_sums(uint32_t ta, uint32_t tc, int j0, int row, float& den, float& fu) {
    uint32_t av[32], cv[32];
    tmem_ld32(ta, av);
    tmem_ld32(tc, cv);
    tmem_ld_wait();
#pragma unroll
    for (int k = 0; k < 32; ++k) {
        if (j0 + k <= row) {
            const float av_k = __uint_as_float(av[k]);
            den += av_k;
            fu = fmaf(av_k, __uint_as_float(cv[k]), fu);
        }
    }
}

// Two / four consecutive tensor-memory columns of this thread's lane.
__device__ __forceinline__ void tmem_st2(uint32_t taddr, const uint32_t (&r)[2]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x2.b32 [%0], {%1, %2};" ::"r"(taddr), "r"(r[0]), "r"(r[1])
                 : "memory");
}
__device__ __forceinline__ void tmem_ld4(uint32_t taddr, uint32_t (&r)[4]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(taddr)
                 : "memory");
}

// Query pass, persistent over the call's tile ranges (grid R.G, 256 threads).  Thread t is
// query row t % 128 with features 128 (t / 128) .. +127 of it (the same split as the
// bidirectional query pass), and feature row t of the key features and of the running prefix
// state.  dq cancels strongly (sum_f G_f (omega_f - s x) with sum_f G_f = 0), so every product
// inside a chunk takes the key features as bf16 pairs hi + lo, and B as a pair too; the query
// features enter A as bf16, and the parts from before the chunk take the same rounded values,
// so that den and dO . out are exact for them.  Shared memory holds the pairs of 64 keys at a
// time: the scores and B Phi_K run in two key halves, each half's features recomputed from its
// projection when its turn comes.  Tensor memory per chunk (columns):
//   P0  P_K^T halves [0,128) [128,256) -> key features hi + lo in place (keys 0..63 also in
//       shared memory)
//   P1  dS halves [256,320) [320,384), P_Q [0,256)
//   P2  U = dO S~^T [256,512) -> bf16 Phi_Q over [0,64) [128,192)
//   P3  A (keys 0..63) [256,320), C [384,512), P_K^T of keys 64..127 [320,384) [192,256)
//   P4  A (keys 64..127) [256,320) -> B = tril(C - go) hi, lo over C: keys 64c .. +63 of
//       thread half c at [384 + 64c, +32) and [416 + 64c, +32); row partials exchanged in
//       columns 320..323
//   P5  U = dO S~^T + B Phi_K (keys 64..127) [0,256), P_K^T of keys 0..63 [256,320) [320,384)
//   P6  U += B Phi_K (keys 0..63), P_Q again [256,512) -> G hi over U, lo over P
//   P7  dq [64,128)
template <int KIND>
__global__ void __launch_bounds__(kBwdThreads, 1)
k_tc_cbwd_q(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
            const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
            const __grid_constant__ CUtensorMap tm_w, const float* __restrict__ prefix,
            const float* __restrict__ kshift, __nv_bfloat16* __restrict__ dq, float4* __restrict__ rowstat, int H,
            int L, float s, Ranges R, int* err) {
    constexpr bool POS = KIND == FAVOR_KERNEL_SOFTMAX_POS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1k(smem_raw);
    const uint32_t s_w = smem_u32(sm);
    const uint32_t s_img = s_w + kCbImgOff;
    const uint32_t s_q = s_w + kCbTiles, s_k = s_q + kTileBytes, s_v = s_k + kTileBytes, s_do = s_v + kTileBytes;
    const uint32_t s_khi = s_w + kCbPhi, s_klo = s_khi + 2 * kPhiBlock;   // 64 keys' features hi | lo
    float* zv = reinterpret_cast<float*>(sm + kCbVec);                     // z of the chunk's prefix
    float* kc = zv + kM;                                                    // key column terms
    float* redg = reinterpret_cast<float*>(sm + kCbPhi);                   // gsum partials, in the features
    CbBars* bars = reinterpret_cast<CbBars*>(sm + kCbBars);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int row = tid & (kTile - 1), ch = tid >> 7;
    const int cta = blockIdx.x;
    const int g0 = cta * R.per, g1 = min(R.T, g0 + R.per);

    cb_init(bars);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    const uint32_t tl = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    const float a = s * kLog2e;
    CbPending pend;
    int w_h = -1;
    if (g0 < g1) {
        w_h = (g0 / R.tph) % H;
        if (tid == 0) {
            cb_load_omega(&tm_w, sm, bars, w_h);
            pend.w = 0;
            for (int b = 0; b < 4; ++b) {
                cb_load_tile(b == CB_Q ? &tm_q : b == CB_K ? &tm_k : b == CB_V ? &tm_v : &tm_do, sm, b, bars, g0, R.tph);
                pend.tile[b] = 0;
            }
        }
    }
    bool w_wait = g0 < g1;
    float srun[64];
    float zrun = 0.f;
    bool ok = true;
    int cur_bh = -1;
    uint32_t nw = 0, nmma = 0;
    for (int g = g0, it = 0; g < g1; ++g, ++it) {
        const int bh = g / R.tph, tile = g - bh * R.tph, h = bh % H;
        const int tok0 = tile * kTile, tok = tok0 + row;
        const bool live = tok < L;
        const uint32_t tpar = (uint32_t)(it & 1);
        const bool more = g + 1 < g1;
        __syncthreads();   // the previous chunk is done with its buffers and tensor memory
        if (bh != cur_bh) {
            if (h != w_h) {
                if (tid == 0) {
                    cb_load_omega(&tm_w, sm, bars, h);
                    pend.w = (int)(nw & 1);
                }
                w_h = h;
                w_wait = true;
            }
            // the piece's prefix state, feature row tid, and its image
            const float* pre = prefix + ((size_t)bh * R.pstride + (cta - first_cta(R, bh))) * (kM * (kDV + 1)) +
                               (size_t)tid * (kDV + 1);
#pragma unroll
            for (int c = 0; c < 64; ++c) srun[c] = pre[c];
            zrun = pre[kDV];
            cb_write_image(s_img, (uint32_t)tid, srun, 1.f);
            zv[tid] = zrun;
            fence_async_smem();
            cur_bh = bh;
            if (w_wait) {
                ok = __syncthreads_and(mbar_wait(&bars->w, nw & 1, err, 60));
                ++nw;
                w_wait = false;
                if (!ok) break;
                pend.w = -1;
            }
        }
        // ---- P0: key projection (transposed) -> key features (hi + lo), their sums
        ok = __syncthreads_and(mbar_wait(&bars->tile[CB_K], tpar, err, 61));
        if (!ok) break;
        pend.tile[CB_K] = -1;
        if (tid == 0) {
            tc_fence_after();
            cb_project(tmem, s_w, s_k, 128);
            cb_project(tmem + 128, s_w + 128 * 128, s_k, 128);
            mma_commit(&bars->mma);
        }
        if (tid < kTile) {
            const bool kl = tok0 + tid < L;
            if (POS) kc[tid] = kl ? -(0.5f * s * s * row_sqnorm(s_k, (uint32_t)tid) + kshift[h]) * kLog2e : -INFINITY;
            else kc[tid] = kl ? s : 0.f;
        }
        ok = __syncthreads_and(mbar_wait(&bars->mma, nmma & 1, err, 62));
        ++nmma;
        if (!ok) break;
        tc_fence_after();
        float zc = cb_key_row_hl<KIND, true, true>(tl + 128 * ch, s_khi, s_klo, (uint32_t)tid, a, kc);
        zc += cb_key_row_hl<KIND, false, true>(tl + 128 * ch + 64, s_khi, s_klo, (uint32_t)tid, a, kc + 64);
        tmem_st_wait();
        fence_async_smem();
        tc_fence_before();
        ok = __syncthreads_and(mbar_wait(&bars->tile[CB_Q], tpar, err, 63) &&
                               mbar_wait(&bars->tile[CB_V], tpar, err, 58));
        if (!ok) break;
        pend.tile[CB_Q] = pend.tile[CB_V] = -1;
        // ---- P1: the chunk's state increment dS = Phi_K^T V (hi + lo), the query projection
        if (tid == 0) {
            tc_fence_after();
            cb_state_inc(tmem + 256, tmem + 320, tmem, tmem + 128, s_v);
            issue_projection(tmem, s_q, s_w, 256);
            mma_commit(&bars->mma);
        }
        uint4 qrow[4];
#pragma unroll
        for (uint32_t c4 = 0; c4 < 4; ++c4)
            qrow[c4] = POS ? ld_shared_v4(s_q + sw128((uint32_t)row, 4 * (uint32_t)ch + c4)) : make_uint4(0, 0, 0, 0);
        ok = __syncthreads_and(mbar_wait(&bars->mma, nmma & 1, err, 65));
        ++nmma;
        if (!ok) break;
        tc_fence_after();
        {
            uint32_t d0[32], d1[32];
            tmem_ld32(tl + 256 + 64 * ch, d0);
            tmem_ld32(tl + 288 + 64 * ch, d1);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                srun[i] += __uint_as_float(d0[i]);
                srun[32 + i] += __uint_as_float(d1[i]);
            }
            zrun += zc;
        }
        // the row's largest projection over all 256 features (both halves of the row are read)
        float mx = -INFINITY;
#pragma unroll 1
        for (int cc = 0; cc < 8; ++cc) {
            uint32_t pw[32];
            tmem_ld32(tl + 32 * cc, pw);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) mx = fmaxf(mx, __uint_as_float(pw[i]));
        }
        const int eq = POS ? 0 : (s * mx > 0.f ? max(-100, min(100, ilog2f(s * mx) + 1)) : 0);
        const float c = -mx * a;
        tc_fence_before();
        ok = __syncthreads_and(mbar_wait(&bars->tile[CB_O], tpar, err, 64));
        if (!ok) break;
        pend.tile[CB_O] = -1;
        // ---- P2: U = dO S~^T (the prefix part); query features, den and dO . out of the prefix
        if (tid == 0) {
            tc_fence_after();
            cb_state_mult(tmem + 256, s_do, s_img);
            mma_commit(&bars->mma);
        }
        ok = __syncthreads_and(mbar_wait(&bars->mma, nmma & 1, err, 57));
        ++nmma;
        if (!ok) break;
        tc_fence_after();
        float den = 0.f, fu = 0.f;   // from the bf16 query features, as A uses them
#pragma unroll 1
        for (int cc = 0; cc < 4; ++cc) {
            uint32_t pw[32], uw[32];
            tmem_ld32(tl + 128 * ch + 32 * cc, pw);
            tmem_ld32(tl + 256 + 128 * ch + 32 * cc, uw);
            tmem_ld_wait();
            uint32_t fw[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float p0 = __uint_as_float(pw[2 * i]), p1 = __uint_as_float(pw[2 * i + 1]);
                fw[i] = POS ? pack_bf16(ex2(fmaf(p0, a, c)), ex2(fmaf(p1, a, c)))
                            : pack_bf16(fmaxf(s * p0, 0.f), fmaxf(s * p1, 0.f));
                const float f0 = bf16lo(fw[i]), f1 = bf16hi(fw[i]);
                const int k = 128 * ch + 32 * cc + 2 * i;
                den = fmaf(f0, zv[k], fmaf(f1, zv[k + 1], den));
                fu = fmaf(f0, __uint_as_float(uw[2 * i]), fmaf(f1, __uint_as_float(uw[2 * i + 1]), fu));
            }
            tmem_st16(tl + 128 * ch + 16 * cc, fw);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncthreads();
        // ---- P3: A for keys 0..63 (hi + lo), C = dO V^T, projections of keys 64..127
        if (tid == 0) {
            tc_fence_after();
            cb_scores_half(tmem + 256, tmem, tmem + 128, s_khi, s_klo);
            cb_project(tmem + 384, s_do, s_v, 128);
            cb_project(tmem + 320, s_w, s_k + 64 * 128, 64);
            cb_project(tmem + 192, s_w + 128 * 128, s_k + 64 * 128, 64);
            mma_commit(&bars->mma);
        }
        ok = __syncthreads_and(mbar_wait(&bars->mma, nmma & 1, err, 66));
        ++nmma;
        if (!ok) break;
        if (tid == 0 && more) {
            cb_load_tile(&tm_v, sm, CB_V, bars, g + 1, R.tph);
            pend.tile[CB_V] = (int)(tpar ^ 1);
        }
        tc_fence_after();
        cb_masked_sums(tl + 256 + 32 * ch, tl + 384 + 32 * ch, 32 * ch, row, den, fu);
        cb_key_row_hl<KIND, true, false>(ch == 0 ? tl + 320 : tl + 192, s_khi, s_klo, (uint32_t)tid, a, kc + 64);
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        // ---- P4: A for keys 64..127; den, go; B = tril(C - go) as hi + lo
        if (tid == 0) {
            tc_fence_after();
            cb_scores_half(tmem + 256, tmem, tmem + 128, s_khi, s_klo);
            mma_commit(&bars->mma);
        }
        ok = __syncthreads_and(mbar_wait(&bars->mma, nmma & 1, err, 59));
        ++nmma;
        if (!ok) break;
        tc_fence_after();
        cb_masked_sums(tl + 256 + 32 * ch, tl + 448 + 32 * ch, 64 + 32 * ch, row, den, fu);
        {
            // the row's two partials through tensor-memory columns 320..323
            const uint32_t xw[2] = {__float_as_uint(den), __float_as_uint(fu)};
            tmem_st2(tl + 320 + 2 * ch, xw);
            tmem_st_wait();
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        {
            uint32_t xr[4];
            tmem_ld4(tl + 320, xr);
            tmem_ld_wait();
            den = __uint_as_float(xr[0]) + __uint_as_float(xr[2]);
            fu = __uint_as_float(xr[1]) + __uint_as_float(xr[3]);
        }
        const float inv = den != 0.f ? 1.f / den : 0.f;
        const float go = fu * inv;
        if (live && ch == 0) rowstat[(size_t)bh * L + tok] = make_float4(den, POS ? s * mx : 0.f, go, (float)eq);
        {
            uint32_t c0[32], c1[32];
            tmem_ld32(tl + 384 + 64 * ch, c0);
            tmem_ld32(tl + 416 + 64 * ch, c1);
            tmem_ld_wait();
            uint32_t h0[16], h1[16], l0[16], l1[16];
            const int j0 = 64 * ch;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                split_pack(j0 + 2 * i <= row ? __uint_as_float(c0[2 * i]) - go : 0.f,
                           j0 + 2 * i + 1 <= row ? __uint_as_float(c0[2 * i + 1]) - go : 0.f, h0[i], l0[i]);
                split_pack(j0 + 32 + 2 * i <= row ? __uint_as_float(c1[2 * i]) - go : 0.f,
                           j0 + 33 + 2 * i <= row ? __uint_as_float(c1[2 * i + 1]) - go : 0.f, h1[i], l1[i]);
            }
            tmem_st16(tl + 384 + 64 * ch, h0);
            tmem_st16(tl + 400 + 64 * ch, h1);
            tmem_st16(tl + 416 + 64 * ch, l0);
            tmem_st16(tl + 432 + 64 * ch, l1);
            tmem_st_wait();
        }
        tc_fence_before();
        __syncthreads();
        // ---- P5: U = dO S~^T + B Phi_K (keys 64..127), projections of keys 0..63
        if (tid == 0) {
            tc_fence_after();
            cb_state_mult(tmem, s_do, s_img);
            cb_weighted_half(tmem, tmem + 448, tmem + 480, s_khi, s_klo);
            cb_project(tmem + 256, s_w, s_k, 64);
            cb_project(tmem + 320, s_w + 128 * 128, s_k, 64);
            mma_commit(&bars->mma);
        }
        ok = __syncthreads_and(mbar_wait(&bars->mma, nmma & 1, err, 67));
        ++nmma;
        if (!ok) break;
        if (tid == 0 && more) {
            cb_load_tile(&tm_k, sm, CB_K, bars, g + 1, R.tph);
            pend.tile[CB_K] = (int)(tpar ^ 1);
        }
        tc_fence_after();
        cb_key_row_hl<KIND, true, false>(tl + 256 + 64 * ch, s_khi, s_klo, (uint32_t)tid, a, kc);
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        // ---- P6: U += B Phi_K (keys 0..63), the query projection again; G
        if (tid == 0) {
            tc_fence_after();
            cb_weighted_half(tmem, tmem + 384, tmem + 416, s_khi, s_klo);
            issue_projection(tmem + 256, s_q, s_w, 256);
            mma_commit(&bars->mma);
        }
        ok = __syncthreads_and(mbar_wait(&bars->mma, nmma & 1, err, 56));
        ++nmma;
        if (!ok) break;
        if (tid == 0 && more) {
            cb_load_tile(&tm_q, sm, CB_Q, bars, g + 1, R.tph);
            cb_load_tile(&tm_do, sm, CB_O, bars, g + 1, R.tph);
            pend.tile[CB_Q] = pend.tile[CB_O] = (int)(tpar ^ 1);
        }
        tc_fence_after();
        float gsum = 0.f;
#pragma unroll 1
        for (int cc = 0; cc < 4; ++cc) {
            uint32_t pw[32], uw[32];
            tmem_ld32(tl + 256 + 128 * ch + 32 * cc, pw);
            tmem_ld32(tl + 128 * ch + 32 * cc, uw);
            tmem_ld_wait();
            uint32_t hw[16], lw[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                float gg[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int k = 2 * i + e;
                    const float pv = __uint_as_float(pw[k]);
                    const float dphi = (__uint_as_float(uw[k]) - zv[128 * ch + 32 * cc + k] * go) * inv;
                    const float gv = POS ? dphi * ex2(fmaf(pv, a, c)) : (pv > 0.f ? dphi : 0.f);
                    gg[e] = gv;
                    gsum += gv;
                }
                split_pack(gg[0], gg[1], hw[i], lw[i]);
            }
            tmem_st16(tl + 128 * ch + 16 * cc, hw);
            tmem_st16(tl + 256 + 128 * ch + 16 * cc, lw);
        }
        tmem_st_wait();
        redg[ch * kTile + row] = gsum;
        tc_fence_before();
        __syncthreads();
        // ---- P7: dq = G omega; meanwhile the next chunk's prefix image
        if (tid == 0) {
            tc_fence_after();
            cb_grad_omega(tmem + 64, tmem, tmem + 128, tmem + 256, tmem + 384, s_w);
            mma_commit(&bars->mma);
        }
        cb_write_image(s_img, (uint32_t)tid, srun, 1.f);
        zv[tid] = zrun;
        fence_async_smem();
        ok = __syncthreads_and(mbar_wait(&bars->mma, nmma & 1, err, 68));
        ++nmma;
        if (!ok) break;
        tc_fence_after();
        gsum = redg[row] + redg[kTile + row];
        cb_store_grad<KIND>(live ? dq + ((size_t)bh * L + tok) * kD : nullptr, tl + 64 + 32 * ch, ch, s, gsum, qrow);
        tc_fence_before();
    }
    if (!ok && tid == 0) pend.drain(bars, err, 69);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

// Key pass for dk, persistent over the call's tile ranges in reverse (grid R.G, 256 threads).
// Thread t is key row t % 128 with features 128 (t / 128) .. +127 of it, and feature row t of the
// query features and of the running suffix state.  The in-chunk term W Phi~_Q takes f16 operands:
// the query features f as the query pass scaled them (2^-eq_i; positive: f <= 1), W_ji = (C_ji -
// go_i) 2^eq_i / den_i times 2^-ew_j (the row's largest to [2^13, 2^14)), and V row j times
// 2^-ew_j so that U stays one sum.  Tensor memory per chunk (columns):
//   P_Q^T halves [256,384) [384,512) -> query features hi + lo in place (and f16 in shared memory)
//   dT halves [0,64) [64,128), C^T = V dO^T [128,256) -> W over [128,160) [192,224)
//   U = V T~^T + W Phi~_Q [256,512), P_K [0,256) -> G hi over U, lo over P
//   dk [64,128)
template <int KIND>
__global__ void __launch_bounds__(kBwdThreads, 1)
k_tc_cbwd_k(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
            const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
            const __grid_constant__ CUtensorMap tm_w, const float* __restrict__ suffix,
            const float* __restrict__ kshift, const float4* __restrict__ rowstat, __nv_bfloat16* __restrict__ dk,
            int H, int L, float s, Ranges R, int* err) {
    constexpr bool POS = KIND == FAVOR_KERNEL_SOFTMAX_POS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1k(smem_raw);
    const uint32_t s_w = smem_u32(sm);
    const uint32_t s_img = s_w + kCbImgOff;
    const uint32_t s_q = s_w + kCbTiles, s_k = s_q + kTileBytes, s_v = s_k + kTileBytes, s_do = s_v + kTileBytes;
    const uint32_t s_phi = s_w + kCbPhi;
    float* tv = reinterpret_cast<float*>(sm + kCbVec);                 // t of the chunk's suffix
    float* qs = reinterpret_cast<float*>(sm + kCbTiles);               // query terms [3][128], W scales [2][128]
    float* redg = reinterpret_cast<float*>(sm + kCbPhi);               // gsum partials, in the features
    CbBars* bars = reinterpret_cast<CbBars*>(sm + kCbBars);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int row = tid & (kTile - 1), ch = tid >> 7;
    const int cta = blockIdx.x;
    const int g0 = cta * R.per, g1 = min(R.T, g0 + R.per);

    cb_init(bars);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    const uint32_t tl = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    const float a = s * kLog2e;
    CbPending pend;
    int w_h = -1;
    if (g0 < g1) {
        w_h = ((g1 - 1) / R.tph) % H;
        if (tid == 0) {
            cb_load_omega(&tm_w, sm, bars, w_h);
            pend.w = 0;
            for (int b = 0; b < 4; ++b) {
                cb_load_tile(b == CB_Q ? &tm_q : b == CB_K ? &tm_k : b == CB_V ? &tm_v : &tm_do, sm, b, bars, g1 - 1,
                             R.tph);
                pend.tile[b] = 0;
            }
        }
    }
    bool w_wait = g0 < g1;
    float trun[64];
    float tz = 0.f;
    bool ok = true;
    int cur_bh = -1;
    uint32_t nw = 0, nmma = 0;
    for (int g = g1 - 1, it = 0; g >= g0; --g, ++it) {
        const int bh = g / R.tph, tile = g - bh * R.tph, h = bh % H;
        const int tok0 = tile * kTile, tok = tok0 + row;
        const bool live = tok < L;
        const uint32_t tpar = (uint32_t)(it & 1);
        const bool more = g > g0;
        __syncthreads();   // the previous chunk is done with its buffers and tensor memory
        if (bh != cur_bh) {
            if (h != w_h) {
                if (tid == 0) {
                    cb_load_omega(&tm_w, sm, bars, h);
                    pend.w = (int)(nw & 1);
                }
                w_h = h;
                w_wait = true;
            }
            // the piece's suffix state, feature row tid
            const float* suf = suffix + ((size_t)bh * R.pstride + (cta - first_cta(R, bh))) * (kM * (kDV + 1)) +
                               (size_t)tid * (kDV + 1);
#pragma unroll
            for (int c = 0; c < 64; ++c) trun[c] = suf[c];
            tz = suf[kDV];
            cb_write_image(s_img, (uint32_t)tid, trun, 1.f);
            tv[tid] = tz;
            fence_async_smem();
            cur_bh = bh;
            if (w_wait) {
                ok = __syncthreads_and(mbar_wait(&bars->w, nw & 1, err, 70));
                ++nw;
                w_wait = false;
                if (!ok) break;
                pend.w = -1;
            }
        }
        // ---- the transposed query projection -> query features
        ok = __syncthreads_and(mbar_wait(&bars->tile[CB_Q], tpar, err, 71) &&
                               mbar_wait(&bars->tile[CB_K], tpar, err, 72));
        if (!ok) break;
        pend.tile[CB_Q] = pend.tile[CB_K] = -1;
        if (tid == 0) {
            tc_fence_after();
            cb_project(tmem + 256, s_w, s_q, 128);
            cb_project(tmem + 384, s_w + 128 * 128, s_q, 128);
            mma_commit(&bars->mma);
        }
        // query terms of token tok0 + tid (tid < 128): exponent offset (positive) or f16 scale
        // (ReLU) of the query pass, 2^eq / den, -go; zero for tokens past L and zero denominators
        float qoff = POS ? -INFINITY : 0.f, qmt = 0.f, qgo = 0.f;
        if (tid < kTile && tok0 + tid < L) {
            const float4 rs = rowstat[(size_t)bh * L + tok0 + tid];
            const int eq = (int)rs.w;
            qoff = POS ? -rs.y * kLog2e : s * exp2i(-eq);
            qmt = rs.x != 0.f ? exp2i(eq) / rs.x : 0.f;
            qgo = rs.z;
        }
        // this key row: exponent offset (or ReLU scale) and, for the epilogue, its half of k
        const float kc = live ? (POS ? -(0.5f * s * s * row_sqnorm(s_k, (uint32_t)row) + kshift[h]) * kLog2e : s)
                              : (POS ? -INFINITY : 0.f);
        uint4 krow[4];
#pragma unroll
        for (uint32_t c4 = 0; c4 < 4; ++c4)
            krow[c4] = POS ? ld_shared_v4(s_k + sw128((uint32_t)row, 4 * (uint32_t)ch + c4)) : make_uint4(0, 0, 0, 0);
        ok = __syncthreads_and(mbar_wait(&bars->mma, nmma & 1, err, 73));
        ++nmma;
        if (!ok) break;
        tc_fence_after();
        if (tid < kTile) {   // the Q tile is read: it holds the query terms until the next load
            qs[tid] = qoff;
            qs[kTile + tid] = qmt;
            qs[2 * kTile + tid] = -qgo;
        }
        __syncthreads();
        float tzc = 0.f;
#pragma unroll 1
        for (int u = 0; u < 2; ++u)
            tzc += cb_feature_row<KIND, true>(tl + 256 + 128 * ch + 64 * u, s_phi + (uint32_t)u * 2 * kPhiBlock,
                                              (uint32_t)tid, a, qs + 64 * u, qs + kTile + 64 * u, 1.f,
                                              qs + 2 * kTile + 64 * u);
        tmem_st_wait();
        fence_async_smem();
        tc_fence_before();
        ok = __syncthreads_and(mbar_wait(&bars->tile[CB_V], tpar, err, 78) &&
                               mbar_wait(&bars->tile[CB_O], tpar, err, 78));
        if (!ok) break;
        pend.tile[CB_V] = pend.tile[CB_O] = -1;
        // ---- dT = Phi~_Q^T dO (features hi + lo), C^T = V dO^T
        if (tid == 0) {
            tc_fence_after();
            cb_state_inc(tmem, tmem + 64, tmem + 256, tmem + 384, s_do);
            cb_project(tmem + 128, s_v, s_do, 128);
            mma_commit(&bars->mma);
        }
        ok = __syncthreads_and(mbar_wait(&bars->mma, nmma & 1, err, 74));
        ++nmma;
        if (!ok) break;
        tc_fence_after();
        {
            uint32_t d0[32], d1[32];
            tmem_ld32(tl + 64 * ch, d0);
            tmem_ld32(tl + 32 + 64 * ch, d1);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                trun[i] += __uint_as_float(d0[i]);
                trun[32 + i] += __uint_as_float(d1[i]);
            }
            tz += tzc;
        }
        // queries 64 ch .. +63 of key row `row`: W = tril(C^T - go) 2^eq / den, its row scale
        const uint32_t tcw = tl + 128 + 64 * ch;
        uint32_t x0[32], x1[32];
        tmem_ld32(tcw, x0);
        tmem_ld32(tcw + 32, x1);
        tmem_ld_wait();
        const int i0 = 64 * ch;
        {
            const float* ngo = qs + 2 * kTile + i0;
            const float* mt = qs + kTile + i0;
            float bm = 0.f;
#pragma unroll
            for (int k = 0; k < 32; ++k) {
                const float w0 = i0 + k >= row ? (__uint_as_float(x0[k]) + ngo[k]) * mt[k] : 0.f;
                const float w1 = i0 + 32 + k >= row ? (__uint_as_float(x1[k]) + ngo[32 + k]) * mt[32 + k] : 0.f;
                x0[k] = __float_as_uint(w0);
                x1[k] = __float_as_uint(w1);
                bm = fmaxf(bm, fmaxf(fabsf(w0), fabsf(w1)));
            }
            qs[3 * kTile + ch * kTile + row] = bm;
        }
        __syncthreads();
        const int ew = f16_scale_exp(fmaxf(qs[3 * kTile + row], qs[4 * kTile + row]));
        {
            const float ws = exp2i(-ew);
            uint32_t w0[16], w1[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                w0[i] = pack_f16(__uint_as_float(x0[2 * i]) * ws, __uint_as_float(x0[2 * i + 1]) * ws);
                w1[i] = pack_f16(__uint_as_float(x1[2 * i]) * ws, __uint_as_float(x1[2 * i + 1]) * ws);
            }
            tmem_st16(tcw, w0);
            tmem_st16(tcw + 16, w1);
            // this key row's v (columns 32 ch .. +31) times 2^-ew in place
#pragma unroll
            for (uint32_t c4 = 0; c4 < 4; ++c4) {
                const uint32_t addr = s_v + sw128((uint32_t)row, 4 * (uint32_t)ch + c4);
                const uint4 x = ld_shared_v4(addr);
                const uint32_t xin[4] = {x.x, x.y, x.z, x.w};
                uint32_t y[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) y[i] = pack_bf16(bf16lo(xin[i]) * ws, bf16hi(xin[i]) * ws);
                st_shared_v4(addr, y[0], y[1], y[2], y[3]);
            }
            fence_async_smem();
            tmem_st_wait();
        }
        tc_fence_before();
        __syncthreads();
        // ---- U = V' T~^T + W' Phi~_Q (= 2^-ew_j U), the key projection
        if (tid == 0) {
            tc_fence_after();
            if (more) {   // the query terms are read
                cb_load_tile(&tm_q, sm, CB_Q, bars, g - 1, R.tph);
                pend.tile[CB_Q] = (int)(tpar ^ 1);
            }
            cb_state_mult(tmem + 256, s_v, s_img);
            cb_weighted_features(tmem + 256, tmem + 128, tmem + 192, s_phi);
            issue_projection(tmem, s_k, s_w, 256);
            mma_commit(&bars->mma);
        }
        ok = __syncthreads_and(mbar_wait(&bars->mma, nmma & 1, err, 75));
        ++nmma;
        if (!ok) break;
        if (tid == 0 && more) {
            cb_load_tile(&tm_k, sm, CB_K, bars, g - 1, R.tph);
            cb_load_tile(&tm_v, sm, CB_V, bars, g - 1, R.tph);
            cb_load_tile(&tm_do, sm, CB_O, bars, g - 1, R.tph);
            pend.tile[CB_K] = pend.tile[CB_V] = pend.tile[CB_O] = (int)(tpar ^ 1);
        }
        tc_fence_after();
        float gsum = 0.f;
        {
            const float us = exp2i(ew);
#pragma unroll 1
            for (int cc = 0; cc < 4; ++cc) {
                uint32_t pw[32], uw[32];
                tmem_ld32(tl + 128 * ch + 32 * cc, pw);
                tmem_ld32(tl + 256 + 128 * ch + 32 * cc, uw);
                tmem_ld_wait();
                uint32_t hw[16], lw[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    float gg[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int k = 2 * i + e;
                        const float pv = __uint_as_float(pw[k]);
                        const float dphi = fmaf(__uint_as_float(uw[k]), us, tv[128 * ch + 32 * cc + k]);
                        const float gv = POS ? dphi * ex2(fmaf(pv, a, kc)) : (pv * kc > 0.f ? dphi : 0.f);
                        gg[e] = gv;
                        gsum += gv;
                    }
                    split_pack(gg[0], gg[1], hw[i], lw[i]);
                }
                tmem_st16(tl + 256 + 128 * ch + 16 * cc, hw);
                tmem_st16(tl + 128 * ch + 16 * cc, lw);
            }
        }
        tmem_st_wait();
        cb_write_image(s_img, (uint32_t)tid, trun, 1.f);   // the previous chunk's suffix
        fence_async_smem();
        redg[ch * kTile + row] = gsum;
        tc_fence_before();
        __syncthreads();
        // ---- dk = G omega
        if (tid == 0) {
            tc_fence_after();
            cb_grad_omega(tmem + 64, tmem + 256, tmem + 384, tmem, tmem + 128, s_w);
            mma_commit(&bars->mma);
        }
        tv[tid] = tz;   // t of the previous chunk's suffix (the current one is read)
        ok = __syncthreads_and(mbar_wait(&bars->mma, nmma & 1, err, 77));
        ++nmma;
        if (!ok) break;
        tc_fence_after();
        gsum = redg[row] + redg[kTile + row];
        cb_store_grad<KIND>(live ? dk + ((size_t)bh * L + tok) * kD : nullptr, tl + 64 + 32 * ch, ch, s, gsum, krow);
        tc_fence_before();
    }
    if (!ok && tid == 0) pend.drain(bars, err, 79);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

// Key pass for dv (bf16 operands: dv subtracts nothing), persistent over the call's tile ranges in
// reverse (grid R.G, 256 threads), the same thread roles.  Tensor memory per chunk (columns):
//   P_K [0,256), P_Q^T halves [256,384) [384,512) -> packed Phi_K over [0,64) [128,192), scaled
//       query features hi + lo in place (and bf16 in shared memory)
//   dT halves [64,128) [192,256), A^T = Phi_K Phi~_Q^T [256,384) -> tril over [256,288) [320,352)
//   dv [64,128)
template <int KIND>
__global__ void __launch_bounds__(kBwdThreads, 1)
k_tc_cbwd_v(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
            const __grid_constant__ CUtensorMap tm_do, const __grid_constant__ CUtensorMap tm_w,
            const float* __restrict__ suffix, const float* __restrict__ kshift, const float4* __restrict__ rowstat,
            __nv_bfloat16* __restrict__ dvv, int H, int L, float s, Ranges R, int* err) {
    constexpr bool POS = KIND == FAVOR_KERNEL_SOFTMAX_POS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1k(smem_raw);
    const uint32_t s_w = smem_u32(sm);
    const uint32_t s_img = s_w + kCbImgOff;
    const uint32_t s_q = s_w + kCbTiles, s_k = s_q + kTileBytes, s_do = s_k + 2 * kTileBytes;
    const uint32_t s_phi = s_w + kCbPhi;
    float* qs = reinterpret_cast<float*>(sm + kCbTiles);               // query terms [128], in the Q tile
    CbBars* bars = reinterpret_cast<CbBars*>(sm + kCbBars);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int row = tid & (kTile - 1), ch = tid >> 7;
    const int cta = blockIdx.x;
    const int g0 = cta * R.per, g1 = min(R.T, g0 + R.per);

    cb_init(bars);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    const uint32_t tl = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    const float a = s * kLog2e;
    CbPending pend;
    int w_h = -1;
    if (g0 < g1) {
        w_h = ((g1 - 1) / R.tph) % H;
        if (tid == 0) {
            cb_load_omega(&tm_w, sm, bars, w_h);
            pend.w = 0;
            cb_load_tile(&tm_q, sm, CB_Q, bars, g1 - 1, R.tph);
            cb_load_tile(&tm_k, sm, CB_K, bars, g1 - 1, R.tph);
            cb_load_tile(&tm_do, sm, CB_O, bars, g1 - 1, R.tph);
            pend.tile[CB_Q] = pend.tile[CB_K] = pend.tile[CB_O] = 0;
        }
    }
    bool w_wait = g0 < g1;
    float trun[64];
    bool ok = true;
    int cur_bh = -1;
    uint32_t nw = 0, nmma = 0;
    for (int g = g1 - 1, it = 0; g >= g0; --g, ++it) {
        const int bh = g / R.tph, tile = g - bh * R.tph, h = bh % H;
        const int tok0 = tile * kTile, tok = tok0 + row;
        const bool live = tok < L;
        const uint32_t tpar = (uint32_t)(it & 1);
        const bool more = g > g0;
        __syncthreads();   // the previous chunk is done with its buffers and tensor memory
        if (bh != cur_bh) {
            if (h != w_h) {
                if (tid == 0) {
                    cb_load_omega(&tm_w, sm, bars, h);
                    pend.w = (int)(nw & 1);
                }
                w_h = h;
                w_wait = true;
            }
            const float* suf = suffix + ((size_t)bh * R.pstride + (cta - first_cta(R, bh))) * (kM * (kDV + 1)) +
                               (size_t)tid * (kDV + 1);
#pragma unroll
            for (int c = 0; c < 64; ++c) trun[c] = suf[c];
            cb_write_image(s_img, (uint32_t)tid, trun, 1.f);
            fence_async_smem();
            cur_bh = bh;
            if (w_wait) {
                ok = __syncthreads_and(mbar_wait(&bars->w, nw & 1, err, 80));
                ++nw;
                w_wait = false;
                if (!ok) break;
                pend.w = -1;
            }
        }
        // ---- key projection and the transposed query projection
        ok = __syncthreads_and(mbar_wait(&bars->tile[CB_Q], tpar, err, 81) &&
                               mbar_wait(&bars->tile[CB_K], tpar, err, 82));
        if (!ok) break;
        pend.tile[CB_Q] = pend.tile[CB_K] = -1;
        if (tid == 0) {
            tc_fence_after();
            issue_projection(tmem, s_k, s_w, 256);
            cb_project(tmem + 256, s_w, s_q, 128);
            cb_project(tmem + 384, s_w + 128 * 128, s_q, 128);
            mma_commit(&bars->mma);
        }
        // query term of token tok0 + tid (tid < 128): phi~ = phi / den directly, through the
        // exponent offset (positive) or the scale (ReLU); zero past L and for zero denominators
        float qoff = POS ? -INFINITY : 0.f;
        if (tid < kTile && tok0 + tid < L) {
            const float4 rs = rowstat[(size_t)bh * L + tok0 + tid];
            if (rs.x > 0.f) qoff = POS ? -rs.y * kLog2e - log2f(rs.x) : s / rs.x;
        }
        const float kc = live ? (POS ? -(0.5f * s * s * row_sqnorm(s_k, (uint32_t)row) + kshift[h]) * kLog2e : s)
                              : (POS ? -INFINITY : 0.f);
        ok = __syncthreads_and(mbar_wait(&bars->mma, nmma & 1, err, 83));
        ++nmma;
        if (!ok) break;
        tc_fence_after();
        if (tid < kTile) qs[tid] = qoff;   // the Q tile is read
        __syncthreads();
#pragma unroll 1
        for (int u = 0; u < 2; ++u)
            cb_feature_row<KIND, false>(tl + 256 + 128 * ch + 64 * u, s_phi + (uint32_t)u * 2 * kPhiBlock,
                                        (uint32_t)tid, a, qs + 64 * u, nullptr, 1.f, nullptr);
#pragma unroll 1
        for (int cc = 0; cc < 4; ++cc) {
            uint32_t pw[32];
            tmem_ld32(tl + 128 * ch + 32 * cc, pw);
            tmem_ld_wait();
            uint32_t fw[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float p0 = __uint_as_float(pw[2 * i]), p1 = __uint_as_float(pw[2 * i + 1]);
                fw[i] = POS ? pack_bf16(ex2(fmaf(p0, a, kc)), ex2(fmaf(p1, a, kc)))
                            : pack_bf16(fmaxf(p0 * kc, 0.f), fmaxf(p1 * kc, 0.f));
            }
            tmem_st16(tl + 128 * ch + 16 * cc, fw);
        }
        tmem_st_wait();
        fence_async_smem();
        tc_fence_before();
        ok = __syncthreads_and(mbar_wait(&bars->tile[CB_O], tpar, err, 84));
        if (!ok) break;
        pend.tile[CB_O] = -1;
        // ---- dT = Phi~_Q^T dO (features hi + lo), A^T = Phi_K Phi~_Q^T
        if (tid == 0) {
            tc_fence_after();
            if (more) {   // the query terms are read
                cb_load_tile(&tm_q, sm, CB_Q, bars, g - 1, R.tph);
                pend.tile[CB_Q] = (int)(tpar ^ 1);
            }
            cb_state_inc(tmem + 64, tmem + 192, tmem + 256, tmem + 384, s_do);
            cb_scores<false>(tmem + 256, tmem, tmem + 128, s_phi);
            mma_commit(&bars->mma);
        }
        ok = __syncthreads_and(mbar_wait(&bars->mma, nmma & 1, err, 85));
        ++nmma;
        if (!ok) break;
        tc_fence_after();
        {
            uint32_t d0[32], d1[32];
            tmem_ld32(tl + 64 + 128 * ch, d0);
            tmem_ld32(tl + 96 + 128 * ch, d1);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                trun[i] += __uint_as_float(d0[i]);
                trun[32 + i] += __uint_as_float(d1[i]);
            }
        }
        {
            // tril(A^T) for queries 64 ch .. +63 of key row `row`, packed in place
            const uint32_t ta = tl + 256 + 64 * ch;
            uint32_t x0[32], x1[32];
            tmem_ld32(ta, x0);
            tmem_ld32(ta + 32, x1);
            tmem_ld_wait();
            const int i0 = 64 * ch;
            uint32_t w0[16], w1[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                w0[i] = pack_bf16(i0 + 2 * i >= row ? __uint_as_float(x0[2 * i]) : 0.f,
                                  i0 + 2 * i + 1 >= row ? __uint_as_float(x0[2 * i + 1]) : 0.f);
                w1[i] = pack_bf16(i0 + 32 + 2 * i >= row ? __uint_as_float(x1[2 * i]) : 0.f,
                                  i0 + 33 + 2 * i >= row ? __uint_as_float(x1[2 * i + 1]) : 0.f);
            }
            tmem_st16(ta, w0);
            tmem_st16(ta + 16, w1);
            tmem_st_wait();
        }
        tc_fence_before();
        __syncthreads();
        // ---- dv = Phi_K T~ + tril(A^T) dO
        if (tid == 0) {
            tc_fence_after();
            const uint32_t id_o = make_idesc(128, 64, 0, 1);
            const uint64_t bth = make_desc(s_img, 8192, 1024, SW_128B), btl = make_desc(s_img + kSBytes, 8192, 1024, SW_128B);
            const uint64_t bdo = make_desc(s_do, 8192, 1024, SW_128B);
#pragma unroll
            for (int kk = 0; kk < 16; ++kk)
                mma_ts(tmem + 64, kk < 8 ? tmem + 8 * kk : tmem + 128 + 8 * (kk - 8), bth + 128 * kk, id_o, kk > 0 ? 1u : 0u);
#pragma unroll
            for (int kk = 0; kk < 16; ++kk)
                mma_ts(tmem + 64, kk < 8 ? tmem + 8 * kk : tmem + 128 + 8 * (kk - 8), btl + 128 * kk, id_o, 1u);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                mma_ts(tmem + 64, tmem + 256 + 64 * (kk >> 2) + 8 * (kk & 3), bdo + 128 * kk, id_o, 1u);
            mma_commit(&bars->mma);
        }
        ok = __syncthreads_and(mbar_wait(&bars->mma, nmma & 1, err, 86));
        ++nmma;
        if (!ok) break;
        if (tid == 0 && more) {
            cb_load_tile(&tm_k, sm, CB_K, bars, g - 1, R.tph);
            cb_load_tile(&tm_do, sm, CB_O, bars, g - 1, R.tph);
            pend.tile[CB_K] = pend.tile[CB_O] = (int)(tpar ^ 1);
        }
        tc_fence_after();
        {
            uint32_t v0[32];
            tmem_ld32(tl + 64 + 32 * ch, v0);
            tmem_ld_wait();
            if (live) {
                uint4* dst = reinterpret_cast<uint4*>(dvv + ((size_t)bh * L + tok) * kDV);
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) {
                    uint32_t wv[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        wv[i] = pack_bf16(__uint_as_float(v0[8 * c4 + 2 * i]), __uint_as_float(v0[8 * c4 + 2 * i + 1]));
                    dst[4 * ch + c4] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
                }
            }
        }
        cb_write_image(s_img, (uint32_t)tid, trun, 1.f);   // the previous chunk's suffix
        fence_async_smem();
        tc_fence_before();
    }
    if (!ok && tid == 0) pend.drain(bars, err, 89);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

// In place, per head: piece p <- the sum of the pieces before it (REV false) or after it (REV
// true), fixed order.  grid (m (dv+1) / 256 up, B*H).
template <bool REV>
__global__ void k_piece_scan(float* __restrict__ part, Ranges R) {
    constexpr int n = kM * (kDV + 1);
    const int bh = blockIdx.y;
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const int np = last_cta(R, bh) - first_cta(R, bh) + 1;
    float* p = part + (size_t)bh * R.pstride * n + i;
    float run = 0.f;
    for (int k = 0; k < np; ++k) {
        const int q = REV ? np - 1 - k : k;
        const float t = p[(size_t)q * n];
        p[(size_t)q * n] = run;
        run += t;
    }
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

constexpr size_t kSmemCb = 1024 + kCbBars + sizeof(CbBars);
static_assert(kSmemCb <= 232448, "causal backward shared memory");
static_assert(3 * kTile * 4 <= kTileBytes && 6 * kTile * 4 <= kTileBytes, "row partials fit a tile buffer");

void allow_cbwd_once() {
    static std::once_flag once;
    std::call_once(once, [] {
        allow_smem(k_tc_cbwd_q<FAVOR_KERNEL_SOFTMAX_POS>, kSmemCb);
        allow_smem(k_tc_cbwd_q<FAVOR_KERNEL_RELU>, kSmemCb);
        allow_smem(k_tc_cbwd_k<FAVOR_KERNEL_SOFTMAX_POS>, kSmemCb);
        allow_smem(k_tc_cbwd_k<FAVOR_KERNEL_RELU>, kSmemCb);
        allow_smem(k_tc_cbwd_v<FAVOR_KERNEL_SOFTMAX_POS>, kSmemCb);
        allow_smem(k_tc_cbwd_v<FAVOR_KERNEL_RELU>, kSmemCb);
        cudaGetLastError();
    });
}

template <int KIND>
favor_status tc_causal_backward_t(const Handle& h, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                                  const CUtensorMap& mdo, const CUtensorMap& mw, void* dq, void* dk, void* dv, int BH,
                                  int L, const Ranges& R, cudaStream_t st) {
    float4* rowstat = reinterpret_cast<float4*>(h.ws_rowstat);
    const dim3 sgrid((kM * (kDV + 1) + 255) / 256, BH);
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
        k_piece_scan<false><<<sgrid, 256, 0, st>>>(h.ws_partial, R);
        count_launch();
        if ((e = check_launch("backward prefix scan kernel")) != FAVOR_OK) return e;
    }
    {
        ProfScope ps(h, PROF_BWD_QUERY, st);
        k_tc_cbwd_q<KIND><<<R.G, kBwdThreads, kSmemCb, st>>>(mq, mk, mv, mdo, mw, h.ws_partial, h.kshift,
                                                               (__nv_bfloat16*)dq, rowstat, h.H, L, h.s, R, h.dev_err);
        count_launch();
        if ((e = check_launch("causal backward query kernel")) != FAVOR_OK) return e;
        k_tc_bstate<KIND, 1><<<R.G, kBStateThreads, kSmemBState, st>>>(mq, mdo, mw, h.kshift, rowstat, h.ws_partial,
                                                                         h.H, L, h.s, R, h.dev_err);
        count_launch();
        if ((e = check_launch("backward query-state kernel")) != FAVOR_OK) return e;
    }
    {
        ProfScope ps(h, PROF_COMBINE, st);
        k_piece_scan<true><<<sgrid, 256, 0, st>>>(h.ws_partial, R);
        count_launch();
        if ((e = check_launch("backward suffix scan kernel")) != FAVOR_OK) return e;
    }
    ProfScope ps(h, PROF_BWD_KEY, st);
    k_tc_cbwd_k<KIND><<<R.G, kBwdThreads, kSmemCb, st>>>(mq, mk, mv, mdo, mw, h.ws_partial, h.kshift, rowstat,
                                                           (__nv_bfloat16*)dk, h.H, L, h.s, R, h.dev_err);
    count_launch();
    if ((e = check_launch("causal backward key kernel")) != FAVOR_OK) return e;
    k_tc_cbwd_v<KIND><<<R.G, kBwdThreads, kSmemCb, st>>>(mq, mk, mdo, mw, h.ws_partial, h.kshift, rowstat,
                                                           (__nv_bfloat16*)dv, h.H, L, h.s, R, h.dev_err);
    count_launch();
    return check_launch("causal backward value kernel");
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

favor_status tc_causal_backward(const Handle& h, const void* q, const void* k, const void* v, const void* dout,
                                void* dq, void* dk, void* dv, int B, int L, cudaStream_t st) {
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dout) || !aligned16(dq) || !aligned16(dk) ||
        !aligned16(dv))
        return simt_causal_backward(h, q, k, v, dout, dq, dk, dv, B, L, st);
    allow_bwd_once();
    allow_cbwd_once();
    const int BH = B * h.H;
    const Ranges R = plan_ranges(BH, L, h.num_sms);
    if ((size_t)BH * R.pstride > h.ws_partial_rows)
        return set_error(FAVOR_ERR_INVALID_ARG, "backward workspace too small (%d x %d rows)", BH, R.pstride);
    CUtensorMap mq, mk, mv, mdo, mw;
    if (!map_tokens(&mq, q, BH, L) || !map_tokens(&mk, k, BH, L) || !map_tokens(&mv, v, BH, L) ||
        !map_tokens(&mdo, dout, BH, L) || !map_omega(&mw, h.omega_bf16, h.H))
        return set_error(FAVOR_ERR_CUDA, "cuTensorMapEncodeTiled failed");
    if (h.kind == FAVOR_KERNEL_SOFTMAX_POS)
        return tc_causal_backward_t<FAVOR_KERNEL_SOFTMAX_POS>(h, mq, mk, mv, mdo, mw, dq, dk, dv, BH, L, R, st);
    return tc_causal_backward_t<FAVOR_KERNEL_RELU>(h, mq, mk, mv, mdo, mw, dq, dk, dv, BH, L, R, st);
}

}  // namespace favor
