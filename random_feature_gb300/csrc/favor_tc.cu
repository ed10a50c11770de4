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
//   state kernel : [0,256) projection halves P0, P1 | [256,416) [S | z] halves (2 x 80 columns)
//   readout      : two 256-column tile slots: projection, then Phi_Q packed in [0,64) and
//                  [192,256), [num | den] in [64,144)
//   causal       : three rotating 128-column slots (query projection halves -> packed Phi_Q and
//                  num; key projection halves -> A -> packed tril(A)) | [384,512) S halves
#include <cmath>
#include <cstddef>
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>

#include "favor_internal.h"
#include "tc_common.cuh"
#include "tc_ptx.cuh"

namespace favor {
namespace {

using namespace tc;

struct Bars {
    uint64_t tma;
    uint64_t mma;
    uint32_t tmem_base;
    uint32_t pad;
};

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

__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&r)[64]) {
    uint32_t (&lo)[32] = *reinterpret_cast<uint32_t(*)[32]>(&r[0]);
    uint32_t (&hi)[32] = *reinterpret_cast<uint32_t(*)[32]>(&r[32]);
    tmem_ld32(taddr, lo);
    tmem_ld32(taddr + 32, hi);
}

// ====================================================================== state
// Persistent, warp-specialised.  The key projection is computed transposed,
// D[feature r, token j] = omega_r . k_j + c_j / a, per half of 128 features
// (tensor-memory slots P0, P1: lane = feature, column = token), where the
// per-token exponent offset c_j = -(s^2 ||k_j||^2 / 2 + kappa) log2(e) enters
// through one extra K-step: [c_j/a as bf16 hi + lo] against a pair of ones.
// Feature warps then need only f = 2^(a * D): they read a slot once
// (releasing it at once for the next tile's projection), accumulate z_r in
// registers, and write the features packed (bf16) to Phi0 / Phi1, the A
// operand (tensor memory) of S_half += Phi^T_half V.  Trigonometric features
// (rows [omega; omega]): only P0 is projected (the rows repeat), and the two
// warps of a lane quarter split its tokens, each writing sin of s D into Phi0
// and cos into Phi1 from one range reduction, times the token's
// h(s k_j) = exp(s^2 ||k_j||^2 / 2), which the norm warp writes per stage.
//   tensor memory: P0 [0,128) P1 [128,256) Phi0 [256,320) Phi1 [320,384) S0 [384,448) S1 [448,512)
//   warp 0: TMA producer   warp 1: projection MMAs   warp 2: state MMAs
//   warp 3: key norms -> offsets (positive features) or h(s k_j) (trigonometric)
//   warps 4..11: features; lane quarter q = warp % 4, half h = (warp - 4) / 4
// The two MMA streams are independent (projections read omega and K, state
// updates read Phi and V) and a single issuing thread is the bottleneck, so each
// has its own thread; a K/V stage is released when both have committed.
constexpr int kNS = 5;                 // K/V pipeline stages
constexpr int kStateThreads = 384;
constexpr uint32_t kExtStage = kTile * 32;        // K-side extra K-step: [128 tokens][16] bf16, no swizzle
constexpr uint32_t kExtOmega = kM * 32;           // omega side: [256 features][16] bf16 = (1, 1, 0, ...)

// Row r of a no-swizzle K-major [rows][16] bf16 operand: core matrices of
// 8 rows x 16 B (SBO = 256 between row groups, LBO = 128 to elements 8..15).
__device__ __forceinline__ uint32_t ext_row(uint32_t r) { return (r >> 3) * 256u + (r & 7u) * 16u; }

struct StBars {
    uint64_t kv_full[kNS], kv_empty[kNS];
    uint64_t ext_full[kNS];
    uint64_t w_full, w_empty;
    uint64_t p_full[2], p_empty[2];
    uint64_t phi_full[2], phi_empty[2];
    uint64_t acc_full, acc_empty;
    uint64_t zx;   // trigonometric: the feature warps' z hand-over at a piece end
    uint32_t tmem_base;
};

template <int KIND, bool GATED = false>
__global__ void __launch_bounds__(kStateThreads, 1)
k_tc_state(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
           const __grid_constant__ CUtensorMap tm_w, const float* __restrict__ kshift, const float* __restrict__ wlog,
           float* __restrict__ part, int H, int L, float s, Ranges R, int* err) {
    constexpr bool POS = KIND == FAVOR_KERNEL_SOFTMAX_POS;
    constexpr bool TRIG = KIND == FAVOR_KERNEL_SOFTMAX_TRIG;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1k(smem_raw);
    const uint32_t s_w = smem_u32(sm);
    const uint32_t s_kv = s_w + kOmegaBytes;                 // stage i: K at +2i*16K, V at +(2i+1)*16K
    const uint32_t s_ext = s_kv + kNS * 2 * kTileBytes;      // stage i: K-side extra block at +i*4K
    const uint32_t s_wext = s_ext + kNS * kExtStage;         // omega-side extra block
    StBars* bars = reinterpret_cast<StBars*>(sm + (s_wext - s_w) + kExtOmega);
    const int c = blockIdx.x;
    const int g0 = c * R.per;
    const int g1 = min(R.T, g0 + R.per);
    const int n = g1 - g0;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const float a = s * kLog2e;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kNS; ++i) {
            mbar_init(&bars->kv_full[i], 1);
            mbar_init(&bars->kv_empty[i], 2);
            mbar_init(&bars->ext_full[i], 1);
        }
        mbar_init(&bars->w_full, 1);
        mbar_init(&bars->w_empty, 1);
        // trigonometric: all eight feature warps read P0 and write both Phi halves
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars->p_full[i], 1);
            mbar_init(&bars->p_empty[i], TRIG ? 8 : 4);
            mbar_init(&bars->phi_full[i], TRIG ? 8 : 4);
            mbar_init(&bars->phi_empty[i], 1);
        }
        mbar_init(&bars->acc_full, 1);
        mbar_init(&bars->acc_empty, 8);
        mbar_init(&bars->zx, 8);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&bars->tmem_base, 512);
        tmem_relinquish();
    }
    if (POS && warp >= 4) {
        // zero the K-side extra blocks; omega side = 1 in elements 0 and 1 of every row
        uint32_t* e = reinterpret_cast<uint32_t*>(sm + (s_ext - s_w));
        for (int i = threadIdx.x - 128; i < (int)(kNS * kExtStage / 4); i += kStateThreads - 128) e[i] = 0u;
        uint32_t* wx = reinterpret_cast<uint32_t*>(sm + (s_wext - s_w));
        for (int i = threadIdx.x - 128; i < (int)(kExtOmega / 4); i += kStateThreads - 128)
            wx[i] = ((i & 63) < 32 && (i & 3) == 0) ? 0x3F803F80u : 0u;   // word 0 of core 0 of each row
        fence_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int cur_h = -1;
            uint32_t wph = 0;
            for (int i = 0; i < n; ++i) {
                const int g = g0 + i, bh = g / R.tph, h = bh % H, tok0 = (g % R.tph) * kTile;
                const int st = i % kNS;
                if (i >= kNS && !mbar_wait(&bars->kv_empty[st], ((i / kNS) - 1) & 1, err, 101)) break;
                if (h != cur_h) {
                    if (cur_h >= 0) {
                        if (!mbar_wait(&bars->w_empty, wph, err, 102)) break;
                        wph ^= 1;
                    }
                    mbar_expect_tx(&bars->w_full, kOmegaBytes);
                    tma_load_2d(sm, &tm_w, &bars->w_full, 0, h * kM);
                    cur_h = h;
                }
                mbar_expect_tx(&bars->kv_full[st], 2 * kTileBytes);
                tma_load_3d(sm + (s_kv - s_w) + 2 * st * kTileBytes, &tm_k, &bars->kv_full[st], 0, tok0, bh);
                tma_load_3d(sm + (s_kv - s_w) + (2 * st + 1) * kTileBytes, &tm_v, &bars->kv_full[st], 0, tok0, bh);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------ projection MMAs
        // P_h (features 128h.., tokens) = omega rows x K tile (+ offsets for positive features)
        if (lane == 0 && n > 0) {
            const uint32_t id_p = make_idesc(128, 128, 0, 0);
            uint32_t wph = 0;
            int tih = g0 % R.tph;               // tile index within the current head
            const bool multi_head = H > 1;      // a new bh means new omega only when H > 1
            int st = 0;
            for (int i = 0; i < n; ++i) {
                if (i == 0 || (tih == 0 && multi_head)) {
                    if (!mbar_wait(&bars->w_full, wph, err, 111)) break;
                    wph ^= 1;
                }
                if (!mbar_wait(&bars->kv_full[st], (i / kNS) & 1, err, 112)) break;
                if (POS && !mbar_wait(&bars->ext_full[st], (i / kNS) & 1, err, 113)) break;
                bool ok = true;
                for (int hp = 0; hp < (TRIG ? 1 : 2); ++hp) {   // trigonometric: rows 128.. repeat 0..127
                    if (i > 0 && !mbar_wait(&bars->p_empty[hp], (i - 1) & 1, err, 114 + hp)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t a0 = make_desc(s_w + hp * 128 * 128, 16, 1024, SW_128B);
                    const uint64_t b0 = make_desc(s_kv + 2 * st * kTileBytes, 16, 1024, SW_128B);
                    const uint32_t d = tmem + 128 * hp;
                    mma_ss(d, a0, b0, id_p, 0u);
                    mma_ss(d, a0 + 2, b0 + 2, id_p, 1u);
                    mma_ss(d, a0 + 4, b0 + 4, id_p, 1u);
                    mma_ss(d, a0 + 6, b0 + 6, id_p, 1u);
                    if (POS)
                        mma_ss(d, make_desc(s_wext + hp * 128 * 32, 128, 256, SW_NONE),
                               make_desc(s_ext + st * kExtStage, 128, 256, SW_NONE), id_p, 1u);
                    mma_commit(&bars->p_full[hp]);
                }
                if (!ok) break;
                mma_commit(&bars->kv_empty[st]);                       // K side of the stage is read
                if (i + 1 < n && tih == R.tph - 1 && multi_head) mma_commit(&bars->w_empty);
                tih = (tih + 1 == R.tph) ? 0 : tih + 1;
                st = (st + 1 == kNS) ? 0 : st + 1;
            }
        }
    } else if (warp == 2) {
        // ----------------------------------------------------------- state MMAs
        // S_h += Phi^T_h (tensor memory, packed bf16) x V tile (smem, MN-major)
        if (lane == 0 && n > 0) {
            const uint32_t id_s = make_idesc(128, 64, 0, 1);
            int piece = 0;
            int tih = g0 % R.tph;
            int st = 0;
            bool ok = true;
            for (int i = 0; i < n && ok; ++i) {
                const bool first = (i == 0) || tih == 0;
                const bool last = (i == n - 1) || tih == R.tph - 1;
                if (first && i > 0) {
                    ok = mbar_wait(&bars->acc_empty, (piece - 1) & 1, err, 117);
                    if (!ok) break;
                }
                for (int hp = 0; hp < 2 && ok; ++hp) {
                    ok = mbar_wait(&bars->phi_full[hp], i & 1, err, 118 + hp);
                    if (!ok) break;
                    tc_fence_after();
                    const uint64_t b0 = make_desc(s_kv + (2 * st + 1) * kTileBytes, 8192, 1024, SW_128B);
                    const uint32_t d = tmem + 384 + 64 * hp;
                    const uint32_t ap = tmem + 256 + 64 * hp;
                    mma_ts(d, ap, b0, id_s, first ? 0u : 1u);
#pragma unroll
                    for (int kk = 1; kk < 8; ++kk) mma_ts(d, ap + 8 * kk, b0 + 128 * kk, id_s, 1u);
                    mma_commit(&bars->phi_empty[hp]);
                }
                if (!ok) break;
                mma_commit(&bars->kv_empty[st]);                       // V side of the stage is read
                if (last) {
                    mma_commit(&bars->acc_full);
                    ++piece;
                }
                tih = (tih + 1 == R.tph) ? 0 : tih + 1;
                st = (st + 1 == kNS) ? 0 : st + 1;
            }
        }
    } else if (warp == 3) {
        // ---------------------------------------------------------- key norms
        // Per token, positive features: x = c_j / a with c_j = -(s^2 ||k_j||^2 / 2 +
        // kappa_h) log2(e) (a huge negative value past L), written as bf16 hi + lo
        // into the stage's K-side extra block; trigonometric features: the factor
        // h(s k_j) as fp32 in the same block, for the feature warps.  Four tokens per lane.
        if (POS || TRIG || GATED) {
            int kap_h = -1;
            float kap = 0.f;
            const float inv_s = 1.f / s, inv_a = 1.f / a;
            for (int i = 0; i < n; ++i) {
                const int g = g0 + i, bh = g / R.tph, h = bh % H, tok0 = (g % R.tph) * kTile;
                const int st = i % kNS;
                if (h != kap_h) {
                    kap = __ldg(kshift + h);
                    kap_h = h;
                }
                if (!mbar_wait(&bars->kv_full[st], (i / kNS) & 1, err, 131)) break;
                float nrm[4] = {0.f, 0.f, 0.f, 0.f};
                if (POS || TRIG) {
                    row_sqnorm2(s_kv + 2 * st * kTileBytes, (uint32_t)lane, (uint32_t)(lane + 32), nrm[0], nrm[1]);
                    row_sqnorm2(s_kv + 2 * st * kTileBytes, (uint32_t)(lane + 64), (uint32_t)(lane + 96), nrm[2], nrm[3]);
                }
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const uint32_t j = (uint32_t)(lane + 32 * t);
                    // gated calls: the key's log2 weight toward its piece's end
                    const float wl = (GATED && tok0 + (int)j < L) ? __ldg(wlog + (size_t)bh * L + tok0 + j) : 0.f;
                    if (GATED && !POS) {
                        // ReLU: the weight itself, a column factor for the feature warps
                        const float wk = (tok0 + (int)j < L && wl > -1.0e29f) ? exp2f(wl) : 0.f;
                        reinterpret_cast<float*>(sm + (s_ext - s_w) + st * kExtStage)[j] = wk;
                    } else if (TRIG) {
                        // h(s k_j) = exp(s^2 ||k_j||^2 / 2), 0 past L, one fp32 per token
                        const float hk = (tok0 + (int)j < L) ? expf(0.5f * s * s * nrm[t]) : 0.f;
                        reinterpret_cast<float*>(sm + (s_ext - s_w) + st * kExtStage)[j] = hk;
                    } else {
                        // positive: the weight enters the exponent offset (x in projection units, f = 2^(a D))
                        const float x = (tok0 + (int)j < L && wl > -1.0e29f)
                                            ? -(0.5f * s * nrm[t] + kap * inv_s) + wl * inv_a
                                            : -1.0e30f;
                        const float hi = __bfloat162float(__float2bfloat16_rn(x));
                        const float lo = x - hi;
                        st_shared_v4(s_ext + st * kExtStage + ext_row(j), pack_bf16(hi, lo), 0u, 0u, 0u);
                    }
                }
                fence_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->ext_full[st]);
            }
        }
    } else {
        // ------------------------------------------------------------ features
        const int q = warp & 3;
        const int hp = (warp - 4) >> 2;
        const uint32_t lane_off = (uint32_t)(32 * q) << 16;
        const uint32_t tp = tmem + lane_off + 128 * hp;           // projection slot
        const uint32_t tf = tmem + lane_off + 256 + 64 * hp;      // packed features
        int piece = 0;
        float z0 = 0.f, z1 = 0.f, zc0 = 0.f, zc1 = 0.f;   // zc: cos sums (trigonometric)
        for (int i = 0; i < n; ++i) {
            const int g = g0 + i, bh = g / R.tph;
            const bool last = (i == n - 1) || ((g + 1) / R.tph) != bh;
            if (TRIG) {
                // P0 holds the 128 distinct projections; warp (q, h) takes tokens [64h, 64h+64)
                // and writes sin into Phi0 and cos into Phi1 (one range reduction per pair),
                // times the token's h(s k_j)
                if (!mbar_wait(&bars->p_full[0], i & 1, err, 121)) break;
                tc_fence_after();
                uint32_t p[64];
                tmem_ld64(tmem + lane_off + 64 * hp, p);
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->p_empty[0]);
                const int st = i % kNS;
                if (!mbar_wait(&bars->ext_full[st], (i / kNS) & 1, err, 122)) break;
                const float4* hk = reinterpret_cast<const float4*>(sm + (s_ext - s_w) + st * kExtStage) + 16 * hp;
                uint32_t ws[32], wc[32];
#pragma unroll
                for (int k4 = 0; k4 < 16; ++k4) {
                    const float4 h4 = hk[k4];
                    const float hh[4] = {h4.x, h4.y, h4.z, h4.w};
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int k2 = 2 * k4 + e;
                        float s0, c0, s1, c1;
                        sincos_pair(s * __uint_as_float(p[2 * k2]), s0, c0);
                        sincos_pair(s * __uint_as_float(p[2 * k2 + 1]), s1, c1);
                        s0 *= hh[2 * e];
                        c0 *= hh[2 * e];
                        s1 *= hh[2 * e + 1];
                        c1 *= hh[2 * e + 1];
                        z0 += s0;
                        z1 += s1;
                        zc0 += c0;
                        zc1 += c1;
                        ws[k2] = pack_bf16(s0, s1);
                        wc[k2] = pack_bf16(c0, c1);
                    }
                }
                if (i > 0 && !(mbar_wait(&bars->phi_empty[0], (i - 1) & 1, err, 123) &&
                               mbar_wait(&bars->phi_empty[1], (i - 1) & 1, err, 123)))
                    break;
                tc_fence_after();
                const uint32_t t0 = tmem + lane_off + 256 + 32 * hp, t1 = t0 + 64;
                tmem_st16(t0, *reinterpret_cast<uint32_t(*)[16]>(&ws[0]));
                tmem_st16(t0 + 16, *reinterpret_cast<uint32_t(*)[16]>(&ws[16]));
                tmem_st16(t1, *reinterpret_cast<uint32_t(*)[16]>(&wc[0]));
                tmem_st16(t1 + 16, *reinterpret_cast<uint32_t(*)[16]>(&wc[16]));
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&bars->phi_full[0]);
                    mbar_arrive(&bars->phi_full[1]);
                }
                if (last) {
                    if (!mbar_wait(&bars->acc_full, piece & 1, err, 124)) break;
                    tc_fence_after();
                    uint32_t sv[64];
                    tmem_ld64(tmem + lane_off + 384 + 64 * hp, sv);
                    tmem_ld_wait();
                    // z of this warp's feature row (sin row r for h = 0, cos row 128 + r for
                    // h = 1): its own token half plus the partner warp's, handed over in the
                    // omega-side extra block (unused by this kind)
                    float* zx = reinterpret_cast<float*>(sm + (s_wext - s_w));
                    const uint32_t r = 32 * q + lane;
                    if (hp == 0) zx[128 + r] = zc0 + zc1;
                    else zx[r] = z0 + z1;
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars->zx);   // release: the warp's writes above
                    if (!mbar_wait(&bars->zx, piece & 1, err, 125)) break;
                    const float zt = hp == 0 ? (z0 + z1) + zx[r] : (zc0 + zc1) + zx[128 + r];
                    const int pc = c - first_cta(R, bh);
                    float* o = part + ((size_t)bh * R.pstride + pc) * (kM * (kDV + 1)) + (128 * hp + r);
#pragma unroll
                    for (int k2 = 0; k2 < 64; ++k2) o[(size_t)k2 * kM] = __uint_as_float(sv[k2]);
                    o[(size_t)64 * kM] = zt;
                    z0 = z1 = zc0 = zc1 = 0.f;
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars->acc_empty);
                    ++piece;
                }
                continue;
            }
            if (!mbar_wait(&bars->p_full[hp], i & 1, err, 121)) break;
            tc_fence_after();
            uint32_t p[128];
            {
                uint32_t (&p0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&p[0]);
                uint32_t (&p1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&p[32]);
                uint32_t (&p2)[32] = *reinterpret_cast<uint32_t(*)[32]>(&p[64]);
                uint32_t (&p3)[32] = *reinterpret_cast<uint32_t(*)[32]>(&p[96]);
                tmem_ld32(tp, p0);
                tmem_ld32(tp + 32, p1);
                tmem_ld32(tp + 64, p2);
                tmem_ld32(tp + 96, p3);
            }
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->p_empty[hp]);
            // features into registers first: the exps overlap the previous tile's
            // state MMAs, which still read this warp's Phi region
            uint32_t w[64];
            if (GATED && !POS) {
                // ReLU, gated: max(p, 0) times the key's weight toward its piece's end
                const int st = i % kNS;
                if (!mbar_wait(&bars->ext_full[st], (i / kNS) & 1, err, 122)) break;
                const float4* wk = reinterpret_cast<const float4*>(sm + (s_ext - s_w) + st * kExtStage);
#pragma unroll
                for (int k4 = 0; k4 < 32; ++k4) {
                    const float4 w4 = wk[k4];
                    const float ww[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int k2 = 2 * k4 + e;
                        const float f0 = fmaxf(__uint_as_float(p[2 * k2]), 0.f) * ww[2 * e];
                        const float f1 = fmaxf(__uint_as_float(p[2 * k2 + 1]), 0.f) * ww[2 * e + 1];
                        z0 += f0;
                        z1 += f1;
                        w[k2] = pack_bf16(f0, f1);
                    }
                }
            } else {
#pragma unroll
                for (int k2 = 0; k2 < 64; ++k2) {
                    const float x0 = __uint_as_float(p[2 * k2]), x1 = __uint_as_float(p[2 * k2 + 1]);
                    float f0, f1;
                    if (POS) {
                        f0 = ex2(x0 * a);
                        f1 = ex2(x1 * a);
                    } else {
                        // ReLU: rows past L are zero (TMA fill), so their projection is 0
                        f0 = fmaxf(x0, 0.f);
                        f1 = fmaxf(x1, 0.f);
                    }
                    z0 += f0;
                    z1 += f1;
                    w[k2] = pack_bf16(f0, f1);
                }
            }
            if (i > 0 && !mbar_wait(&bars->phi_empty[hp], (i - 1) & 1, err, 123)) break;
            tc_fence_after();
#pragma unroll
            for (int cc = 0; cc < 4; ++cc)
                tmem_st16(tf + 16 * cc, *reinterpret_cast<uint32_t(*)[16]>(&w[16 * cc]));
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->phi_full[hp]);
            if (last) {
                if (!mbar_wait(&bars->acc_full, piece & 1, err, 124)) break;
                tc_fence_after();
                uint32_t sv[64];
                tmem_ld64(tmem + lane_off + 384 + 64 * hp, sv);
                tmem_ld_wait();
                const int pc = c - first_cta(R, bh);
                // piece state stored column-major, [65][256]: a warp's 32 features are
                // 128 contiguous bytes for every column
                float* o = part + ((size_t)bh * R.pstride + pc) * (kM * (kDV + 1)) + (128 * hp + 32 * q + lane);
#pragma unroll
                for (int k2 = 0; k2 < 64; ++k2) o[(size_t)k2 * kM] = __uint_as_float(sv[k2]);
                o[(size_t)64 * kM] = z0 + z1;
                z0 = z1 = 0.f;
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->acc_empty);
                ++piece;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, 512);
}

// ================================================ reduce + pack (bidirectional)
// grid (ceil(256*65/256), B*H).  Sum a head's pieces in order and write the
// bf16 operand image of the readout: S~ as a [256][64] SW128 block, then a
// second [256][64] SW128 block with z~ in column 0 (its other columns stay at
// the zeros the workspace was created with).
__global__ void k_reduce_pack(const float* __restrict__ part, uint8_t* __restrict__ image, Ranges R) {
    const int bh = blockIdx.y;
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    constexpr int n = kM * (kDV + 1);
    if (i >= n) return;
    const int np = last_cta(R, bh) - first_cta(R, bh) + 1;
    const float* p = part + (size_t)bh * R.pstride * n + i;
    float acc = 0.f;
    int j = 0;
    for (; j + 8 <= np; j += 8) {       // loads first, then the additions in order
        float v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) v[u] = p[(size_t)(j + u) * n];
#pragma unroll
        for (int u = 0; u < 8; ++u) acc += v[u];
    }
    for (; j < np; ++j) acc += p[(size_t)j * n];
    const int e = i / kM, r = i - e * kM;   // piece states are column-major [65][256]
    uint8_t* img = image + (size_t)bh * (2 * kSBytes);
    const __nv_bfloat16 b = __float2bfloat16_rn(acc);
    if (e < kDV) {
        const uint32_t off = (uint32_t)r * 128u + ((((uint32_t)e >> 3) ^ ((uint32_t)r & 7u)) << 4) + ((uint32_t)e & 7u) * 2u;
        *reinterpret_cast<__nv_bfloat16*>(img + off) = b;
    } else {
        *reinterpret_cast<__nv_bfloat16*>(img + kSBytes + (uint32_t)r * 128u + (((uint32_t)r & 7u) << 4)) = b;
    }
}

// Causal: piece j of head bh <- sum of pieces 0..j-1 (exclusive prefix, in order).
// One thread per 4 consecutive elements (float4); pieces in register batches of 8.
__global__ void k_scan_pieces(float* __restrict__ part, Ranges R) {
    const int bh = blockIdx.y;
    const int i4 = blockIdx.x * blockDim.x + threadIdx.x;
    constexpr int n = kM * (kDV + 1);
    static_assert(n % 4 == 0, "float4 scan");
    if (i4 >= n / 4) return;
    const int np = last_cta(R, bh) - first_cta(R, bh) + 1;
    float4* p = reinterpret_cast<float4*>(part + (size_t)bh * R.pstride * n) + i4;
    float4 run = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < np; j += 8) {
        float4 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)
            if (j + u < np) v[u] = p[(size_t)(j + u) * (n / 4)];
#pragma unroll
        for (int u = 0; u < 8; ++u)
            if (j + u < np) {
                p[(size_t)(j + u) * (n / 4)] = run;
                run.x += v[u].x;
                run.y += v[u].y;
                run.z += v[u].z;
                run.w += v[u].w;
            }
    }
}

// Gated causal calls (RFA-Gate): decayed prefix of pieces.  Piece j of head
// bh <- prefix_j, prefix_0 = 0, prefix_{j+1} = d_j prefix_j + piece_j, with d_j
// the product of piece j's gates (the pieces hold their keys weighted toward
// their own end).  One thread per element.
__global__ void k_scan_pieces_decay(float* __restrict__ part, const float* __restrict__ pdecay, Ranges R) {
    const int bh = blockIdx.y;
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    constexpr int n = kM * (kDV + 1);
    if (i >= n) return;
    const int np = last_cta(R, bh) - first_cta(R, bh) + 1;
    float* p = part + (size_t)bh * R.pstride * n + i;
    const float* d = pdecay + (size_t)bh * R.pstride;
    float run = 0.f;
    for (int j = 0; j < np; ++j) {
        const float v = p[(size_t)j * n];
        p[(size_t)j * n] = run;
        run = fmaf(run, d[j], v);
    }
}

// Gated causal calls: per token of a piece (the ranges of the state kernel cut
// at head boundaries), the log2 weight of its key toward the piece's end,
//   wlog_j = sum_{l in (j, end]} log2 g_l + log2(1 - g_j)   (-1e30 where 1 - g_j = 0 or past L),
// and per piece the product of its gates (pdecay, indexed like the piece
// states).  Gates are clamped below at 2^-126, so a zero gate ends the history
// without turning any sum into -inf.  grid R.G (one block per range), 128 threads.
__global__ void __launch_bounds__(128) k_gate_weights(const float* __restrict__ gate, float* __restrict__ wlog,
                                                      float* __restrict__ pdecay, int L, Ranges R) {
    __shared__ float wsum[4];
    const int cta = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g0 = cta * R.per, g1 = min(R.T, g0 + R.per);
    float run = 0.f;   // log2 of the product of the piece's gates after the current tile
    int cur_bh = -1;
    for (int g = g1 - 1; g >= g0; --g) {   // backwards: each piece from its end
        const int bh = g / R.tph, tok = (g % R.tph) * kTile + tid;
        if (bh != cur_bh) {
            if (cur_bh >= 0 && tid == 0) pdecay[(size_t)cur_bh * R.pstride + (cta - first_cta(R, cur_bh))] = exp2f(run);
            run = 0.f;
            cur_bh = bh;
        }
        const bool live = tok < L;
        const float gv = live ? gate[(size_t)bh * L + tok] : 1.f;
        const float lg = log2f(fmaxf(gv, 1.17549435e-38f));
        float sfx = lg;   // sum over tokens tid..(end of the warp)
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float t = __shfl_down_sync(0xffffffffu, sfx, o);
            if (lane + o < 32) sfx += t;
        }
        if (lane == 0) wsum[warp] = sfx;
        __syncthreads();
        float later = 0.f;
        for (int w = warp + 1; w < 4; ++w) later += wsum[w];
        const float tile_sum = (wsum[0] + wsum[1]) + (wsum[2] + wsum[3]);
        __syncthreads();
        if (live) {
            const float one_m = 1.f - gv;
            wlog[(size_t)bh * L + tok] = one_m > 0.f ? (sfx + later - lg + run) + log2f(one_m) : -1.0e30f;
        }
        run += tile_sum;
    }
    if (cur_bh >= 0 && tid == 0) pdecay[(size_t)cur_bh * R.pstride + (cta - first_cta(R, cur_bh))] = exp2f(run);
}

// ============================================================ stateful calls
// state[bh][r][e] += scale * sum over the head's pieces (in order) of the
// column-major piece states: public state rows from the state kernel's sums.
__global__ void k_accum_cols(const float* __restrict__ part, float* __restrict__ state, Ranges R, float scale) {
    const int bh = blockIdx.y;
    const int i = blockIdx.x * blockDim.x + threadIdx.x;   // column-major index e * 256 + r
    constexpr int n = kM * (kDV + 1);
    if (i >= n) return;
    const int np = last_cta(R, bh) - first_cta(R, bh) + 1;
    const float* p = part + (size_t)bh * R.pstride * n + i;
    float a = 0.f;
    for (int j = 0; j < np; ++j) a += p[(size_t)j * n];
    const int e = i / kM, r = i - e * kM;
    state[(size_t)bh * n + (size_t)r * (kDV + 1) + e] += scale * a;
}

// Readout operand image (as k_reduce_pack writes it) from a public state
// [256][65] fp32: S~ block and z~ in column 0 of the second block, bf16.
__global__ void k_pack_state(const float* __restrict__ state, uint8_t* __restrict__ image) {
    const int bh = blockIdx.y;
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    constexpr int n = kM * (kDV + 1);
    if (i >= n) return;
    const int r = i / (kDV + 1), e = i - r * (kDV + 1);
    uint8_t* img = image + (size_t)bh * (2 * kSBytes);
    const __nv_bfloat16 b = __float2bfloat16_rn(state[(size_t)bh * n + i]);
    if (e < kDV) {
        const uint32_t off = (uint32_t)r * 128u + ((((uint32_t)e >> 3) ^ ((uint32_t)r & 7u)) << 4) + ((uint32_t)e & 7u) * 2u;
        *reinterpret_cast<__nv_bfloat16*>(img + off) = b;
    } else {
        *reinterpret_cast<__nv_bfloat16*>(img + kSBytes + (uint32_t)r * 128u + (((uint32_t)r & 7u) << 4)) = b;
    }
}

// ==================================================================== readout
// Persistent over the same flattened (head, tile) ranges as the state kernel;
// omega and the head's [S~ | z~] image are reloaded only when the range moves
// to another head.  Per 128-query tile t (tensor-memory slot t mod 2, 256 columns):
//   P = Q omega^T (N = 256)                     -> slot [0,256)
//   Phi_Q = exp2(a P - a max_r P) packed bf16   -> [0,64) (features 0..127), [192,256) (128..255)
//           (ReLU: max(P, 0); trigonometric, rows [omega; omega]: P of the first 128
//           rows only, then sin and cos of s P from one range reduction, without
//           h(x), a factor of the row that cancels in num / den)
//   [num | den] = Phi_Q [S~ | z~] (N = 80)      -> [64,144)
//   out = num / den, staged in shared memory and written by one TMA store
// (Eq. 4 of Rethinking Attention with Performers).  The feature and output
// work of tile t+1 overlaps the contraction of tile t.
//   warp 0: TMA producer (one thread polls the Q ring, omega and the image)
//   warp 1: projection MMAs; warp 2: [num | den] MMAs (separate issuers, so each
//   goes as soon as its own inputs are ready)
//   warps 4..19: four groups of four (lane = query), group g owns features
//   [64g, 64g+64): it loads them once, the groups swap row maxima, and each
//   writes its packed features and then output columns [16g, 16g+16).
constexpr int kReadoutThreads = 640;
constexpr int kRStages = 3;
constexpr uint32_t kRImage = 2 * kSBytes;   // [S~ | z~] image: two [256][64] SW128 blocks

struct RdBars {
    uint64_t q_full[kRStages], q_empty[kRStages];
    uint64_t w_full, w_empty, img_full, img_empty;
    uint64_t pq_full[2], phiq_full[2], o_full[2], slot_free[2];
    uint64_t mxb, stage_full, stage_free[2];
    uint32_t tmem_base;
};

// Packed destination column of feature quarter g (16-column steps k = 0, 1).
__device__ __forceinline__ uint32_t quarter_dst(int g) { return g < 2 ? 32u * g : 192u + 32u * (g - 2); }

template <int KIND>
__global__ void __launch_bounds__(kReadoutThreads, 1)
k_tc_readout(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_w,
             const __grid_constant__ CUtensorMap tm_o, const uint8_t* __restrict__ image, int H, int L, float s,
             Ranges R, int* err) {
    constexpr bool POS = KIND == FAVOR_KERNEL_SOFTMAX_POS;
    constexpr bool TRIG = KIND == FAVOR_KERNEL_SOFTMAX_TRIG;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1k(smem_raw);
    const uint32_t s_w = smem_u32(sm);
    const uint32_t s_q = s_w + kOmegaBytes;                   // Q ring
    const uint32_t s_img = s_q + kRStages * kTileBytes;       // [S~ | z~]: 2 blocks of 32 KB
    const uint32_t s_stage = s_img + kRImage;                 // output staging, 2 x 16 KB
    const uint32_t s_mx = s_stage + 2 * kTileBytes;           // row maxima [2 tiles][4 quarters][128]
    RdBars* bars = reinterpret_cast<RdBars*>(sm + (s_mx - s_w) + 2 * 4 * kTile * 4);
    const int cta = blockIdx.x;
    const int g0 = cta * R.per, g1 = min(R.T, g0 + R.per);
    const int n = g1 - g0;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const float a = s * kLog2e;

    if (threadIdx.x == 0) {
        uint64_t* b = reinterpret_cast<uint64_t*>(bars);
        // order and arrival counts follow the fields of RdBars
        const int counts[] = {1, 1, 1, 1, 1, 1,   1, 1, 1, 1,   1, 1, 16, 16, 1, 1, 16, 16,   16, 16, 1, 1};
        static_assert(sizeof(counts) / sizeof(int) * sizeof(uint64_t) == offsetof(RdBars, tmem_base), "barrier table");
        for (int i = 0; i < (int)(sizeof(counts) / sizeof(int)); ++i) mbar_init(b + i, counts[i]);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&bars->tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int nq = 0, nw = 0, ni = 0;               // next Q tile; tiles covered by loaded omega / image
            int wseg = 0, iseg = 0;                   // omega / image loads done so far
            long long t0 = clock64();
            while (nq < n || nw < n || ni < n) {
                bool progress = false;
                if (nq < n && (nq < kRStages || mbar_test_wait(&bars->q_empty[nq % kRStages], ((nq / kRStages) + 1) & 1))) {
                    const int g = g0 + nq;
                    mbar_expect_tx(&bars->q_full[nq % kRStages], kTileBytes);
                    tma_load_3d(sm + (s_q - s_w) + (nq % kRStages) * kTileBytes, &tm_q, &bars->q_full[nq % kRStages], 0,
                                (g % R.tph) * kTile, g / R.tph);
                    ++nq;
                    progress = true;
                }
                if (nw < n && (wseg == 0 || mbar_test_wait(&bars->w_empty, (wseg - 1) & 1))) {
                    const int h = ((g0 + nw) / R.tph) % H;
                    mbar_expect_tx(&bars->w_full, kOmegaBytes);
                    tma_load_2d(sm, &tm_w, &bars->w_full, 0, h * kM);
                    while (nw < n && ((g0 + nw) / R.tph) % H == h) ++nw;   // tiles of this omega segment
                    ++wseg;
                    progress = true;
                }
                if (ni < n && (iseg == 0 || mbar_test_wait(&bars->img_empty, (iseg - 1) & 1))) {
                    const int bh = (g0 + ni) / R.tph;
                    mbar_expect_tx(&bars->img_full, kRImage);
                    bulk_load(sm + (s_img - s_w), image + (size_t)bh * kRImage, kRImage, &bars->img_full);
                    while (ni < n && (g0 + ni) / R.tph == bh) ++ni;
                    ++iseg;
                    progress = true;
                }
                if (progress) {
                    t0 = clock64();
                } else {
                    __nanosleep(64);
                    if (clock64() - t0 > (4LL << 30)) {
                        atomicCAS(err, 0, 301);
                        break;
                    }
                }
            }
        }
    } else if (warp == 1) {
        // --------------------------------------------------- projection MMAs
        // P for tile u: an omega segment start waits w_full; the last P of a segment frees omega
        if (lane == 0) {
            uint32_t wph = 0;
            for (int u = 0; u < n; ++u) {
                const int g = g0 + u, h = (g / R.tph) % H;
                const bool seg_start = u == 0 || ((g - 1) / R.tph) % H != h;
                const bool seg_end = u + 1 < n && ((g + 1) / R.tph) % H != h;
                const uint32_t sl = tmem + 256u * (uint32_t)(u & 1);
                if (seg_start) {
                    if (!mbar_wait(&bars->w_full, wph, err, 311)) break;
                    wph ^= 1;
                }
                if (!mbar_wait(&bars->q_full[u % kRStages], (u / kRStages) & 1, err, 312)) break;
                if (u >= 2 && !mbar_wait(&bars->slot_free[u & 1], ((u >> 1) - 1) & 1, err, 313)) break;
                tc_fence_after();
                // trigonometric: the rows repeat after 128, so project the first 128 only
                issue_projection(sl, s_q + (u % kRStages) * kTileBytes, s_w, TRIG ? 128 : 256);
                mma_commit(&bars->pq_full[u & 1]);
                mma_commit(&bars->q_empty[u % kRStages]);
                if (seg_end) mma_commit(&bars->w_empty);
            }
        }
    } else if (warp == 2) {
        // ---------------------------------------------------- [num | den] MMAs
        if (lane == 0) {
            const uint32_t id_o = make_idesc(128, 80, 0, 1);
            uint32_t iph = 0;
            for (int t = 0; t < n; ++t) {
                const int bh = (g0 + t) / R.tph;
                const bool seg_start = t == 0 || (g0 + t - 1) / R.tph != bh;
                const bool seg_end = t + 1 < n && (g0 + t + 1) / R.tph != bh;
                const uint32_t sl = tmem + 256u * (uint32_t)(t & 1);
                if (seg_start) {
                    if (!mbar_wait(&bars->img_full, iph, err, 314)) break;
                    iph ^= 1;
                }
                if (!mbar_wait(&bars->phiq_full[t & 1], (t >> 1) & 1, err, 315)) break;
                tc_fence_after();
                // B MN-major, N = 80 over two 64-wide blocks (LBO = 32 KB)
                const uint64_t b0 = make_desc(s_img, kSBytes, 1024, SW_128B);
#pragma unroll
                for (int kk = 0; kk < 16; ++kk)
                    mma_ts(sl + 64, kk < 8 ? sl + 8 * kk : sl + 192 + 8 * (kk - 8), b0 + 128 * kk, id_o,
                           kk > 0 ? 1u : 0u);
                mma_commit(&bars->o_full[t & 1]);
                if (seg_end) mma_commit(&bars->img_empty);
            }
        }
    } else if (warp >= 4) {
        // ------------------------------------------------ features and output
        const int grp = (warp - 4) >> 2, q = warp & 3;
        const uint32_t row = 32 * q + lane;
        const uint32_t tl = tmem + ((uint32_t)(32 * q) << 16);
        float* mx = reinterpret_cast<float*>(sm + (s_mx - s_w));
        bool ok = true;
        auto features = [&](int u) -> bool {
            const uint32_t sl = tl + 256u * (uint32_t)(u & 1);
            if (!mbar_wait(&bars->pq_full[u & 1], (u >> 1) & 1, err, 321)) return false;
            tc_fence_after();
            if (TRIG) {
                // group g: projections [32g, 32g+32) -> sin features [32g, ..) packed in
                // [16g, 16g+16), cos features [128 + 32g, ..) packed in [192 + 16g, ..)
                uint32_t p[32];
                tmem_ld32(sl + 32u * (uint32_t)grp, p);
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->mxb);   // every group's projections are in registers
                if (!mbar_wait(&bars->mxb, u & 1, err, 322)) return false;
                tc_fence_after();
                uint32_t ws[16], wc[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    float s0, c0, s1, c1;
                    sincos_pair(s * __uint_as_float(p[2 * i]), s0, c0);
                    sincos_pair(s * __uint_as_float(p[2 * i + 1]), s1, c1);
                    ws[i] = pack_bf16(s0, s1);
                    wc[i] = pack_bf16(c0, c1);
                }
                tmem_st16(sl + 16u * (uint32_t)grp, ws);
                tmem_st16(sl + 192u + 16u * (uint32_t)grp, wc);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->phiq_full[u & 1]);
                return true;
            }
            uint32_t p[64];
            tmem_ld64(sl + 64u * (uint32_t)grp, p);
            tmem_ld_wait();
            float m = -INFINITY;
            if (POS) {
                float m0 = -INFINITY, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
#pragma unroll
                for (int i = 0; i < 64; i += 4) {
                    m0 = fmaxf(m0, __uint_as_float(p[i]));
                    m1 = fmaxf(m1, __uint_as_float(p[i + 1]));
                    m2 = fmaxf(m2, __uint_as_float(p[i + 2]));
                    m3 = fmaxf(m3, __uint_as_float(p[i + 3]));
                }
                m = fmaxf(fmaxf(m0, m1), fmaxf(m2, m3));
                mx[((u & 1) * 4 + grp) * kTile + row] = m;
            }
            // every group holds its projections in registers past this point, so
            // the packed features may overwrite any group's fp32 columns
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->mxb);
            if (!mbar_wait(&bars->mxb, u & 1, err, 322)) return false;
            tc_fence_after();
            float c = 0.f;
            if (POS) {
                const float* mr = mx + (u & 1) * 4 * kTile + row;
                c = fmaxf(fmaxf(mr[0], mr[kTile]), fmaxf(mr[2 * kTile], mr[3 * kTile])) * a;
            }
            const uint32_t dst = sl + quarter_dst(grp);
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                uint32_t w[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    float f0, f1;
                    if (POS) {
                        f0 = ex2(fmaf(__uint_as_float(p[32 * k + 2 * i]), a, -c));
                        f1 = ex2(fmaf(__uint_as_float(p[32 * k + 2 * i + 1]), a, -c));
                    } else {
                        f0 = fmaxf(__uint_as_float(p[32 * k + 2 * i]), 0.f);
                        f1 = fmaxf(__uint_as_float(p[32 * k + 2 * i + 1]), 0.f);
                    }
                    w[i] = pack_bf16(f0, f1);
                }
                tmem_st16(dst + 16 * k, w);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->phiq_full[u & 1]);
            return true;
        };
        if (n > 0) ok = features(0);
        for (int t = 0; t < n && ok; ++t) {
            if (t + 1 < n && !(ok = features(t + 1))) break;
            // output tile t: this group's 16 columns of num / den
            const int g = g0 + t, bh = g / R.tph, tok0 = (g % R.tph) * kTile;
            const uint32_t sl = tl + 256u * (uint32_t)(t & 1);
            if (!mbar_wait(&bars->o_full[t & 1], (t >> 1) & 1, err, 323)) break;
            tc_fence_after();
            uint32_t nv[16], dz[16];
            tmem_ld16(sl + 64 + 16 * grp, nv);
            tmem_ld16(sl + 128, dz);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->slot_free[t & 1]);
            const uint32_t stage = s_stage + (uint32_t)(t & 1) * kTileBytes;
            if (t >= 2 && !mbar_wait(&bars->stage_free[t & 1], ((t >> 1) - 1) & 1, err, 324)) break;
            const float den = __uint_as_float(dz[0]);
            const float inv = den != 0.f ? 1.f / den : 0.f;
#pragma unroll
            for (uint32_t c = 0; c < 2; ++c)
                st_shared_v4(stage + sw128(row, 2 * grp + c),
                             pack_bf16(__uint_as_float(nv[8 * c + 0]) * inv, __uint_as_float(nv[8 * c + 1]) * inv),
                             pack_bf16(__uint_as_float(nv[8 * c + 2]) * inv, __uint_as_float(nv[8 * c + 3]) * inv),
                             pack_bf16(__uint_as_float(nv[8 * c + 4]) * inv, __uint_as_float(nv[8 * c + 5]) * inv),
                             pack_bf16(__uint_as_float(nv[8 * c + 6]) * inv, __uint_as_float(nv[8 * c + 7]) * inv));
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->stage_full);
            if (warp == 4 && lane == 0) {
                if (!mbar_wait(&bars->stage_full, t & 1, err, 325)) break;
                tma_store_3d(&tm_o, stage, 0, tok0, bh);
                bulk_commit();
                bulk_wait_read<1>();   // the previous tile's store has read its buffer
                if (t >= 1) mbar_arrive(&bars->stage_free[(t - 1) & 1]);
            }
        }
        if (warp == 4 && lane == 0) bulk_wait<0>();   // output stores complete before exit
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, 512);
}

// ===================================================================== causal
// Persistent over ranges, chunks of 128 tokens.  For chunk t of head bh with
// state S(t), z(t) (the sums over all earlier keys of the head):
//   num = Phi_Q S~(t) + tril(Phi_Q Phi_K^T) V       (tensor cores)
//   den = Phi_Q z(t)  + rowsum tril(Phi_Q Phi_K^T)  (fp32 on the CUDA cores, from the same
//                                                    bf16-rounded Phi_Q and tril(A) the numerator uses)
//   out = num / den,   S(t+1) = S(t) + Phi_K^T V,   z(t+1) = z(t) + Phi_K^T 1
// (App. B.1 Eq. 11 of Rethinking Attention with Performers, taken chunk by chunk).
//
// Roles (576 threads, 18 warps):
//   warp 0      TMA producer: one thread keeps the Q, K and V streams and omega independent
//   warp 1      the MMA issuer: one thread issues every contraction in a fixed order
//   warps 2..5  query group A (lane = query row): norm shift, features of half 0 and their
//               part of Phi_Q z, then the causal mask of A and its row sums
//   warps 6..9  query group B: norm shift, features of half 1 and their part of Phi_Q z,
//               then the output rows (num / den, stored from registers)
//   warps 10..17 key warps, two per lane quarter: warps 10..13 take tokens 0..63 of the
//               tile, warps 14..17 tokens 64..127 (lane = feature of the quarter); key norms
//               (first four), key features into Phi_K, z, and the S~ / z~ refresh
//
// Tensor memory: three rotating 128-column slots and the fp32 state in
// [384,512) (two halves of 64 columns, lane = feature).  Chunk t uses
//   X: P_Q half 0 -> Phi_Q half 0 packed in [0,64); num in [64,128)
//   Y: P_Q half 1 -> Phi_Q half 1 packed in [0,64)
//   Z: P_K^T half 0, then half 1, then A, then tril(A) packed in [0,64)
// and chunk t+1 takes X' = Z, Y' = X, Z' = Y.  One thread issues all MMAs, and
// tcgen05.mma from one thread run in issue order, so a projection of chunk
// t+1 that is issued after the last MMA of chunk t reading its slot needs no
// wait for that MMA; it waits only for CUDA-core reads of the slot.  Issue
// order of iteration t:
//   A(t) over feature half 0 (as soon as half 0's query features are in), A
//   over half 1, the inter term (once the S~ image of t is in), key projection
//   half 0 of t+1, the state update of t, key projection half 1 of t+1, the
//   intra term of t, query projection halves 0 and 1 of t+1.
// The key warps run one step ahead of the state: they compute chunk t+1's
// features while the state update of t is queued, holding them in registers
// until that update has read Phi_K, then refresh S~ and publish z~ of t+2.
//
// Query shift: features are exp2(a p - c) with c = a W_h ||q|| and W_h the
// largest row norm of the head's omega, so omega_r . q <= W_h ||q|| (Cauchy-
// Schwarz) keeps every feature at most 1 without a pass over the row; c is a
// per-row constant, so it cancels between num and den.  Key features are
// exp2(a p + c_j) with the per-token offset c_j = -(s^2 ||k_j||^2 / 2 +
// kappa_h) log2(e) taken from shared memory (-1e30 for rows past L).
//
// Trigonometric kind (rows [omega; omega]): sin of s p in half 0, cos in half
// 1, the keys times h(s k_j) from cs (query_half_trig, key_half_row_trig).
//
// Gated calls (GATED, RFA-Gate): warp 10 scans each chunk's gates into C_i
// (cumulative log2 gate), T_j = C_j - log2(1 - g_j), the keys' state weights
// 2^(C_last - C_j) (1 - g_j) and the decay 2^C_last (g_full).  After A has read
// Phi_Q the query groups scale it by 2^C_i (phiq_scaled: the inter term then
// carries that row factor) and the mask multiplies A_ij by 2^(C_i - T_j);
// after A has read Phi_K the key warps weight it for the state update
// (phik_w); the refresh writes the S~ image of S and then S 2^C_last back for
// the update to accumulate onto.
constexpr int kCausalThreads = 576;

struct CaBars {
    uint64_t q_full, k_full, v_full, w_full, q_empty, k_empty, v_empty, w_empty;
    uint64_t pq0_full, pq1_full, phiq0_full, phiq1_full, pk_full, pk_free, cs_full, phik_full;
    uint64_t phik_free, a_full, am_full, s_full, st_full, ai_done, o_full, o_empty;
    uint64_t z_full, zx_full, mma_done, stage_full, stage_free[2];
    uint64_t g_full[2], phiq_scaled, phik_w;   // gated calls only
    uint32_t tmem_base;
};

// Slot of role 0 (X), 1 (Y) or 2 (Z) for a chunk with index t, r3 = t mod 3.
__device__ __forceinline__ uint32_t ca_slot(int role, int r3) {
    int i = role - r3;
    i += (i < 0) ? 3 : 0;
    return 128u * (uint32_t)i;
}

// Features of one query half, 32 projections at a time, packed in place into
// the first 64 columns at taddr; returns sum_r f_r z~_r over the half's z~
// (fp32 in shared memory at zaddr), taken over the bf16-rounded features.
// The block loop stays rolled: the kernel's roles run different code at the
// same time, and unrolled bodies overflow the instruction cache.
template <int KIND>
__device__ __noinline__ float query_half(uint32_t taddr, float a, float c, uint32_t zaddr) {
    float d0 = 0.f, d1 = 0.f;
#pragma unroll 1
    for (int blk = 0; blk < 4; ++blk) {
        uint32_t p[32], w[16];
        tmem_ld32(taddr + 32 * blk, p);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint4 z4a = ld_shared_v4(zaddr + 4 * (32 * blk + 8 * j));
            const uint4 z4b = ld_shared_v4(zaddr + 4 * (32 * blk + 8 * j + 4));
            const float zz[8] = {__uint_as_float(z4a.x), __uint_as_float(z4a.y), __uint_as_float(z4a.z),
                                 __uint_as_float(z4a.w), __uint_as_float(z4b.x), __uint_as_float(z4b.y),
                                 __uint_as_float(z4b.z), __uint_as_float(z4b.w)};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int e = 8 * j + 2 * i;
                float f0, f1;
                if (KIND == FAVOR_KERNEL_SOFTMAX_POS) {
                    f0 = ex2(fmaf(__uint_as_float(p[e]), a, -c));
                    f1 = ex2(fmaf(__uint_as_float(p[e + 1]), a, -c));
                } else {
                    f0 = fmaxf(__uint_as_float(p[e]), 0.f);
                    f1 = fmaxf(__uint_as_float(p[e + 1]), 0.f);
                }
                const uint32_t pk = pack_bf16(f0, f1);
                d0 = fmaf(bf16lo(pk), zz[2 * i], d0);
                d1 = fmaf(bf16hi(pk), zz[2 * i + 1], d1);
                w[4 * j + i] = pk;
            }
        }
        // packed block blk lands in columns [16 blk, 16 blk + 16), all of which were read already
        tmem_st16(taddr + 16 * blk, w);
    }
    return d0 + d1;
}

// Features of one query half, 32 projections at a time, packed in place into
// the first 64 columns at taddr; returns sum_r f_r z~_r over the half's z~
// (fp32 in shared memory at zaddr), taken over the bf16-rounded features.
// This copy serves the trigonometric kind: sin (half 0) or cos (half 1, COS)
// of a p, where the caller passes a = s (c is unused).
// The block loop stays rolled: the kernel's roles run different code at the
// same time, and unrolled bodies overflow the instruction cache.
template <int KIND, bool COS>
__device__ __noinline__ float query_half_trig(uint32_t taddr, float a, float c, uint32_t zaddr) {
    float d0 = 0.f, d1 = 0.f;
#pragma unroll 1
    for (int blk = 0; blk < 4; ++blk) {
        uint32_t p[32], w[16];
        tmem_ld32(taddr + 32 * blk, p);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint4 z4a = ld_shared_v4(zaddr + 4 * (32 * blk + 8 * j));
            const uint4 z4b = ld_shared_v4(zaddr + 4 * (32 * blk + 8 * j + 4));
            const float zz[8] = {__uint_as_float(z4a.x), __uint_as_float(z4a.y), __uint_as_float(z4a.z),
                                 __uint_as_float(z4a.w), __uint_as_float(z4b.x), __uint_as_float(z4b.y),
                                 __uint_as_float(z4b.z), __uint_as_float(z4b.w)};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int e = 8 * j + 2 * i;
                float f0, f1;
                if (KIND == FAVOR_KERNEL_SOFTMAX_POS) {
                    f0 = ex2(fmaf(__uint_as_float(p[e]), a, -c));
                    f1 = ex2(fmaf(__uint_as_float(p[e + 1]), a, -c));
                } else if (KIND == FAVOR_KERNEL_SOFTMAX_TRIG) {
                    f0 = sincos_reduced(a * __uint_as_float(p[e]), COS);
                    f1 = sincos_reduced(a * __uint_as_float(p[e + 1]), COS);
                } else {
                    f0 = fmaxf(__uint_as_float(p[e]), 0.f);
                    f1 = fmaxf(__uint_as_float(p[e + 1]), 0.f);
                }
                const uint32_t pk = pack_bf16(f0, f1);
                d0 = fmaf(bf16lo(pk), zz[2 * i], d0);
                d1 = fmaf(bf16hi(pk), zz[2 * i + 1], d1);
                w[4 * j + i] = pk;
            }
        }
        // packed block blk lands in columns [16 blk, 16 blk + 16), all of which were read already
        tmem_st16(taddr + 16 * blk, w);
    }
    return d0 + d1;
}

// Causal mask of one row of A (fp32, 128 columns at taddr), packed in place into
// [0,64); returns the row sum of the kept bf16-rounded values.  Blocks of keys
// entirely after every row of the warp (blk > q) are written as zeros unread.
__device__ __noinline__ float mask_row(uint32_t taddr, int row, int q) {
    float s0 = 0.f, s1 = 0.f;
#pragma unroll 1
    for (int blk = 0; blk < 4; ++blk) {
        uint32_t w[16];
        if (blk <= q) {
            uint32_t p[32];
            tmem_ld32(taddr + 32 * blk, p);
            tmem_ld_wait();
            const int lim = row - 32 * blk;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float f0 = (2 * i <= lim) ? __uint_as_float(p[2 * i]) : 0.f;
                const float f1 = (2 * i + 1 <= lim) ? __uint_as_float(p[2 * i + 1]) : 0.f;
                w[i] = pack_bf16(f0, f1);
                s0 += bf16lo(w[i]);
                s1 += bf16hi(w[i]);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) w[i] = 0u;
        }
        tmem_st16(taddr + 16 * blk, w);
    }
    return s0 + s1;
}

// Key features of feature row r for the 64 tokens [64u, 64u + 64) of the tile
// (their projections: 64 fp32 columns at taddr, offsets folded in by c_j), 32
// columns at a time; `release` (if not null) is arrived once both blocks are in
// registers, so the slot may take the next projection while the rest is
// computed.  f = exp2(a p + c_j) (positive, c_j from cs) or max(p, 0) (ReLU),
// packed to bf16 in registers; then, after `gate` (if not null: Phi_K's
// previous contents are no longer read) has completed the phase of parity
// gate_par, stored into Phi_K [feature][token] (token block u of 64, 128-byte
// swizzle).  Returns the sum of the features; *ok = false if the gate's wait
// gave up (nothing stored).
template <int KIND>
__device__ __noinline__ float key_half_row(uint32_t taddr, uint64_t* release, uint64_t* gate, uint32_t gate_par,
                                           int* err, bool* ok, uint32_t phi, uint32_t r, float a, uint32_t cs) {
    uint32_t w[32];
    float z0 = 0.f, z1 = 0.f;
#pragma unroll
    for (int blk = 0; blk < 2; ++blk) {
        uint32_t p[32];
        tmem_ld32(taddr + 32 * blk, p);
        tmem_ld_wait();
        if (blk == 1 && release) {
            tc_fence_before();
            __syncwarp();
            if ((threadIdx.x & 31) == 0) mbar_arrive(release);
        }
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
            float c8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            if (KIND == FAVOR_KERNEL_SOFTMAX_POS) {
                const uint32_t ca_addr = cs + 4 * (32 * blk + 8 * cc);
                const uint4 ca = ld_shared_v4(ca_addr), cb = ld_shared_v4(ca_addr + 16);
                c8[0] = __uint_as_float(ca.x); c8[1] = __uint_as_float(ca.y);
                c8[2] = __uint_as_float(ca.z); c8[3] = __uint_as_float(ca.w);
                c8[4] = __uint_as_float(cb.x); c8[5] = __uint_as_float(cb.y);
                c8[6] = __uint_as_float(cb.z); c8[7] = __uint_as_float(cb.w);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float x0 = __uint_as_float(p[8 * cc + 2 * i]), x1 = __uint_as_float(p[8 * cc + 2 * i + 1]);
                float f0, f1;
                if (KIND == FAVOR_KERNEL_SOFTMAX_POS) {
                    f0 = ex2(fmaf(x0, a, c8[2 * i]));
                    f1 = ex2(fmaf(x1, a, c8[2 * i + 1]));
                } else {
                    f0 = fmaxf(x0, 0.f);
                    f1 = fmaxf(x1, 0.f);
                }
                z0 += f0;
                z1 += f1;
                w[16 * blk + 4 * cc + i] = pack_bf16(f0, f1);
            }
        }
    }
    if (gate && !mbar_wait(gate, gate_par, err, 258)) {
        *ok = false;
        return 0.f;
    }
#pragma unroll
    for (int cc = 0; cc < 8; ++cc) st_shared_v4(phi + sw128(r, (uint32_t)cc), w[4 * cc], w[4 * cc + 1], w[4 * cc + 2], w[4 * cc + 3]);
    return z0 + z1;
}

// Key features of feature row r for the 64 tokens [64u, 64u + 64) of the tile
// (their projections: 64 fp32 columns at taddr, offsets folded in by c_j), 32
// columns at a time; `release` (if not null) is arrived once both blocks are in
// registers, so the slot may take the next projection while the rest is
// computed.  f = exp2(a p + c_j) (positive, c_j from cs) or max(p, 0) (ReLU),
// packed to bf16 in registers; then, after `gate` (if not null: Phi_K's
// previous contents are no longer read) has completed the phase of parity
// gate_par, stored into Phi_K [feature][token] (token block u of 64, 128-byte
// swizzle).  Returns the sum of the features; *ok = false if the gate's wait
// gave up (nothing stored).  This copy serves the trigonometric kind: sin (or
// cos, COS) of a p times the token's h(s k_j) from cs, where the caller passes a = s.
template <int KIND, bool COS>
__device__ __noinline__ float key_half_row_trig(uint32_t taddr, uint64_t* release, uint64_t* gate, uint32_t gate_par,
                                           int* err, bool* ok, uint32_t phi, uint32_t r, float a, uint32_t cs) {
    uint32_t w[32];
    float z0 = 0.f, z1 = 0.f;
#pragma unroll
    for (int blk = 0; blk < 2; ++blk) {
        uint32_t p[32];
        tmem_ld32(taddr + 32 * blk, p);
        tmem_ld_wait();
        if (blk == 1 && release) {
            tc_fence_before();
            __syncwarp();
            if ((threadIdx.x & 31) == 0) mbar_arrive(release);
        }
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
            float c8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            if (KIND == FAVOR_KERNEL_SOFTMAX_POS || KIND == FAVOR_KERNEL_SOFTMAX_TRIG) {
                const uint32_t ca_addr = cs + 4 * (32 * blk + 8 * cc);
                const uint4 ca = ld_shared_v4(ca_addr), cb = ld_shared_v4(ca_addr + 16);
                c8[0] = __uint_as_float(ca.x); c8[1] = __uint_as_float(ca.y);
                c8[2] = __uint_as_float(ca.z); c8[3] = __uint_as_float(ca.w);
                c8[4] = __uint_as_float(cb.x); c8[5] = __uint_as_float(cb.y);
                c8[6] = __uint_as_float(cb.z); c8[7] = __uint_as_float(cb.w);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float x0 = __uint_as_float(p[8 * cc + 2 * i]), x1 = __uint_as_float(p[8 * cc + 2 * i + 1]);
                float f0, f1;
                if (KIND == FAVOR_KERNEL_SOFTMAX_POS) {
                    f0 = ex2(fmaf(x0, a, c8[2 * i]));
                    f1 = ex2(fmaf(x1, a, c8[2 * i + 1]));
                } else if (KIND == FAVOR_KERNEL_SOFTMAX_TRIG) {
                    f0 = sincos_reduced(a * x0, COS) * c8[2 * i];
                    f1 = sincos_reduced(a * x1, COS) * c8[2 * i + 1];
                } else {
                    f0 = fmaxf(x0, 0.f);
                    f1 = fmaxf(x1, 0.f);
                }
                z0 += f0;
                z1 += f1;
                w[16 * blk + 4 * cc + i] = pack_bf16(f0, f1);
            }
        }
    }
    if (gate && !mbar_wait(gate, gate_par, err, 258)) {
        *ok = false;
        return 0.f;
    }
#pragma unroll
    for (int cc = 0; cc < 8; ++cc) st_shared_v4(phi + sw128(r, (uint32_t)cc), w[4 * cc], w[4 * cc + 1], w[4 * cc + 2], w[4 * cc + 3]);
    return z0 + z1;
}

// Gated calls: packed bf16 feature row (64 columns at taddr) times f, in place.
__device__ __noinline__ void scale_packed_row(uint32_t taddr, float f) {
#pragma unroll 1
    for (int blk = 0; blk < 2; ++blk) {
        uint32_t w[32];
        tmem_ld32(taddr + 32 * blk, w);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) w[i] = pack_bf16(bf16lo(w[i]) * f, bf16hi(w[i]) * f);
        tmem_st16(taddr + 32 * blk, *reinterpret_cast<uint32_t(*)[16]>(&w[0]));
        tmem_st16(taddr + 32 * blk + 16, *reinterpret_cast<uint32_t(*)[16]>(&w[16]));
    }
}

// Gated calls: the causal mask of one row of A with the decay of the gates,
// A_ij 2^(C_i - T_j) for j <= i (C_i the row's cumulative log2 gate, T_j =
// C_j - log2(1 - g_j) at tcol, fp32 in shared memory), packed in place into
// [0,64); returns the row sum of the kept bf16-rounded values.
__device__ __noinline__ float mask_row_gated(uint32_t taddr, int row, int q, float ci, uint32_t tcol) {
    float s0 = 0.f, s1 = 0.f;
#pragma unroll 1
    for (int blk = 0; blk < 4; ++blk) {
        uint32_t w[16];
        if (blk <= q) {
            uint32_t p[32];
            tmem_ld32(taddr + 32 * blk, p);
            tmem_ld_wait();
            const int lim = row - 32 * blk;
#pragma unroll
            for (int j4 = 0; j4 < 8; ++j4) {
                const uint4 t4 = ld_shared_v4(tcol + 4 * (32 * blk + 4 * j4));
                const float tt[4] = {__uint_as_float(t4.x), __uint_as_float(t4.y), __uint_as_float(t4.z),
                                     __uint_as_float(t4.w)};
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int i = 2 * j4 + e;
                    const float f0 = (2 * i <= lim) ? __uint_as_float(p[2 * i]) * ex2(ci - tt[2 * e]) : 0.f;
                    const float f1 = (2 * i + 1 <= lim) ? __uint_as_float(p[2 * i + 1]) * ex2(ci - tt[2 * e + 1]) : 0.f;
                    w[i] = pack_bf16(f0, f1);
                    s0 += bf16lo(w[i]);
                    s1 += bf16hi(w[i]);
                }
            }
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) w[i] = 0u;
        }
        tmem_st16(taddr + 16 * blk, w);
    }
    return s0 + s1;
}

// Gated calls: the S~ image row r from the fp32 state row (64 columns at
// taddr), then the state row times the chunk's decay d, written back.
__device__ __noinline__ void refresh_decay_row(uint32_t taddr, uint32_t img, uint32_t r, float d) {
#pragma unroll 1
    for (int blk = 0; blk < 2; ++blk) {
        uint32_t sv[32];
        tmem_ld32(taddr + 32 * blk, sv);
        tmem_ld_wait();
#pragma unroll
        for (uint32_t c = 0; c < 4; ++c)
            st_shared_v4(img + sw128(r, 4 * blk + c),
                         pack_bf16(__uint_as_float(sv[8 * c]), __uint_as_float(sv[8 * c + 1])),
                         pack_bf16(__uint_as_float(sv[8 * c + 2]), __uint_as_float(sv[8 * c + 3])),
                         pack_bf16(__uint_as_float(sv[8 * c + 4]), __uint_as_float(sv[8 * c + 5])),
                         pack_bf16(__uint_as_float(sv[8 * c + 6]), __uint_as_float(sv[8 * c + 7])));
#pragma unroll
        for (int i = 0; i < 32; ++i) sv[i] = __float_as_uint(__uint_as_float(sv[i]) * d);
        tmem_st16(taddr + 32 * blk, *reinterpret_cast<uint32_t(*)[16]>(&sv[0]));
        tmem_st16(taddr + 32 * blk + 16, *reinterpret_cast<uint32_t(*)[16]>(&sv[16]));
    }
}

// Gated calls: Phi_K row r of token block u (64 tokens at phi) times the keys'
// state weights (fp32 at wcol, the block's 64 tokens), in place; returns the
// sum of the weighted bf16-rounded values.
__device__ __noinline__ float weight_phik_row(uint32_t phi, uint32_t r, uint32_t wcol) {
    float z0 = 0.f, z1 = 0.f;
#pragma unroll 1
    for (uint32_t cc = 0; cc < 8; ++cc) {
        const uint4 v = ld_shared_v4(phi + sw128(r, cc));
        const uint4 wa = ld_shared_v4(wcol + 4 * (8 * cc)), wb = ld_shared_v4(wcol + 4 * (8 * cc + 4));
        const uint32_t x[4] = {v.x, v.y, v.z, v.w};
        const float wt[8] = {__uint_as_float(wa.x), __uint_as_float(wa.y), __uint_as_float(wa.z), __uint_as_float(wa.w),
                             __uint_as_float(wb.x), __uint_as_float(wb.y), __uint_as_float(wb.z), __uint_as_float(wb.w)};
        uint32_t y[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            y[i] = pack_bf16(bf16lo(x[i]) * wt[2 * i], bf16hi(x[i]) * wt[2 * i + 1]);
            z0 += bf16lo(y[i]);
            z1 += bf16hi(y[i]);
        }
        st_shared_v4(phi + sw128(r, cc), y[0], y[1], y[2], y[3]);
    }
    return z0 + z1;
}

// S~ image row r from the fp32 state row (64 columns at taddr).
__device__ __noinline__ void refresh_row(uint32_t taddr, uint32_t img, uint32_t r) {
#pragma unroll 1
    for (int blk = 0; blk < 2; ++blk) {
        uint32_t sv[32];
        tmem_ld32(taddr + 32 * blk, sv);
        tmem_ld_wait();
#pragma unroll
        for (uint32_t c = 0; c < 4; ++c)
            st_shared_v4(img + sw128(r, 4 * blk + c),
                         pack_bf16(__uint_as_float(sv[8 * c]), __uint_as_float(sv[8 * c + 1])),
                         pack_bf16(__uint_as_float(sv[8 * c + 2]), __uint_as_float(sv[8 * c + 3])),
                         pack_bf16(__uint_as_float(sv[8 * c + 4]), __uint_as_float(sv[8 * c + 5])),
                         pack_bf16(__uint_as_float(sv[8 * c + 6]), __uint_as_float(sv[8 * c + 7])));
    }
}

// fp32 state row (64 columns at taddr), S~ image row r from a prefix in global
// memory stored column-major (element e of the row at src[e * 256]).
__device__ __noinline__ void load_prefix_row(const float* src, uint32_t taddr, uint32_t img, uint32_t r) {
#pragma unroll 1
    for (int blk = 0; blk < 4; ++blk) {
        uint32_t sv[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) sv[i] = __float_as_uint(src[(size_t)(16 * blk + i) * kM]);
        tmem_st16(taddr + 16 * blk, sv);
#pragma unroll
        for (uint32_t c = 0; c < 2; ++c)
            st_shared_v4(img + sw128(r, 2 * blk + c),
                         pack_bf16(__uint_as_float(sv[8 * c]), __uint_as_float(sv[8 * c + 1])),
                         pack_bf16(__uint_as_float(sv[8 * c + 2]), __uint_as_float(sv[8 * c + 3])),
                         pack_bf16(__uint_as_float(sv[8 * c + 4]), __uint_as_float(sv[8 * c + 5])),
                         pack_bf16(__uint_as_float(sv[8 * c + 6]), __uint_as_float(sv[8 * c + 7])));
    }
}

// Gated calls: as load_prefix_row, the fp32 state row times the chunk's decay d.
template <bool SCALED>
__device__ __noinline__ void load_prefix_row_scaled(const float* src, uint32_t taddr, uint32_t img, uint32_t r, float d) {
#pragma unroll 1
    for (int blk = 0; blk < 4; ++blk) {
        uint32_t sv[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) sv[i] = __float_as_uint(src[(size_t)(16 * blk + i) * kM]);
        if (SCALED) {
            uint32_t sd[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) sd[i] = __float_as_uint(__uint_as_float(sv[i]) * d);
            tmem_st16(taddr + 16 * blk, sd);
        } else {
            tmem_st16(taddr + 16 * blk, sv);
        }
#pragma unroll
        for (uint32_t c = 0; c < 2; ++c)
            st_shared_v4(img + sw128(r, 2 * blk + c),
                         pack_bf16(__uint_as_float(sv[8 * c]), __uint_as_float(sv[8 * c + 1])),
                         pack_bf16(__uint_as_float(sv[8 * c + 2]), __uint_as_float(sv[8 * c + 3])),
                         pack_bf16(__uint_as_float(sv[8 * c + 4]), __uint_as_float(sv[8 * c + 5])),
                         pack_bf16(__uint_as_float(sv[8 * c + 6]), __uint_as_float(sv[8 * c + 7])));
    }
}

// Output row `row` of a chunk: num (64 fp32 columns at taddr) / den as bf16,
// written into a [128][64] staging image in the 128-byte swizzled layout of
// the output tensor map (one TMA store per chunk writes it out; rows past L
// are clipped by the map).  32 columns at a time; `done` (the slot's release)
// is arrived once both blocks are in registers.
__device__ __noinline__ void out_row(uint32_t taddr, uint32_t stage, uint32_t row, float den, uint64_t* done) {
    const float inv = den != 0.f ? 1.f / den : 0.f;
#pragma unroll 1
    for (int blk = 0; blk < 2; ++blk) {
        uint32_t nv[32];
        tmem_ld32(taddr + 32 * blk, nv);
        tmem_ld_wait();
        if (blk == 1) {
            tc_fence_before();
            __syncwarp();
            if ((threadIdx.x & 31) == 0) mbar_arrive(done);
        }
#pragma unroll
        for (uint32_t c = 0; c < 4; ++c)
            st_shared_v4(stage + sw128(row, 4 * blk + c),
                         pack_bf16(__uint_as_float(nv[8 * c + 0]) * inv, __uint_as_float(nv[8 * c + 1]) * inv),
                         pack_bf16(__uint_as_float(nv[8 * c + 2]) * inv, __uint_as_float(nv[8 * c + 3]) * inv),
                         pack_bf16(__uint_as_float(nv[8 * c + 4]) * inv, __uint_as_float(nv[8 * c + 5]) * inv),
                         pack_bf16(__uint_as_float(nv[8 * c + 6]) * inv, __uint_as_float(nv[8 * c + 7]) * inv));
    }
}

// MMAs of the causal kernel (issued by one thread).
//   D[128 x 128] = X tile [128 rows][64] . omega rows [w0, w0+128) -- a projection of
//   128 rows (query rows of a Q tile, or transposed: features of omega against a K tile)
__device__ __forceinline__ void ca_project(uint32_t d, uint32_t a_tile, uint32_t b_tile) {
    const uint32_t id = make_idesc(128, 128, 0, 0);
    const uint64_t a0 = make_desc(a_tile, 16, 1024, SW_128B);
    const uint64_t b0 = make_desc(b_tile, 16, 1024, SW_128B);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) mma_ss(d, a0 + 2 * kk, b0 + 2 * kk, id, kk > 0 ? 1u : 0u);
}

template <int KIND, bool GATED = false>
__global__ void __launch_bounds__(kCausalThreads, 1)
k_tc_causal(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
            const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_w,
            const __grid_constant__ CUtensorMap tm_o, const float* __restrict__ kshift, const float* __restrict__ wmax,
            const float* __restrict__ prefix, const float* __restrict__ gate, int H, int L, float s, Ranges R,
            int* err) {
    constexpr bool POS = KIND == FAVOR_KERNEL_SOFTMAX_POS;
    constexpr bool TRIG = KIND == FAVOR_KERNEL_SOFTMAX_TRIG;
    constexpr bool KOFF = POS || TRIG;   // per-key terms from the K tile: offsets, or h(s k_j)
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1k(smem_raw);
    const uint32_t s_w = smem_u32(sm);
    const uint32_t s_q = s_w + kOmegaBytes;
    const uint32_t s_k = s_q + kTileBytes;
    const uint32_t s_v = s_k + kTileBytes;
    const uint32_t s_phi = s_v + kTileBytes;                  // Phi_K [256 features][128 tokens]: 2 blocks of 64 tokens
    const uint32_t s_st = s_phi + 4 * kPhiBlock;              // S~ [256 features][64], MN-major B operand
    const uint32_t s_stage = s_st + kSBytes;                  // output staging, 2 x [128][64] bf16 (1 KB aligned)
    const uint32_t s_cs = s_stage + 2 * kTileBytes;           // key offsets c_j, [2 chunk parities][128]
    const uint32_t s_z = s_cs + 2 * kTile * 4;                // z~ fp32 [2 chunk parities][256]
    const uint32_t s_zp = s_z + 2 * kM * 4;                   // key-warp z exchange [256]
    const uint32_t s_dsh = s_zp + kM * 4;                     // group A's den part per row [128]
    CaBars* bars = reinterpret_cast<CaBars*>(sm + (s_dsh - s_w) + kTile * 4);
    // gated calls, per chunk parity: C_i (cumulative log2 gate), T_j = C_j - log2(1 - g_j),
    // the keys' state weights 2^(C_last - C_j) (1 - g_j), then [2] chunk decays
    const uint32_t s_gr = (s_dsh + kTile * 4 + (uint32_t)sizeof(CaBars) + 15u) & ~15u;
    const uint32_t s_gt = s_gr + 2 * kTile * 4;
    const uint32_t s_gb = s_gt + 2 * kTile * 4;
    const int cta = blockIdx.x;
    const int g0 = cta * R.per, g1 = min(R.T, g0 + R.per);
    const int n = g1 - g0;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const float a = s * kLog2e;
    const float fa = TRIG ? s : a;   // the feature functions' scale of the projection
    const bool multi_head = H > 1;

    if (threadIdx.x == 0) {
        uint64_t* b = reinterpret_cast<uint64_t*>(bars);
        // order and arrival counts follow the fields of CaBars
        // (each barrier completes once per chunk -- pk_full twice, at parities 0 and 1 --
        // so a parity wait cannot miss a phase)
        const int counts[] = {1, 1, 1, 1, POS ? 9 : 1, KOFF ? 5 : 1, 1, 1,
                              1, 1, 4, 4, 1, 8, 4, 8,
                              1, 1, 4, 1, 8, 1, 1, 4,
                              8, 8, 1, 4, 1, 1,
                              1, 1, 8, 8};
        static_assert(sizeof(counts) / sizeof(int) * sizeof(uint64_t) == offsetof(CaBars, tmem_base), "barrier table");
        for (int i = 0; i < (int)(sizeof(counts) / sizeof(int)); ++i) mbar_init(b + i, counts[i]);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&bars->tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        // One thread keeps the Q, K and V streams independent: it polls each
        // stream's empty barrier and issues whichever next load is free.  It
        // also reloads omega at a head change, before the first Q tile of the
        // new head.  Gives up after about two seconds without progress, then
        // waits (bounded) for the loads it issued.
        if (lane == 0) {
            const CUtensorMap* maps[3] = {&tm_q, &tm_k, &tm_v};
            uint64_t* fulls[3] = {&bars->q_full, &bars->k_full, &bars->v_full};
            uint64_t* empties[3] = {&bars->q_empty, &bars->k_empty, &bars->v_empty};
            const uint32_t dsts[3] = {s_q - s_w, s_k - s_w, s_v - s_w};
            int next[3] = {0, 0, 0};
            int cur_h = -1, wloads = 0;
            uint32_t wph = 0;
            long long t0 = clock64();
            bool failed = false;
            while (next[0] < n || next[1] < n || next[2] < n) {
                bool progress = false;
#pragma unroll
                for (int sidx = 0; sidx < 3; ++sidx) {
                    const int t = next[sidx];
                    if (t >= n) continue;
                    if (t > 0 && !mbar_test_wait(empties[sidx], (t - 1) & 1)) continue;
                    const int g = g0 + t, bh = g / R.tph, h = bh % H, tok0 = (g % R.tph) * kTile;
                    if (sidx == 0 && h != cur_h) {
                        if (cur_h >= 0) {
                            if (!mbar_test_wait(&bars->w_empty, wph)) continue;
                            wph ^= 1;
                        }
                        mbar_expect_tx(&bars->w_full, kOmegaBytes);
                        tma_load_2d(sm, &tm_w, &bars->w_full, 0, h * kM);
                        cur_h = h;
                        ++wloads;
                    }
                    mbar_expect_tx(fulls[sidx], kTileBytes);
                    tma_load_3d(sm + dsts[sidx], maps[sidx], fulls[sidx], 0, tok0, bh);
                    next[sidx] = t + 1;
                    progress = true;
                }
                if (progress) {
                    t0 = clock64();
                } else {
                    __nanosleep(32);
                    if (clock64() - t0 > (4LL << 30)) {
                        atomicCAS(err, 0, 201);
                        failed = true;
                        break;
                    }
                }
            }
            if (failed) {
                // no copy may still be writing shared memory when the block exits
                for (int sidx = 0; sidx < 3; ++sidx)
                    if (next[sidx] > 0) mbar_wait_for(fulls[sidx], (next[sidx] - 1) & 1, nullptr, 0, 1LL << 28);
                if (wloads > 0) mbar_wait_for(&bars->w_full, (wloads - 1) & 1, nullptr, 0, 1LL << 28);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && n > 0) {
            const uint32_t id_a = make_idesc(128, 128, 0, 1);
            const uint32_t id_o = make_idesc(128, 64, 0, 1);
            const uint64_t bk = make_desc(s_phi, 2 * kPhiBlock, 1024, SW_128B);   // Phi_K, N = token (2 blocks)
            const uint64_t bs = make_desc(s_st, 8192, 1024, SW_128B);             // S~, N = value column
            const uint64_t bv = make_desc(s_v, 8192, 1024, SW_128B);              // V, N = value column
            uint32_t wph = 0;
            bool ok = true;
            int t = 0;
            // projections of chunk 0
            do {
                ok = mbar_wait(&bars->w_full, wph, err, 211) && mbar_wait(&bars->k_full, 0, err, 212);
                if (!ok) break;
                wph ^= 1;
                tc_fence_after();
                ca_project(tmem + ca_slot(2, 0), s_w, s_k);                    // P_K^T half 0 -> Z
                mma_commit(&bars->pk_full);
                if (!(ok = mbar_wait(&bars->q_full, 0, err, 213))) break;
                tc_fence_after();
                ca_project(tmem + ca_slot(0, 0), s_q, s_w);                    // P_Q half 0 -> X
                mma_commit(&bars->pq0_full);
                if (!(ok = mbar_wait(&bars->pk_free, 0, err, 214))) break;
                tc_fence_after();
                ca_project(tmem + ca_slot(2, 0), s_w + 128 * 128, s_k);        // P_K^T half 1 -> Z
                mma_commit(&bars->pk_full);
                mma_commit(&bars->k_empty);
                ca_project(tmem + ca_slot(1, 0), s_q, s_w + 128 * 128);        // P_Q half 1 -> Y
                mma_commit(&bars->pq1_full);
                mma_commit(&bars->q_empty);
                if (n > 1 && multi_head && (g0 + 1) % R.tph == 0) mma_commit(&bars->w_empty);
            } while (0);
            for (t = 0; t < n && ok; ++t) {
                const uint32_t ph = t & 1;
                const int r3 = t % 3, r3n = (t + 1) % 3;
                const uint32_t X = tmem + ca_slot(0, r3), Y = tmem + ca_slot(1, r3), Z = tmem + ca_slot(2, r3);
                const bool more = t + 1 < n;
                const bool new_w = more && multi_head && (g0 + t + 1) % R.tph == 0;
                const uint32_t Xn = tmem + ca_slot(0, r3n), Yn = tmem + ca_slot(1, r3n), Zn = tmem + ca_slot(2, r3n);
                // A = Phi_Q Phi_K^T, feature half 0 as soon as its query features are in, then half 1
                if (!(ok = mbar_wait(&bars->phiq0_full, ph, err, 221) && mbar_wait(&bars->phik_full, ph, err, 222))) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) mma_ts(Z, X + 8 * kk, bk + 128 * kk, id_a, kk > 0 ? 1u : 0u);
                if (!(ok = mbar_wait(&bars->phiq1_full, ph, err, 224))) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 8; kk < 16; ++kk) mma_ts(Z, Y + 8 * (kk - 8), bk + 128 * kk, id_a, 1u);
                mma_commit(&bars->a_full);
                // inter term num = Phi_Q S~(t) once the S~ / z~ image of this chunk is in (gated:
                // and the query groups have scaled Phi_Q by 2^C_i, now that A has read it)
                if (!(ok = mbar_wait(&bars->st_full, ph, err, 223))) break;
                if (GATED && !(ok = mbar_wait(&bars->phiq_scaled, ph, err, 233))) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) mma_ts(X + 64, X + 8 * kk, bs + 128 * kk, id_o, kk > 0 ? 1u : 0u);
#pragma unroll
                for (int kk = 8; kk < 16; ++kk) mma_ts(X + 64, Y + 8 * (kk - 8), bs + 128 * kk, id_o, 1u);
                mma_commit(&bars->ai_done);
                if (more) {
                    // key projection half 0 of chunk t+1 into Z' = Y (its last reader, the inter term, is issued)
                    if (new_w) {
                        if (!(ok = mbar_wait(&bars->w_full, wph, err, 226))) break;
                        wph ^= 1;
                    }
                    if (!(ok = mbar_wait(&bars->k_full, (t + 1) & 1, err, 227))) break;
                    tc_fence_after();
                    ca_project(Zn, s_w, s_k);
                    mma_commit(&bars->pk_full);
                }
                // state: S_h += Phi_K^T_h V (A = Phi_K rows of half h, K-major over tokens); the key
                // warps keep chunk t+1's features in registers until it has read Phi_K
                if (!(ok = mbar_wait(&bars->v_full, ph, err, 225))) break;
                // gated: the key warps have weighted Phi_K toward the chunk's end
                if (GATED && !(ok = mbar_wait(&bars->phik_w, ph, err, 234))) break;
                tc_fence_after();
#pragma unroll
                for (int hp = 0; hp < 2; ++hp) {
                    const uint64_t a0 = make_desc(s_phi + hp * 128 * 128, 16, 1024, SW_128B);
                    const uint32_t d = tmem + 384 + 64 * hp;
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_ss(d, a0 + (uint64_t)((((kk >> 2) * 2 * kPhiBlock) + (kk & 3) * 32) >> 4), bv + 128 * kk,
                               id_o, 1u);
                }
                mma_commit(&bars->s_full);
                mma_commit(&bars->phik_free);
                if (more) {
                    // key projection half 1 of t+1 once half 0's projections are in registers
                    if (!(ok = mbar_wait(&bars->pk_free, (t + 1) & 1, err, 230))) break;
                    tc_fence_after();
                    ca_project(Zn, s_w + 128 * 128, s_k);
                    mma_commit(&bars->pk_full);
                    mma_commit(&bars->k_empty);
                }
                // intra term: num += tril(A) V
                if (!(ok = mbar_wait(&bars->am_full, ph, err, 228))) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) mma_ts(X + 64, Z + 8 * kk, bv + 128 * kk, id_o, 1u);
                mma_commit(&bars->o_full);
                mma_commit(&bars->v_empty);
                if (more) {
                    // query projection half 0 of t+1 into X' = Z (tril(A) read above, mask read before am_full)
                    if (!(ok = mbar_wait(&bars->q_full, (t + 1) & 1, err, 229))) break;
                    tc_fence_after();
                    ca_project(Xn, s_q, s_w);
                    mma_commit(&bars->pq0_full);
                    // query projection half 1 of t+1 into Y' = X once the output has read num
                    if (!(ok = mbar_wait(&bars->o_empty, ph, err, 231))) break;
                    tc_fence_after();
                    ca_project(Yn, s_q, s_w + 128 * 128);
                    mma_commit(&bars->pq1_full);
                    mma_commit(&bars->q_empty);
                    if (t + 2 < n && multi_head && (g0 + t + 2) % R.tph == 0) mma_commit(&bars->w_empty);
                }
            }
            // every MMA issued has completed before tensor memory is freed
            mma_commit(&bars->mma_done);
            mbar_wait_for(&bars->mma_done, 0, ok ? err : nullptr, 232, ok ? (4LL << 30) : (1LL << 28));
        }
    } else if (warp < 10) {
        // ----------------------------------------------------------- query groups
        const bool grpA = warp < 6;
        const int q = warp & 3;
        const uint32_t row = 32 * q + lane;
        const uint32_t tl = tmem + ((uint32_t)(32 * q) << 16);
        float* dsh = reinterpret_cast<float*>(sm + (s_dsh - s_w));
        int wh = -1;
        float W = 0.f;
        for (int t = 0; t < n; ++t) {
            const uint32_t ph = t & 1;
            const int g = g0 + t, bh = g / R.tph, h = bh % H, tok0 = (g % R.tph) * kTile;
            const int r3 = t % 3;
            // row shift from the query norm (positive features)
            float c = 0.f;
            if (POS) {
                if (!mbar_wait(&bars->q_full, ph, err, 241)) break;
                if (h != wh) {
                    W = __ldg(wmax + h);
                    wh = h;
                }
                c = a * W * sqrtf(row_sqnorm(s_q, row));
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->q_empty);
            }
            if (!mbar_wait(&bars->z_full, ph, err, 242)) break;   // z~ of this chunk
            const uint32_t zt = s_z + ph * kM * 4;
            if (grpA) {
                if (!mbar_wait(&bars->pq0_full, ph, err, 243)) break;
                tc_fence_after();
                float dA;
                if constexpr (TRIG) dA = query_half_trig<KIND, false>(tl + ca_slot(0, r3), fa, c, zt);
                else dA = query_half<KIND>(tl + ca_slot(0, r3), a, c, zt);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->phiq0_full);
                // causal mask: keep key j <= query row, packed in place into Z[0,64)
                if (!mbar_wait(&bars->a_full, ph, err, 244)) break;
                tc_fence_after();
                float rs, ei = 1.f;
                if (GATED) {
                    // A has read Phi_Q: scale it by 2^C_i for the inter term, then the decayed mask
                    if (!mbar_wait(&bars->g_full[t & 1], (t >> 1) & 1, err, 247)) break;
                    const float ci = reinterpret_cast<const float*>(sm + (s_gr - s_w))[(t & 1) * kTile + row];
                    ei = exp2f(ci);
                    scale_packed_row(tl + ca_slot(0, r3), ei);
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars->phiq_scaled);
                    rs = mask_row_gated(tl + ca_slot(2, r3), (int)row, q, ci, s_gt + (t & 1) * kTile * 4);
                } else {
                    rs = mask_row(tl + ca_slot(2, r3), (int)row, q);
                }
                dsh[row] = ei * dA + rs;
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->am_full);
            } else {
                if (!mbar_wait(&bars->pq1_full, ph, err, 245)) break;
                tc_fence_after();
                float dB;
                if constexpr (TRIG) dB = query_half_trig<KIND, true>(tl + ca_slot(1, r3), fa, c, zt + 4 * 128);
                else dB = query_half<KIND>(tl + ca_slot(1, r3), a, c, zt + 4 * 128);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->phiq1_full);
                if (GATED) {
                    // once A has read Phi_Q: its half 1 times 2^C_i for the inter term
                    if (!mbar_wait(&bars->a_full, ph, err, 250)) break;
                    if (!mbar_wait(&bars->g_full[t & 1], (t >> 1) & 1, err, 247)) break;
                    tc_fence_after();
                    const float ei = exp2f(reinterpret_cast<const float*>(sm + (s_gr - s_w))[(t & 1) * kTile + row]);
                    scale_packed_row(tl + ca_slot(1, r3), ei);
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars->phiq_scaled);
                    dB *= ei;
                }
                // output rows: num / den, den = this half + group A's half and row sum
                if (!mbar_wait(&bars->o_full, ph, err, 246)) break;
                if (!mbar_wait(&bars->am_full, ph, err, 247)) break;   // dsh of this chunk is visible
                tc_fence_after();
                // num / den staged in shared memory, written by one TMA store (rows past L are clipped)
                if (t >= 2 && !mbar_wait(&bars->stage_free[ph], ((t >> 1) - 1) & 1, err, 248)) break;
                const uint32_t stage = s_stage + ph * kTileBytes;
                out_row(tl + ca_slot(0, r3) + 64, stage, row, dB + dsh[row], &bars->o_empty);
                fence_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->stage_full);
                if (warp == 6 && lane == 0) {
                    if (!mbar_wait(&bars->stage_full, ph, err, 249)) break;
                    tma_store_3d(&tm_o, stage, 0, tok0, bh);
                    bulk_commit();
                    bulk_wait_read<1>();   // the previous chunk's store has read its buffer
                    if (t >= 1) mbar_arrive(&bars->stage_free[ph ^ 1]);
                }
            }
        }
    } else {
        // ------------------------------------------------------------- key warps
        // lane quarter q = warp % 4.  Warps 10..13 (u = 0): tokens [0,64) of the tile,
        // features r0 = 32q + lane (half 0) and r0 + 128 (half 1); warps 14..17 (u = 1):
        // tokens [64,128).  The u = 0 warps compute the key offsets and own row r0 of
        // S~ / z~, the u = 1 warps row r0 + 128.  Per chunk t: the key features of t
        // (held in registers until the state update of t-1 has read Phi_K), then the
        // S~ refresh of t (the inter term of t waits for it, the state update of t
        // follows that), then z~ of t+1 for the query groups.
        const int q = warp & 3, u = (warp - 10) >> 2;
        const uint32_t r0 = 32 * q + lane;
        const uint32_t rown = r0 + 128 * (uint32_t)u;        // the state row this thread owns
        const uint32_t tl = tmem + ((uint32_t)(32 * q) << 16);
        float* zs = reinterpret_cast<float*>(sm + (s_z - s_w));
        float* zp = reinterpret_cast<float*>(sm + (s_zp - s_w));
        float* cs = reinterpret_cast<float*>(sm + (s_cs - s_w));
        float zpre = 0.f;           // z of the piece's prefix for row rown
        float zr[2] = {0.f, 0.f};   // this thread's running sums over its tokens, rows r0 and r0 + 128
        int cur_bh = -1, kap_h = -1, nzx = 0;
        float kap = 0.f;
        bool ok = true;
        // gated calls: warp 10 scans each chunk's gates, four tokens per lane; the
        // next chunk's gates are loaded a chunk ahead
        const bool scanner = GATED && warp == 10;
        float4 gnext = make_float4(1.f, 1.f, 1.f, 1.f);
        auto load_gates = [&](int tt) {
            const int gg = g0 + tt, bb = gg / R.tph, tk = (gg % R.tph) * kTile + 4 * lane;
            float v[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) v[e] = tk + e < L ? __ldg(gate + (size_t)bb * L + tk + e) : 1.f;
            return make_float4(v[0], v[1], v[2], v[3]);
        };
        if (scanner && n > 0) gnext = load_gates(0);
        float* gflt = reinterpret_cast<float*>(sm + (s_gr - s_w));   // C_i | T_j | weights | decays, by parity
        for (int t = 0; t < n && ok; ++t) {
            const uint32_t ph = t & 1;
            const int g = g0 + t, bh = g / R.tph, h = bh % H, tok0 = (g % R.tph) * kTile;
            const int r3 = t % 3;
            const uint32_t Z = tl + ca_slot(2, r3);
            if (scanner) {
                // this chunk's cumulative log2 gates C_i (gates clamped below at 2^-126; past L a
                // gate of 1 with weight 0), T_j = C_j - log2(1 - g_j), the keys' state weights
                // 2^(C_last - C_j) (1 - g_j) and the chunk decay 2^C_last
                const float4 g4 = gnext;
                if (t + 1 < n) gnext = load_gates(t + 1);
                const float gv[4] = {g4.x, g4.y, g4.z, g4.w};
                float c[4], acc = 0.f;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    acc += log2f(fmaxf(gv[e], 1.17549435e-38f));
                    c[e] = acc;
                }
                float off = acc;   // inclusive scan of the lanes' sums
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float x = __shfl_up_sync(0xffffffffu, off, o);
                    if (lane >= o) off += x;
                }
                const float total = __shfl_sync(0xffffffffu, off, 31);
                off -= acc;   // exclusive
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int tok = 4 * lane + e;
                    const float ci = c[e] + off, om = 1.f - gv[e];
                    gflt[ph * kTile + tok] = ci;
                    gflt[2 * kTile + ph * kTile + tok] = om > 0.f ? ci - log2f(om) : 1.0e30f;
                    gflt[4 * kTile + ph * kTile + tok] = om > 0.f ? exp2f(total - ci) * om : 0.f;
                }
                if (lane == 0) gflt[6 * kTile + ph] = exp2f(total);
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->g_full[ph]);
            }
            float gdec = 1.f;   // the chunk's decay of the carried state (gated calls)
            if (GATED) {
                if (!(ok = mbar_wait(&bars->g_full[ph], (t >> 1) & 1, err, 261))) break;
                gdec = gflt[6 * kTile + ph];
            }
            // key offsets of this chunk (tokens 32q + lane), in cs[t & 1]: exponent offsets
            // (positive features) or the factors h(s k_j) (trigonometric)
            if (KOFF && u == 0) {
                if (!(ok = mbar_wait(&bars->k_full, ph, err, 251))) break;
                if (h != kap_h) {
                    kap = __ldg(kshift + h);
                    kap_h = h;
                }
                const float nrm = row_sqnorm(s_k, r0);
                if constexpr (TRIG)
                    cs[ph * kTile + r0] = (tok0 + (int)r0 < L) ? expf(0.5f * s * s * nrm) : 0.f;
                else
                    cs[ph * kTile + r0] = (tok0 + (int)r0 < L) ? -(0.5f * s * s * nrm + kap) * kLog2e : -1.0e30f;
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&bars->k_empty);
                    mbar_arrive(&bars->cs_full);
                }
            }
            const bool piece_start = bh != cur_bh;
            if (piece_start) {
                // the piece's prefix: fp32 state row and S~ image row, z~ of this chunk
                if (t > 0) {
                    ok = mbar_wait(&bars->s_full, ph ^ 1, err, 252) && mbar_wait(&bars->ai_done, ph ^ 1, err, 253);
                    if (!ok) break;
                    tc_fence_after();
                }
                const float* pre = prefix + ((size_t)bh * R.pstride + (cta - first_cta(R, bh))) * (kM * (kDV + 1));
                if constexpr (GATED) load_prefix_row_scaled<true>(pre + rown, tl + 384 + 64 * u, s_st, rown, gdec);
                else load_prefix_row(pre + rown, tl + 384 + 64 * u, s_st, rown);
                zpre = pre[(size_t)64 * kM + rown];
                zr[0] = zr[1] = 0.f;
                zs[ph * kM + rown] = zpre;
                tmem_st_wait();
                fence_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&bars->st_full);
                    mbar_arrive(&bars->z_full);
                }
                cur_bh = bh;
            }
            // key features, half 0 then half 1, of this warp's 64 tokens
            float zc[2];
#pragma unroll 1
            for (int hp = 0; hp < 2; ++hp) {
                if (!(ok = mbar_wait(&bars->pk_full, (uint32_t)hp, err, 255 + hp))) break;
                if (hp == 0 && KOFF && !(ok = mbar_wait(&bars->cs_full, ph, err, 257))) break;
                tc_fence_after();
                // half 0's projections go to registers first (then the slot may take half 1);
                // stores into Phi_K wait until the state update of t-1 has read it
                if constexpr (TRIG) {
                    const uint32_t kt = Z + 64 * (uint32_t)u, kphi = s_phi + (uint32_t)u * 2 * kPhiBlock;
                    const uint32_t kcs = s_cs + (ph * kTile + 64 * (uint32_t)u) * 4, kr = r0 + 128 * (uint32_t)hp;
                    uint64_t* krel = hp == 0 ? &bars->pk_free : nullptr;
                    uint64_t* kgate = (hp == 0 && t > 0) ? &bars->phik_free : nullptr;
                    zc[hp] = hp == 1 ? key_half_row_trig<KIND, true>(kt, krel, kgate, ph ^ 1, err, &ok, kphi, kr, fa, kcs)
                                     : key_half_row_trig<KIND, false>(kt, krel, kgate, ph ^ 1, err, &ok, kphi, kr, fa, kcs);
                } else {
                    zc[hp] = key_half_row<KIND>(Z + 64 * (uint32_t)u, hp == 0 ? &bars->pk_free : nullptr,
                                                (hp == 0 && t > 0) ? &bars->phik_free : nullptr, ph ^ 1, err, &ok,
                                                s_phi + (uint32_t)u * 2 * kPhiBlock, r0 + 128 * (uint32_t)hp, a,
                                                s_cs + (ph * kTile + 64 * (uint32_t)u) * 4);
                }
                if (!ok) break;
            }
            if (!ok) break;
            if (!GATED) {
                zr[0] += zc[0];
                zr[1] += zc[1];
            }
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->phik_full);
            // S~ image of this chunk from the running state S(t) (after the state update of t-1;
            // the inter term of t-1 has read the previous image)
            if (!piece_start) {
                ok = mbar_wait(&bars->s_full, ph ^ 1, err, 252) && mbar_wait(&bars->ai_done, ph ^ 1, err, 253);
                if (!ok) break;
                tc_fence_after();
                if (GATED) {
                    // the image of S(t-1) for the inter term, and S(t-1) times the chunk's decay
                    // for the state update of t to accumulate onto
                    refresh_decay_row(tl + 384 + 64 * u, s_st, rown, gdec);
                    tmem_st_wait();
                } else {
                    refresh_row(tl + 384 + 64 * u, s_st, rown);
                }
                fence_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->st_full);
            }
            if (GATED) {
                // once A has read Phi_K: weight this thread's two rows of it by the keys' state
                // weights (the state update reads them next); the running sums decay the same way
                if (!(ok = mbar_wait(&bars->a_full, ph, err, 262))) break;
                const uint32_t wcol = s_gr + (4 * kTile + ph * kTile + 64 * (uint32_t)u) * 4;
                const uint32_t phi = s_phi + (uint32_t)u * 2 * kPhiBlock;
                const float zw0 = weight_phik_row(phi, r0, wcol);
                const float zw1 = weight_phik_row(phi, r0 + 128, wcol);
                fence_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->phik_w);
                zr[0] = fmaf(gdec, zr[0], zw0);
                zr[1] = fmaf(gdec, zr[1], zw1);
                zpre *= gdec;
            }
            // z~ of chunk t+1 (same piece): this thread's sums plus the partner warp's for row rown
            if (t + 1 < n && (g + 1) / R.tph == bh) {
                // both query groups are past their wait for z~ of t (A(t) needed their features),
                // so the next phase of z_full cannot be mistaken for this one
                if (!(ok = mbar_wait(&bars->a_full, ph, err, 260))) break;
                zp[r0 + 128 * (uint32_t)(1 - u)] = zr[1 - u];
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->zx_full);
                if (!(ok = mbar_wait(&bars->zx_full, (uint32_t)(nzx & 1), err, 259))) break;
                ++nzx;
                zs[(ph ^ 1) * kM + rown] = zpre + zr[u] + zp[rown];
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->z_full);
            }
        }
    }
    if (threadIdx.x == 6 * 32) bulk_wait<0>();   // output stores complete before exit
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, 512);
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

// ======================================================== bounded-wait check
// One thread waits on an mbarrier phase that nothing completes, with a limit
// of `limit` cycles: the wait must give up, write `code` to the error word and
// return.  No copies, tensor memory or other warps are involved.
__global__ void k_wait_expiry(int* err, long long limit, int code) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait_for(&bar, 0, err, code, limit);
}

// ================================================================ host side
constexpr size_t kSmemState = 1024 + kOmegaBytes + kNS * 2 * kTileBytes + kNS * kExtStage + kExtOmega + sizeof(StBars);
constexpr size_t kSmemReadout = 1024 + kOmegaBytes + kRStages * kTileBytes + kRImage + 2 * kTileBytes +
                                 2 * 4 * kTile * 4 + sizeof(RdBars);
constexpr size_t kSmemCausal = 1024 + kOmegaBytes + 3 * kTileBytes + 4 * kPhiBlock + kSBytes + 2 * kTileBytes + 2 * kTile * 4 +
                                3 * kM * 4 + kTile * 4 + sizeof(CaBars) + 16 + 6 * kTile * 4 + 64;
static_assert(kSmemCausal <= 232448, "causal shared memory");
constexpr size_t kSmemFmap = 1024 + kOmegaBytes + kTileBytes + 64;

void allow_all_once() {
    static std::once_flag once;
    std::call_once(once, [] {
        allow_smem(k_tc_state<FAVOR_KERNEL_SOFTMAX_POS>, kSmemState);
        allow_smem(k_tc_state<FAVOR_KERNEL_RELU>, kSmemState);
        allow_smem(k_tc_state<FAVOR_KERNEL_SOFTMAX_TRIG>, kSmemState);
        allow_smem(k_tc_state<FAVOR_KERNEL_SOFTMAX_POS, true>, kSmemState);
        allow_smem(k_tc_state<FAVOR_KERNEL_RELU, true>, kSmemState);
        allow_smem(k_tc_readout<FAVOR_KERNEL_SOFTMAX_POS>, kSmemReadout);
        allow_smem(k_tc_readout<FAVOR_KERNEL_RELU>, kSmemReadout);
        allow_smem(k_tc_readout<FAVOR_KERNEL_SOFTMAX_TRIG>, kSmemReadout);
        allow_smem(k_tc_causal<FAVOR_KERNEL_SOFTMAX_POS>, kSmemCausal);
        allow_smem(k_tc_causal<FAVOR_KERNEL_RELU>, kSmemCausal);
        allow_smem(k_tc_causal<FAVOR_KERNEL_SOFTMAX_TRIG>, kSmemCausal);
        allow_smem(k_tc_causal<FAVOR_KERNEL_SOFTMAX_POS, true>, kSmemCausal);
        allow_smem(k_tc_causal<FAVOR_KERNEL_RELU, true>, kSmemCausal);
        allow_smem(k_tc_feature_map<FAVOR_KERNEL_SOFTMAX_POS>, kSmemFmap);
        allow_smem(k_tc_feature_map<FAVOR_KERNEL_RELU>, kSmemFmap);
        cudaGetLastError();
    });
}

// wlog: null, or the gated call's per-token log2 key weights (k_gate_weights).
favor_status launch_state(const Handle& h, const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mw,
                          int BH, int L, const Ranges& R, cudaStream_t st, const float* wlog = nullptr) {
    if ((size_t)BH * R.pstride > h.ws_partial_rows)
        return set_error(FAVOR_ERR_INVALID_ARG, "state workspace too small (%d x %d rows)", BH, R.pstride);
    ProfScope ps(h, PROF_STATE, st);
    const dim3 g(R.G), b(kStateThreads);
    if (wlog && h.kind == FAVOR_KERNEL_SOFTMAX_POS)
        k_tc_state<FAVOR_KERNEL_SOFTMAX_POS, true><<<g, b, kSmemState, st>>>(mk, mv, mw, h.kshift, wlog, h.ws_partial,
                                                                            h.H, L, h.s, R, h.dev_err);
    else if (wlog)
        k_tc_state<FAVOR_KERNEL_RELU, true><<<g, b, kSmemState, st>>>(mk, mv, mw, h.kshift, wlog, h.ws_partial, h.H, L,
                                                                     h.s, R, h.dev_err);
    else if (h.kind == FAVOR_KERNEL_SOFTMAX_POS)
        k_tc_state<FAVOR_KERNEL_SOFTMAX_POS><<<g, b, kSmemState, st>>>(mk, mv, mw, h.kshift, nullptr, h.ws_partial,
                                                                      h.H, L, h.s, R, h.dev_err);
    else if (h.kind == FAVOR_KERNEL_SOFTMAX_TRIG)
        k_tc_state<FAVOR_KERNEL_SOFTMAX_TRIG><<<g, b, kSmemState, st>>>(mk, mv, mw, h.kshift, nullptr, h.ws_partial,
                                                                       h.H, L, h.s, R, h.dev_err);
    else
        k_tc_state<FAVOR_KERNEL_RELU><<<g, b, kSmemState, st>>>(mk, mv, mw, h.kshift, nullptr, h.ws_partial, h.H, L,
                                                               h.s, R, h.dev_err);
    count_launch();
    return check_launch("tensor-core state kernel");
}

}  // namespace

favor_status launch_wait_expiry(const Handle& h, long long limit, int code, cudaStream_t st) {
    k_wait_expiry<<<1, 32, 0, st>>>(h.dev_err, limit, code);
    count_launch();
    return check_launch("bounded-wait check kernel");
}

bool tc_supported(const Handle& h) {
    return h.dtype == FAVOR_DTYPE_BF16 && h.d == kD && h.dv == kDV && h.m == kM && h.cc_major >= 10 &&
           encode_fn() != nullptr;
}

favor_status tc_feature_map(const Handle& h, const void* x, void* phi, int B, int L, cudaStream_t st) {
    // the plain trigonometric map (with h(x)) stays on the CUDA cores
    if (!aligned16(x) || !aligned16(phi) || h.kind == FAVOR_KERNEL_SOFTMAX_TRIG)
        return simt_feature_map(h, x, phi, B, L, st);
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
    Ranges R = plan_ranges(BH, L, h.num_sms);
    CUtensorMap mq, mk, mv, mw;
    if (!map_tokens(&mq, q, BH, L) || !map_tokens(&mk, k, BH, L) || !map_tokens(&mv, v, BH, L) ||
        !map_omega(&mw, h.omega_bf16, h.H))
        return set_error(FAVOR_ERR_CUDA, "cuTensorMapEncodeTiled failed");
    favor_status s = launch_state(h, mk, mv, mw, BH, L, R, st);
    if (s != FAVOR_OK) return s;
    {
        dim3 grid((kM * (kDV + 1) + 255) / 256, BH);
        ProfScope ps(h, PROF_COMBINE, st);
        k_reduce_pack<<<grid, 256, 0, st>>>(h.ws_partial, (uint8_t*)h.ws_tc, R);
        count_launch();
        s = check_launch("reduce/pack kernel");
        if (s != FAVOR_OK) return s;
    }
    CUtensorMap mo;
    if (!map_tokens(&mo, out, BH, L)) return set_error(FAVOR_ERR_CUDA, "cuTensorMapEncodeTiled failed");
    ProfScope ps(h, PROF_READOUT, st);
    if (h.kind == FAVOR_KERNEL_SOFTMAX_POS)
        k_tc_readout<FAVOR_KERNEL_SOFTMAX_POS><<<R.G, kReadoutThreads, kSmemReadout, st>>>(
            mq, mw, mo, (const uint8_t*)h.ws_tc, h.H, L, h.s, R, h.dev_err);
    else if (h.kind == FAVOR_KERNEL_SOFTMAX_TRIG)
        k_tc_readout<FAVOR_KERNEL_SOFTMAX_TRIG><<<R.G, kReadoutThreads, kSmemReadout, st>>>(
            mq, mw, mo, (const uint8_t*)h.ws_tc, h.H, L, h.s, R, h.dev_err);
    else
        k_tc_readout<FAVOR_KERNEL_RELU><<<R.G, kReadoutThreads, kSmemReadout, st>>>(
            mq, mw, mo, (const uint8_t*)h.ws_tc, h.H, L, h.s, R, h.dev_err);
    count_launch();
    return check_launch("tensor-core readout kernel");
}

favor_status tc_causal(const Handle& h, const void* q, const void* k, const void* v, void* out, int B, int L,
                       cudaStream_t st) {
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
        return simt_causal(h, q, k, v, out, B, L, st);
    allow_all_once();
    const int BH = B * h.H;
    Ranges R = plan_ranges(BH, L, h.num_sms);
    CUtensorMap mq, mk, mv, mw, mo;
    if (!map_tokens(&mq, q, BH, L) || !map_tokens(&mk, k, BH, L) || !map_tokens(&mv, v, BH, L) ||
        !map_tokens(&mo, out, BH, L) || !map_omega(&mw, h.omega_bf16, h.H))
        return set_error(FAVOR_ERR_CUDA, "cuTensorMapEncodeTiled failed");
    favor_status s;
    if (R.pstride > 1) {
        s = launch_state(h, mk, mv, mw, BH, L, R, st);
        if (s != FAVOR_OK) return s;
        dim3 g2((kM * (kDV + 1) / 4 + 255) / 256, BH);
        ProfScope ps(h, PROF_COMBINE, st);
        k_scan_pieces<<<g2, 256, 0, st>>>(h.ws_partial, R);
        count_launch();
        s = check_launch("piece scan kernel");
    } else {
        s = cudaMemsetAsync(h.ws_partial, 0, (size_t)BH * kM * (kDV + 1) * sizeof(float), st) == cudaSuccess
                ? FAVOR_OK
                : set_error(FAVOR_ERR_CUDA, "cudaMemsetAsync failed");
    }
    if (s != FAVOR_OK) return s;
    ProfScope ps(h, PROF_CAUSAL, st);
    if (h.kind == FAVOR_KERNEL_SOFTMAX_POS)
        k_tc_causal<FAVOR_KERNEL_SOFTMAX_POS><<<R.G, kCausalThreads, kSmemCausal, st>>>(
            mq, mk, mv, mw, mo, h.kshift, h.omega_wmax, h.ws_partial, nullptr, h.H, L, h.s, R, h.dev_err);
    else if (h.kind == FAVOR_KERNEL_SOFTMAX_TRIG)
        k_tc_causal<FAVOR_KERNEL_SOFTMAX_TRIG><<<R.G, kCausalThreads, kSmemCausal, st>>>(
            mq, mk, mv, mw, mo, h.kshift, h.omega_wmax, h.ws_partial, nullptr, h.H, L, h.s, R, h.dev_err);
    else
        k_tc_causal<FAVOR_KERNEL_RELU><<<R.G, kCausalThreads, kSmemCausal, st>>>(
            mq, mk, mv, mw, mo, h.kshift, h.omega_wmax, h.ws_partial, nullptr, h.H, L, h.s, R, h.dev_err);
    count_launch();
    return check_launch("tensor-core causal kernel");
}

// RFA-Gate causal attention on the tensor cores (positive and ReLU features):
// per-token key weights toward each piece's end and the pieces' decays, the
// weighted piece states, their decayed prefix, then the gated chunk kernel.
favor_status tc_causal_gated(const Handle& h, const void* q, const void* k, const void* v, const float* gate, void* out,
                             int B, int L, cudaStream_t st) {
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
        return simt_causal(h, q, k, v, out, B, L, st, gate);
    allow_all_once();
    const int BH = B * h.H;
    Ranges R = plan_ranges(BH, L, h.num_sms);
    CUtensorMap mq, mk, mv, mw, mo;
    if (!map_tokens(&mq, q, BH, L) || !map_tokens(&mk, k, BH, L) || !map_tokens(&mv, v, BH, L) ||
        !map_tokens(&mo, out, BH, L) || !map_omega(&mw, h.omega_bf16, h.H))
        return set_error(FAVOR_ERR_CUDA, "cuTensorMapEncodeTiled failed");
    favor_status s;
    if (R.pstride > 1) {
        {
            ProfScope ps(h, PROF_COMBINE, st);
            // the per-token log2 weights fit the causal backward's row statistics buffer
            k_gate_weights<<<R.G, 128, 0, st>>>(gate, h.ws_rowstat, h.ws_segdecay, L, R);
            count_launch();
            s = check_launch("gate weights kernel");
            if (s != FAVOR_OK) return s;
        }
        s = launch_state(h, mk, mv, mw, BH, L, R, st, h.ws_rowstat);
        if (s != FAVOR_OK) return s;
        dim3 g2((kM * (kDV + 1) + 255) / 256, BH);
        ProfScope ps(h, PROF_COMBINE, st);
        k_scan_pieces_decay<<<g2, 256, 0, st>>>(h.ws_partial, h.ws_segdecay, R);
        count_launch();
        s = check_launch("decayed piece scan kernel");
    } else {
        s = cudaMemsetAsync(h.ws_partial, 0, (size_t)BH * kM * (kDV + 1) * sizeof(float), st) == cudaSuccess
                ? FAVOR_OK
                : set_error(FAVOR_ERR_CUDA, "cudaMemsetAsync failed");
    }
    if (s != FAVOR_OK) return s;
    ProfScope ps(h, PROF_CAUSAL, st);
    if (h.kind == FAVOR_KERNEL_SOFTMAX_POS)
        k_tc_causal<FAVOR_KERNEL_SOFTMAX_POS, true><<<R.G, kCausalThreads, kSmemCausal, st>>>(
            mq, mk, mv, mw, mo, h.kshift, h.omega_wmax, h.ws_partial, gate, h.H, L, h.s, R, h.dev_err);
    else
        k_tc_causal<FAVOR_KERNEL_RELU, true><<<R.G, kCausalThreads, kSmemCausal, st>>>(
            mq, mk, mv, mw, mo, h.kshift, h.omega_wmax, h.ws_partial, gate, h.H, L, h.s, R, h.dev_err);
    count_launch();
    return check_launch("tensor-core gated causal kernel");
}

favor_status tc_kv_state(const Handle& h, const void* k, const void* v, float* state, int B, int L, cudaStream_t st) {
    if (!aligned16(k) || !aligned16(v)) return simt_kv_state(h, k, v, state, B, L, st);
    allow_all_once();
    const int BH = B * h.H;
    Ranges R = plan_ranges(BH, L, h.num_sms);
    CUtensorMap mk, mv, mw;
    if (!map_tokens(&mk, k, BH, L) || !map_tokens(&mv, v, BH, L) || !map_omega(&mw, h.omega_bf16, h.H))
        return set_error(FAVOR_ERR_CUDA, "cuTensorMapEncodeTiled failed");
    favor_status s = launch_state(h, mk, mv, mw, BH, L, R, st);
    if (s != FAVOR_OK) return s;
    // the state kernel leaves out m^-1/2 (trigonometric: (m/2)^-1/2), and its ReLU
    // features are of k, not s*k
    const float scale = (h.kind == FAVOR_KERNEL_RELU ? h.s : 1.f) /
                        sqrtf((float)(h.kind == FAVOR_KERNEL_SOFTMAX_TRIG ? kM / 2 : kM));
    dim3 grid((kM * (kDV + 1) + 255) / 256, BH);
    ProfScope ps(h, PROF_COMBINE, st);
    k_accum_cols<<<grid, 256, 0, st>>>(h.ws_partial, state, R, scale);
    count_launch();
    return check_launch("state accumulate kernel");
}

favor_status tc_attn_from_state(const Handle& h, const void* q, const float* state, void* out, int B, int L,
                                cudaStream_t st) {
    if (!aligned16(q) || !aligned16(out)) return simt_attn_from_state(h, q, state, out, B, L, st);
    allow_all_once();
    const int BH = B * h.H;
    Ranges R = plan_ranges(BH, L, h.num_sms);
    CUtensorMap mq, mw, mo;
    if (!map_tokens(&mq, q, BH, L) || !map_tokens(&mo, out, BH, L) || !map_omega(&mw, h.omega_bf16, h.H))
        return set_error(FAVOR_ERR_CUDA, "cuTensorMapEncodeTiled failed");
    {
        dim3 grid((kM * (kDV + 1) + 255) / 256, BH);
        ProfScope ps(h, PROF_COMBINE, st);
        k_pack_state<<<grid, 256, 0, st>>>(state, (uint8_t*)h.ws_tc);
        count_launch();
        favor_status s = check_launch("state pack kernel");
        if (s != FAVOR_OK) return s;
    }
    ProfScope ps(h, PROF_READOUT, st);
    if (h.kind == FAVOR_KERNEL_SOFTMAX_POS)
        k_tc_readout<FAVOR_KERNEL_SOFTMAX_POS><<<R.G, kReadoutThreads, kSmemReadout, st>>>(
            mq, mw, mo, (const uint8_t*)h.ws_tc, h.H, L, h.s, R, h.dev_err);
    else if (h.kind == FAVOR_KERNEL_SOFTMAX_TRIG)
        k_tc_readout<FAVOR_KERNEL_SOFTMAX_TRIG><<<R.G, kReadoutThreads, kSmemReadout, st>>>(
            mq, mw, mo, (const uint8_t*)h.ws_tc, h.H, L, h.s, R, h.dev_err);
    else
        k_tc_readout<FAVOR_KERNEL_RELU><<<R.G, kReadoutThreads, kSmemReadout, st>>>(
            mq, mw, mo, (const uint8_t*)h.ws_tc, h.H, L, h.s, R, h.dev_err);
    count_launch();
    return check_launch("tensor-core readout kernel");
}

}  // namespace favor
