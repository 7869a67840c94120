// Bifocal causal GQA prefill attention: TMA + tcgen05 (TMEM accumulators).
//
// What it computes (Jet-Long: "local RoPE-faithful window" + "long-range
// window" merged by inclusion-exclusion, abstract and ResearchPod transcript
// on the prefill phase): for query i and key j <= i,
//   score = tau <q_i, k_j>                          if i - j < w   (exact RoPE)
//   score = tau <R_{delta_i} q_i, R_{delta_j} k_j>  if i - j >= w  (aliased)
// and one softmax over all keys -- which is what local(window) + remote(all)
// - remote(window) on log-sum-exp statistics equals.  The aliased view is an
// on-the-fly correction rotation of the exact-RoPE q/k held in shared memory.
//
// One CTA owns a 128-row query tile of one head and walks its key tiles
// 0..diagonal.  A per-tile classifier picks the view: exact tiles run Q.K^T,
// remote tiles run Qg.Kg^T on the K tile corrected in place, band tiles (the
// ones the window edge crosses) run both and select per element.
//
// Warp roles (320 threads):
//   warp 0      TMA producer (Q once, K/V tiles through an NS-stage ring)
//   warp 1      TMEM allocator + single-thread tcgen05.mma issuer
//   warps 2-5   softmax (one query row per thread, TMEM lane = row) + epilogue
//   warps 6-9   correction: Qg once, then every remote/band K tile in place
// TMEM (512 columns): S0 [0,128), S1 [128,256), O [256, 256+D).
// Shared memory: Q, Qg (SW128, two 64-column boxes when D = 128), NS K and V
// stages, one P tile (bf16, SW128 K-major) -- all 1024-byte aligned.
#include <math.h>
#include <stdio.h>

#include "jl_common.cuh"
#include "sm100_ptx.cuh"
#include "tile_class.cuh"

namespace {

using namespace jl::ptx;

constexpr int kBM = 128, kBN = 128;
constexpr int kThreads = 320;
constexpr float kLn2 = 0.6931471805599453f;
// Lazy rescaling: the running maximum used as the exponent offset is moved
// only when a row's maximum grows by more than this (log2 units), so P stays
// <= 2^8 and O is rarely rescaled in TMEM.
constexpr float kRescaleThreshold = 8.0f;

template <int D>
struct Cfg {
    static constexpr int NS = (D == 128) ? 2 : 3;
    static constexpr int REGION = kBM * 64 * 2;  // one 128-row x 64-column bf16 box: 16 KB
    static constexpr int NREG = D / 64;          // boxes per 128-row tile
    static constexpr int TILE = kBM * D * 2;     // Q / K / V tile bytes
    static constexpr int PBYTES = kBM * kBN * 2; // P tile bytes
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_QG = OFF_Q + TILE;
    static constexpr int OFF_K = OFF_QG + TILE;
    static constexpr int OFF_V = OFF_K + NS * TILE;
    static constexpr int OFF_P = OFF_V + NS * TILE;
    static constexpr int OFF_BAR = OFF_P + PBYTES;
    static constexpr int BAR_BYTES = 256;
    static constexpr int SMEM = OFF_BAR + BAR_BYTES + 1024;  // + alignment slack
    // barrier indices
    static constexpr int B_QFULL = 0, B_QGFULL = 1, B_KFULL = 2, B_VFULL = 2 + NS,
                         B_KVEMPTY = 2 + 2 * NS, B_KGFULL = 2 + 3 * NS, B_SEDONE = 2 + 4 * NS,
                         B_SFULL = 3 + 4 * NS, B_SEMPTY = 5 + 4 * NS, B_PFULL = 7 + 4 * NS,
                         B_ODONE = 8 + 4 * NS, B_DRAIN = 9 + 4 * NS, NBAR = 10 + 4 * NS;
    static_assert(NBAR * 8 <= 192, "barrier area");
    static_assert(SMEM <= 232448, "shared memory budget");
};

struct Params {
    __nv_bfloat16 *out;  // [B, S, Hq, D]
    float *lse;          // [B, Hq, S]
    int *status;
    int B, Hq, Hkv, S, w, g, grp, n_qtiles;
    float scale_log2;    // tau * log2(e)
};

// Byte offset of 16-byte chunk `cc` of row `n` inside a 128-byte-swizzled box.
__device__ __forceinline__ uint32_t sw128(int n, int cc)
{
    return (uint32_t)(n * 128 + ((cc ^ (n & 7)) << 4));
}

// Rotate rows of a 128-row bf16 tile (SW128 boxes) from src to dst by
// delta_p, p = p0 + row, for the pairs this thread owns, writing fp16: the
// corrected operands feed a kind::f16 MMA with fp16 A and B, whose 11-bit
// significand keeps the rounding of the aliased view ~8x below bf16's (the
// rotation preserves each pair's norm, so |x| < 46000 stays finite).  Thread t of the 128-thread
// group owns chunk pair c = t % CPR (pairs d = 8c..8c+7) and rows
// n0 + RPS*k.  Angles: exact fixed-point phase at the first row, then a
// recurrence of unit complex steps (delta moves by one of two constants per
// RPS rows).
template <int D>
struct Corrector {
    static constexpr int CPR = D / 16;       // chunk pairs per row
    static constexpr int RPS = 128 / CPR;    // rows per step
    static constexpr int STEPS = 128 / RPS;  // rows per thread
    int c, n0, g, rs;
    float ac[8], as_[8], bc[8], bs_[8];      // step rotations A, B
    unsigned long long F[8];

    __device__ void init(int t, int g_, const jl::PhaseTable &pt)
    {
        c = t % CPR;
        n0 = t / CPR;
        g = g_;
        const int qs = RPS / g;
        rs = RPS % g;
#pragma unroll
        for (int e = 0; e < 8; e++) {
            F[e] = pt.f[8 * c + e];
            jl::phase_sincos(qs - RPS, F[e], &as_[e], &ac[e]);
            jl::phase_sincos(qs + 1 - RPS, F[e], &bs_[e], &bc[e]);
        }
    }

    __device__ void run(uint32_t src, uint32_t dst, int p0) const
    {
        constexpr uint32_t REGION = Cfg<D>::REGION;
        float zc[8], zs[8];
        int p = p0 + n0;
        const int dp = jl::delta_pos(p, g);
#pragma unroll
        for (int e = 0; e < 8; e++) jl::phase_sincos(dp, F[e], &zs[e], &zc[e]);
        int jm = p % g;
#pragma unroll
        for (int k = 0; k < STEPS; k++) {
            const int n = n0 + RPS * k;
            uint32_t off_lo, off_hi;
            if (D == 128) {
                off_lo = sw128(n, c);
                off_hi = REGION + off_lo;
            } else {
                off_lo = sw128(n, c);
                off_hi = sw128(n, c + 4);
            }
            uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
            asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                         : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3)
                         : "r"(src + off_lo));
            asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                         : "=r"(b0), "=r"(b1), "=r"(b2), "=r"(b3)
                         : "r"(src + off_hi));
            uint32_t av[4] = {a0, a1, a2, a3}, bv[4] = {b0, b1, b2, b3}, ao[4], bo[4];
#pragma unroll
            for (int e = 0; e < 4; e++) {
                float x0 = jl::bf16lo(av[e]), x1 = jl::bf16hi(av[e]);
                float y0 = jl::bf16lo(bv[e]), y1 = jl::bf16hi(bv[e]);
                const float c0 = zc[2 * e], s0 = zs[2 * e], c1 = zc[2 * e + 1], s1 = zs[2 * e + 1];
                ao[e] = jl::pack_f16x2(x0 * c0 - y0 * s0, x1 * c1 - y1 * s1);
                bo[e] = jl::pack_f16x2(y0 * c0 + x0 * s0, y1 * c1 + x1 * s1);
            }
            asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(dst + off_lo), "r"(ao[0]),
                         "r"(ao[1]), "r"(ao[2]), "r"(ao[3])
                         : "memory");
            asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(dst + off_hi), "r"(bo[0]),
                         "r"(bo[1]), "r"(bo[2]), "r"(bo[3])
                         : "memory");
            // advance the rotation by RPS rows
            jm += rs;
            const bool carry = jm >= g;
            if (carry) jm -= g;
#pragma unroll
            for (int e = 0; e < 8; e++) {
                const float sc = carry ? bc[e] : ac[e], ss = carry ? bs_[e] : as_[e];
                const float nc = zc[e] * sc - zs[e] * ss;
                const float ns = zs[e] * sc + zc[e] * ss;
                zc[e] = nc;
                zs[e] = ns;
            }
        }
    }
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                   const __grid_constant__ CUtensorMap tv, const Params p,
                   const __grid_constant__ jl::PhaseTable pt)
{
    using C = Cfg<D>;
    constexpr int NS = C::NS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~(uintptr_t)1023);
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sQ = sbase + C::OFF_Q, sQG = sbase + C::OFF_QG, sK = sbase + C::OFF_K,
                   sV = sbase + C::OFF_V, sP = sbase + C::OFF_P;
    const uint32_t bar0 = sbase + C::OFF_BAR;
    auto bar = [&](int idx) -> uint32_t { return bar0 + 8u * (uint32_t)idx; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_BAR + 192);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_BAR + 196);
    const WaitCtx wc{p.status, abort_flag};

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bh = blockIdx.x;
    const int b = bh / p.Hq, h = bh % p.Hq, hk = h / p.grp;
    const int qt = p.n_qtiles - 1 - (int)blockIdx.y;  // longest rows first
    const int i0 = qt * kBM;
    const int T = qt + 1;                             // key tiles 0..qt
    const int S = p.S, w = p.w, g = p.g;
    const bool any_corr = jl::tile_class(i0, 0, kBM, kBN, S, w, g) != jl::kTileExact;

    if (threadIdx.x == 0) {
        mbar_init(bar(C::B_QFULL), 1);
        mbar_init(bar(C::B_QGFULL), 128);
        for (int s = 0; s < NS; s++) {
            mbar_init(bar(C::B_KFULL + s), 1);
            mbar_init(bar(C::B_VFULL + s), 1);
            mbar_init(bar(C::B_KVEMPTY + s), 1);
            mbar_init(bar(C::B_KGFULL + s), 128);
        }
        mbar_init(bar(C::B_SEDONE), 1);
        mbar_init(bar(C::B_SFULL + 0), 1);
        mbar_init(bar(C::B_SFULL + 1), 1);
        mbar_init(bar(C::B_SEMPTY + 0), 128);
        mbar_init(bar(C::B_SEMPTY + 1), 128);
        mbar_init(bar(C::B_PFULL), 128);
        mbar_init(bar(C::B_ODONE), 1);
        mbar_init(bar(C::B_DRAIN), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tS = tmem, tO = tmem + 256;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tmap(&tq);
            prefetch_tmap(&tk);
            prefetch_tmap(&tv);
            mbar_arrive_expect_tx(bar(C::B_QFULL), C::TILE);
#pragma unroll
            for (int r = 0; r < C::NREG; r++)
                tma_load_4d(sQ + r * C::REGION, &tq, bar(C::B_QFULL), r * 64, h, i0, b);
            int issued = 0;
            for (int it = 0; it < T; it++) {
                const int s = it % NS, u = it / NS;
                if (!wait_bar(bar(C::B_KVEMPTY + s), (u & 1) ^ 1, wc)) break;
                mbar_arrive_expect_tx(bar(C::B_KFULL + s), C::TILE);
#pragma unroll
                for (int r = 0; r < C::NREG; r++)
                    tma_load_4d(sK + s * C::TILE + r * C::REGION, &tk, bar(C::B_KFULL + s), r * 64, hk,
                                it * kBN, b);
                mbar_arrive_expect_tx(bar(C::B_VFULL + s), C::TILE);
#pragma unroll
                for (int r = 0; r < C::NREG; r++)
                    tma_load_4d(sV + s * C::TILE + r * C::REGION, &tv, bar(C::B_VFULL + s), r * 64, hk,
                                it * kBN, b);
                issued = it + 1;
            }
            if (*abort_flag) {
                // let the copies already issued land before the CTA retires
                drain_bar(bar(C::B_QFULL), 0);
                for (int it = issued - NS < 0 ? 0 : issued - NS; it < issued; it++) {
                    drain_bar(bar(C::B_KFULL + it % NS), (it / NS) & 1);
                    drain_bar(bar(C::B_VFULL + it % NS), (it / NS) & 1);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idS = idesc_bf16_f32(kBM, kBN, false, false);
            constexpr uint32_t idSG = idesc_f16_f32(kBM, kBN, false, false);
            constexpr uint32_t idPV = idesc_bf16_f32(kBM, D, false, true);
            auto issue_qk = [&](uint32_t dcol, uint32_t a_base, uint32_t b_base, uint32_t idesc) {
#pragma unroll
                for (int k = 0; k < D / 16; k++) {
                    const uint32_t off = (k >> 2) * C::REGION + (k & 3) * 32;
                    mma_f16_ss(tS + dcol, sdesc_sw128(a_base + off, 16, 1024),
                                sdesc_sw128(b_base + off, 16, 1024), idesc, k > 0 ? 1u : 0u);
                }
            };
            bool ok = wait_bar(bar(C::B_QFULL), 0, wc);
            if (ok && any_corr) ok = wait_bar(bar(C::B_QGFULL), 0, wc);
            uint32_t ub_par = 0;  // bit b: parity of the next fill of S buffer b
            uint32_t cu_par = 0;  // bit s: parity of the next correction of stage s
            int slot = 0;
            auto issue_pv = [&](int t) -> bool {
                const int s = t % NS;
                if (!wait_bar(bar(C::B_PFULL), t & 1, wc)) return false;
                if (!wait_bar(bar(C::B_VFULL + s), (t / NS) & 1, wc)) return false;
                tc_fence_after();
                const uint32_t vb = sV + s * C::TILE;
#pragma unroll
                for (int k = 0; k < kBN / 16; k++) {
                    const uint32_t aoff = (k >> 2) * C::REGION + (k & 3) * 32;
                    mma_f16_ss(tO, sdesc_sw128(sP + aoff, 16, 1024),
                                sdesc_sw128(vb + k * 2048, C::REGION, 1024), idPV,
                                (t > 0 || k > 0) ? 1u : 0u);
                }
                mma_commit(bar(C::B_KVEMPTY + s));
                mma_commit(bar(C::B_ODONE));
                return true;
            };
            for (int it = 0; ok && it < T; it++) {
                const int cls = jl::tile_class(i0, it * kBN, kBM, kBN, S, w, g);
                const int s = it % NS;
                const uint32_t kb = sK + s * C::TILE;
                if (!(ok = wait_bar(bar(C::B_KFULL + s), (it / NS) & 1, wc))) break;
                const int b0 = slot & 1;
                if (!(ok = wait_bar(bar(C::B_SEMPTY + b0), ((ub_par >> b0) & 1) ^ 1, wc))) break;
                if (cls == jl::kTileRemote) {
                    if (!(ok = wait_bar(bar(C::B_KGFULL + s), (cu_par >> s) & 1, wc))) break;
                    cu_par ^= 1u << s;
                    tc_fence_after();
                    issue_qk(128u * b0, sQG, kb, idSG);
                } else {
                    tc_fence_after();
                    issue_qk(128u * b0, sQ, kb, idS);
                }
                mma_commit(bar(C::B_SFULL + b0));
                ub_par ^= 1u << b0;
                if (cls == jl::kTileBand) {
                    mma_commit(bar(C::B_SEDONE));
                    const int b1 = b0 ^ 1;
                    if (!(ok = wait_bar(bar(C::B_SEMPTY + b1), ((ub_par >> b1) & 1) ^ 1, wc))) break;
                    if (!(ok = wait_bar(bar(C::B_KGFULL + s), (cu_par >> s) & 1, wc))) break;
                    cu_par ^= 1u << s;
                    tc_fence_after();
                    issue_qk(128u * b1, sQG, kb, idSG);
                    mma_commit(bar(C::B_SFULL + b1));
                    ub_par ^= 1u << b1;
                    slot += 2;
                } else {
                    slot += 1;
                }
                if (it >= 1 && !(ok = issue_pv(it - 1))) break;
            }
            if (ok) ok = issue_pv(T - 1);
            if (!ok) {
                // make sure no MMA is still running before TMEM is released
                mma_commit(bar(C::B_DRAIN));
                drain_bar(bar(C::B_DRAIN), 0);
            }
        }
        __syncwarp();
    } else if (warp < 6) {
        // ------------------------------------------------------------ softmax
        const int q4 = warp & 3;
        const int row = 32 * q4 + lane;
        const int i = i0 + row;
        const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
        float m_used = -INFINITY, l = 0.f;
        uint32_t ub_par = 0;  // bit b: parity of the next fill of S buffer b
        int slot = 0;
        bool ok = true;
        // the score of column e of a 32-column chunk, scaled to log2 units and
        // masked (causal, past-the-end keys); band tiles select the view
        auto score = [&](uint32_t xe, uint32_t ye, int j, bool band, bool need_mask) -> float {
            float sv = __uint_as_float(xe);
            if (band && i - j >= w) sv = __uint_as_float(ye);
            if ((band || need_mask) && (j > i || j >= S)) return -INFINITY;
            return sv * p.scale_log2;
        };
        for (int it = 0; it < T; it++) {
            const int cls = jl::tile_class(i0, it * kBN, kBM, kBN, S, w, g);
            const int j0 = it * kBN;
            const int b0 = slot & 1, b1 = b0 ^ 1;
            const bool band = (cls == jl::kTileBand);
            if (!(ok = wait_bar_warp(bar(C::B_SFULL + b0), (ub_par >> b0) & 1, wc))) break;
            if (band && !(ok = wait_bar_warp(bar(C::B_SFULL + b1), (ub_par >> b1) & 1, wc))) break;
            tc_fence_after();
            const bool need_mask = (j0 + kBN - 1 > i0) || (j0 + kBN > S);
            const uint32_t sx = tS + lane_base + 128u * b0, sy = tS + lane_base + 128u * b1;
            // pass 1: row maximum
            float mx = -INFINITY;
#pragma unroll 1
            for (int ch = 0; ch < kBN / 32; ch++) {
                uint32_t x[32], y[32];
                tmem_ld32(sx + 32u * ch, x);
                if (band) tmem_ld32(sy + 32u * ch, y);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 32; e++)
                    mx = fmaxf(mx, score(x[e], band ? y[e] : 0u, j0 + 32 * ch + e, band, need_mask));
            }
            const float m_new = fmaxf(m_used, mx);
            const bool rescale = m_new > m_used + kRescaleThreshold;
            float factor = 1.f;
            if (rescale) {
                factor = exp2f(m_used - m_new);
                m_used = m_new;
                l *= factor;
            }
            // P buffer and O are free once PV of the previous tile is done
            if (it >= 1) {
                if (!(ok = wait_bar_warp(bar(C::B_ODONE), (it - 1) & 1, wc))) break;
                tc_fence_after();
                if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
                    for (int ch = 0; ch < D / 32; ch++) {
                        uint32_t o[32];
                        tmem_ld32(tO + lane_base + 32u * ch, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int e = 0; e < 32; e++) o[e] = __float_as_uint(__uint_as_float(o[e]) * factor);
                        tmem_st32(tO + lane_base + 32u * ch, o);
                    }
                    tmem_st_wait();
                }
            }
            // pass 2: P = 2^(score - m_used), bf16, into the SW128 K-major P tile
#pragma unroll 1
            for (int ch = 0; ch < kBN / 32; ch++) {
                uint32_t x[32], y[32];
                tmem_ld32(sx + 32u * ch, x);
                if (band) tmem_ld32(sy + 32u * ch, y);
                tmem_ld_wait();
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; e++) {
                    const int j = j0 + 32 * ch + 2 * e;
                    const float p0 = exp2f(score(x[2 * e], band ? y[2 * e] : 0u, j, band, need_mask) - m_used);
                    const float p1 =
                        exp2f(score(x[2 * e + 1], band ? y[2 * e + 1] : 0u, j + 1, band, need_mask) - m_used);
                    l += p0 + p1;
                    pk[e] = jl::pack_bf16x2(p0, p1);
                }
                const uint32_t region = sP + (ch >> 1) * C::REGION;
#pragma unroll
                for (int q = 0; q < 4; q++) {
                    const int cc = (ch & 1) * 4 + q;
                    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(region + sw128(row, cc)),
                                 "r"(pk[4 * q]), "r"(pk[4 * q + 1]), "r"(pk[4 * q + 2]), "r"(pk[4 * q + 3])
                                 : "memory");
                }
            }
            // S buffers fully read; P visible to the tensor core; O rescaled
            tc_fence_before();
            mbar_arrive(bar(C::B_SEMPTY + b0));
            if (band) mbar_arrive(bar(C::B_SEMPTY + b1));
            ub_par ^= 1u << b0;
            if (band) ub_par ^= 1u << b1;
            slot += band ? 2 : 1;
            fence_proxy_async_smem();
            mbar_arrive(bar(C::B_PFULL));
        }
        // ------------------------------------------------------------ epilogue
        if (ok) ok = wait_bar_warp(bar(C::B_ODONE), (T - 1) & 1, wc);
        if (ok) {
            tc_fence_after();
            const float inv_l = 1.f / l;
            __nv_bfloat16 *orow = p.out + (((size_t)b * S + i) * p.Hq + h) * D;
#pragma unroll
            for (int ch = 0; ch < D / 32; ch++) {
                uint32_t o[32];
                tmem_ld32(tO + lane_base + 32u * ch, o);
                tmem_ld_wait();
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; e++)
                    pk[e] = jl::pack_bf16x2(__uint_as_float(o[2 * e]) * inv_l,
                                            __uint_as_float(o[2 * e + 1]) * inv_l);
                if (i < S) {
                    uint4 *dst = reinterpret_cast<uint4 *>(orow + 32 * ch);
#pragma unroll
                    for (int q = 0; q < 4; q++)
                        dst[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
                }
            }
            if (i < S) p.lse[((size_t)b * p.Hq + h) * S + i] = (m_used + log2f(l)) * kLn2;
        }
    } else {
        // ------------------------------------------------------------ correction
        if (any_corr) {
            const int t = threadIdx.x - 192;
            Corrector<D> cor;
            cor.init(t, g, pt);
            bool ok = wait_bar_warp(bar(C::B_QFULL), 0, wc);
            if (ok) {
                cor.run(sQ, sQG, i0);
                fence_proxy_async_smem();
                mbar_arrive(bar(C::B_QGFULL));
            }
            int nb = 0;
            for (int it = 0; ok && it < T; it++) {
                const int cls = jl::tile_class(i0, it * kBN, kBM, kBN, S, w, g);
                if (cls == jl::kTileExact) continue;
                const int s = it % NS;
                if (!(ok = wait_bar_warp(bar(C::B_KFULL + s), (it / NS) & 1, wc))) break;
                if (cls == jl::kTileBand) {
                    if (!(ok = wait_bar_warp(bar(C::B_SEDONE), nb & 1, wc))) break;
                    nb++;
                    tc_fence_after();
                }
                const uint32_t kb = sK + s * C::TILE;
                cor.run(kb, kb, it * kBN);
                fence_proxy_async_smem();
                mbar_arrive(bar(C::B_KGFULL + s));
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        fn = reinterpret_cast<EncodeTiledFn>(ptr);
    }
    return fn;
}

// [B, S, H, D] bf16 viewed as a 4-D tensor {D, H, S, B}; box {64, 1, 128, 1},
// 128-byte swizzle, zero fill outside the tensor.
bool make_bshd_map(CUtensorMap *m, const void *base, int B, int S, int H, int D)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)S, (cuuint64_t)B};
    cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2, (cuuint64_t)S * H * D * 2};
    cuuint32_t box[4] = {64, 1, 128, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int D>
int launch(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv, const Params &p,
           const jl::PhaseTable &pt, cudaStream_t st)
{
    auto kern = prefill_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<D>::SMEM);
    if (e != cudaSuccess) return jl::cuda_status(e);
    dim3 grid((unsigned)(p.B * p.Hq), (unsigned)p.n_qtiles, 1);
    kern<<<grid, kThreads, Cfg<D>::SMEM, st>>>(tq, tk, tv, p, pt);
    return jl::cuda_status(cudaGetLastError());
}

}  // namespace

extern "C" int jl_bifocal_prefill(const void *q, const void *k, const void *v, void *out, float *lse,
                                  int B, int Hq, int Hkv, int S, int D, int L_pre, int w,
                                  double theta, void *stream)
{
    if (!q || !k || !v || !out || !lse) return JL_ERR_ARG;
    if (B < 1 || Hq < 1 || Hkv < 1 || S < 1 || L_pre < 1 || w < 1 || !(theta > 0.0) ||
        Hq % Hkv != 0)
        return JL_ERR_ARG;
    if (D != 64 && D != 128) return JL_ERR_UNSUPPORTED;
    if (!jl::aligned16(q) || !jl::aligned16(k) || !jl::aligned16(v) || !jl::aligned16(out) ||
        !jl::aligned16(lse))
        return JL_ERR_ALIGN;
    if ((long long)B * S * Hq * D > ((long long)1 << 46)) return JL_ERR_OVERFLOW;
    const long long n_qtiles = ((long long)S + kBM - 1) / kBM;
    if ((long long)B * Hq > 0x7fffffffLL || n_qtiles > 65535) return JL_ERR_OVERFLOW;
    jl::PhaseTable pt;
    if (!jl::make_phase_table(&pt, D, theta)) return JL_ERR_ARG;
    CUtensorMap tq, tk, tv;
    if (!make_bshd_map(&tq, q, B, S, Hq, D) || !make_bshd_map(&tk, k, B, S, Hkv, D) ||
        !make_bshd_map(&tv, v, B, S, Hkv, D))
        return JL_ERR_CUDA;
    Params p;
    p.out = (__nv_bfloat16 *)out;
    p.lse = lse;
    p.status = jl::status_word_ptr();
    p.B = B;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.S = S;
    p.w = w;
    p.g = (int)jl::group_factor_host(S, L_pre);
    p.grp = Hq / Hkv;
    p.n_qtiles = (int)n_qtiles;
    p.scale_log2 = (float)(1.0 / sqrt((double)D) * 1.4426950408889634);
    cudaStream_t st = (cudaStream_t)stream;
    return D == 128 ? launch<128>(tq, tk, tv, p, pt, st) : launch<64>(tq, tk, tv, p, pt, st);
}
