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
// One CTA owns a 128-row query tile of NH heads that share a kv head (GQA
// pair when Hq/Hkv is even), so every K/V tile it loads and every K tile it
// corrects serves 2 x 128 query rows.  Its key tiles are visited as a
// sequence of "virtual tiles": first the remote phase -- every key tile
// wholly outside the window plus the remote part of the tiles the window
// edge crosses -- on Q corrected in place, then the exact phase -- the exact
// part of those edge tiles plus every tile inside the window -- on Q
// reloaded.  An edge tile thus appears twice with complementary masks; the
// online softmax does not care in which order keys arrive.
//
// Warp roles (480 threads):
//   warps 0-3   softmax of head 0 (one query row per thread, TMEM lane = row)
//   warps 4-7   softmax of head 1 (idle when NH = 1)
//   warps 8-11  correction: Q of every head once, then every remote K tile
//   warp 12     TMA producer: Q and the K ring (NK stages)
//   warp 13     TMEM allocator + single-thread tcgen05.mma issuer
//   warp 14     TMA producer: the V ring (NV stages), so K loads -- which the
//               correction must finish before their QK -- never queue
//               behind a V slot
// TMEM (512 columns): S_n at [128n, 128n+128) with P_n (bf16) written over
// its first 64 columns, O_n at [256 + 128n, 256 + 128n + D).
// MMA order per virtual tile v: PV_0(v), QK_0(v+1), PV_1(v), QK_1(v+1): the
// QK of the next tile for a head follows that head's PV in the in-order
// tensor pipe, so it may overwrite S_n/P_n without a wait, and each softmax
// group works while the tensor core serves the other head.
#include <math.h>
#include <stdio.h>
#include <string.h>

#include "jl_common.cuh"
#include "sm100_ptx.cuh"
#include "tile_class.cuh"
#include "corrector.cuh"

namespace {

using namespace jl::ptx;

constexpr int kBM = 128, kBN = 128;
constexpr int kThreads = 480;
constexpr float kLn2 = 0.6931471805599453f;
// Lazy rescaling: the running maximum used as the exponent offset is moved
// only when a row's maximum grows by more than this (log2 units), so P stays
// <= 2^8 and O is rarely rescaled in TMEM.
constexpr float kRescaleThreshold = 8.0f;

template <int D, int NH>
struct Cfg {
    static constexpr int REGION = kBM * 64 * 2;  // one 128-row x 64-column box: 16 KB
    static constexpr int NREG = D / 64;          // boxes per 128-row tile
    static constexpr int TILE = kBM * D * 2;     // Q / K / V tile bytes
    static constexpr int NK = (D == 128) ? 3 : 4;                     // K ring stages
    static constexpr int NV = (D == 128) ? (NH == 2 ? 2 : 3) : 4;     // V ring stages
    // a V stage is refilled only after the PV that frees it, and that PV
    // follows the MMA issuer's wait on GO[v % NK] -- so the V producer's
    // arrival for tile v lands in that barrier's phase for v only if NV <= NK
    static_assert(NV <= NK, "V ring deeper than the K ring");
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + NH * TILE;
    static constexpr int OFF_V = OFF_K + NK * TILE;
    static constexpr int OFF_BAR = OFF_V + NV * TILE;
    static constexpr int BAR_BYTES = 512;
    static constexpr int SMEM = OFF_BAR + BAR_BYTES + 1024;  // + alignment slack
    // barrier indices
    static constexpr int B_QFULL = 0, B_K0READY = 1, B_QFREE = 2, B_DRAIN = 3, B_KFULL = 4,
                         B_KEMPTY = B_KFULL + NK, B_GO = B_KEMPTY + NK, B_VFULL = B_GO + NK,
                         B_VEMPTY = B_VFULL + NV, B_SFULL = B_VEMPTY + NV, B_PFULL = B_SFULL + 2,
                         B_ODONE = B_PFULL + 2, NBAR = B_ODONE + 2;
    static constexpr int OFF_TMEM_SLOT = 448, OFF_ABORT = 452;
    static_assert(NBAR * 8 <= OFF_TMEM_SLOT, "barrier area");
    static_assert(SMEM <= 232448, "shared memory budget");
};

struct Params {
    __nv_bfloat16 *out;  // row 0 of this launch's rows; batch stride q_rows rows
    float *lse;          // column 0 of this launch's rows; row stride lse_stride
    int *status;
    // S: keys (positions 0..S-1, the length that sets g); the Sq query rows sit
    // at positions pos0..pos0+Sq-1 = S-Sq..S-1 (pos0 = 0, Sq = S: full prefill)
    int B, Hq, Hkv, S, Sq, pos0, w, g, grp, n_qtiles, pairs;  // pairs = grp / NH
    int q_rows;          // rows per batch entry of q / out (>= Sq)
    int lse_stride;      // elements between (b, h) rows of lse (>= Sq)
    int qshift;          // added to the query's correction offset (query-shift variant)
    int sliding;         // sliding-window layer: keys with i - j >= w are not attended
    float scale_log2;    // tau * log2(e)
};

__device__ __forceinline__ float fast_exp2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// The virtual-tile sequence of one query tile (identical in every role).
// Key-tile classes are monotone in the key tile index kt: remote, then band
// (the window edge), then exact.  The remote phase visits kt in [0, nr)
// (remote and band tiles, remote part), the exact phase kt in [kb, qt]
// (band and exact tiles, exact part).
struct Visit {
    int nr, kb, T;

    // query rows from absolute position i0; kt_last = the last key tile any of
    // them reaches (the diagonal tile)
    __device__ void init(int i0, int kt_last, int S, int w, int g)
    {
        // first kt whose class is not remote; first kt whose class is exact
        int lo = 0, hi = kt_last;  // class(kt_last) is never remote (distance 0 < w)
        while (lo < hi) {
            int mid = (lo + hi) >> 1;
            if (jl::tile_class(i0, mid * kBN, kBM, kBN, S, w, g) == jl::kTileRemote) lo = mid + 1;
            else hi = mid;
        }
        kb = lo;
        lo = kb;
        hi = kt_last + 1;
        while (lo < hi) {
            int mid = (lo + hi) >> 1;
            if (jl::tile_class(i0, mid * kBN, kBM, kBN, S, w, g) == jl::kTileExact) hi = mid;
            else lo = mid + 1;
        }
        nr = lo;  // tiles [0, nr) have a remote part
        T = nr + (kt_last + 1 - kb);
    }

    __device__ __forceinline__ int kt(int v) const { return v < nr ? v : kb + (v - nr); }
    __device__ __forceinline__ bool remote(int v) const { return v < nr; }
};

template <int D, int NH>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                   const __grid_constant__ CUtensorMap tv, const Params p,
                   const __grid_constant__ jl::PhaseTable pt, const __grid_constant__ RotConsts rc)
{
    using C = Cfg<D, NH>;
    constexpr int NK = C::NK, NV = C::NV;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~(uintptr_t)1023);
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sQ = sbase + C::OFF_Q, sK = sbase + C::OFF_K, sV = sbase + C::OFF_V;
    const uint32_t bar0 = sbase + C::OFF_BAR;
    auto bar = [&](int idx) -> uint32_t { return bar0 + 8u * (uint32_t)idx; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_BAR + C::OFF_TMEM_SLOT);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_BAR + C::OFF_ABORT);
    const WaitCtx wc{p.status, abort_flag};

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // blockIdx.x walks (query tile, head pair) with the pair fastest and the
    // longest rows first; blockIdx.y is (batch, kv head).  Every wave of CTAs
    // thus works on one kv head, whose K/V (64 MB at 128K) stays in L2.
    const int hp = (int)blockIdx.x % p.pairs;
    const int qt = p.n_qtiles - 1 - (int)blockIdx.x / p.pairs;
    const int hk = (int)blockIdx.y % p.Hkv;
    const int b = (int)blockIdx.y / p.Hkv;
    const int h0 = hk * p.grp + hp * NH;  // first head of this CTA
    const int q_row0 = qt * kBM;   // first row of the tile in q / out / lse
    const int i0 = p.pos0 + q_row0;  // its position
    const int S = p.S, w = p.w, g = p.g;
    // tiles are classified against the window as for any g > 1 when the layer
    // is a sliding window (g itself plays no part there)
    const int g_cls = p.sliding ? 2 : g;
    Visit vis;
    vis.init(i0, (min(i0 + kBM, S) - 1) / kBN, S, w, g_cls);
    if (p.sliding) {
        // nothing outside the window is attended: no remote phase
        vis.T -= vis.nr;
        vis.nr = 0;
    }
    const int T = vis.T, NR = vis.nr;

    if (threadIdx.x == 0) {
        mbar_init(bar(C::B_QFULL), 1);
        mbar_init(bar(C::B_K0READY), 128);
        mbar_init(bar(C::B_QFREE), 1);
        mbar_init(bar(C::B_DRAIN), 1);
        for (int s = 0; s < NK; s++) {
            mbar_init(bar(C::B_KFULL + s), 1);
            mbar_init(bar(C::B_KEMPTY + s), 1);
            // head 0's softmax, the correction warps and the V producer
            mbar_init(bar(C::B_GO + s), 128 + 128 + 1);
        }
        for (int s = 0; s < NV; s++) {
            mbar_init(bar(C::B_VFULL + s), 1);
            mbar_init(bar(C::B_VEMPTY + s), 1);
        }
        for (int n = 0; n < 2; n++) {
            mbar_init(bar(C::B_SFULL + n), 1);
            mbar_init(bar(C::B_PFULL + n), 128);
            mbar_init(bar(C::B_ODONE + n), 1);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 13) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 12) {
        // ------------------------------------------------------------ producer: Q and K
        if (lane == 0) {
            prefetch_tmap(&tq);
            prefetch_tmap(&tk);
            auto load_q = [&]() {
                mbar_arrive_expect_tx(bar(C::B_QFULL), NH * C::TILE);
#pragma unroll
                for (int n = 0; n < NH; n++)
#pragma unroll
                    for (int r = 0; r < C::NREG; r++)
                        tma_load_4d(sQ + n * C::TILE + r * C::REGION, &tq, bar(C::B_QFULL), r * 64,
                                    h0 + n, q_row0, b);
            };
            load_q();
            int issued = 0;
            bool ok = true;
            for (int v = 0; v < T; v++) {
                if (v == NR && NR > 0) {
                    // the remote phase has finished reading the corrected Q
                    if (!(ok = wait_bar(bar(C::B_QFREE), 0, wc))) break;
                    load_q();
                }
                const int sk = v % NK;
                if (!(ok = wait_bar(bar(C::B_KEMPTY + sk), ((v / NK) & 1) ^ 1, wc))) break;
                mbar_arrive_expect_tx(bar(C::B_KFULL + sk), C::TILE);
#pragma unroll
                for (int r = 0; r < C::NREG; r++)
                    tma_load_4d(sK + sk * C::TILE + r * C::REGION, &tk, bar(C::B_KFULL + sk), r * 64, hk,
                                vis.kt(v) * kBN, b);
                issued = v + 1;
            }
            if (!ok) {
                // let the copies already issued land before the CTA retires
                for (int v = issued - NK < 0 ? 0 : issued - NK; v < issued; v++)
                    drain_bar(bar(C::B_KFULL + v % NK), (v / NK) & 1);
            }
        }
    } else if (warp == 14) {
        // ------------------------------------------------------------ producer: V
        if (lane == 0) {
            prefetch_tmap(&tv);
            int issued = 0;
            bool ok = true;
            for (int v = 0; v < T; v++) {
                const int sv = v % NV;
                if (!(ok = wait_bar(bar(C::B_VEMPTY + sv), ((v / NV) & 1) ^ 1, wc))) break;
                mbar_arrive_expect_tx(bar(C::B_VFULL + sv), C::TILE);
#pragma unroll
                for (int r = 0; r < C::NREG; r++)
                    tma_load_4d(sV + sv * C::TILE + r * C::REGION, &tv, bar(C::B_VFULL + sv), r * 64, hk,
                                vis.kt(v) * kBN, b);
                issued = v + 1;
                // V(v) landed: one of the three arrivals that let tile v's PV go
                if (!(ok = wait_bar(bar(C::B_VFULL + sv), (v / NV) & 1, wc))) break;
                mbar_arrive(bar(C::B_GO + v % NK));
            }
            if (!ok) {
                for (int v = issued - NV < 0 ? 0 : issued - NV; v < issued; v++)
                    drain_bar(bar(C::B_VFULL + v % NV), (v / NV) & 1);
            }
        }
    } else if (warp == 13) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idS = idesc_bf16_f32(kBM, kBN, false, false);
            constexpr uint32_t idSG = idesc_f16_f32(kBM, kBN, false, false);
            constexpr uint32_t idPV = idesc_bf16_f32(kBM, D, false, true);
            // The issuing thread runs at most about one MMA ahead of the tensor
            // pipe, and every mbarrier wait it makes costs ~200 cycles of pipe
            // time even when the phase is already complete (the SS MMAs keep
            // shared memory busy).  So it waits twice per virtual tile: on
            // GO[v % NK] -- head 0's P(v) written, V(v) landed, K(v+1) landed and
            // (remote) corrected, Q reloaded before the first exact QK -- and on
            // head 1's P(v).  The first QK waits on K0READY (Q and K(0) ready).
            bool ok = wait_bar(bar(C::B_K0READY), 0, wc);
            tc_fence_after();
            // S_n = Q_n K^T.  The descriptors are built once per operand tile and
            // advanced by each k-step's byte offset (>> 4), keeping the issuing
            // thread's instructions between MMAs to a minimum.
            auto qk_head = [&](int v, int n) {
                const uint64_t dk = sdesc_sw128(sK + (v % NK) * C::TILE, 16, 1024);
                const uint64_t dq = sdesc_sw128(sQ + n * C::TILE, 16, 1024);
                const uint32_t id = vis.remote(v) ? idSG : idS;
#pragma unroll
                for (int k = 0; k < D / 16; k++) {
                    const uint64_t o = (uint64_t)(((k >> 2) * C::REGION + (k & 3) * 32) >> 4);
                    mma_f16_ss(tmem + 128u * n, dq + o, dk + o, id, k > 0 ? 1u : 0u);
                }
                mma_commit(bar(C::B_SFULL + n));
                if (n == NH - 1) {
                    mma_commit(bar(C::B_KEMPTY + v % NK));
                    if (v == NR - 1) mma_commit(bar(C::B_QFREE));
                }
            };
            if (ok)
                for (int n = 0; n < NH; n++) qk_head(0, n);
            for (int v = 0; ok && v < T; v++) {
                const int sv = v % NV;
                const uint64_t dv = sdesc_sw128(sV + sv * C::TILE, C::REGION, 1024);
                for (int n = 0; n < NH; n++) {
                    if (n == 0) ok = wait_bar(bar(C::B_GO + v % NK), (v / NK) & 1, wc);
                    else ok = wait_bar(bar(C::B_PFULL + n), v & 1, wc);
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll
                    for (int k = 0; k < kBN / 16; k++)
                        mma_f16_ts(tmem + 256u + 128u * n, tmem + 128u * n + 8u * k,
                                   dv + (uint64_t)((k * 2048) >> 4), idPV, (v > 0 || k > 0) ? 1u : 0u);
                    mma_commit(bar(C::B_ODONE + n));
                    if (n == NH - 1) mma_commit(bar(C::B_VEMPTY + sv));
                    if (v + 1 < T) qk_head(v + 1, n);
                }
            }
            if (!ok) {
                // make sure no MMA is still running before TMEM is released
                mma_commit(bar(C::B_DRAIN));
                drain_bar(bar(C::B_DRAIN), 0);
            }
        }
        __syncwarp();
    } else if (warp < 8) {
        // ------------------------------------------------------------ softmax
        const int n = warp >> 2;  // head slot
        if (n < NH) {
            const int q4 = warp & 3;
            const int row = 32 * q4 + lane;
            const int i = i0 + row;
            const int h = h0 + n;
            const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
            const uint32_t tS = tmem + lane_base + 128u * n;
            const uint32_t tO = tmem + lane_base + 256u + 128u * n;
            const float sc = p.scale_log2;
            float m_used = -INFINITY, l = 0.f;  // m_used in log2 units
            bool ok = true;
            const jl::f32x2 sc2 = jl::f2(sc, sc);
            for (int v = 0; v < T; v++) {
                const int kt = vis.kt(v);
                const bool remote = vis.remote(v);
                const int j0 = kt * kBN;
                const bool band = jl::tile_class(i0, j0, kBM, kBN, S, w, g_cls) == jl::kTileBand;
                const bool masked = band || (j0 + kBN - 1 > i0) || (j0 + kBN > S);
                // load 64 score columns (half hh) as raw fp32 bits with both TMEM
                // loads in flight; keys that are in the future, past the end, or
                // (edge tiles) of the other view -> -inf
                auto load_half = [&](int hh, uint32_t (&x)[64]) {
                    tmem_ld32(tS + 64u * hh, *reinterpret_cast<uint32_t(*)[32]>(&x[0]));
                    tmem_ld32(tS + 64u * hh + 32u, *reinterpret_cast<uint32_t(*)[32]>(&x[32]));
                    tmem_ld_wait();
                    if (masked) {
#pragma unroll
                        for (int e = 0; e < 64; e++) {
                            const int j = j0 + 64 * hh + e;
                            bool d = (j > i || j >= S);
                            if (band) d = d || (remote ? (i - j < w) : (i - j >= w));
                            if (d) x[e] = 0xff800000u;
                        }
                    }
                };
                // P = 2^(s*sc - m) for half hh, bf16 pairs into S columns 32hh..32hh+31
                auto exp_half = [&](int hh, const uint32_t (&x)[64], jl::f32x2 nm, jl::f32x2 &lsum) {
#pragma unroll
                    for (int q = 0; q < 2; q++) {
                        uint32_t pk[16];
#pragma unroll
                        for (int e = 0; e < 16; e++) {
                            const int k2 = 32 * q + 2 * e;
                            const jl::f32x2 t =
                                jl::fma2(jl::f2(__uint_as_float(x[k2]), __uint_as_float(x[k2 + 1])), sc2, nm);
                            float t0, t1;
                            jl::f2_split(t, t0, t1);
                            const jl::f32x2 pp = jl::f2(fast_exp2(t0), fast_exp2(t1));
                            lsum = jl::add2(lsum, pp);
                            pk[e] = jl::f2_to_bf16x2(pp);
                        }
                        tmem_st16(tS + 32u * hh + 16u * q, pk);
                    }
                };
                if (!(ok = wait_bar_warp(bar(C::B_SFULL + n), v & 1, wc))) break;
                tc_fence_after();
                // One pass over the scores, 64 columns at a time, against a
                // running exponent offset m_cur (log2 units).  A half whose
                // maximum exceeds m_cur by more than the threshold raises m_cur
                // by an integer k (so the P already written is rescaled by the
                // exact power of two 2^-k), or sets it when the row had no key
                // yet.  S is never read again after its P is written.
                float m_cur = m_used;
                jl::f32x2 lsum = jl::f2(0.f, 0.f);
#pragma unroll 1
                for (int hh = 0; hh < 2; hh++) {
                    uint32_t x[64];
                    load_half(hh, x);
                    float cm = -INFINITY;
#pragma unroll
                    for (int e = 0; e < 32; e++)
                        cm = jl::fmax3(cm, __uint_as_float(x[2 * e]), __uint_as_float(x[2 * e + 1]));
                    cm *= sc;
                    const bool raise = cm > m_cur + kRescaleThreshold;
                    float f = 1.f;
                    if (raise) {
                        if (m_cur == -INFINITY) {
                            m_cur = cm;  // the first half of this row holds only zeros
                        } else {
                            // an integer step to at least the new maximum, so the
                            // factor is an exact power of two (0 once below the
                            // smallest fp32 subnormal) and no P exceeds 2^8
                            const float k = ceilf(cm - m_cur);
                            m_cur += k;
                            f = k >= 150.f ? 0.f : ldexpf(1.f, -(int)k);
                        }
                    }
                    if (hh > 0 && __any_sync(0xffffffffu, raise && f != 1.f)) {
                        lsum = jl::mul2(lsum, jl::f2(f, f));
                        tmem_st_wait();  // the first half's P has landed
#pragma unroll 1
                        for (int c2 = 0; c2 < 2; c2++) {
                            uint32_t pk[16];
                            tmem_ld16(tS + 16u * c2, pk);
                            tmem_ld_wait();
#pragma unroll
                            for (int e = 0; e < 16; e++)
                                pk[e] = jl::f2_to_bf16x2(jl::mul2(jl::bf16x2_to_f2(pk[e]), jl::f2(f, f)));
                            tmem_st16(tS + 16u * c2, pk);
                        }
                    }
                    const float m_off = (m_cur == -INFINITY) ? 0.f : m_cur;
                    exp_half(hh, x, jl::f2(-m_off, -m_off), lsum);
                }
                // the tile moved the row's offset: bring O and l to the new one
                const bool moved = m_cur != m_used;
                const bool need_o = moved && m_used != -INFINITY;
                const float factor = need_o ? exp2f(m_used - m_cur) : (moved ? 0.f : 1.f);
                l *= factor;
                if (v >= 1 && __any_sync(0xffffffffu, need_o)) {
                    // O holds PV of tiles < v (complete: this head's QK(v) followed
                    // its PV(v-1) in the in-order tensor pipe); rows whose offset
                    // did not move (or that have no key yet) scale by 1
                    const float fo = need_o ? factor : 1.f;
                    if (!(ok = wait_bar_warp(bar(C::B_ODONE + n), (v - 1) & 1, wc))) break;
                    tc_fence_after();
#pragma unroll 1
                    for (int ch = 0; ch < D / 32; ch++) {
                        uint32_t o[32];
                        tmem_ld32(tO + 32u * ch, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int e = 0; e < 32; e++) o[e] = __float_as_uint(__uint_as_float(o[e]) * fo);
                        tmem_st32(tO + 32u * ch, o);
                    }
                }
                m_used = m_cur;
                float l0, l1;
                jl::f2_split(lsum, l0, l1);
                l += l0 + l1;
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(n == 0 ? bar(C::B_GO + v % NK) : bar(C::B_PFULL + n));
            }
            // ------------------------------------------------------------ epilogue
            if (ok) ok = wait_bar_warp(bar(C::B_ODONE + n), (T - 1) & 1, wc);
            if (ok) {
                tc_fence_after();
                // a row sum that is not finite comes from an infinite or NaN score
                // (an input or corrected operand out of range): report it
                if (!(l < INFINITY)) jl::record_status(p.status, JL_ERR_GUARD);
                const float inv_l = 1.f / l;
                const int il = i - p.pos0;  // row in out / lse (valid while i < S)
                __nv_bfloat16 *orow = p.out + (((size_t)b * p.q_rows + il) * p.Hq + h) * D;
#pragma unroll 1
                for (int ch = 0; ch < D / 32; ch++) {
                    uint32_t o[32];
                    tmem_ld32(tO + 32u * ch, o);
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
                if (i < S) p.lse[((size_t)b * p.Hq + h) * p.lse_stride + il] = (m_used + log2f(l)) * kLn2;
            }
        }
    } else {
        // ------------------------------------------------------------ correction
        // Makes K(u) ready for QK(u): waits for it to land and, on a remote
        // tile, rotates it in place; then arrives on the barrier the MMA issuer
        // waits on before QK(u) -- K0READY for u = 0 (after correcting Q when
        // the CTA has a remote phase), else GO[(u-1) % NK]; before the first
        // exact tile it also waits for the exact Q to be reloaded.  u = T loads
        // nothing (tile T-1's PV has no QK after it) and only arrives.
        const int t = threadIdx.x - 256;
        Corrector<D> cor;
        if (NR > 0) cor.init(t, g, pt, rc);
        bool ok = wait_bar_warp(bar(C::B_QFULL), 0, wc);
        if (ok && NR > 0) {
#pragma unroll 1
            for (int n = 0; n < NH; n++) cor.run_q(sQ + n * C::TILE, i0, p.qshift);
        }
        for (int u = 0; ok && u <= T; u++) {
            if (u < T) {
                const int sk = u % NK;
                if (!(ok = wait_bar_warp(bar(C::B_KFULL + sk), (u / NK) & 1, wc))) break;
                if (u < NR) cor.run_k(sK + sk * C::TILE, u);
                if (u == NR && NR > 0 && !(ok = wait_bar_warp(bar(C::B_QFULL), 1, wc))) break;
                if (u <= NR) fence_proxy_async_smem();
            }
            // An arrival for tile u-1 must not land in GO's phase for tile
            // u-1-NK.  For u < T the landing of K(u) orders it (the stage is
            // refilled only after QK(u-NK), which follows the issuer's wait on
            // that phase); the last one has no K to wait for, so it waits for
            // that phase itself.
            if (u == T && T - 1 >= NK &&
                !(ok = wait_bar_warp(bar(C::B_GO + (T - 1) % NK), (((T - 1) / NK) & 1) ^ 1, wc)))
                break;
            mbar_arrive(u == 0 ? bar(C::B_K0READY) : bar(C::B_GO + (u - 1) % NK));
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 13) tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------------------- pair kernel
// The same computation with two SMs per tile (cta_group::2 MMAs, M = 256): a
// cluster of two CTAs covers one 128-row query tile of FOUR heads that share a
// kv head, two heads per CTA.  Each CTA loads -- and on remote tiles corrects
// -- one half of every K tile (64 keys), and loads one half of every V tile
// (64 of the 128 dims), so per SM the correction work and the K / V
// shared-memory traffic are half those of the single-CTA kernel while every
// corrected key still serves 4 x 128 query rows.  One thread of the even CTA
// issues the MMAs of both (A rows from each CTA's own Q or P, B split along N
// between the CTAs, D in each CTA's own TMEM) and multicasts every commit to
// both CTAs' barriers; warps of either CTA arrive on the even CTA's barriers
// through the cluster window.  Roles, virtual tiles and barrier phases are
// those of prefill_kernel; arrivals on the even CTA's barriers come one per
// warp.
struct PairCfg {
    static constexpr int D = 128;
    static constexpr int QTILE = kBM * D * 2;   // one head's 128 query rows: 32 KB
    static constexpr int QREG = kBM * 128;      // one 64-column box of it: 16 KB
    static constexpr int KHALF = 64 * D * 2;    // 64 keys x 128 dims: 16 KB
    static constexpr int KREG = 64 * 128;       // one 64-column box of it: 8 KB
    static constexpr int VHALF = kBN * 64 * 2;  // 128 keys x 64 dims: 16 KB
    static constexpr int NK = 4, NV = 4;
    static_assert(NV <= NK, "V ring deeper than the K ring");
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + 2 * QTILE;
    static constexpr int OFF_V = OFF_K + NK * KHALF;
    static constexpr int OFF_BAR = OFF_V + NV * VHALF;
    static constexpr int SMEM = OFF_BAR + 512 + 1024;  // + alignment slack
    static constexpr int B_QFULL = 0, B_K0READY = 1, B_QFREE = 2, B_DRAIN = 3, B_KFULL = 4,
                         B_KEMPTY = B_KFULL + NK, B_GO = B_KEMPTY + NK, B_VFULL = B_GO + NK,
                         B_VEMPTY = B_VFULL + NV, B_SFULL = B_VEMPTY + NV, B_PFULL = B_SFULL + 2,
                         B_ODONE = B_PFULL + 2, NBAR = B_ODONE + 2;
    static constexpr int OFF_TMEM_SLOT = 448, OFF_ABORT = 452;
    static_assert(NBAR * 8 <= OFF_TMEM_SLOT, "barrier area");
    static_assert(SMEM <= 232448, "shared memory budget");
    // arrivals on the even CTA's barriers: one per warp of both CTAs
    static constexpr uint32_t K0_COUNT = 2 * 4;           // correction warps
    static constexpr uint32_t GO_COUNT = 2 * (4 + 4 + 1);  // head-0 softmax, correction, V producer
    static constexpr uint32_t P1_COUNT = 2 * 4;           // head-1 softmax
    static constexpr uint16_t BOTH = 0x3;
};

__global__ void __launch_bounds__(kThreads, 1)
    prefill_pair_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                        const __grid_constant__ CUtensorMap tv, const Params p,
                        const __grid_constant__ jl::PhaseTable pt, const __grid_constant__ RotConsts rc)
{
    using C = PairCfg;
    constexpr int D = C::D, NK = C::NK, NV = C::NV;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~(uintptr_t)1023);
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sQ = sbase + C::OFF_Q, sK = sbase + C::OFF_K, sV = sbase + C::OFF_V;
    const uint32_t bar0 = sbase + C::OFF_BAR;
    auto bar = [&](int idx) -> uint32_t { return bar0 + 8u * (uint32_t)idx; };
    // the even CTA's copy of a barrier, in the cluster window
    auto lead = [&](int idx) -> uint32_t { return mapa_shared(bar(idx), 0); };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_BAR + C::OFF_TMEM_SLOT);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_BAR + C::OFF_ABORT);
    const WaitCtx wc{p.status, abort_flag};

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();  // = blockIdx.x & 1
    // blockIdx.x >> 1 walks (query tile, quad of heads), quad fastest, longest
    // rows first; the rank picks the head pair of the quad
    const int quads = p.pairs / 2;
    const int cl = (int)blockIdx.x >> 1;
    const int qt = p.n_qtiles - 1 - cl / quads;
    const int hk = (int)blockIdx.y % p.Hkv;
    const int b = (int)blockIdx.y / p.Hkv;
    const int h0 = hk * p.grp + (2 * (cl % quads) + (int)rank) * 2;
    const int q_row0 = qt * kBM;
    const int i0 = p.pos0 + q_row0;
    const int S = p.S, w = p.w, g = p.g;
    const int g_cls = p.sliding ? 2 : g;
    Visit vis;
    vis.init(i0, (min(i0 + kBM, S) - 1) / kBN, S, w, g_cls);
    if (p.sliding) {
        vis.T -= vis.nr;
        vis.nr = 0;
    }
    const int T = vis.T, NR = vis.nr;

    if (threadIdx.x == 0) {
        mbar_init(bar(C::B_QFULL), 1);
        mbar_init(bar(C::B_K0READY), C::K0_COUNT);
        mbar_init(bar(C::B_QFREE), 1);
        mbar_init(bar(C::B_DRAIN), 1);
        for (int s = 0; s < NK; s++) {
            mbar_init(bar(C::B_KFULL + s), 1);
            mbar_init(bar(C::B_KEMPTY + s), 1);
            mbar_init(bar(C::B_GO + s), C::GO_COUNT);
        }
        for (int s = 0; s < NV; s++) {
            mbar_init(bar(C::B_VFULL + s), 1);
            mbar_init(bar(C::B_VEMPTY + s), 1);
        }
        for (int n = 0; n < 2; n++) {
            mbar_init(bar(C::B_SFULL + n), 1);
            mbar_init(bar(C::B_PFULL + n), C::P1_COUNT);
            mbar_init(bar(C::B_ODONE + n), 1);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 13) {
        tmem_alloc2(smem_u32(tmem_slot), 512);
        tmem_relinquish2();
    }
    // both CTAs' barriers and TMEM exist before anyone arrives or issues
    __syncwarp();
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 12) {
        // ------------------------------------------------------------ producer: Q and K halves
        if (lane == 0) {
            prefetch_tmap(&tq);
            prefetch_tmap(&tk);
            auto load_q = [&]() {
                mbar_arrive_expect_tx(bar(C::B_QFULL), 2 * C::QTILE);
#pragma unroll
                for (int n = 0; n < 2; n++)
#pragma unroll
                    for (int r = 0; r < 2; r++)
                        tma_load_4d(sQ + n * C::QTILE + r * C::QREG, &tq, bar(C::B_QFULL), r * 64, h0 + n,
                                    q_row0, b);
            };
            load_q();
            int issued = 0;
            bool ok = true;
            for (int v = 0; v < T; v++) {
                if (v == NR && NR > 0) {
                    if (!(ok = wait_bar_cl(bar(C::B_QFREE), 0, wc))) break;
                    load_q();
                }
                const int sk = v % NK;
                if (!(ok = wait_bar_cl(bar(C::B_KEMPTY + sk), ((v / NK) & 1) ^ 1, wc))) break;
                mbar_arrive_expect_tx(bar(C::B_KFULL + sk), C::KHALF);
#pragma unroll
                for (int r = 0; r < 2; r++)
                    tma_load_4d(sK + sk * C::KHALF + r * C::KREG, &tk, bar(C::B_KFULL + sk), r * 64, hk,
                                vis.kt(v) * kBN + 64 * (int)rank, b);
                issued = v + 1;
            }
            if (!ok) {
                for (int v = issued - NK < 0 ? 0 : issued - NK; v < issued; v++)
                    drain_bar(bar(C::B_KFULL + v % NK), (v / NK) & 1);
            }
        }
    } else if (warp == 14) {
        // ------------------------------------------------------------ producer: V halves
        if (lane == 0) {
            prefetch_tmap(&tv);
            int issued = 0;
            bool ok = true;
            for (int v = 0; v < T; v++) {
                const int sv = v % NV;
                if (!(ok = wait_bar_cl(bar(C::B_VEMPTY + sv), ((v / NV) & 1) ^ 1, wc))) break;
                mbar_arrive_expect_tx(bar(C::B_VFULL + sv), C::VHALF);
                tma_load_4d(sV + sv * C::VHALF, &tv, bar(C::B_VFULL + sv), 64 * (int)rank, hk, vis.kt(v) * kBN, b);
                issued = v + 1;
                if (!(ok = wait_bar(bar(C::B_VFULL + sv), (v / NV) & 1, wc))) break;
                mbar_arrive_peer(lead(C::B_GO + v % NK));
            }
            if (!ok) {
                for (int v = issued - NV < 0 ? 0 : issued - NV; v < issued; v++)
                    drain_bar(bar(C::B_VFULL + v % NV), (v / NV) & 1);
            }
        }
    } else if (warp == 13) {
        // ------------------------------------------------------------ MMA issuer (even CTA)
        if (lane == 0 && rank == 0) {
            constexpr uint32_t idS = idesc_bf16_f32(2 * kBM, kBN, false, false);
            constexpr uint32_t idSG = idesc_f16_f32(2 * kBM, kBN, false, false);
            constexpr uint32_t idPV = idesc_bf16_f32(2 * kBM, D, false, true);
            bool ok = wait_bar_cl(bar(C::B_K0READY), 0, wc);
            tc_fence_after();
            auto qk_head = [&](int v, int n) {
                const uint64_t dk = sdesc_sw128(sK + (v % NK) * C::KHALF, 16, 1024);
                const uint64_t dq = sdesc_sw128(sQ + n * C::QTILE, 16, 1024);
                const uint32_t id = vis.remote(v) ? idSG : idS;
#pragma unroll
                for (int k = 0; k < D / 16; k++) {
                    const uint64_t oq = (uint64_t)(((k >> 2) * C::QREG + (k & 3) * 32) >> 4);
                    const uint64_t ok_ = (uint64_t)(((k >> 2) * C::KREG + (k & 3) * 32) >> 4);
                    mma2_f16_ss(tmem + 128u * n, dq + oq, dk + ok_, id, k > 0 ? 1u : 0u);
                }
                mma2_commit_mc(bar(C::B_SFULL + n), C::BOTH);
                if (n == 1) {
                    mma2_commit_mc(bar(C::B_KEMPTY + v % NK), C::BOTH);
                    if (v == NR - 1) mma2_commit_mc(bar(C::B_QFREE), C::BOTH);
                }
            };
            if (ok)
                for (int n = 0; n < 2; n++) qk_head(0, n);
            for (int v = 0; ok && v < T; v++) {
                const int sv = v % NV;
                const uint64_t dv = sdesc_sw128(sV + sv * C::VHALF, C::VHALF, 1024);
                for (int n = 0; n < 2; n++) {
                    if (n == 0) ok = wait_bar_cl(bar(C::B_GO + v % NK), (v / NK) & 1, wc);
                    else ok = wait_bar_cl(bar(C::B_PFULL + 1), v & 1, wc);
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll
                    for (int k = 0; k < kBN / 16; k++)
                        mma2_f16_ts(tmem + 256u + 128u * n, tmem + 128u * n + 8u * k,
                                    dv + (uint64_t)((k * 2048) >> 4), idPV, (v > 0 || k > 0) ? 1u : 0u);
                    mma2_commit_mc(bar(C::B_ODONE + n), C::BOTH);
                    if (n == 1) mma2_commit_mc(bar(C::B_VEMPTY + sv), C::BOTH);
                    if (v + 1 < T) qk_head(v + 1, n);
                }
            }
            if (!ok) {
                // no MMA may still run when the CTAs release TMEM and shared memory
                mma2_commit_mc(bar(C::B_DRAIN), 0x1);
                drain_bar(bar(C::B_DRAIN), 0);
            }
        }
        __syncwarp();
    } else if (warp < 8) {
        // ------------------------------------------------------------ softmax
        const int n = warp >> 2;  // head slot
        const int q4 = warp & 3;
        const int row = 32 * q4 + lane;
        const int i = i0 + row;
        const int h = h0 + n;
        const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
        const uint32_t tS = tmem + lane_base + 128u * n;
        const uint32_t tO = tmem + lane_base + 256u + 128u * n;
        const float sc = p.scale_log2;
        float m_used = -INFINITY, l = 0.f;  // m_used in log2 units
        bool ok = true;
        const jl::f32x2 sc2 = jl::f2(sc, sc);
        for (int v = 0; v < T; v++) {
            const int kt = vis.kt(v);
            const bool remote = vis.remote(v);
            const int j0 = kt * kBN;
            const bool band = jl::tile_class(i0, j0, kBM, kBN, S, w, g_cls) == jl::kTileBand;
            const bool masked = band || (j0 + kBN - 1 > i0) || (j0 + kBN > S);
            auto load_half = [&](int hh, uint32_t (&x)[64]) {
                tmem_ld32(tS + 64u * hh, *reinterpret_cast<uint32_t(*)[32]>(&x[0]));
                tmem_ld32(tS + 64u * hh + 32u, *reinterpret_cast<uint32_t(*)[32]>(&x[32]));
                tmem_ld_wait();
                if (masked) {
#pragma unroll
                    for (int e = 0; e < 64; e++) {
                        const int j = j0 + 64 * hh + e;
                        bool d = (j > i || j >= S);
                        if (band) d = d || (remote ? (i - j < w) : (i - j >= w));
                        if (d) x[e] = 0xff800000u;
                    }
                }
            };
            auto exp_half = [&](int hh, const uint32_t (&x)[64], jl::f32x2 nm, jl::f32x2 &lsum) {
#pragma unroll
                for (int q = 0; q < 2; q++) {
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; e++) {
                        const int k2 = 32 * q + 2 * e;
                        const jl::f32x2 t =
                            jl::fma2(jl::f2(__uint_as_float(x[k2]), __uint_as_float(x[k2 + 1])), sc2, nm);
                        float t0, t1;
                        jl::f2_split(t, t0, t1);
                        const jl::f32x2 pp = jl::f2(fast_exp2(t0), fast_exp2(t1));
                        lsum = jl::add2(lsum, pp);
                        pk[e] = jl::f2_to_bf16x2(pp);
                    }
                    tmem_st16(tS + 32u * hh + 16u * q, pk);
                }
            };
            if (!(ok = wait_bar_warp_cl(bar(C::B_SFULL + n), v & 1, wc))) break;
            tc_fence_after();
            float m_cur = m_used;
            jl::f32x2 lsum = jl::f2(0.f, 0.f);
#pragma unroll 1
            for (int hh = 0; hh < 2; hh++) {
                uint32_t x[64];
                load_half(hh, x);
                float cm = -INFINITY;
#pragma unroll
                for (int e = 0; e < 32; e++)
                    cm = jl::fmax3(cm, __uint_as_float(x[2 * e]), __uint_as_float(x[2 * e + 1]));
                cm *= sc;
                const bool raise = cm > m_cur + kRescaleThreshold;
                float f = 1.f;
                if (raise) {
                    if (m_cur == -INFINITY) {
                        m_cur = cm;
                    } else {
                        const float k = ceilf(cm - m_cur);
                        m_cur += k;
                        f = k >= 150.f ? 0.f : ldexpf(1.f, -(int)k);
                    }
                }
                if (hh > 0 && __any_sync(0xffffffffu, raise && f != 1.f)) {
                    lsum = jl::mul2(lsum, jl::f2(f, f));
                    tmem_st_wait();
#pragma unroll 1
                    for (int c2 = 0; c2 < 2; c2++) {
                        uint32_t pk[16];
                        tmem_ld16(tS + 16u * c2, pk);
                        tmem_ld_wait();
#pragma unroll
                        for (int e = 0; e < 16; e++)
                            pk[e] = jl::f2_to_bf16x2(jl::mul2(jl::bf16x2_to_f2(pk[e]), jl::f2(f, f)));
                        tmem_st16(tS + 16u * c2, pk);
                    }
                }
                const float m_off = (m_cur == -INFINITY) ? 0.f : m_cur;
                exp_half(hh, x, jl::f2(-m_off, -m_off), lsum);
            }
            const bool moved = m_cur != m_used;
            const bool need_o = moved && m_used != -INFINITY;
            const float factor = need_o ? exp2f(m_used - m_cur) : (moved ? 0.f : 1.f);
            l *= factor;
            if (v >= 1 && __any_sync(0xffffffffu, need_o)) {
                const float fo = need_o ? factor : 1.f;
                if (!(ok = wait_bar_warp_cl(bar(C::B_ODONE + n), (v - 1) & 1, wc))) break;
                tc_fence_after();
#pragma unroll 1
                for (int ch = 0; ch < D / 32; ch++) {
                    uint32_t o[32];
                    tmem_ld32(tO + 32u * ch, o);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 32; e++) o[e] = __float_as_uint(__uint_as_float(o[e]) * fo);
                    tmem_st32(tO + 32u * ch, o);
                }
            }
            m_used = m_cur;
            float l0, l1;
            jl::f2_split(lsum, l0, l1);
            l += l0 + l1;
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_peer(n == 0 ? lead(C::B_GO + v % NK) : lead(C::B_PFULL + 1));
        }
        // ------------------------------------------------------------ epilogue
        if (ok) ok = wait_bar_warp_cl(bar(C::B_ODONE + n), (T - 1) & 1, wc);
        if (ok) {
            tc_fence_after();
            if (!(l < INFINITY)) jl::record_status(p.status, JL_ERR_GUARD);
            const float inv_l = 1.f / l;
            const int il = i - p.pos0;
            __nv_bfloat16 *orow = p.out + (((size_t)b * p.q_rows + il) * p.Hq + h) * D;
#pragma unroll 1
            for (int ch = 0; ch < D / 32; ch++) {
                uint32_t o[32];
                tmem_ld32(tO + 32u * ch, o);
                tmem_ld_wait();
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; e++)
                    pk[e] = jl::pack_bf16x2(__uint_as_float(o[2 * e]) * inv_l, __uint_as_float(o[2 * e + 1]) * inv_l);
                if (i < S) {
                    uint4 *dst = reinterpret_cast<uint4 *>(orow + 32 * ch);
#pragma unroll
                    for (int q = 0; q < 4; q++)
                        dst[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
                }
            }
            if (i < S) p.lse[((size_t)b * p.Hq + h) * p.lse_stride + il] = (m_used + log2f(l)) * kLn2;
        }
    } else {
        // ------------------------------------------------------------ correction
        // As in prefill_kernel, for this CTA's half of every K tile: K(u) ready
        // (landed, and corrected if remote) -> one arrival per warp on the even
        // CTA's K0READY (u = 0) or GO[(u-1) % NK].  The final arrival (u = T) has
        // no K tile to order it after GO's phase for tile T-1-NK; the commit that
        // frees the stage of QK(T-NK) -- issued right after the issuer's wait on
        // that phase -- does, and it reaches this CTA's KEMPTY.
        const int t = threadIdx.x - 256;
        Corrector<D, 128> corq;
        Corrector<D, 64> cork;
        if (NR > 0) {
            corq.init(t, g, pt, rc);
            cork.init(t, g, pt, rc);
        }
        bool ok = wait_bar_warp(bar(C::B_QFULL), 0, wc);
        if (ok && NR > 0) {
#pragma unroll 1
            for (int n = 0; n < 2; n++) corq.run_q(sQ + n * C::QTILE, i0, p.qshift);
        }
        for (int u = 0; ok && u <= T; u++) {
            if (u < T) {
                const int sk = u % NK;
                if (!(ok = wait_bar_warp(bar(C::B_KFULL + sk), (u / NK) & 1, wc))) break;
                if (u < NR) cork.run_k(sK + sk * C::KHALF, u, 64 * (int)rank);
                if (u == NR && NR > 0 && !(ok = wait_bar_warp(bar(C::B_QFULL), 1, wc))) break;
                if (u <= NR) fence_proxy_async_smem();
            }
            if (u == T && T - 1 >= NK &&
                !(ok = wait_bar_warp_cl(bar(C::B_KEMPTY + (T - NK) % NK), ((T - NK) / NK) & 1, wc)))
                break;
            __syncwarp();
            if (lane == 0) mbar_arrive_peer(u == 0 ? lead(C::B_K0READY) : lead(C::B_GO + (u - 1) % NK));
        }
    }

    // every MMA has completed (the epilogues waited for the last ones, an
    // aborting issuer drained them) before either CTA releases TMEM or exits
    __syncwarp();
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    if (warp == 13) tmem_dealloc2(tmem, 512);
}

int launch_pair(const CUtensorMap &tq, const CUtensorMap &tk64, const CUtensorMap &tv, const Params &p,
                const jl::PhaseTable &pt, const RotConsts &rc, cudaStream_t st)
{
    cudaError_t e = cudaFuncSetAttribute(prefill_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         PairCfg::SMEM);
    if (e != cudaSuccess) return jl::cuda_status(e);
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3((unsigned)(p.pairs * p.n_qtiles), (unsigned)(p.B * p.Hkv), 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = PairCfg::SMEM;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return jl::cuda_status(cudaLaunchKernelEx(&cfg, prefill_pair_kernel, tq, tk64, tv, p, pt, rc));
}

// ---------------------------------------------------------------- few-key rows
// Rows at positions below kFewKeyRows see fewer than kFewKeyRows keys.  The
// tile kernel rounds to 16 bits what it feeds the tensor cores: P to bf16
// (relative error up to 2^-9) while out and lse are normalised by the fp32
// sum of P, and, in the remote view, the corrected q and k to fp16 (2^-11
// each, about 4e-4 on one score).  Over many keys these errors average down in
// out and in the log-sum-exp; over a handful they do not (a row of two keys
// whose V rows differ by 8 can miss out by 2^-9 * 4 plus its own rounding).
// This kernel recomputes those rows in fp32 on CUDA cores -- the same
// definition, key by key -- and overwrites what the tile kernel wrote for
// them.  Its cost is at most kFewKeyRows rows of at most kFewKeyRows keys per
// call.
constexpr int kFewKeyRows = 256;
constexpr int kFewThreads = 128;

struct FewRowParams {
    const __nv_bfloat16 *q;  // row 0 at position pos0; batch stride q_rows rows
    const __nv_bfloat16 *k;  // [B, n_cap, Hkv, D]
    const __nv_bfloat16 *v;
    __nv_bfloat16 *out;      // as q
    float *lse;              // column 0 at position pos0; row stride lse_stride
    int Hq, Hkv, q_rows, lse_stride, n_cap;
    int pos0;    // position of q / out / lse row 0
    int first;   // position of the first row recomputed (block x = 0)
    int w, g;
    int qshift;   // added to the query's correction offset
    int sliding;  // keys with i - j >= w are not attended
    float scale_log2;
};

template <int D>
__global__ void __launch_bounds__(kFewThreads)
    few_key_rows_kernel(const FewRowParams a, const __grid_constant__ jl::PhaseTable pt)
{
    constexpr int HALF = D / 2;
    __shared__ float sq[D], sqg[D], sc[kFewKeyRows], red[kFewThreads / 32];
    const int i = a.first + (int)blockIdx.x;  // absolute position of the query row
    const int h = (int)blockIdx.y, b = (int)blockIdx.z;
    const int hk = h / (a.Hq / a.Hkv);
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const size_t qrow = ((size_t)b * a.q_rows + (i - a.pos0)) * a.Hq + h;
    for (int d = t; d < D; d += kFewThreads) sq[d] = __bfloat162float(a.q[qrow * D + d]);
    __syncthreads();
    const int di = jl::delta_pos(i, a.g) + a.qshift;
    for (int d = t; d < HALF; d += kFewThreads) {
        float sn, cs;
        jl::phase_sincos(di, pt.f[d], &sn, &cs);
        sqg[d] = sq[d] * cs - sq[d + HALF] * sn;
        sqg[d + HALF] = sq[d + HALF] * cs + sq[d] * sn;
    }
    __syncthreads();
    // scores (log2 units) of keys 0..i: exact inside the window, corrected outside
    for (int j = t; j <= i; j += kFewThreads) {
        const __nv_bfloat16 *kj = a.k + (((size_t)b * a.n_cap + j) * a.Hkv + hk) * D;
        float acc = 0.f;
        const uint4 *k16 = reinterpret_cast<const uint4 *>(kj);  // 8 bf16 per 16-byte load
        if (i - j < a.w || (a.g == 1 && !a.sliding)) {
            float acc2 = 0.f;
#pragma unroll 4
            for (int c8 = 0; c8 < D / 8; c8++) {
                const uint4 u = k16[c8];
                const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int e = 0; e < 4; e++) {
                    acc = fmaf(sq[8 * c8 + 2 * e], jl::bf16lo(w4[e]), acc);
                    acc2 = fmaf(sq[8 * c8 + 2 * e + 1], jl::bf16hi(w4[e]), acc2);
                }
            }
            acc += acc2;
        } else if (a.sliding) {
            acc = -INFINITY;  // outside a sliding window: not attended
        } else {
            const int dj = jl::delta_pos(j, a.g);
#pragma unroll 1
            for (int c8 = 0; c8 < HALF / 8; c8++) {
                const uint4 ul = k16[c8], uh = k16[HALF / 8 + c8];
                const uint32_t lo4[4] = {ul.x, ul.y, ul.z, ul.w}, hi4[4] = {uh.x, uh.y, uh.z, uh.w};
#pragma unroll
                for (int e = 0; e < 8; e++) {
                    const int d = 8 * c8 + e;
                    float sn, cs;
                    jl::phase_sincos(dj, pt.f[d], &sn, &cs);
                    const float x = (e & 1) ? jl::bf16hi(lo4[e / 2]) : jl::bf16lo(lo4[e / 2]);
                    const float y = (e & 1) ? jl::bf16hi(hi4[e / 2]) : jl::bf16lo(hi4[e / 2]);
                    acc = fmaf(sqg[d], x * cs - y * sn, acc);
                    acc = fmaf(sqg[d + HALF], y * cs + x * sn, acc);
                }
            }
        }
        sc[j] = acc * a.scale_log2;
    }
    __syncthreads();
    // row maximum and sum of 2^(s - m)
    float m = -INFINITY;
    for (int j = t; j <= i; j += kFewThreads) m = fmaxf(m, sc[j]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) red[warp] = m;
    __syncthreads();
    m = red[0];
#pragma unroll
    for (int q = 1; q < kFewThreads / 32; q++) m = fmaxf(m, red[q]);
    __syncthreads();
    float l = 0.f;
    for (int j = t; j <= i; j += kFewThreads) {
        const float pj = exp2f(sc[j] - m);
        sc[j] = pj;
        l += pj;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    if (lane == 0) red[warp] = l;
    __syncthreads();
    l = 0.f;
#pragma unroll
    for (int q = 0; q < kFewThreads / 32; q++) l += red[q];
    const float inv_l = 1.f / l;
    for (int d = t; d < D; d += kFewThreads) {
        const __nv_bfloat16 *vd = a.v + ((size_t)b * a.n_cap * a.Hkv + hk) * D + d;
        const size_t vs = (size_t)a.Hkv * D;  // one key further
        float o[4] = {0.f, 0.f, 0.f, 0.f};
        int j = 0;
        for (; j + 3 <= i; j += 4) {
#pragma unroll
            for (int u = 0; u < 4; u++) o[u] = fmaf(sc[j + u], __bfloat162float(vd[(j + u) * vs]), o[u]);
        }
        for (; j <= i; j++) o[0] = fmaf(sc[j], __bfloat162float(vd[j * vs]), o[0]);
        a.out[qrow * D + d] = __float2bfloat16_rn(((o[0] + o[1]) + (o[2] + o[3])) * inv_l);
    }
    if (t == 0) a.lse[((size_t)b * a.Hq + h) * a.lse_stride + (i - a.pos0)] = (m + log2f(l)) * kLn2;
}

// ---------------------------------------------------------------- host side
template <int D, int NH>
int launch(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv, const Params &p,
           const jl::PhaseTable &pt, const RotConsts &rc, cudaStream_t st)
{
    auto kern = prefill_kernel<D, NH>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<D, NH>::SMEM);
    if (e != cudaSuccess) return jl::cuda_status(e);
    dim3 grid((unsigned)(p.pairs * p.n_qtiles), (unsigned)(p.B * p.Hkv), 1);
    kern<<<grid, kThreads, Cfg<D, NH>::SMEM, st>>>(tq, tk, tv, p, pt, rc);
    return jl::cuda_status(cudaGetLastError());
}

}  // namespace

// Arguments shared by every launch of one prefill call (already validated).
struct PrefillCall {
    const void *k, *v;
    int B, Hq, Hkv, n_cap, D, w;
    int q_rows, lse_stride;  // batch stride of q / out (rows), row stride of lse
    int sliding;
    int pair;  // kernel choice: 0 one CTA (JL_PREFILL_ONE_CTA), 1 automatic, 2 two SMs (JL_PREFILL_CTA_PAIR)
    jl::PhaseTable pt;
    float scale_log2;
    cudaStream_t st;
};

// One launch: the Sq query rows at positions pos0..pos0+Sq-1 (q, out and lse
// point at the first of them) over the keys at positions 0..pos0+Sq-1, with
// group factor g and the query's correction offset shifted by qshift.
static int prefill_rows(const PrefillCall &c, const void *q, void *out, float *lse, int Sq, int pos0,
                        int g, int qshift)
{
    const int S = pos0 + Sq;
    const int D = c.D;
    const long long n_qtiles = ((long long)Sq + kBM - 1) / kBM;
    if ((long long)c.Hq * n_qtiles > 0x7fffffffLL) return JL_ERR_OVERFLOW;
    CUtensorMap tq, tk, tv;
    if (!jl::make_bshd_map(&tq, q, c.B, Sq, c.q_rows, c.Hq, D, 64, 128, true) ||
        !jl::make_bshd_map(&tk, c.k, c.B, S, c.n_cap, c.Hkv, D, 64, 128, true) ||
        !jl::make_bshd_map(&tv, c.v, c.B, S, c.n_cap, c.Hkv, D, 64, 128, true))
        return JL_ERR_CUDA;
    Params p;
    p.out = (__nv_bfloat16 *)out;
    p.lse = lse;
    p.status = jl::status_word_ptr();
    p.B = c.B;
    p.Hq = c.Hq;
    p.Hkv = c.Hkv;
    p.S = S;
    p.Sq = Sq;
    p.pos0 = pos0;
    p.w = c.w;
    p.g = g;
    p.grp = c.Hq / c.Hkv;
    p.n_qtiles = (int)n_qtiles;
    p.q_rows = c.q_rows;
    p.lse_stride = c.lse_stride;
    p.qshift = qshift;
    p.sliding = c.sliding;
    // two heads of a GQA group per CTA when the group size is even
    const int nh = (p.grp % 2 == 0) ? 2 : 1;
    p.pairs = p.grp / nh;
    p.scale_log2 = c.scale_log2;
    // step rotations of the correction (rows per step: 16 at D = 128, 32 at D = 64)
    RotConsts rc;
    make_rot_consts(c.pt, D, g, &rc);
    int rc_launch;
    // The two-SM kernel applies at D = 128 with four heads (or a multiple) per
    // kv head; by default it runs where the launch has remote keys, since it
    // halves each SM's correction work, and the one-CTA kernel runs the plain
    // (all-exact) launches, whose handshakes it keeps on one SM.
    const bool pair_fits = D == 128 && p.grp % 4 == 0;
    const bool has_remote = g > 1 && !c.sliding && S - 1 >= c.w;
    if (pair_fits && (c.pair == 2 || (c.pair == 1 && has_remote))) {
        // four heads per kv head or a multiple: a CTA pair per query tile of four heads
        CUtensorMap tk64;
        if (!jl::make_bshd_map(&tk64, c.k, c.B, S, c.n_cap, c.Hkv, D, 64, 64, true)) return JL_ERR_CUDA;
        rc_launch = launch_pair(tq, tk64, tv, p, c.pt, rc, c.st);
    } else if (D == 128)
        rc_launch = nh == 2 ? launch<128, 2>(tq, tk, tv, p, c.pt, rc, c.st) : launch<128, 1>(tq, tk, tv, p, c.pt, rc, c.st);
    else
        rc_launch = nh == 2 ? launch<64, 2>(tq, tk, tv, p, c.pt, rc, c.st) : launch<64, 1>(tq, tk, tv, p, c.pt, rc, c.st);
    if (rc_launch != JL_OK) return rc_launch;
    // rows below kFewKeyRows are redone in fp32
    const int few_lo = pos0;
    const int few_hi = S < kFewKeyRows ? S : kFewKeyRows;
    if (few_lo < few_hi) {
        FewRowParams f;
        f.q = (const __nv_bfloat16 *)q;
        f.k = (const __nv_bfloat16 *)c.k;
        f.v = (const __nv_bfloat16 *)c.v;
        f.out = (__nv_bfloat16 *)out;
        f.lse = lse;
        f.Hq = c.Hq;
        f.Hkv = c.Hkv;
        f.q_rows = c.q_rows;
        f.lse_stride = c.lse_stride;
        f.n_cap = c.n_cap;
        f.pos0 = pos0;
        f.first = few_lo;
        f.w = c.w;
        f.g = g;
        f.qshift = qshift;
        f.sliding = c.sliding;
        f.scale_log2 = c.scale_log2;
        dim3 grid((unsigned)(few_hi - few_lo), (unsigned)c.Hq, (unsigned)c.B);
        if (D == 128) few_key_rows_kernel<128><<<grid, kFewThreads, 0, c.st>>>(f, c.pt);
        else few_key_rows_kernel<64><<<grid, kFewThreads, 0, c.st>>>(f, c.pt);
        return jl::cuda_status(cudaGetLastError());
    }
    return JL_OK;
}

// Prefill of Sq queries at positions n_past..n_past+Sq-1 over the keys at
// positions 0..n_past+Sq-1 (k / v: [B, n_cap, Hkv, D], rows past the keys
// are never read), s = n_past + Sq, with the variant flags of the header.
static int prefill_impl(const void *q, const void *k, const void *v, void *out, float *lse, int B, int Hq,
                        int Hkv, int Sq, int n_past, int n_cap, int D, int L_pre, int w, double theta,
                        unsigned flags, void *stream)
{
    if (!q || !k || !v || !out || !lse) return JL_ERR_ARG;
    if (B < 1 || Hq < 1 || Hkv < 1 || Sq < 1 || n_past < 0 || L_pre < 1 || w < 1 ||
        !(theta > 0.0) || Hq % Hkv != 0)
        return JL_ERR_ARG;
    if (flags & ~(unsigned)(JL_VARIANT_PER_QUERY_G | JL_VARIANT_SLIDING | JL_VARIANT_QUERY_SHIFT |
                            JL_PREFILL_CTA_PAIR | JL_PREFILL_ONE_CTA))
        return JL_ERR_ARG;
    if ((flags & JL_PREFILL_CTA_PAIR) && (flags & JL_PREFILL_ONE_CTA)) return JL_ERR_ARG;
    const int pair = (flags & JL_PREFILL_CTA_PAIR) ? 2 : (flags & JL_PREFILL_ONE_CTA) ? 0 : 1;
    flags &= ~(unsigned)(JL_PREFILL_CTA_PAIR | JL_PREFILL_ONE_CTA);
    if ((flags & JL_VARIANT_SLIDING) && flags != JL_VARIANT_SLIDING) return JL_ERR_ARG;
    if ((flags & JL_VARIANT_PER_QUERY_G) && (flags & JL_VARIANT_QUERY_SHIFT)) return JL_ERR_UNSUPPORTED;
    if ((long long)n_past + Sq > 0x7fffffffLL) return JL_ERR_OVERFLOW;
    const int S = n_past + Sq;
    if (n_cap < S) return JL_ERR_ARG;
    if (D != 64 && D != 128) return JL_ERR_UNSUPPORTED;
    if (!jl::aligned16(q) || !jl::aligned16(k) || !jl::aligned16(v) || !jl::aligned16(out) ||
        !jl::aligned16(lse))
        return JL_ERR_ALIGN;
    if ((long long)B * Sq * Hq * D > ((long long)1 << 46) ||
        (long long)B * n_cap * Hkv * D > ((long long)1 << 46))
        return JL_ERR_OVERFLOW;
    if ((long long)B * Hkv > 65535 || Hq > 65535) return JL_ERR_OVERFLOW;
    long long g_call = jl::group_factor_host(S, L_pre);
    int qshift = 0;
    if (flags & JL_VARIANT_QUERY_SHIFT) {
        g_call = jl::group_factor_shift_host(S, L_pre, w);
        if (g_call < 1) return JL_ERR_ARG;  // no g keeps the shifted distances inside L_pre
        qshift = (int)(w - w / g_call);
    }
    if (g_call > 0x7fffffffLL) return JL_ERR_OVERFLOW;
    PrefillCall c;
    c.k = k;
    c.v = v;
    c.B = B;
    c.Hq = Hq;
    c.Hkv = Hkv;
    c.n_cap = n_cap;
    c.D = D;
    c.w = w;
    c.q_rows = Sq;
    c.lse_stride = Sq;
    c.sliding = (flags & JL_VARIANT_SLIDING) ? 1 : 0;
    c.pair = pair;
    if (!jl::make_phase_table(&c.pt, D, theta)) return JL_ERR_ARG;
    c.scale_log2 = (float)(1.0 / sqrt((double)D) * 1.4426950408889634);
    c.st = (cudaStream_t)stream;
    if (c.sliding) return prefill_rows(c, q, out, lse, Sq, n_past, 1, 0);
    if (!(flags & JL_VARIANT_PER_QUERY_G)) return prefill_rows(c, q, out, lse, Sq, n_past, (int)g_call, qshift);
    // per-query group factor: row i has s = i + 1, so g = ceil((i + 1) / L_pre) is
    // constant on the rows [(g-1) L_pre, g L_pre); each such range is one launch whose
    // rows see the keys before them -- the chunk of a prefill of length g L_pre
    const size_t row_bytes = (size_t)Hq * D * sizeof(__nv_bfloat16);
    for (int a = n_past; a < S;) {
        const long long g = jl::group_factor_host((long long)a + 1, L_pre);
        const long long end_ll = g * (long long)L_pre;
        const int b = end_ll < S ? (int)end_ll : S;
        const size_t r = (size_t)(a - n_past);
        const int rc = prefill_rows(c, (const char *)q + r * row_bytes, (char *)out + r * row_bytes, lse + r,
                                    b - a, a, (int)g, 0);
        if (rc != JL_OK) return rc;
        a = b;
    }
    return JL_OK;
}

extern "C" int jl_bifocal_prefill(const void *q, const void *k, const void *v, void *out, float *lse,
                                  int B, int Hq, int Hkv, int S, int D, int L_pre, int w,
                                  double theta, void *stream)
{
    return prefill_impl(q, k, v, out, lse, B, Hq, Hkv, S, 0, S, D, L_pre, w, theta, 0u, stream);
}

extern "C" int jl_bifocal_prefill_chunk(const void *q, const void *k_cache, const void *v_cache,
                                        void *out, float *lse, int B, int Hq, int Hkv, int S_new,
                                        int n_past, int n_cap, int D, int L_pre, int w, double theta,
                                        void *stream)
{
    return prefill_impl(q, k_cache, v_cache, out, lse, B, Hq, Hkv, S_new, n_past, n_cap, D, L_pre, w,
                        theta, 0u, stream);
}

extern "C" int jl_bifocal_prefill_ex(const void *q, const void *k_cache, const void *v_cache, void *out,
                                     float *lse, int B, int Hq, int Hkv, int S_new, int n_past, int n_cap,
                                     int D, int L_pre, int w, double theta, unsigned flags, void *stream)
{
    return prefill_impl(q, k_cache, v_cache, out, lse, B, Hq, Hkv, S_new, n_past, n_cap, D, L_pre, w,
                        theta, flags, stream);
}
