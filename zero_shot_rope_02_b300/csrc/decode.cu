// Bifocal single-token decode over an exact-RoPE bf16 KV cache (split-KV).
//
// The cache keeps the original positions and is never rewritten; keys that
// fall outside the local window are corrected by the rotation R_{delta_j} at
// lookup time (ResearchPod transcript on caching; Jet-Long abstract: the
// correction is applied on the fly).  The query at position n-1 is corrected
// once by R_{delta_{n-1}}.
//
// HBM-bound.  A CTA owns one contiguous chunk of one kv head's keys and
// serves all Hq/Hkv query heads of that kv head.  A producer warp streams the
// chunk's K and V rows in 64-key blocks through a 3-stage TMA ring; four
// compute warps score a block (correcting its remote keys), fold it into a
// running log-sum-exp per head, and accumulate P.V, all from shared memory
// in packed f32x2 arithmetic.  The last CTA of each (batch, kv head) to
// finish merges the per-chunk partial statistics.
//
// Rotation angles of remote keys come from a chain of unit complex numbers:
// a thread's keys are KPS apart and, when g divides KPS, delta changes by
// the same amount every KPS keys, so each key's rotation is the previous one
// times a constant; the chain is re-anchored from the exact fixed-point
// phase every kReanchorBlocks blocks.  Other g take the exact phase per key.
//
// The paged variant serves a batch whose sequences have their own lengths:
// each CTA reads its sequence's length from the device and derives from it
// g, the exact / remote split and the chain's step rotation, and the
// producer finds each 64-key block's page in the sequence's block table.  Its
// split plan is sized for the longest sequence; splits past a shorter
// sequence's end load nothing and leave an empty partial for the merge.
#include <math.h>
#include <string.h>

#include "jl_common.cuh"
#include "sm100_ptx.cuh"

namespace {

using namespace jl::ptx;

constexpr int kCompute = 128;           // compute threads (4 warps)
constexpr int kThreads = kCompute + 32; // + one producer warp
constexpr int kKB = 64;                 // keys per block
constexpr int kNS = 3;                  // TMA ring stages
constexpr int kReanchorBlocks = 32;
constexpr float kLn2 = 0.6931471805599453f;

// Host-computed rotation per KPS keys for the chained angles, per pair d,
// as cosine / sine / negated-sine arrays (consecutive d load as one f32x2).
struct DecRot {
    alignas(8) float c[64];
    alignas(8) float s[64];
    alignas(8) float ns[64];
    int uni;  // g divides KPS
};

struct DecodeArgs {
    const __nv_bfloat16 *q;  // [B, Hq, D]
    __nv_bfloat16 *out;      // [B, Hq, D]
    float *lse;              // [B, Hq]
    int *counters;           // [B * Hkv]
    float *part_ml;          // [B, Hq, splits, 2]
    float *part_o;           // [B, Hq, splits, D]
    int *status;
    int Hq, Hkv, n, w, g, splits, chunk;
    int qshift;              // added to the query's correction offset (query-shift variant)
    float scale_log2;        // tau * log2(e)
    // paged variant: per-sequence lengths and the page table (device), the
    // pages' row count, table width and the pretrained window (g per sequence)
    const int *seq_lens;     // [B]
    const int *block_table;  // [B, max_pages]
    int page_size, max_pages, num_pages, L;
};

// Named barrier over the compute warps only (the producer warp never joins).
__device__ __forceinline__ void compute_sync()
{
    asm volatile("bar.sync 1, %0;" ::"n"(kCompute) : "memory");
}

template <int D, int GRP>
struct DecCfg {
    static constexpr int BLOCK_BYTES = kKB * D * 2;  // one K or V block
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = OFF_K + kNS * BLOCK_BYTES;
    static constexpr int OFF_Q = OFF_V + kNS * BLOCK_BYTES;   // fp32 [GRP][D] exact q
    static constexpr int OFF_QG = OFF_Q + GRP * D * 4;        // fp32 [GRP][D] corrected q
    static constexpr int OFF_SC = OFF_QG + GRP * D * 4;       // fp32 [GRP][kKB] scores / p
    static constexpr int OFF_ST = OFF_SC + GRP * kKB * 4;     // fp32 m[GRP], l[GRP], fac[GRP]
    static constexpr int OFF_MW = OFF_ST + 3 * GRP * 4 + 16;  // merge weights [GRP][256]
    static constexpr int OFF_BAR = (OFF_MW + GRP * 256 * 4 + 15) / 16 * 16;
    static constexpr int SMEM = OFF_BAR + 2 * kNS * 8 + 16;
    // end-of-chunk reduction buffer [KPS3][GRP][D] fp32 aliases the K/V ring
    static constexpr int VC = D / 8, KPS3 = kCompute / VC;
    static_assert(KPS3 * GRP * D * 4 <= 2 * kNS * BLOCK_BYTES, "reduction buffer");
};

// PAGED: the keys of sequence b live in pages of a shared pool, page p of it
// at block_table[b][p]; its length n_b comes from seq_lens[b] and sets its own
// g.  Otherwise the cache is [B, n_cap, Hkv, D] and every sequence has length n.
template <int D, int GRP, bool PAGED>
__global__ void __launch_bounds__(kThreads, 2)
    decode_kernel(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                  const DecodeArgs a, const __grid_constant__ jl::PhaseTable pt,
                  const __grid_constant__ DecRot rot)
{
    using C = DecCfg<D, GRP>;
    constexpr int HALF = D / 2;
    constexpr int CPK = D / 16;          // threads per key in scoring (8 pairs each)
    constexpr int KPS = kCompute / CPK;  // keys per scoring step (16 or 32)
    constexpr int ITEMS = kKB / KPS;     // scoring steps per block
    constexpr int VC = C::VC;            // threads per V row (8 dims each)
    constexpr int KPS3 = C::KPS3;        // keys per PV step
    constexpr int VITEMS = kKB / KPS3;

    extern __shared__ __align__(128) uint8_t smem[];
    float *sq = reinterpret_cast<float *>(smem + C::OFF_Q);
    float *sqg = reinterpret_cast<float *>(smem + C::OFF_QG);
    float *sc = reinterpret_cast<float *>(smem + C::OFF_SC);
    float *st_m = reinterpret_cast<float *>(smem + C::OFF_ST);
    float *st_l = st_m + GRP;
    float *st_f = st_l + GRP;
    float *mw = reinterpret_cast<float *>(smem + C::OFF_MW);
    const uint32_t sbase = smem_u32(smem);
    auto full = [&](int s) -> uint32_t { return sbase + C::OFF_BAR + 8u * s; };
    auto empty = [&](int s) -> uint32_t { return sbase + C::OFF_BAR + 8u * (kNS + s); };
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_BAR + 2 * kNS * 8);
    volatile int &s_last = *reinterpret_cast<volatile int *>(smem + C::OFF_BAR + 2 * kNS * 8 + 4);
    const WaitCtx wc{a.status, abort_flag};

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int split = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
    int n = a.n, g = a.g;
    if constexpr (PAGED) {
        // a length the plan or the page table cannot cover is clamped (never
        // read past either) and reported
        const int n_lim = min(a.max_pages * a.page_size, a.splits * a.chunk);
        n = a.seq_lens[b];
        if (n < 1 || n > n_lim) {
            if (tid == 0 && split == 0 && hk == 0) jl::record_status(a.status, JL_ERR_GUARD);
            n = min(max(n, 1), n_lim);
        }
        g = (n <= a.L) ? 1 : (n - 1) / a.L + 1;
    }
    const int j_begin = split * a.chunk;
    const int j_end = min(n, j_begin + a.chunk);
    const int nblk = (j_end - j_begin + kKB - 1) / kKB;
    const int j_split = (g > 1) ? max(0, n - a.w) : 0;  // keys below are remote

    if (tid == 0) {
        for (int s = 0; s < kNS; s++) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), kCompute / 32);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == kCompute / 32) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tmap(&tk);
            prefetch_tmap(&tv);
            int issued = 0;
            bool ok = true;
            for (int blk = 0; blk < nblk; blk++) {
                const int s = blk % kNS;
                if (!(ok = wait_bar(empty(s), ((blk / kNS) & 1) ^ 1, wc))) break;
                mbar_arrive_expect_tx(full(s), 2 * C::BLOCK_BYTES);
                const int row = j_begin + blk * kKB;
                int r_in = row, unit = b;
                if constexpr (PAGED) {
                    // a page id outside the pool reads zeros (TMA bounds), never
                    // faults, and is reported: those keys would score 0 with V = 0
                    unit = a.block_table[(size_t)b * a.max_pages + row / a.page_size];
                    r_in = row % a.page_size;
                    if ((unsigned)unit >= (unsigned)a.num_pages) jl::record_status(a.status, JL_ERR_GUARD);
                }
                tma_load_4d(sbase + C::OFF_K + s * C::BLOCK_BYTES, &tk, full(s), 0, hk, r_in, unit);
                tma_load_4d(sbase + C::OFF_V + s * C::BLOCK_BYTES, &tv, full(s), 0, hk, r_in, unit);
                issued = blk + 1;
            }
            if (!ok)
                for (int blk = issued - kNS < 0 ? 0 : issued - kNS; blk < issued; blk++)
                    drain_bar(full(blk % kNS), (blk / kNS) & 1);
        }
        return;
    }

    // ---------------------------------------------------------------- compute
    // exact and corrected query of the GRP heads of this kv head, fp32
    const __nv_bfloat16 *qb = a.q + ((size_t)b * a.Hq + (size_t)hk * GRP) * D;
    for (int e = tid; e < GRP * D; e += kCompute) sq[e] = __bfloat162float(qb[e]);
    if (tid < GRP) {
        st_m[tid] = -INFINITY;
        st_l[tid] = 0.f;
    }
    compute_sync();
    if (g > 1) {
        const int di = jl::delta_pos(n - 1, g) + a.qshift;
        for (int d = tid; d < HALF; d += kCompute) {
            float sn, cs;
            jl::phase_sincos(di, pt.f[d], &sn, &cs);
#pragma unroll
            for (int h = 0; h < GRP; h++) {
                const float x0 = sq[h * D + d], x1 = sq[h * D + d + HALF];
                sqg[h * D + d] = x0 * cs - x1 * sn;
                sqg[h * D + d + HALF] = x1 * cs + x0 * sn;
            }
        }
    }
    compute_sync();

    // scoring layout: thread (c, r) owns pairs 8c..8c+7 of keys r + KPS*i
    const int c = tid % CPK, r = tid / CPK;
    // PV layout: thread (dc, r3) owns dims 8dc..8dc+7 of keys r3 + KPS3*i
    const int dc = tid % VC, r3 = tid / VC;
    jl::f32x2 qr[GRP][8];  // this thread's 16 query values per head (pairs of consecutive dims)
    int qmode = -1;        // which query qr holds: 0 exact, 1 corrected
    auto load_q = [&](int mode) {
        const float *src = mode ? sqg : sq;
#pragma unroll
        for (int h = 0; h < GRP; h++)
#pragma unroll
            for (int e = 0; e < 4; e++) {
                qr[h][e] = jl::f2(src[h * D + 8 * c + 2 * e], src[h * D + 8 * c + 2 * e + 1]);
                qr[h][4 + e] = jl::f2(src[h * D + HALF + 8 * c + 2 * e], src[h * D + HALF + 8 * c + 2 * e + 1]);
            }
        qmode = mode;
    };
    // rotation chain of this thread's next remote key
    jl::f32x2 zc[4], zs[4];
    int chain_next = -1;  // key the chain currently refers to
    const bool uni = PAGED ? (KPS % g == 0) : (rot.uni != 0);
    auto anchor = [&](int j) {
        const int dj = jl::delta_pos(j, g);
#pragma unroll
        for (int q = 0; q < 4; q++) {
            float s0, c0, s1, c1;
            jl::phase_sincos(dj, pt.f[8 * c + 2 * q], &s0, &c0);
            jl::phase_sincos(dj, pt.f[8 * c + 2 * q + 1], &s1, &c1);
            zc[q] = jl::f2(c0, c1);
            zs[q] = jl::f2(s0, s1);
        }
    };
    // the chain's per-KPS-keys rotation for this thread's pairs, in registers
    jl::f32x2 rcs[4], rsn[4], rns[4];
#pragma unroll
    for (int q = 0; q < 4; q++) {
        if constexpr (PAGED) {
            // this sequence's g: delta moves by KPS/g - KPS per KPS keys (g | KPS)
            const int step = KPS / g - KPS;
            float s0, c0, s1, c1;
            jl::phase_sincos(step, pt.f[8 * c + 2 * q], &s0, &c0);
            jl::phase_sincos(step, pt.f[8 * c + 2 * q + 1], &s1, &c1);
            rcs[q] = jl::f2(c0, c1);
            rsn[q] = jl::f2(s0, s1);
            rns[q] = jl::f2(-s0, -s1);
        } else {
            rcs[q] = *reinterpret_cast<const jl::f32x2 *>(rot.c + 8 * c + 2 * q);
            rsn[q] = *reinterpret_cast<const jl::f32x2 *>(rot.s + 8 * c + 2 * q);
            rns[q] = *reinterpret_cast<const jl::f32x2 *>(rot.ns + 8 * c + 2 * q);
        }
    }
    jl::f32x2 acc[GRP][4];
#pragma unroll
    for (int h = 0; h < GRP; h++)
#pragma unroll
        for (int e = 0; e < 4; e++) acc[h][e] = jl::f2(0.f, 0.f);

    bool ok = true;
    for (int blk = 0; blk < nblk; blk++) {
        const int s = blk % kNS;
        if (!(ok = wait_bar_warp(full(s), (blk / kNS) & 1, wc))) break;
        const int j0 = j_begin + blk * kKB;
        const uint8_t *kblk = smem + C::OFF_K + s * C::BLOCK_BYTES;
        const uint8_t *vblk = smem + C::OFF_V + s * C::BLOCK_BYTES;
        const bool any_remote = j0 < j_split;
        const bool any_exact = j0 + kKB > j_split;

        // ---- scores of this block (log2 units), one pass per view present
        for (int mode = any_remote ? 1 : 0; mode >= (any_exact ? 0 : 1); mode--) {
            if (qmode != mode) load_q(mode);
#pragma unroll 1
            for (int it = 0; it < ITEMS; it++) {
                const int kk = r + KPS * it;
                const int j = j0 + kk;
                const uint4 lo4 = *reinterpret_cast<const uint4 *>(kblk + kk * (D * 2) + 16 * c);
                const uint4 hi4 = *reinterpret_cast<const uint4 *>(kblk + kk * (D * 2) + D + 16 * c);
                const uint32_t lw[4] = {lo4.x, lo4.y, lo4.z, lo4.w};
                const uint32_t hw[4] = {hi4.x, hi4.y, hi4.z, hi4.w};
                jl::f32x2 kx[8];
                if (mode == 1) {
                    // corrected key: (x, y) -> (x c - y s, y c + x s)
                    if (!uni || chain_next != j || ((j - j_begin) / kKB) % kReanchorBlocks == 0 && it == 0)
                        anchor(j);
#pragma unroll
                    for (int q = 0; q < 4; q++) {
                        const jl::f32x2 x = jl::bf16x2_to_f2(lw[q]), y = jl::bf16x2_to_f2(hw[q]);
                        const jl::f32x2 ny = y ^ 0x8000000080000000ull;
                        kx[q] = jl::fma2(x, zc[q], jl::mul2(ny, zs[q]));
                        kx[4 + q] = jl::fma2(y, zc[q], jl::mul2(x, zs[q]));
                    }
                    if (uni) {
                        // advance the chain to key j + KPS
#pragma unroll
                        for (int q = 0; q < 4; q++) {
                            const jl::f32x2 nc = jl::fma2(zc[q], rcs[q], jl::mul2(zs[q], rns[q]));
                            const jl::f32x2 ns = jl::fma2(zs[q], rcs[q], jl::mul2(zc[q], rsn[q]));
                            zc[q] = nc;
                            zs[q] = ns;
                        }
                        chain_next = j + KPS;
                    }
                } else {
#pragma unroll
                    for (int q = 0; q < 4; q++) {
                        kx[q] = jl::bf16x2_to_f2(lw[q]);
                        kx[4 + q] = jl::bf16x2_to_f2(hw[q]);
                    }
                }
                float part[GRP];
#pragma unroll
                for (int h = 0; h < GRP; h++) {
                    jl::f32x2 t = jl::mul2(qr[h][0], kx[0]);
#pragma unroll
                    for (int e = 1; e < 8; e++) t = jl::fma2(qr[h][e], kx[e], t);
                    float t0, t1;
                    jl::f2_split(t, t0, t1);
                    part[h] = t0 + t1;
                }
#pragma unroll
                for (int h = 0; h < GRP; h++)
#pragma unroll
                    for (int o = 1; o < CPK; o <<= 1) part[h] += __shfl_xor_sync(0xffffffffu, part[h], o);
                const bool mine = (j < j_split) == (mode == 1);
                const bool valid = j < j_end;
#pragma unroll
                for (int h = 0; h < GRP; h++)
                    if (h % CPK == c && mine)
                        sc[h * kKB + kk] = valid ? part[h] * a.scale_log2 : -INFINITY;
            }
        }
        compute_sync();

        // ---- running log-sum-exp per head: warp h folds the block in
        for (int h = warp; h < GRP; h += kCompute / 32) {
            const float s0 = sc[h * kKB + lane], s1 = sc[h * kKB + lane + 32];
            float bm = fmaxf(s0, s1);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, o));
            const float m_old = st_m[h];
            const float m_new = fmaxf(m_old, bm);
            const float off = (m_new == -INFINITY) ? 0.f : m_new;
            const float p0 = exp2f(s0 - off), p1 = exp2f(s1 - off);
            sc[h * kKB + lane] = p0;
            sc[h * kKB + lane + 32] = p1;
            float sum = p0 + p1;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
            if (lane == 0) {
                // an infinite or NaN score (an input or corrected key out of range)
                if (!(sum < INFINITY)) jl::record_status(a.status, JL_ERR_GUARD);
                const float fac = (m_old == -INFINITY) ? 0.f : exp2f(m_old - off);
                st_l[h] = st_l[h] * fac + sum;
                st_m[h] = m_new;
                st_f[h] = fac;
            }
        }
        compute_sync();

        // ---- P . V
#pragma unroll
        for (int h = 0; h < GRP; h++) {
            const jl::f32x2 f = jl::f2(st_f[h], st_f[h]);
#pragma unroll
            for (int e = 0; e < 4; e++) acc[h][e] = jl::mul2(acc[h][e], f);
        }
#pragma unroll 2
        for (int it = 0; it < VITEMS; it++) {
            const int kk = r3 + KPS3 * it;
            uint4 v4 = *reinterpret_cast<const uint4 *>(vblk + kk * (D * 2) + 16 * dc);
            // a page's rows past the sequence hold whatever the pool held: zero
            // them (their p is 0, but 0 * NaN would still poison O)
            if (PAGED && j0 + kk >= j_end) v4 = make_uint4(0u, 0u, 0u, 0u);
            const jl::f32x2 vx[4] = {jl::bf16x2_to_f2(v4.x), jl::bf16x2_to_f2(v4.y), jl::bf16x2_to_f2(v4.z),
                                     jl::bf16x2_to_f2(v4.w)};
#pragma unroll
            for (int h = 0; h < GRP; h++) {
                const float pv = sc[h * kKB + kk];
                const jl::f32x2 p2 = jl::f2(pv, pv);
#pragma unroll
                for (int e = 0; e < 4; e++) acc[h][e] = jl::fma2(p2, vx[e], acc[h][e]);
            }
        }
        // this warp is done with stage s (scores of the next block overwrite
        // sc only after the next compute_sync, which every warp reaches after
        // its PV)
        __syncwarp();
        if (lane == 0) mbar_arrive(empty(s));
        compute_sync();
    }
    if (!ok) return;

    // ---- reduce the KPS3 key slots; o[h][d] unnormalised (buffer aliases the ring)
    float *red = reinterpret_cast<float *>(smem + C::OFF_K);
#pragma unroll
    for (int h = 0; h < GRP; h++)
#pragma unroll
        for (int e = 0; e < 4; e++) {
            float lo, hi;
            jl::f2_split(acc[h][e], lo, hi);
            red[(r3 * GRP + h) * D + dc * 8 + 2 * e] = lo;
            red[(r3 * GRP + h) * D + dc * 8 + 2 * e + 1] = hi;
        }
    compute_sync();
    const size_t hq0 = (size_t)b * a.Hq + (size_t)hk * GRP;
    if (a.splits == 1) {
        for (int t = tid; t < GRP * D; t += kCompute) {
            const int h = t / D, d = t % D;
            float o = 0.f;
#pragma unroll
            for (int q = 0; q < KPS3; q++) o += red[(q * GRP + h) * D + d];
            a.out[(hq0 + h) * D + d] = __float2bfloat16_rn(o / st_l[h]);
        }
        if (tid < GRP) a.lse[hq0 + tid] = (st_m[tid] + log2f(st_l[tid])) * kLn2;
        return;
    }
    for (int t = tid; t < GRP * D; t += kCompute) {
        const int h = t / D, d = t % D;
        float o = 0.f;
#pragma unroll
        for (int q = 0; q < KPS3; q++) o += red[(q * GRP + h) * D + d];
        a.part_o[((hq0 + h) * a.splits + split) * D + d] = o;
    }
    if (tid < GRP) {
        a.part_ml[((hq0 + tid) * a.splits + split) * 2 + 0] = st_m[tid];
        a.part_ml[((hq0 + tid) * a.splits + split) * 2 + 1] = st_l[tid];
    }
    __threadfence();
    compute_sync();
    if (tid == 0) {
        const int ticket = atomicAdd(&a.counters[b * a.Hkv + hk], 1);
        s_last = (ticket == a.splits - 1);
    }
    compute_sync();
    if (!s_last) return;
    __threadfence();

    // ---- last CTA of this (b, kv head): merge the partial statistics
    // weights w_s = 2^(m_s - M) with M = max m_s; L = sum l_s w_s
    for (int h = warp; h < GRP; h += kCompute / 32) {
        const float *ml = a.part_ml + (hq0 + h) * a.splits * 2;
        float m = -INFINITY;
        for (int q = lane; q < a.splits; q += 32) m = fmaxf(m, __ldcg(ml + 2 * q));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        const float off = (m == -INFINITY) ? 0.f : m;
        float L = 0.f;
        for (int q = lane; q < a.splits; q += 32) {
            const float wgt = exp2f(__ldcg(ml + 2 * q) - off);
            mw[h * 256 + q] = wgt;
            L += wgt * __ldcg(ml + 2 * q + 1);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
        if (lane == 0) {
            st_m[h] = m;
            st_l[h] = L;
        }
    }
    compute_sync();
    // each thread: 4 consecutive dims of one head, 8 splits' loads in flight
    for (int t = tid; t < GRP * D / 4; t += kCompute) {
        const int h = (4 * t) / D, d = (4 * t) % D;
        const float *po = a.part_o + (hq0 + h) * a.splits * D + d;
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
        int q = 0;
        for (; q + 8 <= a.splits; q += 8) {
            float4 x[8];
#pragma unroll
            for (int u = 0; u < 8; u++) x[u] = __ldcg(reinterpret_cast<const float4 *>(po + (size_t)(q + u) * D));
#pragma unroll
            for (int u = 0; u < 8; u++) {
                const float wgt = mw[h * 256 + q + u];
                o.x = fmaf(wgt, x[u].x, o.x);
                o.y = fmaf(wgt, x[u].y, o.y);
                o.z = fmaf(wgt, x[u].z, o.z);
                o.w = fmaf(wgt, x[u].w, o.w);
            }
        }
        for (; q < a.splits; q++) {
            const float4 x = __ldcg(reinterpret_cast<const float4 *>(po + (size_t)q * D));
            const float wgt = mw[h * 256 + q];
            o.x = fmaf(wgt, x.x, o.x);
            o.y = fmaf(wgt, x.y, o.y);
            o.z = fmaf(wgt, x.z, o.z);
            o.w = fmaf(wgt, x.w, o.w);
        }
        const float inv = 1.f / st_l[h];
        __nv_bfloat16 *dst = a.out + (hq0 + h) * D + d;
        *reinterpret_cast<uint2 *>(dst) = make_uint2(jl::pack_bf16x2(o.x * inv, o.y * inv),
                                                     jl::pack_bf16x2(o.z * inv, o.w * inv));
    }
    if (tid < GRP) a.lse[hq0 + tid] = (st_m[tid] + log2f(st_l[tid])) * kLn2;
    if (tid == 0) a.counters[b * a.Hkv + hk] = 0;  // ready for the next call
}

// Split plan: as many CTAs as the kernel keeps resident (two per SM: shared
// memory and registers allow two), at most 256 splits per (batch, kv head),
// chunks a multiple of the 64-key block.  splits_cap bounds splits for every
// n, and the workspace is sized by it, so one workspace serves every cache
// length for the same (B, Hq, Hkv, D).
struct Plan {
    int splits, chunk, splits_cap;
};

int resident_ctas(int) { return 2; }

Plan make_plan(int B, int Hkv, int grp, int n)
{
    const long long target_ctas = 148LL * resident_ctas(grp);
    long long per_head = (target_ctas + (long long)B * Hkv - 1) / ((long long)B * Hkv);
    if (per_head < 1) per_head = 1;
    if (per_head > 256) per_head = 256;
    long long chunk = (n + per_head - 1) / per_head;
    chunk = (chunk + kKB - 1) / kKB * kKB;
    long long splits = (n + chunk - 1) / chunk;  // <= per_head
    return Plan{(int)splits, (int)chunk, (int)per_head};
}

// Paged batches mix lengths, so the split count is sized for the longest
// sequence as if it alone filled the GPU (every resident CTA over its kv
// heads); the splits of shorter sequences past their end exit at once.
Plan make_paged_plan(int Hkv, int grp, int max_n)
{
    long long per_head = (148LL * resident_ctas(grp) + Hkv - 1) / Hkv;
    if (per_head > 256) per_head = 256;
    long long chunk = (max_n + per_head - 1) / per_head;
    chunk = (chunk + kKB - 1) / kKB * kKB;
    long long splits = (max_n + chunk - 1) / chunk;
    return Plan{(int)splits, (int)chunk, (int)per_head};
}

size_t ws_layout(int B, int Hq, int Hkv, int D, const Plan &p, size_t *off_ml, size_t *off_o)
{
    size_t cnt = ((size_t)B * Hkv * sizeof(int) + 255) / 256 * 256;
    size_t ml = ((size_t)B * Hq * p.splits_cap * 2 * sizeof(float) + 255) / 256 * 256;
    size_t o = (size_t)B * Hq * p.splits_cap * D * sizeof(float);
    if (off_ml) *off_ml = cnt;
    if (off_o) *off_o = cnt + ml;
    return cnt + ml + o;
}

bool shapes_ok(int B, int Hq, int Hkv, int n, int D)
{
    return B >= 1 && Hq >= 1 && Hkv >= 1 && n >= 1 && Hq % Hkv == 0 && (D == 64 || D == 128);
}

// Per-call host work that depends only on (D, theta, g) is cached per thread.
struct HostCache {
    int D = 0, g = 0;
    double theta = 0.0;
    jl::PhaseTable pt;
    DecRot rot;
};

bool host_tables(int D, double theta, int g, const jl::PhaseTable **pt, const DecRot **rot)
{
    thread_local HostCache hc;
    if (hc.D != D || hc.theta != theta || hc.g != g) {
        if (!jl::make_phase_table(&hc.pt, D, theta)) return false;
        memset(&hc.rot, 0, sizeof(hc.rot));
        const int kps = kCompute / (D / 16);
        hc.rot.uni = (kps % g == 0) ? 1 : 0;
        const long long step = kps / g - kps;  // delta moves by this per KPS keys when g | KPS
        for (int d = 0; d < D / 2; d++) {
            jl::rotation_host(hc.pt, d, step, &hc.rot.c[d], &hc.rot.s[d]);
            hc.rot.ns[d] = -hc.rot.s[d];
        }
        hc.D = D;
        hc.theta = theta;
        hc.g = g;
    }
    *pt = &hc.pt;
    *rot = &hc.rot;
    return true;
}

template <int D, int GRP, bool PAGED>
int launch(const DecodeArgs &a, int B, const CUtensorMap &tk, const CUtensorMap &tv,
           const jl::PhaseTable &pt, const DecRot &rot, cudaStream_t st)
{
    using C = DecCfg<D, GRP>;
    auto kern = decode_kernel<D, GRP, PAGED>;
    static bool attr_set[64] = {false};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return jl::cuda_status(cudaGetLastError());
    if (!attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return jl::cuda_status(e);
        attr_set[dev] = true;
    }
    dim3 grid(a.splits, a.Hkv, B);
    kern<<<grid, kThreads, C::SMEM, st>>>(tk, tv, a, pt, rot);
    return jl::cuda_status(cudaGetLastError());
}

template <bool PAGED>
int dispatch(int D, int grp, const DecodeArgs &a, int B, const CUtensorMap &tk, const CUtensorMap &tv,
             const jl::PhaseTable &pt, const DecRot &rot, cudaStream_t st)
{
    if (D == 128) {
        switch (grp) {
        case 1: return launch<128, 1, PAGED>(a, B, tk, tv, pt, rot, st);
        case 2: return launch<128, 2, PAGED>(a, B, tk, tv, pt, rot, st);
        case 4: return launch<128, 4, PAGED>(a, B, tk, tv, pt, rot, st);
        default: return launch<128, 8, PAGED>(a, B, tk, tv, pt, rot, st);
        }
    }
    switch (grp) {
    case 1: return launch<64, 1, PAGED>(a, B, tk, tv, pt, rot, st);
    case 2: return launch<64, 2, PAGED>(a, B, tk, tv, pt, rot, st);
    case 4: return launch<64, 4, PAGED>(a, B, tk, tv, pt, rot, st);
    default: return launch<64, 8, PAGED>(a, B, tk, tv, pt, rot, st);
    }
}

// Every argument check of the contiguous-cache decode that does not depend on
// the workspace: run before anything is enqueued, by both entry points that
// take that cache.
int decode_args_status(const void *q, const void *k_cache, const void *v_cache, const void *out,
                       const float *lse, int B, int Hq, int Hkv, int n, int n_cap, int D, int L_pre,
                       int w, double theta)
{
    if (!q || !k_cache || !v_cache || !out || !lse) return JL_ERR_ARG;
    if (B < 1 || Hq < 1 || Hkv < 1 || n < 1 || n_cap < n || L_pre < 1 || w < 1 || !(theta > 0.0) ||
        Hq % Hkv != 0)
        return JL_ERR_ARG;
    if (D != 64 && D != 128) return JL_ERR_UNSUPPORTED;
    const int grp = Hq / Hkv;
    if (grp != 1 && grp != 2 && grp != 4 && grp != 8) return JL_ERR_UNSUPPORTED;
    if (!jl::aligned16(q) || !jl::aligned16(out) || !jl::aligned16(lse) || !jl::aligned16(k_cache) ||
        !jl::aligned16(v_cache))
        return JL_ERR_ALIGN;
    if ((long long)B * n_cap * Hkv * D > ((long long)1 << 46)) return JL_ERR_OVERFLOW;
    return JL_OK;
}

// The argument checks and workspace layout both entry points share; fills the
// length-independent fields of `a`.
int common_setup(DecodeArgs &a, const void *q, void *out, float *lse, int B, int Hq, int Hkv, int n,
                 int D, int L_pre, int w, double theta, void *workspace, size_t ws_bytes, bool paged)
{
    if (!q || !out || !lse) return JL_ERR_ARG;
    if (B < 1 || Hq < 1 || Hkv < 1 || n < 1 || L_pre < 1 || w < 1 || !(theta > 0.0) || Hq % Hkv != 0)
        return JL_ERR_ARG;
    if (D != 64 && D != 128) return JL_ERR_UNSUPPORTED;
    const int grp = Hq / Hkv;
    if (grp != 1 && grp != 2 && grp != 4 && grp != 8) return JL_ERR_UNSUPPORTED;
    if (!jl::aligned16(q) || !jl::aligned16(out) || !jl::aligned16(lse)) return JL_ERR_ALIGN;
    Plan p = paged ? make_paged_plan(Hkv, grp, n) : make_plan(B, Hkv, grp, n);
    size_t off_ml = 0, off_o = 0;
    size_t need = ws_layout(B, Hq, Hkv, D, p, &off_ml, &off_o);
    if (!workspace || ws_bytes < need) return JL_ERR_WORKSPACE;
    if (!jl::aligned16(workspace)) return JL_ERR_ALIGN;
    memset(&a, 0, sizeof(a));
    a.q = (const __nv_bfloat16 *)q;
    a.out = (__nv_bfloat16 *)out;
    a.lse = lse;
    char *ws = (char *)workspace;
    a.counters = (int *)ws;
    a.part_ml = (float *)(ws + off_ml);
    a.part_o = (float *)(ws + off_o);
    a.status = jl::status_word_ptr();
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.n = n;
    a.w = w;
    a.L = L_pre;
    a.splits = p.splits;
    a.chunk = p.chunk;
    a.scale_log2 = (float)(1.0 / sqrt((double)D) * 1.4426950408889634);
    return JL_OK;
}

}  // namespace

extern "C" size_t jl_bifocal_decode_workspace_size(int B, int Hq, int Hkv, int n, int D)
{
    if (!shapes_ok(B, Hq, Hkv, n, D)) return 0;
    Plan p = make_plan(B, Hkv, Hq / Hkv, n);
    return ws_layout(B, Hq, Hkv, D, p, nullptr, nullptr);
}

extern "C" size_t jl_bifocal_decode_paged_workspace_size(int B, int Hq, int Hkv, int max_n, int D)
{
    if (!shapes_ok(B, Hq, Hkv, max_n, D)) return 0;
    return ws_layout(B, Hq, Hkv, D, make_paged_plan(Hkv, Hq / Hkv, max_n), nullptr, nullptr);
}

// The contiguous-cache decode with group factor g and the query's correction
// offset shifted by qshift (arguments already checked by decode_args_status).
static int decode_impl(const void *q, const void *k_cache, const void *v_cache, void *out, float *lse,
                       int B, int Hq, int Hkv, int n, int n_cap, int D, int L_pre, int w, double theta,
                       int g, int qshift, void *workspace, size_t ws_bytes, void *stream)
{
    DecodeArgs a;
    int rc = common_setup(a, q, out, lse, B, Hq, Hkv, n, D, L_pre, w, theta, workspace, ws_bytes, false);
    if (rc != JL_OK) return rc;
    a.g = g;
    a.qshift = qshift;
    const jl::PhaseTable *pt = nullptr;
    const DecRot *rot = nullptr;
    if (!host_tables(D, theta, a.g, &pt, &rot)) return JL_ERR_ARG;
    CUtensorMap tk, tv;
    // only rows [0, n) are mapped: the block that holds key n-1 reads zeros past
    // it, never the cache's unused capacity (0 * NaN would poison P.V)
    if (!jl::make_bshd_map(&tk, k_cache, B, n, n_cap, Hkv, D, D, kKB, false) ||
        !jl::make_bshd_map(&tv, v_cache, B, n, n_cap, Hkv, D, D, kKB, false))
        return JL_ERR_CUDA;
    return dispatch<false>(D, Hq / Hkv, a, B, tk, tv, *pt, *rot, (cudaStream_t)stream);
}

extern "C" int jl_bifocal_decode(const void *q, const void *k_cache, const void *v_cache, void *out,
                                 float *lse, int B, int Hq, int Hkv, int n, int n_cap, int D,
                                 int L_pre, int w, double theta, void *workspace, size_t ws_bytes,
                                 void *stream)
{
    const int rc = decode_args_status(q, k_cache, v_cache, out, lse, B, Hq, Hkv, n, n_cap, D, L_pre, w,
                                      theta);
    if (rc != JL_OK) return rc;
    return decode_impl(q, k_cache, v_cache, out, lse, B, Hq, Hkv, n, n_cap, D, L_pre, w, theta,
                       (int)jl::group_factor_host(n, L_pre), 0, workspace, ws_bytes, stream);
}

extern "C" int jl_bifocal_decode_ex(const void *q, const void *k_cache, const void *v_cache, void *out,
                                    float *lse, int B, int Hq, int Hkv, int n, int n_cap, int D, int L_pre,
                                    int w, double theta, unsigned flags, void *workspace, size_t ws_bytes,
                                    void *stream)
{
    int rc = decode_args_status(q, k_cache, v_cache, out, lse, B, Hq, Hkv, n, n_cap, D, L_pre, w, theta);
    if (rc != JL_OK) return rc;
    if (flags & ~(unsigned)(JL_VARIANT_PER_QUERY_G | JL_VARIANT_SLIDING | JL_VARIANT_QUERY_SHIFT))
        return JL_ERR_ARG;
    if ((flags & JL_VARIANT_SLIDING) && flags != JL_VARIANT_SLIDING) return JL_ERR_ARG;
    if (flags & JL_VARIANT_SLIDING) {
        // only the last min(n, w) keys are attended, all exact: the plain decode
        // over the cache rows from n - w on (g = 1; positions play no part in
        // exact scores of exact-RoPE vectors).  The view keeps the cache's batch
        // stride of n_cap rows; its last batch entry ends at row n <= n_cap.
        const int n_in = n < w ? n : w;
        const size_t skip = (size_t)(n - n_in) * Hkv * D * sizeof(__nv_bfloat16);
        return decode_impl(q, (const char *)k_cache + skip, (const char *)v_cache + skip, out, lse, B, Hq,
                           Hkv, n_in, n_cap, D, n_in, w, theta, 1, 0, workspace, ws_bytes, stream);
    }
    if (flags & JL_VARIANT_QUERY_SHIFT) {
        const long long g = jl::group_factor_shift_host(n, L_pre, w);
        if (g < 1) return JL_ERR_ARG;
        return decode_impl(q, k_cache, v_cache, out, lse, B, Hq, Hkv, n, n_cap, D, L_pre, w, theta, (int)g,
                           (int)(w - w / g), workspace, ws_bytes, stream);
    }
    // per-query g: the single query at n - 1 has the call's length n
    return decode_impl(q, k_cache, v_cache, out, lse, B, Hq, Hkv, n, n_cap, D, L_pre, w, theta,
                       (int)jl::group_factor_host(n, L_pre), 0, workspace, ws_bytes, stream);
}

extern "C" int jl_bifocal_decode_paged(const void *q, const void *k_pages, const void *v_pages,
                                       const int *block_table, const int *seq_lens, void *out,
                                       float *lse, int B, int Hq, int Hkv, int D, int page_size,
                                       int num_pages, int max_pages, int max_n, int L_pre, int w,
                                       double theta, void *workspace, size_t ws_bytes, void *stream)
{
    if (!k_pages || !v_pages || !block_table || !seq_lens) return JL_ERR_ARG;
    if (page_size < kKB || page_size % kKB != 0 || num_pages < 1 || max_pages < 1 ||
        (long long)max_pages * page_size > 0x7fffffffLL || max_n > max_pages * page_size)
        return JL_ERR_ARG;
    DecodeArgs a;
    int rc = common_setup(a, q, out, lse, B, Hq, Hkv, max_n, D, L_pre, w, theta, workspace, ws_bytes, true);
    if (rc != JL_OK) return rc;
    if (!jl::aligned16(k_pages) || !jl::aligned16(v_pages) ||
        (reinterpret_cast<uintptr_t>(block_table) & 3u) || (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
        return JL_ERR_ALIGN;
    if ((long long)num_pages * page_size * Hkv * D > ((long long)1 << 46)) return JL_ERR_OVERFLOW;
    a.seq_lens = seq_lens;
    a.block_table = block_table;
    a.page_size = page_size;
    a.max_pages = max_pages;
    a.num_pages = num_pages;
    const jl::PhaseTable *pt = nullptr;
    const DecRot *rot = nullptr;
    if (!host_tables(D, theta, 1, &pt, &rot)) return JL_ERR_ARG;  // per-sequence g on the device
    CUtensorMap tk, tv;
    // the pool as num_pages units of page_size rows: a page id outside it reads zeros
    if (!jl::make_bshd_map(&tk, k_pages, num_pages, page_size, page_size, Hkv, D, D, kKB, false) ||
        !jl::make_bshd_map(&tv, v_pages, num_pages, page_size, page_size, Hkv, D, D, kKB, false))
        return JL_ERR_CUDA;
    return dispatch<true>(D, Hq / Hkv, a, B, tk, tv, *pt, *rot, (cudaStream_t)stream);
}

// ---------------------------------------------------------------- no-allocation entry point
// Decode for callers that must not allocate device memory: the split-KV
// scratch lives in a fixed file-scope device array instead of a caller
// workspace.
namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)JL_DECODE_NOALLOC_SCRATCH_BYTES;

// The scratch itself.  Every GPU that loads this library holds it until the
// process exits.  In host code this name is only a stand-in for the device
// object, never a device address: the address comes from
// cudaGetSymbolAddress, per device.
static __device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

// Device address of g_decode_scratch on the current device, looked up on the
// first call made with that device current and cached afterwards.
void *noalloc_scratch_address(int *status)
{
    static void *addr[64] = {nullptr};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        *status = JL_ERR_CUDA;
        return nullptr;
    }
    if (!addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_decode_scratch);
        if (e != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            *status = JL_ERR_CUDA;
            return nullptr;
        }
        addr[dev] = p;
    }
    return addr[dev];
}

}  // namespace

extern "C" int jl_bifocal_decode_noalloc(const void *q, const void *k_cache, const void *v_cache,
                                         void *out, float *lse, int B, int Hq, int Hkv, int n,
                                         int n_cap, int D, int L_pre, int w, double theta,
                                         void *stream)
{
    // every check runs before the scratch is touched: a rejected call enqueues nothing
    const int rc = decode_args_status(q, k_cache, v_cache, out, lse, B, Hq, Hkv, n, n_cap, D, L_pre, w,
                                      theta);
    if (rc != JL_OK) return rc;
    const Plan p = make_plan(B, Hkv, Hq / Hkv, n);
    size_t off_ml = 0, off_o = 0;
    const size_t need = ws_layout(B, Hq, Hkv, D, p, &off_ml, &off_o);
    if (need > kNoAllocScratchBytes) return JL_ERR_WORKSPACE;  // beyond the fixed scratch
    int status = JL_OK;
    void *scratch = noalloc_scratch_address(&status);
    if (!scratch) return status;
    // the arrival counters must start at zero; the array keeps whatever the
    // previous call (of any size) left in it
    cudaError_t e = cudaMemsetAsync(scratch, 0, off_ml, (cudaStream_t)stream);
    if (e != cudaSuccess) return jl::cuda_status(e);
    return jl_bifocal_decode(q, k_cache, v_cache, out, lse, B, Hq, Hkv, n, n_cap, D, L_pre, w, theta,
                             scratch, kNoAllocScratchBytes, stream);
}
