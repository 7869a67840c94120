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
#include "corrector.cuh"

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
    int page_size, max_pages, num_pages, L, B;
    int part_stride;         // tensor-core paged decode: splits per (batch, head) in the partial layout
};

// Named barrier over the compute warps only (the producer warp never joins).
__device__ __forceinline__ void compute_sync()
{
    asm volatile("bar.sync 1, %0;" ::"n"(kCompute) : "memory");
}

// The same barrier, returning whether `v` holds in every compute thread: a
// wait that gave up in one warp makes all of them leave together.
__device__ __forceinline__ bool compute_sync_and(bool v)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, 1, %2, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "n"(kCompute)
        : "memory");
    return r != 0;
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
    static constexpr int SMEM = OFF_BAR + 2 * kNS * 8 + 32;  // + abort, last, the paged plan
    // end-of-chunk reduction buffer [KPS3][GRP][D] fp32 aliases the K/V ring
    static constexpr int VC = D / 8, KPS3 = kCompute / VC;
    static_assert(KPS3 * GRP * D * 4 <= 2 * kNS * BLOCK_BYTES, "reduction buffer");
};

// PAGED: the keys of sequence b live in pages of a shared pool, page p of it
// at block_table[b][p]; its length n_b comes from seq_lens[b] and sets its own
// g.  Otherwise the cache is [B, n_cap, Hkv, D] and every sequence has length n.
// Resident CTAs per SM the kernel is built for: two, or one for eight heads
// per kv head, whose per-thread accumulators need more than the 168
// registers two CTAs of 160 threads leave.
template <int GRP>
struct DecOcc {
    static constexpr int CTAS = GRP <= 4 ? 2 : 1;
};

// The end of a split: once its partial statistics are written, the last CTA
// of the (batch, kv head) to finish merges all ns of them into out and lse
// and resets the arrival counter.  Run by the 128 threads of the compute
// group (thread indices 0..127); mw, st_m and st_l are shared scratch of
// GRP * 256, GRP and GRP floats.
template <int D, int GRP>
__device__ void ticket_and_merge(const DecodeArgs &a, int b, int hk, int ns, int stride, float *mw,
                                 float *st_m, float *st_l, volatile int &s_last)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const size_t hq0 = (size_t)b * a.Hq + (size_t)hk * GRP;
    __threadfence();
    compute_sync();
    if (tid == 0) {
        const int ticket = atomicAdd(&a.counters[b * a.Hkv + hk], 1);
        s_last = (ticket == ns - 1);
    }
    compute_sync();
    if (!s_last) return;
    __threadfence();

    // ---- last CTA of this (b, kv head): merge the partial statistics
    // weights w_s = 2^(m_s - M) with M = max m_s; L = sum l_s w_s
    for (int h = warp; h < GRP; h += kCompute / 32) {
        const float *ml = a.part_ml + (hq0 + h) * stride * 2;
        float m = -INFINITY;
        for (int q = lane; q < ns; q += 32) m = fmaxf(m, __ldcg(ml + 2 * q));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        const float off = (m == -INFINITY) ? 0.f : m;
        float L = 0.f;
        for (int q = lane; q < ns; q += 32) {
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
        const float *po = a.part_o + (hq0 + h) * stride * D + d;
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
        int q = 0;
        for (; q + 8 <= ns; q += 8) {
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
        for (; q < ns; q++) {
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

template <int D, int GRP, bool PAGED>
__global__ void __launch_bounds__(kThreads, DecOcc<GRP>::CTAS)
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
    const int hk = blockIdx.y;
    // this CTA's sequence b, its split, the sequence's split count ns, and the
    // split capacity of the partial-statistics layout
    int b = blockIdx.z, split = blockIdx.x, ns = a.splits, chunk = a.chunk;
    const int stride = a.splits;
    int n = a.n, g = a.g;
    if constexpr (PAGED) {
        // Splits in proportion to the sequences' lengths: one chunk size for
        // the whole batch from its total key count, so every CTA of the grid
        // (a.splits per kv head, plus at most one more per sequence) has about
        // the same number of keys.  Lengths outside [1, min(max_n, what the
        // page table covers)] are clamped (never read past the table) and
        // reported.
        volatile int *s_plan = reinterpret_cast<volatile int *>(smem + C::OFF_BAR + 2 * kNS * 8 + 8);
        if (tid == 0) {
            const int n_lim = min(a.max_pages * a.page_size, a.n);
            long long tot = 0;
            bool bad = false;
            for (int s = 0; s < a.B; s++) {
                const int ls = a.seq_lens[s];
                bad = bad || ls < 1 || ls > n_lim;
                tot += min(max(ls, 1), n_lim);
            }
            if (bad && blockIdx.x == 0 && hk == 0) jl::record_status(a.status, JL_ERR_GUARD);
            long long ch = (tot + a.splits - 1) / a.splits;
            ch = (ch + kKB - 1) / kKB * kKB;
            int bb = -1, sp = 0, nsb = 0, nb = 0, cum = 0;
            for (int s = 0; s < a.B; s++) {
                const int ls = min(max(a.seq_lens[s], 1), n_lim);
                const int sb = (int)((ls + ch - 1) / ch);
                if ((int)blockIdx.x < cum + sb) {
                    bb = s;
                    sp = (int)blockIdx.x - cum;
                    nsb = sb;
                    nb = ls;
                    break;
                }
                cum += sb;
            }
            s_plan[0] = bb;
            s_plan[1] = sp;
            s_plan[2] = nsb;
            s_plan[3] = nb;
            s_plan[4] = (int)ch;
        }
        __syncthreads();
        b = s_plan[0];
        if (b < 0) return;  // past the last sequence's splits: no work
        split = s_plan[1];
        ns = s_plan[2];
        n = s_plan[3];
        chunk = s_plan[4];
        g = (n <= a.L) ? 1 : (n - 1) / a.L + 1;
    }
    const int j_begin = split * chunk;
    const int j_end = min(n, j_begin + chunk);
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
    if (ns == 1) {
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
        a.part_o[((hq0 + h) * stride + split) * D + d] = o;
    }
    if (tid < GRP) {
        a.part_ml[((hq0 + tid) * stride + split) * 2 + 0] = st_m[tid];
        a.part_ml[((hq0 + tid) * stride + split) * 2 + 1] = st_l[tid];
    }
    ticket_and_merge<D, GRP>(a, b, hk, ns, stride, mw, st_m, st_l, s_last);
}

// ---------------------------------------------------------------- tensor-core decode
// The same split-KV decode with the dot products and P.V on the tensor core
// (head dimension 128, contiguous cache).  A CTA streams its chunk of one kv
// head's keys in 128-key tiles and computes S^T = K Q^T (M = 128 keys, N = 16
// columns holding the GRP query heads) and O^T += V^T P^T (M = 128 dims, the
// V tile read as an MN-major A operand), accumulators in TMEM.  Remote tiles
// are rotated in place by the correction warps (fp16 operands, the corrected
// query on the other side); the tile the window edge crosses is scored twice,
// exactly before the correction rotates it and aliased after.  What is left
// on the CUDA cores per key is the correction and a handful of softmax
// instructions, so the kernel streams K and V at HBM speed where the scalar
// kernel above is bound by its instruction issue.
//
// Warp roles (352 threads):
//   warps 0-3  softmax: thread t owns key t of a tile (TMEM lane t of S^T) and
//              dim t of O^T; then the epilogue and the merge of the splits
//   warps 4-7  correction of remote K tiles (rows 16 apart per thread)
//   warp 8     TMA producer of the K ring
//   warp 9     TMA producer of the V ring
//   warp 10    TMEM allocator and single-thread MMA issuer
// TMEM (128 columns): S^T of tile v at 32 (v % 2) (the tile's own view) and
// 32 (v % 2) + 16 (the exact view of the edge tile), O^T at 64.
constexpr int kTcKeys = 128;
constexpr int kTcNS = 3;
constexpr int kTcThreads = 352;
constexpr int kTcN = 16;
constexpr float kTcRescaleThreshold = 8.0f;  // log2 units, as the prefill's lazy offset
// Shorter contiguous caches take the scalar kernel; the paged batch takes this
// kernel for every length, its shorter sequences with P split into two bf16
// parts for P.V.
constexpr int kTcMinKeys = 256;

struct TcCfg {
    static constexpr int D = 128;
    static constexpr int TILE = kTcKeys * D * 2;     // one K or V tile: 32 KB
    static constexpr int REGION = kTcKeys * 64 * 2;  // one 64-column box of it: 16 KB
    static constexpr int HALF = REGION / 2;          // 64 rows of a box (one paged load): 8 KB
    static constexpr int QBOX = kTcN * 128;          // 16 rows x 64 16-bit values: 2 KB
    static constexpr int OPND = 2 * QBOX;            // a 16 x 128 operand (Q^T or P^T): 4 KB
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = OFF_K + kTcNS * TILE;
    static constexpr int OFF_QE = OFF_V + kTcNS * TILE;  // exact q, bf16
    static constexpr int OFF_QR = OFF_QE + OPND;         // corrected q, fp16
    static constexpr int OFF_P = OFF_QR + OPND;          // P^T high and low parts, two tiles
    static constexpr int OFF_RED = OFF_P + 4 * OPND;     // fp32 [2][4 warps][8 heads] maxima, [4][16] sums
    static constexpr int OFF_RC = OFF_RED + (2 * 4 * 8 + 4 * 16) * 4;  // paged: this sequence's RotConsts
    static constexpr int OFF_BAR = (OFF_RC + (int)sizeof(RotConsts) + 15) / 16 * 16;
    static constexpr int B_KFULL = 0, B_KEMPTY = B_KFULL + kTcNS, B_KREADY = B_KEMPTY + kTcNS,
                         B_VFULL = B_KREADY + kTcNS, B_VEMPTY = B_VFULL + kTcNS, B_SFULL = B_VEMPTY + kTcNS,
                         B_PFULL = B_SFULL + 2, B_ODONE = B_PFULL + 2, B_QREADY = B_ODONE + 2,
                         B_BANDQK = B_QREADY + 1, B_DRAIN = B_BANDQK + 1, B_VREADY = B_DRAIN + 1,
                         NBAR = B_VREADY + 1;
    static constexpr int OFF_TMEM_SLOT = NBAR * 8, OFF_ABORT = OFF_TMEM_SLOT + 4, OFF_LAST = OFF_ABORT + 4,
                         OFF_PLAN = OFF_LAST + 4;  // paged: 5 ints
    static constexpr int SMEM = OFF_BAR + OFF_PLAN + 5 * 4 + 1024;  // + alignment slack
    static_assert(SMEM <= 232448, "shared memory budget");
    // the merge's scratch (GRP x 256 weights, then m and l) reuses the K ring
    static_assert(8 * 256 * 4 + 2 * 8 * 4 <= kTcNS * TILE, "merge scratch");
};

__device__ __forceinline__ uint32_t tc_opnd_off(int row, int col)
{
    // byte offset of 16-bit element (row, col) of a 16 x 128 K-major operand
    // stored as two 128-byte-swizzled boxes of 64 columns
    return (uint32_t)((col >> 6) * TcCfg::QBOX + row * 128 + ((((col & 63) >> 3) ^ (row & 7)) << 4) +
                      (col & 7) * 2);
}

template <int GRP, bool PAGED>
__global__ void __launch_bounds__(kTcThreads, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                     const DecodeArgs a, const __grid_constant__ jl::PhaseTable pt,
                     const __grid_constant__ RotConsts rc)
{
    using C = TcCfg;
    constexpr int D = C::D, NS = kTcNS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~(uintptr_t)1023);
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sK = sbase + C::OFF_K, sV = sbase + C::OFF_V, sQE = sbase + C::OFF_QE,
                   sQR = sbase + C::OFF_QR, sP = sbase + C::OFF_P;
    auto bar = [&](int idx) -> uint32_t { return sbase + C::OFF_BAR + 8u * (uint32_t)idx; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_BAR + C::OFF_TMEM_SLOT);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_BAR + C::OFF_ABORT);
    volatile int &s_last = *reinterpret_cast<volatile int *>(smem + C::OFF_BAR + C::OFF_LAST);
    float *red = reinterpret_cast<float *>(smem + C::OFF_RED);
    const WaitCtx wc{a.status, abort_flag};

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int hk = blockIdx.y;
    // this CTA's sequence b, its split, the sequence's split count ns and
    // length n, the chunk size, and the split stride of the partial layout
    int b = blockIdx.z, split = blockIdx.x, ns = a.splits, n = a.n, chunk = a.chunk, g = a.g;
    const int stride = PAGED ? a.part_stride : a.splits;
    // Programmatic dependent launch: let the next kernel of the stream start
    // its launch now (every CTA of this grid is resident once all have
    // passed here), and read nothing another kernel may still write before
    // the previous one completed.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if constexpr (PAGED) asm volatile("griddepcontrol.wait;" ::: "memory");
    if constexpr (PAGED) {
        // Splits in proportion to the lengths: the smallest chunk (a multiple
        // of the 128-key tile) for which the batch needs at most gridDim.x
        // CTAs per kv head, so one wave serves every sequence.
        volatile int *s_plan = reinterpret_cast<volatile int *>(smem + C::OFF_BAR + C::OFF_PLAN);
        if (tid == 0) {
            const int n_lim = min(a.max_pages * a.page_size, a.n);
            bool bad = false;
            for (int q = 0; q < a.B; q++) {
                const int ls = a.seq_lens[q];
                bad = bad || ls < 1 || ls > n_lim;
            }
            if (bad && blockIdx.x == 0 && hk == 0) jl::record_status(a.status, JL_ERR_GUARD);
            auto need = [&](long long ch) {
                long long cnt = 0;
                for (int q = 0; q < a.B; q++) cnt += (min(max(a.seq_lens[q], 1), n_lim) + ch - 1) / ch;
                return cnt;
            };
            // need(ch) is non-increasing in ch; at one tile-rounded chunk of the
            // longest length it is B <= gridDim.x
            long long lo = 1, hi = ((long long)n_lim + kTcKeys - 1) / kTcKeys;
            while (lo < hi) {
                const long long mid = (lo + hi) >> 1;
                if (need(mid * kTcKeys) <= (long long)gridDim.x) hi = mid;
                else lo = mid + 1;
            }
            const long long ch = lo * kTcKeys;
            int bb = -1, sp = 0, nsb = 0, nb = 0, cum = 0;
            for (int q = 0; q < a.B; q++) {
                const int ls = min(max(a.seq_lens[q], 1), n_lim);
                const int sb = (int)((ls + ch - 1) / ch);
                if ((int)blockIdx.x < cum + sb) {
                    bb = q;
                    sp = (int)blockIdx.x - cum;
                    nsb = sb;
                    nb = ls;
                    break;
                }
                cum += sb;
            }
            s_plan[0] = bb;
            s_plan[1] = sp;
            s_plan[2] = nsb;
            s_plan[3] = nb;
            s_plan[4] = (int)ch;
        }
        __syncthreads();
        b = s_plan[0];
        if (b < 0) return;  // past the last sequence's splits: no work (nothing allocated yet)
        split = s_plan[1];
        ns = s_plan[2];
        n = s_plan[3];
        chunk = s_plan[4];
        g = (n <= a.L) ? 1 : (n - 1) / a.L + 1;
    }
    const int j_begin = split * chunk;
    const int j_end = min(n, j_begin + chunk);
    const int T = (j_end - j_begin + kTcKeys - 1) / kTcKeys;
    // Over fewer than kTcMinKeys keys the rounding of P to bf16 is not averaged
    // out: P.V then takes P as a high and a low bf16 part (P to ~2^-17).
    const bool split_p = n < kTcMinKeys;
    const int j_split = (g > 1) ? max(0, n - a.w) : 0;  // keys below are remote
    const bool any_remote = j_begin < j_split;
    // tile classes: 0 exact, 1 remote, 2 crossed by the window edge
    auto tclass = [&](int v) -> int {
        const int j0 = j_begin + v * kTcKeys;
        return j0 >= j_split ? 0 : (j0 + kTcKeys <= j_split ? 1 : 2);
    };

    if (tid == 0) {
        for (int s = 0; s < NS; s++) {
            mbar_init(bar(C::B_KFULL + s), 1);
            mbar_init(bar(C::B_KEMPTY + s), 1);
            mbar_init(bar(C::B_KREADY + s), 4);  // one per correction warp
            mbar_init(bar(C::B_VFULL + s), 1);
            mbar_init(bar(C::B_VEMPTY + s), 1);
        }
        for (int s = 0; s < 2; s++) {
            mbar_init(bar(C::B_SFULL + s), 1);
            mbar_init(bar(C::B_PFULL + s), 4);  // one per softmax warp
        }
        mbar_init(bar(C::B_ODONE), 1);
        mbar_init(bar(C::B_ODONE + 1), 1);
        mbar_init(bar(C::B_QREADY), 4);
        mbar_init(bar(C::B_BANDQK), 1);
        mbar_init(bar(C::B_DRAIN), 1);
        mbar_init(bar(C::B_VREADY), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 10) {
        tmem_alloc(smem_u32(tmem_slot), 128);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    if constexpr (!PAGED) asm volatile("griddepcontrol.wait;" ::: "memory");
    const size_t hq0 = (size_t)b * a.Hq + (size_t)hk * GRP;
    bool ok = true;
    float m_run[GRP], l_run[GRP], lr_run[GRP];  // softmax state (warps 0-3)

    if (warp == 8 || warp == 9) {
        // ------------------------------------------------------------ producers: K (warp 8), V (warp 9)
        if (lane == 0) {
            const bool is_k = warp == 8;
            const CUtensorMap *m = is_k ? &tk : &tv;
            const uint32_t ring = is_k ? sK : sV;
            const int b_full = is_k ? C::B_KFULL : C::B_VFULL, b_empty = is_k ? C::B_KEMPTY : C::B_VEMPTY;
            prefetch_tmap(m);
            int issued = 0;
            for (int v = 0; v < T; v++) {
                const int s = v % NS;
                if (!(ok = wait_bar(bar(b_empty + s), ((v / NS) & 1) ^ 1, wc))) break;
                const int row0 = j_begin + v * kTcKeys;
                if constexpr (PAGED) {
                    // two 64-row halves, each from its own page (page sizes are
                    // multiples of 64); a half wholly past the sequence loads nothing.
                    // A page id outside the pool reads zeros (TMA bounds) and is reported.
                    const int halves = (j_end - row0 > 64) ? 2 : 1;
                    mbar_arrive_expect_tx(bar(b_full + s), halves * 2 * C::HALF);
                    for (int hh = 0; hh < halves; hh++) {
                        const int row = row0 + 64 * hh;
                        const int page = a.block_table[(size_t)b * a.max_pages + row / a.page_size];
                        if ((unsigned)page >= (unsigned)a.num_pages) jl::record_status(a.status, JL_ERR_GUARD);
#pragma unroll
                        for (int r = 0; r < 2; r++)
                            tma_load_4d(ring + s * C::TILE + r * C::REGION + hh * C::HALF, m, bar(b_full + s),
                                        r * 64, hk, row % a.page_size, page);
                    }
                } else {
                    mbar_arrive_expect_tx(bar(b_full + s), C::TILE);
#pragma unroll
                    for (int r = 0; r < 2; r++)
                        tma_load_4d(ring + s * C::TILE + r * C::REGION, m, bar(b_full + s), r * 64, hk, row0, b);
                }
                issued = v + 1;
            }
            if (!ok)
                for (int v = issued - NS < 0 ? 0 : issued - NS; v < issued; v++)
                    drain_bar(bar(b_full + v % NS), (v / NS) & 1);
        }
        if constexpr (PAGED) {
            if (warp == 9) {
                // The last tile's V rows past the sequence hold whatever the pool
                // (or an earlier tile) left there: zero them before its P.V, where
                // 0 * NaN would still poison O.  The issuer waits on VREADY for it.
                __syncwarp();
                ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                const int v = T - 1, s = v % NS;
                if (ok) ok = wait_bar_warp(bar(C::B_VFULL + s), (v / NS) & 1, wc);
                if (ok) {
                    const int valid = j_end - (j_begin + v * kTcKeys);  // 1..128 rows hold keys
                    const int nz = (kTcKeys - valid) * 8;              // 16-byte chunks per box
                    for (int e = lane; e < 2 * nz; e += 32) {
                        const int r = e / nz, rem = e % nz;
                        *reinterpret_cast<uint4 *>(smem + C::OFF_V + s * C::TILE + r * C::REGION +
                                                   (valid + rem / 8) * 128 + (rem % 8) * 16) =
                            make_uint4(0u, 0u, 0u, 0u);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(C::B_VREADY));
                }
            }
        }
    } else if (warp == 10) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idE = idesc_bf16_f32(128, kTcN, false, false);
            constexpr uint32_t idR = idesc_f16_f32(128, kTcN, false, false);
            constexpr uint32_t idPV = idesc_bf16_f32(128, kTcN, true, false);  // A = V^T, MN-major
            auto qk = [&](int v, int group, uint32_t qaddr, uint32_t id) {
                const uint64_t dk = sdesc_sw128(sK + (v % NS) * C::TILE, 16, 1024);
                const uint64_t dq = sdesc_sw128(qaddr, 16, 1024);
#pragma unroll
                for (int k = 0; k < D / 16; k++)
                    mma_f16_ss(tmem + 32u * (v & 1) + 16u * group,
                               dk + (uint64_t)(((k >> 2) * C::REGION + (k & 3) * 32) >> 4),
                               dq + (uint64_t)(((k >> 2) * C::QBOX + (k & 3) * 32) >> 4), id, k > 0 ? 1u : 0u);
            };
            // S^T(v): the edge tile's exact scores first, on the raw tile
            auto qk_tile = [&](int v) -> bool {
                const int s = v % NS, cls = tclass(v);
                if (cls == 2) {
                    if (!wait_bar(bar(C::B_KFULL + s), (v / NS) & 1, wc)) return false;
                    tc_fence_after();
                    qk(v, 1, sQE, idE);
                    mma_commit(bar(C::B_BANDQK));
                }
                if (!wait_bar(bar(C::B_KREADY + s), (v / NS) & 1, wc)) return false;
                tc_fence_after();
                if (cls == 0) qk(v, 0, sQE, idE);
                else qk(v, 0, sQR, idR);
                mma_commit(bar(C::B_SFULL + (v & 1)));
                mma_commit(bar(C::B_KEMPTY + s));
                return true;
            };
            ok = wait_bar(bar(C::B_QREADY), 0, wc);
            tc_fence_after();
            if (ok) ok = qk_tile(0);
            for (int v = 0; ok && v < T; v++) {
                // QK of the next tile goes first: its softmax overlaps this P.V
                if (v + 1 < T && !(ok = qk_tile(v + 1))) break;
                const int s = v % NS;
                if (!(ok = wait_bar(bar(C::B_PFULL + (v & 1)), (v >> 1) & 1, wc))) break;
                // the paged batch's last tile: V with its rows past the sequence zeroed
                const bool vready = PAGED && v == T - 1;
                if (!(ok = wait_bar(bar(vready ? C::B_VREADY : C::B_VFULL + s), vready ? 0u : (v / NS) & 1, wc)))
                    break;
                tc_fence_after();
                const uint64_t dv = sdesc_sw128(sV + s * C::TILE, C::REGION, 1024);
                // P.V on the rounded P, or P = P_hi + P_lo (bf16 each) over few keys:
                // O^T += V^T P_hi^T (+ V^T P_lo^T)
                for (int part = 0; part < (split_p ? 2 : 1); part++) {
                    const uint64_t dp = sdesc_sw128(sP + (2 * (v & 1) + part) * C::OPND, 16, 1024);
#pragma unroll
                    for (int k = 0; k < kTcKeys / 16; k++)
                        mma_f16_ss(tmem + 64u, dv + (uint64_t)((k * 2048) >> 4),
                                   dp + (uint64_t)(((k >> 2) * C::QBOX + (k & 3) * 32) >> 4), idPV,
                                   (v > 0 || part > 0 || k > 0) ? 1u : 0u);
                }
                mma_commit(bar(C::B_VEMPTY + s));
                mma_commit(bar(C::B_ODONE + (v & 1)));
            }
            if (!ok) {
                // no MMA may still run when TMEM is released
                mma_commit(bar(C::B_DRAIN));
                drain_bar(bar(C::B_DRAIN), 0);
            }
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ------------------------------------------------------------ correction
        // Makes K(v) ready for its QK: rotates a tile with remote keys in place
        // (the edge tile after its exact QK has read it) and arrives on KREADY.
        const int t = tid - 128;
        Corrector<D> cor;
        if constexpr (PAGED) {
            // this sequence's g sets the step rotations: build them in shared
            // memory from the exact phase (pairs d = t, 64 threads), as the host
            // does for the contiguous cache
            RotConsts *src = reinterpret_cast<RotConsts *>(smem + C::OFF_RC);
            if (any_remote && t < D / 2) {
                const int rps = 128 / (D / 16);
                const int qs = rps / g;
                const int offs[4] = {qs - rps, qs + 1 - rps, 2 * (qs - rps), (64 / rps) * (qs - rps)};
                float cs[4], sn[4];
#pragma unroll
                for (int u = 0; u < 4; u++) jl::phase_sincos(offs[u], pt.f[t], &sn[u], &cs[u]);
                src->ac[t] = cs[0];
                src->as[t] = sn[0];
                src->ans[t] = -sn[0];
                src->bc[t] = cs[1];
                src->bs[t] = sn[1];
                src->bns[t] = -sn[1];
                src->a2c[t] = cs[2];
                src->a2s[t] = sn[2];
                src->a2ns[t] = -sn[2];
                src->skc[t] = cs[3];
                src->sks[t] = sn[3];
                if (t == 0) src->uni = (rps % g == 0) ? 1 : 0;
            }
            asm volatile("bar.sync 2, 128;" ::: "memory");  // the correction warps only
            if (any_remote) cor.init(t, g, pt, *src);
        } else {
            if (any_remote) cor.init(t, g, pt, rc);
        }
        for (int v = 0; ok && v < T; v++) {
            const int s = v % NS, cls = tclass(v);
            if (!(ok = wait_bar_warp(bar(C::B_KFULL + s), (v / NS) & 1, wc))) break;
            if (cls == 2 && !(ok = wait_bar_warp(bar(C::B_BANDQK), 0, wc))) break;
            if (cls != 0) {
                cor.run_k(sK + s * C::TILE, (j_begin + v * kTcKeys) / kTcKeys);
                fence_proxy_async_smem();
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::B_KREADY + s));
        }
    } else {
        // ------------------------------------------------------------ softmax
        const int t = tid;
        const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
        const __nv_bfloat16 *qb = a.q + hq0 * D;
        // Q^T operands: rows h < GRP hold the heads, the rest zero
        for (int e = t; e < kTcN * 16; e += 128) {
            const int h = e >> 4, cc = e & 15;
            uint4 x = make_uint4(0u, 0u, 0u, 0u);
            if (h < GRP) x = *reinterpret_cast<const uint4 *>(qb + h * D + cc * 8);
            *reinterpret_cast<uint4 *>(smem + C::OFF_QE + tc_opnd_off(h, cc * 8)) = x;
        }
        if (any_remote) {
            // corrected query at offset delta_{n-1} + qshift, fp16
            const int di = jl::delta_pos(n - 1, g) + a.qshift;
            for (int e = t; e < kTcN * 8; e += 128) {
                const int h = e >> 3, cc = e & 7;
                uint32_t lo[4] = {0u, 0u, 0u, 0u}, hi[4] = {0u, 0u, 0u, 0u};
                if (h < GRP) {
                    const uint4 x4 = *reinterpret_cast<const uint4 *>(qb + h * D + cc * 8);
                    const uint4 y4 = *reinterpret_cast<const uint4 *>(qb + h * D + 64 + cc * 8);
                    const uint32_t xw[4] = {x4.x, x4.y, x4.z, x4.w}, yw[4] = {y4.x, y4.y, y4.z, y4.w};
#pragma unroll
                    for (int e2 = 0; e2 < 4; e2++) {
                        float xs[2], ys[2], xo[2], yo[2];
                        jl::f2_split(jl::bf16x2_to_f2(xw[e2]), xs[0], xs[1]);
                        jl::f2_split(jl::bf16x2_to_f2(yw[e2]), ys[0], ys[1]);
#pragma unroll
                        for (int u = 0; u < 2; u++) {
                            float sn, cs;
                            jl::phase_sincos(di, pt.f[cc * 8 + 2 * e2 + u], &sn, &cs);
                            xo[u] = xs[u] * cs - ys[u] * sn;
                            yo[u] = ys[u] * cs + xs[u] * sn;
                        }
                        lo[e2] = jl::f2_to_f16x2(jl::f2(xo[0], xo[1]));
                        hi[e2] = jl::f2_to_f16x2(jl::f2(yo[0], yo[1]));
                    }
                }
                *reinterpret_cast<uint4 *>(smem + C::OFF_QR + tc_opnd_off(h, cc * 8)) =
                    make_uint4(lo[0], lo[1], lo[2], lo[3]);
                *reinterpret_cast<uint4 *>(smem + C::OFF_QR + tc_opnd_off(h, 64 + cc * 8)) =
                    make_uint4(hi[0], hi[1], hi[2], hi[3]);
            }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(C::B_QREADY));

#pragma unroll
        for (int h = 0; h < GRP; h++) {
            m_run[h] = -INFINITY;
            l_run[h] = 0.f;
            lr_run[h] = 0.f;
        }
        const float sc = a.scale_log2;
        for (int v = 0; v < T; v++) {
            const int j = j_begin + v * kTcKeys + t;
            const int cls = tclass(v);
            const bool got = wait_bar_warp(bar(C::B_SFULL + (v & 1)), (v >> 1) & 1, wc);
            float x[GRP], mx[GRP];
            float *rm = red + (v & 1) * 32;
            if (got) {
                tc_fence_after();
                uint32_t sa[16], sb[16];
                tmem_ld16(tmem + lane_base + 32u * (v & 1), sa);
                if (cls == 2) tmem_ld16(tmem + lane_base + 32u * (v & 1) + 16u, sb);
                tmem_ld_wait();
                const bool valid = j < j_end;
                const bool exact_b = cls == 2 && j >= j_split;
#pragma unroll
                for (int h = 0; h < GRP; h++) {
                    const float raw = __uint_as_float(exact_b ? sb[h] : sa[h]);
                    x[h] = valid ? raw * sc : -INFINITY;
                    mx[h] = x[h];
                }
                // the tile's maximum per head over the 128 keys
#pragma unroll
                for (int o = 16; o > 0; o >>= 1)
#pragma unroll
                    for (int h = 0; h < GRP; h++) mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], o));
                if (lane == 0)
#pragma unroll
                    for (int h = 0; h < GRP; h++) rm[warp * 8 + h] = mx[h];
            }
            if (!(ok = compute_sync_and(got))) break;
            // Lazy offset (as in the prefill): moved only when the maximum grows
            // by more than the threshold, by an integer, so rescaling is by an
            // exact power of two.  Every thread takes the same decision.
            float f[GRP];
            bool moved = false;
#pragma unroll
            for (int h = 0; h < GRP; h++) {
                const float tm = fmaxf(fmaxf(rm[h], rm[8 + h]), fmaxf(rm[16 + h], rm[24 + h]));
                f[h] = 1.f;
                if (tm > m_run[h] + kTcRescaleThreshold) {
                    if (m_run[h] == -INFINITY) {
                        m_run[h] = tm;  // no key of this head so far carried weight
                    } else {
                        const float k = ceilf(tm - m_run[h]);
                        m_run[h] += k;
                        f[h] = k >= 150.f ? 0.f : ldexpf(1.f, -(int)k);
                        l_run[h] *= f[h];
                        lr_run[h] *= f[h];
                        moved = true;
                    }
                }
            }
            if (moved && v > 0) {
                // O^T holds P.V of tiles < v once the P.V of tile v-1 completed
                const bool done = wait_bar_warp(bar(C::B_ODONE + ((v - 1) & 1)), ((v - 1) >> 1) & 1, wc);
                if (!(ok = compute_sync_and(done))) break;
                tc_fence_after();
                uint32_t o[16];
                tmem_ld16(tmem + lane_base + 64u, o);
                tmem_ld_wait();
#pragma unroll
                for (int h = 0; h < GRP; h++) o[h] = __float_as_uint(__uint_as_float(o[h]) * f[h]);
                tmem_st16(tmem + lane_base + 64u, o);
                tmem_st_wait();
            }
            // P^T(v), rounded to bf16 (and over few keys its low part too).
            // lr sums the P that P.V multiplies and normalises out; l, the fp32
            // sum, gives lse.  The buffers were last read by the P.V of tile
            // v-2, which completed before QK(v) (one issuing thread, in-order pipe).
            uint8_t *pbuf = smem + C::OFF_P + 2 * (v & 1) * C::OPND;
#pragma unroll
            for (int h = 0; h < GRP; h++) {
                const float off = (m_run[h] == -INFINITY) ? 0.f : m_run[h];
                const float pv = exp2f(x[h] - off);
                const __nv_bfloat16 ph = __float2bfloat16_rn(pv);
                const float phf = __bfloat162float(ph);
                l_run[h] += pv;
                *reinterpret_cast<__nv_bfloat16 *>(pbuf + tc_opnd_off(h, t)) = ph;
                if (split_p) {
                    const __nv_bfloat16 pl = __float2bfloat16_rn(pv - phf);
                    lr_run[h] += phf + __bfloat162float(pl);
                    *reinterpret_cast<__nv_bfloat16 *>(pbuf + C::OPND + tc_opnd_off(h, t)) = pl;
                } else {
                    lr_run[h] += phf;
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::B_PFULL + (v & 1)));
        }
        // ------------------------------------------------------------ epilogue (TMEM part)
        // P.V(v) completes a phase of ODONE[v % 2].  With QK(v+1) issued before
        // P.V(v), the P.V of the last two tiles may both be in flight here, and
        // on one barrier no parity wait would be right (the last phase's parity
        // also names the one before the previous); on ODONE[(T-1) % 2] the
        // phase of P.V(T-1) is at most one behind (SFULL(T-1) implied P.V(T-3)
        // complete), and its completion implies P.V(T-2)'s (one issuing
        // thread, in-order pipe).  The rescale's wait above is unambiguous the
        // same way.
        if (ok) ok = compute_sync_and(wait_bar_warp(bar(C::B_ODONE + ((T - 1) & 1)), ((T - 1) >> 1) & 1, wc));
        float o_h[GRP];
        if (ok) {
            tc_fence_after();
            uint32_t o[16];
            tmem_ld16(tmem + lane_base + 64u, o);
            tmem_ld_wait();
#pragma unroll
            for (int h = 0; h < GRP; h++) o_h[h] = __uint_as_float(o[h]);
            // row sums over the 128 keys of every tile: per-thread parts -> totals
#pragma unroll
            for (int o2 = 16; o2 > 0; o2 >>= 1)
#pragma unroll
                for (int h = 0; h < GRP; h++) {
                    l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], o2);
                    lr_run[h] += __shfl_xor_sync(0xffffffffu, lr_run[h], o2);
                }
            float *rs = red + 64;
            if (lane == 0)
#pragma unroll
                for (int h = 0; h < GRP; h++) {
                    rs[warp * 16 + h] = l_run[h];
                    rs[warp * 16 + 8 + h] = lr_run[h];
                }
            compute_sync();
#pragma unroll
            for (int h = 0; h < GRP; h++) {
                l_run[h] = (rs[h] + rs[16 + h]) + (rs[32 + h] + rs[48 + h]);
                lr_run[h] = (rs[8 + h] + rs[24 + h]) + (rs[40 + h] + rs[56 + h]);
            }
            if (t == 0)
#pragma unroll
                for (int h = 0; h < GRP; h++)
                    // an infinite or NaN score (an input or corrected operand out of range)
                    if (!(l_run[h] < INFINITY)) jl::record_status(a.status, JL_ERR_GUARD);
            if (ns == 1) {
#pragma unroll
                for (int h = 0; h < GRP; h++) {
                    a.out[(hq0 + h) * D + t] = __float2bfloat16_rn(o_h[h] / lr_run[h]);
                    if (t == h) a.lse[hq0 + h] = (m_run[h] + log2f(l_run[h])) * kLn2;
                }
            } else {
#pragma unroll
                for (int h = 0; h < GRP; h++) {
                    // the merge weighs splits by l: o scaled to the fp32 sum
                    a.part_o[((hq0 + h) * stride + split) * D + t] = o_h[h] * (l_run[h] / lr_run[h]);
                    if (t == h) {
                        a.part_ml[((hq0 + h) * stride + split) * 2 + 0] = m_run[h];
                        a.part_ml[((hq0 + h) * stride + split) * 2 + 1] = l_run[h];
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 10) tmem_dealloc(tmem, 128);
    // the K ring is free now: the merge's scratch
    if (warp < 4 && ok && ns > 1) {
        float *mw = reinterpret_cast<float *>(smem + C::OFF_K);
        ticket_and_merge<D, GRP>(a, b, hk, ns, stride, mw, mw + GRP * 256, mw + GRP * 256 + 8, s_last);
    }
}

// Split plan: as many CTAs as the kernel keeps resident (two per SM up to four
// heads per kv head, one above), at most 256 splits per (batch, kv head),
// chunks a multiple of the 64-key block.  splits_cap bounds splits for every
// n, and the workspace is sized by it, so one workspace serves every cache
// length for the same (B, Hq, Hkv, D).
struct Plan {
    int splits, chunk, splits_cap;
};

int resident_ctas(int grp) { return grp <= 4 ? DecOcc<4>::CTAS : DecOcc<8>::CTAS; }

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

// Paged batches mix lengths: the grid gives every kv head splits_cap CTAs
// (every resident CTA over the kv heads), which the kernel shares out among
// the sequences in proportion to their lengths (it reads them on the device).
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
    DecRot rot;     // the scalar kernel's chain step
    RotConsts rc;   // the tensor-core kernel's tile correction
};

bool host_tables(int D, double theta, int g, const jl::PhaseTable **pt, const DecRot **rot,
                 const RotConsts **rc = nullptr)
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
        make_rot_consts(hc.pt, D, g, &hc.rc);
        hc.D = D;
        hc.theta = theta;
        hc.g = g;
    }
    *pt = &hc.pt;
    *rot = &hc.rot;
    if (rc) *rc = &hc.rc;
    return true;
}

// Split plan of the tensor-core kernel: one CTA per SM (its rings take most
// of the shared memory), a single wave of at most 148 CTAs, chunks a multiple
// of the 128-key tile; never more splits than the scalar plan's capacity, so
// the same workspace serves both.
Plan make_tc_plan(int B, int Hkv, int n, int splits_cap)
{
    long long per_head = 148LL / ((long long)B * Hkv);
    if (per_head < 1) per_head = 1;
    if (per_head > splits_cap) per_head = splits_cap;
    long long chunk = (n + per_head - 1) / per_head;
    chunk = (chunk + kTcKeys - 1) / kTcKeys * kTcKeys;
    const long long splits = (n + chunk - 1) / chunk;
    return Plan{(int)splits, (int)chunk, splits_cap};
}

template <int GRP, bool PAGED>
int launch_tc(const DecodeArgs &a, int B, const CUtensorMap &tk, const CUtensorMap &tv,
              const jl::PhaseTable &pt, const RotConsts &rc, cudaStream_t st)
{
    auto kern = decode_tc_kernel<GRP, PAGED>;
    static bool attr_set[64] = {false};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return jl::cuda_status(cudaGetLastError());
    if (!attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, TcCfg::SMEM);
        if (e != cudaSuccess) return jl::cuda_status(e);
        attr_set[dev] = true;
    }
    // paged: a.splits CTAs per kv head, shared out by the device in proportion
    // to the lengths (at most that many are needed; the surplus exits at once)
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(a.splits, a.Hkv, PAGED ? 1 : B);
    cfg.blockDim = dim3(kTcThreads, 1, 1);
    cfg.dynamicSmemBytes = TcCfg::SMEM;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return jl::cuda_status(cudaLaunchKernelEx(&cfg, kern, tk, tv, a, pt, rc));
}

template <bool PAGED>
int dispatch_tc(int grp, const DecodeArgs &a, int B, const CUtensorMap &tk, const CUtensorMap &tv,
                const jl::PhaseTable &pt, const RotConsts &rc, cudaStream_t st)
{
    switch (grp) {
    case 1: return launch_tc<1, PAGED>(a, B, tk, tv, pt, rc, st);
    case 2: return launch_tc<2, PAGED>(a, B, tk, tv, pt, rc, st);
    case 4: return launch_tc<4, PAGED>(a, B, tk, tv, pt, rc, st);
    default: return launch_tc<8, PAGED>(a, B, tk, tv, pt, rc, st);
    }
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
    // paged: a.splits CTAs per kv head shared by the batch in proportion to the
    // lengths, plus one per sequence for rounding; the surplus exits at once
    dim3 grid(PAGED ? a.splits + B : a.splits, a.Hkv, PAGED ? 1 : B);
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
    // paged: the CTA target per kv head (the device derives each sequence's
    // share); otherwise this length's split count
    a.splits = paged ? p.splits_cap : p.splits;
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
    const RotConsts *rcs = nullptr;
    if (!host_tables(D, theta, a.g, &pt, &rot, &rcs)) return JL_ERR_ARG;
    CUtensorMap tk, tv;
    if (D == 128 && n >= kTcMinKeys) {
        // the tensor-core kernel: 128-key tiles as two 64-column swizzled boxes
        const Plan p = make_tc_plan(B, Hkv, n, make_plan(B, Hkv, Hq / Hkv, n).splits_cap);
        a.splits = p.splits;
        a.chunk = p.chunk;
        if (!jl::make_bshd_map(&tk, k_cache, B, n, n_cap, Hkv, D, 64, kTcKeys, true) ||
            !jl::make_bshd_map(&tv, v_cache, B, n, n_cap, Hkv, D, 64, kTcKeys, true))
            return JL_ERR_CUDA;
        return dispatch_tc<false>(Hq / Hkv, a, B, tk, tv, *pt, *rcs, (cudaStream_t)stream);
    }
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
    a.B = B;
    const jl::PhaseTable *pt = nullptr;
    const DecRot *rot = nullptr;
    const RotConsts *rcs = nullptr;
    if (!host_tables(D, theta, 1, &pt, &rot, &rcs)) return JL_ERR_ARG;  // per-sequence g on the device
    CUtensorMap tk, tv;
    if (D == 128) {
        // the tensor-core kernel: one wave of CTAs (148 / Hkv per kv head, at
        // least one per sequence), 64-row halves of its 128-key tiles loaded
        // page by page.  The partial layout's split stride stays within the
        // workspace's capacity: past it every sequence has one split.
        long long per_head = 148LL / Hkv;
        if (per_head > a.splits) per_head = a.splits;  // the workspace's split capacity
        if (per_head < 1) per_head = 1;
        const long long grid_x = per_head > B ? per_head : B;
        a.part_stride = (int)(grid_x < a.splits ? grid_x : a.splits);
        a.splits = (int)grid_x;
        if (!jl::make_bshd_map(&tk, k_pages, num_pages, page_size, page_size, Hkv, D, 64, 64, true) ||
            !jl::make_bshd_map(&tv, v_pages, num_pages, page_size, page_size, Hkv, D, 64, 64, true))
            return JL_ERR_CUDA;
        return dispatch_tc<true>(Hq / Hkv, a, B, tk, tv, *pt, *rcs, (cudaStream_t)stream);
    }
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
