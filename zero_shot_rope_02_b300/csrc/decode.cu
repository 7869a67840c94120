// Bifocal single-token decode over an exact-RoPE bf16 KV cache (split-KV).
//
// The cache keeps the original positions and is never rewritten; keys that
// fall outside the local window are corrected by the rotation R_{delta_j} at
// lookup time (ResearchPod transcript on caching; Jet-Long abstract: the
// correction is applied on the fly).  The query at position n-1 is corrected
// once by R_{delta_{n-1}}.  HBM-bound: every CTA streams one contiguous chunk
// of one kv head's keys and values with 128-bit non-allocating loads, serving
// all Hq/Hkv query heads that share the kv head, and produces partial
// log-sum-exp statistics; the last CTA of each (batch, kv head) to finish
// merges the partials.
//
// Rotation angles along a thread's key sequence come from a recurrence: a
// thread steps KPS keys at a time, and delta changes by one of two constants
// per step, so the rotation is advanced by one of two precomputed unit
// complex numbers and re-anchored from the exact fixed-point phase every
// kReanchor steps.
#include <math.h>

#include "jl_common.cuh"

namespace {

constexpr int kThreads = 128;
constexpr int kUnroll = 4;
constexpr int kReanchor = 32;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ uint4 ldg_stream(const uint4 *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

struct DecodeArgs {
    const __nv_bfloat16 *q;  // [B, Hq, D]
    const __nv_bfloat16 *k;  // [B, n_cap, Hkv, D]
    const __nv_bfloat16 *v;
    __nv_bfloat16 *out;      // [B, Hq, D]
    float *lse;              // [B, Hq]
    int *counters;           // [B * Hkv]
    float *part_ml;          // [B, Hq, splits, 2]
    float *part_o;           // [B, Hq, splits, D]
    int *status;
    int Hq, Hkv, n, n_cap, w, g, splits, chunk;
    float scale_log2;        // tau * log2(e)
};

// Shared-memory carve-up (floats): q[GRP][D], qg[GRP][D], sc[GRP][chunk],
// red[KPS3][GRP][D], plus small reduction scratch.
template <int D, int GRP>
struct Smem {
    static constexpr int VC = D / 8;            // threads per V row (phase 3)
    static constexpr int KPS3 = kThreads / VC;  // keys per step in phase 3
    static size_t bytes(int chunk)
    {
        return sizeof(float) * (size_t)(2 * GRP * D + GRP * chunk + KPS3 * GRP * D + 4 * GRP * 4 +
                                        2 * GRP + 2 * GRP * 256);
    }
};

template <int D, int GRP>
__global__ void __launch_bounds__(kThreads) decode_kernel(const DecodeArgs a,
                                                          const __grid_constant__ jl::PhaseTable pt)
{
    constexpr int HALF = D / 2;
    constexpr int CPK = D / 16;           // threads per key in phase 1 (8 pairs each)
    constexpr int KPS = kThreads / CPK;   // keys per step in phase 1
    constexpr int VC = Smem<D, GRP>::VC;
    constexpr int KPS3 = Smem<D, GRP>::KPS3;

    extern __shared__ __align__(16) float smem[];
    float *sq = smem;                       // exact q, fp32
    float *sqg = sq + GRP * D;              // corrected q
    float *sc = sqg + GRP * D;              // [GRP][chunk] scores (log2 units) then p
    float *red = sc + GRP * a.chunk;        // [KPS3][GRP][D]
    float *wred = red + KPS3 * GRP * D;     // [4 warps][GRP] x 4
    float *stat = wred + 4 * GRP * 4;       // m[GRP], l[GRP]
    float *mw = stat + 2 * GRP;             // merge weights [GRP][256]
    __shared__ int s_last;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int split = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
    const int n = a.n, g = a.g;
    const int j_begin = split * a.chunk;
    const int j_end = min(n, j_begin + a.chunk);
    const int cnt = j_end - j_begin;
    const int i = n - 1;                    // query position
    const int j_split = max(0, n - a.w);    // keys below are remote

    // ---- phase 0: the GRP query heads of this kv head, exact and corrected
    const __nv_bfloat16 *qb = a.q + ((size_t)b * a.Hq + (size_t)hk * GRP) * D;
    for (int e = tid; e < GRP * D; e += kThreads) sq[e] = __bfloat162float(qb[e]);
    __syncthreads();
    if (g > 1) {
        const int di = jl::delta_pos(i, g);
        for (int d = tid; d < HALF; d += kThreads) {
            float s, c;
            jl::phase_sincos(di, pt.f[d], &s, &c);
#pragma unroll
            for (int h = 0; h < GRP; h++) {
                float x0 = sq[h * D + d], x1 = sq[h * D + d + HALF];
                sqg[h * D + d] = x0 * c - x1 * s;
                sqg[h * D + d + HALF] = x1 * c + x0 * s;
            }
        }
    }
    __syncthreads();

    // ---- phase 1: scores
    {
        const int c = tid % CPK, r = tid / CPK;
        const size_t row_stride = (size_t)a.Hkv * D / 8;  // uint4 per position
        const uint4 *kb = reinterpret_cast<const uint4 *>(a.k) +
                          ((size_t)b * a.n_cap * a.Hkv + hk) * (D / 8);
        float qr[GRP][16];

        auto load_q = [&](const float *src) {
#pragma unroll
            for (int h = 0; h < GRP; h++)
#pragma unroll
                for (int e = 0; e < 8; e++) {
                    qr[h][e] = src[h * D + 8 * c + e];
                    qr[h][8 + e] = src[h * D + HALF + 8 * c + e];
                }
        };
        // dot of one key chunk pair with the GRP queries, reduced over the CPK
        // threads of the key; thread c then writes head(s) c, c+CPK, ...
        auto score_key = [&](const float kx[16], int jj, bool valid) {
            float part[GRP];
#pragma unroll
            for (int h = 0; h < GRP; h++) {
                float acc = 0.f;
#pragma unroll
                for (int e = 0; e < 16; e++) acc = fmaf(qr[h][e], kx[e], acc);
                part[h] = acc;
            }
#pragma unroll
            for (int h = 0; h < GRP; h++)
#pragma unroll
                for (int o = 1; o < CPK; o <<= 1) part[h] += __shfl_xor_sync(0xffffffffu, part[h], o);
            if (valid) {
#pragma unroll
                for (int h = 0; h < GRP; h++)
                    if (h % CPK == c) sc[h * a.chunk + (jj - j_begin)] = part[h] * a.scale_log2;
            }
        };

        // remote keys [j_begin, min(j_end, j_split)) when g > 1
        const int rem_end = (g > 1) ? min(j_end, j_split) : j_begin;
        if (rem_end > j_begin) {
            load_q(sqg);
            const int q0 = KPS / g, r0 = KPS % g;
            float sac[8], sas[8], sbc[8], sbs[8], zc[8], zs[8];
#pragma unroll
            for (int e = 0; e < 8; e++) {
                jl::phase_sincos(q0 - KPS, pt.f[8 * c + e], &sas[e], &sac[e]);
                jl::phase_sincos(q0 + 1 - KPS, pt.f[8 * c + e], &sbs[e], &sbc[e]);
            }
            int j = j_begin + r;
            int jm = j % g;
            int since = kReanchor;  // forces an exact anchor on the first key
            // iterate in warp-uniform trip counts so the shuffles stay converged
            const int nsteps = (rem_end - j_begin + KPS - 1) / KPS;
            for (int s0 = 0; s0 < nsteps; s0 += kUnroll) {
                uint4 lo[kUnroll], hi[kUnroll];
#pragma unroll
                for (int u = 0; u < kUnroll; u++) {
                    int jj = j + u * KPS;
                    if (s0 + u < nsteps && jj < rem_end) {
                        const uint4 *row = kb + (size_t)jj * row_stride;
                        lo[u] = ldg_stream(row + c);
                        hi[u] = ldg_stream(row + c + CPK);
                    } else {
                        lo[u] = make_uint4(0, 0, 0, 0);
                        hi[u] = lo[u];
                    }
                }
#pragma unroll
                for (int u = 0; u < kUnroll; u++) {
                    if (s0 + u >= nsteps) break;  // uniform across the warp
                    int jj = j + u * KPS;
                    if (since >= kReanchor) {
                        int dj = jl::delta_pos(jj, g);
#pragma unroll
                        for (int e = 0; e < 8; e++) jl::phase_sincos(dj, pt.f[8 * c + e], &zs[e], &zc[e]);
                        since = 0;
                    }
                    uint32_t lw[4] = {lo[u].x, lo[u].y, lo[u].z, lo[u].w};
                    uint32_t hw[4] = {hi[u].x, hi[u].y, hi[u].z, hi[u].w};
                    float kx[16];
#pragma unroll
                    for (int e = 0; e < 4; e++) {
                        float a0 = jl::bf16lo(lw[e]), a1 = jl::bf16hi(lw[e]);
                        float b0 = jl::bf16lo(hw[e]), b1 = jl::bf16hi(hw[e]);
                        kx[2 * e] = a0 * zc[2 * e] - b0 * zs[2 * e];
                        kx[2 * e + 1] = a1 * zc[2 * e + 1] - b1 * zs[2 * e + 1];
                        kx[8 + 2 * e] = b0 * zc[2 * e] + a0 * zs[2 * e];
                        kx[8 + 2 * e + 1] = b1 * zc[2 * e + 1] + a1 * zs[2 * e + 1];
                    }
                    score_key(kx, jj, jj < rem_end);
                    // advance the rotation to key jj + KPS
                    jm += r0;
                    bool carry = jm >= g;
                    if (carry) jm -= g;
#pragma unroll
                    for (int e = 0; e < 8; e++) {
                        float sc_ = carry ? sbc[e] : sac[e], ss_ = carry ? sbs[e] : sas[e];
                        float nc = zc[e] * sc_ - zs[e] * ss_;
                        float ns = zs[e] * sc_ + zc[e] * ss_;
                        zc[e] = nc;
                        zs[e] = ns;
                    }
                    since++;
                }
                j += kUnroll * KPS;
            }
        }

        // exact keys [max(j_begin, rem_end), j_end)
        const int ex_begin = max(j_begin, rem_end);
        if (ex_begin < j_end) {
            load_q(sq);
            const int nsteps = (j_end - ex_begin + KPS - 1) / KPS;
            int j = ex_begin + r;
            for (int s0 = 0; s0 < nsteps; s0 += kUnroll) {
                uint4 lo[kUnroll], hi[kUnroll];
#pragma unroll
                for (int u = 0; u < kUnroll; u++) {
                    int jj = j + u * KPS;
                    if (s0 + u < nsteps && jj < j_end) {
                        const uint4 *row = kb + (size_t)jj * row_stride;
                        lo[u] = ldg_stream(row + c);
                        hi[u] = ldg_stream(row + c + CPK);
                    } else {
                        lo[u] = make_uint4(0, 0, 0, 0);
                        hi[u] = lo[u];
                    }
                }
#pragma unroll
                for (int u = 0; u < kUnroll; u++) {
                    if (s0 + u >= nsteps) break;
                    int jj = j + u * KPS;
                    uint32_t lw[4] = {lo[u].x, lo[u].y, lo[u].z, lo[u].w};
                    uint32_t hw[4] = {hi[u].x, hi[u].y, hi[u].z, hi[u].w};
                    float kx[16];
#pragma unroll
                    for (int e = 0; e < 4; e++) {
                        kx[2 * e] = jl::bf16lo(lw[e]);
                        kx[2 * e + 1] = jl::bf16hi(lw[e]);
                        kx[8 + 2 * e] = jl::bf16lo(hw[e]);
                        kx[8 + 2 * e + 1] = jl::bf16hi(hw[e]);
                    }
                    score_key(kx, jj, jj < j_end);
                }
                j += kUnroll * KPS;
            }
        }
    }
    __syncthreads();

    // ---- phase 2: per-head max and exp over the chunk
    for (int h = 0; h < GRP; h++) {
        float *row = sc + h * a.chunk;
        float m = -INFINITY;
        for (int t = tid; t < cnt; t += kThreads) m = fmaxf(m, row[t]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (lane == 0) wred[warp * GRP + h] = m;
    }
    __syncthreads();
    if (tid < GRP) {
        float m = wred[tid];
        for (int w_ = 1; w_ < kThreads / 32; w_++) m = fmaxf(m, wred[w_ * GRP + tid]);
        stat[tid] = m;
    }
    __syncthreads();
    for (int h = 0; h < GRP; h++) {
        float *row = sc + h * a.chunk;
        const float m = stat[h];
        float l = 0.f;
        for (int t = tid; t < cnt; t += kThreads) {
            float p = exp2f(row[t] - m);
            row[t] = p;
            l += p;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
        if (lane == 0) wred[4 * GRP + warp * GRP + h] = l;
    }
    __syncthreads();
    if (tid < GRP) {
        float l = 0.f;
        for (int w_ = 0; w_ < kThreads / 32; w_++) l += wred[4 * GRP + w_ * GRP + tid];
        stat[GRP + tid] = l;
    }

    // ---- phase 3: P . V over the chunk
    {
        const int dc = tid % VC, r = tid / VC;
        const size_t row_stride = (size_t)a.Hkv * D / 8;
        const uint4 *vb = reinterpret_cast<const uint4 *>(a.v) +
                          ((size_t)b * a.n_cap * a.Hkv + hk) * (D / 8);
        float acc[GRP][8];
#pragma unroll
        for (int h = 0; h < GRP; h++)
#pragma unroll
            for (int e = 0; e < 8; e++) acc[h][e] = 0.f;
        for (int j = j_begin + r; j < j_end; j += kUnroll * KPS3) {
            uint4 vv[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; u++) {
                int jj = j + u * KPS3;
                vv[u] = (jj < j_end) ? ldg_stream(vb + (size_t)jj * row_stride + dc) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < kUnroll; u++) {
                int jj = j + u * KPS3;
                if (jj >= j_end) break;
                uint32_t vw[4] = {vv[u].x, vv[u].y, vv[u].z, vv[u].w};
                float vx[8];
#pragma unroll
                for (int e = 0; e < 4; e++) {
                    vx[2 * e] = jl::bf16lo(vw[e]);
                    vx[2 * e + 1] = jl::bf16hi(vw[e]);
                }
#pragma unroll
                for (int h = 0; h < GRP; h++) {
                    float p = sc[h * a.chunk + (jj - j_begin)];
#pragma unroll
                    for (int e = 0; e < 8; e++) acc[h][e] = fmaf(p, vx[e], acc[h][e]);
                }
            }
        }
#pragma unroll
        for (int h = 0; h < GRP; h++)
#pragma unroll
            for (int e = 0; e < 8; e++) red[(r * GRP + h) * D + dc * 8 + e] = acc[h][e];
    }
    __syncthreads();

    // reduce over the KPS3 key slots; o[h][d] unnormalised
    const size_t hq0 = (size_t)b * a.Hq + (size_t)hk * GRP;
    if (a.splits == 1) {
        for (int t = tid; t < GRP * D; t += kThreads) {
            int h = t / D, d = t % D;
            float o = 0.f;
#pragma unroll
            for (int r = 0; r < KPS3; r++) o += red[(r * GRP + h) * D + d];
            a.out[(hq0 + h) * D + d] = __float2bfloat16_rn(o / stat[GRP + h]);
        }
        if (tid < GRP) a.lse[hq0 + tid] = (stat[tid] + log2f(stat[GRP + tid])) * kLn2;
        return;
    }
    for (int t = tid; t < GRP * D; t += kThreads) {
        int h = t / D, d = t % D;
        float o = 0.f;
#pragma unroll
        for (int r = 0; r < KPS3; r++) o += red[(r * GRP + h) * D + d];
        a.part_o[((hq0 + h) * a.splits + split) * D + d] = o;
    }
    if (tid < GRP) {
        a.part_ml[((hq0 + tid) * a.splits + split) * 2 + 0] = stat[tid];
        a.part_ml[((hq0 + tid) * a.splits + split) * 2 + 1] = stat[GRP + tid];
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        int ticket = atomicAdd(&a.counters[b * a.Hkv + hk], 1);
        s_last = (ticket == a.splits - 1);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();

    // ---- last CTA of this (b, kv head): merge the partial statistics
    // weights w_s = 2^(m_s - M) / L with M = max m_s, L = sum l_s 2^(m_s - M)
    for (int h = 0; h < GRP; h++) {
        const float *ml = a.part_ml + (hq0 + h) * a.splits * 2;
        float m = -INFINITY;
        for (int s = tid; s < a.splits; s += kThreads) m = fmaxf(m, __ldcg(ml + 2 * s));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (lane == 0) wred[warp * GRP + h] = m;
    }
    __syncthreads();
    if (tid < GRP) {
        float m = wred[tid];
        for (int w_ = 1; w_ < kThreads / 32; w_++) m = fmaxf(m, wred[w_ * GRP + tid]);
        stat[tid] = m;
    }
    __syncthreads();
    for (int h = 0; h < GRP; h++) {
        const float *ml = a.part_ml + (hq0 + h) * a.splits * 2;
        const float M = stat[h];
        float l = 0.f;
        for (int s = tid; s < a.splits; s += kThreads) {
            float wgt = exp2f(__ldcg(ml + 2 * s) - M);
            mw[h * 256 + s] = wgt;
            l += wgt * __ldcg(ml + 2 * s + 1);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
        if (lane == 0) wred[4 * GRP + warp * GRP + h] = l;
    }
    __syncthreads();
    if (tid < GRP) {
        float l = 0.f;
        for (int w_ = 0; w_ < kThreads / 32; w_++) l += wred[4 * GRP + w_ * GRP + tid];
        stat[GRP + tid] = l;
    }
    __syncthreads();
    for (int t = tid; t < GRP * D; t += kThreads) {
        int h = t / D, d = t % D;
        const float *po = a.part_o + (hq0 + h) * a.splits * D + d;
        float o0 = 0.f, o1 = 0.f;
        int s = 0;
        for (; s + 1 < a.splits; s += 2) {
            o0 = fmaf(mw[h * 256 + s], __ldcg(po + (size_t)s * D), o0);
            o1 = fmaf(mw[h * 256 + s + 1], __ldcg(po + (size_t)(s + 1) * D), o1);
        }
        if (s < a.splits) o0 = fmaf(mw[h * 256 + s], __ldcg(po + (size_t)s * D), o0);
        a.out[(hq0 + h) * D + d] = __float2bfloat16_rn((o0 + o1) / stat[GRP + h]);
    }
    if (tid < GRP) a.lse[hq0 + tid] = (stat[tid] + log2f(stat[GRP + tid])) * kLn2;
    if (tid == 0) a.counters[b * a.Hkv + hk] = 0;  // ready for the next call
}

// Split plan: enough CTAs to keep every SM streaming, chunks of 256..2048
// keys (a multiple of 64), at most 256 splits per (batch, kv head).
struct Plan {
    int splits, chunk;
};

Plan make_plan(int B, int Hkv, int n)
{
    const long long target_ctas = 148 * 4;
    long long per_head = (target_ctas + (long long)B * Hkv - 1) / ((long long)B * Hkv);
    if (per_head < 1) per_head = 1;
    long long chunk = (n + per_head - 1) / per_head;
    chunk = (chunk + 63) / 64 * 64;
    if (chunk < 256) chunk = 256;
    if (chunk > 2048) chunk = 2048;
    long long splits = (n + chunk - 1) / chunk;
    if (splits > 256) {
        splits = 256;
        chunk = ((n + splits - 1) / splits + 63) / 64 * 64;
        splits = (n + chunk - 1) / chunk;
    }
    return Plan{(int)splits, (int)chunk};
}

size_t ws_layout(int B, int Hq, int Hkv, int D, const Plan &p, size_t *off_ml, size_t *off_o)
{
    size_t cnt = ((size_t)B * Hkv * sizeof(int) + 255) / 256 * 256;
    size_t ml = ((size_t)B * Hq * p.splits * 2 * sizeof(float) + 255) / 256 * 256;
    size_t o = (size_t)B * Hq * p.splits * D * sizeof(float);
    if (off_ml) *off_ml = cnt;
    if (off_o) *off_o = cnt + ml;
    return cnt + ml + o;
}

bool shapes_ok(int B, int Hq, int Hkv, int n, int D)
{
    return B >= 1 && Hq >= 1 && Hkv >= 1 && n >= 1 && Hq % Hkv == 0 && (D == 64 || D == 128);
}

template <int D, int GRP>
int launch(const DecodeArgs &a, int B, const jl::PhaseTable &pt, cudaStream_t st)
{
    size_t smem = Smem<D, GRP>::bytes(a.chunk);
    auto kern = decode_kernel<D, GRP>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return jl::cuda_status(e);
    dim3 grid(a.splits, a.Hkv, B);
    kern<<<grid, kThreads, smem, st>>>(a, pt);
    return jl::cuda_status(cudaGetLastError());
}

}  // namespace

extern "C" size_t jl_bifocal_decode_workspace_size(int B, int Hq, int Hkv, int n, int D)
{
    if (!shapes_ok(B, Hq, Hkv, n, D)) return 0;
    Plan p = make_plan(B, Hkv, n);
    return ws_layout(B, Hq, Hkv, D, p, nullptr, nullptr);
}

extern "C" int jl_bifocal_decode(const void *q, const void *k_cache, const void *v_cache, void *out,
                                 float *lse, int B, int Hq, int Hkv, int n, int n_cap, int D,
                                 int L_pre, int w, double theta, void *workspace, size_t ws_bytes,
                                 void *stream)
{
    if (!q || !k_cache || !v_cache || !out || !lse) return JL_ERR_ARG;
    if (B < 1 || Hq < 1 || Hkv < 1 || n < 1 || n_cap < n || L_pre < 1 || w < 1 ||
        !(theta > 0.0) || Hq % Hkv != 0)
        return JL_ERR_ARG;
    if (D != 64 && D != 128) return JL_ERR_UNSUPPORTED;
    const int grp = Hq / Hkv;
    if (grp != 1 && grp != 2 && grp != 4 && grp != 8) return JL_ERR_UNSUPPORTED;
    if (!jl::aligned16(q) || !jl::aligned16(k_cache) || !jl::aligned16(v_cache) ||
        !jl::aligned16(out) || !jl::aligned16(lse))
        return JL_ERR_ALIGN;
    if ((long long)B * n_cap * Hkv * D > ((long long)1 << 46)) return JL_ERR_OVERFLOW;
    Plan p = make_plan(B, Hkv, n);
    size_t off_ml = 0, off_o = 0;
    size_t need = ws_layout(B, Hq, Hkv, D, p, &off_ml, &off_o);
    if (!workspace || ws_bytes < need) return JL_ERR_WORKSPACE;
    if (!jl::aligned16(workspace)) return JL_ERR_ALIGN;
    jl::PhaseTable pt;
    if (!jl::make_phase_table(&pt, D, theta)) return JL_ERR_ARG;

    DecodeArgs a;
    a.q = (const __nv_bfloat16 *)q;
    a.k = (const __nv_bfloat16 *)k_cache;
    a.v = (const __nv_bfloat16 *)v_cache;
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
    a.n_cap = n_cap;
    a.w = w;
    a.g = (int)jl::group_factor_host(n, L_pre);
    a.splits = p.splits;
    a.chunk = p.chunk;
    a.scale_log2 = (float)(1.0 / sqrt((double)D) * 1.4426950408889634);
    cudaStream_t st = (cudaStream_t)stream;
    if (D == 128) {
        switch (grp) {
        case 1: return launch<128, 1>(a, B, pt, st);
        case 2: return launch<128, 2>(a, B, pt, st);
        case 4: return launch<128, 4>(a, B, pt, st);
        default: return launch<128, 8>(a, B, pt, st);
        }
    }
    switch (grp) {
    case 1: return launch<64, 1>(a, B, pt, st);
    case 2: return launch<64, 2>(a, B, pt, st);
    case 4: return launch<64, 4>(a, B, pt, st);
    default: return launch<64, 8>(a, B, pt, st);
    }
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
    if (!q || !k_cache || !v_cache || !out || !lse) return JL_ERR_ARG;
    if (B < 1 || Hq < 1 || Hkv < 1 || n < 1 || n_cap < n || L_pre < 1 || w < 1 ||
        !(theta > 0.0) || Hq % Hkv != 0)
        return JL_ERR_ARG;
    if (D != 64 && D != 128) return JL_ERR_UNSUPPORTED;
    const Plan p = make_plan(B, Hkv, n);
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
