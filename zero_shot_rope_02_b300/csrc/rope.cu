// Exact RoPE, in place on bf16 [B, S, H, D]: the "local RoPE-faithful window"
// of the Jet-Long abstract keeps the original, unscaled frequencies; this
// kernel produces the exact-RoPE q, k and cache rows that the prefill and
// decode kernels consume (and later correct on the fly for remote keys).
//
// Bandwidth-bound: each thread owns one row and eight rotation pairs, i.e. a
// 16-byte chunk of the first half of the head vector and the matching chunk
// of the second half, loaded and stored with 128-bit accesses.  Angles come
// from the exact 64-bit phase p * F_d, so large positions lose no precision.
#include "jl_common.cuh"

namespace {

// Pairs 8c..8c+7 of one row at position p: a holds x_d, b holds x_{d+D/2}
// (d = 8c .. 8c+7), rotated by p * theta_d and rounded to bf16.  Both RoPE
// kernels below use this, so their results are bit-identical.
__device__ __forceinline__ void rotate8(uint4 &a, uint4 &b, long long p, int c, const jl::PhaseTable &pt)
{
    uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
    uint32_t ao[4], bo[4];
#pragma unroll
    for (int e = 0; e < 4; e++) {
        float s0, c0, s1, c1;
        jl::phase_sincos(p, pt.f[8 * c + 2 * e], &s0, &c0);
        jl::phase_sincos(p, pt.f[8 * c + 2 * e + 1], &s1, &c1);
        float x0 = jl::bf16lo(av[e]), x1 = jl::bf16hi(av[e]);
        float y0 = jl::bf16lo(bv[e]), y1 = jl::bf16hi(bv[e]);
        ao[e] = jl::pack_bf16x2(x0 * c0 - y0 * s0, x1 * c1 - y1 * s1);
        bo[e] = jl::pack_bf16x2(y0 * c0 + x0 * s0, y1 * c1 + x1 * s1);
    }
    a = make_uint4(ao[0], ao[1], ao[2], ao[3]);
    b = make_uint4(bo[0], bo[1], bo[2], bo[3]);
}

// One thread per (row, chunk of 8 pairs); requires (D/2) % 8 == 0.
__global__ void __launch_bounds__(256) rope_vec8_kernel(uint4 *x, long long rows, int S, int H,
                                                        int D, long long pos0,
                                                        const __grid_constant__ jl::PhaseTable pt)
{
    const int half = D / 2;
    const int chunks = half / 8;
    long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= rows * chunks) return;
    long long r = t / chunks;
    int c = (int)(t - r * chunks);
    long long s = (r / H) % S;
    long long p = pos0 + s;
    uint4 *row = x + r * (D / 8);
    uint4 a = row[c];           // x_d,       d = 8c .. 8c+7
    uint4 b = row[c + chunks];  // x_{d+D/2}
    rotate8(a, b, p, c, pt);
    row[c] = a;
    row[c + chunks] = b;
}

// RoPE fused into the KV-cache write: the new tokens' raw k and their v
// ([B, S_new, H, D]) go to cache rows n_past .. n_past+S_new-1 of
// [B, n_cap, H, D], k rotated at its position on the way.  One read and one
// write of each byte, instead of a rotation in place plus two copies.  One
// thread per (row, chunk of 8 pairs) moves its chunks of both k and v.
__global__ void __launch_bounds__(256) rope_cache_write_kernel(const uint4 *k_raw, const uint4 *v,
                                                               uint4 *k_cache, uint4 *v_cache,
                                                               long long rows, int S_new, int H, int D,
                                                               long long n_past, int n_cap,
                                                               const __grid_constant__ jl::PhaseTable pt)
{
    const int chunks = D / 16;
    long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= rows * chunks) return;
    long long r = t / chunks;  // row of [B, S_new, H]
    int c = (int)(t - r * chunks);
    const long long h = r % H, bs = r / H;
    const long long s = bs % S_new, b = bs / S_new;
    const long long p = n_past + s;
    const long long dst = ((b * n_cap + p) * H + h) * (D / 8);
    const uint4 *ks = k_raw + r * (D / 8), *vs = v + r * (D / 8);
    uint4 a = ks[c], bb = ks[c + chunks];
    rotate8(a, bb, p, c, pt);
    k_cache[dst + c] = a;
    k_cache[dst + c + chunks] = bb;
    v_cache[dst + c] = vs[c];
    v_cache[dst + c + chunks] = vs[c + chunks];
}

// One thread per (row, pair): any even D.
__global__ void __launch_bounds__(256) rope_scalar_kernel(__nv_bfloat16 *x, long long rows, int S,
                                                          int H, int D, long long pos0,
                                                          const __grid_constant__ jl::PhaseTable pt)
{
    const int half = D / 2;
    long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= rows * half) return;
    long long r = t / half;
    int d = (int)(t - r * half);
    long long s = (r / H) % S;
    float sn, cs;
    jl::phase_sincos(pos0 + s, pt.f[d], &sn, &cs);
    __nv_bfloat16 *row = x + r * D;
    float a = __bfloat162float(row[d]), b = __bfloat162float(row[d + half]);
    row[d] = __float2bfloat16_rn(a * cs - b * sn);
    row[d + half] = __float2bfloat16_rn(b * cs + a * sn);
}

}  // namespace

extern "C" int jl_rope_apply(void *x, int B, int S, int H, int D, int64_t pos0, double theta,
                             void *stream)
{
    if (!x || B < 1 || S < 1 || H < 1 || D < 2 || pos0 < 0 || !(theta > 0.0)) return JL_ERR_ARG;
    if ((D & 1) || D / 2 > jl::kMaxPairs) return JL_ERR_UNSUPPORTED;
    if (!jl::aligned16(x)) return JL_ERR_ALIGN;
    if (pos0 > ((int64_t)1 << 62) - S) return JL_ERR_OVERFLOW;
    const long long rows = (long long)B * S * H;
    // one launch: at most 2^31 - 1 blocks of 256 threads (one per row and pair at worst)
    if (rows > ((long long)1 << 40) || rows * (D / 2) / 256 >= 0x7fffffffLL) return JL_ERR_OVERFLOW;
    jl::PhaseTable pt;
    if (!jl::make_phase_table(&pt, D, theta)) return JL_ERR_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    if ((D / 2) % 8 == 0) {
        long long work = rows * (D / 16);
        long long blocks = (work + 255) / 256;
        rope_vec8_kernel<<<(unsigned)blocks, 256, 0, st>>>((uint4 *)x, rows, S, H, D, pos0, pt);
    } else {
        long long work = rows * (D / 2);
        long long blocks = (work + 255) / 256;
        rope_scalar_kernel<<<(unsigned)blocks, 256, 0, st>>>((__nv_bfloat16 *)x, rows, S, H, D,
                                                             pos0, pt);
    }
    return jl::cuda_status(cudaGetLastError());
}

extern "C" int jl_rope_cache_write(const void *k_raw, const void *v, void *k_cache, void *v_cache, int B,
                                   int S_new, int H, int D, int n_past, int n_cap, double theta,
                                   void *stream)
{
    if (!k_raw || !v || !k_cache || !v_cache || B < 1 || S_new < 1 || H < 1 || n_past < 0 ||
        !(theta > 0.0))
        return JL_ERR_ARG;
    if ((long long)n_past + S_new > n_cap) return JL_ERR_ARG;
    if (D < 16 || D % 16 != 0 || D / 2 > jl::kMaxPairs) return JL_ERR_UNSUPPORTED;
    if (!jl::aligned16(k_raw) || !jl::aligned16(v) || !jl::aligned16(k_cache) || !jl::aligned16(v_cache))
        return JL_ERR_ALIGN;
    const long long rows = (long long)B * S_new * H;
    if (rows > ((long long)1 << 40) || rows * (D / 16) / 256 >= 0x7fffffffLL ||
        (long long)B * n_cap * H * D > ((long long)1 << 46))
        return JL_ERR_OVERFLOW;
    jl::PhaseTable pt;
    if (!jl::make_phase_table(&pt, D, theta)) return JL_ERR_ARG;
    const long long work = rows * (D / 16);
    rope_cache_write_kernel<<<(unsigned)((work + 255) / 256), 256, 0, (cudaStream_t)stream>>>(
        (const uint4 *)k_raw, (const uint4 *)v, (uint4 *)k_cache, (uint4 *)v_cache, rows, S_new, H, D,
        n_past, n_cap, pt);
    return jl::cuda_status(cudaGetLastError());
}
