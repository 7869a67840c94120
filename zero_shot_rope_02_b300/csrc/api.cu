// Host side of the C ABI that every kernel file shares: status strings, the
// group-factor rule, the fixed-point rotation phases, the device status word
// and the debug exports.
#include <math.h>
#include <stdio.h>

#include "jl_common.cuh"
#include "sm100_ptx.cuh"
#include "tile_class.cuh"

// Device status word: kernels record JL_ERR_TIMEOUT / JL_ERR_GUARD here
// instead of trapping.  One per device that loads the library.
__device__ int g_jl_status_word;

namespace jl {

bool make_phase_table(PhaseTable *t, int D, double theta)
{
    if (!t || D < 2 || (D & 1) || D / 2 > kMaxPairs || !(theta > 0.0) || !isfinite(theta))
        return false;
    const int h = D / 2;
    for (int d = 0; d < kMaxPairs; d++) t->f[d] = 0ull;
    for (int d = 0; d < h; d++) {
        // theta_d / (2 pi) turns, reduced mod 1, as a 64-bit binary fraction.
        long double turns = powl((long double)theta, -2.0L * d / (long double)D) /
                            (2.0L * 3.14159265358979323846264338327950288L);
        turns -= floorl(turns);
        long double scaled = ldexpl(turns, 64);
        unsigned long long f;
        if (scaled >= 18446744073709551616.0L)
            f = 0ull;  // rounds up to a whole turn
        else
            f = (unsigned long long)scaled;
        t->f[d] = f;
    }
    return true;
}

void rotation_host(const PhaseTable &t, int d, long long offset, float *c, float *s)
{
    const unsigned long long ph = (unsigned long long)offset * t.f[d];
    const double turns = (double)(long long)ph * 5.42101086242752217003726400434970855712890625e-20;  // 2^-64
    const double a = turns * 6.283185307179586476925286766559;
    *c = (float)cos(a);
    *s = (float)sin(a);
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled through the runtime's driver entry point (the
// library does not link libcuda itself).
static EncodeTiledFn encode_fn()
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

// Encoded maps per host thread, keyed by everything the encoding depends on:
// repeated calls on the same tensors (a decode step's caches, one per layer;
// benchmark loops) skip the driver's encode.  Open addressing on a hash of the
// key; a full probe sequence evicts its first slot.
namespace {
struct MapKey {
    const void *base;
    int B, S, S_cap, H, D, box_d, box_rows, sw;
    bool operator==(const MapKey &o) const
    {
        return base == o.base && B == o.B && S == o.S && S_cap == o.S_cap && H == o.H && D == o.D &&
               box_d == o.box_d && box_rows == o.box_rows && sw == o.sw;
    }
    uint64_t hash() const
    {
        uint64_t h = reinterpret_cast<uintptr_t>(base) * 0x9E3779B97F4A7C15ull;
        const int f[8] = {B, S, S_cap, H, D, box_d, box_rows, sw};
        for (int i = 0; i < 8; i++) h = (h ^ (uint64_t)(uint32_t)f[i]) * 0x100000001B3ull;
        return h ^ (h >> 29);
    }
};
struct MapCache {
    static constexpr int N = 256, PROBE = 8;
    MapKey key[N];
    CUtensorMap map[N];
    bool used[N] = {};
};
}  // namespace

static bool encode_bshd_map(CUtensorMap *m, const void *base, int B, int S, int S_cap, int H, int D,
                            int box_d, int box_rows, bool swizzle128);

bool make_bshd_map(CUtensorMap *m, const void *base, int B, int S, int S_cap, int H, int D,
                   int box_d, int box_rows, bool swizzle128)
{
    thread_local MapCache cache;
    const MapKey k{base, B, S, S_cap, H, D, box_d, box_rows, swizzle128 ? 1 : 0};
    const int h0 = (int)(k.hash() % MapCache::N);
    int slot = -1;
    for (int p = 0; p < MapCache::PROBE; p++) {
        const int i = (h0 + p) % MapCache::N;
        if (cache.used[i] && cache.key[i] == k) {
            *m = cache.map[i];
            return true;
        }
        if (!cache.used[i] && slot < 0) slot = i;
    }
    if (!encode_bshd_map(m, base, B, S, S_cap, H, D, box_d, box_rows, swizzle128)) return false;
    if (slot < 0) slot = h0;
    cache.key[slot] = k;
    cache.map[slot] = *m;
    cache.used[slot] = true;
    return true;
}

static bool encode_bshd_map(CUtensorMap *m, const void *base, int B, int S, int S_cap, int H, int D,
                            int box_d, int box_rows, bool swizzle128)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn || S < 1 || S > S_cap) return false;
    cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)S, (cuuint64_t)B};
    // byte strides of dims 1..3 (H, S, B); a batch entry spans S_cap rows
    cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2, (cuuint64_t)S_cap * H * D * 2};
    cuuint32_t box[4] = {(cuuint32_t)box_d, 1, (cuuint32_t)box_rows, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int *status_word_ptr()
{
    static int *cache[64] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return nullptr;
    }
    if (!cache[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_jl_status_word) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        cache[dev] = static_cast<int *>(p);
    }
    return cache[dev];
}

int cuda_status(cudaError_t e)
{
    if (e == cudaSuccess) return JL_OK;
    cudaGetLastError();
    return JL_ERR_CUDA;
}

}  // namespace jl

namespace {

__global__ void grouped_positions_kernel(int32_t *out, int64_t S, int g)
{
    int64_t p = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (p < S) out[p] = jl::grouped_pos((int)p, g);
}

// One warp waits on an mbarrier that nothing ever arrives on, through the
// same bounded warp-wide wait the attention kernels use, with a short limit:
// the wait must give up, record JL_ERR_TIMEOUT and let the kernel return.
__global__ void wait_timeout_kernel(int *status, unsigned long long limit_ns, int *gave_up)
{
    __shared__ __align__(8) unsigned long long bar;
    __shared__ int abort_flag;
    const uint32_t b = jl::ptx::smem_u32(&bar);
    if (threadIdx.x == 0) {
        jl::ptx::mbar_init(b, 1);
        abort_flag = 0;
        jl::ptx::fence_mbar_init();
    }
    __syncwarp();
    const jl::ptx::WaitCtx wc{status, &abort_flag, limit_ns};
    const bool ok = jl::ptx::wait_bar_warp(b, 0, wc);
    if (threadIdx.x == 0) *gave_up = ok ? 0 : 1;
}

__global__ void tile_classes_kernel(int8_t *out, int S, int w, int g, int nt)
{
    int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= nt * nt) return;
    int qi = t / nt, kj = t % nt;
    out[t] = (int8_t)jl::tile_class(qi * 128, kj * 128, 128, 128, S, w, g);
}

}  // namespace

extern "C" {

const char *jl_status_string(int status)
{
    switch (status) {
    case JL_OK: return "JL_OK";
    case JL_ERR_ARG: return "JL_ERR_ARG: argument out of range";
    case JL_ERR_ALIGN: return "JL_ERR_ALIGN: pointer not 16-byte aligned";
    case JL_ERR_UNSUPPORTED: return "JL_ERR_UNSUPPORTED: shape without a kernel";
    case JL_ERR_OVERFLOW: return "JL_ERR_OVERFLOW: size overflows";
    case JL_ERR_CUDA: return "JL_ERR_CUDA: CUDA call or launch failed";
    case JL_ERR_TIMEOUT: return "JL_ERR_TIMEOUT: a bounded device wait expired";
    case JL_ERR_WORKSPACE: return "JL_ERR_WORKSPACE: workspace missing or too small";
    case JL_ERR_GUARD: return "JL_ERR_GUARD: an in-kernel guard fired";
    default: return "unknown jl_status";
    }
}

const char *jl_version(void) { return "0.1.0"; }

int jl_group_factor(int64_t s, int64_t L_pre, int32_t *g_out)
{
    if (!g_out || s < 1 || L_pre < 1) return JL_ERR_ARG;
    int64_t g = jl::group_factor_host(s, L_pre);
    if (g > INT32_MAX) return JL_ERR_OVERFLOW;
    *g_out = (int32_t)g;
    return JL_OK;
}

int jl_group_factor_ex(int64_t s, int64_t L_pre, int64_t w, unsigned flags, int32_t *g_out)
{
    if (!g_out || s < 1 || L_pre < 1 || w < 1) return JL_ERR_ARG;
    if (flags & ~(unsigned)(JL_VARIANT_PER_QUERY_G | JL_VARIANT_SLIDING | JL_VARIANT_QUERY_SHIFT))
        return JL_ERR_ARG;
    if ((flags & JL_VARIANT_SLIDING) && flags != JL_VARIANT_SLIDING) return JL_ERR_ARG;
    int64_t g = jl::group_factor_host(s, L_pre);
    if (flags & JL_VARIANT_SLIDING) g = 1;
    if (flags & JL_VARIANT_QUERY_SHIFT) {
        g = jl::group_factor_shift_host(s, L_pre, w);
        if (g < 1) return JL_ERR_ARG;
    }
    if (g > INT32_MAX) return JL_ERR_OVERFLOW;
    *g_out = (int32_t)g;
    return JL_OK;
}

int jl_debug_grouped_positions(int64_t S, int64_t L_pre, int32_t *out_dev, void *stream)
{
    if (!out_dev || S < 1 || L_pre < 1) return JL_ERR_ARG;
    if (S > INT32_MAX) return JL_ERR_OVERFLOW;
    int g = (int)jl::group_factor_host(S, L_pre);
    int64_t blocks = (S + 255) / 256;
    grouped_positions_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(out_dev, S, g);
    return jl::cuda_status(cudaGetLastError());
}

int jl_debug_tile_classes(int S, int L_pre, int w, int8_t *out_dev, void *stream)
{
    if (!out_dev || S < 1 || L_pre < 1 || w < 1) return JL_ERR_ARG;
    int nt = (S + 127) / 128;
    int g = (int)jl::group_factor_host(S, L_pre);
    int64_t n = (int64_t)nt * nt;
    tile_classes_kernel<<<(unsigned)((n + 255) / 256), 256, 0, (cudaStream_t)stream>>>(out_dev, S, w,
                                                                                      g, nt);
    return jl::cuda_status(cudaGetLastError());
}

int jl_debug_wait_timeout(int64_t limit_ns, int *gave_up_dev, void *stream)
{
    if (!gave_up_dev || limit_ns < 1 || limit_ns > 100000000) return JL_ERR_ARG;
    int *st = jl::status_word_ptr();
    if (!st) return JL_ERR_CUDA;
    wait_timeout_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(st, (unsigned long long)limit_ns, gave_up_dev);
    return jl::cuda_status(cudaGetLastError());
}

int jl_debug_status(int *status_out)
{
    if (!status_out) return JL_ERR_ARG;
    int v = 0;
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpyFromSymbol(&v, g_jl_status_word, sizeof(int));
    if (e == cudaSuccess) {
        int zero = 0;
        e = cudaMemcpyToSymbol(g_jl_status_word, &zero, sizeof(int));
    }
    if (e != cudaSuccess) return jl::cuda_status(e);
    *status_out = v;
    return JL_OK;
}

}  // extern "C"
