// Shared device/host helpers of the Dynamic Bifocal RoPE library: the exact
// fixed-point phase used for every rotation angle, the group-factor and
// aliasing integer rules, the device status word and bounded waits.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "../../include/jetlong.h"

namespace jl {

// Largest supported D/2 for the rotation tables (D <= 256).
constexpr int kMaxPairs = 128;

// Rotation frequencies as exact fixed-point phases: F[d] = theta_d / (2*pi)
// in units of 2^-64 turns, reduced mod 1 turn.  The phase of an integer
// offset p is then (uint64)(p * F[d]) mod 2^64 -- the multiply wraps for
// free, negative p included -- so a rotation angle never loses the bits that
// an fp32 product p*theta_d would drop at p ~ 1e5.
struct PhaseTable {
    unsigned long long f[kMaxPairs];
};

// Host: fill F[d] for d < D/2 (theta_d = theta^(-2d/D), the RoPE frequencies
// of the "local RoPE-faithful window").  Returns false on bad arguments.
bool make_phase_table(PhaseTable *t, int D, double theta);

// Host: TMA tensor map over a bf16 [B, S_cap, H, D] tensor of which rows
// [0, S) of every batch entry are mapped, viewed as the 4-D tensor {D, H, S,
// B} (batch stride S_cap rows); box {box_d, 1, box_rows, 1}; 128-byte swizzle
// or none.  Loads outside the mapped rows read zeros, so rows at or past S
// (a cache's unused capacity, whatever it holds) never reach a kernel.
// False if the driver refuses it.
bool make_bshd_map(CUtensorMap *m, const void *base, int B, int S, int S_cap, int H, int D,
                   int box_d, int box_rows, bool swizzle128);

// Host: cos / sin of the angle offset * theta_d, from the same exact
// fixed-point phase the device uses, evaluated in double precision.
void rotation_host(const PhaseTable &t, int d, long long offset, float *c, float *s);

// Host: group factor g = max(1, ceil(s / L)) -- the smallest integer g with
// floor((s-1)/g) <= L-1 (ResearchPod summary: smallest integer grouping).
inline int64_t group_factor_host(int64_t s, int64_t L) { return s <= L ? 1 : (s + L - 1) / L; }

// Host: group factor of the query-shift variant -- the smallest g >= 1 with
// floor((s-1)/g) + w - floor(w/g) <= L-1, the largest aliased distance once the
// aliased query position is shifted by w - floor(w/g) (Self-Extend's grouping,
// named as a baseline in the ResearchPod summary).  -1 when no g does (w >= L
// while s > L).  Smaller g than the unshifted factor cannot work (the shift is
// >= 0), and g = max(s, w) + 1 always does once w < L, so the search ends.
inline int64_t group_factor_shift_host(int64_t s, int64_t L, int64_t w)
{
    if (s <= L) return 1;
    if (w >= L) return -1;
    for (int64_t g = (s + L - 1) / L;; g++)
        if ((s - 1) / g + (w - w / g) <= L - 1) return g;
}

// Host: pointer to the device status word of the current device (cached per
// device).  Returns nullptr if CUDA is unusable.
int *status_word_ptr();

// Host: cudaError -> JL status, clearing the sticky-free error state.
int cuda_status(cudaError_t e);

// Host: true when p is 16-byte aligned.
inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---------------------------------------------------------------- device side

// sin/cos of the angle p * theta_d given its fixed-point frequency F.
// The top 32 bits of the 64-bit phase are a signed fraction of a half turn
// in [-1, 1); sincospif evaluates it.
__device__ __forceinline__ void phase_sincos(long long p, unsigned long long F, float *s, float *c)
{
    unsigned long long ph = static_cast<unsigned long long>(p) * F;
    int hi = static_cast<int>(ph >> 32);
    float x = static_cast<float>(hi) * 4.656612873077392578125e-10f;  // 2^-31
    sincospif(x, s, c);
}

// floor(p / g) for p >= 0, g >= 1.
__device__ __forceinline__ int grouped_pos(int p, int g) { return p / g; }

// delta_p = floor(p/g) - p  (<= 0): the correction offset of position p.
__device__ __forceinline__ int delta_pos(int p, int g) { return p / g - p; }

__device__ __forceinline__ void record_status(int *status, int code)
{
    if (status) atomicCAS(status, 0, code);
}

__device__ __forceinline__ unsigned long long globaltimer_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Upper bound of any single wait inside a kernel; far above the longest
// legitimate wait (a few microseconds), far below a watchdog.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ float bf16lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

// Two fp32 -> packed bf16x2 (round to nearest even); `lo` in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

// Two fp32 -> packed fp16x2 (round to nearest even); `lo` in the low half.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi)
{
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

// Packed fp32 pairs (f32x2 arithmetic of the sm_100 family): one 64-bit
// register holds (lo, hi); one instruction does two fp32 operations.
typedef unsigned long long f32x2;

__device__ __forceinline__ f32x2 f2(float lo, float hi)
{
    f32x2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ void f2_split(f32x2 v, float &lo, float &hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

__device__ __forceinline__ f32x2 fma2(f32x2 a, f32x2 b, f32x2 c)
{
    f32x2 r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}

__device__ __forceinline__ f32x2 mul2(f32x2 a, f32x2 b)
{
    f32x2 r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

__device__ __forceinline__ f32x2 sub2(f32x2 a, f32x2 b)
{
    f32x2 r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

__device__ __forceinline__ f32x2 add2(f32x2 a, f32x2 b)
{
    f32x2 r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

// Both bf16 halves of a packed word, widened exactly to an fp32 pair.
__device__ __forceinline__ f32x2 bf16x2_to_f2(uint32_t u) { return f2(bf16lo(u), bf16hi(u)); }

// fp32 pair -> packed fp16x2 (round to nearest even), lo in the low half.
__device__ __forceinline__ uint32_t f2_to_f16x2(f32x2 v)
{
    float lo, hi;
    f2_split(v, lo, hi);
    return pack_f16x2(lo, hi);
}

// fp32 pair -> packed bf16x2 (round to nearest even), lo in the low half.
__device__ __forceinline__ uint32_t f2_to_bf16x2(f32x2 v)
{
    float lo, hi;
    f2_split(v, lo, hi);
    return pack_bf16x2(lo, hi);
}

// Three-input fp32 maximum.
__device__ __forceinline__ float fmax3(float a, float b, float c)
{
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

}  // namespace jl
