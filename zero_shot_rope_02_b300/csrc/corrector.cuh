// Correction rotation of 128-row operand tiles held in shared memory, shared
// by the prefill and decode kernels.
//
// The aliased (remote) view of Jet-Long's bifocal attention scores a key at
// position p as if it sat at floor(p/g): its exact-RoPE vector is turned by
// the rotation R_{delta_p}, delta_p = floor(p/g) - p, on the fly (abstract and
// ResearchPod transcript: no second rotated copy of the cache).  The tiles are
// the TMA's 128-byte-swizzled boxes of 64 columns; the rotated values are
// written back in place as fp16 for a kind::f16 MMA.
#pragma once

#include <stdint.h>
#include <string.h>

#include "jl_common.cuh"

namespace {

constexpr int kCorrTileRows = 128;  // rows of one operand tile

// Byte offset of 16-byte chunk `cc` of row `n` inside a 128-byte-swizzled box.
__device__ __forceinline__ uint32_t sw128(int n, int cc)
{
    return (uint32_t)(n * 128 + ((cc ^ (n & 7)) << 4));
}

// Unit rotations per rotation pair d, computed on the host from the exact
// fixed-point phase, as cosine, sine and negated sine arrays (pairs of
// consecutive d load as one f32x2): a = rotation by (RPS/g - RPS) * theta_d
// (RPS rows further, no group boundary crossed), b = by (RPS/g + 1 - RPS) *
// theta_d (one boundary crossed), a2 = by twice a.
struct RotConsts {
    alignas(8) float ac[64];
    alignas(8) float as[64];
    alignas(8) float ans[64];
    alignas(8) float bc[64];
    alignas(8) float bs[64];
    alignas(8) float bns[64];
    alignas(8) float a2c[64];
    alignas(8) float a2s[64];
    alignas(8) float a2ns[64];
    // the 64 rows another CTA holds in the paired kernel (uniform steps only)
    alignas(8) float skc[64];
    alignas(8) float sks[64];
    int uni;  // g divides RPS: every RPS-row step is a
};

// Rotates 128-row bf16 tiles (SW128 boxes) in place by delta_p, p = p0 + row,
// writing fp16: the corrected operands feed a kind::f16 MMA with fp16 A and
// B, whose 11-bit significand keeps the rounding of the aliased view ~8x
// below bf16's (the rotation preserves each pair's norm, so |x| < 46000
// stays finite).  Thread t of the 128-thread group owns chunk pair
// c = t % CPR (pairs d = 8c..8c+7) and rows n0 + RPS*k; the arithmetic runs
// on packed fp32 pairs (two consecutive d per instruction).
//
// Angles.  When g divides RPS, delta moves by the same amount every RPS rows,
// so two chains of unit complex numbers (even and odd steps of this thread's
// rows, each advanced by a2) cover a tile with independent work, and after a
// tile they have advanced exactly to the first rows of the next tile: the
// remote K tiles come in order 0, 1, 2, ..., so the chains carry over and
// are re-anchored from the exact phase only every kReanchorTiles tiles.
// Otherwise every tile is anchored exactly and each step picks a or b.
//
// ROWS = 64 serves the pair kernel, whose CTAs hold one half of each K tile:
// its chains then skip the other CTA's 64 rows after every tile.
template <int D, int ROWS = 128>
struct Corrector {
    static constexpr int CPR = D / 16;        // chunk pairs per row
    static constexpr int RPS = 128 / CPR;     // rows per step
    static constexpr int STEPS = ROWS / RPS;  // rows per thread
    static constexpr int kReanchorTiles = 32;
    static constexpr uint32_t REGION = ROWS * 64 * 2;  // one 64-column box of the tile
    int c, n0, g, next_kt;
    int jm;  // generic chain: position of its next row, mod g
    bool uni;
    const unsigned long long *F;  // this thread's 8 phases (parameter space)
    const RotConsts *rc;
    jl::f32x2 ec[4], es[4], oc[4], os[4];  // chains: rows n0 and n0 + RPS of tile next_kt

    __device__ void init(int t, int g_, const jl::PhaseTable &pt, const RotConsts &rc_)
    {
        c = t % CPR;
        n0 = t / CPR;
        g = g_;
        F = pt.f + 8 * c;
        rc = &rc_;
        uni = rc_.uni != 0;
        next_kt = -1;
    }

    __device__ __forceinline__ void offsets(int n, uint32_t &lo, uint32_t &hi) const
    {
        lo = sw128(n, c);
        hi = (D == 128) ? REGION + lo : sw128(n, c + 4);
    }

    __device__ __forceinline__ static jl::f32x2 ld2(const float *p)
    {
        return *reinterpret_cast<const jl::f32x2 *>(p);
    }

    // (x, y) -> (x c - y s, y c + x s) for 8 pairs, fp16 out
    __device__ __forceinline__ static void rotate(const uint32_t (&a)[4], const uint32_t (&b)[4],
                                                  const jl::f32x2 (&zc)[4], const jl::f32x2 (&zs)[4],
                                                  uint32_t (&ao)[4], uint32_t (&bo)[4])
    {
#pragma unroll
        for (int q = 0; q < 4; q++) {
            const jl::f32x2 x = jl::bf16x2_to_f2(a[q]), y = jl::bf16x2_to_f2(b[q]);
            ao[q] = jl::f2_to_f16x2(jl::sub2(jl::mul2(x, zc[q]), jl::mul2(y, zs[q])));
            bo[q] = jl::f2_to_f16x2(jl::fma2(y, zc[q], jl::mul2(x, zs[q])));
        }
    }

    // z <- z * (cos + i sin) for the 8 pairs, given cos / sin / -sin arrays
    __device__ __forceinline__ static void cmul(jl::f32x2 (&zc)[4], jl::f32x2 (&zs)[4],
                                                const jl::f32x2 (&rcs)[4], const jl::f32x2 (&rsn)[4],
                                                const jl::f32x2 (&rns)[4])
    {
#pragma unroll
        for (int q = 0; q < 4; q++) {
            const jl::f32x2 nc = jl::fma2(zc[q], rcs[q], jl::mul2(zs[q], rns[q]));
            const jl::f32x2 ns = jl::fma2(zs[q], rcs[q], jl::mul2(zc[q], rsn[q]));
            zc[q] = nc;
            zs[q] = ns;
        }
    }

    __device__ __forceinline__ static void ld4(uint32_t addr, uint32_t (&r)[4])
    {
        asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                     : "r"(addr));
    }

    __device__ __forceinline__ static void st4(uint32_t addr, const uint32_t (&r)[4])
    {
        asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(r[0]), "r"(r[1]),
                     "r"(r[2]), "r"(r[3])
                     : "memory");
    }

    __device__ void sincos8(int off, jl::f32x2 (&zc)[4], jl::f32x2 (&zs)[4]) const
    {
#pragma unroll
        for (int q = 0; q < 4; q++) {
            float s0, c0, s1, c1;
            jl::phase_sincos(off, F[2 * q], &s0, &c0);
            jl::phase_sincos(off, F[2 * q + 1], &s1, &c1);
            zc[q] = jl::f2(c0, c1);
            zs[q] = jl::f2(s0, s1);
        }
    }

    // exact anchors of both chains at rows p and p + RPS (offsets delta + off)
    __device__ void anchor(int p, int off = 0)
    {
        sincos8(jl::delta_pos(p, g) + off, ec, es);
        sincos8(jl::delta_pos(p + RPS, g) + off, oc, os);
    }

    // g divides RPS: rows n0 + 2k*RPS on the even chain, n0 + (2k+1)*RPS on
    // the odd one, both advanced by a2 after every pair of rows
    __device__ void run_uni(uint32_t tile)
    {
        jl::f32x2 rcs[4], rsn[4], rns[4];
#pragma unroll
        for (int q = 0; q < 4; q++) {
            rcs[q] = ld2(rc->a2c + 8 * c + 2 * q);
            rsn[q] = ld2(rc->a2s + 8 * c + 2 * q);
            rns[q] = ld2(rc->a2ns + 8 * c + 2 * q);
        }
#pragma unroll 1
        for (int k = 0; k < STEPS / 2; k++) {
            const int ne = n0 + 2 * k * RPS, no = ne + RPS;
            uint32_t le, he, lo_, ho;
            offsets(ne, le, he);
            offsets(no, lo_, ho);
            uint32_t a0[4], b0[4], a1[4], b1[4], r0[4], q0[4], r1[4], q1[4];
            ld4(tile + le, a0);
            ld4(tile + he, b0);
            ld4(tile + lo_, a1);
            ld4(tile + ho, b1);
            rotate(a0, b0, ec, es, r0, q0);
            rotate(a1, b1, oc, os, r1, q1);
            st4(tile + le, r0);
            st4(tile + he, q0);
            st4(tile + lo_, r1);
            st4(tile + ho, q1);
            cmul(ec, es, rcs, rsn, rns);
            cmul(oc, os, rcs, rsn, rns);
        }
    }

    // Any g: one chain (ec, es) over this thread's rows, RPS apart; from row p
    // to p + RPS the offset moves by RPS/g - RPS, plus one when a group
    // boundary falls in between (jm = p mod g tracks that), so each step
    // multiplies by the rotation a or b, both held in registers.  `skip` more
    // steps follow without rotating (rows another CTA holds), leaving the
    // chain at the first row of the next 128-row tile.
    __device__ void run_generic(uint32_t tile, int skip)
    {
        jl::f32x2 ac2[4], as2[4], bc2[4], bs2[4];
#pragma unroll
        for (int q = 0; q < 4; q++) {
            const int i = 8 * c + 2 * q;
            ac2[q] = ld2(rc->ac + i);
            as2[q] = ld2(rc->as + i);
            bc2[q] = ld2(rc->bc + i);
            bs2[q] = ld2(rc->bs + i);
        }
        const int rs = RPS % g;
        auto step = [&]() {
            jm += rs;
            const bool carry = jm >= g;
            if (carry) jm -= g;
#pragma unroll
            for (int q = 0; q < 4; q++) {
                const jl::f32x2 rc2 = carry ? bc2[q] : ac2[q];
                const jl::f32x2 rs2 = carry ? bs2[q] : as2[q];
                const jl::f32x2 nc = jl::sub2(jl::mul2(ec[q], rc2), jl::mul2(es[q], rs2));
                const jl::f32x2 ns = jl::fma2(es[q], rc2, jl::mul2(ec[q], rs2));
                ec[q] = nc;
                es[q] = ns;
            }
        };
#pragma unroll 1
        for (int k = 0; k < STEPS; k++) {
            uint32_t lo_, hi_;
            offsets(n0 + RPS * k, lo_, hi_);
            uint32_t a[4], b[4], ao[4], bo[4];
            ld4(tile + lo_, a);
            ld4(tile + hi_, b);
            rotate(a, b, ec, es, ao, bo);
            st4(tile + lo_, ao);
            st4(tile + hi_, bo);
            step();
        }
#pragma unroll 1
        for (int k = 0; k < skip; k++) step();
    }

    // exact anchor of the generic chain at row p (offset delta + off)
    __device__ void anchor_generic(int p, int off = 0)
    {
        sincos8(jl::delta_pos(p, g) + off, ec, es);
        jm = p % g;
    }

    // the query tile at rows p0..p0+127, offsets delta + qshift (leaves the K
    // chains to be re-anchored)
    __device__ void run_q(uint32_t tile, int p0, int qshift)
    {
        if (uni) {
            anchor(p0 + n0, qshift);
            run_uni(tile);
        } else {
            anchor_generic(p0 + n0, qshift);
            run_generic(tile, 0);
        }
        next_kt = -1;
    }

    // remote K tile kt (tiles arrive in increasing order); row0 = position of
    // the held rows' first row within the 128-key tile (0, or 64 for the
    // second half in the pair kernel)
    __device__ void run_k(uint32_t tile, int kt, int row0 = 0)
    {
        if (uni) {
            if (kt != next_kt || kt % kReanchorTiles == 0) anchor(kt * kCorrTileRows + row0 + n0);
            run_uni(tile);
            if constexpr (ROWS < kCorrTileRows) {
                // skip the 64 rows the other CTA holds: one rotation per chain
                static_assert(kCorrTileRows - ROWS == 64, "the skip rotation covers 64 rows");
                jl::f32x2 rcs[4], rsn[4], rns[4];
#pragma unroll
                for (int q = 0; q < 4; q++) {
                    rcs[q] = ld2(rc->skc + 8 * c + 2 * q);
                    rsn[q] = ld2(rc->sks + 8 * c + 2 * q);
                    rns[q] = rsn[q] ^ 0x8000000080000000ull;
                }
                cmul(ec, es, rcs, rsn, rns);
                cmul(oc, os, rcs, rsn, rns);
            }
            next_kt = kt + 1;
        } else {
            if (kt != next_kt || kt % kReanchorTiles == 0) anchor_generic(kt * kCorrTileRows + row0 + n0);
            run_generic(tile, (kCorrTileRows - ROWS) / RPS);
            next_kt = kt + 1;
        }
    }
};


// Host: the step rotations of the correction for group factor g at head
// dimension D (rows per step: 16 at D = 128, 32 at D = 64).
inline void make_rot_consts(const jl::PhaseTable &pt, int D, int g, RotConsts *rc)
{
    memset(rc, 0, sizeof(*rc));
    const int rps = 128 / (D / 16);
    const long long qs = rps / g;
    rc->uni = (rps % g == 0) ? 1 : 0;
    for (int d = 0; d < D / 2; d++) {
        jl::rotation_host(pt, d, qs - rps, &rc->ac[d], &rc->as[d]);
        jl::rotation_host(pt, d, qs + 1 - rps, &rc->bc[d], &rc->bs[d]);
        jl::rotation_host(pt, d, 2 * (qs - rps), &rc->a2c[d], &rc->a2s[d]);
        rc->ans[d] = -rc->as[d];
        rc->bns[d] = -rc->bs[d];
        rc->a2ns[d] = -rc->a2s[d];
        jl::rotation_host(pt, d, (64 / rps) * (qs - rps), &rc->skc[d], &rc->sks[d]);
    }
}

}  // namespace
