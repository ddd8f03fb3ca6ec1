// rope_smem.cuh -- RoPE applied to a tile in shared memory as it arrives from TMA
// (the rotation of "NanoEuler: C와 CUDA로 밑바닥부터 구축한 GPT-2 규모의 LLM", 기술 사양,
// RoPE bullet: adjacent pairs (2i, 2i+1) of the row at position t turn by t*theta^(-2i/D):
// (x0, x1) -> (x0 c - x1 s, x0 s + x1 c)).
//
// A tile is [ROWS x D] in the 128-byte-swizzled layout TMA writes (one 128-byte chunk
// of the row per ROWS*128-byte slab), split in 16-byte units.  Thread t of NT always
// takes the same unit u = t % UPR (so the same PPU frequency pairs) of rows
// r0 = t / UPR, r0 + RSTEP, r0 + 2*RSTEP, ... with RSTEP = NT / UPR.  Its angles
// therefore form an arithmetic progression: the cos/sin of the first row come from the
// table (one load per tile, which the caller can issue a tile early) and every further
// row is reached by one more rotation by RSTEP*w (angle addition; the step is the
// table row RSTEP).  Rows at or beyond T hold TMA's zero fill and stay zero.
//
// Output forms:
//   ROPE_F16       bf16 in -> fp16 in place (logit operand: 3 more mantissa bits than
//                  bf16, so the rounding of Q', K' does not dominate the logits)
//   ROPE_BF16_F16  bf16 in -> bf16 in place and an fp16 copy at `dst16`
//   ROPE_TF32      fp32 in -> fp32 rounded to TF32 (round to nearest) in place
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include "kernels.h"
#include "ptx.cuh"

namespace ne {

enum RopeMode { ROPE_F16 = 0, ROPE_BF16_F16 = 1, ROPE_TF32 = 2 };

__device__ __forceinline__ uint32_t f32_to_tf32_rna(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ uint32_t pack_half2(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t pack_bf162(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

// The rotation (x0, x1) -> (x0 c - x1 s, x0 s + x1 c) with its roundings fixed by
// explicit intrinsics: left to the compiler, the contraction of a product into an FMA
// may differ between two instantiations of the same kernel, and so would the results.
__device__ __forceinline__ float rot0(float x0, float x1, float c, float s) {
    return __fmaf_rn(x0, c, __fmul_rn(-x1, s));
}
__device__ __forceinline__ float rot1(float x0, float x1, float c, float s) {
    return __fmaf_rn(x0, s, __fmul_rn(x1, c));
}

template <int D, int ROWS, int NT, int MODE>
struct RopeTile {
    static constexpr int ES = MODE == ROPE_TF32 ? 4 : 2;
    static constexpr int UPR = D * ES / 16;        // 16-byte units per row
    static constexpr int PPU = 16 / ES / 2;        // (cos, sin) pairs per unit: 4 or 2
    static constexpr int F4 = PPU / 2;             // float4 table reads per unit
    static constexpr int RSTEP = NT / UPR;         // rows between a thread's units
    static constexpr int KSTEPS = ROWS / RSTEP;    // units per thread per tile
    static_assert(NT % UPR == 0 && ROWS % RSTEP == 0, "thread layout");
    static_assert(RSTEP < kRopeTableMinRows, "step row must exist in the table");

    int unit, r0;
    float4 step[F4];                               // (cos, sin) of RSTEP * w for this unit's pairs

    __device__ __forceinline__ void init(int t, const float2* __restrict__ rope) {
        unit = t % UPR;
        r0 = t / UPR;
        const float4* sp = reinterpret_cast<const float4*>(rope + (size_t)RSTEP * (D / 2) + unit * PPU);
#pragma unroll
        for (int e = 0; e < F4; ++e) step[e] = __ldg(sp + e);
    }
    // cos/sin of this thread's first row of the tile starting at position pos0.
    __device__ __forceinline__ void load_base(float4 (&b)[F4], int pos0, int T,
                                              const float2* __restrict__ rope) const {
        const int pos = pos0 + r0 < T ? pos0 + r0 : 0;
        const float4* bp = reinterpret_cast<const float4*>(rope + (size_t)pos * (D / 2) + unit * PPU);
#pragma unroll
        for (int e = 0; e < F4; ++e) b[e] = __ldg(bp + e);
    }
    // Rotates the tile; with CHECK, returns true if an fp16 output of a row before
    // zero_row would have overflowed (without, the caller detects overflow downstream and
    // this returns false).  Rows zero_row and later (padding past a sequence's length) are
    // then overwritten with zeros; the rotation itself reads every row unconditionally, so
    // the common case (no padding in the tile) runs the plain loop.
    template <bool CHECK = true>
    __device__ __forceinline__ bool apply(uint8_t* base, uint8_t* dst16, float4 (&b)[F4],
                                          int zero_row = ROWS) const {
        float amax = 0.f;
#pragma unroll
        for (int k = 0; k < KSTEPS; ++k) {
            const int row = r0 + k * RSTEP;
            const uint32_t off = (unit >> 3) * ROWS * 128 + sw128_offset(row, unit & 7);
            const uint4 raw = *reinterpret_cast<const uint4*>(base + off);
            if constexpr (MODE == ROPE_TF32) {
                const float4 cs = b[0];
                const float x0 = __uint_as_float(raw.x), x1 = __uint_as_float(raw.y);
                const float x2 = __uint_as_float(raw.z), x3 = __uint_as_float(raw.w);
                *reinterpret_cast<uint4*>(base + off) =
                    make_uint4(f32_to_tf32_rna(rot0(x0, x1, cs.x, cs.y)), f32_to_tf32_rna(rot1(x0, x1, cs.x, cs.y)),
                               f32_to_tf32_rna(rot0(x2, x3, cs.z, cs.w)), f32_to_tf32_rna(rot1(x2, x3, cs.z, cs.w)));
            } else {
                const float cs[8] = {b[0].x, b[0].y, b[0].z, b[0].w, b[1].x, b[1].y, b[1].z, b[1].w};
                const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
                uint32_t o16[4], ob[4];
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(&w[p]);
                    const float x0 = __low2float(v), x1 = __high2float(v);
                    const float c = cs[2 * p], s = cs[2 * p + 1];
                    const float y0 = rot0(x0, x1, c, s), y1 = rot1(x0, x1, c, s);
                    if constexpr (CHECK) amax = fmaxf(amax, row < zero_row ? fmaxf(fabsf(y0), fabsf(y1)) : 0.f);
                    o16[p] = pack_half2(y0, y1);
                    if constexpr (MODE == ROPE_BF16_F16) ob[p] = pack_bf162(y0, y1);
                }
                if constexpr (MODE == ROPE_F16) {
                    *reinterpret_cast<uint4*>(base + off) = make_uint4(o16[0], o16[1], o16[2], o16[3]);
                } else {
                    *reinterpret_cast<uint4*>(base + off) = make_uint4(ob[0], ob[1], ob[2], ob[3]);
                    *reinterpret_cast<uint4*>(dst16 + off) = make_uint4(o16[0], o16[1], o16[2], o16[3]);
                }
            }
            if (k + 1 < KSTEPS) {   // advance every pair's angle by RSTEP * w
#pragma unroll
                for (int e = 0; e < F4; ++e) {
                    const float4 c = b[e], s = step[e];
                    b[e] = make_float4(rot0(c.x, c.y, s.x, s.y), rot1(c.x, c.y, s.x, s.y),
                                       rot0(c.z, c.w, s.z, s.w), rot1(c.z, c.w, s.z, s.w));
                }
            }
        }
        if (zero_row < ROWS) {      // padding rows: zeros in every output
#pragma unroll
            for (int k = 0; k < KSTEPS; ++k) {
                const int row = r0 + k * RSTEP;
                if (row < zero_row) continue;
                const uint32_t off = (unit >> 3) * ROWS * 128 + sw128_offset(row, unit & 7);
                *reinterpret_cast<uint4*>(base + off) = make_uint4(0u, 0u, 0u, 0u);
                if constexpr (MODE == ROPE_BF16_F16) *reinterpret_cast<uint4*>(dst16 + off) = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        return amax > 65504.f;   // largest finite fp16
    }
};

// One-shot form: rotate rows [pos0, pos0 + ROWS) of a tile with thread t of NT.  Rows at
// positions len and later (padding of a shorter sequence) are written as zeros.
template <int D, int ROWS, int NT, int MODE, bool CHECK = true>
__device__ __forceinline__ bool rope_tile_smem(uint8_t* base, uint8_t* dst16, int pos0, int T, int t,
                                               const float2* __restrict__ rope, int len) {
    RopeTile<D, ROWS, NT, MODE> rt;
    rt.init(t, rope);
    float4 b[RopeTile<D, ROWS, NT, MODE>::F4];
    rt.load_base(b, pos0, T, rope);
    return rt.template apply<CHECK>(base, dst16, b, len - pos0);
}

}  // namespace ne
