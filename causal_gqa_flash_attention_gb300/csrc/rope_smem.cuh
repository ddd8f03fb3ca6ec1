// rope_smem.cuh -- RoPE applied to a tile in shared memory as it arrives from TMA
// (the rotation of "NanoEuler: C와 CUDA로 밑바닥부터 구축한 GPT-2 규모의 LLM", 기술 사양,
// RoPE bullet: adjacent pairs (2i, 2i+1) of the row at position t turn by t*theta^(-2i/D):
// (x0, x1) -> (x0 c - x1 s, x0 s + x1 c)).
//
// A tile is [ROWS x D] in the 128-byte-swizzled layout TMA writes (one 128-byte chunk
// of the row per ROWS*128-byte slab).  NT threads split the tile into 16-byte units;
// each thread loads the cos/sin of a batch of units first (the table lives in L2) and
// only then rotates, so the table latency is paid once per batch.  Rows at or beyond T
// hold TMA's zero fill; they use the table row of position 0 and stay zero.
//
// Output forms:
//   ROPE_F16       bf16 in -> fp16 in place (logit operand: 3 more mantissa bits than
//                  bf16, so the rounding of Q', K' does not dominate the logits)
//   ROPE_BF16_F16  bf16 in -> bf16 in place and an fp16 copy at `dst16`
//   ROPE_TF32      fp32 in -> fp32 rounded to TF32 (round to nearest) in place
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
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

// Largest finite fp16 is 65504; a rotated value above it would become inf.
__device__ __forceinline__ bool f16_overflow(float a) { return fabsf(a) > 65504.f; }

// Rotates rows [pos0, pos0 + ROWS) of a tile; thread t of NT.  Returns true if an
// fp16 output would have overflowed (the caller reports it).
template <int D, int ROWS, int NT, int MODE>
__device__ __forceinline__ bool rope_tile_smem(uint8_t* base, uint8_t* dst16, int pos0, int T, int t,
                                               const float2* __restrict__ rope) {
    constexpr int ES = MODE == ROPE_TF32 ? 4 : 2;
    constexpr int UPR = D * ES / 16;           // 16-byte units per row
    constexpr int PPU = 16 / ES / 2;           // (cos, sin) pairs per unit: 4 or 2
    constexpr int F4 = PPU / 2;                // float4 table loads per unit
    constexpr int TOTAL = ROWS * UPR;
    static_assert(TOTAL % NT == 0, "tile units must split evenly");
    constexpr int PER = TOTAL / NT;
    constexpr int BATCH = PER < 8 ? PER : 8;
    static_assert(PER % BATCH == 0, "batches must split evenly");
    bool overflow = false;
#pragma unroll
    for (int b0 = 0; b0 < PER; b0 += BATCH) {
        float4 tab[BATCH][F4];
        uint4 raw[BATCH];
        uint32_t off[BATCH];
#pragma unroll
        for (int k = 0; k < BATCH; ++k) {
            const int ul = t + (b0 + k) * NT;
            const int row = ul / UPR, unit = ul % UPR;
            const int pos = pos0 + row < T ? pos0 + row : 0;
            off[k] = (unit >> 3) * ROWS * 128 + sw128_offset(row, unit & 7);
            const float4* tp = reinterpret_cast<const float4*>(rope + (size_t)pos * (D / 2) + unit * PPU);
#pragma unroll
            for (int e = 0; e < F4; ++e) tab[k][e] = __ldg(tp + e);
            raw[k] = *reinterpret_cast<const uint4*>(base + off[k]);
        }
#pragma unroll
        for (int k = 0; k < BATCH; ++k) {
            if constexpr (MODE == ROPE_TF32) {
                const float4 cs = tab[k][0];
                const float x0 = __uint_as_float(raw[k].x), x1 = __uint_as_float(raw[k].y);
                const float x2 = __uint_as_float(raw[k].z), x3 = __uint_as_float(raw[k].w);
                *reinterpret_cast<uint4*>(base + off[k]) =
                    make_uint4(f32_to_tf32_rna(x0 * cs.x - x1 * cs.y), f32_to_tf32_rna(x0 * cs.y + x1 * cs.x),
                               f32_to_tf32_rna(x2 * cs.z - x3 * cs.w), f32_to_tf32_rna(x2 * cs.w + x3 * cs.z));
            } else {
                const float cs[8] = {tab[k][0].x, tab[k][0].y, tab[k][0].z, tab[k][0].w,
                                     tab[k][1].x, tab[k][1].y, tab[k][1].z, tab[k][1].w};
                const uint32_t w[4] = {raw[k].x, raw[k].y, raw[k].z, raw[k].w};
                uint32_t o16[4], ob[4];
#pragma unroll
                for (int p = 0; p < 4; ++p) {
                    const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(&w[p]);
                    const float x0 = __low2float(v), x1 = __high2float(v);
                    const float c = cs[2 * p], s = cs[2 * p + 1];
                    const float y0 = x0 * c - x1 * s, y1 = x0 * s + x1 * c;
                    overflow |= f16_overflow(y0) | f16_overflow(y1);
                    o16[p] = pack_half2(y0, y1);
                    if constexpr (MODE == ROPE_BF16_F16) ob[p] = pack_bf162(y0, y1);
                }
                if constexpr (MODE == ROPE_F16) {
                    *reinterpret_cast<uint4*>(base + off[k]) = make_uint4(o16[0], o16[1], o16[2], o16[3]);
                } else {
                    *reinterpret_cast<uint4*>(base + off[k]) = make_uint4(ob[0], ob[1], ob[2], ob[3]);
                    *reinterpret_cast<uint4*>(dst16 + off[k]) = make_uint4(o16[0], o16[1], o16[2], o16[3]);
                }
            }
        }
    }
    return overflow;
}

}  // namespace ne
