// attn_decode.cu -- one decode step of causal GQA + RoPE attention over a key/value
// cache: in every sequence b the newest token, at position len_b - 1, attends in each
// query head to the cached positions 0 .. len_b - 1 of its kv head.  That is row
// len_b - 1 of the causal attention of the training kernels (same RoPE, grouped heads and
// scale), computed for one query row per head.  The CUDA port runs inference as well as
// training ("NanoEuler: C와 CUDA로 밑바닥부터 구축한 GPT-2 규모의 LLM", CUDA 엔진 및 성능),
// and the chat command generates a continuation token by token ("NanoEuler – 순수
// C/CUDA로 처음부터 만든 GPT-2 규모 언어 모델", Code Example).
//
// One query row per head means a matrix-vector product per head: the step is bound by
// the HBM read of the cache (2 * len * D elements per kv head), not by arithmetic, so it
// runs on the CUDA cores with plain 16-byte loads; tensor cores would only add staging.
//
// Split-sequence layout: a CTA takes one (batch, kv head, group of HPC query heads of
// that kv head) and one chunk of positions, so the G query heads of a kv head share a
// single read of its keys and values, and a short batch still fills the GPU.  A key row
// of D elements is read by LPK = D / EPL lanes (16 bytes each); a warp covers 32 / LPK
// rows per step, each lane group keeping its own running max m, sum l and output o.  The
// lane groups, then the warps, are merged with the usual rescaling at the end; a second
// kernel merges the chunks when there is more than one.  The keys arrive unrotated, as
// in the training kernels, and are rotated in registers from the fp32 (cos, sin) table.
// No wait of any kind: nothing to bound.
#include <cuda_bf16.h>
#include "kernels.h"
#include "ptx.cuh"

namespace ne {
namespace {

constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;
constexpr int kUnroll = 4;          // key rows in flight per lane group
constexpr int kChunkQuantum = 64;   // chunks are whole multiples of this many positions
constexpr int kTargetCtas = 608;    // 4 CTAs per SM on 152 SMs

// One 16-byte load of a row, widened to fp32.
template <typename T>
struct Row16;
template <>
struct Row16<__nv_bfloat16> {
    static constexpr int N = 8;
    __device__ static void widen(const uint4& u, float (&f)[8]) {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(w[i] << 16);               // low half: element 2i
            f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);   // high half: element 2i+1
        }
    }
    __device__ static void store(void* dst, float x) { *static_cast<__nv_bfloat16*>(dst) = __float2bfloat16_rn(x); }
};
template <>
struct Row16<float> {
    static constexpr int N = 4;
    __device__ static void widen(const uint4& u, float (&f)[4]) {
        f[0] = __uint_as_float(u.x);
        f[1] = __uint_as_float(u.y);
        f[2] = __uint_as_float(u.z);
        f[3] = __uint_as_float(u.w);
    }
    __device__ static void store(void* dst, float x) { *static_cast<float*>(dst) = x; }
};

// Rotate N consecutive elements (N/2 adjacent pairs, the first pair index e0/2) of a row
// at position t: (x0, x1) -> (x0 c - x1 s, x0 s + x1 c), as packed f32x2 operations:
// (x0, x0) (c, s) + (-x1, x1) (s, c).  The chunk kernel is bound by its instruction
// stream, so its arithmetic runs two lanes of a float2 per instruction where it can.
template <int N>
__device__ __forceinline__ void rotate(float (&x)[N], const float2* __restrict__ rope, int t, int half, int e0) {
    const float4* tab = reinterpret_cast<const float4*>(rope + (size_t)t * half + e0 / 2);
#pragma unroll
    for (int i = 0; i < N / 4; ++i) {
        const float4 cs = __ldg(tab + i);   // (cos, sin) of pairs 2i and 2i+1 of this slice
        const float a0 = x[4 * i], a1 = x[4 * i + 1], b0 = x[4 * i + 2], b1 = x[4 * i + 3];
        const float2 ra = __ffma2_rn(make_float2(-a1, a1), make_float2(cs.y, cs.x),
                                     __fmul2_rn(make_float2(a0, a0), make_float2(cs.x, cs.y)));
        const float2 rb = __ffma2_rn(make_float2(-b1, b1), make_float2(cs.w, cs.z),
                                     __fmul2_rn(make_float2(b0, b0), make_float2(cs.z, cs.w)));
        x[4 * i] = ra.x;
        x[4 * i + 1] = ra.y;
        x[4 * i + 2] = rb.x;
        x[4 * i + 3] = rb.y;
    }
}

// Merge running softmax state (m2, l2, o2) into (m, l, o); m in log2 units of the scaled
// logits, -inf for an empty state.
template <int N>
__device__ __forceinline__ void merge(float& m, float& l, float (&o)[N], float m2, float l2, const float (&o2)[N]) {
    const float mx = fmaxf(m, m2);
    const float ref = mx == -INFINITY ? 0.f : mx;
    const float w1 = ex2(m - ref), w2 = ex2(m2 - ref);
    l = l * w1 + l2 * w2;
#pragma unroll
    for (int e = 0; e < N; ++e) o[e] = o[e] * w1 + o2[e] * w2;
    m = mx;
}

template <typename TIn, int D, int HPC>
__global__ void __launch_bounds__(kThreads, HPC <= 3 ? 4 : 3) attn_decode_kernel(DecodeArgs a) {
    constexpr int EPL = Row16<TIn>::N;    // elements per lane per row
    constexpr int LPK = D / EPL;          // lanes per key row
    constexpr int KPW = 32 / LPK;         // key rows per warp per step
    constexpr int KPS = KPW * kWarps;     // key rows per CTA per step
    static_assert(LPK >= 4 && 32 % LPK == 0, "lane layout");
    static_assert(kChunkQuantum % (KPS * kUnroll) == 0, "a chunk is whole steps");
    __shared__ float s_m[kWarps][HPC], s_l[kWarps][HPC];
    __shared__ __align__(16) float s_o[kWarps][HPC][D];

    griddep_launch_dependents();
    griddep_wait();   // the cache or q may come from the kernel before this one

    const int split = blockIdx.x;
    const int hkv = blockIdx.y / a.n_hgrp;
    const int h0 = hkv * a.G + (blockIdx.y % a.n_hgrp) * HPC;   // first query head of the CTA
    const int b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int slot = lane / LPK;          // key row of the warp's step this lane group takes
    const int e0 = (lane % LPK) * EPL;    // first element of the row this lane holds
    const int half = D / 2;

    int len = a.seq_lens[b];
    if (len < 1 || len > a.Tmax) {        // reported, then clamped so every read stays in bounds
        if (split == 0 && blockIdx.y == 0 && threadIdx.x == 0) report_error(a.err, SITE_DECODE_LEN);
        len = len < 1 ? 1 : a.Tmax;
    }
    const int j0 = split * a.chunk;
    const int j1 = min(j0 + a.chunk, len);

    // The new token's query rows, rotated at position len - 1 and scaled by log2(e)/sqrt(D).
    float qr[HPC][EPL];
#pragma unroll
    for (int h = 0; h < HPC; ++h) {
        const uint4 u = __ldg(reinterpret_cast<const uint4*>(
            static_cast<const TIn*>(a.q) + ((size_t)b * a.Hq + h0 + h) * D + e0));
        Row16<TIn>::widen(u, qr[h]);
        rotate<EPL>(qr[h], a.rope, len - 1, half, e0);
#pragma unroll
        for (int e = 0; e < EPL; ++e) qr[h][e] *= a.scale_log2;
    }

    float m[HPC], l[HPC], o[HPC][EPL];
#pragma unroll
    for (int h = 0; h < HPC; ++h) {
        m[h] = -INFINITY;
        l[h] = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) o[h][e] = 0.f;
    }

    const size_t pos_stride = (size_t)a.Hkv * D;   // elements between consecutive positions
    const size_t base = ((size_t)b * a.Tmax * a.Hkv + hkv) * D + e0;
    const TIn* kp = static_cast<const TIn*>(a.k) + base;
    const TIn* vp = static_cast<const TIn*>(a.v) + base;
    // The loop runs on the warp's first row, so every lane of a warp takes the same
    // iterations (the shuffles below need the whole warp); rows past j1 load nothing.
    for (int jw = j0 + warp * KPW; jw < j1; jw += KPS * kUnroll) {
        uint4 kr[kUnroll], vr[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int j = jw + slot + u * KPS;
            if (j < j1) {
                kr[u] = __ldg(reinterpret_cast<const uint4*>(kp + (size_t)j * pos_stride));
                vr[u] = __ldg(reinterpret_cast<const uint4*>(vp + (size_t)j * pos_stride));
            } else {
                kr[u] = make_uint4(0, 0, 0, 0);
                vr[u] = make_uint4(0, 0, 0, 0);
            }
        }
        float s[kUnroll][HPC];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int j = jw + slot + u * KPS;
            float kf[EPL];
            Row16<TIn>::widen(kr[u], kf);
            rotate<EPL>(kf, a.rope, j < j1 ? j : 0, half, e0);
#pragma unroll
            for (int h = 0; h < HPC; ++h) {
                float2 acc = make_float2(0.f, 0.f);   // even and odd elements
#pragma unroll
                for (int e = 0; e < EPL; e += 2)
                    acc = __ffma2_rn(make_float2(qr[h][e], qr[h][e + 1]), make_float2(kf[e], kf[e + 1]), acc);
                s[u][h] = acc.x + acc.y;
            }
        }
#pragma unroll
        for (int off = 1; off < LPK; off <<= 1)
#pragma unroll
            for (int u = 0; u < kUnroll; ++u)
#pragma unroll
                for (int h = 0; h < HPC; ++h) s[u][h] += __shfl_xor_sync(0xffffffffu, s[u][h], off);
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
            if (jw + slot + u * KPS >= j1)
#pragma unroll
                for (int h = 0; h < HPC; ++h) s[u][h] = -INFINITY;
        float vf[kUnroll][EPL];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) Row16<TIn>::widen(vr[u], vf[u]);
#pragma unroll
        for (int h = 0; h < HPC; ++h) {
            float mx = m[h];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) mx = fmaxf(mx, s[u][h]);
            const float ref = mx == -INFINITY ? 0.f : mx;
            const float c = ex2(m[h] - ref);
            float p[kUnroll], psum = 0.f;
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                p[u] = ex2(s[u][h] - ref);
                psum += p[u];
            }
            l[h] = l[h] * c + psum;
#pragma unroll
            for (int e = 0; e < EPL; e += 2) {
                float2 acc = __fmul2_rn(make_float2(o[h][e], o[h][e + 1]), make_float2(c, c));
#pragma unroll
                for (int u = 0; u < kUnroll; ++u)
                    acc = __ffma2_rn(make_float2(p[u], p[u]), make_float2(vf[u][e], vf[u][e + 1]), acc);
                o[h][e] = acc.x;
                o[h][e + 1] = acc.y;
            }
            m[h] = mx;
        }
    }

    // Merge the warp's lane groups (lanes with the same e0 hold the same elements).
#pragma unroll
    for (int off = LPK; off < 32; off <<= 1)
#pragma unroll
        for (int h = 0; h < HPC; ++h) {
            float o2[EPL];
#pragma unroll
            for (int e = 0; e < EPL; ++e) o2[e] = __shfl_xor_sync(0xffffffffu, o[h][e], off);
            const float m2 = __shfl_xor_sync(0xffffffffu, m[h], off);
            const float l2 = __shfl_xor_sync(0xffffffffu, l[h], off);
            merge<EPL>(m[h], l[h], o[h], m2, l2, o2);
        }
    if (slot == 0) {
#pragma unroll
        for (int h = 0; h < HPC; ++h) {
#pragma unroll
            for (int e = 0; e < EPL; ++e) s_o[warp][h][e0 + e] = o[h][e];
            if (lane == 0) {
                s_m[warp][h] = m[h];
                s_l[warp][h] = l[h];
            }
        }
    }
    __syncthreads();

    // Merge the warps: thread i takes element i % D of head i / D.
    for (int i = threadIdx.x; i < HPC * D; i += kThreads) {
        const int h = i / D, d = i % D;
        float mx = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) mx = fmaxf(mx, s_m[w][h]);
        const float ref = mx == -INFINITY ? 0.f : mx;
        float lsum = 0.f, acc = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float wt = ex2(s_m[w][h] - ref);
            lsum += s_l[w][h] * wt;
            acc += s_o[w][h][d] * wt;
        }
        const size_t row = (size_t)b * a.Hq + h0 + h;
        if (a.n_split == 1) {
            // One chunk holds the whole sequence (position 0 included): l > 0.
            Row16<TIn>::store(static_cast<TIn*>(a.o) + row * D + d, acc / lsum);
            if (d == 0) a.lse[row] = (mx + __log2f(lsum)) * 0.6931471805599453f;
        } else {
            a.part_o[(row * a.n_split + split) * D + d] = acc;
            if (d == 0) a.part_ml[row * a.n_split + split] = make_float2(mx, lsum);
        }
    }
}

// Merge of the chunks of one (batch, query head): thread d takes element d.
template <typename TIn>
__global__ void __launch_bounds__(128) attn_decode_combine_kernel(DecodeArgs a, int D) {
    griddep_launch_dependents();
    griddep_wait();   // the chunk partials come from the kernel before this one
    const size_t row = blockIdx.x;
    const int d = threadIdx.x;
    const float2* ml = a.part_ml + row * a.n_split;
    float mx = -INFINITY;
    for (int s = 0; s < a.n_split; ++s) mx = fmaxf(mx, ml[s].x);
    // The first chunk always holds position 0, so mx is finite.
    float lsum = 0.f, acc = 0.f;
    const float* po = a.part_o + row * a.n_split * D + d;
    for (int s = 0; s < a.n_split; ++s) {
        const float2 v = ml[s];
        const float wt = ex2(v.x - mx);   // 0 for an empty chunk (m = -inf)
        lsum += v.y * wt;
        acc += po[(size_t)s * D] * wt;
    }
    Row16<TIn>::store(static_cast<TIn*>(a.o) + row * D + d, acc / lsum);
    if (d == 0) a.lse[row] = (mx + __log2f(lsum)) * 0.6931471805599453f;
}

template <typename TIn, int D>
cudaError_t launch_decode_t(const DecodePlan& p, const DecodeArgs& a, cudaStream_t st) {
    const dim3 grid(p.n_split, a.Hkv * p.n_hgrp, a.B);
    cudaError_t e;
    switch (p.hpc) {
        case 4: e = launch_k(attn_decode_kernel<TIn, D, 4>, grid, dim3(kThreads), 0, st, a); break;
        case 3: e = launch_k(attn_decode_kernel<TIn, D, 3>, grid, dim3(kThreads), 0, st, a); break;
        case 2: e = launch_k(attn_decode_kernel<TIn, D, 2>, grid, dim3(kThreads), 0, st, a); break;
        default: e = launch_k(attn_decode_kernel<TIn, D, 1>, grid, dim3(kThreads), 0, st, a); break;
    }
    if (e != cudaSuccess || p.n_split == 1) return e;
    return launch_k(attn_decode_combine_kernel<TIn>, dim3(a.B * a.Hq), dim3(D), 0, st, a, D);
}

}  // namespace

DecodePlan decode_plan(int B, int Tmax, int Hq, int Hkv) {
    DecodePlan p;
    const int G = Hq / Hkv;
    p.hpc = G % 4 == 0 ? 4 : G % 3 == 0 ? 3 : G % 2 == 0 ? 2 : 1;
    p.n_hgrp = G / p.hpc;
    const long long groups = (long long)B * Hkv * p.n_hgrp;
    const long long quanta = (Tmax + kChunkQuantum - 1) / kChunkQuantum;
    long long want = (kTargetCtas + groups - 1) / (groups > 0 ? groups : 1);
    if (want < 1) want = 1;
    if (want > quanta) want = quanta;
    const long long per = (quanta + want - 1) / want;   // quanta per chunk
    p.chunk = (int)(per * kChunkQuantum);
    p.n_split = (int)((Tmax + p.chunk - 1) / p.chunk);
    if (p.n_split < 1) p.n_split = 1;
    return p;
}

cudaError_t launch_decode(bool f32, int D, const DecodePlan& p, const DecodeArgs& a, cudaStream_t st) {
    if (f32) return D == 32 ? launch_decode_t<float, 32>(p, a, st) : launch_decode_t<float, 64>(p, a, st);
    return D == 64 ? launch_decode_t<__nv_bfloat16, 64>(p, a, st) : launch_decode_t<__nv_bfloat16, 128>(p, a, st);
}

}  // namespace ne
