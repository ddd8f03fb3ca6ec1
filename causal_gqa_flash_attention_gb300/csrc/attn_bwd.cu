// attn_bwd.cu -- backward of causal GQA + RoPE attention on tcgen05 tensor cores.
//
// The hand-written backward of "NanoEuler: C와 CUDA로 밑바닥부터 구축한 GPT-2 규모의
// LLM" (검증 및 안정성), for the attention of the same page's 기술 사양 (RoPE, GQA) and
// 커널 구현 (tiling, no T x T matrix).  With s = 1/sqrt(D), Q' = R Q, K' = R K:
//   P  = exp(s Q'K'^T - LSE)  (recomputed from the forward's LSE, causal mask)
//   dV = sum_heads P^T dO,  dP = dO V^T,  dS = P o (dP - Delta),  Delta = rowsum(dO o O)
//   dK = R^T sum_heads s dS^T Q',  dQ = R^T s dS K'
// Three kernels on one stream:
//   bwd_pre   Delta = rowsum(dO o O) (fp32) and zeroing of the fp32 dQ accumulator;
//   bwd_main  KV-major: one CTA per (batch, kv head, 128-key tile) loops over the G
//             query heads of its group and every query tile on or after the diagonal.
//             dK and dV accumulate in TMEM across the whole group (no atomics); each
//             (head, query tile) step adds its dS K' into the fp32 dQ accumulator;
//   bwd_post  dQ = s R^T (accumulator), cast to the output dtype.
//
// bwd_main warp roles (512 threads).  One thread issues a tcgen05.mma only every
// ~100 cycles, so three warps issue UMMAs, each for its own accumulators:
//   warp 0      TMA producer: K, V once; Q and dO tiles into a ring.
//   warp 1      TMEM allocator (all 512 columns); issuer A: S^T = K'Q'^T (fp16), dP^T = V dO^T.
//   warp 2      issuer B: dV += P^T dO (P^T from TMEM), dK' += dS^T Q'.
//   warp 3      issuer C: dQ' partial = dS K'.
//   warps 4-7   RoPE on K once and on every Q tile; drain of the dQ partial (thread =
//               query row) into the fp32 accumulator with 16-byte atomics.
//   warps 8-15  two groups, thread = key row, each on half of the query columns: P^T
//               and dS^T from S^T, dP^T, LSE, Delta; P^T to TMEM, dS^T (bf16) to shared
//               memory; at the end group 0 writes dK (inverse rotation), group 1 dV.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include "kernels.h"
#include "ptx.cuh"
#include "rope_smem.cuh"

namespace ne {

namespace {

// ------------------------------------------------------------------------ pre
// Delta[b,h,t] = sum_d dO[b,t,h,d] * O[b,t,h,d]; also zeroes dq_acc and, when q16 is set
// (bf16 tensors), writes Q' = R_t Q rounded to fp16 (the logit and dK' operand of the
// head_dim-64 main kernel, so each query row is rotated once instead of once per key
// tile).  A group of LPR lanes takes one row (D elements); rows are [B,T,Hq] in memory
// order.  Each warp zeroes the accumulator rows of the units it reads: interleaving the
// zero stores with the loads row by row kept HBM busier than a zeroing sweep followed by
// the loads.
// DELTA_ONLY (after the training forward, which stored R Q and zeroed the accumulator):
// the pass only reads O and dO, so it keeps four row units in flight per thread.
template <typename Tin, int D, bool VL, bool DELTA_ONLY = false>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const BwdPreArgs a) {
    constexpr int EPV = 16 / sizeof(Tin);        // elements per 16-byte vector
    constexpr int LPR = D / EPV;                 // lanes per row (8 or 16)
    constexpr int RPW = 32 / LPR;                // rows per warp unit
    // Units per pass: with the rotation and the zero stores one was fastest when measured;
    // the loads alone need more in flight.
    constexpr int U = DELTA_ONLY ? 4 : 1;
    constexpr int ZPL = D / 4 / LPR;             // 16-byte zero stores per lane per row
    griddep_launch_dependents();
    griddep_wait();
    // Index math in 32 bits (rows * D < 2^31 is checked at the API) with the divisions
    // by Hq and T as multiply-shifts: the 64-bit divide sequences dominated this pass's
    // instruction count.
    const uint32_t lane = threadIdx.x & 31;
    const uint32_t sub = lane / LPR, li = lane % LPR;
    const uint32_t wg = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const uint32_t nw = (gridDim.x * blockDim.x) >> 5;
    const uint32_t rows = (uint32_t)a.rows;
    const uint4* o4 = static_cast<const uint4*>(a.o);
    const uint4* g4 = static_cast<const uint4*>(a.dO);
    const bool rot = !DELTA_ONLY && sizeof(Tin) == 2 && a.q16 != nullptr;
    bool ovf = false;
    for (uint32_t r0 = wg * RPW + sub; r0 - sub < rows; r0 += nw * RPW * U) {
        uint4 ov[U], gv[U], qv[U];
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const uint32_t row = r0 + k * nw * RPW;
            if (row < rows) {
                ov[k] = o4[row * LPR + li];
                gv[k] = g4[row * LPR + li];
                if (rot) qv[k] = static_cast<const uint4*>(a.q)[row * LPR + li];
            } else {
                ov[k] = gv[k] = qv[k] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        if constexpr (sizeof(Tin) == 2) {
            if (rot) {
                // Lane li holds elements 8li .. 8li+7 of the row: pairs 4li .. 4li+3.
#pragma unroll
                for (int k = 0; k < U; ++k) {
                    const uint32_t row = r0 + k * nw * RPW;
                    if (row >= rows) continue;
                    const uint32_t bt = fast_div(row, a.div_hq);
                    const uint32_t bb = fast_div(bt, a.div_t);
                    const uint32_t t = bt - bb * (uint32_t)a.T;
                    // Padding positions (past the sequence's length) get R Q = 0.
                    const bool pad = VL && (int)t >= seq_len(a.seq_lens, (int)bb, a.T);
                    const float4* cs4 = reinterpret_cast<const float4*>(a.rope + (size_t)t * a.rope_ld + 4 * li);
                    const float4 c01 = __ldg(cs4), c23 = __ldg(cs4 + 1);
                    const float cs[8] = {c01.x, c01.y, c01.z, c01.w, c23.x, c23.y, c23.z, c23.w};
                    const uint32_t wq[4] = {qv[k].x, qv[k].y, qv[k].z, qv[k].w};
                    uint32_t o16[4];
#pragma unroll
                    for (int pr = 0; pr < 4; ++pr) {
                        const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wq[pr]));
                        const float c = cs[2 * pr], sn = cs[2 * pr + 1];
                        const float y0 = pad ? 0.f : rot0(x.x, x.y, c, sn), y1 = pad ? 0.f : rot1(x.x, x.y, c, sn);
                        ovf |= fmaxf(fabsf(y0), fabsf(y1)) > 65504.f;
                        const __half2 h = __floats2half2_rn(y0, y1);
                        o16[pr] = *reinterpret_cast<const uint32_t*>(&h);
                    }
                    static_cast<uint4*>(a.q16)[row * LPR + li] = make_uint4(o16[0], o16[1], o16[2], o16[3]);
                }
            }
        }
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const uint32_t row = r0 + k * nw * RPW;
            if (!DELTA_ONLY && row < rows && a.dq_acc) {
                float4* z = reinterpret_cast<float4*>(a.dq_acc + (size_t)row * D);
#pragma unroll
                for (int e = 0; e < ZPL; ++e) z[li + e * LPR] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
#pragma unroll
        for (int k = 0; k < U; ++k) {
            float acc = 0.f;
            if constexpr (sizeof(Tin) == 2) {
                const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(&ov[k]);
                const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&gv[k]);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 of = __bfloat1622float2(o2[e]), gf = __bfloat1622float2(g2[e]);
                    acc = fmaf(of.x, gf.x, acc);
                    acc = fmaf(of.y, gf.y, acc);
                }
            } else {
                acc = __uint_as_float(ov[k].x) * __uint_as_float(gv[k].x) +
                      __uint_as_float(ov[k].y) * __uint_as_float(gv[k].y) +
                      __uint_as_float(ov[k].z) * __uint_as_float(gv[k].z) +
                      __uint_as_float(ov[k].w) * __uint_as_float(gv[k].w);
            }
#pragma unroll
            for (int off = LPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            const uint32_t row = r0 + k * nw * RPW;
            if (row < rows && li == 0) {
                const uint32_t bt = fast_div(row, a.div_hq), b = fast_div(bt, a.div_t);
                const uint32_t h = row - bt * (uint32_t)a.Hq, t = bt - b * (uint32_t)a.T;
                a.delta[(b * (uint32_t)a.Hq + h) * (uint32_t)a.T + t] =
                    !VL || (int)t < seq_len(a.seq_lens, (int)b, a.T) ? acc : 0.f;
            }
        }
    }
    if (ovf) report_error(a.err, SITE_RANGE);   // a rotated query beyond the fp16 range
}

// ------------------------------------------------------------------------ post
// dq[row] = s * R_t^T dq_acc[row].  A thread takes 8 consecutive elements (4 pairs) of
// a row, U such groups in flight per pass; the (cos, sin) table is L2-resident.
template <typename Tout, int D>
__global__ void __launch_bounds__(256) bwd_post_kernel(const BwdPostArgs a) {
    constexpr int G8 = D / 8;                    // 8-element groups per row
    constexpr int U = 2;
    griddep_launch_dependents();
    griddep_wait();
    // 32-bit index math (rows * D < 2^31), divisions by Hq and T as multiply-shifts.
    const uint32_t n = (uint32_t)a.rows * G8;
    const uint32_t tg = blockIdx.x * blockDim.x + threadIdx.x;
    const uint32_t nt = gridDim.x * blockDim.x;
    const float4* acc4 = reinterpret_cast<const float4*>(a.dq_acc);
    const float4* rope4 = reinterpret_cast<const float4*>(a.rope);
    for (uint32_t i0 = tg; i0 < n; i0 += nt * U) {
        float4 g[U][2], cs[U][2];
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const uint32_t idx = i0 + k * nt;
            if (idx < n) {
                const uint32_t row = idx / G8;
                const uint32_t c8 = idx % G8;
                const uint32_t bt = fast_div(row, a.div_hq);
                const uint32_t t = bt - fast_div(bt, a.div_t) * (uint32_t)a.T;
                g[k][0] = acc4[idx * 2];
                g[k][1] = acc4[idx * 2 + 1];
                cs[k][0] = __ldg(rope4 + (size_t)t * (a.rope_ld / 2) + 2 * c8);
                cs[k][1] = __ldg(rope4 + (size_t)t * (a.rope_ld / 2) + 2 * c8 + 1);
            }
        }
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const uint32_t idx = i0 + k * nt;
            if (idx >= n) continue;
            float y[8];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const float4 v = g[k][h], c = cs[k][h];
                y[4 * h + 0] = a.scale * (v.x * c.x + v.y * c.y);
                y[4 * h + 1] = a.scale * (-v.x * c.y + v.y * c.x);
                y[4 * h + 2] = a.scale * (v.z * c.z + v.w * c.w);
                y[4 * h + 3] = a.scale * (-v.z * c.w + v.w * c.z);
            }
            if constexpr (sizeof(Tout) == 2) {
                uint4 o;
                __nv_bfloat162 p0 = __floats2bfloat162_rn(y[0], y[1]), p1 = __floats2bfloat162_rn(y[2], y[3]);
                __nv_bfloat162 p2 = __floats2bfloat162_rn(y[4], y[5]), p3 = __floats2bfloat162_rn(y[6], y[7]);
                o.x = *reinterpret_cast<uint32_t*>(&p0);
                o.y = *reinterpret_cast<uint32_t*>(&p1);
                o.z = *reinterpret_cast<uint32_t*>(&p2);
                o.w = *reinterpret_cast<uint32_t*>(&p3);
                reinterpret_cast<uint4*>(a.dq)[idx] = o;
            } else {
                reinterpret_cast<float4*>(a.dq)[idx * 2] = make_float4(y[0], y[1], y[2], y[3]);
                reinterpret_cast<float4*>(a.dq)[idx * 2 + 1] = make_float4(y[4], y[5], y[6], y[7]);
            }
        }
    }
}

// ------------------------------------------------------------------------ main
template <int D>
struct BwdCfg {
    static constexpr int ES = 2;
    static constexpr int BKV = 128;                 // key rows per CTA
    static constexpr int BQ = 128;                  // query rows per step
    static constexpr int ROWB = D * ES;
    static constexpr int NCH = ROWB / 128;
    static constexpr int EPC = 64;
    static constexpr int NQS = D <= 64 ? 2 : 1;     // Q/dO stages
    static constexpr bool DS_ALIASES_Q16 = D > 64;  // dS^T reuses the fp16 Q' buffer
    static constexpr int KV_BYTES = BKV * ROWB;
    static constexpr int Q_BYTES = BQ * ROWB;
    static constexpr int STAGE_BYTES = 3 * Q_BYTES; // Q' (bf16) | Q' (fp16) | dO
    static constexpr int DS_BYTES = BKV * BQ * 2;   // dS^T bf16 [key][query]
    static constexpr int DQ_STAGE = BQ * 128;       // one 32-column fp32 chunk of dQ' for a bulk reduce-add
    static constexpr int SMEM =
        1024 + 3 * KV_BYTES + NQS * STAGE_BYTES + (DS_ALIASES_Q16 ? 0 : DS_BYTES) + DQ_STAGE;
    // TMEM columns
    static constexpr int S_COL = 0;                 // S^T, then P^T (bf16 packed)
    static constexpr int DP_COL = 128;              // dP^T
    static constexpr int DV_COL = 256;
    static constexpr int DK_COL = 256 + D;
    static constexpr int DQ_COL = D <= 64 ? 256 + 2 * D : 128;  // D = 128 shares dP^T's columns
    static constexpr bool DQ_ALIASES_DP = D > 64;
    // P^T (bf16, 64 packed columns): its own columns when they fit (D = 64), so the next
    // step's S^T can be issued before dV has read P^T; over S^T otherwise.
    static constexpr bool PT_OWN = 256 + 3 * D + 64 <= 512;
    static constexpr int PT_COL = PT_OWN ? 256 + 3 * D : 0;
    // Packed P^T column of query column q (TMEM column pair q/2).  Sharing S^T's columns,
    // each half of the queries is packed into the first half of its own 64 S^T columns,
    // which its group has already read.
    static __device__ __forceinline__ int pt_col(int q) {
        return PT_OWN ? PT_COL + (q >> 1) : S_COL + (q >> 1) + ((q >> 6) << 5);
    }
    static constexpr int KSTEPS_D = ROWB / 32;      // K-steps over head_dim
    static constexpr int KSTEPS_Q = BQ / 16;        // K-steps over query rows
    static constexpr int KSTEPS_KV = BKV / 16;      // K-steps over key rows
    static constexpr int THREADS = 512;
    static_assert(SMEM <= 227 * 1024, "shared memory");
    static_assert(DS_BYTES == Q_BYTES || !DS_ALIASES_Q16, "alias needs equal sizes");
};

// VL: per-sequence lengths (padded batch).  Without them every length is T, rows past T
// arrive as TMA's zero fill, and the padding code compiles away.
template <int D, bool VL>
__global__ void __launch_bounds__(512, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_dq, const BwdArgs a) {
    using C = BwdCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sK = smem;                            // K' bf16 (rotated in place)
    uint8_t* sK16 = sK + C::KV_BYTES;              // K' fp16 (logit operand)
    uint8_t* sV = sK16 + C::KV_BYTES;
    uint8_t* sStage = sV + C::KV_BYTES;            // NQS x (Q' bf16 | Q' fp16 | dO)
    uint8_t* sdS = C::DS_ALIASES_Q16 ? sStage + C::Q_BYTES : sStage + C::NQS * C::STAGE_BYTES;
    uint8_t* sDQ = sStage + C::NQS * C::STAGE_BYTES + (C::DS_ALIASES_Q16 ? 0 : C::DS_BYTES);   // dQ' chunk
    auto stage_q = [&](int s) { return sStage + s * C::STAGE_BYTES; };
    auto stage_q16 = [&](int s) { return sStage + s * C::STAGE_BYTES + C::Q_BYTES; };

    __shared__ __align__(8) uint64_t bar_kv_full, bar_k_ready, bar_s_full, bar_dp_full, bar_ds_ready,
        bar_p_free, bar_ds_free, bar_dq_full, bar_dq_free, bar_dkv_full, bar_final, bar_sdp_read;
    __shared__ __align__(8) uint64_t bar_qdo_full[C::NQS], bar_q_ready[C::NQS], bar_qdo_empty[C::NQS];
    __shared__ __align__(8) uint64_t bar_rows[2];   // LSE/Delta of a query tile staged (double buffer)
    __shared__ __align__(8) uint64_t bar_dqs_free, bar_dqs_full;   // dQ' chunk: read by its reduce / staged
    __shared__ __align__(16) float s_lse[2][C::BQ];
    __shared__ __align__(16) float s_delta[2][C::BQ];
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int hkv = blockIdx.x, b = blockIdx.y, j = blockIdx.z;
    const int T = a.T, G = a.G;
    const int kv0 = j * C::BKV;
    // Query tiles end at the sequence's length (T without per-sequence lengths); a key
    // tile wholly past it has no query tile and writes zero gradients.
    const int len = VL ? seq_len(a.seq_lens, b, T) : T;
    const int n_qt = (len + C::BQ - 1) / C::BQ;
    const int i_first = kv0 / C::BQ;
    const int per_head = n_qt > i_first ? n_qt - i_first : 0;
    const int n_it = G * per_head;

    if (tid == 0) {
        mbar_init(smem_u32(&bar_kv_full), 1);
        mbar_init(smem_u32(&bar_k_ready), 128);
        mbar_init(smem_u32(&bar_s_full), 1);
        mbar_init(smem_u32(&bar_dp_full), 1);
        mbar_init(smem_u32(&bar_ds_ready), 256);
        mbar_init(smem_u32(&bar_p_free), 1);
        mbar_init(smem_u32(&bar_sdp_read), 256);   // S^T and dP^T of a step are in registers
        mbar_init(smem_u32(&bar_ds_free), 2);      // dK issuer and dQ issuer
        mbar_init(smem_u32(&bar_dq_full), 1);
        mbar_init(smem_u32(&bar_dq_free), 128);
        mbar_init(smem_u32(&bar_dkv_full), 1);
        mbar_init(smem_u32(&bar_final), 3);        // one commit per issuer
        mbar_init(smem_u32(&bar_rows[0]), 256);
        mbar_init(smem_u32(&bar_rows[1]), 256);
        mbar_init(smem_u32(&bar_dqs_free), 1);       // the thread that issued the reduce
        mbar_init(smem_u32(&bar_dqs_full), 128);     // every row of the chunk
        for (int s = 0; s < C::NQS; ++s) {
            mbar_init(smem_u32(&bar_qdo_full[s]), 1);
            mbar_init(smem_u32(&bar_q_ready[s]), 128);
            mbar_init(smem_u32(&bar_qdo_empty[s]), 2);   // dK issuer and dQ issuer
        }
        abort_flag = 0;
        fence_mbar_init();
        // The tensor maps are kernel parameters, not outputs of an earlier kernel: fetch
        // them before the dependency wait, under the previous kernel's tail.
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        tma_prefetch_desc(&tm_do);
        tma_prefetch_desc(&tm_dq);
    }
    if (warp == 1) {
        __syncwarp();
        tmem_alloc(smem_u32(&tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    griddep_launch_dependents();   // after the TMEM allocation
    griddep_wait();                // LSE, Delta and the zeroed accumulator are visible
    const uint32_t tm = tmem_slot;
    const WaitCtx w{a.err, &abort_flag, a.timeout_ns};

    // Shared-memory descriptors, built once; a step or a stage only moves the start address.
    auto kdesc = [](const void* p) { return sdesc(smem_u32(p), 16, 1024); };        // K-major
    auto mndesc = [](const void* p, uint32_t lbo) { return sdesc(smem_u32(p), lbo, 1024); };  // MN-major

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint32_t kvf = smem_u32(&bar_kv_full);
            mbar_arrive_expect_tx(kvf, 2 * C::KV_BYTES);
            for (int c = 0; c < C::NCH; ++c) {
                tma_load_4d(smem_u32(sK + c * C::BKV * 128), &tm_k, kvf, c * C::EPC, hkv, kv0, b);
                tma_load_4d(smem_u32(sV + c * C::BKV * 128), &tm_v, kvf, c * C::EPC, hkv, kv0, b);
            }
            int issued = 0;
            for (int it = 0; it < n_it; ++it) {
                const int s = it % C::NQS;
                const int h = hkv * G + it / per_head;
                const int q0 = (i_first + it % per_head) * C::BQ;
                if (it >= C::NQS &&
                    !mbar_wait(smem_u32(&bar_qdo_empty[s]), ((it / C::NQS) - 1) & 1, w, SITE_BWD_QDO_EMPTY))
                    break;
                const uint32_t f = smem_u32(&bar_qdo_full[s]);
                mbar_arrive_expect_tx(f, 2 * C::Q_BYTES);
                for (int c = 0; c < C::NCH; ++c) {
                    tma_load_4d(smem_u32(stage_q(s) + c * C::BQ * 128), &tm_q, f, c * C::EPC, h, q0, b);
                    tma_load_4d(smem_u32(stage_q(s) + 2 * C::Q_BYTES + c * C::BQ * 128), &tm_do, f, c * C::EPC, h,
                                q0, b);
                }
                ++issued;
            }
            mbar_wait_drain(kvf, 0, w, SITE_BWD_DRAIN);
            for (int it = max(0, issued - C::NQS); it < issued; ++it)
                mbar_wait_drain(smem_u32(&bar_qdo_full[it % C::NQS]), (it / C::NQS) & 1, w, SITE_BWD_DRAIN);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ issuer A: S^T, dP^T
        // Each issuer warp runs its loop and waits together (UMMA operands stay warp-
        // uniform) and one elected lane issues each batch with its commits: a loop run by
        // lane 0 alone cost several instructions per UMMA.
        {
            constexpr uint32_t id_s = idesc_make(FMT_F16, 128, C::BQ, false, false);   // S^T (fp16 Q', K')
            constexpr uint32_t id_dp = idesc_make(FMT_BF16, 128, C::BQ, false, false); // dP^T
            const uint64_t dK16 = kdesc(sK16), dV = kdesc(sV), dQ0 = kdesc(stage_q(0));
            bool ok = mbar_wait_warp(smem_u32(&bar_k_ready), 0, w, SITE_BWD_KV);
            for (int it = 0; ok && it < n_it; ++it) {
                const int s = it % C::NQS;
                const uint32_t so = s * C::STAGE_BYTES;
                if (!(ok = mbar_wait_warp(smem_u32(&bar_q_ready[s]), (it / C::NQS) & 1, w, SITE_BWD_Q_READY))) break;
                // The previous step's S^T and dP^T must have been read out of TMEM; when P^T
                // shares S^T's columns, dV must also have read P^T.
                if (it > 0) {
                    const uint32_t bar = smem_u32(C::PT_OWN ? &bar_sdp_read : &bar_p_free);
                    if (!(ok = mbar_wait_warp(bar, (it - 1) & 1, w, SITE_BWD_DS_READY))) break;
                }
                tc_fence_after();
                const uint64_t dQ16 = sdesc_add(dQ0, so + C::Q_BYTES), dO = sdesc_add(dQ0, so + 2 * C::Q_BYTES);
                if (elect_one()) {
#pragma unroll
                    for (int ks = 0; ks < C::KSTEPS_D; ++ks) {  // S^T = K' Q'^T, K = head_dim
                        const uint32_t off = (ks * 32 >> 7) * C::BKV * 128 + (ks * 32 & 127);
                        const uint32_t offq = (ks * 32 >> 7) * C::BQ * 128 + (ks * 32 & 127);
                        umma_ss<false>(tm + C::S_COL, sdesc_add(dK16, off), sdesc_add(dQ16, offq), id_s, ks > 0);
                    }
                    umma_commit(smem_u32(&bar_s_full));
                }
                __syncwarp();
                if constexpr (C::DQ_ALIASES_DP) {               // dQ of the previous step sits in dP^T's columns
                    if (it > 0 && !(ok = mbar_wait_warp(smem_u32(&bar_dq_free), (it - 1) & 1, w, SITE_BWD_DQ_FREE)))
                        break;
                    tc_fence_after();
                }
                if (elect_one()) {
#pragma unroll
                    for (int ks = 0; ks < C::KSTEPS_D; ++ks) {  // dP^T = V dO^T
                        const uint32_t off = (ks * 32 >> 7) * C::BKV * 128 + (ks * 32 & 127);
                        const uint32_t offq = (ks * 32 >> 7) * C::BQ * 128 + (ks * 32 & 127);
                        umma_ss<false>(tm + C::DP_COL, sdesc_add(dV, off), sdesc_add(dO, offq), id_dp, ks > 0);
                    }
                    umma_commit(smem_u32(&bar_dp_full));
                }
                __syncwarp();
            }
            if (elect_one()) umma_commit(smem_u32(&bar_final));
            __syncwarp();
        }
    } else if (warp == 2) {
        // ------------------------------------------------------------ issuer B: dV, dK
        {
            constexpr uint32_t id_dv = idesc_make(FMT_BF16, 128, D, false, true);      // B MN-major
            const uint64_t dQmn0 = mndesc(stage_q(0), C::BQ * 128), dDS0 = kdesc(sdS);
            bool ok = true;
            for (int it = 0; ok && it < n_it; ++it) {
                const int s = it % C::NQS;
                const uint32_t so = s * C::STAGE_BYTES;
                const uint64_t dDS = sdesc_add(dDS0, C::DS_ALIASES_Q16 ? so : 0);
                if (!(ok = mbar_wait_warp(smem_u32(&bar_ds_ready), it & 1, w, SITE_BWD_DS_READY))) break;
                tc_fence_after();
                const uint64_t dOmn = sdesc_add(dQmn0, so + 2 * C::Q_BYTES), dQmn = sdesc_add(dQmn0, so);
                if (elect_one()) {
#pragma unroll
                    for (int ks = 0; ks < C::KSTEPS_Q; ++ks)     // dV += P^T dO (P^T from TMEM)
                        umma_ts<false>(tm + C::DV_COL, tm + C::pt_col(ks * 16), sdesc_add(dOmn, ks * 16 * 128), id_dv,
                                       (it > 0 || ks > 0) ? 1u : 0u);
                    umma_commit(smem_u32(&bar_p_free));
#pragma unroll
                    for (int ks = 0; ks < C::KSTEPS_Q; ++ks) {   // dK' += dS^T Q'
                        const uint32_t off = (ks * 32 >> 7) * C::BKV * 128 + (ks * 32 & 127);
                        umma_ss<false>(tm + C::DK_COL, sdesc_add(dDS, off), sdesc_add(dQmn, ks * 16 * 128), id_dv,
                                       (it > 0 || ks > 0) ? 1u : 0u);
                    }
                    umma_commit(smem_u32(&bar_qdo_empty[s]));
                    umma_commit(smem_u32(&bar_ds_free));
                }
                __syncwarp();
            }
            if (elect_one()) {
                umma_commit(smem_u32(&bar_dkv_full));
                umma_commit(smem_u32(&bar_final));
            }
            __syncwarp();
        }
    } else if (warp == 3) {
        // ------------------------------------------------------------ issuer C: dQ
        {
            constexpr uint32_t id_dq = idesc_make(FMT_BF16, 128, D, true, true);       // A, B MN-major
            const uint64_t dKmn = mndesc(sK, C::BKV * 128), dDSmn0 = mndesc(sdS, C::BKV * 128);
            bool ok = true;
            for (int it = 0; ok && it < n_it; ++it) {
                const int s = it % C::NQS;
                const uint64_t dDSmn = sdesc_add(dDSmn0, C::DS_ALIASES_Q16 ? s * C::STAGE_BYTES : 0);
                if (!(ok = mbar_wait_warp(smem_u32(&bar_ds_ready), it & 1, w, SITE_BWD_DS_READY))) break;
                if (it > 0 && !(ok = mbar_wait_warp(smem_u32(&bar_dq_free), (it - 1) & 1, w, SITE_BWD_DQ_FREE))) break;
                if constexpr (C::DQ_ALIASES_DP) {               // dQ overwrites dP^T: issuer A's dP^T is done
                    if (!(ok = mbar_wait_warp(smem_u32(&bar_dp_full), it & 1, w, SITE_BWD_DP_FULL))) break;
                }
                tc_fence_after();
                if (elect_one()) {
#pragma unroll
                    for (int ks = 0; ks < C::KSTEPS_KV; ++ks)    // dQ'_part = dS K'
                        umma_ss<false>(tm + C::DQ_COL, sdesc_add(dDSmn, ks * 16 * 128), sdesc_add(dKmn, ks * 16 * 128),
                                       id_dq, ks > 0);
                    umma_commit(smem_u32(&bar_dq_full));
                    umma_commit(smem_u32(&bar_qdo_empty[s]));
                    umma_commit(smem_u32(&bar_ds_free));
                }
                __syncwarp();
            }
            if (elect_one()) umma_commit(smem_u32(&bar_final));
            __syncwarp();
        }
    } else if (warp < 8) {
        // ------------------------------------------------------------ RoPE on K and Q; dQ drain
        // Thread r: RoPE units of the K tile and of every Q tile, and query row r of the dQ
        // partial (TMEM lane r), added into the fp32 accumulator.  The Q of step it+1 is
        // rotated before the dQ of step it is drained.
        // The drain stages 32 columns of the partial at a time (16 KB) and adds each chunk
        // with one bulk tensor reduce-add (per-thread 16-byte atomics kept the accumulator's
        // traffic in flight on every thread and made the drain the longest-stalled role).
        // Chunk kk (over all steps) waits until the reduce of chunk kk - 1 has read the
        // staging tile.
        const int r = tid - 128;
        const uint32_t lt = tm + ((uint32_t)((warp & 3) * 32) << 16);
        bool ovf = false;
        int kk = 0;                                    // dQ' chunks staged so far
        auto drain = [&](int it) -> bool {
            const int h = hkv * G + it / per_head;
            const int q0 = (i_first + it % per_head) * C::BQ;
            if (!mbar_wait_warp(smem_u32(&bar_dq_full), it & 1, w, SITE_BWD_DQ_FULL)) return false;
            tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < D; c += 32, ++kk) {
                uint32_t v[32];
                tmem_ld32(lt + C::DQ_COL + c, v);
                tmem_wait_ld();
                reg_fence32(v);
                if (c + 32 >= D) {
                    tc_fence_before();
                    mbar_arrive(smem_u32(&bar_dq_free));
                }
                if (kk > 0) {
                    if (r == 0) {
                        bulk_wait_group_read0();
                        mbar_arrive(smem_u32(&bar_dqs_free));
                    }
                    if (!mbar_wait_warp(smem_u32(&bar_dqs_free), (kk - 1) & 1, w, SITE_BWD_DQ_FREE)) return false;
                }
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    *reinterpret_cast<uint4*>(sDQ + sw128_offset(r, u)) =
                        make_uint4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
                fence_proxy_async_smem();
                mbar_arrive(smem_u32(&bar_dqs_full));
                bool issued = true;
                if (r == 0) {
                    issued = mbar_wait(smem_u32(&bar_dqs_full), kk & 1, w, SITE_BWD_DQ_FULL);
                    if (issued) {
                        // Rows at or beyond T lie outside the tensor map and are skipped.
                        tma_reduce_add_4d(&tm_dq, smem_u32(sDQ), c, h, q0, b);
                        bulk_commit_group();
                    }
                }
                if (!__all_sync(0xffffffffu, issued)) return false;
            }
            return true;
        };
        bool ok = mbar_wait_warp(smem_u32(&bar_kv_full), 0, w, SITE_BWD_KV);
        if (ok) {
            ovf |= rope_tile_smem<D, C::BKV, 128, ROPE_BF16_F16>(sK, sK16, kv0, T, r, a.rope,
                                                                 VL ? len : kv0 + C::BKV);
            fence_proxy_async_smem();
            mbar_arrive(smem_u32(&bar_k_ready));
        }
        for (int it = 0; ok && it <= n_it; ++it) {
            if (it < n_it) {
                const int s = it % C::NQS;
                const int q0 = (i_first + it % per_head) * C::BQ;
                if (!(ok = mbar_wait_warp(smem_u32(&bar_qdo_full[s]), (it / C::NQS) & 1, w, SITE_BWD_QDO_FULL))) break;
                // With dS^T living in the fp16 Q' buffer, the previous step's dK/dQ MMAs
                // must be done with it before it is overwritten.
                if (C::DS_ALIASES_Q16 && it > 0 &&
                    !(ok = mbar_wait_warp(smem_u32(&bar_ds_free), (it - 1) & 1, w, SITE_BWD_DS_FREE)))
                    break;
                ovf |= rope_tile_smem<D, C::BQ, 128, ROPE_BF16_F16>(stage_q(s), stage_q16(s), q0, T, r, a.rope,
                                                                    VL ? len : q0 + C::BQ);
                fence_proxy_async_smem();
                mbar_arrive(smem_u32(&bar_q_ready[s]));
            }
            if (it > 0 && !(ok = drain(it - 1))) break;
        }
        if (r == 0) bulk_wait_group0();   // the last reduces have completed before the CTA exits
        if (ovf) report_error(a.err, SITE_RANGE);
    } else {
        // ------------------------------------------------------------ P^T, dS^T; dK, dV epilogue
        // Two groups share every key row: group g (warps 8-11 / 12-15) takes query columns
        // [64g, 64g + 64) of S^T and dP^T, so each SMSP has two such warps to overlap.
        const int g = (warp - 8) >> 2;
        const int r = (warp & 3) * 32 + lane;          // key row = TMEM lane
        const int kvpos = kv0 + r;
        const int cbase = 64 * g;
        const uint32_t lt = tm + ((uint32_t)((warp & 3) * 32) << 16);
        const float sl2 = a.scale_log2;
        bool ok = true;
        // LSE/Delta of step it sit in s_lse/s_delta[it & 1]; the rows of step it+1 are
        // fetched while step it runs and published at its end.  A buffer is rewritten only
        // after every thread has passed the step that read it (bar_rows of the next step).
        auto row_vals = [&](int it, float& lv, float& dv) {
            const int h = hkv * G + it / per_head;
            const int qpos = (i_first + it % per_head) * C::BQ + cbase + (r & 63);
            const size_t rix = ((size_t)b * a.Hq + h) * T + qpos;
            lv = qpos < len ? a.lse[rix] * 1.4426950408889634f : 0.f;
            dv = qpos < len ? a.delta[rix] : 0.f;
        };
        auto publish = [&](int it, float lv, float dv) {
            if (r < 64) {                         // negated: added by packed FMA / add
                s_lse[it & 1][cbase + r] = -lv;
                s_delta[it & 1][cbase + r] = -dv;
            }
            mbar_arrive(smem_u32(&bar_rows[it & 1]));
        };
        {
            float lv, dv;
            if (r < 64 && n_it > 0) row_vals(0, lv, dv);
            publish(0, lv, dv);
        }
        for (int it = 0; it < n_it; ++it) {
            const int q0 = (i_first + it % per_head) * C::BQ;
            const int sb = it & 1;
            uint8_t* dsb = C::DS_ALIASES_Q16 ? stage_q16(it % C::NQS) : sdS;
            if (!mbar_wait_warp(smem_u32(&bar_rows[sb]), (it >> 1) & 1, w, SITE_BWD_S_FULL)) { ok = false; break; }
            float lv_n = 0.f, dv_n = 0.f;
            if (it + 1 < n_it && r < 64) row_vals(it + 1, lv_n, dv_n);    // in flight during this step
            // Per-element masks: the causal diagonal, and queries past the length (padding).
            const bool diag = kv0 + C::BKV - 1 > q0 || (VL && q0 + C::BQ > len);
            if (!mbar_wait_warp(smem_u32(&bar_s_full), it & 1, w, SITE_BWD_S_FULL)) { ok = false; break; }
            if (!mbar_wait_warp(smem_u32(&bar_dp_full), it & 1, w, SITE_BWD_DP_FULL)) { ok = false; break; }
            if (it > 0 && !mbar_wait_warp(smem_u32(&bar_ds_free), (it - 1) & 1, w, SITE_BWD_DS_FREE)) { ok = false; break; }
            tc_fence_after();
            // P^T goes to its own columns: dV of the previous step must have read them.
            if (C::PT_OWN && it > 0 && !mbar_wait_warp(smem_u32(&bar_p_free), (it - 1) & 1, w, SITE_BWD_DS_READY)) {
                ok = false;
                break;
            }
            // Four 16-query chunks; the TMEM loads of chunk c+1 are in flight while chunk c
            // is computed.  Once the last chunk is in registers the MMA issuer may overwrite
            // S^T and dP^T with the next step's.
            auto chunk = [&](int c, uint32_t (&sr)[16], uint32_t (&dr)[16]) {
                uint32_t pk[8], dk[8];
                const float4* l4 = reinterpret_cast<const float4*>(&s_lse[sb][cbase + c]);
                const float4* d4 = reinterpret_cast<const float4*>(&s_delta[sb][cbase + c]);
                const float2 sl2v = make_float2(sl2, sl2);
#pragma unroll
                for (int e = 0; e < 16; e += 4) {
                    // -LSE log2(e) and -Delta (negated when staged): the exponent argument,
                    // dP - Delta and P (dP - Delta) run as packed f32x2 pairs of queries.
                    const float4 lv = l4[e >> 2], dv = d4[e >> 2];   // broadcast reads
                    const float2 x01 = __ffma2_rn(make_float2(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])),
                                                  sl2v, make_float2(lv.x, lv.y));
                    const float2 x23 = __ffma2_rn(make_float2(__uint_as_float(sr[e + 2]), __uint_as_float(sr[e + 3])),
                                                  sl2v, make_float2(lv.z, lv.w));
                    float p[4] = {ex2(x01.x), ex2(x01.y), ex2(x23.x), ex2(x23.y)};
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        if (diag && (kvpos > q0 + cbase + c + e + k || (VL && q0 + cbase + c + e + k >= len))) p[k] = 0.f;
                    const float2 g01 = __fmul2_rn(make_float2(p[0], p[1]),
                                                  __fadd2_rn(make_float2(__uint_as_float(dr[e]), __uint_as_float(dr[e + 1])),
                                                             make_float2(dv.x, dv.y)));
                    const float2 g23 = __fmul2_rn(make_float2(p[2], p[3]),
                                                  __fadd2_rn(make_float2(__uint_as_float(dr[e + 2]), __uint_as_float(dr[e + 3])),
                                                             make_float2(dv.z, dv.w)));
                    const float gg[4] = {g01.x, g01.y, g23.x, g23.y};
                    pk[e >> 1] = pack_bf162(p[0], p[1]);
                    pk[(e >> 1) + 1] = pack_bf162(p[2], p[3]);
                    dk[e >> 1] = pack_bf162(gg[0], gg[1]);
                    dk[(e >> 1) + 1] = pack_bf162(gg[2], gg[3]);
                }
                tmem_st8(lt + C::pt_col(cbase + c), pk);
                uint8_t* base = dsb + g * C::BKV * 128;
                const int u0 = c >> 3;
                *reinterpret_cast<uint4*>(base + sw128_offset(r, u0)) = make_uint4(dk[0], dk[1], dk[2], dk[3]);
                *reinterpret_cast<uint4*>(base + sw128_offset(r, u0 + 1)) = make_uint4(dk[4], dk[5], dk[6], dk[7]);
            };
            uint32_t sa[16], da[16], sb2[16], db2[16];
            const uint32_t scol = lt + C::S_COL + cbase, dcol = lt + C::DP_COL + cbase;
            tmem_ld16(scol, sa);
            tmem_ld16(dcol, da);
            tmem_wait_ld16(sa);
            tmem_wait_ld16(da);
            tmem_ld16(scol + 16, sb2);
            tmem_ld16(dcol + 16, db2);
            chunk(0, sa, da);
            tmem_wait_ld16(sb2);
            tmem_wait_ld16(db2);
            tmem_ld16(scol + 32, sa);
            tmem_ld16(dcol + 32, da);
            chunk(16, sb2, db2);
            tmem_wait_ld16(sa);
            tmem_wait_ld16(da);
            tmem_ld16(scol + 48, sb2);
            tmem_ld16(dcol + 48, db2);
            chunk(32, sa, da);
            tmem_wait_ld16(sb2);
            tmem_wait_ld16(db2);
            if constexpr (C::PT_OWN) {
                tc_fence_before();
                mbar_arrive(smem_u32(&bar_sdp_read));
            }
            chunk(48, sb2, db2);
            fence_proxy_async_smem();
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(smem_u32(&bar_ds_ready));
            if (it + 1 < n_it) publish(it + 1, lv_n, dv_n);
        }
        // Epilogue, key row r of this CTA's tile: group 0 writes dK = s R^T dK', group 1 dV.
        if (ok && mbar_wait_warp(smem_u32(&bar_dkv_full), 0, w, SITE_BWD_DKV)) {
            tc_fence_after();
            const bool valid = kvpos < T;
            // Keys past the sequence's length (or a tile with no query tile) get zeros.
            const bool live = !VL || (kvpos < len && n_it > 0);
            const size_t orow = (((size_t)b * T + (valid ? kvpos : 0)) * a.Hkv + hkv) * D;
#pragma unroll 1
            for (int c = 0; c < D; c += 32) {
                uint32_t x[32];
                tmem_ld32(lt + (g == 0 ? C::DK_COL : C::DV_COL) + c, x);
                tmem_wait_ld();
                reg_fence32(x);
                if (!valid) continue;
                if (!live) {
#pragma unroll
                    for (int e = 0; e < 32; ++e) x[e] = 0u;
                }
                uint32_t pk[16];
                if (g == 0) {
                    const float4* tab = reinterpret_cast<const float4*>(a.rope + (size_t)kvpos * (D / 2) + c / 2);
#pragma unroll
                    for (int e = 0; e < 32; e += 4) {
                        const float4 cs = __ldg(tab + e / 4);
                        const float g0 = __uint_as_float(x[e]) * a.scale, g1 = __uint_as_float(x[e + 1]) * a.scale;
                        const float g2 = __uint_as_float(x[e + 2]) * a.scale, g3 = __uint_as_float(x[e + 3]) * a.scale;
                        // R^T: the rotation by -angle.
                        pk[e >> 1] = pack_bf162(rot0(g0, g1, cs.x, -cs.y), rot1(g0, g1, cs.x, -cs.y));
                        pk[(e >> 1) + 1] = pack_bf162(rot0(g2, g3, cs.z, -cs.w), rot1(g2, g3, cs.z, -cs.w));
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 32; e += 2) pk[e >> 1] = pack_bf162(__uint_as_float(x[e]), __uint_as_float(x[e + 1]));
                }
                uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(g == 0 ? a.dk : a.dv) + orow + c);
#pragma unroll
                for (int e = 0; e < 4; ++e) dst[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
            }
        }
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        mbar_wait_drain(smem_u32(&bar_final), 0, w, SITE_BWD_DRAIN);
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tm, 512);
    }
}

template <int D, bool VL>
cudaError_t launch_bwd_vl(int B, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const CUtensorMap& tdo, const CUtensorMap& tdq, const BwdArgs& a, cudaStream_t st) {
    using C = BwdCfg<D>;
    auto kfn = attn_bwd_kernel<D, VL>;
    cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    dim3 grid(a.Hkv, B, a.n_kvt);
    return launch_k(kfn, grid, dim3(C::THREADS), C::SMEM, st, tq, tk, tv, tdo, tdq, a);
}

template <int D>
cudaError_t launch_bwd_t(int B, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const CUtensorMap& tdo, const CUtensorMap& tdq, const BwdArgs& a, cudaStream_t st) {
    return a.seq_lens ? launch_bwd_vl<D, true>(B, tq, tk, tv, tdo, tdq, a, st)
                      : launch_bwd_vl<D, false>(B, tq, tk, tv, tdo, tdq, a, st);
}

int grid_for(long long work, int per_block) {
    long long blocks = (work + per_block - 1) / per_block;
    if (blocks > 152 * 8) blocks = 152 * 8;
    return (int)(blocks < 1 ? 1 : blocks);
}

}  // namespace

template <bool VL>
cudaError_t launch_bwd_pre_vl(bool tf32, const BwdPreArgs& a, cudaStream_t st) {
    const dim3 g(grid_for(a.rows * 8, 256)), blk(256);
    if (!tf32 && !a.q16 && !a.dq_acc) {          // after the training forward (bf16, D <= 64)
        if (a.D == 32) return launch_k(bwd_pre_kernel<__nv_bfloat16, 32, VL, true>, g, blk, 0, st, a);
        if (a.D == 64) return launch_k(bwd_pre_kernel<__nv_bfloat16, 64, VL, true>, g, blk, 0, st, a);
    }
    if (!tf32) {
        if (a.D == 32) return launch_k(bwd_pre_kernel<__nv_bfloat16, 32, VL>, g, blk, 0, st, a);
        if (a.D == 64) return launch_k(bwd_pre_kernel<__nv_bfloat16, 64, VL>, g, blk, 0, st, a);
        if (a.D == 128) return launch_k(bwd_pre_kernel<__nv_bfloat16, 128, VL>, g, blk, 0, st, a);
    } else {
        if (a.D == 32) return launch_k(bwd_pre_kernel<float, 32, VL>, g, blk, 0, st, a);
        if (a.D == 64) return launch_k(bwd_pre_kernel<float, 64, VL>, g, blk, 0, st, a);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_bwd_pre(bool tf32, const BwdPreArgs& a, cudaStream_t st) {
    if (a.rows == 0) return cudaSuccess;
    return a.seq_lens ? launch_bwd_pre_vl<true>(tf32, a, st) : launch_bwd_pre_vl<false>(tf32, a, st);
}

cudaError_t launch_bwd_post(bool tf32, const BwdPostArgs& a, cudaStream_t st) {
    if (a.rows == 0) return cudaSuccess;
    const dim3 g(grid_for(a.rows * (a.D / 8), 256)), blk(256);
    if (!tf32) {
        if (a.D == 32) return launch_k(bwd_post_kernel<__nv_bfloat16, 32>, g, blk, 0, st, a);
        if (a.D == 64) return launch_k(bwd_post_kernel<__nv_bfloat16, 64>, g, blk, 0, st, a);
        if (a.D == 128) return launch_k(bwd_post_kernel<__nv_bfloat16, 128>, g, blk, 0, st, a);
    } else {
        if (a.D == 32) return launch_k(bwd_post_kernel<float, 32>, g, blk, 0, st, a);
        if (a.D == 64) return launch_k(bwd_post_kernel<float, 64>, g, blk, 0, st, a);
    }
    return cudaErrorInvalidValue;
}

int bwd_q_box_rows(bool tf32, int D) {
    if (tf32) return bwd_tf32_q_box_rows();
    return D <= 64 ? bwd_d64_q_box_rows() : BwdCfg<128>::BQ;
}

cudaError_t launch_bwd(bool tf32, int D, int B, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdq, const BwdArgs& a,
                       cudaStream_t st) {
    if (tf32) return cudaErrorNotSupported;
    if (D == 64 || D == 32) return launch_bwd_d64(B, tq, tk, tv, tdo, tdq, a, st);   // 32: zero-padded to 64
    if (D == 128) return launch_bwd_t<128>(B, tq, tk, tv, tdo, tdq, a, st);
    return cudaErrorInvalidValue;
}

}  // namespace ne
