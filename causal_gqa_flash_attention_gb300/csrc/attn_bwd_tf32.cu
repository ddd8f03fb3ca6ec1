// attn_bwd_tf32.cu -- backward of causal GQA + RoPE attention for fp32 tensors on TF32
// tensor cores (the hand-written backward of "NanoEuler: C와 CUDA로 밑바닥부터 구축한
// GPT-2 규모의 LLM", 검증 및 안정성, for the attention of its 기술 사양 and 커널 구현).
//
// Same mathematics as the bf16 backward (attn_bwd.cu); the layout differs because TF32
// UMMAs only read K-major operands.  One CTA per (batch, kv head, 128-key tile) loops
// over the G query heads and every 64-query tile at or after the diagonal:
//   S^T  = K' Q'^T           M=128 keys, N=64 queries     A = K', B = Q'
//   dP^T = V dO^T            M=128, N=64                  A = V,  B = dO
//   P^T, dS^T (fp32, TF32-rounded) written back to TMEM over S^T and dP^T (two TMEM
//   buffers, by step parity); dS also to shared memory as [query][key] (the K-major A
//   of the dQ product)
//   dV  += P^T dO            A = P^T (TMEM), B = dO^T     (dO transposed in smem)
//   dK' += dS^T Q'           A = dS^T (TMEM), B = Q'^T    (Q' transposed in smem)
//   dQ'_part = dS K'         M=64 queries, N=D, K=128 keys; A = dS, B = K'^T
// The M=64 accumulator puts query row m in TMEM lane 32*(m/16) + m%16.
// Warp roles (384 threads): warp 0 TMA; warp 1 TMEM allocator and UMMA issuer (all
// products, in order, so every TMEM and smem reuse is ordered by the one issuer);
// warps 4-7 RoPE on K and Q', TF32 rounding of V and dO, the transposes, then the dQ
// drain; warps 8-11 P^T, dS^T and dS (thread = key row) and the dK/dV epilogue.  (Warps
// 2-3 taking dO's rounding and transpose measured slower: the roles share the shared-
// memory bandwidth with the SS products, and the gradient warps slowed by more than the
// transposes gained.)
// Two Q' | dO stages (one for Q'^T | dO^T) and two S^T | dP^T buffers in TMEM: step
// it's tiles load into stage it % 2 once step it - 2 is done with it and are rotated and
// rounded in place while step it - 1 runs; S^T and dP^T of step it + 1 (whose operands
// need no transpose) are issued as soon as its tiles are rotated, before the dV, dK and
// dQ products of step it, so the gradient warps go from one step to the next without
// waiting for those.  The transposes wait only for the dK product of the step before
// (the last reader of Q'^T and dO^T), and the gradient warps write dS to shared memory
// only after the previous step's dQ product has read it.  (With one stage and one
// buffer, each step began with the load, rotation and transposes of its tiles after
// every product of the step before had completed: 273 us against 221.5 with two
// stages at B16 T512.)
#include "kernels.h"
#include "ptx.cuh"
#include "rope_smem.cuh"

namespace ne {

namespace {

template <int D>
struct BwdTf32Cfg {
    static constexpr int BKV = 128, BQ = 64;
    static constexpr int ROWB = D * 4;
    static constexpr int NCH = ROWB / 128;            // 128-byte chunks per row
    static constexpr int KV_BYTES = BKV * ROWB;       // K', V, K'^T
    static constexpr int Q_BYTES = BQ * ROWB;         // Q', Q'^T, dO, dO^T
    static constexpr int STAGE_BYTES = 2 * Q_BYTES;   // one Q' | dO stage (two stages)
    static constexpr int DS_BYTES = BQ * BKV * 4;     // dS [query][key]
    static constexpr int SMEM = 1024 + 3 * KV_BYTES + 2 * STAGE_BYTES + 2 * Q_BYTES + DS_BYTES;
    // S^T / P^T of buffer b at 128 b, dP^T / dS^T at 128 b + 64; dV, dK', dQ' after both.
    static constexpr int DV_COL = 256, DK_COL = 256 + D, DQ_COL = 256 + 2 * D;
    static constexpr int TMEM_COLS = 512;
    static_assert(DQ_COL + D <= TMEM_COLS, "TMEM columns");
    static __device__ __forceinline__ uint32_t s_col(int it) { return (uint32_t)((it & 1) * 128); }
    static __device__ __forceinline__ uint32_t dp_col(int it) { return (uint32_t)((it & 1) * 128 + 64); }
    static_assert(SMEM <= 227 * 1024, "shared memory");
};

// dst[d][r] = src[r][d] for a fp32 tile of ROWS rows x D columns in the 128-byte
// swizzled layout (both K-major, 32 elements per 128-byte chunk); NT threads.
template <int D, int ROWS, int NT = 128>
__device__ __forceinline__ void transpose_f32(const uint8_t* src, uint8_t* dst, int t) {
    constexpr int UNITS = D * ROWS / 4;
    // A warp takes 32 consecutive columns d of the same four rows: conflict-free reads
    // (one row, every bank once under the 128-byte swizzle) and writes (eight rows d per
    // quarter-warp at swizzle-spread chunk positions).  Rows fastest put a warp's reads
    // on two or four banks.
#pragma unroll 4
    for (int ul = t; ul < UNITS; ul += NT) {
        const int d = ul % D, r0 = 4 * (ul / D);
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
            w[k] = *reinterpret_cast<const uint32_t*>(src + (d >> 5) * ROWS * 128 + sw128_offset(r0 + k, (d & 31) >> 2) +
                                                      (d & 3) * 4);
        *reinterpret_cast<uint4*>(dst + (r0 >> 5) * D * 128 + sw128_offset(d, (r0 & 31) >> 2)) =
            make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// Round a fp32 tile to TF32 (nearest) in place; NT threads.
template <int BYTES, int NT = 128>
__device__ __forceinline__ void round_tf32(uint8_t* p, int t) {
#pragma unroll 4
    for (int i = t; i < BYTES / 16; i += NT) {
        uint4 v = reinterpret_cast<uint4*>(p)[i];
        v.x = f32_to_tf32_rna(__uint_as_float(v.x));
        v.y = f32_to_tf32_rna(__uint_as_float(v.y));
        v.z = f32_to_tf32_rna(__uint_as_float(v.z));
        v.w = f32_to_tf32_rna(__uint_as_float(v.w));
        reinterpret_cast<uint4*>(p)[i] = v;
    }
}

// VL: per-sequence lengths (padded batch).  Without them every length is T, rows past T
// arrive as TMA's zero fill, and the padding code compiles away.
template <int D, bool VL>
__global__ void __launch_bounds__(384, 1)
    attn_bwd_tf32_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                         const BwdArgs a) {
    using C = BwdTf32Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sK = smem;                       // K' [128][D]
    uint8_t* sKT = sK + C::KV_BYTES;          // K'^T [D][128]
    uint8_t* sV = sKT + C::KV_BYTES;          // V [128][D]
    uint8_t* sStage = sV + C::KV_BYTES;       // stage s: Q' [64][D] | dO [64][D]
    uint8_t* sQT = sStage + 2 * C::STAGE_BYTES;   // Q'^T [D][64]
    uint8_t* sOT = sQT + C::Q_BYTES;          // dO^T [D][64]
    uint8_t* sdS = sOT + C::Q_BYTES;          // dS [64][128]
    auto stage_q = [&](int it) { return sStage + (it & 1) * C::STAGE_BYTES; };
    auto stage_o = [&](int it) { return sStage + (it & 1) * C::STAGE_BYTES + C::Q_BYTES; };

    __shared__ __align__(8) uint64_t bar_kv_full, bar_k_ready, bar_q_rot, bar_q_ready, bar_qt_free, bar_ds_ready,
        bar_dq_full, bar_dq_free, bar_dkv_full, bar_final, bar_aux;
    __shared__ __align__(8) uint64_t bar_stage_full[2], bar_stage_free[2], bar_s_full[2];
    __shared__ __align__(8) uint64_t bar_rows[2];
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
    auto step_h = [&](int it) { return hkv * G + it / per_head; };
    auto step_q0 = [&](int it) { return (i_first + it % per_head) * C::BQ; };

    if (tid == 0) {
        mbar_init(smem_u32(&bar_kv_full), 1);
        mbar_init(smem_u32(&bar_k_ready), 128);
        mbar_init(smem_u32(&bar_stage_full[0]), 1);
        mbar_init(smem_u32(&bar_stage_full[1]), 1);
        // A stage is free once the S^T and dP^T products (a commit) and the transposes
        // (the 128 RoPE threads) have read it.
        mbar_init(smem_u32(&bar_stage_free[0]), 1 + 128);
        mbar_init(smem_u32(&bar_stage_free[1]), 1 + 128);
        mbar_init(smem_u32(&bar_q_rot), 128);
        mbar_init(smem_u32(&bar_q_ready), 128);
        mbar_init(smem_u32(&bar_qt_free), 1);
        mbar_init(smem_u32(&bar_s_full[0]), 1);
        mbar_init(smem_u32(&bar_s_full[1]), 1);
        mbar_init(smem_u32(&bar_ds_ready), 128);
        mbar_init(smem_u32(&bar_dq_full), 1);
        mbar_init(smem_u32(&bar_dq_free), 128);
        mbar_init(smem_u32(&bar_dkv_full), 1);
        mbar_init(smem_u32(&bar_final), 1);
        mbar_init(smem_u32(&bar_aux), 128);        // intra-group sync of the RoPE/transpose warps
        mbar_init(smem_u32(&bar_rows[0]), 128);
        mbar_init(smem_u32(&bar_rows[1]), 128);
        abort_flag = 0;
        fence_mbar_init();
        // The tensor maps are kernel parameters, not outputs of an earlier kernel: fetch
        // them before the dependency wait, under the previous kernel's tail.
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        tma_prefetch_desc(&tm_do);
    }
    if (warp == 1) {
        __syncwarp();
        tmem_alloc(smem_u32(&tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    griddep_launch_dependents();   // after the TMEM allocation
    griddep_wait();                // LSE, Delta and the zeroed accumulator are visible
    const uint32_t tm = tmem_slot;
    const WaitCtx w{a.err, &abort_flag, a.timeout_ns};

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint32_t kvf = smem_u32(&bar_kv_full);
            mbar_arrive_expect_tx(kvf, 2 * C::KV_BYTES);
            for (int c = 0; c < C::NCH; ++c) {
                tma_load_4d(smem_u32(sK + c * C::BKV * 128), &tm_k, kvf, c * 32, hkv, kv0, b);
                tma_load_4d(smem_u32(sV + c * C::BKV * 128), &tm_v, kvf, c * 32, hkv, kv0, b);
            }
            int issued = 0;
            for (int it = 0; it < n_it; ++it) {
                // Stage it % 2 is free once step it - 2 has read it.
                if (it >= 2 && !mbar_wait(smem_u32(&bar_stage_free[it & 1]), ((it >> 1) - 1) & 1, w,
                                          SITE_BWD_QDO_EMPTY))
                    break;
                const uint32_t f = smem_u32(&bar_stage_full[it & 1]);
                mbar_arrive_expect_tx(f, 2 * C::Q_BYTES);
                for (int c = 0; c < C::NCH; ++c) {
                    tma_load_4d(smem_u32(stage_q(it) + c * C::BQ * 128), &tm_q, f, c * 32, step_h(it), step_q0(it), b);
                    tma_load_4d(smem_u32(stage_o(it) + c * C::BQ * 128), &tm_do, f, c * 32, step_h(it), step_q0(it), b);
                }
                ++issued;
            }
            mbar_wait_drain(kvf, 0, w, SITE_BWD_DRAIN);
            // The last load of each stage has landed (earlier ones were waited for by the
            // RoPE warps before the stage was reused).
            for (int it = issued - 2 > 0 ? issued - 2 : 0; it < issued; ++it)
                mbar_wait_drain(smem_u32(&bar_stage_full[it & 1]), (it >> 1) & 1, w, SITE_BWD_DRAIN);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ UMMA issuer (all products)
        // The whole warp runs the loop and its waits, so the UMMA operands stay
        // warp-uniform, and one elected lane issues each batch with its commits (a loop
        // run by lane 0 alone cost several instructions per UMMA, 48 UMMAs a step).
        {
            constexpr uint32_t id_sp = idesc_make(FMT_TF32, 128, C::BQ, false, false);   // S^T, dP^T
            constexpr uint32_t id_vk = idesc_make(FMT_TF32, 128, D, false, false);       // dV, dK
            constexpr uint32_t id_q = idesc_make(FMT_TF32, 64, D, false, false);         // dQ (M = 64)
            const uint64_t dK = sdesc(smem_u32(sK), 16, 1024), dKT = sdesc(smem_u32(sKT), 16, 1024);
            const uint64_t dV = sdesc(smem_u32(sV), 16, 1024), dQ0 = sdesc(smem_u32(stage_q(0)), 16, 1024);
            const uint64_t dQT = sdesc(smem_u32(sQT), 16, 1024), dO0 = sdesc(smem_u32(stage_o(0)), 16, 1024);
            const uint64_t dOT = sdesc(smem_u32(sOT), 16, 1024), dS = sdesc(smem_u32(sdS), 16, 1024);
            // K-step ks covers 8 fp32 = 32 bytes of the K dimension: chunk ks/4, offset (ks%4)*32.
            auto koff = [](int ks, int rows) { return (uint32_t)((ks >> 2) * rows * 128 + (ks & 3) * 32); };
            // S^T and dP^T of step it into TMEM buffer it % 2, once its Q' and dO are
            // rotated and rounded (their buffer's previous products, dV and dK of step
            // it - 2, were issued earlier by this warp and run first).
            auto sdp = [&](int it) -> bool {
                if (!mbar_wait_warp(smem_u32(&bar_q_rot), it & 1, w, SITE_BWD_Q_READY)) return false;
                tc_fence_after();
                const uint64_t dQ = sdesc_add(dQ0, (it & 1) * C::STAGE_BYTES);
                const uint64_t dO = sdesc_add(dO0, (it & 1) * C::STAGE_BYTES);
                const uint32_t sc = tm + C::s_col(it), dc = tm + C::dp_col(it);
                if (elect_one()) {
#pragma unroll
                    for (int ks = 0; ks < D / 8; ++ks)
                        umma_ss<true>(sc, sdesc_add(dK, koff(ks, C::BKV)), sdesc_add(dQ, koff(ks, C::BQ)), id_sp, ks > 0);
#pragma unroll
                    for (int ks = 0; ks < D / 8; ++ks)
                        umma_ss<true>(dc, sdesc_add(dV, koff(ks, C::BKV)), sdesc_add(dO, koff(ks, C::BQ)), id_sp, ks > 0);
                    umma_commit(smem_u32(&bar_s_full[it & 1]));
                    umma_commit(smem_u32(&bar_stage_free[it & 1]));
                }
                __syncwarp();
                return true;
            };
            bool ok = mbar_wait_warp(smem_u32(&bar_k_ready), 0, w, SITE_BWD_KV) && (n_it == 0 || sdp(0));
            for (int it = 0; ok && it < n_it; ++it) {
                if (it + 1 < n_it && !(ok = sdp(it + 1))) break;
                if (!(ok = mbar_wait_warp(smem_u32(&bar_ds_ready), it & 1, w, SITE_BWD_DS_READY))) break;
                if (!(ok = mbar_wait_warp(smem_u32(&bar_q_ready), it & 1, w, SITE_BWD_Q_READY))) break;   // transposes
                tc_fence_after();
                const uint32_t sc = tm + C::s_col(it), dc = tm + C::dp_col(it);
                if (elect_one()) {
#pragma unroll
                    for (int ks = 0; ks < C::BQ / 8; ++ks)   // dV += P^T dO, K = queries
                        umma_ts<true>(tm + C::DV_COL, sc + ks * 8, sdesc_add(dOT, koff(ks, D)), id_vk,
                                      (it > 0 || ks > 0) ? 1u : 0u);
#pragma unroll
                    for (int ks = 0; ks < C::BQ / 8; ++ks)   // dK' += dS^T Q'
                        umma_ts<true>(tm + C::DK_COL, dc + ks * 8, sdesc_add(dQT, koff(ks, D)), id_vk,
                                      (it > 0 || ks > 0) ? 1u : 0u);
                    umma_commit(smem_u32(&bar_qt_free));    // Q'^T and dO^T are read
                }
                __syncwarp();
                if (it > 0 && !(ok = mbar_wait_warp(smem_u32(&bar_dq_free), (it - 1) & 1, w, SITE_BWD_DQ_FREE))) break;
                tc_fence_after();
                if (elect_one()) {
#pragma unroll
                    for (int ks = 0; ks < C::BKV / 8; ++ks)  // dQ'_part = dS K', K = keys
                        umma_ss<true>(tm + C::DQ_COL, sdesc_add(dS, koff(ks, C::BQ)), sdesc_add(dKT, koff(ks, D)), id_q,
                                      ks > 0);
                    umma_commit(smem_u32(&bar_dq_full));
                }
                __syncwarp();
            }
            if (elect_one()) {
                umma_commit(smem_u32(&bar_dkv_full));
                umma_commit(smem_u32(&bar_final));
            }
            __syncwarp();
        }
    } else if (warp >= 4 && warp < 8) {
        // ------------------------------------------------------------ RoPE, rounding, transposes; dQ drain
        const int r = tid - 128;
        const uint32_t lt = tm + ((uint32_t)((warp & 3) * 32) << 16);
        int aux_uses = 0;
        // The transposes read rows rotated or rounded by other threads of the group.
        auto group_sync = [&]() -> bool {
            mbar_arrive(smem_u32(&bar_aux));
            return mbar_wait_warp(smem_u32(&bar_aux), (aux_uses++) & 1, w, SITE_BWD_KV);
        };
        auto drain = [&](int it) -> bool {
            if (!mbar_wait_warp(smem_u32(&bar_dq_full), it & 1, w, SITE_BWD_DQ_FULL)) return false;
            tc_fence_after();
            uint32_t v[D];
            tmem_ld_cols<D / 32>(lt + C::DQ_COL, v);
            tc_fence_before();
            mbar_arrive(smem_u32(&bar_dq_free));
            const int qrow = (warp & 3) * 16 + lane;           // M=64 layout: lanes 0-15 of each quarter
            const int qpos = step_q0(it) + qrow;
            if (lane < 16 && qpos < T) {
                float* dst = a.dq_acc + (((size_t)b * T + qpos) * a.Hq + step_h(it)) * D;
#pragma unroll
                for (int e = 0; e < D; e += 4)
                    atomicAdd(reinterpret_cast<float4*>(dst + e),
                              make_float4(__uint_as_float(v[e]), __uint_as_float(v[e + 1]), __uint_as_float(v[e + 2]),
                                          __uint_as_float(v[e + 3])));
            }
            return true;
        };
        bool ok = mbar_wait_warp(smem_u32(&bar_kv_full), 0, w, SITE_BWD_KV);
        if (ok) {
            rope_tile_smem<D, C::BKV, 128, ROPE_TF32>(sK, nullptr, kv0, T, r, a.rope, VL ? len : kv0 + C::BKV);
            round_tf32<C::KV_BYTES>(sV, r);
            ok = group_sync();
        }
        if (ok) {
            transpose_f32<D, C::BKV>(sK, sKT, r);
            fence_proxy_async_smem();
            mbar_arrive(smem_u32(&bar_k_ready));
        }
        // Rotation of step it's Q' and rounding of its dO in place; the q_rot barrier
        // (every thread of the group) also orders them before the transposes.  The table
        // row of the next step's rotation is fetched right after this one, so its latency
        // overlaps the transposes and the drain.
        using RopeQ = RopeTile<D, C::BQ, 128, ROPE_TF32>;
        RopeQ rq;
        rq.init(r, a.rope);
        float4 qbase[RopeQ::F4];
        if (n_it > 0) rq.load_base(qbase, step_q0(0), T, a.rope);
        auto rotate = [&](int it) -> bool {
            if (!mbar_wait_warp(smem_u32(&bar_stage_full[it & 1]), (it >> 1) & 1, w, SITE_BWD_QDO_FULL)) return false;
            rq.template apply<false>(stage_q(it), nullptr, qbase, (VL ? len : step_q0(it) + C::BQ) - step_q0(it));
            round_tf32<C::Q_BYTES>(stage_o(it), r);
            fence_proxy_async_smem();
            mbar_arrive(smem_u32(&bar_q_rot));
            if (it + 1 < n_it) rq.load_base(qbase, step_q0(it + 1), T, a.rope);
            return true;
        };
        if (ok && n_it > 0) ok = rotate(0);
        for (int it = 0; ok && it < n_it; ++it) {
            if (!(ok = mbar_wait_warp(smem_u32(&bar_q_rot), it & 1, w, SITE_BWD_Q_READY))) break;
            // Q'^T and dO^T of step it - 1 have been read by its dV and dK products.
            if (it > 0 && !(ok = mbar_wait_warp(smem_u32(&bar_qt_free), (it - 1) & 1, w, SITE_BWD_Q_READY))) break;
            transpose_f32<D, C::BQ>(stage_q(it), sQT, r);
            transpose_f32<D, C::BQ>(stage_o(it), sOT, r);
            fence_proxy_async_smem();
            mbar_arrive(smem_u32(&bar_q_ready));
            mbar_arrive(smem_u32(&bar_stage_free[it & 1]));
            // The next rotation completes the next q_rot phase: first the issuer must have
            // passed this one (its S^T and dP^T of step it are done), or on the first step
            // q_rot could run two phases past the issuer's wait.
            if (it + 1 < n_it && !(ok = mbar_wait_warp(smem_u32(&bar_s_full[it & 1]), (it >> 1) & 1, w, SITE_BWD_S_FULL)))
                break;
            if (it + 1 < n_it && !(ok = rotate(it + 1))) break;
            if (it > 0 && !(ok = drain(it - 1))) break;
        }
        if (ok && n_it > 0) drain(n_it - 1);
    } else if (warp >= 8) {
        // ------------------------------------------------------------ P^T, dS^T, dS; dK, dV epilogue
        const int r = tid - 256;                       // key row = TMEM lane
        const int kvpos = kv0 + r;
        const uint32_t lt = tm + ((uint32_t)((warp & 3) * 32) << 16);
        const float sl2 = a.scale_log2;
        bool ok = true;
        auto row_vals = [&](int it, float& lv, float& dv) {
            const int qpos = step_q0(it) + r;
            const size_t rix = ((size_t)b * a.Hq + step_h(it)) * T + qpos;
            lv = qpos < len ? a.lse[rix] * 1.4426950408889634f : 0.f;
            dv = qpos < len ? a.delta[rix] : 0.f;
        };
        auto publish = [&](int it, float lv, float dv) {
            if (r < C::BQ) {
                s_lse[it & 1][r] = -lv;     // negated: added by packed FMA / add
                s_delta[it & 1][r] = -dv;
            }
            mbar_arrive(smem_u32(&bar_rows[it & 1]));
        };
        {
            float lv = 0.f, dv = 0.f;
            if (r < C::BQ && n_it > 0) row_vals(0, lv, dv);
            publish(0, lv, dv);
        }
        for (int it = 0; it < n_it; ++it) {
            const int q0 = step_q0(it);
            const int sb = it & 1;
            if (!mbar_wait_warp(smem_u32(&bar_rows[sb]), (it >> 1) & 1, w, SITE_BWD_S_FULL)) { ok = false; break; }
            float lv_n = 0.f, dv_n = 0.f;
            if (it + 1 < n_it && r < C::BQ) row_vals(it + 1, lv_n, dv_n);
            if (!mbar_wait_warp(smem_u32(&bar_s_full[it & 1]), (it >> 1) & 1, w, SITE_BWD_S_FULL)) { ok = false; break; }
            tc_fence_after();
            uint32_t sr[64], dr[64];
            tmem_ld_cols<2>(lt + C::s_col(it), sr);
            tmem_ld_cols<2>(lt + C::dp_col(it), dr);
            const bool diag = kv0 + C::BKV - 1 > q0;
            const bool tail = VL && q0 + C::BQ > len;          // queries past the length are padding
#pragma unroll
            for (int c0 = 0; c0 < 64; c0 += 4) {
                // Four queries' -LSE log2(e) and -Delta per 16-byte read; the exponent
                // argument, dP - Delta and the product run as packed f32x2 pairs of queries.
                const float4 l4 = *reinterpret_cast<const float4*>(&s_lse[sb][c0]);
                const float4 d4 = *reinterpret_cast<const float4*>(&s_delta[sb][c0]);
                const float2 nl[2] = {make_float2(l4.x, l4.y), make_float2(l4.z, l4.w)};
                const float2 nd[2] = {make_float2(d4.x, d4.y), make_float2(d4.z, d4.w)};
#pragma unroll
                for (int e = 0; e < 4; e += 2) {
                    const int c = c0 + e;
                    const float2 x = __ffma2_rn(make_float2(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])),
                                                make_float2(sl2, sl2), nl[e >> 1]);
                    float p0 = ex2(x.x), p1 = ex2(x.y);
                    if ((diag && kvpos > q0 + c) || (tail && q0 + c >= len)) p0 = 0.f;
                    if ((diag && kvpos > q0 + c + 1) || (tail && q0 + c + 1 >= len)) p1 = 0.f;
                    const float2 g = __fmul2_rn(make_float2(p0, p1),
                                                __fadd2_rn(make_float2(__uint_as_float(dr[c]), __uint_as_float(dr[c + 1])),
                                                           nd[e >> 1]));
                    sr[c] = f32_to_tf32_rna(p0);
                    sr[c + 1] = f32_to_tf32_rna(p1);
                    dr[c] = f32_to_tf32_rna(g.x);
                    dr[c + 1] = f32_to_tf32_rna(g.y);
                }
            }
            tmem_st32(lt + C::s_col(it), *reinterpret_cast<uint32_t(*)[32]>(sr));
            tmem_st32(lt + C::s_col(it) + 32, *reinterpret_cast<uint32_t(*)[32]>(sr + 32));
            tmem_st32(lt + C::dp_col(it), *reinterpret_cast<uint32_t(*)[32]>(dr));
            tmem_st32(lt + C::dp_col(it) + 32, *reinterpret_cast<uint32_t(*)[32]>(dr + 32));
            // dS to shared memory once the dQ product of step it - 1 has read the buffer.
            if (it > 0 && !mbar_wait_warp(smem_u32(&bar_dq_full), (it - 1) & 1, w, SITE_BWD_DQ_FULL)) { ok = false; break; }
#pragma unroll
            for (int c = 0; c < 64; ++c)   // dS [query c][key r]: key chunk r/32, 4-byte element (r%32) of row c
                *reinterpret_cast<uint32_t*>(sdS + (r >> 5) * C::BQ * 128 + sw128_offset(c, (r & 31) >> 2) + (r & 3) * 4) =
                    dr[c];
            fence_proxy_async_smem();
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(smem_u32(&bar_ds_ready));
            if (it + 1 < n_it) publish(it + 1, lv_n, dv_n);
        }
        // dK = s R^T dK', dV (fp32): key row r of this CTA's tile
        if (ok && mbar_wait_warp(smem_u32(&bar_dkv_full), 0, w, SITE_BWD_DKV)) {
            tc_fence_after();
            const bool valid = kvpos < T;
            // Keys past the sequence's length (or a tile with no query tile) get zeros.
            const bool live = !VL || (kvpos < len && n_it > 0);
            const size_t orow = (((size_t)b * T + (valid ? kvpos : 0)) * a.Hkv + hkv) * D;
#pragma unroll 1
            for (int c = 0; c < D; c += 32) {
                uint32_t kr[32], vr[32];
                tmem_ld32(lt + C::DK_COL + c, kr);
                tmem_ld32(lt + C::DV_COL + c, vr);
                tmem_wait_ld();
                reg_fence32(kr);
                reg_fence32(vr);
                if (!valid) continue;
                if (!live) {
#pragma unroll
                    for (int e = 0; e < 32; ++e) kr[e] = vr[e] = 0u;
                }
                const float4* tab = reinterpret_cast<const float4*>(a.rope + (size_t)kvpos * (D / 2) + c / 2);
                float4* dkp = reinterpret_cast<float4*>(static_cast<float*>(a.dk) + orow + c);
                float4* dvp = reinterpret_cast<float4*>(static_cast<float*>(a.dv) + orow + c);
#pragma unroll
                for (int e = 0; e < 32; e += 4) {
                    const float4 cs = __ldg(tab + e / 4);
                    const float g0 = __uint_as_float(kr[e]) * a.scale, g1 = __uint_as_float(kr[e + 1]) * a.scale;
                    const float g2 = __uint_as_float(kr[e + 2]) * a.scale, g3 = __uint_as_float(kr[e + 3]) * a.scale;
                    dkp[e / 4] = make_float4(rot0(g0, g1, cs.x, -cs.y), rot1(g0, g1, cs.x, -cs.y),   // R^T
                                             rot0(g2, g3, cs.z, -cs.w), rot1(g2, g3, cs.z, -cs.w));
                    dvp[e / 4] = make_float4(__uint_as_float(vr[e]), __uint_as_float(vr[e + 1]),
                                             __uint_as_float(vr[e + 2]), __uint_as_float(vr[e + 3]));
                }
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
        tmem_dealloc(tm, C::TMEM_COLS);
    }
}

template <int D>
cudaError_t launch_t(int B, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                     const CUtensorMap& tdo, const BwdArgs& a, cudaStream_t st) {
    using C = BwdTf32Cfg<D>;
    auto kfn = a.seq_lens ? attn_bwd_tf32_kernel<D, true> : attn_bwd_tf32_kernel<D, false>;
    cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    dim3 grid(a.Hkv, B, a.n_kvt);
    return launch_k(kfn, grid, dim3(384), C::SMEM, st, tq, tk, tv, tdo, a);
}

}  // namespace

int bwd_tf32_q_box_rows() { return BwdTf32Cfg<64>::BQ; }

cudaError_t launch_bwd_tf32(int D, int B, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const BwdArgs& a, cudaStream_t st) {
    if (D == 32) return launch_t<32>(B, tq, tk, tv, tdo, a, st);
    if (D == 64) return launch_t<64>(B, tq, tk, tv, tdo, a, st);
    return cudaErrorInvalidValue;
}

}  // namespace ne
