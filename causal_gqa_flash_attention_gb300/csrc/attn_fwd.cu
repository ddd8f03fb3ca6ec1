// attn_fwd.cu -- forward of causal GQA + RoPE attention on tcgen05 tensor cores.
//
// Method: FlashAttention tiling with an online softmax, so the T x T score matrix is
// never stored ("NanoEuler: C와 CUDA로 밑바닥부터 구축한 GPT-2 규모의 LLM", 커널 구현);
// RoPE on queries and keys and grouped-query heads (same page, 기술 사양); causal mask
// j <= i ("Tiny hackable CUDA language model implementation", Core Mechanics).
//
// One CTA owns two consecutive 128-row query subtiles (u = 0, 1) of one (batch, query
// head) and walks the key/value tiles up to the diagonal; every K/V tile is loaded and
// rotated once for both subtiles.  Warp roles (384 threads, one CTA per SM):
//   warp 0       TMA producer: Q0, Q1 once, then K/V tiles into an NS-stage ring.
//   warp 1       TMEM allocator (512 columns) and UMMA issuer.  Order per tile j:
//                PV0(j), S0(j+1), PV1(j), S1(j+1), so each softmax group works on one
//                subtile while the tensor core runs the other's MMAs.
//   warps 2-3    RoPE on every K tile in place (fp16 logit operand; TF32: rounded fp32)
//                and, for TF32, V transposed (TF32 UMMA reads K-major operands only).
//   warps 4-7    softmax of subtile 0; warps 8-11 softmax of subtile 1.  Thread r owns
//                query row r (TMEM lane r): it rotates its Q row block once, then per
//                tile reads the S row from TMEM, updates the running max m and sum l,
//                writes P (bf16, or TF32 fp32) back over S, rescales its O row when m
//                grew by more than 2^8, and at the end writes O / l (staged in shared
//                memory, stored by TMA) and LSE.
// TMEM: S0 [0,128), S1 [128,256), O0 [256,256+D), O1 [256+D,256+2D).
// Every wait is bounded (WaitCtx); a CTA that gives up records an error code, drains
// its own copies and MMAs, frees its TMEM and exits.
#include <cuda_bf16.h>
#include "kernels.h"
#include "ptx.cuh"
#include "rope_smem.cuh"

namespace ne {

namespace {

#define kNegInf (-__int_as_float(0x7f800000))

template <bool TF32, int D>
struct FwdCfg {
    static constexpr int ES = TF32 ? 4 : 2;            // element bytes
    static constexpr int BM = 128;                     // query rows per subtile
    static constexpr int ROWB = D * ES;                // bytes per row
    static constexpr int BN = (TF32 && D == 64) ? 64 : 128;  // key rows per tile
    static constexpr int NCH = ROWB / 128;             // 128-byte chunks per row
    static constexpr int EPC = 128 / ES;               // elements per chunk
    static constexpr int Q_BYTES = BM * ROWB;          // one subtile
    static constexpr int KV_BYTES = BN * ROWB;
    static constexpr int VT_BYTES = TF32 ? BN * ROWB : 0;
    static constexpr int STAGE_BYTES = 2 * KV_BYTES + VT_BYTES;
    static constexpr int NS = (2 * Q_BYTES + 3 * STAGE_BYTES <= 200 * 1024) ? 3 : 2;
    static constexpr int SMEM = 1024 + 2 * Q_BYTES + NS * STAGE_BYTES;
    static constexpr int O_COL = 256;
    static constexpr int S_KSTEPS = ROWB / 32;         // 32-byte K-steps of S = Q K^T
    static constexpr int PV_KSTEPS = BN * ES / 32;     // K-steps of O += P V
    static constexpr int PV_ROWS = 32 / ES;            // key rows per PV K-step
    static constexpr uint32_t FMT_S = TF32 ? FMT_TF32 : FMT_F16;
    static constexpr uint32_t FMT_PV = TF32 ? FMT_TF32 : FMT_BF16;
    static constexpr int MODE = TF32 ? ROPE_TF32 : ROPE_F16;
    static constexpr int THREADS = 384;
    static_assert(ROWB % 128 == 0, "rows must be whole 128-byte chunks");
    static_assert(D <= 128, "two O subtiles must fit next to two S tiles in 512 TMEM columns");
    static_assert(SMEM <= 227 * 1024, "shared memory");
};

// TF32 only: Vt[d][r] = tf32(V[r][d]) for a [ROWS x D] fp32 tile, written K-major (key
// index contiguous, 32 keys per 128-byte chunk); NT threads.
template <int D, int ROWS, int NT>
__device__ __forceinline__ void transpose_v_tf32(const uint8_t* src, uint8_t* dst, int t) {
    constexpr int UNITS = D * ROWS / 4;       // 16-byte units of the transposed tile
    constexpr int UPR = ROWS / 4;             // units per transposed row
#pragma unroll 4
    for (int ul = t; ul < UNITS; ul += NT) {
        const int d = ul / UPR, u = ul % UPR;  // transposed row d, keys 4u .. 4u+3
        const int r0 = 4 * u;
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint8_t* s = src + (d >> 5) * ROWS * 128 + sw128_offset(r0 + k, (d & 31) >> 2) + (d & 3) * 4;
            w[k] = f32_to_tf32_rna(*reinterpret_cast<const float*>(s));
        }
        *reinterpret_cast<uint4*>(dst + (r0 >> 5) * D * 128 + sw128_offset(d, (r0 & 31) >> 2)) =
            make_uint4(w[0], w[1], w[2], w[3]);
    }
}

template <bool TF32, int D>
__global__ void __launch_bounds__(384, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                    const FwdArgs a) {
    using C = FwdCfg<TF32, D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem;                               // Q0 | Q1 (later: O staging)
    uint8_t* sStage = sQ + 2 * C::Q_BYTES;            // NS x (K | V | Vt)

    __shared__ __align__(8) uint64_t bar_q_full, bar_final;
    __shared__ __align__(8) uint64_t bar_q_ready[2], bar_s_full[2], bar_p_ready[2], bar_o_done[2], bar_o_staged[2];
    __shared__ __align__(8) uint64_t bar_kv_full[C::NS], bar_k_ready[C::NS], bar_kv_empty[C::NS];
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = blockIdx.x, b = blockIdx.y;
    const int pair = a.n_qt - 1 - (int)blockIdx.z;    // heaviest query tiles launch first
    const int hkv = h / a.G;
    const int T = a.T;
    const int q0 = pair * 2 * C::BM;
    int n_u[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const int qu = q0 + u * C::BM;
        n_u[u] = qu < T ? min(qu + C::BM - 1, T - 1) / C::BN + 1 : 0;
    }
    const int n_kv = max(n_u[0], n_u[1]);
    const int n_qsub = n_u[1] > 0 ? 2 : 1;

    if (tid == 0) {
        mbar_init(smem_u32(&bar_q_full), 1);
        mbar_init(smem_u32(&bar_final), 1);
        for (int u = 0; u < 2; ++u) {
            mbar_init(smem_u32(&bar_q_ready[u]), 128);
            mbar_init(smem_u32(&bar_s_full[u]), 1);
            mbar_init(smem_u32(&bar_p_ready[u]), 128);
            mbar_init(smem_u32(&bar_o_done[u]), 1);
            mbar_init(smem_u32(&bar_o_staged[u]), 128);
        }
        for (int s = 0; s < C::NS; ++s) {
            mbar_init(smem_u32(&bar_kv_full[s]), 1);
            mbar_init(smem_u32(&bar_k_ready[s]), 64);
            mbar_init(smem_u32(&bar_kv_empty[s]), 1);
        }
        abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        __syncwarp();
        tmem_alloc(smem_u32(&tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = tmem_slot;
    const WaitCtx w{a.err, &abort_flag, a.timeout_ns};
    auto stage_k = [&](int s) { return sStage + s * C::STAGE_BYTES; };
    auto stage_v = [&](int s) { return sStage + s * C::STAGE_BYTES + C::KV_BYTES; };
    auto stage_vt = [&](int s) { return sStage + s * C::STAGE_BYTES + 2 * C::KV_BYTES; };

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            const uint32_t qf = smem_u32(&bar_q_full);
            mbar_arrive_expect_tx(qf, n_qsub * C::Q_BYTES);
            for (int u = 0; u < n_qsub; ++u)
                for (int c = 0; c < C::NCH; ++c)
                    tma_load_4d(smem_u32(sQ + u * C::Q_BYTES + c * C::BM * 128), &tm_q, qf, c * C::EPC, h,
                                q0 + u * C::BM, b);
            int issued = 0;
            for (int j = 0; j < n_kv; ++j) {
                const int s = j % C::NS;
                if (j >= C::NS &&
                    !mbar_wait(smem_u32(&bar_kv_empty[s]), ((j / C::NS) - 1) & 1, w, SITE_FWD_KV_EMPTY))
                    break;
                const uint32_t full = smem_u32(&bar_kv_full[s]);
                mbar_arrive_expect_tx(full, 2 * C::KV_BYTES);
                for (int c = 0; c < C::NCH; ++c) {
                    tma_load_4d(smem_u32(stage_k(s) + c * C::BN * 128), &tm_k, full, c * C::EPC, hkv, j * C::BN, b);
                    tma_load_4d(smem_u32(stage_v(s) + c * C::BN * 128), &tm_v, full, c * C::EPC, hkv, j * C::BN, b);
                }
                ++issued;
            }
            // Teardown: every copy this CTA started must have landed before exit.
            mbar_wait_drain(qf, 0, w, SITE_FWD_DRAIN);
            for (int j = max(0, issued - C::NS); j < issued; ++j)
                mbar_wait_drain(smem_u32(&bar_kv_full[j % C::NS]), (j / C::NS) & 1, w, SITE_FWD_DRAIN);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ UMMA issuer
        if (lane == 0) {
            constexpr uint32_t id_s = idesc_make(C::FMT_S, 128, C::BN, false, false);
            constexpr uint32_t id_o = idesc_make(C::FMT_PV, 128, D, false, !TF32);
            auto issue_s = [&](int u, int j) {
                const int s = j % C::NS;
                const uint32_t qa = smem_u32(sQ + u * C::Q_BYTES), ka = smem_u32(stage_k(s));
#pragma unroll
                for (int ks = 0; ks < C::S_KSTEPS; ++ks) {
                    const uint32_t byte = ks * 32;
                    umma_ss<TF32>(tm + u * 128, sdesc(qa + (byte >> 7) * C::BM * 128 + (byte & 127), 16, 1024),
                                  sdesc(ka + (byte >> 7) * C::BN * 128 + (byte & 127), 16, 1024), id_s, ks > 0);
                }
                umma_commit(smem_u32(&bar_s_full[u]));
            };
            auto issue_pv = [&](int u, int j) -> bool {
                if (!mbar_wait(smem_u32(&bar_p_ready[u]), j & 1, w, SITE_FWD_P_READY)) return false;
                tc_fence_after();
                const int s = j % C::NS;
#pragma unroll
                for (int ks = 0; ks < C::PV_KSTEPS; ++ks) {
                    uint64_t bd;
                    if constexpr (TF32) {
                        const uint32_t byte = ks * 32;   // V^T [D x BN], K-major, 32 keys per chunk
                        bd = sdesc(smem_u32(stage_vt(s)) + (byte >> 7) * D * 128 + (byte & 127), 16, 1024);
                    } else {                            // V [BN x D], MN-major, D chunks BN*128 apart
                        bd = sdesc(smem_u32(stage_v(s)) + ks * C::PV_ROWS * 128, C::BN * 128, 1024);
                    }
                    umma_ts<TF32>(tm + C::O_COL + u * D, tm + u * 128 + ks * 8, bd, id_o, (j > 0 || ks > 0) ? 1u : 0u);
                }
                umma_commit(smem_u32(&bar_o_done[u]));
                return true;
            };
            bool ok = true;
            for (int u = 0; u < n_qsub && ok; ++u) ok = mbar_wait(smem_u32(&bar_q_ready[u]), 0, w, SITE_FWD_Q);
            ok = ok && mbar_wait(smem_u32(&bar_k_ready[0]), 0, w, SITE_FWD_K_READY);
            if (ok) {
                tc_fence_after();
                if (n_u[0] > 0) issue_s(0, 0);
                if (n_u[1] > 0) issue_s(1, 0);
            }
            for (int j = 0; ok && j < n_kv; ++j) {
                if (j < n_u[0] && !(ok = issue_pv(0, j))) break;
                const bool nxt = j + 1 < n_kv;
                if (nxt) {
                    const int s1 = (j + 1) % C::NS;
                    if (!(ok = mbar_wait(smem_u32(&bar_k_ready[s1]), ((j + 1) / C::NS) & 1, w, SITE_FWD_K_READY)))
                        break;
                    tc_fence_after();
                    if (j + 1 < n_u[0]) issue_s(0, j + 1);
                }
                if (j < n_u[1] && !(ok = issue_pv(1, j))) break;
                umma_commit(smem_u32(&bar_kv_empty[j % C::NS]));
                if (nxt && j + 1 < n_u[1]) issue_s(1, j + 1);
            }
            umma_commit(smem_u32(&bar_final));
        }
    } else if (warp < 4) {
        // ------------------------------------------------------------ RoPE on K (+ V^T)
        const int rt = tid - 64;
        bool ovf = false;
        for (int j = 0; j < n_kv; ++j) {
            const int s = j % C::NS;
            if (!mbar_wait_warp(smem_u32(&bar_kv_full[s]), (j / C::NS) & 1, w, SITE_FWD_KV_FULL)) break;
            if constexpr (TF32) transpose_v_tf32<D, C::BN, 64>(stage_v(s), stage_vt(s), rt);
            ovf |= rope_tile_smem<D, C::BN, 64, C::MODE>(stage_k(s), nullptr, j * C::BN, T, rt, a.rope);
            fence_proxy_async_smem();
            mbar_arrive(smem_u32(&bar_k_ready[s]));
        }
        if (ovf) atomicCAS(a.err, 0, SITE_RANGE);
    } else {
        // ------------------------------------------------------------ softmax (subtile u)
        const int u = (warp - 4) >> 2;
        const int r = tid - 128 - 128 * u;            // query row = TMEM lane
        const int qsub0 = q0 + u * C::BM;
        const int qpos = qsub0 + r;
        const int n = n_u[u];
        const uint32_t lt = tm + ((uint32_t)((warp & 3) * 32) << 16);
        const uint32_t s_col = u * 128, o_col = C::O_COL + u * D;
        uint8_t* sQu = sQ + u * C::Q_BYTES;
        const float sl2 = a.scale_log2;
        float m_used = kNegInf, l = 0.f;
        bool ok = n > 0;
        if (ok && mbar_wait_warp(smem_u32(&bar_q_full), 0, w, SITE_FWD_Q)) {
            if (rope_tile_smem<D, C::BM, 128, C::MODE>(sQu, nullptr, qsub0, T, r, a.rope))
                atomicCAS(a.err, 0, SITE_RANGE);
            fence_proxy_async_smem();
            mbar_arrive(smem_u32(&bar_q_ready[u]));
        } else {
            ok = false;
        }
        for (int j = 0; ok && j < n; ++j) {
            if (!mbar_wait_warp(smem_u32(&bar_s_full[u]), j & 1, w, SITE_FWD_S_FULL)) { ok = false; break; }
            tc_fence_after();
            uint32_t sr[C::BN];
            tmem_ld_cols<C::BN / 32>(lt + s_col, sr);
            const int kv0 = j * C::BN;
            if (kv0 + C::BN - 1 > qsub0) {          // tile crosses the diagonal: mask j > i
#pragma unroll
                for (int e = 0; e < C::BN; ++e)
                    if (kv0 + e > qpos) sr[e] = __float_as_uint(kNegInf);
            }
            // Row max over 8 independent chains (one warp per SMSP runs this: a single
            // dependent chain of BN maxes would serialise on the FMNMX latency).
            float m8[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) m8[k] = __uint_as_float(sr[k]);
#pragma unroll
            for (int e = 8; e < C::BN; ++e) m8[e & 7] = fmaxf(m8[e & 7], __uint_as_float(sr[e]));
            const float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                                   fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
            const float m_tile = mx * sl2;
            // A row whose max grew by more than 2^8 rescales l and its O row; the others
            // keep their max (p <= 2^8 stays exact).  TMEM access is warp-collective, so
            // a warp rescales when any lane needs it (alpha = 1 elsewhere).  O is idle
            // here: the PV of tile j-1 finished before S of tile j was issued.
            const bool need = j > 0 && m_tile > m_used + 8.f;
            if (j == 0) m_used = m_tile;
            if (__any_sync(0xffffffffu, need)) {
                const float alpha = need ? ex2(m_used - m_tile) : 1.f;
                l *= alpha;
                if (need) m_used = m_tile;
                if (!mbar_wait_warp(smem_u32(&bar_o_done[u]), (j - 1) & 1, w, SITE_FWD_O_DONE)) { ok = false; break; }
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < D; c += 32) {
                    uint32_t orow[32];
                    tmem_ld_cols<1>(lt + o_col + c, orow);
#pragma unroll
                    for (int e = 0; e < 32; ++e) orow[e] = __float_as_uint(__uint_as_float(orow[e]) * alpha);
                    tmem_st32(lt + o_col + c, orow);
                }
            }
            float s8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            const float neg_m = -m_used;
#pragma unroll
            for (int c = 0; c < C::BN; c += 32) {
                if constexpr (TF32) {
                    uint32_t pk[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const float p = ex2(fmaf(__uint_as_float(sr[c + e]), sl2, neg_m));
                        s8[e & 7] += p;
                        pk[e] = f32_to_tf32_rna(p);
                    }
                    tmem_st32(lt + s_col + c, pk);
                } else {
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        const float p0 = ex2(fmaf(__uint_as_float(sr[c + e]), sl2, neg_m));
                        const float p1 = ex2(fmaf(__uint_as_float(sr[c + e + 1]), sl2, neg_m));
                        s8[e & 7] += p0;
                        s8[(e + 1) & 7] += p1;
                        pk[e >> 1] = pack_bf162(p0, p1);
                    }
                    tmem_st16(lt + s_col + (c >> 1), pk);
                }
            }
            l += ((s8[0] + s8[1]) + (s8[2] + s8[3])) + ((s8[4] + s8[5]) + (s8[6] + s8[7]));
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(smem_u32(&bar_p_ready[u]));
        }
        // Epilogue: O / l staged (swizzled) in this subtile's Q buffer, stored by TMA;
        // LSE = natural log of the partition sum of the scaled logits.
        if (ok && mbar_wait_warp(smem_u32(&bar_o_done[u]), (n - 1) & 1, w, SITE_FWD_O_DONE)) {
            tc_fence_after();
            const float inv_l = 1.f / l;
#pragma unroll
            for (int c = 0; c < D; c += 32) {
                uint32_t orow[32];
                tmem_ld_cols<1>(lt + o_col + c, orow);
                if constexpr (TF32) {
                    uint8_t* dst = sQu + (c >> 5) * C::BM * 128;
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        *reinterpret_cast<float4*>(dst + sw128_offset(r, k)) =
                            make_float4(__uint_as_float(orow[4 * k]) * inv_l, __uint_as_float(orow[4 * k + 1]) * inv_l,
                                        __uint_as_float(orow[4 * k + 2]) * inv_l,
                                        __uint_as_float(orow[4 * k + 3]) * inv_l);
                } else {
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 32; e += 2)
                        pk[e >> 1] = pack_bf162(__uint_as_float(orow[e]) * inv_l, __uint_as_float(orow[e + 1]) * inv_l);
                    uint8_t* dst = sQu + (c >> 6) * C::BM * 128;
                    const int u0 = (c & 63) >> 3;
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        *reinterpret_cast<uint4*>(dst + sw128_offset(r, u0 + k)) =
                            make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
                }
            }
            fence_proxy_async_smem();
            mbar_arrive(smem_u32(&bar_o_staged[u]));
            if (qpos < T) a.lse[((size_t)b * a.Hq + h) * T + qpos] = (m_used + log2f(l)) * 0.6931471805599453f;
            if (r == 0 && mbar_wait(smem_u32(&bar_o_staged[u]), 0, w, SITE_FWD_O_DONE)) {
                for (int c = 0; c < C::NCH; ++c)
                    tma_store_4d(&tm_o, smem_u32(sQu + c * C::BM * 128), c * C::EPC, h, qsub0, b);
                bulk_commit_group();
                bulk_wait_group_read0();
            }
        }
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        mbar_wait_drain(smem_u32(&bar_final), 0, w, SITE_FWD_DRAIN);
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tm, 512);
    }
}

template <bool TF32, int D>
cudaError_t launch_fwd_t(int B, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const CUtensorMap& to, const FwdArgs& a, cudaStream_t st) {
    using C = FwdCfg<TF32, D>;
    auto kfn = attn_fwd_kernel<TF32, D>;
    cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    dim3 grid(a.Hq, B, a.n_qt);
    kfn<<<grid, C::THREADS, C::SMEM, st>>>(tq, tk, tv, to, a);
    return cudaGetLastError();
}

}  // namespace

int fwd_kv_box_rows(bool tf32, int D) { return (tf32 && D == 64) ? 64 : 128; }

cudaError_t launch_fwd(bool tf32, int D, int B, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, const CUtensorMap& to, const FwdArgs& a, cudaStream_t st) {
    if (!tf32) {
        if (D == 64) return launch_fwd_t<false, 64>(B, tq, tk, tv, to, a, st);
        if (D == 128) return launch_fwd_t<false, 128>(B, tq, tk, tv, to, a, st);
    } else {
        if (D == 32) return launch_fwd_t<true, 32>(B, tq, tk, tv, to, a, st);
        if (D == 64) return launch_fwd_t<true, 64>(B, tq, tk, tv, to, a, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace ne
