// attn_bwd_d64.cu -- backward main kernel for head_dim 64 (bf16 tensors): the hand-written
// backward of "NanoEuler: C와 CUDA로 밑바닥부터 구축한 GPT-2 규모의 LLM" (검증 및 안정성)
// for the causal GQA + RoPE attention of the same page (기술 사양, 커널 구현).  With
// s = 1/sqrt(D), Q' = R Q, K' = R K (rows rotated by their positions):
//   P^T  = exp(s K'Q'^T - LSE)            recomputed per tile from the forward's LSE
//   dP^T = V dO^T,  dS^T = P^T o (dP^T - Delta)
//   dV  += P^T dO,  dK' += dS^T Q',  dQ' = dS K'   (dK = s R^T dK', dQ = s R^T dQ')
//
// One CTA per (batch, kv head, 128-key tile) loops over the G query heads of its group
// and every 128-query tile on or after the diagonal; dK and dV stay in TMEM for the whole
// group (no atomics).  Each query tile is taken as two 64-query half-steps, and the two
// softmax-gradient warp groups take alternate half-steps (group h the half h of every
// tile): while one group waits on its barriers, the other keeps the special-function unit
// busy with its exponentials.  dQ' of a whole 128-query tile is one M = 128 MMA over the
// two halves' dS; the drain warps stage it in shared memory and one TMA bulk reduce-add
// per tile adds it into the fp32 accumulator.
//
// A chain of K-step MMAs into one accumulator, plus its commit and the waiter's wake-up,
// takes ~600 cycles on an idle tensor pipe and more under load, so S^T, dP^T and P^T are
// double-buffered in TMEM (one buffer per warp group): those of half-step i+2 are issued
// as soon as its group holds half-step i's in registers.
//
// Operand precision: Q', K' and dS are fp16 (logits and dS keep 3 more mantissa bits
// than bf16; a rotated value or a dS beyond the fp16 range is reported as an error, never
// silently saturated); P^T, V and dO are bf16.  Every MMA has one operand type.  Q' comes
// rotated and rounded to fp16 from the preprocess kernel (each query row is rotated once,
// not once per key tile); K' is rotated here.
//
// Warp roles (512 threads, one CTA per SM):
//   warp 0      TMA producer (K, V once; Q, dO half tiles into an NQS ring) and the dQ'
//               issuer (once per 128-query tile).
//   warp 1      TMEM allocator; S^T issuer.
//   warp 2      dP^T issuer.
//   warp 3      dV and dK' issuer.
//   warps 4-7   RoPE of K once (in place, to fp16), and the dQ' drain (thread = query row
//               of the tile = TMEM lane) through the staging tile.
//   warps 8-15  two groups of 128 threads (thread = key row = TMEM lane); group h takes
//               the half-steps h, h+2, ... (all 64 query columns, in two 32-column
//               chunks); at the end group 0 writes dK (inverse rotation, scale), group 1 dV.
// TMEM: S^T of buffer b (= warp group) at 128b and dP^T at 128b + 64 (64 cols each),
// packed bf16 P^T of buffer b at 256 + 32b, dV at 320, dK' at 384, dQ' at 448.
// Shared memory: K' (fp16), V, NQS x (Q' half | dO half), two dS^T tiles [key][query], the
// fp32 dQ' staging tile (two 128-byte-swizzled column chunks, as the reduce's box expects).
// Every wait is bounded; a CTA that gives up records an error code, drains its own copies
// and MMAs and frees its TMEM.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include "kernels.h"
#include "ptx.cuh"
#include "rope_smem.cuh"

namespace ne {

namespace {

struct Bwd64 {
    static constexpr int D = 64;
    static constexpr int BKV = 128;                  // key rows per CTA
    static constexpr int BT = 128;                   // query rows per tile
    static constexpr int BH = 64;                    // query rows per half-step
    static constexpr int KV_BYTES = BKV * 128;       // one 128-byte row per key
    static constexpr int H_BYTES = BH * 128;         // a Q or dO half tile
    static constexpr int STAGE_BYTES = 2 * H_BYTES;  // Q' | dO
    static constexpr int NQS = 5;                    // half-step stages
    static constexpr int DS_TILE = BKV * BT * 2;     // dS^T [key][query] fp16: two 64-query chunks
    static constexpr int DS_CHUNK = BKV * 128;
    static constexpr int DQ_STAGE = BT * D * 4;      // fp32 dQ' of a tile: two 32-column chunks
    static constexpr int SMEM = 1024 + 2 * KV_BYTES + NQS * STAGE_BYTES + 2 * DS_TILE + DQ_STAGE;
    static constexpr int PT_COL = 256, DV_COL = 320, DK_COL = 384, DQ_COL = 448;
    static constexpr int THREADS = 512;
    static_assert(SMEM <= 227 * 1024, "shared memory");
};

// (query head, first query row) of tile tau, advanced one tile at a time: the tiles of a
// CTA run over the G heads of its kv group and, per head, the 128-query tiles j .. n_qt-1.
// (Dividing tau by the per-head count in the loops would go through the special-function
// unit, which the exponentials keep busy.)
struct TileWalk {
    int h, qt;
    __device__ __forceinline__ void init(int hkv, int G, int j) {
        h = hkv * G;
        qt = j;
    }
    __device__ __forceinline__ void next(int j, int n_qt) {
        if (++qt == n_qt) {
            qt = j;
            ++h;
        }
    }
    __device__ __forceinline__ int q0() const { return qt * Bwd64::BT; }
};

// One 32-query chunk of one key row: P^T = exp2(S^T s log2e - LSE log2e) and
// dS^T = P^T o (dP^T - Delta), packed to bf16 (P^T) and fp16 (dS^T).  With MASK, query i
// of the chunk is masked (P = 0) when i < kl: kl is the key's lane when the warp's 32
// keys and the chunk's queries start at the same position, and 32 when every key
// follows every query (the chunk is all zero).
// amax2 keeps the largest |dS| as packed fp16, so a value past the fp16 range shows up
// as infinity.
// nlse2 and ndelta hold -LSE log2(e) and -Delta of the chunk's queries, so that the
// exponent argument, dP - Delta and the product P (dP - Delta) run as packed f32x2
// instructions, two queries each.
template <bool MASK>
__device__ __forceinline__ void grad_chunk(const uint32_t (&sr)[32], const uint32_t (&dr)[32], const float* nlse2,
                                           const float* ndelta, float sl2, int kl, int qlim, uint32_t (&pk)[16],
                                           uint32_t (&dk)[16], __half2& amax2) {
    const float4* l4 = reinterpret_cast<const float4*>(nlse2);
    const float4* d4 = reinterpret_cast<const float4*>(ndelta);
    const float2 sl2v = make_float2(sl2, sl2);
#pragma unroll
    for (int e = 0; e < 32; e += 4) {
        const float4 lq4 = l4[e >> 2], dq4 = d4[e >> 2];   // broadcast reads
        const float2 x01 = __ffma2_rn(make_float2(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])), sl2v,
                                      make_float2(lq4.x, lq4.y));
        const float2 x23 = __ffma2_rn(make_float2(__uint_as_float(sr[e + 2]), __uint_as_float(sr[e + 3])), sl2v,
                                      make_float2(lq4.z, lq4.w));
        float p[4] = {ex2(x01.x), ex2(x01.y), ex2(x23.x), ex2(x23.y)};
        if (MASK) {
#pragma unroll
            for (int k = 0; k < 4; ++k)
                if (kl > e + k || e + k >= qlim) p[k] = 0.f;
        }
        const float2 g01 = __fadd2_rn(make_float2(__uint_as_float(dr[e]), __uint_as_float(dr[e + 1])),
                                      make_float2(dq4.x, dq4.y));
        const float2 g23 = __fadd2_rn(make_float2(__uint_as_float(dr[e + 2]), __uint_as_float(dr[e + 3])),
                                      make_float2(dq4.z, dq4.w));
        const float2 d01 = __fmul2_rn(make_float2(p[0], p[1]), g01);
        const float2 d23 = __fmul2_rn(make_float2(p[2], p[3]), g23);
        const float ds[4] = {d01.x, d01.y, d23.x, d23.y};
        pk[e >> 1] = pack_bf162(p[0], p[1]);
        pk[(e >> 1) + 1] = pack_bf162(p[2], p[3]);
        dk[e >> 1] = pack_half2(ds[0], ds[1]);
        dk[(e >> 1) + 1] = pack_half2(ds[2], ds[3]);
        amax2 = __hmax2(amax2, __habs2(*reinterpret_cast<const __half2*>(&dk[e >> 1])));
        amax2 = __hmax2(amax2, __habs2(*reinterpret_cast<const __half2*>(&dk[(e >> 1) + 1])));
    }
}

__device__ __forceinline__ uint32_t s_col(int b) { return (uint32_t)(128 * b); }
__device__ __forceinline__ uint32_t dp_col(int b) { return (uint32_t)(128 * b + 64); }
// Packed P^T of buffer b: 64 queries in 32 columns.
__device__ __forceinline__ uint32_t pt_col(int b) { return (uint32_t)(Bwd64::PT_COL + 32 * b); }

// VL: per-sequence lengths (padded batch).  Without them every length is T, rows past T
// arrive as TMA's zero fill, and the padding code compiles away.
template <bool VL>
__global__ void __launch_bounds__(512, 1)
    attn_bwd_d64_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                        const __grid_constant__ CUtensorMap tm_dq, const BwdArgs a) {
    using C = Bwd64;
    constexpr int D = C::D;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sK = smem;                              // K, rotated in place to fp16
    uint8_t* sV = sK + C::KV_BYTES;
    uint8_t* sStage = sV + C::KV_BYTES;              // NQS x (Q half | dO half)
    uint8_t* sDS = sStage + C::NQS * C::STAGE_BYTES; // two dS^T tiles
    uint8_t* sDQ = sDS + 2 * C::DS_TILE;             // dQ' staging for the bulk reduce
    auto stage_q = [&](int s) { return sStage + s * C::STAGE_BYTES; };
    auto stage_do = [&](int s) { return sStage + s * C::STAGE_BYTES + C::H_BYTES; };
    auto ds_tile = [&](int tb) { return sDS + tb * C::DS_TILE; };

    __shared__ __align__(8) uint64_t bar_kv_full, bar_k_ready, bar_dkv_full, bar_final;
    __shared__ __align__(8) uint64_t bar_qdo_full[C::NQS], bar_qdo_empty[C::NQS];
    __shared__ __align__(8) uint64_t bar_sdp_full[2];                 // [S^T/dP^T buffer]: both MMAs done
    __shared__ __align__(8) uint64_t bar_sp_read[2];                  // ... read into registers
    __shared__ __align__(8) uint64_t bar_ds_half[2];   // [half]: P^T and the dS^T half of a half-step written
    __shared__ __align__(8) uint64_t bar_ds_tile[2];   // [dS^T tile buffer]: both halves written
    __shared__ __align__(8) uint64_t bar_ds_free[2];   // [dS^T tile buffer]: dK' and dQ' done with it
    __shared__ __align__(8) uint64_t bar_dq_full, bar_dq_free;          // dQ' TMEM accumulator
    __shared__ __align__(8) uint64_t bar_stage_free, bar_staged;   // dQ' staging tile
    __shared__ __align__(16) float s_lse[8][2][64];    // [softmax warp][buffer][query column]
    __shared__ __align__(16) float s_delta[8][2][64];
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // Grid order: (kv head, batch row) fastest, so the first CTAs to start are every
    // group's first key tiles, the heaviest; or, when the fp32 dQ' accumulator is larger
    // than about a third of the L2 and a group has at most 16 key tiles, key tile
    // fastest, so the CTAs running together add into the accumulators of several groups
    // and their reduce-adds stay in L2 (B32 T2048: 816 -> 741 us; B128 T512: 325 -> 299).
    // With 64 and 128 key tiles per group that order measured slower (T8192 +2%, T16384
    // +1.4%): the CTAs running together then all add into one or two groups, and the
    // heaviest tiles of the last groups start late.  32 (T4096) is not measured and keeps
    // the heaviest-first order.
    const int hkv = a.group_major ? (int)blockIdx.y : (int)blockIdx.x;
    const int b = a.group_major ? (int)blockIdx.z : (int)blockIdx.y;
    const int j = a.group_major ? (int)blockIdx.x : (int)blockIdx.z;
    const int T = a.T, G = a.G;
    const int kv0 = j * C::BKV;
    // Query tiles end at the sequence's length (T without per-sequence lengths); a key
    // tile wholly past it has no query tile and writes zero gradients.
    const int len = VL ? seq_len(a.seq_lens, b, T) : T;
    const int n_qt = (len + C::BT - 1) / C::BT;
    const int per_head = n_qt > j ? n_qt - j : 0;    // 128-query tiles on or after the diagonal
    const int n_tiles = G * per_head;
    const int n_hs = 2 * n_tiles;

    if (tid == 0) {
        mbar_init(smem_u32(&bar_kv_full), 1);
        mbar_init(smem_u32(&bar_k_ready), 128);

        mbar_init(smem_u32(&bar_dkv_full), 1);
        mbar_init(smem_u32(&bar_final), 4);          // one commit per UMMA issuer
        for (int s = 0; s < C::NQS; ++s) {
            mbar_init(smem_u32(&bar_qdo_full[s]), 1);
            mbar_init(smem_u32(&bar_qdo_empty[s]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&bar_sdp_full[i]), 2);   // the S^T and the dP^T issuer
            mbar_init(smem_u32(&bar_sp_read[i]), 128);   // the warp group of buffer i
            mbar_init(smem_u32(&bar_ds_half[i]), 128);   // the warp group of half i
            mbar_init(smem_u32(&bar_ds_tile[i]), 256);
            mbar_init(smem_u32(&bar_ds_free[i]), 2);  // dK' issuer (after the odd half) and dQ' issuer
        }
        mbar_init(smem_u32(&bar_stage_free), 1);
        mbar_init(smem_u32(&bar_dq_full), 1);
        mbar_init(smem_u32(&bar_dq_free), 128);
        mbar_init(smem_u32(&bar_staged), 128);
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

    auto kdesc = [](const void* p) { return sdesc(smem_u32(p), 16, 1024); };                 // K-major
    auto mndesc = [](const void* p, uint32_t lbo) { return sdesc(smem_u32(p), lbo, 1024); };  // MN-major

    // The issuing warps (0-3) run their loops with all 32 lanes, so that descriptors and
    // loop state stay warp-uniform; one elected lane issues each batch of MMAs and their
    // commits in one branch (an election per MMA took several times the instructions),
    // and lane 0 issues the TMA copies.
    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer + dQ' issuer
        const uint32_t kvf = smem_u32(&bar_kv_full);
        if (lane == 0) {
            mbar_arrive_expect_tx(kvf, 2 * C::KV_BYTES);
            tma_load_4d(smem_u32(sK), &tm_k, kvf, 0, hkv, kv0, b);
            tma_load_4d(smem_u32(sV), &tm_v, kvf, 0, hkv, kv0, b);
        }
        int issued = 0;
        TileWalk lw;                                 // tile of the next half-step to load
        lw.init(hkv, G, j);
        auto load = [&](int hs) -> bool {
            const int s = hs % C::NQS;
            if (hs >= C::NQS &&
                !mbar_wait_warp(smem_u32(&bar_qdo_empty[s]), ((hs / C::NQS) - 1) & 1, w, SITE_BWD_QDO_EMPTY))
                return false;
            if (lane == 0) {
                const uint32_t f = smem_u32(&bar_qdo_full[s]);
                const int h = lw.h, q0 = lw.q0() + (hs & 1) * C::BH;
                mbar_arrive_expect_tx(f, 2 * C::H_BYTES);
                tma_load_4d(smem_u32(stage_q(s)), &tm_q, f, 0, h, q0, b);
                tma_load_4d(smem_u32(stage_do(s)), &tm_do, f, 0, h, q0, b);
            }
            if (hs & 1) lw.next(j, n_qt);
            ++issued;
            return true;
        };
        bool ok = true;
        for (int hs = 0; ok && hs < C::NQS && hs < n_hs; ++hs) ok = load(hs);
        constexpr uint32_t id_dq = idesc_make(FMT_F16, 128, D, true, true);   // A, B MN-major
        const uint64_t dKmn = mndesc(sK, C::BKV * 128);
        if (ok) ok = mbar_wait_warp(smem_u32(&bar_k_ready), 0, w, SITE_BWD_KV);
        for (int tau = 0; ok && tau < n_tiles; ++tau) {
            const int tb = tau & 1;
            if (!(ok = mbar_wait_warp(smem_u32(&bar_ds_tile[tb]), (tau >> 1) & 1, w, SITE_BWD_DS_READY))) break;
            // The drain warps have taken the previous tile's dQ' out of TMEM.
            if (tau >= 1 && !(ok = mbar_wait_warp(smem_u32(&bar_dq_free), (tau - 1) & 1, w, SITE_BWD_DQ_FREE)))
                break;
            tc_fence_after();
            const uint64_t dSmn = mndesc(ds_tile(tb), C::DS_CHUNK);
            if (elect_one()) {
#pragma unroll
                for (int ks = 0; ks < C::BKV / 16; ++ks)    // dQ' = dS K', K = key rows
                    umma_ss<false>(tm + C::DQ_COL, sdesc_add(dSmn, ks * 16 * 128), sdesc_add(dKmn, ks * 16 * 128),
                                   id_dq, ks > 0);
                umma_commit(smem_u32(&bar_dq_full));
                umma_commit(smem_u32(&bar_ds_free[tb]));
            }
            __syncwarp();
            for (int hs = 2 * tau + C::NQS; ok && hs < 2 * tau + C::NQS + 2 && hs < n_hs; ++hs) ok = load(hs);
        }
        umma_commit_e(smem_u32(&bar_final));
        // Teardown: every copy this CTA started must have landed before exit.
        if (lane == 0) {
            mbar_wait_drain(kvf, 0, w, SITE_BWD_DRAIN);
            for (int hs = max(0, issued - C::NQS); hs < issued; ++hs)
                mbar_wait_drain(smem_u32(&bar_qdo_full[hs % C::NQS]), (hs / C::NQS) & 1, w, SITE_BWD_DRAIN);
        }
    } else if (warp == 1 || warp == 2) {
        // ------------------------------------------------------------ S^T (warp 1) / dP^T (warp 2)
        const bool is_s = warp == 1;
        // S^T = K'Q'^T on fp16 operands, dP^T = V dO^T on bf16.
        const uint32_t id = is_s ? idesc_make(FMT_F16, 128, C::BH, false, false)
                                 : idesc_make(FMT_BF16, 128, C::BH, false, false);
        const uint64_t dA = kdesc(is_s ? sK : sV);
        const uint64_t dB0 = kdesc(is_s ? stage_q(0) : stage_do(0));
        // S^T waits for the rotated K' (once), both for the copies of Q' / dO.
        bool ok = is_s ? mbar_wait_warp(smem_u32(&bar_k_ready), 0, w, SITE_BWD_KV)
                       : mbar_wait_warp(smem_u32(&bar_kv_full), 0, w, SITE_BWD_KV);
        for (int hs = 0; ok && hs < n_hs; ++hs) {
            const int s = hs % C::NQS, bf = hs & 1;
            if (!(ok = mbar_wait_warp(smem_u32(&bar_qdo_full[s]), (hs / C::NQS) & 1, w, SITE_BWD_QDO_FULL))) break;
            // Buffer bf is free once its warp group holds half-step hs-2's S^T and dP^T in
            // registers.
            if (hs >= 2 &&
                !(ok = mbar_wait_warp(smem_u32(&bar_sp_read[bf]), ((hs - 2) >> 1) & 1, w, SITE_BWD_DS_READY)))
                break;
            tc_fence_after();
            const uint64_t dB = sdesc_add(dB0, s * C::STAGE_BYTES);
            const uint32_t dcol = tm + (is_s ? s_col(bf) : dp_col(bf));
            if (elect_one()) {                              // one elected lane issues the batch
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks)        // K = head_dim: 16 per step (32 bytes)
                    umma_ss<false>(dcol, sdesc_add(dA, ks * 32), sdesc_add(dB, ks * 32), id, ks > 0);
                umma_commit(smem_u32(&bar_sdp_full[bf]));
            }
            __syncwarp();
        }
        umma_commit_e(smem_u32(&bar_final));
    } else if (warp == 3) {
        // ------------------------------------------------------------ dV, dK' issuer
        constexpr uint32_t id_dv = idesc_make(FMT_BF16, 128, D, false, true);   // B (dO) MN-major
        constexpr uint32_t id_dk = idesc_make(FMT_F16, 128, D, false, true);    // B (Q') MN-major
        const uint64_t dQmn0 = mndesc(stage_q(0), C::H_BYTES), dOmn0 = mndesc(stage_do(0), C::H_BYTES);
        bool ok = true;
        for (int hs = 0; ok && hs < n_hs; ++hs) {
            const int s = hs % C::NQS, half = hs & 1, tau = hs >> 1, tb = tau & 1;
            if (!(ok = mbar_wait_warp(smem_u32(&bar_ds_half[half]), tau & 1, w, SITE_BWD_DS_READY))) break;
            tc_fence_after();
            const uint64_t dOmn = sdesc_add(dOmn0, s * C::STAGE_BYTES), dQmn = sdesc_add(dQmn0, s * C::STAGE_BYTES);
            const uint64_t dDS = kdesc(ds_tile(tb) + half * C::DS_CHUNK);
            if (elect_one()) {
#pragma unroll
                for (int ks = 0; ks < C::BH / 16; ++ks)     // dV += P^T dO (P^T from TMEM), K = queries
                    umma_ts<false>(tm + C::DV_COL, tm + pt_col(half) + 8 * ks, sdesc_add(dOmn, ks * 16 * 128), id_dv,
                                   (hs > 0 || ks > 0) ? 1u : 0u);
#pragma unroll
                for (int ks = 0; ks < C::BH / 16; ++ks)     // dK' += dS^T Q', K = queries
                    umma_ss<false>(tm + C::DK_COL, sdesc_add(dDS, ks * 32), sdesc_add(dQmn, ks * 16 * 128), id_dk,
                                   (hs > 0 || ks > 0) ? 1u : 0u);
                umma_commit(smem_u32(&bar_qdo_empty[s]));
                if (half == 1) umma_commit(smem_u32(&bar_ds_free[tb]));
            }
            __syncwarp();
        }
        umma_commit_e(smem_u32(&bar_dkv_full));
        umma_commit_e(smem_u32(&bar_final));
    } else if (warp < 8) {
        // ------------------------------------------------------------ RoPE on K and Q; dQ' drain
        const int r = tid - 128;
        const uint32_t lt = tm + ((uint32_t)((warp & 3) * 32) << 16);
        bool ovf = false;
        bool ok = mbar_wait_warp(smem_u32(&bar_kv_full), 0, w, SITE_BWD_KV);
        if (ok) {
            ovf |= rope_tile_smem<D, C::BKV, 128, ROPE_F16, true>(sK, nullptr, kv0, T, r, a.rope,
                                                                   VL ? len : kv0 + C::BKV);
            fence_proxy_async_smem();
            mbar_arrive(smem_u32(&bar_k_ready));
        }
        TileWalk dw;
        dw.init(hkv, G, j);
        for (int tau = 0; ok && tau < n_tiles; ++tau, dw.next(j, n_qt)) {
            if (!(ok = mbar_wait_warp(smem_u32(&bar_dq_full), tau & 1, w, SITE_BWD_DQ_FULL))) break;
            tc_fence_after();
            uint32_t v[64];
            tmem_ld_cols<2>(lt + C::DQ_COL, v);
            tc_fence_before();
            mbar_arrive(smem_u32(&bar_dq_free));
            // The staging tile is free once the previous tile's reduce has read it.
            if (tau > 0) {
                if (r == 0) {
                    bulk_wait_group_read0();
                    mbar_arrive(smem_u32(&bar_stage_free));
                }
                if (!(ok = mbar_wait_warp(smem_u32(&bar_stage_free), (tau - 1) & 1, w, SITE_BWD_DQ_FREE))) break;
            }
#pragma unroll
            for (int c = 0; c < 2; ++c)
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    *reinterpret_cast<uint4*>(sDQ + c * (C::BT * 128) + sw128_offset(r, u)) =
                        make_uint4(v[32 * c + 4 * u], v[32 * c + 4 * u + 1], v[32 * c + 4 * u + 2], v[32 * c + 4 * u + 3]);
            fence_proxy_async_smem();
            mbar_arrive(smem_u32(&bar_staged));
            bool issued = true;
            if (r == 0) {
                issued = mbar_wait(smem_u32(&bar_staged), tau & 1, w, SITE_BWD_DQ_FULL);
                if (issued) {
                    // Rows at or beyond T lie outside the tensor map and are skipped.
                    const int h = dw.h, q0 = dw.q0();
                    tma_reduce_add_4d(&tm_dq, smem_u32(sDQ), 0, h, q0, b);
                    tma_reduce_add_4d(&tm_dq, smem_u32(sDQ + C::BT * 128), 32, h, q0, b);
                    bulk_commit_group();
                }
            }
            if (!(ok = __all_sync(0xffffffffu, issued))) break;   // the warp leaves the loop together
        }
        if (r == 0) bulk_wait_group0();   // the last reduces have completed before the CTA exits
        if (ovf) report_error(a.err, SITE_RANGE);
    } else {
        // ------------------------------------------------------------ P^T, dS^T; dK, dV epilogue
        const int g = (warp - 8) >> 2;                   // warp group = half index = TMEM buffer
        const int r = (warp & 3) * 32 + lane;            // key row = TMEM lane
        const int kvpos = kv0 + r;
        const int kw = kv0 + (warp & 3) * 32;            // first key row of this warp
        const uint32_t lt = tm + ((uint32_t)((warp & 3) * 32) << 16);
        const float sl2 = a.scale_log2;
        __half2 amax2 = __floats2half2_rn(0.f, 0.f);
        bool ok = true;
        // LSE / Delta of the 64 query columns: lanes l and l+32 fetch columns l and l+32 of
        // the group's next half-step while the current one runs, and the warp stages them in
        // its own double-buffered slot (read back as broadcasts; __syncwarp orders the warp's
        // own writes and reads, so no cross-warp barrier is needed).  The loaded values are
        // not touched until they are staged (a use right after the load would stall).
        const int sw = warp - 8;
        // Half-step hs = 2 tau + g lies in tile tau; `cur` walks the group's current tile,
        // `nxt` the one after it.
        TileWalk cur, nxt;
        cur.init(hkv, G, j);
        nxt = cur;
        nxt.next(j, n_qt);
        auto row_vals = [&](const TileWalk& tw, float (&lv)[2], float (&dv)[2]) {
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int qpos = tw.q0() + g * C::BH + lane + 32 * k;
                const size_t rix = ((size_t)b * a.Hq + tw.h) * T + qpos;
                lv[k] = 0.f;
                dv[k] = 0.f;
                if (qpos < len) {
                    lv[k] = __ldg(a.lse + rix);
                    dv[k] = __ldg(a.delta + rix);
                }
            }
        };
        auto publish = [&](int hs, const float (&lv)[2], const float (&dv)[2]) {
            const int buf = (hs >> 1) & 1;
#pragma unroll
            for (int k = 0; k < 2; ++k) {       // negated: added by packed FMA / add
                s_lse[sw][buf][lane + 32 * k] = -(lv[k] * 1.4426950408889634f);
                s_delta[sw][buf][lane + 32 * k] = -dv[k];
            }
            __syncwarp();
        };
        if (g < n_hs) {
            float lv[2], dv[2];
            row_vals(cur, lv, dv);
            publish(g, lv, dv);
        }
        for (int hs = g; hs < n_hs; hs += 2, cur = nxt, nxt.next(j, n_qt)) {
            const int tau = hs >> 1, tb = tau & 1, buf = (hs >> 1) & 1;
            const int q0 = cur.q0() + g * C::BH;
            float lv_n[2] = {0.f, 0.f}, dv_n[2] = {0.f, 0.f};
            if (hs + 2 < n_hs) row_vals(nxt, lv_n, dv_n);   // in flight during this half-step
            if (!(ok = mbar_wait_warp(smem_u32(&bar_sdp_full[g]), (hs >> 1) & 1, w, SITE_BWD_S_FULL))) break;
            tc_fence_after();
            uint8_t* dsbase = ds_tile(tb) + g * C::DS_CHUNK;
#pragma unroll
            for (int c = 0; c < 2; ++c) {                // two 32-query chunks
                uint32_t sr[32], dr[32];
                tmem_ld32(lt + s_col(g) + 32 * c, sr);
                tmem_ld32(lt + dp_col(g) + 32 * c, dr);
                tmem_wait_ld();
                reg_fence32(sr);
                reg_fence32(dr);
                if (c == 1) {                            // the buffer may take half-step hs+2
                    tc_fence_before();
                    mbar_arrive(smem_u32(&bar_sp_read[g]));
                }
                // The causal mask on the block of this warp's 32 keys and the chunk's 32
                // queries (both start on 32-row boundaries) is warp-uniform: every key
                // after every query, none, or the diagonal block (key lane masked for the
                // queries before it).
                uint32_t pk[16], dk[16];
                const int qc = q0 + 32 * c;
                const float* lrow = &s_lse[sw][buf][32 * c];
                const float* drow = &s_delta[sw][buf][32 * c];
                // Queries of the chunk at or past the sequence's length are padding (masked).
                const int qlim = VL ? len - qc : 32;
                if (kw < qc && qlim >= 32) grad_chunk<false>(sr, dr, lrow, drow, sl2, -1, 32, pk, dk, amax2);
                else grad_chunk<true>(sr, dr, lrow, drow, sl2, kw < qc ? -1 : (kw == qc ? lane : 32), qlim, pk, dk, amax2);
                if (c == 0) {
                    // P^T buffer g is free once dV of half-step hs-2 has read it: that
                    // half-step's stage release, committed after its dK' (issued after its
                    // dV by the same thread), says so.  The dS^T tile buffer is free once
                    // dK' and dQ' of tile tau-2 have read it.
                    if (hs >= 2 && !(ok = mbar_wait_warp(smem_u32(&bar_qdo_empty[(hs - 2) % C::NQS]),
                                                         ((hs - 2) / C::NQS) & 1, w, SITE_BWD_DS_READY)))
                        break;
                    if (tau >= 2 &&
                        !(ok = mbar_wait_warp(smem_u32(&bar_ds_free[tb]), ((tau - 2) >> 1) & 1, w, SITE_BWD_DS_FREE)))
                        break;
                    tc_fence_after();
                }
                tmem_st16(lt + pt_col(g) + 16 * c, pk);
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    *reinterpret_cast<uint4*>(dsbase + sw128_offset(r, 4 * c + k)) =
                        make_uint4(dk[4 * k], dk[4 * k + 1], dk[4 * k + 2], dk[4 * k + 3]);
            }
            if (!ok) break;
            fence_proxy_async_smem();
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(smem_u32(&bar_ds_half[g]));
            mbar_arrive(smem_u32(&bar_ds_tile[tb]));
            if (hs + 2 < n_hs) publish(hs + 2, lv_n, dv_n);
        }
        // A dS beyond the fp16 range rounded to infinity.
        if (fmaxf(__low2float(amax2), __high2float(amax2)) > 65504.f) report_error(a.err, SITE_RANGE);
        // Epilogue, key row r of this CTA's tile: group 0 writes dK = s R^T dK', group 1 dV.
        if (ok && mbar_wait_warp(smem_u32(&bar_dkv_full), 0, w, SITE_BWD_DKV)) {
            tc_fence_after();
            const bool valid = kvpos < T;
            // Keys past the sequence's length (or a tile with no query tile) get zeros.
            const bool live = !VL || (kvpos < len && n_hs > 0);
            // The tensors' row is a.dr wide: at head_dim 32 the kernel runs zero-padded to
            // 64 columns and stores only the first 32.
            const size_t orow = (((size_t)b * T + (valid ? kvpos : 0)) * a.Hkv + hkv) * a.dr;
#pragma unroll 1
            for (int c = 0; c < a.dr; c += 32) {
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

}  // namespace

int bwd_d64_q_box_rows() { return Bwd64::BH; }

cudaError_t launch_bwd_d64(int B, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const CUtensorMap& tdo, const CUtensorMap& tdq, const BwdArgs& a, cudaStream_t st) {
    auto kfn = a.seq_lens ? attn_bwd_d64_kernel<true> : attn_bwd_d64_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, Bwd64::SMEM);
    if (e != cudaSuccess) return e;
    BwdArgs ag = a;
    ag.group_major = (double)B * a.T * a.Hq * Bwd64::D * 4 > 48e6 && a.n_kvt <= 16 ? 1 : 0;
    const dim3 grid = ag.group_major ? dim3(a.n_kvt, a.Hkv, B) : dim3(a.Hkv, B, a.n_kvt);
    return launch_k(kfn, grid, dim3(Bwd64::THREADS), Bwd64::SMEM, st, tq, tk, tv, tdo, tdq, ag);
}

}  // namespace ne
