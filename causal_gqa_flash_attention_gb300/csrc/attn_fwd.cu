// attn_fwd.cu -- forward of causal GQA + RoPE attention on tcgen05 tensor cores.
//
// Method: FlashAttention tiling with an online softmax, so the T x T score matrix is
// never stored ("NanoEuler: C와 CUDA로 밑바닥부터 구축한 GPT-2 규모의 LLM", 커널 구현);
// RoPE on queries and keys and grouped-query heads (same page, 기술 사양); causal mask
// j <= i ("Tiny hackable CUDA language model implementation", Core Mechanics).
//
// Persistent kernel: one CTA per SM walks a static list of work units.  A unit is two
// consecutive 128-row query subtiles (u = 0, 1) of one (batch, query head); the units are
// numbered heaviest first (latest query rows) and dealt to the CTAs in snake order
// (round r goes left to right when r is even, right to left when odd), which balances
// the causal work about as well as greedy longest-first.  Inside a unit the CTA walks
// 64-key tiles up to the diagonal; every K/V tile is loaded and rotated once for both
// subtiles.  The pipeline does not drain between units: the next unit's Q is loaded and
// rotated, and its first S tiles are computed, while the softmax warps finish the
// current one, so a CTA pays its set-up (TMEM allocation, barrier set-up, first loads)
// once instead of once per unit.  Warp roles (480 threads):
//   warp 0       TMA producer: Q pairs into NQB buffers, K/V tiles into an NS-stage ring.
//   warp 1, 2    UMMA issuer of subtile 0 / 1 (warp 1 also owns the 512 TMEM columns);
//                the whole warp runs the loop, one elected lane issues.  Over the
//                subtile's tiles in order (across units), S(t+2) = Q'K'^T goes into S
//                buffer t % 2 right after PV(t) = P(t) V, two tiles ahead of the softmax.
//   warps 3, 12-14  RoPE: each unit's Q pair, then every K tile, in place (fp16 logit
//                operand; TF32: rounded fp32) and, for TF32, V transposed (TF32 UMMA reads
//                K-major operands only).
//   warps 4-7    softmax of subtile 0; warps 8-11 softmax of subtile 1.  Thread r owns
//                query row r (TMEM lane r): per tile it reads the S row from TMEM, updates
//                the running max m and sum l, writes P (bf16, or TF32 fp32) back over S,
//                rescales its O row when m grew by more than 2^8; at the end of a unit it
//                writes O / l (staged in the unit's Q buffer, stored by TMA) and LSE.
// TMEM: S buffers (u, b) at 64 * (2u + b), b = 0, 1; O_u at 256 + u * D.  A unit's first
// PV overwrites O_u; it needs P of the unit's first tile, which the softmax threads write
// only after their epilogue has read the previous unit's O_u.
// Every wait is bounded (WaitCtx); a CTA that gives up records an error code, drains
// its own copies and MMAs, frees its TMEM and exits.
#include <climits>
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
    static constexpr int BN = 64;                      // key rows per tile
    static constexpr int ROWB = D * ES;                // bytes per row
    static constexpr int NCH = ROWB / 128;             // 128-byte chunks per row
    static constexpr int EPC = 128 / ES;               // elements per chunk
    static constexpr int Q_BYTES = BM * ROWB;          // one subtile
    static constexpr int KV_BYTES = BN * ROWB;
    static constexpr int VT_BYTES = TF32 ? BN * ROWB : 0;
    static constexpr int STAGE_BYTES = 2 * KV_BYTES + VT_BYTES;
    static constexpr int QBUF = 2 * Q_BYTES;           // one Q buffer: both subtiles
    // Two Q buffers (the next unit's Q lands while this one runs) where that leaves at
    // least four K/V stages; otherwise one.
    static constexpr int NQB = (220 * 1024 - 2 * QBUF) / STAGE_BYTES >= 4 ? 2 : 1;
    static constexpr int NS_FIT = (220 * 1024 - NQB * QBUF) / STAGE_BYTES;
    static constexpr int NS = NS_FIT > 6 ? 6 : NS_FIT; // K/V pipeline stages
    static constexpr int SMEM = 1024 + NQB * QBUF + NS * STAGE_BYTES;
    static constexpr int O_COL = 256;                  // O_u at O_COL + u*D
    static constexpr int S_KSTEPS = ROWB / 32;         // 32-byte K-steps of S = Q K^T
    static constexpr int PV_KSTEPS = BN * ES / 32;     // K-steps of O += P V
    static constexpr int PV_ROWS = 32 / ES;            // key rows per PV K-step
    static constexpr uint32_t FMT_S = TF32 ? FMT_TF32 : FMT_F16;
    static constexpr uint32_t FMT_PV = TF32 ? FMT_TF32 : FMT_BF16;
    static constexpr int MODE = TF32 ? ROPE_TF32 : ROPE_F16;
    static constexpr int THREADS = 480;             // 15 warps
    static constexpr int ROPE_THREADS = 128;        // warps 3, 12, 13, 14
    static_assert(ROWB % 128 == 0, "rows must be whole 128-byte chunks");
    static_assert(D <= 128, "O subtiles must fit next to four S buffers in 512 TMEM columns");
    static_assert(NS >= 3, "need at least three K/V stages (S runs two tiles ahead)");
    static_assert(NQB == 1 || NS >= 4, "S of the next unit may wait inside a unit's loop: four stages");
    static_assert(SMEM <= 227 * 1024, "shared memory");
};

// Bytes of the zero tile the training forward stores into the dQ' accumulator (fp32:
// 128 rows x 32 columns per store).
constexpr int kZeroTileBytes = 128 * 128;

// TMEM column of S buffer `buf` (0/1) of subtile u.
__device__ __forceinline__ uint32_t s_col(int u, int buf) { return (uint32_t)((u * 2 + buf) * 64); }

// Zeroes rows zero_row .. ROWS-1 of a [ROWS x NCH*128 bytes] tile in the 128-byte-swizzled
// layout (padding past a sequence's length); thread t of NT.
template <int ROWS, int NCH, int NT>
__device__ __forceinline__ void zero_rows(uint8_t* base, int zero_row, int t) {
    for (int idx = t; idx < ROWS * NCH * 8; idx += NT) {
        const int c = idx / (ROWS * 8), rem = idx - c * (ROWS * 8), row = rem >> 3;
        if (row >= zero_row)
            *reinterpret_cast<uint4*>(base + c * ROWS * 128 + sw128_offset(row, rem & 7)) = make_uint4(0u, 0u, 0u, 0u);
    }
}

// TF32 only: Vt[d][r] = tf32(V[r][d]) for a [ROWS x D] fp32 tile, written K-major (key
// index contiguous, 32 keys per 128-byte chunk); NT threads.  Keys zero_row and later
// (padding) are written as zeros.
template <int D, int ROWS, int NT>
__device__ __forceinline__ void transpose_v_tf32(const uint8_t* src, uint8_t* dst, int t, int zero_row) {
    constexpr int UNITS = D * ROWS / 4;       // 16-byte units of the transposed tile
    // A warp takes 32 consecutive columns d of the same four keys: its reads of one key
    // row cover eight 16-byte chunks x four words (every bank once in the 128-byte
    // swizzle) and its 16-byte writes go to eight rows d per quarter-warp, whose chunk
    // positions the swizzle spreads.  (Keys fastest put a warp's reads on two banks.)
#pragma unroll 4
    for (int ul = t; ul < UNITS; ul += NT) {
        const int d = ul % D, u = ul / D;      // transposed row d, keys 4u .. 4u+3
        const int r0 = 4 * u;
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint8_t* s = src + (d >> 5) * ROWS * 128 + sw128_offset(r0 + k, (d & 31) >> 2) + (d & 3) * 4;
            w[k] = r0 + k < zero_row ? f32_to_tf32_rna(*reinterpret_cast<const float*>(s)) : 0u;
        }
        *reinterpret_cast<uint4*>(dst + (r0 >> 5) * D * 128 + sw128_offset(d, (r0 & 31) >> 2)) =
            make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// Per-row online-softmax state of one softmax thread.
struct RowState {
    float m_used;   // max (log2 domain, scaled) the exponentials are taken against
    float l;        // running sum of exp2(x * sl2 - m_used)
};

// One key tile of one softmax thread: mask, max, rescale decision (and O rescale),
// exp2, P written back over this tile's S buffer, p_ready arrival.  j is the tile's
// index within the unit, t its index in the subtile's sequence of tiles over all units
// (S buffer t % 2; barrier phases), g its index in the CTA's K/V sequence.  Returns
// false when a wait ran out.
template <bool TF32, int D>
__device__ __forceinline__ bool softmax_tile(uint32_t (&sr)[64], int j, int t, int g, int u, int qsub0, int qpos,
                                             uint32_t lt, float sl2, RowState& st, uint64_t* bar_kv_empty,
                                             uint64_t* bar_p_ready, const WaitCtx& w) {
    using C = FwdCfg<TF32, D>;
    const int kv0 = j * C::BN;
    if (kv0 + C::BN - 1 > qsub0) {   // tile crosses the diagonal: mask keys after the row
#pragma unroll
        for (int e = 0; e < C::BN; ++e)
            if (kv0 + e > qpos) sr[e] = __float_as_uint(kNegInf);
    }
    // Row max with three-input maxima over four independent chains (a single dependent
    // chain would serialise on the max latency).
    float m4[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) m4[k] = __uint_as_float(sr[k]);
#pragma unroll
    for (int e = 4; e < C::BN; e += 8)
#pragma unroll
        for (int k = 0; k < 4; ++k) m4[k] = fmax3(m4[k], __uint_as_float(sr[e + k]), __uint_as_float(sr[e + 4 + k]));
    const float mx = fmaxf(fmax3(m4[0], m4[1], m4[2]), m4[3]);
    const float m_tile = __fmul_rn(mx, sl2);   // (not contracted into a use below)
    // An fp16 operand that overflowed (|rotated q or k| > 65504) turns logits into inf or
    // NaN; a finite row max rules that out for the whole row (masked rows are -inf).
    if (!(fabsf(mx) < __int_as_float(0x7f800000)) && !(mx == kNegInf)) report_error(w.err, SITE_RANGE);
    // A row whose max grew by more than 2^8 rescales l and its O row; the others keep
    // their max (p <= 2^8 stays exact).  TMEM access is warp-collective, so a warp
    // rescales when any lane needs it (alpha = 1 elsewhere).  O is idle once the PV of
    // the previous tile is done (PV(t) needs this thread's P(t)); that tile's stage
    // release, which both issuers commit after their PV of it, says so.  (The release
    // barrier cannot have run a phase further: the stage's next tile is not loaded
    // before this release.)
    const bool need = j > 0 && m_tile > st.m_used + 8.f;
    if (j == 0) st.m_used = m_tile;
    if (__any_sync(0xffffffffu, need)) {
        const float alpha = need ? ex2(st.m_used - m_tile) : 1.f;
        st.l = __fmul_rn(st.l, alpha);   // (no FMA contraction with the sum below)
        if (need) st.m_used = m_tile;
        if (!mbar_wait_warp(smem_u32(&bar_kv_empty[(g - 1) % C::NS]), ((g - 1) / C::NS) & 1, w, SITE_FWD_O_DONE))
            return false;
        tc_fence_after();
        const uint32_t oc = C::O_COL + u * D;
#pragma unroll 1
        for (int c = 0; c < D; c += 16) {   // 16 columns at a time: two S tiles are live in registers
            uint32_t orow[16];
            tmem_ld16(lt + oc + c, orow);
            tmem_wait_ld16(orow);
#pragma unroll
            for (int e = 0; e < 16; ++e) orow[e] = __float_as_uint(__uint_as_float(orow[e]) * alpha);
            tmem_st16(lt + oc + c, orow);
        }
    }
    float s8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float2 s2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
    const float neg_m = -st.m_used;
    const uint32_t sc = lt + s_col(u, t & 1);
#pragma unroll
    for (int c = 0; c < C::BN; c += 32) {
        if constexpr (TF32) {
            // Two scores per instruction, as in the bf16 branch.
            uint32_t pk[32];
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
                const float2 x = __ffma2_rn(make_float2(__uint_as_float(sr[c + e]), __uint_as_float(sr[c + e + 1])),
                                            make_float2(sl2, sl2), make_float2(neg_m, neg_m));
                const float2 pp = make_float2(ex2(x.x), ex2(x.y));
                s2[(e >> 1) & 3] = __fadd2_rn(s2[(e >> 1) & 3], pp);
                pk[e] = f32_to_tf32_rna(pp.x);
                pk[e + 1] = f32_to_tf32_rna(pp.y);
            }
            tmem_st32(sc + c, pk);
        } else {
            // Two scores per instruction: the exponent argument and the partial sums run
            // as packed f32x2 FMA / add.
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
                const float2 x = __ffma2_rn(make_float2(__uint_as_float(sr[c + e]), __uint_as_float(sr[c + e + 1])),
                                            make_float2(sl2, sl2), make_float2(neg_m, neg_m));
                const float2 pp = make_float2(ex2(x.x), ex2(x.y));
                s2[(e >> 1) & 3] = __fadd2_rn(s2[(e >> 1) & 3], pp);
                pk[e >> 1] = pack_bf162(pp.x, pp.y);
            }
            tmem_st16(sc + (c >> 1), pk);
        }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) s8[2 * k] += s2[k].x + s2[k].y;
    st.l = __fadd_rn(st.l, ((s8[0] + s8[1]) + (s8[2] + s8[3])) + ((s8[4] + s8[5]) + (s8[6] + s8[7])));
    tmem_wait_st();
    tc_fence_before();
    mbar_arrive(smem_u32(&bar_p_ready[u * 2 + (t & 1)]));
    return true;
}

// Work unit U of the persistent schedule: (batch, query head, pair of 128-row query
// subtiles), numbered heaviest first (the pair holding the latest query rows).
struct FwdUnit {
    int b, h, q0;
    int len;       // the sequence's length (T without per-sequence lengths)
    int n_u[2];    // key tiles of subtile u (0: subtile at or past the length)
    int n_kv;      // key tiles the unit loads: max(n_u)
    int n_qsub;    // subtiles holding positions before the length (at least 1)
};

template <int BM, int BN, bool VL>
__device__ __forceinline__ FwdUnit fwd_unit(int U, const FwdArgs& a) {
    FwdUnit f;
    // Multiply-shift divisions: this decode is inlined in every role, and the generic
    // integer-divide sequences made up much of the kernel's code.
    const int rank = (int)fast_div((uint32_t)U, a.div_bh), rem = U - rank * (a.B * a.Hq);
    f.b = (int)fast_div((uint32_t)rem, a.div_hq);
    f.h = rem - f.b * a.Hq;
    f.q0 = (a.n_qt - 1 - rank) * 2 * BM;
    f.len = VL ? seq_len(a.seq_lens, f.b, a.T) : a.T;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const int qu = f.q0 + u * BM;
        f.n_u[u] = qu < f.len ? min(qu + BM - 1, f.len - 1) / BN + 1 : 0;
    }
    f.n_kv = max(f.n_u[0], f.n_u[1]);
    f.n_qsub = f.n_u[1] > 0 ? 2 : 1;
    return f;
}

// The k-th unit of this CTA, or -1 past the end: round k takes units k*G .. k*G+G-1
// (G CTAs), left to right for even k and right to left for odd k.
__device__ __forceinline__ int fwd_unit_index(int k, int n_units) {
    const int G = (int)gridDim.x, c = (int)blockIdx.x;
    const long long U = (long long)k * G + ((k & 1) ? G - 1 - c : c);
    return U < n_units ? (int)U : -1;
}

// Walks one subtile's tiles over the CTA's units in order, skipping units where the
// subtile lies beyond T: unit iteration k (-1 at the end), tile j of n, and kvb, the
// index of the unit's first K/V tile in the CTA's K/V sequence.
template <int BM, int BN, bool VL>
struct FwdWalk {
    int k, j, n, n_kv, kvb;
    __device__ __forceinline__ void load(int kk, int u, const FwdArgs& a) {
        const int U = fwd_unit_index(kk, a.n_units);
        k = U < 0 ? -1 : kk;
        if (U >= 0) {
            const FwdUnit f = fwd_unit<BM, BN, VL>(U, a);
            n = u == 0 ? f.n_u[0] : f.n_u[1];   // (a select: no local-memory array)
            n_kv = f.n_kv;
        }
    }
    __device__ __forceinline__ void skip_empty(int u, const FwdArgs& a) {
        while (k >= 0 && n == 0) {
            kvb += n_kv;
            load(k + 1, u, a);
        }
    }
    __device__ __forceinline__ void init(int u, const FwdArgs& a) {
        j = 0;
        kvb = 0;
        load(0, u, a);
        skip_empty(u, a);
    }
    __device__ __forceinline__ void advance(int u, const FwdArgs& a) {
        if (++j == n) {
            j = 0;
            kvb += n_kv;
            load(k + 1, u, a);
            skip_empty(u, a);
        }
    }
};

// VL: per-sequence lengths (padded batch).  Without them every length is T, rows past T
// arrive as TMA's zero fill, and the padding code below compiles away.
// SAVE (training forward, bf16 head_dim <= 64): the rotated fp16 queries R Q, which the
// backward uses as its logit and dK' operand, are stored from shared memory once rotated
// (tm_q16), and the backward's fp32 dQ' accumulator rows of each unit are zeroed by TMA
// stores of a zero tile (tm_dqz).  This kernel leaves HBM mostly idle, so the backward's
// preprocess pass no longer reads Q or writes these 37.8 MB (B16 T512 Hq12 D64).
template <bool TF32, int D, bool VL, bool SAVE>
__global__ void __launch_bounds__(480, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                    const __grid_constant__ CUtensorMap tm_q16, const __grid_constant__ CUtensorMap tm_dqz,
                    const FwdArgs a) {
    using C = FwdCfg<TF32, D>;
    static_assert(!SAVE || (!TF32 && D == 64 && !VL), "the training forward is the bf16 head_dim-64 kernel");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem;                               // NQB x (Q0 | Q1), later O staging
    uint8_t* sStage = sQ + C::NQB * C::QBUF;          // NS x (K | V | Vt)
    uint8_t* sZero = sStage + C::NS * C::STAGE_BYTES;  // SAVE: a zero tile [128 rows x 128 bytes]

    __shared__ __align__(8) uint64_t bar_final;
    __shared__ __align__(8) uint64_t bar_q_full[2], bar_q_ready[2], bar_q_empty[2];   // [Q buffer]
    __shared__ __align__(8) uint64_t bar_q16_read[2];  // [Q buffer] SAVE: the R Q store has read it
    __shared__ __align__(8) uint64_t bar_o_final[2], bar_o_staged[2];  // [subtile]
    __shared__ __align__(8) uint64_t bar_s_full[4], bar_p_ready[4];     // [u * 2 + buffer]
    __shared__ __align__(8) uint64_t bar_kv_full[C::NS], bar_k_ready[C::NS], bar_kv_empty[C::NS];
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int T = a.T;

    if (tid == 0) {
        mbar_init(smem_u32(&bar_final), 2);              // one commit per UMMA issuer
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&bar_q_full[i]), 1);
            mbar_init(smem_u32(&bar_q_ready[i]), C::ROPE_THREADS);
            mbar_init(smem_u32(&bar_q_empty[i]), 2);     // one arrival per subtile epilogue
            mbar_init(smem_u32(&bar_q16_read[i]), 1);    // the storing RoPE thread
            mbar_init(smem_u32(&bar_o_final[i]), 1);     // the last PV of a unit
            mbar_init(smem_u32(&bar_o_staged[i]), 128);
        }
        for (int i = 0; i < 4; ++i) {
            mbar_init(smem_u32(&bar_s_full[i]), 1);
            mbar_init(smem_u32(&bar_p_ready[i]), 128);
        }
        for (int s = 0; s < C::NS; ++s) {
            mbar_init(smem_u32(&bar_kv_full[s]), 1);
            mbar_init(smem_u32(&bar_k_ready[s]), C::ROPE_THREADS);
            mbar_init(smem_u32(&bar_kv_empty[s]), 2);    // one commit per UMMA issuer
        }
        abort_flag = 0;
        fence_mbar_init();
        // The tensor maps are kernel parameters, not outputs of an earlier kernel: fetch
        // them before the dependency wait, under the previous kernel's tail.
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        tma_prefetch_desc(&tm_o);
        if constexpr (SAVE) {
            tma_prefetch_desc(&tm_q16);
            tma_prefetch_desc(&tm_dqz);
        }
    }
    if constexpr (SAVE) {
        for (int i = tid; i < kZeroTileBytes / 16; i += C::THREADS)
            reinterpret_cast<uint4*>(sZero)[i] = make_uint4(0u, 0u, 0u, 0u);
        fence_proxy_async_smem();      // read by TMA stores after the barrier below
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
    griddep_wait();                // inputs of earlier kernels on the stream are visible
    const uint32_t tm = tmem_slot;
    const WaitCtx w{a.err, &abort_flag, a.timeout_ns};
    auto q_buf = [&](int k) { return sQ + (k % C::NQB) * C::QBUF; };
    auto stage_k = [&](int s) { return sStage + s * C::STAGE_BYTES; };
    auto stage_v = [&](int s) { return sStage + s * C::STAGE_BYTES + C::KV_BYTES; };
    auto stage_vt = [&](int s) { return sStage + s * C::STAGE_BYTES + 2 * C::KV_BYTES; };

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int issued = 0;                           // K/V tiles loaded so far
            int last_k0 = -1, last_k1 = -1;           // last unit loaded into Q buffer 0 / 1
            bool ok = true;
            for (int k = 0; ok; ++k) {
                const int U = fwd_unit_index(k, a.n_units);
                if (U < 0) break;
                const FwdUnit f = fwd_unit<C::BM, C::BN, VL>(U, a);
                const int qb = k % C::NQB;
                // The Q buffer is free once both epilogues of unit k - NQB stored their O.
                if (k >= C::NQB &&
                    !(ok = mbar_wait(smem_u32(&bar_q_empty[qb]), ((k / C::NQB) - 1) & 1, w, SITE_FWD_Q)))
                    break;
                if (VL && seq_len_bad(a.seq_lens, f.b, T)) report_error(a.err, SITE_VARLEN_LEN);
                const uint32_t qf = smem_u32(&bar_q_full[qb]);
                mbar_arrive_expect_tx(qf, f.n_qsub * C::Q_BYTES);
                for (int u = 0; u < f.n_qsub; ++u)
                    for (int c = 0; c < C::NCH; ++c)
                        tma_load_4d(smem_u32(q_buf(k) + u * C::Q_BYTES + c * C::BM * 128), &tm_q, qf, c * C::EPC,
                                    f.h, f.q0 + u * C::BM, f.b);
                // Training forward: the unit's dQ' accumulator rows are zeroed by stores of
                // the zero tile (fp32, 128 rows x 32 columns each), one after each K/V tile
                // request rather than all at once ahead of them.
                int zs = 0;
                const int n_zs = SAVE ? f.n_qsub * ((a.dr + 31) / 32) : 0;
                auto zero_store = [&]() {
                    if (zs < n_zs) {
                        const int per = (a.dr + 31) / 32;
                        tma_store_4d(&tm_dqz, smem_u32(sZero), (zs % per) * 32, f.h, f.q0 + (zs / per) * C::BM, f.b);
                        bulk_commit_group();
                        ++zs;
                    }
                };
                if (qb == 0) last_k0 = k;
                else last_k1 = k;
                const int hkv = f.h / a.G;
                for (int j = 0; j < f.n_kv; ++j) {
                    const int g = issued, s = g % C::NS;
                    if (g >= C::NS &&
                        !(ok = mbar_wait(smem_u32(&bar_kv_empty[s]), ((g / C::NS) - 1) & 1, w, SITE_FWD_KV_EMPTY)))
                        break;
                    const uint32_t full = smem_u32(&bar_kv_full[s]);
                    mbar_arrive_expect_tx(full, 2 * C::KV_BYTES);
                    for (int c = 0; c < C::NCH; ++c) {
                        tma_load_4d(smem_u32(stage_k(s) + c * C::BN * 128), &tm_k, full, c * C::EPC, hkv, j * C::BN,
                                    f.b);
                        tma_load_4d(smem_u32(stage_v(s) + c * C::BN * 128), &tm_v, full, c * C::EPC, hkv, j * C::BN,
                                    f.b);
                    }
                    ++issued;
                    if constexpr (SAVE) zero_store();
                }
                if constexpr (SAVE)
                    while (ok && zs < n_zs) zero_store();
            }
            // Teardown: every copy this CTA started must have landed before exit.
            if (last_k0 >= 0) mbar_wait_drain(smem_u32(&bar_q_full[0]), (last_k0 / C::NQB) & 1, w, SITE_FWD_DRAIN);
            if (last_k1 >= 0) mbar_wait_drain(smem_u32(&bar_q_full[1]), (last_k1 / C::NQB) & 1, w, SITE_FWD_DRAIN);
            for (int g = max(0, issued - C::NS); g < issued; ++g)
                mbar_wait_drain(smem_u32(&bar_kv_full[g % C::NS]), (g / C::NS) & 1, w, SITE_FWD_DRAIN);
            if constexpr (SAVE) bulk_wait_group0();   // the zero stores have completed
        }
    } else if (warp < 3) {
        // ------------------------------------------------------------ UMMA issuers
        // Each subtile has its own issuing warp (1 + u).  The whole warp runs the loop, so
        // the UMMA operands stay warp-uniform, and one elected lane issues each batch in
        // one branch: an election per UMMA, or a loop run by one lane alone (operands no
        // longer provably uniform), took several times the instructions.  This role's
        // steps are the kernel's critical path: clock64 traces put a 64-key tile at ~1.7K
        // cycles with the softmax work removed, almost all of it waits, elections and
        // bookkeeping between UMMA batches.  So the PV of a tile and the S the two-tile
        // window then admits go out as one batch when the S can go at once (its K' tile
        // rotated, its Q' already waited for).
        // Tiles are numbered t = 0, 1, ... over all units of the CTA; S(t) goes to S
        // buffer t % 2, two tiles ahead of the softmax, and overwrites P(t-2), whose PV
        // the same lane issued earlier (one thread's UMMAs execute in order).
        const int u = warp - 1;
        constexpr uint32_t id_s = idesc_make(C::FMT_S, 128, C::BN, false, false);
        constexpr uint32_t id_o = idesc_make(C::FMT_PV, 128, D, false, !TF32);
        // Descriptors are built once; a K-step, a stage or a Q buffer only moves the start
        // address.
        const uint64_t dq0 = sdesc(smem_u32(sQ + u * C::Q_BYTES), 16, 1024);
        const uint64_t dk0 = sdesc(smem_u32(stage_k(0)), 16, 1024);
        const uint64_t dv0 = TF32 ? sdesc(smem_u32(stage_vt(0)), 16, 1024)
                                  : sdesc(smem_u32(stage_v(0)), C::BN * 128, 1024);
        const uint32_t ocol = tm + C::O_COL + u * D;
        auto k_ready = [&](int g) {
            const bool r = mbar_wait_warp(smem_u32(&bar_k_ready[g % C::NS]), (g / C::NS) & 1, w, SITE_FWD_K_READY);
            tc_fence_after();
            return r;
        };
        int t_s = 0;                                  // S tiles issued
        int qr_next = 0;                              // first unit whose Q' this issuer has not waited for
        FwdWalk<C::BM, C::BN, VL> sw;                 // the next tile to issue S for
        sw.init(u, a);
        // S(t_s) of tile sw: the UMMAs and the commit (run by the elected lane).
        auto s_mmas = [&]() {
            const int g = sw.kvb + sw.j;
            const uint64_t dq = sdesc_add(dq0, (sw.k % C::NQB) * C::QBUF);
            const uint64_t dk = sdesc_add(dk0, (g % C::NS) * C::STAGE_BYTES);
            const uint32_t dcol = tm + s_col(u, t_s & 1);
#pragma unroll
            for (int ks = 0; ks < C::S_KSTEPS; ++ks) {
                const uint32_t byte = ks * 32;
                umma_ss<TF32>(dcol, sdesc_add(dq, (byte >> 7) * C::BM * 128 + (byte & 127)),
                              sdesc_add(dk, (byte >> 7) * C::BN * 128 + (byte & 127)), id_s, ks > 0);
            }
            umma_commit(smem_u32(&bar_s_full[u * 2 + (t_s & 1)]));
        };
        // Waits, in unit order, for the rotated Q of units qr_next .. upto.  A unit where
        // this subtile has no rows frees its Q buffer here (one of the buffer's two
        // releases; its softmax warps take no part): then the buffer's next phase needs
        // this issuer to have seen the current one, on every path, and neither this
        // issuer's nor the RoPE warps' waits on the Q barriers can fall a phase behind
        // (a run of units with no rows at all could otherwise cycle a buffer twice before
        // they looked).
        auto q_sync = [&](int upto) -> bool {
            for (; qr_next <= upto; ++qr_next) {
                const int U = fwd_unit_index(qr_next, a.n_units);
                if (U < 0) break;
                if (!mbar_wait_warp(smem_u32(&bar_q_ready[qr_next % C::NQB]), (qr_next / C::NQB) & 1, w, SITE_FWD_Q))
                    return false;
                const FwdUnit f = fwd_unit<C::BM, C::BN, VL>(U, a);
                if ((u == 0 ? f.n_u[0] : f.n_u[1]) == 0 && lane == 0)
                    mbar_arrive(smem_u32(&bar_q_empty[qr_next % C::NQB]));
                __syncwarp();
            }
            return true;
        };
        // The waits S(t_s) needs: Q' of its unit (and of every unit before it) and its
        // rotated K' tile.
        auto s_waits = [&]() -> bool {
            if (sw.j == 0 && !q_sync(sw.k)) return false;
            return k_ready(sw.kvb + sw.j);
        };
        int t = 0, g = 0;                             // PV tiles issued; K/V tiles passed
        // S runs at most two tiles ahead of PV, and an S wait must never depend on this
        // issuer's own later steps:
        // - unit: the Q of unit k lands once the epilogues of unit k - NQB have read O,
        //   which needs this issuer's PVs of that unit, so S stays within NQB - 1 units
        //   of the PV walk (k_cur);
        // - K/V tile: the tile g_s loads into the stage of tile g_s - NS, which this
        //   issuer has released only below g_rel (the PV walk's tiles, including those
        //   beyond its diagonal, which it releases without use), so g_s < g_rel + NS.
        //   (The producer loads every Q after the K/V tiles of the unit before it, so
        //   this bound also covers the Q load.)
        // A subtile with no tiles in several units in a row (its rows past the sequence)
        // would otherwise wait for the Q or K of a unit two or more ahead while still
        // holding the stages of the units between.
        auto may_issue = [&](int k_cur, int t_pv, int g_rel) {
            return sw.k >= 0 && t_s < t_pv + 2 && sw.k <= k_cur + (C::NQB - 1) && sw.kvb + sw.j < g_rel + C::NS;
        };
        // The PV walk: every K/V tile g of every unit in order, tile jp of unit kp, of
        // which the first np are this subtile's (the rest lie beyond its diagonal).
        int kp = 0, jp = 0, np = 0, nkv = 0;
        auto load_pv = [&]() -> bool {
            for (;; ++kp) {                           // units with no K/V tile load nothing
                const int U = fwd_unit_index(kp, a.n_units);
                if (U < 0) return false;
                const FwdUnit f = fwd_unit<C::BM, C::BN, VL>(U, a);
                np = u == 0 ? f.n_u[0] : f.n_u[1];
                nkv = f.n_kv;
                if (nkv > 0) return true;
            }
        };
        bool more = load_pv();
        bool ok = q_sync(more ? kp : INT_MAX);
        // One loop: every issue decision of the role in one short body, so the warp's code
        // stays in the instruction cache beside the softmax and RoPE warps' code.  Every
        // K/V stage is released by both issuers, in order; a tile beyond the subtile's
        // diagonal is released without use, but only once the stage really holds it
        // (k_ready), so the release never runs a phase ahead.
        while (ok) {
            if (may_issue(kp, t, g)) {                // an S on its own (start, unit change)
                if (!(ok = s_waits())) break;
                if (elect_one()) s_mmas();
                __syncwarp();
                ++t_s;
                sw.advance(u, a);
                continue;
            }
            if (!more) break;
            const uint32_t kv_empty = smem_u32(&bar_kv_empty[g % C::NS]);
            if (jp < np) {
                if (!(ok = mbar_wait_warp(smem_u32(&bar_p_ready[u * 2 + (t & 1)]), (t >> 1) & 1, w,
                                          SITE_FWD_P_READY)))
                    break;
                // The S this PV admits joins the batch if it needs no wait: its unit's Q'
                // was waited for and its K' tile is already rotated (a test, not a wait).
                bool fuse = may_issue(kp, t + 1, g + 1) && !(sw.j == 0 && qr_next <= sw.k);
                if (fuse) {
                    const int gs = sw.kvb + sw.j;
                    fuse = __all_sync(0xffffffffu, mbar_test(smem_u32(&bar_k_ready[gs % C::NS]), (gs / C::NS) & 1));
                }
                tc_fence_after();
                const uint64_t dv = sdesc_add(dv0, (g % C::NS) * C::STAGE_BYTES);
                const uint32_t pcol = tm + s_col(u, t & 1);
                const bool last = jp == np - 1;
                if (elect_one()) {
#pragma unroll
                    for (int ks = 0; ks < C::PV_KSTEPS; ++ks) {
                        // TF32: V^T [D x BN] K-major, 32 keys per chunk; bf16: V [BN x D]
                        // MN-major, PV_ROWS keys per K-step.
                        const uint32_t off =
                            TF32 ? ((ks * 32) >> 7) * D * 128 + ((ks * 32) & 127) : ks * C::PV_ROWS * 128;
                        umma_ts<TF32>(ocol, pcol + ks * 8, sdesc_add(dv, off), id_o, (jp > 0 || ks > 0) ? 1u : 0u);
                    }
                    if (last) umma_commit(smem_u32(&bar_o_final[u]));
                    umma_commit(kv_empty);
                    if (fuse) s_mmas();
                }
                __syncwarp();
                ++t;
                if (fuse) {
                    ++t_s;
                    sw.advance(u, a);
                }
            } else {
                if (!(ok = k_ready(g))) break;
                umma_commit_e(kv_empty);
            }
            ++g;
            if (++jp == nkv) {
                jp = 0;
                ++kp;
                more = load_pv();
                if (!(ok = q_sync(more ? kp : INT_MAX))) break;
            }
        }
        if (ok) q_sync(INT_MAX);
        umma_commit_e(smem_u32(&bar_final));
    } else if (warp == 3 || warp >= 12) {
        // ------------------------------------------------------------ RoPE on Q and K (+ V^T)
        // One branch for all four warps: a second inlined copy of this code measurably
        // slowed the kernel (instruction fetch).
        const int rt = lane + (warp == 3 ? 0 : 32 * (warp - 11));
        using RopeK = RopeTile<D, C::BN, C::ROPE_THREADS, C::MODE>;
        using RopeQ = RopeTile<D, C::BM, C::ROPE_THREADS, C::MODE>;
        RopeK rk;
        rk.init(rt, a.rope);
        RopeQ rq;
        rq.init(rt, a.rope);
        int g = 0;
        bool ok = true;
        int q16_pending = -1;                         // SAVE: unit whose R Q store may still be reading
        auto q16_release = [&]() {
            if (SAVE && rt == 0 && q16_pending >= 0) {
                bulk_wait_group_read0();
                mbar_arrive(smem_u32(&bar_q16_read[q16_pending % C::NQB]));
                q16_pending = -1;
            }
        };
        for (int k = 0; ok; ++k) {
            const int U = fwd_unit_index(k, a.n_units);
            if (U < 0) break;
            const FwdUnit f = fwd_unit<C::BM, C::BN, VL>(U, a);
            uint8_t* qbuf = q_buf(k);
            q16_release();
            // The table rows are fetched before the wait, so their latency overlaps it.
            float4 qa[RopeQ::F4], qc[RopeQ::F4], kn[RopeK::F4];
            rq.load_base(qa, f.q0, T, a.rope);
            rq.load_base(qc, f.q0 + C::BM, T, a.rope);
            rk.load_base(kn, 0, T, a.rope);
            if (!(ok = mbar_wait_warp(smem_u32(&bar_q_full[k % C::NQB]), (k / C::NQB) & 1, w, SITE_FWD_Q))) break;
            // Rows past the sequence's length (padding) are zeroed, so whatever the caller
            // left there never reaches an MMA.
            // One copy of the rotation code for both subtiles (instruction cache).
#pragma unroll 1
            for (int s2 = 0; s2 < f.n_qsub; ++s2) {
                float4 qb[RopeQ::F4];
#pragma unroll
                for (int e = 0; e < RopeQ::F4; ++e) qb[e] = s2 ? qc[e] : qa[e];
                rq.template apply<false>(qbuf + s2 * C::Q_BYTES, nullptr, qb, VL ? f.len - f.q0 - s2 * C::BM : C::BM);
            }
            fence_proxy_async_smem();
            if constexpr (SAVE) {
                // Every rotation of the unit is done (the four RoPE warps), then one thread
                // stores R Q.  The buffer later stages the unit's O: the epilogue waits for
                // bar_q16_read, which this thread arrives on once TMA has read the tile (at
                // its next unit, or after its loop): waiting here delayed the unit's S.
                named_bar_sync(1, C::ROPE_THREADS);
                if (rt == 0) {
                    for (int s2 = 0; s2 < f.n_qsub; ++s2)
                        tma_store_4d(&tm_q16, smem_u32(qbuf + s2 * C::Q_BYTES), 0, f.h, f.q0 + s2 * C::BM, f.b);
                    bulk_commit_group();
                    q16_pending = k;
                }
            }
            mbar_arrive(smem_u32(&bar_q_ready[k % C::NQB]));
            for (int j = 0; j < f.n_kv; ++j, ++g) {
                const int s = g % C::NS;
                float4 cur[RopeK::F4];
#pragma unroll
                for (int e = 0; e < RopeK::F4; ++e) cur[e] = kn[e];
                if (j + 1 < f.n_kv) rk.load_base(kn, (j + 1) * C::BN, T, a.rope);   // one tile early
                if (!(ok = mbar_wait_warp(smem_u32(&bar_kv_full[s]), (g / C::NS) & 1, w, SITE_FWD_KV_FULL))) break;
                const int kz = VL ? f.len - j * C::BN : C::BN;   // first padding row of the tile
                if constexpr (TF32) {
                    transpose_v_tf32<D, C::BN, C::ROPE_THREADS>(stage_v(s), stage_vt(s), rt, kz);
                } else if (VL && kz < C::BN) {
                    zero_rows<C::BN, C::NCH, C::ROPE_THREADS>(stage_v(s), kz, rt);
                }
                rk.template apply<false>(stage_k(s), nullptr, cur, kz);
                fence_proxy_async_smem();
                mbar_arrive(smem_u32(&bar_k_ready[s]));
            }
        }
        if constexpr (SAVE) {
            q16_release();
            if (rt == 0) bulk_wait_group0();   // the R Q stores have completed
        }
    } else if (warp >= 4 && warp < 12) {
        // ------------------------------------------------------------ softmax (subtile u)
        const int u = (warp - 4) >> 2;
        const int r = tid - 128 - 128 * u;            // query row = TMEM lane
        const uint32_t lt = tm + ((uint32_t)((warp & 3) * 32) << 16);
        const uint32_t o_col = C::O_COL + u * D;
        const float sl2 = a.scale_log2;
        int t = 0, n_epi = 0;                         // tiles and epilogues of this subtile so far
        int kvb = 0, n_kv = 0;                        // first K/V tile of the unit, its K/V tiles
        bool ok = true;
        for (int k = 0; ok; ++k, kvb += n_kv) {
            // Only what the tiles need stays live through the tile loop (the softmax
            // holds a 64-register S row); the epilogue decodes the unit again.
            int n, qsub0;
            {
                const int U = fwd_unit_index(k, a.n_units);
                if (U < 0) break;
                const FwdUnit f = fwd_unit<C::BM, C::BN, VL>(U, a);
                n = u == 0 ? f.n_u[0] : f.n_u[1];
                qsub0 = f.q0 + u * C::BM;
                n_kv = f.n_kv;
            }
            const int qb = k % C::NQB;
            if (n == 0) {                             // subtile at or past the sequence's length
                // (Its issuer frees the unit's Q buffer for it.)
                // Padding rows inside T: O = 0 and LSE = -inf (a softmax over no keys).
                const int qpos = qsub0 + r;
                if (VL && qpos < T) {
                    const FwdUnit f = fwd_unit<C::BM, C::BN, VL>(fwd_unit_index(k, a.n_units), a);
                    const size_t row = ((size_t)f.b * T + qpos) * a.Hq + f.h;
                    // The tensors' row is a.dr wide (bf16 head_dim 32 runs zero-padded to 64).
                    const int rb = a.dr * C::ES;
                    uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(a.o) + row * rb);
                    for (int e = 0; e < rb / 16; ++e) dst[e] = make_uint4(0u, 0u, 0u, 0u);
                    a.lse[((size_t)f.b * a.Hq + f.h) * T + qpos] = kNegInf;
                }
                continue;
            }
            const int qpos = qsub0 + r;
            RowState st{kNegInf, 0.f};
            for (int j = 0; j < n; ++j, ++t) {
                if (!(ok = mbar_wait_warp(smem_u32(&bar_s_full[u * 2 + (t & 1)]), (t >> 1) & 1, w, SITE_FWD_S_FULL)))
                    break;
                tc_fence_after();
                uint32_t sr[64];
                tmem_ld_cols<2>(lt + s_col(u, t & 1), sr);
                if (!(ok = softmax_tile<TF32, D>(sr, j, t, kvb + j, u, qsub0, qpos, lt, sl2, st, bar_kv_empty,
                                                 bar_p_ready, w)))
                    break;
            }
            if (!ok) break;
            // Epilogue: O / l staged (swizzled) in this subtile's half of the unit's Q
            // buffer (its S MMAs completed before its last PV did), stored by TMA; LSE =
            // natural log of the partition sum of the scaled logits.  The unit's last PV
            // has its own barrier, one phase per unit: on the per-PV barrier both of the
            // last two PVs may have completed before this wait starts, and the parity of
            // the older one would then name a phase that is still to come.
            if (!(ok = mbar_wait_warp(smem_u32(&bar_o_final[u]), n_epi & 1, w, SITE_FWD_O_DONE))) break;
            // Training forward: the R Q store of this unit has read the buffer O is staged in.
            if (SAVE && !(ok = mbar_wait_warp(smem_u32(&bar_q16_read[qb]), (k / C::NQB) & 1, w, SITE_FWD_O_DONE)))
                break;
            tc_fence_after();
            const FwdUnit f = fwd_unit<C::BM, C::BN, VL>(fwd_unit_index(k, a.n_units), a);
            uint8_t* sQu = q_buf(k) + u * C::Q_BYTES;
            // Padding rows (past the sequence's length) store O = 0 and LSE = -inf; their
            // accumulators are finite (their Q, and the padding K and V, were zeroed).
            const bool live = !VL || qpos < f.len;
            const float inv_l = live ? 1.f / st.l : 0.f;
#pragma unroll
            for (int c = 0; c < D; c += 32) {
                uint32_t orow[32];
                tmem_ld_cols<1>(lt + o_col + c, orow);
                if constexpr (TF32) {
                    uint8_t* dst = sQu + (c >> 5) * C::BM * 128;
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        *reinterpret_cast<float4*>(dst + sw128_offset(r, kk)) =
                            make_float4(__uint_as_float(orow[4 * kk]) * inv_l, __uint_as_float(orow[4 * kk + 1]) * inv_l,
                                        __uint_as_float(orow[4 * kk + 2]) * inv_l,
                                        __uint_as_float(orow[4 * kk + 3]) * inv_l);
                } else {
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 32; e += 2)
                        pk[e >> 1] = pack_bf162(__uint_as_float(orow[e]) * inv_l, __uint_as_float(orow[e + 1]) * inv_l);
                    uint8_t* dst = sQu + (c >> 6) * C::BM * 128;
                    const int u0 = (c & 63) >> 3;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        *reinterpret_cast<uint4*>(dst + sw128_offset(r, u0 + kk)) =
                            make_uint4(pk[4 * kk], pk[4 * kk + 1], pk[4 * kk + 2], pk[4 * kk + 3]);
                }
            }
            tc_fence_before();
            fence_proxy_async_smem();
            mbar_arrive(smem_u32(&bar_o_staged[u]));
            if (qpos < T)
                a.lse[((size_t)f.b * a.Hq + f.h) * T + qpos] =
                    live ? (st.m_used + log2f(st.l)) * 0.6931471805599453f : kNegInf;
            bool stored = true;
            if (r == 0) {
                stored = mbar_wait(smem_u32(&bar_o_staged[u]), n_epi & 1, w, SITE_FWD_O_DONE);
                if (stored) {
                    for (int c = 0; c < C::NCH; ++c)
                        tma_store_4d(&tm_o, smem_u32(sQu + c * C::BM * 128), c * C::EPC, f.h, qsub0, f.b);
                    bulk_commit_group();
                    bulk_wait_group_read0();          // the buffer may take the next Q
                    mbar_arrive(smem_u32(&bar_q_empty[qb]));
                }
            }
            if (!(ok = __all_sync(0xffffffffu, stored))) break;   // the warp leaves the loop together
            ++n_epi;
        }
        if (r == 0) bulk_wait_group0();               // the last O store has completed
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

template <bool TF32, int D, bool VL, bool SAVE = false>
cudaError_t launch_fwd_t(int B, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const CUtensorMap& to, const CUtensorMap& tq16, const CUtensorMap& tdqz, const FwdArgs& a,
                         cudaStream_t st) {
    using C = FwdCfg<TF32, D>;
    auto kfn = attn_fwd_kernel<TF32, D, VL, SAVE>;
    constexpr int smem = C::SMEM + (SAVE ? kZeroTileBytes : 0);
    static_assert(smem <= 227 * 1024, "shared memory");
    cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    // One CTA per SM (the shared memory allows no second), each walking its units.
    dim3 grid(a.n_units < sms ? a.n_units : sms);
    return launch_k(kfn, grid, dim3(C::THREADS), smem, st, tq, tk, tv, to, tq16, tdqz, a);
}

}  // namespace

int fwd_kv_box_rows(bool tf32, int D) { return 64; }

template <bool VL>
cudaError_t launch_fwd_vl(bool tf32, int D, int B, const CUtensorMap& tq, const CUtensorMap& tk,
                          const CUtensorMap& tv, const CUtensorMap& to, const CUtensorMap& tq16,
                          const CUtensorMap& tdqz, const FwdArgs& a, cudaStream_t st) {
    if (!tf32) {
        // head_dim 32 runs the 64-wide kernel: its 128-byte TMA boxes read the upper 32
        // columns as zeros and the O store clips them.
        if (D == 64 || D == 32) return launch_fwd_t<false, 64, VL>(B, tq, tk, tv, to, tq16, tdqz, a, st);
        if (D == 128) return launch_fwd_t<false, 128, VL>(B, tq, tk, tv, to, tq16, tdqz, a, st);
    } else {
        if (D == 32) return launch_fwd_t<true, 32, VL>(B, tq, tk, tv, to, tq16, tdqz, a, st);
        if (D == 64) return launch_fwd_t<true, 64, VL>(B, tq, tk, tv, to, tq16, tdqz, a, st);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_fwd(bool tf32, int D, int B, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, const CUtensorMap& to, const CUtensorMap& tq16,
                       const CUtensorMap& tdqz, const FwdArgs& a, cudaStream_t st) {
    if (a.save) {
        if (tf32 || !(D == 64 || D == 32) || a.seq_lens) return cudaErrorInvalidValue;
        return launch_fwd_t<false, 64, false, true>(B, tq, tk, tv, to, tq16, tdqz, a, st);
    }
    return a.seq_lens ? launch_fwd_vl<true>(tf32, D, B, tq, tk, tv, to, tq16, tdqz, a, st)
                      : launch_fwd_vl<false>(tf32, D, B, tq, tk, tv, to, tq16, tdqz, a, st);
}

}  // namespace ne
