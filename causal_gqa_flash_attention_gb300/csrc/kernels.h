// kernels.h -- internal interface between the C-ABI layer (api.cu) and the kernel
// translation units.  Not part of the public ABI.
#pragma once
#include <cstdint>
#include <utility>
#include <cuda.h>
#include <cuda_runtime.h>

namespace ne {

// Device error codes written by bounded waits (first writer wins).  The low byte is
// the wait site; the host maps any nonzero word to NE_ERR_DEVICE_TIMEOUT.
enum WaitSite : int {
    SITE_FWD_Q = 0x101, SITE_FWD_KV_FULL, SITE_FWD_KV_EMPTY, SITE_FWD_K_READY, SITE_FWD_S_FULL,
    SITE_FWD_P_READY, SITE_FWD_O_DONE, SITE_FWD_DRAIN,
    SITE_BWD_KV = 0x201, SITE_BWD_QDO_FULL, SITE_BWD_QDO_EMPTY, SITE_BWD_Q_READY, SITE_BWD_S_FULL,
    SITE_BWD_DP_FULL, SITE_BWD_DS_READY, SITE_BWD_DS_FREE, SITE_BWD_DQ_FULL, SITE_BWD_DQ_FREE,
    SITE_BWD_DKV, SITE_BWD_DRAIN,
    SITE_SELFTEST = 0x301,
    SITE_PRO_EMPTY = 0x501, SITE_PRO_READY, SITE_PRO_FULL, SITE_PRO_ACC, SITE_PRO_DRAIN,
    // Not a wait: a rotated q/k value exceeded the fp16 range of the logit operand.
    SITE_RANGE = 0x401,
    // Not a wait: a decode call got a sequence length outside [1, T_max].
    SITE_DECODE_LEN = 0x402,
    // Not a wait: a variable-length call got a sequence length outside [0, T].
    SITE_VARLEN_LEN = 0x403,
};

// Length of sequence b: T when the call has no per-sequence lengths, else seq_lens[b]
// clamped to [0, T] (the caller reports a length outside that range).
__device__ __forceinline__ int seq_len(const int* seq_lens, int b, int T) {
    if (!seq_lens) return T;
    const int l = __ldg(seq_lens + b);
    return l < 0 ? 0 : (l > T ? T : l);
}
__device__ __forceinline__ bool seq_len_bad(const int* seq_lens, int b, int T) {
    if (!seq_lens) return false;
    const int l = __ldg(seq_lens + b);
    return l < 0 || l > T;
}

// Rows of the interleaved RoPE table the kernels read: at least this many (shorter
// sequences get a padded table), because the in-kernel angle-addition steps read
// table row RSTEP (at most 32).
constexpr int kRopeTableMinRows = 64;
inline int rope_table_rows(int T) { return T > kRopeTableMinRows ? T : kRopeTableMinRows; }

// Division by a runtime divisor d >= 1 of dividends below 2^31, without the divide
// sequence: q = (n * m) >> k with k = 31 + ceil(log2 d) and m = floor(2^k / d) + 1,
// computed once on the host.  With m d = 2^k + e, 0 < e <= d, the error n e / (d 2^k)
// stays below 1/d for n < 2^31 (n e < 2^31 d <= 2^k), so q = floor(n / d) exactly.
struct FastDiv {
    uint32_t m, k;
};
inline FastDiv make_fastdiv(uint32_t d) {
    uint32_t s = 0;
    while ((1ull << s) < d) ++s;
    const uint32_t k = 31 + s;
    return FastDiv{(uint32_t)((1ull << k) / d + 1), k};
}
__device__ __forceinline__ uint32_t fast_div(uint32_t n, FastDiv f) {
    return (uint32_t)(((uint64_t)n * f.m) >> f.k);
}

struct FwdArgs {
    void* o;                 // [B,T,Hq,D], input dtype
    float* lse;              // [B,Hq,T]
    const float2* rope;      // [T, D/2] (cos, sin)
    int B, T, Hq, G, n_qt;   // n_qt = ceil(T / 256): pairs of 128-row query tiles
    int n_units;             // B * Hq * n_qt work units of the persistent kernel
    float scale_log2;        // log2(e) / sqrt(D)
    int* err;
    unsigned long long timeout_ns;
    const int* seq_lens;     // [B] per-sequence lengths (positions at or past are padding), or null
    int dr;                  // the tensors' head_dim (bf16 32 runs the 64-wide kernel, zero-padded)
    FastDiv div_bh, div_hq;  // by B * Hq and by Hq (the unit decode)
    int save;                // training forward: store R Q (fp16) and zero the dQ' accumulator
};

struct BwdPreArgs {
    const void* o;           // [B,T,Hq,D]
    const void* dO;          // [B,T,Hq,D]
    float* delta;            // [B,Hq,T]
    float* dq_acc;           // [B,T,Hq,D] fp32, zeroed here (null: zeroed by the training forward)
    long long rows;          // B*T*Hq
    int T, Hq, D;
    const void* q;           // [B,T,Hq,D] bf16: rotated into q16 when q16 is set
    void* q16;               // [B,T,Hq,D] fp16 R Q, or nullptr
    const float2* rope;      // [T, D/2] (cos, sin), when q16 is set
    int* err;                // device error word (an fp16 overflow of R Q), may be null
    FastDiv div_hq, div_t;   // by Hq and by T (row = (b T + t) Hq + h)
    const int* seq_lens;     // [B] or null: Delta and R Q are zero at padding positions
    int rope_ld;             // (cos, sin) pairs per row of `rope` (>= D/2)
};

struct BwdArgs {
    const float* lse;        // [B,Hq,T]
    const float* delta;      // [B,Hq,T]
    float* dq_acc;           // [B,T,Hq,D] fp32 accumulator of R dQ / s
    void* dk;                // [B,T,Hkv,D]
    void* dv;                // [B,T,Hkv,D]
    const float2* rope;      // [T, D/2]
    int T, Hq, Hkv, G, n_kvt;
    float scale_log2;        // log2(e) / sqrt(D)
    float scale;             // 1 / sqrt(D)
    int* err;
    unsigned long long timeout_ns;
    const int* seq_lens;     // [B] or null: padding queries and keys get zero gradients
    int dr;                  // the tensors' head_dim (bf16 32 runs the 64-wide kernel, zero-padded)
    int group_major;         // set by the launcher: CTA order (key tile fastest) of attn_bwd_d64_kernel
};

// RMSNorm -> QKV projection -> RoPE prologue (qkv_prologue.cu), bf16 tensors.
struct ProArgs {
    const float* inv_rms;    // [M] 1 / root-mean-square of each token row
    void* q;                 // [B,T,Hq,D]
    void* k;                 // [B,T,Hkv,D]
    void* v;                 // [B,T,Hkv,D]
    const float2* rope;      // [>= T, D/2] (cos, sin)
    int M, T, dim, Hq, Hkv, D;   // M = B * T token rows
    int rotate;              // nonzero: RoPE on the query and key heads
    int* err;
    unsigned long long timeout_ns;
};

struct BwdPostArgs {
    const float* dq_acc;     // [B,T,Hq,D]
    void* dq;                // [B,T,Hq,D]
    const float2* rope;
    long long rows;          // B*T*Hq
    int T, Hq, D;
    float scale;
    FastDiv div_hq, div_t;   // by Hq and by T
    int rope_ld;             // (cos, sin) pairs per row of `rope` (>= D/2)
};

struct DecodeArgs {
    const void* q;           // [B, Hq, D]: query row of each sequence's newest token, unrotated
    const void* k;           // [B, Tmax, Hkv, D] key cache, unrotated
    const void* v;           // [B, Tmax, Hkv, D] value cache
    const int* seq_lens;     // [B]: cached positions of each sequence, newest token included
    void* o;                 // [B, Hq, D]
    float* lse;              // [B, Hq]
    float* part_o;           // [B, Hq, n_split, D] unnormalised chunk outputs (n_split > 1)
    float2* part_ml;         // [B, Hq, n_split] (running max in log2 units, sum) per chunk
    const float2* rope;      // [>= Tmax, D/2] (cos, sin)
    int B, Tmax, Hq, Hkv, G;
    int n_hgrp, n_split, chunk;   // from decode_plan()
    float scale_log2;        // log2(e) / sqrt(D)
    int* err;
};

// Work split of a decode call: hpc query heads per CTA (a divisor of G), n_hgrp = G / hpc
// head groups per kv head, and the positions cut into n_split chunks of `chunk` rows.
struct DecodePlan {
    int hpc, n_hgrp, n_split, chunk;
};
DecodePlan decode_plan(int B, int Tmax, int Hq, int Hkv);

// Programmatic dependent launch: every kernel of the library is launched with
// programmatic stream serialization (unless NE_ATTN_PDL=0), so it can be scheduled while
// the previous kernel on the stream drains.  Each kernel does its on-chip set-up first,
// then `griddepcontrol.wait` before its first global-memory access; kernels that own
// TMEM signal `launch_dependents` only after their allocation, so a dependent CTA never
// holds TMEM that a still-unallocated CTA of its predecessor needs.
bool pdl_enabled();

template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                     Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Prologue: tx maps x [M, dim] bf16 with (64 x 128) boxes, tw maps W [N, dim] bf16 with
// (64 x prologue_tile_n()) boxes.
int prologue_tile_n();
cudaError_t launch_qkv_prologue(const CUtensorMap& tx, const CUtensorMap& tw, const ProArgs& a, cudaStream_t st);
// The pass before the prologue GEMM: wg [N, dim] = w [N, dim] times gamma [dim] along
// each row (bf16), and inv_rms [M] = 1 / sqrt(mean of the squares of row m of x [M, dim]
// bf16 + eps); dim % 8 == 0.
cudaError_t launch_prologue_prep(const void* w, const void* gamma, void* wg, long long N, const void* x,
                                 float* inv_rms, int M, int dim, float eps, cudaStream_t st);
// Tile rows of the key/value tensor maps the forward kernel expects.
int fwd_kv_box_rows(bool tf32, int D);
// Launchers: return cudaSuccess or the launch error.
// ld: (cos, sin) pairs per table row (default D/2); pairs D/2 .. ld-1 get angle 0.
cudaError_t launch_rope_table(float* cos_out, float* sin_out, float2* interleaved, int T, int D,
                              double theta, cudaStream_t st, int ld = 0);
// `tq16` / `tdqz` map the backward workspace's fp16 R Q and fp32 dQ' accumulator; read only
// when a.save is set (bf16 head_dim 32/64, no per-sequence lengths).
cudaError_t launch_fwd(bool tf32, int D, int B, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, const CUtensorMap& to, const CUtensorMap& tq16,
                       const CUtensorMap& tdqz, const FwdArgs& a, cudaStream_t st);
cudaError_t launch_bwd_pre(bool tf32, const BwdPreArgs& a, cudaStream_t st);
// `tdq` maps the fp32 dQ accumulator (used by the head_dim-64 kernel).
cudaError_t launch_bwd(bool tf32, int D, int B, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdq, const BwdArgs& a,
                       cudaStream_t st);
cudaError_t launch_bwd_post(bool tf32, const BwdPostArgs& a, cudaStream_t st);
// head_dim 64, bf16: the half-step kernel; its Q and dO tensor maps use bwd_d64_q_box_rows() rows,
// and it adds dQ' into the accumulator through `tdq` (fp32 [B,T,Hq,D], 128-row boxes).
int bwd_d64_q_box_rows();
cudaError_t launch_bwd_d64(int B, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const CUtensorMap& tdo, const CUtensorMap& tdq, const BwdArgs& a, cudaStream_t st);
// Rows of the Q / dO tensor-map boxes the backward main kernel for (dtype, D) expects.
int bwd_q_box_rows(bool tf32, int D);
// fp32 tensors on TF32 tensor cores; its Q and dO tensor maps use bwd_tf32_q_box_rows() rows.
int bwd_tf32_q_box_rows();
cudaError_t launch_bwd_tf32(int D, int B, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const BwdArgs& a, cudaStream_t st);
cudaError_t launch_selftest_wait(int* err, unsigned long long timeout_ns, cudaStream_t st);
// Decode step: the chunk kernel and, when n_split > 1, the merge of the chunks.
cudaError_t launch_decode(bool f32, int D, const DecodePlan& p, const DecodeArgs& a, cudaStream_t st);

}  // namespace ne
