/*
 * neattn.h -- C ABI of libneattn: fused causal grouped-query self-attention with
 * rotary position embeddings (RoPE), forward and backward, on sm_103a tensor cores.
 *
 * What is computed (page title, section):
 *   - causal self-attention, each position attending to itself and earlier
 *     positions ("Tiny hackable CUDA language model implementation", Core Mechanics,
 *     causal self-attention bullet);
 *   - grouped-query attention: Hkv key/value heads, each shared by G = Hq / Hkv
 *     query heads; query head h reads key/value head h / G ("NanoEuler: C와 CUDA로
 *     밑바닥부터 구축한 GPT-2 규모의 LLM", 기술 사양, GQA bullet, and 모델 구성);
 *   - RoPE on queries and keys (same page, 기술 사양, RoPE bullet): adjacent pairs
 *     (2i, 2i+1) of a row at position t are rotated by the angle t * theta^(-2i/D),
 *     (x0, x1) -> (x0 cos - x1 sin, x0 sin + x1 cos), positions t = 0 .. T-1;
 *   - FlashAttention-style tiling with an online softmax, so the T x T score matrix
 *     is never stored (same page, 커널 구현);
 *   - the hand-written backward pass (same page, 검증 및 안정성).
 *   O = softmax(s * Q' K'^T + causal mask) V with s = 1/sqrt(D), Q' = R Q, K' = R K.
 *   LSE[b,h,t] = natural log of sum_j exp(s * q'_t . k'_j) over j <= t.
 *
 * Layouts (all row-major, dense, no padding):
 *   q, o, dO, dq : [B, T, Hq,  D]      k, v, dk, dv : [B, T, Hkv, D]
 *   lse          : [B, Hq, T] fp32     rope tables  : [T, D/2] fp32
 * The bf16 entry points take __nv_bfloat16 tensors and compute with bf16 tensor-core
 * inputs and fp32 accumulation; the *_f32 entry points take fp32 tensors and use TF32
 * tensor cores with fp32 accumulation.  Outputs have the input dtype, lse is fp32.
 *
 * Supported shapes: B >= 0, T >= 0 (any T, ragged tails included), Hq % Hkv == 0,
 * D in {32, 64, 128} for bf16 and {32, 64} for f32 (others return NE_ERR_UNSUPPORTED;
 * bf16 32 runs on the head_dim-64 kernels with zero-padded columns; fp32 128 does not
 * fit the kernels' shared memory: a 128-row fp32 tile of 128 columns is 64 KB),
 * B * T * max(Hq, 1) * D < 2^31.  Every tensor pointer must be 16-byte aligned.
 *
 * Ownership: the caller owns every tensor and the backward workspace.  The library
 * owns only small per-device caches (RoPE tables per (D, theta), one device error
 * word), created on first use and released by ne_shutdown().  A table serves every T up
 * to its length; a call with a longer T builds one of twice the length (or T's), and the
 * shorter table is kept until ne_shutdown() (kernels in flight may still read it), so a
 * caller whose T grows step by step (a growing KV cache) holds at most about twice the
 * largest table (T * D/2 * 8 bytes).  All pointers are device
 * pointers unless stated otherwise.
 *
 * Streams: every call enqueues its kernels on `stream` (NULL = legacy default stream)
 * and returns without synchronising, except that a call that needs a new or longer RoPE
 * table for its (device, D, theta) builds it and synchronises `stream` once; make such
 * a call (the longest T) before any stream capture.  Argument errors return before anything
 * is enqueued.  Device-side failures (a bounded wait inside a kernel that ran out,
 * see ne_get_device_error) are reported asynchronously.
 *
 * Threading: calls are thread-safe; ne_last_error() is per thread.
 */
#ifndef NEATTN_H
#define NEATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream. */
typedef struct CUstream_st* ne_stream_t;

typedef enum {
    NE_OK = 0,
    NE_ERR_INVALID_ARG = 1,     /* bad pointer, shape or size; nothing was enqueued */
    NE_ERR_UNSUPPORTED = 2,     /* valid but not implemented (e.g. head_dim) */
    NE_ERR_CUDA = 3,            /* a CUDA runtime/driver call failed; see ne_last_error() */
    NE_ERR_DEVICE_TIMEOUT = 4,  /* a kernel's bounded wait ran out (ne_get_device_error) */
    NE_ERR_NO_DEVICE = 5        /* no CUDA device, or not an sm_103 device */
} ne_status;

/* RoPE cos/sin table (the rotation of the RoPE bullet, same page): for t < T and
 * i < D/2, cos_out[t*(D/2)+i] = cos(t * theta^(-2i/D)) and likewise sin_out.  Angles
 * are formed in fp64 on the device and stored as fp32.  cos_out/sin_out: device
 * pointers to T*D/2 floats each.  D must be even and > 0, theta > 0. */
ne_status ne_rope_table(float* cos_out, float* sin_out, int T, int D, double theta,
                        ne_stream_t stream);

/* Forward (커널 구현: tiling + online softmax).  q [B,T,Hq,D], k and v [B,T,Hkv,D] in,
 * o [B,T,Hq,D] and lse [B,Hq,T] (fp32) out.  bf16 tensors. */
ne_status ne_attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                      int B, int T, int Hq, int Hkv, int D, double rope_theta,
                      ne_stream_t stream);
/* Same with fp32 tensors on TF32 tensor cores. */
ne_status ne_attn_fwd_f32(const float* q, const float* k, const float* v, float* o, float* lse,
                          int B, int T, int Hq, int Hkv, int D, double rope_theta,
                          ne_stream_t stream);

/* Bytes of device workspace ne_attn_bwd needs for this shape (0 on a bad shape).
 * Layout: Delta fp32 [B,Hq,T] at offset 0, then (256-byte aligned) the fp32 dQ
 * accumulator [B,T,Hq,D], then (256-byte aligned) the rotated queries R Q as fp16
 * [B,T,Hq,D] (used by the bf16 head_dim-64 kernel).  All are rewritten by every call. */
size_t ne_attn_bwd_workspace_size(int B, int T, int Hq, int Hkv, int D);

/* Backward (검증 및 안정성: the hand-written backward), the vector-Jacobian product of
 * <dO, O> for the forward above.  Inputs q, k, v, o, lse, dO as the forward wrote or
 * read them; outputs dq [B,T,Hq,D], dk and dv [B,T,Hkv,D] in the input dtype.  The
 * gradient of every kv head is summed over its G query heads.  `workspace` must hold
 * ne_attn_bwd_workspace_size() bytes (256-byte aligned); it is caller-owned scratch. */
ne_status ne_attn_bwd(const void* q, const void* k, const void* v, const void* o,
                      const float* lse, const void* dO, void* dq, void* dk, void* dv,
                      int B, int T, int Hq, int Hkv, int D, double rope_theta,
                      void* workspace, size_t workspace_bytes, ne_stream_t stream);
ne_status ne_attn_bwd_f32(const float* q, const float* k, const float* v, const float* o,
                          const float* lse, const float* dO, float* dq, float* dk, float* dv,
                          int B, int T, int Hq, int Hkv, int D, double rope_theta,
                          void* workspace, size_t workspace_bytes, ne_stream_t stream);

/* Training pair: the forward and backward of one layer sharing that layer's backward
 * workspace (the pages train with the forward and backward kernels of 커널 구현 and
 * 검증 및 안정성, same page).  ne_attn_fwd_train computes what ne_attn_fwd computes and,
 * for bf16 head_dim 32 and 64, also fills the workspace for the later backward: the
 * rotated queries R Q as fp16 and a zeroed fp32 dQ accumulator (the forward rotates the
 * queries anyway, and its HBM is mostly idle).  ne_attn_bwd_train then computes what
 * ne_attn_bwd computes while skipping that work, so its preprocess pass only forms Delta.
 * Same arguments as ne_attn_fwd / ne_attn_bwd plus the workspace (as for ne_attn_bwd:
 * ne_attn_bwd_workspace_size() bytes, 256-byte aligned, caller-owned).  Contract: the
 * backward must get the same workspace, the same q, k, v, shape and theta, and nothing
 * may write the workspace between the two calls (one workspace per layer in flight).
 * For f32 tensors and head_dim 128 the pair is exactly ne_attn_fwd + ne_attn_bwd (the
 * forward leaves the workspace alone and the backward fills it itself). */
ne_status ne_attn_fwd_train(const void* q, const void* k, const void* v, void* o, float* lse,
                            void* workspace, size_t workspace_bytes, int B, int T, int Hq, int Hkv, int D,
                            double rope_theta, ne_stream_t stream);
ne_status ne_attn_fwd_train_f32(const float* q, const float* k, const float* v, float* o, float* lse,
                                void* workspace, size_t workspace_bytes, int B, int T, int Hq, int Hkv,
                                int D, double rope_theta, ne_stream_t stream);
ne_status ne_attn_bwd_train(const void* q, const void* k, const void* v, const void* o,
                            const float* lse, const void* dO, void* dq, void* dk, void* dv,
                            int B, int T, int Hq, int Hkv, int D, double rope_theta,
                            void* workspace, size_t workspace_bytes, ne_stream_t stream);
ne_status ne_attn_bwd_train_f32(const float* q, const float* k, const float* v, const float* o,
                                const float* lse, const float* dO, float* dq, float* dk, float* dv,
                                int B, int T, int Hq, int Hkv, int D, double rope_theta,
                                void* workspace, size_t workspace_bytes, ne_stream_t stream);

/* Variable-length sequences in a padded batch: the supervised fine-tuning data of
 * "NanoEuler: C와 CUDA로 밑바닥부터 구축한 GPT-2 규모의 LLM" (2단계 학습 프로세스, SFT bullet)
 * pads sequences of different lengths to one T, and the padding must not take part.
 * Same tensors and layouts as ne_attn_fwd / ne_attn_bwd, plus
 *   seq_lens [B] int32 (device memory, 4-byte aligned): sequence b occupies positions
 *            0 .. seq_lens[b]-1 of row b; positions seq_lens[b] .. T-1 are padding.
 * The valid positions of sequence b get the results of the same call on that sequence
 * alone with T = seq_lens[b] (RoPE positions start at 0 in every row).
 * Padding never takes part: no valid query attends to a padding key, padding queries
 * and keys get zero outputs and gradients (o, dq, dk, dv = 0) and lse = -inf (the log of
 * an empty sum).  Padding entries of q and k are not read as values (the kernels zero
 * them before any MMA); padding entries of v and dO must be finite (e.g. zeros, as
 * padding usually is): they meet zero weights inside tensor-core products, where a NaN
 * or infinity would still propagate.  A length outside [0, T] is clamped on the device
 * and reported by ne_get_device_error() as NE_ERR_INVALID_ARG; a length of 0 is an
 * empty sequence.  The backward takes the workspace of ne_attn_bwd. */
ne_status ne_attn_fwd_varlen(const void* q, const void* k, const void* v, const int* seq_lens, void* o,
                             float* lse, int B, int T, int Hq, int Hkv, int D, double rope_theta,
                             ne_stream_t stream);
ne_status ne_attn_fwd_varlen_f32(const float* q, const float* k, const float* v, const int* seq_lens,
                                 float* o, float* lse, int B, int T, int Hq, int Hkv, int D,
                                 double rope_theta, ne_stream_t stream);
ne_status ne_attn_bwd_varlen(const void* q, const void* k, const void* v, const void* o,
                             const float* lse, const void* dO, const int* seq_lens, void* dq, void* dk,
                             void* dv, int B, int T, int Hq, int Hkv, int D, double rope_theta,
                             void* workspace, size_t workspace_bytes, ne_stream_t stream);
ne_status ne_attn_bwd_varlen_f32(const float* q, const float* k, const float* v, const float* o,
                                 const float* lse, const float* dO, const int* seq_lens, float* dq,
                                 float* dk, float* dv, int B, int T, int Hq, int Hkv, int D,
                                 double rope_theta, void* workspace, size_t workspace_bytes,
                                 ne_stream_t stream);

/* Backward that allocates nothing (there is no counterpart of this call on the
 * pages: it is a deployment convenience).  Same computation, arguments and outputs
 * as ne_attn_bwd for bf16 tensors, but without a workspace argument: its scratch
 * (RoPE table, Delta, fp32 dQ accumulator, rotated queries) lives in one file-scope
 * device array of 48 MiB that every GPU loading the library keeps until the process exits.  It is for
 * callers that cannot call cudaMalloc at this point: code that runs while a stream
 * is being captured into a CUDA graph (allocation is not allowed there), runtimes
 * whose own allocator already owns the device's free memory, or real-time loops that
 * forbid allocation after start-up.  It calls no cudaMalloc, cudaFree or allocating
 * library routine.
 *  - Limit: round256(max(T,64)*P*8) + round256(B*Hq*T*4) + round256(B*T*Hq*D*4)
 *    + (D <= 64 ? B*T*Hq*D*2 : 0) <= 50331648 bytes, P = max(D,64)/2 (the GPU-pipeline shape B=16 T=512
 *    Hq=12 D=64 uses 38.3 MB); larger shapes
 *    return NE_ERR_INVALID_ARG before anything is enqueued.
 *  - The first call on a device looks up the array's device address (once per
 *    device, with that device current); make that first call before any stream
 *    capture.
 *  - All calls share the one array, which keeps the last call's contents; every call
 *    rewrites what it reads.  Calls whose kernels overlap on the GPU (two streams, or
 *    two threads) race on the scratch and produce wrong gradients: serialise them.
 *  - Device-side errors (a bounded wait that ran out, or an MMA operand beyond the
 *    fp16 range: a rotated q or k, or dS) are recorded in a second file-scope device
 *    word beside the scratch, not in the allocated word ne_get_device_error() reads;
 *    read them with ne_noalloc_get_device_error(). */
ne_status ne_attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                              const float* lse, const void* dO, void* dq, void* dk, void* dv,
                              int B, int T, int Hq, int Hkv, int D, double rope_theta,
                              ne_stream_t stream);
/* The error report of the allocation-free calls (no counterpart on the pages).
 * Synchronises `stream`, then reads and clears the current device's static error word
 * of ne_attn_bwd_noalloc; allocates nothing.  Returns NE_ERR_INVALID_ARG when an MMA
 * operand left the fp16 range (the outputs of that call are invalid),
 * NE_ERR_DEVICE_TIMEOUT when a bounded wait ran out, NE_ERR_CUDA when the
 * synchronisation failed, else NE_OK.  Like the scratch, the word is shared by all
 * calls on a device. */
ne_status ne_noalloc_get_device_error(ne_stream_t stream);

/* Decode step over a key/value cache: the newest token of every sequence attends to
 * all cached positions of its sequence.  For sequence b with len = seq_lens[b] the
 * newest token sits at position len - 1, and the result is row len - 1 of the causal
 * attention above over positions 0 .. len - 1: the same RoPE, grouped heads, scale and
 * LSE convention.  The CUDA engine of "NanoEuler: C와 CUDA로 밑바닥부터 구축한 GPT-2 규모의
 * LLM" (CUDA 엔진 및 성능) runs inference as well as training, and its chat command
 * generates token by token ("NanoEuler – 순수 C/CUDA로 처음부터 만든 GPT-2 규모 언어
 * 모델", Code Example).
 *   q        [B, Hq, D]        query rows of the newest tokens, unrotated (in)
 *   k_cache  [B, T_max, Hkv, D] keys, unrotated, positions 0 .. len-1 valid; the newest
 *                              token's key must already be written at len - 1 (in)
 *   v_cache  [B, T_max, Hkv, D] values, same positions (in)
 *   seq_lens [B] int32         1 <= len <= T_max (device memory, 4-byte aligned) (in)
 *   o        [B, Hq, D]        output rows, input dtype (out)
 *   lse      [B, Hq] fp32      natural log of the softmax denominator (out)
 * Rows at positions >= len are never read.  `workspace` holds
 * ne_attn_decode_workspace_size() bytes (256-byte aligned, caller-owned, rewritten by
 * every call); it may be NULL when that size is 0.  A seq_lens entry outside
 * [1, T_max] is clamped on the device and reported by ne_get_device_error() as
 * NE_ERR_INVALID_ARG; that sequence's outputs are then invalid.
 * Supported: D in {64, 128} (bf16) or {32, 64} (f32), Hq % Hkv == 0, 1 <= B <= 65535,
 * 1 <= T_max <= 2^30; B == 0 is a no-op.  Arithmetic is fp32 throughout (no tensor cores: one
 * query row per head is a matrix-vector product, bound by the read of the cache). */
size_t ne_attn_decode_workspace_size(int B, int T_max, int Hq, int Hkv, int D);
ne_status ne_attn_decode(const void* q, const void* k_cache, const void* v_cache,
                         const int* seq_lens, void* o, float* lse, int B, int T_max, int Hq,
                         int Hkv, int D, double rope_theta, void* workspace,
                         size_t workspace_bytes, ne_stream_t stream);
ne_status ne_attn_decode_f32(const float* q, const float* k_cache, const float* v_cache,
                             const int* seq_lens, float* o, float* lse, int B, int T_max,
                             int Hq, int Hkv, int D, double rope_theta, void* workspace,
                             size_t workspace_bytes, ne_stream_t stream);

/* The steps before attention in every layer, fused into one tensor-core GEMM ("NanoEuler:
 * C와 CUDA로 밑바닥부터 구축한 GPT-2 규모의 LLM", 기술 사양: RMSNorm as pre-normalization
 * without bias, RoPE on queries and keys; the model has no biases): for token row m of x,
 *   r_m = sqrt(mean_c x_mc^2 + eps),   y_m = W (x_m o gamma) / r_m,
 * split into query heads (rows 0 .. Hq*D-1 of W), key heads (next Hkv*D rows) and value
 * heads (last Hkv*D rows).  With rotate != 0 the query and key heads are rotated by the
 * RoPE of the attention calls (position m mod T, theta rope_theta); the attention calls
 * take unrotated q and k (they rotate as their tiles load), so the form they consume is
 * rotate = 0.
 *   x     [B, T, dim] bf16 (in)          gamma [dim] bf16 (in)
 *   w     [(Hq + 2 Hkv) * D, dim] bf16, row-major (in: row n holds output feature n)
 *   q     [B, T, Hq, D] bf16 (out)       k, v  [B, T, Hkv, D] bf16 (out)
 *   workspace: caller-owned device scratch of ne_qkv_prologue_workspace_size(B, T, dim,
 *              Hq, Hkv, D) bytes, 256-byte aligned; each call rewrites it with
 *              W diag(gamma) (bf16) and the reciprocal root-mean-square of every token row
 *              (fp32), formed by two small passes before the GEMM.
 * Arithmetic: bf16 tensor-core products with fp32 accumulation; the gain is folded into
 * the weights (W diag(gamma), rounded to bf16, formed on the device by each call), the
 * root-mean-square is fp32.  Supported: D in {32, 64, 128}, dim a multiple of 8,
 * Hq % Hkv == 0, B*T*dim and B*T*(Hq + 2 Hkv)*D below 2^31, eps >= 0.  Pointers 16-byte
 * aligned.  A call that needs a new or longer RoPE table builds it and synchronises
 * `stream` once (as the attention calls do). */
size_t ne_qkv_prologue_workspace_size(int B, int T, int dim, int Hq, int Hkv, int D);
ne_status ne_qkv_prologue(const void* x, const void* gamma, const void* w, void* q, void* k, void* v,
                          int B, int T, int dim, int Hq, int Hkv, int D, double eps,
                          double rope_theta, int rotate, void* workspace, size_t workspace_bytes,
                          ne_stream_t stream);

/* Human-readable name of a status code (static string). */
const char* ne_status_string(ne_status s);
/* Detail of the last error on the calling thread ("" if none). */
const char* ne_last_error(void);

/* Synchronises `stream`, then reads and clears the current device's error word.
 * Returns NE_ERR_DEVICE_TIMEOUT if a kernel's bounded wait ran out since the last
 * check (the kernel then skipped the rest of its work and its outputs are invalid),
 * NE_ERR_CUDA if the synchronisation failed, else NE_OK. */
ne_status ne_get_device_error(ne_stream_t stream);

/* Wall-clock limit of every bounded wait inside the kernels (default 2000 ms, or
 * NE_ATTN_TIMEOUT_MS from the environment).  0 restores the default. */
void ne_set_wait_timeout_ms(uint32_t ms);

/* Diagnostic: launches one tiny kernel whose bounded wait can never be satisfied, so
 * it runs out after `timeout_ms` and records NE_ERR_DEVICE_TIMEOUT in the device error
 * word, exactly as a stalled attention kernel would.  Used to test the error path
 * without faulting or hanging the GPU. */
ne_status ne_selftest_wait_timeout(uint32_t timeout_ms, ne_stream_t stream);

/* Diagnostic timing of the kernels behind the calls above.  While enabled (on != 0),
 * every call records a CUDA event before and after each kernel it launches, on the
 * call's stream; ne_profile_totals() synchronises the current device and returns, per
 * phase, the summed milliseconds and the number of launches since enabling:
 * phase 0 forward, 1 backward Delta preprocess, 2 backward main, 3 backward dQ
 * epilogue.  Enabling again restarts the sums and reuses the events already made;
 * disabling (on == 0) frees them.  Not thread-safe; off by default. */
void ne_profile_enable(int on);
ne_status ne_profile_totals(double ms_out[4], int launches_out[4]);

/* Releases the library's per-device caches (RoPE tables, error words). */
void ne_shutdown(void);

#ifdef __cplusplus
}
#endif

#endif /* NEATTN_H */
