// api.cu -- the C ABI declared in include/neattn.h: argument validation, status
// codes, per-device caches (RoPE tables, device error word), TMA tensor-map encoding
// and kernel launches.  No compute happens here; every step runs in the kernels.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <tuple>
#include <utility>
#include <vector>

#include "kernels.h"
#include "neattn.h"

namespace {

thread_local std::string g_last_error;

ne_status fail(ne_status s, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return s;
}

ne_status cuda_fail(cudaError_t e, const char* what) {
    return fail(NE_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

// ------------------------------------------------------------------ per-device state
struct DeviceState {
    int* err_word = nullptr;                                           // device int
    // RoPE tables per (D, pairs per row, theta bits): rows and pointer.  A table serves
    // every T up to its rows; a longer T builds one twice as long (or T's), and the
    // shorter one is kept until ne_shutdown (a kernel in flight may still read it), so
    // a caller whose T grows step by step costs at most twice the largest table.
    std::map<std::tuple<int, int, uint64_t>, std::pair<int, float2*>> rope;
    std::vector<float2*> rope_retired;
};

std::mutex g_mu;
std::map<int, DeviceState> g_dev;
uint32_t g_timeout_ms = 0;   // 0 = default

unsigned long long timeout_ns() {
    uint32_t ms = g_timeout_ms;
    if (ms == 0) {
        const char* env = std::getenv("NE_ATTN_TIMEOUT_MS");
        long v = env ? std::strtol(env, nullptr, 10) : 0;
        ms = v > 0 ? (uint32_t)v : 2000u;
    }
    return (unsigned long long)ms * 1000000ull;
}

ne_status current_device(int* dev) {
    cudaError_t e = cudaGetDevice(dev);
    if (e != cudaSuccess) return fail(NE_ERR_NO_DEVICE, "no CUDA device: %s", cudaGetErrorString(e));
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, *dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, *dev);
    if (major != 10 || minor != 3)
        return fail(NE_ERR_NO_DEVICE, "device %d is sm_%d%d; libneattn is built for sm_103a only", *dev, major,
                    minor);
    return NE_OK;
}

// Device error word of the current device (allocated once).
ne_status error_word(int dev, int** out) {
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState& ds = g_dev[dev];
    if (!ds.err_word) {
        cudaError_t e = cudaMalloc(&ds.err_word, sizeof(int));
        if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(error word)");
        e = cudaMemset(ds.err_word, 0, sizeof(int));
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemset(error word)");
    }
    *out = ds.err_word;
    return NE_OK;
}

// Cached interleaved (cos, sin) table [T, ld] (ld >= D/2 pairs per row; pairs past D/2
// hold angle 0) for the current device.  Built on `st` by the rope kernel the first
// time; that first build synchronises `st`.
ne_status rope_cache(int dev, int T, int D, double theta, cudaStream_t st, const float2** out, int ld = 0) {
    if (ld < D / 2) ld = D / 2;
    uint64_t tb;
    std::memcpy(&tb, &theta, sizeof(tb));
    const auto key = std::make_tuple(D, ld, tb);
    const int need = ne::rope_table_rows(T);
    int rows = need;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        auto& m = g_dev[dev].rope;
        auto it = m.find(key);
        if (it != m.end()) {
            if (it->second.first >= need) {
                *out = it->second.second;
                return NE_OK;
            }
            rows = std::max(need, 2 * it->second.first);   // geometric growth
        }
    }
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cap) == cudaSuccess && cap != cudaStreamCaptureStatusNone)
        return fail(NE_ERR_UNSUPPORTED,
                    "first call for T=%d D=%d theta=%g on this device happened inside stream capture; "
                    "make one call before capturing",
                    T, D, theta);
    float2* buf = nullptr;
    size_t bytes = (size_t)rows * ld * sizeof(float2);
    cudaError_t e = cudaMalloc(&buf, bytes);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(rope table)");
    e = ne::launch_rope_table(nullptr, nullptr, buf, rows, D, theta, st, ld);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) {
        cudaFree(buf);
        return cuda_fail(e, "rope table build");
    }
    std::lock_guard<std::mutex> lk(g_mu);
    auto& m = g_dev[dev].rope;
    auto it = m.find(key);
    if (it != m.end() && it->second.first >= need) {   // another thread won the race
        cudaFree(buf);
        *out = it->second.second;
    } else {
        if (it != m.end()) g_dev[dev].rope_retired.push_back(it->second.second);
        m[key] = std::make_pair(rows, buf);
        *out = buf;
    }
    return NE_OK;
}

// ------------------------------------------------------------------ phase timing (diagnostic)
// Events come from a pool that survives re-enabling, so a timed region pays only the
// two cudaEventRecord calls per launch once the pool has grown.
struct PhaseProfile {
    bool on = false;
    std::vector<cudaEvent_t> pool;          // 2 per recorded launch
    std::vector<int> phase;                 // phase of recorded launch i
    size_t used = 0;                        // launches recorded since enabling
};
PhaseProfile g_prof;

// Records `launch` between two events when profiling is on.
template <typename F>
cudaError_t timed(int phase, cudaStream_t st, F&& launch) {
    if (!g_prof.on) return launch();
    const size_t i = g_prof.used;
    while (g_prof.pool.size() < 2 * (i + 1)) {
        cudaEvent_t ev = nullptr;
        if (cudaEventCreate(&ev) != cudaSuccess) return launch();
        g_prof.pool.push_back(ev);
    }
    if (g_prof.phase.size() < i + 1) g_prof.phase.resize(i + 1);
    cudaEventRecord(g_prof.pool[2 * i], st);
    cudaError_t e = launch();
    cudaEventRecord(g_prof.pool[2 * i + 1], st);
    g_prof.phase[i] = phase;
    g_prof.used = i + 1;
    return e;
}

// ------------------------------------------------------------------ tensor maps
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

ne_status encode_fn(EncodeTiledFn* out) {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    if (!fn) return fail(NE_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    *out = fn;
    return NE_OK;
}

// Tiled map over a [B, T, H, D] tensor: box = (128 bytes of D, 1 head, rows, 1 batch),
// 128-byte swizzle, zero fill out of bounds (ragged T tails).
ne_status map_bthd(CUtensorMap* m, const void* ptr, bool f32, int B, int T, int H, int D, int rows,
                   bool f16 = false) {
    EncodeTiledFn enc;
    ne_status s = encode_fn(&enc);
    if (s != NE_OK) return s;
    const int es = f32 ? 4 : 2;
    cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)B};
    cuuint64_t strides[3] = {(cuuint64_t)D * es, (cuuint64_t)H * D * es, (cuuint64_t)T * H * D * es};
    cuuint32_t box[4] = {(cuuint32_t)(128 / es), 1, (cuuint32_t)rows, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    const CUtensorMapDataType dt = f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                       : (f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
    CUresult r = enc(m, dt, 4,
                     const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(NE_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return NE_OK;
}

// Tiled map over a row-major bf16 matrix [rows, cols]: box = (64 columns = 128 bytes,
// box_rows rows), 128-byte swizzle, zero fill out of bounds.
ne_status map_rows_bf16(CUtensorMap* m, const void* ptr, long long rows, int cols, int box_rows) {
    EncodeTiledFn enc;
    ne_status s = encode_fn(&enc);
    if (s != NE_OK) return s;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(NE_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return NE_OK;
}

// ------------------------------------------------------------------ validation
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

ne_status check_shape(int B, int T, int Hq, int Hkv, int D, double theta, bool f32) {
    if (B < 0 || T < 0) return fail(NE_ERR_INVALID_ARG, "B and T must be >= 0 (B=%d T=%d)", B, T);
    if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0)
        return fail(NE_ERR_INVALID_ARG, "need Hq > 0, Hkv > 0 and Hq %% Hkv == 0 (Hq=%d Hkv=%d)", Hq, Hkv);
    if (!(theta > 0.0) || !std::isfinite(theta)) return fail(NE_ERR_INVALID_ARG, "rope_theta must be finite and > 0");
    if (D <= 0 || D % 2 != 0) return fail(NE_ERR_INVALID_ARG, "D must be even and > 0 (D=%d)", D);
    if (f32 ? (D != 32 && D != 64) : (D != 32 && D != 64 && D != 128))
        return fail(NE_ERR_UNSUPPORTED, "head_dim D=%d is not supported for %s (supported: %s)", D,
                    f32 ? "f32" : "bf16", f32 ? "32, 64" : "32, 64, 128");
    const long long elems = (long long)B * T * Hq * D;
    if (elems >= (1LL << 31)) return fail(NE_ERR_INVALID_ARG, "B*T*Hq*D must be < 2^31");
    return NE_OK;
}

ne_status check_ptrs(std::initializer_list<const void*> ps) {
    for (const void* p : ps) {
        if (!p) return fail(NE_ERR_INVALID_ARG, "null tensor pointer");
        if (!aligned16(p)) return fail(NE_ERR_INVALID_ARG, "tensor pointer %p is not 16-byte aligned", p);
    }
    return NE_OK;
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Backward workspace: Delta fp32 [B,Hq,T] | dQ accumulator fp32 [B,T,Hq,D] | rotated fp16
// Q' [B,T,Hq,D] (written by the preprocess kernel for the bf16 head_dim-64 kernel).
struct BwdWs {
    size_t delta, acc, q16, total;
};
BwdWs bwd_ws_layout(int B, int T, int Hq, int D) {
    BwdWs l;
    l.delta = 0;
    l.acc = round_up((size_t)B * Hq * T * sizeof(float), 256);
    l.q16 = l.acc + round_up((size_t)B * T * Hq * D * sizeof(float), 256);
    l.total = l.q16 + (size_t)B * T * Hq * D * 2;
    return l;
}
size_t bwd_ws_bytes(int B, int T, int Hq, int D) { return bwd_ws_layout(B, T, Hq, D).total; }
// The bf16 head_dim-64 kernel reads Q rotated ahead of time by the preprocess kernel.
bool bwd_uses_q16(bool f32, int D) { return !f32 && D <= 64; }
// bf16 head_dim 32 runs on the 64-wide kernels with the upper 32 columns zero (128-byte
// TMA boxes over 64-byte rows read zeros there and clip stores); their RoPE table has
// 32 (cos, sin) pairs per row, the last 16 at angle 0.
int rope_ld(bool f32, int D) { return !f32 && D == 32 ? 32 : D / 2; }

// ------------------------------------------------------------------ forward / backward
// Per-sequence lengths of a variable-length call: a device int32 array [B], 4-byte aligned.
ne_status check_seq_lens(const int* seq_lens) {
    if (!seq_lens || (reinterpret_cast<uintptr_t>(seq_lens) & 3u) != 0)
        return fail(NE_ERR_INVALID_ARG, "seq_lens must be a non-null, 4-byte aligned device pointer");
    return NE_OK;
}

// The backward workspace must be non-null, 256-byte aligned and large enough.
ne_status check_ws(const void* ws, size_t ws_bytes, int B, int T, int Hq, int D) {
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0)
        return fail(NE_ERR_INVALID_ARG, "workspace must be non-null and 256-byte aligned");
    const size_t need = bwd_ws_bytes(B, T, Hq, D);
    if (ws_bytes < need)
        return fail(NE_ERR_INVALID_ARG, "workspace too small: %zu bytes given, %zu needed", ws_bytes, need);
    return NE_OK;
}

// seq_lens: null, or (variable-length calls) the device lengths [B] of the sequences.
// ws: null, or (training forward) the backward workspace that receives R Q and a zeroed
// dQ' accumulator where the backward uses them (bf16, head_dim 32 or 64).
ne_status attn_fwd_impl(bool f32, const void* q, const void* k, const void* v, void* o, float* lse, int B, int T,
                        int Hq, int Hkv, int D, double theta, const int* seq_lens, bool varlen, cudaStream_t st,
                        void* ws = nullptr, size_t ws_bytes = 0, bool train = false) {
    g_last_error.clear();
    ne_status s = check_shape(B, T, Hq, Hkv, D, theta, f32);
    if (s != NE_OK) return s;
    if (B == 0 || T == 0) return NE_OK;
    if ((s = check_ptrs({q, k, v, o, lse})) != NE_OK) return s;
    if (varlen && (s = check_seq_lens(seq_lens)) != NE_OK) return s;
    if (train && (s = check_ws(ws, ws_bytes, B, T, Hq, D)) != NE_OK) return s;
    int dev;
    if ((s = current_device(&dev)) != NE_OK) return s;
    int* err;
    if ((s = error_word(dev, &err)) != NE_OK) return s;
    const float2* rope;
    if ((s = rope_cache(dev, T, D, theta, st, &rope, rope_ld(f32, D))) != NE_OK) return s;
    CUtensorMap tq, tk, tv, to;
    const int kv_rows = ne::fwd_kv_box_rows(f32, D);
    if ((s = map_bthd(&tq, q, f32, B, T, Hq, D, 128)) != NE_OK) return s;
    if ((s = map_bthd(&tk, k, f32, B, T, Hkv, D, kv_rows)) != NE_OK) return s;
    if ((s = map_bthd(&tv, v, f32, B, T, Hkv, D, kv_rows)) != NE_OK) return s;
    if ((s = map_bthd(&to, o, f32, B, T, Hq, D, 128)) != NE_OK) return s;
    ne::FwdArgs a;
    a.o = o;
    a.lse = lse;
    a.rope = rope;
    a.B = B;
    a.T = T;
    a.Hq = Hq;
    a.G = Hq / Hkv;
    a.n_qt = (T + 255) / 256;
    a.n_units = B * Hq * a.n_qt;
    a.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)D));
    a.err = err;
    a.timeout_ns = timeout_ns();
    a.seq_lens = seq_lens;
    a.dr = D;
    a.div_bh = ne::make_fastdiv((uint32_t)(B * Hq));   // B, Hq >= 1 here
    a.div_hq = ne::make_fastdiv((uint32_t)Hq);
    // The training forward fills the backward's R Q and zeroes its dQ' accumulator where
    // the backward reads them (bf16 head_dim <= 64); elsewhere it is the plain forward.
    a.save = train && bwd_uses_q16(f32, D) ? 1 : 0;
    CUtensorMap tq16, tdqz;
    std::memset(&tq16, 0, sizeof(tq16));
    std::memset(&tdqz, 0, sizeof(tdqz));
    if (a.save) {
        const BwdWs wl = bwd_ws_layout(B, T, Hq, D);
        if ((s = map_bthd(&tq16, static_cast<char*>(ws) + wl.q16, false, B, T, Hq, D, 128, true)) != NE_OK) return s;
        if ((s = map_bthd(&tdqz, static_cast<char*>(ws) + wl.acc, true, B, T, Hq, D, 128)) != NE_OK) return s;
    }
    cudaError_t e = timed(0, st, [&] { return ne::launch_fwd(f32, D, B, tq, tk, tv, to, tq16, tdqz, a, st); });
    if (e != cudaSuccess) return cuda_fail(e, "attn_fwd launch");
    return NE_OK;
}

// train: the workspace holds what the training forward left there (R Q and the zeroed
// dQ' accumulator, for bf16 head_dim <= 64), so the preprocess pass only forms Delta.
ne_status attn_bwd_impl(bool f32, const void* q, const void* k, const void* v, const void* o, const float* lse,
                        const void* dO, void* dq, void* dk, void* dv, int B, int T, int Hq, int Hkv, int D,
                        double theta, void* ws, size_t ws_bytes, const int* seq_lens, bool varlen, cudaStream_t st,
                        bool train = false) {
    g_last_error.clear();
    ne_status s = check_shape(B, T, Hq, Hkv, D, theta, f32);
    if (s != NE_OK) return s;
    if (B == 0 || T == 0) return NE_OK;
    if ((s = check_ptrs({q, k, v, o, lse, dO, dq, dk, dv})) != NE_OK) return s;
    if (varlen && (s = check_seq_lens(seq_lens)) != NE_OK) return s;
    if ((s = check_ws(ws, ws_bytes, B, T, Hq, D)) != NE_OK) return s;
    int dev;
    if ((s = current_device(&dev)) != NE_OK) return s;
    int* err;
    if ((s = error_word(dev, &err)) != NE_OK) return s;
    const float2* rope;
    if ((s = rope_cache(dev, T, D, theta, st, &rope, rope_ld(f32, D))) != NE_OK) return s;
    const BwdWs wl = bwd_ws_layout(B, T, Hq, D);
    float* delta = static_cast<float*>(ws);
    float* dq_acc = reinterpret_cast<float*>(static_cast<char*>(ws) + wl.acc);
    void* q16 = bwd_uses_q16(f32, D) ? static_cast<char*>(ws) + wl.q16 : nullptr;
    const long long rows = (long long)B * T * Hq;

    const bool prepared = train && q16 != nullptr;   // R Q stored and dQ' zeroed by the forward
    ne::BwdPreArgs pa{o, dO, delta, prepared ? nullptr : dq_acc, rows, T, Hq, D, q, prepared ? nullptr : q16, rope,
                      err, ne::make_fastdiv((uint32_t)Hq), ne::make_fastdiv((uint32_t)T), seq_lens, rope_ld(f32, D)};
    cudaError_t e = timed(1, st, [&] { return ne::launch_bwd_pre(f32, pa, st); });
    if (e != cudaSuccess) return cuda_fail(e, "attn_bwd preprocess launch");

    CUtensorMap tq, tk, tv, tdo, tdq;
    const int q_rows = ne::bwd_q_box_rows(f32, D);
    if ((s = map_bthd(&tq, q16 ? q16 : q, f32, B, T, Hq, D, q_rows, q16 != nullptr)) != NE_OK) return s;
    if ((s = map_bthd(&tk, k, f32, B, T, Hkv, D, 128)) != NE_OK) return s;
    if ((s = map_bthd(&tv, v, f32, B, T, Hkv, D, 128)) != NE_OK) return s;
    if ((s = map_bthd(&tdo, dO, f32, B, T, Hq, D, q_rows)) != NE_OK) return s;
    std::memset(&tdq, 0, sizeof(tdq));
    if (!f32 && (s = map_bthd(&tdq, dq_acc, true, B, T, Hq, D, 128)) != NE_OK) return s;
    ne::BwdArgs a = {};
    a.lse = lse;
    a.delta = delta;
    a.dq_acc = dq_acc;
    a.dk = dk;
    a.dv = dv;
    a.rope = rope;
    a.T = T;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.G = Hq / Hkv;
    a.n_kvt = (T + 127) / 128;
    a.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)D));
    a.scale = (float)(1.0 / std::sqrt((double)D));
    a.err = err;
    a.timeout_ns = timeout_ns();
    a.seq_lens = seq_lens;
    a.dr = D;
    e = timed(2, st, [&] {
        return f32 ? ne::launch_bwd_tf32(D, B, tq, tk, tv, tdo, a, st)
                   : ne::launch_bwd(f32, D, B, tq, tk, tv, tdo, tdq, a, st);
    });
    if (e != cudaSuccess) return cuda_fail(e, "attn_bwd launch");

    ne::BwdPostArgs qa{dq_acc, dq, rope, rows, T, Hq, D, a.scale, ne::make_fastdiv((uint32_t)Hq),
                          ne::make_fastdiv((uint32_t)T), rope_ld(f32, D)};
    e = timed(3, st, [&] { return ne::launch_bwd_post(f32, qa, st); });
    if (e != cudaSuccess) return cuda_fail(e, "attn_bwd dq epilogue launch");
    return NE_OK;
}

// ------------------------------------------------------------------ decode
// Decode workspace (only when the positions are cut into more than one chunk):
// unnormalised chunk outputs fp32 [B, Hq, n_split, D], then (256-byte aligned) the
// per-chunk (max, sum) pairs [B, Hq, n_split] float2.
size_t decode_part_o_bytes(int B, int Hq, int D, const ne::DecodePlan& p) {
    return round_up((size_t)B * Hq * p.n_split * D * sizeof(float), 256);
}
size_t decode_ws_bytes(int B, int Tmax, int Hq, int Hkv, int D) {
    const ne::DecodePlan p = ne::decode_plan(B, Tmax, Hq, Hkv);
    if (p.n_split <= 1) return 0;
    return decode_part_o_bytes(B, Hq, D, p) + (size_t)B * Hq * p.n_split * sizeof(float2);
}

ne_status attn_decode_impl(bool f32, const void* q, const void* k, const void* v, const int* seq_lens, void* o,
                           float* lse, int B, int Tmax, int Hq, int Hkv, int D, double theta, void* ws,
                           size_t ws_bytes, cudaStream_t st) {
    g_last_error.clear();
    // Head, head_dim and theta rules as for the forward; the cache is indexed in 64 bits.
    ne_status s = check_shape(B, 1, Hq, Hkv, D, theta, f32);
    if (s != NE_OK) return s;
    if (!f32 && D == 32)
        return fail(NE_ERR_UNSUPPORTED, "decode supports head_dim 64 and 128 for bf16 (32 and 64 for f32)");
    if (B > 65535) return fail(NE_ERR_INVALID_ARG, "decode needs B <= 65535 (B=%d)", B);
    if (B == 0) return NE_OK;
    if (Tmax < 1 || Tmax > (1 << 30))
        return fail(NE_ERR_INVALID_ARG, "decode needs 1 <= T_max <= 2^30: the cache holds the newest token (T_max=%d)",
                    Tmax);
    if ((s = check_ptrs({q, k, v, o, lse})) != NE_OK) return s;
    if (!seq_lens || (reinterpret_cast<uintptr_t>(seq_lens) & 3u) != 0)
        return fail(NE_ERR_INVALID_ARG, "seq_lens must be a non-null, 4-byte aligned device pointer");
    const size_t need = decode_ws_bytes(B, Tmax, Hq, Hkv, D);
    if (need > 0 && (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0))
        return fail(NE_ERR_INVALID_ARG, "workspace must be non-null and 256-byte aligned (%zu bytes needed)", need);
    if (ws_bytes < need)
        return fail(NE_ERR_INVALID_ARG, "workspace too small: %zu bytes given, %zu needed", ws_bytes, need);
    int dev;
    if ((s = current_device(&dev)) != NE_OK) return s;
    int* err;
    if ((s = error_word(dev, &err)) != NE_OK) return s;
    const float2* rope;
    if ((s = rope_cache(dev, Tmax, D, theta, st, &rope)) != NE_OK) return s;
    const ne::DecodePlan p = ne::decode_plan(B, Tmax, Hq, Hkv);
    ne::DecodeArgs a;
    a.q = q;
    a.k = k;
    a.v = v;
    a.seq_lens = seq_lens;
    a.o = o;
    a.lse = lse;
    a.part_o = need ? static_cast<float*>(ws) : nullptr;
    a.part_ml = need ? reinterpret_cast<float2*>(static_cast<char*>(ws) + decode_part_o_bytes(B, Hq, D, p)) : nullptr;
    a.rope = rope;
    a.B = B;
    a.Tmax = Tmax;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.G = Hq / Hkv;
    a.n_hgrp = p.n_hgrp;
    a.n_split = p.n_split;
    a.chunk = p.chunk;
    a.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)D));
    a.err = err;
    cudaError_t e = ne::launch_decode(f32, D, p, a, st);
    if (e != cudaSuccess) return cuda_fail(e, "attn_decode launch");
    return NE_OK;
}

// Reads a device error word (the stream that wrote it is already synchronised), clears
// it, and maps a nonzero code to its status.
ne_status read_and_clear(int* err) {
    int h = 0;
    cudaError_t e = cudaMemcpy(&h, err, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "read device error word");
    if (h == 0) return NE_OK;
    e = cudaMemset(err, 0, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e, "clear device error word");
    if (h == ne::SITE_DECODE_LEN)
        return fail(NE_ERR_INVALID_ARG,
                    "a decode call got a seq_lens entry outside [1, T_max]; it was clamped and the outputs of "
                    "that sequence are invalid");
    if (h == ne::SITE_VARLEN_LEN)
        return fail(NE_ERR_INVALID_ARG,
                    "a variable-length call got a seq_lens entry outside [0, T]; it was clamped and the outputs of "
                    "that sequence are invalid");
    if (h == ne::SITE_RANGE)
        return fail(NE_ERR_INVALID_ARG,
                    "a rotated q or k value or a dS value exceeded 65504, the fp16 range of an MMA operand of "
                    "the bf16 path; the outputs of that call are invalid");
    return fail(NE_ERR_DEVICE_TIMEOUT, "a bounded wait inside a kernel ran out (site 0x%x)", h);
}

// ------------------------------------------------------------------ allocation-free backward
// Scratch of ne_attn_bwd_noalloc: a file-scope device array (every GPU that loads the
// library holds it until the process exits).  Layout per call: RoPE table
// [T, D/2] float2 | Delta [B, Hq, T] fp32 | dQ accumulator [B, T, Hq, D] fp32, each
// part starting on a 256-byte boundary.
constexpr size_t kNoAllocScratchBytes = size_t(48) << 20;
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];
// The error word of the allocation-free calls, beside their scratch (zero at load):
// the kernels they launch record range errors and bounded-wait timeouts here, and
// ne_noalloc_get_device_error() reads and clears it.
__device__ int g_noalloc_err;

// Device addresses of g_noalloc_scratch and g_noalloc_err per device ordinal.  In host
// code the names are only host-side stand-ins, so the addresses come from
// cudaGetSymbolAddress, taken once per device with that device current.
constexpr int kMaxDevices = 64;
void* g_noalloc_ptr[kMaxDevices] = {};
int* g_noalloc_err_ptr[kMaxDevices] = {};
std::mutex g_noalloc_mu;

ne_status noalloc_scratch(int dev, void** out, int** err_out) {
    if (dev < 0 || dev >= kMaxDevices) return fail(NE_ERR_UNSUPPORTED, "device ordinal %d >= %d", dev, kMaxDevices);
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        void* pe = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(scratch)");
        e = cudaGetSymbolAddress(&pe, g_noalloc_err);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(error word)");
        g_noalloc_err_ptr[dev] = static_cast<int*>(pe);
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    *err_out = g_noalloc_err_ptr[dev];
    return NE_OK;
}

}  // namespace

namespace ne {
bool pdl_enabled() {
    static const bool on = [] {
        const char* env = std::getenv("NE_ATTN_PDL");
        return !(env && env[0] == '0');
    }();
    return on;
}
}  // namespace ne

extern "C" {

ne_status ne_rope_table(float* cos_out, float* sin_out, int T, int D, double theta, ne_stream_t stream) {
    g_last_error.clear();
    if (T < 0 || D <= 0 || D % 2 != 0) return fail(NE_ERR_INVALID_ARG, "need T >= 0 and even D > 0");
    if (!(theta > 0.0) || !std::isfinite(theta)) return fail(NE_ERR_INVALID_ARG, "theta must be finite and > 0");
    if (T == 0) return NE_OK;
    if (!cos_out || !sin_out) return fail(NE_ERR_INVALID_ARG, "null output pointer");
    int dev;
    ne_status s = current_device(&dev);
    if (s != NE_OK) return s;
    cudaError_t e = ne::launch_rope_table(cos_out, sin_out, nullptr, T, D, theta, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "rope table launch");
    return NE_OK;
}

ne_status ne_attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int T, int Hq,
                      int Hkv, int D, double rope_theta, ne_stream_t stream) {
    return attn_fwd_impl(false, q, k, v, o, lse, B, T, Hq, Hkv, D, rope_theta, nullptr, false, (cudaStream_t)stream);
}

ne_status ne_attn_fwd_f32(const float* q, const float* k, const float* v, float* o, float* lse, int B, int T,
                          int Hq, int Hkv, int D, double rope_theta, ne_stream_t stream) {
    return attn_fwd_impl(true, q, k, v, o, lse, B, T, Hq, Hkv, D, rope_theta, nullptr, false, (cudaStream_t)stream);
}

ne_status ne_attn_fwd_train(const void* q, const void* k, const void* v, void* o, float* lse, void* workspace,
                            size_t workspace_bytes, int B, int T, int Hq, int Hkv, int D, double rope_theta,
                            ne_stream_t stream) {
    return attn_fwd_impl(false, q, k, v, o, lse, B, T, Hq, Hkv, D, rope_theta, nullptr, false, (cudaStream_t)stream,
                         workspace, workspace_bytes, true);
}

ne_status ne_attn_fwd_train_f32(const float* q, const float* k, const float* v, float* o, float* lse, void* workspace,
                                size_t workspace_bytes, int B, int T, int Hq, int Hkv, int D, double rope_theta,
                                ne_stream_t stream) {
    return attn_fwd_impl(true, q, k, v, o, lse, B, T, Hq, Hkv, D, rope_theta, nullptr, false, (cudaStream_t)stream,
                         workspace, workspace_bytes, true);
}

ne_status ne_attn_bwd_train(const void* q, const void* k, const void* v, const void* o, const float* lse,
                            const void* dO, void* dq, void* dk, void* dv, int B, int T, int Hq, int Hkv, int D,
                            double rope_theta, void* workspace, size_t workspace_bytes, ne_stream_t stream) {
    return attn_bwd_impl(false, q, k, v, o, lse, dO, dq, dk, dv, B, T, Hq, Hkv, D, rope_theta, workspace,
                         workspace_bytes, nullptr, false, (cudaStream_t)stream, true);
}

ne_status ne_attn_bwd_train_f32(const float* q, const float* k, const float* v, const float* o, const float* lse,
                                const float* dO, float* dq, float* dk, float* dv, int B, int T, int Hq, int Hkv,
                                int D, double rope_theta, void* workspace, size_t workspace_bytes,
                                ne_stream_t stream) {
    return attn_bwd_impl(true, q, k, v, o, lse, dO, dq, dk, dv, B, T, Hq, Hkv, D, rope_theta, workspace,
                         workspace_bytes, nullptr, false, (cudaStream_t)stream, true);
}

size_t ne_attn_bwd_workspace_size(int B, int T, int Hq, int Hkv, int D) {
    if (B < 0 || T < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Hq % Hkv != 0) return 0;
    return bwd_ws_bytes(B, T, Hq, D);
}

ne_status ne_attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
                      void* dq, void* dk, void* dv, int B, int T, int Hq, int Hkv, int D, double rope_theta,
                      void* workspace, size_t workspace_bytes, ne_stream_t stream) {
    return attn_bwd_impl(false, q, k, v, o, lse, dO, dq, dk, dv, B, T, Hq, Hkv, D, rope_theta, workspace,
                         workspace_bytes, nullptr, false, (cudaStream_t)stream);
}

ne_status ne_attn_bwd_f32(const float* q, const float* k, const float* v, const float* o, const float* lse,
                          const float* dO, float* dq, float* dk, float* dv, int B, int T, int Hq, int Hkv, int D,
                          double rope_theta, void* workspace, size_t workspace_bytes, ne_stream_t stream) {
    return attn_bwd_impl(true, q, k, v, o, lse, dO, dq, dk, dv, B, T, Hq, Hkv, D, rope_theta, workspace,
                         workspace_bytes, nullptr, false, (cudaStream_t)stream);
}

ne_status ne_attn_fwd_varlen(const void* q, const void* k, const void* v, const int* seq_lens, void* o, float* lse,
                             int B, int T, int Hq, int Hkv, int D, double rope_theta, ne_stream_t stream) {
    return attn_fwd_impl(false, q, k, v, o, lse, B, T, Hq, Hkv, D, rope_theta, seq_lens, true, (cudaStream_t)stream);
}

ne_status ne_attn_fwd_varlen_f32(const float* q, const float* k, const float* v, const int* seq_lens, float* o,
                                 float* lse, int B, int T, int Hq, int Hkv, int D, double rope_theta,
                                 ne_stream_t stream) {
    return attn_fwd_impl(true, q, k, v, o, lse, B, T, Hq, Hkv, D, rope_theta, seq_lens, true, (cudaStream_t)stream);
}

ne_status ne_attn_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const float* lse,
                             const void* dO, const int* seq_lens, void* dq, void* dk, void* dv, int B, int T, int Hq,
                             int Hkv, int D, double rope_theta, void* workspace, size_t workspace_bytes,
                             ne_stream_t stream) {
    return attn_bwd_impl(false, q, k, v, o, lse, dO, dq, dk, dv, B, T, Hq, Hkv, D, rope_theta, workspace,
                         workspace_bytes, seq_lens, true, (cudaStream_t)stream);
}

ne_status ne_attn_bwd_varlen_f32(const float* q, const float* k, const float* v, const float* o, const float* lse,
                                 const float* dO, const int* seq_lens, float* dq, float* dk, float* dv, int B, int T,
                                 int Hq, int Hkv, int D, double rope_theta, void* workspace, size_t workspace_bytes,
                                 ne_stream_t stream) {
    return attn_bwd_impl(true, q, k, v, o, lse, dO, dq, dk, dv, B, T, Hq, Hkv, D, rope_theta, workspace,
                         workspace_bytes, seq_lens, true, (cudaStream_t)stream);
}

size_t ne_attn_decode_workspace_size(int B, int T_max, int Hq, int Hkv, int D) {
    if (B <= 0 || T_max <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Hq % Hkv != 0) return 0;
    return decode_ws_bytes(B, T_max, Hq, Hkv, D);
}

ne_status ne_attn_decode(const void* q, const void* k_cache, const void* v_cache, const int* seq_lens, void* o,
                         float* lse, int B, int T_max, int Hq, int Hkv, int D, double rope_theta, void* workspace,
                         size_t workspace_bytes, ne_stream_t stream) {
    return attn_decode_impl(false, q, k_cache, v_cache, seq_lens, o, lse, B, T_max, Hq, Hkv, D, rope_theta,
                            workspace, workspace_bytes, (cudaStream_t)stream);
}

ne_status ne_attn_decode_f32(const float* q, const float* k_cache, const float* v_cache, const int* seq_lens,
                             float* o, float* lse, int B, int T_max, int Hq, int Hkv, int D, double rope_theta,
                             void* workspace, size_t workspace_bytes, ne_stream_t stream) {
    return attn_decode_impl(true, q, k_cache, v_cache, seq_lens, o, lse, B, T_max, Hq, Hkv, D, rope_theta,
                            workspace, workspace_bytes, (cudaStream_t)stream);
}

// W diag(gamma) (bf16), then 1/rms of every token row (fp32).
static size_t prologue_weight_bytes(int dim, int Hq, int Hkv, int D) {
    return round_up((size_t)(Hq + 2 * Hkv) * D * dim * 2, 256);
}
size_t ne_qkv_prologue_workspace_size(int B, int T, int dim, int Hq, int Hkv, int D) {
    if (B < 0 || T < 0 || dim <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0) return 0;
    return prologue_weight_bytes(dim, Hq, Hkv, D) + round_up((size_t)B * T * 4, 256);
}

ne_status ne_qkv_prologue(const void* x, const void* gamma, const void* w, void* q, void* k, void* v, int B, int T,
                          int dim, int Hq, int Hkv, int D, double eps, double rope_theta, int rotate,
                          void* workspace, size_t workspace_bytes, ne_stream_t stream) {
    g_last_error.clear();
    cudaStream_t st = (cudaStream_t)stream;
    if (B < 0 || T < 0) return fail(NE_ERR_INVALID_ARG, "B and T must be >= 0 (B=%d T=%d)", B, T);
    if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0)
        return fail(NE_ERR_INVALID_ARG, "need Hq > 0, Hkv > 0 and Hq %% Hkv == 0 (Hq=%d Hkv=%d)", Hq, Hkv);
    if (D != 32 && D != 64 && D != 128)
        return fail(NE_ERR_UNSUPPORTED, "head_dim D=%d is not supported (supported: 32, 64, 128)", D);
    if (dim <= 0 || dim % 8 != 0) return fail(NE_ERR_INVALID_ARG, "dim must be a positive multiple of 8 (dim=%d)", dim);
    if (!(eps >= 0.0) || !std::isfinite(eps)) return fail(NE_ERR_INVALID_ARG, "eps must be finite and >= 0");
    if (!(rope_theta > 0.0) || !std::isfinite(rope_theta))
        return fail(NE_ERR_INVALID_ARG, "rope_theta must be finite and > 0");
    const long long M = (long long)B * T;
    const long long N = (long long)(Hq + 2 * Hkv) * D;
    if (M * dim >= (1LL << 31) || M * N >= (1LL << 31) || (M + 127) / 128 > 65535)
        return fail(NE_ERR_INVALID_ARG, "shape too large: B*T*dim and B*T*(Hq+2Hkv)*D must be < 2^31");
    if (M == 0) return NE_OK;
    ne_status s;
    if ((s = check_ptrs({x, gamma, w, q, k, v})) != NE_OK) return s;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return fail(NE_ERR_INVALID_ARG, "workspace must be non-null and 256-byte aligned");
    if (workspace_bytes < ne_qkv_prologue_workspace_size(B, T, dim, Hq, Hkv, D))
        return fail(NE_ERR_INVALID_ARG, "workspace too small: %zu bytes given, %zu needed", workspace_bytes,
                    ne_qkv_prologue_workspace_size(B, T, dim, Hq, Hkv, D));
    if ((reinterpret_cast<uintptr_t>(gamma) & 15u) != 0 || (reinterpret_cast<uintptr_t>(w) & 15u) != 0)
        return fail(NE_ERR_INVALID_ARG, "gamma and w must be 16-byte aligned");
    int dev;
    if ((s = current_device(&dev)) != NE_OK) return s;
    int* err;
    if ((s = error_word(dev, &err)) != NE_OK) return s;
    const float2* rope;
    if ((s = rope_cache(dev, T, D, rope_theta, st, &rope)) != NE_OK) return s;
    CUtensorMap tx, tw;
    if ((s = map_rows_bf16(&tx, x, M, dim, 128)) != NE_OK) return s;
    // The gain folded into the weights, W' = W diag(gamma), and the 1/rms of every token
    // row after them in the workspace.
    float* inv_rms = reinterpret_cast<float*>(static_cast<char*>(workspace) + prologue_weight_bytes(dim, Hq, Hkv, D));
    cudaError_t e = ne::launch_prologue_prep(w, gamma, workspace, N, x, inv_rms, (int)M, dim, (float)eps, st);
    if (e != cudaSuccess) return cuda_fail(e, "prologue prep launch");
    if ((s = map_rows_bf16(&tw, workspace, N, dim, ne::prologue_tile_n())) != NE_OK) return s;
    ne::ProArgs a;
    a.q = q;
    a.k = k;
    a.v = v;
    a.rope = rope;
    a.M = (int)M;
    a.T = T;
    a.dim = dim;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.D = D;
    a.inv_rms = inv_rms;
    a.rotate = rotate;
    a.err = err;
    a.timeout_ns = timeout_ns();
    e = ne::launch_qkv_prologue(tx, tw, a, st);
    if (e != cudaSuccess) return cuda_fail(e, "qkv prologue launch");
    return NE_OK;
}

const char* ne_status_string(ne_status s) {
    switch (s) {
        case NE_OK: return "NE_OK";
        case NE_ERR_INVALID_ARG: return "NE_ERR_INVALID_ARG";
        case NE_ERR_UNSUPPORTED: return "NE_ERR_UNSUPPORTED";
        case NE_ERR_CUDA: return "NE_ERR_CUDA";
        case NE_ERR_DEVICE_TIMEOUT: return "NE_ERR_DEVICE_TIMEOUT";
        case NE_ERR_NO_DEVICE: return "NE_ERR_NO_DEVICE";
    }
    return "NE_UNKNOWN_STATUS";
}

const char* ne_last_error(void) { return g_last_error.c_str(); }

ne_status ne_get_device_error(ne_stream_t stream) {
    g_last_error.clear();
    int dev;
    ne_status s = current_device(&dev);
    if (s != NE_OK) return s;
    int* err;
    if ((s = error_word(dev, &err)) != NE_OK) return s;
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    return read_and_clear(err);
}

ne_status ne_noalloc_get_device_error(ne_stream_t stream) {
    g_last_error.clear();
    int dev;
    ne_status s = current_device(&dev);
    if (s != NE_OK) return s;
    void* base;
    int* err;
    if ((s = noalloc_scratch(dev, &base, &err)) != NE_OK) return s;
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    return read_and_clear(err);
}

void ne_set_wait_timeout_ms(uint32_t ms) { g_timeout_ms = ms; }

ne_status ne_selftest_wait_timeout(uint32_t timeout_ms, ne_stream_t stream) {
    g_last_error.clear();
    int dev;
    ne_status s = current_device(&dev);
    if (s != NE_OK) return s;
    int* err;
    if ((s = error_word(dev, &err)) != NE_OK) return s;
    cudaError_t e = ne::launch_selftest_wait(err, (unsigned long long)timeout_ms * 1000000ull, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "selftest launch");
    return NE_OK;
}

void ne_profile_enable(int on) {
    g_prof.used = 0;
    g_prof.on = on != 0;
    if (!g_prof.on) {
        for (cudaEvent_t ev : g_prof.pool) cudaEventDestroy(ev);
        g_prof.pool.clear();
        g_prof.phase.clear();
    }
}

ne_status ne_profile_totals(double ms_out[4], int launches_out[4]) {
    g_last_error.clear();
    if (!ms_out || !launches_out) return fail(NE_ERR_INVALID_ARG, "null output");
    for (int i = 0; i < 4; ++i) {
        ms_out[i] = 0.0;
        launches_out[i] = 0;
    }
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
    for (size_t i = 0; i < g_prof.used; ++i) {
        float ms = 0.f;
        const int ph = g_prof.phase[i];
        if (cudaEventElapsedTime(&ms, g_prof.pool[2 * i], g_prof.pool[2 * i + 1]) == cudaSuccess && ph >= 0 && ph < 4) {
            ms_out[ph] += ms;
            launches_out[ph] += 1;
        }
    }
    return NE_OK;
}

void ne_shutdown(void) {
    std::lock_guard<std::mutex> lk(g_mu);
    int cur = 0;
    cudaGetDevice(&cur);
    for (auto& kv : g_dev) {
        cudaSetDevice(kv.first);
        if (kv.second.err_word) cudaFree(kv.second.err_word);
        for (auto& r : kv.second.rope) cudaFree(r.second.second);
        for (float2* p : kv.second.rope_retired) cudaFree(p);
    }
    g_dev.clear();
    cudaSetDevice(cur);
}

ne_status ne_attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                              const void* dO, void* dq, void* dk, void* dv, int B, int T, int Hq, int Hkv, int D,
                              double rope_theta, ne_stream_t stream) {
    g_last_error.clear();
    cudaStream_t st = (cudaStream_t)stream;
    ne_status s = check_shape(B, T, Hq, Hkv, D, rope_theta, false);
    if (s != NE_OK) return s;
    if (B == 0 || T == 0) return NE_OK;
    if ((s = check_ptrs({q, k, v, o, lse, dO, dq, dk, dv})) != NE_OK) return s;
    const int ld = rope_ld(false, D);
    const size_t rope_bytes = round_up((size_t)ne::rope_table_rows(T) * ld * sizeof(float2), 256);
    const size_t delta_bytes = round_up((size_t)B * Hq * T * sizeof(float), 256);
    const size_t acc_bytes = round_up((size_t)B * T * Hq * D * sizeof(float), 256);
    const size_t q16_bytes = bwd_uses_q16(false, D) ? (size_t)B * T * Hq * D * 2 : 0;
    if (rope_bytes + delta_bytes + acc_bytes + q16_bytes > kNoAllocScratchBytes)
        return fail(NE_ERR_INVALID_ARG,
                    "ne_attn_bwd_noalloc: this shape needs %zu bytes of scratch, above its fixed maximum of %zu "
                    "(%zu MiB); use ne_attn_bwd with a caller-allocated workspace",
                    rope_bytes + delta_bytes + acc_bytes + q16_bytes, kNoAllocScratchBytes, kNoAllocScratchBytes >> 20);
    int dev;
    if ((s = current_device(&dev)) != NE_OK) return s;
    void* base;
    int* err;
    if ((s = noalloc_scratch(dev, &base, &err)) != NE_OK) return s;
    float2* rope = static_cast<float2*>(base);
    float* delta = reinterpret_cast<float*>(static_cast<char*>(base) + rope_bytes);
    float* dq_acc = reinterpret_cast<float*>(static_cast<char*>(base) + rope_bytes + delta_bytes);
    void* q16 = q16_bytes ? static_cast<char*>(base) + rope_bytes + delta_bytes + acc_bytes : nullptr;
    const long long rows = (long long)B * T * Hq;

    // The table is rebuilt on every call: the scratch keeps whatever the last call left.
    cudaError_t e = ne::launch_rope_table(nullptr, nullptr, rope, ne::rope_table_rows(T), D, rope_theta, st, ld);
    if (e != cudaSuccess) return cuda_fail(e, "rope table launch");
    ne::BwdPreArgs pa{o, dO, delta, dq_acc, rows, T, Hq, D, q, q16, rope, err,   // also zeroes dq_acc
                      ne::make_fastdiv((uint32_t)Hq), ne::make_fastdiv((uint32_t)T), nullptr, ld};
    e = ne::launch_bwd_pre(false, pa, st);
    if (e != cudaSuccess) return cuda_fail(e, "attn_bwd preprocess launch");
    CUtensorMap tq, tk, tv, tdo, tdq;
    const int q_rows = ne::bwd_q_box_rows(false, D);
    if ((s = map_bthd(&tq, q16 ? q16 : q, false, B, T, Hq, D, q_rows, q16 != nullptr)) != NE_OK) return s;
    if ((s = map_bthd(&tk, k, false, B, T, Hkv, D, 128)) != NE_OK) return s;
    if ((s = map_bthd(&tv, v, false, B, T, Hkv, D, 128)) != NE_OK) return s;
    if ((s = map_bthd(&tdo, dO, false, B, T, Hq, D, q_rows)) != NE_OK) return s;
    std::memset(&tdq, 0, sizeof(tdq));
    if ((s = map_bthd(&tdq, dq_acc, true, B, T, Hq, D, 128)) != NE_OK) return s;
    ne::BwdArgs a = {};
    a.lse = lse;
    a.delta = delta;
    a.dq_acc = dq_acc;
    a.dk = dk;
    a.dv = dv;
    a.rope = rope;
    a.T = T;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.G = Hq / Hkv;
    a.n_kvt = (T + 127) / 128;
    a.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)D));
    a.scale = (float)(1.0 / std::sqrt((double)D));
    a.err = err;                // the static error word of the allocation-free calls
    a.timeout_ns = timeout_ns();
    a.seq_lens = nullptr;
    a.dr = D;
    e = ne::launch_bwd(false, D, B, tq, tk, tv, tdo, tdq, a, st);
    if (e != cudaSuccess) return cuda_fail(e, "attn_bwd launch");
    ne::BwdPostArgs qa{dq_acc, dq, rope, rows, T, Hq, D, a.scale, ne::make_fastdiv((uint32_t)Hq),
                          ne::make_fastdiv((uint32_t)T), ld};
    e = ne::launch_bwd_post(false, qa, st);
    if (e != cudaSuccess) return cuda_fail(e, "attn_bwd dq epilogue launch");
    return NE_OK;
}

}  // extern "C"
