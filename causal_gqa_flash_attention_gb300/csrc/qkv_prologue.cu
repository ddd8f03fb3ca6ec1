// qkv_prologue.cu -- the steps before attention in every layer, fused into one tcgen05
// GEMM: RMSNorm (pre-normalization, gain gamma, no bias), one bias-free projection to the
// query, key and value heads, and RoPE on the query and key heads ("NanoEuler: C와 CUDA로
// 밑바닥부터 구축한 GPT-2 규모의 LLM", 기술 사양: RMSNorm, RoPE and GQA bullets; the pages
// run this projection on cuBLAS TF32 tensor cores, 커널 구현).  For token row m:
//   r_m = sqrt(mean_c x_mc^2 + eps),   y_m = W (x_m o gamma) / r_m
// with W [(Hq + 2 Hkv) D, dim] (query heads, then key heads, then value heads).  Since
// 1/r_m is one factor per output row, it is applied to the fp32 accumulator in the
// epilogue; gamma is folded into the weights once per call (W' = W diag(gamma)) and
// 1/r_m is formed once per row, both by a small pass into the caller's workspace before
// the GEMM, so x goes from TMA straight to the MMA and the GEMM's ring has one reader.
//
// Persistent, one CTA per SM walking 128-row x 256-column output tiles; the dim (K) axis
// streams through an NS-stage ring of 64-column chunks (x: 128 rows, W': 256 rows, 128
// bytes each, 128-byte-swizzled by TMA) that only the MMAs read.  Warp roles (192
// threads):
//   warp 0      TMA producer.
//   warp 1      TMEM owner (512 columns) and UMMA issuer: M128 N256 K16, 4 per chunk,
//               into two accumulators (tile i in columns 256 (i % 2)).
//   warps 2-5   epilogue, thread = token row = TMEM lane: acc / r_m, RoPE on query and
//               key heads (position m mod T), bf16 stores; the tile's 1/r_m and (cos,
//               sin) row are fetched one tile early.
// An earlier version summed each row's squares inside this kernel, on four more warps
// reading the ring's x chunks and releasing a stage after their loads.  Under load such
// a warp at times read a stage already refilled with the chunk four ahead (per-chunk
// checksums of the rows it read showed it), although its release followed its loads,
// even with the release made to depend on the loaded data; any change to the warp's
// timing hid it.  Each row block was also summed once per column tile (five times at
// the GPU-pipeline shape); the row pass sums it once.
// clock64 traces of the first version, which multiplied x by gamma in place between TMA
// and MMA, showed that pass (~2.2K cycles a chunk on one warp per SM sub-partition) and
// an epilogue that waited on a table load per chunk (~15K cycles) as the whole cost.
// Every wait is bounded; a CTA that gives up records an error code, drains its own copies
// and MMAs and frees its TMEM.
#include <cuda_bf16.h>
#include "kernels.h"
#include "ptx.cuh"
#include "rope_smem.cuh"

namespace ne {

namespace {

struct ProCfg {
    static constexpr int BM = 128;                  // token rows per tile
    static constexpr int BN = 256;                  // output features per tile
    static constexpr int BK = 64;                   // dim elements per chunk (128 bytes)
    static constexpr int A_BYTES = BM * 128;
    static constexpr int B_BYTES = BN * 128;
    static constexpr int STAGE = A_BYTES + B_BYTES;
    static constexpr int NS = 4;
    static constexpr int SMEM = 1024 + NS * STAGE;
    static constexpr int THREADS = 192;
    static_assert(SMEM <= 227 * 1024, "shared memory");
};

template <int D>
__global__ void __launch_bounds__(192, 1)
    qkv_prologue_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                        const ProArgs a) {
    using C = ProCfg;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    auto st_a = [&](int s) { return smem + s * C::STAGE; };
    auto st_b = [&](int s) { return smem + s * C::STAGE + C::A_BYTES; };

    __shared__ __align__(8) uint64_t bar_full[C::NS], bar_empty[C::NS];
    __shared__ __align__(8) uint64_t bar_acc_full[2], bar_acc_empty[2];   // [accumulator]
    __shared__ __align__(8) uint64_t bar_final;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nk = (a.dim + C::BK - 1) / C::BK;
    const int nh = a.Hq + 2 * a.Hkv;
    const int tiles_n = (nh * D + C::BN - 1) / C::BN, tiles_m = (a.M + C::BM - 1) / C::BM;
    const int n_tiles = tiles_n * tiles_m;
    // This CTA's tiles: blockIdx.x, + gridDim.x, ...  Tile t is (row block t / tiles_n,
    // column block t % tiles_n), so tiles running at the same time share rows of x in L2.
    const int my_tiles = n_tiles > (int)blockIdx.x ? (n_tiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    auto tile_m0 = [&](int i) { return ((int)blockIdx.x + i * (int)gridDim.x) / tiles_n * C::BM; };
    auto tile_n0 = [&](int i) { return ((int)blockIdx.x + i * (int)gridDim.x) % tiles_n * C::BN; };

    if (tid == 0) {
        for (int s = 0; s < C::NS; ++s) {
            mbar_init(smem_u32(&bar_full[s]), 1);
            mbar_init(smem_u32(&bar_empty[s]), 1);   // the chunk's MMAs have completed
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&bar_acc_full[i]), 1);        // the tile's last MMA
            mbar_init(smem_u32(&bar_acc_empty[i]), 128);     // the epilogue threads
        }
        mbar_init(smem_u32(&bar_final), 1);
        abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tm_x);
        tma_prefetch_desc(&tm_w);
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
    griddep_wait();
    const uint32_t tm = tmem_slot;
    const WaitCtx w{a.err, &abort_flag, a.timeout_ns};

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        // One ring over every chunk of every tile of the CTA (chunk g = i nk + kc).
        if (lane == 0) {
            int issued = 0;
            bool ok = true;
            for (int i = 0; ok && i < my_tiles; ++i) {
                const int m0 = tile_m0(i), n0 = tile_n0(i);
                for (int kc = 0; kc < nk; ++kc) {
                    const int g = issued, s = g % C::NS;
                    if (g >= C::NS &&
                        !(ok = mbar_wait(smem_u32(&bar_empty[s]), ((g / C::NS) - 1) & 1, w, SITE_PRO_EMPTY)))
                        break;
                    const uint32_t f = smem_u32(&bar_full[s]);
                    mbar_arrive_expect_tx(f, C::STAGE);
                    tma_load_2d(smem_u32(st_a(s)), &tm_x, f, kc * C::BK, m0);
                    tma_load_2d(smem_u32(st_b(s)), &tm_w, f, kc * C::BK, n0);
                    ++issued;
                }
            }
            // Teardown: every copy this CTA started must have landed before exit.
            for (int g = max(0, issued - C::NS); g < issued; ++g)
                mbar_wait_drain(smem_u32(&bar_full[g % C::NS]), (g / C::NS) & 1, w, SITE_PRO_DRAIN);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ UMMA issuer
        // Tile i accumulates in TMEM columns 256 (i % 2) .. + 255, once the epilogue has
        // read tile i - 2 out of them.
        constexpr uint32_t id = idesc_make(FMT_BF16, 128, C::BN, false, false);
        const uint64_t da0 = sdesc(smem_u32(st_a(0)), 16, 1024), db0 = sdesc(smem_u32(st_b(0)), 16, 1024);
        bool ok = true;
        int g = 0;
        for (int i = 0; ok && i < my_tiles; ++i) {
            const int ab = i & 1;
            if (i >= 2 && !(ok = mbar_wait_warp(smem_u32(&bar_acc_empty[ab]), ((i >> 1) - 1) & 1, w, SITE_PRO_ACC)))
                break;
            tc_fence_after();
            const uint32_t acc = tm + 256 * ab;
            for (int kc = 0; kc < nk; ++kc, ++g) {
                const int s = g % C::NS;
                if (!(ok = mbar_wait_warp(smem_u32(&bar_full[s]), (g / C::NS) & 1, w, SITE_PRO_FULL))) break;
                tc_fence_after();
                const uint64_t da = sdesc_add(da0, s * C::STAGE), db = sdesc_add(db0, s * C::STAGE);
                if (elect_one()) {                    // one elected lane issues the batch
#pragma unroll
                    for (int ks = 0; ks < C::BK / 16; ++ks)   // K = dim, 16 per step (32 bytes)
                        umma_ss<false>(acc, sdesc_add(da, ks * 32), sdesc_add(db, ks * 32), id,
                                       (kc > 0 || ks > 0) ? 1u : 0u);
                    umma_commit(smem_u32(&bar_empty[s]));
                    if (kc == nk - 1) umma_commit(smem_u32(&bar_acc_full[ab]));
                }
                __syncwarp();
            }
        }
        umma_commit_e(smem_u32(&bar_final));   // the teardown's: every MMA of this CTA
    } else {
        // ------------------------------------------------------------ epilogue
        // Thread r: token row r of the tile = TMEM lane (warps 2-5 cover the four lane
        // quarters).  acc / r_m, RoPE on query and key heads (position m mod T), bf16
        // stores; the tile's (cos, sin) table row is fetched one tile early.
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;
        const uint32_t lt = tm + ((uint32_t)(quarter * 32) << 16);
        float4 tabr[D / 4];
        float invr = 0.f;
        auto fetch_row = [&](int i) {
            const int m = tile_m0(i) + r;
            invr = m < a.M ? __ldg(a.inv_rms + m) : 0.f;
            const float4* tr = reinterpret_cast<const float4*>(a.rope + (size_t)(m % a.T) * (D / 2));
#pragma unroll
            for (int e = 0; e < D / 4; ++e)
                tabr[e] = a.rotate && m < a.M ? __ldg(tr + e) : make_float4(0.f, 0.f, 0.f, 0.f);
        };
        if (my_tiles > 0) fetch_row(0);
        bool ok = true;
        for (int i = 0; ok && i < my_tiles; ++i) {
            const int ab = i & 1;
            const int m = tile_m0(i) + r, n0 = tile_n0(i);
            const float inv_r = invr;
            if (!(ok = mbar_wait_warp(smem_u32(&bar_acc_full[ab]), (i >> 1) & 1, w, SITE_PRO_ACC))) break;
            tc_fence_after();
            // Unrolled over the tile's chunks so each chunk's table pairs are registers
            // named at compile time (32 columns = 16 pairs; the tile starts on a head).
#pragma unroll
            for (int c = 0; c < C::BN; c += 32) {
                uint32_t x[32];
                tmem_ld32(lt + 256 * ab + c, x);
                tmem_wait_ld();
                reg_fence32(x);
                if (c + 32 == C::BN) {                   // the accumulator may take tile i + 2
                    tc_fence_before();
                    mbar_arrive(smem_u32(&bar_acc_empty[ab]));
                }
                const int n = n0 + c;                   // first output feature of the chunk
                if (m >= a.M || n >= nh * D) continue;
                const int h = n / D, e0 = n - h * D;    // head and column within it (32 | D)
                static_assert(C::BN % D == 0 || D % C::BN == 0, "chunks line up with heads");
                float y[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) y[e] = __uint_as_float(x[e]) * inv_r;
                if (a.rotate && h < a.Hq + a.Hkv) {     // RoPE on query and key heads
#pragma unroll
                    for (int e = 0; e < 32; e += 4) {
                        const float4 cs = tabr[((c % D) + e) / 4];
                        const float y0 = y[e], y1 = y[e + 1], y2 = y[e + 2], y3 = y[e + 3];
                        y[e] = rot0(y0, y1, cs.x, cs.y);
                        y[e + 1] = rot1(y0, y1, cs.x, cs.y);
                        y[e + 2] = rot0(y2, y3, cs.z, cs.w);
                        y[e + 3] = rot1(y2, y3, cs.z, cs.w);
                    }
                }
                __nv_bfloat16* dst = h < a.Hq ? static_cast<__nv_bfloat16*>(a.q) + ((size_t)m * a.Hq + h) * D
                                     : h < a.Hq + a.Hkv
                                         ? static_cast<__nv_bfloat16*>(a.k) + ((size_t)m * a.Hkv + (h - a.Hq)) * D
                                         : static_cast<__nv_bfloat16*>(a.v) + ((size_t)m * a.Hkv + (h - a.Hq - a.Hkv)) * D;
                uint4* d4 = reinterpret_cast<uint4*>(dst + e0);
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    d4[u] = make_uint4(pack_bf162(y[8 * u], y[8 * u + 1]), pack_bf162(y[8 * u + 2], y[8 * u + 3]),
                                       pack_bf162(y[8 * u + 4], y[8 * u + 5]), pack_bf162(y[8 * u + 6], y[8 * u + 7]));
            }
            if (i + 1 < my_tiles) fetch_row(i + 1);
        }
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        mbar_wait_drain(smem_u32(&bar_final), 0, w, SITE_PRO_DRAIN);
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tm, 512);
    }
}

// The two passes before the GEMM, in one launch: W' = W diag(gamma) (row n, column c of
// the projection times the gain of input column c, rounded to bf16; 8 elements, 16 bytes,
// per thread step), then inv_rms[m] = 1 / sqrt(mean_c x_mc^2 + eps) (one warp per row,
// 16 bytes a lane at a time, the lanes' sums combined by shuffles; dim % 8 == 0).
__global__ void __launch_bounds__(256) prologue_prep_kernel(const __nv_bfloat16* __restrict__ w,
                                                            const __nv_bfloat16* __restrict__ gamma,
                                                            __nv_bfloat16* __restrict__ wg, long long n8,
                                                            const __nv_bfloat16* __restrict__ x,
                                                            float* __restrict__ inv_rms, int M, int dim, float eps) {
    griddep_launch_dependents();
    griddep_wait();
    const int dim8 = dim / 8;
    const uint4* w4 = reinterpret_cast<const uint4*>(w);
    const uint4* g4 = reinterpret_cast<const uint4*>(gamma);
    uint4* o4 = reinterpret_cast<uint4*>(wg);
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n8; i += (long long)gridDim.x * blockDim.x) {
        const uint4 wv = w4[i], gv = __ldg(g4 + (int)(i % dim8));
        const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w}, gw[4] = {gv.x, gv.y, gv.z, gv.w};
        uint32_t o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 wf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ww[e]));
            const float2 gf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gw[e]));
            o[e] = pack_bf162(wf.x * gf.x, wf.y * gf.y);
        }
        o4[i] = make_uint4(o[0], o[1], o[2], o[3]);
    }
    const int lane = threadIdx.x & 31;
    const int warps = (gridDim.x * blockDim.x) >> 5;
    for (int m = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; m < M; m += warps) {
        const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)m * dim);
        float2 ss2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
        for (int c = lane; c < dim8; c += 32) {
            const uint4 v = __ldg(xr + c);
            const uint32_t xw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 xf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&xw[e]));
                ss2[e] = __ffma2_rn(xf, xf, ss2[e]);
            }
        }
        float ss = ((ss2[0].x + ss2[0].y) + (ss2[1].x + ss2[1].y)) + ((ss2[2].x + ss2[2].y) + (ss2[3].x + ss2[3].y));
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
        if (lane == 0) inv_rms[m] = rsqrtf(ss / (float)dim + eps);
    }
}

}  // namespace

int prologue_tile_n() { return ProCfg::BN; }

cudaError_t launch_prologue_prep(const void* w, const void* gamma, void* wg, long long N, const void* x,
                                 float* inv_rms, int M, int dim, float eps, cudaStream_t st) {
    // Enough threads for the rows (a warp each, eight per block), at most eight blocks
    // per SM; the weights are walked grid-stride.
    long long blocks = ((long long)M + 7) / 8;
    if (blocks < (N * dim / 8 + 255) / 256) blocks = (N * dim / 8 + 255) / 256;
    if (blocks > 152 * 8) blocks = 152 * 8;
    return launch_k(prologue_prep_kernel, dim3((unsigned)blocks), dim3(256), 0, st,
                    static_cast<const __nv_bfloat16*>(w), static_cast<const __nv_bfloat16*>(gamma),
                    static_cast<__nv_bfloat16*>(wg), N * dim / 8, static_cast<const __nv_bfloat16*>(x), inv_rms, M,
                    dim, eps);
}

cudaError_t launch_qkv_prologue(const CUtensorMap& tx, const CUtensorMap& tw, const ProArgs& a, cudaStream_t st) {
    auto kfn = a.D == 32 ? qkv_prologue_kernel<32> : a.D == 64 ? qkv_prologue_kernel<64> : qkv_prologue_kernel<128>;
    cudaError_t e = cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, ProCfg::SMEM);
    if (e != cudaSuccess) return e;
    const int N = (a.Hq + 2 * a.Hkv) * a.D;
    const int tiles = ((N + ProCfg::BN - 1) / ProCfg::BN) * ((a.M + ProCfg::BM - 1) / ProCfg::BM);
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    // Persistent: one CTA per SM (the ring takes most of the shared memory), each walking
    // its tiles.
    dim3 grid(tiles < sms ? tiles : sms);
    return launch_k(kfn, grid, dim3(ProCfg::THREADS), ProCfg::SMEM, st, tx, tw, a);
}

}  // namespace ne
