// skinny.cu -- fp8_gemm for few tokens (M <= 128: the decode shapes).
//
// The same block-scaled product as fp8_gemm_kernel ("DeepSeek-V3"
// repository overview, section "FP8 混合精度训练", the linear() excerpt):
//   y[m, n] = bf16( sum_kb RN32(sx[m, kb] * sw[n / 128, kb]) * P_kb[m, n] ),
// P_kb the exact sum over the 128 k of chunk kb of dec(xq) * dec(wq).
//
// With a handful of tokens the work is reading the weight.  So the weight's
// rows take the MMA's 128-row side (a 128-row tile is one row of weight-scale
// blocks, so sw is one number per chunk) and the tokens the N side (padded
// to a multiple of 16); a cluster of S <= 8 CTAs splits K, and its CTAs add their
// partial sums through distributed shared memory: one launch, no workspace.
// Per CTA (192 threads): warp 0 issues the TMA loads of all its chunks at
// once (one stage each), warp 1 the MMAs (four tcgen05.mma.kind::f8f6f4,
// M 128, N = tokens, K 32, per chunk, each chunk into its own TMEM columns,
// so nothing waits for a buffer to be read), warps 2-5 the promotion
// (acc = fma(RN(sx * sw), P_kb, acc) in fp32, chunks in order).  The
// cluster then sums the S partials in rank order, each CTA a 1/S share of
// the tile's rows, and writes bf16.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "internal.h"
#include "ptx.cuh"

namespace fp8bs {
namespace {

constexpr int kSkRows = 128;      // weight rows per tile = TMEM lanes
constexpr int kSkBK = 128;        // K chunk in bytes (fp8 elements) = one scale block
constexpr int kSkMaxTok = 128;    // tokens (MMA N) at most
constexpr int kSkMaxSplit = 8;    // CTAs per cluster (the portable maximum)
constexpr int kSkMaxChunks = 8;   // chunks per CTA: one stage and NP TMEM columns each
constexpr int kSkStageSpace = 192 * 1024;  // shared memory for the stages
constexpr int kSkThreads = 192;
constexpr int kSkEpiWarp0 = 2;    // warps 2-5: TMEM lane quarters 2, 3, 0, 1
static_assert(kSkThreads == 32 * (kSkEpiWarp0 + 4), "one promotion warp per TMEM lane quarter");

// A stage is the weight tile (16 KB) and the token tile (NP rows of 128
// bytes), rounded up to the 128-byte swizzle's 1024-byte atoms: 18 KB for 16
// tokens, 24 KB for 64, 32 KB for 128.
__host__ __device__ constexpr int sk_stage_bytes(int np) { return (kSkRows * kSkBK + np * kSkBK + 1023) / 1024 * 1024; }
// chunks a CTA can hold: one stage and NP TMEM columns (of 512) each
__host__ __device__ constexpr int sk_min(int a, int b) { return a < b ? a : b; }
__host__ __device__ constexpr int sk_max_chunks(int np) {
    return sk_min(sk_min(kSkMaxChunks, 512 / np), kSkStageSpace / sk_stage_bytes(np));
}

struct SkLayout {
    static constexpr int A_BYTES = kSkRows * kSkBK;   // weight tile, 16 KB
    static constexpr int STAGES_END = kSkStageSpace;
    // partial sums [NP][128] fp32, over the stages once every MMA is done
    static constexpr int OFF_RED = 0;
    // promotion factors RN(sx * sw) [chunk][token]
    static constexpr int OFF_F = STAGES_END;
    static constexpr int OFF_BAR = OFF_F + kSkMaxChunks * kSkMaxTok * 4;
    static constexpr int NUM_BARS = 2 * kSkMaxChunks;  // full[j], tfull[j]
    static constexpr int OFF_TMEM = OFF_BAR + NUM_BARS * 8;
    static constexpr int OFF_ABORT = OFF_TMEM + 4;
    static constexpr int BYTES = OFF_ABORT + 4;
    static constexpr int ALLOC = BYTES + 1024;
    static constexpr uint32_t TMEM_COLS = 512;
    static_assert(kSkMaxTok * kSkRows * 4 <= STAGES_END, "the partial sums fit over the stages");
    static_assert(sk_max_chunks(16) == kSkMaxChunks && sk_max_chunks(64) == kSkMaxChunks && sk_max_chunks(128) == 4,
                  "chunks per CTA");
    static_assert(ALLOC <= 227 * 1024, "shared memory per CTA");
};

struct SkParams {
    const float* sx;  // [M, lds]
    int64_t lds;
    const float* sw;  // [ceil(N / 128), KB]
    uint16_t* y;      // [M, ldy]
    int64_t ldy;
    int M, N, KB;
    int NP;           // tokens padded to a multiple of 16 (MMA N)
    int stage;        // bytes per stage, sk_stage_bytes(NP)
    int S;            // CTAs per cluster (K slices)
    int kps;          // chunks per slice
    unsigned* err;
    uint64_t timeout_ns;
};

__device__ __forceinline__ void drain_wait_sk(uint32_t bar, uint32_t parity, const WaitCtl& ctl) {
    int no_abort = 0;
    WaitCtl c2{&no_abort, ctl.err, ctl.timeout_ns};
    bounded_wait(bar, parity, c2);
}

__global__ void __launch_bounds__(kSkThreads, 1)
    fp8_gemm_skinny_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                           const __grid_constant__ SkParams p) {
    using L = SkLayout;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw_s + 1023u) & ~1023u) - raw_s);
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const int tile = blockIdx.x / p.S;
    const int n0 = tile * kSkRows;
    const int kb0 = static_cast<int>(rank) * p.kps;
    const int nk = max(0, min(p.KB, kb0 + p.kps) - kb0);  // this CTA's chunks
    const uint32_t bar0 = sbase + L::OFF_BAR;
    auto full_bar = [&](int j) { return bar0 + 8u * j; };
    auto tfull_bar = [&](int j) { return bar0 + 8u * (kSkMaxChunks + j); };
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_ABORT);
    float* fac = reinterpret_cast<float*>(smem + L::OFF_F);

    if (threadIdx.x == 0) {
        for (int j = 0; j < kSkMaxChunks; ++j) {
            mbar_init(full_bar(j), 1);
            mbar_init(tfull_bar(j), 1);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    // launched with programmatic stream serialisation: the set-up above ran
    // while the kernel before may still be finishing; every global read
    // (operands, scales) and the TMEM allocation come after this wait
    grid_dependency_wait();
    allow_dependents();
    __syncthreads();
    if (warp == 0 && lane == 0) {
        // every chunk of the slice at once, one stage each
        tma_prefetch_desc(&tmW);
        tma_prefetch_desc(&tmX);
        for (int j = 0; j < nk; ++j) {
            const uint32_t st = sbase + static_cast<uint32_t>(j * p.stage);
            mbar_arrive_expect_tx(full_bar(j), static_cast<uint32_t>(L::A_BYTES + p.NP * kSkBK));
            tma_load_2d(st, &tmW, full_bar(j), (kb0 + j) * kSkBK, n0);
            tma_load_2d(st + L::A_BYTES, &tmX, full_bar(j), (kb0 + j) * kSkBK, 0);
        }
    }
    if (warp == 1) tmem_alloc(sbase + L::OFF_TMEM, L::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + L::OFF_TMEM);
    const WaitCtl ctl{abort_flag, p.err, p.timeout_ns};

    if (warp == 0) {
        // every issued load must land before the CTA's shared memory goes away
        if (lane == 0)
            for (int j = 0; j < nk; ++j) drain_wait_sk(full_bar(j), 0, ctl);
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = idesc_e4m3_f32(kSkRows, p.NP);
            for (int j = 0; j < nk; ++j) {
                if (!bounded_wait(full_bar(j), 0, ctl)) break;
                tc_fence_after();
                const uint32_t st = sbase + static_cast<uint32_t>(j * p.stage);
                const uint64_t adesc = sdesc_kmajor_sw128(st);
                const uint64_t bdesc = sdesc_kmajor_sw128(st + L::A_BYTES);
                const uint32_t d = tmem + static_cast<uint32_t>(j * p.NP);
#pragma unroll
                for (int k = 0; k < kSkBK / 32; ++k)  // +32 bytes along K = +2 in the address field
                    umma_e4m3(d, adesc + 2u * k, bdesc + 2u * k, idesc, k > 0 ? 1u : 0u);
                umma_commit(tfull_bar(j));
            }
        }
        __syncwarp();
    } else {
        // promotion: this thread's weight row (TMEM lane), every token column
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const uint32_t taddr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
        // promotion factors RN(sx[m, kb] * sw[tile, kb]) (tokens past M get
        // 0), formed while the first chunk is in flight; the four promotion
        // warps meet at a named barrier before any wait, so all of them reach it
        const int pt = threadIdx.x - 32 * kSkEpiWarp0;
        for (int i = pt; i < nk * p.NP; i += 128) {
            const int j = i / p.NP, m = i % p.NP;
            const int kb = kb0 + j;
            fac[j * kSkMaxTok + m] =
                m < p.M ? __fmul_rn(__ldg(p.sx + static_cast<int64_t>(m) * p.lds + kb),
                                    __ldg(p.sw + static_cast<int64_t>(tile) * p.KB + kb))
                        : 0.0f;
        }
        asm volatile("bar.sync 1, 128;" ::: "memory");
        float acc[kSkMaxTok];
#pragma unroll
        for (int c = 0; c < kSkMaxTok; ++c) acc[c] = 0.0f;
        for (int j = 0; j < nk; ++j) {
            if (!warp_wait(tfull_bar(j), 0, ctl)) break;
            tc_fence_after();
            const float* f = fac + j * kSkMaxTok;
#pragma unroll
            for (int u = 0; u < kSkMaxTok / 16; ++u) {
                if (u * 16 < p.NP) {
                    uint64_t pr[8];
                    tmem_ld_x16_pairs(taddr + static_cast<uint32_t>(j * p.NP + 16 * u), pr);
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        acc[16 * u + 2 * i] = __fmaf_rn(f[16 * u + 2 * i], lo_f32(pr[i]), acc[16 * u + 2 * i]);
                        acc[16 * u + 2 * i + 1] =
                            __fmaf_rn(f[16 * u + 2 * i + 1], hi_f32(pr[i]), acc[16 * u + 2 * i + 1]);
                    }
                }
            }
        }
        // the partial sums, token-major, over the (consumed) stages; those
        // were last written by TMA (async proxy)
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        float* red = reinterpret_cast<float*>(smem + L::OFF_RED);
#pragma unroll
        for (int c = 0; c < kSkMaxTok; ++c)
            if (c < p.NP) red[c * kSkRows + row] = acc[c];
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, L::TMEM_COLS);
    }
    cluster_sync_all();  // every CTA's partial sums are complete and visible
    // this CTA's share of the tile's rows (rp, a multiple of 4): sum the S
    // partials in rank order, four rows at a time, two groups' loads in flight
    const int rp = ((kSkRows + p.S - 1) / p.S + 3) / 4 * 4;
    const int r_lo = static_cast<int>(rank) * rp;
    const int g4 = rp / 4;
    const uint32_t red0 = sbase + L::OFF_RED;
    auto group_load = [&](int g, float4 (&v)[kSkMaxSplit]) {
        const int m = g / g4;
        const int r = r_lo + 4 * (g % g4);
        const bool live = r < kSkRows && m < p.M;
        const uint32_t off = static_cast<uint32_t>((m * kSkRows + r) * 4);
#pragma unroll
        for (int q = 0; q < kSkMaxSplit; ++q)
            v[q] = (live && q < p.S) ? ld_cluster_v4f32(mapa_rank(red0 + off, static_cast<uint32_t>(q)))
                                     : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    };
    auto group_store = [&](int g, const float4 (&v)[kSkMaxSplit]) {
        const int m = g / g4;
        const int r = r_lo + 4 * (g % g4);
        const int n = n0 + r;
        if (r >= kSkRows || m >= p.M || n >= p.N) return;
        float4 sum = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
        for (int q = 0; q < kSkMaxSplit; ++q) {
            if (q < p.S) {
                sum.x = __fadd_rn(sum.x, v[q].x);
                sum.y = __fadd_rn(sum.y, v[q].y);
                sum.z = __fadd_rn(sum.z, v[q].z);
                sum.w = __fadd_rn(sum.w, v[q].w);
            }
        }
        uint16_t* yr = p.y + static_cast<int64_t>(m) * p.ldy + n;
        const uint16_t b0 = __bfloat16_as_ushort(__float2bfloat16_rn(sum.x));
        const uint16_t b1 = __bfloat16_as_ushort(__float2bfloat16_rn(sum.y));
        const uint16_t b2 = __bfloat16_as_ushort(__float2bfloat16_rn(sum.z));
        const uint16_t b3 = __bfloat16_as_ushort(__float2bfloat16_rn(sum.w));
        if (n + 3 < p.N) {  // y is 16-byte aligned and ldy % 8 == 0: n % 4 == 0 is 8-byte aligned
            *reinterpret_cast<uint2*>(yr) = make_uint2(b0 | (static_cast<uint32_t>(b1) << 16),
                                                       b2 | (static_cast<uint32_t>(b3) << 16));
        } else {
            yr[0] = b0;
            if (n + 1 < p.N) yr[1] = b1;
            if (n + 2 < p.N) yr[2] = b2;
        }
    };
    const int ng = g4 * p.M;
    for (int g = threadIdx.x; g < ng; g += 2 * kSkThreads) {
        float4 va[kSkMaxSplit], vb[kSkMaxSplit];
        group_load(g, va);
        const bool second = g + kSkThreads < ng;
        if (second) group_load(g + kSkThreads, vb);
        group_store(g, va);
        if (second) group_store(g + kSkThreads, vb);
    }
    cluster_sync_all();  // no CTA leaves while a peer may still read its partial sums
}

}  // namespace

static int sk_np(int64_t M) { return static_cast<int>(std::max<int64_t>(16, (M + 15) / 16 * 16)); }

bool gemm_skinny_applies(int64_t M, int64_t N, int64_t K) {
    if (M < 1 || M > kSkMaxTok || N < 1 || K < kSkBK || K % kSkBK != 0) return false;
    return K / kSkBK <= static_cast<int64_t>(kSkMaxSplit) * sk_max_chunks(sk_np(M));
}

cudaError_t launch_gemm_skinny(const GemmArgs& a, const DeviceInfo& dev, cudaStream_t stream) {
    if (!gemm_skinny_applies(a.M, a.N, a.K)) return cudaErrorInvalidValue;
    {
        static bool ready[64];
        if (dev.device < 0 || dev.device >= 64) return cudaErrorInvalidDevice;
        if (!ready[dev.device]) {
            const cudaError_t e = cudaFuncSetAttribute(fp8_gemm_skinny_kernel,
                                                       cudaFuncAttributeMaxDynamicSharedMemorySize, SkLayout::ALLOC);
            if (e != cudaSuccess) return e;
            ready[dev.device] = true;
        }
    }
    SkParams p{};
    p.sx = a.sx;
    p.lds = a.lds;
    p.sw = a.sw;
    p.y = a.y;
    p.ldy = a.ldy;
    p.M = static_cast<int>(a.M);
    p.N = static_cast<int>(a.N);
    p.KB = static_cast<int>(a.K / kSkBK);
    p.NP = sk_np(a.M);
    p.stage = sk_stage_bytes(p.NP);
    p.kps = (p.KB + kSkMaxSplit - 1) / kSkMaxSplit;  // <= sk_max_chunks(NP), by gemm_skinny_applies
    p.S = (p.KB + p.kps - 1) / p.kps;                 // every CTA gets at least one chunk
    p.err = dev.err;
    p.timeout_ns = wait_timeout_ns();
    // weight rows: boxes of 128 rows x 128 bytes; tokens: boxes of NP rows
    // (rows past M read as zero)
    CUtensorMap tmW, tmX;
    cudaError_t e;
    if ((e = make_tmap_2d(&tmW, a.wq, 1, a.K, a.N, a.K, kSkBK, kSkRows, 128)) != cudaSuccess) return e;
    if ((e = make_tmap_2d(&tmX, a.xq, 1, a.K, a.M, a.K, kSkBK, p.NP, 128)) != cudaSuccess) return e;
    const int tiles = static_cast<int>((a.N + kSkRows - 1) / kSkRows);
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(p.S);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(tiles * p.S));
    cfg.blockDim = dim3(kSkThreads);
    cfg.dynamicSmemBytes = SkLayout::ALLOC;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, fp8_gemm_skinny_kernel, tmW, tmX, p);
}

}  // namespace fp8bs
