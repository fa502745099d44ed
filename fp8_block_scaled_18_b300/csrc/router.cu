// router.cu -- the MoE router on the device: gate logits on the tensor cores
// (bf16 x bf16 -> fp32), sigmoid affinities, bias-steered group-limited
// top-k and the gate values, then the routing tables by a stable counting
// sort of the selections by expert.
//
// What it follows: sigmoid scoring, 8 expert groups of which 4 are kept,
// top-8 of 256, route_scale 2.5 (config block of "671B 参数如何「激活」37B？");
// the per-expert bias enters the selection only, the FFN output keeps the
// original affinities, and no token is dropped (page 2 of the DeepSeek-V3
// notes, section 2-2); gating stays in higher precision than FP8 (section
// 2-4 of the same notes), so the logits come from bf16 operands with fp32
// accumulation.  Where the pages are silent: a group's score is the largest
// biased affinity in it, ties go to the lower index, and the gate values are
// the chosen affinities normalised to sum 1, times route_scale.
#include <cuda.h>
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace fp8bs {
namespace {

// ------------------------------------------------------------------ gate
//
// One CTA per 128 tokens, 192 threads: warp 0 TMA producer (x tile 128 x 64
// bf16 and the gate weight E x 64 bf16 per 128-byte K chunk, 128-byte
// swizzle, kGateStages-deep ring), warp 1 MMA issuer (four
// tcgen05.mma.kind::f16, M 128, N E, K 16, per chunk, all accumulating in one
// TMEM region of E fp32 columns; owns the TMEM allocation), warps 2-5 the
// epilogue, one token (TMEM lane) per thread: after the last chunk each
// thread reads its E logits back twice from TMEM -- first for the group
// scores, then for the top-k inside the kept groups -- and writes its ids
// and gate values.
constexpr int kGateM = 128;
constexpr int kGateK = 64;            // bf16 elements per 128-byte chunk
constexpr int kGateStages = 4;
constexpr int kGateMaxE = 256;
constexpr int kGateMaxGroups = 32;
constexpr int kGateMaxTopK = 16;

struct GateLayout {
    static constexpr int A_BYTES = kGateM * 128;
    static constexpr int B_BYTES = kGateMaxE * 128;
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = kGateStages * A_BYTES;
    static constexpr int OFF_BAR = OFF_B + kGateStages * B_BYTES;  // full[S], empty[S], done
    static constexpr int NUM_BARS = 2 * kGateStages + 1;
    static constexpr int OFF_TMEM = OFF_BAR + NUM_BARS * 8;
    static constexpr int OFF_ABORT = OFF_TMEM + 4;
    static constexpr int OFF_BIAS = (OFF_ABORT + 4 + 15) & ~15;
    static constexpr int BYTES = OFF_BIAS + kGateMaxE * 4;
    static constexpr int ALLOC = BYTES + 1024;
    static constexpr uint32_t TMEM_COLS = 256;
};

struct GateParams {
    const float* bias;  // [E] or nullptr
    int32_t* ids;       // [T, top_k]
    float* w;           // [T, top_k]
    int T, KB, E, n_groups, topk_groups, top_k;
    float route_scale;
    unsigned* err;
    uint64_t timeout_ns;
};

// tcgen05.mma kind::f16, fp32 accumulate, A = B = bf16, both K-major, M x N.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Waits on an mbarrier while draining async work before exit: ignores the
// abort flag (the work must land first) but keeps the time limit.
__device__ __forceinline__ bool drain_wait_g(uint32_t bar, uint32_t parity, const WaitCtl& ctl) {
    int no_abort = 0;
    WaitCtl c2{&no_abort, ctl.err, ctl.timeout_ns};
    const bool ok = bounded_wait(bar, parity, c2);
    __syncwarp();
    return ok;
}

__device__ __forceinline__ float sigmoid_f32(float v) { return __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-v))); }

__global__ void __launch_bounds__(192, 1)
    moe_gate_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                    const __grid_constant__ GateParams p) {
    using L = GateLayout;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw_s + 1023u) & ~1023u) - raw_s);
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t bar0 = sbase + L::OFF_BAR;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (kGateStages + s); };
    const uint32_t done_bar = bar0 + 8u * (2 * kGateStages);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_ABORT);
    float* bias_s = reinterpret_cast<float*>(smem + L::OFF_BIAS);

    if (threadIdx.x == 32) {
        tma_prefetch_desc(&tmX);
        tma_prefetch_desc(&tmW);
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < kGateStages; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        mbar_init(done_bar, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    grid_dependency_wait();
    allow_dependents();
    if (warp == 1) tmem_alloc(sbase + L::OFF_TMEM, L::TMEM_COLS);
    for (int e = threadIdx.x; e < p.E; e += blockDim.x) bias_s[e] = p.bias ? p.bias[e] : 0.0f;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + L::OFF_TMEM);
    const WaitCtl ctl{abort_flag, p.err, p.timeout_ns};
    const int m0 = blockIdx.x * kGateM;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        const uint32_t tx = static_cast<uint32_t>(L::A_BYTES + p.E * 128);
        int kb = 0;
        for (; kb < p.KB; ++kb) {
            const int s = kb % kGateStages;
            const uint32_t ph = (kb / kGateStages) & 1u;
            if (!warp_wait(empty_bar(s), ph ^ 1u, ctl)) break;
            if (lane == 0) {
                mbar_arrive_expect_tx(full_bar(s), tx);
                tma_load_2d(sbase + L::OFF_A + s * L::A_BYTES, &tmX, full_bar(s), kb * kGateK, m0);
                tma_load_2d(sbase + L::OFF_B + s * L::B_BYTES, &tmW, full_bar(s), kb * kGateK, 0);
            }
            __syncwarp();
        }
        // every issued load must land before the CTA's shared memory goes away
        const int first = kb > kGateStages ? kb - kGateStages : 0;
        for (int j = first; j < kb; ++j) drain_wait_g(full_bar(j % kGateStages), (j / kGateStages) & 1u, ctl);
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        const uint32_t idesc = idesc_bf16_f32(kGateM, p.E);
        bool issued = false;
        for (int kb = 0; kb < p.KB; ++kb) {
            const int s = kb % kGateStages;
            if (!warp_wait(full_bar(s), (kb / kGateStages) & 1u, ctl)) break;
            tc_fence_after();
            if (lane == 0) {
                const uint64_t adesc = sdesc_kmajor_sw128(sbase + L::OFF_A + s * L::A_BYTES);
                const uint64_t bdesc = sdesc_kmajor_sw128(sbase + L::OFF_B + s * L::B_BYTES);
#pragma unroll
                for (int k = 0; k < 4; ++k)  // K 16 = 32 bytes = +2 in the address field
                    umma_bf16(tmem, adesc + 2u * k, bdesc + 2u * k, idesc, (kb > 0 || k > 0) ? 1u : 0u);
                umma_commit(empty_bar(s));
            }
            issued = true;
            __syncwarp();
        }
        // Publish the sums (also after a wait that gave up: the status word
        // then reports the failure and the outputs are not to be used).
        if (lane == 0) umma_commit(done_bar);
        __syncwarp();
        if (issued) drain_wait_g(done_bar, 0, ctl);
    } else {
        // ------------------------------------------------------------ epilogue
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const int m = m0 + row;
        const uint32_t taddr0 = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
        const bool ok = warp_wait(done_bar, 0, ctl);
        tc_fence_after();
        if (ok) {
            const int per = p.E / p.n_groups;
            float gmax[kGateMaxGroups];
            for (int g = 0; g < p.n_groups; ++g) gmax[g] = -INFINITY;
            // pass 1: group scores (largest biased affinity per group)
            for (int c = 0; c < p.E; c += 16) {
                uint64_t pr[8];
                __syncwarp();
                tmem_ld_x16_pairs(taddr0 + c, pr);
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int e = c + i;
                    const float l = (i & 1) ? hi_f32(pr[i >> 1]) : lo_f32(pr[i >> 1]);
                    const float b = __fadd_rn(sigmoid_f32(l), bias_s[e]);
                    const int g = e / per;
                    gmax[g] = fmaxf(gmax[g], b);
                }
            }
            // the best topk_groups groups, lower index on ties
            uint32_t keep = 0;
            for (int r = 0; r < p.topk_groups; ++r) {
                int best = -1;
                for (int g = 0; g < p.n_groups; ++g)
                    if (!((keep >> g) & 1u) && (best < 0 || gmax[g] > gmax[best])) best = g;
                keep |= 1u << best;
            }
            // pass 2: top-k of the kept groups' experts by biased affinity,
            // kept sorted (descending; an equal score goes after: lower index first)
            float tb[kGateMaxTopK], ts[kGateMaxTopK];
            int te[kGateMaxTopK];
            int n = 0;
            for (int c = 0; c < p.E; c += 16) {
                // every lane loads every slice (the kept groups differ per
                // token, and the TMEM load is a warp-wide instruction)
                uint64_t pr[8];
                __syncwarp();
                tmem_ld_x16_pairs(taddr0 + c, pr);
                for (int i = 0; i < 16; ++i) {
                    const int e = c + i;
                    if (!((keep >> (e / per)) & 1u)) continue;
                    const float l = (i & 1) ? hi_f32(pr[i >> 1]) : lo_f32(pr[i >> 1]);
                    const float s = sigmoid_f32(l);
                    const float b = __fadd_rn(s, bias_s[e]);
                    if (n == p.top_k && !(b > tb[n - 1])) continue;
                    int pos = n < p.top_k ? n : p.top_k - 1;
                    while (pos > 0 && tb[pos - 1] < b) {
                        tb[pos] = tb[pos - 1];
                        ts[pos] = ts[pos - 1];
                        te[pos] = te[pos - 1];
                        --pos;
                    }
                    tb[pos] = b;
                    ts[pos] = s;
                    te[pos] = e;
                    if (n < p.top_k) ++n;
                }
            }
            if (m < p.T) {
                float ssum = 0.0f;
                for (int r = 0; r < p.top_k; ++r) ssum = __fadd_rn(ssum, ts[r]);
                int32_t* idr = p.ids + static_cast<int64_t>(m) * p.top_k;
                float* wr = p.w + static_cast<int64_t>(m) * p.top_k;
                for (int r = 0; r < p.top_k; ++r) {
                    idr[r] = te[r];
                    wr[r] = __fmul_rn(__fdiv_rn(ts[r], ssum), p.route_scale);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, L::TMEM_COLS);
    }
}

// ------------------------------------------------------------------ routing tables
//
// One CTA of 1024 threads.  The expert counts come from shared-memory
// atomics (a count is the same whatever the order), their exclusive scan
// gives the offsets, and each selection's row is offsets[e] + the number of
// earlier tokens that chose e.  That rank is formed without any ordering
// race: tokens are taken 1024 at a time, one per thread; each warp marks, per
// expert, the lanes that chose it (a 32-bit mask built with atomicOr), a scan
// over the warps gives each warp's base per expert, and a lane's rank is its
// warp's base plus the number of lower lanes in the mask.  Rows start as
// token -1 / gate 0, so a row no selection reaches (a token naming an expert
// twice) is visible as an out-of-range id downstream.
constexpr int kRouteThreads = 1024;
constexpr int kRouteWarps = kRouteThreads / 32;
constexpr int kRouteMaxE = 256;

struct RouteSmem {
    uint32_t mask[kRouteWarps][kRouteMaxE];
    int32_t base[kRouteWarps][kRouteMaxE];
    int32_t next[kRouteMaxE];
    int32_t scan[kRouteMaxE + 1];
};

__global__ void __launch_bounds__(kRouteThreads, 1)
    moe_route_kernel(const int32_t* __restrict__ ids, const float* __restrict__ w, int T, int top_k, int E,
                     int32_t* __restrict__ offsets, int32_t* __restrict__ token_of_row,
                     int32_t* __restrict__ rows_of_token, float* __restrict__ weight_of_row,
                     unsigned* __restrict__ err) {
    extern __shared__ uint8_t route_smem_raw[];
    RouteSmem& sm = *reinterpret_cast<RouteSmem*>(route_smem_raw);
    auto& mask = sm.mask;
    auto& base = sm.base;
    auto& next = sm.next;
    auto& scan = sm.scan;
    grid_dependency_wait();
    allow_dependents();
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int wp = tid >> 5;
    const int64_t R = static_cast<int64_t>(T) * top_k;
    for (int e = tid; e < E; e += kRouteThreads) next[e] = 0;
    for (int64_t r = tid; r < R; r += kRouteThreads) {
        token_of_row[r] = -1;
        weight_of_row[r] = 0.0f;
    }
    __syncthreads();
    // counts
    bool bad = false;
    for (int64_t i = tid; i < R; i += kRouteThreads) {
        const int e = ids[i];
        if (e >= 0 && e < E) atomicAdd(&next[e], 1); else bad = true;
    }
    __syncthreads();
    // exclusive scan of the counts (one warp; E <= 256)
    if (wp == 0) {
        int run = 0;
        for (int e0 = 0; e0 < E; e0 += 32) {
            const int e = e0 + lane;
            const int c = e < E ? next[e] : 0;
            int incl = c;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += v;
            }
            if (e < E) scan[e] = run + incl - c;
            run += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) scan[E] = run;
    }
    __syncthreads();
    for (int e = tid; e <= E; e += kRouteThreads) offsets[e] = scan[e];
    for (int e = tid; e < E; e += kRouteThreads) next[e] = scan[e];  // first free row of each expert
    __syncthreads();
    const uint32_t lt = (1u << lane) - 1u;
    for (int t0 = 0; t0 < T; t0 += kRouteThreads) {
        for (int i = tid; i < kRouteWarps * E; i += kRouteThreads) mask[i / E][i % E] = 0u;
        __syncthreads();
        const int t = t0 + tid;
        if (t < T) {
            for (int k = 0; k < top_k; ++k) {
                const int e = ids[static_cast<int64_t>(t) * top_k + k];
                if (e >= 0 && e < E) {
                    const uint32_t old = atomicOr(&mask[wp][e], 1u << lane);
                    if (old & (1u << lane)) bad = true;  // the same expert twice for one token
                }
            }
        }
        __syncthreads();
        for (int e = tid; e < E; e += kRouteThreads) {
            int run = next[e];
            for (int q = 0; q < kRouteWarps; ++q) {
                base[q][e] = run;
                run += __popc(mask[q][e]);
            }
            next[e] = run;
        }
        __syncthreads();
        if (t < T) {
            for (int k = 0; k < top_k; ++k) {
                const int64_t i = static_cast<int64_t>(t) * top_k + k;
                const int e = ids[i];
                int32_t r = -1;
                if (e >= 0 && e < E) {
                    r = base[wp][e] + __popc(mask[wp][e] & lt);
                    token_of_row[r] = t;
                    weight_of_row[r] = w[i];
                }
                rows_of_token[i] = r;
            }
        }
        __syncthreads();
    }
    if (bad) atomicOr(err, kDevErrIndex);
}

}  // namespace

cudaError_t launch_moe_gate(const uint16_t* x, int64_t ldx, const uint16_t* wg, const float* bias, int64_t T,
                            int64_t dim, int E, int n_groups, int topk_groups, int top_k, float route_scale,
                            int32_t* ids, float* w, const DeviceInfo& dev, cudaStream_t stream) {
    CUtensorMap tmX, tmW;
    cudaError_t e;
    if ((e = make_tmap_2d(&tmX, x, 2, dim, T, ldx * 2, kGateK, kGateM, true)) != cudaSuccess) return e;
    if ((e = make_tmap_2d(&tmW, wg, 2, dim, E, dim * 2, kGateK, E, true)) != cudaSuccess) return e;
    {
        static bool ready[64];
        if (dev.device < 0 || dev.device >= 64) return cudaErrorInvalidDevice;
        if (!ready[dev.device]) {
            e = cudaFuncSetAttribute(moe_gate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, GateLayout::ALLOC);
            if (e != cudaSuccess) return e;
            ready[dev.device] = true;
        }
    }
    GateParams p{};
    p.bias = bias;
    p.ids = ids;
    p.w = w;
    p.T = static_cast<int>(T);
    p.KB = static_cast<int>(dim / kGateK);
    p.E = E;
    p.n_groups = n_groups;
    p.topk_groups = topk_groups;
    p.top_k = top_k;
    p.route_scale = route_scale;
    p.err = dev.err;
    p.timeout_ns = wait_timeout_ns();
    const int grid = static_cast<int>((T + kGateM - 1) / kGateM);
    return launch_pdl(moe_gate_kernel, dim3(grid), dim3(192), GateLayout::ALLOC, stream, tmX, tmW, p);
}

cudaError_t launch_moe_route(const int32_t* ids, const float* w, int64_t T, int top_k, int E, int32_t* offsets,
                             int32_t* token_of_row, int32_t* rows_of_token, float* weight_of_row,
                             const DeviceInfo& dev, cudaStream_t stream) {
    static bool ready[64];
    if (dev.device < 0 || dev.device >= 64) return cudaErrorInvalidDevice;
    if (!ready[dev.device]) {
        const cudaError_t e = cudaFuncSetAttribute(moe_route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(sizeof(RouteSmem)));
        if (e != cudaSuccess) return e;
        ready[dev.device] = true;
    }
    return launch_pdl(moe_route_kernel, dim3(1), dim3(kRouteThreads), sizeof(RouteSmem), stream, ids, w,
                      static_cast<int>(T), top_k, E, offsets, token_of_row, rows_of_token, weight_of_row, dev.err);
}

}  // namespace fp8bs
