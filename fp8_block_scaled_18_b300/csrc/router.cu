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

#include <algorithm>

#include "internal.h"
#include "ptx.cuh"

namespace fp8bs {
namespace {

// ------------------------------------------------------------------ gate
//
// One CTA per 128 tokens, 576 threads: warp 0 TMA producer (x tile 128 x 64
// bf16 and the gate weight E x 64 bf16 per 128-byte K chunk, 128-byte
// swizzle, kGateStages-deep ring), warp 1 MMA issuer (four
// tcgen05.mma.kind::f16, M 128, N E, K 16, per chunk, all accumulating in one
// TMEM region of E fp32 columns; owns the TMEM allocation), warps 2-17 the
// epilogue: four warps per TMEM lane quarter, each taking a quarter of the
// experts (columns) of its 32 tokens.  Once the sums are complete the
// pipeline's shared memory is reused:
//   1. each thread turns its columns' logits into affinities s = sigmoid(l)
//      and stores them, expert-major, in shared memory;
//   2. each thread forms the scores (largest s + bias) of the groups
//      g = its quarter index mod 4 for its token;
//   3. each thread picks its token's kept groups (all four threads of a token
//      pick the same ones) and keeps a sorted top-k of its columns inside
//      them by biased affinity, ties to the lower expert;
//   4. one thread per token merges the four partial lists (in expert
//      order, so ties still go to the lower expert), normalises the chosen
//      affinities and writes ids and gate values.
// The phases are separated by mbarriers with bounded waits.
constexpr int kGateM = 128;
constexpr int kGateK = 64;            // bf16 elements per 128-byte chunk
constexpr int kGateStages = 4;
constexpr int kGateMaxE = 256;
constexpr int kGateMaxGroups = 32;
constexpr int kGateMaxTopK = 16;
constexpr int kGateEpiWarp0 = 2;
constexpr int kGateEpiWarps = 16;
constexpr int kGateThreads = 32 * (kGateEpiWarp0 + kGateEpiWarps);

struct GateLayout {
    static constexpr int A_BYTES = kGateM * 128;
    static constexpr int B_BYTES = kGateMaxE * 128;
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = kGateStages * A_BYTES;
    // full[S], empty[S], done, then the epilogue's three phase barriers
    static constexpr int OFF_BAR = OFF_B + kGateStages * B_BYTES;
    static constexpr int NUM_BARS = 2 * kGateStages + 1 + 3;
    static constexpr int OFF_TMEM = OFF_BAR + NUM_BARS * 8;
    static constexpr int OFF_ABORT = OFF_TMEM + 4;
    static constexpr int OFF_BIAS = (OFF_ABORT + 4 + 15) & ~15;
    static constexpr int BYTES = OFF_BIAS + kGateMaxE * 4;
    static constexpr int ALLOC = BYTES + 1024;
    static constexpr uint32_t TMEM_COLS = 256;
    // epilogue tables, over the pipeline stages once the sums are complete:
    // affinities [E][128 tokens] fp32, group scores [32][128] fp32, partial
    // top-k lists [4 quarters][16][128] expert ids (int16)
    static constexpr int OFF_S = 0;
    static constexpr int OFF_G = OFF_S + kGateMaxE * kGateM * 4;
    static constexpr int OFF_P = OFF_G + kGateMaxGroups * kGateM * 4;
    static constexpr int EPI_END = OFF_P + 4 * kGateMaxTopK * kGateM * 2;
    static_assert(EPI_END <= OFF_BAR, "the epilogue tables fit in the pipeline stages");
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

// Sorted insertion of (v, e) into a descending list of n <= kGateMaxTopK
// entries (static indices, so the list stays in registers): an entry moves
// down only past strictly smaller values, so equal values keep the order in
// which they arrived.
__device__ __forceinline__ void topk_insert(float (&lb)[kGateMaxTopK], int (&le)[kGateMaxTopK], int n, float v,
                                            int e) {
#pragma unroll
    for (int i = 0; i < kGateMaxTopK; ++i) {
        if (i < n && v > lb[i]) {
            const float tb = lb[i];
            const int te = le[i];
            lb[i] = v;
            le[i] = e;
            v = tb;
            e = te;
        }
    }
}

__global__ void __launch_bounds__(kGateThreads, 1)
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
    auto phase_bar = [&](int i) { return bar0 + 8u * (2 * kGateStages + 1 + i); };
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
        for (int i = 0; i < 3; ++i) mbar_init(phase_bar(i), kGateEpiWarps);
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
        const int quarter = warp & 3;              // TMEM lane quarter this warp may read
        const int tok = quarter * 32 + lane;       // the token (TMEM lane) of this thread
        const int sl = (warp - kGateEpiWarp0) >> 2;  // which quarter of the experts
        const int m = m0 + tok;
        const uint32_t taddr0 = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
        // this thread's columns: 16-column units [u0, u1) of the E / 16
        const int units = p.E / 16;
        const int u0 = sl * units / 4, u1 = (sl + 1) * units / 4;
        const int per = p.E / p.n_groups;
        float* S = reinterpret_cast<float*>(smem + L::OFF_S);      // [e][tok]
        float* Gs = reinterpret_cast<float*>(smem + L::OFF_G);     // [g][tok]
        int16_t* P = reinterpret_cast<int16_t*>(smem + L::OFF_P);  // [sl][k][tok]
        auto phase = [&](int i) {  // all epilogue warps reach phase i
            __syncwarp();
            if (lane == 0) mbar_arrive(phase_bar(i));
            return warp_wait(phase_bar(i), 0, ctl);
        };
        bool ok = warp_wait(done_bar, 0, ctl);
        tc_fence_after();
        // the stages were last written by TMA (async proxy); the tables below
        // overwrite them with ordinary stores
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        // 1. affinities of this thread's columns
        if (ok) {
            for (int u = u0; u < u1; ++u) {
                uint64_t pr[8];
                tmem_ld_x16_pairs(taddr0 + 16 * u, pr);
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float l = (i & 1) ? hi_f32(pr[i >> 1]) : lo_f32(pr[i >> 1]);
                    S[(16 * u + i) * kGateM + tok] = sigmoid_f32(l);
                }
            }
        }
        ok = phase(0) && ok;
        // 2. group scores: the largest biased affinity of each group g = sl (mod 4)
        if (ok) {
            for (int g = sl; g < p.n_groups; g += 4) {
                float gm = -INFINITY;
                for (int e = g * per; e < (g + 1) * per; ++e) gm = fmaxf(gm, __fadd_rn(S[e * kGateM + tok], bias_s[e]));
                Gs[g * kGateM + tok] = gm;
            }
        }
        ok = phase(1) && ok;
        // 3. the kept groups (the topk_groups best, lower index on ties), then
        //    a sorted top-k of this thread's columns inside them
        if (ok) {
            uint32_t keep = 0;
            for (int r = 0; r < p.topk_groups; ++r) {
                int best = -1;
                float bv = 0.0f;
                for (int g = 0; g < p.n_groups; ++g) {
                    const float v = Gs[g * kGateM + tok];
                    if (!((keep >> g) & 1u) && (best < 0 || v > bv)) {
                        best = g;
                        bv = v;
                    }
                }
                keep |= 1u << best;
            }
            float lb[kGateMaxTopK];
            int le[kGateMaxTopK];
#pragma unroll
            for (int i = 0; i < kGateMaxTopK; ++i) {
                lb[i] = -INFINITY;
                le[i] = -1;
            }
            for (int e = 16 * u0; e < 16 * u1; ++e) {
                if (!((keep >> (e / per)) & 1u)) continue;
                topk_insert(lb, le, p.top_k, __fadd_rn(S[e * kGateM + tok], bias_s[e]), e);
            }
#pragma unroll
            for (int i = 0; i < kGateMaxTopK; ++i)
                if (i < p.top_k) P[(sl * kGateMaxTopK + i) * kGateM + tok] = static_cast<int16_t>(le[i]);
        }
        ok = phase(2) && ok;
        // 4. merge the four lists (in expert order), gate values, outputs
        if (ok && sl == 0 && m < p.T) {
            float lb[kGateMaxTopK];
            int le[kGateMaxTopK];
#pragma unroll
            for (int i = 0; i < kGateMaxTopK; ++i) {
                lb[i] = -INFINITY;
                le[i] = -1;
            }
            for (int q = 0; q < 4; ++q) {
                for (int i = 0; i < p.top_k; ++i) {
                    const int e = P[(q * kGateMaxTopK + i) * kGateM + tok];
                    if (e < 0) break;  // a shorter list (fewer kept columns than top_k)
                    topk_insert(lb, le, p.top_k, __fadd_rn(S[e * kGateM + tok], bias_s[e]), e);
                }
            }
            float ls[kGateMaxTopK];
            float ssum = 0.0f;
#pragma unroll
            for (int r = 0; r < kGateMaxTopK; ++r) {
                if (r < p.top_k) {
                    ls[r] = S[le[r] * kGateM + tok];
                    ssum = __fadd_rn(ssum, ls[r]);
                }
            }
            int32_t* idr = p.ids + static_cast<int64_t>(m) * p.top_k;
            float* wr = p.w + static_cast<int64_t>(m) * p.top_k;
#pragma unroll
            for (int r = 0; r < kGateMaxTopK; ++r) {
                if (r < p.top_k) {
                    idr[r] = le[r];
                    wr[r] = __fmul_rn(__fdiv_rn(ls[r], ssum), p.route_scale);
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
// Several CTAs, each owning a contiguous chunk of tokens.  Every CTA counts
// all the selections per expert (shared-memory atomics: a count is the same
// whatever the order), splitting them into those of tokens before its chunk
// and those of its own tokens; the exclusive scan of the totals gives the
// offsets, and expert e's rows for the chunk start at offsets[e] + the count
// of earlier tokens that chose e.  Inside the chunk the rank of a selection
// is formed without any ordering race: tokens are taken kRouteThreads at a
// time, one per thread; each warp marks, per expert, the lanes that chose it
// (a 32-bit mask built with atomicOr), a scan over the warps gives each
// warp's base per expert, and a lane's rank is its warp's base plus the
// number of lower lanes in the mask.  The rows a chunk owns first get token
// -1 / gate 0, so a row no selection reaches (a token naming an expert
// twice) is visible as an out-of-range id downstream.  Re-reading every
// selection per CTA costs T * top_k * 4 bytes of L2 reads per CTA; the grid
// is capped at two CTAs per SM.
constexpr int kRouteThreads = 512;
constexpr int kRouteWarps = kRouteThreads / 32;
constexpr int kRouteMaxE = 256;
constexpr int kRouteChunk = 128;  // tokens per CTA, at least

struct RouteSmem {
    uint32_t mask[kRouteWarps][kRouteMaxE];
    int32_t base[kRouteWarps][kRouteMaxE];
    int32_t total[kRouteMaxE];
    int32_t before[kRouteMaxE];
    int32_t mine[kRouteMaxE];
    int32_t next[kRouteMaxE];
    int32_t scan[kRouteMaxE + 1];
};

__global__ void __launch_bounds__(kRouteThreads)
    moe_route_kernel(const int32_t* __restrict__ ids, const float* __restrict__ w, int T, int top_k, int E,
                     int chunk, int32_t* __restrict__ offsets, int32_t* __restrict__ token_of_row,
                     int32_t* __restrict__ rows_of_token, float* __restrict__ weight_of_row,
                     unsigned* __restrict__ err) {
    extern __shared__ uint8_t route_smem_raw[];
    RouteSmem& sm = *reinterpret_cast<RouteSmem*>(route_smem_raw);
    grid_dependency_wait();
    allow_dependents();
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int wp = tid >> 5;
    const int t_begin = blockIdx.x * chunk;
    const int t_end = min(T, t_begin + chunk);
    const int64_t R = static_cast<int64_t>(T) * top_k;
    const int64_t i_begin = static_cast<int64_t>(t_begin) * top_k;
    const int64_t i_end = static_cast<int64_t>(t_end) * top_k;
    for (int e = tid; e < E; e += kRouteThreads) {
        sm.total[e] = 0;
        sm.before[e] = 0;
        sm.mine[e] = 0;
    }
    __syncthreads();
    // counts over every selection: all tokens, those before this chunk, this chunk's
    bool bad = false;
    for (int64_t i = tid; i < R; i += kRouteThreads) {
        const int e = __ldg(ids + i);
        const bool own = i >= i_begin && i < i_end;
        if (e >= 0 && e < E) {
            atomicAdd(&sm.total[e], 1);
            if (i < i_begin) atomicAdd(&sm.before[e], 1);
            else if (own) atomicAdd(&sm.mine[e], 1);
        } else if (own) {
            bad = true;  // reported by the CTA that owns the token
        }
    }
    __syncthreads();
    // exclusive scan of the totals (one warp; E <= 256)
    if (wp == 0) {
        int run = 0;
        for (int e0 = 0; e0 < E; e0 += 32) {
            const int e = e0 + lane;
            const int c = e < E ? sm.total[e] : 0;
            int incl = c;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += v;
            }
            if (e < E) sm.scan[e] = run + incl - c;
            run += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) sm.scan[E] = run;
    }
    __syncthreads();
    if (blockIdx.x == 0)
        for (int e = tid; e <= E; e += kRouteThreads) offsets[e] = sm.scan[e];
    for (int e = tid; e < E; e += kRouteThreads) {
        const int first = sm.scan[e] + sm.before[e];  // this chunk's first row of expert e
        sm.next[e] = first;
        for (int r = first; r < first + sm.mine[e]; ++r) {
            token_of_row[r] = -1;
            weight_of_row[r] = 0.0f;
        }
    }
    const uint32_t lt = (1u << lane) - 1u;
    for (int t0 = t_begin; t0 < t_end; t0 += kRouteThreads) {
        for (int i = tid; i < kRouteWarps * E; i += kRouteThreads) sm.mask[i / E][i % E] = 0u;
        __syncthreads();
        const int t = t0 + tid;
        if (t < t_end) {
            for (int k = 0; k < top_k; ++k) {
                const int e = __ldg(ids + static_cast<int64_t>(t) * top_k + k);
                if (e >= 0 && e < E) {
                    const uint32_t old = atomicOr(&sm.mask[wp][e], 1u << lane);
                    if (old & (1u << lane)) bad = true;  // the same expert twice for one token
                }
            }
        }
        __syncthreads();
        for (int e = tid; e < E; e += kRouteThreads) {
            int run = sm.next[e];
            for (int q = 0; q < kRouteWarps; ++q) {
                sm.base[q][e] = run;
                run += __popc(sm.mask[q][e]);
            }
            sm.next[e] = run;
        }
        __syncthreads();
        if (t < t_end) {
            for (int k = 0; k < top_k; ++k) {
                const int64_t i = static_cast<int64_t>(t) * top_k + k;
                const int e = __ldg(ids + i);
                int32_t r = -1;
                if (e >= 0 && e < E) {
                    r = sm.base[wp][e] + __popc(sm.mask[wp][e] & lt);
                    token_of_row[r] = t;
                    weight_of_row[r] = __ldg(w + i);
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
    if ((e = make_tmap_2d(&tmX, x, 2, dim, T, ldx * 2, kGateK, kGateM, 128)) != cudaSuccess) return e;
    if ((e = make_tmap_2d(&tmW, wg, 2, dim, E, dim * 2, kGateK, E, 128)) != cudaSuccess) return e;
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
    return launch_pdl(moe_gate_kernel, dim3(grid), dim3(kGateThreads), GateLayout::ALLOC, stream, tmX, tmW, p);
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
    // chunks of at least kRouteChunk tokens, at most two per SM
    const int64_t max_chunks = std::max<int64_t>(1, 2 * static_cast<int64_t>(dev.num_sms));
    const int64_t nchunks = std::max<int64_t>(1, std::min<int64_t>((T + kRouteChunk - 1) / kRouteChunk, max_chunks));
    const int chunk = static_cast<int>(std::max<int64_t>(1, (T + nchunks - 1) / nchunks));
    // T == 0: one CTA still writes the (all-zero) offsets
    const int grid = static_cast<int>(std::max<int64_t>(1, (T + chunk - 1) / chunk));
    return launch_pdl(moe_route_kernel, dim3(grid), dim3(kRouteThreads), sizeof(RouteSmem), stream, ids, w,
                      static_cast<int>(T), top_k, E, chunk, offsets, token_of_row, rows_of_token, weight_of_row,
                      dev.err);
}

}  // namespace fp8bs
