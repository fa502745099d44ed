// quant.cu -- the HBM-bound kernels: act_quant (1x128 groups), weight_quant
// (128x128 blocks), weight_dequant, and the elementwise e4m3 encoder.
//
// Quantisation rule ("DeepSeek-V3" repository overview, section
// "FP8 混合精度训练"): s = amax / 448 over the group or block (fp32, IEEE
// round-to-nearest division), code = e4m3(x / s) with round-to-nearest-even
// and saturation at +-448; an all-zero group has s = 0 and +-0 codes.
#include <cuda_bf16.h>

#include "codec.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace fp8bs {
namespace {

__device__ __forceinline__ uint4 ld_stream(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// ---------------------------------------------------------------- act_quant
//
// Four lanes own one 128-channel group: lane j of the team loads the 16-byte
// chunks j, j+4, j+8, j+12 of the group (each load instruction of the team
// covers 64 contiguous bytes), the amax is reduced over the team with two
// xor-shuffles, and each lane writes its 32 codes as four 8-byte stores.  A
// warp handles eight groups per step; grid-stride over all groups.  Four
// lanes per group (rather than more) keeps the per-group work -- the
// shuffles and the scale -- small against the 32 elements each lane encodes.
constexpr int kAqTeam = 4;
constexpr int kAqGroupsPerWarp = 32 / kAqTeam;

template <bool POW2>
__global__ void __launch_bounds__(256) act_quant_kernel(const uint16_t* __restrict__ x, int64_t KB,
                                                       int64_t ldx, uint8_t* __restrict__ xq, int64_t ldq,
                                                       float* __restrict__ sx, int64_t lds,
                                                       int64_t total_groups) {
    grid_dependency_wait();  // the previous kernel may still read xq / sx
    allow_dependents();
    const int lane = threadIdx.x & 31;
    const int sub = lane & (kAqTeam - 1);
    const int team = lane / kAqTeam;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;

    for (int64_t base = warp * kAqGroupsPerWarp; base < total_groups; base += nwarps * kAqGroupsPerWarp) {
        const int64_t g = base + team;
        const bool valid = g < total_groups;
        uint4 v[4];
        int64_t m = 0, kb = 0;
        if (valid) {
            m = g / KB;
            kb = g - m * KB;
            const uint16_t* p = x + m * ldx + kb * 128;
#pragma unroll
            for (int i = 0; i < 4; ++i) v[i] = ld_stream(p + (sub + kAqTeam * i) * 8);
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) v[i] = make_uint4(0, 0, 0, 0);
        }
        uint32_t amax2 = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) amax2 = absmax_bits8(v[i], amax2);
        amax2 = __vmaxu2(amax2, __shfl_xor_sync(0xffffffffu, amax2, 1));
        amax2 = __vmaxu2(amax2, __shfl_xor_sync(0xffffffffu, amax2, 2));
        if (valid) {
            const float amax = bits_to_amax(amax2);
            const GroupScale gs = POW2 ? group_scale_pow2(amax) : group_scale(amax);
            const bool zero = (amax == 0.0f);
            uint8_t* q = xq + m * ldq + kb * 128;
#pragma unroll
            for (int i = 0; i < 4; ++i)
                *reinterpret_cast<uint2*>(q + (sub + kAqTeam * i) * 8) = encode8(v[i], gs, zero);
            if (sub == 0) sx[m * lds + kb] = gs.s;
        }
    }
}

// ---------------------------------------------------------------- weight_quant
//
// The launch picks 512 threads per block (four 16-byte loads in flight per
// thread) when there are few blocks -- a small weight would otherwise be
// latency-bound -- and 256 (eight loads per thread) otherwise.
//
// One CTA per 128x128 block.  Thread t reads the 16-byte chunk (t % 16) of
// rows (t / 16) + kWqRowStep j (each warp load covers two full
// 256-byte row segments), block amax via warp shuffles and shared memory.
template <int kWqThreads, bool POW2>
__global__ void __launch_bounds__(kWqThreads) weight_quant_kernel(const uint16_t* __restrict__ w, int64_t N, int64_t K,
                                                          uint8_t* __restrict__ wq, float* __restrict__ sw) {
    constexpr int kWqRowStep = kWqThreads / 16;  // rows between a thread's loads
    grid_dependency_wait();
    allow_dependents();
    constexpr int kWqRowsPerThread = 128 / kWqRowStep;
    __shared__ float warp_max[kWqThreads / 32];
    const int kb = blockIdx.x, nb = blockIdx.y;
    const int64_t KB = K / 128;
    const int t = threadIdx.x;
    const int chunk = t & 15;
    const int r0 = t >> 4;
    uint4 raw[kWqRowsPerThread];  // the block stays in registers as packed bf16
    uint32_t amax2 = 0;
#pragma unroll
    for (int j = 0; j < kWqRowsPerThread; ++j) {
        const int64_t n = static_cast<int64_t>(nb) * 128 + r0 + kWqRowStep * j;
        raw[j] = n < N ? ld_stream(w + n * K + static_cast<int64_t>(kb) * 128 + chunk * 8) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int j = 0; j < kWqRowsPerThread; ++j) amax2 = absmax_bits8(raw[j], amax2);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax2 = __vmaxu2(amax2, __shfl_xor_sync(0xffffffffu, amax2, o));
    if ((t & 31) == 0) warp_max[t >> 5] = bits_to_amax(amax2);
    __syncthreads();
    float amax = warp_max[0];
#pragma unroll
    for (int i = 1; i < kWqThreads / 32; ++i) amax = fmaxf(amax, warp_max[i]);
    const GroupScale gs = POW2 ? group_scale_pow2(amax) : group_scale(amax);
    const bool zero = (amax == 0.0f);
#pragma unroll
    for (int j = 0; j < kWqRowsPerThread; ++j) {
        const int64_t n = static_cast<int64_t>(nb) * 128 + r0 + kWqRowStep * j;
        if (n < N)
            *reinterpret_cast<uint2*>(wq + n * K + static_cast<int64_t>(kb) * 128 + chunk * 8) =
                encode8(raw[j], gs, zero);
    }
    if (t == 0) sw[static_cast<int64_t>(nb) * KB + kb] = gs.s;
}

// ---------------------------------------------------------------- weight_dequant
//
// w = bf16_rne(fp32(dec(q)) * s) per 128x128 block.  Work items are 16 rows x
// 128 columns of one block (2 KB of codes): thread t of a 128-thread group
// takes row (t / 8) and the 16-byte chunk (t % 8), so a warp reads four whole
// 128-byte rows and writes 256 contiguous bytes per row.  Each 128-thread
// group strides over the items kDqBatch at a time, the next batch's codes
// and scales loading while the current batch converts and stores
// (2 x kDqBatch loads in flight per thread).
constexpr int kDqItemRows = 16;
constexpr int kDqBatch = 2;

__global__ void __launch_bounds__(256) weight_dequant_kernel(const uint8_t* __restrict__ wq,
                                                            const float* __restrict__ sw, int64_t N, int64_t K,
                                                            uint16_t* __restrict__ w) {
    grid_dependency_wait();  // wq / sw may come from the kernel just before
    allow_dependents();
    const int64_t KB = K / 128;
    const int64_t NB = (N + 127) / 128;
    const int64_t items = NB * KB * (128 / kDqItemRows);
    const int t = threadIdx.x & 127;
    const int row = t >> 3, chunk = t & 7;
    const int64_t groups = 2 * static_cast<int64_t>(gridDim.x);  // two 128-thread groups per CTA
    const int64_t g0 = 2 * static_cast<int64_t>(blockIdx.x) + (threadIdx.x >> 7);
    struct Item {
        int64_t off;  // element offset of the chunk, or -1 when there is none
        uint4 q;
        float s;
    };
    auto fetch = [&](int64_t it, Item& x) {
        x.off = -1;
        if (it >= items) return;
        const int64_t blk = it / (128 / kDqItemRows);
        const int64_t part = it - blk * (128 / kDqItemRows);
        const int64_t nb = blk / KB, kb = blk - nb * KB;
        const int64_t n = nb * 128 + part * kDqItemRows + row;
        if (n >= N) return;
        x.off = n * K + kb * 128 + chunk * 16;
        x.s = __ldg(sw + nb * KB + kb);
        x.q = ld_stream(wq + x.off);
    };
    Item cur[kDqBatch], nxt[kDqBatch];
    // batch b of this group holds items g0 + (b * kDqBatch + i) * groups
#pragma unroll
    for (int i = 0; i < kDqBatch; ++i) fetch(g0 + i * groups, cur[i]);
    for (int64_t base = g0; base < items; base += kDqBatch * groups) {
#pragma unroll
        for (int i = 0; i < kDqBatch; ++i) fetch(base + (kDqBatch + i) * groups, nxt[i]);
#pragma unroll
        for (int i = 0; i < kDqBatch; ++i) {
            const Item& x = cur[i];
            if (x.off < 0) continue;
            const uint32_t words[4] = {x.q.x, x.q.y, x.q.z, x.q.w};
            uint32_t out[8];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float2 f01 = cvt_e4m3x2_to_f32(static_cast<uint16_t>(words[j] & 0xFFFFu));
                const float2 f23 = cvt_e4m3x2_to_f32(static_cast<uint16_t>(words[j] >> 16));
                const __nv_bfloat162 b01 = __floats2bfloat162_rn(__fmul_rn(f01.x, x.s), __fmul_rn(f01.y, x.s));
                const __nv_bfloat162 b23 = __floats2bfloat162_rn(__fmul_rn(f23.x, x.s), __fmul_rn(f23.y, x.s));
                out[2 * j] = *reinterpret_cast<const uint32_t*>(&b01);
                out[2 * j + 1] = *reinterpret_cast<const uint32_t*>(&b23);
            }
            // one 32-byte store: a warp writes four whole 256-byte row segments
            asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(w + x.off), "r"(out[0]),
                         "r"(out[1]), "r"(out[2]), "r"(out[3]), "r"(out[4]), "r"(out[5]), "r"(out[6]), "r"(out[7])
                         : "memory");
        }
#pragma unroll
        for (int i = 0; i < kDqBatch; ++i) cur[i] = nxt[i];
    }
}

// ---------------------------------------------------------------- diagnostics

__global__ void e4m3_encode_kernel(const float* __restrict__ v, int64_t n, uint8_t* __restrict__ q) {
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
        q[i] = static_cast<uint8_t>(cvt_e4m3x2(v[i], 0.0f) & 0xFFu);
}

// One warp waits on a barrier that nothing completes, using the same bounded
// wait as the GEMM pipeline, and records DEVERR_SELFTEST when it gives up.
__global__ void wait_selftest_kernel(unsigned* err, uint64_t timeout_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    __shared__ unsigned local_err;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        local_err = 0;
        fence_barrier_init();
    }
    __syncthreads();
    WaitCtl ctl{&abort_flag, &local_err, timeout_ns};
    const bool ok = bounded_wait(smem_u32(&bar), 0, ctl);
    __syncwarp();
    if (!ok && threadIdx.x == 0) atomicOr(err, DEVERR_SELFTEST);
}

// ---------------------------------------------------------------- act_quant_cols
//
// 128x1 groups (the weight gradient's operands, quantised along the tokens):
// for each column k and each block of 128 rows, amax over the block's valid
// rows, s = amax / 448, and the codes written transposed, xqt[k, m], so that
// each output row holds one channel's tokens contiguously (the layout the
// weight-gradient GEMM contracts over).
//
// A CTA walks tiles of 128 rows x 64 columns (16 KB of bf16) through a
// two-stage shared-memory ring filled with cp.async (16-byte copies; rows
// past M are zero-filled, so they never raise the amax): the next tile is in
// flight while one is encoded, and four CTAs share an SM.  Thread (cq, g)
// takes columns 4cq .. 4cq+3 and rows 8g .. 8g+7: eight 8-byte shared loads
// bring its 32 values, byte permutes regroup them by column, each column's
// partial amax is combined with the warp's other row group by one shuffle
// and left in shared memory; one thread per column then finishes the amax
// over the eight warps and forms the scale once, and every thread encodes
// its columns' eight values with the act_quant codec.  The codes go to a
// 64 x 128-byte staging tile, one row per output channel, its 16-byte
// chunks XOR-swizzled by the writer's column group (a warp's writes spread
// over all 32 banks), and leave as whole 128-byte rows of xqt.
constexpr int kCqRows = 128;
constexpr int kCqCols = 64;
constexpr int kCqStages = 2;
constexpr int kCqTileBytes = kCqRows * kCqCols * 2;        // 16 KB of bf16
constexpr int kCqOutOff = kCqStages * kCqTileBytes;         // staging: 64 channels x 128 codes
constexpr int kCqPamOff = kCqOutOff + kCqCols * kCqRows;    // per-warp column amaxes: 8 x 64 x 4 B
constexpr int kCqGsOff = kCqPamOff + 8 * kCqCols * 4;     // per column: s, 1/s (f32), flags (u8)
constexpr int kCqSmem = kCqGsOff + kCqCols * 9;

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__global__ void __launch_bounds__(256, 4) act_quant_cols_kernel(const uint16_t* __restrict__ x, int64_t M, int64_t K,
                                                               int64_t ldx, uint8_t* __restrict__ xqt, int64_t ldt,
                                                               float* __restrict__ sc, int64_t ldsc) {
    extern __shared__ __align__(128) uint8_t cq_smem[];
    grid_dependency_wait();  // the previous kernel may still read xqt / sc
    allow_dependents();
    const int t = threadIdx.x;
    const int lane = t & 31, w = t >> 5;
    const int cq = t & 15;  // columns 4cq .. 4cq+3 of the tile
    const int g = t >> 4;   // rows 8g .. 8g+7 of the tile
    const int64_t MB = (M + kCqRows - 1) / kCqRows;
    const int64_t CB = K / kCqCols;
    const int64_t G = gridDim.x;
    const uint32_t sbase = smem_u32(cq_smem);
    uint8_t* const stg = cq_smem + kCqOutOff;
    uint32_t* const pam = reinterpret_cast<uint32_t*>(cq_smem + kCqPamOff);
    float* const gs_s = reinterpret_cast<float*>(cq_smem + kCqGsOff);
    float* const gs_r = gs_s + kCqCols;
    uint8_t* const gs_f = reinterpret_cast<uint8_t*>(gs_r + kCqCols);  // bit 0: exact division, bit 1: amax 0
    // tile tt = mb * CB + cb; this CTA's tiles are blockIdx.x + j G, stepped
    // without a division: G = dq CB + dr
    struct TilePos {
        int64_t mb, cb;
    };
    const int64_t dq = G / CB, dr = G - (G / CB) * CB;
    auto advance = [&](TilePos& q) {
        q.cb += dr;
        q.mb += dq;
        if (q.cb >= CB) {
            q.cb -= CB;
            ++q.mb;
        }
    };

    // one tile's copies into stage st: 128 rows x 8 chunks of 16 bytes, four
    // per thread; a group is committed even when there is no tile, so that
    // the group count stays in step with the tiles
    auto issue = [&](const TilePos& q4, int st) {
        if (q4.mb < MB) {
            const int64_t mb = q4.mb;
            const int64_t k0 = q4.cb * kCqCols;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int q = t + 256 * i;
                const int r = q >> 3, ch = q & 7;
                const int64_t row = mb * kCqRows + r;
                const bool ok = row < M;
                cp_async16(sbase + st * kCqTileBytes + r * 128 + ch * 16, ok ? x + row * ldx + k0 + ch * 8 : x,
                           ok ? 16u : 0u);
            }
        }
        cp_async_commit();
    };
    TilePos cur{static_cast<int64_t>(blockIdx.x) / CB, static_cast<int64_t>(blockIdx.x) % CB};
    TilePos pre = cur;
    issue(cur, 0);
    advance(pre);  // one tile ahead of cur from here on
    int st = 0;  // stage of the current tile: this CTA's j-th tile sits in stage j % 2
    for (; cur.mb < MB; advance(cur), advance(pre)) {
        const int64_t mb = cur.mb;
        const int64_t k0 = cur.cb * kCqCols;
        const int64_t m0 = mb * kCqRows;
        cp_async_wait<0>();  // this thread's copies of the current tile have landed
        __syncthreads();     // and everyone's; the previous tile's shared reads are over
        issue(pre, st ^ 1);  // into the stage the previous tile used

        const uint8_t* tile = cq_smem + st * kCqTileBytes;
        uint2 v[8];  // row 8g + r, columns 4cq .. 4cq+3
#pragma unroll
        for (int r = 0; r < 8; ++r) v[r] = *reinterpret_cast<const uint2*>(tile + (8 * g + r) * 128 + cq * 8);
        uint4 col[4];  // column 4cq + j, rows 8g .. 8g+7 (element e in half e of the words)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint32_t wd[4];
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                const uint32_t a = j < 2 ? v[2 * p].x : v[2 * p].y;
                const uint32_t b = j < 2 ? v[2 * p + 1].x : v[2 * p + 1].y;
                wd[p] = __byte_perm(a, b, (j & 1) ? 0x7632 : 0x5410);
            }
            col[j] = make_uint4(wd[0], wd[1], wd[2], wd[3]);
        }
        uint32_t am[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            am[j] = absmax_bits8(col[j], 0u);
            am[j] = __vmaxu2(am[j], __shfl_xor_sync(0xffffffffu, am[j], 16));  // the warp's other row group
        }
        if (lane < 16) *reinterpret_cast<uint4*>(pam + w * kCqCols + 4 * cq) = make_uint4(am[0], am[1], am[2], am[3]);
        __syncthreads();
        if (t < kCqCols) {  // column t: its amax over the eight warps, and its scale
            uint32_t m2 = 0;
#pragma unroll
            for (int ww = 0; ww < 8; ++ww) m2 = __vmaxu2(m2, pam[ww * kCqCols + t]);
            const float amax = bits_to_amax(m2);
            const GroupScale gs = group_scale(amax);
            gs_s[t] = gs.s;
            gs_r[t] = gs.r;
            gs_f[t] = static_cast<uint8_t>((gs.exact_div ? 1u : 0u) | (amax == 0.0f ? 2u : 0u));
            sc[mb * ldsc + k0 + t] = gs.s;
        }
        __syncthreads();
        const float4 s4 = *reinterpret_cast<const float4*>(gs_s + 4 * cq);
        const float4 r4 = *reinterpret_cast<const float4*>(gs_r + 4 * cq);
        const uint32_t f4 = *reinterpret_cast<const uint32_t*>(gs_f + 4 * cq);
        const float sj[4] = {s4.x, s4.y, s4.z, s4.w};
        const float rj[4] = {r4.x, r4.y, r4.z, r4.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t fl = f4 >> (8 * j);
            const GroupScale gs{sj[j], rj[j], (fl & 1u) != 0u};
            const uint2 codes = encode8(col[j], gs, (fl & 2u) != 0u);
            const int c = 4 * cq + j;
            *reinterpret_cast<uint2*>(stg + c * 128 + (((g >> 1) ^ (cq & 7)) * 16) + (g & 1) * 8) = codes;
        }
        __syncthreads();
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int q = t + 256 * h;
            const int c = q >> 3, chl = q & 7;  // channel k0 + c, tokens m0 + 16 chl .. +15
            const uint4 val = *reinterpret_cast<const uint4*>(stg + c * 128 + ((chl ^ ((c >> 2) & 7)) * 16));
            const int64_t m = m0 + 16 * chl;
            uint8_t* out = xqt + (k0 + c) * ldt + m;
            if (m + 16 <= M) {
                *reinterpret_cast<uint4*>(out) = val;
            } else if (m < M) {  // the ragged last block: only the tokens that exist
                const uint64_t lo = (static_cast<uint64_t>(val.y) << 32) | val.x;
                const uint64_t hi = (static_cast<uint64_t>(val.w) << 32) | val.z;
                for (int b = 0; b < static_cast<int>(M - m); ++b)
                    out[b] = static_cast<uint8_t>(b < 8 ? lo >> (8 * b) : hi >> (8 * (b - 8)));
            }
        }
        st ^= 1;
    }
    cp_async_wait<0>();  // only an empty group can remain; leave with none in flight
}

}  // namespace

cudaError_t launch_act_quant(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, uint8_t* xq, int64_t ldq,
                             float* sx, int64_t lds, const DeviceInfo& dev, cudaStream_t stream, bool pow2) {
    const int64_t KB = K / 128;
    const int64_t groups = M * KB;
    const int64_t warps_needed = (groups + kAqGroupsPerWarp - 1) / kAqGroupsPerWarp;
    const int64_t blocks_needed = (warps_needed + 7) / 8;
    const int64_t max_blocks = static_cast<int64_t>(dev.num_sms) * 8;  // 8 x 256 threads per SM
    const int blocks = static_cast<int>(blocks_needed < max_blocks ? blocks_needed : max_blocks);
    if (pow2)
        return launch_pdl(act_quant_kernel<true>, dim3(blocks), dim3(256), 0, stream, x, KB, ldx, xq, ldq, sx, lds,
                          groups);
    return launch_pdl(act_quant_kernel<false>, dim3(blocks), dim3(256), 0, stream, x, KB, ldx, xq, ldq, sx, lds,
                      groups);
}

cudaError_t launch_weight_quant(const uint16_t* w, int64_t N, int64_t K, uint8_t* wq, float* sw,
                                const DeviceInfo& dev, cudaStream_t stream, bool pow2) {
    dim3 grid(static_cast<unsigned>(K / 128), static_cast<unsigned>((N + 127) / 128));
    const bool small = static_cast<int64_t>(grid.x) * grid.y < 2 * static_cast<int64_t>(dev.num_sms);
    if (pow2)
        return small ? launch_pdl(weight_quant_kernel<512, true>, grid, dim3(512), 0, stream, w, N, K, wq, sw)
                     : launch_pdl(weight_quant_kernel<256, true>, grid, dim3(256), 0, stream, w, N, K, wq, sw);
    return small ? launch_pdl(weight_quant_kernel<512, false>, grid, dim3(512), 0, stream, w, N, K, wq, sw)
                 : launch_pdl(weight_quant_kernel<256, false>, grid, dim3(256), 0, stream, w, N, K, wq, sw);
}

cudaError_t launch_weight_dequant(const uint8_t* wq, const float* sw, int64_t N, int64_t K, uint16_t* w,
                                  const DeviceInfo& dev, cudaStream_t stream) {
    const int64_t items = ((N + 127) / 128) * (K / 128) * (128 / kDqItemRows);
    const int64_t want = (items + 2 * kDqBatch - 1) / (2 * kDqBatch);  // CTAs that each get a batch per group
    const int64_t cap = static_cast<int64_t>(dev.num_sms) * 8;       // 8 x 256 threads per SM
    const int blocks = static_cast<int>(want < cap ? want : cap);
    return launch_pdl(weight_dequant_kernel, dim3(blocks), dim3(256), 0, stream, wq, sw, N, K, w);
}

cudaError_t launch_e4m3_encode(const float* v, int64_t n, uint8_t* q, const DeviceInfo& dev,
                               cudaStream_t stream) {
    int64_t blocks = (n + 255) / 256;
    const int64_t cap = static_cast<int64_t>(dev.num_sms) * 16;
    if (blocks > cap) blocks = cap;
    e4m3_encode_kernel<<<static_cast<int>(blocks), 256, 0, stream>>>(v, n, q);
    return cudaGetLastError();
}

cudaError_t launch_wait_selftest(uint64_t timeout_ns, const DeviceInfo& dev, cudaStream_t stream) {
    wait_selftest_kernel<<<1, 32, 0, stream>>>(dev.err, timeout_ns);
    return cudaGetLastError();
}

cudaError_t launch_act_quant_cols(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, uint8_t* xqt, int64_t ldt,
                                  float* sc, int64_t ldsc, const DeviceInfo& dev, cudaStream_t stream) {
    {
        static bool ready[64];
        if (dev.device < 0 || dev.device >= 64) return cudaErrorInvalidDevice;
        if (!ready[dev.device]) {
            const cudaError_t e =
                cudaFuncSetAttribute(act_quant_cols_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kCqSmem);
            if (e != cudaSuccess) return e;
            ready[dev.device] = true;
        }
    }
    const int64_t tiles = ((M + kCqRows - 1) / kCqRows) * (K / kCqCols);
    const int64_t max_blocks = static_cast<int64_t>(dev.num_sms) * 4;  // four 44 KB CTAs per SM
    const int blocks = static_cast<int>(tiles < max_blocks ? tiles : max_blocks);
    return launch_pdl(act_quant_cols_kernel, dim3(blocks), dim3(256), kCqSmem, stream, x, M, K, ldx, xqt, ldt, sc,
                      ldsc);
}

}  // namespace fp8bs
