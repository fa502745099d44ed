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
// weight-gradient GEMM contracts over).  A CTA takes tiles of 128 rows x 64
// columns: the tile is read with 16-byte loads into shared memory, then
// thread (c, g) takes column c and rows 32g .. 32g+31, reduces their amax,
// combines the four partial amaxes of its column through shared memory,
// encodes its 32 values with the act_quant arithmetic and stores its 32
// codes -- contiguous in the transposed output -- as two 16-byte stores.
constexpr int kCqRows = 128;
constexpr int kCqCols = 64;

__global__ void __launch_bounds__(256) act_quant_cols_kernel(const uint16_t* __restrict__ x, int64_t M, int64_t K,
                                                            int64_t ldx, uint8_t* __restrict__ xqt, int64_t ldt,
                                                            float* __restrict__ sc, int64_t ldsc) {
    __shared__ __align__(16) uint16_t tile[kCqRows][kCqCols];
    __shared__ uint32_t pam[4][kCqCols];
    grid_dependency_wait();  // the previous kernel may still read xqt / sc
    allow_dependents();
    const int t = threadIdx.x;
    const int c = t % kCqCols;   // column within the tile
    const int g = t / kCqCols;   // row group of 32
    const int64_t MB = (M + kCqRows - 1) / kCqRows;
    const int64_t CB = K / kCqCols;
    // the tile's 128 rows x 128 bytes: four 16-byte chunks per thread, eight
    // threads per row; rows past M read as zeros (they never raise the amax)
    auto load_tile = [&](int64_t tt, uint4 (&v)[4]) {
        const int64_t mb = tt / CB;
        const int64_t k0 = (tt - mb * CB) * kCqCols;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int q = t + 256 * i;
            const int r = q / 8, ch = q % 8;
            v[i] = make_uint4(0, 0, 0, 0);
            if (tt < MB * CB && mb * kCqRows + r < M) v[i] = ld_stream(x + (mb * kCqRows + r) * ldx + k0 + ch * 8);
        }
    };
    uint4 pre[4];
    load_tile(blockIdx.x, pre);
    for (int64_t tt = blockIdx.x; tt < MB * CB; tt += gridDim.x) {
        const int64_t mb = tt / CB;
        const int64_t k0 = (tt - mb * CB) * kCqCols;
        const int64_t m0 = mb * kCqRows;
        __syncthreads();  // the previous tile's reads of `tile` and `pam` are done
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int q = t + 256 * i;
            *reinterpret_cast<uint4*>(&tile[q / 8][(q % 8) * 8]) = pre[i];
        }
        load_tile(tt + gridDim.x, pre);  // the next tile's loads run during this tile's work
        __syncthreads();
        uint4 v[4];  // rows 32g + 8j .. +7 of column c, as 8 bf16 values each
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint32_t w[4];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                const int r = 32 * g + 8 * j + 2 * h;
                w[h] = static_cast<uint32_t>(tile[r][c]) | (static_cast<uint32_t>(tile[r + 1][c]) << 16);
            }
            v[j] = make_uint4(w[0], w[1], w[2], w[3]);
        }
        uint32_t amax2 = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) amax2 = absmax_bits8(v[j], amax2);
        pam[g][c] = amax2;
        __syncthreads();
        amax2 = __vmaxu2(__vmaxu2(pam[0][c], pam[1][c]), __vmaxu2(pam[2][c], pam[3][c]));
        const float amax = bits_to_amax(amax2);
        const GroupScale gs = group_scale(amax);
        const bool zero = amax == 0.0f;
        uint2 codes[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) codes[j] = encode8(v[j], gs, zero);
        const int64_t mrow = m0 + 32 * g;  // first token of this thread's 32 codes
        uint8_t* out = xqt + (k0 + c) * ldt + mrow;
        if (mrow + 32 <= M) {
            *reinterpret_cast<uint4*>(out) = make_uint4(codes[0].x, codes[0].y, codes[1].x, codes[1].y);
            *reinterpret_cast<uint4*>(out + 16) = make_uint4(codes[2].x, codes[2].y, codes[3].x, codes[3].y);
        } else if (mrow < M) {  // the ragged last block: only the tokens that exist
            const uint32_t wds[8] = {codes[0].x, codes[0].y, codes[1].x, codes[1].y,
                                     codes[2].x, codes[2].y, codes[3].x, codes[3].y};
            for (int b = 0; b < static_cast<int>(M - mrow); ++b) out[b] = static_cast<uint8_t>(wds[b / 4] >> (8 * (b % 4)));
        }
        if (g == 0) sc[mb * ldsc + k0 + c] = gs.s;
    }
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
    const int64_t tiles = ((M + kCqRows - 1) / kCqRows) * (K / kCqCols);
    const int64_t max_blocks = static_cast<int64_t>(dev.num_sms) * 4;
    const int blocks = static_cast<int>(tiles < max_blocks ? tiles : max_blocks);
    return launch_pdl(act_quant_cols_kernel, dim3(blocks), dim3(256), 0, stream, x, M, K, ldx, xqt, ldt, sc, ldsc);
}

}  // namespace fp8bs
