/*
 * fp8bs.h -- C ABI of the FP8 (e4m3) block-scaled linear layer for B300
 * (sm_103a).  Library: libfp8bs.so.
 *
 * The operation is the FP8 branch of DeepSeek-V3's linear(), as printed in the
 * "DeepSeek-V3" repository overview (pomoai hub), section "FP8 混合精度训练":
 *   x, scale = act_quant(x, block_size, scale_fmt)
 *   y = fp8_gemm(x, scale, weight, weight.scale)
 * with weights stored as float8 e4m3 in 128x128 blocks, one fp32 scale per
 * block ("weight_scale_inv"), activations quantised at run time per token per
 * 128 channels, and weight_dequant(weight, weight.scale) as the bf16 branch.
 * fp32 promotion once per 128-wide K chunk follows the Float8 paragraph of the
 * 88811315.cn post on DeepSeek v3 (fp32 accumulation after a fixed number of
 * FP8 multiply-adds) and the qdgithub overview's "FP8 量化" section (blockwise
 * FP8 compute, dequantisation on CUDA cores).
 *
 * Conventions shared by every call
 *   - bf16 values travel as uint16_t bit patterns; e4m3 codes as uint8_t (OCP
 *     E4M3: bias 7, no infinities, 0x7F/0xFF NaN, largest finite 448).
 *   - Every scale is the dequantisation multiplier: value ~= dec(code) * s,
 *     with s = amax / 448 (fp32, IEEE round-to-nearest division) over the
 *     group or block, and code = e4m3(x / s) rounded to nearest-even with
 *     saturation at +-448.  An all-zero group/block gets s = 0 and +-0 codes.
 *   - K must be a multiple of 128.  Row-major everywhere ("ld*" = row stride
 *     in elements).  All pointers are DEVICE pointers owned by the caller; the
 *     library keeps none of them after the call returns and allocates no
 *     device memory in any call (it holds a small static status word per
 *     device, and the fixed scratch array of fp8bs_gemm_noalloc).
 *   - Calls are asynchronous on `stream` (NULL = legacy default stream).
 *     The kernels are launched with programmatic stream serialisation: one
 *     may start its set-up while the previous kernel on the stream finishes,
 *     but it waits for that kernel to complete before it reads or writes any
 *     global memory, so stream order is kept exactly as for plain launches
 *     (also inside CUDA graphs captured from the stream).
 *     Argument errors are returned synchronously and launch nothing.  Errors
 *     inside a kernel (a bounded pipeline wait that expired) are recorded in
 *     the device status word and reported by fp8bs_sync_status().
 *   - M (or total rows) == 0 is a no-op returning FP8BS_OK.
 *   - Thread-safe: calls keep no mutable host state except per-device caches
 *     filled once under a lock.  Those caches (device symbol addresses, kernel
 *     attributes) belong to the device's context: do not call the library
 *     again in a process that reset a device with cudaDeviceReset.
 */
#ifndef FP8BS_H
#define FP8BS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream. */
typedef struct CUstream_st* fp8bs_stream_t;

typedef enum {
    FP8BS_OK = 0,
    FP8BS_ERR_INVALID_ARG = 1,  /* null pointer, negative or inconsistent size */
    FP8BS_ERR_UNSUPPORTED = 2,  /* K % 128 != 0, size beyond the 32-bit index range, no sm_103 device */
    FP8BS_ERR_MISALIGNED = 3,   /* pointer or leading dimension breaks the 16-byte rule */
    FP8BS_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed */
    FP8BS_ERR_TIMEOUT = 5,      /* a kernel's bounded wait expired (see fp8bs_sync_status) */
    FP8BS_ERR_INDEX = 6         /* a device-side row or token id was out of range (see fp8bs_sync_status) */
} fp8bs_status;

/* act_quant: per row m and group g of 128 channels (per token, per 128
 * channels -- "FP8 混合精度训练", dynamic activation quantisation).
 *   x  [M, K] bf16, row stride ldx (ldx % 8 == 0, x 16-byte aligned)
 *   xq [M, K] e4m3, row stride ldq (ldq % 16 == 0, 16-byte aligned)
 *   sx [M, lds] fp32, sx[m*lds + g] = amax_g / 448 for g < K/128
 *      (lds >= K/128, lds % 4 == 0, 16-byte aligned); columns >= K/128 untouched. */
fp8bs_status fp8bs_act_quant(const uint16_t* x, int64_t M, int64_t K, int64_t ldx,
                             uint8_t* xq, int64_t ldq, float* sx, int64_t lds,
                             fp8bs_stream_t stream);

/* weight_quant: per 128x128 block (nb, kb) of w ("以 128×128 分块存储", one
 * fp32 weight_scale_inv per block).  The last row block may be ragged
 * (N % 128 != 0); its amax is taken over its valid rows.
 *   w  [N, K] bf16, dense (row stride K), 16-byte aligned
 *   wq [N, K] e4m3, dense, 16-byte aligned
 *   sw [ceil(N/128), K/128] fp32, dense. */
fp8bs_status fp8bs_weight_quant(const uint16_t* w, int64_t N, int64_t K,
                                uint8_t* wq, float* sw, fp8bs_stream_t stream);

/* act_quant / weight_quant with power-of-two scales: the pages' act_quant
 * takes a scale format (scale_fmt, the linear() excerpt of the "DeepSeek-V3"
 * repository overview) that they do not define.  These calls read it as a
 * UE8M0-style scale -- an unsigned power of two, no mantissa -- rounded up so
 * that nothing saturates: s = 2^e with e the smallest integer such that
 * amax <= 448 * 2^e, codes e4m3(x / s) (x / s is exact; only the encode
 * rounds); an all-zero group or block has s = 0 and +-0 codes.  Arguments,
 * layouts and errors exactly as fp8bs_act_quant / fp8bs_weight_quant; the
 * scales are written as fp32 (exact powers of two), so the outputs feed
 * fp8bs_gemm and fp8bs_weight_dequant unchanged. */
fp8bs_status fp8bs_act_quant_pow2(const uint16_t* x, int64_t M, int64_t K, int64_t ldx,
                                  uint8_t* xq, int64_t ldq, float* sx, int64_t lds,
                                  fp8bs_stream_t stream);
fp8bs_status fp8bs_weight_quant_pow2(const uint16_t* w, int64_t N, int64_t K,
                                     uint8_t* wq, float* sw, fp8bs_stream_t stream);

/* weight_dequant (the bf16 branch of linear(); also the FP8->BF16 checkpoint
 * cast): w[n,k] = bf16_rne(fp32(dec(wq[n,k])) * sw[n/128, k/128]).
 *   wq [N, K] e4m3 dense, sw [ceil(N/128), K/128] fp32 dense, w [N, K] bf16 dense;
 *   wq and w 16-byte aligned. */
fp8bs_status fp8bs_weight_dequant(const uint8_t* wq, const float* sw, int64_t N, int64_t K,
                                  uint16_t* w, fp8bs_stream_t stream);

/* fp8_gemm ("y = fp8_gemm(x, scale, weight, weight.scale)"):
 *   y[m,n] = bf16_rne( sum_kb fp32( sx[m,kb] * sw[n/128,kb] ) * P_kb[m,n] )
 *   P_kb[m,n] = sum over the 128 k of chunk kb of dec(xq[m,k]) * dec(wq[n,k]),
 * accumulated by the tensor cores in fp32 and promoted (scaled and added in
 * fp32) once per chunk.  Any fp32 summation order is allowed: results satisfy
 * |y - y_exact| <= 2^-8 |y_exact| + 1e-4 sum_k |a_k b_k| elementwise.
 *   xq [M, K] e4m3, row stride K (dense), 16-byte aligned
 *   sx [M, lds] fp32 (lds >= K/128, lds % 4 == 0), 16-byte aligned
 *   wq [N, K] e4m3 dense ("TN": both operands K-major), 16-byte aligned
 *   sw [ceil(N/128), K/128] fp32 dense
 *   y  [M, N] bf16, row stride ldy (ldy >= N, ldy % 8 == 0), 16-byte aligned
 *   workspace: optional device scratch for the split-K path used when M is
 *     small but above the few-token kernel's range; may be NULL (then no
 *     split).  fp8bs_gemm_workspace_size() gives the size that enables the
 *     fastest plan; a smaller buffer selects fewer splits.  Contents on entry
 *     are ignored; the caller must not use it concurrently from another call.
 * Few tokens (M <= 64 with K <= 8192, or M <= 128 with K <= 4096) run a
 * weight-streaming kernel that splits K over a thread-block cluster and adds
 * the pieces in shared memory: one launch, no workspace, the same bits with
 * or without one. */
fp8bs_status fp8bs_gemm(const uint8_t* xq, const float* sx, int64_t lds,
                        const uint8_t* wq, const float* sw,
                        int64_t M, int64_t N, int64_t K,
                        uint16_t* y, int64_t ldy,
                        void* workspace, size_t ws_bytes, fp8bs_stream_t stream);

/* Bytes of workspace that let fp8bs_gemm pick its fastest plan for this shape
 * on the current device (0 when no split is used). */
size_t fp8bs_gemm_workspace_size(int64_t M, int64_t N, int64_t K);

/* fp8_gemm with a fused epilogue: the bias add of the pages' linear()
 * ("DeepSeek-V3" repository overview, "FP8 混合精度训练": y += bias after
 * fp8_gemm) and the re-quantisation of the result back to FP8 that the same
 * section describes ("结果再量化回 FP8").  The pages' code returns a bf16 y;
 * this call produces either or both forms in one pass.
 *   y[m,n]  = bf16_rne( fp8_gemm sum (as fp8bs_gemm) + bias[n] ), the bias
 *             (bf16 [N], may be NULL) added in fp32 before the rounding.
 *   yq, sy  = the bf16 y quantised exactly as fp8bs_act_quant quantises an
 *             input: per row and per group of 128 columns, s = amax/448,
 *             code = e4m3(y / s) -- ready to feed the next fp8 GEMM.
 * y (ldy >= N, ldy % 8 == 0, 16-byte aligned) may be NULL when yq is given;
 * yq [M, ldyq] (ldyq >= N, ldyq % 16 == 0) and sy [M, ldsy] (ldsy >= N/128,
 * ldsy % 4 == 0), both 16-byte aligned, may be NULL (both) when y is given.
 * At least one of y and yq is required (FP8BS_ERR_INVALID_ARG otherwise).
 * yq requires N % 128 == 0 (FP8BS_ERR_UNSUPPORTED otherwise) and runs with
 * 256-column tiles.  This call never splits K, so it needs no workspace.
 * Operand rules and errors otherwise as fp8bs_gemm. */
fp8bs_status fp8bs_gemm_fused(const uint8_t* xq, const float* sx, int64_t lds, const uint8_t* wq, const float* sw,
                              const uint16_t* bias, int64_t M, int64_t N, int64_t K, uint16_t* y, int64_t ldy,
                              uint8_t* yq, int64_t ldyq, float* sy, int64_t ldsy, fp8bs_stream_t stream);

/* grouped fp8_gemm for MoE experts (256 routed experts, top-8 -- "MoE 架构详解"):
 * for each expert g, rows offsets[g] .. offsets[g+1]-1 of xq/sx/y are
 * multiplied by expert g's weight, exactly as fp8bs_gemm.
 *   xq [total_M, K] e4m3 dense, sx [total_M, lds] fp32 (as fp8bs_gemm)
 *   wq [G, N, K] e4m3 dense, sw [G, ceil(N/128), K/128] fp32 dense
 *   offsets_dev: DEVICE int32 [G+1], non-decreasing, offsets[0] = 0,
 *     offsets[G] = total_M (read on the device: no host synchronisation).
 *     A violation is undefined behaviour of the kernel (rows may be skipped
 *     or written twice) but never an out-of-bounds access: every row index
 *     is clamped to [0, total_M).
 *   y  [total_M, N] bf16, row stride ldy (ldy % 8 == 0). */
fp8bs_status fp8bs_grouped_gemm(const uint8_t* xq, const float* sx, int64_t lds,
                                const uint8_t* wq, const float* sw,
                                const int32_t* offsets_dev, int32_t G, int64_t total_M,
                                int64_t N, int64_t K, uint16_t* y, int64_t ldy,
                                fp8bs_stream_t stream);

/* Scratch bytes fp8bs_grouped_gemm needs for G experts of [N, K]: always 0.
 * Its per-expert tile table is built inside each CTA's shared memory from
 * offsets_dev, so the call takes no workspace argument; this size query
 * exists for callers written against a grouped GEMM that takes one. */
size_t fp8bs_grouped_gemm_workspace_size(int32_t G, int64_t N, int64_t K);

/* fp8_gemm for callers that cannot allocate device memory -- code running
 * inside an allocator's or memory pool's own callback, plugin hosts that pass
 * a library only its input and output buffers, and latency-critical paths
 * that must not trigger a (possibly synchronising) device allocation.  The
 * DeepSeek-V3 pages have no counterpart: this is an interface for such
 * callers, computing exactly what fp8bs_gemm computes.
 * Same arguments and results as fp8bs_gemm without the workspace: the
 * split-K scratch of the small-M plan (above the few-token kernel's range,
 * which needs none) comes from a fixed array of
 * FP8BS_NOALLOC_SCRATCH_BYTES inside the library's device image (every device
 * that loads the library holds it until the process exits).  Returns
 * FP8BS_ERR_UNSUPPORTED, launching nothing, when the shape's plan needs more
 * scratch than that (fp8bs_gemm_workspace_size(M, N, K) > the maximum).
 * The first call on a device looks up the array's device address (with that
 * device current); make that first call before any stream capture.  All
 * calls on a device share the array: calls whose kernels overlap on the GPU
 * race and must be serialised by the caller.  Allocates nothing.
 * On 148 SMs the largest scratch any shape's plan asks for is
 * num_sms * 128 * 160 * 4 bytes (12.1 MB: split-K runs with 160-column tiles
 * and at most one (tile, split) piece per SM), so the 32 MiB array serves
 * every valid shape on devices of up to 409 SMs.
 * Like the library's other per-device set-up (the status word's address,
 * kernel attributes), the looked-up address belongs to the device's current
 * context: after cudaDeviceReset the library must not be called again in
 * that process. */
#define FP8BS_NOALLOC_SCRATCH_BYTES (32u << 20)
fp8bs_status fp8bs_gemm_noalloc(const uint8_t* xq, const float* sx, int64_t lds,
                                const uint8_t* wq, const float* sw,
                                int64_t M, int64_t N, int64_t K,
                                uint16_t* y, int64_t ldy, fp8bs_stream_t stream);

/* Backward pass, weight gradient (E4M3 in the backward pass as well as the
 * forward: the Float8 paragraph of the 88811315.cn post on DeepSeek v3).
 * dW = dY^T X contracts over the tokens, so both operands are quantised in
 * 128x1 groups along the tokens -- the contraction dimension of this GEMM,
 * as the forward groups its operands along K.
 *
 * act_quant_cols: per column k and per block of 128 rows (the last block may
 * be ragged: its amax is over the rows that exist), amax = max |x|,
 * s = amax / 448, codes e4m3(x / s) exactly as fp8bs_act_quant computes them,
 * written TRANSPOSED so that each channel's tokens are contiguous:
 *   x   [M, K] bf16, row stride ldx (ldx % 8 == 0, 16-byte aligned)
 *   xqt [K, ldt] e4m3: xqt[k*ldt + m] = code of x[m, k] (ldt >= M,
 *       ldt % 16 == 0, 16-byte aligned); bytes m >= M of a row are untouched
 *   sc  [ceil(M/128), ldsc] fp32: sc[mb*ldsc + k] = s of column k, block mb
 *       (ldsc >= K, 4-byte aligned)
 * K % 64 == 0 (else FP8BS_ERR_UNSUPPORTED); M == 0 or K == 0 is a no-op. */
fp8bs_status fp8bs_act_quant_cols(const uint16_t* x, int64_t M, int64_t K, int64_t ldx,
                                  uint8_t* xqt, int64_t ldt, float* sc, int64_t ldsc,
                                  fp8bs_stream_t stream);

/* gemm_wgrad: dW[n, k] = sum_tb fp32(sdy[tb, n] * sx[tb, k]) * P_tb[n, k],
 * P_tb the sum over the 128 tokens of block tb of dec(dy code) * dec(x code),
 * accumulated in fp32 and promoted once per token block (as fp8bs_gemm
 * promotes once per 128-wide K chunk); dW in fp32.
 *   dyqt [N, lddyt], sdy [ceil(T/128), ldsdy]: fp8bs_act_quant_cols of dY [T, N]
 *   xqt  [K, ldxt],  sx  [ceil(T/128), ldsx]:  fp8bs_act_quant_cols of X  [T, K]
 *   dw   [N, lddw] fp32 (lddw >= K, lddw % 4 == 0, 16-byte aligned)
 * T >= 1 tokens (T == 0: FP8BS_ERR_INVALID_ARG); N or K == 0 is a no-op.
 * Code row strides % 16 == 0 and >= T, scale row strides % 4 == 0, all base
 * pointers 16-byte aligned.  Tokens past T read as zero codes. */
fp8bs_status fp8bs_gemm_wgrad(const uint8_t* dyqt, int64_t lddyt, const float* sdy, int64_t ldsdy,
                              const uint8_t* xqt, int64_t ldxt, const float* sx, int64_t ldsx,
                              int64_t T, int64_t N, int64_t K, float* dw, int64_t lddw,
                              fp8bs_stream_t stream);

/* MoE expert first stage with the SwiGLU activation fused (the pages' Expert
 * forward, "DeepSeek-V3" repository overview, MoE section: w2(silu(w1(x)) *
 * w3(x)); this call computes the part before w2).  For each expert g and
 * each of its rows m (offsets_dev as fp8bs_grouped_gemm):
 *   a = fp8_gemm(xq, sx, w1q[g], sw1[g]),  b = fp8_gemm(xq, sx, w3q[g], sw3[g])
 *   h[m, i] = bf16( bf16(silu(bf16(a))) * bf16(b) ),  silu(v) = v / (1 + e^-v)
 * i.e. the bf16 roundings of the expert forward run on bf16 tensors; silu
 * is evaluated in fp32.  w1q, w3q: e4m3 [G, I, K]; sw1, sw3: fp32
 * [G, I/128, K/128] (each weight quantised on its own, as fp8bs_weight_quant
 * does per expert).  Outputs, at least one of them (FP8BS_ERR_INVALID_ARG
 * otherwise):
 *   h  bf16 [total_M, ldh] (ldh >= I, ldh % 8 == 0, 16-byte aligned), or NULL;
 *   hq e4m3 [total_M, ldhq] and sh fp32 [total_M, ldsh]: h quantised exactly
 *      as fp8bs_act_quant quantises an input (per row, per 128 columns;
 *      ldhq >= I, ldhq % 16 == 0; ldsh >= I/128, ldsh % 4 == 0; both 16-byte
 *      aligned) -- the operand of the w2 GEMM -- or both NULL.
 * I % 128 == 0 (else FP8BS_ERR_UNSUPPORTED).  Other operand rules and errors
 * as fp8bs_grouped_gemm. */
fp8bs_status fp8bs_grouped_gemm_swiglu(const uint8_t* xq, const float* sx, int64_t lds, const uint8_t* w1q,
                                       const float* sw1, const uint8_t* w3q, const float* sw3,
                                       const int32_t* offsets_dev, int32_t G, int64_t total_M, int64_t I,
                                       int64_t K, uint16_t* h, int64_t ldh, uint8_t* hq, int64_t ldhq, float* sh,
                                       int64_t ldsh, fp8bs_stream_t stream);

/* MoE dispatch: gather the quantised token rows into routed (expert-grouped)
 * order, the operand layout of fp8bs_grouped_gemm and
 * fp8bs_grouped_gemm_swiglu.  Every token keeps all of its selected experts
 * (no token dropping: DeepSeek-V3 notes, page 2 section 2-2), so a token
 * routed to k experts appears in k rows.  For r < R, t = token_of_row[r]:
 *   xq_rows[r, 0:K] = xq[t, 0:K]   (e4m3 codes, copied unchanged)
 *   sx_rows[r, 0:K/128] = sx[t, 0:K/128]   (the per-128-channel scales)
 * Quantisation is per token row, so the result equals fp8bs_act_quant of the
 * gathered bf16 rows bit for bit, at 1/k of the quantisation work.
 *   xq [tokens, ldq] (ldq >= K, ldq % 16 == 0, 16-byte aligned), sx [tokens, lds]
 *      (lds >= K/128, 4-byte aligned): as fp8bs_act_quant writes them
 *   token_of_row int32 [R] device (4-byte aligned): source token of each row
 *   xq_rows [R, ldq_rows] (ldq_rows >= K, ldq_rows % 16 == 0, 16-byte aligned),
 *   sx_rows [R, lds_rows] (lds_rows >= K/128, 4-byte aligned); scale columns
 *      >= K/128 untouched.
 * K % 128 == 0 (else FP8BS_ERR_UNSUPPORTED); tokens == 0 with R > 0 is
 * FP8BS_ERR_INVALID_ARG.  A token id outside [0, tokens) is not read: that
 * row is written as zeros (codes and scales) and the next fp8bs_sync_status()
 * reports FP8BS_ERR_INDEX. */
fp8bs_status fp8bs_moe_dispatch(const uint8_t* xq, int64_t ldq, const float* sx, int64_t lds, int64_t tokens,
                                int64_t K, const int32_t* token_of_row, int64_t R, uint8_t* xq_rows,
                                int64_t ldq_rows, float* sx_rows, int64_t lds_rows, fp8bs_stream_t stream);

/* MoE combine: each token's output is its selected experts' outputs weighted
 * by its gate values -- the sigmoid affinities, not the bias-adjusted scores,
 * which only steer the selection (DeepSeek-V3 notes, page 2 section 2-2) --
 * plus an optional dense term z, e.g. the shared experts' output that every
 * token receives (page 3, the DeepSeekMoE shared-expert paragraph) or the
 * residual.  For each token t and column d, r_k = rows_of_token[t, k]:
 *   y[t, d] = bf16_rne( acc ),  acc = z[t, d] (0 if z is NULL), then for
 *   k = 0 .. topk-1 in that order acc = fma(weight_of_row[r_k], yk[r_k, d], acc)
 * in fp32 (one rounding per term, one to bf16 at the end).  So
 *   |y - y_exact| <= 2^-8 |y_exact| + (topk + 1) 2^-24 (|z| + sum_k |w yk|).
 *   yk bf16 [R, ldyk] (ldyk >= dim, ldyk % 8 == 0, 16-byte aligned): the
 *      expert outputs in routed order (fp8bs_grouped_gemm's y)
 *   weight_of_row fp32 [R] (4-byte aligned): the gate value of each routed row
 *   rows_of_token int32 [tokens, topk] dense (4-byte aligned): the routed rows of each token
 *   z bf16 [tokens, ldz] (ldz >= dim, ldz % 8 == 0, 16-byte aligned) or NULL;
 *      z may be y itself (same pointer and ldz == ldy), no other overlap
 *      (FP8BS_ERR_INVALID_ARG)
 *   y bf16 [tokens, ldy] (ldy >= dim, ldy % 8 == 0, 16-byte aligned).
 * dim % 8 == 0 (else FP8BS_ERR_UNSUPPORTED).  topk == 0 gives y = bf16(z) (or
 * zeros).  A row id outside [0, R) contributes nothing and the next
 * fp8bs_sync_status() reports FP8BS_ERR_INDEX. */
fp8bs_status fp8bs_moe_combine(const uint16_t* yk, int64_t ldyk, int64_t R, const float* weight_of_row,
                               const int32_t* rows_of_token, int64_t tokens, int32_t topk, int64_t dim,
                               const uint16_t* z, int64_t ldz, uint16_t* y, int64_t ldy, fp8bs_stream_t stream);

/* MoE router (gate): for each token t, the sigmoid affinities
 * s_e = sigmoid(x_t . wg_e) of the E routed experts, computed from the bf16
 * operands with fp32 accumulation on the tensor cores (gating stays in
 * higher precision than FP8: DeepSeek-V3 notes, page 2 section 2-4); the
 * selection looks at s_e + bias_e, the gate values at s_e alone (page 2
 * section 2-2).  The experts form n_groups equal groups of consecutive
 * indices; a group's score is its largest biased affinity; the topk_groups
 * best groups are kept, and the top_k best biased affinities among their
 * experts are chosen (ties to the lower index throughout).  Gate values:
 * w_k = s_k / (sum of the chosen s) * route_scale (DeepSeek-V3: sigmoid
 * scoring, 8 groups keep 4, top-8 of 256, route_scale 2.5 -- config block
 * of "671B 参数如何「激活」37B？").  All in fp32; the sigmoid uses expf.
 *   x  bf16 [T, ldx] (ldx >= dim, ldx % 8 == 0, 16-byte aligned)
 *   wg bf16 [E, dim] dense, 16-byte aligned; bias fp32 [E] or NULL (zeros)
 *   ids int32 [T, top_k]: the chosen experts, best biased affinity first
 *   weights fp32 [T, top_k]: their gate values
 * dim % 64 == 0 and E % 16 == 0, E <= 256 (else FP8BS_ERR_UNSUPPORTED);
 * n_groups divides E, n_groups <= 32, 1 <= topk_groups <= n_groups,
 * 1 <= top_k <= 16 and top_k <= topk_groups * E / n_groups (else
 * FP8BS_ERR_INVALID_ARG).  Near-ties may resolve differently from an exact
 * (fp64) router: the logits carry fp32 rounding.  A token whose biased
 * affinities include NaN or -inf (non-finite x or bias) may get id -1 in a
 * slot, with gate value computed as if that affinity were 0; fp8bs_moe_route
 * then reports FP8BS_ERR_INDEX. */
fp8bs_status fp8bs_moe_gate(const uint16_t* x, int64_t ldx, const uint16_t* wg, const float* bias, int64_t T,
                            int64_t dim, int32_t E, int32_t n_groups, int32_t topk_groups, int32_t top_k,
                            float route_scale, int32_t* ids, float* weights, fp8bs_stream_t stream);

/* MoE routing tables: the (token, k) selections grouped by expert, tokens in
 * order within an expert (a stable counting sort; the same result on every
 * run) -- the layout fp8bs_moe_dispatch, the grouped GEMMs and
 * fp8bs_moe_combine take:
 *   offsets int32 [E+1]: expert e's routed rows are offsets[e] .. offsets[e+1]-1
 *   token_of_row int32 [T*top_k], weight_of_row fp32 [T*top_k]: per routed row
 *      its token and gate value
 *   rows_of_token int32 [T, top_k]: the routed row of selection (t, k)
 * from ids int32 [T, top_k] and weights fp32 [T, top_k] (fp8bs_moe_gate's
 * outputs).  E <= 256 and top_k <= 16 (else FP8BS_ERR_UNSUPPORTED); all
 * pointers 4-byte aligned.  An id outside [0, E) gets no row (rows_of_token -1); a token
 * naming one expert twice leaves a row with token -1 and gate 0; both set
 * FP8BS_ERR_INDEX for the next fp8bs_sync_status(). */
fp8bs_status fp8bs_moe_route(const int32_t* ids, const float* weights, int64_t T, int32_t top_k, int32_t E,
                             int32_t* offsets, int32_t* token_of_row, int32_t* rows_of_token, float* weight_of_row,
                             fp8bs_stream_t stream);

/* Synchronise `stream`, then report and clear this device's status word:
 * FP8BS_ERR_TIMEOUT if a kernel's bounded wait expired since the last call,
 * else FP8BS_ERR_INDEX if a MoE gather met an out-of-range id, FP8BS_ERR_CUDA
 * if the stream reports a CUDA error, else FP8BS_OK. */
fp8bs_status fp8bs_sync_status(fp8bs_stream_t stream);

/* Static, human-readable name of a status. */
const char* fp8bs_status_string(fp8bs_status status);

/* --- diagnostics -------------------------------------------------------- */

/* The e4m3 encoder the quantisers use, applied elementwise: q[i] = e4m3(v[i])
 * (round to nearest-even, saturate to +-448, NaN -> NaN code).  For testing
 * the device conversion against the format definition.  v, q device arrays
 * of n elements (any alignment). */
fp8bs_status fp8bs_e4m3_encode_f32(const float* v, int64_t n, uint8_t* q, fp8bs_stream_t stream);

/* Launch a one-warp kernel that waits, with the library's bounded wait, on a
 * barrier nothing ever completes, giving up after timeout_ns nanoseconds.
 * The next fp8bs_sync_status() must then report FP8BS_ERR_TIMEOUT.  Exercises
 * the failure path without faulting or hanging the GPU. */
fp8bs_status fp8bs_debug_wait_timeout(uint64_t timeout_ns, fp8bs_stream_t stream);

/* Library version, (major << 16) | (minor << 8) | patch. */
int fp8bs_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FP8BS_H */
