/*
 * awq.h -- C ABI of libawq, a GB300 (sm_103a) implementation of the group-wise
 * INT4 weight-only quantized linear layer (AWQ W4A16) and its W4A8 variant.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every pointer argument is a DEVICE pointer on the current CUDA device,
 *    unless the comment says otherwise.  The caller owns every buffer; the
 *    library allocates nothing (scratch space is the caller's `workspace`).
 *  - fp16 values travel as raw IEEE binary16 bits in uint16_t.
 *  - Matrices are dense and row-major.  M = tokens, K = input features
 *    (reduction), N = output features, group_size = input channels per
 *    quantization group (128 on the GPU path).
 *  - Every call is asynchronous on `stream` (NULL = the legacy default
 *    stream).  Argument checks run on the host before anything is launched;
 *    a failing check returns a negative status and launches nothing.  No
 *    C++ exception crosses this boundary.
 *  - Packing ("older" AWQ format): a packed int32 word c of a row holds the
 *    4-bit codes of logical columns 8c..8c+7; nibble slot i (bits 4i..4i+3)
 *    holds column 8c + map[i] with map = [0, 2, 4, 6, 1, 3, 5, 7].
 *    Source: "Speed up AWQ 2.5x with updated kernel" (vLLM pull request),
 *    casper-hansen's list of format differences between the older and the
 *    new AWQ format.
 *  - Pointers to matrices must be 16-byte aligned (AWQ_EALIGN otherwise).
 */
#ifndef AWQ_H_
#define AWQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream; NULL selects the legacy default stream. */
typedef struct CUstream_st *awq_stream_t;

typedef enum {
  AWQ_OK = 0,
  AWQ_EINVAL = -1,      /* a size or shape argument is out of range */
  AWQ_EALIGN = -2,      /* a matrix pointer is not 16-byte aligned */
  AWQ_EARCH = -3,       /* the current device is not a compute-capability 10.3 GPU */
  AWQ_ECUDA = -4,       /* a CUDA runtime call or a kernel launch failed */
  AWQ_ETIMEOUT = -5,    /* a bounded device-side wait expired (awq_last_device_error) */
  AWQ_EWORKSPACE = -6,  /* workspace NULL or smaller than awq_workspace_bytes() */
  AWQ_ENULL = -7        /* a required pointer is NULL */
} awq_status;

/* Operation selector for awq_workspace_bytes(). */
typedef enum {
  AWQ_OP_GEMV = 0,
  AWQ_OP_GEMM = 1,
  AWQ_OP_W4A8_GEMM = 2,
  AWQ_OP_GEMV_PREPACKED = 3,
  AWQ_OP_GEMV_BF16 = 4,
  AWQ_OP_GEMM_BF16 = 5,
  AWQ_OP_W4A8_GROUPED = 6
} awq_op;

/* Human-readable name of a status code (static string, never NULL). */
const char *awq_status_string(awq_status status);

/*
 * awq_pack -- pack 4-bit codes into AWQ int32 words.
 * q: uint8 [rows, n] codes (values above 15 are clamped to 15);
 * packed: int32 [rows, n/8].  n % 8 == 0, rows >= 0.
 * Source: the older-format order map ("Speed up AWQ 2.5x with updated
 * kernel", casper-hansen's format differences); the clamp follows the packer
 * fix reported in "Support W4A8 quantization for vllm" (HandH1998's reply to
 * brisker about the missing clamp in the per-channel pack).
 */
awq_status awq_pack(const uint8_t *q, int64_t rows, int64_t n, int32_t *packed,
                    awq_stream_t stream);

/* awq_unpack -- inverse of awq_pack: packed int32 [rows, n/8] -> uint8 codes [rows, n]. */
awq_status awq_unpack(const int32_t *packed, int64_t rows, int64_t n, uint8_t *q,
                      awq_stream_t stream);

/*
 * Order maps of the two AWQ formats: the older one (map [0, 2, 4, 6, 1, 3, 5, 7], the format every
 * other entry point takes) and the new one (map [0, 1, ..., 7]: nibble slot i holds column 8c + i).
 * Source: "Speed up AWQ 2.5x with updated kernel", casper-hansen's list of format differences.  The
 * new format's other differences (skipped zeros, calculate_zeros_width) are not specified there and
 * are not supported.
 */
typedef enum { AWQ_ORDER_OLD = 0, AWQ_ORDER_NEW = 1 } awq_order;

/* awq_pack_order / awq_unpack_order -- awq_pack / awq_unpack with the order map chosen by `order`
 * (AWQ_EINVAL for another value).  Codes above 15 are clamped as by awq_pack. */
awq_status awq_pack_order(const uint8_t *q, int64_t rows, int64_t n, awq_order order, int32_t *packed,
                          awq_stream_t stream);
awq_status awq_unpack_order(const int32_t *packed, int64_t rows, int64_t n, awq_order order,
                            uint8_t *q, awq_stream_t stream);

/*
 * awq_dequant -- W[k, n] = fp16_RN((q[k, n] - z[k / g, n]) * s[k / g, n]).
 * qweight int32 [K, N/8]; qzeros int32 [K/g, N/8] or NULL for the symmetric
 * variant (z = 8); scales fp16 [K/g, N]; w fp16 [K, N] (output).
 * K % group_size == 0, N % 8 == 0, group_size in {32, 64, 128, 256}.
 * The result is bit-identical to the correctly rounded product.
 * Source: the qweight / scales / qzeros / group_size operands of the AWQ
 * kernels ("Speed up AWQ 2.5x with updated kernel", dispatch snippet);
 * symmetric variant: "Marlin symmetric quantization and inference".
 */
awq_status awq_dequant(const int32_t *qweight, const int32_t *qzeros, const uint16_t *scales,
                       int64_t K, int64_t N, int32_t group_size, uint16_t *w,
                       awq_stream_t stream);

/*
 * awq_workspace_bytes -- bytes of caller-owned workspace that awq_gemv,
 * awq_gemm or w4a8_gemm need for the given shape and split_k (0 = the
 * library's automatic choice, which this function resolves the same way the
 * compute call does).  Returns 0 when no workspace is needed.
 *
 * Workspace contract: before its FIRST use the workspace must be zero-filled
 * (cudaMemsetAsync); every call that completes leaves its tile counters at
 * zero again, so consecutive calls on one stream can reuse it without
 * re-zeroing.  Calls that may run concurrently need separate workspaces.
 * After AWQ_ETIMEOUT, zero the workspace again before reusing it.
 */
size_t awq_workspace_bytes(awq_op op, int64_t M, int64_t K, int64_t N, int32_t split_k);

/*
 * awq_gemv -- y = x * W for M <= 16 tokens (decode), W dequantized on the fly.
 * x fp16 [M, K]; qweight int32 [K, N/8]; qzeros int32 [K/128, N/8] or NULL
 * (symmetric, z = 8); scales fp16 [K/128, N]; y fp16 [M, N] (output).
 * 1 <= M <= 16 (0 = no-op), K % 128 == 0, N % 32 == 0, group_size == 128.
 * M > 8 runs as two 8-token halves sharing each dequantized weight, which is
 * made as W = fp16_RN((q - z) * s) like awq_dequant's.
 * split_k: number of CTAs per 512-column tile, whose K slices are reduced in
 * fp32 (0 = automatic: a persistent grid of one CTA per SM, each owning an
 * equal share of the (tile, 64-row block) units; 1 = one CTA per tile, no
 * shared tile).  When tiles are shared the grid never exceeds one CTA per SM,
 * so a larger split_k is clamped: a tile is completed by the CTA holding its
 * first 64-row block, which waits (bounded) for the other contributors'
 * partials, so the call assumes its CTAs can all be resident at once (no
 * other kernel holding SMs indefinitely).  The fp16 output is rounded once
 * from the fp32 sum, adding the partials in a fixed order (bit-reproducible).
 * Needs a workspace when a tile is shared by several CTAs
 * (awq_workspace_bytes() > 0).  For M <= 8 the group's zero point and scale
 * are applied to fp32 sums of the integer codes, so the products use
 * s * (q - z) in fp32 rather than its fp16 rounding (well inside the fp16
 * output tolerance).
 * Source: the M <= 8 branch of the dispatch snippet, gemv_forward_cuda(inputs,
 * qweight, scales, qzeros, group_size) ("Speed up AWQ 2.5x with updated kernel").
 */
awq_status awq_gemv(const uint16_t *x, const int32_t *qweight, const int32_t *qzeros,
                    const uint16_t *scales, uint16_t *y, int64_t M, int64_t K, int64_t N,
                    int32_t group_size, int32_t split_k, void *workspace,
                    size_t workspace_bytes, awq_stream_t stream);

/*
 * awq_gemv_noalloc -- awq_gemv for callers that cannot allocate device memory.
 * The pages have no counterpart to this entry point; it exists for callers such as a
 * plugin inside an inference runtime that owns all device memory and gives the plugin
 * no allocator, or a serving loop that forbids allocation after start-up (cudaMalloc
 * may synchronize the device).  Same arguments, results and checks as awq_gemv, minus
 * the workspace: the split-K scratch lives in a fixed 8 MiB array inside the library
 * on every GPU that loads it, held until the process exits.  The call allocates
 * nothing (no cudaMalloc / cudaFree, no allocating library routine).
 *  - The first call on each device resolves the array's device address
 *    (cudaGetSymbolAddress with that device current); make that first call before
 *    any stream capture.
 *  - Automatic split (split_k = 0) shrinks the split until its scratch fits 8 MiB
 *    (split 1 needs none); an explicit split_k whose scratch (64 KB of tickets +
 *    contributors per tile * tiles * T * 512 * 4 bytes, with T = 8 token rows per
 *    partial for M <= 8 and T = 16 for 9..16 tokens; the same size
 *    awq_workspace_bytes(AWQ_OP_GEMV, ...) gives awq_gemv) exceeds 8 MiB is rejected
 *    with AWQ_EWORKSPACE.
 *  - Every call shares the array and clears the tickets it needs on `stream` before
 *    its kernel; calls whose kernels overlap on the GPU (other streams, other host
 *    threads) race on the array and must be serialized by the caller.
 *  - A bounded device wait that expires is recorded in the same device error word as
 *    awq_gemv's (read it with awq_last_device_error); that word is also a fixed
 *    variable inside the library, so reporting allocates nothing.
 */
awq_status awq_gemv_noalloc(const uint16_t *x, const int32_t *qweight, const int32_t *qzeros,
                            const uint16_t *scales, uint16_t *y, int64_t M, int64_t K, int64_t N,
                            int32_t group_size, int32_t split_k, awq_stream_t stream);

/*
 * Prepared decode weights.  The decode GEMV reads its weights fastest from a copy laid out for it,
 * made once when the layer is loaded (the pages' W4A8 kernel shuffles its int4 weights offline in
 * the same spirit: "Support W4A8 quantization for vllm", HandH1998 on the 8 INT4 weights of one
 * INT32 shuffled offline so that every thread of a warp fetches the right weights).  The copy holds
 * exactly the codes, zero points and scales of the AWQ layer, rearranged: for each 256-column tile
 * (tile-major) and each 128-row group, one 17024-byte unit of
 *   - codes as uint32 words [warp w: 4][16-row step i: 8][lane l: 32][column pair b: 4]; word
 *     (w, i, l, b), with g = l / 4, t = l % 4, even column ce = 256 T + 64 w + 8 g + 2 b, odd column
 *     co = ce + 1 and rows k = 128 G + 16 i + (2t, 2t+1, 2t+8, 2t+9), holds from the lowest nibble
 *     up q[2t, ce], q[2t, co], q[2t+8, ce], q[2t+8, co], q[2t+1, ce], q[2t+1, co], q[2t+9, ce],
 *     q[2t+9, co];
 *   - zero points as uint32 words [w: 4][g: 8], nibble c = z of column 256 T + 64 w + 8 g + c
 *     (8 for the symmetric variant);
 *   - scales as fp16 [w: 4][g: 8][c: 8] of the same columns.
 * Columns at or beyond N hold code 0, zero point 0 and scale 0.
 *
 * awq_prepacked_bytes -- bytes of the prepared copy: ceil(N / 256) * (K / 128) * 17024
 * (0 for a shape the GEMV does not take: K % 128 != 0 or N % 32 != 0).
 */
size_t awq_prepacked_bytes(int64_t K, int64_t N);

/*
 * awq_prepack_gemv -- writes the prepared copy of an AWQ layer (group size 128) into `packed`
 * (device memory of at least awq_prepacked_bytes(K, N) bytes, 16-byte aligned, caller-owned).
 * qweight int32 [K, N/8]; qzeros int32 [K/128, N/8] or NULL (symmetric, z = 8); scales fp16
 * [K/128, N].  K % 128 == 0, N % 32 == 0.  AWQ_EINVAL for a shape outside that or a `packed_bytes`
 * below the size needed.  Bit-exact and reversible (awq_unprepack_gemv).
 */
awq_status awq_prepack_gemv(const int32_t *qweight, const int32_t *qzeros, const uint16_t *scales,
                            int64_t K, int64_t N, int32_t group_size, void *packed,
                            size_t packed_bytes, awq_stream_t stream);

/*
 * awq_unprepack_gemv -- the inverse: the AWQ words, zero points (packed like AWQ qzeros; pass NULL
 * to skip them, e.g. for a symmetric layer) and scales that `packed` was made from.
 */
awq_status awq_unprepack_gemv(const void *packed, int64_t K, int64_t N, int32_t *qweight,
                              int32_t *qzeros, uint16_t *scales, awq_stream_t stream);

/*
 * awq_gemv_prepacked -- y = x * W for M <= 8 tokens on the prepared copy: the same result as
 * awq_gemv (the same fold of zero point and scale into fp32 sums, one rounding of the output; the
 * fp32 summation order differs).  x fp16 [M, K], packed from awq_prepack_gemv, y fp16 [M, N].
 * 1 <= M <= 8 (0 = no-op), K % 128 == 0, N % 32 == 0.  split_k as for awq_gemv, over 256-column
 * tiles: a tile shared by several CTAs is completed by the CTA holding its first group, which waits
 * (bounded) for the other contributors, so the call assumes its CTAs can all be resident at once.
 * Needs a workspace when a tile is shared (awq_workspace_bytes(AWQ_OP_GEMV_PREPACKED, ...) > 0;
 * same contract as awq_gemv's).  Two of its CTAs fit on one SM, so with programmatic dependent launch
 * the next call's CTAs stream their weights while this call finishes.
 * Source: as awq_gemv (the M <= 8 branch of the dispatch snippet in "Speed up AWQ 2.5x with updated
 * kernel").
 */
awq_status awq_gemv_prepacked(const uint16_t *x, const void *packed, uint16_t *y, int64_t M,
                              int64_t K, int64_t N, int32_t split_k, void *workspace,
                              size_t workspace_bytes, awq_stream_t stream);

/*
 * awq_gemm -- y = x * W on the tensor cores (tcgen05, fp16 x fp16 -> fp32 in
 * tensor memory) for any M >= 1 (intended for M > 8: prefill).
 * Same operands and layouts as awq_gemv; K % 128 == 0, N % 32 == 0,
 * group_size == 128.  split_k: K slices reduced in fp32 (0 = automatic).
 * Source: the M > 8 branch of the dispatch snippet, gemmv2_forward_cuda(
 * inputs, qweight, scales, qzeros, group_size, split_k_iters) ("Speed up AWQ
 * 2.5x with updated kernel").
 */
awq_status awq_gemm(const uint16_t *x, const int32_t *qweight, const int32_t *qzeros,
                    const uint16_t *scales, uint16_t *y, int64_t M, int64_t K, int64_t N,
                    int32_t group_size, int32_t split_k, void *workspace,
                    size_t workspace_bytes, awq_stream_t stream);

/*
 * bf16 variant of the W4A16 layer.  Many models are trained in bf16 ("Support W4A8 quantization for
 * vllm": brisker's question on bf16 support and HandH1998's answer that the W4A8 kernel there does not
 * support it).  These entry points take bf16 activations and scales (raw bf16 bits in uint16_t, the
 * upper half of an IEEE binary32) and write bf16 outputs; codes and zero points are packed as for the
 * fp16 entry points.
 *
 * awq_dequant_bf16 -- W[k, n] = bf16_RN((q[k, n] - z[k / g, n]) * s[k / g, n]); same arguments and
 * checks as awq_dequant, bf16 scales and output.  Bit-identical to the correctly rounded product.
 *
 * awq_gemv_bf16 -- y = x * W for M <= 16 tokens, bf16 x [M, K], scales, y [M, N].  Every weight is
 * made exactly as awq_dequant_bf16 makes it and multiplied on the tensor pipe with fp32 accumulation;
 * the output is rounded once.  Runs the 8-token instance of the decode kernel up to 8 tokens and the
 * 16-token one above (workspace: awq_workspace_bytes(AWQ_OP_GEMV_BF16, ...), sized for 16 token rows
 * of partials whatever M); split_k and the residency assumption as for awq_gemv.
 *
 * awq_gemm_bf16 -- the tensor-core GEMM (tcgen05 kind::f16 with bf16 A and B) for any M >= 1, bf16
 * x, scales and y; workspace awq_workspace_bytes(AWQ_OP_GEMM_BF16, ...); otherwise as awq_gemm.
 */
awq_status awq_dequant_bf16(const int32_t *qweight, const int32_t *qzeros, const uint16_t *scales,
                            int64_t K, int64_t N, int32_t group_size, uint16_t *w,
                            awq_stream_t stream);
awq_status awq_gemv_bf16(const uint16_t *x, const int32_t *qweight, const int32_t *qzeros,
                         const uint16_t *scales, uint16_t *y, int64_t M, int64_t K, int64_t N,
                         int32_t group_size, int32_t split_k, void *workspace,
                         size_t workspace_bytes, awq_stream_t stream);
awq_status awq_gemm_bf16(const uint16_t *x, const int32_t *qweight, const int32_t *qzeros,
                         const uint16_t *scales, uint16_t *y, int64_t M, int64_t K, int64_t N,
                         int32_t group_size, int32_t split_k, void *workspace,
                         size_t workspace_bytes, awq_stream_t stream);

/*
 * w4a8_quant_act -- per-token dynamic int8 quantization of activations.
 * x fp16 [M, K]; xq int8 [M, K] (output); s_tok fp32 [M] (output).
 * s_tok[m] = fp32(fp16_RN(absmax_k |x[m, k]| / 127)) computed in fp32,
 * xq = clamp(rint(x / s_tok), -128, 127); an all-zero row gives s = 0, xq = 0.
 * M >= 1, K % 8 == 0.
 * Source: "Support W4A8 quantization for vllm", the dynamic_quant function of
 * brisker's consistency script and HandH1998's note that s1 is the dynamic
 * per-token scale computed online.
 */
awq_status w4a8_quant_act(const uint16_t *x, int8_t *xq, float *s_tok, int64_t M, int64_t K,
                          awq_stream_t stream);

/*
 * w4a8_gemm -- W4A8 product with exact int32 accumulation.
 * xq int8 [M, K]; s_tok fp32 [M]; wq int32 [K, N/8] holding u = q + 8 for
 * signed int4 weights q in [-8, 7], AWQ packing; s_ch fp16 [N] per-output-
 * channel scales; y fp16 [M, N] (output); acc_out int32 [M, N] (optional
 * output of the exact accumulator, NULL to skip).
 * acc[m, n] = sum_k xq[m, k] * q[k, n] (exact), y = fp16_RN((fp32(acc) *
 * s_tok[m]) * fp32(s_ch[n])).  K % 128 == 0, N % 32 == 0.
 * Always needs a workspace (it holds an fp16 copy of xq for the fp16 tensor
 * path; every int8 and int4 value and every product is exact in fp16/fp32).
 * split_k: K slices reduced in int32 across CTAs (0 = automatic).  Inside a
 * CTA every 16384 inputs get their own fp32 tensor-memory accumulator (two at
 * most), so each fp32 sum is an exact integer; K beyond 32768 per slice is
 * split across CTAs.  With 128 or more tokens and K <= 16384 a CTA covers 256
 * output channels with one accumulator each (two 128-channel blocks sharing
 * every activation tile).
 * With at most 16 tokens the product runs on the decode GEMV instead (up to 8
 * tokens it takes sum (1024 + u) x and sum x per 64-row block, exact integers
 * in fp32, and subtracts the offset exactly; from 9 to 16 tokens it makes the
 * weights u - 8 exactly in fp16; fp32 sums stay below 2^24 within a CTA and
 * are added as int32 across CTAs), whenever its plan for split_k keeps each
 * CTA's rows of a 512-column tile within 16384; otherwise on the GEMM.
 * The results are identical either way.
 * Source: "Support W4A8 quantization for vllm": marlin_qqq_gemm(a, b_q_weight,
 * s1, s2, s3, workspace, size_m, size_n, size_k) in tlrmchlsmth's review;
 * HandH1998's per-channel dequantization (int4 to int8, channel scale on the
 * output); alexm's note that the global reduce works on int32 elements in a
 * temporary buffer C.
 */
awq_status w4a8_gemm(const int8_t *xq, const float *s_tok, const int32_t *wq,
                     const uint16_t *s_ch, uint16_t *y, int32_t *acc_out, int64_t M, int64_t K,
                     int64_t N, int32_t split_k, void *workspace, size_t workspace_bytes,
                     awq_stream_t stream);

/*
 * w4a8_linear -- w4a8_quant_act and w4a8_gemm in one call, from fp16 activations.
 * x fp16 [M, K]; wq, s_ch, y, acc_out, split_k, workspace as for w4a8_gemm
 * (the same workspace size: awq_workspace_bytes(AWQ_OP_W4A8_GEMM, ...));
 * s_tok fp32 [M] (output, required: the per-token scales the epilogue uses);
 * xq_out int8 [M, K] (optional output of the codes, NULL to skip).
 * The quantization writes the codes widened to fp16 straight into the
 * workspace for the fp16 tensor path, so the int8 codes need not round-trip
 * through memory.  Results are bit-identical to w4a8_quant_act followed by
 * w4a8_gemm.
 * Source: "Support W4A8 quantization for vllm": the description's news list
 * (dynamic activation quantization fused into the QQQ linear method) and
 * HandH1998's reply on moving the activation quantization out of the
 * surrounding layers into the linear method; the per-token scale computed
 * online.
 */
awq_status w4a8_linear(const uint16_t *x, const int32_t *wq, const uint16_t *s_ch, uint16_t *y,
                       int32_t *acc_out, int8_t *xq_out, float *s_tok, int64_t M, int64_t K,
                       int64_t N, int32_t split_k, void *workspace, size_t workspace_bytes,
                       awq_stream_t stream);

/*
 * W4A8 with per-group weight factors.  The per-channel W4A8 kernel widens an int4 weight to int8 by a
 * shift of 4 and applies the channel scale to the output; per-group weight quantization needs a group
 * scale as well as the channel scale, and the reduction stays on int32 ("Support W4A8 quantization for
 * vllm": HandH1998 on FragS_GROUP and FragS_CHANNEL, on dequant_per_channel as a shift of 4 bits, alexm
 * on the int32 global reduce; marlin_qqq_gemm(a, b_q_weight, s1, s2, s3, ...)).  Reading of the group
 * scale: s3 [K/128, N] holds integers in [1, 16] (fp16 storage), the per-group factor that turns the
 * int4 weight into an int8 one; s3 = 16 everywhere is the per-channel kernel.
 *   acc[m, n] = sum_k xq[m, k] * ((u[k, n] - 8) * s3[k / 128, n])   (exact, int32)
 *   y[m, n]   = fp16_RN((fp32(acc) * s_tok[m]) * fp32(s2[n]))
 * Factors outside the integers 1..16 give unspecified (but memory-safe) results.
 *
 * w4a8_gemm_grouped -- from int8 codes: xq int8 [M, K], s_tok fp32 [M], wq int32 [K, N/8] (AWQ-packed
 * u = q + 8), s3 fp16 [K/128, N], s2 fp16 [N], y fp16 [M, N], acc_out int32 [M, N] (optional).  Runs the
 * tensor-core GEMM for every M: weights (u - 8) * s3 made exactly in fp16, codes widened to fp16 in the
 * workspace, each 1024 rows in their own fp32 tensor-memory accumulator (an exact integer: |code| <= 128,
 * |weight| <= 128), token tiles of at most 64, K beyond one slice of 512 / tile * 1024 rows reduced across
 * CTAs in int32.  K % 128 == 0, N % 32 == 0, group_size == 128.  Workspace:
 * awq_workspace_bytes(AWQ_OP_W4A8_GROUPED, ...).
 *
 * w4a8_linear_grouped -- the same from fp16 activations, quantized per token as w4a8_quant_act does
 * (s_tok fp32 [M] output, required; xq_out int8 [M, K] optional), one call.
 */
awq_status w4a8_gemm_grouped(const int8_t *xq, const float *s_tok, const int32_t *wq,
                             const uint16_t *s3, const uint16_t *s2, uint16_t *y, int32_t *acc_out,
                             int64_t M, int64_t K, int64_t N, int32_t group_size, int32_t split_k,
                             void *workspace, size_t workspace_bytes, awq_stream_t stream);
awq_status w4a8_linear_grouped(const uint16_t *x, const int32_t *wq, const uint16_t *s3,
                               const uint16_t *s2, uint16_t *y, int32_t *acc_out, int8_t *xq_out,
                               float *s_tok, int64_t M, int64_t K, int64_t N, int32_t group_size,
                               int32_t split_k, void *workspace, size_t workspace_bytes,
                               awq_stream_t stream);

/*
 * awq_last_device_error -- reads and clears the device-side error word of the
 * current device (synchronous: waits for the device).  *code receives 0 when
 * no bounded wait expired since the last read, else the id of the wait that
 * gave up.  Returns AWQ_ETIMEOUT when *code != 0.
 */
awq_status awq_last_device_error(int32_t *code);

/*
 * awq_selftest_wait_timeout -- runs, on `stream`, one bounded device-side wait on
 * an mbarrier that nothing arrives on, with a limit of `limit_ns` nanoseconds
 * (0 < limit_ns <= 2e9) instead of the kernels' 2 s.  The wait expires, records
 * id 901 in the device error word and returns; awq_last_device_error() then
 * reports AWQ_ETIMEOUT with code 901, and the context stays usable.  It lets a
 * caller (and the tests) check the failure path of every kernel's waits without
 * faulting or hanging the GPU.  No source passage: the pages describe no
 * failure handling.  Returns AWQ_EINVAL for a limit outside the range,
 * AWQ_EARCH off sm_103, AWQ_ECUDA when the launch fails.
 */
awq_status awq_selftest_wait_timeout(int64_t limit_ns, awq_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* AWQ_H_ */
