/*
 * exl3.h -- C ABI of libexl3.so, the EXL3 trellis-quantized linear layer on sm_103a.
 *
 * The layer computes
 *
 *     y = svh * H_N( Wq^T-contraction( H_K(x * suh) * 2^-4 ) ) * 2^-3
 *
 * where H_K / H_N are block-diagonal 128-point Hadamard transforms and Wq is
 * decoded on the fly from 16x16 trellis tiles (cuda-exl3 README, "Why custom
 * kernels" and "One op per layer"; TensorFold PR #740, "Arithmetic").
 *
 * Conventions shared by every call:
 *  - All tensor pointers are DEVICE pointers owned by the caller, C-contiguous,
 *    16-byte aligned.  The library allocates nothing and keeps no per-layer
 *    state; it never synchronises the host.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    Work is enqueued asynchronously on it.
 *  - Every argument is validated on the host before anything is launched.  An
 *    invalid call returns EXL3_EINVAL (or EXL3_EWORKSPACE) and launches nothing.
 *    A launch failure returns EXL3_ECUDA; exl3_last_error() gives the CUDA text.
 *  - fp16 / bf16 values are passed as their 16-bit patterns (uint16_t).
 *  - m == 0 is an empty batch: the call returns EXL3_OK and launches nothing;
 *    the activation, output and workspace pointers may then be NULL.
 *    m may be at most EXL3_MAX_ROWS.
 *  - k and n are multiples of 128 (whole Hadamard blocks; cuda-exl3 README,
 *    "Loading into a dim vLLM has padded").  bits is 1..8 (cuda-exl3 README,
 *    "What is supported").
 *  - Padded dims (same passage).  A dim padded for tensor parallelism is padded
 *    by whole 128-blocks, and the library needs nothing special for it:
 *      output (n) pad: the caller sets svh = 0 on the pad columns; those outputs
 *        are then exactly zero whatever trellis words sit behind them (every
 *        code decodes finite), and the real columns are unchanged because the
 *        output rotation mixes only inside a 128-column block;
 *      input (k) pad: when loading a checkpoint layer of K_real rows into a dim
 *        of K rows, the caller copies the K_real/16 trellis tile rows and the
 *        K_real suh entries per shard that exist and zeroes the rest (it must
 *        not read past the checkpoint's end), and the activations carry exact
 *        zeros on the pad positions (the producing layer's padded output
 *        already does).  The result equals the unpadded layer's, byte for byte
 *        for exl3_gemm (the extra k16 steps add exact zeros).
 */
#ifndef EXL3_H
#define EXL3_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { EXL3_CB_3INST = 0, EXL3_CB_MCG = 1, EXL3_CB_MUL1 = 2 } exl3_codebook_t;
typedef enum { EXL3_F16 = 0, EXL3_BF16 = 1 } exl3_dtype_t;
typedef enum {
  EXL3_OK = 0,
  EXL3_EINVAL = 1,       /* bad shape, pointer, alignment, width, codebook or shard map */
  EXL3_EUNSUPPORTED = 2, /* valid request this build does not implement */
  EXL3_EWORKSPACE = 3,   /* split-k accumulator too small */
  EXL3_ECUDA = 4         /* a CUDA launch or runtime call failed */
} exl3_status_t;

/* Largest batch (rows of x) one call accepts. */
#define EXL3_MAX_ROWS (1 << 22)

/* Maximum number of fused shards in one call (qkv = 3, gate_up = 2). */
#define EXL3_MAX_SHARDS 8

/*
 * exl3_input_transform -- input rotation of every shard in one pass over x.
 *
 * TensorFold PR #740, "Arithmetic" step 1; cuda-exl3 README, "One op per layer"
 * (activation transform fused, bf16 -> fp16 folded into the load).  For each
 * shard s, row r and 128-block b of k:
 *     xh[s][r][128b+i] = fp16_rne( 2^-4 * sum_j H[i][j] * (x[r][128b+j] * suh[s][128b+j]) )
 * with H[i][j] = (-1)^popcount(i & j), the product x*suh exact in fp32 and the
 * sum taken as a radix-2 butterfly in fp32 with a fixed order of adds.
 *
 *   x        device, [m][k] of x_dtype (bf16 or fp16)
 *   suh      device, fp16 [num_shards][k]
 *   xh       device, fp16 [num_shards][m][k] (output)
 */
exl3_status_t exl3_input_transform(const void* x, exl3_dtype_t x_dtype, int64_t m, int64_t k,
                                   const uint16_t* suh, int32_t num_shards, uint16_t* xh,
                                   void* stream);

/*
 * exl3_input_transform_swiglu -- the down-projection's input transform with the
 * gated MLP's SwiGLU folded in (cuda-exl3 README, "MoE throughput": folding
 * SwiGLU into the down-projection's input transform removes an elementwise
 * pass).  The pages print no formula; this library reads it as the usual
 * SwiGLU with the gate first:
 *     h[r][j]      = silu(g) * u,  g = gate_up[r][j], u = gate_up[r][k + j],
 *                    silu(g) = g / (1 + e^-g), in fp32
 *     xh[s][r][:]  = as exl3_input_transform with h in place of x
 * (the layout a gate_up layer fused as two shards of width k writes).
 *   gate_up  device, [m][2k] of dtype (bf16 or fp16), 16-byte aligned
 *   suh      device, fp16 [num_shards][k]
 *   xh       device, fp16 [num_shards][m][k] (output)
 * Validation and the empty batch as for exl3_input_transform.
 */
exl3_status_t exl3_input_transform_swiglu(const void* gate_up, exl3_dtype_t dtype, int64_t m, int64_t k,
                                          const uint16_t* suh, int32_t num_shards, uint16_t* xh,
                                          void* stream);

/*
 * exl3_gemm -- trellis decode fused into the contraction, output rotation fused
 * into the epilogue, all shards of a fused layer in one launch.
 *
 * cuda-exl3 README, "Why custom kernels" (a block owns its columns and the whole
 * k extent, so the output Hadamard and svh fold into the epilogue) and "Notes on
 * the format" (trellis and svh concatenate along n; one suh row, hence one xh
 * slice, per shard).  TensorFold PR #740, "Arithmetic" steps 2-3.
 *     z[r][c]  = sum_k xh[s(c)][r][k] * Wq[k][c]      (fp16 products, fp32 sums)
 *     y[r][c]  = out_rne( svh[c] * 2^-3 * sum_j H[i][j] z[r][128b+j] ),  c = 128b+i
 * Wq[k][c] is decoded from trellis tile (k/16, c/16).  The fp32 sum over k runs
 * in a fixed order that does not depend on m, so each row's bytes are the same
 * at every batch size.
 *
 *   xh         device, fp16 [num_shards][m][k] (exl3_input_transform's output)
 *   trellis    device, int16 [k/16][n/16][16*bits]
 *   bits       1..8;  cb: codebook id
 *   svh        device, fp16 [n]
 *   shard_cols HOST, int32 [num_shards+1]: 0 = c_0 < c_1 < ... < c_S = n, multiples
 *              of 128; shard s owns output columns [c_s, c_{s+1})
 *   y          device, [m][n] of y_dtype (output)
 *
 * Launch overlap: the GEMM kernel is launched with programmatic stream
 * serialization, and exl3_input_transform's kernel lets its dependents start
 * early.  So the GEMM may begin (and read trellis and svh) while the kernel
 * before it in the stream is still running, provided that kernel allows it;
 * it reads xh and writes y only after that kernel has completed.  A caller's
 * own kernel that allows early dependents must therefore not write the
 * trellis or svh that the following GEMM uses.
 */
exl3_status_t exl3_gemm(const uint16_t* xh, int64_t m, int64_t k, const int16_t* trellis,
                        int32_t bits, exl3_codebook_t cb, const uint16_t* svh,
                        const int32_t* shard_cols, int32_t num_shards, void* y,
                        exl3_dtype_t y_dtype, int64_t n, void* stream);

/*
 * Split-k variant.  cuda-exl3 README, "One op per layer" (split-k for narrow
 * layers: partials go to an fp32 accumulator that a second kernel turns into
 * outputs while zeroing it again); TensorFold PR #740, "Arithmetic" (k
 * blocks split into a number of parts fixed by the shape, parts added in part
 * order).  Part p covers a contiguous range of k: whole 256-row units when
 * k/128 is even and P <= k/256 (so a part never splits a four-atom stage),
 * else whole 128-row blocks, in either case part p takes units
 * [p*U/P, (p+1)*U/P) of the U units; its
 * fp32 partial goes to acc[p][r][c]; the epilogue sums p = 0..P-1 in order,
 * applies the output rotation, writes y and writes zeros back to acc.
 *
 * exl3_splitk_parts(k, n) is the number of parts P; it depends on the shape only
 * (never on m), so rows stay byte-equal across batch sizes.  It is a pure host
 * function.  exl3_splitk_workspace_bytes(m, k, n) = P * m * n * 4.
 *
 *   acc        device, fp32 [P][m][n].  Its contents on entry do not matter:
 *              each part stores every partial it owns (plain stores, no
 *              accumulation into acc) before the epilogue reads it.  The
 *              epilogue writes zeros back, the pages' re-zeroed accumulator,
 *              so with P > 1 acc is all zero when the call's work completes;
 *              nothing relies on that.  With P = 1 the call computes what
 *              exl3_gemm computes, with no partials and no epilogue, and
 *              leaves acc as it found it.  Calls that share one acc must be
 *              ordered on one stream.
 *   acc_bytes  size of acc in bytes; smaller than the workspace size -> EXL3_EWORKSPACE
 *   other arguments as exl3_gemm.
 * If a kernel of the call gives up on a bounded wait (exl3_device_status then
 * reports it), its part skips its stores and y is undefined for that call.
 */
int32_t exl3_splitk_parts(int64_t k, int64_t n);
size_t exl3_splitk_workspace_bytes(int64_t m, int64_t k, int64_t n);
exl3_status_t exl3_gemm_splitk(const uint16_t* xh, int64_t m, int64_t k, const int16_t* trellis,
                               int32_t bits, exl3_codebook_t cb, const uint16_t* svh,
                               const int32_t* shard_cols, int32_t num_shards, void* y,
                               exl3_dtype_t y_dtype, int64_t n, float* acc, size_t acc_bytes,
                               void* stream);

/*
 * Mixture of experts (cuda-exl3 README, "What is supported" and "MoE notes").
 * Routed (token, expert) pairs arrive block-aligned, the layout vLLM's
 * moe_align_block_size writes: pairs sorted by expert, each expert's run padded
 * to whole blocks of `block` rows, so every block belongs to one expert.
 *   sorted_ids    device int32 [rows]: pair index token * topk + slot of each
 *                 padded row; any value outside [0, num_tokens * topk) marks
 *                 a padding row
 *   block_expert  device int32 [rows / block]: expert of each block; -1 (or an
 *                 id >= num_experts) marks a block of no expert, which both
 *                 calls skip (such blocks may sit between live ones)
 *   block         16, 32 or 128; rows a multiple of block (16 is the pages'
 *                 floor, used when few tokens reach each expert: cuda-exl3
 *                 README, "MoE notes")
 *
 * exl3_moe_input_transform: since suh is per expert (and per shard), the input
 * rotation happens after routing: each padded row of a live block gets its
 * token's x rotated with its block's expert's suh, as exl3_input_transform
 * computes it; padding rows get zeros; rows of skipped blocks are not written.
 *   x    device, [num_tokens][k] of x_dtype
 *   suh  device, fp16 [num_experts][num_shards][k]
 *   xh   device, fp16 [num_shards][rows][k] (output)
 *
 * exl3_moe_gemm: the grouped GEMM.  Each live block's rows go through its
 * expert's layer exactly as exl3_gemm computes it (same fixed fp32 order, so a
 * row's bytes equal exl3_gemm's with that expert); skipped blocks' rows of y
 * are not written.
 *   xh       device, fp16 [num_shards][rows][k] (exl3_moe_input_transform's output)
 *   trellis  device, int16 [num_experts][k/16][n/16][16*bits] (experts stacked)
 *   svh      device, fp16 [num_experts][n]
 *   y        device, [rows][n] of y_dtype (output, in padded-row order; the
 *            weighted combine over each token's top-k rows is the caller's)
 * Validation and empty input as for exl3_gemm; EXL3_EINVAL also for a block
 * size other than 16, 32 or 128, rows not a multiple of it, or no experts.  The
 * kernel reads block_expert before it waits for the previous kernel in the
 * stream, like the trellis (see exl3_gemm).
 */
exl3_status_t exl3_moe_input_transform(const void* x, exl3_dtype_t x_dtype, int64_t num_tokens, int64_t k,
                                       const int32_t* sorted_ids, int64_t rows, int32_t topk,
                                       const int32_t* block_expert, int32_t block, const uint16_t* suh,
                                       int32_t num_shards, int32_t num_experts, uint16_t* xh, void* stream);
exl3_status_t exl3_moe_gemm(const uint16_t* xh, int64_t rows, int64_t k, const int16_t* trellis,
                            int32_t bits, exl3_codebook_t cb, const uint16_t* svh,
                            const int32_t* shard_cols, int32_t num_shards, const int32_t* block_expert,
                            int32_t block, int32_t num_experts, void* y, exl3_dtype_t y_dtype, int64_t n,
                            void* stream);

/*
 * exl3_moe_combine: the weighted sum of each token's top-k expert rows, the
 * step after the grouped GEMM (the pages leave it to the caller: cuda-exl3
 * README, "MoE notes"; the routing layout is the one above).
 *   out[t, :] = sum over s = 0 .. topk-1, in that order, of
 *               weights[t, s] * y[row(t, s), :]
 * where row(t, s) is the padded row of a live block (expert id in
 * [0, num_experts)) whose sorted_ids entry is the pair t * topk + s; a pair
 * with no such row adds nothing (a token with none gets zeros).  The sum is
 * fp32, one fused multiply-add per slot in slot order, then one rounding to
 * out_dtype; padding rows and rows of blocks of no expert are never read.
 *   y          device, [rows][n] of y_dtype (exl3_moe_gemm's output)
 *   weights    device, fp32 [num_tokens][topk] (the router's top-k weights)
 *   pair_rows  device, int32 [num_tokens * topk] scratch owned by the caller:
 *              the call writes the row of every routed pair into it first and
 *              checks each entry it reads against sorted_ids and block_expert,
 *              so it needs no clearing between calls
 *   out        device, [num_tokens][n] of out_dtype (output)
 * Each pair must appear in at most one row of a live block (the layout above
 * guarantees it; with duplicates the row taken is unspecified).  Two kernel
 * launches on `stream`, no synchronisation, no allocation.  EXL3_EINVAL for
 * sizes out of range, rows not a multiple of block, a block size other than
 * 16, 32 or 128, topk outside 1..64, no experts, or a missing or misaligned
 * pointer; num_tokens == 0 does nothing.
 */
exl3_status_t exl3_moe_combine(const void* y, exl3_dtype_t y_dtype, int64_t rows, int64_t n,
                               const int32_t* sorted_ids, const int32_t* block_expert, int32_t block,
                               int32_t num_experts, const float* weights, int64_t num_tokens, int32_t topk,
                               int32_t* pair_rows, void* out, exl3_dtype_t out_dtype, void* stream);

/*
 * exl3_gemm_splitk_noalloc -- the split-k GEMM for callers that cannot allocate.
 *
 * The pages have no counterpart to this call; it exists for callers that have
 * no way to obtain a device workspace (a plugin inside a host program that owns
 * the allocator, or code that must not call cudaMalloc because it would
 * synchronise the device or break a fixed memory budget).  It computes exactly
 * what exl3_gemm_splitk computes, with the same arguments minus the workspace:
 * the fp32 partials go to a scratch array built into the library, of
 * EXL3_NOALLOC_SCRATCH_BYTES per GPU, held on every GPU that loads the library
 * until the process exits.  It calls no allocator.
 *
 *  - Size limit: exl3_splitk_workspace_bytes(m, k, n) must not exceed
 *    EXL3_NOALLOC_SCRATCH_BYTES; a larger request returns EXL3_EWORKSPACE and
 *    launches nothing (use exl3_gemm_splitk with your own workspace instead).
 *  - Each call looks up the scratch array's address in the current device's
 *    context (a lookup that allocates nothing), so no address outlives a
 *    context: after cudaDeviceReset the next call uses the new context's array.
 *    Loading the module on a device happens at its first call; make that call
 *    before any stream capture on that device.
 *  - Every call shares the one array.  Calls whose work may overlap on the GPU
 *    (different streams, or different threads without ordering) race on it and
 *    give wrong results; order them on one stream.  Each call overwrites every
 *    partial it reads, so what an earlier call left behind does no harm.
 *  - As for exl3_gemm_splitk, y is undefined for a call during which
 *    exl3_device_status records a wait that gave up.
 */
#define EXL3_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)
exl3_status_t exl3_gemm_splitk_noalloc(const uint16_t* xh, int64_t m, int64_t k, const int16_t* trellis,
                                       int32_t bits, exl3_codebook_t cb, const uint16_t* svh,
                                       const int32_t* shard_cols, int32_t num_shards, void* y,
                                       exl3_dtype_t y_dtype, int64_t n, void* stream);

/*
 * Test-only entry points (they run the same device decode as exl3_gemm).
 *
 * exl3_test_codebook: out[s] = fp16 bits of codebook cb at state s, s = 0..65535
 *   (TensorFold PR #740, "Tests": all 65,536 states of each codebook).  The
 *   library decodes with two instruction sequences (one per kernel family);
 *   a state where they disagree reads 0xFFFF, a NaN no state decodes to.
 *   out: device, uint16 [65536].
 * exl3_test_unpack: wq[k][n] = decoded weights of the whole trellis as fp16 bits
 *   (TensorFold PR #740, "Tests": random tiles at every width and codebook).
 *   trellis: device int16 [k/16][n/16][16*bits]; wq: device uint16 [k][n].
 *   k and n need only be multiples of 16 here.
 */
exl3_status_t exl3_test_codebook(exl3_codebook_t cb, uint16_t* out, void* stream);
exl3_status_t exl3_test_unpack(const int16_t* trellis, int32_t bits, exl3_codebook_t cb,
                               int64_t k, int64_t n, uint16_t* wq, void* stream);

/*
 * exl3_test_gemm_shape: exl3_gemm (acc == NULL) or exl3_gemm_splitk (acc !=
 * NULL, same workspace rules) with the kernel's tile shape fixed by the caller
 * instead of chosen from the call's sizes.  Every tile shape computes each
 * output element with the same k16 steps in the same order, so the result must
 * be byte-equal to the one the library picks; tests use this to check each
 * shape.  No counterpart in the pages: the tiling is this library's own.
 *   tile_shape: 0 = 32-column strips (m <= 32, k/128 even, no split-k),
 *     1 = 64-column strips (m <= 32), 2 = 128 columns (m <= 32),
 *     3 = 128 columns x 128 rows, 4 = 128 columns x 256 rows,
 *     5 = 256 columns x 256 rows (n and shard edges multiples of 256),
 *     6 = pair of 128-column x 256-row CTAs sharing decoded weights,
 *     7 = pair of 256-column x 256-row CTAs (edges multiples of 256),
 *     8 = 128 columns, four k atoms per stage (m <= 32, k/128 even, no split-k),
 *     9 = 96-column strips in clusters of four CTAs over three Hadamard blocks
 *         (m <= 32, k/128 even, no split-k, n and shard edges multiples of 384),
 *     10 = 96 columns x 128 rows, 11 = 96 columns x 256 rows (clusters of four
 *         as in 9; n and shard edges multiples of 384),
 *     12 = 32-column strips with eight k atoms per stage (m <= 32, k a
 *         multiple of 512, no split-k), 13 = 64-column strips with four
 *         (m <= 32, k/128 even, no split-k), 14 = 96-column strips holding
 *         64 rows with four (m <= 64, k/128 even, no split-k, n and shard
 *         edges multiples of 384), 15 = 64-column strips holding 64 rows with
 *         four (m <= 64, k/128 even, no split-k), 16 = 64-column strips of
 *         128 rows with four (k/128 even, no split-k), 17 = 32-column strips
 *         of 128 rows with four (k/128 even, no split-k).
 *     The decoded weights as the tensor core's 128-row operand and the batch
 *     rows as the narrow one (18, 19, 21, 23 keep the decoded weights in
 *     tensor memory, 20 and 22 in shared memory):
 *     18 = 128 columns, four k atoms per stage (m <= 32, k/128 even; under
 *         split-k only when its parts are whole 256-row units of k), 19 =
 *         128 columns, two k atoms (m <= 32), 20 = 96-column
 *         strips in clusters of four, four k atoms (m <= 32, k/128 even, no
 *         split-k, n and shard edges multiples of 384), 21 and 22 = 18 and 20
 *         holding 16 rows (m <= 16), 23 = 19 holding 16 rows (m <= 16),
 *         24 = 18 holding 64 rows (m <= 64), 25 = 19 holding 64 rows
 *         (m <= 64), 26 = 19 holding 128 rows (m <= 128), 27 = 20 holding
 *         64 rows (m <= 64), 28 = 18 holding 128 rows (m <= 128; two k
 *         atoms per stage at 7-8 bits).
 * Returns EXL3_EUNSUPPORTED, launching nothing, when the shape cannot run the
 * call (the conditions in parentheses).
 */
#define EXL3_TEST_TILE_SHAPES 29
exl3_status_t exl3_test_gemm_shape(int32_t tile_shape, const uint16_t* xh, int64_t m, int64_t k,
                                   const int16_t* trellis, int32_t bits, exl3_codebook_t cb,
                                   const uint16_t* svh, const int32_t* shard_cols, int32_t num_shards,
                                   void* y, exl3_dtype_t y_dtype, int64_t n, float* acc, size_t acc_bytes,
                                   void* stream);

/*
 * exl3_test_tile_plan: the cost model's plan for an exl3_gemm call (split = 0)
 * or exl3_gemm_splitk call (split = 1) of the given sizes, computed on the host
 * with no launch (the SM count of the current device, 152 when there is none).
 * out[0] = tile shape (numbered as in exl3_test_gemm_shape); for a pair shape
 * whose partial last wave runs as a second launch of smaller tiles (or of
 * 128-column pairs), out[1] =
 * that launch's shape, out[2] = pair tiles of the first launch, out[3] and
 * out[4] = first row and first column of the second launch; otherwise
 * out[1] = -1 and out[2..4] = 0.  EXL3_EINVAL for invalid sizes or shard map.
 * No counterpart in the pages: the tiling is this library's own.
 */
exl3_status_t exl3_test_tile_plan(int64_t m, int64_t k, int64_t n, const int32_t* shard_cols, int32_t num_shards,
                                  int32_t split, int64_t* out);

/*
 * Tile-shape autotune (off by default).  The best tile for a batch size
 * depends on the layer's shape too, so the shape is timed once per distinct
 * shape and cached, never while a CUDA graph is being captured, and the cost
 * model stays the fallback for captured work (cuda-exl3 README, "Where the
 * time goes").  Here the split-k parts are fixed by (k, n) so that rows stay
 * byte-equal across batch sizes; only the tile shape is tuned.
 * When enabled, the first uncaptured exl3_gemm / exl3_gemm_splitk call of each
 * key (device, width, codebook, k, n, shard edges, split parts, batch bucket:
 * m <= 32, else the next power of two of m) times every tile shape that can
 * run it on the caller's stream, synchronising the host, and caches the
 * fastest (the cost model's shape unless another is more than 2% faster).
 * The timing launches write the call's own y (or acc) several times; the
 * result is the final launch's, and every shape computes the same bytes, so
 * tuning never changes a result.  A call under capture uses the cached shape
 * of its key if there is one (tune in an eager warm-up to reach captured
 * work), else the cost model's, and never tunes.
 *   exl3_set_autotune(1 | 0): EXL3_EINVAL for any other value.
 *   exl3_clear_autotune(): forget every cached key.
 *   exl3_autotune_entries(): the number of cached keys.
 */
exl3_status_t exl3_set_autotune(int32_t enable);
exl3_status_t exl3_clear_autotune(void);
int64_t exl3_autotune_entries(void);

/*
 * exl3_device_status -- read and clear the library's device-side error flags.
 * Every wait inside the kernels is bounded; a kernel that gives up sets bit 0
 * (EXL3_DEVERR_WAIT_TIMEOUT) and skips its stores instead of hanging.  This call
 * synchronises the current device (it is meant for tests and diagnostics).
 *   flags: host pointer, receives the OR of all flags set since the last call.
 */
#define EXL3_DEVERR_WAIT_TIMEOUT 1u
exl3_status_t exl3_device_status(uint32_t* flags);

/*
 * exl3_test_wait_timeout -- test-only: the failure path of the bounded waits.
 * One CTA waits, with the same bounded mbarrier wait every kernel of the
 * library uses, on a barrier that nothing arrives on.  The wait gives up after
 * 2 s, the kernel sets EXL3_DEVERR_WAIT_TIMEOUT (read by exl3_device_status)
 * and writes *out = 0 (1 would mean the wait had returned).  It faults
 * nothing and leaves the context usable.  No counterpart in the pages.
 *   out: device uint32, 4-byte aligned; EXL3_EINVAL when null or misaligned.
 */
exl3_status_t exl3_test_wait_timeout(uint32_t* out, void* stream);

/* Static text for a status code. */
const char* exl3_status_string(exl3_status_t status);
/* Text of the last CUDA error seen by this thread's calls ("" if none). */
const char* exl3_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* EXL3_H */
