/*
 * hc.h -- C ABI of the width-sharded ("halo-exchange") Conv2d for GB300.
 *
 * What it computes: the Shard(3) convolution of the NVIDIA technical blog
 * "Perception model training for autonomous vehicles with tensor
 * parallelism" (design section: input and output Shard(3) along W, weight and
 * bias Replicate; backward grad_input Shard(3), grad_weight / grad_bias
 * _Partial; Figures 1 and 2: halo exchange, concat, local conv, crop) and of
 * its Chinese write-up at kwkr.cn news/18980 (section 2.2: halo exchange,
 * concat, crop, and in backward zero-padding plus exchange of grad_output;
 * section 3.2: the exchange / local F.conv2d / crop override).  The W shards
 * are virtual: equal column blocks of one tensor in one GPU's memory.  A shard
 * reads its halo columns straight from its neighbours' blocks (zeros past the
 * image edge); the per-shard _Partial gradients are summed in a fixed order.
 *
 * Conventions for every call:
 *   - Tensors are fp32, NCHW, contiguous, in device memory, 16-byte aligned.
 *     Weights are [C_out][C_in/groups][kh][kw]; bias and grad_bias [C_out].
 *   - The caller owns every buffer, including the workspace.  The library
 *     allocates no device memory and does not synchronise, except in
 *     hc_sync_check.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  Calls are asynchronous on it.
 *   - Argument errors are returned before anything is launched.  A failed
 *     launch returns HC_ERR_CUDA.  A kernel that gives up waiting records
 *     HC_ERR_TIMEOUT in a device status word that hc_sync_check reports.
 *   - Results are deterministic: no floating-point atomics; every sum has a
 *     fixed order, so repeated calls give bit-identical outputs.
 */
#ifndef HC_H
#define HC_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    HC_OK = 0,
    HC_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misaligned pointer  */
    HC_ERR_UNSUPPORTED = 2,   /* valid convolution, but not a supported plan */
    HC_ERR_WORKSPACE = 3,     /* workspace missing or too small              */
    HC_ERR_CUDA = 4,          /* a CUDA call or launch failed                */
    HC_ERR_TIMEOUT = 5        /* a kernel gave up waiting (see hc_sync_check)*/
} hc_status;

/* The convolution (input, weight, bias, stride, padding, groups -- the
 * arguments of the _conv_forward override, kwkr.cn section 3.2) plus the
 * number of W shards and, optionally, of H shards.  Square stride and padding;
 * no dilation.
 *   num_shards    W blocks (Shard(3)), >= 1.
 *   num_shards_h  H blocks (Shard(2), kwkr.cn 5.2: the sharded dimension
 *                 switches to the height at very high resolution); 0 or 1 for
 *                 none.  With both, the shards form a row x column grid and
 *                 shard q = a * num_shards + b holds row block a and column
 *                 block b. */
typedef struct {
    int N, C_in, H, W, C_out, kh, kw, stride, padding, groups, num_shards;
    int num_shards_h;
} hc_conv_desc;

/* One shard of the plan: input columns [in_begin, in_end) (its Shard(3)
 * block), halo_left / halo_right columns read from the neighbouring blocks,
 * and the output columns [out_begin, out_end) it owns after the crop. */
typedef struct {
    int in_begin, in_end, halo_left, halo_right, out_begin, out_end;
} hc_shard_extent;

/* Kernel families; HC_ALGO_AUTO picks the fastest one that supports the desc. */
typedef enum {
    HC_ALGO_AUTO = 0,
    HC_ALGO_DIRECT = 1,       /* plain direct convolution, any groups / stride  */
    HC_ALGO_DEPTHWISE = 2,    /* groups == C, odd k, stride 1, padding (k-1)/2  */
    HC_ALGO_TC_3XTF32 = 3,    /* groups == 1: tcgen05 implicit GEMM; forward and
                                 grad_input on 3xTF32, the weight gradient (not
                                 space-to-depth) on three bf16 pieces per operand */
    HC_ALGO_TC_BF16X6 = 4     /* groups 1, padding 0, C_out a multiple of 128,
                                 W_out % 8 == 0, W / num_shards / stride a
                                 multiple of 32, and either
                                 1x1 / stride 1 with C_in a multiple of 128 and
                                 H*W a multiple of 128, or
                                 k = stride <= 4 (space-to-depth) with
                                 stride^2 * C_in a multiple of 8 and W_out a
                                 multiple of 128:
                                 tcgen05 GEMM on three bf16 pieces per operand
                                 (a = a0 + a1 + a2, six products a_i*b_j with
                                 i + j <= 2, fp32 accumulation), operands in
                                 NCHW order with no transposed copies           */
} hc_algo;

/* Shard(3) plan (NVIDIA blog, design section; kwkr.cn 2.1 and 2.2).
 * W is split into num_shards blocks of Wl = W / num_shards columns.  Shard r
 * owns input columns [r*Wl, (r+1)*Wl) and output columns
 * [r*Wl/stride, (r+1)*Wl/stride) (the last shard also takes output columns
 * past W/stride).  halo_left is the number of columns left of its block that
 * its owned outputs read (padding for the layouts here), halo_right the number
 * right of it (k - padding - stride when positive): for the pages' 5x5 /
 * padding 2 / stride 1 example, 2 and 2.
 *   ext   out: num_shards entries (caller-owned host memory).
 *   H_out, W_out  out (may be NULL): output size, (in + 2p - k) / s + 1.
 * Returns HC_ERR_INVALID_ARG for an invalid convolution, HC_ERR_UNSUPPORTED
 * when W % num_shards, Wl % stride or padding % stride is non-zero, or when a
 * halo is wider than Wl (a halo may only come from the adjacent shards). */
hc_status hc_shard_plan(const hc_conv_desc* d, hc_shard_extent* ext, int* H_out, int* W_out);

/* The row plan: the same rule on H with the kernel height (in_* / out_* are
 * rows, halo_left / halo_right the halo rows above / below the block).  With
 * num_shards_h <= 1 it is one extent of every row with no halo rows (no row
 * neighbours; the padding supplies the image edges).
 *   ext   out: max(1, num_shards_h) entries.
 * HC_ERR_UNSUPPORTED as for hc_shard_plan, on H. */
hc_status hc_shard_plan_rows(const hc_conv_desc* d, hc_shard_extent* ext);

/* Workspace bytes that hc_conv2d_fwd (pass 0), hc_conv2d_bwd (pass 1) or
 * hc_conv2d_bwd_reuse (pass 2) needs for this desc with HC_ALGO_AUTO (use
 * hc_conv2d_workspace_size_algo for a fixed algorithm).  Zero is a valid
 * answer; ws may then be NULL. */
hc_status hc_conv2d_workspace_size(const hc_conv_desc* d, int pass, size_t* bytes);
hc_status hc_conv2d_workspace_size_algo(const hc_conv_desc* d, int pass, hc_algo algo, size_t* bytes);

/* Which algorithm HC_ALGO_AUTO runs for this desc and pass. */
hc_status hc_conv2d_select(const hc_conv_desc* d, int pass, hc_algo* algo);

/* Forward (NVIDIA blog Figure 1; kwkr.cn 2.2 steps 1-3 and 3.2): per shard,
 * halo exchange + concat, local conv, crop to the owned output columns; the
 * shards' outputs together form y (Shard(3)).
 *   x    [N][C_in][H][W]           in
 *   w    [C_out][C_in/groups][kh][kw] in (Replicate)
 *   bias [C_out] or NULL           in
 *   y    [N][C_out][H_out][W_out]  out
 *   ws, ws_bytes: workspace of at least hc_conv2d_workspace_size(d, 0) bytes. */
hc_status hc_conv2d_fwd(const hc_conv_desc* d, const float* x, const float* w, const float* bias, float* y,
                        void* ws, size_t ws_bytes, void* stream);
hc_status hc_conv2d_fwd_algo(const hc_conv_desc* d, const float* x, const float* w, const float* bias, float* y,
                             void* ws, size_t ws_bytes, void* stream, hc_algo algo);

/* Backward (NVIDIA blog design section and Figure 2; kwkr.cn 2.2): per shard,
 * the grad_output block is extended by the halo of its neighbours' grad_output
 * (zeros past the image edge), grad_input of the owned input columns is the
 * local transposed conv, and the shard's _Partial grad_weight / grad_bias are
 * the local sums over its own output columns.  The partials are then summed
 * over shards in shard order (the pages' cross-device reduce-sum).
 *   x, w, gy   in ([N][C_out][H_out][W_out] for gy)
 *   gx         out [N][C_in][H][W], or NULL to skip
 *   gw         out [C_out][C_in/groups][kh][kw], or NULL to skip
 *   gb         out [C_out], or NULL to skip
 *   gw_partials out [Q][C_out][C_in/groups][kh][kw], or NULL
 *   gb_partials out [Q][C_out], or NULL
 *     Q = num_shards * max(1, num_shards_h), shard q = a * num_shards + b owning
 *     output rows of row block a and columns of column block b; the full
 *     gradients are the sums over q in increasing order.
 *   ws, ws_bytes: workspace of at least hc_conv2d_workspace_size(d, 1) bytes. */
hc_status hc_conv2d_bwd(const hc_conv_desc* d, const float* x, const float* w, const float* gy, float* gx, float* gw,
                        float* gb, float* gw_partials, float* gb_partials, void* ws, size_t ws_bytes, void* stream);
hc_status hc_conv2d_bwd_algo(const hc_conv_desc* d, const float* x, const float* w, const float* gy, float* gx,
                             float* gw, float* gb, float* gw_partials, float* gb_partials, void* ws, size_t ws_bytes,
                             void* stream, hc_algo algo);

/* Backward pass that reuses the forward pass's operand copy of x instead of
 * rebuilding it (the way a training step keeps forward state for its
 * backward pass).  With HC_ALGO_TC_BF16X6 the forward workspace begins with
 * the bf16 pieces of x (or of its space-to-depth image), which the weight
 * gradient reads; the other algorithms keep nothing between the passes, and
 * for them the call is hc_conv2d_bwd_algo (fwd_ws is not read).
 *   fwd_ws, fwd_ws_bytes: the workspace of the last hc_conv2d_fwd(_algo) call
 *     with this desc, this x and the same algorithm, not written since; at
 *     least hc_conv2d_workspace_size(d, 0) bytes, 256-byte aligned
 *     (HC_ERR_INVALID_ARG if NULL or misaligned, HC_ERR_WORKSPACE if too
 *     small, for HC_ALGO_TC_BF16X6).
 *   ws, ws_bytes: at least hc_conv2d_workspace_size(d, 2) bytes.
 * Every other argument as for hc_conv2d_bwd; the results are bit-identical to
 * hc_conv2d_bwd's. */
hc_status hc_conv2d_bwd_reuse(const hc_conv_desc* d, const float* x, const float* w, const float* gy, float* gx,
                              float* gw, float* gb, float* gw_partials, float* gb_partials, void* ws,
                              size_t ws_bytes, const void* fwd_ws, size_t fwd_ws_bytes, void* stream, hc_algo algo);

/* Backward pass of a convolution on the branch of a residual block (the
 * ConvNeXt-XL blocks the pages train, NVIDIA blog design section: out = x +
 * branch(x)): grad_input also receives the gradient that reaches x along the
 * skip connection.
 *   residual: that gradient, same shape and layout as x (device, 16-byte
 *     aligned); it must not overlap gx (HC_ERR_INVALID_ARG if NULL,
 *     misaligned or equal to gx).
 *   gx: required (not NULL); receives grad_input + residual.
 * The depthwise family adds the residual in its grad_input epilogue (one more
 * read, no extra pass over gx); the other families run their backward pass and
 * then add it (hc_add_inplace).  Every other argument, the workspace and the
 * errors as for hc_conv2d_bwd_algo; gw, gb and the partials are unchanged. */
hc_status hc_conv2d_bwd_residual(const hc_conv_desc* d, const float* x, const float* w, const float* gy,
                                 const float* residual, float* gx, float* gw, float* gb, float* gw_partials,
                                 float* gb_partials, void* ws, size_t ws_bytes, void* stream, hc_algo algo);

/* A GELU (exact form, hc_gelu_fwd) next to a convolution, folded into the
 * passes that read the tensor it touches -- the MLP pattern 1x1 -> GELU -> 1x1
 * of a ConvNeXt block, with h the first conv's output:
 *   second conv:  hc_conv2d_fwd_act(..., x = h, HC_ACT_GELU_INPUT) and
 *                 hc_conv2d_bwd_act(..., HC_ACT_GELU_INPUT), whose grad_input is
 *                 the gradient with respect to GELU(h);
 *   first conv:   hc_conv2d_fwd (its output is h) and hc_conv2d_bwd_act(...,
 *                 gy = that gradient, HC_ACT_GELU_OUTPUT, y_pre = h), which runs on
 *                 gy * GELU'(h), the gradient with respect to h.
 * GELU(h) and the separate GELU backward pass are never materialised. */
typedef enum {
    HC_ACT_NONE = 0,
    HC_ACT_GELU_INPUT = 1,  /* the conv's input is GELU(x) */
    HC_ACT_GELU_OUTPUT = 2  /* the conv's output y feeds GELU(y) */
} hc_act;

/* Forward pass with a GELU: HC_ACT_GELU_INPUT gives y = conv(GELU(x)) + bias,
 * GELU(x) going straight into the operand pieces as x is read;
 * HC_ACT_GELU_OUTPUT and HC_ACT_NONE give the plain conv (the output is the
 * pre-activation).  GELU needs HC_ALGO_TC_BF16X6 (or HC_ALGO_AUTO picking it)
 * and a 1x1 stride-1 conv, else HC_ERR_UNSUPPORTED.  Arguments and workspace as
 * for hc_conv2d_fwd. */
hc_status hc_conv2d_fwd_act(const hc_conv_desc* d, const float* x, const float* w, const float* bias, float* y,
                            void* ws, size_t ws_bytes, void* stream, hc_algo algo, hc_act act);

/* Backward pass with a GELU:
 *   HC_ACT_GELU_INPUT: the backward of hc_conv2d_fwd_act(HC_ACT_GELU_INPUT): gw,
 *     gb of the conv on GELU(x); gx = the gradient with respect to the conv's
 *     input GELU(x) (GELU'(x) is left to the consumer: the first conv's
 *     HC_ACT_GELU_OUTPUT backward, or hc_gelu_bwd).  y_pre is not read.
 *   HC_ACT_GELU_OUTPUT: gy is the gradient with respect to GELU(y_pre), y_pre
 *     ([N][C_out][H_out][W_out]) the conv's output; the pass runs on
 *     gy * GELU'(y_pre), formed as gy is read, and gx, gw, gb, partials are the
 *     conv's gradients for it (HC_ERR_INVALID_ARG if y_pre is NULL).
 * fwd_ws: the workspace of this conv's forward call (hc_conv2d_fwd_act with the
 * same desc, x and act, or hc_conv2d_fwd for HC_ACT_GELU_OUTPUT), read as by
 * hc_conv2d_bwd_reuse (ws then needs pass-2 bytes), or NULL (pass-1 bytes).
 * Same support rule as hc_conv2d_fwd_act. */
hc_status hc_conv2d_bwd_act(const hc_conv_desc* d, const float* x, const float* w, const float* gy, float* gx,
                            float* gw, float* gb, float* gw_partials, float* gb_partials, void* ws, size_t ws_bytes,
                            const void* fwd_ws, size_t fwd_ws_bytes, void* stream, hc_algo algo, hc_act act,
                            const float* y_pre);

/* Halo exchange + concat made explicit (kwkr.cn 2.2 steps 1-2): for every
 * shard q of the row x column grid, x_ext[q] is its block of x with the halo
 * rows above / below (hc_shard_plan_rows) and halo columns left / right
 * (hc_shard_plan) around it, zeros past the image edge.  x_ext is
 * [Q][N][C_in][He][We], Q = num_shards * max(1, num_shards_h),
 * We = max over column shards of halo_left + Wl + halo_right and He the same
 * over row shards (H when there is one row shard); a shard with narrower halos
 * leaves its unused trailing rows / columns zero.  A pure copy (bit-exact). */
hc_status hc_halo_gather(const hc_conv_desc* d, const float* x, float* x_ext, void* stream);

/* ---- One rank of a multi-device Shard(3) layout ----------------------------
 * The pages' design puts each column block on its own device, which receives
 * its halo columns from the neighbouring devices (NVIDIA blog, design section
 * and Figure 1; kwkr.cn 2.2: halo exchange, concat, local conv, crop) and may
 * compute the region away from the block edges while the halo is in flight
 * (kwkr.cn 5.2).  A rank keeps its block of Wl = W / num_shards columns in the
 * halo-padded layout x_pad [N][C][H][Wl + 2 * HC_HALO_COLS]: its own columns at
 * [HC_HALO_COLS, HC_HALO_COLS + Wl), the HC_HALO_COLS columns left of them
 * holding the left neighbour's last columns and those right of them the right
 * neighbour's first columns (zeros past the image edge), so the pages' concat
 * is the layout itself.  A halo exchange moves HC_HALO_COLS columns each way:
 * hc_halo_pack on the sender, the caller's transport (NCCL send / recv, a peer
 * copy), hc_halo_unpack on the receiver.  Every call takes the GLOBAL desc d
 * (W the full width, num_shards the number of ranks); the work is one block's.
 * Tensors: fp32, device memory, 16-byte aligned; x_pad rows are Wl + 8 floats. */
#define HC_HALO_COLS 4

/* Column tiles of one rank's block that a call computes (128-column tiles,
 * T = Wl / 128 of them). */
typedef enum {
    HC_TILES_ALL = 0,       /* every tile                                          */
    HC_TILES_INTERIOR = 1,  /* tiles 1 .. T-2: they read no halo column            */
    HC_TILES_EDGE = 2       /* tiles 0 and T-1: they read the halo columns         */
} hc_tiles;

/* x_pad's own columns from the rank's block x_local [N][C][H][Wl]; both margins
 * zeroed.  HC_ERR_INVALID_ARG for null or misaligned pointers or Wl % 4 != 0. */
hc_status hc_halo_pad(const hc_conv_desc* d, const float* x_local, float* x_pad, void* stream);

/* The HC_HALO_COLS edge columns of x_pad's own block that a neighbour needs,
 * packed as buf [N*C*H][HC_HALO_COLS]: side 0 the first ones (the left
 * neighbour's right margin), side 1 the last ones (the right neighbour's left
 * margin).  A pure copy. */
hc_status hc_halo_pack(const hc_conv_desc* d, const float* x_pad, int side, float* buf, void* stream);

/* A packed halo (hc_halo_pack of the neighbour) into x_pad's margin: side 0
 * the left margin, side 1 the right one; buf NULL writes zeros (the image
 * edge).  A pure copy. */
hc_status hc_halo_unpack(const hc_conv_desc* d, const float* buf, int side, float* x_pad, void* stream);

/* Forward of one rank: y [N][C][H][Wl], its block's output columns, from x_pad
 * whose margins hold the exchanged halo.  tiles selects the column tiles: an
 * HC_TILES_INTERIOR call reads only the block's own columns, so it may run
 * while the halo is in flight, and an HC_TILES_EDGE call after it completes
 * the output (bit-identical to one HC_TILES_ALL call).  Depthwise
 * convolutions (groups = C_in = C_out, K in {3, 5, 7}, stride 1, padding
 * (K-1)/2 <= HC_HALO_COLS) with Wl a multiple of 128 and no row shards;
 * HC_ERR_UNSUPPORTED otherwise. */
hc_status hc_conv2d_fwd_rank(const hc_conv_desc* d, const float* x_pad, const float* w, const float* bias, float* y,
                             hc_tiles tiles, void* stream);

/* Workspace bytes of hc_conv2d_bwd_rank (the per-tile weight-gradient partials). */
hc_status hc_conv2d_workspace_size_rank(const hc_conv_desc* d, size_t* bytes);

/* Backward of one rank (the pages' backward on one device): gy_pad is
 * grad_output in the halo-padded layout, its margins exchanged like x's (the
 * zero-pad + exchange of grad_output, kwkr.cn 2.2).  Outputs (each nullable):
 * gx [N][C][H][Wl] the block's grad_input; gw_part [C][1][K][K] and gb_part
 * [C] this rank's _Partial grad_weight / grad_bias, which summed over the
 * ranks in rank order (hc_sum_partials) give the full gradients.  An
 * HC_TILES_INTERIOR call followed by an HC_TILES_EDGE call on the same
 * workspace computes what one HC_TILES_ALL call does (grad_input
 * bit-identical; the weight gradient's tile sums may split differently across
 * blocks, within rounding); the call covering the edge tiles (ALL or EDGE) also
 * reduces the partials.  Same support as hc_conv2d_fwd_rank. */
hc_status hc_conv2d_bwd_rank(const hc_conv_desc* d, const float* x_pad, const float* w, const float* gy_pad,
                             float* gx, float* gw_part, float* gb_part, void* ws, size_t ws_bytes, hc_tiles tiles,
                             void* stream);

/* out[k] = sum_{r < count} parts[r * n + k] with r ascending: the ranks'
 * gathered _Partial gradients summed in rank order, the deterministic form of
 * the pages' all-reduce (NVIDIA blog, design section). */
hc_status hc_sum_partials(const float* parts, int count, long long n, float* out, void* stream);

/* Depthwise backward that allocates nothing.  The pages have no counterpart:
 * this entry point exists for callers that may not allocate device memory at
 * the point of the call -- for example code running under another framework's
 * memory allocator that forbids raw cudaMalloc, or a latency-critical loop that
 * must not allocate after start-up (cudaMalloc can block and synchronise the
 * device) -- and so cannot provide the workspace hc_conv2d_bwd takes.
 *
 * It computes exactly what hc_conv2d_bwd_algo(..., HC_ALGO_DEPTHWISE) computes
 * (same kernels, same arguments minus the workspace), but keeps its scratch
 * (the per-tile and per-shard partial weight / bias gradients) in a 16 MiB
 * statically sized device array that lives in the library: every GPU that
 * loads the library holds those 16 MiB until the process exits.  The caller
 * still passes all inputs and outputs.
 *   - Sizes whose scratch would exceed 16 MiB are rejected with
 *     HC_ERR_WORKSPACE before anything is launched; so are descs the depthwise
 *     kernels do not cover (HC_ERR_UNSUPPORTED).
 *   - A call looks up the current device's address of the array (with that
 *     device current) unless its stream is being captured; a call into a
 *     capturing stream reuses the address of the device's last lookup, so make
 *     one call on the device before any stream capture (a capture with no
 *     earlier call returns HC_ERR_UNSUPPORTED).
 *   - All calls share the one array and it keeps the last call's contents;
 *     every scratch value a call reads is written earlier in the same call, so
 *     nothing needs clearing, but calls that overlap on the GPU (different
 *     streams, or different host threads) race on it and must be serialised
 *     by the caller. */
hc_status hc_conv2d_bwd_depthwise_noalloc(const hc_conv_desc* d, const float* x, const float* w, const float* gy,
                                          float* gx, float* gw, float* gb, float* gw_partials, float* gb_partials,
                                          void* stream);

/* ---- ConvNeXt block pointwise ops (channels first, shard-local: no halo) ----
 * The pages train ConvNeXt-XL (NVIDIA blog, design section), whose blocks put
 * a LayerNorm over channels, a GELU and a layer scale + residual around the
 * depthwise and 1x1 convolutions.  Tensors are [N][C][HW] fp32 (NCHW with H*W
 * flattened), device memory, 16-byte aligned; gamma / beta are [C].  Parameter
 * gradients are per-block partial sums added in a fixed order (the workspace
 * holds the partials).  Invalid sizes or pointers: HC_ERR_INVALID_ARG. */

/* Workspace bytes for hc_layernorm_c_bwd and hc_layerscale_residual_bwd. */
hc_status hc_pointwise_workspace_size(int N, int C, long long HW, size_t* bytes);

/* LayerNorm over C at every (n, position): mean, biased variance,
 * y = (x - mean) / sqrt(var + eps) * gamma[c] + beta[c].  mean / rstd
 * ([N][HW], may be NULL) keep the statistics for the backward pass. */
hc_status hc_layernorm_c_fwd(int N, int C, long long HW, const float* x, const float* gamma, const float* beta,
                             float eps, float* y, float* mean, float* rstd, void* stream);

/* LayerNorm backward: with xhat = (x - mean) * rstd and g = gy * gamma,
 * gx = rstd * (g - mean_c(g) - xhat * mean_c(g * xhat));
 * ggamma[c] = sum gy * xhat, gbeta[c] = sum gy over n and positions (either
 * may be NULL; then ws may be NULL too). */
hc_status hc_layernorm_c_bwd(int N, int C, long long HW, const float* x, const float* gamma, const float* mean,
                             const float* rstd, const float* gy, float* gx, float* ggamma, float* gbeta, void* ws,
                             size_t ws_bytes, void* stream);

/* GELU, exact form y = x * (1 + erf(x / sqrt 2)) / 2, over n elements. */
hc_status hc_gelu_fwd(long long n, const float* x, float* y, void* stream);

/* GELU backward: gx = gy * (Phi(x) + x * exp(-x^2 / 2) / sqrt(2 pi)). */
hc_status hc_gelu_bwd(long long n, const float* x, const float* gy, float* gx, void* stream);

/* y += x over n elements: joins the residual's gradient (the block output's
 * gradient itself) with the gradient that comes back through the branch. */
hc_status hc_add_inplace(long long n, float* y, const float* x, void* stream);

/* Layer scale and residual: out = res + gamma[c] * branch. */
hc_status hc_layerscale_residual_fwd(int N, int C, long long HW, const float* res, const float* branch,
                                     const float* gamma, float* out, void* stream);

/* Backward: gbranch = gamma[c] * gy (NULL to skip), ggamma[c] = sum branch * gy;
 * the residual's gradient is gy itself. */
hc_status hc_layerscale_residual_bwd(int N, int C, long long HW, const float* branch, const float* gamma,
                                     const float* gy, float* gbranch, float* ggamma, void* ws, size_t ws_bytes,
                                     void* stream);

/* DropPath (stochastic depth) keep mask with a shard-consistent draw (NVIDIA
 * blog design section: ConvNeXt-XL's DropPath Bernoulli draw must agree across
 * devices; kwkr.cn 3.1 and 6.1: a distributed DropPath layer keeps the RNG
 * consistent, every DropPath layer uses the same seed).
 *   mask[n] = 1 / (1 - drop_prob) if sample n keeps its branch, else 0,
 * for n in [0, N).  The draw for sample n is output number offset + n of a
 * SplitMix64 generator seeded with `seed` (Steele, Lea, Flood 2014), kept iff
 * its top 24 bits are >= floor(drop_prob * 2^24): it depends on (seed, offset,
 * n) only, so any shard or device holding sample n -- or a slice of the batch
 * called with offset + its first sample -- draws the same value.
 *   mask  out [N] device fp32.  drop_prob in [0, 1), else HC_ERR_INVALID_ARG. */
hc_status hc_drop_path_mask(int N, float drop_prob, unsigned long long seed, unsigned long long offset, float* mask,
                            void* stream);
/* hc_layerscale_residual_fwd / _bwd with a per-sample DropPath mask (from
 * hc_drop_path_mask; NULL = keep all): out = res + mask[n] * gamma[c] * branch;
 * backward gbranch = mask[n] * gamma[c] * gy, ggamma[c] = sum mask[n] * branch * gy. */
hc_status hc_layerscale_droppath_fwd(int N, int C, long long HW, const float* res, const float* branch,
                                     const float* gamma, const float* mask, float* out, void* stream);
hc_status hc_layerscale_droppath_bwd(int N, int C, long long HW, const float* branch, const float* gamma,
                                     const float* mask, const float* gy, float* gbranch, float* ggamma, void* ws,
                                     size_t ws_bytes, void* stream);

/* One training step of a convolution -- hc_conv2d_fwd then, when ws_fwd and
 * ws_bwd do not overlap, hc_conv2d_bwd_reuse (reading x's operand copy from
 * ws_fwd; ws_bwd needs hc_conv2d_workspace_size(d, 2) bytes), else
 * hc_conv2d_bwd (pass-1 bytes), with the automatic algorithm and every
 * argument as in those calls; either way the results equal hc_conv2d_fwd +
 * hc_conv2d_bwd -- captured into a
 * CUDA graph that replays with one launch (LibreYOLO documentation, page "Grafy
 * CUDA": a graph records a fixed kernel sequence and the addresses it uses;
 * replay must match eager execution bit for bit, which it does here since every
 * kernel is deterministic).  For small problems the step costs its launch
 * latency; the graph removes most of it.  The graph is bound to the pointers
 * given here: replays read the inputs' current contents and overwrite the
 * outputs.  gx, gw, gb may be NULL as in hc_conv2d_bwd (no partial outputs).
 * Capture runs on a private stream and launches nothing.  *out receives a handle
 * owned by the caller (hc_step_graph_destroy); on any error *out is NULL and the
 * status is the failing call's. */
typedef struct hc_step_graph_s* hc_step_graph;
hc_status hc_conv2d_step_graph_create(const hc_conv_desc* d, const float* x, const float* w, const float* bias,
                                      float* y, const float* gy, float* gx, float* gw, float* gb, void* ws_fwd,
                                      size_t ws_fwd_bytes, void* ws_bwd, size_t ws_bwd_bytes, hc_step_graph* out);
/* Replays the step on `stream` (asynchronous; HC_ERR_CUDA if the launch fails). */
hc_status hc_step_graph_launch(hc_step_graph g, void* stream);
/* Releases the graph (NULL is a no-op). */
hc_status hc_step_graph_destroy(hc_step_graph g);

/* Synchronises `stream`, then returns (and clears) the first error a kernel
 * recorded in the device status word, HC_ERR_CUDA for an asynchronous CUDA
 * error, or HC_OK. */
hc_status hc_sync_check(void* stream);

/* Self-test of failure detection.  Launches one kernel that waits on an
 * mbarrier nothing ever arrives on; after wait_us microseconds (1 .. 2e6) of
 * the GPU's global timer it gives up, records HC_ERR_TIMEOUT in the device
 * status word -- the same path every pipelined kernel of the library takes
 * when a wait runs out -- and returns, leaving the context usable.  The next
 * hc_sync_check on `stream` then returns HC_ERR_TIMEOUT (and clears it).
 * Returns HC_ERR_INVALID_ARG for an out-of-range wait_us. */
hc_status hc_selftest_timeout(int wait_us, void* stream);

/* Static English text for a status code. */
const char* hc_status_string(hc_status s);

/* Number of kernels this library has launched since it was loaded. */
unsigned long long hc_launch_count(void);

/* Reproducibility hook (the pages have no counterpart): the number of SMs the
 * library sizes its persistent grids and split counts for; 0 (the default)
 * uses the device's.  Results are bit-identical from call to call for a fixed
 * count; another count partitions the fixed-order sums differently and may
 * round differently, within the stated tolerances -- this hook lets a test see
 * both on one GPU.  Process-wide; set it before querying workspace sizes (the
 * tensor-core weight-gradient split count, hence its workspace, depends on
 * it).  HC_ERR_INVALID_ARG for a negative count. */
hc_status hc_set_sm_count(int sms);

/* Per-kernel device timing (a measurement aid; the pages have no counterpart).
 * hc_trace_enable(1): from then on every launcher records a CUDA event on its
 * stream before its first kernel and one after every kernel, so each kernel's
 * device time is the interval between the event before it and its own on the
 * same stream.  Launches into a stream that is being captured are not traced.
 * hc_trace_enable(0) stops recording.  While off, the cost is one atomic load
 * per launch; while on, one event record per launch.
 * hc_trace_collect: waits for the recorded events, adds the intervals up per
 * kernel name into out[0 .. *n_entries) (caller-owned host memory; names that
 * do not fit in max_entries are dropped) and clears the record.  Returns
 * HC_ERR_CUDA if an event could not be read (its interval is left out). */
typedef struct {
    char name[48];
    int launches;
    double total_ms;
} hc_trace_entry;
hc_status hc_trace_enable(int on);
hc_status hc_trace_collect(hc_trace_entry* out, int max_entries, int* n_entries);

#ifdef __cplusplus
}
#endif

#endif /* HC_H */
