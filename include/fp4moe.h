/*
 * fp4moe.h -- C ABI of libfp4moe.so: the forward pass of an MoE layer with
 * FP4 (E2M1) expert weights on one NVIDIA GB300 (sm_103a).
 *
 * The layer ("DeepSeek-V4揭秘：细粒度专家并行隐藏通信时延，FP4量化与TileLang协同优化百万Token上下文",
 * itsolotime.com/archives/32374, section 1.1: four stages -- dispatch,
 * linear-1, linear-2, combine) is, for every token t:
 *   z      = x_t . gate_w  (+ bias)                  fp32, fixed order (below)
 *   S      = top-k experts by z                       ties -> lower expert index
 *   w_j    = sqrt(softplus(z_j)) / sum_j sqrt(softplus(z_j))
 *            (gate activation of "DeepSeek V4架构学习笔记", 67808.cn/a/484462.html,
 *            DeepSeekMoE paragraph; renormalised to sum 1)
 *   xq     = FP8 E4M3 of x_t, one power-of-two scale per 128 channels
 *            (FP8 dispatch, section 1.4 of the first page)
 *   h_e    = silu(xq W13_e[gate]^T) * (xq W13_e[up]^T)    -> FP8, scale per 128
 *   y_e    = bf16(h_e W2_e^T)                          (BF16 combine payload)
 *   out_t  = bf16( sum_j w_j * y_{e_j} )   fp32 fused multiply-adds in slot order
 * with expert weights stored as MXFP4: E2M1 codes plus one UE8M0 power-of-two
 * scale per 32 elements along K (section 4, "FP4 量化感知训练", of the first
 * page; the FP4 -> FP8 step is exact, so the contraction runs on FP8 tensor
 * cores with the 1x32 scales applied by the block-scaled MMA).
 *
 * Conventions for every function:
 *  - Pointers marked "device" are caller-owned device memory; the library
 *    never frees them and keeps no pointer after the call returns.
 *  - All work is enqueued on `stream` (a cudaStream_t passed as void*; NULL =
 *    legacy default stream).  No function synchronises the stream except
 *    moe_get_device_status.
 *  - Every argument is checked on the host before anything is launched; on an
 *    argument error the outputs are left untouched and nothing is enqueued.
 *  - Return value: MOE_OK or an error code; nothing throws across the ABI.
 *    Asynchronous device errors surface as MOE_ERR_CUDA from a later call, or
 *    through moe_get_device_status.
 *  - Shapes: T >= 0 (T == 0 is a no-op that returns MOE_OK), d % 128 == 0,
 *    inter % 128 == 0, 1 <= k <= 8, k <= E <= 256, T * k < 2^31
 *    (moe_backward_h: d % 256 == 0, inter % 256 == 0).
 *  - Alignment: every device pointer 16-byte aligned; packed weights 32-byte
 *    aligned (the tensor-memory-access rule for packed 4-bit data).
 *  - Results are deterministic: repeated calls give identical bits, and a
 *    token's output bits do not depend on the other tokens in the batch.
 */
#ifndef FP4MOE_H
#define FP4MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum moe_status {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,        /* NULL or misaligned pointer, negative size */
    MOE_ERR_UNSUPPORTED_SHAPE = 2,  /* shape outside the supported set above */
    MOE_ERR_CUDA = 3,               /* a CUDA runtime call failed */
    MOE_ERR_WORKSPACE = 4,          /* workspace allocation failed or too small */
    MOE_ERR_TIMEOUT = 5,            /* a kernel gave up waiting on a barrier */
    MOE_ERR_UNSUPPORTED_DEVICE = 6, /* the current device is not sm_103 */
    MOE_ERR_DEVICE_FAULT = 7        /* a kernel flagged bad data (e.g. expert id out of range) */
} moe_status;

/* Human-readable name of a status code (static string, never NULL). */
const char *moe_status_string(moe_status s);

/* Library version as 10000*major + 100*minor + patch. */
int moe_version(void);

/*
 * moe_pack_fp4 -- MXFP4 weight quantisation (first page, section 4) into the
 * tiled layout moe_forward reads.
 *   w        device, fp32 [E][N][K] row-major (K contiguous)
 *   rule     per 32 consecutive K-elements: X = floor(log2(max |w|)) - 2
 *            (X = -127 for an all-zero block), clamped to [-127, 127]; codes
 *            are the round-to-nearest-even E2M1 of w * 2^-X saturated to +-6,
 *            the scale is the UE8M0 byte X + 127.
 *   layout   each expert's [N][K] matrix is cut into 128 x 128 blocks, NB = N/128
 *            rows and KB = K/128 columns of them.  With H = ceil(NB/2), row
 *            block n/128 is half h = (n/128 >= H) of pair j = n/128 - h * H; at
 *            K block k/128 the two blocks of pair j are adjacent:
 *              b = e * NB * KB + (j * KB + k/128) * 2 + h        (j < NB/2)
 *            (for W13 the gate and up rows of the same channels).  When NB is
 *            odd the last row block (j = NB/2) stands alone, its K blocks
 *            consecutive: b = e * NB * KB + 2 * (NB/2) * KB + k/128.  Then:
 *   w_fp4    device, E*N*K/2 bytes: block b at b * 8192, its row n % 128 at
 *            (n % 128) * 64, two codes per byte, the low nibble holding the
 *            even k (so one block is 8 KB of contiguous memory)
 *   w_scale  device, E*N*K/32 bytes: block b at b * 512, the scale of row
 *            r = n % 128 and 32-element sub-block j = (k % 128) / 32 at byte
 *            (r % 32) * 16 + (r / 32) * 4 + j (the order the tensor cores'
 *            scale-factor copy reads, so the forward loads it with one copy)
 * For the layer: W13 is [E][2*inter][d] (rows 0..inter-1 = gate projection,
 * inter..2*inter-1 = up projection), W2 is [E][d][inter].
 * Requires N % 128 == 0, K % 128 == 0.  Load-time operation, off the hot path.
 */
moe_status moe_pack_fp4(const float *w, uint8_t *w_fp4, uint8_t *w_scale,
                        int E, int N, int K, void *stream);

/*
 * moe_fp4_to_fp8t -- FP8 weights for the backward pass of FP4 quantisation-
 * aware training (first page, section 4: the FP4 weights are dequantised to
 * FP8 for compute, losslessly while the 1x32 sub-block scales inside each
 * 128x128 FP8 block stay within a ratio; gradients use these FP8 weights, and
 * 128x128 blocks transpose without re-quantisation).  For every 128x128 block
 * of W[e] ([N][K]): block exponent B = (largest 1x32 exponent X of the block)
 * - 6, clamped to >= -127; each element is E4M3(code * 2^(X - B)) rounded to
 * nearest even -- exactly the FP4 value over 2^B when X - B >= -8, i.e. when
 * the block's sub-block scales span at most 2^14.
 *   w_fp4, w_scale  device, moe_pack_fp4 output (tiled layout) of W [E][N][K]
 *   w8t             device, E*K*N bytes, 16-byte aligned: the transposed
 *                   matrix W[e]^T ([K][N]) in 128 x 128 blocks of 16 KB, the
 *                   E4M3 code of W[e][n][k] at byte (k % 128) * 128 + n % 128
 *                   of block fp8t(e, k/128, n/128); row blocks pair as
 *                   (2j, 2j+1) with RB = K/128, CB = N/128, J = RB/2:
 *                     fp8t(e, rb, cb) = e*RB*CB + ((rb/2)*CB + cb)*2 + rb%2
 *                   for rb < 2J, and e*RB*CB + 2*J*CB + cb for an odd last
 *                   row block (so the backward GEMM reads 256 rows of one
 *                   K stage as 32 KB of contiguous memory)
 *   s8t             device, E*(K/128)*(N/128) bytes: B + 127 of block (bn, bk)
 *                   at (e * K/128 + bk) * N/128 + bn
 * Requires N % 128 == 0, K % 128 == 0.  Argument errors are reported before
 * any launch; the outputs are written on the stream.  Load-time operation
 * (once per weight update), off the forward's hot path.
 */
moe_status moe_fp4_to_fp8t(const uint8_t *w_fp4, const uint8_t *w_scale, uint8_t *w8t, uint8_t *s8t,
                           int E, int N, int K, void *stream);

/*
 * moe_quantize_act -- FP8 E4M3 activation quantisation (first page, section 1.4,
 * "FP8 dispatch").  One power-of-two scale per token per 128 channels:
 * e = the smallest integer with max|x| <= 448 * 2^e (e = 0 for an all-zero
 * group), clamped to [-127, 127]; xq = round-to-nearest-even E4M3 of x * 2^-e.
 *   x   device, bf16 bit patterns [T][d]
 *   xq  device, uint8 E4M3 codes [T][d]
 *   xs  device, uint8 [T][d/128], byte e + 127
 * This is the quantisation the forward pass applies to x (same kernel).
 */
moe_status moe_quantize_act(const uint16_t *x, uint8_t *xq, uint8_t *xs,
                            int T, int d, void *stream);

/*
 * moe_route -- gate and top-k ("DeepSeek V4架构学习笔记", DeepSeekMoE paragraph).
 *   x          device, bf16 [T][d]
 *   gate_w     device, fp32 [d][E]
 *   gate_bias  device, fp32 [E] added to the logits, or NULL
 *   topk_idx   device, int32 [T][k]: slot j holds the j-th largest logit's
 *              expert (logits descending, ties to the lower expert index)
 *   topk_w     device, fp32 [T][k]: w_j = s_j / sum_j s_j (fp32 sum in slot
 *              order), s_j = fp32(sqrt(softplus(z_j))) evaluated in double;
 *              w_j = 1/k if the sum is 0
 * Logits use a fixed fp32 order so routing is exactly reproducible: for each
 * (t, e), 32 partial sums over channels i = l, l+32, ... accumulated with fused
 * multiply-adds in increasing i, then added as a binary tree with offsets
 * 16, 8, 4, 2, 1 (partial[l] += partial[l + off]); the bias is added last.
 * Inputs must be finite.  Allocates stream-ordered scratch: T*E*4 bytes, plus
 * E*d*8 + E*4 + T*4 bytes from MOE_GATE_TC_MIN_TOKENS tokens on (the
 * tensor-core gate below, which gives the same routing bits).
 */
moe_status moe_route(const uint16_t *x, const float *gate_w, const float *gate_bias,
                     int32_t *topk_idx, float *topk_w, int T, int d, int E, int k, void *stream);

/*
 * moe_route_noalloc -- moe_route for callers that cannot allocate device
 * memory at call time (a serving loop whose allocator already owns all free
 * device memory, a latency-critical loop that forbids allocator calls after
 * start-up, a host program that does not let libraries call cudaMalloc).
 * Same arguments, results and checks as moe_route; the pages describe
 * nothing of the kind (it exists only for such callers).
 * Its T*E fp32 logits live in a fixed 4 MiB array of device memory that
 * every device loading the library holds until the process exits; the call
 * allocates nothing.  Limit: T * E <= 1048576 (e.g. 4096 tokens with 256
 * experts); larger shapes return MOE_ERR_WORKSPACE without launching.
 * The first call on a device looks up that array's device address (once per
 * device, with the device current); make that first call before any stream
 * capture.  Where the CUDA driver loads a library's device code lazily (its
 * default), that first call is also when the driver loads the code holding
 * the array and so reserves its 4 MiB: make it at start-up, with the other
 * allocations; every later call allocates nothing.  All calls share the
 * array: calls that overlap on the GPU (e.g. on two streams at once) race and
 * must be serialised by the caller.
 */
moe_status moe_route_noalloc(const uint16_t *x, const float *gate_w, const float *gate_bias,
                             int32_t *topk_idx, float *topk_w, int T, int d, int E, int k, void *stream);

/*
 * moe_dispatch_plan -- expert-contiguous layout of the P = T*k token-expert
 * pairs (first page, section 1.1 "dispatch"; section 3.2: a fixed token order
 * keeps results deterministic).  Pair p = t*k + j.
 *   topk_idx        device, int32 [T][k], values in [0, E)
 *   expert_offsets  device, int32 [E+1]: start of expert e's group; [E] = P
 *   sorted_pair     device, int32 [P]: pairs by ascending expert, ascending p
 *                   within an expert (a stable counting sort)
 *   pair_pos        device, int32 [P]: inverse of sorted_pair
 * An out-of-range expert index sets MOE_ERR_DEVICE_FAULT in the device status
 * word (see moe_get_device_status) and the outputs are then unspecified.
 */
moe_status moe_dispatch_plan(const int32_t *topk_idx, int32_t *expert_offsets,
                             int32_t *sorted_pair, int32_t *pair_pos,
                             int T, int E, int k, void *stream);

/*
 * moe_forward -- the whole layer: gate + top-k, FP8 quantisation of x,
 * dispatch plan, grouped GEMM1 (W13; each tile gathers its tokens' FP8 rows,
 * the dispatch; fused SwiGLU and FP8 re-quantisation of
 * h with one power-of-two scale per 128 channels), grouped GEMM2 (W2, output
 * rounded to bf16) and the combine out_t = bf16(fp32 fused multiply-add chain
 * over slots j = 0..k-1 of w_j * y_j).
 *   x                  device, bf16 [T][d]
 *   gate_w             device, fp32 [d][E]
 *   w13_fp4, w13_scale device, moe_pack_fp4 output (tiled) for W13 [E][2*inter][d]
 *   w2_fp4,  w2_scale  device, moe_pack_fp4 output (tiled) for W2 [E][d][inter]
 *   out                device, bf16 [T][d]
 * Workspace (moe_workspace_size bytes) is allocated stream-ordered on `stream`
 * and released on it before return.
 */
moe_status moe_forward(const uint16_t *x, const float *gate_w,
                       const uint8_t *w13_fp4, const uint8_t *w13_scale,
                       const uint8_t *w2_fp4, const uint8_t *w2_scale,
                       uint16_t *out, int T, int d, int inter, int E, int k, void *stream);

/* Options of moe_forward_ex.  Zero-initialise and set what is needed. */
typedef struct moe_forward_opts {
    const float *gate_bias;    /* device fp32 [E] added to the logits, or NULL */
    void *workspace;           /* device, >= moe_workspace_size bytes, 256-byte
                                  aligned; NULL = allocate on the stream */
    size_t workspace_bytes;
    int32_t *topk_idx_out;     /* optional device copies of the routing: [T][k] */
    float *topk_w_out;         /* [T][k] */
    int32_t *pair_pos_out;     /* [T*k] position of pair t*k+j in expert order */
    uint32_t flags;            /* 0, or MOE_FLAG_TEST_STALL_GEMM2 (tests only) */
    void **stage_events;       /* optional: MOE_STAGE_COUNT + 1 caller-created
                                  cudaEvent_t, recorded on the stream before the
                                  first stage, between stages and after the last
                                  (per-stage timing); NULL = none */
    float *gu_out;             /* optional (training): device fp32 [T*k][2*inter], 32-byte
                                  aligned: g and u of every pair in expert order (row
                                  workspace pair position, g at [p][c], u at [p][inter + c]),
                                  the tensor-core fp32 sums GEMM1 applies SwiGLU to; the
                                  input moe_backward_h needs.  NULL = not kept */
    const void *gate_prep;     /* optional: moe_prepare_gate's buffer for this gate_w
                                  (256-byte aligned).  From MOE_GATE_TC_MIN_TOKENS
                                  tokens the forward then reads gate_w's split and
                                  norms from it instead of computing them per call;
                                  the results are the same bits.  NULL = compute */
} moe_forward_opts;

/*
 * moe_prepare_gate -- gate_w's form for the tensor-core gate (large batches),
 * computed once per gate_w like moe_pack_fp4's packed experts: gate_w
 * transposed (fp32 [E][d]), split into bf16 high and low parts ([E][d] each),
 * and an upper bound of each expert's weight norm (fp32 [E]).  Pass the buffer
 * as moe_forward_opts.gate_prep; prepare again after changing gate_w.
 *   gate_w  device fp32 [d][E], 16-byte aligned
 *   prep    device, moe_gate_prep_size(d, E) bytes, 256-byte aligned
 * Requires d % 128 == 0, 1 <= E <= 256.  Load-time operation.
 */
size_t moe_gate_prep_size(int d, int E);
moe_status moe_prepare_gate(const float *gate_w, void *prep, int d, int E, void *stream);

/* Test only (failure detection without a GPU fault): GEMM2 waits for a
 * GEMM1 completion count that is never published, before it issues any copy.
 * Its bounded wait (FP4MOE_TIMEOUT_MS, default 2000 ms) runs out, every CTA
 * leaves through its exit path, and moe_get_device_status then reports
 * MOE_ERR_TIMEOUT.  The output of that call is not computed; the next call
 * runs normally. */
#define MOE_FLAG_TEST_STALL_GEMM2 0x1u

/* Stages of moe_forward_ex, in launch order (index into stage_events). */
enum {
    MOE_STAGE_GATE = 0,   /* fixed-order fp32 gate logits */
    MOE_STAGE_TOPK,       /* top-k, weights and FP8 quantisation of x */
    MOE_STAGE_PLAN,       /* dispatch plan (stable counting sort) + scale tiles */
    MOE_STAGE_DISPATCH,   /* copy of the FP8 token rows of densely filled tiles into expert order */
    MOE_STAGE_GEMM1,      /* grouped W13 GEMM (gathers the rows of sparse tiles) + SwiGLU + FP8 */
    MOE_STAGE_GEMM2,      /* grouped W2 GEMM, bf16 output */
    MOE_STAGE_COMBINE,    /* slot-order weighted combine */
    MOE_STAGE_COUNT
};

/* moe_forward with options (gate bias, caller workspace, routing outputs).
 * With a caller workspace the call allocates nothing and can be captured in a
 * CUDA graph. */
moe_status moe_forward_ex(const uint16_t *x, const float *gate_w,
                          const uint8_t *w13_fp4, const uint8_t *w13_scale,
                          const uint8_t *w2_fp4, const uint8_t *w2_scale,
                          uint16_t *out, int T, int d, int inter, int E, int k,
                          void *stream, const moe_forward_opts *opts);

/*
 * moe_backward_h -- the first GEMM of the layer's backward pass in FP4
 * quantisation-aware training, with the SwiGLU backward fused (first page,
 * section 4: the backward computes with the FP8 weights the FP4 weights
 * dequantise to -- moe_fp4_to_fp8t -- and transposed 128 x 128 blocks are not
 * re-quantised; section 3.2: fixed summation order, no atomics).  For every
 * token-expert pair p = t*k + j routed to expert e, in the forward's expert
 * order (pair position pos = pair_pos[p]):
 *   dy     = topk_w[t][j] * dout[t]                       fp32
 *   dyq    = E4M3 of dy, one power-of-two scale per 128 channels (the rule of
 *            moe_quantize_act)
 *   dh     = W2[e]^T dyq                                  block-scaled FP8 MMA, fp32
 *   dg     = dh * u * s * (1 + g * (1 - s)),  du = dh * g * s,  s = 1 / (1 + e^-g)
 *            (g, u: the forward's, from moe_forward_opts.gu_out)
 *   [dg; du] -> E4M3 codes with one power-of-two scale per 128 channels
 *   dout           device, bf16 [T][d]: the gradient at the layer output
 *   w2_fp8t        device, moe_fp4_to_fp8t output for W2 ([E][d][inter]): E4M3
 *                  codes of W2^T ([E][inter][d]) in that function's 16 KB
 *                  blocks, 16-byte aligned
 *   w2_s8t         device, its block exponents [E][inter/128][d/128]
 *   gu             device, fp32 [T*k][2*inter] (moe_forward_opts.gu_out)
 *   fwd_workspace  device, the workspace of the forward call that produced gu
 *                  (its routing and dispatch-plan regions are read)
 *   workspace      device scratch of moe_backward_h_workspace_size bytes,
 *                  256-byte aligned, or NULL (then allocated stream-ordered)
 *   dgu            device, E4M3 codes [T*k][2*inter] in expert order, 32-byte aligned:
 *                  dg at [pos][c], du at [pos][inter + c]
 *   dgu_scale      device, [T*k][2*inter/128]: byte e + 127 of each 128 channels
 *   dgu_f32        device, fp32 [T*k][2*inter] (the unquantised dg, du), or NULL
 * Requires d % 256 == 0 and inter % 256 == 0, 1 <= k <= 8, k <= E <= 256.
 * Argument errors are reported before anything is enqueued.
 */
size_t moe_backward_h_workspace_size(int T, int d, int inter, int E, int k);
moe_status moe_backward_h(const uint16_t *dout, const uint8_t *w2_fp8t, const uint8_t *w2_s8t, const float *gu,
                          const void *fwd_workspace, void *workspace, size_t workspace_bytes, uint8_t *dgu,
                          uint8_t *dgu_scale, float *dgu_f32, int T, int d, int inter, int E, int k, void *stream);

/*
 * moe_backward_x -- the second GEMM of the layer's backward pass (the same
 * passages as moe_backward_h): the gradient at the layer input through the
 * experts.  For every pair p = t*k + j routed to expert e, at its expert-order
 * position pos:
 *   dx_p   = W13[e]^T [dg; du]_p                          block-scaled FP8 MMA, fp32,
 *                                                         rounded to bf16 (like y)
 *   dx[t]  = bf16( sum over j = 0..k-1, in slot order, of dx_{t*k+j} )   fp32 sum
 * (the routing weights' own gradient is not part of dx: routing is held fixed).
 *   dgu, dgu_scale  device, moe_backward_h's outputs (E4M3 [T*k][2*inter] in
 *                   expert order, 16-byte aligned, and [T*k][2*inter/128])
 *   w13_fp8t        device, moe_fp4_to_fp8t output for W13 ([E][2*inter][d]):
 *                   E4M3 codes of W13^T ([E][d][2*inter]) in 16 KB blocks,
 *                   16-byte aligned
 *   w13_s8t         device, its block exponents [E][d/128][2*inter/128]
 *   fwd_workspace   device, the workspace of the forward call (routing and
 *                   dispatch plan)
 *   workspace       device scratch of moe_backward_x_workspace_size bytes,
 *                   256-byte aligned, or NULL (then allocated stream-ordered)
 *   dx              device, bf16 [T][d], 16-byte aligned
 * Requires d % 256 == 0 and inter % 256 == 0, 1 <= k <= 8, k <= E <= 256.
 * Argument errors are reported before anything is enqueued.
 */
/*
 * moe_backward_w -- the master weights' gradients (first page, section 4: the
 * gradient passes straight through the FP4 quantisation to the FP32 master
 * weights; section 3.2: fixed summation order).  For every expert e, over its
 * pairs p in the forward's expert order (ascending pair id: token order, then
 * slot order), with every operand its E4M3 code times its power-of-two scale:
 *   dW2[e]  = sum_p dy_p (x) h_p          fp32 [E][d][inter]
 *   dW13[e] = sum_p [dg; du]_p (x) x_p    fp32 [E][2*inter][d]
 * (dy_p as moe_backward_h quantised it, h_p and x_p as the forward's GEMMs read
 * them, [dg; du]_p as moe_backward_h wrote it).  The operands are dequantised to
 * bf16 (exact for E4M3 times a power of two within bf16's range) and the sums
 * run on the bf16 tensor cores in fp32, in pair order.  Experts without pairs
 * get zero gradients.
 *   fwd_workspace     device, the forward call's workspace (plan, xq, hq and scales)
 *   bwd_h_workspace   device, the workspace moe_backward_h was given (its dy
 *                     codes and scales are read; moe_backward_h must have been
 *                     called with a caller workspace, not NULL)
 *   dgu, dgu_scale    device, moe_backward_h's outputs, dgu 16-byte aligned
 *   dW13, dW2         device, fp32 outputs, 32-byte aligned
 *   workspace         device scratch of moe_backward_w_workspace_size bytes,
 *                     256-byte aligned, or NULL (then allocated stream-ordered)
 * Requires d % 256 == 0 and inter % 256 == 0, 1 <= k <= 8, k <= E <= 256.
 * Argument errors are reported before anything is enqueued.
 */
size_t moe_backward_w_workspace_size(int T, int d, int inter, int E, int k);
moe_status moe_backward_w(const void *fwd_workspace, const void *bwd_h_workspace, const uint8_t *dgu,
                          const uint8_t *dgu_scale, float *dW13, float *dW2, void *workspace, size_t workspace_bytes,
                          int T, int d, int inter, int E, int k, void *stream);

/*
 * moe_backward_dw -- the gradient with respect to the routing weights (the
 * backward of the weighted combine, first page section 1.4): for every pair
 * p = t*k + j, dw[p] = sum over c of dout[t][c] * y_p[c], y_p the pair's bf16
 * expert output that the forward kept in its workspace (fp32 sum, lane-strided
 * partial sums and a fixed tree; deterministic).  Routing is held fixed: the
 * gate's own backward is the caller's.
 *   dout           device, bf16 [T][d], 16-byte aligned
 *   fwd_workspace  device, the forward call's workspace (y and the plan are read)
 *   dw             device, fp32 [T][k]
 * Requires the forward's shapes.  Argument errors are reported before
 * anything is enqueued.
 */
moe_status moe_backward_dw(const uint16_t *dout, const void *fwd_workspace, float *dw, int T, int d, int inter, int E,
                           int k, void *stream);

size_t moe_backward_x_workspace_size(int T, int d, int inter, int E, int k);
moe_status moe_backward_x(const uint8_t *dgu, const uint8_t *dgu_scale, const uint8_t *w13_fp8t,
                          const uint8_t *w13_s8t, const void *fwd_workspace, void *workspace, size_t workspace_bytes,
                          uint16_t *dx, int T, int d, int inter, int E, int k, void *stream);

/* Bytes of workspace moe_forward_ex needs for these shapes (0 for bad shapes). */
size_t moe_workspace_size(int T, int d, int inter, int E, int k);

/* Workspace regions, for inspecting intermediates in tests and tools.
 * moe_workspace_layout writes the byte offset of each region into
 * offsets[MOE_WS_COUNT] and its row stride in bytes into strides[MOE_WS_COUNT]
 * (either may be NULL) and returns the total size (0 for bad shapes). */
enum {
    MOE_WS_XQ = 0,        /* uint8 E4M3 [T][d] */
    MOE_WS_XS,            /* uint8 [T][stride], first d/128 bytes of a row used */
    MOE_WS_LOGITS,        /* fp32 [T][E]: below MOE_GATE_TC_MIN_TOKENS tokens (or E not a
                             multiple of 64) the fixed-order logits; from there on the
                             tensor-core approximations a, each within
                             c(d) ||x_t|| ||w_e|| + 2^-22 |a| + d 2^-125 of the
                             fixed-order logit (the gate path below) */
    MOE_WS_TOPK_IDX,      /* int32 [T][k] */
    MOE_WS_TOPK_W,        /* fp32 [T][k] */
    MOE_WS_EXPERT_OFFSETS,/* int32 [E+1] */
    MOE_WS_SORTED_PAIR,   /* int32 [P] */
    MOE_WS_PAIR_POS,      /* int32 [P] */
    MOE_WS_TILE_PREFIX,   /* int32 [E+1] running count of the GEMMs' row tiles of R pairs each:
                             R = 16 when T*k <= 8*E, 32 when <= 20*E, 64 when <= 48*E, else 128 */
    MOE_WS_HQ,            /* uint8 E4M3 [P][inter], rows in expert order */
    MOE_WS_HS_TILES,      /* uint8 scales of hq per row tile m (R rows, as above) and
                             group g of four 128-channel groups: 512-byte blocks
                             at (m * ceil(inter/512) + g) * 512, the byte of row r
                             and group 4g + j at (r % 32) * 16 + (r / 32) * 4 + j */
    MOE_WS_Y,             /* bf16 [P][d], rows in expert order */
    MOE_WS_XQ_SORTED,     /* uint8 E4M3 [P][d]: row p = xq of the pair's token, expert order;
                             written only when T*k >= 16*E, for the rows of tiles holding
                             more than 16 pairs (the others are gathered from xq inside
                             GEMM1) */
    MOE_WS_XS_TILES,      /* scales of the expert-ordered pair rows (their tokens' xs), laid
                             out like MOE_WS_HS_TILES with d */
    MOE_WS_PLAN_COUNTS,   /* int32 per-chunk expert counts of the dispatch plan (large batches) */
    MOE_WS_TILE_DONE,     /* int32 per GEMM row tile: GEMM1 epilogue warps that have stored
                             the tile's hq rows and scales (GEMM2 starts a row tile once all
                             of them have), then one int32 total over all tiles */
    MOE_WS_TOPK_Z,        /* fp32 [T][k]: the fixed-order logits of the selected experts */
    /* the tensor-core gate's scratch (empty below MOE_GATE_TC_MIN_TOKENS tokens): */
    MOE_WS_GATE_WT,       /* fp32 [E][d]: gate_w transposed */
    MOE_WS_GATE_WHI,      /* bf16 [E][d]: its high parts (round to nearest even) */
    MOE_WS_GATE_WLO,      /* bf16 [E][d]: w - hi, rounded to bf16 */
    MOE_WS_GATE_WNORM,    /* fp32 [E]: upper bounds of ||w_e||_2 */
    MOE_WS_GATE_NCAND,    /* int32 [T]: experts whose logit was computed in the fixed
                             order (the candidates of the certified top-k) */
    MOE_WS_COUNT
};

/* Gate path.  From this many tokens on (with E a multiple of 64, at most
 * 256), the logits are first approximated on the tensor cores: gate_w is
 * split into bf16 parts hi + lo (|w - hi - lo| <= 2^-16 |w|) and
 * a = x . (hi + lo) + bias is accumulated in fp32, restarting every 128
 * channels.  Each a_e lies within D_e = c(d) ||x_t|| ||w_e|| + 2^-22 |a_e| +
 * d 2^-125 of the fixed-order logit z_e (c(d) = 1.026 (2^-16 + 17 * 2^-17 +
 * (5 d/128 + 5) 2^-24): the split, 16 MMAs per chunk at 2^-17 each, the chunk
 * sums, the fixed order's own rounding; the last term, products flushed below
 * the normal range).  Every expert of the exact top-k has
 * a_e + D_e >= L, the k-th largest a_e - D_e; for those candidates alone the
 * fixed-order logit is computed, and the top-k, its slot order and the
 * weights come from those.  The routing is therefore bit-identical to the
 * CUDA-core path's for every token, whatever the batch. */
#define MOE_GATE_TC_MIN_TOKENS 1024
size_t moe_workspace_layout(int T, int d, int inter, int E, int k,
                            size_t *offsets, size_t *strides);

/* Synchronises `stream`, then reads and clears the library's device status
 * word: MOE_OK, MOE_ERR_TIMEOUT (a kernel gave up on a bounded wait) or
 * MOE_ERR_DEVICE_FAULT (a kernel found bad data); MOE_ERR_CUDA if the
 * synchronisation itself failed. */
moe_status moe_get_device_status(void *stream);

#ifdef __cplusplus
}
#endif

#endif /* FP4MOE_H */
