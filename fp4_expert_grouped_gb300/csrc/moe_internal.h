// moe_internal.h -- host-side declarations shared by the library's translation
// units (launchers of the kernels in kernels.cu and gemm.cu).  Not installed.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "fp4moe.h"

namespace fp4moe {

// SM count and device address of the status word of the current device
// (MOE_ERR_UNSUPPORTED_DEVICE unless it is an sm_103 part).
moe_status device_query(int *num_sms, unsigned **status);

// Tile sizes of the grouped GEMM (fixed for every batch size, so a token's
// result never depends on how many other tokens share its expert).
constexpr int kTileM = 128;   // pair rows (tokens) per tile = MMA M
constexpr int kTileN = 256;   // weight rows per tile = MMA N
constexpr int kTileK = 128;   // K per pipeline stage

// Tiled MXFP4 weight layout written by moe_pack_fp4 (see fp4moe.h): the
// matrix [N][K] of an expert is cut into 128 x 128 blocks, NB = N/128 rows of
// them.  The row blocks form pairs: with H = ceil(NB/2), row block n128 is
// half h = (n128 >= H) of pair j = n128 - h * H, i.e. pair j holds row blocks
// j and j + H (for W13 the gate and up rows of the same channels; for W2
// output rows [128 j, +128) and [128 (j + H), +128)).  At K block k128 the two
// blocks of pair j are neighbours:
//   b = e * NB * K/128 + (j * K/128 + k128) * 2 + h          (j < NB/2),
// so a GEMM tile fetches both with one TMA box and one scale copy.  When NB
// is odd, the last pair (j = NB/2) holds row block j alone, its K blocks
// consecutive after the others:
//   b = e * NB * K/128 + 2 * (NB/2) * K/128 + k128.
// Block b holds
//   codes:  8192 bytes at b * 8192, row r (0..127) at r * 64, two codes per
//           byte, low nibble = even k
//   scales: 512 bytes at b * 512, the UE8M0 byte of row r and 32-element
//           sub-block j (0..3) at (r % 32) * 16 + (r / 32) * 4 + j -- the
//           order the tensor-core scale-factor copy reads.
constexpr int kBlockCodeBytes = 128 * 64;
constexpr int kBlockScaleBytes = 512;
// pairs of row blocks (GEMM tiles of 256 weight rows) of an N-row matrix
__host__ __device__ inline int weight_pairs(int N) { return (N / 128 + 1) / 2; }
// whether pair j of an N-row matrix holds a single row block
__host__ __device__ inline bool weight_pair_single(int j, int N) { return (N / 128) % 2 == 1 && j == (N / 128) / 2; }
__host__ __device__ inline long long weight_block(long long e, int n128, int k128, int N, int K)
{
    const int NB = N / 128, KB = K / 128, H = (NB + 1) / 2;
    const int h = n128 >= H ? 1 : 0;
    const int j = n128 - h * H;
    const long long base = e * NB * KB;
    return j < NB / 2 ? base + ((long long)j * KB + k128) * 2 + h : base + 2LL * (NB / 2) * KB + k128;
}

// Block number of 128 x 128 block (rb, cb) of expert e's transposed FP8
// weights (moe_fp4_to_fp8t: R = K rows, C = N columns per expert, 16 KB per
// block, row r at r * 128).  Row blocks pair as (2j, 2j + 1): a pair's two
// blocks are neighbours at every column block, so the backward GEMM's 256-row
// operand of one K stage is 32 KB of contiguous memory; with R/128 odd the
// last row block is alone, its column blocks consecutive after the pairs'.
__host__ __device__ inline long long fp8t_block(int e, int rb, int cb, int R, int C)
{
    const int RB = R / 128, CB = C / 128, J = RB / 2;
    const long long base = (long long)e * RB * CB;
    const int j = rb >> 1;
    return j < J ? base + ((long long)j * CB + cb) * 2 + (rb & 1) : base + 2LL * J * CB + cb;
}

__host__ __device__ inline int sf_byte(int r, int j) { return (r % 32) * 16 + (r / 32) * 4 + j; }

// Activation scales of the GEMM operands (xq rows for GEMM1, hq rows for
// GEMM2) use the same 512-byte order per 128-row tile and per group of four
// 128-channel stages: byte j of row r in group g is the scale of stage 4g + j.
__host__ __device__ inline int stage_groups(int K) { return (K / 128 + 3) / 4; }

struct Shapes {
    int T, d, inter, E, k;
    long long P() const { return (long long)T * k; }
};

// Workspace layout (byte offsets, row strides).
struct Workspace {
    size_t off[32];
    size_t stride[32];
    size_t total;
};
bool workspace_layout(const Shapes &s, Workspace *ws);

// Row stride of the per-token scale array written by the top-k kernel
// (a multiple of 4 so one 32-bit word holds four consecutive groups).
inline int scale_row_stride(int channels) { return ((channels / 128) + 3) / 4 * 4; }

// upper bound on the number of 128-row tiles of the expert-ordered pairs
// Pair rows per GEMM row tile: 16 for batches averaging at most 8 pairs per
// expert, 32 up to 20, 64 up to 48, 128 otherwise.  At the top of each range
// about one expert in 200 (32-row tiles) or 75 (64-row tiles) holds more
// pairs than a tile and streams its weights twice.  A small batch's tiles
// hold a few rows each, and the shared memory a 128-row A slot takes is
// better spent on a deeper ring of weight stages (the GEMMs then stream
// weights at ~90% of HBM bandwidth instead of ~80%).  The MMA still computes
// 128 rows; rows past the tile's own are discarded, so a row's result does
// not depend on the tile size.
__host__ __device__ inline int gemm_tile_rows(long long P, int E)
{
    return P <= 8LL * E ? 16 : P <= 20LL * E ? 32 : P <= 48LL * E ? 64 : kTileM;
}

// Upper bound of the row tiles of all experts: every expert's last tile may
// be partial.
inline long long max_row_tiles(long long P, int E, int tile_rows)
{
    return (P + tile_rows - 1) / tile_rows + (P < E ? P : E);
}

// Launch with programmatic stream serialisation: the kernel may be scheduled
// while the previous grid in the stream finishes; every kernel of the library
// waits on the previous grid (griddepcontrol.wait) before reading or writing
// global memory, so this is safe after any predecessor.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// ---- launchers (kernels.cu) ----------------------------------------------
// rows = E * N; writes the tiled layout above (N % 128 == 0, K % 128 == 0)
cudaError_t launch_pack_fp4(const float *w, uint8_t *w_fp4, uint8_t *w_scale, int E, int N, int K, cudaStream_t st);
// FP8 weights for the backward pass, transposed (N % 128 == 0, K % 128 == 0):
// w8t [E][K][N] E4M3 codes, s8t [E][K/128][N/128] block exponents + 127
cudaError_t launch_fp4_to_fp8t(const uint8_t *w_fp4, const uint8_t *w_scale, uint8_t *w8t, uint8_t *s8t, int E, int N,
                               int K, cudaStream_t st);
cudaError_t launch_quantize(const uint16_t *x, uint8_t *xq, uint8_t *xs, int xs_stride, int T, int d,
                            cudaStream_t st);
cudaError_t launch_gate_logits(const uint16_t *x, const float *gate_w, const float *bias, float *z, int T, int d,
                               int E, cudaStream_t st);
// top-k + weights for every token; optionally quantises x in the same pass
// (xq/xs may be NULL).
cudaError_t launch_topk(const float *z, int32_t *topk_idx, float *topk_w, const uint16_t *x, uint8_t *xq,
                        uint8_t *xs, int xs_stride, int T, int d, int E, int k, unsigned *status, cudaStream_t st,
                        float *topk_z = nullptr);
// dispatch plan; tile_prefix may be NULL.  cta_counts: plan_scratch_bytes()
// of scratch for large P (NULL runs the plan as one CTA whatever P).
// With xs_tiles, also writes every pair's token scales (xs [T][xs_stride],
// d channels) into the GEMM's per-tile scale layout.
cudaError_t launch_plan(const int32_t *topk_idx, int32_t *expert_offsets, int32_t *sorted_pair, int32_t *pair_pos,
                        int32_t *tile_prefix, int *cta_counts, int T, int E, int k, unsigned *status, cudaStream_t st,
                        const uint8_t *xs = nullptr, int xs_stride = 0, uint8_t *xs_tiles = nullptr, int d = 0,
                        int tile_rows = kTileM, int *tile_done = nullptr, int n_tile_done = 0);
size_t plan_scratch_bytes(long long P, int E);
// With 128-row tiles, tiles holding more than kDenseTileRows pairs read their
// A rows from an expert-ordered copy (written by launch_dispatch_dense): one
// TMA box of kDenseBoxRows rows when they fit, else one 128-row box; the
// others gather them from xq, four rows per TMA gather, inside GEMM1.  An A
// stage costs about one TMA request's worth per box or gather whatever its
// bytes: four-row gathers suit a handful of rows, a single box the rest.
constexpr int kDenseTileRows = 16;
constexpr int kDenseBoxRows = 32;
// copy of xq row t into row pair_pos[t * k + j] of xq_sorted, for every pair
// whose position falls in a tile holding more than kDenseTileRows pairs
cudaError_t launch_dispatch_dense(const uint8_t *xq, const int32_t *pair_pos, const int32_t *topk_idx,
                                  const int32_t *expert_offsets, uint8_t *xq_sorted, int T, int d, int k,
                                  cudaStream_t st);
cudaError_t launch_combine(const uint16_t *y, const int32_t *pair_pos, const float *topk_w, uint16_t *out, int T,
                           int d, int k, cudaStream_t st);

// ---- tensor-core gate with certified routing (gate_tc.cu) -----------------
// Batches of at least kGateTcMinTokens tokens (E a multiple of 64, at most
// 256) compute approximate logits on the tensor cores and then the exact
// fixed-order logits of the candidate experts only; the routing is the same
// bits either way.
constexpr long long kGateTcMinTokens = 1024;
bool gate_uses_tc(long long T, int d, int E);
// c(d) of the bound |approx - fixed-order logit| <= c(d) ||x|| ||w_e|| + 2^-22 |approx|
float gate_bound_coefficient(int d);
struct GateScratch {
    float *wt;          // fp32 [E][d]: gate_w transposed
    uint16_t *whi;      // bf16 [E][d]: its high parts
    uint16_t *wlo;      // bf16 [E][d]: w - hi rounded to bf16
    float *wn;          // fp32 [E]: upper bounds of the experts' weight norms
    float *approx;      // fp32 [T][E]: tensor-core logits (+ bias)
    int32_t *ncand;     // int32 [T]: candidate experts per token (or NULL)
    bool prepared;      // wt, whi, wlo, wn already hold gate_w's (moe_prepare_gate)
};
// gate_w's transposed fp32 rows, bf16 split and weight norms into g
cudaError_t launch_gate_prep(const float *gate_w, const GateScratch &g, int d, int E, cudaStream_t st);
// where moe_prepare_gate puts them in its buffer
struct GatePrepLayout {
    size_t wt, whi, wlo, wn, total;
};
inline GatePrepLayout gate_prep_layout(int d, int E)
{
    auto up = [](size_t v) { return (v + 255) / 256 * 256; };
    GatePrepLayout l;
    l.wt = 0;
    l.whi = up((size_t)E * d * 4);
    l.wlo = l.whi + up((size_t)E * d * 2);
    l.wn = l.wlo + up((size_t)E * d * 2);
    l.total = l.wn + up((size_t)E * 4);
    return l;
}
// the tensor-core logits: gate_w split and transposed, the weight norms, then
// g.approx = x . (hi + lo) + bias
cudaError_t launch_gate_tc_logits(const uint16_t *x, const float *gate_w, const float *bias, const GateScratch &g,
                                  int T, int d, int E, int num_sms, unsigned *status, unsigned long long timeout_ns,
                                  cudaStream_t st);
// then the certified top-k (+ FP8 quantisation of x when xq is given);
// topk_z (or NULL): the selected experts' fixed-order logits
cudaError_t launch_gate_certify(const uint16_t *x, const float *bias, const GateScratch &g, int32_t *topk_idx,
                                float *topk_w, float *topk_z, uint8_t *xq, uint8_t *xs, int xs_stride, int T, int d,
                                int E, int k, unsigned *status, cudaStream_t st);

// ---- grouped GEMMs (gemm.cu) ---------------------------------------------
struct GemmArgs {
    // A: GEMM1 -- quantised tokens xq [T][K], gathered in the kernel by
    // sorted_pair (row = pair p -> token p / k); GEMM2 -- hq [P][K] rows in
    // expert order.  Scales per 128-row tile in the 512-byte order,
    // [tiles][stage_groups(K)][512].
    int tile_rows;                   // gemm_tile_rows(P, E): 16 or 128 pair rows per tile
    // per row tile: GEMM1 epilogue warps done with its hq rows and scales
    // (GEMM1 adds, GEMM2 waits for all of them; zeroed by the plan)
    int *tile_done;
    int *all_done;                   // the same arrivals summed over all row tiles
    const uint8_t *a;
    // GEMM1 only: expert-ordered copy of the A rows of the tiles holding more
    // than kDenseTileRows pairs ([P][K]; NULL: every tile gathers)
    const uint8_t *a_dense;
    const uint8_t *a_scale_tiles;
    const int32_t *sorted_pair;
    int k;
    long long a_rows;
    // B: tiled MXFP4 weights of all experts (codes + scales), N rows, K columns
    const uint8_t *b;
    const uint8_t *b_scale;
    int N;
    int K;
    // plan
    const int32_t *expert_offsets;   // [E+1]
    const int32_t *tile_prefix;      // [E+1]
    int E;
    long long P;
    // outputs: GEMM1 -> hq [P][inter] + hs tiles [tiles][stage_groups(inter)][512];
    // GEMM2 -> y bf16 [P][d]
    uint8_t *hq;
    uint8_t *hs_tiles;
    uint16_t *y;
    unsigned *status;
    unsigned long long timeout_ns;
    int num_sms;
    // GEMM2, tests only: wait for a GEMM1 count that never comes (before any
    // copy), so the bounded wait expires
    int stall_test;
    // GEMM1 (training): g and u of every pair, fp32 [P][2 inter] in expert
    // order (g at [p][c], u at [p][inter + c]); NULL = not kept
    float *gu_out;
    // MODE 3 (backward, dh = W2^T dy and the SwiGLU backward): the forward's
    // g, u (as gu_out), and the outputs [dg; du] as E4M3 codes [P][2 inter] +
    // scales [P][2 inter / 128], optionally also fp32 [P][2 inter]
    const float *gu_in;
    uint8_t *dgu;
    uint8_t *dgu_scale;
    float *dgu_f32;
};
cudaError_t launch_gemm1(const GemmArgs &a, int inter, cudaStream_t st);
cudaError_t launch_gemm2(const GemmArgs &a, int d, cudaStream_t st);
// dh = W2^T dy per pair on the FP8 weights (B = W2^T in moe_fp4_to_fp8t's
// 16 KB blocks, N = inter rows, K = d; scales as the block-exponent image in
// the tiled scale layout) with the SwiGLU backward fused
cudaError_t launch_gemm_dgrad_h(const GemmArgs &a, int inter, cudaStream_t st);
// dx of every pair = W13^T [dg; du] on the FP8 W13 (B = W13^T in 16 KB blocks,
// N = d rows, K = 2 inter), bf16 into y [P][d]
cudaError_t launch_gemm_dgrad_x(const GemmArgs &a, int d, cudaStream_t st);

} // namespace fp4moe
