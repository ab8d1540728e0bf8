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

struct Shapes {
    int T, d, inter, E, k;
    long long P() const { return (long long)T * k; }
};

// Workspace layout (byte offsets, row strides).
struct Workspace {
    size_t off[16];
    size_t stride[16];
    size_t total;
};
bool workspace_layout(const Shapes &s, Workspace *ws);

// Row strides of the per-row scale arrays used by the GEMM (multiple of 4 so a
// 4-byte word covers four consecutive 128-channel groups).
inline int scale_row_stride(int channels) { return ((channels / 128) + 3) / 4 * 4; }

// ---- launchers (kernels.cu) ----------------------------------------------
cudaError_t launch_pack_fp4(const float *w, uint8_t *w_fp4, uint8_t *w_scale, long long rows, int K,
                            cudaStream_t st);
cudaError_t launch_quantize(const uint16_t *x, uint8_t *xq, uint8_t *xs, int xs_stride, int T, int d,
                            cudaStream_t st);
cudaError_t launch_gate_logits(const uint16_t *x, const float *gate_w, const float *bias, float *z, int T, int d,
                               int E, cudaStream_t st);
// top-k + weights for every token; optionally quantises x in the same pass
// (xq/xs may be NULL).
cudaError_t launch_topk(const float *z, int32_t *topk_idx, float *topk_w, const uint16_t *x, uint8_t *xq,
                        uint8_t *xs, int xs_stride, int T, int d, int E, int k, unsigned *status, cudaStream_t st);
// dispatch plan; tile_prefix may be NULL.
cudaError_t launch_plan(const int32_t *topk_idx, int32_t *expert_offsets, int32_t *sorted_pair, int32_t *pair_pos,
                        int32_t *tile_prefix, int T, int E, int k, unsigned *status, cudaStream_t st);
// copy every pair's quantised token row into expert order
cudaError_t launch_dispatch(const uint8_t *xq, const uint8_t *xs, int xs_stride, const int32_t *sorted_pair,
                            uint8_t *xq_sorted, uint8_t *xs_sorted, long long P, int d, int k, cudaStream_t st);
cudaError_t launch_combine(const uint16_t *y, const int32_t *pair_pos, const float *topk_w, uint16_t *out, int T,
                           int d, int k, cudaStream_t st);

// ---- grouped GEMMs (gemm.cu) ---------------------------------------------
struct GemmArgs {
    // A: pair rows in expert order, E4M3 [P][K] with per-row scales [P][a_scale_stride]
    const uint8_t *a;
    const uint8_t *a_scale;
    int a_scale_stride;
    // B: packed weights of all experts [E][N][K/2] + UE8M0 scales [E][N][K/32]
    const uint8_t *b;
    const uint8_t *b_scale;
    int N;
    int K;
    // plan
    const int32_t *expert_offsets;   // [E+1]
    const int32_t *tile_prefix;      // [E+1]
    int E;
    long long P;
    // outputs: GEMM1 -> hq [P][inter] + hs [P][hs_stride]; GEMM2 -> y bf16 [P][d]
    uint8_t *hq;
    uint8_t *hs;
    int hs_stride;
    uint16_t *y;
    unsigned *status;
    unsigned long long timeout_ns;
    int num_sms;
};
cudaError_t launch_gemm1(const GemmArgs &a, int inter, cudaStream_t st);
cudaError_t launch_gemm2(const GemmArgs &a, int d, cudaStream_t st);
// upper bound on the number of tiles for the persistent grid size
inline long long max_row_tiles(long long P, int E)
{
    return (P + kTileM - 1) / kTileM + (P < E ? P : E);
}

} // namespace fp4moe
