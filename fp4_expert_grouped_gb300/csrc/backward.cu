// backward.cu -- the first GEMM of the MoE layer's backward pass in FP4
// quantisation-aware training, and its C ABI entry (moe_backward_h).
//
// "DeepSeek-V4揭秘：细粒度专家并行隐藏通信时延，FP4量化与TileLang协同优化百万Token上下文"
// (itsolotime.com/archives/32374), section 4: the backward computes with the
// FP8 weights the FP4 weights dequantise to (moe_fp4_to_fp8t), transposed
// 128 x 128 blocks without re-quantisation.  Per token-expert pair p (token t,
// slot j, expert e), in the forward's expert order:
//   dy_p       = w_tj dout_t                      (the gradient at y_p)
//   dyq_p      = E4M3 of dy_p, one power-of-two scale per 128 channels
//   dh_p       = W2[e]^T dyq_p                    (FP8 x FP8 block-scaled MMA)
//   dg, du     = the SwiGLU backward with the forward's g, u
//   [dg; du]   = E4M3, one power-of-two scale per 128 channels
// Section 3.2 (determinism): no atomics, every sum in a fixed order.
#include "moe_device.cuh"
#include "moe_internal.h"

#include <cstring>

namespace fp4moe {

// The weights' block exponents as the tensor cores' scale-factor image: for
// expert e, 256-row block nb of W^T ([R][C]: W2^T with R = inter, C = d, or
// W13^T with R = d, C = 2 inter) and K block ks, two 512-byte blocks (rows
// 0-127 and 128-255) at ((e * R/256 + nb) * C/128 + ks) * 2 + h, every byte of
// block h the exponent of 128 x 128 block (2 nb + h, ks) -- the tiled scale
// layout of moe_pack_fp4 with N = R, K = C, all four 1 x 32 scales of a row
// equal.  One thread per 16 bytes.
__global__ void __launch_bounds__(256) bwd_scale_image_kernel(const uint8_t *__restrict__ s8t, uint8_t *__restrict__ img,
                                                              long long n16, int R, int C)
{
    pdl_wait();
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n16) {
        const long long b = i / 32;                       // 512-byte block
        const int h = (int)(b & 1);
        const long long q = b >> 1;
        const int KB = C / 128, J = R / 256;
        const int ks = (int)(q % KB);
        const long long ej = q / KB;
        const int nb = (int)(ej % J);
        const long long e = ej / J;
        // s8t as moe_fp4_to_fp8t writes it: [E][R/128][C/128]
        const uint32_t v = s8t[(e * (R / 128) + 2 * nb + h) * KB + ks];
        const uint32_t w = v * 0x01010101u;
        reinterpret_cast<uint4 *>(img)[i] = make_uint4(w, w, w, w);
    }
    pdl_trigger();
}

// dy of every pair, quantised into expert order: one warp per token.  The
// token's dout row is read once (a warp per pair position re-read it k times,
// scattered, mostly from DRAM) and each of its k pairs gets dy = w_tj * dout_t
// in fp32, then E4M3 with one power-of-two scale per 128 channels (the
// activations' rule), written at the pair's expert-order position; the scale
// bytes go to the GEMM's per-tile scale layout (row tiles of R pairs, as the
// forward's plan numbers them).
__global__ void __launch_bounds__(256) bwd_dy_kernel(const uint16_t *__restrict__ dout, const float *__restrict__ topk_w,
                                                     const int32_t *__restrict__ topk_idx,
                                                     const int32_t *__restrict__ pair_pos,
                                                     const int32_t *__restrict__ expert_offsets,
                                                     const int32_t *__restrict__ tile_prefix, uint8_t *__restrict__ dyq,
                                                     uint8_t *__restrict__ dys_tiles, int T, int d, int k, int R)
{
    pdl_wait();
    const int t = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    if (t >= T) return;
    const int lane = threadIdx.x & 31;
    const int G4 = stage_groups(d);
    float w[8];
    uint8_t *qrow[8];
    uint8_t *srow[8];                                // the pair's scale byte of group 0
#pragma unroll
    for (int j = 0; j < 8; j++) {
        w[j] = 0.f;
        qrow[j] = nullptr;
        srow[j] = nullptr;
        if (j < k) {
            const int p = t * k + j;
            const int pos = pair_pos[p];
            const int e = topk_idx[p];
            w[j] = topk_w[p];
            const int local = pos - expert_offsets[e];
            const long long m = tile_prefix[e] + local / R;
            qrow[j] = dyq + (size_t)pos * d;
            srow[j] = dys_tiles + (size_t)m * G4 * kBlockScaleBytes + sf_byte(local % R, 0);
        }
    }
    const uint4 *src = reinterpret_cast<const uint4 *>(dout + (size_t)t * d);
    const int n8 = d / 8;
    for (int c = lane; c - lane < n8; c += 32) {
        uint4 cur = make_uint4(0, 0, 0, 0);
        if (c < n8) cur = __ldg(src + c);
        const uint32_t u[4] = {cur.x, cur.y, cur.z, cur.w};
        float x[8];
#pragma unroll
        for (int i = 0; i < 4; i++) {
            x[2 * i] = bf16_bits_to_f32(u[i] & 0xFFFFu);
            x[2 * i + 1] = bf16_bits_to_f32(u[i] >> 16);
        }
        const int grp = c / 16;                          // 128-channel group = K stage of the GEMM
#pragma unroll
        for (int j = 0; j < 8; j++) {
            if (j >= k) break;
            float v[8];
#pragma unroll
            for (int i = 0; i < 8; i++) v[i] = w[j] * x[i];
            float amax = 0.f;
#pragma unroll
            for (int i = 0; i < 8; i++) amax = fmaxf(amax, fabsf(v[i]));
#pragma unroll
            for (int off = 8; off >= 1; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
            if (c < n8) {
                const int ex = e4m3_scale_exp(amax);
                const float sc = exp2i(-ex);
                uint2 q;
                q.x = cvt_e4m3x2(v[0] * sc, v[1] * sc) | (cvt_e4m3x2(v[2] * sc, v[3] * sc) << 16);
                q.y = cvt_e4m3x2(v[4] * sc, v[5] * sc) | (cvt_e4m3x2(v[6] * sc, v[7] * sc) << 16);
                reinterpret_cast<uint2 *>(qrow[j])[c] = q;
                if ((lane & 15) == 0)
                    srow[j][(size_t)(grp / 4) * kBlockScaleBytes + grp % 4] = (uint8_t)(ex + 127);
            }
        }
    }
    pdl_trigger();
}

// [dg; du]'s scales, row-major [P][G] (G = 2 inter / 128) as moe_backward_h
// writes them, into the GEMM's per-tile scale layout: row r of row tile m,
// 128-channel group grp at (m * stage_groups(2 inter) + grp / 4) * 512 +
// sf_byte(r, grp % 4).  One thread per byte.
__global__ void __launch_bounds__(256) bwd_sf_tiles_kernel(const uint8_t *__restrict__ scale,
                                                           const int32_t *__restrict__ topk_idx,
                                                           const int32_t *__restrict__ sorted_pair,
                                                           const int32_t *__restrict__ expert_offsets,
                                                           const int32_t *__restrict__ tile_prefix,
                                                           uint8_t *__restrict__ tiles, long long P, int G, int k, int R)
{
    pdl_wait();
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < P * G) {
        const long long pos = i / G;
        const int grp = (int)(i % G);
        const int e = topk_idx[sorted_pair[pos]];
        const int local = (int)(pos - expert_offsets[e]);
        const long long m = tile_prefix[e] + local / R;
        const int r = local % R;
        tiles[(m * stage_groups(G * 128) + grp / 4) * kBlockScaleBytes + sf_byte(r, grp % 4)] = scale[i];
    }
    pdl_trigger();
}

// dw[t][j] = dout[t] . y[pair_pos[t k + j]] (the routing weight's gradient;
// y is the forward's bf16 expert output, kept in its workspace): one warp per
// pair, lane l summing channels 8 l .. 8 l + 7 of every 256 in fp32 (each
// product of two bf16 values exact), then the xor tree.
__global__ void __launch_bounds__(256) bwd_dw_kernel(const uint16_t *__restrict__ dout, const uint16_t *__restrict__ y,
                                                     const int32_t *__restrict__ pair_pos, float *__restrict__ dw,
                                                     long long P, int d, int k)
{
    pdl_wait();
    const long long p = (long long)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    if (p >= P) return;
    const int lane = threadIdx.x & 31;
    const uint4 *a = reinterpret_cast<const uint4 *>(dout + (size_t)(p / k) * d);
    const uint4 *b = reinterpret_cast<const uint4 *>(y + (size_t)__ldg(pair_pos + p) * d);
    float acc = 0.f;
    for (int c = lane; c < d / 8; c += 32) {
        const uint4 u = __ldg(a + c), v = __ldg(b + c);
        const uint32_t uu[4] = {u.x, u.y, u.z, u.w}, vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; i++) {
            acc = fmaf(bf16_bits_to_f32(uu[i] & 0xFFFFu), bf16_bits_to_f32(vv[i] & 0xFFFFu), acc);
            acc = fmaf(bf16_bits_to_f32(uu[i] >> 16), bf16_bits_to_f32(vv[i] >> 16), acc);
        }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) acc = acc + __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) dw[p] = acc;
    pdl_trigger();
}

namespace {

bool aligned_to(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
size_t round_up256(size_t v) { return (v + 255) / 256 * 256; }

bool bwd_shape_ok(int T, int d, int inter, int E, int k)
{
    if (T < 0 || d <= 0 || inter <= 0 || E <= 0 || k <= 0) return false;
    if (d % 256 || inter % 256) return false;
    if (k > 8 || k > E || E > 256) return false;
    if ((long long)T * k >= (1ll << 31)) return false;
    return true;
}

// scratch of moe_backward_h: dyq [P][d], its scale tiles, the scale image
struct BwdLayout {
    size_t dyq, dys, img, total;
};
BwdLayout bwd_layout(int T, int d, int inter, int E, int k)
{
    const long long P = (long long)T * k;
    const int R = gemm_tile_rows(P, E);
    const size_t tiles = (size_t)max_row_tiles(P, E, R);
    BwdLayout l;
    l.dyq = 0;
    l.dys = round_up256((size_t)P * d);
    l.img = l.dys + round_up256(tiles * stage_groups(d) * kBlockScaleBytes);
    l.total = l.img + round_up256((size_t)E * (inter / 128) * (d / 128) * kBlockScaleBytes);
    return l;
}

// scratch of moe_backward_x: each pair's dx (bf16 [P][d]), the [dg; du] scales
// in tile layout, the scale image of W13^T
struct BwdXLayout {
    size_t dxp, sft, img, total;
};
BwdXLayout bwdx_layout(int T, int d, int inter, int E, int k)
{
    const long long P = (long long)T * k;
    const int R = gemm_tile_rows(P, E);
    const size_t tiles = (size_t)max_row_tiles(P, E, R);
    BwdXLayout l;
    l.dxp = 0;
    l.sft = round_up256((size_t)P * d * 2);
    l.img = l.sft + round_up256(tiles * stage_groups(2 * inter) * kBlockScaleBytes);
    l.total = l.img + round_up256((size_t)E * (d / 128) * (2 * inter / 128) * kBlockScaleBytes);
    return l;
}

} // namespace

// moe_backward_h's scratch as moe_backward_w reads it: dy's E4M3 codes
// [P][d] in expert order at offset 0, their scales in the GEMM's tile layout
size_t bwd_h_dy_offset() { return 0; }
size_t bwd_h_dys_offset(int T, int d, int inter, int E, int k) { return bwd_layout(T, d, inter, E, k).dys; }

} // namespace fp4moe

using namespace fp4moe;

extern "C" size_t moe_backward_h_workspace_size(int T, int d, int inter, int E, int k)
{
    if (!bwd_shape_ok(T, d, inter, E, k)) return 0;
    return bwd_layout(T, d, inter, E, k).total;
}

extern "C" moe_status moe_backward_h(const uint16_t *dout, const uint8_t *w2_fp8t, const uint8_t *w2_s8t,
                                     const float *gu, const void *fwd_workspace, void *workspace,
                                     size_t workspace_bytes, uint8_t *dgu, uint8_t *dgu_scale, float *dgu_f32, int T,
                                     int d, int inter, int E, int k, void *stream)
{
    if (!dout || !w2_fp8t || !w2_s8t || !gu || !fwd_workspace || !dgu || !dgu_scale) return MOE_ERR_INVALID_ARG;
    if (T < 0 || d <= 0 || inter <= 0 || E <= 0 || k <= 0) return MOE_ERR_INVALID_ARG;
    if (!aligned_to(dout, 16) || !aligned_to(w2_fp8t, 16) || !aligned_to(gu, 32) || !aligned_to(dgu, 32) ||
        !aligned_to(fwd_workspace, 256) || (dgu_f32 && !aligned_to(dgu_f32, 32)))
        return MOE_ERR_INVALID_ARG;
    if (!bwd_shape_ok(T, d, inter, E, k)) return MOE_ERR_UNSUPPORTED_SHAPE;
    const BwdLayout L = bwd_layout(T, d, inter, E, k);
    if (workspace && (!aligned_to(workspace, 256) || workspace_bytes < L.total)) return MOE_ERR_WORKSPACE;
    if (T == 0) return MOE_OK;
    int num_sms = 0;
    unsigned *status = nullptr;
    moe_status st = device_query(&num_sms, &status);
    if (st != MOE_OK) return st;
    Workspace fw;
    if (!workspace_layout(Shapes{T, d, inter, E, k}, &fw)) return MOE_ERR_UNSUPPORTED_SHAPE;
    const uint8_t *fb = static_cast<const uint8_t *>(fwd_workspace);
    const long long P = (long long)T * k;
    const int R = gemm_tile_rows(P, E);

    cudaStream_t s = (cudaStream_t)stream;
    uint8_t *base = static_cast<uint8_t *>(workspace);
    bool owned = false;
    if (!base) {
        void *p = nullptr;
        if (cudaMallocAsync(&p, L.total, s) != cudaSuccess) {
            cudaGetLastError();
            return MOE_ERR_WORKSPACE;
        }
        base = static_cast<uint8_t *>(p);
        owned = true;
    }
    const int32_t *topk_idx = reinterpret_cast<const int32_t *>(fb + fw.off[MOE_WS_TOPK_IDX]);
    const float *topk_w = reinterpret_cast<const float *>(fb + fw.off[MOE_WS_TOPK_W]);
    const int32_t *offs = reinterpret_cast<const int32_t *>(fb + fw.off[MOE_WS_EXPERT_OFFSETS]);
    const int32_t *pair_pos = reinterpret_cast<const int32_t *>(fb + fw.off[MOE_WS_PAIR_POS]);
    const int32_t *tile_prefix = reinterpret_cast<const int32_t *>(fb + fw.off[MOE_WS_TILE_PREFIX]);
    uint8_t *dyq = base + L.dyq, *dys = base + L.dys, *img = base + L.img;

    const long long n16 = (long long)E * (inter / 128) * (d / 128) * (kBlockScaleBytes / 16);
    cudaError_t e = launch_pdl(bwd_scale_image_kernel, dim3((unsigned)((n16 + 255) / 256)), dim3(256), 0, s, w2_s8t,
                               img, n16, inter, d);
    if (e == cudaSuccess)
        e = launch_pdl(bwd_dy_kernel, dim3((unsigned)((T + 7) / 8)), dim3(256), 0, s, dout, topk_w, topk_idx,
                       pair_pos, offs, tile_prefix, dyq, dys, T, d, k, R);
    if (e == cudaSuccess) {
        GemmArgs g;
        std::memset(&g, 0, sizeof g);
        g.tile_rows = R;
        g.a = dyq;
        g.a_scale_tiles = dys;
        g.k = k;
        g.a_rows = P;
        g.b = w2_fp8t;
        g.b_scale = img;
        g.N = inter;
        g.K = d;
        g.expert_offsets = offs;
        g.tile_prefix = tile_prefix;
        g.E = E;
        g.P = P;
        g.status = status;
        g.timeout_ns = 2000000000ull;
        g.num_sms = num_sms;
        g.gu_in = gu;
        g.dgu = dgu;
        g.dgu_scale = dgu_scale;
        g.dgu_f32 = dgu_f32;
        e = launch_gemm_dgrad_h(g, inter, s);
    }
    if (owned) {
        cudaError_t f = cudaFreeAsync(base, s);
        if (e == cudaSuccess) e = f;
    }
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

extern "C" size_t moe_backward_x_workspace_size(int T, int d, int inter, int E, int k)
{
    if (!bwd_shape_ok(T, d, inter, E, k)) return 0;
    return bwdx_layout(T, d, inter, E, k).total;
}

extern "C" moe_status moe_backward_x(const uint8_t *dgu, const uint8_t *dgu_scale, const uint8_t *w13_fp8t,
                                     const uint8_t *w13_s8t, const void *fwd_workspace, void *workspace,
                                     size_t workspace_bytes, uint16_t *dx, int T, int d, int inter, int E, int k,
                                     void *stream)
{
    if (!dgu || !dgu_scale || !w13_fp8t || !w13_s8t || !fwd_workspace || !dx) return MOE_ERR_INVALID_ARG;
    if (T < 0 || d <= 0 || inter <= 0 || E <= 0 || k <= 0) return MOE_ERR_INVALID_ARG;
    if (!aligned_to(dgu, 16) || !aligned_to(w13_fp8t, 16) || !aligned_to(dx, 16) || !aligned_to(fwd_workspace, 256))
        return MOE_ERR_INVALID_ARG;
    if (!bwd_shape_ok(T, d, inter, E, k)) return MOE_ERR_UNSUPPORTED_SHAPE;
    const BwdXLayout L = bwdx_layout(T, d, inter, E, k);
    if (workspace && (!aligned_to(workspace, 256) || workspace_bytes < L.total)) return MOE_ERR_WORKSPACE;
    if (T == 0) return MOE_OK;
    int num_sms = 0;
    unsigned *status = nullptr;
    moe_status st = device_query(&num_sms, &status);
    if (st != MOE_OK) return st;
    Workspace fw;
    if (!workspace_layout(Shapes{T, d, inter, E, k}, &fw)) return MOE_ERR_UNSUPPORTED_SHAPE;
    const uint8_t *fb = static_cast<const uint8_t *>(fwd_workspace);
    const long long P = (long long)T * k;
    const int R = gemm_tile_rows(P, E);
    const int G = 2 * inter / 128;

    cudaStream_t s = (cudaStream_t)stream;
    uint8_t *base = static_cast<uint8_t *>(workspace);
    bool owned = false;
    if (!base) {
        void *p = nullptr;
        if (cudaMallocAsync(&p, L.total, s) != cudaSuccess) {
            cudaGetLastError();
            return MOE_ERR_WORKSPACE;
        }
        base = static_cast<uint8_t *>(p);
        owned = true;
    }
    const int32_t *topk_idx = reinterpret_cast<const int32_t *>(fb + fw.off[MOE_WS_TOPK_IDX]);
    const int32_t *offs = reinterpret_cast<const int32_t *>(fb + fw.off[MOE_WS_EXPERT_OFFSETS]);
    const int32_t *sorted_pair = reinterpret_cast<const int32_t *>(fb + fw.off[MOE_WS_SORTED_PAIR]);
    const int32_t *pair_pos = reinterpret_cast<const int32_t *>(fb + fw.off[MOE_WS_PAIR_POS]);
    const int32_t *tile_prefix = reinterpret_cast<const int32_t *>(fb + fw.off[MOE_WS_TILE_PREFIX]);
    uint16_t *dxp = reinterpret_cast<uint16_t *>(base + L.dxp);
    uint8_t *sft = base + L.sft, *img = base + L.img;

    const long long n16 = (long long)E * (d / 128) * G * (kBlockScaleBytes / 16);
    cudaError_t e = launch_pdl(bwd_scale_image_kernel, dim3((unsigned)((n16 + 255) / 256)), dim3(256), 0, s, w13_s8t,
                               img, n16, d, 2 * inter);
    if (e == cudaSuccess)
        e = launch_pdl(bwd_sf_tiles_kernel, dim3((unsigned)((P * G + 255) / 256)), dim3(256), 0, s, dgu_scale, topk_idx,
                       sorted_pair, offs, tile_prefix, sft, P, G, k, R);
    if (e == cudaSuccess) {
        GemmArgs g;
        std::memset(&g, 0, sizeof g);
        g.tile_rows = R;
        g.a = dgu;
        g.a_scale_tiles = sft;
        g.k = k;
        g.a_rows = P;
        g.b = w13_fp8t;
        g.b_scale = img;
        g.N = d;
        g.K = 2 * inter;
        g.expert_offsets = offs;
        g.tile_prefix = tile_prefix;
        g.E = E;
        g.P = P;
        g.y = dxp;
        g.status = status;
        g.timeout_ns = 2000000000ull;
        g.num_sms = num_sms;
        e = launch_gemm_dgrad_x(g, d, s);
    }
    if (e == cudaSuccess) e = launch_combine(dxp, pair_pos, nullptr, dx, T, d, k, s);
    if (owned) {
        cudaError_t f = cudaFreeAsync(base, s);
        if (e == cudaSuccess) e = f;
    }
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

extern "C" moe_status moe_backward_dw(const uint16_t *dout, const void *fwd_workspace, float *dw, int T, int d,
                                      int inter, int E, int k, void *stream)
{
    if (!dout || !fwd_workspace || !dw) return MOE_ERR_INVALID_ARG;
    if (T < 0 || d <= 0 || inter <= 0 || E <= 0 || k <= 0) return MOE_ERR_INVALID_ARG;
    if (!aligned_to(dout, 16) || !aligned_to(fwd_workspace, 256) || !aligned_to(dw, 4)) return MOE_ERR_INVALID_ARG;
    Workspace fw;
    if (!workspace_layout(Shapes{T, d, inter, E, k}, &fw)) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (T == 0) return MOE_OK;
    int num_sms = 0;
    unsigned *status = nullptr;
    moe_status st = device_query(&num_sms, &status);
    if (st != MOE_OK) return st;
    const uint8_t *fb = static_cast<const uint8_t *>(fwd_workspace);
    const long long P = (long long)T * k;
    const cudaError_t e = launch_pdl(bwd_dw_kernel, dim3((unsigned)((P + 7) / 8)), dim3(256), 0, (cudaStream_t)stream,
                                     dout, reinterpret_cast<const uint16_t *>(fb + fw.off[MOE_WS_Y]),
                                     reinterpret_cast<const int32_t *>(fb + fw.off[MOE_WS_PAIR_POS]), dw, P, d, k);
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
