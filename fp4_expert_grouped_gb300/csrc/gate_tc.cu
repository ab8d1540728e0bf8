// gate_tc.cu -- gate + top-k for large batches: tensor-core logits with a
// proven error bound, and the routing decided exactly as by the fixed fp32
// order of the gate logits.
//
// The routing contract (fixed-order fp32 logits z = x . gate_w + bias, top-k
// by z with ties to the lower expert, weights sqrt(softplus(z)) renormalised;
// "DeepSeek V4架构学习笔记", 67808.cn/a/484462.html, DeepSeekMoE paragraph)
// takes T*d*E fp32 fused multiply-adds on the CUDA cores, a quarter of the
// layer's time at the largest batches.  Here the dense contraction runs on the
// tensor cores instead, and exactness is kept by certification:
//
//   1. gate_w is split into bf16 hi + lo parts (w = hi + lo + r, |r| <= 2^-16 |w|)
//      and transposed ([E][d], the operand layout of the MMA).
//   2. a = x . (hi + lo) + bias on tcgen05 (bf16 x bf16, fp32 accumulate).  The
//      accumulation restarts every 128 channels (16 MMAs) in one of two
//      tensor-memory buffers, and the 128-channel sums are added in fp32 in
//      registers, so the tensor core's own rounding enters only over 16
//      instructions.
//   3. per token, a bound D_e >= |a_e - z_e| (z_e the fixed-order logit) from
//      the norms: D_e = c(d) ||x|| ||w_e|| + 2^-22 |a_e| + d 2^-125, c(d) from
//      the error terms of both computations (see gate_bound_coefficient).  With L the
//      k-th largest a_e - D_e, every expert of the exact top-k has
//      a_e + D_e >= L; those are the candidates (k plus, typically, a fraction
//      of one).  Their fixed-order logits are computed exactly as the
//      CUDA-core gate computes them (32 chains of fused multiply-adds, then
//      the xor tree), and the top-k, the slot order and the weights come from
//      those exact logits.  So the routing and its weights are bit-identical
//      to the fixed-order gate's, and to the oracle's, for any batch.
//
// Section 3.1 of "DeepSeek-V4揭秘：细粒度专家并行隐藏通信时延，FP4量化与TileLang协同优化百万Token上下文"
// (itsolotime.com/archives/32374): the result of a token does not depend on
// the batch.  The approximate logits may (they never reach an output); the
// certified routing does not.
#include "moe_device.cuh"
#include "moe_internal.h"

#include <cmath>

namespace fp4moe {

// An upper bound of sqrt(v) for v an fp32 sum of n squares accumulated with
// fused multiply-adds (see gate_wnorm_kernel).
__device__ __forceinline__ float norm_upper_bound(float ssq, int n)
{
    const float ub = __fmaf_ru(ssq, 1.0f + 0x1p-10f, __fmul_ru((float)n, 0x1p-149f));
    return __fmul_ru(__fsqrt_ru(ub), 1.0f + 0x1p-20f);
}

// ---------------------------------------------------------------------------
// 1. split + transpose of gate_w, and the experts' weight norms
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) gate_split_kernel(const float *__restrict__ gw, float *__restrict__ wt,
                                                         uint16_t *__restrict__ whi, uint16_t *__restrict__ wlo,
                                                         int d, int E)
{
    pdl_wait();
    __shared__ float tile[32][33];
    const int i0 = blockIdx.x * 32, e0 = blockIdx.y * 32;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    for (int r = ty; r < 32; r += 8) {
        const int e = e0 + tx;
        tile[r][tx] = e < E ? __ldg(gw + (size_t)(i0 + r) * E + e) : 0.f;
    }
    __syncthreads();
    for (int r = ty; r < 32; r += 8) {
        const int e = e0 + r, i = i0 + tx;
        if (e < E) {
            const float w = tile[tx][r];
            const __nv_bfloat16 hi = __float2bfloat16_rn(w);
            // w - hi is exact in fp32 (hi is w rounded to 8 significant bits)
            const __nv_bfloat16 lo = __float2bfloat16_rn(w - __bfloat162float(hi));
            wt[(size_t)e * d + i] = w;
            whi[(size_t)e * d + i] = __bfloat16_as_ushort(hi);
            wlo[(size_t)e * d + i] = __bfloat16_as_ushort(lo);
        }
    }
    pdl_trigger();
}

// Upper bound of ||w_e||_2: the fp32 sum of squares (32 fused multiply-add
// chains and a tree, relative error below 2^-16 for d < 2^19; once the terms
// are subnormal each step may lose up to 2^-150 more) raised by 2^-10 plus
// d 2^-149, its square root rounded up and raised by 2^-20.
__global__ void __launch_bounds__(256) gate_wnorm_kernel(const float *__restrict__ wt, float *__restrict__ wn, int d,
                                                         int E)
{
    pdl_wait();
    const int e = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (e < E) {
        float s = 0.f;
        for (int i = lane; i < d; i += 32) {
            const float v = __ldg(wt + (size_t)e * d + i);
            s = fmaf(v, v, s);
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) s = s + __shfl_xor_sync(0xffffffffu, s, off);
        if (lane == 0) wn[e] = norm_upper_bound(s, d);
    }
    pdl_trigger();
}

// ---------------------------------------------------------------------------
// 2. a = x . (hi + lo) + bias on the tensor cores
// ---------------------------------------------------------------------------
namespace gtc {

constexpr int BM = 128;                // tokens per tile (MMA M)
constexpr int SK = 32;                 // channels per ring stage: 64-byte rows of bf16
constexpr int CHUNK_STAGES = 4;        // 128 channels per accumulation chunk
constexpr int STAGES = 5;
constexpr int EPI_WARPS = 8;
constexpr int NUM_THREADS = (2 + EPI_WARPS) * 32;
constexpr int A_STAGE = BM * SK * 2;   // 8 KB of x

template <int NH>                      // 64 * NH experts per work unit
struct Cfg {
    static constexpr int E = 64 * NH;
    static constexpr int B_STAGE = E * SK * 2;                 // hi (or lo) rows of one stage
    static constexpr uint32_t STAGE_TX = A_STAGE + 2 * B_STAGE;
    static constexpr int OFF_A = 0;
    static constexpr int OFF_BHI = OFF_A + STAGES * A_STAGE;
    static constexpr int OFF_BLO = OFF_BHI + STAGES * B_STAGE;
    static constexpr int OFF_BAR = OFF_BLO + STAGES * B_STAGE;
    // full and empty per stage; full and empty per accumulator buffer; exit drain
    static constexpr int OFF_MISC = OFF_BAR + (2 * STAGES + 4 + 1) * 8;
    static constexpr int SMEM_USED = OFF_MISC + 16;
    static constexpr int SMEM_BYTES = SMEM_USED + 1024;         // slack for 1024-byte alignment
    // two accumulator buffers of E fp32 columns
    static constexpr uint32_t TMEM_COLS = 2 * E <= 128 ? 128 : 2 * E <= 256 ? 256 : 512;
    // MMA: kind::f16, fp32 accumulator (bit 4), A and B bf16 (bits 7, 10), both
    // K-major, N = E, M = 128
    static constexpr uint32_t IDESC = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(E >> 3) << 17) |
                                      ((uint32_t)(BM >> 4) << 24);
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");
    static_assert(B_STAGE % 512 == 0, "64-byte swizzle atoms stay aligned");
};

// A work unit is 128 tokens x 64 * NH experts (column block cb of the E_all
// experts); a small batch splits the experts over several units so that more
// SMs stream the weights.  Warp roles (320 threads): warp 0 producer (TMA
// loads of x and of the unit's hi and lo weight rows, 32 channels per stage),
// warp 1 tensor-memory owner and MMA issuer (one thread: per stage two MMAs of
// K = 16 on hi, two on lo), warps 2-9 epilogue (two per 32-lane quarter, each
// with half of the unit's experts: per 128-channel chunk, the buffer's fp32
// sums added into registers; at the end of the unit the bias is added and the
// row stored).
template <int NH>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gate_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmHi,
                   const __grid_constant__ CUtensorMap tmLo, const float *__restrict__ bias, float *__restrict__ approx,
                   int T, int d, int E_all, unsigned *status, unsigned long long timeout_ns)
{
    using C = Cfg<NH>;
    constexpr int E = C::E;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    uint64_t *empty = full + STAGES;
    uint64_t *acc_full = full + 2 * STAGES;      // [2]
    uint64_t *acc_empty = acc_full + 2;          // [2]
    uint64_t *drain = acc_empty + 2;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; s++) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; b++) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], EPI_WARPS);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmX);
        tma_prefetch_desc(&tmHi);
        tma_prefetch_desc(&tmLo);
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, C::TMEM_COLS);
        tmem_relinquish();
    }
    pdl_wait();                                  // x and the split weights come from earlier work
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const int ncb = E_all / E;                   // column blocks per token tile
    const int n_units = (T + BM - 1) / BM * ncb;
    const int nst = d / SK;                      // stages per tile
    const int nch = nst / CHUNK_STAGES;          // chunks per tile (d % 128 == 0)

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            uint32_t stage = 0, phase = 0;
            long long armed = 0;
            for (int u = blockIdx.x; u < n_units && !*abort_flag; u += gridDim.x) {
                const int tile = u / ncb, e0 = (u - tile * ncb) * E;
                for (int s = 0; s < nst; s++) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, timeout_ns, abort_flag)) {
                        *abort_flag = 1;
                        break;
                    }
                    uint64_t *fb = &full[stage];
                    armed++;
                    mbar_arrive_expect_tx(fb, C::STAGE_TX);
                    tma_load_2d(smem + C::OFF_A + stage * A_STAGE, &tmX, fb, s * SK, tile * BM);
                    tma_load_2d(smem + C::OFF_BHI + stage * C::B_STAGE, &tmHi, fb, s * SK, e0);
                    tma_load_2d(smem + C::OFF_BLO + stage * C::B_STAGE, &tmLo, fb, s * SK, e0);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // leave no copy in flight: the last use of every slot armed so far
            for (int s = 0; s < STAGES; s++) {
                if (armed <= s) continue;
                mbar_wait_drain(&full[s], s < (int)stage ? phase : (phase ^ 1u), timeout_ns);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            uint32_t stage = 0, phase = 0, gc = 0;
            const uint32_t sbase = smem_u32(smem);
            bool ok = true;
            for (int u = blockIdx.x; ok && u < n_units && !*abort_flag; u += gridDim.x) {
                for (int c = 0; ok && c < nch; c++, gc++) {
                    const uint32_t b = gc & 1u, use = gc >> 1;
                    if (!mbar_wait(&acc_empty[b], (use & 1u) ^ 1u, timeout_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t dcol = tmem + b * E;
                    for (int s = 0; s < CHUNK_STAGES; s++) {
                        if (!mbar_wait(&full[stage], phase, timeout_ns, abort_flag)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint64_t ad = sdesc_kmajor_sw64(sbase + C::OFF_A + stage * A_STAGE);
                        const uint64_t hd = sdesc_kmajor_sw64(sbase + C::OFF_BHI + stage * C::B_STAGE);
                        const uint64_t ld = sdesc_kmajor_sw64(sbase + C::OFF_BLO + stage * C::B_STAGE);
                        // K = 16 per MMA: 32 bytes along the 64-byte row (descriptor
                        // start address in 16-byte units)
#pragma unroll
                        for (int kk = 0; kk < 2; kk++)
                            tc_mma_bf16(dcol, ad + 2 * kk, hd + 2 * kk, C::IDESC, (s | kk) != 0);
#pragma unroll
                        for (int kk = 0; kk < 2; kk++) tc_mma_bf16(dcol, ad + 2 * kk, ld + 2 * kk, C::IDESC, 1u);
                        tc_commit(&empty[stage]);
                        if (++stage == STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                    if (ok) tc_commit(&acc_full[b]);
                }
            }
            if (!ok) *abort_flag = 1;
            // tensor memory is freed below: let this thread's MMAs finish
            tc_commit(drain);
            mbar_wait_drain(drain, 0, timeout_ns);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3, half = (warp - 2) >> 2;
        const int r = q * 32 + lane;
        const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(half * (E / 2));
        uint32_t gc = 0;
        for (int u = blockIdx.x; u < n_units && !*abort_flag; u += gridDim.x) {
            float sum[32 * NH];
#pragma unroll
            for (int i = 0; i < 32 * NH; i++) sum[i] = 0.f;
            bool ok = true;
            for (int c = 0; c < nch; c++, gc++) {
                const uint32_t b = gc & 1u, use = gc >> 1;
                if (!mbar_wait(&acc_full[b], use & 1u, timeout_ns, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int i = 0; i < NH; i++) {
                    uint32_t v[32];
                    tmem_ld32(lane_base + b * E + 32 * i, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; j++) sum[32 * i + j] = sum[32 * i + j] + __uint_as_float(v[j]);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&acc_empty[b]);
            }
            if (!ok) {
                *abort_flag = 1;
                break;
            }
            const int tile = u / ncb, e0 = (u - tile * ncb) * E;
            const int t = tile * BM + r;
            if (t < T) {
                float *dst = approx + (size_t)t * E_all + e0 + half * (E / 2);
#pragma unroll
                for (int i = 0; i < 32 * NH; i += 8) {
                    uint32_t w[8];
#pragma unroll
                    for (int m = 0; m < 8; m++) {
                        float v = sum[i + m];
                        if (bias) v = v + __ldg(bias + e0 + half * (E / 2) + i + m);
                        w[m] = __float_as_uint(v);
                    }
                    st_global_v8(dst + i, w);
                }
            }
        }
    }

    pdl_trigger();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (threadIdx.x == 0 && *abort_flag) flag_status(status, kStatusTimeout);
    if (warp == 1) tmem_dealloc(tmem, C::TMEM_COLS);
}

} // namespace gtc

// ---------------------------------------------------------------------------
// 3. per token: bounds, candidates, their exact fixed-order logits, top-k,
//    weights; the FP8 quantisation of x in the same pass
// ---------------------------------------------------------------------------

// The token's bf16 row, 8 channels per lane and step, quantised to E4M3 with
// one power-of-two scale per 128 channels when qrow is given (two groups per
// step, one per half-warp: the rule of moe_quantize_act); returns this lane's
// part of the row's sum of squares.  The row is read B steps (B KB) at a
// time, all loads in flight together: the row comes from DRAM, and one
// dependent load per step made this the longest part of a token's work.  B =
// 8 up to d = 4096 (two batches), 12 above (three batches instead of four at
// d = 7168: certify 349 -> 326 us at 16K tokens; at d = 4096 the larger batch
// only cost registers).
template <int B>
__device__ __forceinline__ float quant_row_ssq(const uint16_t *__restrict__ xrow, uint8_t *__restrict__ qrow,
                                               uint8_t *__restrict__ srow, int d, int s_stride)
{
    const int lane = threadIdx.x & 31;
    const int n8 = d / 8;
    const uint4 *src = reinterpret_cast<const uint4 *>(xrow);
    float ssq = 0.f;
    for (int c0 = 0; c0 < n8; c0 += 32 * B) {
        uint4 cur[B];
#pragma unroll
        for (int b = 0; b < B; b++) {
            const int c = c0 + 32 * b + lane;
            cur[b] = c < n8 ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int b = 0; b < B; b++) {
            const int c = c0 + 32 * b + lane;
            if (c0 + 32 * b >= n8) break;                  // warp-uniform
            const uint32_t u[4] = {cur[b].x, cur[b].y, cur[b].z, cur[b].w};
            float v[8];
#pragma unroll
            for (int i = 0; i < 4; i++) {
                v[2 * i] = bf16_bits_to_f32(u[i] & 0xFFFFu);
                v[2 * i + 1] = bf16_bits_to_f32(u[i] >> 16);
            }
            float amax = 0.f;
#pragma unroll
            for (int i = 0; i < 8; i++) {
                amax = fmaxf(amax, fabsf(v[i]));
                ssq = fmaf(v[i], v[i], ssq);
            }
            if (qrow) {
#pragma unroll
                for (int off = 8; off >= 1; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
                if (c < n8) {
                    const int e = e4m3_scale_exp(amax);
                    const float sc = exp2i(-e);
                    uint2 q;
                    q.x = cvt_e4m3x2(v[0] * sc, v[1] * sc) | (cvt_e4m3x2(v[2] * sc, v[3] * sc) << 16);
                    q.y = cvt_e4m3x2(v[4] * sc, v[5] * sc) | (cvt_e4m3x2(v[6] * sc, v[7] * sc) << 16);
                    reinterpret_cast<uint2 *>(qrow)[c] = q;
                    if ((lane & 15) == 0) srow[c / 16] = (uint8_t)(e + 127);
                }
            }
        }
    }
    if (qrow)
        for (int g = d / 128 + lane; g < s_stride; g += 32) srow[g] = 0;
    return ssq;
}

// Order-preserving 32-bit image of a float (-0 taken as +0).
__device__ __forceinline__ uint32_t ord_f32(float v)
{
    const uint32_t u = __float_as_uint(v + 0.0f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float unord_f32(uint32_t o)
{
    return __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o);
}

constexpr int kCertWarps = 4;           // tokens per CTA (a warp each)

// The fixed-order logits of GS candidate experts ec[0..GS) of one token, by
// one warp: lane l runs chain l (channels l, l+32, ... with fused
// multiply-adds), the xor tree adds the chains in the fixed order's pairs, the
// bias comes last; the result goes to the lane holding that expert.  U channel
// steps of all GS experts' weights (and of x) are loaded before their
// multiply-adds: U = 8 for a group of 8, more for the smaller groups that take
// the last candidates (32 for one, 16 for two or four), so that every group
// keeps about 70 loads per lane in flight (the step is latency-bound: a group
// of one at U = 8 took as long as a group of eight).
template <int GS>
__device__ __forceinline__ void exact_logits(const int *ec_list, const uint16_t *__restrict__ xrow,
                                             const float *__restrict__ wt, const float *__restrict__ bias, int d,
                                             int lane, float (&zx)[8])
{
    int ec[GS];
    const float *wp[GS];
#pragma unroll
    for (int c = 0; c < GS; c++) {
        ec[c] = ec_list[c];
        wp[c] = wt + (size_t)ec[c] * d + lane;
    }
    const uint16_t *xp = xrow + lane;
    float acc[GS];
#pragma unroll
    for (int c = 0; c < GS; c++) acc[c] = 0.f;
    const int nj = d / 32;
    constexpr int U = GS == 1 ? 32 : GS <= 4 ? 16 : 8;
    int j = 0;
    for (; j + U <= nj; j += U) {
        float xv[U], wv[GS][U];
#pragma unroll
        for (int u = 0; u < U; u++) xv[u] = bf16_bits_to_f32(__ldg(xp + (j + u) * 32));
#pragma unroll
        for (int c = 0; c < GS; c++)
#pragma unroll
            for (int u = 0; u < U; u++) wv[c][u] = __ldg(wp[c] + (j + u) * 32);
#pragma unroll
        for (int u = 0; u < U; u++)
#pragma unroll
            for (int c = 0; c < GS; c++) acc[c] = fmaf(xv[u], wv[c][u], acc[c]);
    }
    for (; j + 8 <= nj; j += 8) {             // what is left of the U-step blocks, 8 steps at a time
        float xv[8], wv[GS][8];
#pragma unroll
        for (int u = 0; u < 8; u++) xv[u] = bf16_bits_to_f32(__ldg(xp + (j + u) * 32));
#pragma unroll
        for (int c = 0; c < GS; c++)
#pragma unroll
            for (int u = 0; u < 8; u++) wv[c][u] = __ldg(wp[c] + (j + u) * 32);
#pragma unroll
        for (int u = 0; u < 8; u++)
#pragma unroll
            for (int c = 0; c < GS; c++) acc[c] = fmaf(xv[u], wv[c][u], acc[c]);
    }
    for (; j < nj; j += 4) {                 // d % 256 == 128: four steps left
        float xv[4], wv[GS][4];
#pragma unroll
        for (int u = 0; u < 4; u++) xv[u] = bf16_bits_to_f32(__ldg(xp + (j + u) * 32));
#pragma unroll
        for (int c = 0; c < GS; c++)
#pragma unroll
            for (int u = 0; u < 4; u++) wv[c][u] = __ldg(wp[c] + (j + u) * 32);
#pragma unroll
        for (int u = 0; u < 4; u++)
#pragma unroll
            for (int c = 0; c < GS; c++) acc[c] = fmaf(xv[u], wv[c][u], acc[c]);
    }
#pragma unroll
    for (int c = 0; c < GS; c++) {
        float v = acc[c];
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) v = v + __shfl_xor_sync(0xffffffffu, v, off);
        if (bias) v = v + __ldg(bias + ec[c]);
#pragma unroll
        for (int m = 0; m < 8; m++) zx[m] = (ec[c] == lane + 32 * m) ? v : zx[m];
    }
}

template <int QB>
__global__ void __launch_bounds__(kCertWarps * 32) gate_certify_kernel(
    const uint16_t *__restrict__ x, const float *__restrict__ approx, const float *__restrict__ wt,
    const float *__restrict__ wn, const float *__restrict__ bias, float crel, int32_t *__restrict__ topk_idx,
    float *__restrict__ topk_w, float *__restrict__ topk_z, int32_t *__restrict__ ncand, uint8_t *__restrict__ xq,
    uint8_t *__restrict__ xs, int xs_stride, int T, int d, int E, int k, unsigned *status)
{
    pdl_wait();
    extern __shared__ __align__(16) uint8_t cert_smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * kCertWarps + warp;
    if (t >= T) return;
    int *cl = reinterpret_cast<int *>(cert_smem) + warp * 256;     // the token's candidates

    // the row, its quantisation and an upper bound of ||x||_2 (as for the weights)
    float ssq = quant_row_ssq<QB>(x + (size_t)t * d, xq ? xq + (size_t)t * d : nullptr,
                              xq ? xs + (size_t)t * xs_stride : nullptr, d, xs_stride);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) ssq = ssq + __shfl_xor_sync(0xffffffffu, ssq, off);
    const float xn = norm_upper_bound(ssq, d);
    // products the tensor core may flush to zero (below 2^-126 each)
    const float d_abs = __fmul_ru((float)d, 0x1p-125f);

    // bounds of every logit: [a - D, a + D] holds the fixed-order logit
    float lb[8], ub[8];
#pragma unroll
    for (int m = 0; m < 8; m++) {
        const int e = lane + 32 * m;
        lb[m] = -INFINITY;
        ub[m] = -INFINITY;
        if (e < E) {
            const float a = __ldg(approx + (size_t)t * E + e);
            const float D = __fadd_ru(__fadd_ru(__fmul_ru(__fmul_ru(crel, xn), __ldg(wn + e)),
                                                __fmul_ru(0x1p-22f, fabsf(a))),
                                      d_abs);
            if (isfinite(a) && isfinite(D)) {
                lb[m] = __fsub_rd(a, D);
                ub[m] = __fadd_ru(a, D);
            } else {
                ub[m] = INFINITY;            // no usable bound: a candidate
            }
        }
    }
    // L = the k-th largest lower bound
    float L = -INFINITY;
    {
        uint64_t key[8];
#pragma unroll
        for (int m = 0; m < 8; m++) {
            const int e = lane + 32 * m;
            key[m] = e < E ? ((uint64_t)ord_f32(lb[m]) << 32) | (uint32_t)(0xFFFFFFFFu - (uint32_t)e) : 0ull;
        }
        for (int j = 0; j < k; j++) {
            uint64_t best = key[0];
#pragma unroll
            for (int m = 1; m < 8; m++) best = key[m] > best ? key[m] : best;
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) {
                const uint64_t o = __shfl_xor_sync(0xffffffffu, best, off);
                best = o > best ? o : best;
            }
            const int e = (int)(0xFFFFFFFFu - (uint32_t)best);
#pragma unroll
            for (int m = 0; m < 8; m++) key[m] = ((e & 31) == lane && m == (e >> 5)) ? 0ull : key[m];
            if (j == k - 1) L = unord_f32((uint32_t)(best >> 32));
        }
    }
    // candidates: upper bound reaching L (the exact top-k is among them)
    unsigned cmask[8];
    int n = 0;
    const unsigned lt = (1u << lane) - 1u;
#pragma unroll
    for (int m = 0; m < 8; m++) {
        const int e = lane + 32 * m;
        const bool cand = e < E && !(ub[m] < L);
        cmask[m] = __ballot_sync(0xffffffffu, cand);
        if (cand) cl[n + __popc(cmask[m] & lt)] = e;
        n += __popc(cmask[m]);
    }
    __syncwarp();

    // the candidates' fixed-order logits, in groups of 8, then 4, 2, 1
    float zx[8];
#pragma unroll
    for (int m = 0; m < 8; m++) zx[m] = 0.f;
    const uint16_t *xrow = x + (size_t)t * d;
    int g = 0;
    for (; g + 8 <= n; g += 8) exact_logits<8>(cl + g, xrow, wt, bias, d, lane, zx);
    if (g + 4 <= n) {
        exact_logits<4>(cl + g, xrow, wt, bias, d, lane, zx);
        g += 4;
    }
    if (g + 2 <= n) {
        exact_logits<2>(cl + g, xrow, wt, bias, d, lane, zx);
        g += 2;
    }
    if (g < n) exact_logits<1>(cl + g, xrow, wt, bias, d, lane, zx);

    // top-k of the candidates by exact logit (descending, ties to the lower
    // expert), weights from those logits -- as the CUDA-core top-k does
    uint64_t key[8];
    bool bad = false;
#pragma unroll
    for (int m = 0; m < 8; m++) {
        const int e = lane + 32 * m;
        uint64_t kk = 0;
        if ((cmask[m] >> lane) & 1u) {
            float v = zx[m];
            if (isnan(v)) {
                bad = true;
                v = -INFINITY;
            }
            kk = ((uint64_t)ord_f32(v) << 32) | (uint32_t)(0xFFFFFFFFu - (uint32_t)e);
        }
        key[m] = kk;
    }
    float my_z = 0.f;
    int my_e = 0;
    for (int j = 0; j < k; j++) {
        uint64_t best = key[0];
#pragma unroll
        for (int m = 1; m < 8; m++) best = key[m] > best ? key[m] : best;
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) {
            const uint64_t o = __shfl_xor_sync(0xffffffffu, best, off);
            best = o > best ? o : best;
        }
        const int e = (int)(0xFFFFFFFFu - (uint32_t)best);
#pragma unroll
        for (int m = 0; m < 8; m++) key[m] = ((e & 31) == lane && m == (e >> 5)) ? 0ull : key[m];
        if (lane == j) {
            my_z = unord_f32((uint32_t)(best >> 32));
            my_e = e;
        }
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) flag_status(status, kStatusBadData);
    float s = 0.f;
    if (lane < k) {
        const double zd = (double)my_z;
        const double sp = (zd > 0.0 ? zd : 0.0) + log1p(exp(-fabs(zd)));
        s = (float)sqrt(sp);
    }
    float S = 0.f;
    for (int j = 0; j < k; j++) S = S + __shfl_sync(0xffffffffu, s, j);
    if (lane < k) {
        topk_idx[(size_t)t * k + lane] = my_e;
        topk_w[(size_t)t * k + lane] = (S == 0.f) ? 1.0f / (float)k : s / S;
        if (topk_z) topk_z[(size_t)t * k + lane] = my_z;
    }
    if (ncand && lane == 0) ncand[t] = n;
    pdl_trigger();
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
bool gate_uses_tc(long long T, int d, int E)
{
    return T >= kGateTcMinTokens && E % 64 == 0 && E >= 64 && E <= 256 && d % 128 == 0;
}

// c(d) of the bound |a - z| <= c(d) ||x|| ||w_e|| + 2^-22 |a| + d 2^-125
// (Cauchy-Schwarz: sum_i |x_i w_i| <= ||x|| ||w_e||; the last term covers
// products below the normal range that the tensor core may flush), the sum of:
//   2^-16              the split: |w - hi - lo| <= 2^-16 |w|
//   17 u_tc (1 + 2^-6) the tensor core over one 128-channel chunk, 16 MMAs of
//                      K = 16, each assumed to add its products to the
//                      accumulator with error <= u_tc (|acc| + sum |products|);
//                      u_tc = 2^-17 allows 7 bits of loss against fp32 (the
//                      measured worst case is recorded beside the tests)
//   (d/128) 2^-24      the fp32 running sum of the d/128 chunk sums
//   (d/32 + 5) 2^-24   the fixed-order logit against the exact dot product
//                      (chains of d/32 fused multiply-adds, a 5-level tree)
// each first-order term raised by 2^-6 for the second-order ones; the bias
// additions on both sides are covered by the 2^-22 |a| term.
float gate_bound_coefficient(int d)
{
    const double u = 0x1p-24, u_tc = 0x1p-17;
    const double c = 0x1p-16 + 17.0 * u_tc + (d / 128.0) * u + (d / 32.0 + 5.0) * u;
    return (float)(c * (1.0 + 0x1p-6) * 1.01);
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn gate_encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// bf16 rows [rows][d], a 32-channel x box_rows box, 64-byte swizzle (rows past
// the end read as zeros)
static bool make_map_bf16(CUtensorMap *m, const void *base, long long rows, int d, int box_rows)
{
    EncodeTiledFn enc = gate_encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)d * 2};
    cuuint32_t box[2] = {(cuuint32_t)gtc::SK, (cuuint32_t)box_rows};
    cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int NH>
static cudaError_t launch_gate_tc_cfg(const CUtensorMap &mx, const CUtensorMap &mh, const CUtensorMap &ml,
                                      const float *bias, float *approx, int T, int d, int E, int num_sms,
                                      unsigned *status, unsigned long long timeout_ns, cudaStream_t st)
{
    using C = gtc::Cfg<NH>;
    auto kern = gtc::gate_tc_kernel<NH>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (err != cudaSuccess) return err;
    const int units = (T + gtc::BM - 1) / gtc::BM * (E / C::E);
    const int grid = units < num_sms ? units : num_sms;
    return launch_pdl(kern, dim3(grid), dim3(gtc::NUM_THREADS), C::SMEM_BYTES, st, mx, mh, ml, bias, approx, T, d, E,
                      status, timeout_ns);
}

// Experts per work unit (64 * NH of the E): each unit streams its 128 tokens'
// x and its experts' hi and lo rows through one SM at the SM's copy rate, so
// the launch takes about (units per SM, rounded up) x (x bytes + weight
// bytes of a unit).  Splitting the experts pays when the token tiles alone
// leave SMs idle: on 152 SMs with E = 256, 4096 tokens (32 tiles) run units
// of 64 experts, 8192 tokens units of 128, 16384 tokens units of all 256.
static int gate_tc_experts_per_unit(int T, int E, int num_sms)
{
    const long long tiles = (T + gtc::BM - 1) / gtc::BM;
    int best = E;
    long long best_cost = -1;
    for (int ncb = 1; ncb <= 4; ncb *= 2) {
        if (E % (64 * ncb) != 0) continue;
        const int ecta = E / ncb;
        const long long units = tiles * ncb;
        const long long rounds = (units + num_sms - 1) / num_sms;
        // per unit: x 128 rows x 2 bytes, weights ecta rows x 4 bytes (hi, lo)
        const long long cost = rounds * (2LL * gtc::BM + 4LL * ecta);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = ecta;
        }
    }
    return best;
}

cudaError_t launch_gate_prep(const float *gate_w, const GateScratch &g, int d, int E, cudaStream_t st)
{
    cudaError_t err = launch_pdl(gate_split_kernel, dim3(d / 32, (E + 31) / 32), dim3(256), 0, st, gate_w, g.wt, g.whi,
                                 g.wlo, d, E);
    if (err != cudaSuccess) return err;
    return launch_pdl(gate_wnorm_kernel, dim3((E + 7) / 8), dim3(256), 0, st, (const float *)g.wt, g.wn, d, E);
}

cudaError_t launch_gate_tc_logits(const uint16_t *x, const float *gate_w, const float *bias, const GateScratch &g,
                                  int T, int d, int E, int num_sms, unsigned *status, unsigned long long timeout_ns,
                                  cudaStream_t st)
{
    if (T == 0) return cudaSuccess;
    if (!gate_uses_tc(T, d, E)) return cudaErrorInvalidValue;
    cudaError_t err = cudaSuccess;
    if (!g.prepared) {
        err = launch_gate_prep(gate_w, g, d, E, st);
        if (err != cudaSuccess) return err;
    }
    const int ecta = gate_tc_experts_per_unit(T, E, num_sms);
    CUtensorMap mx, mh, ml;
    if (!make_map_bf16(&mx, x, T, d, gtc::BM) || !make_map_bf16(&mh, g.whi, E, d, ecta) ||
        !make_map_bf16(&ml, g.wlo, E, d, ecta))
        return cudaErrorInvalidValue;
    switch (ecta / 64) {
    case 1: err = launch_gate_tc_cfg<1>(mx, mh, ml, bias, g.approx, T, d, E, num_sms, status, timeout_ns, st); break;
    case 2: err = launch_gate_tc_cfg<2>(mx, mh, ml, bias, g.approx, T, d, E, num_sms, status, timeout_ns, st); break;
    case 3: err = launch_gate_tc_cfg<3>(mx, mh, ml, bias, g.approx, T, d, E, num_sms, status, timeout_ns, st); break;
    default: err = launch_gate_tc_cfg<4>(mx, mh, ml, bias, g.approx, T, d, E, num_sms, status, timeout_ns, st); break;
    }
    return err;
}

cudaError_t launch_gate_certify(const uint16_t *x, const float *bias, const GateScratch &g, int32_t *topk_idx,
                                float *topk_w, float *topk_z, uint8_t *xq, uint8_t *xs, int xs_stride, int T, int d,
                                int E, int k, unsigned *status, cudaStream_t st)
{
    if (T == 0) return cudaSuccess;
    const size_t smem = (size_t)kCertWarps * 256 * 4;
    auto kern = d > 4096 ? gate_certify_kernel<12> : gate_certify_kernel<8>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    return launch_pdl(kern, dim3((T + kCertWarps - 1) / kCertWarps), dim3(kCertWarps * 32), smem, st,
                      x, (const float *)g.approx, (const float *)g.wt, (const float *)g.wn, bias,
                      gate_bound_coefficient(d), topk_idx, topk_w, topk_z, g.ncand, xq, xs, xs_stride, T, d, E, k,
                      status);
}

} // namespace fp4moe
