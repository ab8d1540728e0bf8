// kernels.cu -- the CUDA-core stages of the MoE layer forward:
//   MXFP4 weight packing, FP8 E4M3 activation quantisation, fixed-order gate
//   logits, warp-level top-k with sqrt(softplus) weights, the stable
//   counting-sort dispatch plan, the dispatch copy into expert order and the
//   slot-order combine.
//
// Sources: "DeepSeek-V4揭秘：细粒度专家并行隐藏通信时延，FP4量化与TileLang协同优化百万Token上下文"
// (itsolotime.com/archives/32374): section 1.1 (dispatch / combine stages),
// 1.4 (FP8 dispatch, BF16 combine), 3.1-3.2 (batch invariance, no
// atomic-order-dependent sums), 4 (MXFP4 expert weights).
// "DeepSeek V4架构学习笔记" (67808.cn/a/484462.html), DeepSeekMoE paragraph:
// the sqrt(softplus(.)) gate activation.
#include "moe_device.cuh"
#include "moe_internal.h"

#include <algorithm>
#include <climits>

namespace fp4moe {

// ---------------------------------------------------------------------------
// MXFP4 packing into the tiled layout (moe_internal.h).  One thread per 8
// consecutive K elements; four threads share a 32-element block (scale
// X = floor(log2 amax) - 2, codes = RNE E2M1 of w * 2^-X saturated to +-6,
// low nibble = even element).  The codes of row n, columns k..k+7 land at
// block b = weight_block(e, n/128, k/128), row n % 128, byte (k % 128)/2; the
// scale byte at b * 512 + sf_byte(n % 128, (k % 128) / 32).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) pack_fp4_kernel(const float *__restrict__ w, uint8_t *__restrict__ w_fp4,
                                                       uint8_t *__restrict__ w_scale, long long n8, int N, int K)
{
    pdl_wait();
    const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const bool valid = gid < n8;
    float v[8];
    if (valid) {
        const float4 a = __ldg(reinterpret_cast<const float4 *>(w) + 2 * gid);
        const float4 b = __ldg(reinterpret_cast<const float4 *>(w) + 2 * gid + 1);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else {
#pragma unroll
        for (int i = 0; i < 8; i++) v[i] = 0.f;
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 8; i++) amax = fmaxf(amax, fabsf(v[i]));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    const int ef = (int)((__float_as_uint(amax) >> 23) & 0xFF);
    int X = (amax == 0.f || ef == 0) ? -127 : ef - 127 - 2;
    X = X < -127 ? -127 : X;
    const float s = exp2i(-X);
    uint32_t codes = 0;
#pragma unroll
    for (int i = 0; i < 4; i++) codes |= cvt_e2m1x2(v[2 * i] * s, v[2 * i + 1] * s) << (8 * i);
    if (valid) {
        const long long el = gid * 8;
        const long long row = el / K;                  // e * N + n
        const int k0 = (int)(el % K);
        const long long e = row / N;
        const int n = (int)(row % N);
        const long long blk = weight_block(e, n / 128, k0 / 128, N, K);
        const int r = n % 128;
        *reinterpret_cast<uint32_t *>(w_fp4 + blk * kBlockCodeBytes + r * 64 + (k0 % 128) / 2) = codes;
        if ((gid & 3) == 0) w_scale[blk * kBlockScaleBytes + sf_byte(r, (k0 % 128) / 32)] = (uint8_t)(X + 127);
    }
    pdl_trigger();
}

cudaError_t launch_pack_fp4(const float *w, uint8_t *w_fp4, uint8_t *w_scale, int E, int N, int K, cudaStream_t st)
{
    const long long n8 = (long long)E * N * (K / 8);
    if (n8 == 0) return cudaSuccess;
    const long long blocks = (n8 + 255) / 256;
    return launch_pdl(pack_fp4_kernel, dim3((unsigned)blocks), dim3(256), 0, st, w, w_fp4, w_scale, n8, N, K);
}

// ---------------------------------------------------------------------------
// FP8 weights for the backward pass (FP4 QAT): every 128 x 128 block of the
// packed weights becomes E4M3 codes at one power-of-two block scale B (the
// block's largest 1x32 exponent - 6, at least -127), written transposed.
// One CTA per block: the scales' maximum, the codes staged in shared memory,
// then warp w writes the 16 codes of rows n = 16w .. 16w+15 of every output
// row k as a 16-byte vector (lane q takes output rows 2q and 2q + 1, the two
// codes of byte q of each code row, so the lanes read one shared 32-byte span
// and the reads broadcast).  A value code * 2^(X - B) is exact in fp32 down to
// its subnormals (it is below E4M3's half-ulp, so rounds to a signed zero,
// whenever it is smaller), and the E4M3 conversion rounds to nearest even.
// ---------------------------------------------------------------------------

// 2^e as fp32 for any e (subnormal, or zero below 2^-149)
__device__ __forceinline__ float pow2_any(int e)
{
    if (e >= -126) return __uint_as_float((uint32_t)(e + 127) << 23);
    if (e >= -149) return __uint_as_float(1u << (e + 149));
    return 0.f;
}

constexpr int kF8tRow = 64;                   // shared-memory row of 128 codes
constexpr long long kF8tBlockBytes = 128 * 128;   // one 128 x 128 block of E4M3 codes

__global__ void __launch_bounds__(256) fp4_to_fp8t_kernel(const uint8_t *__restrict__ w_fp4,
                                                          const uint8_t *__restrict__ w_scale,
                                                          uint8_t *__restrict__ w8t, uint8_t *__restrict__ s8t,
                                                          int N, int K)
{
    pdl_wait();
    __shared__ __align__(16) uint8_t codes[128 * kF8tRow];
    __shared__ __align__(16) uint8_t sc[kBlockScaleBytes];
    __shared__ int s_max[8];
    const int NB = N / 128, KB = K / 128;
    const int bk = blockIdx.x % KB, bn = (blockIdx.x / KB) % NB, e = blockIdx.x / (KB * NB);
    const long long blk = weight_block(e, bn, bk, N, K);
    const uint8_t *src = w_fp4 + blk * kBlockCodeBytes;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    // codes: 8 KB, 32 bytes per thread, into rows of kF8tRow bytes
    {
        const int r = t >> 1, half = t & 1;
        const uint4 *g = reinterpret_cast<const uint4 *>(src + r * 64 + half * 32);
        uint4 *d = reinterpret_cast<uint4 *>(codes + r * kF8tRow + half * 32);
        d[0] = __ldg(g);
        d[1] = __ldg(g + 1);
    }
    int m = -127;
    {
        const uint16_t two = __ldg(reinterpret_cast<const uint16_t *>(w_scale + blk * kBlockScaleBytes) + t);
        reinterpret_cast<uint16_t *>(sc)[t] = two;
        m = max((int)(two & 0xFF), (int)(two >> 8)) - 127;
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, off));
    if (lane == 0) s_max[warp] = m;
    __syncthreads();
    int S = s_max[0];
#pragma unroll
    for (int w = 1; w < 8; w++) S = max(S, s_max[w]);
    const int B = max(S - 6, -127);
    if (t == 0) s8t[((long long)e * KB + bk) * NB + bn] = (uint8_t)(B + 127);
    // Every 32-code sub-block (row n, sub-block j of K) shares one shift
    // X - B, so the E4M3 codes of its eight magnitudes {0, .5, 1, 1.5, 2, 3,
    // 4, 6} x 2^(X-B) are converted once into a table (the same products and
    // the same conversion as code by code); a code is then a byte select plus
    // its sign bit (E4M3 is sign-symmetric, -0 included).
    __shared__ uint2 lut[128 * 4];
    for (int i = t; i < 128 * 4; i += 256) {
        const int n = i >> 2, j = i & 3;
        const float p = pow2_any((int)sc[sf_byte(n, j)] - 127 - B);
        lut[i] = make_uint2(cvt_e4m3x2(0.f * p, 0.5f * p) | (cvt_e4m3x2(1.f * p, 1.5f * p) << 16),
                            cvt_e4m3x2(2.f * p, 3.f * p) | (cvt_e4m3x2(4.f * p, 6.f * p) << 16));
    }
    __syncthreads();
    // output rows k = 2q and 2q + 1 of the block (both codes of one byte),
    // 16 codes (16 rows n) per lane and row
    const int n0 = warp * 16;
    for (int q = lane; q < 64; q += 32) {
        const int j = q >> 4;                     // 32-element sub-block of K
        uint32_t out0[4] = {0, 0, 0, 0}, out1[4] = {0, 0, 0, 0};
#pragma unroll
        for (int u = 0; u < 16; u++) {
            const int n = n0 + u;
            const uint32_t byte = codes[n * kF8tRow + q];
            const uint2 L = lut[n * 4 + j];
            const uint32_t lo = byte & 15u, hi = byte >> 4;
            const uint32_t c0 = (__byte_perm(L.x, L.y, lo & 7u) & 0xFFu) | ((lo & 8u) << 4);
            const uint32_t c1 = (__byte_perm(L.x, L.y, hi & 7u) & 0xFFu) | ((hi & 8u) << 4);
            out0[u >> 2] |= c0 << (8 * (u & 3));
            out1[u >> 2] |= c1 << (8 * (u & 3));
        }
        uint8_t *dst = w8t + fp8t_block(e, bk, bn, K, N) * kF8tBlockBytes + (2 * q) * 128 + n0;
        *reinterpret_cast<uint4 *>(dst) = make_uint4(out0[0], out0[1], out0[2], out0[3]);
        *reinterpret_cast<uint4 *>(dst + 128) = make_uint4(out1[0], out1[1], out1[2], out1[3]);
    }
    pdl_trigger();
}

cudaError_t launch_fp4_to_fp8t(const uint8_t *w_fp4, const uint8_t *w_scale, uint8_t *w8t, uint8_t *s8t, int E, int N,
                               int K, cudaStream_t st)
{
    const long long blocks = (long long)E * (N / 128) * (K / 128);
    if (blocks == 0) return cudaSuccess;
    if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
    return launch_pdl(fp4_to_fp8t_kernel, dim3((unsigned)blocks), dim3(256), 0, st, w_fp4, w_scale, w8t, s8t, N, K);
}

// ---------------------------------------------------------------------------
// FP8 quantisation of one 128-channel group of a bf16 row by one warp:
// each lane handles 4 channels; returns the group's scale exponent e.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int quant_group_warp(const uint16_t *__restrict__ xg, uint8_t *__restrict__ qg)
{
    const int lane = threadIdx.x & 31;
    const uint2 raw = __ldg(reinterpret_cast<const uint2 *>(xg) + lane);
    float v[4] = {bf16_bits_to_f32(raw.x & 0xFFFFu), bf16_bits_to_f32(raw.x >> 16),
                  bf16_bits_to_f32(raw.y & 0xFFFFu), bf16_bits_to_f32(raw.y >> 16)};
    float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    const int e = e4m3_scale_exp(amax);
    const float s = exp2i(-e);
    const uint32_t q = cvt_e4m3x2(v[0] * s, v[1] * s) | (cvt_e4m3x2(v[2] * s, v[3] * s) << 16);
    reinterpret_cast<uint32_t *>(qg)[lane] = q;
    return e;
}

// A whole row by one warp: 8 channels per lane, so a step covers two groups
// (lanes 0-15 the first, each half reducing its own amax); the next step's
// 16-byte loads are issued before the current step is converted.
__device__ __forceinline__ void quant_row_warp(const uint16_t *__restrict__ xrow, uint8_t *__restrict__ qrow,
                                               uint8_t *__restrict__ srow, int d, int s_stride)
{
    const int lane = threadIdx.x & 31;
    const int G = d / 128;
    const int n8 = d / 8;                              // 8-channel pieces of the row
    const uint4 *src = reinterpret_cast<const uint4 *>(xrow);
    uint4 nxt = make_uint4(0, 0, 0, 0);
    if (lane < n8) nxt = __ldg(src + lane);
    for (int c = lane; c - lane < n8; c += 32) {
        const uint4 cur = nxt;
        if (c + 32 < n8) nxt = __ldg(src + c + 32);
        const uint32_t u[4] = {cur.x, cur.y, cur.z, cur.w};
        float v[8];
#pragma unroll
        for (int i = 0; i < 4; i++) {
            v[2 * i] = bf16_bits_to_f32(u[i] & 0xFFFFu);
            v[2 * i + 1] = bf16_bits_to_f32(u[i] >> 16);
        }
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < 8; i++) amax = fmaxf(amax, fabsf(v[i]));
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
    for (int g = G + lane; g < s_stride; g += 32) srow[g] = 0;
}

__global__ void __launch_bounds__(256) quantize_kernel(const uint16_t *__restrict__ x, uint8_t *__restrict__ xq,
                                                       uint8_t *__restrict__ xs, int xs_stride, int T, int d)
{
    pdl_wait();
    const int t = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    if (t >= T) return;
    quant_row_warp(x + (size_t)t * d, xq + (size_t)t * d, xs + (size_t)t * xs_stride, d, xs_stride);
    pdl_trigger();
}

cudaError_t launch_quantize(const uint16_t *x, uint8_t *xq, uint8_t *xs, int xs_stride, int T, int d,
                            cudaStream_t st)
{
    if (T == 0) return cudaSuccess;
    return launch_pdl(quantize_kernel, dim3((T + 7) / 8), dim3(256), 0, st, x, xq, xs, xs_stride, T, d);
}

// ---------------------------------------------------------------------------
// Gate logits in the fixed fp32 order: for each (t, e) and l = 0..31 a partial
// sum over channels i = l, l+32, ... (increasing i, fused multiply-adds), then
// a binary tree with offsets 16..1.  Here warp lane l IS partial sum l: a warp
// owns a TW x EW tile of (token, expert) pairs, every lane accumulates its
// channel subsequence for all of them, and the final xor-butterfly adds
// exactly the tree's pairs (each add is commutative, so every lane ends with
// the tree's total).  Chunks of CH (128 or 256) channels of x and gate_w are
// staged in shared memory through a STAGES-deep cp.async pipeline.
// ---------------------------------------------------------------------------
namespace gate {

__device__ __forceinline__ void cp_async_16_zfill(void *dst, const void *src, bool pred)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(pred ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_4_zfill(void *dst, const void *src, bool pred)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(pred ? 4 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }
} // namespace gate

template <int TW, int EW, int WT, int WE, bool VEC_W, int CH, int STAGES, bool PF = false>
__global__ void __launch_bounds__(WT *WE * 32) gate_logits_kernel(const uint16_t *__restrict__ x,
                                                                  const float *__restrict__ gate_w,
                                                                  const float *__restrict__ bias,
                                                                  float *__restrict__ z, int T, int d, int E)
{
    pdl_wait();
    using namespace gate;
    constexpr int NT = WT * WE * 32;
    constexpr int CT = TW * WT;           // tokens per CTA
    constexpr int CE = EW * WE;           // experts per CTA
    constexpr int WROW = CE + 4;          // padded gate_w row in shared memory (floats)
    constexpr int XROW = CH + 8;          // padded x row (bf16 elements)
    static_assert(CE % 4 == 0, "expert tile must be a multiple of 4");
    static_assert(CH % 32 == 0, "channel chunk must be a multiple of 32");

    extern __shared__ __align__(16) unsigned char smem_raw[];
    uint16_t *xs_ = reinterpret_cast<uint16_t *>(smem_raw);                       // [STAGES][CT][XROW]
    float *ws_ = reinterpret_cast<float *>(smem_raw + STAGES * CT * XROW * 2);     // [STAGES][CH][WROW]

    const int t0 = blockIdx.x * CT;
    const int e0 = blockIdx.y * CE;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wt = warp / WE, we = warp % WE;
    const int nch = d / CH;

    auto load_chunk = [&](int c) {
        if (c >= nch) return;
        const int st = c % STAGES;
        const int i0 = c * CH;
        uint16_t *xd = xs_ + st * CT * XROW;
        for (int q = threadIdx.x; q < CT * (CH / 8); q += NT) {
            const int r = q / (CH / 8), c8 = q % (CH / 8);
            const int t = t0 + r;
            const bool ok = t < T;
            cp_async_16_zfill(xd + r * XROW + c8 * 8, x + (size_t)(ok ? t : 0) * d + i0 + c8 * 8, ok);
        }
        float *wd = ws_ + st * CH * WROW;
        if (VEC_W) {
            for (int q = threadIdx.x; q < CH * (CE / 4); q += NT) {
                const int r = q / (CE / 4), c4 = q % (CE / 4);
                const int e = e0 + c4 * 4;
                const bool ok = e < E;
                cp_async_16_zfill(wd + r * WROW + c4 * 4, gate_w + (size_t)(i0 + r) * E + (ok ? e : 0), ok);
            }
        } else {
            for (int q = threadIdx.x; q < CH * CE; q += NT) {
                const int r = q / CE, c1 = q % CE;
                const int e = e0 + c1;
                const bool ok = e < E;
                cp_async_4_zfill(wd + r * WROW + c1, gate_w + (size_t)(i0 + r) * E + (ok ? e : 0), ok);
            }
        }
    };

    // Accumulators of adjacent experts are packed in pairs: one packed FMA
    // (two IEEE single-precision fused multiply-adds, each rounded exactly as
    // fmaf) updates both with the same x value, halving the instruction count.
    float2 acc[TW][EW / 2];
#pragma unroll
    for (int a = 0; a < TW; a++)
#pragma unroll
        for (int b = 0; b < EW / 2; b++) acc[a][b] = make_float2(0.f, 0.f);

#pragma unroll
    for (int s = 0; s < STAGES - 1; s++) {
        load_chunk(s);
        cp_async_commit();
    }
    for (int c = 0; c < nch; c++) {
        cp_async_wait<STAGES - 2>();
        __syncthreads();
        load_chunk(c + STAGES - 1);
        cp_async_commit();
        const int st = c % STAGES;
        const uint16_t *xb = xs_ + st * CT * XROW + (wt * TW) * XROW;
        const float *wb = ws_ + st * CH * WROW + we * EW;
        // operands of channel step q (this lane's channel q * 32 + lane)
        auto load_ops = [&](int q, float2 (&xv)[TW], float2 (&wv)[EW / 2]) {
            const int i = q * 32 + lane;
#pragma unroll
            for (int a = 0; a < TW; a++) {
                const float xf = bf16_bits_to_f32(xb[a * XROW + i]);
                xv[a] = make_float2(xf, xf);
            }
#pragma unroll
            for (int b = 0; b < EW; b += 4) {
                const float4 f = *reinterpret_cast<const float4 *>(wb + i * WROW + b);
                wv[b / 2] = make_float2(f.x, f.y);
                wv[b / 2 + 1] = make_float2(f.z, f.w);
            }
        };
        if constexpr (PF) {
            // next step's operands load while this step's multiply-adds issue
            float2 xv[2][TW];
            float2 wv[2][EW / 2];
            load_ops(0, xv[0], wv[0]);
#pragma unroll
            for (int q = 0; q < CH / 32; q++) {
                if (q + 1 < CH / 32) load_ops(q + 1, xv[(q + 1) & 1], wv[(q + 1) & 1]);
#pragma unroll
                for (int a = 0; a < TW; a++)
#pragma unroll
                    for (int b = 0; b < EW / 2; b++) acc[a][b] = __ffma2_rn(xv[q & 1][a], wv[q & 1][b], acc[a][b]);
            }
        } else {
#pragma unroll
            for (int q = 0; q < CH / 32; q++) {
                float2 xv[TW];
                float2 wv[EW / 2];
                load_ops(q, xv, wv);
#pragma unroll
                for (int a = 0; a < TW; a++)
#pragma unroll
                    for (int b = 0; b < EW / 2; b++) acc[a][b] = __ffma2_rn(xv[a], wv[b], acc[a][b]);
            }
        }
    }
    cp_async_wait<0>();

    float tot[TW][EW];
#pragma unroll
    for (int a = 0; a < TW; a++)
#pragma unroll
        for (int b = 0; b < EW; b++) {
            float v = (b & 1) ? acc[a][b / 2].y : acc[a][b / 2].x;
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) v = v + __shfl_xor_sync(0xffffffffu, v, off);
            tot[a][b] = v;
        }
    // every lane holds every total; lane (a*EW+b) % 32 writes pair (a, b)
#pragma unroll
    for (int a = 0; a < TW; a++)
#pragma unroll
        for (int b = 0; b < EW; b++) {
            if (((a * EW + b) & 31) != lane) continue;
            const int t = t0 + wt * TW + a, e = e0 + we * EW + b;
            if (t < T && e < E) {
                float v = tot[a][b];
                if (bias) v = v + bias[e];
                z[(size_t)t * E + e] = v;
            }
        }
    pdl_trigger();
}

template <int TW, int EW, int WT, int WE, bool VEC_W, int CH = 128, int STAGES = 4, bool PF = false>
static cudaError_t launch_gate_cfg(const uint16_t *x, const float *gate_w, const float *bias, float *z, int T, int d,
                                   int E, cudaStream_t st)
{
    constexpr int CT = TW * WT, CE = EW * WE;
    if (d % CH) return cudaErrorInvalidValue;
    const size_t smem = (size_t)STAGES * (CT * (CH + 8) * 2 + CH * (CE + 4) * 4);
    auto kern = gate_logits_kernel<TW, EW, WT, WE, VEC_W, CH, STAGES, PF>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    dim3 grid((T + CT - 1) / CT, (E + CE - 1) / CE);
    return launch_pdl(kern, grid, dim3(WT * WE * 32), smem, st, x, gate_w, bias, z, T, d, E);
}

// Small batches: the 32 lane partial sums of every logit are split over a
// cluster of four CTAs, eight each (partial l = 8 g + j in the CTA of cluster
// rank g), so a batch of a few tiles still spreads over four times as many
// CTAs, each with a quarter of the channels.  Every partial is the same
// fused multiply-add chain over its channels in order as in the kernel above.
// Lane 8 u + j runs partial 8 g + j for tokens [TW u, TW u + TW) of its warp's
// 4 TW tokens and all EW experts of its warp.  CTA 0 of the cluster then adds
// the 32 partials of each logit in the same xor-tree order (pairs 16 apart,
// then 8, 4, 2, 1), reading the other CTAs' partials from their shared memory.
// Both cluster barriers are taken unconditionally by every thread; the CTAs of
// a cluster are resident together, so neither can wait forever.
__device__ __forceinline__ void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ float ld_cluster_f32(const float *local, uint32_t rank)
{
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
    return v;
}

constexpr int kGateSplit = 4;                 // CTAs per cluster (partial-sum groups)

template <int TW, int EW, int WT, int WE, int CH, int STAGES>
__global__ void __cluster_dims__(1, 1, kGateSplit) __launch_bounds__(WT *WE * 32)
    gate_logits_split_kernel(const uint16_t *__restrict__ x, const float *__restrict__ gate_w,
                             const float *__restrict__ bias, float *__restrict__ z, int T, int d, int E)
{
    pdl_wait();
    using namespace gate;
    constexpr int L = 32 / kGateSplit;        // partials per CTA
    constexpr int NT = WT * WE * 32;
    constexpr int CT = TW * (32 / L) * WT;    // tokens per CTA
    constexpr int CE = EW * WE;               // experts per CTA
    constexpr int CC = CH / kGateSplit;       // this CTA's channels of a chunk (L of every 32)
    constexpr int XROW = CC + 8;              // padded x row (bf16 elements)
    constexpr int WROW = CE + 4;              // padded gate_w row (floats)
    static_assert(L == 8, "one 16-byte x copy per 32-channel block");
    static_assert(CE % 4 == 0 && CH % 32 == 0, "tile shape");
    static_assert(STAGES * (CT * XROW * 2 + CC * WROW * 4) >= L * CT * CE * 4, "partials fit the staging memory");

    extern __shared__ __align__(16) unsigned char smem_raw[];
    uint16_t *xs_ = reinterpret_cast<uint16_t *>(smem_raw);                       // [STAGES][CT][XROW]
    float *ws_ = reinterpret_cast<float *>(smem_raw + STAGES * CT * XROW * 2);     // [STAGES][CC][WROW]
    float *part = reinterpret_cast<float *>(smem_raw);                            // [L][CT][CE] after the loop

    const int g = blockIdx.z;                 // rank in the cluster (cluster = the grid's z extent)
    const int t0 = blockIdx.x * CT;
    const int e0 = blockIdx.y * CE;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wt = warp / WE, we = warp % WE;
    const int j = lane % L, u = lane / L;
    const int nch = d / CH;

    auto load_chunk = [&](int c) {
        if (c >= nch) return;
        const int st = c % STAGES;
        const int i0 = c * CH;
        uint16_t *xd = xs_ + st * CT * XROW;
        for (int q = threadIdx.x; q < CT * (CH / 32); q += NT) {
            const int r = q / (CH / 32), b = q % (CH / 32);
            const int t = t0 + r;
            const bool ok = t < T;
            cp_async_16_zfill(xd + r * XROW + b * L, x + (size_t)(ok ? t : 0) * d + i0 + b * 32 + g * L, ok);
        }
        float *wd = ws_ + st * CC * WROW;
        for (int q = threadIdx.x; q < CC * (CE / 4); q += NT) {
            const int r = q / (CE / 4), c4 = q % (CE / 4);
            const int ch = i0 + (r / L) * 32 + g * L + r % L;
            const int e = e0 + c4 * 4;
            const bool ok = e < E;
            cp_async_16_zfill(wd + r * WROW + c4 * 4, gate_w + (size_t)ch * E + (ok ? e : 0), ok);
        }
    };

    float2 acc[TW][EW / 2];
#pragma unroll
    for (int a = 0; a < TW; a++)
#pragma unroll
        for (int b = 0; b < EW / 2; b++) acc[a][b] = make_float2(0.f, 0.f);

#pragma unroll
    for (int s = 0; s < STAGES - 1; s++) {
        load_chunk(s);
        cp_async_commit();
    }
    const int tl0 = wt * TW * (32 / L) + u * TW;   // this lane's first token in the CTA tile
    for (int c = 0; c < nch; c++) {
        cp_async_wait<STAGES - 2>();
        __syncthreads();
        load_chunk(c + STAGES - 1);
        cp_async_commit();
        const int st = c % STAGES;
        const uint16_t *xb = xs_ + st * CT * XROW + tl0 * XROW;
        const float *wb = ws_ + st * CC * WROW + we * EW;
#pragma unroll
        for (int b = 0; b < CH / 32; b++) {
            const int i = b * L + j;             // channel 32 b + 8 g + j of the chunk
            float2 xv[TW];
            float2 wv[EW / 2];
#pragma unroll
            for (int a = 0; a < TW; a++) {
                const float xf = bf16_bits_to_f32(xb[a * XROW + i]);
                xv[a] = make_float2(xf, xf);
            }
#pragma unroll
            for (int q = 0; q < EW; q += 4) {
                const float4 f = *reinterpret_cast<const float4 *>(wb + i * WROW + q);
                wv[q / 2] = make_float2(f.x, f.y);
                wv[q / 2 + 1] = make_float2(f.z, f.w);
            }
#pragma unroll
            for (int a = 0; a < TW; a++)
#pragma unroll
                for (int q = 0; q < EW / 2; q++) acc[a][q] = __ffma2_rn(xv[a], wv[q], acc[a][q]);
        }
    }
    cp_async_wait<0>();
    __syncthreads();                          // staging memory free for the partials
#pragma unroll
    for (int a = 0; a < TW; a++)
#pragma unroll
        for (int q = 0; q < EW / 2; q++) {
            float *pp = part + ((size_t)j * CT + tl0 + a) * CE + we * EW + 2 * q;
            pp[0] = acc[a][q].x;
            pp[1] = acc[a][q].y;
        }
    cluster_sync_all();
    if (g == 0) {
        for (int o = threadIdx.x; o < CT * CE; o += NT) {
            const int tl = o / CE, el = o % CE;
            float p[32];
#pragma unroll
            for (int l = 0; l < 32; l++) p[l] = ld_cluster_f32(part + ((size_t)(l % L) * CT + tl) * CE + el, l / L);
#pragma unroll
            for (int h = 16; h >= 1; h >>= 1)
#pragma unroll
                for (int l = 0; l < h; l++) p[l] = p[l] + p[l + h];
            const int t = t0 + tl, e = e0 + el;
            if (t < T && e < E) {
                float v = p[0];
                if (bias) v = v + bias[e];
                z[(size_t)t * E + e] = v;
            }
        }
    }
    cluster_sync_all();                       // the partials stay readable until CTA 0 is done
    pdl_trigger();
}

template <int TW, int EW, int WT, int WE, int CH, int STAGES>
static cudaError_t launch_gate_split_cfg(const uint16_t *x, const float *gate_w, const float *bias, float *z, int T,
                                         int d, int E, cudaStream_t st)
{
    constexpr int CT = TW * 4 * WT, CE = EW * WE, CC = CH / kGateSplit;
    if (d % CH || E % 4) return cudaErrorInvalidValue;
    const size_t smem = (size_t)STAGES * (CT * (CC + 8) * 2 + CC * (CE + 4) * 4);
    auto kern = gate_logits_split_kernel<TW, EW, WT, WE, CH, STAGES>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    dim3 grid((T + CT - 1) / CT, (E + CE - 1) / CE, kGateSplit);
    return launch_pdl(kern, grid, dim3(WT * WE * 32), smem, st, x, gate_w, bias, z, T, d, E);
}

cudaError_t launch_gate_logits(const uint16_t *x, const float *gate_w, const float *bias, float *z, int T, int d,
                               int E, cudaStream_t st)
{
    if (T == 0) return cudaSuccess;
    // Tile shapes measured at E = 256 (all give the same bits), as (token x
    // expert) warp tiles and warps per CTA: 6 x 16 tiles, 4 x 2 warps (two
    // CTAs of 24 x 32 per SM) from 1536 tokens on (T=2048: 165 -> 135 us,
    // T=4096: 272 -> 234 us, T=16384 at d=7168: 1489 -> 1457 us against
    // 8 x 16 tiles of 6 x 2 warps); 4 x 16 tiles, 8 x 1 warps from 192 (T=512:
    // 60 -> 47 us); 4 x 8 tiles, 4 x 2 warps below.  256-channel chunks
    // (fewer block barriers) where d allows, else 128 channels.  The largest and
    // smallest shapes load each channel step's operands during the previous
    // step's multiply-adds (T=128: 24.3 -> 22.7 us, T=16384: 1453 -> 1428 us).
    // E not a multiple of 4 loads gate_w by words.  Batches whose 16 x 16 tiles
    // would leave SMs idle split every logit's partial sums over clusters of
    // four CTAs (T=40: 23 -> 17 us; E=64 at T=128: 23 -> 14 us).
    if (E % 4 == 0 && d % 256 == 0 && (long long)((T + 15) / 16) * ((E + 15) / 16) < 128)
        return launch_gate_split_cfg<2, 8, 1, 4, 256, 4>(x, gate_w, bias, z, T, d, E, st);
    if (E % 4) {
        return T >= 2048 ? launch_gate_cfg<8, 16, 4, 2, false>(x, gate_w, bias, z, T, d, E, st)
                         : launch_gate_cfg<4, 8, 4, 1, false>(x, gate_w, bias, z, T, d, E, st);
    }
    if (d % 256) {
        if (T >= 1536) return launch_gate_cfg<6, 16, 4, 2, true, 128, 4>(x, gate_w, bias, z, T, d, E, st);
        if (T >= 192) return launch_gate_cfg<4, 16, 8, 1, true, 128, 4>(x, gate_w, bias, z, T, d, E, st);
        return launch_gate_cfg<4, 8, 4, 1, true>(x, gate_w, bias, z, T, d, E, st);
    }
    if (T >= 1536) return launch_gate_cfg<6, 16, 4, 2, true, 256, 2, true>(x, gate_w, bias, z, T, d, E, st);
    if (T >= 192) return launch_gate_cfg<4, 16, 8, 1, true, 256, 3>(x, gate_w, bias, z, T, d, E, st);
    return launch_gate_cfg<4, 8, 4, 2, true, 256, 3, true>(x, gate_w, bias, z, T, d, E, st);
}

// ---------------------------------------------------------------------------
// Top-k + weights.  Selection order: larger logit first, equal logits -> lower
// expert index.  s_j = fp32(sqrt(softplus(z_j))) with softplus(z) =
// max(z, 0) + log1p(exp(-|z|)) in double; w_j = s_j / S, S the fp32 sum of
// s_j in slot order (w_j = 1/k when S == 0).
// One CTA of 8 warps per token: warp 0 selects the experts while all 8 warps
// quantise the token's 128-channel groups of x (when xq is given), so the
// groups' loads are in flight together rather than one after another.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void topk_warp(const float *__restrict__ zt, int32_t *__restrict__ idx_out,
                                          float *__restrict__ w_out, float *__restrict__ z_out, int E, int k,
                                          unsigned *status)
{
    const int lane = threadIdx.x & 31;
    float v[8];
    bool bad = false;
#pragma unroll
    for (int m = 0; m < 8; m++) {
        const int e = lane + 32 * m;
        float val = -INFINITY;
        if (e < E) {
            val = zt[e];
            if (isnan(val)) {
                bad = true;
                val = -INFINITY;
            }
        }
        v[m] = val;
    }
    // Selection on 64-bit keys: the logit's bits mapped to an unsigned order
    // (-0 taken as +0, so equal logits compare equal), then the inverted expert
    // index, so the larger key is the larger logit and, among equal logits,
    // the lower expert.  Each round is one max over the lane's keys and a
    // 5-step butterfly; the winner's owner clears its key.
    uint64_t key[8];
#pragma unroll
    for (int m = 0; m < 8; m++) {
        const int e = lane + 32 * m;
        uint64_t kk = 0;
        if (e < E) {
            const uint32_t u = __float_as_uint(v[m] + 0.0f);
            const uint32_t o = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
            kk = ((uint64_t)o << 32) | (uint32_t)(0xFFFFFFFFu - (uint32_t)e);
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
        const bool mine = (e & 31) == lane;
#pragma unroll
        for (int m = 0; m < 8; m++) key[m] = (mine && m == (e >> 5)) ? 0ull : key[m];
        if (lane == j) {
            const uint32_t o = (uint32_t)(best >> 32);
            my_z = __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o);
            my_e = e;
        }
    }
    if (bad && lane == 0) flag_status(status, kStatusBadData);
    float s = 0.f;
    if (lane < k) {
        const double zd = (double)my_z;
        const double sp = (zd > 0.0 ? zd : 0.0) + log1p(exp(-fabs(zd)));
        s = (float)sqrt(sp);
    }
    float S = 0.f;
    for (int j = 0; j < k; j++) S = S + __shfl_sync(0xffffffffu, s, j);
    if (lane < k) {
        idx_out[lane] = my_e;
        w_out[lane] = (S == 0.f) ? 1.0f / (float)k : s / S;
        if (z_out) z_out[lane] = my_z;
    }
}

constexpr int kTopkWarps = 8;

__global__ void __launch_bounds__(kTopkWarps * 32) topk_kernel(const float *__restrict__ z, int32_t *__restrict__ topk_idx,
                                                               float *__restrict__ topk_w, const uint16_t *__restrict__ x,
                                                               uint8_t *__restrict__ xq, uint8_t *__restrict__ xs,
                                                               int xs_stride, int T, int d, int E, int k,
                                                               unsigned *status, float *__restrict__ topk_z)
{
    pdl_wait();
    const int t = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp == 0)
        topk_warp(z + (size_t)t * E, topk_idx + (size_t)t * k, topk_w + (size_t)t * k,
                  topk_z ? topk_z + (size_t)t * k : nullptr, E, k, status);
    if (!xq) return;
    const uint16_t *xrow = x + (size_t)t * d;
    uint8_t *qrow = xq + (size_t)t * d;
    uint8_t *srow = xs + (size_t)t * xs_stride;
    const int G = d / 128;
    // warp 0 selects; the other warps quantise
    for (int g = warp - 1; warp > 0 && g < G; g += kTopkWarps - 1) {
        const int e = quant_group_warp(xrow + g * 128, qrow + g * 128);
        if (lane == 0) srow[g] = (uint8_t)(e + 127);
    }
    for (int g = G + threadIdx.x; g < xs_stride; g += blockDim.x) srow[g] = 0;
    pdl_trigger();
}

// Large batches: one warp per token (top-k, then that token's quantisation);
// enough tokens are in flight that the per-group latency is hidden.
__global__ void __launch_bounds__(256) topk_warp_per_token_kernel(const float *__restrict__ z,
                                                                  int32_t *__restrict__ topk_idx,
                                                                  float *__restrict__ topk_w,
                                                                  const uint16_t *__restrict__ x,
                                                                  uint8_t *__restrict__ xq, uint8_t *__restrict__ xs,
                                                                  int xs_stride, int T, int d, int E, int k,
                                                                  unsigned *status, float *__restrict__ topk_z)
{
    pdl_wait();
    const int t = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    if (t >= T) return;
    topk_warp(z + (size_t)t * E, topk_idx + (size_t)t * k, topk_w + (size_t)t * k,
              topk_z ? topk_z + (size_t)t * k : nullptr, E, k, status);
    if (xq) quant_row_warp(x + (size_t)t * d, xq + (size_t)t * d, xs + (size_t)t * xs_stride, d, xs_stride);
    pdl_trigger();
}

cudaError_t launch_topk(const float *z, int32_t *topk_idx, float *topk_w, const uint16_t *x, uint8_t *xq,
                        uint8_t *xs, int xs_stride, int T, int d, int E, int k, unsigned *status, cudaStream_t st,
                        float *topk_z)
{
    if (T == 0) return cudaSuccess;
    if (T >= 2048)
        return launch_pdl(topk_warp_per_token_kernel, dim3((T + 7) / 8), dim3(256), 0, st, z, topk_idx, topk_w, x, xq,
                          xs, xs_stride, T, d, E, k, status, topk_z);
    return launch_pdl(topk_kernel, dim3(T), dim3(kTopkWarps * 32), 0, st, z, topk_idx, topk_w, x, xq, xs, xs_stride, T,
                      d, E, k, status, topk_z);
}

// ---------------------------------------------------------------------------
// Dispatch plan (stable counting sort of the pairs by expert), no atomics on
// positions.  The pairs are cut into C contiguous chunks, one per CTA, and
// each CTA's chunk into 32 warp chunks.  A warp counts its pairs per expert
// in a private row of a shared table (match_any groups equal experts of a
// 32-pair step; each group's leader adds its size), so counting needs no
// atomics.  With C > 1 a first kernel publishes each CTA's per-expert
// counts; the scatter kernel (every CTA) turns all counts into global
// offsets, gives each warp the first free slot per expert of its chunk, then
// walks its pairs in order placing each at slot + rank among equal experts
// earlier in the step.  The result is the unique stable order.
// Up to kPlanFusedMaxPairs pairs a single kernel does it all: each of its
// CTAs (kPlanFusedChunk pairs each) counts every pair itself -- the per-expert
// totals and the pairs before its chunk -- so no CTA waits for another, and
// the scattered stores of the pairs' scale words spread over many SMs.
// ---------------------------------------------------------------------------
constexpr int kPlanWarps = 32;
constexpr int kPlanPairsPerCta = 2048;
constexpr int kPlanFusedChunk = 256;
constexpr int kPlanFusedWarps = 8;      // one 32-pair step per warp
constexpr long long kPlanFusedSmallPairs = 8192;
constexpr long long kPlanFusedMaxPairs = 32768;

// Count this CTA's pairs into the warp rows cnt[warp][e]; returns nothing,
// flags out-of-range experts (treated as expert 0 so the plan stays a bijection).
template <int NW>
__device__ __forceinline__ void plan_count_warps(const int32_t *__restrict__ topk_idx, int *cnt, long long pb,
                                                 long long pe, int E, bool *bad)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long n = pe - pb;
    const long long wchunk = (n + NW - 1) / NW;
    const long long wb = pb + warp * wchunk;
    const long long we = (wb + wchunk < pe) ? wb + wchunk : pe;
    int *my = cnt + warp * E;
    for (long long base = wb; base < we; base += 32) {
        const long long p = base + lane;
        const bool valid = p < we;
        int e = valid ? __ldg(topk_idx + p) : -1;
        if (valid && (e < 0 || e >= E)) {
            *bad = true;
            e = 0;
        }
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        if (valid && lane == __ffs(peers) - 1) my[e] += __popc(peers);
    }
}

__global__ void __launch_bounds__(kPlanWarps * 32) plan_count_kernel(const int32_t *__restrict__ topk_idx,
                                                                     int *__restrict__ cta_counts, long long P, int E,
                                                                     unsigned *status)
{
    pdl_wait();
    extern __shared__ int cnt[];                  // [kPlanWarps][E]
    for (int i = threadIdx.x; i < kPlanWarps * E; i += blockDim.x) cnt[i] = 0;
    __syncthreads();
    const long long pb = (long long)blockIdx.x * kPlanPairsPerCta;
    const long long pe = (pb + kPlanPairsPerCta < P) ? pb + kPlanPairsPerCta : P;
    bool bad = false;
    plan_count_warps<kPlanWarps>(topk_idx, cnt, pb, pe, E, &bad);
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int sum = 0;
        for (int w = 0; w < kPlanWarps; w++) sum += cnt[w * E + e];
        cta_counts[(size_t)blockIdx.x * E + e] = sum;
    }
    if (bad) flag_status(status, kStatusBadData);
    pdl_trigger();
}

// cta_counts == NULL: a single CTA covers all pairs (no count kernel needed).
template <int NW>
__global__ void __launch_bounds__(NW * 32) plan_scatter_kernel(const int32_t *__restrict__ topk_idx,
                                                                       const int *__restrict__ cta_counts,
                                                                       int32_t *__restrict__ expert_offsets,
                                                                       int32_t *__restrict__ sorted_pair,
                                                                       int32_t *__restrict__ pair_pos,
                                                                       int32_t *__restrict__ tile_prefix, long long P,
                                                                       int E, unsigned *status,
                                                                       const uint8_t *__restrict__ xs, int xs_stride,
                                                                       uint8_t *__restrict__ xs_tiles, int G4, int k,
                                                                       int tile_rows, int *__restrict__ tile_done,
                                                                       int n_tile_done, int chunk_pairs)
{
    pdl_wait();
    if (blockIdx.x == 0)
        for (int i = threadIdx.x; i < n_tile_done; i += blockDim.x) tile_done[i] = 0;
    extern __shared__ int cnt[];                  // [NW][E]
    __shared__ int tot[257];                      // per-expert total, then this CTA's first slot
    __shared__ int pre[257];                      // pairs of the expert in earlier CTAs
    __shared__ int tiles[257];
    __shared__ int goff[257];                     // expert's first slot in expert order
    __shared__ int gtp[257];                      // expert's first row tile (tile_rows pairs each)
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int C = gridDim.x;
    // several CTAs and no count kernel: every CTA counts all pairs itself
    const bool fused = C > 1 && !cta_counts;
    for (int i = threadIdx.x; i < NW * E; i += blockDim.x) cnt[i] = 0;
    for (int i = threadIdx.x; i < E; i += blockDim.x) {
        tot[i] = 0;
        pre[i] = 0;
    }
    __syncthreads();
    const long long chunk = C > 1 ? chunk_pairs : P;
    const long long pb = (long long)blockIdx.x * chunk;
    const long long pe = (pb + chunk < P) ? pb + chunk : P;
    bool bad = false;
    plan_count_warps<NW>(topk_idx, cnt, pb, pe, E, &bad);
    if (fused) {
        // per-expert totals and pairs before this chunk (order-free counts);
        // four 16-byte index loads in flight per thread
        auto count = [&](int e, long long p) {
            if (e < 0 || e >= E) e = 0;
            atomicAdd(&tot[e], 1);
            if (p < pb) atomicAdd(&pre[e], 1);
        };
        const long long nv = (reinterpret_cast<uintptr_t>(topk_idx) & 15) ? 0 : P / 4;
        const int4 *v4 = reinterpret_cast<const int4 *>(topk_idx);
        for (long long i0 = threadIdx.x; i0 < nv; i0 += 4 * (long long)blockDim.x) {
            int4 q[4];
#pragma unroll
            for (int u = 0; u < 4; u++) {
                const long long i = i0 + (long long)u * blockDim.x;
                q[u] = i < nv ? __ldg(v4 + i) : make_int4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < 4; u++) {
                const long long i = i0 + (long long)u * blockDim.x;
                if (i < nv) {
                    count(q[u].x, 4 * i);
                    count(q[u].y, 4 * i + 1);
                    count(q[u].z, 4 * i + 2);
                    count(q[u].w, 4 * i + 3);
                }
            }
        }
        for (long long p = 4 * nv + threadIdx.x; p < P; p += blockDim.x) count(__ldg(topk_idx + p), p);
    }
    __syncthreads();

    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int before = 0, total = 0;
        if (fused) {
            before = pre[e];
            total = tot[e];
        } else if (cta_counts) {
            // the other CTAs' counts of expert e, sixteen loads in flight at a
            // time (integer sums: any order gives the same totals)
            int c = 0;
            for (; c + 16 <= C; c += 16) {
                int v[16];
#pragma unroll
                for (int u = 0; u < 16; u++) v[u] = __ldg(cta_counts + (size_t)(c + u) * E + e);
#pragma unroll
                for (int u = 0; u < 16; u++) {
                    if (c + u < (int)blockIdx.x) before += v[u];
                    total += v[u];
                }
            }
            for (; c < C; c++) {
                const int v = __ldg(cta_counts + (size_t)c * E + e);
                if (c < (int)blockIdx.x) before += v;
                total += v;
            }
        } else {
            for (int w = 0; w < NW; w++) total += cnt[w * E + e];
        }
        tot[e] = total;
        pre[e] = before;
        tiles[e] = (total + tile_rows - 1) / tile_rows;
    }
    __syncthreads();
    if (warp == 0) {
        int run = 0, trun = 0;
        for (int e0 = 0; e0 < E; e0 += 32) {
            const int e = e0 + lane;
            const int c = e < E ? tot[e] : 0;
            const int tc = e < E ? tiles[e] : 0;
            int inc = c, tinc = tc;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int a = __shfl_up_sync(0xffffffffu, inc, off);
                const int b = __shfl_up_sync(0xffffffffu, tinc, off);
                if (lane >= off) {
                    inc += a;
                    tinc += b;
                }
            }
            if (e < E) {
                if (blockIdx.x == 0) {
                    expert_offsets[e] = run + inc - c;
                    if (tile_prefix) tile_prefix[e] = trun + tinc - tc;
                }
                goff[e] = run + inc - c;
                gtp[e] = trun + tinc - tc;
                tot[e] = run + inc - c + pre[e];      // this CTA's first slot for expert e
            }
            run += __shfl_sync(0xffffffffu, inc, 31);
            trun += __shfl_sync(0xffffffffu, tinc, 31);
        }
        if (lane == 0 && blockIdx.x == 0) {
            expert_offsets[E] = run;
            if (tile_prefix) tile_prefix[E] = trun;
        }
    }
    __syncthreads();
    // each warp's first slot per expert
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int run = tot[e];
        for (int w = 0; w < NW; w++) {
            const int c = cnt[w * E + e];
            cnt[w * E + e] = run;
            run += c;
        }
    }
    __syncthreads();

    const long long n = pe - pb;
    const long long wchunk = (n + NW - 1) / NW;
    const long long wb = pb + warp * wchunk;
    const long long we = (wb + wchunk < pe) ? wb + wchunk : pe;
    int *my = cnt + warp * E;
    const unsigned lt_mask = (1u << lane) - 1u;
    for (long long base = wb; base < we; base += 32) {
        const long long p = base + lane;
        const bool valid = p < we;
        int e = valid ? __ldg(topk_idx + p) : -1;
        if (valid && (e < 0 || e >= E)) e = 0;
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        int pos = 0;
        if (valid) pos = my[e] + __popc(peers & lt_mask);
        __syncwarp();
        if (valid && lane == __ffs(peers) - 1) my[e] += __popc(peers);
        __syncwarp();
        if (valid) {
            sorted_pair[pos] = (int32_t)p;
            pair_pos[p] = pos;
            if (xs_tiles) {
                // the pair's token scales into the GEMM's per-tile scale layout:
                // tile m = first tile of e + local / tile_rows, row local % tile_rows
                const int local = pos - goff[e];
                const long long m = gtp[e] + local / tile_rows;
                const int r = local % tile_rows;
                const uint32_t *src = reinterpret_cast<const uint32_t *>(xs + (size_t)(p / k) * xs_stride);
                uint8_t *dst = xs_tiles + (size_t)m * G4 * kBlockScaleBytes + sf_byte(r, 0);
                for (int g0 = 0; g0 < G4; g0 += 8) {
                    uint32_t w[8];
#pragma unroll
                    for (int u = 0; u < 8; u++) w[u] = g0 + u < G4 ? __ldg(src + g0 + u) : 0u;
#pragma unroll
                    for (int u = 0; u < 8; u++)
                        if (g0 + u < G4)
                            *reinterpret_cast<uint32_t *>(dst + (size_t)(g0 + u) * kBlockScaleBytes) = w[u];
                }
            }
        }
    }
    if (bad && !cta_counts) flag_status(status, kStatusBadData);
    pdl_trigger();
}

cudaError_t launch_plan(const int32_t *topk_idx, int32_t *expert_offsets, int32_t *sorted_pair, int32_t *pair_pos,
                        int32_t *tile_prefix, int *cta_counts, int T, int E, int k, unsigned *status, cudaStream_t st,
                        const uint8_t *xs, int xs_stride, uint8_t *xs_tiles, int d, int tile_rows, int *tile_done,
                        int n_tile_done)
{
    const int G4 = xs_tiles ? stage_groups(d) : 0;
    const long long P = (long long)T * k;
    const size_t smem = (size_t)kPlanWarps * E * sizeof(int);
    const size_t smem_small = (size_t)kPlanFusedWarps * E * sizeof(int);
    const long long C = (P + kPlanPairsPerCta - 1) / kPlanPairsPerCta;
    if (P <= kPlanFusedMaxPairs || !cta_counts) {
        // one kernel: kPlanFusedChunk pairs per CTA up to kPlanFusedMaxPairs
        // pairs; one CTA for all pairs beyond that when there is no scratch
        if (P <= kPlanFusedMaxPairs) {
            const long long CF = std::max(1LL, (P + kPlanFusedChunk - 1) / kPlanFusedChunk);
            // eight warps (one 32-pair step each, cheaper block barriers) while
            // every CTA's count of all pairs stays short; 32 beyond that
            if (P <= kPlanFusedSmallPairs)
                return launch_pdl(plan_scatter_kernel<kPlanFusedWarps>, dim3((unsigned)CF), dim3(kPlanFusedWarps * 32),
                                  smem_small, st, topk_idx, (const int *)nullptr, expert_offsets, sorted_pair,
                                  pair_pos, tile_prefix, P, E, status, xs, xs_stride, xs_tiles, G4, k, tile_rows,
                                  tile_done, n_tile_done, kPlanFusedChunk);
            return launch_pdl(plan_scatter_kernel<kPlanWarps>, dim3((unsigned)CF), dim3(kPlanWarps * 32), smem, st,
                              topk_idx, (const int *)nullptr, expert_offsets, sorted_pair, pair_pos, tile_prefix, P, E,
                              status, xs, xs_stride, xs_tiles, G4, k, tile_rows, tile_done, n_tile_done,
                              kPlanFusedChunk);
        }
        return launch_pdl(plan_scatter_kernel<kPlanWarps>, dim3(1), dim3(kPlanWarps * 32), smem, st, topk_idx,
                          (const int *)nullptr, expert_offsets, sorted_pair, pair_pos, tile_prefix, P, E, status, xs,
                          xs_stride, xs_tiles, G4, k, tile_rows, tile_done, n_tile_done, kPlanFusedChunk);
    }
    cudaError_t err = launch_pdl(plan_count_kernel, dim3((unsigned)C), dim3(kPlanWarps * 32), smem, st, topk_idx,
                                 cta_counts, P, E, status);
    if (err != cudaSuccess) return err;
    return launch_pdl(plan_scatter_kernel<kPlanWarps>, dim3((unsigned)C), dim3(kPlanWarps * 32), smem, st, topk_idx,
                      (const int *)cta_counts, expert_offsets, sorted_pair, pair_pos, tile_prefix, P, E, status, xs,
                      xs_stride, xs_tiles, G4, k, tile_rows, tile_done, n_tile_done, kPlanPairsPerCta);
}

// Scratch for the multi-CTA plan: per-CTA expert counts.
size_t plan_scratch_bytes(long long P, int E)
{
    const long long C = (P + kPlanPairsPerCta - 1) / kPlanPairsPerCta;
    return C > 1 ? (size_t)C * E * sizeof(int) : 0;
}

// ---------------------------------------------------------------------------
// Combine: out[t][c] = bf16(acc), acc = fmaf(w_j, y_j[c], acc) over slots
// j = 0..k-1 from acc = 0 -- a fixed order, no atomics.  One thread per
// (token, 8 channels).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) combine_kernel(const uint16_t *__restrict__ y,
                                                      const int32_t *__restrict__ pair_pos,
                                                      const float *__restrict__ topk_w, uint16_t *__restrict__ out,
                                                      int T, int d, int k, int out32)
{
    pdl_wait();
    // one thread per 16 channels of a token: the k slot rows are loaded up
    // front (32 bytes each), then added in slot order with fused multiply-adds
    // (weights 1 when topk_w is NULL: the backward's sum of a token's dx rows,
    // a fused multiply-add by 1 being the plain fp32 sum)
    const int per_tok = d / 16;
    const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (gid >= (long long)T * per_tok) return;
    const int t = (int)(gid / per_tok), c16 = (int)(gid % per_tok);
    uint32_t v[8][8];
    float w[8];
#pragma unroll
    for (int j = 0; j < 8; j++) {
        if (j < k) {
            w[j] = topk_w ? __ldg(topk_w + (size_t)t * k + j) : 1.0f;
            const int pos = __ldg(pair_pos + (size_t)t * k + j);
            ld_global_nc_v8(v[j], y + (size_t)pos * d + 16 * c16);
        }
    }
    float acc[16];
#pragma unroll
    for (int i = 0; i < 16; i++) acc[i] = 0.f;
#pragma unroll
    for (int j = 0; j < 8; j++) {
        if (j < k) {
#pragma unroll
            for (int i = 0; i < 8; i++) {
                acc[2 * i] = fmaf(w[j], bf16_bits_to_f32(v[j][i] & 0xFFFFu), acc[2 * i]);
                acc[2 * i + 1] = fmaf(w[j], bf16_bits_to_f32(v[j][i] >> 16), acc[2 * i + 1]);
            }
        }
    }
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 8; i++) o[i] = pack_bf16x2(acc[2 * i], acc[2 * i + 1]);
    uint16_t *dst = out + (size_t)t * d + 16 * c16;
    if (out32) {
        st_global_v8(dst, o);
    } else {                                   // out is only 16-byte aligned
        reinterpret_cast<uint4 *>(dst)[0] = make_uint4(o[0], o[1], o[2], o[3]);
        reinterpret_cast<uint4 *>(dst)[1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
    pdl_trigger();
}

// ---------------------------------------------------------------------------
// Dense dispatch copy: row pos of the expert-ordered activations is the
// quantised row of token sorted_pair[pos] / k, written only where pos falls in
// a tile of more than kDenseTileRows pairs.  One warp per token: its xq row is
// read once (32-byte vectors) and written to each of its pairs' positions that
// need it -- reading the row once per pair instead, in expert order, doubled
// the DRAM traffic (the scattered re-reads of xq do not stay in L2).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) dispatch_dense_kernel(const uint8_t *__restrict__ xq,
                                                             const int32_t *__restrict__ pair_pos,
                                                             const int32_t *__restrict__ topk_idx,
                                                             const int32_t *__restrict__ expert_offsets,
                                                             uint8_t *__restrict__ xq_sorted, int T, int d, int k)
{
    pdl_wait();
    const int t = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    if (t < T) {
        const int lane = threadIdx.x & 31;
        uint8_t *dst[8];                       // NULL: the pair's tile gathers its rows
        bool any = false;
#pragma unroll
        for (int j = 0; j < 8; j++) {
            dst[j] = nullptr;
            if (j < k) {
                const int pos = __ldg(pair_pos + (size_t)t * k + j);
                const int e = __ldg(topk_idx + (size_t)t * k + j);
                const int begin = __ldg(expert_offsets + e), count = __ldg(expert_offsets + e + 1) - begin;
                const int tile_first = (pos - begin) / kTileM * kTileM;
                if (count - tile_first > kDenseTileRows) {
                    dst[j] = xq_sorted + (size_t)pos * d;
                    any = true;
                }
            }
        }
        if (any) {
            const uint8_t *src = xq + (size_t)t * d;
            for (int i = lane; i < d / 32; i += 32) {
                uint32_t r[8];
                ld_global_nc_v8(r, src + 32 * i);
#pragma unroll
                for (int j = 0; j < 8; j++)
                    if (dst[j]) st_global_v8(dst[j] + 32 * i, r);
            }
        }
    }
    pdl_trigger();
}

cudaError_t launch_dispatch_dense(const uint8_t *xq, const int32_t *pair_pos, const int32_t *topk_idx,
                                  const int32_t *expert_offsets, uint8_t *xq_sorted, int T, int d, int k,
                                  cudaStream_t st)
{
    if (T == 0) return cudaSuccess;
    return launch_pdl(dispatch_dense_kernel, dim3((unsigned)((T + 7) / 8)), dim3(256), 0, st, xq, pair_pos, topk_idx,
                      expert_offsets, xq_sorted, T, d, k);
}

cudaError_t launch_combine(const uint16_t *y, const int32_t *pair_pos, const float *topk_w, uint16_t *out, int T,
                           int d, int k, cudaStream_t st)
{
    const long long n = (long long)T * (d / 16);
    if (n == 0) return cudaSuccess;
    const int out32 = (reinterpret_cast<uintptr_t>(out) % 32) == 0;
    return launch_pdl(combine_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, st, y, pair_pos, topk_w, out, T,
                      d, k, out32);
}

} // namespace fp4moe
