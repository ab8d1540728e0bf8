// wgrad.cu -- the weight gradients of the MoE layer's backward pass in FP4
// quantisation-aware training, and their C ABI entry (moe_backward_w).
//
// "DeepSeek-V4揭秘：细粒度专家并行隐藏通信时延，FP4量化与TileLang协同优化百万Token上下文"
// (itsolotime.com/archives/32374), section 4: the gradients reach the FP32
// master weights unchanged (straight through the FP4 quantisation); section
// 3.2: sums in a fixed order, no atomics.  For every expert e, over its pairs
// p in the forward's expert order (ascending pair id: token order, then slot):
//   dW2[e]  = sum_p dy_p (x) h_p          [d][inter]      dy_p: E4M3 of w dout
//   dW13[e] = sum_p [dg; du]_p (x) x_p    [2 inter][d]    as the dgrad GEMMs read them
// with every operand the E4M3 code times its power-of-two scale.  The
// contraction runs over an expert's pairs, along which the operands' scales
// change (one per pair and 128 channels), so the block-scaled FP8 MMA cannot
// take them as they are: each operand is dequantised to bf16 (exact: an E4M3
// value times a power of two has at most four significant bits) and
// transposed so that the pairs are contiguous, and the GEMM runs on the bf16
// tensor cores with fp32 accumulation.
#include "moe_device.cuh"
#include "moe_internal.h"

#include <cstring>

namespace fp4moe {

namespace wg {

constexpr int BM = 128;                    // output rows per tile (MMA M)
constexpr int BN = 256;                    // output columns per tile (MMA N)
constexpr int SK = 64;                     // pairs per stage: one 128-byte bf16 row chunk
constexpr int STAGES = 4;
constexpr int A_STAGE = BM * SK * 2;       // 16 KB
constexpr int B_STAGE = BN * SK * 2;       // 32 KB
constexpr int EPI_WARPS = 8;
constexpr int NUM_THREADS = (2 + EPI_WARPS) * 32;
constexpr int MAX_E = 256;
constexpr int OFF_A = 0;
constexpr int OFF_B = OFF_A + STAGES * A_STAGE;
constexpr int OFF_BAR = OFF_B + STAGES * B_STAGE;
constexpr int OFF_MISC = OFF_BAR + (2 * STAGES + 4 + 1) * 8;   // full/empty per stage, acc full/empty x2, drain
constexpr int OFF_KB = OFF_MISC + 16;                           // kbase[E+1]
// per epilogue warp, 32 rows x 32 fp32 columns: the accumulator rows, one per
// lane, regrouped into whole 128-byte lines for the stores
constexpr int STG_WARP = 32 * 32 * 4;
constexpr int OFF_STG = (OFF_KB + (MAX_E + 1) * 4 + 127) / 128 * 128;
constexpr int SMEM_USED = OFF_STG + EPI_WARPS * STG_WARP;
constexpr int SMEM_BYTES = SMEM_USED + 1024;
constexpr uint32_t TMEM_COLS = 512;        // two 256-column accumulators (no scale factors for bf16)
// kind::f16, fp32 accumulator (bit 4), A and B bf16 (bits 7, 10), K-major, N = 256, M = 128
constexpr uint32_t IDESC = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");

} // namespace wg

// Where an operand row's codes and scales live (see wg_operand_kernel).
struct WgSource {
    const uint8_t *codes;      // E4M3 rows of `width` bytes
    const uint8_t *scale;      // per 128 channels: row-major [rows][scale_stride], or the GEMM tile layout
    int scale_stride;          // row-major stride; 0: tile layout (row tile of R rows, stage_groups(width) groups)
    int by_token;              // row index = the pair's token (xq) instead of its position
};

__device__ __forceinline__ float e4m3_value(uint32_t code)
{
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((unsigned short)code));
    return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
}

// kbase[e] = sum over e' < e of e's pair count rounded up to a multiple of SK:
// where expert e's pairs start along the transposed operands' columns (the
// padding columns hold zeros).  One CTA.
__global__ void __launch_bounds__(256) wg_kbase_kernel(const int32_t *__restrict__ expert_offsets, int32_t *kbase, int E)
{
    pdl_wait();
    if (threadIdx.x == 0) {
        int acc = 0;
        for (int e = 0; e < E; e++) {
            kbase[e] = acc;
            const int n = expert_offsets[e + 1] - expert_offsets[e];
            acc += (n + wg::SK - 1) / wg::SK * wg::SK;
        }
        kbase[E] = acc;
    }
    pdl_trigger();
}

// out[c][kcol] (bf16, row stride kp) = the dequantised operand of channel c of
// the pair at padded column kcol (zero in padding columns).  A CTA transposes
// a block of 64 columns x 256 channels through shared memory; every 64-column
// block belongs to one expert.  Each thread loads four 16-byte pieces of one
// pair's codes up front (a single piece per thread left the loads latency-bound:
// about 0.55 of HBM).
constexpr int kWgOpChannels = 256;
__global__ void __launch_bounds__(256) wg_operand_kernel(WgSource src, const int32_t *__restrict__ kbase,
                                                         const int32_t *__restrict__ expert_offsets,
                                                         const int32_t *__restrict__ tile_prefix,
                                                         const int32_t *__restrict__ sorted_pair, uint16_t *out,
                                                         long long kp, int width, int E, int k, int R)
{
    pdl_wait();
    __shared__ uint16_t tileT[kWgOpChannels][64 + 2];   // [channel][column], padded against bank conflicts
    __shared__ int s_e;
    const long long col0 = (long long)blockIdx.x * 64;
    const int c0 = blockIdx.y * kWgOpChannels;
    if (col0 >= kbase[E]) return;                 // beyond the last expert's columns: never read
    if (threadIdx.x == 0) {
        int lo = 0, hi = E - 1;                   // the expert with kbase[e] <= col0 < kbase[e+1]
        while (lo < hi) {
            const int mid = (lo + hi + 1) / 2;
            if (kbase[mid] <= col0) lo = mid;
            else hi = mid - 1;
        }
        s_e = lo;
    }
    __syncthreads();
    const int e = s_e;
    const int n_e = expert_offsets[e + 1] - expert_offsets[e];
    // load: thread t takes column i = t / 4 and channels 16 (t % 4) + 64 j .. +16, j = 0..3
    {
        const int i = threadIdx.x >> 2, cq = (threadIdx.x & 3) * 16;
        const int local = (int)(col0 - kbase[e]) + i;
        if (local < n_e) {
            const long long pos = expert_offsets[e] + local;
            const long long row = src.by_token ? sorted_pair[pos] / k : pos;
            uint4 raw[4];
#pragma unroll
            for (int j = 0; j < 4; j++)
                raw[j] = __ldg(reinterpret_cast<const uint4 *>(src.codes + row * width + c0 + cq + 64 * j));
            float sc[2];                              // the block's two 128-channel groups
#pragma unroll
            for (int h = 0; h < 2; h++) {
                const int grp = c0 / 128 + h;
                int sb;
                if (src.scale_stride) {
                    sb = src.scale[row * src.scale_stride + grp];
                } else {
                    const long long m = tile_prefix[e] + local / R;
                    sb = src.scale[(m * stage_groups(width) + grp / 4) * kBlockScaleBytes + sf_byte(local % R, grp % 4)];
                }
                sc[h] = exp2i(sb - 127);
            }
#pragma unroll
            for (int j = 0; j < 4; j++) {
                const uint32_t w[4] = {raw[j].x, raw[j].y, raw[j].z, raw[j].w};
#pragma unroll
                for (int u = 0; u < 16; u++)
                    tileT[64 * j + cq + u][i] = __bfloat16_as_ushort(
                        __float2bfloat16_rn(e4m3_value((w[u >> 2] >> (8 * (u & 3))) & 0xFFu) * sc[j >> 1]));
            }
        } else {
#pragma unroll
            for (int j = 0; j < 4; j++)
#pragma unroll
                for (int u = 0; u < 16; u++) tileT[64 * j + cq + u][i] = 0;
        }
    }
    __syncthreads();
    // store: 256 rows of 128 bytes, 16 bytes per thread and pass
#pragma unroll
    for (int pass = 0; pass < 8; pass++) {
        const int idx = threadIdx.x + pass * 256;
        const int c = idx >> 3, j = (idx & 7) * 8;
        uint32_t w[4];
#pragma unroll
        for (int u = 0; u < 4; u++) w[u] = (uint32_t)tileT[c][j + 2 * u] | ((uint32_t)tileT[c][j + 2 * u + 1] << 16);
        *reinterpret_cast<uint4 *>(out + (size_t)(c0 + c) * kp + col0 + j) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    pdl_trigger();
}

// dW[e] tile (mb, nb) = sum over e's padded columns of A^T[rows][cols] B^T[cols]:
// persistent, one CTA per SM; warp 0 loads both operands' 64-column stages by
// TMA (128-byte swizzle), one thread of warp 1 issues four bf16 MMAs of K = 16
// per stage into one of two tensor-memory accumulators, warps 2-9 store the
// finished accumulator as fp32 (two warps per 32-lane quarter, 128 columns
// each) while the next tile accumulates in the other.  Experts without pairs
// get zero tiles.  Every wait is bounded.
__global__ void __launch_bounds__(wg::NUM_THREADS, 1)
    wgrad_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const int32_t *__restrict__ kbase_g, float *__restrict__ out, int E, int Mout, int Nout,
                 unsigned *status, unsigned long long timeout_ns)
{
    using namespace wg;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + OFF_BAR);
    uint64_t *empty = full + STAGES;
    uint64_t *acc_full = empty + STAGES;          // [2]
    uint64_t *acc_empty = acc_full + 2;           // [2]
    uint64_t *drain = acc_empty + 2;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + OFF_MISC + 4);
    int *kb = reinterpret_cast<int *>(smem + OFF_KB);
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
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, TMEM_COLS);
        tmem_relinquish();
    }
    pdl_wait();                                   // the operands and kbase come from earlier work
    for (int i = threadIdx.x; i <= E; i += NUM_THREADS) kb[i] = kbase_g[i];
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const int MB = Mout / BM, NB = Nout / BN;
    const long long n_tiles = (long long)E * MB * NB;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            uint32_t stage = 0, phase = 0;
            long long armed = 0;
            for (long long tile = blockIdx.x; tile < n_tiles && !*abort_flag; tile += gridDim.x) {
                const int e = (int)(tile / (MB * NB)), rem = (int)(tile % (MB * NB));
                const int mb = rem / NB, nb = rem % NB;
                const int nk = (kb[e + 1] - kb[e]) / SK;
                for (int s = 0; s < nk; s++) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, timeout_ns, abort_flag)) {
                        *abort_flag = 1;
                        break;
                    }
                    uint64_t *fb = &full[stage];
                    armed++;
                    mbar_arrive_expect_tx(fb, A_STAGE + B_STAGE);
                    tma_load_2d(smem + OFF_A + stage * A_STAGE, &tmA, fb, kb[e] + s * SK, mb * BM);
                    tma_load_2d(smem + OFF_B + stage * B_STAGE, &tmB, fb, kb[e] + s * SK, nb * BN);
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
            for (long long tile = blockIdx.x; ok && tile < n_tiles && !*abort_flag; tile += gridDim.x) {
                const int e = (int)(tile / (MB * NB));
                const int nk = (kb[e + 1] - kb[e]) / SK;
                if (nk == 0) continue;                // a zero tile: no accumulator
                const uint32_t b = gc & 1u, use = gc >> 1;
                gc++;
                if (!mbar_wait(&acc_empty[b], (use & 1u) ^ 1u, timeout_ns, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t dcol = tmem + b * BN;
                for (int s = 0; s < nk; s++) {
                    if (!mbar_wait(&full[stage], phase, timeout_ns, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = sdesc_kmajor_sw128(sbase + OFF_A + stage * A_STAGE);
                    const uint64_t bd = sdesc_kmajor_sw128(sbase + OFF_B + stage * B_STAGE);
                    // K = 16 per MMA: 32 bytes along the 128-byte row (descriptor
                    // start address in 16-byte units)
#pragma unroll
                    for (int kk = 0; kk < 4; kk++) tc_mma_bf16(dcol, ad + 2 * kk, bd + 2 * kk, IDESC, (s | kk) != 0);
                    tc_commit(&empty[stage]);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (ok) tc_commit(&acc_full[b]);
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
        const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(half * (BN / 2));
        uint32_t gc = 0;
        for (long long tile = blockIdx.x; tile < n_tiles && !*abort_flag; tile += gridDim.x) {
            const int e = (int)(tile / (MB * NB)), rem = (int)(tile % (MB * NB));
            const int mb = rem / NB, nb = rem % NB;
            const int nk = (kb[e + 1] - kb[e]) / SK;
            if (nk == 0) {                            // an expert without pairs: zero gradient
                float *dst = out + ((size_t)e * Mout + (size_t)mb * BM + r) * Nout + (size_t)nb * BN + half * (BN / 2);
                const uint32_t z[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
                for (int i = 0; i < BN / 2; i += 8) st_global_v8(dst + i, z);
                continue;
            }
            const uint32_t b = gc & 1u, use = gc >> 1;
            gc++;
            if (!mbar_wait(&acc_full[b], use & 1u, timeout_ns, abort_flag)) {
                *abort_flag = 1;
                break;
            }
            tc_fence_after();
            uint32_t v0[32], v1[32], v2[32], v3[32];
            tmem_ld32(lane_base + b * BN, v0);
            tmem_ld32(lane_base + b * BN + 32, v1);
            tmem_ld32(lane_base + b * BN + 64, v2);
            tmem_ld32(lane_base + b * BN + 96, v3);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[b]);
            // Each lane holds one output row; stored as they are, every store
            // instruction touched 32 lines (one sector each) and the stores
            // throttled the kernel.  So each 32-column chunk goes through
            // shared memory (16-byte units XOR-swizzled by the row: no bank
            // conflicts either way) and comes back as row segments: four lanes
            // per 128-byte line, eight whole lines per store instruction.
            const uint32_t stg = smem_u32(smem + OFF_STG + (warp - 2) * STG_WARP);
            float *const dst0 = out + ((size_t)e * Mout + (size_t)mb * BM + q * 32) * Nout + (size_t)nb * BN +
                                half * (BN / 2);
            const int rs = lane >> 2, ps = lane & 3;
#pragma unroll
            for (int c = 0; c < 4; c++) {
                const uint32_t *v = c == 0 ? v0 : c == 1 ? v1 : c == 2 ? v2 : v3;
#pragma unroll
                for (int j = 0; j < 8; j++)
                    st_shared_v4(stg + lane * 128 + 16 * (j ^ (lane & 7)), v[4 * j], v[4 * j + 1], v[4 * j + 2],
                                 v[4 * j + 3]);
                __syncwarp();
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    const int rr = 8 * i + rs;
                    uint32_t w[8];
                    ld_shared_v4(stg + rr * 128 + 16 * ((2 * ps) ^ (rr & 7)), w[0], w[1], w[2], w[3]);
                    ld_shared_v4(stg + rr * 128 + 16 * ((2 * ps + 1) ^ (rr & 7)), w[4], w[5], w[6], w[7]);
                    st_global_v8(dst0 + (size_t)rr * Nout + 32 * c + 8 * ps, w);
                }
                __syncwarp();
            }
        }
    }

    pdl_trigger();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (threadIdx.x == 0 && *abort_flag) flag_status(status, kStatusTimeout);
    if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
}

namespace {

bool aligned_to(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
size_t round_up256(size_t v) { return (v + 255) / 256 * 256; }

bool wg_shape_ok(int T, int d, int inter, int E, int k)
{
    if (T < 0 || d <= 0 || inter <= 0 || E <= 0 || k <= 0) return false;
    if (d % 256 || inter % 256) return false;
    if (k > 8 || k > E || E > wg::MAX_E) return false;
    if ((long long)T * k >= (1ll << 31)) return false;
    return true;
}

// columns of the transposed operands: every expert's pairs rounded up to SK
long long wg_cols(int T, int E, int k) { return ((long long)T * k + (long long)E * (wg::SK - 1)) / wg::SK * wg::SK; }

// scratch of moe_backward_w: kbase, then two transposed bf16 operands
// (dy [d][cols] and h [inter][cols] for dW2, then, reusing the space,
// [dg; du] [2 inter][cols] and x [d][cols] for dW13)
struct WgLayout {
    size_t kbase, opA, opB, total;
    long long cols;
};
WgLayout wg_layout(int T, int d, int inter, int E, int k)
{
    WgLayout l;
    l.cols = wg_cols(T, E, k);
    l.kbase = 0;
    l.opA = round_up256((size_t)(E + 1) * 4);
    const size_t a_bytes = (size_t)(d > 2 * inter ? d : 2 * inter) * l.cols * 2;
    l.opB = l.opA + round_up256(a_bytes);
    l.total = l.opB + round_up256((size_t)d * l.cols * 2);
    return l;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn wg_encode_fn()
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

// bf16 [rows][cols] (row stride cols), a 64-column x box_rows box, 128-byte swizzle
bool make_map_bf16_rows(CUtensorMap *m, const void *base, long long rows, long long cols, int box_rows)
{
    EncodeTiledFn enc = wg_encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {(cuuint32_t)wg::SK, (cuuint32_t)box_rows};
    cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct WgPlan {
    const int32_t *offs, *tile_prefix, *sorted_pair;
    int32_t *kbase;
    long long cols;
    int E, k, R;
};

cudaError_t wg_operand(const WgPlan &pl, const WgSource &src, uint16_t *out, int width, cudaStream_t st)
{
    const dim3 grid((unsigned)(pl.cols / 64), (unsigned)(width / kWgOpChannels));
    return launch_pdl(wg_operand_kernel, grid, dim3(256), 0, st, src, (const int32_t *)pl.kbase, pl.offs,
                      pl.tile_prefix, pl.sorted_pair, out, pl.cols, width, pl.E, pl.k, pl.R);
}

cudaError_t wg_gemm(const WgPlan &pl, const uint16_t *a, int Mout, const uint16_t *b, int Nout, float *out,
                    int num_sms, unsigned *status, cudaStream_t st)
{
    CUtensorMap ma, mb;
    if (!make_map_bf16_rows(&ma, a, Mout, pl.cols, wg::BM) || !make_map_bf16_rows(&mb, b, Nout, pl.cols, wg::BN))
        return cudaErrorInvalidValue;
    cudaError_t err = cudaFuncSetAttribute(wgrad_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, wg::SMEM_BYTES);
    if (err != cudaSuccess) return err;
    const long long tiles = (long long)pl.E * (Mout / wg::BM) * (Nout / wg::BN);
    const int grid = (int)(tiles < num_sms ? tiles : num_sms);
    return launch_pdl(wgrad_kernel, dim3(grid), dim3(wg::NUM_THREADS), wg::SMEM_BYTES, st, ma, mb,
                      (const int32_t *)pl.kbase, out, pl.E, Mout, Nout, status, 2000000000ull);
}

} // namespace

// The scratch of moe_backward_h (dy codes and their scale tiles), as that
// function lays it out.
size_t bwd_h_dy_offset();
size_t bwd_h_dys_offset(int T, int d, int inter, int E, int k);

} // namespace fp4moe

using namespace fp4moe;

extern "C" size_t moe_backward_w_workspace_size(int T, int d, int inter, int E, int k)
{
    if (!wg_shape_ok(T, d, inter, E, k)) return 0;
    return wg_layout(T, d, inter, E, k).total;
}

extern "C" moe_status moe_backward_w(const void *fwd_workspace, const void *bwd_h_workspace, const uint8_t *dgu,
                                     const uint8_t *dgu_scale, float *dW13, float *dW2, void *workspace,
                                     size_t workspace_bytes, int T, int d, int inter, int E, int k, void *stream)
{
    if (!fwd_workspace || !bwd_h_workspace || !dgu || !dgu_scale || !dW13 || !dW2) return MOE_ERR_INVALID_ARG;
    if (T < 0 || d <= 0 || inter <= 0 || E <= 0 || k <= 0) return MOE_ERR_INVALID_ARG;
    if (!aligned_to(fwd_workspace, 256) || !aligned_to(bwd_h_workspace, 256) || !aligned_to(dgu, 16) ||
        !aligned_to(dW13, 32) || !aligned_to(dW2, 32))
        return MOE_ERR_INVALID_ARG;
    if (!wg_shape_ok(T, d, inter, E, k)) return MOE_ERR_UNSUPPORTED_SHAPE;
    const WgLayout L = wg_layout(T, d, inter, E, k);
    if (workspace && (!aligned_to(workspace, 256) || workspace_bytes < L.total)) return MOE_ERR_WORKSPACE;
    if (T == 0) {
        // no pairs: both gradients are zero
        cudaStream_t s = (cudaStream_t)stream;
        if (cudaMemsetAsync(dW2, 0, (size_t)E * d * inter * 4, s) != cudaSuccess ||
            cudaMemsetAsync(dW13, 0, (size_t)E * 2 * inter * d * 4, s) != cudaSuccess)
            return MOE_ERR_CUDA;
        return MOE_OK;
    }
    int num_sms = 0;
    unsigned *status = nullptr;
    moe_status st = device_query(&num_sms, &status);
    if (st != MOE_OK) return st;
    Workspace fw;
    if (!workspace_layout(Shapes{T, d, inter, E, k}, &fw)) return MOE_ERR_UNSUPPORTED_SHAPE;
    const uint8_t *fb = static_cast<const uint8_t *>(fwd_workspace);
    const uint8_t *hb = static_cast<const uint8_t *>(bwd_h_workspace);
    const long long P = (long long)T * k;

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
    WgPlan pl;
    pl.offs = reinterpret_cast<const int32_t *>(fb + fw.off[MOE_WS_EXPERT_OFFSETS]);
    pl.tile_prefix = reinterpret_cast<const int32_t *>(fb + fw.off[MOE_WS_TILE_PREFIX]);
    pl.sorted_pair = reinterpret_cast<const int32_t *>(fb + fw.off[MOE_WS_SORTED_PAIR]);
    pl.kbase = reinterpret_cast<int32_t *>(base + L.kbase);
    pl.cols = L.cols;
    pl.E = E;
    pl.k = k;
    pl.R = gemm_tile_rows(P, E);
    uint16_t *opA = reinterpret_cast<uint16_t *>(base + L.opA);
    uint16_t *opB = reinterpret_cast<uint16_t *>(base + L.opB);

    // dW2 = sum dy (x) h: A = dy^T [d][cols], B = h^T [inter][cols]
    WgSource dy{hb + bwd_h_dy_offset(), hb + bwd_h_dys_offset(T, d, inter, E, k), 0, 0};
    WgSource hq{fb + fw.off[MOE_WS_HQ], fb + fw.off[MOE_WS_HS_TILES], 0, 0};
    // dW13 = sum [dg; du] (x) x: A = [dg; du]^T [2 inter][cols], B = x^T [d][cols]
    WgSource gu{dgu, dgu_scale, 2 * inter / 128, 0};
    WgSource xq{fb + fw.off[MOE_WS_XQ], fb + fw.off[MOE_WS_XS], (int)fw.stride[MOE_WS_XS], 1};

    cudaError_t e = launch_pdl(wg_kbase_kernel, dim3(1), dim3(256), 0, s, pl.offs, pl.kbase, E);
    if (e == cudaSuccess) e = wg_operand(pl, dy, opA, d, s);
    if (e == cudaSuccess) e = wg_operand(pl, hq, opB, inter, s);
    if (e == cudaSuccess) e = wg_gemm(pl, opA, d, opB, inter, dW2, num_sms, status, s);
    if (e == cudaSuccess) e = wg_operand(pl, gu, opA, 2 * inter, s);
    if (e == cudaSuccess) e = wg_operand(pl, xq, opB, d, s);
    if (e == cudaSuccess) e = wg_gemm(pl, opA, 2 * inter, opB, d, dW13, num_sms, status, s);
    if (owned) {
        cudaError_t f = cudaFreeAsync(base, s);
        if (e == cudaSuccess) e = f;
    }
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
