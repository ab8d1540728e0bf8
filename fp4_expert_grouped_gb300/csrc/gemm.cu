// gemm.cu -- persistent grouped GEMMs of the expert FFN on tcgen05 tensor cores.
//
// Linear-1 and linear-2 of the MoE layer ("DeepSeek-V4揭秘：细粒度专家并行隐藏通信时延，FP4量化与TileLang协同优化百万Token上下文",
// itsolotime.com/archives/32374, section 1.1; SwiGLU gate/up/down, section 1.4)
// with FP4 E2M1 expert weights carrying one UE8M0 scale per 32 K-elements
// (section 4: FP4 -> FP8 is exact, so the contraction runs as a block-scaled
// FP8 x FP4 MMA) and FP8 E4M3 activations with one power-of-two scale per
// 128 channels.  No split-K: every output element is reduced over the whole K
// by one MMA chain in a fixed order, whatever the batch (section 3.1).
//
// Tile = (expert e, 128 consecutive pair rows of e, 256 weight rows).  Tiles
// are numbered expert-major (inside an expert: weight block major, row block
// minor), and the persistent CTAs (one per SM) walk them round-robin, so at
// any moment the SMs work on a "wave" of neighbouring experts whose weight
// blocks are shared through L2, and the TMA loads of the next tiles run while
// the current tile's MMAs execute.
//
// Warp roles (192 threads):
//   warp 0      producer: TMA tile loads of A (pair rows, E4M3) and B (weights,
//               E2M1 spread to one byte per code by the copy engine) plus
//               4-byte cp.async copies of the scale factors, into a 4-stage ring
//   warp 1      tensor-memory owner and MMA issuer (one elected thread):
//               scale factors -> tensor memory (tcgen05.cp), then 4 MMAs of
//               K = 32 per stage into a 128 x 256 fp32 accumulator
//   warps 2-5   epilogue: tcgen05.ld of the accumulator, then
//               GEMM1: h = silu(g) * u, FP8 re-quantisation per 128 channels
//               GEMM2: rounding to bf16
// Every wait is bounded; on a timeout the CTA flags the status word and exits.
#include "moe_device.cuh"
#include "moe_internal.h"

namespace fp4moe {
namespace gg {

constexpr int BM = kTileM;
constexpr int BN = kTileN;
constexpr int BK = kTileK;
constexpr int STAGES = 4;
constexpr int A_STAGE = BM * BK;          // 16 KB of E4M3
constexpr int B_STAGE = BN * BK;          // 32 KB: 256 rows x 128 codes, one byte per code in shared memory
constexpr int B_HALF = B_STAGE / 2;
constexpr int SFA_STAGE = 512;            // 128 rows x 4 bytes
constexpr int SFB_STAGE = 1024;           // 256 rows x 4 bytes
constexpr int OFF_A = 0;
constexpr int OFF_B = OFF_A + STAGES * A_STAGE;
constexpr int OFF_SFA = OFF_B + STAGES * B_STAGE;
constexpr int OFF_SFB = OFF_SFA + STAGES * SFA_STAGE;
constexpr int OFF_BAR = OFF_SFB + STAGES * SFB_STAGE;
constexpr int OFF_MISC = OFF_BAR + (2 * STAGES + 2) * 8;
constexpr int OFF_PLAN = OFF_MISC + 16;
constexpr int PLAN_INTS = 260;
constexpr int SMEM_USED = OFF_PLAN + 2 * PLAN_INTS * 4;
constexpr int SMEM_BYTES = SMEM_USED + 1024;   // slack for 1024-byte alignment
constexpr int NUM_THREADS = 192;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t ACC_COL = 0;
constexpr uint32_t SFA_COL = 256;
constexpr uint32_t SFB_COL = 264;
constexpr uint32_t FULL_ARRIVALS = 1 + 32;     // expect_tx arrival + one cp.async arrival per producer lane
// Transaction bytes per stage.  The copy of packed 4-bit data spreads every
// 8-byte group of 16 codes over a 16-byte slot (codes in the low 8 bytes, the
// high 8 bytes left as they were), but the barrier's transaction count
// advances by the packed bytes: half the shared-memory footprint of B.
constexpr uint32_t STAGE_TX = A_STAGE + B_STAGE / 2;

// Instruction descriptor of the block-scaled MMA: A = E4M3 (format 0),
// B = E2M1 (format 5), both K-major, N = 256, M = 128, UE8M0 scales.
constexpr uint32_t IDESC_BASE = (0u << 7) | (5u << 10) | ((uint32_t)(BN >> 3) << 17) | (1u << 23) |
                                ((uint32_t)(BM >> 4) << 24);

static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");

struct Tile {
    int e, n_block, row0, valid;
};

__device__ __forceinline__ Tile decode_tile(long long tile, const int *s_tp, const int *s_offs, int E, int nb)
{
    int lo = 0, hi = E;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((long long)s_tp[mid] * nb <= tile) lo = mid;
        else hi = mid - 1;
    }
    Tile t;
    t.e = lo;
    const int mb = s_tp[lo + 1] - s_tp[lo];
    const long long local = tile - (long long)s_tp[lo] * nb;
    const int m_block = (int)(local % mb);
    t.n_block = (int)(local / mb);
    t.row0 = s_offs[lo] + m_block * BM;
    const int rem = s_offs[lo + 1] - t.row0;
    t.valid = rem < BM ? rem : BM;
    return t;
}

template <int MODE>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const GemmArgs g, const int out_dim)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + OFF_BAR);
    uint64_t *empty = full + STAGES;
    uint64_t *acc_full = full + 2 * STAGES;
    uint64_t *acc_empty = acc_full + 1;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + OFF_MISC + 4);
    int *s_offs = reinterpret_cast<int *>(smem + OFF_PLAN);
    int *s_tp = s_offs + PLAN_INTS;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int E = g.E;

    for (int i = threadIdx.x; i <= E; i += NUM_THREADS) {
        s_offs[i] = g.expert_offsets[i];
        s_tp[i] = g.tile_prefix[i];
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; s++) {
            mbar_init(&full[s], FULL_ARRIVALS);
            mbar_init(&empty[s], 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, 128);
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
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    const int nb = (MODE == 1) ? out_dim / 128 : out_dim / BN;
    const long long total_tiles = (long long)s_tp[E] * nb;
    const int nk = g.K / BK;
    const uint64_t tmo = g.timeout_ns;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        uint32_t stage = 0, phase = 0;
        const uint32_t sfa_base = OFF_SFA, sfb_base = OFF_SFB;
        for (long long tile = blockIdx.x; tile < total_tiles && !*abort_flag; tile += gridDim.x) {
            const Tile ti = decode_tile(tile, s_tp, s_offs, E, nb);
            int rb0, rb1;
            if (MODE == 1) {
                rb0 = ti.n_block * 128;
                rb1 = out_dim + ti.n_block * 128;
            } else {
                rb0 = ti.n_block * BN;
                rb1 = rb0 + 128;
            }
            const uint8_t *arow[4];
#pragma unroll
            for (int j = 0; j < 4; j++) {
                const int r = lane + 32 * j;
                arow[j] = g.a_scale + (size_t)(ti.row0 + (r < ti.valid ? r : 0)) * g.a_scale_stride;
            }
            const uint8_t *brow[8];
#pragma unroll
            for (int j = 0; j < 8; j++) {
                const int r = lane + 32 * (j & 3);
                const int wrow = (j < 4 ? rb0 : rb1) + r;
                brow[j] = g.b_scale + ((size_t)ti.e * g.N + wrow) * (size_t)(g.K / 32);
            }
            for (int ks = 0; ks < nk; ks++) {
                if (!mbar_wait(&empty[stage], phase ^ 1u, tmo, abort_flag)) {
                    *abort_flag = 1;
                    break;
                }
                uint8_t *sa = smem + OFF_A + stage * A_STAGE;
                uint8_t *sb = smem + OFF_B + stage * B_STAGE;
                if (lane == 0) {
                    mbar_arrive_expect_tx(&full[stage], STAGE_TX);
                    tma_load_2d(sa, &tmA, &full[stage], ks * BK, ti.row0);
                    tma_load_3d(sb, &tmB, &full[stage], ks * BK, rb0, ti.e);
                    tma_load_3d(sb + B_HALF, &tmB, &full[stage], ks * BK, rb1, ti.e);
                }
                // scale words, written straight into the layout tcgen05.cp
                // expects: row r of a 128-row block -> word (r % 32) * 4 + r / 32
                uint8_t *sfa = smem + sfa_base + stage * SFA_STAGE;
                uint8_t *sfb = smem + sfb_base + stage * SFB_STAGE;
#pragma unroll
                for (int j = 0; j < 4; j++) cp_async_4(sfa + (lane * 4 + j) * 4, arow[j] + 4 * (ks >> 2));
#pragma unroll
                for (int j = 0; j < 8; j++)
                    cp_async_4(sfb + (j >> 2) * 512 + (lane * 4 + (j & 3)) * 4, brow[j] + 4 * ks);
                cp_async_arrive_noinc(&full[stage]);
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        uint32_t stage = 0, phase = 0, acc_phase = 0;
        const uint32_t sbase = smem_u32(smem);
        for (long long tile = blockIdx.x; tile < total_tiles && !*abort_flag; tile += gridDim.x) {
            if (!mbar_wait(acc_empty, acc_phase ^ 1u, tmo, abort_flag)) {
                *abort_flag = 1;
                break;
            }
            tc_fence_after();
            bool ok = true;
            for (int ks = 0; ks < nk; ks++) {
                if (!mbar_wait(&full[stage], phase, tmo, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (lane == 0) {
                    fence_proxy_async_smem();
                    const uint32_t sfa = sbase + OFF_SFA + stage * SFA_STAGE;
                    const uint32_t sfb = sbase + OFF_SFB + stage * SFB_STAGE;
                    tc_cp_32x128b_warpx4(tmem + SFA_COL, sdesc_sf(sfa));
                    tc_cp_32x128b_warpx4(tmem + SFB_COL, sdesc_sf(sfb));
                    tc_cp_32x128b_warpx4(tmem + SFB_COL + 4, sdesc_sf(sfb + 512));
                    const uint64_t adesc = sdesc_kmajor_sw128(sbase + OFF_A + stage * A_STAGE);
                    const uint64_t bdesc = sdesc_kmajor_sw128(sbase + OFF_B + stage * B_STAGE);
#pragma unroll
                    for (int kk = 0; kk < BK / 32; kk++) {
                        // A scales: one byte per 128 channels, byte (ks % 4) of the word;
                        // B scales: one byte per 32 K-elements, byte kk of the word
                        const uint32_t idesc = IDESC_BASE | ((uint32_t)kk << 4) | ((uint32_t)(ks & 3) << 29);
                        tc_mma_mx(tmem + ACC_COL, adesc + 2 * kk, bdesc + 2 * kk, idesc, tmem + SFA_COL,
                                  tmem + SFB_COL, (ks | kk) != 0);
                    }
                    tc_commit(&empty[stage]);
                }
                __syncwarp();
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) {
                *abort_flag = 1;
                break;
            }
            if (lane == 0) tc_commit(acc_full);
            __syncwarp();
            acc_phase ^= 1u;
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;                    // tensor-memory lane quarter of this warp
        const int r = q * 32 + lane;               // accumulator row = pair row in the tile
        const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16) + ACC_COL;
        uint32_t acc_phase = 0;
        for (long long tile = blockIdx.x; tile < total_tiles && !*abort_flag; tile += gridDim.x) {
            const Tile ti = decode_tile(tile, s_tp, s_offs, E, nb);
            if (!mbar_wait(acc_full, acc_phase, tmo, abort_flag)) {
                *abort_flag = 1;
                break;
            }
            tc_fence_after();
            const size_t row = (size_t)ti.row0 + r;
            if (MODE == 1) {
                float h[128];
#pragma unroll
                for (int c = 0; c < 4; c++) {
                    uint32_t gr[32], ur[32];
                    tmem_ld32(trow + 32 * c, gr);
                    tmem_ld32(trow + 128 + 32 * c, ur);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; i++) {
                        const float gv = __uint_as_float(gr[i]);
                        const float uv = __uint_as_float(ur[i]);
                        h[32 * c + i] = gv / (1.0f + expf(-gv)) * uv;
                    }
                }
                tc_fence_before();
                mbar_arrive(acc_empty);
                float amax = 0.f;
#pragma unroll
                for (int i = 0; i < 128; i++) amax = fmaxf(amax, fabsf(h[i]));
                const int e = e4m3_scale_exp(amax);
                const float s = exp2i(-e);
                if (r < ti.valid) {
                    uint4 *dst = reinterpret_cast<uint4 *>(g.hq + row * out_dim + (size_t)ti.n_block * 128);
#pragma unroll
                    for (int v = 0; v < 8; v++) {
                        uint32_t w[4];
#pragma unroll
                        for (int u = 0; u < 4; u++) {
                            const int b = 16 * v + 4 * u;
                            w[u] = cvt_e4m3x2(h[b] * s, h[b + 1] * s) | (cvt_e4m3x2(h[b + 2] * s, h[b + 3] * s) << 16);
                        }
                        dst[v] = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                    g.hs[row * g.hs_stride + ti.n_block] = (uint8_t)(e + 127);
                }
            } else {
                uint32_t pk[128];
#pragma unroll
                for (int c = 0; c < 8; c++) {
                    uint32_t v[32];
                    tmem_ld32(trow + 32 * c, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 16; i++)
                        pk[16 * c + i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
                }
                tc_fence_before();
                mbar_arrive(acc_empty);
                if (r < ti.valid) {
                    uint4 *dst = reinterpret_cast<uint4 *>(g.y + row * out_dim + (size_t)ti.n_block * BN);
#pragma unroll
                    for (int v = 0; v < 32; v++) dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
                }
            }
            acc_phase ^= 1u;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (threadIdx.x == 0 && *abort_flag) flag_status(g.status, kStatusTimeout);
    if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
}

} // namespace gg

// ---------------------------------------------------------------------------
// Host side: tensor maps and launch
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode_fn()
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

// A operand: E4M3 rows [rows][K], 128 x 128 box, 128-byte swizzle.
static bool make_map_a(CUtensorMap *m, const uint8_t *a, long long rows, int K)
{
    EncodeTiledFn enc = get_encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)K};
    cuuint32_t box[2] = {(cuuint32_t)gg::BK, (cuuint32_t)gg::BM};
    cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(a), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// B operand: packed E2M1 [E][N][K/2]; the copy engine spreads each 8-byte
// group of 16 codes over 16 bytes of shared memory, the layout the FP8/FP6/FP4
// MMA reads.  128 x 128 box, 128-byte swizzle.
static bool make_map_b(CUtensorMap *m, const uint8_t *b, int E, int N, int K)
{
    EncodeTiledFn enc = get_encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)K, (cuuint64_t)N, (cuuint64_t)E};
    cuuint64_t strides[2] = {(cuuint64_t)K / 2, (cuuint64_t)N * (cuuint64_t)K / 2};
    cuuint32_t box[3] = {(cuuint32_t)gg::BK, 128, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 3, const_cast<uint8_t *>(b), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int MODE>
static cudaError_t launch_gemm(const GemmArgs &a, int out_dim, cudaStream_t st)
{
    if (a.P == 0) return cudaSuccess;
    CUtensorMap ma, mb;
    if (!make_map_a(&ma, a.a, a.P, a.K)) return cudaErrorInvalidValue;
    if (!make_map_b(&mb, a.b, a.E, a.N, a.K)) return cudaErrorInvalidValue;
    auto kern = gg::grouped_gemm_kernel<MODE>;
    static bool attr_set[2] = {false, false};
    if (!attr_set[MODE - 1]) {
        cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, gg::SMEM_BYTES);
        if (err != cudaSuccess) return err;
        attr_set[MODE - 1] = true;
    }
    const int nb = (MODE == 1) ? out_dim / 128 : out_dim / gg::BN;
    const long long tiles = max_row_tiles(a.P, a.E) * nb;
    const int grid = (int)(tiles < a.num_sms ? tiles : a.num_sms);
    kern<<<grid, gg::NUM_THREADS, gg::SMEM_BYTES, st>>>(ma, mb, a, out_dim);
    return cudaGetLastError();
}

cudaError_t launch_gemm1(const GemmArgs &a, int inter, cudaStream_t st) { return launch_gemm<1>(a, inter, st); }
cudaError_t launch_gemm2(const GemmArgs &a, int d, cudaStream_t st) { return launch_gemm<2>(a, d, st); }

} // namespace fp4moe
