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
// Warp roles (320 threads; 352 with the scale-factor warp of 16-, 32- and
// 64-row tiles):
//   warp 0      producer: GEMM1 gathers the tile's token rows of A (E4M3)
//               with four-row TMA gathers (the dispatch to expert order
//               happens here);
//               GEMM2 loads A rows (hq) as TMA boxes (only the 16-row boxes
//               holding valid rows when a tile is sparsely filled); TMA
//               loads of B (weights, E2M1 spread to one byte per code by the
//               copy engine; the weights are stored in contiguous 8 KB blocks)
//               and 512-byte bulk copies of scale factors stored in the
//               tensor cores' scale-factor order, into a 4-stage ring
//   warp 1      tensor-memory owner and MMA issuer (one elected thread):
//               A's scale factors -> tensor memory (tcgen05.cp, every fourth
//               stage), then 4 MMAs of K = 32 per stage into a 128 x 256 fp32
//               accumulator
//   warp 10     (16/32/64-row tiles) B's scale factors -> tensor memory, one copy
//               pair per stage; otherwise the MMA thread copies them
//   warps 2-9   epilogue, two warps per 32-lane quarter of tensor memory, each
//               with half of the columns: tcgen05.ld to registers, release of
//               the accumulator to the MMA warp, then
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
constexpr int A_SMALL_ROWS = 16;          // row box used when a tile holds <= SMALL_TILE_ROWS valid rows
constexpr int SMALL_TILE_ROWS = 64;
constexpr int SFA_STAGE = 512;            // 128 rows x 4 bytes
constexpr int SFB_STAGE = 1024;           // 256 rows x 4 bytes
constexpr int B_STAGE = BN * BK;          // 32 KB: 256 rows x 128 codes, one byte per code in shared memory
constexpr int PLAN_INTS = 260;
constexpr int EPI_WARPS = 8;              // two warps per 32-lane quarter of tensor memory
constexpr int SF_WARP = 2 + EPI_WARPS;    // B scale-factor copies into tensor memory (16/32/64-row tiles)

// Shared-memory layout per tile size TR (pair rows per tile).  TR = 128: a
// 4-stage ring of 48 KB stages (A 16 KB, B 32 KB).  TR = 16: A slots of 2 KB
// and a 6-stage ring (50% more weight bytes in flight); TR = 32 and 64: 4 and
// 8 KB slots, 5 stages (a sixth does not fit).  The MMA always reads 128 A
// rows (16 KB) from a slot's start; with smaller slots the rows past TR come
// from whatever follows the slot in shared memory and only feed accumulator
// rows that are discarded.  The A slots therefore come first.
template <int TR>
struct Cfg {
    static constexpr int STAGES = TR == 16 ? 6 : TR <= 64 ? 5 : 4;
    // 16/32/64-row tiles stream weights through a deep ring: a separate warp copies
    // B's scale factors into tensor memory, keeping the MMA thread's per-stage
    // issue work under the stage's MMA time (decode GEMM1 363 -> 352 us).  With
    // 128-row tiles and a 4-deep ring the extra hop's latency cost more (large
    // batches 1-3% slower), so there the MMA thread copies them itself.
    static constexpr bool SF_WARP = TR <= 64;
    // 32-lane quarters of tensor memory holding the tile's rows (the
    // epilogue warps of the others have nothing to do)
    static constexpr int EPI_Q = TR >= 128 ? 4 : (TR + 31) / 32;
    static constexpr int NUM_THREADS = (SF_WARP ? 3 + EPI_WARPS : 2 + EPI_WARPS) * 32;
    static constexpr int A_STAGE = TR * BK;
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + STAGES * A_STAGE;
    static constexpr int OFF_SFA = OFF_B + STAGES * B_STAGE;
    static constexpr int OFF_SFB = OFF_SFA + STAGES * SFA_STAGE;
    static constexpr int OFF_AMAX = OFF_SFB + STAGES * SFB_STAGE;          // [2 tile parities][2 halves][128 rows] fp32
    static constexpr int OFF_BAR = OFF_AMAX + 2 * 2 * BM * 4;
    // full, empty, sf_ready per stage; acc_full, acc_empty; one amax-exchange
    // barrier per lane quarter; two for the exit drain (MMA thread, scale warp)
    static constexpr int OFF_MISC = OFF_BAR + (3 * STAGES + 2 + 4 + 2) * 8;
    static constexpr int OFF_PLAN = OFF_MISC + 16;
    static constexpr int SMEM_USED = OFF_PLAN + 2 * PLAN_INTS * 4;
    static constexpr int SMEM_BYTES = SMEM_USED + 1024;   // slack for 1024-byte alignment
    static_assert((STAGES - 1) * A_STAGE + BM * BK <= SMEM_USED, "MMA A reads stay in shared memory");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");
};
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t ACC_COL = 0;
// Scale factors in tensor memory.  B's (8 columns) change every stage and get
// a column set per ring stage; A's (4 columns) hold the scales of four
// consecutive stages (one byte each), so they are copied once per group of
// four stages into one of two slots alternating by group.  A copy therefore
// never writes columns that MMAs still to run will read.
constexpr uint32_t SFB_COL0 = 256;
constexpr uint32_t SFB_COLS_PER_STAGE = 8;
constexpr uint32_t SFA_COL0 = SFB_COL0 + 6 * SFB_COLS_PER_STAGE;   // after the deepest ring's B columns
static_assert(SFA_COL0 + 2 * 4 <= TMEM_COLS, "tensor memory budget");
// The backward's epilogue (MODE 3) parks 96 of each thread's 128 accumulator
// columns here (96 per epilogue warp of a lane quarter), so that it can
// release the accumulator at once without holding all 128 in registers.
constexpr uint32_t STASH_COLS = 96;
constexpr uint32_t STASH_COL0 = SFA_COL0 + 2 * 4;
static_assert(STASH_COL0 + 2 * STASH_COLS <= TMEM_COLS, "tensor memory budget");
// Full-barrier arrivals: the producer's expect_tx arrival alone (every copy
// into a stage is a TMA or bulk copy counted in transaction bytes).
__host__ __device__ constexpr uint32_t full_arrivals(int) { return 1; }
// Transaction bytes of B per stage.  The copy of packed 4-bit data spreads
// every 8-byte group of 16 codes over a 16-byte slot (codes in the low 8
// bytes, the high 8 bytes left as they were), but the barrier's transaction
// count advances by the packed bytes: half the shared-memory footprint.
// MODE 3 reads FP8 weights: one byte per code in global and shared memory.
template <int MODE>
__host__ __device__ constexpr uint32_t b_stage_tx() { return MODE >= 3 ? B_STAGE : B_STAGE / 2; }

// Instruction descriptor of the block-scaled MMA: A = E4M3 (format 0), B =
// E2M1 (format 5; E4M3 for the backward's FP8 weights, MODE 3), both K-major,
// N = 256, M = 128, UE8M0 scales.
template <int MODE>
__host__ __device__ constexpr uint32_t idesc_base()
{
    return (0u << 7) | ((MODE >= 3 ? 0u : 5u) << 10) | ((uint32_t)(BN >> 3) << 17) | (1u << 23) |
           ((uint32_t)(BM >> 4) << 24);
}

// SwiGLU backward of one channel (the backward GEMM's epilogue):
//   dg = dh u s (1 + g (1 - s)),  du = dh g s,  s = 1 / (1 + e^-g),
// with the hardware exp2 and reciprocal approximations and every other
// rounding explicit, so that the epilogue's two passes get the same bits.
__device__ __forceinline__ void swiglu_backward(float dh, float g, float u, float &dg, float &du)
{
    const float s = __fdividef(1.0f, __fadd_rn(1.0f, __expf(-g)));
    dg = __fmul_rn(__fmul_rn(__fmul_rn(dh, u), s), __fmaf_rn(g, __fsub_rn(1.0f, s), 1.0f));
    du = __fmul_rn(__fmul_rn(dh, g), s);
}

struct Tile {
    int e, m_tile, n_block, row0, valid;   // m_tile: index of the row tile among all experts' tiles
};

__device__ __forceinline__ Tile decode_tile(long long tile, const int *s_tp, const int *s_offs, int E, int nb, int TR)
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
    t.m_tile = s_tp[lo] + m_block;
    t.n_block = (int)(local / mb);
    t.row0 = s_offs[lo] + m_block * TR;
    const int rem = s_offs[lo + 1] - t.row0;
    t.valid = rem < TR ? rem : TR;
    return t;
}

// DENSE (GEMM1 only): some tiles read A from the expert-ordered copy.  A
// separate instantiation keeps that path's code out of the gather-only
// producer, whose loop is sensitive to its size when the GEMM streams weights.
// TR: pair rows per tile (16 or 128).
template <int MODE, bool DENSE, int TR>
__global__ void __launch_bounds__(Cfg<TR>::NUM_THREADS, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA2,
                        const __grid_constant__ CUtensorMap tmA3,
                        const __grid_constant__ CUtensorMap tmB, const GemmArgs g, const int out_dim)
{
    using C = Cfg<TR>;
    constexpr bool SFW = C::SF_WARP;
    constexpr int NUM_THREADS = C::NUM_THREADS;
    constexpr int STAGES = C::STAGES;
    constexpr int A_STAGE = C::A_STAGE;
    constexpr int OFF_A = C::OFF_A, OFF_B = C::OFF_B, OFF_SFA = C::OFF_SFA, OFF_SFB = C::OFF_SFB;
    constexpr int OFF_AMAX = C::OFF_AMAX, OFF_BAR = C::OFF_BAR, OFF_MISC = C::OFF_MISC, OFF_PLAN = C::OFF_PLAN;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + OFF_BAR);
    uint64_t *empty = full + STAGES;
    uint64_t *sf_ready = full + 2 * STAGES;    // the stage's B scale factors are in tensor memory
    uint64_t *acc_full = full + 3 * STAGES;
    uint64_t *acc_empty = acc_full + 1;
    uint64_t *xbar = acc_empty + 1;            // [4] amax exchange of the two epilogue warps of a lane quarter
    uint64_t *drain = xbar + 4;                // [2] exit: MMA thread's, scale warp's tensor-core work done
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + OFF_MISC + 4);
    int *s_offs = reinterpret_cast<int *>(smem + OFF_PLAN);
    int *s_tp = s_offs + PLAN_INTS;
    float *s_amax = reinterpret_cast<float *>(smem + OFF_AMAX);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int E = g.E;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; s++) {
            mbar_init(&full[s], full_arrivals(MODE));
            mbar_init(&empty[s], 1);
            mbar_init(&sf_ready[s], 1);
        }
        mbar_init(acc_full, 1);
        // small tiles: only the epilogue warps of the lane quarters holding rows
        mbar_init(acc_empty, C::EPI_Q * 2);       // one arrival per epilogue warp
        for (int i = 0; i < 4; i++) mbar_init(&xbar[i], 64);
        mbar_init(&drain[0], 1);
        mbar_init(&drain[1], 1);
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmA2);
        if (DENSE) tma_prefetch_desc(&tmA3);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, TMEM_COLS);
        tmem_relinquish();
    }
    // Everything above overlaps the previous kernel's tail.  GEMM1 waits for
    // its inputs (the plan, the dispatch copy).  GEMM2 does not wait for GEMM1
    // to finish: the plan it reads was complete before GEMM1 started, and each
    // of its row tiles waits for that tile's GEMM1 epilogue warps (tile_done)
    // before loading the tile's hq rows, so GEMM2 tiles of early experts run
    // while GEMM1 finishes the last ones.
    if (MODE != 2) pdl_wait();
    for (int i = threadIdx.x; i <= E; i += NUM_THREADS) {
        s_offs[i] = g.expert_offsets[i];
        s_tp[i] = g.tile_prefix[i];
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // GEMM1: let GEMM2 launch now; its CTAs take each SM a GEMM1 CTA leaves
    if (MODE == 1) pdl_trigger();
    const uint32_t tmem = *tmem_holder;

    // GEMM2: one tile per pair of W2's 128-row blocks (the last alone when
    // d / 128 is odd)
    const int nb = (MODE == 1) ? out_dim / 128 : MODE == 2 ? weight_pairs(out_dim) : out_dim / BN;
    const long long total_tiles = (long long)s_tp[E] * nb;
    const int nk = g.K / BK;
    const uint64_t tmo = g.timeout_ns;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        // Lane 0 issues the TMA and bulk copies of each stage: two 8 KB blocks
        // of B codes (spread to one byte per code in shared memory by the 4-bit
        // copy) and the 512-byte scale-factor blocks already in the tensor
        // cores' order; for GEMM2 also the A rows (hq, expert order) as TMA
        // boxes.  For GEMM1 the warp gathers the A rows -- the tile's
        // tokens' rows of xq, i.e. the dispatch to expert order -- one TMA
        // gather of four rows per lane, only for the groups holding valid
        // rows; the copy engine applies the 128-byte swizzle.
        // (Prefetching B into L2 ahead of the ring was measured and made every
        // workload slower.)
        uint32_t stage = 0, phase = 0;
        long long armed = 0;                                // stages armed so far (exit drain)
        const int ga = stage_groups(g.K);                   // activation scale groups per tile
        bool gemm1_done = false;                            // GEMM2: all of GEMM1's tiles published
        for (long long tile = blockIdx.x; tile < total_tiles && !*abort_flag; tile += gridDim.x) {
            const Tile ti = decode_tile(tile, s_tp, s_offs, E, nb, TR);
            // The tile's two 128-row weight blocks (GEMM1: gate rows and up rows
            // of channels [128 t, 128 t + 128); GEMM2: output rows [128 t, +128)
            // and [d/2 + 128 t, +128)) are adjacent blocks of the tiled layout,
            // pair t: blocks blk + 2 ks and blk + 2 ks + 1.
            const long long blk = weight_block(ti.e, ti.n_block, 0, g.N, g.K);
            // a pair of one row block: its K blocks are consecutive, and only
            // its 512 bytes of scales are fetched (the box's second block is
            // whatever follows, or zeros past the end, and feeds discarded
            // accumulator columns)
            const bool single = MODE == 2 && weight_pair_single(ti.n_block, g.N);
            const int bstride = single ? 1 : 2;
            const uint32_t sfb_bytes = single ? kBlockScaleBytes : 2 * kBlockScaleBytes;
            const bool small = TR <= 64 || ti.valid <= SMALL_TILE_ROWS;   // 16/32/64-row tiles: always 16-row boxes
            const int a_boxes = small ? (ti.valid + A_SMALL_ROWS - 1) / A_SMALL_ROWS : 1;
            // GEMM1: a dense tile reads its rows from the expert-ordered copy, a
            // sparse one gathers them (four rows per TMA gather)
            const bool dense = DENSE && ti.valid > kDenseTileRows;
            // a dense tile of at most 32 rows loads one 32-row box of the copy,
            // a larger 128-row tile one 128-row box: one TMA request either way
            // (the requests, not the bytes, are what an A stage costs); a
            // 64-row tile of more than 32 rows two 32-row boxes (its A slot
            // holds 64 rows)
            const bool dense_big = dense && TR == 128 && ti.valid > kDenseBoxRows;
            const int dense_boxes = dense && !dense_big ? (ti.valid + kDenseBoxRows - 1) / kDenseBoxRows : 0;
            const int a_gathers = (MODE == 1 && !dense) ? (ti.valid + 3) / 4 : 0;
            const uint32_t a_tx = (MODE == 1) ? (dense_big ? (uint32_t)A_STAGE
                                                 : dense ? (uint32_t)dense_boxes * kDenseBoxRows * BK
                                                         : (uint32_t)a_gathers * 4 * BK)
                                              : (small ? a_boxes * A_SMALL_ROWS * BK : A_STAGE);
            // A's scales change every fourth stage, and only those stages' copy is
            // read (the MMA thread moves it into tensor memory there)
            const uint32_t stage_tx = a_tx + b_stage_tx<MODE>() + sfb_bytes;
            const uint8_t *a_sf = g.a_scale_tiles + (size_t)ti.m_tile * ga * SFA_STAGE;
            // GEMM2: the tile's hq rows and scales are complete once every GEMM1
            // epilogue warp that stores them (one per 128-channel block of
            // inter and per working epilogue warp) has published its part
            // (once GEMM1 has finished altogether no tile needs to wait: the
            // first look at the total usually says so, costing one load per CTA)
            if (MODE == 2 && !gemm1_done) {
                const int per_tile = C::EPI_Q * 2 * (g.K / 128);
                // (test flag: a count GEMM1 never reaches, so the wait runs out
                // before this CTA issues any copy)
                if (lane == 0) {
                    if (!g.stall_test && ld_acquire(g.all_done) >= per_tile * s_tp[E]) {
                        gemm1_done = true;
                        fence_proxy_async_global();
                    } else if (wait_counter(g.tile_done + ti.m_tile, per_tile + (g.stall_test ? 1 : 0), tmo,
                                            abort_flag)) {
                        fence_proxy_async_global();
                    } else {
                        *abort_flag = 1;
                    }
                }
                gemm1_done = __shfl_sync(0xffffffffu, gemm1_done, 0);
                if (*abort_flag) break;
            }
            // GEMM1: lane l gathers rows 4l .. 4l+3 of the tile, i.e. the xq
            // rows of their tokens; rows past the tile's last valid row repeat
            // its token, so every gathered row is in bounds
            int tok[4] = {0, 0, 0, 0};
            if (MODE == 1 && lane < a_gathers) {
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    const int r = min(4 * lane + i, ti.valid - 1);
                    tok[i] = __ldg(g.sorted_pair + ti.row0 + r) / g.k;
                }
            }
            for (int ks = 0; ks < nk; ks++) {
                if (!mbar_wait(&empty[stage], phase ^ 1u, tmo, abort_flag)) {
                    *abort_flag = 1;
                    break;
                }
                uint8_t *sa = smem + OFF_A + stage * A_STAGE;
                uint8_t *sb = smem + OFF_B + stage * B_STAGE;
                uint64_t *fb = &full[stage];
                armed++;
                if (lane == 0) {
                    mbar_arrive_expect_tx(fb, stage_tx + ((ks & 3) == 0 ? SFA_STAGE : 0));
                    if (dense_big) tma_load_2d(sa, &tmA2, fb, ks * BK, ti.row0);
                    for (int b = 0; b < dense_boxes; b++)
                        tma_load_2d(sa + b * kDenseBoxRows * BK, &tmA3, fb, ks * BK, ti.row0 + b * kDenseBoxRows);
                    if (MODE >= 2) {
                        if (small) {
                            for (int b = 0; b < a_boxes; b++)
                                tma_load_2d(sa + b * A_SMALL_ROWS * BK, &tmA2, fb, ks * BK, ti.row0 + b * A_SMALL_ROWS);
                        } else {
                            tma_load_2d(sa, &tmA, fb, ks * BK, ti.row0);
                        }
                    }
                    if (MODE >= 3)   // tiled FP8 weights: the tile's two 128-row blocks at K block ks, 32 KB
                        tma_load_2d(sb, &tmB, fb, 0, (int)(fp8t_block(ti.e, 2 * ti.n_block, ks, g.N, g.K) * 128));
                    else
                        tma_load_3d(sb, &tmB, fb, 0, 0, (int)(blk + bstride * ks));
                    if ((ks & 3) == 0)
                        bulk_copy_g2s(smem + OFF_SFA + stage * SFA_STAGE, a_sf + (ks >> 2) * SFA_STAGE, SFA_STAGE, fb);
                    uint8_t *sfb = smem + OFF_SFB + stage * SFB_STAGE;
                    bulk_copy_g2s(sfb, g.b_scale + (blk + bstride * ks) * kBlockScaleBytes, sfb_bytes, fb);
                }
                if (MODE == 1) {
                    __syncwarp();   // the stage's expect_tx is armed before any gather lands
                    if (lane < a_gathers)
                        tma_gather4(sa + lane * 4 * BK, &tmA, fb, ks * BK, tok[0], tok[1], tok[2], tok[3]);
                }
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        // Leave no copy of this CTA in flight: wait for the last use of every
        // slot armed so far (already complete unless a wait above gave up).
        // Slots below `stage` were last armed in this lap of the ring, the
        // others in the previous one.
        if (lane == 0) {
            for (int s = 0; s < STAGES; s++) {
                if (armed <= s) continue;
                mbar_wait_drain(&full[s], s < (int)stage ? phase : (phase ^ 1u), tmo);
            }
        }
        __syncwarp();
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
                // the stage's operands have landed and its B scale factors are in
                // tensor memory (the scale-factor warp waited for the former)
                if (!mbar_wait(SFW ? &sf_ready[stage] : &full[stage], phase, tmo, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t sfa = sbase + OFF_SFA + stage * SFA_STAGE;
                    const uint32_t sfa_col = tmem + SFA_COL0 + ((ks >> 2) & 1) * 4;
                    const uint32_t sfb_col = tmem + SFB_COL0 + stage * SFB_COLS_PER_STAGE;
                    // A's scales change every fourth stage; copying them here, in
                    // order with this thread's MMAs, keeps the two slots safe
                    if ((ks & 3) == 0) tc_cp_32x128b_warpx4(sfa_col, sdesc_sf(sfa));
                    if (!SFW) {
                        const uint32_t sfb = sbase + OFF_SFB + stage * SFB_STAGE;
                        tc_cp_32x128b_warpx4(sfb_col, sdesc_sf(sfb));
                        tc_cp_32x128b_warpx4(sfb_col + 4, sdesc_sf(sfb + 512));
                    }
                    const uint64_t adesc = sdesc_kmajor_sw128(sbase + OFF_A + stage * A_STAGE);
                    const uint64_t bdesc = sdesc_kmajor_sw128(sbase + OFF_B + stage * B_STAGE);
#pragma unroll
                    for (int kk = 0; kk < BK / 32; kk++) {
                        // A scales: one byte per 128 channels, byte (ks % 4) of the word;
                        // B scales: one byte per 32 K-elements, byte kk of the word
                        const uint32_t idesc = idesc_base<MODE>() | ((uint32_t)kk << 4) | ((uint32_t)(ks & 3) << 29);
                        tc_mma_mx(tmem + ACC_COL, adesc + 2 * kk, bdesc + 2 * kk, idesc, sfa_col, sfb_col,
                                  (ks | kk) != 0);
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
        // tensor memory is freed below: let this thread's MMAs and copies finish
        if (lane == 0) {
            tc_commit(&drain[0]);
            mbar_wait_drain(&drain[0], 0, tmo);
        }
        __syncwarp();
    } else if (SFW && warp == SF_WARP) {
        // ------------------------------------------------------- B scale factors
        // Same tile and stage walk as the MMA warp: once a stage is full, copy
        // its B scale factors into the stage's tensor-memory columns and signal
        // sf_ready.  This keeps the two copies per stage off the MMA thread,
        // whose per-stage issue work must stay under the stage's MMA time.  The
        // copies wait for the stage's full barrier, which completes only once
        // the MMAs of the stage's previous use have finished.
        uint32_t stage = 0, phase = 0;
        const uint32_t sbase = smem_u32(smem);
        bool ok = true;
        for (long long tile = blockIdx.x; ok && tile < total_tiles && !*abort_flag; tile += gridDim.x) {
            for (int ks = 0; ks < nk; ks++) {
                if (!mbar_wait(&full[stage], phase, tmo, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t sfb = sbase + OFF_SFB + stage * SFB_STAGE;
                    const uint32_t sfb_col = tmem + SFB_COL0 + stage * SFB_COLS_PER_STAGE;
                    tc_cp_32x128b_warpx4(sfb_col, sdesc_sf(sfb));
                    tc_cp_32x128b_warpx4(sfb_col + 4, sdesc_sf(sfb + 512));
                    tc_commit(&sf_ready[stage]);
                }
                __syncwarp();
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        if (!ok) *abort_flag = 1;
        if (lane == 0) {
            tc_commit(&drain[1]);
            mbar_wait_drain(&drain[1], 0, tmo);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        // Eight warps: warp w reads tensor-memory lanes 32 * (w % 4) ..; the two
        // warps of a lane quarter split the columns (half = 0 or 1).  Each
        // thread copies its accumulator slice to registers, releases the
        // accumulator (so the next tile's MMAs start), then finishes.
        const int q = warp & 3;
        const int half = (warp - 2) >> 2;
        const int r = q * 32 + lane;               // accumulator row = pair row in the tile
        const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16) + ACC_COL;
        uint32_t acc_phase = 0, tpar = 0;
        // small tiles have no rows in the lane quarters from EPI_Q on
        for (long long tile = blockIdx.x; q < C::EPI_Q && tile < total_tiles && !*abort_flag;
             tile += gridDim.x) {
            const Tile ti = decode_tile(tile, s_tp, s_offs, E, nb, TR);
            if (MODE == 3 && r < ti.valid) {
                // the backward's epilogue reads this row's g and u of the tile's
                // channels: start bringing them into L2 while the tile accumulates
                const float *gp = g.gu_in + ((size_t)ti.row0 + r) * (2 * (size_t)out_dim) +
                                  (size_t)ti.n_block * BN + 128 * half;
                prefetch_l2_bulk(gp, 128 * sizeof(float));
                prefetch_l2_bulk(gp + out_dim, 128 * sizeof(float));
            }
            if (!mbar_wait(acc_full, acc_phase, tmo, abort_flag)) {
                *abort_flag = 1;
                break;
            }
            tc_fence_after();
            const size_t row = (size_t)ti.row0 + r;
            if (MODE == 1) {
                // channels [64 * half, 64 * half + 64) of the tile's 128: gate
                // columns at 64 * half, up columns at 128 + 64 * half
                uint32_t g0[32], g1[32], u0[32], u1[32];
                tmem_ld32(trow + 64 * half, g0);
                tmem_ld32(trow + 64 * half + 32, g1);
                tmem_ld32(trow + 128 + 64 * half, u0);
                tmem_ld32(trow + 128 + 64 * half + 32, u1);
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(acc_empty);
                if (g.gu_out && r < ti.valid) {
                    // training: keep g and u (fp32) for the backward's SwiGLU
                    float *gd = g.gu_out + row * (2 * (size_t)out_dim) + (size_t)ti.n_block * 128 + 64 * half;
                    float *ud = gd + out_dim;
#pragma unroll
                    for (int i = 0; i < 64; i += 8) {
                        uint32_t wg[8], wu[8];
#pragma unroll
                        for (int u = 0; u < 8; u++) {
                            wg[u] = i < 32 ? g0[i + u] : g1[i - 32 + u];
                            wu[u] = i < 32 ? u0[i + u] : u1[i - 32 + u];
                        }
                        st_global_v8(gd + i, wg);
                        st_global_v8(ud + i, wu);
                    }
                }
                // SwiGLU with the hardware exp2 and reciprocal approximations
                // (a few ulp of fp32); h is rounded to E4M3 (3 mantissa bits)
                // right below, so this error is about 1e-4 of the FP8 step.
                // The accurate library exp and IEEE division, unrolled 64
                // times, made the epilogue code large enough to slow the
                // producer and MMA warps that share the SM's instruction cache.
                float h[64];
                float amax = 0.f;
#pragma unroll
                for (int i = 0; i < 32; i++) {
                    const float ga = __uint_as_float(g0[i]), gb = __uint_as_float(g1[i]);
                    h[i] = __fdividef(ga, 1.0f + __expf(-ga)) * __uint_as_float(u0[i]);
                    h[32 + i] = __fdividef(gb, 1.0f + __expf(-gb)) * __uint_as_float(u1[i]);
                    amax = fmaxf(amax, fmaxf(fabsf(h[i]), fabsf(h[32 + i])));
                }
                // the 128-channel amax spans both halves: swap partial maxima
                // through shared memory (slots alternate between tiles) and a
                // per-quarter barrier whose phase i belongs to this CTA's tile i
                float *xa = s_amax + tpar * 2 * BM;
                xa[half * BM + r] = amax;
                mbar_arrive(&xbar[q]);
                if (!mbar_wait(&xbar[q], tpar, tmo, abort_flag)) {
                    *abort_flag = 1;
                    break;
                }
                amax = fmaxf(amax, xa[(1 - half) * BM + r]);
                const int e = e4m3_scale_exp(amax);
                const float s = exp2i(-e);
                if (r < ti.valid) {
                    uint8_t *dst = g.hq + row * out_dim + (size_t)ti.n_block * 128 + 64 * half;
#pragma unroll
                    for (int v = 0; v < 2; v++) {
                        uint32_t w[8];
#pragma unroll
                        for (int u = 0; u < 8; u++) {
                            const int b = 32 * v + 4 * u;
                            w[u] = cvt_e4m3x2(h[b] * s, h[b + 1] * s) | (cvt_e4m3x2(h[b + 2] * s, h[b + 3] * s) << 16);
                        }
                        st_global_v8(dst + 32 * v, w);
                    }
                    if (half == 0)
                        g.hs_tiles[((size_t)ti.m_tile * stage_groups(out_dim) + (ti.n_block >> 2)) * SFA_STAGE +
                                   sf_byte(r, ti.n_block & 3)] = (uint8_t)(e + 127);
                }
                // this warp's rows of the tile are stored: publish them to GEMM2
                __syncwarp();
                if (lane == 0) {
                    red_release_add(g.tile_done + ti.m_tile, 1);
                    red_release_add(g.all_done, 1);
                }
            } else if (MODE == 3) {
                // Backward (QAT): the accumulator is dh for channels c0 .. c0+127
                // of the pair (half h of the tile: channels 256 n_block + 128 h).
                // SwiGLU backward with the forward's g and u:
                //   dg = dh u s (1 + g (1 - s)),  du = dh g s,  s = 1 / (1 + e^-g);
                // [dg; du] quantised to E4M3 with one power-of-two scale per 128
                // channels (the activations' rule).  The accumulator is released
                // at once: the thread's columns 32..127 are parked in spare
                // tensor-memory columns and 0..31 kept in registers, so the next
                // tile's MMAs run while this tile's g and u (prefetched into L2
                // while it accumulated) are read.  Pass 0 finds the two amaxes,
                // pass 1 recomputes and stores.
                const int I = out_dim;
                const int c0 = ti.n_block * BN + 128 * half;
                const bool live = r < ti.valid;
                const float *grow = g.gu_in + row * (2 * (size_t)I);
                const uint32_t stash = tmem + ((uint32_t)(q * 32) << 16) + STASH_COL0 + STASH_COLS * half;
                uint32_t v0[32], w[32];
#pragma unroll
                for (int c = 1; c < 4; c++) {
                    tmem_ld32(trow + 128 * half + 32 * c, w);
                    tmem_ld_wait();
                    tmem_st32(stash + 32 * (c - 1), w);
                }
                tmem_ld32(trow + 128 * half, v0);
                tmem_ld_wait();
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(acc_empty);
                // 32 channels per group: the group's g and u (eight 32-byte loads
                // per lane, issued together so that one memory round trip
                // serves the group), then its dh (group 0 from the registers,
                // the others from the parked columns).  The loads do not
                // allocate in L1: each lane reads its own row, 32 rows per warp
                // load, and caching those lines in L1 (the default for
                // read-only loads) made the whole kernel 1.8x slower at 16K
                // tokens (4.0 -> 2.26 ms), the operand pipeline starved.  Every
                // lane runs both passes (the tensor-memory loads are
                // warp-collective); lanes of rows past the tile's last pair
                // read zeros and store nothing.
                float amax_g = 0.f, amax_u = 0.f;
#pragma unroll
                for (int c = 0; c < 4; c++) {
                    uint32_t a[4][8], b[4][8];
#pragma unroll
                    for (int q8 = 0; q8 < 4; q8++) {
                        if (live) {
                            ld_global_nc_na_v8(a[q8], grow + c0 + 32 * c + 8 * q8);
                            ld_global_nc_na_v8(b[q8], grow + I + c0 + 32 * c + 8 * q8);
                        } else {
#pragma unroll
                            for (int u = 0; u < 8; u++) a[q8][u] = b[q8][u] = 0u;
                        }
                    }
                    if (c > 0) {
                        tmem_ld32(stash + 32 * (c - 1), w);
                        tmem_ld_wait();
                    }
                    const uint32_t *v = c == 0 ? v0 : w;
#pragma unroll
                    for (int q8 = 0; q8 < 4; q8++)
#pragma unroll
                        for (int u = 0; u < 8; u++) {
                            float dg, du;
                            swiglu_backward(__uint_as_float(v[8 * q8 + u]), __uint_as_float(a[q8][u]),
                                            __uint_as_float(b[q8][u]), dg, du);
                            amax_g = fmaxf(amax_g, fabsf(dg));
                            amax_u = fmaxf(amax_u, fabsf(du));
                        }
                }
                const int eg = e4m3_scale_exp(amax_g), eu = e4m3_scale_exp(amax_u);
                const float sg = exp2i(-eg), su = exp2i(-eu);
                // pass 1's loads may not be hoisted into pass 0 (the scheduler
                // would keep both passes' operands live): their addresses take a
                // zero the compiler cannot see through, the sign bit of the
                // non-negative amax
                const float *grow1 = grow + (__float_as_uint(fmaxf(amax_g, amax_u)) >> 31);
                uint8_t *qrow = g.dgu + row * (2 * (size_t)I);
                float *frow = g.dgu_f32 ? g.dgu_f32 + row * (2 * (size_t)I) : nullptr;
#pragma unroll
                for (int c = 0; c < 4; c++) {
                    uint32_t a[4][8], b[4][8];
#pragma unroll
                    for (int q8 = 0; q8 < 4; q8++) {
                        if (live) {
                            ld_global_nc_na_v8(a[q8], grow1 + c0 + 32 * c + 8 * q8);
                            ld_global_nc_na_v8(b[q8], grow1 + I + c0 + 32 * c + 8 * q8);
                        } else {
#pragma unroll
                            for (int u = 0; u < 8; u++) a[q8][u] = b[q8][u] = 0u;
                        }
                    }
                    if (c > 0) {
                        tmem_ld32(stash + 32 * (c - 1), w);
                        tmem_ld_wait();
                    }
                    const uint32_t *v = c == 0 ? v0 : w;
                    uint32_t wg[8], wu[8];               // one 32-byte sector of codes per lane each
#pragma unroll
                    for (int q8 = 0; q8 < 4; q8++)
#pragma unroll
                        for (int h4 = 0; h4 < 2; h4++) {
                            float dg[4], du[4];
#pragma unroll
                            for (int u = 0; u < 4; u++)
                                swiglu_backward(__uint_as_float(v[8 * q8 + 4 * h4 + u]),
                                                __uint_as_float(a[q8][4 * h4 + u]),
                                                __uint_as_float(b[q8][4 * h4 + u]), dg[u], du[u]);
                            wg[2 * q8 + h4] =
                                cvt_e4m3x2(dg[0] * sg, dg[1] * sg) | (cvt_e4m3x2(dg[2] * sg, dg[3] * sg) << 16);
                            wu[2 * q8 + h4] =
                                cvt_e4m3x2(du[0] * su, du[1] * su) | (cvt_e4m3x2(du[2] * su, du[3] * su) << 16);
                            if (live && frow) {
                                *reinterpret_cast<float4 *>(frow + c0 + 32 * c + 8 * q8 + 4 * h4) =
                                    make_float4(dg[0], dg[1], dg[2], dg[3]);
                                *reinterpret_cast<float4 *>(frow + I + c0 + 32 * c + 8 * q8 + 4 * h4) =
                                    make_float4(du[0], du[1], du[2], du[3]);
                            }
                        }
                    if (live) {
                        st_global_v8(qrow + c0 + 32 * c, wg);
                        st_global_v8(qrow + I + c0 + 32 * c, wu);
                    }
                }
                if (live) {
                    uint8_t *srow = g.dgu_scale + row * (2 * (size_t)I / 128);
                    srow[c0 / 128] = (uint8_t)(eg + 127);
                    srow[(I + c0) / 128] = (uint8_t)(eu + 127);
                }
            } else if (MODE == 4) {
                // Backward (QAT), dx of each pair: the accumulator holds output
                // columns 256 n_block + 128 h .. +128 (the tile's two row blocks
                // of W13^T are consecutive); rounded to bf16 like the forward's y
                uint32_t v0[32], v1[32], v2[32], v3[32];
                tmem_ld32(trow + 128 * half, v0);
                tmem_ld32(trow + 128 * half + 32, v1);
                tmem_ld32(trow + 128 * half + 64, v2);
                tmem_ld32(trow + 128 * half + 96, v3);
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(acc_empty);
                if (r < ti.valid) {
                    uint16_t *dst = g.y + row * out_dim + (size_t)ti.n_block * BN + 128 * half;
#pragma unroll
                    for (int c = 0; c < 4; c++) {
                        const uint32_t *v = c == 0 ? v0 : c == 1 ? v1 : c == 2 ? v2 : v3;
#pragma unroll
                        for (int j = 0; j < 2; j++) {
                            uint32_t w[8];
#pragma unroll
                            for (int u = 0; u < 8; u++)
                                w[u] = pack_bf16x2(__uint_as_float(v[16 * j + 2 * u]), __uint_as_float(v[16 * j + 2 * u + 1]));
                            st_global_v8(dst + 32 * c + 16 * j, w);
                        }
                    }
                }
            } else {
                uint32_t v0[32], v1[32], v2[32], v3[32];
                tmem_ld32(trow + 128 * half, v0);
                tmem_ld32(trow + 128 * half + 32, v1);
                tmem_ld32(trow + 128 * half + 64, v2);
                tmem_ld32(trow + 128 * half + 96, v3);
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(acc_empty);
                // accumulator half h holds output columns of weight block
                // n_block + h * ceil(d/256) (the tile's pair of blocks; none for
                // half 1 of a pair of one block)
                const int ob = ti.n_block + half * weight_pairs(out_dim);
                if (r < ti.valid && ob < out_dim / 128) {
                    uint16_t *dst = g.y + row * out_dim + (size_t)ob * 128;
#pragma unroll
                    for (int c = 0; c < 4; c++) {
                        const uint32_t *v = c == 0 ? v0 : c == 1 ? v1 : c == 2 ? v2 : v3;
#pragma unroll
                        for (int j = 0; j < 2; j++) {
                            uint32_t w[8];
#pragma unroll
                            for (int u = 0; u < 8; u++)
                                w[u] = pack_bf16x2(__uint_as_float(v[16 * j + 2 * u]), __uint_as_float(v[16 * j + 2 * u + 1]));
                            st_global_v8(dst + 32 * c + 16 * j, w);
                        }
                    }
                }
            }
            acc_phase ^= 1u;
            tpar ^= 1u;
        }
    }

    if (MODE >= 2) pdl_trigger();
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

// A operand: E4M3 rows [rows][K], 128-channel x box_rows box, 128-byte swizzle.
static bool make_map_a(CUtensorMap *m, const uint8_t *a, long long rows, int K, int box_rows)
{
    EncodeTiledFn enc = get_encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)K};
    cuuint32_t box[2] = {(cuuint32_t)gg::BK, (cuuint32_t)box_rows};
    cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(a), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// B operand: tiled MXFP4 codes, 128 x 128 blocks of 8 KB (row r at r * 64);
// the copy engine spreads each 8-byte group of 16 codes over 16 bytes of
// shared memory, the layout the FP8/FP6/FP4 MMA reads.  Two adjacent blocks
// (a tile's pair) per box, landing as its two 128-row halves; 128-byte
// swizzle.
static bool make_map_b(CUtensorMap *m, const uint8_t *b, long long blocks)
{
    EncodeTiledFn enc = get_encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {128, 128, (cuuint64_t)blocks};
    cuuint64_t strides[2] = {64, (cuuint64_t)kBlockCodeBytes};
    cuuint32_t box[3] = {128, 128, 2};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 3, const_cast<uint8_t *>(b), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int MODE>
static cudaError_t launch_gemm(const GemmArgs &a, int out_dim, cudaStream_t st)
{
    if (a.P == 0) return cudaSuccess;
    CUtensorMap ma, ma2, ma3, mb;
    // GEMM1 gathers single rows of xq (box one row high); GEMM2 reads
    // contiguous expert-ordered rows of hq.  The second A map: GEMM1 -- 128-row
    // boxes of the dense tiles' copy (when there is one); GEMM2 -- 16-row boxes.
    // The third: GEMM1 -- 32-row boxes of the copy.
    if (!make_map_a(&ma, a.a, a.a_rows, a.K, MODE == 1 ? 1 : gg::BM)) return cudaErrorInvalidValue;
    if (MODE == 1 && a.a_dense) {
        if (!make_map_a(&ma2, a.a_dense, a.P, a.K, gg::BM)) return cudaErrorInvalidValue;
        if (!make_map_a(&ma3, a.a_dense, a.P, a.K, kDenseBoxRows)) return cudaErrorInvalidValue;
    } else if (!make_map_a(&ma2, a.a, a.a_rows, a.K, MODE == 1 ? 1 : gg::A_SMALL_ROWS)) {
        return cudaErrorInvalidValue;
    }
    if (!make_map_b(&mb, a.b, (long long)a.E * (a.N / 128) * (a.K / 128))) return cudaErrorInvalidValue;
    const bool dense = MODE == 1 && a.a_dense;
    auto kern = gg::grouped_gemm_kernel<MODE, false, 128>;
    int smem = gg::Cfg<128>::SMEM_BYTES;
    int threads = gg::Cfg<128>::NUM_THREADS;
    if (a.tile_rows == 16) {
        if (dense) return cudaErrorInvalidValue;   // the copy exists from 16 pairs per expert on
        kern = gg::grouped_gemm_kernel<MODE, false, 16>;
        smem = gg::Cfg<16>::SMEM_BYTES;
        threads = gg::Cfg<16>::NUM_THREADS;
    } else if (a.tile_rows == 32) {
        kern = gg::grouped_gemm_kernel<MODE, false, 32>;
        smem = gg::Cfg<32>::SMEM_BYTES;
        threads = gg::Cfg<32>::NUM_THREADS;
        if constexpr (MODE == 1)
            if (dense) kern = gg::grouped_gemm_kernel<1, true, 32>;
    } else if (a.tile_rows == 64) {
        kern = gg::grouped_gemm_kernel<MODE, false, 64>;
        smem = gg::Cfg<64>::SMEM_BYTES;
        threads = gg::Cfg<64>::NUM_THREADS;
        if constexpr (MODE == 1)
            if (dense) kern = gg::grouped_gemm_kernel<1, true, 64>;
    } else if (a.tile_rows == 128) {
        if constexpr (MODE == 1)
            if (dense) kern = gg::grouped_gemm_kernel<1, true, 128>;
    } else {
        return cudaErrorInvalidValue;
    }
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    const int nb = (MODE == 1) ? out_dim / 128 : weight_pairs(out_dim);
    const long long tiles = max_row_tiles(a.P, a.E, a.tile_rows) * nb;
    const int grid = (int)(tiles < a.num_sms ? tiles : a.num_sms);
    if (!(MODE == 1 && a.a_dense)) ma3 = ma2;   // unused
    return launch_pdl(kern, dim3(grid), dim3(threads), smem, st, ma, ma2, ma3, mb, a, out_dim);
}

// FP8 weight rows [rows][K] (the backward's transposed weights), a 128-byte x
// 256-row box, 128-byte swizzle
// The tiled FP8 weights of moe_fp4_to_fp8t as rows of 128 bytes (every block
// row); a box is 256 of them: two neighbouring blocks, 128-byte swizzle.
static bool make_map_fp8_tiled(CUtensorMap *m, const uint8_t *b, long long rows)
{
    EncodeTiledFn enc = get_encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)gg::BK, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)gg::BK};
    cuuint32_t box[2] = {(cuuint32_t)gg::BK, (cuuint32_t)gg::BN};
    cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(b), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The backward's GEMMs on the tiled FP8 weights: MODE 3 (dh = W2^T dy with the
// SwiGLU backward, out_dim = inter) and MODE 4 (dx of each pair = W13^T [dg; du],
// out_dim = d).
template <int MODE>
static cudaError_t launch_gemm_fp8b(const GemmArgs &a, int out_dim, cudaStream_t st)
{
    if (a.P == 0) return cudaSuccess;
    CUtensorMap ma, ma2, mb;
    if (!make_map_a(&ma, a.a, a.a_rows, a.K, gg::BM) || !make_map_a(&ma2, a.a, a.a_rows, a.K, gg::A_SMALL_ROWS) ||
        !make_map_fp8_tiled(&mb, a.b, (long long)a.E * a.N * (a.K / 128)))
        return cudaErrorInvalidValue;
    auto kern = gg::grouped_gemm_kernel<MODE, false, 128>;
    int smem = gg::Cfg<128>::SMEM_BYTES, threads = gg::Cfg<128>::NUM_THREADS;
    if (a.tile_rows == 16) {
        kern = gg::grouped_gemm_kernel<MODE, false, 16>;
        smem = gg::Cfg<16>::SMEM_BYTES;
        threads = gg::Cfg<16>::NUM_THREADS;
    } else if (a.tile_rows == 32) {
        kern = gg::grouped_gemm_kernel<MODE, false, 32>;
        smem = gg::Cfg<32>::SMEM_BYTES;
        threads = gg::Cfg<32>::NUM_THREADS;
    } else if (a.tile_rows == 64) {
        kern = gg::grouped_gemm_kernel<MODE, false, 64>;
        smem = gg::Cfg<64>::SMEM_BYTES;
        threads = gg::Cfg<64>::NUM_THREADS;
    } else if (a.tile_rows != 128) {
        return cudaErrorInvalidValue;
    }
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    const long long tiles = max_row_tiles(a.P, a.E, a.tile_rows) * (out_dim / gg::BN);
    const int grid = (int)(tiles < a.num_sms ? tiles : a.num_sms);
    return launch_pdl(kern, dim3(grid), dim3(threads), smem, st, ma, ma2, ma2, mb, a, out_dim);
}

cudaError_t launch_gemm_dgrad_h(const GemmArgs &a, int inter, cudaStream_t st) { return launch_gemm_fp8b<3>(a, inter, st); }
cudaError_t launch_gemm_dgrad_x(const GemmArgs &a, int d, cudaStream_t st) { return launch_gemm_fp8b<4>(a, d, st); }

cudaError_t launch_gemm1(const GemmArgs &a, int inter, cudaStream_t st) { return launch_gemm<1>(a, inter, st); }
cudaError_t launch_gemm2(const GemmArgs &a, int d, cudaStream_t st) { return launch_gemm<2>(a, d, st); }

} // namespace fp4moe
