// api.cu -- the C ABI of libfp4moe.so (declared in include/fp4moe.h).
//
// Host side only: argument checks (all before anything is enqueued), the
// workspace layout, the launch sequence of the layer forward on the caller's
// stream, and the device status word that kernels raise on a bounded-wait
// timeout or on bad data.
#include "fp4moe.h"
#include "moe_internal.h"
#include "moe_device.cuh"

#include <cstdlib>
#include <cstring>
#include <mutex>

namespace fp4moe {

__device__ unsigned g_status_word;

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    bool init = false;
    bool supported = false;
    int num_sms = 0;
    unsigned *status = nullptr;     // device address of g_status_word
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

moe_status device_info(DeviceInfo **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_dev_mu);
    DeviceInfo &di = g_dev[dev];
    if (!di.init) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return MOE_ERR_CUDA;
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return MOE_ERR_CUDA;
        di.supported = (major == 10 && minor == 3);
        di.num_sms = sms;
        di.status = static_cast<unsigned *>(p);
        di.init = true;
    }
    *out = &di;
    return di.supported ? MOE_OK : MOE_ERR_UNSUPPORTED_DEVICE;
}

unsigned long long timeout_ns()
{
    static unsigned long long v = 0;
    if (v == 0) {
        unsigned long long ms = 2000;
        if (const char *s = std::getenv("FP4MOE_TIMEOUT_MS")) {
            char *end = nullptr;
            unsigned long long t = std::strtoull(s, &end, 10);
            if (end != s && t > 0) ms = t;
        }
        v = ms * 1000000ull;
    }
    return v;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool layer_shape_ok(int T, int d, int inter, int E, int k)
{
    if (T < 0 || d <= 0 || inter <= 0 || E <= 0 || k <= 0) return false;
    if (d % 128 || inter % 128) return false;
    if (k > 8 || k > E || E > 256) return false;
    if ((long long)T * k >= (1ll << 31)) return false;
    return true;
}

} // namespace

moe_status device_query(int *num_sms, unsigned **status)
{
    DeviceInfo *di;
    moe_status st = device_info(&di);
    if (st != MOE_OK) return st;
    *num_sms = di->num_sms;
    *status = di->status;
    return MOE_OK;
}

bool workspace_layout(const Shapes &s, Workspace *ws)
{
    if (!layer_shape_ok(s.T, s.d, s.inter, s.E, s.k)) return false;
    const size_t T = s.T, d = s.d, I = s.inter, E = s.E, k = s.k, P = T * k;
    const size_t xs_stride = scale_row_stride(s.d);
    const size_t tiles = (size_t)max_row_tiles((long long)P, s.E, gemm_tile_rows((long long)P, s.E));
    const size_t xs_tiles = tiles * stage_groups(s.d) * kBlockScaleBytes;
    const size_t hs_tiles = tiles * stage_groups(s.inter) * kBlockScaleBytes;
    size_t bytes[MOE_WS_COUNT], stride[MOE_WS_COUNT];
    bytes[MOE_WS_XQ] = T * d;                stride[MOE_WS_XQ] = d;
    bytes[MOE_WS_XS] = T * xs_stride;        stride[MOE_WS_XS] = xs_stride;
    bytes[MOE_WS_LOGITS] = T * E * 4;        stride[MOE_WS_LOGITS] = E * 4;
    bytes[MOE_WS_TOPK_IDX] = P * 4;          stride[MOE_WS_TOPK_IDX] = k * 4;
    bytes[MOE_WS_TOPK_W] = P * 4;            stride[MOE_WS_TOPK_W] = k * 4;
    bytes[MOE_WS_EXPERT_OFFSETS] = (E + 1) * 4; stride[MOE_WS_EXPERT_OFFSETS] = 4;
    bytes[MOE_WS_SORTED_PAIR] = P * 4;       stride[MOE_WS_SORTED_PAIR] = 4;
    bytes[MOE_WS_PAIR_POS] = P * 4;          stride[MOE_WS_PAIR_POS] = 4;
    bytes[MOE_WS_TILE_PREFIX] = (E + 1) * 4; stride[MOE_WS_TILE_PREFIX] = 4;
    bytes[MOE_WS_HQ] = P * I;                stride[MOE_WS_HQ] = I;
    bytes[MOE_WS_HS_TILES] = hs_tiles;       stride[MOE_WS_HS_TILES] = stage_groups(s.inter) * kBlockScaleBytes;
    bytes[MOE_WS_Y] = P * d * 2;             stride[MOE_WS_Y] = d * 2;
    bytes[MOE_WS_XQ_SORTED] = P * d;         stride[MOE_WS_XQ_SORTED] = d;
    bytes[MOE_WS_XS_TILES] = xs_tiles;       stride[MOE_WS_XS_TILES] = stage_groups(s.d) * kBlockScaleBytes;
    bytes[MOE_WS_PLAN_COUNTS] = plan_scratch_bytes((long long)P, s.E);
    stride[MOE_WS_PLAN_COUNTS] = (size_t)s.E * 4;
    bytes[MOE_WS_TILE_DONE] = (tiles + 1) * 4; stride[MOE_WS_TILE_DONE] = 4;
    bytes[MOE_WS_TOPK_Z] = P * 4;            stride[MOE_WS_TOPK_Z] = k * 4;
    const bool tc = gate_uses_tc(s.T, s.d, s.E);
    bytes[MOE_WS_GATE_WT] = tc ? E * d * 4 : 0;   stride[MOE_WS_GATE_WT] = d * 4;
    bytes[MOE_WS_GATE_WHI] = tc ? E * d * 2 : 0;  stride[MOE_WS_GATE_WHI] = d * 2;
    bytes[MOE_WS_GATE_WLO] = tc ? E * d * 2 : 0;  stride[MOE_WS_GATE_WLO] = d * 2;
    bytes[MOE_WS_GATE_WNORM] = tc ? E * 4 : 0;    stride[MOE_WS_GATE_WNORM] = 4;
    bytes[MOE_WS_GATE_NCAND] = tc ? T * 4 : 0;    stride[MOE_WS_GATE_NCAND] = 4;
    size_t off = 0;
    for (int i = 0; i < MOE_WS_COUNT; i++) {
        ws->off[i] = off;
        ws->stride[i] = stride[i];
        off = round_up(off + bytes[i], 256);
    }
    ws->total = off;
    return true;
}

} // namespace fp4moe

using namespace fp4moe;

extern "C" {

const char *moe_status_string(moe_status s)
{
    switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED_SHAPE: return "MOE_ERR_UNSUPPORTED_SHAPE";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
    case MOE_ERR_UNSUPPORTED_DEVICE: return "MOE_ERR_UNSUPPORTED_DEVICE";
    case MOE_ERR_DEVICE_FAULT: return "MOE_ERR_DEVICE_FAULT";
    }
    return "MOE_ERR_UNKNOWN";
}

int moe_version(void) { return 100; }

moe_status moe_pack_fp4(const float *w, uint8_t *w_fp4, uint8_t *w_scale, int E, int N, int K, void *stream)
{
    if (!w || !w_fp4 || !w_scale) return MOE_ERR_INVALID_ARG;
    if (E < 0 || N < 0 || K < 0) return MOE_ERR_INVALID_ARG;
    if (!aligned(w, 16) || !aligned(w_fp4, 16) || !aligned(w_scale, 16)) return MOE_ERR_INVALID_ARG;
    if (K % 128 || N % 128) return MOE_ERR_UNSUPPORTED_SHAPE;
    if ((long long)E * N * K == 0) return MOE_OK;
    DeviceInfo *di;
    moe_status st = device_info(&di);
    if (st != MOE_OK) return st;
    return cuda_status(launch_pack_fp4(w, w_fp4, w_scale, E, N, K, (cudaStream_t)stream));
}

moe_status moe_fp4_to_fp8t(const uint8_t *w_fp4, const uint8_t *w_scale, uint8_t *w8t, uint8_t *s8t, int E, int N,
                           int K, void *stream)
{
    if (!w_fp4 || !w_scale || !w8t || !s8t) return MOE_ERR_INVALID_ARG;
    if (E < 0 || N < 0 || K < 0) return MOE_ERR_INVALID_ARG;
    if (!aligned(w_fp4, 16) || !aligned(w_scale, 16) || !aligned(w8t, 16)) return MOE_ERR_INVALID_ARG;
    if (K % 128 || N % 128) return MOE_ERR_UNSUPPORTED_SHAPE;
    if ((long long)E * N * K == 0) return MOE_OK;
    if ((long long)E * (N / 128) * (K / 128) > 0x7FFFFFFFLL) return MOE_ERR_UNSUPPORTED_SHAPE;
    DeviceInfo *di;
    moe_status st = device_info(&di);
    if (st != MOE_OK) return st;
    return cuda_status(launch_fp4_to_fp8t(w_fp4, w_scale, w8t, s8t, E, N, K, (cudaStream_t)stream));
}

moe_status moe_quantize_act(const uint16_t *x, uint8_t *xq, uint8_t *xs, int T, int d, void *stream)
{
    if (!x || !xq || !xs) return MOE_ERR_INVALID_ARG;
    if (T < 0 || d <= 0) return MOE_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(xq, 16)) return MOE_ERR_INVALID_ARG;
    if (d % 128) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (T == 0) return MOE_OK;
    DeviceInfo *di;
    moe_status st = device_info(&di);
    if (st != MOE_OK) return st;
    return cuda_status(launch_quantize(x, xq, xs, d / 128, T, d, (cudaStream_t)stream));
}

moe_status moe_route(const uint16_t *x, const float *gate_w, const float *gate_bias, int32_t *topk_idx,
                     float *topk_w, int T, int d, int E, int k, void *stream)
{
    if (!x || !gate_w || !topk_idx || !topk_w) return MOE_ERR_INVALID_ARG;
    if (T < 0 || d <= 0 || E <= 0 || k <= 0) return MOE_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(gate_w, 16) || !aligned(topk_idx, 4) || !aligned(topk_w, 4) ||
        (gate_bias && !aligned(gate_bias, 4)))
        return MOE_ERR_INVALID_ARG;
    if (d % 128 || k > 8 || k > E || E > 256 || (long long)T * k >= (1ll << 31)) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (T == 0) return MOE_OK;
    DeviceInfo *di;
    moe_status st = device_info(&di);
    if (st != MOE_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    const bool tc = gate_uses_tc(T, d, E);
    // logits [T][E]; with the tensor-core gate also gate_w transposed (fp32)
    // and split (two bf16), the weight norms and the candidate counts
    const size_t zb = round_up((size_t)T * E * 4, 256), wtb = round_up((size_t)E * d * 4, 256),
                 wpb = round_up((size_t)E * d * 2, 256), wnb = round_up((size_t)E * 4, 256);
    const size_t bytes = zb + (tc ? wtb + 2 * wpb + wnb + (size_t)T * 4 : 0);
    void *z = nullptr;
    if (cudaMallocAsync(&z, bytes, s) != cudaSuccess) {
        cudaGetLastError();                      // nothing was enqueued; leave no error behind
        return MOE_ERR_WORKSPACE;
    }
    cudaError_t e;
    if (tc) {
        uint8_t *b = static_cast<uint8_t *>(z);
        GateScratch g;
        g.approx = reinterpret_cast<float *>(b);
        g.wt = reinterpret_cast<float *>(b + zb);
        g.whi = reinterpret_cast<uint16_t *>(b + zb + wtb);
        g.wlo = reinterpret_cast<uint16_t *>(b + zb + wtb + wpb);
        g.wn = reinterpret_cast<float *>(b + zb + wtb + 2 * wpb);
        g.ncand = reinterpret_cast<int32_t *>(b + zb + wtb + 2 * wpb + wnb);
        g.prepared = false;
        e = launch_gate_tc_logits(x, gate_w, gate_bias, g, T, d, E, di->num_sms, di->status, timeout_ns(), s);
        if (e == cudaSuccess)
            e = launch_gate_certify(x, gate_bias, g, topk_idx, topk_w, nullptr, nullptr, nullptr, 0, T, d, E, k,
                                    di->status, s);
    } else {
        e = launch_gate_logits(x, gate_w, gate_bias, (float *)z, T, d, E, s);
        if (e == cudaSuccess)
            e = launch_topk((const float *)z, topk_idx, topk_w, nullptr, nullptr, nullptr, 0, T, d, E, k, di->status,
                            s);
    }
    cudaError_t f = cudaFreeAsync(z, s);
    return cuda_status(e != cudaSuccess ? e : f);
}

moe_status moe_dispatch_plan(const int32_t *topk_idx, int32_t *expert_offsets, int32_t *sorted_pair,
                             int32_t *pair_pos, int T, int E, int k, void *stream)
{
    if (!topk_idx || !expert_offsets || !sorted_pair || !pair_pos) return MOE_ERR_INVALID_ARG;
    if (T < 0 || E <= 0 || k <= 0) return MOE_ERR_INVALID_ARG;
    if (!aligned(topk_idx, 4) || !aligned(expert_offsets, 4) || !aligned(sorted_pair, 4) || !aligned(pair_pos, 4))
        return MOE_ERR_INVALID_ARG;
    if (k > 8 || k > E || E > 256 || (long long)T * k >= (1ll << 31)) return MOE_ERR_UNSUPPORTED_SHAPE;
    DeviceInfo *di;
    moe_status st = device_info(&di);
    if (st != MOE_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    const size_t scratch = plan_scratch_bytes((long long)T * k, E);
    void *counts = nullptr;
    if (scratch && cudaMallocAsync(&counts, scratch, s) != cudaSuccess) {
        cudaGetLastError();                      // nothing was enqueued; leave no error behind
        return MOE_ERR_WORKSPACE;
    }
    cudaError_t e = launch_plan(topk_idx, expert_offsets, sorted_pair, pair_pos, nullptr, (int *)counts, T, E, k,
                                di->status, s);
    cudaError_t f = counts ? cudaFreeAsync(counts, s) : cudaSuccess;
    return cuda_status(e != cudaSuccess ? e : f);
}

size_t moe_workspace_layout(int T, int d, int inter, int E, int k, size_t *offsets, size_t *strides)
{
    Workspace ws;
    if (!workspace_layout(Shapes{T, d, inter, E, k}, &ws)) return 0;
    for (int i = 0; i < MOE_WS_COUNT; i++) {
        if (offsets) offsets[i] = ws.off[i];
        if (strides) strides[i] = ws.stride[i];
    }
    return ws.total;
}

size_t moe_gate_prep_size(int d, int E)
{
    if (d <= 0 || E <= 0 || d % 128 || E > 256) return 0;
    return gate_prep_layout(d, E).total;
}

moe_status moe_prepare_gate(const float *gate_w, void *prep, int d, int E, void *stream)
{
    if (!gate_w || !prep || !aligned(gate_w, 16) || !aligned(prep, 256)) return MOE_ERR_INVALID_ARG;
    if (d <= 0 || E <= 0) return MOE_ERR_INVALID_ARG;
    if (d % 128 || E > 256) return MOE_ERR_UNSUPPORTED_SHAPE;
    int num_sms = 0;
    unsigned *status = nullptr;
    moe_status st = device_query(&num_sms, &status);
    if (st != MOE_OK) return st;
    const GatePrepLayout gl = gate_prep_layout(d, E);
    uint8_t *gp = static_cast<uint8_t *>(prep);
    GateScratch g;
    std::memset(&g, 0, sizeof g);
    g.wt = reinterpret_cast<float *>(gp + gl.wt);
    g.whi = reinterpret_cast<uint16_t *>(gp + gl.whi);
    g.wlo = reinterpret_cast<uint16_t *>(gp + gl.wlo);
    g.wn = reinterpret_cast<float *>(gp + gl.wn);
    return launch_gate_prep(gate_w, g, d, E, (cudaStream_t)stream) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

size_t moe_workspace_size(int T, int d, int inter, int E, int k)
{
    return moe_workspace_layout(T, d, inter, E, k, nullptr, nullptr);
}

moe_status moe_forward_ex(const uint16_t *x, const float *gate_w, const uint8_t *w13_fp4, const uint8_t *w13_scale,
                          const uint8_t *w2_fp4, const uint8_t *w2_scale, uint16_t *out, int T, int d, int inter,
                          int E, int k, void *stream, const moe_forward_opts *opts)
{
    if (!x || !gate_w || !w13_fp4 || !w13_scale || !w2_fp4 || !w2_scale || !out) return MOE_ERR_INVALID_ARG;
    if (T < 0 || d <= 0 || inter <= 0 || E <= 0 || k <= 0) return MOE_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(gate_w, 16) || !aligned(out, 16) || !aligned(w13_fp4, 32) ||
        !aligned(w2_fp4, 32) || !aligned(w13_scale, 16) || !aligned(w2_scale, 16))
        return MOE_ERR_INVALID_ARG;
    moe_forward_opts o;
    std::memset(&o, 0, sizeof o);
    if (opts) o = *opts;
    if (o.flags & ~MOE_FLAG_TEST_STALL_GEMM2) return MOE_ERR_INVALID_ARG;
    if (o.gate_bias && !aligned(o.gate_bias, 4)) return MOE_ERR_INVALID_ARG;
    if ((o.topk_idx_out && !aligned(o.topk_idx_out, 4)) || (o.topk_w_out && !aligned(o.topk_w_out, 4)) ||
        (o.pair_pos_out && !aligned(o.pair_pos_out, 4)) || (o.gu_out && !aligned(o.gu_out, 32)) ||
        (o.gate_prep && !aligned(o.gate_prep, 256)))
        return MOE_ERR_INVALID_ARG;
    if (!layer_shape_ok(T, d, inter, E, k)) return MOE_ERR_UNSUPPORTED_SHAPE;
    Workspace ws;
    workspace_layout(Shapes{T, d, inter, E, k}, &ws);
    if (o.workspace && (!aligned(o.workspace, 256) || o.workspace_bytes < ws.total)) return MOE_ERR_WORKSPACE;
    if (T == 0) return MOE_OK;
    DeviceInfo *di;
    moe_status st = device_info(&di);
    if (st != MOE_OK) return st;

    cudaStream_t s = (cudaStream_t)stream;
    uint8_t *base = static_cast<uint8_t *>(o.workspace);
    bool owned = false;
    if (!base) {
        void *p = nullptr;
        if (cudaMallocAsync(&p, ws.total, s) != cudaSuccess) {
            cudaGetLastError();                  // nothing was enqueued; leave no error behind
            return MOE_ERR_WORKSPACE;
        }
        base = static_cast<uint8_t *>(p);
        owned = true;
    }
    auto at = [&](int r) { return base + ws.off[r]; };
    uint8_t *xq = at(MOE_WS_XQ), *xs = at(MOE_WS_XS);
    float *logits = reinterpret_cast<float *>(at(MOE_WS_LOGITS));
    int32_t *topk_idx = reinterpret_cast<int32_t *>(at(MOE_WS_TOPK_IDX));
    float *topk_w = reinterpret_cast<float *>(at(MOE_WS_TOPK_W));
    int32_t *offs = reinterpret_cast<int32_t *>(at(MOE_WS_EXPERT_OFFSETS));
    int32_t *sorted_pair = reinterpret_cast<int32_t *>(at(MOE_WS_SORTED_PAIR));
    int32_t *pair_pos = reinterpret_cast<int32_t *>(at(MOE_WS_PAIR_POS));
    int32_t *tile_prefix = reinterpret_cast<int32_t *>(at(MOE_WS_TILE_PREFIX));
    uint8_t *hq = at(MOE_WS_HQ), *hs_tiles = at(MOE_WS_HS_TILES);
    uint16_t *y = reinterpret_cast<uint16_t *>(at(MOE_WS_Y));
    uint8_t *xs_tiles = at(MOE_WS_XS_TILES);
    const int xs_stride = (int)ws.stride[MOE_WS_XS];
    const long long P = (long long)T * k;

    cudaError_t e = cudaSuccess;
    auto mark = [&](int stage) {
        if (o.stage_events && e == cudaSuccess) e = cudaEventRecord((cudaEvent_t)o.stage_events[stage], s);
    };
    float *topk_z = reinterpret_cast<float *>(at(MOE_WS_TOPK_Z));
    mark(MOE_STAGE_GATE);
    if (gate_uses_tc(T, d, E)) {
        // tensor-core logits, then (the top-k stage) the certified top-k with
        // the candidates' fixed-order logits and the FP8 quantisation of x
        GateScratch gs;
        if (o.gate_prep) {                      // gate_w's split and norms, prepared at load time
            const GatePrepLayout gl = gate_prep_layout(d, E);
            uint8_t *gp = static_cast<uint8_t *>(const_cast<void *>(o.gate_prep));
            gs.wt = reinterpret_cast<float *>(gp + gl.wt);
            gs.whi = reinterpret_cast<uint16_t *>(gp + gl.whi);
            gs.wlo = reinterpret_cast<uint16_t *>(gp + gl.wlo);
            gs.wn = reinterpret_cast<float *>(gp + gl.wn);
            gs.prepared = true;
        } else {
            gs.wt = reinterpret_cast<float *>(at(MOE_WS_GATE_WT));
            gs.whi = reinterpret_cast<uint16_t *>(at(MOE_WS_GATE_WHI));
            gs.wlo = reinterpret_cast<uint16_t *>(at(MOE_WS_GATE_WLO));
            gs.wn = reinterpret_cast<float *>(at(MOE_WS_GATE_WNORM));
            gs.prepared = false;
        }
        gs.approx = logits;
        gs.ncand = reinterpret_cast<int32_t *>(at(MOE_WS_GATE_NCAND));
        if (e == cudaSuccess)
            e = launch_gate_tc_logits(x, gate_w, o.gate_bias, gs, T, d, E, di->num_sms, di->status, timeout_ns(), s);
        mark(MOE_STAGE_TOPK);
        if (e == cudaSuccess)
            e = launch_gate_certify(x, o.gate_bias, gs, topk_idx, topk_w, topk_z, xq, xs, xs_stride, T, d, E, k,
                                    di->status, s);
    } else {
        if (e == cudaSuccess) e = launch_gate_logits(x, gate_w, o.gate_bias, logits, T, d, E, s);
        mark(MOE_STAGE_TOPK);
        if (e == cudaSuccess)
            e = launch_topk(logits, topk_idx, topk_w, x, xq, xs, xs_stride, T, d, E, k, di->status, s, topk_z);
    }
    mark(MOE_STAGE_PLAN);
    if (e == cudaSuccess)
        e = launch_plan(topk_idx, offs, sorted_pair, pair_pos, tile_prefix,
                        reinterpret_cast<int *>(at(MOE_WS_PLAN_COUNTS)), T, E, k, di->status, s, xs, xs_stride,
                        xs_tiles, d, gemm_tile_rows(P, E), reinterpret_cast<int *>(at(MOE_WS_TILE_DONE)),
                        (int)max_row_tiles(P, E, gemm_tile_rows(P, E)) + 1);
    // From 16 pairs per expert on average, tiles of more than 16 pairs read A
    // from an expert-ordered copy.  Smaller batches gather every tile and skip
    // the copy: their GEMM1 streams weights, and the gather-only kernel (a
    // smaller producer loop) does that faster.  Either way the rows the MMA
    // sees for valid pairs are the same bytes, so the output does not depend
    // on this choice.
    mark(MOE_STAGE_DISPATCH);
    uint8_t *xq_sorted = P >= 16ll * E ? at(MOE_WS_XQ_SORTED) : nullptr;
    if (e == cudaSuccess && xq_sorted)
        e = launch_dispatch_dense(xq, pair_pos, topk_idx, offs, xq_sorted, T, d, k, s);
    mark(MOE_STAGE_GEMM1);
    GemmArgs g;
    std::memset(&g, 0, sizeof g);
    g.expert_offsets = offs;
    g.tile_prefix = tile_prefix;
    g.E = E;
    g.P = P;
    g.status = di->status;
    g.timeout_ns = timeout_ns();
    g.num_sms = di->num_sms;
    g.tile_rows = gemm_tile_rows(P, E);
    g.tile_done = reinterpret_cast<int *>(at(MOE_WS_TILE_DONE));
    g.all_done = g.tile_done + max_row_tiles(P, E, g.tile_rows);
    if (e == cudaSuccess) {
        g.a = xq;
        g.a_dense = xq_sorted;
        g.a_rows = T;
        g.sorted_pair = sorted_pair;
        g.k = k;
        g.a_scale_tiles = xs_tiles;
        g.b = w13_fp4;
        g.b_scale = w13_scale;
        g.N = 2 * inter;
        g.K = d;
        g.hq = hq;
        g.hs_tiles = hs_tiles;
        g.gu_out = o.gu_out;
        e = launch_gemm1(g, inter, s);
        g.gu_out = nullptr;
    }
    mark(MOE_STAGE_GEMM2);
    if (e == cudaSuccess) {
        g.a = hq;
        g.a_dense = nullptr;
        g.a_rows = P;
        g.a_scale_tiles = hs_tiles;
        g.b = w2_fp4;
        g.b_scale = w2_scale;
        g.N = d;
        g.K = inter;
        g.y = y;
        g.stall_test = (o.flags & MOE_FLAG_TEST_STALL_GEMM2) ? 1 : 0;
        e = launch_gemm2(g, d, s);
    }
    mark(MOE_STAGE_COMBINE);
    if (e == cudaSuccess) e = launch_combine(y, pair_pos, topk_w, out, T, d, k, s);
    mark(MOE_STAGE_COUNT);
    if (e == cudaSuccess && o.topk_idx_out)
        e = cudaMemcpyAsync(o.topk_idx_out, topk_idx, (size_t)P * 4, cudaMemcpyDeviceToDevice, s);
    if (e == cudaSuccess && o.topk_w_out)
        e = cudaMemcpyAsync(o.topk_w_out, topk_w, (size_t)P * 4, cudaMemcpyDeviceToDevice, s);
    if (e == cudaSuccess && o.pair_pos_out)
        e = cudaMemcpyAsync(o.pair_pos_out, pair_pos, (size_t)P * 4, cudaMemcpyDeviceToDevice, s);
    if (owned) {
        cudaError_t f = cudaFreeAsync(base, s);
        if (e == cudaSuccess) e = f;
    }
    return cuda_status(e);
}

moe_status moe_forward(const uint16_t *x, const float *gate_w, const uint8_t *w13_fp4, const uint8_t *w13_scale,
                       const uint8_t *w2_fp4, const uint8_t *w2_scale, uint16_t *out, int T, int d, int inter, int E,
                       int k, void *stream)
{
    return moe_forward_ex(x, gate_w, w13_fp4, w13_scale, w2_fp4, w2_scale, out, T, d, inter, E, k, stream, nullptr);
}

moe_status moe_get_device_status(void *stream)
{
    DeviceInfo *di;
    moe_status st = device_info(&di);
    if (st != MOE_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
    unsigned v = 0;
    if (cudaMemcpy(&v, di->status, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
    const unsigned zero = 0;
    if (cudaMemcpy(di->status, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess) return MOE_ERR_CUDA;
    if (v & kStatusTimeout) return MOE_ERR_TIMEOUT;
    if (v & kStatusBadData) return MOE_ERR_DEVICE_FAULT;
    return MOE_OK;
}

} // extern "C"
