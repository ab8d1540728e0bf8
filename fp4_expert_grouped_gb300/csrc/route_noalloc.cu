// route_noalloc.cu -- moe_route without any device allocation.
//
// moe_route needs T*E fp32 logits of scratch between its two kernels and gets
// them from the stream-ordered allocator.  Some callers cannot allocate at
// call time: a serving loop that handed all free device memory to its own
// pool at start-up (an allocation would fail or force that pool to shrink),
// a latency-critical loop whose rules forbid allocator calls after
// initialisation (an allocation can block on the device or fragment memory),
// or a host program that owns device memory through its own allocator and
// forbids libraries from calling cudaMalloc behind its back.
// moe_route_noalloc serves them: its scratch is a fixed array in device
// global memory that belongs to this library, so the call itself allocates
// nothing.
//
// The array below exists once on every device that loads the library and
// stays there until the process exits.  Every call shares it; nothing in it
// has to start at zero, because each call writes every logit it later reads.
// Two calls that run at the same time on the device (e.g. on two streams)
// race on it.
#include "fp4moe.h"
#include "moe_internal.h"

#include <mutex>

namespace fp4moe {
namespace {

// 1 Mi fp32 logits = 4 MiB: T * E <= 1048576 (e.g. 4096 tokens with 256 experts).
constexpr size_t kNoallocLogits = size_t(1) << 20;

static __device__ __align__(256) float g_route_scratch[kNoallocLogits];

// In host code `g_route_scratch` only names a host-side shadow of the array,
// not a device address.  The device address is looked up once per device
// (with that device current) and cached here.
constexpr int kMaxDev = 64;
float *g_scratch_addr[kMaxDev];
std::mutex g_scratch_mu;

cudaError_t scratch_for_current_device(float **out)
{
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        err = cudaGetSymbolAddress(&p, g_route_scratch);
        if (err != cudaSuccess) return err;
        g_scratch_addr[dev] = static_cast<float *>(p);
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

bool aligned_to(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

} // namespace
} // namespace fp4moe

using namespace fp4moe;

extern "C" moe_status moe_route_noalloc(const uint16_t *x, const float *gate_w, const float *gate_bias,
                                        int32_t *topk_idx, float *topk_w, int T, int d, int E, int k, void *stream)
{
    if (!x || !gate_w || !topk_idx || !topk_w) return MOE_ERR_INVALID_ARG;
    if (T < 0 || d <= 0 || E <= 0 || k <= 0) return MOE_ERR_INVALID_ARG;
    if (!aligned_to(x, 16) || !aligned_to(gate_w, 16) || !aligned_to(topk_idx, 4) || !aligned_to(topk_w, 4) ||
        (gate_bias && !aligned_to(gate_bias, 4)))
        return MOE_ERR_INVALID_ARG;
    if (d % 128 || k > 8 || k > E || E > 256 || (long long)T * k >= (1ll << 31)) return MOE_ERR_UNSUPPORTED_SHAPE;
    if ((size_t)T * (size_t)E > kNoallocLogits) return MOE_ERR_WORKSPACE;   // beyond the fixed scratch
    if (T == 0) return MOE_OK;
    int num_sms = 0;
    unsigned *status = nullptr;
    moe_status st = device_query(&num_sms, &status);
    if (st != MOE_OK) return st;
    float *z = nullptr;
    if (scratch_for_current_device(&z) != cudaSuccess) return MOE_ERR_CUDA;
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = launch_gate_logits(x, gate_w, gate_bias, z, T, d, E, s);
    if (e == cudaSuccess)
        e = launch_topk(z, topk_idx, topk_w, nullptr, nullptr, nullptr, 0, T, d, E, k, status, s);
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
