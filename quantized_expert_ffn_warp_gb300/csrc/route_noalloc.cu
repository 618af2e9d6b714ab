// moe_route_topk_noalloc: routing (exact router logits, top-k, softmax
// weights) without a layer object and without allocating device memory.
//
// Callers that cannot allocate at the point of routing use it -- e.g. a
// scheduler that picks the experts to stage before any layer exists, on a
// device whose memory its own pool already holds; there a cudaMalloc fails or
// synchronises the device and stalls every other stream.  The routing kernel
// needs scratch (per-(token, expert) 128-bit logit sums and per-token-block
// tickets, both zero on entry); here it lives in one fixed file-scope device
// buffer, so the call's size is bounded by that buffer.  Its address is looked
// up once per device (the first call on a device does this setup).  Every
// call clears the must-be-zero part on its stream before the kernel, so a
// call never depends on what an earlier one left.  Calls whose executions
// overlap share the buffer and race.
#include <cuda_runtime.h>

#include <functional>
#include <mutex>

#include "internal.cuh"

namespace qe {
bool device_pointer(const void *p);
int router_k_slices(int H, int E, int n, int num_sms);
int record_failure(int code, const char *msg);
int record_success();
void configure_router_kernel(size_t smem);
cudaError_t launch_route_scratch(const __half *x, const __half *rw, const float *bias, int n,
                                 int H, int E, int k, int ks, unsigned long long *sums,
                                 unsigned *tickets,
                                 int *status, int32_t *idx, float *w, cudaStream_t st);
}  // namespace qe

namespace {

// Scratch layout: [status word, padded to 256 B][tickets][sums]
constexpr size_t kStatusBytes = 256;
constexpr size_t kTicketBytes = 4 * ((MOE_NOALLOC_MAX_SCORES + 7) / 8);   // 8 KB
constexpr size_t kSumsOffset = kStatusBytes + kTicketBytes;                // 16-byte aligned
constexpr size_t kSumBytes = 24;   // three 64-bit limbs per (token, expert)
constexpr size_t kScratchBytes = kSumsOffset + kSumBytes * MOE_NOALLOC_MAX_SCORES;   // ~392 KB
static_assert(kSumsOffset % 256 == 0, "sums must stay aligned");

static __device__ __align__(256) unsigned char g_route_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;

struct DeviceSetup {
    std::once_flag once;
    unsigned char *base = nullptr;
    int num_sms = 0;
    cudaError_t err = cudaSuccess;
};
DeviceSetup g_setup[kMaxDevices];

void setup_device(DeviceSetup &s, int dev)
{
    void *p = nullptr;
    s.err = cudaGetSymbolAddress(&p, g_route_scratch);
    if (s.err == cudaSuccess)
        s.err = cudaDeviceGetAttribute(&s.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (s.err == cudaSuccess) {
        qe::configure_router_kernel((size_t)8 * 1024 * sizeof(int2));
        s.err = cudaGetLastError();
    }
    if (s.err == cudaSuccess)
        s.base = static_cast<unsigned char *>(p);
}

}  // namespace

extern "C" int moe_route_topk_noalloc(const void *x, const void *router_w,
                                      const float *router_bias, int n, int H, int E, int k,
                                      int32_t *topk_idx, float *topk_w, void *stream)
{
    using namespace qe;
    if (!x || !router_w || !topk_idx || !topk_w)
        return record_failure(MOE_ERR_INVALID_ARG, "null pointer argument");
    if (H < kGroup || H > 16384 || H % kGroup)
        return record_failure(MOE_ERR_INVALID_ARG, "hidden must be a multiple of 128 in 128..16384");
    if (E < 1 || E > kMaxExperts)
        return record_failure(MOE_ERR_INVALID_ARG, "n_experts must be in 1..1024");
    if (k < 1 || k > kMaxTopK || k > E)
        return record_failure(MOE_ERR_INVALID_ARG, "top_k must be in 1..min(32, n_experts)");
    if (n < 1)
        return record_failure(MOE_ERR_INVALID_ARG, "n_tokens must be at least 1");
    if ((long long)n * E > MOE_NOALLOC_MAX_SCORES)
        return record_failure(MOE_ERR_INVALID_ARG,
                              "n_tokens * n_experts exceeds MOE_NOALLOC_MAX_SCORES (16384)");
    // the routing kernel reads x in 16-byte words, router_w in 8-byte words
    // and the others as their own element type; a misaligned pointer would
    // fault on the device
    const auto mis = [](const void *p, uintptr_t a) { return ((uintptr_t)p & (a - 1)) != 0; };
    if (mis(router_w, 8) || mis(x, 16) || (router_bias && mis(router_bias, 4)) ||
        mis(topk_idx, 4) || mis(topk_w, 4))
        return record_failure(MOE_ERR_INVALID_ARG,
                              "misaligned pointer (x needs 16 bytes, router_w 8, router_bias, "
                              "topk_idx and topk_w 4)");
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return record_failure(MOE_ERR_CUDA, "no usable current CUDA device");
    }
    if (!device_pointer(x) || !device_pointer(router_w) || !device_pointer(topk_idx) ||
        !device_pointer(topk_w) || (router_bias && !device_pointer(router_bias)))
        return record_failure(MOE_ERR_INVALID_ARG, "arguments must be device pointers");
    DeviceSetup &s = g_setup[dev];
    std::call_once(s.once, setup_device, std::ref(s), dev);
    if (s.err != cudaSuccess || !s.base)
        return record_failure(MOE_ERR_CUDA, "scratch setup failed on this device");

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int *status = reinterpret_cast<int *>(s.base);
    unsigned *tickets = reinterpret_cast<unsigned *>(s.base + kStatusBytes);
    unsigned long long *sums = reinterpret_cast<unsigned long long *>(s.base + kSumsOffset);
    // status, every ticket and the n * E sums this call uses
    const size_t clear = kSumsOffset + kSumBytes * (size_t)n * E;
    if (cudaMemsetAsync(s.base, 0, clear, st) != cudaSuccess) {
        cudaGetLastError();
        return record_failure(MOE_ERR_CUDA, "clearing the routing scratch failed");
    }
    const int ks = router_k_slices(H, E, n, s.num_sms);
    const cudaError_t e = launch_route_scratch(
        static_cast<const __half *>(x), static_cast<const __half *>(router_w), router_bias, n, H,
        E, k, ks, sums, tickets, status, topk_idx, topk_w, st);
    if (e != cudaSuccess)
        return record_failure(MOE_ERR_CUDA, cudaGetErrorString(e));
    return record_success();
}
