// Expert-parallel layer across GPUs: the routed experts are partitioned by id
// over `world` ranks ("Strata" article, section 5.2: with two cards the expert
// cache is sharded per card).  Rank r owns experts [r E / world,
// (r + 1) E / world).  Each rank routes its own tokens, sends every (token,
// slot) pair's activation row to the owner of its expert, the owner runs its
// experts on the rows it received (one weight read per expert for all of
// them), the rows come back, and the source rank combines them.  Two
// layer-free kernels here frame the exchange:
//   - dispatch: per pair p = t k + j, its destination rank, its position in
//     the send buffer (pairs grouped by destination, pair order kept inside a
//     destination), the owner's local expert id, and the row x[t] copied to
//     that position; plus the rows per destination;
//   - combine: out[t] = x[t] + sum_j w[t][j] y[pos(t, j)] + sigmoid(x[t] . wg)
//     y_sh[t], in fp32 in slot order, rounded once to fp16.
// The exchange itself is the caller's all-to-all (NCCL); no remote memory is
// touched here.
#include <cuda_fp16.h>

#include "internal.cuh"

namespace qe {

constexpr int kEpThreads = 1024;
constexpr int kEpWarps = kEpThreads / 32;
constexpr int kEpMaxWorld = 32;

__host__ __device__ __forceinline__ int ep_owner(int e, int E, int world)
{
    return (int)(((long long)(e + 1) * world - 1) / E);
}

__host__ __device__ __forceinline__ int ep_first(int r, int E, int world)
{
    return (int)((long long)r * E / world);
}

// One CTA: counts per destination, then stable positions (chunks of 1024
// pairs in order; inside a chunk, warp order then lane order).
__global__ void __launch_bounds__(kEpThreads) ep_plan_kernel(
    const int32_t *__restrict__ idx, int P, int E, int world, int32_t *__restrict__ send_expert,
    int32_t *__restrict__ pos_of_pair, int32_t *__restrict__ dest_counts, int *__restrict__ bad_out)
{
    __shared__ int cnt[kEpMaxWorld], base[kEpMaxWorld];
    __shared__ int wcnt[kEpWarps][kEpMaxWorld];
    pdl_enter();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid < kEpMaxWorld)
        cnt[tid] = 0;
    __syncthreads();
    int bad = 0;
    for (int p = tid; p < P; p += kEpThreads) {
        const int e = idx[p];
        if (e < 0 || e >= E)
            bad = 1;
        else
            atomicAdd(&cnt[ep_owner(e, E, world)], 1);
    }
    __syncthreads();
    if (tid == 0) {
        int run = 0;
        for (int r = 0; r < world; r++) {
            base[r] = run;
            dest_counts[r] = cnt[r];
            run += cnt[r];
        }
    }
    __syncthreads();
    const unsigned lt = (1u << lane) - 1u;
    for (int c0 = 0; c0 < P; c0 += kEpThreads) {
        const int p = c0 + tid;
        const int e = p < P ? idx[p] : -1;
        const bool ok = e >= 0 && e < E;
        const int d = ok ? ep_owner(e, E, world) : -1;
        const unsigned peers = __match_any_sync(0xffffffffu, ok ? d : -2 - lane);
        const int rank = __popc(peers & lt);
        if (lane < kEpMaxWorld)
            wcnt[warp][lane] = 0;
        __syncwarp();
        if (ok && rank == 0)
            wcnt[warp][d] = __popc(peers);
        __syncthreads();
        // exclusive prefix over the warps of this chunk, per destination
        if (tid < world) {
            int run = 0;
            for (int w = 0; w < kEpWarps; w++) {
                const int v = wcnt[w][tid];
                wcnt[w][tid] = run;
                run += v;
            }
            cnt[tid] = run;   // this chunk's pairs per destination
        }
        __syncthreads();
        if (ok) {
            const int pos = base[d] + wcnt[warp][d] + rank;
            pos_of_pair[p] = pos;
            send_expert[pos] = e - ep_first(d, E, world);
        } else if (p < P) {
            pos_of_pair[p] = -1;
        }
        __syncthreads();
        if (tid < world)
            base[tid] += cnt[tid];
        __syncthreads();
    }
    if (bad)
        atomicOr(bad_out, 1);
}

// send_x[pos_of_pair[p]] = x[p / k]: one CTA per pair, 16-byte columns.
__global__ void __launch_bounds__(256) ep_gather_kernel(const __half *__restrict__ x, int H, int k,
                                                       const int32_t *__restrict__ pos_of_pair,
                                                       __half *__restrict__ send_x)
{
    pdl_enter();
    const int p = blockIdx.x;
    const int pos = pos_of_pair[p];
    if (pos < 0)
        return;
    const uint4 *src = reinterpret_cast<const uint4 *>(x + (long long)(p / k) * H);
    uint4 *dst = reinterpret_cast<uint4 *>(send_x + (long long)pos * H);
    for (int i = threadIdx.x; i < H / 8; i += blockDim.x)
        dst[i] = src[i];
}

constexpr int kEcThreads = 256;
constexpr int kEcCols = kEcThreads * 8;

// out[t] = x[t] (residual) + sum_j w[t][j] y[pos(t, j)] + sigmoid(x[t] . wg) y_sh[t]
__global__ void __launch_bounds__(kEcThreads) ep_combine_kernel(
    const __half *__restrict__ x, int H, int k, const float *__restrict__ w,
    const int32_t *__restrict__ pos_of_pair, const __half *__restrict__ y,
    const __half *__restrict__ gate_w, const __half *__restrict__ y_sh, int residual,
    __half *__restrict__ out)
{
    __shared__ float red[kEcThreads / 32];
    pdl_enter();
    const int t = blockIdx.x;
    const __half *xr = x + (long long)t * H;
    float gate = 0.f;
    if (y_sh) {
        float z = 0.f;
        for (int c = threadIdx.x * 8; c < H; c += kEcThreads * 8) {
            const uint4 xv = *reinterpret_cast<const uint4 *>(xr + c);
            const uint4 gv = *reinterpret_cast<const uint4 *>(gate_w + c);
            const __half2 *xh = reinterpret_cast<const __half2 *>(&xv);
            const __half2 *gh = reinterpret_cast<const __half2 *>(&gv);
#pragma unroll
            for (int i = 0; i < 4; i++) {
                const float2 a = __half22float2(xh[i]), b = __half22float2(gh[i]);
                z = fmaf(a.x, b.x, z);
                z = fmaf(a.y, b.y, z);
            }
        }
#pragma unroll
        for (int d = 16; d > 0; d >>= 1)
            z += __shfl_xor_sync(0xffffffffu, z, d);
        if ((threadIdx.x & 31) == 0)
            red[threadIdx.x >> 5] = z;
        __syncthreads();
        z = 0.f;
#pragma unroll
        for (int i = 0; i < kEcThreads / 32; i++)
            z += red[i];
        gate = 1.0f / (1.0f + expf(-z));
    }
    const int c = blockIdx.y * kEcCols + threadIdx.x * 8;
    if (c >= H)
        return;
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; i++)
        acc[i] = 0.f;
    if (residual) {
        const uint4 xv = *reinterpret_cast<const uint4 *>(xr + c);
        const __half2 *xh = reinterpret_cast<const __half2 *>(&xv);
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const float2 a = __half22float2(xh[i]);
            acc[2 * i] = a.x;
            acc[2 * i + 1] = a.y;
        }
    }
    auto add_row = [&](const __half *row, float wt) {
        const uint4 v = *reinterpret_cast<const uint4 *>(row + c);
        const __half2 *h = reinterpret_cast<const __half2 *>(&v);
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const float2 a = __half22float2(h[i]);
            acc[2 * i] = fmaf(wt, a.x, acc[2 * i]);
            acc[2 * i + 1] = fmaf(wt, a.y, acc[2 * i + 1]);
        }
    };
    for (int j = 0; j < k; j++) {
        const int pos = pos_of_pair[t * k + j];
        if (pos >= 0)
            add_row(y + (long long)pos * H, w[t * k + j]);
    }
    if (y_sh)
        add_row(y_sh + (long long)t * H, gate);
    uint4 ov;
    __half2 *oh = reinterpret_cast<__half2 *>(&ov);
#pragma unroll
    for (int i = 0; i < 4; i++)
        oh[i] = __floats2half2_rn(acc[2 * i], acc[2 * i + 1]);
    *reinterpret_cast<uint4 *>(out + (long long)t * H + c) = ov;
}

}  // namespace qe

namespace qe {
int record_failure(int code, const char *msg);
int record_success();
bool device_pointer(const void *p);
}  // namespace qe

namespace {
bool misaligned(const void *p, uintptr_t a) { return ((uintptr_t)p & (a - 1)) != 0; }
}  // namespace

extern "C" int moe_ep_dispatch(const void *x, int n, int H, const int32_t *topk_idx, int k,
                               int E, int world, void *send_x, int32_t *send_expert,
                               int32_t *pos_of_pair, int32_t *dest_counts, int *status,
                               void *stream)
{
    using namespace qe;
    if (!x || !topk_idx || !send_x || !send_expert || !pos_of_pair || !dest_counts || !status)
        return record_failure(MOE_ERR_INVALID_ARG, "null pointer argument");
    if (n < 1 || k < 1 || k > kMaxTopK || E < 1 || E > kMaxExperts || k > E)
        return record_failure(MOE_ERR_INVALID_ARG, "bad n_tokens, top_k or n_experts");
    if (world < 1 || world > kEpMaxWorld || world > E)
        return record_failure(MOE_ERR_INVALID_ARG, "world must be in 1..min(32, n_experts)");
    if (H < kGroup || H > 16384 || H % kGroup)
        return record_failure(MOE_ERR_INVALID_ARG, "hidden must be a multiple of 128 in 128..16384");
    if ((long long)n * k > (1LL << 24))
        return record_failure(MOE_ERR_INVALID_ARG, "n_tokens * top_k too large");
    if (misaligned(x, 16) || misaligned(send_x, 16) || misaligned(topk_idx, 4) ||
        misaligned(send_expert, 4) || misaligned(pos_of_pair, 4) || misaligned(dest_counts, 4) ||
        misaligned(status, 4))
        return record_failure(MOE_ERR_INVALID_ARG, "misaligned pointer");
    if (!device_pointer(x) || !device_pointer(topk_idx) || !device_pointer(send_x) ||
        !device_pointer(send_expert) || !device_pointer(pos_of_pair) ||
        !device_pointer(dest_counts) || !device_pointer(status))
        return record_failure(MOE_ERR_INVALID_ARG, "arguments must be device pointers");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int P = n * k;
    cudaError_t e = launch_pdl(ep_plan_kernel, dim3(1), dim3(kEpThreads), 0, st, topk_idx, P, E,
                               world, send_expert, pos_of_pair, dest_counts, status);
    if (e == cudaSuccess)
        e = launch_pdl(ep_gather_kernel, dim3(P), dim3(256), 0, st,
                       static_cast<const __half *>(x), H, k,
                       static_cast<const int32_t *>(pos_of_pair), static_cast<__half *>(send_x));
    if (e != cudaSuccess) {
        cudaGetLastError();
        return record_failure(MOE_ERR_CUDA, cudaGetErrorString(e));
    }
    return record_success();
}

extern "C" int moe_ep_combine(const void *x, int n, int H, int k, const float *topk_w,
                              const int32_t *pos_of_pair, const void *y_rows,
                              const void *sh_gate_w, const void *y_shared, int residual,
                              void *out, void *stream)
{
    using namespace qe;
    if (!x || !topk_w || !pos_of_pair || !y_rows || !out)
        return record_failure(MOE_ERR_INVALID_ARG, "null pointer argument");
    if ((sh_gate_w == nullptr) != (y_shared == nullptr))
        return record_failure(MOE_ERR_INVALID_ARG, "sh_gate_w and y_shared go together");
    if (n < 1 || k < 1 || k > kMaxTopK || (residual != 0 && residual != 1))
        return record_failure(MOE_ERR_INVALID_ARG, "bad n_tokens, top_k or residual");
    if (H < kGroup || H > 16384 || H % kGroup)
        return record_failure(MOE_ERR_INVALID_ARG, "hidden must be a multiple of 128 in 128..16384");
    if (misaligned(x, 16) || misaligned(y_rows, 16) || misaligned(out, 16) ||
        misaligned(topk_w, 4) || misaligned(pos_of_pair, 4) ||
        (y_shared && (misaligned(y_shared, 16) || misaligned(sh_gate_w, 16))))
        return record_failure(MOE_ERR_INVALID_ARG, "misaligned pointer");
    const char *a = static_cast<const char *>(x), *b = static_cast<const char *>(out);
    const size_t bytes = (size_t)n * H * 2;
    if (a < b + bytes && b < a + bytes)
        return record_failure(MOE_ERR_INVALID_ARG, "out overlaps x");
    if (!device_pointer(x) || !device_pointer(topk_w) || !device_pointer(pos_of_pair) ||
        !device_pointer(y_rows) || !device_pointer(out) ||
        (y_shared && (!device_pointer(y_shared) || !device_pointer(sh_gate_w))))
        return record_failure(MOE_ERR_INVALID_ARG, "arguments must be device pointers");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    dim3 grid(n, (H + kEcCols - 1) / kEcCols);
    cudaError_t e = launch_pdl(ep_combine_kernel, grid, dim3(kEcThreads), 0, st,
                               static_cast<const __half *>(x), H, k, topk_w, pos_of_pair,
                               static_cast<const __half *>(y_rows),
                               static_cast<const __half *>(sh_gate_w),
                               static_cast<const __half *>(y_shared), residual,
                               static_cast<__half *>(out));
    if (e != cudaSuccess) {
        cudaGetLastError();
        return record_failure(MOE_ERR_CUDA, cudaGetErrorString(e));
    }
    return record_success();
}
