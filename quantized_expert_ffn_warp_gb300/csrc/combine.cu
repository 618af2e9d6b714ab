// Weighted combine + residual + sigmoid-gated shared expert, one fused kernel
// ("Flash-MoE" article, section 3: MoE combine, residual and sigmoid gate in
// one kernel):
//   out[t] = x[t] + sum_j w[t][j] * y[pos(t, j)] + sigmoid(x[t] . wg) * y_sh[t]
// accumulated in fp32 in slot order, rounded once to fp16 (nearest even).
// The residual rows come from xres: x itself, or the un-normalised rows when
// the layer runs on RMSNorm-ed tokens.
#include <cuda_fp16.h>

#include "internal.cuh"

namespace qe {

constexpr int kCombThreads = 256;
constexpr int kCombCols = kCombThreads * 8;   // columns per CTA

__global__ void __launch_bounds__(kCombThreads) combine_kernel(
    const __half *__restrict__ x, const __half *__restrict__ xres, __half *__restrict__ out,
    const float *__restrict__ w,
    const int32_t *__restrict__ pos_of_pair, const float *__restrict__ y,
    const __half *__restrict__ gate_w, int n, int H, int k, int P, int has_shared, int residual)
{
    __shared__ float red[kCombThreads / 32];
    pdl_enter();
    const int t = blockIdx.x;
    const __half *xr = x + (long long)t * H;
    float gate = 0.f;
    if (has_shared) {
        float z = 0.f;
        for (int c = threadIdx.x * 8; c < H; c += kCombThreads * 8) {
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
        for (int i = 0; i < kCombThreads / 32; i++)
            z += red[i];
        gate = 1.0f / (1.0f + expf(-z));
    }
    const int c = blockIdx.y * kCombCols + threadIdx.x * 8;
    if (c >= H)
        return;
    float acc[8];
    if (residual) {
        const uint4 xv = *reinterpret_cast<const uint4 *>(xres + (long long)t * H + c);
        const __half2 *xh = reinterpret_cast<const __half2 *>(&xv);
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const float2 a = __half22float2(xh[i]);
            acc[2 * i] = a.x;
            acc[2 * i + 1] = a.y;
        }
    } else {
#pragma unroll
        for (int i = 0; i < 8; i++)
            acc[i] = 0.f;
    }
    for (int j = 0; j < k; j++) {
        const int pos = pos_of_pair[t * k + j];
        if (pos < 0)
            continue;
        const float wj = w[t * k + j];
        const float4 *yr = reinterpret_cast<const float4 *>(y + (long long)pos * H + c);
        const float4 a = yr[0], b = yr[1];
        acc[0] = fmaf(wj, a.x, acc[0]);
        acc[1] = fmaf(wj, a.y, acc[1]);
        acc[2] = fmaf(wj, a.z, acc[2]);
        acc[3] = fmaf(wj, a.w, acc[3]);
        acc[4] = fmaf(wj, b.x, acc[4]);
        acc[5] = fmaf(wj, b.y, acc[5]);
        acc[6] = fmaf(wj, b.z, acc[6]);
        acc[7] = fmaf(wj, b.w, acc[7]);
    }
    if (has_shared) {
        const float4 *yr = reinterpret_cast<const float4 *>(y + (long long)(P + t) * H + c);
        const float4 a = yr[0], b = yr[1];
        acc[0] = fmaf(gate, a.x, acc[0]);
        acc[1] = fmaf(gate, a.y, acc[1]);
        acc[2] = fmaf(gate, a.z, acc[2]);
        acc[3] = fmaf(gate, a.w, acc[3]);
        acc[4] = fmaf(gate, b.x, acc[4]);
        acc[5] = fmaf(gate, b.y, acc[5]);
        acc[6] = fmaf(gate, b.z, acc[6]);
        acc[7] = fmaf(gate, b.w, acc[7]);
    }
    uint4 ov;
    __half2 *oh = reinterpret_cast<__half2 *>(&ov);
#pragma unroll
    for (int i = 0; i < 4; i++)
        oh[i] = __floats2half2_rn(acc[2 * i], acc[2 * i + 1]);
    *reinterpret_cast<uint4 *>(out + (long long)t * H + c) = ov;
}

cudaError_t launch_combine(const LayerDev &L, const Workspace &ws, const __half *x,
                           const __half *xres, __half *out, int n, cudaStream_t st)
{
    dim3 grid(n, (L.H + kCombCols - 1) / kCombCols);
    return launch_pdl(combine_kernel, grid, dim3(kCombThreads), 0, st, x, xres, out,
                      static_cast<const float *>(ws.w), static_cast<const int32_t *>(ws.pos_of_pair),
                      static_cast<const float *>(ws.y), L.sh_gate_w, n, L.H, L.k, n * L.k,
                      L.has_shared, L.residual);
}

}  // namespace qe
