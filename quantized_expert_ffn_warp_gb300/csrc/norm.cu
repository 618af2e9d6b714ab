// Two-pass RMSNorm of the residual stream in front of the router ("Flash-MoE"
// article, section 3: two-pass RMSNorm among the kernels of a layer).  Pass 1
// the mean square of a row, pass 2 the row scaled by 1 / sqrt(ms + eps) and
// the gain.  The pages give no precision; the fp16 values it writes are
// within one ulp of the correctly rounded real value (and equal to it almost
// always).  They are the tokens the router and the experts see, so that a
// given input always routes the same way the fp32 steps follow one fixed
// order, each one IEEE operation rounded to nearest even (no contraction):
//   - the squares r_h^2 (exact in fp32);
//   - per group of 128 consecutive h: lane l adds the squares of h = 4l ..
//     4l+3 left to right, then the lanes combine by a butterfly (xor 16, 8,
//     4, 2, 1);
//   - the group sums added in group order, starting from 0;
//   - ms = sum / H; v = ms + eps; rs = 1 / sqrt(v);
//   - xn_h = fp16((r_h * rs) * g_h).
// One CTA per token; H is a multiple of 128 and at most 16384.
#include <cuda_fp16.h>

#include "internal.cuh"

namespace qe {

constexpr int kNormThreads = 256;
constexpr int kNormMaxGroups = 16384 / kGroup;

__global__ void __launch_bounds__(kNormThreads) rmsnorm_kernel(const __half *__restrict__ r,
                                                              const __half *__restrict__ g,
                                                              float eps, int H,
                                                              __half *__restrict__ xn)
{
    __shared__ float part[kNormMaxGroups];
    __shared__ float rs_sm;
    pdl_enter();
    const int t = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = H / kGroup;
    const __half *row = r + (long long)t * H;
    for (int gg = warp; gg < G; gg += kNormThreads / 32) {
        const uint2 v = *reinterpret_cast<const uint2 *>(row + gg * kGroup + 4 * lane);
        const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&v.x));
        const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&v.y));
        float s = __fadd_rn(__fadd_rn(__fadd_rn(__fmul_rn(a.x, a.x), __fmul_rn(a.y, a.y)),
                                      __fmul_rn(b.x, b.x)),
                            __fmul_rn(b.y, b.y));
#pragma unroll
        for (int d = 16; d > 0; d >>= 1)
            s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, d));
        if (lane == 0)
            part[gg] = s;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        float sum = 0.0f;
        for (int gg = 0; gg < G; gg++)
            sum = __fadd_rn(sum, part[gg]);
        const float ms = __fdiv_rn(sum, (float)H);
        rs_sm = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, eps)));
    }
    __syncthreads();
    const float rs = rs_sm;
    __half *out = xn + (long long)t * H;
    for (int h = threadIdx.x * 8; h < H; h += kNormThreads * 8) {
        const uint4 rv = *reinterpret_cast<const uint4 *>(row + h);
        const uint4 gv = *reinterpret_cast<const uint4 *>(g + h);
        const __half2 *rh = reinterpret_cast<const __half2 *>(&rv);
        const __half2 *gh = reinterpret_cast<const __half2 *>(&gv);
        uint4 ov;
        __half2 *oh = reinterpret_cast<__half2 *>(&ov);
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const float2 a = __half22float2(rh[i]), w = __half22float2(gh[i]);
            oh[i] = __halves2half2(__float2half_rn(__fmul_rn(__fmul_rn(a.x, rs), w.x)),
                                   __float2half_rn(__fmul_rn(__fmul_rn(a.y, rs), w.y)));
        }
        *reinterpret_cast<uint4 *>(out + h) = ov;
    }
}

cudaError_t launch_rmsnorm(const __half *r, const __half *g, float eps, int n, int H,
                           __half *xn, cudaStream_t st)
{
    return launch_pdl(rmsnorm_kernel, dim3(n), dim3(kNormThreads), 0, st, r, g, eps, H, xn);
}

}  // namespace qe
