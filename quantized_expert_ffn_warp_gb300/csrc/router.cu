// Router: exact logits and warp-level top-k with softmax renormalisation.
//
// The router scores every expert from the token's hidden state and keeps the
// k best ("12GB显卡跑68GB大模型：Betelgeuse引擎实测22 tok/s", MoE background;
// top-2 of 64 in the "Strata" article, section 1.1; top-4 of 512 in the
// "Flash-MoE" article, section 1).  A logit here is the exact sum of the
// exact fp16 x fp16 products rounded once to fp32, so routing does not depend
// on how the dot product is split across threads and blocks.
//
// Exactness: an fp16 value is M * 2^(s - 24) with |M| < 2^11 and s in
// [0, 29].  Write s = 15*c + r with c in {0, 1}, r in [0, 14]; then
// X = M << r is a signed integer below 2^25 and the value is X * 2^(15c - 24).
// A product of two such values is X*W * 2^(15(cx+cw) - 48): an int64 product
// below 2^50 in one of three classes cx + cw = 0, 1, 2.  Each thread keeps
// one int64 accumulator per class (at most 8192 terms per thread: no
// overflow), the three are merged into one 128-bit integer (scale 2^-48) and
// the 128-bit partial sums are added exactly across lanes and K-slices.
#include <cuda_fp16.h>

#include "internal.cuh"

namespace qe {

constexpr int kRtTok = 8;     // tokens per CTA
constexpr int kRtWarps = 8;   // experts per CTA (one per warp)

// Split an fp16 bit pattern into the class-0 and class-1 integers described
// above (exactly one of them non-zero, or both zero).  inf/nan count as 0 and
// raise the non-finite flag.
__device__ __forceinline__ int2 split_half(uint32_t b, int &bad)
{
    const int e = (b >> 10) & 31, f = b & 1023;
    const int M = e ? (f | 1024) : f;
    const int s = (e ? e : 1) - 1;
    const int cls = s >= 15;
    int v = M << (s - 15 * cls);
    if (b & 0x8000)
        v = -v;
    if (e == 31) {
        bad = 1;
        v = 0;
    }
    return cls ? make_int2(0, v) : make_int2(v, 0);
}

__global__ void __launch_bounds__(256) router_partial_kernel(const uint16_t *__restrict__ x,
                                                             const uint16_t *__restrict__ rw,
                                                             int n, int H, int E, int kslice,
                                                             ulonglong2 *__restrict__ part,
                                                             int *__restrict__ status)
{
    extern __shared__ int2 xs[];   // [kRtTok][4][kslice/4]
    const int q4 = kslice / 4;
    const int t0 = blockIdx.y * kRtTok, ks = blockIdx.z;
    const int nt = min(kRtTok, n - t0);
    const long long k0 = (long long)ks * kslice;
    int bad = 0;
    for (int i = threadIdx.x; i < kRtTok * kslice; i += blockDim.x) {
        const int t = i / kslice, hl = i - t * kslice;
        int2 v = make_int2(0, 0);
        if (t < nt)
            v = split_half(x[(long long)(t0 + t) * H + k0 + hl], bad);
        xs[(t * 4 + (hl & 3)) * q4 + (hl >> 2)] = v;
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = blockIdx.x * kRtWarps + warp;
    if (e < E) {
        long long A0[kRtTok], A1[kRtTok], A2[kRtTok];
#pragma unroll
        for (int t = 0; t < kRtTok; t++)
            A0[t] = A1[t] = A2[t] = 0;
        const uint2 *wrow = reinterpret_cast<const uint2 *>(rw + (long long)e * H + k0);
        for (int q = lane; q < q4; q += 32) {
            const uint2 wv = __ldg(wrow + q);
            const uint32_t hb[4] = {wv.x & 0xFFFF, wv.x >> 16, wv.y & 0xFFFF, wv.y >> 16};
#pragma unroll
            for (int i = 0; i < 4; i++) {
                const int2 w = split_half(hb[i], bad);
                const int2 *xp = xs + i * q4 + q;
#pragma unroll
                for (int t = 0; t < kRtTok; t++) {
                    const int2 xv = xp[t * 4 * q4];
                    A0[t] += (long long)xv.x * w.x;
                    A1[t] += (long long)xv.x * w.y;
                    A1[t] += (long long)xv.y * w.x;
                    A2[t] += (long long)xv.y * w.y;
                }
            }
        }
#pragma unroll
        for (int t = 0; t < kRtTok; t++) {
            if (t >= nt)
                break;
            __int128 s = (__int128)A0[t] + ((__int128)A1[t] << 15) + ((__int128)A2[t] << 30);
            unsigned long long lo = (unsigned long long)s;
            long long hi = (long long)(s >> 64);
#pragma unroll
            for (int d = 16; d > 0; d >>= 1) {
                const unsigned long long olo = __shfl_xor_sync(0xffffffffu, lo, d);
                const long long ohi = __shfl_xor_sync(0xffffffffu, hi, d);
                const unsigned long long nlo = lo + olo;
                hi = hi + ohi + (nlo < lo ? 1 : 0);
                lo = nlo;
            }
            if (lane == 0)
                part[((long long)ks * n + t0 + t) * E + e] = make_ulonglong2(lo, (unsigned long long)hi);
        }
    }
    if (bad)
        atomicOr(status, MOE_STATUS_NONFINITE);
}

// value = s * 2^-48 rounded once to fp32 (nearest, ties to even).
__device__ __forceinline__ float round_scaled(unsigned long long lo, long long hi)
{
    const bool neg = hi < 0;
    unsigned __int128 m = ((unsigned __int128)(unsigned long long)hi << 64) | lo;
    if (neg)
        m = ~m + 1;
    if (m == 0)
        return 0.0f;
    const unsigned long long mh = (unsigned long long)(m >> 64);
    const int p = mh ? 127 - __clzll((long long)mh) : 63 - __clzll((long long)(unsigned long long)m);
    unsigned int mant;
    int shift = 0;
    if (p <= 23) {
        mant = (unsigned int)m;
    } else {
        shift = p - 23;
        unsigned __int128 q = m >> shift;
        const unsigned __int128 rem = m - (q << shift);
        const unsigned __int128 half = (unsigned __int128)1 << (shift - 1);
        if (rem > half || (rem == half && (q & 1)))
            q += 1;
        if (q >> 24) {
            q >>= 1;
            shift += 1;
        }
        mant = (unsigned int)q;
    }
    // mant * 2^(shift - 48) with mant in [2^23, 2^24) (or smaller, exact): normal range
    const float f = ldexpf((float)mant, shift - 48);
    return neg ? -f : f;
}

// kPer = experts per lane (E <= 32 * kPer).
template <int kPer>
__global__ void __launch_bounds__(256) topk_kernel(const ulonglong2 *__restrict__ part, int ks,
                                                   int n, int E, int k,
                                                   const float *__restrict__ bias,
                                                   int32_t *__restrict__ idx,
                                                   float *__restrict__ wout,
                                                   float *__restrict__ logits)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + warp;
    if (t >= n)
        return;
    float lv[kPer];
#pragma unroll
    for (int i = 0; i < kPer; i++) {
        const int e = lane + 32 * i;
        lv[i] = 0.f;
        if (e < E) {
            unsigned long long lo = 0;
            long long hi = 0;
#pragma unroll 8
            for (int s = 0; s < ks; s++) {
                const ulonglong2 v = part[((long long)s * n + t) * E + e];
                const unsigned long long nlo = lo + v.x;
                hi = hi + (long long)v.y + (nlo < lo ? 1 : 0);
                lo = nlo;
            }
            float l = round_scaled(lo, hi);
            if (bias)
                l = __fadd_rn(l, bias[e]);
            lv[i] = l;
            if (logits)
                logits[(long long)t * E + e] = l;
        }
    }
    unsigned int taken = 0;
    float my_v = 0.f;
    int my_e = 0;
    for (int j = 0; j < k; j++) {
        float bv = 0.f;
        int be = -1;
#pragma unroll
        for (int i = 0; i < kPer; i++) {
            const int e = lane + 32 * i;
            if (e < E && !((taken >> i) & 1u) && (be < 0 || lv[i] > bv)) {
                bv = lv[i];
                be = e;
            }
        }
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, d);
            const int oe = __shfl_xor_sync(0xffffffffu, be, d);
            const bool take = oe >= 0 && (be < 0 || ov > bv || (ov == bv && oe < be));
            if (take) {
                bv = ov;
                be = oe;
            }
        }
        if ((be & 31) == lane)
            taken |= 1u << (be >> 5);
        if (lane == j) {
            my_v = bv;
            my_e = be;
        }
    }
    const float mx = __shfl_sync(0xffffffffu, my_v, 0);
    const float ex = lane < k ? expf(my_v - mx) : 0.f;
    float den = ex;
#pragma unroll
    for (int d = 16; d > 0; d >>= 1)
        den += __shfl_xor_sync(0xffffffffu, den, d);
    if (lane < k) {
        idx[(long long)t * k + lane] = my_e;
        wout[(long long)t * k + lane] = ex / den;
    }
}

void configure_router_kernel(size_t smem)
{
    cudaFuncSetAttribute(router_partial_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)smem);
}

cudaError_t launch_router(const LayerDev &L, const Workspace &ws, const __half *x, int n, int ks,
                          cudaStream_t st)
{
    const int kslice = L.H / ks;
    const int E = L.E;
    dim3 grid((E + kRtWarps - 1) / kRtWarps, (n + kRtTok - 1) / kRtTok, ks);
    const size_t smem = (size_t)kRtTok * kslice * sizeof(int2);
    router_partial_kernel<<<grid, 256, smem, st>>>(reinterpret_cast<const uint16_t *>(x),
                                                   reinterpret_cast<const uint16_t *>(L.router_w),
                                                   n, L.H, E, kslice, ws.partials, ws.hdr + 2);
    return cudaGetLastError();
}

cudaError_t launch_topk(const LayerDev &L, const Workspace &ws, int n, int ks, int want_logits,
                        cudaStream_t st)
{
    float *lg = want_logits ? ws.logits : nullptr;
    const dim3 grid((n + 7) / 8);
    if (L.E <= 64)
        topk_kernel<2><<<grid, 256, 0, st>>>(ws.partials, ks, n, L.E, L.k, L.router_bias, ws.idx, ws.w, lg);
    else if (L.E <= 128)
        topk_kernel<4><<<grid, 256, 0, st>>>(ws.partials, ks, n, L.E, L.k, L.router_bias, ws.idx, ws.w, lg);
    else if (L.E <= 256)
        topk_kernel<8><<<grid, 256, 0, st>>>(ws.partials, ks, n, L.E, L.k, L.router_bias, ws.idx, ws.w, lg);
    else if (L.E <= 512)
        topk_kernel<16><<<grid, 256, 0, st>>>(ws.partials, ks, n, L.E, L.k, L.router_bias, ws.idx, ws.w, lg);
    else
        topk_kernel<32><<<grid, 256, 0, st>>>(ws.partials, ks, n, L.E, L.k, L.router_bias, ws.idx, ws.w, lg);
    return cudaGetLastError();
}

}  // namespace qe
