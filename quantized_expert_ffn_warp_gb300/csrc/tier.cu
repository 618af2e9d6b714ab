// Expert residency tiers: hot experts resident in HBM, cold experts in host
// memory, a bounded pool of device slots for the cold experts in use.
//
// The pages' offload engines keep the most frequently routed experts on the
// GPU and the rest in host RAM ("Luce Spark", sections 1-2: per-(layer,
// expert) routing frequencies pick the set pinned on the GPU; the weights of
// the experts that miss it are copied in on demand, behind the matmuls), hold
// the experts in use in a pool of VRAM slots, and resolve which routed
// experts are present on the device, in the stream, instead of asking the host
// ("Betelgeuse", the VRAM slot pool and the in-stream GPU doorbell with one
// CUDA Graph replay).
//
// On GB300 the cold tier is pinned host memory that the SMs read in place
// over NVLink-C2C.  Per forward, after the grouping has counted the tokens of
// every expert, two kernels run in the layer's stream with no host round
// trip:
//   - stage_decide_kernel (one CTA): every touched expert that is not
//     resident either already has a slot (a hit: the slot is marked used by
//     this call) or needs one (a miss).  The misses take, in expert order,
//     the free slots that this call does not use, least recently used first
//     (ties to the lower slot); an evicted expert loses its slot.  It writes
//     the device base pointer of each touched cold expert's records, which
//     the FFN kernels read, and the list of copies;
//   - stage_copy_kernel (grid): copies the missed experts' records (gate/up
//     and down streams) from host memory into their slots with 16-byte loads.
// The FFN kernels then read every expert from device memory.
// If a call touched more cold experts than free slots -- impossible when the
// pool holds at least min(cold experts, max_tokens * top_k) slots, which
// moe_layer_set_residency requires -- the surplus experts read an all-zero
// record block (their outputs are 0) and MOE_STATUS_TIER_OVERFLOW is set.
#include <cuda_runtime.h>

#include "internal.cuh"

namespace qe {

constexpr int kDecideThreads = 1024;

__global__ void __launch_bounds__(kDecideThreads) stage_decide_kernel(TierDev t,
                                                                      const int32_t *counts)
{
    __shared__ unsigned call;
    __shared__ int n_miss, n_cand;
    __shared__ int miss_scan[kDecideThreads];
    pdl_enter();
    const int tid = threadIdx.x;
    if (tid == 0) {
        call = *t.call + 1;
        *t.call = call;
    }
    __syncthreads();
    // pass 1: hits mark their slot, misses are counted (expert order)
    int miss = 0;
    const int e = tid;
    if (e < t.E && counts[e] > 0) {
        const int s = t.slot_of[e];
        if (s >= 0) {
            t.slot_used[s] = call;
            t.ebase_gu[e] = t.slot_gu + (long long)s * t.gu_bytes;
            t.ebase_dn[e] = t.slot_dn + (long long)s * t.dn_bytes;
            atomicAdd(&t.stats[0], 1ull);
        } else if (s == kNoSlot) {
            miss = 1;
        }
    }
    miss_scan[tid] = miss;
    __syncthreads();
    for (int d = 1; d < kDecideThreads; d <<= 1) {   // inclusive scan of the miss flags
        const int v = tid >= d ? miss_scan[tid - d] : 0;
        __syncthreads();
        miss_scan[tid] += v;
        __syncthreads();
    }
    if (tid == kDecideThreads - 1)
        n_miss = miss_scan[tid];
    // pass 2: rank of each free slot (not used by this call) by (last use, slot)
    int rank = -1;
    const int s = tid;
    if (s < t.S && t.slot_used[s] != call) {
        const unsigned u = t.slot_used[s];
        rank = 0;
        for (int o = 0; o < t.S; o++) {
            const unsigned uo = t.slot_used[o];
            if (uo != call && (uo < u || (uo == u && o < s)))
                rank++;
        }
    }
    if (tid == 0)
        n_cand = 0;
    __syncthreads();
    if (rank >= 0)
        atomicAdd(&n_cand, 1);
    __syncthreads();
    // the r-th miss (expert order) takes the free slot of rank r
    if (rank >= 0 && rank < n_miss) {
        // find the expert of the rank-th miss: miss_scan is the inclusive count
        int lo = 0, hi = t.E - 1;
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (miss_scan[mid] > rank)
                hi = mid;
            else
                lo = mid + 1;
        }
        const int me = lo;
        const int old = t.slot_expert[s];
        if (old >= 0) {
            t.slot_of[old] = kNoSlot;
            t.ebase_gu[old] = t.zero;
            t.ebase_dn[old] = t.zero;
        }
        t.slot_expert[s] = me;
        t.slot_used[s] = call;
        t.copies[rank] = s;
        t.copies[t.S + rank] = me;
    }
    __syncthreads();   // evictions (writes of ebase[old]) before the new owners' writes
    if (rank >= 0 && rank < n_miss) {
        const int me = t.copies[t.S + rank];
        t.slot_of[me] = s;
        t.ebase_gu[me] = t.slot_gu + (long long)s * t.gu_bytes;
        t.ebase_dn[me] = t.slot_dn + (long long)s * t.dn_bytes;
    }
    if (tid == 0) {
        const int done = min(n_miss, n_cand);
        *t.n_copy = done;
        t.stats[1] += (unsigned long long)n_miss;
        if (n_miss > n_cand)
            atomicOr(t.status, MOE_STATUS_TIER_OVERFLOW);
    }
    // misses beyond the free slots (only when the pool is smaller than the
    // required minimum) read the zero expert
    if (e < t.E && miss && miss_scan[e] > n_cand) {
        t.ebase_gu[e] = t.zero;
        t.ebase_dn[e] = t.zero;
    }
}

constexpr int kStageThreads = 256;
constexpr int kStageUnroll = 4;   // 16-byte loads in flight per thread

__device__ __forceinline__ void stage_addr(const TierDev &t, long long i, long long per_gu,
                                           long long per, const uint4 *&src, uint4 *&dst)
{
    const int c = (int)(i / per);
    const long long u = i - (long long)c * per;
    const int s = t.copies[c], e = t.copies[t.S + c];
    if (u < per_gu) {
        src = reinterpret_cast<const uint4 *>(t.host_gu + (long long)e * t.gu_bytes) + u;
        dst = reinterpret_cast<uint4 *>(t.slot_gu + (long long)s * t.gu_bytes) + u;
    } else {
        src = reinterpret_cast<const uint4 *>(t.host_dn + (long long)e * t.dn_bytes) + (u - per_gu);
        dst = reinterpret_cast<uint4 *>(t.slot_dn + (long long)s * t.dn_bytes) + (u - per_gu);
    }
}

// Copy of the missed experts' records into their slots: the copy list is
// split into 16-byte units over the grid, kStageUnroll loads of a thread in
// flight before its stores (host memory answers slowly: the bytes in flight
// set the rate); the loads read host memory in place.
__global__ void __launch_bounds__(kStageThreads) stage_copy_kernel(TierDev t)
{
    pdl_enter();
    const int n = *t.n_copy;
    const long long per_gu = t.gu_bytes / 16, per_dn = t.dn_bytes / 16, per = per_gu + per_dn;
    const long long total = per * n;
    const long long stride = (long long)gridDim.x * kStageThreads;
    for (long long i0 = (long long)blockIdx.x * kStageThreads + threadIdx.x; i0 < total;
         i0 += stride * kStageUnroll) {
        uint4 v[kStageUnroll];
        uint4 *dst[kStageUnroll];
#pragma unroll
        for (int j = 0; j < kStageUnroll; j++) {
            const long long i = i0 + j * stride;
            dst[j] = nullptr;
            if (i < total) {
                const uint4 *src;
                stage_addr(t, i, per_gu, per, src, dst[j]);
                v[j] = __ldcs(src);   // streamed once: no need to keep it in the caches
            }
        }
#pragma unroll
        for (int j = 0; j < kStageUnroll; j++)
            if (dst[j])
                *dst[j] = v[j];
    }
}

cudaError_t launch_stage(const TierDev &t, const Workspace &ws, int num_sms, cudaStream_t st)
{
    cudaError_t e = launch_pdl(stage_decide_kernel, dim3(1), dim3(kDecideThreads), 0, st, t,
                               static_cast<const int32_t *>(ws.counts));
    if (e != cudaSuccess)
        return e;
    return launch_pdl(stage_copy_kernel, dim3(4 * num_sms), dim3(kStageThreads), 0, st, t);
}

}  // namespace qe
