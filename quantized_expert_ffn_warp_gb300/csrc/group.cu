// Token-to-expert grouping: histogram, exclusive scan and a stable scatter.
//
// Each expert's work is aggregated across tokens so that one read of its
// weights serves all of them (the per-expert task queue
// Map{expert_id: Vec(request_id, input_tokens)} of "为什么12G显存笔记本能跑
// MoE-16B", section 2.3; "Strata" section 2.3: requests that share an expert
// read its weights once).  Here the queue is realised as counts, offsets and a
// permutation of the flat pair ids p = t*k + j, stably sorted by expert: the
// pairs of one expert keep their pair order.
//
// One CTA of 32 warps.  Warp w owns a contiguous slice of the pairs.  A
// per-(warp, expert) histogram turned into per-warp bases, plus ranks among
// equal experts inside each 32-pair step (warp match), give every pair its
// sorted position without atomics on the positions, so the order is
// deterministic and stable.  The same kernel cuts each expert's list into
// work entries for the FFN kernels and appends the shared expert's: experts
// with at least `big` tokens (big > 0) get entries of up to gtok tokens
// for the tensor-core GEMM kernels, the others entries of up to kMaxTokTile
// tokens for the decode kernels.
#include "internal.cuh"

namespace qe {

constexpr int kGroupThreads = 1024;
constexpr int kGroupWarps = kGroupThreads / 32;

size_t group_smem_bytes(int E)
{
    return sizeof(int) * ((size_t)kGroupWarps * E + 3 * (size_t)E + 3 + 3 * kGroupWarps);
}

__global__ void __launch_bounds__(kGroupThreads) group_kernel(
    const int32_t *__restrict__ idx, int n, int k, int E, int has_shared, int big, int gtok,
    int *__restrict__ hdr, Entry *__restrict__ entries, int4 *__restrict__ gentries,
    int32_t *__restrict__ counts, int32_t *__restrict__ offsets,
    int32_t *__restrict__ perm, int32_t *__restrict__ pos_of_pair,
    int32_t *__restrict__ tok_of_pos)
{
    extern __shared__ int sm[];
    pdl_enter();
    int *whist = sm;                           // [32][E]
    int *off = whist + kGroupWarps * E;        // [E]   exclusive offsets
    int *ebase = off + E;                      // [E]   exclusive decode-entry bases
    int *gbase = ebase + E;                    // [E]   exclusive GEMM-entry bases
    int *wt = gbase + E;                       // [3][32] warp totals for the scans
    int *tot = wt + 3 * kGroupWarps;           // [3] totals
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int P = n * k;
    const int S = (P + kGroupWarps - 1) / kGroupWarps;
    const int p_beg = min(P, warp * S), p_end = min(P, p_beg + S);

    for (int i = tid; i < kGroupWarps * E; i += kGroupThreads)
        whist[i] = 0;
    __syncthreads();

    int bad = 0;
    for (int p = p_beg + lane; p < p_end; p += 32) {
        const int e = idx[p];
        if (e < 0 || e >= E)
            bad = 1;
        else
            atomicAdd(&whist[warp * E + e], 1);
    }
    if (bad)
        atomicOr(&hdr[2], MOE_STATUS_BAD_EXPERT);
    __syncthreads();

    // per expert: exclusive prefix over warps, total count, entry counts
    int c_mine = 0, ch_mine = 0, cg_mine = 0;
    for (int e = tid; e < E; e += kGroupThreads) {
        int run = 0;
        for (int w = 0; w < kGroupWarps; w++) {
            const int v = whist[w * E + e];
            whist[w * E + e] = run;
            run += v;
        }
        c_mine = run;
        const bool gemm = big > 0 && run >= big;
        ch_mine = gemm ? 0 : (run + kMaxTokTile - 1) / kMaxTokTile;
        cg_mine = gemm ? (run + gtok - 1) / gtok : 0;
        counts[e] = run;
    }
    // block exclusive scan of (count, decode entries, GEMM entries) over
    // experts: E <= 1024 = one per thread
    int v0 = c_mine, v1 = ch_mine, v2 = cg_mine;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int u0 = __shfl_up_sync(0xffffffffu, v0, d);
        const int u1 = __shfl_up_sync(0xffffffffu, v1, d);
        const int u2 = __shfl_up_sync(0xffffffffu, v2, d);
        if (lane >= d) {
            v0 += u0;
            v1 += u1;
            v2 += u2;
        }
    }
    if (lane == 31) {
        wt[warp] = v0;
        wt[kGroupWarps + warp] = v1;
        wt[2 * kGroupWarps + warp] = v2;
    }
    __syncthreads();
    if (warp == 0) {
        int a0 = wt[lane], a1 = wt[kGroupWarps + lane], a2 = wt[2 * kGroupWarps + lane];
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int u0 = __shfl_up_sync(0xffffffffu, a0, d);
            const int u1 = __shfl_up_sync(0xffffffffu, a1, d);
            const int u2 = __shfl_up_sync(0xffffffffu, a2, d);
            if (lane >= d) {
                a0 += u0;
                a1 += u1;
                a2 += u2;
            }
        }
        wt[lane] = a0;
        wt[kGroupWarps + lane] = a1;
        wt[2 * kGroupWarps + lane] = a2;
        if (lane == 31) {
            tot[0] = a0;
            tot[1] = a1;
            tot[2] = a2;
        }
    }
    __syncthreads();
    if (tid < E) {
        const int pre0 = warp ? wt[warp - 1] : 0, pre1 = warp ? wt[kGroupWarps + warp - 1] : 0;
        const int pre2 = warp ? wt[2 * kGroupWarps + warp - 1] : 0;
        off[tid] = pre0 + v0 - c_mine;
        ebase[tid] = pre1 + v1 - ch_mine;
        gbase[tid] = pre2 + v2 - cg_mine;
        offsets[tid] = off[tid];
    }
    if (tid == 0)
        offsets[E] = tot[0];
    __syncthreads();

    // stable scatter: walk the warp's slice in order, 32 pairs per step
    const unsigned lt = (1u << lane) - 1u;
    for (int base = p_beg; base < p_end; base += 32) {
        const int p = base + lane;
        const bool valid = p < p_end;
        int e = valid ? idx[p] : -1;
        const bool ok = valid && e >= 0 && e < E;
        const int key = ok ? e : -2 - lane;   // unmatched keys for skipped lanes
        const unsigned peers = __match_any_sync(0xffffffffu, key);
        const int rank = __popc(peers & lt);
        if (ok) {
            const int pos = off[e] + whist[warp * E + e] + rank;
            perm[pos] = p;
            pos_of_pair[p] = pos;
            tok_of_pos[pos] = p / k;
        } else if (valid) {
            pos_of_pair[p] = -1;
        }
        __syncwarp();
        if (ok && rank == 0)
            whist[warp * E + e] += __popc(peers);
        __syncwarp();
    }

    __syncthreads();   // perm is complete

    // work entries: routed experts in expert order, then the shared expert
    for (int e = tid; e < E; e += kGroupThreads) {
        const int c = c_mine, nb = ch_mine;
        for (int j = 0; j < nb; j++) {
            Entry en;
            en.expert = e;
            en.start = off[e] + j * kMaxTokTile;
            en.ntok = min(kMaxTokTile, c - j * kMaxTokTile);
            en.pad = 0;
            for (int i = 0; i < kMaxTokTile; i++)
                en.tok[i] = perm[en.start + min(i, en.ntok - 1)] / k;
            entries[ebase[e] + j] = en;
        }
        for (int j = 0; j < cg_mine; j++)
            gentries[gbase[e] + j] =
                make_int4(e, off[e] + j * gtok, min(gtok, c - j * gtok), 0);
    }
    const int n_r = tot[1];
    const bool sh_gemm = has_shared && big > 0 && n >= big;
    const int n_s = has_shared && !sh_gemm ? (n + kMaxTokTile - 1) / kMaxTokTile : 0;
    const int g_r = tot[2];
    const int g_s = sh_gemm ? (n + gtok - 1) / gtok : 0;
    for (int j = tid; j < g_s; j += kGroupThreads)
        gentries[g_r + j] = make_int4(E, P + j * gtok, min(gtok, n - j * gtok), 0);
    for (int j = tid; j < n_s; j += kGroupThreads) {
        Entry en;
        en.expert = E;
        en.start = P + j * kMaxTokTile;
        en.ntok = min(kMaxTokTile, n - j * kMaxTokTile);
        en.pad = 0;
        for (int i = 0; i < kMaxTokTile; i++)
            en.tok[i] = j * kMaxTokTile + min(i, en.ntok - 1);
        entries[n_r + j] = en;
    }
    if (has_shared)
        for (int t = tid; t < n; t += kGroupThreads)
            tok_of_pos[P + t] = t;
    if (tid == 0) {
        hdr[0] = n_r;
        hdr[1] = n_s;
        hdr[4] = g_r;
        hdr[5] = g_s;
    }
}

void configure_group_kernel(size_t smem)
{
    cudaFuncSetAttribute(group_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

cudaError_t launch_group(const LayerDev &L, const Workspace &ws, int n, int big, int gtok,
                         cudaStream_t st)
{
    return launch_pdl(group_kernel, dim3(1), dim3(kGroupThreads), group_smem_bytes(L.E), st,
                      static_cast<const int32_t *>(ws.idx), n, L.k, L.E, L.has_shared, big, gtok,
                      ws.hdr,
                      ws.entries, ws.gentries, ws.counts, ws.offsets, ws.perm, ws.pos_of_pair,
                      ws.tok_of_pos);
}

}  // namespace qe
