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
// one int64 accumulator per class (a K slice holds at most 1024 values, so a
// thread adds at most 64 terms below 2^50 to one accumulator: no overflow),
// the lanes of a warp add theirs exactly (a reduce-scatter that leaves each
// token's class sums with a few lanes), those merge them into one 128-bit
// integer (scale 2^-48) and add the K slice's total into the token's sum,
// kept as three 64-bit limbs of 40, 40 and 48 bits (bits 0-39,
// 40-79 and the signed rest) with three fire-and-forget atomic adds: each
// limb has 24 bits of headroom, so no carry has to travel between limbs
// until the sum is read.  Integer addition is associative, so the sum does
// not depend on the order in which slices arrive.
//
// One launch does the whole routing step: the last CTA to finish a block of
// 8 tokens (a per-block ticket counter) rounds those tokens' sums, runs top-k
// and the softmax, and clears the sums and its ticket for the next call.
#include <cuda_fp16.h>

#include "internal.cuh"

namespace qe {

constexpr int kRtTok = 8;     // tokens per CTA (one top-k warp each)
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

// Bit i set when expert lane + 32 i exists.
template <int kPer>
__device__ __forceinline__ unsigned valid_mask(int E, int lane)
{
    unsigned m = 0;
#pragma unroll
    for (int i = 0; i < kPer; i++)
        if (lane + 32 * i < E)
            m |= 1u << i;
    return m;
}

// The k largest of the logits lv (expert lane + 32 i) whose bit is set in
// avail, by (logit desc, expert id asc), and their softmax weights, written
// to idx/wout of token t.  One warp.
// Each round takes every lane's best remaining logit by a max tree over its
// kPer slots (log2 kPer dependent steps), then a warp argmax; the winner's
// slot becomes -inf.  Logits are finite, and an unavailable slot (-inf) is
// never chosen while k experts are available, as they always are.
template <int kPer>
__device__ __forceinline__ void select_topk(const float (&lv)[kPer], unsigned avail, int k, int t,
                                            int32_t *__restrict__ idx, float *__restrict__ wout)
{
    const int lane = threadIdx.x & 31;
    const float ninf = __int_as_float(0xff800000);
    float v[kPer];
#pragma unroll
    for (int i = 0; i < kPer; i++)
        v[i] = (avail >> i) & 1u ? lv[i] : ninf;
    float my_v = 0.f;
    int my_e = 0;
    for (int j = 0; j < k; j++) {
        float tv[kPer];
        int ti[kPer];
#pragma unroll
        for (int i = 0; i < kPer; i++) {
            tv[i] = v[i];
            ti[i] = i;
        }
#pragma unroll
        for (int w = kPer / 2; w > 0; w >>= 1)
#pragma unroll
            for (int i = 0; i < w; i++)
                if (tv[i + w] > tv[i] || (tv[i + w] == tv[i] && ti[i + w] < ti[i])) {
                    tv[i] = tv[i + w];
                    ti[i] = ti[i + w];
                }
        float bv = tv[0];
        int be = lane + 32 * ti[0];
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, d);
            const int oe = __shfl_xor_sync(0xffffffffu, be, d);
            if (ov > bv || (ov == bv && oe < be)) {
                bv = ov;
                be = oe;
            }
        }
        if ((be & 31) == lane) {
#pragma unroll
            for (int i = 0; i < kPer; i++)
                if (i == (be >> 5))
                    v[i] = ninf;
        }
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

// Logit of (token t, expert e) from its exact sum: round(sum) + bias.  The
// three limbs are read first (exact_limbs), so that a thread's loads of
// several sums are in flight together, then the sum is cleared for the next
// call and rounded (exact_finish).
struct Limbs {
    unsigned long long l0, l1, l2;
};

__device__ __forceinline__ Limbs exact_limbs(int t, int e, const unsigned long long *sums, int E)
{
    const unsigned long long *p = sums + ((long long)t * E + e) * 3;
    return Limbs{__ldcg(p), __ldcg(p + 1), __ldcg(p + 2)};
}

__device__ __forceinline__ float exact_finish(const Limbs &m, int t, int e,
                                              unsigned long long *sums, int E,
                                              const float *__restrict__ bias)
{
    unsigned long long *p = sums + ((long long)t * E + e) * 3;
    __stcg(p, 0ull);
    __stcg(p + 1, 0ull);
    __stcg(p + 2, 0ull);
    const __int128 v = (__int128)m.l0 + ((__int128)m.l1 << 40) + ((__int128)(long long)m.l2 << 80);
    float l = round_scaled((unsigned long long)v, (long long)(v >> 64));
    if (bias)
        l = __fadd_rn(l, bias[e]);
    return l;
}

// Grouping of all P <= kFusedPairs pairs of the call by one CTA of 256
// threads (the last routing CTA of the call to finish), with the outputs of
// the separate grouping kernel: counts, offsets, the stable permutation,
// pos_of_pair, tok_of_pos, the decode and GEMM work entries and the entry
// counts in hdr.  Pair p = threadIdx.x: its sorted position is its expert's
// offset, plus the pairs of that expert in the earlier 32-pair warp slices,
// plus its rank among equal experts inside its own slice (warp match), so
// the order is stable and deterministic.  The router's expert ids are always
// valid.
__device__ void group_fused(const RouteExtras &g, const int32_t *idx, int n, int k, int E, int *sm)
{
    constexpr int NW = 8;
    const int P = n * k;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int *whist = sm;                // [NW][E] pairs of expert e in warp slice w, then their prefix
    int *off = whist + NW * E;      // [E] exclusive offsets
    int *eb = off + E;              // [E] decode-entry bases
    int *gb = eb + E;               // [E] GEMM-entry bases
    int *cnt = gb + E;              // [E] counts
    int *stok = cnt + E;            // [kFusedPairs] token of sorted position
    int *wt = stok + kFusedPairs;   // [3][NW] inclusive warp totals of the scans
    int *tot = wt + 3 * NW;         // [3] totals
    for (int i = tid; i < NW * E; i += blockDim.x)
        whist[i] = 0;
    const bool valid = tid < P;
    const int e = valid ? __ldcg(idx + tid) : -1;
    __syncthreads();
    const unsigned peers = __match_any_sync(0xffffffffu, valid ? e : -2 - lane);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    if (valid && rank == 0)
        whist[warp * E + e] = __popc(peers);
    __syncthreads();

    // experts 4 tid .. 4 tid + 3: prefix over the warp slices, counts, entries
    int c4[4], h4[4], g4[4];
    int s0 = 0, s1 = 0, s2 = 0;
#pragma unroll
    for (int j = 0; j < 4; j++) {
        const int ex = 4 * tid + j;
        int run = 0;
        if (ex < E) {
            for (int w = 0; w < NW; w++) {
                const int v = whist[w * E + ex];
                whist[w * E + ex] = run;
                run += v;
            }
            cnt[ex] = run;
            g.counts[ex] = run;
        }
        const bool gemm = g.big > 0 && run >= g.big;
        c4[j] = run;
        h4[j] = gemm ? 0 : (run + kMaxTokTile - 1) / kMaxTokTile;
        g4[j] = gemm ? (run + g.gtok - 1) / g.gtok : 0;
        s0 += c4[j];
        s1 += h4[j];
        s2 += g4[j];
    }
    // block exclusive scan of (pairs, decode entries, GEMM entries)
    int v0 = s0, v1 = s1, v2 = s2;
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
        wt[NW + warp] = v1;
        wt[2 * NW + warp] = v2;
    }
    __syncthreads();
    if (warp == 0) {
        int a0 = lane < NW ? wt[lane] : 0, a1 = lane < NW ? wt[NW + lane] : 0;
        int a2 = lane < NW ? wt[2 * NW + lane] : 0;
#pragma unroll
        for (int d = 1; d < NW; d <<= 1) {
            const int u0 = __shfl_up_sync(0xffffffffu, a0, d);
            const int u1 = __shfl_up_sync(0xffffffffu, a1, d);
            const int u2 = __shfl_up_sync(0xffffffffu, a2, d);
            if (lane >= d) {
                a0 += u0;
                a1 += u1;
                a2 += u2;
            }
        }
        __syncwarp();
        if (lane < NW) {
            wt[lane] = a0;
            wt[NW + lane] = a1;
            wt[2 * NW + lane] = a2;
        }
        if (lane == NW - 1) {
            tot[0] = a0;
            tot[1] = a1;
            tot[2] = a2;
        }
    }
    __syncthreads();
    int p0 = (warp ? wt[warp - 1] : 0) + v0 - s0;
    int p1 = (warp ? wt[NW + warp - 1] : 0) + v1 - s1;
    int p2 = (warp ? wt[2 * NW + warp - 1] : 0) + v2 - s2;
#pragma unroll
    for (int j = 0; j < 4; j++) {
        const int ex = 4 * tid + j;
        if (ex < E) {
            off[ex] = p0;
            eb[ex] = p1;
            gb[ex] = p2;
            g.offsets[ex] = p0;
        }
        p0 += c4[j];
        p1 += h4[j];
        p2 += g4[j];
    }
    if (tid == 0)
        g.offsets[E] = tot[0];
    __syncthreads();

    // stable scatter
    if (valid) {
        const int pos = off[e] + whist[warp * E + e] + rank;
        g.perm[pos] = tid;
        g.pos_of_pair[tid] = pos;
        g.tok_of_pos[pos] = tid / k;
        stok[pos] = tid / k;
    }
    __syncthreads();

    // work entries: routed experts in expert order, then the shared expert
#pragma unroll
    for (int j = 0; j < 4; j++) {
        const int ex = 4 * tid + j;
        if (ex >= E)
            continue;
        const int c = cnt[ex];
        for (int q = 0; q < h4[j]; q++) {
            Entry en;
            en.expert = ex;
            en.start = off[ex] + q * kMaxTokTile;
            en.ntok = min(kMaxTokTile, c - q * kMaxTokTile);
            en.pad = 0;
#pragma unroll
            for (int i = 0; i < kMaxTokTile; i++)
                en.tok[i] = stok[en.start + min(i, en.ntok - 1)];
            g.entries[eb[ex] + q] = en;
        }
        for (int q = 0; q < g4[j]; q++)
            g.gentries[gb[ex] + q] =
                make_int4(ex, off[ex] + q * g.gtok, min(g.gtok, c - q * g.gtok), 0);
    }
    const int n_r = tot[1];
    const bool sh_gemm = g.has_shared && g.big > 0 && n >= g.big;
    const int n_s = g.has_shared && !sh_gemm ? (n + kMaxTokTile - 1) / kMaxTokTile : 0;
    const int g_r = tot[2];
    const int g_s = sh_gemm ? (n + g.gtok - 1) / g.gtok : 0;
    for (int j = tid; j < g_s; j += blockDim.x)
        g.gentries[g_r + j] = make_int4(E, P + j * g.gtok, min(g.gtok, n - j * g.gtok), 0);
    for (int j = tid; j < n_s; j += blockDim.x) {
        Entry en;
        en.expert = E;
        en.start = P + j * kMaxTokTile;
        en.ntok = min(kMaxTokTile, n - j * kMaxTokTile);
        en.pad = 0;
#pragma unroll
        for (int i = 0; i < kMaxTokTile; i++)
            en.tok[i] = j * kMaxTokTile + min(i, en.ntok - 1);
        g.entries[n_r + j] = en;
    }
    if (g.has_shared)
        for (int t = tid; t < n; t += blockDim.x)
            g.tok_of_pos[P + t] = t;
    if (tid == 0) {
        g.hdr[0] = n_r;
        g.hdr[1] = n_s;
        g.hdr[4] = g_r;
        g.hdr[5] = g_s;
    }
}

// The same grouping for calls of at most 32 pairs by one warp (lane = pair),
// with the same outputs: a CTA-wide grouping spends most of its time in its
// barriers when there are only a few pairs.  Counts through shared memory;
// one warp scan over the experts in chunks of 32 gives, packed in one word,
// the exclusive offsets and the bases of each expert's decode and GEMM
// entries (each of the three sums is at most 32 here, so 10-bit fields hold
// them); positions from the offsets and the rank among equal experts (warp
// match); entries written by the first pair of each expert.
__device__ void group_small(const RouteExtras &g, const int32_t *idx, int n, int k, int E, int *sm)
{
    const int P = n * k;
    const int lane = threadIdx.x & 31;
    int *cnt = sm;          // [E] counts, then the packed exclusive scan
    int *stok = sm + E;     // [32] token of sorted position
    for (int e = lane; e < E; e += 32)
        cnt[e] = 0;
    __syncwarp();
    const bool valid = lane < P;
    const int e = valid ? __ldcg(idx + lane) : -1;
    const unsigned peers = __match_any_sync(0xffffffffu, valid ? e : -2 - lane);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    const bool leader = valid && rank == 0;
    const int c = __popc(peers);
    if (leader)
        cnt[e] = c;
    __syncwarp();
    // per expert: count | decode entries << 10 | GEMM entries << 20; four
    // 32-expert chunks per step, their warp scans independent of each other
    int run = 0;
    for (int e0 = 0; e0 < E; e0 += 128) {
        int v[4], pk[4], incl[4];
#pragma unroll
        for (int c = 0; c < 4; c++) {
            const int ee = e0 + 32 * c + lane;
            v[c] = ee < E ? cnt[ee] : 0;
            const bool gm = g.big > 0 && v[c] >= g.big;
            pk[c] = v[c] | (gm ? 0 : (v[c] + kMaxTokTile - 1) / kMaxTokTile) << 10 |
                    (gm ? (v[c] + g.gtok - 1) / g.gtok : 0) << 20;
            incl[c] = pk[c];
        }
#pragma unroll
        for (int d = 1; d < 32; d <<= 1)
#pragma unroll
            for (int c = 0; c < 4; c++) {
                const int u = __shfl_up_sync(0xffffffffu, incl[c], d);
                if (lane >= d)
                    incl[c] += u;
            }
#pragma unroll
        for (int c = 0; c < 4; c++) {
            const int ee = e0 + 32 * c + lane;
            if (ee < E) {
                const int ex = run + incl[c] - pk[c];
                g.counts[ee] = v[c];
                g.offsets[ee] = ex & 1023;
                cnt[ee] = ex;
            }
            run += __shfl_sync(0xffffffffu, incl[c], 31);
        }
    }
    if (lane == 0)
        g.offsets[E] = run & 1023;
    __syncwarp();
    const int pk = valid ? cnt[e] : 0;
    const int off = pk & 1023;
    if (valid) {
        const int pos = off + rank;
        g.perm[pos] = lane;
        g.pos_of_pair[lane] = pos;
        g.tok_of_pos[pos] = lane / k;
        stok[pos] = lane / k;
    }
    __syncwarp();
    // entries of this lane's expert (leaders only) at the bases the scan gave
    const bool gemm = leader && g.big > 0 && c >= g.big;
    const int nh = leader && !gemm ? (c + kMaxTokTile - 1) / kMaxTokTile : 0;
    const int ng = gemm ? (c + g.gtok - 1) / g.gtok : 0;
    const int hb = (pk >> 10) & 1023, gbase = pk >> 20;
    const int n_r = (run >> 10) & 1023, g_r = run >> 20;
    for (int j = 0; j < nh; j++) {
        Entry en;
        en.expert = e;
        en.start = off + j * kMaxTokTile;
        en.ntok = min(kMaxTokTile, c - j * kMaxTokTile);
        en.pad = 0;
#pragma unroll
        for (int i = 0; i < kMaxTokTile; i++)
            en.tok[i] = stok[en.start + min(i, en.ntok - 1)];
        g.entries[hb + j] = en;
    }
    for (int j = 0; j < ng; j++)
        g.gentries[gbase + j] = make_int4(e, off + j * g.gtok, min(g.gtok, c - j * g.gtok), 0);
    const bool sh_gemm = g.has_shared && g.big > 0 && n >= g.big;
    const int n_s = g.has_shared && !sh_gemm ? (n + kMaxTokTile - 1) / kMaxTokTile : 0;
    const int g_s = sh_gemm ? (n + g.gtok - 1) / g.gtok : 0;
    for (int j = lane; j < g_s; j += 32)
        g.gentries[g_r + j] = make_int4(E, P + j * g.gtok, min(g.gtok, n - j * g.gtok), 0);
    for (int j = lane; j < n_s; j += 32) {
        Entry en;
        en.expert = E;
        en.start = P + j * kMaxTokTile;
        en.ntok = min(kMaxTokTile, n - j * kMaxTokTile);
        en.pad = 0;
#pragma unroll
        for (int i = 0; i < kMaxTokTile; i++)
            en.tok[i] = j * kMaxTokTile + min(i, en.ntok - 1);
        g.entries[n_r + j] = en;
    }
    if (g.has_shared)
        for (int t = lane; t < n; t += 32)
            g.tok_of_pos[P + t] = t;
    if (lane == 0) {
        g.hdr[0] = n_r;
        g.hdr[1] = n_s;
        g.hdr[4] = g_r;
        g.hdr[5] = g_s;
    }
}

// The CTA that closes the call's last unit (token block or token) groups the
// pairs: every thread's top-k writes are fenced before the call-wide ticket.
// Returns after resetting the ticket; sm is the CTA's dynamic shared memory.
// With a single unit this CTA wrote every top-k result itself, and a CTA
// barrier makes them visible to its threads: no ticket.
__device__ __forceinline__ void group_if_last(const RouteExtras &fg, unsigned units,
                                              const int32_t *idx, int n, int k, int E, int *sm,
                                              int *flag)
{
    const bool small = n * k <= 32;
    if (units == 1) {
        __syncthreads();
        if (!small)
            group_fused(fg, idx, n, k, E, sm);
        else if (threadIdx.x < 32)
            group_small(fg, idx, n, k, E, sm);
        return;
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0)
        *flag = atomicAdd(fg.ticket, 1u) == units - 1;
    __syncthreads();
    if (!*flag)
        return;
    __threadfence();
    if (!small)
        group_fused(fg, idx, n, k, E, sm);
    else if (threadIdx.x < 32)
        group_small(fg, idx, n, k, E, sm);
    if (threadIdx.x == 0)
        *fg.ticket = 0;
}

// Grid (ceil(E/8), ceil(n/kTok), ks): CTA (bx, by, bz) scores experts
// 8bx..8bx+7 (one per warp) for tokens kTok by .. kTok by + kTok - 1 over K
// slice bz.  kTok = 8, or 4 or 1 for calls of at most that many tokens (less
// work on empty slots).
template <int kPer, int kTok>
__global__ void __launch_bounds__(256) router_kernel(
    const uint16_t *__restrict__ x, const uint16_t *__restrict__ rw, int n, int H, int E, int k,
    int kslice, unsigned long long *sums, unsigned *tickets, const float *__restrict__ bias,
    int32_t *__restrict__ idx, float *__restrict__ wout, float *__restrict__ logits,
    int *__restrict__ status, const RouteExtras fg)
{
    extern __shared__ int2 xs[];   // [kTok][4][kslice/4]; then the logits [kTok][E]
    __shared__ int last_cta;
    const int q4 = kslice / 4;
    const int t0 = blockIdx.y * kTok, ks = blockIdx.z;
    const int nt = min(kTok, n - t0);
    const long long k0 = (long long)ks * kslice;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = blockIdx.x * kRtWarps + warp;
    pdl_enter();
    // this warp's first (token, group) activation sum of the K slice: its
    // load is issued now and reduced after the dot products
    const int gps = kslice / kGroup;
    const int xs_p0 = blockIdx.x * kRtWarps + warp, xs_step = gridDim.x * kRtWarps;
    uint2 xs_v = make_uint2(0u, 0u);
    if (fg.xsum && xs_p0 < nt * gps)
        xs_v = group_sum128_load(reinterpret_cast<const __half *>(x) +
                                 (long long)(t0 + xs_p0 / gps) * H + k0 + (xs_p0 % gps) * kGroup);
    int bad = 0;
    // the warp's first weights, loaded while the activations are staged
    const uint2 *wrow = reinterpret_cast<const uint2 *>(rw + (long long)(e < E ? e : 0) * H + k0);
    const uint2 wv0 = e < E && lane < q4 ? __ldg(wrow + lane) : make_uint2(0u, 0u);
    // stage the split activations: 16-byte loads (8 values), up to kStageLd
    // of them in flight per thread before any is split
    constexpr int kStageLd = 4;
    const int c8 = kslice / 8;   // 16-byte words per token row of the slice
    for (int i0 = threadIdx.x; i0 < kTok * c8; i0 += kStageLd * blockDim.x) {
        uint4 v[kStageLd];
#pragma unroll
        for (int j = 0; j < kStageLd; j++) {
            const int i = i0 + j * blockDim.x;
            const int t = i / c8, c = i - t * c8;
            v[j] = make_uint4(0u, 0u, 0u, 0u);
            if (i < kTok * c8 && t < nt)
                v[j] = *reinterpret_cast<const uint4 *>(x + (long long)(t0 + t) * H + k0 + 8 * c);
        }
#pragma unroll
        for (int j = 0; j < kStageLd; j++) {
            const int i = i0 + j * blockDim.x;
            if (i >= kTok * c8)
                break;
            const int t = i / c8, c = i - t * c8;
            const uint32_t w[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
            for (int h = 0; h < 8; h++) {
                const int hl = 8 * c + h;
                xs[(t * 4 + (hl & 3)) * q4 + (hl >> 2)] =
                    split_half((w[h >> 1] >> (16 * (h & 1))) & 0xFFFF, bad);
            }
        }
    }
    __syncthreads();
    if (e < E) {
        long long A0[kTok], A1[kTok], A2[kTok];
#pragma unroll
        for (int t = 0; t < kTok; t++)
            A0[t] = A1[t] = A2[t] = 0;
        for (int q = lane; q < q4; q += 32) {
            const uint2 wv = q == lane ? wv0 : __ldg(wrow + q);
            const uint32_t hb[4] = {wv.x & 0xFFFF, wv.x >> 16, wv.y & 0xFFFF, wv.y >> 16};
#pragma unroll
            for (int i = 0; i < 4; i++) {
                const int2 w = split_half(hb[i], bad);
                const int2 *xp = xs + i * q4 + q;
#pragma unroll
                for (int t = 0; t < kTok; t++) {
                    const int2 xv = xp[t * 4 * q4];
                    A0[t] += (long long)xv.x * w.x;
                    A1[t] += (long long)xv.x * w.y;
                    A1[t] += (long long)xv.y * w.x;
                    A2[t] += (long long)xv.y * w.y;
                }
            }
        }
        // reduce-scatter over the warp: each halving step keeps one half of
        // the tokens (lane bit d set: the upper half) and adds the partner's
        // share of it, so after log2(kTok) steps the lanes 4t..4t+3 (kTok = 8)
        // hold token t, whose sum the remaining steps complete; the class
        // sums stay separate int64s (at most 32 x 64 terms below 2^50 each:
        // no overflow) and are merged once per token
        constexpr int kL = kTok == 8 ? 3 : kTok == 4 ? 2 : 0;
#pragma unroll
        for (int c = kTok, d = 16; c > 1; c >>= 1, d >>= 1) {
            const bool up = lane & d;
#pragma unroll
            for (int j = 0; j < c / 2; j++) {
                const long long k0v = up ? A0[c / 2 + j] : A0[j], s0v = up ? A0[j] : A0[c / 2 + j];
                const long long k1v = up ? A1[c / 2 + j] : A1[j], s1v = up ? A1[j] : A1[c / 2 + j];
                const long long k2v = up ? A2[c / 2 + j] : A2[j], s2v = up ? A2[j] : A2[c / 2 + j];
                A0[j] = k0v + __shfl_xor_sync(0xffffffffu, s0v, d);
                A1[j] = k1v + __shfl_xor_sync(0xffffffffu, s1v, d);
                A2[j] = k2v + __shfl_xor_sync(0xffffffffu, s2v, d);
            }
        }
#pragma unroll
        for (int d = 16 >> kL; d > 0; d >>= 1) {
            A0[0] += __shfl_xor_sync(0xffffffffu, A0[0], d);
            A1[0] += __shfl_xor_sync(0xffffffffu, A1[0], d);
            A2[0] += __shfl_xor_sync(0xffffffffu, A2[0], d);
        }
        const int t = (lane >> (5 - kL)) & (kTok - 1);
        if ((lane & ((32 >> kL) - 1)) == 0 && t < nt) {
            const __int128 s =
                (__int128)A0[0] + ((__int128)A1[0] << 15) + ((__int128)A2[0] << 30);
            const unsigned long long lo = (unsigned long long)s;
            const unsigned long long hi = (unsigned long long)(s >> 64);
            unsigned long long *dst = sums + ((long long)(t0 + t) * E + e) * 3;
            atomicAdd(dst, lo & ((1ull << 40) - 1));
            atomicAdd(dst + 1, (lo >> 40) | ((hi & 0xFFFFull) << 24));
            atomicAdd(dst + 2, (unsigned long long)((long long)hi >> 16));
            __threadfence();
        }
    }
    if (fg.xsum) {   // this CTA's share of the (token, group) sums of its K slice
        const int G = H / kGroup;
        for (int p = xs_p0; p < nt * gps; p += xs_step) {
            const int t = p / gps, gg = p - t * gps;
            group_sum128_store(
                p == xs_p0 ? xs_v
                           : group_sum128_load(reinterpret_cast<const __half *>(x) +
                                               (long long)(t0 + t) * H + k0 + gg * kGroup),
                fg.xsum + (((long long)(t0 + t) * G + k0 / kGroup + gg) << fg.xsplit), fg.xsplit);
        }
    }
    if (bad)
        atomicOr(status, MOE_STATUS_NONFINITE);
    // the last CTA of this token block to finish ranks its tokens
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned total = gridDim.x * gridDim.z;
        last_cta = atomicAdd(&tickets[blockIdx.y], 1u) == total - 1;
    }
    __syncthreads();
    if (!last_cta)
        return;
    __threadfence();
    // every thread rounds a share of the block's (token, expert) sums, then
    // warp t ranks token t
    float *lsm = reinterpret_cast<float *>(xs);
    for (int i = threadIdx.x; i < nt * E; i += 2 * blockDim.x) {
        // two sums per step: both loads in flight before either is cleared
        const int i2 = i + blockDim.x;
        const int t = i / E, e2 = i - t * E;
        const int u = i2 / E, f2 = i2 - u * E;
        const Limbs a = exact_limbs(t0 + t, e2, sums, E);
        Limbs b{0ull, 0ull, 0ull};
        if (i2 < nt * E)
            b = exact_limbs(t0 + u, f2, sums, E);
        const float la = exact_finish(a, t0 + t, e2, sums, E, bias);
        lsm[i] = la;
        if (logits)
            logits[(long long)(t0 + t) * E + e2] = la;
        if (i2 < nt * E) {
            const float lb = exact_finish(b, t0 + u, f2, sums, E, bias);
            lsm[i2] = lb;
            if (logits)
                logits[(long long)(t0 + u) * E + f2] = lb;
        }
    }
    __syncthreads();
    if (warp < nt) {
        float lv[kPer];
#pragma unroll
        for (int i = 0; i < kPer; i++) {
            const int e2 = lane + 32 * i;
            lv[i] = e2 < E ? lsm[warp * E + e2] : 0.f;
        }
        select_topk<kPer>(lv, valid_mask<kPer>(E, lane), k, t0 + warp, idx, wout);
    }
    if (threadIdx.x == 0)
        tickets[blockIdx.y] = 0;
    if (fg.on)   // the logits in shared memory are no longer needed
        group_if_last(fg, gridDim.y, idx, n, k, E, reinterpret_cast<int *>(xs), &last_cta);
}

// ------------------------------------------------------------ large batches
//
// For many tokens the exact dot products of every (token, expert) pair cost
// far more than the routing decision needs.  The large-batch route computes
// approximate logits with fp32 FMAs (a tiled SIMT GEMM), bounds their error
// rigorously, and computes exact logits (the same exact integer sum, rounded
// once, plus the bias) only for the experts that could still be among a
// token's k best.  An expert is dropped only when k others are certainly
// above it, so the selection, the logits it uses and the softmax weights are
// identical to the exact route's.
//
// Error bound: every approximate logit is a sum of H exact products in fp32,
// each term passing through at most H + ks roundings of relative size 2^-24
// (sequential FMAs within a K slice, then the atomic merge of ks slices), so
// |approx - exact| <= (H + ks) 2^-24 sum |x_h w_h| / (1 - (H + ks) 2^-24)
// <= (H + ks) 2^-24 ||x||_2 ||w||_2 (1 + small), taken here with a factor 2
// of margin; the rounding of the exact sum to fp32 and of the bias add add at
// most 2^-23 |logit| each.

constexpr int kApT = 64, kApE = 64, kApK = 32;   // approx tile: tokens, experts, K chunk

__global__ void __launch_bounds__(256) router_approx_kernel(const __half *__restrict__ x,
                                                            const __half *__restrict__ rw, int n,
                                                            int H, int E, int kz,
                                                            float *__restrict__ approx)
{
    __shared__ __align__(16) float xs_s[kApK][kApT + 4];
    __shared__ __align__(16) float ws_s[kApK][kApE + 4];
    pdl_enter();
    const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
    const int t0 = blockIdx.y * kApT, e0 = blockIdx.x * kApE;
    const int kbeg = blockIdx.z * kz, kend = min(H, kbeg + kz);
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; i++)
#pragma unroll
        for (int j = 0; j < 4; j++)
            acc[i][j] = 0.f;
    const int r = tid >> 2, c8 = (tid & 3) * 8;   // staging: row r, halves c8 .. c8 + 7
    for (int kc = kbeg; kc < kend; kc += kApK) {
        uint4 xv = make_uint4(0u, 0u, 0u, 0u), wv = make_uint4(0u, 0u, 0u, 0u);
        if (t0 + r < n)
            xv = *reinterpret_cast<const uint4 *>(x + (long long)(t0 + r) * H + kc + c8);
        if (e0 + r < E)
            wv = *reinterpret_cast<const uint4 *>(rw + (long long)(e0 + r) * H + kc + c8);
        const __half2 *xh = reinterpret_cast<const __half2 *>(&xv);
        const __half2 *wh = reinterpret_cast<const __half2 *>(&wv);
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const float2 xf = __half22float2(xh[i]), wf = __half22float2(wh[i]);
            xs_s[c8 + 2 * i][r] = xf.x;
            xs_s[c8 + 2 * i + 1][r] = xf.y;
            ws_s[c8 + 2 * i][r] = wf.x;
            ws_s[c8 + 2 * i + 1][r] = wf.y;
        }
        __syncthreads();
#pragma unroll 8
        for (int kk = 0; kk < kApK; kk++) {
            const float4 a = *reinterpret_cast<const float4 *>(&xs_s[kk][4 * ty]);
            const float4 b = *reinterpret_cast<const float4 *>(&ws_s[kk][4 * tx]);
            const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
            for (int i = 0; i < 4; i++)
#pragma unroll
                for (int j = 0; j < 4; j++)
                    acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const int t = t0 + 4 * ty + i;
        if (t >= n)
            continue;
#pragma unroll
        for (int j = 0; j < 4; j++) {
            const int e = e0 + 4 * tx + j;
            if (e < E)
                atomicAdd(approx + (long long)t * E + e, acc[i][j]);
        }
    }
}

constexpr int kRfCand = 64;   // candidates per round of the refine kernel

// Exact partial sum, as a 128-bit integer at scale 2^-48, of the fp16
// products of x and w over h in [h0, h1) (8-element steps per lane).
// Warp-collective; lane 0 returns the warp's total.
__device__ __forceinline__ void exact_partial(const uint16_t *__restrict__ xr,
                                              const uint16_t *__restrict__ wr, int h0, int h1,
                                              int &bad, unsigned long long &lo_out,
                                              unsigned long long &hi_out)
{
    const int lane = threadIdx.x & 31;
    long long A0 = 0, A1 = 0, A2 = 0;
    for (int h = h0 + lane * 8; h < h1; h += 256) {
        const uint4 xv = *reinterpret_cast<const uint4 *>(xr + h);
        const uint4 wv = *reinterpret_cast<const uint4 *>(wr + h);
        const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w}, ww[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
        for (int i = 0; i < 8; i++) {
            const int2 a = split_half((xw[i >> 1] >> (16 * (i & 1))) & 0xFFFF, bad);
            const int2 b = split_half((ww[i >> 1] >> (16 * (i & 1))) & 0xFFFF, bad);
            A0 += (long long)a.x * b.x;
            A1 += (long long)a.x * b.y;
            A1 += (long long)a.y * b.x;
            A2 += (long long)a.y * b.y;
        }
    }
    const __int128 s = (__int128)A0 + ((__int128)A1 << 15) + ((__int128)A2 << 30);
    unsigned long long lo = (unsigned long long)s;
    unsigned long long hi = (unsigned long long)(s >> 64);
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) {
        const unsigned long long olo = __shfl_xor_sync(0xffffffffu, lo, d);
        const unsigned long long ohi = __shfl_xor_sync(0xffffffffu, hi, d);
        const unsigned long long nlo = lo + olo;
        hi = hi + ohi + (nlo < lo ? 1ull : 0ull);
        lo = nlo;
    }
    lo_out = lo;
    hi_out = hi;
}

// One CTA of 8 warps per token: bounds from the approximate logits (read and
// cleared for the next call), the candidate set, exact logits of the
// candidates (the 8 warps split H, exact 128-bit partials summed by warp 0),
// then the same top-k and softmax as the exact route.
template <int kPer>
__global__ void __launch_bounds__(256) router_refine_kernel(
    const __half *__restrict__ x, const __half *__restrict__ rw, const float *__restrict__ rnorm,
    int n, int H, int E, int k, int ks, float *approx, const float *__restrict__ bias,
    int32_t *__restrict__ idx, float *__restrict__ wout, int *__restrict__ status,
    const RouteExtras fg)
{
    extern __shared__ int gsm[];   // the fused grouping's work space
    __shared__ float red_f[8];
    __shared__ int cand_e[kRfCand];
    __shared__ int n_round;
    __shared__ unsigned long long part[8][kRfCand][2];
    pdl_enter();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x;
    const uint16_t *xr = reinterpret_cast<const uint16_t *>(x) + (long long)t * H;
    // ||x_t||^2 in fp32
    float s2 = 0.f;
    for (int h = threadIdx.x * 8; h < H; h += 256 * 8) {
        const uint4 v = *reinterpret_cast<const uint4 *>(xr + h);
        const __half2 *p = reinterpret_cast<const __half2 *>(&v);
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const float2 f = __half22float2(p[i]);
            s2 = fmaf(f.x, f.x, s2);
            s2 = fmaf(f.y, f.y, s2);
        }
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1)
        s2 += __shfl_xor_sync(0xffffffffu, s2, d);
    if (lane == 0)
        red_f[warp] = s2;
    __syncthreads();
    s2 = 0.f;
#pragma unroll
    for (int w = 0; w < 8; w++)
        s2 += red_f[w];
    // bounds and candidates (warp 0)
    const float gam = 2.0f * (float)(H + ks + 8) * 5.9604644775390625e-08f;
    const float scale = gam * sqrtf(s2) * 1.001f;
    const unsigned valid = valid_mask<kPer>(E, lane);
    unsigned cand = 0;
    float lv[kPer];
    if (warp == 0) {
        float lo[kPer], hi[kPer];
#pragma unroll
        for (int i = 0; i < kPer; i++) {
            const int e = lane + 32 * i;
            lo[i] = -INFINITY;
            hi[i] = INFINITY;
            lv[i] = -INFINITY;
            if (e < E) {
                float *p = approx + (long long)t * E + e;
                const float a = __ldcg(p);
                __stcg(p, 0.f);
                const float bb = bias ? bias[e] : 0.f;
                const float b = scale * rnorm[e];
                const float c = a + bb;
                const float m = b + 2.4e-7f * (fabsf(a) + fabsf(bb) + b + fabsf(c)) + 1e-30f;
                if (isfinite(c - m) && isfinite(c + m)) {
                    lo[i] = c - m;
                    hi[i] = c + m;
                }
            }
        }
        // T = k-th largest lower bound; an expert whose upper bound is below T
        // has k experts certainly above it
        unsigned taken = 0;
        float T = -INFINITY;
        for (int j = 0; j < k; j++) {
            float bv = -INFINITY;
            int be = -1;
#pragma unroll
            for (int i = 0; i < kPer; i++)
                if (((valid >> i) & 1u) && !((taken >> i) & 1u) && (be < 0 || lo[i] > bv)) {
                    bv = lo[i];
                    be = lane + 32 * i;
                }
#pragma unroll
            for (int d = 16; d > 0; d >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, d);
                const int oe = __shfl_xor_sync(0xffffffffu, be, d);
                if (oe >= 0 && (be < 0 || ov > bv || (ov == bv && oe < be))) {
                    bv = ov;
                    be = oe;
                }
            }
            if (be >= 0 && (be & 31) == lane)
                taken |= 1u << (be >> 5);
            T = bv;
        }
#pragma unroll
        for (int i = 0; i < kPer; i++)
            if (((valid >> i) & 1u) && hi[i] >= T)
                cand |= 1u << i;
    } else if (fg.xsum) {   // the token's activation group sums, by warps 1..7
        const int G = H / kGroup;
        for (int gg = warp - 1; gg < G; gg += 7)
            group_sum128_store(group_sum128_load(x + (long long)t * H + gg * kGroup),
                               fg.xsum + (((long long)t * G + gg) << fg.xsplit), fg.xsplit);
    }
    // exact logits of the candidates, in rounds of up to kRfCand
    int bad = 0;
    int next_i = 0;   // warp 0: candidate enumeration cursor (slot i, then lanes)
    unsigned rest = cand;
    for (;;) {
        if (warp == 0) {
            int cnt = 0;
            for (; next_i < kPer && cnt < kRfCand; next_i++) {
                const unsigned m = __ballot_sync(0xffffffffu, (rest >> next_i) & 1u);
                const int c = __popc(m);
                if (cnt + c > kRfCand)
                    break;
                if ((rest >> next_i) & 1u)
                    cand_e[cnt + __popc(m & ((1u << lane) - 1u))] = lane + 32 * next_i;
                cnt += c;
            }
            if (lane == 0)
                n_round = cnt;
        }
        __syncthreads();
        const int nr = n_round;
        if (nr == 0)
            break;
        const int h0 = warp * (H / 8), h1 = h0 + H / 8;
        for (int c = 0; c < nr; c++) {
            const int e = cand_e[c];
            unsigned long long plo, phi;
            exact_partial(xr, reinterpret_cast<const uint16_t *>(rw) + (long long)e * H, h0, h1,
                          bad, plo, phi);
            if (lane == 0) {
                part[warp][c][0] = plo;
                part[warp][c][1] = phi;
            }
        }
        __syncthreads();
        if (warp == 0) {
            for (int c = 0; c < nr; c++) {
                unsigned long long lo = 0, hi = 0;
#pragma unroll
                for (int w = 0; w < 8; w++) {
                    const unsigned long long nlo = lo + part[w][c][0];
                    hi = hi + part[w][c][1] + (nlo < lo ? 1ull : 0ull);
                    lo = nlo;
                }
                const int e = cand_e[c];
                float l = round_scaled(lo, (long long)hi);
                if (bias)
                    l = __fadd_rn(l, bias[e]);
#pragma unroll
                for (int i = 0; i < kPer; i++)
                    if ((e >> 5) == i && (e & 31) == lane)
                        lv[i] = l;
            }
        }
        __syncthreads();
    }
    if (warp == 0)
        select_topk<kPer>(lv, cand, k, t, idx, wout);
    if (bad)
        atomicOr(status, MOE_STATUS_NONFINITE);
    if (fg.on)
        group_if_last(fg, gridDim.x, idx, n, k, E, gsm, &n_round);
}

// Upper bounds of the router rows' 2-norms (fp64 sums of exact squares,
// rounded up).  One warp per expert; run once at layer creation.
__global__ void router_rnorm_kernel(const __half *__restrict__ rw, int H, int E,
                                    float *__restrict__ rnorm)
{
    const int e = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (e >= E)
        return;
    double s = 0.0;
    for (int h = lane; h < H; h += 32) {
        const double v = (double)__half2float(rw[(long long)e * H + h]);
        s += v * v;
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1)
        s += __shfl_xor_sync(0xffffffffu, s, d);
    if (lane == 0)
        rnorm[e] = __double2float_ru(sqrt(s) * (1.0 + 1e-9));
}

cudaError_t launch_router_rnorm(const LayerDev &L, float *rnorm, cudaStream_t st)
{
    router_rnorm_kernel<<<(L.E + 7) / 8, 256, 0, st>>>(L.router_w, L.H, L.E, rnorm);
    return cudaGetLastError();
}

template <int kPer>
static cudaError_t route_large_impl(const LayerDev &L, const Workspace &ws, const __half *x, int n,
                                    int num_sms, const RouteExtras &fg, cudaStream_t st)
{
    const int tiles = ((L.E + kApE - 1) / kApE) * ((n + kApT - 1) / kApT);
    int ks = (2 * num_sms + tiles - 1) / tiles;
    ks = max(1, min(ks, L.H / kApK));
    const int kz = ((L.H / ks + kApK - 1) / kApK) * kApK;
    ks = (L.H + kz - 1) / kz;
    const dim3 grid((L.E + kApE - 1) / kApE, (n + kApT - 1) / kApT, ks);
    cudaError_t e = launch_pdl(router_approx_kernel, grid, dim3(256), 0, st, x, L.router_w, n, L.H,
                               L.E, kz, ws.approx);
    if (e != cudaSuccess)
        return e;
    return launch_pdl(router_refine_kernel<kPer>, dim3(n), dim3(256),
                      fg.on ? fused_group_smem(L.E) : 0, st, x, L.router_w,
                      static_cast<const float *>(ws.rnorm), n, L.H, L.E, L.k, ks, ws.approx,
                      L.router_bias, ws.idx, ws.w, ws.hdr + 2, fg);
}

cudaError_t launch_route_large(const LayerDev &L, const Workspace &ws, const __half *x, int n,
                               int num_sms, const RouteExtras &fg, cudaStream_t st)
{
    if (L.E <= 64)
        return route_large_impl<2>(L, ws, x, n, num_sms, fg, st);
    if (L.E <= 128)
        return route_large_impl<4>(L, ws, x, n, num_sms, fg, st);
    if (L.E <= 256)
        return route_large_impl<8>(L, ws, x, n, num_sms, fg, st);
    if (L.E <= 512)
        return route_large_impl<16>(L, ws, x, n, num_sms, fg, st);
    return route_large_impl<32>(L, ws, x, n, num_sms, fg, st);
}

template <int kPer>
static void configure_one(size_t smem)
{
    cudaFuncSetAttribute(router_kernel<kPer, kRtTok>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)smem);
    cudaFuncSetAttribute(router_kernel<kPer, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)smem);
    cudaFuncSetAttribute(router_kernel<kPer, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)smem);
    cudaFuncSetAttribute(router_refine_kernel<kPer>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)fused_group_smem(kMaxExperts));
}

void configure_router_kernel(size_t smem)
{
    configure_one<2>(smem);
    configure_one<4>(smem);
    configure_one<8>(smem);
    configure_one<16>(smem);
    configure_one<32>(smem);
}

// Dynamic shared memory of a routing CTA: the split activations of its K
// slice, later reused for its tokens' logits.
static size_t router_smem(int tok, int kslice, int E)
{
    const size_t a = (size_t)tok * kslice * sizeof(int2), b = (size_t)tok * E * sizeof(float);
    return a > b ? a : b;
}

template <int kPer, int kTok>
static cudaError_t route_tok(const LayerDev &L, const Workspace &ws, const __half *x, int n,
                             int ks, float *lg, const RouteExtras &fg, cudaStream_t st)
{
    const int kslice = L.H / ks;
    const dim3 grid((L.E + kRtWarps - 1) / kRtWarps, (n + kTok - 1) / kTok, ks);
    size_t smem = router_smem(kTok, kslice, L.E);
    if (fg.on && fused_group_smem(L.E) > smem)
        smem = fused_group_smem(L.E);
    return launch_pdl(router_kernel<kPer, kTok>, grid, dim3(kRtWarps * 32), smem, st,
                      reinterpret_cast<const uint16_t *>(x),
                      reinterpret_cast<const uint16_t *>(L.router_w), n, L.H, L.E, L.k, kslice,
                      ws.sums, ws.tickets, L.router_bias, ws.idx, ws.w, lg, ws.hdr + 2, fg);
}

template <int kPer>
static cudaError_t route_impl(const LayerDev &L, const Workspace &ws, const __half *x, int n,
                              int ks, float *lg, const RouteExtras &fg, cudaStream_t st)
{
    if (n == 1)
        return route_tok<kPer, 1>(L, ws, x, n, ks, lg, fg, st);
    if (n <= 4)
        return route_tok<kPer, 4>(L, ws, x, n, ks, lg, fg, st);
    return route_tok<kPer, kRtTok>(L, ws, x, n, ks, lg, fg, st);
}

template <int kPer, int kTok>
static void route_scratch_tok(const uint16_t *xb, const uint16_t *wb, const float *bias, int n,
                              int H, int E, int k, int ks, unsigned long long *sums,
                              unsigned *tickets, int *status, int32_t *idx, float *w,
                              cudaStream_t st)
{
    const int kslice = H / ks;
    const dim3 grid((E + kRtWarps - 1) / kRtWarps, (n + kTok - 1) / kTok, ks);
    const size_t smem = router_smem(kTok, kslice, E);
    router_kernel<kPer, kTok><<<grid, kRtWarps * 32, smem, st>>>(
        xb, wb, n, H, E, k, kslice, sums, tickets, bias, idx, w, nullptr, status, RouteExtras{});
}

template <int kPer>
static void route_scratch(const uint16_t *xb, const uint16_t *wb, const float *bias, int n,
                          int H, int E, int k, int ks, unsigned long long *sums,
                          unsigned *tickets, int *status, int32_t *idx, float *w,
                          cudaStream_t st)
{
    if (n == 1)
        route_scratch_tok<kPer, 1>(xb, wb, bias, n, H, E, k, ks, sums, tickets, status, idx, w,
                                   st);
    else if (n <= 4)
        route_scratch_tok<kPer, 4>(xb, wb, bias, n, H, E, k, ks, sums, tickets, status, idx, w,
                                   st);
    else
        route_scratch_tok<kPer, kRtTok>(xb, wb, bias, n, H, E, k, ks, sums, tickets, status, idx,
                                        w, st);
}

// The same routing kernel on caller-provided scratch: sums [n][E] and
// tickets [ceil(n/8)] zero on entry (cleared again by the kernel), status one
// word.
cudaError_t launch_route_scratch(const __half *x, const __half *rw, const float *bias, int n,
                                 int H, int E, int k, int ks, unsigned long long *sums,
                                 unsigned *tickets,
                                 int *status, int32_t *idx, float *w, cudaStream_t st)
{
    const uint16_t *xb = reinterpret_cast<const uint16_t *>(x);
    const uint16_t *wb = reinterpret_cast<const uint16_t *>(rw);
    if (E <= 64)
        route_scratch<2>(xb, wb, bias, n, H, E, k, ks, sums, tickets, status, idx, w, st);
    else if (E <= 128)
        route_scratch<4>(xb, wb, bias, n, H, E, k, ks, sums, tickets, status, idx, w, st);
    else if (E <= 256)
        route_scratch<8>(xb, wb, bias, n, H, E, k, ks, sums, tickets, status, idx, w, st);
    else if (E <= 512)
        route_scratch<16>(xb, wb, bias, n, H, E, k, ks, sums, tickets, status, idx, w, st);
    else
        route_scratch<32>(xb, wb, bias, n, H, E, k, ks, sums, tickets, status, idx, w, st);
    return cudaGetLastError();
}

// Activation group sums of n tokens: one CTA per token, warp w takes the
// groups w, w + 8, ...
__global__ void __launch_bounds__(256) xsum_kernel(const __half *__restrict__ x, int H,
                                                   float *__restrict__ xsum, int split)
{
    pdl_enter();
    const int t = blockIdx.x, warp = threadIdx.x >> 5, G = H / kGroup;
    for (int gg = warp; gg < G; gg += 8)
        group_sum128_store(group_sum128_load(x + (long long)t * H + gg * kGroup),
                           xsum + (((long long)t * G + gg) << split), split);
}

cudaError_t launch_xsum(const LayerDev &L, const Workspace &ws, const __half *x, int n,
                        cudaStream_t st)
{
    return launch_pdl(xsum_kernel, dim3(n), dim3(256), 0, st, x, L.H, ws.xsum,
                      L.wbits == 2 ? 1 : 0);
}

cudaError_t launch_route(const LayerDev &L, const Workspace &ws, const __half *x, int n, int ks,
                         int want_logits, const RouteExtras &fg, cudaStream_t st)
{
    float *lg = want_logits ? ws.logits : nullptr;
    if (L.E <= 64)
        return route_impl<2>(L, ws, x, n, ks, lg, fg, st);
    if (L.E <= 128)
        return route_impl<4>(L, ws, x, n, ks, lg, fg, st);
    if (L.E <= 256)
        return route_impl<8>(L, ws, x, n, ks, lg, fg, st);
    if (L.E <= 512)
        return route_impl<16>(L, ws, x, n, ks, lg, fg, st);
    return route_impl<32>(L, ws, x, n, ks, lg, fg, st);
}

}  // namespace qe
