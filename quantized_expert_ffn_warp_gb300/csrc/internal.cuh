// Internal declarations shared by the CUDA translation units of the layer.
#pragma once
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe_layer.h"

namespace qe {

// Programmatic dependent launch: the forward's kernels are launched so that
// each may start while its predecessor drains; every such kernel first
// waits for the predecessor's completion (and memory) before it touches
// global memory, then lets its own successor launch.
__device__ __forceinline__ void pdl_enter()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t st, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

constexpr int kGroup = 128;      // quantisation group along K

// Sum of the 128 fp16 values p[0..127] (one quantisation group of one
// activation row) in fp32, in one fixed order: lane l adds p[4l..4l+3] in
// sequence, then a butterfly over the lanes.  Warp-collective; every lane
// returns the sum.  The same order wherever it is computed, so the sums do
// not depend on which kernel produced them.
// The lane's share of a group (issue early, reduce later).
__device__ __forceinline__ uint2 group_sum128_load(const __half *p)
{
    return *reinterpret_cast<const uint2 *>(p + 4 * (threadIdx.x & 31));
}

__device__ __forceinline__ float group_sum128_reduce(uint2 v)
{
    const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&v.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&v.y));
    float s = ((a.x + a.y) + b.x) + b.y;
#pragma unroll
    for (int d = 16; d > 0; d >>= 1)
        s += __shfl_xor_sync(0xffffffffu, s, d);
    return s;
}

__device__ __forceinline__ float group_sum128(const __half *p)
{
    return group_sum128_reduce(group_sum128_load(p));
}

// The group sum of v (as group_sum128_reduce) into dst[0] by lane 0, or with
// split the two partial sums over the positions k % 4 < 2 and k % 4 >= 2
// into dst[0], dst[1] (the 2-bit gate/up kernels scale the activations of
// the latter by 1/16 before the MMA).  Every lane of the warp calls it.
__device__ __forceinline__ void group_sum128_store(uint2 v, float *dst, int split)
{
    const int lane = threadIdx.x & 31;
    if (!split) {
        const float s = group_sum128_reduce(v);
        if (lane == 0)
            dst[0] = s;
        return;
    }
    const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&v.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&v.y));
    float lo = a.x + a.y, hi = b.x + b.y;
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) {
        lo += __shfl_xor_sync(0xffffffffu, lo, d);
        hi += __shfl_xor_sync(0xffffffffu, hi, d);
    }
    if (lane == 0) {
        dst[0] = lo;
        dst[1] = hi;
    }
}
constexpr int kRowTile = 16;     // rows per packed tile (MMA M)
constexpr int kChunkBytes = 512; // packed bytes per (row tile, chunk): 32 lanes x 16 B

// Slot of lane (g = lane / 4, t = lane % 4)'s 16-byte word inside a 512-byte
// chunk: the words of row pair g sit in 64-byte run g, rotated by g / 2, so
// that both the 8 lanes of a quarter warp (two runs) and the 8 row pairs
// reading their runs' t-th words (the tensor-memory dequantisation) touch 8
// different 16-byte bank groups.
__host__ __device__ __forceinline__ int chunk_slot(int g, int t)
{
    return 4 * g + ((t + (g >> 1)) & 3);
}
constexpr int kMetaBytes = 48;   // per (row tile, group): 16 fp16 scales + 16 u8 zeros
constexpr int kMaxTokTile = 8;   // tokens per decode work entry (one MMA N tile)
// Tokens per GEMM work entry (tcgen05 MMA N): 64, or 128 for calls that
// average at least 128 tokens per expert (gemm.cu); the workspace is sized
// for the smaller.
constexpr int kGemmTok = 64;
constexpr int kGemmTokWide = 128;
constexpr int kMaxExperts = 1024;
constexpr int kMaxTopK = 32;
constexpr int kPhases = 5;  // route, group, gate_up, down, combine

// Packed weight records of one stream (the gate/up pair, or down) for every
// expert: [E][128-row tile][K/128][upt units][rec].  A record holds two slots of one 16-row
// tile and 128-group each: the CPG chunks of 512 bytes of codes (CPG = 2 for
// 4-bit, 1 for 2-bit) followed by the 48-byte scale/zero block, so the bytes a
// warp needs for one group are one contiguous run.  Gate/up: a unit is one
// row tile, the slots are the gate and the up matrix.  Down (paired): a unit
// is two consecutive row tiles 2p, 2p+1 of the one matrix, in slots 0 and 1.
struct PackedRecs {
    const uint8_t *recs;
    int n_rt, n_groups;      // units (row tiles, or row-tile pairs), 128-groups along K
    int pair;                // 1: a unit is two row tiles of one matrix
    int upt;                 // units per 128-row tile (8, or 4 pairs)
    int rec;                 // bytes per (unit, group) record
    long long expert_bytes;  // bytes per expert
    // Tiered layers: base of each routed expert's records in device memory
    // ([E], written by the staging kernels before the FFN kernels run); null
    // for a layer whose experts are all at recs + e * expert_bytes.
    const uint8_t *const *ebase;
};

// Base of routed expert e's records (the shared expert is never tiered).
__device__ __forceinline__ const uint8_t *expert_records(const PackedRecs &pr, long long e)
{
    return pr.ebase ? pr.ebase[e] : pr.recs + e * pr.expert_bytes;
}

// Work entry: `ntok` tokens (<= kMaxTokTile) of expert `expert` (E = the
// shared expert) whose rows in the sorted activation buffers start at `start`;
// tok[i] is the token of row start + i (tok[i] = tok[0] for i >= ntok, so
// every slot names a valid row).
struct Entry {
    int expert, start, ntok, pad;
    int tok[kMaxTokTile];
};

struct Workspace {
    int *hdr;               // [0] routed / [1] shared decode entries, [2] status bits,
                            // [4] routed / [5] shared GEMM entries
    Entry *entries;         // [max_entries]
    int4 *gentries;         // [max_gentries] GEMM entries (expert, start, ntok, 0)
    __half *xs;             // [P + n][H] x rows in sorted-position order (GEMM path)
    int32_t *idx;           // [P] top-k expert ids
    float *w;               // [P] top-k weights
    int32_t *counts;        // [E]
    int32_t *offsets;       // [E+1]
    int32_t *perm;          // [P]
    int32_t *pos_of_pair;   // [P] sorted position of pair p (-1: skipped)
    int32_t *tok_of_pos;    // [P + n] token of sorted position
    float *logits;          // [n][E]
    float *approx;          // [n][E] approximate logits of the large-batch route; zero between calls
    float *rnorm;           // [E] upper bounds of the router rows' 2-norms (layer constant)
    unsigned long long *sums;   // [n][E][3] exact router sums as 40/40/48-bit limbs; zero between calls
    unsigned *tickets;      // [ceil(n/8) + 1] router CTAs finished per token block, then
                            // token blocks (or tokens) finished per call; zero between calls
    float *xsum;            // [n][H/128] group sums of the tokens' activations (gate/up zero
                            // points); 2-bit layers: [n][H/128][2] partial sums
    __half *xn;             // [n][H] RMSNorm-ed tokens of a forward with the norm in front
    __half *h;              // [P + n][max(I, I_sh)] SwiGLU activations
    float *y;               // [P + n][H] expert outputs
    int max_entries, max_gentries;
};

// Extra outputs of a routing launch.
// Grouping: for calls of at most kFusedPairs (token, expert) pairs the last
// CTA of the whole call (a call-wide ticket) groups the pairs, with the same
// outputs as the separate grouping kernel, and the forward skips that launch
// (on = 0: no grouping).
// Activation group sums: with xsum set, the launch also writes the fp32 sum of
// every (token, 128-group) of x (group_sum128), which the gate/up kernels use
// for the zero-point term.
constexpr int kFusedPairs = 256;
struct RouteExtras {
    int on;                 // 1: group the pairs at the end of routing
    int big;                // experts with >= big tokens get GEMM entries (0: none)
    int gtok;               // tokens per GEMM entry (kGemmTok or kGemmTokWide)
    int has_shared;
    unsigned *ticket;       // call-wide ticket, zero between calls
    int *hdr;
    Entry *entries;
    int4 *gentries;
    int32_t *counts, *offsets, *perm, *pos_of_pair, *tok_of_pos;
    float *xsum;            // [n][H/128] or null
    int xsplit;             // 1: [n][H/128][2] partial sums (2-bit layers)
};
// Dynamic shared memory of the fused grouping (256 threads).
__host__ __device__ constexpr size_t fused_group_smem(int E)
{
    return sizeof(int) * (8 * (size_t)E + 4 * (size_t)E + kFusedPairs + 3 * 8 + 3);
}

struct LayerDev {
    int H, I, E, k, wbits, has_shared, I_sh, residual, max_tokens;
    PackedRecs gu, dn;          // routed experts
    PackedRecs sh_gu, sh_dn;    // shared expert
    const __half *router_w;     // [E][H]
    const float *router_bias;   // [E] or null
    const __half *sh_gate_w;    // [H]
};

// ---- kernels / launchers (defined in their .cu files) --------------------
// Repack matrix `m` (of `mats`) of a stream from the canonical layout into
// the records `out` (see PackedRecs).
cudaError_t launch_repack(const uint8_t *codes, const uint16_t *scales, const uint8_t *zeros,
                          int n_exp, int rows, int K, int wbits, int m, int mats, int pair,
                          uint8_t *out, cudaStream_t st);

// Router logits, top-k and softmax weights in one launch (K split in ks
// slices); with fg.on the same launch also groups the pairs, and with fg.xsum
// it writes the activation group sums.
cudaError_t launch_route(const LayerDev &L, const Workspace &ws, const __half *x, int n, int ks,
                         int want_logits, const RouteExtras &fg, cudaStream_t st);
// The same routing for large batches: approximate logits with an error bound,
// exact logits of the candidate experts only (identical results).
cudaError_t launch_route_large(const LayerDev &L, const Workspace &ws, const __half *x, int n,
                               int num_sms, const RouteExtras &fg, cudaStream_t st);
cudaError_t launch_router_rnorm(const LayerDev &L, float *rnorm, cudaStream_t st);
// Grouping; experts with at least `big` tokens (big > 0) go to the GEMM path.
cudaError_t launch_group(const LayerDev &L, const Workspace &ws, int n, int big, int gtok,
                         cudaStream_t st);
// x rows in sorted-position order for the GEMM path (routed pairs, then the
// shared expert's tokens).
cudaError_t launch_gather(const LayerDev &L, const Workspace &ws, const __half *x, int n,
                          cudaStream_t st);
// tcgen05 grouped GEMM over the GEMM entries; `bmap` is the TMA map of the B
// operand source (xs for gate/up, h for down); gtok: tokens per GEMM entry
// (kGemmTok or kGemmTokWide, as the grouping used).
cudaError_t launch_gemm_gateup(const LayerDev &L, const Workspace &ws, const CUtensorMap &bmap,
                               int gtok, int grid, cudaStream_t st);
cudaError_t launch_gemm_down(const LayerDev &L, const Workspace &ws, const CUtensorMap &bmap,
                             int gtok, int grid, cudaStream_t st);
void configure_gemm_kernels();
// Decode FFN kernels (entries of at most kMaxTokTile tokens).
cudaError_t launch_gateup(const LayerDev &L, const Workspace &ws, const __half *x, int grid,
                          cudaStream_t st);
cudaError_t launch_down(const LayerDev &L, const Workspace &ws, int grid, cudaStream_t st);
// Group sums of the activations of n tokens (into ws.xsum), for calls whose
// routing was given by the caller (the routing launches write them otherwise).
cudaError_t launch_xsum(const LayerDev &L, const Workspace &ws, const __half *x, int n,
                        cudaStream_t st);
// x: the layer's input tokens (shared-expert gate); xres: the residual rows.
cudaError_t launch_combine(const LayerDev &L, const Workspace &ws, const __half *x,
                           const __half *xres, __half *out, int n, cudaStream_t st);
// Expert residency tiers: per call, find the touched experts that live in
// host memory, give each a device slot (hits keep theirs, misses take the
// least recently used free ones) and copy the misses' records into them.
constexpr int kPinned = -2;   // slot_of[e] of a resident expert
constexpr int kNoSlot = -1;   // slot_of[e] of a cold expert without a slot

// Device state of a tiered layer (device pointers, except host_*: pinned host
// memory mapped for the device).
struct TierDev {
    int E, S;                       // experts, slots
    int *slot_of;                   // [E] slot of expert e, kNoSlot, or kPinned
    int *slot_expert;               // [S] expert held by slot s, or -1
    unsigned *slot_used;            // [S] last call that used slot s (0: never)
    unsigned *call;                 // [1] calls staged so far
    int *copies;                    // [S] slot of each miss of the call, then [S] its expert
    int *n_copy;                    // [1] misses of the call that got a slot
    unsigned long long *stats;      // [2] hits, misses over all calls
    int *status;                    // the layer's device status word
    const uint8_t **ebase_gu, **ebase_dn;   // [E] record bases the FFN kernels read
    uint8_t *slot_gu, *slot_dn;     // [S] slots of each stream
    const uint8_t *host_gu, *host_dn;       // every expert's records (mapped host memory)
    const uint8_t *zero;            // an all-zero expert of the larger stream (device)
    long long gu_bytes, dn_bytes;   // bytes of one expert per stream
};
cudaError_t launch_stage(const TierDev &t, const Workspace &ws, int num_sms, cudaStream_t st);
// Kernel copy of `bytes` (a multiple of 16) between device-reachable buffers.
cudaError_t launch_copy(void *dst, const void *src, size_t bytes, int num_sms, cudaStream_t st);
// Two-pass RMSNorm of r [n][H] with gain g [H] into xn [n][H].
cudaError_t launch_rmsnorm(const __half *r, const __half *g, float eps, int n, int H,
                           __half *xn, cudaStream_t st);

int ffn_blocks_per_sm(int wbits);
size_t group_smem_bytes(int E);

}  // namespace qe
