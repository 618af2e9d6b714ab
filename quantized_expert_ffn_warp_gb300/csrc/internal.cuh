// Internal declarations shared by the CUDA translation units of the layer.
#pragma once
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe_layer.h"

namespace qe {

constexpr int kGroup = 128;      // quantisation group along K
constexpr int kRowTile = 16;     // rows per packed tile (MMA M)
constexpr int kChunkBytes = 512; // packed bytes per (row tile, chunk): 32 lanes x 16 B
constexpr int kMetaBytes = 48;   // per (row tile, group): 16 fp16 scales + 16 u8 zeros
constexpr int kMaxTokTile = 16;  // tokens per FFN work entry (2 MMA N tiles)
constexpr int kMaxExperts = 1024;
constexpr int kMaxTopK = 32;
constexpr int kPhases = 6;

// One packed matrix type (gate, up or down) for every expert.
// codes: [E][rows/16][K/chunkK][32 lanes] uint4; meta: [E][rows/16][K/128][48 B].
// chunkK = 64 (4-bit) or 128 (2-bit): one 16-byte lane word covers 4 (4-bit)
// or 8 (2-bit) MMA k-steps of 16.
struct PackedMat {
    const uint4 *codes;
    const uint8_t *meta;
    int rows, K;
    int n_rt, n_chunks, n_groups;
    long long expert_codes;  // uint4 per expert
    long long expert_meta;   // bytes per expert
};

// Work entry: `ntok` tokens (<= kMaxTokTile) of expert `expert` (E = the
// shared expert) whose rows in the sorted activation buffers start at `start`.
struct Entry {
    int expert, start, ntok, pad;
};

struct Workspace {
    int *hdr;               // [0] routed entries, [1] shared entries, [2] status bits
    Entry *entries;         // [max_entries]
    int32_t *idx;           // [P] top-k expert ids
    float *w;               // [P] top-k weights
    int32_t *counts;        // [E]
    int32_t *offsets;       // [E+1]
    int32_t *perm;          // [P]
    int32_t *pos_of_pair;   // [P] sorted position of pair p (-1: skipped)
    int32_t *tok_of_pos;    // [P + n] token of sorted position
    float *logits;          // [n][E]
    ulonglong2 *partials;   // [ks][n][E] exact router partial sums (lo, hi)
    float *sh_gate;         // [n] sigmoid gate of the shared expert
    __half *h;              // [P + n][max(I, I_sh)] SwiGLU activations
    float *y;               // [P + n][H] expert outputs
    int max_entries;
};

struct LayerDev {
    int H, I, E, k, wbits, has_shared, I_sh, residual, max_tokens;
    PackedMat mat[3], sh[3];
    const __half *router_w;     // [E][H]
    const float *router_bias;   // [E] or null
    const __half *sh_gate_w;    // [H]
};

// ---- kernels / launchers (defined in their .cu files) --------------------
cudaError_t launch_repack(const uint8_t *codes, const uint16_t *scales, const uint8_t *zeros,
                          int n_exp, int rows, int K, int wbits, uint4 *out_codes,
                          uint8_t *out_meta, cudaStream_t st);

cudaError_t launch_router(const LayerDev &L, const Workspace &ws, const __half *x, int n, int ks,
                          cudaStream_t st);
cudaError_t launch_topk(const LayerDev &L, const Workspace &ws, int n, int ks, int want_logits,
                        cudaStream_t st);
cudaError_t launch_group(const LayerDev &L, const Workspace &ws, int n, cudaStream_t st);
cudaError_t launch_gateup(const LayerDev &L, const Workspace &ws, const __half *x, int n, int grid,
                          cudaStream_t st);
cudaError_t launch_down(const LayerDev &L, const Workspace &ws, int n, int grid, cudaStream_t st);
cudaError_t launch_combine(const LayerDev &L, const Workspace &ws, const __half *x, __half *out,
                           int n, cudaStream_t st);

int ffn_blocks_per_sm(int wbits);
size_t group_smem_bytes(int E);

}  // namespace qe
