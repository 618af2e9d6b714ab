// Host side of the C ABI declared in include/moe_layer.h: validation, weight
// repacking, workspace ownership and the stream-ordered launch sequence
//   router partial sums -> top-k + softmax -> grouping -> gate/up + SwiGLU ->
//   down -> combine + residual + shared expert.
// No host synchronisation and no allocation happen after moe_layer_create.
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdarg>
#include <cstdio>
#include <algorithm>
#include <cstring>
#include <new>
#include <vector>

#include "internal.cuh"

namespace qe {
void configure_group_kernel(size_t smem);
void configure_router_kernel(size_t smem);
void configure_ffn_kernels();
}  // namespace qe

// Default expert-FFN kernel choice of a 4-bit layer.  The decode kernels
// are bound by the work per record, and an expert with c tokens costs them
// ceil(c / 8) passes over its weights (one per 8-token entry); the GEMM
// kernels pass once, but one 128-row tile per SM at a time, so they pay off
// only when the experts that reach the threshold bring enough tiles to keep
// the SMs busy.  Layers whose routed expert alone has at least one gate/up
// tile per SM take experts of kDefaultGemmMinTokens (9: two entries or more)
// tokens and up to the GEMM kernels; the others keep every expert on the
// decode kernels, as do layers with hidden, inter or shared_inter below
// kShortKGemm (fewer than 4 steps per tile: the GEMM pipeline never fills).
// Measured: the 14336-wide 64-expert layer at 256 tokens 1463 us at 9
// against 1768 us decode only; the 4096-wide 64-expert layer at 64 tokens
// 304 us decode only against 327 us at 9 and 309 us at 33; the 512-expert
// layer (inter 1024) at 64 tokens 282 us against 304 us at 17 or 33.
constexpr int kDefaultGemmMinTokens = 9;
constexpr int kShortKGemm = 512;
// Routing computes exact logits only for the candidate experts (approximate
// logits with an error bound select them) from kLargeRouteTokens tokens on,
// or from kManyExpertTokens tokens when there are many experts; the all-pairs
// exact kernel stays for small batches, where it is one short launch.
constexpr int kLargeRouteTokens = 64;
constexpr int kLargeRouteExperts = 128;
constexpr int kManyExpertTokens = 8;
#ifndef QE_LARGE_ROUTE_ALL
#define QE_LARGE_ROUTE_ALL 0
#endif

using namespace qe;

namespace {

thread_local char g_err[512];

int fail(int code, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return code;
}

int ok()
{
    g_err[0] = 0;
    return MOE_OK;
}

constexpr int kProfRing = 256;

}  // namespace

namespace qe {
// moe_last_error() bookkeeping for entry points in other translation units.
int record_failure(int code, const char *msg) { return fail(code, "%s", msg); }
int record_success() { return ok(); }
}  // namespace qe

struct moe_layer {
    moe_cfg_t cfg{};
    LayerDev dev{};
    Workspace ws{};
    int device = 0;
    int num_sms = 0;
    int grid_ffn = 0;
    int gemm_min_tokens = 0;          // 0: every expert on the decode kernels
    CUtensorMap map_xs{}, map_h{};    // TMA maps of the GEMM path's B operands
    int64_t weight_bytes = 0, workspace_bytes = 0, expert_bytes = 0, shared_bytes = 0;
    std::vector<void *> allocs;
    // expert residency tiers (moe_layer_set_residency)
    int tiered = 0;                   // routed experts read through tier.ebase_*
    int n_resident = 0;
    TierDev tier{};
    std::vector<void *> tier_allocs;  // device memory of the tiers (resident, slots, state)
    void *host_gu = nullptr, *host_dn = nullptr;   // pinned host copies of every expert
    // per-phase timing
    int prof_on = 0, prof_active = 0;
    cudaEvent_t *prof_ev = nullptr;   // [kProfRing][kPhases + 1]
    int prof_head = 0, prof_pending = 0;
    double prof_ms[kPhases] = {};
    int prof_calls = 0;
};

namespace {

cudaError_t dalloc(moe_layer *L, void **p, size_t bytes)
{
    *p = nullptr;
    if (bytes == 0)
        bytes = 16;
    cudaError_t e = cudaMalloc(p, bytes);
    if (e == cudaSuccess)
        L->allocs.push_back(*p);
    return e;
}

void release(moe_layer *L)
{
    if (!L)
        return;
    cudaDeviceSynchronize();
    for (void *p : L->allocs)
        cudaFree(p);
    L->allocs.clear();
    for (void *p : L->tier_allocs)
        cudaFree(p);
    L->tier_allocs.clear();
    if (L->host_gu)
        cudaFreeHost(L->host_gu);
    if (L->host_dn)
        cudaFreeHost(L->host_dn);
    if (L->prof_ev) {
        for (int i = 0; i < kProfRing * (kPhases + 1); i++)
            if (L->prof_ev[i])
                cudaEventDestroy(L->prof_ev[i]);
        delete[] L->prof_ev;
        L->prof_ev = nullptr;
    }
    delete L;
}

bool is_device_ptr(const void *p)
{
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

// K-slices of the router: kslice = H / ks must be a multiple of 128 and at most
// 1024 (shared memory); enough CTAs to cover the SMs twice where possible.
int choose_ks(int H, int E, int n, int num_sms)
{
    const int units = H / kGroup;
    const long long ctas = (long long)((E + 7) / 8) * ((n + 7) / 8);
    int best = 0;
    for (int ks = 1; ks <= units; ks++) {
        if (units % ks || H / ks > 1024)
            continue;
        best = ks;
        if (ctas * ks >= 2LL * num_sms)
            break;
    }
    return best;
}

int check_cfg(const moe_cfg_t *c)
{
    if (c->group_size != kGroup)
        return fail(MOE_ERR_UNSUPPORTED, "group_size %d: only 128 is supported", c->group_size);
    if (c->wbits != 4 && c->wbits != 2)
        return fail(MOE_ERR_UNSUPPORTED, "wbits %d: only 4 and 2 are supported", c->wbits);
    if (c->io_dtype != MOE_FP16)
        return fail(MOE_ERR_UNSUPPORTED, "io_dtype %d: only MOE_FP16 is supported", c->io_dtype);
    if (c->hidden <= 0 || c->hidden % kGroup || c->hidden > 16384)
        return fail(MOE_ERR_INVALID_ARG, "hidden %d: need a multiple of 128 in [128, 16384]",
                    c->hidden);
    if (c->inter <= 0 || c->inter % kGroup || c->inter > 65536)
        return fail(MOE_ERR_INVALID_ARG, "inter %d: need a multiple of 128 in [128, 65536]",
                    c->inter);
    if (c->n_experts < 1 || c->n_experts > kMaxExperts)
        return fail(MOE_ERR_INVALID_ARG, "n_experts %d: need 1..%d", c->n_experts, kMaxExperts);
    if (c->top_k < 1 || c->top_k > c->n_experts || c->top_k > kMaxTopK)
        return fail(MOE_ERR_INVALID_ARG, "top_k %d: need 1..min(n_experts, %d)", c->top_k,
                    kMaxTopK);
    if (c->has_shared != 0 && c->has_shared != 1)
        return fail(MOE_ERR_INVALID_ARG, "has_shared must be 0 or 1");
    if (c->has_shared && (c->shared_inter <= 0 || c->shared_inter % kGroup ||
                          c->shared_inter > 65536))
        return fail(MOE_ERR_INVALID_ARG, "shared_inter %d: need a multiple of 128",
                    c->shared_inter);
    if (c->residual != 0 && c->residual != 1)
        return fail(MOE_ERR_INVALID_ARG, "residual must be 0 or 1");
    if (c->max_tokens < 1 || c->max_tokens > 65536)
        return fail(MOE_ERR_INVALID_ARG, "max_tokens %d: need 1..65536", c->max_tokens);
    if ((long long)c->max_tokens * c->top_k > (1LL << 24))
        return fail(MOE_ERR_INVALID_ARG, "max_tokens * top_k too large");
    return MOE_OK;
}

int check_weight_ptrs(const moe_cfg_t *c, const moe_packed_weights_t *w)
{
    for (int m = 0; m < 3; m++)
        if (!w->codes[m] || !w->scales[m] || !w->zeros[m])
            return fail(MOE_ERR_INVALID_ARG, "null expert weight pointer (matrix %d)", m);
    if (!w->router_w)
        return fail(MOE_ERR_INVALID_ARG, "null router_w");
    if (c->has_shared) {
        for (int m = 0; m < 3; m++)
            if (!w->sh_codes[m] || !w->sh_scales[m] || !w->sh_zeros[m])
                return fail(MOE_ERR_INVALID_ARG, "null shared weight pointer (matrix %d)", m);
        if (!w->sh_gate_w)
            return fail(MOE_ERR_INVALID_ARG, "null sh_gate_w");
    }
    return MOE_OK;
}

#define CK(call)                                                                            \
    do {                                                                                     \
        cudaError_t e_ = (call);                                                             \
        if (e_ != cudaSuccess) {                                                             \
            int code_ = e_ == cudaErrorMemoryAllocation ? MOE_ERR_OOM : MOE_ERR_CUDA;         \
            fail(code_, "%s: %s (%s:%d)", #call, cudaGetErrorString(e_), __FILE__, __LINE__); \
            cudaGetLastError();                                                              \
            return code_;                                                                    \
        }                                                                                    \
    } while (0)

// Records of one stream: `mats` matrices (rows x K each) of n_exp experts.
int build_stream(moe_layer *L, PackedRecs *pr, int n_exp, int rows, int K, int mats,
                 const uint8_t *const *codes, const uint16_t *const *scales,
                 const uint8_t *const *zeros)
{
    const int wb = L->cfg.wbits;
    const int code = (kGroup * wb / 8) * kRowTile;   // codes of 16 rows x 128 K
    const int pair = mats == 1;   // one matrix: two row tiles per record
    pr->n_rt = pair ? rows / (2 * kRowTile) : rows / kRowTile;
    pr->n_groups = K / kGroup;
    pr->pair = pair;
    pr->upt = pair ? 4 : 8;
    pr->rec = 2 * (code + kMetaBytes);
    pr->expert_bytes = (long long)pr->n_rt * pr->n_groups * pr->rec;
    void *p = nullptr;
    const size_t bytes = (size_t)n_exp * pr->expert_bytes;
    CK(dalloc(L, &p, bytes));
    L->weight_bytes += bytes;
    pr->recs = static_cast<const uint8_t *>(p);
    for (int m = 0; m < mats; m++)
        CK(launch_repack(codes[m], scales[m], zeros[m], n_exp, rows, K, wb, m, mats, pair,
                         static_cast<uint8_t *>(p), 0));
    return MOE_OK;
}

// 2-D TMA map of a row-major fp16 matrix [rows][cols]: boxes of 32 rows x
// 64 columns (128 bytes) with the 128-byte swizzle the MMA operand expects.
bool encode_rows(CUtensorMap *map, const void *base, uint64_t cols, uint64_t rows)
{
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    if (!encode) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn) {
            cudaGetLastError();
            return false;
        }
        encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {64, 32};
    const cuuint32_t estr[2] = {1, 1};
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int create_impl(const moe_cfg_t *cfg, const moe_packed_weights_t *w, moe_layer *L)
{
    L->cfg = *cfg;
    const moe_cfg_t &c = L->cfg;
    CK(cudaGetDevice(&L->device));
    CK(cudaDeviceGetAttribute(&L->num_sms, cudaDevAttrMultiProcessorCount, L->device));
    // every weight pointer must be device memory
    const void *ptrs[] = {w->codes[0], w->codes[1], w->codes[2], w->scales[0], w->scales[1],
                          w->scales[2], w->zeros[0], w->zeros[1], w->zeros[2], w->router_w};
    for (const void *p : ptrs)
        if (!is_device_ptr(p))
            return fail(MOE_ERR_INVALID_ARG, "weight pointer %p is not device memory", p);
    if (w->router_bias && !is_device_ptr(w->router_bias))
        return fail(MOE_ERR_INVALID_ARG, "router_bias is not device memory");
    if (c.has_shared) {
        const void *sp[] = {w->sh_codes[0], w->sh_codes[1], w->sh_codes[2], w->sh_scales[0],
                            w->sh_scales[1], w->sh_scales[2], w->sh_zeros[0], w->sh_zeros[1],
                            w->sh_zeros[2], w->sh_gate_w};
        for (const void *p : sp)
            if (!is_device_ptr(p))
                return fail(MOE_ERR_INVALID_ARG, "shared weight pointer %p is not device memory",
                            p);
    }
    LayerDev &D = L->dev;
    D.H = c.hidden;
    D.I = c.inter;
    D.E = c.n_experts;
    D.k = c.top_k;
    D.wbits = c.wbits;
    D.has_shared = c.has_shared;
    D.I_sh = c.has_shared ? c.shared_inter : 0;
    D.residual = c.residual;
    D.max_tokens = c.max_tokens;

    const int H = D.H, I = D.I, E = D.E;
    int rc;
    if ((rc = build_stream(L, &D.gu, E, I, H, 2, w->codes, w->scales, w->zeros)) ||
        (rc = build_stream(L, &D.dn, E, H, I, 1, w->codes + 2, w->scales + 2, w->zeros + 2)))
        return rc;
    L->expert_bytes = 3LL * I * H * c.wbits / 8 + 3LL * I * (H / kGroup) * 3;
    if (c.has_shared) {
        const int Is = D.I_sh;
        if ((rc = build_stream(L, &D.sh_gu, 1, Is, H, 2, w->sh_codes, w->sh_scales,
                               w->sh_zeros)) ||
            (rc = build_stream(L, &D.sh_dn, 1, H, Is, 1, w->sh_codes + 2, w->sh_scales + 2,
                               w->sh_zeros + 2)))
            return rc;
        L->shared_bytes = 3LL * Is * H * c.wbits / 8 + 3LL * Is * (H / kGroup) * 3;
    }
    void *p;
    CK(dalloc(L, &p, (size_t)E * H * 2));
    CK(cudaMemcpy(p, w->router_w, (size_t)E * H * 2, cudaMemcpyDeviceToDevice));
    D.router_w = static_cast<const __half *>(p);
    L->weight_bytes += (int64_t)E * H * 2;
    if (w->router_bias) {
        CK(dalloc(L, &p, (size_t)E * 4));
        CK(cudaMemcpy(p, w->router_bias, (size_t)E * 4, cudaMemcpyDeviceToDevice));
        D.router_bias = static_cast<const float *>(p);
        L->weight_bytes += (int64_t)E * 4;
    }
    if (c.has_shared) {
        CK(dalloc(L, &p, (size_t)H * 2));
        CK(cudaMemcpy(p, w->sh_gate_w, (size_t)H * 2, cudaMemcpyDeviceToDevice));
        D.sh_gate_w = static_cast<const __half *>(p);
        L->weight_bytes += (int64_t)H * 2;
    }

    // workspace for max_tokens
    Workspace &ws = L->ws;
    const long long n = c.max_tokens, P = n * c.top_k;
    const long long Imax = I > D.I_sh ? I : D.I_sh;
    ws.max_entries = (int)(E + 2 * ((P + kMaxTokTile - 1) / kMaxTokTile) +
                           (n + kMaxTokTile - 1) / kMaxTokTile + 8);
    ws.max_gentries = (int)(E + (P + kGemmTok - 1) / kGemmTok + (n + kGemmTok - 1) / kGemmTok + 8);
    size_t before = 0;
    struct Req {
        void **dst;
        size_t bytes;
    } reqs[] = {
        {(void **)&ws.hdr, 64},
        {(void **)&ws.entries, sizeof(Entry) * (size_t)ws.max_entries},
        {(void **)&ws.gentries, sizeof(int4) * (size_t)ws.max_gentries},
        {(void **)&ws.xs, c.wbits == 4 ? 2 * (size_t)((P + n) * H) : 0},
        {(void **)&ws.idx, 4 * (size_t)P},
        {(void **)&ws.w, 4 * (size_t)P},
        {(void **)&ws.counts, 4 * (size_t)E},
        {(void **)&ws.offsets, 4 * (size_t)(E + 1)},
        {(void **)&ws.perm, 4 * (size_t)P},
        {(void **)&ws.pos_of_pair, 4 * (size_t)P},
        {(void **)&ws.tok_of_pos, 4 * (size_t)(P + n)},
        {(void **)&ws.logits, 4 * (size_t)(n * E)},
        {(void **)&ws.approx, 4 * (size_t)(n * E)},
        {(void **)&ws.rnorm, 4 * (size_t)E},
        {(void **)&ws.sums, 24 * (size_t)(n * E)},
        {(void **)&ws.tickets, 4 * (size_t)((n + 7) / 8 + 1)},
        {(void **)&ws.xsum, 4 * (size_t)(n * (H / kGroup)) * (c.wbits == 2 ? 2 : 1)},
        {(void **)&ws.xn, 2 * (size_t)(n * H)},
        {(void **)&ws.h, 2 * (size_t)((P + n) * Imax)},
        {(void **)&ws.y, 4 * (size_t)((P + n) * H)},
    };
    for (auto &r : reqs) {
        CK(dalloc(L, r.dst, r.bytes));
        before += r.bytes;
    }
    L->workspace_bytes = (int64_t)before;
    CK(cudaMemset(ws.hdr, 0, 64));
    CK(cudaMemset(ws.sums, 0, 24 * (size_t)(n * E)));
    CK(cudaMemset(ws.tickets, 0, 4 * (size_t)((n + 7) / 8 + 1)));
    CK(cudaMemset(ws.approx, 0, 4 * (size_t)(n * E)));
    CK(launch_router_rnorm(D, ws.rnorm, 0));

    // the attribute belongs to the kernel, not to this layer: the size for the
    // largest expert count, so that no later layer lowers it under an earlier one
    configure_group_kernel(group_smem_bytes(kMaxExperts));
    configure_router_kernel((size_t)8 * 1024 * sizeof(int2));
    configure_ffn_kernels();
    if (c.wbits == 4) {
        configure_gemm_kernels();
        const uint64_t rows = (uint64_t)(P + n);
        if (!encode_rows(&L->map_xs, ws.xs, (uint64_t)H, rows) ||
            !encode_rows(&L->map_h, ws.h, (uint64_t)Imax, rows))
            return fail(MOE_ERR_CUDA, "TMA tensor map encoding failed");
        const int kmin = std::min(std::min(H, I), D.has_shared ? D.I_sh : I);
        const bool fills = 2 * I / 128 >= L->num_sms;   // gate/up 128-row tiles of one expert
        L->gemm_min_tokens = kmin >= kShortKGemm && fills ? kDefaultGemmMinTokens : 0;
    }
    const int bps = ffn_blocks_per_sm(c.wbits);
    L->grid_ffn = L->num_sms * (bps > 0 ? bps : 1);
    CK(cudaGetLastError());
    CK(cudaDeviceSynchronize());
    return MOE_OK;
}

int check_call(moe_layer *L, const void *x, int n)
{
    if (!L)
        return fail(MOE_ERR_INVALID_ARG, "null layer");
    if (!x)
        return fail(MOE_ERR_INVALID_ARG, "null x");
    if (n < 1 || n > L->cfg.max_tokens)
        return fail(MOE_ERR_INVALID_ARG, "n_tokens %d outside 1..%d", n, L->cfg.max_tokens);
    if (reinterpret_cast<uintptr_t>(x) % 16)
        return fail(MOE_ERR_INVALID_ARG, "x must be 16-byte aligned");
    return MOE_OK;
}

void prof_mark(moe_layer *L, int phase, cudaStream_t st)
{
    if (!L->prof_active)
        return;
    cudaEvent_t *set = L->prof_ev + (size_t)L->prof_head * (kPhases + 1);
    cudaEventRecord(set[phase], st);
}

void prof_begin(moe_layer *L)
{
    L->prof_active = L->prof_on;
    if (!L->prof_on)
        return;
    // the set about to be overwritten holds a forward kProfRing calls old
    if (L->prof_pending == kProfRing) {
        cudaEvent_t *set = L->prof_ev + (size_t)L->prof_head * (kPhases + 1);
        cudaEventSynchronize(set[kPhases]);
        for (int ph = 0; ph < kPhases; ph++) {
            float ms = 0.f;
            cudaEventElapsedTime(&ms, set[ph], set[ph + 1]);
            L->prof_ms[ph] += ms;
        }
        L->prof_calls++;
        L->prof_pending--;
    }
}

void prof_end(moe_layer *L)
{
    if (!L->prof_active)
        return;
    L->prof_active = 0;
    L->prof_head = (L->prof_head + 1) % kProfRing;
    L->prof_pending++;
}

// Per-expert token count from which an expert runs on the GEMM kernels in a
// call of n tokens (0: none can): an expert has at most n tokens, and the
// shared expert exactly n.
int gemm_big(const moe_layer *L, int n)
{
    return L->gemm_min_tokens > 0 && n >= L->gemm_min_tokens ? L->gemm_min_tokens : 0;
}

// Tokens per GEMM entry for a call of n tokens: 128 when the call averages
// at least 128 tokens per expert, else 64.  The 128-token kernels keep one
// accumulator set (the other half of tensor memory holds the A ring), so a
// tile's epilogue is not hidden behind the next tile's MMAs; they pay off
// once most entries are full (the 14336-wide 64-expert layer: 4317 against
// 5134 us at 4096 tokens, 8176 against 9519 us at 8192; 1920 against 1825 us
// at 1024).
int gemm_tok(const moe_layer *L, int n)
{
    return (long long)n * L->dev.k >= (long long)kGemmTokWide * L->dev.E ? kGemmTokWide
                                                                          : kGemmTok;
}

// `grouped`: the routing launch has already grouped the pairs.  xres: the
// residual rows (x itself unless the layer runs on RMSNorm-ed tokens).
int run_tail(moe_layer *L, const void *x, void *out, int n, int grouped, const void *xres,
             cudaStream_t st)
{
    const LayerDev &D = L->dev;
    const Workspace &ws = L->ws;
    const int big = gemm_big(L, n), gtok = gemm_tok(L, n);
    if (!grouped)
        CK(launch_group(D, ws, n, big, gtok, st));
    if (L->tiered && L->n_resident < D.E)   // give the touched cold experts device slots
        CK(launch_stage(L->tier, ws, L->num_sms, st));
    prof_mark(L, 2, st);
    CK(launch_gateup(D, ws, static_cast<const __half *>(x), L->grid_ffn, st));
    if (big) {
        CK(launch_gather(D, ws, static_cast<const __half *>(x), n, st));
        CK(launch_gemm_gateup(D, ws, L->map_xs, gtok, L->num_sms, st));
    }
    prof_mark(L, 3, st);
    CK(launch_down(D, ws, L->grid_ffn, st));
    if (big)
        CK(launch_gemm_down(D, ws, L->map_h, gtok, L->num_sms, st));
    prof_mark(L, 4, st);
    CK(launch_combine(D, ws, static_cast<const __half *>(x), static_cast<const __half *>(xres),
                      static_cast<__half *>(out), n, st));
    prof_mark(L, 5, st);
    return MOE_OK;
}

// Routing of n tokens.  With group_big >= 0 and at most kFusedPairs pairs
// the same launch also groups the pairs (GEMM threshold group_big) and
// *grouped is set; otherwise the caller launches the grouping kernel.
int run_route(moe_layer *L, const void *x, int n, int want_logits, int group_big, int *grouped,
              cudaStream_t st)
{
    prof_mark(L, 0, st);
    const Workspace &ws = L->ws;
    RouteExtras fg{};
    if (group_big >= 0 && (long long)n * L->dev.k <= kFusedPairs) {
        fg.on = 1;
        fg.big = group_big;
        fg.gtok = gemm_tok(L, n);
        fg.has_shared = L->dev.has_shared;
        fg.ticket = ws.tickets + (L->cfg.max_tokens + 7) / 8;
        fg.hdr = ws.hdr;
        fg.entries = ws.entries;
        fg.gentries = ws.gentries;
        fg.counts = ws.counts;
        fg.offsets = ws.offsets;
        fg.perm = ws.perm;
        fg.pos_of_pair = ws.pos_of_pair;
        fg.tok_of_pos = ws.tok_of_pos;
    }
    if (grouped)
        *grouped = fg.on;
    if (!want_logits)
        fg.xsum = ws.xsum;
    fg.xsplit = L->dev.wbits == 2 ? 1 : 0;
    if (!want_logits &&
        (QE_LARGE_ROUTE_ALL || n >= kLargeRouteTokens ||
         (L->dev.E >= kLargeRouteExperts && n >= kManyExpertTokens))) {
        CK(launch_route_large(L->dev, ws, static_cast<const __half *>(x), n, L->num_sms, fg, st));
    } else {
        const int ks = choose_ks(L->dev.H, L->dev.E, n, L->num_sms);
        CK(launch_route(L->dev, ws, static_cast<const __half *>(x), n, ks, want_logits, fg, st));
    }
    prof_mark(L, 1, st);
    return MOE_OK;
}

// The address through which the SMs reach p: p itself for device and
// managed memory, the mapped address of pinned host memory; null otherwise.
const void *device_reachable(const void *p)
{
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged)
        return p;
    if (a.type == cudaMemoryTypeHost)
        return a.devicePointer;
    return nullptr;
}

// Checks out and sets *dout to the address the combine kernel writes:
// device memory, or pinned host memory written in place.
int check_out(moe_layer *L, const void *x, const void *out, int n, void **dout)
{
    if (!out)
        return fail(MOE_ERR_INVALID_ARG, "null out");
    if (reinterpret_cast<uintptr_t>(out) % 16)
        return fail(MOE_ERR_INVALID_ARG, "out must be 16-byte aligned");
    const char *a = static_cast<const char *>(x), *b = static_cast<const char *>(out);
    const size_t bytes = (size_t)n * L->cfg.hidden * 2;
    if (a < b + bytes && b < a + bytes)
        return fail(MOE_ERR_INVALID_ARG, "out overlaps x");
    *dout = const_cast<void *>(device_reachable(out));
    if (!*dout)
        return fail(MOE_ERR_INVALID_ARG, "out is neither device memory nor pinned host memory");
    return MOE_OK;
}

int check_norm_args(const void *gamma, float eps)
{
    if (!gamma)
        return fail(MOE_ERR_INVALID_ARG, "null gamma");
    if (reinterpret_cast<uintptr_t>(gamma) % 16)
        return fail(MOE_ERR_INVALID_ARG, "gamma must be 16-byte aligned");
    if (!(eps >= 0.0f) || eps > 3.0e38f)
        return fail(MOE_ERR_INVALID_ARG, "eps must be finite and >= 0");
    return MOE_OK;
}

int norm_launch(const __half *r, const __half *g, float eps, int n, int H, __half *xn,
                cudaStream_t st)
{
    CK(launch_rmsnorm(r, g, eps, n, H, xn, st));
    return MOE_OK;
}

}  // namespace

namespace qe {
// Host helpers shared with the layer-free entry point.
bool device_pointer(const void *p) { return is_device_ptr(p); }
int router_k_slices(int H, int E, int n, int num_sms) { return choose_ks(H, E, n, num_sms); }
}  // namespace qe

extern "C" {

int moe_layer_create(const moe_cfg_t *cfg, const moe_packed_weights_t *w, moe_layer_t **out)
{
    if (!out)
        return fail(MOE_ERR_INVALID_ARG, "null out handle");
    *out = nullptr;
    if (!cfg)
        return fail(MOE_ERR_INVALID_ARG, "null cfg");
    if (!w)
        return fail(MOE_ERR_INVALID_ARG, "null weights");
    int rc = check_cfg(cfg);
    if (rc)
        return rc;
    if ((rc = check_weight_ptrs(cfg, w)))
        return rc;
    moe_layer *L = new (std::nothrow) moe_layer();
    if (!L)
        return fail(MOE_ERR_OOM, "host allocation failed");
    rc = create_impl(cfg, w, L);
    if (rc) {
        char saved[sizeof(g_err)];
        memcpy(saved, g_err, sizeof(saved));
        release(L);
        memcpy(g_err, saved, sizeof(saved));
        return rc;
    }
    *out = L;
    return ok();
}

void moe_layer_destroy(moe_layer_t *layer) { release(layer); }

int moe_route_topk(moe_layer_t *L, const void *x, int n, int32_t *topk_idx, float *topk_w,
                   int32_t *counts, int32_t *offsets, int32_t *perm, void *stream)
{
    int rc = check_call(L, x, n);
    if (rc)
        return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t P = (size_t)n * L->cfg.top_k, E = L->cfg.n_experts;
    int grouped = 0;
    if ((rc = run_route(L, x, n, 0, 0, &grouped, st)))
        return rc;
    if (!grouped)
        CK(launch_group(L->dev, L->ws, n, 0, kGemmTok, st));
    if (topk_idx)
        CK(cudaMemcpyAsync(topk_idx, L->ws.idx, 4 * P, cudaMemcpyDeviceToDevice, st));
    if (topk_w)
        CK(cudaMemcpyAsync(topk_w, L->ws.w, 4 * P, cudaMemcpyDeviceToDevice, st));
    if (counts)
        CK(cudaMemcpyAsync(counts, L->ws.counts, 4 * E, cudaMemcpyDeviceToDevice, st));
    if (offsets)
        CK(cudaMemcpyAsync(offsets, L->ws.offsets, 4 * (E + 1), cudaMemcpyDeviceToDevice, st));
    if (perm)
        CK(cudaMemcpyAsync(perm, L->ws.perm, 4 * P, cudaMemcpyDeviceToDevice, st));
    return ok();
}

int moe_router_logits(moe_layer_t *L, const void *x, int n, float *logits, void *stream)
{
    int rc = check_call(L, x, n);
    if (rc)
        return rc;
    if (!logits)
        return fail(MOE_ERR_INVALID_ARG, "null logits");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if ((rc = run_route(L, x, n, 1, -1, nullptr, st)))
        return rc;
    CK(cudaMemcpyAsync(logits, L->ws.logits, 4 * (size_t)n * L->cfg.n_experts,
                       cudaMemcpyDeviceToDevice, st));
    return ok();
}

int moe_forward(moe_layer_t *L, const void *x, void *out, int n, void *stream)
{
    int rc = check_call(L, x, n);
    if (rc)
        return rc;
    void *dout = nullptr;
    if ((rc = check_out(L, x, out, n, &dout)))
        return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    prof_begin(L);
    int grouped = 0;
    if ((rc = run_route(L, x, n, 0, gemm_big(L, n), &grouped, st)) ||
        (rc = run_tail(L, x, dout, n, grouped, x, st))) {
        L->prof_active = 0;
        return rc;
    }
    prof_end(L);
    return ok();
}

int moe_forward_routed(moe_layer_t *L, const void *x, const int32_t *topk_idx,
                       const float *topk_w, void *out, int n, void *stream)
{
    int rc = check_call(L, x, n);
    if (rc)
        return rc;
    if (!topk_idx || !topk_w)
        return fail(MOE_ERR_INVALID_ARG, "null routing input");
    void *dout = nullptr;
    if ((rc = check_out(L, x, out, n, &dout)))
        return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t P = (size_t)n * L->cfg.top_k;
    CK(cudaMemcpyAsync(L->ws.idx, topk_idx, 4 * P, cudaMemcpyDeviceToDevice, st));
    CK(cudaMemcpyAsync(L->ws.w, topk_w, 4 * P, cudaMemcpyDeviceToDevice, st));
    CK(launch_xsum(L->dev, L->ws, static_cast<const __half *>(x), n, st));
    if ((rc = run_tail(L, x, dout, n, 0, x, st)))
        return rc;
    return ok();
}

int moe_forward_prenorm(moe_layer_t *L, const void *resid, const void *gamma, float eps,
                        void *out, int n, void *stream)
{
    int rc = check_call(L, resid, n);
    if (rc)
        return rc;
    if ((rc = check_norm_args(gamma, eps)))
        return rc;
    void *dout = nullptr;
    if ((rc = check_out(L, resid, out, n, &dout)))
        return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const __half *xn = L->ws.xn;
    prof_begin(L);
    int grouped = 0;
    if ((rc = norm_launch(static_cast<const __half *>(resid), static_cast<const __half *>(gamma),
                          eps, n, L->cfg.hidden, L->ws.xn, st)) ||
        (rc = run_route(L, xn, n, 0, gemm_big(L, n), &grouped, st)) ||
        (rc = run_tail(L, xn, dout, n, grouped, resid, st))) {
        L->prof_active = 0;
        return rc;
    }
    prof_end(L);
    return ok();
}

int moe_rmsnorm(const void *resid, const void *gamma, float eps, int n, int hidden, void *xn,
                void *stream)
{
    if (!resid || !xn)
        return fail(MOE_ERR_INVALID_ARG, "null resid or xn");
    if (reinterpret_cast<uintptr_t>(resid) % 16 || reinterpret_cast<uintptr_t>(xn) % 16)
        return fail(MOE_ERR_INVALID_ARG, "resid and xn must be 16-byte aligned");
    if (n < 1)
        return fail(MOE_ERR_INVALID_ARG, "n_tokens %d: need >= 1", n);
    if (hidden <= 0 || hidden % kGroup || hidden > 16384)
        return fail(MOE_ERR_INVALID_ARG, "hidden %d: need a multiple of 128 in [128, 16384]",
                    hidden);
    int rc = check_norm_args(gamma, eps);
    if (rc)
        return rc;
    if ((rc = norm_launch(static_cast<const __half *>(resid), static_cast<const __half *>(gamma),
                          eps, n, hidden, static_cast<__half *>(xn),
                          static_cast<cudaStream_t>(stream))))
        return rc;
    return ok();
}

int moe_copy(void *dst, const void *src, size_t bytes, void *stream)
{
    if (bytes == 0)
        return ok();
    if (!dst || !src)
        return fail(MOE_ERR_INVALID_ARG, "null dst or src");
    if (reinterpret_cast<uintptr_t>(dst) % 16 || reinterpret_cast<uintptr_t>(src) % 16 ||
        bytes % 16)
        return fail(MOE_ERR_INVALID_ARG, "dst, src and bytes must be multiples of 16 bytes");
    const char *a = static_cast<const char *>(dst), *b = static_cast<const char *>(src);
    if (a < b + bytes && b < a + bytes)
        return fail(MOE_ERR_INVALID_ARG, "dst overlaps src");
    void *d = const_cast<void *>(device_reachable(dst));
    const void *s = device_reachable(src);
    if (!d || !s)
        return fail(MOE_ERR_INVALID_ARG,
                    "dst and src must be device, managed or pinned (mapped) host memory");
    int dev = 0, sms = 0;
    CK(cudaGetDevice(&dev));
    CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    CK(launch_copy(d, s, bytes, sms, static_cast<cudaStream_t>(stream)));
    return ok();
}

int moe_check_status(moe_layer_t *L, int *bits)
{
    if (bits)
        *bits = 0;
    if (!L)
        return fail(MOE_ERR_INVALID_ARG, "null layer");
    CK(cudaDeviceSynchronize());
    int v = 0;
    CK(cudaMemcpy(&v, L->ws.hdr + 2, sizeof(int), cudaMemcpyDeviceToHost));
    CK(cudaMemset(L->ws.hdr + 2, 0, sizeof(int)));
    CK(cudaDeviceSynchronize());
    if (bits)
        *bits = v;
    if (v)
        return fail(MOE_ERR_DEVICE_STATUS, "device status bits 0x%x", v);
    return ok();
}

int moe_layer_set_gemm_min_tokens(moe_layer_t *L, int min_tokens)
{
    if (!L)
        return fail(MOE_ERR_INVALID_ARG, "null layer");
    if (min_tokens < 0)
        return fail(MOE_ERR_INVALID_ARG, "min_tokens must be >= 0");
    if (min_tokens > 0 && L->cfg.wbits != 4)
        return fail(MOE_ERR_UNSUPPORTED, "the GEMM kernels take 4-bit layers only");
    L->gemm_min_tokens = min_tokens;
    return ok();
}

int moe_layer_info(const moe_layer_t *L, moe_layer_info_t *info)
{
    if (!L || !info)
        return fail(MOE_ERR_INVALID_ARG, "null argument");
    info->weight_bytes = L->weight_bytes;
    info->workspace_bytes = L->workspace_bytes;
    info->expert_bytes = L->expert_bytes;
    info->shared_bytes = L->shared_bytes;
    info->num_sms = L->num_sms;
    info->grid_ffn = L->grid_ffn;
    info->n_phases = kPhases;
    info->gemm_min_tokens = L->gemm_min_tokens;
    return ok();
}

int moe_profile_enable(moe_layer_t *L, int on)
{
    if (!L)
        return fail(MOE_ERR_INVALID_ARG, "null layer");
    if (on && !L->prof_ev) {
        L->prof_ev = new (std::nothrow) cudaEvent_t[kProfRing * (kPhases + 1)]();
        if (!L->prof_ev)
            return fail(MOE_ERR_OOM, "host allocation failed");
        for (int i = 0; i < kProfRing * (kPhases + 1); i++)
            CK(cudaEventCreate(&L->prof_ev[i]));
    }
    L->prof_on = on ? 1 : 0;
    return ok();
}

int moe_profile_read(moe_layer_t *L, float *ms, int n, int *calls)
{
    if (!L)
        return fail(MOE_ERR_INVALID_ARG, "null layer");
    if (L->prof_ev) {
        // drain every pending set, oldest first
        int idx = (L->prof_head - L->prof_pending + kProfRing) % kProfRing;
        for (; L->prof_pending > 0; L->prof_pending--, idx = (idx + 1) % kProfRing) {
            cudaEvent_t *set = L->prof_ev + (size_t)idx * (kPhases + 1);
            CK(cudaEventSynchronize(set[kPhases]));
            for (int ph = 0; ph < kPhases; ph++) {
                float v = 0.f;
                if (cudaEventElapsedTime(&v, set[ph], set[ph + 1]) == cudaSuccess)
                    L->prof_ms[ph] += v;
                else
                    cudaGetLastError();
            }
            L->prof_calls++;
        }
    }
    for (int i = 0; i < n && i < kPhases; i++)
        if (ms)
            ms[i] = (float)L->prof_ms[i];
    if (calls)
        *calls = L->prof_calls;
    for (int i = 0; i < kPhases; i++)
        L->prof_ms[i] = 0;
    L->prof_calls = 0;
    return ok();
}

const char *moe_last_error(void) { return g_err; }

int moe_residency_plan(const int64_t *counts, int n_experts, int n_resident, int32_t *resident)
{
    if (!counts || !resident)
        return fail(MOE_ERR_INVALID_ARG, "null counts or resident");
    if (n_experts < 1 || n_experts > kMaxExperts)
        return fail(MOE_ERR_INVALID_ARG, "n_experts %d: need 1..%d", n_experts, kMaxExperts);
    if (n_resident < 0 || n_resident > n_experts)
        return fail(MOE_ERR_INVALID_ARG, "n_resident %d: need 0..n_experts", n_resident);
    for (int e = 0; e < n_experts; e++)
        if (counts[e] < 0)
            return fail(MOE_ERR_INVALID_ARG, "negative count for expert %d", e);
    // the n_resident most frequently routed experts, ties to the lower id:
    // repeated selection of the largest remaining count
    std::vector<char> taken((size_t)n_experts, 0);
    for (int i = 0; i < n_resident; i++) {
        int best = -1;
        for (int e = 0; e < n_experts; e++)
            if (!taken[e] && (best < 0 || counts[e] > counts[best]))
                best = e;
        taken[best] = 1;
        resident[i] = best;
    }
    return ok();
}

int moe_layer_set_residency(moe_layer_t *L, const int32_t *resident, int n_resident,
                            int n_slots)
{
    if (!L)
        return fail(MOE_ERR_INVALID_ARG, "null layer");
    const int E = L->cfg.n_experts;
    if (n_resident < 0 || n_resident > E)
        return fail(MOE_ERR_INVALID_ARG, "n_resident %d: need 0..%d", n_resident, E);
    if (n_resident > 0 && !resident)
        return fail(MOE_ERR_INVALID_ARG, "null resident list");
    std::vector<int> pos((size_t)E, -1);   // position in the resident list
    for (int i = 0; i < n_resident; i++) {
        const int e = resident[i];
        if (e < 0 || e >= E)
            return fail(MOE_ERR_INVALID_ARG, "resident expert %d outside 0..%d", e, E - 1);
        if (pos[e] >= 0)
            return fail(MOE_ERR_INVALID_ARG, "resident expert %d listed twice", e);
        pos[e] = i;
    }
    const int cold = E - n_resident;
    const long long need = std::min<long long>(cold, (long long)L->cfg.max_tokens * L->cfg.top_k);
    if (cold == 0)
        n_slots = 0;
    else if (n_slots < need || n_slots > cold)
        return fail(MOE_ERR_INVALID_ARG,
                    "n_slots %d: need min(cold experts, max_tokens * top_k) = %lld .. %d",
                    n_slots, need, cold);
    LayerDev &D = L->dev;
    const long long gb = D.gu.expert_bytes, db = D.dn.expert_bytes;
    CK(cudaDeviceSynchronize());
    if (!L->tiered) {
        // every expert's records into pinned host memory; the device copy goes
        CK(cudaHostAlloc(&L->host_gu, (size_t)E * gb, cudaHostAllocMapped));
        CK(cudaHostAlloc(&L->host_dn, (size_t)E * db, cudaHostAllocMapped));
        CK(cudaMemcpy(L->host_gu, D.gu.recs, (size_t)E * gb, cudaMemcpyDeviceToHost));
        CK(cudaMemcpy(L->host_dn, D.dn.recs, (size_t)E * db, cudaMemcpyDeviceToHost));
        for (const void *full : {static_cast<const void *>(D.gu.recs),
                                 static_cast<const void *>(D.dn.recs)}) {
            for (size_t i = 0; i < L->allocs.size(); i++)
                if (L->allocs[i] == full) {
                    CK(cudaFree(L->allocs[i]));
                    L->allocs.erase(L->allocs.begin() + (long)i);
                    break;
                }
        }
        L->weight_bytes -= (int64_t)E * (gb + db);
    } else {
        for (void *p : L->tier_allocs)
            CK(cudaFree(p));
        L->tier_allocs.clear();
        L->weight_bytes -= L->tier.E ? (int64_t)(L->n_resident + L->tier.S) * (gb + db) +
                                           std::max(gb, db)
                                     : 0;
    }
    L->tiered = 1;
    L->n_resident = n_resident;
    TierDev &t = L->tier;
    t = TierDev{};
    t.E = E;
    t.S = n_slots;
    t.gu_bytes = gb;
    t.dn_bytes = db;
    t.status = L->ws.hdr + 2;
    auto tal = [&](void **p, size_t bytes) -> cudaError_t {
        *p = nullptr;
        cudaError_t e = cudaMalloc(p, bytes ? bytes : 16);
        if (e == cudaSuccess)
            L->tier_allocs.push_back(*p);
        return e;
    };
    void *res_gu, *res_dn, *zero;
    CK(tal(&res_gu, (size_t)n_resident * gb));
    CK(tal(&res_dn, (size_t)n_resident * db));
    CK(tal(reinterpret_cast<void **>(&t.slot_gu), (size_t)n_slots * gb));
    CK(tal(reinterpret_cast<void **>(&t.slot_dn), (size_t)n_slots * db));
    CK(tal(&zero, (size_t)std::max(gb, db)));
    CK(cudaMemset(zero, 0, (size_t)std::max(gb, db)));
    t.zero = static_cast<const uint8_t *>(zero);
    CK(tal(reinterpret_cast<void **>(&t.slot_of), 4 * (size_t)E));
    CK(tal(reinterpret_cast<void **>(&t.slot_expert), 4 * (size_t)(n_slots + 1)));
    CK(tal(reinterpret_cast<void **>(&t.slot_used), 4 * (size_t)(n_slots + 1)));
    CK(tal(reinterpret_cast<void **>(&t.call), 4));
    CK(tal(reinterpret_cast<void **>(&t.copies), 8 * (size_t)(n_slots + 1)));
    CK(tal(reinterpret_cast<void **>(&t.n_copy), 4));
    CK(tal(reinterpret_cast<void **>(&t.stats), 16));
    CK(tal(reinterpret_cast<void **>(&t.ebase_gu), 8 * (size_t)E));
    CK(tal(reinterpret_cast<void **>(&t.ebase_dn), 8 * (size_t)E));
    void *hg = nullptr, *hd = nullptr;
    CK(cudaHostGetDevicePointer(&hg, L->host_gu, 0));
    CK(cudaHostGetDevicePointer(&hd, L->host_dn, 0));
    t.host_gu = static_cast<const uint8_t *>(hg);
    t.host_dn = static_cast<const uint8_t *>(hd);
    // resident experts into their device block, in list order
    std::vector<int> slot_of((size_t)E);
    std::vector<const uint8_t *> eb_gu((size_t)E), eb_dn((size_t)E);
    for (int e = 0; e < E; e++) {
        if (pos[e] >= 0) {
            uint8_t *g = static_cast<uint8_t *>(res_gu) + (size_t)pos[e] * gb;
            uint8_t *d = static_cast<uint8_t *>(res_dn) + (size_t)pos[e] * db;
            CK(cudaMemcpy(g, static_cast<uint8_t *>(L->host_gu) + (size_t)e * gb, (size_t)gb,
                          cudaMemcpyHostToDevice));
            CK(cudaMemcpy(d, static_cast<uint8_t *>(L->host_dn) + (size_t)e * db, (size_t)db,
                          cudaMemcpyHostToDevice));
            slot_of[e] = kPinned;
            eb_gu[e] = g;
            eb_dn[e] = d;
        } else {
            slot_of[e] = kNoSlot;
            eb_gu[e] = t.zero;
            eb_dn[e] = t.zero;
        }
    }
    CK(cudaMemcpy(t.slot_of, slot_of.data(), 4 * (size_t)E, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(t.ebase_gu, eb_gu.data(), 8 * (size_t)E, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(t.ebase_dn, eb_dn.data(), 8 * (size_t)E, cudaMemcpyHostToDevice));
    CK(cudaMemset(t.slot_expert, 0xFF, 4 * (size_t)(n_slots + 1)));
    CK(cudaMemset(t.slot_used, 0, 4 * (size_t)(n_slots + 1)));
    CK(cudaMemset(t.call, 0, 4));
    CK(cudaMemset(t.n_copy, 0, 4));
    CK(cudaMemset(t.stats, 0, 16));
    D.gu.ebase = t.ebase_gu;
    D.dn.ebase = t.ebase_dn;
    D.gu.recs = t.zero;
    D.dn.recs = t.zero;
    L->weight_bytes += (int64_t)(n_resident + n_slots) * (gb + db) + std::max(gb, db);
    CK(cudaDeviceSynchronize());
    return ok();
}

int moe_layer_tier_stats(moe_layer_t *L, uint64_t *hits, uint64_t *misses, int *slots_filled)
{
    if (!L)
        return fail(MOE_ERR_INVALID_ARG, "null layer");
    if (!L->tiered)
        return fail(MOE_ERR_INVALID_ARG, "layer has no residency tiers");
    unsigned long long st[2] = {0, 0};
    CK(cudaDeviceSynchronize());
    CK(cudaMemcpy(st, L->tier.stats, 16, cudaMemcpyDeviceToHost));
    if (hits)
        *hits = st[0];
    if (misses)
        *misses = st[1];
    if (slots_filled) {
        std::vector<int> se((size_t)L->tier.S + 1);
        CK(cudaMemcpy(se.data(), L->tier.slot_expert, 4 * (size_t)(L->tier.S + 1),
                      cudaMemcpyDeviceToHost));
        int f = 0;
        for (int i = 0; i < L->tier.S; i++)
            f += se[i] >= 0;
        *slots_filled = f;
    }
    return ok();
}

int moe_layer_tier_slots(moe_layer_t *L, int32_t *slot_expert, int n)
{
    if (!L || !slot_expert)
        return fail(MOE_ERR_INVALID_ARG, "null argument");
    if (!L->tiered || n < L->tier.S)
        return fail(MOE_ERR_INVALID_ARG, "layer has no tiers or n < slots");
    CK(cudaDeviceSynchronize());
    if (L->tier.S)
        CK(cudaMemcpy(slot_expert, L->tier.slot_expert, 4 * (size_t)L->tier.S,
                      cudaMemcpyDeviceToHost));
    return ok();
}

}  // extern "C"
