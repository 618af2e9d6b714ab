// Expert FFN for large per-expert batches: a grouped GEMM on the tcgen05
// tensor cores with the accumulators in tensor memory.
//
// Once an expert serves many tokens the FFN is a dense contraction (the
// "Strata" article, section 3.4, verifies several tokens per weight read; the
// MoE-16B article, section 4.2, hands dequantised weights to a GEMM).  Here
// the weights stay packed in HBM (the same records as the decode kernels:
// 16-row tile x 128-group, codes then the 48-byte scale/zero block) and are
// dequantised inside the kernel, W = (q - zero) * scale ("Strata" section
// 2.2), rounded once to fp16 as the MMA's A operand, never written back.
//
// Work item: (GEMM entry = up to TOK (64 or 128) consecutive sorted positions
// of one expert, 128-row tile of the output features), ordered row tile first so
// that the entries of one expert run side by side and share each weight
// read in L2.  Swap-AB: the 128 weight rows are the MMA's M (A operand, in
// tensor memory), the entry's tokens its N (a multiple of 16, B
// operand in shared memory; N = 16..64).  One persistent CTA per SM,
// warp-specialised:
//   - code producer warp (one lane): per step (below), one bulk copy of the
//     tile's records (8 row tiles, one or two 128-groups) into a code ring;
//   - B producer warp (one lane): per 64 K, TMA tensor loads of the
//     activation rows (32-row boxes, 128-byte swizzle) into a B ring;
//   - dequant warps: one thread per weight row (its tensor-memory lane) and
//     half of each 64-K chunk; LOP3 magic-number unpack, exact q - z in fp16,
//     one rounding multiply by the scale, stored into an A ring in tensor
//     memory with tcgen05.st;
//   - two MMA warps (one lane each) with independent accumulator chains
//     (gate and up; or, for down, the even and odd 128-groups), because one
//     thread can issue a tcgen05 operation only every ~110 cycles: kind::f16
//     (fp16 x fp16 -> fp32), A from tensor memory; a step's A and B stages
//     are released by one barrier that both chains commit to;
//   - four epilogue warps (one per 32-lane quarter of tensor memory): sum the
//     chains and write h = silu(g) * u (fp16) or y (fp32), then release the
//     accumulator set.  There are two sets, used by alternate tiles, so that
//     a tile's epilogue overlaps the next tile's MMAs instead of stalling the
//     whole pipeline at every tile boundary.
// Every wait is bounded in time; on expiry the waiting thread raises
// MOE_STATUS_TIMEOUT and an abort flag, every role leaves its loop, the MMA
// lanes wait (bounded) for their MMAs and the producers for their copies, and
// the tensor memory is freed on every path.
//
// A pipeline step holds two 128-row x 128-K matrices in both kernels: the
// gate and the up rows of one 128-group, or the rows of two consecutive
// 128-groups of down.  The step's fixed cost (barrier round trips, the
// commit) is then paid once per 16 KB of codes in both; a down step of one
// group took as long as a gate/up step of two matrices.
#include <cuda.h>
#include <cuda_fp16.h>

#include "internal.cuh"

namespace qe {

namespace {

constexpr int kGM = 128;                  // weight rows per tile (MMA M)
constexpr int kGEpi = 4;                  // epilogue warps (one per tensor-memory lane quarter)
constexpr int kBox = 32;                  // rows per TMA box
constexpr int kRec4 = 1024 + kMetaBytes;  // one matrix of a 4-bit record
constexpr int kChains = 2;                // MMA warps, one accumulator chain each

// Geometry of the kernel for entries of up to TOK tokens.  TOK = 64: two
// accumulator sets, used by alternate tiles, so that a tile's epilogue
// overlaps the next tile's MMAs; TOK = 128: one set (2 x 128 columns), the
// other half of tensor memory holding the A ring, and 4 code stages so that
// the larger B stages fit in shared memory.
template <bool GU, int TOK>
struct GGeo {
    static constexpr int batom = TOK * 128;             // TOK rows x 64 K, fp16 (one swizzle atom column)
    static constexpr int bbytes = 2 * batom;            // B rows of one 128-group (two 64-K atoms)
    static constexpr int acc_bufs = TOK == kGemmTok ? 2 : 1;   // accumulator sets
    static constexpr int acc_cols = kChains * TOK;      // tensor-memory columns of one set
    static constexpr int acol0 = acc_bufs * acc_cols;   // first tensor-memory column of the A ring
    // matrices of a step: gate and up of one 128-group, or two 128-groups of down
    static constexpr int mats = 2;
    static constexpr int gps = GU ? 1 : 2;                // 128-groups per step
    static constexpr int deq = 8 * mats;                  // dequant warps: (matrix, quarter, K half)
    static constexpr int epi0 = deq;                      // first epilogue warp (epi0 % 4 == 0)
    static constexpr int prod = deq + kGEpi;              // code producer warp
    static constexpr int bprod = prod + 1;                // B producer warp
    static constexpr int mma0 = bprod + 1;                // MMA warps mma0, mma0 + 1
    static constexpr int threads = (mma0 + kChains) * 32;
    static constexpr int cs = TOK == kGemmTok ? 6 : 4;    // code stages (one step each)
    static constexpr int a_cols = mats * 64;              // tensor-memory columns per A stage
    // A and B stages (one step each), in lockstep: what tensor memory holds
    // beside the two accumulators
    static constexpr int as = (512 - acol0) / a_cols < 8 ? (512 - acol0) / a_cols : 8;
    static constexpr int bs = as;
    static constexpr int b_stage = gps * bbytes;
    static constexpr int rec = (GU ? 2 : 1) * kRec4;      // bytes per 16-row tile and group
    static constexpr int code_group = 8 * rec;            // a 128-row tile's records of one group
    static constexpr int code_stage = 16 * kRec4;
    static constexpr int b_off = 0;
    static constexpr int c_off = b_off + bs * b_stage;
    static constexpr int bar_off = c_off + cs * code_stage;
    static constexpr int nbars = 2 * cs + 2 * as + bs + 2 * acc_bufs + kChains;
    static constexpr int smem = bar_off + nbars * 8 + 16 + 1024;   // + alignment slack
    static constexpr int tmem_cols = 512;
};
template <bool GU, int TOK>
constexpr bool ggeo_ok()
{
    using G = GGeo<GU, TOK>;
    return G::smem <= 227 * 1024 && G::c_off % 1024 == 0 && G::rec % 16 == 0 &&
           G::bar_off % 8 == 0 && G::epi0 % 4 == 0 && G::acol0 <= 256 &&
           G::acol0 + G::as * G::a_cols <= 512 && TOK % kBox == 0 && G::as >= 2 &&
           G::code_stage == G::gps * G::code_group;
}
static_assert(ggeo_ok<true, kGemmTok>() && ggeo_ok<false, kGemmTok>() &&
                  ggeo_ok<true, kGemmTokWide>() && ggeo_ok<false, kGemmTokWide>(),
              "GEMM stages fit shared and tensor memory");

// Steps of a 128-row tile, and the 128-groups of step j.
template <bool GU>
__device__ __forceinline__ int tile_steps(const PackedRecs &pr)
{
    constexpr int gps = GU ? 1 : 2;
    return (pr.n_groups + gps - 1) / gps;
}

template <bool GU>
__device__ __forceinline__ int step_groups(const PackedRecs &pr, int j)
{
    constexpr int gps = GU ? 1 : 2;
    return min(gps, pr.n_groups - j * gps);
}

constexpr unsigned long long kGWaitNs = 2000000000ull;   // 2 s

__device__ __forceinline__ uint32_t saddr(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ unsigned long long now_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void bar_init(uint32_t b, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(b), "r"(count) : "memory");
}

__device__ __forceinline__ void bar_arrive(uint32_t b)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(b) : "memory");
}

__device__ __forceinline__ void bar_expect_tx(uint32_t b, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(b), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool bar_try(uint32_t b, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(b), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase of `parity`; false on expiry or abort.
__device__ __forceinline__ bool bar_wait(uint32_t b, uint32_t parity, volatile int *abort_flag)
{
    if (bar_try(b, parity))
        return true;
    const unsigned long long t0 = now_ns();
    for (unsigned it = 0;; it++) {
        if (bar_try(b, parity))
            return true;
        if ((it & 15) == 15 && (*abort_flag || now_ns() - t0 > kGWaitNs))
            return false;
    }
}

// Copy with an L2 evict-first policy: streamed data that no one reads again.
__device__ __forceinline__ void bulk_copy_ef(uint32_t dst, const void *src, uint32_t bytes,
                                             uint32_t b, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(b), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t evict_first_policy()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            uint32_t b)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(b)
        : "memory");
}

__device__ __forceinline__ void tc_fence_before()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major operand in the 128-byte
// swizzled layout: rows of 128 bytes (64 fp16 of K), 8-row groups 1024 bytes
// apart; the start address advances by 32 bytes per 16-K step.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr)
{
    return (uint64_t)((addr >> 4) & 0x3FFFu)       // start address
           | ((uint64_t)1 << 16)                   // leading offset (unused when swizzled)
           | ((uint64_t)(1024 >> 4) << 32)         // stride between 8-row groups
           | ((uint64_t)1 << 46)                   // descriptor version
           | ((uint64_t)2 << 61);                  // 128-byte swizzle
}

// Instruction descriptor, kind::f16: fp32 accumulate, fp16 A and B, both
// K-major, M = 128, N = n (multiple of 16, 16..256).
__device__ __forceinline__ uint32_t idesc_f16(int n)
{
    return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(kGM >> 4) << 24);
}

// tcgen05.mma kind::f16 with A read from tensor memory (M rows in lanes, K
// packed two fp16 per 32-bit column) and B from a shared-memory descriptor.
__device__ __forceinline__ void umma_ta(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                        uint32_t accumulate)
{
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}"
        ::"r"(d), "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

// 32 consecutive 32-bit columns of this warp's 32 tensor-memory lanes.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
        "%28, %29, %30, %31, %32};"
        ::"r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]),
          "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]),
          "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]),
          "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]),
          "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void umma_commit(uint32_t b)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 ::"r"(b)
                 : "memory");
}

// 16 consecutive fp32 columns of this warp's 32 tensor-memory lanes.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16])
{
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; i++)
        v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ uint32_t lop_magic(uint32_t a, uint32_t mask)
{
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(mask), "r"(0x64006400u));
    return d;
}

__device__ __forceinline__ uint32_t h2u(__half2 h)
{
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ __half2 u2h(uint32_t u)
{
    return *reinterpret_cast<__half2 *>(&u);
}

struct GemmArgs {
    PackedRecs r, s;        // routed and shared-expert records of this stream
    const int4 *gentries;
    const int *hdr;
    int *status;
    void *out;              // gate/up: h (fp16); down: y (fp32), rows by sorted position
    long long out_ld;
};

struct GTile {
    int expert, start, ntok, mt;
    bool shared;
};

// Tile t: routed tiles first, row tile major (the entries of one 128-row
// tile are consecutive, so the entries of one expert share the weight read),
// then the shared expert's.
__device__ __forceinline__ GTile gemm_tile(const GemmArgs &a, unsigned t, unsigned n_r,
                                           unsigned n_s, unsigned mt_r)
{
    GTile g;
    unsigned ei;
    if (t < n_r * mt_r) {
        const unsigned mt = t / n_r;
        ei = t - mt * n_r;
        g.mt = (int)mt;
        g.shared = false;
    } else {
        const unsigned j = t - n_r * mt_r, mt = j / n_s;
        ei = n_r + (j - mt * n_s);
        g.mt = (int)mt;
        g.shared = true;
    }
    const int4 e = a.gentries[ei];
    g.expert = e.x;
    g.start = e.y;
    g.ntok = e.z;
    return g;
}

// Dequantisation constants of one weight row: its scale, and the fp16
// multiplier and offset that turn the LOP3 magic-number field (1024 + q for
// rows g of a 16-row tile, 1024 + 16 q for rows g + 8) into the exact q - z.
struct RowDeq {
    uint32_t mask;          // nibble mask of this row's fields
    __half2 mul, add, scale;
};

__device__ __forceinline__ RowDeq row_deq(const uint8_t *meta, int g, int hi)
{
    const __half s = reinterpret_cast<const __half *>(meta)[2 * g + hi];
    const unsigned z = meta[32 + 2 * g + hi];
    RowDeq d;
    d.mask = hi ? 0x00F000F0u : 0x000F000Fu;
    d.mul = __float2half2_rn(hi ? 0.0625f : 1.0f);
    d.add = __float2half2_rn(hi ? -(64.0f + (float)z) : -(1024.0f + (float)z));
    d.scale = __half2half2(s);
    return d;
}

// One code word (four consecutive K of this row) into two fp16 pairs.
__device__ __forceinline__ void deq_row_word(uint32_t w, const RowDeq &d, uint32_t &p0,
                                             uint32_t &p1)
{
    p0 = h2u(__hmul2(__hfma2(u2h(lop_magic(w, d.mask)), d.mul, d.add), d.scale));
    p1 = h2u(__hmul2(__hfma2(u2h(lop_magic(w >> 8, d.mask)), d.mul, d.add), d.scale));
}

template <bool GU, int TOK>
__global__ void __launch_bounds__(GGeo<GU, TOK>::threads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap bmap, GemmArgs a)
{
    using G = GGeo<GU, TOK>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (saddr(smem_raw) & 1023u)) & 1023u);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + G::bar_off);
    const uint32_t code_full = saddr(bars), code_empty = code_full + 8 * G::cs;
    // stage_empty[s]: the MMAs reading A stage s and B stage s have completed
    const uint32_t a_full = code_empty + 8 * G::cs, stage_empty = a_full + 8 * G::as;
    const uint32_t b_full = stage_empty + 8 * G::as;
    const uint32_t acc_full = b_full + 8 * G::bs;   // [acc_bufs]
    const uint32_t acc_empty = acc_full + 8 * G::acc_bufs;   // [acc_bufs]
    const uint32_t drain = acc_empty + 8 * G::acc_bufs;      // [kChains], one per MMA warp
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + G::nbars);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    if (threadIdx.x == 0) {
        for (int s = 0; s < G::cs; s++) {
            bar_init(code_full + 8 * s, 1);
            bar_init(code_empty + 8 * s, G::deq);
        }
        for (int s = 0; s < G::as; s++) {
            bar_init(a_full + 8 * s, G::deq);
            bar_init(stage_empty + 8 * s, kChains);
            bar_init(b_full + 8 * s, 1);
        }
        for (int i = 0; i < G::acc_bufs; i++) {
            bar_init(acc_full + 8 * i, kChains);
            bar_init(acc_empty + 8 * i, kGEpi);
        }
        for (int c = 0; c < kChains; c++)
            bar_init(drain + 8 * c, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == G::mma0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(saddr(tmem_slot)), "r"((uint32_t)G::tmem_cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_enter();

    const unsigned n_r = (unsigned)a.hdr[4], n_s = (unsigned)a.hdr[5];
    // 128-row tiles: 8 row tiles, or 4 row-tile pairs of a paired stream
    const unsigned mt_r = (unsigned)a.r.n_rt / (a.r.pair ? 4 : 8);
    const unsigned mt_s = (unsigned)a.s.n_rt / (a.s.pair ? 4 : 8);
    const unsigned total = n_r * mt_r + n_s * mt_s;
    bool ok = true;

    if (warp == G::prod) {
        // ------------------------------------------------------ code producer
        if (lane == 0) {
            unsigned cc = 0;
            const uint64_t policy = evict_first_policy();
            for (unsigned t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const GTile tl = gemm_tile(a, t, n_r, n_s, mt_r);
                const PackedRecs &pr = tl.shared ? a.s : a.r;
                const uint8_t *base = expert_records(pr, tl.shared ? 0 : tl.expert);
                // the tile's records of one group are one contiguous block
                // (consecutive groups follow each other: a step's records are one block)
                const long long tile_base = (long long)tl.mt * pr.n_groups * pr.upt;
                const int nst = tile_steps<GU>(pr);
                for (int j = 0; j < nst; j++) {
                    const uint32_t s = cc % G::cs;
                    if (!bar_wait(code_empty + 8 * s, ((cc / G::cs) & 1) ^ 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t bytes = step_groups<GU>(pr, j) * G::code_group;
                    bar_expect_tx(code_full + 8 * s, bytes);
                    const uint8_t *src =
                        base + (tile_base + (long long)j * G::gps * pr.upt) * pr.rec;
                    // the codes are read once: evict them first, so that the B rows,
                    // which every row tile of the expert reads, stay in L2
                    bulk_copy_ef(saddr(smem + G::c_off + s * G::code_stage), src, bytes,
                                 code_full + 8 * s, policy);
                    ++cc;
                }
            }
            if (!ok) {
                *abort_flag = 1;
                atomicOr(a.status, MOE_STATUS_TIMEOUT);
                for (unsigned i = cc > (unsigned)G::cs ? cc - G::cs : 0; i < cc; i++) {
                    const unsigned long long t0 = now_ns();
                    while (!bar_try(code_full + 8 * (i % G::cs), (i / G::cs) & 1) &&
                           now_ns() - t0 < kGWaitNs) {
                    }
                }
            }
        }
        __syncwarp();
    } else if (warp == G::bprod) {
        // ------------------------------------------------------ B producer
        if (lane == 0) {
            unsigned bc = 0;
            for (unsigned t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const GTile tl = gemm_tile(a, t, n_r, n_s, mt_r);
                const PackedRecs &pr = tl.shared ? a.s : a.r;
                const int nb = (tl.ntok + kBox - 1) / kBox;
                const int nst = tile_steps<GU>(pr);
                for (int j = 0; j < nst; j++) {
                    const uint32_t b = bc % G::bs;
                    if (!bar_wait(stage_empty + 8 * b, ((bc / G::bs) & 1) ^ 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const int ng = step_groups<GU>(pr, j);
                    bar_expect_tx(b_full + 8 * b, ng * 2 * nb * kBox * 128);
                    const uint32_t bdst = saddr(smem + G::b_off + b * G::b_stage);
                    for (int gs = 0; gs < ng; gs++)
                        for (int at = 0; at < 2; at++)
                            for (int i = 0; i < nb; i++)
                                tma_load_2d(bdst + gs * G::bbytes + at * G::batom + i * kBox * 128,
                                            &bmap, (j * G::gps + gs) * kGroup + at * 64,
                                            tl.start + i * kBox, b_full + 8 * b);
                    ++bc;
                }
            }
            if (!ok) {
                *abort_flag = 1;
                atomicOr(a.status, MOE_STATUS_TIMEOUT);
                for (unsigned i = bc > (unsigned)G::bs ? bc - G::bs : 0; i < bc; i++) {
                    const unsigned long long t0 = now_ns();
                    while (!bar_try(b_full + 8 * (i % G::bs), (i / G::bs) & 1) &&
                           now_ns() - t0 < kGWaitNs) {
                    }
                }
            }
        }
        __syncwarp();
    } else if (warp >= G::mma0) {
        // ------------------------------------------------------ MMA issuers
        // chain c = warp - mma0, into its own accumulator: matrix c of every
        // step (gate/up: gate or up; down: the 128-groups of parity c)
        const int ch = warp - G::mma0;
        if (lane == 0) {
            unsigned ac = 0, ti = 0;
            bool issued = false;

            for (unsigned t = blockIdx.x; t < total && ok; t += gridDim.x, ti++) {
                const GTile tl = gemm_tile(a, t, n_r, n_s, mt_r);
                const PackedRecs &pr = tl.shared ? a.s : a.r;
                const int nmma = ((max(tl.ntok, 16) + 15) / 16) * 16;
                const uint32_t idesc = idesc_f16(nmma);
                // accumulator set ti % 2, used for the (ti / 2)-th time
                const uint32_t ab = ti % G::acc_bufs, use = ti / G::acc_bufs;
                const uint32_t dacc = tmem + ab * G::acc_cols + ch * TOK;
                if (!bar_wait(acc_empty + 8 * ab, (use & 1) ^ 1, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                bool first = true;
                const int nst = tile_steps<GU>(pr);
                for (int j = 0; j < nst && ok; j++) {
                    const uint32_t as = ac % G::as;
                    if (!bar_wait(a_full + 8 * as, (ac / G::as) & 1, abort_flag) ||
                        !bar_wait(b_full + 8 * as, (ac / G::as) & 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t abase = tmem + G::acol0 + as * G::a_cols + ch * 64;
                    // gate/up: both chains read the step's one B group; down: chain c
                    // reads group c of the step, absent in an odd tail
                    const uint32_t bbase =
                        saddr(smem + G::b_off + as * G::b_stage + (GU ? 0 : ch * G::bbytes));
                    if (GU || ch < step_groups<GU>(pr, j)) {
#pragma unroll
                        for (int kk = 0; kk < 8; kk++) {   // 16 K each: A 8 columns, B 32 bytes of an atom
                            const uint64_t bd =
                                sw128_desc(bbase + (kk >> 2) * G::batom + (kk & 3) * 32);
                            umma_ta(dacc, abase + kk * 8, bd, idesc, first ? 0u : 1u);
                            first = false;
                        }
                    }
                    issued = true;
                    umma_commit(stage_empty + 8 * as);
                    ++ac;
                }
                if (ok)
                    umma_commit(acc_full + 8 * ab);
            }
            if (!ok) {
                *abort_flag = 1;
                atomicOr(a.status, MOE_STATUS_TIMEOUT);
            }
            if (issued) {   // every MMA issued has completed before the memory is freed
                umma_commit(drain + 8 * ch);
                const unsigned long long t0 = now_ns();
                while (!bar_try(drain + 8 * ch, 0) && now_ns() - t0 < kGWaitNs) {
                }
            }
        }
        __syncwarp();
    } else if (warp >= G::epi0) {
        // ------------------------------------------------------ epilogue
        // rows 32 q + lane of the tile (q = this warp's tensor-memory lane
        // quarter); the chains are summed in a fixed order
        const int q = warp & 3;
        unsigned ti = 0;
        for (unsigned t = blockIdx.x; t < total && ok; t += gridDim.x, ti++) {
            const GTile tl = gemm_tile(a, t, n_r, n_s, mt_r);
            const uint32_t ab = ti % G::acc_bufs, use = ti / G::acc_bufs;
            if (!bar_wait(acc_full + 8 * ab, use & 1, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int row = tl.mt * kGM + 32 * q + lane;
            const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16) + ab * G::acc_cols;
            // down with a single 128-group: chain 1 issued nothing
            const bool two = GU || (tl.shared ? a.s : a.r).n_groups > 1;
            const int nchunks = (tl.ntok + 15) / 16;
            for (int ci = 0; ci < nchunks; ci++) {
                float d0[16], d1[16];
                tmem_ld16(taddr + ci * 16, d0);               // chain 0: gate, or even groups
                if (two)
                    tmem_ld16(taddr + TOK + ci * 16, d1);    // chain 1: up, or odd groups
                if (GU) {
                    __half *h = reinterpret_cast<__half *>(a.out);
#pragma unroll
                    for (int i = 0; i < 16; i++) {
                        const int col = ci * 16 + i;
                        if (col < tl.ntok) {
                            const float gv = d0[i], uv = d1[i];
                            h[(long long)(tl.start + col) * a.out_ld + row] =
                                __float2half_rn(gv / (1.0f + expf(-gv)) * uv);
                        }
                    }
                } else {
                    float *y = reinterpret_cast<float *>(a.out);
#pragma unroll
                    for (int i = 0; i < 16; i++) {
                        const int col = ci * 16 + i;
                        if (col < tl.ntok)
                            y[(long long)(tl.start + col) * a.out_ld + row] =
                                two ? d0[i] + d1[i] : d0[i];
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                bar_arrive(acc_empty + 8 * ab);
        }
        if (!ok && lane == 0) {
            *abort_flag = 1;
            atomicOr(a.status, MOE_STATUS_TIMEOUT);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------ dequant
        // warp = (chunk kh, matrix m, lane quarter q): thread = tile row
        // r = 32 q + lane (its tensor-memory lane) and the 64-K chunk kh of its
        // matrix's 128-group, i.e. 32 columns of the A stage
        const int q = warp & 3, m = (warp >> 2) & 1, kh = warp >> 3;
        const int r = 32 * q + lane, rt = r >> 4, g = r & 7, hi = (r >> 3) & 1;
        const uint32_t tlane = (uint32_t)(32 * q) << 16;
        unsigned cc = 0;
        for (unsigned t = blockIdx.x; t < total && ok; t += gridDim.x) {
            const GTile tl = gemm_tile(a, t, n_r, n_s, mt_r);
            const PackedRecs &pr = tl.shared ? a.s : a.r;
            const int nst = tile_steps<GU>(pr);
            for (int j = 0; j < nst && ok; j++) {
                const uint32_t s = cc % G::cs, as = cc % G::as;
                if (!bar_wait(code_full + 8 * s, (cc / G::cs) & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                // down's odd tail: the step has no second group
                const bool live = GU || m < step_groups<GU>(pr, j);
                // this row's slot of the record of its row tile (gate/up: slot m of
                // the record; down: the record of group m of the step); codes of
                // rows g, g + 8 for K [16 tq, 16 tq + 16) of chunk kh sit at
                // kh * 512 + chunk_slot(g, tq) * 16
                const uint8_t *rec = smem + G::c_off + s * G::code_stage +
                                     (GU ? rt * G::rec + m * kRec4 : m * G::code_group + rt * G::rec);
                RowDeq d{};
                uint4 cw[4] = {};
                if (live) {
                    d = row_deq(rec + 1024, g, hi);
#pragma unroll
                    for (int v = 0; v < 4; v++)
                        cw[v] = *reinterpret_cast<const uint4 *>(rec + kh * kChunkBytes +
                                                                 chunk_slot(g, v) * 16);
                }
                __syncwarp();
                if (lane == 0)   // the codes are in registers: the stage may be refilled
                    bar_arrive(code_empty + 8 * s);
                if (!bar_wait(stage_empty + 8 * as, ((cc / G::as) & 1) ^ 1, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (live) {
                    uint32_t col[32];
#pragma unroll
                    for (int v = 0; v < 4; v++) {
                        const uint32_t w4[4] = {cw[v].x, cw[v].y, cw[v].z, cw[v].w};
#pragma unroll
                        for (int jw = 0; jw < 4; jw++)
                            deq_row_word(w4[jw], d, col[8 * v + 2 * jw], col[8 * v + 2 * jw + 1]);
                    }
                    tmem_st32(tmem + tlane + G::acol0 + as * G::a_cols + m * 64 + kh * 32, col);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    bar_arrive(a_full + 8 * as);
                ++cc;
            }
        }
        if (!ok && lane == 0) {
            *abort_flag = 1;
            atomicOr(a.status, MOE_STATUS_TIMEOUT);
        }
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == G::mma0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"((uint32_t)G::tmem_cols)
                     : "memory");
}

// xs[r] = x[tok_of_pos[r]]; a position no pair filled this call (possible
// only after skipped pairs) gets zeros.
__global__ void gather_kernel(const __half *__restrict__ x, const int32_t *__restrict__ tok_of_pos,
                              int rows, int n, int H, __half *__restrict__ xs)
{
    pdl_enter();
    const int r = blockIdx.x;
    if (r >= rows)
        return;
    const int tok = tok_of_pos[r];
    uint4 *dst = reinterpret_cast<uint4 *>(xs + (long long)r * H);
    if (tok < 0 || tok >= n) {
        for (int i = threadIdx.x; i < H / 8; i += blockDim.x)
            dst[i] = make_uint4(0, 0, 0, 0);
        return;
    }
    const uint4 *src = reinterpret_cast<const uint4 *>(x + (long long)tok * H);
    for (int i = threadIdx.x; i < H / 8; i += blockDim.x)
        dst[i] = src[i];
}

template <bool GU, int TOK>
void set_gemm_smem()
{
    cudaFuncSetAttribute(gemm_kernel<GU, TOK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         GGeo<GU, TOK>::smem);
}

template <bool GU>
cudaError_t launch_gemm(const GemmArgs &a, const CUtensorMap &bmap, int gtok, int grid,
                        cudaStream_t st)
{
    if (gtok == kGemmTokWide)
        return launch_pdl(gemm_kernel<GU, kGemmTokWide>, dim3(grid),
                          dim3(GGeo<GU, kGemmTokWide>::threads), GGeo<GU, kGemmTokWide>::smem, st,
                          bmap, a);
    return launch_pdl(gemm_kernel<GU, kGemmTok>, dim3(grid), dim3(GGeo<GU, kGemmTok>::threads),
                      GGeo<GU, kGemmTok>::smem, st, bmap, a);
}

}  // namespace

void configure_gemm_kernels()
{
    set_gemm_smem<true, kGemmTok>();
    set_gemm_smem<false, kGemmTok>();
    set_gemm_smem<true, kGemmTokWide>();
    set_gemm_smem<false, kGemmTokWide>();
}

cudaError_t launch_gather(const LayerDev &L, const Workspace &ws, const __half *x, int n,
                          cudaStream_t st)
{
    const int rows = n * L.k + (L.has_shared ? n : 0);
    return launch_pdl(gather_kernel, dim3(rows), dim3(128), 0, st, x,
                      static_cast<const int32_t *>(ws.tok_of_pos), rows, n, L.H, ws.xs);
}

cudaError_t launch_gemm_gateup(const LayerDev &L, const Workspace &ws, const CUtensorMap &bmap,
                               int gtok, int grid, cudaStream_t st)
{
    GemmArgs a{};
    a.r = L.gu;
    a.s = L.has_shared ? L.sh_gu : L.gu;
    a.gentries = ws.gentries;
    a.hdr = ws.hdr;
    a.status = ws.hdr + 2;
    a.out = ws.h;
    a.out_ld = L.I > L.I_sh ? L.I : L.I_sh;
    return launch_gemm<true>(a, bmap, gtok, grid, st);
}

cudaError_t launch_gemm_down(const LayerDev &L, const Workspace &ws, const CUtensorMap &bmap,
                             int gtok, int grid, cudaStream_t st)
{
    GemmArgs a{};
    a.r = L.dn;
    a.s = L.has_shared ? L.sh_dn : L.dn;
    a.gentries = ws.gentries;
    a.hdr = ws.hdr;
    a.status = ws.hdr + 2;
    a.out = ws.y;
    a.out_ld = L.H;
    return launch_gemm<false>(a, bmap, gtok, grid, st);
}

}  // namespace qe
