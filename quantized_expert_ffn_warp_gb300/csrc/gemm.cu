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
// Work item: (GEMM entry = up to 256 consecutive sorted positions of one
// expert, 128-row tile of the output features).  Swap-AB: the 128 weight rows
// are the MMA's M, the entry's tokens its N (16..256, a multiple of 16).
// One persistent CTA per SM, warp-specialised:
//   - code producer warp (one lane): per 128-group, 8 bulk copies of the
//     row tiles' records into a code ring;
//   - B producer warp (one lane): per 64 K, TMA tensor loads of the
//     activation rows (32-row boxes, 128-byte swizzle) into a B ring; the two
//     producers run independently, so the weight prefetch depth is the code
//     ring's, not the B ring's;
//   - dequant warps, one per (16-row tile, matrix): unpack their part of each
//     record (LOP3 magic-number unpack, exact q - z in fp16, one rounding
//     multiply by the scale) into an A ring laid out as the MMA's K-major
//     128-byte-swizzled operand;
//   - MMA warp (one lane): allocates tensor memory, issues tcgen05.mma
//     kind::f16 (fp16 x fp16 -> fp32) for gate and up (or down) into one of
//     two accumulator buffers, and signals stage release and tile completion
//     with tcgen05.commit;
//   - four epilogue warps (one per 32-lane quarter of tensor memory): read
//     the finished buffer and write h = silu(g) * u (fp16) or y (fp32) while
//     the next tile accumulates into the other buffer.
// Every wait is bounded in time; on expiry the waiting thread raises
// MOE_STATUS_TIMEOUT and an abort flag, every role leaves its loop, the MMA
// lane waits (bounded) for its MMAs and the producer for its copies, and the
// tensor memory is freed on every path.
#include <cuda.h>
#include <cuda_fp16.h>

#include "internal.cuh"

namespace qe {

namespace {

constexpr int kGM = 128;                  // weight rows per tile (MMA M)
constexpr int kGEpi = 4;                  // epilogue warps (one per tensor-memory lane quarter)
constexpr int kABytes = kGM * 128;        // one matrix, 64 K, fp16: 16 KB
constexpr int kBBytes = kGemmTok * 128;   // kGemmTok rows x 64 K, fp16
constexpr int kBox = 32;                  // rows per TMA box
constexpr int kRec4 = 1024 + kMetaBytes;  // one matrix of a 4-bit record
static_assert(kGemmTok % kBox == 0 && kGemmTok <= 128, "two accumulator buffers fit in TMEM");

template <bool GU>
struct GGeo {
    static constexpr int mats = GU ? 2 : 1;
    static constexpr int deq = 8 * mats;                  // dequant warps: (row tile, matrix)
    static constexpr int epi0 = deq;                      // first epilogue warp (epi0 % 4 == 0)
    static constexpr int prod = deq + kGEpi;              // code producer warp
    static constexpr int bprod = prod + 1;                // B producer warp
    static constexpr int mma = bprod + 1;                 // MMA warp
    static constexpr int threads = (mma + 1) * 32;
    static constexpr int cs = GU ? 4 : 10;                // code stages (one 128-group)
    static constexpr int as = GU ? 3 : 4;                 // A stages (64 K of each matrix)
    static constexpr int bs = GU ? 3 : 4;                 // B stages (64 K x kGemmTok tokens)
    static constexpr int rec = mats * kRec4;
    static constexpr int code_stage = 8 * rec;
    static constexpr int a_stage = mats * kABytes;
    static constexpr int a_off = 0;
    static constexpr int b_off = a_off + as * a_stage;
    static constexpr int c_off = b_off + bs * kBBytes;
    static constexpr int bar_off = c_off + cs * code_stage;
    static constexpr int nbars = 2 * cs + 2 * as + 2 * bs + 5;
    static constexpr int smem = bar_off + nbars * 8 + 16 + 1024;   // + alignment slack
    static constexpr int buf_cols = mats * kGemmTok;               // one accumulator buffer
    static constexpr int tmem_cols = 2 * buf_cols;                 // 512 or 256
};
static_assert(GGeo<true>::smem <= 227 * 1024, "gate/up GEMM stages exceed shared memory");
static_assert(GGeo<false>::smem <= 227 * 1024, "down GEMM stages exceed shared memory");
static_assert(GGeo<true>::b_off % 1024 == 0 && GGeo<true>::c_off % 1024 == 0, "1 KB alignment");
static_assert(GGeo<false>::b_off % 1024 == 0 && GGeo<false>::c_off % 1024 == 0, "1 KB alignment");
static_assert(GGeo<true>::rec % 16 == 0 && GGeo<false>::rec % 16 == 0, "16-byte copies");
static_assert(GGeo<true>::bar_off % 8 == 0 && GGeo<false>::bar_off % 8 == 0, "barrier alignment");
static_assert(GGeo<true>::epi0 % 4 == 0 && GGeo<false>::epi0 % 4 == 0, "epilogue lane quarters");
static_assert(GGeo<true>::tmem_cols == 512 && GGeo<false>::tmem_cols == 256, "tensor memory");

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

__device__ __forceinline__ void bulk_copy(uint32_t dst, const void *src, uint32_t bytes,
                                          uint32_t b)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(b)
        : "memory");
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

__device__ __forceinline__ void umma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                     uint32_t accumulate)
{
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}"
        ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
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

__device__ __forceinline__ GTile gemm_tile(const GemmArgs &a, unsigned t, unsigned n_r,
                                           unsigned mt_r, unsigned mt_s)
{
    GTile g;
    unsigned ei;
    if (t < n_r * mt_r) {
        ei = t / mt_r;
        g.mt = (int)(t - ei * mt_r);
        g.shared = false;
    } else {
        const unsigned j = t - n_r * mt_r, es = j / mt_s;
        ei = n_r + es;
        g.mt = (int)(j - es * mt_s);
        g.shared = true;
    }
    const int4 e = a.gentries[ei];
    g.expert = e.x;
    g.start = e.y;
    g.ntok = e.z;
    return g;
}

// One 32-bit word of codes (rows g and g+8, four consecutive K) into four
// fp16 pairs: W = (q - z) * s rounded once.  Rows g hold 1024 + q after the
// magic-number LOP3, rows g+8 hold 1024 + 16 q; both differences are exact.
struct DeqConst {
    __half2 zg, sg;     // row g: 1024 + z, scale
    __half2 zg8, sg8;   // row g+8: -(64 + z), scale
};

__device__ __forceinline__ void deq_word(uint32_t w, const DeqConst &c, uint32_t (&rg)[2],
                                         uint32_t (&rg8)[2])
{
    const __half2 sixteenth = __float2half2_rn(0.0625f);
    const uint32_t w8 = w >> 8;
    rg[0] = h2u(__hmul2(__hsub2(u2h(lop_magic(w, 0x000F000Fu)), c.zg), c.sg));
    rg[1] = h2u(__hmul2(__hsub2(u2h(lop_magic(w8, 0x000F000Fu)), c.zg), c.sg));
    rg8[0] = h2u(__hmul2(__hfma2(u2h(lop_magic(w, 0x00F000F0u)), sixteenth, c.zg8), c.sg8));
    rg8[1] = h2u(__hmul2(__hfma2(u2h(lop_magic(w8, 0x00F000F0u)), sixteenth, c.zg8), c.sg8));
}

__device__ __forceinline__ DeqConst deq_const(const uint8_t *meta, int g)
{
    const __half2 s = *reinterpret_cast<const __half2 *>(meta + 4 * g);
    const unsigned z = *reinterpret_cast<const uint16_t *>(meta + 32 + 2 * g);
    DeqConst c;
    c.zg = __float2half2_rn(1024.0f + (float)(z & 0xFF));
    c.zg8 = __float2half2_rn(-(64.0f + (float)(z >> 8)));
    c.sg = __half2half2(__low2half(s));
    c.sg8 = __half2half2(__high2half(s));
    return c;
}

template <bool GU>
__global__ void __launch_bounds__(GGeo<GU>::threads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap bmap, GemmArgs a)
{
    using G = GGeo<GU>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (saddr(smem_raw) & 1023u)) & 1023u);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + G::bar_off);
    const uint32_t code_full = saddr(bars), code_empty = code_full + 8 * G::cs;
    const uint32_t a_full = code_empty + 8 * G::cs, a_empty = a_full + 8 * G::as;
    const uint32_t b_full = a_empty + 8 * G::as, b_empty = b_full + 8 * G::bs;
    const uint32_t acc_full = b_empty + 8 * G::bs;  // [2]
    const uint32_t acc_empty = acc_full + 16;       // [2]
    const uint32_t drain = acc_empty + 16;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + G::nbars);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    if (threadIdx.x == 0) {
        for (int s = 0; s < G::cs; s++) {
            bar_init(code_full + 8 * s, 1);
            bar_init(code_empty + 8 * s, G::deq);
        }
        for (int s = 0; s < G::as; s++) {
            bar_init(a_full + 8 * s, G::deq);
            bar_init(a_empty + 8 * s, 1);
        }
        for (int s = 0; s < G::bs; s++) {
            bar_init(b_full + 8 * s, 1);
            bar_init(b_empty + 8 * s, 1);
        }
        for (int j = 0; j < 2; j++) {
            bar_init(acc_full + 8 * j, 1);
            bar_init(acc_empty + 8 * j, kGEpi);
        }
        bar_init(drain, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == G::mma) {
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
            for (unsigned t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const GTile tl = gemm_tile(a, t, n_r, mt_r, mt_s);
                const PackedRecs &pr = tl.shared ? a.s : a.r;
                const uint8_t *base = pr.recs + (long long)(tl.shared ? 0 : tl.expert) *
                                                    pr.expert_bytes;
                for (int gi = 0; gi < pr.n_groups; gi++) {
                    const uint32_t s = cc % G::cs;
                    if (!bar_wait(code_empty + 8 * s, ((cc / G::cs) & 1) ^ 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    bar_expect_tx(code_full + 8 * s, G::code_stage);
                    // the tile's 8 row tiles: 8 records, or 4 records of row-tile pairs
                    const uint32_t dst = saddr(smem + G::c_off + s * G::code_stage);
                    const int nu = pr.pair ? 4 : 8;
                    for (int u = 0; u < nu; u++)
                        bulk_copy(dst + u * pr.rec,
                                  base + ((long long)(nu * tl.mt + u) * pr.n_groups + gi) * pr.rec,
                                  pr.rec, code_full + 8 * s);
                    ++cc;
                }
            }
            if (!ok) {
                *abort_flag = 1;
                atomicOr(a.status, MOE_STATUS_TIMEOUT);
                // the last stages issued land before the CTA leaves
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
                const GTile tl = gemm_tile(a, t, n_r, mt_r, mt_s);
                const PackedRecs &pr = tl.shared ? a.s : a.r;
                const int nb = (tl.ntok + kBox - 1) / kBox;
                for (int kc = 0; kc < 2 * pr.n_groups; kc++) {
                    const uint32_t b = bc % G::bs;
                    if (!bar_wait(b_empty + 8 * b, ((bc / G::bs) & 1) ^ 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    bar_expect_tx(b_full + 8 * b, nb * kBox * 128);
                    const uint32_t bdst = saddr(smem + G::b_off + b * kBBytes);
                    for (int j = 0; j < nb; j++)
                        tma_load_2d(bdst + j * kBox * 128, &bmap, kc * 64, tl.start + j * kBox,
                                    b_full + 8 * b);
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
    } else if (warp == G::mma) {
        // ------------------------------------------------------ MMA issuer
        if (lane == 0) {
            unsigned ac = 0, bc = 0, ti = 0;
            bool issued = false;
            for (unsigned t = blockIdx.x; t < total && ok; t += gridDim.x, ti++) {
                const GTile tl = gemm_tile(a, t, n_r, mt_r, mt_s);
                const PackedRecs &pr = tl.shared ? a.s : a.r;
                const int nmma = ((max(tl.ntok, 16) + 15) / 16) * 16;
                const uint32_t idesc = idesc_f16(nmma);
                const uint32_t j = ti & 1;
                if (!bar_wait(acc_empty + 8 * j, ((ti >> 1) & 1) ^ 1, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t dbuf = tmem + j * G::buf_cols;
                for (int gi = 0; gi < pr.n_groups && ok; gi++) {
                    for (int c = 0; c < 2; c++) {
                        const uint32_t as = ac % G::as, bs = bc % G::bs;
                        if (!bar_wait(a_full + 8 * as, (ac / G::as) & 1, abort_flag) ||
                            !bar_wait(b_full + 8 * bs, (bc / G::bs) & 1, abort_flag)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t abase = saddr(smem + G::a_off + as * G::a_stage);
                        const uint32_t bbase = saddr(smem + G::b_off + bs * kBBytes);
#pragma unroll
                        for (int kk = 0; kk < 4; kk++) {
                            const uint64_t bd = sw128_desc(bbase + kk * 32);
#pragma unroll
                            for (int m = 0; m < G::mats; m++)
                                umma(dbuf + m * kGemmTok, sw128_desc(abase + m * kABytes + kk * 32),
                                     bd, idesc, (gi | c | kk) != 0);
                        }
                        issued = true;
                        umma_commit(a_empty + 8 * as);
                        umma_commit(b_empty + 8 * bs);
                        ++ac;
                        ++bc;
                    }
                }
                if (ok)
                    umma_commit(acc_full + 8 * j);
            }
            if (!ok) {
                *abort_flag = 1;
                atomicOr(a.status, MOE_STATUS_TIMEOUT);
            }
            if (issued) {   // every MMA issued has completed before the memory is freed
                umma_commit(drain);
                const unsigned long long t0 = now_ns();
                while (!bar_try(drain, 0) && now_ns() - t0 < kGWaitNs) {
                }
            }
        }
        __syncwarp();
    } else if (warp >= G::epi0) {
        // ------------------------------------------------------ epilogue
        // rows 32 q + lane of the tile (q = this warp's tensor-memory lane quarter)
        const int q = warp & 3;
        unsigned ti = 0;
        for (unsigned t = blockIdx.x; t < total && ok; t += gridDim.x, ti++) {
            const GTile tl = gemm_tile(a, t, n_r, mt_r, mt_s);
            const uint32_t j = ti & 1;
            if (!bar_wait(acc_full + 8 * j, (ti >> 1) & 1, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int row = tl.mt * kGM + 32 * q + lane;
            const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16) + j * G::buf_cols;
            const int nchunks = (tl.ntok + 15) / 16;
            for (int ci = 0; ci < nchunks; ci++) {
                float d0[16];
                tmem_ld16(taddr + ci * 16, d0);
                if (GU) {
                    float d1[16];
                    tmem_ld16(taddr + kGemmTok + ci * 16, d1);
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
                            y[(long long)(tl.start + col) * a.out_ld + row] = d0[i];
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                bar_arrive(acc_empty + 8 * j);
        }
        if (!ok && lane == 0) {
            *abort_flag = 1;
            atomicOr(a.status, MOE_STATUS_TIMEOUT);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------ dequant
        // warp = (matrix m, row tile rt): lane (g, tq) owns rows g, g + 8 of
        // the row tile and K [16 tq, 16 tq + 16) of each 64-K chunk
        const int rt = warp & 7, m = warp >> 3;
        const int g = lane >> 2, tq = lane & 3;
        const int r0 = rt * 16 + g, r1 = r0 + 8;
        unsigned cc = 0, ac = 0;
        for (unsigned t = blockIdx.x; t < total && ok; t += gridDim.x) {
            const GTile tl = gemm_tile(a, t, n_r, mt_r, mt_s);
            const PackedRecs &pr = tl.shared ? a.s : a.r;
            for (int gi = 0; gi < pr.n_groups && ok; gi++) {
                const uint32_t s = cc % G::cs;
                if (!bar_wait(code_full + 8 * s, (cc / G::cs) & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                const uint8_t *rec = smem + G::c_off + s * G::code_stage + rt * G::rec + m * kRec4;
                const DeqConst dc = deq_const(rec + 1024, g);
                const uint4 qv[2] = {*reinterpret_cast<const uint4 *>(rec + lane * 16),
                                     *reinterpret_cast<const uint4 *>(rec + 512 + lane * 16)};
                __syncwarp();
                if (lane == 0)   // the codes are in registers: the stage may be refilled
                    bar_arrive(code_empty + 8 * s);
                ++cc;
                for (int c = 0; c < 2; c++) {
                    const uint32_t as = ac % G::as;
                    if (!bar_wait(a_empty + 8 * as, ((ac / G::as) & 1) ^ 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t wq[4] = {qv[c].x, qv[c].y, qv[c].z, qv[c].w};
                    uint32_t rg[4][2], rg8[4][2];
#pragma unroll
                    for (int jw = 0; jw < 4; jw++)
                        deq_word(wq[jw], dc, rg[jw], rg8[jw]);
                    // row r, 16-byte chunk ch of the 128-byte row, swizzled by r & 7
                    uint8_t *am = smem + G::a_off + as * G::a_stage + m * kABytes;
#pragma unroll
                    for (int h = 0; h < 2; h++) {
                        const int ch = 2 * tq + h;
                        *reinterpret_cast<uint4 *>(am + r0 * 128 + ((ch ^ (r0 & 7)) << 4)) =
                            make_uint4(rg[2 * h][0], rg[2 * h][1], rg[2 * h + 1][0],
                                       rg[2 * h + 1][1]);
                        *reinterpret_cast<uint4 *>(am + r1 * 128 + ((ch ^ (r1 & 7)) << 4)) =
                            make_uint4(rg8[2 * h][0], rg8[2 * h][1], rg8[2 * h + 1][0],
                                       rg8[2 * h + 1][1]);
                    }
                    // generic-proxy writes become visible to the tensor core's reads
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    __syncwarp();
                    if (lane == 0)
                        bar_arrive(a_full + 8 * as);
                    ++ac;
                }
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
    if (warp == G::mma)
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

template <bool GU>
void set_gemm_smem()
{
    cudaFuncSetAttribute(gemm_kernel<GU>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         GGeo<GU>::smem);
}

}  // namespace

void configure_gemm_kernels()
{
    set_gemm_smem<true>();
    set_gemm_smem<false>();
}

cudaError_t launch_gather(const LayerDev &L, const Workspace &ws, const __half *x, int n,
                          cudaStream_t st)
{
    const int rows = n * L.k + (L.has_shared ? n : 0);
    return launch_pdl(gather_kernel, dim3(rows), dim3(128), 0, st, x,
                      static_cast<const int32_t *>(ws.tok_of_pos), rows, n, L.H, ws.xs);
}

cudaError_t launch_gemm_gateup(const LayerDev &L, const Workspace &ws, const CUtensorMap &bmap,
                               int grid, cudaStream_t st)
{
    GemmArgs a{};
    a.r = L.gu;
    a.s = L.has_shared ? L.sh_gu : L.gu;
    a.gentries = ws.gentries;
    a.hdr = ws.hdr;
    a.status = ws.hdr + 2;
    a.out = ws.h;
    a.out_ld = L.I > L.I_sh ? L.I : L.I_sh;
    return launch_pdl(gemm_kernel<true>, dim3(grid), dim3(GGeo<true>::threads), GGeo<true>::smem, st,
                      bmap, a);
}

cudaError_t launch_gemm_down(const LayerDev &L, const Workspace &ws, const CUtensorMap &bmap,
                             int grid, cudaStream_t st)
{
    GemmArgs a{};
    a.r = L.dn;
    a.s = L.has_shared ? L.sh_dn : L.dn;
    a.gentries = ws.gentries;
    a.hdr = ws.hdr;
    a.status = ws.hdr + 2;
    a.out = ws.y;
    a.out_ld = L.H;
    return launch_pdl(gemm_kernel<false>, dim3(grid), dim3(GGeo<false>::threads), GGeo<false>::smem,
                      st, bmap, a);
}

}  // namespace qe
