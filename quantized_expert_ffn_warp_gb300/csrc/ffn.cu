// Expert FFN: weight repacking and the fused dequant x GEMV/GEMM kernels.
//
// Group-wise INT4 (or 2-bit) weights W = (q - zero) * scale, one fp16 scale
// and zero point per 128 consecutive K elements ("Strata" article, section
// 2.2; "为什么12G显存笔记本能跑MoE-16B" section 4.2: the codes are unpacked
// inside the kernel and never written back as fp16), gate/up projection with
// SwiGLU h = silu(g) * u, then the down projection ("Flash-MoE" article,
// section 3: dequant matvec, fused SwiGLU).  Decode is bound by the bytes of
// the touched experts' weights ("Strata" section 1.1), so the kernels stream
// each expert's codes exactly once per call and keep every token routed to
// that expert in the same pass ("Strata" sections 2.3 and 3.4: one weight
// read serves every token that shares the expert).
//
// Packed layout (built by repack): one record per (expert, unit, 128-group)
// with two slots, each the codes of one 16-row tile and group followed by its
// 48-byte scale/zero block (8 pairs (row g, row g+8) of fp16 scales, then 8
// pairs of byte zero points).  Gate/up: the unit is a row tile and the slots
// are the gate and the up matrix.  Down: the unit is a pair of row tiles and
// the slots are its two tiles, so both kinds of record are processed alike,
// two 16-row MMA operands sharing one activation fragment.
// The codes of a record are CPG chunks of 512 bytes (CPG = 2 for 4-bit, 1 for
// 2-bit), one 16-byte word per lane of a warp (at chunk_slot(g, t)): lane
// (g = lane/4, t = lane%4) owns rows g and g+8 and the K range
// [t*CK/4, (t+1)*CK/4) of the 64-K (4-bit) or 128-K (2-bit) chunk, and the
// fields inside each 32-bit word are
// ordered so that a LOP3 with the fp16 magic number 0x6400 turns two of them
// into the two fp16 halves of one register of the A fragment of an m16n8k16
// tensor-core MMA.  The K order inside a lane's slice is the natural one, so
// the activation operand is one contiguous 16-byte load per 8 K and token.
//
// Arithmetic: a LOP3 turns two fields into the fp16 pair 1024 + q (or
// 1024 + 16q for the rows g+8 of a 4-bit word), the exact field value.  The
// MMA multiplies fragments by the fp16 activations and accumulates in fp32
// over one 128-group; per group and row the kernel then adds s times the
// group's sum of (q - z) a to the row's fp32 total (s / 16 for the rows g+8
// of a 4-bit word).  The zero point enters in one of two exact-or-bounded
// ways:
//   gate/up: the MMA takes the raw fields, and the group sum is corrected
//     by the zero point's field value zf = 1024 + z (or 1024 + 16z) times
//     the group's activation sum, sum (1024 + q) a - zf sum a, in one fp32
//     FMA.  The activation sums (fp32, one fixed summation order) come with
//     the routing launch, so the per-weight work is one LOP3 per two
//     weights.  The 2-bit fields of a register carry 4^j q (j = 0..3); with
//     the activations of each k-step's second register scaled by 1/16 (one
//     exact HMUL2 per 16 weights), rows g see q and rows g+8 4q at every k,
//     and the correction takes two activation partial sums (k % 4 < 2 and
//     k % 4 >= 2) with zf = 1024 + z and 64 + z (rows g+8: 1024 + 4z and
//     64 + 4z), in two FMAs.
//   down: the fragments are made the exact small integer q - z before the
//     MMA, by one HSUB2 (4-bit) or by the HFMA2 that 2-bit fields need
//     anyway (2-bit: x 4^-j with the zero point in the addend).
// The tensor core is the multiply-add engine because the per-weight ALU
// budget at HBM speed (about 2.5 issue slots per weight) leaves no room for a
// scalar convert and FMA per weight.  On this part a legacy m16n8k16 MMA costs
// the issuing sub-partition about ten cycles in which little else issues, so
// the 16 MMAs of a record are these kernels' largest cost, and every ALU
// instruction per weight removed around them shows in the time.
#include <cuda_fp16.h>

#include "internal.cuh"

namespace qe {

// ------------------------------------------------------------ repacking

__host__ __device__ constexpr int code_bytes(int wb)
{
    return kGroup * wb / 8 * kRowTile;   // codes of 16 rows x 128 K
}

// Record order: [expert][128-row tile][group][unit of the tile], u units per
// 128-row tile (8 row tiles, or 4 row-tile pairs): the records a 128-row
// tile needs for one K group are one contiguous block, and a row tile's
// records of consecutive groups are u records apart.
__host__ __device__ __forceinline__ long long rec_index(long long e, int unit, int grp, int n_units,
                                                        int G, int u)
{
    return ((e * (n_units / u) + unit / u) * G + grp) * u + unit % u;
}

template <int WB>
__global__ void repack_codes_kernel(const uint8_t *__restrict__ canon, int n_exp, int rows,
                                    int K, int m, int mats, int pair, uint8_t *__restrict__ out)
{
    constexpr int CK = 256 / WB, CPG = kGroup / CK, CODE = code_bytes(WB);
    const int n_rt = rows / kRowTile, n_c = K / CK, G = K / kGroup;
    const int rec = (pair ? 2 : mats) * (CODE + kMetaBytes);
    const long long total = (long long)n_exp * n_rt * n_c * 32;
    const long long row_bytes = (long long)K * WB / 8;
    for (long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x; gid < total;
         gid += (long long)gridDim.x * blockDim.x) {
        const int lane = (int)(gid & 31);
        long long rest = gid >> 5;
        const int c = (int)(rest % n_c);
        rest /= n_c;
        const int rt = (int)(rest % n_rt);
        const long long e = rest / n_rt;
        const int g = lane >> 2, t = lane & 3;
        const uint8_t *ra = canon + (e * rows + rt * kRowTile + g) * row_bytes;
        const uint8_t *rb = ra + 8 * row_bytes;
        uint32_t wd[4];
        if (WB == 4) {
#pragma unroll
            for (int j = 0; j < 4; j++) {
                const int k0 = c * 64 + 16 * t + 4 * j;
                const uint32_t a0 = ra[k0 / 2], a1 = ra[k0 / 2 + 1];
                const uint32_t b0 = rb[k0 / 2], b1 = rb[k0 / 2 + 1];
                // row g: k0, k0+1, k0+2, k0+3 -> nibbles 0, 4, 2, 6
                // row g+8:                    -> nibbles 1, 5, 3, 7
                wd[j] = (a0 & 15) | ((b0 & 15) << 4) | ((a1 & 15) << 8) | ((b1 & 15) << 12) |
                        ((a0 >> 4) << 16) | ((b0 >> 4) << 20) | ((a1 >> 4) << 24) |
                        ((b1 >> 4) << 28);
            }
        } else {
#pragma unroll
            for (int w = 0; w < 4; w++) {
                uint32_t word = 0;
#pragma unroll
                for (int hs = 0; hs < 2; hs++) {
                    const int j = 2 * w + hs;
                    const int k0 = c * 128 + 32 * t + 4 * j;
                    const uint32_t a = ra[k0 / 4], b = rb[k0 / 4];
                    const int base = 4 * hs;
                    // k-step fields: row g (k0, k0+1) -> (base, base+8); row g+8 ->
                    // (base+1, base+9); row g (k0+2, k0+3) -> (base+2, base+10);
                    // row g+8 (k0+2, k0+3) -> (base+3, base+11)
                    word |= ((a >> 0) & 3) << (2 * (base + 0));
                    word |= ((a >> 2) & 3) << (2 * (base + 8));
                    word |= ((b >> 0) & 3) << (2 * (base + 1));
                    word |= ((b >> 2) & 3) << (2 * (base + 9));
                    word |= ((a >> 4) & 3) << (2 * (base + 2));
                    word |= ((a >> 6) & 3) << (2 * (base + 10));
                    word |= ((b >> 4) & 3) << (2 * (base + 3));
                    word |= ((b >> 6) & 3) << (2 * (base + 11));
                }
                wd[w] = word;
            }
        }
        // paired layout: row tiles 2p and 2p+1 share a record, in slots 0 and 1
        const int slot = pair ? (rt & 1) : m;
        const long long r = rec_index(e, pair ? rt >> 1 : rt, c / CPG, pair ? n_rt / 2 : n_rt, G,
                                      pair ? 4 : 8);
        uint8_t *dst =
            out + r * rec + slot * (CODE + kMetaBytes) + (c % CPG) * kChunkBytes +
            chunk_slot(g, t) * 16;
        *reinterpret_cast<uint4 *>(dst) = make_uint4(wd[0], wd[1], wd[2], wd[3]);
    }
}

template <int WB>
__global__ void repack_meta_kernel(const uint16_t *__restrict__ scales,
                                   const uint8_t *__restrict__ zeros, int n_exp, int rows, int K,
                                   int m, int mats, int pair, uint8_t *__restrict__ out)
{
    constexpr int CODE = code_bytes(WB);
    const int G = K / kGroup, n_rt = rows / kRowTile;
    const int rec = (pair ? 2 : mats) * (CODE + kMetaBytes);
    const long long total = (long long)n_exp * n_rt * G * kRowTile;
    for (long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x; gid < total;
         gid += (long long)gridDim.x * blockDim.x) {
        const int r = (int)(gid % kRowTile);
        long long rest = gid / kRowTile;
        const int grp = (int)(rest % G);
        rest /= G;
        const int rt = (int)(rest % n_rt);
        const long long e = rest / n_rt;
        const long long src = (e * rows + rt * kRowTile + r) * G + grp;
        const int slot = pair ? (rt & 1) : m;
        const long long rr = rec_index(e, pair ? rt >> 1 : rt, grp, pair ? n_rt / 2 : n_rt, G,
                                       pair ? 4 : 8);
        uint8_t *dst = out + rr * rec + slot * (CODE + kMetaBytes) + CODE;
        const int gp = r & 7, half = r >> 3;   // (row g, row g+8) pairs
        reinterpret_cast<uint16_t *>(dst)[2 * gp + half] = scales[src];
        dst[32 + 2 * gp + half] = zeros[src];
    }
}

cudaError_t launch_repack(const uint8_t *codes, const uint16_t *scales, const uint8_t *zeros,
                          int n_exp, int rows, int K, int wbits, int m, int mats, int pair,
                          uint8_t *out, cudaStream_t st)
{
    const int threads = 256, blocks = 4096;
    if (wbits == 4) {
        repack_codes_kernel<4><<<blocks, threads, 0, st>>>(codes, n_exp, rows, K, m, mats, pair,
                                                           out);
        repack_meta_kernel<4><<<blocks, threads, 0, st>>>(scales, zeros, n_exp, rows, K, m, mats,
                                                          pair, out);
    } else {
        repack_codes_kernel<2><<<blocks, threads, 0, st>>>(codes, n_exp, rows, K, m, mats, pair,
                                                           out);
        repack_meta_kernel<2><<<blocks, threads, 0, st>>>(scales, zeros, n_exp, rows, K, m, mats,
                                                          pair, out);
    }
    return cudaGetLastError();
}

// ------------------------------------------------------------ device helpers

__device__ __forceinline__ uint4 ld_act(const void *p)
{
    return __ldg(reinterpret_cast<const uint4 *>(p));
}

// (a & mask) | 0x64006400: the two selected fields become fp16 1024 + field.
__device__ __forceinline__ uint32_t lop_magic(uint32_t a, uint32_t mask)
{
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(mask), "r"(0x64006400u));
    return d;
}

__device__ __forceinline__ uint32_t hmul2_u(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ uint32_t hfma2_u(uint32_t a, uint32_t b, uint32_t c)
{
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// A fragment of one k-step as raw magic-number fields.  4-bit: rows g hold
// 1024 + q, rows g+8 1024 + 16q.  2-bit: the four registers hold 1024 + q
// (rows g, first k half), 1024 + 4q (rows g+8, first half), 1024 + 16q (rows
// g, second half), 1024 + 64q (rows g+8, second half); the B register of the
// second half is scaled by 1/16 (load_b), so rows g see q and rows g+8 4q
// throughout, plus 1024 x or 64 x.
template <int WB>
__device__ __forceinline__ void frag(uint32_t w, int hs, uint32_t (&a)[4])
{
    if (WB == 4) {
        const uint32_t w8 = w >> 8;
        a[0] = lop_magic(w, 0x000F000Fu);
        a[1] = lop_magic(w, 0x00F000F0u);
        a[2] = lop_magic(w8, 0x000F000Fu);
        a[3] = lop_magic(w8, 0x00F000F0u);
    } else {
        const uint32_t v = hs ? (w >> 8) : w;
        a[0] = lop_magic(v, 0x00030003u);
        a[1] = lop_magic(v, 0x000C000Cu);
        a[2] = lop_magic(v, 0x00300030u);
        a[3] = lop_magic(v, 0x00C000C0u);
    }
}

// Scale and zero-point terms of one (matrix, group) for a lane's rows g, g+8.
// ZC (zero point by correction, the gate/up kernels): the MMA sees the raw
// field values (frag) and the group's sum is corrected in fp32 by the field
// value of the zero point times the group sum of the activations: 4-bit
// zf = 1024 + z (rows g) or 1024 + 16z (rows g+8); 2-bit, per partial sum
// (k % 4 < 2, k % 4 >= 2): 1024 + z and 64 + z (rows g), 1024 + 4z and
// 64 + 4z (rows g+8).  Otherwise (down kernels) the fragments are made exact
// q - z before the MMA: z_lo, z_hi are the zero point's field values for one
// HSUB2, and for 2-bit rows c1..c3 the addends that turn the HFMA2 of the
// shifted fields into q - z.
struct GroupMeta {
    float s_lo, s_hi;      // scale of the row's group sum
    float zf_lo, zf_hi;    // ZC: field value of the zero point (2-bit: first partial sum)
    float zf2_lo, zf2_hi;  // ZC, 2-bit: for the second partial sum
    __half2 z_lo, z_hi;    // otherwise: field value of the zero point, both halves
    __half2 c1, c2, c3;    // otherwise, 2-bit: -(256 + z_hi), -(64 + z_lo), -(16 + z_hi)
};

// 2^23 + b as fp32, b the byte of v named by the selector's low nibble (one
// PRMT: byte b, then bytes 0, 0 and 0x4B of 2^23's bit pattern).
__device__ __forceinline__ float byte_plus_2p23(unsigned v, unsigned sel)
{
    unsigned d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(v), "r"(0x4B000000u), "r"(sel));
    return __uint_as_float(d);
}

template <int WB, bool ZC>
__device__ __forceinline__ GroupMeta group_meta(const uint8_t *meta, int g)
{
    const float2 s = __half22float2(*reinterpret_cast<const __half2 *>(meta + 4 * g));
    const unsigned z = *reinterpret_cast<const uint16_t *>(meta + 32 + 2 * g);
    GroupMeta k;
    k.s_lo = s.x;
    // 4-bit rows g+8 carry 16q: scale s/16; 2-bit ZC rows g+8 carry 4q
    k.s_hi = WB == 4 ? s.y * 0.0625f : ZC ? s.y * 0.25f : s.y;
    if (ZC) {
        // bytes z_lo (0) and z_hi (1) into the low byte of 2^23 (exact), then
        // the zero points' field values, each exact in one FADD or FFMA
        const float zl = byte_plus_2p23(z, 0x7540u);
        const float zh = byte_plus_2p23(z, 0x7541u);
        k.zf_lo = zl - 8387584.0f;                               // 1024 + z: - (2^23 - 1024)
        if (WB == 4) {
            k.zf_hi = fmaf(zh, 16.0f, -134216704.0f);            // 16 (2^23 + z) - (2^27 - 1024)
        } else {
            k.zf2_lo = zl - 8388544.0f;                          // 64 + z: - (2^23 - 64)
            k.zf_hi = fmaf(zh, 4.0f, -33553408.0f);              // 4 (2^23 + z) - (2^25 - 1024)
            k.zf2_hi = fmaf(zh, 4.0f, -33554368.0f);             // 4 (2^23 + z) - (2^25 - 64)
        }
    } else {
        const float zl = (float)(z & 0xFF), zh = (float)(z >> 8);
        k.z_lo = __float2half2_rn(1024.0f + zl);
        if (WB == 4) {
            k.z_hi = __float2half2_rn(1024.0f + 16.0f * zh);
        } else {
            k.z_hi = __float2half2_rn(1024.0f + zh);
            k.c1 = __float2half2_rn(-(256.0f + zh));
            k.c2 = __float2half2_rn(-(64.0f + zl));
            k.c3 = __float2half2_rn(-(16.0f + zh));
        }
    }
    return k;
}

// 2-bit A fragment of one k-step made exact q - z directly: register 0 by
// one HSUB2 of its 1024 + q fields, registers 1..3 by one HFMA2 of the
// shifted fields (1024 + 4^j q) x 4^-j + c_j, exact because the result is a
// small integer.
__device__ __forceinline__ void frag2_exact(uint32_t w, int hs, const GroupMeta &k,
                                            uint32_t (&a)[4])
{
    const uint32_t v = hs ? (w >> 8) : w;
    const uint32_t r0 = lop_magic(v, 0x00030003u);
    const __half2 d0 = __hsub2(*reinterpret_cast<const __half2 *>(&r0), k.z_lo);
    a[0] = *reinterpret_cast<const uint32_t *>(&d0);
    a[1] = hfma2_u(lop_magic(v, 0x000C000Cu), 0x34003400u, *reinterpret_cast<const uint32_t *>(&k.c1));
    a[2] = hfma2_u(lop_magic(v, 0x00300030u), 0x2C002C00u, *reinterpret_cast<const uint32_t *>(&k.c2));
    a[3] = hfma2_u(lop_magic(v, 0x00C000C0u), 0x24002400u, *reinterpret_cast<const uint32_t *>(&k.c3));
}

// The fields of an A fragment minus the zero-point fields of their rows
// (registers 0, 2: rows g; 1, 3: rows g+8): exact small integers.
__device__ __forceinline__ void sub_zero(uint32_t (&a)[4], const GroupMeta &k)
{
#pragma unroll
    for (int r = 0; r < 4; r++) {
        const __half2 d = __hsub2(*reinterpret_cast<const __half2 *>(&a[r]), r & 1 ? k.z_hi : k.z_lo);
        a[r] = *reinterpret_cast<const uint32_t *>(&d);
    }
}

// ------------------------------------------------------------ FFN kernels
//
// One persistent CTA per SM holding kWG warp groups of kWW warps.  Work items
// are (entry, 16-row tile); warp group v of the grid (of V) takes the
// contiguous item range [total v / V, total (v+1) / V), so consecutive items
// mostly share an entry and its activation rows.  Inside a group, warp w owns
// the K slice [w G / kWW, (w+1) G / kWW) of 128-groups of every item, so the
// warps of a group split each row tile's K range and never need the same
// bytes.
//
// Every warp streams its own K slices through a private ring of kS stages.
// A unit is up to UG consecutive groups of one item, i.e. UG consecutive
// records: lane 0 issues one bulk asynchronous copy per unit (at least 2 KB,
// because the copy engine starts a bounded number of copies per microsecond
// per SM), completing on the stage's mbarrier, kS - 1 units ahead of the one
// being multiplied, across item boundaries.  No warp waits on another warp to
// get its data.  The warp reads the codes and scales from shared memory and
// the activations through L1, and multiplies on the tensor core.  After an
// item's last unit every warp of the group writes its partial sums to one of
// two reduction slots and counts itself in; the last warp to arrive reduces
// the slot in a fixed warp order and writes h (gate/up, after SwiGLU) or y
// (down).  The work entries are copied into shared memory once per kernel.
//
// Every wait (on a stage's mbarrier or on a reduction slot) is bounded in
// time: on expiry the warp raises MOE_STATUS_TIMEOUT and an abort flag makes
// the other warps of its group stop; every warp waits (again bounded) for its
// own copies still in flight before it leaves.

struct FfnArgs {
    PackedRecs r, s;       // routed and shared-expert records of this stream
    const Entry *entries;
    const int *hdr;
    int *status;
    const __half *act;     // gate/up: x [n][H] by token; down: h [P+n][ld] by position
    long long act_ld;
    void *out;             // gate/up: h (fp16); down: y (fp32)
    long long out_ld;
    const float *xsum;     // gate/up: [n][H/128] activation group sums (2-bit: [n][H/128][2])
    int xs_ld;
};

#ifndef QE_FFN_WW
#define QE_FFN_WW 4
#endif
#ifndef QE_FFN_WG
#define QE_FFN_WG 4
#endif
#ifndef QE_FFN_STAGES
#define QE_FFN_STAGES 3
#endif
#ifndef QE_FFN_ENTCAP
#define QE_FFN_ENTCAP 768
#endif
#ifndef QE_FFN_MINCOPY
#define QE_FFN_MINCOPY 2048
#endif
constexpr int kWW = QE_FFN_WW;                           // warps per group
constexpr int kS = QE_FFN_STAGES;                        // stages per warp
constexpr int kEntCap = QE_FFN_ENTCAP;                   // entries kept in shared memory
constexpr int kMinCopy = QE_FFN_MINCOPY;                 // bytes per bulk copy, at least

// Kernel shape: kWG warp groups of kWW warps per CTA (more warps measured
// slower); an entry holds at most 8 tokens, one MMA column tile.
constexpr int kWG = QE_FFN_WG;
constexpr int kFfnThreads = kWW * kWG * 32;
constexpr int kRed = kWW * 2 * 4 * 32;   // floats of a reduction slot: [warp][mat][4][32]
static_assert(kMaxTokTile == 8, "one 8-token MMA tile per entry");

template <int WB, bool GU>
struct Geo {
    static constexpr int mats = 2;                       // record slots (gate/up, or 2 row tiles)
    static constexpr int cpg = kGroup / (256 / WB);      // chunks per group
    static constexpr int code = code_bytes(WB);          // bytes of codes per matrix and group
    static constexpr int rec = mats * (code + kMetaBytes);
    static constexpr int ug = (kMinCopy + rec - 1) / rec;   // groups per unit
    static constexpr int stage = ug * rec;
    static constexpr int ring = kS * stage;              // per warp
    static constexpr int group = kWW * ring + 2 * kRed * 4 + 64;
    static constexpr int warp_ctl = kS * 8;              // mbarriers per warp
    static constexpr int smem = kWG * group + kFfnThreads / 32 * warp_ctl + kEntCap * 16;
};
static_assert(Geo<4, true>::smem <= 227 * 1024, "gate/up stages exceed shared memory");
static_assert(Geo<4, false>::smem <= 227 * 1024, "down stages exceed shared memory");
static_assert(Geo<2, true>::smem <= 227 * 1024, "gate/up stages exceed shared memory");
static_assert(Geo<2, false>::smem <= 227 * 1024, "down stages exceed shared memory");
static_assert(Geo<4, true>::stage % 16 == 0 && Geo<2, false>::stage % 16 == 0, "16-byte copies");

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ unsigned long long global_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

constexpr unsigned long long kWaitLimitNs = 2000000000ull;   // 2 s

// Bounded wait for the phase of `parity` to complete.  False on expiry or
// when another warp of the group has aborted.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag)
{
    if (mbar_try(bar, parity))
        return true;
    const unsigned long long t0 = global_ns();
    for (unsigned it = 0;; it++) {
        if (mbar_try(bar, parity))
            return true;
        if ((it & 15) == 15 && (*abort_flag || global_ns() - t0 > kWaitLimitNs))
            return false;
    }
}

// Shared-memory counters with acquire/release ordering at CTA scope.
__device__ __forceinline__ unsigned atom_inc_acq_rel(unsigned *p, unsigned wrap)
{
    unsigned old;
    asm volatile("atom.acq_rel.cta.shared::cta.inc.u32 %0, [%1], %2;"
                 : "=r"(old)
                 : "r"(smem_addr(p)), "r"(wrap)
                 : "memory");
    return old;
}

__device__ __forceinline__ int ld_acquire(const volatile int *p)
{
    int v;
    asm volatile("ld.acquire.cta.shared::cta.s32 %0, [%1];"
                 : "=r"(v)
                 : "r"(smem_addr(const_cast<const int *>(p)))
                 : "memory");
    return v;
}

__device__ __forceinline__ void st_release(volatile int *p, int v)
{
    asm volatile("st.release.cta.shared::cta.s32 [%0], %1;" ::"r"(smem_addr(const_cast<int *>(p))),
                 "r"(v)
                 : "memory");
}

#ifndef QE_FFN_EVF
#define QE_FFN_EVF 1
#endif
// Bulk copy of streamed codes; with QE_FFN_EVF they leave L2 first, so that
// the activations, which every row tile of an entry reads, stay resident.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                         uint32_t bar)
{
#if QE_FFN_EVF
    uint64_t policy;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
#else
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
        : "memory");
#endif
}

// Compact copy of the work entries (expert, start, ntok) in shared memory;
// entries beyond kEntCap are read from global memory.
struct EntTab {
    const int4 *sm;
    const Entry *gl;
    __device__ __forceinline__ int4 get(unsigned ei) const
    {
        if (ei < (unsigned)kEntCap)
            return sm[ei];
        const Entry &e = gl[ei];
        return make_int4(e.expert, e.start, e.ntok, 0);
    }
};

struct Item {
    unsigned ei;      // entry index
    int expert, start, ntok;
    int rt;
    bool shared;
};

// Item `it` of the flat (entry, row tile) order: routed entries first, then
// the shared expert's.  32-bit arithmetic: item counts stay below 2^31.
// (Running the row tiles of an expert's sibling entries back to back, so
// that their second reads hit L2, measured 1-7% slower: the decode kernels
// are bound by the work per record, not by where its bytes come from.)
__device__ __forceinline__ Item decode_item(const FfnArgs &a, const EntTab &tab, unsigned it,
                                            unsigned n_r)
{
    Item r;
    const unsigned tiles_r = a.r.n_rt, tiles_s = a.s.n_rt;
    const unsigned routed = n_r * tiles_r;
    if (it < routed) {
        r.ei = it / tiles_r;
        r.rt = (int)(it - r.ei * tiles_r);
        r.shared = false;
    } else {
        const unsigned j = it - routed, es = j / tiles_s;
        r.ei = n_r + es;
        r.rt = (int)(j - es * tiles_s);
        r.shared = true;
    }
    const int4 e = tab.get(r.ei);
    r.expert = e.x;
    r.start = e.y;
    r.ntok = e.z;
    return r;
}

// A warp's work: the items [first, first + J) of its group, and in each item
// its own K slice of 128-groups [b, b + M) cut into units of up to UG groups
// (routed items first, then shared ones), so the item and groups of the
// warp's u-th unit follow in closed form.
struct Sched {
    unsigned n_r;
    bool solo;                // every warp owns whole items (short K): no K split
    unsigned first, J_r, J;   // items of the group (routed ones first)
    unsigned b_r, M_r, N_r;   // routed items: slice start, slice size, units per item
    unsigned b_s, M_s, N_s;   // shared items: likewise
    unsigned U;               // units of this warp
};

// With at most kSoloGroups groups along K a K split would leave each warp a
// group or two per item and the cross-warp reduction would dominate: then
// every warp takes whole items (contiguous ranges of its own) instead.
constexpr unsigned kSoloGroups = 2 * kWW;

template <int UG, int WG>
__device__ __forceinline__ Sched make_sched(const FfnArgs &a, int wg, int wl)
{
    Sched c;
    c.n_r = (unsigned)a.hdr[0];
    const unsigned n_s = (unsigned)a.hdr[1];
    const unsigned routed = c.n_r * a.r.n_rt, total = routed + n_s * a.s.n_rt;
    c.solo = (unsigned)a.r.n_groups <= kSoloGroups &&
             (n_s == 0 || (unsigned)a.s.n_groups <= kSoloGroups);
    const unsigned long long v = ((unsigned long long)blockIdx.x * WG + wg) * (c.solo ? kWW : 1) +
                                 (c.solo ? wl : 0);
    const unsigned long long V = (unsigned long long)gridDim.x * WG * (c.solo ? kWW : 1);
    c.first = (unsigned)(total * v / V);
    const unsigned last = (unsigned)(total * (v + 1) / V);
    c.J = last - c.first;
    c.J_r = routed > c.first ? min(routed - c.first, c.J) : 0;
    const unsigned G_r = a.r.n_groups, G_s = a.s.n_groups;
    const unsigned ws = c.solo ? 0 : wl, nw = c.solo ? 1 : kWW;
    c.b_r = ws * G_r / nw;
    c.M_r = (ws + 1) * G_r / nw - c.b_r;
    c.N_r = (c.M_r + UG - 1) / UG;
    c.b_s = ws * G_s / nw;
    c.M_s = (ws + 1) * G_s / nw - c.b_s;
    c.N_s = (c.M_s + UG - 1) / UG;
    c.U = c.J_r * c.N_r + (c.J - c.J_r) * c.N_s;
    return c;
}

struct WarpRing {
    uint8_t *stage0;          // kS stages of this warp
    uint64_t *full;           // [kS]
};

// Activation row pointer of a lane for one entry: token g of the entry
// (every slot of an entry names a valid row; the C columns of absent tokens
// are not written).
struct LaneCtx {
    const __half *arow;
    int xo[2];   // gate/up: activation-sum rows of the lane's C columns 2t, 2t+1
};

// Activations of one 128-group for the B operand: 8 k-steps x 4 fp16 =
// 4 x uint4; with ZC also the group sums of the lane's C columns (4-bit:
// xs[0], xs[1] for columns 2t, 2t+1; 2-bit: the partial sums (k % 4 < 2,
// k % 4 >= 2) of column 2t in xs[0], xs[1] and of 2t+1 in xs[2], xs[3]; the
// second register of every k-step, the positions k % 4 >= 2 of the lane's
// contiguous 32-value slice, is scaled by 1/16, exactly).
template <int WB, bool ZC>
__device__ __forceinline__ void load_b(const LaneCtx &lc, int gg, uint4 (&b)[4], float (&xs)[4],
                                       const float *xsum)
{
    if (ZC && WB == 4) {
        xs[0] = __ldg(xsum + lc.xo[0] + gg);
        xs[1] = __ldg(xsum + lc.xo[1] + gg);
    } else if (ZC) {
        const float2 c0 = __ldg(reinterpret_cast<const float2 *>(xsum + lc.xo[0] + 2 * gg));
        const float2 c1 = __ldg(reinterpret_cast<const float2 *>(xsum + lc.xo[1] + 2 * gg));
        xs[0] = c0.x;
        xs[1] = c0.y;
        xs[2] = c1.x;
        xs[3] = c1.y;
    }
    constexpr int CK = 256 / WB;
    constexpr int CPG = kGroup / CK;
#pragma unroll
    for (int v = 0; v < 4; v++) {
        // 4-bit: chunk v/2, uint4 v%2 of the lane's 16-half slice; 2-bit: uint4 v
        const int off = WB == 4 ? (gg * CPG + (v >> 1)) * CK + 8 * (v & 1) : gg * CK + 8 * v;
        b[v] = ld_act(lc.arow + off);
        if (ZC && WB == 2) {
            b[v].y = hmul2_u(b[v].y, 0x2C002C00u);   // x 1/16
            b[v].w = hmul2_u(b[v].w, 0x2C002C00u);
        }
    }
}

// One record (one 128-group of one or two matrices), activations in b.
// The down kernels, whose fragments take a subtraction, run two accumulator
// chains per matrix (even and odd k-steps), which keeps consecutive MMAs
// independent; the gate/up kernels, whose fragments come straight from the
// LOP3s, are faster with one (4-bit: 57.7 against 56.5 us on the 64-expert
// decode bench) -- fewer registers to zero and to add.
template <int WB, bool GU>
__device__ __forceinline__ void group_mma(const uint8_t *rec, const uint4 (&b)[4],
                                          const float (&xs)[4], float (&tot0)[4],
                                          float (&tot1)[4])
{
    // gate/up: zero point by the activation-sum correction; down: fragments
    // made exact q - z (one HSUB2 per register, or frag2_exact)
    constexpr bool ZC = GU;
    using G = Geo<WB, GU>;
    constexpr int CPG = G::cpg;
    const int lane = threadIdx.x & 31, g = lane >> 2;
    const int word = chunk_slot(g, lane & 3) * 16;
    const uint8_t *codes0 = rec;
    const uint8_t *meta0 = rec + G::code;
    const uint8_t *codes1 = meta0 + kMetaBytes;
    const uint8_t *meta1 = codes1 + G::code;
    uint4 q0[CPG], q1[CPG];
#pragma unroll
    for (int cc = 0; cc < CPG; cc++) {
        q0[cc] = *reinterpret_cast<const uint4 *>(codes0 + cc * kChunkBytes + word);
        q1[cc] = *reinterpret_cast<const uint4 *>(codes1 + cc * kChunkBytes + word);
    }
    const GroupMeta k0 = group_meta<WB, ZC>(meta0, g);
    const GroupMeta k1 = group_meta<WB, ZC>(meta1, g);
    constexpr int CH = ZC ? 1 : 2;   // accumulator chains per matrix
    float acc0[CH][4], acc1[CH][4];
#pragma unroll
    for (int c = 0; c < CH; c++)
#pragma unroll
        for (int r = 0; r < 4; r++)
            acc0[c][r] = acc1[c][r] = 0.f;
    const uint32_t *bb = reinterpret_cast<const uint32_t *>(&b[0]);
#pragma unroll
    for (int step = 0; step < 8; step++) {
        const int cc = WB == 4 ? step >> 2 : 0;
        const int wd = WB == 4 ? step & 3 : step >> 1;
        const int hs = WB == 4 ? 0 : step & 1;
        const int ch = CH == 2 ? step & 1 : 0;
        uint32_t af[4];
        if (ZC) {
            frag<WB>((&q0[cc].x)[wd], hs, af);
        } else if (WB == 2) {
            frag2_exact((&q0[cc].x)[wd], hs, k0, af);
        } else {
            frag<WB>((&q0[cc].x)[wd], hs, af);
            sub_zero(af, k0);
        }
        mma16816(acc0[ch], af, bb[2 * step], bb[2 * step + 1]);
        if (ZC) {
            frag<WB>((&q1[cc].x)[wd], hs, af);
        } else if (WB == 2) {
            frag2_exact((&q1[cc].x)[wd], hs, k1, af);
        } else {
            frag<WB>((&q1[cc].x)[wd], hs, af);
            sub_zero(af, k1);
        }
        mma16816(acc1[ch], af, bb[2 * step], bb[2 * step + 1]);
    }
    float a0 = acc0[0][0], a1 = acc0[0][1], a2 = acc0[0][2], a3 = acc0[0][3];
    float c0 = acc1[0][0], c1 = acc1[0][1], c2 = acc1[0][2], c3 = acc1[0][3];
    if (CH == 2) {
        a0 += acc0[CH - 1][0];
        a1 += acc0[CH - 1][1];
        a2 += acc0[CH - 1][2];
        a3 += acc0[CH - 1][3];
        c0 += acc1[CH - 1][0];
        c1 += acc1[CH - 1][1];
        c2 += acc1[CH - 1][2];
        c3 += acc1[CH - 1][3];
    }
    if (ZC && WB == 4) {   // C columns 2t, 2t+1: subtract zf x (activation sum)
        a0 = fmaf(-k0.zf_lo, xs[0], a0);
        a1 = fmaf(-k0.zf_lo, xs[1], a1);
        a2 = fmaf(-k0.zf_hi, xs[0], a2);
        a3 = fmaf(-k0.zf_hi, xs[1], a3);
        c0 = fmaf(-k1.zf_lo, xs[0], c0);
        c1 = fmaf(-k1.zf_lo, xs[1], c1);
        c2 = fmaf(-k1.zf_hi, xs[0], c2);
        c3 = fmaf(-k1.zf_hi, xs[1], c3);
    } else if (ZC) {       // the same per partial sum: column 2t xs[0..1], 2t+1 xs[2..3]
        a0 = fmaf(-k0.zf2_lo, xs[1], fmaf(-k0.zf_lo, xs[0], a0));
        a1 = fmaf(-k0.zf2_lo, xs[3], fmaf(-k0.zf_lo, xs[2], a1));
        a2 = fmaf(-k0.zf2_hi, xs[1], fmaf(-k0.zf_hi, xs[0], a2));
        a3 = fmaf(-k0.zf2_hi, xs[3], fmaf(-k0.zf_hi, xs[2], a3));
        c0 = fmaf(-k1.zf2_lo, xs[1], fmaf(-k1.zf_lo, xs[0], c0));
        c1 = fmaf(-k1.zf2_lo, xs[3], fmaf(-k1.zf_lo, xs[2], c1));
        c2 = fmaf(-k1.zf2_hi, xs[1], fmaf(-k1.zf_hi, xs[0], c2));
        c3 = fmaf(-k1.zf2_hi, xs[3], fmaf(-k1.zf_hi, xs[2], c3));
    }
    tot0[0] = fmaf(k0.s_lo, a0, tot0[0]);
    tot0[1] = fmaf(k0.s_lo, a1, tot0[1]);
    tot0[2] = fmaf(k0.s_hi, a2, tot0[2]);
    tot0[3] = fmaf(k0.s_hi, a3, tot0[3]);
    tot1[0] = fmaf(k1.s_lo, c0, tot1[0]);
    tot1[1] = fmaf(k1.s_lo, c1, tot1[1]);
    tot1[2] = fmaf(k1.s_hi, c2, tot1[2]);
    tot1[3] = fmaf(k1.s_hi, c3, tot1[3]);
}

// Reduction of one item by the last warp to arrive: outputs (r, lane)
// summed over the group's warps in a fixed order.
template <bool GU>
__device__ __forceinline__ void finish_item(const FfnArgs &a, const Item &t, const float *red)
{
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int r = 0; r < 4; r++) {
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int w = 0; w < kWW; w++) {
            s0 += red[((w * 2 + 0) * 4 + r) * 32 + lane];
            s1 += red[((w * 2 + 1) * 4 + r) * 32 + lane];
        }
        const int tn = 2 * (lane & 3) + (r & 1);         // token inside the entry
        const int rr = (lane >> 2) + 8 * (r >> 1);       // row inside a 16-row tile
        if (tn < t.ntok) {
            const long long orow = (long long)(t.start + tn) * a.out_ld;
            if (GU) {   // slots: gate, up of row tile rt
                const float hv = s0 / (1.0f + expf(-s0)) * s1;
                reinterpret_cast<__half *>(a.out)[orow + t.rt * kRowTile + rr] =
                    __float2half_rn(hv);
            } else {    // slots: row tiles 2 rt and 2 rt + 1
                float *y = reinterpret_cast<float *>(a.out) + orow + t.rt * 2 * kRowTile + rr;
                y[0] = s0;
                y[kRowTile] = s1;
            }
        }
    }
}

// Output of an item computed by one warp alone (no reduction).
template <bool GU>
__device__ __forceinline__ void finish_solo(const FfnArgs &a, const Item &t, const float (&tot0)[4],
                                            const float (&tot1)[4])
{
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int r = 0; r < 4; r++) {
        const float s0 = tot0[r], s1 = tot1[r];
        const int tn = 2 * (lane & 3) + (r & 1);         // token inside the entry
        const int rr = (lane >> 2) + 8 * (r >> 1);       // row inside a 16-row tile
        if (tn < t.ntok) {
            const long long orow = (long long)(t.start + tn) * a.out_ld;
            if (GU) {
                const float hv = s0 / (1.0f + expf(-s0)) * s1;
                reinterpret_cast<__half *>(a.out)[orow + t.rt * kRowTile + rr] =
                    __float2half_rn(hv);
            } else {
                float *y = reinterpret_cast<float *>(a.out) + orow + t.rt * 2 * kRowTile + rr;
                y[0] = s0;
                y[kRowTile] = s1;
            }
        }
    }
}

struct GroupCtl {
    float *red;               // [2][kRed]
    int red_floats;           // floats per slot
    unsigned *red_cnt;        // [2] warps that wrote their partials into the slot
    volatile int *red_done;   // [2] 1 + index of the last item reduced from the slot
    volatile int *abort_flag;
};

// Partial sums of item j into slot j&1 (once the item two back has been
// reduced from it); the last warp to arrive reduces the item.  False when the
// wait for the slot gave up.
template <bool GU>
__device__ __forceinline__ bool reduce_item(const FfnArgs &a, const Item &t, unsigned j,
                                            const float (&tot0)[4], const float (&tot1)[4],
                                            const GroupCtl &gc, int wl)
{
    const int lane = threadIdx.x & 31;
    const int slot = j & 1;
    bool ok = true;
    if (lane == 0) {
        const unsigned long long t0 = global_ns();
        while (ld_acquire(&gc.red_done[slot]) < (int)j - 1) {
            if (*gc.abort_flag || global_ns() - t0 > kWaitLimitNs) {
                ok = false;
                break;
            }
        }
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok)
        return false;
    __syncwarp();
    float *red = gc.red + slot * gc.red_floats;
#pragma unroll
    for (int r = 0; r < 4; r++) {
        red[((wl * 2 + 0) * 4 + r) * 32 + lane] = tot0[r];
        red[((wl * 2 + 1) * 4 + r) * 32 + lane] = tot1[r];
    }
    __syncwarp();
    unsigned last = 0;
    if (lane == 0)   // releases this warp's partials, acquires the others' (wraps to 0)
        last = atom_inc_acq_rel(&gc.red_cnt[slot], kWW - 1) == kWW - 1;
    last = __shfl_sync(0xffffffffu, last, 0);
    if (last) {
        __syncwarp();   // lane 0's fence precedes every lane's reads of the slot
        finish_item<GU>(a, t, red);
        __syncwarp();
        if (lane == 0)
            st_release(&gc.red_done[slot], (int)j + 1);
    }
    return true;
}

// Position in the group's contiguous item sequence, advanced one item at a
// time without divisions: routed entries [0, n_r) then shared ones.
struct Cursor {
    unsigned ei;            // entry index
    int rt;                 // 16-row tile
    bool shared;
    int expert, start, ntok;
};

__device__ __forceinline__ void cursor_at(Cursor &cu, const FfnArgs &a, const EntTab &tab,
                                          unsigned it, unsigned n_r)
{
    const Item t = decode_item(a, tab, it, n_r);
    cu.ei = t.ei;
    cu.rt = t.rt;
    cu.shared = t.shared;
    cu.expert = t.expert;
    cu.start = t.start;
    cu.ntok = t.ntok;
}

__device__ __forceinline__ void cursor_next(Cursor &cu, const FfnArgs &a, const EntTab &tab,
                                            unsigned n_r)
{
    if (++cu.rt == (cu.shared ? a.s.n_rt : a.r.n_rt)) {
        cu.rt = 0;
        if (++cu.ei >= n_r)
            cu.shared = true;
        const int4 e = tab.get(cu.ei);
        cu.expert = e.x;
        cu.start = e.y;
        cu.ntok = e.z;
    }
}

// Copy issuer of one warp (state kept by lane 0): the item and unit of the
// next unit to issue, and the first record of that item's slice.
struct Issuer {
    Cursor cu;
    unsigned k;             // unit inside the item
    unsigned N, M;          // units and groups of this warp's slice in the item
    const uint8_t *base;    // record of group b of the item
    long long stride;       // bytes between the item's records of consecutive groups
};

template <int WB, bool GU>
__device__ __forceinline__ void issuer_item(Issuer &is, const FfnArgs &a, const Sched &c)
{
    using G = Geo<WB, GU>;
    const PackedRecs &pr = is.cu.shared ? a.s : a.r;
    const long long e = is.cu.shared ? 0 : is.cu.expert;
    const unsigned b = is.cu.shared ? c.b_s : c.b_r;
    is.N = is.cu.shared ? c.N_s : c.N_r;
    is.M = is.cu.shared ? c.M_s : c.M_r;
    is.k = 0;
    // unit rt's record of group b; its next groups follow pr.upt records apart
    is.base = expert_records(pr, e) + rec_index(0, is.cu.rt, b, pr.n_rt, pr.n_groups, pr.upt) * G::rec;
    is.stride = (long long)pr.upt * G::rec;
}

// Issue the next unit into stage s and advance (lane 0).  The caller issues
// only while units remain, so the cursor never passes the group's last item.
template <int WB, bool GU>
__device__ __forceinline__ void issue_next(Issuer &is, const FfnArgs &a, const EntTab &tab,
                                           const Sched &c, const WarpRing &wr, int s)
{
    using G = Geo<WB, GU>;
    while (is.k == is.N) {   // items where this warp has no groups
        cursor_next(is.cu, a, tab, c.n_r);
        issuer_item<WB, GU>(is, a, c);
    }
    const unsigned ng = min((unsigned)G::ug, is.M - is.k * G::ug);
    const uint32_t fb = smem_addr(&wr.full[s]);
    mbar_expect_tx(fb, ng * G::rec);
    const uint8_t *src = is.base + (long long)is.k * G::ug * is.stride;
    for (unsigned i = 0; i < ng; i++)   // one copy per record: consecutive groups are apart
        bulk_g2s(smem_addr(wr.stage0 + (size_t)s * G::stage + i * G::rec), src + i * is.stride,
                 G::rec, fb);
    ++is.k;
}

template <int WB, bool GU>
__global__ void __launch_bounds__(kFfnThreads, 1) ffn_kernel(FfnArgs a)
{
    using G = Geo<WB, GU>;
    constexpr int CK = 256 / WB;
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wg = warp / kWW, wl = warp % kWW;
    uint8_t *gbase = smem + (size_t)wg * G::group;
    WarpRing wr;
    wr.stage0 = gbase + (size_t)wl * G::ring;
    wr.full = reinterpret_cast<uint64_t *>(smem + (size_t)kWG * G::group) + warp * kS;
    GroupCtl gc;
    gc.red = reinterpret_cast<float *>(gbase + kWW * G::ring);
    gc.red_floats = kRed;
    gc.red_cnt = reinterpret_cast<unsigned *>(gc.red + 2 * kRed);
    gc.red_done = reinterpret_cast<volatile int *>(gc.red_cnt + 2);
    gc.abort_flag = gc.red_done + 2;
    int4 *ent_sm = reinterpret_cast<int4 *>(smem + (size_t)kWG * G::group +
                                            kFfnThreads / 32 * G::warp_ctl);
    const EntTab tab{ent_sm, a.entries};
    pdl_enter();

    const unsigned n_ent = (unsigned)(a.hdr[0] + a.hdr[1]);
    for (unsigned i = threadIdx.x; i < n_ent && i < (unsigned)kEntCap; i += kFfnThreads) {
        const int4 e = *reinterpret_cast<const int4 *>(&a.entries[i]);
        ent_sm[i] = make_int4(e.x, e.y, e.z, 0);
    }
    if (wl == 0 && lane == 0) {
        gc.red_cnt[0] = gc.red_cnt[1] = 0;
        gc.red_done[0] = gc.red_done[1] = 0;
        *gc.abort_flag = 0;
    }
    if (lane == 0) {
        for (int s = 0; s < kS; s++)
            mbar_init(smem_addr(&wr.full[s]), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    const Sched c = make_sched<G::ug, kWG>(a, wg, wl);
    if (c.J == 0)
        return;
    Cursor cu;                       // the item being multiplied
    cursor_at(cu, a, tab, c.first, c.n_r);
    Issuer is;                       // the next unit to copy (lane 0)
    unsigned issued = 0;
    if (lane == 0) {
        is.cu = cu;
        issuer_item<WB, GU>(is, a, c);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        for (; issued + 1 < (unsigned)kS && issued < c.U; issued++)
            issue_next<WB, GU>(is, a, tab, c, wr, issued);
    }
    const int g = lane >> 2, tq = lane & 3;
    unsigned u = 0;
    bool ok = true;
    for (unsigned j = 0; j < c.J && ok; j++) {
        if (j)
            cursor_next(cu, a, tab, c.n_r);
        const Item t{cu.ei, cu.expert, cu.start, cu.ntok, cu.rt, cu.shared};
        LaneCtx lc;
        {
            const long long row = GU ? a.entries[t.ei].tok[g] : t.start + min(g, t.ntok - 1);
            lc.arow = a.act + row * a.act_ld + tq * (CK / 4);
            if (GU) {   // every slot of an entry names a valid token
                lc.xo[0] = a.entries[t.ei].tok[2 * tq] * a.xs_ld;
                lc.xo[1] = a.entries[t.ei].tok[2 * tq + 1] * a.xs_ld;
            }
        }
        const unsigned N = t.shared ? c.N_s : c.N_r;
        const unsigned M = t.shared ? c.M_s : c.M_r;
        const unsigned gb = t.shared ? c.b_s : c.b_r;
        float tot0[4] = {0.f, 0.f, 0.f, 0.f}, tot1[4] = {0.f, 0.f, 0.f, 0.f};
        for (unsigned k = 0; k < N && ok; k++, u++) {
            // refill the stage freed by the previous unit, kS - 1 units ahead
            // (the stage's previous contents were read into registers and
            // consumed before the __syncwarp that ended the previous unit)
            if (lane == 0 && issued < c.U) {
                issue_next<WB, GU>(is, a, tab, c, wr, issued % kS);
                ++issued;
            }
            const int s = u % kS;
            const uint8_t *stage = wr.stage0 + (size_t)s * G::stage;
            const unsigned ng = min((unsigned)G::ug, M - k * G::ug);
            const unsigned g0 = gb + k * G::ug;
            uint4 b[4];
            float xs[4];
            load_b<WB, GU>(lc, g0, b, xs, a.xsum);
            if (!mbar_wait(smem_addr(&wr.full[s]), (u / kS) & 1, gc.abort_flag)) {
                ok = false;
                break;
            }
            for (unsigned i = 0; i < ng; i++) {
                if (i)
                    load_b<WB, GU>(lc, g0 + i, b, xs, a.xsum);
                group_mma<WB, GU>(stage + i * G::rec, b, xs, tot0, tot1);
            }
            __syncwarp();   // every lane has read the stage before it is refilled
        }
        if (!ok)
            break;
        if (c.solo) {
            finish_solo<GU>(a, t, tot0, tot1);
            if (*gc.abort_flag)
                ok = false;
            continue;
        }
        if (!reduce_item<GU>(a, t, j, tot0, tot1, gc, wl) || *gc.abort_flag)
            ok = false;
    }
    if (!ok && lane == 0) {
        *gc.abort_flag = 1;
        atomicOr(a.status, MOE_STATUS_TIMEOUT);
        // copies still in flight into this warp's ring land before it leaves
        // (only possible after an abort: otherwise every issued unit was waited on)
        for (unsigned uu = u; uu < issued; uu++) {
            const unsigned long long t0 = global_ns();
            while (!mbar_try(smem_addr(&wr.full[uu % kS]), (uu / kS) & 1) &&
                   global_ns() - t0 < kWaitLimitNs) {
            }
        }
    }
}

template <int WB, bool GU>
static void set_smem()
{
    cudaFuncSetAttribute(ffn_kernel<WB, GU>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         Geo<WB, GU>::smem);
}

void configure_ffn_kernels()
{
    set_smem<4, true>();
    set_smem<2, true>();
    set_smem<4, false>();
    set_smem<2, false>();
}

int ffn_blocks_per_sm(int wbits)
{
    (void)wbits;
    return 1;
}

template <int WB, bool GU>
static cudaError_t launch_ffn(const FfnArgs &a, int grid, cudaStream_t st)
{
    return launch_pdl(ffn_kernel<WB, GU>, dim3(grid), dim3(kFfnThreads), Geo<WB, GU>::smem, st, a);
}

cudaError_t launch_gateup(const LayerDev &L, const Workspace &ws, const __half *x, int grid,
                          cudaStream_t st)
{
    FfnArgs a{};
    a.r = L.gu;
    a.s = L.has_shared ? L.sh_gu : L.gu;
    a.entries = ws.entries;
    a.hdr = ws.hdr;
    a.status = ws.hdr + 2;
    a.act = x;
    a.act_ld = L.H;
    a.out = ws.h;
    a.out_ld = L.I > L.I_sh ? L.I : L.I_sh;
    a.xsum = ws.xsum;
    a.xs_ld = (L.H / kGroup) * (L.wbits == 2 ? 2 : 1);   // 2-bit: two partial sums per group
    return L.wbits == 4 ? launch_ffn<4, true>(a, grid, st) : launch_ffn<2, true>(a, grid, st);
}

cudaError_t launch_down(const LayerDev &L, const Workspace &ws, int grid, cudaStream_t st)
{
    FfnArgs a{};
    a.r = L.dn;
    a.s = L.has_shared ? L.sh_dn : L.dn;
    a.entries = ws.entries;
    a.hdr = ws.hdr;
    a.status = ws.hdr + 2;
    a.act = ws.h;
    a.act_ld = L.I > L.I_sh ? L.I : L.I_sh;
    a.out = ws.y;
    a.out_ld = L.H;
    return L.wbits == 4 ? launch_ffn<4, false>(a, grid, st) : launch_ffn<2, false>(a, grid, st);
}

}  // namespace qe
