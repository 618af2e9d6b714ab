// Expert FFN: weight repacking and the fused dequant x GEMV/GEMM kernels.
//
// Group-wise INT4 (or 2-bit) weights W = (q - zero) * scale, one fp16 scale
// and zero point per 128 consecutive K elements ("Strata" article, section
// 2.2; "为什么12G显存笔记本能跑MoE-16B" section 4.2: the codes are unpacked
// inside the kernel and never written back as fp16), gate/up projection with
// SwiGLU h = silu(g) * u, then the down projection ("Flash-MoE" article,
// section 3: dequant matvec, fused SwiGLU).  Decode is bound by the bytes of
// the touched experts' weights ("Strata" section 1.1), so the kernels stream
// each expert's codes exactly once per call with 128-bit coalesced loads and
// keep every token routed to that expert in the same pass ("Strata" section
// 2.3 and 3.4: one weight read serves every token that shares the expert).
//
// Packed layout (built by repack): for every (expert, 16-row tile, K chunk)
// 512 contiguous bytes, one 16-byte word per lane of a warp.  A chunk spans
// 64 K (4-bit) or 128 K (2-bit).  Lane (g = lane/4, t = lane%4) owns rows g
// and g+8 of the tile and the K range [t*CK/4, (t+1)*CK/4) of the chunk; the
// nibbles (2-bit fields) inside each 32-bit word are ordered so that the
// magic-number conversion below yields, with one LOP3 and one HFMA2 per two
// weights, exactly the A fragment of an m16n8k16 tensor-core MMA.  The K
// order inside a lane's slice is the natural one, so the activation operand
// is one contiguous 16-byte load per 8 K and token.
//
// Arithmetic: q - z is exact in fp16; x (or h) is fp16; the MMA accumulates
// the exact products in fp32 over one 128-group; the group sum is multiplied
// by its fp32-widened scale and added to an fp32 total.  The tensor core is
// used as the multiply-add engine because the per-weight ALU budget at HBM
// speed (about 2.5 issue slots per weight) does not leave room for scalar
// convert + FMA; the kernel stays bound by the weight stream.
#include <cuda_fp16.h>

#include "internal.cuh"

namespace qe {

// ------------------------------------------------------------ repacking

template <int WB>
__global__ void repack_codes_kernel(const uint8_t *__restrict__ canon, int n_exp, int rows,
                                    int K, uint4 *__restrict__ out)
{
    const int CK = 256 / WB;
    const int n_rt = rows / kRowTile, n_c = K / CK;
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
        out[gid] = make_uint4(wd[0], wd[1], wd[2], wd[3]);
    }
}

__global__ void repack_meta_kernel(const uint16_t *__restrict__ scales,
                                   const uint8_t *__restrict__ zeros, int n_exp, int rows, int K,
                                   uint8_t *__restrict__ out)
{
    const int G = K / kGroup, n_rt = rows / kRowTile;
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
        uint8_t *dst = out + ((e * n_rt + rt) * G + grp) * kMetaBytes;
        reinterpret_cast<uint16_t *>(dst)[r] = scales[src];
        dst[32 + r] = zeros[src];
    }
}

cudaError_t launch_repack(const uint8_t *codes, const uint16_t *scales, const uint8_t *zeros,
                          int n_exp, int rows, int K, int wbits, uint4 *out_codes,
                          uint8_t *out_meta, cudaStream_t st)
{
    const int threads = 256, blocks = 4096;
    if (wbits == 4)
        repack_codes_kernel<4><<<blocks, threads, 0, st>>>(codes, n_exp, rows, K, out_codes);
    else
        repack_codes_kernel<2><<<blocks, threads, 0, st>>>(codes, n_exp, rows, K, out_codes);
    repack_meta_kernel<<<blocks, threads, 0, st>>>(scales, zeros, n_exp, rows, K, out_meta);
    return cudaGetLastError();
}

// ------------------------------------------------------------ device helpers

__device__ __forceinline__ uint4 ld_stream(const uint4 *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

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

__device__ __forceinline__ uint32_t hfma2_u(uint32_t a, uint32_t b, uint32_t c)
{
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ uint32_t hadd2_u(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("add.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
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

__device__ __forceinline__ uint32_t half2_bits(float v)
{
    const __half h = __float2half_rn(v);
    const uint32_t u = __half_as_ushort(h);
    return u | (u << 16);
}

// Per (matrix, group) constants of one lane: fp32 scales of rows g and g+8 and
// the fp16x2 offsets that turn magic-number fields into q - z.
struct GroupConst {
    float s_lo, s_hi;   // rows g, g+8
    uint32_t c[4];      // offsets for the 4 field positions of a word
};

template <int WB>
__device__ __forceinline__ GroupConst load_group(const uint8_t *meta, int g)
{
    GroupConst k;
    const __half *sc = reinterpret_cast<const __half *>(meta);
    k.s_lo = __half2float(sc[g]);
    k.s_hi = __half2float(sc[g + 8]);
    const int z_lo = meta[32 + g], z_hi = meta[32 + g + 8];
    if (WB == 4) {
        // field scale 1 (rows g) and 16 (rows g+8, multiplied back by 1/16)
        k.c[0] = half2_bits(-(1024.0f + z_lo));
        k.c[1] = half2_bits(-(64.0f + z_hi));
        k.c[2] = k.c[0];
        k.c[3] = k.c[1];
    } else {
        // field scales 1, 4, 16, 64 -> rows g, g+8, g, g+8
        k.c[0] = half2_bits(-(1024.0f + z_lo));
        k.c[1] = half2_bits(-(256.0f + z_hi));
        k.c[2] = half2_bits(-(64.0f + z_lo));
        k.c[3] = half2_bits(-(16.0f + z_hi));
    }
    return k;
}

// A fragment (rows g / g+8, 4 K each) of one k-step from one 32-bit word
// (4-bit) or half a word (2-bit: step 0 = low byte pair, 1 = high).
__device__ __forceinline__ void frag4(uint32_t w, const GroupConst &k, uint32_t (&a)[4])
{
    const uint32_t w8 = w >> 8;
    a[0] = hadd2_u(lop_magic(w, 0x000F000Fu), k.c[0]);
    a[1] = hfma2_u(lop_magic(w, 0x00F000F0u), 0x2C002C00u, k.c[1]);   // x 1/16
    a[2] = hadd2_u(lop_magic(w8, 0x000F000Fu), k.c[0]);
    a[3] = hfma2_u(lop_magic(w8, 0x00F000F0u), 0x2C002C00u, k.c[1]);
}

__device__ __forceinline__ void frag2(uint32_t w, const GroupConst &k, uint32_t (&a)[4])
{
    a[0] = hadd2_u(lop_magic(w, 0x00030003u), k.c[0]);
    a[1] = hfma2_u(lop_magic(w, 0x000C000Cu), 0x34003400u, k.c[1]);   // x 1/4
    a[2] = hfma2_u(lop_magic(w, 0x00300030u), 0x2C002C00u, k.c[2]);   // x 1/16
    a[3] = hfma2_u(lop_magic(w, 0x00C000C0u), 0x24002400u, k.c[3]);   // x 1/64
}

// ------------------------------------------------------------ FFN kernels

struct FfnArgs {
    PackedMat m0, m1;      // routed matrices (gate, up) or (down, -)
    PackedMat s0, s1;      // shared-expert matrices
    const Entry *entries;
    const int *hdr;
    const int32_t *tok_of_pos;
    const __half *act;     // gate/up: x [n][H] by token; down: h [P+n][ld] by position
    long long act_ld;
    void *out;             // gate/up: h (fp16); down: y (fp32)
    long long out_ld;
    int E;
    int tiles_r, tiles_s;
};

constexpr int kFfnThreads = 256;
constexpr int kFfnWarps = kFfnThreads / 32;

// One expert's slice of a packed matrix: its row tile `rt` base pointers.
struct MatView {
    const uint4 *codes;    // + chunk * 32 + lane
    const uint8_t *meta;   // + group * kMetaBytes
    int n_c;
};

__device__ __forceinline__ MatView mat_view(const PackedMat &m, long long e, int rt)
{
    MatView v;
    v.codes = m.codes + e * m.expert_codes + (long long)rt * m.n_chunks * 32;
    v.meta = m.meta + e * m.expert_meta + (long long)rt * m.n_groups * kMetaBytes;
    v.n_c = m.n_chunks;
    return v;
}

template <int WB, bool GU, int NT>
__device__ __forceinline__ void ffn_item(const FfnArgs &a, const MatView V0, const MatView V1,
                                         int rt, const Entry &en, float *red)
{
    constexpr int CK = 256 / WB;     // K per chunk
    constexpr int CPG = kGroup / CK; // chunks per group
    constexpr int BV = CK / 32;      // uint4 activation loads per chunk and token
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int n_c = V0.n_c;
    const int c_begin = warp * n_c / kFfnWarps, c_end = (warp + 1) * n_c / kFfnWarps;

    float tot0[NT][4], tot1[NT][4];
#pragma unroll
    for (int i = 0; i < NT; i++)
#pragma unroll
        for (int r = 0; r < 4; r++)
            tot0[i][r] = tot1[i][r] = 0.f;

    if (c_begin < c_end) {
        const uint4 *cp0 = V0.codes + lane;
        const uint4 *cp1 = GU ? V1.codes + lane : cp0;
        const uint8_t *mp0 = V0.meta;
        const uint8_t *mp1 = GU ? V1.meta : mp0;

        const __half *arow[NT];
        bool aval[NT];
#pragma unroll
        for (int i = 0; i < NT; i++) {
            const int tn = g + 8 * i;
            aval[i] = tn < en.ntok;
            const int pos = en.start + (aval[i] ? tn : 0);
            const long long row = GU ? a.tok_of_pos[pos] : pos;
            arow[i] = a.act + row * a.act_ld + t * (CK / 4);
        }

        float acc0[NT][4], acc1[NT][4];
        GroupConst k0{}, k1{};
        uint4 cur0 = ld_stream(cp0 + (long long)c_begin * 32);
        uint4 cur1 = GU ? ld_stream(cp1 + (long long)c_begin * 32) : cur0;
        uint4 nxt0 = cur0, nxt1 = cur1;
        if (c_begin + 1 < c_end) {
            nxt0 = ld_stream(cp0 + (long long)(c_begin + 1) * 32);
            if (GU)
                nxt1 = ld_stream(cp1 + (long long)(c_begin + 1) * 32);
        }
        for (int c = c_begin; c < c_end; c++) {
            const uint4 q0 = cur0, q1 = cur1;
            cur0 = nxt0;
            cur1 = nxt1;
            if (c + 2 < c_end) {
                nxt0 = ld_stream(cp0 + (long long)(c + 2) * 32);
                if (GU)
                    nxt1 = ld_stream(cp1 + (long long)(c + 2) * 32);
            }
            uint4 b[NT][BV];
#pragma unroll
            for (int i = 0; i < NT; i++)
#pragma unroll
                for (int v = 0; v < BV; v++)
                    b[i][v] = aval[i] ? ld_act(arow[i] + (long long)c * CK + 8 * v)
                                      : make_uint4(0, 0, 0, 0);
            if (c == c_begin || c % CPG == 0) {
                const int grp = c / CPG;
                k0 = load_group<WB>(mp0 + grp * kMetaBytes, g);
                if (GU)
                    k1 = load_group<WB>(mp1 + grp * kMetaBytes, g);
#pragma unroll
                for (int i = 0; i < NT; i++)
#pragma unroll
                    for (int r = 0; r < 4; r++)
                        acc0[i][r] = acc1[i][r] = 0.f;
            }
            const uint32_t w0[4] = {q0.x, q0.y, q0.z, q0.w};
            const uint32_t w1[4] = {q1.x, q1.y, q1.z, q1.w};
#pragma unroll
            for (int wd = 0; wd < 4; wd++) {
#pragma unroll
                for (int hs = 0; hs < (WB == 4 ? 1 : 2); hs++) {
                    const int step = WB == 4 ? wd : 2 * wd + hs;   // k-step inside the chunk
                    uint32_t af[4];
                    if (WB == 4)
                        frag4(w0[wd], k0, af);
                    else
                        frag2(hs ? (w0[wd] >> 8) : w0[wd], k0, af);
#pragma unroll
                    for (int i = 0; i < NT; i++) {
                        const uint32_t *bb = reinterpret_cast<const uint32_t *>(&b[i][0]);
                        mma16816(acc0[i], af, bb[2 * step], bb[2 * step + 1]);
                    }
                    if (GU) {
                        if (WB == 4)
                            frag4(w1[wd], k1, af);
                        else
                            frag2(hs ? (w1[wd] >> 8) : w1[wd], k1, af);
#pragma unroll
                        for (int i = 0; i < NT; i++) {
                            const uint32_t *bb = reinterpret_cast<const uint32_t *>(&b[i][0]);
                            mma16816(acc1[i], af, bb[2 * step], bb[2 * step + 1]);
                        }
                    }
                }
            }
            if (c + 1 == c_end || (c + 1) % CPG == 0) {
#pragma unroll
                for (int i = 0; i < NT; i++) {
                    tot0[i][0] = fmaf(acc0[i][0], k0.s_lo, tot0[i][0]);
                    tot0[i][1] = fmaf(acc0[i][1], k0.s_lo, tot0[i][1]);
                    tot0[i][2] = fmaf(acc0[i][2], k0.s_hi, tot0[i][2]);
                    tot0[i][3] = fmaf(acc0[i][3], k0.s_hi, tot0[i][3]);
                    if (GU) {
                        tot1[i][0] = fmaf(acc1[i][0], k1.s_lo, tot1[i][0]);
                        tot1[i][1] = fmaf(acc1[i][1], k1.s_lo, tot1[i][1]);
                        tot1[i][2] = fmaf(acc1[i][2], k1.s_hi, tot1[i][2]);
                        tot1[i][3] = fmaf(acc1[i][3], k1.s_hi, tot1[i][3]);
                    }
                }
            }
        }
    }

    // deterministic cross-warp reduction: red[warp][mat][i][r][lane]
#pragma unroll
    for (int i = 0; i < NT; i++)
#pragma unroll
        for (int r = 0; r < 4; r++) {
            red[(((warp * 2 + 0) * NT + i) * 4 + r) * 32 + lane] = tot0[i][r];
            if (GU)
                red[(((warp * 2 + 1) * NT + i) * 4 + r) * 32 + lane] = tot1[i][r];
        }
    __syncthreads();
    if (warp == 0) {
#pragma unroll
        for (int i = 0; i < NT; i++)
#pragma unroll
            for (int r = 0; r < 4; r++) {
                float s0 = 0.f, s1 = 0.f;
                for (int w = 0; w < kFfnWarps; w++) {
                    s0 += red[(((w * 2 + 0) * NT + i) * 4 + r) * 32 + lane];
                    if (GU)
                        s1 += red[(((w * 2 + 1) * NT + i) * 4 + r) * 32 + lane];
                }
                const int tn = 2 * t + (r & 1) + 8 * i;    // token inside the entry
                const int row = rt * kRowTile + g + 8 * (r >> 1);
                if (tn < en.ntok) {
                    const long long orow = (long long)(en.start + tn) * a.out_ld;
                    if (GU) {
                        const float hv = s0 / (1.0f + expf(-s0)) * s1;
                        reinterpret_cast<__half *>(a.out)[orow + row] = __float2half_rn(hv);
                    } else {
                        reinterpret_cast<float *>(a.out)[orow + row] = s0;
                    }
                }
            }
    }
    __syncthreads();
}

template <int WB, bool GU>
__global__ void __launch_bounds__(kFfnThreads, 2) ffn_kernel(FfnArgs a)
{
    __shared__ float red[kFfnWarps * 2 * 2 * 4 * 32];
    const long long n_r = a.hdr[0], n_s = a.hdr[1];
    const long long total = n_r * a.tiles_r + n_s * a.tiles_s;
    for (long long it = blockIdx.x; it < total; it += gridDim.x) {
        long long ei;
        int rt;
        bool shared;
        if (it < n_r * a.tiles_r) {
            ei = it / a.tiles_r;
            rt = (int)(it % a.tiles_r);
            shared = false;
        } else {
            const long long j = it - n_r * a.tiles_r;
            ei = n_r + j / a.tiles_s;
            rt = (int)(j % a.tiles_s);
            shared = true;
        }
        const Entry en = a.entries[ei];
        const MatView V0 = shared ? mat_view(a.s0, 0, rt) : mat_view(a.m0, en.expert, rt);
        const MatView V1 = !GU ? V0 : shared ? mat_view(a.s1, 0, rt) : mat_view(a.m1, en.expert, rt);
        if (en.ntok <= 8)
            ffn_item<WB, GU, 1>(a, V0, V1, rt, en, red);
        else
            ffn_item<WB, GU, 2>(a, V0, V1, rt, en, red);
    }
}

template <int WB, bool GU>
static int blocks_per_sm_for()
{
    int nb = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, ffn_kernel<WB, GU>, kFfnThreads, 0);
    return nb;
}

int ffn_blocks_per_sm(int wbits)
{
    int a = wbits == 4 ? blocks_per_sm_for<4, true>() : blocks_per_sm_for<2, true>();
    int b = wbits == 4 ? blocks_per_sm_for<4, false>() : blocks_per_sm_for<2, false>();
    return a < b ? a : b;
}

cudaError_t launch_gateup(const LayerDev &L, const Workspace &ws, const __half *x, int n, int grid,
                          cudaStream_t st)
{
    FfnArgs a{};
    a.m0 = L.mat[0];
    a.m1 = L.mat[1];
    if (L.has_shared) {
        a.s0 = L.sh[0];
        a.s1 = L.sh[1];
    } else {
        a.s0 = L.mat[0];
        a.s1 = L.mat[1];
    }
    a.entries = ws.entries;
    a.hdr = ws.hdr;
    a.tok_of_pos = ws.tok_of_pos;
    a.act = x;
    a.act_ld = L.H;
    a.out = ws.h;
    a.out_ld = L.I > L.I_sh ? L.I : L.I_sh;
    a.E = L.E;
    a.tiles_r = L.I / kRowTile;
    a.tiles_s = L.has_shared ? L.I_sh / kRowTile : 1;
    if (L.wbits == 4)
        ffn_kernel<4, true><<<grid, kFfnThreads, 0, st>>>(a);
    else
        ffn_kernel<2, true><<<grid, kFfnThreads, 0, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_down(const LayerDev &L, const Workspace &ws, int n, int grid, cudaStream_t st)
{
    FfnArgs a{};
    a.m0 = L.mat[2];
    a.m1 = L.mat[2];
    a.s0 = L.has_shared ? L.sh[2] : L.mat[2];
    a.s1 = a.s0;
    a.entries = ws.entries;
    a.hdr = ws.hdr;
    a.tok_of_pos = ws.tok_of_pos;
    a.act = ws.h;
    a.act_ld = L.I > L.I_sh ? L.I : L.I_sh;
    a.out = ws.y;
    a.out_ld = L.H;
    a.E = L.E;
    a.tiles_r = L.H / kRowTile;
    a.tiles_s = L.H / kRowTile;
    if (L.wbits == 4)
        ffn_kernel<4, false><<<grid, kFfnThreads, 0, st>>>(a);
    else
        ffn_kernel<2, false><<<grid, kFfnThreads, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace qe
