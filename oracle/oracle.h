/*
 * CPU oracle for the quantised MoE layer forward.  TEST INFRASTRUCTURE ONLY:
 * only the tests, the smoke check and the benchmark's CPU-baseline leg use
 * it.  Independent of the CUDA path (no shared code or headers).
 *
 * All buffers are host memory, row-major, caller-owned.  fp16 values are
 * passed as their uint16 bit patterns.  Every function returns 0 on success,
 * -1 on an invalid argument and -2 when host memory runs out.
 */
#ifndef QEFFN_ORACLE_H
#define QEFFN_ORACLE_H
#include <stdint.h>

typedef struct {
    int hidden, inter, n_experts, top_k, group, wbits, has_shared, shared_inter;
    /* stacked routed experts: [E][rows][K*wbits/8], [E][rows][K/group] x2 */
    const uint8_t *codes[3];
    const uint16_t *scales[3];
    const uint8_t *zeros[3];
    const uint16_t *router_w; /* fp16 [E][H] */
    const float *router_bias; /* fp32 [E] or NULL */
    const uint8_t *sh_codes[3];
    const uint16_t *sh_scales[3];
    const uint8_t *sh_zeros[3];
    const uint16_t *sh_gate_w; /* fp16 [H] */
} oracle_layer_t;

double oracle_half_to_double(uint16_t h);
uint16_t oracle_double_to_half(double v);
int oracle_unpack_codes(const uint8_t *codes, int64_t rows, int K, int wbits, uint8_t *q);
int oracle_dequant(const uint8_t *codes, const uint16_t *scales, const uint8_t *zeros,
                   int64_t rows, int K, int wbits, int group, double *w);
int oracle_router_logits(const uint16_t *x, int n, int H, const uint16_t *router_w,
                         const float *bias, int E, float *logits);
int oracle_topk(const float *logits, int n, int E, int k, int32_t *idx, float *w32, double *w64);
int oracle_group(const int32_t *idx, int n, int k, int E, int32_t *counts, int32_t *offsets,
                 int32_t *perm);
/* e = -1 selects the shared expert; y [T][H] in fp64 */
int oracle_expert_ffn(const oracle_layer_t *L, int e, const uint16_t *x, int T, double *y);
/* Routing for all n tokens; FFN and combine only for the n_sel tokens listed
 * in `tokens` (NULL with n_sel == n: all tokens).  out64/out16 are
 * [n_sel][H].  Any output pointer may be NULL. */
int oracle_forward(const oracle_layer_t *L, const uint16_t *x, int n, const int32_t *tokens,
                   int n_sel, float *logits, int32_t *idx, float *w32, int32_t *counts,
                   int32_t *offsets, int32_t *perm, double *out64, uint16_t *out16);
/* Two-pass RMSNorm r [n][H] x gain g [H] -> fp16 xn [n][H]: the fp64
 * definition rounded once to fp16. */
int oracle_rmsnorm(const uint16_t *r, const uint16_t *g, float eps, int n, int H, uint16_t *xn);
/* OpenMP threads of the parallel loops (n <= 0: unchanged), and their count. */
void oracle_set_num_threads(int n);
int oracle_num_threads(void);
#endif
