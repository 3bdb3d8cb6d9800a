/*
 * fp64 CPU oracle for the per-token multi-LoRA delta.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path links, loads or calls
 * this file; only the tests, the smoke check and the benchmark's CPU-baseline
 * leg do. It shares no code, header or constant with the CUDA library.
 *
 * What it computes, for every listed token t and one injected linear layer:
 *
 *     s = token_slot_idx[t]
 *     s == -1 (base model only), s out of range, or slot s empty (rank 0):
 *         y_out[t][i] = y_in[t][i]
 *     otherwise, with r = rank[s] (the adapter's own rank, "r" in the PEFT
 *     adapter_config.json shown on the "vLLM LoRA Resolver 插件详解" page,
 *     section 3.2, with use_rslora false):
 *         v[k]        = sum_j A[s][k][j] * x[t][j]           k < r
 *         y_out[t][i] = y_in[t][i] + (alpha[s] / r) * sum_k B[s][i][k] * v[k]
 *
 * A is [S][R][d_in] and B is [S][d_out][R] (ranks zero-padded to R =
 * max_lora_rank, the slot table of the "Multi-LoRA 适配器缓存生产实战" page,
 * section 核心原理, parameter table). Everything is in double precision, with
 * no rounding of the intermediate v and no rounding of the output. Inputs are
 * read as the exact values the device sees (bf16 bit patterns decoded, or
 * fp32).
 *
 * The loop bound over k is r_s by default. With loop_padded = 1 the loop runs
 * over all R padded ranks (the appended zeros); the tests use that to pin the
 * zero-padding invariance.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_F32 = 0, ORACLE_BF16 = 1 };

/* Read element i of an array of the given element type as a double. */
static double elem(const void *base, int dtype, size_t i)
{
    if (dtype == ORACLE_F32)
        return (double)((const float *)base)[i];
    uint32_t bits = (uint32_t)((const uint16_t *)base)[i] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

int oracle_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Thread count for the calls that follow (timing runs only; results do not
 * depend on it: each token's sums run in one thread in a fixed order). */
void oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/*
 * y_out is [n_list][d_out], one row per listed token (tokens[n] indexes x,
 * y_in and token_slot_idx). Returns 0, or -1 on bad arguments.
 */
int oracle_lora_apply(int n_list, const int64_t *tokens,
                      int d_in, int d_out, int S, int R, int dtype,
                      const void *x, const void *y_in,
                      const void *A_pool, const void *B_pool,
                      const int32_t *rank, const double *alpha,
                      const int32_t *token_slot_idx, int loop_padded,
                      double *y_out)
{
    if (n_list < 0 || d_in <= 0 || d_out <= 0 || S <= 0 || R <= 0)
        return -1;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 4) reduction(| : bad)
    for (int n = 0; n < n_list; n++) {
        int64_t t = tokens[n];
        double *out = y_out + (size_t)n * d_out;
        for (int i = 0; i < d_out; i++)
            out[i] = elem(y_in, dtype, (size_t)t * d_out + i);

        int s = token_slot_idx[t];
        if (s < 0 || s >= S || rank[s] <= 0)
            continue;
        int r = rank[s];
        if (r > R) {
            bad = 1;
            continue;
        }
        int kmax = loop_padded ? R : r;
        double scale = alpha[s] / (double)r;

        double *v = (double *)malloc(sizeof(double) * (size_t)kmax);
        if (!v) {
            bad = 1;
            continue;
        }
        /* shrink: v = A_s . x_t */
        for (int k = 0; k < kmax; k++) {
            double acc = 0.0;
            size_t arow = ((size_t)s * R + k) * (size_t)d_in;
            for (int j = 0; j < d_in; j++)
                acc += elem(A_pool, dtype, arow + j) * elem(x, dtype, (size_t)t * d_in + j);
            v[k] = acc;
        }
        /* expand: y_t += scale * B_s . v */
        for (int i = 0; i < d_out; i++) {
            double acc = 0.0;
            size_t brow = ((size_t)s * d_out + i) * (size_t)R;
            for (int k = 0; k < kmax; k++)
                acc += elem(B_pool, dtype, brow + k) * v[k];
            out[i] += scale * acc;
        }
        free(v);
    }
    return bad ? -1 : 0;
}
