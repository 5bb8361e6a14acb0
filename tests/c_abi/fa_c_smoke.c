/*
 * The C ABI of include/fa.h used from plain C, with no Python or PyTorch in
 * the process: device buffers from the CUDA runtime, one fa_forward call per
 * case, fa_check_device_error, and a rejected call whose reason is read back
 * through fa_last_error.  Every output row is compared with the CPU oracle
 * (oracle/oracle.c, linked into this test program only).
 *
 * Inputs: a SplitMix64 stream (Steele, Lea and Flood, OOPSLA 2014) mapped to
 * uniform values in [-2, 2), rounded to bf16 (round to nearest even); the
 * oracle reads the same values as float.  Cases: a ragged non-causal problem
 * at d = 64 and a causal one at d = 128 (several key tiles and a ragged tail
 * each), O stored as fp32 so the comparison sees no output rounding.
 *
 * Exit status 0 when every check passes; a message on stderr otherwise.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "fa.h"

int oracle_attention_rows(const float *q, const float *k, const float *v, int64_t B, int64_t H, int64_t N,
                          int64_t d, double scale, int causal, const int64_t *rows, int64_t nrows, double *o,
                          double *lse, double *work);

static uint64_t splitmix64(uint64_t *state)
{
    uint64_t z = (*state += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

/* bf16 bits of x, round to nearest even (finite inputs) */
static uint16_t to_bf16(float x)
{
    uint32_t u;
    memcpy(&u, &x, 4);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

static float from_bf16(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float x;
    memcpy(&x, &u, 4);
    return x;
}

/* n bf16 values (bits) and the same values as float */
static void fill(uint64_t seed, size_t n, uint16_t *bits, float *vals)
{
    uint64_t st = seed;
    for (size_t i = 0; i < n; ++i) {
        const double u = (double)(splitmix64(&st) >> 11) * (1.0 / 9007199254740992.0);
        bits[i] = to_bf16((float)(4.0 * u - 2.0));
        vals[i] = from_bf16(bits[i]);
    }
}

#define CHECK_CUDA(call)                                                                  \
    do {                                                                                  \
        cudaError_t e_ = (call);                                                          \
        if (e_ != cudaSuccess) {                                                          \
            fprintf(stderr, "%s failed: %s\n", #call, cudaGetErrorString(e_));            \
            return 1;                                                                     \
        }                                                                                 \
    } while (0)

static int run_case(int64_t B, int64_t H, int64_t N, int64_t d, int causal, uint64_t seed)
{
    const size_t n = (size_t)(B * H * N * d), rows = (size_t)(B * H * N);
    const double scale = 1.0 / sqrt((double)d);
    uint16_t *hq = malloc(n * 2), *hk = malloc(n * 2), *hv = malloc(n * 2);
    float *fq = malloc(n * 4), *fk = malloc(n * 4), *fv = malloc(n * 4), *ho = malloc(n * 4), *hl = malloc(rows * 4);
    double *ro = malloc(n * 8), *rl = malloc(rows * 8), *work = malloc((size_t)N * 8);
    int64_t *ids = malloc(rows * 8);
    if (!hq || !hk || !hv || !fq || !fk || !fv || !ho || !hl || !ro || !rl || !work || !ids) {
        fprintf(stderr, "host allocation failed\n");
        return 1;
    }
    fill(seed, n, hq, fq);
    fill(seed + 1, n, hk, fk);
    fill(seed + 2, n, hv, fv);

    void *dq, *dk, *dv, *dout;
    float *dlse;
    CHECK_CUDA(cudaMalloc(&dq, n * 2));
    CHECK_CUDA(cudaMalloc(&dk, n * 2));
    CHECK_CUDA(cudaMalloc(&dv, n * 2));
    CHECK_CUDA(cudaMalloc(&dout, n * 4));
    CHECK_CUDA(cudaMalloc((void **)&dlse, rows * 4));
    CHECK_CUDA(cudaMemcpy(dq, hq, n * 2, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dk, hk, n * 2, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dv, hv, n * 2, cudaMemcpyHostToDevice));

    char msg[256];
    fa_status st = fa_forward(dq, dk, dv, dout, dlse, B, H, N, d, (float)scale, causal, FA_BF16, FA_FP32, NULL);
    if (st != FA_OK) {
        fa_last_error(msg, sizeof(msg));
        fprintf(stderr, "fa_forward: status %d: %s\n", (int)st, msg);
        return 1;
    }
    st = fa_check_device_error(NULL);
    if (st != FA_OK) {
        fa_last_error(msg, sizeof(msg));
        fprintf(stderr, "fa_check_device_error: status %d: %s\n", (int)st, msg);
        return 1;
    }
    CHECK_CUDA(cudaMemcpy(ho, dout, n * 4, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(hl, dlse, rows * 4, cudaMemcpyDeviceToHost));

    for (size_t r = 0; r < rows; ++r) ids[r] = (int64_t)r;
    if (oracle_attention_rows(fq, fk, fv, B, H, N, d, scale, causal, ids, (int64_t)rows, ro, rl, work) != 0) {
        fprintf(stderr, "oracle failed\n");
        return 1;
    }
    double max_o = 0.0, sum_o = 0.0, max_l = 0.0;
    for (size_t i = 0; i < n; ++i) {
        const double e = fabs((double)ho[i] - ro[i]);
        max_o = e > max_o ? e : max_o;
        sum_o += e;
    }
    for (size_t r = 0; r < rows; ++r) {
        const double e = fabs((double)hl[r] - rl[r]);
        max_l = e > max_l ? e : max_l;
    }
    const double mean_o = sum_o / (double)n;
    printf("B=%lld H=%lld N=%lld d=%lld causal=%d: O max %.3e mean %.3e, LSE max %.3e\n", (long long)B,
           (long long)H, (long long)N, (long long)d, causal, max_o, mean_o, max_l);
    /* bf16 inputs, fp32 O: the stated bounds O max 1e-2, mean 1e-3, LSE 1e-3 */
    const int ok = max_o <= 1e-2 && mean_o <= 1e-3 && max_l <= 1e-3;

    cudaFree(dq);
    cudaFree(dk);
    cudaFree(dv);
    cudaFree(dout);
    cudaFree(dlse);
    free(hq), free(hk), free(hv), free(fq), free(fk), free(fv), free(ho), free(hl), free(ro), free(rl), free(work),
        free(ids);
    if (!ok) fprintf(stderr, "parity bound exceeded\n");
    return ok ? 0 : 1;
}

int main(void)
{
    printf("%s\n", fa_version());
    if (run_case(1, 2, 300, 64, 0, 7001) != 0) return 1;
    if (run_case(2, 1, 333, 128, 1, 7101) != 0) return 1;

    /* a rejected call: N = 0 never reaches the GPU and says why */
    const fa_status st = fa_forward(NULL, NULL, NULL, NULL, NULL, 1, 1, 0, 64, 0.125f, 0, FA_BF16, FA_BF16, NULL);
    char msg[256];
    const fa_status last = fa_last_error(msg, sizeof(msg));
    if (st != FA_ERR_INVALID_ARG || last != st || msg[0] == '\0') {
        fprintf(stderr, "invalid call: status %d (recorded %d), message \"%s\"\n", (int)st, (int)last, msg);
        return 1;
    }
    /* a cut-down copy still ends in a NUL */
    char small[8];
    fa_last_error(small, sizeof(small));
    if (strlen(small) != sizeof(small) - 1) {
        fprintf(stderr, "truncated message has length %zu\n", strlen(small));
        return 1;
    }
    printf("rejected as expected: %s\n", msg);
    printf("ok\n");
    return 0;
}
