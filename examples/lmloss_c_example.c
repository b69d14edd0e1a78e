/*
 * Using the lmloss C ABI from C, with no Python: one loss and gradient call on
 * a batch read from files.
 *
 *   lmloss_c_example T V logits.f32 targets.i64 grad_out.f32 [host]
 *
 * logits.f32 holds T*V float32 values (row-major), targets.i64 T int64 targets
 * (-100 ignores a row).  The gradient of the token-mean loss is written to
 * grad_out.f32 (T*V float32), and the five losses (total, cross-entropy,
 * z-loss, KL, policy) are printed on one line.  The z-loss weight is 1e-4.
 * With "host" the logits stay in host memory (registered as pinned) and
 * lmloss_forward_backward_host copies them itself, in row chunks under the
 * chunks' kernels; the results are the same bits.
 *
 * Build (from the repository root, after the library is built):
 *   cc -std=c11 -Iinclude -I/usr/local/cuda/include examples/lmloss_c_example.c \
 *      -Llm_head_vocab_gb300/_build -llmloss -L/usr/local/cuda/lib64 -lcudart \
 *      -Wl,-rpath,$PWD/lm_head_vocab_gb300/_build -o lmloss_c_example
 */
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "lmloss.h"

static int read_file(const char* path, void* buf, size_t bytes)
{
    FILE* f = fopen(path, "rb");
    if (!f) return -1;
    size_t n = fread(buf, 1, bytes, f);
    fclose(f);
    return n == bytes ? 0 : -1;
}

static int write_file(const char* path, const void* buf, size_t bytes)
{
    FILE* f = fopen(path, "wb");
    if (!f) return -1;
    size_t n = fwrite(buf, 1, bytes, f);
    fclose(f);
    return n == bytes ? 0 : -1;
}

#define CHECK_CUDA(x)                                                             \
    do {                                                                          \
        cudaError_t e_ = (x);                                                     \
        if (e_ != cudaSuccess) {                                                  \
            fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_));             \
            return 1;                                                             \
        }                                                                         \
    } while (0)

#define CHECK_LMLOSS(x)                                                           \
    do {                                                                          \
        lmloss_status s_ = (x);                                                   \
        if (s_ != LMLOSS_OK) {                                                    \
            fprintf(stderr, "%s: %s\n", #x, lmloss_status_string(s_));           \
            return 1;                                                             \
        }                                                                         \
    } while (0)

int main(int argc, char** argv)
{
    if (argc != 6 && !(argc == 7 && strcmp(argv[6], "host") == 0)) {
        fprintf(stderr, "usage: %s T V logits.f32 targets.i64 grad_out.f32 [host]\n", argv[0]);
        return 2;
    }
    const int from_host = argc == 7;
    const int64_t T = atoll(argv[1]), V = atoll(argv[2]);
    if (T < 1 || V < 1) {
        fprintf(stderr, "T and V must be positive\n");
        return 2;
    }
    const size_t n = (size_t)T * (size_t)V;
    float* x = (float*)malloc(n * sizeof(float));
    float* g = (float*)malloc(n * sizeof(float));
    int64_t* t = (int64_t*)malloc((size_t)T * sizeof(int64_t));
    if (!x || !g || !t) return 1;
    if (read_file(argv[3], x, n * sizeof(float)) || read_file(argv[4], t, (size_t)T * sizeof(int64_t))) {
        fprintf(stderr, "cannot read the inputs\n");
        return 1;
    }

    float *d_x, *d_g, *d_loss;
    int64_t* d_t;
    CHECK_CUDA(cudaMalloc((void**)&d_x, n * sizeof(float)));
    CHECK_CUDA(cudaMalloc((void**)&d_g, n * sizeof(float)));
    CHECK_CUDA(cudaMalloc((void**)&d_t, (size_t)T * sizeof(int64_t)));
    CHECK_CUDA(cudaMalloc((void**)&d_loss, 5 * sizeof(float)));
    if (from_host)
        CHECK_CUDA(cudaHostRegister(x, n * sizeof(float), cudaHostRegisterDefault));
    else
        CHECK_CUDA(cudaMemcpy(d_x, x, n * sizeof(float), cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(d_t, t, (size_t)T * sizeof(int64_t), cudaMemcpyHostToDevice));

    lmloss_handle h = NULL;
    CHECK_LMLOSS(lmloss_create(&h, 0, T, 0));

    lmloss_args a;
    memset(&a, 0, sizeof a);
    a.logits = d_x;
    a.T = T;
    a.V = V;
    a.ld = V;
    a.dtype = LMLOSS_FP32;
    a.reduction = LMLOSS_REDUCE_TOKEN_MEAN;
    a.targets = d_t;
    a.ce_weight = 1.0f;
    a.z_alpha = 1e-4f;
    a.temperature = 1.0f;
    a.denominator = 1.0;
    a.grad_out = d_g;
    a.loss_out = d_loss;
    CHECK_LMLOSS(lmloss_check_args(&a));
    if (from_host)   /* d_x receives the logits from x, chunk by chunk */
        CHECK_LMLOSS(lmloss_forward_backward_host(h, &a, x, NULL, 0, 0));
    else
        CHECK_LMLOSS(lmloss_forward_backward(h, &a, 0));   /* the default stream */
    CHECK_CUDA(cudaStreamSynchronize(0));
    CHECK_LMLOSS(lmloss_get_device_error(h));

    float loss[5];
    CHECK_CUDA(cudaMemcpy(loss, d_loss, sizeof loss, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(g, d_g, n * sizeof(float), cudaMemcpyDeviceToHost));
    if (write_file(argv[5], g, n * sizeof(float))) {
        fprintf(stderr, "cannot write %s\n", argv[5]);
        return 1;
    }
    printf("%.9g %.9g %.9g %.9g %.9g\n", loss[0], loss[1], loss[2], loss[3], loss[4]);

    CHECK_LMLOSS(lmloss_destroy(h));
    if (from_host) CHECK_CUDA(cudaHostUnregister(x));
    cudaFree(d_x);
    cudaFree(d_g);
    cudaFree(d_t);
    cudaFree(d_loss);
    free(x);
    free(g);
    free(t);
    return 0;
}
