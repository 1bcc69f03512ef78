/*
 * A C consumer of liblce_gb300.so through include/lce.h alone: plain C11 and the
 * CUDA runtime, no C++ and no Python. It reads the inputs from files, runs the
 * fused forward + backward (lce_fwd_bwd) on a stream of its own, checks the
 * device-side status, and writes the outputs back to files:
 *
 *     lce_c_client N D V chunk DIR
 *
 * DIR holds H.bin (N*D bf16 bit patterns), W.bin (V*D bf16) and y.bin (N int64);
 * the client writes loss.bin (1 fp32), lse.bin (N fp32), dH.bin (N*D bf16) and
 * dW.bin (V*D fp32) into it. Exit status 0 on success, non-zero with a message on
 * stderr otherwise.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "lce.h"

static void *read_file(const char *dir, const char *name, size_t bytes) {
    char path[4096];
    snprintf(path, sizeof(path), "%s/%s", dir, name);
    FILE *f = fopen(path, "rb");
    if (!f) return NULL;
    void *buf = malloc(bytes ? bytes : 1);
    if (buf && fread(buf, 1, bytes, f) != bytes) {
        free(buf);
        buf = NULL;
    }
    fclose(f);
    return buf;
}

static int write_file(const char *dir, const char *name, const void *buf, size_t bytes) {
    char path[4096];
    snprintf(path, sizeof(path), "%s/%s", dir, name);
    FILE *f = fopen(path, "wb");
    if (!f) return 0;
    const int ok = fwrite(buf, 1, bytes, f) == bytes;
    fclose(f);
    return ok;
}

#define CHECK_CUDA(x)                                                               \
    do {                                                                            \
        cudaError_t e_ = (x);                                                       \
        if (e_ != cudaSuccess) {                                                    \
            fprintf(stderr, "%s failed: %s\n", #x, cudaGetErrorString(e_));         \
            return 2;                                                               \
        }                                                                           \
    } while (0)

#define CHECK_LCE(x)                                                                \
    do {                                                                            \
        lce_status s_ = (x);                                                        \
        if (s_ != LCE_OK) {                                                         \
            fprintf(stderr, "%s failed: %s\n", #x, lce_status_string(s_));          \
            return 3;                                                               \
        }                                                                           \
    } while (0)

int main(int argc, char **argv) {
    if (argc != 6) {
        fprintf(stderr, "usage: %s N D V chunk DIR\n", argv[0]);
        return 1;
    }
    const int64_t N = atoll(argv[1]), D = atoll(argv[2]), V = atoll(argv[3]);
    const int64_t chunk = atoll(argv[4]);
    const char *dir = argv[5];
    if (N <= 0 || D <= 0 || V <= 0 || chunk <= 0) {
        fprintf(stderr, "sizes must be positive\n");
        return 1;
    }
    const size_t h_bytes = (size_t)N * D * 2, w_bytes = (size_t)V * D * 2;
    const size_t y_bytes = (size_t)N * 8, dw_bytes = (size_t)V * D * 4;
    void *H_h = read_file(dir, "H.bin", h_bytes);
    void *W_h = read_file(dir, "W.bin", w_bytes);
    void *y_h = read_file(dir, "y.bin", y_bytes);
    void *dH_h = malloc(h_bytes), *dW_h = malloc(dw_bytes);
    float *lse_h = (float *)malloc((size_t)N * 4);
    float loss_h = 0.f;
    if (!H_h || !W_h || !y_h || !dH_h || !dW_h || !lse_h) {
        fprintf(stderr, "reading the inputs from %s failed\n", dir);
        return 1;
    }

    size_t ws_bytes = 0;
    CHECK_LCE(lce_workspace_size(N, D, V, chunk, &ws_bytes));
    cudaStream_t stream;
    CHECK_CUDA(cudaStreamCreateWithFlags(&stream, cudaStreamNonBlocking));
    void *H, *W, *y, *dH, *ws;
    float *loss, *lse, *dW;
    CHECK_CUDA(cudaMalloc(&H, h_bytes));
    CHECK_CUDA(cudaMalloc(&W, w_bytes));
    CHECK_CUDA(cudaMalloc(&y, y_bytes));
    CHECK_CUDA(cudaMalloc(&dH, h_bytes));
    CHECK_CUDA(cudaMalloc((void **)&dW, dw_bytes));
    CHECK_CUDA(cudaMalloc((void **)&loss, 16));
    CHECK_CUDA(cudaMalloc((void **)&lse, (size_t)N * 4));
    CHECK_CUDA(cudaMalloc(&ws, ws_bytes));
    CHECK_CUDA(cudaMemcpyAsync(H, H_h, h_bytes, cudaMemcpyHostToDevice, stream));
    CHECK_CUDA(cudaMemcpyAsync(W, W_h, w_bytes, cudaMemcpyHostToDevice, stream));
    CHECK_CUDA(cudaMemcpyAsync(y, y_h, y_bytes, cudaMemcpyHostToDevice, stream));

    /* dloss = NULL: an upstream gradient of 1 */
    CHECK_LCE(lce_fwd_bwd(H, W, (const int64_t *)y, NULL, N, D, V, -100, chunk, loss, lse, dH, dW,
                          ws, ws_bytes, (lce_stream_t)stream));
    CHECK_LCE(lce_read_status(ws, (lce_stream_t)stream));

    CHECK_CUDA(cudaMemcpyAsync(&loss_h, loss, 4, cudaMemcpyDeviceToHost, stream));
    CHECK_CUDA(cudaMemcpyAsync(lse_h, lse, (size_t)N * 4, cudaMemcpyDeviceToHost, stream));
    CHECK_CUDA(cudaMemcpyAsync(dH_h, dH, h_bytes, cudaMemcpyDeviceToHost, stream));
    CHECK_CUDA(cudaMemcpyAsync(dW_h, dW, dw_bytes, cudaMemcpyDeviceToHost, stream));
    CHECK_CUDA(cudaStreamSynchronize(stream));
    if (!write_file(dir, "loss.bin", &loss_h, 4) || !write_file(dir, "lse.bin", lse_h, (size_t)N * 4) ||
        !write_file(dir, "dH.bin", dH_h, h_bytes) || !write_file(dir, "dW.bin", dW_h, dw_bytes)) {
        fprintf(stderr, "writing the outputs to %s failed\n", dir);
        return 1;
    }
    printf("lce_c_client: library version %d, loss %.6f, %d launches\n", lce_version(), loss_h,
           lce_last_launch_count());
    cudaFree(H); cudaFree(W); cudaFree(y); cudaFree(dH); cudaFree(dW);
    cudaFree(loss); cudaFree(lse); cudaFree(ws);
    cudaStreamDestroy(stream);
    free(H_h); free(W_h); free(y_h); free(dH_h); free(dW_h); free(lse_h);
    return 0;
}
