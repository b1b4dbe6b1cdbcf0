/*
 * A plain C99 caller of libswiglu: it includes only swiglu.h and the CUDA
 * runtime's C API, allocates device memory itself and runs the forward, the
 * out-of-place backward and the in-place backward through the C ABI.
 *
 *   c_caller DTYPE ROWS N IN_FILE OUT_FILE
 *
 * IN_FILE holds x [ROWS, 2N] then dy [ROWS, N], raw, in the element type
 * (DTYPE 0 = fp32, 1 = bf16).  OUT_FILE receives y [ROWS, N], dx [ROWS, 2N]
 * and the in-place dx [ROWS, 2N], then y and dx again as computed from
 * page-locked host buffers by swiglu_gateup_fwd_bwd_host (its own device
 * staging buffer and three streams), raw.  Exit status 0 on success;
 * otherwise the failing call and its status string go to stderr.
 */
#include <cuda_runtime_api.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "swiglu.h"

static int check_cuda(cudaError_t e, const char *what) {
    if (e != cudaSuccess) {
        fprintf(stderr, "%s: %s\n", what, cudaGetErrorString(e));
        return 1;
    }
    return 0;
}

static int check(swiglu_status_t st, const char *what) {
    if (st != SWIGLU_OK) {
        fprintf(stderr, "%s: %s (CUDA error %d)\n", what, swiglu_status_string(st),
                swiglu_last_cuda_error());
        return 1;
    }
    return 0;
}

int main(int argc, char **argv) {
    if (argc != 6) {
        fprintf(stderr, "usage: %s DTYPE ROWS N IN_FILE OUT_FILE\n", argv[0]);
        return 2;
    }
    const swiglu_dtype_t dtype = (swiglu_dtype_t)atoi(argv[1]);
    const int64_t rows = atoll(argv[2]), n = atoll(argv[3]);
    const size_t eb = dtype == SWIGLU_F32 ? 4 : 2;
    const size_t bx = (size_t)rows * 2 * n * eb, by = (size_t)rows * n * eb;
    unsigned char *host = malloc(bx + by), *out = malloc(by + 2 * bx);
    void *x = NULL, *dy = NULL, *y = NULL, *dx = NULL;
    FILE *f = fopen(argv[4], "rb");
    if (!host || !out || !f || fread(host, 1, bx + by, f) != bx + by) {
        fprintf(stderr, "cannot read %s\n", argv[4]);
        return 2;
    }
    fclose(f);
    if (check_cuda(cudaMalloc(&x, bx), "cudaMalloc") || check_cuda(cudaMalloc(&dy, by), "cudaMalloc") ||
        check_cuda(cudaMalloc(&y, by), "cudaMalloc") || check_cuda(cudaMalloc(&dx, bx), "cudaMalloc"))
        return 1;
    if (check_cuda(cudaMemcpy(x, host, bx, cudaMemcpyHostToDevice), "copy x") ||
        check_cuda(cudaMemcpy(dy, host + bx, by, cudaMemcpyHostToDevice), "copy dy"))
        return 1;
    /* contiguous rows: row strides 2n (x, dx) and n (y, dy); NULL stream */
    if (check(swiglu_gateup_fwd(x, y, rows, n, 2 * n, n, dtype, NULL), "swiglu_gateup_fwd") ||
        check(swiglu_gateup_bwd(dy, x, dx, rows, n, n, 2 * n, 2 * n, dtype, 0, NULL),
              "swiglu_gateup_bwd"))
        return 1;
    if (check_cuda(cudaMemcpy(out, y, by, cudaMemcpyDeviceToHost), "copy y") ||
        check_cuda(cudaMemcpy(out + by, dx, bx, cudaMemcpyDeviceToHost), "copy dx"))
        return 1;
    /* in place: the gradient over x, dx = NULL and dx_row_stride = 0 */
    if (check(swiglu_gateup_bwd(dy, x, NULL, rows, n, n, 2 * n, 0, dtype, 1, NULL),
              "swiglu_gateup_bwd in place") ||
        check_cuda(cudaMemcpy(out + by + bx, x, bx, cudaMemcpyDeviceToHost), "copy x"))
        return 1;
    /* end to end from host memory: chunks of about a third of the rows,
     * two staging slots, three streams */
    const int64_t chunk = rows / 3 + 1;
    const int depth = 2;
    size_t staging_bytes = 0;
    void *hx = NULL, *hdy = NULL, *hy = NULL, *hdx = NULL, *staging = NULL;
    cudaStream_t s[3];
    if (check(swiglu_gateup_fwd_bwd_host_staging_size(chunk, n, dtype, depth, &staging_bytes),
              "swiglu_gateup_fwd_bwd_host_staging_size") ||
        check_cuda(cudaMalloc(&staging, staging_bytes), "cudaMalloc staging") ||
        check_cuda(cudaMallocHost(&hx, bx), "cudaMallocHost") ||
        check_cuda(cudaMallocHost(&hdy, by), "cudaMallocHost") ||
        check_cuda(cudaMallocHost(&hy, by), "cudaMallocHost") ||
        check_cuda(cudaMallocHost(&hdx, bx), "cudaMallocHost"))
        return 1;
    for (int i = 0; i < 3; ++i)
        if (check_cuda(cudaStreamCreate(&s[i]), "cudaStreamCreate")) return 1;
    memcpy(hx, host, bx);
    memcpy(hdy, host + bx, by);
    if (check(swiglu_gateup_fwd_bwd_host(hx, hdy, hy, hdx, rows, n, dtype, staging, staging_bytes,
                                         chunk, depth, s[0], s[1], s[2]),
              "swiglu_gateup_fwd_bwd_host"))
        return 1;
    f = fopen(argv[5], "wb");
    if (!f || fwrite(out, 1, by + 2 * bx, f) != by + 2 * bx || fwrite(hy, 1, by, f) != by ||
        fwrite(hdx, 1, bx, f) != bx) {
        fprintf(stderr, "cannot write %s\n", argv[5]);
        return 2;
    }
    fclose(f);
    for (int i = 0; i < 3; ++i) cudaStreamDestroy(s[i]);
    cudaFreeHost(hx);
    cudaFreeHost(hdy);
    cudaFreeHost(hy);
    cudaFreeHost(hdx);
    cudaFree(staging);
    cudaFree(x);
    cudaFree(dy);
    cudaFree(y);
    cudaFree(dx);
    free(host);
    free(out);
    printf("ok: abi version %d\n", swiglu_abi_version());
    return 0;
}
