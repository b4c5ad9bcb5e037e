/* mlp_block.c -- a caller of the tensor-parallel MLP block's C ABI written in
 * plain C99, with no Python and no C++ in the process: the forward pass
 * Y = GeLU(X A + b1) B + b2 + residual over t shards and its backward pass
 * ("Megatron-LM: Tensor Model Parallel", Figure 3(a): A split by columns, B
 * by rows; the g operator's sum after the row-parallel GEMM, the f
 * operator's sum of the input gradient), through tp_mlp_forward and
 * tp_mlp_backward on one CUDA stream.
 *
 *   mlp_block T h F t in.bin out.bin
 *
 * in.bin holds the raw bf16 bits of X [T,h], A [h,F], b1 [F], B [F,h],
 * b2 [h], residual [T,h] and dY [T,h], row-major, in that order.  out.bin
 * receives Y [T,h], Z [T,F], H [T,F], dX [T,h], dA [h,F], dB [F,h] as bf16
 * bits, then db1 [F] and db2 [h] as float32.
 *
 * Exit status: 0 on success; 2 bad arguments; 3 a file could not be read or
 * written; 4 a CUDA runtime call failed; 5 the library returned an error
 * (its status text is printed). */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime_api.h>

#include "tpmlp.h"

enum { N_IN = 7, N_OUT = 8 };

static int cuda_ok(cudaError_t e, const char* what) {
    if (e == cudaSuccess) return 1;
    fprintf(stderr, "%s: %s\n", what, cudaGetErrorString(e));
    return 0;
}

static int lib_ok(int status, const char* what) {
    if (status == TPMLP_OK) return 1;
    fprintf(stderr, "%s: %s (status %d, CUDA error %d)\n", what, tp_mlp_status_string(status),
            status, tpmlp_last_cuda_error());
    return 0;
}

int main(int argc, char** argv) {
    if (argc != 7) {
        fprintf(stderr, "usage: %s T h F t in.bin out.bin\n", argv[0]);
        return 2;
    }
    const long long T = atoll(argv[1]), h = atoll(argv[2]), F = atoll(argv[3]);
    const int t = atoi(argv[4]);
    if (T < 1 || h < 1 || F < 1 || t < 1) return 2;

    /* element counts and byte sizes of every tensor, inputs then outputs */
    const long long in_elems[N_IN] = {T * h, h * F, F, F * h, h, T * h, T * h};
    const long long out_elems[N_OUT] = {T * h, T * F, T * F, T * h, h * F, F * h, F, h};
    const size_t out_size[N_OUT] = {2, 2, 2, 2, 2, 2, 4, 4};

    void* dev_in[N_IN] = {0};
    void* dev_out[N_OUT] = {0};
    void* host = NULL;
    void* workspace = NULL;
    void* fwd_workspace = NULL;
    cudaStream_t stream = NULL;
    int rc = 4;
    size_t most = 0;
    for (int i = 0; i < N_IN; ++i)
        if ((size_t)in_elems[i] * 2 > most) most = (size_t)in_elems[i] * 2;
    for (int i = 0; i < N_OUT; ++i)
        if ((size_t)out_elems[i] * out_size[i] > most) most = (size_t)out_elems[i] * out_size[i];
    host = malloc(most);
    if (host == NULL) return 3;

    if (!cuda_ok(cudaStreamCreateWithFlags(&stream, cudaStreamNonBlocking), "stream")) goto done;
    FILE* in = fopen(argv[5], "rb");
    if (in == NULL) {
        rc = 3;
        goto done;
    }
    for (int i = 0; i < N_IN; ++i) {
        const size_t bytes = (size_t)in_elems[i] * 2;
        if (fread(host, 1, bytes, in) != bytes) {
            fclose(in);
            rc = 3;
            goto done;
        }
        if (!cuda_ok(cudaMalloc(&dev_in[i], bytes), "cudaMalloc") ||
            !cuda_ok(cudaMemcpy(dev_in[i], host, bytes, cudaMemcpyHostToDevice), "copy in")) {
            fclose(in);
            goto done;
        }
    }
    fclose(in);
    for (int i = 0; i < N_OUT; ++i)
        if (!cuda_ok(cudaMalloc(&dev_out[i], (size_t)out_elems[i] * out_size[i]), "cudaMalloc"))
            goto done;

    const tpmlp_bf16 *X = dev_in[0], *A = dev_in[1], *b1 = dev_in[2], *B = dev_in[3],
                     *b2 = dev_in[4], *residual = dev_in[5], *dY = dev_in[6];
    tpmlp_bf16 *Y = dev_out[0], *Z = dev_out[1], *H = dev_out[2], *dX = dev_out[3],
               *dA = dev_out[4], *dB = dev_out[5];
    float *db1 = dev_out[6], *db2 = dev_out[7];

    /* the caller owns every buffer, the workspaces included; the forward's
       is optional (it lets the row-parallel GEMM split its reduction) */
    const size_t fwd_ws_bytes = tp_mlp_forward_workspace_bytes((int)T, (int)h, (int)F, t);
    if (fwd_ws_bytes > 0 && !cuda_ok(cudaMalloc(&fwd_workspace, fwd_ws_bytes), "cudaMalloc"))
        goto done;
    const size_t ws_bytes = tp_mlp_backward_workspace_bytes((int)T, (int)h, (int)F, t);
    if (ws_bytes == 0) {
        fprintf(stderr, "tp_mlp_backward_workspace_bytes: shape rejected\n");
        rc = 5;
        goto done;
    }
    if (!cuda_ok(cudaMalloc(&workspace, ws_bytes), "cudaMalloc")) goto done;

    rc = 5;
    if (!lib_ok(tp_mlp_forward(X, A, b1, B, b2, residual, (int)T, (int)h, (int)F, t, Y, Z, H,
                               fwd_workspace, fwd_ws_bytes, stream),
                "tp_mlp_forward"))
        goto done;
    if (!lib_ok(tp_mlp_backward(dY, X, A, B, Z, H, (int)T, (int)h, (int)F, t, dX, dA, dB, db1,
                                db2, workspace, ws_bytes, stream),
                "tp_mlp_backward"))
        goto done;
    rc = 4;
    if (!cuda_ok(cudaStreamSynchronize(stream), "synchronize")) goto done;
    rc = 5;
    if (!lib_ok(tpmlp_device_status(), "device status")) goto done;

    rc = 3;
    FILE* out = fopen(argv[6], "wb");
    if (out == NULL) goto done;
    for (int i = 0; i < N_OUT; ++i) {
        const size_t bytes = (size_t)out_elems[i] * out_size[i];
        if (!cuda_ok(cudaMemcpy(host, dev_out[i], bytes, cudaMemcpyDeviceToHost), "copy out")) {
            fclose(out);
            rc = 4;
            goto done;
        }
        if (fwrite(host, 1, bytes, out) != bytes) {
            fclose(out);
            goto done;
        }
    }
    rc = fclose(out) == 0 ? 0 : 3;

done:
    for (int i = 0; i < N_IN; ++i) cudaFree(dev_in[i]);
    for (int i = 0; i < N_OUT; ++i) cudaFree(dev_out[i]);
    cudaFree(workspace);
    cudaFree(fwd_workspace);
    if (stream != NULL) cudaStreamDestroy(stream);
    free(host);
    return rc;
}
