/*
 * Host cost of one rowops_softmax call, measured from C: the C ABI's own
 * per-call work (argument checks, kernel choice, launch) without any Python
 * or ctypes layer. Workload: fp32 1024 x 768 softmax (6.3 MB, L2-resident,
 * launch-bound), the size at which host cost decides the call rate.
 *
 * Prints one JSON line:
 *   host_us_per_call    wall time of the calls alone (each batch of calls is
 *                       issued, timed, and only then synchronised)
 *   events_us_per_call  CUDA events around back-to-back calls: what a caller
 *                       sees per call when the host issues as fast as it can
 *   graph_us_per_call   the same kernels captured once in a CUDA graph and
 *                       replayed: the device's own time per launch
 * Exit status 0 on success, 1 on a CUDA or rowops error.
 */
#define _POSIX_C_SOURCE 199309L
#include <stdio.h>
#include <stdlib.h>
#include <time.h>

#include <cuda_runtime.h>

#include "rowops.h"

#define CK(call)                                                                      \
    do {                                                                              \
        cudaError_t e_ = (call);                                                      \
        if (e_ != cudaSuccess) {                                                      \
            fprintf(stderr, "%s failed: %s\n", #call, cudaGetErrorString(e_));        \
            return 1;                                                                 \
        }                                                                             \
    } while (0)

static double now_us(void) {
    struct timespec ts;
    clock_gettime(CLOCK_MONOTONIC, &ts);
    return ts.tv_sec * 1e6 + ts.tv_nsec / 1e3;
}

int main(void) {
    const int64_t M = 1024, N = 768;
    const int batch = 256, batches = 40, graph_calls = 256;
    float *x = NULL, *y = NULL;
    CK(cudaMalloc((void**)&x, (size_t)(M * N) * sizeof(float)));
    CK(cudaMalloc((void**)&y, (size_t)(M * N) * sizeof(float)));
    CK(cudaMemset(x, 0, (size_t)(M * N) * sizeof(float)));
    cudaStream_t s;
    CK(cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking));
    for (int i = 0; i < 200; ++i)
        if (rowops_softmax(x, y, M, N, N, ROWOPS_F32, s) != ROWOPS_OK) return 1;
    CK(cudaStreamSynchronize(s));

    /* host cost: issue a batch, time only the issuing, then drain */
    double host = 0.0;
    for (int b = 0; b < batches; ++b) {
        const double t0 = now_us();
        for (int i = 0; i < batch; ++i)
            if (rowops_softmax(x, y, M, N, N, ROWOPS_F32, s) != ROWOPS_OK) return 1;
        host += now_us() - t0;
        CK(cudaStreamSynchronize(s));
    }

    /* events around back-to-back calls */
    cudaEvent_t e0, e1;
    CK(cudaEventCreate(&e0));
    CK(cudaEventCreate(&e1));
    const int calls = batch * 8;
    CK(cudaEventRecord(e0, s));
    for (int i = 0; i < calls; ++i)
        if (rowops_softmax(x, y, M, N, N, ROWOPS_F32, s) != ROWOPS_OK) return 1;
    CK(cudaEventRecord(e1, s));
    CK(cudaEventSynchronize(e1));
    float ev_ms = 0.f;
    CK(cudaEventElapsedTime(&ev_ms, e0, e1));

    /* the same calls in a CUDA graph */
    cudaGraph_t g;
    cudaGraphExec_t ge;
    CK(cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal));
    for (int i = 0; i < graph_calls; ++i)
        if (rowops_softmax(x, y, M, N, N, ROWOPS_F32, s) != ROWOPS_OK) return 1;
    CK(cudaStreamEndCapture(s, &g));
    CK(cudaGraphInstantiate(&ge, g, 0));
    CK(cudaGraphLaunch(ge, s));
    CK(cudaStreamSynchronize(s));
    CK(cudaEventRecord(e0, s));
    for (int r = 0; r < 4; ++r) CK(cudaGraphLaunch(ge, s));
    CK(cudaEventRecord(e1, s));
    CK(cudaEventSynchronize(e1));
    float gr_ms = 0.f;
    CK(cudaEventElapsedTime(&gr_ms, e0, e1));

    printf("{\"workload\": \"softmax fp32 1024x768\", \"host_us_per_call\": %.3f, \"events_us_per_call\": %.3f, "
           "\"graph_us_per_call\": %.3f}\n",
           host / (double)(batch * batches), ev_ms * 1000.0 / calls, gr_ms * 1000.0 / (4 * graph_calls));
    CK(cudaGraphExecDestroy(ge));
    CK(cudaGraphDestroy(g));
    CK(cudaFree(x));
    CK(cudaFree(y));
    return 0;
}
