/* A C program that uses the library only through include/rar.h and the CUDA
 * runtime: the worked example of "Ring All-Reduce, in depth" ("Tracing four
 * GPUs": rank r holds (r + 1) x [1, 10, 100, 1000]; every rank ends with
 * [10, 100, 1000, 10000] and sends six elements), on each engine.  Exits 0
 * when every check passes. */
#include <stdio.h>
#include <string.h>

#include <cuda_runtime.h>

#include "rar.h"

#define CHECK(cond, ...)                                  \
    do {                                                  \
        if (!(cond)) {                                    \
            fprintf(stderr, "FAILED: " __VA_ARGS__);      \
            fprintf(stderr, "\n");                        \
            return 1;                                     \
        }                                                 \
    } while (0)

static int run_engine(int engine) {
    const int p = 4;
    const size_t n = 4;
    float host[4][4];
    void *dev[4];
    for (int r = 0; r < p; r++) {
        const float base[4] = {1.0f, 10.0f, 100.0f, 1000.0f};
        for (size_t i = 0; i < n; i++) host[r][i] = (float)(r + 1) * base[i];
        CHECK(cudaMalloc(&dev[r], n * sizeof(float)) == cudaSuccess, "cudaMalloc");
        CHECK(cudaMemcpy(dev[r], host[r], n * sizeof(float), cudaMemcpyHostToDevice) == cudaSuccess, "copy in");
    }
    rar_options opt;
    memset(&opt, 0, sizeof(opt));
    opt.engine = engine;
    rar_handle h = NULL;
    int rc = rar_init(&h, 0, &opt);
    CHECK(rc == RAR_OK, "rar_init: %d %s", rc, rar_last_error(NULL));
    rc = rar_allreduce(h, dev, p, n, RAR_FLOAT32, RAR_SUM, NULL);
    CHECK(rc == RAR_OK, "rar_allreduce: %d %s", rc, rar_last_error(h));
    CHECK(rar_status(h) == RAR_OK, "rar_status: %s", rar_last_error(h));
    unsigned long long sends[4];
    CHECK(rar_send_counts(h, sends, p) == RAR_OK, "rar_send_counts");
    const float expect[4] = {10.0f, 100.0f, 1000.0f, 10000.0f};
    for (int r = 0; r < p; r++) {
        float got[4];
        CHECK(cudaMemcpy(got, dev[r], n * sizeof(float), cudaMemcpyDeviceToHost) == cudaSuccess, "copy out");
        for (size_t i = 0; i < n; i++)
            CHECK(got[i] == expect[i], "engine %d rank %d element %zu: %g", engine, r, i, (double)got[i]);
        if (engine == RAR_ENGINE_RING) CHECK(sends[r] == 6, "engine %d rank %d sent %llu", engine, r, sends[r]);
    }
    /* argument errors come back as codes */
    CHECK(rar_allreduce(h, dev, 0, n, RAR_FLOAT32, RAR_SUM, NULL) == RAR_EINVAL, "p = 0 accepted");
    CHECK(rar_allreduce(h, dev, p, n, RAR_INT32, RAR_AVG, NULL) == RAR_EUNSUPPORTED, "int32 avg accepted");
    CHECK(rar_destroy(h) == RAR_OK, "rar_destroy");
    for (int r = 0; r < p; r++) cudaFree(dev[r]);
    return 0;
}

int main(void) {
    const int engines[] = {RAR_ENGINE_FUSED, RAR_ENGINE_RING, RAR_ENGINE_RING_BIDIR, RAR_ENGINE_FUSED_TREE,
                           RAR_ENGINE_TREE};
    CHECK(rar_version() == RAR_VERSION, "version");
    for (unsigned k = 0; k < sizeof(engines) / sizeof(engines[0]); k++)
        if (run_engine(engines[k])) return 1;
    printf("c-abi roundtrip ok\n");
    return 0;
}
