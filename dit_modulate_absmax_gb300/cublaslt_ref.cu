// cublaslt_ref.cu -- reference timing of cuBLASLt's block-scaled NVFP4 GEMM on
// operands prepared by this library (a measurement tool, not part of the
// library: nothing in libh3fp4.so calls cuBLASLt).
//
//   cublaslt_ref DIR M N K REPS ALPHA [OUT]
//
// DIR holds aq.bin (activation QDATA [ceil128(M), K/2]), asf.bin (its scales
// in the 128x4-atom layout), bq.bin (weight QDATA [N, K/2]) and bsf.bin (its
// scales), as written by compare_cublaslt.py.  Computes C[M, N] (row-major
// bf16) = ALPHA * A B^T with cuBLASLt (VEC16_UE4M3 block scales; cuBLAS's
// column-major "A" is the weight, its "B" the activation), runs it twice
// untimed and REPS times between CUDA events, and prints
//   TIMED <wall start> <wall end> <ms per call>
// (wall clock in seconds, to bin sampled GPU clocks).  With OUT, the last
// output is written there.
#include <cublasLt.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <ctime>
#include <vector>

#define CHECK(x)                                                                          \
    do {                                                                                  \
        const int e_ = static_cast<int>(x);                                               \
        if (e_ != 0) {                                                                    \
            std::fprintf(stderr, "%s failed with %d (line %d)\n", #x, e_, __LINE__);      \
            std::exit(1);                                                                 \
        }                                                                                 \
    } while (0)

static double wall_s()
{
    timespec t;
    clock_gettime(CLOCK_REALTIME, &t);
    return t.tv_sec + 1e-9 * t.tv_nsec;
}

static void *load(const char *dir, const char *name, size_t bytes)
{
    char path[1024];
    std::snprintf(path, sizeof path, "%s/%s", dir, name);
    FILE *f = std::fopen(path, "rb");
    if (!f) {
        std::fprintf(stderr, "cannot open %s\n", path);
        std::exit(1);
    }
    std::vector<uint8_t> h(bytes, 0);
    const size_t got = std::fread(h.data(), 1, bytes, f);
    std::fclose(f);
    if (got != bytes) {
        std::fprintf(stderr, "%s: %zu of %zu bytes\n", path, got, bytes);
        std::exit(1);
    }
    void *d = nullptr;
    CHECK(cudaMalloc(&d, bytes));
    CHECK(cudaMemcpy(d, h.data(), bytes, cudaMemcpyHostToDevice));
    return d;
}

int main(int argc, char **argv)
{
    if (argc < 7) {
        std::fprintf(stderr, "usage: %s DIR M N K REPS ALPHA [OUT]\n", argv[0]);
        return 2;
    }
    const char *dir = argv[1];
    const int M = std::atoi(argv[2]), N = std::atoi(argv[3]), K = std::atoi(argv[4]), reps = std::atoi(argv[5]);
    const float alpha_h = static_cast<float>(std::atof(argv[6])), beta_h = 0.f;
    const size_t m128 = (static_cast<size_t>(M) + 127) / 128 * 128;
    void *A = load(dir, "aq.bin", m128 * K / 2), *SA = load(dir, "asf.bin", m128 * K / 16);
    void *B = load(dir, "bq.bin", static_cast<size_t>(N) * K / 2), *SB = load(dir, "bsf.bin", static_cast<size_t>(N) * K / 16);
    void *C = nullptr, *ws = nullptr;
    float *alpha = nullptr, *beta = nullptr;
    const size_t ws_bytes = 64u << 20;
    CHECK(cudaMalloc(&C, static_cast<size_t>(M) * N * 2));
    CHECK(cudaMalloc(&ws, ws_bytes));
    CHECK(cudaMalloc(&alpha, 4));
    CHECK(cudaMalloc(&beta, 4));
    CHECK(cudaMemcpy(alpha, &alpha_h, 4, cudaMemcpyHostToDevice));
    CHECK(cudaMemcpy(beta, &beta_h, 4, cudaMemcpyHostToDevice));

    cublasLtHandle_t lt;
    CHECK(cublasLtCreate(&lt));
    cublasLtMatmulDesc_t op;
    CHECK(cublasLtMatmulDescCreate(&op, CUBLAS_COMPUTE_32F, CUDA_R_32F));
    const cublasOperation_t ta = CUBLAS_OP_T, tb = CUBLAS_OP_N;
    CHECK(cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_TRANSA, &ta, sizeof ta));
    CHECK(cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_TRANSB, &tb, sizeof tb));
    const cublasLtMatmulMatrixScale_t vec16 = CUBLASLT_MATMUL_MATRIX_SCALE_VEC16_UE4M3;
    CHECK(cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_A_SCALE_MODE, &vec16, sizeof vec16));
    CHECK(cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_B_SCALE_MODE, &vec16, sizeof vec16));
    CHECK(cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_A_SCALE_POINTER, &SB, sizeof SB));
    CHECK(cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_B_SCALE_POINTER, &SA, sizeof SA));
    const cublasLtPointerMode_t pm = CUBLASLT_POINTER_MODE_DEVICE;
    CHECK(cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_POINTER_MODE, &pm, sizeof pm));
    cublasLtMatrixLayout_t la, lb, lc;
    CHECK(cublasLtMatrixLayoutCreate(&la, CUDA_R_4F_E2M1, K, N, K));
    CHECK(cublasLtMatrixLayoutCreate(&lb, CUDA_R_4F_E2M1, K, M, K));
    CHECK(cublasLtMatrixLayoutCreate(&lc, CUDA_R_16BF, N, M, N));
    cublasLtMatmulPreference_t pref;
    CHECK(cublasLtMatmulPreferenceCreate(&pref));
    CHECK(cublasLtMatmulPreferenceSetAttribute(pref, CUBLASLT_MATMUL_PREF_MAX_WORKSPACE_BYTES, &ws_bytes,
                                               sizeof ws_bytes));
    cublasLtMatmulHeuristicResult_t res;
    int nres = 0;
    CHECK(cublasLtMatmulAlgoGetHeuristic(lt, op, la, lb, lc, lc, pref, 1, &res, &nres));
    if (nres < 1) {
        std::fprintf(stderr, "no cuBLASLt algorithm for M=%d N=%d K=%d\n", M, N, K);
        return 1;
    }
    auto call = [&] {
        CHECK(cublasLtMatmul(lt, op, alpha, B, la, A, lb, beta, C, lc, C, lc, &res.algo, ws, ws_bytes, 0));
    };
    call();
    call();
    cudaEvent_t e0, e1;
    CHECK(cudaEventCreate(&e0));
    CHECK(cudaEventCreate(&e1));
    CHECK(cudaDeviceSynchronize());
    const double w0 = wall_s();
    CHECK(cudaEventRecord(e0));
    for (int i = 0; i < reps; ++i)
        call();
    CHECK(cudaEventRecord(e1));
    CHECK(cudaEventSynchronize(e1));
    const double w1 = wall_s();
    float ms = 0.f;
    CHECK(cudaEventElapsedTime(&ms, e0, e1));
    std::printf("TIMED %.3f %.3f %.5f\n", w0, w1, ms / reps);
    if (argc > 7) {
        std::vector<uint8_t> h(static_cast<size_t>(M) * N * 2);
        CHECK(cudaMemcpy(h.data(), C, h.size(), cudaMemcpyDeviceToHost));
        FILE *f = std::fopen(argv[7], "wb");
        if (!f || std::fwrite(h.data(), 1, h.size(), f) != h.size()) {
            std::fprintf(stderr, "cannot write %s\n", argv[7]);
            return 1;
        }
        std::fclose(f);
    }
    return 0;
}
