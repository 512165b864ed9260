// cublaslt_gemm.cu -- the vendor library's block-scaled GEMMs timed on the
// shapes of the quantized linear layer, as a reference point for the
// library's own kernels (bench.py --vs-cublaslt builds and runs it).
//
// D (M x N, fp32, row-major) = A (M x K) B (N x K)^T with A and B NVFP4
// (E2M1 codes, one UE4M3 scale per 16 elements, cuBLASLt's VEC16_UE4M3
// scale mode) or FP8 E4M3.  cuBLASLt is column-major, so the call computes
// D^T = B A^T: its "A" is our B (K x N, op T) and its "B" our A (K x M, op N).
// Operands hold constant codes (1.0) and unit scales; the timing does not
// depend on the values.  Every heuristic candidate (up to 8) is timed over
// `reps` back-to-back launches on the same buffers (L2-warm); the best is
// printed as one JSON line.
//
// usage: cublaslt_gemm nvfp4|fp8 M N K [reps]
#include <cublasLt.h>
#include <cuda_runtime.h>

#include <cstdio>
#include <cstdlib>
#include <cstring>

#define CHECK(x)                                                                      \
  do {                                                                                \
    const int e_ = (int)(x);                                                          \
    if (e_ != 0) {                                                                    \
      std::printf("{\"error\": \"%s returned %d\"}\n", #x, e_);                        \
      return 1;                                                                       \
    }                                                                                 \
  } while (0)

int main(int argc, char** argv) {
  if (argc < 5) {
    std::printf("{\"error\": \"usage: cublaslt_gemm nvfp4|fp8 M N K [reps]\"}\n");
    return 2;
  }
  const bool fp4 = std::strcmp(argv[1], "nvfp4") == 0;
  const long long M = std::atoll(argv[2]), N = std::atoll(argv[3]), K = std::atoll(argv[4]);
  const int reps = argc > 5 ? std::atoi(argv[5]) : 20;
  if (M <= 0 || N <= 0 || K <= 0 || K % 32 != 0 || reps <= 0) {
    std::printf("{\"error\": \"bad shape\"}\n");
    return 2;
  }
  const size_t a_bytes = fp4 ? (size_t)M * K / 2 : (size_t)M * K;
  const size_t b_bytes = fp4 ? (size_t)N * K / 2 : (size_t)N * K;
  const size_t d_bytes = (size_t)M * N * 4;
  void *A = nullptr, *B = nullptr, *D = nullptr, *sA = nullptr, *sB = nullptr, *ws = nullptr;
  const size_t ws_bytes = 64u << 20;
  CHECK(cudaMalloc(&A, a_bytes));
  CHECK(cudaMalloc(&B, b_bytes));
  CHECK(cudaMalloc(&D, d_bytes));
  CHECK(cudaMalloc(&ws, ws_bytes));
  CHECK(cudaMemset(A, fp4 ? 0x22 : 0x38, a_bytes));   // E2M1 pairs of 1.0 / E4M3 1.0
  CHECK(cudaMemset(B, fp4 ? 0x22 : 0x38, b_bytes));

  cublasLtHandle_t lt;
  CHECK(cublasLtCreate(&lt));
  cublasLtMatmulDesc_t desc;
  CHECK(cublasLtMatmulDescCreate(&desc, CUBLAS_COMPUTE_32F, CUDA_R_32F));
  const cublasOperation_t op_t = CUBLAS_OP_T, op_n = CUBLAS_OP_N;
  CHECK(cublasLtMatmulDescSetAttribute(desc, CUBLASLT_MATMUL_DESC_TRANSA, &op_t, sizeof op_t));
  CHECK(cublasLtMatmulDescSetAttribute(desc, CUBLASLT_MATMUL_DESC_TRANSB, &op_n, sizeof op_n));
  if (fp4) {
    // one scale byte per 16 elements, rows padded to 128 and blocks to 4
    const size_t sa_bytes = (size_t)((N + 127) / 128 * 128) * (size_t)((K / 16 + 3) / 4 * 4);
    const size_t sb_bytes = (size_t)((M + 127) / 128 * 128) * (size_t)((K / 16 + 3) / 4 * 4);
    CHECK(cudaMalloc(&sA, sa_bytes));
    CHECK(cudaMalloc(&sB, sb_bytes));
    CHECK(cudaMemset(sA, 0x38, sa_bytes));   // UE4M3 1.0
    CHECK(cudaMemset(sB, 0x38, sb_bytes));
    const cublasLtMatmulMatrixScale_t mode = CUBLASLT_MATMUL_MATRIX_SCALE_VEC16_UE4M3;
    CHECK(cublasLtMatmulDescSetAttribute(desc, CUBLASLT_MATMUL_DESC_A_SCALE_MODE, &mode, sizeof mode));
    CHECK(cublasLtMatmulDescSetAttribute(desc, CUBLASLT_MATMUL_DESC_B_SCALE_MODE, &mode, sizeof mode));
    CHECK(cublasLtMatmulDescSetAttribute(desc, CUBLASLT_MATMUL_DESC_A_SCALE_POINTER, &sA, sizeof sA));
    CHECK(cublasLtMatmulDescSetAttribute(desc, CUBLASLT_MATMUL_DESC_B_SCALE_POINTER, &sB, sizeof sB));
  }
  const cudaDataType ab = fp4 ? CUDA_R_4F_E2M1 : CUDA_R_8F_E4M3;
  cublasLtMatrixLayout_t la, lb, ld;
  CHECK(cublasLtMatrixLayoutCreate(&la, ab, K, N, K));
  CHECK(cublasLtMatrixLayoutCreate(&lb, ab, K, M, K));
  CHECK(cublasLtMatrixLayoutCreate(&ld, CUDA_R_32F, N, M, N));
  cublasLtMatmulPreference_t pref;
  CHECK(cublasLtMatmulPreferenceCreate(&pref));
  CHECK(cublasLtMatmulPreferenceSetAttribute(pref, CUBLASLT_MATMUL_PREF_MAX_WORKSPACE_BYTES, &ws_bytes,
                                             sizeof ws_bytes));
  cublasLtMatmulHeuristicResult_t cand[8];
  int ncand = 0;
  CHECK(cublasLtMatmulAlgoGetHeuristic(lt, desc, la, lb, ld, ld, pref, 8, cand, &ncand));
  if (ncand == 0) {
    std::printf("{\"error\": \"no algorithm\"}\n");
    return 1;
  }
  const float alpha = 1.0f, beta = 0.0f;
  cudaEvent_t e0, e1;
  CHECK(cudaEventCreate(&e0));
  CHECK(cudaEventCreate(&e1));
  float best = 1e30f;
  for (int c = 0; c < ncand; ++c) {
    CHECK(cublasLtMatmul(lt, desc, &alpha, B, la, A, lb, &beta, D, ld, D, ld, &cand[c].algo, ws, ws_bytes, 0));
    CHECK(cudaDeviceSynchronize());
    CHECK(cudaEventRecord(e0));
    for (int r = 0; r < reps; ++r)
      CHECK(cublasLtMatmul(lt, desc, &alpha, B, la, A, lb, &beta, D, ld, D, ld, &cand[c].algo, ws, ws_bytes, 0));
    CHECK(cudaEventRecord(e1));
    CHECK(cudaEventSynchronize(e1));
    float ms = 0.0f;
    CHECK(cudaEventElapsedTime(&ms, e0, e1));
    if (ms / reps < best) best = ms / reps;
  }
  std::printf("{\"fmt\": \"%s\", \"M\": %lld, \"N\": %lld, \"K\": %lld, \"candidates\": %d, \"ms\": %.5f, "
              "\"tflops\": %.1f}\n",
              fp4 ? "nvfp4" : "fp8", M, N, K, ncand, best, 2.0 * M * N * K / (best * 1e-3) / 1e12);
  cublasLtMatmulPreferenceDestroy(pref);
  cublasLtMatrixLayoutDestroy(la);
  cublasLtMatrixLayoutDestroy(lb);
  cublasLtMatrixLayoutDestroy(ld);
  cublasLtMatmulDescDestroy(desc);
  cublasLtDestroy(lt);
  cudaFree(A);
  cudaFree(B);
  cudaFree(D);
  cudaFree(ws);
  if (sA) cudaFree(sA);
  if (sB) cudaFree(sB);
  return 0;
}
