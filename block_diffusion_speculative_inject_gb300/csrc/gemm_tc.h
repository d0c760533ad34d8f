// Tensor-core (tcgen05 / TMEM / TMA) GEMM for bf16 operands — internal interface.
#pragma once
#include "common.cuh"

namespace dflash {

struct TcGemm;

// Creates the per-context GEMM state (driver entry point for tensor maps, SM count, the
// device error flag its bounded waits raise).
cudaError_t tc_gemm_create(TcGemm **out, int device, int num_sms, int *err_flag);
void tc_gemm_destroy(TcGemm *t);
// bf16 2-D tensor map over a row-major [rows, cols] matrix with row stride ld elements,
// box {box_cols, box_rows}, 128-byte swizzle. False if the driver rejects it.
bool tc_encode_2d(TcGemm *t, const void *ptr, unsigned long long rows, unsigned long long cols,
                  unsigned long long ld, unsigned box_cols, unsigned box_rows, void *map_out);

// Incremented whenever an internal buffer (split-K workspace) is reallocated; captured
// graphs that used the old buffer must be re-captured.
int tc_gemm_generation(const TcGemm *t);

// Split-K factor the GEMM will use, and the floats its partials need in partials mode.
int tc_gemm_splits(const TcGemm *t, const GemmDesc &d);

// Number of kernel launches tc_gemm_run issues for this GEMM.
int tc_gemm_launches(const TcGemm *t, const GemmDesc &d);
// Runs Y = epilogue(X . W^T) for bf16 W and a bf16 (or bf16 hi/lo pair) X.
cudaError_t tc_gemm_run(TcGemm *t, const GemmDesc &d, cudaStream_t s);

}  // namespace dflash
