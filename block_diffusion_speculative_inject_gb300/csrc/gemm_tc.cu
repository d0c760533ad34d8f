// Tensor-core GEMM (placeholder until the tcgen05 kernel lands): disabled.
#include "gemm_tc.h"

namespace dflash {
struct TcGemm { int dummy; };
cudaError_t tc_gemm_create(TcGemm **out, int, int) { *out = nullptr; return cudaSuccess; }
void tc_gemm_destroy(TcGemm *t) { delete t; }
int tc_gemm_launches(const TcGemm *, const GemmDesc &) { return 0; }
cudaError_t tc_gemm_run(TcGemm *, const GemmDesc &, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace dflash
