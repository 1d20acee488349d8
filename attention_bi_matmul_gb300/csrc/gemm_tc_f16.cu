// gemm_tc_f16.cu -- instantiations of the tensor-core GEMM for f16 operands.
#include "gemm_tc.cuh"

namespace bi {

bi_status launch_gemm_tc_f16(const void *a, int64_t lda, const void *b, int64_t ldb, bool b_nk,
                            const GemmArgs &args, const TcConfig &cfg, cudaStream_t s) {
    return launch_gemm_tc_typed<__half>(a, lda, b, ldb, b_nk, args, BI_F16, cfg, s);
}

bi_status init_gemm_tc_f16() { return init_tc_all<__half>(); }

}  // namespace bi
