// gemm_tc_bf16.cu -- instantiations of the tensor-core GEMM for bf16 operands.
#include "gemm_tc.cuh"

namespace bi {

bi_status launch_gemm_tc_bf16(const void *a, int64_t lda, const void *b, int64_t ldb, bool b_nk,
                            const GemmArgs &args, const TcConfig &cfg, cudaStream_t s) {
    return launch_gemm_tc_typed<__nv_bfloat16>(a, lda, b, ldb, b_nk, args, BI_BF16, cfg, s);
}

bi_status init_gemm_tc_bf16() { return init_tc_all<__nv_bfloat16>(); }

}  // namespace bi
