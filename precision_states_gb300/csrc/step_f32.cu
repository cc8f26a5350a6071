// step_f32.cu -- fused step instantiations with FP32 m, v (and m2).
#include "step_kernel.cuh"

namespace psopt {

cudaError_t launch_step_fp32_states(int grad_dtype, int algo, const StepArgs& a, int sm_count,
                                    cudaStream_t s) {
  if (grad_dtype == OPT_BF16) {
    if (algo == ALGO_ADEMAMIX) return launch_one<OPT_BF16, SC_F32, ALGO_ADEMAMIX, false>(a, sm_count, s);
    return launch_one<OPT_BF16, SC_F32, ALGO_ADAMW, false>(a, sm_count, s);
  }
  if (algo == ALGO_ADEMAMIX) return launch_one<OPT_F32, SC_F32, ALGO_ADEMAMIX, false>(a, sm_count, s);
  return launch_one<OPT_F32, SC_F32, ALGO_ADAMW, false>(a, sm_count, s);
}

}  // namespace psopt
