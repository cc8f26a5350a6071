// step_lowp.cu -- fused AdamW instantiations with a BF16 first moment and a
// BF16 / E4M3 / E2M2 second moment, nearest or stochastic rounding.
#include "step_bulk.cuh"
#include "step_kernel.cuh"

namespace psopt {

template <int GT, int COMBO, bool SR>
static cudaError_t launch_lowp(const StepArgs& a, int sm_count, cudaStream_t s) {
  if constexpr (StepShape<GT, COMBO, ALGO_ADAMW, SR>::kBulk) return launch_bulk<GT, COMBO, SR>(a, sm_count, s);
  else return launch_one<GT, COMBO, ALGO_ADAMW, SR>(a, sm_count, s);
}

template <int GT>
static cudaError_t dispatch_lowp(int combo, int stochastic, const StepArgs& a, int sm_count,
                                 cudaStream_t s) {
  switch (combo) {
    case SC_BF16_BF16:
      return stochastic ? launch_lowp<GT, SC_BF16_BF16, true>(a, sm_count, s) : launch_lowp<GT, SC_BF16_BF16, false>(a, sm_count, s);
    case SC_BF16_E4M3:
      return stochastic ? launch_lowp<GT, SC_BF16_E4M3, true>(a, sm_count, s) : launch_lowp<GT, SC_BF16_E4M3, false>(a, sm_count, s);
    case SC_BF16_E2M2:
      return stochastic ? launch_lowp<GT, SC_BF16_E2M2, true>(a, sm_count, s) : launch_lowp<GT, SC_BF16_E2M2, false>(a, sm_count, s);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_step_lowp_states(int grad_dtype, int combo, int stochastic, const StepArgs& a,
                                    int sm_count, cudaStream_t s) {
  if (grad_dtype == OPT_BF16) return dispatch_lowp<OPT_BF16>(combo, stochastic, a, sm_count, s);
  return dispatch_lowp<OPT_F32>(combo, stochastic, a, sm_count, s);
}

}  // namespace psopt
