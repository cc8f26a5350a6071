// step_f32.cu -- fused step instantiations with FP32 m, v (and m2), and the
// device step counter that lets a captured CUDA graph replay the step.
#include "step_dyn.cuh"
#include "step_kernel.cuh"

namespace psopt {

namespace {

// One thread: advance the plan's step counter and form the step's scalar
// block.  Every field but the two bias corrections is the same each step
// and comes from the host (`base`); the corrections are formed here, in
// double from the FP32 hyperparameters and rounded once, as the host does
// ("Investigate SM103 bias-correction broadcast in 32-bit optimizers",
// 'Problem': one computation per step, not one per thread).
__global__ void step_scalars_kernel(opt_step_scalars base, int64_t* counter, opt_step_scalars* out) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  const int64_t t = *counter + 1;
  *counter = t;
  base.inv_bc1 = (float)(1.0 / (1.0 - pow((double)base.beta1, (double)t)));
  base.inv_bc2 = (float)(1.0 / (1.0 - pow((double)base.beta2, (double)t)));
  *out = base;
}

__global__ void set_step_kernel(int64_t* counter, int64_t value) {
  if (threadIdx.x == 0 && blockIdx.x == 0) *counter = value;
}

template <int GT, int ALGO>
cudaError_t launch_f32(const StepArgs& a, int sm_count, cudaStream_t s) {
  if (a.d_sc != nullptr) return launch_dyn<GT, SC_F32, ALGO, false, true>(a, sm_count, s);
  return launch_dyn<GT, SC_F32, ALGO, false, false>(a, sm_count, s);
}

}  // namespace

cudaError_t launch_step_fp32_states(int grad_dtype, int algo, const StepArgs& a, int sm_count,
                                    cudaStream_t s) {
  if (grad_dtype == OPT_BF16) {
    if (algo == ALGO_ADEMAMIX) return launch_f32<OPT_BF16, ALGO_ADEMAMIX>(a, sm_count, s);
    return launch_f32<OPT_BF16, ALGO_ADAMW>(a, sm_count, s);
  }
  if (algo == ALGO_ADEMAMIX) return launch_f32<OPT_F32, ALGO_ADEMAMIX>(a, sm_count, s);
  return launch_f32<OPT_F32, ALGO_ADAMW>(a, sm_count, s);
}

cudaError_t launch_step_scalars(const opt_step_scalars& base, int64_t* counter, opt_step_scalars* out,
                                cudaStream_t s) {
  step_scalars_kernel<<<1, 32, 0, s>>>(base, counter, out);
  return cudaGetLastError();
}

cudaError_t launch_set_step(int64_t* counter, int64_t value, cudaStream_t s) {
  set_step_kernel<<<1, 32, 0, s>>>(counter, value);
  return cudaGetLastError();
}

}  // namespace psopt
