// k_step_ademamix.cu -- step kernels of AdEMAMix.
#include "k_step8.cuh"
#include "k_step32.cuh"

namespace bnb8 {

#define BNB8_DISPATCH(OPTV, DTV, MODEV, CALL8, CALL32) \
  if (optim == OPTV && dtype == DTV && mode == MODEV) \
    return bits == 8 ? CALL8<OPTV, DTV, MODEV>(a, grid, s) : CALL32<OPTV, DTV, MODEV>(a, grid, s);

cudaError_t launch_step_ademamix(int bits, int optim, int dtype, int mode, const StepArgs& a,
                                int grid, cudaStream_t s) {
  BNB8_DISPATCH(ADEMAMIX, DT_F32, MODE_STEP, launch_step8_t, launch_step32_t)
  BNB8_DISPATCH(ADEMAMIX, DT_F32, MODE_NORM, launch_step8_t, launch_step32_t)
  BNB8_DISPATCH(ADEMAMIX, DT_F32, MODE_BCLIP, launch_step8_t, launch_step32_t)
  BNB8_DISPATCH(ADEMAMIX, DT_F32, MODE_TWMAX, launch_step8_t, launch_step32_t)
  BNB8_DISPATCH(ADEMAMIX, DT_F32, MODE_TWSTEP, launch_step8_t, launch_step32_t)
  BNB8_DISPATCH(ADEMAMIX, DT_BF16, MODE_STEP, launch_step8_t, launch_step32_t)
  BNB8_DISPATCH(ADEMAMIX, DT_BF16, MODE_NORM, launch_step8_t, launch_step32_t)
  BNB8_DISPATCH(ADEMAMIX, DT_BF16, MODE_BCLIP, launch_step8_t, launch_step32_t)
  BNB8_DISPATCH(ADEMAMIX, DT_BF16, MODE_TWMAX, launch_step8_t, launch_step32_t)
  BNB8_DISPATCH(ADEMAMIX, DT_BF16, MODE_TWSTEP, launch_step8_t, launch_step32_t)
  BNB8_DISPATCH(ADEMAMIX, DT_F16, MODE_STEP, launch_step8_t, launch_step32_t)
  BNB8_DISPATCH(ADEMAMIX, DT_F16, MODE_NORM, launch_step8_t, launch_step32_t)
  BNB8_DISPATCH(ADEMAMIX, DT_F16, MODE_BCLIP, launch_step8_t, launch_step32_t)
  BNB8_DISPATCH(ADEMAMIX, DT_F16, MODE_TWMAX, launch_step8_t, launch_step32_t)
  BNB8_DISPATCH(ADEMAMIX, DT_F16, MODE_TWSTEP, launch_step8_t, launch_step32_t)
  return cudaErrorInvalidValue;
}

#undef BNB8_DISPATCH
#define BNB8_DISPATCH(OPTV, DTV, MODEV, CALL8, CALL32) \
  if (optim == OPTV && dtype == DTV && mode == MODEV) \
    return bits == 8 ? CALL8<OPTV, DTV, MODEV>() : CALL32<OPTV, DTV, MODEV>();

int ctas_step_ademamix(int bits, int optim, int dtype, int mode) {
  BNB8_DISPATCH(ADEMAMIX, DT_F32, MODE_STEP, ctas_step8_t, ctas_step32_t)
  BNB8_DISPATCH(ADEMAMIX, DT_F32, MODE_NORM, ctas_step8_t, ctas_step32_t)
  BNB8_DISPATCH(ADEMAMIX, DT_F32, MODE_BCLIP, ctas_step8_t, ctas_step32_t)
  BNB8_DISPATCH(ADEMAMIX, DT_F32, MODE_TWMAX, ctas_step8_t, ctas_step32_t)
  BNB8_DISPATCH(ADEMAMIX, DT_F32, MODE_TWSTEP, ctas_step8_t, ctas_step32_t)
  BNB8_DISPATCH(ADEMAMIX, DT_BF16, MODE_STEP, ctas_step8_t, ctas_step32_t)
  BNB8_DISPATCH(ADEMAMIX, DT_BF16, MODE_NORM, ctas_step8_t, ctas_step32_t)
  BNB8_DISPATCH(ADEMAMIX, DT_BF16, MODE_BCLIP, ctas_step8_t, ctas_step32_t)
  BNB8_DISPATCH(ADEMAMIX, DT_BF16, MODE_TWMAX, ctas_step8_t, ctas_step32_t)
  BNB8_DISPATCH(ADEMAMIX, DT_BF16, MODE_TWSTEP, ctas_step8_t, ctas_step32_t)
  BNB8_DISPATCH(ADEMAMIX, DT_F16, MODE_STEP, ctas_step8_t, ctas_step32_t)
  BNB8_DISPATCH(ADEMAMIX, DT_F16, MODE_NORM, ctas_step8_t, ctas_step32_t)
  BNB8_DISPATCH(ADEMAMIX, DT_F16, MODE_BCLIP, ctas_step8_t, ctas_step32_t)
  BNB8_DISPATCH(ADEMAMIX, DT_F16, MODE_TWMAX, ctas_step8_t, ctas_step32_t)
  BNB8_DISPATCH(ADEMAMIX, DT_F16, MODE_TWSTEP, ctas_step8_t, ctas_step32_t)
  return 1;
}

#undef BNB8_DISPATCH

}  // namespace bnb8
