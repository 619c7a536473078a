// k_step_adam.cu -- step kernels of the 2-state optimizers (Adam, AdamW).
#include "k_step8.cuh"
#include "k_step32.cuh"

namespace bnb8 {

#define BNB8_DISPATCH(OPTV, DTV, MODEV, CALL8, CALL32) \
  if (optim == OPTV && dtype == DTV && mode == MODEV) \
    return bits == 8 ? CALL8<OPTV, DTV, MODEV>(a, grid, s) : CALL32<OPTV, DTV, MODEV>(a, grid, s);

cudaError_t launch_step_adam(int bits, int optim, int dtype, int mode, const StepArgs& a,
                                int grid, cudaStream_t s) {
  BNB8_DISPATCH(ADAM, DT_F32, MODE_STEP, launch_step8_t, launch_step32_t)
  BNB8_DISPATCH(ADAM, DT_F32, MODE_NORM, launch_step8_t, launch_step32_t)
  BNB8_DISPATCH(ADAM, DT_F32, MODE_BCLIP, launch_step8_t, launch_step32_t)
  BNB8_DISPATCH(ADAM, DT_F32, MODE_TWMAX, launch_step8_t, launch_step32_t)
  BNB8_DISPATCH(ADAM, DT_F32, MODE_TWSTEP, launch_step8_t, launch_step32_t)
  BNB8_DISPATCH(ADAM, DT_BF16, MODE_STEP, launch_step8_t, launch_step32_t)
  BNB8_DISPATCH(ADAM, DT_BF16, MODE_NORM, launch_step8_t, launch_step32_t)
  BNB8_DISPATCH(ADAM, DT_BF16, MODE_BCLIP, launch_step8_t, launch_step32_t)
  BNB8_DISPATCH(ADAM, DT_BF16, MODE_TWMAX, launch_step8_t, launch_step32_t)
  BNB8_DISPATCH(ADAM, DT_BF16, MODE_TWSTEP, launch_step8_t, launch_step32_t)
  BNB8_DISPATCH(ADAM, DT_F16, MODE_STEP, launch_step8_t, launch_step32_t)
  BNB8_DISPATCH(ADAM, DT_F16, MODE_NORM, launch_step8_t, launch_step32_t)
  BNB8_DISPATCH(ADAM, DT_F16, MODE_BCLIP, launch_step8_t, launch_step32_t)
  BNB8_DISPATCH(ADAM, DT_F16, MODE_TWMAX, launch_step8_t, launch_step32_t)
  BNB8_DISPATCH(ADAM, DT_F16, MODE_TWSTEP, launch_step8_t, launch_step32_t)
  BNB8_DISPATCH(ADAMW, DT_F32, MODE_STEP, launch_step8_t, launch_step32_t)
  BNB8_DISPATCH(ADAMW, DT_F32, MODE_NORM, launch_step8_t, launch_step32_t)
  BNB8_DISPATCH(ADAMW, DT_F32, MODE_BCLIP, launch_step8_t, launch_step32_t)
  BNB8_DISPATCH(ADAMW, DT_F32, MODE_TWMAX, launch_step8_t, launch_step32_t)
  BNB8_DISPATCH(ADAMW, DT_F32, MODE_TWSTEP, launch_step8_t, launch_step32_t)
  BNB8_DISPATCH(ADAMW, DT_BF16, MODE_STEP, launch_step8_t, launch_step32_t)
  BNB8_DISPATCH(ADAMW, DT_BF16, MODE_NORM, launch_step8_t, launch_step32_t)
  BNB8_DISPATCH(ADAMW, DT_BF16, MODE_BCLIP, launch_step8_t, launch_step32_t)
  BNB8_DISPATCH(ADAMW, DT_BF16, MODE_TWMAX, launch_step8_t, launch_step32_t)
  BNB8_DISPATCH(ADAMW, DT_BF16, MODE_TWSTEP, launch_step8_t, launch_step32_t)
  BNB8_DISPATCH(ADAMW, DT_F16, MODE_STEP, launch_step8_t, launch_step32_t)
  BNB8_DISPATCH(ADAMW, DT_F16, MODE_NORM, launch_step8_t, launch_step32_t)
  BNB8_DISPATCH(ADAMW, DT_F16, MODE_BCLIP, launch_step8_t, launch_step32_t)
  BNB8_DISPATCH(ADAMW, DT_F16, MODE_TWMAX, launch_step8_t, launch_step32_t)
  BNB8_DISPATCH(ADAMW, DT_F16, MODE_TWSTEP, launch_step8_t, launch_step32_t)
  return cudaErrorInvalidValue;
}

#undef BNB8_DISPATCH
#define BNB8_DISPATCH(OPTV, DTV, MODEV, CALL8, CALL32) \
  if (optim == OPTV && dtype == DTV && mode == MODEV) \
    return bits == 8 ? CALL8<OPTV, DTV, MODEV>() : CALL32<OPTV, DTV, MODEV>();

int ctas_step_adam(int bits, int optim, int dtype, int mode) {
  BNB8_DISPATCH(ADAM, DT_F32, MODE_STEP, ctas_step8_t, ctas_step32_t)
  BNB8_DISPATCH(ADAM, DT_F32, MODE_NORM, ctas_step8_t, ctas_step32_t)
  BNB8_DISPATCH(ADAM, DT_F32, MODE_BCLIP, ctas_step8_t, ctas_step32_t)
  BNB8_DISPATCH(ADAM, DT_F32, MODE_TWMAX, ctas_step8_t, ctas_step32_t)
  BNB8_DISPATCH(ADAM, DT_F32, MODE_TWSTEP, ctas_step8_t, ctas_step32_t)
  BNB8_DISPATCH(ADAM, DT_BF16, MODE_STEP, ctas_step8_t, ctas_step32_t)
  BNB8_DISPATCH(ADAM, DT_BF16, MODE_NORM, ctas_step8_t, ctas_step32_t)
  BNB8_DISPATCH(ADAM, DT_BF16, MODE_BCLIP, ctas_step8_t, ctas_step32_t)
  BNB8_DISPATCH(ADAM, DT_BF16, MODE_TWMAX, ctas_step8_t, ctas_step32_t)
  BNB8_DISPATCH(ADAM, DT_BF16, MODE_TWSTEP, ctas_step8_t, ctas_step32_t)
  BNB8_DISPATCH(ADAM, DT_F16, MODE_STEP, ctas_step8_t, ctas_step32_t)
  BNB8_DISPATCH(ADAM, DT_F16, MODE_NORM, ctas_step8_t, ctas_step32_t)
  BNB8_DISPATCH(ADAM, DT_F16, MODE_BCLIP, ctas_step8_t, ctas_step32_t)
  BNB8_DISPATCH(ADAM, DT_F16, MODE_TWMAX, ctas_step8_t, ctas_step32_t)
  BNB8_DISPATCH(ADAM, DT_F16, MODE_TWSTEP, ctas_step8_t, ctas_step32_t)
  BNB8_DISPATCH(ADAMW, DT_F32, MODE_STEP, ctas_step8_t, ctas_step32_t)
  BNB8_DISPATCH(ADAMW, DT_F32, MODE_NORM, ctas_step8_t, ctas_step32_t)
  BNB8_DISPATCH(ADAMW, DT_F32, MODE_BCLIP, ctas_step8_t, ctas_step32_t)
  BNB8_DISPATCH(ADAMW, DT_F32, MODE_TWMAX, ctas_step8_t, ctas_step32_t)
  BNB8_DISPATCH(ADAMW, DT_F32, MODE_TWSTEP, ctas_step8_t, ctas_step32_t)
  BNB8_DISPATCH(ADAMW, DT_BF16, MODE_STEP, ctas_step8_t, ctas_step32_t)
  BNB8_DISPATCH(ADAMW, DT_BF16, MODE_NORM, ctas_step8_t, ctas_step32_t)
  BNB8_DISPATCH(ADAMW, DT_BF16, MODE_BCLIP, ctas_step8_t, ctas_step32_t)
  BNB8_DISPATCH(ADAMW, DT_BF16, MODE_TWMAX, ctas_step8_t, ctas_step32_t)
  BNB8_DISPATCH(ADAMW, DT_BF16, MODE_TWSTEP, ctas_step8_t, ctas_step32_t)
  BNB8_DISPATCH(ADAMW, DT_F16, MODE_STEP, ctas_step8_t, ctas_step32_t)
  BNB8_DISPATCH(ADAMW, DT_F16, MODE_NORM, ctas_step8_t, ctas_step32_t)
  BNB8_DISPATCH(ADAMW, DT_F16, MODE_BCLIP, ctas_step8_t, ctas_step32_t)
  BNB8_DISPATCH(ADAMW, DT_F16, MODE_TWMAX, ctas_step8_t, ctas_step32_t)
  BNB8_DISPATCH(ADAMW, DT_F16, MODE_TWSTEP, ctas_step8_t, ctas_step32_t)
  return 1;
}

#undef BNB8_DISPATCH

cudaError_t launch_tw_store(int optim, const StepArgs& a, cudaStream_t s) {
  switch (optim) {
    case ADAM: return launch_tw_store_t<ADAM>(a, s);
    case ADAMW: return launch_tw_store_t<ADAMW>(a, s);
    case MOMENTUM: return launch_tw_store_t<MOMENTUM>(a, s);
    case RMSPROP: return launch_tw_store_t<RMSPROP>(a, s);
    case ADAGRAD: return launch_tw_store_t<ADAGRAD>(a, s);
    case LION: return launch_tw_store_t<LION>(a, s);
    case ADEMAMIX: return launch_tw_store_t<ADEMAMIX>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace bnb8
