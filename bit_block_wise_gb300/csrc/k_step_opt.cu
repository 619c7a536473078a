// k_step_opt.cu -- the step kernels of one optimizer (all dtypes and modes).
// The build compiles this file once per optimizer with -DBNB8_OPT=<Optim>, so
// the optimizers' kernels compile in parallel.
#include "k_step8.cuh"
#include "k_step32.cuh"

#ifndef BNB8_OPT
#error "compile with -DBNB8_OPT=<optimizer number>"
#endif

namespace bnb8 {

namespace {
template <int DT, int MODE>
cudaError_t launch_one(int bits, const StepArgs& a, int grid, cudaStream_t s) {
  return bits == 8 ? launch_step8_t<BNB8_OPT, DT, MODE>(a, grid, s)
                   : launch_step32_t<BNB8_OPT, DT, MODE>(a, grid, s);
}
template <int DT>
cudaError_t launch_dt(int bits, int mode, const StepArgs& a, int grid, cudaStream_t s) {
  switch (mode) {
    case MODE_STEP: return launch_one<DT, MODE_STEP>(bits, a, grid, s);
    case MODE_NORM: return launch_one<DT, MODE_NORM>(bits, a, grid, s);
    case MODE_BCLIP: return launch_one<DT, MODE_BCLIP>(bits, a, grid, s);
    case MODE_TWMAX: return launch_one<DT, MODE_TWMAX>(bits, a, grid, s);
    case MODE_TWSTEP: return launch_one<DT, MODE_TWSTEP>(bits, a, grid, s);
    default: return cudaErrorInvalidValue;
  }
}
template <int DT, int MODE>
int ctas_one(int bits) {
  return bits == 8 ? ctas_step8_t<BNB8_OPT, DT, MODE>() : ctas_step32_t<BNB8_OPT, DT, MODE>();
}
template <int DT>
int ctas_dt(int bits, int mode) {
  switch (mode) {
    case MODE_STEP: return ctas_one<DT, MODE_STEP>(bits);
    case MODE_NORM: return ctas_one<DT, MODE_NORM>(bits);
    case MODE_BCLIP: return ctas_one<DT, MODE_BCLIP>(bits);
    case MODE_TWMAX: return ctas_one<DT, MODE_TWMAX>(bits);
    case MODE_TWSTEP: return ctas_one<DT, MODE_TWSTEP>(bits);
    default: return 1;
  }
}
}  // namespace

template <>
cudaError_t launch_step_opt<BNB8_OPT>(int bits, int dtype, int mode, const StepArgs& a, int grid,
                                      cudaStream_t s) {
  switch (dtype) {
    case DT_F32: return launch_dt<DT_F32>(bits, mode, a, grid, s);
    case DT_BF16: return launch_dt<DT_BF16>(bits, mode, a, grid, s);
    case DT_F16: return launch_dt<DT_F16>(bits, mode, a, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

template <>
int ctas_step_opt<BNB8_OPT>(int bits, int dtype, int mode) {
  switch (dtype) {
    case DT_F32: return ctas_dt<DT_F32>(bits, mode);
    case DT_BF16: return ctas_dt<DT_BF16>(bits, mode);
    case DT_F16: return ctas_dt<DT_F16>(bits, mode);
    default: return 1;
  }
}

template <>
cudaError_t tw_store_opt<BNB8_OPT>(const StepArgs& a, cudaStream_t s) {
  return launch_tw_store_t<BNB8_OPT>(a, s);
}

}  // namespace bnb8
