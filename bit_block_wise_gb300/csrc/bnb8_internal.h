// bnb8_internal.h -- launch arguments shared by the host library (bnb8_api.cu)
// and the kernel translation units.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace bnb8 {

// Per-device one-time set-up (a kernel's shared-memory limit, the device
// address of a symbol) is cached in arrays of kMaxDevices atomics, so that
// host threads calling the library at the same time never race on the cache.
// Devices with a larger ordinal skip the cache and redo the set-up per call.
constexpr int kMaxDevices = 64;

// cudaFuncSetAttribute(fn, MaxDynamicSharedMemorySize, bytes) once per device.
inline cudaError_t set_smem_limit_once(const void* fn, int bytes,
                                       std::atomic<unsigned char>* done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool cached = dev >= 0 && dev < kMaxDevices;
  if (cached && done[dev].load(std::memory_order_acquire) != 0) return cudaSuccess;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && cached) done[dev].store(1, std::memory_order_release);
  return e;
}

// Bits of the library's device status word (StepArgs::status).
constexpr uint32_t kStatusWaitTimeout = 1u;  // a bounded wait for an async copy ran out

constexpr int kThreads = 512;       // threads per CTA of every step / quantize kernel
constexpr int kMaxTensors = 96;     // descriptors per launch (kernel parameter space)
constexpr int kTblSize = 5892;      // search-table entries per map: 2 signs x 2946 buckets
constexpr int kTblZero = 2946;      // entry of the smallest positive bucket

enum Optim { ADAM = 0, ADAMW = 1, MOMENTUM = 2, RMSPROP = 3, ADAGRAD = 4, LION = 5, ADEMAMIX = 6 };
enum Dtype { DT_F32 = 0, DT_BF16 = 1, DT_F16 = 2 };
// MODE_STEP: the update; MODE_NORM: the per-tensor max_unorm pre-pass;
// MODE_BCLIP: the update with max_unorm applied per block (no pre-pass);
// MODE_TWMAX: tensor-wise quantization's first pass, the new absmax of each
// state of each tensor (the update is computed, nothing is stored);
// MODE_TWSTEP: tensor-wise quantization's step (requantized with that absmax).
enum Mode { MODE_STEP = 0, MODE_NORM = 1, MODE_BCLIP = 2, MODE_TWMAX = 3, MODE_TWSTEP = 4 };

// One tensor of a launch.  Pointers are device pointers.
struct DevTensor {
  void* p;
  const void* g;
  void* s1;      // first state (AdEMAMix: m1 then m2)
  void* s2;      // second state (Adam v, AdEMAMix nu)
  float* a1;     // absmax of s1 (AdEMAMix: [2, nblocks])
  float* a2;     // absmax of s2
  int64_t n;
  int64_t first_block;  // index of the tensor's first block in the launch
  int32_t index;        // position in the caller's tensor list (clip / out_scale slot)
  // bit 0: every stream of this tensor is aligned for vector access; bit 1:
  // also for 16-byte bulk copies of whole chunks (multiples of 256 elements)
  int32_t vec_ok;
  int32_t nblocks;      // ceil(n / B)
  int32_t units;        // the ring step's work units: ceil(n / max(512, B))
};

// Per-step scalars (host: binary64, rounded once) and the tensor table.
struct StepArgs {
  float b1, b2, b3t, omb1, omb2, omb3t;
  float step_size, eps_hat, inv_bc1, alpha_t, decay, wd, gscale;
  float max_unorm, unorm_c;  // MODE_BCLIP: limit and |direction| = unorm_c * |u|
  int32_t skip_zeros;
  int32_t log2B;
  int32_t ntensors;
  int64_t total_blocks;
  const float* qmap1;
  const float* qmap2;
  const float* clip;     // per-tensor step multipliers (by DevTensor::index) or nullptr
  float2* partials;      // MODE_NORM: per-block (sum u^2, sum p^2), indexed by launch block
  // Tensor-wise quantization (one absmax per state per tensor): absmax
  // arrays hold one value per state; tw_acc[4 * index + k] is the new absmax
  // bit pattern of state k (max-reduced by MODE_TWMAX) and [4 * index + 3]
  // is nonzero if any element of the tensor is updated.
  int32_t tensorwise;
  // 1 if a zero gradient over zero moments has the update direction of its
  // (signed zero) numerator exactly: eps_hat > 0 and finite, and finite
  // betas, 1 - betas and gradient scale
  int32_t zero_ratio;
  uint32_t* tw_acc;
  int32_t nsm;             // SMs of the device (persistent grids sized in the launcher)
  int32_t stall_test;      // test hook: one warp withholds a copy so that its wait runs out
  // 1 if every tensor of the launch has vec_ok == 3 and n a multiple of
  // max(512, B): all its 512-element chunks are whole and bulk-copyable
  int32_t whole;
  int64_t ring_units;      // sum of DevTensor::units
  uint64_t wait_ns;        // bound of every wait for an async copy
  uint32_t* status;        // the library's device status word (kStatus* bits are or-ed in)
  // The carried parameter norm (BNB8_CARRY_PNORM): a MODE_STEP launch with
  // carry_out set leaves the sum of the new p^2 of each block in
  // partials[block].y; the launch with carry_writer set then stores carry_write
  // in *carry_stamp.  A MODE_NORM launch whose *carry_stamp equals
  // carry_expect takes those sums instead of reading p for them.
  int32_t carry_out;
  int32_t carry_writer;
  uint64_t* carry_stamp;
  uint64_t carry_expect;
  uint64_t carry_write;
  // MODE_NORM: the per-tensor tickets of the reduction that follows (CTA 0
  // sets tickets[0, ntensors) to 0), or null
  uint32_t* tickets;
  DevTensor t[kMaxTensors];
};

struct QuantArgs {
  const void* x;
  uint8_t* codes;
  float* absmax;
  const float* qmap;
  int64_t n;
  int64_t total_blocks;
  int32_t log2B;
};

struct DequantArgs {
  const uint8_t* codes;
  const float* absmax;
  const float* qmap;
  void* out;
  int64_t n;
  int32_t log2B;
};

// The per-tensor max_unorm reduction of the pre-pass's block partials, one
// launch in two levels: a CTA per chunk of kUnormChunk blocks of a tensor sums
// the chunk in binary64 and writes the two sums in place over the chunk's
// first two partials; the CTA that completes a tensor's last chunk (a ticket
// per tensor, zeroed by the pre-pass) adds the tensor's chunk sums in chunk
// order (a one-block chunk keeps its binary32 partial) and writes the
// multiplier.
constexpr int64_t kUnormChunk = 512;

struct FinalizeArgs {
  float2* partials;
  float* out_scale;        // indexed by DevTensor::index
  double unorm_c;          // |update direction| = unorm_c * |u|
  double max_unorm;
  int32_t ntensors;
  int64_t first_block[kMaxTensors + 1];
  int64_t first_chunk[kMaxTensors + 1];  // chunks of tensors 0..t-1
  int32_t index[kMaxTensors];
  uint64_t* stamp_clear;   // set to 0 (the carried norm's stamp), or null
  uint32_t* tickets;       // [ntensors], zero on entry
};

// Kernel launchers (defined in the kernel translation units).  Each returns
// the cudaError_t of its launch.  bits = 8 (block-wise codes) or 32.
// One optimizer's kernels (k_step_opt.cu, compiled once per optimizer): the
// step in each mode, its resident CTAs per SM, and tensor-wise
// quantization's last step (the new absmax of every tensor of a launch from
// tw_acc into its absmax arrays, tensors with an update only).
template <int OPT>
cudaError_t launch_step_opt(int bits, int dtype, int mode, const StepArgs& a, int grid, cudaStream_t s);
template <int OPT>
int ctas_step_opt(int bits, int dtype, int mode);
template <int OPT>
cudaError_t tw_store_opt(const StepArgs& a, cudaStream_t s);
#define BNB8_DECLARE_OPT(OPTV)                                                                \
  template <>                                                                                 \
  cudaError_t launch_step_opt<OPTV>(int, int, int, const StepArgs&, int, cudaStream_t);      \
  template <>                                                                                 \
  int ctas_step_opt<OPTV>(int, int, int);                                                     \
  template <>                                                                                 \
  cudaError_t tw_store_opt<OPTV>(const StepArgs&, cudaStream_t);
BNB8_DECLARE_OPT(ADAM)
BNB8_DECLARE_OPT(ADAMW)
BNB8_DECLARE_OPT(MOMENTUM)
BNB8_DECLARE_OPT(RMSPROP)
BNB8_DECLARE_OPT(ADAGRAD)
BNB8_DECLARE_OPT(LION)
BNB8_DECLARE_OPT(ADEMAMIX)
#undef BNB8_DECLARE_OPT
cudaError_t launch_quantize(int dtype, const QuantArgs& a, int grid, cudaStream_t s);
cudaError_t launch_dequantize(int dtype, const DequantArgs& a, int grid, cudaStream_t s);
cudaError_t launch_unorm_finalize(const FinalizeArgs& a, cudaStream_t s);  // both levels, one launch
cudaError_t launch_fill(float* out, int n, float v, cudaStream_t s);

// Resident CTAs per SM of a step kernel (sizes the persistent grids).
int quantize_ctas_per_sm(int dtype);

}  // namespace bnb8
