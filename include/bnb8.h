/*
 * bnb8.h -- C ABI of the GB300 (sm_103a) 8-bit block-wise optimizer library.
 *
 * The library implements one hot path: the optimizer step with 8-bit
 * block-wise dynamically quantized states, as described by
 *   - "8-bit Optimizers via Block-wise Quantization" (Dettmers et al.),
 *     abstract: block-wise quantization (independently normalised blocks of
 *     B elements) with a dynamic, non-linear data type;
 *   - bitsandbytes docs "optim_overview.md": Optimizer2State /
 *     Optimizer1State parameters (lr, betas, eps, weight_decay,
 *     min_8bit_size, max_unorm, skip_zeros, alpha, t_alpha, t_beta3);
 *   - "[XPU] Implemented 8bit optimizers in triton #1692", benchmark script:
 *     the per-parameter state tensors state1/qmap1/absmax1 and
 *     state2/qmap2/absmax2, the AdEMAMix m1_m2 stacking, and
 *     F.dequantize_blockwise(code, absmax, A, blocksize);
 *   - "Support skip_zeros in the XPU Triton optimizer kernels #2097":
 *     skip_zeros semantics (raw gradient tested before weight decay).
 *
 * Conventions shared by every entry point
 *   - Every function returns an int status (enum bnb8_status).  On failure
 *     bnb8_last_error() returns a message for the calling thread.  No
 *     exception or abort crosses this boundary.
 *   - Device work is enqueued asynchronously on the caller's stream
 *     (a cudaStream_t, passed as struct CUstream_st*; NULL = legacy default
 *     stream).  No function synchronizes the device.  BNB8_ECUDA reports a
 *     launch error; errors raised later by the device surface on the stream.
 *   - The caller owns every buffer.  The library allocates no device or host
 *     memory that outlives a call; scratch comes from a caller-provided
 *     workspace (bnb8_workspace_size).  The exceptions are the fixed
 *     scratch array behind bnb8_unorm_static and the paged buffers that
 *     bnb8_paged_alloc hands to the caller (see there).
 *   - Pointers marked "device" must be device-accessible memory of the
 *     current device.  Calls are reentrant; calls on different streams that
 *     touch the same buffers race, as with any CUDA kernel.
 *   - Element counts are int64_t; a tensor with n == 0 is skipped.
 *   - Dtypes: BNB8_F32 (IEEE binary32), BNB8_BF16 (bfloat16), BNB8_F16
 *     (IEEE binary16).  All arithmetic is binary32; a value is rounded to its
 *     storage dtype once, to nearest even.
 *   - Block sizes: a power of two from 64 to 4096.  The last block of a
 *     tensor may be partial.  The step functions also take blocksize 0:
 *     tensor-wise quantization, one absmax per state per tensor.
 */
#ifndef BNB8_H
#define BNB8_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* the type behind cudaStream_t */

enum bnb8_status {
  BNB8_OK = 0,
  BNB8_EINVAL = 1,       /* bad argument: null pointer, size, dtype, block size, optimizer */
  BNB8_EUNSUPPORTED = 2, /* valid request this build does not implement */
  BNB8_ECUDA = 3,        /* a CUDA runtime call or kernel launch failed */
  BNB8_EWORKSPACE = 4    /* workspace missing, misaligned or smaller than required */
};

enum bnb8_dtype { BNB8_F32 = 0, BNB8_BF16 = 1, BNB8_F16 = 2 };

enum bnb8_optim {
  BNB8_ADAM = 0,     /* 2-state; weight decay coupled into the gradient (torch.optim.Adam) */
  BNB8_ADAMW = 1,    /* 2-state; decoupled weight decay (torch.optim.AdamW) */
  BNB8_MOMENTUM = 2, /* 1-state; SGD with momentum beta1, no dampening */
  BNB8_RMSPROP = 3,  /* 1-state; smoothing constant alpha = beta1 */
  BNB8_ADAGRAD = 4,  /* 1-state */
  BNB8_LION = 5,     /* 1-state; decoupled weight decay */
  BNB8_ADEMAMIX = 6  /* two EMAs of g (m1, m2) and nu; decoupled weight decay */
};

/* One parameter tensor and its optimizer state (all device pointers).
 *   p        parameter, n elements of hparams.dtype, updated in place.
 *   g        gradient, n elements of the same dtype, read only.
 *   s1, s2   state arrays.  state_bits == 8: uint8 codes; state_bits == 32:
 *            binary32 values.  2-state optimizers: s1 = first moment
 *            (qmap1), s2 = second moment (qmap2).  1-state: s1 only.
 *            AdEMAMix: s1 holds m1 then m2 ([2, n], both on qmap1),
 *            s2 holds nu (qmap2).  Unused slots may be NULL.
 *   absmax1, absmax2
 *            state_bits == 8 only: binary32 per-block scales, ceil(n/B)
 *            entries for s2 and for 1-/2-state s1; AdEMAMix absmax1 is
 *            [2, ceil(n/B)] (m1 scales, then m2 scales).
 *   n        number of elements.
 *   state_bits  8 (block-wise dynamic quantization) or 32 (binary32 states;
 *            the docs page's min_8bit_size rule keeps tensors below 4096
 *            elements at 32 bits -- the caller picks per tensor).
 * Zero states: codes equal to the code of 0.0 in their map
 * (bnb8_qmap_code(qmap, 0.0f, &code)) with absmax 0, or binary32 zeros.
 * Alignment: any element alignment is accepted; p/g/state arrays aligned to
 * 16 bytes (codes: 8 bytes, AdEMAMix needs n % 8 == 0 for the m2 half) take
 * the vectorised path. */
typedef struct bnb8_tensor {
  void* p;
  const void* g;
  void* s1;
  void* s2;
  float* absmax1;
  float* absmax2;
  int64_t n;
  int32_t state_bits;
  int32_t reserved; /* must be 0 */
} bnb8_tensor;

/* Hyperparameters of one update, shared by every tensor of a call.
 *   optim       enum bnb8_optim; must match the entry point.
 *   dtype       enum bnb8_dtype of p and g.
 *   blocksize   B, a power of two in [64, 4096]; or 0: tensor-wise 8-bit
 *               states ("8-bit Optimizers via Block-wise Quantization"
 *               compares block-wise against this), one absmax per state per
 *               tensor (absmax1/absmax2 hold 1 value; AdEMAMix absmax1 = [2]).
 *               A first pass finds each tensor's new absmax, the step then
 *               requantizes with it; needs a workspace (bnb8_workspace_size);
 *               BNB8_UNORM_PER_BLOCK is BNB8_EINVAL with it.
 *   skip_zeros  nonzero: where the raw gradient is exactly 0 the parameter
 *               and its states keep their values; a block whose gradient is
 *               all zero keeps its codes and absmax bit-identical.
 *   lr, beta1, beta2, eps, weight_decay   as on the docs page.
 *   beta3, alpha, t_alpha, t_beta3        AdEMAMix only (t_* == 0: no
 *               warm-up schedule).
 *   gnorm_scale multiplies the raw gradient (1.0 = off).
 *   max_unorm   0 = off.  Otherwise, per tensor, if ||update direction|| >
 *               max_unorm * ||p|| the step is scaled down to that norm (a
 *               pre-pass over g, p and the states; needs a workspace).
 *   flags       0, or BNB8_UNORM_PER_BLOCK: max_unorm taken per block of
 *               blocksize elements instead of per tensor ("optim_overview.md":
 *               the maximum value to normalize each block with, read
 *               literally): each block whose ||update direction|| exceeds
 *               max_unorm * ||p of the block|| is scaled down to it.  The
 *               norms are formed inside the step (no pre-pass, no workspace);
 *               the multiplier matches the binary64 definition to 1e-6.
 *               BNB8_CARRY_PNORM, BNB8_TEST_STALL_WAIT: see enum bnb8_flags.
 *               Other bits: BNB8_EINVAL.
 *   step        1-based number of this update (bias corrections, schedules). */
typedef struct bnb8_hparams {
  int32_t optim;
  int32_t dtype;
  int32_t blocksize;
  int32_t skip_zeros;
  float lr, beta1, beta2, beta3, alpha, eps, weight_decay, gnorm_scale, max_unorm;
  int32_t flags; /* 0 or BNB8_UNORM_PER_BLOCK, BNB8_CARRY_PNORM, BNB8_TEST_STALL_WAIT */
  int64_t step;
  int64_t t_alpha;
  int64_t t_beta3;
} bnb8_hparams;

enum bnb8_flags {
  BNB8_UNORM_PER_BLOCK = 1, /* max_unorm per block instead of per tensor */
  /* With max_unorm per tensor: the step also leaves, in the workspace, the
   * per-block sums of the squares of the NEW parameters, stamped with the
   * tensor list (its p pointers, sizes, state bits, block size, dtype and
   * optimizer) and the step number.  The next call with step + 1, the same
   * list and the same workspace finds the stamp and takes ||p|| for its
   * max_unorm test from those sums: it reads no p for the norm, and none at
   * all in the pre-pass when the update direction does not depend on p
   * (decoupled weight decay, or weight_decay 0).  Any other call recomputes
   * the norm; every pre-pass (bnb8_unorm included) clears the stamp, so a
   * workspace shared between lists or calls only loses the shortcut.  The
   * caller must not change p between the two calls, and a step that raised
   * BNB8_STATUS_WAIT_TIMEOUT leaves no usable sums.  The sums are binary32
   * per block, as the pre-pass forms them, but in the step's own summation
   * order: the multiplier matches the binary64 definition to 1e-6 either
   * way.  Tensor-wise steps (blocksize 0) and skip_zeros steps ignore the
   * flag. */
  BNB8_CARRY_PNORM = 2,
  /* Test hook of the bounded waits (not for training): in a plain step
   * (no skip_zeros, blocksize >= 256, max_unorm off or per tensor) one warp
   * of the step kernel withholds one of its own asynchronous copies, so its
   * wait for that copy runs out after 1 s.  The kernel then records
   * BNB8_STATUS_WAIT_TIMEOUT in the device status (bnb8_device_status) and
   * returns normally; the blocks of that warp are left partly or wholly
   * unstepped.  No other flag bit is defined. */
  BNB8_TEST_STALL_WAIT = 0x100
};

/* Message describing the last failure on this thread ("" if none). */
const char* bnb8_last_error(void);

/* Bits of the device status word. */
enum bnb8_device_status_bits {
  /* a step kernel's bounded wait for one of its asynchronous copies ran out
   * (1 s); the call's results are incomplete */
  BNB8_STATUS_WAIT_TIMEOUT = 1
};

/* The library keeps one 32-bit status word per device (a variable of the
 * library's device code): the step kernels or-in enum bnb8_device_status_bits
 * when a device-side wait gives up, instead of hanging or trapping.  This
 * call copies the current device's word to *status (host), after the device
 * has finished its work (it synchronizes the device), and zeroes the word if
 * clear is nonzero.  Errors: BNB8_EINVAL (status NULL), BNB8_ECUDA. */
int bnb8_device_status(uint32_t* status, int clear);

/* Library version, major * 10000 + minor * 100 + patch. */
int bnb8_version(void);

/* Fill out[256] (host memory) with the dynamic quantization map, ascending.
 * Data type ("8-bit Optimizers via Block-wise Quantization", abstract, and the
 * citing description of dynamic exponent types): a sign bit (signed map
 * only), k zero bits giving the exponent 10^-k, an indicator bit, then f
 * fraction bits whose 2^f codes are the midpoints of 2^f equal steps of
 * [0.1, 1].  Signed: k = 0..6, f = 6-k, plus 0 and +1.0.  Unsigned: k = 0..6,
 * f = 7-k, plus 0 and +1.0.  Formed in binary64, rounded once.
 * Returns BNB8_EINVAL if out is NULL. */
int bnb8_create_qmap(int is_signed, float* out);

/* The code the nearest-level rule of block-wise quantization gives a
 * normalised value x under a map (host): the number of map midpoints
 * fl((qmap[j] + qmap[j+1]) * 0.5), j = 0..254, strictly below x (the nearest
 * level, ties to the lower one) -- the rule bnb8_quantize_blockwise and the
 * step functions apply to every value ("8-bit Optimizers via Block-wise
 * Quantization", abstract: a value is stored as the index of its level in the
 * dynamic data type).  Its use is the initial state: an all-zero state is
 * the code of 0.0 in every element, for whatever map the caller steps with.
 *   qmap   256 binary32 values, strictly ascending (host memory).
 *   x      the value; code receives its code.
 * Errors: BNB8_EINVAL if qmap or code is NULL, x is NaN, or qmap is not
 * strictly ascending. */
int bnb8_qmap_code(const float* qmap, float x, uint8_t* code);

/* Block-wise quantization (device): for each block of B elements of x,
 * absmax[b] = max |x| over the block and codes[i] = the number of map
 * midpoints (q[j] + q[j+1]) / 2 strictly below x[i] * (1 / absmax[b])
 * (nearest level, ties to the lower one; 0 / absmax 0 for an all-zero block).
 * A NaN in a block makes its absmax NaN (the IEEE 754-2019 maximum); the
 * block is then normalised by 0 as an all-zero block is, so its values take
 * the code of 0 and the NaN code 0.
 *   x       n elements of dtype.
 *   qmap    256 binary32 map values, strictly ascending (device).
 *   codes   n uint8 (device, written).   absmax  ceil(n/B) binary32 (written).
 * Errors: BNB8_EINVAL for null pointers (n > 0), n < 0, bad dtype or B. */
int bnb8_quantize_blockwise(const void* x, int dtype, int64_t n, const float* qmap, int blocksize,
                            uint8_t* codes, float* absmax, struct CUstream_st* stream);

/* Block-wise dequantization (device), the inverse used by
 * F.dequantize_blockwise(code, absmax, A, blocksize): out[i] =
 * qmap[codes[i]] * absmax[i / B], rounded once to dtype. */
int bnb8_dequantize_blockwise(const uint8_t* codes, const float* absmax, const float* qmap,
                              int blocksize, int64_t n, void* out, int dtype,
                              struct CUstream_st* stream);

/* Bytes of workspace the step functions and bnb8_unorm need for this tensor
 * list: the per-tensor max_unorm pre-pass's stamp, multipliers, partials and
 * the reduction's tickets (hp->max_unorm > 0 without BNB8_UNORM_PER_BLOCK)
 * plus 16 bytes per tensor for tensor-wise
 * quantization (hp->blocksize 0); 0 when neither applies.  Returns 0 and
 * sets the error message on invalid arguments. */
size_t bnb8_workspace_size(const bnb8_tensor* tensors, int ntensors, const bnb8_hparams* hp);

/* One optimizer update of every tensor in the list (host array of
 * descriptors; the list is read during the call only).
 * Per element, in binary32, each operation rounded once; a product that is
 * added (x*y + z below) is one fused multiply-add, rounded once:
 *   g = g_raw * gnorm_scale; if coupled decay and wd != 0: g = wd*p + g
 *   Adam/AdamW  m = b1*m + ((1-b1)*g);  v = b2*v + ((1-b2)*(g*g));
 *               u = m / (sqrt(v) + eps*sqrt(1-b2^t));  step = lr*sqrt(1-b2^t)/(1-b1^t)
 *   decoupled decay and wd != 0: p = p * (1 - lr*wd)
 *   p = -(step * clip)*u + p
 * 8-bit states are dequantized (qmap[code] * absmax), updated, and
 * requantized with a fresh per-block absmax (NaN when a new state of the
 * block is NaN, as in bnb8_quantize_blockwise) after p is written from the
 * unquantized new states.  skip_zeros and max_unorm as in bnb8_hparams.
 *   qmap1, qmap2  device maps (256 binary32, ascending) for s1 and s2 of
 *                 8-bit tensors; unused for 32-bit tensors.
 *   workspace     device scratch of at least bnb8_workspace_size() bytes,
 *                 256-byte aligned; may be NULL when that size is 0.
 * Errors: BNB8_EINVAL (bad descriptor or hparams, hp->optim not ADAM/ADAMW),
 * BNB8_EWORKSPACE, BNB8_ECUDA. */
int bnb8_step_2state(const bnb8_tensor* tensors, int ntensors, const bnb8_hparams* hp,
                     const float* qmap1, const float* qmap2, void* workspace,
                     size_t workspace_bytes, struct CUstream_st* stream);

/* 1-state update (MOMENTUM, RMSPROP, ADAGRAD, LION); qmap1 is the map of s1
 * (signed for Momentum and Lion, unsigned for RMSprop and Adagrad).
 *   Momentum  m = b1*m + g;  u = m;                         step = lr
 *   RMSprop   v = b1*v + (1-b1)*g*g;  u = g/(sqrt(v) + eps); step = lr
 *   Adagrad   v = v + g*g;  u = g/(sqrt(v) + eps);           step = lr
 *   Lion      c = b1*m + (1-b1)*g;  u = sign(c);  m = b2*m + (1-b2)*g;  step = lr
 * Momentum, RMSprop and Adagrad couple weight decay into g; Lion decouples.
 * Other arguments and errors as bnb8_step_2state. */
int bnb8_step_1state(const bnb8_tensor* tensors, int ntensors, const bnb8_hparams* hp,
                     const float* qmap1, void* workspace, size_t workspace_bytes,
                     struct CUstream_st* stream);

/* AdEMAMix update: m1 = b1*m1 + (1-b1)*g;  m2 = b3_t*m2 + (1-b3_t)*g;
 * nu = b2*nu + (1-b2)*g*g;
 * u = (m1 / (1-b1^t) + alpha_t*m2) / (sqrt(nu) + eps*sqrt(1-b2^t));
 * step = lr*sqrt(1-b2^t); decoupled decay.  alpha_t = min(t*alpha/t_alpha,
 * alpha) and b3_t = min(exp(ln b1 ln b3 / ((1-t/T) ln b3 + (t/T) ln b1)), b3)
 * with T = t_beta3 (no schedule when t_alpha / t_beta3 are 0).  m1 and m2
 * share qmap1 (s1 = [2, n], absmax1 = [2, nblocks]); nu uses qmap2. */
int bnb8_step_ademamix(const bnb8_tensor* tensors, int ntensors, const bnb8_hparams* hp,
                       const float* qmap1, const float* qmap2, void* workspace,
                       size_t workspace_bytes, struct CUstream_st* stream);

/* The max_unorm pre-pass on its own (per-tensor reading; hp->flags with
 * BNB8_UNORM_PER_BLOCK is BNB8_EINVAL here): writes, for every tensor i of the list,
 * out_scale[i] (device binary32) = the step multiplier the update would use
 * (max_unorm * ||p|| / ||d|| if ||d|| > max_unorm * ||p||, else 1), where d
 * is the update direction of this step without lr and without decoupled
 * decay (Adam: u*sqrt(1-b2^t)/(1-b1^t); AdEMAMix: u*sqrt(1-b2^t); 1-state:
 * u) and skipped elements contribute 0.  Nothing else is written.
 * qmap2 may be NULL for 1-state optimizers.  Needs a workspace of
 * bnb8_workspace_size() bytes computed with this hp (max_unorm > 0). */
int bnb8_unorm(const bnb8_tensor* tensors, int ntensors, const bnb8_hparams* hp,
               const float* qmap1, const float* qmap2, float* out_scale, void* workspace,
               size_t workspace_bytes, struct CUstream_st* stream);

/* bnb8_unorm without a workspace, for callers that cannot allocate device
 * memory: for example code whose device memory is all handed out by a host
 * framework's pool that must see every allocation, or a hot loop where a
 * cudaMalloc / cudaFree would stall the device.  This entry point calls no
 * allocator; its scratch (the per-block partial norms of up to 262,144
 * blocks, 2 MiB, and the reduction's tickets) is a fixed array compiled into
 * the library, which every GPU that loads the library holds until the process
 * exits.  The paper has no counterpart: this is a deployment variant of
 * bnb8_unorm.
 *   Same arguments, results and errors as bnb8_unorm, minus the workspace.
 *   A list with more than 262,144 blocks (over all tensors, at hp->blocksize)
 *   is rejected with BNB8_EWORKSPACE.
 *   The first call on a device looks up the array's device address (once per
 *   device, with that device current); make that first call before any stream
 *   capture on the device.
 *   All calls on a device share the one array, so calls whose work overlaps
 *   on the GPU (different streams, no ordering between them) race and give
 *   undefined results; calls on one stream, or otherwise ordered, are safe.
 *   Each call writes every partial it reads before reading it, so whatever an
 *   earlier call left in the array does not matter. */
int bnb8_unorm_static(const bnb8_tensor* tensors, int ntensors, const bnb8_hparams* hp,
                      const float* qmap1, const float* qmap2, float* out_scale,
                      struct CUstream_st* stream);

/* Paged optimizer state ("optim_overview.md": the is_paged argument of the
 * optimizers; "[XPU] Implemented 8bit optimizers in triton #1692", benchmark
 * script: PagedAdam8bit, PagedAdamW8bit, PagedLion8bit, PagedAdEMAMix8bit):
 * state arrays (s1, s2, absmax1, absmax2) in CUDA managed memory, which the
 * driver pages between host and device memory under device-memory pressure,
 * so that states larger than free device memory still step.  The step functions take such arrays
 * unchanged (any device-accessible pointer); these three calls allocate,
 * place and free them.  They need a device with concurrent managed access
 * (cudaDevAttrConcurrentManagedAccess), else BNB8_EUNSUPPORTED. */

/* *out = `bytes` of managed memory (cudaMallocManaged, attached globally),
 * for the current device; contents undefined.  The caller frees it with
 * bnb8_paged_free.  Errors: BNB8_EINVAL (out NULL, bytes 0),
 * BNB8_EUNSUPPORTED, BNB8_ECUDA (out of memory among others). */
int bnb8_paged_alloc(size_t bytes, void** out);

/* Migrates [ptr, ptr + bytes) of a bnb8_paged_alloc buffer, asynchronously
 * on `stream`, to device `device` (an ordinal >= 0), or to host memory for
 * device == BNB8_PAGED_HOST.  The paged optimizers call it for every state
 * array, to the device, before each step on the step's stream, so the step
 * kernel finds its pages resident instead of faulting them in one by one.
 * Migration is a placement hint: the data stay valid wherever they live.
 * bytes == 0 does nothing.  Errors: BNB8_EINVAL (ptr NULL with bytes > 0,
 * device < -1), BNB8_EUNSUPPORTED, BNB8_ECUDA. */
int bnb8_paged_prefetch(const void* ptr, size_t bytes, int device, struct CUstream_st* stream);

enum { BNB8_PAGED_HOST = -1 };

/* Frees a bnb8_paged_alloc buffer (NULL: nothing).  Like cudaFree, it waits
 * for the device to finish work that may use the buffer. */
int bnb8_paged_free(void* ptr);

#ifdef __cplusplus
}
#endif

#endif /* BNB8_H */
