// bnb8_api.cu -- the C ABI of include/bnb8.h: argument validation, per-step
// scalars (binary64, rounded once), tensor lists split into 8-bit and 32-bit
// launches, workspace layout, and the kernel launches.  Host code is built
// with -ffp-contract=off so every scalar below is one fixed expression.
#include <cuda_runtime.h>

#include <atomic>
#include <climits>
#include <cmath>
#include <cstdarg>
#include <cstddef>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "bnb8.h"
#include "bnb8_internal.h"

using namespace bnb8;

namespace {

thread_local std::string g_last_error;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(BNB8_ECUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int elem_size(int dtype) { return dtype == BNB8_F32 ? 4 : 2; }

bool valid_dtype(int dtype) { return dtype == BNB8_F32 || dtype == BNB8_BF16 || dtype == BNB8_F16; }

int log2_blocksize(int blocksize) {
  for (int l = 6; l <= 12; ++l)
    if (blocksize == (1 << l)) return l;
  return -1;
}

int nstates(int optim) {
  if (optim == BNB8_ADAM || optim == BNB8_ADAMW) return 2;
  if (optim == BNB8_ADEMAMIX) return 3;
  return 1;
}

int nmaps(int optim) {
  return (optim == BNB8_ADAM || optim == BNB8_ADAMW || optim == BNB8_ADEMAMIX) ? 2 : 1;
}

// SM count of the current device (cached per device; a larger ordinal than
// the cache holds is queried on every call).
int sm_count() {
  static std::atomic<int> cache[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 1;
  const bool cached = dev < kMaxDevices;
  if (cached) {
    const int c = cache[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
  if (cached) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

// ---- per-step scalars -------------------------------------------------------
// Adam / AdamW: lr/(1-b1^t) * m/(sqrt(v)/sqrt(1-b2^t) + eps) is evaluated as
// step_size * m/(sqrt(v) + eps_hat) with step_size = lr*sqrt(bc2)/bc1 and
// eps_hat = eps*sqrt(bc2).  AdEMAMix (alpha and beta3 warm-up of the AdEMAMix
// optimizer, t_alpha / t_beta3 on the docs page): alpha_t = min(t*alpha/T_a,
// alpha), beta3_t = min(exp(ln b1 ln b3 / ((1 - t/T_b) ln b3 + (t/T_b) ln b1)), b3).
struct Scalars {
  float b1, b2, b3t, omb1, omb2, omb3t, step_size, eps_hat, inv_bc1, alpha_t, decay;
  double unorm_c;
};

Scalars make_scalars(const bnb8_hparams& hp) {
  Scalars s;
  std::memset(&s, 0, sizeof(s));
  const double t = static_cast<double>(hp.step);
  const double b1 = hp.beta1, b2 = hp.beta2, b3 = hp.beta3;
  const double lr = hp.lr, eps = hp.eps, wd = hp.weight_decay;
  const double bc1 = 1.0 - std::pow(b1, t);
  const double bc2 = 1.0 - std::pow(b2, t);
  s.b1 = hp.beta1;
  s.b2 = hp.beta2;
  s.omb1 = static_cast<float>(1.0 - b1);
  s.omb2 = static_cast<float>(1.0 - b2);
  s.decay = static_cast<float>(1.0 - lr * wd);
  s.step_size = hp.lr;
  s.eps_hat = hp.eps;
  s.unorm_c = 1.0;
  if (hp.optim == BNB8_ADAM || hp.optim == BNB8_ADAMW) {
    s.step_size = static_cast<float>(lr * std::sqrt(bc2) / bc1);
    s.eps_hat = static_cast<float>(eps * std::sqrt(bc2));
    s.unorm_c = std::sqrt(bc2) / bc1;
  } else if (hp.optim == BNB8_ADEMAMIX) {
    const double alpha = hp.alpha;
    double at = alpha;
    if (hp.t_alpha > 0) {
      const double ramp = t * alpha / static_cast<double>(hp.t_alpha);
      at = ramp < alpha ? ramp : alpha;
    }
    double b3t = b3;
    if (hp.t_beta3 > 0) {
      const double r = t / static_cast<double>(hp.t_beta3);
      const double lb1 = std::log(b1), lb3 = std::log(b3);
      const double v = std::exp(lb1 * lb3 / ((1.0 - r) * lb3 + r * lb1));
      b3t = v < b3 ? v : b3;
    }
    s.alpha_t = static_cast<float>(at);
    s.b3t = static_cast<float>(b3t);
    s.omb3t = static_cast<float>(1.0 - static_cast<double>(s.b3t));
    s.inv_bc1 = static_cast<float>(1.0 / bc1);
    s.step_size = static_cast<float>(lr * std::sqrt(bc2));
    s.eps_hat = static_cast<float>(eps * std::sqrt(bc2));
    s.unorm_c = std::sqrt(bc2);
  }
  return s;
}

int check_hparams(const bnb8_hparams* hp, const int* allowed, int nallowed, int* log2B) {
  if (hp == nullptr) return fail(BNB8_EINVAL, "hparams is NULL");
  bool ok = false;
  for (int i = 0; i < nallowed; ++i) ok = ok || hp->optim == allowed[i];
  if (!ok) return fail(BNB8_EINVAL, "optimizer %d not handled by this entry point", hp->optim);
  if (!valid_dtype(hp->dtype)) return fail(BNB8_EINVAL, "unknown dtype %d", hp->dtype);
  // blocksize 0: tensor-wise quantization (one absmax per state per tensor);
  // the kernels then cut each tensor into groups of 256 elements for work
  *log2B = hp->blocksize == 0 ? 8 : log2_blocksize(hp->blocksize);
  if (*log2B < 0)
    return fail(BNB8_EINVAL, "blocksize %d is neither 0 nor a power of two in [64, 4096]",
                hp->blocksize);
  if (hp->blocksize == 0 && (hp->flags & BNB8_UNORM_PER_BLOCK) != 0)
    return fail(BNB8_EINVAL, "BNB8_UNORM_PER_BLOCK needs blocks (blocksize 0 is tensor-wise)");
  const int known = BNB8_UNORM_PER_BLOCK | BNB8_CARRY_PNORM | BNB8_TEST_STALL_WAIT;
  if ((hp->flags & ~known) != 0)
    return fail(BNB8_EINVAL, "hparams.flags: unknown bits 0x%x", hp->flags & ~known);
  if (hp->step < 1) return fail(BNB8_EINVAL, "step must be >= 1 (got %lld)", (long long)hp->step);
  if (hp->t_alpha < 0 || hp->t_beta3 < 0) return fail(BNB8_EINVAL, "t_alpha / t_beta3 must be >= 0");
  if (!(hp->max_unorm >= 0.0f) || std::isinf(hp->max_unorm))
    return fail(BNB8_EINVAL, "max_unorm must be finite and >= 0");
  return BNB8_OK;
}

// Validate one descriptor; sets *vec to DevTensor::vec_ok's bits: 1 if every
// stream is aligned for the vector path, 3 if also for whole-chunk bulk copies.
int check_tensor(const bnb8_tensor& t, int i, const bnb8_hparams& hp, int* vec) {
  if (t.n < 0) return fail(BNB8_EINVAL, "tensor %d: n < 0", i);
  if (t.reserved != 0) return fail(BNB8_EINVAL, "tensor %d: reserved must be 0", i);
  if (t.state_bits != 8 && t.state_bits != 32)
    return fail(BNB8_EINVAL, "tensor %d: state_bits must be 8 or 32 (got %d)", i, t.state_bits);
  if (t.n > (int64_t(1) << 50)) return fail(BNB8_EINVAL, "tensor %d: n too large", i);
  *vec = 0;
  if (t.n == 0) return BNB8_OK;
  const int ns = nstates(hp.optim);
  const int es = elem_size(hp.dtype);
  if (t.p == nullptr || t.g == nullptr || t.s1 == nullptr)
    return fail(BNB8_EINVAL, "tensor %d: p, g and s1 must not be NULL", i);
  if (ns >= 2 && t.s2 == nullptr) return fail(BNB8_EINVAL, "tensor %d: s2 must not be NULL", i);
  if (!aligned(t.p, es) || !aligned(t.g, es))
    return fail(BNB8_EINVAL, "tensor %d: p and g must be aligned to their element size", i);
  if (t.state_bits == 8) {
    if (t.absmax1 == nullptr || (ns >= 2 && nmaps(hp.optim) == 2 && t.absmax2 == nullptr))
      return fail(BNB8_EINVAL, "tensor %d: absmax arrays must not be NULL for 8-bit state", i);
    if (!aligned(t.absmax1, 4) || (t.absmax2 != nullptr && !aligned(t.absmax2, 4)))
      return fail(BNB8_EINVAL, "tensor %d: absmax arrays must be 4-byte aligned", i);
  } else {
    if (!aligned(t.s1, 4) || (t.s2 != nullptr && !aligned(t.s2, 4)))
      return fail(BNB8_EINVAL, "tensor %d: 32-bit states must be 4-byte aligned", i);
  }
  bool v = aligned(t.p, 16) && aligned(t.g, 16);
  bool bulk = false;
  if (t.state_bits == 8) {
    // bulk copies of whole chunks want 16-byte aligned code streams too
    // (AdEMAMix's m2 half starts n bytes into s1)
    bulk = v && aligned(t.s1, 16) && (ns < 2 || aligned(t.s2, 16)) &&
           (hp.optim != BNB8_ADEMAMIX || t.n % 16 == 0);
    v = v && aligned(t.s1, 8) && (ns < 2 || aligned(t.s2, 8));
    if (hp.optim == BNB8_ADEMAMIX) v = v && (t.n % 8 == 0);
  } else {
    v = v && aligned(t.s1, 16) && (ns < 2 || aligned(t.s2, 16));
    if (hp.optim == BNB8_ADEMAMIX) v = v && (t.n % 4 == 0);
  }
  *vec = v ? (bulk ? 3 : 1) : 0;
  return BNB8_OK;
}

struct Plan {
  struct Chunk {
    int bits;
    std::vector<int> idx;          // positions in the caller's list
    int64_t total_blocks = 0;
    int64_t partial_offset = 0;    // first block in the workspace partials
  };
  std::vector<Chunk> chunks;
  std::vector<char> vec;
  int64_t all_blocks = 0;
};

int make_plan(const bnb8_tensor* ts, int nt, const bnb8_hparams& hp, int log2B,
              const float* qmap1, const float* qmap2, Plan* plan) {
  if (nt < 0) return fail(BNB8_EINVAL, "ntensors < 0");
  if (nt > 0 && ts == nullptr) return fail(BNB8_EINVAL, "tensors is NULL");
  plan->vec.assign(nt, 0);
  bool any8 = false;
  for (int i = 0; i < nt; ++i) {
    int v = 0;
    const int rc = check_tensor(ts[i], i, hp, &v);
    if (rc != BNB8_OK) return rc;
    plan->vec[i] = static_cast<char>(v);
    if (ts[i].n > 0 && ts[i].state_bits == 8) any8 = true;
  }
  if (any8) {
    if (qmap1 == nullptr || (nmaps(hp.optim) == 2 && qmap2 == nullptr))
      return fail(BNB8_EINVAL, "8-bit tensors need qmap1%s", nmaps(hp.optim) == 2 ? " and qmap2" : "");
    if (!aligned(qmap1, 4) || (qmap2 != nullptr && !aligned(qmap2, 4)))
      return fail(BNB8_EINVAL, "qmaps must be 4-byte aligned");
  }
  // 8-bit tensors whose chunks are all whole for the ring step (aligned, a
  // multiple of max(512, B) elements) are launched apart from the others,
  // so that their launches take the ring's whole-chunk variant
  const int64_t unit = int64_t(1) << (log2B > 9 ? log2B : 9);
  auto whole = [&](int i) { return plan->vec[i] == 3 && ts[i].n % unit == 0; };
  int64_t offset = 0;
  for (int bits : {8, 32}) {
    for (int group = 0; group < (bits == 8 ? 2 : 1); ++group) {
      Plan::Chunk cur;
      cur.bits = bits;
      for (int i = 0; i < nt; ++i) {
        if (ts[i].n == 0 || ts[i].state_bits != bits) continue;
        if (bits == 8 && whole(i) != (group == 0)) continue;
        if (static_cast<int>(cur.idx.size()) == kMaxTensors) {
          cur.partial_offset = offset;
          offset += cur.total_blocks;
          plan->chunks.push_back(cur);
          cur = Plan::Chunk();
          cur.bits = bits;
        }
        cur.idx.push_back(i);
        cur.total_blocks += (ts[i].n + (int64_t(1) << log2B) - 1) >> log2B;
      }
      if (!cur.idx.empty()) {
        cur.partial_offset = offset;
        offset += cur.total_blocks;
        plan->chunks.push_back(cur);
      }
    }
  }
  plan->all_blocks = offset;
  // the 8-bit kernels index the blocks of one launch with 32-bit integers (a
  // list that fits in HBM is far below the limit at B >= 64)
  for (const Plan::Chunk& c : plan->chunks)
    if (c.total_blocks > INT32_MAX)
      return fail(BNB8_EUNSUPPORTED, "%lld blocks in one launch (at most %d)",
                  static_cast<long long>(c.total_blocks), INT32_MAX);
  return BNB8_OK;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// The library's device status word (one per device that loads the library):
// kernels or-in kStatus* bits, bnb8_device_status reads and clears it.
__device__ uint32_t g_device_status;

// Device address of g_device_status on the current device, looked up once per
// device (atomics: host threads may race on the first call) and cached.
int device_status_addr(uint32_t** out) {
  static std::atomic<uint32_t*> addr[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  const bool cached = dev >= 0 && dev < kMaxDevices;
  uint32_t* a = cached ? addr[dev].load(std::memory_order_acquire) : nullptr;
  if (a == nullptr) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_device_status);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(device status)");
    a = static_cast<uint32_t*>(ptr);
    if (cached) addr[dev].store(a, std::memory_order_release);
  }
  *out = a;
  return BNB8_OK;
}

// Bound of every wait for an async copy inside the step kernels.
constexpr uint64_t kWaitLimitNs = 1000000000ull;

// Workspace layout when the per-tensor pre-pass runs: [the carried norm's
// stamp, in its own 256 bytes][per-tensor max_unorm multipliers][per-block
// partials][the reduction's tickets, one word per tensor of a launch]; then
// [4 words per tensor] of tensor-wise absmax accumulators when blocksize is
// 0.  The stamp sits at the same place for every tensor list, so any call
// that reuses the workspace for another list replaces it.
constexpr size_t kStampBytes = 256;
constexpr size_t kTicketBytes = (kMaxTensors * sizeof(uint32_t) + 255) / 256 * 256;
size_t partials_offset(int nt) { return kStampBytes + align256(static_cast<size_t>(nt) * sizeof(float)); }
size_t tickets_offset(int nt, int64_t all_blocks) {
  return partials_offset(nt) + align256(static_cast<size_t>(all_blocks) * sizeof(float2));
}
size_t workspace_bytes_for(int nt, int64_t all_blocks) { return tickets_offset(nt, all_blocks) + kTicketBytes; }

// The carried norm's stamp: a hash of the tensor list and the settings that
// shape its partials (FNV-1a over 64-bit words), mixed with a step number.
uint64_t list_hash(const bnb8_tensor* ts, int nt, const bnb8_hparams& hp) {
  uint64_t h = 0xcbf29ce484222325ull;
  auto mix = [&](uint64_t v) {
    for (int i = 0; i < 8; ++i) {
      h ^= (v >> (8 * i)) & 0xffu;
      h *= 0x100000001b3ull;
    }
  };
  mix(static_cast<uint64_t>(hp.optim));
  mix(static_cast<uint64_t>(hp.dtype));
  mix(static_cast<uint64_t>(hp.blocksize));
  mix(static_cast<uint64_t>(nt));
  for (int i = 0; i < nt; ++i) {
    mix(reinterpret_cast<uintptr_t>(ts[i].p));
    mix(static_cast<uint64_t>(ts[i].n));
    mix(static_cast<uint64_t>(ts[i].state_bits));
  }
  return h;
}
uint64_t carry_stamp_for(uint64_t list, int64_t step) {
  uint64_t z = list ^ (static_cast<uint64_t>(step) * 0x9e3779b97f4a7c15ull);
  z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
  z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
  return (z ^ (z >> 31)) | 1ull;  // never 0, the contents of a cleared workspace
}
size_t tw_bytes_for(int nt) { return align256(static_cast<size_t>(nt) * 4 * sizeof(uint32_t)); }

StepArgs make_args(const Plan::Chunk& c, const bnb8_tensor* ts, const Plan& plan,
                   const bnb8_hparams& hp, const Scalars& sc, int log2B, const float* qmap1,
                   const float* qmap2) {
  StepArgs a;
  std::memset(&a, 0, sizeof(a));
  a.b1 = sc.b1;
  a.b2 = sc.b2;
  a.b3t = sc.b3t;
  a.omb1 = sc.omb1;
  a.omb2 = sc.omb2;
  a.omb3t = sc.omb3t;
  a.step_size = sc.step_size;
  a.eps_hat = sc.eps_hat;
  a.inv_bc1 = sc.inv_bc1;
  a.alpha_t = sc.alpha_t;
  a.decay = sc.decay;
  a.wd = hp.weight_decay;
  a.gscale = hp.gnorm_scale;
  a.max_unorm = hp.max_unorm;
  a.unorm_c = static_cast<float>(sc.unorm_c);
  a.skip_zeros = hp.skip_zeros != 0;
  a.zero_ratio = sc.eps_hat > 0.0f && std::isfinite(sc.eps_hat) && std::isfinite(sc.b1) &&
                 std::isfinite(sc.b2) && std::isfinite(sc.omb1) && std::isfinite(sc.omb2) &&
                 std::isfinite(hp.gnorm_scale);
  a.tensorwise = hp.blocksize == 0 ? 1 : 0;
  a.nsm = sm_count();
  a.stall_test = (hp.flags & BNB8_TEST_STALL_WAIT) != 0 ? 1 : 0;
  a.wait_ns = kWaitLimitNs;
  a.log2B = log2B;
  a.ntensors = static_cast<int32_t>(c.idx.size());
  a.total_blocks = c.total_blocks;
  a.qmap1 = qmap1;
  a.qmap2 = qmap2;
  int64_t fb = 0;
  a.whole = 1;
  a.ring_units = 0;
  const int log2U = log2B > 9 ? log2B : 9;  // a ring unit: max(512, B) elements
  const int64_t unit = int64_t(1) << log2U;
  for (size_t k = 0; k < c.idx.size(); ++k) {
    const bnb8_tensor& t = ts[c.idx[k]];
    DevTensor& d = a.t[k];
    d.p = t.p;
    d.g = t.g;
    d.s1 = t.s1;
    d.s2 = t.s2;
    d.a1 = t.absmax1;
    d.a2 = t.absmax2;
    d.n = t.n;
    d.first_block = fb;
    d.index = c.idx[k];
    d.vec_ok = plan.vec[c.idx[k]];
    d.nblocks = static_cast<int32_t>((t.n + (int64_t(1) << log2B) - 1) >> log2B);
    d.units = static_cast<int32_t>((t.n + unit - 1) >> log2U);
    a.ring_units += d.units;
    if (d.vec_ok != 3 || t.n % unit != 0) a.whole = 0;
    fb += d.nblocks;
  }
  return a;
}

cudaError_t launch_family(int bits, int optim, int dtype, int mode, const StepArgs& a, int grid,
                          cudaStream_t s) {
  switch (optim) {
    case BNB8_ADAM: return launch_step_opt<ADAM>(bits, dtype, mode, a, grid, s);
    case BNB8_ADAMW: return launch_step_opt<ADAMW>(bits, dtype, mode, a, grid, s);
    case BNB8_MOMENTUM: return launch_step_opt<MOMENTUM>(bits, dtype, mode, a, grid, s);
    case BNB8_RMSPROP: return launch_step_opt<RMSPROP>(bits, dtype, mode, a, grid, s);
    case BNB8_ADAGRAD: return launch_step_opt<ADAGRAD>(bits, dtype, mode, a, grid, s);
    case BNB8_LION: return launch_step_opt<LION>(bits, dtype, mode, a, grid, s);
    case BNB8_ADEMAMIX: return launch_step_opt<ADEMAMIX>(bits, dtype, mode, a, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t tw_store_family(int optim, const StepArgs& a, cudaStream_t s) {
  switch (optim) {
    case BNB8_ADAM: return tw_store_opt<ADAM>(a, s);
    case BNB8_ADAMW: return tw_store_opt<ADAMW>(a, s);
    case BNB8_MOMENTUM: return tw_store_opt<MOMENTUM>(a, s);
    case BNB8_RMSPROP: return tw_store_opt<RMSPROP>(a, s);
    case BNB8_ADAGRAD: return tw_store_opt<ADAGRAD>(a, s);
    case BNB8_LION: return tw_store_opt<LION>(a, s);
    case BNB8_ADEMAMIX: return tw_store_opt<ADEMAMIX>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

int grid_for(int bits, int optim, int dtype, int mode, int64_t total_blocks, int log2B) {
  // resident CTAs per SM of each kernel (the same on every device of a process)
  static std::atomic<int> cache[2][7][3][5];
  std::atomic<int>& slot = cache[bits == 8 ? 0 : 1][optim][dtype][mode];
  int c = slot.load(std::memory_order_relaxed);
  if (c == 0) {
    switch (optim) {
      case BNB8_ADAM: c = ctas_step_opt<ADAM>(bits, dtype, mode); break;
      case BNB8_ADAMW: c = ctas_step_opt<ADAMW>(bits, dtype, mode); break;
      case BNB8_MOMENTUM: c = ctas_step_opt<MOMENTUM>(bits, dtype, mode); break;
      case BNB8_RMSPROP: c = ctas_step_opt<RMSPROP>(bits, dtype, mode); break;
      case BNB8_ADAGRAD: c = ctas_step_opt<ADAGRAD>(bits, dtype, mode); break;
      case BNB8_LION: c = ctas_step_opt<LION>(bits, dtype, mode); break;
      default: c = ctas_step_opt<ADEMAMIX>(bits, dtype, mode); break;
    }
    slot.store(c, std::memory_order_relaxed);
  }
  const int groups_per_cta = kThreads / ((1 << log2B) >> 3);
  const int64_t need = (total_blocks + groups_per_cta - 1) / groups_per_cta;
  const int64_t persistent = static_cast<int64_t>(sm_count()) * c;
  return static_cast<int>(need < persistent ? need : persistent);
}

// max_unorm pre-pass + finalize into out_scale[caller index].  fill: every
// entry of out_scale is first set to 1 (the caller reads the multipliers of
// empty tensors too); the step reads only those of the tensors it updates,
// which the finalize writes, and skips that launch.
int run_unorm(const Plan& plan, const bnb8_tensor* ts, int nt, const bnb8_hparams& hp,
              const Scalars& sc, int log2B, const float* qmap1, const float* qmap2,
              float* out_scale, float2* partials, uint32_t* tickets, cudaStream_t stream, bool fill,
              uint64_t* stamp = nullptr, uint64_t carry_expect = 0) {
  cudaError_t e = fill ? launch_fill(out_scale, nt, 1.0f, stream) : cudaSuccess;  // n == 0 tensors keep 1
  if (e != cudaSuccess) return cuda_fail(e, "unorm fill");
  for (size_t ci = 0; ci < plan.chunks.size(); ++ci) {
    const Plan::Chunk& c = plan.chunks[ci];
    StepArgs a = make_args(c, ts, plan, hp, sc, log2B, qmap1, qmap2);
    a.partials = partials + c.partial_offset;
    // carry_expect 0: no carried norm (a stamp is never 0)
    a.carry_stamp = carry_expect != 0 ? stamp : nullptr;
    a.carry_expect = carry_expect;
    a.tickets = tickets;   // zeroed by the pre-pass for the reduction that follows
    const int grid = grid_for(c.bits, hp.optim, hp.dtype, MODE_NORM, c.total_blocks, log2B);
    e = launch_family(c.bits, hp.optim, hp.dtype, MODE_NORM, a, grid, stream);
    if (e != cudaSuccess) return cuda_fail(e, "unorm pre-pass launch");
    FinalizeArgs f;
    std::memset(&f, 0, sizeof(f));
    f.partials = a.partials;
    f.out_scale = out_scale;
    f.unorm_c = sc.unorm_c;
    f.max_unorm = hp.max_unorm;
    f.ntensors = a.ntensors;
    f.tickets = tickets;
    // these partials no longer hold a carried norm: the last finalize clears
    // the stamp (a step that carries the norm writes a new one after it)
    f.stamp_clear = ci + 1 == plan.chunks.size() ? stamp : nullptr;
    int64_t chunks = 0;
    for (int k = 0; k < a.ntensors; ++k) {
      f.first_block[k] = a.t[k].first_block;
      f.first_chunk[k] = chunks;
      f.index[k] = a.t[k].index;
      const int64_t nb = (k + 1 < a.ntensors ? a.t[k + 1].first_block : c.total_blocks) -
                         a.t[k].first_block;
      chunks += (nb + kUnormChunk - 1) / kUnormChunk;
    }
    f.first_block[a.ntensors] = c.total_blocks;
    f.first_chunk[a.ntensors] = chunks;
    e = launch_unorm_finalize(f, stream);
    if (e != cudaSuccess) return cuda_fail(e, "unorm finalize launch");
  }
  (void)nt;
  return BNB8_OK;
}

int step_common(const bnb8_tensor* ts, int nt, const bnb8_hparams* hp, const int* allowed,
                int nallowed, const float* qmap1, const float* qmap2, void* ws, size_t ws_bytes,
                cudaStream_t stream) {
  int log2B = 0;
  int rc = check_hparams(hp, allowed, nallowed, &log2B);
  if (rc != BNB8_OK) return rc;
  Plan plan;
  rc = make_plan(ts, nt, *hp, log2B, qmap1, qmap2, &plan);
  if (rc != BNB8_OK) return rc;
  if (plan.chunks.empty()) return BNB8_OK;
  const Scalars sc = make_scalars(*hp);
  const float* clip = nullptr;
  // per-block max_unorm: the norms are formed inside the step itself
  const bool per_block = hp->max_unorm > 0.0f && (hp->flags & BNB8_UNORM_PER_BLOCK) != 0;
  const int mode = per_block ? MODE_BCLIP : MODE_STEP;
  const bool prepass = hp->max_unorm > 0.0f && !per_block;
  const bool tw = hp->blocksize == 0;
  const size_t need = (prepass ? workspace_bytes_for(nt, plan.all_blocks) : 0) + (tw ? tw_bytes_for(nt) : 0);
  if (need > 0 && (ws == nullptr || !aligned(ws, 256) || ws_bytes < need))
    return fail(BNB8_EWORKSPACE, "%s needs a 256-byte aligned workspace of %zu bytes (got %zu)",
                prepass ? "max_unorm" : "tensor-wise quantization", need, ws_bytes);
  uint32_t* status = nullptr;
  rc = device_status_addr(&status);
  if (rc != BNB8_OK) return rc;
  uint32_t* tw_acc = tw ? reinterpret_cast<uint32_t*>(
                              static_cast<char*>(ws) + (prepass ? workspace_bytes_for(nt, plan.all_blocks) : 0))
                        : nullptr;
  float2* partials = nullptr;
  uint64_t* stamp = nullptr;      // the carried norm's stamp (workspace offset 0)
  // no carry with blocksize 0 (tensor-wise steps leave no per-block sums) or
  // with skip_zeros (a skipped block reads no p, so it could not leave its sum)
  const bool carry = prepass && !tw && hp->skip_zeros == 0 && (hp->flags & BNB8_CARRY_PNORM) != 0;
  const uint64_t list = carry ? list_hash(ts, nt, *hp) : 0;
  if (prepass) {
    float* scales = reinterpret_cast<float*>(static_cast<char*>(ws) + kStampBytes);
    partials = reinterpret_cast<float2*>(static_cast<char*>(ws) + partials_offset(nt));
    stamp = static_cast<uint64_t*>(ws);
    uint32_t* tickets = reinterpret_cast<uint32_t*>(static_cast<char*>(ws) + tickets_offset(nt, plan.all_blocks));
    rc = run_unorm(plan, ts, nt, *hp, sc, log2B, qmap1, qmap2, scales, partials, tickets, stream, false, stamp,
                   carry ? carry_stamp_for(list, hp->step - 1) : 0);
    if (rc != BNB8_OK) return rc;
    clip = scales;
  }
  if (tw) {
    // tensor-wise: the new absmax of every state of every 8-bit tensor first
    cudaError_t e = launch_fill(reinterpret_cast<float*>(tw_acc), 4 * nt, 0.0f, stream);
    if (e != cudaSuccess) return cuda_fail(e, "tensor-wise fill");
    for (const Plan::Chunk& c : plan.chunks) {
      if (c.bits != 8) continue;
      StepArgs a = make_args(c, ts, plan, *hp, sc, log2B, qmap1, qmap2);
      a.clip = clip;
      a.tw_acc = tw_acc;
      const int grid = grid_for(8, hp->optim, hp->dtype, MODE_TWMAX, c.total_blocks, log2B);
      e = launch_family(8, hp->optim, hp->dtype, MODE_TWMAX, a, grid, stream);
      if (e != cudaSuccess) return cuda_fail(e, "tensor-wise max launch");
    }
  }
  for (size_t ci = 0; ci < plan.chunks.size(); ++ci) {
    const Plan::Chunk& c = plan.chunks[ci];
    StepArgs a = make_args(c, ts, plan, *hp, sc, log2B, qmap1, qmap2);
    a.clip = clip;
    a.tw_acc = tw_acc;
    a.status = status;
    if (carry) {
      // every launch leaves its blocks' sums of p^2; the last one stamps them
      a.carry_out = 1;
      a.partials = partials + c.partial_offset;
      a.carry_stamp = stamp;
      a.carry_writer = ci + 1 == plan.chunks.size() ? 1 : 0;
      a.carry_write = carry_stamp_for(list, hp->step);
    }
    const int m = (tw && c.bits == 8) ? MODE_TWSTEP : mode;
    const int grid = grid_for(c.bits, hp->optim, hp->dtype, m, c.total_blocks, log2B);
    const cudaError_t e = launch_family(c.bits, hp->optim, hp->dtype, m, a, grid, stream);
    if (e != cudaSuccess) return cuda_fail(e, "step launch");
  }
  if (tw) {
    // the new absmax is stored once every CTA has dequantized with the old
    for (const Plan::Chunk& c : plan.chunks) {
      if (c.bits != 8) continue;
      StepArgs a = make_args(c, ts, plan, *hp, sc, log2B, qmap1, qmap2);
      a.tw_acc = tw_acc;
      const cudaError_t e = tw_store_family(hp->optim, a, stream);
      if (e != cudaSuccess) return cuda_fail(e, "tensor-wise store launch");
    }
  }
  return BNB8_OK;
}

}  // namespace

extern "C" {

const char* bnb8_last_error(void) { return g_last_error.c_str(); }

int bnb8_version(void) { return 300; }  // 0.3.0: paged state

// Dynamic map (see include/bnb8.h).  Levels are emitted directly in ascending
// order: the negative levels from the largest magnitude down, zero, the
// positive levels from the smallest up, then +1.0.
int bnb8_create_qmap(int is_signed, float* out) {
  if (out == nullptr) return fail(BNB8_EINVAL, "out is NULL");
  static const double kPow10[7] = {1.0, 10.0, 100.0, 1000.0, 10000.0, 100000.0, 1000000.0};
  auto level = [](int k, int f, int nfrac) {
    return (0.1 + (static_cast<double>(f) + 0.5) * (0.9 / nfrac)) / kPow10[k];
  };
  int i = 0;
  if (is_signed) {
    for (int k = 0; k <= 6; ++k) {
      const int nfrac = 1 << (6 - k);
      for (int f = nfrac - 1; f >= 0; --f) out[i++] = static_cast<float>(-level(k, f, nfrac));
    }
    out[i++] = 0.0f;
    for (int k = 6; k >= 0; --k) {
      const int nfrac = 1 << (6 - k);
      for (int f = 0; f < nfrac; ++f) out[i++] = static_cast<float>(level(k, f, nfrac));
    }
  } else {
    out[i++] = 0.0f;
    for (int k = 6; k >= 0; --k) {
      const int nfrac = 1 << (7 - k);
      for (int f = 0; f < nfrac; ++f) out[i++] = static_cast<float>(level(k, f, nfrac));
    }
  }
  out[i++] = 1.0f;
  return i == 256 ? BNB8_OK : fail(BNB8_EUNSUPPORTED, "internal: map has %d levels", i);
}

// Nearest-level code on the host: the count of binary32 midpoints below x,
// each midpoint formed as (q[j] + q[j+1]) * 0.5 with one rounding per
// operation, as the kernels form them.
int bnb8_qmap_code(const float* qmap, float x, uint8_t* code) {
  if (qmap == nullptr || code == nullptr) return fail(BNB8_EINVAL, "qmap and code must not be NULL");
  if (std::isnan(x)) return fail(BNB8_EINVAL, "x is NaN");
  for (int j = 0; j < 255; ++j)
    if (!(qmap[j] < qmap[j + 1]))
      return fail(BNB8_EINVAL, "qmap is not strictly ascending at index %d", j);
  int c = 0;
  for (int j = 0; j < 255; ++j) {
    const float mid = (qmap[j] + qmap[j + 1]) * 0.5f;
    if (mid < x) ++c;
  }
  *code = static_cast<uint8_t>(c);
  return BNB8_OK;
}

int bnb8_quantize_blockwise(const void* x, int dtype, int64_t n, const float* qmap, int blocksize,
                            uint8_t* codes, float* absmax, struct CUstream_st* stream) {
  if (!valid_dtype(dtype)) return fail(BNB8_EINVAL, "unknown dtype %d", dtype);
  const int log2B = log2_blocksize(blocksize);
  if (log2B < 0) return fail(BNB8_EINVAL, "blocksize %d is not a power of two in [64, 4096]", blocksize);
  if (n < 0) return fail(BNB8_EINVAL, "n < 0");
  if (n == 0) return BNB8_OK;
  if (x == nullptr || qmap == nullptr || codes == nullptr || absmax == nullptr)
    return fail(BNB8_EINVAL, "x, qmap, codes and absmax must not be NULL");
  if (!aligned(x, elem_size(dtype)) || !aligned(absmax, 4) || !aligned(qmap, 4))
    return fail(BNB8_EINVAL, "x, qmap or absmax misaligned");
  QuantArgs a;
  a.x = x;
  a.codes = codes;
  a.absmax = absmax;
  a.qmap = qmap;
  a.n = n;
  a.total_blocks = (n + blocksize - 1) >> log2B;
  a.log2B = log2B;
  const int groups_per_cta = kThreads / (blocksize >> 3);
  const int64_t need = (a.total_blocks + groups_per_cta - 1) / groups_per_cta;
  const int64_t persistent = static_cast<int64_t>(sm_count()) * quantize_ctas_per_sm(dtype);
  const int grid = static_cast<int>(need < persistent ? need : persistent);
  const cudaError_t e = launch_quantize(dtype, a, grid, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? BNB8_OK : cuda_fail(e, "quantize launch");
}

int bnb8_dequantize_blockwise(const uint8_t* codes, const float* absmax, const float* qmap,
                              int blocksize, int64_t n, void* out, int dtype,
                              struct CUstream_st* stream) {
  if (!valid_dtype(dtype)) return fail(BNB8_EINVAL, "unknown dtype %d", dtype);
  const int log2B = log2_blocksize(blocksize);
  if (log2B < 0) return fail(BNB8_EINVAL, "blocksize %d is not a power of two in [64, 4096]", blocksize);
  if (n < 0) return fail(BNB8_EINVAL, "n < 0");
  if (n == 0) return BNB8_OK;
  if (codes == nullptr || absmax == nullptr || qmap == nullptr || out == nullptr)
    return fail(BNB8_EINVAL, "codes, absmax, qmap and out must not be NULL");
  if (!aligned(out, elem_size(dtype)) || !aligned(absmax, 4) || !aligned(qmap, 4))
    return fail(BNB8_EINVAL, "out, qmap or absmax misaligned");
  DequantArgs a;
  a.codes = codes;
  a.absmax = absmax;
  a.qmap = qmap;
  a.out = out;
  a.n = n;
  a.log2B = log2B;
  const int64_t chunks = (n + 7) >> 3;
  const int64_t need = (chunks + 255) / 256;
  const int64_t cap = static_cast<int64_t>(sm_count()) * 8;
  const int grid = static_cast<int>(need < cap ? need : cap);
  const cudaError_t e = launch_dequantize(dtype, a, grid, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? BNB8_OK : cuda_fail(e, "dequantize launch");
}

size_t bnb8_workspace_size(const bnb8_tensor* tensors, int ntensors, const bnb8_hparams* hp) {
  static const int all[] = {BNB8_ADAM, BNB8_ADAMW, BNB8_MOMENTUM, BNB8_RMSPROP,
                            BNB8_ADAGRAD, BNB8_LION, BNB8_ADEMAMIX};
  int log2B = 0;
  if (check_hparams(hp, all, 7, &log2B) != BNB8_OK) return 0;
  const bool prepass = hp->max_unorm > 0.0f && (hp->flags & BNB8_UNORM_PER_BLOCK) == 0;
  const bool tw = hp->blocksize == 0;
  if (!prepass && !tw) return 0;
  if (ntensors < 0 || (ntensors > 0 && tensors == nullptr)) {
    fail(BNB8_EINVAL, "bad tensor list");
    return 0;
  }
  int64_t blocks = 0;
  for (int i = 0; i < ntensors; ++i) {
    if (tensors[i].n < 0) {
      fail(BNB8_EINVAL, "tensor %d: n < 0", i);
      return 0;
    }
    blocks += (tensors[i].n + (int64_t(1) << log2B) - 1) >> log2B;
  }
  return (prepass ? workspace_bytes_for(ntensors, blocks) : 0) + (tw ? tw_bytes_for(ntensors) : 0);
}

int bnb8_device_status(uint32_t* status, int clear) {
  if (status == nullptr) return fail(BNB8_EINVAL, "status is NULL");
  *status = 0u;
  uint32_t* addr = nullptr;
  int rc = device_status_addr(&addr);
  if (rc != BNB8_OK) return rc;
  cudaError_t e = cudaMemcpy(status, addr, sizeof(uint32_t), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "reading the device status");
  if (clear) {
    e = cudaMemset(addr, 0, sizeof(uint32_t));
    if (e != cudaSuccess) return cuda_fail(e, "clearing the device status");
    e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "clearing the device status");
  }
  return BNB8_OK;
}

int bnb8_step_2state(const bnb8_tensor* tensors, int ntensors, const bnb8_hparams* hp,
                     const float* qmap1, const float* qmap2, void* workspace,
                     size_t workspace_bytes, struct CUstream_st* stream) {
  static const int allowed[] = {BNB8_ADAM, BNB8_ADAMW};
  return step_common(tensors, ntensors, hp, allowed, 2, qmap1, qmap2, workspace, workspace_bytes,
                     reinterpret_cast<cudaStream_t>(stream));
}

int bnb8_step_1state(const bnb8_tensor* tensors, int ntensors, const bnb8_hparams* hp,
                     const float* qmap1, void* workspace, size_t workspace_bytes,
                     struct CUstream_st* stream) {
  static const int allowed[] = {BNB8_MOMENTUM, BNB8_RMSPROP, BNB8_ADAGRAD, BNB8_LION};
  return step_common(tensors, ntensors, hp, allowed, 4, qmap1, nullptr, workspace,
                     workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

int bnb8_step_ademamix(const bnb8_tensor* tensors, int ntensors, const bnb8_hparams* hp,
                       const float* qmap1, const float* qmap2, void* workspace,
                       size_t workspace_bytes, struct CUstream_st* stream) {
  static const int allowed[] = {BNB8_ADEMAMIX};
  return step_common(tensors, ntensors, hp, allowed, 1, qmap1, qmap2, workspace, workspace_bytes,
                     reinterpret_cast<cudaStream_t>(stream));
}

int bnb8_unorm(const bnb8_tensor* tensors, int ntensors, const bnb8_hparams* hp,
               const float* qmap1, const float* qmap2, float* out_scale, void* workspace,
               size_t workspace_bytes, struct CUstream_st* stream) {
  static const int all[] = {BNB8_ADAM, BNB8_ADAMW, BNB8_MOMENTUM, BNB8_RMSPROP,
                            BNB8_ADAGRAD, BNB8_LION, BNB8_ADEMAMIX};
  int log2B = 0;
  int rc = check_hparams(hp, all, 7, &log2B);
  if (rc != BNB8_OK) return rc;
  if ((hp->flags & BNB8_UNORM_PER_BLOCK) != 0)
    return fail(BNB8_EINVAL, "the max_unorm pre-pass computes per-tensor multipliers; "
                             "BNB8_UNORM_PER_BLOCK has none");
  if (ntensors > 0 && out_scale == nullptr) return fail(BNB8_EINVAL, "out_scale is NULL");
  if (out_scale != nullptr && !aligned(out_scale, 4)) return fail(BNB8_EINVAL, "out_scale misaligned");
  Plan plan;
  rc = make_plan(tensors, ntensors, *hp, log2B, qmap1, qmap2, &plan);
  if (rc != BNB8_OK) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (hp->max_unorm <= 0.0f || plan.chunks.empty()) {
    const cudaError_t e = launch_fill(out_scale, ntensors, 1.0f, s);
    return e == cudaSuccess ? BNB8_OK : cuda_fail(e, "unorm fill");
  }
  const size_t need = workspace_bytes_for(ntensors, plan.all_blocks);
  if (workspace == nullptr || !aligned(workspace, 256) || workspace_bytes < need)
    return fail(BNB8_EWORKSPACE, "unorm needs a 256-byte aligned workspace of %zu bytes (got %zu)",
                need, workspace_bytes);
  float2* partials = reinterpret_cast<float2*>(static_cast<char*>(workspace) + partials_offset(ntensors));
  uint32_t* tickets =
      reinterpret_cast<uint32_t*>(static_cast<char*>(workspace) + tickets_offset(ntensors, plan.all_blocks));
  const Scalars sc = make_scalars(*hp);
  return run_unorm(plan, tensors, ntensors, *hp, sc, log2B, qmap1, qmap2, out_scale, partials, tickets, s, true,
                   static_cast<uint64_t*>(workspace));
}

}  // extern "C"

// ---------------------------------------------------------------------------
// bnb8_unorm_static: bnb8_unorm for callers that cannot allocate device
// memory.  The per-block partial norms live in one file-scope device array
// instead of a caller workspace.  Every GPU that loads this library holds the
// array (2 MiB) until the process exits; all calls on a device share it.
// ---------------------------------------------------------------------------
namespace {

constexpr int64_t kStaticScratchBlocks = int64_t(1) << 18;  // float2 partials: 2 MiB

struct StaticScratch {
  float2 partials[kStaticScratchBlocks];
  uint32_t tickets[kMaxTensors];
};
__device__ __align__(256) StaticScratch g_static_scratch;

// Device address of g_static_scratch on the current device, looked up once per
// device (with that device current) and cached.  Host code must not use the
// array's name as a pointer: on the host it only stands in for the symbol.
// The cache entries are atomics: host threads making their first call on a
// device at the same time both look the address up and store the same value.
int static_scratch(StaticScratch** out) {
  static std::atomic<StaticScratch*> addr[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices)
    return fail(BNB8_EUNSUPPORTED, "device ordinal %d out of range", dev);
  StaticScratch* a = addr[dev].load(std::memory_order_acquire);
  if (a == nullptr) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_static_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static scratch)");
    a = static_cast<StaticScratch*>(ptr);
    addr[dev].store(a, std::memory_order_release);
  }
  *out = a;
  return BNB8_OK;
}

}  // namespace

extern "C" int bnb8_unorm_static(const bnb8_tensor* tensors, int ntensors, const bnb8_hparams* hp,
                                 const float* qmap1, const float* qmap2, float* out_scale,
                                 struct CUstream_st* stream) {
  static const int all[] = {BNB8_ADAM, BNB8_ADAMW, BNB8_MOMENTUM, BNB8_RMSPROP,
                            BNB8_ADAGRAD, BNB8_LION, BNB8_ADEMAMIX};
  int log2B = 0;
  int rc = check_hparams(hp, all, 7, &log2B);
  if (rc != BNB8_OK) return rc;
  if ((hp->flags & BNB8_UNORM_PER_BLOCK) != 0)
    return fail(BNB8_EINVAL, "the max_unorm pre-pass computes per-tensor multipliers; "
                             "BNB8_UNORM_PER_BLOCK has none");
  if (ntensors > 0 && out_scale == nullptr) return fail(BNB8_EINVAL, "out_scale is NULL");
  if (out_scale != nullptr && !aligned(out_scale, 4)) return fail(BNB8_EINVAL, "out_scale misaligned");
  Plan plan;
  rc = make_plan(tensors, ntensors, *hp, log2B, qmap1, qmap2, &plan);
  if (rc != BNB8_OK) return rc;
  if (hp->max_unorm > 0.0f && plan.all_blocks > kStaticScratchBlocks)
    return fail(BNB8_EWORKSPACE,
                "bnb8_unorm_static handles at most %lld blocks per call (this list has %lld); "
                "use bnb8_unorm with a workspace",
                (long long)kStaticScratchBlocks, (long long)plan.all_blocks);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (hp->max_unorm <= 0.0f || plan.chunks.empty()) {
    const cudaError_t e = launch_fill(out_scale, ntensors, 1.0f, s);
    return e == cudaSuccess ? BNB8_OK : cuda_fail(e, "unorm fill");
  }
  StaticScratch* scratch = nullptr;
  rc = static_scratch(&scratch);
  if (rc != BNB8_OK) return rc;
  // every partial a call reads is written by the same call's pre-pass first,
  // and the pre-pass zeroes the tickets, so the contents left by an earlier
  // call need no clearing
  const Scalars sc = make_scalars(*hp);
  char* base = reinterpret_cast<char*>(scratch);   // a device address: offsets only
  return run_unorm(plan, tensors, ntensors, *hp, sc, log2B, qmap1, qmap2, out_scale,
                   reinterpret_cast<float2*>(base + offsetof(StaticScratch, partials)),
                   reinterpret_cast<uint32_t*>(base + offsetof(StaticScratch, tickets)), s, true);
}

// ---------------------------------------------------------------------------
// Paged state: state arrays in CUDA managed memory, which the driver pages
// between host and device memory; the step kernels read them like any other
// device-accessible memory.  Placement is by explicit prefetch on the step's
// stream.
// ---------------------------------------------------------------------------
namespace {

// BNB8_OK if device `dev` can page managed memory while kernels run
// (concurrent managed access), which the prefetch and the paged buffers need.
int check_managed(int dev) {
  int cma = 0;
  const cudaError_t e = cudaDeviceGetAttribute(&cma, cudaDevAttrConcurrentManagedAccess, dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(concurrent managed access)");
  if (cma == 0) return fail(BNB8_EUNSUPPORTED, "device %d has no concurrent managed access", dev);
  return BNB8_OK;
}

}  // namespace

extern "C" {

int bnb8_paged_alloc(size_t bytes, void** out) {
  if (out == nullptr) return fail(BNB8_EINVAL, "out is NULL");
  *out = nullptr;
  if (bytes == 0) return fail(BNB8_EINVAL, "bytes is 0");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  const int rc = check_managed(dev);
  if (rc != BNB8_OK) return rc;
  void* p = nullptr;
  e = cudaMallocManaged(&p, bytes, cudaMemAttachGlobal);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMallocManaged");
  *out = p;
  return BNB8_OK;
}

int bnb8_paged_prefetch(const void* ptr, size_t bytes, int device, struct CUstream_st* stream) {
  if (bytes == 0) return BNB8_OK;
  if (ptr == nullptr) return fail(BNB8_EINVAL, "ptr is NULL");
  if (device < BNB8_PAGED_HOST) return fail(BNB8_EINVAL, "device %d is neither an ordinal nor BNB8_PAGED_HOST", device);
  int dev = device;
  if (dev == BNB8_PAGED_HOST) {
    const cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  }
  const int rc = check_managed(dev);
  if (rc != BNB8_OK) return rc;
  cudaMemLocation loc;
  std::memset(&loc, 0, sizeof(loc));
  loc.type = device == BNB8_PAGED_HOST ? cudaMemLocationTypeHost : cudaMemLocationTypeDevice;
  loc.id = device == BNB8_PAGED_HOST ? 0 : device;
  const cudaError_t e =
      cudaMemPrefetchAsync(ptr, bytes, loc, 0, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemPrefetchAsync");
  return BNB8_OK;
}

int bnb8_paged_free(void* ptr) {
  if (ptr == nullptr) return BNB8_OK;
  const cudaError_t e = cudaFree(ptr);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFree(paged)");
  return BNB8_OK;
}

}  // extern "C"
