// k_quant.cu -- stand-alone block-wise quantize / dequantize, the max_unorm
// finalize reduction and a fill kernel (sm_103a).
//
// Quantize ("8-bit Optimizers via Block-wise Quantization", abstract:
// independently normalised blocks): per block of B elements, absmax = max |x|
// and code = number of map midpoints below x * (1/absmax), through the same
// shared-memory bucket table as the step kernels.  Dequantize
// ("[XPU] Implemented 8bit optimizers in triton #1692", benchmark script,
// F.dequantize_blockwise): out = qmap[code] * absmax[block].
#include "bnb8_device.cuh"

namespace bnb8 {

struct QuantSmem {
  static constexpr int kQ = 0;
  static constexpr int kMid = kQ + 256 * 4;
  static constexpr int kTbl = kMid + 256 * 4;
  static constexpr int kRed = kTbl + kTblSize * 4;
  static constexpr int kBytes = kRed + 2 * (kThreads / 32) * 4 * 4;
};

template <int DT>
__global__ void __launch_bounds__(kThreads, 2) k_quantize(const __grid_constant__ QuantArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  float* sq = reinterpret_cast<float*>(smem + QuantSmem::kQ);
  float* smid = reinterpret_cast<float*>(smem + QuantSmem::kMid);
  uint32_t* stbl = reinterpret_cast<uint32_t*>(smem + QuantSmem::kTbl);
  float* sred = reinterpret_cast<float*>(smem + QuantSmem::kRed);
  __shared__ int s_bad, s_below;
  __shared__ int s_scan[32];
  const int tid = threadIdx.x;
  for (int i = tid; i < 256; i += kThreads) sq[i] = a.qmap[i];
  if (tid == 0) s_bad = 0;
  __syncthreads();
  for (int i = tid; i < 256; i += kThreads) smid[i] = i < 255 ? (sq[i] + sq[i + 1]) * 0.5f : 0.0f;
  __syncthreads();
  build_tables<1>(smid, stbl, &s_bad, &s_below, s_scan);
  const bool fast_map = s_bad == 0;

  const int log2B = a.log2B;
  const int GT = (1 << log2B) >> 3;
  const int groups_per_cta = kThreads / GT;
  const int lane = tid & 31;
  const int glocal = tid / GT;
  const int gtid = tid & (GT - 1);
  const int64_t stride = static_cast<int64_t>(gridDim.x) * groups_per_cta;
  const int64_t warp_g0 = static_cast<int64_t>(blockIdx.x) * groups_per_cta + ((tid & ~31) / GT);
  const int in_warp = GT < 32 ? lane / GT : 0;
  const bool vec = true;  // alignment of x and codes is checked by the host for the vector path
  int parity = 0;
  for (int64_t base = warp_g0; base < a.total_blocks; base += stride) {
    const int64_t gb = base + in_warp;
    const bool active = gb < a.total_blocks;
    const int64_t e0 = (gb << log2B) + static_cast<int64_t>(gtid) * 8;
    const int64_t left = active ? a.n - e0 : 0;
    const int valid = left >= 8 ? 8 : (left > 0 ? static_cast<int>(left) : 0);
    float x[8];
    load8<DT, true>(a.x, e0, valid, vec && (reinterpret_cast<uintptr_t>(a.x) & 15) == 0, x);
    uint32_t r[1] = {0u};
#pragma unroll
    for (int j = 0; j < 8; ++j) r[0] = max(r[0], __float_as_uint(fabsf(x[j])));
    group_max_bits<1>(r, GT, glocal, reinterpret_cast<uint32_t*>(sred), parity);
    parity ^= 1;
    if (!active) continue;
    const float amax = __uint_as_float(r[0]);
    const float inv = amax > 0.0f ? __frcp_rn(amax) : 0.0f;
    uint32_t e[8];
    if (fast_map && r[0] <= 0x7f7fffffu && inv <= FLT_MAX) {
#pragma unroll
      for (int j = 0; j < 8; ++j) e[j] = encode_fast(x[j], inv, stbl + kTblZero);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) e[j] = encode_search(x[j] * inv, smid);
    }
    const uint32_t lo = __byte_perm(__byte_perm(e[0], e[1], 0x0062u), __byte_perm(e[2], e[3], 0x0062u), 0x5410u);
    const uint32_t hi = __byte_perm(__byte_perm(e[4], e[5], 0x0062u), __byte_perm(e[6], e[7], 0x0062u), 0x5410u);
    store_codes(a.codes, e0, valid, (reinterpret_cast<uintptr_t>(a.codes) & 7) == 0,
                make_uint2(lo, hi));
    if (gtid == 0) a.absmax[gb] = amax;
  }
}

template <int DT>
__global__ void __launch_bounds__(256) k_dequantize(const __grid_constant__ DequantArgs a) {
  __shared__ float sq[256];
  sq[threadIdx.x] = a.qmap[threadIdx.x];
  __syncthreads();
  const bool vec_out = (reinterpret_cast<uintptr_t>(a.out) & 15) == 0;
  const bool vec_in = (reinterpret_cast<uintptr_t>(a.codes) & 7) == 0;
  const int64_t nchunks = (a.n + 7) >> 3;
  for (int64_t c = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; c < nchunks;
       c += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t e0 = c << 3;
    const int64_t left = a.n - e0;
    const int valid = left >= 8 ? 8 : static_cast<int>(left);
    const uint2 cw = load_codes(a.codes, e0, valid, vec_in);
    const float am = a.absmax[e0 >> a.log2B];  // B >= 64: all 8 elements share a block
    float x[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) x[j] = sq[code_byte(cw, j)] * am;
    store8<DT>(a.out, e0, valid, vec_out, x);
  }
}

// One CTA per chunk of up to kUnormChunk blocks of one tensor.  Level 1: its
// binary64 sums (sum u^2, sum p^2) in a fixed order (thread i takes blocks i,
// i + 256, ...; then a tree) replace the chunk's first two partials (a chunk
// of a single block is left as it is).  Level 2, in the CTA that takes the
// tensor's last ticket: the tensor's chunk sums in the same fixed order
// (thread i takes chunks i, i + 256, ...; then a tree), and the multiplier.
__global__ void __launch_bounds__(256) k_unorm_reduce(const __grid_constant__ FinalizeArgs a) {
  __shared__ double su[256], sp[256];
  __shared__ int s_last;
  const int64_t c = blockIdx.x;
  // the tensor of chunk c: the last t with first_chunk[t] <= c
  int lo = 0, hi = a.ntensors - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (a.first_chunk[mid] <= c) lo = mid;
    else hi = mid - 1;
  }
  const int t = lo;
  auto tree = [&](double u, double p) {
    su[threadIdx.x] = u;
    sp[threadIdx.x] = p;
    __syncthreads();
    for (int o = 128; o > 0; o >>= 1) {
      if (threadIdx.x < o) {
        su[threadIdx.x] += su[threadIdx.x + o];
        sp[threadIdx.x] += sp[threadIdx.x + o];
      }
      __syncthreads();
    }
  };
  const int64_t b0 = a.first_block[t] + (c - a.first_chunk[t]) * kUnormChunk;
  const int64_t b1 = b0 + kUnormChunk < a.first_block[t + 1] ? b0 + kUnormChunk : a.first_block[t + 1];
  if (b1 - b0 >= 2) {
    double u = 0.0, p = 0.0;
    for (int64_t b = b0 + threadIdx.x; b < b1; b += blockDim.x) {
      const float2 v = a.partials[b];
      u += static_cast<double>(v.x);
      p += static_cast<double>(v.y);
    }
    tree(u, p);   // (every partial of the chunk has been read before the first barrier)
    if (threadIdx.x == 0) {
      double* out = reinterpret_cast<double*>(a.partials + b0);
      out[0] = su[0];
      out[1] = sp[0];
    }
  }
  // the ticket: the sums above are visible device-wide before it is taken
  const int64_t nchunks = a.first_chunk[t + 1] - a.first_chunk[t];
  if (threadIdx.x == 0) {
    __threadfence();
    s_last = atomicAdd(a.tickets + t, 1u) + 1u == static_cast<uint32_t>(nchunks);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  double u = 0.0, p = 0.0;
  for (int64_t k = threadIdx.x; k < nchunks; k += blockDim.x) {
    const int64_t k0 = a.first_block[t] + k * kUnormChunk;
    const int64_t k1 = k0 + kUnormChunk < a.first_block[t + 1] ? k0 + kUnormChunk : a.first_block[t + 1];
    if (k1 - k0 >= 2) {
      // written by other CTAs: read past the L1
      const double* in = reinterpret_cast<const double*>(a.partials + k0);
      u += __ldcg(in);
      p += __ldcg(in + 1);
    } else {
      const float2 v = __ldcg(a.partials + k0);
      u += static_cast<double>(v.x);
      p += static_cast<double>(v.y);
    }
  }
  tree(u, p);
  if (threadIdx.x == 0) {
    const double unorm = a.unorm_c * sqrt(su[0]);
    const double limit = a.max_unorm * sqrt(sp[0]);
    a.out_scale[a.index[t]] = (a.max_unorm > 0.0 && unorm > limit) ? static_cast<float>(limit / unorm)
                                                                    : 1.0f;
    if (t == 0 && a.stamp_clear != nullptr) *a.stamp_clear = 0ull;
  }
}

__global__ void k_fill(float* out, int n, float v) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) out[i] = v;
}

cudaError_t launch_quantize(int dtype, const QuantArgs& a, int grid, cudaStream_t s) {
  constexpr int bytes = QuantSmem::kBytes;
  static std::atomic<unsigned char> configured[3][kMaxDevices];
  const void* fn = dtype == DT_F32 ? reinterpret_cast<const void*>(k_quantize<DT_F32>)
                   : dtype == DT_BF16 ? reinterpret_cast<const void*>(k_quantize<DT_BF16>)
                                      : reinterpret_cast<const void*>(k_quantize<DT_F16>);
  const cudaError_t e = set_smem_limit_once(fn, bytes, configured[dtype]);
  if (e != cudaSuccess) return e;
  if (dtype == DT_F32) k_quantize<DT_F32><<<grid, kThreads, bytes, s>>>(a);
  else if (dtype == DT_BF16) k_quantize<DT_BF16><<<grid, kThreads, bytes, s>>>(a);
  else k_quantize<DT_F16><<<grid, kThreads, bytes, s>>>(a);
  return cudaGetLastError();
}

int quantize_ctas_per_sm(int dtype) {
  constexpr int bytes = QuantSmem::kBytes;
  const void* fn = dtype == DT_F32 ? reinterpret_cast<const void*>(k_quantize<DT_F32>)
                   : dtype == DT_BF16 ? reinterpret_cast<const void*>(k_quantize<DT_BF16>)
                                      : reinterpret_cast<const void*>(k_quantize<DT_F16>);
  cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kThreads, bytes) != cudaSuccess) return 1;
  return n > 0 ? n : 1;
}

cudaError_t launch_dequantize(int dtype, const DequantArgs& a, int grid, cudaStream_t s) {
  if (dtype == DT_F32) k_dequantize<DT_F32><<<grid, 256, 0, s>>>(a);
  else if (dtype == DT_BF16) k_dequantize<DT_BF16><<<grid, 256, 0, s>>>(a);
  else k_dequantize<DT_F16><<<grid, 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_unorm_finalize(const FinalizeArgs& a, cudaStream_t s) {
  const int64_t chunks = a.first_chunk[a.ntensors];   // >= 1 per tensor (no empty tensor)
  if (chunks <= 0) return cudaSuccess;
  k_unorm_reduce<<<static_cast<unsigned>(chunks), 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_fill(float* out, int n, float v, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  k_fill<<<(n + 255) / 256, 256, 0, s>>>(out, n, v);
  return cudaGetLastError();
}

}  // namespace bnb8
