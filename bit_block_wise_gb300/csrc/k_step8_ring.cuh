// k_step8_ring.cuh -- the fused 8-bit block-wise optimizer step with a
// per-warp asynchronous-copy ring (sm_103a; MODE_STEP without skip_zeros,
// blocks of 256 elements or more).
//
// The step moves about 16 bytes per element and computes on every one, so
// it is held back less by arithmetic than by how many bytes each SM keeps in
// flight.  Here every warp owns a two-stage ring in shared memory: while it
// computes on one 256-element chunk, the bulk copy engine (cp.async.bulk,
// completion counted on an mbarrier) is already bringing in p, g and the
// code streams of its next two chunks, so the registers hold only the chunk
// being computed.  One CTA of up to 32 warps runs per SM; its first copies
// are issued before the map tables are built, so the table build overlaps
// the first loads.
//
// Arithmetic, per element and per block, is the same as k_step8's packed
// path ("8-bit Optimizers via Block-wise Quantization", abstract: blocks
// quantized independently, in parallel): dequantize through the map in
// shared memory times the block absmax, update in binary32, store p, reduce
// the new absmax (one warp per 256 elements; warps of a larger block meet at
// a named barrier), requantize through the bucket table.
//
// Element mapping inside a chunk (chosen so that every global store of a
// warp covers one contiguous span): 32-bit p/g -- lane l holds elements
// 4l..4l+3 and 128+4l..128+4l+3; 16-bit p/g -- elements 8l..8l+7.  A lane's
// eight codes per state follow its elements.
//
// Every wait is bounded: a copy that does not land within StepArgs::wait_ns
// sets BNB8_STATUS_WAIT_TIMEOUT in *StepArgs::status, and the warp stops
// computing, lets its copies still in flight land (again bounded) and keeps
// only its part in the block barriers of its group.
#pragma once

#include "bnb8_device.cuh"

namespace bnb8 {

// ---------------------------------------------------------------------------
// async-copy and mbarrier primitives (inline PTX)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes) : "memory");
}
// global -> shared bulk copy; bytes and both addresses 16-byte aligned
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
// one more arrival on bar once this thread's earlier cp.async copies have landed
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0u;
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Wait for the phase of `parity` to complete, for at most limit_ns.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_ns() - t0 > limit_ns) return false;
  return true;
}

// ---------------------------------------------------------------------------
// geometry and shared memory layout
// ---------------------------------------------------------------------------
// A warp takes 512 elements (a chunk) per iteration, in one of three shapes:
//  SH_TWO (blocksize 256): two passes of 8 elements a lane, one block each;
//         24 warps of up to 80 registers.
//  SH_BIG (blocksize >= 512, where the park fits): two passes of 8 elements
//         a lane of one block, the first pass's new states parked in shared
//         memory until the block's absmax is known; 24 warps.
//  SH_ONE (blocksize >= 512 otherwise): one pass of 16 elements a lane; 16
//         warps of up to 128 registers.
// Either way the per-chunk work (the wait, the copies of the next chunk,
// the chunk's bookkeeping) is paid once per 512 elements.
constexpr int kChunk = 512;                              // elements per warp and iteration
constexpr int kLog2Chunk = 9;
template <bool SEQ>
struct RingShape {
  static constexpr int kWarps = SEQ ? 24 : 16;
  static constexpr int kPasses = SEQ ? 2 : 1;
  static constexpr int kQuads = SEQ ? 2 : 4;             // quads of 4 elements a lane per pass
  static constexpr int kNE = 4 * kQuads;                 // elements a lane per pass
};
enum RingShapeId { SH_ONE = 0, SH_TWO = 1, SH_BIG = 2 };
// Warps per CTA: the two-pass shapes run 24 warps of at most 80 registers,
// AdEMAMix (three states) 20 warps of at most 96; the one-pass shape 16 of
// at most 128.
template <int OPT, int SH>
__host__ __device__ constexpr int ring_warps() {
  return SH == SH_ONE ? 16 : (OPT == ADEMAMIX ? 20 : 24);
}
template <int OPT, int DT, int SH>
struct RingSmem {
  static constexpr bool SEQ = SH != SH_ONE;
  static constexpr int NS = Traits<OPT>::NS;
  static constexpr int NM = Traits<OPT>::NM;
  static constexpr int ES = DT == DT_F32 ? 4 : 2;
  // one stage: p | g | codes of each state | absmax | header
  static constexpr int kSP = 0;
  static constexpr int kSG = kSP + kChunk * ES;
  static constexpr int kSC = kSG + kChunk * ES;
  static constexpr int kSA = kSC + NS * kChunk;          // absmax of the chunk's blocks [block][state]
  static constexpr int kSH = kSA + 32;                    // the chunk's header (ChunkRef)
  static constexpr int kStage = kSH + 16;
  static_assert(kStage % 16 == 0, "stages keep 16-byte alignment");
  static_assert(2 * NS * 4 <= 32, "absmax slots of two blocks");
  // CTA layout: maps, midpoints, bucket tables, reduction slots, rings, barriers
  static constexpr int kQ = 0;
  static constexpr int kMid = kQ + NM * 256 * 4;
  static constexpr int kTbl = kMid + NM * 256 * 4;
  static constexpr int kRed = kTbl + NM * kTblSize * 4;
  static constexpr int kRedBytes = 2 * 32 * 4 * 4;       // 2 parities x 32 warps x 4 values
  static constexpr int kRing = kRed + kRedBytes;
  // the opt-in shared memory of an sm_100-class CTA (227 KB), less room for
  // the kernel's static shared variables
  static constexpr int kBudget = 232448 - 1024;
  static constexpr int kWarps = ring_warps<OPT, SH>();
  // two stages where they fit (while one chunk is computed the next is in
  // flight), else one: a chunk is read into registers first thing, so the
  // copy of the next one overlaps the rest of the iteration
  static constexpr int kStages = kRing + kWarps * 2 * (kStage + 8) <= kBudget ? 2 : 1;
  static_assert(kRing + kWarps * kStages * (kStage + 8) <= kBudget, "the ring fits");
  static constexpr int kBars = kRing + kWarps * kStages * kStage;
  // SEQ with blocks of 512 or more: each warp parks its first pass's new
  // states (NS x 256 floats) until the block's absmax is known; offered only
  // where the park fits beside the same number of stages
  static constexpr int kParkWarp = NS * 256 * 4;
  static constexpr bool kPark =
      SH == SH_BIG && NS <= 2 && kRing + kWarps * (kStages * (kStage + 8) + kParkWarp) <= kBudget;
  static constexpr int kPark0 = kBars + kWarps * kStages * 8;
  static_assert(kPark0 % 16 == 0, "the park keeps 16-byte alignment");
  static constexpr int kBytes = kPark0 + (kPark ? kWarps * kParkWarp : 0);
};

// ---------------------------------------------------------------------------
// work units and chunks
// ---------------------------------------------------------------------------
// A unit is what one group of G warps computes together: 512 elements (two
// blocks of 256, or one of 512) when B <= 512, one block when B > 512 (then
// G = B / 512 warps, one 512-element chunk each).  DevTensor::units counts a
// tensor's units, StepArgs::ring_units the launch's.
//
// A chunk: warp j's 512 elements of unit u of tensor t, starting at element
// e0, v of them present (0..512).
struct ChunkRef {
  int64_t e0;
  int32_t u;
  int32_t t;
  int32_t v;
};

// A warp's position in the launch's tensor list: tensor t and unit u in it.
// A warp's units ascend, so it only moves forward.
struct ChunkCursor {
  int32_t t;
  int32_t u;
};
__device__ __forceinline__ void cursor_settle(const StepArgs& a, ChunkCursor& c) {
  int32_t nu;
  while (c.u >= (nu = a.t[c.t].units) && c.t + 1 < a.ntensors) {
    c.u -= nu;
    ++c.t;
  }
}
// log2 of the elements of a unit: max(9, log2B).
__device__ __forceinline__ int unit_shift(const StepArgs& a) {
  return a.log2B > kLog2Chunk ? a.log2B : kLog2Chunk;
}
// WHOLE: every chunk of the launch is whole (the host checked it).
template <bool WHOLE>
__device__ __forceinline__ ChunkRef cursor_chunk(const StepArgs& a, const ChunkCursor& c, int j) {
  ChunkRef r;
  r.t = c.t;
  r.u = c.u;
  r.e0 = (static_cast<int64_t>(c.u) << unit_shift(a)) + j * kChunk;
  if (WHOLE || c.u + 1 < a.t[c.t].units) {
    r.v = kChunk;  // every unit but a tensor's last is whole
  } else {
    const int64_t left = a.t[c.t].n - r.e0;
    r.v = left >= kChunk ? kChunk : (left > 0 ? static_cast<int>(left) : 0);
  }
  return r;
}
// The tensor block of half h of a chunk of unit u (two blocks per chunk when
// B = 256, else one).
__device__ __forceinline__ int32_t chunk_block(bool two, int32_t u, int h) {
  return two ? 2 * u + h : u;
}

template <int OPT>
__device__ __forceinline__ const uint8_t* code_stream(const DevTensor& d, int k) {
  if (OPT == ADEMAMIX) {
    return k == 0 ? static_cast<const uint8_t*>(d.s1)
                  : (k == 1 ? static_cast<const uint8_t*>(d.s1) + d.n
                            : static_cast<const uint8_t*>(d.s2));
  }
  return static_cast<const uint8_t*>(k == 0 ? d.s1 : d.s2);
}
template <int OPT>
__device__ __forceinline__ float* absmax_stream(const DevTensor& d, int k) {
  if (OPT == ADEMAMIX) return k == 0 ? d.a1 : (k == 1 ? d.a1 + d.nblocks : d.a2);
  return k == 0 ? d.a1 : d.a2;
}

// Offset (elements) of quad q (0..3) of lane l inside a chunk.  32-bit
// p/g: quad q holds elements 128q + 4l ..; 16-bit: half h = q / 2 holds
// elements 256h + 8l .. 256h + 8l + 7.  Either way quads 0, 1 of a lane lie
// in the chunk's first 256 elements and 2, 3 in its second.
template <int DT>
__device__ __forceinline__ int quad_offset(int lane, int q) {
  return DT == DT_F32 ? (q * 128 + lane * 4) : ((q >> 1) * 256 + lane * 8 + (q & 1) * 4);
}

// Lane's elements of quads q0 .. q0 + NQ - 1 (q0, NQ even) from a stage (p or g).
template <int DT, int NQ>
__device__ __forceinline__ void stage_load(const unsigned char* base, int lane, int q0,
                                           float (&x)[4 * NQ]) {
  if (DT == DT_F32) {
#pragma unroll
    for (int i = 0; i < NQ; ++i) {
      const float4 u = reinterpret_cast<const float4*>(base + (q0 + i) * 512)[lane];
      x[4 * i] = u.x; x[4 * i + 1] = u.y; x[4 * i + 2] = u.z; x[4 * i + 3] = u.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < NQ / 2; ++i) {
      const uint4 v = reinterpret_cast<const uint4*>(base + (q0 / 2 + i) * 512)[lane];
      x[8 * i + 0] = lo_half(v.x, DT); x[8 * i + 1] = hi_half(v.x, DT);
      x[8 * i + 2] = lo_half(v.y, DT); x[8 * i + 3] = hi_half(v.y, DT);
      x[8 * i + 4] = lo_half(v.z, DT); x[8 * i + 5] = hi_half(v.z, DT);
      x[8 * i + 6] = lo_half(v.w, DT); x[8 * i + 7] = hi_half(v.w, DT);
    }
  }
}
// Lane's codes of one state for quads q0 .. q0 + NQ - 1 from a stage: word i
// holds the codes of quad q0 + i.
template <int DT, int NQ>
__device__ __forceinline__ void stage_codes(const unsigned char* base, int lane, int q0,
                                            uint32_t (&w)[NQ]) {
  if (DT == DT_F32) {
#pragma unroll
    for (int i = 0; i < NQ; ++i) w[i] = reinterpret_cast<const uint32_t*>(base + (q0 + i) * 128)[lane];
  } else {
#pragma unroll
    for (int i = 0; i < NQ / 2; ++i) {
      const uint2 v = reinterpret_cast<const uint2*>(base + (q0 / 2 + i) * 256)[lane];
      w[2 * i] = v.x;
      w[2 * i + 1] = v.y;
    }
  }
}
template <int NQ>
__device__ __forceinline__ uint32_t code_of(const uint32_t (&w)[NQ], int e) {
  return __byte_perm(w[e >> 2], 0u, 0x4440u | static_cast<uint32_t>(e & 3));
}

// The same from global memory (chunks that are partial or whose tensor is
// not aligned for bulk copies); absent elements read as 0.
template <int DT, int NQ>
__device__ __forceinline__ void global_load(const void* base, int64_t e0, int v, int lane, int q0,
                                            float (&x)[4 * NQ]) {
#pragma unroll
  for (int i = 0; i < NQ; ++i) {
    const int o = quad_offset<DT>(lane, q0 + i);
#pragma unroll
    for (int k = 0; k < 4; ++k) x[4 * i + k] = (o + k < v) ? Elem<DT>::ld(base, e0 + o + k) : 0.0f;
  }
}
template <int DT, int NQ>
__device__ __forceinline__ void global_codes(const uint8_t* base, int64_t e0, int v, int lane,
                                             int q0, uint32_t (&w)[NQ]) {
#pragma unroll
  for (int i = 0; i < NQ; ++i) {
    const int o = quad_offset<DT>(lane, q0 + i);
    w[i] = 0u;
#pragma unroll
    for (int k = 0; k < 4; ++k)
      if (o + k < v) w[i] |= static_cast<uint32_t>(base[e0 + o + k]) << (8 * k);
  }
}

// Store the lane's elements of quads q0 .. of p: a full chunk of an aligned
// tensor (vec: DevTensor::vec_ok bit 0) as contiguous spans per warp, else
// element by element.
template <int DT, int NQ>
__device__ __forceinline__ void ring_store(void* base, int64_t e0, int v, bool vec, int lane, int q0,
                                           const float (&x)[4 * NQ]) {
  if (vec && v == kChunk) {
    if (DT == DT_F32) {
      float* b = static_cast<float*>(base) + e0;
#pragma unroll
      for (int i = 0; i < NQ; ++i)
        reinterpret_cast<float4*>(b + 128 * (q0 + i))[lane] =
            make_float4(x[4 * i], x[4 * i + 1], x[4 * i + 2], x[4 * i + 3]);
    } else {
      uint16_t* b = static_cast<uint16_t*>(base) + e0;
#pragma unroll
      for (int i = 0; i < NQ / 2; ++i)
        reinterpret_cast<uint4*>(b + 256 * (q0 / 2 + i))[lane] =
            make_uint4(pack_half2<DT>(x[8 * i], x[8 * i + 1]), pack_half2<DT>(x[8 * i + 2], x[8 * i + 3]),
                       pack_half2<DT>(x[8 * i + 4], x[8 * i + 5]),
                       pack_half2<DT>(x[8 * i + 6], x[8 * i + 7]));
    }
    return;
  }
#pragma unroll
  for (int i = 0; i < NQ; ++i) {
    const int o = quad_offset<DT>(lane, q0 + i);
#pragma unroll
    for (int k = 0; k < 4; ++k)
      if (o + k < v) Elem<DT>::st(base, e0 + o + k, x[4 * i + k]);
  }
}
template <int DT, int NQ>
__device__ __forceinline__ void ring_store_codes(uint8_t* base, int64_t e0, int v, bool vec,
                                                 int lane, int q0, const uint32_t (&w)[NQ]) {
  if (vec && v == kChunk) {
    if (DT == DT_F32) {
#pragma unroll
      for (int i = 0; i < NQ; ++i) reinterpret_cast<uint32_t*>(base + e0 + 128 * (q0 + i))[lane] = w[i];
    } else {
#pragma unroll
      for (int i = 0; i < NQ / 2; ++i)
        reinterpret_cast<uint2*>(base + e0 + 256 * (q0 / 2 + i))[lane] = make_uint2(w[2 * i], w[2 * i + 1]);
    }
    return;
  }
#pragma unroll
  for (int i = 0; i < NQ; ++i) {
    const int o = quad_offset<DT>(lane, q0 + i);
#pragma unroll
    for (int k = 0; k < 4; ++k)
      if (o + k < v) base[e0 + o + k] = static_cast<uint8_t>((w[i] >> (8 * k)) & 0xffu);
  }
}

// Maximum of the NS absmax bit patterns over the G warps of a group: a warp
// max (redux.sync), then, for G > 1, the warps' results meet in red (two
// parities of 32 warps x 4 values) at named barrier 1 + group.
template <int NS>
__device__ __forceinline__ void ring_group_max(uint32_t (&v)[NS], int G, int warp, int lane,
                                               uint32_t* red, int parity) {
#pragma unroll
  for (int k = 0; k < NS; ++k) v[k] = __reduce_max_sync(0xffffffffu, v[k]);
  if (G > 1) {
    uint32_t* slot = red + parity * 32 * 4;
    if (lane == 0) {
#pragma unroll
      for (int k = 0; k < NS; ++k) slot[warp * 4 + k] = v[k];
    }
    const int grp = warp / G;
    named_barrier(1 + grp, G * 32);
    const int w0 = grp * G;
#pragma unroll
    for (int k = 0; k < NS; ++k)
      v[k] = __reduce_max_sync(0xffffffffu, lane < G ? slot[(w0 + lane) * 4 + k] : 0u);
  }
}

// Sum of v over the G warps of a group, in a fixed order (as ring_group_max).
__device__ __forceinline__ float ring_group_sum(float v, int G, int warp, int lane, uint32_t* red,
                                                int parity) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if (G > 1) {
    float* slot = reinterpret_cast<float*>(red + parity * 32 * 4);
    if (lane == 0) slot[warp * 4] = v;
    const int grp = warp / G;
    named_barrier(1 + grp, G * 32);
    const int w0 = grp * G;
    float acc = slot[w0 * 4];
    for (int w = 1; w < G; ++w) acc += slot[(w0 + w) * 4];
    v = acc;
  }
  return v;
}

// Sums of (x, y) over the G warps of a group (G > 1), in a fixed order.
__device__ __forceinline__ float2 ring_group_sum2(float2 v, int G, int warp, int lane, uint32_t* red,
                                                  int parity) {
  float* slot = reinterpret_cast<float*>(red + parity * 32 * 4);
  if (lane == 0) {
    slot[warp * 4] = v.x;
    slot[warp * 4 + 1] = v.y;
  }
  const int grp = warp / G;
  named_barrier(1 + grp, G * 32);
  const int w0 = grp * G;
  float2 acc = make_float2(slot[w0 * 4], slot[w0 * 4 + 1]);
  for (int w = 1; w < G; ++w) {
    acc.x += slot[(w0 + w) * 4];
    acc.y += slot[(w0 + w) * 4 + 1];
  }
  return acc;
}

// WHOLE: every tensor of the launch is aligned for bulk copies and a
// multiple of max(512, B) elements, so every chunk is whole and streams
// through the ring; the element-wise paths for ragged or misaligned chunks are
// compiled out.  SH: the shape (RingShapeId).
// RM (ring mode): RING_STEP the step; RING_NORM the per-tensor max_unorm
// pre-pass: the same update directions u, summed per block as (sum u^2,
// sum p^2) into StepArgs::partials, nothing else written (with a carried
// norm, BNB8_CARRY_PNORM, the p^2 sums are already there, and p is not even
// read when the direction does not need it); RING_BCLIP the step with
// max_unorm per block: each block's directions are kept until its
// unorm_c * ||u|| and ||p|| are known, and the block's multiplier scales its
// step.
enum RingMode { RING_STEP = 0, RING_NORM = 1, RING_BCLIP = 2 };
template <int OPT, int DT, bool WHOLE, int SH, int RM>
__global__ void __launch_bounds__(ring_warps<OPT, SH>() * 32, 1)
    k_step8_ring(const __grid_constant__ StepArgs a) {
  constexpr bool NORM = RM == RING_NORM;
  constexpr bool BCLIP = RM == RING_BCLIP;
  constexpr bool SEQ = SH != SH_ONE;
  constexpr bool BIG = SH == SH_BIG;
  using L = RingSmem<OPT, DT, SH>;
  using R = RingShape<SEQ>;
  constexpr int NS = L::NS;
  constexpr int NM = L::NM;
  constexpr int ES = L::ES;
  constexpr int NQ = R::kQuads;
  constexpr int NE = R::kNE;
  constexpr int kStages = L::kStages;
  extern __shared__ __align__(128) unsigned char ring_smem[];
  unsigned char* smem = ring_smem;
  float* sq = reinterpret_cast<float*>(smem + L::kQ);
  float* smid = reinterpret_cast<float*>(smem + L::kMid);
  uint32_t* stbl = reinterpret_cast<uint32_t*>(smem + L::kTbl);
  uint32_t* sred = reinterpret_cast<uint32_t*>(smem + L::kRed);
  __shared__ int s_bad[2];
  __shared__ int s_below[2];
  __shared__ int s_scan[2 * 32];

  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  unsigned char* ring = smem + L::kRing + warp * kStages * L::kStage;
  float* park = reinterpret_cast<float*>(smem + L::kPark0) + warp * (L::kParkWarp / 4);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBars) + warp * kStages;

  // ---- geometry: groups of G warps share a unit ----
  const bool two = SH == SH_TWO || (SH == SH_ONE && a.log2B == 8);   // two blocks per chunk
  const int G = a.log2B > kLog2Chunk ? (1 << (a.log2B - kLog2Chunk)) : 1;
  const int nwarps = static_cast<int>(blockDim.x >> 5);   // a multiple of G (host)
  const int gpc = nwarps / G;                              // groups per CTA
  const int j = warp % G;                                  // chunk of the unit
  const int32_t NG = static_cast<int32_t>(gridDim.x) * gpc;
  const int32_t b0 = static_cast<int32_t>(blockIdx.x) * gpc + warp / G;
  const int32_t TB = static_cast<int32_t>(a.ring_units);
  // the pre-pass zeroes the tickets of the reduction launched after it
  if (NORM && a.tickets != nullptr && blockIdx.x == 0 && tid < a.ntensors) a.tickets[tid] = 0u;
  // the pre-pass with a carried parameter norm
  const bool carried = NORM && a.carry_stamp != nullptr && *a.carry_stamp == a.carry_expect;
  const bool read_p = !(carried && (Traits<OPT>::DECOUPLED || a.wd == 0.0f));
  // the pre-pass's directions from the hardware approximations
  const bool approx = NORM && ratio_approx_ok(a.eps_hat);

  // ---- the ring: barriers, then the first chunks' copies ----
  if (lane < kStages) mbar_init(bars + lane, 2);   // the bulk copies' arrival and the absmax copies'
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  __syncwarp();
  // copies of a whole chunk c into stage s: p, g and the code streams in bulk
  // (counted in bytes), the absmax of its blocks by cp.async (counted by the
  // second arrival)
  auto issue = [&](const ChunkRef& c, int s) {
    const DevTensor& d = a.t[c.t];
    unsigned char* st = ring + s * L::kStage;
    mbar_expect_tx(bars + s, read_p ? L::kSA : L::kSA - kChunk * ES);
    if (read_p)
      bulk_g2s(st + L::kSP, static_cast<const unsigned char*>(d.p) + c.e0 * ES, kChunk * ES, bars + s);
    bulk_g2s(st + L::kSG, static_cast<const unsigned char*>(d.g) + c.e0 * ES, kChunk * ES, bars + s);
#pragma unroll
    for (int k = 0; k < NS; ++k)
      bulk_g2s(st + L::kSC + k * kChunk, code_stream<OPT>(d, k) + c.e0, kChunk, bars + s);
    const int32_t lb = chunk_block(two, c.u, 0);
#pragma unroll
    for (int k = 0; k < NS; ++k) {
      cp_async4(st + L::kSA + 4 * k, absmax_stream<OPT>(d, k) + lb);
      if (two) cp_async4(st + L::kSA + 4 * (NS + k), absmax_stream<OPT>(d, k) + lb + 1);
    }
    cp_async_arrive(bars + s);
  };
  const bool stall_test = a.stall_test != 0 && blockIdx.x == 0 && warp == 0;
  // per stage (bit s): the parity to wait for; a chunk to wait for (want);
  // copies issued and not yet seen to land (inflight)
  uint32_t phase = 0u, want = 0u, inflight = 0u;
  // the cursor of the next chunk to issue (kStages ahead of the one
  // computed); each issued chunk leaves its ChunkRef in its stage's header
  ChunkCursor cur{0, b0};
  cursor_settle(a, cur);
  auto put_header = [&](const ChunkRef& c, int s) {
    if (lane == 0)
      *reinterpret_cast<int4*>(ring + s * L::kStage + L::kSH) =
          make_int4(static_cast<int>(c.e0), static_cast<int>(c.e0 >> 32), c.u, c.t | (c.v << 16));
  };
  for (int s = 0; s < kStages; ++s) {
    const int32_t b = b0 + s * NG;
    if (b < TB) {
      const ChunkRef c = cursor_chunk<WHOLE>(a, cur, j);
      put_header(c, s);
      if (WHOLE || (c.v == kChunk && (a.t[c.t].vec_ok & 2))) {
        // the stall test withholds this warp's first copy: its wait must run out
        const bool withhold = stall_test && s == 0;
        if (lane == 0 && !withhold) issue(c, s);
        want |= 1u << s;
        if (!withhold) inflight |= 1u << s;
      }
      cur.u += NG;
      cursor_settle(a, cur);
    }
  }
  __syncwarp();

  // ---- maps, midpoints and bucket tables (the first copies land meanwhile) ----
  for (int i = tid; i < NM * 256; i += blockDim.x) sq[i] = i < 256 ? a.qmap1[i] : a.qmap2[i - 256];
  if (tid < 2) s_bad[tid] = 0;
  __syncthreads();
  for (int i = tid; i < NM * 256; i += blockDim.x) {
    const int m = i >> 8, k = i & 255;
    smid[i] = k < 255 ? (sq[m * 256 + k] + sq[m * 256 + k + 1]) * 0.5f : 0.0f;
  }
  __syncthreads();
  build_tables<NM>(smid, stbl, s_bad, s_below, s_scan, static_cast<int>(blockDim.x));
  const bool fast_map[2] = {s_bad[0] == 0, s_bad[1] == 0};
  const bool nonneg_map[2] = {sq[0] >= 0.0f, NM > 1 && sq[256] >= 0.0f};

  // ---- the chunk loop ----
  bool ok = true;          // false once a wait has run out: the warp only keeps its barriers
  int parity = 0;          // reduction-slot parity (G > 1)
  int s = 0;                // the stage of this chunk
  for (int32_t b = b0; b < TB; b += NG, s = (s + 1 == kStages) ? 0 : s + 1) {
    ChunkRef c;
    {
      const int4 h = *reinterpret_cast<const int4*>(ring + s * L::kStage + L::kSH);
      c.e0 = static_cast<int64_t>(static_cast<uint32_t>(h.x)) | (static_cast<int64_t>(h.y) << 32);
      c.u = h.z;
      c.t = h.w & 0xffff;
      c.v = h.w >> 16;
    }
    const DevTensor& d = a.t[c.t];
    const int32_t lb0 = chunk_block(two, c.u, 0);
    // the chunk's second half has elements (and, B = 256, is a second block)
    const bool half1 = WHOLE || c.v > 256;
    const bool second = two && half1;
    const bool have = (WHOLE || c.v > 0) && ok;   // (before this chunk's wait)
    bool staged = false;     // the chunk is in stage s (else read from global memory)
    if ((want >> s) & 1u) {
      if (ok) {
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(bars + s, (phase >> s) & 1u, a.wait_ns));
        if (!ok && lane == 0) atomicOr(a.status, kStatusWaitTimeout);
      }
      if (ok) {
        phase ^= 1u << s;
        want &= ~(1u << s);
        inflight &= ~(1u << s);
        staged = true;
      }
    }
    const unsigned char* st = ring + s * L::kStage;
    // refill stage s with the chunk kStages ahead, once every read of this
    // chunk from the stage is done
    auto refill = [&]() {
      __syncwarp();
      if (ok) {
        const int32_t bn = b + kStages * NG;
        if (bn < TB) {
          const ChunkRef cn = cursor_chunk<WHOLE>(a, cur, j);
          if (lane == 0) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          put_header(cn, s);
          if (WHOLE || (cn.v == kChunk && (a.t[cn.t].vec_ok & 2))) {
            if (lane == 0) issue(cn, s);
            want |= 1u << s;
            inflight |= 1u << s;
          }
          cur.u += NG;
          cursor_settle(a, cur);
        }
      }
    };
    const float eff = a.step_size * (a.clip != nullptr ? a.clip[d.index] : 1.0f);
    // SEQ, blocks of 512 or more: the block's lane maxima and sums over both passes
    uint32_t mxc[NS];
#pragma unroll
    for (int k = 0; k < NS; ++k) mxc[k] = 0u;
    float usq_c = 0.0f, psq_c = 0.0f;

    // requantize the lane's new states svx of quads q0x.. with the block
    // absmax mxh (per block half) and store their codes.  The usual case:
    // every state's absmax lies in [2^-125, 2^125] (or is 0, an all-zero
    // block) and every map takes the table: one Newton reciprocal per block
    // and state and the table lookups, no other tests.
    auto encode_store = [&](const float (&svx)[NS][NE], int q0x, const uint32_t (&mxh)[2][NS]) {
      constexpr int NH = SEQ ? 1 : 2;   // block halves of a pass
      auto hf = [](int e) { return SEQ ? 0 : (e >> 3); };
      uint32_t enc[NS][NE];
      bool usual = true;
#pragma unroll
      for (int k = 0; k < NS; ++k) {
        const int m = Traits<OPT>::map_of(k);
#pragma unroll
        for (int h = 0; h < NH; ++h)
          usual = usual && (mxh[h][k] - 0x01000000u <= 0x7D000000u || mxh[h][k] == 0u);
        usual = usual && fast_map[m] && (!Traits<OPT>::nonneg(k) || nonneg_map[m]);
      }
      if (usual) {
#pragma unroll
        for (int k = 0; k < NS; ++k) {
          float inv[NH];
#pragma unroll
          for (int h = 0; h < NH; ++h) {
            const float amk = __uint_as_float(mxh[h][k]);
            const float y = rcp_approx(amk);
            const float r = __fmaf_rn(__fmaf_rn(-amk, y, 1.0f), y, y);
            inv[h] = mxh[h][k] == 0u ? 0.0f : r;
          }
          const uint32_t* tz = stbl + Traits<OPT>::map_of(k) * kTblSize + kTblZero;
#pragma unroll
          for (int e = 0; e < NE; e += 2) {
            const float2 xn = mul2(make_float2(svx[k][e], svx[k][e + 1]), f2(inv[hf(e)]));
            if (Traits<OPT>::nonneg(k)) {
              enc[k][e] = encode_xn_nonneg(xn.x, tz);
              enc[k][e + 1] = encode_xn_nonneg(xn.y, tz);
            } else {
              enc[k][e] = encode_xn(xn.x, tz);
              enc[k][e + 1] = encode_xn(xn.y, tz);
            }
          }
        }
      } else {
        // absmax tiny, huge or not finite, or a map the table cannot take
#pragma unroll
        for (int k = 0; k < NS; ++k) {
          const int m = Traits<OPT>::map_of(k);
          const uint32_t* tz = stbl + m * kTblSize + kTblZero;
          const float* md = smid + m * 256;
#pragma unroll
          for (int h = 0; h < NH; ++h) {
            const float inv = rcp_block(__uint_as_float(mxh[h][k]));
            const bool fast = fast_map[m] && mxh[h][k] <= 0x7f7fffffu && inv <= FLT_MAX;
#pragma unroll
            for (int e = 8 * h; e < 8 * h + 8; ++e) {
              if (!fast) enc[k][e] = encode_search(svx[k][e] * inv, md);
              else if (Traits<OPT>::nonneg(k) && nonneg_map[m]) enc[k][e] = encode_fast_nonneg(svx[k][e], inv, tz);
              else enc[k][e] = encode_fast(svx[k][e], inv, tz);
            }
          }
        }
      }
#pragma unroll
      for (int k = 0; k < NS; ++k) {
        // byte 2 of each entry is the code
        uint32_t w[NQ];
#pragma unroll
        for (int i = 0; i < NQ; ++i)
          w[i] = __byte_perm(__byte_perm(enc[k][4 * i], enc[k][4 * i + 1], 0x0062u),
                             __byte_perm(enc[k][4 * i + 2], enc[k][4 * i + 3], 0x0062u), 0x5410u);
        ring_store_codes<DT, NQ>(const_cast<uint8_t*>(code_stream<OPT>(d, k)), c.e0,
                                 WHOLE ? kChunk : c.v, WHOLE || (d.vec_ok & 1) != 0, lane, q0x, w);
      }
    };

#pragma unroll
    for (int pass = 0; pass < R::kPasses; ++pass) {
      const int q0 = pass * NQ;            // first quad of the pass
      // pass h of SEQ covers block lb0 + h; !SEQ covers the chunk's blocks at once
      const bool have_p = have && ok && (!SEQ || pass == 0 || half1);
      float am[2][NS];       // absmax of the blocks of the pass's elements (halves 0, 1)
      float p[NE], g[NE];
      uint32_t cw[NS][NQ];
      if (staged) {
        if (read_p) {
          stage_load<DT, NQ>(st + L::kSP, lane, q0, p);
        } else {
#pragma unroll
          for (int e = 0; e < NE; ++e) p[e] = 0.0f;
        }
        stage_load<DT, NQ>(st + L::kSG, lane, q0, g);
#pragma unroll
        for (int k = 0; k < NS; ++k) stage_codes<DT, NQ>(st + L::kSC + k * kChunk, lane, q0, cw[k]);
        const float* sa = reinterpret_cast<const float*>(st + L::kSA);
#pragma unroll
        for (int k = 0; k < NS; ++k) {
          if (SEQ) {
            am[0][k] = am[1][k] = sa[(two ? pass : 0) * NS + k];
          } else {
            am[0][k] = sa[k];
            am[1][k] = two ? sa[NS + k] : sa[k];
          }
        }
      } else if (!WHOLE && have_p) {
#pragma unroll
        for (int k = 0; k < NS; ++k) {
          if (SEQ) {
            am[0][k] = am[1][k] = absmax_stream<OPT>(d, k)[lb0 + (two ? pass : 0)];
          } else {
            am[0][k] = absmax_stream<OPT>(d, k)[lb0];
            am[1][k] = second ? absmax_stream<OPT>(d, k)[lb0 + 1] : am[0][k];
          }
        }
        if (read_p) {
          global_load<DT, NQ>(d.p, c.e0, c.v, lane, q0, p);
        } else {
#pragma unroll
          for (int e = 0; e < NE; ++e) p[e] = 0.0f;
        }
        global_load<DT, NQ>(d.g, c.e0, c.v, lane, q0, g);
#pragma unroll
        for (int k = 0; k < NS; ++k)
          global_codes<DT, NQ>(code_stream<OPT>(d, k), c.e0, c.v, lane, q0, cw[k]);
      }
      if (pass + 1 == R::kPasses) refill();

      // ---- dequantize and update; new states in sv, running max of |s| per
      // ---- block half in mx ----
      float sv[NS][NE];
      uint32_t mx[2][NS];
      float psq[2] = {0.0f, 0.0f};   // sum of p^2 per block half (carried norm; NORM: the old p)
      float usq[2] = {0.0f, 0.0f};   // NORM, BCLIP: sum of u^2 per block half
      float2 usq2[2] = {f2(0.0f), f2(0.0f)};   // NORM, BCLIP: the same on pairs (whole chunks)
      float ud[BCLIP ? NE : 1];      // BCLIP: the directions, applied once the block's clip is known
#pragma unroll
      for (int k = 0; k < NS; ++k) mx[0][k] = mx[1][k] = 0u;
      // the block half of element e of this pass
      auto half_of = [](int e) { return SEQ ? 0 : (e >> 3); };
      // element e of this pass is present (partial chunks)
      const bool full = WHOLE || c.v == kChunk;
      auto present = [&](int e) { return full || quad_offset<DT>(lane, q0 + (e >> 2)) + (e & 3) < c.v; };
      // NORM, BCLIP: the directions of elements e, e + 1 into their block half's sums
      auto add_u2 = [&](int e, float2 u) {
        if (full) {
          usq2[half_of(e)] = fma2(u, u, usq2[half_of(e)]);
        } else {
          if (present(e)) usq[half_of(e)] = usq[half_of(e)] + u.x * u.x;
          if (present(e + 1)) usq[half_of(e)] = usq[half_of(e)] + u.y * u.y;
        }
      };
      if (have_p) {
        // optimizers whose direction is n / (sqrt(v) + eps)
        constexpr bool kRatio = OPT == ADAM || OPT == ADAMW || OPT == RMSPROP || OPT == ADAGRAD ||
                                OPT == ADEMAMIX;
        constexpr int kV = (OPT == ADAM || OPT == ADAMW) ? 1 : (OPT == ADEMAMIX ? 2 : 0);
        float gk[NE];            // RMSprop, Adagrad: the scaled gradient, their numerator
        // running minima of (bits of v) - 1 and 2|n|'s bits - 2: a zero maps
        // to the top of the range, so a minimum below the threshold means a
        // nonzero v or numerator under 2^-100 (outside the fast ratio's range)
        uint32_t lo_v = 0xffffffffu, lo_n = 0xffffffffu;
        uint32_t nmax = 0u;      // max |numerator| of the lane (bit pattern)
        // pass 1: the new states (Momentum and Lion: also the new p)
#pragma unroll
        for (int e = 0; e < NE; e += 2) {
          const int h = half_of(e);
          float2 stt[3];
#pragma unroll
          for (int k = 0; k < 3; ++k)
            stt[k] = k < NS ? mul2(make_float2(sq[Traits<OPT>::map_of(k) * 256 + code_of<NQ>(cw[k], e)],
                                               sq[Traits<OPT>::map_of(k) * 256 + code_of<NQ>(cw[k], e + 1)]),
                                   f2(am[h][k]))
                            : f2(0.0f);
          float2 pp = make_float2(p[e], p[e + 1]);
          float2 gg = mul2(make_float2(g[e], g[e + 1]), f2(a.gscale));
          if (!Traits<OPT>::DECOUPLED && a.wd != 0.0f) gg = fma2(f2(a.wd), pp, gg);
          if (OPT == ADAM || OPT == ADAMW) {
            const float2 m = fma2(f2(a.b1), stt[0], mul2(f2(a.omb1), gg));
            const float2 v = fma2(f2(a.b2), stt[1], mul2(f2(a.omb2), mul2(gg, gg)));
            sv[0][e] = m.x; sv[0][e + 1] = m.y;
            sv[1][e] = v.x; sv[1][e + 1] = v.y;
            if (!NORM) {
              lo_n = min_tiny_n(lo_n, m);
              lo_v = min_tiny_v(lo_v, v);
            }
          } else if (OPT == RMSPROP || OPT == ADAGRAD) {
            const float2 v = OPT == RMSPROP ? fma2(f2(a.b1), stt[0], mul2(f2(a.omb1), mul2(gg, gg)))
                                            : fma2(gg, gg, stt[0]);
            sv[0][e] = v.x; sv[0][e + 1] = v.y;
            gk[e] = gg.x; gk[e + 1] = gg.y;
            if (!NORM) {
              nmax = absmax_nan(nmax, gg.x, gg.y);
              lo_n = min_tiny_n(lo_n, gg);
              lo_v = min_tiny_v(lo_v, v);
            }
          } else if (OPT == ADEMAMIX) {
            const float2 m1 = fma2(f2(a.b1), stt[0], mul2(f2(a.omb1), gg));
            const float2 m2 = fma2(f2(a.b3t), stt[1], mul2(f2(a.omb3t), gg));
            const float2 nu = fma2(f2(a.b2), stt[2], mul2(f2(a.omb2), mul2(gg, gg)));
            const float2 num = fma2(m1, f2(a.inv_bc1), mul2(f2(a.alpha_t), m2));
            sv[0][e] = m1.x; sv[0][e + 1] = m1.y;
            sv[1][e] = m2.x; sv[1][e + 1] = m2.y;
            sv[2][e] = nu.x; sv[2][e + 1] = nu.y;
            if (!NORM) {
              nmax = absmax_nan(nmax, num.x, num.y);
              lo_n = min_tiny_n(lo_n, num);
              lo_v = min_tiny_v(lo_v, nu);
            }
          } else if (OPT == MOMENTUM) {
            const float2 m = fma2(f2(a.b1), stt[0], gg);
            sv[0][e] = m.x; sv[0][e + 1] = m.y;
            if (NORM || BCLIP) add_u2(e, m);
            if (BCLIP) {
              ud[e] = m.x; ud[e + 1] = m.y;
            } else if (!NORM) {
              pair_apply<OPT>(a, -eff, pp, m);
              p[e] = pp.x; p[e + 1] = pp.y;
            }
          } else {  // LION
            const float2 cc = fma2(f2(a.b1), stt[0], mul2(f2(a.omb1), gg));
            const float2 m = fma2(f2(a.b2), stt[0], mul2(f2(a.omb2), gg));
            sv[0][e] = m.x; sv[0][e + 1] = m.y;
            if (NORM || BCLIP) {
              float2 u;
              u.x = cc.x > 0.0f ? 1.0f : (cc.x < 0.0f ? -1.0f : 0.0f);
              u.y = cc.y > 0.0f ? 1.0f : (cc.y < 0.0f ? -1.0f : 0.0f);
              add_u2(e, u);
              if (BCLIP) {
                ud[e] = u.x; ud[e + 1] = u.y;
              }
            } else {
              // p + (-eff)*sign(c) with the product formed by bits: -eff
              // with c's sign folded in where |c| > 0, else the signed zero
              // -eff * (+0); the one rounding is the sum's, as in the FMA
              const float2 t = lion_term(-eff, cc);
              if (Traits<OPT>::DECOUPLED && a.wd != 0.0f) pp = mul2(pp, f2(a.decay));
              pp = __fadd2_rn(pp, t);
              p[e] = pp.x; p[e + 1] = pp.y;
            }
          }
        }
        // absent elements of a partial chunk keep state 0 (they do not count in the absmax)
        if (!WHOLE && c.v < kChunk) {
#pragma unroll
          for (int i = 0; i < NQ; ++i) {
            const int o = quad_offset<DT>(lane, q0 + i);
#pragma unroll
            for (int e = 0; e < 4; ++e)
              if (o + e >= c.v) {
#pragma unroll
                for (int k = 0; k < NS; ++k) sv[k][4 * i + e] = 0.0f;
                if (OPT == RMSPROP || OPT == ADAGRAD) gk[4 * i + e] = 0.0f;
              }
          }
        }
        // (the pre-pass requantizes nothing: no absmax)
        if constexpr (!NORM) {
#pragma unroll
          for (int k = 0; k < NS; ++k)
#pragma unroll
            for (int e = 0; e < NE; e += 2)
              mx[half_of(e)][k] = absmax_nan(mx[half_of(e)][k], sv[k][e], sv[k][e + 1]);
        }
        if constexpr (kRatio && NORM) {
          // the pre-pass: u only for its norm, from the hardware
          // approximations (within 2^-21 relative) where eps allows, else
          // from the IEEE operations
          auto numer = [&](int e) -> float2 {
            if (OPT == RMSPROP || OPT == ADAGRAD) return make_float2(gk[e], gk[e + 1]);
            if (OPT == ADEMAMIX)
              return fma2(make_float2(sv[0][e], sv[0][e + 1]), f2(a.inv_bc1),
                          mul2(f2(a.alpha_t), make_float2(sv[1][e], sv[1][e + 1])));
            return make_float2(sv[0][e], sv[0][e + 1]);
          };
          if (approx) {
#pragma unroll
            for (int e = 0; e < NE; e += 2)
              add_u2(e, ratio2_approx(numer(e), make_float2(sv[kV][e], sv[kV][e + 1]), a.eps_hat));
          } else {
#pragma unroll
            for (int e = 0; e < NE; e += 2)
              add_u2(e, ratio2_ieee_slow(numer(e), make_float2(sv[kV][e], sv[kV][e + 1]), a.eps_hat));
          }
        } else if constexpr (kRatio) {
          // pass 2: u = n / (sqrt(v) + eps) and the new p; the fast ratio
          // when every operand of the lane lies in its range, the IEEE
          // operations else
          const uint32_t vmax = mx[0][kV] > mx[1][kV] ? mx[0][kV] : mx[1][kV];
          if (OPT == ADAM || OPT == ADAMW) nmax = mx[0][0] > mx[1][0] ? mx[0][0] : mx[1][0];
          const bool fast = lo_v >= kRatioLoV && lo_n >= kRatioLoN && a.eps_hat >= 0x1p-60f &&
                            a.eps_hat <= 0x1p20f && vmax <= kRatioMaxV && nmax <= kRatioMaxN;
          auto numer = [&](int e) -> float2 {
            if (OPT == RMSPROP || OPT == ADAGRAD) return make_float2(gk[e], gk[e + 1]);
            if (OPT == ADEMAMIX)
              return fma2(make_float2(sv[0][e], sv[0][e + 1]), f2(a.inv_bc1),
                          mul2(f2(a.alpha_t), make_float2(sv[1][e], sv[1][e + 1])));
            return make_float2(sv[0][e], sv[0][e + 1]);
          };
          // the direction of elements e, e + 1 into the sums, the kept
          // directions or the new p
          auto use_u = [&](int e, float2 u) {
            if (NORM || BCLIP) add_u2(e, u);
            if (BCLIP) {
              ud[e] = u.x; ud[e + 1] = u.y;
            } else if (!NORM) {
              float2 pp = make_float2(p[e], p[e + 1]);
              pair_apply<OPT>(a, -eff, pp, u);
              p[e] = pp.x; p[e + 1] = pp.y;
            }
          };
          // RMSprop, Adagrad: a lane whose numerators (the scaled gradients)
          // are all +-0 has u = n exactly, since then d = sqrt(v) + eps > 0
          // (no v is NaN, eps > 0) and +-0 / d = +-0: the untouched rows of
          // an embedding skip the square root and the division
          const bool zero_n = (OPT == RMSPROP || OPT == ADAGRAD) && nmax == 0u &&
                              vmax <= 0x7f800000u && a.eps_hat > 0.0f;
          if (zero_n) {
#pragma unroll
            for (int e = 0; e < NE; e += 2) use_u(e, numer(e));
          } else if (fast) {
#pragma unroll
            for (int e = 0; e < NE; e += 2)
              use_u(e, ratio2_fast(numer(e), make_float2(sv[kV][e], sv[kV][e + 1]), a.eps_hat));
          } else {
#pragma unroll
            for (int e = 0; e < NE; e += 2)
              use_u(e, ratio2_ieee_slow(numer(e), make_float2(sv[kV][e], sv[kV][e + 1]), a.eps_hat));
          }
        }
        if (NORM || BCLIP) {
          // the parameter norm of the step's input (unless carried)
          if (!carried) {
            float2 psq2[2] = {f2(0.0f), f2(0.0f)};
#pragma unroll
            for (int e = 0; e < NE; e += 2) {
              // absent elements of a partial chunk hold p = 0
              const float2 pp = make_float2(p[e], p[e + 1]);
              psq2[half_of(e)] = fma2(pp, pp, psq2[half_of(e)]);
            }
            psq[0] = psq2[0].x + psq2[0].y;
            psq[1] = psq2[1].x + psq2[1].y;
          }
#pragma unroll
          for (int h = 0; h < 2; ++h) usq[h] = usq[h] + (usq2[h].x + usq2[h].y);
        }
        if (RM == RING_STEP)
          ring_store<DT, NQ>(d.p, c.e0, WHOLE ? kChunk : c.v, WHOLE || (d.vec_ok & 1) != 0, lane, q0, p);
        if (RM == RING_STEP && a.carry_out) {
          // the squares of p as stored (rounded to the dtype); the registers
          // of a partial chunk's absent elements hold no parameter
#pragma unroll
          for (int e = 0; e < NE; ++e) {
            const float q = Elem<DT>::stored(p[e]);
            if (WHOLE || quad_offset<DT>(lane, q0 + (e >> 2)) + (e & 3) < c.v)
              psq[half_of(e)] = psq[half_of(e)] + q * q;
          }
        }
      } else {
#pragma unroll
        for (int k = 0; k < NS; ++k)
#pragma unroll
          for (int e = 0; e < NE; ++e) sv[k][e] = 0.0f;
      }

      if constexpr (BIG && RM != RING_BCLIP) {
        // Blocks of 512 elements or more: both passes belong to one block
        // (G warps share it).  The first pass parks its new states in
        // shared memory; after the second the block's absmax and sums are
        // reduced (every warp of the group takes part) and both passes are
        // requantized with the block's reciprocal.
#pragma unroll
        for (int k = 0; k < NS; ++k) mxc[k] = mxc[k] > mx[0][k] ? mxc[k] : mx[0][k];
        usq_c = usq_c + usq[0];
        psq_c = psq_c + psq[0];
        if (pass == 0) {
          if (!NORM && have_p) {
#pragma unroll
            for (int k = 0; k < NS; ++k)
#pragma unroll
              for (int i = 0; i < NE / 4; ++i)
                reinterpret_cast<float4*>(park + k * 256)[i * 32 + lane] =
                    make_float4(sv[k][4 * i], sv[k][4 * i + 1], sv[k][4 * i + 2], sv[k][4 * i + 3]);
          }
          continue;
        }
        const bool have_blk = have && ok;
        if constexpr (NORM) {
          float2 r = make_float2(usq_c, psq_c);
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            r.x += __shfl_xor_sync(0xffffffffu, r.x, o);
            r.y += __shfl_xor_sync(0xffffffffu, r.y, o);
          }
          if (G > 1) {
            r = ring_group_sum2(r, G, warp, lane, sred, parity);
            parity ^= 1;
          }
          if (have_blk && j == 0 && lane == 0) {
            if (carried) a.partials[d.first_block + lb0].x = r.x;
            else a.partials[d.first_block + lb0] = r;
          }
        } else {
          if (a.carry_out) {
            const float bsq = ring_group_sum(psq_c, G, warp, lane, sred, parity);
            parity ^= 1;
            if (have_blk && j == 0 && lane == 0)
              reinterpret_cast<float*>(a.partials + d.first_block + lb0)[1] = bsq;
          }
          ring_group_max<NS>(mxc, G, warp, lane, sred, parity);
          parity ^= 1;
          if (have_blk) {
            uint32_t mxh[2][NS];
#pragma unroll
            for (int k = 0; k < NS; ++k) mxh[0][k] = mxh[1][k] = mxc[k];
            if (have_p) encode_store(sv, q0, mxh);
            // the first pass's states back from the park
#pragma unroll
            for (int k = 0; k < NS; ++k)
#pragma unroll
              for (int i = 0; i < NE / 4; ++i) {
                const float4 v = reinterpret_cast<const float4*>(park + k * 256)[i * 32 + lane];
                sv[k][4 * i] = v.x; sv[k][4 * i + 1] = v.y; sv[k][4 * i + 2] = v.z; sv[k][4 * i + 3] = v.w;
              }
            encode_store(sv, 0, mxh);
            if (j == 0 && lane == 0) {
#pragma unroll
              for (int k = 0; k < NS; ++k) absmax_stream<OPT>(d, k)[lb0] = __uint_as_float(mxc[k]);
            }
          }
        }
        continue;
      }

      if constexpr (BCLIP) {
        // the block's sums (every lane receives them; every warp of a group
        // takes part, those without elements with zeros), its multiplier,
        // the step
        float2 r0 = make_float2(usq[0], psq[0]), r1 = make_float2(usq[1], psq[1]);
        if (!SEQ && !two) r0 = make_float2(usq[0] + usq[1], psq[0] + psq[1]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          r0.x += __shfl_xor_sync(0xffffffffu, r0.x, o);
          r0.y += __shfl_xor_sync(0xffffffffu, r0.y, o);
          if (!SEQ) {
            r1.x += __shfl_xor_sync(0xffffffffu, r1.x, o);
            r1.y += __shfl_xor_sync(0xffffffffu, r1.y, o);
          }
        }
        if (!SEQ && !two && G > 1) {
          r0 = ring_group_sum2(r0, G, warp, lane, sred, parity);
          parity ^= 1;
        }
        if (!SEQ && !two) r1 = r0;
        if (have_p) {
          float effb[2];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const float2 r = h == 0 ? r0 : r1;
            const float unorm = a.unorm_c * sqrtf(r.x);
            const float limit = a.max_unorm * sqrtf(r.y);
            effb[h] = eff * (unorm > limit ? limit / unorm : 1.0f);
          }
#pragma unroll
          for (int e = 0; e < NE; e += 2) {
            float2 pp = make_float2(p[e], p[e + 1]);
            pair_apply<OPT>(a, -effb[half_of(e)], pp, make_float2(ud[e], ud[e + 1]));
            p[e] = pp.x; p[e + 1] = pp.y;
          }
          ring_store<DT, NQ>(d.p, c.e0, WHOLE ? kChunk : c.v, WHOLE || (d.vec_ok & 1) != 0, lane, q0, p);
        }
      }

      if constexpr (NORM) {
        // ---- the blocks' (sum u^2, sum p^2) ----
        if (two) {
          float2 r0 = make_float2(usq[0], psq[0]), r1 = make_float2(usq[1], psq[1]);
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            r0.x += __shfl_xor_sync(0xffffffffu, r0.x, o);
            r0.y += __shfl_xor_sync(0xffffffffu, r0.y, o);
            if (!SEQ) {
              r1.x += __shfl_xor_sync(0xffffffffu, r1.x, o);
              r1.y += __shfl_xor_sync(0xffffffffu, r1.y, o);
            }
          }
          if (have_p && lane == 0) {
            const int32_t blk = d.first_block + lb0 + (SEQ ? pass : 0);
            if (carried) a.partials[blk].x = r0.x;
            else a.partials[blk] = r0;
            if (!SEQ && second) {
              if (carried) a.partials[blk + 1].x = r1.x;
              else a.partials[blk + 1] = r1;
            }
          }
        } else {
          float2 r = make_float2(usq[0] + usq[1], psq[0] + psq[1]);
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            r.x += __shfl_xor_sync(0xffffffffu, r.x, o);
            r.y += __shfl_xor_sync(0xffffffffu, r.y, o);
          }
          if (G > 1) {
            r = ring_group_sum2(r, G, warp, lane, sred, parity);
            parity ^= 1;
          }
          if (have_p && j == 0 && lane == 0) {
            if (carried) a.partials[d.first_block + lb0].x = r.x;
            else a.partials[d.first_block + lb0] = r;
          }
        }
        continue;
      }

      // ---- each block's new absmax (every warp of the group takes part) ----
      if (SEQ) {
#pragma unroll
        for (int k = 0; k < NS; ++k) mx[0][k] = mx[1][k] = __reduce_max_sync(0xffffffffu, mx[0][k]);
      } else if (two) {
        // two blocks of 256 in the chunk, one warp each way: warp maxima
#pragma unroll
        for (int k = 0; k < NS; ++k) {
          mx[0][k] = __reduce_max_sync(0xffffffffu, mx[0][k]);
          mx[1][k] = __reduce_max_sync(0xffffffffu, mx[1][k]);
        }
      } else {
#pragma unroll
        for (int k = 0; k < NS; ++k) mx[0][k] = mx[0][k] > mx[1][k] ? mx[0][k] : mx[1][k];
        ring_group_max<NS>(mx[0], G, warp, lane, sred, parity);
        parity ^= 1;
#pragma unroll
        for (int k = 0; k < NS; ++k) mx[1][k] = mx[0][k];
      }
      if (RM == RING_STEP && a.carry_out) {
        if (two) {
          float s0 = psq[0], s1 = psq[1];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            s0 += __shfl_xor_sync(0xffffffffu, s0, o);
            if (!SEQ) s1 += __shfl_xor_sync(0xffffffffu, s1, o);
          }
          if (have_p && lane == 0) {
            const int32_t blk = d.first_block + lb0 + (SEQ ? pass : 0);
            reinterpret_cast<float*>(a.partials + blk)[1] = s0;
            if (!SEQ && second) reinterpret_cast<float*>(a.partials + blk + 1)[1] = s1;
          }
        } else {
          const float bsq = ring_group_sum(psq[0] + psq[1], G, warp, lane, sred, parity);
          parity ^= 1;
          if (have_p && j == 0 && lane == 0)
            reinterpret_cast<float*>(a.partials + d.first_block + lb0)[1] = bsq;
        }
      }
      if (!have_p) continue;

      // ---- requantize and store codes (and, once per block, the absmax) ----
      encode_store(sv, q0, mx);
      if (j == 0 && lane == 0) {
#pragma unroll
        for (int k = 0; k < NS; ++k) {
          if (SEQ) {
            absmax_stream<OPT>(d, k)[lb0 + pass] = __uint_as_float(mx[0][k]);
          } else {
            absmax_stream<OPT>(d, k)[lb0] = __uint_as_float(mx[0][k]);
            if (second) absmax_stream<OPT>(d, k)[lb0 + 1] = __uint_as_float(mx[1][k]);
          }
        }
      }
    }
  }

  if (RM == RING_STEP && a.carry_writer && blockIdx.x == 0 && threadIdx.x == 0)
    *a.carry_stamp = a.carry_write;

  // ---- a wait ran out: let this warp's copies still in flight land ----
  if (!ok && lane == 0) {
    for (int s = 0; s < kStages; ++s)
      if ((inflight >> s) & 1u) mbar_wait_bounded(bars + s, (phase >> s) & 1u, a.wait_ns);
  }
}

// CTA size for a launch: as many warps as the ring holds, whole groups.
// (at most 15 groups: named barriers 1..15 are the groups' meeting points)
template <int OPT, int SH>
__host__ __forceinline__ int ring_threads(int log2B) {
  const int G = log2B > kLog2Chunk ? (1 << (log2B - kLog2Chunk)) : 1;
  int groups = ring_warps<OPT, SH>() / G;
  if (G > 1 && groups > 15) groups = 15;
  return groups * G * 32;
}

template <int OPT, int DT, bool WHOLE, int SH, int RM>
cudaError_t launch_step8_ring_w(const StepArgs& a, cudaStream_t s) {
  using L = RingSmem<OPT, DT, SH>;
  static std::atomic<unsigned char> configured[kMaxDevices];
  cudaError_t e = set_smem_limit_once(reinterpret_cast<const void*>(k_step8_ring<OPT, DT, WHOLE, SH, RM>),
                                      L::kBytes, configured);
  if (e != cudaSuccess) return e;
  const int threads = ring_threads<OPT, SH>(a.log2B);
  const int G = a.log2B > kLog2Chunk ? (1 << (a.log2B - kLog2Chunk)) : 1;
  const int64_t groups = threads / 32 / G;
  const int64_t need = (a.ring_units + groups - 1) / groups;
  const int grid = static_cast<int>(need < a.nsm ? need : a.nsm);
  k_step8_ring<OPT, DT, WHOLE, SH, RM><<<grid, threads, L::kBytes, s>>>(a);
  return cudaGetLastError();
}

// Blocksize 256: two passes of a block each (24 warps); larger blocks: two
// passes of one block with the first pass parked (24 warps) where the park
// fits, else one pass over the chunk (16 warps).
template <int OPT, int DT, int RM>
cudaError_t launch_step8_ring(const StepArgs& a, cudaStream_t s) {
  if (a.log2B == 8)
    return a.whole ? launch_step8_ring_w<OPT, DT, true, SH_TWO, RM>(a, s)
                   : launch_step8_ring_w<OPT, DT, false, SH_TWO, RM>(a, s);
  if constexpr (RM != RING_BCLIP && RingSmem<OPT, DT, SH_BIG>::kPark) {
    return a.whole ? launch_step8_ring_w<OPT, DT, true, SH_BIG, RM>(a, s)
                   : launch_step8_ring_w<OPT, DT, false, SH_BIG, RM>(a, s);
  } else {
    return a.whole ? launch_step8_ring_w<OPT, DT, true, SH_ONE, RM>(a, s)
                   : launch_step8_ring_w<OPT, DT, false, SH_ONE, RM>(a, s);
  }
}

}  // namespace bnb8
