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
// shared memory layout
// ---------------------------------------------------------------------------
// Warps per CTA (one CTA per SM): fewer warps leave each thread more
// registers (65536 / threads), more warps keep more copies in flight.
#ifndef BNB8_RING_WARPS
#define BNB8_RING_WARPS 24
#endif
constexpr int kRingWarps = BNB8_RING_WARPS;
// Stages per warp: while one chunk is computed, the next kRingStages - 1 are
// in flight.
#ifndef BNB8_RING_STAGES
#define BNB8_RING_STAGES 2
#endif
constexpr int kRingStages = BNB8_RING_STAGES;
template <int OPT, int DT>
struct RingSmem {
  static constexpr int NS = Traits<OPT>::NS;
  static constexpr int NM = Traits<OPT>::NM;
  static constexpr int ES = DT == DT_F32 ? 4 : 2;
  static constexpr int kChunk = 256;                     // elements per warp and iteration
  // one stage: p | g | codes of each state
  static constexpr int kSP = 0;
  static constexpr int kSG = kSP + kChunk * ES;
  static constexpr int kSC = kSG + kChunk * ES;
  static constexpr int kSA = kSC + NS * kChunk;          // the block's absmax of each state
  static constexpr int kSH = kSA + 16;                    // the chunk's header (ChunkRef)
  static constexpr int kStage = kSH + 16;
  static_assert(kStage % 16 == 0, "stages keep 16-byte alignment");
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
  static constexpr int kFit = (kBudget - kRing) / (kRingStages * (kStage + 8));
  static constexpr int kWarps = kFit < kRingWarps ? kFit : kRingWarps;
  static_assert(kWarps >= 16, "the ring leaves room for at least 16 warps");
  static constexpr int kBars = kRing + kWarps * kRingStages * kStage;
  static constexpr int kBytes = kBars + kWarps * kRingStages * 8;
};

// ---------------------------------------------------------------------------
// per-chunk addressing
// ---------------------------------------------------------------------------
// A chunk: warp j's 256 elements of local block lb of tensor t, starting at
// element e0, v of them present (0..256).
struct ChunkRef {
  int64_t e0;
  int32_t lb;
  int32_t t;
  int32_t v;
};

__device__ __forceinline__ int32_t tensor_blocks(const StepArgs& a, int t) { return a.t[t].nblocks; }

// A warp's position in the launch's tensor list: tensor t and local block lb
// in it.  A warp's blocks ascend, so it only moves forward.
struct ChunkCursor {
  int32_t t;
  int32_t lb;
};
__device__ __forceinline__ void cursor_settle(const StepArgs& a, ChunkCursor& c) {
  int32_t nb;
  while (c.lb >= (nb = tensor_blocks(a, c.t)) && c.t + 1 < a.ntensors) {
    c.lb -= nb;
    ++c.t;
  }
}
// WHOLE: every chunk of the launch is whole (the host checked it).
template <bool WHOLE>
__device__ __forceinline__ ChunkRef cursor_chunk(const StepArgs& a, const ChunkCursor& c, int j) {
  ChunkRef r;
  r.t = c.t;
  r.lb = c.lb;
  r.e0 = (static_cast<int64_t>(c.lb) << a.log2B) + j * 256;
  if (WHOLE || c.lb + 1 < tensor_blocks(a, c.t)) {
    r.v = 256;  // every block but a tensor's last is whole
  } else {
    const int64_t left = a.t[c.t].n - r.e0;
    r.v = left >= 256 ? 256 : (left > 0 ? static_cast<int>(left) : 0);
  }
  return r;
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
__device__ __forceinline__ float* absmax_stream(const DevTensor& d, int k, int32_t nblocks) {
  if (OPT == ADEMAMIX) return k == 0 ? d.a1 : (k == 1 ? d.a1 + nblocks : d.a2);
  return k == 0 ? d.a1 : d.a2;
}

// Offset (elements) of quad q (0, 1) of lane l inside a chunk.
template <int DT>
__device__ __forceinline__ int quad_offset(int lane, int q) {
  return DT == DT_F32 ? (q * 128 + lane * 4) : (lane * 8 + q * 4);
}

// Lane's 8 elements of a full chunk from a stage (p or g).
template <int DT>
__device__ __forceinline__ void stage_load8(const unsigned char* base, int lane, float (&x)[8]) {
  if (DT == DT_F32) {
    const float4 u = reinterpret_cast<const float4*>(base)[lane];
    const float4 w = reinterpret_cast<const float4*>(base + 512)[lane];
    x[0] = u.x; x[1] = u.y; x[2] = u.z; x[3] = u.w;
    x[4] = w.x; x[5] = w.y; x[6] = w.z; x[7] = w.w;
  } else {
    const uint4 v = reinterpret_cast<const uint4*>(base)[lane];
    x[0] = lo_half(v.x, DT); x[1] = hi_half(v.x, DT);
    x[2] = lo_half(v.y, DT); x[3] = hi_half(v.y, DT);
    x[4] = lo_half(v.z, DT); x[5] = hi_half(v.z, DT);
    x[6] = lo_half(v.w, DT); x[7] = hi_half(v.w, DT);
  }
}
// Lane's 8 codes of one state from a stage.
template <int DT>
__device__ __forceinline__ uint2 stage_codes(const unsigned char* base, int lane) {
  if (DT == DT_F32)
    return make_uint2(reinterpret_cast<const uint32_t*>(base)[lane],
                      reinterpret_cast<const uint32_t*>(base + 128)[lane]);
  return reinterpret_cast<const uint2*>(base)[lane];
}

// Lane's elements straight from global memory (chunks that are partial or
// whose tensor is not aligned for bulk copies); absent elements read as 0.
template <int DT>
__device__ __forceinline__ void global_load8(const void* base, int64_t e0, int v, int lane,
                                             float (&x)[8]) {
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int o = quad_offset<DT>(lane, q);
#pragma unroll
    for (int i = 0; i < 4; ++i) x[4 * q + i] = (o + i < v) ? Elem<DT>::ld(base, e0 + o + i) : 0.0f;
  }
}
template <int DT>
__device__ __forceinline__ uint2 global_codes(const uint8_t* base, int64_t e0, int v, int lane) {
  uint32_t w[2] = {0u, 0u};
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int o = quad_offset<DT>(lane, q);
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (o + i < v) w[q] |= static_cast<uint32_t>(base[e0 + o + i]) << (8 * i);
  }
  return make_uint2(w[0], w[1]);
}

// Store the lane's 8 elements of p: a full chunk of an aligned tensor (vec:
// DevTensor::vec_ok bit 0) as one contiguous span per warp, else element by
// element.
template <int DT>
__device__ __forceinline__ void ring_store8(void* base, int64_t e0, int v, bool vec, int lane,
                                            const float (&x)[8]) {
  if (vec && v == 256) {
    if (DT == DT_F32) {
      float* b = static_cast<float*>(base) + e0;
      reinterpret_cast<float4*>(b)[lane] = make_float4(x[0], x[1], x[2], x[3]);
      reinterpret_cast<float4*>(b + 128)[lane] = make_float4(x[4], x[5], x[6], x[7]);
    } else {
      uint4* b = reinterpret_cast<uint4*>(static_cast<uint16_t*>(base) + e0);
      b[lane] = make_uint4(pack_half2<DT>(x[0], x[1]), pack_half2<DT>(x[2], x[3]),
                           pack_half2<DT>(x[4], x[5]), pack_half2<DT>(x[6], x[7]));
    }
    return;
  }
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int o = quad_offset<DT>(lane, q);
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (o + i < v) Elem<DT>::st(base, e0 + o + i, x[4 * q + i]);
  }
}
template <int DT>
__device__ __forceinline__ void ring_store_codes(uint8_t* base, int64_t e0, int v, bool vec,
                                                 int lane, uint2 c) {
  if (vec && v == 256) {
    if (DT == DT_F32) {
      reinterpret_cast<uint32_t*>(base + e0)[lane] = c.x;
      reinterpret_cast<uint32_t*>(base + e0 + 128)[lane] = c.y;
    } else {
      reinterpret_cast<uint2*>(base + e0)[lane] = c;
    }
    return;
  }
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int o = quad_offset<DT>(lane, q);
    const uint32_t w = q == 0 ? c.x : c.y;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (o + i < v) base[e0 + o + i] = static_cast<uint8_t>((w >> (8 * i)) & 0xffu);
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

// WHOLE: every tensor of the launch is aligned for bulk copies and a
// multiple of max(256, B) elements, so every chunk is whole and streams
// through the ring; the element-wise paths for ragged or misaligned chunks are
// compiled out.
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

template <int OPT, int DT, bool WHOLE>
__global__ void __launch_bounds__(kRingWarps * 32, 1) k_step8_ring(const __grid_constant__ StepArgs a) {
  using L = RingSmem<OPT, DT>;
  constexpr int NS = L::NS;
  constexpr int NM = L::NM;
  constexpr int ES = L::ES;
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
  unsigned char* ring = smem + L::kRing + warp * kRingStages * L::kStage;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBars) + warp * kRingStages;

  // ---- geometry: groups of G warps share a block of G * 256 elements ----
  const int G = a.log2B > 8 ? (1 << (a.log2B - 8)) : 1;
  const int nwarps = static_cast<int>(blockDim.x >> 5);   // a multiple of G (host)
  const int gpc = nwarps / G;                              // groups per CTA
  const int j = warp % G;                                  // chunk of the block
  const int32_t NG = static_cast<int32_t>(gridDim.x) * gpc;
  const int32_t b0 = static_cast<int32_t>(blockIdx.x) * gpc + warp / G;
  const int32_t TB = static_cast<int32_t>(a.total_blocks);

  // ---- the ring: barriers, then the first two chunks' copies ----
  if (lane < kRingStages) mbar_init(bars + lane, 2);   // the bulk copies' arrival and the absmax copies'
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  __syncwarp();
  // copies of chunk c (of launch block b) into stage s: p, g and the code
  // streams in bulk (counted in bytes), the block's absmax values by cp.async
  // (counted by the second arrival)
  auto issue = [&](const ChunkRef& c, int s) {
    const DevTensor& d = a.t[c.t];
    unsigned char* st = ring + s * L::kStage;
    mbar_expect_tx(bars + s, L::kSA);
    bulk_g2s(st + L::kSP, static_cast<const unsigned char*>(d.p) + c.e0 * ES, 256 * ES, bars + s);
    bulk_g2s(st + L::kSG, static_cast<const unsigned char*>(d.g) + c.e0 * ES, 256 * ES, bars + s);
#pragma unroll
    for (int k = 0; k < NS; ++k)
      bulk_g2s(st + L::kSC + k * 256, code_stream<OPT>(d, k) + c.e0, 256, bars + s);
    const int32_t nbt = OPT == ADEMAMIX ? tensor_blocks(a, c.t) : 0;
#pragma unroll
    for (int k = 0; k < NS; ++k) cp_async4(st + L::kSA + 4 * k, absmax_stream<OPT>(d, k, nbt) + c.lb);
    cp_async_arrive(bars + s);
  };
  const bool stall_test = a.stall_test != 0 && blockIdx.x == 0 && warp == 0;
  // per stage (bit s): the parity to wait for; a chunk to wait for (want);
  // copies issued and not yet seen to land (inflight)
  uint32_t phase = 0u, want = 0u, inflight = 0u;
  // the cursor of the next chunk to issue (two ahead of the one computed);
  // each issued chunk leaves its ChunkRef in its stage's header
  ChunkCursor cur{0, b0};
  cursor_settle(a, cur);
  auto put_header = [&](const ChunkRef& c, int s) {
    if (lane == 0)
      *reinterpret_cast<int4*>(ring + s * L::kStage + L::kSH) =
          make_int4(static_cast<int>(c.e0), static_cast<int>(c.e0 >> 32), c.lb, c.t | (c.v << 16));
  };
  for (int s = 0; s < kRingStages; ++s) {
    const int32_t b = b0 + s * NG;
    if (b < TB) {
      const ChunkRef c = cursor_chunk<WHOLE>(a, cur, j);
      put_header(c, s);
      if (WHOLE || (c.v == 256 && (a.t[c.t].vec_ok & 2))) {
        // the stall test withholds this warp's first copy: its wait must run out
        const bool withhold = stall_test && s == 0;
        if (lane == 0 && !withhold) issue(c, s);
        want |= 1u << s;
        if (!withhold) inflight |= 1u << s;
      }
      cur.lb += NG;
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
  for (int32_t b = b0; b < TB; b += NG, s = (s + 1 == kRingStages) ? 0 : s + 1) {
    ChunkRef c;
    {
      const int4 h = *reinterpret_cast<const int4*>(ring + s * L::kStage + L::kSH);
      c.e0 = static_cast<int64_t>(static_cast<uint32_t>(h.x)) | (static_cast<int64_t>(h.y) << 32);
      c.lb = h.z;
      c.t = h.w & 0xffff;
      c.v = h.w >> 16;
    }
    const DevTensor& d = a.t[c.t];
    const int32_t nb = OPT == ADEMAMIX ? tensor_blocks(a, c.t) : 0;
    const int32_t lb = c.lb;
    float am[NS];

    float p[8], g[8];
    uint2 cw[NS];
    bool have = (WHOLE || c.v > 0) && ok;
    if ((want >> s) & 1u) {
      if (ok) {
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(bars + s, (phase >> s) & 1u, a.wait_ns));
        if (!ok) {
          have = false;
          if (lane == 0) atomicOr(a.status, kStatusWaitTimeout);
        }
      }
      if (ok) {
        phase ^= 1u << s;
        want &= ~(1u << s);
        inflight &= ~(1u << s);
        const unsigned char* st = ring + s * L::kStage;
        stage_load8<DT>(st + L::kSP, lane, p);
        stage_load8<DT>(st + L::kSG, lane, g);
#pragma unroll
        for (int k = 0; k < NS; ++k) cw[k] = stage_codes<DT>(st + L::kSC + k * 256, lane);
#pragma unroll
        for (int k = 0; k < NS; ++k) am[k] = reinterpret_cast<const float*>(st + L::kSA)[k];
      }
    } else if (!WHOLE && have) {
#pragma unroll
      for (int k = 0; k < NS; ++k) am[k] = absmax_stream<OPT>(d, k, nb)[lb];
      global_load8<DT>(d.p, c.e0, c.v, lane, p);
      global_load8<DT>(d.g, c.e0, c.v, lane, g);
#pragma unroll
      for (int k = 0; k < NS; ++k) cw[k] = global_codes<DT>(code_stream<OPT>(d, k), c.e0, c.v, lane);
    }
    // refill this stage with the chunk two ahead (its reads above are done)
    __syncwarp();
    if (ok) {
      const int32_t bn = b + kRingStages * NG;
      if (bn < TB) {
        const ChunkRef cn = cursor_chunk<WHOLE>(a, cur, j);
        if (lane == 0) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        put_header(cn, s);
        if (WHOLE || (cn.v == 256 && (a.t[cn.t].vec_ok & 2))) {
          if (lane == 0) issue(cn, s);
          want |= 1u << s;
          inflight |= 1u << s;
        }
        cur.lb += NG;
        cursor_settle(a, cur);
      }
    }

    // ---- dequantize and update; new states in sv, running max of |s| in mx ----
    float sv[NS][8];
    uint32_t mx[NS];
    float psq = 0.0f;        // sum of the new p^2 (the carried norm)
#pragma unroll
    for (int k = 0; k < NS; ++k) mx[k] = 0u;
    const float eff = a.step_size * (a.clip != nullptr ? a.clip[d.index] : 1.0f);
    if (have) {
      // optimizers whose direction is n / (sqrt(v) + eps)
      constexpr bool kRatio = OPT == ADAM || OPT == ADAMW || OPT == RMSPROP || OPT == ADAGRAD ||
                              OPT == ADEMAMIX;
      constexpr int kV = (OPT == ADAM || OPT == ADAMW) ? 1 : (OPT == ADEMAMIX ? 2 : 0);
      float gk[8];             // RMSprop, Adagrad: the scaled gradient, their numerator
      // running minima of (bits of v) - 1 and 2|n|'s bits - 2: a zero maps to
      // the top of the range, so a minimum below the threshold means a nonzero
      // v or numerator under 2^-100 (outside the fast ratio's range)
      uint32_t lo_v = 0xffffffffu, lo_n = 0xffffffffu;
      uint32_t nmax = 0u;      // max |numerator| of the lane (bit pattern)
      // pass 1: the new states (Momentum and Lion: also the new p)
#pragma unroll
      for (int e = 0; e < 8; e += 2) {
        float2 st[3];
#pragma unroll
        for (int k = 0; k < 3; ++k)
          st[k] = k < NS ? mul2(make_float2(sq[Traits<OPT>::map_of(k) * 256 + code_byte(cw[k], e)],
                                            sq[Traits<OPT>::map_of(k) * 256 + code_byte(cw[k], e + 1)]),
                                f2(am[k]))
                         : f2(0.0f);
        float2 pp = make_float2(p[e], p[e + 1]);
        float2 gg = mul2(make_float2(g[e], g[e + 1]), f2(a.gscale));
        if (!Traits<OPT>::DECOUPLED && a.wd != 0.0f) gg = fma2(f2(a.wd), pp, gg);
        if (OPT == ADAM || OPT == ADAMW) {
          const float2 m = fma2(f2(a.b1), st[0], mul2(f2(a.omb1), gg));
          const float2 v = fma2(f2(a.b2), st[1], mul2(f2(a.omb2), mul2(gg, gg)));
          sv[0][e] = m.x; sv[0][e + 1] = m.y;
          sv[1][e] = v.x; sv[1][e + 1] = v.y;
          lo_n = min_tiny_n(lo_n, m);
          lo_v = min_tiny_v(lo_v, v);
        } else if (OPT == RMSPROP || OPT == ADAGRAD) {
          const float2 v = OPT == RMSPROP ? fma2(f2(a.b1), st[0], mul2(f2(a.omb1), mul2(gg, gg)))
                                          : fma2(gg, gg, st[0]);
          sv[0][e] = v.x; sv[0][e + 1] = v.y;
          gk[e] = gg.x; gk[e + 1] = gg.y;
          nmax = absmax_nan(nmax, gg.x, gg.y);
          lo_n = min_tiny_n(lo_n, gg);
          lo_v = min_tiny_v(lo_v, v);
        } else if (OPT == ADEMAMIX) {
          const float2 m1 = fma2(f2(a.b1), st[0], mul2(f2(a.omb1), gg));
          const float2 m2 = fma2(f2(a.b3t), st[1], mul2(f2(a.omb3t), gg));
          const float2 nu = fma2(f2(a.b2), st[2], mul2(f2(a.omb2), mul2(gg, gg)));
          const float2 num = fma2(m1, f2(a.inv_bc1), mul2(f2(a.alpha_t), m2));
          sv[0][e] = m1.x; sv[0][e + 1] = m1.y;
          sv[1][e] = m2.x; sv[1][e + 1] = m2.y;
          sv[2][e] = nu.x; sv[2][e + 1] = nu.y;
          nmax = absmax_nan(nmax, num.x, num.y);
          lo_n = min_tiny_n(lo_n, num);
          lo_v = min_tiny_v(lo_v, nu);
        } else if (OPT == MOMENTUM) {
          const float2 m = fma2(f2(a.b1), st[0], gg);
          sv[0][e] = m.x; sv[0][e + 1] = m.y;
          pair_apply<OPT>(a, -eff, pp, m);
          p[e] = pp.x; p[e + 1] = pp.y;
        } else {  // LION
          const float2 c = fma2(f2(a.b1), st[0], mul2(f2(a.omb1), gg));
          float2 u;
          u.x = c.x > 0.0f ? 1.0f : (c.x < 0.0f ? -1.0f : 0.0f);
          u.y = c.y > 0.0f ? 1.0f : (c.y < 0.0f ? -1.0f : 0.0f);
          const float2 m = fma2(f2(a.b2), st[0], mul2(f2(a.omb2), gg));
          sv[0][e] = m.x; sv[0][e + 1] = m.y;
          pair_apply<OPT>(a, -eff, pp, u);
          p[e] = pp.x; p[e + 1] = pp.y;
        }
      }
      // absent elements of a partial chunk keep state 0 (they do not count in the absmax)
      if (!WHOLE && c.v < 256) {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int o = quad_offset<DT>(lane, q);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (o + e >= c.v) {
#pragma unroll
              for (int k = 0; k < NS; ++k) sv[k][4 * q + e] = 0.0f;
              if (OPT == RMSPROP || OPT == ADAGRAD) gk[4 * q + e] = 0.0f;
            }
        }
      }
#pragma unroll
      for (int k = 0; k < NS; ++k)
#pragma unroll
        for (int e = 0; e < 8; e += 2) mx[k] = absmax_nan(mx[k], sv[k][e], sv[k][e + 1]);
      if constexpr (kRatio) {
        // pass 2: u = n / (sqrt(v) + eps) and the new p; the fast ratio when
        // every operand of the lane lies in its range, the IEEE operations else
        if (OPT == ADAM || OPT == ADAMW) nmax = mx[0];
        const bool fast = lo_v >= kRatioLoV && lo_n >= kRatioLoN && a.eps_hat >= 0x1p-60f &&
                          a.eps_hat <= 0x1p20f && mx[kV] <= kRatioMaxV && nmax <= kRatioMaxN;
        auto numer = [&](int e) -> float2 {
          if (OPT == RMSPROP || OPT == ADAGRAD) return make_float2(gk[e], gk[e + 1]);
          if (OPT == ADEMAMIX)
            return fma2(make_float2(sv[0][e], sv[0][e + 1]), f2(a.inv_bc1),
                        mul2(f2(a.alpha_t), make_float2(sv[1][e], sv[1][e + 1])));
          return make_float2(sv[0][e], sv[0][e + 1]);
        };
        if (fast) {
#pragma unroll
          for (int e = 0; e < 8; e += 2) {
            const float2 u = ratio2_fast(numer(e), make_float2(sv[kV][e], sv[kV][e + 1]), a.eps_hat);
            float2 pp = make_float2(p[e], p[e + 1]);
            pair_apply<OPT>(a, -eff, pp, u);
            p[e] = pp.x; p[e + 1] = pp.y;
          }
        } else {
#pragma unroll
          for (int e = 0; e < 8; e += 2) {
            const float2 u = ratio2_ieee_slow(numer(e), make_float2(sv[kV][e], sv[kV][e + 1]), a.eps_hat);
            float2 pp = make_float2(p[e], p[e + 1]);
            pair_apply<OPT>(a, -eff, pp, u);
            p[e] = pp.x; p[e + 1] = pp.y;
          }
        }
      }
      ring_store8<DT>(d.p, c.e0, WHOLE ? 256 : c.v, WHOLE || (d.vec_ok & 1) != 0, lane, p);
      if (a.carry_out) {
        // the squares of p as stored (rounded to the dtype); the registers
        // of a ragged chunk's absent elements hold no parameter
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float q = Elem<DT>::stored(p[e]);
          if (WHOLE || quad_offset<DT>(lane, e >> 2) + (e & 3) < c.v) psq = psq + q * q;
        }
      }
    } else {
#pragma unroll
      for (int k = 0; k < NS; ++k)
#pragma unroll
        for (int e = 0; e < 8; ++e) sv[k][e] = 0.0f;
    }

    // ---- the block's new absmax (every warp of the group takes part) ----
    ring_group_max<NS>(mx, G, warp, lane, sred, parity);
    parity ^= 1;
    if (a.carry_out) {
      const float bsq = ring_group_sum(psq, G, warp, lane, sred, parity);
      parity ^= 1;
      if (have && j == 0 && lane == 0)
        reinterpret_cast<float*>(a.partials + d.first_block + lb)[1] = bsq;
    }
    if (!have) continue;

    // ---- requantize and store codes (and, once per block, the absmax) ----
    // The usual case: every state's absmax lies in [2^-125, 2^125] (or is 0,
    // an all-zero block) and every map takes the table: one Newton
    // reciprocal per state and the table lookups, no other tests.
    uint32_t enc[NS][8];
    bool usual = true;
#pragma unroll
    for (int k = 0; k < NS; ++k) {
      const int m = Traits<OPT>::map_of(k);
      usual = usual && fast_map[m] && (mx[k] - 0x01000000u <= 0x7D000000u || mx[k] == 0u) &&
              (!Traits<OPT>::nonneg(k) || nonneg_map[m]);
    }
    if (usual) {
#pragma unroll
      for (int k = 0; k < NS; ++k) {
        const float amk = __uint_as_float(mx[k]);
        const float y = rcp_approx(amk);
        const float r = __fmaf_rn(__fmaf_rn(-amk, y, 1.0f), y, y);
        const float inv = mx[k] == 0u ? 0.0f : r;
        const uint32_t* tz = stbl + Traits<OPT>::map_of(k) * kTblSize + kTblZero;
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
          const float2 xn = mul2(make_float2(sv[k][e], sv[k][e + 1]), f2(inv));
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
        const float inv = rcp_block(__uint_as_float(mx[k]));
        const bool fast = fast_map[m] && mx[k] <= 0x7f7fffffu && inv <= FLT_MAX;
        const uint32_t* tz = stbl + m * kTblSize + kTblZero;
        const float* md = smid + m * 256;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          if (!fast) enc[k][e] = encode_search(sv[k][e] * inv, md);
          else if (Traits<OPT>::nonneg(k) && nonneg_map[m]) enc[k][e] = encode_fast_nonneg(sv[k][e], inv, tz);
          else enc[k][e] = encode_fast(sv[k][e], inv, tz);
        }
      }
    }
#pragma unroll
    for (int k = 0; k < NS; ++k) {
      // byte 2 of each entry is the code
      const uint32_t lo = __byte_perm(__byte_perm(enc[k][0], enc[k][1], 0x0062u),
                                      __byte_perm(enc[k][2], enc[k][3], 0x0062u), 0x5410u);
      const uint32_t hi = __byte_perm(__byte_perm(enc[k][4], enc[k][5], 0x0062u),
                                      __byte_perm(enc[k][6], enc[k][7], 0x0062u), 0x5410u);
      ring_store_codes<DT>(const_cast<uint8_t*>(code_stream<OPT>(d, k)), c.e0, WHOLE ? 256 : c.v,
                           WHOLE || (d.vec_ok & 1) != 0, lane, make_uint2(lo, hi));
      if (j == 0 && lane == 0) absmax_stream<OPT>(d, k, nb)[lb] = __uint_as_float(mx[k]);
    }
  }

  if (a.carry_writer && blockIdx.x == 0 && threadIdx.x == 0) *a.carry_stamp = a.carry_write;

  // ---- a wait ran out: let this warp's copies still in flight land ----
  if (!ok && lane == 0) {
    for (int s = 0; s < kRingStages; ++s)
      if ((inflight >> s) & 1u) mbar_wait_bounded(bars + s, (phase >> s) & 1u, a.wait_ns);
  }
}

// CTA size for a launch: as many warps as the ring holds, whole groups.
// (at most 15 groups: named barriers 1..15 are the groups' meeting points)
template <int OPT, int DT>
__host__ __forceinline__ int ring_threads(int log2B) {
  const int G = log2B > 8 ? (1 << (log2B - 8)) : 1;
  int groups = RingSmem<OPT, DT>::kWarps / G;
  if (G > 1 && groups > 15) groups = 15;
  return groups * G * 32;
}

template <int OPT, int DT, bool WHOLE>
cudaError_t launch_step8_ring_w(const StepArgs& a, cudaStream_t s) {
  using L = RingSmem<OPT, DT>;
  static std::atomic<unsigned char> configured[kMaxDevices];
  cudaError_t e = set_smem_limit_once(reinterpret_cast<const void*>(k_step8_ring<OPT, DT, WHOLE>),
                                      L::kBytes, configured);
  if (e != cudaSuccess) return e;
  const int threads = ring_threads<OPT, DT>(a.log2B);
  const int G = a.log2B > 8 ? (1 << (a.log2B - 8)) : 1;
  const int64_t groups = threads / 32 / G;
  const int64_t need = (a.total_blocks + groups - 1) / groups;
  const int grid = static_cast<int>(need < a.nsm ? need : a.nsm);
  k_step8_ring<OPT, DT, WHOLE><<<grid, threads, L::kBytes, s>>>(a);
  return cudaGetLastError();
}

template <int OPT, int DT>
cudaError_t launch_step8_ring(const StepArgs& a, cudaStream_t s) {
  return a.whole ? launch_step8_ring_w<OPT, DT, true>(a, s) : launch_step8_ring_w<OPT, DT, false>(a, s);
}

}  // namespace bnb8
