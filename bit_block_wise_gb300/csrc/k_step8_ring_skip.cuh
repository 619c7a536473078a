// k_step8_ring_skip.cuh -- the 8-bit step with skip_zeros on a per-warp ring
// (blocksize 256).
//
// skip_zeros ("Support skip_zeros in the XPU Triton optimizer kernels
// #2097"): an element whose raw gradient is exactly zero keeps its parameter
// and state; a block whose gradient is all zero is not touched at all.  On
// sparse gradients (an embedding whose rows are mostly zero) most blocks are
// such blocks, so the step is a stream of g with a few live blocks in it.
//
// Here every warp streams the gradient of its 512-element chunks through a
// ring of shared-memory stages (bulk copies, as in k_step8_ring, but of g
// alone, so the ring holds several chunks ahead).  A chunk with a nonzero
// gradient in either of its two blocks then fetches its p, codes and absmax
// into the warp's own live buffer (bulk copies on a second mbarrier, one
// round trip per chunk), and its live blocks are stepped and requantized
// exactly as in the plain step, with the skipped elements' old parameter and
// dequantized states kept.  Blocks with an all-zero gradient cost a
// shared-memory read and a warp vote on the OR of the raw gradient words'
// magnitude bits; only live blocks are widened to binary32.  The warps of a
// CTA take their chunks from a shared counter, so that the warp that meets
// more live chunks takes fewer.
#pragma once

#include "k_step8_ring.cuh"

namespace bnb8 {

template <int OPT, int DT>
struct SkipSmem {
  static constexpr int NS = Traits<OPT>::NS;
  static constexpr int NM = Traits<OPT>::NM;
  static constexpr int ES = DT == DT_F32 ? 4 : 2;
  static constexpr int kWarps = 24;
  // one stage: g of a chunk | header
  static constexpr int kSG = 0;
  static constexpr int kSH = kChunk * ES;
  static constexpr int kStage = kSH + 16;
  // the warp's live buffer: a chunk's p | codes of each state | absmax [block][state]
  static constexpr int kLP = 0;
  static constexpr int kLC = kChunk * ES;
  static constexpr int kLA = kLC + NS * kChunk;
  static constexpr int kLive = kLA + 32;
  static_assert(2 * NS * 4 <= 32, "absmax slots of two blocks");
  static_assert(kStage % 16 == 0 && kLive % 16 == 0, "16-byte alignment");
  // CTA layout: maps, midpoints, bucket tables, rings, stage barriers, live
  // buffers, live barriers
  static constexpr int kQ = 0;
  static constexpr int kMid = kQ + NM * 256 * 4;
  static constexpr int kTbl = kMid + NM * 256 * 4;
  static constexpr int kRing = kTbl + NM * kTblSize * 4;
  static constexpr int kBudget = 232448 - 1024;
  static constexpr int per_warp(int s) { return s * (kStage + 8) + kLive + 8; }
  // as many stages (up to 4) as fit: the ring runs that many chunks ahead
  static constexpr int kStages = kRing + kWarps * per_warp(4) <= kBudget   ? 4
                                 : kRing + kWarps * per_warp(3) <= kBudget ? 3
                                 : kRing + kWarps * per_warp(2) <= kBudget ? 2
                                                                           : 1;
  static_assert(kRing + kWarps * per_warp(kStages) <= kBudget, "the ring fits");
  static constexpr int kBars = kRing + kWarps * kStages * kStage;
  static constexpr int kLive0 = kBars + kWarps * kStages * 8;
  static_assert(kLive0 % 16 == 0, "live buffers keep 16-byte alignment");
  static constexpr int kLiveBars = kLive0 + kWarps * kLive;
  static constexpr int kBytes = kLiveBars + kWarps * 8;
};

// A lane's 8 gradient elements of one pass as they sit in a stage (the
// layout of stage_load: one 16-byte word group for 16-bit values, two for
// binary32), before they are widened.
template <int DT>
struct RawG {
  uint4 w[DT == DT_F32 ? 2 : 1];
};
template <int DT>
__device__ __forceinline__ void stage_raw(const unsigned char* base, int lane, int q0, RawG<DT>& r) {
  if (DT == DT_F32) {
#pragma unroll
    for (int i = 0; i < 2; ++i) r.w[i] = reinterpret_cast<const uint4*>(base + (q0 + i) * 512)[lane];
  } else {
    r.w[0] = reinterpret_cast<const uint4*>(base + (q0 / 2) * 512)[lane];
  }
}
// The same from global memory (a ragged chunk), absent elements as 0.
template <int DT>
__device__ __forceinline__ void global_raw(const void* base, int64_t e0, int v, int lane, int q0,
                                           RawG<DT>& r) {
  if (DT == DT_F32) {
    const uint32_t* b = static_cast<const uint32_t*>(base) + e0;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int o = quad_offset<DT>(lane, q0 + i);
      r.w[i].x = o < v ? b[o] : 0u;
      r.w[i].y = o + 1 < v ? b[o + 1] : 0u;
      r.w[i].z = o + 2 < v ? b[o + 2] : 0u;
      r.w[i].w = o + 3 < v ? b[o + 3] : 0u;
    }
  } else {
    const uint16_t* b = static_cast<const uint16_t*>(base) + e0;
    const int o = quad_offset<DT>(lane, q0);   // 8 consecutive elements
    uint32_t h[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) h[k] = o + k < v ? b[o + k] : 0u;
    r.w[0] = make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16),
                        h[6] | (h[7] << 16));
  }
}
template <int DT>
__device__ __forceinline__ void raw_zero(RawG<DT>& r) {
#pragma unroll
  for (int i = 0; i < (DT == DT_F32 ? 2 : 1); ++i) r.w[i] = make_uint4(0u, 0u, 0u, 0u);
}
// Whether any of the 8 values is nonzero: the OR of their magnitude bits
// (+0 and -0 are zero; subnormals, infinities and NaN are not), which is
// the comparison g != 0 on each value.
template <int DT>
__device__ __forceinline__ bool raw_nonzero(const RawG<DT>& r) {
  constexpr uint32_t kMag = DT == DT_F32 ? 0x7fffffffu : 0x7fff7fffu;
  uint32_t o = 0u;
#pragma unroll
  for (int i = 0; i < (DT == DT_F32 ? 2 : 1); ++i) o |= r.w[i].x | r.w[i].y | r.w[i].z | r.w[i].w;
  return (o & kMag) != 0u;
}
// The values, in stage_load's order.
template <int DT>
__device__ __forceinline__ void raw_widen(const RawG<DT>& r, float (&x)[8]) {
  if (DT == DT_F32) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      x[4 * i] = __uint_as_float(r.w[i].x); x[4 * i + 1] = __uint_as_float(r.w[i].y);
      x[4 * i + 2] = __uint_as_float(r.w[i].z); x[4 * i + 3] = __uint_as_float(r.w[i].w);
    }
  } else {
    const uint4 v = r.w[0];
    x[0] = lo_half(v.x, DT); x[1] = hi_half(v.x, DT);
    x[2] = lo_half(v.y, DT); x[3] = hi_half(v.y, DT);
    x[4] = lo_half(v.z, DT); x[5] = hi_half(v.z, DT);
    x[6] = lo_half(v.w, DT); x[7] = hi_half(v.w, DT);
  }
}

// WHOLE: every tensor of the launch is aligned for bulk copies and a
// multiple of 512 elements (the host checked it).
template <int OPT, int DT, bool WHOLE>
__global__ void __launch_bounds__(24 * 32, 1) k_step8_skip_ring(const __grid_constant__ StepArgs a) {
  using L = SkipSmem<OPT, DT>;
  constexpr int NS = L::NS;
  constexpr int NM = L::NM;
  constexpr int ES = L::ES;
  constexpr int kStages = L::kStages;
  extern __shared__ __align__(128) unsigned char ring_smem[];
  unsigned char* smem = ring_smem;
  float* sq = reinterpret_cast<float*>(smem + L::kQ);
  float* smid = reinterpret_cast<float*>(smem + L::kMid);
  uint32_t* stbl = reinterpret_cast<uint32_t*>(smem + L::kTbl);
  __shared__ int s_bad[2];
  __shared__ int s_below[2];
  __shared__ int s_scan[2 * 32];
  __shared__ int32_t s_next;   // the CTA's next chunk to hand out

  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  if (tid == 0) s_next = 0;
  __syncthreads();
  unsigned char* ring = smem + L::kRing + warp * kStages * L::kStage;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBars) + warp * kStages;
  unsigned char* live = smem + L::kLive0 + warp * L::kLive;
  uint64_t* lbar = reinterpret_cast<uint64_t*>(smem + L::kLiveBars) + warp;

  // The CTA's units are blockIdx.x + k * gridDim.x; its warps take the next
  // k from a shared counter as they go (a warp's units still ascend).  Live
  // chunks cost far more than dead ones and fall at random, so a fixed
  // share per warp would leave the warp with the most live chunks running
  // long after the others.
  const int32_t TB = static_cast<int32_t>(a.ring_units);
  auto grab = [&]() -> int32_t {
    int32_t k = 0;
    if (lane == 0) k = atomicAdd(&s_next, 1);
    k = __shfl_sync(0xffffffffu, k, 0);
    // (k exceeds TB / gridDim by at most one take per stage of each warp,
    // so u does not wrap)
    const uint32_t u = blockIdx.x + static_cast<uint32_t>(k) * gridDim.x;
    return u < static_cast<uint32_t>(TB) ? static_cast<int32_t>(u) : TB;
  };

  // ---- the ring of gradient chunks, and the live buffer ----
  if (lane < kStages) mbar_init(bars + lane, 1);   // the bulk copy's arrival
  if (lane == 0) mbar_init(lbar, 2);               // the bulk copies' arrival and the absmax copies'
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  __syncwarp();
  auto issue = [&](const ChunkRef& c, int s) {
    const DevTensor& d = a.t[c.t];
    mbar_expect_tx(bars + s, kChunk * ES);
    bulk_g2s(ring + s * L::kStage + L::kSG, static_cast<const unsigned char*>(d.g) + c.e0 * ES,
             kChunk * ES, bars + s);
  };
  uint32_t phase = 0u, want = 0u, inflight = 0u;
  uint32_t lphase = 0u;
  bool linflight = false;
  ChunkCursor cur{0, 0};
  int32_t at = 0;              // the cursor's unit over the launch
  uint32_t held = 0u;          // stages holding a chunk
  auto move_to = [&](int32_t un) {
    cur.u += un - at;
    at = un;
    cursor_settle(a, cur);
  };
  auto put_header = [&](const ChunkRef& c, int s) {
    if (lane == 0)
      *reinterpret_cast<int4*>(ring + s * L::kStage + L::kSH) =
          make_int4(static_cast<int>(c.e0), static_cast<int>(c.e0 >> 32), c.u, c.t | (c.v << 16));
  };
  for (int s = 0; s < kStages; ++s) {
    const int32_t un = grab();
    if (un >= TB) break;
    move_to(un);
    const ChunkRef c = cursor_chunk<WHOLE>(a, cur, 0);
    put_header(c, s);
    if (WHOLE || (c.v == kChunk && (a.t[c.t].vec_ok & 2))) {
      if (lane == 0) issue(c, s);
      want |= 1u << s;
      inflight |= 1u << s;
    }
    held |= 1u << s;
  }
  __syncwarp();

  // ---- maps, midpoints and bucket tables ----
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
  bool ok = true;
  // the stages are refilled in turn, so those holding a chunk follow each
  // other from s on; the loop ends at the first empty one
  for (int s = 0; (held >> s) & 1u; s = (s + 1 == kStages) ? 0 : s + 1) {
    ChunkRef c;
    {
      const int4 h = *reinterpret_cast<const int4*>(ring + s * L::kStage + L::kSH);
      c.e0 = static_cast<int64_t>(static_cast<uint32_t>(h.x)) | (static_cast<int64_t>(h.y) << 32);
      c.u = h.z;
      c.t = h.w & 0xffff;
      c.v = h.w >> 16;
    }
    const DevTensor& d = a.t[c.t];
    const bool have = (WHOLE || c.v > 0) && ok;
    bool staged = false;
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
    // ---- the gradient of both blocks of the chunk: from a stage as raw
    // ---- words (whether a block is live is a test on their bits; only a
    // ---- live block's are widened), from global memory as values ----
    RawG<DT> gr[2];
    int vbs[2];
#pragma unroll
    for (int pass = 0; pass < 2; ++pass) {
      const int rest = c.v - 256 * pass;
      vbs[pass] = WHOLE ? 256 : (rest > 256 ? 256 : (rest > 0 ? rest : 0));
      if (staged) stage_raw<DT>(ring + s * L::kStage + L::kSG, lane, 2 * pass, gr[pass]);
      else if (!WHOLE && have && vbs[pass] > 0) global_raw<DT>(d.g, c.e0, c.v, lane, 2 * pass, gr[pass]);
      else raw_zero<DT>(gr[pass]);   // (absent elements read as 0)
    }
    // refill this stage with the warp's next chunk
    __syncwarp();
    held &= ~(1u << s);
    if (ok) {
      const int32_t un = grab();
      if (un < TB) {
        move_to(un);
        const ChunkRef cn = cursor_chunk<WHOLE>(a, cur, 0);
        if (lane == 0) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        put_header(cn, s);
        if (WHOLE || (cn.v == kChunk && (a.t[cn.t].vec_ok & 2))) {
          if (lane == 0) issue(cn, s);
          want |= 1u << s;
          inflight |= 1u << s;
        }
        held |= 1u << s;
      }
    }
    if (!(have && ok)) continue;
    // a block whose raw gradient is all zero is left as it is
    bool blk_live[2];
#pragma unroll
    for (int pass = 0; pass < 2; ++pass) blk_live[pass] = __any_sync(0xffffffffu, raw_nonzero<DT>(gr[pass]));
    if (!blk_live[0] && !blk_live[1]) continue;
    float gc[2][8];
#pragma unroll
    for (int pass = 0; pass < 2; ++pass) raw_widen<DT>(gr[pass], gc[pass]);
    const float eff = a.step_size * (a.clip != nullptr ? a.clip[d.index] : 1.0f);
    const bool vec = WHOLE || (d.vec_ok & 1) != 0;

    // ---- the live chunk's p, codes and absmax, one round trip ----
    const bool bulk = WHOLE || (c.v == kChunk && (d.vec_ok & 2));
    if (bulk) {
      // (the buffer's previous contents were read before this warp's votes)
      if (lane == 0) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_expect_tx(lbar, kChunk * ES + NS * kChunk);
        bulk_g2s(live + L::kLP, static_cast<const unsigned char*>(d.p) + c.e0 * ES, kChunk * ES, lbar);
#pragma unroll
        for (int k = 0; k < NS; ++k)
          bulk_g2s(live + L::kLC + k * kChunk, code_stream<OPT>(d, k) + c.e0, kChunk, lbar);
#pragma unroll
        for (int k = 0; k < NS; ++k) {
          cp_async4(live + L::kLA + 4 * k, absmax_stream<OPT>(d, k) + 2 * c.u);
          cp_async4(live + L::kLA + 4 * (NS + k), absmax_stream<OPT>(d, k) + 2 * c.u + 1);
        }
        cp_async_arrive(lbar);
      }
      linflight = true;
      ok = __all_sync(0xffffffffu, mbar_wait_bounded(lbar, lphase, a.wait_ns));
      if (!ok) {
        if (lane == 0) atomicOr(a.status, kStatusWaitTimeout);
        continue;
      }
      lphase ^= 1u;
      linflight = false;
    }

#pragma unroll
    for (int pass = 0; pass < 2; ++pass) {
      if (!blk_live[pass]) continue;
      const int q0 = 2 * pass;
      const int vb = vbs[pass];
      const float (&g)[8] = gc[pass];
      const int32_t lb = 2 * c.u + pass;
      float p[8];
      uint32_t cw[NS][2];
      float am[NS];
      if (bulk) {
        stage_load<DT, 2>(live + L::kLP, lane, q0, p);
#pragma unroll
        for (int k = 0; k < NS; ++k) stage_codes<DT, 2>(live + L::kLC + k * kChunk, lane, q0, cw[k]);
#pragma unroll
        for (int k = 0; k < NS; ++k) am[k] = reinterpret_cast<const float*>(live + L::kLA)[pass * NS + k];
      } else {
        global_load<DT, 2>(d.p, c.e0, c.v, lane, q0, p);
#pragma unroll
        for (int k = 0; k < NS; ++k) global_codes<DT, 2>(code_stream<OPT>(d, k), c.e0, c.v, lane, q0, cw[k]);
#pragma unroll
        for (int k = 0; k < NS; ++k) am[k] = absmax_stream<OPT>(d, k)[lb];
      }

      // ---- dequantize and update; a zero raw gradient keeps the element's
      // ---- parameter and its old (dequantized) states ----
      constexpr bool kRatio = OPT == ADAM || OPT == ADAMW || OPT == RMSPROP || OPT == ADAGRAD ||
                              OPT == ADEMAMIX;
      constexpr int kV = (OPT == ADAM || OPT == ADAMW) ? 1 : (OPT == ADEMAMIX ? 2 : 0);
      float sv[NS][8];
      float gk[8];
      uint32_t mx[NS];
#pragma unroll
      for (int k = 0; k < NS; ++k) mx[k] = 0u;
      uint32_t lo_v = 0xffffffffu, lo_n = 0xffffffffu, nmax = 0u;
      auto keep = [](bool skip, float old_v, float new_v) { return skip ? old_v : new_v; };
#pragma unroll
      for (int e = 0; e < 8; e += 2) {
        const bool k0 = g[e] == 0.0f, k1 = g[e + 1] == 0.0f;
        float2 stt[3];
#pragma unroll
        for (int k = 0; k < 3; ++k)
          stt[k] = k < NS ? mul2(make_float2(sq[Traits<OPT>::map_of(k) * 256 + code_of<2>(cw[k], e)],
                                             sq[Traits<OPT>::map_of(k) * 256 + code_of<2>(cw[k], e + 1)]),
                                 f2(am[k]))
                          : f2(0.0f);
        float2 pp = make_float2(p[e], p[e + 1]);
        float2 gg = mul2(make_float2(g[e], g[e + 1]), f2(a.gscale));
        if (!Traits<OPT>::DECOUPLED && a.wd != 0.0f) gg = fma2(f2(a.wd), pp, gg);
        if (OPT == ADAM || OPT == ADAMW) {
          const float2 m = fma2(f2(a.b1), stt[0], mul2(f2(a.omb1), gg));
          const float2 v = fma2(f2(a.b2), stt[1], mul2(f2(a.omb2), mul2(gg, gg)));
          sv[0][e] = keep(k0, stt[0].x, m.x); sv[0][e + 1] = keep(k1, stt[0].y, m.y);
          sv[1][e] = keep(k0, stt[1].x, v.x); sv[1][e + 1] = keep(k1, stt[1].y, v.y);
          lo_n = min_tiny_n(lo_n, make_float2(sv[0][e], sv[0][e + 1]));
          lo_v = min_tiny_v(lo_v, make_float2(sv[1][e], sv[1][e + 1]));
        } else if (OPT == RMSPROP || OPT == ADAGRAD) {
          const float2 v = OPT == RMSPROP ? fma2(f2(a.b1), stt[0], mul2(f2(a.omb1), mul2(gg, gg)))
                                          : fma2(gg, gg, stt[0]);
          sv[0][e] = keep(k0, stt[0].x, v.x); sv[0][e + 1] = keep(k1, stt[0].y, v.y);
          gk[e] = gg.x; gk[e + 1] = gg.y;
          nmax = absmax_nan(nmax, gg.x, gg.y);
          lo_n = min_tiny_n(lo_n, gg);
          lo_v = min_tiny_v(lo_v, make_float2(sv[0][e], sv[0][e + 1]));
        } else if (OPT == ADEMAMIX) {
          const float2 m1 = fma2(f2(a.b1), stt[0], mul2(f2(a.omb1), gg));
          const float2 m2 = fma2(f2(a.b3t), stt[1], mul2(f2(a.omb3t), gg));
          const float2 nu = fma2(f2(a.b2), stt[2], mul2(f2(a.omb2), mul2(gg, gg)));
          sv[0][e] = keep(k0, stt[0].x, m1.x); sv[0][e + 1] = keep(k1, stt[0].y, m1.y);
          sv[1][e] = keep(k0, stt[1].x, m2.x); sv[1][e + 1] = keep(k1, stt[1].y, m2.y);
          sv[2][e] = keep(k0, stt[2].x, nu.x); sv[2][e + 1] = keep(k1, stt[2].y, nu.y);
          const float2 num = fma2(make_float2(sv[0][e], sv[0][e + 1]), f2(a.inv_bc1),
                                  mul2(f2(a.alpha_t), make_float2(sv[1][e], sv[1][e + 1])));
          nmax = absmax_nan(nmax, num.x, num.y);
          lo_n = min_tiny_n(lo_n, num);
          lo_v = min_tiny_v(lo_v, make_float2(sv[2][e], sv[2][e + 1]));
        } else if (OPT == MOMENTUM) {
          const float2 m = fma2(f2(a.b1), stt[0], gg);
          sv[0][e] = keep(k0, stt[0].x, m.x); sv[0][e + 1] = keep(k1, stt[0].y, m.y);
          pair_apply<OPT>(a, -eff, pp, m);
          p[e] = keep(k0, p[e], pp.x); p[e + 1] = keep(k1, p[e + 1], pp.y);
        } else {  // LION
          const float2 cc = fma2(f2(a.b1), stt[0], mul2(f2(a.omb1), gg));
          const float2 m = fma2(f2(a.b2), stt[0], mul2(f2(a.omb2), gg));
          sv[0][e] = keep(k0, stt[0].x, m.x); sv[0][e + 1] = keep(k1, stt[0].y, m.y);
          // p + (-eff)*sign(c), the product formed by bits (lion_term)
          if (Traits<OPT>::DECOUPLED && a.wd != 0.0f) pp = mul2(pp, f2(a.decay));
          pp = __fadd2_rn(pp, lion_term(-eff, cc));
          p[e] = keep(k0, p[e], pp.x); p[e + 1] = keep(k1, p[e + 1], pp.y);
        }
      }
      // absent elements of a partial chunk keep state 0 (they do not count in the absmax)
      if (!WHOLE && vb < 256) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int o = quad_offset<DT>(lane, q0 + i) - 256 * pass;
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (o + e >= vb) {
#pragma unroll
              for (int k = 0; k < NS; ++k) sv[k][4 * i + e] = 0.0f;
              if (OPT == RMSPROP || OPT == ADAGRAD) gk[4 * i + e] = 0.0f;
            }
        }
      }
#pragma unroll
      for (int k = 0; k < NS; ++k)
#pragma unroll
        for (int e = 0; e < 8; e += 2) mx[k] = absmax_nan(mx[k], sv[k][e], sv[k][e + 1]);
      if constexpr (kRatio) {
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
        auto apply = [&](int e, float2 u) {
          float2 pp = make_float2(p[e], p[e + 1]);
          pair_apply<OPT>(a, -eff, pp, u);
          p[e] = keep(g[e] == 0.0f, p[e], pp.x);
          p[e + 1] = keep(g[e + 1] == 0.0f, p[e + 1], pp.y);
        };
        if (fast) {
#pragma unroll
          for (int e = 0; e < 8; e += 2)
            apply(e, ratio2_fast(numer(e), make_float2(sv[kV][e], sv[kV][e + 1]), a.eps_hat));
        } else {
#pragma unroll
          for (int e = 0; e < 8; e += 2)
            apply(e, ratio2_ieee_slow(numer(e), make_float2(sv[kV][e], sv[kV][e + 1]), a.eps_hat));
        }
      }
      ring_store<DT, 2>(d.p, c.e0, WHOLE ? kChunk : c.v, vec, lane, q0, p);

      // ---- the block's new absmax, requantization, codes and absmax ----
#pragma unroll
      for (int k = 0; k < NS; ++k) mx[k] = __reduce_max_sync(0xffffffffu, mx[k]);
      uint32_t enc[NS][8];
#pragma unroll
      for (int k = 0; k < NS; ++k) {
        const int m = Traits<OPT>::map_of(k);
        const uint32_t* tz = stbl + m * kTblSize + kTblZero;
        const float inv = rcp_block(__uint_as_float(mx[k]));
        const bool fastk = fast_map[m] && mx[k] <= 0x7f7fffffu && inv <= FLT_MAX;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          if (!fastk) enc[k][e] = encode_search(sv[k][e] * inv, smid + m * 256);
          else if (Traits<OPT>::nonneg(k) && nonneg_map[m]) enc[k][e] = encode_fast_nonneg(sv[k][e], inv, tz);
          else enc[k][e] = encode_fast(sv[k][e], inv, tz);
        }
        uint32_t w[2];
#pragma unroll
        for (int i = 0; i < 2; ++i)
          w[i] = __byte_perm(__byte_perm(enc[k][4 * i], enc[k][4 * i + 1], 0x0062u),
                             __byte_perm(enc[k][4 * i + 2], enc[k][4 * i + 3], 0x0062u), 0x5410u);
        ring_store_codes<DT, 2>(const_cast<uint8_t*>(code_stream<OPT>(d, k)), c.e0, WHOLE ? kChunk : c.v,
                                vec, lane, q0, w);
        if (lane == 0) absmax_stream<OPT>(d, k)[lb] = __uint_as_float(mx[k]);
      }
    }
  }

  // ---- a wait ran out: let this warp's copies still in flight land ----
  if (!ok && lane == 0) {
    for (int s2 = 0; s2 < kStages; ++s2)
      if ((inflight >> s2) & 1u) mbar_wait_bounded(bars + s2, (phase >> s2) & 1u, a.wait_ns);
    if (linflight) mbar_wait_bounded(lbar, lphase, a.wait_ns);
  }
}

template <int OPT, int DT, bool WHOLE>
cudaError_t launch_step8_skip_ring_w(const StepArgs& a, cudaStream_t s) {
  using L = SkipSmem<OPT, DT>;
  static std::atomic<unsigned char> configured[kMaxDevices];
  cudaError_t e = set_smem_limit_once(reinterpret_cast<const void*>(k_step8_skip_ring<OPT, DT, WHOLE>),
                                      L::kBytes, configured);
  if (e != cudaSuccess) return e;
  const int threads = L::kWarps * 32;
  const int64_t need = (a.ring_units + L::kWarps - 1) / L::kWarps;
  const int grid = static_cast<int>(need < a.nsm ? need : a.nsm);
  k_step8_skip_ring<OPT, DT, WHOLE><<<grid, threads, L::kBytes, s>>>(a);
  return cudaGetLastError();
}

// skip_zeros, blocksize 256 (the caller checks both).
template <int OPT, int DT>
cudaError_t launch_step8_skip_ring(const StepArgs& a, cudaStream_t s) {
  return a.whole ? launch_step8_skip_ring_w<OPT, DT, true>(a, s)
                 : launch_step8_skip_ring_w<OPT, DT, false>(a, s);
}

}  // namespace bnb8
