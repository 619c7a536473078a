// k_step8.cuh -- the fused 8-bit block-wise optimizer step (and its max_unorm
// pre-pass) for sm_103a.
//
// One HBM pass per step ("8-bit Optimizers via Block-wise Quantization",
// abstract: blocks are quantized independently, in parallel): for each
// block of B elements a group of B/8 threads (8 elements per thread) loads
// p, g and the uint8 codes with 16/8-byte vector loads, dequantizes the codes
// through the map in shared memory times the block absmax, applies the
// optimizer update in binary32, writes p, reduces the new per-block absmax
// with warp shuffles (plus a named barrier for B > 256), and requantizes
// through the shared-memory bucket table (one lookup per value).
//
// Persistent grid: every CTA builds the map tables once, then its groups
// stride over the blocks of all tensors of the launch.
#pragma once

#include "bnb8_device.cuh"
#include "k_step8_ring.cuh"
#include "k_step8_ring_skip.cuh"

namespace bnb8 {

template <int OPT>
struct StatePtrs {
  uint8_t* c[3];
  float* a[3];
};

template <int OPT>
__device__ __forceinline__ StatePtrs<OPT> state_ptrs(const DevTensor& d, int64_t nblocks) {
  StatePtrs<OPT> r;
  r.c[0] = static_cast<uint8_t*>(d.s1);
  r.a[0] = d.a1;
  if (OPT == ADEMAMIX) {
    r.c[1] = static_cast<uint8_t*>(d.s1) + d.n;
    r.a[1] = d.a1 + nblocks;
    r.c[2] = static_cast<uint8_t*>(d.s2);
    r.a[2] = d.a2;
  } else {
    r.c[1] = static_cast<uint8_t*>(d.s2);
    r.a[1] = d.a2;
    r.c[2] = nullptr;
    r.a[2] = nullptr;
  }
  return r;
}

// shared memory layout (bytes)
template <int OPT, int MODE>
struct Step8Smem {
  static constexpr int NM = Traits<OPT>::NM;
  static constexpr int kQ = 0;                                   // float q[NM][256]
  static constexpr int kMid = kQ + NM * 256 * 4;                 // float mid[NM][256]
  static constexpr int kTbl = kMid + NM * 256 * 4;               // uint32 tbl[NM][kTblSize]
  static constexpr int kRed = kTbl + ((MODE == MODE_STEP || MODE == MODE_BCLIP || MODE == MODE_TWSTEP) ? NM * kTblSize * 4 : 0);
  static constexpr int kBytes = kRed + 2 * (kThreads / 32) * 4 * 4;
};

// Requantize the NS new states of one group and store codes and absmax.
// mx holds the group's absmax bit patterns.  Every lane computes the NS
// reciprocals itself: independent of each other, they are shorter on the
// critical path than one reciprocal followed by a shuffle.
template <int OPT>
__device__ __forceinline__ void requantize_store(const float (&s)[Traits<OPT>::NS][8],
                                                 const uint32_t (&mx)[Traits<OPT>::NS],
                                                 const StatePtrs<OPT>& sp, int64_t e0,
                                                 int64_t blk, int valid, bool vec, int gtid,
                                                 const bool (&fast_map)[2],
                                                 const bool (&nonneg_map)[2],
                                                 const uint32_t* stbl, const float* smid,
                                                 bool store_absmax = true) {
  constexpr int NS = Traits<OPT>::NS;
  if (!store_absmax) gtid = 1;  // tensor-wise: the absmax is stored after the pass
  float inv[NS];
  bool all_fast = true;
#pragma unroll
  for (int k = 0; k < NS; ++k) {
    const int m = Traits<OPT>::map_of(k);
    const float amk = __uint_as_float(mx[k]);
    inv[k] = amk > 0.0f ? __frcp_rn(amk) : 0.0f;
    all_fast = all_fast && fast_map[m] && mx[k] <= 0x7f7fffffu && inv[k] <= FLT_MAX &&
               (!Traits<OPT>::nonneg(k) || nonneg_map[m]);
  }
  if (all_fast) {
    // the usual case: every state takes the table path, in one straight-line
    // block so that the lookups of all states overlap
    uint32_t e[NS][8];
#pragma unroll
    for (int k = 0; k < NS; ++k) {
      const uint32_t* tz = stbl + Traits<OPT>::map_of(k) * kTblSize + kTblZero;
#pragma unroll
      for (int j = 0; j < 8; ++j)
        e[k][j] = Traits<OPT>::nonneg(k) ? encode_fast_nonneg(s[k][j], inv[k], tz)
                                         : encode_fast(s[k][j], inv[k], tz);
    }
#pragma unroll
    for (int k = 0; k < NS; ++k) {
      const uint32_t lo = __byte_perm(__byte_perm(e[k][0], e[k][1], 0x0062u), __byte_perm(e[k][2], e[k][3], 0x0062u), 0x5410u);
      const uint32_t hi = __byte_perm(__byte_perm(e[k][4], e[k][5], 0x0062u), __byte_perm(e[k][6], e[k][7], 0x0062u), 0x5410u);
      store_codes(sp.c[k], e0, valid, vec, make_uint2(lo, hi));
      if (gtid == 0) sp.a[k][blk] = __uint_as_float(mx[k]);
    }
    return;
  }
#pragma unroll
  for (int k = 0; k < NS; ++k) {
    const int m = Traits<OPT>::map_of(k);
    const float amax = __uint_as_float(mx[k]);
    // the table path needs a finite absmax and reciprocal (no NaN / inf)
    const bool fast = fast_map[m] && mx[k] <= 0x7f7fffffu && inv[k] <= FLT_MAX;
    uint32_t e[8];
    if (fast) {
      const uint32_t* tz = stbl + m * kTblSize + kTblZero;
      if (Traits<OPT>::nonneg(k) && nonneg_map[m]) {
#pragma unroll
        for (int j = 0; j < 8; ++j) e[j] = encode_fast_nonneg(s[k][j], inv[k], tz);
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) e[j] = encode_fast(s[k][j], inv[k], tz);
      }
    } else {
      const float* md = smid + m * 256;
#pragma unroll
      for (int j = 0; j < 8; ++j) e[j] = encode_search(s[k][j] * inv[k], md);
    }
    // byte 2 of each e[j] is the code
    const uint32_t lo = __byte_perm(__byte_perm(e[0], e[1], 0x0062u), __byte_perm(e[2], e[3], 0x0062u), 0x5410u);
    const uint32_t hi = __byte_perm(__byte_perm(e[4], e[5], 0x0062u), __byte_perm(e[6], e[7], 0x0062u), 0x5410u);
    store_codes(sp.c[k], e0, valid, vec, make_uint2(lo, hi));
    if (gtid == 0) sp.a[k][blk] = amax;
  }
}

// Eight zero gradients over zero states of RMSprop or Adagrad, on packed
// pairs (StepArgs::zero_ratio holds): the state and p update as usual, with
// the update direction the scaled gradient itself, which is the exact value
// of g / (sqrt(+0) + eps_hat) (pair_dir ZERO).
template <int OPT>
__device__ __forceinline__ void zero_rows_update(const StepArgs& a, const float* sq, uint2 cw,
                                                 float am, float (&p)[8], const float (&g)[8],
                                                 float eff, float (&s)[8], uint32_t& mx) {
#pragma unroll
  for (int j = 0; j < 8; j += 2) {
    float2 st[3] = {mul2(make_float2(sq[code_byte(cw, j)], sq[code_byte(cw, j + 1)]), f2(am)),
                    f2(0.0f), f2(0.0f)};
    float2 pp = make_float2(p[j], p[j + 1]);
    pair_update<OPT, true>(a, -eff, pp, make_float2(g[j], g[j + 1]), st);
    p[j] = pp.x;
    p[j + 1] = pp.y;
    s[j] = st[0].x;
    s[j + 1] = st[0].y;
    mx = absmax_nan(mx, st[0].x, st[0].y);
  }
}

template <int OPT, int DT, int MODE, bool SKIP>
__global__ void __launch_bounds__(kThreads, 2) k_step8(const __grid_constant__ StepArgs a) {
  constexpr int NS = Traits<OPT>::NS;
  constexpr int NM = Traits<OPT>::NM;
  using L = Step8Smem<OPT, MODE>;
  extern __shared__ __align__(16) unsigned char smem[];
  float* sq = reinterpret_cast<float*>(smem + L::kQ);
  float* smid = reinterpret_cast<float*>(smem + L::kMid);
  uint32_t* stbl = reinterpret_cast<uint32_t*>(smem + L::kTbl);
  float* sred = reinterpret_cast<float*>(smem + L::kRed);
  __shared__ int s_bad[2];
  __shared__ uint32_t s_tw[4];  // MODE_TWMAX: this CTA's new absmax bits per state, any-update
  __shared__ int s_below[2];
  __shared__ int s_scan[2 * 32];

  const int tid = threadIdx.x;
  // the pre-pass zeroes the tickets of the reduction launched after it
  if (MODE == MODE_NORM && a.tickets != nullptr && blockIdx.x == 0 && tid < a.ntensors) a.tickets[tid] = 0u;
  // the pre-pass with a carried parameter norm (BNB8_CARRY_PNORM): the sums
  // of p^2 are already in the partials; p is not read when the direction does
  // not depend on it
  const bool carried = MODE == MODE_NORM && a.carry_stamp != nullptr && *a.carry_stamp == a.carry_expect;
  const bool read_p = !(carried && (Traits<OPT>::DECOUPLED || a.wd == 0.0f));
  // ---- stage the maps, midpoints and (step mode) the bucket tables ----
  for (int i = tid; i < NM * 256; i += kThreads) sq[i] = i < 256 ? a.qmap1[i] : a.qmap2[i - 256];
  if (tid < 2) s_bad[tid] = 0;
  if (tid < 4) s_tw[tid] = 0u;
  __syncthreads();
  // Rows with a zero gradient over zero states (untouched rows of an
  // embedding) skip the square root and division of RMSprop and Adagrad,
  // exactly (pair_dir ZERO).  Adam keeps one path: at its register budget a
  // second copy of the packed loop costs more on dense gradients than the
  // zero rows gain.
  constexpr bool kZeroPath = (OPT == RMSPROP || OPT == ADAGRAD) && MODE == MODE_STEP;
  static_assert(!kZeroPath || NS == 1, "the zero check reads one state absmax");
  bool fin = true;
  for (int i = tid; i < NM * 256; i += kThreads) {
    const int m = i >> 8, k = i & 255;
    smid[i] = k < 255 ? (sq[m * 256 + k] + sq[m * 256 + k + 1]) * 0.5f : 0.0f;
    if (kZeroPath) fin = fin && fabsf(sq[i]) <= FLT_MAX;
  }
  // whether every map level is finite (a zero absmax then dequantizes to zeros)
  bool maps_finite = false;
  if constexpr (kZeroPath) {
    maps_finite = __syncthreads_and(fin) != 0;
  } else {
    __syncthreads();
  }
  if (MODE == MODE_STEP || MODE == MODE_BCLIP || MODE == MODE_TWSTEP) {
    build_tables<NM>(smid, stbl, s_bad, s_below, s_scan);
  }
  const bool fast_map[2] = {s_bad[0] == 0, s_bad[1] == 0};
  // the map's lowest level is its first (ascending maps)
  const bool nonneg_map[2] = {sq[0] >= 0.0f, NM > 1 && sq[256] >= 0.0f};

  // ---- group geometry ----
  const int log2B = a.log2B;
  const int64_t B = int64_t(1) << log2B;
  const int GT = static_cast<int>(B >> 3);   // threads per block
  const int groups_per_cta = kThreads / GT;
  const int groups_per_warp = GT < 32 ? 32 / GT : 1;
  const int lane = tid & 31;
  const int glocal = tid / GT;
  const int gtid = tid & (GT - 1);
  // block indices of a launch fit in 32 bits (the host checks it)
  const int32_t stride = static_cast<int32_t>(gridDim.x) * groups_per_cta;
  // warp-uniform loop base: the first group of this warp
  const int32_t warp_g0 = static_cast<int32_t>(blockIdx.x) * groups_per_cta + ((tid & ~31) / GT);
  const int in_warp = GT < 32 ? lane / GT : 0;
  // lanes of this thread's group inside its warp (GT < 32)
  const uint32_t gmask = GT >= 32 ? 0xffffffffu : (((1u << GT) - 1u) << (in_warp * GT));
  // parity selects the half of the reduction scratch; it flips after every
  // group reduction so that consecutive reductions never share a slot
  int parity = 0;

  // Tensors are visited in order; within a tensor this warp's groups take the
  // blocks gb = base + in_warp, base stepping by the grid's group count, so
  // every per-tensor value is loaded once.  A warp whose groups straddle a
  // tensor boundary (blocks of fewer than 256 elements) visits that base once
  // per tensor, with disjoint groups active.
  for (int t = 0; t < a.ntensors; ++t) {
    const DevTensor& d = a.t[t];
    const int32_t fb = static_cast<int32_t>(d.first_block);
    const int64_t n = d.n;
    const int32_t nb = static_cast<int32_t>((n + B - 1) >> log2B);
    const int32_t end = fb + nb;
    // tensor-wise: one absmax per state (index 0; AdEMAMix's absmax1 is
    // [2, 1]); a tensor none of whose elements is updated (skip_zeros) is
    // left untouched
    const bool tw = MODE == MODE_TWMAX || MODE == MODE_TWSTEP ||
                    (MODE == MODE_NORM && a.tensorwise != 0);
    const StatePtrs<OPT> sp = state_ptrs<OPT>(d, tw ? 1 : nb);
    const bool vec = d.vec_ok != 0;
    const float eff = a.step_size * (a.clip != nullptr ? a.clip[d.index] : 1.0f);
    if (MODE == MODE_TWSTEP && a.tw_acc[4 * d.index + 3] == 0u) continue;
    // first warp base whose groups can reach this tensor
    const int32_t lo = fb - (groups_per_warp - 1);
    int32_t base = warp_g0;
    if (base < lo) base += ((lo - base + stride - 1) / stride) * stride;

    // Where the registers allow, the next block's absmax (2-state with
    // binary32 p: Adam, AdamW) or codes and absmax (1-state) are loaded
    // before this block's requantization, overlapping their latency with it;
    // the other kernels would spill and keep the plain order
    constexpr bool kAheadAm = MODE == MODE_STEP && !SKIP && (NS == 1 || (NS == 2 && DT == DT_F32));
    constexpr bool kAheadCodes = MODE == MODE_STEP && !SKIP && NS == 1;
    const bool zero_ok = kZeroPath && a.zero_ratio != 0 && maps_finite &&
                         (Traits<OPT>::DECOUPLED || a.wd == 0.0f);
    bool have_n = false;
    uint2 cwn[NS];
    float amn[NS];
    for (; base < end; base += stride) {
      const int32_t blk = base + in_warp - fb;
      const bool active = blk >= 0 && blk < nb;
      const int64_t e0 = (static_cast<int64_t>(blk) << log2B) + gtid * 8;
      const int64_t left = active ? n - e0 : 0;
      const int valid = left >= 8 ? 8 : (left > 0 ? static_cast<int>(left) : 0);
      const bool full = vec && valid == 8;

      float p[8], g[8];
      uint2 cw[NS];
      float am[NS];
      if ((MODE == MODE_STEP || MODE == MODE_BCLIP || MODE == MODE_TWSTEP) && SKIP) {
        // skip_zeros: read g first; a block whose gradient is all zero is left
        // untouched, so its p, codes and absmax are never read.  Groups of
        // fewer than 32 threads skip only when their whole warp may.
        load8<DT, true>(d.g, e0, valid, vec, g);
        bool nz = false;
#pragma unroll
        for (int j = 0; j < 8; ++j) nz = nz || (j < valid && g[j] != 0.0f);
        bool group_nz;
        if (GT <= 32) {
          group_nz = __any_sync(0xffffffffu, nz);
        } else {
          uint32_t v[1] = {nz ? 1u : 0u};
          group_max_bits<1>(v, GT, glocal, reinterpret_cast<uint32_t*>(sred), parity);
          parity ^= 1;
          group_nz = v[0] != 0u;
        }
        if (!group_nz && !tw) continue;
        load8<DT, false>(d.p, e0, valid, vec, p);
      } else {
        if (MODE != MODE_NORM || read_p) {
          load8<DT, false>(d.p, e0, valid, vec, p);
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) p[e] = 0.0f;
        }
        load8<DT, true>(d.g, e0, valid, vec, g);
      }
#pragma unroll
      for (int k = 0; k < NS; ++k) {
        cw[k] = kAheadCodes && have_n ? cwn[k] : load_codes(sp.c[k], e0, valid, vec);
        am[k] = kAheadAm && have_n ? amn[k] : (active ? sp.a[k][tw ? 0 : blk] : 0.0f);
      }

      // ---- dequantize, update; new states in s, running max of |s| in mx ----
      float s[NS][8];
      uint32_t mx[NS];
#pragma unroll
      for (int k = 0; k < NS; ++k) mx[k] = 0u;
      float usq = 0.0f, psq = 0.0f;
      bool any = false;
      float ud[8];          // MODE_BCLIP: update directions, applied after the block's clip
      uint32_t held = 0u;   // MODE_BCLIP: elements left as they are (skipped)
      if (!SKIP && __all_sync(0xffffffffu, full)) {
        // every thread of the warp holds 8 present, aligned elements: a
        // straight-line path on packed pairs, no per-element predicates
        bool zero = false;
        if constexpr (kZeroPath) {
          if (zero_ok) {
            uint32_t o = 0u;
#pragma unroll
            for (int j = 0; j < 8; ++j) o |= __float_as_uint(g[j]);
            zero = (o << 1) == 0u && am[0] == 0.0f;  // eight +-0 gradients, zero states
          }
          if (zero) zero_rows_update<OPT>(a, sq, cw[0], am[0], p, g, eff, s[0], mx[0]);
        }
        if (!zero) {
#pragma unroll
          for (int j = 0; j < 8; j += 2) {
            float2 st[3];
#pragma unroll
            for (int k = 0; k < 3; ++k)
              st[k] = k < NS ? mul2(make_float2(sq[Traits<OPT>::map_of(k) * 256 + code_byte(cw[k], j)],
                                                sq[Traits<OPT>::map_of(k) * 256 + code_byte(cw[k], j + 1)]),
                                    f2(am[k]))
                             : f2(0.0f);
            if (MODE != MODE_STEP) psq = psq + p[j] * p[j] + p[j + 1] * p[j + 1];
            float2 pp = make_float2(p[j], p[j + 1]);
            float2 u;
            if (MODE == MODE_BCLIP) {
              u = pair_dir<OPT>(a, pp, make_float2(g[j], g[j + 1]), st);
              ud[j] = u.x;
              ud[j + 1] = u.y;
            } else {
              u = pair_update<OPT>(a, -eff, pp, make_float2(g[j], g[j + 1]), st);
              p[j] = pp.x;
              p[j + 1] = pp.y;
            }
            if (MODE != MODE_STEP) usq = usq + u.x * u.x + u.y * u.y;
#pragma unroll
            for (int k = 0; k < NS; ++k) {
              s[k][j] = st[k].x;
              s[k][j + 1] = st[k].y;
              mx[k] = absmax_nan(mx[k], st[k].x, st[k].y);
            }
          }
        }
        any = true;
      } else if (full) {
        // whole group of 8 present: no per-element predicates
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          float st[3];
#pragma unroll
          for (int k = 0; k < 3; ++k)
            st[k] = k < NS ? sq[Traits<OPT>::map_of(k) * 256 + code_byte(cw[k], j)] * am[k] : 0.0f;
          if (MODE != MODE_STEP) psq = psq + p[j] * p[j];
          bool skipped;
          float u;
          if (MODE == MODE_BCLIP) {
            u = elem_dir<OPT, SKIP>(a, p[j], g[j], st, skipped);
            ud[j] = u;
            if (skipped) held |= 1u << j;
          } else {
            u = elem_update<OPT, SKIP>(a, eff, p[j], g[j], st, skipped);
          }
          if (SKIP) any = any || !skipped;
          if (MODE != MODE_STEP) usq = usq + u * u;
#pragma unroll
          for (int k = 0; k < NS; ++k) {
            s[k][j] = st[k];
            mx[k] = absmax_nan(mx[k], st[k], 0.0f);
          }
        }
        if (!SKIP) any = true;
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          float st[3];
#pragma unroll
          for (int k = 0; k < 3; ++k)
            st[k] = k < NS ? sq[Traits<OPT>::map_of(k) * 256 + code_byte(cw[k], j)] * am[k] : 0.0f;
          if (MODE != MODE_STEP && j < valid) psq = psq + p[j] * p[j];
          bool skipped = true;
          float u = 0.0f;
          if (MODE == MODE_BCLIP) {
            if (j < valid) u = elem_dir<OPT, SKIP>(a, p[j], g[j], st, skipped);
            ud[j] = u;
            if (skipped) held |= 1u << j;
          } else if (j < valid) {
            u = elem_update<OPT, SKIP>(a, eff, p[j], g[j], st, skipped);
          }
          if (!skipped) any = true;
          if (MODE != MODE_STEP) usq = usq + u * u;
#pragma unroll
          for (int k = 0; k < NS; ++k) {
            s[k][j] = j < valid ? st[k] : 0.0f;
            mx[k] = absmax_nan(mx[k], s[k][j], 0.0f);
          }
        }
      }

      if constexpr (MODE == MODE_NORM) {
        float r[2] = {usq, psq};
        group_reduce<2, false>(r, GT, glocal, sred, parity);
        parity ^= 1;
        if (active && gtid == 0) {
          if (carried) a.partials[fb + blk].x = r[0];
          else a.partials[fb + blk] = make_float2(r[0], r[1]);
        }
        continue;
      }
      if constexpr (MODE == MODE_TWMAX) {
        // the tensor's new absmax: warp maxima into this CTA's shared
        // accumulators (flushed to tw_acc once per tensor below)
#pragma unroll
        for (int k = 0; k < NS; ++k) {
          const uint32_t w = __reduce_max_sync(0xffffffffu, mx[k]);
          if (lane == 0 && w != 0u) atomicMax(&s_tw[k], w);
        }
        if (__any_sync(0xffffffffu, any && active) && lane == 0) atomicOr(&s_tw[3], 1u);
        continue;
      }
      if constexpr (MODE == MODE_BCLIP) {
        // max_unorm per block: U = unorm_c * ||u||, P = ||p|| over the block
        // (group sums as in the pre-pass); clip the step if U > max_unorm * P
        float r[2] = {usq, psq};
        group_reduce<2, false>(r, GT, glocal, sred, parity);
        parity ^= 1;
        const float unorm = a.unorm_c * sqrtf(r[0]);
        const float limit = a.max_unorm * sqrtf(r[1]);
        const float eff_b = eff * (unorm > limit ? limit / unorm : 1.0f);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (!((held >> j) & 1u)) elem_apply<OPT>(a, eff_b, p[j], ud[j]);
      }

      // p does not depend on the new absmax: store it now (skipped elements
      // write back their unchanged bits; a group with nothing updated writes
      // only when skip_zeros could not leave its warp early, with the same
      // bits)
      if (active && any) store8<DT>(d.p, e0, valid, vec, p);
      if (MODE == MODE_STEP && a.carry_out) {
        // the block's sum of the new p^2 as stored (skipped elements keep theirs)
        float r[1] = {0.0f};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float q = Elem<DT>::stored(p[e]);
          if (e < valid) r[0] = r[0] + q * q;
        }
        group_reduce<1, false>(r, GT, glocal, sred, parity);
        parity ^= 1;
        if (active && gtid == 0) a.partials[fb + blk].y = r[0];
      }
      if (kAheadAm) {
        // the next block of this tensor, when all 8 of this thread's elements
        // exist there and its streams are aligned (else it loads as usual)
        have_n = false;
        const int32_t blk_n = base + stride + in_warp - fb;
        if (vec && blk_n < nb) {
          const int64_t e0n = (static_cast<int64_t>(blk_n) << log2B) + gtid * 8;
          if (e0n + 8 <= n) {
#pragma unroll
            for (int k = 0; k < NS; ++k) {
              if (kAheadCodes) cwn[k] = load_codes(sp.c[k], e0n, 8, true);
              amn[k] = sp.a[k][tw ? 0 : blk_n];
            }
            have_n = true;
          }
        }
      }

      // ---- new absmax per state (bit patterns of non-negative values) ----
      if (tw) {
#pragma unroll
        for (int k = 0; k < NS; ++k) mx[k] = a.tw_acc[4 * d.index + k];
      } else {
        group_max_bits<NS>(mx, GT, glocal, reinterpret_cast<uint32_t*>(sred), parity);
        parity ^= 1;
      }
      if (SKIP) {
        // whether any element of the group was updated
        bool group_any;
        if (GT >= 32) {
          group_any = __any_sync(0xffffffffu, any);
          if (GT > 32) {
            uint32_t v[1] = {group_any ? 1u : 0u};
            group_max_bits<1>(v, GT, glocal, reinterpret_cast<uint32_t*>(sred), parity);
            parity ^= 1;
            group_any = v[0] != 0u;
          }
        } else {
          group_any = (__ballot_sync(0xffffffffu, any) & gmask) != 0u;
        }
        if (!group_any && !tw) continue;  // nothing updated: codes and absmax untouched
      }
      // inactive lanes compute along (valid 0) and store nothing
      requantize_store<OPT>(s, mx, sp, e0, blk, active ? valid : 0, vec, active ? gtid : 1,
                            fast_map, nonneg_map, stbl, smid, !tw);
    }
    if constexpr (MODE == MODE_TWMAX) {
      // this CTA's share of the tensor's new absmax, once per tensor
      __syncthreads();
      if (tid < NS) {
        if (s_tw[tid] != 0u) atomicMax(&a.tw_acc[4 * d.index + tid], s_tw[tid]);
        s_tw[tid] = 0u;
      } else if (tid == 3) {
        if (s_tw[3] != 0u) atomicOr(&a.tw_acc[4 * d.index + 3], 1u);
        s_tw[3] = 0u;
      }
      __syncthreads();
    }
  }
  if (MODE == MODE_STEP && a.carry_writer && blockIdx.x == 0 && threadIdx.x == 0)
    *a.carry_stamp = a.carry_write;
}

// Tensor-wise quantization: after the step, the new absmax of each updated
// tensor of the launch (one thread per tensor).
template <int OPT>
__global__ void k_tw_store(const __grid_constant__ StepArgs a) {
  constexpr int NS = Traits<OPT>::NS;
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= a.ntensors) return;
  const DevTensor& d = a.t[t];
  const uint32_t* acc = a.tw_acc + 4 * d.index;
  if (acc[3] == 0u) return;
  const StatePtrs<OPT> sp = state_ptrs<OPT>(d, 1);
#pragma unroll
  for (int k = 0; k < NS; ++k) sp.a[k][0] = __uint_as_float(acc[k]);
}

template <int OPT>
cudaError_t launch_tw_store_t(const StepArgs& a, cudaStream_t s) {
  k_tw_store<OPT><<<(a.ntensors + 127) / 128, 128, 0, s>>>(a);
  return cudaGetLastError();
}

template <int OPT, int DT, int MODE, bool SKIP>
cudaError_t launch_step8_skip(const StepArgs& a, int grid, cudaStream_t s) {
  constexpr int bytes = Step8Smem<OPT, MODE>::kBytes;
  static std::atomic<unsigned char> configured[kMaxDevices];  // the attribute is per device
  const cudaError_t e = set_smem_limit_once(
      reinterpret_cast<const void*>(k_step8<OPT, DT, MODE, SKIP>), bytes, configured);
  if (e != cudaSuccess) return e;
  k_step8<OPT, DT, MODE, SKIP><<<grid, kThreads, bytes, s>>>(a);
  return cudaGetLastError();
}

template <int OPT, int DT, int MODE>
cudaError_t launch_step8_t(const StepArgs& a, int grid, cudaStream_t s) {
  // the plain step, its max_unorm pre-pass and the step with max_unorm per
  // block, over blocks of 256 elements or more: the async-copy ring
  if constexpr (MODE == MODE_STEP) {
    // skip_zeros over blocks of 256: the gradient streams through the ring,
    // live blocks fetch the rest
    if (a.skip_zeros && a.log2B == 8 && a.tensorwise == 0) return launch_step8_skip_ring<OPT, DT>(a, s);
  }
  if constexpr (MODE == MODE_STEP || MODE == MODE_NORM || MODE == MODE_BCLIP) {
    if (!a.skip_zeros && a.log2B >= 8 && a.tensorwise == 0)
      return launch_step8_ring<OPT, DT, MODE == MODE_STEP ? RING_STEP
                                        : (MODE == MODE_NORM ? RING_NORM : RING_BCLIP)>(a, s);
  }
  return a.skip_zeros ? launch_step8_skip<OPT, DT, MODE, true>(a, grid, s)
                      : launch_step8_skip<OPT, DT, MODE, false>(a, grid, s);
}

template <int OPT, int DT, int MODE>
int ctas_step8_t() {
  constexpr int bytes = Step8Smem<OPT, MODE>::kBytes;
  cudaFuncSetAttribute(k_step8<OPT, DT, MODE, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       bytes);
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_step8<OPT, DT, MODE, false>, kThreads,
                                                    bytes) != cudaSuccess)
    return 1;
  return n > 0 ? n : 1;
}

}  // namespace bnb8
