// k_step32.cuh -- the optimizer step with binary32 states, for tensors the
// caller keeps at 32-bit state (bitsandbytes docs "optim_overview.md":
// min_8bit_size, default 4096 elements), and its max_unorm pre-pass.  Same
// element update, thread geometry and block partition as the 8-bit kernel, so
// one launch block of the pre-pass covers B elements in both.
#pragma once

#include "bnb8_device.cuh"

namespace bnb8 {

template <int OPT, int DT, int MODE>
__global__ void __launch_bounds__(kThreads, 2) k_step32(const __grid_constant__ StepArgs a) {
  constexpr int NS = Traits<OPT>::NS;
  __shared__ float sred[2 * (kThreads / 32) * 4];
  const int tid = threadIdx.x;
  const int log2B = a.log2B;
  const int B = 1 << log2B;
  const int GT = B >> 3;
  const int groups_per_cta = kThreads / GT;
  const int lane = tid & 31;
  const int glocal = tid / GT;
  const int gtid = tid & (GT - 1);
  const int64_t stride = static_cast<int64_t>(gridDim.x) * groups_per_cta;
  const int64_t warp_g0 = static_cast<int64_t>(blockIdx.x) * groups_per_cta + ((tid & ~31) / GT);
  const int in_warp = GT < 32 ? lane / GT : 0;
  int parity = 0;
  // the pre-pass zeroes the tickets of the reduction launched after it
  if (MODE == MODE_NORM && a.tickets != nullptr && blockIdx.x == 0 && tid < a.ntensors) a.tickets[tid] = 0u;
  // the pre-pass with a carried parameter norm (see k_step8)
  const bool carried = MODE == MODE_NORM && a.carry_stamp != nullptr && *a.carry_stamp == a.carry_expect;
  const bool read_p = !(carried && (Traits<OPT>::DECOUPLED || a.wd == 0.0f));

  for (int64_t base = warp_g0; base < a.total_blocks; base += stride) {
    const int64_t gb = base + in_warp;
    const bool active = gb < a.total_blocks;
    const int t = active ? (a.ntensors > 1 ? find_tensor(a, gb) : 0) : 0;
    const DevTensor& d = a.t[t];
    const int64_t blk = active ? gb - d.first_block : 0;
    const int64_t e0 = (blk << log2B) + static_cast<int64_t>(gtid) * 8;
    const int64_t left = active ? d.n - e0 : 0;
    const int valid = left >= 8 ? 8 : (left > 0 ? static_cast<int>(left) : 0);
    const bool vec = d.vec_ok != 0;
    float* sp[3] = {static_cast<float*>(d.s1),
                    OPT == ADEMAMIX ? static_cast<float*>(d.s1) + d.n : static_cast<float*>(d.s2),
                    static_cast<float*>(d.s2)};

    float p[8], g[8], s[NS][8];
    if (MODE != MODE_NORM || read_p) {
      load8<DT, false>(d.p, e0, valid, vec, p);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) p[j] = 0.0f;
    }
    load8<DT, true>(d.g, e0, valid, vec, g);
#pragma unroll
    for (int k = 0; k < NS; ++k) load8<DT_F32, false>(sp[k], e0, valid, vec, s[k]);
    const float clip = (a.clip != nullptr && active) ? a.clip[d.index] : 1.0f;
    const float eff = a.step_size * clip;

    float usq = 0.0f, psq = 0.0f;
    bool any = false;
    float ud[8];          // MODE_BCLIP: update directions, applied after the block's clip
    uint32_t held = 0u;   // MODE_BCLIP: elements left as they are (skipped)
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      float st[3];
#pragma unroll
      for (int k = 0; k < 3; ++k) st[k] = k < NS ? s[k][j] : 0.0f;
      if (MODE != MODE_STEP && j < valid) psq = psq + p[j] * p[j];
      bool skipped = true;
      float u = 0.0f;
      if (MODE == MODE_BCLIP) {
        if (j < valid) u = elem_dir<OPT>(a, p[j], g[j], st, skipped);
        ud[j] = u;
        if (skipped) held |= 1u << j;
      } else if (j < valid) {
        u = elem_update<OPT>(a, eff, p[j], g[j], st, skipped);
      }
      if (!skipped) any = true;
      if (MODE != MODE_STEP) usq = usq + u * u;
#pragma unroll
      for (int k = 0; k < NS; ++k) s[k][j] = st[k];
    }
    if constexpr (MODE == MODE_NORM) {
      float r[2] = {usq, psq};
      group_reduce<2, false>(r, GT, glocal, sred, parity);
      parity ^= 1;
      if (active && gtid == 0) {
        if (carried) a.partials[gb].x = r[0];
        else a.partials[gb] = make_float2(r[0], r[1]);
      }
      continue;
    }
    if constexpr (MODE == MODE_BCLIP) {
      // max_unorm per block of B elements, as in the 8-bit kernel
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
    if (MODE == MODE_STEP && a.carry_out) {
      // the block's sum of the new p^2 as stored, for the next step's max_unorm
      float r[1] = {0.0f};
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float q = Elem<DT>::stored(p[j]);
        if (j < valid) r[0] = r[0] + q * q;
      }
      group_reduce<1, false>(r, GT, glocal, sred, parity);
      parity ^= 1;
      if (active && gtid == 0) a.partials[gb].y = r[0];
    }
    if (!any) continue;  // every element skipped: leave them untouched
    store8<DT>(d.p, e0, valid, vec, p);
#pragma unroll
    for (int k = 0; k < NS; ++k) store8<DT_F32>(sp[k], e0, valid, vec, s[k]);
  }
  if (MODE == MODE_STEP && a.carry_writer && blockIdx.x == 0 && threadIdx.x == 0)
    *a.carry_stamp = a.carry_write;
}

template <int OPT, int DT, int MODE>
cudaError_t launch_step32_t(const StepArgs& a, int grid, cudaStream_t s) {
  if constexpr (MODE == MODE_TWMAX || MODE == MODE_TWSTEP) {
    return cudaErrorInvalidValue;  // 32-bit states have no absmax
  } else {
    k_step32<OPT, DT, MODE><<<grid, kThreads, 0, s>>>(a);
    return cudaGetLastError();
  }
}

template <int OPT, int DT, int MODE>
int ctas_step32_t() {
  if constexpr (MODE == MODE_TWMAX || MODE == MODE_TWSTEP) return 1;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k_step32<OPT, DT, MODE>, kThreads, 0) !=
      cudaSuccess)
    return 1;
  return n > 0 ? n : 1;
}

}  // namespace bnb8
