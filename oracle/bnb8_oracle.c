/*
 * bnb8_oracle.c -- reference (oracle) implementation of the 8-bit block-wise
 * dynamic-quantized optimizer step.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plain, single-threaded CPU
 * statement of what the GPU library computes.  Only the test suite, the smoke
 * check and the benchmark's CPU-baseline leg may load it.  It shares no code,
 * header, table or constant generator with the CUDA library.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -fPIC -shared
 *        (no FMA contraction, so every float operation below is rounded once,
 *        in the order written; all state arithmetic is IEEE binary32).
 *
 * Sources (web pages on the method):
 *  [P1] "[XPU] Implemented 8bit optimizers in triton #1692" (bitsandbytes pull
 *       request): the benchmark script `test_optimizer8bit` names the state
 *       tensors (state1/state2, qmap1/qmap2, absmax1/absmax2), the AdEMAMix
 *       stacked m1_m2 layout, the 32-bit torch comparators and the tolerances.
 *  [P2] "optim_overview.md" (bitsandbytes docs): Optimizer2State /
 *       Optimizer1State parameters and defaults (lr, betas, eps,
 *       weight_decay, min_8bit_size, max_unorm, skip_zeros, alpha, t_alpha,
 *       t_beta3).
 *  [P3] "Support skip_zeros in the XPU Triton optimizer kernels #2097":
 *       skip_zeros leaves parameter and states untouched where the raw
 *       (pre-weight-decay) gradient is exactly zero.
 *  [P4] "8-bit Optimizers via Block-wise Quantization" (Dettmers et al.),
 *       abstract and introduction: block-wise quantization with independent
 *       per-block normalisation; dynamic (sign / base-10 exponent / fraction)
 *       quantization; a citing paper ("The case for 4-bit precision") states the
 *       data type: one sign bit, then a run of zero bits whose length is the
 *       base-10 exponent, then the fraction.
 *
 * The pages print neither the update equations nor the 256 map values.  Every
 * place where this file takes a reading of its own is marked READING below.
 *
 * Parity status of each function (what pins it in the CPU test suite):
 *  oracle_create_qmap        pinned: independent byte-structure enumeration,
 *                            closed-form values, monotonicity, symmetry.  The
 *                            exact bitsandbytes table values are parity
 *                            unpinned (not on the pages).
 *  oracle_code               pinned: brute-force nearest level; tie rule.
 *  oracle_quantize_blockwise pinned: exact round trip of every level, error
 *                            bound, absmax = max |x|.
 *  oracle_step (32-bit)      pinned: torch.optim Adam/AdamW/SGD/RMSprop/Adagrad;
 *                            Lion and AdEMAMix closed forms and special cases.
 *  oracle_step (8-bit)       pinned: tracks the 32-bit torch optimizers within
 *                            the benchmark script's tolerances; skip_zeros and
 *                            max_unorm invariants; checkpoint round trip.
 *  oracle_param_sumsq        pinned: Pythagorean closed forms in every
 *                            dtype, exactly rounded sums (math.fsum), and the
 *                            P of the next step's max_unorm test.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---- enums (the oracle's own numbering) --------------------------------- */
enum { OR_F32 = 0, OR_BF16 = 1, OR_F16 = 2 };
enum {
  OR_ADAM = 0, OR_ADAMW = 1, OR_MOMENTUM = 2, OR_RMSPROP = 3,
  OR_ADAGRAD = 4, OR_LION = 5, OR_ADEMAMIX = 6
};

typedef struct {
  int optim;
  float lr, beta1, beta2, beta3, alpha, eps, weight_decay, gnorm_scale, max_unorm;
  int64_t step;     /* 1-based step number of the update being taken */
  int64_t t_alpha;  /* AdEMAMix alpha warm-up length, 0 = no schedule */
  int64_t t_beta3;  /* AdEMAMix beta3 warm-up length, 0 = no schedule */
  int skip_zeros;
  int unorm_per_block; /* max_unorm per quantization block instead of per tensor */
} oracle_hparams;

/* Per-step scalars, computed once in binary64 and rounded once to binary32. */
typedef struct {
  float b1, b2, b3t;        /* decay rates (b3t: scheduled AdEMAMix beta3) */
  float omb1, omb2, omb3t;  /* 1 - b */
  float step_size;          /* multiplies the update direction u */
  float eps_hat;            /* eps as it appears in the denominator */
  float inv_bc1;            /* AdEMAMix: 1 / (1 - beta1^t) */
  float alpha_t;            /* AdEMAMix: scheduled alpha */
  float decay;              /* decoupled weight decay factor 1 - lr*wd */
  double unorm_c;           /* |true update direction| = unorm_c * |u| */
} step_scalars;

/* ---- storage dtypes ------------------------------------------------------ */
/* bfloat16 <-> binary32: bfloat16 is the top half of a binary32; narrowing
 * rounds to nearest, ties to even. */
float oracle_bf16_to_f32(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

uint16_t oracle_f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x0040u); /* quiet NaN */
  uint32_t kept_lsb = (u >> 16) & 1u;
  u += 0x7fffu + kept_lsb;
  return (uint16_t)(u >> 16);
}

/* IEEE binary16 <-> binary32 (round to nearest even, gradual underflow). */
float oracle_f16_to_f32(uint16_t h) {
  uint32_t sign = (uint32_t)(h & 0x8000u) << 16;
  uint32_t e = (h >> 10) & 0x1fu, m = h & 0x3ffu;
  float f;
  if (e == 0) {
    f = (float)m * (1.0f / 16777216.0f); /* m * 2^-24, exact */
    uint32_t u;
    memcpy(&u, &f, 4);
    u |= sign;
    memcpy(&f, &u, 4);
    return f;
  }
  uint32_t u;
  if (e == 31) u = sign | 0x7f800000u | (m << 13);
  else u = sign | ((e + 112u) << 23) | (m << 13);
  memcpy(&f, &u, 4);
  return f;
}

uint16_t oracle_f32_to_f16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
  uint32_t a = u & 0x7fffffffu;
  if (a > 0x7f800000u) return (uint16_t)(sign | 0x7e00u);   /* NaN */
  if (a >= 0x477ff000u) return (uint16_t)(sign | 0x7c00u);  /* >= 65520 rounds to inf */
  if (a >= 0x38800000u) {                                   /* normal binary16 range */
    uint32_t e = (a >> 23) - 112u;
    uint32_t mant = a & 0x7fffffu;
    uint32_t h = (e << 10) | (mant >> 13);
    uint32_t rest = mant & 0x1fffu;
    if (rest > 0x1000u || (rest == 0x1000u && (h & 1u))) h += 1u;
    return (uint16_t)(sign | h);
  }
  /* subnormal binary16: count units of 2^-24, rounding to nearest even */
  float fa;
  memcpy(&fa, &a, 4);
  float units = nearbyintf(fa * 16777216.0f);
  return (uint16_t)(sign | (uint16_t)units);
}

static float load_elem(const void* base, int dtype, int64_t i) {
  if (dtype == OR_F32) return ((const float*)base)[i];
  if (dtype == OR_BF16) return oracle_bf16_to_f32(((const uint16_t*)base)[i]);
  return oracle_f16_to_f32(((const uint16_t*)base)[i]);
}

static void store_elem(void* base, int dtype, int64_t i, float v) {
  if (dtype == OR_F32) ((float*)base)[i] = v;
  else if (dtype == OR_BF16) ((uint16_t*)base)[i] = oracle_f32_to_bf16(v);
  else ((uint16_t*)base)[i] = oracle_f32_to_f16(v);
}

void oracle_convert(const float* in, int64_t n, void* out, int dtype) {
  for (int64_t i = 0; i < n; ++i) store_elem(out, dtype, i, in[i]);
}

void oracle_widen(const void* in, int dtype, int64_t n, float* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = load_elem(in, dtype, i);
}

/* ---- the dynamic quantization map ---------------------------------------
 * [P4] abstract: dynamic quantization is non-linear and precise for both
 * small and large magnitudes; the citing snippet gives the bit layout: a sign
 * bit, then k zero bits meaning the base-10 exponent -k, then an indicator
 * bit, then the linear fraction bits.
 * READING (values): with f fraction bits the 2^f fraction codes are the
 * midpoints of 2^f equal sub-intervals of [0.1, 1], scaled by 10^-k.  Signed
 * map: k = 0..6 with 6-k fraction bits -> 127 positive levels, their
 * negatives, zero, and +1.0 in the remaining (negative-zero) slot.  Unsigned
 * map (no sign bit): k = 0..6 with 7-k fraction bits -> 254 levels, zero and
 * +1.0.  Values are formed in binary64 and rounded once; the table is sorted
 * ascending.  +1.0 is present so that the element holding the block maximum
 * is stored without loss.
 */
void oracle_create_qmap(int is_signed, float* out) {
  double v[256];
  int cnt = 0;
  for (int k = 0; k <= 6; ++k) {
    int fbits = is_signed ? 6 - k : 7 - k;
    int nfrac = 1 << fbits;
    double scale = pow(10.0, -(double)k);
    for (int f = 0; f < nfrac; ++f) {
      double frac = 0.1 + ((double)f + 0.5) * (0.9 / (double)nfrac);
      v[cnt++] = scale * frac;
      if (is_signed) v[cnt++] = -scale * frac;
    }
  }
  v[cnt++] = 0.0;
  v[cnt++] = 1.0;
  /* plain insertion sort, ascending */
  for (int i = 1; i < cnt; ++i) {
    double x = v[i];
    int j = i - 1;
    while (j >= 0 && v[j] > x) {
      v[j + 1] = v[j];
      --j;
    }
    v[j + 1] = x;
  }
  for (int i = 0; i < 256; ++i) out[i] = (float)v[i];
}

/* READING (nearest code): the decision points are the binary32 midpoints
 * mid_i = (q_i + q_{i+1}) * 0.5 between neighbouring levels, and the code of
 * a normalised value xn is the number of midpoints strictly below it, so an
 * exact tie goes to the lower level. */
void oracle_midpoints(const float* q, float* mid) {
  for (int i = 0; i < 255; ++i) mid[i] = (q[i] + q[i + 1]) * 0.5f;
}

int oracle_code(const float* mid, float xn) {
  int c = 0;
  for (int i = 0; i < 255; ++i)
    if (mid[i] < xn) c += 1;
  return c;
}

/* READING (normalisation): absmax = max |x| over the block (exact); the
 * reciprocal 1/absmax is taken once per block in binary32 (0 for an all-zero
 * block) and each element is normalised by one multiplication.
 * READING (a NaN in the block): the maximum is the IEEE 754-2019 maximum,
 * which is NaN when any operand is NaN.  The reciprocal of a NaN absmax is 0
 * (as for an all-zero block), so every value of the block takes the code of
 * 0 and the NaN the code of NaN (no midpoint lies below it: code 0); the NaN
 * absmax makes the whole block NaN when it is next dequantized.  A maximum
 * that skipped the NaN would instead store it as the lowest level times a
 * finite absmax: a finite, wrong state. */
static float block_inverse(float absmax) {
  return absmax > 0.0f ? 1.0f / absmax : 0.0f;
}
/* max |x| over x[0..n) with the IEEE 754-2019 maximum's NaN rule */
static float block_absmax(const float* x, int64_t n) {
  float amax = 0.0f;
  for (int64_t i = 0; i < n; ++i) {
    float a = fabsf(x[i]);
    if (isnan(a)) return a;
    if (a > amax) amax = a;
  }
  return amax;
}

/* [P4] abstract: block-wise quantization splits the tensor into blocks of B
 * elements that are normalised and quantized independently; [P1] benchmark
 * script: F.dequantize_blockwise(code, absmax, A, blocksize) is the inverse.
 * The last block may be shorter than B. */
void oracle_quantize_blockwise(const void* x, int dtype, int64_t n, const float* q,
                               int64_t B, uint8_t* codes, float* absmax) {
  float mid[255];
  oracle_midpoints(q, mid);
  int64_t nblocks = (n + B - 1) / B;
  for (int64_t b = 0; b < nblocks; ++b) {
    int64_t lo = b * B, hi = lo + B < n ? lo + B : n;
    float amax = 0.0f;   /* as block_absmax, over the block's loaded values */
    for (int64_t i = lo; i < hi; ++i) {
      float a = fabsf(load_elem(x, dtype, i));
      if (isnan(a)) { amax = a; break; }
      if (a > amax) amax = a;
    }
    absmax[b] = amax;
    float inv = block_inverse(amax);
    for (int64_t i = lo; i < hi; ++i)
      codes[i] = (uint8_t)oracle_code(mid, load_elem(x, dtype, i) * inv);
  }
}

void oracle_dequantize_blockwise(const uint8_t* codes, const float* absmax, const float* q,
                                 int64_t B, int64_t n, void* out, int dtype) {
  for (int64_t i = 0; i < n; ++i) store_elem(out, dtype, i, q[codes[i]] * absmax[i / B]);
}

/* ---- per-step scalars -----------------------------------------------------
 * [P2] Optimizer2State/Optimizer1State parameters; the step count t is the
 * 1-based number of the update.  Formed in binary64, rounded once.
 * AdEMAMix schedules (Pagliardini et al., "The AdEMAMix Optimizer", the
 * alpha and beta3 warm-up schedulers referred to by t_alpha / t_beta3 on
 * [P2]):  alpha_t = min(t*alpha/T_alpha, alpha);
 *         beta3_t = min(exp(ln b1 * ln b3 / ((1 - t/T) ln b3 + (t/T) ln b1)), b3).
 */
void oracle_scalars(const oracle_hparams* hp, step_scalars* sc) {
  double t = (double)hp->step;
  double b1 = (double)hp->beta1, b2 = (double)hp->beta2, b3 = (double)hp->beta3;
  double lr = (double)hp->lr, eps = (double)hp->eps, wd = (double)hp->weight_decay;
  double bc1 = 1.0 - pow(b1, t);
  double bc2 = 1.0 - pow(b2, t);
  memset(sc, 0, sizeof(*sc));
  sc->b1 = hp->beta1;
  sc->b2 = hp->beta2;
  sc->omb1 = (float)(1.0 - b1);
  sc->omb2 = (float)(1.0 - b2);
  sc->decay = (float)(1.0 - lr * wd);
  sc->unorm_c = 1.0;
  sc->step_size = hp->lr;
  sc->eps_hat = hp->eps;
  switch (hp->optim) {
    case OR_ADAM:
    case OR_ADAMW:
      /* lr/bc1 * m/(sqrt(v)/sqrt(bc2) + eps) == (lr*sqrt(bc2)/bc1) * m/(sqrt(v) + eps*sqrt(bc2)) */
      sc->step_size = (float)(lr * sqrt(bc2) / bc1);
      sc->eps_hat = (float)(eps * sqrt(bc2));
      sc->unorm_c = sqrt(bc2) / bc1;
      break;
    case OR_ADEMAMIX: {
      double a = (double)hp->alpha;
      double at = a;
      if (hp->t_alpha > 0) {
        double ramp = t * a / (double)hp->t_alpha;
        at = ramp < a ? ramp : a;
      }
      double b3t = b3;
      if (hp->t_beta3 > 0) {
        double r = t / (double)hp->t_beta3;
        double lb1 = log(b1), lb3 = log(b3);
        double s = exp(lb1 * lb3 / ((1.0 - r) * lb3 + r * lb1));
        b3t = s < b3 ? s : b3;
      }
      sc->alpha_t = (float)at;
      sc->b3t = (float)b3t;
      sc->omb3t = (float)(1.0 - (double)sc->b3t);
      sc->inv_bc1 = (float)(1.0 / bc1);
      sc->step_size = (float)(lr * sqrt(bc2));
      sc->eps_hat = (float)(eps * sqrt(bc2));
      sc->unorm_c = sqrt(bc2);
      break;
    }
    default:
      break;
  }
}

static int nstates(int optim) {
  if (optim == OR_ADAM || optim == OR_ADAMW) return 2;
  if (optim == OR_ADEMAMIX) return 3;
  return 1;
}

static int decoupled(int optim) {
  return optim == OR_ADAMW || optim == OR_LION || optim == OR_ADEMAMIX;
}

/* ---- one element of one optimizer ----------------------------------------
 * READING (update equations): the pages name torch's 32-bit optimizers as the
 * comparators ([P1] benchmark script: torch.optim.Adam / AdamW / SGD(lr,
 * momentum) / RMSprop(lr, alpha), Lion, the AdEMAMix reference) but print no
 * equations and no operation order.  The textbook forms below reproduce those
 * optimizers with zero initial state.  Every operation is one binary32
 * rounding, in this order; fma(a, b, c) is IEEE 754 fusedMultiplyAdd (a*b+c
 * rounded once), used wherever a product is added to something:
 *
 *   g  = g_raw * gnorm_scale;   coupled decay (Adam, Momentum, RMSprop,
 *                               Adagrad) when wd != 0:  g = fma(wd, p, g)
 *   Adam/AdamW: m = fma(b1, m, (1-b1)*g);  v = fma(b2, v, (1-b2)*(g*g))
 *               u = m / (sqrt(v) + eps_hat)
 *   Momentum:   m = fma(b1, m, g);         u = m
 *   RMSprop:    v = fma(b1, v, (1-b1)*(g*g));  u = g / (sqrt(v) + eps)
 *   Adagrad:    v = fma(g, g, v);          u = g / (sqrt(v) + eps)
 *   Lion:       c = fma(b1, m, (1-b1)*g);  u = sign(c);  m = fma(b2, m, (1-b2)*g)
 *   AdEMAMix:   m1 = fma(b1, m1, (1-b1)*g);  m2 = fma(b3t, m2, (1-b3t)*g);
 *               nu = fma(b2, nu, (1-b2)*(g*g));
 *               u = fma(m1, inv_bc1, alpha_t*m2) / (sqrt(nu) + eps_hat)
 *   decoupled decay (AdamW, Lion, AdEMAMix) when wd != 0:  p = p * (1 - lr*wd)
 *   p = fma(-(step_size * clip), u, p)
 *
 * [P3] skip_zeros: where the raw gradient is exactly zero the parameter and
 * the states keep their old values (tested before gnorm_scale and decay).
 */
typedef struct {
  float s[3];  /* new state values */
  float u;     /* update direction (0 where skipped) */
  float p;     /* new parameter value */
  int skipped;
} elem_result;

static elem_result update_element(const oracle_hparams* hp, const step_scalars* sc,
                                  float step_eff, float p, float g_raw, const float* s_old) {
  elem_result r;
  int ns = nstates(hp->optim);
  for (int j = 0; j < 3; ++j) r.s[j] = j < ns ? s_old[j] : 0.0f;
  r.u = 0.0f;
  r.p = p;
  r.skipped = hp->skip_zeros && g_raw == 0.0f;
  if (r.skipped) return r;

  float wd = hp->weight_decay;
  float g = g_raw * hp->gnorm_scale;
  if (!decoupled(hp->optim) && wd != 0.0f) g = fmaf(wd, p, g);

  float u = 0.0f;
  switch (hp->optim) {
    case OR_ADAM:
    case OR_ADAMW: {
      float m = fmaf(sc->b1, s_old[0], sc->omb1 * g);
      float v = fmaf(sc->b2, s_old[1], sc->omb2 * (g * g));
      u = m / (sqrtf(v) + sc->eps_hat);
      r.s[0] = m;
      r.s[1] = v;
      break;
    }
    case OR_MOMENTUM: {
      float m = fmaf(sc->b1, s_old[0], g);
      u = m;
      r.s[0] = m;
      break;
    }
    case OR_RMSPROP: {
      float v = fmaf(sc->b1, s_old[0], sc->omb1 * (g * g));
      u = g / (sqrtf(v) + sc->eps_hat);
      r.s[0] = v;
      break;
    }
    case OR_ADAGRAD: {
      float v = fmaf(g, g, s_old[0]);
      u = g / (sqrtf(v) + sc->eps_hat);
      r.s[0] = v;
      break;
    }
    case OR_LION: {
      float c = fmaf(sc->b1, s_old[0], sc->omb1 * g);
      u = c > 0.0f ? 1.0f : (c < 0.0f ? -1.0f : 0.0f);
      r.s[0] = fmaf(sc->b2, s_old[0], sc->omb2 * g);
      break;
    }
    case OR_ADEMAMIX: {
      float m1 = fmaf(sc->b1, s_old[0], sc->omb1 * g);
      float m2 = fmaf(sc->b3t, s_old[1], sc->omb3t * g);
      float nu = fmaf(sc->b2, s_old[2], sc->omb2 * (g * g));
      u = fmaf(m1, sc->inv_bc1, sc->alpha_t * m2) / (sqrtf(nu) + sc->eps_hat);
      r.s[0] = m1;
      r.s[1] = m2;
      r.s[2] = nu;
      break;
    }
    default:
      break;
  }
  if (decoupled(hp->optim) && wd != 0.0f) p = p * sc->decay;
  r.p = fmaf(-step_eff, u, p);
  r.u = u;
  return r;
}

/* ---- state access (8-bit codes or 32-bit floats) -------------------------
 * [P1] benchmark script, statenames: Adam-family tensors carry state1/qmap1/
 * absmax1 (first moment, signed map) and state2/qmap2/absmax2 (second moment,
 * unsigned map); AdEMAMix keeps m1 and m2 stacked as state1 = [2, N] codes
 * with absmax1 = [2, nblocks] sharing qmap1, and nu in state2.
 * READING (1-state map choice): Momentum and Lion states are signed (qmap1
 * should be the signed map), RMSprop and Adagrad states are non-negative
 * (the caller passes the unsigned map as qmap1).  The oracle uses whatever
 * map it is given.
 */
typedef struct {
  void* base;            /* uint8 codes or float values */
  float* absmax;         /* per block (8-bit only) */
  const float* q;        /* the map (8-bit only) */
} state_ref;

static void state_refs(int optim, int state_bits, int64_t n, int64_t B, void* s1, void* s2,
                       float* absmax1, float* absmax2, const float* q1, const float* q2,
                       state_ref* out) {
  int64_t nb = (n + B - 1) / B;
  int64_t esz = state_bits == 8 ? 1 : 4;
  memset(out, 0, 3 * sizeof(state_ref));
  out[0].base = s1;
  out[0].absmax = absmax1;
  out[0].q = q1;
  if (optim == OR_ADEMAMIX) {
    out[1].base = (char*)s1 + n * esz;
    out[1].absmax = absmax1 ? absmax1 + nb : NULL;
    out[1].q = q1;
    out[2].base = s2;
    out[2].absmax = absmax2;
    out[2].q = q2;
  } else {
    out[1].base = s2;
    out[1].absmax = absmax2;
    out[1].q = q2;
  }
}

static float read_state(const state_ref* s, int state_bits, int64_t i, int64_t B) {
  if (state_bits == 32) return ((const float*)s->base)[i];
  return s->q[((const uint8_t*)s->base)[i]] * s->absmax[i / B];
}

/* ---- max_unorm -------------------------------------------------------------
 * [P2] max_unorm: "the maximum value to normalize each block with", default
 * 0.0 (off).  READING: per tensor, with U = ||d|| the norm of the true update
 * direction d = unorm_c * u (lr excluded, decoupled decay excluded, skipped
 * elements contribute 0) and P = ||p|| before the step: if U > max_unorm * P
 * the step is multiplied by max_unorm * P / U.  Sums are taken in binary64.
 */
float oracle_unorm_scale(const oracle_hparams* hp, const void* p, const void* g, void* s1,
                         void* s2, float* absmax1, float* absmax2, int64_t n, int state_bits,
                         int dtype, int64_t B, const float* q1, const float* q2, double* U_out,
                         double* P_out) {
  step_scalars sc;
  oracle_scalars(hp, &sc);
  state_ref st[3];
  state_refs(hp->optim, state_bits, n, B, s1, s2, absmax1, absmax2, q1, q2, st);
  int ns = nstates(hp->optim);
  double usum = 0.0, psum = 0.0;
  for (int64_t i = 0; i < n; ++i) {
    float s_old[3] = {0.0f, 0.0f, 0.0f};
    for (int j = 0; j < ns; ++j) s_old[j] = read_state(&st[j], state_bits, i, B);
    float pv = load_elem(p, dtype, i);
    elem_result r = update_element(hp, &sc, sc.step_size, pv, load_elem(g, dtype, i), s_old);
    usum += (double)r.u * (double)r.u;
    psum += (double)pv * (double)pv;
  }
  double unorm = sc.unorm_c * sqrt(usum);
  double pnorm = sqrt(psum);
  if (U_out) *U_out = unorm;
  if (P_out) *P_out = pnorm;
  double limit = (double)hp->max_unorm * pnorm;
  if (hp->max_unorm > 0.0f && unorm > limit) return (float)(limit / unorm);
  return 1.0f;
}

/* The squared parameter norm, sum of p[i]^2 in binary64 in element order.
 * It is the P^2 of the max_unorm test above when p is the parameter as the
 * call finds it, so for the parameter one step leaves it is the P^2 of the
 * next step's test: the quantity a step that carries the norm forward forms
 * while it writes p.  ([P2] max_unorm, as read above.) */
double oracle_param_sumsq(const void* p, int dtype, int64_t n) {
  double psum = 0.0;
  for (int64_t i = 0; i < n; ++i) {
    const double v = (double)load_elem(p, dtype, i);
    psum += v * v;
  }
  return psum;
}

/* READING (the alternative, per block): the same test with U and P taken
 * over one block of B elements (the quantization blocks of 8-bit states; the
 * same partition of a tensor with 32-bit states), each block getting its own
 * multiplier.  Elements lo..hi-1 of the tensor; sums in binary64, in element
 * order. */
static float block_unorm_scale(const oracle_hparams* hp, const step_scalars* sc, const void* p,
                               const void* g, const state_ref* st, int ns, int state_bits,
                               int dtype, int64_t B, int64_t lo, int64_t hi) {
  double usum = 0.0, psum = 0.0;
  for (int64_t i = lo; i < hi; ++i) {
    float s_old[3] = {0.0f, 0.0f, 0.0f};
    for (int j = 0; j < ns; ++j) s_old[j] = read_state(&st[j], state_bits, i, B);
    float pv = load_elem(p, dtype, i);
    elem_result r = update_element(hp, sc, sc->step_size, pv, load_elem(g, dtype, i), s_old);
    usum += (double)r.u * (double)r.u;
    psum += (double)pv * (double)pv;
  }
  double unorm = sc->unorm_c * sqrt(usum);
  double limit = (double)hp->max_unorm * sqrt(psum);
  if (hp->max_unorm > 0.0f && unorm > limit) return (float)(limit / unorm);
  return 1.0f;
}

/* ---- the optimizer step on one tensor --------------------------------------
 * One update of parameter p with gradient g (same dtype) and its states.
 * 8-bit states: for every block, dequantize the old states (code -> q[code] *
 * absmax), update every element, write p (one rounding to its dtype), then
 * requantize each new state with a fresh absmax.  READING: p is updated from
 * the unquantized binary32 new states; requantization follows.  A block in
 * which every element was skipped (skip_zeros) keeps its codes and absmax
 * bit-identical; otherwise skipped elements re-enter requantization with
 * their old dequantized values.
 * 32-bit states ([P2] min_8bit_size: smaller tensors keep 32-bit state): the
 * same element update with binary32 state arrays.
 * Returns the step multiplier applied (1 unless max_unorm clipped).
 * oracle_step_clipped takes the multiplier from the caller (clip_in >= 0)
 * so that a subset of a tensor's blocks can be stepped with the multiplier
 * of the whole tensor; blocks are otherwise independent.
 */
float oracle_step_clipped(const oracle_hparams* hp, void* p, const void* g, void* s1, void* s2,
                          float* absmax1, float* absmax2, int64_t n, int state_bits, int dtype,
                          int64_t B, const float* q1, const float* q2, float clip_in) {
  step_scalars sc;
  oracle_scalars(hp, &sc);
  const int per_block = hp->unorm_per_block && hp->max_unorm > 0.0f;
  float clip = 1.0f;
  if (per_block)
    clip = 1.0f; /* each block takes its own multiplier below */
  else if (clip_in >= 0.0f)
    clip = clip_in; /* a multiplier the caller took from oracle_unorm_scale on the whole tensor */
  else if (hp->max_unorm > 0.0f)
    clip = oracle_unorm_scale(hp, p, g, s1, s2, absmax1, absmax2, n, state_bits, dtype, B, q1,
                              q2, NULL, NULL);
  float step_eff = sc.step_size * clip;

  state_ref st[3];
  state_refs(hp->optim, state_bits, n, B, s1, s2, absmax1, absmax2, q1, q2, st);
  int ns = nstates(hp->optim);

  if (state_bits == 32) {
    for (int64_t i = 0; i < n; ++i) {
      if (per_block && i % B == 0) {
        int64_t hi = i + B < n ? i + B : n;
        step_eff = sc.step_size *
                   block_unorm_scale(hp, &sc, p, g, st, ns, 32, dtype, B, i, hi);
      }
      float s_old[3] = {0.0f, 0.0f, 0.0f};
      for (int j = 0; j < ns; ++j) s_old[j] = ((float*)st[j].base)[i];
      elem_result r =
          update_element(hp, &sc, step_eff, load_elem(p, dtype, i), load_elem(g, dtype, i), s_old);
      if (r.skipped) continue;
      for (int j = 0; j < ns; ++j) ((float*)st[j].base)[i] = r.s[j];
      store_elem(p, dtype, i, r.p);
    }
    return clip;
  }

  float mids[3][255];
  for (int j = 0; j < ns; ++j) oracle_midpoints(st[j].q, mids[j]);
  float* snew = (float*)malloc(sizeof(float) * 3 * (size_t)B);
  float* pnew = (float*)malloc(sizeof(float) * (size_t)B);
  int* skipped = (int*)malloc(sizeof(int) * (size_t)B);
  int64_t nblocks = (n + B - 1) / B;
  for (int64_t b = 0; b < nblocks; ++b) {
    int64_t lo = b * B, hi = lo + B < n ? lo + B : n;
    int any_update = 0;
    if (per_block)
      step_eff = sc.step_size * block_unorm_scale(hp, &sc, p, g, st, ns, 8, dtype, B, lo, hi);
    for (int64_t i = lo; i < hi; ++i) {
      float s_old[3] = {0.0f, 0.0f, 0.0f};
      for (int j = 0; j < ns; ++j) s_old[j] = read_state(&st[j], 8, i, B);
      elem_result r =
          update_element(hp, &sc, step_eff, load_elem(p, dtype, i), load_elem(g, dtype, i), s_old);
      for (int j = 0; j < ns; ++j) snew[j * B + (i - lo)] = r.s[j];
      pnew[i - lo] = r.p;
      skipped[i - lo] = r.skipped;
      if (!r.skipped) any_update = 1;
    }
    if (!any_update) continue; /* all skipped: codes, absmax and p untouched */
    for (int64_t i = lo; i < hi; ++i)
      if (!skipped[i - lo]) store_elem(p, dtype, i, pnew[i - lo]);
    for (int j = 0; j < ns; ++j) {
      float amax = block_absmax(snew + j * B, hi - lo);
      st[j].absmax[b] = amax;
      float inv = block_inverse(amax);
      uint8_t* codes = (uint8_t*)st[j].base;
      for (int64_t i = lo; i < hi; ++i)
        codes[i] = (uint8_t)oracle_code(mids[j], snew[j * B + (i - lo)] * inv);
    }
  }
  free(snew);
  free(pnew);
  free(skipped);
  return clip;
}

/* The step on a whole tensor: the max_unorm multiplier (if any) is computed
 * from this tensor. */
float oracle_step(const oracle_hparams* hp, void* p, const void* g, void* s1, void* s2,
                  float* absmax1, float* absmax2, int64_t n, int state_bits, int dtype, int64_t B,
                  const float* q1, const float* q2) {
  return oracle_step_clipped(hp, p, g, s1, s2, absmax1, absmax2, n, state_bits, dtype, B, q1, q2,
                             -1.0f);
}
