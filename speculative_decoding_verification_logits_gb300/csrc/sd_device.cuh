// Device code shared by the translation units of the verify library:
// element types, float-float arithmetic, Philox, row geometry, the
// streaming loop and the per-sequence cluster kernel, plus the host
// helpers both launch paths use.
#pragma once


#include "sd_verify.h"

#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

namespace cg = cooperative_groups;

namespace sdv {

constexpr int kU = 4;                        // 16-byte vectors per thread per step
constexpr int kDepth = 3;                    // steps in each thread's copy ring
constexpr int kMaxWarps = 16;                // threads per CTA <= 512
constexpr int kMaxCS = 16;                   // cluster size limit
constexpr int kMaxRows = 2 * SD_MAX_K + 2;   // K+1 target, K draft, 1 bonus
constexpr float kRebase = 16.f;              // log2 headroom of the exp offset
constexpr float kBig = 1048576.f;            // a step sum above 2^20 moves the offset
constexpr float kL2eHi = 1.44269502162933349609375f;  // log2(e) = hi + lo
constexpr float kL2eLo = 1.925963033500011e-08f;

enum Mode : int { kVerify = 0, kPredict = 1 };
enum RowKind : int { kTarget = 0, kDraft = 1, kBonus = 2 };
enum RowFlag : int { kNeedExp = 1, kNeedArg = 2, kNeedKeys = 4 };

// Piece record of the split launch: the statistics of one CTA's piece of
// one row ({m, idx, c, zhi, zlo}) and its best keys ({value, index bits}).
constexpr int kRecBytes = 96;
constexpr int kRecKeys = 8;
constexpr int kMaxStreamGrid = 1024;         // CTAs of the streaming grid
constexpr int kMaxParts = 16;                // streaming CTAs covering one row

struct Params {
  const uint8_t *target;   // [B][K+1][V]
  const uint8_t *draft;    // [B][K][V]
  const uint8_t *bonus;    // [B][V] or null
  const int32_t *tokens;   // [B][K]
  const float *temps;      // [B]
  const int32_t *keys_in;  // [B][n_keys_in][2] or null
  int32_t *keys_out;       // [B][n_keys_out][2] or null
  int32_t *num_accepted, *out_tokens, *tau;
  uint8_t *hit;
  int32_t *offsets, *packed;
  float *ratio_out, *p_out, *q_out;
  int32_t *argmax_out;
  int32_t *status;
  uint64_t seed;
  int64_t row_base;
  int32_t B, K, V;
  int32_t mode;
  int32_t keys;            // build keys in this pass
  int32_t compact;
  int32_t n_keys_in, n_keys_out;
  int32_t cs, slice;       // cluster size, vocabulary slice per CTA (draw pass)
  int32_t rowsplit;        // stream split: 1 row-major over the sequence, 0 by slice
  int32_t fanout[SD_MAX_K + 1];
  int32_t fan_off[SD_MAX_K + 2];
  // Split launch (a flat streaming grid, then the per-sequence finish): the
  // rows of all sequences in groups g = 0..K for positions j = K - g; group
  // g holds, sequence by sequence, row x_j (the bonus draft row for j = K,
  // draft row j below) if present, then target row j.  grp_x[g]: x_j absent
  // (0), present for the sampled sequences only (1), for all sequences (2).
  uint8_t *ws;             // piece records [gstream + rows][kRecBytes]
  int32_t spr;             // streaming steps per row
  int32_t gstream;         // CTAs of the streaming grid
  int8_t grp_x[SD_MAX_K + 1];
  size_t ws_bytes;         // bytes at ws
  int32_t chk;             // SD_FLAG_CHECK_FINITE: rows read are checked
  int32_t kf;              // key candidates per piece record (split launch)
  int32_t pw;              // split finish: draw iterations per warp (mass rows)
};

// ------------------------------------------------------------------ Philox --
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11): ten rounds of two
// 32x32->64 multiplies of counter words 0 and 2 by the round multipliers,
// high halves xored with the other counter words and the key, key bumped
// by the Weyl increments between rounds.  Only output word 0 is used.
__device__ __forceinline__ uint32_t philox_w0(uint64_t seed, uint32_t row, uint32_t pos,
                                              uint32_t slot) {
  uint32_t c0 = row, c1 = pos, c2 = slot, c3 = 0u;
  uint32_t k0 = (uint32_t)seed, k1 = (uint32_t)(seed >> 32);
#pragma unroll 1
  for (int r = 0; r < 10; ++r) {
    const uint32_t m0 = 0xD2511F53u, m1 = 0xCD9E8D57u;
    const uint32_t hi0 = __umulhi(m0, c0), lo0 = m0 * c0;
    const uint32_t hi1 = __umulhi(m1, c2), lo1 = m1 * c2;
    const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
    c0 = n0;
    c1 = lo1;
    c2 = n2;
    c3 = lo0;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return c0;
}

// u in (0, 1], a multiple of 2^-24: exact in float.
__device__ __forceinline__ float uniform_u(uint64_t seed, int64_t row, int pos, int slot) {
  const uint32_t x = philox_w0(seed, (uint32_t)row, (uint32_t)pos, (uint32_t)slot);
  return (float)((x >> 8) + 1u) * 5.9604644775390625e-8f;
}

// ------------------------------------------------------------- primitives --
// 2^x on the special-function unit.  Results below 2^-126 flush to zero, far
// below anything that moves a sum of at least 1.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// s = log2(e) / T rounded to float: log2(e) = kL2eHi + kL2eLo divided with
// one correction step.  Every kernel derives a row's scale from T this way.
__device__ __forceinline__ float log2e_over(float T) {
  const float q = __fdiv_rn(kL2eHi, T);
  return q + __fdiv_rn(fmaf(-q, T, kL2eHi) + kL2eLo, T);
}

// ---------------------------------------------- float-float arithmetic --
// Sums and products carried as an unevaluated pair hi + lo: Knuth's two-sum,
// Dekker's fast two-sum (|a| >= |b|) and the fma form of the exact product,
// about 48 significant bits on the fp32 pipe.  (The fp64 pipe of this part
// is slow enough that a handful of dependent double operations costs
// microseconds.)
struct ff {
  float hi, lo;
};
__device__ __forceinline__ ff two_sum(float a, float b) {
  const float s = a + b;
  const float bb = s - a;
  return ff{s, (a - (s - bb)) + (b - bb)};
}
__device__ __forceinline__ ff fast_two_sum(float a, float b) {
  const float s = a + b;
  return ff{s, b - (s - a)};
}
__device__ __forceinline__ ff two_prod(float a, float b) {
  const float p = a * b;
  return ff{p, fmaf(a, b, -p)};
}
__device__ __forceinline__ ff ff_add(ff x, ff y) {
  const ff t = two_sum(x.hi, y.hi);
  return fast_two_sum(t.hi, t.lo + (x.lo + y.lo));
}
__device__ __forceinline__ ff ff_add_f(ff x, float y) {
  const ff t = two_sum(x.hi, y);
  return fast_two_sum(t.hi, t.lo + x.lo);
}
__device__ __forceinline__ ff ff_sub(ff x, ff y) { return ff_add(x, ff{-y.hi, -y.lo}); }
__device__ __forceinline__ ff ff_mul_f(ff x, float y) {
  const ff p = two_prod(x.hi, y);
  return fast_two_sum(p.hi, fmaf(x.lo, y, p.lo));
}
__device__ __forceinline__ bool ff_gt(ff x, ff y) {
  return x.hi > y.hi || (x.hi == y.hi && x.lo > y.lo);
}
__device__ __forceinline__ bool ff_pos(ff x) { return x.hi > 0.f; }
__device__ __forceinline__ float ff_f(ff x) { return x.hi + x.lo; }
// a / b for float-float a, b > 0, rounded to float: one correction step on
// the float quotient with the remainder carried exactly (within an ulp).
__device__ __forceinline__ float ff_ratio(ff a, ff b) {
  const float q0 = __fdiv_rn(a.hi, b.hi);
  const ff p = two_prod(q0, b.hi);
  const float r = ((a.hi - p.hi) - p.lo) + fmaf(-q0, b.lo, a.lo);
  return q0 + __fdiv_rn(r, b.hi);
}
__device__ __forceinline__ ff ff_shfl(ff x, int src) {
  __syncwarp();
  return ff{__shfl_sync(0xffffffffu, x.hi, src), __shfl_sync(0xffffffffu, x.lo, src)};
}
__device__ __forceinline__ ff ff_shfl_up(ff x, int o) {
  return ff{__shfl_up_sync(0xffffffffu, x.hi, o), __shfl_up_sync(0xffffffffu, x.lo, o)};
}
__device__ __forceinline__ ff ff_shfl_xor(ff x, int o) {
  return ff{__shfl_xor_sync(0xffffffffu, x.hi, o), __shfl_xor_sync(0xffffffffu, x.lo, o)};
}
// inclusive warp scan and warp sum
static __device__ __noinline__ ff ff_warp_scan(ff x) {
  const int lane = threadIdx.x & 31;
  __syncwarp();
#pragma unroll 1
  for (int o = 1; o < 32; o <<= 1) {
    ff y = ff_shfl_up(x, o);
    y.hi = lane >= o ? y.hi : 0.f;  // adding (0, 0) leaves x as it is
    y.lo = lane >= o ? y.lo : 0.f;
    x = ff_add(x, y);
  }
  return x;
}
static __device__ __noinline__ ff ff_warp_sum(ff x) {
  __syncwarp();
#pragma unroll 1
  for (int o = 16; o > 0; o >>= 1) x = ff_add(x, ff_shfl_xor(x, o));
  return x;
}

// 2^(x.hi + x.lo) without a double-precision transcendental: the integer
// part of hi scales the result exactly, the fraction (hi - n exact, plus
// lo) goes through ex2 (relative error about 2^-22).  Below 2^-126: 0.
static __device__ __noinline__ float exp2_ff(ff x) {
  if (!(x.hi > -126.f)) return 0.f;
  if (x.hi >= 128.f) return INFINITY;
  const float n = floorf(x.hi);
  return ldexpf(ex2((x.hi - n) + x.lo), (int)n);
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
// 16-byte asynchronous copy global -> shared (L2 only), per thread
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// 16-byte global load through L2 only (read-once data)
__device__ __forceinline__ uint4 ld_stream(const uint8_t *p) {
  return __ldcg(reinterpret_cast<const uint4 *>(p));
}

__device__ __forceinline__ void kahan_add(float &sum, float &comp, float v) {
  const float y = v - comp;
  const float t = sum + y;
  comp = (t - sum) - y;
  sum = t;
}

__device__ __forceinline__ float warp_max(float v) {
  __syncwarp();
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
  __syncwarp();
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ int warp_min_i(int v) {
  __syncwarp();
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// ------------------------------------------------------ packed fp32 pairs --
// Two fp32 lanes per instruction (fma / add on a 64-bit register pair).
__device__ __forceinline__ uint64_t pk2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void upk2(uint64_t r, float &lo, float &hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// Order-preserving integer image of a float (-0 taken as +0), so warp-wide
// float minima and maxima run as single integer reductions.
__device__ __forceinline__ int ford(float x) {
  const int i = __float_as_int(x);
  return i >= 0 ? i : (i == (int)0x80000000 ? 0 : (i ^ 0x7fffffff));
}
__device__ __forceinline__ float fdeord(int i) { return __int_as_float(i >= 0 ? i : (i ^ 0x7fffffff)); }
// Every warp-collective helper below first reconverges the warp: lanes that
// took different sides of an earlier branch may otherwise reach the
// collective separately, and each such collective then costs hundreds of
// cycles.
__device__ __forceinline__ float rmax_f(float x) {
  __syncwarp();
  return fdeord(__reduce_max_sync(0xffffffffu, ford(x)));
}
__device__ __forceinline__ float rmin_f(float x) {
  __syncwarp();
  return fdeord(__reduce_min_sync(0xffffffffu, ford(x)));
}
__device__ __forceinline__ int rmin_i(int x) {
  __syncwarp();
  return __reduce_min_sync(0xffffffffu, x);
}
__device__ __forceinline__ unsigned ballot(bool p) {
  __syncwarp();
  return __ballot_sync(0xffffffffu, p);
}

// Warp-wide best (value desc, then index asc) of one candidate per lane.
__device__ __forceinline__ void warp_best(float &v, int &i) {
  const float mv = rmax_f(v);
  i = rmin_i(v == mv ? i : INT32_MAX);
  v = mv;
}

// --------------------------------------------------------- element types --
template <typename E>
struct Elt;
template <>
struct Elt<float> {
  static constexpr int kSize = 4;
  static constexpr int kPerVec = 4;
  static constexpr uint32_t kNegInfWord = 0xFF800000u;
  static __device__ __forceinline__ void unpack(const uint4 &v, float *f) {
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
  }
  static __device__ __forceinline__ float vmax(const uint4 &v) {
    return fmaxf(fmaxf(__uint_as_float(v.x), __uint_as_float(v.y)),
                 fmaxf(__uint_as_float(v.z), __uint_as_float(v.w)));
  }
  static __device__ __forceinline__ float load_global(const uint8_t *p) {
    return __ldg(reinterpret_cast<const float *>(p));
  }
  // max of the 4 values where a NaN wins: NaN or +inf anywhere shows here
  static __device__ __forceinline__ float vmax_nan(const uint4 &v) {
    float a, b, c;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(a) : "f"(__uint_as_float(v.x)), "f"(__uint_as_float(v.y)));
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(b) : "f"(__uint_as_float(v.z)), "f"(__uint_as_float(v.w)));
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(c) : "f"(a), "f"(b));
    return c;
  }
};
template <>
struct Elt<__nv_bfloat16> {
  static constexpr int kSize = 2;
  static constexpr int kPerVec = 8;
  static constexpr uint32_t kNegInfWord = 0xFF80FF80u;
  static __device__ __forceinline__ void unpack(const uint4 &v, float *f) {
    f[0] = __uint_as_float(v.x << 16);
    f[1] = __uint_as_float(v.x & 0xffff0000u);
    f[2] = __uint_as_float(v.y << 16);
    f[3] = __uint_as_float(v.y & 0xffff0000u);
    f[4] = __uint_as_float(v.z << 16);
    f[5] = __uint_as_float(v.z & 0xffff0000u);
    f[6] = __uint_as_float(v.w << 16);
    f[7] = __uint_as_float(v.w & 0xffff0000u);
  }
  // max of the 8 values with packed bf16x2 maxima (exact), then widened
  static __device__ __forceinline__ float vmax(const uint4 &v) {
    const __nv_bfloat162 a = __hmax2(*reinterpret_cast<const __nv_bfloat162 *>(&v.x),
                                     *reinterpret_cast<const __nv_bfloat162 *>(&v.y));
    const __nv_bfloat162 c = __hmax2(*reinterpret_cast<const __nv_bfloat162 *>(&v.z),
                                     *reinterpret_cast<const __nv_bfloat162 *>(&v.w));
    const __nv_bfloat162 m = __hmax2(a, c);
    const uint32_t w = *reinterpret_cast<const uint32_t *>(&m);
    return fmaxf(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
  }
  static __device__ __forceinline__ float load_global(const uint8_t *p) {
    return __uint_as_float((uint32_t)__ldg(reinterpret_cast<const unsigned short *>(p)) << 16);
  }
  // max of the 8 values where a NaN wins (packed bf16x2 maxima), widened
  static __device__ __forceinline__ float vmax_nan(const uint4 &v) {
    uint32_t a, c, m;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(a) : "r"(v.x), "r"(v.y));
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(c) : "r"(v.z), "r"(v.w));
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(m) : "r"(a), "r"(c));
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(__uint_as_float(m << 16)),
        "f"(__uint_as_float(m & 0xffff0000u)));
    return r;
  }
};

// ---------------------------------------------------------------- rows ----
// What a row's stream computes: exp-sums (E), argmax (A), key vectors (K).
enum RowType : int { kRowE = 0, kRowEA = 1, kRowA = 2, kRowK = 3, kRowEK = 4 };

// One logit row as this CTA sees it: the slice [v0, v1) occupies `nvec`
// 16-byte vectors starting at `gbase`, the 16-byte boundary at or below
// element v0 (element v0 sits `hp` bytes into vector 0).  Vectors in
// [qlo, qhi) lie wholly inside the slice and are copied with cp.async; the
// (at most two) others are assembled from element loads with -inf in the
// bytes outside the slice, so every vector a thread sees is a plain list of
// logits with -inf padding.  Step t covers vectors [t NT kU, (t+1) NT kU);
// steps [sf0, sf1) lie wholly inside [qlo, qhi).  `qd` is the vector holding
// the token excluded from this row's keys (-1 if it is not in this slice).
struct RowInfo {
  const uint8_t *g;      // element 0 of the row
  const uint8_t *gbase;  // 16-byte boundary at or below element v0
  int v0, v1;            // the elements [v0, v1) of the row this CTA covers
  int kind, j, type;     // RowKind, position, RowType
  int excl;              // token excluded from the keys (-1: none)
  int fan;               // keys wanted from this row
  float s;               // log2(e) / T of the row's sequence (split stream)
  int rec;               // piece record of this row (split stream)
  int hp, nvec, nsteps, qlo, qhi, sf0, sf1, qd, qd_step;
};

// Element index of element i of slice vector q.
__device__ __forceinline__ int elem_index(int v0, int hp, int q, int i, int sz) {
  return v0 + (q * 16 - hp) / sz + i;
}

template <int NT>
__device__ __noinline__ void row_geometry(RowInfo &R, int v0, int v1, int sz) {
  constexpr int kStepVec = NT * kU;
  R.gbase = R.g;
  R.v0 = v0;
  R.v1 = v1;
  R.hp = R.nvec = R.nsteps = R.qlo = R.qhi = R.sf0 = R.sf1 = 0;
  R.qd = R.qd_step = -1;
  if (v1 <= v0) return;
  const uintptr_t a0 = (uintptr_t)(R.g + (int64_t)v0 * sz);
  const uintptr_t a1 = (uintptr_t)(R.g + (int64_t)v1 * sz);
  const uintptr_t gf = a0 & ~(uintptr_t)15, gl = (a1 + 15) & ~(uintptr_t)15;
  R.gbase = reinterpret_cast<const uint8_t *>(gf);
  R.hp = (int)(a0 - gf);
  R.nvec = (int)((gl - gf) / 16);
  R.nsteps = (R.nvec + kStepVec - 1) / kStepVec;
  R.qlo = R.hp == 0 ? 0 : 1;
  R.qhi = (a1 & 15) == 0 ? R.nvec : R.nvec - 1;
  R.sf0 = R.qlo > 0 ? 1 : 0;
  R.sf1 = umax(R.sf0, R.qhi / kStepVec);
  if (R.excl >= v0 && R.excl < v1) {
    R.qd = ((R.excl - v0) * sz + R.hp) / 16;
    R.qd_step = R.qd / kStepVec;
  }
}

// Vector q of row R's slice assembled from element loads (ragged ends), or
// all -inf past the slice.
template <typename E>
__device__ __noinline__ uint4 load_vec_slow(const RowInfo &R, int q, int v0, int v1) {
  constexpr int sz = Elt<E>::kSize, N = Elt<E>::kPerVec;
  const uint32_t ninf = Elt<E>::kNegInfWord;
  uint32_t w[4] = {ninf, ninf, ninf, ninf};
  if (q < R.nvec) {
#pragma unroll
    for (int i = 0; i < N; ++i) {
      const int e = elem_index(v0, R.hp, q, i, sz);
      if (e >= v0 && e < v1) {
        if (sz == 4) {
          w[i] = __ldg(reinterpret_cast<const unsigned int *>(R.g + (int64_t)e * 4));
        } else {
          const uint32_t h = __ldg(reinterpret_cast<const unsigned short *>(R.g + (int64_t)e * 2));
          w[i >> 1] = (i & 1) ? ((w[i >> 1] & 0x0000ffffu) | (h << 16))
                              : ((w[i >> 1] & 0xffff0000u) | h);
        }
      }
    }
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// Vector q of row R's slice read directly (128-bit load through L2 when it
// lies inside the slice).
template <typename E>
__device__ __forceinline__ uint4 load_vec_direct(const RowInfo &R, int q, int v0, int v1) {
  if (q >= R.qlo && q < R.qhi) return __ldcg(reinterpret_cast<const uint4 *>(R.gbase + 16 * q));
  return load_vec_slow<E>(R, q, v0, v1);
}

// -------------------------------------------------------- shared memory --
// Per-warp statistics of one row: max, sum z of 2^(l s + c), offset c,
// lowest index of the max.
struct WStat {
  float m, z, c;
  int idx;
};
// Per-CTA statistics of one row, pushed into every CTA of the cluster.
struct CStat {
  float m;
  int idx;
  float c;
  float zhi, zlo;  // sum of 2^(l s + c) as a float-float pair
};

// Dynamic shared memory carve-out (byte offsets), identical on host and
// device.  nrows: rows streamed per sequence; npos: K + 1 key positions;
// KF: keys kept per row; cs: cluster size.
struct Layout {
  int ring, wstat, wsel, cstat, ckeys, cmass, pmass, pw, total;
};
// Steps of 64 vectors in one warp's share of a slice of `slice` elements.
__host__ __device__ inline int pass_steps(int slice, int sz, int NT) {
  const int nvec = (slice * sz + 31) / 16 + 1, nw = NT / 32;
  return ((nvec + nw - 1) / nw + 63) / 64;
}
__host__ __device__ inline int align128(int x) { return (x + 127) & ~127; }
__host__ __device__ inline Layout make_layout(int NT, int nrows, int npos, int KF, int cs,
                                              int slice, int sz) {
  const int nw = NT / 32, kf = KF > 0 ? KF : 1, kp = KF > 0 ? npos : 0;
  Layout L;
  int o = 0;
  L.ring = o;                                   // [kDepth][kU][NT] 16-byte vectors
  o = align128(o + kDepth * kU * NT * 16);
  L.wstat = o;                                  // [nrows][nw] WStat
  o = align128(o + 16 * nrows * nw);
  L.wsel = o;                                   // [npos][nw][KF] key vectors chosen by each warp
  o = align128(o + 4 * kp * nw * kf);
  L.cstat = o;                                  // [cs][nrows] CStat, slot p written by CTA p
  o = align128(o + 20 * cs * nrows);
  L.ckeys = o;                                  // [cs][npos][KF] {value, index}
  o = align128(o + 8 * cs * kp * kf);
  L.cmass = o;                                  // [2][cs] float-float: slice masses of the draw
  o = align128(o + 16 * cs);
  L.pw = pass_steps(slice, sz, NT);
  L.pmass = o;                                  // [nw][pw][32] float: masses of the draw
  o = align128(o + 4 * nw * L.pw * 32);
  L.total = o;
  return L;
}

struct Static {
  RowInfo rows[kMaxRows];
  int trow[SD_MAX_K + 1];  // row slot of target row j
  int drow[SD_MAX_K + 1];  // row slot of draft row j (K: bonus row), -1 if absent
  int nrows;
  int dvalid;
  int d[SD_MAX_K];         // drafted tokens
  float ld_t[SD_MAX_K];    // target logit of d_j
  float ld_d[SD_MAX_K];    // draft logit of d_j
  float M[kMaxRows];       // combined row statistics: max,
  float C[kMaxRows];       //   offset C: sum over the row of 2^(l s) = Z 2^-C
  ff Z[kMaxRows];
  int amax[kMaxRows];      //   lowest index of the max
  int2 keys[(SD_MAX_K + 1) * SD_MAX_FANOUT];  // this sequence's keys (fused prediction)
  RowInfo dt, dd;             // draw: target and draft row at m on the vocabulary slice
  int m, kind, owner, valid;  // kind: 0 none, 1 residual at m, 2 from p at m
  ff t_loc;
  int cstar;
  ff wmass[kMaxWarps];        // draw: mass of each warp's range, and its prefix
  ff wpre[kMaxWarps];
  int wsel;                   //   the warp holding the crossing point
  ff t_w;
  int red_i[kMaxWarps];
  float u_acc[SD_MAX_K];      // accept uniforms u(b, j, 0)
  float u_draw[SD_MAX_K + 1]; // draw uniforms u(b, m, 1) for every m
  int fvalid;                 // 0: a row read failed the finiteness check
  int tok;
};

// Copy-ahead cursor: the next step this thread copies.
struct Issuer {
  const uint8_t *ptr;  // this thread's vector 0 of `step`
  uint32_t slot;       // shared address of this thread's vector 0 in the slot to fill
  int row, step, nsteps, sf0, sf1, qlo, qhi;
};

template <int NT>
__device__ __forceinline__ void issuer_row(Issuer &I, const Static &S, int nrows) {
  while (I.row < nrows && S.rows[I.row].nsteps == 0) ++I.row;
  if (I.row < nrows) {
    const RowInfo &R = S.rows[I.row];
    I.step = 0;
    I.nsteps = R.nsteps;
    I.sf0 = R.sf0;
    I.sf1 = R.sf1;
    I.qlo = R.qlo;
    I.qhi = R.qhi;
    I.ptr = R.gbase + 16 * threadIdx.x;
  }
}

// --------------------------------------------------------- finalization --
// Exclusive scan of tau and packing of out_tokens, one CTA.  `cg_loads`
// reads values written by other CTAs of the same grid through L2.
static __device__ void compact_block(int B, int K, const int32_t *out_tokens, const int32_t *tau,
                              int32_t *offsets, int32_t *packed, int32_t *status, bool cg_loads,
                              int *red) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int carry = 0;
  constexpr int kPre = 16;  // rows this short are read along with their tau
  const bool pre_on = K + 1 <= kPre;
  for (int base = 0; base < B; base += blockDim.x) {
    const int b = base + threadIdx.x;
    int t = 0;
    int pre[kPre];
    if (b < B && pre_on) {
      const int32_t *src = out_tokens + (int64_t)b * (K + 1);
#pragma unroll
      for (int i = 0; i < kPre; ++i)
        if (i <= K) pre[i] = cg_loads ? __ldcg(src + i) : src[i];
    }
    if (b < B) {
      t = cg_loads ? __ldcg(tau + b) : tau[b];
      if (t < 0 || t > K + 1) {
        if (status) atomicOr(status, (int)SD_STATUS_BAD_TOKEN);
        t = 0;
      }
    }
    int x = t;  // inclusive warp scan
    __syncwarp();
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      x += lane >= o ? y : 0;
    }
    if (lane == 31) red[w] = x;
    __syncthreads();
    if (w == 0) {
      int v = lane < nw ? red[lane] : 0;
      __syncwarp();
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, v, o);
        v += lane >= o ? y : 0;
      }
      if (lane < nw) red[lane] = v;  // inclusive warp totals
    }
    __syncthreads();
    const int excl = carry + (w > 0 ? red[w - 1] : 0) + x - t;
    if (b < B) {
      offsets[b] = excl;
      if (pre_on) {
#pragma unroll
        for (int i = 0; i < kPre; ++i)
          if (i < t) packed[excl + i] = pre[i];
      } else {
        const int32_t *src = out_tokens + (int64_t)b * (K + 1);
        for (int i = 0; i < t; ++i) packed[excl + i] = cg_loads ? __ldcg(src + i) : src[i];
      }
    }
    carry += red[nw - 1];
    __syncthreads();
  }
  if (threadIdx.x == 0) offsets[B] = carry;
}


// ------------------------------------------------------------ streaming --
__device__ __forceinline__ uint64_t sub2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// Weights of the sampling pass for the elements of one target vector, two
// lanes per instruction: the residual Zt (p - q)+ =
// max(0, 2^(l s + Ct) - R 2^(l' s + Cd)) with R = Zt / Zd (r2 holds R, cd2
// Cd), or Zt p = 2^(l s + Ct) for a draw from p.  R is applied as a product
// rather than folded into the exponent, which would add the error of a
// hardware log2 to every draft weight.
template <typename E>
__device__ __forceinline__ void pass_weights(const uint4 &tv, const uint4 &dv, bool residual,
                                             uint64_t s2, uint64_t ct2, uint64_t cd2, uint64_t r2,
                                             float *w) {
  constexpr int N = Elt<E>::kPerVec;
  float ft[N], fd[N];
  Elt<E>::unpack(tv, ft);
  Elt<E>::unpack(dv, fd);
#pragma unroll
  for (int i = 0; i < N; i += 2) {
    float a, b;
    upk2(fma2(pk2(ft[i], ft[i + 1]), s2, ct2), a, b);
    uint64_t p = pk2(ex2(a), ex2(b));
    if (residual) {
      float c, d;
      upk2(fma2(pk2(fd[i], fd[i + 1]), s2, cd2), c, d);
      p = sub2(p, mul2(pk2(ex2(c), ex2(d)), r2));
    }
    upk2(p, w[i], w[i + 1]);
    if (residual) {
      w[i] = fmaxf(0.f, w[i]);
      w[i + 1] = fmaxf(0.f, w[i + 1]);
    }
  }
}

// Mass of one target vector in the sampling pass (sum of its weights).
template <typename E>
__device__ __forceinline__ float vec_mass(const uint4 &tv, const uint4 &dv, bool residual,
                                          uint64_t s2, uint64_t ct2, uint64_t cd2, uint64_t r2) {
  constexpr int N = Elt<E>::kPerVec;
  float w[N];
  pass_weights<E>(tv, dv, residual, s2, ct2, cd2, r2, w);
  uint64_t acc = pk2(w[0], w[1]);
#pragma unroll
  for (int i = 2; i < N; i += 2) acc = add2(acc, pk2(w[i], w[i + 1]));
  float lo, hi;
  upk2(acc, lo, hi);
  return lo + hi;
}

// Per-thread state of the row being streamed.
template <int KF>
struct RowAcc {
  static constexpr int KFm = KF > 0 ? KF : 1;
  float m;        // running max
  float c;        // exp offset: z = sum 2^(l s + c); +inf before the first finite value
  float z, zc;    // Kahan sum and compensation
  uint4 bv;       // first vector that reached the running max
  int bq;         // its slice vector index
  float kv[KFm];  // keys: this thread's best vectors by (masked max, index)
  int kq[KFm];
  float theta;    // keys: lower bound of the warp's KF-th best vector max
  __device__ __forceinline__ void reset() {
    m = -INFINITY;
    c = INFINITY;
    z = zc = 0.f;
    bq = -1;
    theta = -INFINITY;
#pragma unroll
    for (int k = 0; k < KFm; ++k) {
      kv[k] = -INFINITY;
      kq[k] = INT32_MAX;
    }
  }
};

// Sum of 2^(l s + c) over this thread's vectors of one step, two lanes per
// instruction; vectors k >= kv are skipped unless FULL.
template <typename E, bool FULL>
__device__ __forceinline__ float exp_sum(const uint4 (&v)[kU], int kv, uint64_t s2, uint64_t c2) {
  constexpr int N = Elt<E>::kPerVec;
  static_assert(kU == 4, "the combine below pairs four vectors");
  uint64_t acc[kU];
#pragma unroll
  for (int k = 0; k < kU; ++k) {
    acc[k] = 0ull;  // the pair (+0, +0)
    if (FULL || k < kv) {
      float f[N];
      Elt<E>::unpack(v[k], f);
#pragma unroll
      for (int i = 0; i < N; i += 2) {
        float a, b;
        upk2(fma2(pk2(f[i], f[i + 1]), s2, c2), a, b);
        const uint64_t e = pk2(ex2(a), ex2(b));
        acc[k] = i == 0 ? e : add2(acc[k], e);
      }
    }
  }
  float lo, hi;
  upk2(add2(add2(acc[0], acc[1]), add2(acc[2], acc[3])), lo, hi);
  return lo + hi;
}

template <typename E, bool FULL>
__device__ __forceinline__ float step_max(const uint4 (&v)[kU], int kv, float *vm) {
  float g = -INFINITY;
#pragma unroll
  for (int k = 0; k < kU; ++k) {
    vm[k] = (FULL || k < kv) ? Elt<E>::vmax(v[k]) : -INFINITY;
    g = fmaxf(g, vm[k]);
  }
  return g;
}

// What a row's stream computes (flags, uniform per row).
enum : int { kFExp = 1, kFArg = 2, kFKeys = 4, kFChk = 8 };

__device__ __forceinline__ int row_flags(int type, bool chk) {
  int f = chk ? kFChk : 0;
  if (type == kRowE || type == kRowEA || type == kRowEK) f |= kFExp;
  if (type == kRowEA || type == kRowA) f |= kFArg;
  if (type == kRowK || type == kRowEK) f |= kFKeys;
  return f;
}

__device__ __forceinline__ void st_shared16(uint32_t a, const uint4 &w) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(w.x), "r"(w.y), "r"(w.z),
               "r"(w.w)
               : "memory");
}

// Copy one step (kU vectors per thread) into the next ring slot.  Vectors
// wholly inside the piece are copied with cp.async; the ragged ends are
// assembled from element loads and past the piece the slot gets -inf, both
// stored by this thread, which alone reads its slots.
template <typename E, int NT>
__device__ __forceinline__ void issue_fill(Issuer &I, const Static &S, int nrows, uint32_t ring_t) {
  constexpr int kStepVec = NT * kU;
  constexpr uint32_t kSlot = kU * NT * 16;
  if (I.row < nrows) {
    if (I.step >= I.sf0 && I.step < I.sf1) {
#pragma unroll
      for (int k = 0; k < kU; ++k) cp_async16(I.slot + k * NT * 16, I.ptr + k * NT * 16);
    } else {
      const RowInfo &R = S.rows[I.row];
#pragma unroll 1
      for (int k = 0; k < kU; ++k) {
        const int q = I.step * kStepVec + k * NT + (int)threadIdx.x;
        if (q >= I.qlo && q < I.qhi) {
          cp_async16(I.slot + k * NT * 16, I.ptr + k * NT * 16);
        } else {
          const uint32_t ni = Elt<E>::kNegInfWord;
          const uint4 w = q < R.nvec ? load_vec_slow<E>(R, q, R.v0, R.v1) : make_uint4(ni, ni, ni, ni);
          st_shared16(I.slot + k * NT * 16, w);
        }
      }
    }
    I.ptr += kStepVec * 16;
    if (++I.step == I.nsteps) {
      ++I.row;
      issuer_row<NT>(I, S, nrows);
    }
  }
  cp_commit();
  I.slot += kSlot;
  if (I.slot == ring_t + kDepth * kSlot) I.slot = ring_t;
}

// One step of one row: kU whole vectors per thread (-inf padded).  kFExp:
// offset exp-sum; kFArg: running max and the first vector that reached it;
// kFKeys: the thread's best KF vectors by masked max; kFChk: NaN or +inf
// seen.  The running max is kept for every row but the exp-only ones (the
// finiteness check and the offset of the others use it).
template <typename E, int KF, int NT>
__device__ __forceinline__ void step_gen(RowAcc<KF> &A, const uint4 (&v)[kU], int step, int fl,
                                         int qd_step, int qd, int excl, int v0, int hp, float s,
                                         uint64_t s2, bool &bad) {
  constexpr int sz = Elt<E>::kSize, N = Elt<E>::kPerVec;
  const int qbase = step * (NT * kU) + threadIdx.x;
  float vm[kU];
  if (fl == kFExp) {
    // Exp-only rows: the offset comes from the first step that has a finite
    // value and moves only when a step's sum shows a far larger value (no
    // running max: nothing reads it for these rows).
    if (A.c == INFINITY) {
      const float g = step_max<E, true>(v, kU, vm);
      if (g > -INFINITY) A.c = -(g * s);
    }
    if (A.c != INFINITY) {
      float ss = exp_sum<E, true>(v, kU, s2, pk2(A.c, A.c));
      if (!(ss <= kBig)) {
        const float cn = -(step_max<E, true>(v, kU, vm) * s);
        if (cn < A.c) {
          const float f = ex2(cn - A.c);
          A.z *= f;
          A.zc *= f;
          A.c = cn;
        }
        ss = exp_sum<E, true>(v, kU, s2, pk2(A.c, A.c));
      }
      kahan_add(A.z, A.zc, ss);
    }
    return;
  }
  const float gmax = step_max<E, true>(v, kU, vm);
  if (fl & kFChk) {
#pragma unroll
    for (int k = 0; k < kU; ++k) bad |= !(Elt<E>::vmax_nan(v[k]) < INFINITY);
  }
  if (gmax > A.m) {
    A.m = gmax;
    if (fl & kFArg) {
      int kb = kU - 1;
#pragma unroll
      for (int k = kU - 1; k >= 0; --k)
        if (vm[k] == gmax) kb = k;
#pragma unroll
      for (int k = 0; k < kU; ++k)
        if (k == kb) {
          A.bv = v[k];
          A.bq = qbase + k * NT;
        }
    }
    if (fl & kFExp) {
      const float cn = -(gmax * s);
      if (A.c == INFINITY) {
        A.c = cn;
      } else if (A.c - cn > kRebase) {  // the max rose by more than kRebase (log2)
        const float f = ex2(cn - A.c);
        A.z *= f;
        A.zc *= f;
        A.c = cn;
      }
    }
  }
  if ((fl & kFExp) && A.c != INFINITY)
    kahan_add(A.z, A.zc, exp_sum<E, true>(v, kU, s2, pk2(A.c, A.c)));
  if constexpr (KF > 0) {
  if (fl & kFKeys) {
    // The top-KF elements of a set lie in its top-KF vectors ranked by
    // (max, index): every vector holding one of them has a max at least the
    // KF-th value, and at most KF vectors reach it.  Track those vectors.
    if (step == qd_step) {
#pragma unroll
      for (int k = 0; k < kU; ++k) {
        const int q = qbase + k * NT;
        if (q == qd) {  // the vector holding the excluded token: its max without it
          float f[N];
          Elt<E>::unpack(v[k], f);
          float mm = -INFINITY;
#pragma unroll
          for (int i = 0; i < N; ++i)
            if (elem_index(v0, hp, q, i, sz) != excl) mm = fmaxf(mm, f[i]);
          vm[k] = mm;
        }
      }
    }
    if (step == 0) {  // the warp's KF-th best first vector bounds the rest from below
      const int lane = threadIdx.x & 31;
      float x = vm[0], th = -INFINITY;
#pragma unroll
      for (int r = 0; r < KF; ++r) {
        th = rmax_f(x);
        const unsigned w = ballot(x == th);
        if (lane == __ffs(w) - 1) x = -INFINITY;
      }
      A.theta = th;
    }
    const float vbest = fmaxf(fmaxf(vm[0], vm[1]), fmaxf(vm[2], vm[3]));
    if (vbest > A.kv[KF - 1] && vbest >= A.theta) {  // rare once the row is under way
#pragma unroll
      for (int k = 0; k < kU; ++k) {
        if (vm[k] > A.kv[KF - 1] && vm[k] >= A.theta) {
          A.kv[KF - 1] = vm[k];
          A.kq[KF - 1] = qbase + k * NT;
#pragma unroll
          for (int x = KF - 1; x > 0; --x) {
            if (A.kv[x] > A.kv[x - 1]) {  // later vectors lose ties
              const float t1 = A.kv[x];
              A.kv[x] = A.kv[x - 1];
              A.kv[x - 1] = t1;
              const int t2 = A.kq[x];
              A.kq[x] = A.kq[x - 1];
              A.kq[x - 1] = t2;
            }
          }
        }
      }
    }
  }
  }
}

// End of a row piece: warp statistics into `ws` (a piece that failed the
// finiteness check gets a NaN sum), the warp's best KF key vectors into
// wsel[0..KF).
template <typename E, int KF>
__device__ __forceinline__ void row_end_gen(RowAcc<KF> &A, int fl, bool bad, int v0, int hp,
                                            WStat *ws, int *wsel) {
  constexpr int sz = Elt<E>::kSize, N = Elt<E>::kPerVec;
  constexpr int KFm = RowAcc<KF>::KFm;
  const int lane = threadIdx.x & 31;
  WStat st{-INFINITY, 0.f, INFINITY, INT32_MAX};
  const float mw = rmax_f(A.m);
  st.m = mw;
  if (fl & kFArg) {
    int idx = INT32_MAX;
    if (A.m == mw && mw > -INFINITY && A.bq >= 0) {
      float f[N];
      Elt<E>::unpack(A.bv, f);
#pragma unroll
      for (int i = N - 1; i >= 0; --i)
        if (f[i] == mw) idx = elem_index(v0, hp, A.bq, i, sz);
    }
    st.idx = rmin_i(idx);
  }
  if (fl & kFExp) {
    const bool has = A.z > 0.f;
    const float cw = rmin_f(has ? A.c : INFINITY);  // smallest offset: the largest max
    const float zt = has ? (A.z - A.zc) * ex2(cw - A.c) : 0.f;
    st.z = warp_sum(zt);
    st.c = cw;
  }
  if ((fl & kFChk) && ballot(bad) != 0u) st.z = __int_as_float(0x7fffffff);
  if (lane == 0) *ws = st;
  if (KF > 0 && (fl & kFKeys)) {
#pragma unroll
    for (int r = 0; r < KFm; ++r) {
      float bv = A.kv[0];
      int bq = A.kq[0];
      warp_best(bv, bq);
      if (bq != INT32_MAX && A.kq[0] == bq) {
#pragma unroll
        for (int x = 0; x < KFm - 1; ++x) {
          A.kv[x] = A.kv[x + 1];
          A.kq[x] = A.kq[x + 1];
        }
        A.kv[KFm - 1] = -INFINITY;
        A.kq[KFm - 1] = INT32_MAX;
      }
      if (lane == 0) wsel[r] = bv > -INFINITY ? bq : INT32_MAX;
    }
  }
  A.reset();
}

// The crossing point of a warp's values x (one per lane, in index order)
// for target t: the first lane with positive mass whose inclusive prefix
// exceeds t; if none (rounding put t at or past the total), the last lane
// with positive mass (crossed = 0); l = -1 when no lane has mass.  `before`
// is the prefix before lane l, `total` the warp's sum.  Whole warp.
struct Cross {
  int l, crossed;
  ff before, total;
};
static __device__ __noinline__ Cross ff_cross(ff x, ff t) {
  const ff incl = ff_warp_scan(x);
  const unsigned cross = ballot(ff_pos(x) && ff_gt(incl, t));
  const unsigned pos = ballot(ff_pos(x));
  Cross c;
  c.crossed = cross != 0u;
  c.l = cross ? __ffs(cross) - 1 : (pos ? 31 - __clz(pos) : -1);
  c.before = ff_shfl(ff_sub(incl, x), c.l < 0 ? 0 : c.l);
  if (c.l < 0) c.before = ff{0.f, 0.f};
  c.total = ff_shfl(incl, 31);
  return c;
}

constexpr int kFinCH = 8;  // draw iterations whose loads a warp keeps in flight together

// Weights pass of the draw over one warp's contiguous share [wq0, wq1) of
// this CTA's slice vectors: iteration it covers vectors wq0 + 32 it + lane.
// Writes the mass of each (iteration, lane) to pmw[it][lane] and returns the
// lane's total (Kahan-summed) as a float-float pair.  Whole vectors are read
// with all loads of a chunk in flight at once; the at most two ragged
// vectors of the slice are assembled afterwards, and a draft row off the
// target's vector grid takes the element-wise loop.
template <typename E>
__device__ __noinline__ ff draw_pass(const RowInfo &Rt, const RowInfo &Rd, const RowInfo &Rdt,
                                     bool residual, bool d_vec, int wq0, int wq1, int v0, int v1,
                                     uint64_t s2, uint64_t ct2, uint64_t cd2, uint64_t r2,
                                     float *pmw) {
  const int lane = threadIdx.x & 31;
  const int nit = (wq1 - wq0 + 31) / 32;
  const uint32_t ni = Elt<E>::kNegInfWord;
  float tsum = 0.f, tcomp = 0.f;
  if (residual && !d_vec) {
#pragma unroll 1
    for (int it = 0; it < nit; ++it) {
      const int q = wq0 + it * 32 + lane;
      float ms = 0.f;
      if (q < wq1)
        ms = vec_mass<E>(load_vec_direct<E>(Rt, q, v0, v1), load_vec_slow<E>(Rdt, q, v0, v1), true,
                         s2, ct2, cd2, r2);
      pmw[it * 32 + lane] = ms;
      kahan_add(tsum, tcomp, ms);
    }
    return two_sum(tsum, -tcomp);
  }
  const uint8_t *const tg = Rt.gbase;
  const uint8_t *const dg = residual ? Rd.gbase : Rt.gbase;
  const int tlo = Rt.qlo, thi = Rt.qhi;
#pragma unroll 1
  for (int it0 = 0; it0 < nit; it0 += kFinCH) {
    uint4 tv[kFinCH], dv[kFinCH];
#pragma unroll
    for (int c = 0; c < kFinCH; ++c) {
      const int q = wq0 + (it0 + c) * 32 + lane;
      tv[c] = dv[c] = make_uint4(ni, ni, ni, ni);
      if (q < wq1 && q >= tlo && q < thi) {
        tv[c] = __ldcg(reinterpret_cast<const uint4 *>(tg + 16 * q));
        if (residual) dv[c] = __ldcg(reinterpret_cast<const uint4 *>(dg + 16 * q));
      }
    }
#pragma unroll
    for (int c = 0; c < kFinCH; ++c) {
      if (it0 + c < nit) {
        const float ms = vec_mass<E>(tv[c], dv[c], residual, s2, ct2, cd2, r2);
        pmw[(it0 + c) * 32 + lane] = ms;
        kahan_add(tsum, tcomp, ms);
      }
    }
  }
  // the ragged vectors, by the lanes that own them: vector 0 when the slice
  // starts off the 16-byte grid (tlo = 1), the last when it ends off it
#pragma unroll 1
  for (int x = 0; x < 2; ++x) {
    const int q = x == 0 ? (tlo > 0 ? 0 : -1) : (thi < Rt.nvec ? Rt.nvec - 1 : -1);
    if (q < wq0 || q >= wq1 || (x == 1 && q == 0 && tlo > 0)) continue;
    if (((q - wq0) & 31) == lane) {
      const uint4 tvv = load_vec_slow<E>(Rt, q, v0, v1);
      const uint4 dvv = residual ? load_vec_slow<E>(Rd, q, v0, v1) : tvv;
      const float ms = vec_mass<E>(tvv, dvv, residual, s2, ct2, cd2, r2);
      pmw[((q - wq0) >> 5) * 32 + lane] = ms;
      kahan_add(tsum, tcomp, ms);
    }
  }
  return two_sum(tsum, -tcomp);
}

// The CTA's best KF elements (value desc, index asc) of key row R from the
// NW x KF vectors its warps kept, by one warp: the lanes expand the vectors
// into elements (without the excluded token, -inf and anything outside the
// slice), then KF rounds of a warp-wide best.  Lane 0 writes them to out[]
// as {value, index bits}; no candidate: {-inf, INT32_MAX}.
template <typename E, int KF, int NT>
__device__ __noinline__ void cta_keys(const RowInfo &R, const int *wsel, int v0, int v1,
                                      float2 *out) {
  constexpr int sz = Elt<E>::kSize, N = Elt<E>::kPerVec, NW = NT / 32;
  constexpr int NC = NW * KF;
  constexpr int PER = (NC + 31) / 32;
  const int lane = threadIdx.x & 31;
  float cv[PER * N];
  int ci[PER * N];
  uint4 x[PER];
  int qv[PER];
#pragma unroll
  for (int h = 0; h < PER; ++h) {
    const int c = lane + 32 * h;
    qv[h] = c < NC ? wsel[c] : INT32_MAX;
    if (qv[h] != INT32_MAX) x[h] = load_vec_direct<E>(R, qv[h], v0, v1);
  }
#pragma unroll
  for (int h = 0; h < PER; ++h) {
    float f[N];
    if (qv[h] != INT32_MAX) Elt<E>::unpack(x[h], f);
#pragma unroll
    for (int i = 0; i < N; ++i) {
      cv[h * N + i] = -INFINITY;
      ci[h * N + i] = INT32_MAX;
      if (qv[h] != INT32_MAX) {
        const int e = elem_index(v0, R.hp, qv[h], i, sz);
        if (e >= v0 && e < v1 && e != R.excl && f[i] > -INFINITY) {
          cv[h * N + i] = f[i];
          ci[h * N + i] = e;
        }
      }
    }
  }
#pragma unroll 1
  for (int r = 0; r < KF; ++r) {
    float bv = -INFINITY;
    int bi = INT32_MAX;
#pragma unroll
    for (int t = 0; t < PER * N; ++t)
      if (cv[t] > bv || (cv[t] == bv && ci[t] < bi)) {
        bv = cv[t];
        bi = ci[t];
      }
    warp_best(bv, bi);
#pragma unroll
    for (int t = 0; t < PER * N; ++t)
      if (bi != INT32_MAX && ci[t] == bi) {
        cv[t] = -INFINITY;
        ci[t] = INT32_MAX;
      }
    if (lane == 0) out[r] = make_float2(bi == INT32_MAX ? -INFINITY : bv, __int_as_float(bi));
  }
}

// ------------------------------------------------------------ the kernel --
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}
// A full cluster barrier (release / acquire) for code that every thread of
// every warp reaches together.  The .aligned form keeps each warp converged
// past the barrier; the unaligned form that cluster_group::sync() uses may
// release the threads of a warp separately, and the float-float shuffle code
// that follows it then ran several times slower.
__device__ __forceinline__ void cluster_sync_aligned() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" :::
               "memory");
}

// The sequence's outputs, by one warp: lane j writes token j, the lanes
// test the keys together.
static __device__ __forceinline__ void seq_outputs(const Params &P, const Static &S, int b,
                                                   bool tvalid) {
  const int lane = threadIdx.x & 31, K = P.K;
  int32_t *out = P.out_tokens + (int64_t)b * (K + 1);
  const bool valid = S.valid != 0;
  const int mm = valid ? S.m : -1, tok = S.tok;
  for (int j = lane; j <= K; j += 32) {
    const int v = !valid ? -1 : (j < mm ? S.d[j] : (j == mm ? tok : -1));
    out[j] = v;
  }
  bool h = false;
  if (valid && P.hit) {
    if (P.keys) {
      for (int k2 = lane; k2 < P.n_keys_out; k2 += 32)
        h |= S.keys[k2].x == mm && S.keys[k2].y == tok;
    } else if (P.keys_in) {
      const int32_t *kb = P.keys_in + (int64_t)b * P.n_keys_in * 2;
      for (int k2 = lane; k2 < P.n_keys_in; k2 += 32)
        h |= kb[2 * k2] == mm && kb[2 * k2 + 1] == tok;
    }
  }
  const bool hit = ballot(h) != 0u;
  if (lane == 0) {
    P.num_accepted[b] = valid ? mm : 0;
    P.tau[b] = valid ? mm + 1 : 0;
    if (P.hit) P.hit[b] = (uint8_t)(hit ? 1 : 0);
    if (!valid && P.status)
      atomicOr(P.status, (tvalid ? 0 : (int)SD_STATUS_BAD_TEMP) |
                             (S.dvalid ? 0 : (int)SD_STATUS_BAD_TOKEN) |
                             ((tvalid && S.dvalid && !S.fvalid) ? (int)SD_STATUS_NONFINITE : 0));
  }
}

template <typename E, int KF, int NT>
__global__ void __launch_bounds__(NT, 2) sd_seq_kernel(const __grid_constant__ Params P) {
  constexpr int sz = Elt<E>::kSize, NV = Elt<E>::kPerVec;
  constexpr int KFm = KF > 0 ? KF : 1;
  constexpr int NW = NT / 32;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int cs = P.cs;
  const int b = blockIdx.x / cs;
  const int K = P.K;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  __shared__ Static S;
  extern __shared__ __align__(128) uint8_t dyn[];

  // launched as a programmatic dependent of the stream's previous kernel:
  // nothing is read before that kernel has finished and its writes are
  // visible (the launch itself overlaps its tail)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // every CTA of the cluster has started before any pushes into its memory
  cluster_arrive_relaxed();

  const int v0 = min(rank * P.slice, P.V);
  const int v1 = min(v0 + P.slice, P.V);
  const bool verify = P.mode == kVerify;
  // both loads issued before anything waits on either
  const int d_pre = (warp == 0 && lane < K) ? P.tokens[(int64_t)b * K + (K - 1 - lane)] : -1;
  const float T = verify ? P.temps[b] : 0.f;
  const bool tvalid = !verify || ((T >= 0.f) && (T <= 3.4e38f));  // rejects NaN / inf / < 0
  const bool sampled = verify && tvalid && T > 0.f;
  // scaled logits x = l s with s = log2(e) / T rounded to float; every
  // exponential below uses this same s
  const float s = sampled ? log2e_over(T) : 0.f;
  const bool has_bonus = P.keys && P.bonus && P.fanout[K] > 0;

  // ---- the rows this CTA streams, in order: bonus, target K, then
  // (draft j, target j) for j = K-1..0.  Lane l of warp 0 places position
  // j = K-1-l; warp 1 the bonus row and target row K.
  float my_lt = -INFINITY, my_ld = -INFINITY;  // logits at d_j (lane j of warp 0)
  const int base = (has_bonus ? 1 : 0) + (verify ? 1 : 0);
  if (warp == 0) {
    const int l = lane, j = K - 1 - l;
    const bool act = l < K;
    const int fj = (act && P.keys) ? P.fanout[j] : 0;
    const bool dpres = act && (sampled || fj > 0);
    const unsigned dm = ballot(dpres);
    const int d = d_pre;
    if (act) S.d[j] = d;
    const bool dok = !act || (d >= 0 && d < P.V);
    const bool dvalid = __all_sync(0xffffffffu, dok);
    const int r_d = base + __popc(dm & ((1u << l) - 1u)) + (verify ? l : 0);
    const int r_t = r_d + (dpres ? 1 : 0);
    if (dpres) {
      RowInfo &R = S.rows[r_d];
      R.g = P.draft + ((int64_t)b * K + j) * P.V * sz;
      R.kind = kDraft;
      R.j = j;
      R.type = sampled ? (fj > 0 ? kRowEK : kRowE) : kRowK;
      R.excl = d;
      R.fan = fj;
      S.drow[j] = r_d;
    } else if (act) {
      S.drow[j] = -1;
    }
    if (act && verify) {
      RowInfo &R = S.rows[r_t];
      R.g = P.target + ((int64_t)b * (K + 1) + j) * P.V * sz;
      R.kind = kTarget;
      R.j = j;
      R.type = sampled ? (P.argmax_out ? kRowEA : kRowE) : kRowA;
      R.excl = -1;
      R.fan = 0;
      S.trow[j] = r_t;
    }
    if (act && sampled && dvalid) {
      my_lt = Elt<E>::load_global(P.target + (((int64_t)b * (K + 1) + j) * P.V + d) * sz);
      my_ld = Elt<E>::load_global(P.draft + (((int64_t)b * K + j) * P.V + d) * sz);
    }
    if (lane == 0) {
      S.nrows = base + __popc(dm) + (verify ? K : 0);
      S.dvalid = dvalid ? 1 : 0;
    }
    // the uniforms of the accept test at every position and of the draw at
    // every possible outcome position, ahead of the chain that uses them
    if (sampled)
      for (int q = lane; q <= K; q += 32) {
        if (q < K) S.u_acc[q] = uniform_u(P.seed, P.row_base + b, q, 0);
        S.u_draw[q] = uniform_u(P.seed, P.row_base + b, q, 1);
      }
  } else if (warp == 1 && lane < 2) {
    if (lane == 0 && has_bonus) {
      RowInfo &R = S.rows[0];
      R.g = P.bonus + (int64_t)b * P.V * sz;
      R.kind = kBonus;
      R.j = K;
      R.type = kRowK;
      R.excl = -1;
      R.fan = P.fanout[K];
      S.drow[K] = 0;
    } else if (lane == 0) {
      S.drow[K] = -1;
    }
    if (lane == 1 && verify) {
      RowInfo &R = S.rows[has_bonus ? 1 : 0];
      R.g = P.target + ((int64_t)b * (K + 1) + K) * P.V * sz;
      R.kind = kTarget;
      R.j = K;
      R.type = sampled ? (P.argmax_out ? kRowEA : kRowE) : kRowA;
      R.excl = -1;
      R.fan = 0;
      S.trow[K] = has_bonus ? 1 : 0;
    }
  }
  __syncthreads();

  const int nrows = S.nrows;
  // ---- the part of each row this CTA streams: either the vocabulary slice
  // [v0, v1) of every row, or an equal share of the sequence's rows laid end
  // to end in stream order, cut at whole streaming steps of a row (a few row
  // pieces per CTA instead of a piece of every row)
  if (tid < nrows) {
    RowInfo &R = S.rows[tid];
    if (P.rowsplit) {
      constexpr int ue = NT * kU * 16 / sz;  // elements per streaming step
      const int spr = (P.V + ue - 1) / ue;   // steps per row
      const int64_t U = (int64_t)nrows * spr;
      const int64_t u_lo = U * rank / cs, u_hi = U * (rank + 1) / cs;
      const int64_t r0 = (int64_t)tid * spr;
      const int64_t a = (u_lo > r0 ? u_lo : r0) - r0;
      const int64_t e = (u_hi < r0 + spr ? u_hi : r0 + spr) - r0;
      R.v0 = e > a ? (int)(a * ue) : 0;
      R.v1 = e > a ? (int)(e * ue < P.V ? e * ue : (int64_t)P.V) : 0;
    } else {
      R.v0 = v0;
      R.v1 = v1;
    }
    row_geometry<NT>(R, R.v0, R.v1, sz);
  }
  __syncthreads();
  const int npos = K + 1;
  const Layout L = make_layout(NT, nrows, npos, KF, cs, P.slice, sz);
  uint8_t *ring = dyn + L.ring;
  const uint32_t ring_t = smem_u32(ring) + tid * 16;
  WStat *wstat = reinterpret_cast<WStat *>(dyn + L.wstat);
  int *wsel = reinterpret_cast<int *>(dyn + L.wsel);
  CStat *cstat = reinterpret_cast<CStat *>(dyn + L.cstat);
  float2 *ckeys = reinterpret_cast<float2 *>(dyn + L.ckeys);  // .x value, .y index bits
  ff *cmass = reinterpret_cast<ff *>(dyn + L.cmass);
  float *pmass = reinterpret_cast<float *>(dyn + L.pmass);

  // ---- stream every row once: one row loop for every kind of row
  {
    Issuer I;
    I.row = 0;
    I.slot = ring_t;
    issuer_row<NT>(I, S, nrows);
#pragma unroll
    for (int d = 0; d < kDepth - 1; ++d) issue_fill<E, NT>(I, S, nrows, ring_t);
    uint32_t c_off = tid * 16;
    RowAcc<KF> A;
    A.reset();
    const bool chk = P.chk != 0;
    const uint64_t s2 = pk2(s, s);
    constexpr uint32_t kSlot = kU * NT * 16;
#pragma unroll 1
    for (int r = 0; r < nrows; ++r) {
      const RowInfo &R = S.rows[r];
      WStat *ws = &wstat[r * NW + warp];
      int *wk = &wsel[(R.j * NW + warp) * KFm];
      const int fl = row_flags(R.type, chk);
      if (R.nsteps == 0) {  // this CTA holds none of the row
        if (lane == 0) *ws = WStat{-INFINITY, 0.f, INFINITY, INT32_MAX};
        if (KF > 0 && (fl & kFKeys) && lane < KFm) wk[lane] = INT32_MAX;
        continue;
      }
      const int nsteps = R.nsteps, qd_step = R.qd_step, qd = R.qd, excl = R.excl;
      const int rv0 = R.v0, hp = R.hp;
      bool bad = false;
#pragma unroll 1
      for (int step = 0; step < nsteps; ++step) {
        issue_fill<E, NT>(I, S, nrows, ring_t);
        cp_wait<kDepth - 1>();  // this step's copies have landed
        const uint8_t *src = ring + c_off;
        uint4 v[kU];
#pragma unroll
        for (int k = 0; k < kU; ++k) v[k] = *reinterpret_cast<const uint4 *>(src + k * NT * 16);
        step_gen<E, KF, NT>(A, v, step, fl, qd_step, qd, excl, rv0, hp, s, s2, bad);
        c_off += kSlot;
        if (c_off >= kDepth * kSlot) c_off -= kDepth * kSlot;
      }
      row_end_gen<E, KF>(A, fl, bad, rv0, hp, ws, wk);
    }
    cp_wait<0>();
  }
  // the packing launch that follows may be scheduled from here on
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (warp == 0 && lane < K) {
    S.ld_t[lane] = my_lt;  // lane l holds position K-1-l
    S.ld_d[lane] = my_ld;
  }
  __syncthreads();

  // ---- CTA statistics per row (thread per row), pushed into every CTA (a
  // warp with a NaN sum, from the finiteness check, makes the sum NaN)
  cluster_wait();  // pairs with the arrive at the top
  if (tid < nrows) {
    const int r = tid;
    float M = -INFINITY;
    bool poison = false;
#pragma unroll 1
    for (int w = 0; w < NW; ++w) M = fmaxf(M, wstat[r * NW + w].m);
    int I = INT32_MAX;
    float C = INFINITY;
#pragma unroll 1
    for (int w = 0; w < NW; ++w) {
      const WStat x = wstat[r * NW + w];
      if (x.m == M) I = min(I, x.idx);
      if (x.z > 0.f) C = fminf(C, x.c);
      poison |= x.z != x.z;
    }
    ff Z{0.f, 0.f};
#pragma unroll 1
    for (int w = 0; w < NW; ++w) {
      const WStat x = wstat[r * NW + w];
      if (x.z > 0.f) Z = ff_add(Z, two_prod(x.z, ex2(C - x.c)));
    }
    if (poison) Z.hi = __int_as_float(0x7fffffff);
    CStat cst;
    cst.m = M;
    cst.idx = I;
    cst.c = C;
    cst.zhi = Z.hi;
    cst.zlo = Z.lo;
#pragma unroll 1
    for (int p = 0; p < cs; ++p) *cluster.map_shared_rank(&cstat[rank * nrows + r], p) = cst;
  }
  if (KF > 0) {
    for (int r = warp; r < nrows; r += NW) {
      const RowInfo &R = S.rows[r];
      if (!(R.type == kRowK || R.type == kRowEK)) continue;
      // the CTA's keys staged in the idle ring, then pushed to every CTA
      float2 *stage = reinterpret_cast<float2 *>(ring) + R.j * KFm;
      if (R.nsteps > 0) {
        cta_keys<E, KFm, NT>(R, &wsel[R.j * NW * KFm], R.v0, R.v1, stage);
      } else if (lane < KFm) {
        stage[lane] = make_float2(-INFINITY, __int_as_float(INT32_MAX));
      }
      __syncwarp();
#pragma unroll 1
      for (int x = lane; x < KFm * cs; x += 32)
        *cluster.map_shared_rank(&ckeys[(rank * npos + R.j) * KFm + x % KFm], x / KFm) =
            stage[x % KFm];
    }
  }
  cluster_sync_aligned();  // (1) every CTA's statistics are in every CTA

  // ---- combine the cluster's statistics (same arithmetic in every CTA)
  if (tid == 0) S.fvalid = 1;
  __syncthreads();
  if (tid < nrows) {
    const int r = tid;
    float M = -INFINITY;
#pragma unroll 1
    for (int p = 0; p < cs; ++p) M = fmaxf(M, cstat[p * nrows + r].m);
    int I = INT32_MAX;
    float C = INFINITY;
#pragma unroll 1
    for (int p = 0; p < cs; ++p) {
      const CStat &x = cstat[p * nrows + r];
      if (x.m == M) I = min(I, x.idx);
      if (x.zhi > 0.f) C = fminf(C, x.c);
    }
    ff Z{0.f, 0.f};
    bool poison = false;
#pragma unroll 1
    for (int p = 0; p < cs; ++p) {
      const CStat &x = cstat[p * nrows + r];
      if (x.zhi > 0.f) Z = ff_add(Z, ff_mul_f(ff{x.zhi, x.zlo}, ex2(C - x.c)));
      poison |= x.zhi != x.zhi;
    }
    S.M[r] = M;
    S.C[r] = C;
    S.Z[r] = Z;
    S.amax[r] = I == INT32_MAX ? 0 : I;
    if (P.chk && (poison || !(M > -INFINITY))) S.fvalid = 0;
  }
  if (KF > 0 && P.keys) {
    // keys of each position: the best fan of the cs x KF CTA candidates
    for (int j = warp; j <= K; j += NW) {
      const int fan = P.fanout[j];
      if (fan <= 0) continue;
      int2 *kdst = &S.keys[P.fan_off[j]];
      int32_t *kout = P.keys_out ? P.keys_out + ((int64_t)b * P.n_keys_out + P.fan_off[j]) * 2
                                 : nullptr;
      const bool present = S.drow[j] >= 0;
      constexpr int PER = (kMaxCS * KFm + 31) / 32;
      float cv[PER];
      int ci[PER];
#pragma unroll
      for (int h = 0; h < PER; ++h) {
        const int c = lane + 32 * h;  // candidate c: CTA c / KF, rank c % KF
        cv[h] = -INFINITY;
        ci[h] = INT32_MAX;
        if (present && c < cs * KFm) {
          const float2 e = ckeys[((c / KFm) * npos + j) * KFm + c % KFm];
          cv[h] = e.x;
          ci[h] = __float_as_int(e.y);
        }
      }
      for (int r2 = 0; r2 < fan; ++r2) {
        float bv = -INFINITY;
        int bi = INT32_MAX;
#pragma unroll
        for (int h = 0; h < PER; ++h)
          if (cv[h] > bv || (cv[h] == bv && ci[h] < bi)) {
            bv = cv[h];
            bi = ci[h];
          }
        warp_best(bv, bi);
#pragma unroll
        for (int h = 0; h < PER; ++h)
          if (bi != INT32_MAX && ci[h] == bi) {
            cv[h] = -INFINITY;
            ci[h] = INT32_MAX;
          }
        if (lane == 0) {
          const int2 key = bi == INT32_MAX ? make_int2(-1, -1) : make_int2(j, bi);
          kdst[r2] = key;
          if (rank == 0 && kout) {
            kout[2 * r2] = key.x;
            kout[2 * r2 + 1] = key.y;
          }
        }
      }
    }
  }
  __syncthreads();

  if (verify) {
    // ---- accept tests, one lane per position (K <= 32: warp 0)
    if (warp == 0) {
      const int j = lane;
      const bool dvalid = S.dvalid != 0;
      int rej = 0;
      if (j < K) {
        const int rt = S.trow[j];
        const int d = S.d[j];
        int a = 0;
        if (!sampled) {
          a = (dvalid && d == S.amax[rt]) ? 1 : 0;
        } else if (dvalid) {
          const int rd = S.drow[j];
          const float lt = S.ld_t[K - 1 - j], ldr = S.ld_d[K - 1 - j];
          // log2 of 2^(l_d s + C), carried as float-float (the products exact)
          const ff xt = ff_add_f(two_prod(lt, s), S.C[rt]);
          const ff xd = ff_add_f(two_prod(ldr, s), S.C[rd]);
          const float zt = ff_f(S.Z[rt]), zd = ff_f(S.Z[rd]);
          const float r = (ldr == -INFINITY)
                              ? INFINITY  // q(d) = 0
                              : exp2_ff(ff_sub(xt, xd)) * ff_ratio(S.Z[rd], S.Z[rt]);
          const float u = S.u_acc[j];
          a = (u <= r) ? 1 : 0;
          if (rank == 0) {
            const int64_t pj = (int64_t)b * K + j;
            if (P.ratio_out) P.ratio_out[pj] = r;
            if (P.p_out) P.p_out[pj] = __fdiv_rn(exp2_ff(xt), zt);
            if (P.q_out) P.q_out[pj] = __fdiv_rn(exp2_ff(xd), zd);
          }
        }
        rej = !a;
      }
      const unsigned rejects = ballot(rej);
      if (sampled && tvalid && dvalid && S.fvalid && lane < 2) {  // the rows the draw reads
        const int mm = rejects ? __ffs(rejects) - 1 : K;
        if (lane == 0) {
          S.dt = S.rows[S.trow[mm]];
          row_geometry<NT>(S.dt, v0, v1, sz);
        } else if (mm < K) {
          S.dd = S.rows[S.drow[mm]];
          row_geometry<NT>(S.dd, v0, v1, sz);
        }
      }
      if (lane == 0) {
        const int mm = rejects ? __ffs(rejects) - 1 : K;
        S.m = mm;
        S.valid = (tvalid && dvalid && S.fvalid) ? 1 : 0;
        S.kind = 0;
        S.owner = 0;
        S.tok = -1;
        S.cstar = 0;
        if (S.valid) {
          if (!sampled) S.tok = S.amax[S.trow[mm]];
          else S.kind = mm < K ? 1 : 2;
        }
      }
    }
    if (rank == 0 && P.argmax_out)
      for (int j = tid; j <= K; j += NT) P.argmax_out[(int64_t)b * (K + 1) + j] = S.amax[S.trow[j]];
    __syncthreads();

    // ---- one inverse-CDF draw per sequence (residual at m, or p at K).
    // Each warp takes a contiguous range of the slice and lane l the two
    // consecutive vectors 2l, 2l+1 of each 64-vector step, so the masses kept
    // per (step, lane) are in index order.  The CTA holding the crossing
    // point finds its warp, step and lane from those masses, and that lane
    // re-reads only its two vectors.
    for (int attempt = 0; attempt < 2 && S.kind != 0; ++attempt) {
      const int mm = S.m;
      const bool residual = S.kind == 1;
      const RowInfo &Rt = S.dt;
      const RowInfo *Rd = residual ? &S.dd : nullptr;
      const bool d_vec = residual && Rd->hp == Rt.hp;  // same vector grid
      RowInfo Rdt;  // otherwise: the draft row read element-wise on the target's grid
      if (residual && !d_vec) {
        Rdt = Rt;
        Rdt.g = Rd->g;
        Rdt.qlo = 1;
        Rdt.qhi = 0;
      }
      const float Ct = S.C[S.trow[mm]];
      const float Cd = residual ? S.C[S.drow[mm]] : 0.f;
      const float Rz = residual ? ff_ratio(S.Z[S.trow[mm]], S.Z[S.drow[mm]]) : 0.f;
      const uint64_t s2 = pk2(s, s), ct2 = pk2(Ct, Ct);
      const uint64_t cd2 = pk2(Cd, Cd), r2 = pk2(Rz, Rz);  // draft weights times R
      const int wr = (Rt.nvec + NW - 1) / NW;  // vectors per warp
      const int wq0 = min(warp * wr, Rt.nvec), wq1 = min(wq0 + wr, Rt.nvec);
      const int wsteps = (wq1 - wq0 + 2 * 32 - 1) / (2 * 32);
      float *pmw = pmass + warp * L.pw * 32;  // [step][lane] masses of this warp
      {
        constexpr uint32_t kSlot = kU * NT * 16;
        // step u: target vectors into ring vectors 0, 1; draft into 2, 3.  The
        // rows' fields are kept in registers: the copy instructions clobber
        // memory, so fields read through a reference would be reloaded.
        const uint8_t *const tg = Rt.gbase;
        const uint8_t *const dg = d_vec ? Rd->gbase : Rt.gbase;
        const int tlo = max(Rt.qlo, wq0), thi = min(Rt.qhi, wq1);  // vectors copied whole
        int i_u = 0;
        auto issue_pass = [&](int slot) {
          if (i_u < wsteps) {
            const int qa = wq0 + i_u * 64 + 2 * lane;
            const uint32_t sl = ring_t + slot * kSlot;
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              const int q = qa + k;
              if (q >= tlo && q < thi) {
                cp_async16(sl + k * NT * 16, tg + 16 * q);
                if (d_vec) cp_async16(sl + (2 + k) * NT * 16, dg + 16 * q);
              }
            }
            ++i_u;
          }
          cp_commit();
        };
#pragma unroll 1
        for (int d = 0; d < kDepth - 1; ++d) issue_pass(d);
        float tsum = 0.f, tcomp = 0.f;
#pragma unroll 1
        for (int u = 0; u < wsteps; ++u) {
          issue_pass((u + kDepth - 1) % kDepth);
          cp_wait<kDepth - 1>();
          const uint8_t *slot = ring + (u % kDepth) * kSlot + tid * 16;
          float ms = 0.f;
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const int q = wq0 + u * 64 + 2 * lane + k;
            if (q < wq1) {
              uint4 tv, dv;
              if (q >= tlo && q < thi) {
                tv = *reinterpret_cast<const uint4 *>(slot + k * NT * 16);
                dv = d_vec ? *reinterpret_cast<const uint4 *>(slot + (2 + k) * NT * 16) : tv;
              } else {
                tv = load_vec_slow<E>(Rt, q, v0, v1);
                dv = d_vec ? load_vec_slow<E>(*Rd, q, v0, v1) : tv;
              }
              if (residual && !d_vec) dv = load_vec_slow<E>(Rdt, q, v0, v1);
              ms += vec_mass<E>(tv, dv, residual, s2, ct2, cd2, r2);
            }
          }
          pmw[u * 32 + lane] = ms;
          kahan_add(tsum, tcomp, ms);
        }
        cp_wait<0>();
        const ff wm = ff_warp_sum(two_sum(tsum, -tcomp));
        if (lane == 0) S.wmass[warp] = wm;
      }
      __syncthreads();
      if (warp == 0) {
        // prefix over the warps, the CTA mass pushed into every CTA
        const ff m_l = lane < NW ? S.wmass[lane] : ff{0.f, 0.f};
        const ff incl = ff_warp_scan(m_l);
        if (lane < NW) S.wpre[lane] = ff_sub(incl, m_l);
        const ff tot_cta = ff_shfl(incl, 31);
        if (lane < cs) *cluster.map_shared_rank(&cmass[attempt * cs + rank], lane) = tot_cta;
      }
      cluster_sync_aligned();  // (2) slice masses are in every CTA
      if (warp == 0) {
        const ff sc = lane < cs ? cmass[attempt * cs + lane] : ff{0.f, 0.f};  // lane c: CTA c
        const ff incl = ff_warp_scan(sc);
        const ff tot = ff_shfl(incl, 31);
        if (ff_pos(tot) || !residual) {
          const float u = S.u_draw[mm];
          const ff t = ff_mul_f(tot, u);
          const unsigned cross = ballot(ff_pos(sc) && ff_gt(incl, t));
          const unsigned pos = ballot(ff_pos(sc));
          // the first CTA whose range passes t; if rounding put t past the
          // total, the last CTA with mass
          const int cstar = cross ? __ffs(cross) - 1 : (pos ? 31 - __clz(pos) : 0);
          const ff before = ff_shfl(ff_sub(incl, sc), cstar);
          if (lane == 0) {
            S.cstar = cstar;
            S.t_loc = ff_sub(t, before);
            S.owner = cstar;
          }
        } else if (lane == 0) {
          S.kind = 2;  // identically zero residual: draw from p at m
        }
      }
      __syncthreads();
      if (S.kind == 2 && residual) continue;  // every CTA takes this branch
      if (rank == S.cstar) {
        if (warp == 0) {
          // the crossing warp: the first whose range passes t_loc, else the
          // last with mass
          const ff m_l = lane < NW ? S.wmass[lane] : ff{0.f, 0.f};
          const ff pre = lane < NW ? S.wpre[lane] : ff{0.f, 0.f};
          const unsigned cross =
              ballot(ff_pos(m_l) && ff_gt(ff_add(pre, m_l), S.t_loc));
          const unsigned pos = ballot(ff_pos(m_l));
          const int ws = cross ? __ffs(cross) - 1 : (pos ? 31 - __clz(pos) : 0);
          if (lane == 0) {
            S.wsel = ws;
            S.t_w = ff_sub(S.t_loc, S.wpre[ws]);
          }
        }
        __syncthreads();
        if (warp == S.wsel) {
          const ff tw = S.t_w;
          // the crossing step: step masses (lane t sums row t of the warp's
          // [step][lane] masses, reading it rotated across the banks)
          int tsel = -1, tlast = -1;
          ff before{0.f, 0.f}, before_last{0.f, 0.f}, cum{0.f, 0.f};
#pragma unroll 1
          for (int tb = 0; tb < wsteps && tsel < 0; tb += 32) {
            const int t = tb + lane;
            ff mt{0.f, 0.f};
            if (t < wsteps) {  // pairwise: five dependent levels instead of 32
              ff v[16];
#pragma unroll
              for (int i = 0; i < 16; ++i)
                v[i] = two_sum(pmw[t * 32 + ((2 * i + lane) & 31)],
                               pmw[t * 32 + ((2 * i + 1 + lane) & 31)]);
#pragma unroll
              for (int w2 = 8; w2 > 0; w2 >>= 1)
#pragma unroll
                for (int i = 0; i < w2; ++i) v[i] = ff_add(v[i], v[i + w2]);
              mt = v[0];
            }
            const ff incl = ff_warp_scan(mt);
            const unsigned cross =
                ballot(ff_pos(mt) && ff_gt(ff_add(cum, incl), tw));
            const unsigned pos = ballot(ff_pos(mt));
            if (cross) {
              const int l = __ffs(cross) - 1;
              tsel = tb + l;
              before = ff_add(cum, ff_shfl(ff_sub(incl, mt), l));
            } else if (pos) {
              const int l = 31 - __clz(pos);
              tlast = tb + l;
              before_last = ff_add(cum, ff_shfl(ff_sub(incl, mt), l));
            }
            cum = ff_add(cum, ff_shfl(incl, 31));
          }
          if (tsel < 0) {  // rounding put the target past the warp's mass
            tsel = tlast;
            before = before_last;
          }
          // the crossing lane within that step
          int lsel = -1;
          ff before_l{0.f, 0.f};
          if (tsel >= 0) {
            const float ml = pmw[tsel * 32 + lane];
            const ff incl = ff_warp_scan(ff{ml, 0.f});
            const unsigned cross =
                ballot(ml > 0.f && ff_gt(ff_add(before, incl), tw));
            const unsigned pos = ballot(ml > 0.f);
            lsel = cross ? __ffs(cross) - 1 : (pos ? 31 - __clz(pos) : -1);
            if (lsel >= 0) before_l = ff_add(before, ff_shfl(ff_add_f(incl, -ml), lsel));
          }
          if (lsel >= 0) {
            // the crossing lane's two vectors, one element per lane (lane
            // k NV + i: element i of vector k, i.e. index order), a scan of
            // the weights from before_l, the first element past tw; if
            // rounding leaves none, the last element with weight
            const int k = lane / NV, i = lane % NV;
            const int q = wq0 + tsel * 64 + 2 * lsel + k;
            float w = 0.f;
            int e = -1;
            if (lane < 2 * NV && q < wq1) {
              const uint4 tvv = load_vec_direct<E>(Rt, q, v0, v1);
              uint4 dvv = tvv;
              if (residual)
                dvv = d_vec ? load_vec_direct<E>(*Rd, q, v0, v1) : load_vec_slow<E>(Rdt, q, v0, v1);
              float ww[NV];
              pass_weights<E>(tvv, dvv, residual, s2, ct2, cd2, r2, ww);
              float wi = 0.f;
#pragma unroll
              for (int ii = 0; ii < NV; ++ii)
                if (ii == i) wi = ww[ii];
              const int ei = elem_index(v0, Rt.hp, q, i, sz);
              if (ei >= v0 && ei < v1 && wi > 0.f) {
                w = wi;
                e = ei;
              }
            }
            const ff cw = ff_add(before_l, ff_warp_scan(ff{w, 0.f}));
            const unsigned cross = ballot(e >= 0 && ff_gt(cw, tw));
            const unsigned pos = ballot(e >= 0);
            const int ls = cross ? __ffs(cross) - 1 : (pos ? 31 - __clz(pos) : 0);
            const int tok = __shfl_sync(0xffffffffu, e, ls);
            if (lane == 0) S.tok = tok >= 0 ? tok : S.amax[S.trow[mm]];
          }
          if (lsel < 0 && lane == 0) S.tok = S.amax[S.trow[mm]];  // no mass in this warp
        }
        __syncthreads();
      }
      break;
    }

    // ---- the sequence's outputs (owning CTA, one warp)
    if (rank == S.owner && warp == 0) seq_outputs(P, S, b, tvalid);
  }
  // No CTA touches another's shared memory after barrier (1) or (2), which
  // every CTA passes, so the CTAs may leave independently.
}


// The packing step launched right behind the verify kernel as its
// programmatic dependent: it may become resident early and waits here until
// every verify CTA has finished and its writes are visible.
static __global__ void __launch_bounds__(1024) sd_compact_after_kernel(
    int B, int K, const int32_t *out_tokens, const int32_t *tau, int32_t *offsets,
    int32_t *packed, int32_t *status) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  __shared__ int red[32];
  compact_block(B, K, out_tokens, tau, offsets, packed, status, false, red);
}

// ------------------------------------------------------------------- host --
static int env_int(const char *name, int dflt) {
  const char *s = getenv(name);
  return s && *s ? atoi(s) : dflt;
}

// Host-side state is kept per device: a process may drive several GPUs, and
// SM counts, kernel attributes and occupancy answers belong to one of them.
// An NVTX range named after the C-ABI entry point, open while the call does
// its host work and enqueues its launches (a profiler shows each call's
// launches under its name).  Header-only NVTX: without a tool attached a
// push or pop is a call through an empty slot.
struct NvtxRange {
  explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange &) = delete;
  NvtxRange &operator=(const NvtxRange &) = delete;
};

constexpr int kMaxDevices = 64;

static int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    dev = 0;
  }
  return dev;
}

static int sm_count() {
  static int n[kMaxDevices];
  const int dev = current_device();
  if (n[dev] <= 0) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    n[dev] = v > 0 ? v : 1;
  }
  return n[dev];
}

// Sets a kernel's dynamic shared-memory limit (and, for cluster kernels, the
// non-portable cluster sizes) once on each device it is launched on.
struct FuncAttrs {
  std::mutex mu;
  bool done[kMaxDevices] = {};
  void apply(const void *fn, int smem_cap, bool clusters, const char *what) {
    const int dev = current_device();
    std::lock_guard<std::mutex> g(mu);
    if (done[dev]) return;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_cap) !=
        cudaSuccess)
      fprintf(stderr, "sd_verify: shared-memory limit of %s not set: %s\n", what,
              cudaGetErrorString(cudaGetLastError()));
    if (clusters &&
        cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
      cudaGetLastError();
    done[dev] = true;
  }
};

static const int kDynSmemCap = 227 * 1024 - (int)sizeof(Static) - 256;

template <typename E, int KF, int NT>
static void *kernel_fn() {
  static FuncAttrs attrs;
  void *fn = (void *)sd_seq_kernel<E, KF, NT>;
  attrs.apply(fn, kDynSmemCap, true, "the cluster kernel");
  return fn;
}

// Rows streamed per sequence (upper bound used for the shared-memory size).
static int rows_per_seq(const Params &P) {
  int n = P.mode == kVerify ? 2 * P.K + 1 : P.K;
  if (P.keys && P.bonus && P.fanout[P.K] > 0) n += 1;
  return std::max(n, 1);
}

// The packing of all sequences' tokens, as a programmatic dependent of the
// verify launch just issued on the same stream.
static sd_status_t launch_compact_after(const Params &P, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1, 1, 1);
  cfg.blockDim = dim3(1024, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, sd_compact_after_kernel, (int)P.B, (int)P.K,
                                           (const int32_t *)P.out_tokens, (const int32_t *)P.tau,
                                           P.offsets, P.packed, P.status);
  if (e != cudaSuccess) {
    fprintf(stderr, "sd_verify packing launch failed: %s\n", cudaGetErrorString(e));
    return SD_ERR_CUDA;
  }
  return SD_OK;
}
// Vocabulary slice of one CTA for cluster size cs (a multiple of 16 elements).
// Whole streaming steps (NT kU vectors) per slice where that still leaves
// every CTA some vocabulary, so only the last CTA of a cluster meets a
// partial step; otherwise a multiple of 16 elements.
static int slice_for(int V, int cs, int sz, int NT) {
  const int64_t even = ((int64_t)V + cs - 1) / cs;
  const int64_t step = (int64_t)NT * kU * 16 / sz;
  const int64_t whole = (even + step - 1) / step * step;
  if ((cs - 1) * whole < V) return (int)whole;
  return (int)((even + 15) / 16 * 16);
}

template <typename E, int KF, int NT>
static int smem_bytes(const Params &P, int cs) {
  return make_layout(NT, rows_per_seq(P), P.K + 1, KF, cs, slice_for(P.V, cs, Elt<E>::kSize, NT),
                     Elt<E>::kSize)
      .total;
}

// Clusters of cs CTAs with `smem` bytes each that the device holds at once.
template <typename E, int KF, int NT>
static int max_active_clusters(int cs, int smem) {
  static std::mutex mu;
  static int cache[kMaxDevices][kMaxCS + 1][8];
  static int cache_smem[kMaxDevices][kMaxCS + 1][8];
  const int dev = current_device();
  void *fn = kernel_fn<E, KF, NT>();
  std::lock_guard<std::mutex> g(mu);
  const int slot = (smem / 1024) % 8;
  if (cache_smem[dev][cs][slot] == smem + 1) return cache[dev][cs][slot];
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)cs, 1, 1);
  cfg.blockDim = dim3(NT, 1, 1);
  cfg.dynamicSmemBytes = (size_t)smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  cache[dev][cs][slot] = n;
  cache_smem[dev][cs][slot] = smem + 1;
  return n;
}

// Cluster size: the largest cs up to about SDV_CPS (default 2) CTAs per SM
// for which all B clusters are resident at once (one wave); if none is,
// the size that leaves the fewest waves.
template <typename E, int KF, int NT>
static int choose_cs(const Params &P) {
  const int forced = env_int("SDV_CS", 0);
  if (forced) return forced;
  const int per_sm = std::max(1, env_int("SDV_CPS", 2));
  const int B = std::max(P.B, 1);
  const int target = (int)std::min<int64_t>(
      kMaxCS, std::max<int64_t>(1, (int64_t)per_sm * sm_count() / B));
  int best = -1;
  int64_t best_waves = INT64_MAX;
  for (int cs = target; cs >= 1; --cs) {
    const int smem = smem_bytes<E, KF, NT>(P, cs);
    if (smem > kDynSmemCap) break;
    const int n = max_active_clusters<E, KF, NT>(cs, smem);
    if (n <= 0) continue;
    if (n >= B) return cs;
    const int64_t waves = (B + n - 1) / n;
    if (waves < best_waves) {
      best_waves = waves;
      best = cs;
    }
  }
  if (best > 0) return best;
  for (int cs = target; cs <= kMaxCS; ++cs)
    if (smem_bytes<E, KF, NT>(P, cs) <= kDynSmemCap) return cs;
  return kMaxCS;
}


// The split launch (sd_split.cu): SD_ERR_UNSUPPORTED when the request does
// not fit its limits, before anything is launched.
size_t split_workspace_bytes(int64_t B, int K);
template <typename E, int KF>
sd_status_t launch_split(Params &P, size_t ws_bytes, cudaStream_t stream);

}  // namespace sdv
