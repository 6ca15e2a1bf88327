// GB300 (sm_103a) kernels of the speculative-decoding verify step.
//
// Layout of the work: one thread-block cluster per sequence (row b of the
// batch).  The cluster's CTAs split the vocabulary into contiguous slices;
// each CTA streams its slice of every logit row of the sequence -- target
// rows K..0 and draft rows K-1..0, plus the optional draft row of the bonus
// position.  Each thread copies its own 16-byte vectors a few steps ahead
// into its own shared-memory slots (cp.async, so no block-wide barrier is
// needed while streaming) and keeps only per-row statistics in registers:
// max, lowest-index argmax, the sum of 2^(l s + c) (s = log2(e) / T, c a
// per-thread offset carried exactly into the combine) and, for draft rows,
// the few vectors that can hold the top-F keys.  One exchange over
// distributed shared memory gives every CTA the statistics of all K+1
// positions, so each CTA evaluates the left-to-right accept scan itself and
// all of them agree on the first rejection m.  Only then is a single
// inverse-CDF draw needed per sequence: over the residual max(0, p - q) at m,
// or over p at the bonus position K.  The CTAs re-read their slices of those
// one or two rows (rows are streamed in the order K..0, so the likely m ~ 0
// rows were read last and are still in L2), exchange slice masses, and the
// CTA holding the crossing point scans it.  The owning CTA writes the
// sequence's tokens and tau, and the last sequence to finish (one atomic
// counter) packs all sequences' tokens.  Nothing waits on another cluster
// and there are no spin-waits.
//
// Method sources (web pages, stated in prose there):
//  "What is speculative decoding" explainer (lotook.com): the four-stage loop
//    (greedy match; keep a token the target rates at least as high as the
//    draft, else keep it with the probability ratio; resample the first
//    rejection from a residual of both distributions; bonus token at K+1).
//  "Speculative Speculative Decoding" blog (jiwasawa.github.io), "Saguaro
//    1. Outcome Prediction": keys from the draft logits' top tokens with a
//    fan-out per position.
//  "LLMの生成を5倍速くする「D3D」を図で読む" (animemo.app), 検証のしくみ③,
//    検証のまとめ, ヒット / ミス: greedy worked example, tau, hit test.
// Readings where the pages are silent are listed in include/sd_verify.h.

#include "sd_verify.h"

#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

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
constexpr int kMaxSliceVec = 4096;           // vectors in one row slice
constexpr float kRebase = 16.f;              // log2 headroom of the exp offset

enum Mode : int { kVerify = 0, kPredict = 1 };
enum RowKind : int { kTarget = 0, kDraft = 1, kBonus = 2 };
enum RowFlag : int { kNeedExp = 1, kNeedArg = 2, kNeedKeys = 4 };

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
  int32_t *done_counter;   // workspace
  uint64_t seed;
  int64_t row_base;
  int32_t B, K, V;
  int32_t mode;
  int32_t keys;            // build keys in this pass
  int32_t compact;
  int32_t n_keys_in, n_keys_out;
  int32_t cs, slice;       // cluster size, vocabulary slice per CTA
  int32_t fanout[SD_MAX_K + 1];
  int32_t fan_off[SD_MAX_K + 2];
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
#pragma unroll
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

// u in (0, 1], a multiple of 2^-24: exact in float and double.
__device__ __forceinline__ double uniform_u(uint64_t seed, int64_t row, int pos, int slot) {
  const uint32_t x = philox_w0(seed, (uint32_t)row, (uint32_t)pos, (uint32_t)slot);
  return (double)((x >> 8) + 1u) * (1.0 / 16777216.0);
}

// ------------------------------------------------------------- primitives --
// 2^x on the special-function unit.  Results below 2^-126 flush to zero, far
// below anything that moves a sum of at least 1.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 2^d for a double d without a double-precision transcendental: the integer
// part goes into the float exponent, the fraction (exact in double) through
// ex2 (relative error about 2^-22).  Results below the normal range are 0.
__device__ __forceinline__ float exp2_split(double d) {
  if (!(d > -126.0)) return 0.f;
  if (d >= 128.0) return INFINITY;
  const double n = floor(d);
  const float y = ex2((float)(d - n));  // in [1, 2)
  return __int_as_float(__float_as_int(y) + ((int)n << 23));
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
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ int warp_min_i(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Order of (value, index) candidates: larger value first, then lower index.
__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

// Warp-wide best (value desc, index asc) of one candidate per lane.
__device__ __forceinline__ void warp_best(float &v, int &i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, o);
    const int oi = __shfl_xor_sync(0xffffffffu, i, o);
    if (better(ov, oi, v, i)) {
      v = ov;
      i = oi;
    }
  }
}

// Bitonic sort of one value per lane, descending; returns this lane's value.
__device__ __forceinline__ float warp_sort_desc(float v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const float o = __shfl_xor_sync(0xffffffffu, v, j);
      const bool up = ((lane & k) == 0);
      const bool lower = ((lane & j) == 0);
      v = (lower == up) ? fmaxf(v, o) : fminf(v, o);
    }
  }
  return v;
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
};

// ---------------------------------------------------------------- rows ----
// One logit row as this CTA sees it: the slice [v0, v1) occupies `nvec`
// 16-byte vectors starting at `gbase`, the 16-byte boundary at or below
// element v0 (element v0 sits `hp` bytes into vector 0).  Vectors in
// [qlo, qhi) lie wholly inside the slice and are copied with cp.async; the
// (at most two) others are assembled from element loads with -inf in the
// bytes outside the slice, so every vector a thread sees is a plain list of
// logits with -inf padding.  `qd` is the vector holding the token excluded
// from this row's keys (-1 if it is not in this slice).
struct RowInfo {
  const uint8_t *g;      // element 0 of the row
  const uint8_t *gbase;  // 16-byte boundary at or below element v0
  int kind, j;           // RowKind, position
  int flags;             // RowFlag bits
  int excl;              // token excluded from the keys (-1: none)
  int fan;               // keys wanted from this row
  int hp, nvec, nsteps, qlo, qhi, qd;
};

// Element index of element i of slice vector q.
__device__ __forceinline__ int elem_index(int v0, int hp, int q, int i, int sz) {
  return v0 + (q * 16 - hp) / sz + i;
}

template <int NT>
__device__ __forceinline__ void row_geometry(RowInfo &R, int v0, int v1, int sz) {
  constexpr int kStepVec = NT * kU;
  R.gbase = R.g;
  R.hp = R.nvec = R.nsteps = R.qlo = R.qhi = 0;
  R.qd = -1;
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
  if (R.excl >= v0 && R.excl < v1) R.qd = ((R.excl - v0) * sz + R.hp) / 16;
}

// Vector q of row R's slice assembled from element loads (ragged ends, or
// -inf past the slice).
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

// Vector q of row R's slice read directly (128-bit load when it lies inside
// the slice), -inf past `R.nvec`.
template <typename E>
__device__ __forceinline__ uint4 load_vec_direct(const RowInfo &R, int q, int v0, int v1) {
  if (q >= R.qlo && q < R.qhi) return ld_stream(R.gbase + 16 * q);
  return load_vec_slow<E>(R, q, v0, v1);
}

// One 16-byte vector q (< qend) of row R into this thread's k-th slot of
// ring slot `slot`; ragged ends are read when consumed.
template <int NT>
__device__ __forceinline__ void issue_vec(const RowInfo &R, int q, int qend, uint32_t ring,
                                          int slot, int k) {
  if (q < qend && q >= R.qlo && q < R.qhi)
    cp_async16(ring + (uint32_t)(((slot * kU + k) * NT + threadIdx.x) * 16), R.gbase + 16 * q);
}
template <typename E, int NT>
__device__ __forceinline__ uint4 fetch_vec(const RowInfo &R, int q, int qend, const uint8_t *ring,
                                           int slot, int k, int v0, int v1) {
  if (q < qend && q >= R.qlo && q < R.qhi)
    return *reinterpret_cast<const uint4 *>(ring + ((slot * kU + k) * NT + threadIdx.x) * 16);
  if (q >= qend || q >= R.nvec) {
    const uint32_t w = Elt<E>::kNegInfWord;
    return make_uint4(w, w, w, w);
  }
  return load_vec_slow<E>(R, q, v0, v1);
}

// Each thread copies its own kU vectors of one step of row R into its own
// slots of ring slot `slot` (vectors inside the slice only).
template <int NT>
__device__ __forceinline__ void issue_unit(const RowInfo &R, int step, uint32_t ring, int slot) {
  constexpr int kStepVec = NT * kU;
#pragma unroll
  for (int k = 0; k < kU; ++k) {
    const int q = step * kStepVec + threadIdx.x + k * NT;
    if (q >= R.qlo && q < R.qhi)
      cp_async16(ring + (uint32_t)(((slot * kU + k) * NT + threadIdx.x) * 16), R.gbase + 16 * q);
  }
}
// Vector k of this thread's part of one step: from the ring, or assembled.
template <typename E, int NT>
__device__ __forceinline__ uint4 unit_vec(const RowInfo &R, int step, int k, const uint8_t *ring,
                                          int slot, int v0, int v1) {
  constexpr int kStepVec = NT * kU;
  const int q = step * kStepVec + threadIdx.x + k * NT;
  if (q >= R.qlo && q < R.qhi)
    return *reinterpret_cast<const uint4 *>(ring + ((slot * kU + k) * NT + threadIdx.x) * 16);
  if (q >= R.nvec) {  // past the slice
    const uint32_t w = Elt<E>::kNegInfWord;
    return make_uint4(w, w, w, w);
  }
  return load_vec_slow<E>(R, q, v0, v1);
}

// -------------------------------------------------------- shared memory --
// Dynamic shared memory carve-out (byte offsets), identical on host and
// device.  nrows: rows streamed per sequence; KF: keys kept per row.
struct Layout {
  int ring, wstat, wtop, part_m, part_i, part_c, part_z, part_tv, part_ti, total;
};
__host__ __device__ inline int align128(int x) { return (x + 127) & ~127; }
__host__ __device__ inline Layout make_layout(int NT, int nrows, int KF) {
  const int nw = NT / 32;
  Layout L;
  int o = 0;
  L.ring = o;                                    // [kDepth][kU][NT] 16-byte slots
  o = align128(o + kDepth * kU * NT * 16);
  L.wstat = o;                                   // [nrows][nw] WStat
  o = align128(o + 16 * nrows * nw);
  L.wtop = o;                                    // [nrows][nw][KF] {v, i}
  o = align128(o + 8 * nrows * nw * KF);
  L.part_m = o;                                  // [nrows] float
  o = align128(o + 4 * nrows);
  L.part_i = o;                                  // [nrows] int
  o = align128(o + 4 * nrows);
  L.part_c = o;                                  // [nrows] float
  o = align128(o + 4 * nrows);
  L.part_z = o;                                  // [nrows] double
  o = align128(o + 8 * nrows);
  L.part_tv = o;                                 // [nrows][KF] float
  o = align128(o + 4 * nrows * KF);
  L.part_ti = o;                                 // [nrows][KF] int
  o = align128(o + 4 * nrows * KF);
  L.total = o;
  return L;
}

// Warp partial of one row: max, sum z of 2^(l s + c), offset c, argmax.
struct WStat {
  float m, z, c;
  int idx;
};

struct Static {
  RowInfo rows[kMaxRows];
  int trow[SD_MAX_K + 1];  // row slot of target row j
  int drow[SD_MAX_K + 1];  // row slot of draft row j (K: bonus row), -1 if absent
  int nrows;
  int d[SD_MAX_K];         // drafted tokens
  float ld_t[SD_MAX_K];    // target logit of d_j
  float ld_d[SD_MAX_K];    // draft logit of d_j
  float M[kMaxRows];       // combined row statistics: max,
  float C[kMaxRows];       //   offset C: sum over the row of 2^(l s) = Z 2^-C
  double Z[kMaxRows];
  int amax[kMaxRows];      //   lowest index of the max
  int m, kind, owner, valid;  // kind: 0 none, 1 residual at m, 2 from p at m
  double t_loc;
  int cstar;
  double s_part;              // this CTA's mass of the sampling pass
  double wmass[kMaxWarps];    //   per warp (contiguous ranges), and its prefix
  double wpre[kMaxWarps];
  int wsel;                   //   the warp holding the crossing point
  double t_w;
  double red_d[kMaxWarps];
  int red_i[kMaxWarps];
  int tok;
  int flag_compact;
};

// --------------------------------------------------------- finalization --
// Exclusive scan of tau and packing of out_tokens, one CTA.  `cg_loads`
// reads values written by other CTAs of the same grid through L2.
__device__ void compact_block(int B, int K, const int32_t *out_tokens, const int32_t *tau,
                              int32_t *offsets, int32_t *packed, int32_t *status, bool cg_loads,
                              int *red) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int carry = 0;
  for (int base = 0; base < B; base += blockDim.x) {
    const int b = base + threadIdx.x;
    int t = 0;
    if (b < B) {
      t = cg_loads ? __ldcg(tau + b) : tau[b];
      if (t < 0 || t > K + 1) {
        if (status) atomicOr(status, (int)SD_STATUS_BAD_TOKEN);
        t = 0;
      }
    }
    int x = t;  // inclusive warp scan
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) red[w] = x;
    __syncthreads();
    if (w == 0) {
      int v = lane < nw ? red[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += y;
      }
      if (lane < nw) red[lane] = v;  // inclusive warp totals
    }
    __syncthreads();
    const int excl = carry + (w > 0 ? red[w - 1] : 0) + x - t;
    if (b < B) {
      offsets[b] = excl;
      const int32_t *src = out_tokens + (int64_t)b * (K + 1);
      for (int i = 0; i < t; ++i) packed[excl + i] = cg_loads ? __ldcg(src + i) : src[i];
    }
    carry += red[nw - 1];
    __syncthreads();
  }
  if (threadIdx.x == 0) offsets[B] = carry;
}

// ------------------------------------------------------------ the kernel --
// Weights of the sampling pass for the elements of one target vector:
// residual Zt (p - q)+ = max(0, 2^(l s + Ct) - 2^(l' s + Cd) R), R = Zt / Zd,
// or Zt p = 2^(l s + Ct) for a draw from p.
template <typename E>
__device__ __forceinline__ void pass_weights(const float *ft, const float *fd, bool residual,
                                             float Ct, float Cd, float s, float R, float *w) {
  constexpr int N = Elt<E>::kPerVec;
#pragma unroll
  for (int k = 0; k < N; ++k) {
    const float pt = ex2(fmaf(ft[k], s, Ct));
    w[k] = residual ? fmaxf(0.f, pt - ex2(fmaf(fd[k], s, Cd)) * R) : pt;
  }
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

// One step of one row: kU vectors per thread.
template <typename E, int KF, int NT>
__device__ __forceinline__ void process_step(RowAcc<KF> &A, int flags, int hp, int qd, int excl,
                                             int step, const uint4 *v, int v0, float s) {
  constexpr int sz = Elt<E>::kSize, N = Elt<E>::kPerVec;
  const int qbase = step * (NT * kU) + threadIdx.x;
  float vm[kU];
  float gmax = -INFINITY;
#pragma unroll
  for (int k = 0; k < kU; ++k) {
    vm[k] = Elt<E>::vmax(v[k]);
    gmax = fmaxf(gmax, vm[k]);
  }
  if (gmax > A.m) {
    A.m = gmax;
    if (flags & kNeedArg) {
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
  }
  if ((flags & kNeedExp) && gmax > -INFINITY) {
    const float cg = -(gmax * s);
    if (A.c == INFINITY) {
      A.c = cg;
    } else if (A.c - cg > kRebase) {  // the max rose by more than kRebase (log2)
      const float f = ex2(cg - A.c);
      A.z *= f;
      A.zc *= f;
      A.c = cg;
    }
    float vs[kU];  // independent per-vector sums, then one compensated add
#pragma unroll
    for (int k = 0; k < kU; ++k) {
      float f[N];
      Elt<E>::unpack(v[k], f);
#pragma unroll
      for (int i = 0; i < N; ++i) f[i] = ex2(fmaf(f[i], s, A.c));
#pragma unroll
      for (int h = N / 2; h > 0; h >>= 1)
#pragma unroll
        for (int i = 0; i < h; ++i) f[i] += f[i + h];
      vs[k] = f[0];
    }
#pragma unroll
    for (int h = kU / 2; h > 0; h >>= 1)
#pragma unroll
      for (int k = 0; k < h; ++k) vs[k] += vs[k + h];
    kahan_add(A.z, A.zc, vs[0]);
  }
  if (KF > 0 && (flags & kNeedKeys)) {
    // The top-KF elements of a set lie in its top-KF vectors ranked by
    // (max, index): every vector holding one of them has a max at least the
    // KF-th value, and at most KF vectors reach it.  Track those vectors.
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
    if (step == 0) {  // first step of the row: a warp-wide lower bound
      const float srt = warp_sort_desc(vm[0]);
      A.theta = __shfl_sync(0xffffffffu, srt, KF - 1);
    }
#pragma unroll
    for (int k = 0; k < kU; ++k) {
      if (vm[k] > A.kv[KF - 1] && vm[k] >= A.theta) {
        A.kv[KF - 1] = vm[k];
        A.kq[KF - 1] = qbase + k * NT;
#pragma unroll
        for (int x = KF - 1; x > 0; --x) {
          if (better(A.kv[x], A.kq[x], A.kv[x - 1], A.kq[x - 1])) {
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

// End of a row: warp-level statistics into wstat / wtop.
template <typename E, int KF>
__device__ __forceinline__ void row_end(RowAcc<KF> &A, const RowInfo &R, int v0, int v1,
                                        WStat *ws, float2 *wt) {
  constexpr int sz = Elt<E>::kSize, N = Elt<E>::kPerVec;
  constexpr int KFm = RowAcc<KF>::KFm;
  const int lane = threadIdx.x & 31;
  const float mw = warp_max(A.m);
  int idx = INT32_MAX;
  if ((R.flags & kNeedArg) && A.m == mw && A.m > -INFINITY && A.bq >= 0) {
    float f[N];
    Elt<E>::unpack(A.bv, f);
#pragma unroll
    for (int i = N - 1; i >= 0; --i)
      if (f[i] == A.m) idx = elem_index(v0, R.hp, A.bq, i, sz);
  }
  const int iw = warp_min_i(idx);
  const bool has = A.z > 0.f;
  const float cw = -warp_max(has ? -A.c : -INFINITY);  // min offset of the warp
  const float zt = has ? (A.z - A.zc) * ex2(cw - A.c) : 0.f;
  const float zw = warp_sum(zt);
  if (lane == 0) *ws = WStat{mw, zw, cw, iw};
  if (KF > 0 && (R.flags & kNeedKeys)) {
    // the warp's best KF vectors, then its best KF elements among them
    int selq[KFm];
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
      selq[r] = bv > -INFINITY ? bq : INT32_MAX;
    }
    constexpr int NC = KFm * N;                   // candidate elements
    constexpr int PER = (NC + 31) / 32;           // per lane
    float cv[PER];
    int ci[PER];
#pragma unroll
    for (int h = 0; h < PER; ++h) {
      cv[h] = -INFINITY;
      ci[h] = INT32_MAX;
      const int c = lane + 32 * h;
      if (c < NC) {
        int qq = INT32_MAX;
#pragma unroll
        for (int r = 0; r < KFm; ++r)
          if (r == c / N) qq = selq[r];
        if (qq != INT32_MAX) {
          const int e = elem_index(v0, R.hp, qq, c % N, sz);
          if (e >= v0 && e < v1 && e != R.excl) {
            const float x = Elt<E>::load_global(R.g + (int64_t)e * sz);
            if (x > -INFINITY) {
              cv[h] = x;
              ci[h] = e;
            }
          }
        }
      }
    }
#pragma unroll
    for (int r = 0; r < KFm; ++r) {
      int hb = 0;
#pragma unroll
      for (int h = 1; h < PER; ++h)
        if (better(cv[h], ci[h], cv[hb], ci[hb])) hb = h;
      float bv = -INFINITY;
      int bi = INT32_MAX;
#pragma unroll
      for (int h = 0; h < PER; ++h)
        if (h == hb) {
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
      if (lane == 0) wt[r] = make_float2(bv, __int_as_float(bi));
    }
  }
  A.reset();
}

template <typename E, int KF, int NT>
__global__ void __launch_bounds__(NT, 768 / NT) sd_seq_kernel(const __grid_constant__ Params P) {
  constexpr int sz = Elt<E>::kSize, NV = Elt<E>::kPerVec;
  constexpr int KFm = KF > 0 ? KF : 1;
  constexpr int NW = NT / 32;
  constexpr int kStepVec = NT * kU;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int cs = P.cs;
  const int b = blockIdx.x / cs;
  const int K = P.K;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  __shared__ Static S;
  extern __shared__ __align__(128) uint8_t dyn[];

  const int v0 = min(rank * P.slice, P.V);
  const int v1 = min(v0 + P.slice, P.V);
  const bool verify = P.mode == kVerify;
  const float T = verify ? P.temps[b] : 0.f;
  const bool tvalid = !verify || ((T >= 0.f) && (T <= 3.4e38f));  // rejects NaN / inf / < 0
  const bool sampled = verify && tvalid && T > 0.f;
  // scaled logits x = l s with s = log2(e) / T rounded to float; every
  // exponential below uses this same s
  const float s = sampled ? (float)(1.4426950408889634 / (double)T) : 0.f;
  const double sd = (double)s;

  // ---- drafted tokens
  int dvalid_local = 1;
  int my_d = -1;
  for (int j = tid; j < K; j += NT) {
    const int d = P.tokens[(int64_t)b * K + j];
    S.d[j] = d;
    if (!(d >= 0 && d < P.V)) dvalid_local = 0;
    if (j == tid) my_d = d;
  }
  const bool dvalid = __syncthreads_and(dvalid_local) != 0;

  // ---- the rows this CTA streams, in order (bonus, K, then K-1..0)
  if (tid == 0) {
    int n = 0;
    const int64_t V = P.V;
    for (int j = 0; j <= K; ++j) {
      S.trow[j] = -1;
      S.drow[j] = -1;
    }
    auto add = [&](const uint8_t *g, int kind, int j, int flags, int excl, int fan) {
      RowInfo &R = S.rows[n];
      R.g = g;
      R.kind = kind;
      R.j = j;
      R.flags = flags;
      R.excl = excl;
      R.fan = fan;
      row_geometry<NT>(R, v0, v1, sz);
      if (kind == kTarget) S.trow[j] = n;
      else S.drow[j] = n;
      ++n;
    };
    const int fK = P.keys ? P.fanout[K] : 0;
    if (fK > 0 && P.bonus) add(P.bonus + (int64_t)b * V * sz, kBonus, K, kNeedKeys, -1, fK);
    if (verify)
      add(P.target + ((int64_t)b * (K + 1) + K) * V * sz, kTarget, K,
          kNeedArg | (sampled ? kNeedExp : 0), -1, 0);
    for (int j = K - 1; j >= 0; --j) {
      const int fj = P.keys ? P.fanout[j] : 0;
      if (sampled || fj > 0)
        add(P.draft + ((int64_t)b * K + j) * V * sz, kDraft, j,
            (sampled ? kNeedExp : 0) | (fj > 0 ? kNeedKeys : 0), S.d[j], fj);
      if (verify)
        add(P.target + ((int64_t)b * (K + 1) + j) * V * sz, kTarget, j,
            kNeedArg | (sampled ? kNeedExp : 0), -1, 0);
    }
    S.nrows = n;
    S.flag_compact = 0;
  }
  __syncthreads();

  // the logits at the drafted tokens: loaded now, used after the stream
  float my_lt = -INFINITY, my_ld = -INFINITY;
  if (tid < K && sampled && my_d >= 0 && my_d < P.V) {
    my_lt = Elt<E>::load_global(P.target + (((int64_t)b * (K + 1) + tid) * P.V + my_d) * sz);
    my_ld = Elt<E>::load_global(P.draft + (((int64_t)b * K + tid) * P.V + my_d) * sz);
  }

  const int nrows = S.nrows;
  const Layout L = make_layout(NT, nrows, KF);
  uint8_t *ring = dyn + L.ring;
  const uint32_t ring_s = smem_u32(ring);
  WStat *wstat = reinterpret_cast<WStat *>(dyn + L.wstat);
  float2 *wtop = reinterpret_cast<float2 *>(dyn + L.wtop);  // .x value, .y index bits
  float *part_m = reinterpret_cast<float *>(dyn + L.part_m);
  int *part_i = reinterpret_cast<int *>(dyn + L.part_i);
  float *part_c = reinterpret_cast<float *>(dyn + L.part_c);
  double *part_z = reinterpret_cast<double *>(dyn + L.part_z);
  float *part_tv = reinterpret_cast<float *>(dyn + L.part_tv);
  int *part_ti = reinterpret_cast<int *>(dyn + L.part_ti);

  // ---- stream every row once.  Each thread copies its own vectors
  // kDepth-1 steps ahead into its own ring slots (cp.async).
  int total = 0;
  for (int r = 0; r < nrows; ++r) total += S.rows[r].nsteps;
  RowAcc<KF> A;
  A.reset();
  auto advance = [&](int &row, int &step) {
    ++step;
    while (row < nrows && step >= S.rows[row].nsteps) {
      ++row;
      step = 0;
    }
  };
  int i_row = 0, i_step = 0;  // next step to copy
  while (i_row < nrows && S.rows[i_row].nsteps == 0) ++i_row;
  int c_row = i_row, c_step = 0;  // step being consumed
  auto issue_next = [&](int slot) {
    if (i_row < nrows) {
      issue_unit<NT>(S.rows[i_row], i_step, ring_s, slot);
      advance(i_row, i_step);
    }
    cp_commit();
  };
#pragma unroll
  for (int d = 0; d < kDepth - 1; ++d) issue_next(d);
  for (int st = 0; st < total; ++st) {
    issue_next((st + kDepth - 1) % kDepth);
    cp_wait<kDepth - 1>();  // this step's copies have landed
    const RowInfo &R = S.rows[c_row];
    const int flags = R.flags, hp = R.hp, qd = R.qd, excl = R.excl, nsteps = R.nsteps;
    uint4 cur[kU];
#pragma unroll
    for (int k = 0; k < kU; ++k)
      cur[k] = unit_vec<E, NT>(R, c_step, k, ring, st % kDepth, v0, v1);
    process_step<E, KF, NT>(A, flags, hp, qd, excl, c_step, cur, v0, s);
    if (c_step == nsteps - 1)
      row_end<E, KF>(A, S.rows[c_row], v0, v1, &wstat[c_row * NW + warp],
                     &wtop[(c_row * NW + warp) * KFm]);
    advance(c_row, c_step);
  }
  cp_wait<0>();

  // rows with an empty slice (this CTA holds no vocabulary) still need entries
  if (total == 0) {
    for (int x = tid; x < nrows * NW; x += NT) wstat[x] = WStat{-INFINITY, 0.f, INFINITY, INT32_MAX};
    if (KF > 0)
      for (int x = tid; x < nrows * NW * KFm; x += NT)
        wtop[x] = make_float2(-INFINITY, __int_as_float(INT32_MAX));
  }
  if (tid < K) {
    S.ld_t[tid] = my_lt;
    S.ld_d[tid] = my_ld;
  }
  __syncthreads();

  // ---- CTA statistics per row (one warp per row)
  for (int r = warp; r < nrows; r += NW) {
    const RowInfo &R = S.rows[r];
    const WStat wsl = lane < NW ? wstat[r * NW + lane] : WStat{-INFINITY, 0.f, INFINITY, INT32_MAX};
    const float Mc = warp_max(wsl.m);
    const int ic = warp_min_i(wsl.m == Mc ? wsl.idx : INT32_MAX);
    const bool has = wsl.z > 0.f;
    const float cb = -warp_max(has ? -wsl.c : -INFINITY);
    const double term = has ? (double)wsl.z * (double)ex2(cb - wsl.c) : 0.0;
    const double Zc = warp_sum_d(term);
    if (lane == 0) {
      part_m[r] = Mc;
      part_i[r] = ic;
      part_c[r] = cb;
      part_z[r] = Zc;
    }
    if (KF > 0 && (R.flags & kNeedKeys)) {
      // NW x KF candidates; lane l holds candidates l, l + 32, ...
      constexpr int PER = (NW * KFm + 31) / 32;
      float cv[PER];
      int ci[PER];
#pragma unroll
      for (int h = 0; h < PER; ++h) {
        const int c = lane + 32 * h;
        cv[h] = -INFINITY;
        ci[h] = INT32_MAX;
        if (c < NW * KFm) {
          const float2 e = wtop[r * NW * KFm + c];
          cv[h] = e.x;
          ci[h] = __float_as_int(e.y);
        }
      }
      for (int r2 = 0; r2 < KFm; ++r2) {
        int hb = 0;
#pragma unroll
        for (int h = 1; h < PER; ++h)
          if (better(cv[h], ci[h], cv[hb], ci[hb])) hb = h;
        float bv = -INFINITY;
        int bi = INT32_MAX;
#pragma unroll
        for (int h = 0; h < PER; ++h)
          if (h == hb) {
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
          part_tv[r * KFm + r2] = bv;
          part_ti[r * KFm + r2] = bi;
        }
      }
    }
  }
  cluster.sync();  // (1) every CTA's per-row partials are ready

  // ---- combine the cluster's partials (same arithmetic in every CTA)
  for (int r = warp; r < nrows; r += NW) {
    const RowInfo &R = S.rows[r];
    float pm = -INFINITY, pc = INFINITY;
    double pz = 0.0;
    int pi = INT32_MAX;
    if (lane < cs) {
      pm = *cluster.map_shared_rank(&part_m[r], lane);
      pc = *cluster.map_shared_rank(&part_c[r], lane);
      pz = *cluster.map_shared_rank(&part_z[r], lane);
      pi = *cluster.map_shared_rank(&part_i[r], lane);
    }
    const float M = warp_max(pm);
    const int am = warp_min_i(pm == M ? pi : INT32_MAX);
    const bool has = pz > 0.0;
    const float C = -warp_max(has ? -pc : -INFINITY);
    const double term = has ? pz * (double)ex2(C - pc) : 0.0;
    const double Z = warp_sum_d(term);
    if (lane == 0) {
      S.M[r] = M;
      S.C[r] = C;
      S.Z[r] = Z;
      S.amax[r] = am == INT32_MAX ? 0 : am;
    }
    if (KF > 0 && (R.flags & kNeedKeys) && rank == 0 && P.keys_out) {
      // merge cs x KF candidates into this row's keys
      constexpr int PER = (kMaxCS * KFm + 31) / 32;
      float cv[PER];
      int ci[PER];
#pragma unroll
      for (int h = 0; h < PER; ++h) {
        const int c = lane + 32 * h;  // candidate c: peer c / KF, rank c % KF
        cv[h] = -INFINITY;
        ci[h] = INT32_MAX;
        if (c < cs * KFm) {
          cv[h] = *cluster.map_shared_rank(&part_tv[r * KFm + c % KFm], c / KFm);
          ci[h] = *cluster.map_shared_rank(&part_ti[r * KFm + c % KFm], c / KFm);
        }
      }
      int32_t *kout = P.keys_out + ((int64_t)b * P.n_keys_out + P.fan_off[R.j]) * 2;
      for (int r2 = 0; r2 < R.fan; ++r2) {
        int hb = 0;
#pragma unroll
        for (int h = 1; h < PER; ++h)
          if (better(cv[h], ci[h], cv[hb], ci[hb])) hb = h;
        float bv = -INFINITY;
        int bi = INT32_MAX;
#pragma unroll
        for (int h = 0; h < PER; ++h)
          if (h == hb) {
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
          kout[2 * r2] = bi == INT32_MAX ? -1 : R.j;
          kout[2 * r2 + 1] = bi == INT32_MAX ? -1 : bi;
        }
      }
    }
  }
  // keys of the bonus position when there is no bonus row: empty slots
  if (P.keys && P.keys_out && rank == 0 && tid == 0 && P.fanout[K] > 0 && S.drow[K] < 0) {
    int32_t *kout = P.keys_out + ((int64_t)b * P.n_keys_out + P.fan_off[K]) * 2;
    for (int r2 = 0; r2 < P.fanout[K]; ++r2) {
      kout[2 * r2] = -1;
      kout[2 * r2 + 1] = -1;
    }
  }
  __syncthreads();

  if (verify) {
    // ---- accept tests, one lane per position (K <= 32: warp 0)
    if (warp == 0) {
      const int j = lane;
      int rej = 0;
      if (j < K) {
        const int rt = S.trow[j];
        const int d = S.d[j];
        int a = 0;
        if (!sampled) {
          a = (dvalid && d == S.amax[rt]) ? 1 : 0;
        } else if (dvalid) {
          const int rd = S.drow[j];
          // log2 of 2^(l_d s + C): the product of two floats is exact in double
          const double xt = (double)S.ld_t[j] * sd + (double)S.C[rt];
          const double xd = (double)S.ld_d[j] * sd + (double)S.C[rd];
          const float r = (S.ld_d[j] == -INFINITY)
                              ? INFINITY  // q(d) = 0
                              : exp2_split(xt - xd) * ((float)S.Z[rd] / (float)S.Z[rt]);
          const double u = uniform_u(P.seed, P.row_base + b, j, 0);
          a = (u <= (double)r) ? 1 : 0;
          if (rank == 0) {
            const int64_t pj = (int64_t)b * K + j;
            if (P.ratio_out) P.ratio_out[pj] = r;
            if (P.p_out) P.p_out[pj] = exp2_split(xt) / (float)S.Z[rt];
            if (P.q_out) P.q_out[pj] = exp2_split(xd) / (float)S.Z[rd];
          }
        }
        rej = !a;
      }
      const unsigned rejects = __ballot_sync(0xffffffffu, rej);
      if (lane == 0) {
        const int mm = rejects ? __ffs(rejects) - 1 : K;
        S.m = mm;
        S.valid = (tvalid && dvalid) ? 1 : 0;
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
    // Each warp takes a contiguous range of the slice, so warp masses are in
    // index order; the owning CTA finds the crossing warp, which re-scans its
    // range in 32-vector chunks.
    for (int attempt = 0; attempt < 2 && S.kind != 0; ++attempt) {
      const int mm = S.m;
      const bool residual = S.kind == 1;
      const RowInfo &Rt = S.rows[S.trow[mm]];
      const RowInfo *Rd = residual ? &S.rows[S.drow[mm]] : nullptr;
      const bool d_vec = residual && Rd->hp == Rt.hp;  // same vector grid
      const float Ct = S.C[S.trow[mm]];
      const float Cd = residual ? S.C[S.drow[mm]] : 0.f;
      const float Rz = residual ? (float)(S.Z[S.trow[mm]] / S.Z[S.drow[mm]]) : 0.f;
      const int wr = (Rt.nvec + NW - 1) / NW;  // vectors per warp
      const int wq0 = min(warp * wr, Rt.nvec), wq1 = min(wq0 + wr, Rt.nvec);
      const int wsteps = (wr + 32 * kU - 1) / (32 * kU);
      // weights of this lane's vector q of the target (and draft) row
      auto vec_mass = [&](uint4 tvec, uint4 dvec, int q, bool dv_ok) -> float {
        float ft[NV], fd[NV], w[NV];
        Elt<E>::unpack(tvec, ft);
        if (residual) {
          if (dv_ok) {
            Elt<E>::unpack(dvec, fd);
          } else {
#pragma unroll
            for (int i = 0; i < NV; ++i) {
              const int e = elem_index(v0, Rt.hp, q, i, sz);
              fd[i] = (e >= v0 && e < v1) ? Elt<E>::load_global(Rd->g + (int64_t)e * sz)
                                          : -INFINITY;
            }
          }
        }
        pass_weights<E>(ft, fd, residual, Ct, Cd, s, Rz, w);
#pragma unroll
        for (int h = NV / 2; h > 0; h >>= 1)
#pragma unroll
          for (int i = 0; i < h; ++i) w[i] += w[i + h];
        return w[0];
      };
      // units: target step t, then (same vector grid) draft step t
      const int per = d_vec ? 2 : 1;
      const int nunits = wsteps * per;
      int i_u = 0;
      auto issue_pass = [&](int slot) {
        if (i_u < nunits) {
          const RowInfo &RR = (i_u % per == 0) ? Rt : *Rd;
          const int t = i_u / per;
#pragma unroll
          for (int k = 0; k < kU; ++k)
            issue_vec<NT>(RR, wq0 + t * 32 * kU + k * 32 + lane, wq1, ring_s, slot, k);
          ++i_u;
        }
        cp_commit();
      };
#pragma unroll
      for (int d = 0; d < kDepth - 1; ++d) issue_pass(d);
      float tsum = 0.f, tcomp = 0.f;
      uint4 tv4[kU];
      for (int u = 0; u < nunits; ++u) {
        issue_pass((u + kDepth - 1) % kDepth);
        cp_wait<kDepth - 1>();
        const int t = u / per;
        if (u % per == 0) {
#pragma unroll
          for (int k = 0; k < kU; ++k)
            tv4[k] = fetch_vec<E, NT>(Rt, wq0 + t * 32 * kU + k * 32 + lane, wq1, ring, u % kDepth,
                                      k, v0, v1);
          if (per == 2) continue;  // the draft unit follows
        }
        float vs[kU];
#pragma unroll
        for (int k = 0; k < kU; ++k) {
          const int q = wq0 + t * 32 * kU + k * 32 + lane;
          uint4 dvec = tv4[k];
          if (d_vec) dvec = fetch_vec<E, NT>(*Rd, q, wq1, ring, u % kDepth, k, v0, v1);
          vs[k] = q < wq1 ? vec_mass(tv4[k], dvec, q, d_vec) : 0.f;
        }
#pragma unroll
        for (int h = kU / 2; h > 0; h >>= 1)
#pragma unroll
          for (int k = 0; k < h; ++k) vs[k] += vs[k + h];
        kahan_add(tsum, tcomp, vs[0]);
      }
      cp_wait<0>();
      // warp masses, their prefix, the CTA mass
      const double wm = warp_sum_d((double)tsum - (double)tcomp);
      if (lane == 0) S.wmass[warp] = wm;
      __syncthreads();
      if (warp == 0) {
        const double m_l = lane < NW ? S.wmass[lane] : 0.0;
        double incl = m_l;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const double y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        if (lane < NW) S.wpre[lane] = incl - m_l;
        if (lane == 31) S.s_part = incl;
      }
      cluster.sync();  // (2) slice masses ready
      if (warp == 0) {
        // prefix of the slice masses over the cluster (lane c: CTA c)
        const double sc = lane < cs ? *cluster.map_shared_rank(&S.s_part, lane) : 0.0;
        double incl = sc;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const double y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        const double tot = __shfl_sync(0xffffffffu, incl, 31);
        if (tot > 0.0 || !residual) {
          const double u = uniform_u(P.seed, P.row_base + b, mm, 1);
          const double t = u * tot;
          const unsigned cross = __ballot_sync(0xffffffffu, sc > 0.0 && incl > t);
          const unsigned pos = __ballot_sync(0xffffffffu, sc > 0.0);
          // the first CTA whose range passes t; if rounding put t past the
          // total, the last CTA with mass
          const int cstar = cross ? __ffs(cross) - 1 : (pos ? 31 - __clz(pos) : 0);
          const double before = __shfl_sync(0xffffffffu, incl - sc, cstar);
          if (lane == 0) {
            S.cstar = cstar;
            S.t_loc = t - before;
            S.owner = cstar;
          }
        } else if (lane == 0) {
          S.kind = 2;  // identically zero residual: draw from p at m
        }
      }
      __syncthreads();
      if (residual && S.kind == 2) {
        cluster.sync();  // peers are done reading this CTA's mass
        continue;
      }
      if (rank == S.cstar) {
        // the crossing warp: the first whose range passes t_loc, else the
        // last with mass
        if (warp == 0) {
          const double m_l = lane < NW ? S.wmass[lane] : 0.0;
          const double pre = lane < NW ? S.wpre[lane] : 0.0;
          const unsigned cross = __ballot_sync(0xffffffffu, m_l > 0.0 && pre + m_l > S.t_loc);
          const unsigned pos = __ballot_sync(0xffffffffu, m_l > 0.0);
          const int ws = cross ? __ffs(cross) - 1 : (pos ? 31 - __clz(pos) : 0);
          if (lane == 0) {
            S.wsel = ws;
            S.t_w = S.t_loc - S.wpre[ws];
          }
        }
        __syncthreads();
        if (warp == S.wsel) {
          // masses of this warp's vectors, in index order, into the (now
          // idle) ring memory; then a chunked scan
          float *vm_s = reinterpret_cast<float *>(ring);
          const int nq = wq1 - wq0;
          for (int base = 0; base < nq; base += 32 * kU) {
            uint4 tvv[kU], dvv[kU];
#pragma unroll
            for (int k = 0; k < kU; ++k) {
              const int q = wq0 + base + k * 32 + lane;
              tvv[k] = q < wq1 ? load_vec_direct<E>(Rt, q, v0, v1) : tvv[0];
              dvv[k] = (q < wq1 && d_vec) ? load_vec_direct<E>(*Rd, q, v0, v1) : tvv[k];
            }
#pragma unroll
            for (int k = 0; k < kU; ++k) {
              const int q = wq0 + base + k * 32 + lane;
              if (q < wq1) vm_s[q - wq0] = vec_mass(tvv[k], dvv[k], q, d_vec);
            }
          }
          __syncwarp();
          const double tw = S.t_w;
          double cum = 0.0;
          int qsel = -1;
          double before = 0.0;
          int qlast = -1;
          double before_last = 0.0;
          for (int base = 0; base < nq && qsel < 0; base += 32) {
            const int i = base + lane;
            const double mv = i < nq ? (double)vm_s[i] : 0.0;
            double incl = mv;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
              const double y = __shfl_up_sync(0xffffffffu, incl, o);
              if (lane >= o) incl += y;
            }
            const unsigned cross = __ballot_sync(0xffffffffu, mv > 0.0 && cum + incl > tw);
            const unsigned pos = __ballot_sync(0xffffffffu, mv > 0.0);
            if (cross) {
              const int l = __ffs(cross) - 1;
              qsel = wq0 + base + l;
              before = cum + __shfl_sync(0xffffffffu, incl - mv, l);
            } else if (pos) {
              const int l = 31 - __clz(pos);
              qlast = wq0 + base + l;
              before_last = cum + __shfl_sync(0xffffffffu, incl - mv, l);
            }
            cum += __shfl_sync(0xffffffffu, incl, 31);
          }
          if (qsel < 0) {  // rounding put the target past this warp's mass
            qsel = qlast;
            before = before_last;
          }
          if (lane == 0) {
            int tok = -1, klast = -1;
            if (qsel >= 0) {
              float ft[NV], fd[NV], w[NV];
              Elt<E>::unpack(load_vec_direct<E>(Rt, qsel, v0, v1), ft);
              if (residual) Elt<E>::unpack(load_vec_direct<E>(*Rd, qsel, v0, v1), fd);
              if (residual && !d_vec) {
#pragma unroll
                for (int i = 0; i < NV; ++i) {
                  const int e = elem_index(v0, Rt.hp, qsel, i, sz);
                  fd[i] = (e >= v0 && e < v1) ? Elt<E>::load_global(Rd->g + (int64_t)e * sz)
                                              : -INFINITY;
                }
              }
              pass_weights<E>(ft, fd, residual, Ct, Cd, s, Rz, w);
              double c2 = before;
              for (int i = 0; i < NV; ++i) {
                const int e = elem_index(v0, Rt.hp, qsel, i, sz);
                if (e < v0 || e >= v1 || !(w[i] > 0.f)) continue;
                klast = e;
                if (tok < 0 && c2 + (double)w[i] > tw) tok = e;
                c2 += (double)w[i];
              }
              if (tok < 0) tok = klast;
            }
            if (tok < 0) tok = S.amax[S.trow[mm]];  // degenerate: no mass in this slice
            S.tok = tok;
          }
        }
        __syncthreads();
      }
      break;
    }

    // ---- the sequence's outputs (owning CTA)
    if (rank == S.owner && tid == 0) {
      int32_t *out = P.out_tokens + (int64_t)b * (K + 1);
      if (!S.valid) {
        for (int j = 0; j <= K; ++j) out[j] = -1;
        P.num_accepted[b] = 0;
        P.tau[b] = 0;
        if (P.hit) P.hit[b] = 0;
        if (P.status)
          atomicOr(P.status, (tvalid ? 0 : (int)SD_STATUS_BAD_TEMP) |
                                 (dvalid ? 0 : (int)SD_STATUS_BAD_TOKEN));
      } else {
        const int mm = S.m, tok = S.tok;
        for (int j = 0; j < mm; ++j) out[j] = S.d[j];
        out[mm] = tok;
        for (int j = mm + 1; j <= K; ++j) out[j] = -1;
        P.num_accepted[b] = mm;
        P.tau[b] = mm + 1;
        if (P.hit) {
          int h = 0;
          if (P.keys && P.keys_out) {
            // written by rank 0 of this cluster before barrier (2), or by
            // this very CTA when it is rank 0
            const int32_t *kb = P.keys_out + (int64_t)b * P.n_keys_out * 2;
            for (int k2 = 0; k2 < P.n_keys_out; ++k2)
              if (__ldcg(kb + 2 * k2) == mm && __ldcg(kb + 2 * k2 + 1) == tok) h = 1;
          } else if (P.keys_in) {
            const int32_t *kb = P.keys_in + (int64_t)b * P.n_keys_in * 2;
            for (int k2 = 0; k2 < P.n_keys_in; ++k2)
              if (kb[2 * k2] == mm && kb[2 * k2 + 1] == tok) h = 1;
          }
          P.hit[b] = (uint8_t)h;
        }
      }
      if (P.compact) {
        __threadfence();
        const int done = atomicAdd(P.done_counter, 1);
        if (done == P.B - 1) {
          __threadfence();
          S.flag_compact = 1;
        }
      }
    }
    __syncthreads();
    if (S.flag_compact) {
      compact_block(P.B, K, P.out_tokens, P.tau, P.offsets, P.packed, P.status, true, S.red_i);
      if (tid == 0) *P.done_counter = 0;
    }
  }
  cluster.sync();  // peers may still read this CTA's shared memory
}

__global__ void sd_compact_kernel(int B, int K, const int32_t *out_tokens, const int32_t *tau,
                                  int32_t *offsets, int32_t *packed, int32_t *status) {
  __shared__ int red[32];
  compact_block(B, K, out_tokens, tau, offsets, packed, status, false, red);
}

__global__ void sd_uniforms_kernel(uint64_t seed, int n, const int32_t *row, const int32_t *pos,
                                   const int32_t *slot, double *out) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) out[i] = uniform_u(seed, row[i], pos[i], slot[i]);
}

// ------------------------------------------------------------------- host --
static int env_int(const char *name, int dflt) {
  const char *s = getenv(name);
  return s && *s ? atoi(s) : dflt;
}

static int sm_count() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 1;
  }
  return n;
}

static const int kDynSmemCap = 227 * 1024 - (int)sizeof(Static) - 256;

template <typename E, int KF, int NT>
static void *kernel_fn() {
  static std::once_flag once;
  void *fn = (void *)sd_seq_kernel<E, KF, NT>;
  std::call_once(once, [fn] {
    cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kDynSmemCap);
    cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    cudaGetLastError();
  });
  return fn;
}

// Rows streamed per sequence (upper bound used for the shared-memory size).
static int rows_per_seq(const Params &P) {
  int n = P.mode == kVerify ? 2 * P.K + 1 : P.K;
  if (P.keys && P.bonus && P.fanout[P.K] > 0) n += 1;
  return std::max(n, 1);
}

// Cluster size: slices of at most kMaxSliceVec vectors, then enough CTAs to
// give every SM two, at most kMaxCS.
static int choose_cs(int B, int V, int sz) {
  const int forced = env_int("SDV_CS", 0);
  if (forced) return forced;
  int cs = 1;
  while (cs < kMaxCS && (((int64_t)V + cs - 1) / cs * sz + 31) / 16 + 2 > kMaxSliceVec) cs <<= 1;
  while (cs < kMaxCS && (int64_t)B * cs < 2LL * sm_count()) cs <<= 1;
  return cs;
}

template <typename E, int KF, int NT>
static sd_status_t launch_nt(Params &P, int cs, cudaStream_t stream) {
  constexpr int sz = Elt<E>::kSize;
  P.cs = cs;
  P.slice = (int)((((int64_t)P.V + cs - 1) / cs + 15) / 16 * 16);
  const Layout L = make_layout(NT, rows_per_seq(P), KF);
  if (L.total > kDynSmemCap) return SD_ERR_UNSUPPORTED;
  void *fn = kernel_fn<E, KF, NT>();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(P.B * cs), 1, 1);
  cfg.blockDim = dim3(NT, 1, 1);
  cfg.dynamicSmemBytes = (size_t)L.total;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (env_int("SDV_VERBOSE", 0))
    fprintf(stderr, "sd_verify: mode=%d B=%d K=%d V=%d cs=%d NT=%d slice=%d KF=%d smem=%d\n",
            P.mode, P.B, P.K, P.V, cs, NT, P.slice, KF, L.total);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, (void (*)(const Params))fn, P);
  if (e != cudaSuccess) {
    fprintf(stderr, "sd_verify launch failed: %s\n", cudaGetErrorString(e));
    return SD_ERR_CUDA;
  }
  return SD_OK;
}

// 512-thread CTAs when the grid would leave SMs short of warps.
template <typename E, int KF>
static sd_status_t launch_kf(Params &P, cudaStream_t s) {
  constexpr int sz = Elt<E>::kSize;
  const int cs = choose_cs(P.B, P.V, sz);
  if (cs < 1 || cs > kMaxCS) return SD_ERR_INVALID_ARG;
  int nt = env_int("SDV_NT", 0);
  if (nt != 256 && nt != 512) nt = 256;
  return nt == 512 ? launch_nt<E, KF, 512>(P, cs, s) : launch_nt<E, KF, 256>(P, cs, s);
}

template <typename E>
static sd_status_t launch(Params &P, cudaStream_t s) {
  int fmax = 0;
  if (P.keys)
    for (int k = 0; k <= P.K; ++k) fmax = std::max(fmax, P.fanout[k]);
  if (fmax == 0) {
    P.keys = 0;
    return launch_kf<E, 0>(P, s);
  }
  if (fmax <= 2) return launch_kf<E, 2>(P, s);
  if (fmax <= 4) return launch_kf<E, 4>(P, s);
  return launch_kf<E, 8>(P, s);
}

static sd_status_t dispatch(Params &P, sd_dtype_t dt, cudaStream_t s) {
  return dt == SD_BF16 ? launch<__nv_bfloat16>(P, s) : launch<float>(P, s);
}

static bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

}  // namespace sdv

using namespace sdv;

extern "C" {

size_t sd_verify_workspace_size(int32_t B, int32_t K) {
  if (B < 0 || K < 0 || K > SD_MAX_K) return 0;
  return 256;  // one completion counter, padded
}

sd_status_t sd_verify(const sd_verify_args *a, void *stream) {
  if (!a) return SD_ERR_INVALID_ARG;
  if (a->B < 0 || a->K < 0 || a->K > SD_MAX_K || a->V < 1 || a->V > SD_MAX_V)
    return SD_ERR_INVALID_ARG;
  if (a->dtype != SD_F32 && a->dtype != SD_BF16) return SD_ERR_INVALID_ARG;
  if ((int64_t)a->B * kMaxCS > INT32_MAX) return SD_ERR_INVALID_ARG;
  const bool predict = (a->flags & SD_FLAG_PREDICT) != 0;
  const bool compact = (a->flags & SD_FLAG_COMPACT) != 0;
  if (a->flags & ~(SD_FLAG_PREDICT | SD_FLAG_COMPACT)) return SD_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  if (compact && !a->offsets) return SD_ERR_INVALID_ARG;
  if (a->B == 0) {
    if (compact && cudaMemsetAsync(a->offsets, 0, sizeof(int32_t), s) != cudaSuccess)
      return SD_ERR_CUDA;
    return SD_OK;
  }
  if (!a->target_logits || !a->temperature || !a->num_accepted || !a->out_tokens || !a->tau)
    return SD_ERR_INVALID_ARG;
  if (a->K > 0 && (!a->draft_logits || !a->draft_tokens)) return SD_ERR_INVALID_ARG;
  if (compact && !a->packed) return SD_ERR_INVALID_ARG;
  if (!a->workspace || !aligned(a->workspace, 16) ||
      a->workspace_bytes < sd_verify_workspace_size(a->B, a->K))
    return SD_ERR_INVALID_ARG;
  if (a->cache_keys && a->n_keys < 0) return SD_ERR_INVALID_ARG;
  const size_t esz = a->dtype == SD_BF16 ? 2 : 4;
  if (!aligned(a->target_logits, esz) || (a->draft_logits && !aligned(a->draft_logits, esz)))
    return SD_ERR_INVALID_ARG;

  Params P;
  memset(&P, 0, sizeof(P));
  P.mode = kVerify;
  P.target = (const uint8_t *)a->target_logits;
  P.draft = (const uint8_t *)a->draft_logits;
  P.tokens = a->draft_tokens;
  P.temps = a->temperature;
  P.num_accepted = a->num_accepted;
  P.out_tokens = a->out_tokens;
  P.tau = a->tau;
  P.hit = a->hit;
  P.offsets = a->offsets;
  P.packed = a->packed;
  P.ratio_out = a->accept_ratio;
  P.p_out = a->p_draft;
  P.q_out = a->q_draft;
  P.argmax_out = a->target_argmax;
  P.status = a->status;
  P.seed = a->seed;
  P.row_base = a->row_base;
  P.B = a->B;
  P.K = a->K;
  P.V = a->V;
  P.compact = compact ? 1 : 0;
  P.done_counter = (int32_t *)a->workspace;
  if (predict) {
    if (!a->fanout_host || !a->keys_out) return SD_ERR_INVALID_ARG;
    if (a->draft_bonus_logits && !aligned(a->draft_bonus_logits, esz)) return SD_ERR_INVALID_ARG;
    int off = 0;
    for (int k = 0; k <= a->K; ++k) {
      const int f = a->fanout_host[k];
      if (f < 0 || f > SD_MAX_FANOUT) return SD_ERR_INVALID_ARG;
      P.fanout[k] = f;
      P.fan_off[k] = off;
      off += f;
    }
    P.fan_off[a->K + 1] = off;
    P.keys = off > 0 ? 1 : 0;
    P.keys_out = a->keys_out;
    P.n_keys_out = off;
    P.bonus = (const uint8_t *)a->draft_bonus_logits;
  } else {
    P.keys_in = a->cache_keys;
    P.n_keys_in = a->cache_keys ? a->n_keys : 0;
  }
  return dispatch(P, a->dtype, s);
}

sd_status_t sd_outcome_predict(int32_t B, int32_t K, int32_t V, sd_dtype_t dtype,
                               const void *draft_logits, const int32_t *draft_tokens,
                               const void *draft_bonus_logits, const int32_t *fanout_host,
                               int32_t *keys, int32_t *n_keys_out, int32_t *status,
                               void *stream) {
  if (B < 0 || K < 0 || K > SD_MAX_K || V < 1 || V > SD_MAX_V) return SD_ERR_INVALID_ARG;
  if (dtype != SD_F32 && dtype != SD_BF16) return SD_ERR_INVALID_ARG;
  if (!fanout_host) return SD_ERR_INVALID_ARG;
  if ((int64_t)B * kMaxCS > INT32_MAX) return SD_ERR_INVALID_ARG;
  Params P;
  memset(&P, 0, sizeof(P));
  int off = 0;
  for (int k = 0; k <= K; ++k) {
    const int f = fanout_host[k];
    if (f < 0 || f > SD_MAX_FANOUT) return SD_ERR_INVALID_ARG;
    P.fanout[k] = f;
    P.fan_off[k] = off;
    off += f;
  }
  P.fan_off[K + 1] = off;
  if (n_keys_out) *n_keys_out = off;
  if (B == 0 || off == 0) return SD_OK;
  if (!keys || (K > 0 && (!draft_logits || !draft_tokens))) return SD_ERR_INVALID_ARG;
  const size_t esz = dtype == SD_BF16 ? 2 : 4;
  if ((draft_logits && !aligned(draft_logits, esz)) ||
      (draft_bonus_logits && !aligned(draft_bonus_logits, esz)))
    return SD_ERR_INVALID_ARG;
  P.mode = kPredict;
  P.draft = (const uint8_t *)draft_logits;
  P.bonus = (const uint8_t *)draft_bonus_logits;
  P.tokens = draft_tokens;
  P.keys = 1;
  P.keys_out = keys;
  P.n_keys_out = off;
  P.status = status;
  P.B = B;
  P.K = K;
  P.V = V;
  return dispatch(P, dtype, (cudaStream_t)stream);
}

sd_status_t sd_compact(int32_t B, int32_t K, const int32_t *out_tokens, const int32_t *tau,
                       int32_t *offsets, int32_t *packed, int32_t *status, void *stream) {
  if (B < 0 || K < 0 || K > SD_MAX_K || !offsets) return SD_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  if (B == 0) {
    return cudaMemsetAsync(offsets, 0, sizeof(int32_t), s) == cudaSuccess ? SD_OK : SD_ERR_CUDA;
  }
  if (!out_tokens || !tau || !packed) return SD_ERR_INVALID_ARG;
  sd_compact_kernel<<<1, 1024, 0, s>>>(B, K, out_tokens, tau, offsets, packed, status);
  return cudaGetLastError() == cudaSuccess ? SD_OK : SD_ERR_CUDA;
}

sd_status_t sd_uniforms(uint64_t seed, int32_t n, const int32_t *row, const int32_t *pos,
                        const int32_t *slot, double *out, void *stream) {
  if (n < 0) return SD_ERR_INVALID_ARG;
  if (n == 0) return SD_OK;
  if (!row || !pos || !slot || !out) return SD_ERR_INVALID_ARG;
  sd_uniforms_kernel<<<(n + 255) / 256, 256, 0, (cudaStream_t)stream>>>(seed, n, row, pos, slot,
                                                                        out);
  return cudaGetLastError() == cudaSuccess ? SD_OK : SD_ERR_CUDA;
}

size_t sd_verify_args_size(void) { return sizeof(sd_verify_args); }

const char *sd_version(void) { return "sdverify 0.2 (sm_103a)"; }

const char *sd_status_string(sd_status_t s) {
  switch (s) {
    case SD_OK: return "SD_OK";
    case SD_ERR_INVALID_ARG: return "SD_ERR_INVALID_ARG";
    case SD_ERR_UNSUPPORTED: return "SD_ERR_UNSUPPORTED";
    case SD_ERR_CUDA: return "SD_ERR_CUDA";
  }
  return "unknown";
}

}  // extern "C"
