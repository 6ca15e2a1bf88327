// GB300 (sm_103a) kernels of the speculative-decoding verify step.
//
// One thread-block cluster works on one (row b, position j) item at a time:
// its CTAs split the vocabulary into contiguous slices, bring their slice of
// target row j and draft row j into shared memory with 1-D TMA bulk copies
// (each logit read from HBM exactly once), reduce max / argmax / sum of
// exponentials per slice, and exchange the per-CTA partials over
// distributed shared memory.  Every CTA of the cluster then holds the same
// row statistics and takes the same decisions.  A position whose draft is
// rejected, and the bonus position K, draw their token right there from
// the slices still resident in shared memory (inverse CDF over the
// residual max(0, p - q) or over p), so no logit is read twice.  The item's
// owner CTA publishes its result to global scratch; the last item of a row
// to finish (an atomic counter, no spin-waits) runs that row's
// left-to-right accept scan, writes tau / the emitted tokens / the hit
// test, and the last row to finish packs all rows' tokens.  The kernel is
// persistent: clusters loop over items with a two-stage shared-memory
// pipeline so that the bulk copies of the next item overlap the reductions
// of the current one.
//
// Method sources (web pages, stated in prose there):
//  "What is speculative decoding" explainer (lotook.com): the four-stage
//    loop (greedy match; keep a token the target rates at least as high as
//    the draft, else keep it with the probability ratio; resample the first
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

#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <map>
#include <tuple>
#include <algorithm>

namespace cg = cooperative_groups;

namespace sdv {

constexpr int kMaxF = SD_MAX_FANOUT;
constexpr int kMaxK = SD_MAX_K;
constexpr int kMaxCS = 16;
constexpr int kCandCap = 512;           // top-F candidate buffer per CTA
constexpr int kThreads = 512;     // threads per CTA
constexpr unsigned kWaitSpins = 1u << 24;  // bounded mbarrier wait (~1 s with backoff)

enum Mode : int { kVerify = 0, kPredict = 1 };

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
  int32_t *row_counter;    // [B]   workspace
  int32_t *done_counter;   // [1]   workspace
  int32_t *pos_token;      // [B][K+1] workspace
  int8_t *pos_accept;      // [B][K+1] workspace
  uint64_t seed;
  int64_t row_base;
  int32_t B, K, V;
  int32_t mode;
  int32_t keys;            // build keys in this pass
  int32_t compact;         // pack tokens at the end
  int32_t n_keys_in, n_keys_out;
  int32_t cs, nstage, slice, region;
  int32_t n_items;
  int32_t fanout[kMaxK + 1];
  int32_t fan_off[kMaxK + 2];
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
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0u;
}

// Bounded wait on one phase of an mbarrier; false if it gave up.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity) {
  for (unsigned i = 0; i < kWaitSpins; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (i > 32) __nanosleep(64);
  }
  return false;
}

// 1-D TMA bulk copy global -> this CTA's shared memory, completion counted
// in bytes on the mbarrier.  dst, src and bytes are multiples of 16.
__device__ __forceinline__ void bulk_copy_g2s(void *dst, const void *src, uint32_t bytes,
                                              uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// 2^x on the special-function unit (x <= 0 here; results below 2^-126 flush
// to zero, far below anything that moves a sum of at least 1).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
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

struct Red {
  float f[32];
  int i[32];
  double d[32];
};

__device__ float block_max(float v, Red &r) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_max(v);
  if (lane == 0) r.f[w] = v;
  __syncthreads();
  float x = lane < nw ? r.f[lane] : -INFINITY;
  x = warp_max(x);
  __syncthreads();
  return x;
}
__device__ int block_min_i(int v, Red &r) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_min_i(v);
  if (lane == 0) r.i[w] = v;
  __syncthreads();
  int x = lane < nw ? r.i[lane] : INT32_MAX;
  x = warp_min_i(x);
  __syncthreads();
  return x;
}
// Sum in double, combined in a fixed order (warp tree, then warps in order).
__device__ double block_sum_d(double v, Red &r) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_sum_d(v);
  if (lane == 0) r.d[w] = v;
  __syncthreads();
  double x = lane < nw ? r.d[lane] : 0.0;
  x = warp_sum_d(x);
  __syncthreads();
  return x;
}

// --------------------------------------------------------- element types --
template <typename E>
struct Elt;
template <>
struct Elt<float> {
  static constexpr int kSize = 4;
  static constexpr int kPerVec = 4;
  static __device__ __forceinline__ void unpack(const uint4 &v, float *f) {
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
  }
  static __device__ __forceinline__ float load(const uint8_t *p) {
    return *reinterpret_cast<const float *>(p);
  }
  static __device__ __forceinline__ float load_global(const uint8_t *p) {
    return __ldg(reinterpret_cast<const float *>(p));
  }
  static __device__ __forceinline__ void store_neg_inf(uint8_t *p) {
    *reinterpret_cast<uint32_t *>(p) = 0xFF800000u;
  }
  static __device__ __forceinline__ void copy_elem(uint8_t *dst, const uint8_t *src) {
    *reinterpret_cast<uint32_t *>(dst) = __ldg(reinterpret_cast<const unsigned int *>(src));
  }
};
template <>
struct Elt<__nv_bfloat16> {
  static constexpr int kSize = 2;
  static constexpr int kPerVec = 8;
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
  static __device__ __forceinline__ float load(const uint8_t *p) {
    return __uint_as_float((uint32_t)(*reinterpret_cast<const uint16_t *>(p)) << 16);
  }
  static __device__ __forceinline__ float load_global(const uint8_t *p) {
    return __uint_as_float((uint32_t)__ldg(reinterpret_cast<const unsigned short *>(p)) << 16);
  }
  static __device__ __forceinline__ void store_neg_inf(uint8_t *p) {
    *reinterpret_cast<uint16_t *>(p) = (uint16_t)0xFF80u;
  }
  static __device__ __forceinline__ void copy_elem(uint8_t *dst, const uint8_t *src) {
    *reinterpret_cast<uint16_t *>(dst) = __ldg(reinterpret_cast<const unsigned short *>(src));
  }
};

// Where one CTA's slice [v0, v1) of one logit row sits in shared memory.
// The region mirrors the global 16-byte alignment of the slice: element
// v0 is at byte `hp` and vector q covers global bytes [g_first + 16q, +16).
// Bytes of the first/last vector outside the slice hold -inf.
struct Slice {
  int v0, v1;       // element range
  int hp;           // head pad in bytes
  int nvec;         // 16-byte vectors in the region
  __device__ __forceinline__ int first_elem(int q, int sz) const {
    return v0 + (q * 16 - hp) / sz;
  }
};

__device__ __forceinline__ Slice make_slice(const uint8_t *row, int v0, int v1, int sz) {
  Slice s;
  s.v0 = v0;
  s.v1 = v1;
  const uintptr_t a0 = (uintptr_t)(row + (int64_t)v0 * sz);
  const uintptr_t a1 = (uintptr_t)(row + (int64_t)v1 * sz);
  const uintptr_t gf = a0 & ~(uintptr_t)15, gl = (a1 + 15) & ~(uintptr_t)15;
  s.hp = (int)(a0 - gf);
  s.nvec = v1 > v0 ? (int)((gl - gf) / 16) : 0;
  return s;
}

// Issued by one thread: the bulk copy of the 16-byte-aligned interior of the
// slice, plain loads for the ragged head and tail, -inf in the pad bytes.
// Returns the bytes the bulk copy will deliver.
template <typename E>
__device__ uint32_t bulk_bytes(const uint8_t *row, const Slice &s) {
  constexpr int sz = Elt<E>::kSize;
  if (s.v1 <= s.v0) return 0;
  const uintptr_t a0 = (uintptr_t)(row + (int64_t)s.v0 * sz);
  const uintptr_t a1 = (uintptr_t)(row + (int64_t)s.v1 * sz);
  const uintptr_t lo = (a0 + 15) & ~(uintptr_t)15, hi = a1 & ~(uintptr_t)15;
  return hi > lo ? (uint32_t)(hi - lo) : 0u;
}

template <typename E>
__device__ void issue_slice(uint8_t *region, const uint8_t *row, const Slice &s, uint64_t *bar) {
  constexpr int sz = Elt<E>::kSize;
  if (s.v1 <= s.v0) return;
  const uintptr_t a0 = (uintptr_t)(row + (int64_t)s.v0 * sz);
  const uintptr_t a1 = (uintptr_t)(row + (int64_t)s.v1 * sz);
  const uintptr_t gf = a0 & ~(uintptr_t)15, gl = (a1 + 15) & ~(uintptr_t)15;
  const uintptr_t lo = (a0 + 15) & ~(uintptr_t)15, hi = a1 & ~(uintptr_t)15;
  uintptr_t plain_hi = a1;  // end of the head part loaded with plain loads
  if (hi > lo) {
    uint32_t off = (uint32_t)(lo - gf), bytes = (uint32_t)(hi - lo);
    const uint8_t *src = reinterpret_cast<const uint8_t *>(lo);
    // chunks of at most 64 KiB per instruction
    while (bytes > 0) {
      const uint32_t n = bytes > 65536u ? 65536u : bytes;
      bulk_copy_g2s(region + off, src, n, bar);
      off += n;
      src += n;
      bytes -= n;
    }
    plain_hi = lo;
    for (uintptr_t a = hi; a < a1; a += sz)
      Elt<E>::copy_elem(region + (a - gf), reinterpret_cast<const uint8_t *>(a));
  }
  for (uintptr_t a = a0; a < plain_hi; a += sz)
    Elt<E>::copy_elem(region + (a - gf), reinterpret_cast<const uint8_t *>(a));
  for (uintptr_t a = gf; a < a0; a += sz) Elt<E>::store_neg_inf(region + (a - gf));
  for (uintptr_t a = a1; a < gl; a += sz) Elt<E>::store_neg_inf(region + (a - gf));
}

// ------------------------------------------------------------ item layout --
struct Item {
  int b, j;
  float T;
  bool tvalid, sampled;   // temperature valid / T > 0
  int d;                  // drafted token at j (-1 at j == K)
  bool dvalid;
  bool need_t, need_1;    // target row j / second row (draft j or bonus)
  const uint8_t *trow, *row1;
  int fan;                // keys to build at this position (0 if none)
};

template <typename E>
__device__ __forceinline__ Item describe(const Params &P, int it) {
  constexpr int sz = Elt<E>::kSize;
  Item I;
  I.b = it / (P.K + 1);
  I.j = it - I.b * (P.K + 1);
  const float T = P.temps ? P.temps[I.b] : 0.f;
  I.T = T;
  I.tvalid = (T >= 0.f) && (T <= 3.4e38f);  // rejects NaN, negative, inf
  I.sampled = I.tvalid && T > 0.f;
  I.d = I.j < P.K ? P.tokens[(int64_t)I.b * P.K + I.j] : -1;
  I.dvalid = I.j < P.K ? (I.d >= 0 && I.d < P.V) : true;
  I.fan = P.keys ? P.fanout[I.j] : 0;
  const int64_t V = P.V;
  if (P.mode == kPredict) {
    I.need_t = false;
    I.trow = nullptr;
    if (I.j < P.K) {
      I.row1 = P.draft + ((int64_t)I.b * P.K + I.j) * V * sz;
      I.need_1 = I.fan > 0;
    } else {
      I.row1 = P.bonus ? P.bonus + (int64_t)I.b * V * sz : nullptr;
      I.need_1 = I.fan > 0 && P.bonus != nullptr;
    }
  } else {
    I.need_t = true;
    I.trow = P.target + ((int64_t)I.b * (P.K + 1) + I.j) * V * sz;
    if (I.j < P.K) {
      I.row1 = P.draft + ((int64_t)I.b * P.K + I.j) * V * sz;
      I.need_1 = I.sampled || I.fan > 0;
    } else {
      I.row1 = P.bonus ? P.bonus + (int64_t)I.b * V * sz : nullptr;
      I.need_1 = I.fan > 0 && P.bonus != nullptr;
    }
    if (!I.need_1) I.row1 = nullptr;
  }
  return I;
}

// ------------------------------------------------------- per-CTA partials --
struct alignas(16) Part {
  float mt;       // target slice max
  int at;         // first index of mt in the slice (INT32_MAX if none)
  double zt;      // sum 2^((l - mt) s) over the slice
  float ld;       // target logit of the drafted token (if in slice)
  int has_ld;
  float m1;       // second row: slice max
  double z1;      // second row: sum 2^((l - m1) s)
  float l1d;      // second row logit of the drafted token (if in slice)
  int has_l1d;
  int nc;         // top-F candidates found in the slice
  float cv[kMaxF];
  int ci[kMaxF];
  double s;       // mass of the sampling pass over the slice
};
static_assert(sizeof(Part) % 16 == 0, "Part is copied in 16-byte units");

// Decisions every CTA of a cluster derives identically from the partials.
struct Decision {
  float M, M1;
  double Zt, Z1;
  int amax;
  int accept;
  int sample;     // 0 none, 1 residual, 2 from p (bonus / empty residual)
  float s_hi, s_lo;
  float A, Bq;    // 1/Zt and 1/Z1 as floats (sampling pass weights)
  double t;       // u * S of the sampling pass
  int cstar;      // CTA that owns the sampled token
  double t_loc;   // target within the owning CTA's slice
  float ratio, p_d, q_d;
  int token;
  int owner;
};

struct Smem {
  uint64_t bar[2];
  Part part[2];
  Part peer[kMaxCS];      // local copies of the cluster's partials
  double zterm[kMaxCS], z1term[kMaxCS], sterm[kMaxCS];
  Red red;
  Decision dec;
  int cand_n;
  int found_thread;
  int tok;
  int flag_compact;
  int found_q;
};

// ----------------------------------------------------- slice reductions --
template <typename E>
__device__ __forceinline__ float slice_max(const uint8_t *reg, const Slice &s) {
  float m = -INFINITY;
  for (int q = threadIdx.x; q < s.nvec; q += blockDim.x) {
    float f[Elt<E>::kPerVec];
    Elt<E>::unpack(*reinterpret_cast<const uint4 *>(reg + 16 * q), f);
#pragma unroll
    for (int k = 0; k < Elt<E>::kPerVec; ++k) m = fmaxf(m, f[k]);
  }
  return m;
}

// first index (in [v0, v1)) of a value equal to target among this thread's vectors
template <typename E>
__device__ __forceinline__ int slice_first_eq(const uint8_t *reg, const Slice &s, float target) {
  constexpr int sz = Elt<E>::kSize;
  for (int q = threadIdx.x; q < s.nvec; q += blockDim.x) {
    float f[Elt<E>::kPerVec];
    Elt<E>::unpack(*reinterpret_cast<const uint4 *>(reg + 16 * q), f);
    const int e0 = s.first_elem(q, sz);
#pragma unroll
    for (int k = 0; k < Elt<E>::kPerVec; ++k) {
      const int e = e0 + k;
      if (f[k] == target && e >= s.v0 && e < s.v1) return e;
    }
  }
  return INT32_MAX;
}

// sum over the slice of 2^((l - m) s), s = s_hi + s_lo (s_lo >= 0 so that
// -inf logits give 2^-inf = 0 without inf - inf)
template <typename E>
__device__ __forceinline__ float slice_expsum(const uint8_t *reg, const Slice &s, float m,
                                              float s_hi, float s_lo) {
  float sum = 0.f, comp = 0.f;
  for (int q = threadIdx.x; q < s.nvec; q += blockDim.x) {
    float f[Elt<E>::kPerVec];
    Elt<E>::unpack(*reinterpret_cast<const uint4 *>(reg + 16 * q), f);
    float e[Elt<E>::kPerVec];
#pragma unroll
    for (int k = 0; k < Elt<E>::kPerVec; ++k) {
      const float dl = f[k] - m;
      e[k] = ex2(fmaf(dl, s_hi, dl * s_lo));
    }
#pragma unroll
    for (int w = Elt<E>::kPerVec / 2; w > 0; w >>= 1)
#pragma unroll
      for (int k = 0; k < w; ++k) e[k] += e[k + w];
    kahan_add(sum, comp, e[0]);
  }
  return sum;
}

// Weights of the sampling pass for the Elt::kPerVec elements of target
// vector q: residual max(0, 2^x A - 2^y Bq) (mode 1) or 2^x A (mode 2),
// x = (l - M) s, y = (l' - M1) s.  Elements outside the slice weigh 0.
template <typename E>
__device__ __forceinline__ void sample_weights(const uint8_t *rt, const Slice &st,
                                               const uint8_t *r1, const Slice &s1, int q,
                                               const Decision &D, float *w) {
  constexpr int sz = Elt<E>::kSize, N = Elt<E>::kPerVec;
  float f[N];
  Elt<E>::unpack(*reinterpret_cast<const uint4 *>(rt + 16 * q), f);
#pragma unroll
  for (int k = 0; k < N; ++k) {
    const float dl = f[k] - D.M;
    w[k] = ex2(fmaf(dl, D.s_hi, dl * D.s_lo)) * D.A;
  }
  if (D.sample == 1) {
    float g[N];
    if (s1.hp == st.hp) {
      Elt<E>::unpack(*reinterpret_cast<const uint4 *>(r1 + 16 * q), g);
    } else {
      const int e0 = st.first_elem(q, sz);
#pragma unroll
      for (int k = 0; k < N; ++k) {
        const int e = e0 + k;
        g[k] = (e >= s1.v0 && e < s1.v1) ? Elt<E>::load(r1 + s1.hp + (e - s1.v0) * sz)
                                         : -INFINITY;
      }
    }
#pragma unroll
    for (int k = 0; k < N; ++k) {
      const float dl = g[k] - D.M1;
      const float qv = ex2(fmaf(dl, D.s_hi, dl * D.s_lo)) * D.Bq;
      w[k] = fmaxf(0.f, w[k] - qv);
    }
  }
  const int e0 = st.first_elem(q, sz);
#pragma unroll
  for (int k = 0; k < N; ++k) {
    const int e = e0 + k;
    if (e < st.v0 || e >= st.v1) w[k] = 0.f;
  }
}

// ------------------------------------------------------------- top-F keys --
// Ordered key of (value, index): larger value first, then lower index.
__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

// Bitonic sort of one value per lane, descending; returns this lane's value.
__device__ __forceinline__ float warp_sort_desc(float v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const float o = __shfl_xor_sync(0xffffffffu, v, j);
      const bool up = ((lane & k) == 0);         // block sorted descending
      const bool lower = ((lane & j) == 0);
      v = (lower == up) ? fmaxf(v, o) : fminf(v, o);
    }
  }
  return v;
}

// Top-`fan` (value desc, index asc) of the slice excluding index `excl` and
// -inf values.  m_thread: this thread's slice max.  Result left in
// sm.part[par].cv/ci/nc by thread 0.
template <typename E>
__device__ void slice_topf(const uint8_t *reg, const Slice &s, float m_thread, int fan, int excl,
                           float *cand_v, int *cand_i, Smem &sm, Part &out) {
  constexpr int sz = Elt<E>::kSize, N = Elt<E>::kPerVec;
  const int lane = threadIdx.x & 31;
  // threshold: the (fan+1)-th largest thread maximum of the best warp is a
  // lower bound of the (fan+1)-th largest value of the slice, so every
  // top-fan element other than `excl` is >= theta.
  const float sorted = warp_sort_desc(m_thread);
  float th = __shfl_sync(0xffffffffu, sorted, fan);  // fan <= kMaxF < 32
  th = block_max(th, sm.red);
  if (threadIdx.x == 0) sm.cand_n = 0;
  __syncthreads();
  for (int q = threadIdx.x; q < s.nvec; q += blockDim.x) {
    float f[N];
    Elt<E>::unpack(*reinterpret_cast<const uint4 *>(reg + 16 * q), f);
    const int e0 = s.first_elem(q, sz);
#pragma unroll
    for (int k = 0; k < N; ++k) {
      if (f[k] >= th && f[k] > -INFINITY) {
        const int e = e0 + k;
        if (e != excl && e >= s.v0 && e < s.v1) {
          const int slot = atomicAdd(&sm.cand_n, 1);
          if (slot < kCandCap) {
            cand_v[slot] = f[k];
            cand_i[slot] = e;
          }
        }
      }
    }
  }
  __syncthreads();
  const int n = sm.cand_n;
  if (n > kCandCap) {
    // many ties at the threshold: exact selection by repeated block argmax
    float last_v = INFINITY;
    int last_i = -1;
    for (int r = 0; r < fan; ++r) {
      float bv = -INFINITY;
      int bi = INT32_MAX;
      for (int q = threadIdx.x; q < s.nvec; q += blockDim.x) {
        float f[N];
        Elt<E>::unpack(*reinterpret_cast<const uint4 *>(reg + 16 * q), f);
        const int e0 = s.first_elem(q, sz);
#pragma unroll
        for (int k = 0; k < N; ++k) {
          const int e = e0 + k;
          if (e == excl || e < s.v0 || e >= s.v1 || !(f[k] > -INFINITY)) continue;
          if (!better(last_v, last_i, f[k], e) || (f[k] == last_v && e == last_i)) continue;
          if (better(f[k], e, bv, bi)) {
            bv = f[k];
            bi = e;
          }
        }
      }
      const float mv = block_max(bv, sm.red);
      const int mi = block_min_i(bv == mv ? bi : INT32_MAX, sm.red);
      if (threadIdx.x == 0) {
        if (mv > -INFINITY && mi != INT32_MAX) {
          out.cv[r] = mv;
          out.ci[r] = mi;
          out.nc = r + 1;
        }
      }
      last_v = mv;
      last_i = mi;
      if (!(mv > -INFINITY) || mi == INT32_MAX) break;
    }
    __syncthreads();
    return;
  }
  // warp 0 selects the best `fan` candidates
  if (threadIdx.x < 32) {
    int taken = 0;  // bit r set: this lane's r-th candidate already chosen
    int nc = 0;
    for (int r = 0; r < fan; ++r) {
      float bv = -INFINITY;
      int bi = INT32_MAX, bslot = -1;
      for (int c = lane, t = 0; c < n; c += 32, ++t) {
        if (taken & (1 << t)) continue;
        if (better(cand_v[c], cand_i[c], bv, bi)) {
          bv = cand_v[c];
          bi = cand_i[c];
          bslot = t;
        }
      }
      float wv = bv;
      int wi = bi;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, wv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, wi, o);
        if (better(ov, oi, wv, wi)) {
          wv = ov;
          wi = oi;
        }
      }
      if (wi == INT32_MAX) break;
      if (bi == wi && bslot >= 0) taken |= 1 << bslot;
      if (lane == 0) {
        out.cv[r] = wv;
        out.ci[r] = wi;
      }
      nc = r + 1;
    }
    if (lane == 0) out.nc = nc;
  }
  __syncthreads();
}

// --------------------------------------------------------- row finalizer --
// Runs on one thread once all K+1 positions of row b have published.
__device__ void finalize_row(const Params &P, int b) {
  const int K = P.K;
  const float T = P.temps[b];
  const bool tvalid = (T >= 0.f) && (T <= 3.4e38f);
  bool dvalid = true;
  for (int j = 0; j < K; ++j) {
    const int d = P.tokens[(int64_t)b * K + j];
    if (d < 0 || d >= P.V) dvalid = false;
  }
  int32_t *out = P.out_tokens + (int64_t)b * (K + 1);
  int32_t *ptok = P.pos_token + (int64_t)b * (K + 1);
  int8_t *pacc = P.pos_accept + (int64_t)b * (K + 1);
  if (!tvalid || !dvalid) {
    for (int j = 0; j <= K; ++j) {  // leave the scratch zeroed
      ptok[j] = 0;
      pacc[j] = 0;
    }
    for (int j = 0; j <= K; ++j) out[j] = -1;
    P.num_accepted[b] = 0;
    P.tau[b] = 0;
    if (P.hit) P.hit[b] = 0;
    if (P.status) atomicOr(P.status, (tvalid ? 0 : (int)SD_STATUS_BAD_TEMP) |
                                         (dvalid ? 0 : (int)SD_STATUS_BAD_TOKEN));
    return;
  }
  int n_acc = K;
  const int8_t *acc = P.pos_accept + (int64_t)b * (K + 1);
  for (int j = 0; j < K; ++j) {
    if (__ldcg(reinterpret_cast<const signed char *>(acc + j)) == 0) {
      n_acc = j;
      break;
    }
  }
  const int tok = __ldcg(ptok + n_acc);
  for (int j = 0; j <= K; ++j) {  // leave the scratch zeroed for the next call
    ptok[j] = 0;
    pacc[j] = 0;
  }
  for (int j = 0; j < n_acc; ++j) out[j] = P.tokens[(int64_t)b * K + j];
  out[n_acc] = tok;
  for (int j = n_acc + 1; j <= K; ++j) out[j] = -1;
  P.num_accepted[b] = n_acc;
  P.tau[b] = n_acc + 1;
  if (P.hit) {
    int h = 0;
    if (P.keys && P.keys_out) {
      const int32_t *kb = P.keys_out + (int64_t)b * P.n_keys_out * 2;
      for (int k = 0; k < P.n_keys_out; ++k)
        if (__ldcg(kb + 2 * k) == n_acc && __ldcg(kb + 2 * k + 1) == tok) h = 1;
    } else if (P.keys_in) {
      const int32_t *kb = P.keys_in + (int64_t)b * P.n_keys_in * 2;
      for (int k = 0; k < P.n_keys_in; ++k)
        if (kb[2 * k] == n_acc && kb[2 * k + 1] == tok) h = 1;
    }
    P.hit[b] = (uint8_t)h;
  }
}

// Exclusive scan of tau and packing of out_tokens, one CTA.  `cg_loads`
// reads values written by other CTAs of the same grid through L2.
__device__ void compact_block(int B, int K, const int32_t *out_tokens, const int32_t *tau,
                              int32_t *offsets, int32_t *packed, int32_t *status, bool cg_loads,
                              Red &red) {
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
    if (lane == 31) red.i[w] = x;
    __syncthreads();
    if (w == 0) {
      int v = lane < nw ? red.i[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += y;
      }
      if (lane < nw) red.i[lane] = v;  // inclusive warp totals
    }
    __syncthreads();
    const int excl = carry + (w > 0 ? red.i[w - 1] : 0) + x - t;
    if (b < B) {
      offsets[b] = excl;
      const int32_t *src = out_tokens + (int64_t)b * (K + 1);
      for (int i = 0; i < t; ++i) packed[excl + i] = cg_loads ? __ldcg(src + i) : src[i];
    }
    carry += red.i[nw - 1];
    __syncthreads();
  }
  if (threadIdx.x == 0) offsets[B] = carry;
}

// ------------------------------------------------------------ the kernel --
template <typename E>
__global__ void __launch_bounds__(kThreads, 1) sd_verify_kernel(const __grid_constant__ Params P) {
  constexpr int sz = Elt<E>::kSize, NV = Elt<E>::kPerVec;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int cs = P.cs;
  const int cid = blockIdx.x / cs;
  const int ncl = gridDim.x / cs;

  __shared__ Smem sm;
  extern __shared__ __align__(128) uint8_t dyn[];
  // dynamic layout: stages (2 regions each), csum, candidate buffer
  uint8_t *stage_base[2] = {dyn, dyn + (P.nstage > 1 ? 2 * P.region : 0)};
  float *csum = reinterpret_cast<float *>(dyn + P.nstage * 2 * P.region);
  const int nvec_max = P.region / 16;
  float *cand_v = csum + nvec_max;
  int *cand_i = reinterpret_cast<int *>(cand_v + kCandCap);

  const int v0 = min(rank * P.slice, P.V);
  const int v1 = min(v0 + P.slice, P.V);

  if (threadIdx.x == 0) {
    mbar_init(&sm.bar[0], 1);
    mbar_init(&sm.bar[1], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    sm.flag_compact = 0;
  }
  __syncthreads();

  uint32_t phase[2] = {0u, 0u};
  bool timed_out = false;
  int late_stage = -1;       // stage whose bounded wait gave up
  uint32_t late_parity = 0u;

  auto issue = [&](int k) {
    // thread 0 only: loads of the k-th item of this cluster into stage k % nstage
    const int it = cid + k * ncl;
    const Item I = describe<E>(P, it);
    uint8_t *sb = stage_base[k % P.nstage];
    uint64_t *bar = &sm.bar[k % P.nstage];
    Slice st{}, s1{};
    uint32_t tx = 0;
    if (I.need_t) {
      st = make_slice(I.trow, v0, v1, sz);
      tx += bulk_bytes<E>(I.trow, st);
    }
    if (I.need_1) {
      s1 = make_slice(I.row1, v0, v1, sz);
      tx += bulk_bytes<E>(I.row1, s1);
    }
    // the stage was last read through the generic proxy; order those reads
    // before the bulk copies (async proxy) overwrite it
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    mbar_arrive_expect_tx(bar, tx);
    if (I.need_t) issue_slice<E>(sb, I.trow, st, bar);
    if (I.need_1) issue_slice<E>(sb + P.region, I.row1, s1, bar);
  };

  const int n_mine = cid < P.n_items ? (P.n_items - 1 - cid) / ncl + 1 : 0;
  if (threadIdx.x == 0 && n_mine > 0) issue(0);

  for (int k = 0; k < n_mine; ++k) {
    const int it = cid + k * ncl;
    const int par = k & 1;
    const int stg = k % P.nstage;
    if (threadIdx.x == 0) {
      if (P.nstage > 1 && k + 1 < n_mine) issue(k + 1);
      else if (P.nstage == 1 && k > 0) issue(k);
    }
    if (!mbar_wait_bounded(&sm.bar[stg], phase[stg])) {
      timed_out = true;
      late_stage = stg;
      late_parity = phase[stg];
    }
    phase[stg] ^= 1u;
    __syncthreads();

    const Item I = describe<E>(P, it);
    const uint8_t *rt = stage_base[stg];
    const uint8_t *r1 = stage_base[stg] + P.region;
    Slice st{}, s1{};
    if (I.need_t) st = make_slice(I.trow, v0, v1, sz);
    if (I.need_1) s1 = make_slice(I.row1, v0, v1, sz);
    const double s_d = I.sampled ? 1.4426950408889634 / (double)I.T : 0.0;
    // s = s_hi + s_lo with s_lo > 0, so that (-inf) * s_lo stays -inf
    const float s_hi = __double2float_rd(s_d);
    const float s_lo = fmaxf((float)(s_d - (double)s_hi), 1.17549435e-38f);
    Part &mine = sm.part[par];

    // ---- target row j: max, argmax, sum of exponentials, logit of d_j
    if (I.need_t) {
      const float mt = slice_max<E>(rt, st);
      const float Mc = block_max(mt, sm.red);
      int at = mt == Mc ? slice_first_eq<E>(rt, st, Mc) : INT32_MAX;
      at = block_min_i(at, sm.red);
      double zc = 0.0;
      if (I.sampled) zc = block_sum_d((double)slice_expsum<E>(rt, st, Mc, s_hi, s_lo), sm.red);
      if (threadIdx.x == 0) {
        mine.mt = Mc;
        mine.at = at;
        mine.zt = zc;
        mine.has_ld = 0;
        mine.ld = -INFINITY;
        if (I.j < P.K && I.dvalid && I.d >= st.v0 && I.d < st.v1) {
          mine.has_ld = 1;
          mine.ld = Elt<E>::load(rt + st.hp + (I.d - st.v0) * sz);
        }
      }
    }
    // ---- second row (draft row j, or the bonus draft row at j == K)
    if (threadIdx.x == 0) {
      mine.nc = 0;
      mine.has_l1d = 0;
      mine.m1 = -INFINITY;
      mine.z1 = 0.0;
      if (!I.need_t) {
        mine.mt = -INFINITY;
        mine.at = INT32_MAX;
        mine.zt = 0.0;
        mine.has_ld = 0;
      }
    }
    if (I.need_1) {
      const float m1 = slice_max<E>(r1, s1);
      const float M1c = block_max(m1, sm.red);
      double z1 = 0.0;
      if (I.sampled && I.j < P.K && P.mode == kVerify)
        z1 = block_sum_d((double)slice_expsum<E>(r1, s1, M1c, s_hi, s_lo), sm.red);
      if (threadIdx.x == 0) {
        mine.m1 = M1c;
        mine.z1 = z1;
        if (I.j < P.K && I.dvalid && I.d >= s1.v0 && I.d < s1.v1) {
          mine.has_l1d = 1;
          mine.l1d = Elt<E>::load(r1 + s1.hp + (I.d - s1.v0) * sz);
        }
      }
      if (I.fan > 0) {
        __syncthreads();
        slice_topf<E>(r1, s1, m1, I.fan, I.j < P.K ? I.d : -1, cand_v, cand_i, sm, mine);
      }
    }
    cluster.sync();

    // ---- gather the cluster's partials (one thread per peer, 16-byte loads)
    if ((int)threadIdx.x < cs) {
      const int4 *src =
          reinterpret_cast<const int4 *>(cluster.map_shared_rank(&sm.part[par], (int)threadIdx.x));
      int4 *dst = reinterpret_cast<int4 *>(&sm.peer[threadIdx.x]);
#pragma unroll
      for (int w = 0; w < (int)(sizeof(Part) / 16); ++w) dst[w] = src[w];
    }
    __syncthreads();
    // ---- combine them (same order in every CTA, so every CTA decides alike)
    if (threadIdx.x == 0) {
      float M = -INFINITY, M1 = -INFINITY;
      for (int c = 0; c < cs; ++c) {
        M = fmaxf(M, sm.peer[c].mt);
        M1 = fmaxf(M1, sm.peer[c].m1);
      }
      sm.dec.M = M;
      sm.dec.M1 = M1;
    }
    __syncthreads();
    if ((int)threadIdx.x < cs) {
      const Part &pc = sm.peer[threadIdx.x];
      sm.zterm[threadIdx.x] = (I.need_t && I.sampled && pc.zt > 0.0)
                                  ? pc.zt * exp2(((double)pc.mt - (double)sm.dec.M) * s_d)
                                  : 0.0;
      sm.z1term[threadIdx.x] = (I.need_1 && I.sampled && pc.z1 > 0.0)
                                   ? pc.z1 * exp2(((double)pc.m1 - (double)sm.dec.M1) * s_d)
                                   : 0.0;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      Decision D;
      D.s_hi = s_hi;
      D.s_lo = s_lo;
      D.accept = 0;
      D.sample = 0;
      D.token = -1;
      D.owner = 0;
      D.ratio = NAN;
      D.p_d = NAN;
      D.q_d = NAN;
      D.M = sm.dec.M;
      D.M1 = sm.dec.M1;
      D.Zt = 0.0;
      D.Z1 = 0.0;
      float ld = -INFINITY, l1d = -INFINITY;
      int amax = INT32_MAX;
      for (int c = 0; c < cs; ++c) {
        const Part &pc = sm.peer[c];
        if (I.need_t) {
          if (amax == INT32_MAX && pc.mt == D.M && pc.at != INT32_MAX) amax = pc.at;
          D.Zt += sm.zterm[c];
          if (pc.has_ld) ld = pc.ld;
        }
        if (I.need_1) {
          D.Z1 += sm.z1term[c];
          if (pc.has_l1d) l1d = pc.l1d;
        }
      }
      D.amax = amax == INT32_MAX ? 0 : amax;
      if (P.mode == kVerify) {
        if (I.j < P.K) {
          if (!I.sampled) {
            D.accept = (I.dvalid && I.d == D.amax) ? 1 : 0;
          } else if (I.dvalid) {
            const double pd = exp2(((double)ld - (double)D.M) * s_d) / D.Zt;
            const double qd = exp2(((double)l1d - (double)D.M1) * s_d) / D.Z1;
            const double r = qd > 0.0 ? pd / qd : INFINITY;
            const double u = uniform_u(P.seed, P.row_base + I.b, I.j, 0);
            D.accept = (u <= r) ? 1 : 0;
            D.ratio = (float)r;
            D.p_d = (float)pd;
            D.q_d = (float)qd;
          }
        }
        if (I.sampled && I.dvalid) {
          if (I.j == P.K) D.sample = 2;
          else if (!D.accept) D.sample = 1;
        }
        if (!I.sampled) D.token = D.amax;
        D.A = (float)(1.0 / D.Zt);
        D.Bq = I.j < P.K && I.sampled ? (float)(1.0 / D.Z1) : 0.f;
      }
      sm.dec = D;
    }
    __syncthreads();

    // ---- sampling pass: residual at a rejection, or p at the bonus position
    if (sm.dec.sample != 0) {
      for (int attempt = 0; attempt < 2; ++attempt) {
        const Decision &D = sm.dec;
        float tsum = 0.f, tcomp = 0.f;
        for (int q = threadIdx.x; q < st.nvec; q += blockDim.x) {
          float w[NV];
          sample_weights<E>(rt, st, r1, s1, q, D, w);
#pragma unroll
          for (int h = NV / 2; h > 0; h >>= 1)
#pragma unroll
            for (int k2 = 0; k2 < h; ++k2) w[k2] += w[k2 + h];
          csum[q] = w[0];
          kahan_add(tsum, tcomp, w[0]);
        }
        const double Sc = block_sum_d((double)tsum, sm.red);
        if (threadIdx.x == 0) mine.s = Sc;
        cluster.sync();
        if ((int)threadIdx.x < cs)
          sm.sterm[threadIdx.x] = cluster.map_shared_rank(&sm.part[par], (int)threadIdx.x)->s;
        __syncthreads();
        if (threadIdx.x == 0) {
          Decision &Dw = sm.dec;
          double S = 0.0;
          const double *pre = sm.sterm;
          for (int c = 0; c < cs; ++c) S += pre[c];
          if (S > 0.0 || Dw.sample == 2) {
            const double u = uniform_u(P.seed, P.row_base + I.b, I.j, 1);
            const double t = u * S;
            int cstar = -1, last_pos = -1;
            double acc = 0.0, acc_star = 0.0;
            for (int c = 0; c < cs; ++c) {
              if (pre[c] > 0.0) {
                last_pos = c;
                if (cstar < 0 && acc + pre[c] > t) {
                  cstar = c;
                  acc_star = acc;
                }
              }
              acc += pre[c];
            }
            if (cstar < 0) {  // rounding pushed t past the total
              cstar = last_pos < 0 ? 0 : last_pos;
              acc_star = 0.0;
              for (int c = 0; c < cstar; ++c) acc_star += pre[c];
            }
            Dw.t = t;
            Dw.cstar = cstar;
            Dw.t_loc = t - acc_star;
            Dw.owner = cstar;
            sm.found_thread = 0;  // non-zero: retry
          } else {
            // empty residual: draw from p instead
            Dw.sample = 2;
            sm.found_thread = 1;
          }
        }
        __syncthreads();
        if (sm.found_thread == 0) break;
        // all CTAs retry with mode 2 (uniform decision: same S everywhere)
        cluster.sync();
      }
      // inverse CDF inside the owning CTA
      const Decision &D = sm.dec;
      if (rank == D.cstar) {
        const int nt = blockDim.x;
        const int per = (st.nvec + nt - 1) / nt;
        const int q0 = min(threadIdx.x * per, st.nvec), q1 = min(q0 + per, st.nvec);
        double mysum = 0.0;
        for (int q = q0; q < q1; ++q) mysum += (double)csum[q];
        // exclusive block scan of mysum (double)
        const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
        double x = mysum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const double y = __shfl_up_sync(0xffffffffu, x, o);
          if (lane >= o) x += y;
        }
        if (lane == 31) sm.red.d[w] = x;
        __syncthreads();
        if (w == 0) {
          double v = lane < nw ? sm.red.d[lane] : 0.0;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const double y = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += y;
          }
          if (lane < nw) sm.red.d[lane] = v;
        }
        __syncthreads();
        const double pre = (w > 0 ? sm.red.d[w - 1] : 0.0) + x - mysum;
        const bool crosses = mysum > 0.0 && pre + mysum > D.t_loc;
        int first = block_min_i(crosses ? (int)threadIdx.x : INT32_MAX, sm.red);
        if (first == INT32_MAX) first = -block_min_i(mysum > 0.0 ? -(int)threadIdx.x : INT32_MAX, sm.red);
        if (first == INT32_MAX || first < 0) first = 0;
        if ((int)threadIdx.x == first) {
          double cum = pre;
          int qs = -1, qlast = -1;
          for (int q = q0; q < q1; ++q) {
            if (csum[q] > 0.f) qlast = q;
            if (qs < 0 && csum[q] > 0.f && cum + (double)csum[q] > D.t_loc) qs = q;
            if (qs < 0) cum += (double)csum[q];
          }
          if (qs < 0) {
            qs = qlast;
            cum = pre;
            for (int q = q0; q < qs; ++q) cum += (double)csum[q];
          }
          int tok = -1, klast = -1;
          if (qs >= 0) {
            float wv[NV];
            sample_weights<E>(rt, st, r1, s1, qs, D, wv);
            const int e0 = st.first_elem(qs, sz);
            double c2 = cum;
            for (int k2 = 0; k2 < NV; ++k2) {
              if (wv[k2] > 0.f) {
                klast = e0 + k2;
                if (tok < 0 && c2 + (double)wv[k2] > D.t_loc) tok = e0 + k2;
                c2 += (double)wv[k2];
              }
            }
            if (tok < 0) tok = klast;
          }
          if (tok < 0) tok = D.amax;  // nothing positive in this slice (degenerate)
          sm.tok = tok;
        }
        __syncthreads();
        if (threadIdx.x == 0) sm.dec.token = sm.tok;
      }
    }
    __syncthreads();

    // ---- publish (owner CTA): per-position results, keys, counters
    const Decision &D = sm.dec;
    if (rank == D.owner && threadIdx.x == 0) {
      const int64_t pk = (int64_t)I.b * (P.K + 1) + I.j;
      if (P.mode == kVerify) {
        if (I.j < P.K) P.pos_accept[pk] = (int8_t)D.accept;
        P.pos_token[pk] = D.token;
        if (P.argmax_out) P.argmax_out[pk] = D.amax;
        if (I.j < P.K && I.sampled) {
          const int64_t pj = (int64_t)I.b * P.K + I.j;
          if (P.ratio_out) P.ratio_out[pj] = D.ratio;
          if (P.p_out) P.p_out[pj] = D.p_d;
          if (P.q_out) P.q_out[pj] = D.q_d;
        }
      }
      if (I.fan > 0 && P.keys_out) {
        // merge the cluster's candidate lists
        float lv = INFINITY;
        int li = -1;
        int32_t *kout = P.keys_out + ((int64_t)I.b * P.n_keys_out + P.fan_off[I.j]) * 2;
        for (int r = 0; r < I.fan; ++r) {
          float bv = -INFINITY;
          int bi = INT32_MAX;
          if (I.need_1) {
            for (int c = 0; c < cs; ++c) {
              const Part *pc = &sm.peer[c];
              for (int x2 = 0; x2 < pc->nc; ++x2) {
                const float v = pc->cv[x2];
                const int ix = pc->ci[x2];
                if (better(lv, li, v, ix) && !(v == lv && ix == li) && better(v, ix, bv, bi)) {
                  bv = v;
                  bi = ix;
                }
              }
            }
          }
          if (bi == INT32_MAX) {
            kout[2 * r] = -1;
            kout[2 * r + 1] = -1;
          } else {
            kout[2 * r] = I.j;
            kout[2 * r + 1] = bi;
            lv = bv;
            li = bi;
          }
        }
      }
      if (P.mode == kVerify) {
        __threadfence();
        const int old = atomicAdd(&P.row_counter[I.b], 1);
        if (old == P.K) {
          __threadfence();
          finalize_row(P, I.b);
          P.row_counter[I.b] = 0;
          if (P.compact) {
            __threadfence();
            const int done = atomicAdd(P.done_counter, 1);
            if (done == P.B - 1) {
              __threadfence();
              sm.flag_compact = 1;
            }
          }
        }
      }
    }
    __syncthreads();
    if (sm.flag_compact) {
      compact_block(P.B, P.K, P.out_tokens, P.tau, P.offsets, P.packed, P.status, true, sm.red);
      if (threadIdx.x == 0) {
        *P.done_counter = 0;
        sm.flag_compact = 0;
      }
      __syncthreads();
    }
  }

  // Every issued copy was waited for in the loop; after a wait that gave up,
  // wait once more (bounded) so that no copy is in flight at exit.
  if (timed_out && threadIdx.x == 0) {
    (void)mbar_wait_bounded(&sm.bar[late_stage], late_parity);
    if (P.status) atomicOr(P.status, (int)SD_STATUS_TIMEOUT);
  }
  // peers may still read this CTA's partials
  cluster.sync();
}

__global__ void sd_compact_kernel(int B, int K, const int32_t *out_tokens, const int32_t *tau,
                                  int32_t *offsets, int32_t *packed, int32_t *status) {
  __shared__ Red red;
  compact_block(B, K, out_tokens, tau, offsets, packed, status, false, red);
}

__global__ void sd_uniforms_kernel(uint64_t seed, int n, const int32_t *row, const int32_t *pos,
                                   const int32_t *slot, double *out) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) out[i] = uniform_u(seed, row[i], pos[i], slot[i]);
}

// ------------------------------------------------------------------- host --
struct Plan {
  int cs, nstage, nt, slice, region, smem, clusters;
};

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct WsLayout {
  size_t done, row_counter, pos_token, pos_accept, total;
};
static WsLayout ws_layout(int B, int K) {
  WsLayout L;
  const size_t n = (size_t)B * (size_t)(K + 1);
  L.done = 0;
  L.row_counter = 16;
  L.pos_token = align_up(L.row_counter + 4 * (size_t)B, 16);
  L.pos_accept = align_up(L.pos_token + 4 * n, 16);
  L.total = align_up(L.pos_accept + n, 256);
  return L;
}

static const size_t kDynSmemCap = 227 * 1024 - sizeof(Smem) - 256;

template <typename E>
static void *kernel_ptr() {
  static std::once_flag once;
  void *fn = (void *)sd_verify_kernel<E>;
  std::call_once(once, [fn] {
    cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDynSmemCap);
    cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    cudaGetLastError();
  });
  return fn;
}

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

static size_t smem_bytes(int nstage, int region, bool cand) {
  size_t b = (size_t)nstage * 2 * region;      // stages
  b += (size_t)(region / 16) * 4;              // csum
  b += (size_t)kCandCap * 8;                   // candidates (always reserved)
  (void)cand;
  return align_up(b, 128);
}

// Resident clusters for a configuration (cached).
static int active_clusters(void *fn, int cs, int nt, size_t smem) {
  static std::mutex mu;
  static std::map<std::tuple<void *, int, int, size_t>, int> cache;
  std::lock_guard<std::mutex> g(mu);
  auto key = std::make_tuple(fn, cs, nt, smem);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cs * 64, 1, 1);
  cfg.blockDim = dim3(nt, 1, 1);
  cfg.dynamicSmemBytes = smem;
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
  cache[key] = n;
  return n;
}

template <typename E>
static bool make_plan(int items, int V, int rows_per_item, Plan &pl) {
  constexpr int sz = Elt<E>::kSize;
  (void)rows_per_item;
  void *fn = kernel_ptr<E>();
  const int nt = kThreads;
  const int force_cs = env_int("SDV_CS", 0);
  const int force_ns = env_int("SDV_NSTAGE", 0);
  const size_t smem_cap = kDynSmemCap;
  const int sms = sm_count();
  int best_cs = -1, best_ns = 1;
  double best_cost = 1e300;
  for (int cs = 1; cs <= kMaxCS; cs <<= 1) {
    if (force_cs && cs != force_cs) continue;
    const int slice = (int)align_up((size_t)((V + cs - 1) / cs), 16);
    const int region = (int)align_up((size_t)slice * sz + 32, 128);
    for (int ns = 1; ns <= 2; ++ns) {
      if (force_ns && ns != force_ns) continue;
      const size_t smem = smem_bytes(ns, region, true);
      if (smem > smem_cap) continue;
      const int ac = active_clusters(fn, cs, nt, smem);
      if (ac <= 0) continue;
      // cost model: waves of items over resident clusters, each item's
      // slice streamed at the SM's share of bandwidth; a single stage
      // cannot overlap the next item's copy with this item's reductions.
      const double waves = (double)((items + ac - 1) / ac);
      const double per_item = (double)slice * sz * 2.0;  // bytes per CTA per item
      const double active_frac = (double)std::min(items, ac) * cs / (double)sms;
      double cost = waves * per_item * (ns == 1 && waves > 1 ? 1.8 : 1.0) /
                    std::min(1.0, std::max(active_frac, 1e-3));
      cost += waves * 3000.0;  // per-item fixed latency (syncs), in byte units
      if (cost < best_cost * 0.999) {
        best_cost = cost;
        best_cs = cs;
        best_ns = ns;
      }
    }
  }
  if (best_cs < 0) return false;
  pl.cs = best_cs;
  pl.nstage = best_ns;
  pl.nt = nt;
  pl.slice = (int)align_up((size_t)((V + best_cs - 1) / best_cs), 16);
  pl.region = (int)align_up((size_t)pl.slice * sz + 32, 128);
  pl.smem = (int)smem_bytes(pl.nstage, pl.region, true);
  const int ac = active_clusters(fn, pl.cs, nt, pl.smem);
  pl.clusters = std::max(1, std::min(items, ac));
  return true;
}

template <typename E>
static sd_status_t launch(Params &P, cudaStream_t stream) {
  Plan pl;
  const int rows = 2;
  if (!make_plan<E>(P.n_items, P.V, rows, pl)) return SD_ERR_UNSUPPORTED;
  P.cs = pl.cs;
  P.nstage = pl.nstage;
  P.slice = pl.slice;
  P.region = pl.region;
  void *fn = kernel_ptr<E>();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(pl.clusters * pl.cs, 1, 1);
  cfg.blockDim = dim3(pl.nt, 1, 1);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = pl.cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (env_int("SDV_VERBOSE", 0))
    fprintf(stderr, "sd_verify plan: mode=%d items=%d cs=%d nstage=%d nt=%d slice=%d smem=%d clusters=%d\n",
            P.mode, P.n_items, pl.cs, pl.nstage, pl.nt, pl.slice, pl.smem, pl.clusters);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, (void (*)(const Params))fn, P);
  if (e != cudaSuccess) {
    fprintf(stderr, "sd_verify launch failed: %s\n", cudaGetErrorString(e));
    return SD_ERR_CUDA;
  }
  return SD_OK;
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
  return ws_layout(B, K).total;
}

sd_status_t sd_verify(const sd_verify_args *a, void *stream) {
  if (!a) return SD_ERR_INVALID_ARG;
  if (a->B < 0 || a->K < 0 || a->K > SD_MAX_K || a->V < 1 || a->V > SD_MAX_V)
    return SD_ERR_INVALID_ARG;
  if (a->dtype != SD_F32 && a->dtype != SD_BF16) return SD_ERR_INVALID_ARG;
  if ((int64_t)a->B * (a->K + 1) > INT32_MAX) return SD_ERR_INVALID_ARG;
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
  const WsLayout L = ws_layout(a->B, a->K);
  uint8_t *ws = (uint8_t *)a->workspace;
  P.done_counter = (int32_t *)(ws + L.done);
  P.row_counter = (int32_t *)(ws + L.row_counter);
  P.pos_token = (int32_t *)(ws + L.pos_token);
  P.pos_accept = (int8_t *)(ws + L.pos_accept);
  P.n_items = a->B * (a->K + 1);
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
  P.n_items = B * (K + 1);
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

const char *sd_version(void) { return "sdverify 0.1 (sm_103a)"; }

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
