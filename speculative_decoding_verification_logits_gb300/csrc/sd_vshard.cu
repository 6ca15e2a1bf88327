// Vocabulary-sharded verify: the target's logits split over the vocabulary
// across S devices (tensor-parallel ranks), as when the target runs sharded
// over several GPUs ("Speculative Speculative Decoding" blog
// (jiwasawa.github.io), performance and hardware: the target on four GPUs).
//
// The verify step needs, per logit row, the maximum, its lowest index and
// the sum of 2^(l s + c) over the whole vocabulary, and one inverse-CDF draw
// over the whole vocabulary.  Sharded, that becomes three kernels with an
// exchange between them:
//   stats  per shard: the statistics of every row over the shard's columns
//          (the same records as the split launch's streaming pieces, indices
//          global), its key candidates, and the logits at the drafted tokens
//          the shard owns;                               -> all-gather
//   mass   per shard: every shard combines all shards' records identically,
//          runs the accept scan (the same decision everywhere) and computes
//          its own columns' mass of the draw's distribution at the first
//          rejection m (the residual max(0, p - q), and p for the identically
//          zero residual);                                -> all-gather
//   pick   per shard: the prefix over the shards' masses names the shard
//          holding u * S (the first level of a two-level inverse CDF); that
//          shard alone scans its columns (the second level) and writes the
//          token; every shard writes the rest of the outputs, which are the
//          same everywhere.                               -> all-reduce (max)
// The last exchange fills the one slot per row that only its owner wrote:
// callers pre-fill out_tokens with -1 and hit with 0, so an element-wise
// maximum over the shards (or, on one device, running the shards in turn on
// the same outputs) completes them.  The result equals the unsharded verify
// (the same records are combined in the same order as the split launch's
// pieces, up to where the rows are cut).

#include "sd_device.cuh"

namespace sdv {

constexpr int kVsNT = 256;
constexpr int kVsNW = kVsNT / 32;
constexpr int kVsParts = 8;              // column parts of a shard (mass CTAs per sequence)
constexpr int kVsMass = 16 * kVsParts;   // bytes per sequence in a mass block
constexpr int kVsCH = 4;  // vectors per row a mass thread loads before using them

// Columns [a, e) of part p of a shard of vs columns: kVsParts near-equal
// ranges of whole 16-column groups, the last one taking the rest.
__host__ __device__ inline void vs_part(int vs, int p, int &a, int &e) {
  const int len = ((vs + kVsParts - 1) / kVsParts + 15) / 16 * 16;
  a = p * len < vs ? p * len : vs;
  e = a + len < vs ? a + len : vs;
}

struct VsParams {
  const uint8_t *target, *draft, *bonus;  // this shard's columns
  const int32_t *tokens;
  const float *temps;
  int32_t *keys_out, *num_accepted, *out_tokens, *tau;
  uint8_t *hit;
  int32_t *status;
  uint8_t *stats;            // this shard's stats block (stats kernel)
  const uint8_t *stats_all;  // S stats blocks (mass, pick)
  uint8_t *mass;             // this shard's mass block (mass kernel)
  const uint8_t *mass_all;   // S mass blocks (pick)
  size_t stats_bytes;
  uint64_t seed;
  int64_t row_base;
  int32_t B, K, V, S, shard, v0, vs;
  int32_t keys, chk, kf, n_keys, pw;
  int32_t fanout[SD_MAX_K + 1];
  int32_t fan_off[SD_MAX_K + 2];
};

__host__ __device__ inline size_t vs_stats_bytes(int64_t B, int K) {
  return (size_t)(B * (2 * (int64_t)K + 2) * kRecBytes + B * (int64_t)(K > 0 ? K : 1) * 16);
}

// Slot t of a sequence's rows: t = j (0..K) is target row j; t = K + 1 + j
// the draft row j (j < K) or the bonus draft row (j = K).  Whether a row is
// read (the same rule as the single-device launches).
__device__ __forceinline__ bool vs_present(const VsParams &P, int t, bool sampled) {
  if (t <= P.K) return true;
  const int j = t - (P.K + 1);
  if (j < P.K) return sampled || (P.keys && P.fanout[j] > 0);
  return P.keys && P.bonus && P.fanout[P.K] > 0;
}

// ------------------------------------------------------------------ stats --
// One CTA per (row slot, sequence): the row's statistics over this shard's
// columns, written as a record; the target row j < K also writes the logits
// at d_j when this shard owns d_j.
template <typename E, int KF>
__global__ void __launch_bounds__(kVsNT) sd_vshard_stats_kernel(const __grid_constant__ VsParams P) {
  constexpr int NT = kVsNT, NW = kVsNW, sz = Elt<E>::kSize;
  constexpr int KFm = KF > 0 ? KF : 1;
  const int slot = blockIdx.x, b = blockIdx.y, K = P.K;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  __shared__ RowInfo R;
  __shared__ WStat wst[NW];
  __shared__ int wsel[NW * KFm];
  __shared__ float2 kst[KFm];
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const float T = P.temps[b];
  const bool sampled = T > 0.f && T <= 3.4e38f;
  const float s = sampled ? log2e_over(T) : 0.f;
  const bool is_x = slot > K;
  const int j = is_x ? slot - (K + 1) : slot;
  uint8_t *rec = P.stats + ((int64_t)b * (2 * K + 2) + slot) * kRecBytes;
  if (!is_x && j < K && tid == 0) {
    const int d = P.tokens[(int64_t)b * K + j];
    const bool own = d >= P.v0 && d < P.v0 + P.vs;
    float4 dl = make_float4(__int_as_float(0x7fffffff), __int_as_float(0x7fffffff), 0.f, 0.f);
    if (own) {
      dl.x = Elt<E>::load_global(P.target + (((int64_t)b * (K + 1) + j) * P.vs + (d - P.v0)) * sz);
      dl.y = Elt<E>::load_global(P.draft + (((int64_t)b * K + j) * P.vs + (d - P.v0)) * sz);
      dl.z = 1.f;
    }
    *reinterpret_cast<float4 *>(P.stats + (int64_t)P.B * (2 * K + 2) * kRecBytes +
                                ((int64_t)b * K + j) * 16) = dl;
  }
  if (!vs_present(P, slot, sampled)) {
    if (tid < 8) {
      float *r = reinterpret_cast<float *>(rec);
      if (tid == 0) {
        *reinterpret_cast<float4 *>(r) = make_float4(-INFINITY, __int_as_float(INT32_MAX), INFINITY, 0.f);
        r[4] = 0.f;
      }
      reinterpret_cast<float2 *>(rec + 32)[tid] = make_float2(-INFINITY, __int_as_float(INT32_MAX));
    }
    return;
  }
  int type;
  if (!is_x) type = sampled ? kRowE : kRowA;
  else if (j < K) type = sampled ? (P.keys && P.fanout[j] > 0 ? kRowEK : kRowE) : kRowK;
  else type = kRowK;
  const int fl = row_flags(type, P.chk != 0);
  if (tid == 0) {
    if (!is_x) R.g = P.target + ((int64_t)b * (K + 1) + j) * P.vs * sz;
    else if (j < K) R.g = P.draft + ((int64_t)b * K + j) * P.vs * sz;
    else R.g = P.bonus + (int64_t)b * P.vs * sz;
    R.excl = -1;
    if (is_x && j < K && (fl & kFKeys)) {
      const int d = P.tokens[(int64_t)b * K + j];
      if (d >= P.v0 && d < P.v0 + P.vs) R.excl = d - P.v0;
    }
    row_geometry<NT>(R, 0, P.vs, sz);
  }
  __syncthreads();
  RowAcc<KF> A;
  A.reset();
  bool bad = false;
  const uint64_t s2 = pk2(s, s);
  const uint32_t ni = Elt<E>::kNegInfWord;
#pragma unroll 1
  for (int step = 0; step < R.nsteps; ++step) {
    uint4 v[kU];
#pragma unroll
    for (int k = 0; k < kU; ++k) {
      const int q = step * NT * kU + k * NT + tid;
      if (q >= R.qlo && q < R.qhi) v[k] = __ldcg(reinterpret_cast<const uint4 *>(R.gbase + 16 * q));
      else v[k] = make_uint4(ni, ni, ni, ni);
    }
#pragma unroll 1
    for (int k = 0; k < kU; ++k) {  // the ragged ends, from element loads
      const int q = step * NT * kU + k * NT + tid;
      if ((q < R.qlo || q >= R.qhi) && q < R.nvec) {
        const uint4 w = load_vec_slow<E>(R, q, 0, P.vs);
        if (k == 0) v[0] = w;
        else if (k == 1) v[1] = w;
        else if (k == 2) v[2] = w;
        else v[3] = w;
      }
    }
    step_gen<E, KF, NT>(A, v, step, fl, R.qd_step, R.qd, R.excl, 0, R.hp, s, s2, bad);
  }
  row_end_gen<E, KF>(A, fl, bad, 0, R.hp, &wst[warp], &wsel[warp * KFm]);
  __syncthreads();
  if (tid == 0) {
    float M = -INFINITY;
    bool poison = false;
    for (int w = 0; w < NW; ++w) M = fmaxf(M, wst[w].m);
    int Ix = INT32_MAX;
    float C = INFINITY;
    for (int w = 0; w < NW; ++w) {
      if (wst[w].m == M) Ix = min(Ix, wst[w].idx);
      if (wst[w].z > 0.f) C = fminf(C, wst[w].c);
      poison |= wst[w].z != wst[w].z;
    }
    ff Z{0.f, 0.f};
    for (int w = 0; w < NW; ++w)
      if (wst[w].z > 0.f) Z = ff_add(Z, two_prod(wst[w].z, ex2(C - wst[w].c)));
    if (poison) Z.hi = __int_as_float(0x7fffffff);
    float *r = reinterpret_cast<float *>(rec);
    *reinterpret_cast<float4 *>(r) =
        make_float4(M, __int_as_float(Ix == INT32_MAX ? Ix : Ix + P.v0), C, Z.hi);
    r[4] = Z.lo;
  }
  if (warp == 0) {
    if (KF > 0 && (fl & kFKeys)) {
      cta_keys<E, KFm, NT>(R, wsel, 0, P.vs, kst);
      __syncwarp();
    }
    if (lane < 8) {
      float2 e = make_float2(-INFINITY, __int_as_float(INT32_MAX));
      if (KF > 0 && (fl & kFKeys) && lane < KFm) {
        e = kst[lane];
        const int ix = __float_as_int(e.y);
        if (ix != INT32_MAX) e.y = __int_as_float(ix + P.v0);
      }
      reinterpret_cast<float2 *>(rec + 32)[lane] = e;
    }
  }
}

// ------------------------------------------------------------ decision --
// What every shard decides the same way from all shards' records.
struct VsS {
  float M[kMaxRows], C[kMaxRows];
  ff Z[kMaxRows];
  int amax[kMaxRows];
  int d[SD_MAX_K];
  float ld_t[SD_MAX_K], ld_d[SD_MAX_K];
  float u_acc[SD_MAX_K], u_draw[SD_MAX_K + 1];
  int2 keys[(SD_MAX_K + 1) * SD_MAX_FANOUT];
  RowInfo dt, dd, ddt;
  ff wmass[kVsNW];
  ff t_loc, t_w;
  int m, kind, valid, dvalid, fvalid, tok, owner, wsel, part;
};

// Combine of every row over the shards (warp per row, lane p = shard p, the
// records' combine of the split launch), the logits at the drafted tokens
// from their owners, and the accept scan: m, kind, validity.
template <typename E>
__device__ void vs_decide(const VsParams &P, VsS &S, int b, float s, bool tvalid, bool sampled) {
  constexpr int NW = kVsNW;
  const int K = P.K, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nslot = 2 * K + 2;
  if (warp == 0) {
    const int d = lane < K ? P.tokens[(int64_t)b * K + lane] : 0;
    const bool dvalid = __all_sync(0xffffffffu, lane >= K || (d >= 0 && d < P.V));
    if (lane < K) {
      S.d[lane] = d;
      float lt = -INFINITY, ld = -INFINITY;
      for (int p = 0; p < P.S; ++p) {
        const float4 dl = __ldcg(reinterpret_cast<const float4 *>(
            P.stats_all + (int64_t)p * P.stats_bytes + (int64_t)P.B * nslot * kRecBytes +
            ((int64_t)b * K + lane) * 16));
        if (dl.z == 1.f) {
          lt = dl.x;
          ld = dl.y;
        }
      }
      S.ld_t[lane] = lt;
      S.ld_d[lane] = ld;
    }
    if (lane == 0) {
      S.dvalid = dvalid ? 1 : 0;
      S.fvalid = 1;
    }
    if (sampled)
      for (int q = lane; q <= K; q += 32) {
        if (q < K) S.u_acc[q] = uniform_u(P.seed, P.row_base + b, q, 0);
        S.u_draw[q] = uniform_u(P.seed, P.row_base + b, q, 1);
      }
  }
  __syncthreads();
#pragma unroll 1
  for (int r = warp; r < nslot; r += NW) {
    CStat x{-INFINITY, INT32_MAX, INFINITY, 0.f, 0.f};
    if (lane < P.S) {
      const float *rp = reinterpret_cast<const float *>(
          P.stats_all + (int64_t)lane * P.stats_bytes + ((int64_t)b * nslot + r) * kRecBytes);
      const float4 a4 = __ldcg(reinterpret_cast<const float4 *>(rp));
      x = CStat{a4.x, __float_as_int(a4.y), a4.z, a4.w, __ldcg(rp + 4)};
    }
    const bool poison = ballot(x.zhi != x.zhi) != 0u;
    const float M = rmax_f(x.m);
    const int I = rmin_i(x.m == M ? x.idx : INT32_MAX);
    const float C = rmin_f(x.zhi > 0.f ? x.c : INFINITY);
    const ff zt = x.zhi > 0.f ? ff_mul_f(ff{x.zhi, x.zlo}, ex2(C - x.c)) : ff{0.f, 0.f};
    const ff Z = ff_warp_sum(zt);
    if (lane == 0) {
      S.M[r] = M;
      S.C[r] = C;
      S.Z[r] = Z;
      S.amax[r] = I == INT32_MAX ? 0 : I;
      if (P.chk && vs_present(P, r, sampled) && (poison || !(M > -INFINITY))) S.fvalid = 0;
    }
  }
  __syncthreads();
  if (warp == 0) {
    const int j = lane;
    const bool dvalid = S.dvalid != 0;
    int rej = 0;
    if (j < K) {
      int a = 0;
      if (!sampled) {
        a = (dvalid && S.d[j] == S.amax[j]) ? 1 : 0;
      } else if (dvalid) {
        const int rd = K + 1 + j;
        const float lt = S.ld_t[j], ldr = S.ld_d[j];
        const ff xt = ff_add_f(two_prod(lt, s), S.C[j]);
        const ff xd = ff_add_f(two_prod(ldr, s), S.C[rd]);
        const float r = (ldr == -INFINITY) ? INFINITY
                                           : exp2_ff(ff_sub(xt, xd)) * ff_ratio(S.Z[rd], S.Z[j]);
        a = (S.u_acc[j] <= r) ? 1 : 0;
      }
      rej = !a;
    }
    const unsigned rejects = ballot(rej);
    if (lane == 0) {
      const int mm = rejects ? __ffs(rejects) - 1 : K;
      const bool valid = tvalid && dvalid && S.fvalid != 0;
      S.m = mm;
      S.valid = valid ? 1 : 0;
      S.kind = 0;
      S.tok = -1;
      S.owner = -1;
      if (valid) {
        if (!sampled) S.tok = S.amax[mm];
        else S.kind = mm < K ? 1 : 2;
      }
    }
  }
  __syncthreads();
}

// The rows the draw reads, on columns [a, e) of this shard.
template <typename E>
__device__ void vs_draw_rows(const VsParams &P, VsS &S, int b, int a, int e) {
  constexpr int sz = Elt<E>::kSize;
  const int K = P.K, mm = S.m;
  if (threadIdx.x == 0 && S.kind != 0) {
    S.dt.g = P.target + ((int64_t)b * (K + 1) + mm) * P.vs * sz;
    S.dt.excl = -1;
    row_geometry<kVsNT>(S.dt, a, e, sz);
    if (mm < K) {
      S.dd.g = P.draft + ((int64_t)b * K + mm) * P.vs * sz;
      S.dd.excl = -1;
      row_geometry<kVsNT>(S.dd, a, e, sz);
      S.ddt = S.dt;  // the draft row read element-wise on the target's grid
      S.ddt.g = S.dd.g;
      S.ddt.qlo = 1;
      S.ddt.qhi = 0;
    }
  }
  __syncthreads();
}

// ------------------------------------------------------------------- mass --
// One CTA per (sequence, part of the shard's columns): the decision, then
// the part's mass of the residual at m and of p at m (the fallback for an
// identically zero residual), one float-float pair each per part.
template <typename E>
__global__ void __launch_bounds__(kVsNT) sd_vshard_mass_kernel(const __grid_constant__ VsParams P) {
  constexpr int NT = kVsNT, NW = kVsNW;
  const int b = blockIdx.x, part = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  __shared__ VsS S;
  __shared__ ff red[2][NW];
  int pa, pe;  // this CTA's columns of the shard
  vs_part(P.vs, part, pa, pe);
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const float T = P.temps[b];
  const bool tvalid = (T >= 0.f) && (T <= 3.4e38f);
  const bool sampled = tvalid && T > 0.f;
  const float s = sampled ? log2e_over(T) : 0.f;
  vs_decide<E>(P, S, b, s, tvalid, sampled);
  vs_draw_rows<E>(P, S, b, pa, pe);
  ff mres{0.f, 0.f}, mp{0.f, 0.f};
  if (S.kind != 0) {
    const int mm = S.m;
    const bool residual = S.kind == 1;
    const float Ct = S.C[mm];
    const float Cd = residual ? S.C[P.K + 1 + mm] : 0.f;
    const float Rz = residual ? ff_ratio(S.Z[mm], S.Z[P.K + 1 + mm]) : 0.f;
    const uint64_t s2 = pk2(s, s), ct2 = pk2(Ct, Ct), cd2 = pk2(Cd, Cd), r2 = pk2(Rz, Rz);
    const bool d_vec = residual && S.dd.hp == S.dt.hp;
    float a = 0.f, ac = 0.f, p = 0.f, pc = 0.f;
    // kVsCH vectors of each row per thread in flight at once, then their masses
    const int nvec = S.dt.nvec;
#pragma unroll 1
    for (int q0 = tid; q0 < nvec; q0 += NT * kVsCH) {
      uint4 tv[kVsCH], dv[kVsCH];
#pragma unroll
      for (int c = 0; c < kVsCH; ++c) {
        const int q = q0 + c * NT;
        if (q < nvec) {
          tv[c] = load_vec_direct<E>(S.dt, q, pa, pe);
          if (residual)
            dv[c] = d_vec ? load_vec_direct<E>(S.dd, q, pa, pe)
                          : load_vec_slow<E>(S.ddt, q, pa, pe);
        }
      }
#pragma unroll
      for (int c = 0; c < kVsCH; ++c) {
        if (q0 + c * NT < nvec) {
          if (residual) kahan_add(a, ac, vec_mass<E>(tv[c], dv[c], true, s2, ct2, cd2, r2));
          kahan_add(p, pc, vec_mass<E>(tv[c], tv[c], false, s2, ct2, cd2, r2));
        }
      }
    }
    mres = ff_warp_sum(two_sum(a, -ac));
    mp = ff_warp_sum(two_sum(p, -pc));
  }
  if (lane == 0) {
    red[0][warp] = mres;
    red[1][warp] = mp;
  }
  __syncthreads();
  if (tid == 0) {
    ff x{0.f, 0.f}, y{0.f, 0.f};
    for (int w = 0; w < NW; ++w) {
      x = ff_add(x, red[0][w]);
      y = ff_add(y, red[1][w]);
    }
    *reinterpret_cast<float4 *>(P.mass + (int64_t)b * kVsMass + 16 * part) =
        make_float4(x.hi, x.lo, y.hi, y.lo);
  }
}

// ------------------------------------------------------------------- pick --
// One CTA per sequence: the decision again, the keys from all shards'
// candidates, the shard holding u * S and, in it, the part holding it; that
// shard scans the part's columns (warp, iteration, lane, element, as the
// split launch's finish does) and writes the token.  Every shard writes the outputs that are the same everywhere.
template <typename E>
__global__ void __launch_bounds__(kVsNT) sd_vshard_pick_kernel(const __grid_constant__ VsParams P) {
  constexpr int NW = kVsNW;
  constexpr int sz = Elt<E>::kSize, NV = Elt<E>::kPerVec;
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = P.K, nslot = 2 * K + 2;
  __shared__ VsS S;
  extern __shared__ __align__(128) float pm[];  // [NW][pw][32] masses of the draw
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const float T = P.temps[b];
  const bool tvalid = (T >= 0.f) && (T <= 3.4e38f);
  const bool sampled = tvalid && T > 0.f;
  const float s = sampled ? log2e_over(T) : 0.f;
  vs_decide<E>(P, S, b, s, tvalid, sampled);
  // keys of each position: the best fan of all shards' candidates
  if (P.keys) {
    const int kf = P.kf;
#pragma unroll 1
    for (int j = warp; j <= K; j += NW) {
      const int fan = P.fanout[j];
      if (fan <= 0) continue;
      const int xs = K + 1 + j;
      constexpr int PER = (32 * 8 + 31) / 32;
      float cv[PER];
      int ci[PER];
#pragma unroll
      for (int h = 0; h < PER; ++h) {
        const int c = lane + 32 * h;  // candidate c: shard c / kf, rank c % kf
        cv[h] = -INFINITY;
        ci[h] = INT32_MAX;
        if (c < P.S * kf) {
          const float2 e = __ldcg(reinterpret_cast<const float2 *>(
              P.stats_all + (int64_t)(c / kf) * P.stats_bytes +
              ((int64_t)b * nslot + xs) * kRecBytes + 32 + (c % kf) * 8));
          cv[h] = e.x;
          ci[h] = __float_as_int(e.y);
        }
      }
      int32_t *kout = P.keys_out ? P.keys_out + ((int64_t)b * P.n_keys + P.fan_off[j]) * 2 : nullptr;
#pragma unroll 1
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
          S.keys[P.fan_off[j] + r2] = key;
          if (kout) {
            kout[2 * r2] = key.x;
            kout[2 * r2 + 1] = key.y;
          }
        }
      }
    }
  }
  if (S.kind != 0 && warp == 0) {
    // the shard holding u * S: prefix over the shards' masses (lane p: shard
    // p, the sum of its parts in order)
    const int mm = S.m;
    ff x{0.f, 0.f}, y{0.f, 0.f};
    if (lane < P.S) {
#pragma unroll
      for (int q = 0; q < kVsParts; ++q) {
        const float4 m4 = __ldcg(reinterpret_cast<const float4 *>(
            P.mass_all + (int64_t)lane * P.B * kVsMass + (int64_t)b * kVsMass + 16 * q));
        x = ff_add(x, ff{m4.x, m4.y});
        y = ff_add(y, ff{m4.z, m4.w});
      }
    }
    const ff tres = ff_warp_sum(x);
    // a draw from p at the bonus position, or for an identically zero residual
    const bool use_p = S.kind == 2 || !ff_pos(tres);
    const ff xs = use_p ? y : x;
    const ff tot = use_p ? ff_warp_sum(y) : tres;
    const ff t = ff_mul_f(tot, S.u_draw[mm]);
    const Cross c = ff_cross(xs, t);
    if (lane == 0) {
      S.owner = c.l < 0 ? 0 : c.l;
      S.t_loc = ff_sub(t, c.before);
      if (use_p) S.kind = 2;
    }
  }
  __syncthreads();
  if (S.kind != 0 && S.owner == P.shard) {
    // the part of this shard holding u * S (lane q: part q)
    if (warp == 0) {
      ff mq{0.f, 0.f};
      if (lane < kVsParts) {
        const float4 m4 = __ldcg(reinterpret_cast<const float4 *>(
            P.mass_all + (int64_t)P.shard * P.B * kVsMass + (int64_t)b * kVsMass + 16 * lane));
        mq = S.kind == 2 ? ff{m4.z, m4.w} : ff{m4.x, m4.y};
      }
      const Cross c = ff_cross(mq, S.t_loc);
      if (lane == 0) {
        S.part = c.l < 0 ? 0 : c.l;
        S.t_loc = ff_sub(S.t_loc, c.before);
      }
    }
    __syncthreads();
    int pa, pe;  // the part's columns, which the draw scans
    vs_part(P.vs, S.part, pa, pe);
    vs_draw_rows<E>(P, S, b, pa, pe);
    const int mm = S.m;
    const bool residual = S.kind == 1;
    const RowInfo &Rt = S.dt;
    const bool d_vec = residual && S.dd.hp == Rt.hp;
    const float Ct = S.C[mm];
    const float Cd = residual ? S.C[K + 1 + mm] : 0.f;
    const float Rz = residual ? ff_ratio(S.Z[mm], S.Z[K + 1 + mm]) : 0.f;
    const uint64_t s2 = pk2(s, s), ct2 = pk2(Ct, Ct), cd2 = pk2(Cd, Cd), r2 = pk2(Rz, Rz);
    const int nvec = Rt.nvec;
    const int wr = (nvec + NW - 1) / NW;
    const int wq0 = min(warp * wr, nvec), wq1 = min(wq0 + wr, nvec);
    float *pmw = pm + warp * P.pw * 32;
    const ff lm = draw_pass<E>(Rt, S.dd, S.ddt, residual, d_vec, wq0, wq1, pa, pe, s2, ct2, cd2,
                               r2, pmw);
    const ff wm = ff_warp_sum(lm);
    if (lane == 0) S.wmass[warp] = wm;
    __syncthreads();
    if (warp == 0) {
      const ff m_l = lane < NW ? S.wmass[lane] : ff{0.f, 0.f};
      const Cross c = ff_cross(m_l, S.t_loc);
      if (lane == 0) {
        S.wsel = c.l < 0 ? 0 : c.l;
        S.t_w = ff_sub(S.t_loc, c.before);
      }
    }
    __syncthreads();
    if (warp == S.wsel) {
      const int nit = (wq1 - wq0 + 31) / 32;
      ff cum{0.f, 0.f};
      int isel = -1;
      ff t_it{0.f, 0.f};
#pragma unroll 1
      for (int tb = 0; tb < nit; tb += 32) {
        const int t = tb + lane;
        ff mt{0.f, 0.f};
        if (t < nit) {
          ff a0{0.f, 0.f}, a1{0.f, 0.f};
#pragma unroll 4
          for (int i = 0; i < 32; i += 2) {
            a0 = ff_add_f(a0, pmw[t * 32 + ((i + lane) & 31)]);
            a1 = ff_add_f(a1, pmw[t * 32 + ((i + 1 + lane) & 31)]);
          }
          mt = ff_add(a0, a1);
        }
        const ff rem = ff_sub(S.t_w, cum);
        const Cross c = ff_cross(mt, rem);
        if (c.l >= 0) {
          isel = tb + c.l;
          t_it = ff_sub(rem, c.before);
          if (c.crossed) break;
        }
        cum = ff_add(cum, c.total);
      }
      int tok = -1;
      if (isel >= 0) {
        const Cross cl = ff_cross(ff{pmw[isel * 32 + lane], 0.f}, t_it);
        if (cl.l >= 0) {
          const ff t_l = ff_sub(t_it, cl.before);
          const int q = wq0 + isel * 32 + cl.l;
          const int i = lane % NV;
          const uint4 tvv = load_vec_direct<E>(Rt, q, pa, pe);
          uint4 dvv = tvv;
          if (residual)
            dvv = d_vec ? load_vec_direct<E>(S.dd, q, pa, pe) : load_vec_slow<E>(S.ddt, q, pa, pe);
          float ww[NV];
          pass_weights<E>(tvv, dvv, residual, s2, ct2, cd2, r2, ww);
          float wi = 0.f;
#pragma unroll
          for (int ii = 0; ii < NV; ++ii)
            if (ii == i) wi = ww[ii];
          const int ei = elem_index(pa, Rt.hp, q, i, sz);
          const bool ok = lane < NV && ei >= pa && ei < pe && wi > 0.f;
          const Cross ce = ff_cross(ff{ok ? wi : 0.f, 0.f}, t_l);
          tok = __shfl_sync(0xffffffffu, ei, ce.l < 0 ? 0 : ce.l);
          if (ce.l < 0) tok = -1;
        }
      }
      // rounding left no element: the shard's largest logit of row m stands in
      if (lane == 0) S.tok = tok >= 0 ? tok + P.v0 : S.amax[mm];
    }
    __syncthreads();
  }
  // ---- outputs: every shard writes what is the same everywhere; the token
  // of a sampled row and its hit flag only on the owning shard
  if (warp == 0) {
    const bool valid = S.valid != 0;
    const bool mine = S.kind == 0 || S.owner == P.shard;
    const int mm = valid ? S.m : -1, tok = S.tok;
    int32_t *out = P.out_tokens + (int64_t)b * (K + 1);
    for (int j = lane; j <= K; j += 32) {
      if (!valid) out[j] = -1;
      else if (j < mm) out[j] = S.d[j];
      else if (j > mm) out[j] = -1;
      else if (mine) out[j] = tok;
    }
    bool h = false;
    if (valid && mine && P.hit && P.keys)
      for (int k2 = lane; k2 < P.n_keys; k2 += 32) h |= S.keys[k2].x == mm && S.keys[k2].y == tok;
    const bool hit = ballot(h) != 0u;
    if (lane == 0) {
      P.num_accepted[b] = valid ? mm : 0;
      P.tau[b] = valid ? mm + 1 : 0;
      if (P.hit && (mine || !valid)) P.hit[b] = (uint8_t)(hit ? 1 : 0);
      if (!valid && P.status) {
        int bits = 0;
        if (!tvalid) bits |= (int)SD_STATUS_BAD_TEMP;
        if (!S.dvalid) bits |= (int)SD_STATUS_BAD_TOKEN;
        if (tvalid && S.dvalid && !S.fvalid) bits |= (int)SD_STATUS_NONFINITE;
        atomicOr(P.status, bits);
      }
    }
  }
}

// ===================================================================== host

static sd_status_t vs_params(const sd_vshard_args *a, VsParams &P) {
  if (!a) return SD_ERR_INVALID_ARG;
  if (a->B < 0 || a->K < 0 || a->K > SD_MAX_K || a->V < 1 || a->V > SD_MAX_V) return SD_ERR_INVALID_ARG;
  if (a->S < 1 || a->S > 32 || a->shard < 0 || a->shard >= a->S) return SD_ERR_INVALID_ARG;
  if (a->v0 < 0 || a->vs < 1 || (int64_t)a->v0 + a->vs > a->V) return SD_ERR_INVALID_ARG;
  if (a->dtype != SD_F32 && a->dtype != SD_BF16) return SD_ERR_INVALID_ARG;
  if (a->flags & ~(SD_FLAG_PREDICT | SD_FLAG_CHECK_FINITE)) return SD_ERR_INVALID_ARG;
  memset(&P, 0, sizeof(P));
  P.target = (const uint8_t *)a->target_logits;
  P.draft = (const uint8_t *)a->draft_logits;
  P.tokens = a->draft_tokens;
  P.temps = a->temperature;
  P.keys_out = a->keys_out;
  P.num_accepted = a->num_accepted;
  P.out_tokens = a->out_tokens;
  P.tau = a->tau;
  P.hit = a->hit;
  P.status = a->status;
  P.seed = a->seed;
  P.row_base = a->row_base;
  P.B = a->B;
  P.K = a->K;
  P.V = a->V;
  P.S = a->S;
  P.shard = a->shard;
  P.v0 = a->v0;
  P.vs = a->vs;
  P.chk = (a->flags & SD_FLAG_CHECK_FINITE) ? 1 : 0;
  P.stats_bytes = vs_stats_bytes(a->B, a->K);
  const size_t esz = a->dtype == SD_BF16 ? 2 : 4;
  if (a->B > 0) {
    if (!P.target || !P.temps) return SD_ERR_INVALID_ARG;
    if (a->K > 0 && (!P.draft || !P.tokens)) return SD_ERR_INVALID_ARG;
    if ((uintptr_t)P.target % esz || (P.draft && (uintptr_t)P.draft % esz)) return SD_ERR_INVALID_ARG;
  }
  if (a->flags & SD_FLAG_PREDICT) {
    if (!a->fanout_host) return SD_ERR_INVALID_ARG;
    int off = 0;
    for (int k = 0; k <= a->K; ++k) {
      const int f = a->fanout_host[k];
      if (f < 0 || f > SD_MAX_FANOUT) return SD_ERR_INVALID_ARG;
      P.fanout[k] = f;
      P.fan_off[k] = off;
      off += f;
    }
    P.fan_off[a->K + 1] = off;
    P.n_keys = off;
    P.keys = off > 0 ? 1 : 0;
    P.bonus = (const uint8_t *)a->draft_bonus_logits;
    if (P.bonus && (uintptr_t)P.bonus % esz) return SD_ERR_INVALID_ARG;
  }
  int fmax = 0;
  for (int k = 0; k <= a->K && P.keys; ++k) fmax = std::max(fmax, P.fanout[k]);
  P.kf = fmax == 0 ? 1 : (fmax <= 2 ? 2 : (fmax <= 4 ? 4 : 8));
  return SD_OK;
}

static sd_status_t vs_launch(const void *fn, dim3 grid, int smem, const VsParams &P,
                             cudaStream_t s, const char *what) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kVsNT, 1, 1);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, (void (*)(const VsParams))fn, P);
  if (e != cudaSuccess) {
    fprintf(stderr, "%s launch failed: %s\n", what, cudaGetErrorString(e));
    return SD_ERR_CUDA;
  }
  return SD_OK;
}

template <typename E>
static const void *vs_stats_fn(int kf) {
  if (kf <= 1) return (const void *)sd_vshard_stats_kernel<E, 0>;
  if (kf == 2) return (const void *)sd_vshard_stats_kernel<E, 2>;
  if (kf == 4) return (const void *)sd_vshard_stats_kernel<E, 4>;
  return (const void *)sd_vshard_stats_kernel<E, 8>;
}

static const int kVsSmemCap = 227 * 1024 - (int)sizeof(VsS) - 256;

template <typename E>
static const void *vs_pick_fn() {
  static FuncAttrs attrs;
  const void *fn = (const void *)sd_vshard_pick_kernel<E>;
  attrs.apply(fn, kVsSmemCap, false, "the sharded pick kernel");
  return fn;
}

}  // namespace sdv

using namespace sdv;

extern "C" {

size_t sd_vshard_stats_bytes(int32_t B, int32_t K) {
  if (B < 0 || K < 0 || K > SD_MAX_K) return 0;
  return vs_stats_bytes(B, K);
}

size_t sd_vshard_mass_bytes(int32_t B) { return B < 0 ? 0 : (size_t)B * kVsMass; }

sd_status_t sd_vshard_stats(const sd_vshard_args *a, void *stats, void *stream) {
  sdv::NvtxRange nvtx_range("sd_vshard_stats");
  VsParams P;
  const sd_status_t st = vs_params(a, P);
  if (st != SD_OK) return st;
  if (P.B == 0) return SD_OK;
  if (!stats || (uintptr_t)stats % 16) return SD_ERR_INVALID_ARG;
  P.stats = (uint8_t *)stats;
  const dim3 grid((unsigned)(2 * P.K + 2), (unsigned)P.B, 1);
  const void *fn = a->dtype == SD_BF16 ? vs_stats_fn<__nv_bfloat16>(P.keys ? P.kf : 0)
                                       : vs_stats_fn<float>(P.keys ? P.kf : 0);
  return vs_launch(fn, grid, 0, P, (cudaStream_t)stream, "sd_vshard_stats");
}

sd_status_t sd_vshard_mass(const sd_vshard_args *a, const void *stats_all, void *mass,
                           void *stream) {
  sdv::NvtxRange nvtx_range("sd_vshard_mass");
  VsParams P;
  const sd_status_t st = vs_params(a, P);
  if (st != SD_OK) return st;
  if (P.B == 0) return SD_OK;
  if (!stats_all || !mass || (uintptr_t)stats_all % 16 || (uintptr_t)mass % 16)
    return SD_ERR_INVALID_ARG;
  P.stats_all = (const uint8_t *)stats_all;
  P.mass = (uint8_t *)mass;
  const void *fn = a->dtype == SD_BF16 ? (const void *)sd_vshard_mass_kernel<__nv_bfloat16>
                                       : (const void *)sd_vshard_mass_kernel<float>;
  return vs_launch(fn, dim3((unsigned)P.B, kVsParts, 1), 0, P, (cudaStream_t)stream,
                   "sd_vshard_mass");
}

sd_status_t sd_vshard_pick(const sd_vshard_args *a, const void *stats_all, const void *mass_all,
                           void *stream) {
  sdv::NvtxRange nvtx_range("sd_vshard_pick");
  VsParams P;
  const sd_status_t st = vs_params(a, P);
  if (st != SD_OK) return st;
  if (P.B == 0) return SD_OK;
  if (!stats_all || !mass_all || (uintptr_t)stats_all % 16 || (uintptr_t)mass_all % 16)
    return SD_ERR_INVALID_ARG;
  if (!P.num_accepted || !P.out_tokens || !P.tau) return SD_ERR_INVALID_ARG;
  if (P.keys && !P.keys_out) return SD_ERR_INVALID_ARG;
  P.stats_all = (const uint8_t *)stats_all;
  P.mass_all = (const uint8_t *)mass_all;
  const int sz = a->dtype == SD_BF16 ? 2 : 4;
  int pa, pe;  // the draw scans one part of the shard: part 0 is the largest
  vs_part(P.vs, 0, pa, pe);
  const int nvec = (int)(((int64_t)(pe - pa) * sz + 31) / 16) + 1;
  P.pw = ((nvec + kVsNW - 1) / kVsNW + 31) / 32;
  const int smem = 4 * kVsNW * P.pw * 32;
  if (smem > kVsSmemCap) return SD_ERR_UNSUPPORTED;
  const void *fn = a->dtype == SD_BF16 ? vs_pick_fn<__nv_bfloat16>() : vs_pick_fn<float>();
  return vs_launch(fn, dim3((unsigned)P.B, 1, 1), smem, P, (cudaStream_t)stream, "sd_vshard_pick");
}

}  // extern "C"
