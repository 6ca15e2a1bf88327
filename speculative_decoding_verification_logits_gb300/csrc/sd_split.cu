// Split launch of the verify step: a flat streaming grid over the logit rows
// of all sequences, then a compact per-sequence finish.
//
// Streaming grid.  About two CTAs per SM stream the rows of all sequences
// laid end to end; every CTA gets the same number of 16 KB streaming steps,
// so every SM moves the same bytes.  Rows are grouped by position, j = K
// first: in group j, sequence after sequence, draft row j (the bonus draft
// row for j = K) when the sequence needs it, then target row j; draft rows
// with keys and target rows alternate, so every CTA sees the same mix of
// row kinds.  The rows of the first positions, where a rejection is
// likeliest, come last, so that the finish finds them in L2 when a round's
// logits fit there.  A CTA issues its first copies as soon as it knows where
// its rows are, before it loads the temperatures and drafted tokens that say
// what each row is streamed for.  One row loop serves every kind of row (the statistics a row needs --
// offset exp-sum, argmax, key vectors, the finiteness check -- are switched
// per row), and ragged vectors are assembled into the copy ring where they
// are issued, so the loop always consumes whole steps.  Per row piece the
// CTA writes a record: max, lowest-index argmax, the offset exp-sum as a
// float-float pair and its best key candidates.
//
// Finish.  One thread-block cluster per sequence, launched as a
// programmatic dependent of the streaming grid: its prologue (drafted
// tokens, their logits, the uniforms, the sequence's place in the flat
// order, the geometry of every row the draw may read) reads only inputs and
// overlaps the stream's tail.  Then every CTA
// combines the records of each row in the same order, so all CTAs take the
// same accept decisions; warp 0 runs the accept scan while the other warps
// merge the key candidates.  The draw (residual max(0, p - q) at the first
// rejection m, or p at the bonus position) splits the vocabulary over the
// cluster's CTAs: each warp reads its contiguous share of the two rows with
// all of its loads in flight at once, keeps one mass per (iteration, lane),
// and the CTA masses are exchanged over distributed shared memory.  The CTA
// holding u * S then narrows the crossing down warp -> iteration -> lane ->
// element with one float-float search routine.  The kernel is kept small
// (loops, one shared search routine, no per-kind copies of the row code):
// the chain after the stream runs once per sequence, and straight-line code
// that misses the instruction caches costs several cycles per instruction.
//
// Method sources (web pages): "What is speculative decoding" explainer
// (lotook.com), the four-stage loop and the FAQ on losslessness;
// "Speculative Speculative Decoding" blog (jiwasawa.github.io), Saguaro
// 1. Outcome Prediction; "LLMの生成を5倍速くする「D3D」を図で読む"
// (animemo.app), 検証のまとめ.  Readings where they are silent are listed in
// include/sd_verify.h.

#include "sd_device.cuh"

namespace sdv {

// =========================================================== streaming grid

// Dynamic shared memory of the streaming kernel (byte offsets).
struct FlatLayout {
  int ring, wstat, wsel, rank, total;
};
__host__ __device__ inline FlatLayout flat_layout(int NT, int KF, int B) {
  const int nw = NT / 32, kf = KF > 0 ? KF : 1;
  FlatLayout L;
  int o = 0;
  L.ring = o;  // [kDepth][kU][NT] 16-byte vectors
  o = align128(o + kDepth * kU * NT * 16);
  L.wstat = o;  // [kMaxRows][nw] WStat
  o = align128(o + 16 * kMaxRows * nw);
  L.wsel = o;  // [kMaxRows][nw][KF] key vectors chosen by each warp
  o = align128(o + 4 * kMaxRows * nw * kf);
  L.rank = o;  // [B + 1] sampled sequences before each sequence
  o = align128(o + 4 * (B + 1));
  L.total = o;
  return L;
}

// CTAs of the streaming kernel per SM (three, where the registers allow it
// for rows without key tracking, measured slower: more CTAs contend for the
// same HBM bandwidth and the last wave of steps ends later).
template <int KF>
constexpr int stream_ctas_per_sm() { return 2; }

template <typename E, int KF, int NT>
__global__ void __launch_bounds__(NT, stream_ctas_per_sm<KF>())
    sd_flat_stream_kernel(const __grid_constant__ Params P) {
  constexpr int sz = Elt<E>::kSize;
  constexpr int KFm = KF > 0 ? KF : 1;
  constexpr int NW = NT / 32;
  constexpr int ue = NT * kU * 16 / sz;  // elements per streaming step
  constexpr uint32_t kSlot = kU * NT * 16;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = P.K;

  __shared__ Static S;
  __shared__ int goff[SD_MAX_K + 2];
  __shared__ int wcnt[kMaxWarps];
  extern __shared__ __align__(128) uint8_t dyn[];
  // Launched as a programmatic dependent of the stream's previous kernel:
  // nothing is read before that kernel has finished.  Then the finish grid
  // may be scheduled at once: its CTAs take the place of streaming CTAs as
  // those exit and run their prologue meanwhile (reading only inputs; their
  // griddepcontrol.wait still waits for this whole grid).
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const FlatLayout FL = flat_layout(NT, KF, P.B);
  uint8_t *ring = dyn + FL.ring;
  const uint32_t ring_t = smem_u32(ring) + tid * 16;
  WStat *wstat = reinterpret_cast<WStat *>(dyn + FL.wstat);
  int *wsel = reinterpret_cast<int *>(dyn + FL.wsel);
  int *rank = reinterpret_cast<int *>(dyn + FL.rank);

  // ---- rank[b]: sampled sequences before b, b = 0..B (a block-wide scan;
  // only groups whose draft rows belong to the sampled sequences need it)
  bool sonly = false;
  for (int g = 0; g <= K; ++g) sonly |= P.grp_x[g] == 1;
  int ns = 0;
  if (sonly) {
#pragma unroll 1
    for (int x0 = 0; x0 < P.B; x0 += NT) {
      const int x = x0 + tid;
      const float tx = x < P.B ? P.temps[x] : 0.f;
      const bool sx = tx > 0.f && tx <= 3.4e38f;
      const unsigned m = ballot(sx);
      if (lane == 0) wcnt[warp] = __popc(m);
      __syncthreads();
      int before = 0, total = 0;
#pragma unroll 1
      for (int w = 0; w < NW; ++w) {
        before += w < warp ? wcnt[w] : 0;
        total += wcnt[w];
      }
      if (x < P.B) rank[x] = ns + before + __popc(m & ((1u << lane) - 1u));
      ns += total;
      __syncthreads();
    }
    if (tid == 0) rank[P.B] = ns;
  }
  if (tid == 0) {
    int o = 0;
    for (int g = 0; g <= K; ++g) {
      goff[g] = o;
      o += P.B + (P.grp_x[g] == 2 ? P.B : (P.grp_x[g] == 1 ? ns : 0));
    }
    goff[K + 1] = o;
  }
  __syncthreads();

  // ---- this CTA's steps [u_lo, u_hi) of the flat stream, cut into pieces
  const int64_t U = (int64_t)goff[K + 1] * P.spr, G = gridDim.x;
  const int64_t u_lo = U * blockIdx.x / G, u_hi = U * (blockIdx.x + 1) / G;
  if (u_hi <= u_lo) return;  // more CTAs than steps
  const int64_t r_first = u_lo / P.spr;
  const int nrows = (int)((u_hi - 1) / P.spr - r_first + 1);  // <= kMaxRows (host)
  int rb = 0, rfj = 0;  // this thread's row: its sequence and fan-out
  if (tid < nrows) {
    // flat row r: group g (position j = K - g), place i in the group
    const int64_t r = r_first + tid;
    int g = 0;
    while (g < K && goff[g + 1] <= r) ++g;
    const int i = (int)(r - goff[g]), j = K - g, gx = P.grp_x[g];
    int b = i;
    bool isx = false;
    if (gx == 2) {
      b = i >> 1;
      isx = (i & 1) == 0;
    } else if (gx == 1) {  // the last b with b + rank[b] <= i
      int lo = 0, hi = P.B - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (mid + rank[mid] <= i) lo = mid;
        else hi = mid - 1;
      }
      b = lo;
      isx = rank[b + 1] > rank[b] && i == b + rank[b];
    }
    // where the row is (all the first copies need); what it is streamed for
    // depends on inputs and is filled in once those copies are under way
    const int fj = (isx && g > 0 && P.keys) ? P.fanout[j] : 0;
    RowInfo &R = S.rows[tid];
    R.kind = isx ? (g == 0 ? kBonus : kDraft) : kTarget;
    R.j = j;
    R.rec = blockIdx.x + (int)r;
    R.excl = -1;
    R.fan = 0;
    if (R.kind == kTarget) {
      R.g = P.target + ((int64_t)b * (K + 1) + j) * P.V * sz;
    } else if (R.kind == kDraft) {
      R.g = P.draft + ((int64_t)b * K + j) * P.V * sz;
      R.fan = fj;
    } else {
      R.g = P.bonus + (int64_t)b * P.V * sz;
      R.fan = P.fanout[K];
    }
    const int64_t r0 = r * P.spr;
    const int64_t a = (u_lo > r0 ? u_lo : r0) - r0;
    const int64_t e = (u_hi < r0 + P.spr ? u_hi : r0 + P.spr) - r0;
    row_geometry<NT>(R, (int)(a * ue), (int)(e * ue < P.V ? e * ue : (int64_t)P.V), sz);
    rb = b;
    rfj = fj;
  }
  __syncthreads();

  // ---- stream the pieces: one row loop for every kind of row
  {
    Issuer I;
    I.row = 0;
    I.slot = ring_t;
    issuer_row<NT>(I, S, nrows);
#pragma unroll
    for (int d = 0; d < kDepth - 1; ++d) issue_fill<E, NT>(I, S, nrows, ring_t);
    // with the first copies in flight: the row's scale and statistics (from
    // the sequence's temperature) and the drafted token the keys exclude
    if (tid < nrows) {
      RowInfo &R = S.rows[tid];
      const float T = P.temps[rb];  // both loads issued before either is used
      const int tok = rfj > 0 ? P.tokens[(int64_t)rb * K + R.j] : -1;
      const bool sampled = T > 0.f && T <= 3.4e38f;
      R.s = sampled ? log2e_over(T) : 0.f;
      if (R.kind == kTarget) {
        R.type = sampled ? (P.argmax_out ? kRowEA : kRowE) : kRowA;
      } else if (R.kind == kDraft) {
        R.type = sampled ? (rfj > 0 ? kRowEK : kRowE) : kRowK;
        if (rfj > 0) {
          R.excl = tok;
          if (tok >= R.v0 && tok < R.v1) {  // the piece's vector holding it
            R.qd = ((tok - R.v0) * sz + R.hp) / 16;
            R.qd_step = R.qd / (NT * kU);
          }
        }
      } else {
        R.type = kRowK;
      }
    }
    __syncthreads();
    uint32_t c_off = tid * 16;
    RowAcc<KF> A;
    A.reset();
    const bool chk = P.chk != 0;
#pragma unroll 1
    for (int r = 0; r < nrows; ++r) {
      const RowInfo &R = S.rows[r];
      const int fl = row_flags(R.type, chk);
      const float s = R.s;
      const uint64_t s2 = pk2(s, s);
      const int nsteps = R.nsteps, qd_step = R.qd_step, qd = R.qd, excl = R.excl;
      const int v0 = R.v0, hp = R.hp;
      bool bad = false;
#pragma unroll 1
      for (int step = 0; step < nsteps; ++step) {
        issue_fill<E, NT>(I, S, nrows, ring_t);
        cp_wait<kDepth - 1>();  // this step's copies have landed
        const uint8_t *src = ring + c_off;
        uint4 v[kU];
#pragma unroll
        for (int k = 0; k < kU; ++k) v[k] = *reinterpret_cast<const uint4 *>(src + k * NT * 16);
        step_gen<E, KF, NT>(A, v, step, fl, qd_step, qd, excl, v0, hp, s, s2, bad);
        c_off += kSlot;
        if (c_off >= kDepth * kSlot) c_off -= kDepth * kSlot;
      }
      row_end_gen<E, KF>(A, fl, bad, v0, hp, &wstat[r * NW + warp], &wsel[(r * NW + warp) * KFm]);
    }
    cp_wait<0>();
  }
  __syncthreads();

  // ---- one record per piece: a warp per row, lane w holding warp w's
  // statistics, combined by warp-wide reductions (a warp with a NaN sum,
  // from the finiteness check, makes the piece's sum NaN)
#pragma unroll 1
  for (int r = warp; r < nrows; r += NW) {
    const WStat x = lane < NW ? wstat[r * NW + lane] : WStat{-INFINITY, 0.f, INFINITY, INT32_MAX};
    const float M = rmax_f(x.m);
    const int Ix = rmin_i(x.m == M ? x.idx : INT32_MAX);
    const float C = rmin_f(x.z > 0.f ? x.c : INFINITY);
    const bool poison = ballot(x.z != x.z) != 0u;
    ff Z = ff_warp_sum(x.z > 0.f ? two_prod(x.z, ex2(C - x.c)) : ff{0.f, 0.f});
    if (poison) Z.hi = __int_as_float(0x7fffffff);
    if (lane == 0) {
      float *rec = reinterpret_cast<float *>(P.ws + (int64_t)S.rows[r].rec * kRecBytes);
      *reinterpret_cast<float4 *>(rec) = make_float4(M, __int_as_float(Ix), C, Z.hi);
      rec[4] = Z.lo;
    }
  }
  if (KF > 0) {
#pragma unroll 1
    for (int r = warp; r < nrows; r += NW) {
      const RowInfo &R = S.rows[r];
      if (!(R.type == kRowK || R.type == kRowEK)) continue;
      cta_keys<E, KFm, NT>(R, &wsel[r * NW * KFm], R.v0, R.v1,
                           reinterpret_cast<float2 *>(P.ws + (int64_t)R.rec * kRecBytes + 32));
    }
  }
}

// =================================================================== finish

constexpr int kFinNT = 256;
constexpr int kFinNW = kFinNT / 32;

// Row slots of one sequence in the finish: slot j (0..K) is target row j,
// slot K + 1 + j the draft row j (j < K) or the bonus draft row (j = K).
struct FinS {
  int rflat[kMaxRows];  // the slot's row in the flat stream, -1 if absent
  int pc0[kMaxRows];    // first streaming CTA over the row
  int npc[kMaxRows];    // streaming CTAs over the row (piece records)
  float M[kMaxRows];
  float C[kMaxRows];
  ff Z[kMaxRows];
  int amax[kMaxRows];
  int d[SD_MAX_K];
  float ld_t[SD_MAX_K], ld_d[SD_MAX_K];
  float u_acc[SD_MAX_K];
  float u_draw[SD_MAX_K + 1];
  int2 keys[(SD_MAX_K + 1) * SD_MAX_FANOUT];
  RowInfo dt, dd;  // draw: target and draft row at m on this CTA's slice
  RowInfo ddt;     // the draft row read element-wise on the target's vector grid
  RowInfo geo[2 * SD_MAX_K + 1];  // every row the draw may read: target j, then draft j
  ff wmass[kFinNW];
  ff cmass[2][kMaxCS];  // per-CTA masses of the draw, entry c pushed by CTA c
  ff t_loc, t_w;
  int m, kind, valid, dvalid, fvalid, tok, owner, cstar, wsel;
};

// The sequence's outputs, by one warp: lane j writes token j, the lanes test
// the keys together.
static __device__ void fin_outputs(const Params &P, const FinS &S, int b, bool tvalid) {
  const int lane = threadIdx.x & 31, K = P.K;
  int32_t *out = P.out_tokens + (int64_t)b * (K + 1);
  const bool valid = S.valid != 0;
  const int mm = valid ? S.m : -1, tok = S.tok;
  for (int j = lane; j <= K; j += 32) out[j] = !valid ? -1 : (j < mm ? S.d[j] : (j == mm ? tok : -1));
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
    if (!valid && P.status) {
      int bits = 0;
      if (!tvalid) bits |= (int)SD_STATUS_BAD_TEMP;
      if (!S.dvalid) bits |= (int)SD_STATUS_BAD_TOKEN;
      if (tvalid && S.dvalid && !S.fvalid) bits |= (int)SD_STATUS_NONFINITE;
      atomicOr(P.status, bits);
    }
  }
}

template <typename E>
__global__ void __launch_bounds__(kFinNT, 2) sd_finish_kernel(const __grid_constant__ Params P) {
  constexpr int NT = kFinNT, NW = kFinNW;
  constexpr int sz = Elt<E>::kSize, NV = Elt<E>::kPerVec;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int cs = P.cs;
  const int b = blockIdx.x / cs;
  const int K = P.K;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nslot = 2 * K + 2;

  __shared__ FinS S;
  extern __shared__ __align__(128) float pm[];  // [NW][pw][32] masses of the draw

  // every CTA of the cluster has started before any pushes into its memory
  cluster_arrive_relaxed();

  // ---- prologue: inputs only (the streaming grid may still be running)
  const float T = P.temps[b];
  const bool tvalid = (T >= 0.f) && (T <= 3.4e38f);  // rejects NaN / inf / < 0
  const bool sampled = tvalid && T > 0.f;
  const float s = sampled ? log2e_over(T) : 0.f;
  if (warp == 0) {
    const int d = lane < K ? P.tokens[(int64_t)b * K + lane] : 0;
    const bool dok = lane >= K || (d >= 0 && d < P.V);
    const bool dvalid = __all_sync(0xffffffffu, dok);
    if (lane < K) {
      S.d[lane] = d;
      float lt = -INFINITY, ld = -INFINITY;
      if (sampled && dvalid) {
        lt = Elt<E>::load_global(P.target + (((int64_t)b * (K + 1) + lane) * P.V + d) * sz);
        ld = Elt<E>::load_global(P.draft + (((int64_t)b * K + lane) * P.V + d) * sz);
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
  // this sequence's place among the sampled sequences places its rows in
  // the flat stream; streaming CTA c covered steps [U c / G, U (c+1) / G)
  int ns = 0, rk = 0;
#pragma unroll 1
  for (int x0 = 0; x0 < P.B; x0 += NT) {
    const int x = x0 + tid;
    const float tx = x < P.B ? P.temps[x] : 0.f;
    const bool sx = tx > 0.f && tx <= 3.4e38f;
    ns += __syncthreads_count(sx);
    rk += __syncthreads_count(sx && x < b);
  }
  if (tid < nslot) {
    const int is_x = tid > K, j = is_x ? tid - (K + 1) : tid;
    const int g = K - j;
    int64_t off = 0, rtot = 0;
    for (int x = 0; x <= K; ++x) {
      const int n = P.B + (P.grp_x[x] == 2 ? P.B : (P.grp_x[x] == 1 ? ns : 0));
      if (x < g) off += n;
      rtot += n;
    }
    const int gx = P.grp_x[g];
    const bool xpres = gx == 2 || (gx == 1 && sampled);
    const int64_t r = off + b + (gx == 2 ? b : (gx == 1 ? rk : 0)) + ((!is_x && xpres) ? 1 : 0);
    const int64_t U = rtot * P.spr, G = P.gstream;
    const int c0 = (int)(((r * P.spr + 1) * G - 1) / U);
    const int c1 = (int)(((r + 1) * P.spr * G - 1) / U);
    S.rflat[tid] = (is_x && !xpres) ? -1 : (int)r;
    S.pc0[tid] = c0;
    S.npc[tid] = c1 - c0 + 1;
  }
  // the geometry of every row the draw may read on this CTA's slice (the
  // first rejection picks two of them)
  const int v0 = min(rank * P.slice, P.V);
  const int v1 = min(v0 + P.slice, P.V);
  if (sampled && tid < 2 * K + 1) {
    RowInfo &R = S.geo[tid];
    R.g = tid <= K ? P.target + ((int64_t)b * (K + 1) + tid) * P.V * sz
                   : P.draft + ((int64_t)b * K + (tid - K - 1)) * P.V * sz;
    R.excl = -1;
    row_geometry<NT>(R, v0, v1, sz);
  }
  __syncthreads();

  // ---- the streaming grid has finished and its records are visible
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // ---- row statistics: one warp per row, lane p holding piece p (the same
  // arithmetic in every CTA of the cluster)
  const bool chk = P.chk != 0;
  // the records of two of a warp's rows are loaded together, then reduced
#pragma unroll 1
  for (int r0 = warp; r0 < nslot; r0 += 2 * NW) {
  float4 ra[2];
  float rb[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int r = r0 + i * NW;
    ra[i] = make_float4(-INFINITY, __int_as_float(INT32_MAX), INFINITY, 0.f);
    rb[i] = 0.f;
    if (r < nslot && S.rflat[r] >= 0 && lane < S.npc[r]) {
      const float *rp = reinterpret_cast<const float *>(
          P.ws + (int64_t)(S.pc0[r] + lane + S.rflat[r]) * kRecBytes);
      ra[i] = __ldcg(reinterpret_cast<const float4 *>(rp));
      rb[i] = __ldcg(rp + 4);
    }
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int r = r0 + i * NW;
    if (r >= nslot || S.rflat[r] < 0) continue;
    const CStat x{ra[i].x, __float_as_int(ra[i].y), ra[i].z, ra[i].w, rb[i]};
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
      if (chk && (poison || !(M > -INFINITY))) S.fvalid = 0;
    }
  }
  }
  __syncthreads();

  if (warp == 0) {
    // ---- accept tests, one lane per position (K <= 32)
    const int j = lane;
    const bool dvalid = S.dvalid != 0;
    int rej = 0;
    if (j < K) {
      const int d = S.d[j];
      int a = 0;
      if (!sampled) {
        a = (dvalid && d == S.amax[j]) ? 1 : 0;
      } else if (dvalid) {
        const int rd = K + 1 + j;
        const float lt = S.ld_t[j], ldr = S.ld_d[j];
        // log2 of 2^(l_d s + C), carried as float-float (the products exact)
        const ff xt = ff_add_f(two_prod(lt, s), S.C[j]);
        const ff xd = ff_add_f(two_prod(ldr, s), S.C[rd]);
        const float zt = ff_f(S.Z[j]), zd = ff_f(S.Z[rd]);
        const float r = (ldr == -INFINITY) ? INFINITY  // q(d) = 0
                                           : exp2_ff(ff_sub(xt, xd)) * ff_ratio(S.Z[rd], S.Z[j]);
        a = (S.u_acc[j] <= r) ? 1 : 0;
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
    const int mm = rejects ? __ffs(rejects) - 1 : K;
    const bool valid = tvalid && dvalid && S.fvalid != 0;
    if (sampled && valid && lane < 2 && (lane == 0 || mm < K))  // the rows the draw reads
      (lane == 0 ? S.dt : S.dd) = S.geo[lane == 0 ? mm : K + 1 + mm];
    __syncwarp();
    if (sampled && valid && lane == 0 && mm < K && S.dd.hp != S.dt.hp) {
      S.ddt = S.dt;
      S.ddt.g = S.dd.g;
      S.ddt.qlo = 1;  // every vector assembled from element loads
      S.ddt.qhi = 0;
    }
    if (lane == 0) {
      S.m = mm;
      S.valid = valid ? 1 : 0;
      S.kind = 0;
      S.owner = 0;
      S.tok = -1;
      S.cstar = 0;
      if (valid) {
        if (!sampled) S.tok = S.amax[mm];
        else S.kind = mm < K ? 1 : 2;
      }
    }
    if (rank == 0 && P.argmax_out)
      for (int jj = lane; jj <= K; jj += 32) P.argmax_out[(int64_t)b * (K + 1) + jj] = S.amax[jj];
  } else if (P.keys) {
    // ---- keys of each position: the best fan of the pieces' candidates
    const int kf = P.kf;
#pragma unroll 1
    for (int j = warp - 1; j <= K; j += NW - 1) {
      const int fan = P.fanout[j];
      if (fan <= 0) continue;
      const int xs = K + 1 + j;
      const bool present = S.rflat[xs] >= 0;
      const int ncand = present ? S.npc[xs] * kf : 0;
      constexpr int PER = (kMaxParts * 8 + 31) / 32;
      float cv[PER];
      int ci[PER];
#pragma unroll
      for (int h = 0; h < PER; ++h) {
        const int c = lane + 32 * h;  // candidate c: piece c / kf, rank c % kf
        cv[h] = -INFINITY;
        ci[h] = INT32_MAX;
        if (c < ncand) {
          const float2 e = __ldcg(reinterpret_cast<const float2 *>(
              P.ws + (int64_t)(S.pc0[xs] + c / kf + S.rflat[xs]) * kRecBytes + 32 + (c % kf) * 8));
          cv[h] = e.x;
          ci[h] = __float_as_int(e.y);
        }
      }
      int2 *kdst = &S.keys[P.fan_off[j]];
      int32_t *kout =
          P.keys_out ? P.keys_out + ((int64_t)b * P.n_keys_out + P.fan_off[j]) * 2 : nullptr;
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
          kdst[r2] = key;
          if (rank == 0 && kout) {
            kout[2 * r2] = key.x;
            kout[2 * r2 + 1] = key.y;
          }
        }
      }
    }
  }
  cluster_wait();  // pairs with the arrive at the top: every CTA has started
  __syncthreads();

  // ---- one inverse-CDF draw per sequence (residual at m, or p at K)
#pragma unroll 1
  for (int attempt = 0; attempt < 2 && S.kind != 0; ++attempt) {
    const int mm = S.m;
    const bool residual = S.kind == 1;
    const RowInfo &Rt = S.dt;
    const bool d_vec = residual && S.dd.hp == Rt.hp;  // the same vector grid
    const RowInfo &Rdt = S.ddt;  // otherwise: element-wise on the target's grid
    const float Ct = S.C[mm];
    const float Cd = residual ? S.C[K + 1 + mm] : 0.f;
    const float Rz = residual ? ff_ratio(S.Z[mm], S.Z[K + 1 + mm]) : 0.f;
    const uint64_t s2 = pk2(s, s), ct2 = pk2(Ct, Ct);
    const uint64_t cd2 = pk2(Cd, Cd), r2 = pk2(Rz, Rz);  // draft weights times R
    const int nvec = Rt.nvec;
    const int wr = (nvec + NW - 1) / NW;  // vectors per warp
    const int wq0 = min(warp * wr, nvec), wq1 = min(wq0 + wr, nvec);
    float *pmw = pm + warp * P.pw * 32;  // [iteration][lane] masses of this warp
    const ff lm =
        draw_pass<E>(Rt, S.dd, Rdt, residual, d_vec, wq0, wq1, v0, v1, s2, ct2, cd2, r2, pmw);
    const ff wm = ff_warp_sum(lm);
    if (lane == 0) S.wmass[warp] = wm;
    __syncthreads();
    if (warp == 0) {
      // the CTA's mass into every CTA of the cluster
      const ff m_l = lane < NW ? S.wmass[lane] : ff{0.f, 0.f};
      const ff tot_cta = ff_warp_sum(m_l);
      if (lane < cs) *cluster.map_shared_rank(&S.cmass[attempt][rank], lane) = tot_cta;
    }
    cluster_sync_aligned();  // slice masses are in every CTA
    if (warp == 0) {
      const ff sc = lane < cs ? S.cmass[attempt][lane] : ff{0.f, 0.f};  // lane c: CTA c
      const ff tot = ff_warp_sum(sc);
      if (ff_pos(tot) || !residual) {
        const ff t = ff_mul_f(tot, S.u_draw[mm]);
        const Cross c = ff_cross(sc, t);
        if (lane == 0) {
          S.cstar = c.l < 0 ? 0 : c.l;
          S.t_loc = ff_sub(t, c.before);
          S.owner = S.cstar;
        }
      } else if (lane == 0) {
        S.kind = 2;  // identically zero residual: draw from p at m
      }
    }
    __syncthreads();
    if (S.kind == 2 && residual) continue;  // every CTA takes this branch
    if (rank == S.cstar) {
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
        // the crossing iteration: lane t sums the 32 lane masses of
        // iteration tb + t (reading its row rotated across the banks)
        const int nit = (wq1 - wq0 + 31) / 32;
        ff tw = S.t_w, cum{0.f, 0.f};
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
          const ff rem = ff_sub(tw, cum);
          const Cross c = ff_cross(mt, rem);
          if (c.l >= 0) {  // a crossing here, or the last iteration with mass so far
            isel = tb + c.l;
            t_it = ff_sub(rem, c.before);
            if (c.crossed) break;
          }
          cum = ff_add(cum, c.total);
        }
        int tok = -1;
        if (isel >= 0) {
          // the crossing lane within that iteration
          const Cross cl = ff_cross(ff{pmw[isel * 32 + lane], 0.f}, t_it);
          if (cl.l >= 0) {
            const ff t_l = ff_sub(t_it, cl.before);
            // that lane's vector, one element per lane (index order), the
            // first element past t_l; if rounding leaves none, the last one
            // with weight
            const int q = wq0 + isel * 32 + cl.l;
            const int i = lane % NV;
            uint4 tvv = load_vec_direct<E>(Rt, q, v0, v1);
            uint4 dvv = tvv;
            if (residual)
              dvv = d_vec ? load_vec_direct<E>(S.dd, q, v0, v1) : load_vec_slow<E>(Rdt, q, v0, v1);
            float ww[NV];
            pass_weights<E>(tvv, dvv, residual, s2, ct2, cd2, r2, ww);
            float wi = 0.f;
#pragma unroll
            for (int ii = 0; ii < NV; ++ii)
              if (ii == i) wi = ww[ii];
            const int ei = elem_index(v0, Rt.hp, q, i, sz);
            const bool ok = lane < NV && ei >= v0 && ei < v1 && wi > 0.f;
            const Cross ce = ff_cross(ff{ok ? wi : 0.f, 0.f}, t_l);
            tok = __shfl_sync(0xffffffffu, ei, ce.l < 0 ? 0 : ce.l);
            if (ce.l < 0) tok = -1;
          }
        }
        if (lane == 0) S.tok = tok >= 0 ? tok : S.amax[mm];
      }
      __syncthreads();
    }
    break;
  }

  // ---- the sequence's outputs (owning CTA, one warp)
  if (rank == S.owner && warp == 0) fin_outputs(P, S, b, tvalid);
  // No CTA touches another's shared memory after the last cluster barrier,
  // which every CTA passes, so the CTAs may leave independently.
}

// ===================================================================== host

// Dynamic shared memory the streaming kernel may use: the 227 KB a CTA can
// hold less its static part (Static, the class offsets, the warp counts).
static const int kFlatSmemCap = 227 * 1024 - (int)sizeof(Static) - 1024;
static const int kFinSmemCap = 227 * 1024 - (int)sizeof(FinS) - 256;

template <typename E, int KF, int NT>
static void *flat_fn() {
  static FuncAttrs attrs;
  void *fn = (void *)sd_flat_stream_kernel<E, KF, NT>;
  attrs.apply(fn, kFlatSmemCap, false, "the streaming kernel");
  return fn;
}

template <typename E>
static void *fin_fn() {
  static FuncAttrs attrs;
  void *fn = (void *)sd_finish_kernel<E>;
  attrs.apply(fn, kFinSmemCap, true, "the finish kernel");
  return fn;
}

// Vocabulary slice of one finish CTA: an even share, a multiple of 16
// elements (so a 16-byte aligned row keeps its slices aligned).
static int fin_slice(int V, int cs) { return (int)((((int64_t)V + cs - 1) / cs + 15) / 16 * 16); }

// Iterations of 32 vectors one warp of the finish takes in the draw over a
// slice of `slice` elements (the slice may start off the 16-byte grid).
static int fin_pw(int slice, int sz) {
  const int nvec = (int)(((int64_t)slice * sz + 31) / 16) + 1;
  return ((nvec + kFinNW - 1) / kFinNW + 31) / 32;
}
static int fin_smem(int pw) { return align128(4 * kFinNW * pw * 32); }

// Clusters of cs finish CTAs with `smem` bytes each that the device holds at once.
template <typename E>
static int fin_active_clusters(int cs, int smem) {
  static std::mutex mu;
  static int cache[kMaxDevices][kMaxCS + 1];
  static int cache_smem[kMaxDevices][kMaxCS + 1];
  const int dev = current_device();
  void *fn = fin_fn<E>();
  std::lock_guard<std::mutex> g(mu);
  if (cache_smem[dev][cs] == smem + 1) return cache[dev][cs];
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)cs, 1, 1);
  cfg.blockDim = dim3(kFinNT, 1, 1);
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
  cache[dev][cs] = n;
  cache_smem[dev][cs] = smem + 1;
  return n;
}

// Cluster size of the finish: the largest cs up to about two CTAs per SM for
// which all B clusters are resident at once; if none is, the size that
// leaves the fewest waves.
template <typename E>
static int choose_fin_cs(const Params &P) {
  constexpr int sz = Elt<E>::kSize;
  const int forced = env_int("SDV_CS", 0);
  if (forced >= 1 && forced <= kMaxCS) return forced;
  const int per_sm = std::max(1, env_int("SDV_CPS", 2));
  const int B = std::max(P.B, 1);
  const int target = (int)std::min<int64_t>(
      kMaxCS, std::max<int64_t>(1, (int64_t)per_sm * sm_count() / B));
  int best = -1;
  int64_t best_waves = INT64_MAX;
  for (int cs = target; cs >= 1; --cs) {
    const int smem = fin_smem(fin_pw(fin_slice(P.V, cs), sz));
    if (smem > kFinSmemCap) break;
    const int n = fin_active_clusters<E>(cs, smem);
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
    if (fin_smem(fin_pw(fin_slice(P.V, cs), sz)) <= kFinSmemCap) return cs;
  return kMaxCS;
}

// Groups of the flat stream (see Params): g = 0..K for position K - g.
// rmin / rmax: rows of all sequences when none / all of them are sampled.
static void flat_groups(Params &P, int64_t &rmin, int64_t &rmax) {
  rmin = rmax = 0;
  const bool has_bonus = P.keys && P.bonus && P.fanout[P.K] > 0;
  for (int g = 0; g <= P.K; ++g) {
    const int j = P.K - g;
    int x;
    if (g == 0) x = has_bonus ? 2 : 0;
    else x = (P.keys && P.fanout[j] > 0) ? 2 : 1;
    P.grp_x[g] = (int8_t)x;
    rmax += P.B + (x > 0 ? P.B : 0);
    rmin += P.B + (x == 2 ? P.B : 0);
  }
}

// Bytes of piece records the split launch needs at most: one per row of
// every sequence plus one per streaming CTA (a CTA's range cuts at most one
// row it shares with the next CTA).
size_t split_workspace_bytes(int64_t B, int K) {
  return (size_t)(kMaxStreamGrid + B * (2 * (int64_t)K + 2)) * kRecBytes;
}

template <typename E, int KF>
sd_status_t launch_split(Params &P, size_t ws_bytes, cudaStream_t stream) {
  constexpr int NT = 256, sz = Elt<E>::kSize;
  constexpr int ue = NT * kU * 16 / sz;
  if (P.mode != kVerify || !P.ws || P.B < 1) return SD_ERR_UNSUPPORTED;
  int64_t rmin = 0, rmax = 0;
  flat_groups(P, rmin, rmax);
  P.spr = (P.V + ue - 1) / ue;
  P.kf = KF > 0 ? KF : 1;
  // Two CTAs per SM.  Never more CTAs than steps (no CTA is empty),
  // nor so many that one row spans more than kMaxParts CTAs.
  int64_t G = std::min<int64_t>((int64_t)stream_ctas_per_sm<KF>() * sm_count(), kMaxStreamGrid);
  const int forced = env_int("SDV_GRID", 0);
  if (forced > 0) G = std::min<int64_t>(forced, kMaxStreamGrid);
  G = std::min<int64_t>({G, (int64_t)(kMaxParts - 1) * rmin, rmin * P.spr});
  if (G < 1) return SD_ERR_UNSUPPORTED;
  // a CTA's range must touch at most kMaxRows rows
  const int64_t steps = (rmax * P.spr + G - 1) / G;
  if ((steps + P.spr - 1) / P.spr + 1 > kMaxRows) return SD_ERR_UNSUPPORTED;
  if ((size_t)(G + rmax) * kRecBytes > ws_bytes) return SD_ERR_INVALID_ARG;
  const FlatLayout FL = flat_layout(NT, KF, P.B);
  if (FL.total > kFlatSmemCap) return SD_ERR_UNSUPPORTED;
  P.gstream = (int)G;
  const int cs = choose_fin_cs<E>(P);
  if (cs < 1 || cs > kMaxCS) return SD_ERR_UNSUPPORTED;
  P.cs = cs;
  P.slice = fin_slice(P.V, cs);
  P.rowsplit = 0;
  P.pw = fin_pw(P.slice, sz);
  const int fsmem = fin_smem(P.pw);
  if (fsmem > kFinSmemCap) return SD_ERR_UNSUPPORTED;

  // the streaming grid: a programmatic dependent of the stream's previous
  // kernel (it waits for it before reading anything)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)G, 1, 1);
  cfg.blockDim = dim3(NT, 1, 1);
  cfg.dynamicSmemBytes = (size_t)FL.total;
  cfg.stream = stream;
  cudaLaunchAttribute attr0[1];
  attr0[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr0[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr0;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, (void (*)(const Params))flat_fn<E, KF, NT>(), P);
  if (e != cudaSuccess) {
    fprintf(stderr, "sd_verify stream launch failed: %s\n", cudaGetErrorString(e));
    return SD_ERR_CUDA;
  }
  // the finish: one cluster per sequence, a programmatic dependent
  cudaLaunchConfig_t cfg2 = {};
  cfg2.gridDim = dim3((unsigned)(P.B * cs), 1, 1);
  cfg2.blockDim = dim3(kFinNT, 1, 1);
  cfg2.dynamicSmemBytes = (size_t)fsmem;
  cfg2.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg2.attrs = attr;
  cfg2.numAttrs = 2;
  if (env_int("SDV_VERBOSE", 0))
    fprintf(stderr, "sd_verify split: B=%d K=%d V=%d G=%d spr=%d cs=%d slice=%d KF=%d "
            "smem=%d/%d\n", P.B, P.K, P.V, (int)G, P.spr, cs, P.slice, KF, FL.total, fsmem);
  e = cudaLaunchKernelEx(&cfg2, (void (*)(const Params))fin_fn<E>(), P);
  if (e != cudaSuccess) {
    fprintf(stderr, "sd_verify finish launch failed: %s\n", cudaGetErrorString(e));
    return SD_ERR_CUDA;
  }
  if (P.compact) return launch_compact_after(P, stream);
  return SD_OK;
}

template sd_status_t launch_split<float, 0>(Params &, size_t, cudaStream_t);
template sd_status_t launch_split<float, 2>(Params &, size_t, cudaStream_t);
template sd_status_t launch_split<float, 4>(Params &, size_t, cudaStream_t);
template sd_status_t launch_split<float, 8>(Params &, size_t, cudaStream_t);
template sd_status_t launch_split<__nv_bfloat16, 0>(Params &, size_t, cudaStream_t);
template sd_status_t launch_split<__nv_bfloat16, 2>(Params &, size_t, cudaStream_t);
template sd_status_t launch_split<__nv_bfloat16, 4>(Params &, size_t, cudaStream_t);
template sd_status_t launch_split<__nv_bfloat16, 8>(Params &, size_t, cudaStream_t);

}  // namespace sdv
