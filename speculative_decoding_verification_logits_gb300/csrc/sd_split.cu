// Split launch of the verify step: a flat streaming grid, then the
// per-sequence finish.
//
// The cluster kernel gives each sequence its own cluster, which leaves SMs
// unevenly loaded whenever the clusters do not tile the device exactly, and
// makes every CTA of a cluster wait for the slowest one before the accept
// scan.  Here the streaming is one grid of about two CTAs per SM over all
// logit rows of all sequences laid end to end.  Every CTA gets the same
// number of streaming steps (16 KB each), so every SM moves the same number
// of bytes.  Rows are grouped by position, j = K first: in group j, sequence
// after sequence, draft row j (the bonus draft row for j = K), when the
// sequence needs it, then target row j.  Draft rows with keys and target
// rows alternate, so every CTA sees the same mix of row kinds.  A CTA's
// range usually cuts one or two rows.
// It writes, per row piece, the statistics the combine needs (max,
// lowest-index argmax, offset exp-sum) and its best key candidates, to a
// record in caller-provided scratch.  The rows of the first positions, where
// a rejection is likeliest, come last in the flat order (streamed by the
// last CTAs of the grid); the draw re-reads its two rows from L2 when a
// round's logits fit there, from HBM otherwise.
//
// The finish is sd_seq_kernel<..., SPLIT = true>: one cluster per sequence,
// launched as a programmatic dependent of the streaming grid; its CTAs take
// the place of streaming CTAs as those exit (the register file holds no
// more) and run their prologue (row table, drafted tokens, their logits, the
// uniforms, the sequence's place in the flat order).  After griddepcontrol.wait
// it combines the records of each of its rows in the same order in every CTA,
// merges the key candidates, and continues exactly as the cluster kernel does
// after its first exchange: accept scan, one inverse-CDF draw over the
// cluster's vocabulary slices, outputs.  The packing launch follows as before.

#include "sd_device.cuh"

namespace sdv {

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

template <typename E, int KF, int NT>
__global__ void __launch_bounds__(NT, 2) sd_flat_stream_kernel(const __grid_constant__ Params P) {
  constexpr int sz = Elt<E>::kSize;
  constexpr int KFm = KF > 0 ? KF : 1;
  constexpr int NW = NT / 32;
  constexpr int ue = NT * kU * 16 / sz;  // elements per streaming step
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = P.K;

  __shared__ Static S;
  __shared__ int goff[SD_MAX_K + 2];
  __shared__ int wcnt[kMaxWarps];
  extern __shared__ __align__(128) uint8_t dyn[];
  // Launched as a programmatic dependent of the stream's previous kernel:
  // nothing is read before that kernel has finished.  Then the finish grid
  // may be scheduled at once: its CTAs take the place of streaming CTAs as
  // those exit and run their prologue meanwhile (reading only inputs, now
  // complete; their griddepcontrol.wait still waits for this whole grid).
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
    const float T = P.temps[b];
    const bool sampled = T > 0.f && T <= 3.4e38f;
    RowInfo &R = S.rows[tid];
    R.kind = isx ? (g == 0 ? kBonus : kDraft) : kTarget;
    R.j = j;
    R.s = sampled ? log2e_over(T) : 0.f;
    R.rec = blockIdx.x + (int)r;
    R.excl = -1;
    R.fan = 0;
    if (R.kind == kTarget) {
      R.g = P.target + ((int64_t)b * (K + 1) + j) * P.V * sz;
      R.type = sampled ? (P.argmax_out ? kRowEA : kRowE) : kRowA;
    } else if (R.kind == kDraft) {
      const int fj = P.keys ? P.fanout[j] : 0;
      R.g = P.draft + ((int64_t)b * K + j) * P.V * sz;
      R.type = sampled ? (fj > 0 ? kRowEK : kRowE) : kRowK;
      R.fan = fj;
      if (fj > 0) R.excl = P.tokens[(int64_t)b * K + j];
    } else {
      R.g = P.bonus + (int64_t)b * P.V * sz;
      R.type = kRowK;
      R.fan = P.fanout[K];
    }
    const int64_t r0 = r * P.spr;
    const int64_t a = (u_lo > r0 ? u_lo : r0) - r0;
    const int64_t e = (u_hi < r0 + P.spr ? u_hi : r0 + P.spr) - r0;
    row_geometry<NT>(R, (int)(a * ue), (int)(e * ue < P.V ? e * ue : (int64_t)P.V), sz);
  }
  __syncthreads();

  // ---- stream the pieces (the same row loops as the cluster kernel, with
  // each row's own scale)
  {
    Issuer I;
    I.row = 0;
    I.slot = ring_t;
    issuer_row<NT>(I, S, nrows);
#pragma unroll
    for (int d = 0; d < kDepth - 1; ++d) issue_step<NT>(I, S, nrows, ring_t);
    uint32_t c_off = tid * 16;
    RowAcc<KF> A;
    A.reset();
    for (int r = 0; r < nrows; ++r) {
      const RowInfo &R = S.rows[r];
      WStat *ws = &wstat[r * NW + warp];
      int *wk = &wsel[(r * NW + warp) * KFm];
      const float s = R.s;
      const uint64_t s2 = pk2(s, s);
      switch (R.type) {
        case kRowE:
          stream_row<E, KF, NT, true, false, false>(A, R, I, S, nrows, ring, ring_t, c_off, R.v0, R.v1,
                                                   s, s2, ws, wk);
          break;
        case kRowEA:
          stream_row<E, KF, NT, true, true, false>(A, R, I, S, nrows, ring, ring_t, c_off, R.v0, R.v1,
                                                  s, s2, ws, wk);
          break;
        case kRowA:
          stream_row<E, KF, NT, false, true, false>(A, R, I, S, nrows, ring, ring_t, c_off, R.v0,
                                                   R.v1, s, s2, ws, wk);
          break;
        default:
          if (KF > 0) {
            if (R.type == kRowK)
              stream_row<E, KF, NT, false, false, (KF > 0)>(A, R, I, S, nrows, ring, ring_t, c_off,
                                                            R.v0, R.v1, s, s2, ws, wk);
            else
              stream_row<E, KF, NT, true, false, (KF > 0)>(A, R, I, S, nrows, ring, ring_t, c_off,
                                                           R.v0, R.v1, s, s2, ws, wk);
          }
          break;
      }
    }
    cp_wait<0>();
  }
  __syncthreads();

  // ---- one record per piece: the warps combined as in the cluster kernel
  if (tid < nrows) {
    const int r = tid;
    float M = -INFINITY;
#pragma unroll 1
    for (int w = 0; w < NW; ++w) M = fmaxf(M, wstat[r * NW + w].m);
    int Ix = INT32_MAX;
    float C = INFINITY;
#pragma unroll 1
    for (int w = 0; w < NW; ++w) {
      const WStat x = wstat[r * NW + w];
      if (x.m == M) Ix = min(Ix, x.idx);
      if (x.z > 0.f) C = fminf(C, x.c);
    }
    ff Z{0.f, 0.f};
#pragma unroll 1
    for (int w = 0; w < NW; ++w) {
      const WStat x = wstat[r * NW + w];
      if (x.z > 0.f) Z = ff_add(Z, two_prod(x.z, ex2(C - x.c)));
    }
    float *rec = reinterpret_cast<float *>(P.ws + (int64_t)S.rows[r].rec * kRecBytes);
    *reinterpret_cast<float4 *>(rec) = make_float4(M, __int_as_float(Ix), C, Z.hi);
    rec[4] = Z.lo;
  }
  if (KF > 0) {
    for (int r = warp; r < nrows; r += NW) {
      const RowInfo &R = S.rows[r];
      if (!(R.type == kRowK || R.type == kRowEK)) continue;
      cta_keys<E, KFm, NT>(R, &wsel[r * NW * KFm], R.v0, R.v1,
                           reinterpret_cast<float2 *>(P.ws + (int64_t)R.rec * kRecBytes + 32));
    }
  }
}

// ------------------------------------------------------------------- host --
// Dynamic shared memory the streaming kernel may use: the 227 KB a CTA can
// hold less its static part (Static, the class offsets, the warp counts).
static const int kFlatSmemCap = 227 * 1024 - (int)sizeof(Static) - 1024;

template <typename E, int KF, int NT>
static void *flat_fn() {
  static std::once_flag once;
  void *fn = (void *)sd_flat_stream_kernel<E, KF, NT>;
  std::call_once(once, [fn] {
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kFlatSmemCap) !=
        cudaSuccess)
      fprintf(stderr, "sd_verify: shared-memory limit of the streaming kernel not set: %s\n",
              cudaGetErrorString(cudaGetLastError()));
  });
  return fn;
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
  // About two CTAs per SM.  Never more CTAs than steps (no CTA is empty),
  // nor so many that one row spans more than kMaxParts CTAs.
  int64_t G = std::min<int64_t>(2LL * sm_count(), kMaxStreamGrid);
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
  const int cs = choose_cs<E, KF, NT, true>(P);
  if (cs < 1 || cs > kMaxCS) return SD_ERR_UNSUPPORTED;
  P.cs = cs;
  P.slice = slice_for(P.V, cs, sz, NT);
  P.rowsplit = 0;
  const Layout L = make_layout(NT, rows_per_seq(P), P.K + 1, KF, cs, P.slice, sz);
  if (L.total > kDynSmemCap) return SD_ERR_UNSUPPORTED;

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
  cfg2.blockDim = dim3(NT, 1, 1);
  cfg2.dynamicSmemBytes = (size_t)L.total;
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
            "smem=%d/%d\n", P.B, P.K, P.V, (int)G, P.spr, cs, P.slice, KF, FL.total, L.total);
  e = cudaLaunchKernelEx(&cfg2, (void (*)(const Params))kernel_fn<E, KF, NT, true>(), P);
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
