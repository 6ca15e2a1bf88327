// GB300 (sm_103a) library of the speculative-decoding verify step: the C ABI
// entry points, their argument checks and the choice of launch plan, the
// packing kernels and the uniforms audit kernel.
//
// Two launch plans compute the verify step (the kernels are in
// sd_device.cuh and sd_split.cu):
//  * the cluster kernel: one thread-block cluster per sequence.  Its CTAs
//    split the vocabulary (or the sequence's rows laid end to end) and
//    stream every logit row of the sequence once -- target rows K..0, draft
//    rows K-1..0, the optional draft row of the bonus position -- keeping
//    per-row statistics in registers (max, lowest-index argmax, the sum of
//    2^(l s + c), the vectors that can hold the top-F keys).  One exchange
//    over distributed shared memory gives every CTA the statistics of all
//    positions, so every CTA runs the left-to-right accept scan itself and
//    they agree on the first rejection m.  One inverse-CDF draw follows:
//    over the residual max(0, p - q) at m, or over p at the bonus position;
//    the CTAs re-read their slices of those rows (streamed last, so mostly
//    from L2), exchange slice masses, and the CTA holding the crossing point
//    scans it.  The owning CTA writes the sequence's tokens and tau.
//  * the split launch (with caller scratch): a flat streaming grid over the
//    rows of all sequences writes per-piece statistics, and a per-sequence
//    finish -- the cluster kernel's code after its exchange -- combines them.
// A one-CTA packing launch follows either as its programmatic dependent.
// Nothing waits on another cluster and there are no spin-waits.
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
#include "sd_device.cuh"

namespace sdv {


__global__ void sd_compact_kernel(int B, int K, const int32_t *out_tokens, const int32_t *tau,
                                  int32_t *offsets, int32_t *packed, int32_t *status) {
  __shared__ int red[32];
  compact_block(B, K, out_tokens, tau, offsets, packed, status, false, red);
}


__global__ void sd_uniforms_kernel(uint64_t seed, int n, const int32_t *row, const int32_t *pos,
                                   const int32_t *slot, double *out) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) out[i] = (double)uniform_u(seed, row[i], pos[i], slot[i]);
}



template <typename E, int KF, int NT>
static sd_status_t launch_nt(Params &P, cudaStream_t stream) {
  constexpr int sz = Elt<E>::kSize;
  const int cs = choose_cs<E, KF, NT>(P);
  if (cs < 1 || cs > kMaxCS) return SD_ERR_INVALID_ARG;
  P.cs = cs;
  P.slice = slice_for(P.V, cs, sz, NT);
  // Row-major split where a slice of every row would leave each CTA at most
  // two streaming steps per row (per-row work then outweighs the steps);
  // SDV_ROWSPLIT=0/1 forces either.
  {
    const int rs = env_int("SDV_ROWSPLIT", -1);
    P.rowsplit = rs >= 0 ? (rs ? 1 : 0) : (P.slice <= 2 * (NT * kU * 16 / sz) ? 1 : 0);
  }
  const Layout L = make_layout(NT, rows_per_seq(P), P.K + 1, KF, cs, P.slice, sz);
  if (L.total > kDynSmemCap) return SD_ERR_UNSUPPORTED;
  void *fn = kernel_fn<E, KF, NT>();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(P.B * cs), 1, 1);
  cfg.blockDim = dim3(NT, 1, 1);
  cfg.dynamicSmemBytes = (size_t)L.total;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // a programmatic dependent of the stream's previous kernel: the kernel
  // waits for it before reading anything, the launch overlaps its tail
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (env_int("SDV_VERBOSE", 0))
    fprintf(stderr,
            "sd_verify: mode=%d B=%d K=%d V=%d cs=%d NT=%d slice=%d rowsplit=%d KF=%d smem=%d\n",
            P.mode, P.B, P.K, P.V, cs, NT, P.slice, P.rowsplit, KF, L.total);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, (void (*)(const Params))fn, P);
  if (e != cudaSuccess) {
    fprintf(stderr, "sd_verify launch failed: %s\n", cudaGetErrorString(e));
    return SD_ERR_CUDA;
  }
  if (P.compact) return launch_compact_after(P, stream);
  return SD_OK;
}

// With scratch from the caller, the split launch (a flat streaming grid over
// all sequences' rows, every SM moving the same bytes, then the compact
// finish); without scratch, or when the request is outside the split
// launch's limits, the cluster kernel.  SDV_SPLIT=0 forces the cluster
// kernel.
template <typename E, int KF>
static sd_status_t launch_kf(Params &P, cudaStream_t s) {
  const int mode = env_int("SDV_SPLIT", -1);
  const bool split = P.ws != nullptr && mode != 0 && P.mode == kVerify;
  if (split) {
    const sd_status_t st = launch_split<E, KF>(P, P.ws_bytes, s);
    if (st != SD_ERR_UNSUPPORTED) return st;
  }
  return launch_nt<E, KF, 256>(P, s);
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
  return split_workspace_bytes(B, K);
}

sd_status_t sd_verify(const sd_verify_args *a, void *stream) {
  sdv::NvtxRange nvtx_range("sd_verify");
  if (!a) return SD_ERR_INVALID_ARG;
  if (a->B < 0 || a->K < 0 || a->K > SD_MAX_K || a->V < 1 || a->V > SD_MAX_V)
    return SD_ERR_INVALID_ARG;
  if (a->dtype != SD_F32 && a->dtype != SD_BF16) return SD_ERR_INVALID_ARG;
  if ((int64_t)a->B * kMaxCS > INT32_MAX) return SD_ERR_INVALID_ARG;
  const bool predict = (a->flags & SD_FLAG_PREDICT) != 0;
  const bool compact = (a->flags & SD_FLAG_COMPACT) != 0;
  if (a->flags & ~(SD_FLAG_PREDICT | SD_FLAG_COMPACT | SD_FLAG_CHECK_FINITE))
    return SD_ERR_INVALID_ARG;
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
  if (a->workspace && !aligned(a->workspace, 16)) return SD_ERR_INVALID_ARG;
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
  P.chk = (a->flags & SD_FLAG_CHECK_FINITE) ? 1 : 0;
  P.ws = (uint8_t *)a->workspace;
  P.ws_bytes = a->workspace ? a->workspace_bytes : 0;
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
  sdv::NvtxRange nvtx_range("sd_outcome_predict");
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
  sdv::NvtxRange nvtx_range("sd_compact");
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
  sdv::NvtxRange nvtx_range("sd_uniforms");
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
