// N-gram / prompt-lookup drafting ("What is speculative decoding"
// explainer (lotook.com), FAQ on drafting without a separate model: find a
// span of the prompt and recent output matching the text's ending and copy
// the tokens that follow it; "Speculative Speculative Decoding" blog
// (jiwasawa.github.io), Saguaro fallback: an n-gram model as the light
// drafter at large batch).
//
// For each sequence, among the places j (1 <= j < len) where a copy could
// start, the best is the one whose preceding tokens share the longest
// suffix with the history (capped at n_max, at least n_min), latest first:
// the same as trying n = n_max..n_min and taking the latest earlier
// occurrence of the last n tokens.  A cluster of up to four CTAs per row;
// in round r thread t takes the kJP places j = len - 1 - t - q NT - r NT kJP,
// computes the common suffix length c(j) by comparing h[j-1-s] with
// h[len-1-s] (consecutive threads read consecutive tokens), and keeps the
// maximum of the packed key (c << 26 | j).  CTA i of the cluster takes the
// rounds i, i + cs, ...; a round whose CTA maximum has c = n_max ends that
// CTA's scan (its later rounds hold smaller j); an atomic maximum in rank
// 0's shared memory and one cluster barrier give the row's key.

#include "sd_device.cuh"

namespace sdv {

constexpr int kNgramMax = 16;   // longest n-gram compared
constexpr int kJBits = 26;      // j < 2^26 in the packed key
constexpr int kJP = 8;          // positions per thread per round
constexpr int kNgramCS = 4;     // CTAs per row (a cluster)

template <int NT>
__global__ void __launch_bounds__(NT) sd_ngram_kernel(int L, int K, int n_max, int n_min,
                                                      const int32_t *history,
                                                      const int32_t *lengths, int32_t *drafts,
                                                      int32_t *count, int32_t *match_pos,
                                                      int32_t *match_n) {
  constexpr int NW = NT / 32;
  cg::cluster_group cluster = cg::this_cluster();
  const int cs = (int)cluster.num_blocks(), rank = (int)cluster.block_rank();
  const int b = blockIdx.x / cs, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // a programmatic dependent of the stream's previous kernel: nothing is read
  // before it has finished; the next launch may be scheduled at once
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int32_t *h = history + (int64_t)b * L;
  const int n_tok = min(max(__ldg(lengths + b), 0), L);
  __shared__ int32_t pat[kNgramMax];   // pat[s] = h[len-1-s]
  __shared__ unsigned wbest[NW];
  __shared__ unsigned best;            // this CTA's best key
  __shared__ unsigned cbest;           // rank 0: the cluster's best key
  if (tid < n_max) pat[tid] = tid < n_tok ? __ldg(h + n_tok - 1 - tid) : -1;
  if (tid == 0) best = cbest = 0u;
  cluster_sync_aligned();  // every CTA has started (and zeroed cbest) before any push
  // CTA `rank` of the row's cluster takes rounds rank, rank + cs, ...: its
  // own rounds hold decreasing places, so a full-length match ends them
  for (int j0 = n_tok - 1 - rank * NT * kJP; j0 >= 1; j0 -= cs * NT * kJP) {
    // kJP places per thread per round, NT apart, so that every load of the
    // round is coalesced and kJP of them are in flight per thread
    int32_t last[kJP];
#pragma unroll
    for (int q = 0; q < kJP; ++q) {
      const int j = j0 - tid - q * NT;
      last[q] = j >= 1 ? __ldg(h + j - 1) : -1;
    }
    unsigned key = 0u;
#pragma unroll
    for (int q = 0; q < kJP; ++q) {
      const int j = j0 - tid - q * NT;
      if (j >= 1 && last[q] == pat[0]) {
        int c = 1;
        while (c < n_max && j - 1 - c >= 0 && __ldg(h + j - 1 - c) == pat[c]) ++c;
        if (c >= n_min) key = max(key, ((unsigned)c << kJBits) | (unsigned)j);
      }
    }
    key = __reduce_max_sync(0xffffffffu, key);
    if (lane == 0) wbest[warp] = key;
    __syncthreads();
    if (tid == 0) {
      unsigned m = best;
      for (int w = 0; w < NW; ++w) m = max(m, wbest[w]);
      best = m;
    }
    __syncthreads();
    if ((best >> kJBits) == (unsigned)n_max) break;  // nothing later can beat it
  }
  if (tid == 0) atomicMax(cluster.map_shared_rank(&cbest, 0), best);
  cluster_sync_aligned();  // every CTA's best is in rank 0
  if (rank != 0) return;
  const unsigned key = cbest;
  const int c = (int)(key >> kJBits), j = (int)(key & ((1u << kJBits) - 1u));
  for (int k = tid; k < K; k += NT) {
    const int src = j + k;
    drafts[(int64_t)b * K + k] = (key != 0u && src < n_tok) ? __ldg(h + src) : -1;
  }
  if (tid == 0) {
    count[b] = key != 0u ? min(K, n_tok - j) : 0;
    match_pos[b] = key != 0u ? j - c : -1;
    match_n[b] = key != 0u ? c : -1;
  }
}

}  // namespace sdv

using namespace sdv;

extern "C" sd_status_t sd_ngram_draft(int32_t B, int32_t L, int32_t K, int32_t n_max,
                                      int32_t n_min, const int32_t *history,
                                      const int32_t *lengths, int32_t *drafts, int32_t *count,
                                      int32_t *match_pos, int32_t *match_n, void *stream) {
  sdv::NvtxRange nvtx_range("sd_ngram_draft");
  if (B < 0 || L < 0 || L >= (1 << kJBits) || K < 0 || K > SD_MAX_K) return SD_ERR_INVALID_ARG;
  if (n_min < 1 || n_max < n_min || n_max > kNgramMax) return SD_ERR_INVALID_ARG;
  if (B == 0) return SD_OK;
  if (!history || !lengths || !count || !match_pos || !match_n || (K > 0 && !drafts))
    return SD_ERR_INVALID_ARG;
  // a cluster of CTAs per row: rows of up to one round need one CTA, longer
  // ones split their rounds over up to kNgramCS CTAs
  const int64_t rounds = ((int64_t)L + 256 * kJP - 1) / (256 * kJP);
  const int cs = (int)std::max<int64_t>(1, std::min<int64_t>(kNgramCS, rounds));
  if ((int64_t)B * cs > INT32_MAX) return SD_ERR_INVALID_ARG;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(B * cs), 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = (cudaStream_t)stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, sd_ngram_kernel<256>, L, K, n_max, n_min,
                                           history, lengths, drafts, count, match_pos, match_n);
  return e == cudaSuccess ? SD_OK : SD_ERR_CUDA;
}
