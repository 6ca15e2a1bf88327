// KV-cache rollback after a verify round ("What is speculative decoding"
// explainer (lotook.com), FAQ on speculative decoding and the KV cache: the
// engine rolls both models' KV caches back and truncates them, dropping the
// entries of rejected drafts before the next cycle).
//
// Row b holds kv_len[b] entries in pages of page_size entries listed in
// block_table[b][..]; the round appended `appended` of them and confirms
// the first tau[b].  One CTA: a thread per row computes the new length and
// how many pages it frees, a block-wide scan gives every row its place in
// the packed list of freed page ids, and the row moves its freed ids there
// and clears their table slots.  Rows beyond the CTA's size are taken in
// further passes, the scan carried over.

#include "sd_device.cuh"

namespace sdv {

__global__ void __launch_bounds__(1024) sd_kv_rollback_kernel(
    int B, int page_size, int max_pages, int appended, const int32_t *kv_len,
    const int32_t *tau, int32_t *block_table, int32_t *new_len, int32_t *freed,
    int32_t *free_offsets) {
  // a programmatic dependent of the stream's previous kernel: nothing is read
  // before it has finished; the next launch may be scheduled at once
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __shared__ int red[32];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int carry = 0;
  for (int base = 0; base < B; base += blockDim.x) {
    const int b = base + threadIdx.x;
    int nf = 0, still = 0, used = 0;
    if (b < B) {
      const int kv = kv_len[b];
      const int before = max(kv - appended, 0);  // entries older than the round
      const int keep = min(min(max(tau[b], 0), appended), kv - before);
      const int n_new = before + keep;
      used = min((kv + page_size - 1) / page_size, max_pages);
      still = (n_new + page_size - 1) / page_size;
      nf = max(used - still, 0);
      new_len[b] = n_new;
    }
    // exclusive scan of the freed-page counts over the CTA
    int x = nf;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      x += lane >= o ? y : 0;
    }
    if (lane == 31) red[w] = x;
    __syncthreads();
    if (w == 0) {
      int v = lane < nw ? red[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, v, o);
        v += lane >= o ? y : 0;
      }
      if (lane < nw) red[lane] = v;
    }
    __syncthreads();
    const int at = carry + (w > 0 ? red[w - 1] : 0) + x - nf;
    if (b < B) {
      free_offsets[b] = at;
      int32_t *row = block_table + (int64_t)b * max_pages;
      for (int p = max(still, 0); p < used; ++p) {
        freed[at + (p - still)] = row[p];
        row[p] = -1;
      }
    }
    carry += red[nw - 1];
    __syncthreads();
  }
  if (threadIdx.x == 0) free_offsets[B] = carry;
}

}  // namespace sdv

using namespace sdv;

extern "C" sd_status_t sd_kv_rollback(int32_t B, int32_t page_size, int32_t max_pages,
                                      int32_t appended, const int32_t *kv_len,
                                      const int32_t *tau, int32_t *block_table,
                                      int32_t *new_len, int32_t *freed, int32_t *free_offsets,
                                      void *stream) {
  sdv::NvtxRange nvtx_range("sd_kv_rollback");
  if (B < 0 || page_size < 1 || max_pages < 0 || appended < 0 || !free_offsets)
    return SD_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  if (B == 0)
    return cudaMemsetAsync(free_offsets, 0, sizeof(int32_t), s) == cudaSuccess ? SD_OK
                                                                             : SD_ERR_CUDA;
  if (!kv_len || !tau || !new_len || (max_pages > 0 && (!block_table || !freed)))
    return SD_ERR_INVALID_ARG;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1, 1, 1);
  cfg.blockDim = dim3(1024, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, sd_kv_rollback_kernel, (int)B, (int)page_size,
                                           (int)max_pages, (int)appended, kv_len, tau,
                                           block_table, new_len, freed, free_offsets);
  return e == cudaSuccess ? SD_OK : SD_ERR_CUDA;
}
