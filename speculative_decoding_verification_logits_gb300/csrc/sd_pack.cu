// The drafter's next pass, packed from the verify step's outcome keys
// ("LLMの生成を5倍速くする「D3D」を図で読む" (animemo.app), sections
// 答え:ありうる結果すべてに、先回りして下書きする and パック:24ブロックを
// 1回の計算で): every possible outcome of the round under verification
// (a rejection at draft k replaced by candidate c, or all drafts accepted
// and a bonus token c) gets a block of K+1 tokens -- c as its anchor and K
// mask tokens to be drafted -- and all of them, together with the block
// under verification, go into one input of the drafter.  Each block sees
// the shared prefix, the first k+1 tokens of the block under verification
// (its anchor and the drafts a rejection at k keeps) and itself; that count
// is the block's ctx.
//
// Integer layout work: one thread per slot of the pack, consecutive threads
// on consecutive slots of a block, so every read and write is coalesced.
// For the D3D shape (K = 15, 23 keys, 16 sequences) the pack is 48 KB of
// output; the launch is latency-bound.

#include "sd_device.cuh"

namespace sdv {

__global__ void __launch_bounds__(256) sd_d3d_pack_kernel(
    int B, int K, int n_keys, const int2 *keys, const int32_t *draft_tokens,
    const int32_t *anchor, const int32_t *anchor_pos, int32_t mask, int32_t *tokens,
    int32_t *positions, int32_t *ctx, int64_t total) {
  // a programmatic dependent of the stream's previous kernel: nothing is read
  // before it has finished; the next launch may be scheduled at once
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int L = K + 1, nb = 1 + n_keys;
  for (int64_t x = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; x < total;
       x += (int64_t)gridDim.x * blockDim.x) {
    const int i = (int)(x % L);            // slot in the block
    const int64_t bb = x / L;              // b * nb + block
    const int blk = (int)(bb % nb);
    const int b = (int)(bb / nb);
    int t, p, c;
    if (blk == 0) {  // the block under verification: anchor, then the drafts
      t = i == 0 ? __ldg(anchor + b) : __ldg(draft_tokens + (int64_t)b * K + (i - 1));
      p = __ldg(anchor_pos + b) + i;
      c = 0;
    } else {
      const int2 key = __ldg(keys + (int64_t)b * n_keys + (blk - 1));
      if (key.x < 0 || key.x > K || key.y < 0) {  // empty key slot: empty block
        t = p = c = -1;
      } else {  // c replaces draft k (or follows all K): its position, then masks
        t = i == 0 ? key.y : mask;
        p = __ldg(anchor_pos + b) + 1 + key.x + i;
        c = key.x + 1;
      }
    }
    tokens[x] = t;
    positions[x] = p;
    if (i == 0) ctx[bb] = c;
  }
}

}  // namespace sdv

using namespace sdv;

extern "C" sd_status_t sd_d3d_pack(int32_t B, int32_t K, int32_t n_keys, const int32_t *keys,
                                   const int32_t *draft_tokens, const int32_t *anchor,
                                   const int32_t *anchor_pos, int32_t mask_token,
                                   int32_t *tokens, int32_t *positions, int32_t *ctx,
                                   void *stream) {
  sdv::NvtxRange nvtx_range("sd_d3d_pack");
  if (B < 0 || K < 0 || K > SD_MAX_K || n_keys < 0 || n_keys > (SD_MAX_K + 1) * SD_MAX_FANOUT)
    return SD_ERR_INVALID_ARG;
  if (B == 0) return SD_OK;
  if (!anchor || !anchor_pos || !tokens || !positions || !ctx) return SD_ERR_INVALID_ARG;
  if ((K > 0 && !draft_tokens) || (n_keys > 0 && !keys)) return SD_ERR_INVALID_ARG;
  if (keys && ((uintptr_t)keys % 8) != 0) return SD_ERR_INVALID_ARG;  // read as int2 pairs
  const int64_t total = (int64_t)B * (1 + n_keys) * (K + 1);
  const int64_t blocks = std::min<int64_t>((total + 255) / 256, 8LL * sm_count());
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks, 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = (cudaStream_t)stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, sd_d3d_pack_kernel, (int)B, (int)K, (int)n_keys,
                                           reinterpret_cast<const int2 *>(keys), draft_tokens,
                                           anchor, anchor_pos, mask_token, tokens, positions, ctx,
                                           total);
  return e == cudaSuccess ? SD_OK : SD_ERR_CUDA;
}
