// Allocation-free entry point: sd_verify with a scratch area that lives in
// the library itself.
//
// Some callers cannot allocate device memory at the point where they verify
// a round: a runtime whose memory is fully carved up by its own pool before
// serving starts, a plugin that is handed only the tensors it works on, or
// code that must not call into an allocator between two steps.  For them
// sd_verify_noalloc runs the split launch (flat streaming grid, then the
// per-sequence finish) with its piece records in g_sd_scratch below, a
// file-scope device array of kStaticScratchBytes that every GPU which loads
// this library holds until the process exits.  The caller still passes all
// inputs and outputs.
//
// Host code cannot hand g_sd_scratch to a kernel by name: on the host that
// name is a stand-in object, not a device address.  The first call on each
// device therefore looks the array's device address up with
// cudaGetSymbolAddress, with that device current, and keeps it; later calls
// reuse it.

#include "sd_device.cuh"

namespace sdv {

// Piece records of the split launch for (G + rows) <= 21845 records of 96
// bytes: (1024 + B (2K + 2)) <= 21845, e.g. B = 256 sequences at K = 32.
constexpr size_t kStaticScratchBytes = (size_t)2 << 20;
static __device__ __align__(256) uint8_t g_sd_scratch[kStaticScratchBytes];

static std::mutex g_scratch_mu;
static void *g_scratch_addr[kMaxDevices];

// Device address of g_sd_scratch on the current device (looked up once).
static sd_status_t static_scratch(void **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return SD_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return SD_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> g(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_sd_scratch);
    if (e != cudaSuccess || !p) {
      fprintf(stderr, "sd_verify_noalloc: no device address for the static scratch: %s\n",
              cudaGetErrorString(e));
      return SD_ERR_CUDA;
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return SD_OK;
}

}  // namespace sdv

using namespace sdv;

extern "C" sd_status_t sd_verify_noalloc(const sd_verify_args *args, void *stream) {
  sdv::NvtxRange nvtx_range("sd_verify_noalloc");
  if (!args) return SD_ERR_INVALID_ARG;
  if (args->workspace || args->workspace_bytes)
    return SD_ERR_INVALID_ARG;  // the static scratch replaces the caller's
  const size_t need = sd_verify_workspace_size(args->B, args->K);
  if (need == 0) return SD_ERR_INVALID_ARG;  // B or K out of range
  if (need > kStaticScratchBytes) {
    fprintf(stderr,
            "sd_verify_noalloc: a batch of B=%d, K=%d needs %zu bytes of scratch; the static "
            "scratch holds %zu (at most 1024 + B (2K + 2) = %zu records of 96 bytes)\n",
            args->B, args->K, need, kStaticScratchBytes, kStaticScratchBytes / kRecBytes);
    return SD_ERR_UNSUPPORTED;
  }
  void *scratch = nullptr;
  const sd_status_t st = static_scratch(&scratch);
  if (st != SD_OK) return st;
  sd_verify_args a = *args;
  a.workspace = scratch;
  a.workspace_bytes = kStaticScratchBytes;
  return sd_verify(&a, stream);
}
