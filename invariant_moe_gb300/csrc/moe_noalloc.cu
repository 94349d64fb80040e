// moe_noalloc.cu -- bi_moe_forward for callers that cannot allocate device
// memory.
//
// Some callers cannot call cudaMalloc at the point where they run the MoE
// layer: code inside a custom allocator or a memory-pool callback, runtimes
// that own every byte of device memory and forbid allocations behind their
// back, and launch paths that must not touch the allocator at all.  For them
// this entry point takes its scratch space from a fixed array in the
// library's own device memory instead of a caller-provided workspace.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds kNoAllocScratchBytes of memory for it until the process exits.
// Host code cannot use the array's name as a device address (on the host it is
// only a stand-in symbol), so the device address is looked up with
// cudaGetSymbolAddress, with the device current, on the first call made on
// that device -- and again on the first call after the current context
// changes (a cudaDeviceReset, or a caller in a context other than the
// device's primary one loads the module anew, possibly at another address).
// Make the first call of each context before any stream capture begins.
#include <mutex>

#include "bimoe_internal.cuh"

namespace bimoe {

// 64 MiB: the workspace of decode-sized batches, e.g. up to 605 tokens of a
// Qwen3-30B-A3B-shaped layer (H=2048, E=128, top-8, I=768) or 291 tokens of
// an H=4096, E=256, top-8, I=2048 layer.  Must match BI_NOALLOC_SCRATCH_BYTES
// in bimoe.h.
constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;
static_assert(kNoAllocScratchBytes == BI_NOALLOC_SCRATCH_BYTES, "scratch size out of sync");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

static std::mutex g_noalloc_mu;
static void *g_noalloc_ptr[64] = {};
static ContextSetup g_noalloc_ctx;

// Device address of the scratch array in the current context of the current
// device (looked up once per device and context).  Returns null and sets the
// error message on failure.
static void *noalloc_scratch() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    set_error("bi_moe_forward_noalloc: no usable current device");
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[dev] || g_noalloc_ctx.pending(dev)) {
    g_noalloc_ptr[dev] = nullptr;
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();  // do not leave the error for an unrelated later check
      set_error("bi_moe_forward_noalloc: cudaGetSymbolAddress failed: %s", cudaGetErrorString(e));
      return nullptr;
    }
    g_noalloc_ptr[dev] = p;
    g_noalloc_ctx.done(dev);
  }
  return g_noalloc_ptr[dev];
}

}  // namespace bimoe

extern "C" BI_API bi_status bi_moe_forward_noalloc(const bi_bf16 *x, const int32_t *ids,
                                                   const float *wts, const bi_bf16 *w13,
                                                   const bi_bf16 *w2, bi_bf16 *out, int64_t M,
                                                   int64_t H, int64_t E, int32_t top_k, int64_t I,
                                                   bi_stream_t stream) {
  const size_t need = bi_moe_workspace_bytes(M, H, E, top_k, I);
  if (need == 0) {
    // invalid sizes (bi_moe_workspace_bytes is 0 only for those): the
    // regular checks report them; nothing is launched
    const bi_status st = bi_moe_forward(x, ids, wts, w13, w2, out, M, H, E, top_k, I, nullptr, 0, stream);
    return st == BI_OK ? BI_ERR_INVALID_ARG : st;
  }
  if (M == 0) return BI_OK;  // valid sizes, nothing to do
  if (need > bimoe::kNoAllocScratchBytes) {
    bimoe::set_error(
        "bi_moe_forward_noalloc: these sizes need %zu bytes of scratch but the built-in array "
        "holds %zu bytes (M=%lld H=%lld E=%lld top_k=%d I=%lld); use bi_moe_forward with a "
        "caller-provided workspace",
        need, bimoe::kNoAllocScratchBytes, (long long)M, (long long)H, (long long)E, top_k,
        (long long)I);
    return BI_ERR_WORKSPACE;
  }
  void *scratch = bimoe::noalloc_scratch();
  if (!scratch) return BI_ERR_CUDA;
  return bi_moe_forward(x, ids, wts, w13, w2, out, M, H, E, top_k, I, scratch,
                        bimoe::kNoAllocScratchBytes, stream);
}
