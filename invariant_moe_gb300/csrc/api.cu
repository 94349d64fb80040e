// api.cu -- the extern "C" entry points of libbimoe.so: argument checks,
// workspace layout, TMA descriptor encoding, and the device error word.
// All arithmetic happens in the kernels of router.cu, topk.cu, moe_route.cu
// and moe_gemm.cu.
#include <cstdarg>
#include <cstdio>
#include <atomic>
#include <mutex>

#include "bimoe_internal.cuh"

namespace bimoe {

bi_status launch_router(const float *, const float *, const float *, float *, int64_t, int64_t,
                        int64_t, int, cudaStream_t);
bi_status launch_router_bf16(const void *, const float *, const float *, float *, int64_t, int64_t,
                             int64_t, int, cudaStream_t, unsigned *zero_words, int n_zero);
bi_status launch_topk_window(const float *, int64_t, const int64_t *, const int64_t *, int64_t,
                             int64_t, int32_t, int32_t *, cudaStream_t);
bi_status launch_router_negctl(const float *, const float *, const float *, float *, int64_t,
                               int64_t, int64_t, cudaStream_t);
bi_status launch_cast_bf16_f32(const void *, float *, int64_t, cudaStream_t);
bi_status launch_topk(const float *, int32_t *, float *, float *, int64_t, int64_t, int32_t,
                      cudaStream_t);
size_t permute_scratch_bytes(int64_t M, int64_t E);
bi_status launch_permute(const int32_t *, int32_t *, int32_t *, int64_t, int64_t, int32_t, void *,
                         cudaStream_t, uint32_t *slot_mask);
bi_status launch_gather(const void *, const int32_t *, const int32_t *, int64_t, int64_t, int64_t,
                        int32_t, void *, cudaStream_t);
bi_status launch_combine(const float *, void *, int64_t, int64_t, int32_t, bool, cudaStream_t,
                         const uint32_t *slot_mask);
bi_status launch_gate_up(const void *, const int32_t *, const int32_t *, const float *,
                         const void *, void *, int64_t, int64_t, int64_t, int32_t, int64_t,
                         cudaStream_t);
int set_gemm_variant(int v);
bi_status launch_gate_up_tokens(const void *, int64_t, const int32_t *, const int32_t *, const float *,
                                const void *, void *, int64_t, int64_t, int32_t, int64_t, cudaStream_t);
bool decode_path_ok(int64_t M, int64_t E, int32_t top_k);
size_t decode_counter_count(int64_t M, int64_t H);
bi_status launch_moe_decode(const void *, const int32_t *, const float *, const void *, const void *, void *,
                            float *, int *, void *, int64_t, int64_t, int64_t, int32_t, int64_t, cudaStream_t,
                            const float *scores, int32_t *ids_out, float *wts_out);
int set_decode_fused(int mode);
bool decode_fused_ok(int64_t M, int64_t H, int64_t E, int32_t top_k, int64_t I);
int64_t decode_fused_ready_count(int64_t M, int64_t E, int32_t top_k, int64_t I);
bi_status launch_moe_decode_fused(const void *, const void *, const void *, void *, float *, int *, unsigned *,
                                  void *, int64_t, int64_t, int64_t, int32_t, int64_t, cudaStream_t,
                                  const float *scores, int32_t *ids_out, float *wts_out);
// How bi_moe_forward feeds the gate/up GEMM its token rows: 0 automatic (the
// copy), 1 the gather kernel's contiguous copy, 2 gathered by the GEMM itself
// (tile::gather4).  Measured on GB300 at M=4096 the GEMM gathering its own
// rows is 3x slower (DSv4-shaped gate/up 4.31 ms against 1.45 ms; Qwen-shaped
// 0.339 against 0.220 ms): the TMA issues the 128-byte row gathers at about
// 20 cycles per row per SM, well below what the MMAs consume; at decode sizes
// the two are within noise.
static std::atomic<int> g_gate_up_feed{0};
static bool feed_in_gemm() { return g_gate_up_feed.load() == 2; }
bi_status launch_down(const void *, const int32_t *, const int32_t *, const void *, float *,
                      int64_t, int64_t, int64_t, int32_t, int64_t, cudaStream_t);
bi_status launch_fp32_fma_probe(float *, int64_t, int32_t, cudaStream_t);
bool router_topk_fused_supported(int64_t M, int64_t K, int64_t N, int32_t top_k);
template <typename XT>
bi_status launch_router_topk_fused(const XT *, const float *, const float *, float *, float *, int32_t *,
                                   float *, int64_t, int64_t, int64_t, int32_t, cudaStream_t);
// Batches up to this many rows take the one-kernel router + top-k (when its
// cluster can be scheduled); larger ones the router grid and the selection
// grid.  Both give the same bits.  0: the one-kernel path runs only when
// forced (schedule 10): measured on GB300 it is slower than the chained grids
// (DSv4 router shape, M=1: 10.9 us against 8.6 us; the 16 SMs of one
// cluster each stream 256 KB of the weight, and the two grids spread it over
// all SMs).
constexpr int64_t kFusedRouterTopkMaxM = 0;
bi_status launch_gather_routing(const int32_t *, const float *, const int32_t *, const int32_t *, int64_t,
                                int64_t, int64_t, int32_t *, float *, cudaStream_t);
bi_status launch_scatter_contrib(const float *, const int32_t *, const int32_t *, int64_t, int64_t, int64_t,
                                 float *, cudaStream_t);
bi_status launch_wait_timeout_probe(int, cudaStream_t);

// ------------------------------------------------------------ error state --
static thread_local char g_msg[512] = "";

void set_error(const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof g_msg, fmt, ap);
  va_end(ap);
}

// One word per device: kernels record the first BI_DEVERR_* they hit.
__device__ int g_device_error;

constexpr int kMaxDevices = 64;
static std::mutex g_mu;
static int *g_err_ptr[kMaxDevices] = {};
static ContextSetup g_err_ctx;
static int g_sms[kMaxDevices] = {};

static int current_device() {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess) return 0;
  return d;
}

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);

unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  if (!get_current || !get_id) return 0;
  CUcontext c = nullptr;
  if (get_current(&c) != CUDA_SUCCESS || c == nullptr) return 0;
  unsigned long long id = 0;
  if (get_id(c, &id) != CUDA_SUCCESS) return 0;
  return id + 1;  // 0 stays "no context"
}

int *device_error_word() {
  const int d = current_device();
  if (d >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  // the word's address belongs to the context the module is loaded in
  if (!g_err_ptr[d] || g_err_ctx.pending(d)) {
    void *p = nullptr;
    g_err_ptr[d] = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) == cudaSuccess) {
      g_err_ptr[d] = static_cast<int *>(p);
      g_err_ctx.done(d);
    }
  }
  return g_err_ptr[d];
}

int num_sms() {
  const int d = current_device();
  if (d >= kMaxDevices) return 148;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_sms[d]) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, d) != cudaSuccess || v <= 0) v = 148;
    g_sms[d] = v;
  }
  return g_sms[d];
}

// ------------------------------------------------------------ TMA encode --
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

bool make_tma_2d_f32(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols,
                     uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) {
    set_error("cuTensorMapEncodeTiled is not available from the driver");
    return false;
  }
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 4};
  const cuuint32_t box[2] = {32, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void *>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error("cuTensorMapEncodeTiled failed (%d) for fp32 [%llu x %llu]", (int)r,
              (unsigned long long)rows, (unsigned long long)cols);
    return false;
  }
  return true;
}

bool make_tma_2d_bf16(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols,
                      uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) {
    set_error("cuTensorMapEncodeTiled is not available from the driver");
    return false;
  }
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error("cuTensorMapEncodeTiled failed (%d) for [%llu x %llu]", (int)r,
              (unsigned long long)rows, (unsigned long long)cols);
    return false;
  }
  return true;
}

bool make_tma_inter_bf16(CUtensorMap *map, const void *base, uint64_t rows, uint64_t I, uint64_t K) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) {
    set_error("cuTensorMapEncodeTiled is not available from the driver");
    return false;
  }
  if (rows % 16 != 0 || I % 16 != 0) {
    set_error("interleaved weight map needs rows and I multiples of 16");
    return false;
  }
  const cuuint64_t dims[4] = {K, 16, 2, rows / 16};
  const cuuint64_t strides[3] = {K * 2, I * K * 2, 16 * K * 2};
  const cuuint32_t box[4] = {64, 16, 2, 4};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides, box,
                        estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error("cuTensorMapEncodeTiled failed (%d) for the interleaved map [%llu x %llu], I=%llu", (int)r,
              (unsigned long long)rows, (unsigned long long)K, (unsigned long long)I);
    return false;
  }
  return true;
}

// ------------------------------------------------------- MoE workspace --
static size_t align256(size_t v) { return (v + 255) / 256 * 256; }

struct MoeWorkspace {
  size_t offsets, perm, slot_mask, scratch, xperm, act, contrib, counters, gridbar, total;
};

static MoeWorkspace moe_layout(int64_t M, int64_t H, int64_t E, int32_t top_k, int64_t I) {
  MoeWorkspace w{};
  const size_t P = static_cast<size_t>(M) * top_k;
  size_t off = 0;
  w.offsets = off; off += align256((E + 1) * sizeof(int32_t));
  w.perm = off;    off += align256(P * sizeof(int32_t));
  w.slot_mask = off; off += align256(static_cast<size_t>(M) * sizeof(uint32_t));
  w.scratch = off; off += align256(permute_scratch_bytes(M, E));
  w.xperm = off;   off += align256(P * H * 2);
  w.act = off;     off += align256(P * I * 2);
  w.contrib = off; off += align256(P * H * sizeof(float));
  w.counters = off; off += align256(decode_counter_count(M, H) * sizeof(int));
  w.gridbar = off; off += 4096;  // the one-launch decode layer's ready counts (at most 1024)
  w.total = off;
  return w;
}

static bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

static bi_status check_moe_dims(int64_t M, int64_t H, int64_t E, int32_t top_k, int64_t I) {
  if (M < 0 || H <= 0 || E <= 0 || I <= 0) {
    set_error("negative or zero size (M=%lld H=%lld E=%lld I=%lld)", (long long)M, (long long)H,
              (long long)E, (long long)I);
    return BI_ERR_INVALID_ARG;
  }
  if (top_k < 1 || top_k > 16 || top_k > E) {
    set_error("top_k=%d outside [1, min(16, E)]", top_k);
    return BI_ERR_INVALID_ARG;
  }
  if (E > 1024 || H % 128 != 0 || I % 128 != 0) {
    set_error("unsupported MoE shape (needs H%%128==0, I%%128==0, E<=1024): H=%lld I=%lld E=%lld",
              (long long)H, (long long)I, (long long)E);
    return BI_ERR_UNSUPPORTED;
  }
  if (M * top_k >= (int64_t(1) << 31) || M * top_k * H >= (int64_t(1) << 40) ||
      E * 2 * I >= (int64_t(1) << 31) || E * H >= (int64_t(1) << 31)) {
    set_error("MoE sizes exceed the 32-bit index range");
    return BI_ERR_UNSUPPORTED;
  }
  return BI_OK;
}

}  // namespace bimoe

using namespace bimoe;

#define BI_REQUIRE(cond, code, ...) \
  do {                              \
    if (!(cond)) {                  \
      set_error(__VA_ARGS__);       \
      return code;                  \
    }                               \
  } while (0)

extern "C" {

BI_API const char *bi_status_str(bi_status s) {
  switch (s) {
    case BI_OK: return "BI_OK";
    case BI_ERR_INVALID_ARG: return "BI_ERR_INVALID_ARG";
    case BI_ERR_UNSUPPORTED: return "BI_ERR_UNSUPPORTED";
    case BI_ERR_WORKSPACE: return "BI_ERR_WORKSPACE";
    case BI_ERR_CUDA: return "BI_ERR_CUDA";
    case BI_ERR_DEVICE: return "BI_ERR_DEVICE";
  }
  return "BI_ERR_UNKNOWN";
}

BI_API const char *bi_last_error_message(void) { return g_msg; }

BI_API const char *bi_version(void) { return "bimoe 0.1 sm_103a"; }

BI_API bi_status bi_device_error(int32_t *code) {
  BI_REQUIRE(code, BI_ERR_INVALID_ARG, "code is NULL");
  int v = 0, zero = 0;
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpyFromSymbol(&v, g_device_error, sizeof v);
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof zero);
  if (e != cudaSuccess) {
    set_error("reading the device error word: %s", cudaGetErrorString(e));
    return BI_ERR_CUDA;
  }
  *code = v;
  return BI_OK;
}

BI_API bi_status bi_cast_bf16_to_f32(const bi_bf16 *x, float *y, int64_t n, bi_stream_t stream) {
  BI_REQUIRE(n >= 0, BI_ERR_INVALID_ARG, "n < 0");
  if (n == 0) return BI_OK;
  BI_REQUIRE(x && y, BI_ERR_INVALID_ARG, "null pointer");
  return launch_cast_bf16_f32(x, y, n, reinterpret_cast<cudaStream_t>(stream));
}

static bi_status router_checks(const void *x, const float *w, float *y, int64_t M, int64_t K,
                               int64_t N) {
  BI_REQUIRE(M >= 0 && K > 0 && N > 0, BI_ERR_INVALID_ARG, "bad sizes M=%lld K=%lld N=%lld",
             (long long)M, (long long)K, (long long)N);
  BI_REQUIRE(M == 0 || (x && w && y), BI_ERR_INVALID_ARG, "null pointer");
  BI_REQUIRE(K % 128 == 0 && K <= 32768 && N <= 4096, BI_ERR_UNSUPPORTED,
             "router recipe needs K %% 128 == 0, K <= 32768, N <= 4096 (K=%lld N=%lld)",
             (long long)K, (long long)N);
  BI_REQUIRE(M * K < (int64_t(1) << 40) && M * N < (int64_t(1) << 31), BI_ERR_UNSUPPORTED,
             "router sizes exceed the index range");
  BI_REQUIRE(M == 0 || (aligned(x, 16) && aligned(w, 16)), BI_ERR_INVALID_ARG,
             "x and w must be 16-byte aligned");
  return BI_OK;
}

BI_API bi_status bi_router_gemm_schedule(const float *x, const float *w, const float *bias,
                                         float *y, int64_t M, int64_t K, int64_t N,
                                         int32_t schedule, bi_stream_t stream) {
  bi_status st = router_checks(x, w, y, M, K, N);
  if (st != BI_OK) return st;
  BI_REQUIRE(schedule >= 0 && schedule <= 9, BI_ERR_INVALID_ARG, "schedule %d", schedule);
  if (M == 0) return BI_OK;
  return launch_router(x, w, bias, y, M, K, N, schedule, reinterpret_cast<cudaStream_t>(stream));
}

BI_API bi_status bi_router_gemm(const float *x, const float *w, const float *bias, float *y,
                                int64_t M, int64_t K, int64_t N, bi_stream_t stream) {
  return bi_router_gemm_schedule(x, w, bias, y, M, K, N, 0, stream);
}

BI_API bi_status bi_router_gemm_bf16_schedule(const bi_bf16 *x, const float *w, const float *bias,
                                              float *y, int64_t M, int64_t K, int64_t N,
                                              int32_t schedule, bi_stream_t stream) {
  bi_status st = router_checks(x, w, y, M, K, N);
  if (st != BI_OK) return st;
  BI_REQUIRE(schedule >= 0 && schedule <= 9, BI_ERR_INVALID_ARG, "schedule %d", schedule);
  if (M == 0) return BI_OK;
  return launch_router_bf16(x, w, bias, y, M, K, N, schedule, reinterpret_cast<cudaStream_t>(stream), nullptr, 0);
}

BI_API bi_status bi_router_gemm_bf16(const bi_bf16 *x, const float *w, const float *bias, float *y,
                                     int64_t M, int64_t K, int64_t N, bi_stream_t stream) {
  return bi_router_gemm_bf16_schedule(x, w, bias, y, M, K, N, 0, stream);
}

BI_API bi_status bi_router_gemm_splitk_negctl(const float *x, const float *w, const float *bias,
                                              float *y, int64_t M, int64_t K, int64_t N,
                                              bi_stream_t stream) {
  bi_status st = router_checks(x, w, y, M, K, N);
  if (st != BI_OK) return st;
  if (M == 0) return BI_OK;
  return launch_router_negctl(x, w, bias, y, M, K, N, reinterpret_cast<cudaStream_t>(stream));
}

BI_API bi_status bi_topk(const float *scores, float *probs, int32_t *ids, float *wts, int64_t M,
                         int64_t E, int32_t top_k, bi_stream_t stream) {
  BI_REQUIRE(M >= 0, BI_ERR_INVALID_ARG, "M < 0");
  BI_REQUIRE(E >= 1 && E <= 512, BI_ERR_UNSUPPORTED, "E=%lld outside [1, 512]", (long long)E);
  BI_REQUIRE(top_k >= 1 && top_k <= 16 && top_k <= E, BI_ERR_INVALID_ARG,
             "top_k=%d outside [1, min(16, E)]", top_k);
  BI_REQUIRE(M * E < (int64_t(1) << 31), BI_ERR_UNSUPPORTED, "M*E exceeds the index range");
  if (M == 0) return BI_OK;
  BI_REQUIRE(scores && ids && wts, BI_ERR_INVALID_ARG, "null pointer");
  return launch_topk(scores, ids, wts, probs, M, E, top_k, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"

static bi_status launch_router_any(const float *x, const float *w, const float *b, float *y, int64_t M,
                                   int64_t K, int64_t N, int schedule, cudaStream_t s) {
  return launch_router(x, w, b, y, M, K, N, schedule, s);
}
static bi_status launch_router_any(const __nv_bfloat16 *x, const float *w, const float *b, float *y,
                                   int64_t M, int64_t K, int64_t N, int schedule, cudaStream_t s) {
  return launch_router_bf16(x, w, b, y, M, K, N, schedule, s, nullptr, 0);
}

// Router + selection: schedule 0 picks by M (the one-kernel path for small
// batches, else the router grid chained with the selection grid), 10 forces
// the one-kernel path, 1..9 force a router schedule followed by the selection
// grid.
template <typename XT>
static bi_status router_topk_impl(const XT *x, const float *w, const float *bias, float *y, float *probs,
                                  int32_t *ids, float *wts, int64_t M, int64_t K, int64_t N, int32_t top_k,
                                  int32_t schedule, bi_stream_t stream) {
  bi_status st = router_checks(x, w, y, M, K, N);
  if (st != BI_OK) return st;
  BI_REQUIRE(schedule >= 0 && schedule <= 10, BI_ERR_INVALID_ARG, "schedule %d", schedule);
  BI_REQUIRE(N <= 512, BI_ERR_UNSUPPORTED, "selection needs N <= 512 (N=%lld)", (long long)N);
  BI_REQUIRE(top_k >= 1 && top_k <= 16 && top_k <= N, BI_ERR_INVALID_ARG,
             "top_k=%d outside [1, min(16, N)]", top_k);
  if (M == 0) return BI_OK;
  BI_REQUIRE(ids && wts, BI_ERR_INVALID_ARG, "null pointer");
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (schedule == 10) return launch_router_topk_fused(x, w, bias, y, probs, ids, wts, M, K, N, top_k, s);
  if (schedule == 0 && M <= kFusedRouterTopkMaxM && router_topk_fused_supported(M, K, N, top_k)) {
    st = launch_router_topk_fused(x, w, bias, y, probs, ids, wts, M, K, N, top_k, s);
    if (st != BI_ERR_UNSUPPORTED) return st;  // else its cluster cannot be scheduled: two grids
  }
  if ((st = launch_router_any(x, w, bias, y, M, K, N, schedule, s)) != BI_OK) return st;
  return launch_topk(y, ids, wts, probs, M, N, top_k, s);
}

extern "C" {

BI_API bi_status bi_router_topk_schedule(const float *x, const float *w, const float *bias,
                                         float *y, float *probs, int32_t *ids, float *wts,
                                         int64_t M, int64_t K, int64_t N, int32_t top_k,
                                         int32_t schedule, bi_stream_t stream) {
  return router_topk_impl(x, w, bias, y, probs, ids, wts, M, K, N, top_k, schedule, stream);
}

BI_API bi_status bi_router_topk_bf16_schedule(const bi_bf16 *x, const float *w, const float *bias,
                                              float *y, float *probs, int32_t *ids, float *wts,
                                              int64_t M, int64_t K, int64_t N, int32_t top_k,
                                              int32_t schedule, bi_stream_t stream) {
  return router_topk_impl(reinterpret_cast<const __nv_bfloat16 *>(x), w, bias, y, probs, ids, wts, M, K, N,
                          top_k, schedule, stream);
}

BI_API bi_status bi_router_topk(const float *x, const float *w, const float *bias, float *y,
                                float *probs, int32_t *ids, float *wts, int64_t M, int64_t K,
                                int64_t N, int32_t top_k, bi_stream_t stream) {
  return bi_router_topk_schedule(x, w, bias, y, probs, ids, wts, M, K, N, top_k, 0, stream);
}

BI_API bi_status bi_router_topk_bf16(const bi_bf16 *x, const float *w, const float *bias, float *y,
                                     float *probs, int32_t *ids, float *wts, int64_t M, int64_t K,
                                     int64_t N, int32_t top_k, bi_stream_t stream) {
  return bi_router_topk_bf16_schedule(x, w, bias, y, probs, ids, wts, M, K, N, top_k, 0, stream);
}

BI_API bi_status bi_topk_window(const float *scores, int64_t ld, const int64_t *row_start,
                                const int64_t *row_end, int64_t n_rows, int64_t num_cols,
                                int32_t k, int32_t *out, bi_stream_t stream) {
  BI_REQUIRE(n_rows >= 0 && num_cols >= 0 && ld >= num_cols, BI_ERR_INVALID_ARG,
             "bad sizes n_rows=%lld num_cols=%lld ld=%lld", (long long)n_rows,
             (long long)num_cols, (long long)ld);
  BI_REQUIRE(num_cols <= 8192, BI_ERR_UNSUPPORTED, "num_cols=%lld > 8192", (long long)num_cols);
  BI_REQUIRE(k >= 1 && k <= 8192, BI_ERR_INVALID_ARG, "k=%d outside [1, 8192]", k);
  BI_REQUIRE(n_rows < (int64_t(1) << 31) && n_rows * ld < (int64_t(1) << 62), BI_ERR_UNSUPPORTED,
             "sizes exceed the index range");
  if (n_rows == 0) return BI_OK;
  BI_REQUIRE(out && (scores || num_cols == 0), BI_ERR_INVALID_ARG, "null pointer");
  return launch_topk_window(scores, ld, row_start, row_end, n_rows, num_cols, k, out,
                            reinterpret_cast<cudaStream_t>(stream));
}

BI_API bi_status bi_fp32_fma_probe(float *out, int64_t blocks, int32_t iters, bi_stream_t stream) {
  BI_REQUIRE(out && blocks > 0 && blocks < (int64_t(1) << 31) && iters > 0, BI_ERR_INVALID_ARG,
             "bad probe arguments");
  return launch_fp32_fma_probe(out, blocks, iters, reinterpret_cast<cudaStream_t>(stream));
}

BI_API bi_status bi_wait_timeout_probe(int32_t which, bi_stream_t stream) {
  BI_REQUIRE(which == 0 || which == 1, BI_ERR_INVALID_ARG, "wait probe %d not in {0, 1}", which);
  return launch_wait_timeout_probe(which, reinterpret_cast<cudaStream_t>(stream));
}

BI_API size_t bi_moe_workspace_bytes(int64_t M, int64_t H, int64_t E, int32_t top_k, int64_t I) {
  if (check_moe_dims(M, H, E, top_k, I) != BI_OK) return 0;
  return moe_layout(M, H, E, top_k, I).total;
}

BI_API size_t bi_moe_permute_workspace_bytes(int64_t M, int64_t E) {
  if (M < 0 || E <= 0) return 0;
  return align256(permute_scratch_bytes(M, E));
}

BI_API bi_status bi_moe_permute(const int32_t *ids, int32_t *offsets, int32_t *perm, int64_t M,
                                int64_t E, int32_t top_k, void *workspace, size_t workspace_bytes,
                                bi_stream_t stream) {
  BI_REQUIRE(M >= 0 && E >= 1 && E <= 1024, BI_ERR_INVALID_ARG, "bad sizes M=%lld E=%lld",
             (long long)M, (long long)E);
  BI_REQUIRE(top_k >= 1 && top_k <= 16 && top_k <= E, BI_ERR_INVALID_ARG, "top_k=%d", top_k);
  BI_REQUIRE(M * top_k < (int64_t(1) << 31), BI_ERR_UNSUPPORTED, "M*top_k exceeds int32");
  BI_REQUIRE(offsets, BI_ERR_INVALID_ARG, "offsets is NULL");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (M == 0) {
    if (cudaMemsetAsync(offsets, 0, (E + 1) * sizeof(int32_t), s) != cudaSuccess) {
      set_error("cudaMemsetAsync failed");
      return BI_ERR_CUDA;
    }
    return BI_OK;
  }
  BI_REQUIRE(ids && perm && workspace, BI_ERR_INVALID_ARG, "null pointer");
  BI_REQUIRE(workspace_bytes >= bi_moe_permute_workspace_bytes(M, E), BI_ERR_WORKSPACE,
             "workspace %zu < %zu bytes", workspace_bytes, bi_moe_permute_workspace_bytes(M, E));
  return launch_permute(ids, offsets, perm, M, E, top_k, workspace, s, nullptr);
}

BI_API bi_status bi_moe_gather(const bi_bf16 *x, const int32_t *offsets, const int32_t *perm,
                               bi_bf16 *x_perm, int64_t M, int64_t H, int64_t E, int32_t top_k,
                               bi_stream_t stream) {
  BI_REQUIRE(M >= 0 && H > 0 && H % 8 == 0 && E >= 1, BI_ERR_INVALID_ARG, "bad sizes (H %% 8 == 0)");
  BI_REQUIRE(top_k >= 1 && top_k <= 16, BI_ERR_INVALID_ARG, "top_k=%d", top_k);
  BI_REQUIRE(M * top_k < (int64_t(1) << 31), BI_ERR_UNSUPPORTED, "M*top_k exceeds int32");
  if (M == 0) return BI_OK;
  BI_REQUIRE(x && offsets && perm && x_perm, BI_ERR_INVALID_ARG, "null pointer");
  BI_REQUIRE(aligned(x, 16) && aligned(x_perm, 16), BI_ERR_INVALID_ARG,
             "x and x_perm must be 16-byte aligned");
  return launch_gather(x, perm, offsets, M * top_k, H, E, top_k, x_perm,
                       reinterpret_cast<cudaStream_t>(stream));
}

BI_API bi_status bi_moe_gate_up(const bi_bf16 *x_perm, const int32_t *offsets, const int32_t *perm,
                                const float *wts, const bi_bf16 *w13, bi_bf16 *act, int64_t M,
                                int64_t H, int64_t E, int32_t top_k, int64_t I,
                                bi_stream_t stream) {
  bi_status st = check_moe_dims(M, H, E, top_k, I);
  if (st != BI_OK) return st;
  if (M == 0) return BI_OK;
  BI_REQUIRE(x_perm && offsets && perm && wts && w13 && act, BI_ERR_INVALID_ARG, "null pointer");
  BI_REQUIRE(aligned(x_perm, 16) && aligned(w13, 16), BI_ERR_INVALID_ARG,
             "x_perm/w13 must be 16-byte aligned");
  return launch_gate_up(x_perm, offsets, perm, wts, w13, act, M * top_k, H, E, top_k, I,
                        reinterpret_cast<cudaStream_t>(stream));
}

BI_API bi_status bi_moe_gate_up_tokens(const bi_bf16 *x, const int32_t *offsets, const int32_t *perm,
                                       const float *wts, const bi_bf16 *w13, bi_bf16 *act, int64_t M,
                                       int64_t H, int64_t E, int32_t top_k, int64_t I, bi_stream_t stream) {
  bi_status st = check_moe_dims(M, H, E, top_k, I);
  if (st != BI_OK) return st;
  if (M == 0) return BI_OK;
  BI_REQUIRE(x && offsets && perm && wts && w13 && act, BI_ERR_INVALID_ARG, "null pointer");
  BI_REQUIRE(aligned(x, 16) && aligned(w13, 16), BI_ERR_INVALID_ARG, "x/w13 must be 16-byte aligned");
  return launch_gate_up_tokens(x, M, offsets, perm, wts, w13, act, H, E, top_k, I,
                               reinterpret_cast<cudaStream_t>(stream));
}

BI_API bi_status bi_moe_down(const bi_bf16 *act, const int32_t *offsets, const int32_t *perm,
                             const bi_bf16 *w2, float *contrib, int64_t M, int64_t H, int64_t E,
                             int32_t top_k, int64_t I, bi_stream_t stream) {
  bi_status st = check_moe_dims(M, H, E, top_k, I);
  if (st != BI_OK) return st;
  if (M == 0) return BI_OK;
  BI_REQUIRE(act && offsets && perm && w2 && contrib, BI_ERR_INVALID_ARG, "null pointer");
  BI_REQUIRE(aligned(act, 16) && aligned(w2, 16), BI_ERR_INVALID_ARG,
             "act/w2 must be 16-byte aligned");
  return launch_down(act, offsets, perm, w2, contrib, M * top_k, H, E, top_k, I,
                     reinterpret_cast<cudaStream_t>(stream));
}

BI_API bi_status bi_moe_combine(const float *contrib, bi_bf16 *out, int64_t M, int64_t H,
                                int32_t top_k, bi_stream_t stream) {
  BI_REQUIRE(M >= 0 && H > 0 && H % 4 == 0, BI_ERR_INVALID_ARG, "bad sizes (H %% 4 == 0 needed)");
  BI_REQUIRE(top_k >= 1 && top_k <= 16, BI_ERR_INVALID_ARG, "top_k=%d", top_k);
  if (M == 0) return BI_OK;
  BI_REQUIRE(contrib && out, BI_ERR_INVALID_ARG, "null pointer");
  BI_REQUIRE(aligned(contrib, 16) && aligned(out, 8), BI_ERR_INVALID_ARG,
             "contrib must be 16-byte and out 8-byte aligned");
  return launch_combine(contrib, out, M, H, top_k, false, reinterpret_cast<cudaStream_t>(stream), nullptr);
}

BI_API bi_status bi_moe_combine_consume(float *contrib, bi_bf16 *out, int64_t M, int64_t H,
                                        int32_t top_k, bi_stream_t stream) {
  BI_REQUIRE(M >= 0 && H > 0 && H % 4 == 0, BI_ERR_INVALID_ARG, "bad sizes (H %% 4 == 0 needed)");
  BI_REQUIRE(top_k >= 1 && top_k <= 16, BI_ERR_INVALID_ARG, "top_k=%d", top_k);
  if (M == 0) return BI_OK;
  BI_REQUIRE(contrib && out, BI_ERR_INVALID_ARG, "null pointer");
  BI_REQUIRE(aligned(contrib, 16) && aligned(out, 8), BI_ERR_INVALID_ARG,
             "contrib must be 16-byte and out 8-byte aligned");
  return launch_combine(contrib, out, M, H, top_k, true, reinterpret_cast<cudaStream_t>(stream), nullptr);
}

BI_API bi_status bi_moe_gather_routing(const int32_t *ids, const float *wts, const int32_t *offsets,
                                       const int32_t *perm, int32_t *lid, float *pw, int64_t M, int64_t E,
                                       int32_t top_k, int64_t experts_per_rank, bi_stream_t stream) {
  BI_REQUIRE(M >= 0 && E >= 1 && E <= 1024, BI_ERR_INVALID_ARG, "bad sizes M=%lld E=%lld", (long long)M,
             (long long)E);
  BI_REQUIRE(top_k >= 1 && top_k <= 16 && top_k <= E, BI_ERR_INVALID_ARG, "top_k=%d", top_k);
  BI_REQUIRE(experts_per_rank >= 1 && experts_per_rank <= E && E % experts_per_rank == 0, BI_ERR_INVALID_ARG,
             "experts_per_rank=%lld must divide E=%lld", (long long)experts_per_rank, (long long)E);
  BI_REQUIRE(M * top_k < (int64_t(1) << 31), BI_ERR_UNSUPPORTED, "M*top_k exceeds int32");
  if (M == 0) return BI_OK;
  BI_REQUIRE(ids && wts && offsets && perm && lid && pw, BI_ERR_INVALID_ARG, "null pointer");
  return launch_gather_routing(ids, wts, offsets, perm, M * top_k, E, experts_per_rank, lid, pw,
                               reinterpret_cast<cudaStream_t>(stream));
}

BI_API bi_status bi_moe_scatter_contrib(const float *rows, const int32_t *offsets, const int32_t *perm,
                                        float *contrib, int64_t M, int64_t H, int64_t E, int32_t top_k,
                                        bi_stream_t stream) {
  BI_REQUIRE(M >= 0 && H > 0 && H % 4 == 0 && E >= 1 && E <= 1024, BI_ERR_INVALID_ARG,
             "bad sizes (H %% 4 == 0 needed)");
  BI_REQUIRE(top_k >= 1 && top_k <= 16, BI_ERR_INVALID_ARG, "top_k=%d", top_k);
  BI_REQUIRE(M * top_k < (int64_t(1) << 31), BI_ERR_UNSUPPORTED, "M*top_k exceeds int32");
  if (M == 0) return BI_OK;
  BI_REQUIRE(rows && offsets && perm && contrib, BI_ERR_INVALID_ARG, "null pointer");
  BI_REQUIRE(aligned(rows, 16) && aligned(contrib, 16), BI_ERR_INVALID_ARG,
             "rows and contrib must be 16-byte aligned");
  return launch_scatter_contrib(rows, offsets, perm, M * top_k, H, E, contrib,
                                reinterpret_cast<cudaStream_t>(stream));
}

BI_API bi_status bi_moe_forward(const bi_bf16 *x, const int32_t *ids, const float *wts,
                                const bi_bf16 *w13, const bi_bf16 *w2, bi_bf16 *out, int64_t M,
                                int64_t H, int64_t E, int32_t top_k, int64_t I, void *workspace,
                                size_t workspace_bytes, bi_stream_t stream) {
  bi_status st = check_moe_dims(M, H, E, top_k, I);
  if (st != BI_OK) return st;
  if (M == 0) return BI_OK;
  BI_REQUIRE(x && ids && wts && w13 && w2 && out && workspace, BI_ERR_INVALID_ARG, "null pointer");
  BI_REQUIRE(aligned(x, 16) && aligned(w13, 16) && aligned(w2, 16) && aligned(out, 8) &&
                 aligned(workspace, 256),
             BI_ERR_INVALID_ARG, "misaligned pointer (x/w13/w2 16 B, out 8 B, workspace 256 B)");
  const MoeWorkspace L = moe_layout(M, H, E, top_k, I);
  BI_REQUIRE(workspace_bytes >= L.total, BI_ERR_WORKSPACE, "workspace %zu < %zu bytes",
             workspace_bytes, L.total);
  char *ws = static_cast<char *>(workspace);
  int32_t *offsets = reinterpret_cast<int32_t *>(ws + L.offsets);
  int32_t *perm = reinterpret_cast<int32_t *>(ws + L.perm);
  void *xperm = ws + L.xperm;
  void *act = ws + L.act;
  float *contrib = reinterpret_cast<float *>(ws + L.contrib);
  uint32_t *slot_mask = reinterpret_cast<uint32_t *>(ws + L.slot_mask);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int64_t P = M * top_k;
  if (g_gate_up_feed.load() == 0 && decode_path_ok(M, E, top_k)) {
    // decode-sized batch: two launches, the routing derived inside the GEMMs
    // and the combine fused into the down GEMM
    return launch_moe_decode(x, ids, wts, w13, w2, act, contrib, reinterpret_cast<int *>(ws + L.counters), out,
                             M, H, E, top_k, I, s, nullptr, nullptr, nullptr);
  }
  if ((st = launch_permute(ids, offsets, perm, M, E, top_k, ws + L.scratch, s, slot_mask)) != BI_OK)
    return st;
  if (feed_in_gemm()) {
    // the gate/up GEMM gathers the token rows from x itself
    if ((st = launch_gate_up_tokens(x, M, offsets, perm, wts, w13, act, H, E, top_k, I, s)) != BI_OK)
      return st;
  } else {
    if ((st = launch_gather(x, perm, offsets, P, H, E, top_k, xperm, s)) != BI_OK) return st;
    if ((st = launch_gate_up(xperm, offsets, perm, wts, w13, act, P, H, E, top_k, I, s)) != BI_OK)
      return st;
  }
  if ((st = launch_down(act, offsets, perm, w2, contrib, P, H, E, top_k, I, s)) != BI_OK) return st;
  // a pair skipped for a bad id (recorded in the device error word) adds
  // nothing: the combine sums the slots the permutation marked valid
  return launch_combine(contrib, out, M, H, top_k, true, s, slot_mask);
}

BI_API bi_status bi_moe_layer(const bi_bf16 *x, const float *w_router, const float *bias,
                              const bi_bf16 *w13, const bi_bf16 *w2, bi_bf16 *out, float *scores,
                              int32_t *ids, float *wts, int64_t M, int64_t H, int64_t E, int32_t top_k,
                              int64_t I, void *workspace, size_t workspace_bytes, bi_stream_t stream) {
  bi_status st = check_moe_dims(M, H, E, top_k, I);
  if (st != BI_OK) return st;
  BI_REQUIRE(E <= 512, BI_ERR_UNSUPPORTED, "the layer's selection needs E <= 512 (E=%lld)", (long long)E);
  if ((st = router_checks(x, w_router, scores, M, H, E)) != BI_OK) return st;
  if (M == 0) return BI_OK;
  BI_REQUIRE(x && w_router && w13 && w2 && out && scores && ids && wts && workspace, BI_ERR_INVALID_ARG,
             "null pointer");
  BI_REQUIRE(aligned(x, 16) && aligned(w13, 16) && aligned(w2, 16) && aligned(out, 8) && aligned(workspace, 256),
             BI_ERR_INVALID_ARG, "misaligned pointer (x/w13/w2 16 B, out 8 B, workspace 256 B)");
  const MoeWorkspace L = moe_layout(M, H, E, top_k, I);
  BI_REQUIRE(workspace_bytes >= L.total, BI_ERR_WORKSPACE, "workspace %zu < %zu bytes", workspace_bytes, L.total);
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  char *ws = static_cast<char *>(workspace);
  const bool decode = g_gate_up_feed.load() == 0 && decode_path_ok(M, E, top_k);
  // decode-sized batch with the one-launch expert path: the router zeroes
  // its combine counters and ready counts (one range: the counters, the
  // padding after them, the ready counts)
  const bool fused = decode && decode_fused_ok(M, H, E, top_k, I);
  unsigned *zero_from = fused ? reinterpret_cast<unsigned *>(ws + L.counters) : nullptr;
  const int n_zero = fused ? static_cast<int>((L.gridbar - L.counters) / 4 + decode_fused_ready_count(M, E, top_k, I))
                           : 0;
  if ((st = launch_router_bf16(x, w_router, bias, scores, M, H, E, 0, s, zero_from, n_zero)) != BI_OK) return st;
  if (fused)
    return launch_moe_decode_fused(x, w13, w2, ws + L.act, reinterpret_cast<float *>(ws + L.contrib),
                                   reinterpret_cast<int *>(ws + L.counters), reinterpret_cast<unsigned *>(ws + L.gridbar),
                                   out, M, H, E, top_k, I, s, scores, ids, wts);
  if (decode) {
    // decode-sized batch: the gate/up GEMM selects the experts itself
    return launch_moe_decode(x, nullptr, nullptr, w13, w2, ws + L.act, reinterpret_cast<float *>(ws + L.contrib),
                             reinterpret_cast<int *>(ws + L.counters), out, M, H, E, top_k, I, s, scores, ids, wts);
  }
  if ((st = launch_topk(scores, ids, wts, nullptr, M, E, top_k, s)) != BI_OK) return st;
  return bi_moe_forward(x, ids, wts, w13, w2, out, M, H, E, top_k, I, workspace, workspace_bytes, stream);
}

}  // extern "C"

BI_API bi_status bi_moe_gate_up_feed(int32_t mode, int32_t *previous) {
  BI_REQUIRE(mode >= 0 && mode <= 2, BI_ERR_INVALID_ARG, "feed mode %d not in {0, 1, 2}", mode);
  const int old = g_gate_up_feed.exchange(mode);
  if (previous) *previous = old;
  return BI_OK;
}

BI_API bi_status bi_moe_decode_fused(int32_t mode, int32_t *previous) {
  BI_REQUIRE(mode == 0 || mode == 1, BI_ERR_INVALID_ARG, "decode layer mode %d not in {0, 1}", mode);
  const int old = bimoe::set_decode_fused(mode);
  if (previous) *previous = old;
  return BI_OK;
}

BI_API bi_status bi_moe_gemm_variant(int32_t variant, int32_t *previous) {
  BI_REQUIRE(variant >= 0 && variant <= 4, BI_ERR_INVALID_ARG, "variant %d not in {0, ..., 4}", variant);
  const int old = bimoe::set_gemm_variant(variant);
  if (previous) *previous = old;
  return BI_OK;
}
