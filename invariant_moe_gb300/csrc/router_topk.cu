// router_topk.cu -- decode-sized router GEMM, sigmoid and top-k selection in
// one kernel.
//
// Source: "[BI][DSv4] Batch-invariant GateLinear router with fp32 persistent
// matmul", sections "Perf" (at decode sizes the router's cost is per-call
// latency, paid in every layer of every decode step) and "A correction to why
// the key excludes M" (the reduction recipe may not depend on M); "[BI][DSv4]
// Pin sparse-MLA decode and prefill scheduling under batch invariance", commit
// log (the deterministic per-row top-k).
//
// For a batch of at most kRtMaxM token rows, one thread-block cluster owns all
// N scores of its rows: CTA c of the cluster computes columns [16c, 16c + 16)
// for every row, parks them in its shared memory, and after a cluster barrier
// one warp per row reads the row's N scores from the cluster's shared memory
// (distributed shared memory) and selects its top_k with the same warp
// selection as bi_topk.  No score makes a round trip through global memory
// before the selection, and there is no second launch.
//
// Per-element arithmetic is the router recipe of router.cu, unchanged: slice
// s = fp32 FMA chain over k = 128s .. 128s+127 in increasing k from +0.0,
// slices added in slice order into a running sum starting at +0.0, bias added
// last.  So y, ids, wts and probs are bit for bit those of bi_router_gemm
// followed by bi_topk (the tests compare them).
//
// Layout of the work.  K runs in stages of 8 slices (1024 k); a stage brings
// the CTA's 16 weight-row pieces (4 KB each, 1-D bulk copies into rows padded
// to 4112 bytes, which makes the lanes' 16-byte loads conflict free) and the
// batch's token rows into a ring as deep as shared memory allows (2-4
// stages); the copies of a stage are issued by one lane each of warp 0.  Warp
// w evaluates slice w of the stage; lane l takes column l % 16 and rows
// l / 16, l / 16 + 2.  After each stage one thread per (row, column) adds the
// stage's 8 slice partials to its running sum in slice order.
#include "router_common.cuh"
#include "topk_warp.cuh"

namespace bimoe {

constexpr int kRtCols = 16;                       // columns per CTA
constexpr int kRtStageSlices = 8;                 // slices per stage (one per warp)
constexpr int kRtStageK = kRtStageSlices * kSlice;  // 1024
constexpr int kRtWPitch = kRtStageK + 4;          // floats per staged weight piece
constexpr int kRtThreads = 32 * kRtStageSlices;   // 256
constexpr int kRtMaxM = 4;                        // rows per call
constexpr int kRtMaxCluster = 16;                 // N <= 256

template <int MR, typename XT>
struct RtCfg {
  static constexpr int kWBytes = kRtCols * kRtWPitch * 4;                 // 65,792
  static constexpr int kXBytes = MR * kRtStageK * static_cast<int>(sizeof(XT));
  static constexpr int kStageBytes = kWBytes + kXBytes;
  static constexpr int kPartBytes = 2 * MR * kRtCols * kRtStageSlices * 4;
  static constexpr int kScoreBytes = MR * kRtCols * 4;
  static constexpr int kFixed = kPartBytes + kScoreBytes + 8 * 4 + 16;
  static constexpr int kFit = (227 * 1024 - kFixed) / kStageBytes;
  static constexpr int kStages = kFit < 4 ? kFit : 4;  // ring depth
  static_assert(kStages >= 2, "ring");
  static constexpr int kSmem = kStages * kStageBytes + kFixed;
  static_assert(kWBytes % 16 == 0 && kXBytes % 16 == 0, "bulk copy alignment");
  static_assert(kSmem <= 227 * 1024, "shared memory");
};

// Load of an fp32 from the shared memory of a CTA of the cluster (address
// from mapa).
__device__ __forceinline__ float ld_dsmem_f32(uint32_t cluster_addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(cluster_addr) : "memory");
  return v;
}

template <int MR, typename XT>
__global__ void __launch_bounds__(kRtThreads, 1)
    router_topk_cluster_kernel(const XT *__restrict__ x, const float *__restrict__ w,
                               const float *__restrict__ bias, float *__restrict__ y,
                               float *__restrict__ probs, int32_t *__restrict__ ids,
                               float *__restrict__ wts, int M, int K, int N, int top_k, int *err) {
  using C = RtCfg<MR, XT>;
  extern __shared__ __align__(16) uint8_t rt_smem[];
  uint8_t *ring = rt_smem;
  constexpr int kRtStages = C::kStages;
  float *part = reinterpret_cast<float *>(rt_smem + kRtStages * C::kStageBytes);  // [2][MR][16][8]
  float *sc = part + 2 * MR * kRtCols * kRtStageSlices;                             // [MR][16]
  uint64_t *full = reinterpret_cast<uint64_t *>(sc + MR * kRtCols);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(full + kRtStages);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cta = static_cast<int>(cluster_ctarank());
  const int ncta = N / kRtCols;
  const int col = lane & 15;         // this lane's column of the CTA's 16
  const int R = K / kRtStageK;        // stages

  if (tid == 0) {
    for (int s = 0; s < kRtStages; ++s) mbar_init(smem_u32(&full[s]), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  griddep_wait();  // x may come from the previous kernel on the stream

  // warp 0 issues a stage's copies, one per lane: lanes 0-15 the 16 weight
  // pieces, lanes 16.. the M token rows
  auto issue = [&](int r) {
    const int b = r % kRtStages;
    uint8_t *st = ring + b * C::kStageBytes;
    const uint32_t bar = smem_u32(&full[b]);
    const uint32_t xbytes = kRtStageK * static_cast<uint32_t>(sizeof(XT));
    if (lane == 0) mbar_arrive_expect_tx(bar, kRtCols * kRtStageK * 4 + static_cast<uint32_t>(M) * xbytes);
    __syncwarp();
    if (lane < kRtCols)
      bulk_g2s(smem_u32(st + lane * kRtWPitch * 4),
               w + static_cast<size_t>(cta * kRtCols + lane) * K + static_cast<size_t>(r) * kRtStageK,
               kRtStageK * 4, bar);
    else if (lane - kRtCols < M)
      bulk_g2s(smem_u32(st + C::kWBytes + (lane - kRtCols) * kRtStageK * sizeof(XT)),
               x + static_cast<size_t>(lane - kRtCols) * K + static_cast<size_t>(r) * kRtStageK, xbytes, bar);
  };
  if (warp == 0)
    for (int r = 0; r < R && r < kRtStages; ++r) issue(r);

  float rs = 0.0f;  // running sum of thread tid < MR*16: row tid / 16, column tid % 16
  int done = 0;     // stages consumed
  for (int r = 0; r < R; ++r) {
    const int b = r % kRtStages;
    const bool got = mbar_wait(smem_u32(&full[b]), static_cast<uint32_t>((r / kRtStages) & 1), abort_flag, err);
    if (__syncthreads_or(got ? 0 : 1)) break;
    const uint8_t *st = ring + b * C::kStageBytes;
    const float *wl = reinterpret_cast<const float *>(st) + col * kRtWPitch + warp * kSlice;
    const XT *xs = reinterpret_cast<const XT *>(st + C::kWBytes) + warp * kSlice;
    float p[(MR + 1) / 2];
#pragma unroll
    for (int i = 0; i < (MR + 1) / 2; ++i) p[i] = 0.0f;
#pragma unroll 8
    for (int k = 0; k < kSlice; k += 4) {
      const float4 wv = *reinterpret_cast<const float4 *>(wl + k);
#pragma unroll
      for (int i = 0; i < (MR + 1) / 2; ++i) {
        const int m = (lane >> 4) + 2 * i;
        if (m < MR) {
          const float4 xv = ld_x4(xs + m * kRtStageK + k);
          p[i] = __fmaf_rn(xv.x, wv.x, p[i]);
          p[i] = __fmaf_rn(xv.y, wv.y, p[i]);
          p[i] = __fmaf_rn(xv.z, wv.z, p[i]);
          p[i] = __fmaf_rn(xv.w, wv.w, p[i]);
        }
      }
    }
    float *pr = part + (r & 1) * MR * kRtCols * kRtStageSlices;
#pragma unroll
    for (int i = 0; i < (MR + 1) / 2; ++i) {
      const int m = (lane >> 4) + 2 * i;
      if (m < MR) pr[(m * kRtCols + col) * kRtStageSlices + warp] = p[i];
    }
    __syncthreads();  // the ring slot is free and the partials are in place
    done = r + 1;
    if (warp == 0 && r + kRtStages < R) issue(r + kRtStages);
    if (tid < MR * kRtCols) {
      const float *q = pr + tid * kRtStageSlices;
#pragma unroll
      for (int j = 0; j < kRtStageSlices; ++j) rs = __fadd_rn(rs, q[j]);
    }
  }
  const bool aborted = done < R;
  if (aborted && tid == 0) {
    // let every copy still in flight land before the CTA can leave
    for (int r = done; r < R && r < done + kRtStages; ++r)
      mbar_wait(smem_u32(&full[r % kRtStages]), static_cast<uint32_t>((r / kRtStages) & 1), nullptr, err);
  }
  if (!aborted && tid < MR * kRtCols) {
    const int m = tid / kRtCols, c = tid % kRtCols;
    float v = rs;
    if (bias) v = __fadd_rn(v, bias[cta * kRtCols + c]);
    sc[m * kRtCols + c] = v;
    if (m < M) y[static_cast<size_t>(m) * N + cta * kRtCols + c] = v;
  }
  // every CTA's scores are in its shared memory before anyone reads them
  cluster_sync_all();
  const int m = cta + ncta * warp;  // this warp's row, if any (rows < 8 * ncta >= M)
  if (!aborted && m < M) {
    const uint32_t base = smem_u32(&sc[m * kRtCols]);
    auto load = [&](int j) { return ld_dsmem_f32(mapa_shared(base + 4u * (j % kRtCols), j / kRtCols)); };
    float *prow = probs ? probs + static_cast<size_t>(m) * N : nullptr;
    int32_t *irow = ids + static_cast<size_t>(m) * top_k;
    float *wrow = wts + static_cast<size_t>(m) * top_k;
    if (N <= 32) topk_select_warp<1>(load, N, top_k, irow, wrow, prow, lane);
    else if (N <= 64) topk_select_warp<2>(load, N, top_k, irow, wrow, prow, lane);
    else if (N <= 128) topk_select_warp<4>(load, N, top_k, irow, wrow, prow, lane);
    else topk_select_warp<8>(load, N, top_k, irow, wrow, prow, lane);
  }
  // no CTA leaves while another may still read its shared memory
  cluster_sync_all();
}

// ------------------------------------------------------------------- host --
// Shapes the one-kernel path takes: N a multiple of 16 up to 256 (one cluster
// of N/16 CTAs), K a multiple of 512, top_k <= 16, M <= kRtMaxM.
bool router_topk_fused_supported(int64_t M, int64_t K, int64_t N, int32_t top_k) {
  return M >= 1 && M <= kRtMaxM && N % kRtCols == 0 && N / kRtCols >= 1 &&
         N / kRtCols <= kRtMaxCluster && K % kRtStageK == 0 && top_k >= 1 && top_k <= 16 && top_k <= N;
}

template <int MR, typename XT>
static bi_status launch_rt(const XT *x, const float *w, const float *b, float *y, float *probs,
                           int32_t *ids, float *wts, int64_t M, int64_t K, int64_t N, int32_t top_k,
                           cudaStream_t stream) {
  using Cf = RtCfg<MR, XT>;
  auto kern = router_topk_cluster_kernel<MR, XT>;
  const int ncta = static_cast<int>(N / kRtCols);
  static ContextSetup setup;
  static int schedulable[64][kRtMaxCluster + 1];  // per device: 1 yes, -1 no, 0 not checked
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) {
    set_error("device ordinal %d out of range", dev);
    return BI_ERR_CUDA;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(ncta);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(ncta));
  cfg.blockDim = dim3(kRtThreads);
  cfg.dynamicSmemBytes = Cf::kSmem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (setup.pending(dev)) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cf::kSmem) != cudaSuccess ||
        cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
      cudaGetLastError();
      set_error("router+top-k cluster kernel: cannot set its attributes");
      return BI_ERR_CUDA;
    }
    for (int c = 0; c <= kRtMaxCluster; ++c) schedulable[dev][c] = 0;
    setup.done(dev);
  }
  if (schedulable[dev][ncta] == 0) {
    // a cluster of up to 16 CTAs with ~200 KB of shared memory each needs
    // that many SMs free in one GPC; ask once per context and size
    int clusters = 0;
    const cudaError_t e = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
    if (e != cudaSuccess) cudaGetLastError();
    schedulable[dev][ncta] = (e == cudaSuccess && clusters > 0) ? 1 : -1;
  }
  if (schedulable[dev][ncta] < 0) {
    set_error("router+top-k: a cluster of %d CTAs cannot be scheduled on this device", ncta);
    return BI_ERR_UNSUPPORTED;
  }
  cfg.numAttrs = 2;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, x, w, b, y, probs, ids, wts, static_cast<int>(M),
                                           static_cast<int>(K), static_cast<int>(N), top_k,
                                           device_error_word());
  if (e != cudaSuccess) {
    cudaGetLastError();
    set_error("router+top-k cluster kernel launch: %s", cudaGetErrorString(e));
    return BI_ERR_CUDA;
  }
  return BI_OK;
}

// One launch: y, ids, wts (and probs) for M <= kRtMaxM rows.  Returns
// BI_ERR_UNSUPPORTED (and launches nothing) when the shape is not one the
// kernel takes or its cluster cannot be scheduled; the caller then takes the
// two-grid path, which gives the same bits.
template <typename XT>
bi_status launch_router_topk_fused(const XT *x, const float *w, const float *b, float *y, float *probs,
                                   int32_t *ids, float *wts, int64_t M, int64_t K, int64_t N, int32_t top_k,
                                   cudaStream_t stream) {
  if (!router_topk_fused_supported(M, K, N, top_k)) {
    set_error("router+top-k one-kernel path: unsupported shape (M=%lld K=%lld N=%lld top_k=%d)",
              (long long)M, (long long)K, (long long)N, top_k);
    return BI_ERR_UNSUPPORTED;
  }
  if (M == 1) return launch_rt<1, XT>(x, w, b, y, probs, ids, wts, M, K, N, top_k, stream);
  if (M == 2) return launch_rt<2, XT>(x, w, b, y, probs, ids, wts, M, K, N, top_k, stream);
  return launch_rt<4, XT>(x, w, b, y, probs, ids, wts, M, K, N, top_k, stream);
}

template bi_status launch_router_topk_fused<float>(const float *, const float *, const float *, float *,
                                                   float *, int32_t *, float *, int64_t, int64_t, int64_t,
                                                   int32_t, cudaStream_t);
template bi_status launch_router_topk_fused<__nv_bfloat16>(const __nv_bfloat16 *, const float *, const float *,
                                                           float *, float *, int32_t *, float *, int64_t,
                                                           int64_t, int64_t, int32_t, cudaStream_t);

}  // namespace bimoe
