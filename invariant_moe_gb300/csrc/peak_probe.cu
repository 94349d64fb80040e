// peak_probe.cu -- FP32 FMA throughput probe used by the benchmark to
// measure the FP32 (non-tensor) roofline denominator of this GPU, and the
// wait-timeout probe the tests use to exercise the bounded-wait discipline.
//
// Every thread runs kChains independent __fmaf_rn chains for `iters` steps
// (no memory traffic inside the loop), so the kernel is bound by the FP32
// pipe alone; one result per thread is written so the work cannot be
// removed.  The probe is not part of the MoE path.
#include "bimoe_internal.cuh"

namespace bimoe {

constexpr int kChains = 16;

__global__ void __launch_bounds__(256) fp32_fma_probe_kernel(float *__restrict__ out, int iters,
                                                             float a, float b) {
  float v[kChains];
#pragma unroll
  for (int c = 0; c < kChains; ++c) v[c] = static_cast<float>(threadIdx.x + c) * 1e-7f;
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int c = 0; c < kChains; ++c) v[c] = __fmaf_rn(v[c], a, b);
  }
  float s = 0.0f;
#pragma unroll
  for (int c = 0; c < kChains; ++c) s = __fadd_rn(s, v[c]);
  out[static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x] = s;
}

// One thread waits, through one of the library's bounded waits, for
// something that never happens: which = 0, a phase of an mbarrier that
// nothing arrives on; which = 1, an arrival count (a word of this probe that
// nothing raises) to reach 1.  The wait gives up after its limit, records
// BI_DEVERR_WAIT_TIMEOUT in the device error word and the kernel returns
// normally.
__device__ unsigned g_probe_count;  // zero, never written

__global__ void wait_timeout_probe_kernel(int which, int *err) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  if (which == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_barrier_init();
    (void)mbar_wait(smem_u32(&bar), 0, nullptr, err);
  } else {
    (void)wait_count_geq(&g_probe_count, 1u, nullptr, err);
  }
}

bi_status launch_wait_timeout_probe(int which, cudaStream_t stream) {
  wait_timeout_probe_kernel<<<1, 32, 0, stream>>>(which, device_error_word());
  BI_CHECK_LAUNCH();
  return BI_OK;
}

bi_status launch_fp32_fma_probe(float *out, int64_t blocks, int32_t iters, cudaStream_t stream) {
  fp32_fma_probe_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(out, iters, 0.999999f,
                                                                           1e-7f);
  BI_CHECK_LAUNCH();
  return BI_OK;
}

}  // namespace bimoe
