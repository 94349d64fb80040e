// peak_probe.cu -- FP32 FMA throughput probe used by the benchmark to
// measure the FP32 (non-tensor) roofline denominator of this GPU.
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

bi_status launch_fp32_fma_probe(float *out, int64_t blocks, int32_t iters, cudaStream_t stream) {
  fp32_fma_probe_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(out, iters, 0.999999f,
                                                                           1e-7f);
  BI_CHECK_LAUNCH();
  return BI_OK;
}

}  // namespace bimoe
