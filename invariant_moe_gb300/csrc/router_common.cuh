// router_common.cuh -- pieces of the fp32 router's per-element recipe shared
// by the router kernels (router.cu) and the fused decode router + top-k
// kernel (router_topk.cu): the slice length, staging pitches, the exact
// widening of bf16 tokens, and the cp.async / 1-D bulk copy wrappers.
#pragma once

#include "bimoe_internal.cuh"

namespace bimoe {

constexpr int kSlice = 128;

// Padded shared row for one slice (128 fp32 + 4): lanes walking different
// slices along k then read distinct banks.
constexpr int kSlicePad = kSlice + 4;

// x may be fp32 or bf16 (the MoE layer's tokens); a bf16 value converts to
// fp32 exactly (its bits are the high half of the fp32's), so both give the
// same per-element sequence.  Shared-memory row pitches (elements) keep every
// row 16-byte aligned for the bulk / cp.async copies.
template <typename XT> struct XPitch;
template <> struct XPitch<float> { static constexpr int slice = kSlicePad, round = 8 * kSlice + 4; };
template <> struct XPitch<__nv_bfloat16> { static constexpr int slice = kSlice + 8, round = 8 * kSlice + 8; };

// Four consecutive x values from shared memory, as fp32.
__device__ __forceinline__ float4 ld_x4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ float4 ld_x4(const __nv_bfloat16 *p) {
  const uint2 u = *reinterpret_cast<const uint2 *>(p);
  return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                     __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
}


__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// 1-D bulk copy global -> shared (TMA engine), completion counted in bytes
// on an mbarrier.  Addresses 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

}  // namespace bimoe
