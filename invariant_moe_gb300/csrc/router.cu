// router.cu -- fp32 GateLinear router GEMM y = x W^T (+ b) on CUDA cores.
//
// Source: "[BI][DSv4] Batch-invariant GateLinear router with fp32 persistent
// matmul", sections "What" (fp32 scores, bias kept) and "A correction to why
// the key excludes M" (the reduction order is a contract that must not depend
// on M).  Tensor cores are not used: TF32 would round the operands, and the
// page's tolerance (atol 2e-3 / rtol 1e-4) is an fp32 one.
//
// Per-element reduction recipe (fixed by K, identical in every schedule):
//   K is cut into S = K/128 contiguous slices;
//   p_s = fmaf chain over k = 128s .. 128s+127 in increasing k, from +0.0f;
//   acc = +0.0f; acc = acc + p_s for s = 0 .. S-1 (round-to-nearest adds);
//   y = acc (+ b[n], added last).
// Every operation is an explicit __fmaf_rn / __fadd_rn, so the compiler has no
// contraction or reassociation freedom.  Schedules differ only in which
// thread evaluates which p_s and in tile sizes; they are chosen from M for
// speed:
//   rows    (M <= 8)      one warp per weight row, lanes own slices: streams
//                         W once at HBM rate for decode batches
//   sliced  (8 < M < 384) 8x32 output tile per CTA, one warp per slice, the
//                         partials combined in slice order through smem
//   tiled   (M >= 384)    64x64 register-tiled FFMA kernel, 8x8 outputs per
//                         thread, slices summed into a running register sum
#include "bimoe_internal.cuh"

namespace bimoe {

constexpr int kSlice = 128;

// -------------------------------------------------------------------- rows --
// Lane l of a warp serves weight row n = n0 + l / LPR and slices
// s = l % LPR, l % LPR + LPR, ...; MR token rows share each W load.
template <int MR>
__global__ void __launch_bounds__(32) router_rows_kernel(const float *__restrict__ x,
                                                         const float *__restrict__ w,
                                                         const float *__restrict__ bias,
                                                         float *__restrict__ y, int M, int K,
                                                         int N, int LPR) {
  extern __shared__ float part[];  // [rows_per_warp][MR][S]
  const int lane = threadIdx.x;
  const int S = K / kSlice;
  const int rpw = 32 / LPR;
  const int r = lane / LPR;
  const int n = blockIdx.x * rpw + r;
  const int m0 = blockIdx.y * MR;
  if (n < N) {
    const float4 *w4 = reinterpret_cast<const float4 *>(w + static_cast<size_t>(n) * K);
    const float4 *x4[MR];
#pragma unroll
    for (int i = 0; i < MR; ++i) {
      const int m = min(m0 + i, M - 1);
      x4[i] = reinterpret_cast<const float4 *>(x + static_cast<size_t>(m) * K);
    }
    for (int s = lane % LPR; s < S; s += LPR) {
      float p[MR];
#pragma unroll
      for (int i = 0; i < MR; ++i) p[i] = 0.0f;
#pragma unroll 8
      for (int j = 0; j < kSlice / 4; ++j) {
        const float4 wv = __ldg(w4 + s * (kSlice / 4) + j);
#pragma unroll
        for (int i = 0; i < MR; ++i) {
          const float4 xv = __ldg(x4[i] + s * (kSlice / 4) + j);
          p[i] = __fmaf_rn(xv.x, wv.x, p[i]);
          p[i] = __fmaf_rn(xv.y, wv.y, p[i]);
          p[i] = __fmaf_rn(xv.z, wv.z, p[i]);
          p[i] = __fmaf_rn(xv.w, wv.w, p[i]);
        }
      }
#pragma unroll
      for (int i = 0; i < MR; ++i) part[(r * MR + i) * S + s] = p[i];
    }
  }
  __syncwarp();
  for (int c = lane; c < rpw * MR; c += 32) {
    const int rr = c / MR, i = c % MR;
    const int nn = blockIdx.x * rpw + rr;
    const int m = m0 + i;
    if (nn < N && m < M) {
      float acc = 0.0f;
      for (int s = 0; s < S; ++s) acc = __fadd_rn(acc, part[c * S + s]);
      if (bias) acc = __fadd_rn(acc, bias[nn]);
      y[static_cast<size_t>(m) * N + nn] = acc;
    }
  }
}

// ------------------------------------------------------------------ sliced --
// CTA = G warps, output tile 8 (m) x 32 (n): lane l owns column n0 + l and
// the 8 rows.  In round r warp g evaluates slice s = r*G + g for the whole
// tile; partials meet in shared memory and thread (i, l) adds them to its
// running sum in slice order.
template <int G>
__global__ void __launch_bounds__(32 * G) router_sliced_kernel(const float *__restrict__ x,
                                                               const float *__restrict__ w,
                                                               const float *__restrict__ bias,
                                                               float *__restrict__ y, int M,
                                                               int K, int N) {
  __shared__ float part[G][8][32];
  const int lane = threadIdx.x & 31;
  const int g = threadIdx.x >> 5;
  const int S = K / kSlice;
  const int n0 = blockIdx.x * 32;
  const int m0 = blockIdx.y * 8;
  const int nl = min(n0 + lane, N - 1);
  const float4 *w4 = reinterpret_cast<const float4 *>(w + static_cast<size_t>(nl) * K);
  const float4 *x4[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    x4[i] = reinterpret_cast<const float4 *>(x + static_cast<size_t>(min(m0 + i, M - 1)) * K);
  // combine role: thread t owns output (m0 + t/32, n0 + t%32) for t < 256
  const int ci = threadIdx.x >> 5, cl = threadIdx.x & 31;
  float acc = 0.0f;
  for (int base = 0; base < S; base += G) {
    const int s = base + g;
    if (s < S) {
      float p[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) p[i] = 0.0f;
#pragma unroll 4
      for (int j = 0; j < kSlice / 4; ++j) {
        const float4 wv = __ldg(w4 + s * (kSlice / 4) + j);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 xv = __ldg(x4[i] + s * (kSlice / 4) + j);
          p[i] = __fmaf_rn(xv.x, wv.x, p[i]);
          p[i] = __fmaf_rn(xv.y, wv.y, p[i]);
          p[i] = __fmaf_rn(xv.z, wv.z, p[i]);
          p[i] = __fmaf_rn(xv.w, wv.w, p[i]);
        }
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) part[g][i][lane] = p[i];
    }
    __syncthreads();
    if (threadIdx.x < 256) {
      const int ng = min(G, S - base);
      for (int gg = 0; gg < ng; ++gg) acc = __fadd_rn(acc, part[gg][ci][cl]);
    }
    __syncthreads();
  }
  if (threadIdx.x < 256) {
    const int m = m0 + ci, n = n0 + cl;
    if (m < M && n < N) {
      if (bias) acc = __fadd_rn(acc, bias[n]);
      y[static_cast<size_t>(m) * N + n] = acc;
    }
  }
}

// ------------------------------------------------------------------- tiled --
// 64x64 output tile, 64 threads in an 8x8 grid, 8x8 outputs per thread (rows
// tr*4+{0..3} and 32+tr*4+{0..3}, same for columns).  K advances in chunks of
// 16 through double-buffered, transposed shared-memory tiles; at every
// 128-element slice boundary the chain value is added to the running sum and
// restarted from +0.0f.
constexpr int kTBM = 64, kTBN = 64, kTBK = 16, kTPad = 4;

__global__ void __launch_bounds__(64) router_tiled_kernel(const float *__restrict__ x,
                                                          const float *__restrict__ w,
                                                          const float *__restrict__ bias,
                                                          float *__restrict__ y, int M, int K,
                                                          int N) {
  __shared__ __align__(16) float xs[2][kTBK][kTBM + kTPad];
  __shared__ __align__(16) float ws[2][kTBK][kTBN + kTPad];
  const int tid = threadIdx.x;
  const int tr = tid >> 3, tc = tid & 7;
  const int m0 = blockIdx.y * kTBM, n0 = blockIdx.x * kTBN;
  const float4 *xg = reinterpret_cast<const float4 *>(
      x + static_cast<size_t>(min(m0 + tid, M - 1)) * K);
  const float4 *wg = reinterpret_cast<const float4 *>(
      w + static_cast<size_t>(min(n0 + tid, N - 1)) * K);

  float p[8][8], acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      p[i][j] = 0.0f;
      acc[i][j] = 0.0f;
    }

  float4 xr[4], wr[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    xr[q] = __ldg(xg + q);
    wr[q] = __ldg(wg + q);
  }
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    xs[0][4 * q + 0][tid] = xr[q].x;
    xs[0][4 * q + 1][tid] = xr[q].y;
    xs[0][4 * q + 2][tid] = xr[q].z;
    xs[0][4 * q + 3][tid] = xr[q].w;
    ws[0][4 * q + 0][tid] = wr[q].x;
    ws[0][4 * q + 1][tid] = wr[q].y;
    ws[0][4 * q + 2][tid] = wr[q].z;
    ws[0][4 * q + 3][tid] = wr[q].w;
  }
  __syncthreads();

  const int nchunks = K / kTBK;
  constexpr int kChunksPerSlice = kSlice / kTBK;
  for (int c = 0; c < nchunks; ++c) {
    const int buf = c & 1;
    const bool more = (c + 1) < nchunks;
    if (more) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        xr[q] = __ldg(xg + (c + 1) * (kTBK / 4) + q);
        wr[q] = __ldg(wg + (c + 1) * (kTBK / 4) + q);
      }
    }
#pragma unroll
    for (int k = 0; k < kTBK; ++k) {
      const float4 a0 = *reinterpret_cast<const float4 *>(&xs[buf][k][tr * 4]);
      const float4 a1 = *reinterpret_cast<const float4 *>(&xs[buf][k][32 + tr * 4]);
      const float4 b0 = *reinterpret_cast<const float4 *>(&ws[buf][k][tc * 4]);
      const float4 b1 = *reinterpret_cast<const float4 *>(&ws[buf][k][32 + tc * 4]);
      const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) p[i][j] = __fmaf_rn(a[i], b[j], p[i][j]);
    }
    if ((c + 1) % kChunksPerSlice == 0) {
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          acc[i][j] = __fadd_rn(acc[i][j], p[i][j]);
          p[i][j] = 0.0f;
        }
    }
    if (more) {
      const int nb = buf ^ 1;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        xs[nb][4 * q + 0][tid] = xr[q].x;
        xs[nb][4 * q + 1][tid] = xr[q].y;
        xs[nb][4 * q + 2][tid] = xr[q].z;
        xs[nb][4 * q + 3][tid] = xr[q].w;
        ws[nb][4 * q + 0][tid] = wr[q].x;
        ws[nb][4 * q + 1][tid] = wr[q].y;
        ws[nb][4 * q + 2][tid] = wr[q].z;
        ws[nb][4 * q + 3][tid] = wr[q].w;
      }
    }
    __syncthreads();
  }

#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int m = m0 + (i < 4 ? tr * 4 + i : 32 + tr * 4 + (i - 4));
    if (m >= M) continue;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int n = n0 + (j < 4 ? tc * 4 + j : 32 + tc * 4 + (j - 4));
      if (n >= N) continue;
      float v = acc[i][j];
      if (bias) v = __fadd_rn(v, bias[n]);
      y[static_cast<size_t>(m) * N + n] = v;
    }
  }
}

// ------------------------------------------------------- negative control --
// One thread per output; the K split depends on M (the defect the recipe
// above exists to rule out).  Test use only.
__global__ void router_negctl_kernel(const float *__restrict__ x, const float *__restrict__ w,
                                     const float *__restrict__ bias, float *__restrict__ y, int M,
                                     int K, int N, int L) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= M * N) return;
  const int m = idx / N, n = idx % N;
  const float *xr = x + static_cast<size_t>(m) * K;
  const float *wr = w + static_cast<size_t>(n) * K;
  float acc = 0.0f;
  for (int s0 = 0; s0 < K; s0 += L) {
    float p = 0.0f;
    for (int k = s0; k < s0 + L; ++k) p = __fmaf_rn(xr[k], wr[k], p);
    acc = __fadd_rn(acc, p);
  }
  if (bias) acc = __fadd_rn(acc, bias[n]);
  y[idx] = acc;
}

// -------------------------------------------------------------------- cast --
__global__ void cast_bf16_f32_kernel(const __nv_bfloat16 *__restrict__ x, float *__restrict__ y,
                                     int64_t n) {
  const int64_t i0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) * 8;
  if (i0 + 8 <= n && (reinterpret_cast<uintptr_t>(x) & 15) == 0 &&
      (reinterpret_cast<uintptr_t>(y) & 15) == 0) {
    const uint4 v = *reinterpret_cast<const uint4 *>(x + i0);
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&v);
    float4 a, b;
    float2 f0 = __bfloat1622float2(h[0]), f1 = __bfloat1622float2(h[1]);
    float2 f2 = __bfloat1622float2(h[2]), f3 = __bfloat1622float2(h[3]);
    a = make_float4(f0.x, f0.y, f1.x, f1.y);
    b = make_float4(f2.x, f2.y, f3.x, f3.y);
    reinterpret_cast<float4 *>(y + i0)[0] = a;
    reinterpret_cast<float4 *>(y + i0)[1] = b;
  } else {
    for (int64_t i = i0; i < i0 + 8 && i < n; ++i) y[i] = __bfloat162float(x[i]);
  }
}

// ------------------------------------------------------------------- host --
bi_status launch_router(const float *x, const float *w, const float *b, float *y, int64_t M,
                        int64_t K, int64_t N, int schedule, cudaStream_t stream) {
  const int S = static_cast<int>(K / kSlice);
  if (schedule == 0) schedule = (M <= 8) ? 1 : (M < 384 ? 2 : 3);
  if (schedule == 1) {
    int LPR = 1;
    while (LPR * 2 <= S && LPR * 2 <= 32) LPR *= 2;
    const int rpw = 32 / LPR;
    const int mr = M <= 1 ? 1 : (M <= 2 ? 2 : (M <= 4 ? 4 : 8));
    dim3 grid(static_cast<unsigned>((N + rpw - 1) / rpw), static_cast<unsigned>((M + mr - 1) / mr));
    const size_t smem = static_cast<size_t>(rpw) * mr * S * sizeof(float);
    if (grid.y > 65535u || smem > 48 * 1024) {
      set_error("router rows schedule: M=%lld or K=%lld too large for it", (long long)M,
                (long long)K);
      return BI_ERR_UNSUPPORTED;
    }
    switch (mr) {
      case 1: router_rows_kernel<1><<<grid, 32, smem, stream>>>(x, w, b, y, (int)M, (int)K, (int)N, LPR); break;
      case 2: router_rows_kernel<2><<<grid, 32, smem, stream>>>(x, w, b, y, (int)M, (int)K, (int)N, LPR); break;
      case 4: router_rows_kernel<4><<<grid, 32, smem, stream>>>(x, w, b, y, (int)M, (int)K, (int)N, LPR); break;
      default: router_rows_kernel<8><<<grid, 32, smem, stream>>>(x, w, b, y, (int)M, (int)K, (int)N, LPR); break;
    }
  } else if (schedule == 2) {
    dim3 grid(static_cast<unsigned>((N + 31) / 32), static_cast<unsigned>((M + 7) / 8));
    if (grid.y > 65535u) {
      set_error("router sliced schedule: M=%lld too large for it", (long long)M);
      return BI_ERR_UNSUPPORTED;
    }
    if (S % 16 == 0)
      router_sliced_kernel<16><<<grid, 512, 0, stream>>>(x, w, b, y, (int)M, (int)K, (int)N);
    else
      router_sliced_kernel<8><<<grid, 256, 0, stream>>>(x, w, b, y, (int)M, (int)K, (int)N);
  } else if (schedule == 3) {
    dim3 grid(static_cast<unsigned>((N + kTBN - 1) / kTBN), static_cast<unsigned>((M + kTBM - 1) / kTBM));
    if (grid.y > 65535u) {
      set_error("router tiled schedule: M=%lld too large for it", (long long)M);
      return BI_ERR_UNSUPPORTED;
    }
    router_tiled_kernel<<<grid, 64, 0, stream>>>(x, w, b, y, (int)M, (int)K, (int)N);
  } else {
    set_error("unknown router schedule %d", schedule);
    return BI_ERR_INVALID_ARG;
  }
  BI_CHECK_LAUNCH();
  return BI_OK;
}

bi_status launch_router_negctl(const float *x, const float *w, const float *b, float *y,
                               int64_t M, int64_t K, int64_t N, cudaStream_t stream) {
  const int L = (M <= 16 && K % 256 == 0) ? 256 : static_cast<int>(K);
  const int64_t total = M * N;
  const int threads = 256;
  router_negctl_kernel<<<static_cast<unsigned>((total + threads - 1) / threads), threads, 0, stream>>>(
      x, w, b, y, (int)M, (int)K, (int)N, L);
  BI_CHECK_LAUNCH();
  return BI_OK;
}

bi_status launch_cast_bf16_f32(const void *x, float *y, int64_t n, cudaStream_t stream) {
  const int threads = 256;
  const int64_t blocks = (n + threads * 8 - 1) / (threads * 8);
  cast_bf16_f32_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
      static_cast<const __nv_bfloat16 *>(x), y, n);
  BI_CHECK_LAUNCH();
  return BI_OK;
}

}  // namespace bimoe
