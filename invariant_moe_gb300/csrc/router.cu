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
//   rows    (M <= 2; M <= 4 where split does not apply) one warp per weight
//           row and up to 4 token rows, lanes own slices: streams W
//   split   (2 < M < 3072) the slices spread over a cluster of 2..8 CTAs,
//           one slice per warp, lane tiles of 2x2 .. 8x4 outputs picked from
//           M; the slice partials meet in shared memory and are summed in
//           slice order across the cluster (distributed shared memory)
//   sliced  (4 < M < 384 where split does not apply) 8x16 output tile per
//           CTA, one warp per slice, partials combined through smem
//   tiled   (M >= 3072; M >= 384 where split does not apply) register-tiled
//           FFMA kernel over 128 or 256 columns, TMR x TN outputs per thread
//           (7x8 once the 28-row tiles cover 70 % of the SMs, else 7x4 or
//           smaller), cp.async ring, slices summed into a running sum; extra
//           groups of warps split the slices of a tile (partials joined in
//           slice order)
// split applies when K/128 splits into 2..8 CTAs of 4 or 8 slices.
// x is fp32, or bf16 (the MoE layer's tokens) read as its exact fp32 values;
// both give the same bits.
#include "router_common.cuh"

namespace bimoe {

// -------------------------------------------------------------------- rows --
// One warp per weight row n and MR token rows; lane l owns slice l of each
// group of 32 slices.  Each lane bulk-copies its slice of the W row and of
// the MR x rows (512 B each) into padded shared rows, then runs its MR
// chains from there; the partials meet in shared memory and lane i < MR adds
// them in slice order.
template <int MR, typename XT>
__global__ void __launch_bounds__(32) router_rows_kernel(const XT *__restrict__ x,
                                                         const float *__restrict__ w,
                                                         const float *__restrict__ bias,
                                                         float *__restrict__ y, int M, int K,
                                                         int N, int *err, unsigned *zero_words, int n_zero) {
  constexpr int XP = XPitch<XT>::slice;
  extern __shared__ __align__(16) float sm[];
  float *ws = sm;                                              // [32][kSlicePad]
  XT *xs = reinterpret_cast<XT *>(sm + 32 * kSlicePad);        // [MR][32][XP]
  float *part = reinterpret_cast<float *>(xs + MR * 32 * XP);  // [MR][S]
  __shared__ __align__(8) uint64_t bar;
  const int lane = threadIdx.x;
  griddep_wait();
  // a single wave of one-warp CTAs: the next grid on the stream (which waits
  // for this one before reading anything) may start beside it (the decode
  // layer's expert launch sets up its CTAs meanwhile)
  griddep_launch_dependents();
  if (zero_words && blockIdx.x == 0 && blockIdx.y == 0)
    for (int i = lane; i < n_zero; i += 32) zero_words[i] = 0u;
  const int S = K / kSlice;
  const int n = blockIdx.x;
  const int m0 = blockIdx.y * MR;
  const float *wrow = w + static_cast<size_t>(n) * K;
  const uint32_t b = smem_u32(&bar);
  if (lane == 0) {
    mbar_init(b, 1);
    fence_barrier_init();
  }
  __syncwarp();
  uint32_t phase = 0;
  for (int g0 = 0; g0 < S; g0 += 32) {
    const int ns = min(32, S - g0);
    if (lane == 0)
      mbar_arrive_expect_tx(b, static_cast<uint32_t>(ns) * kSlice * (4 + MR * sizeof(XT)));
    __syncwarp();
    if (lane < ns) {
      const int k0 = (g0 + lane) * kSlice;
      bulk_g2s(smem_u32(ws + lane * kSlicePad), wrow + k0, kSlice * 4, b);
#pragma unroll
      for (int i = 0; i < MR; ++i)
        bulk_g2s(smem_u32(xs + (i * 32 + lane) * XP),
                 x + static_cast<size_t>(min(m0 + i, M - 1)) * K + k0, kSlice * sizeof(XT), b);
    }
    const bool got = mbar_wait(b, phase, nullptr, err);
    if (!__all_sync(0xffffffffu, got)) {
      if (!got) mbar_wait(b, phase, nullptr, err);  // let the copies land before exit
      return;
    }
    phase ^= 1u;
    if (lane < ns) {
      float p[MR];
#pragma unroll
      for (int i = 0; i < MR; ++i) p[i] = 0.0f;
      const float *wl = ws + lane * kSlicePad;
#pragma unroll 8
      for (int k = 0; k < kSlice; k += 4) {
        const float4 wv = *reinterpret_cast<const float4 *>(wl + k);
#pragma unroll
        for (int i = 0; i < MR; ++i) {
          const float4 xv = ld_x4(xs + (i * 32 + lane) * XP + k);
          p[i] = __fmaf_rn(xv.x, wv.x, p[i]);
          p[i] = __fmaf_rn(xv.y, wv.y, p[i]);
          p[i] = __fmaf_rn(xv.z, wv.z, p[i]);
          p[i] = __fmaf_rn(xv.w, wv.w, p[i]);
        }
      }
#pragma unroll
      for (int i = 0; i < MR; ++i) part[i * S + g0 + lane] = p[i];
    }
    __syncwarp();
  }
  if (lane < MR && m0 + lane < M) {
    float acc = 0.0f;
    const float *pr = part + lane * S;
#pragma unroll 8
    for (int sl = 0; sl < S; ++sl) acc = __fadd_rn(acc, pr[sl]);
    if (bias) acc = __fadd_rn(acc, bias[n]);
    y[static_cast<size_t>(m0 + lane) * N + n] = acc;
  }
}

// ------------------------------------------------------------------ sliced --
// CTA = 8 warps, output tile 8 (m) x 16 (n).  K is processed in rounds of 8
// slices; in a round warp g evaluates slice 8r+g for the whole tile, lane l
// owning rows {l/8, l/8+4} x columns {l%8, l%8+8}.  A round's 8 x rows and
// 16 W rows (8 slices = 4 KB contiguous each) are bulk-copied into a
// double-buffered shared tile (row stride 1028 floats: conflict-free for
// lanes reading different rows at the same k) while the previous round
// computes.  Partials meet in shared memory and thread (i, j) adds them to
// its running sum in slice order.
constexpr int kSlMT = 8, kSlNT = 16, kSlG = 8;
constexpr int kSlRow = kSlG * kSlice + 4;  // floats per staged W row
// bytes of one stage: MT x rows (element type XT) then NT W rows
template <typename XT>
__host__ __device__ constexpr int sl_stage_bytes() {
  return kSlMT * XPitch<XT>::round * static_cast<int>(sizeof(XT)) + kSlNT * kSlRow * 4;
}

template <typename XT>
__global__ void __launch_bounds__(256) router_sliced_kernel(const XT *__restrict__ x,
                                                            const float *__restrict__ w,
                                                            const float *__restrict__ bias,
                                                            float *__restrict__ y, int M, int K,
                                                            int N, int *err, unsigned *zero_words, int n_zero) {
  constexpr int XP = XPitch<XT>::round;
  constexpr int kStageB = sl_stage_bytes<XT>();
  extern __shared__ __align__(16) float sm[];
  uint8_t *stage_buf = reinterpret_cast<uint8_t *>(sm);                     // [2] x [MT][XP] XT, W [NT][kSlRow]
  float *part = reinterpret_cast<float *>(stage_buf + 2 * kStageB);         // [G][MT][NT]
  auto xrow = [&](int buf, int row) {
    return reinterpret_cast<XT *>(stage_buf + buf * kStageB) + row * XP;
  };
  auto wrow = [&](int buf, int row) {
    return reinterpret_cast<float *>(stage_buf + buf * kStageB + kSlMT * XP * sizeof(XT)) + row * kSlRow;
  };
  __shared__ __align__(8) uint64_t bars[2];
  const int tid = threadIdx.x;
  griddep_wait();
  if (zero_words && blockIdx.x == 0 && blockIdx.y == 0)
    for (int i = tid; i < n_zero; i += 256) zero_words[i] = 0u;
  const int g = tid >> 5, lane = tid & 31;
  const int S = K / kSlice;
  const int rounds = (S + kSlG - 1) / kSlG;
  const int m0 = blockIdx.y * kSlMT, n0 = blockIdx.x * kSlNT;

  if (tid == 0) {
    mbar_init(smem_u32(&bars[0]), 1);
    mbar_init(smem_u32(&bars[1]), 1);
    fence_barrier_init();
  }
  __syncthreads();
  // lanes of warp 0 issue the copies of a round: row q (< 24) by lane q
  auto load_round = [&](int rd) {
    if (g != 0) return;
    const int buf = rd & 1;
    const uint32_t b = smem_u32(&bars[buf]);
    const int ns = min(kSlG, S - rd * kSlG);
    const uint32_t xbytes = static_cast<uint32_t>(ns) * kSlice * sizeof(XT);
    const uint32_t wbytes = static_cast<uint32_t>(ns) * kSlice * 4;
    if (lane == 0) mbar_arrive_expect_tx(b, xbytes * kSlMT + wbytes * kSlNT);
    __syncwarp();
    if (lane < kSlMT) {
      bulk_g2s(smem_u32(xrow(buf, lane)),
               x + static_cast<size_t>(min(m0 + lane, M - 1)) * K + rd * kSlG * kSlice, xbytes, b);
    } else if (lane < kSlMT + kSlNT) {
      bulk_g2s(smem_u32(wrow(buf, lane - kSlMT)),
               w + static_cast<size_t>(min(n0 + lane - kSlMT, N - 1)) * K + rd * kSlG * kSlice, wbytes, b);
    }
  };

  const int cr = lane >> 3, cc = lane & 7;  // compute role: rows cr, cr+4; cols cc, cc+8
  const int oi = tid >> 4, oj = tid & 15;   // combine role (tid < 128)
  float acc = 0.0f;
  bool ok = true;
  load_round(0);
  uint32_t phases = 0;  // bit b: parity of the next wait on bars[b]
  for (int rd = 0; rd < rounds; ++rd) {
    if (rd + 1 < rounds) load_round(rd + 1);
    const int buf = rd & 1;
    if (!mbar_wait(smem_u32(&bars[buf]), (phases >> buf) & 1u, nullptr, err)) ok = false;
    phases ^= 1u << buf;
    if (__syncthreads_or(!ok)) break;
    const int sl = rd * kSlG + g;
    if (sl < S) {
      float p00 = 0.0f, p01 = 0.0f, p10 = 0.0f, p11 = 0.0f;
      const XT *x0 = xrow(buf, cr) + g * kSlice;
      const XT *x1 = xrow(buf, cr + 4) + g * kSlice;
      const float *w0 = wrow(buf, cc) + g * kSlice;
      const float *w1 = wrow(buf, cc + 8) + g * kSlice;
#pragma unroll 8
      for (int k = 0; k < kSlice; k += 4) {
        const float4 a0 = ld_x4(x0 + k);
        const float4 a1 = ld_x4(x1 + k);
        const float4 b0 = *reinterpret_cast<const float4 *>(w0 + k);
        const float4 b1 = *reinterpret_cast<const float4 *>(w1 + k);
        p00 = __fmaf_rn(a0.x, b0.x, p00); p01 = __fmaf_rn(a0.x, b1.x, p01);
        p10 = __fmaf_rn(a1.x, b0.x, p10); p11 = __fmaf_rn(a1.x, b1.x, p11);
        p00 = __fmaf_rn(a0.y, b0.y, p00); p01 = __fmaf_rn(a0.y, b1.y, p01);
        p10 = __fmaf_rn(a1.y, b0.y, p10); p11 = __fmaf_rn(a1.y, b1.y, p11);
        p00 = __fmaf_rn(a0.z, b0.z, p00); p01 = __fmaf_rn(a0.z, b1.z, p01);
        p10 = __fmaf_rn(a1.z, b0.z, p10); p11 = __fmaf_rn(a1.z, b1.z, p11);
        p00 = __fmaf_rn(a0.w, b0.w, p00); p01 = __fmaf_rn(a0.w, b1.w, p01);
        p10 = __fmaf_rn(a1.w, b0.w, p10); p11 = __fmaf_rn(a1.w, b1.w, p11);
      }
      float *pg = part + g * kSlMT * kSlNT;
      pg[cr * kSlNT + cc] = p00;
      pg[cr * kSlNT + cc + 8] = p01;
      pg[(cr + 4) * kSlNT + cc] = p10;
      pg[(cr + 4) * kSlNT + cc + 8] = p11;
    }
    __syncthreads();
    if (tid < kSlMT * kSlNT) {
      const int ng = min(kSlG, S - rd * kSlG);
      for (int gg = 0; gg < ng; ++gg) acc = __fadd_rn(acc, part[(gg * kSlMT + oi) * kSlNT + oj]);
    }
  }
  if (!ok) {
    // let any copy still in flight land before the CTA exits
    if (tid == 0)
      for (int bb = 0; bb < 2; ++bb) mbar_wait(smem_u32(&bars[bb]), (phases >> bb) & 1u, nullptr, err);
    __syncthreads();
    return;
  }
  if (tid < kSlMT * kSlNT) {
    const int m = m0 + oi, n = n0 + oj;
    if (m < M && n < N) {
      if (bias) acc = __fadd_rn(acc, bias[n]);
      y[static_cast<size_t>(m) * N + n] = acc;
    }
  }
}

// ------------------------------------------------------------------- tiled --
// Register-tiled FFMA kernel for large M.  A group of RB x CB warps (row
// blocks x column blocks of 8*TN columns) covers a BM x BN output tile;
// thread (r, c) of a warp owns rows base + 4i + r (i < TMR) and columns
// base + 8j + c (j < TN).  K advances in chunks of 32 through an NSTG-stage
// cp.async ring of [rows][32 + 4] fp32 tiles (k contiguous, padded so the
// 16-byte loads along k are bank-conflict free); each chunk is consumed four
// k at a time, each output's chain in increasing k.  Every 128 k (4 chunks)
// the chain value is added to the running sum and restarted from +0.0f.
// TW: the W chunk is one TMA copy per group and stage into the 128-byte
// swizzled layout instead (no per-thread copies; 16-byte chunk c of row r
// lands at chunk c ^ (r % 8), which keeps the 8-row loads conflict free).
// A CTA holds G groups over the same tile: group g evaluates slices g, g+G,
// ... and after each round of G slices group 0 adds the round's partials to
// the running sum in slice order through shared memory.  A thread loads
// TMR + TN values per k for TMR x TN FMAs, so the FMA pipe can be at most
// TMR*TN / (4 (TMR + TN)) busy under the shared-memory load rate (one
// wavefront per loaded register per warp): 64 % for 7x4, 93 % for 7x8.
constexpr int kTBK = 32;              // k per chunk
constexpr int kTLd = kTBK + 4;        // padded smem row length (floats)

template <int TMR, int TN, int RB, int CB, int G, int NSTG, typename XT, bool TW = false>
struct TiledCfg {
  static constexpr int GT = 32 * RB * CB;  // threads per group
  static constexpr int BM = RB * 4 * TMR, BN = CB * 8 * TN;
  // x is staged as fp32 whatever its type: bf16 x is widened once as it is
  // written to shared memory instead of at every use
  static constexpr int XLd = kTLd;
  // W rows: padded to 36 floats (cp.async), or 32 floats in the 128-byte
  // swizzled layout a TMA copy writes (TW)
  static constexpr int WLd = TW ? kTBK : kTLd;
  static constexpr int XS = BM * XLd;                                     // x floats per stage
  static constexpr int WS = BN * WLd;                                     // W floats per stage
  // floats of one group's ring (TW: the W stages lead it, and every ring
  // starts 1024-byte aligned, as the swizzled TMA copies need)
  static constexpr int GS = TW ? (NSTG * (XS + WS) + 255) / 256 * 256 : NSTG * (XS + WS);
  static constexpr int PB = (G - 1) * TMR * TN * GT;                      // partial floats
  static constexpr size_t kSmem = (static_cast<size_t>(G) * GS + PB) * sizeof(float) + (TW ? 1024 : 0);
  static constexpr int kMinBlocks = (TMR > 4 || G > 1 || TN > 4) ? 1 : 2;
  static_assert(!TW || ((WS * 4) % 1024 == 0 && (GS * 4) % 1024 == 0), "TW: W stages keep 1024-byte alignment");
};

template <int TMR, int TN, int RB, int CB, int G, int NSTG, typename XT, bool TW = false>
__global__ void __launch_bounds__(TiledCfg<TMR, TN, RB, CB, G, NSTG, XT, TW>::GT * G,
                                  TiledCfg<TMR, TN, RB, CB, G, NSTG, XT, TW>::kMinBlocks)
    router_tiled_kernel(const __grid_constant__ CUtensorMap tmW, const XT *__restrict__ x,
                        const float *__restrict__ w, const float *__restrict__ bias, float *__restrict__ y,
                        int M, int K, int N, int *err) {
  using Cf = TiledCfg<TMR, TN, RB, CB, G, NSTG, XT, TW>;
  constexpr int GT = Cf::GT, BM = Cf::BM, BN = Cf::BN, XLd = Cf::XLd, WLd = Cf::WLd;
  constexpr int XS = Cf::XS, WS = Cf::WS, GS = Cf::GS;
  extern __shared__ __align__(16) float smem_raw_f[];
  // TW: one TMA copy of a group's [BN][32] W chunk per stage, completing on
  // the stage's mbarrier
  __shared__ __align__(8) uint64_t wbar[TW ? G * NSTG : 1];
  float *smem_f = TW ? reinterpret_cast<float *>((reinterpret_cast<uintptr_t>(smem_raw_f) + 1023) &
                                                 ~static_cast<uintptr_t>(1023))
                     : smem_raw_f;

  griddep_wait();
  const int grp = threadIdx.x / GT;
  const int tid = threadIdx.x % GT;
  float *ws = smem_f + grp * GS;                // [NSTG][BN][WLd]
  float *xs = smem_f + grp * GS + NSTG * WS;    // [NSTG][BM][XLd] fp32
  float *pb = smem_f + G * GS;               // [G-1][TMR*TN][GT] slice partials of groups >= 1
  if (TW) {
    if (threadIdx.x == 0) {
      for (int i = 0; i < G * NSTG; ++i) mbar_init(smem_u32(&wbar[i]), 1);
      fence_barrier_init();
    }
    __syncthreads();
  }
  const int warp = tid >> 5, lane = tid & 31;
  const int rb = warp / CB, cb = warp % CB;
  const int r = lane >> 3, c = lane & 7;
  const int m0 = blockIdx.x * BM, n0 = blockIdx.y * BN;
  constexpr int kCPS = kSlice / kTBK;        // chunks per slice
  constexpr bool kBf16 = sizeof(XT) == 2;
  // first k of the group's local chunk lc
  auto chunk_k0 = [&](int lc) { return ((lc / kCPS) * G + grp) * kSlice + (lc % kCPS) * kTBK; };

  // global -> shared copy of the group's local chunk lc (16-byte pieces;
  // rows past M / N read a clamped valid row and are never stored); bf16 x
  // goes through registers (xload / xstore) instead
  auto load_chunk = [&](int lc, int stage) {
    const int k0 = chunk_k0(lc);
    constexpr int XPC = kBf16 ? 0 : kTBK / 4, WPC = TW ? 0 : kTBK / 4;  // pieces per row
    float *xst = xs + stage * (BM * XLd);
    if (TW && tid == 0) {
      const uint32_t bar = smem_u32(&wbar[grp * NSTG + stage]);
      mbar_arrive_expect_tx(bar, static_cast<uint32_t>(WS * 4));
      tma_load_2d(smem_u32(ws + stage * WS), &tmW, bar, k0, n0);
    }
    for (int q = tid; q < BM * XPC + BN * WPC; q += GT) {
      if (q < BM * XPC) {
        constexpr int XPCd = XPC > 0 ? XPC : 1;  // (bf16 x never gets here)
        const int row = q / XPCd, piece = q % XPCd;
        const int gm = min(m0 + row, M - 1);
        cp_async16(smem_u32(xst + row * XLd + piece * 4),
                   reinterpret_cast<const float *>(x) + static_cast<size_t>(gm) * K + k0 + piece * 4);
      } else {
        constexpr int WPCd = WPC > 0 ? WPC : 1;  // (TW never gets here)
        const int wr = (q - BM * XPC) / WPCd, piece = (q - BM * XPC) % WPCd;
        const int gn = min(n0 + wr, N - 1);
        cp_async16(smem_u32(ws + stage * WS + wr * WLd + piece * 4),
                   w + static_cast<size_t>(gn) * K + k0 + piece * 4);
      }
    }
  };
  constexpr int XPT = kBf16 ? (BM * 4 + GT - 1) / GT : 1;  // 16-byte bf16 pieces per thread
  uint4 xreg[XPT];
  auto xload = [&](int lc) {  // bf16 x of chunk lc into registers
    const int k0 = chunk_k0(lc);
#pragma unroll
    for (int t = 0; t < XPT; ++t) {
      const int q = tid + t * GT;
      if (q < BM * 4) {
        const int gm = min(m0 + q / 4, M - 1);
        xreg[t] = __ldg(reinterpret_cast<const uint4 *>(x + static_cast<size_t>(gm) * K + k0 + (q % 4) * 8));
      }
    }
  };
  auto xstore = [&](int stage) {  // ... widened to fp32 into the stage
    float *xst = xs + stage * (BM * XLd);
#pragma unroll
    for (int t = 0; t < XPT; ++t) {
      const int q = tid + t * GT;
      if (q < BM * 4) {
        const uint4 u = xreg[t];
        float4 *d = reinterpret_cast<float4 *>(xst + (q / 4) * XLd + (q % 4) * 8);
        d[0] = make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                           __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
        d[1] = make_float4(__uint_as_float(u.z << 16), __uint_as_float(u.z & 0xffff0000u),
                           __uint_as_float(u.w << 16), __uint_as_float(u.w & 0xffff0000u));
      }
    }
  };

  float p[TMR][TN], acc[TMR][TN];
#pragma unroll
  for (int i = 0; i < TMR; ++i)
#pragma unroll
    for (int j = 0; j < TN; ++j) {
      p[i][j] = 0.0f;
      acc[i][j] = 0.0f;
    }

  const int nchunks = K / kTBK / G;  // per group (G divides the slice count)
#pragma unroll
  for (int s = 0; s < NSTG - 1; ++s) {
    if (s < nchunks) {
      load_chunk(s, s);
      if (kBf16) {
        xload(s);
        xstore(s);
      }
    }
    cp_async_commit();
  }
  const int xrow0 = rb * 4 * TMR + r;  // + 4i
  const int wrow0 = cb * 8 * TN + c;   // + 8j
  for (int ch = 0; ch < nchunks; ++ch) {
    cp_async_wait<NSTG - 2>();
    __syncthreads();
    const int nx = ch + NSTG - 1;  // the chunk staged during this one
    if (nx < nchunks) {
      load_chunk(nx, nx % NSTG);
      if (kBf16) xload(nx);  // lands in registers while this chunk computes
    }
    cp_async_commit();
    const float *xb = xs + (ch % NSTG) * (BM * XLd);
    const float *wb = ws + (ch % NSTG) * WS;
    // TW: the chunk's W copy (a wait that times out records
    // BI_DEVERR_WAIT_TIMEOUT; the kernel goes on, its outputs undefined)
    if (TW) mbar_wait(smem_u32(&wbar[grp * NSTG + ch % NSTG]), static_cast<uint32_t>((ch / NSTG) & 1), nullptr, err);
#pragma unroll
    for (int kk = 0; kk < kTBK; kk += 4) {
      float4 xv[TMR], wv[TN];
#pragma unroll
      for (int i = 0; i < TMR; ++i)
        xv[i] = ld_x4(xb + (xrow0 + 4 * i) * XLd + kk);
#pragma unroll
      for (int j = 0; j < TN; ++j)
        // TW: 16-byte chunk kk/4 of row r sits at chunk (kk/4) ^ (r % 8), and
        // r % 8 = wrow0 % 8 for every j
        wv[j] = *reinterpret_cast<const float4 *>(wb + (wrow0 + 8 * j) * WLd +
                                                  (TW ? (((kk >> 2) ^ (wrow0 & 7)) << 2) : kk));
#pragma unroll
      for (int i = 0; i < TMR; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) {
          p[i][j] = __fmaf_rn(xv[i].x, wv[j].x, p[i][j]);
          p[i][j] = __fmaf_rn(xv[i].y, wv[j].y, p[i][j]);
          p[i][j] = __fmaf_rn(xv[i].z, wv[j].z, p[i][j]);
          p[i][j] = __fmaf_rn(xv[i].w, wv[j].w, p[i][j]);
        }
    }
    // the stage of chunk nx held chunk ch - 1, which every thread finished
    // before this iteration's barrier
    if (kBf16 && nx < nchunks) xstore(nx % NSTG);
    if ((ch + 1) % kCPS == 0) {
      // end of a round of G slices: the slice partials join the running sum
      // in slice order (group 0's slice first, then group 1's, ...)
      if (G > 1) {
        if (grp > 0) {
#pragma unroll
          for (int i = 0; i < TMR; ++i)
#pragma unroll
            for (int j = 0; j < TN; ++j) pb[((grp - 1) * TMR * TN + i * TN + j) * GT + tid] = p[i][j];
        }
        __syncthreads();
      }
      if (grp == 0) {
#pragma unroll
        for (int i = 0; i < TMR; ++i)
#pragma unroll
          for (int j = 0; j < TN; ++j) {
            float a = __fadd_rn(acc[i][j], p[i][j]);
#pragma unroll
            for (int g2 = 1; g2 < G; ++g2) a = __fadd_rn(a, pb[((g2 - 1) * TMR * TN + i * TN + j) * GT + tid]);
            acc[i][j] = a;
          }
      }
#pragma unroll
      for (int i = 0; i < TMR; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) p[i][j] = 0.0f;
    }
  }
  cp_async_wait<0>();
  if (grp != 0) return;

#pragma unroll
  for (int i = 0; i < TMR; ++i) {
    const int m = m0 + xrow0 + 4 * i;
    if (m >= M) continue;
#pragma unroll
    for (int j = 0; j < TN; ++j) {
      const int n = n0 + wrow0 + 8 * j;
      if (n >= N) continue;
      float v = acc[i][j];
      if (bias) v = __fadd_rn(v, bias[n]);
      y[static_cast<size_t>(m) * N + n] = v;
    }
  }
}

template <int TMR, int TN, int RB, int CB, int G, int NSTG, typename XT, bool TW = false>
static bi_status launch_tiled_t(const XT *x, const float *w, const float *b, float *y, int64_t M,
                                int64_t K, int64_t N, cudaStream_t stream) {
  using Cf = TiledCfg<TMR, TN, RB, CB, G, NSTG, XT, TW>;
  static_assert(Cf::kSmem <= 227 * 1024, "shared memory");
  static ContextSetup attr_done;  // the shared-memory attribute is per context
  int dev = 0;
  cudaGetDevice(&dev);
  if (attr_done.pending(dev)) {
    if (cudaFuncSetAttribute(router_tiled_kernel<TMR, TN, RB, CB, G, NSTG, XT, TW>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(Cf::kSmem)) !=
        cudaSuccess) {
      cudaGetLastError();  // do not leave the error for an unrelated later check
      set_error("router tiled: cannot reserve %zu bytes of shared memory", Cf::kSmem);
      return BI_ERR_CUDA;
    }
    attr_done.done(dev);
  }
  dim3 grid(static_cast<unsigned>((M + Cf::BM - 1) / Cf::BM), static_cast<unsigned>((N + Cf::BN - 1) / Cf::BN));
  CUtensorMap tmW;
  memset(&tmW, 0, sizeof(tmW));
  if (TW && !make_tma_2d_f32(&tmW, w, static_cast<uint64_t>(N), static_cast<uint64_t>(K), Cf::BN))
    return BI_ERR_CUDA;
  return launch_chained(router_tiled_kernel<TMR, TN, RB, CB, G, NSTG, XT, TW>, grid, dim3(Cf::GT * G), Cf::kSmem,
                        stream, 1, tmW, x, w, b, y, (int)M, (int)K, (int)N, device_error_word());
}

// The classic shapes: 8 warps per group, 4 columns per thread, 3 stages.
template <int TMR, int CB, int G, typename XT>
static bi_status launch_tiled4(const XT *x, const float *w, const float *b, float *y, int64_t M,
                               int64_t K, int64_t N, cudaStream_t stream) {
  return launch_tiled_t<TMR, 4, 8 / CB, CB, G, 3, XT>(x, w, b, y, M, K, N, stream);
}

// Wide lane tiles (7 rows x 8 columns per thread): groups of 4 warps over 256
// columns with two slice groups, or of 2 warps over 128 columns with four;
// either way 28-row CTA tiles of 256 threads (147 CTAs at M = 4096).  A CTA
// runs its whole K loop in about the same time at any M (255 registers, two
// warps per scheduler), so the schedule pays once the 28-row tiles cover
// most SMs: measured on GB300 at M = 4096, 62.5 vs 75.0 us (K=2048, N=128,
// bf16 x) and 226.5 vs 233.8 us (K=4096, N=256) against the 7x4 tiles.
static bool wide_ok(int64_t K, int64_t N) {
  const int64_t S = K / kSlice;
  return N <= 128 ? S % 4 == 0 : S % 2 == 0;
}

template <typename XT>
static bi_status launch_tiled_wide(const XT *x, const float *w, const float *b, float *y, int64_t M,
                                   int64_t K, int64_t N, cudaStream_t stream) {
  const int64_t S = K / kSlice;
  if (N <= 128) {
    if (S % 4 != 0) {
      set_error("router wide tiles: K/128 = %lld slices do not split over 4 groups", (long long)S);
      return BI_ERR_UNSUPPORTED;
    }
    return launch_tiled_t<7, 8, 1, 2, 4, 2, XT>(x, w, b, y, M, K, N, stream);
  }
  if (S % 2 != 0) {
    set_error("router wide tiles: K/128 = %lld slices do not split over 2 groups", (long long)S);
    return BI_ERR_UNSUPPORTED;
  }
  // 256 columns: W chunks by TMA (measured on GB300, DSv4-shaped router at
  // M=4096: 217.6 vs 224.7 us with bf16 x, 211.1 vs 225.3 us with fp32 x;
  // for the 128-column tiles above the cp.async ring stays, 60.9 vs 62.3 us)
  return launch_tiled_t<7, 8, 1, 4, 2, 2, XT, true>(x, w, b, y, M, K, N, stream);
}

// Tile shape for the tiled schedule: the (column blocks, rows per thread)
// pair with the smallest per-SM load ceil(CTAs / SMs) * TMR, taking the first
// of a preference list on ties (measured on GB300: a full-width 7-row tile
// for the widest batches, 128-column tiles with fewer rows otherwise).
template <typename XT>
static bi_status launch_tiled(const XT *x, const float *w, const float *b, float *y, int64_t M,
                              int64_t K, int64_t N, cudaStream_t stream) {
  struct Shape { int cb, tmr; };
  static const Shape wide[] = {{8, 7}, {8, 8}, {4, 4}, {4, 3}, {4, 2}, {4, 1}};
  static const Shape narrow[] = {{4, 4}, {4, 3}, {4, 2}, {4, 1}};
  const bool is_wide = N > 128;
  const Shape *list = is_wide ? wide : narrow;
  const int nlist = is_wide ? 6 : 4;
  const int sms = num_sms();
  Shape pick = list[0];
  int64_t best = INT64_MAX;
  for (int i = 0; i < nlist; ++i) {
    const Shape sh = list[i];
    const int bm = (8 / sh.cb) * 4 * sh.tmr, bn = sh.cb * 32;
    const int64_t ctas = ((M + bm - 1) / bm) * ((N + bn - 1) / bn);
    const int64_t cost = ((ctas + sms - 1) / sms) * sh.tmr;
    if (cost < best) {
      best = cost;
      pick = sh;
    }
  }
  // Two slice groups per CTA (512 threads) when the tile is small enough
  // (<= 4 rows per thread) and leaves SMs idle: the groups share the tile's
  // output rows and columns and split its slices, so the grid has twice the
  // warps for the same CTA count (measured: 4-6 % faster on the
  // K=2048/N=128 router at M >= 1024 and on K=4096/N=256 at M=1024).
  {
    const int bm = (8 / pick.cb) * 4 * pick.tmr, bn = pick.cb * 32;
    const int64_t ctas = ((M + bm - 1) / bm) * ((N + bn - 1) / bn);
    if (pick.tmr <= 4 && ctas < sms && (K / kSlice) % 2 == 0) {
      switch (pick.cb * 16 + pick.tmr) {
        case 4 * 16 + 4: return launch_tiled4<4, 4, 2, XT>(x, w, b, y, M, K, N, stream);
        case 4 * 16 + 3: return launch_tiled4<3, 4, 2, XT>(x, w, b, y, M, K, N, stream);
        case 4 * 16 + 2: return launch_tiled4<2, 4, 2, XT>(x, w, b, y, M, K, N, stream);
        default: return launch_tiled4<1, 4, 2, XT>(x, w, b, y, M, K, N, stream);
      }
    }
  }
  switch (pick.cb * 16 + pick.tmr) {
    case 8 * 16 + 7: return launch_tiled4<7, 8, 1, XT>(x, w, b, y, M, K, N, stream);
    case 8 * 16 + 8: return launch_tiled4<8, 8, 1, XT>(x, w, b, y, M, K, N, stream);
    case 4 * 16 + 4: return launch_tiled4<4, 4, 1, XT>(x, w, b, y, M, K, N, stream);
    case 4 * 16 + 3: return launch_tiled4<3, 4, 1, XT>(x, w, b, y, M, K, N, stream);
    case 4 * 16 + 2: return launch_tiled4<2, 4, 1, XT>(x, w, b, y, M, K, N, stream);
    default: return launch_tiled4<1, 4, 1, XT>(x, w, b, y, M, K, N, stream);
  }
}

// ------------------------------------------------------------------- split --
// Slice-parallel kernel for small and medium M.  The S slices of every output
// are spread over a cluster of C = S / L CTAs of L warps, one slice per warp,
// so a batch of a few rows still keeps most SMs busy and each warp's lane
// tile can be as large as the batch allows.  Warp w of cluster rank r
// evaluates slice s = rL + w for the CTA's whole BM x BN block: lane (a, b)
// owns rows a + 4i (i < TM) and columns b + 8j (j < TN).  The warp streams its
// slice of x and W through a warp-private ring of NST chunks of CK k
// (cp.async, 16-byte pieces, rows padded by 16 bytes so lanes reading
// different rows at one k hit different banks), so no warp waits for another.  After the chain the warp parks its slice partials in
// its own shared memory; a cluster barrier; then each CTA takes 1/C of the
// block's outputs and sums, for each, the S partials in slice order (rank r's
// shared memory holds slices rL .. rL+L-1), then adds the bias.  The sum order
// is the recipe's; only the placement of the chains differs.
constexpr int kSpLM = 4, kSpLN = 8;  // lanes along rows x lanes along columns
constexpr int kSpMaxC = 8;           // portable cluster size

template <int TM, int TN, int NST, typename XT, int CK>
struct SplitCfg {
  static constexpr int BM = kSpLM * TM, BN = kSpLN * TN;
  static constexpr int XLd = CK + 16 / static_cast<int>(sizeof(XT));  // x row pitch (elements)
  static constexpr int WLd = CK + 4;                                  // W row pitch (floats)
  static constexpr int XB = BM * XLd * static_cast<int>(sizeof(XT));  // bytes of one x chunk
  static constexpr int WB = BN * WLd * 4;                             // bytes of one W chunk
  static constexpr int WARP_BYTES = NST * (XB + WB);                  // one warp's ring
  static_assert(BM * BN * 4 <= WARP_BYTES, "a warp's partials must fit in its ring");
};

__device__ __forceinline__ float ld_dsmem_f32(uint32_t cluster_addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(cluster_addr));
  return v;
}

template <int TM, int TN, int NST, int L, typename XT, int CK, bool ROLL = false>
__global__ void __launch_bounds__(32 * L) router_split_kernel(const XT *__restrict__ x,
                                                              const float *__restrict__ w,
                                                              const float *__restrict__ bias,
                                                              float *__restrict__ y, int M, int K,
                                                              int N, unsigned *zero_words, int n_zero) {
  using Cf = SplitCfg<TM, TN, NST, XT, CK>;
  constexpr int BM = Cf::BM, BN = Cf::BN, XLd = Cf::XLd, WLd = Cf::WLd;
  constexpr int kChunks = kSlice / CK;
  extern __shared__ __align__(16) uint8_t sp_smem[];

  griddep_wait();
  if (zero_words && blockIdx.x == 0 && blockIdx.y == 0)
    for (int i = threadIdx.x; i < n_zero; i += 32 * L) zero_words[i] = 0u;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int C = K / kSlice / L;  // CTAs per cluster (the launch's cluster size)
  const int rank = static_cast<int>(cluster_ctarank());
  const int n0 = (blockIdx.x / C) * BN, m0 = blockIdx.y * BM;
  const int s = rank * L + warp;  // this warp's slice
  uint8_t *mine = sp_smem + warp * Cf::WARP_BYTES;
  XT *xr = reinterpret_cast<XT *>(mine);                   // [NST][BM][XLd]
  float *wr = reinterpret_cast<float *>(mine + NST * Cf::XB);  // [NST][BN][WLd]

  // chunk q (k = 128 s + CK q ...) of the warp's x rows and W rows into stage st
  auto load = [&](int q, int st) {
    const int k0 = s * kSlice + q * CK;
    constexpr int XE = 16 / static_cast<int>(sizeof(XT));  // x elements per piece
    constexpr int XPC = CK / XE, WPC = CK / 4;             // pieces per row
    static_assert((BM * XPC) % 32 == 0 && (BN * WPC) % 32 == 0, "whole warps of pieces");
#pragma unroll
    for (int t = 0; t < BM * XPC / 32; ++t) {
      const int i = lane + 32 * t, row = i / XPC, pc = i % XPC;
      const int gm = min(m0 + row, M - 1);
      cp_async16(smem_u32(xr + (st * BM + row) * XLd + pc * XE),
                 x + static_cast<size_t>(gm) * K + k0 + pc * XE);
    }
#pragma unroll
    for (int t = 0; t < BN * WPC / 32; ++t) {
      const int i = lane + 32 * t, row = i / WPC, pc = i % WPC;
      const int gn = min(n0 + row, N - 1);
      cp_async16(smem_u32(wr + (st * BN + row) * WLd + pc * 4),
                 w + static_cast<size_t>(gn) * K + k0 + pc * 4);
    }
  };

  float p[TM][TN];
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int j = 0; j < TN; ++j) p[i][j] = 0.0f;

#pragma unroll
  for (int q = 0; q < NST - 1; ++q) {
    if (q < kChunks) load(q, q);
    cp_async_commit();
  }
  const int a = lane / kSpLN, b = lane % kSpLN;
  // ROLL: a runtime loop over the slice's chunks.  Unrolled, the slice is
  // several thousand instructions of straight-line code that each warp runs
  // once, and instruction fetch becomes the main stall once the warps' FMA
  // work is long enough (measured on GB300, K=4096/N=256: 8-20 % faster for
  // bf16 x at M >= 128, for fp32 x at M >= 1024; 1-7 % slower below)
#pragma unroll(ROLL ? 1 : kChunks)
  for (int q = 0; q < kChunks; ++q) {
    cp_async_wait<NST - 2>();
    __syncwarp();  // every lane's pieces of chunk q landed; stage of q-1 free
    if (q + NST - 1 < kChunks) load(q + NST - 1, (q + NST - 1) % NST);
    cp_async_commit();
    const XT *xb = xr + (q % NST) * BM * XLd;
    const float *wb = wr + (q % NST) * BN * WLd;
#pragma unroll
    for (int kk = 0; kk < CK; kk += 4) {
      float4 xv[TM], wv[TN];
#pragma unroll
      for (int i = 0; i < TM; ++i) xv[i] = ld_x4(xb + (a + kSpLM * i) * XLd + kk);
#pragma unroll
      for (int j = 0; j < TN; ++j)
        wv[j] = *reinterpret_cast<const float4 *>(wb + (b + kSpLN * j) * WLd + kk);
#pragma unroll
      for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) {
          p[i][j] = __fmaf_rn(xv[i].x, wv[j].x, p[i][j]);
          p[i][j] = __fmaf_rn(xv[i].y, wv[j].y, p[i][j]);
          p[i][j] = __fmaf_rn(xv[i].z, wv[j].z, p[i][j]);
          p[i][j] = __fmaf_rn(xv[i].w, wv[j].w, p[i][j]);
        }
    }
  }
  cp_async_wait<0>();
  __syncwarp();  // the ring is read out: the warp's partials go over it
  float *part = reinterpret_cast<float *>(mine);  // [BM][BN]
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int j = 0; j < TN; ++j) part[(a + kSpLM * i) * BN + b + kSpLN * j] = p[i][j];

  cluster_sync_all();  // every slice partial of the block is in place

  // this CTA's share of the block's outputs, each summed over all S slices
  constexpr int E = BM * BN;
  const int per = (E + C - 1) / C;
  const int e_end = min(E, (rank + 1) * per);
  const uint32_t base = smem_u32(sp_smem);
  for (int e = rank * per + static_cast<int>(threadIdx.x); e < e_end; e += 32 * L) {
    float v[kSpMaxC][L];
#pragma unroll
    for (int r = 0; r < kSpMaxC; ++r) {
      if (r < C) {
        const uint32_t rb = mapa_shared(base, static_cast<uint32_t>(r)) + static_cast<uint32_t>(e) * 4u;
#pragma unroll
        for (int l = 0; l < L; ++l) v[r][l] = ld_dsmem_f32(rb + static_cast<uint32_t>(l * Cf::WARP_BYTES));
      }
    }
    float acc = 0.0f;
#pragma unroll
    for (int r = 0; r < kSpMaxC; ++r) {
      if (r < C) {
#pragma unroll
        for (int l = 0; l < L; ++l) acc = __fadd_rn(acc, v[r][l]);
      }
    }
    const int m = m0 + e / BN, n = n0 + e % BN;
    if (m < M && n < N) {
      if (bias) acc = __fadd_rn(acc, bias[n]);
      y[static_cast<size_t>(m) * N + n] = acc;
    }
  }
  cluster_sync_all();  // no CTA leaves while a peer still reads its partials
}

template <int TM, int TN, int NST, int CK, int L, typename XT, bool ROLL>
static bi_status launch_split_t(const XT *x, const float *w, const float *b, float *y, int64_t M,
                                int64_t K, int64_t N, cudaStream_t stream, unsigned *zw, int nz) {
  using Cf = SplitCfg<TM, TN, NST, XT, CK>;
  const int C = static_cast<int>(K / kSlice) / L;
  const size_t smem = static_cast<size_t>(L) * Cf::WARP_BYTES;
  static ContextSetup attr_done;  // the shared-memory attribute is per context
  int dev = 0;
  cudaGetDevice(&dev);
  if (attr_done.pending(dev)) {
    if (cudaFuncSetAttribute(router_split_kernel<TM, TN, NST, L, XT, CK, ROLL>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
        cudaSuccess) {
      cudaGetLastError();
      set_error("router split: cannot reserve %zu bytes of shared memory", smem);
      return BI_ERR_CUDA;
    }
    attr_done.done(dev);
  }
  dim3 grid(static_cast<unsigned>(C * ((N + Cf::BN - 1) / Cf::BN)),
            static_cast<unsigned>((M + Cf::BM - 1) / Cf::BM));
  return launch_chained(router_split_kernel<TM, TN, NST, L, XT, CK, ROLL>, grid, dim3(32 * L), smem, stream, C,
                        x, w, b, y, (int)M, (int)K, (int)N, zw, nz);
}

// Lane tiles of the split schedule (outputs per thread TM x TN, ring depth,
// k per chunk).  The 8x4 tile streams 16-k chunks: 40 KB per CTA instead of
// 74, so four of its CTAs share an SM (register-limited) instead of three.
struct SplitTile { int tm, tn, nst, ck; };
constexpr SplitTile kSplitTiles[] = {{2, 2, 4, 32}, {4, 2, 4, 32}, {4, 4, 3, 32}, {8, 4, 2, 16}};
constexpr int kNumSplitTiles = 4;

// Warps per CTA for the split schedule (slices per CTA), 0 if the slice count
// does not split into 2..8 CTAs of 4 or 8 warps.
static int split_warps(int64_t K) {
  const int64_t S = K / kSlice;
  if (S % 4 == 0 && S / 4 >= 2 && S / 4 <= kSpMaxC) return 4;
  if (S % 8 == 0 && S / 8 >= 2 && S / 8 <= kSpMaxC) return 8;
  return 0;
}

// Tile for M: the largest lane tile that still gives at least 1.5 CTAs per
// SM, else the smallest.  A CTA of few warps is latency-bound, so spreading
// the work over more CTAs beats the better load/FMA ratio of a larger tile
// until the SMs are covered (measured on GB300 for K=4096/N=256 and
// K=2048/N=128, M = 1 .. 1024).
static int split_pick(int64_t M, int64_t N, int C) {
  const int64_t want = 3 * static_cast<int64_t>(num_sms()) / 2;
  for (int t = kNumSplitTiles - 1; t > 0; --t) {
    const int64_t bm = kSpLM * kSplitTiles[t].tm, bn = kSpLN * kSplitTiles[t].tn;
    if (C * ((N + bn - 1) / bn) * ((M + bm - 1) / bm) >= want) return t;
  }
  return 0;
}

template <int L, typename XT, bool ROLL>
static bi_status launch_split_r(const XT *x, const float *w, const float *b, float *y, int64_t M,
                                int64_t K, int64_t N, int tile, cudaStream_t stream, unsigned *zw, int nz) {
  switch (tile) {
    case 0: return launch_split_t<2, 2, 4, 32, L, XT, ROLL>(x, w, b, y, M, K, N, stream, zw, nz);
    case 1: return launch_split_t<4, 2, 4, 32, L, XT, ROLL>(x, w, b, y, M, K, N, stream, zw, nz);
    case 2: return launch_split_t<4, 4, 3, 32, L, XT, ROLL>(x, w, b, y, M, K, N, stream, zw, nz);
    default: return launch_split_t<8, 4, 2, 16, L, XT, ROLL>(x, w, b, y, M, K, N, stream, zw, nz);
  }
}

// The chunk loop rolled where that measured faster (see router_split_kernel).
template <int L, typename XT>
static bi_status launch_split_l(const XT *x, const float *w, const float *b, float *y, int64_t M,
                                int64_t K, int64_t N, int tile, cudaStream_t stream, unsigned *zw, int nz) {
  const bool roll = M >= (sizeof(XT) == 2 ? 128 : 1024);
  return roll ? launch_split_r<L, XT, true>(x, w, b, y, M, K, N, tile, stream, zw, nz)
              : launch_split_r<L, XT, false>(x, w, b, y, M, K, N, tile, stream, zw, nz);
}

// tile < 0: chosen from M.  Needs split_warps(K) != 0.
template <typename XT>
static bi_status launch_split(const XT *x, const float *w, const float *b, float *y, int64_t M,
                              int64_t K, int64_t N, int tile, cudaStream_t stream, unsigned *zw, int nz) {
  const int L = split_warps(K);
  const int C = static_cast<int>(K / kSlice) / L;
  if (tile < 0) tile = split_pick(M, N, C);
  return L == 4 ? launch_split_l<4, XT>(x, w, b, y, M, K, N, tile, stream, zw, nz)
                : launch_split_l<8, XT>(x, w, b, y, M, K, N, tile, stream, zw, nz);
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
  griddep_wait();
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
// zero_words (optional): n_zero words that the launched kernel sets to 0
// after its predecessors on the stream have finished (the rows, split and
// sliced schedules; the decode layer's one-launch expert path counts arrivals
// on them).
template <typename XT>
static bi_status launch_router_t(const XT *x, const float *w, const float *b, float *y, int64_t M,
                                 int64_t K, int64_t N, int schedule, cudaStream_t stream,
                                 unsigned *zero_words, int n_zero) {
  const int S = static_cast<int>(K / kSlice);
  // automatic: rows for one or two tokens, the cluster split up to ~3K rows,
  // the tiled kernel beyond (measured crossover on GB300: the split is 27 %
  // faster at M=2048 for K=2048/N=128 and level for K=4096/N=256; the tiled
  // kernel is level or faster at M=4096)
  if (schedule == 0) {
    if (M <= 2) schedule = 1;
    else if (M < 3072 && split_warps(K)) schedule = 4;
    else if (M < 384) schedule = (M <= 4) ? 1 : 2;
    else schedule = (wide_ok(K, N) && (M + 27) / 28 >= 7 * num_sms() / 10) ? 9 : 3;
  }
  if (schedule >= 4 && schedule <= 4 + kNumSplitTiles) {  // 4 auto tile, 5.. forced
    if (!split_warps(K)) {
      set_error("router split schedule: K=%lld does not split into 2..8 CTAs of 4 or 8 slices",
                (long long)K);
      return BI_ERR_UNSUPPORTED;
    }
    if ((M + 7) / 8 > 65535) {
      set_error("router split schedule: M=%lld too large for it", (long long)M);
      return BI_ERR_UNSUPPORTED;
    }
    const bi_status st = launch_split(x, w, b, y, M, K, N, schedule - 5, stream, zero_words, n_zero);
    if (st != BI_OK) return st;
  } else if (schedule == 1) {
    const int mr = M <= 1 ? 1 : (M <= 2 ? 2 : 4);
    dim3 grid(static_cast<unsigned>(N), static_cast<unsigned>((M + mr - 1) / mr));
    const size_t smem = static_cast<size_t>(32) * kSlicePad * sizeof(float) +
                        static_cast<size_t>(mr) * 32 * XPitch<XT>::slice * sizeof(XT) +
                        static_cast<size_t>(mr) * S * sizeof(float);
    if (grid.y > 65535u) {
      set_error("router rows schedule: M=%lld too large for it", (long long)M);
      return BI_ERR_UNSUPPORTED;
    }
#define BI_ROWS(R)                                                                                     \
  {                                                                                                    \
    static ContextSetup attr;                                                                          \
    int dv = 0;                                                                                        \
    cudaGetDevice(&dv);                                                                                \
    if (attr.pending(dv)) {                                                                            \
      cudaFuncSetAttribute(router_rows_kernel<R, XT>, cudaFuncAttributeMaxDynamicSharedMemorySize, 100000); \
      attr.done(dv);                                                                                   \
    }                                                                                                  \
    const bi_status st_ = launch_chained(router_rows_kernel<R, XT>, grid, dim3(32), smem, stream, 1, x, w, \
                                         b, y, (int)M, (int)K, (int)N, device_error_word(), zero_words, n_zero); \
    if (st_ != BI_OK) return st_;                                                                    \
  }
    if (mr == 1) BI_ROWS(1) else if (mr == 2) BI_ROWS(2) else BI_ROWS(4)
#undef BI_ROWS
  } else if (schedule == 2) {
    dim3 grid(static_cast<unsigned>((N + kSlNT - 1) / kSlNT), static_cast<unsigned>((M + kSlMT - 1) / kSlMT));
    const size_t smem = 2 * static_cast<size_t>(sl_stage_bytes<XT>()) + kSlG * kSlMT * kSlNT * sizeof(float);
    if (grid.y > 65535u) {
      set_error("router sliced schedule: M=%lld too large for it", (long long)M);
      return BI_ERR_UNSUPPORTED;
    }
    static ContextSetup attr;
    int dv = 0;
    cudaGetDevice(&dv);
    if (attr.pending(dv)) {
      cudaFuncSetAttribute(router_sliced_kernel<XT>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
      attr.done(dv);
    }
    const bi_status st = launch_chained(router_sliced_kernel<XT>, grid, dim3(256), smem, stream, 1, x, w, b,
                                        y, (int)M, (int)K, (int)N, device_error_word(), zero_words, n_zero);
    if (st != BI_OK) return st;
  } else if (zero_words) {
    set_error("router schedule %d cannot zero words", schedule);
    return BI_ERR_UNSUPPORTED;
  } else if (schedule == 9) {
    if ((M + 27) / 28 > 2147483647LL) {
      set_error("router wide schedule: M=%lld too large for it", (long long)M);
      return BI_ERR_UNSUPPORTED;
    }
    const bi_status st = launch_tiled_wide(x, w, b, y, M, K, N, stream);
    if (st != BI_OK) return st;
  } else if (schedule == 3) {
    if ((M + 3) / 4 > 65535LL * 8 * 4) {
      set_error("router tiled schedule: M=%lld too large for it", (long long)M);
      return BI_ERR_UNSUPPORTED;
    }
    const bi_status st = launch_tiled(x, w, b, y, M, K, N, stream);
    if (st != BI_OK) return st;
  } else {
    set_error("unknown router schedule %d", schedule);
    return BI_ERR_INVALID_ARG;
  }
  BI_CHECK_LAUNCH();
  return BI_OK;
}

bi_status launch_router(const float *x, const float *w, const float *b, float *y, int64_t M,
                        int64_t K, int64_t N, int schedule, cudaStream_t stream) {
  return launch_router_t<float>(x, w, b, y, M, K, N, schedule, stream, nullptr, 0);
}

// The same router on bf16 x (converted exactly to fp32 as it is read).
bi_status launch_router_bf16(const void *x, const float *w, const float *b, float *y, int64_t M,
                             int64_t K, int64_t N, int schedule, cudaStream_t stream, unsigned *zero_words,
                             int n_zero) {
  return launch_router_t<__nv_bfloat16>(static_cast<const __nv_bfloat16 *>(x), w, b, y, M, K, N,
                                        schedule, stream, zero_words, n_zero);
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
  return launch_chained(cast_bf16_f32_kernel, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0,
                        stream, 1, static_cast<const __nv_bfloat16 *>(x), y, n);
}

}  // namespace bimoe
