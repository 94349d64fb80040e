// moe_gemm.cu -- grouped expert GEMMs on 5th-generation tensor cores.
//
// Source: "Batch-invariance generation with vLLM fused-MoE backend at
// improved performance", section "What's included": the expert GEMMs pin the
// K-reduction recipe (a fixed K step, fp32 accumulation, no split-K); tiling
// along M/N does not touch the bits.  The activation applies the routing
// probability with fp32 math and one bf16 round (the strict-review summary:
// gate|up half split, single final bf16 round).
//
// Design (sm_103a):
//   * swap-AB: the weight rows are the MMA "M" side (128 rows of one expert),
//     the tokens routed to that expert are the "N" side (128 per tile), K runs
//     over the hidden (gate/up) or intermediate (down) dimension.
//   * one instruction shape for every M: tcgen05.mma.cta_group::1.kind::f16,
//     M=128, N=128, K=16, bf16 operands, fp32 accumulator in tensor memory.
//     K advances in steps of 64 (one 128-byte swizzle atom: four MMAs) in
//     increasing k, always accumulating into the same tensor-memory tile,
//     with no split-K: each output element sees the same instruction sequence
//     whatever the batch is.
//   * TMA (cp.async.bulk.tensor, 128-byte swizzle) stages weight and token
//     tiles through a 4-6 deep shared-memory ring guarded by mbarriers.
//   * warp roles: warp 0 issues TMA, warp 1 owns tensor memory and issues the
//     MMAs from one thread, warps 2-5 drain the accumulator (tcgen05.ld) and
//     run the epilogue.  Accumulators are double-buffered in tensor memory so
//     the epilogue of one tile overlaps the MMAs of the next.
//   * persistent grid (at most one CTA per SM); tiles are ordered expert,
//     weight block, token block so the token blocks sharing a weight block run
//     back to back and read it from L2.
//   * gate/up: two accumulators per tile (gate rows j, up rows I+j); the
//     epilogue computes act = bf16(silu(g) * u * p) in fp32.
//   * down: one accumulator; the epilogue writes fp32 contributions to row
//     token*top_k + slot.
#include "bimoe_internal.cuh"

namespace bimoe {

constexpr int kBM = 128;                 // weight rows per tile (MMA M)
constexpr int kBN = 128;                 // tokens per tile (MMA N)
constexpr int kBK = 64;                  // K step per stage (one swizzle atom)
constexpr int kUK = 16;                  // K of one MMA
constexpr int kTileBytes = kBM * kBK * 2;  // one 128 x 64 bf16 operand tile
constexpr int kGemmThreads = 192;

template <bool GATE_UP>
struct GemmCfg {
  static constexpr int kNumA = GATE_UP ? 2 : 1;
  static constexpr int kStages = GATE_UP ? 4 : 6;
  static constexpr int kStageBytes = (kNumA + 1) * kTileBytes;
  static constexpr int kAccCols = GATE_UP ? 2 * kBN : kBN;  // per accumulator buffer
  static constexpr int kTmemCols = 2 * kAccCols;             // double buffered
  static constexpr int kAuxBytes = 8192;
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kAuxBytes;
};

struct GemmParams {
  const int32_t *offsets;  // [E+1] first permuted position of each expert
  const int32_t *perm;     // [P] pair id (token*top_k + slot) of each position
  const float *wts;        // [M*top_k] routing probabilities (gate/up only)
  void *out;               // gate/up: act bf16 [P, I]; down: contrib fp32 [M*top_k, H]
  int E;
  int K;                   // reduction length (H for gate/up, I for down)
  int n_wb;                // 128-row weight blocks per expert (I/128 or H/128)
  int out_ld;              // output row length (I or H)
  int a_rows_per_expert;   // rows of the weight tensor per expert (2I or H)
  int up_offset;           // row offset of the up half (I), gate/up only
  int *err;
};

struct TileInfo {
  int e, wb, tok0, ntok;
};

__device__ __forceinline__ TileInfo decode_tile(int tile, const int *tile_prefix,
                                                const GemmParams &p) {
  int lo = 0, hi = p.E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tile_prefix[mid] <= tile) lo = mid;
    else hi = mid - 1;
  }
  TileInfo t;
  t.e = lo;
  const int local = tile - tile_prefix[lo];
  const int beg = __ldg(p.offsets + lo);
  const int cnt = __ldg(p.offsets + lo + 1) - beg;
  const int ntt = (cnt + kBN - 1) / kBN;
  t.wb = local / ntt;
  const int tt = local - t.wb * ntt;
  t.tok0 = beg + tt * kBN;
  t.ntok = min(kBN, cnt - tt * kBN);
  return t;
}

template <bool GATE_UP>
__global__ void __launch_bounds__(kGemmThreads, 1)
    moe_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const GemmParams prm) {
  using C = GemmCfg<GATE_UP>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *tiles = smem;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kStages * C::kStageBytes);
  uint64_t *full = bars;
  uint64_t *empty = bars + C::kStages;
  uint64_t *tfull = bars + 2 * C::kStages;
  uint64_t *tempty = tfull + 2;
  uint64_t *drain = tempty + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  int *tile_prefix = reinterpret_cast<int *>(tmem_slot + 4);  // [E+1]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nkb = prm.K / kBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(&tfull[a]), 1);
      mbar_init(smem_u32(&tempty[a]), 128);
    }
    mbar_init(smem_u32(drain), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  if (warp == 2) {
    // tile_prefix[e] = tiles of experts < e; each lane scans a contiguous chunk
    const int per = (prm.E + 31) / 32;
    const int e0 = min(lane * per, prm.E), e1 = min(e0 + per, prm.E);
    int local = 0;
    for (int e = e0; e < e1; ++e) {
      const int cnt = __ldg(prm.offsets + e + 1) - __ldg(prm.offsets + e);
      local += prm.n_wb * ((cnt + kBN - 1) / kBN);
    }
    int incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += v;
    }
    int run = incl - local;
    for (int e = e0; e < e1; ++e) {
      tile_prefix[e] = run;
      const int cnt = __ldg(prm.offsets + e + 1) - __ldg(prm.offsets + e);
      run += prm.n_wb * ((cnt + kBN - 1) / kBN);
    }
    if (lane == 31) tile_prefix[prm.E] = incl;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total_tiles = tile_prefix[prm.E];

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_mask = 0, issued_parity = 0;
      for (int tile = blockIdx.x; tile < total_tiles && !*abort_flag; tile += gridDim.x) {
        const TileInfo ti = decode_tile(tile, tile_prefix, prm);
        const int a_row = ti.e * prm.a_rows_per_expert + ti.wb * kBM;
        bool ok = true;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(smem_u32(&empty[stage]), phase ^ 1u, abort_flag, prm.err)) {
            ok = false;
            break;
          }
          uint8_t *st = tiles + stage * C::kStageBytes;
          const uint32_t fb = smem_u32(&full[stage]);
          mbar_arrive_expect_tx(fb, C::kStageBytes);
          tma_load_2d(smem_u32(st), &tmA, fb, kb * kBK, a_row);
          if (GATE_UP) tma_load_2d(smem_u32(st + kTileBytes), &tmA, fb, kb * kBK, a_row + prm.up_offset);
          tma_load_2d(smem_u32(st + C::kNumA * kTileBytes), &tmB, fb, kb * kBK, ti.tok0);
          issued_mask |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
      }
      if (*abort_flag) {
        // let every copy this thread started land before the CTA can exit
        for (int s = 0; s < C::kStages; ++s)
          if ((issued_mask >> s) & 1u)
            mbar_wait(smem_u32(&full[s]), (issued_parity >> s) & 1u, nullptr, prm.err);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(kBM, kBN);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool issued_any = false;
      for (int tile = blockIdx.x; tile < total_tiles && !*abort_flag; tile += gridDim.x) {
        if (!mbar_wait(smem_u32(&tempty[acc]), acc_phase ^ 1u, abort_flag, prm.err)) break;
        tc_fence_after();
        const uint32_t d0 = tmem_base + static_cast<uint32_t>(acc * C::kAccCols);
        bool ok = true;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(smem_u32(&full[stage]), phase, abort_flag, prm.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(tiles + stage * C::kStageBytes);
          const uint32_t b0 = a0 + C::kNumA * kTileBytes;
#pragma unroll
          for (int k = 0; k < kBK / kUK; ++k) {
            const uint32_t acc_in = (kb | k) != 0 ? 1u : 0u;
            const uint64_t bdesc = sdesc_sw128(b0 + k * kUK * 2);
            umma_f16(d0, sdesc_sw128(a0 + k * kUK * 2), bdesc, idesc, acc_in);
            if (GATE_UP)
              umma_f16(d0 + kBN, sdesc_sw128(a0 + kTileBytes + k * kUK * 2), bdesc, idesc, acc_in);
          }
          issued_any = true;
          umma_commit(smem_u32(&empty[stage]));
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(smem_u32(&tfull[acc]));
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (*abort_flag && issued_any) {
        // wait for the MMAs in flight before tensor memory is released
        umma_commit(smem_u32(drain));
        mbar_wait(smem_u32(drain), 0, nullptr, prm.err);
      }
    }
    __syncwarp();
  } else {
    // --------------------------------------------------------- epilogue --
    const int q = warp & 3;        // tensor-memory lane quarter of this warp
    const int row = q * 32 + lane;  // weight row inside the tile
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
      const TileInfo ti = decode_tile(tile, tile_prefix, prm);
      if (!mbar_wait(smem_u32(&tfull[acc]), acc_phase, abort_flag, prm.err)) break;
      tc_fence_after();
      const uint32_t tbase =
          tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * C::kAccCols);
      const int col = ti.wb * kBM + row;
      for (int c0 = 0; c0 < ti.ntok; c0 += 32) {
        uint32_t d[32];
        tmem_ld32(tbase + c0, d);
        // per-token data: lane c holds token c0 + c, broadcast by shuffles
        const bool tv = c0 + lane < ti.ntok;
        const int my_pair = tv ? __ldg(prm.perm + ti.tok0 + c0 + lane) : 0;
        if (GATE_UP) {
          uint32_t u[32];
          tmem_ld32(tbase + kBN + c0, u);
          const float my_p = tv ? __ldg(prm.wts + my_pair) : 0.0f;
          tmem_ld_wait();
          __nv_bfloat16 *act = static_cast<__nv_bfloat16 *>(prm.out);
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const float pc = __shfl_sync(0xffffffffu, my_p, c);
            if (c0 + c < ti.ntok) {
              const float g = __uint_as_float(d[c]);
              const float uu = __uint_as_float(u[c]);
              const float sg = __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-g)));
              const float a = __fmul_rn(__fmul_rn(__fmul_rn(g, sg), uu), pc);
              act[static_cast<size_t>(ti.tok0 + c0 + c) * prm.out_ld + col] = __float2bfloat16_rn(a);
            }
          }
        } else {
          tmem_ld_wait();
          float *contrib = static_cast<float *>(prm.out);
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const int pair = __shfl_sync(0xffffffffu, my_pair, c);
            if (c0 + c < ti.ntok)
              contrib[static_cast<size_t>(pair) * prm.out_ld + col] = __uint_as_float(d[c]);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&tempty[acc]));
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

// ------------------------------------------------------------------- host --
template <bool GATE_UP>
static bi_status launch_gemm(const CUtensorMap &tmA, const CUtensorMap &tmB, const GemmParams &p,
                             int64_t P, cudaStream_t stream) {
  using C = GemmCfg<GATE_UP>;
  static bool attr_done[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(moe_gemm_kernel<GATE_UP>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) {
      set_error("cudaFuncSetAttribute: %s", cudaGetErrorString(e));
      return BI_ERR_CUDA;
    }
    attr_done[dev] = true;
  }
  // upper bound on the number of tiles (token blocks per expert <= P/128 + 1)
  const int64_t ub = static_cast<int64_t>(p.n_wb) * (std::min<int64_t>(p.E, P) + P / kBN + 1);
  const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(num_sms(), ub)));
  moe_gemm_kernel<GATE_UP><<<grid, kGemmThreads, C::kSmemBytes, stream>>>(tmA, tmB, p);
  BI_CHECK_LAUNCH();
  return BI_OK;
}

bi_status launch_gate_up(const void *x_perm, const int32_t *offsets, const int32_t *perm,
                         const float *wts, const void *w13, void *act, int64_t P, int64_t H,
                         int64_t E, int32_t top_k, int64_t I, cudaStream_t stream) {
  (void)top_k;
  CUtensorMap tmA, tmB;
  if (!make_tma_2d_bf16(&tmA, w13, static_cast<uint64_t>(E * 2 * I), static_cast<uint64_t>(H), kBM) ||
      !make_tma_2d_bf16(&tmB, x_perm, static_cast<uint64_t>(P), static_cast<uint64_t>(H), kBN))
    return BI_ERR_CUDA;
  GemmParams p{offsets, perm, wts, act, (int)E, (int)H, (int)(I / kBM), (int)I, (int)(2 * I), (int)I,
               device_error_word()};
  return launch_gemm<true>(tmA, tmB, p, P, stream);
}

bi_status launch_down(const void *act, const int32_t *offsets, const int32_t *perm, const void *w2,
                      float *contrib, int64_t P, int64_t H, int64_t E, int32_t top_k, int64_t I,
                      cudaStream_t stream) {
  (void)top_k;
  CUtensorMap tmA, tmB;
  if (!make_tma_2d_bf16(&tmA, w2, static_cast<uint64_t>(E * H), static_cast<uint64_t>(I), kBM) ||
      !make_tma_2d_bf16(&tmB, act, static_cast<uint64_t>(P), static_cast<uint64_t>(I), kBN))
    return BI_ERR_CUDA;
  GemmParams p{offsets, perm, nullptr, contrib, (int)E, (int)I, (int)(H / kBM), (int)H, (int)H, 0,
               device_error_word()};
  return launch_gemm<false>(tmA, tmB, p, P, stream);
}

}  // namespace bimoe
