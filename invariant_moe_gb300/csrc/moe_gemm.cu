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
//   * swap-AB: weight rows are the MMA "M" side, the tokens routed to one
//     expert are the "N" side (up to 256 per tile), K runs over the hidden
//     (gate/up) or intermediate (down) dimension.
//   * tcgen05.mma kind::f16 per K=16 step: bf16 operands, fp32 accumulator in
//     tensor memory, N = the tile's token count rounded up to 16.  K advances
//     in steps of 64 (one 128-byte swizzle atom, four MMAs) in increasing k
//     into the same accumulator, no split-K: each output element sees the
//     same K order whatever the batch is (the instruction's M and N only
//     decide how many rows and token columns are computed; the tests check
//     that neither the batch nor the variant below changes a bit).
//   * three variants of one kernel template (bi_moe_gemm_variant selects;
//     automatic by shape and batch):
//       - one CTA per tile, cta_group::1, M=128 weight rows.  gate/up: 128
//         gate rows j0.. and the 128 matching up rows I+j0.. against up to
//         128 tokens, two MMAs per K step sharing the token tile into two
//         accumulators; down: 128 rows of W2 against up to 256 tokens.
//       - CTA pairs, cta_group::2 (output features a multiple of 256): two
//         SMs of a cluster share a tile of 256 weight rows; each stages its
//         own 128 rows and HALF of the token rows, and one thread of the even
//         CTA issues M=256 MMAs reading the token rows from both SMs, so each
//         SM stages 40 KB (gate/up) or 32 KB (down) per K step instead of 48.
//       - interleaved gate/up rows (gate/up), in CTA pairs (automatic for
//         H >= 4096 once the experts average 64 or more rows) or one CTA
//         per tile (automatic for the smallest decode batches): each CTA
//         holds 64 gate rows and the matching 64 up rows against up to 256
//         tokens (one 4-D TMA copy lands the 16-row gate and up groups
//         interleaved); a lane and its partner lane swap half of each chunk.
//     and two token-tile widths: up to 128/256 tokens, or NARROW tiles of up
//     to 32 tokens with the deepest ring shared memory allows, for batches of
//     at most 16 rows per expert on average (decode), where the weight
//     stream is the whole cost (automatic choice there: one CTA per tile).
//   * the epilogue computes act = bf16(silu(g) * u * p) (gate/up) or writes
//     fp32 contributions to row token*top_k + slot (down).
//   * TMA (cp.async.bulk.tensor, 128-byte swizzle) fills a ring of stages;
//     accumulators are double buffered (2 x 256 tensor-memory columns) so the
//     epilogue of one tile overlaps the MMAs of the next.
//   * warp roles: warp 0 issues TMA, warp 1 owns tensor memory and issues the
//     MMAs (each loop inside one elect_one() block: a single thread issues a
//     stage's copies or MMAs back to back with uniform operands), warps 2-5
//     drain the accumulator (tcgen05.ld).  Every mbarrier wait is bounded.
//   * persistent grid (one CTA, or CTA pair, per SM or SM pair); tiles are
//     ordered expert, weight block, token block, so the token blocks of a
//     weight block run back to back and share it through L2.
//   * decode-sized batches: every CTA derives the routing itself (DECODE);
//     in the layer call the gate/up and down GEMMs can run as one launch
//     (moe_decode_layer_kernel: the gate/up tiles, then the down tiles with
//     the combine fused, each down K block loaded once the gate/up tile that
//     stores it has finished: a bounded wait).
#include <atomic>
#include <mutex>

#include "bimoe_internal.cuh"
#include "topk_warp.cuh"

namespace bimoe {

constexpr int kBM = 128;                    // MMA M: weight rows per tile
constexpr int kBK = 64;                     // K per stage (one swizzle atom of bf16)
constexpr int kUK = 16;                     // K of one MMA
constexpr int kTileBytes = kBM * kBK * 2;   // 16 KB: one 128-row operand tile
constexpr int kAccCols = 256;               // tensor-memory columns per accumulator buffer
constexpr int kNumAcc = 2;                  // double-buffered
constexpr int kTmemCols = kNumAcc * kAccCols;
constexpr int kGemmThreads = 192;
constexpr int kAuxBytes = 12288;            // barriers, tile prefix, expert offsets

// gate/up: A = gate + up tiles (32 KB), up to 128 tokens, two 128-column
// accumulators per buffer.  down: A = one tile (16 KB), up to 256 tokens, one
// 256-column accumulator per buffer.  One CTA per tile stages all the tile's
// token rows (48 KB stages, 4 deep); a CTA pair stages half of them per SM
// (40 KB x 5 for gate/up, 32 KB x 6 for down).
// INTER (gate/up): each CTA stages 64 gate rows and the matching 64 up rows
// as one 128-row A operand, against up to 256 tokens (for a pair, 128 token
// rows per SM and one M=256 x N=256 MMA per K step; alone, one M=128 MMA).
// The rows go in 16-row groups, gate rows of 16 features then the up rows of
// the same 16, so each tensor-memory lane quarter (one epilogue warp) holds
// both halves of its features and a lane swaps half of a chunk with
// lane ^ 16 by shuffle.
// NARROW (decode-sized batches): tiles of at most 32 tokens, so a stage is
// almost all weight bytes and the ring is as deep as shared memory allows;
// with few tokens per expert a CTA's time is the weight stream, and the
// bytes it keeps in flight set its rate.
constexpr int kSmemLimit = 227 * 1024;

template <bool GATE_UP, bool PAIR, bool INTER = false, bool NARROW = false>
struct GemmCfg {
  static_assert(!INTER || GATE_UP, "interleaved rows are a gate/up layout");
  static constexpr int kBN = NARROW ? 32 : ((GATE_UP && !INTER) ? 128 : 256);  // tokens per tile (largest MMA N)
  static constexpr int kBNc = PAIR ? kBN / 2 : kBN; // token rows staged per CTA
  static constexpr int kABytes = (GATE_UP && !INTER ? 2 : 1) * kTileBytes;
  static constexpr int kStageBytes = kABytes + kBNc * kBK * 2;
  // 2 warp pairs x (g, u) halves of 16 x 32 fp32, then one decision flag per epilogue warp
  static constexpr int kXchgBytes = 0;
  static constexpr int kNarrowStages = (kSmemLimit - 1024 - kAuxBytes - kXchgBytes) / kStageBytes;
  static constexpr int kStages =
      NARROW ? (kNarrowStages < 16 ? kNarrowStages : 16) : (PAIR ? (GATE_UP && !INTER ? 5 : 6) : 4);
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kAuxBytes + kXchgBytes;
  static_assert(kSmemBytes <= kSmemLimit, "shared memory");
  static_assert(kStageBytes % 1024 == 0 && kABytes % 1024 == 0, "swizzle atoms");
};

struct GemmParams {
  const int32_t *offsets;  // [E+1] first permuted position of each expert
  const int32_t *perm;     // [P] pair id (token*top_k + slot) of each position
  const float *wts;        // [M*top_k] routing probabilities (gate/up only)
  void *out;               // gate/up: act bf16 [P, I]; down: contrib fp32 [M*top_k, H]
  int E;
  int K;                   // reduction length (H for gate/up, I for down)
  int n_wb;                // weight blocks per expert (output features / wb_rows)
  int wb_rows;             // output features per weight block (128, or 256 for a CTA pair)
  int out_ld;              // output row length (I or H)
  int a_rows_per_expert;   // rows of the weight tensor per expert (2I or H)
  int up_offset;           // row offset of the up half (I), gate/up only
  int *err;
  int P;                   // (token, slot) pairs: rows of the token operand and of the output
  int top_k;               // slots per token (GATHER: token of pair id q = q / top_k)
  // DECODE only: the kernel derives offsets / perm from the expert ids itself
  const int32_t *ids;      // [M, top_k]
  int M;                   // tokens
  int *counters;           // [M, n_fb32] contributions summed per (token, 32-feature block)
  __nv_bfloat16 *lout;     // [M, out_ld] layer output (down: the fused combine writes it)
  int n_fb32;              // out_ld / 32
  // DECODE gate/up of the whole layer (bi_moe_layer): the router scores
  // [M, E]; every CTA selects the top_k experts of each row itself (the
  // selection of bi_topk) and CTA 0 writes ids / wts for the caller and the
  // down GEMM.  Null otherwise.
  const float *scores;
  int32_t *ids_out;
  float *wts_out;
};

// The down phase of the one-launch decode layer (moe_decode_layer_kernel):
// its shape, and the counts the gate/up tiles' epilogue warps arrive on.
struct DownPhase {
  void *out;              // contributions fp32 [M*top_k, H]
  int K;                  // I
  int n_wb;               // weight blocks per expert (H / 128)
  int wb_rows;            // 128
  int out_ld;             // H
  int a_rows_per_expert;  // H
  unsigned *ready;        // [gate/up tiles] arrivals (4 per tile: its epilogue warps); zero before the launch
};

// Decode-sized batches (bi_moe_forward with M * top_k <= kDecodeMaxP):
// every CTA of the two expert GEMMs derives the routing from the expert ids
// itself, so no permutation, gather or combine kernel runs (see DECODE).
// One warp routes the pairs (a lane per pair), so the path stops at 32
// pairs; below that the decode path won on every GB300 measured (layer
// time, CUDA-graph replay, cold L2, two boxes: Qwen3-30B-A3B-shaped M = 1 / 4:
// 42.4-44.1 / 87.3-87.9 us against 44.9-46.9 / 89.5-89.6 us; DSv4-shaped
// M = 1 / 4: 104.4-106.7 / 293.6-295.1 against 110.6-110.8 / 295.4-298.7 us);
// at 64 pairs (M = 8) it was within +-2.5 us either way, beyond it slower.
constexpr int kDecodeMaxP = 32;
// the one-launch decode layer's ready counts (one per gate/up tile) fit in a
// workspace region of this many words
constexpr int kDecodeReadyMax = 1024;
// the aux region holds the barriers (at most 16 stages), the tile prefix and
// expert offsets for E <= 1024, the decode routing tables and the gathered
// rows' tokens (at most 256)
static_assert(8 * (2 * 16 + 2 * kNumAcc + 1) + 16 + 4 * (2 * 1025 + 8 * kDecodeMaxP + 1 + 256) <= kAuxBytes,
              "aux shared memory");

struct TileInfo {
  int e, wb, tok0, ntok;
};

// A compile-time phase for the per-tile code of the producer and epilogue
// (gate/up or down), so that each phase's loops are compiled on their own.
template <bool GU>
struct PhaseTag {
  static constexpr bool value = GU;
};

template <int kBN>
__device__ __forceinline__ TileInfo decode_tile(int tile, const int *tile_prefix,
                                                const int *offs, const GemmParams &p) {
  int lo = 0, hi = p.E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tile_prefix[mid] <= tile) lo = mid;
    else hi = mid - 1;
  }
  TileInfo t;
  t.e = lo;
  const int local = tile - tile_prefix[lo];
  const int beg = offs[lo];
  const int cnt = offs[lo + 1] - beg;
  const int ntt = (cnt + kBN - 1) / kBN;
  t.wb = local / ntt;
  const int tt = local - t.wb * ntt;
  t.tok0 = beg + tt * kBN;
  t.ntok = min(kBN, cnt - tt * kBN);
  return t;
}

// Routing of a decode-sized batch (at most 32 pairs), computed by one warp of
// every CTA from the expert ids, lane i holding pair i = token * top_k +
// slot; the result equals the permutation kernels': the valid pairs grouped
// by expert in increasing expert order, in token order inside an expert (a
// token holds an expert at most once).  A slot whose id is outside [0,E) or
// repeats an earlier slot of its row is skipped.  Writes, for the nv valid
// pairs at positions p < nv: perm_s[p] = pair id, tokp_s[p] = its token; for
// the nd distinct experts d (increasing): dexp_s[d] = expert, dbeg_s[d] =
// its first position, dcnt_s[d] = its pairs; tok_s[m] = mask of token m's
// valid slots.  Returns nd on every lane.
__device__ __forceinline__ int decode_routing_warp(const int32_t *ids, const int32_t *ids_s, int M, int top_k,
                                                   int E, int *perm_s, int *tokp_s, int *dexp_s, int *dbeg_s,
                                                   int *dcnt_s, uint32_t *tok_s, int *err, bool report,
                                                   int lane) {
  const int P = M * top_k;
  const int m = lane / top_k;
  int e = -1;
  if (lane < P) e = ids ? __ldg(ids + lane) : ids_s[lane];
  bool ok = lane < P && e >= 0 && e < E;
  if (lane < P && !ok && report) report_error(err, BI_DEVERR_BAD_EXPERT_ID);
  const uint32_t lower = (1u << lane) - 1u;
  // an earlier slot of the same token holding the same expert
  const uint32_t dup = __match_any_sync(0xffffffffu, ok ? static_cast<uint32_t>(m * E + e) : 0x80000000u | lane);
  if (ok && (dup & lower)) {
    ok = false;
    if (report) report_error(err, BI_DEVERR_REPEATED_EXPERT);
  }
  const uint32_t valid = __ballot_sync(0xffffffffu, ok);
  const uint32_t same = __match_any_sync(0xffffffffu, ok ? e : E + lane);  // lanes of this expert
  const bool head = ok && !(same & lower);                                 // first lane of its expert
  const uint32_t heads = __ballot_sync(0xffffffffu, head);
  // valid pairs (and distinct experts) of smaller experts
  int less = 0, dless = 0;
  for (int j = 0; j < P; ++j) {
    const int ej = __shfl_sync(0xffffffffu, e, j);
    const bool lt = ((valid >> j) & 1u) && ej < e;
    less += lt;
    dless += lt && ((heads >> j) & 1u);
  }
  if (ok) {
    const int pos = less + __popc(same & lower);
    perm_s[pos] = lane;
    tokp_s[pos] = m;
    if (head) {
      dexp_s[dless] = e;
      dbeg_s[dless] = less;
      dcnt_s[dless] = __popc(same);
    }
  }
  if (lane < M) {
    const uint32_t slots = top_k >= 32 ? 0xffffffffu : (1u << top_k) - 1u;
    tok_s[lane] = (valid >> (lane * top_k)) & slots;  // lane * top_k <= 32 - top_k
  }
  return __popc(heads);
}

// act = silu(g) * u * p: a fixed fp32 sequence, one bf16 rounding.
__device__ __forceinline__ __nv_bfloat16 swiglu_p(float g, float u, float p) {
  const float sg = __fdividef(g, __fadd_rn(1.0f, __expf(-g)));
  return __float2bfloat16_rn(__fmul_rn(__fmul_rn(sg, u), p));
}

// GATHER (gate/up): tmB maps the token matrix x [M, H] itself with a box of
// one row, and the producer warp gathers each tile's token rows (pair
// perm[p] belongs to token perm[p] / top_k) with tile::gather4 loads, one
// group of 4 rows per lane, instead of a tiled load from the gathered copy
// x_perm.  The bytes that land in shared memory are the same rows in the same
// swizzled layout, so the MMAs -- and the bits -- are unchanged.
// DECODE (decode-sized batches, one CTA per tile, narrow tiles): offsets and
// perm are not read from memory; every CTA derives them from the expert ids
// (decode_routing_warp).  gate/up (with GATHER) also zeroes the arrival counters
// and the output rows of tokens with no valid slot; down fuses the top-k
// combine: after storing its fp32 contributions, each epilogue warp counts
// one arrival per token of the tile on that token's counter for the warp's 32
// features, and the warp whose arrival completes the count (all the token's
// valid slots stored) sums the k contributions in slot order and writes the
// bf16 output -- the same sequence of adds as the combine kernel.  No warp
// waits for another.
// FUSED (moe_decode_layer_kernel): the DECODE gate/up GEMM (interleaved rows,
// GATHER) and the DECODE down GEMM in one launch of at most one CTA per SM.
// The tile list is the gate/up tiles, then the down tiles (tmA2 / tmB2 / dn:
// W2 and the activations); both phases use the same 20 KB stages.  K block
// kb of a down tile (64 activation features of its expert's tokens) is what
// gate/up tile (expert, kb) stores, so each epilogue warp arrives on
// dn.ready[gate/up tile] once that tile's activations are stored, and the
// producer loads a down stage's W2 rows at once but its activation rows only
// when the count of that K block's gate/up tile is complete (a bounded
// wait): the down MMAs run as the gate/up tiles they need finish.  The
// combine counters and dn.ready are zeroed before the launch (by the
// router kernel of the same layer call), not here: CTAs start at different
// moments and no point of this launch orders them all.
template <bool GATE_UP, bool PAIR, bool INTER, bool NARROW, bool GATHER, bool DECODE, bool FUSED,
          int RING_DROP = 0>
__device__ __forceinline__ void moe_gemm_body(const CUtensorMap &tmA, const CUtensorMap &tmB, const GemmParams &prm,
                                              const CUtensorMap &tmA2, const CUtensorMap &tmB2,
                                              const DownPhase &dn) {
  static_assert(!FUSED || (GATE_UP && INTER && NARROW && GATHER && DECODE && !PAIR), "fused decode layer");
  static_assert(!FUSED || (GemmCfg<true, false, true, true>::kStageBytes == GemmCfg<false, false, false, true>::kStageBytes &&
                           GemmCfg<true, false, true, true>::kABytes == GemmCfg<false, false, false, true>::kABytes &&
                           GemmCfg<true, false, true, true>::kBN == GemmCfg<false, false, false, true>::kBN),
                "both phases of the fused decode layer share one stage layout");
  static_assert(!GATHER || GATE_UP, "the token gather feeds the gate/up GEMM");
  static_assert(!DECODE || (NARROW && !PAIR), "the decode path runs narrow tiles, one CTA per tile");
  static_assert(!DECODE || !GATE_UP || GATHER, "decode gate/up gathers its token rows");
  using C = GemmCfg<GATE_UP, PAIR, INTER, NARROW>;
  constexpr int kBN = C::kBN;
  constexpr int kStages = C::kStages - RING_DROP;  // FUSED beside the router: one stage fewer
  constexpr int kStageBytes = C::kStageBytes;
  constexpr int kABytes = C::kABytes;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *tiles = smem;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kStages * kStageBytes);
  uint64_t *full = bars;
  uint64_t *empty = bars + kStages;
  uint64_t *tfull = bars + 2 * kStages;
  uint64_t *tempty = tfull + kNumAcc;
  uint64_t *drain = tempty + kNumAcc;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  int *tile_prefix = reinterpret_cast<int *>(tmem_slot + 4);  // [E+1]
  int *offs = tile_prefix + prm.E + 1;                        // [E+1] copy of prm.offsets
  // DECODE: the routing derived in the prologue (decode_routing_warp)
  int *perm_s = offs + prm.E + 1;                                        // pair id at position p
  int *tokp_s = perm_s + kDecodeMaxP;                                    // its token
  int *vexp_s = tokp_s + kDecodeMaxP;                                    // selected ids (own_select)
  float *wts_s = reinterpret_cast<float *>(vexp_s + kDecodeMaxP);        // selected weights
  uint32_t *tok_s = reinterpret_cast<uint32_t *>(wts_s + kDecodeMaxP);  // valid slots of token m
  int *dexp_s = reinterpret_cast<int *>(tok_s + kDecodeMaxP);           // distinct experts ...
  int *dbeg_s = dexp_s + kDecodeMaxP;                                    // ... their first position
  int *dcnt_s = dbeg_s + kDecodeMaxP;                                    // ... and pair count
  int *nd_s = dcnt_s + kDecodeMaxP;                                      // number of distinct experts
  int *grow_s = nd_s + 1;  // GATHER: token of each gathered row of the current tile [kBNc]
  // routing probability of pair id q (selected in this CTA for the layer)
  const bool own_select = DECODE && GATE_UP && prm.scores != nullptr;
  auto wts_at = [&](int q) { return own_select ? wts_s[q] : __ldg(prm.wts + q); };
  // pair id at permuted position p
  auto perm_at = [&](int p) {
    if constexpr (DECODE) return perm_s[p];
    else return __ldg(prm.perm + p);
  };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // K blocks of a tile (the down tiles of FUSED reduce over dn.K)
  auto nkb_of = [&](bool gu) { return ((FUSED && !gu) ? dn.K : prm.K) / kBK; };
  // A CTA pair walks the tile list as one unit: both CTAs see the same tiles.
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const bool leader = rank == 0;
  const int unit0 = PAIR ? static_cast<int>(cluster_id_x()) : static_cast<int>(blockIdx.x);
  const int nunits = PAIR ? static_cast<int>(num_clusters_x()) : static_cast<int>(gridDim.x);
  auto wait = [&](uint32_t bar, uint32_t parity, volatile int *ab) {
    return PAIR ? mbar_wait_cl(bar, parity, ab, prm.err) : mbar_wait(bar, parity, ab, prm.err);
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int a = 0; a < kNumAcc; ++a) {
      mbar_init(smem_u32(&tfull[a]), 1);
      // pair: one arrival per epilogue warp of both CTAs, on the even CTA's barrier
      mbar_init(smem_u32(&tempty[a]), PAIR ? 8 : 128);
    }
    mbar_init(smem_u32(drain), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (FUSED) {
      tma_prefetch_desc(&tmA2);
      tma_prefetch_desc(&tmB2);
    }
  }
  if (warp == 1) {
    if (PAIR) {
      if (lane == 0) *tmem_slot = 0u;
      __syncwarp();
      tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(tmem_slot), kTmemCols);
      tmem_relinquish();
    }
  }
  // Nothing above reads what earlier kernels write (the tensor maps are
  // parameters), so it overlaps their end; from here on the offsets,
  // permutation and operands are read.  (Tensor memory is never held by a
  // predecessor on the same SM: only these GEMM kernels allocate it and their
  // CTAs need most of an SM's shared memory.)
  griddep_wait();
  if constexpr (DECODE) {
    if (own_select) {
      // the layer's top-k selection, row m by warp m % 6 (rows < M <= 64),
      // into shared memory; CTA 0 also writes it out
      for (int m = warp; m < prm.M; m += kGemmThreads / 32) {
        const float *row = prm.scores + static_cast<size_t>(m) * prm.E;
        auto load = [&](int j) { return __ldcg(row + j); };
        int32_t *irow = vexp_s + m * prm.top_k;
        float *wrow = wts_s + m * prm.top_k;
        if (prm.E <= 32) topk_select_warp<1>(load, prm.E, prm.top_k, irow, wrow, nullptr, lane);
        else if (prm.E <= 64) topk_select_warp<2>(load, prm.E, prm.top_k, irow, wrow, nullptr, lane);
        else if (prm.E <= 128) topk_select_warp<4>(load, prm.E, prm.top_k, irow, wrow, nullptr, lane);
        else if (prm.E <= 256) topk_select_warp<8>(load, prm.E, prm.top_k, irow, wrow, nullptr, lane);
        else topk_select_warp<16>(load, prm.E, prm.top_k, irow, wrow, nullptr, lane);
      }
      __syncthreads();
      if (blockIdx.x == 0 && warp >= 2)
        for (int i = threadIdx.x - 64; i < prm.M * prm.top_k; i += kGemmThreads - 64) {
          prm.ids_out[i] = vexp_s[i];
          prm.wts_out[i] = wts_s[i];
        }
    }
    if (warp == 0) {
      const int nd = decode_routing_warp(own_select ? nullptr : prm.ids, vexp_s, prm.M, prm.top_k, prm.E, perm_s,
                                         tokp_s, dexp_s, dbeg_s, dcnt_s, tok_s, prm.err,
                                         GATE_UP && blockIdx.x == 0, lane);
      if (lane == 0) *nd_s = nd;
    } else if (GATE_UP && !FUSED) {
      // for the down GEMM that follows: its arrival counters start at zero
      const int nc = prm.M * prm.n_fb32;
      for (int i = blockIdx.x * (kGemmThreads - 32) + threadIdx.x - 32; i < nc; i += gridDim.x * (kGemmThreads - 32))
        prm.counters[i] = 0;
    }
  } else {
    // the expert offsets in shared memory: one global round trip for all
    // threads instead of a chain of dependent loads in the tile scan below
    for (int i = threadIdx.x; i <= prm.E; i += kGemmThreads) offs[i] = __ldg(prm.offsets + i);
    __syncthreads();
  }
  if (!DECODE && warp == 2) {
    // tile_prefix[e] = tiles of experts < e; each lane scans a contiguous chunk
    const int per = (prm.E + 31) / 32;
    const int e0 = min(lane * per, prm.E), e1 = min(e0 + per, prm.E);
    // offsets that are not non-decreasing inside [0, P] would put tiles
    // outside the operands: then the kernel does no tile and records the error
    bool bad = lane == 0 && (offs[0] < 0 || offs[prm.E] > prm.P);
    int local = 0;
    for (int e = e0; e < e1; ++e) {
      const int cnt = offs[e + 1] - offs[e];
      bad = bad || cnt < 0;
      local += prm.n_wb * ((max(cnt, 0) + kBN - 1) / kBN);
    }
    bad = __any_sync(0xffffffffu, bad);
    int incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += v;
    }
    int run = incl - local;
    for (int e = e0; e < e1; ++e) {
      tile_prefix[e] = run;
      const int cnt = offs[e + 1] - offs[e];
      run += prm.n_wb * ((max(cnt, 0) + kBN - 1) / kBN);
    }
    if (lane == 31) tile_prefix[prm.E] = bad ? 0 : incl;
    if (bad && lane == 0) report_error(prm.err, BI_DEVERR_BAD_PERMUTATION);
  }
  tc_fence_before();
  __syncthreads();
  // the peer's barriers are initialised before anything is sent to them
  if (PAIR) cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // FUSED: the gate/up tiles (n_gu of them), then the down tiles
  const int n_gu = DECODE ? *nd_s * prm.n_wb : 0;
  const int total_tiles = DECODE ? (FUSED ? n_gu + *nd_s * dn.n_wb : n_gu) : tile_prefix[prm.E];
  auto gu_tile = [&](int tile) { return FUSED ? tile < n_gu : GATE_UP; };
  if (DECODE && GATE_UP && blockIdx.x == 0 && warp >= 2) {
    // tokens with no valid slot (no tile stores them) get zero output rows
    for (int m = 0; m < prm.M; ++m)
      if (tok_s[m] == 0u)
        for (int h = threadIdx.x - 64; h < prm.n_fb32 * 32; h += kGemmThreads - 64)
          prm.lout[static_cast<size_t>(m) * prm.n_fb32 * 32 + h] = __float2bfloat16_rn(0.0f);
  }
  // the tile's expert, weight block and token range
  auto tile_at = [&](int tile) {
    if constexpr (DECODE) {
      // one token tile per distinct expert (at most 32 pairs), its weight
      // blocks in order (FUSED: the gate/up list, then the down list)
      TileInfo t;
      int local = tile, nwb = prm.n_wb;
      if (FUSED && tile >= n_gu) {
        local = tile - n_gu;
        nwb = dn.n_wb;
      }
      const int d = local / nwb;
      t.e = dexp_s[d];
      t.wb = local - d * nwb;
      t.tok0 = dbeg_s[d];
      t.ntok = dcnt_s[d];
      return t;
    } else {
      return decode_tile<kBN>(tile, tile_prefix, offs, prm);
    }
  };

  // The producer and MMA loops run on one elected lane of their warp alone
  // (waits, copies, MMAs, commits).  Measured on GB300 (a tcgen05.mma
  // probe): an elect and a warp sync around every MMA cost ~250 cycles an
  // MMA; a loop inside one `if (elect_one())` block ~60 cycles at N=16 (the
  // tensor rate at N=256); the same loop under `if (lane == 0)` ~150, as
  // the operands leave uniform registers.
  if (warp == 0) {
    // ------------------------------------------------------ TMA producer --
    int stage = 0;
    uint32_t phase = 0;
    uint32_t issued_mask = 0, issued_parity = 0;
    // one tile's copies; returns false when the tile loop must stop
    auto produce = [&](auto phase_tag, int tile) -> bool {
      constexpr bool gu = decltype(phase_tag)::value;
      constexpr bool gather_t = GATHER && gu;
      const TileInfo ti = tile_at(tile);
      const int nkb_t = nkb_of(gu);
      const int a_row = (FUSED && !gu) ? ti.e * dn.a_rows_per_expert + ti.wb * dn.wb_rows
                                       : ti.e * prm.a_rows_per_expert + ti.wb * prm.wb_rows +
                                             static_cast<int>(rank) * (INTER ? kBM / 2 : kBM);
      // pair: the odd CTA stages tokens N/2.. of the tile's MMA N
      const int b_row = ti.tok0 + (rank ? ((ti.ntok + 15) & ~15) / 2 : 0);
      constexpr int kGroups = C::kBNc / 4;
      // GATHER: only this CTA's real token rows are fetched, four per
      // gather, and the stage expects exactly those bytes.  The MMA N is the
      // tile's tokens rounded up to 16; the columns past the real tokens read
      // whatever rows the stage held before and are never stored (an
      // accumulator column depends on its own B row only).  A gathered row
      // costs the copy engine far more than a row of a tiled box, so at
      // decode sizes (one token: 4 rows instead of 16) this sets the stage
      // rate.
      const int half = ((ti.ntok + 15) & ~15) / 2;  // PAIR: token rows staged per CTA
      auto real_groups = [&](int r) {
        const int rows = PAIR ? max(0, min(ti.ntok - r * half, half)) : ti.ntok;
        return min(kGroups, (rows + 3) / 4);
      };
      const int ngroups = gather_t ? real_groups(static_cast<int>(rank)) : kGroups;
      const uint32_t stage_bytes = gather_t ? static_cast<uint32_t>(kABytes + ngroups * 4 * kBK * 2)
                                            : static_cast<uint32_t>(kStageBytes);
      const uint32_t pair_bytes =
          GATHER ? static_cast<uint32_t>(2 * kABytes + (real_groups(0) + real_groups(1)) * 4 * kBK * 2)
                 : 2u * static_cast<uint32_t>(kStageBytes);
      if (gather_t) {
        // the token of each gathered row (the warp fills the table, lane 0
        // issues); rows past the tile's tokens (and any position whose perm
        // entry is not a pair id, reported by the epilogue) fetch token 0,
        // whose columns the epilogue never stores
        for (int q = lane; q < ngroups * 4; q += 32) {
          const int pos = b_row + q;
          int tok = 0;
          if (pos < ti.tok0 + ti.ntok) {
            if constexpr (DECODE) {
              tok = tokp_s[pos];
            } else {
              const int pq = perm_at(pos);
              if (static_cast<unsigned>(pq) < static_cast<unsigned>(prm.P)) tok = pq / prm.top_k;
            }
          }
          grow_s[q] = tok;
        }
        __syncwarp();
      }
      bool ok = true;
      const bool el = elect_one();
      if (el) {
        // FUSED down tile: the stages (consecutive in the ring, from
        // dq_stage, K blocks from dq_kb) whose weight rows are loading and
        // whose activation rows wait for their gate/up tile; K block kb's is
        // gate/up tile d * n_wb + kb, d the tile's distinct expert
        int dq_n = 0, dq_stage = 0, dq_kb = 0;
        const unsigned *rdy = nullptr;
        if constexpr (FUSED && !gu) rdy = dn.ready + ((tile - n_gu) / dn.n_wb) * prm.n_wb;
        // issue the waiting stages' activation loads in K order while their
        // gate/up tiles are stored; `block` waits (bounded) for the first
        // one, `all` for every one (after a timeout a load is issued all the
        // same, so every armed stage completes; the abort flag then stops
        // the MMAs and the epilogue)
        auto flush = [&](bool block, bool all) {
          bool fenced = false;
          while (dq_n > 0) {
            const unsigned *f = rdy + dq_kb;
            if (ld_acquire_gpu(f) < 4u) {
              if (!block) break;
              wait_count_geq(f, 4u, abort_flag, prm.err);
              block = all;
            }
            if (!fenced) {
              fence_proxy_async_global();  // the activations were stored through the generic proxy
              fenced = true;
            }
            tma_load_2d(smem_u32(tiles + dq_stage * kStageBytes + kABytes), &tmB2, smem_u32(&full[dq_stage]),
                        dq_kb * kBK, b_row);
            dq_stage = dq_stage + 1 == kStages ? 0 : dq_stage + 1;
            ++dq_kb;
            --dq_n;
          }
        };
        for (int kb = 0; kb < nkb_t; ++kb) {
          if (!wait(smem_u32(&empty[stage]), phase ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          uint8_t *st = tiles + stage * kStageBytes;
          if (PAIR) {
            // both CTAs' copies complete on the even CTA's barrier, which the
            // even CTA arms with the bytes of both
            const uint32_t fb = mapa_shared(smem_u32(&full[stage]), 0);
            if (leader) mbar_arrive_expect_tx(smem_u32(&full[stage]), pair_bytes);
            if (INTER) {
              // 16 gate rows, the 16 up rows of the same features, and so on
              // for four groups: one copy through the 4-D interleaved map
              tma_load_4d_pair(smem_u32(st), &tmA, fb, kb * kBK, 0, 0, a_row / 16);
            } else {
              tma_load_2d_pair(smem_u32(st), &tmA, fb, kb * kBK, a_row);
              if (GATE_UP)
                tma_load_2d_pair(smem_u32(st + kTileBytes), &tmA, fb, kb * kBK, a_row + prm.up_offset);
            }
            if (!GATHER) tma_load_2d_pair(smem_u32(st + kABytes), &tmB, fb, kb * kBK, b_row);
            else
              for (int g = 0; g < ngroups; ++g)
                tma_gather4_pair(smem_u32(st + kABytes + g * 4 * kBK * 2), &tmB, fb, kb * kBK, grow_s[4 * g],
                                 grow_s[4 * g + 1], grow_s[4 * g + 2], grow_s[4 * g + 3]);
          } else {
            const uint32_t fb = smem_u32(&full[stage]);
            mbar_arrive_expect_tx(fb, stage_bytes);
            if (INTER && gu) {
              tma_load_4d(smem_u32(st), &tmA, fb, kb * kBK, 0, 0, a_row / 16);
            } else {
              tma_load_2d(smem_u32(st), (FUSED && !gu) ? &tmA2 : &tmA, fb, kb * kBK, a_row);
            }
            if (GATE_UP && !INTER)
              tma_load_2d(smem_u32(st + kTileBytes), &tmA, fb, kb * kBK, a_row + prm.up_offset);
            if (FUSED && !gu) {
              // the stage's activation rows wait for their gate/up tile (the
              // barrier already expects their bytes); with the ring all
              // waiting, wait for the first; at the tile's last K block, for
              // all
              if (dq_n++ == 0) {
                dq_stage = stage;
                dq_kb = kb;
              }
              flush(dq_n == kStages || kb == nkb_t - 1, kb == nkb_t - 1);
            } else if (!gather_t) {
              tma_load_2d(smem_u32(st + kABytes), (FUSED && !gu) ? &tmB2 : &tmB, fb, kb * kBK, b_row);
            } else
              for (int g = 0; g < ngroups; ++g)
                tma_gather4(smem_u32(st + kABytes + g * 4 * kBK * 2), &tmB, fb, kb * kBK, grow_s[4 * g],
                            grow_s[4 * g + 1], grow_s[4 * g + 2], grow_s[4 * g + 3]);
          }
          issued_mask |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (FUSED && dq_n > 0) flush(true, true);  // only after a failed wait: complete the armed stages
      }
      // the ring state back on every lane (this also keeps grow_s until every
      // gather of the tile is issued)
      const int src = __ffs(__ballot_sync(0xffffffffu, el)) - 1;
      stage = __shfl_sync(0xffffffffu, stage, src);
      phase = __shfl_sync(0xffffffffu, phase, src);
      issued_mask = __shfl_sync(0xffffffffu, issued_mask, src);
      issued_parity = __shfl_sync(0xffffffffu, issued_parity, src);
      return __shfl_sync(0xffffffffu, ok ? 1 : 0, src) != 0;
    };
    for (int tile = unit0; tile < total_tiles; tile += nunits) {
      if (__shfl_sync(0xffffffffu, *abort_flag, 0) != 0) break;
      bool cont;
      if constexpr (FUSED) {
        cont = tile < n_gu ? produce(PhaseTag<true>{}, tile) : produce(PhaseTag<false>{}, tile);
      } else {
        cont = produce(PhaseTag<GATE_UP>{}, tile);
      }
      if (!cont) break;
    }
    if (lane == 0 && *abort_flag) {
      // let every copy this warp started land before the CTA can exit
      if (!PAIR || leader) {
        for (int s = 0; s < kStages; ++s)
          if ((issued_mask >> s) & 1u) wait(smem_u32(&full[s]), (issued_parity >> s) & 1u, nullptr);
      }
      if (PAIR) {
        // the odd CTA's copies complete on the even CTA's barriers: give
        // them time to land (copies take microseconds; this path only runs
        // after a wait has already given up)
        const unsigned long long t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 200000ull) {
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer --
    if (!leader) {
      // odd CTA of a pair: the even CTA's final commit arrives here
      if (lane == 0) wait(smem_u32(drain), 0, nullptr);
    } else if (elect_one()) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool issued_any = false;
      for (int tile = unit0; tile < total_tiles && !*abort_flag; tile += nunits) {
        // the MMA N covers the tile's real tokens (a multiple of 16), so a
        // ragged last tile of an expert does not pay for padding columns
        const TileInfo ti = tile_at(tile);
        const int nkb_t = FUSED && tile >= n_gu ? dn.K / kBK : prm.K / kBK;
        const uint32_t idesc = idesc_bf16_f32(PAIR ? 2 * kBM : kBM, (ti.ntok + 15) & ~15);
        if (!wait(smem_u32(&tempty[acc]), acc_phase ^ 1u, abort_flag)) break;
        tc_fence_after();
        const uint32_t d0 = tmem_base + static_cast<uint32_t>(acc * kAccCols);
        bool ok = true;
        for (int kb = 0; kb < nkb_t; ++kb) {
          if (!wait(smem_u32(&full[stage]), phase, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(tiles + stage * kStageBytes);
          const uint32_t b0 = a0 + kABytes;
          // the stage's MMAs back to back, then the commit that frees the
          // stage (in both CTAs of a pair) once they are done
#pragma unroll
          for (int k = 0; k < kBK / kUK; ++k) {
            const uint32_t acc_in = (kb | k) != 0 ? 1u : 0u;
            const uint64_t bdesc = sdesc_sw128(b0 + k * kUK * 2);
            const uint64_t adesc = sdesc_sw128(a0 + k * kUK * 2);
            const uint64_t udesc = sdesc_sw128(a0 + kTileBytes + k * kUK * 2);
            if (PAIR) {
              umma_f16_pair(d0, adesc, bdesc, idesc, acc_in);
              if (GATE_UP && !INTER) umma_f16_pair(d0 + kBN, udesc, bdesc, idesc, acc_in);
            } else {
              umma_f16(d0, adesc, bdesc, idesc, acc_in);
              if (GATE_UP && !INTER) umma_f16(d0 + kBN, udesc, bdesc, idesc, acc_in);
            }
          }
          if (PAIR) umma_commit_pair(smem_u32(&empty[stage]), 0x3);
          else umma_commit(smem_u32(&empty[stage]));
          issued_any = true;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if (PAIR) umma_commit_pair(smem_u32(&tfull[acc]), 0x3);
        else umma_commit(smem_u32(&tfull[acc]));
        if (++acc == kNumAcc) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (PAIR || (*abort_flag && issued_any)) {
        // pair: always, telling both CTAs that every MMA into their tensor
        // memory (and every read of their shared memory) has completed;
        // single CTA: after an abort, before tensor memory is released
        if (PAIR) umma_commit_pair(smem_u32(drain), 0x3);
        else umma_commit(smem_u32(drain));
        wait(smem_u32(drain), 0, nullptr);
      }
    }
    __syncwarp();
  } else {
    // --------------------------------------------------------- epilogue --
    // Warp w reads tensor-memory lanes 32*(w%4).. (weight rows of the tile);
    // the per-token data of a tile (pair ids, probabilities) is loaded one
    // tile ahead, lane l holding token 32i + l, so the dependent global loads
    // overlap the wait for the accumulator.
    const int q = warp & 3;
    const int row = q * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    int nx_pair[kBN / 32];
    float nx_p[kBN / 32];
    auto prefetch = [&](int tile) {
      const TileInfo t = tile_at(tile);
#pragma unroll
      for (int i = 0; i < kBN / 32; ++i) {
        const int c = 32 * i + lane;
        nx_pair[i] = c < t.ntok ? perm_at(t.tok0 + c) : 0;
        nx_p[i] = 0.0f;
      }
      if (gu_tile(tile)) {
        // a perm entry that is not a pair id reads no probability (checked
        // again, and reported, when the tile is stored)
#pragma unroll
        for (int i = 0; i < kBN / 32; ++i) {
          const int c = 32 * i + lane;
          const bool ok = static_cast<unsigned>(nx_pair[i]) < static_cast<unsigned>(prm.P);
          nx_p[i] = c < t.ntok && ok ? wts_at(nx_pair[i]) : 0.0f;
        }
      }
    };
    // one tile's epilogue; returns false when the tile loop must stop
    auto consume = [&](auto phase_tag, int tile) -> bool {
      constexpr bool gu = decltype(phase_tag)::value;
      const TileInfo ti = tile_at(tile);
      // per-phase output (the down tiles of FUSED write dn.out)
      const int out_ld_t = (FUSED && !gu) ? dn.out_ld : prm.out_ld;
      void *out_t = (FUSED && !gu) ? dn.out : prm.out;
      int my_pair[kBN / 32];
      float my_p[kBN / 32];
#pragma unroll
      for (int i = 0; i < kBN / 32; ++i) {
        my_pair[i] = nx_pair[i];
        my_p[i] = nx_p[i];
      }
      if (tile + nunits < total_tiles) prefetch(tile + nunits);
      // one decision per warp (lanes can disagree at the instant a wait gives up)
      const bool okw = __all_sync(0xffffffffu, wait(smem_u32(&tfull[acc]), acc_phase, abort_flag) ? 1 : 0) != 0;
      if (!okw) return false;
      {
        // perm entries of this tile that are not pair ids (the loads landed
        // long ago): reported once; nothing is stored through them below
        bool badp = false;
#pragma unroll
        for (int i = 0; i < kBN / 32; ++i)
          badp = badp || (32 * i + lane < ti.ntok &&
                          static_cast<unsigned>(my_pair[i]) >= static_cast<unsigned>(prm.P));
        if (badp) report_error(prm.err, BI_DEVERR_BAD_PERMUTATION);
      }
      tc_fence_after();
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                             static_cast<uint32_t>(acc * kAccCols);
      const int col = (INTER && gu) ? ti.wb * prm.wb_rows + static_cast<int>(rank) * (kBM / 2) + 16 * q + (lane & 15)
                                    : ti.wb * ((FUSED && !gu) ? dn.wb_rows : prm.wb_rows) +
                                          static_cast<int>(rank) * kBM + row;
#pragma unroll
      for (int i = 0; i < kBN / 32; ++i) {
        const int c0 = 32 * i;
        if (c0 >= ti.ntok) break;  // warp-uniform (and the same for both warps of a pair)
        uint32_t d[32];
        tmem_ld32(tbase + c0, d);
        if (INTER && gu) {
          // lanes 0-15 hold the gate rows of 16 features, lanes 16-31 the up
          // rows of the same features: the gate lane keeps tokens 0-15 of the
          // chunk and hands 16-31 to its partner (lane ^ 16), which hands
          // back the up values of tokens 0-15; each finishes 16 tokens
          tmem_ld_wait();
          const bool is_gate = lane < 16;
          __nv_bfloat16 *act = static_cast<__nv_bfloat16 *>(prm.out);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float mine = __uint_as_float(is_gate ? d[j] : d[16 + j]);
            const float other = __shfl_xor_sync(0xffffffffu, __uint_as_float(is_gate ? d[16 + j] : d[j]), 16);
            const int c = is_gate ? j : 16 + j;
            const float pc = __shfl_sync(0xffffffffu, my_p[i], c);
            const float g = is_gate ? mine : other;
            const float u = is_gate ? other : mine;
            if (c0 + c < ti.ntok)
              act[static_cast<size_t>(ti.tok0 + c0 + c) * prm.out_ld + col] = swiglu_p(g, u, pc);
          }
        } else if (GATE_UP && !INTER) {
          uint32_t u[32];
          tmem_ld32(tbase + kBN + c0, u);
          tmem_ld_wait();
          __nv_bfloat16 *act = static_cast<__nv_bfloat16 *>(prm.out);
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const float pc = __shfl_sync(0xffffffffu, my_p[i], c);
            if (c0 + c < ti.ntok)
              act[static_cast<size_t>(ti.tok0 + c0 + c) * prm.out_ld + col] =
                  swiglu_p(__uint_as_float(d[c]), __uint_as_float(u[c]), pc);
          }
        } else {
          tmem_ld_wait();
          float *contrib = static_cast<float *>(out_t);
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const int pair = __shfl_sync(0xffffffffu, my_pair[i], c);
            if (c0 + c < ti.ntok && static_cast<unsigned>(pair) < static_cast<unsigned>(prm.P))
              contrib[static_cast<size_t>(pair) * out_ld_t + col] = __uint_as_float(d[c]);
          }
        }
      }
      if (FUSED && gu) {
        // this warp's activation stores of the tile are done: one arrival on
        // the tile's count, which the down stages of its K block wait on.
        // The warp barrier orders every lane's stores before lane 0's
        // release (cumulative, GPU scope); the proxy fence orders them
        // before async-proxy (TMA) reads.  (A fence in every lane before the
        // warp barrier measured ~0.9 us slower per decode layer.)
        __syncwarp();
        if (lane == 0) {
          fence_proxy_async_global();
          red_release_gpu_add(dn.ready + tile, 1u);
        }
      }
      // the accumulator is free once its tensor-memory loads have completed
      // (tcgen05.wait::ld above); the arrival does not wait for this tile's
      // global stores, which only later kernels read
      tc_fence_before();
      if (PAIR) {
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster_relaxed(mapa_shared(smem_u32(&tempty[acc]), 0));
      } else {
        mbar_arrive_relaxed(smem_u32(&tempty[acc]));
      }
      if (DECODE && !gu) {
        // fused combine for this warp's 32 features (see DECODE above): one
        // arrival per token, an acquire-release add by the token's lane after
        // the warp barrier (which orders every lane's contribution stores
        // before it; measured 0.3-0.9 us per decode layer faster than a fence
        // in every lane before the add and another before the sum), and each
        // (token, 32-feature block) completed here is summed by this warp
        // once a second warp barrier orders the acquire before every lane's
        // loads
        const int fb32 = (ti.wb * ((FUSED && !gu) ? dn.wb_rows : prm.wb_rows) + q * 32) / 32;
        float *contrib = static_cast<float *>(out_t);
        __syncwarp();
        int tok = 0;
        bool last = false;
        if (lane < ti.ntok) {  // NARROW: at most 32 tokens per tile
          tok = tokp_s[ti.tok0 + lane];
          const int need = __popc(tok_s[tok]);
          last = atom_add_acq_rel_gpu(prm.counters + tok * prm.n_fb32 + fb32, 1) == need - 1;
        }
        unsigned todo = __ballot_sync(0xffffffffu, last);
        if (todo) __syncwarp();
        while (todo) {
          const int src = __ffs(todo) - 1;
          todo &= todo - 1;
          const int m = __shfl_sync(0xffffffffu, tok, src);
          const uint32_t valid = tok_s[m];
          const size_t f = static_cast<size_t>(fb32) * 32 + lane;
          float sum = 0.0f;
          bool any = false;
          for (int t = 0; t < prm.top_k; ++t) {
            if (!((valid >> t) & 1u)) continue;
            const float v = __ldcg(contrib + static_cast<size_t>(m * prm.top_k + t) * out_ld_t + f);
            sum = any ? __fadd_rn(sum, v) : v;
            any = true;
          }
          prm.lout[static_cast<size_t>(m) * out_ld_t + f] = __float2bfloat16_rn(sum);
        }
      }
      if (++acc == kNumAcc) {
        acc = 0;
        acc_phase ^= 1u;
      }
      return true;
    };
    if (unit0 < total_tiles) prefetch(unit0);
    for (int tile = unit0; tile < total_tiles; tile += nunits) {
      bool cont;
      if constexpr (FUSED) {
        cont = tile < n_gu ? consume(PhaseTag<true>{}, tile) : consume(PhaseTag<false>{}, tile);
      } else {
        cont = consume(PhaseTag<GATE_UP>{}, tile);
      }
      if (!cont) break;
    }
  }

  tc_fence_before();
  __syncthreads();
  // neither CTA of a pair leaves (or frees tensor memory) while the other
  // may still signal its barriers
  if (PAIR) cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    if (PAIR) tmem_dealloc_pair(tmem_base, kTmemCols);
    else tmem_dealloc(tmem_base, kTmemCols);
  }
}

template <bool GATE_UP, bool PAIR, bool INTER, bool NARROW, bool GATHER = false, bool DECODE = false>
__global__ void __launch_bounds__(kGemmThreads, 1)
    moe_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ GemmParams prm) {
  moe_gemm_body<GATE_UP, PAIR, INTER, NARROW, GATHER, DECODE, false>(tmA, tmB, prm, tmA, tmB, DownPhase{});
}

// The expert path of a decode-sized layer in one launch (FUSED above): at
// most one CTA per SM, all resident at once.  RING_DROP = 1: a ring one
// stage shorter, so that a CTA fits on an SM beside a CTA of the one-warp
// router kernel, which lets its dependents start at once.
template <int RING_DROP>
__global__ void __launch_bounds__(kGemmThreads, 1)
    moe_decode_layer_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                            const __grid_constant__ GemmParams prm, const __grid_constant__ CUtensorMap tmA2,
                            const __grid_constant__ CUtensorMap tmB2, const __grid_constant__ DownPhase dn) {
  moe_gemm_body<true, false, true, true, true, true, true, RING_DROP>(tmA, tmB, prm, tmA2, tmB2, dn);
}

// ------------------------------------------------------------------- host --
// 0 = automatic, 1 = one CTA per tile, 2 = CTA pairs, 3 = CTA pairs with
// interleaved gate/up rows for the gate/up GEMM (CTA pairs for down); the
// automatic choice is pick_variant below.  The interleaved rows lose at
// H=2048 (20 % slower on the gate/up GEMM), where the shorter K loop no
// longer hides the epilogue's exchange.
static std::atomic<int> g_gemm_variant{0};

int set_gemm_variant(int v) { return g_gemm_variant.exchange(v); }

template <bool GATE_UP, bool PAIR, bool INTER, bool NARROW, bool GATHER, bool DECODE = false>
static bi_status launch_gemm(const CUtensorMap &tmA, const CUtensorMap &tmB, const GemmParams &p,
                             int64_t P, cudaStream_t stream) {
  using C = GemmCfg<GATE_UP, PAIR, INTER, NARROW>;
  static std::mutex mu;
  static int max_units[64] = {};  // CTAs (or CTA pairs) resident at once, per device
  static ContextSetup setup;      // the shared-memory attribute is per context
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) {
    set_error("device ordinal %d out of range", dev);
    return BI_ERR_CUDA;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.blockDim = dim3(kGemmThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  if (PAIR) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  {
    std::lock_guard<std::mutex> lk(mu);
    if (max_units[dev] == 0 || setup.pending(dev)) {
      cudaError_t e = cudaFuncSetAttribute(moe_gemm_kernel<GATE_UP, PAIR, INTER, NARROW, GATHER, DECODE>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
      if (e != cudaSuccess) {
        cudaGetLastError();  // do not leave the error for an unrelated later check
        set_error("cudaFuncSetAttribute: %s", cudaGetErrorString(e));
        return BI_ERR_CUDA;
      }
      int units = num_sms();
      if (PAIR) {
        cfg.gridDim = dim3(2 * (num_sms() / 2));
        int clusters = 0;
        e = cudaOccupancyMaxActiveClusters(&clusters, moe_gemm_kernel<GATE_UP, PAIR, INTER, NARROW, GATHER, DECODE>, &cfg);
        if (e != cudaSuccess || clusters <= 0) {
          cudaGetLastError();
          set_error("cudaOccupancyMaxActiveClusters: %s (%d clusters)", cudaGetErrorString(e), clusters);
          return BI_ERR_CUDA;
        }
        units = clusters;
      }
      max_units[dev] = units;
      setup.done(dev);
    }
  }
  // upper bound on the number of tiles (token blocks per expert <= P/kBN + 1)
  const int64_t ub = static_cast<int64_t>(p.n_wb) * (std::min<int64_t>(p.E, P) + P / C::kBN + 1);
  const int units = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(max_units[dev], ub)));
  cfg.gridDim = dim3(PAIR ? 2 * units : units);
  // a programmatic dependent of the previous kernel on the stream (every
  // kernel of the library waits for its predecessors before reading)
  cudaLaunchAttribute attr2[2];
  attr2[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr2[0].val.programmaticStreamSerializationAllowed = 1;
  int nattr = 1;
  if (PAIR) attr2[nattr++] = attr[0];
  cfg.attrs = attr2;
  cfg.numAttrs = nattr;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, moe_gemm_kernel<GATE_UP, PAIR, INTER, NARROW, GATHER, DECODE>, tmA, tmB, p);
  if (e != cudaSuccess) {
    set_error("moe_gemm launch: %s", cudaGetErrorString(e));
    return BI_ERR_CUDA;
  }
  BI_CHECK_LAUNCH();
  return BI_OK;
}

// Which variant runs for `features` output features per expert (1 one CTA
// per tile, 2 CTA pairs, 3 CTA pairs with interleaved gate/up rows), or -1
// (error set) when a forced pair variant does not fit.  Automatic choice:
// interleaved gate/up rows for wide tokens (K >= 4096) once the experts
// average 64 or more rows (P >= 64 E); measured on GB300 for the DSv4-shaped
// layer (H=4096, E=256, I=2048): 3 % faster at M=4096 (128 rows per
// expert), 3-5 % slower at M <= 1024, where plain pairs win.
static bool use_narrow(int64_t P, int64_t E);

static int pick_variant(int64_t features, bool gate_up, int64_t K, int64_t P, int64_t E) {
  const int v = g_gemm_variant.load();
  const bool fits = features % (2 * kBM) == 0;
  // NARROW tiles: one CTA per tile (measured on GB300: 2-6 % faster than
  // CTA pairs at M <= 256 on both the Qwen- and DSv4-shaped layers); for
  // gate/up, 64-feature tiles with interleaved rows when even those fit in
  // one wave on the SMs (twice the CTAs streaming the touched weights: the
  // Qwen-shaped layer at M=1, 96 tiles, 44.1 vs 47.9 us; a second wave,
  // as for the DSv4-shaped layer at M=1, makes them slower)
  if (v == 0 && use_narrow(P, E))
    return (gate_up && std::min(E, P) * (features / (kBM / 2)) <= num_sms()) ? 4 : 1;
  if (gate_up && (v == 3 || (v == 0 && K >= 4096 && P >= 64 * E)))
    return 3;  // 128 features per CTA pair: any I % 128 == 0
  if (v == 4) return gate_up ? 4 : 1;  // 64 features per CTA (gate/up); down: one CTA per tile
  if (v >= 2 && !fits) {
    set_error("CTA-pair expert GEMMs need output features %% 256 == 0 (got %lld)",
              static_cast<long long>(features));
    return -1;
  }
  return (v == 1 || !fits) ? 1 : 2;
}

// Batches of at most 16 (token, expert) pairs per expert on average run the
// NARROW tiles (measured on GB300: the DSv4-shaped layer at M = 1 / 16 / 64 /
// 256 went from 135 / 878 / 1829 / 2139 us to 112 / 810 / 1727 / 2003 us,
// 94-96 % of the copy bandwidth over the touched weights for M >= 16; the
// Qwen-shaped layer at M=256, 16 pairs per expert, from 260 to 251 us; at 32
// and 64 pairs per expert the wide tiles win by 15-40 %).
static bool use_narrow(int64_t P, int64_t E) { return P <= 16 * E; }

// tok: the gathered copy [P, K] (GATHER = false: tiled loads of kBNc rows),
// or the token matrix [tok_rows = M, K] itself (GATHER: one-row box for
// tile::gather4).
template <bool GATE_UP, bool PAIR, bool INTER, bool NARROW, bool GATHER = false, bool DECODE = false>
static bi_status run_gemm(const void *wt, int64_t w_rows, uint32_t box_a, const void *tok, int64_t P,
                          int64_t K, const GemmParams &p, cudaStream_t stream, int64_t tok_rows = 0) {
  CUtensorMap tmA, tmB;
  const bool amap = INTER ? make_tma_inter_bf16(&tmA, wt, static_cast<uint64_t>(w_rows),
                                                static_cast<uint64_t>(p.up_offset), static_cast<uint64_t>(K))
                          : make_tma_2d_bf16(&tmA, wt, static_cast<uint64_t>(w_rows), static_cast<uint64_t>(K), box_a);
  if (!amap ||
      !make_tma_2d_bf16(&tmB, tok, static_cast<uint64_t>(GATHER ? tok_rows : P), static_cast<uint64_t>(K),
                        GATHER ? 1u : static_cast<uint32_t>(GemmCfg<GATE_UP, PAIR, INTER, NARROW>::kBNc)))
    return BI_ERR_CUDA;
  return launch_gemm<GATE_UP, PAIR, INTER, NARROW, GATHER, DECODE>(tmA, tmB, p, P, stream);
}

// Gate/up GEMM.  tok is the gathered copy x_perm [P, H] (GATHER = false) or
// the token matrix x [M, H] whose rows the GEMM gathers itself (GATHER).
template <bool GATHER>
static bi_status gate_up_any(const void *tok, int64_t M, const int32_t *offsets, const int32_t *perm,
                             const float *wts, const void *w13, void *act, int64_t P, int64_t H, int64_t E,
                             int32_t top_k, int64_t I, cudaStream_t stream) {
  const int v = pick_variant(I, true, H, P, E);
  if (v < 0) return BI_ERR_UNSUPPORTED;
  const bool pair = v == 2 || v == 3, inter = v == 3 || v == 4, narrow = use_narrow(P, E);
  // features per tile: 128 (one CTA), 256 (pair), 128 (pair, interleaved:
  // 64 per CTA), 64 (one CTA, interleaved)
  const int wb_rows = inter ? (pair ? kBM : kBM / 2) : (pair ? 2 * kBM : kBM);
  const uint32_t box_a = kBM;  // (interleaved tiles use the 4-D map)
  GemmParams p{offsets, perm, wts, act, (int)E, (int)H, (int)(I / wb_rows), wb_rows, (int)I,
               (int)(2 * I), (int)I, device_error_word(), (int)P, (int)top_k, nullptr, 0, nullptr, nullptr, 0};
  const int64_t wr = E * 2 * I;
  if (inter && pair)
    return narrow ? run_gemm<true, true, true, true, GATHER>(w13, wr, box_a, tok, P, H, p, stream, M)
                  : run_gemm<true, true, true, false, GATHER>(w13, wr, box_a, tok, P, H, p, stream, M);
  if (pair)
    return narrow ? run_gemm<true, true, false, true, GATHER>(w13, wr, box_a, tok, P, H, p, stream, M)
                  : run_gemm<true, true, false, false, GATHER>(w13, wr, box_a, tok, P, H, p, stream, M);
  if (inter)
    return narrow ? run_gemm<true, false, true, true, GATHER>(w13, wr, box_a, tok, P, H, p, stream, M)
                  : run_gemm<true, false, true, false, GATHER>(w13, wr, box_a, tok, P, H, p, stream, M);
  return narrow ? run_gemm<true, false, false, true, GATHER>(w13, wr, box_a, tok, P, H, p, stream, M)
                : run_gemm<true, false, false, false, GATHER>(w13, wr, box_a, tok, P, H, p, stream, M);
}

bi_status launch_gate_up(const void *x_perm, const int32_t *offsets, const int32_t *perm,
                         const float *wts, const void *w13, void *act, int64_t P, int64_t H,
                         int64_t E, int32_t top_k, int64_t I, cudaStream_t stream) {
  return gate_up_any<false>(x_perm, 0, offsets, perm, wts, w13, act, P, H, E, top_k, I, stream);
}

bi_status launch_gate_up_tokens(const void *x, int64_t M, const int32_t *offsets, const int32_t *perm,
                                const float *wts, const void *w13, void *act, int64_t H, int64_t E,
                                int32_t top_k, int64_t I, cudaStream_t stream) {
  return gate_up_any<true>(x, M, offsets, perm, wts, w13, act, M * top_k, H, E, top_k, I, stream);
}

bi_status launch_down(const void *act, const int32_t *offsets, const int32_t *perm, const void *w2,
                      float *contrib, int64_t P, int64_t H, int64_t E, int32_t top_k, int64_t I,
                      cudaStream_t stream) {
  const int v = pick_variant(H, false, I, P, E);
  if (v < 0) return BI_ERR_UNSUPPORTED;
  const bool pair = v >= 2, narrow = use_narrow(P, E);
  const int wb_rows = pair ? 2 * kBM : kBM;
  GemmParams p{offsets, perm, nullptr, contrib, (int)E, (int)I, (int)(H / wb_rows), wb_rows, (int)H,
               (int)H, 0, device_error_word(), (int)P, (int)top_k, nullptr, 0, nullptr, nullptr, 0};
  if (pair)
    return narrow ? run_gemm<false, true, false, true>(w2, E * H, kBM, act, P, I, p, stream)
                  : run_gemm<false, true, false, false>(w2, E * H, kBM, act, P, I, p, stream);
  return narrow ? run_gemm<false, false, false, true>(w2, E * H, kBM, act, P, I, p, stream)
                : run_gemm<false, false, false, false>(w2, E * H, kBM, act, P, I, p, stream);
}

// ------------------------------------------------------------- decode --
// The expert path of a decode-sized batch in two launches: gate/up (routing
// derived in every CTA, token rows gathered from x, counters zeroed) and down
// (routing derived again, the top-k combine fused).  Taken by bi_moe_forward
// for M * top_k <= kDecodeMaxP under the automatic variant choice, where
// the narrow one-CTA tiles apply anyway; same bits as the permutation,
// gather, GEMM and combine kernels (tested).
bool decode_path_ok(int64_t M, int64_t E, int32_t top_k) {
  const int64_t P = M * top_k;
  return P >= 1 && P <= kDecodeMaxP && use_narrow(P, E) && g_gemm_variant.load() == 0;
}

size_t decode_counter_count(int64_t M, int64_t H) { return static_cast<size_t>(M) * (H / 32); }

// scores non-null (bi_moe_layer): ids / wts are outputs, selected from the
// router scores inside the gate/up GEMM (E <= 512).
bi_status launch_moe_decode(const void *x, const int32_t *ids, const float *wts, const void *w13, const void *w2,
                            void *act, float *contrib, int *counters, void *out, int64_t M, int64_t H,
                            int64_t E, int32_t top_k, int64_t I, cudaStream_t stream, const float *scores = nullptr,
                            int32_t *ids_out = nullptr, float *wts_out = nullptr) {
  const int64_t P = M * top_k;
  __nv_bfloat16 *lout = static_cast<__nv_bfloat16 *>(out);
  const int v = pick_variant(I, true, H, P, E);  // narrow: 4 (interleaved 64-feature tiles) or 1
  const bool inter = v == 4;
  const int wb_rows = inter ? kBM / 2 : kBM;
  const uint32_t box_a = kBM;  // (interleaved tiles use the 4-D map)
  GemmParams g{nullptr, nullptr, wts, act, (int)E, (int)H, (int)(I / wb_rows), wb_rows, (int)I, (int)(2 * I),
               (int)I, device_error_word(), (int)P, (int)top_k, ids, (int)M, counters, lout, (int)(H / 32),
               scores, ids_out, wts_out};
  bi_status st = inter ? run_gemm<true, false, true, true, true, true>(w13, E * 2 * I, box_a, x, P, H, g, stream, M)
                       : run_gemm<true, false, false, true, true, true>(w13, E * 2 * I, box_a, x, P, H, g, stream, M);
  if (st != BI_OK) return st;
  // down reads the ids the gate/up GEMM selected (complete before it starts)
  GemmParams d{nullptr, nullptr, nullptr, contrib, (int)E, (int)I, (int)(H / kBM), kBM, (int)H, (int)H, 0,
               device_error_word(), (int)P, (int)top_k, scores ? ids_out : ids, (int)M, counters, lout,
               (int)(H / 32)};
  return run_gemm<false, false, false, true, false, true>(w2, E * H, kBM, act, P, I, d, stream);
}

// The decode-sized layer's expert path in one launch (moe_decode_layer_kernel),
// for bi_moe_layer: where the decode gate/up GEMM runs 64-feature
// interleaved tiles (their count fits one wave on the SMs), so that both
// phases share the stage layout.  The caller zeroes the combine counters
// (M * H / 32) and ready[0 .. min(E, M * top_k) * I / 64) in a kernel earlier
// on the stream (the router's).  0 = automatic, 1 = never (the two
// GEMM launches of launch_moe_decode instead).
static std::atomic<int> g_decode_fused{0};

int set_decode_fused(int mode) { return g_decode_fused.exchange(mode); }

// Gate/up tiles of the one-launch decode layer (at most): the ready counts.
int64_t decode_fused_ready_count(int64_t M, int64_t E, int32_t top_k, int64_t I) {
  return std::min<int64_t>(E, M * top_k) * (I / (kBM / 2));
}

bool decode_fused_ok(int64_t M, int64_t H, int64_t E, int32_t top_k, int64_t I) {
  const int64_t P = M * top_k;
  return g_decode_fused.load() == 0 && decode_path_ok(M, E, top_k) && pick_variant(I, true, H, P, E) == 4 &&
         decode_fused_ready_count(M, E, top_k, I) <= kDecodeReadyMax;
}

bi_status launch_moe_decode_fused(const void *x, const void *w13, const void *w2, void *act, float *contrib,
                                  int *counters, unsigned *ready, void *out, int64_t M, int64_t H, int64_t E,
                                  int32_t top_k, int64_t I, cudaStream_t stream, const float *scores,
                                  int32_t *ids_out, float *wts_out) {
  using C = GemmCfg<true, false, true, true>;
  const int64_t P = M * top_k;
  constexpr int wb_rows = kBM / 2;  // 64 interleaved gate/up features per tile
  GemmParams g{nullptr, nullptr, nullptr, act, (int)E, (int)H, (int)(I / wb_rows), wb_rows, (int)I, (int)(2 * I),
               (int)I, device_error_word(), (int)P, (int)top_k, nullptr, (int)M, counters,
               static_cast<__nv_bfloat16 *>(out), (int)(H / 32), scores, ids_out, wts_out};
  const DownPhase dn{contrib, (int)I, (int)(H / kBM), kBM, (int)H, (int)H, ready};
  CUtensorMap tmA, tmB, tmA2, tmB2;
  if (!make_tma_inter_bf16(&tmA, w13, static_cast<uint64_t>(E * 2 * I), static_cast<uint64_t>(I),
                           static_cast<uint64_t>(H)) ||
      !make_tma_2d_bf16(&tmB, x, static_cast<uint64_t>(M), static_cast<uint64_t>(H), 1u) ||
      !make_tma_2d_bf16(&tmA2, w2, static_cast<uint64_t>(E * H), static_cast<uint64_t>(I), kBM) ||
      !make_tma_2d_bf16(&tmB2, act, static_cast<uint64_t>(P), static_cast<uint64_t>(I), C::kBNc))
    return BI_ERR_CUDA;
  // At M <= 2 the router before this launch is the one-warp rows kernel,
  // which lets its dependents start at once: a ring one stage shorter (9 x
  // 20 KB) fits beside one of its CTAs, so the CTAs of this launch are
  // resident and set up before the router ends (measured on GB300: the
  // Qwen3-30B-A3B-shaped layer at M=1 0.2 us faster cold, an H=1024 / E=16
  // one at M=2 0.7 us; where the router is the cluster split schedule, the
  // shorter ring alone cost 0.3-0.5 us, so it keeps 10 stages)
  const bool beside_router = M <= 2;
  void (*kern)(CUtensorMap, CUtensorMap, GemmParams, CUtensorMap, CUtensorMap, DownPhase) =
      beside_router ? moe_decode_layer_kernel<1> : moe_decode_layer_kernel<0>;
  const int smem = C::kSmemBytes - (beside_router ? C::kStageBytes : 0);
  static std::mutex mu;
  static ContextSetup setup[2];  // the shared-memory attribute is per context
  int dev = 0;
  cudaGetDevice(&dev);
  {
    std::lock_guard<std::mutex> lk(mu);
    if (setup[beside_router].pending(dev)) {
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      int per_sm = 0;
      if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kGemmThreads, smem);
      if (e != cudaSuccess || per_sm < 1) {
        cudaGetLastError();
        set_error("decode layer kernel: cannot be resident (%s, %d per SM)", cudaGetErrorString(e), per_sm);
        return BI_ERR_CUDA;
      }
      setup[beside_router].done(dev);
    }
  }
  // CTAs wait on one another, so all must be resident: at most one per SM
  // (its shared memory allows no second), a cooperative launch
  const int64_t tiles_ub = std::min<int64_t>(P, E) * (I / wb_rows + H / kBM);
  const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(num_sms(), tiles_ub)));
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeCooperative;
  attr[1].val.cooperative = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kGemmThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, tmA, tmB, g, tmA2, tmB2, dn);
  if (e != cudaSuccess) {
    set_error("decode layer launch: %s", cudaGetErrorString(e));
    return BI_ERR_CUDA;
  }
  BI_CHECK_LAUNCH();
  return BI_OK;
}

}  // namespace bimoe
