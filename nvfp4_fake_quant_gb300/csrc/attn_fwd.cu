// Attn-QAT forward on sm_103a: two passes over the keys per 128-query tile.
//
//   pass 1: S = Q~ K~^T (tcgen05 BF16 UMMA into TMEM), m = rowmax(scale*S)
//   pass 2: S again, P = exp(scale*S - m), l += sum P, P~ = fq16(P) per 16 keys
//           (in registers, one query row per thread), P~ -> TMEM (over the S
//           columns already read) -> O += P~ V~ (tcgen05 F16 UMMA, A from TMEM)
//   epilogue: O / l -> bf16, LSE = m + ln l, m
//
// The second pass exists because P~ is referenced to the final row max m
// ("Attn-QAT Training" guide, "Architecture-specific Triton routing": exact
// statistics); a running max would quantize P against a moving reference.
// Q~, K~ (bf16) and V~ (f16, exact) are produced by the quantizer before this
// kernel.  P~ values are code * E4M3 scale <= 1.03125 with <= 6 significant
// bits and V~ values have <= 7, so both are exact in f16 and the P~V~ UMMA
// runs on f16 operands.
//
// Roles (576 threads, one CTA per SM, two 128-query tiles per CTA):
//   warps 0-15 softmax, two warpgroups per query tile (64 key columns each);
//              thread t owns query row t = TMEM lane t
//   warp 16    TMA producer
//   warp 17    TMEM allocator and UMMA issuer
// (both as converged warps, one elected lane issuing).
// Buffers: two Q~ tiles and a 5-stage K~/V~ ring in shared memory; TMEM columns
// [0,256) hold S_0, S_1 (and P~_0, P~_1 over them) and [256,512) the O_0, O_1
// accumulators.  Warpgroup hf of tile i writes the f16 pairs of its 64 keys
// into the first 32 of its own 64 S columns, which it has already loaded:
// the 16-key slice kk of P~_i is at column 128 i + 64 (kk / 4) + 8 (kk % 4).
//
// Modes (template kMode; the dense form and the auxiliary output run
// attn_fwd_fp4_kernel, so only the block-sparse mode is instantiated):
//   kDense   every key tile, one K/V load per step shared by the two query tiles
//            (the structure the block-sparse mode specialises);
//   kSparse  block-sparse: query tile i runs over its own listed key tiles, one
//            load per query tile per step; pass 1 on FP4 UMMAs.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "nvq_internal.h"
#include "nvq_ptx.cuh"
#include "nvq_quant.cuh"

namespace nvq {

namespace {

constexpr int kPairThreads = 256;  // two softmax warpgroups per query tile
constexpr int kPairWarps = 8;
constexpr int kTmaWarp = 16;
constexpr int kMmaWarp = 17;
constexpr int kThreads = 576;
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint32_t kAtomBlock = 128u * 128u;  // bytes of one 64-column block of a 128-row tile
constexpr int kDense = 0, kSparse = 1;  // forward modes

// K/V tile ring (K and V tiles interleave in pass 2): 5 slots, 4 in the
// block-sparse mode, whose two query tiles' FP4 codes take the room of the fifth.
template <int D, int kMode>
struct FwdLayout {
  static constexpr int kRing = kMode == kSparse ? 4 : 5;
  static constexpr uint32_t kTileBytes = 128u * D * 2u;
  static constexpr uint32_t kCodeBytes = 128u * D / 2;      // E2M1 codes of a 128-row tile
  static constexpr uint32_t kScBytes = (D / 64) * 512u;     // their scale blocks
  static constexpr uint32_t kC4 = (kCodeBytes + kScBytes + 1023u) / 1024u * 1024u;
  static constexpr uint32_t kQ = 0;                          // [2] query tiles
  static constexpr uint32_t kRingOff = kQ + 2u * kTileBytes;
  static constexpr uint32_t kX = kRingOff + kRing * kTileBytes;  // [2 tiles][128] f32
  // codes + scale blocks of Q~ for the FP4 pass 1 of the block-sparse mode, one
  // per query tile
  static constexpr uint32_t kQ4s = kX + 1024u;
  static constexpr uint32_t kBars = kQ4s + (kMode == kSparse ? 2u * kC4 : 0u);
  static constexpr uint32_t kNumBars = 1 + 2 * kRing + 2 * 4 + 1;
  static constexpr uint32_t kTmemSlot = kBars + kNumBars * 8u;
  static constexpr uint32_t kAbort = kTmemSlot + 4u;
  static constexpr uint32_t kUsed = kAbort + 4u;
  static constexpr uint32_t kAlloc =
      (kUsed + 1024u) > 150u * 1024u ? (kUsed + 1024u) : 150u * 1024u;
};

__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Grid: (ceil(Nq / 256), H, B).  Each CTA owns two 128-query tiles; softmax
// warpgroups 2i and 2i+1 (warps 8i..8i+7) own tile i, 64 key columns each.  TMEM: S_i at [128 i, 128 i + 128),
// O_i at [256 + 128 i, 256 + 128 i + D).  The UMMA warp ping-pongs the two
// tiles so that one warpgroup's softmax overlaps the other's UMMAs.
template <int D, int kMode>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tq4,
                    const __grid_constant__ CUtensorMap tk4, const uint8_t* __restrict__ q_sc,
                    const uint8_t* __restrict__ k_sc, __nv_bfloat16* __restrict__ o,
                    float* __restrict__ stats, int Nq, int Nkv,
                    int H, float scale, int causal, const int* __restrict__ kv_list, int topk,
                    int* __restrict__ err) {
  constexpr bool sparse = kMode == kSparse;
  constexpr int kQTiles = 2;  // query tiles per CTA
  using L = FwdLayout<D, kMode>;
  constexpr int kRing = L::kRing;
  constexpr bool fp4_pass1 = kMode == kSparse;  // pass-1 S on FP4 UMMAs
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023u) &
                                             ~static_cast<uintptr_t>(1023u));
  const int warp = threadIdx.x >> 5;
  const int h = blockIdx.y, b = blockIdx.z;
  const int q0 = blockIdx.x * kQTiles * kTile;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBars);
  uint64_t* q_full = bars + 0;
  uint64_t* r_full = bars + 1;              // [kRing]
  uint64_t* r_empty = bars + 1 + kRing;     // [kRing]
  uint64_t* s_full = bars + 1 + 2 * kRing;  // [2]
  uint64_t* s_free = s_full + 2;            // [2]
  uint64_t* p_full = s_full + 4;            // [2]
  uint64_t* o_full = s_full + 6;            // [2]
  uint64_t* mma_drain = s_full + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + L::kAbort);

  const int n_kv_all = (Nkv + kTile - 1) / kTile;
  // causal: the second query tile sees one more key tile than the first; both
  // run over it (the first tile's part of it is fully masked); block-sparse:
  // topk listed key tiles per query tile
  int n_kv;
  if (sparse) {
    n_kv = topk;
  } else {
    n_kv = causal ? min(n_kv_all, 2 * static_cast<int>(blockIdx.x) + 2) : n_kv_all;
  }

  if (threadIdx.x == 0) {
    *abort = 0;
    mbar_init(q_full, 1);
    for (int s = 0; s < kRing; ++s) {
      mbar_init(&r_full[s], 1);
      mbar_init(&r_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], kPairWarps);
      mbar_init(&p_full[i], kPairWarps);
      mbar_init(&o_full[i], 1);
    }
    mbar_init(mma_drain, 1);
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // Block-sparse: query tile i attends to the key tiles list_i[0..topk); a K or V
  // step then loads one tile per query tile.  Dense: key tile j at step j, one
  // load shared by both query tiles.
  constexpr bool per_pair = sparse;  // one K or V load per pair and step
  constexpr int nt = per_pair ? 2 : 1;      // loads per K or V step
  const int n_qt = (Nq + kTile - 1) / kTile;
  const int* list0 = nullptr;
  const int* list1 = nullptr;
  if (sparse) {
    const int qt0 = 2 * static_cast<int>(blockIdx.x);
    const int64_t base = (static_cast<int64_t>(b) * H + h) * n_qt;
    list0 = kv_list + (base + qt0) * topk;
    list1 = kv_list + (base + min(qt0 + 1, n_qt - 1)) * topk;  // a missing tile's rows are masked
  }
  auto key_tile = [&](int i, int j) -> int {
    return sparse ? (i ? list1[j] : list0[j]) : j;
  };

  if (warp == kTmaWarp) {
    // ------------------------------------------------------------ producer
    // Load order: Q0, Q1; pass 1: K(j) for every step j; pass 2: K(0), then V(j),
    // K(j+1) for every step j; K(j), V(j) are one load (dense) or one per query
    // tile (sparse), in tile order.
    tma_prefetch_desc(&tq);
    tma_prefetch_desc(&tk);
    tma_prefetch_desc(&tv);
    // Q~ codes and scale blocks for the FP4 S of pass 1 (a query tile past the
    // last one, the missing second tile of the block-sparse mode, gets zero
    // codes and no scales: its rows are never written)
    const int qt0 = static_cast<int>(blockIdx.x) * kQTiles;
    uint32_t q4_bytes = 0;
    if constexpr (fp4_pass1)
      for (int i = 0; i < kQTiles; ++i)
        q4_bytes += L::kCodeBytes + (qt0 + i < n_qt ? L::kScBytes : 0u);
    mbar_arrive_expect_tx_w(q_full, static_cast<uint32_t>(kQTiles) * L::kTileBytes + q4_bytes);
#pragma unroll
    for (int i = 0; i < kQTiles; ++i)
#pragma unroll
      for (int blk = 0; blk < D / 64; ++blk)
        tma_load_4d_w(smem + L::kQ + i * L::kTileBytes + blk * kAtomBlock, &tq, blk * 64,
                      q0 + i * kTile, h, b, q_full);
    if constexpr (fp4_pass1) {
      tma_prefetch_desc(&tq4);
      tma_prefetch_desc(&tk4);
      for (int i = 0; i < kQTiles; ++i) {
        uint8_t* q4 = smem + L::kQ4s + i * L::kC4;
        tma_load_4d_w(q4, &tq4, 0, q0 + i * kTile, h, b, q_full);
        if (qt0 + i < n_qt)
          bulk_load_w(q4 + L::kCodeBytes,
                      q_sc + ((static_cast<int64_t>(b) * H + h) * n_qt + qt0 + i) * L::kScBytes,
                      L::kScBytes, q_full);
      }
    }
    int last[kRing];
    for (int s = 0; s < kRing; ++s) last[s] = -1;
    bool ok = true;
    int li = 0;
    auto load = [&](const CUtensorMap* map, int tile) -> bool {
      const int slot = li % kRing;
      const uint32_t use = static_cast<uint32_t>(li / kRing);
      if (!mbar_wait_warp(&r_empty[slot], (use & 1u) ^ 1u, abort)) return false;
      mbar_arrive_expect_tx_w(&r_full[slot], L::kTileBytes);
#pragma unroll
      for (int blk = 0; blk < D / 64; ++blk)
        tma_load_4d_w(smem + L::kRingOff + slot * L::kTileBytes + blk * kAtomBlock, map, blk * 64,
                      tile * kTile, h, b, &r_full[slot]);
      last[slot] = static_cast<int>(use & 1u);
      ++li;
      return true;
    };
    // FP4 pass 1: K~ as codes + scale blocks (a key tile past the last one gets
    // zero codes and no scales: its scores are masked)
    auto load4 = [&](int tile) -> bool {
      const int slot = li % kRing;
      const uint32_t use = static_cast<uint32_t>(li / kRing);
      if (!mbar_wait_warp(&r_empty[slot], (use & 1u) ^ 1u, abort)) return false;
      const bool have = tile < n_kv_all;
      uint8_t* dst = smem + L::kRingOff + slot * L::kTileBytes;
      mbar_arrive_expect_tx_w(&r_full[slot], L::kCodeBytes + (have ? L::kScBytes : 0u));
      tma_load_4d_w(dst, &tk4, 0, tile * kTile, h, b, &r_full[slot]);
      if (have)
        bulk_load_w(dst + L::kCodeBytes,
                    k_sc + ((static_cast<int64_t>(b) * H + h) * n_kv_all + tile) * L::kScBytes,
                    L::kScBytes, &r_full[slot]);
      last[slot] = static_cast<int>(use & 1u);
      ++li;
      return true;
    };
    for (int j = 0; j < n_kv && ok; ++j)
      for (int i = 0; i < nt && ok; ++i)
        ok = fp4_pass1 ? load4(key_tile(i, j)) : load(&tk, key_tile(i, j));
    for (int i = 0; i < nt && ok; ++i) ok = load(&tk, key_tile(i, 0));
    for (int j = 0; j < n_kv && ok; ++j) {
      for (int i = 0; i < nt && ok; ++i) ok = load(&tv, key_tile(i, j));
      if (j + 1 < n_kv)
        for (int i = 0; i < nt && ok; ++i) ok = load(&tk, key_tile(i, j + 1));
    }
    if (!ok) {
      mbar_wait_warp(q_full, 0, nullptr, 10000000ull);
      for (int s = 0; s < kRing; ++s)
        if (last[s] >= 0) mbar_wait_warp(&r_full[s], static_cast<uint32_t>(last[s]), nullptr, 10000000ull);
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------------- MMA
    constexpr uint32_t idesc_s = idesc_f16(128, 128, 1, 0, 0);
    constexpr uint32_t idesc_pv = idesc_f16(128, D, 0, 0, 1);
    const uint32_t q_addr = smem_u32(smem + L::kQ);
    const uint32_t ring_addr = smem_u32(smem + L::kRingOff);
    int li = 0;  // ring load index being consumed
    auto wait_slot = [&](int idx) -> bool {
      return mbar_wait_warp(&r_full[idx % kRing], static_cast<uint32_t>((idx / kRing) & 1), abort);
    };
    auto issue_s = [&](int i, int idx) {  // S_i = Q~_i K~^T, K~ in ring slot of load idx
      const uint32_t kb = ring_addr + (idx % kRing) * L::kTileBytes;
      const uint32_t qb = q_addr + i * L::kTileBytes;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk >> 2) * kAtomBlock + (kk & 3) * 32;
        umma_f16_ss_w(tmem + i * 128, sdesc_sw128(qb + off, 16, 1024), sdesc_sw128(kb + off, 16, 1024),
                      idesc_s, kk > 0 ? 1u : 0u);
      }
      umma_commit_w(&s_full[i]);
    };
    // O_i += P~_i V~ with P~_i read from TMEM, V~ in the ring slot of load idx
    auto issue_pv = [&](int i, int idx, bool acc) {
      const uint32_t vb = ring_addr + (idx % kRing) * L::kTileBytes;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        umma_f16_ts_w(tmem + 256 + i * 128, tmem + i * 128 + 64 * (kk >> 2) + 8 * (kk & 3),
                      sdesc_sw128(vb + kk * 2048, kAtomBlock, 1024), idesc_pv,
                      (acc || kk > 0) ? 1u : 0u);
    };
    // Load idx of query tile i within a step whose loads start at `base`; a dense
    // load serves both tiles and is released after tile 1's UMMAs.
    auto tile_load = [&](int base, int i) { return base + (per_pair ? i : 0); };
    auto release = [&](int base, int i) {
      if (per_pair || i == 1) umma_commit_w(&r_empty[tile_load(base, i) % kRing]);
    };
    // Pass 1 of the block-sparse mode: S on block-scaled
    // FP4 UMMAs from the codes of Q~ and K~.  Pass 1 only needs the row maxima,
    // and the O columns [256, 512) are not live yet, so they hold the scale
    // operands: query tile qi's at [256 + 8 qi + 4 kk), those of pass-1 load c
    // at [272 + 8 (c % 4) + 4 kk).  A copy for load c comes after the release of
    // S_i two steps earlier, so the load that used its region last (c - 4) has
    // completed.
    constexpr uint32_t idesc_s4 = idesc_mxf4nvf4(128, 128);
    constexpr uint32_t lay4 = D == 128 ? 4u : 6u;  // (D/2)-byte swizzle of code rows
    constexpr uint32_t sbo4 = 8u * (D / 2);
    auto q4_addr = [&](int qi) { return smem_u32(smem + L::kQ4s + qi * L::kC4); };
    auto issue_s4 = [&](int i, int idx) {
      const int qi = i;  // query tile of S_i
      const uint32_t kb = ring_addr + (idx % kRing) * L::kTileBytes;
      const uint32_t sc = 272u + 8u * static_cast<uint32_t>(idx % 4);
      const uint32_t qa = q4_addr(qi);
#pragma unroll
      for (int kk = 0; kk < D / 64; ++kk)
        tmem_cp_32x128_x4_w(tmem + sc + 4 * kk, kb + L::kCodeBytes + kk * 512);
#pragma unroll
      for (int kk = 0; kk < D / 64; ++kk)
        umma_fp4_ss_w(tmem + i * 128, sdesc(qa + 32 * kk, 16, sbo4, lay4),
                      sdesc(kb + 32 * kk, 16, sbo4, lay4), idesc_s4,
                      tmem + 256 + 8 * qi + 4 * kk, tmem + sc + 4 * kk, kk > 0 ? 1u : 0u);
      umma_commit_w(&s_full[i]);
    };
    bool ok = mbar_wait_warp(q_full, 0, abort);
    if (fp4_pass1 && ok) {  // the Q~ scales stay in TMEM for pass 1
      tc_fence_after();
      for (int qi = 0; qi < kQTiles; ++qi)
#pragma unroll
        for (int kk = 0; kk < D / 64; ++kk)
          tmem_cp_32x128_x4_w(tmem + 256 + 8 * qi + 4 * kk, q4_addr(qi) + L::kCodeBytes + kk * 512);
    }
    // pass 1: S_0(j), S_1(j) for the row maxima
    for (int j = 0; j < n_kv && ok; ++j, li += nt) {
      for (int i = 0; i < 2 && ok; ++i) {
        if ((per_pair || i == 0) && !(ok = wait_slot(tile_load(li, i)))) break;
        if (j > 0 && !(ok = mbar_wait_warp(&s_free[i], static_cast<uint32_t>((j - 1) & 1), abort))) break;
        tc_fence_after();
        if constexpr (fp4_pass1) {
          issue_s4(i, tile_load(li, i));
        } else {
          issue_s(i, tile_load(li, i));
        }
        release(li, i);
      }
    }
    // pass 2 prologue: S_0(0), S_1(0)
    for (int i = 0; i < 2 && ok; ++i) {
      if ((per_pair || i == 0) && !(ok = wait_slot(tile_load(li, i)))) break;
      if (!(ok = mbar_wait_warp(&s_free[i], static_cast<uint32_t>((n_kv - 1) & 1), abort))) break;
      tc_fence_after();
      issue_s(i, tile_load(li, i));
      release(li, i);
    }
    li += nt;
    for (int j = 0; j < n_kv && ok; ++j) {
      const int vbase = li;  // V(j)
      li += nt;
      const int kbase = (j + 1 < n_kv) ? li : -1;  // K(j+1)
      if (kbase >= 0) li += nt;
      for (int i = 0; i < 2 && ok; ++i) {
        if ((per_pair || i == 0) && !(ok = wait_slot(tile_load(vbase, i)))) break;
        if (!(ok = mbar_wait_warp(&p_full[i], static_cast<uint32_t>(j & 1), abort))) break;
        tc_fence_after();
        issue_pv(i, tile_load(vbase, i), j > 0);
        release(vbase, i);
        if (kbase >= 0) {
          if ((per_pair || i == 0) && !(ok = wait_slot(tile_load(kbase, i)))) break;
          // S_i(j+1): S_i was read before p_full_i(j), and the UMMAs run in
          // issue order, so PV_i(j) reads P~_i before S_i(j+1) overwrites it
          issue_s(i, tile_load(kbase, i));
          release(kbase, i);
        }
      }
    }
    if (ok) {
      umma_commit_w(&o_full[0]);
      umma_commit_w(&o_full[1]);
    }
    umma_commit_w(mma_drain);
    mbar_wait_warp(mma_drain, 0, nullptr, 10000000ull);
  } else {
    // ------------------------------------------------------------ softmax
    // Warpgroups 2i and 2i+1 own query tile i; half `hf` of the pair owns key
    // columns [64 hf, 64 hf + 64) of S_i and O columns [hf D/2, (hf+1) D/2).
    // Row maxima and sums are combined across the pair through shared memory.
    const int wg = warp >> 2;
    const int ti = wg >> 1;                // query tile
    const int hf = wg & 1;                 // half of the key columns
    const int t = threadIdx.x & 127;       // row in the tile == TMEM lane
    const int tile_q0 = q0 + ti * kTile;
    const int qrow = tile_q0 + t;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t s_col = static_cast<uint32_t>(ti * 128 + hf * 64);
    const float c1 = scale * kLog2e;
    // half 1 posts its partial, half 0 combines and posts the result back
    float* xchg = reinterpret_cast<float*>(smem + L::kX) + ti * 128;
    const uint32_t pair_bar = 1u + static_cast<uint32_t>(ti);
    bool ok = true;
    float mraw = -INFINITY;
    uint32_t r[32];
    for (int j = 0; j < n_kv && ok; ++j) {
      if (!(ok = mbar_wait_warp(&s_full[ti], static_cast<uint32_t>(j & 1), abort))) break;
      tc_fence_after();
      const int kt = key_tile(ti, j);
      const bool edge = kt < 0 || (kt * kTile + kTile > Nkv) || (causal && kt * kTile + kTile - 1 > tile_q0);
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        tmem_ld32(tmem + lane_base + s_col + c * 32, r);
        tmem_wait_ld();
        if (!edge) {
#pragma unroll
          for (int i = 0; i < 32; i += 2) mraw = max3(mraw, __uint_as_float(r[i]), __uint_as_float(r[i + 1]));
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int key = kt * kTile + hf * 64 + c * 32 + i;
            if (key >= 0 && key < Nkv && (!causal || key <= qrow)) mraw = fmaxf(mraw, __uint_as_float(r[i]));
          }
        }
      }
      tc_fence_before();
      mbar_arrive_warp(&s_free[ti]);
    }
    // combine the row maxima of the pair (always reached, also after an abort)
    if (hf == 1) xchg[t] = mraw;
    named_bar_sync(pair_bar, kPairThreads);
    if (hf == 0) xchg[t] = mraw = fmaxf(mraw, xchg[t]);
    named_bar_sync(pair_bar, kPairThreads);
    if (hf == 1) mraw = xchg[t];
    const float m = mraw * scale;
    const float negmb = -m * kLog2e;
    const uint64_t c12 = pk2(c1, c1), nmb2 = pk2(negmb, negmb);
    uint64_t l2 = pk2(0.f, 0.f);
    for (int j = 0; j < n_kv && ok; ++j) {
      if (!(ok = mbar_wait_warp(&s_full[ti], static_cast<uint32_t>((n_kv + j) & 1), abort))) break;
      tc_fence_after();
      // S_i(j) complete implies PV_i(j-1) complete (issued earlier): P~_i(j-1) is consumed
      const int kt = key_tile(ti, j);
      const bool edge = kt < 0 || (kt * kTile + kTile > Nkv) || (causal && kt * kTile + kTile - 1 > tile_q0);
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        tmem_ld32(tmem + lane_base + s_col + c * 32, r);
        tmem_wait_ld();
        float x[32];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          up2(fma2(pk2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])), c12, nmb2),
              x[2 * i], x[2 * i + 1]);
        if (edge) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int key = kt * kTile + hf * 64 + c * 32 + i;
            if (!(key >= 0 && key < Nkv && (!causal || key <= qrow))) x[i] = -INFINITY;
          }
        }
        uint32_t pt[16];  // P~ of these 32 keys as f16 pairs
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
          float pp[16];
          uint32_t (&ph)[8] = *reinterpret_cast<uint32_t(*)[8]>(pt + 8 * hb);
          pquant16_pmax(x + 16 * hb, pp, ph);
#pragma unroll
          for (int u = 0; u < 8; ++u) l2 = add2(l2, pk2(pp[2 * u], pp[2 * u + 1]));
        }
        // keys [64 hf + 32 c, +32) -> columns [64 hf + 16 c, +16) of S_i, already loaded
        tmem_st16(tmem + lane_base + s_col + c * 16, pt);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive_warp(&p_full[ti]);
    }
    float l_lo, l_hi;
    up2(l2, l_lo, l_hi);
    float l = l_lo + l_hi;
    const bool have_o = ok && mbar_wait_warp(&o_full[ti], 0, abort);
    if (hf == 1) xchg[t] = l;
    named_bar_sync(pair_bar, kPairThreads);
    if (hf == 0) xchg[t] = l = l + xchg[t];
    named_bar_sync(pair_bar, kPairThreads);
    if (hf == 1) l = xchg[t];
    if (have_o) {
      tc_fence_after();
      const float inv_l = 1.0f / l;
      __nv_bfloat16* orow = o + ((static_cast<int64_t>(b) * Nq + qrow) * H + h) * D + hf * (D / 2);
      const uint32_t o_col = 256u + static_cast<uint32_t>(ti * 128 + hf * (D / 2));
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        tmem_ld32(tmem + lane_base + o_col + c * 32, r);
        tmem_wait_ld();
        if (qrow < Nq) {
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            __nv_bfloat162 v2 = __floats2bfloat162_rn(__uint_as_float(r[2 * i]) * inv_l,
                                                      __uint_as_float(r[2 * i + 1]) * inv_l);
            w[i] = *reinterpret_cast<uint32_t*>(&v2);
          }
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int u = 0; u < 4; ++u)
            dst[u] = make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
        }
      }
      if (qrow < Nq && hf == 0) {
        float* st = stats + (static_cast<int64_t>(b) * H + h) * 2 * Nq;
        st[qrow] = m + logf(l);
        st[Nq + qrow] = m;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  report_abort(abort, err);
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

template <int D>
cudaError_t launch_sparse_d(const AttnShape& s, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, const CUtensorMap& tq4, const CUtensorMap& tk4,
                            const uint8_t* q_sc, const uint8_t* k_sc, void* o, float* stats,
                            const int* kv_list, int topk, int* err, cudaStream_t stream) {
  using L = FwdLayout<D, kSparse>;
  const int q_per_cta = 2 * kTile;
  const dim3 grid((s.Nq + q_per_cta - 1) / q_per_cta, s.H, s.B);
  cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel<D, kSparse>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (e != cudaSuccess) return e;
  attn_fwd_kernel<D, kSparse><<<grid, kThreads, L::kAlloc, stream>>>(
      tq, tk, tv, tq4, tk4, q_sc, k_sc, static_cast<__nv_bfloat16*>(o), stats, s.Nq, s.Nkv, s.H,
      s.scale, s.causal, kv_list, topk, err);
  return cudaGetLastError();
}

cudaError_t launch_attn_fwd(const AttnShape& s, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, const CUtensorMap& tq4, const CUtensorMap& tk4,
                            const uint8_t* q_sc, const uint8_t* k_sc, void* o, float* stats,
                            const int* kv_list, int topk, int* err, cudaStream_t stream) {
  if (kv_list == nullptr || q_sc == nullptr || k_sc == nullptr) return cudaErrorInvalidValue;
  return s.D == 128 ? launch_sparse_d<128>(s, tq, tk, tv, tq4, tk4, q_sc, k_sc, o, stats,
                                           kv_list, topk, err, stream)
                    : launch_sparse_d<64>(s, tq, tk, tv, tq4, tk4, q_sc, k_sc, o, stats, kv_list,
                                          topk, err, stream);
}

}  // namespace nvq
