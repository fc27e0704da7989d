// Attn-QAT forward with S = Q~ K~^T on block-scaled FP4 UMMAs (sm_103a).
//
// The same two passes as the BF16 forward ("Attn-QAT Training" guide,
// "Architecture-specific Triton routing": statistics against the final row
// max), computing the same values:
//   pass 1: S = Q~ K~^T, m = rowmax(scale*S)
//   pass 2: S again, P = exp(scale*S - m), l += sum P, P~ = fq16(P) per 16 keys,
//           O += P~ V~ (F16 UMMA, P~ read from TMEM)
//   epilogue: O / l -> bf16, LSE = m + ln l, m.
// Q~ and K~ arrive as packed E2M1 codes with their E4M3 scales per 16 elements
// of D (the quantizer's outputs); the kind::mxf4nvf4 UMMA multiplies the codes
// and applies both scales, so each S element is the sum of the same exact
// products code_q*s_q*code_k*s_k that a BF16 UMMA on Q~, K~ would add up.
//
// One 128-query tile per CTA.  S tiles live in TMEM buffers of 128 columns:
// three in pass 1 (columns [0, 384); O is not live yet, tile j in buffer
// j % 3), two in pass 2 (columns [0, 256), tile j in buffer j % 2), so the
// UMMAs of the next tiles run while the softmax works on the current one.  In
// pass 1 warpgroup w takes the whole tiles j = w (mod 4): four tiles are read
// at once, and each tile costs one wait and one release per warp of one
// warpgroup instead of all sixteen warps.  In pass 2 the four warpgroups share
// every tile, warpgroup w owning keys [32 w, 32 w + 32) of it; P~ of a tile is
// written over the first 16 of each warpgroup's 32 columns, which it has
// already loaded, and P~V~ reads it from there.
//
// Every tcgen05 instruction and every mbarrier wait costs the issuing warp tens
// of cycles, more in total than the tensor work of the small FP4 UMMAs, so the
// UMMAs come from two warps: the S warp (the even pass-1 tiles and every
// pass-2 S, with their scale copies) and the PV warp (the odd pass-1 tiles,
// then P~V~).  Before the S warp overwrites a pass-2 buffer
// it waits for the PV warp's commit of the P~V~ that read the buffer.
//
// TMEM: S buffers, O at [256, 256 + D) (pass 2), the Q~ scale operand at
// [384 + 4 kk), the K~ scale operand of tile counter g at [392 + 8 (g % 12) +
// 4 kk) (kk: 64-element group of D).  The issuing warp copies a tile's scales
// before it waits for the tile's S buffer, so the copy is off the path from
// "buffer released" to "UMMA running".  Twelve copies rotate, and a copy never
// overwrites scales an UMMA in flight may still read.  Pass 1: the warp
// copying the scales of tile g fired tile g - 4 after the release of tile
// g - 7, whose S the other warp fired after the release of tile g - 10, a
// tile of this warp fired after its tile g - 12; so tile g - 12, the region's
// last reader, has completed.  Pass 2: the S warp has waited for the P~V~ of
// the tile before, which follows the softmax of tile g - 4, and pass 2 starts
// after every pass-1 tile has been read.
//
// Pass-1 barriers are indexed so that every barrier is waited on by one role
// in phase order (an mbarrier parity wait cannot tell a phase from the one two
// ahead): s1_full[j % 12] (waited by warpgroup j % 4 only), s1_free[j % 6]
// (waited by the issuer of tile j + 3 only), and one pass1_done barrier the
// softmax warps arrive on after their last pass-1 tile.
//
// Roles (608 threads, one CTA per SM): warps 0-15 softmax, warp 16 TMA
// producer, warp 17 TMEM allocator and S issuer, warp 18 P~V~ issuer
// (converged warps, one elected lane issuing).  Shared memory: Q~ codes and
// scales, a ring of K~ tiles (codes + scales), a ring of V~ tiles (f16).
//
// Auxiliary-output form (kAux; the "auxiliary output" of the Attn-QAT
// backward, "use_high_prec_o"): next to O it accumulates O_hp = P V~ / l from
// the unquantized P (f16).  O_hp takes the TMEM columns [256 + D, 256 + 2 D),
// so pass 2 runs on half tiles of 64 keys: half u (keys [64 (u % 2), +64) of
// tile u / 2) is one N = 64 UMMA pair into buffer u % 3 of three 64-column
// buffers [0, 192); warpgroup w owns keys [16 w, 16 w + 16) of every half and
// writes, over the 16 columns it has loaded, P~ (f16 pairs) into the first 8
// and P into the next 8.  The P~V~ warp adds both into O and O_hp.  The Q~
// scale operand of pass 2 sits at [192, 192 + D/16) (pass 1's copy is under
// O_hp), the K~ scale operand of pass-2 tile j at [200 + 8 (j % 4), +8); a
// half reads the scale columns of its 64 keys, 2 (u % 2) columns in (key n of
// a 128-key region is at column n / 32).  Pass 1 is unchanged.
//
// Block-sparse form (kSparseFwd; the "VSA" fine branch, "vsqa-preview-1.3b
// metadata.json", attention.selection): step j of both passes visits key tile
// list[j] of the query tile's topk selected tiles instead of tile j; the TMA
// warp loads the listed tiles, nothing else changes (the sparse calls take
// N % 128 == 0 and no causal mask, so no listed key is masked).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "nvq_internal.h"
#include "nvq_ptx.cuh"
#include "nvq_quant.cuh"

namespace nvq {

namespace {

constexpr int kThreads = 608;
constexpr int kSoftmaxWarps = 16;
constexpr int kTmaWarp = 16;
constexpr int kSWarp = 17;
constexpr int kPvWarp = 18;
constexpr int kKRing = 6;
constexpr int kVRing = 4;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kDenseFwd = 0, kAuxFwd = 1, kSparseFwd = 2;  // kernel modes
constexpr uint32_t kScA = 384, kScB = 392;  // TMEM columns of the scale operands
constexpr int kScRegions = 12;               // K~ scale copies at kScB + 8 r, up to 488
// auxiliary-output pass 2: the Q~ scale operand and four K~ scale regions
constexpr uint32_t kScA2 = 192, kScB2 = 200;
constexpr int kScRegions2 = 4;

template <int D>
struct Fp4Layout {
  static constexpr uint32_t kCodeBytes = 128u * D / 2;   // codes of a 128-row tile
  static constexpr uint32_t kScBytes = (D / 64) * 512u;  // its scale blocks
  static constexpr uint32_t kKSlot = (kCodeBytes + kScBytes + 1023u) / 1024u * 1024u;
  static constexpr uint32_t kVSlot = 128u * D * 2u;
  static constexpr uint32_t kQ = 0;
  static constexpr uint32_t kKRingOff = kKSlot;  // the Q~ tile takes one K~ slot's room
  static constexpr uint32_t kVRingOff = kKRingOff + kKRing * kKSlot;
  static constexpr uint32_t kX = kVRingOff + kVRing * kVSlot;  // [4 warpgroups][128] f32
  static constexpr uint32_t kBars = kX + 4u * 128u * 4u;
  // q_full, k_full/k_empty, v_full/v_empty, s1_full[12], s1_free[6], pass1_done,
  // s_full[3], p_full[3], pv_done[3] (two of each without the auxiliary output),
  // o_full, drain x2, q_sc_ready
  static constexpr uint32_t kNumBars = 1 + 2 * kKRing + 2 * kVRing + 12 + 6 + 1 + 9 + 4;
  static constexpr uint32_t kTmemSlot = kBars + kNumBars * 8u;
  static constexpr uint32_t kAbort = kTmemSlot + 4u;
  static constexpr uint32_t kAlloc = kAbort + 4u + 1024u;
};

// Grid: (ceil(Nq / 128), H, B).  kMode: kDenseFwd, kAuxFwd (o_hp) or
// kSparseFwd (kv_list: int32 [B, H, ceil(Nq/128), topk], the key tiles of each
// query tile, in the order they are visited).
template <int D, int kMode>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_fp4_kernel(const __grid_constant__ CUtensorMap tq,
                        const __grid_constant__ CUtensorMap tk,
                        const __grid_constant__ CUtensorMap tv, const uint8_t* __restrict__ q_sc,
                        const uint8_t* __restrict__ k_sc, __nv_bfloat16* __restrict__ o,
                        __nv_bfloat16* __restrict__ o_hp, float* __restrict__ stats, int Nq,
                        int Nkv, int H, float scale, int causal,
                        const int* __restrict__ kv_list, int topk, int* __restrict__ err) {
  constexpr bool kAux = kMode == kAuxFwd;
  constexpr bool kSparse = kMode == kSparseFwd;
  using L = Fp4Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023u) &
                                             ~static_cast<uintptr_t>(1023u));
  const int warp = threadIdx.x >> 5;
  const int h = blockIdx.y, b = blockIdx.z;
  const int qt = blockIdx.x;
  const int q0 = qt * kTile;
  const int64_t bh = static_cast<int64_t>(b) * H + h;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBars);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;           // [kKRing]
  uint64_t* k_empty = k_full + kKRing;   // [kKRing]
  uint64_t* v_full = k_empty + kKRing;   // [kVRing]
  uint64_t* v_empty = v_full + kVRing;   // [kVRing]
  uint64_t* s1_full = v_empty + kVRing;  // pass 1 [12]: tile j -> j % 12
  uint64_t* s1_free = s1_full + 12;      // pass 1 [6]: tile j -> j % 6
  uint64_t* pass1_done = s1_free + 6;
  uint64_t* s_full = pass1_done + 1;     // pass 2 [3]
  uint64_t* p_full = s_full + 3;         // pass 2 [3]
  uint64_t* pv_done = p_full + 3;        // pass 2 [3]
  uint64_t* o_full = pv_done + 3;
  uint64_t* drain = o_full + 1;          // [2]: S warp, PV warp
  uint64_t* q_sc_ready = drain + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + L::kAbort);

  const int n_kt = (Nkv + kTile - 1) / kTile;
  const int n_qt = (Nq + kTile - 1) / kTile;
  // key tiles this query tile sees (causal: up to its diagonal tile;
  // block-sparse: its topk listed tiles, step j visiting tile list[j])
  const int nk = kSparse ? topk : causal ? min(n_kt, qt + 1) : n_kt;
  const int* list = kSparse ? kv_list + (bh * n_qt + qt) * topk : nullptr;

  if (threadIdx.x == 0) {
    *abort = 0;
    mbar_init(q_full, 1);
    for (int s = 0; s < kKRing; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < kVRing; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int i = 0; i < 12; ++i) mbar_init(&s1_full[i], 1);
    for (int i = 0; i < 6; ++i) mbar_init(&s1_free[i], kSoftmaxWarps / 4);
    mbar_init(pass1_done, kSoftmaxWarps);
    for (int i = 0; i < 3; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], kSoftmaxWarps);
      mbar_init(&pv_done[i], 1);
    }
    mbar_init(&drain[0], 1);
    mbar_init(&drain[1], 1);
    mbar_init(o_full, 1);
    mbar_init(q_sc_ready, 1);
    fence_mbar_init();
  }
  if (warp == kSWarp) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // S into TMEM column `col` = Q~ K~^T for K~ load `kl` (loads are numbered in
  // the producer's order), tile counter g (which scale copy), completion on
  // `bar`; the K~ slot is released after the UMMAs.  Issued by a converged warp.
  constexpr uint32_t idesc_s = idesc_mxf4nvf4(128, 128);
  constexpr uint32_t lay = D == 128 ? 4u : 6u;  // (D/2)-byte swizzle of the code rows
  constexpr uint32_t sbo = 8u * (D / 2);
  const uint32_t q_addr = smem_u32(smem + L::kQ);
  const uint32_t k_ring = smem_u32(smem + L::kKRingOff);
  // the K~ scale region of tile counter g
  auto sc_region = [&](int g) { return kScB + 8u * static_cast<uint32_t>(g % kScRegions); };
  // prep_s: wait for the K~ tile of load kl and copy its scales into TMEM column sc
  auto prep_s = [&](int kl, uint32_t sc) -> bool {
    const int slot = kl % kKRing;
    if (!mbar_wait_warp(&k_full[slot], static_cast<uint32_t>((kl / kKRing) & 1), abort))
      return false;
    tc_fence_after();
    const uint32_t kb = k_ring + slot * L::kKSlot;
#pragma unroll
    for (int kk = 0; kk < D / 64; ++kk)
      tmem_cp_32x128_x4_w(tmem + sc + 4 * kk, kb + L::kCodeBytes + kk * 512);
    return true;
  };
  // Descriptors of the Q~ codes (fixed) and of a K~ slot's codes: a 64-element
  // K step is 32 bytes on (2 in the descriptor's start-address field).
  uint64_t q_d[D / 64];
#pragma unroll
  for (int kk = 0; kk < D / 64; ++kk) q_d[kk] = sdesc(q_addr + 32 * kk, 16, sbo, lay);
  auto k_desc = [&](uint32_t kb, uint64_t (&kd)[D / 64]) {
    kd[0] = sdesc(kb, 16, sbo, lay);
    if constexpr (D == 128) kd[1] = kd[0] + 2;
  };
  // fire_s: the UMMAs of a prepared tile (after its S buffer is free) and their
  // commits as one group; the K~ slot is released by a commit here in pass 2,
  // by the softmax in pass 1
  auto fire_s = [&](uint32_t col, int kl, int g, uint64_t* bar) {
    const int slot = kl % kKRing;
    uint64_t kd[D / 64];
    k_desc(k_ring + slot * L::kKSlot, kd);
    umma_fp4_group_w<D / 64>(tmem + col, q_d, kd, idesc_s, tmem + kScA, tmem + sc_region(g),
                             bar_u32(bar), g >= nk ? bar_u32(&k_empty[slot]) : 0u);
  };
  // Auxiliary output, pass 2: half hh (keys [64 hh, 64 hh + 64)) of the K~ tile
  // of load kl into the 64-column buffer at `col`; the tile's scales at column sc
  constexpr uint32_t idesc_h = idesc_mxf4nvf4(128, 64);
  auto fire_half = [&](uint32_t col, int kl, uint32_t sc, int hh, uint64_t* bar) {
    const int slot = kl % kKRing;
    uint64_t kd[D / 64];
    k_desc(k_ring + slot * L::kKSlot + static_cast<uint32_t>(hh) * 64u * (D / 2), kd);
    umma_fp4_group_w<D / 64>(tmem + col, q_d, kd, idesc_h, tmem + kScA2,
                             tmem + sc + 2 * static_cast<uint32_t>(hh), bar_u32(bar),
                             hh == 1 ? bar_u32(&k_empty[slot]) : 0u);
  };
  // Pass 1, tile j (load j) into buffer j % 3 once the softmax has loaded tile
  // j - 3 from there.  The S warp takes the even tiles, the P~V~ warp (idle
  // until pass 2) the odd ones.
  auto pass1 = [&](int first) -> bool {
    bool ok = true;
    for (int j = first; j < nk && ok; j += 2) {
      if (!(ok = prep_s(j, sc_region(j)))) break;
      if (j >= 3 && !(ok = mbar_wait_warp(&s1_free[(j - 3) % 6],
                                          static_cast<uint32_t>(((j - 3) / 6) & 1), abort)))
        break;
      tc_fence_after();
      fire_s(128u * (j % 3), j, j, &s1_full[j % 12]);
    }
    return ok;
  };

  if (warp == kTmaWarp) {
    // ------------------------------------------------------------ producer
    // Q~; pass 1: K(j) for every tile j; pass 2: K(0), K(1), then per tile
    // V(j) and K(j + 2) (the order the two UMMA warps first use them in).
    tma_prefetch_desc(&tq);
    tma_prefetch_desc(&tk);
    tma_prefetch_desc(&tv);
    mbar_arrive_expect_tx_w(q_full, L::kCodeBytes + L::kScBytes);
    tma_load_4d_w(smem + L::kQ, &tq, 0, q0, h, b, q_full);
    bulk_load_w(smem + L::kQ + L::kCodeBytes, q_sc + (bh * n_qt + qt) * L::kScBytes, L::kScBytes,
                q_full);
    int k_last[kKRing], v_last[kVRing];
    for (int s = 0; s < kKRing; ++s) k_last[s] = -1;
    for (int s = 0; s < kVRing; ++s) v_last[s] = -1;
    int kli = 0, vli = 0;
    bool ok = true;
    // key tile of step j (a listed tile outside [0, n_kt), which the caller must
    // not pass, reads zero codes and no scales instead of memory it does not own)
    auto tile_of = [&](int j) { return kSparse ? __ldg(list + j) : j; };
    auto load_k = [&](int tile) -> bool {
      const int slot = kli % kKRing;
      const uint32_t use = static_cast<uint32_t>(kli / kKRing);
      if (!mbar_wait_warp(&k_empty[slot], (use & 1u) ^ 1u, abort)) return false;
      uint8_t* dst = smem + L::kKRingOff + slot * L::kKSlot;
      const bool have = !kSparse || (tile >= 0 && tile < n_kt);
      mbar_arrive_expect_tx_w(&k_full[slot], L::kCodeBytes + (have ? L::kScBytes : 0u));
      tma_load_4d_w(dst, &tk, 0, tile * kTile, h, b, &k_full[slot]);
      if (have)
        bulk_load_w(dst + L::kCodeBytes, k_sc + (bh * n_kt + tile) * L::kScBytes, L::kScBytes,
                    &k_full[slot]);
      k_last[slot] = static_cast<int>(use & 1u);
      ++kli;
      return true;
    };
    auto load_v = [&](int tile) -> bool {
      const int slot = vli % kVRing;
      const uint32_t use = static_cast<uint32_t>(vli / kVRing);
      if (!mbar_wait_warp(&v_empty[slot], (use & 1u) ^ 1u, abort)) return false;
      uint8_t* dst = smem + L::kVRingOff + slot * L::kVSlot;
      mbar_arrive_expect_tx_w(&v_full[slot], L::kVSlot);
#pragma unroll
      for (int blk = 0; blk < D / 64; ++blk)
        tma_load_4d_w(dst + blk * (128u * 128u), &tv, blk * 64, tile * kTile, h, b, &v_full[slot]);
      v_last[slot] = static_cast<int>(use & 1u);
      ++vli;
      return true;
    };
    for (int j = 0; j < nk && ok; ++j) ok = load_k(tile_of(j));
    for (int j = 0; j < 2 && j < nk && ok; ++j) ok = load_k(tile_of(j));
    for (int j = 0; j < nk && ok; ++j) {
      ok = load_v(tile_of(j));
      if (ok && j + 2 < nk) ok = load_k(tile_of(j + 2));
    }
    if (!ok) {  // let the copies in flight land before the block exits
      mbar_wait_warp(q_full, 0, nullptr, 10000000ull);
      for (int s = 0; s < kKRing; ++s)
        if (k_last[s] >= 0)
          mbar_wait_warp(&k_full[s], static_cast<uint32_t>(k_last[s]), nullptr, 10000000ull);
      for (int s = 0; s < kVRing; ++s)
        if (v_last[s] >= 0)
          mbar_wait_warp(&v_full[s], static_cast<uint32_t>(v_last[s]), nullptr, 10000000ull);
    }
  } else if (warp == kSWarp) {
    // ------------------------------------------------------------ S issuer
    bool ok = mbar_wait_warp(q_full, 0, abort);
    if (ok) {  // the Q~ scales stay in TMEM for the whole kernel
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < D / 64; ++kk)
        tmem_cp_32x128_x4_w(tmem + kScA + 4 * kk, q_addr + L::kCodeBytes + kk * 512);
      // the P~V~ warp issues S UMMAs that read them: signal the copy's completion
      umma_commit_w(q_sc_ready);
    }
    if (ok) ok = pass1(0);
    // every pass-1 tile loaded by the softmax (pass 2 reuses the columns)
    if (ok) ok = mbar_wait_warp(pass1_done, 0, abort);
    if constexpr (!kAux) {
      // Pass 2 (tile counter g = nk + j): tiles 0 and 1 at once, then tile j + 2
      // into buffer j % 2 once the P~V~ of tile j, the last reader of its P~, is done.
      for (int j = 0; j < 2 && j < nk && ok; ++j) {
        if (!(ok = prep_s(nk + j, sc_region(nk + j)))) break;
        fire_s(128u * j, nk + j, nk + j, &s_full[j]);
      }
      for (int j = 0; j + 2 < nk && ok; ++j) {
        const int buf = j & 1;
        if (!(ok = prep_s(nk + j + 2, sc_region(nk + j + 2)))) break;
        if (!(ok = mbar_wait_warp(&pv_done[buf], static_cast<uint32_t>((j >> 1) & 1), abort)))
          break;
        tc_fence_after();
        fire_s(128u * buf, nk + j + 2, nk + j + 2, &s_full[buf]);
      }
    } else {
      // Pass 2 on half tiles: the Q~ scales again (pass 1's copy lies under
      // O_hp), then half u into buffer u % 3 once the P~V~ of half u - 3, the
      // last reader of that buffer, is done.  A tile's K~ scales are copied at
      // its first half into region j % 4: the copy for tile j follows the wait
      // for the P~V~ of half 2 j - 4, so the S UMMAs of tile j - 2 and before,
      // the last readers of the region, have completed.
      if (ok) {
#pragma unroll
        for (int kk = 0; kk < D / 64; ++kk)
          tmem_cp_32x128_x4_w(tmem + kScA2 + 4 * kk, q_addr + L::kCodeBytes + kk * 512);
      }
      for (int u = 0; u < 2 * nk && ok; ++u) {
        const int j = u >> 1, hh = u & 1, c = u % 3;
        const uint32_t sc = kScB2 + 8u * static_cast<uint32_t>(j % kScRegions2);
        if (hh == 0 && !(ok = prep_s(nk + j, sc))) break;
        if (u >= 3 &&
            !(ok = mbar_wait_warp(&pv_done[c], static_cast<uint32_t>(((u - 3) / 3) & 1), abort)))
          break;
        tc_fence_after();
        fire_half(64u * c, nk + j, sc, hh, &s_full[c]);
      }
    }
    umma_commit_w(&drain[0]);
    mbar_wait_warp(&drain[0], 0, nullptr, 10000000ull);
  } else if (warp == kPvWarp) {
    // ------------------------------------------------------------ P~V~ issuer
    constexpr uint32_t idesc_pv = idesc_f16(128, D, 0, 0, 1);
    const uint32_t v_ring = smem_u32(smem + L::kVRingOff);
    // V~ slot s: descriptor of its first 16 keys, 2048 * s on from slot 0's
    const uint64_t v_d0 = sdesc_sw128(v_ring, 128u * 128u, 1024);
    auto v_desc = [&](int slot) { return v_d0 + static_cast<uint64_t>(slot) * (L::kVSlot >> 4); };
    // the Q~ scale copy (S warp) precedes the odd pass-1 tiles' UMMAs
    bool ok = mbar_wait_warp(q_sc_ready, 0, abort);
    if (ok) {
      tc_fence_after();
      ok = pass1(1);
    }
    for (int j = 0; j < nk && ok && !kAux; ++j) {
      const int buf = j & 1, slot = j % kVRing;
      if (!(ok = mbar_wait_warp(&v_full[slot], static_cast<uint32_t>((j / kVRing) & 1), abort))) break;
      if (!(ok = mbar_wait_warp(&p_full[buf], static_cast<uint32_t>((j >> 1) & 1), abort))) break;
      tc_fence_after();
      // keys [16 kk, 16 kk + 16): warpgroup kk / 2, its P~ columns 8 (kk % 2)
      uint32_t a[8];
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        a[kk] = tmem + 128u * static_cast<uint32_t>(buf) + 32 * (kk >> 1) + 8 * (kk & 1);
      umma_f16_ts8_w(tmem + 256, a, v_desc(slot), idesc_pv, j > 0 ? 1u : 0u,
                     bar_u32(&pv_done[buf]), bar_u32(&v_empty[slot]));
    }
    // auxiliary output: per half u, keys [64 hh + 16 w, +16) from warpgroup w's
    // columns of buffer u % 3, P~ into O and P into O_hp
    for (int u = 0; u < 2 * nk && ok && kAux; ++u) {
      const int j = u >> 1, hh = u & 1, c = u % 3, slot = j % kVRing;
      if (hh == 0 &&
          !(ok = mbar_wait_warp(&v_full[slot], static_cast<uint32_t>((j / kVRing) & 1), abort)))
        break;
      if (!(ok = mbar_wait_warp(&p_full[c], static_cast<uint32_t>((u / 3) & 1), abort))) break;
      tc_fence_after();
      uint32_t a[4];
#pragma unroll
      for (int w = 0; w < 4; ++w) a[w] = tmem + 64u * static_cast<uint32_t>(c) + 16 * w;
      umma_f16_ts4x2_w(tmem + 256, tmem + 256 + D, a, v_desc(slot) + 512u * hh, idesc_pv,
                       u > 0 ? 1u : 0u, bar_u32(&pv_done[c]),
                       hh == 1 ? bar_u32(&v_empty[slot]) : 0u);
    }
    if (ok) umma_commit_w(o_full);
    umma_commit_w(&drain[1]);
    mbar_wait_warp(&drain[1], 0, nullptr, 10000000ull);
  } else if (warp < kSoftmaxWarps) {
    // ------------------------------------------------------------ softmax
    const int wg = warp >> 2;            // keys [32 wg, 32 wg + 32) of every tile
    const int t = threadIdx.x & 127;     // query row in the tile == TMEM lane
    const int qrow = q0 + t;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const float c1 = scale * kLog2e;
    float* xchg = reinterpret_cast<float*>(smem + L::kX);  // [4][128]
    auto key0 = [&](int j) { return j * kTile + 32 * wg; };
    auto is_edge = [&](int k0) { return k0 + 32 > Nkv || (causal && k0 + 31 > q0); };
    bool ok = true;
    float mraw = -INFINITY;
    uint32_t r[32];
    {
      // pass 1: warpgroup wg, tiles j = wg (mod 4), all 128 keys of each
      uint32_t r2[32];
      for (int j = wg; j < nk && ok; j += 4) {
        if (!(ok = mbar_wait_warp(&s1_full[j % 12], static_cast<uint32_t>((j / 12) & 1), abort)))
          break;
        tc_fence_after();
        if ((warp & 3) == 0) mbar_arrive_warp(&k_empty[j % kKRing]);  // S_j read its K~ slot
        const uint32_t col = 128u * static_cast<uint32_t>(j % 3);
        // (block-sparse: N % 128 == 0 and non-causal, so no listed tile has a
        // masked key)
        const int k0 = j * kTile;
        const bool edge = !kSparse && (k0 + kTile > Nkv || (causal && k0 + kTile - 1 > q0));
        float mx[4] = {mraw, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          tmem_ld32(tmem + lane_base + col + 64 * hf, r);
          tmem_ld32(tmem + lane_base + col + 64 * hf + 32, r2);
          tmem_wait_ld();
          if (hf == 1) {
            tc_fence_before();
            mbar_arrive_warp(&s1_free[j % 6]);
          }
          if (!edge) {
#pragma unroll
            for (int i = 0; i < 16; i += 2) {
              mx[0] = max3f(mx[0], __uint_as_float(r[i]), __uint_as_float(r[i + 1]));
              mx[1] = max3f(mx[1], __uint_as_float(r[16 + i]), __uint_as_float(r[17 + i]));
              mx[2] = max3f(mx[2], __uint_as_float(r2[i]), __uint_as_float(r2[i + 1]));
              mx[3] = max3f(mx[3], __uint_as_float(r2[16 + i]), __uint_as_float(r2[17 + i]));
            }
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const int key = k0 + 64 * hf + i, key2 = key + 32;
              if (key < Nkv && (!causal || key <= qrow)) mx[i & 1] = fmaxf(mx[i & 1], __uint_as_float(r[i]));
              if (key2 < Nkv && (!causal || key2 <= qrow))
                mx[2 + (i & 1)] = fmaxf(mx[2 + (i & 1)], __uint_as_float(r2[i]));
            }
          }
        }
        mraw = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
      }
      mbar_arrive_warp(pass1_done);
    }
    // row maximum over the four warpgroups (always reached, also after an abort)
    xchg[wg * 128 + t] = mraw;
    named_bar_sync(1, 512);
    mraw = fmaxf(fmaxf(xchg[t], xchg[128 + t]), fmaxf(xchg[256 + t], xchg[384 + t]));
    named_bar_sync(1, 512);  // read before the sums reuse the area
    const float m = mraw * scale;
    const float negmb = -m * kLog2e;
    const uint64_t c12 = pk2(c1, c1), nmb2 = pk2(negmb, negmb);
    uint64_t l2 = pk2(0.f, 0.f);
    // auxiliary output: half u, keys [64 hh + 16 wg, +16) of tile j
    for (int u = 0; u < 2 * nk && ok && kAux; ++u) {
      const int j = u >> 1, hh = u & 1, c = u % 3;
      if (!(ok = mbar_wait_warp(&s_full[c], static_cast<uint32_t>((u / 3) & 1), abort))) break;
      tc_fence_after();
      const uint32_t col = 64u * c + 16u * wg;
      uint32_t r16[16];
      tmem_ld16(tmem + lane_base + col, r16);
      tmem_wait_ld();
      float x[16];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        up2(fma2(pk2(__uint_as_float(r16[2 * i]), __uint_as_float(r16[2 * i + 1])), c12, nmb2),
            x[2 * i], x[2 * i + 1]);
      const int k0 = j * kTile + 64 * hh + 16 * wg;
      if (k0 + 16 > Nkv || (causal && k0 + 15 > q0)) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int key = k0 + i;
          if (!(key < Nkv && (!causal || key <= qrow))) x[i] = -INFINITY;
        }
      }
      // P~ (f16 pairs) into the first 8 of the 16 columns just loaded, P into the next 8
      uint32_t pw[16];
      float pp[16];
      pquant16(x, pp, *reinterpret_cast<uint32_t(*)[8]>(pw));
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        l2 = add2(l2, pk2(pp[2 * i], pp[2 * i + 1]));
        __half2 h2 = __floats2half2_rn(pp[2 * i], pp[2 * i + 1]);
        pw[8 + i] = *reinterpret_cast<uint32_t*>(&h2);
      }
      tmem_st16(tmem + lane_base + col, pw);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive_warp(&p_full[c]);
    }
    for (int j = 0; j < nk && ok && !kAux; ++j) {
      const int buf = j & 1;
      if (!(ok = mbar_wait_warp(&s_full[buf], static_cast<uint32_t>((j >> 1) & 1), abort))) break;
      tc_fence_after();
      const uint32_t col = 128u * buf + 32u * wg;
      tmem_ld32(tmem + lane_base + col, r);
      tmem_wait_ld();
      float x[32];
#pragma unroll
      for (int i = 0; i < 16; ++i)
        up2(fma2(pk2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])), c12, nmb2),
            x[2 * i], x[2 * i + 1]);
      const int k0 = key0(j);
      if (!kSparse && is_edge(k0)) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int key = k0 + i;
          if (!(key < Nkv && (!causal || key <= qrow))) x[i] = -INFINITY;
        }
      }
      uint32_t pt[16];  // P~ of these 32 keys as f16 pairs
#pragma unroll
      for (int hb = 0; hb < 2; ++hb) {
        float pp[16];
        uint32_t (&ph)[8] = *reinterpret_cast<uint32_t(*)[8]>(pt + 8 * hb);
        pquant16(x + 16 * hb, pp, ph);
#pragma unroll
        for (int u = 0; u < 8; ++u) l2 = add2(l2, pk2(pp[2 * u], pp[2 * u + 1]));
      }
      tmem_st16(tmem + lane_base + col, pt);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive_warp(&p_full[buf]);
    }
    float l_lo, l_hi;
    up2(l2, l_lo, l_hi);
    float l = l_lo + l_hi;
    const bool have_o = ok && mbar_wait_warp(o_full, 0, abort);
    xchg[wg * 128 + t] = l;
    named_bar_sync(1, 512);
    l = (xchg[t] + xchg[128 + t]) + (xchg[256 + t] + xchg[384 + t]);
    if (have_o) {
      tc_fence_after();
      const float inv_l = 1.0f / l;
      // warpgroup wg writes O columns [wg D/4, (wg + 1) D/4) (and the same of O_hp)
      constexpr int kCols = D / 4;
#pragma unroll
      for (int oi = 0; oi < (kAux ? 2 : 1); ++oi) {
        const uint32_t o_col = 256u + static_cast<uint32_t>(oi * D + wg * kCols);
        uint32_t w[kCols / 2];
        if constexpr (kCols == 32) {
          tmem_ld32(tmem + lane_base + o_col, r);
        } else {
          uint32_t (&r16)[16] = *reinterpret_cast<uint32_t(*)[16]>(r);
          tmem_ld16(tmem + lane_base + o_col, r16);
        }
        tmem_wait_ld();
        if (qrow < Nq) {
#pragma unroll
          for (int i = 0; i < kCols / 2; ++i) {
            __nv_bfloat162 v2 = __floats2bfloat162_rn(__uint_as_float(r[2 * i]) * inv_l,
                                                      __uint_as_float(r[2 * i + 1]) * inv_l);
            w[i] = *reinterpret_cast<uint32_t*>(&v2);
          }
          __nv_bfloat16* orow = (oi ? o_hp : o) +
                                ((static_cast<int64_t>(b) * Nq + qrow) * H + h) * D + wg * kCols;
          uint4* dst = reinterpret_cast<uint4*>(orow);
#pragma unroll
          for (int u = 0; u < kCols / 8; ++u)
            dst[u] = make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
        }
      }
      if (qrow < Nq && wg == 0) {
        float* st = stats + bh * 2 * Nq;
        st[qrow] = m + logf(l);
        st[Nq + qrow] = m;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  report_abort(abort, err);
  if (warp == kSWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, int kMode>
cudaError_t launch_fp4_d(const AttnShape& s, const CUtensorMap& tq, const CUtensorMap& tk,
                         const CUtensorMap& tv, const uint8_t* q_sc, const uint8_t* k_sc, void* o,
                         void* o_hp, float* stats, const int* kv_list, int topk, int* err,
                         cudaStream_t stream) {
  using L = Fp4Layout<D>;
  static_assert(L::kAlloc <= 227u * 1024u, "shared memory");
  const dim3 grid((s.Nq + kTile - 1) / kTile, s.H, s.B);
  cudaError_t e = cudaFuncSetAttribute(attn_fwd_fp4_kernel<D, kMode>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (e != cudaSuccess) return e;
  attn_fwd_fp4_kernel<D, kMode><<<grid, kThreads, L::kAlloc, stream>>>(
      tq, tk, tv, q_sc, k_sc, static_cast<__nv_bfloat16*>(o), static_cast<__nv_bfloat16*>(o_hp),
      stats, s.Nq, s.Nkv, s.H, s.scale, s.causal, kv_list, topk, err);
  return cudaGetLastError();
}

template <int kMode>
cudaError_t launch_fp4_mode(const AttnShape& s, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, const uint8_t* q_sc, const uint8_t* k_sc,
                            void* o, void* o_hp, float* stats, const int* kv_list, int topk,
                            int* err, cudaStream_t stream) {
  return s.D == 128 ? launch_fp4_d<128, kMode>(s, tq, tk, tv, q_sc, k_sc, o, o_hp, stats, kv_list,
                                               topk, err, stream)
                    : launch_fp4_d<64, kMode>(s, tq, tk, tv, q_sc, k_sc, o, o_hp, stats, kv_list,
                                              topk, err, stream);
}

}  // namespace

cudaError_t launch_attn_fwd_fp4(const AttnShape& s, const CUtensorMap& tq, const CUtensorMap& tk,
                                const CUtensorMap& tv, const uint8_t* q_sc, const uint8_t* k_sc,
                                void* o, void* o_hp, float* stats, const int* kv_list, int topk,
                                int* err, cudaStream_t stream) {
  if (o_hp != nullptr && kv_list != nullptr) return cudaErrorInvalidValue;
  if (kv_list != nullptr)
    return launch_fp4_mode<kSparseFwd>(s, tq, tk, tv, q_sc, k_sc, o, nullptr, stats, kv_list, topk,
                                       err, stream);
  if (o_hp != nullptr)
    return launch_fp4_mode<kAuxFwd>(s, tq, tk, tv, q_sc, k_sc, o, o_hp, stats, nullptr, 0, err,
                                    stream);
  return launch_fp4_mode<kDenseFwd>(s, tq, tk, tv, q_sc, k_sc, o, nullptr, stats, nullptr, 0, err,
                                    stream);
}

}  // namespace nvq
