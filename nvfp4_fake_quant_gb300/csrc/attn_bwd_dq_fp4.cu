// Attn-QAT straight-through backward, dQ part (query-outer), with S = Q~ K~^T
// on block-scaled FP4 UMMAs (tcgen05 kind::mxf4nvf4).
//
//   dQ = scale * dS K~,   dS = A * (dP - delta),   A = P / l = exp(scale*S - m) / l,
//   dP = dO V~^T,         S = Q~ K~^T
// ("attn_qat_train" API page, attn_qat_train(): straight-through backward on the
// quantized operands).  dQ needs P, not P~, so no quantization happens here.
// Q~ and K~ come in for S as packed E2M1 codes with their E4M3 block scales
// (the quantizer's outputs; the UMMA applies the scales, so S is the same sum
// of exact products as with BF16 operands); K~ also comes in as bf16 for dQ.
//
// One CTA per (128-query tile, head, batch).  The Q~ codes and dO stay in
// shared memory; per 128-key step j the K~ codes, V~ and the bf16 K~ stream in
// (K~ codes through 2 slots, V~ through 2, bf16 K~ through 3: it is held from
// the step's S until its dQ).  Per step:
//   S_j = Q~ K~_j^T (FP4), dP_j = dO V~_j^T (BF16)   (M = 128, N = 128, TMEM)
//   dS_j                                              (elementwise, bf16, TMEM)
//   dQ += dS_j K~_j                                   (BF16 UMMA, A = dS_j in TMEM)
// S and dP have one TMEM buffer each, released as soon as the elementwise
// warps have loaded them, so S_{j+1} and dP_{j+1} run while dS_j is computed.
// dS has one buffer: dQ_j is issued as soon as dS_j is stored and finishes
// while the elementwise warps compute dS_{j+1}.
//
// Roles (608 threads, one CTA per SM): warps 0-15 elementwise, warpgroup g owns
// keys [32g, 32g+32) of every step (thread t = query row t = TMEM lane t) and
// D/4 dQ columns at the end; warp 16 issues TMA, warp 17 allocates TMEM and
// issues the S and dP UMMAs, warp 18 the dQ UMMAs (converged warps, one elected
// lane issuing).  Each tcgen05 instruction and mbarrier wait costs its warp
// tens of cycles, so one warp issuing all three products would be the critical
// path; the two issuers touch disjoint TMEM (S, dP vs dQ, dS) and synchronise
// only through the elementwise warps' barriers.
// TMEM: S [0,128), dP [128,256), dQ [256,256+D), dS [384,448), the Q~ scale
// operand at [448 + 4 kk), the K~ scale operand of step j at [456 + 8 (j % 2)
// + 4 kk) (kk: 64-element group of D).  The copy for step j overwrites the
// scales of step j - 2, whose UMMAs completed before the release of S_{j-2},
// which the issuing warp waited on before S_{j-1}.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "nvq_internal.h"
#include "nvq_ptx.cuh"
#include "nvq_quant.cuh"

namespace nvq {

namespace {

constexpr int kElemWarps = 16;
constexpr int kTmaWarp = 16;
constexpr int kMmaWarp = 17;   // S, dP
constexpr int kDqWarp = 18;    // dQ
constexpr int kThreads = 608;
constexpr int kStep = 128;  // keys per step
constexpr int kKSlots = 3;   // bf16 K~ tiles in shared memory
constexpr int kK4Slots = 2;  // K~ code tiles in shared memory
constexpr int kVSlots = 2;   // V~ tiles in shared memory
constexpr uint32_t kColS = 0, kColDP = 128, kColDQ = 256, kColDS = 384;
constexpr uint32_t kScA = 448, kScB = 456;  // TMEM columns of the scale operands
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct DqLayout {
  static constexpr uint32_t kTileBytes = 128u * D * 2u;  // a bf16 128-row tile (dO, K~, V~)
  static constexpr uint32_t kBlock = 128u * 128u;        // 64-column block of a 128-row tile
  static constexpr uint32_t kCodeBytes = 128u * D / 2;   // E2M1 codes of a 128-row tile
  static constexpr uint32_t kScBytes = (D / 64) * 512u;  // its scale blocks
  static constexpr uint32_t kC4 = (kCodeBytes + kScBytes + 1023u) / 1024u * 1024u;
  static constexpr uint32_t kQ = 0;                            // Q~ codes + scales
  static constexpr uint32_t kDO = kQ + kC4;
  static constexpr uint32_t kK = kDO + kTileBytes;             // [kKSlots] bf16 K~
  static constexpr uint32_t kK4 = kK + kKSlots * kTileBytes;   // [kK4Slots] K~ codes + scales
  static constexpr uint32_t kV = kK4 + kK4Slots * kC4;         // [kVSlots]
  static constexpr uint32_t kBars = kV + kVSlots * kTileBytes;
  static constexpr uint32_t kNumBars = 1 + 2 * (kKSlots + kK4Slots + kVSlots) + 2 + 2 + 3;
  static constexpr uint32_t kTmemSlot = kBars + kNumBars * 8u;
  static constexpr uint32_t kAbort = kTmemSlot + 4u;
  static constexpr uint32_t kUsed = kAbort + 4u;
  static constexpr uint32_t kAlloc =
      (kUsed + 1024u) > 150u * 1024u ? (kUsed + 1024u) : 150u * 1024u;
};

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Grid: (ceil(Nq / 128), H, B).  tq4, tk4: packed codes of Q~, K~ (box of D/2
// bytes x 128 rows); q_sc, k_sc: their scale blocks; tdo, tk, tv: bf16 dO, K~, V~.
// kSparse: the query tile's steps run over its listed key tiles
// kv_list[b][h][qt][0..topk) instead of all of them.
template <int D, bool kSparse>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_dq_fp4_kernel(const __grid_constant__ CUtensorMap tq4,
                           const __grid_constant__ CUtensorMap tdo,
                           const __grid_constant__ CUtensorMap tk4,
                           const __grid_constant__ CUtensorMap tk,
                           const __grid_constant__ CUtensorMap tv,
                           const uint8_t* __restrict__ q_sc, const uint8_t* __restrict__ k_sc,
                           const float* __restrict__ stats, const float* __restrict__ delta,
                           __nv_bfloat16* __restrict__ dq, int Nq, int Nkv, int H, float scale,
                           int causal, const int* __restrict__ kv_list, int topk,
                           int* __restrict__ err) {
  using L = DqLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023u) &
                                             ~static_cast<uintptr_t>(1023u));
  const int warp = threadIdx.x >> 5;
  const int qt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int q0 = qt * kTile;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBars);
  uint64_t* q_full = bars + 0;
  uint64_t* k_full = bars + 1;                     // [kKSlots]
  uint64_t* k_empty = k_full + kKSlots;            // [kKSlots]
  uint64_t* k4_full = k_empty + kKSlots;           // [kK4Slots]
  uint64_t* k4_empty = k4_full + kK4Slots;         // [kK4Slots]
  uint64_t* v_full = k4_empty + kK4Slots;          // [kVSlots]
  uint64_t* v_empty = v_full + kVSlots;            // [kVSlots]
  uint64_t* sdp_full = v_empty + kVSlots;          // S_j and dP_j are in TMEM
  uint64_t* sdp_free = sdp_full + 1;               // every elementwise warp has loaded them
  uint64_t* ds_full = sdp_full + 2;                // dS_j is in TMEM
  uint64_t* ds_free = sdp_full + 3;                // dQ += dS_j K~_j is done
  uint64_t* dq_done = sdp_full + 4;
  uint64_t* mma_drain = sdp_full + 5;              // [2]: S/dP warp, dQ warp
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + L::kAbort);

  const int n_all = (Nkv + kStep - 1) / kStep;
  const int64_t bh = static_cast<int64_t>(b) * H + h;
  // steps: every key tile (causal: Nq == Nkv, kStep == kTile, up to the
  // diagonal), or the listed ones (block-sparse)
  const int* list = kSparse ? kv_list + (bh * ((Nq + kTile - 1) / kTile) + qt) * topk : nullptr;
  const int n = kSparse ? topk : causal ? min(n_all, q0 / kStep + 1) : n_all;
  auto ktile = [&](int j) -> int { return kSparse ? list[j] : j; };

  if (threadIdx.x == 0) {
    *abort = 0;
    mbar_init(q_full, 1);
    for (int s = 0; s < kKSlots; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < kK4Slots; ++s) {
      mbar_init(&k4_full[s], 1);
      mbar_init(&k4_empty[s], 1);
    }
    for (int s = 0; s < kVSlots; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    mbar_init(sdp_full, 1);
    mbar_init(sdp_free, kElemWarps);
    mbar_init(ds_full, kElemWarps);
    mbar_init(ds_free, 1);
    mbar_init(dq_done, 1);
    mbar_init(&mma_drain[0], 1);
    mbar_init(&mma_drain[1], 1);
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

  if (warp == kTmaWarp) {
    // ------------------------------------------------------------ producer
    // Q~ codes and dO once; then per step j: K~_j codes, V~_j, bf16 K~_j (the
    // order the UMMAs need them: S_j, dP_j, then dQ_j after S_{j+1}, dP_{j+1}).
    const int n_qt = (Nq + kTile - 1) / kTile;
    const int n_kt = n_all;
    tma_prefetch_desc(&tq4);
    tma_prefetch_desc(&tdo);
    tma_prefetch_desc(&tk4);
    tma_prefetch_desc(&tk);
    tma_prefetch_desc(&tv);
    mbar_arrive_expect_tx_w(q_full, L::kCodeBytes + L::kScBytes + L::kTileBytes);
    tma_load_4d_w(smem + L::kQ, &tq4, 0, q0, h, b, q_full);
    bulk_load_w(smem + L::kQ + L::kCodeBytes, q_sc + (bh * n_qt + qt) * L::kScBytes, L::kScBytes,
                q_full);
#pragma unroll
    for (int blk = 0; blk < D / 64; ++blk)
      tma_load_4d_w(smem + L::kDO + blk * L::kBlock, &tdo, blk * 64, q0, h, b, q_full);
    int last_k[kKSlots], last_k4[kK4Slots], last_v[kVSlots];
    for (int s = 0; s < kKSlots; ++s) last_k[s] = -1;
    for (int s = 0; s < kK4Slots; ++s) last_k4[s] = -1;
    for (int s = 0; s < kVSlots; ++s) last_v[s] = -1;
    bool ok = true;
    for (int j = 0; j < n && ok; ++j) {
      const int ks = j % kKSlots, k4s = j % kK4Slots, vs = j % kVSlots;
      const uint32_t ku = static_cast<uint32_t>(j / kKSlots);
      const uint32_t k4u = static_cast<uint32_t>(j / kK4Slots), vu = static_cast<uint32_t>(j / kVSlots);
      if (!(ok = mbar_wait_warp(&k4_empty[k4s], (k4u & 1u) ^ 1u, abort))) break;
      uint8_t* k4dst = smem + L::kK4 + k4s * L::kC4;
      const int kt = ktile(j);
      mbar_arrive_expect_tx_w(&k4_full[k4s], L::kCodeBytes + L::kScBytes);
      tma_load_4d_w(k4dst, &tk4, 0, kt * kStep, h, b, &k4_full[k4s]);
      bulk_load_w(k4dst + L::kCodeBytes, k_sc + (bh * n_kt + kt) * L::kScBytes, L::kScBytes,
                  &k4_full[k4s]);
      last_k4[k4s] = static_cast<int>(k4u & 1u);
      if (!(ok = mbar_wait_warp(&v_empty[vs], (vu & 1u) ^ 1u, abort))) break;
      mbar_arrive_expect_tx_w(&v_full[vs], L::kTileBytes);
#pragma unroll
      for (int blk = 0; blk < D / 64; ++blk)
        tma_load_4d_w(smem + L::kV + vs * L::kTileBytes + blk * L::kBlock, &tv, blk * 64,
                      kt * kStep, h, b, &v_full[vs]);
      last_v[vs] = static_cast<int>(vu & 1u);
      if (!(ok = mbar_wait_warp(&k_empty[ks], (ku & 1u) ^ 1u, abort))) break;
      mbar_arrive_expect_tx_w(&k_full[ks], L::kTileBytes);
#pragma unroll
      for (int blk = 0; blk < D / 64; ++blk)
        tma_load_4d_w(smem + L::kK + ks * L::kTileBytes + blk * L::kBlock, &tk, blk * 64,
                      kt * kStep, h, b, &k_full[ks]);
      last_k[ks] = static_cast<int>(ku & 1u);
    }
    if (!ok) {  // let the loads already issued land before the block exits
      mbar_wait_warp(q_full, 0, nullptr, 10000000ull);
      for (int s = 0; s < kKSlots; ++s)
        if (last_k[s] >= 0) mbar_wait_warp(&k_full[s], static_cast<uint32_t>(last_k[s]), nullptr, 10000000ull);
      for (int s = 0; s < kK4Slots; ++s)
        if (last_k4[s] >= 0) mbar_wait_warp(&k4_full[s], static_cast<uint32_t>(last_k4[s]), nullptr, 10000000ull);
      for (int s = 0; s < kVSlots; ++s)
        if (last_v[s] >= 0) mbar_wait_warp(&v_full[s], static_cast<uint32_t>(last_v[s]), nullptr, 10000000ull);
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------------- MMA
    // S_j, dP_j as soon as their tiles are in and the elementwise warps have
    // loaded S_{j-1}, dP_{j-1}; dQ_j comes from the other issuing warp.
    constexpr uint32_t idesc_s4 = idesc_mxf4nvf4(128, kStep);      // S (FP4, N = 128 keys)
    constexpr uint32_t idesc_p = idesc_f16(128, kStep, 1, 0, 0);   // dP (N = 128 keys)
    constexpr uint32_t lay = D == 128 ? 4u : 6u;                   // (D/2)-byte swizzle of code rows
    constexpr uint32_t sbo = 8u * (D / 2);
    const uint32_t q_addr = smem_u32(smem + L::kQ);
    const uint32_t do_addr = smem_u32(smem + L::kDO);
    const uint32_t k4_addr = smem_u32(smem + L::kK4);
    const uint32_t v_addr = smem_u32(smem + L::kV);
    // S_j and dP_j, once their tiles are in and every warp has loaded S_{j-1},
    // dP_{j-1}.  The K~ scales are copied before that last wait, off the path
    // from the release to the UMMAs (their columns were last read by S_{j-2},
    // complete since this warp saw S_{j-2} and dP_{j-2} released).
    // Descriptors, computed once: the Q~ codes (a 64-element K step is 32 bytes,
    // 2 in the start-address field), dO and the V~ slots (K step kk of a
    // K-major bf16 tile at byte (kk / 4) 16384 + (kk % 4) 32)
    uint64_t q_d[D / 64], dp_ad[D / 16], dp_bd[kVSlots][D / 16];
#pragma unroll
    for (int kk = 0; kk < D / 64; ++kk) q_d[kk] = sdesc(q_addr + 32 * kk, 16, sbo, lay);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const uint32_t off = (kk >> 2) * L::kBlock + (kk & 3) * 32;
      dp_ad[kk] = sdesc_sw128(do_addr + off, 16, 1024);
#pragma unroll
      for (int vs = 0; vs < kVSlots; ++vs)
        dp_bd[vs][kk] = sdesc_sw128(v_addr + vs * L::kTileBytes + off, 16, 1024);
    }
    static_assert(kVSlots == 2, "the V~ slot is a branch below");
    auto issue_step = [&](int j) -> bool {
      const int k4s = j % kK4Slots, vs = j % kVSlots;
      if (!mbar_wait_warp(&k4_full[k4s], static_cast<uint32_t>((j / kK4Slots) & 1), abort))
        return false;
      tc_fence_after();
      const uint32_t kb = k4_addr + k4s * L::kC4;
      const uint32_t sc = kScB + 8u * static_cast<uint32_t>(j & 1);
#pragma unroll
      for (int kk = 0; kk < D / 64; ++kk)
        tmem_cp_32x128_x4_w(tmem + sc + 4 * kk, kb + L::kCodeBytes + kk * 512);
      if (!mbar_wait_warp(&v_full[vs], static_cast<uint32_t>((j / kVSlots) & 1), abort))
        return false;
      if (j > 0 && !mbar_wait_warp(sdp_free, static_cast<uint32_t>((j - 1) & 1), abort)) return false;
      tc_fence_after();
      uint64_t kd[D / 64];
      kd[0] = sdesc(kb, 16, sbo, lay);
      if constexpr (D == 128) kd[1] = kd[0] + 2;
      // S, then the K~ codes of step j are no longer needed
      umma_fp4_group_w<D / 64>(tmem + kColS, q_d, kd, idesc_s4, tmem + kScA, tmem + sc,
                               bar_u32(&k4_empty[k4s]), 0u);
      // dP, then S_j and dP_j are in TMEM and V~_j is no longer needed
      if (vs)
        umma_f16_group_w<D / 16>(tmem + kColDP, dp_ad, dp_bd[1], idesc_p, 0u, bar_u32(sdp_full),
                                 bar_u32(&v_empty[1]));
      else
        umma_f16_group_w<D / 16>(tmem + kColDP, dp_ad, dp_bd[0], idesc_p, 0u, bar_u32(sdp_full),
                                 bar_u32(&v_empty[0]));
      return true;
    };
    bool ok = mbar_wait_warp(q_full, 0, abort);
    if (ok) {  // the Q~ scales stay in TMEM for the whole kernel
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < D / 64; ++kk)
        tmem_cp_32x128_x4_w(tmem + kScA + 4 * kk, q_addr + L::kCodeBytes + kk * 512);
    }
    for (int j = 0; j < n && ok; ++j) ok = issue_step(j);
    umma_commit_w(&mma_drain[0]);
    mbar_wait_warp(&mma_drain[0], 0, nullptr, 10000000ull);
  } else if (warp == kDqWarp) {
    // ---------------------------------------------------------------- dQ
    constexpr uint32_t idesc_q = idesc_f16(128, D, 1, 0, 1);  // dQ (A in TMEM, B MN-major)
    const uint32_t k_addr = smem_u32(smem + L::kK);
    const uint64_t k_d0 = sdesc_sw128(k_addr, L::kBlock, 1024);  // bf16 K~ slot 0, keys 0-15
    uint32_t a[8];  // dS_j, 16 keys (8 columns) per K step
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) a[kk] = tmem + kColDS + kk * 8;
    bool ok = true;
    for (int j = 0; j < n && ok; ++j) {
      const int ks = j % kKSlots;
      if (!(ok = mbar_wait_warp(ds_full, static_cast<uint32_t>(j & 1), abort)) ||
          !(ok = mbar_wait_warp(&k_full[ks], static_cast<uint32_t>((j / kKSlots) & 1), abort)))
        break;
      tc_fence_after();
      // dQ += dS K~: contraction over the 128 keys; then bf16 K~_j is no longer needed
      static_assert(kStep == 128, "eight K steps of 16 keys");
      umma_f16_ts8_w(tmem + kColDQ, a, k_d0 + static_cast<uint64_t>(ks) * (L::kTileBytes >> 4),
                     idesc_q, j > 0 ? 1u : 0u, bar_u32(ds_free), bar_u32(&k_empty[ks]));
    }
    if (ok) umma_commit_w(dq_done);
    umma_commit_w(&mma_drain[1]);
    mbar_wait_warp(&mma_drain[1], 0, nullptr, 10000000ull);
  } else {
    // --------------------------------------------------------- elementwise
    const int g = warp >> 2;                // warpgroup: keys [32g, 32g+32) of each step
    const int t = threadIdx.x & 127;        // query row in the tile == TMEM lane
    const int qrow = q0 + t;
    const bool row_ok = qrow < Nq;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const float* st = stats + (static_cast<int64_t>(b) * H + h) * 2 * Nq;
    const float m = row_ok ? st[Nq + qrow] : 0.f;
    const float lse = row_ok ? st[qrow] : 0.f;
    const float dl = row_ok ? delta[(static_cast<int64_t>(b) * H + h) * Nq + qrow] : 0.f;
    const float c1 = scale * kLog2e;
    const float negmb = -m * kLog2e;
    const float inv_l = ex2_f32((m - lse) * kLog2e);  // 1 / l
    const uint64_t c12 = pk2(c1, c1), nmb2 = pk2(negmb, negmb);
    // dS = P * (sl dP - sl delta), sl = scale / l (dS carries the softmax scale)
    const float sl = scale * inv_l;
    const uint64_t sl2 = pk2(sl, sl), nsd2 = pk2(-sl * dl, -sl * dl);
    const uint32_t kc = static_cast<uint32_t>(g * 32);
    bool ok = true;
    uint32_t rs[32], rd[32];
    for (int j = 0; j < n && ok; ++j) {
      const int kt = ktile(j);
      const int key0 = kt * kStep + static_cast<int>(kc);
      const bool edge = !row_ok || (kt * kStep + kStep > Nkv) ||
                        (causal && kt * kStep + kStep - 1 > q0);
      if (!(ok = mbar_wait_warp(sdp_full, static_cast<uint32_t>(j & 1), abort))) break;
      tc_fence_after();
      tmem_ld32(tmem + lane_base + kColS + kc, rs);
      tmem_ld32(tmem + lane_base + kColDP + kc, rd);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive_warp(sdp_free);  // S_{j+1} and dP_{j+1} may overwrite them now
      // dS = (scale / l) * exp(scale*S - m) * (dP - delta), 32 keys, as
      // P * fma(dP, sl, -sl * delta)
      uint32_t dsw[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        float x0, x1;
        up2(fma2(pk2(__uint_as_float(rs[2 * i]), __uint_as_float(rs[2 * i + 1])), c12, nmb2), x0, x1);
        if (edge) {
          const int k0 = key0 + 2 * i;
          if (!(row_ok && k0 < Nkv && (!causal || k0 <= qrow))) x0 = -INFINITY;
          if (!(row_ok && k0 + 1 < Nkv && (!causal || k0 + 1 <= qrow))) x1 = -INFINITY;
        }
        const uint64_t t2 = fma2(pk2(__uint_as_float(rd[2 * i]), __uint_as_float(rd[2 * i + 1])), sl2, nsd2);
        float d0, d1;
        up2(mul2(pk2(ex2_f32(x0), ex2_f32(x1)), t2), d0, d1);
        dsw[i] = pack_bf16(d0, d1);
      }
      // the dS buffer is free once dQ += dS_{j-1} K~_{j-1} is done
      if (j >= 1 && !(ok = mbar_wait_warp(ds_free, static_cast<uint32_t>((j - 1) & 1), abort)))
        break;
      tc_fence_after();
      tmem_st16(tmem + lane_base + kColDS + (kc >> 1), dsw);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive_warp(ds_full);
    }
    if (ok && (ok = mbar_wait_warp(dq_done, 0, abort))) {
      tc_fence_after();
      constexpr int kCols = D / 4;  // dQ columns of this warpgroup
      __nv_bfloat16* dst = dq + ((static_cast<int64_t>(b) * Nq + qrow) * H + h) * D + g * kCols;
      uint32_t w[kCols / 2];
#pragma unroll
      for (int c = 0; c < kCols / 16; ++c) {
        uint32_t r[16];
        tmem_ld16(tmem + lane_base + kColDQ + g * kCols + c * 16, r);
        tmem_wait_ld();
#pragma unroll
        for (int u = 0; u < 8; ++u)
          w[c * 8 + u] = pack_bf16(__uint_as_float(r[2 * u]), __uint_as_float(r[2 * u + 1]));
      }
      if (row_ok) {
#pragma unroll
        for (int u = 0; u < kCols / 8; ++u)
          reinterpret_cast<uint4*>(dst)[u] = make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
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

template <int D, bool kSparse>
cudaError_t launch_dq4_t(const AttnShape& s, const CUtensorMap& tq4, const CUtensorMap& tdo,
                         const CUtensorMap& tk4, const CUtensorMap& tk, const CUtensorMap& tv,
                         const uint8_t* q_sc, const uint8_t* k_sc, const float* stats,
                         const float* delta, void* dq, const int* kv_list, int topk, int* err,
                         cudaStream_t stream) {
  using L = DqLayout<D>;
  static_assert(L::kAlloc <= 227u * 1024u, "shared memory");
  const dim3 grid((s.Nq + kTile - 1) / kTile, s.H, s.B);
  cudaError_t e = cudaFuncSetAttribute(attn_bwd_dq_fp4_kernel<D, kSparse>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (e != cudaSuccess) return e;
  attn_bwd_dq_fp4_kernel<D, kSparse><<<grid, kThreads, L::kAlloc, stream>>>(
      tq4, tdo, tk4, tk, tv, q_sc, k_sc, stats, delta, static_cast<__nv_bfloat16*>(dq), s.Nq,
      s.Nkv, s.H, s.scale, s.causal, kv_list, topk, err);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_bwd_dq_fp4(const AttnShape& s, const CUtensorMap& tq4,
                                   const CUtensorMap& tdo, const CUtensorMap& tk4,
                                   const CUtensorMap& tk, const CUtensorMap& tv,
                                   const uint8_t* q_sc, const uint8_t* k_sc, const float* stats,
                                   const float* delta, void* dq, const int* kv_list, int topk,
                                   int* err, cudaStream_t stream) {
  if (kv_list != nullptr)
    return s.D == 128 ? launch_dq4_t<128, true>(s, tq4, tdo, tk4, tk, tv, q_sc, k_sc, stats, delta, dq, kv_list, topk, err, stream)
                      : launch_dq4_t<64, true>(s, tq4, tdo, tk4, tk, tv, q_sc, k_sc, stats, delta, dq, kv_list, topk, err, stream);
  return s.D == 128 ? launch_dq4_t<128, false>(s, tq4, tdo, tk4, tk, tv, q_sc, k_sc, stats, delta, dq, nullptr, 0, err, stream)
                    : launch_dq4_t<64, false>(s, tq4, tdo, tk4, tk, tv, q_sc, k_sc, stats, delta, dq, nullptr, 0, err, stream);
}

}  // namespace nvq
