// Attn-QAT straight-through backward, dQ part (query-outer), with S on BF16
// UMMAs: the block-sparse form (the dense form runs attn_bwd_dq_fp4_kernel; the
// kernel template keeps the dense structure the block-sparse one specialises,
// but only the block-sparse instances are built).
//
//   dQ = scale * dS K~,   dS = A * (dP - delta),   A = P / l = exp(scale*S - m) / l,
//   dP = dO V~^T,         S = Q~ K~^T
// ("attn_qat_train" API page, attn_qat_train(): straight-through backward on the
// quantized operands).  dQ needs P, not P~, so no quantization happens here.
//
// One CTA per (128-query tile, head, batch).  Q~ and dO stay in shared memory;
// K~ and V~ stream in 128-key tiles (K~ through 3 slots, V~ through 2: K~_j is
// held from S_j until dQ_j, V~_j only until dP_j).  Per 128-key step j:
//   S_j = Q~ K~_j^T, dP_j = dO V~_j^T   (BF16 UMMA, M = 128, N = 128, into TMEM)
//   dS_j                                 (elementwise, bf16, stored back into TMEM)
//   dQ += dS_j K~_j                      (BF16 UMMA with A = dS_j read from TMEM)
// and dQ is written once, in bf16: no atomics, no fp32 accumulator in HBM.
// S and dP have one TMEM buffer each: the elementwise warps release it as soon
// as they have loaded their columns, so S_{j+1} and dP_{j+1} run on the tensor
// cores while dS_j is being computed; dS has two buffers.
//
// Roles (576 threads, one CTA per SM): warps 0-15 elementwise, warpgroup g owns
// keys [32g, 32g+32) of every step (thread t = query row t = TMEM lane t) and
// D/4 dQ columns at the end; warp 16 issues TMA, warp 17 allocates TMEM and
// issues the UMMAs (both as converged warps, one elected lane issuing).
// TMEM: S [0,128), dP [128,256), dQ [256,256+D), dS_b [384+64b, 448+64b).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "nvq_internal.h"
#include "nvq_ptx.cuh"
#include "nvq_quant.cuh"

namespace nvq {

namespace {

constexpr int kElemWarps = 16;
constexpr int kTmaWarp = 16;
constexpr int kMmaWarp = 17;
constexpr int kThreads = 576;
constexpr int kStep = 128;  // keys per step
constexpr int kKSlots = 3;  // K~ tiles in shared memory
constexpr int kVSlots = 2;  // V~ tiles in shared memory
constexpr uint32_t kColS = 0, kColDP = 128, kColDQ = 256, kColDS = 384;
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct DqLayout {
  static constexpr uint32_t kTileBytes = 128u * D * 2u;  // any 128-row tile (Q~, dO, K~, V~)
  static constexpr uint32_t kBlock = 128u * 128u;        // 64-column block of a 128-row tile
  static constexpr uint32_t kQ = 0;
  static constexpr uint32_t kDO = kQ + kTileBytes;
  static constexpr uint32_t kK = kDO + kTileBytes;            // [kKSlots]
  static constexpr uint32_t kV = kK + kKSlots * kTileBytes;   // [kVSlots]
  static constexpr uint32_t kBars = kV + kVSlots * kTileBytes;
  static constexpr uint32_t kNumBars = 1 + 2 * (kKSlots + kVSlots) + 2 + 2 * 2 + 2;
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

template <int D, bool kSparse>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tdo,
                       const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
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
  uint64_t* v_full = k_empty + kKSlots;            // [kVSlots]
  uint64_t* v_empty = v_full + kVSlots;            // [kVSlots]
  uint64_t* sdp_full = v_empty + kVSlots;          // S_j and dP_j are in TMEM
  uint64_t* sdp_free = sdp_full + 1;               // every elementwise warp has loaded them
  uint64_t* ds_full = sdp_full + 2;                // [2] dS_j is in TMEM buffer j % 2
  uint64_t* ds_free = sdp_full + 4;                // [2] dQ += dS_j K~_j is done
  uint64_t* dq_done = sdp_full + 6;
  uint64_t* mma_drain = sdp_full + 7;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + L::kAbort);

  const int n_all = (Nkv + kStep - 1) / kStep;
  // steps: every key tile (dense; causal: Nq == Nkv, kStep == kTile) or the topk
  // key tiles listed for this query tile (block-sparse)
  const int n = kSparse ? topk : causal ? min(n_all, q0 / kStep + 1) : n_all;
  const int* list = !kSparse ? nullptr
      : kv_list + ((static_cast<int64_t>(b) * H + h) * ((Nq + kTile - 1) / kTile) + qt) * topk;
  auto key_tile = [&](int j) -> int { return kSparse ? list[j] : j; };

  if (threadIdx.x == 0) {
    *abort = 0;
    mbar_init(q_full, 1);
    for (int s = 0; s < kKSlots; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < kVSlots; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    mbar_init(sdp_full, 1);
    mbar_init(sdp_free, kElemWarps);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ds_full[i], kElemWarps);
      mbar_init(&ds_free[i], 1);
    }
    mbar_init(dq_done, 1);
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

  if (warp == kTmaWarp) {
    // ------------------------------------------------------------ producer
    // Q~, dO once; then K~_0, V~_0, K~_1, V~_1, ... into their slots
    tma_prefetch_desc(&tq);
    tma_prefetch_desc(&tdo);
    tma_prefetch_desc(&tk);
    tma_prefetch_desc(&tv);
    mbar_arrive_expect_tx_w(q_full, 2u * L::kTileBytes);
#pragma unroll
    for (int blk = 0; blk < D / 64; ++blk) {
      tma_load_4d_w(smem + L::kQ + blk * L::kBlock, &tq, blk * 64, q0, h, b, q_full);
      tma_load_4d_w(smem + L::kDO + blk * L::kBlock, &tdo, blk * 64, q0, h, b, q_full);
    }
    int last_k[kKSlots], last_v[kVSlots];
    for (int s = 0; s < kKSlots; ++s) last_k[s] = -1;
    for (int s = 0; s < kVSlots; ++s) last_v[s] = -1;
    bool ok = true;
    for (int j = 0; j < n && ok; ++j) {
      const int ks = j % kKSlots, vs = j % kVSlots;
      const uint32_t ku = static_cast<uint32_t>(j / kKSlots), vu = static_cast<uint32_t>(j / kVSlots);
      if (!(ok = mbar_wait_warp(&k_empty[ks], (ku & 1u) ^ 1u, abort))) break;
      mbar_arrive_expect_tx_w(&k_full[ks], L::kTileBytes);
#pragma unroll
      for (int blk = 0; blk < D / 64; ++blk)
        tma_load_4d_w(smem + L::kK + ks * L::kTileBytes + blk * L::kBlock, &tk, blk * 64,
                      key_tile(j) * kStep, h, b, &k_full[ks]);
      last_k[ks] = static_cast<int>(ku & 1u);
      if (!(ok = mbar_wait_warp(&v_empty[vs], (vu & 1u) ^ 1u, abort))) break;
      mbar_arrive_expect_tx_w(&v_full[vs], L::kTileBytes);
#pragma unroll
      for (int blk = 0; blk < D / 64; ++blk)
        tma_load_4d_w(smem + L::kV + vs * L::kTileBytes + blk * L::kBlock, &tv, blk * 64,
                      key_tile(j) * kStep, h, b, &v_full[vs]);
      last_v[vs] = static_cast<int>(vu & 1u);
    }
    if (!ok) {  // let the loads already issued land before the block exits
      mbar_wait_warp(q_full, 0, nullptr, 10000000ull);
      for (int s = 0; s < kKSlots; ++s)
        if (last_k[s] >= 0) mbar_wait_warp(&k_full[s], static_cast<uint32_t>(last_k[s]), nullptr, 10000000ull);
      for (int s = 0; s < kVSlots; ++s)
        if (last_v[s] >= 0) mbar_wait_warp(&v_full[s], static_cast<uint32_t>(last_v[s]), nullptr, 10000000ull);
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------------- MMA
    // Order: S_0, dP_0; then per step j: S_{j+1}, dP_{j+1} (as soon as the
    // elementwise warps have loaded S_j and dP_j), then dQ_j (once dS_j is stored).
    constexpr uint32_t idesc_s = idesc_f16(128, kStep, 1, 0, 0);  // S, dP (N = 128 keys)
    constexpr uint32_t idesc_q = idesc_f16(128, D, 1, 0, 1);      // dQ (A in TMEM, B MN-major)
    const uint32_t q_addr = smem_u32(smem + L::kQ);
    const uint32_t do_addr = smem_u32(smem + L::kDO);
    const uint32_t k_addr = smem_u32(smem + L::kK);
    const uint32_t v_addr = smem_u32(smem + L::kV);
    // D_tile (128 x 128 keys) = A (128 x D, K-major) * B^T (B = 128 keys x D, K-major)
    auto issue_qk = [&](uint32_t a_addr, uint32_t b_addr, uint32_t dcol) {
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk >> 2) * L::kBlock + (kk & 3) * 32;
        umma_f16_ss_w(tmem + dcol, sdesc_sw128(a_addr + off, 16, 1024),
                      sdesc_sw128(b_addr + off, 16, 1024), idesc_s, kk > 0 ? 1u : 0u);
      }
    };
    // S_j and dP_j, once their tiles are in and every warp has loaded S_{j-1}, dP_{j-1}
    auto issue_step = [&](int j) -> bool {
      const int ks = j % kKSlots, vs = j % kVSlots;
      if (!mbar_wait_warp(&k_full[ks], static_cast<uint32_t>((j / kKSlots) & 1), abort) ||
          !mbar_wait_warp(&v_full[vs], static_cast<uint32_t>((j / kVSlots) & 1), abort))
        return false;
      if (j > 0 && !mbar_wait_warp(sdp_free, static_cast<uint32_t>((j - 1) & 1), abort)) return false;
      tc_fence_after();
      issue_qk(q_addr, k_addr + ks * L::kTileBytes, kColS);
      issue_qk(do_addr, v_addr + vs * L::kTileBytes, kColDP);
      umma_commit_w(sdp_full);
      umma_commit_w(&v_empty[vs]);  // V~_j is no longer needed
      return true;
    };
    bool ok = mbar_wait_warp(q_full, 0, abort) && issue_step(0);
    for (int j = 0; j < n && ok; ++j) {
      const int bsel = j & 1;
      if (j + 1 < n && !(ok = issue_step(j + 1))) break;
      if (!(ok = mbar_wait_warp(&ds_full[bsel], static_cast<uint32_t>((j >> 1) & 1), abort))) break;
      tc_fence_after();
      const uint32_t kb = k_addr + (j % kKSlots) * L::kTileBytes;
#pragma unroll
      for (int kk = 0; kk < kStep / 16; ++kk)  // dQ += dS K~: contraction over 128 keys
        umma_f16_ts_w(tmem + kColDQ, tmem + kColDS + bsel * 64 + kk * 8,
                      sdesc_sw128(kb + kk * 2048, L::kBlock, 1024), idesc_q,
                      (j > 0 || kk > 0) ? 1u : 0u);
      umma_commit_w(&ds_free[bsel]);
      umma_commit_w(&k_empty[j % kKSlots]);  // K~_j is no longer needed
    }
    if (ok) umma_commit_w(dq_done);
    umma_commit_w(mma_drain);
    mbar_wait_warp(mma_drain, 0, nullptr, 10000000ull);
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
    const uint64_t sl2 = pk2(scale * inv_l, scale * inv_l);  // dS carries the softmax scale
    const uint64_t ndl2 = pk2(-dl, -dl);
    const uint32_t kc = static_cast<uint32_t>(g * 32);
    bool ok = true;
    uint32_t rs[32], rd[32];
    for (int j = 0; j < n && ok; ++j) {
      const int bsel = j & 1;
      const int kt = key_tile(j);
      const int key0 = kt * kStep + static_cast<int>(kc);
      const bool edge = !row_ok || kt < 0 || (kt * kStep + kStep > Nkv) ||
                        (causal && kt * kStep + kStep - 1 > q0);
      if (!(ok = mbar_wait_warp(sdp_full, static_cast<uint32_t>(j & 1), abort))) break;
      tc_fence_after();
      tmem_ld32(tmem + lane_base + kColS + kc, rs);
      tmem_ld32(tmem + lane_base + kColDP + kc, rd);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive_warp(sdp_free);  // S_{j+1} and dP_{j+1} may overwrite them now
      // dS = (scale / l) * exp(scale*S - m) * (dP - delta), 32 keys
      uint32_t dsw[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        float x0, x1;
        up2(fma2(pk2(__uint_as_float(rs[2 * i]), __uint_as_float(rs[2 * i + 1])), c12, nmb2), x0, x1);
        if (edge) {
          const int k0 = key0 + 2 * i;
          if (!(row_ok && k0 >= 0 && k0 < Nkv && (!causal || k0 <= qrow))) x0 = -INFINITY;
          if (!(row_ok && k0 + 1 >= 0 && k0 + 1 < Nkv && (!causal || k0 + 1 <= qrow))) x1 = -INFINITY;
        }
        const uint64_t a2 = mul2(pk2(ex2_f32(x0), ex2_f32(x1)), sl2);
        float d0, d1;
        up2(mul2(a2, add2(pk2(__uint_as_float(rd[2 * i]), __uint_as_float(rd[2 * i + 1])), ndl2)),
            d0, d1);
        dsw[i] = pack_bf16(d0, d1);
      }
      // dS buffer bsel is free once dQ += dS_{j-2} K~_{j-2} is done
      if (j >= 2 && !(ok = mbar_wait_warp(&ds_free[bsel], static_cast<uint32_t>(((j >> 1) & 1) ^ 1), abort)))
        break;
      tc_fence_after();
      tmem_st16(tmem + lane_base + kColDS + bsel * 64 + (kc >> 1), dsw);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive_warp(&ds_full[bsel]);
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

}  // namespace

template <int D, bool kSparse>
cudaError_t launch_dq_t(const AttnShape& s, const CUtensorMap& tq, const CUtensorMap& tdo,
                        const CUtensorMap& tk, const CUtensorMap& tv, const float* stats,
                        const float* delta, void* dq, const int* kv_list, int topk, int* err,
                        cudaStream_t stream) {
  using L = DqLayout<D>;
  const dim3 grid((s.Nq + kTile - 1) / kTile, s.H, s.B);
  cudaError_t e = cudaFuncSetAttribute(attn_bwd_dq_kernel<D, kSparse>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (e != cudaSuccess) return e;
  attn_bwd_dq_kernel<D, kSparse><<<grid, kThreads, L::kAlloc, stream>>>(
      tq, tdo, tk, tv, stats, delta, static_cast<__nv_bfloat16*>(dq), s.Nq, s.Nkv, s.H, s.scale,
      s.causal, kv_list, topk, err);
  return cudaGetLastError();
}

cudaError_t launch_attn_bwd_dq(const AttnShape& s, const CUtensorMap& tq, const CUtensorMap& tdo,
                               const CUtensorMap& tk, const CUtensorMap& tv, const float* stats,
                               const float* delta, void* dq, const int* kv_list, int topk,
                               int* err, cudaStream_t stream) {
  // block-sparse only: the dense form runs attn_bwd_dq_fp4_kernel
  if (kv_list == nullptr) return cudaErrorInvalidValue;
  if (s.D == 128)
    return launch_dq_t<128, true>(s, tq, tdo, tk, tv, stats, delta, dq, kv_list, topk, err, stream);
  return launch_dq_t<64, true>(s, tq, tdo, tk, tv, stats, delta, dq, kv_list, topk, err, stream);
}

}  // namespace nvq
