// Attn-QAT straight-through backward, dQ part (query-outer).
//
//   dQ = scale * dS K~,   dS = A * (dP - delta),   A = P / l = exp(scale*S - m) / l,
//   dP = dO V~^T,         S = Q~ K~^T
// ("attn_qat_train" API page, attn_qat_train(): straight-through backward on the
// quantized operands).  dQ needs P, not P~, so no quantization happens here.
//
// One CTA per (128-query tile, head, batch).  Q~ and dO stay in shared memory;
// K~ and V~ stream in 64-key tiles through an 8-slot ring.  Per 64-key step:
//   S = Q~ K~^T, dP = dO V~^T   (BF16 UMMA, N = 64, double-buffered in TMEM)
//   dS (elementwise, bf16 into a double-buffered shared tile)
//   dQ += dS K~                  (BF16 UMMA, accumulated in TMEM over all keys)
// and dQ is written once, in bf16: no atomics, no fp32 accumulator in HBM.
//
// Roles (576 threads, one CTA per SM): warps 0-15 elementwise, in two sets of
// eight warps that take alternate steps (set s does steps s, s+2, ...), so one
// set's TMEM loads, exponentials and stores overlap the other set's; within a
// set, warpgroup gg owns keys [32gg, 32gg+32) of the step (thread t = query row
// t = TMEM lane t).  At the end every warpgroup writes D/4 dQ columns.  Warp 16
// issues TMA, warp 17 allocates TMEM and issues the UMMAs.
// TMEM: S of set s at [64s, 64s+64), dP of set s at [128+64s, 192+64s), dQ at
// [256, 256+D).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "nvq_internal.h"
#include "nvq_ptx.cuh"
#include "nvq_quant.cuh"

namespace nvq {

namespace {

constexpr int kElemWarps = 16;
constexpr int kSetWarps = 8;  // elementwise warps per set
constexpr int kTmaWarp = 16;
constexpr int kMmaWarp = 17;
constexpr int kThreads = 576;
constexpr int kStep = 64;   // keys per step
constexpr int kRing = 8;    // K~/V~ tiles in flight
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct DqLayout {
  static constexpr uint32_t kQTile = 128u * D * 2u;        // Q~ or dO tile
  static constexpr uint32_t kKVTile = kStep * D * 2u;       // one 64-key K~ or V~ tile
  static constexpr uint32_t kQBlock = 128u * 128u;          // 64-column block of a 128-row tile
  static constexpr uint32_t kKVBlock = kStep * 128u;        // 64-column block of a 64-row tile
  static constexpr uint32_t kQ = 0;
  static constexpr uint32_t kDO = kQ + kQTile;
  static constexpr uint32_t kRingOff = kDO + kQTile;
  static constexpr uint32_t kDS = kRingOff + kRing * kKVTile;  // [2] x [128 q][64 keys] bf16
  static constexpr uint32_t kDSBytes = 128u * kStep * 2u;
  static constexpr uint32_t kBars = kDS + 2u * kDSBytes;
  static constexpr uint32_t kNumBars = 1 + 2 * kRing + 2 * 3 + 2;
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

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tdo,
                       const __grid_constant__ CUtensorMap tk64, const __grid_constant__ CUtensorMap tv64,
                       const float* __restrict__ stats, const float* __restrict__ delta,
                       __nv_bfloat16* __restrict__ dq, int Nq, int Nkv, int H, float scale,
                       int causal, int* __restrict__ err) {
  using L = DqLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023u) &
                                             ~static_cast<uintptr_t>(1023u));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int qt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int q0 = qt * kTile;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBars);
  uint64_t* q_full = bars + 0;
  uint64_t* r_full = bars + 1;              // [kRing]
  uint64_t* r_empty = bars + 1 + kRing;     // [kRing]
  uint64_t* sdp_full = bars + 1 + 2 * kRing;  // [2] S and dP of a step are in TMEM
  uint64_t* ds_full = sdp_full + 2;           // [2] dS of a step is in shared memory
  uint64_t* ds_free = sdp_full + 4;           // [2] dQ += dS K~ of a step is done
  uint64_t* dq_done = sdp_full + 6;
  uint64_t* mma_drain = sdp_full + 7;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + L::kAbort);

  const int n_all = (Nkv + kStep - 1) / kStep;
  const int n = causal ? min(n_all, (q0 + kTile + kStep - 1) / kStep) : n_all;

  if (threadIdx.x == 0) {
    *abort = 0;
    mbar_init(q_full, 1);
    for (int s = 0; s < kRing; ++s) {
      mbar_init(&r_full[s], 1);
      mbar_init(&r_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sdp_full[i], 1);
      mbar_init(&ds_full[i], kSetWarps);
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
    // Q~, dO once; then K~_0, V~_0, K~_1, V~_1, ... (64-key tiles) through the ring
    tma_prefetch_desc(&tq);
    tma_prefetch_desc(&tdo);
    tma_prefetch_desc(&tk64);
    tma_prefetch_desc(&tv64);
    mbar_arrive_expect_tx_w(q_full, 2u * L::kQTile);
#pragma unroll
    for (int blk = 0; blk < D / 64; ++blk) {
      tma_load_4d_w(smem + L::kQ + blk * L::kQBlock, &tq, blk * 64, q0, h, b, q_full);
      tma_load_4d_w(smem + L::kDO + blk * L::kQBlock, &tdo, blk * 64, q0, h, b, q_full);
    }
    int last[kRing];
    for (int s = 0; s < kRing; ++s) last[s] = -1;
    bool ok = true;
    for (int li = 0; li < 2 * n && ok; ++li) {
      const int slot = li % kRing;
      const uint32_t use = static_cast<uint32_t>(li / kRing);
      if (!(ok = mbar_wait_warp(&r_empty[slot], (use & 1u) ^ 1u, abort))) break;
      const int j = li >> 1;
      mbar_arrive_expect_tx_w(&r_full[slot], L::kKVTile);
#pragma unroll
      for (int blk = 0; blk < D / 64; ++blk)
        tma_load_4d_w(smem + L::kRingOff + slot * L::kKVTile + blk * L::kKVBlock,
                      (li & 1) ? &tv64 : &tk64, blk * 64, j * kStep, h, b, &r_full[slot]);
      last[slot] = static_cast<int>(use & 1u);
    }
    if (!ok) {
      mbar_wait_warp(q_full, 0, nullptr, 10000000ull);
      for (int s = 0; s < kRing; ++s)
        if (last[s] >= 0) mbar_wait_warp(&r_full[s], static_cast<uint32_t>(last[s]), nullptr, 10000000ull);
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------------- MMA
    // Order: S_0, dP_0, S_1, dP_1, then per step j: dQ_j, S_{j+2}, dP_{j+2}.
    constexpr uint32_t idesc_s = idesc_f16(128, kStep, 1, 0, 0);  // S, dP (N = 64 keys)
    constexpr uint32_t idesc_q = idesc_f16(128, D, 1, 0, 1);      // dQ (A K-major, B MN-major)
    const uint32_t q_addr = smem_u32(smem + L::kQ);
    const uint32_t do_addr = smem_u32(smem + L::kDO);
    const uint32_t ring_addr = smem_u32(smem + L::kRingOff);
    const uint32_t ds_addr = smem_u32(smem + L::kDS);
    auto slot_of = [](int li) { return li % kRing; };
    auto wait_tile = [&](int li) -> bool {
      return mbar_wait_warp(&r_full[slot_of(li)], static_cast<uint32_t>((li / kRing) & 1), abort);
    };
    // S_j (or dP_j) = A (128 x D, K-major) * B^T (B = 64 x D tile, K-major)
    auto issue_qk = [&](uint32_t a_addr, int li, uint32_t dcol) {
      const uint32_t bb = ring_addr + slot_of(li) * L::kKVTile;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        umma_f16_ss_w(tmem + dcol,
                      sdesc_sw128(a_addr + (kk >> 2) * L::kQBlock + (kk & 3) * 32, 16, 1024),
                      sdesc_sw128(bb + (kk >> 2) * L::kKVBlock + (kk & 3) * 32, 16, 1024), idesc_s,
                      kk > 0 ? 1u : 0u);
      }
    };
    auto issue_step = [&](int j) -> bool {  // S_j and dP_j into the buffers of set j % 2
      if (!wait_tile(2 * j) || !wait_tile(2 * j + 1)) return false;
      tc_fence_after();
      const int bsel = j & 1;
      issue_qk(q_addr, 2 * j, static_cast<uint32_t>(bsel * kStep));
      issue_qk(do_addr, 2 * j + 1, static_cast<uint32_t>(128 + bsel * kStep));
      umma_commit_w(&sdp_full[bsel]);
      umma_commit_w(&r_empty[slot_of(2 * j + 1)]);  // V~_j is no longer needed
      return true;
    };
    bool ok = mbar_wait_warp(q_full, 0, abort);
    if (ok) ok = issue_step(0);
    if (ok && n > 1) ok = issue_step(1);
    for (int j = 0; j < n && ok; ++j) {
      const int bsel = j & 1;
      if (!(ok = mbar_wait_warp(&ds_full[bsel], static_cast<uint32_t>((j >> 1) & 1), abort))) break;
      tc_fence_after();
      const uint32_t kb = ring_addr + slot_of(2 * j) * L::kKVTile;
      const uint32_t dsb = ds_addr + bsel * L::kDSBytes;
#pragma unroll
      for (int kk = 0; kk < kStep / 16; ++kk)  // dQ += dS K~: contraction over 64 keys
        umma_f16_ss_w(tmem + 256, sdesc_sw128(dsb + kk * 32, 16, 1024),
                      sdesc_sw128(kb + kk * 2048, L::kKVBlock, 1024), idesc_q,
                      (j > 0 || kk > 0) ? 1u : 0u);
      umma_commit_w(&ds_free[bsel]);
      umma_commit_w(&r_empty[slot_of(2 * j)]);  // K~_j is no longer needed
      // set bsel read S_j and dP_j before ds_full_j: step j+2 may reuse them
      if (j + 2 < n) ok = issue_step(j + 2);
    }
    if (ok) umma_commit_w(dq_done);
    umma_commit_w(mma_drain);
    mbar_wait_warp(mma_drain, 0, nullptr, 10000000ull);
  } else {
    // --------------------------------------------------------- elementwise
    const int g = warp >> 2;                // warpgroup 0..3
    const int set = g >> 1;                 // steps set, set + 2, ...
    const int kc = (g & 1) * 32;            // keys [kc, kc + 32) of each step
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
    uint8_t* dsb = smem + L::kDS + set * L::kDSBytes;
    const uint32_t s_col = static_cast<uint32_t>(set * kStep + kc);
    bool ok = true;
    uint32_t rs[32], rd[32];
    for (int j = set, k = 0; j < n && ok; j += 2, ++k) {
      const uint32_t ph = static_cast<uint32_t>(k & 1);
      const int key0 = j * kStep + kc;
      const bool edge = !row_ok || (j * kStep + kStep > Nkv) || (causal && j * kStep + kStep - 1 > q0);
      if (!(ok = mbar_wait_warp(&sdp_full[set], ph, abort))) break;
      tc_fence_after();
      tmem_ld32(tmem + lane_base + s_col, rs);
      tmem_ld32(tmem + lane_base + 128 + s_col, rd);
      tmem_wait_ld();
      // dS = (scale / l) * exp(scale*S - m) * (dP - delta), 32 keys
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
        const uint64_t a2 = mul2(pk2(ex2_f32(x0), ex2_f32(x1)), sl2);
        float d0, d1;
        up2(mul2(a2, add2(pk2(__uint_as_float(rd[2 * i]), __uint_as_float(rd[2 * i + 1])), ndl2)),
            d0, d1);
        dsw[i] = pack_bf16(d0, d1);
      }
      tc_fence_before();
      // this set's dS buffer is free once dQ of its previous step (j - 2) is done
      if (k > 0 && !(ok = mbar_wait_warp(&ds_free[set], ph ^ 1u, abort))) break;
#pragma unroll
      for (int ch = 0; ch < 4; ++ch)
        *reinterpret_cast<uint4*>(dsb + sw128_offset(t, kc + ch * 8, 128)) =
            make_uint4(dsw[4 * ch], dsw[4 * ch + 1], dsw[4 * ch + 2], dsw[4 * ch + 3]);
      fence_proxy_async_smem();
      mbar_arrive_warp(&ds_full[set]);
    }
    if (ok && (ok = mbar_wait_warp(dq_done, 0, abort))) {
      tc_fence_after();
      constexpr int kCols = D / 4;  // dQ columns of this warpgroup
      __nv_bfloat16* dst = dq + ((static_cast<int64_t>(b) * Nq + qrow) * H + h) * D + g * kCols;
      uint32_t w[kCols / 2];
#pragma unroll
      for (int c = 0; c < kCols / 16; ++c) {
        uint32_t r[16];
        tmem_ld16(tmem + lane_base + 256 + g * kCols + c * 16, r);
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

cudaError_t launch_attn_bwd_dq(const AttnShape& s, const CUtensorMap& tq, const CUtensorMap& tdo,
                               const CUtensorMap& tk64, const CUtensorMap& tv64,
                               const float* stats, const float* delta, void* dq, int* err,
                               cudaStream_t stream) {
  const dim3 grid((s.Nq + kTile - 1) / kTile, s.H, s.B);
  auto* dqp = static_cast<__nv_bfloat16*>(dq);
  if (s.D == 128) {
    using L = DqLayout<128>;
    cudaError_t e = cudaFuncSetAttribute(attn_bwd_dq_kernel<128>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
    if (e != cudaSuccess) return e;
    attn_bwd_dq_kernel<128><<<grid, kThreads, L::kAlloc, stream>>>(
        tq, tdo, tk64, tv64, stats, delta, dqp, s.Nq, s.Nkv, s.H, s.scale, s.causal, err);
  } else {
    using L = DqLayout<64>;
    cudaError_t e = cudaFuncSetAttribute(attn_bwd_dq_kernel<64>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
    if (e != cudaSuccess) return e;
    attn_bwd_dq_kernel<64><<<grid, kThreads, L::kAlloc, stream>>>(
        tq, tdo, tk64, tv64, stats, delta, dqp, s.Nq, s.Nkv, s.H, s.scale, s.causal, err);
  }
  return cudaGetLastError();
}

}  // namespace nvq
