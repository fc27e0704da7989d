// Attn-QAT straight-through backward on sm_103a, dK/dV part (key-outer), and
// the delta pre-pass.
//
// Kernels, in launch order (the dQ kernel, attn_bwd_dq_fp4.cu, follows them):
//   bwd_prep    delta_i = sum_d dO_id * O_id (fp32)
//   attn_bwd    one CTA per (128-key tile, head, batch); V~ and the K~ codes stay
//               in shared memory, the dK and dV accumulators in TMEM; the CTA
//               loops over the 128-query tiles i:
//                 S  = Q~ K~^T          (block-scaled FP4 UMMA on the codes -> TMEM;
//                                        the same exact products as the forward's)
//                 P  = exp(scale*S - m) (m from the forward)
//                 P~ = fq16(P) per 16 keys (the forward's code, bit for bit)
//                 dP = dO V~^T          (BF16 UMMA -> TMEM, into S's buffer once S
//                                        has been loaded)
//                 A  = P / l,   dS = scale * A * (dP - delta)
//                 P~/l and dS -> shared memory (bf16, a buffer each)
//                 dV += (P~/l)^T dO, dK += dS^T Q~  (BF16 UMMA)
//               then writes dK and dV (bf16).
// ("attn_qat_train" API page, attn_qat_train(): the backward uses the quantized
// Q, K, V and the quantized P, with straight-through gradients.)
// dQ is computed by a separate query-outer kernel rather than added into an
// fp32 accumulator from here: with 128-key tiles those additions would move
// (N/128) x |dQ| bytes through L2 reductions, which cost more than the extra
// S and dP UMMAs of the second kernel.
//
// The elementwise work (exp, the P~ quantization, dS) is the critical path:
// per tile it takes longer than the tensor pipe's 1664 cycles of products.
// Shared memory (V~, K~ codes, 2 slots of Q~ codes, one bf16 Q~ slot for dK,
// 2 dO slots, the P~ and dS buffers) is what lets P~_i and dS_i go out as soon
// as each 32-key chunk is computed, without waiting for the products that read
// the previous tile's buffers; S on FP4 codes is what frees the room for it.
//
// Roles (352 threads, one CTA per SM): warps 0-7 elementwise in two
// warpgroups, each owning 64 keys of the tile (thread t = query row t = TMEM
// lane t for S/dP, key row t for dK/dV); warp 8 TMA; warp 9 TMEM allocation and
// the S and dP UMMAs; warp 10 the dV and dK UMMAs.
// TMEM columns: [0,128) S and dP in turn, [128,136) K~ scales, [136,152) Q~
// scales (2 slots), [256,256+D) dV, [384,384+D) dK.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "nvq_internal.h"
#include "nvq_ptx.cuh"
#include "nvq_quant.cuh"

namespace nvq {

namespace {

constexpr int kElemWarps = 8;  // two elementwise warpgroups
constexpr int kTmaWarp = 8;
constexpr int kMmaWarp = 9;    // S, dP (the shared S/dP TMEM buffer); allocates TMEM
constexpr int kGradWarp = 10;  // dV, dK
constexpr int kThreads = 352;
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint32_t kAtomBlock = 128u * 128u;  // 64-column block of a 128-row bf16 tile
// TMEM columns
constexpr uint32_t kColSP = 0;     // S_i, then dP_i, then S_{i+1} ... (one 128-column buffer)
constexpr uint32_t kColScK = 128;  // K~ scale operand, 4 columns per 64 elements of D
constexpr uint32_t kColScQ = 136;  // Q~ scale operands, 8 columns per slot, 2 slots
constexpr uint32_t kColDV = 256, kColDK = 384;

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// *p (0 where !pred), loaded where the call stands: as a volatile asm the load
// stays ahead of the barrier waits that follow it instead of sinking to its
// first use a tile later, so its latency hides behind a tile of work.
__device__ __forceinline__ float ld_ahead(const float* p, bool pred) {
  float v;
  asm volatile(
      "{\n\t.reg .pred q;\n\t"
      "setp.ne.b32 q, %2, 0;\n\t"
      "mov.b32 %0, 0;\n\t"
      "@q ld.global.nc.f32 %0, [%1];\n\t}"
      : "=f"(v)
      : "l"(p), "r"(static_cast<int>(pred))
      : "memory");
  return v;
}

template <int D>
struct BwdLayout {
  static constexpr uint32_t kTileBytes = 128u * D * 2u;  // a bf16 128-row tile
  static constexpr uint32_t kCodeBytes = 128u * D / 2;   // E2M1 codes of a 128-row tile
  static constexpr uint32_t kScBytes = (D / 64) * 512u;  // its scale blocks
  static constexpr uint32_t kC4 = (kCodeBytes + kScBytes + 1023u) / 1024u * 1024u;
  static constexpr uint32_t kV = 0;                          // V~ (bf16)
  static constexpr uint32_t kK4 = kV + kTileBytes;           // K~ codes + scales
  static constexpr uint32_t kQ4 = kK4 + kC4;                 // [2] Q~ codes + scales
  static constexpr uint32_t kQB = kQ4 + 2u * kC4;            // bf16 Q~ (for dK)
  static constexpr uint32_t kDO = kQB + kTileBytes;          // [2] dO
  static constexpr uint32_t kP = kDO + 2u * kTileBytes;      // P~/l [128 q][128 keys] bf16
  static constexpr uint32_t kDS = kP + 128u * 128u * 2u;     // dS, the same layout
  static constexpr uint32_t kBars = kDS + 128u * 128u * 2u;
  static constexpr uint32_t kNumBars = 24;
  static constexpr uint32_t kTmemSlot = kBars + kNumBars * 8u;
  static constexpr uint32_t kAbort = kTmemSlot + 4u;
  static constexpr uint32_t kUsed = kAbort + 4u;
  static constexpr uint32_t kAlloc = kUsed + 1024u;
  static_assert(kAlloc <= 232448u, "shared memory of one CTA");
};

// One CTA per (128-key tile, head, batch).  tq4, tk4: packed codes of Q~, K~
// (box of D/2 bytes x 128 rows); q_sc, k_sc: their scale blocks per 128-row
// tile; tq, tv, tdo: bf16 Q~, V~, dO (128-row boxes).
template <int D, bool kSparse>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tq4, const __grid_constant__ CUtensorMap tk4,
                    const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tv,
                    const __grid_constant__ CUtensorMap tdo, const uint8_t* __restrict__ q_sc,
                    const uint8_t* __restrict__ k_sc, const float* __restrict__ stats,
                    const float* __restrict__ delta, __nv_bfloat16* __restrict__ dk,
                    __nv_bfloat16* __restrict__ dv, int Nq, int Nkv, int H, float scale,
                    int causal, const int* __restrict__ q_off, const int* __restrict__ q_list,
                    int q_stride, int* __restrict__ err) {
  using L = BwdLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023u) &
                                             ~static_cast<uintptr_t>(1023u));
  const int warp = threadIdx.x >> 5;
  const int kt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int k0 = kt * kTile;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBars);
  uint64_t* kv_full = bars + 0;    // V~, K~ codes and scales
  uint64_t* q4_full = bars + 1;    // [2]
  uint64_t* q4_empty = bars + 3;   // [2]
  uint64_t* do_full = bars + 5;    // [2]
  uint64_t* do_empty = bars + 7;   // [2]
  uint64_t* qb_full = bars + 9;
  uint64_t* qb_empty = bars + 10;
  uint64_t* s_full = bars + 11;    // S_i in TMEM
  uint64_t* s_free = bars + 12;    // every elementwise warp has loaded S_i
  uint64_t* dp_full = bars + 13;   // dP_i in TMEM
  uint64_t* dp_free = bars + 14;   // every elementwise warp has loaded dP_i
  uint64_t* pt_full = bars + 15;   // P~_i/l stored
  uint64_t* pt_free = bars + 16;   // dV += ... of tile i done
  uint64_t* ds_full = bars + 17;   // dS_i stored
  uint64_t* ds_free = bars + 18;   // dK += ... of tile i done
  uint64_t* dkdv_done = bars + 19;
  uint64_t* mma_drain = bars + 20;  // [2]: S/dP warp, dV/dK warp
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + L::kAbort);

  const int n_q_all = (Nq + kTile - 1) / kTile;
  const int n_kt = (Nkv + kTile - 1) / kTile;
  const int64_t bh = static_cast<int64_t>(b) * H + h;
  // query tiles of this key tile: all (dense; causal from the diagonal on, which
  // needs Nq == Nkv) or those whose block-sparse list holds it (q_off/q_list,
  // per (b, h): offsets [n_kt + 1] and query tiles in ascending order)
  const int i_begin = causal ? kt : 0;
  const int* qsel = nullptr;
  int n_iter = n_q_all - i_begin;
  if (kSparse) {
    const int* off = q_off + bh * (n_kt + 1);
    qsel = q_list + bh * q_stride + off[kt];
    n_iter = off[kt + 1] - off[kt];
  }
  auto qtile = [&](int it) -> int { return kSparse ? qsel[it] : i_begin + it; };

  if (threadIdx.x == 0) {
    *abort = 0;
    mbar_init(kv_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&q4_full[s], 1);
      mbar_init(&q4_empty[s], 1);
      mbar_init(&do_full[s], 1);
      mbar_init(&do_empty[s], 2);  // dP and dV both read dO
    }
    mbar_init(qb_full, 1);
    mbar_init(qb_empty, 1);
    mbar_init(s_full, 1);
    mbar_init(s_free, kElemWarps);
    mbar_init(dp_full, 1);
    mbar_init(dp_free, kElemWarps);
    mbar_init(pt_full, kElemWarps);
    mbar_init(pt_free, 1);
    mbar_init(ds_full, kElemWarps);
    mbar_init(ds_free, 1);
    mbar_init(dkdv_done, 1);
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
    // V~ and the K~ codes once; Q~ codes and dO one tile ahead of the UMMAs
    // (two slots each); bf16 Q~ (one slot, read only by dK) for the current tile.
    tma_prefetch_desc(&tq4);
    tma_prefetch_desc(&tk4);
    tma_prefetch_desc(&tq);
    tma_prefetch_desc(&tv);
    tma_prefetch_desc(&tdo);
    mbar_arrive_expect_tx_w(kv_full, L::kTileBytes + L::kCodeBytes + L::kScBytes);
#pragma unroll
    for (int blk = 0; blk < D / 64; ++blk)
      tma_load_4d_w(smem + L::kV + blk * kAtomBlock, &tv, blk * 64, k0, h, b, kv_full);
    tma_load_4d_w(smem + L::kK4, &tk4, 0, k0, h, b, kv_full);
    bulk_load_w(smem + L::kK4 + L::kCodeBytes, k_sc + (bh * n_kt + kt) * L::kScBytes,
                L::kScBytes, kv_full);
    int last_q4[2] = {-1, -1}, last_do[2] = {-1, -1}, last_qb = -1;
    bool ok = true;
    auto load_q4_do = [&](int it) -> bool {  // Q~ codes and dO of tile it into slot it & 1
      const int st = it & 1;
      const uint32_t u = static_cast<uint32_t>((it >> 1) & 1);
      const int qt = qtile(it);
      if (!mbar_wait_warp(&q4_empty[st], u ^ 1u, abort)) return false;
      uint8_t* q4dst = smem + L::kQ4 + st * L::kC4;
      mbar_arrive_expect_tx_w(&q4_full[st], L::kCodeBytes + L::kScBytes);
      tma_load_4d_w(q4dst, &tq4, 0, qt * kTile, h, b, &q4_full[st]);
      bulk_load_w(q4dst + L::kCodeBytes, q_sc + (bh * n_q_all + qt) * L::kScBytes, L::kScBytes,
                  &q4_full[st]);
      last_q4[st] = static_cast<int>(u);
      if (!mbar_wait_warp(&do_empty[st], u ^ 1u, abort)) return false;
      mbar_arrive_expect_tx_w(&do_full[st], L::kTileBytes);
#pragma unroll
      for (int blk = 0; blk < D / 64; ++blk)
        tma_load_4d_w(smem + L::kDO + st * L::kTileBytes + blk * kAtomBlock, &tdo, blk * 64,
                      qt * kTile, h, b, &do_full[st]);
      last_do[st] = static_cast<int>(u);
      return true;
    };
    if (n_iter > 0) ok = load_q4_do(0);
    for (int it = 0; it < n_iter && ok; ++it) {
      if (it + 1 < n_iter && !(ok = load_q4_do(it + 1))) break;
      const uint32_t u = static_cast<uint32_t>(it & 1);
      if (!(ok = mbar_wait_warp(qb_empty, u ^ 1u, abort))) break;
      mbar_arrive_expect_tx_w(qb_full, L::kTileBytes);
#pragma unroll
      for (int blk = 0; blk < D / 64; ++blk)
        tma_load_4d_w(smem + L::kQB + blk * kAtomBlock, &tq, blk * 64, qtile(it) * kTile, h, b,
                      qb_full);
      last_qb = static_cast<int>(u);
    }
    if (!ok) {  // let the loads already issued land before the block exits
      mbar_wait_warp(kv_full, 0, nullptr, 10000000ull);
      for (int s = 0; s < 2; ++s) {
        if (last_q4[s] >= 0)
          mbar_wait_warp(&q4_full[s], static_cast<uint32_t>(last_q4[s]), nullptr, 10000000ull);
        if (last_do[s] >= 0)
          mbar_wait_warp(&do_full[s], static_cast<uint32_t>(last_do[s]), nullptr, 10000000ull);
      }
      if (last_qb >= 0) mbar_wait_warp(qb_full, static_cast<uint32_t>(last_qb), nullptr, 10000000ull);
    }
  } else if (warp == kMmaWarp || warp == kGradWarp) {
    // ---------------------------------------------------------------- MMA
    // Two issuing warps, as each tcgen05 instruction and mbarrier wait costs
    // its warp tens of cycles and one warp issuing all four products per tile
    // was the critical path.  kMmaWarp: dP_i once the elementwise warps have
    // loaded S_i, S_{i+1} once they have loaded dP_i (S and dP share one TMEM
    // buffer); so dP_i runs while they turn S_i into P~_i, S_{i+1} while they
    // turn dP_i into dS_i.  kGradWarp: dK_{i-1} once dS_{i-1} is stored, dV_i
    // once P~_i is.  The two touch disjoint TMEM; dO's slot is released by
    // both (dP and dV read it).
    constexpr uint32_t idesc_s4 = idesc_mxf4nvf4(128, 128);     // S (FP4, N = 128 keys)
    constexpr uint32_t idesc_p = idesc_f16(128, 128, 1, 0, 0);  // dP (N = 128 keys)
    constexpr uint32_t idesc_t = idesc_f16(128, D, 1, 1, 1);    // dV, dK (A, B MN-major)
    constexpr uint32_t lay = D == 128 ? 4u : 6u;                // (D/2)-byte swizzle of code rows
    constexpr uint32_t sbo = 8u * (D / 2);
    const uint32_t v_addr = smem_u32(smem + L::kV);
    const uint32_t k4_addr = smem_u32(smem + L::kK4);
    const uint32_t q4_addr = smem_u32(smem + L::kQ4);
    const uint32_t qb_addr = smem_u32(smem + L::kQB);
    const uint32_t do_addr = smem_u32(smem + L::kDO);
    const uint32_t p_addr = smem_u32(smem + L::kP);
    const uint32_t ds_addr = smem_u32(smem + L::kDS);
    // Descriptors of every operand the UMMAs read, computed once: a K step
    // moves a descriptor's start address (bits 0-13, address / 16) by the
    // step's byte offset / 16, with no carry out of the field (shared-memory
    // addresses stay below 2^18).
    auto koff = [](int kk) {  // K-major bf16 tile: K step kk (16 elements)
      return static_cast<uint32_t>((kk >> 2) * kAtomBlock + (kk & 3) * 32);
    };
    // S_{it} from slot it & 1: the copy of its Q~ scales to TMEM (their columns
    // were last read by S_{it-2}, complete since dP_{it-1} was issued after
    // S_{it-1} had been loaded) is issued before the wait for the S/dP buffer,
    // then the UMMAs and their commits as one group
    auto prep_s = [&](int it) -> bool {
      const int st = it & 1;
      if (!mbar_wait_warp(&q4_full[st], static_cast<uint32_t>((it >> 1) & 1), abort)) return false;
      tc_fence_after();
      const uint32_t qa = q4_addr + st * L::kC4;
      const uint32_t sc = kColScQ + 8u * static_cast<uint32_t>(st);
#pragma unroll
      for (int kk = 0; kk < D / 64; ++kk)
        tmem_cp_32x128_x4_w(tmem + sc + 4 * kk, qa + L::kCodeBytes + kk * 512);
      return true;
    };
    uint64_t s_ad[2][D / 64], s_bd[D / 64];
#pragma unroll
    for (int kk = 0; kk < D / 64; ++kk) {
      s_bd[kk] = sdesc(k4_addr + 32 * kk, 16, sbo, lay);
#pragma unroll
      for (int st = 0; st < 2; ++st) s_ad[st][kk] = sdesc(q4_addr + st * L::kC4 + 32 * kk, 16, sbo, lay);
    }
    // (the slot is a branch, not an index, so the descriptors stay in registers)
    auto fire_s = [&](int it) {
      if (it & 1)
        umma_fp4_group_w<D / 64>(tmem + kColSP, s_ad[1], s_bd, idesc_s4, tmem + kColScQ + 8u,
                                 tmem + kColScK, bar_u32(s_full), bar_u32(&q4_empty[1]));
      else
        umma_fp4_group_w<D / 64>(tmem + kColSP, s_ad[0], s_bd, idesc_s4, tmem + kColScQ,
                                 tmem + kColScK, bar_u32(s_full), bar_u32(&q4_empty[0]));
    };
    const int w = warp == kMmaWarp ? 0 : 1;
    bool ok = true;
    if (w == 0) {
      // dP = dO V~^T, contraction over D
      uint64_t dp_ad[2][D / 16], dp_bd[D / 16];
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        dp_bd[kk] = sdesc_sw128(v_addr + koff(kk), 16, 1024);
#pragma unroll
        for (int st = 0; st < 2; ++st)
          dp_ad[st][kk] = sdesc_sw128(do_addr + st * L::kTileBytes + koff(kk), 16, 1024);
      }
      ok = mbar_wait_warp(kv_full, 0, abort) && n_iter > 0;
      if (ok) {  // the K~ scales stay in TMEM for the whole kernel
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 64; ++kk)
          tmem_cp_32x128_x4_w(tmem + kColScK + 4 * kk, k4_addr + L::kCodeBytes + kk * 512);
        if ((ok = prep_s(0))) fire_s(0);
      }
      for (int it = 0; it < n_iter && ok; ++it) {
        const uint32_t ph = static_cast<uint32_t>(it & 1);
        const int st = it & 1;
        // dO of this tile (loaded long before) first, then the buffer
        if (!(ok = mbar_wait_warp(&do_full[st], static_cast<uint32_t>((it >> 1) & 1), abort)))
          break;
        if (!(ok = mbar_wait_warp(s_free, ph, abort))) break;
        tc_fence_after();
        if (st)
          umma_f16_group_w<D / 16>(tmem + kColSP, dp_ad[1], dp_bd, idesc_p, 0u, bar_u32(dp_full),
                                   bar_u32(&do_empty[1]));
        else
          umma_f16_group_w<D / 16>(tmem + kColSP, dp_ad[0], dp_bd, idesc_p, 0u, bar_u32(dp_full),
                                   bar_u32(&do_empty[0]));
        if (it + 1 < n_iter) {
          if (!(ok = prep_s(it + 1))) break;
          if (!(ok = mbar_wait_warp(dp_free, ph, abort))) break;
          tc_fence_after();
          fire_s(it + 1);
        }
      }
    } else {
      // dV += (P~/l)^T dO and dK += dS^T Q~, contractions over the 128 queries
      // of a tile (MN-major operands, K step kk at 2048 kk bytes)
      uint64_t dv_ad[8], dv_bd[2][8], dk_ad[8], dk_bd[8];
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        dv_ad[kk] = sdesc_sw128(p_addr + kk * 2048, kAtomBlock, 1024);
        dk_ad[kk] = sdesc_sw128(ds_addr + kk * 2048, kAtomBlock, 1024);
        dk_bd[kk] = sdesc_sw128(qb_addr + kk * 2048, kAtomBlock, 1024);
#pragma unroll
        for (int st = 0; st < 2; ++st)
          dv_bd[st][kk] = sdesc_sw128(do_addr + st * L::kTileBytes + kk * 2048, kAtomBlock, 1024);
      }
      auto issue_dk = [&](int it) -> bool {  // dK += dS^T Q~ (bf16 Q~ first: loaded earlier)
        if (!mbar_wait_warp(qb_full, static_cast<uint32_t>(it & 1), abort) ||
            !mbar_wait_warp(ds_full, static_cast<uint32_t>(it & 1), abort))
          return false;
        tc_fence_after();
        umma_f16_group_w<8>(tmem + kColDK, dk_ad, dk_bd, idesc_t, it > 0 ? 1u : 0u,
                            bar_u32(ds_free), bar_u32(qb_empty));
        return true;
      };
      for (int it = 0; it < n_iter && ok; ++it) {
        if (it > 0 && !(ok = issue_dk(it - 1))) break;
        const int st = it & 1;
        if (!(ok = mbar_wait_warp(&do_full[st], static_cast<uint32_t>((it >> 1) & 1), abort)) ||
            !(ok = mbar_wait_warp(pt_full, static_cast<uint32_t>(it & 1), abort)))
          break;
        tc_fence_after();
        if (st)
          umma_f16_group_w<8>(tmem + kColDV, dv_ad, dv_bd[1], idesc_t, 1u, bar_u32(pt_free),
                              bar_u32(&do_empty[1]));
        else
          umma_f16_group_w<8>(tmem + kColDV, dv_ad, dv_bd[0], idesc_t, it > 0 ? 1u : 0u,
                              bar_u32(pt_free), bar_u32(&do_empty[0]));
      }
      if (ok && n_iter > 0 && (ok = issue_dk(n_iter - 1))) umma_commit_w(dkdv_done);
    }
    umma_commit_w(&mma_drain[w]);
    mbar_wait_warp(&mma_drain[w], 0, nullptr, 10000000ull);
  } else {
    // --------------------------------------------------------- elementwise
    // Warpgroup hg (0, 1) owns keys [64hg, 64hg+64) of every tile as two
    // 32-key chunks; thread t of the group owns query row t (TMEM lane t).
    // Each chunk's P~/l and dS go to shared memory as soon as they are
    // computed (P~ and dS have a buffer each).  dS is stored pre-multiplied by
    // `scale`, so dK comes out scaled.
    const int hg = warp >> 2;
    const int t = threadIdx.x & 127;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const float c1 = scale * kLog2e;
    uint8_t* p_smem = smem + L::kP;
    uint8_t* ds_smem = smem + L::kDS;
    const float* lse_g = stats + bh * 2 * Nq;
    const float* m_g = lse_g + Nq;
    const float* delta_g = delta + bh * Nq;
    const uint32_t key_col = static_cast<uint32_t>(hg * 64);
    bool ok = true;
    uint32_t r[2][32];
    // statistics of this thread's row, prefetched one tile ahead
    auto load_row = [&](int it, float& m, float& lse, float& dl) {
      const int qrow = (it < n_iter ? qtile(it) : 0) * kTile + t;
      const bool in = it < n_iter && qrow < Nq;
      const int qr = in ? qrow : 0;
      m = ld_ahead(m_g + qr, in);
      lse = ld_ahead(lse_g + qr, in);
      dl = ld_ahead(delta_g + qr, in);
    };
    float nm, nlse, ndl;
    load_row(0, nm, nlse, ndl);
    for (int it = 0; it < n_iter && ok; ++it) {
      const int qi = qtile(it);
      const int qrow = qi * kTile + t;
      const bool row_ok = qrow < Nq;
      const float m = nm, lse = nlse, dl = ndl;
      load_row(it + 1, nm, nlse, ndl);
      const float negmb = -m * kLog2e;
      const uint64_t c12 = pk2(c1, c1), nmb2 = pk2(negmb, negmb);
      const float inv_l = ex2((m - lse) * kLog2e);  // 1 / l
      const bool edge = !row_ok || (k0 + kTile > Nkv) || (causal && qi == kt);
      const uint32_t ph = static_cast<uint32_t>(it & 1);
      // ---- P part: S -> P, P~/l
      if (!(ok = mbar_wait_warp(s_full, ph, abort))) break;
      tc_fence_after();
      tmem_ld32(tmem + lane_base + kColSP + key_col, r[0]);
      tmem_ld32(tmem + lane_base + kColSP + key_col + 32, r[1]);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive_warp(s_free);
      // the P~ buffer is free once dV of the previous tile is done
      if (it > 0 && !(ok = mbar_wait_warp(pt_free, ph ^ 1u, abort))) break;
      float pp[4][16];  // P (fp32) of this thread's 64 keys, for dS
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        float x[32];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          up2(fma2(pk2(__uint_as_float(r[c][2 * i]), __uint_as_float(r[c][2 * i + 1])), c12, nmb2),
              x[2 * i], x[2 * i + 1]);
        if (edge) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int key = k0 + key_col + 32 * c + i;
            if (!(row_ok && key < Nkv && (!causal || key <= qrow))) x[i] = -INFINITY;
          }
        }
        uint32_t ptw[2][8];  // P~ / l as bf16x2
        pquant16_scaled_bf16(x, inv_l, pp[2 * c], ptw[0]);
        pquant16_scaled_bf16(x + 16, inv_l, pp[2 * c + 1], ptw[1]);
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          const uint32_t* w = ptw[ch >> 1] + 4 * (ch & 1);
          const uint32_t off = sw128_offset(t, key_col + 32 * c + ch * 8, 128);
          *reinterpret_cast<uint4*>(p_smem + off) = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
      // ---- dS part: dP -> dS = scale * A * (dP - delta), A = P / l
      // The first dP load is issued before the P~ stores are fenced, so the
      // fence's wait for the stores overlaps the load (dP_i is issued when S_i
      // has been loaded, long before this point).
      if (!(ok = mbar_wait_warp(dp_full, ph, abort))) break;
      tc_fence_after();
      // dP one 32-key chunk at a time: the second load waits until the first
      // chunk's P values are consumed, which keeps the register peak (all 64 P
      // values and 64 dP values at once) under what 320 threads may hold
      tmem_ld32(tmem + lane_base + kColSP + key_col, r[0]);
      fence_proxy_async_smem();
      mbar_arrive_warp(pt_full);
      tmem_wait_ld();
      // the dS buffer is free once dK of the previous tile is done
      if (it > 0 && !(ok = mbar_wait_warp(ds_free, ph ^ 1u, abort))) break;
      {
        // dS = P * (sl * dP - sl * delta) with sl = scale / l
        const float sl = scale * inv_l;
        const uint64_t sl2 = pk2(sl, sl), nsd2 = pk2(-sl * dl, -sl * dl);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if (q == 2) {
            tmem_ld32(tmem + lane_base + kColSP + key_col + 32, r[0]);
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive_warp(dp_free);
          }
          uint32_t dsw[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const uint32_t* rr = r[0] + 16 * (q & 1);
            const uint64_t t2 =
                fma2(pk2(__uint_as_float(rr[2 * u]), __uint_as_float(rr[2 * u + 1])), sl2, nsd2);
            float d0, d1;
            up2(mul2(pk2(pp[q][2 * u], pp[q][2 * u + 1]), t2), d0, d1);
            dsw[u] = pack_bf16(d0, d1);
          }
#pragma unroll
          for (int ch = 0; ch < 2; ++ch) {
            const uint32_t off = sw128_offset(t, key_col + 16 * q + ch * 8, 128);
            *reinterpret_cast<uint4*>(ds_smem + off) =
                make_uint4(dsw[4 * ch], dsw[4 * ch + 1], dsw[4 * ch + 2], dsw[4 * ch + 3]);
          }
        }
      }
      fence_proxy_async_smem();
      mbar_arrive_warp(ds_full);
    }
    if (ok && n_iter > 0 && (ok = mbar_wait_warp(dkdv_done, 0, abort))) {
      tc_fence_after();
      // group 0 writes dV, group 1 dK (already scaled); thread t = key row t
      const int key = k0 + t;
      const int64_t base = ((static_cast<int64_t>(b) * Nkv + key) * H + h) * D;
      __nv_bfloat16* dst = (hg == 0 ? dv : dk) + base;
      const uint32_t col = hg == 0 ? kColDV : kColDK;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        tmem_ld32(tmem + lane_base + col + c * 32, r[0]);
        tmem_wait_ld();
        if (key < Nkv) {
          uint32_t w[16];
#pragma unroll
          for (int u = 0; u < 16; ++u)
            w[u] = pack_bf16(__uint_as_float(r[0][2 * u]), __uint_as_float(r[0][2 * u + 1]));
          uint4* pw = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
          for (int u = 0; u < 4; ++u)
            pw[u] = make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
        }
      }
    } else if (ok && n_iter == 0) {
      // no query attends this key tile: zero gradients
      const int key = k0 + t;
      if (key < Nkv) {
        const int64_t base = ((static_cast<int64_t>(b) * Nkv + key) * H + h) * D;
        __nv_bfloat16* dst = (hg == 0 ? dv : dk) + base;
        for (int c = 0; c < D; c += 8)
          *reinterpret_cast<uint4*>(dst + c) = make_uint4(0, 0, 0, 0);
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

// delta[b,h,i] = sum_d dO[b,i,h,d] * O[b,i,h,d].
template <int D>
__global__ void __launch_bounds__(256) bwd_prep_kernel(const __nv_bfloat16* __restrict__ o,
                                                       const __nv_bfloat16* __restrict__ dout,
                                                       float* __restrict__ delta, int B, int Nq,
                                                       int H) {
  // 8 threads per (b, i, h) row; each takes D/8 consecutive elements.
  const int64_t rows = static_cast<int64_t>(B) * Nq * H;
  const int64_t gt = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t row = gt >> 3;
  const int part = static_cast<int>(gt & 7);
  float acc = 0.f;
  if (row < rows) {
    constexpr int E = D / 8;
    const int64_t off = row * D + part * E;
#pragma unroll
    for (int c = 0; c < E; c += 8) {
      const uint4 a = *reinterpret_cast<const uint4*>(o + off + c);
      const uint4 g = *reinterpret_cast<const uint4*>(dout + off + c);
      const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, gw[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        acc = fmaf(__uint_as_float(aw[u] << 16), __uint_as_float(gw[u] << 16), acc);
        acc = fmaf(__uint_as_float(aw[u] & 0xFFFF0000u), __uint_as_float(gw[u] & 0xFFFF0000u),
                   acc);
      }
    }
  }
  acc += __shfl_xor_sync(0xFFFFFFFFu, acc, 1);
  acc += __shfl_xor_sync(0xFFFFFFFFu, acc, 2);
  acc += __shfl_xor_sync(0xFFFFFFFFu, acc, 4);
  if (row < rows && part == 0) {
    const int64_t hh = row % H;
    const int64_t bi = row / H;  // b * Nq + i
    const int64_t i = bi % Nq;
    const int64_t bb = bi / Nq;
    delta[(bb * H + hh) * Nq + i] = acc;
  }
}

// Block-sparse lists transposed, per (b, h) (grid (H, B)): for each key tile
// the query tiles whose list holds it, in ascending order: offsets
// q_off[n_kt + 1] and entries q_list[<= n_qt * topk].  A list that names a key
// tile twice counts it once.  This form rescans the lists per key tile; it
// serves lists whose bitmap (below) would not fit in shared memory.
__global__ void __launch_bounds__(256) tile_transpose_scan_kernel(const int* __restrict__ kv_list,
                                                             int H, int n_qt, int n_kt, int topk,
                                                             int* __restrict__ q_off,
                                                             int* __restrict__ q_list) {
  extern __shared__ int start[];  // [n_kt + 1]
  const int64_t head = static_cast<int64_t>(blockIdx.y) * H + blockIdx.x;
  const int* lst = kv_list + head * n_qt * topk;
  auto holds = [&](int i, int kt) {
    for (int e = 0; e < topk; ++e)
      if (lst[i * topk + e] == kt) return true;
    return false;
  };
  for (int kt = threadIdx.x; kt < n_kt; kt += blockDim.x) {
    int c = 0;
    for (int i = 0; i < n_qt; ++i) c += holds(i, kt) ? 1 : 0;
    start[kt] = c;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int kt = 0; kt < n_kt; ++kt) {
      const int c = start[kt];
      start[kt] = acc;
      acc += c;
    }
    start[n_kt] = acc;
  }
  __syncthreads();
  int* off = q_off + head * (n_kt + 1);
  for (int kt = threadIdx.x; kt <= n_kt; kt += blockDim.x) off[kt] = start[kt];
  int* out = q_list + head * n_qt * topk;
  for (int kt = threadIdx.x; kt < n_kt; kt += blockDim.x) {
    int pos = start[kt];
    for (int i = 0; i < n_qt; ++i)
      if (holds(i, kt)) out[pos++] = i;
  }
}

// The same transpose through a bitmap in shared memory: bit i of row kt says
// that query tile i's list holds key tile kt (entries outside [0, n_kt) are
// ignored, repeats set the same bit).  Then one warp per key tile counts its
// row, one warp forms the offsets, and one warp per key tile writes its query
// tiles in ascending order.  Grid (H, B), 512 threads.
__global__ void __launch_bounds__(512) tile_transpose_kernel(const int* __restrict__ kv_list,
                                                             int H, int n_qt, int n_kt, int topk,
                                                             int* __restrict__ q_off,
                                                             int* __restrict__ q_list) {
  extern __shared__ uint32_t tt_smem[];
  const int words = (n_qt + 31) / 32;
  uint32_t* bits = tt_smem;                                    // [n_kt][words]
  int* start = reinterpret_cast<int*>(tt_smem + n_kt * words);  // [n_kt + 1]
  const int64_t head = static_cast<int64_t>(blockIdx.y) * H + blockIdx.x;
  const int* lst = kv_list + head * n_qt * topk;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
  for (int i = tid; i < n_kt * words; i += blockDim.x) bits[i] = 0u;
  __syncthreads();
  for (int e = tid; e < n_qt * topk; e += blockDim.x) {
    const int i = e / topk, kt = lst[e];
    if (kt >= 0 && kt < n_kt) atomicOr(&bits[kt * words + (i >> 5)], 1u << (i & 31));
  }
  __syncthreads();
  for (int kt = warp; kt < n_kt; kt += nwarps) {
    int c = 0;
    for (int w = lane; w < words; w += 32) c += __popc(bits[kt * words + w]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xFFFFFFFFu, c, o);
    if (lane == 0) start[kt] = c;
  }
  __syncthreads();
  if (warp == 0) {  // exclusive prefix sum, 32 key tiles at a time
    int carry = 0;
    for (int base = 0; base < n_kt; base += 32) {
      const int v = base + lane < n_kt ? start[base + lane] : 0;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += y;
      }
      if (base + lane < n_kt) start[base + lane] = carry + incl - v;
      carry += __shfl_sync(0xFFFFFFFFu, incl, 31);
    }
    if (lane == 0) start[n_kt] = carry;
  }
  __syncthreads();
  int* off = q_off + head * (n_kt + 1);
  for (int kt = tid; kt <= n_kt; kt += blockDim.x) off[kt] = start[kt];
  int* out = q_list + head * n_qt * topk;
  for (int kt = warp; kt < n_kt; kt += nwarps) {
    int pos = start[kt];
    for (int w0 = 0; w0 < words; w0 += 32) {
      const int w = w0 + lane;
      uint32_t m = w < words ? bits[kt * words + w] : 0u;
      const int c = __popc(m);
      int incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += y;
      }
      int p = pos + incl - c;
      while (m != 0u) {
        out[p++] = w * 32 + __ffs(m) - 1;
        m &= m - 1u;
      }
      pos += __shfl_sync(0xFFFFFFFFu, incl, 31);
    }
  }
}

}  // namespace

cudaError_t launch_tile_transpose(const int* kv_list, int B, int H, int n_qt, int n_kt, int topk,
                                  int* q_off, int* q_list, cudaStream_t stream) {
  const size_t words = static_cast<size_t>(n_qt + 31) / 32;
  const size_t smem = (static_cast<size_t>(n_kt) * words + n_kt + 1) * sizeof(uint32_t);
  if (smem <= 48 * 1024) {
    tile_transpose_kernel<<<dim3(H, B), 512, smem, stream>>>(kv_list, H, n_qt, n_kt, topk, q_off,
                                                             q_list);
    return cudaGetLastError();
  }
  const size_t smem_scan = static_cast<size_t>(n_kt + 1) * sizeof(int);
  if (smem_scan > 48 * 1024) return cudaErrorInvalidValue;
  tile_transpose_scan_kernel<<<dim3(H, B), 256, smem_scan, stream>>>(kv_list, H, n_qt, n_kt, topk,
                                                                     q_off, q_list);
  return cudaGetLastError();
}

cudaError_t launch_bwd_prep(const AttnShape& s, const void* o, const void* dout, float* delta,
                            cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(s.B) * s.Nq * s.H;
  const int64_t threads = rows * 8;
  const int grid = static_cast<int>((threads + 255) / 256);
  const auto* op = static_cast<const __nv_bfloat16*>(o);
  const auto* gp = static_cast<const __nv_bfloat16*>(dout);
  if (s.D == 128)
    bwd_prep_kernel<128><<<grid, 256, 0, stream>>>(op, gp, delta, s.B, s.Nq, s.H);
  else
    bwd_prep_kernel<64><<<grid, 256, 0, stream>>>(op, gp, delta, s.B, s.Nq, s.H);
  return cudaGetLastError();
}

template <int D, bool kSparse>
cudaError_t launch_bwd_t(const AttnShape& s, const CUtensorMap& tq4, const CUtensorMap& tk4,
                         const CUtensorMap& tq, const CUtensorMap& tv, const CUtensorMap& tdo,
                         const uint8_t* q_sc, const uint8_t* k_sc, const float* stats,
                         const float* delta, void* dk, void* dv, const int* q_off,
                         const int* q_list, int q_stride, int* err, cudaStream_t stream) {
  using L = BwdLayout<D>;
  const dim3 grid((s.Nkv + kTile - 1) / kTile, s.H, s.B);
  cudaError_t e = cudaFuncSetAttribute(attn_bwd_kernel<D, kSparse>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (e != cudaSuccess) return e;
  attn_bwd_kernel<D, kSparse><<<grid, kThreads, L::kAlloc, stream>>>(
      tq4, tk4, tq, tv, tdo, q_sc, k_sc, stats, delta, static_cast<__nv_bfloat16*>(dk),
      static_cast<__nv_bfloat16*>(dv), s.Nq, s.Nkv, s.H, s.scale, s.causal, q_off, q_list,
      q_stride, err);
  return cudaGetLastError();
}

cudaError_t launch_attn_bwd(const AttnShape& s, const CUtensorMap& tq4, const CUtensorMap& tk4,
                            const CUtensorMap& tq, const CUtensorMap& tv, const CUtensorMap& tdo,
                            const uint8_t* q_sc, const uint8_t* k_sc, const float* stats,
                            const float* delta, void* dk, void* dv, const int* q_off,
                            const int* q_list, int q_stride, int* err, cudaStream_t stream) {
  const bool sp = q_off != nullptr;
  auto go = [&](auto fn) {
    return fn(s, tq4, tk4, tq, tv, tdo, q_sc, k_sc, stats, delta, dk, dv, q_off, q_list, q_stride,
              err, stream);
  };
  if (s.D == 128) return sp ? go(launch_bwd_t<128, true>) : go(launch_bwd_t<128, false>);
  return sp ? go(launch_bwd_t<64, true>) : go(launch_bwd_t<64, false>);
}

}  // namespace nvq
