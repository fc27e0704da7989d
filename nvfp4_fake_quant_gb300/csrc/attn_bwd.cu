// Attn-QAT straight-through backward on sm_103a, dK/dV part (key-outer), and
// the delta pre-pass.
//
// Kernels, in launch order (the dQ kernel, attn_bwd_dq_fp4.cu, follows them):
//   bwd_prep    delta_i = sum_d dO_id * O_id (fp32)
//   attn_bwd    one CTA per (128-key tile, head, batch); K~ and V~ stay in shared
//               memory, the dK and dV accumulators in TMEM; the CTA loops over the
//               128-query tiles:
//                 S  = Q~ K~^T, dP = dO V~^T              (BF16 UMMA -> TMEM)
//                 P  = exp(scale*S - m)                    (m from the forward)
//                 P~ = fq16(P) per 16 keys                 (the forward's code; S here
//                                                           from BF16 UMMAs, the forward's
//                                                           from FP4 ones: equal up to the
//                                                           fp32 summation order)
//                 A  = P / l,   dS = scale * A * (dP - delta)
//                 P~/l and dS -> shared memory (bf16, one buffer used in turn)
//                 dV += (P~/l)^T dO, dK += dS^T Q~         (BF16 UMMA)
//               then writes dK and dV (bf16).
// ("attn_qat_train" API page, attn_qat_train(): the backward uses the quantized
// Q, K, V and the quantized P, with straight-through gradients.)
// dQ is computed by a separate query-outer kernel rather than added into an
// fp32 accumulator from here: with 128-key tiles those additions would move
// (N/128) x |dQ| bytes through L2 reductions, which cost more than the extra
// S and dP UMMAs of the second kernel.
//
// Roles (576 threads, one CTA per SM): warps 0-15 elementwise in four
// warpgroups, each owning 32 keys of the tile (thread t = query row t = TMEM
// lane t for S/dP, key row t for dK/dV), warp 16 TMA, warp 17 TMEM allocation
// and UMMA issue.
// TMEM columns: [0,128) S, [128,256) dP, [256,256+D) dV, [384,384+D) dK.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "nvq_internal.h"
#include "nvq_ptx.cuh"
#include "nvq_quant.cuh"

namespace nvq {

namespace {

constexpr int kElemWarps = 16;  // four elementwise warpgroups
constexpr int kTmaWarp = 16;
constexpr int kMmaWarp = 17;
constexpr int kThreads = 576;
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint32_t kAtomBlock = 128u * 128u;

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

template <int D>
struct BwdLayout {
  static constexpr uint32_t kTileBytes = 128u * D * 2u;
  static constexpr uint32_t kK = 0;
  static constexpr uint32_t kV = kK + kTileBytes;
  static constexpr uint32_t kQ = kV + kTileBytes;        // [2] stages
  static constexpr uint32_t kDO = kQ + 2u * kTileBytes;  // [2] stages
  static constexpr uint32_t kPD = kDO + 2u * kTileBytes; // P~/l, then dS: [128 q][128 keys] bf16
  static constexpr uint32_t kBars = kPD + 128u * 128u * 2u;
  static constexpr uint32_t kNumBars = 16;
  static constexpr uint32_t kStats = kBars + kNumBars * 8u;  // unused padding slot
  static constexpr uint32_t kTmemSlot = kStats + 8u;
  static constexpr uint32_t kAbort = kTmemSlot + 4u;
  static constexpr uint32_t kUsed = kAbort + 4u;
  static constexpr uint32_t kAlloc =
      (kUsed + 1024u) > 150u * 1024u ? (kUsed + 1024u) : 150u * 1024u;
};

template <int D, bool kSparse>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                    const float* __restrict__ stats, const float* __restrict__ delta,
                    __nv_bfloat16* __restrict__ dk,
                    __nv_bfloat16* __restrict__ dv, int Nq, int Nkv, int H, float scale,
                    int causal, const int* __restrict__ q_off, const int* __restrict__ q_list,
                    int q_stride, int* __restrict__ err) {
  using L = BwdLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023u) &
                                             ~static_cast<uintptr_t>(1023u));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int kt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int k0 = kt * kTile;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBars);
  uint64_t* kv_full = bars + 0;
  uint64_t* qdo_full = bars + 1;   // [2]
  uint64_t* qdo_empty = bars + 3;  // [2]
  uint64_t* s_full = bars + 5;
  uint64_t* dp_full = bars + 6;
  uint64_t* pt_full = bars + 7;
  uint64_t* pt_free = bars + 8;
  uint64_t* ds_full = bars + 9;
  uint64_t* ds_free = bars + 10;
  uint64_t* dkdv_done = bars + 11;
  uint64_t* mma_drain = bars + 12;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + L::kAbort);

  const int n_q_all = (Nq + kTile - 1) / kTile;
  // query tiles of this key tile: all (dense; causal from the diagonal on, which
  // needs Nq == Nkv) or those whose block-sparse list holds it (q_off/q_list,
  // per (b, h): offsets [n_kt + 1] and query tiles in ascending order)
  const int i_begin = causal ? kt : 0;
  const int* qsel = nullptr;
  int n_iter = n_q_all - i_begin;
  if (kSparse) {
    const int n_kt = (Nkv + kTile - 1) / kTile;
    const int64_t head = static_cast<int64_t>(b) * H + h;
    const int* off = q_off + head * (n_kt + 1);
    qsel = q_list + head * q_stride + off[kt];
    n_iter = off[kt + 1] - off[kt];
  }
  auto qtile = [&](int it) -> int { return kSparse ? qsel[it] : i_begin + it; };


  if (threadIdx.x == 0) {
    *abort = 0;
    mbar_init(kv_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&qdo_full[s], 1);
      mbar_init(&qdo_empty[s], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(dp_full, 1);
    mbar_init(pt_full, kElemWarps);
    mbar_init(pt_free, 1);
    mbar_init(ds_full, kElemWarps);
    mbar_init(ds_free, 1);
    mbar_init(dkdv_done, 1);
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
    tma_prefetch_desc(&tq);
    tma_prefetch_desc(&tk);
    tma_prefetch_desc(&tv);
    tma_prefetch_desc(&tdo);
    mbar_arrive_expect_tx_w(kv_full, 2u * L::kTileBytes);
#pragma unroll
    for (int blk = 0; blk < D / 64; ++blk) {
      tma_load_4d_w(smem + L::kK + blk * kAtomBlock, &tk, blk * 64, k0, h, b, kv_full);
      tma_load_4d_w(smem + L::kV + blk * kAtomBlock, &tv, blk * 64, k0, h, b, kv_full);
    }
    int last[2] = {-1, -1};
    bool ok = true;
    for (int it = 0; it < n_iter; ++it) {
      const int st = it & 1;
      if (!(ok = mbar_wait_warp(&qdo_empty[st], ((it >> 1) & 1) ^ 1, abort))) break;
      const int qrow0 = qtile(it) * kTile;
      mbar_arrive_expect_tx_w(&qdo_full[st], 2u * L::kTileBytes);
#pragma unroll
      for (int blk = 0; blk < D / 64; ++blk) {
        tma_load_4d_w(smem + L::kQ + st * L::kTileBytes + blk * kAtomBlock, &tq, blk * 64, qrow0,
                      h, b, &qdo_full[st]);
        tma_load_4d_w(smem + L::kDO + st * L::kTileBytes + blk * kAtomBlock, &tdo, blk * 64,
                      qrow0, h, b, &qdo_full[st]);
      }
      last[st] = (it >> 1) & 1;
    }
    if (!ok) {
      mbar_wait_warp(kv_full, 0, nullptr, 10000000ull);
      for (int s2 = 0; s2 < 2; ++s2)
        if (last[s2] >= 0)
          mbar_wait_warp(&qdo_full[s2], static_cast<uint32_t>(last[s2]), nullptr, 10000000ull);
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------------- MMA
    // Issue order per query tile i: dV_i, S_{i+1}, dK_i, dP_{i+1}, so the
    // elementwise work of one tile overlaps the UMMAs of its neighbours.
    constexpr uint32_t idesc_s = idesc_f16(128, 128, 1, 0, 0);  // S, dP
    constexpr uint32_t idesc_t = idesc_f16(128, D, 1, 1, 1);    // dV, dK (A, B MN-major)
    const uint32_t k_addr = smem_u32(smem + L::kK);
    const uint32_t v_addr = smem_u32(smem + L::kV);
    const uint32_t q_addr = smem_u32(smem + L::kQ);
    const uint32_t do_addr = smem_u32(smem + L::kDO);
    const uint32_t pd_addr = smem_u32(smem + L::kPD);
    auto issue_s = [&](int st) {  // S = Q~_st K~^T -> TMEM [0,128)
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk >> 2) * kAtomBlock + (kk & 3) * 32;
        umma_f16_ss_w(tmem + 0, sdesc_sw128(q_addr + st * L::kTileBytes + off, 16, 1024),
                      sdesc_sw128(k_addr + off, 16, 1024), idesc_s, kk > 0 ? 1u : 0u);
      }
      umma_commit_w(s_full);
    };
    auto issue_dp = [&](int st) {  // dP = dO_st V~^T -> TMEM [128,256)
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk >> 2) * kAtomBlock + (kk & 3) * 32;
        umma_f16_ss_w(tmem + 128, sdesc_sw128(do_addr + st * L::kTileBytes + off, 16, 1024),
                      sdesc_sw128(v_addr + off, 16, 1024), idesc_s, kk > 0 ? 1u : 0u);
      }
      umma_commit_w(dp_full);
    };
    bool ok = mbar_wait_warp(kv_full, 0, abort) && (n_iter > 0) && mbar_wait_warp(&qdo_full[0], 0, abort);
    if (ok) {
      tc_fence_after();
      issue_s(0);
      issue_dp(0);
    }
    for (int it = 0; it < n_iter && ok; ++it) {
      const int st = it & 1;
      const uint32_t ph = static_cast<uint32_t>(it & 1);
      if (!(ok = mbar_wait_warp(pt_full, ph, abort))) break;
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)  // dV += (P~/l)^T dO: contraction over 128 queries
        umma_f16_ss_w(tmem + 256, sdesc_sw128(pd_addr + kk * 2048, kAtomBlock, 1024),
                      sdesc_sw128(do_addr + st * L::kTileBytes + kk * 2048, kAtomBlock, 1024),
                      idesc_t, (it > 0 || kk > 0) ? 1u : 0u);
      umma_commit_w(pt_free);
      if (it + 1 < n_iter) {
        if (!(ok = mbar_wait_warp(&qdo_full[st ^ 1], static_cast<uint32_t>(((it + 1) >> 1) & 1), abort)))
          break;
        tc_fence_after();
        issue_s(st ^ 1);  // S was read before pt_full_i
      }
      if (!(ok = mbar_wait_warp(ds_full, ph, abort))) break;
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)  // dK += dS^T Q~: contraction over 128 queries
        umma_f16_ss_w(tmem + 384, sdesc_sw128(pd_addr + kk * 2048, kAtomBlock, 1024),
                      sdesc_sw128(q_addr + st * L::kTileBytes + kk * 2048, kAtomBlock, 1024),
                      idesc_t, (it > 0 || kk > 0) ? 1u : 0u);
      umma_commit_w(ds_free);
      umma_commit_w(&qdo_empty[st]);
      if (it + 1 < n_iter) issue_dp(st ^ 1);  // dP was read before ds_full_i
    }
    if (ok && n_iter > 0) umma_commit_w(dkdv_done);
    umma_commit_w(mma_drain);
    mbar_wait_warp(mma_drain, 0, nullptr, 10000000ull);
  } else {
    // --------------------------------------------------------- elementwise
    // Warpgroup g (0..3) owns keys [32g, 32g+32) of every tile; thread t of the
    // group owns query row t (TMEM lane t).  dS is stored pre-multiplied by
    // `scale`, so dK comes out scaled.
    const int g = warp >> 2;
    const int t = threadIdx.x & 127;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const float c1 = scale * kLog2e;
    uint8_t* pd_smem = smem + L::kPD;
    const float* lse_g = stats + (static_cast<int64_t>(b) * H + h) * 2 * Nq;
    const float* m_g = lse_g + Nq;
    const float* delta_g = delta + (static_cast<int64_t>(b) * H + h) * Nq;
    const uint32_t key_col = static_cast<uint32_t>(g * 32);
    bool ok = true;
    uint32_t r[32];
    // statistics of this thread's row, prefetched one tile ahead
    auto load_row = [&](int it, float& m, float& lse, float& dl) {
      const int qrow = (it < n_iter ? qtile(it) : 0) * kTile + t;
      const bool in = it < n_iter && qrow < Nq;
      m = in ? m_g[qrow] : 0.f;
      lse = in ? lse_g[qrow] : 0.f;
      dl = in ? delta_g[qrow] : 0.f;
    };
    float nm, nlse, ndl;
    load_row(0, nm, nlse, ndl);
    // The dS stores of tile i are fenced and announced (ds_full) early in tile
    // i+1, after S_{i+1} has been loaded, so the stores drain while the warp
    // works instead of stalling it in the fence.
    bool ds_pending = false;
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
      float pp0[16], pp1[16];  // P (fp32) of this thread's 32 keys, for dS
      {
        tmem_ld32(tmem + lane_base + key_col, r);
        tmem_wait_ld();
        float x[32];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          up2(fma2(pk2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])), c12, nmb2),
              x[2 * i], x[2 * i + 1]);
        if (edge) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int key = k0 + key_col + i;
            if (!(row_ok && key < Nkv && (!causal || key <= qrow))) x[i] = -INFINITY;
          }
        }
        if (ds_pending) {  // dS of the previous tile -> dK
          tc_fence_before();
          fence_proxy_async_smem();
          mbar_arrive_warp(ds_full);
          ds_pending = false;
        }
        uint32_t ptw0[8], ptw1[8];  // P~ / l as bf16x2
        pquant16_scaled_bf16(x, inv_l, pp0, ptw0);
        pquant16_scaled_bf16(x + 16, inv_l, pp1, ptw1);
        tc_fence_before();
        // the P~/dS buffer is free once dK of the previous tile is done
        if (it > 0 && !(ok = mbar_wait_warp(ds_free, ph ^ 1u, abort))) break;
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          const uint32_t* w = ch < 2 ? ptw0 + 4 * ch : ptw1 + 4 * (ch - 2);
          const uint32_t off = sw128_offset(t, key_col + ch * 8, 128);
          *reinterpret_cast<uint4*>(pd_smem + off) = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
      // ---- dS part: dP -> dS = scale * A * (dP - delta), A = P / l
      // The first dP load is issued before the P~ stores are fenced, so its
      // latency overlaps their drain.
      if (!(ok = mbar_wait_warp(dp_full, ph, abort))) break;
      tc_fence_after();
      uint32_t dsw[16];
      uint32_t (&r16)[16] = *reinterpret_cast<uint32_t(*)[16]>(r);
      tmem_ld16(tmem + lane_base + 128 + key_col, r16);
      fence_proxy_async_smem();
      mbar_arrive_warp(pt_full);
      {
        // dP in two halves of 16 keys (P stays in fp32 registers meanwhile);
        // dS = P * (sl * dP - sl * delta) with sl = scale / l
        const float sl = scale * inv_l;
        const uint64_t sl2 = pk2(sl, sl), nsd2 = pk2(-sl * dl, -sl * dl);
#pragma unroll
        for (int hv = 0; hv < 2; ++hv) {
          const float* pp = hv ? pp1 : pp0;
          if (hv) tmem_ld16(tmem + lane_base + 128 + key_col + 16, r16);
          tmem_wait_ld();
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const uint64_t t2 = fma2(pk2(__uint_as_float(r16[2 * u]), __uint_as_float(r16[2 * u + 1])), sl2, nsd2);
            float d0, d1;
            up2(mul2(pk2(pp[2 * u], pp[2 * u + 1]), t2), d0, d1);
            dsw[8 * hv + u] = pack_bf16(d0, d1);
          }
        }
      }
      tc_fence_before();
      if (!(ok = mbar_wait_warp(pt_free, ph, abort))) break;
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        const uint32_t off = sw128_offset(t, key_col + ch * 8, 128);
        *reinterpret_cast<uint4*>(pd_smem + off) =
            make_uint4(dsw[4 * ch], dsw[4 * ch + 1], dsw[4 * ch + 2], dsw[4 * ch + 3]);
      }
      ds_pending = true;
    }
    if (ok && ds_pending) {
      tc_fence_before();
      fence_proxy_async_smem();
      mbar_arrive_warp(ds_full);
    }
    if (ok && n_iter > 0 && (ok = mbar_wait_warp(dkdv_done, 0, abort))) {
      tc_fence_after();
      // groups 0, 1 write dV; groups 2, 3 write dK (already scaled); each group
      // D/2 columns; thread t = key row t
      const int key = k0 + t;
      const int64_t base = ((static_cast<int64_t>(b) * Nkv + key) * H + h) * D;
      __nv_bfloat16* dst = (g < 2 ? dv : dk) + base + (g & 1) * (D / 2);
      const uint32_t col = (g < 2 ? 256u : 384u) + static_cast<uint32_t>((g & 1) * (D / 2));
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        tmem_ld32(tmem + lane_base + col + c * 32, r);
        tmem_wait_ld();
        if (key < Nkv) {
          uint32_t w[16];
#pragma unroll
          for (int u = 0; u < 16; ++u)
            w[u] = pack_bf16(__uint_as_float(r[2 * u]), __uint_as_float(r[2 * u + 1]));
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
        __nv_bfloat16* dst = (g < 2 ? dv : dk) + base + (g & 1) * (D / 2);
        for (int c = 0; c < D / 2; c += 8)
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
// tile twice counts it once.
__global__ void __launch_bounds__(256) tile_transpose_kernel(const int* __restrict__ kv_list,
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

}  // namespace

cudaError_t launch_tile_transpose(const int* kv_list, int B, int H, int n_qt, int n_kt, int topk,
                                  int* q_off, int* q_list, cudaStream_t stream) {
  const size_t smem = static_cast<size_t>(n_kt + 1) * sizeof(int);
  if (smem > 48 * 1024) return cudaErrorInvalidValue;
  tile_transpose_kernel<<<dim3(H, B), 256, smem, stream>>>(kv_list, H, n_qt, n_kt, topk, q_off,
                                                           q_list);
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
cudaError_t launch_bwd_t(const AttnShape& s, const CUtensorMap& tq, const CUtensorMap& tk,
                         const CUtensorMap& tv, const CUtensorMap& tdo, const float* stats,
                         const float* delta, void* dk, void* dv, const int* q_off,
                         const int* q_list, int q_stride, int* err, cudaStream_t stream) {
  using L = BwdLayout<D>;
  const dim3 grid((s.Nkv + kTile - 1) / kTile, s.H, s.B);
  cudaError_t e = cudaFuncSetAttribute(attn_bwd_kernel<D, kSparse>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (e != cudaSuccess) return e;
  attn_bwd_kernel<D, kSparse><<<grid, kThreads, L::kAlloc, stream>>>(
      tq, tk, tv, tdo, stats, delta, static_cast<__nv_bfloat16*>(dk),
      static_cast<__nv_bfloat16*>(dv), s.Nq, s.Nkv, s.H, s.scale, s.causal, q_off, q_list,
      q_stride, err);
  return cudaGetLastError();
}

cudaError_t launch_attn_bwd(const AttnShape& s, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, const CUtensorMap& tdo, const float* stats,
                            const float* delta, void* dk, void* dv, const int* q_off,
                            const int* q_list, int q_stride, int* err, cudaStream_t stream) {
  const bool sp = q_off != nullptr;
  if (s.D == 128)
    return sp ? launch_bwd_t<128, true>(s, tq, tk, tv, tdo, stats, delta, dk, dv, q_off, q_list,
                                        q_stride, err, stream)
              : launch_bwd_t<128, false>(s, tq, tk, tv, tdo, stats, delta, dk, dv, q_off, q_list,
                                         q_stride, err, stream);
  return sp ? launch_bwd_t<64, true>(s, tq, tk, tv, tdo, stats, delta, dk, dv, q_off, q_list,
                                     q_stride, err, stream)
            : launch_bwd_t<64, false>(s, tq, tk, tv, tdo, stats, delta, dk, dv, q_off, q_list,
                                      q_stride, err, stream);
}

}  // namespace nvq
