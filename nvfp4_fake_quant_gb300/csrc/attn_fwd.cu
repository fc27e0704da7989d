// Attn-QAT forward on sm_103a: two passes over the keys per 128-query tile.
//
//   pass 1: S = Q~ K~^T (tcgen05 BF16 UMMA into TMEM), m = rowmax(scale*S)
//   pass 2: S again, P = exp(scale*S - m), l += sum P, P~ = fq16(P) per 16 keys
//           (in registers, one query row per thread), P~ -> shared memory ->
//           O += P~ V~ (tcgen05 F16 UMMA into TMEM)
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
// Roles (192 threads, one CTA per SM):
//   warps 0-3  softmax: thread t owns query row t = TMEM lane t
//   warp 4     TMA producer (lane 0)
//   warp 5     TMEM allocator and UMMA issuer (lane 0)
// Buffers: Q~ tile; K~ and V~ rings of 2 stages; one P~ tile; TMEM columns
// [0,128) and [128,256) hold two S tiles, [256, 256+D) the O accumulator.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "nvq_internal.h"
#include "nvq_ptx.cuh"
#include "nvq_quant.cuh"

namespace nvq {

namespace {

constexpr int kThreads = 192;
constexpr int kStages = 2;
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint32_t kAtomBlock = 128u * 128u;  // bytes of one 64-column block of a 128-row tile

template <int D>
struct FwdLayout {
  static constexpr uint32_t kTileBytes = 128u * D * 2u;
  static constexpr uint32_t kQ = 0;
  static constexpr uint32_t kK = kQ + kTileBytes;
  static constexpr uint32_t kV = kK + kStages * kTileBytes;
  static constexpr uint32_t kP = kV + kStages * kTileBytes;
  static constexpr uint32_t kBars = kP + 128u * 128u * 2u;
  static constexpr uint32_t kNumBars = 17;
  static constexpr uint32_t kTmemSlot = kBars + kNumBars * 8u;
  static constexpr uint32_t kAbort = kTmemSlot + 4u;
  static constexpr uint32_t kUsed = kAbort + 4u;
  // >= 1024 slack for aligning the base; at least ~150 KB so that one CTA
  // (and its 512 TMEM columns) owns an SM.
  static constexpr uint32_t kAlloc =
      (kUsed + 1024u) > 150u * 1024u ? (kUsed + 1024u) : 150u * 1024u;
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tv, __nv_bfloat16* __restrict__ o,
                    float* __restrict__ stats, int Nq, int Nkv, int H, float scale, int causal,
                    int* __restrict__ err) {
  using L = FwdLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023u) &
                                             ~static_cast<uintptr_t>(1023u));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int qt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int q0 = qt * kTile;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBars);
  uint64_t* q_full = bars + 0;
  uint64_t* k_full = bars + 1;    // [2]
  uint64_t* k_empty = bars + 3;   // [2]
  uint64_t* v_full = bars + 5;    // [2]
  uint64_t* v_empty = bars + 7;   // [2]
  uint64_t* s_full = bars + 9;    // [2]
  uint64_t* s_empty = bars + 11;  // [2]
  uint64_t* p_full = bars + 13;
  uint64_t* pv_done = bars + 14;
  uint64_t* o_full = bars + 15;
  uint64_t* mma_drain = bars + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + L::kAbort);

  const int n_kv_all = (Nkv + kTile - 1) / kTile;
  const int n_kv = causal ? min(n_kv_all, qt + 1) : n_kv_all;

  if (threadIdx.x == 0) {
    *abort = 0;
    mbar_init(q_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
      mbar_init(&s_full[s], 1);
      mbar_init(&s_empty[s], 128);
    }
    mbar_init(p_full, 128);
    mbar_init(pv_done, 1);
    mbar_init(o_full, 1);
    mbar_init(mma_drain, 1);
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tv);
      int k_last[2] = {-1, -1}, v_last[2] = {-1, -1};
      bool ok = true;
      mbar_arrive_expect_tx(q_full, L::kTileBytes);
#pragma unroll
      for (int blk = 0; blk < D / 64; ++blk)
        tma_load_4d(smem + L::kQ + blk * kAtomBlock, &tq, blk * 64, q0, h, b, q_full);
      uint32_t kit = 0, vit = 0;
      for (int pass = 0; pass < 2 && ok; ++pass) {
        for (int j = 0; j < n_kv && ok; ++j) {
          const uint32_t st = kit & 1u;
          if (!(ok = mbar_wait(&k_empty[st], ((kit >> 1) & 1u) ^ 1u, abort))) break;
          mbar_arrive_expect_tx(&k_full[st], L::kTileBytes);
#pragma unroll
          for (int blk = 0; blk < D / 64; ++blk)
            tma_load_4d(smem + L::kK + st * L::kTileBytes + blk * kAtomBlock, &tk, blk * 64,
                        j * kTile, h, b, &k_full[st]);
          k_last[st] = static_cast<int>((kit >> 1) & 1u);
          ++kit;
          if (pass == 1) {
            const uint32_t vs = vit & 1u;
            if (!(ok = mbar_wait(&v_empty[vs], ((vit >> 1) & 1u) ^ 1u, abort))) break;
            mbar_arrive_expect_tx(&v_full[vs], L::kTileBytes);
#pragma unroll
            for (int blk = 0; blk < D / 64; ++blk)
              tma_load_4d(smem + L::kV + vs * L::kTileBytes + blk * kAtomBlock, &tv, blk * 64,
                          j * kTile, h, b, &v_full[vs]);
            v_last[vs] = static_cast<int>((vit >> 1) & 1u);
            ++vit;
          }
        }
      }
      if (!ok) {
        // drain copies still in flight before the block leaves
        mbar_wait(q_full, 0, nullptr, 10000000ull);
        for (int s = 0; s < 2; ++s) {
          if (k_last[s] >= 0)
            mbar_wait(&k_full[s], static_cast<uint32_t>(k_last[s]), nullptr, 10000000ull);
          if (v_last[s] >= 0)
            mbar_wait(&v_full[s], static_cast<uint32_t>(v_last[s]), nullptr, 10000000ull);
        }
      }
    }
  } else if (warp == 5) {
    // ---------------------------------------------------------------- MMA
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_f16(128, 128, 1, 0, 0);
      constexpr uint32_t idesc_pv = idesc_f16(128, D, 0, 0, 1);
      const uint32_t q_addr = smem_u32(smem + L::kQ);
      const uint32_t k_addr = smem_u32(smem + L::kK);
      const uint32_t v_addr = smem_u32(smem + L::kV);
      const uint32_t p_addr = smem_u32(smem + L::kP);
      uint32_t kit = 0, sc = 0, vit = 0;
      bool ok = mbar_wait(q_full, 0, abort);
      auto issue_s = [&]() -> bool {
        const uint32_t st = kit & 1u;
        if (!mbar_wait(&k_full[st], (kit >> 1) & 1u, abort)) return false;
        const uint32_t sb = sc & 1u;
        if (!mbar_wait(&s_empty[sb], ((sc >> 1) & 1u) ^ 1u, abort)) return false;
        tc_fence_after();
        const uint32_t kb = k_addr + st * L::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kAtomBlock + (kk & 3) * 32;
          umma_f16_ss(tmem + sb * 128, sdesc_sw128(q_addr + off, 16, 1024),
                      sdesc_sw128(kb + off, 16, 1024), idesc_s, kk > 0 ? 1u : 0u);
        }
        umma_commit(&s_full[sb]);
        umma_commit(&k_empty[st]);
        ++kit;
        ++sc;
        return true;
      };
      if (ok) tc_fence_after();
      for (int j = 0; j < n_kv && ok; ++j) ok = issue_s();  // pass 1
      if (ok) ok = issue_s();                                 // pass 2, tile 0
      for (int j = 0; j < n_kv && ok; ++j) {
        if (j + 1 < n_kv && !(ok = issue_s())) break;
        if (!(ok = mbar_wait(p_full, j & 1, abort))) break;
        const uint32_t vs = vit & 1u;
        if (!(ok = mbar_wait(&v_full[vs], (vit >> 1) & 1u, abort))) break;
        tc_fence_after();
        const uint32_t vb = v_addr + vs * L::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t aoff = (kk >> 2) * kAtomBlock + (kk & 3) * 32;
          umma_f16_ss(tmem + 256, sdesc_sw128(p_addr + aoff, 16, 1024),
                      sdesc_sw128(vb + kk * 2048, kAtomBlock, 1024), idesc_pv,
                      (j > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(pv_done);
        umma_commit(&v_empty[vs]);
        ++vit;
      }
      if (ok) umma_commit(o_full);
      umma_commit(mma_drain);
      mbar_wait(mma_drain, 0, nullptr, 10000000ull);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int t = threadIdx.x;  // 0..127 == query row in tile == TMEM lane
    const int qrow = q0 + t;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const float c1 = scale * kLog2e;
    uint8_t* p_smem = smem + L::kP;
    uint32_t sc = 0;
    bool ok = true;
    float mraw = -INFINITY;
    uint32_t r[32];
    for (int j = 0; j < n_kv && ok; ++j) {
      const uint32_t sb = sc & 1u;
      if (!(ok = mbar_wait_warp(&s_full[sb], (sc >> 1) & 1u, abort))) break;
      tc_fence_after();
      const bool edge = (j * kTile + kTile > Nkv) || (causal && j == qt);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        tmem_ld32(tmem + lane_base + sb * 128 + c * 32, r);
        tmem_wait_ld();
        if (!edge) {
#pragma unroll
          for (int i = 0; i < 32; ++i) mraw = fmaxf(mraw, __uint_as_float(r[i]));
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int key = j * kTile + c * 32 + i;
            if (key < Nkv && (!causal || key <= qrow)) mraw = fmaxf(mraw, __uint_as_float(r[i]));
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&s_empty[sb]);
      ++sc;
    }
    const float m = mraw * scale;
    const float mb = m * kLog2e;
    float l = 0.f;
    for (int j = 0; j < n_kv && ok; ++j) {
      const uint32_t sb = sc & 1u;
      if (!(ok = mbar_wait_warp(&s_full[sb], (sc >> 1) & 1u, abort))) break;
      tc_fence_after();
      const bool edge = (j * kTile + kTile > Nkv) || (causal && j == qt);
      uint32_t pk[64];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        tmem_ld32(tmem + lane_base + sb * 128 + c * 32, r);
        tmem_wait_ld();
        float p[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          float pv = ex2(fmaf(__uint_as_float(r[i]), c1, -mb));
          if (edge) {
            const int key = j * kTile + c * 32 + i;
            if (!(key < Nkv && (!causal || key <= qrow))) pv = 0.f;
          }
          p[i] = pv;
          l += pv;
        }
        uint32_t q8[8];
        quant16_p(p, q8);
#pragma unroll
        for (int u = 0; u < 8; ++u) pk[c * 16 + u] = q8[u];
        quant16_p(p + 16, q8);
#pragma unroll
        for (int u = 0; u < 8; ++u) pk[c * 16 + 8 + u] = q8[u];
      }
      tc_fence_before();
      mbar_arrive(&s_empty[sb]);
      ++sc;
      if (j > 0 && !(ok = mbar_wait_warp(pv_done, (j - 1) & 1, abort))) break;
#pragma unroll
      for (int ch = 0; ch < 16; ++ch) {
        *reinterpret_cast<uint4*>(p_smem + sw128_offset(t, ch * 8, 128)) =
            make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
      }
      fence_proxy_async_smem();
      mbar_arrive(p_full);
    }
    if (ok && (ok = mbar_wait_warp(o_full, 0, abort))) {
      tc_fence_after();
      const float inv_l = 1.0f / l;
      __nv_bfloat16* orow = o + ((static_cast<int64_t>(b) * Nq + qrow) * H + h) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        tmem_ld32(tmem + lane_base + 256 + c * 32, r);
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
      if (qrow < Nq) {
        float* st = stats + (static_cast<int64_t>(b) * H + h) * 2 * Nq;
        st[qrow] = m + logf(l);
        st[Nq + qrow] = m;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  report_abort(abort, err);
  if (warp == 5) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

cudaError_t launch_attn_fwd(const AttnShape& s, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, void* o, float* stats, int* err,
                            cudaStream_t stream) {
  const dim3 grid((s.Nq + kTile - 1) / kTile, s.H, s.B);
  auto* op = static_cast<__nv_bfloat16*>(o);
  if (s.D == 128) {
    using L = FwdLayout<128>;
    cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel<128>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
    if (e != cudaSuccess) return e;
    attn_fwd_kernel<128><<<grid, kThreads, L::kAlloc, stream>>>(tq, tk, tv, op, stats, s.Nq, s.Nkv,
                                                                 s.H, s.scale, s.causal, err);
  } else {
    using L = FwdLayout<64>;
    cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel<64>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
    if (e != cudaSuccess) return e;
    attn_fwd_kernel<64><<<grid, kThreads, L::kAlloc, stream>>>(tq, tk, tv, op, stats, s.Nq, s.Nkv,
                                                                s.H, s.scale, s.causal, err);
  }
  return cudaGetLastError();
}

}  // namespace nvq
