// The GEMMs of the NVFP4 linear ("nvfp4_qad.py": nvfp4_gemm and _NVFP4STE),
// written as persistent tcgen05 kernels for sm_103a.
//
//   forward   out[m, n] = alpha * sum_k x~[m, k] w~[n, k] + bias[n]
//             x~, w~ as packed E2M1 codes with one E4M3 scale per 16 elements
//             (the 128x4 tiled scale layout), on block-scaled FP4 MMAs
//             (tcgen05 kind::mxf4nvf4); alpha = 1 / (gsf_w * gsf_x).
//   backward  grad_x = grad w and grad_w = grad^T x, BF16 MMAs (kind::f16),
//             both in one launch.
//
// Shared structure (192 threads, one CTA per SM, a static round-robin of output
// tiles over the CTAs):
//   warp 0      TMA producer: a ring of shared-memory stages, each filled by
//               tensor-map loads of the operand tiles (and, FP4, bulk copies of
//               the matching scale blocks), completing on the stage's "full"
//               mbarrier
//   warp 1      allocates TMEM and issues the MMAs from one elected lane of the
//               converged warp; each stage is released by a commit to its
//               "empty" mbarrier, each finished tile by a commit to its
//               accumulator's "full" mbarrier
//   warps 2-5   epilogue: thread t of warp w reads TMEM lane 32 (w % 4) + t (one
//               output row), converts to bf16 and stores; then releases the
//               accumulator
// Two TMEM accumulators alternate between tiles, so the epilogue of one tile
// runs under the main loop of the next.  Every wait is bounded; a wait that
// gives up stops every role and records a timeout in the device error word.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "nvq_internal.h"
#include "nvq_ptx.cuh"

namespace nvq {

namespace {

constexpr int kThreads = 192;
constexpr int kTmaWarp = 0, kMmaWarp = 1;
constexpr int kEpiWarps = 4;

__device__ __forceinline__ uint32_t pack2_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Parity of use u (0, 1, ...) of a ring slot: consumers wait for u & 1, the
// producer waits for the slot's release with parity (u & 1) ^ 1.
__device__ __forceinline__ uint32_t par(uint32_t u) { return u & 1u; }

// ===================================================================== BF16
// D[m, n] = sum_k A[m, k] B[n, k] for one problem.  An operand is K-major when
// it is stored [rows, K] (row r contiguous in k: box {64 k, rows}), MN-major
// when stored [K, rows] (box {64 rows, 64 k}, 64-row chunks 8 KB apart).
struct Bf16Problem {
  int a_mn, b_mn;
  int n_tiles;          // output tiles along N (256 columns each)
  int k_steps;          // ceil(K / 64)
  int M, N;             // output size
  int tile0, tile1;     // global tile range [tile0, tile1) of this problem
  __nv_bfloat16* out;   // [M, N] row-major
};

constexpr int kBm = 128, kBn = 256, kBk = 64;
constexpr int kBf16Stages = 4;
constexpr uint32_t kBf16A = kBm * kBk * 2;        // 16 KB
constexpr uint32_t kBf16B = kBn * kBk * 2;        // 32 KB
constexpr uint32_t kBf16Stage = kBf16A + kBf16B;  // 48 KB
constexpr uint32_t kBf16Bars = kBf16Stages * kBf16Stage;
constexpr uint32_t kBf16NumBars = 2 * kBf16Stages + 4 + 1;
constexpr uint32_t kBf16Slot = kBf16Bars + kBf16NumBars * 8;
constexpr uint32_t kBf16Abort = kBf16Slot + 4;
constexpr uint32_t kBf16Smem = kBf16Abort + 4 + 1024;  // + alignment slack

__global__ void __launch_bounds__(kThreads, 1)
    gemm_bf16_kernel(const __grid_constant__ CUtensorMap ta0, const __grid_constant__ CUtensorMap tb0,
                     const __grid_constant__ CUtensorMap ta1, const __grid_constant__ CUtensorMap tb1,
                     const Bf16Problem p0, const Bf16Problem p1, int* __restrict__ err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023u) &
                                             ~static_cast<uintptr_t>(1023u));
  const int warp = threadIdx.x >> 5;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBf16Bars);
  uint64_t* full = bars;                      // [kBf16Stages]
  uint64_t* empty = bars + kBf16Stages;       // [kBf16Stages]
  uint64_t* acc_full = bars + 2 * kBf16Stages;  // [2]
  uint64_t* acc_empty = acc_full + 2;           // [2]
  uint64_t* drain = acc_full + 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kBf16Slot);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + kBf16Abort);
  const int total = p1.tile1;

  if (threadIdx.x == 0) {
    *abort = 0;
    for (int s = 0; s < kBf16Stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], kEpiWarps);
    }
    mbar_init(drain, 1);
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
    tma_prefetch_desc(&ta0);
    tma_prefetch_desc(&tb0);
    tma_prefetch_desc(&ta1);
    tma_prefetch_desc(&tb1);
    uint32_t it = 0;
    int issued[kBf16Stages];
    for (int s = 0; s < kBf16Stages; ++s) issued[s] = -1;
    bool ok = true;
    for (int g = blockIdx.x; g < total && ok; g += gridDim.x) {
      const bool second = g >= p1.tile0;
      const Bf16Problem& p = second ? p1 : p0;
      const CUtensorMap* ta = second ? &ta1 : &ta0;
      const CUtensorMap* tb = second ? &tb1 : &tb0;
      const int local = g - p.tile0;
      const int m0 = (local / p.n_tiles) * kBm, n0 = (local % p.n_tiles) * kBn;
      for (int ks = 0; ks < p.k_steps; ++ks, ++it) {
        const int s = static_cast<int>(it % kBf16Stages);
        const uint32_t u = it / kBf16Stages;
        if (!(ok = mbar_wait_warp(&empty[s], par(u) ^ 1u, abort))) break;
        uint8_t* sa = smem + s * kBf16Stage;
        uint8_t* sb = sa + kBf16A;
        mbar_arrive_expect_tx_w(&full[s], kBf16Stage);
        const int k0 = ks * kBk;
        if (p.a_mn) {
          tma_load_4d_w(sa, ta, m0, k0, 0, 0, &full[s]);
          tma_load_4d_w(sa + 8192, ta, m0 + 64, k0, 0, 0, &full[s]);
        } else {
          tma_load_4d_w(sa, ta, k0, m0, 0, 0, &full[s]);
        }
        if (p.b_mn) {
#pragma unroll
          for (int c = 0; c < 4; ++c) tma_load_4d_w(sb + c * 8192, tb, n0 + 64 * c, k0, 0, 0, &full[s]);
        } else {
          tma_load_4d_w(sb, tb, k0, n0, 0, 0, &full[s]);
        }
        issued[s] = static_cast<int>(par(u));
      }
    }
    if (!ok) {  // let the copies already issued land before the block exits
      for (int s = 0; s < kBf16Stages; ++s)
        if (issued[s] >= 0)
          mbar_wait_warp(&full[s], static_cast<uint32_t>(issued[s]), nullptr, 10000000ull);
    }
  } else if (warp == kMmaWarp) {
    // ----------------------------------------------------------------- MMA
    uint32_t it = 0, tcount = 0;
    bool ok = true;
    for (int g = blockIdx.x; g < total && ok; g += gridDim.x, ++tcount) {
      const Bf16Problem& p = g >= p1.tile0 ? p1 : p0;
      const uint32_t idesc = idesc_f16(kBm, kBn, 1, p.a_mn, p.b_mn);
      const uint32_t acc = tcount & 1u;
      if (!(ok = mbar_wait_warp(&acc_empty[acc], par(tcount >> 1) ^ 1u, abort))) break;
      tc_fence_after();
      const uint32_t d = tmem + acc * kBn;
      for (int ks = 0; ks < p.k_steps; ++ks, ++it) {
        const int s = static_cast<int>(it % kBf16Stages);
        if (!(ok = mbar_wait_warp(&full[s], par(it / kBf16Stages), abort))) break;
        tc_fence_after();
        const uint32_t a = smem_u32(smem + s * kBf16Stage), b = a + kBf16A;
#pragma unroll
        for (int kk = 0; kk < kBk / 16; ++kk) {
          const uint64_t ad = p.a_mn ? sdesc_sw128(a + kk * 2048, 8192, 1024)
                                     : sdesc_sw128(a + kk * 32, 16, 1024);
          const uint64_t bd = p.b_mn ? sdesc_sw128(b + kk * 2048, 8192, 1024)
                                     : sdesc_sw128(b + kk * 32, 16, 1024);
          umma_f16_ss_w(d, ad, bd, idesc, (ks > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit_w(&empty[s]);
      }
      if (ok) umma_commit_w(&acc_full[acc]);
    }
    umma_commit_w(drain);
    mbar_wait_warp(drain, 0, nullptr, 10000000ull);
  } else {
    // ------------------------------------------------------------ epilogue
    const uint32_t wq = static_cast<uint32_t>(warp & 3);
    const int r = static_cast<int>(wq * 32 + (threadIdx.x & 31));  // row in the tile
    const uint32_t lane_base = (wq * 32) << 16;
    uint32_t tcount = 0;
    bool ok = true;
    for (int g = blockIdx.x; g < total && ok; g += gridDim.x, ++tcount) {
      const Bf16Problem& p = g >= p1.tile0 ? p1 : p0;
      const int local = g - p.tile0;
      const int row = (local / p.n_tiles) * kBm + r, n0 = (local % p.n_tiles) * kBn;
      const uint32_t acc = tcount & 1u;
      if (!(ok = mbar_wait_warp(&acc_full[acc], par(tcount >> 1), abort))) break;
      tc_fence_after();
      __nv_bfloat16* dst = p.out + static_cast<int64_t>(row) * p.N + n0;
#pragma unroll 1
      for (int c = 0; c < kBn / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + acc * kBn + c * 32, v);
        tmem_wait_ld();
        if (c == kBn / 32 - 1) {
          tc_fence_before();
          mbar_arrive_warp(&acc_empty[acc]);  // the MMA may reuse this accumulator
        }
        if (row < p.M) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int col = n0 + c * 32 + q * 8;
            if (col < p.N)
              *reinterpret_cast<uint4*>(dst + c * 32 + q * 8) = make_uint4(
                  pack2_bf16(__uint_as_float(v[8 * q + 0]), __uint_as_float(v[8 * q + 1])),
                  pack2_bf16(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3])),
                  pack2_bf16(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5])),
                  pack2_bf16(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7])));
          }
        }
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

// ====================================================================== FP4
// out[m, n] = alpha * sum_k (x codes * x scales)[m, k] (w codes * w scales)[n, k]
// + bias[n].  Codes [rows, K/2] bytes (two a byte, the even element in the low
// nibble), loaded in boxes of 128 bytes (256 elements) x 128 rows with the
// 128-byte swizzle; scales in the 128x4 tiled layout, where the block of row
// tile rt and K-step s (64 elements) is the 512 bytes at (rt * K/64 + s) * 512,
// already in the layout the MMA reads from TMEM: one tcgen05.cp per block.
struct Fp4Problem {
  int M, N;
  int n_tiles, k_steps;        // output tiles along N (128 columns), K / 64
  const uint8_t* sx;           // x scales (tiled)
  const uint8_t* sw;           // w scales (tiled)
  const float* alpha;          // device scalar
  const __nv_bfloat16* bias;   // [N] or nullptr
  __nv_bfloat16* out;          // [M, N] row-major
  int tiles;                   // m_tiles * n_tiles
};

constexpr int kF4Bn = 128;
constexpr int kF4Steps = 4;                        // K-steps of 64 per stage
constexpr int kF4Stages = 5;
constexpr uint32_t kF4Codes = 128u * 128u;         // one operand's codes per stage (16 KB)
constexpr uint32_t kF4Sc = kF4Steps * 512u;        // one operand's scale blocks per stage
constexpr uint32_t kF4Stage = 2 * kF4Codes + 2 * kF4Sc;  // 36 KB
constexpr uint32_t kF4Bars = kF4Stages * kF4Stage;
constexpr uint32_t kF4NumBars = 2 * kF4Stages + 4 + 1;
constexpr uint32_t kF4Slot = kF4Bars + kF4NumBars * 8;
constexpr uint32_t kF4Abort = kF4Slot + 4;
constexpr uint32_t kF4Smem = kF4Abort + 4 + 1024;
// TMEM: accumulators [0, 256); scale operands of stage s, step j at
// kF4ScCol + 8 (s * kF4Steps + j) (x) and + 4 (w).
constexpr uint32_t kF4ScCol = 256;
static_assert(kF4ScCol + 8 * kF4Stages * kF4Steps <= 512, "TMEM columns");

__global__ void __launch_bounds__(kThreads, 1)
    gemm_fp4_kernel(const __grid_constant__ CUtensorMap tx, const __grid_constant__ CUtensorMap tw,
                    const Fp4Problem p, int* __restrict__ err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023u) &
                                             ~static_cast<uintptr_t>(1023u));
  const int warp = threadIdx.x >> 5;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kF4Bars);
  uint64_t* full = bars;
  uint64_t* empty = bars + kF4Stages;
  uint64_t* acc_full = bars + 2 * kF4Stages;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_full + 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kF4Slot);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + kF4Abort);
  const int k_stages = (p.k_steps + kF4Steps - 1) / kF4Steps;

  if (threadIdx.x == 0) {
    *abort = 0;
    for (int s = 0; s < kF4Stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], kEpiWarps);
    }
    mbar_init(drain, 1);
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
    tma_prefetch_desc(&tx);
    tma_prefetch_desc(&tw);
    uint32_t it = 0;
    int issued[kF4Stages];
    for (int s = 0; s < kF4Stages; ++s) issued[s] = -1;
    bool ok = true;
    for (int g = blockIdx.x; g < p.tiles && ok; g += gridDim.x) {
      const int mt = g / p.n_tiles, nt = g % p.n_tiles;
      for (int st = 0; st < k_stages; ++st, ++it) {
        const int s = static_cast<int>(it % kF4Stages);
        const uint32_t u = it / kF4Stages;
        if (!(ok = mbar_wait_warp(&empty[s], par(u) ^ 1u, abort))) break;
        const int s0 = st * kF4Steps;
        const int ns = min(kF4Steps, p.k_steps - s0);
        uint8_t* base = smem + s * kF4Stage;
        mbar_arrive_expect_tx_w(&full[s], 2 * kF4Codes + 2 * static_cast<uint32_t>(ns) * 512u);
        tma_load_4d_w(base, &tx, st * 128, mt * 128, 0, 0, &full[s]);
        tma_load_4d_w(base + kF4Codes, &tw, st * 128, nt * kF4Bn, 0, 0, &full[s]);
        bulk_load_w(base + 2 * kF4Codes,
                    p.sx + (static_cast<int64_t>(mt) * p.k_steps + s0) * 512, ns * 512, &full[s]);
        bulk_load_w(base + 2 * kF4Codes + kF4Sc,
                    p.sw + (static_cast<int64_t>(nt) * p.k_steps + s0) * 512, ns * 512, &full[s]);
        issued[s] = static_cast<int>(par(u));
      }
    }
    if (!ok) {
      for (int s = 0; s < kF4Stages; ++s)
        if (issued[s] >= 0)
          mbar_wait_warp(&full[s], static_cast<uint32_t>(issued[s]), nullptr, 10000000ull);
    }
  } else if (warp == kMmaWarp) {
    // ----------------------------------------------------------------- MMA
    constexpr uint32_t idesc = idesc_mxf4nvf4(128, kF4Bn);
    uint32_t it = 0, tcount = 0;
    bool ok = true;
    for (int g = blockIdx.x; g < p.tiles && ok; g += gridDim.x, ++tcount) {
      const uint32_t acc = tcount & 1u;
      if (!(ok = mbar_wait_warp(&acc_empty[acc], par(tcount >> 1) ^ 1u, abort))) break;
      tc_fence_after();
      const uint32_t d = tmem + acc * kF4Bn;
      for (int st = 0; st < k_stages; ++st, ++it) {
        const int s = static_cast<int>(it % kF4Stages);
        if (!(ok = mbar_wait_warp(&full[s], par(it / kF4Stages), abort))) break;
        tc_fence_after();
        const int ns = min(kF4Steps, p.k_steps - st * kF4Steps);
        const uint32_t a = smem_u32(smem + s * kF4Stage), b = a + kF4Codes;
        const uint32_t sa = a + 2 * kF4Codes, sb = sa + kF4Sc;
        for (int j = 0; j < ns; ++j) {
          const uint32_t col = tmem + kF4ScCol + 8u * static_cast<uint32_t>(s * kF4Steps + j);
          // the previous use of these columns (stage s one ring turn ago) is
          // complete: the producer saw stage s released before refilling it
          tmem_cp_32x128_x4_w(col, sa + j * 512);
          tmem_cp_32x128_x4_w(col + 4, sb + j * 512);
          umma_fp4_ss_w(d, sdesc_sw128(a + 32 * j, 16, 1024), sdesc_sw128(b + 32 * j, 16, 1024),
                        idesc, col, col + 4, (st > 0 || j > 0) ? 1u : 0u);
        }
        umma_commit_w(&empty[s]);
      }
      if (ok) umma_commit_w(&acc_full[acc]);
    }
    umma_commit_w(drain);
    mbar_wait_warp(drain, 0, nullptr, 10000000ull);
  } else {
    // ------------------------------------------------------------ epilogue
    const uint32_t wq = static_cast<uint32_t>(warp & 3);
    const int r = static_cast<int>(wq * 32 + (threadIdx.x & 31));
    const uint32_t lane_base = (wq * 32) << 16;
    const float alpha = *p.alpha;
    uint32_t tcount = 0;
    bool ok = true;
    for (int g = blockIdx.x; g < p.tiles && ok; g += gridDim.x, ++tcount) {
      const int row = (g / p.n_tiles) * 128 + r, n0 = (g % p.n_tiles) * kF4Bn;
      const uint32_t acc = tcount & 1u;
      if (!(ok = mbar_wait_warp(&acc_full[acc], par(tcount >> 1), abort))) break;
      tc_fence_after();
      __nv_bfloat16* dst = p.out + static_cast<int64_t>(row) * p.N + n0;
#pragma unroll 1
      for (int c = 0; c < kF4Bn / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + acc * kF4Bn + c * 32, v);
        tmem_wait_ld();
        if (c == kF4Bn / 32 - 1) {
          tc_fence_before();
          mbar_arrive_warp(&acc_empty[acc]);
        }
        if (row < p.M) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int col = n0 + c * 32 + q * 8;
            if (col >= p.N) continue;
            float bv[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            if (p.bias != nullptr) {
              const uint4 braw = __ldg(reinterpret_cast<const uint4*>(p.bias + col));
              const uint32_t bw[4] = {braw.x, braw.y, braw.z, braw.w};
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                bv[2 * i] = __uint_as_float(bw[i] << 16);
                bv[2 * i + 1] = __uint_as_float(bw[i] & 0xFFFF0000u);
              }
            }
            uint32_t o[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
              o[i] = pack2_bf16(fmaf(alpha, __uint_as_float(v[8 * q + 2 * i]), bv[2 * i]),
                                fmaf(alpha, __uint_as_float(v[8 * q + 2 * i + 1]), bv[2 * i + 1]));
            *reinterpret_cast<uint4*>(dst + c * 32 + q * 8) = make_uint4(o[0], o[1], o[2], o[3]);
          }
        }
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

// ---------------------------------------------------- FP4, x resident, W multicast
// The same product for K <= kXresMaxK, with far less operand traffic: a cluster
// of kRc CTAs takes kRc consecutive 128-row tiles of x (one each) and sweeps a
// chunk of W's 128-row tiles together.  Each CTA keeps its x codes in shared
// memory and its x scales in TMEM for the whole chunk; each W stage (256
// K-elements of 128 rows) is loaded once for the cluster, the CTAs fetching its
// four 32-row slices and four 512-byte scale blocks in turn and multicasting
// them to every CTA of the cluster.  A stage is refilled only when all kRc CTAs
// have released it (their MMA commits arrive on every CTA's "empty" barrier).
// Clusters of 2, 1 and 4 measured 0.278, 0.294 and 0.294 ms at the Wan FFN
// up-projection (more pairs fit on the GPU than quads).  x is reloaded box by box
// (256 K-elements): the chunk's last tile releases box b when its stage b is
// done, so the next chunk's x arrives under the current tile's MMAs.  Output
// tiles leave through shared memory by TMA stores (full 128-byte lines).
constexpr int kRc = 2;  // CTAs per cluster (the slice loops also work for 1 and 4)
constexpr int kXresMaxK = 1536;             // x codes (6 boxes of 16 KB) resident
constexpr int kXresBoxes = kXresMaxK / 256;
constexpr int kXresStages = 4;
constexpr uint32_t kXresStage = 16384 + 2048;              // W codes + 4 scale blocks
constexpr uint32_t kXresA = 0;                             // x codes, box b at b * 16 KB
constexpr uint32_t kXresAS = kXresBoxes * 16384;           // x scales, step j at j * 512
constexpr uint32_t kXresB = kXresAS + kXresBoxes * 2048;   // W stages
constexpr uint32_t kXresO = kXresB + kXresStages * kXresStage;  // output staging
constexpr uint32_t kXresBars = kXresO + kEpiWarps * 2 * 4096;
constexpr uint32_t kXresNumBars = 2 * kXresStages + 2 * kXresBoxes + 4 + 1;
constexpr uint32_t kXresSlot = kXresBars + kXresNumBars * 8;
constexpr uint32_t kXresAbort = kXresSlot + 4;
constexpr uint32_t kXresSmem = kXresAbort + 4 + 1024;
// TMEM: accumulators [0, 256), x scales of step j at 256 + 4 j, W scales of
// stage s, step j at kXresBCol + 4 (4 s + j).
constexpr uint32_t kXresBCol = 256 + 4 * 4 * kXresBoxes;
static_assert(kXresBCol + 4 * 4 * kXresStages <= 512, "TMEM columns");

struct XresProblem {
  int M, N, m_tiles, n_tiles, k_steps;
  int n_chunks, chunk_tiles, units;   // unit = (group of kRc x tiles, chunk of W tiles)
  const uint8_t* sx;
  const uint8_t* sw;
  const float* alpha;
  const __nv_bfloat16* bias;
  __nv_bfloat16* out;   // [M, N]: written through tout
};

__global__ void __launch_bounds__(kThreads, 1)
    gemm_fp4_xres_kernel(const __grid_constant__ CUtensorMap tx,
                         const __grid_constant__ CUtensorMap tw32,
                         const __grid_constant__ CUtensorMap tout, const XresProblem p,
                         int* __restrict__ err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023u) &
                                             ~static_cast<uintptr_t>(1023u));
  const int warp = threadIdx.x >> 5;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kXresBars);
  uint64_t* full = bars;                          // [kXresStages] W stage landed (all slices)
  uint64_t* empty = full + kXresStages;           // [kXresStages] released by all kRc CTAs
  uint64_t* a_full = empty + kXresStages;         // [kXresBoxes] x box landed
  uint64_t* a_empty = a_full + kXresBoxes;        // [kXresBoxes] x box no longer read
  uint64_t* acc_full = a_empty + kXresBoxes;      // [2]
  uint64_t* acc_empty = acc_full + 2;             // [2]
  uint64_t* drain = acc_full + 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kXresSlot);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + kXresAbort);
  const int rank = static_cast<int>(cluster_ctarank());
  const int cid = static_cast<int>(cluster_id_x()), ncl = static_cast<int>(cluster_count_x());
  const int k_stages = (p.k_steps + 3) / 4;
  constexpr uint16_t kAll = (1u << kRc) - 1u;

  if (threadIdx.x == 0) {
    *abort = 0;
    for (int s = 0; s < kXresStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kRc);
    }
    for (int b = 0; b < kXresBoxes; ++b) {
      mbar_init(&a_full[b], 1);
      mbar_init(&a_empty[b], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], kEpiWarps);
    }
    mbar_init(drain, 1);
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  cluster_sync_all();  // every CTA's barriers exist before any multicast arrives
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kTmaWarp) {
    // ------------------------------------------------------------ producer
    tma_prefetch_desc(&tx);
    tma_prefetch_desc(&tw32);
    uint32_t it = 0, ucount = 0;
    int issued[kXresStages];
    for (int s = 0; s < kXresStages; ++s) issued[s] = -1;
    bool ok = true;
    for (int u = cid; u < p.units && ok; u += ncl, ++ucount) {
      const int mt = (u / p.n_chunks) * kRc + rank;
      const int nt0 = (u % p.n_chunks) * p.chunk_tiles;
      const int nt1 = min(nt0 + p.chunk_tiles, p.n_tiles);
      const bool x_ok = mt < p.m_tiles;  // past the last x tile: zero codes, no scales
      for (int nt = nt0; nt < nt1 && ok; ++nt) {
        for (int st = 0; st < k_stages; ++st, ++it) {
          const int ns = min(4, p.k_steps - 4 * st);
          if (nt == nt0) {  // this chunk's x box st, once the previous chunk is done with it
            if (!(ok = mbar_wait_warp(&a_empty[st], par(ucount) ^ 1u, abort))) break;
            mbar_arrive_expect_tx_w(&a_full[st], 16384u + (x_ok ? ns * 512u : 0u));
            tma_load_4d_w(smem + kXresA + st * 16384, &tx, st * 128, mt * 128, 0, 0, &a_full[st]);
            if (x_ok)
              bulk_load_w(smem + kXresAS + st * 2048,
                          p.sx + (static_cast<int64_t>(mt) * p.k_steps + 4 * st) * 512, ns * 512,
                          &a_full[st]);
          }
          const int s = static_cast<int>(it % kXresStages);
          if (!(ok = mbar_wait_warp(&empty[s], par(it / kXresStages) ^ 1u, abort))) break;
          uint8_t* stage = smem + kXresB + s * kXresStage;
          mbar_arrive_expect_tx_w(&full[s], 16384u + ns * 512u);
          for (int q = rank; q < 4; q += kRc)  // 32-row slices q of the W tile
            tma_load_4d_mc_w(stage + q * 4096, &tw32, st * 128, nt * 128 + q * 32, 0, 0, &full[s],
                             kAll);
          for (int j = rank; j < ns; j += kRc)  // scale blocks of K-steps j
            bulk_load_mc_w(stage + 16384 + j * 512,
                           p.sw + (static_cast<int64_t>(nt) * p.k_steps + 4 * st + j) * 512, 512,
                           &full[s], kAll);
          issued[s] = static_cast<int>(par(it / kXresStages));
        }
      }
    }
    if (!ok) {  // let the copies already issued land before the block leaves
      for (int s = 0; s < kXresStages; ++s)
        if (issued[s] >= 0)
          mbar_wait_warp(&full[s], static_cast<uint32_t>(issued[s]), nullptr, 10000000ull);
    }
  } else if (warp == kMmaWarp) {
    // ----------------------------------------------------------------- MMA
    constexpr uint32_t idesc = idesc_mxf4nvf4(128, 128);
    uint32_t it = 0, tcount = 0, ucount = 0;
    bool ok = true;
    const uint32_t a_addr = smem_u32(smem + kXresA), as_addr = smem_u32(smem + kXresAS);
    for (int u = cid; u < p.units && ok; u += ncl, ++ucount) {
      const int nt0 = (u % p.n_chunks) * p.chunk_tiles;
      const int nt1 = min(nt0 + p.chunk_tiles, p.n_tiles);
      for (int nt = nt0; nt < nt1 && ok; ++nt, ++tcount) {
        const uint32_t acc = tcount & 1u;
        if (!(ok = mbar_wait_warp(&acc_empty[acc], par(tcount >> 1) ^ 1u, abort))) break;
        tc_fence_after();
        const uint32_t d = tmem + acc * 128;
        for (int st = 0; st < k_stages; ++st, ++it) {
          const int ns = min(4, p.k_steps - 4 * st);
          if (nt == nt0) {  // x box st of this chunk: its scales go to TMEM
            if (!(ok = mbar_wait_warp(&a_full[st], par(ucount), abort))) break;
            tc_fence_after();
            for (int j = 0; j < ns; ++j)
              tmem_cp_32x128_x4_w(tmem + 256 + 4 * (4 * st + j), as_addr + st * 2048 + j * 512);
          }
          const int s = static_cast<int>(it % kXresStages);
          if (!(ok = mbar_wait_warp(&full[s], par(it / kXresStages), abort))) break;
          tc_fence_after();
          const uint32_t b = smem_u32(smem + kXresB + s * kXresStage);
          for (int j = 0; j < ns; ++j) {
            const uint32_t bcol = tmem + kXresBCol + 4 * (4 * s + j);
            tmem_cp_32x128_x4_w(bcol, b + 16384 + j * 512);
            umma_fp4_ss_w(d, sdesc_sw128(a_addr + st * 16384 + 32 * j, 16, 1024),
                          sdesc_sw128(b + 32 * j, 16, 1024), idesc, tmem + 256 + 4 * (4 * st + j),
                          bcol, (st > 0 || j > 0) ? 1u : 0u);
          }
          umma_commit_mc_w(&empty[s], kAll);  // this CTA is done with stage s
          if (nt == nt1 - 1) umma_commit_w(&a_empty[st]);  // and, last tile, with x box st
        }
        if (ok) umma_commit_w(&acc_full[acc]);
      }
    }
    umma_commit_w(drain);
    mbar_wait_warp(drain, 0, nullptr, 10000000ull);
  } else {
    // ------------------------------------------------------------ epilogue
    const uint32_t wq = static_cast<uint32_t>(warp & 3);
    const uint32_t lane = threadIdx.x & 31;
    const uint32_t lane_base = (wq * 32) << 16;
    uint8_t* stage_out = smem + kXresO + (warp - 2) * 8192;
    const float alpha = *p.alpha;
    uint32_t tcount = 0, sc = 0;
    bool ok = true;
    for (int u = cid; u < p.units && ok; u += ncl) {
      const int mt = (u / p.n_chunks) * kRc + rank;
      const int nt0 = (u % p.n_chunks) * p.chunk_tiles;
      const int nt1 = min(nt0 + p.chunk_tiles, p.n_tiles);
      for (int nt = nt0; nt < nt1 && ok; ++nt, ++tcount) {
        const uint32_t acc = tcount & 1u;
        if (!(ok = mbar_wait_warp(&acc_full[acc], par(tcount >> 1), abort))) break;
        tc_fence_after();
#pragma unroll 1
        for (int h = 0; h < 2; ++h, ++sc) {
          uint32_t v[64];
          tmem_ld32(tmem + lane_base + acc * 128 + h * 64, *reinterpret_cast<uint32_t(*)[32]>(v));
          tmem_ld32(tmem + lane_base + acc * 128 + h * 64 + 32,
                    *reinterpret_cast<uint32_t(*)[32]>(v + 32));
          tmem_wait_ld();
          if (h == 1) {
            tc_fence_before();
            mbar_arrive_warp(&acc_empty[acc]);  // the MMA may reuse the accumulator
          }
          const int c0 = nt * 128 + h * 64;
          uint32_t w[32];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            float bv[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            if (p.bias != nullptr && c0 + 8 * q < p.N) {
              const uint4 braw = __ldg(reinterpret_cast<const uint4*>(p.bias + c0 + 8 * q));
              const uint32_t bw[4] = {braw.x, braw.y, braw.z, braw.w};
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                bv[2 * i] = __uint_as_float(bw[i] << 16);
                bv[2 * i + 1] = __uint_as_float(bw[i] & 0xFFFF0000u);
              }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
              w[4 * q + i] = pack2_bf16(fmaf(alpha, __uint_as_float(v[8 * q + 2 * i]), bv[2 * i]),
                                        fmaf(alpha, __uint_as_float(v[8 * q + 2 * i + 1]), bv[2 * i + 1]));
          }
          uint8_t* buf = stage_out + (sc & 1u) * 4096;
          if (lane == 0) bulk_wait_group_read<1>();  // the store from this buffer has read it
          __syncwarp();
          // row `lane`, 16-byte chunk q at chunk position q ^ (lane % 8): the
          // 128-byte swizzle the output tensor map uses (conflict-free writes)
#pragma unroll
          for (int q = 0; q < 8; ++q)
            *reinterpret_cast<uint4*>(buf + lane * 128 + ((q ^ (lane & 7)) << 4)) =
                make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_4d(&tout, buf, c0, mt * 128 + static_cast<int>(wq) * 32, 0, 0);
            bulk_commit_group();
          }
        }
      }
    }
    if (lane == 0) bulk_wait_group<0>();  // every store has completed
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // no CTA leaves while a peer may still write into it
  report_abort(abort, err);
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

int sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
    return 148;
  return sms;
}

}  // namespace

cudaError_t launch_gemm_bf16_pair(const CUtensorMap& ta0, const CUtensorMap& tb0, int a_mn0,
                                  int b_mn0, int64_t M0, int64_t N0, int64_t K0, void* out0,
                                  const CUtensorMap& ta1, const CUtensorMap& tb1, int a_mn1,
                                  int b_mn1, int64_t M1, int64_t N1, int64_t K1, void* out1,
                                  int* err, cudaStream_t stream) {
  auto make = [](int a_mn, int b_mn, int64_t M, int64_t N, int64_t K, void* out, int tile0) {
    Bf16Problem p{};
    p.a_mn = a_mn;
    p.b_mn = b_mn;
    p.M = static_cast<int>(M);
    p.N = static_cast<int>(N);
    p.n_tiles = static_cast<int>((N + kBn - 1) / kBn);
    p.k_steps = static_cast<int>((K + kBk - 1) / kBk);
    const int tiles = out != nullptr ? static_cast<int>((M + kBm - 1) / kBm) * p.n_tiles : 0;
    p.tile0 = tile0;
    p.tile1 = tile0 + tiles;
    p.out = static_cast<__nv_bfloat16*>(out);
    return p;
  };
  const Bf16Problem p0 = make(a_mn0, b_mn0, M0, N0, K0, out0, 0);
  const Bf16Problem p1 = make(a_mn1, b_mn1, M1, N1, K1, out1, p0.tile1);
  const int total = p1.tile1;
  if (total == 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(gemm_bf16_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kBf16Smem);
  if (e != cudaSuccess) return e;
  const int grid = total < sm_count() ? total : sm_count();
  gemm_bf16_kernel<<<grid, kThreads, kBf16Smem, stream>>>(ta0, tb0, ta1, tb1, p0, p1, err);
  return cudaGetLastError();
}

cudaError_t launch_gemm_fp4_xres(const CUtensorMap& tx, const CUtensorMap& tw32,
                                 const CUtensorMap& tout, const uint8_t* sx, const uint8_t* sw,
                                 const float* alpha, const void* bias, int64_t M, int64_t N,
                                 int64_t K, void* out, int* err, cudaStream_t stream) {
  XresProblem p{};
  p.out = static_cast<__nv_bfloat16*>(out);
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.m_tiles = static_cast<int>((M + 127) / 128);
  p.n_tiles = static_cast<int>((N + 127) / 128);
  p.k_steps = static_cast<int>(K / 64);
  p.sx = sx;
  p.sw = sw;
  p.alpha = alpha;
  p.bias = static_cast<const __nv_bfloat16*>(bias);
  cudaError_t e = cudaFuncSetAttribute(gemm_fp4_xres_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kXresSmem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kRc;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kXresSmem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(sm_count() / kRc * kRc));
  int clusters = 0;
  e = cudaOccupancyMaxActiveClusters(&clusters, gemm_fp4_xres_kernel, &cfg);
  if (e != cudaSuccess) return e;
  if (clusters < 1) return cudaErrorInvalidConfiguration;
  // chunks of W tiles per x group: the fewest rounds of (tiles + one x load)
  const int groups = (p.m_tiles + kRc - 1) / kRc;
  int best_nc = 1;
  int64_t best = -1;
  for (int nc = 1; nc <= p.n_tiles; ++nc) {
    const int chunk = (p.n_tiles + nc - 1) / nc;
    const int64_t rounds = (static_cast<int64_t>(groups) * nc + clusters - 1) / clusters;
    const int64_t cost = rounds * (chunk + 1);
    if (best < 0 || cost < best) {
      best = cost;
      best_nc = nc;
    }
  }
  p.chunk_tiles = (p.n_tiles + best_nc - 1) / best_nc;
  p.n_chunks = (p.n_tiles + p.chunk_tiles - 1) / p.chunk_tiles;
  p.units = groups * p.n_chunks;
  const int used = p.units < clusters ? p.units : clusters;
  cfg.gridDim = dim3(static_cast<unsigned>(used * kRc));
  e = cudaLaunchKernelEx(&cfg, gemm_fp4_xres_kernel, tx, tw32, tout, p, err);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_gemm_fp4(const CUtensorMap& tx, const CUtensorMap& tw, const uint8_t* sx,
                            const uint8_t* sw, const float* alpha, const void* bias, int64_t M,
                            int64_t N, int64_t K, void* out, int* err, cudaStream_t stream) {
  Fp4Problem p{};
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.n_tiles = static_cast<int>((N + kF4Bn - 1) / kF4Bn);
  p.k_steps = static_cast<int>(K / 64);
  p.sx = sx;
  p.sw = sw;
  p.alpha = alpha;
  p.bias = static_cast<const __nv_bfloat16*>(bias);
  p.out = static_cast<__nv_bfloat16*>(out);
  p.tiles = static_cast<int>((M + 127) / 128) * p.n_tiles;
  cudaError_t e = cudaFuncSetAttribute(gemm_fp4_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kF4Smem);
  if (e != cudaSuccess) return e;
  const int grid = p.tiles < sm_count() ? p.tiles : sm_count();
  gemm_fp4_kernel<<<grid, kThreads, kF4Smem, stream>>>(tx, tw, p, err);
  return cudaGetLastError();
}

}  // namespace nvq
