// Self-tests of the hardware encodings the attention kernels rely on:
//  * one 128 x N x K tcgen05 kind::f16 BF16 UMMA fed by 128-byte-swizzled TMA
//    tiles through the same shared-memory and instruction descriptors, for
//    K-major and MN-major A and B, and for A stored in TMEM by tcgen05.st;
//  * one 128 x N x (64 or 128) block-scaled kind::mxf4nvf4 UMMA (E2M1 operands
//    from 32- or 64-byte-swizzled TMA tiles, E4M3 scales in TMEM written either
//    by tcgen05.st from a given TMEM image or by tcgen05.cp from shared memory);
//  * a bounded mbarrier wait that is meant to run out.
#include <cuda_runtime.h>

#include "nvq_internal.h"
#include "nvq_ptx.cuh"
#include "nvq_quant.cuh"

namespace nvq {

namespace {

constexpr uint32_t kSmem = 2 * 32768 + 1024 + 64;

// Tile of a row-major [rows, cols] 16-bit matrix as loaded by TMA with a box
// of {64, rows}: column block j (64 columns) at j * rows * 128 bytes.
// a_mn == 2: A is also read straight from global memory (a_glob, row-major
// [128, K]) and stored into TMEM columns [128, 128 + K/2) by tcgen05.st, two
// elements per column, and the UMMA takes A from there.
__global__ void __launch_bounds__(128, 1)
    selftest_umma_kernel(const __grid_constant__ CUtensorMap ta,
                         const __grid_constant__ CUtensorMap tb, const uint32_t* __restrict__ a_glob,
                         float* __restrict__ c, int N, int K, int a_mn, int b_mn,
                         int* __restrict__ err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023u) &
                                             ~static_cast<uintptr_t>(1023u));
  uint8_t* sa = smem;
  uint8_t* sb = smem + 32768;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 65536);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + 65536 + 16);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + 65536 + 20);
  const int warp = threadIdx.x >> 5;
  const bool a_tmem = a_mn == 2;
  const int a_smem_mn = a_tmem ? 0 : a_mn;
  // A is [128, K] (K-major) or [K, 128] (MN-major); B is [N, K] or [K, N].
  const int a_rows = a_smem_mn ? K : 128, a_cols = a_smem_mn ? 128 : K;
  const int b_rows = b_mn ? K : N, b_cols = b_mn ? N : K;
  if (threadIdx.x == 0) {
    *abort = 0;
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
  if (a_tmem) {  // thread t stores row t of A: K/2 columns of packed pairs
    const uint32_t* row = a_glob + static_cast<size_t>(threadIdx.x) * (K / 2);
    for (int cc = 0; cc < K / 32; ++cc) {
      uint32_t r[16];
      for (int i = 0; i < 16; ++i) r[i] = row[cc * 16 + i];
      tmem_st16(tmem + lane_base + 128 + cc * 16, r);
    }
    tmem_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  bool ok = true;
  if (warp == 0) {  // converged warp: the issue path the attention kernels use
    const uint32_t bytes = static_cast<uint32_t>(a_rows * a_cols * 2 + b_rows * b_cols * 2);
    mbar_arrive_expect_tx_w(&bars[0], bytes);
    for (int j = 0; j < a_cols / 64; ++j)
      tma_load_4d_w(sa + j * a_rows * 128, &ta, j * 64, 0, 0, 0, &bars[0]);
    for (int j = 0; j < b_cols / 64; ++j)
      tma_load_4d_w(sb + j * b_rows * 128, &tb, j * 64, 0, 0, 0, &bars[0]);
    ok = mbar_wait_warp(&bars[0], 0, abort);
    if (ok) {
      tc_fence_after();
      const uint32_t idesc = idesc_f16(128, N, 1, a_smem_mn, b_mn);
      const uint32_t a0 = smem_u32(sa), b0 = smem_u32(sb);
      for (int kk = 0; kk < K / 16; ++kk) {
        uint64_t ad, bd;
        if (a_smem_mn)  // rows = K: 16 rows per step; 64-column M chunks a_rows*128 apart
          ad = sdesc_sw128(a0 + kk * 2048, static_cast<uint32_t>(a_rows * 128), 1024);
        else  // rows = M: 32 bytes per K step inside an atom, next atom block a_rows*128 on
          ad = sdesc_sw128(a0 + (kk >> 2) * (a_rows * 128) + (kk & 3) * 32, 16, 1024);
        if (b_mn)
          bd = sdesc_sw128(b0 + kk * 2048, static_cast<uint32_t>(b_rows * 128), 1024);
        else
          bd = sdesc_sw128(b0 + (kk >> 2) * (b_rows * 128) + (kk & 3) * 32, 16, 1024);
        if (a_tmem)
          umma_f16_ts_w(tmem, tmem + 128 + kk * 8, bd, idesc, kk > 0 ? 1u : 0u);
        else
          umma_f16_ss_w(tmem, ad, bd, idesc, kk > 0 ? 1u : 0u);
      }
      umma_commit_w(&bars[1]);
    }
  }
  __syncthreads();
  // every warp waits (warp-uniformly) even when the issue failed: *abort ends it
  const bool done = mbar_wait_warp(&bars[1], 0, abort);
  if (done && !*abort) {
    tc_fence_after();
    const int row = threadIdx.x;
    uint32_t r[32];
    for (int cc = 0; cc < N / 32; ++cc) {
      tmem_ld32(tmem + lane_base + cc * 32, r);
      tmem_wait_ld();
      for (int i = 0; i < 32; ++i) c[row * N + cc * 32 + i] = __uint_as_float(r[i]);
    }
  }
  tc_fence_before();
  __syncthreads();
  report_abort(abort, err);
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

// FP4 probe.  A: E2M1 codes [128, kb] bytes (kb = 32 * nmma, K = 64 * nmma,
// nmma in {1, 2, 4}), B: [N, kb]; both K-major, loaded by TMA with the kb-byte
// swizzle.  TMEM:
// D at columns [0, N), A scales at [256, 288), B scales at [288, 320).
//   mode 0: sf_img (u32 [2][128][32]: A then B, lane-major) is stored into those
//           columns by tcgen05.st;
//   mode 1: sf_src (bytes [2][nmma][512]) is copied into shared memory and from
//           there by tcgen05.cp (32x128b, warpx4): A block kk to column
//           256 + 4 kk, B block kk to 288 + 4 kk.
// UMMA kk reads its scales at column 256 + kk * sf_stride (A), 288 + kk *
// sf_stride (B).  Outputs: c [128, N] f32 and dump (u32 [128][64]): TMEM columns
// [256, 320) after the UMMAs.
constexpr uint32_t kFp4Smem = 1024 + 16384 + 16384 + 4096 + 4096 + 256;

__global__ void __launch_bounds__(128, 1)
    selftest_fp4_kernel(const __grid_constant__ CUtensorMap ta,
                        const __grid_constant__ CUtensorMap tb, const uint32_t* __restrict__ sf_img,
                        const uint8_t* __restrict__ sf_src, float* __restrict__ c,
                        uint32_t* __restrict__ dump, int N, int nmma, int sf_stride, int mode,
                        int* __restrict__ err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023u) &
                                             ~static_cast<uintptr_t>(1023u));
  uint8_t* sa = smem;
  uint8_t* sb = smem + 16384;
  uint8_t* sfs = smem + 32768;  // cp source (4 KB), followed by 4 KB of slack
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 32768 + 4096 + 4096);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 3);
  volatile int* abort = reinterpret_cast<volatile int*>(bars + 4);
  const int warp = threadIdx.x >> 5;
  const int kb = 32 * nmma;
  if (threadIdx.x == 0) {
    *abort = 0;
    for (int i = 0; i < 3; ++i) mbar_init(&bars[i], 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
  if (mode == 0) {
    const int lane_row = threadIdx.x;  // TMEM lane of this thread
#pragma unroll
    for (int m = 0; m < 2; ++m) {
      const uint32_t* img = sf_img + (static_cast<size_t>(m) * 128 + lane_row) * 32;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t r[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) r[i] = img[h * 16 + i];
        tmem_st16(tmem + lane_base + 256 + 32 * m + 16 * h, r);
      }
    }
    tmem_wait_st();
  } else {
    for (int i = threadIdx.x; i < 2 * nmma * 512; i += 128) sfs[i] = sf_src[i];
    for (int i = threadIdx.x; i < 4096; i += 128) sfs[4096 + i] = 0;
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) {
    mbar_arrive_expect_tx_w(&bars[0], static_cast<uint32_t>((128 + N) * kb));
    tma_load_4d_w(sa, &ta, 0, 0, 0, 0, &bars[0]);
    tma_load_4d_w(sb, &tb, 0, 0, 0, 0, &bars[0]);
    if (mbar_wait_warp(&bars[0], 0, abort)) {
      tc_fence_after();
      // 128-, 64- or 32-byte swizzle
      const uint32_t layout = kb == 128 ? 2u : kb == 64 ? 4u : 6u;
      const uint32_t idesc = idesc_mxf4nvf4(128, N);
      if (mode == 1) {
        for (int kk = 0; kk < nmma; ++kk) {
          tmem_cp_32x128_x4_w(tmem + 256 + 4 * kk, smem_u32(sfs + kk * 512));
          tmem_cp_32x128_x4_w(tmem + 288 + 4 * kk, smem_u32(sfs + (nmma + kk) * 512));
        }
      }
      for (int kk = 0; kk < nmma; ++kk)
        umma_fp4_ss_w(tmem, sdesc(smem_u32(sa) + 32 * kk, 16, 8 * kb, layout),
                      sdesc(smem_u32(sb) + 32 * kk, 16, 8 * kb, layout), idesc,
                      tmem + 256 + kk * sf_stride, tmem + 288 + kk * sf_stride, kk > 0 ? 1u : 0u);
      umma_commit_w(&bars[2]);
    }
  }
  __syncthreads();
  const bool done = mbar_wait_warp(&bars[2], 0, abort);
  if (done && !*abort) {
    tc_fence_after();
    const int row = threadIdx.x;
    uint32_t r[32];
    for (int cc = 0; cc < N / 32; ++cc) {
      tmem_ld32(tmem + lane_base + cc * 32, r);
      tmem_wait_ld();
      for (int i = 0; i < 32; ++i) c[row * N + cc * 32 + i] = __uint_as_float(r[i]);
    }
    for (int cc = 0; cc < 2; ++cc) {
      tmem_ld32(tmem + lane_base + 256 + cc * 32, r);
      tmem_wait_ld();
      for (int i = 0; i < 32; ++i) dump[row * 64 + cc * 32 + i] = r[i];
    }
  }
  tc_fence_before();
  __syncthreads();
  report_abort(abort, err);
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

__global__ void selftest_timeout_kernel(int64_t limit_ns, int* __restrict__ err) {
  __shared__ uint64_t bar;
  __shared__ int abort;
  if (threadIdx.x == 0) {
    abort = 0;
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // nothing ever arrives on `bar`: the wait must give up after limit_ns
    mbar_wait(&bar, 0, &abort, static_cast<uint64_t>(limit_ns));
  }
  __syncthreads();
  report_abort(&abort, err);
}

// Is ex2.approx.ftz.f32 non-decreasing?  Every pair of consecutive floats in
// [-200, 2] (in increasing order: bit patterns 0xC3480000 down to 0x80000000,
// then 0 up to 0x40000000); out[0] counts pairs with 2^next < 2^this, out[1]
// is the first such index (all ones if none).
constexpr uint64_t kMonoNeg = 0xC3480000ull - 0x80000000ull + 1;  // -200 .. -0
constexpr uint64_t kMonoN = kMonoNeg + 0x40000000ull + 1;          // .. 2.0

__device__ __forceinline__ float mono_value(uint64_t i) {
  return __uint_as_float(static_cast<uint32_t>(i < kMonoNeg ? 0xC3480000ull - i : i - kMonoNeg));
}

__global__ void __launch_bounds__(256) selftest_ex2_monotone_kernel(
    unsigned long long* __restrict__ out) {
  const uint64_t stride = static_cast<uint64_t>(gridDim.x) * blockDim.x;
  unsigned long long bad = 0, first = ~0ull;
  for (uint64_t i = static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i + 1 < kMonoN;
       i += stride) {
    if (ex2_f32(mono_value(i + 1)) < ex2_f32(mono_value(i))) {
      ++bad;
      first = first < i ? first : i;
    }
  }
  if (bad != 0) {
    atomicAdd(&out[0], bad);
    atomicMin(&out[1], first);
  }
}

}  // namespace

cudaError_t launch_selftest_umma(const CUtensorMap& ta, const CUtensorMap& tb, const void* a,
                                 float* c, int N, int K, int a_mn, int b_mn, int* err,
                                 cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(selftest_umma_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  selftest_umma_kernel<<<1, 128, kSmem, stream>>>(ta, tb, static_cast<const uint32_t*>(a), c, N, K,
                                                  a_mn, b_mn, err);
  return cudaGetLastError();
}

cudaError_t launch_selftest_fp4(const CUtensorMap& ta, const CUtensorMap& tb, const uint32_t* sf_img,
                                const uint8_t* sf_src, float* c, uint32_t* dump, int N, int nmma,
                                int sf_stride, int mode, int* err, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(selftest_fp4_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kFp4Smem);
  if (e != cudaSuccess) return e;
  selftest_fp4_kernel<<<1, 128, kFp4Smem, stream>>>(ta, tb, sf_img, sf_src, c, dump, N, nmma,
                                                     sf_stride, mode, err);
  return cudaGetLastError();
}

cudaError_t launch_selftest_ex2_monotone(unsigned long long* out, cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(out, 0, sizeof(unsigned long long), stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(out + 1, 0xFF, sizeof(unsigned long long), stream);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 152;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  selftest_ex2_monotone_kernel<<<sms * 8, 256, 0, stream>>>(out);
  return cudaGetLastError();
}

cudaError_t launch_selftest_timeout(int64_t limit_ns, int* err, cudaStream_t stream) {
  selftest_timeout_kernel<<<1, 32, 0, stream>>>(limit_ns, err);
  return cudaGetLastError();
}

}  // namespace nvq
