// Video sparse attention (VSA) support for the block-sparse fine attention
// ("vsqa-preview-1.3b metadata.json", attention: kind vsa, cube_shape [4, 4, 8],
// selection sparsity and effective_topk):
//   * vsa_reorder_kernel   token rows between raster (t, h, w) order of the latent
//                          and cube order (cubes in raster order over the cube
//                          grid, tokens in raster order inside a cube); one warp
//                          copies one token's H*D values (contiguous in [B,N,H,D]);
//   * vsa_tile_mean_kernel the fp32 mean of Q or K over each 128-token tile;
//   * vsa_topk_kernel      per query tile, the fp32 scores mean_q . mean_k for
//                          every key tile and the topk of highest score (ties to
//                          the lower index), written in ascending tile order.
// All three are small next to the attention kernels (memory- or latency-bound).
#include <cstdint>

#include <cuda_runtime.h>

#include "nvq_internal.h"

namespace nvq {

namespace {

constexpr int kTileTokens = 128;  // one 4x4x8 cube = one attention tile

struct CubeGrid {
  int T, Hh, W, ct, ch, cw;
};

// Raster index of the token at cube-order position i (I: int, or int64_t when
// a batch's tokens do not fit in 31 bits).
template <typename I>
__device__ __forceinline__ I cube_to_raster(I i, const CubeGrid& g) {
  const I c = static_cast<I>(g.ct) * g.ch * g.cw;
  const I cube = i / c, inner = i - cube * c;
  const int ncw = g.W / g.cw, nch = g.Hh / g.ch;
  const I c2 = cube % ncw, c1 = (cube / ncw) % nch, c0 = cube / (static_cast<I>(ncw) * nch);
  const I a = inner / (g.ch * g.cw), bb = (inner / g.cw) % g.ch, cc = inner % g.cw;
  const I t = c0 * g.ct + a, hh = c1 * g.ch + bb, w = c2 * g.cw + cc;
  return (t * g.Hh + hh) * g.W + w;
}

// Cube-order position of the token at raster index i.
template <typename I>
__device__ __forceinline__ I raster_to_cube(I i, const CubeGrid& g) {
  const I t = i / (static_cast<I>(g.Hh) * g.W);
  const I hh = (i / g.W) % g.Hh, w = i % g.W;
  const int ncw = g.W / g.cw, nch = g.Hh / g.ch;
  const I cube = ((t / g.ct) * nch + hh / g.ch) * ncw + w / g.cw;
  const I inner = ((t % g.ct) * g.ch + hh % g.ch) * g.cw + w % g.cw;
  return cube * (static_cast<I>(g.ct) * g.ch * g.cw) + inner;
}

__device__ __forceinline__ uint4 ld_nc_v4(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ void st_cs_v4(uint4* p, const uint4& v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

// out[b, i] = x[b, src(i)] for rows of `row_vec` 16-byte vectors.  A warp
// copies one row, up to 256 vectors (8 per lane) in flight before any store;
// I: the index type (int whenever all B * n rows fit in 31 bits).
template <typename I>
__global__ void __launch_bounds__(256) vsa_reorder_kernel(const uint4* __restrict__ x,
                                                          uint4* __restrict__ out, int B,
                                                          CubeGrid g, int to_cubes, int row_vec) {
  const I n = static_cast<I>(g.T) * g.Hh * g.W;
  const I rows = n * B;
  const int lane = threadIdx.x & 31;
  const I warps = static_cast<I>(gridDim.x) * (blockDim.x >> 5);
  for (I row = static_cast<I>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); row < rows;
       row += warps) {
    const I b = row / n, i = row - b * n;
    const I src = to_cubes ? cube_to_raster<I>(i, g) : raster_to_cube<I>(i, g);
    const uint4* s = x + (static_cast<int64_t>(b) * n + src) * row_vec;
    uint4* d = out + static_cast<int64_t>(row) * row_vec;
    for (int v0 = 0; v0 < row_vec; v0 += 256) {
      uint4 buf[8];
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (v0 + lane + 32 * k < row_vec) buf[k] = ld_nc_v4(s + v0 + lane + 32 * k);
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (v0 + lane + 32 * k < row_vec) st_cs_v4(d + v0 + lane + 32 * k, buf[k]);
    }
  }
}

// means[b, h, tile, d] = mean over the tile's 128 tokens of x[b, token, h, d] (bf16).
__global__ void vsa_tile_mean_kernel(const uint16_t* __restrict__ x, float* __restrict__ means,
                                     int N, int H, int D) {
  const int tile = blockIdx.x, h = blockIdx.y, b = blockIdx.z, d = threadIdx.x;
  const int n_tiles = N / kTileTokens;
  const uint16_t* p = x + ((static_cast<int64_t>(b) * N + static_cast<int64_t>(tile) * kTileTokens) * H + h) * D + d;
  float acc = 0.f;
  for (int r = 0; r < kTileTokens; ++r)
    acc += __uint_as_float(static_cast<uint32_t>(p[static_cast<int64_t>(r) * H * D]) << 16);
  means[((static_cast<int64_t>(b) * H + h) * n_tiles + tile) * D + d] = acc * (1.0f / kTileTokens);
}

// One CTA per (query tile, h, b), 256 threads.  Selection: the topk tiles of
// highest score, ties to the lower index, written in ascending tile order.
// Up to 256 key tiles, a bitonic sort of one 64-bit key per tile (the score's
// order-preserving bits above the complemented index, sorted descending: higher
// score first, then lower index); beyond that, each tile's rank is counted.
__global__ void __launch_bounds__(256) vsa_topk_kernel(const float* __restrict__ qm,
                                                       const float* __restrict__ km, int H,
                                                       int n, int D, int topk,
                                                       int* __restrict__ out) {
  extern __shared__ __align__(16) unsigned char sh_raw[];
  uint64_t* key = reinterpret_cast<uint64_t*>(sh_raw);   // [256]
  int* wcount = reinterpret_cast<int*>(key + 256);       // [8]
  float* qrow = reinterpret_cast<float*>(wcount + 8);    // [D]
  float* score = qrow + D;                                // [n]
  int* sel = reinterpret_cast<int*>(score + n);           // [n]
  const int i = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int64_t head = static_cast<int64_t>(b) * H + h;
  for (int d = threadIdx.x; d < D; d += blockDim.x) qrow[d] = qm[(head * n + i) * D + d];
  for (int j = threadIdx.x; j < n; j += blockDim.x) sel[j] = 0;
  __syncthreads();
  // scores: one warp per key tile, lanes over d (coalesced rows of km), four
  // tiles at a time so their loads are in flight together; the lane partial
  // sums added by a butterfly; fp32 throughout
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  for (int j0 = warp; j0 < n; j0 += 4 * nwarps) {
    float a[4] = {0.f, 0.f, 0.f, 0.f};
    for (int d = lane; d < D; d += 32) {
      const float qd = qrow[d];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j = j0 + u * nwarps;
        if (j < n) a[u] = fmaf(qd, km[(head * n + j) * D + d], a[u]);
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) a[u] += __shfl_xor_sync(0xFFFFFFFFu, a[u], o);
      const int j = j0 + u * nwarps;
      if (lane == 0 && j < n) score[j] = a[u];
    }
  }
  __syncthreads();
  const int t = threadIdx.x;
  if (n <= 256) {
    uint64_t kv = 0;  // padding sorts last
    if (t < n) {
      const uint32_t bits = __float_as_uint(score[t] + 0.0f);  // -0 as +0: equal scores tie
      const uint32_t ord = (bits & 0x80000000u) ? ~bits : (bits | 0x80000000u);
      kv = (static_cast<uint64_t>(ord) << 32) | static_cast<uint32_t>(~t);
    }
    key[t] = kv;
    __syncthreads();
    for (int size = 2; size <= 256; size <<= 1) {
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        const int p = t ^ stride;
        if (p > t) {
          const uint64_t x0 = key[t], x1 = key[p];
          if (((t & size) == 0) ? x0 < x1 : x0 > x1) {  // descending runs where t & size == 0
            key[t] = x1;
            key[p] = x0;
          }
        }
        __syncthreads();
      }
    }
    if (t < topk && t < n) sel[~static_cast<uint32_t>(key[t])] = 1;
    __syncthreads();
    // ascending output: position = selected tiles before this one (warp ballots)
    const bool f = t < n && sel[t] != 0;
    const uint32_t bal = __ballot_sync(0xFFFFFFFFu, f);
    if (lane == 0) wcount[warp] = __popc(bal);
    __syncthreads();
    if (f) {
      int pos = __popc(bal & ((1u << lane) - 1u));
      for (int w = 0; w < warp; ++w) pos += wcount[w];
      if (pos < topk) out[(head * n + i) * topk + pos] = t;
    }
    return;
  }
  for (int j = threadIdx.x; j < n; j += blockDim.x) {  // rank by (score desc, index asc)
    const float sj = score[j];
    int rank = 0;
    for (int j2 = 0; j2 < n; ++j2) rank += (score[j2] > sj || (score[j2] == sj && j2 < j)) ? 1 : 0;
    sel[j] = rank < topk ? 1 : 0;
  }
  __syncthreads();
  int* o = out + (head * n + i) * topk;
  for (int j = threadIdx.x; j < n; j += blockDim.x) {
    if (!sel[j]) continue;
    int pos = 0;
    for (int j2 = 0; j2 < j; ++j2) pos += sel[j2];
    if (pos < topk) o[pos] = j;  // ranks are distinct for finite scores: exactly topk selected
  }
}

}  // namespace

cudaError_t launch_vsa_reorder(const void* x, int B, int T, int Hh, int W, int H, int D, int ct,
                               int ch, int cw, int to_cubes, void* out, cudaStream_t stream) {
  const CubeGrid g{T, Hh, W, ct, ch, cw};
  const int row_vec = H * D * 2 / 16;
  const int64_t rows = static_cast<int64_t>(B) * T * Hh * W;
  int dev = 0, sms = 152;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t blocks = (rows + 7) / 8;  // 8 warps per block, one row per warp
  const int grid = static_cast<int>(blocks < static_cast<int64_t>(sms) * 16 ? blocks : sms * 16);
  if (rows < (int64_t{1} << 31))
    vsa_reorder_kernel<int><<<grid, 256, 0, stream>>>(
        static_cast<const uint4*>(x), static_cast<uint4*>(out), B, g, to_cubes, row_vec);
  else
    vsa_reorder_kernel<int64_t><<<grid, 256, 0, stream>>>(
        static_cast<const uint4*>(x), static_cast<uint4*>(out), B, g, to_cubes, row_vec);
  return cudaGetLastError();
}

cudaError_t launch_vsa_select(const void* q, const void* k, int B, int N, int H, int D, int topk,
                              int* kv_tiles, float* qm, float* km, cudaStream_t stream) {
  const int n = N / kTileTokens;
  const dim3 grid(n, H, B);
  vsa_tile_mean_kernel<<<grid, D, 0, stream>>>(static_cast<const uint16_t*>(q), qm, N, H, D);
  vsa_tile_mean_kernel<<<grid, D, 0, stream>>>(static_cast<const uint16_t*>(k), km, N, H, D);
  const size_t smem = 256 * 8 + 8 * 4 + static_cast<size_t>(D + 2 * n) * 4;
  if (smem > 48 * 1024) return cudaErrorInvalidValue;
  vsa_topk_kernel<<<grid, 256, smem, stream>>>(qm, km, H, n, D, topk, kv_tiles);
  return cudaGetLastError();
}

}  // namespace nvq
