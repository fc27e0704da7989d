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

// Raster index of the token at cube-order position i.
__device__ __forceinline__ int64_t cube_to_raster(int64_t i, const CubeGrid& g) {
  const int64_t c = static_cast<int64_t>(g.ct) * g.ch * g.cw;
  const int64_t cube = i / c, inner = i - cube * c;
  const int ncw = g.W / g.cw, nch = g.Hh / g.ch;
  const int64_t c2 = cube % ncw, c1 = (cube / ncw) % nch, c0 = cube / (static_cast<int64_t>(ncw) * nch);
  const int64_t a = inner / (g.ch * g.cw), bb = (inner / g.cw) % g.ch, cc = inner % g.cw;
  const int64_t t = c0 * g.ct + a, hh = c1 * g.ch + bb, w = c2 * g.cw + cc;
  return (t * g.Hh + hh) * g.W + w;
}

// Cube-order position of the token at raster index i.
__device__ __forceinline__ int64_t raster_to_cube(int64_t i, const CubeGrid& g) {
  const int64_t t = i / (static_cast<int64_t>(g.Hh) * g.W);
  const int64_t hh = (i / g.W) % g.Hh, w = i % g.W;
  const int ncw = g.W / g.cw, nch = g.Hh / g.ch;
  const int64_t cube = ((t / g.ct) * nch + hh / g.ch) * ncw + w / g.cw;
  const int64_t inner = ((t % g.ct) * g.ch + hh % g.ch) * g.cw + w % g.cw;
  return cube * (static_cast<int64_t>(g.ct) * g.ch * g.cw) + inner;
}

// out[b, i] = x[b, src(i)] for rows of `row_vec` 16-byte vectors.
__global__ void __launch_bounds__(256) vsa_reorder_kernel(const uint4* __restrict__ x,
                                                          uint4* __restrict__ out, int B,
                                                          CubeGrid g, int to_cubes, int row_vec) {
  const int64_t n = static_cast<int64_t>(g.T) * g.Hh * g.W;
  const int64_t rows = n * B;
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
       row < rows; row += warps) {
    const int64_t b = row / n, i = row - b * n;
    const int64_t src = to_cubes ? cube_to_raster(i, g) : raster_to_cube(i, g);
    const uint4* s = x + (b * n + src) * row_vec;
    uint4* d = out + row * row_vec;
    for (int v = lane; v < row_vec; v += 32) d[v] = s[v];
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

// One CTA per (query tile, h, b).
__global__ void __launch_bounds__(256) vsa_topk_kernel(const float* __restrict__ qm,
                                                       const float* __restrict__ km, int H,
                                                       int n, int D, int topk,
                                                       int* __restrict__ out) {
  extern __shared__ float sh[];
  float* qrow = sh;             // [D]
  float* score = sh + D;        // [n]
  int* sel = reinterpret_cast<int*>(score + n);  // [n]
  const int i = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int64_t head = static_cast<int64_t>(b) * H + h;
  for (int d = threadIdx.x; d < D; d += blockDim.x) qrow[d] = qm[(head * n + i) * D + d];
  __syncthreads();
  for (int j = threadIdx.x; j < n; j += blockDim.x) {
    const float* kr = km + (head * n + j) * D;
    float a = 0.f;
    for (int d = 0; d < D; ++d) a = fmaf(qrow[d], kr[d], a);
    score[j] = a;
  }
  __syncthreads();
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
  vsa_reorder_kernel<<<grid, 256, 0, stream>>>(static_cast<const uint4*>(x), static_cast<uint4*>(out),
                                               B, g, to_cubes, row_vec);
  return cudaGetLastError();
}

cudaError_t launch_vsa_select(const void* q, const void* k, int B, int N, int H, int D, int topk,
                              int* kv_tiles, float* qm, float* km, cudaStream_t stream) {
  const int n = N / kTileTokens;
  const dim3 grid(n, H, B);
  vsa_tile_mean_kernel<<<grid, D, 0, stream>>>(static_cast<const uint16_t*>(q), qm, N, H, D);
  vsa_tile_mean_kernel<<<grid, D, 0, stream>>>(static_cast<const uint16_t*>(k), km, N, H, D);
  const size_t smem = static_cast<size_t>(D + 2 * n) * 4;
  if (smem > 48 * 1024) return cudaErrorInvalidValue;
  vsa_topk_kernel<<<grid, 256, smem, stream>>>(qm, km, H, n, D, topk, kv_tiles);
  return cudaGetLastError();
}

}  // namespace nvq
