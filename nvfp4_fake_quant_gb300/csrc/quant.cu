// Standalone NVFP4 quantizer kernels (HBM-bound) and the static global scale.
//
// One thread quantizes one 16-element block: two 16-byte loads, one 32-byte
// output, one scale byte and/or 8 code bytes.  A warp covers 32 consecutive
// blocks of a row (1 KiB of input), so loads and stores are fully coalesced.
// Contiguous operands take a flat grid-stride loop over the blocks (a whole
// number of waves over the SMs); strided ones a 2-D grid (blocks of a row along
// x, rows along y), so no thread divides a 64-bit index.
#include <algorithm>

#include <cuda_runtime.h>

#include "nvq_internal.h"
#include "nvq_ptx.cuh"
#include "nvq_quant.cuh"

namespace nvq {

namespace {

__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

struct Block16 {
  uint4 lo, hi;
};

__device__ __forceinline__ Block16 load_block(const uint16_t* __restrict__ src) {
  return {ld_stream(src), ld_stream(src + 8)};
}

// g: the global scale (1 for the unit modes), inv_g = RN(1/g).
template <int MODE>
__device__ __forceinline__ void quant_block(const Block16& v, const float g, const float inv_g,
                                            uint16_t* __restrict__ out, uint8_t* __restrict__ sc,
                                            uint8_t* __restrict__ cd) {
  const uint32_t xv[8] = {v.lo.x, v.lo.y, v.lo.z, v.lo.w, v.hi.x, v.hi.y, v.hi.z, v.hi.w};
  Q16 q;
  if constexpr (MODE == kStaticBf16) {
    q = out != nullptr ? quant16_static_fast<true>(xv, g, inv_g)
                       : quant16_static_fast<false>(xv, g, inv_g);
  } else {
    q = quant16_unit<MODE == kUnitF16>(xv);
  }
  if (out != nullptr) {
    uint4* dst = reinterpret_cast<uint4*>(out);
    dst[0] = make_uint4(q.out[0], q.out[1], q.out[2], q.out[3]);
    dst[1] = make_uint4(q.out[4], q.out[5], q.out[6], q.out[7]);
  }
  if (sc != nullptr) *sc = static_cast<uint8_t>(q.sbyte);
  if (cd != nullptr) {
    code_signs(xv, q.codes);
    *reinterpret_cast<uint2*>(cd) = make_uint2(q.codes[0], q.codes[1]);
  }
}

// Contiguous operands (row strides equal to the row lengths): block i of the
// flattened matrix at element 16 i, scale byte i, code bytes 8 i.  Each thread
// takes several blocks a pass (a grid stride apart): four with a unit scale, two
// with a static one (whose longer arithmetic needs the registers), and issues
// the next pass's loads before this pass's arithmetic, so that HBM reads stay in
// flight while the threads quantize (the grid is one wave, a few passes each).
template <int MODE>
__global__ void __launch_bounds__(256) fake_quant_flat_kernel(
    const uint16_t* __restrict__ x, int64_t nblocks, const float* __restrict__ gsf,
    uint16_t* __restrict__ out, uint8_t* __restrict__ scales, uint8_t* __restrict__ codes) {
  constexpr int kUnroll = MODE == kStaticBf16 ? 2 : 4;
  const float g = (MODE == kStaticBf16) ? *gsf : 1.0f;
  const float inv_g = (MODE == kStaticBf16) ? __frcp_rn(g) : 1.0f;
  const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x;
  int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  Block16 v[kUnroll];
#pragma unroll
  for (int u = 0; u < kUnroll; ++u)
    if (i + u * step < nblocks) v[u] = load_block(x + (i + u * step) * 16);
  for (; i < nblocks; i += kUnroll * step) {
    // the next pass's loads go out before this pass's arithmetic
    const int64_t in = i + kUnroll * step;
    Block16 nv[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
      if (in + u * step < nblocks) nv[u] = load_block(x + (in + u * step) * 16);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t b = i + u * step;
      if (b < nblocks)
        quant_block<MODE>(v[u], g, inv_g, out != nullptr ? out + b * 16 : nullptr,
                          scales != nullptr ? scales + b : nullptr,
                          codes != nullptr ? codes + b * 8 : nullptr);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) v[u] = nv[u];
  }
}

// Strided operands: rows over grid y, 16-element blocks of a row over grid x.
template <int MODE>
__global__ void __launch_bounds__(256) fake_quant_rows_kernel(
    const uint16_t* __restrict__ x, int64_t rows, int64_t nbc, int64_t ld_x,
    const float* __restrict__ gsf, uint16_t* __restrict__ out, int64_t ld_out,
    uint8_t* __restrict__ scales, int64_t ld_s, uint8_t* __restrict__ codes, int64_t ld_c) {
  const float g = (MODE == kStaticBf16) ? *gsf : 1.0f;
  const float inv_g = (MODE == kStaticBf16) ? __frcp_rn(g) : 1.0f;
  const int64_t cstep = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t r = blockIdx.y; r < rows; r += gridDim.y) {
    for (int64_t cb = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; cb < nbc;
         cb += cstep)
      quant_block<MODE>(load_block(x + r * ld_x + cb * 16), g, inv_g,
                        out != nullptr ? out + r * ld_out + cb * 16 : nullptr,
                        scales != nullptr ? scales + r * ld_s + cb : nullptr,
                        codes != nullptr ? codes + r * ld_c + cb * 8 : nullptr);
  }
}

// Q or K of attention for the block-scaled FP4 UMMA.  x: bf16 [B, N, H, D]
// (contiguous); codes: [B, N, H, D/2] bytes, two E2M1 codes a byte (the even
// element in the low nibble, the sign bit of x on zero codes); scales: for each
// (b, h), 128-token tile t and 64 elements kk of D, one 512-byte block at
// (((b H + h) n_tiles + t) (D/64) + kk) * 512 holding the E4M3 scale of token r
// of the tile, 16-element block j of the 64, at byte (r % 32) * 16 + (r / 32) * 4
// + j -- the tensor-memory layout of the UMMA's scale operand, so that one
// copy per block moves it there.  Tokens of the last tile beyond N get scale 0.
// Blocks i < nblocks are the input's 16-element blocks in memory order (two
// per thread in flight); the npad indices after them zero the padding scales.
__global__ void __launch_bounds__(256) quant_attn_fp4_kernel(
    const uint16_t* __restrict__ x, uint32_t nblocks, uint32_t npad, uint32_t N, uint32_t H,
    uint32_t lg_nbd, uint32_t n_tiles, uint8_t* __restrict__ codes, uint8_t* __restrict__ scales) {
  const uint32_t nbd = 1u << lg_nbd;  // 16-element blocks per row (D / 16)
  const uint32_t nkk = nbd >> 2;      // 64-element groups per row
  const uint32_t step = gridDim.x * blockDim.x;
  auto scale_at = [&](uint32_t bh, uint32_t n, uint32_t cb) -> uint8_t* {
    return scales + ((static_cast<int64_t>(bh) * n_tiles + (n >> 7)) * nkk + (cb >> 2)) * 512 +
           (n & 31u) * 16 + ((n >> 5) & 3u) * 4 + (cb & 3u);
  };
  constexpr uint32_t kUnroll = 2;
  for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < nblocks; i += kUnroll * step) {
    Block16 v[kUnroll];
#pragma unroll
    for (uint32_t u = 0; u < kUnroll; ++u)
      if (i + u * step < nblocks) v[u] = load_block(x + static_cast<int64_t>(i + u * step) * 16);
#pragma unroll
    for (uint32_t u = 0; u < kUnroll; ++u) {
      const uint32_t blk = i + u * step;
      if (blk >= nblocks) continue;
      const uint32_t xv[8] = {v[u].lo.x, v[u].lo.y, v[u].lo.z, v[u].lo.w,
                              v[u].hi.x, v[u].hi.y, v[u].hi.z, v[u].hi.w};
      Q16 q = quant16_unit<false>(xv);
      code_signs(xv, q.codes);
      *reinterpret_cast<uint2*>(codes + static_cast<int64_t>(blk) * 8) =
          make_uint2(q.codes[0], q.codes[1]);
      const uint32_t row = blk >> lg_nbd, cb = blk & (nbd - 1u);
      const uint32_t bn = row / H, h = row - bn * H;
      const uint32_t b = bn / N, n = bn - b * N;
      *scale_at(b * H + h, n, cb) = static_cast<uint8_t>(q.sbyte);
    }
  }
  const uint32_t pad_rows = n_tiles * 128u - N;
  for (uint32_t j = blockIdx.x * blockDim.x + threadIdx.x; j < npad; j += step) {
    const uint32_t cb = j & (nbd - 1u), t = j >> lg_nbd;
    const uint32_t bh = t / pad_rows, n = N + (t - bh * pad_rows);
    *scale_at(bh, n, cb) = 0;
  }
}

// Every quantized form of up to three attention operands in one launch.  Blocks
// of all jobs form one flat index space (job after job, 16-element blocks in
// memory order, two in flight per thread); each block's decision is taken once
// (quant16_unit) and written in every form its job asks for.  The f16 value of
// a code times an E4M3 scale is exact, and so is its bf16 rounding (at most 6
// significant bits), so both copies hold the same numbers.  The indices after
// the blocks zero the scales of the padding tokens of the last 128-token tile
// of every job that writes scale blocks.
__global__ void __launch_bounds__(256) quant_attn_ops_kernel(const AttnOpJobs jobs) {
  const uint32_t nbd = 1u << jobs.lg_nbd;  // 16-element blocks per row (D / 16)
  const uint32_t nkk = nbd >> 2;           // 64-element groups per row
  const uint32_t step = gridDim.x * blockDim.x;
  const uint32_t n0 = jobs.j[0].nblocks, n01 = n0 + jobs.j[1].nblocks;
  const uint32_t total = n01 + jobs.j[2].nblocks;
  auto scale_at = [&](const AttnOpJob& jb, uint32_t bh, uint32_t n, uint32_t cb) -> uint8_t* {
    return jb.scales +
           ((static_cast<int64_t>(bh) * jb.n_tiles + (n >> 7)) * nkk + (cb >> 2)) * 512 +
           (n & 31u) * 16 + ((n >> 5) & 3u) * 4 + (cb & 3u);
  };
  constexpr uint32_t kUnroll = 2;
  for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += kUnroll * step) {
    Block16 v[kUnroll];
    uint32_t jid[kUnroll], blk[kUnroll];
#pragma unroll
    for (uint32_t u = 0; u < kUnroll; ++u) {
      const uint32_t g = i + u * step;
      jid[u] = g < n0 ? 0u : (g < n01 ? 1u : 2u);
      blk[u] = g - (jid[u] == 0 ? 0u : (jid[u] == 1 ? n0 : n01));
      if (g < total) v[u] = load_block(jobs.j[jid[u]].x + static_cast<int64_t>(blk[u]) * 16);
    }
#pragma unroll
    for (uint32_t u = 0; u < kUnroll; ++u) {
      if (i + u * step >= total) continue;
      const AttnOpJob& jb = jobs.j[jid[u]];
      const uint32_t xv[8] = {v[u].lo.x, v[u].lo.y, v[u].lo.z, v[u].lo.w,
                              v[u].hi.x, v[u].hi.y, v[u].hi.z, v[u].hi.w};
      Q16 q = quant16_unit<true>(xv);  // f16 dequantized values
      const int64_t e0 = static_cast<int64_t>(blk[u]) * 16;
      if (jb.f16 != nullptr) {
        uint4* dst = reinterpret_cast<uint4*>(jb.f16 + e0);
        dst[0] = make_uint4(q.out[0], q.out[1], q.out[2], q.out[3]);
        dst[1] = make_uint4(q.out[4], q.out[5], q.out[6], q.out[7]);
      }
      if (jb.bf16 != nullptr) {
        uint32_t w[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          __nv_bfloat162 bv = __floats2bfloat162_rn(f16lo_to_f32(q.out[k]), f16lo_to_f32(q.out[k] >> 16));
          w[k] = *reinterpret_cast<uint32_t*>(&bv) | (q.out[k] & 0x80008000u);  // keeps -0
        }
        uint4* dst = reinterpret_cast<uint4*>(jb.bf16 + e0);
        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
      }
      if (jb.codes != nullptr) {
        code_signs(xv, q.codes);
        *reinterpret_cast<uint2*>(jb.codes + static_cast<int64_t>(blk[u]) * 8) =
            make_uint2(q.codes[0], q.codes[1]);
      }
      if (jb.scales != nullptr) {
        const uint32_t row = blk[u] >> jobs.lg_nbd, cb = blk[u] & (nbd - 1u);
        const uint32_t bn = row / jobs.H, h = row - bn * jobs.H;
        const uint32_t b = bn / jb.N, n = bn - b * jb.N;
        *scale_at(jb, b * jobs.H + h, n, cb) = static_cast<uint8_t>(q.sbyte);
      }
    }
  }
  // padding tokens of the last tile: scale 0
  const uint32_t p0 = jobs.j[0].npad, p01 = p0 + jobs.j[1].npad, ptot = p01 + jobs.j[2].npad;
  for (uint32_t t = blockIdx.x * blockDim.x + threadIdx.x; t < ptot; t += step) {
    const uint32_t j = t < p0 ? 0u : (t < p01 ? 1u : 2u);
    const AttnOpJob& jb = jobs.j[j];
    const uint32_t idx = t - (j == 0 ? 0u : (j == 1 ? p0 : p01));
    const uint32_t pad_rows = jb.n_tiles * 128u - jb.N;
    const uint32_t cb = idx & (nbd - 1u), r = idx >> jobs.lg_nbd;
    const uint32_t bh = r / pad_rows, n = jb.N + (r - bh * pad_rows);
    *scale_at(jb, bh, n, cb) = 0;
  }
}

// Byte offset of the scale of (row r, 16-element block cb) in the 128x4 tiled
// layout of block-scaled FP4 GEMMs: 512-byte tiles of 128 rows x 4 blocks,
// tiles ordered by row tile, then block tile (n_bt tiles per row tile); inside
// a tile, row r sits at (r % 32) * 16 + (r / 32 % 4) * 4 and block cb at cb % 4.
__device__ __forceinline__ int64_t tiled_scale_offset(int64_t r, int64_t cb, int64_t n_bt) {
  return ((r >> 7) * n_bt + (cb >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (cb & 3);
}

// Packed codes (row-major, cols/2 bytes per row) and scales in the tiled layout.
// A flat grid-stride loop over the rows*nbc blocks, each thread loading two
// blocks before quantizing.  A block's (row, block column) is split off its
// flat index once per thread and then advanced by the grid stride's own
// (rows, columns) with one carry, with no division per block.
template <int MODE>
__global__ void __launch_bounds__(256) quant_tiled_kernel(
    const uint16_t* __restrict__ x, int64_t rows, int64_t nbc, int64_t ld_x,
    const float* __restrict__ gsf, uint8_t* __restrict__ codes, uint8_t* __restrict__ scales) {
  const float g = (MODE == kStaticBf16) ? *gsf : 1.0f;
  const float inv_g = (MODE == kStaticBf16) ? __frcp_rn(g) : 1.0f;
  const int64_t total = rows * nbc;
  const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t n_bt = (nbc + 3) / 4;
  const int64_t i0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  int64_t r0 = i0 / nbc, c0 = i0 - r0 * nbc;         // block i
  const int64_t dr = step / nbc, dc = step - dr * nbc;  // the grid stride
  auto advance = [&](int64_t& r, int64_t& c) {
    r += dr;
    c += dc;
    if (c >= nbc) {
      c -= nbc;
      ++r;
    }
  };
  for (int64_t i = i0; i < total; i += 2 * step) {
    int64_t r1 = r0, c1 = c0;
    advance(r1, c1);  // block i + step
    const bool two = i + step < total;
    const Block16 v0 = load_block(x + r0 * ld_x + c0 * 16);
    Block16 v1;
    if (two) v1 = load_block(x + r1 * ld_x + c1 * 16);
    quant_block<MODE>(v0, g, inv_g, nullptr, scales + tiled_scale_offset(r0, c0, n_bt), codes + i * 8);
    if (two)
      quant_block<MODE>(v1, g, inv_g, nullptr, scales + tiled_scale_offset(r1, c1, n_bt),
                        codes + (i + step) * 8);
    r0 = r1;
    c0 = c1;
    advance(r0, c0);  // block i + 2 step
  }
}

// amax(|x|) of a contiguous operand as a flat array of 16-byte vectors, four
// loads in flight per thread.
__global__ void __launch_bounds__(256) amax_flat_kernel(const uint4* __restrict__ x, int64_t nvec,
                                                        unsigned int* __restrict__ amax_bits) {
  const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x;
  uint32_t m = 0;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < nvec;
       i += 4 * step) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      v[u] = i + u * step < nvec ? ld_stream(x + i + u * step) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        m = max(m, w[j] & 0x7FFFu);
        m = max(m, (w[j] >> 16) & 0x7FFFu);
      }
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
  if ((threadIdx.x & 31) == 0 && m != 0) atomicMax(amax_bits, m << 16);  // bf16 -> f32 bits
}

// amax(|x|) as the unsigned bit pattern of a non-negative float (monotone).
__global__ void __launch_bounds__(256) amax_kernel(const uint16_t* __restrict__ x, int64_t rows,
                                                   int64_t cols, int64_t ld_x,
                                                   unsigned int* __restrict__ amax_bits) {
  const int64_t nvec = cols / 8;  // 16-byte vectors per row (cols % 8 handled below)
  const int64_t total = rows * nvec;
  const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x;
  uint32_t m = 0;  // max of |bf16| bit patterns (monotone for non-negative values)
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += step) {
    const int64_t r = i / nvec, c = i - r * nvec;
    const uint4 v = ld_stream(x + r * ld_x + c * 8);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      m = max(m, w[j] & 0x7FFFu);
      m = max(m, (w[j] >> 16) & 0x7FFFu);
    }
  }
  const int64_t tail = cols - nvec * 8;
  if (tail > 0) {
    for (int64_t r = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; r < rows;
         r += step) {
      for (int64_t c = nvec * 8; c < cols; ++c)
        m = max(m, static_cast<uint32_t>(x[r * ld_x + c] & 0x7FFFu));
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
  if ((threadIdx.x & 31) == 0 && m != 0) atomicMax(amax_bits, m << 16);  // bf16 -> f32 bits
}

__global__ void global_sf_finalize_kernel(float* gsf) {
  const float amax = __uint_as_float(*reinterpret_cast<unsigned int*>(gsf));
  *gsf = __fdiv_rn(2688.0f, fmaxf(amax, 1e-12f));
}

int grid_for(int64_t work, int threads) {
  int dev = 0, sms = 152;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t waves = 8;  // 8 x 256-thread blocks resident per SM at most
  int64_t blocks = (work + threads - 1) / threads;
  const int64_t cap = static_cast<int64_t>(sms) * waves;
  if (blocks > cap) blocks = cap;
  return static_cast<int>(blocks < 1 ? 1 : blocks);
}

// One full wave of `Kernel` (resident blocks per SM x SMs), at most enough
// blocks for `work` threads.  The occupancy query runs once per kernel (one
// template instance per kernel).
template <auto Kernel>
int wave_grid(int64_t work, int threads) {
  static int per_sm = 0;
  if (per_sm == 0) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, Kernel, threads, 0) != cudaSuccess ||
        n < 1)
      n = 1;
    per_sm = n;
  }
  int dev = 0, sms = 152;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t blocks = std::min<int64_t>((work + threads - 1) / threads,
                                           static_cast<int64_t>(sms) * per_sm);
  return static_cast<int>(std::max<int64_t>(blocks, 1));
}

}  // namespace

cudaError_t launch_fake_quant(const void* x, int64_t rows, int64_t cols, int64_t ld_x,
                              const float* gsf, int mode, void* out, int64_t ld_out,
                              uint8_t* scales, int64_t ld_s, uint8_t* codes, int64_t ld_c,
                              cudaStream_t stream) {
  const int64_t nbc = cols / 16;
  const int threads = 256;
  const auto* xs = static_cast<const uint16_t*>(x);
  auto* os = static_cast<uint16_t*>(out);
  const bool flat = ld_x == cols && (out == nullptr || ld_out == cols) &&
                    (scales == nullptr || ld_s == nbc) && (codes == nullptr || ld_c == cols / 2);
  if (flat) {
    const int64_t nblocks = rows * nbc;
    const int64_t per_thread = mode == kStaticBf16 ? 2 : 4;  // blocks in flight per thread
    const int64_t work = (nblocks + per_thread - 1) / per_thread;  // threads needed
    switch (mode) {
      case kUnitBf16:
        fake_quant_flat_kernel<kUnitBf16>
            <<<wave_grid<fake_quant_flat_kernel<kUnitBf16>>(work, threads), threads, 0, stream>>>(
                xs, nblocks, gsf, os, scales, codes);
        break;
      case kUnitF16:
        fake_quant_flat_kernel<kUnitF16>
            <<<wave_grid<fake_quant_flat_kernel<kUnitF16>>(work, threads), threads, 0, stream>>>(
                xs, nblocks, gsf, os, scales, codes);
        break;
      default:
        fake_quant_flat_kernel<kStaticBf16>
            <<<wave_grid<fake_quant_flat_kernel<kStaticBf16>>(work, threads), threads, 0, stream>>>(
                xs, nblocks, gsf, os, scales, codes);
        break;
    }
    return cudaGetLastError();
  }
  const int64_t gx = std::min<int64_t>((nbc + threads - 1) / threads, 64);
  const int64_t gy = std::max<int64_t>(1, std::min<int64_t>({rows, 65535, grid_for(rows * nbc, threads) / gx + 1}));
  const dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(gy));
  switch (mode) {
    case kUnitBf16:
      fake_quant_rows_kernel<kUnitBf16><<<grid, threads, 0, stream>>>(
          xs, rows, nbc, ld_x, gsf, os, ld_out, scales, ld_s, codes, ld_c);
      break;
    case kUnitF16:
      fake_quant_rows_kernel<kUnitF16><<<grid, threads, 0, stream>>>(
          xs, rows, nbc, ld_x, gsf, os, ld_out, scales, ld_s, codes, ld_c);
      break;
    default:
      fake_quant_rows_kernel<kStaticBf16><<<grid, threads, 0, stream>>>(
          xs, rows, nbc, ld_x, gsf, os, ld_out, scales, ld_s, codes, ld_c);
      break;
  }
  return cudaGetLastError();
}

size_t tiled_scale_bytes(int64_t rows, int64_t cols) {
  const int64_t nbc = cols / 16;
  return static_cast<size_t>((rows + 127) / 128 * 128) * static_cast<size_t>((nbc + 3) / 4 * 4);
}

cudaError_t launch_quant_tiled(const void* x, int64_t rows, int64_t cols, int64_t ld_x,
                               const float* gsf, uint8_t* codes, uint8_t* scales,
                               cudaStream_t stream) {
  const int64_t nbc = cols / 16;
  // padding rows of the last row tile and padding blocks of the last block tile
  // hold zero scales
  if (rows % 128 != 0 || nbc % 4 != 0) {
    const cudaError_t e = cudaMemsetAsync(scales, 0, tiled_scale_bytes(rows, cols), stream);
    if (e != cudaSuccess) return e;
  }
  const int threads = 256;
  const int64_t work = (rows * nbc + 1) / 2;  // two blocks per thread and pass
  const auto* xs = static_cast<const uint16_t*>(x);
  if (gsf != nullptr)
    quant_tiled_kernel<kStaticBf16>
        <<<wave_grid<quant_tiled_kernel<kStaticBf16>>(work, threads), threads, 0, stream>>>(
            xs, rows, nbc, ld_x, gsf, codes, scales);
  else
    quant_tiled_kernel<kUnitBf16>
        <<<wave_grid<quant_tiled_kernel<kUnitBf16>>(work, threads), threads, 0, stream>>>(
            xs, rows, nbc, ld_x, gsf, codes, scales);
  return cudaGetLastError();
}

size_t attn_fp4_scale_bytes(int B, int N, int H, int D) {
  const size_t n_tiles = (static_cast<size_t>(N) + 127) / 128;
  return static_cast<size_t>(B) * H * n_tiles * (D / 64) * 512;
}

cudaError_t launch_quant_attn_fp4(const void* x, int B, int N, int H, int D, uint8_t* codes,
                                  uint8_t* scales, cudaStream_t stream) {
  const int64_t nblocks = static_cast<int64_t>(B) * N * H * (D / 16);
  const int64_t n_tiles = (N + 127) / 128;
  const int64_t npad = static_cast<int64_t>(B) * H * (n_tiles * 128 - N) * (D / 16);
  if ((D != 64 && D != 128) || nblocks >= (int64_t{1} << 31) || npad >= (int64_t{1} << 31))
    return cudaErrorInvalidValue;
  const int threads = 256;
  const int64_t work = std::max<int64_t>((nblocks + 1) / 2, npad);
  quant_attn_fp4_kernel<<<wave_grid<quant_attn_fp4_kernel>(work, threads), threads, 0, stream>>>(
      static_cast<const uint16_t*>(x), static_cast<uint32_t>(nblocks), static_cast<uint32_t>(npad),
      static_cast<uint32_t>(N), static_cast<uint32_t>(H), D == 128 ? 3u : 2u,
      static_cast<uint32_t>(n_tiles), codes, scales);
  return cudaGetLastError();
}

cudaError_t launch_quant_attn_ops(const AttnOpSpec* specs, int count, int B, int H, int D,
                                  cudaStream_t stream) {
  if ((D != 64 && D != 128) || count < 1 || count > 3) return cudaErrorInvalidValue;
  AttnOpJobs jobs{};
  jobs.H = static_cast<uint32_t>(H);
  jobs.lg_nbd = D == 128 ? 3u : 2u;
  int64_t total = 0, ptot = 0;
  for (int i = 0; i < count; ++i) {
    const AttnOpSpec& sp = specs[i];
    AttnOpJob& jb = jobs.j[i];
    const int64_t nb = static_cast<int64_t>(B) * sp.N * H * (D / 16);
    const int64_t nt = (sp.N + 127) / 128;
    jb.x = static_cast<const uint16_t*>(sp.x);
    jb.codes = sp.codes;
    jb.scales = sp.scales;
    jb.bf16 = static_cast<uint16_t*>(sp.bf16);
    jb.f16 = static_cast<uint16_t*>(sp.f16);
    jb.nblocks = static_cast<uint32_t>(nb);
    jb.N = static_cast<uint32_t>(sp.N);
    jb.n_tiles = static_cast<uint32_t>(nt);
    const int64_t np = sp.scales != nullptr ? static_cast<int64_t>(B) * H * (nt * 128 - sp.N) * (D / 16) : 0;
    jb.npad = static_cast<uint32_t>(np);
    total += nb;
    ptot += np;
  }
  if (total >= (int64_t{1} << 31) || ptot >= (int64_t{1} << 31)) return cudaErrorInvalidValue;
  const int threads = 256;
  const int64_t work = std::max<int64_t>((total + 1) / 2, ptot);
  quant_attn_ops_kernel<<<wave_grid<quant_attn_ops_kernel>(work, threads), threads, 0, stream>>>(jobs);
  return cudaGetLastError();
}

cudaError_t launch_global_sf(const void* x, int64_t rows, int64_t cols, int64_t ld_x, float* gsf,
                             cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(gsf, 0, sizeof(float), stream);
  if (e != cudaSuccess) return e;
  const int threads = 256;
  if (ld_x == cols && cols % 8 == 0) {
    const int64_t nvec = rows * cols / 8;
    amax_flat_kernel<<<wave_grid<amax_flat_kernel>((nvec + 3) / 4, threads), threads, 0, stream>>>(
        static_cast<const uint4*>(x), nvec, reinterpret_cast<unsigned int*>(gsf));
  } else {
    const int grid = grid_for(rows * (cols / 8 > 0 ? cols / 8 : 1), threads);
    amax_kernel<<<grid, threads, 0, stream>>>(static_cast<const uint16_t*>(x), rows, cols, ld_x,
                                              reinterpret_cast<unsigned int*>(gsf));
  }
  global_sf_finalize_kernel<<<1, 1, 0, stream>>>(gsf);
  return cudaGetLastError();
}

}  // namespace nvq
