// Tiled decode support kernels: latent tile gather, seam blending and
// assembly of the blended tiles into the video.
//
// Tiling (the diffusers pull request "[Feature] Implement tiled VAE
// encoding/decoding for Wan model. #11414"): tiles start at multiples of
// the stride and hold min(tile, remaining) pixels.  Each tile is decoded on
// its own; in raster order a tile cross-fades its top rows with the tile
// above and then its left columns with the tile to its left, over the pixels
// the two share; tile (i, j) then supplies the pixels from its origin up to
// the next tile's origin.
//
// Decoded tiles are fp32 [B][3][F][h][w] each, at TileDesc::off in one
// buffer.  All three kernels are memory-bound copies or 3-point blends.
#include <algorithm>

#include "kernels.h"

namespace wan {

namespace {

inline unsigned blocks_for(long long n, int per_block) { return (unsigned)((n + per_block - 1) / per_block); }

// z [B][48][T][h][w] -> zt [(k*B + b)][48][T][th][tw] for the tiles k of
// one batch, whose latent origins are g.r0[k], g.c0[k].
template <typename E>
__global__ void gather_tiles_kernel(const E* __restrict__ z, E* __restrict__ zt, const __grid_constant__ TileGather g,
                                    long long n) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const int x = (int)(i % g.tw);
    long long r = i / g.tw;
    const int y = (int)(r % g.th);
    r /= g.th;
    const long long ct = r % g.CT;  // channel * T + frame
    r /= g.CT;
    const int b = (int)(r % g.B);
    const int k = (int)(r / g.B);
    const long long src = (((long long)b * g.CT + ct) * g.h + g.r0[k] + y) * g.w + g.c0[k] + x;
    zt[i] = z[src];
  }
}

// Blends the tiles (i, d - i) of anti-diagonal d in place.  Every tile they
// read (the one above, the one to the left) lies on diagonal d - 1 and is
// final; a pixel's vertical and then horizontal blend read only its own
// value besides those, so the pixels of a tile are independent.
__global__ void blend_tiles_kernel(float* __restrict__ buf, const __grid_constant__ TileTable tab, int d, int i_lo,
                                   long long planes) {
  const int i = i_lo + blockIdx.y, j = d - i;
  const TileDesc b = tab.t[i * tab.nj + j];
  const int ev = i > 0 ? min(tab.t[(i - 1) * tab.nj + j].h - tab.sh, b.h) : 0;
  const int eh = j > 0 ? min(tab.t[i * tab.nj + j - 1].w - tab.sw, b.w) : 0;
  const long long nb = (long long)ev * b.w + (long long)(b.h - ev) * eh;  // band pixels per plane
  if (nb <= 0) return;
  const TileDesc up = i > 0 ? tab.t[(i - 1) * tab.nj + j] : b;
  const TileDesc lf = j > 0 ? tab.t[i * tab.nj + j - 1] : b;
  const long long n = planes * nb;
  for (long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x; t < n; t += (long long)gridDim.x * blockDim.x) {
    const long long pl = t / nb;
    const long long r = t - pl * nb;
    int y, x;
    if (r < (long long)ev * b.w) {
      y = (int)(r / b.w);
      x = (int)(r - (long long)y * b.w);
    } else {
      const long long r2 = r - (long long)ev * b.w;
      y = ev + (int)(r2 / eh);
      x = (int)(r2 - (long long)(y - ev) * eh);
    }
    float* p = buf + b.off + pl * b.h * b.w + (long long)y * b.w + x;
    float v = *p;
    if (y < ev) {
      const float a = buf[up.off + pl * up.h * up.w + (long long)(y + tab.sh) * up.w + x];
      v = a * ((float)(ev - y) / (float)ev) + v * ((float)y / (float)ev);
    }
    if (x < eh) {
      const float a = buf[lf.off + pl * lf.h * lf.w + (long long)y * lf.w + x + tab.sw];
      v = a * ((float)(eh - x) / (float)eh) + v * ((float)x / (float)eh);
    }
    *p = v;
  }
}

// out [planes][H][W] <- the region of each tile from its origin up to the
// next origin; four pixels per thread (tile edges are multiples of 16).
template <bool F32>
__global__ void assemble_tiles_kernel(const float* __restrict__ buf, void* __restrict__ out,
                                      const __grid_constant__ TileTable tab, int H, int W, long long n4) {
  const int W4 = W / 4;
  for (long long q = (long long)blockIdx.x * blockDim.x + threadIdx.x; q < n4; q += (long long)gridDim.x * blockDim.x) {
    const int X = (int)(q % W4) * 4;
    const long long r = q / W4;
    const int Y = (int)(r % H);
    const long long pl = r / H;
    const int i = min(Y / tab.sh, tab.ni - 1), j = min(X / tab.sw, tab.nj - 1);
    const TileDesc t = tab.t[i * tab.nj + j];
    const float4 v = *reinterpret_cast<const float4*>(buf + t.off + pl * t.h * t.w +
                                                      (long long)(Y - i * tab.sh) * t.w + (X - j * tab.sw));
    const long long o = r * W + X;
    if (F32) {
      *reinterpret_cast<float4*>(static_cast<float*>(out) + o) = v;
    } else {
      uint2 u;
      __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
      u.x = *reinterpret_cast<uint32_t*>(&lo);
      u.y = *reinterpret_cast<uint32_t*>(&hi);
      *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(out) + o) = u;
    }
  }
}

constexpr int kThreads = 256;
constexpr unsigned kMaxBlocks = 152 * 16;  // grid-stride loops beyond 16 blocks per SM

}  // namespace

cudaError_t launch_gather_tiles(const void* z, int elem_bytes, void* zt, const TileGather& g, cudaStream_t s) {
  if (g.n < 1 || g.n > kMaxGather || (elem_bytes != 2 && elem_bytes != 4)) return cudaErrorInvalidValue;
  const long long n = (long long)g.n * g.B * g.CT * g.th * g.tw;
  if (n == 0) return cudaSuccess;
  const unsigned grid = (unsigned)std::min<long long>(blocks_for(n, kThreads), kMaxBlocks);
  if (elem_bytes == 4)
    gather_tiles_kernel<float><<<grid, kThreads, 0, s>>>(static_cast<const float*>(z), static_cast<float*>(zt), g, n);
  else
    gather_tiles_kernel<uint16_t>
        <<<grid, kThreads, 0, s>>>(static_cast<const uint16_t*>(z), static_cast<uint16_t*>(zt), g, n);
  return cudaGetLastError();
}

cudaError_t launch_blend_tiles(float* buf, const TileTable& tab, long long planes, cudaStream_t s) {
  if (tab.ni < 1 || tab.nj < 1 || tab.ni * tab.nj > kMaxTiles) return cudaErrorInvalidValue;
  // largest band of any tile, to size the grid
  long long band = 0;
  for (int i = 0; i < tab.ni; ++i)
    for (int j = 0; j < tab.nj; ++j) {
      const TileDesc& b = tab.t[i * tab.nj + j];
      const int ev = i > 0 ? std::min(tab.t[(i - 1) * tab.nj + j].h - tab.sh, b.h) : 0;
      const int eh = j > 0 ? std::min(tab.t[i * tab.nj + j - 1].w - tab.sw, b.w) : 0;
      band = std::max(band, (long long)ev * b.w + (long long)(b.h - ev) * eh);
    }
  if (band == 0) return cudaSuccess;  // stride == tile: nothing overlaps
  for (int d = 1; d <= tab.ni + tab.nj - 2; ++d) {
    const int i_lo = std::max(0, d - (tab.nj - 1)), i_hi = std::min(d, tab.ni - 1);
    const int nt = i_hi - i_lo + 1;
    const unsigned gx = (unsigned)std::max<long long>(1, std::min<long long>(blocks_for(planes * band, kThreads),
                                                                             kMaxBlocks / nt + 1));
    blend_tiles_kernel<<<dim3(gx, nt), kThreads, 0, s>>>(buf, tab, d, i_lo, planes);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_assemble_tiles(const float* buf, const TileTable& tab, void* out, int out_f32, long long planes,
                                  int H, int W, cudaStream_t s) {
  if (W % 4 || tab.sh < 1 || tab.sw % 4 || tab.ni * tab.nj > kMaxTiles) return cudaErrorInvalidValue;
  const long long n4 = planes * H * (W / 4);
  if (n4 == 0) return cudaSuccess;
  const unsigned grid = (unsigned)std::min<long long>(blocks_for(n4, kThreads), kMaxBlocks);
  if (out_f32)
    assemble_tiles_kernel<true><<<grid, kThreads, 0, s>>>(buf, out, tab, H, W, n4);
  else
    assemble_tiles_kernel<false><<<grid, kThreads, 0, s>>>(buf, out, tab, H, W, n4);
  return cudaGetLastError();
}

}  // namespace wan
