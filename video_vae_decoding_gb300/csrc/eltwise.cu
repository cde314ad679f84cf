// Memory-bound kernels of the decode: RMS norm (+SiLU), frame copies,
// post_quant_conv, attention softmax and V transpose, and weight packing.
// All activations are channels-last bf16; every access is a 16-byte vector of
// 8 channels where the layout allows.  Frame views may address circular
// causal-cache rings (FrameView::fmod).
#include "kernels.h"
#include "ptx.cuh"

namespace wan {

namespace {

__device__ __forceinline__ const __nv_bfloat16* at(const FrameView& v, int b, int f, long long p) {
  return static_cast<const __nv_bfloat16*>(v.base) + b * v.bs + (long long)ring_slot(v.f0 + f, v.fmod) * v.fs +
         p * v.ldc;
}
__device__ __forceinline__ __nv_bfloat16* at_mut(const FrameView& v, int b, int f, long long p) {
  return static_cast<__nv_bfloat16*>(v.base) + b * v.bs + (long long)ring_slot(v.f0 + f, v.fmod) * v.fs + p * v.ldc;
}

inline unsigned blocks_for(long long n, int per_block) { return (unsigned)((n + per_block - 1) / per_block); }

// RMS norm (+ SiLU) over channels.  Grid: (position blocks, frames,
// batch).  A warp normalises R x (32 / G) consecutive positions of one
// frame: G lanes per position (G = 16 for C <= 128, so that narrow widths do
// not leave most lanes idle), lane l of a group holding channels l*8 + j*256
// .. +7 (j < NCH).  All R*NCH 16-byte loads are issued before the first
// reduction, to keep enough bytes in flight.
constexpr int kNormMaxC = 1024;
// SiLU y * sigmoid(y) with sigmoid(y) = (1 + tanh(y / 2)) / 2: one SFU
// operation (tanh.approx, relative error near 2^-11) instead of an exponential
// and a reciprocal, for outputs rounded to bf16 (relative step 2^-8).
__device__ __forceinline__ float silu_tanh(float y) {
  const float h = 0.5f * y;
  float t;
  asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(h));
  return fmaf(h, t, h);
}

template <bool SILU, int R, int NCH, bool SPLIT, int G = 32>
__global__ void __launch_bounds__(256) rms_norm_kernel(FrameView in, FrameView out, const float* __restrict__ gs,
                                                       int C, int P, int in_lo, int out_lo) {
  constexpr int PW = 32 / G;  // positions side by side in a warp
  const int lane = threadIdx.x & (G - 1);
  const int pw0 = (blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32) * R * PW;
  if (pw0 >= P) return;  // warp-uniform
  // position r of this lane group: p0 + r * PW
  const int p0 = pw0 + (int)((threadIdx.x & 31) / G);
  const int f = blockIdx.y, b = blockIdx.z;
  const __nv_bfloat16* src = at(in, b, f, p0);
  __nv_bfloat16* dst0 = at_mut(out, b, f, p0);
  float x[R][NCH][8];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const bool ok = p0 + r * PW < P;
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
      const int c = lane * 8 + j * 256;
      uint4 a4 = make_uint4(0, 0, 0, 0), b4 = make_uint4(0, 0, 0, 0);
      if (ok && c < C) {
        a4 = __ldg(reinterpret_cast<const uint4*>(src + (long long)r * PW * in.ldc + c));
        if (SPLIT) b4 = __ldg(reinterpret_cast<const uint4*>(src + (long long)r * PW * in.ldc + in_lo + c));
      }
      const uint32_t w[4] = {a4.x, a4.y, a4.z, a4.w}, u[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {  // split format: value = hi + lo
        x[r][j][2 * i] = SPLIT ? bf16_lo(w[i]) + bf16_lo(u[i]) : bf16_lo(w[i]);
        x[r][j][2 * i + 1] = SPLIT ? bf16_hi(w[i]) + bf16_hi(u[i]) : bf16_hi(w[i]);
      }
    }
  }
  float rinv[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < NCH; ++j)
#pragma unroll
      for (int i = 0; i < 8; ++i) ss = fmaf(x[r][j][i], x[r][j][i], ss);
    rinv[r] = ss;
  }
#pragma unroll
  for (int o = G / 2; o > 0; o >>= 1)  // within the lane group
#pragma unroll
    for (int r = 0; r < R; ++r) rinv[r] += __shfl_xor_sync(0xffffffffu, rinv[r], o);
#pragma unroll
  for (int r = 0; r < R; ++r) rinv[r] = 1.0f / fmaxf(sqrtf(rinv[r]), 1e-12f);
#pragma unroll
  for (int j = 0; j < NCH; ++j) {
    const int c = lane * 8 + j * 256;
    if (c >= C) continue;
    const float4 g0 = __ldg(reinterpret_cast<const float4*>(gs + c));
    const float4 g1 = __ldg(reinterpret_cast<const float4*>(gs + c + 4));
    const float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
#pragma unroll
    for (int r = 0; r < R; ++r) {
      if (p0 + r * PW >= P) continue;
      __nv_bfloat16* dst = dst0 + (long long)r * PW * out.ldc;
      float y[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        y[i] = x[r][j][i] * (rinv[r] * g[i]);
        // SiLU: y * sigmoid(y).  The split (fp32) format keeps the exponential
        // form (for y << 0 the exponential overflows to +inf and the
        // approximate division returns -0); bf16 outputs take the tanh form.
        if (SILU) y[i] = SPLIT ? __fdividef(y[i], 1.0f + __expf(-y[i])) : silu_tanh(y[i]);
      }
      if (SPLIT) {
        float h[8], l[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          h[i] = __bfloat162float(__float2bfloat16_rn(y[i]));
          l[i] = y[i] - h[i];
        }
        *reinterpret_cast<uint4*>(dst + c) = make_uint4(pack_bf16x2(h[0], h[1]), pack_bf16x2(h[2], h[3]),
                                                        pack_bf16x2(h[4], h[5]), pack_bf16x2(h[6], h[7]));
        *reinterpret_cast<uint4*>(dst + out_lo + c) = make_uint4(pack_bf16x2(l[0], l[1]), pack_bf16x2(l[2], l[3]),
                                                                 pack_bf16x2(l[4], l[5]), pack_bf16x2(l[6], l[7]));
      } else {
        *reinterpret_cast<uint4*>(dst + c) = make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]),
                                                        pack_bf16x2(y[4], y[5]), pack_bf16x2(y[6], y[7]));
      }
    }
  }
}

__global__ void copy_frames_kernel(FrameView in, FrameView out, int C8, int F, int P, long long n) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const int c = (int)(i % C8) * 8;
  long long r = i / C8;
  const long long p = r % P;
  r /= P;
  const int f = (int)(r % F);
  const int b = (int)(r / F);
  *reinterpret_cast<uint4*>(at_mut(out, b, f, p) + c) = *reinterpret_cast<const uint4*>(at(in, b, f, p) + c);
}

// post_quant_conv (1x1x1, kZ -> kZ; kZ = 48 for TI2V-5B, 16 for Wan2.1) on
// NCDHW latents; one thread per position.  With zstat (mean[kZ] then
// std[kZ]) each latent is first de-normalised, z * std[c] + mean[c], in fp32.
template <int kZ>
__global__ void post_quant_kernel(const void* __restrict__ z, int z_f32, int Tz, int t0, int F, int P,
                                  const float* __restrict__ w, const float* __restrict__ bias,
                                  const float* __restrict__ zstat, FrameView out, long long n, int round_z,
                                  int out_lo) {
  __shared__ float sw[kZ * kZ];
  __shared__ float sb[kZ];
  __shared__ float sst[2 * kZ];
  for (int i = threadIdx.x; i < kZ * kZ; i += blockDim.x) sw[i] = w[i];
  for (int i = threadIdx.x; i < kZ; i += blockDim.x) sb[i] = bias[i];
  for (int i = threadIdx.x; i < 2 * kZ; i += blockDim.x) sst[i] = zstat ? zstat[i] : (i < kZ ? 0.f : 1.f);
  __syncthreads();
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const long long p = i % P;
  const int f = (int)((i / P) % F);
  const int b = (int)(i / ((long long)P * F));
  float zin[kZ];
  const long long base = ((long long)b * kZ * Tz + (t0 + f)) * P + p;  // z[b][c][t][p]
#pragma unroll
  for (int c = 0; c < kZ; ++c) {
    const long long o = base + (long long)c * Tz * P;
    zin[c] = z_f32 ? static_cast<const float*>(z)[o]
                   : __bfloat162float(static_cast<const __nv_bfloat16*>(z)[o]);
    if (zstat) zin[c] = fmaf(zin[c], sst[kZ + c], sst[c]);
    if (round_z) zin[c] = __bfloat162float(__float2bfloat16_rn(zin[c]));
  }
  __nv_bfloat16* dst = at_mut(out, b, f, p);
  for (int co = 0; co < kZ; co += 8) {
    float acc[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      float s = sb[co + k];
#pragma unroll
      for (int c = 0; c < kZ; ++c) s = fmaf(sw[(co + k) * kZ + c], zin[c], s);
      acc[k] = s;
    }
    float h[8], l[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      h[k] = out_lo ? __bfloat162float(__float2bfloat16_rn(acc[k])) : acc[k];
      l[k] = acc[k] - h[k];
    }
    *reinterpret_cast<uint4*>(dst + co) = make_uint4(pack_bf16x2(h[0], h[1]), pack_bf16x2(h[2], h[3]),
                                                     pack_bf16x2(h[4], h[5]), pack_bf16x2(h[6], h[7]));
    if (out_lo)
      *reinterpret_cast<uint4*>(dst + out_lo + co) = make_uint4(pack_bf16x2(l[0], l[1]), pack_bf16x2(l[2], l[3]),
                                                                pack_bf16x2(l[4], l[5]), pack_bf16x2(l[6], l[7]));
  }
}

// Rows of up to 4096 scores: one 256-thread block per row, each thread
// holding up to four float4 chunks of the row in registers, so the scores
// are read once and exponentiated once.
constexpr int kSoftmaxRegCols = 4096;
__device__ __forceinline__ float block_reduce(float v, float* red, bool is_max) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float u = __shfl_xor_sync(0xffffffffu, v, o);
    v = is_max ? fmaxf(v, u) : v + u;
  }
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x < 32) {
    float w = threadIdx.x < blockDim.x / 32 ? red[threadIdx.x] : (is_max ? -INFINITY : 0.f);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float u = __shfl_xor_sync(0xffffffffu, w, o);
      w = is_max ? fmaxf(w, u) : w + u;
    }
    if (threadIdx.x == 0) red[0] = w;
  }
  __syncthreads();
  const float r = red[0];
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(256) softmax_rows_reg_kernel(const float* __restrict__ S, long long ld_s,
                                                               __nv_bfloat16* __restrict__ Pm, long long ld_p, int n,
                                                               float scale, int p_lo) {
  const float4* s4 = reinterpret_cast<const float4*>(S + (long long)blockIdx.x * ld_s);
  __nv_bfloat16* p = Pm + (long long)blockIdx.x * ld_p;
  __shared__ float red[32];
  float v[4][4];
  float mx = -INFINITY;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int j = 4 * (threadIdx.x + 256 * k);
    float4 a = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    if (j < n) a = __ldcs(s4 + threadIdx.x + 256 * k);
    v[k][0] = j < n ? a.x : -INFINITY;
    v[k][1] = j + 1 < n ? a.y : -INFINITY;
    v[k][2] = j + 2 < n ? a.z : -INFINITY;
    v[k][3] = j + 3 < n ? a.w : -INFINITY;
#pragma unroll
    for (int i = 0; i < 4; ++i) mx = fmaxf(mx, v[k][i]);
  }
  mx = block_reduce(mx, red, true);
  float sum = 0.f;
#pragma unroll
  for (int k = 0; k < 4; ++k)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[k][i] = expf((v[k][i] - mx) * scale);  // exp(-inf) = 0 past the row
      sum += v[k][i];
    }
  const float inv = 1.0f / block_reduce(sum, red, false);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int j = 4 * (threadIdx.x + 256 * k);
    if (j >= n) continue;
    float h[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = v[k][i] * inv;
    if (j + 3 < n) {
      *reinterpret_cast<uint2*>(p + j) = make_uint2(pack_bf16x2(h[0], h[1]), pack_bf16x2(h[2], h[3]));
      if (p_lo) {
        float l[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) l[i] = h[i] - __bfloat162float(__float2bfloat16_rn(h[i]));
        *reinterpret_cast<uint2*>(p + p_lo + j) = make_uint2(pack_bf16x2(l[0], l[1]), pack_bf16x2(l[2], l[3]));
      }
    } else {
      for (int i = 0; i < 4 && j + i < n; ++i) {
        const __nv_bfloat16 b = __float2bfloat16_rn(h[i]);
        p[j + i] = b;
        if (p_lo) p[p_lo + j + i] = __float2bfloat16_rn(h[i] - __bfloat162float(b));
      }
    }
  }
}

// Longer rows: one 256-thread block per row, three passes over the scores.
__global__ void softmax_rows_kernel(const float* __restrict__ S, long long ld_s, __nv_bfloat16* __restrict__ Pm,
                                    long long ld_p, int n, float scale, int p_lo) {
  const float* s = S + (long long)blockIdx.x * ld_s;
  __nv_bfloat16* p = Pm + (long long)blockIdx.x * ld_p;
  __shared__ float red[32];
  float mx = -INFINITY;
  for (int j = threadIdx.x; j < n; j += blockDim.x) mx = fmaxf(mx, s[j]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = threadIdx.x < blockDim.x / 32 ? red[threadIdx.x] : -INFINITY;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (threadIdx.x == 0) red[0] = v;
  }
  __syncthreads();
  mx = red[0];
  __syncthreads();
  float sum = 0.f;
  for (int j = threadIdx.x; j < n; j += blockDim.x) sum += expf((s[j] - mx) * scale);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = sum;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = threadIdx.x < blockDim.x / 32 ? red[threadIdx.x] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (threadIdx.x == 0) red[0] = v;
  }
  __syncthreads();
  const float inv = 1.0f / red[0];
  for (int j = threadIdx.x; j < n; j += blockDim.x) {
    const float v = expf((s[j] - mx) * scale) * inv;
    const __nv_bfloat16 h = __float2bfloat16_rn(v);
    p[j] = h;
    if (p_lo) p[p_lo + j] = __float2bfloat16_rn(v - __bfloat162float(h));
  }
}

// 64 x 64 tiles through shared memory, 16-byte global accesses: a thread
// loads 8 channels of one position and stores 8 positions of one channel
// (eight threads cover one 128-byte row of the output).  Shared memory holds
// a row per position in 16-byte chunks, chunk q of row r at q ^ ((r / 8) % 8),
// so the eight rows a warp reads together for one channel sit in distinct
// banks.
__global__ void __launch_bounds__(256) transpose_kernel(const __nv_bfloat16* __restrict__ src, long long src_gs,
                                                        int ld_src, __nv_bfloat16* __restrict__ dst, long long dst_gs,
                                                        int ld_dst, int P, int C) {
  __shared__ __align__(16) __nv_bfloat16 tile[64][64];
  const int g = blockIdx.z;
  const int p0 = blockIdx.x * 64, c0 = blockIdx.y * 64;
  const __nv_bfloat16* s = src + g * src_gs;
  __nv_bfloat16* d = dst + g * dst_gs;
  const bool vec = (ld_src % 8 == 0) && (ld_dst % 8 == 0) && (c0 + 64 <= C) && (p0 + 64 <= P);
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int i = threadIdx.x + 256 * k;  // 512 chunks: 64 positions x 8 channel chunks
    const int r = i >> 3, q = i & 7;
    __nv_bfloat16* t = &tile[r][8 * (q ^ ((r >> 3) & 7))];
    const int p = p0 + r;
    if (vec) {
      *reinterpret_cast<uint4*>(t) = __ldg(reinterpret_cast<const uint4*>(s + (long long)p * ld_src + c0 + 8 * q));
    } else {
      for (int e = 0; e < 8; ++e) {
        const int c = c0 + 8 * q + e;
        t[e] = (p < P && c < C) ? s[(long long)p * ld_src + c] : __float2bfloat16_rn(0.f);
      }
    }
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int i = threadIdx.x + 256 * k;  // 512 chunks: 64 channels x 8 position chunks
    const int c = i >> 3, pk = i & 7;     // channel, position chunk (rows 8 pk .. 8 pk + 7)
    const int col = 8 * ((c >> 3) ^ pk) + (c & 7);
    __nv_bfloat16 v[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = tile[8 * pk + e][col];
    __nv_bfloat16* o = d + (long long)(c0 + c) * ld_dst + p0 + 8 * pk;
    if (vec) {
      uint32_t w[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        __nv_bfloat162 pr = __halves2bfloat162(v[2 * j], v[2 * j + 1]);
        w[j] = *reinterpret_cast<uint32_t*>(&pr);
      }
      *reinterpret_cast<uint4*>(o) = make_uint4(w[0], w[1], w[2], w[3]);
    } else if (c0 + c < C) {
      for (int e = 0; e < 8; ++e)
        if (p0 + 8 * pk + e < P) o[e] = v[e];
    }
  }
}

__global__ void pack_weight_kernel(const void* __restrict__ src, int src_f32, int Co, int Ci, int taps,
                                   __nv_bfloat16* __restrict__ dst, int ld, int k0, int ci_pad, long long n, int lo) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const int tap = (int)(i % taps);
  const int ci = (int)((i / taps) % Ci);
  const int co = (int)(i / ((long long)taps * Ci));
  const float v = src_f32 ? static_cast<const float*>(src)[i] : __bfloat162float(static_cast<const __nv_bfloat16*>(src)[i]);
  const __nv_bfloat16 h = __float2bfloat16_rn(v);
  dst[(long long)co * ld + k0 + (long long)tap * ci_pad + ci] = lo ? __float2bfloat16_rn(v - __bfloat162float(h)) : h;
}

__device__ __forceinline__ float load_any(const void* p, int f32, int i, int rnd) {
  const float v = f32 ? static_cast<const float*>(p)[i] : __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
  return rnd ? __bfloat162float(__float2bfloat16_rn(v)) : v;
}

// rows dy of a 3-row kernel that land on source offset a for output phase i
__device__ __forceinline__ bool subpix_tap(int i, int a, int d) {
  return i == 0 ? (a == 0 ? d == 0 : d >= 1) : (a == 0 ? d <= 1 : d == 2);
}

__global__ void pack_subpixel_kernel(const void* __restrict__ src, int src_f32, int Co, int Ci,
                                     __nv_bfloat16* __restrict__ dst, int ld, int co_pad, int k0, int tap_stride,
                                     int round_src, int lo, long long n) {
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= n) return;  // n = 4 phases * Co * Ci * 4 taps
  const int ab = (int)(idx % 4);
  const int ci = (int)((idx / 4) % Ci);
  const int co = (int)((idx / (4LL * Ci)) % Co);
  const int p = (int)(idx / (4LL * Ci * Co));
  const int i = p >> 1, j = p & 1, a = ab >> 1, b = ab & 1;
  float v = 0.f;
  for (int dy = 0; dy < 3; ++dy) {
    if (!subpix_tap(i, a, dy)) continue;
    for (int dx = 0; dx < 3; ++dx) {
      if (!subpix_tap(j, b, dx)) continue;
      const long long o = (((long long)co * Ci + ci) * 3 + dy) * 3 + dx;
      float w = src_f32 ? static_cast<const float*>(src)[o] : __bfloat162float(static_cast<const __nv_bfloat16*>(src)[o]);
      if (round_src) w = __bfloat162float(__float2bfloat16_rn(w));
      v += w;
    }
  }
  const __nv_bfloat16 h = __float2bfloat16_rn(v);
  dst[((long long)p * co_pad + co) * ld + k0 + (long long)ab * tap_stride + ci] =
      lo ? __float2bfloat16_rn(v - __bfloat162float(h)) : h;
}

__global__ void to_f32_kernel(const void* __restrict__ src, int src_f32, const void* __restrict__ src2, int src2_f32,
                              float* __restrict__ dst, int n, float scale, int rnd) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  float v = load_any(src, src_f32, i, rnd) * scale;
  if (src2) v += load_any(src2, src2_f32, i, rnd);
  dst[i] = v;
}

}  // namespace

template <bool SILU, bool SPLIT>
static void norm_dispatch(FrameView in, FrameView out, const float* gs, int C, int B, int F, int P, int in_lo,
                          int out_lo, cudaStream_t s) {
  // 8 warps per block, R x 32 / G positions per warp
  if (C <= 128)
    rms_norm_kernel<SILU, 4, 1, SPLIT, 16><<<dim3(blocks_for(P, 64), F, B), 256, 0, s>>>(in, out, gs, C, P, in_lo,
                                                                                         out_lo);
  else if (C <= 256)
    rms_norm_kernel<SILU, 4, 1, SPLIT><<<dim3(blocks_for(P, 32), F, B), 256, 0, s>>>(in, out, gs, C, P, in_lo, out_lo);
  else if (C <= 512)
    rms_norm_kernel<SILU, 2, 2, SPLIT><<<dim3(blocks_for(P, 16), F, B), 256, 0, s>>>(in, out, gs, C, P, in_lo, out_lo);
  else
    rms_norm_kernel<SILU, 1, 4, SPLIT><<<dim3(blocks_for(P, 8), F, B), 256, 0, s>>>(in, out, gs, C, P, in_lo, out_lo);
}

cudaError_t launch_rms_norm(FrameView in, FrameView out, const float* gs, int C, int B, int F, int P, bool silu,
                            cudaStream_t s, int in_lo, int out_lo) {
  if (C > kNormMaxC || C % 8 || F > 65535 || B > 65535) return cudaErrorInvalidValue;
  if ((long long)B * F * P == 0) return cudaSuccess;
  if ((in_lo != 0) != (out_lo != 0)) return cudaErrorInvalidValue;  // both split or both plain
  if (silu) {
    if (in_lo)
      norm_dispatch<true, true>(in, out, gs, C, B, F, P, in_lo, out_lo, s);
    else
      norm_dispatch<true, false>(in, out, gs, C, B, F, P, in_lo, out_lo, s);
  } else {
    if (in_lo)
      norm_dispatch<false, true>(in, out, gs, C, B, F, P, in_lo, out_lo, s);
    else
      norm_dispatch<false, false>(in, out, gs, C, B, F, P, in_lo, out_lo, s);
  }
  return cudaGetLastError();
}

cudaError_t launch_copy_frames(FrameView in, FrameView out, int C, int B, int F, int P, cudaStream_t s) {
  if (C % 8) return cudaErrorInvalidValue;
  const long long n = (long long)B * F * P * (C / 8);
  if (n == 0) return cudaSuccess;
  copy_frames_kernel<<<blocks_for(n, 256), 256, 0, s>>>(in, out, C / 8, F, P, n);
  return cudaGetLastError();
}

cudaError_t launch_post_quant(const void* z, int z_f32, int Z, int B, int Tz, int t0, int F, int P, const float* w,
                              const float* bias, const float* zstat, FrameView out, int round_z_bf16, cudaStream_t s,
                              int out_lo) {
  if (out.ldc % 8 || out.ldc < Z || (Z != 48 && Z != 16)) return cudaErrorInvalidValue;
  const long long n = (long long)B * F * P;
  if (n == 0) return cudaSuccess;
  if (Z == 48)
    post_quant_kernel<48><<<blocks_for(n, 128), 128, 0, s>>>(z, z_f32, Tz, t0, F, P, w, bias, zstat, out, n,
                                                             round_z_bf16, out_lo);
  else
    post_quant_kernel<16><<<blocks_for(n, 128), 128, 0, s>>>(z, z_f32, Tz, t0, F, P, w, bias, zstat, out, n,
                                                             round_z_bf16, out_lo);
  return cudaGetLastError();
}

cudaError_t launch_softmax_rows(const float* S, long long ld_s, __nv_bfloat16* P, long long ld_p, int n, long long R,
                                float scale, cudaStream_t s, int p_lo) {
  if (R == 0) return cudaSuccess;
  if (R > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  // the register version needs 16-byte aligned rows and even row starts in P
  const bool reg = n <= kSoftmaxRegCols && ld_s % 4 == 0 && ld_p % 4 == 0 && p_lo % 4 == 0 &&
                   reinterpret_cast<uintptr_t>(S) % 16 == 0 && reinterpret_cast<uintptr_t>(P) % 8 == 0;
  if (reg)
    softmax_rows_reg_kernel<<<(unsigned)R, 256, 0, s>>>(S, ld_s, P, ld_p, n, scale, p_lo);
  else
    softmax_rows_kernel<<<(unsigned)R, 256, 0, s>>>(S, ld_s, P, ld_p, n, scale, p_lo);
  return cudaGetLastError();
}

cudaError_t launch_transpose(const __nv_bfloat16* src, long long src_gs, int ld_src, __nv_bfloat16* dst,
                             long long dst_gs, int ld_dst, int G, int P, int C, cudaStream_t s) {
  if (G == 0 || P == 0 || C == 0) return cudaSuccess;
  if (reinterpret_cast<uintptr_t>(src) % 16 || reinterpret_cast<uintptr_t>(dst) % 16 || src_gs % 8 || dst_gs % 8)
    return cudaErrorInvalidValue;
  dim3 grid((P + 63) / 64, (C + 63) / 64, G);
  transpose_kernel<<<grid, 256, 0, s>>>(src, src_gs, ld_src, dst, dst_gs, ld_dst, P, C);
  return cudaGetLastError();
}

cudaError_t launch_pack_weight(const void* src, int src_f32, int Co, int Ci, int taps, __nv_bfloat16* dst, int ld,
                               int k0, int ci_pad, cudaStream_t s, int lo) {
  const long long n = (long long)Co * Ci * taps;
  if (n == 0) return cudaSuccess;
  pack_weight_kernel<<<blocks_for(n, 256), 256, 0, s>>>(src, src_f32, Co, Ci, taps, dst, ld, k0, ci_pad, n, lo);
  return cudaGetLastError();
}

cudaError_t launch_pack_subpixel(const void* src, int src_f32, int Co, int Ci, __nv_bfloat16* dst, int ld, int co_pad,
                                 int k0, int tap_stride, int round_src, int lo, cudaStream_t s) {
  const long long n = 16LL * Co * Ci;
  if (n == 0) return cudaSuccess;
  pack_subpixel_kernel<<<blocks_for(n, 256), 256, 0, s>>>(src, src_f32, Co, Ci, dst, ld, co_pad, k0, tap_stride,
                                                          round_src, lo, n);
  return cudaGetLastError();
}

cudaError_t launch_to_f32(const void* src, int src_f32, const void* src2, int src2_f32, float* dst, int n,
                          float scale, int round_bf16, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  to_f32_kernel<<<blocks_for(n, 256), 256, 0, s>>>(src, src_f32, src2, src2_f32, dst, n, scale, round_bf16);
  return cudaGetLastError();
}

}  // namespace wan
