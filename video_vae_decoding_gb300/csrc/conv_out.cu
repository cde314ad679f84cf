// conv_out of the decoder (page "wan22_vae_decode/reference.py", section
// "What is computed", item 2: causal 3x3x3 conv to 3 colours x 2 x 2 patch
// channels; items 3-4: unpatchify and clamp) with the spatial taps folded
// into the GEMM's N dimension.
//
// With only 12 (or 3) output channels, the plain implicit GEMM would issue
// M=128 x N=16 MMAs whose A operand (4 KB of shared memory per MMA) costs
// far more than the arithmetic.  Here one GEMM computes, for every input
// position p of a 16 x 16 box and every spatial tap s = (dy, dx),
//
//     Y[p, (s, co)] = sum_{dt, ci} X[frame f + dt, p, ci] * W[co, ci, dt, dy, dx]
//
// (M = 256 positions as two M=128 accumulators, N = 9 * Cout rounded up to 16,
// K = 3 time taps x input channels), and the epilogue forms the convolution
// as a shifted sum over the nine taps,
//
//     out[q] = bias + sum_{dy, dx} Y[q + (dy - 1, dx - 1), (dy, dx)],
//
// for the 14 x 14 interior of the box (box origin = interior origin - 1;
// positions outside the frame read zero from the TMA, so their Y is zero,
// which is the conv's zero padding).  The dx sum runs in registers with warp
// shuffles (the three dx neighbours of a position are adjacent lanes of one
// image row), the dy sum through shared memory.  The result is unpatchified
// (channel 4k + 2j + i -> colour k, row 2y + i, column 2x + j) and clamped
// into the NCDHW video, with an optional fp32 copy before the clamp.
//
// Warp roles (384 threads): warp 0 lane 0 TMA producer (per time tap and
// 64-channel block one 16 x 16 x 64 A box and the 64-channel B block of all
// taps), warp 1 lane 0 MMA issuer, warp 2 TMEM allocation, warps 4-11 the
// epilogue (warp w reads TMEM lane quadrant w % 4 of accumulator (w - 4) / 4).
// The accumulators are double-buffered in TMEM; every wait is bounded.
#include "kernels.h"
#include "ptx.cuh"

namespace wan {

namespace {

constexpr int kVThreads = 384;
constexpr int kVEpiThreads = 256;
constexpr int kBox = 16;                    // box edge (positions)
constexpr int kInner = kBox - 2;            // interior edge: 14
constexpr int kVStages = 4;
constexpr int kVABytes = kBox * kBox * kBlockK * 2;  // 32 KB: 256 positions x 64 channels

template <int COUT>
struct VCfg {
  static constexpr int kTaps = 9 * COUT;                 // N columns used
  static constexpr int kN = (kTaps + 15) / 16 * 16;      // 112 or 32
  static constexpr int kAccCols = kN <= 32 ? 32 : (kN <= 64 ? 64 : 128);  // per M=128 accumulator
  static constexpr int kTmemCols = 2 * 2 * kAccCols;     // 2 accumulators x 2 buffers
  static constexpr int kBBytes = kN * kBlockK * 2;       // 14 KB or 4 KB
  static constexpr int kZS = 3 * COUT + 1;               // Z row stride (odd: no bank conflicts)
  static constexpr size_t kSmem = 1024 + (size_t)kVStages * (kVABytes + kBBytes) +
                                  (size_t)kBox * kBox * kZS * 4 + 8 * (2 * kVStages + 5) + 16;
};

struct VTile {
  int f, tx, ty, b;
};
// Unit order: frame, then x, y, batch (the output frames of one spatial box
// run side by side, so an input frame serves its three time taps from L2).
__device__ __forceinline__ VTile vtile(const VideoConvArgs& a, int u) {
  VTile t;
  t.f = u % a.frames;
  u /= a.frames;
  t.tx = u % a.tiles_x;
  u /= a.tiles_x;
  t.ty = u % a.tiles_y;
  t.b = u / a.tiles_y;
  return t;
}

template <int COUT, int VP>
__global__ void __launch_bounds__(kVThreads, 1)
    video_conv_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
                      const __grid_constant__ VideoConvArgs args) {
  using Cfg = VCfg<COUT>;
  constexpr int S = kVStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + S * kVABytes;
  float* zs = reinterpret_cast<float*>(sB + S * Cfg::kBBytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(zs + kBox * kBox * Cfg::kZS);
  uint64_t* empty = full + S;
  uint64_t* tfull = empty + S;   // [2] accumulators ready
  uint64_t* tempty = tfull + 2;  // [2] accumulators drained
  uint64_t* done = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const long long lim = args.wait_limit > 0 ? args.wait_limit : kWaitLimitCycles;
  const int units = args.frames * args.tiles_x * args.tiles_y * args.batches;
  const int kblocks = 3 * args.nkb;  // K blocks per tile: time taps x channel blocks

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&tfull[i]), 1);
      mbar_init(smem_u32(&tempty[i]), kVEpiThreads);
    }
    mbar_init(smem_u32(done), 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_map(&mapA);
    tma_prefetch_map(&mapB);
  }
  if (warp == 2) {
    tmem_alloc(smem_u32(tmem_slot), Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ producer
    int it = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
      const VTile t = vtile(args, u);
      const int x0 = t.tx * kInner - 1, y0 = t.ty * kInner - 1;
      for (int kk = 0; kk < kblocks; ++kk, ++it) {
        const int dt = kk / args.nkb, kb = kk - dt * args.nkb;
        const int s = it % S, r = it / S;
        if (r > 0 && !mbar_wait_bounded(smem_u32(&empty[s]), (r - 1) & 1, args.err, kDevTimeoutEmpty, lim)) {
          ok = false;
          *abort_flag = 1;
          break;
        }
        if (*abort_flag) {
          ok = false;
          break;
        }
        if (it + 1 == args.stall_at1) continue;  // injected failure: this stage never fills
        const uint32_t fb = smem_u32(&full[s]);
        mbar_arrive_expect_tx(fb, kVABytes + Cfg::kBBytes);
        tma_load_5d(smem_u32(sA + s * kVABytes), &mapA, fb, kb * kBlockK, x0, y0,
                    ring_slot(args.src_f0 + t.f + dt, args.src_fmod), t.b);
        tma_load_3d(smem_u32(sB + s * Cfg::kBBytes), &mapB, fb, dt * args.ci_pad + kb * kBlockK, 0, 0);
      }
    }
    // do not leave while copies into this CTA's shared memory are in flight
    for (int j = (it > S ? it - S : 0); j < it; ++j)
      mbar_wait_bounded(smem_u32(&full[j % S]), (j / S) & 1, args.err, kDevTimeoutFull, lim);
  } else if (warp == 1 && lane == 0) {
    // ---------------------------------------------------------- MMA issuer
    constexpr uint32_t idesc = idesc_bf16_f32(kTileM, Cfg::kN);
    int slot = 0, phase = 0, kbc = 0, lt = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x, ++lt) {
      const int buf = lt & 1, use = lt >> 1;
      if (use > 0 && !mbar_wait_bounded(smem_u32(&tempty[buf]), (use - 1) & 1, args.err, kDevTimeoutAccum, lim)) {
        *abort_flag = 1;
        break;
      }
      if (*abort_flag) break;
      tc_fence_after();
      const uint32_t d0 = tmem + buf * 2 * Cfg::kAccCols, d1 = d0 + Cfg::kAccCols;
      bool ok = true;
      for (int kk = 0; kk < kblocks; ++kk) {
        const int s = slot;
        if (!mbar_wait_bounded(smem_u32(&full[s]), phase, args.err, kDevTimeoutFull, lim)) {
          *abort_flag = 1;
          ok = false;
          break;
        }
        if (++slot == S) {
          slot = 0;
          phase ^= 1;
        }
        tc_fence_after();
        const uint64_t a0 = sdesc_k128(smem_u32(sA + s * kVABytes));
        const uint64_t a1 = a0 + (uint64_t)((kTileM * 128) >> 4);  // positions 128..255
        const uint64_t b0 = sdesc_k128(smem_u32(sB + s * Cfg::kBBytes));
        // a channel block that holds only tail_k16 x 16 channels (the rest is
        // TMA zero fill): issue just those K steps
        const bool tail = args.tail_k16 && kbc == args.nkb - 1;
        if (++kbc == args.nkb) kbc = 0;
        if (tail && args.tail_k16 == 2) {
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const uint32_t acc = (kk > 0 || k > 0) ? 1u : 0u;
            umma_bf16(d0, a0 + 2 * k, b0 + 2 * k, idesc, acc);
            umma_bf16(d1, a1 + 2 * k, b0 + 2 * k, idesc, acc);
          }
        } else {
#pragma unroll
          for (int k = 0; k < kBlockK / 16; ++k) {
            const uint32_t acc = (kk > 0 || k > 0) ? 1u : 0u;
            umma_bf16(d0, a0 + 2 * k, b0 + 2 * k, idesc, acc);
            umma_bf16(d1, a1 + 2 * k, b0 + 2 * k, idesc, acc);
          }
        }
        umma_commit(smem_u32(&empty[s]));
      }
      if (!ok) break;
      umma_commit(smem_u32(&tfull[buf]));
    }
    // every MMA of this CTA completes before the TMEM is released
    umma_commit(smem_u32(done));
    mbar_wait_bounded(smem_u32(done), 0, args.err, kDevTimeoutAccum, lim);
  } else if (warp >= 4) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3, h = (warp - 4) >> 2;
    const int m = kTileM * h + 32 * q + lane;  // box position: row m / 16, column m % 16
    const int r = m >> 4, c = m & 15;
    const bool inner = r >= 1 && r <= kInner && c >= 1 && c <= kInner;
    float* zrow = zs + m * Cfg::kZS;
    int lt = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x, ++lt) {
      const int buf = lt & 1, use = lt >> 1;
      bool got = !*abort_flag && mbar_wait_bounded(smem_u32(&tfull[buf]), use & 1, args.err, kDevTimeoutAccum, lim);
      // all epilogue threads agree (and have finished the previous tile's
      // reads of the Z rows) before any of them writes Z
      got = epi_all(got);
      if (!got) {
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      // phase 1: Z[dy][co] = sum_dx Y[(r, c + dx - 1), (dy, dx, co)]
      float z[3 * COUT];
#pragma unroll
      for (int i = 0; i < 3 * COUT; ++i) z[i] = 0.f;
      const uint32_t taddr = tmem + buf * 2 * Cfg::kAccCols + h * Cfg::kAccCols + ((uint32_t)(32 * q) << 16);
#pragma unroll
      for (int ch = 0; ch < Cfg::kN / 16; ++ch) {
        uint32_t rr[16];
        tmem_ld16(taddr + ch * 16, rr);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int n = ch * 16 + j;
          if (n < Cfg::kTaps) {
            const int s9 = n / COUT, co = n % COUT, dy = s9 / 3, dx = s9 % 3;
            float v = __uint_as_float(rr[j]);
            // dx = 0 needs the left neighbour's Y, dx = 2 the right one's
            if (dx == 0) v = __shfl_up_sync(0xffffffffu, v, 1);
            if (dx == 2) v = __shfl_down_sync(0xffffffffu, v, 1);
            z[dy * COUT + co] += v;
          }
        }
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&tempty[buf]));  // the accumulator may be overwritten
#pragma unroll
      for (int i = 0; i < 3 * COUT; ++i) zrow[i] = z[i];
      epi_sync();
      // phase 2: out[q] = bias + Z[row above][dy 0] + Z[this row][dy 1] + Z[row below][dy 2]
      const VTile t = vtile(args, u);
      const int y = t.ty * kInner - 1 + r, x = t.tx * kInner - 1 + c;
      if (inner && y < args.H && x < args.W) {
        float o[COUT];
#pragma unroll
        for (int co = 0; co < COUT; ++co)
          o[co] = __ldg(args.bias + co) + zrow[-kBox * Cfg::kZS + co] + zrow[COUT + co] +
                  zrow[kBox * Cfg::kZS + 2 * COUT + co];
        const int fo = args.out_f0 + t.f;
        if constexpr (VP == 2) {
          const long long base = (long long)t.b * args.vid_bs + (long long)fo * (4LL * args.H * args.W);
#pragma unroll
          for (int k = 0; k < 3; ++k) {
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              const float a0 = o[4 * k + i], a1 = o[4 * k + 2 + i];  // column offsets j = 0, 1
              const long long off = base + k * args.vid_cs + (long long)(2 * y + i) * (2LL * args.W) + 2LL * x;
              if (args.preclamp) *reinterpret_cast<float2*>(args.preclamp + off) = make_float2(a0, a1);
              const float c0 = fminf(fmaxf(a0, -1.f), 1.f), c1 = fminf(fmaxf(a1, -1.f), 1.f);
              if (args.out_f32)
                *reinterpret_cast<float2*>(static_cast<float*>(args.out) + off) = make_float2(c0, c1);
              else
                *reinterpret_cast<uint32_t*>(static_cast<__nv_bfloat16*>(args.out) + off) = pack_bf16x2(c0, c1);
            }
          }
        } else {
          const long long off = (long long)t.b * args.vid_bs + (long long)fo * args.H * args.W + (long long)y * args.W + x;
#pragma unroll
          for (int k = 0; k < 3; ++k) {
            if (args.preclamp) args.preclamp[off + k * args.vid_cs] = o[k];
            const float cl = fminf(fmaxf(o[k], -1.f), 1.f);
            if (args.out_f32)
              static_cast<float*>(args.out)[off + k * args.vid_cs] = cl;
            else
              static_cast<__nv_bfloat16*>(args.out)[off + k * args.vid_cs] = __float2bfloat16_rn(cl);
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, Cfg::kTmemCols);
  }
}

template <int COUT, int VP>
cudaError_t launch_v(const VideoConvLaunch& L, cudaStream_t stream) {
  using Cfg = VCfg<COUT>;
  auto kern = video_conv_kernel<COUT, VP>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cfg::kSmem);
  if (e != cudaSuccess) return e;
  const VideoConvArgs& a = L.args;
  const long long units = (long long)a.frames * a.tiles_x * a.tiles_y * a.batches;
  if (units <= 0) return cudaSuccess;
  if (units > 0x7FFFFFFFLL) return cudaErrorInvalidConfiguration;
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const long long grid = units < sms ? units : sms;  // persistent: one CTA per SM
  kern<<<(unsigned)grid, kVThreads, Cfg::kSmem, stream>>>(L.a, L.b, a);
  return cudaGetLastError();
}

__global__ void pack_tapfold_kernel(const void* __restrict__ src, int src_f32, int Co, int Ci, int ci_pad,
                                    __nv_bfloat16* __restrict__ dst, long long n) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  // src [Co][Ci][3][3][3]: i = ((co * Ci + ci) * 3 + dt) * 9 + s (s = 3 dy + dx)
  const int s = (int)(i % 9);
  const int dt = (int)((i / 9) % 3);
  const int ci = (int)((i / 27) % Ci);
  const int co = (int)(i / (27LL * Ci));
  const float v = src_f32 ? static_cast<const float*>(src)[i] : __bfloat162float(static_cast<const __nv_bfloat16*>(src)[i]);
  dst[(long long)(s * Co + co) * (3 * ci_pad) + dt * ci_pad + ci] = __float2bfloat16_rn(v);
}

}  // namespace

int video_conv_n(int cout) { return (9 * cout + 15) / 16 * 16; }

cudaError_t launch_video_conv(const VideoConvLaunch& L, cudaStream_t stream) {
  const VideoConvArgs& a = L.args;
  if (a.nkb < 1 || a.ci_pad != a.nkb * kBlockK) return cudaErrorInvalidValue;
  if (a.cout == 12 && a.vid_patch == 2) return launch_v<12, 2>(L, stream);
  if (a.cout == 3 && a.vid_patch == 1) return launch_v<3, 1>(L, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_pack_tapfold(const void* src, int src_f32, int Co, int Ci, int ci_pad, __nv_bfloat16* dst,
                                cudaStream_t s) {
  const long long n = 27LL * Co * Ci;
  if (n == 0) return cudaSuccess;
  pack_tapfold_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(src, src_f32, Co, Ci, ci_pad, dst, n);
  return cudaGetLastError();
}

}  // namespace wan
