// Implicit-GEMM convolution / batched GEMM on the sm_103a tensor cores.
//
// One CTA computes a 128 x BN output tile: 128 positions of one output frame
// (a box_w x box_h rectangle: 16 x 8, or 128 x 1 in row mode) by BN output
// channels, accumulated in fp32 in tensor memory.  Warp roles (384 threads):
//   warp 0, lane 0   TMA producer: per K block, one 5-D tile load of the A
//                    activation box (64 channels x pixels, zero-filled
//                    outside the frame) and 3-D loads of the B weight blocks
//   warp 1, lane 0   MMA issuer: tcgen05.mma (M=128, N=BN, K=16), 4 per K
//                    block and tap, then a tcgen05.commit freeing the stage
//   warp 2           TMEM allocation / release
//   warps 4-11       epilogue: tcgen05.ld of the accumulator, bias, residual /
//                    fused RMS norm / DupUp3D / unpatchify, stores
// Shared-memory rings with "full" and "empty" mbarriers per slot overlap the
// loads with the MMAs (plain and row modes: one ring of A + B stages;
// band mode: an A ring and a B ring).  All waits are bounded.
#include "kernels.h"
#include "ptx.cuh"

namespace wan {

// 12 warps: producer (0), MMA issuer (1), TMEM allocator (2), idle (3),
// and 8 epilogue warps (4-11): warp w reads TMEM lanes 32*(w % 4) .. +31 and
// the column half (w - 4) / 4 of the tile.
constexpr int kThreads = 384;
constexpr int kEpiThreads = 256;

// Band mode: A boxes of 16 x 10 positions (a tile's 8 rows and one halo row
// above and below), 20 KB.
constexpr int kBandABox = 16 * kBandBoxRows * 128;
// Row mode: 130 pixels x 128 B, rounded up to whole 1 KB swizzle atoms.
constexpr int kRowABox = 17 * 1024;

template <int BN, bool ROW = false, bool BAND = false, int NDX = 3>
struct ConvCfg {
  // as many stages as fit in 227 KB: 16 KB of A plus BN x 128 B of B each;
  // row mode: a 130-row A box (17 KB) and three taps of B; band mode: A
  // boxes (16 x 10 pixels, 20 KB) and one-tap B blocks in separate rings
  static constexpr int kStages = BAND ? (BN >= 256 ? 5 : 6)
                                      : ROW ? (NDX == 2 ? (BN <= 96 ? 5 : (BN <= 128 ? 4 : 3))
                                                          : (BN <= 96 ? 4 : (BN <= 128 ? 3 : 2)))
                                            : (BN >= 256 ? 4 : (BN > 128 ? 5 : (BN == 128 ? 6 : (BN > 64 ? 7 : 8))));
  static constexpr int kAStages = BAND ? 3 : kStages;  // A slots (the B ring has kStages)
  static constexpr int kABytes = ROW ? kRowABox : BAND ? kBandABox : kTileM * kBlockK * 2;  // 17 / 20 / 16 KB
  static constexpr int kBBytes = (ROW ? NDX : 1) * BN * kBlockK * 2;
  // one accumulator buffer of BN columns; two are allocated, kAccCols apart
  // (a power of two, so the allocation is one too)
  static constexpr int kAccCols = BN <= 32 ? 32 : (BN <= 64 ? 64 : (BN <= 128 ? 128 : 256));
  static constexpr size_t kSmem = 1024 + (size_t)kAStages * kABytes + (size_t)kStages * kBBytes +
                                   8 * (2 * kStages + 2 * kAStages + 7) + 16 + 4 * 2 * 2 * 128;
};

__device__ __forceinline__ void store16(void* dst, int f32, const float (&v)[16], int lo = 0) {
  if (lo) {
    // split format: hi at dst, lo = v - hi at dst + lo
    float h[16], l[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      h[i] = __bfloat162float(__float2bfloat16_rn(v[i]));
      l[i] = v[i] - h[i];
    }
    uint4* d = reinterpret_cast<uint4*>(dst);
    uint4* e = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(dst) + lo);
    d[0] = make_uint4(pack_bf16x2(h[0], h[1]), pack_bf16x2(h[2], h[3]), pack_bf16x2(h[4], h[5]), pack_bf16x2(h[6], h[7]));
    d[1] = make_uint4(pack_bf16x2(h[8], h[9]), pack_bf16x2(h[10], h[11]), pack_bf16x2(h[12], h[13]),
                      pack_bf16x2(h[14], h[15]));
    e[0] = make_uint4(pack_bf16x2(l[0], l[1]), pack_bf16x2(l[2], l[3]), pack_bf16x2(l[4], l[5]), pack_bf16x2(l[6], l[7]));
    e[1] = make_uint4(pack_bf16x2(l[8], l[9]), pack_bf16x2(l[10], l[11]), pack_bf16x2(l[12], l[13]),
                      pack_bf16x2(l[14], l[15]));
    return;
  }
  if (f32) {
    float4* d = reinterpret_cast<float4*>(dst);
#pragma unroll
    for (int i = 0; i < 4; ++i) d[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
  } else {
    uint4* d = reinterpret_cast<uint4*>(dst);
    d[0] = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                      pack_bf16x2(v[6], v[7]));
    d[1] = make_uint4(pack_bf16x2(v[8], v[9]), pack_bf16x2(v[10], v[11]), pack_bf16x2(v[12], v[13]),
                      pack_bf16x2(v[14], v[15]));
  }
}

// v += bias[0..15]: four 16-byte loads (bias buffers are padded with zeros
// to the N tile, 16-byte aligned).
__device__ __forceinline__ void add_bias16(const float* bias, float (&v)[16]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 b = __ldg(reinterpret_cast<const float4*>(bias) + i);
    v[4 * i] += b.x;
    v[4 * i + 1] += b.y;
    v[4 * i + 2] += b.z;
    v[4 * i + 3] += b.w;
  }
}

__device__ __forceinline__ void add16_bf16(const __nv_bfloat16* src, float (&v)[16]) {
  const uint4* s = reinterpret_cast<const uint4*>(src);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint4 a = s[h];
    const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[8 * h + 2 * i] += bf16_lo(w[i]);
      v[8 * h + 2 * i + 1] += bf16_hi(w[i]);
    }
  }
}

// v += src[0..15] (fp32, bf16, or split bf16 with the low halves at src + lo)
__device__ __forceinline__ void add16(const void* src, int f32, float (&v)[16], int lo = 0) {
  if (f32) {
    const float4* s = reinterpret_cast<const float4*>(src);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 a = s[i];
      v[4 * i] += a.x;
      v[4 * i + 1] += a.y;
      v[4 * i + 2] += a.z;
      v[4 * i + 3] += a.w;
    }
    return;
  }
  add16_bf16(static_cast<const __nv_bfloat16*>(src), v);
  if (lo) add16_bf16(static_cast<const __nv_bfloat16*>(src) + lo, v);
}

// Output tile coordinates of linear tile index t (n fastest, then the
// sub-pixel phase, x, y, frame, batch).
struct TileCoord {
  int tn, phase, tx, ty, f, b;
};
// With clusters of CL CTAs, a work unit is CL tiles side by side in x with
// the same N tile; CTA `rank` of the cluster takes x tile unit.x * CL + rank
// (past the frame's right edge when tiles_x is not a multiple of CL: an
// all-out-of-range tile whose loads read zeros and whose stores are masked).
// Unit order: N tile, sub-pixel phase, frame, then x, y, batch.  Frames come
// before space so that the output frames of one spatial tile run side by
// side: each input frame serves three time taps while it is still in L2.
__device__ __forceinline__ int tiles_x_units(const ConvArgs& a, int CL) { return (a.tiles_x + CL - 1) / CL; }
__device__ __forceinline__ TileCoord tile_coord(const ConvArgs& a, int t, int CL = 1, int rank = 0) {
  TileCoord c;
  c.tn = t % a.tiles_n;
  t /= a.tiles_n;
  c.phase = 0;
  if (a.subpix) {
    c.phase = t & 3;
    t >>= 2;
  }
  c.f = t % a.frames;
  t /= a.frames;
  if (a.row) {  // cluster pairs are adjacent rows
    c.tx = t % a.tiles_x;
    t /= a.tiles_x;
    const int ny = (a.tiles_y + CL - 1) / CL;
    c.ty = (t % ny) * CL + rank;
    c.b = t / ny;
    return c;
  }
  const int nx = tiles_x_units(a, CL);
  c.tx = (t % nx) * CL + rank;
  t /= nx;
  c.ty = t % a.tiles_y;
  c.b = t / a.tiles_y;
  return c;
}
// Work units of a launch: N tiles x phases x frames x spatial units x batches.
__host__ __device__ __forceinline__ long long conv_units(const ConvArgs& a, int CL) {
  const long long sp = a.row ? (long long)a.tiles_x * ((a.tiles_y + CL - 1) / CL)
                             : (long long)((a.tiles_x + CL - 1) / CL) * a.tiles_y;
  return (long long)a.tiles_n * (a.subpix ? 4 : 1) * sp * a.frames * a.batches;
}

// Epilogue of a tile that holds all N output channels, with the RMS norm of
// the output fused in.  Pass 1: y = acc + bias (+ residual), its sum of
// squares, and the raw y to `out` if requested.  Pass 2: y again, scaled by
// 1 / max(||y||, 1e-12) and sqrt(C) * gamma, SiLU, to out2.
template <int BN>
__device__ __forceinline__ void epilogue_norm_tile(const ConvArgs& args, uint32_t tbase, int f, int b, long long pos,
                                                   bool valid, int c_begin, int c_end, float* red, int m, int h,
                                                   uint32_t ssbar, uint32_t ss_parity) {
  const void* rp = nullptr;
  if (args.res) {
    const long long ro = (long long)b * args.res_bs + (long long)(args.res_f0 + f) * args.res_fs + pos * args.res_ldc;
    rp = args.res_f32 ? (const void*)(static_cast<const float*>(args.res) + ro)
                      : (const void*)(static_cast<const __nv_bfloat16*>(args.res) + ro);
  }
  const int esz = args.res_f32 ? 4 : 2;
  const long long lim = args.wait_limit > 0 ? args.wait_limit : kWaitLimitCycles;
  float ss = 0.f;
  float rinv = 0.f;
#pragma unroll 1
  for (int pass = 0; pass < 2; ++pass) {
    if (pass == 1) {
      // the other column half's partial sum of squares, through shared memory
      red[h * 128 + m] = ss;
      mbar_arrive(ssbar);
      mbar_wait_bounded(ssbar, ss_parity, args.err, kDevTimeoutAccum, lim);
      ss += red[(1 - h) * 128 + m];
      rinv = 1.0f / fmaxf(sqrtf(ss), 1e-12f);
    }
#pragma unroll 1
    for (int c = c_begin; c < c_end; ++c) {
      const int n0 = c * 16;
      if (n0 >= args.N) break;  // warp-uniform
      __syncwarp();
      uint32_t r[16];
      tmem_ld16(tbase + c * 16, r);
      tmem_ld_wait();
      float v[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
      if (args.bias) add_bias16(args.bias + n0, v);
      if (!valid) continue;
      if (rp) add16(static_cast<const char*>(rp) + (long long)n0 * esz, args.res_f32, v, args.res_lo);
      if (pass == 0) {
#pragma unroll
        for (int i = 0; i < 16; ++i) ss = fmaf(v[i], v[i], ss);
        if (args.out) {
          const long long oo = (long long)b * args.out_bs + (long long)(args.out_f0 + f * args.out_fmul) * args.out_fs +
                               pos * args.out_ldc + n0;
          void* op = args.out_f32 ? (void*)(static_cast<float*>(args.out) + oo)
                                  : (void*)(static_cast<__nv_bfloat16*>(args.out) + oo);
          store16(op, args.out_f32, v, args.out_lo);
        }
      } else {
        float g[16];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float4 g4 = __ldg(reinterpret_cast<const float4*>(args.norm_gs + n0) + i);
          g[4 * i] = g4.x;
          g[4 * i + 1] = g4.y;
          g[4 * i + 2] = g4.z;
          g[4 * i + 3] = g4.w;
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float y = v[i] * (rinv * g[i]);
          if (args.norm_silu) y = __fdividef(y, 1.0f + __expf(-y));
          v[i] = y;
        }
        const long long oo = (long long)b * args.out2_bs +
                             (long long)ring_slot(args.out2_f0 + f, args.out2_fmod) * args.out2_fs +
                             pos * args.out2_ldc + n0;
        store16(static_cast<__nv_bfloat16*>(args.out2) + oo, 0, v, args.out2_lo);
      }
    }
  }
}

// Epilogue of one tile: 4 warps, thread q*32 + lane owns accumulator row
// (TMEM lane) q*32 + lane, i.e. one output position, and walks its BN columns
// 16 at a time.
template <int BN, int EPI>
__device__ __forceinline__ void epilogue_tile(const ConvArgs& args, uint32_t tacc, const TileCoord& tc, int q, int h,
                                              int lane, bool got, float* red, uint32_t ssbar, uint32_t ss_parity) {
  const int m = q * 32 + lane;
  const int pi = tc.phase >> 1, pj = tc.phase & 1;
  const int yy = tc.ty * args.box_h + m / args.box_w;
  const int xx = tc.tx * args.box_w + m % args.box_w;
  const bool valid = got && yy < args.H && xx < args.W;
  const int f = tc.f, b = tc.b;
  const long long pos = args.subpix ? (long long)(2 * yy + pi) * (2 * args.W) + (2 * xx + pj)
                                    : (long long)yy * args.W + xx;
  const uint32_t tbase = tacc + ((uint32_t)(q * 32) << 16);
  constexpr int NC = BN / 16;  // 16-column chunks; half h takes [h*NC/2, (h+1)*NC/2)
  const int c_begin = (h * NC) / 2, c_end = ((h + 1) * NC) / 2;
  if constexpr (EPI == kEpiStore) {
    if (args.norm_gs) {
      epilogue_norm_tile<BN>(args, tbase, f, b, pos, valid, c_begin, c_end, red, m, h, ssbar, ss_parity);
      return;
    }
  }
#pragma unroll 1
  for (int c = c_begin; c < c_end; ++c) {
    const int n0 = tc.tn * BN + c * 16;
    if (n0 >= args.N) break;  // warp-uniform
    __syncwarp();               // tcgen05.ld is .sync.aligned: all 32 lanes together
    uint32_t r[16];
    tmem_ld16(tbase + c * 16, r);
    tmem_ld_wait();
    float v[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
    if (args.bias) add_bias16(args.bias + n0, v);
    if (!valid) continue;       // lanes re-converge at the __syncwarp above
    if constexpr (EPI == kEpiVideo) {
      if (args.vid_patch == 1) {  // three colour channels, no unpatchify
        const long long off = (long long)b * args.vid_bs + (long long)(args.out_f0 + f) * args.H * args.W + pos;
#pragma unroll
        for (int k = 0; k < 3; ++k) {
          if (args.preclamp) args.preclamp[off + k * args.vid_cs] = v[k];
          const float c = fminf(fmaxf(v[k], -1.f), 1.f);
          if (args.out_f32)
            static_cast<float*>(args.out)[off + k * args.vid_cs] = c;
          else
            static_cast<__nv_bfloat16*>(args.out)[off + k * args.vid_cs] = __float2bfloat16_rn(c);
        }
        continue;
      }
      const long long base = (long long)b * args.vid_bs + (long long)(args.out_f0 + f) * (4LL * args.H * args.W);
#pragma unroll
      for (int k = 0; k < 3; ++k) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const float a0 = v[4 * k + i], a1 = v[4 * k + 2 + i];  // column offsets j = 0, 1
          const long long off = base + k * args.vid_cs + (long long)(2 * yy + i) * (2LL * args.W) + 2LL * xx;
          if (args.preclamp) *reinterpret_cast<float2*>(args.preclamp + off) = make_float2(a0, a1);
          const float c0 = fminf(fmaxf(a0, -1.f), 1.f), c1 = fminf(fmaxf(a1, -1.f), 1.f);
          if (args.out_f32)
            *reinterpret_cast<float2*>(static_cast<float*>(args.out) + off) = make_float2(c0, c1);
          else
            *reinterpret_cast<uint32_t*>(static_cast<__nv_bfloat16*>(args.out) + off) = pack_bf16x2(c0, c1);
        }
      }
    } else {
      if constexpr (EPI == kEpiStore) {
        if (args.res) {
          const long long ro =
              (long long)b * args.res_bs + (long long)(args.res_f0 + f) * args.res_fs + pos * args.res_ldc + n0;
          const void* rp = args.res_f32 ? (const void*)(static_cast<const float*>(args.res) + ro)
                                        : (const void*)(static_cast<const __nv_bfloat16*>(args.res) + ro);
          add16(rp, args.res_f32, v, args.res_lo);
        }
      } else {  // kEpiDup
        const int sf = (f + (args.dup_first ? args.dup_ft - 1 : 0)) / args.dup_ft;
        // source position of output (Y, X) is (Y >> 1, X >> 1): in the
        // sub-pixel form that is the tile position itself
        const long long sp = args.subpix ? (long long)yy * args.dup_W + xx
                                         : (long long)(yy >> 1) * args.dup_W + (xx >> 1);
        const __nv_bfloat16* src = static_cast<const __nv_bfloat16*>(args.dup) + (long long)b * args.dup_bs +
                                   (long long)sf * args.dup_fs + sp * args.dup_ldc;
        if (args.dup_pairs) {
          // channel c reads source channel 2c + (row & 1)
          const int odd = args.subpix ? pi : (yy & 1);
          for (int part = 0; part < (args.dup_lo ? 2 : 1); ++part) {
            const uint4* s4 = reinterpret_cast<const uint4*>(src + 2 * n0 + (part ? args.dup_lo : 0));
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              const uint4 a = s4[h];
              const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
              for (int i = 0; i < 4; ++i) v[4 * h + i] += odd ? bf16_hi(w[i]) : bf16_lo(w[i]);
            }
          }
        } else {
          add16(src + n0, 0, v, args.dup_lo);
        }
      }
      int fo = args.out_f0 + f * args.out_fmul;
      int no = n0;
      if (args.interleave_c > 0 && n0 >= args.interleave_c) {
        fo += 1;
        no -= args.interleave_c;
      }
      const long long oo = (long long)b * args.out_bs + (long long)fo * args.out_fs + pos * args.out_ldc + no;
      void* op = args.out_f32 ? (void*)(static_cast<float*>(args.out) + oo)
                              : (void*)(static_cast<__nv_bfloat16*>(args.out) + oo);
      store16(op, args.out_f32, v, args.out_lo);
    }
  }
}

// Persistent kernel: each cluster of CL CTAs walks work units
// blockIdx.x / CL, + gridDim.x / CL, ...  The accumulator is double-buffered
// in TMEM (2 x BN columns), so the epilogue warps drain tile i while the MMA
// issuer accumulates tile i + 1.  With CL = 2 the two CTAs compute adjacent
// tiles (x tiles, or rows in row mode) of the same N tile: each loads half of
// the B block and multicasts it to both, and each MMA issuer frees a B slot
// in both CTAs (the slot's "empty" barrier counts both), so L2 delivers B
// once per pair.
template <int BN, int EPI, int CL, bool ROW, bool BAND, int NDX = 3>
__global__ void __launch_bounds__(kThreads, 1)
    conv_gemm_kernel(const __grid_constant__ CUtensorMap mapA0, const __grid_constant__ CUtensorMap mapA1,
                     const __grid_constant__ CUtensorMap mapB, const __grid_constant__ ConvArgs args) {
  using Cfg = ConvCfg<BN, ROW, BAND, NDX>;
  static_assert(!BAND || CL == 2, "band mode shares B across a pair of CTAs");
  constexpr int S = Cfg::kStages;
  constexpr int SA = Cfg::kAStages;
  constexpr uint32_t kAccCols = Cfg::kAccCols;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + SA * Cfg::kABytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + S * Cfg::kBBytes);
  uint64_t* empty = full + S;
  uint64_t* fullA = empty + S;    // [SA] band mode: A box landed (unused otherwise)
  uint64_t* emptyA = fullA + SA;  // [SA] band mode: A box consumed
  uint64_t* tfull = emptyA + SA;  // [2] accumulator ready (MMA -> epilogue)
  uint64_t* tempty = tfull + 2;  // [2] accumulator drained (epilogue -> MMA)
  uint64_t* done = tempty + 2;   // all MMAs of this CTA complete
  uint64_t* ssbar = done + 1;    // [2] fused norm: both column halves' partial sums written
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ssbar + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* red = reinterpret_cast<float*>(tmem_slot + 4);  // [2 tiles][2 halves][128 rows]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const long long lim = args.wait_limit > 0 ? args.wait_limit : kWaitLimitCycles;
  const int num_units = (int)conv_units(args, CL);
  const int rank = CL > 1 ? (int)cluster_ctarank() : 0;
  const int unit0 = blockIdx.x / CL, unit_step = gridDim.x / CL;
  constexpr uint16_t kPairMask = (1u << CL) - 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), CL);  // one MMA commit per CTA of the cluster
    }
    for (int s = 0; s < SA; ++s) {
      mbar_init(smem_u32(&fullA[s]), 1);
      mbar_init(smem_u32(&emptyA[s]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&tfull[i]), 1);
      mbar_init(smem_u32(&tempty[i]), kEpiThreads);
      mbar_init(smem_u32(&ssbar[i]), kEpiThreads);
    }
    mbar_init(smem_u32(done), 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_map(&mapA0);
    tma_prefetch_map(&mapA1);
    tma_prefetch_map(&mapB);
  }
  if (warp == 2) {
    tmem_alloc(smem_u32(tmem_slot), 2 * kAccCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if constexpr (CL > 1) cluster_sync();  // the peer's barriers exist before any multicast reaches them
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ producer
    int it = 0, ia = 0;  // B (or shared) stages and, in band mode, A boxes issued
    bool ok = true;
    for (int unit = unit0; unit < num_units && ok; unit += unit_step) {
      const TileCoord tc = tile_coord(args, unit, CL, rank);
      if constexpr (BAND) {
        // per tap (dt, dx) and 64-channel block: one 16 x 10 A box (rows from
        // tile start - 1) into the A ring, then its three dy taps' B blocks,
        // one per B slot
        for (int ti = 0; ti < args.n_taps && ok; ++ti) {
          const ConvTap tp = args.taps[ti];
          const int fr = ring_slot(args.src_f0[0] + tc.f + tp.dt, args.src_fmod);
          const int x0 = tc.tx * args.box_w + tp.dx, y0 = tc.ty * args.box_h - 1;
          for (int kb = 0; kb < tp.nkb && ok; ++kb) {
            const int sa = ia % SA;
            const int ra = ia / SA;
            if (ra > 0 && !mbar_wait_bounded(smem_u32(&emptyA[sa]), (ra - 1) & 1, args.err, kDevTimeoutEmpty, lim)) {
              ok = false;
              *abort_flag = 1;
              break;
            }
            if (*abort_flag) {
              ok = false;
              break;
            }
            const uint32_t fa = smem_u32(&fullA[sa]);
            mbar_arrive_expect_tx(fa, Cfg::kABytes);
            tma_load_5d(smem_u32(sA + sa * Cfg::kABytes), &mapA0, fa, tp.a_c0 + kb * kBlockK, x0, y0, fr, tc.b);
            ++ia;
            for (int j = 0; j < 3; ++j, ++it) {
              const int s = it % S;
              const int r = it / S;
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
              mbar_arrive_expect_tx(fb, Cfg::kBBytes);
              tma_load_3d_multicast(smem_u32(sB + s * Cfg::kBBytes + rank * (BN / CL) * kBlockK * 2), &mapB, fb,
                                    tp.b_k0 + j * args.row_bdk + kb * kBlockK, tc.tn * BN + rank * (BN / CL), 0,
                                    kPairMask);
            }
          }
        }
        continue;
      } else if constexpr (ROW) {
        // per tap (dt, dy) and 64-channel block: one 130-pixel A box (x from
        // tile start - 1) and the B blocks of its NDX dx taps.  In the
        // sub-pixel form (NDX = 2) the box starts at the phase's first column
        // offset (j - 1) and the row offset (i - 1) is added; B's third
        // coordinate is the phase
        const int sx = args.subpix ? (tc.phase & 1) : 0, sy = args.subpix ? (tc.phase >> 1) - 1 : 0;
        const int gR = args.subpix ? tc.phase : 0;
        for (int ti = 0; ti < args.n_taps && ok; ++ti) {
          const ConvTap tp = args.taps[ti];
          const int fr = ring_slot(args.src_f0[0] + tc.f + tp.dt, args.src_fmod);
          const int x0 = tc.tx * kTileM - 1 + sx, y0 = tc.ty + tp.dy + sy;
          for (int kb = 0; kb < tp.nkb; ++kb, ++it) {
            const int s = it % S;
            const int r = it / S;
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
            mbar_arrive_expect_tx(fb, (kTileM + 2) * kBlockK * 2 + Cfg::kBBytes);
            tma_load_5d(smem_u32(sA + s * Cfg::kABytes), &mapA0, fb, tp.a_c0 + kb * kBlockK, x0, y0, fr, tc.b);
            for (int j = 0; j < NDX; ++j) {
              const uint32_t dst = smem_u32(sB + s * Cfg::kBBytes + j * (BN * kBlockK * 2) +
                                            rank * (BN / CL) * kBlockK * 2);
              const int k = tp.b_k0 + j * args.row_bdk + kb * kBlockK;
              if constexpr (CL > 1)
                tma_load_3d_multicast(dst, &mapB, fb, k, tc.tn * BN + rank * (BN / CL), gR, kPairMask);
              else
                tma_load_3d(dst, &mapB, fb, k, tc.tn * BN, gR);
            }
          }
        }
        continue;
      }
      const int gB = args.b_per_frame ? (tc.b * args.b_gstride + tc.f) : tc.phase;
      const int sy = args.subpix ? (tc.phase >> 1) - 1 : 0, sx = args.subpix ? (tc.phase & 1) - 1 : 0;
      for (int ti = 0; ti < args.n_taps && ok; ++ti) {
        const ConvTap tp = args.taps[ti];
        const CUtensorMap* am = tp.src ? &mapA1 : &mapA0;
        const int fr = tp.src ? args.src_f0[1] + tc.f + tp.dt : ring_slot(args.src_f0[0] + tc.f + tp.dt, args.src_fmod);
        const int x0 = tc.tx * args.box_w + tp.dx + sx;
        const int y0 = tc.ty * args.box_h + tp.dy + sy;
        for (int kb = 0; kb < tp.nkb; ++kb, ++it) {
          const int s = it % S;
          const int r = it / S;
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
          mbar_arrive_expect_tx(fb, Cfg::kABytes + Cfg::kBBytes);
          tma_load_5d(smem_u32(sA + s * Cfg::kABytes), am, fb, tp.a_c0 + kb * kBlockK, x0, y0, fr, tc.b);
          if constexpr (CL > 1)
            tma_load_3d_multicast(smem_u32(sB + s * Cfg::kBBytes + rank * (Cfg::kBBytes / CL)), &mapB, fb,
                                  tp.b_k0 + kb * kBlockK, tc.tn * BN + rank * (BN / CL), gB, kPairMask);
          else
            tma_load_3d(smem_u32(sB + s * Cfg::kBBytes), &mapB, fb, tp.b_k0 + kb * kBlockK, tc.tn * BN, gB);
        }
      }
    }
    // Do not leave while copies into this CTA's shared memory are in flight.
    for (int j = (it > S ? it - S : 0); j < it; ++j)
      mbar_wait_bounded(smem_u32(&full[j % S]), (j / S) & 1, args.err, kDevTimeoutFull, lim);
    if constexpr (BAND)
      for (int j = (ia > SA ? ia - SA : 0); j < ia; ++j)
        mbar_wait_bounded(smem_u32(&fullA[j % SA]), (j / SA) & 1, args.err, kDevTimeoutFull, lim);
  } else if (warp == 1 && lane == 0) {
    // ---------------------------------------------------------- MMA issuer
    constexpr uint32_t idesc = idesc_bf16_f32(kTileM, BN);
    int lt = 0;
    // The issuing thread is on the critical path: ring slots and phases are
    // tracked incrementally, and the abort flag is read once per tile (every
    // wait is bounded and raises the flag when it runs out).
    int it_slot = 0, it_phase = 0;  // stage ring (the B ring in band mode)
    int kbc = 0;                    // row mode: channel block within the tap
    const int last_kb = args.taps[0].nkb - 1;
    int ia_slot = 0, ia_phase = 0;  // band mode: A ring
    bool ok = true;
    for (int unit = unit0; unit < num_units && ok; unit += unit_step, ++lt) {
      const int buf = lt & 1, use = lt >> 1;
      if (use > 0 && !mbar_wait_bounded(smem_u32(&tempty[buf]), (use - 1) & 1, args.err, kDevTimeoutAccum, lim)) {
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const uint32_t d = tmem + buf * kAccCols;
      if constexpr (BAND) {
        // per A box: its three dy taps from three consecutive B slots; tap dy
        // reads the box from image row dy on (16 pixels = 2 KB = two whole
        // swizzle atoms further); B slots are freed in both CTAs of the pair,
        // the A slot in this CTA only
        if (*abort_flag) {
          ok = false;
          break;
        }
        for (int kk = 0; kk < args.total_kb; ++kk) {
          const int sa = ia_slot;
          if (!mbar_wait_bounded(smem_u32(&fullA[sa]), ia_phase, args.err, kDevTimeoutFull, lim)) {
            *abort_flag = 1;
            ok = false;
            break;
          }
          if (++ia_slot == SA) {
            ia_slot = 0;
            ia_phase ^= 1;
          }
          tc_fence_after();
          const uint64_t a0 = sdesc_k128(smem_u32(sA + sa * Cfg::kABytes));
#pragma unroll
          for (int j = 0; j < 3; ++j) {
            const int s = it_slot;
            if (!mbar_wait_bounded(smem_u32(&full[s]), it_phase, args.err, kDevTimeoutFull, lim)) {
              *abort_flag = 1;
              ok = false;
              break;
            }
            if (++it_slot == S) {
              it_slot = 0;
              it_phase ^= 1;
            }
            tc_fence_after();
            const uint64_t ad = a0 + (uint64_t)((j * 16 * 128) >> 4);
            const uint64_t bd = sdesc_k128(smem_u32(sB + s * Cfg::kBBytes));
#pragma unroll
            for (int k = 0; k < kBlockK / 16; ++k)
              umma_bf16(d, ad + 2 * k, bd + 2 * k, idesc, (kk > 0 || j > 0 || k > 0) ? 1u : 0u);
            umma_commit_multicast(smem_u32(&empty[s]), kPairMask);
          }
          if (!ok) break;
          umma_commit(smem_u32(&emptyA[sa]));
        }
        umma_commit(smem_u32(&tfull[buf]));
        continue;
      }
      if (*abort_flag) {
        ok = false;
        break;
      }
      for (int kk = 0; kk < args.total_kb; ++kk) {
        const int s = it_slot;
        if (!mbar_wait_bounded(smem_u32(&full[s]), it_phase, args.err, kDevTimeoutFull, lim)) {
          *abort_flag = 1;
          ok = false;
          break;
        }
        if (++it_slot == S) {
          it_slot = 0;
          it_phase ^= 1;
        }
        tc_fence_after();
        if constexpr (ROW) {
          // dx tap j reads the A box from row j, 128 B further on: the 128-byte
          // swizzle is undone from the shared-memory address bits, as the TMA
          // applied it, so a start one row into an atom needs nothing else
          // (the descriptor's base-offset field stays 0); and its own B block
          const uint64_t a0 = sdesc_k128(smem_u32(sA + s * Cfg::kABytes));
          const uint64_t b0 = sdesc_k128(smem_u32(sB + s * Cfg::kBBytes));
          // a tap's last channel block may hold only tail_k16 x 16 channels
          // (the rest is TMA zero fill): issue just those K steps
          const bool tail = args.tail_k16 && kbc == last_kb;
          if (++kbc > last_kb) kbc = 0;
          if (tail && args.tail_k16 == 2) {
#pragma unroll
            for (int j = 0; j < NDX; ++j) {
              const uint64_t ad = a0 + (uint64_t)((j * 128) >> 4);
              const uint64_t bd = b0 + (uint64_t)((j * BN * kBlockK * 2) >> 4);
#pragma unroll
              for (int k = 0; k < 2; ++k)
                umma_bf16(d, ad + 2 * k, bd + 2 * k, idesc, (kk > 0 || j > 0 || k > 0) ? 1u : 0u);
            }
          } else {
#pragma unroll
            for (int j = 0; j < NDX; ++j) {
              const uint64_t ad = a0 + (uint64_t)((j * 128) >> 4);
              const uint64_t bd = b0 + (uint64_t)((j * BN * kBlockK * 2) >> 4);
#pragma unroll
              for (int k = 0; k < kBlockK / 16; ++k)
                umma_bf16(d, ad + 2 * k, bd + 2 * k, idesc, (kk > 0 || j > 0 || k > 0) ? 1u : 0u);
            }
          }
        } else {
          const uint64_t ad = sdesc_k128(smem_u32(sA + s * Cfg::kABytes));
          const uint64_t bd = sdesc_k128(smem_u32(sB + s * Cfg::kBBytes));
#pragma unroll
          for (int k = 0; k < kBlockK / 16; ++k)
            umma_bf16(d, ad + 2 * k, bd + 2 * k, idesc, (kk > 0 || k > 0) ? 1u : 0u);
        }
        if constexpr (CL > 1)
          umma_commit_multicast(smem_u32(&empty[s]), kPairMask);
        else
          umma_commit(smem_u32(&empty[s]));
      }
      umma_commit(smem_u32(&tfull[buf]));
    }
    // wait for every MMA of this CTA before the TMEM can be released
    umma_commit(smem_u32(done));
    mbar_wait_bounded(smem_u32(done), 0, args.err, kDevTimeoutAccum, lim);
  } else if (warp >= 4) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3, h = (warp - 4) >> 2;
    int lt = 0;
    for (int unit = unit0; unit < num_units; unit += unit_step, ++lt) {
      const int buf = lt & 1, use = lt >> 1;
      const bool got =
          !*abort_flag && mbar_wait_bounded(smem_u32(&tfull[buf]), use & 1, args.err, kDevTimeoutAccum, lim);
      if (!got) *abort_flag = 1;
      tc_fence_after();
      epilogue_tile<BN, EPI>(args, tmem + buf * kAccCols, tile_coord(args, unit, CL, rank), q, h, lane, got,
                             red + buf * 256, smem_u32(&ssbar[buf]), use & 1);
      tc_fence_before();
      mbar_arrive(smem_u32(&tempty[buf]));
      if (!got) break;
    }
  }
  tc_fence_before();
  __syncthreads();
  // no CTA leaves while its peer's MMA commits or multicast copies may still reach it
  if constexpr (CL > 1) cluster_sync();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 2 * kAccCols);
  }
}

template <int BN, int EPI, int CL, bool ROW = false, bool BAND = false, int NDX = 3>
static cudaError_t launch_t(const ConvLaunch& L, cudaStream_t stream) {
  using Cfg = ConvCfg<BN, ROW, BAND, NDX>;
  auto kern = conv_gemm_kernel<BN, EPI, CL, ROW, BAND, NDX>;
  // The shared-memory opt-in and the number of co-resident clusters depend
  // only on the kernel and the device: set and queried once per device (the
  // cluster occupancy query costs tens of microseconds of host time).
  constexpr int kMaxDev = 64;
  static int resident_cache[kMaxDev] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool cached = dev >= 0 && dev < kMaxDev && resident_cache[dev] > 0;
  if (!cached) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cfg::kSmem);
    if (e != cudaSuccess) return e;
  }
  const ConvArgs& a = L.args;
  const long long units = conv_units(a, CL);
  if (units <= 0) return cudaSuccess;
  if (units > 0x7FFFFFFFLL) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Cfg::kSmem;
  cfg.stream = stream;
  int resident = cached ? resident_cache[dev] : 0;  // CTAs (one per SM) or clusters that fit at once
  if (CL > 1) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3(CL);
    if (!cached) e = cudaOccupancyMaxActiveClusters(&resident, kern, &cfg);
  } else if (!cached) {
    e = cudaDeviceGetAttribute(&resident, cudaDevAttrMultiProcessorCount, dev);
  }
  if (e != cudaSuccess) return e;
  if (resident < 1) return cudaErrorInvalidConfiguration;
  if (!cached && dev >= 0 && dev < kMaxDev) resident_cache[dev] = resident;
  const long long groups = units < resident ? units : resident;  // persistent: one wave of CTAs / clusters
  cfg.gridDim = dim3((unsigned)(groups * CL));
  e = cudaLaunchKernelEx(&cfg, kern, L.a0, L.a1, L.b, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// Clusters of two CTAs share the B block (each loads half and multicasts it)
// for BN = 96, 192 and 256, where the stage's bytes, not the MMAs, would
// otherwise set the pace; the B tensor map's box then holds BN / 2 rows.
static bool conv_clustered(int bn) { return bn == 96 || bn == 192 || bn == 256; }
int conv_b_box_rows(int bn) { return conv_clustered(bn) ? bn / 2 : bn; }

cudaError_t launch_conv(const ConvLaunch& L, cudaStream_t stream) {
  if (L.args.band) {
    if (L.epi != kEpiStore || L.args.subpix || L.args.row) return cudaErrorInvalidValue;
    if (L.bn == 256) return launch_t<256, kEpiStore, 2, false, true>(L, stream);
    if (L.bn == 192) return launch_t<192, kEpiStore, 2, false, true>(L, stream);
    return cudaErrorInvalidValue;
  }
  if (L.args.row) {
    if (L.epi != kEpiStore) return cudaErrorInvalidValue;
    if (L.args.subpix) {  // 2 x 2 taps per phase: two dx taps per A box
      if (L.bn == 96) return launch_t<96, kEpiStore, 2, true, false, 2>(L, stream);
      if (L.bn == 128) return launch_t<128, kEpiStore, 2, true, false, 2>(L, stream);
      if (L.bn == 192) return launch_t<192, kEpiStore, 2, true, false, 2>(L, stream);
      return cudaErrorInvalidValue;
    }
    if (L.bn == 96) return launch_t<96, kEpiStore, 2, true>(L, stream);
    if (L.bn == 128) return launch_t<128, kEpiStore, 2, true>(L, stream);
    if (L.bn == 192) return launch_t<192, kEpiStore, 2, true>(L, stream);
    return cudaErrorInvalidValue;
  }
  if (L.epi == kEpiVideo) {
    if (L.bn != 16) return cudaErrorInvalidValue;
    return launch_t<16, kEpiVideo, 1>(L, stream);
  }
  if (L.epi == kEpiDup) {
    switch (L.bn) {
      case 16: return launch_t<16, kEpiDup, 1>(L, stream);
      case 32: return launch_t<32, kEpiDup, 1>(L, stream);
      case 64: return launch_t<64, kEpiDup, 1>(L, stream);
      case 128: return launch_t<128, kEpiDup, 1>(L, stream);
      case 256: return launch_t<256, kEpiDup, 2>(L, stream);
    }
    return cudaErrorInvalidValue;
  }
  switch (L.bn) {
    case 16: return launch_t<16, kEpiStore, 1>(L, stream);
    case 32: return launch_t<32, kEpiStore, 1>(L, stream);
    case 64: return launch_t<64, kEpiStore, 1>(L, stream);
    case 96: return launch_t<96, kEpiStore, 2>(L, stream);
    case 128: return launch_t<128, kEpiStore, 1>(L, stream);
    case 192: return launch_t<192, kEpiStore, 2>(L, stream);
    case 256: return launch_t<256, kEpiStore, 2>(L, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace wan
