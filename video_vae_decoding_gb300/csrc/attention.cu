// Flash-style mid-block attention core (page "wan22_vae_decode/reference.py",
// "The parts", fourth bullet; the single-head attention of the page "Fix the
// Wan VAE attention block"): per frame, O = softmax(q k^T / sqrt(C)) v over
// the frame's HW positions, without the HW x HW score matrix ever leaving the
// SM.
//
// Two kernels.  flash_attn_kernel (head dims up to 384): one CTA takes 128
// queries of one frame; the score block S = Q K_j^T of 128 keys and the output
// accumulator O (128 x C fp32) both live in tensor memory (128 + C <= 512
// columns); Q stays in shared memory for the whole key loop.
// flash_attn_split_kernel (head dims 512 and 1024) is described further down.
// Per key block j of the first:
//   MMA issuer   S_j = Q K_j^T (M=128, N=128, K=C), then O += P_{j-1} V_{j-1}
//   softmax      row max and exp2 of the scaled scores (online softmax: the
//                running max m only moves when a block's max exceeds it by more
//                than 8 in log2 units, so P <= 256 and O is rescaled rarely),
//                P_j rounded to bf16 into shared memory in the MMA's operand
//                layout, and the row sum l of the rounded values
// and at the end O / l is written as bf16 (the weights of V sum to one).  Keys past HW are masked to -inf;
// queries past HW are computed on zero rows and not stored.
//
// Warp roles (384 threads): warp 0 lane 0 TMA producer (Q once; per key block
// C/64 boxes of 128 keys x 64 channels of K and the V^T boxes of VR rows x 64
// keys, through one 16 KB-slot ring in the order the MMA consumes them), warp
// 1 lane 0 MMA issuer, warp 2 TMEM allocation, warps 4-11 softmax and output
// (two threads per query row = TMEM lane, each taking half of the keys and
// half of the output columns).  Every wait is bounded.
#include "kernels.h"
#include "ptx.cuh"

namespace wan {

namespace {

constexpr int kFThreads = 384;
constexpr int kFStages = 6;
constexpr int kFUnit = 16384;  // one ring slot: 128 x 64 bf16

template <int NQ>  // C = 64 * NQ
struct FCfg {
  static constexpr int C = 64 * NQ;
  static constexpr int VR = (C % 128 == 0) ? 128 : 64;  // V^T rows per box (an MMA's N)
  static constexpr int NV = C / VR;                     // V^T row groups
  static constexpr int kVBytes = VR * 128;              // one V^T box: VR rows x 64 keys
  static constexpr int kTmemCols = (128 + C) <= 256 ? 256 : 512;
  static constexpr size_t kSmem =
      1024 + (size_t)NQ * kFUnit + 2 * kFUnit + (size_t)kFStages * kFUnit + 8 * 32 + 2 * 128 * 4;
};

// 2^x by the SFU's approximation (flushes subnormal results to zero); the
// probabilities it feeds are rounded to bf16.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int NQ>
__global__ void __launch_bounds__(kFThreads, 1)
    flash_attn_kernel(const __grid_constant__ CUtensorMap mapQK, const __grid_constant__ CUtensorMap mapV,
                      const __grid_constant__ FlashArgs args) {
  using Cfg = FCfg<NQ>;
  constexpr int S = kFStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;                    // NQ boxes of 128 queries x 64 channels
  uint8_t* sP = sQ + NQ * kFUnit;        // 2 boxes of 128 queries x 64 keys
  uint8_t* sR = sP + 2 * kFUnit;         // ring
  uint64_t* full = reinterpret_cast<uint64_t*>(sR + S * kFUnit);
  uint64_t* empty = full + S;
  uint64_t* q_full = empty + S;
  uint64_t* s_full = q_full + 1;   // S_j in TMEM
  uint64_t* s_free = s_full + 1;   // S_j read by the softmax threads
  uint64_t* p_full = s_free + 1;   // P_j in shared memory (and O rescaled)
  uint64_t* pv_done = p_full + 1;  // O += P_j V_j complete
  uint64_t* done = pv_done + 1;    // all MMAs of this CTA complete
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // [2 halves][128 rows]: the row max exchange (reused from block to block:
  // the barrier that opens each block orders a block's writes after the
  // previous block's reads)
  float* red = reinterpret_cast<float*>(tmem_slot + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qb = blockIdx.x, f = blockIdx.y, b = blockIdx.z;
  const int nkb = args.nkb;
  const long long lim = args.wait_limit > 0 ? args.wait_limit : kWaitLimitCycles;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    mbar_init(smem_u32(q_full), 1);
    mbar_init(smem_u32(s_full), 1);
    mbar_init(smem_u32(s_free), 256);
    mbar_init(smem_u32(p_full), 256);
    mbar_init(smem_u32(pv_done), 1);
    mbar_init(smem_u32(done), 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_map(&mapQK);
    tma_prefetch_map(&mapV);
  }
  if (warp == 2) {
    tmem_alloc(smem_u32(tmem_slot), Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS = tmem, tO = tmem + 128;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ producer
    mbar_arrive_expect_tx(smem_u32(q_full), NQ * kFUnit);
    for (int u = 0; u < NQ; ++u)
      tma_load_4d(smem_u32(sQ + u * kFUnit), &mapQK, smem_u32(q_full), args.q_c0 + 64 * u, 128 * qb, f, b);
    int it = 0;
    bool ok = true;
    // order of consumption: K_0, then (K_j, V_{j-1}) for j = 1 .. nkb - 1, then V_{nkb-1}
    for (int j = 0; j <= nkb && ok; ++j) {
      const int nk = j < nkb ? NQ : 0, nv = j >= 1 ? 2 * Cfg::NV : 0;
      for (int i = 0; i < nk + nv; ++i, ++it) {
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
        if (i < nk) {
          mbar_arrive_expect_tx(fb, kFUnit);
          tma_load_4d(smem_u32(sR + s * kFUnit), &mapQK, fb, args.k_c0 + 64 * i, 128 * j, f, b);
        } else {
          const int v = i - nk, rg = v >> 1, h = v & 1;  // V^T row group, key half
          mbar_arrive_expect_tx(fb, Cfg::kVBytes);
          tma_load_4d(smem_u32(sR + s * kFUnit), &mapV, fb, 128 * (j - 1) + 64 * h, Cfg::VR * rg, f, b);
        }
      }
    }
    for (int jj = (it > S ? it - S : 0); jj < it; ++jj)
      mbar_wait_bounded(smem_u32(&full[jj % S]), (jj / S) & 1, args.err, kDevTimeoutFull, lim);
    mbar_wait_bounded(smem_u32(q_full), 0, args.err, kDevTimeoutFull, lim);
  } else if (warp == 1 && lane == 0) {
    // ---------------------------------------------------------- MMA issuer
    constexpr uint32_t idS = idesc_bf16_f32(128, 128);
    constexpr uint32_t idO = idesc_bf16_f32(128, Cfg::VR);
    bool ok = mbar_wait_bounded(smem_u32(q_full), 0, args.err, kDevTimeoutFull, lim);
    if (!ok) *abort_flag = 1;
    int slot = 0, phase = 0;
    for (int j = 0; j <= nkb && ok; ++j) {
      if (j < nkb) {
        // S_j = Q K_j^T, once the softmax has read S_{j-1}
        if (j > 0 && !mbar_wait_bounded(smem_u32(s_free), (j - 1) & 1, args.err, kDevTimeoutAccum, lim)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int u = 0; u < NQ && ok; ++u) {
          if (!mbar_wait_bounded(smem_u32(&full[slot]), phase, args.err, kDevTimeoutFull, lim)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = sdesc_k128(smem_u32(sQ + u * kFUnit));
          const uint64_t bd = sdesc_k128(smem_u32(sR + slot * kFUnit));
#pragma unroll
          for (int k = 0; k < 4; ++k) umma_bf16(tS, ad + 2 * k, bd + 2 * k, idS, (u > 0 || k > 0) ? 1u : 0u);
          umma_commit(smem_u32(&empty[slot]));
          if (++slot == S) {
            slot = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        umma_commit(smem_u32(s_full));
      }
      if (j >= 1) {
        // O += P_{j-1} V_{j-1}, once P_{j-1} is written (and O rescaled)
        const int jv = j - 1;
        if (!mbar_wait_bounded(smem_u32(p_full), jv & 1, args.err, kDevTimeoutAccum, lim)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int v = 0; v < 2 * Cfg::NV && ok; ++v) {
          const int rg = v >> 1, h = v & 1;
          if (!mbar_wait_bounded(smem_u32(&full[slot]), phase, args.err, kDevTimeoutFull, lim)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = sdesc_k128(smem_u32(sP + h * kFUnit));
          const uint64_t bd = sdesc_k128(smem_u32(sR + slot * kFUnit));
#pragma unroll
          for (int k = 0; k < 4; ++k)
            umma_bf16(tO + Cfg::VR * rg, ad + 2 * k, bd + 2 * k, idO, (jv > 0 || h > 0 || k > 0) ? 1u : 0u);
          umma_commit(smem_u32(&empty[slot]));
          if (++slot == S) {
            slot = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        umma_commit(smem_u32(pv_done));
      }
    }
    if (!ok) *abort_flag = 1;
    // every MMA of this CTA completes before the TMEM is released
    umma_commit(smem_u32(done));
    mbar_wait_bounded(smem_u32(done), 0, args.err, kDevTimeoutAccum, lim);
  } else if (warp >= 4) {
    // ------------------------------------------------------ softmax, output
    // Eight warps: warp w reads TMEM lane quadrant w % 4, and half hk = (w - 4)
    // / 4 of the row: keys 64 hk .. 64 hk + 63 of each block, output columns
    // hk C/2 .. (hk + 1) C/2.  The two halves of a row exchange their maxima
    // through shared memory, so both take the same reference max; all eight
    // warps agree on every wait's outcome (named barrier 1) before going on.
    const int q = warp & 3, hk = (warp - 4) >> 2;
    const int row = 32 * q + lane;
    const uint32_t lane_off = (uint32_t)(32 * q) << 16;
    constexpr int CH = Cfg::C / 2;  // output columns per half
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nkb; ++j) {
      ok = epi_all(!*abort_flag && mbar_wait_bounded(smem_u32(s_full), j & 1, args.err, kDevTimeoutAccum, lim));
      if (!ok) break;
      tc_fence_after();
      // the raw scores (the scale is applied in the exponent below)
      float t[64];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t r[16];
        tmem_ld16(tS + lane_off + 64 * hk + 16 * c, r);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) t[16 * c + i] = __uint_as_float(r[i]);
      }
      tc_fence_before();
      mbar_arrive(smem_u32(s_free));
      // keys past the frame's positions
      const int kv = args.HW - 128 * j - 64 * hk;
      if (kv < 64) {
#pragma unroll
        for (int i = 0; i < 64; ++i)
          if (i >= kv) t[i] = -INFINITY;
      }
      float mb = t[0];
#pragma unroll
      for (int i = 1; i < 64; ++i) mb = fmaxf(mb, t[i]);
      mb *= args.scale_log2;  // the scale is positive: the max of the scaled scores
      red[hk * 128 + row] = mb;
      epi_sync();
      mb = fmaxf(mb, red[(1 - hk) * 128 + row]);
      float alpha = 1.f;
      if (mb > m + 8.f) {  // move the reference max (and rescale O and l by alpha)
        alpha = exp2f(m - mb);
        m = mb;
      }
      // P in bf16, and the row sum of the rounded values: the weights that
      // multiply V then sum to exactly 1 after the final division by l
      float rs = 0.f;
      const float sc = args.scale_log2;
#pragma unroll
      for (int i = 0; i < 64; ++i) {
        t[i] = __bfloat162float(__float2bfloat16_rn(ex2_approx(fmaf(t[i], sc, -m))));
        rs += t[i];
      }
      l = l * alpha + rs;
      // P buffer free and O stable once O += P_{j-1} V_{j-1} has completed
      if (j > 0) {
        ok = epi_all(mbar_wait_bounded(smem_u32(pv_done), (j - 1) & 1, args.err, kDevTimeoutAccum, lim));
        if (!ok) break;
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
          for (int c = 0; c < CH / 16; ++c) {
            uint32_t r[16];
            tmem_ld16(tO + lane_off + CH * hk + 16 * c, r);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
            tmem_st16(tO + lane_off + CH * hk + 16 * c, r);
          }
          tmem_st_wait();
        }
      }
      // P_j (bf16) in the 128-byte-swizzled K-major layout: row `row`, key
      // chunk c of 8 keys at 16-byte slot c ^ (row & 7) of its 128-byte line
      // (this half's 64 keys are one swizzled block)
      uint8_t* line = sP + hk * kFUnit + row * 128;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const float* v = t + 8 * c;
        const uint4 w = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                                   pack_bf16x2(v[6], v[7]));
        *reinterpret_cast<uint4*>(line + ((c ^ (row & 7)) << 4)) = w;
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(smem_u32(p_full));
    }
    if (ok) ok = epi_all(mbar_wait_bounded(smem_u32(pv_done), (nkb - 1) & 1, args.err, kDevTimeoutAccum, lim));
    if (!ok) {
      *abort_flag = 1;
    } else {
      tc_fence_after();
      // the row's weight sum: both halves' partial sums (taken against the same max)
      red[hk * 128 + row] = l;
      epi_sync();
      const float rl = 1.f / (l + red[(1 - hk) * 128 + row]);
      const int qrow = 128 * qb + row;
      __nv_bfloat16* dst = args.out + (long long)b * args.out_bs + (long long)f * args.out_fs +
                           (long long)qrow * args.out_ldc + CH * hk;
#pragma unroll 1
      for (int c = 0; c < CH / 16; ++c) {
        uint32_t r[16];
        tmem_ld16(tO + lane_off + CH * hk + 16 * c, r);
        tmem_ld_wait();
        if (qrow < args.HW) {
          float v[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]) * rl;
          uint4* d = reinterpret_cast<uint4*>(dst + 16 * c);
          d[0] = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                            pack_bf16x2(v[6], v[7]));
          d[1] = make_uint4(pack_bf16x2(v[8], v[9]), pack_bf16x2(v[10], v[11]), pack_bf16x2(v[12], v[13]),
                            pack_bf16x2(v[14], v[15]));
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

// ---------------------------------------------------------------------------
// Head dims 512 and 1024 (TI2V-5B's mid block).  A 128-query fp32 output
// accumulator is then C x 512 B, more than one SM's TMEM at C = 1024, and the
// 128 x C block of q more than its shared memory.  So NSL = C / 256 CTAs (side
// by side in the grid) take one block of 128 queries: CTA r accumulates
// output columns [256 r, 256 r + 256) (256 TMEM columns) beside a score block
// of 256 keys (the other 256).  Every CTA needs the full scores S_j = Q K_j^T
// (the softmax weights of its output columns), so each computes them from q
// and k chunks that are the same for all NSL CTAs (read from L2 by each), and
// loads the v^T boxes of its own 256 output columns.  (Sharing the q and k
// chunks by cluster multicast measured no faster: L2 was not the limit, and
// clusters of four CTAs fit only four to a GPC.)
// Per key block j (256 keys):
//   MMA issuer   S_j = Q K_j^T over C / 64 stages of (q box 128 x 64, k box
//                256 x 64), M = 128, N = 256; then O += P_{j-1} V_{j-1} over
//                four stages of one v^T box (256 columns x 64 keys)
//   softmax      the same online softmax as the kernel above (lazy reference
//                max, P rounded to bf16, l summed over the rounded values),
//                sixteen warps, four threads per query row with 64 keys and
//                64 output columns each (the SFU's exp2; a mask-free path for
//                all but the last key block).  P_j is formed in registers as
//                soon as S_j is read, so S_{j+1} starts while P_{j-1} V_{j-1}
//                is still running.
// The stages run through a 4-slot ring of 48 KB (four stages in flight: three
// did not cover the load latency).  P_j's boxes 0 and 1 have a 32 KB buffer
// of their own, written as soon as the softmax is done; a P V stage uses only
// the 32 KB B part of its slot (the v^T box), and boxes 2 and 3 live in the A
// part of the slot of their own P V stage (no room for a 64 KB P buffer
// beside four stages).  The softmax threads write box 2 or 3 once that slot's
// previous stage (four positions earlier: one of the last two of S_{j+1}, or
// of the stages before O += P_j V_j if no S follows) has been consumed:
// barrier pfree[kc], which the MMA issuer commits after that stage, completes
// once per key block.  (The slot's "empty" barrier cannot be used: it
// completes four times during S_{j+1}, and a parity wait only tells
// neighbouring phases apart.)  Each box has its own "written" barrier
// p_full[kc], so the P V stage of box 0 need not wait for box 3.
// ---------------------------------------------------------------------------
constexpr int kSThreads = 640;  // warps 0-3 producer, MMA issuer, TMEM allocation, idle; 4-19 softmax
constexpr int kSStages = 4;
constexpr int kSStage = 49152;  // A part 16 KB (q box) + B part 32 KB (k box or v^T box)

template <int NSL>
struct SCfg {
  static constexpr int C = 256 * NSL;
  static constexpr int NC = C / 64;  // 64-channel chunks of the score contraction
  static constexpr size_t kSmem = 1024 + (size_t)kSStages * kSStage + 2 * kFUnit + 192 + 2 * 128 * 4;
};

// The 512 softmax threads (warps 4-19) of the split kernel: named barrier 2.
__device__ __forceinline__ void sm_sync() { asm volatile("bar.sync 2, 512;" ::: "memory"); }
__device__ __forceinline__ bool sm_all(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 2, 512, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)v)
      : "memory");
  return r != 0;
}

// Position of stage kc of O += P_j V_j in the split kernel's stage sequence:
// the NC chunks of S_0, then for j' = 1 .. nkb - 1 the NC chunks of S_j' and
// the four stages of O += P_{j'-1} V_{j'-1}, then those of O += P_{nkb-1}
// V_{nkb-1}.  (Putting the P V stages in the middle of S_j' measured 19%
// slower: the softmax then has no P V MMAs to hide behind.)
__device__ __forceinline__ int split_pv_pos(int j, int nkb, int NC, int kc) {
  return NC * min(j + 2, nkb) + 4 * j + kc;
}

template <int NSL>
__global__ void __launch_bounds__(kSThreads, 1)
    flash_attn_split_kernel(const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapK,
                            const __grid_constant__ CUtensorMap mapV, const __grid_constant__ FlashArgs args) {
  using Cfg = SCfg<NSL>;
  constexpr int S = kSStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sR = smem;                // ring
  uint8_t* sP = sR + S * kSStage;    // P boxes 0 and 1 (boxes 2 and 3 live in ring slots)
  uint64_t* full = reinterpret_cast<uint64_t*>(sP + 2 * kFUnit);
  uint64_t* empty = full + S;
  uint64_t* s_full = empty + S;    // S_j in TMEM
  uint64_t* s_free = s_full + 1;   // S_j read by the softmax threads
  uint64_t* p_full = s_free + 1;   // [4] P_j box kc written (and O rescaled)
  uint64_t* pv_done = p_full + 4;  // O += P_j V_j complete
  uint64_t* done = pv_done + 1;    // all MMAs of this CTA complete
  uint64_t* pfree = done + 1;      // [4] the slot of P box kc is free
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(pfree + 4);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* red = reinterpret_cast<float*>(sP + 2 * kFUnit + 192);  // [2][128 rows]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = blockIdx.x % NSL;  // output column slice
  const int qb = blockIdx.x / NSL, f = blockIdx.y, b = blockIdx.z;
  const int nkb = args.nkb;
  const long long lim = args.wait_limit > 0 ? args.wait_limit : kWaitLimitCycles;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    mbar_init(smem_u32(s_full), 1);
    mbar_init(smem_u32(s_free), 512);
    for (int kc = 0; kc < 4; ++kc) mbar_init(smem_u32(&p_full[kc]), 512);
    mbar_init(smem_u32(pv_done), 1);
    mbar_init(smem_u32(done), 1);
    for (int kc = 0; kc < 4; ++kc) mbar_init(smem_u32(&pfree[kc]), 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_map(&mapQ);
    tma_prefetch_map(&mapK);
    tma_prefetch_map(&mapV);
  }
  if (warp == 2) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS = tmem, tO = tmem + 256;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ producer
    // order of consumption: S stages of block 0, then for j = 1 .. nkb - 1
    // the S stages of block j and the v^T stages of block j - 1, then the
    // v^T stages of block nkb - 1
    int it = 0;
    bool ok = true;
    for (int j = 0; j <= nkb && ok; ++j) {
      const int nk = j < nkb ? Cfg::NC : 0, nv = j >= 1 ? 4 : 0;
      for (int i = 0; i < nk + nv; ++i, ++it) {
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
        const uint32_t slot = smem_u32(sR + s * kSStage);
        if (i < nk) {
          mbar_arrive_expect_tx(fb, kSStage);
          tma_load_4d(slot, &mapQ, fb, args.q_c0 + 64 * i, 128 * qb, f, b);
          tma_load_4d(slot + kFUnit, &mapK, fb, args.k_c0 + 64 * i, 256 * j, f, b);
        } else {
          mbar_arrive_expect_tx(fb, 2 * kFUnit);
          tma_load_4d(slot + kFUnit, &mapV, fb, 256 * (j - 1) + 64 * (i - nk), 256 * rank, f, b);
        }
      }
    }
    // do not leave while copies into this CTA's shared memory are in flight
    for (int jj = (it > S ? it - S : 0); jj < it; ++jj)
      mbar_wait_bounded(smem_u32(&full[jj % S]), (jj / S) & 1, args.err, kDevTimeoutFull, lim);
  } else if (warp == 1 && lane == 0) {
    // ---------------------------------------------------------- MMA issuer
    constexpr uint32_t idN256 = idesc_bf16_f32(128, 256);
    bool ok = true;
    int slot = 0, phase = 0;
    for (int j = 0; j <= nkb && ok; ++j) {
      if (j < nkb) {
        // S_j = Q K_j^T, once the softmax has read S_{j-1}
        if (j > 0 && !mbar_wait_bounded(smem_u32(s_free), (j - 1) & 1, args.err, kDevTimeoutAccum, lim)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int c = 0; c < Cfg::NC && ok; ++c) {
          if (!mbar_wait_bounded(smem_u32(&full[slot]), phase, args.err, kDevTimeoutFull, lim)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = sdesc_k128(smem_u32(sR + slot * kSStage));
          const uint64_t bd = sdesc_k128(smem_u32(sR + slot * kSStage + kFUnit));
#pragma unroll
          for (int k = 0; k < 4; ++k) umma_bf16(tS, ad + 2 * k, bd + 2 * k, idN256, (c > 0 || k > 0) ? 1u : 0u);
          umma_commit(smem_u32(&empty[slot]));
          // the slot's next stage is stage c + 4 - NC of O += P_{j-1} V_{j-1}
          // (or, with a single key block, of O += P_0 V_0): P box 2 or 3 may go in
          if (c >= Cfg::NC - 2 && (j >= 1 || nkb == 1)) umma_commit(smem_u32(&pfree[c + 4 - Cfg::NC]));
          if (++slot == S) {
            slot = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        umma_commit(smem_u32(s_full));
      }
      if (j >= 1) {
        // O += P_{j-1} V_{j-1}: stage kc once P_{j-1} box kc (boxes 0 and 1
        // in the P buffer, 2 and 3 in the A part of the stage's slot) is
        // written and O rescaled
        const int jv = j - 1;
        for (int kc = 0; kc < 4 && ok; ++kc) {
          if (!mbar_wait_bounded(smem_u32(&p_full[kc]), jv & 1, args.err, kDevTimeoutAccum, lim) ||
              !mbar_wait_bounded(smem_u32(&full[slot]), phase, args.err, kDevTimeoutFull, lim)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = sdesc_k128(smem_u32(kc < 2 ? sP + kc * kFUnit : sR + slot * kSStage));
          const uint64_t bd = sdesc_k128(smem_u32(sR + slot * kSStage + kFUnit));
#pragma unroll
          for (int k = 0; k < 4; ++k)
            umma_bf16(tO, ad + 2 * k, bd + 2 * k, idN256, (jv > 0 || kc > 0 || k > 0) ? 1u : 0u);
          umma_commit(smem_u32(&empty[slot]));
          // with no S stages left, the slot's next stage is stage kc of O += P_{nkb-1} V_{nkb-1}
          if (j == nkb - 1 && kc >= 2) umma_commit(smem_u32(&pfree[kc]));
          if (++slot == S) {
            slot = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        umma_commit(smem_u32(pv_done));
      }
    }
    if (!ok) *abort_flag = 1;
    // every MMA of this CTA completes before the TMEM is released
    umma_commit(smem_u32(done));
    mbar_wait_bounded(smem_u32(done), 0, args.err, kDevTimeoutAccum, lim);
  } else if (warp >= 4) {
    // ------------------------------------------------------ softmax, output
    // warp w reads TMEM lane quadrant w % 4; quarter qt = (w - 4) / 4 of the
    // row takes keys 64 qt .. 64 qt + 63 of each block (P box qt) and output
    // columns 64 qt .. 64 qt + 63 of this CTA's 256.  The four quarters of a
    // row exchange their maxima and, at the end, their sums through shared
    // memory; all sixteen warps agree on every wait's outcome.
    const int q = warp & 3, qt = (warp - 4) >> 2;
    const int row = 32 * q + lane;
    const uint32_t lane_off = (uint32_t)(32 * q) << 16;
    const uint32_t tSq = tS + lane_off + 64 * qt, tOq = tO + lane_off + 64 * qt;
    const float sc = args.scale_log2;
    uint8_t* line_base = nullptr;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nkb; ++j) {
      ok = sm_all(!*abort_flag && mbar_wait_bounded(smem_u32(s_full), j & 1, args.err, kDevTimeoutAccum, lim));
      if (!ok) break;
      tc_fence_after();
      const int kv = args.HW - 256 * j - 64 * qt;  // keys of this quarter inside the frame
      // pass 1: the quarter-row max of the raw scores (the scale is positive)
      float mb = -INFINITY;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t r[16];
        tmem_ld16(tSq + 16 * c, r);
        tmem_ld_wait();
        if (kv >= 64) {
#pragma unroll
          for (int i = 0; i < 16; ++i) mb = fmaxf(mb, __uint_as_float(r[i]));
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if (16 * c + i < kv) mb = fmaxf(mb, __uint_as_float(r[i]));
        }
      }
      mb *= sc;
      // the row max over the four quarters: quarters 2 and 3 hand theirs to 0
      // and 1, which leave max(0, 2) and max(1, 3) for all to read
      if (qt >= 2) red[(qt - 2) * 128 + row] = mb;
      sm_sync();
      if (qt < 2) red[qt * 128 + row] = mb = fmaxf(mb, red[qt * 128 + row]);
      sm_sync();
      mb = fmaxf(red[row], red[128 + row]);
      float alpha = 1.f;
      if (mb > m + 8.f) {  // move the reference max (and rescale O and l by alpha)
        alpha = exp2f(m - mb);
        m = mb;
      }
      // pass 2: P in bf16 (registers), and the row sum of the rounded values
      uint32_t pk[32];
      float rs = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t r[16];
        tmem_ld16(tSq + 16 * c, r);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; i += 2) {
          float e0 = ex2_approx(fmaf(__uint_as_float(r[i]), sc, -m));
          float e1 = ex2_approx(fmaf(__uint_as_float(r[i + 1]), sc, -m));
          if (kv < 64) {
            if (16 * c + i >= kv) e0 = 0.f;
            if (16 * c + i + 1 >= kv) e1 = 0.f;
          }
          const uint32_t w = pack_bf16x2(e0, e1);
          rs += bf16_lo(w) + bf16_hi(w);
          pk[8 * c + i / 2] = w;
        }
      }
      tc_fence_before();
      mbar_arrive(smem_u32(s_free));
      l = l * alpha + rs;
      // O stable once O += P_{j-1} V_{j-1} has completed
      if (j > 0) {
        ok = sm_all(mbar_wait_bounded(smem_u32(pv_done), (j - 1) & 1, args.err, kDevTimeoutAccum, lim));
        if (!ok) break;
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            uint32_t r[16];
            tmem_ld16(tOq + 16 * c, r);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
            tmem_st16(tOq + 16 * c, r);
          }
          tmem_st_wait();
        }
      }
      // O is rescaled: the P V stages of the other quarters' boxes may go
      tc_fence_before();
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (k != qt) mbar_arrive(smem_u32(&p_full[k]));
      // P_j box qt: boxes 0 and 1 go to the P buffer (free: O += P_{j-1}
      // V_{j-1} has completed), boxes 2 and 3 to the A part of the slot of
      // their P V stage, free once pfree[qt] completes for the j-th time.
      // This wait is per thread, so that boxes 0 and 1 are not held up: a
      // thread whose wait runs out raises the abort flag and skips its box,
      // and all threads leave together at the next agreement.
      line_base = sP + qt * kFUnit;
      if (qt >= 2) {
        if (!mbar_wait_bounded(smem_u32(&pfree[qt]), j & 1, args.err, kDevTimeoutEmpty, lim)) {
          ok = false;
          *abort_flag = 1;
          continue;
        }
        line_base = sR + (split_pv_pos(j, nkb, Cfg::NC, qt) % S) * kSStage;
      }
      // in the 128-byte-swizzled K-major layout: row `row`, chunk g of 8 keys
      // at 16-byte slot g ^ (row & 7) of its 128-byte line
      uint8_t* line = line_base + row * 128;
#pragma unroll
      for (int g = 0; g < 8; ++g)
        *reinterpret_cast<uint4*>(line + ((g ^ (row & 7)) << 4)) =
            make_uint4(pk[4 * g], pk[4 * g + 1], pk[4 * g + 2], pk[4 * g + 3]);
      fence_proxy_async_smem();
      mbar_arrive(smem_u32(&p_full[qt]));
    }
    // every thread takes part (a thread that left the loop early has ok false)
    ok = sm_all(ok && !*abort_flag &&
                mbar_wait_bounded(smem_u32(pv_done), (nkb - 1) & 1, args.err, kDevTimeoutAccum, lim));
    if (!ok) {
      *abort_flag = 1;
    } else {
      tc_fence_after();
      // the row's weight sum: the four quarters' partial sums (taken against
      // the same max), combined as the maxima were
      if (qt >= 2) red[(qt - 2) * 128 + row] = l;
      sm_sync();
      if (qt < 2) red[qt * 128 + row] += l;
      sm_sync();
      const float rl = 1.f / (red[row] + red[128 + row]);
      const int qrow = 128 * qb + row;
      __nv_bfloat16* dst = args.out + (long long)b * args.out_bs + (long long)f * args.out_fs +
                           (long long)qrow * args.out_ldc + 256 * rank + 64 * qt;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t r[16];
        tmem_ld16(tOq + 16 * c, r);
        tmem_ld_wait();
        if (qrow < args.HW) {
          float v[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]) * rl;
          uint4* d = reinterpret_cast<uint4*>(dst + 16 * c);
          d[0] = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                            pack_bf16x2(v[6], v[7]));
          d[1] = make_uint4(pack_bf16x2(v[8], v[9]), pack_bf16x2(v[10], v[11]), pack_bf16x2(v[12], v[13]),
                            pack_bf16x2(v[14], v[15]));
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int NQ>
cudaError_t launch_f(const FlashLaunch& L, cudaStream_t stream) {
  using Cfg = FCfg<NQ>;
  auto kern = flash_attn_kernel<NQ>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cfg::kSmem);
  if (e != cudaSuccess) return e;
  const FlashArgs& a = L.args;
  if (a.HW <= 0 || a.frames <= 0 || a.batches <= 0) return cudaSuccess;
  dim3 grid((unsigned)((a.HW + 127) / 128), (unsigned)a.frames, (unsigned)a.batches);
  kern<<<grid, kFThreads, Cfg::kSmem, stream>>>(L.q, L.v, a);
  return cudaGetLastError();
}

template <int NSL>
cudaError_t launch_split(const FlashLaunch& L, cudaStream_t stream) {
  using Cfg = SCfg<NSL>;
  auto kern = flash_attn_split_kernel<NSL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cfg::kSmem);
  if (e != cudaSuccess) return e;
  const FlashArgs& a = L.args;
  if (a.HW <= 0 || a.frames <= 0 || a.batches <= 0) return cudaSuccess;
  dim3 grid((unsigned)(NSL * ((a.HW + 127) / 128)), (unsigned)a.frames, (unsigned)a.batches);
  kern<<<grid, kSThreads, Cfg::kSmem, stream>>>(L.q, L.k, L.v, a);
  return cudaGetLastError();
}

}  // namespace

bool flash_attn_supported(int C) { return C % 64 == 0 && C >= 64 && (C <= 384 || C == 512 || C == 1024); }

FlashBoxes flash_attn_boxes(int C) {
  if (C <= 384) return FlashBoxes{128, 128, C % 128 == 0 ? 128 : 64, 128};
  return FlashBoxes{128, 256, 256, 256};
}

double flash_attn_exec_ratio(int C) { return C <= 384 ? 1.0 : (C / 256 + 1) / 2.0; }

cudaError_t launch_flash_attn(const FlashLaunch& L, cudaStream_t stream) {
  const FlashArgs& a = L.args;
  if (!flash_attn_supported(a.C) || a.HW < 0) return cudaErrorInvalidValue;
  const int kb = flash_attn_boxes(a.C).key_block;
  if (a.nkb != (a.HW + kb - 1) / kb) return cudaErrorInvalidValue;
  switch (a.C / 64) {
    case 1: return launch_f<1>(L, stream);
    case 2: return launch_f<2>(L, stream);
    case 3: return launch_f<3>(L, stream);
    case 4: return launch_f<4>(L, stream);
    case 5: return launch_f<5>(L, stream);
    case 6: return launch_f<6>(L, stream);
    case 8: return launch_split<2>(L, stream);
    case 16: return launch_split<4>(L, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace wan
