// Launch descriptors shared by the host planner and the CUDA kernels.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace wan {

// ---------------------------------------------------------------------------
// Implicit-GEMM convolution on the 5th-generation tensor cores.
//
// Output tile: 128 positions (a box_w x box_h spatial rectangle of one output
// frame) x BN output channels.  The K loop walks a list of taps; each tap is
// one kernel offset (dt, dy, dx) of one A source, contributing nkb blocks of
// 64 input channels.  A tiles are TMA-loaded from a channels-last activation
// tensor [B][F][H][W][C] whose out-of-range coordinates read zero, which is
// the convolution's zero padding in space.  Frame coordinates index the
// tensor's frame slots directly: a causal conv's input tensor keeps its two
// history frames in slots 0-1 in front of the current frames.
// ---------------------------------------------------------------------------
constexpr int kMaxTaps = 96;
constexpr int kBandBoxRows = 10;  // band mode: A boxes of 16 x 10 positions (8 rows + 2 halo rows)
constexpr int kTileM = 128;
constexpr int kBlockK = 64;

struct ConvTap {
  int8_t src;     // A source: 0 or 1
  int8_t dt;      // frame offset added to the source frame base
  int8_t dy, dx;  // spatial offsets of the source position (kernel offset minus padding)
  int16_t a_c0;   // first channel of the tap in the A source
  int16_t nkb;    // 64-channel blocks
  int32_t b_k0;   // first K column of the tap in the B operand
};

enum EpiMode : int { kEpiStore = 0, kEpiDup = 1, kEpiVideo = 2 };

struct ConvArgs {
  ConvTap taps[kMaxTaps];
  int n_taps;
  int total_kb;
  // grid = tiles_n * tiles_x * tiles_y * frames * batches CTAs (n fastest)
  int tiles_n, tiles_x, tiles_y, frames, batches;
  int box_w, box_h;      // spatial tile, box_w * box_h == 128
  int H, W;              // output spatial size (equal to the A sources')
  int src_f0[2];         // frame coordinate of output frame 0 in each A source
  int src_fmod;          // > 0: source 0 is a circular ring of src_fmod frame slots (ring_slot)
  int b_per_frame;       // 1: B's third coordinate is b * b_gstride + output frame (batched GEMMs)
  int b_gstride;
  // Sub-pixel form of nearest-x2 + 3x3 conv: the grid carries a phase
  // p = 2i + j (i, j in {0, 1}) per tile; the taps' spatial offsets are
  // shifted by (i - 1, j - 1), B's third coordinate is p, and the output of
  // low-resolution position (y, x) goes to (2y + i, 2x + j) of a 2H x 2W frame.
  int subpix;
  // Row mode (3x3 spatial taps without a shortcut, N tile 96, 128 or 192): a tile
  // is 128 consecutive pixels of one row (box_w 128, box_h 1); every tap
  // (dt, dy) loads one 130-pixel A box (x from -1) that serves its three dx
  // taps at row offsets 0, 1, 2, and the three taps' B blocks, which lie
  // row_bdk K columns apart.  Cluster pairs are adjacent rows (ty).
  int row;
  int tail_k16;  // row mode: K16 steps holding channels in each tap's last block (0: all 4)
  int row_bdk;  // row mode: K stride between dx taps; band mode: between dy taps
  // Band mode (bf16 3x3 spatial taps without a shortcut, N tile 256, 16 x 8
  // tiles): every tap (dt, dx) loads one 16 x 10 A box (rows from -1) into an
  // A ring that serves its three dy taps at 2 KB offsets; the taps' one-tap
  // B blocks go through a separate ring.
  int band;
  int N;                 // valid output channels
  const float* bias;     // fp32, zero-padded to a multiple of 16 values past N, or null
  // output element (b, frame, y, x, n) at
  //   out + b*out_bs + (out_f0 + f*out_fmul + hi)*out_fs + (y*W + x)*out_ldc + n'
  // where, if interleave_c > 0, channels n >= interleave_c go to the next
  // frame (hi = 1) as n' = n - interleave_c.
  void* out;
  int out_f32;
  long long out_bs, out_fs;
  int out_ldc, out_f0, out_fmul, interleave_c;
  // Split format (fp32 decode): a value v is stored as bf16 hi = bf16(v) at
  // channel n and bf16 lo = bf16(v - hi) at channel n + *_lo; 0 = plain.
  int out_lo, res_lo, dup_lo;
  // kEpiStore: optional residual added at the same (b, y, x, n), frame res_f0 + f
  const void* res;
  int res_f32;
  long long res_bs, res_fs;
  int res_ldc, res_f0;
  // kEpiDup: DupUp3D of a half-resolution source, added to the output
  const void* dup;
  long long dup_bs, dup_fs;
  int dup_ldc, dup_W;
  int dup_ft;            // frames per source frame (2 with temporal upsampling, else 1)
  int dup_first;         // first chunk: the first ft-1 copies of frame 0 are dropped
  int dup_pairs;         // 1: channel c reads source 2c + (row & 1) (r = 2); 0: channel c (r = 4ft)
  // kEpiVideo: out = video [B][3][F][2H][2W]; channel 4k + 2j + i -> colour k,
  // row 2y + i, column 2x + j (vid_patch 2); or video [B][3][F][H][W] from
  // channels 0..2 (vid_patch 1); clamped to [-1, 1]; preclamp is the fp32
  // copy before the clamp (optional).
  float* preclamp;
  long long vid_bs, vid_cs;
  int vid_patch;
  // Fused RMS norm (requires one N tile holding all N channels): y = acc +
  // bias (+ residual) is also written normalised over its N channels,
  // y / max(||y||, 1e-12) * norm_gs (then SiLU if norm_silu), to out2 at
  // (b, out2_f0 + f, position); `out` may be null (only the normalised y).
  const float* norm_gs;
  int norm_silu;
  void* out2;
  long long out2_bs, out2_fs;
  int out2_ldc, out2_f0, out2_lo;
  int out2_fmod;         // > 0: out2 is a circular ring of out2_fmod frame slots
  int* err;              // device error word (kDev* codes)
  // Failure-detection self test: a bounded wait gives up after wait_limit
  // SM clocks (0: the default of about 2 s), and the TMA producer withholds
  // the loads of its K iteration number stall_at1 - 1 (0: none), so the MMA
  // issuer's wait for that stage runs out.
  long long wait_limit;
  int stall_at1;
};

struct ConvLaunch {
  CUtensorMap a0, a1, b;
  ConvArgs args;
  int bn;      // 16, 32, 64, 96, 128, 192 or 256 (96 and 192: plain store epilogue only)
  int epi;     // EpiMode
};

cudaError_t launch_conv(const ConvLaunch& L, cudaStream_t stream);
// Rows of the B tensor map's box for an N tile of bn (half of it when a
// cluster of two CTAs shares the B block).
int conv_b_box_rows(int bn);

// ---------------------------------------------------------------------------
// conv_out with the spatial taps folded into N (conv_out.cu): a causal
// 3x3x3 conv of a ring [B][F slots][H][W][ldc] (bf16) to COUT = 12 channels
// (unpatchified 2 x 2, vid_patch 2) or 3 colours (vid_patch 1), clamped into
// the NCDHW video.  One tile = a 16 x 16 box of input positions whose 14 x 14
// interior it outputs.  B = tap-folded weights [N = video_conv_n(cout)][K =
// 3 * ci_pad], row (3 dy + dx) * cout + co, column dt * ci_pad + ci.
// ---------------------------------------------------------------------------
struct VideoConvArgs {
  int H, W;                       // frame size
  int frames, batches;            // output frames, batch
  int tiles_x, tiles_y;           // ceil(W / 14), ceil(H / 14)
  int src_f0;                     // ring slot read by output frame 0 at time tap 0
  int src_fmod;                   // ring slots (circular ring; 0: a plain tensor)
  int ci_pad, nkb;                // channels per time tap (64 nkb)
  int tail_k16;                   // K16 steps holding channels in the last block (0: all 4)
  int cout;                       // 12 or 3
  const float* bias;              // fp32, cout values
  void* out;                      // video [B][3][F][vid_patch H][vid_patch W]
  int out_f32, out_f0, vid_patch;
  long long vid_bs, vid_cs;       // batch and colour strides (elements)
  float* preclamp;                // optional fp32 copy before the clamp
  int* err;                       // device error word (kDev* codes)
  long long wait_limit;           // bounded waits: SM clocks (0: about 2 s)
  int stall_at1;                  // failure injection (0: none)
};
struct VideoConvLaunch {
  CUtensorMap a, b;  // A box 64 x 16 x 16 x 1 x 1; B box 64 x N x 1
  VideoConvArgs args;
};
int video_conv_n(int cout);
cudaError_t launch_video_conv(const VideoConvLaunch& L, cudaStream_t stream);
// src [Co][Ci][3][3][3] (fp32 or bf16) -> dst[(3 dy + dx) * Co + co][dt * ci_pad + ci] bf16
// (rows past 9 Co and channels past Ci are left as they are).
cudaError_t launch_pack_tapfold(const void* src, int src_f32, int Co, int Ci, int ci_pad, __nv_bfloat16* dst,
                                cudaStream_t s);

// ---------------------------------------------------------------------------
// Flash-style attention core (attention.cu): per frame, O = softmax(q k^T *
// scale) v over HW positions, head dim C (a multiple of 64).  q and k are
// channel ranges of one tensor [B][F][HW][ldc] (maps q and k: 4-D (channels,
// HW, F, B)); v comes transposed, [B][F][C][HWp] with zeros past HW (map v:
// 4-D (HWp, C, F, B)).  O is written as bf16 [B][F][HW][out_ldc].  Two
// kernels: C <= 384 keeps S and all of O in one CTA's TMEM; C = 512 or 1024
// runs C / 256 CTAs per 128 queries, CTA r accumulating output columns
// [256 r, 256 r + 256) and each computing the full scores itself.
// flash_attn_boxes gives the box of each map and the key block.
// ---------------------------------------------------------------------------
struct FlashArgs {
  int HW, frames, batches;
  int nkb;             // key blocks: ceil(HW / key_block)
  int C;               // head dim
  int q_c0, k_c0;      // first channel of q and of k in the qk tensor
  float scale_log2;    // log2(e) / sqrt(C)
  __nv_bfloat16* out;
  long long out_bs, out_fs;
  int out_ldc;
  int* err;
  long long wait_limit;
  int stall_at1;       // failure self test: 1-based ring stage the producer never loads (0: none)
};
struct FlashLaunch {
  CUtensorMap q, k, v;
  FlashArgs args;
};
struct FlashBoxes {
  int q_rows, k_rows;  // rows of the q and k boxes (64 channels wide)
  int v_rows;          // rows (channels) of the v^T box (64 keys wide)
  int key_block;       // keys per score block
};
// false if no flash kernel takes head dim C
bool flash_attn_supported(int C);
FlashBoxes flash_attn_boxes(int C);
// tcgen05 work per nominal FLOP (the split kernel recomputes the scores in
// each CTA of its cluster: (C / 256 + 1) / 2)
double flash_attn_exec_ratio(int C);
cudaError_t launch_flash_attn(const FlashLaunch& L, cudaStream_t stream);

// ---------------------------------------------------------------------------
// Memory-bound kernels (channels-last bf16 unless stated).
// A "frame view" addresses element (b, f, p, c) of a tensor as
//   base + b*bs + (f0 + f)*fs + p*ldc + c.
// ---------------------------------------------------------------------------
// With fmod > 0 the tensor is a circular ring of fmod frame slots: frame
// f0 + f lives in slot (f0 + f) mod fmod (f0 < fmod, f < fmod).
struct FrameView {
  void* base;
  long long bs, fs;
  int ldc, f0;
  int fmod;
};
__host__ __device__ __forceinline__ int ring_slot(int f, int fmod) { return (fmod > 0 && f >= fmod) ? f - fmod : f; }

// y = x / max(||x||, 1e-12) * gs (gs = sqrt(C)*gamma, fp32), then SiLU if silu.
// in_lo / out_lo: split-format offsets of the low halves (0 = plain bf16).
cudaError_t launch_rms_norm(FrameView in, FrameView out, const float* gs, int C, int B, int F, int P, bool silu,
                            cudaStream_t s, int in_lo = 0, int out_lo = 0);
// copy F frames of C channels
cudaError_t launch_copy_frames(FrameView in, FrameView out, int C, int B, int F, int P, cudaStream_t s);
// post_quant_conv: z [B][Z][Tz][h][w] (fp32 or bf16, NCDHW), frames t0..t0+F-1
// -> out(b, f, p, 0..Z-1) bf16; channels Z..ldc-1 are left as they are (zero).
// zstat: NULL, or mean[Z] then std[Z] (fp32): the latents are first
// de-normalised to z * std + mean (before the bf16 rounding of round_z_bf16).
cudaError_t launch_post_quant(const void* z, int z_f32, int Z /*48 or 16*/, int B, int Tz, int t0, int F, int P,
                              const float* w /*Z x Z*/,
                              const float* bias, const float* zstat, FrameView out, int round_z_bf16, cudaStream_t s,
                              int out_lo = 0);
// Row softmax of S [R][ld_s] fp32 (n valid columns) scaled by `scale`, into
// P [R][ld_p] bf16.
cudaError_t launch_softmax_rows(const float* S, long long ld_s, __nv_bfloat16* P, long long ld_p, int n, long long R,
                                float scale, cudaStream_t s, int p_lo = 0);
// Vt[g][c][p] = src[g][p][c] (bf16), p < P, c < C; src row stride ld_src.
cudaError_t launch_transpose(const __nv_bfloat16* src, long long src_gs, int ld_src, __nv_bfloat16* dst,
                             long long dst_gs, int ld_dst, int G, int P, int C, cudaStream_t s);
// Weight packing: src [Co][Ci][taps] (fp32 or bf16, taps = kt*kh*kw) ->
// dst[co][k0 + tap*ci_pad + ci] bf16 for co < Co, ci < Ci; dst has ld columns.
// lo = 1 packs the low half bf16(w - bf16(w)) of the split format instead.
cudaError_t launch_pack_weight(const void* src, int src_f32, int Co, int Ci, int taps, __nv_bfloat16* dst, int ld,
                               int k0, int ci_pad, cudaStream_t s, int lo = 0);
// Sub-pixel weights of nearest-x2 + 3x3 conv: src [Co][Ci][3][3] ->
// dst[p][co][k0 + (2a + b)*tap_stride + ci] = sum of src[co][ci][dy][dx] over the
// kernel rows dy that land on source row offset a for output row phase i
// (i = 0: {0} | {1, 2}; i = 1: {0, 1} | {2}) and likewise columns dx for phase
// j, p = 2i + j.  round_src rounds each weight to bf16 before the sum; lo
// packs the low half of the split format.  dst has ld columns and co_pad rows
// per phase.
cudaError_t launch_pack_subpixel(const void* src, int src_f32, int Co, int Ci, __nv_bfloat16* dst, int ld, int co_pad,
                                 int k0, int tap_stride, int round_src, int lo, cudaStream_t s);
// dst[i] = scale * r(src[i]) (+ r(src2[i]) if src2) as fp32; src fp32 or bf16;
// r rounds to the nearest bf16 when round_bf16 is set.
cudaError_t launch_to_f32(const void* src, int src_f32, const void* src2, int src2_f32, float* dst, int n,
                          float scale, int round_bf16, cudaStream_t s);

// ---------------------------------------------------------------------------
// Tiled decode (tiled.cu).  Decoded tiles are fp32 [B][3][F][h][w] each, at
// element offset `off` of one buffer; the table lists them in raster order.
// Passed by value as kernel parameters (kept under the 32 KB limit).
// ---------------------------------------------------------------------------
struct TileDesc {
  long long off;  // element offset of the tile in the buffer (a multiple of 4)
  int h, w;       // pixels (multiples of 8)
};
constexpr int kMaxTiles = 1024;
struct TileTable {
  int ni, nj;  // tile rows and columns
  int sh, sw;  // stride in pixels: tile (i, j) starts at (i*sh, j*sw)
  TileDesc t[kMaxTiles];
};
// One batch of latent tiles of equal size: zt[(k*B + b)][c][t][y][x] =
// z[b][c][t][r0[k] + y][c0[k] + x], CT = 48 * T.
constexpr int kMaxGather = 64;
struct TileGather {
  int n, B, h, w, th, tw;
  long long CT;
  int r0[kMaxGather], c0[kMaxGather];
};
// elem_bytes: 4 (fp32) or 2 (bf16), copied as is.
cudaError_t launch_gather_tiles(const void* z, int elem_bytes, void* zt, const TileGather& g, cudaStream_t s);
// Seam blending in place, one launch per anti-diagonal of tiles; planes =
// B * 3 * F.
cudaError_t launch_blend_tiles(float* buf, const TileTable& tab, long long planes, cudaStream_t s);
// out [planes][H][W] (fp32 or bf16) from the blended tiles.
cudaError_t launch_assemble_tiles(const float* buf, const TileTable& tab, void* out, int out_f32, long long planes,
                                  int H, int W, cudaStream_t s);

}  // namespace wan
