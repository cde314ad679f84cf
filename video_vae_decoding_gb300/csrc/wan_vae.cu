// Host side of the decode: the C ABI of include/wan_vae.h, weight packing,
// the per-chunk launch sequence and the causal-cache ring buffers.
//
// The sequence follows the page "wan22_vae_decode/reference.py", module
// docstring "What is computed" (post_quant_conv; conv_in; mid block; up
// blocks 0-3; norm_out, SiLU, conv_out; unpatchify; clamp), sections
// "The first latent frame yields one frame" and "Causal caches".  A chunk of
// n latent frames runs every layer over all of its frames at once (the
// whole-sequence form of section "Causal caches" restricted to the chunk),
// the 3-frame causal convs reading their two history frames from the front
// slots of a per-conv ring buffer.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <memory>
#include <mutex>
#include <string>
#include <vector>

#include "kernels.h"
#include "wan_vae.h"

using bf16 = __nv_bfloat16;

namespace wan {

thread_local std::string g_last_error;

static wan_status fail(wan_status s, const char* fmt, ...) {
  char buf[1024];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

#define CUDA_TRY(expr)                                                                                     \
  do {                                                                                                     \
    cudaError_t e_ = (expr);                                                                               \
    if (e_ != cudaSuccess)                                                                                 \
      return ::wan::fail(e_ == cudaErrorMemoryAllocation ? WAN_ERR_OOM : WAN_ERR_CUDA, "%s: %s (%s:%d)", #expr, \
                         cudaGetErrorString(e_), __FILE__, __LINE__);                                      \
  } while (0)
#define WAN_TRY(expr)                 \
  do {                                \
    wan_status s_ = (expr);           \
    if (s_ != WAN_OK) return s_;      \
  } while (0)

static inline long long rup(long long a, long long b) { return (a + b - 1) / b * b; }
static inline long long cdiv(long long a, long long b) { return (a + b - 1) / b; }

// ------------------------------------------------------------- tensor maps
static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

static wan_status init_encode() {
  static std::once_flag once;
  static cudaError_t err = cudaSuccess;
  std::call_once(once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (err == cudaSuccess && q == cudaDriverEntryPointSuccess) g_encode = (PFN_cuTensorMapEncodeTiled_v12000)fn;
  });
  if (!g_encode) return fail(WAN_ERR_CUDA, "cuTensorMapEncodeTiled unavailable (%s)", cudaGetErrorString(err));
  return WAN_OK;
}

static wan_status encode(CUtensorMap* m, int rank, const void* base, const uint64_t* dims, const uint64_t* strides,
                         const uint32_t* box) {
  WAN_TRY(init_encode());
  const uint32_t es[5] = {1, 1, 1, 1, 1};
  const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void*>(base), dims,
                              strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(WAN_ERR_INTERNAL, "cuTensorMapEncodeTiled failed (%d), rank %d", (int)r, rank);
  return WAN_OK;
}

// Channels-last bf16 activation tensor [B][F][H][W][ldc]; channels C..ldc-1
// hold zeros.  ldc is a multiple of 64 for tensors that feed the tensor cores.
// A causal conv's ring is circular (fmod = F slots): its logical frame f
// (0, 1 the history, 2.. the chunk's frames) lives in slot (base + f) mod F,
// and after a chunk of n frames base advances by n, so the chunk's last two
// frames become the next chunk's history without being copied.
struct Act {
  bf16* p = nullptr;
  int B = 0, F = 0, H = 0, W = 0, C = 0, ldc = 0;
  int lo = 0;  // split format: low halves at channel offset lo (0: plain bf16)
  int fmod = 0, base = 0;  // circular ring: F slots, logical frame 0 at slot `base`
  // ring: leading logical frames known to hold zeros (the history after a
  // reset: 2); a causal conv skips the taps that would read them
  int zhist = 0;
  int chans() const { return lo ? ldc : C; }  // channels a copy must move
  long long fs() const { return (long long)H * W * ldc; }
  long long bs() const { return (long long)F * fs(); }
  size_t bytes() const { return (size_t)B * bs() * sizeof(bf16); }
  int slot(int f) const { return fmod ? (base + f) % fmod : f; }  // physical slot of logical frame f
  FrameView view(int f0 = 0) const { return FrameView{p, bs(), fs(), ldc, slot(f0), fmod}; }
};

// A-operand map over an activation tensor: dims (C, W, H, F, B), box
// (64, bw, bh, 1, 1).
static wan_status act_map(CUtensorMap* m, const bf16* base, int C, int ldc, int W, int H, int F, int B, long long fs,
                          long long bs, int bw, int bh) {
  const uint64_t dims[5] = {(uint64_t)C, (uint64_t)W, (uint64_t)H, (uint64_t)F, (uint64_t)B};
  const uint64_t strides[4] = {(uint64_t)ldc * 2, (uint64_t)W * ldc * 2, (uint64_t)fs * 2, (uint64_t)bs * 2};
  const uint32_t box[5] = {64, (uint32_t)bw, (uint32_t)bh, 1, 1};
  return encode(m, 5, base, dims, strides, box);
}
// The channel extent is the tensor's own channel count (the split format's
// whole row): a 64-channel block reaching into the padding up to ldc reads
// TMA zero fill there instead of fetching the zeros from memory.
static wan_status act_map(CUtensorMap* m, const Act& a, int bw = 16, int bh = 8) {
  return act_map(m, a.p, a.chans(), a.ldc, a.W, a.H, a.F, a.B, a.fs(), a.bs(), bw, bh);
}
// B-operand map for an N tile of bn: dims (K, N, G), box (64, rows, 1) with
// rows = bn, or bn / 2 when two CTAs of a cluster each load half of the tile.
static wan_status b_map(CUtensorMap* m, const bf16* base, long long K, long long N, long long G, long long ldk,
                        long long gs, int bn) {
  const uint64_t dims[3] = {(uint64_t)K, (uint64_t)N, (uint64_t)G};
  const uint64_t strides[2] = {(uint64_t)ldk * 2, (uint64_t)gs * 2};
  const uint32_t box[3] = {64, (uint32_t)conv_b_box_rows(bn), 1};
  return encode(m, 3, base, dims, strides, box);
}

// -------------------------------------------------------------- allocation
struct DevMem {
  std::vector<void*> ptrs;
  cudaStream_t async = nullptr;  // stream-ordered allocations when set
  bool use_async = false;
  bool dry = false;              // validation pass: check names and shapes only
  wan_status alloc(void** p, size_t bytes) {
    *p = nullptr;
    if (bytes == 0) bytes = 256;
    const cudaError_t e = use_async ? cudaMallocAsync(p, bytes, async) : cudaMalloc(p, bytes);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return fail(e == cudaErrorMemoryAllocation ? WAN_ERR_OOM : WAN_ERR_CUDA, "device allocation of %zu bytes: %s",
                  bytes, cudaGetErrorString(e));
    }
    ptrs.push_back(*p);
    return WAN_OK;
  }
  void release() {
    for (void* p : ptrs) use_async ? cudaFreeAsync(p, async) : cudaFree(p);
    ptrs.clear();
  }
};

// ----------------------------------------------------------- profiling
// Kinds of tensor-core launches, for the per-kind breakdown.
enum LaunchKind {
  kKindConv333 = 0,
  kKindTimeConv = 1,
  kKindResample = 2,
  kKindAttention = 3,
  kKindConvOut = 4,
  kKindNorm = 5,  // memory-bound kinds record algorithmic bytes instead of FLOPs
  kKindMisc = 6,
  kNumKinds = 7
};
struct ProfRec {
  int kind;
  double work;  // nominal FLOPs (tensor-core kinds) or algorithmic bytes
  double exec;  // FLOPs of the arithmetic the kernels actually run (sub-pixel form: 4/9 of nominal)
};
struct Prof {
  bool on = false;
  long long launches = 0;     // every kernel launch enqueued
  std::vector<cudaEvent_t> ev;  // start/end pairs of timed launches
  std::vector<ProfRec> rec;     // one per timed launch
  ~Prof() {
    for (cudaEvent_t e : ev) cudaEventDestroy(e);
  }
  // Events of the next timed launch (null when not profiling); exec < 0
  // means "as nominal".
  wan_status begin(int kind, double work, cudaStream_t s, cudaEvent_t* e1, double exec = -1.0) {
    *e1 = nullptr;
    if (!on) return WAN_OK;
    const size_t i = rec.size();
    while (ev.size() < 2 * (i + 1)) {
      cudaEvent_t e;
      CUDA_TRY(cudaEventCreate(&e));
      ev.push_back(e);
    }
    rec.push_back({kind, work, exec < 0 ? work : exec});
    *e1 = ev[2 * i + 1];
    CUDA_TRY(cudaEventRecord(ev[2 * i], s));
    return WAN_OK;
  }
};
// A memory-bound launch, timed when profiling, with its algorithmic bytes.
#define ELT(prof, kind, bytes, expr)                                   \
  do {                                                                 \
    Prof* p_ = (prof);                                                 \
    cudaEvent_t e1_ = nullptr;                                         \
    if (p_) WAN_TRY(p_->begin((kind), (double)(bytes), s, &e1_));      \
    CUDA_TRY(expr);                                                    \
    if (e1_) CUDA_TRY(cudaEventRecord(e1_, s));                        \
    if (p_) p_->launches++;                                            \
  } while (0)

// ------------------------------------------------------------ packed convs
struct ConvW {
  bf16* w = nullptr;      // [co_pad][ktot], K = tap-major, 64-padded channel blocks per tap
  float* bias = nullptr;  // [Co] (conv bias + shortcut bias)
  int Co = 0, Ci = 0, kt = 1, kh = 1, kw = 1;
  int ci_pad = 0, ktot = 0, co_pad = 0, bn = 0;
  int sc_Ci = 0, sc_ci_pad = 0;  // appended 1x1x1 shortcut conv
  int split = 0;                 // hi/lo weight halves per tap (fp32 decode)
  int subpix = 0;                // 4 phases of 2x2 taps (nearest-x2 + 3x3 conv)
};

// N tile of a conv with co output channels: 256, or 192 where that divides
// co and 256 does not (384, 1152: the Wan2.1 widths); up to 256 channels one
// tile holding them all (96 and 192 exactly, else the next power of two).
static int choose_bn(int co) {
  if (co > 256) return (co % 256 != 0 && co % 192 == 0) ? 192 : 256;
  if (co == 96 || co == 192) return co;
  int b = 16;
  while (b < co) b *= 2;
  return b;
}

struct WeightTable {
  const wan_tensor* t;
  int n;
  const wan_tensor* find(const std::string& name) const {
    for (int i = 0; i < n; ++i)
      if (t[i].name && name == t[i].name) return &t[i];
    return nullptr;
  }
};

static wan_status get_tensor(const WeightTable& wt, const std::string& name, const wan_tensor** out) {
  const wan_tensor* x = wt.find(name);
  if (!x) return fail(WAN_ERR_MISSING_WEIGHT, "missing weight '%s'", name.c_str());
  if (x->dtype != WAN_F32 && x->dtype != WAN_BF16)
    return fail(WAN_ERR_DTYPE, "weight '%s': dtype %d is neither WAN_F32 nor WAN_BF16", name.c_str(), x->dtype);
  if (!x->data) return fail(WAN_ERR_INVALID_ARG, "weight '%s': null data", name.c_str());
  if (x->ndim < 1 || x->ndim > 5) return fail(WAN_ERR_SHAPE, "weight '%s': ndim %d", name.c_str(), x->ndim);
  *out = x;
  return WAN_OK;
}

static long long numel(const wan_tensor* t) {
  long long n = 1;
  for (int i = 0; i < t->ndim; ++i) n *= t->shape[i];
  return n;
}

static wan_status check_shape(const wan_tensor* t, std::vector<long long> want) {
  bool ok = t->ndim == (int)want.size();
  for (int i = 0; ok && i < t->ndim; ++i) ok = t->shape[i] == want[i];
  if (!ok) {
    std::string got, exp;
    for (int i = 0; i < t->ndim; ++i) got += std::to_string(t->shape[i]) + (i + 1 < t->ndim ? "," : "");
    for (size_t i = 0; i < want.size(); ++i) exp += std::to_string(want[i]) + (i + 1 < want.size() ? "," : "");
    return fail(WAN_ERR_SHAPE, "weight '%s': shape [%s], expected [%s]", t->name, got.c_str(), exp.c_str());
  }
  return WAN_OK;
}

// Packs `name` (conv3d [Co,Ci,kt,kh,kw] or conv2d [Co,Ci,kh,kw]) and, if
// given, a 1x1x1 shortcut conv appended along K.
// Split mode (fp32 decode): each tap holds the weights' bf16 high halves
// followed by their low halves, K = taps * 2 * ci_pad (+ 2 * sc_ci_pad).
static wan_status pack_conv(const WeightTable& wt, const std::string& name, int Co, int Ci, int kt, int kh, int kw,
                            bool conv2d, const std::string& sc_name, int sc_Ci, ConvW& cw, DevMem& mem,
                            cudaStream_t s, bool split = false) {
  const wan_tensor *W, *Bi;
  WAN_TRY(get_tensor(wt, name + ".weight", &W));
  WAN_TRY(get_tensor(wt, name + ".bias", &Bi));
  if (conv2d)
    WAN_TRY(check_shape(W, {Co, Ci, kh, kw}));
  else
    WAN_TRY(check_shape(W, {Co, Ci, kt, kh, kw}));
  WAN_TRY(check_shape(Bi, {Co}));
  const wan_tensor *Ws = nullptr, *Bs = nullptr;
  if (!sc_name.empty()) {
    WAN_TRY(get_tensor(wt, sc_name + ".weight", &Ws));
    WAN_TRY(get_tensor(wt, sc_name + ".bias", &Bs));
    WAN_TRY(check_shape(Ws, {Co, sc_Ci, 1, 1, 1}));
    WAN_TRY(check_shape(Bs, {Co}));
  }
  if (mem.dry) return WAN_OK;
  cw.Co = Co;
  cw.Ci = Ci;
  cw.kt = kt;
  cw.kh = kh;
  cw.kw = kw;
  cw.ci_pad = (int)rup(Ci, 64);
  cw.sc_Ci = Ws ? sc_Ci : 0;
  cw.sc_ci_pad = Ws ? (int)rup(sc_Ci, 64) : 0;
  const int taps = kt * kh * kw;
  const int sp = split ? 2 : 1;
  cw.split = split ? 1 : 0;
  cw.ktot = sp * (taps * cw.ci_pad + cw.sc_ci_pad);
  cw.bn = choose_bn(Co);
  cw.co_pad = (int)rup(Co, cw.bn);
  void* p;
  WAN_TRY(mem.alloc(&p, (size_t)cw.co_pad * cw.ktot * sizeof(bf16)));
  cw.w = (bf16*)p;
  CUDA_TRY(cudaMemsetAsync(cw.w, 0, (size_t)cw.co_pad * cw.ktot * sizeof(bf16), s));
  for (int part = 0; part < sp; ++part) {
    CUDA_TRY(launch_pack_weight(W->data, W->dtype == WAN_F32, Co, Ci, taps, cw.w, cw.ktot, part * cw.ci_pad,
                                sp * cw.ci_pad, s, part));
    if (Ws)
      CUDA_TRY(launch_pack_weight(Ws->data, Ws->dtype == WAN_F32, Co, sc_Ci, 1, cw.w, cw.ktot,
                                  sp * taps * cw.ci_pad + part * cw.sc_ci_pad, cw.sc_ci_pad, s, part));
  }
  WAN_TRY(mem.alloc(&p, (size_t)cw.co_pad * sizeof(float)));  // zero-padded to the N tile
  cw.bias = (float*)p;
  CUDA_TRY(cudaMemsetAsync(cw.bias, 0, (size_t)cw.co_pad * sizeof(float), s));
  CUDA_TRY(launch_to_f32(Bi->data, Bi->dtype == WAN_F32, Bs ? Bs->data : nullptr, Bs ? Bs->dtype == WAN_F32 : 0,
                         cw.bias, Co, 1.0f, split ? 0 : 1, s));
  return WAN_OK;
}

// sqrt(C) * gamma in fp32
static wan_status pack_gamma(const WeightTable& wt, const std::string& name, int C, float** out, DevMem& mem,
                             cudaStream_t s, bool split = false) {
  const wan_tensor* g;
  WAN_TRY(get_tensor(wt, name, &g));
  if (numel(g) != C) return fail(WAN_ERR_SHAPE, "weight '%s': %lld values, expected %d", name.c_str(), numel(g), C);
  if (mem.dry) return WAN_OK;
  void* p;
  WAN_TRY(mem.alloc(&p, (size_t)C * sizeof(float)));
  *out = (float*)p;
  CUDA_TRY(launch_to_f32(g->data, g->dtype == WAN_F32, nullptr, 0, *out, C, std::sqrt((float)C), split ? 0 : 1, s));
  return WAN_OK;
}

// upsample2d's 3x3 conv (conv2d [C, C, 3, 3]) on the nearest-x2 input, in
// its sub-pixel form: four 2x2 convs on the low-resolution input, one per
// output phase (row parity i, column parity j), whose weights sum the 3x3
// taps that read the same source pixel (page "The parts", fifth bullet: the
// upsampling only copies values, so the conv of the copies is the conv of
// the source with the taps merged).  K per phase = 4 taps * ci_pad (x2 split).
static wan_status pack_subpix_conv(const WeightTable& wt, const std::string& name, int C, int Co, ConvW& cw,
                                   DevMem& mem, cudaStream_t s, bool split) {
  const wan_tensor *W, *Bi;
  WAN_TRY(get_tensor(wt, name + ".weight", &W));
  WAN_TRY(get_tensor(wt, name + ".bias", &Bi));
  WAN_TRY(check_shape(W, {Co, C, 3, 3}));
  WAN_TRY(check_shape(Bi, {Co}));
  if (mem.dry) return WAN_OK;
  const int sp = split ? 2 : 1;
  cw.Co = Co;
  cw.Ci = C;
  cw.kt = 1;
  cw.kh = 2;
  cw.kw = 2;
  cw.subpix = 1;
  cw.split = split ? 1 : 0;
  cw.ci_pad = (int)rup(C, 64);
  cw.ktot = sp * 4 * cw.ci_pad;
  cw.bn = choose_bn(Co);
  cw.co_pad = (int)rup(Co, cw.bn);
  void* p;
  const size_t bytes = (size_t)4 * cw.co_pad * cw.ktot * sizeof(bf16);
  WAN_TRY(mem.alloc(&p, bytes));
  cw.w = (bf16*)p;
  CUDA_TRY(cudaMemsetAsync(cw.w, 0, bytes, s));
  for (int part = 0; part < sp; ++part)
    CUDA_TRY(launch_pack_subpixel(W->data, W->dtype == WAN_F32, Co, C, cw.w, cw.ktot, cw.co_pad, part * cw.ci_pad,
                                  sp * cw.ci_pad, split ? 0 : 1, part, s));
  WAN_TRY(mem.alloc(&p, (size_t)cw.co_pad * sizeof(float)));  // zero-padded to the N tile
  cw.bias = (float*)p;
  CUDA_TRY(cudaMemsetAsync(cw.bias, 0, (size_t)cw.co_pad * sizeof(float), s));
  CUDA_TRY(launch_to_f32(Bi->data, Bi->dtype == WAN_F32, nullptr, 0, cw.bias, Co, 1.0f, split ? 0 : 1, s));
  return WAN_OK;
}

// conv_out packed for the tap-folded kernel: [n][3 * ci_pad] bf16, row
// (3 dy + dx) * Co + co, column dt * ci_pad + ci (zero elsewhere).
struct TapFoldW {
  bf16* w = nullptr;
  int n = 0, ci_pad = 0, Co = 0, Ci = 0;
};
static wan_status pack_tapfold(const WeightTable& wt, const std::string& name, int Co, int Ci, TapFoldW& tf,
                               DevMem& mem, cudaStream_t s) {
  const wan_tensor* W;
  WAN_TRY(get_tensor(wt, name + ".weight", &W));
  WAN_TRY(check_shape(W, {Co, Ci, 3, 3, 3}));
  if (mem.dry) return WAN_OK;
  tf.Co = Co;
  tf.Ci = Ci;
  tf.ci_pad = (int)rup(Ci, 64);
  tf.n = video_conv_n(Co);
  const size_t bytes = (size_t)tf.n * 3 * tf.ci_pad * sizeof(bf16);
  void* p;
  WAN_TRY(mem.alloc(&p, bytes));
  tf.w = (bf16*)p;
  CUDA_TRY(cudaMemsetAsync(tf.w, 0, bytes, s));
  CUDA_TRY(launch_pack_tapfold(W->data, W->dtype == WAN_F32, Co, Ci, tf.ci_pad, tf.w, s));
  return WAN_OK;
}

// The tap-folded conv_out over F frames of `ring` (output frame f reads
// slots f, f + 1, f + 2) into the video: 16 x 16 input boxes, 14 x 14
// outputs each.
static wan_status video_conv_setup(const TapFoldW& tf, const float* bias, const Act& ring, int F, int patch,
                                   VideoConvLaunch& V) {
  memset(&V, 0, sizeof(V));
  if (ring.lo || ring.ldc < tf.ci_pad) return fail(WAN_ERR_INTERNAL, "tap-folded conv_out on a split or narrow ring");
  WAN_TRY(act_map(&V.a, ring, 16, 16));
  const uint64_t dims[3] = {(uint64_t)3 * tf.ci_pad, (uint64_t)tf.n, 1};
  const uint64_t strides[2] = {(uint64_t)3 * tf.ci_pad * 2, (uint64_t)3 * tf.ci_pad * tf.n * 2};
  const uint32_t box[3] = {64, (uint32_t)tf.n, 1};
  WAN_TRY(encode(&V.b, 3, tf.w, dims, strides, box));
  VideoConvArgs& a = V.args;
  a.H = ring.H;
  a.W = ring.W;
  a.frames = F;
  a.batches = ring.B;
  a.tiles_x = (int)cdiv(ring.W, 14);
  a.tiles_y = (int)cdiv(ring.H, 14);
  a.src_f0 = ring.slot(0);
  a.src_fmod = ring.fmod;
  a.ci_pad = tf.ci_pad;
  a.nkb = tf.ci_pad / 64;
  // the last 64-channel block of 96 (160, ...) channels holds 32 of them
  a.tail_k16 = (tf.Ci % 64 == 32 && ring.chans() == tf.Ci) ? 2 : 0;
  a.cout = tf.Co;
  a.bias = bias;
  a.vid_patch = patch;
  return WAN_OK;
}

}  // namespace wan

using namespace wan;

struct Resnet {
  ConvW c1, c2;  // c2 carries the shortcut when ci != co
  float* g1 = nullptr;
  float* g2 = nullptr;
  int ci = 0, co = 0;
};

struct wan_vae_model {
  int base = 0, dtype = WAN_BF16;
  // decoder variant: TI2V-5B (z 48, 2x2 patch, DupUp3D shortcuts, resamplers
  // keep channels) or Wan2.1 (z 16, no patch, no DupUp3D, resamplers halve)
  int zdim = 48, patch = 2;
  bool wan21 = false;
  int up[4][5] = {};  // per up block: cin, cout, temporal, spatial, resampler out (channels)
  bool split = false;  // fp32 decode: activations and weights as bf16 hi/lo pairs
  float* pq_w = nullptr;
  float* pq_b = nullptr;
  ConvW conv_in;
  Resnet mid[2];
  float* attn_g = nullptr;
  ConvW qkv, proj;
  Resnet ups[4][3];
  ConvW tconv[2];
  ConvW resample[3];
  float* out_g = nullptr;
  ConvW conv_out;
  TapFoldW out_tf;  // conv_out with its spatial taps folded into N (bf16 decode)
  // latent de-normalisation in front of post_quant_conv: mean[48], std[48]
  float* zstat = nullptr;
  bool zstat_on = false;
  DevMem mem;
};

// (in, out, temporal, spatial, resampler out) of the up blocks in units of the
// base dim.  TI2V-5B (page "What is computed": channels 4b, 4b, 4b -> 2b,
// 2b -> b; the resampler keeps the channels and DupUp3D adds the block
// input); Wan2.1 (that model's published configuration: the resampler
// halves the channels, the next block starts from half).
static const int kUp[4][5] = {{4, 4, 1, 1, 4}, {4, 4, 1, 1, 4}, {4, 2, 0, 1, 2}, {2, 1, 0, 0, 0}};
static const int kUpWan21[4][5] = {{4, 4, 1, 1, 2}, {2, 4, 1, 1, 2}, {2, 2, 0, 1, 1}, {1, 1, 0, 0, 0}};
static const int kZdimMax = 48;

static wan_status pack_resnet(const WeightTable& wt, const std::string& name, int ci, int co, Resnet& r, DevMem& mem,
                              cudaStream_t s, bool split) {
  r.ci = ci;
  r.co = co;
  WAN_TRY(pack_gamma(wt, name + ".norm1.gamma", ci, &r.g1, mem, s, split));
  WAN_TRY(pack_gamma(wt, name + ".norm2.gamma", co, &r.g2, mem, s, split));
  WAN_TRY(pack_conv(wt, name + ".conv1", co, ci, 3, 3, 3, false, "", 0, r.c1, mem, s, split));
  WAN_TRY(pack_conv(wt, name + ".conv2", co, co, 3, 3, 3, false, ci != co ? name + ".conv_shortcut" : "", ci, r.c2,
                    mem, s, split));
  return WAN_OK;
}

static wan_status model_build(const wan_tensor* weights, int n, int dtype, cudaStream_t s, wan_vae_model* m) {
  if (!weights || n <= 0) return fail(WAN_ERR_INVALID_ARG, "empty weight table");
  if (dtype != WAN_F32 && dtype != WAN_BF16) return fail(WAN_ERR_DTYPE, "dtype must be WAN_F32 or WAN_BF16, not %d", dtype);
  WeightTable wt{weights, n};
  const wan_tensor *ci, *pq;
  WAN_TRY(get_tensor(wt, "post_quant_conv.weight", &pq));
  if (pq->ndim < 1 || (pq->shape[0] != 48 && pq->shape[0] != 16))
    return fail(WAN_ERR_SHAPE, "post_quant_conv.weight must be [48, 48, 1, 1, 1] (TI2V-5B) or [16, 16, 1, 1, 1] (Wan2.1)");
  const int zd = (int)pq->shape[0];
  m->zdim = zd;
  m->wan21 = zd == 16;
  m->patch = m->wan21 ? 1 : 2;
  WAN_TRY(get_tensor(wt, "decoder.conv_in.weight", &ci));
  if (ci->ndim != 5 || ci->shape[0] % 4 || ci->shape[0] <= 0)
    return fail(WAN_ERR_SHAPE, "decoder.conv_in.weight must be [4b, %d, 3, 3, 3]", zd);
  const int b = (int)(ci->shape[0] / 4);
  if (b % 8 || 4 * b > 1024)
    return fail(WAN_ERR_UNSUPPORTED, "decoder base dim %d: must be a multiple of 8 and at most 256", b);
  m->base = b;
  m->dtype = dtype;
  m->split = dtype == WAN_F32;
  const bool sp = m->split;
  DevMem& mem = m->mem;
  // post_quant_conv 48 -> 48 (fp32, CUDA-core kernel)
  {
    const wan_tensor *w, *bb;
    WAN_TRY(get_tensor(wt, "post_quant_conv.weight", &w));
    WAN_TRY(get_tensor(wt, "post_quant_conv.bias", &bb));
    WAN_TRY(check_shape(w, {zd, zd, 1, 1, 1}));
    WAN_TRY(check_shape(bb, {zd}));
    if (!mem.dry) {
    void* p;
    WAN_TRY(mem.alloc(&p, zd * zd * sizeof(float)));
    m->pq_w = (float*)p;
    WAN_TRY(mem.alloc(&p, zd * sizeof(float)));
    m->pq_b = (float*)p;
    CUDA_TRY(launch_to_f32(w->data, w->dtype == WAN_F32, nullptr, 0, m->pq_w, zd * zd, 1.0f, sp ? 0 : 1, s));
    CUDA_TRY(launch_to_f32(bb->data, bb->dtype == WAN_F32, nullptr, 0, m->pq_b, zd, 1.0f, sp ? 0 : 1, s));
    }
  }
  const int c4 = 4 * b;
  WAN_TRY(pack_conv(wt, "decoder.conv_in", c4, zd, 3, 3, 3, false, "", 0, m->conv_in, mem, s, sp));
  WAN_TRY(pack_resnet(wt, "decoder.mid_block.resnets.0", c4, c4, m->mid[0], mem, s, sp));
  WAN_TRY(pack_resnet(wt, "decoder.mid_block.resnets.1", c4, c4, m->mid[1], mem, s, sp));
  WAN_TRY(pack_gamma(wt, "decoder.mid_block.attentions.0.norm.gamma", c4, &m->attn_g, mem, s, sp));
  WAN_TRY(pack_conv(wt, "decoder.mid_block.attentions.0.to_qkv", 3 * c4, c4, 1, 1, 1, true, "", 0, m->qkv, mem, s, sp));
  WAN_TRY(pack_conv(wt, "decoder.mid_block.attentions.0.proj", c4, c4, 1, 1, 1, true, "", 0, m->proj, mem, s, sp));
  for (int i = 0; i < 4; ++i) {
    const int* u = m->wan21 ? kUpWan21[i] : kUp[i];
    for (int k = 0; k < 5; ++k) m->up[i][k] = (k == 2 || k == 3) ? u[k] : u[k] * b;
    const int cin = m->up[i][0], cout = m->up[i][1];
    const std::string nm = "decoder.up_blocks." + std::to_string(i);
    const std::string ups = nm + (m->wan21 ? ".upsamplers.0" : ".upsampler");
    for (int j = 0; j < 3; ++j)
      WAN_TRY(pack_resnet(wt, nm + ".resnets." + std::to_string(j), j == 0 ? cin : cout, cout, m->ups[i][j], mem, s,
                          sp));
    if (u[2])
      WAN_TRY(pack_conv(wt, ups + ".time_conv", 2 * cout, cout, 3, 1, 1, false, "", 0, m->tconv[i], mem, s, sp));
    if (u[3]) WAN_TRY(pack_subpix_conv(wt, ups + ".resample.1", cout, m->up[i][4], m->resample[i], mem, s, sp));
  }
  WAN_TRY(pack_gamma(wt, "decoder.norm_out.gamma", b, &m->out_g, mem, s, sp));
  WAN_TRY(pack_conv(wt, "decoder.conv_out", 3 * m->patch * m->patch, b, 3, 3, 3, false, "", 0, m->conv_out, mem, s,
                    sp));
  if (!sp) WAN_TRY(pack_tapfold(wt, "decoder.conv_out", 3 * m->patch * m->patch, b, m->out_tf, mem, s));
  if (!mem.dry) CUDA_TRY(cudaGetLastError());
  return WAN_OK;
}

// Checks every name and shape first (no CUDA call), then packs.
static wan_status model_build_checked(const wan_tensor* weights, int n, int dtype, cudaStream_t s, wan_vae_model* m) {
  m->mem.dry = true;
  const wan_status v = model_build(weights, n, dtype, s, m);
  m->mem.dry = false;
  if (v != WAN_OK) return v;
  return model_build(weights, n, dtype, s, m);
}

// ======================================================================
// Stream state: workspace, rings, launch sequence
// ======================================================================
struct AttnBufs {
  Act an, qkv, O;
  float* S = nullptr;
  bf16* P = nullptr;
  bf16* Vt = nullptr;
  int HW = 0, HWs = 0, HWp = 0, Fmax = 0, B = 0, C = 0;
  int sp = 1;  // 2 in split mode: P and V^T rows hold [hi HWp | lo HWp]
  bool flash = false;  // the flash kernel (no S, no P); else score GEMM + row softmax + P V GEMM
  long long ldp() const { return (long long)sp * HWp; }
  long long s_bs() const { return (long long)Fmax * HW * HWs; }
  long long p_bs() const { return (long long)Fmax * HW * ldp(); }
  long long vt_fs() const { return (long long)C * ldp(); }
  long long vt_bs() const { return (long long)Fmax * vt_fs(); }
};

// The flash kernels: one CTA per 128 queries for head dims up to 384 (Wan2.1's
// 384, the narrow test widths), a cluster of C / 256 CTAs for 512 and 1024
// (TI2V-5B).  Other widths and the fp32 split format take the score GEMM, row
// softmax and P V GEMM path.
static bool attention_is_flash(bool split, int C) { return !split && flash_attn_supported(C); }

struct wan_vae_stream {
  const wan_vae_model* m = nullptr;
  Prof prof;
  int B = 0, h = 0, w = 0, nmax = 0;
  bool first = true;
  DevMem mem;
  char* ws = nullptr;
  size_t ws_bytes = 0, ws_used = 0;
  int* err_dev = nullptr;
  int* err_host = nullptr;
  cudaEvent_t err_ev = nullptr;
  bool err_pending = false;
  // level A (h x w)
  Act ringIn, RA[3], HA, ringA[10], tcA, tuA;
  AttnBufs at;
  // level B (2h x 2w)
  Act RB[3], HB, ringB[6], tcB, tuB;
  // level C (4h x 4w)
  Act RC[3], HC, ringC[6];
  // level D (8h x 8w)
  Act RD[3], HD, ringD[6], ringOut;
  std::vector<Act*> rings;
  std::vector<std::pair<Act*, int>> advance;  // rings a chunk consumed, and its frames
  // decode_clip_host: double-buffered latent / video staging, a copy stream
  // and its events, created on first use and kept until destroy
  void* zb[2] = {nullptr, nullptr};
  void* vb[2] = {nullptr, nullptr};
  size_t zb_bytes = 0, vb_bytes = 0;
  cudaStream_t copy_stream = nullptr;
  cudaEvent_t dec_ev[2] = {nullptr, nullptr}, d2h_ev[2] = {nullptr, nullptr};
};

static wan_status ws_take(wan_vae_stream* st, size_t bytes, void** p) {
  const size_t off = rup(st->ws_used, 256);
  if (off + bytes > st->ws_bytes) return fail(WAN_ERR_INTERNAL, "workspace plan overflow");
  *p = st->ws + off;
  st->ws_used = off + bytes;
  return WAN_OK;
}

// Declares (plan pass, ws == null) or places an activation tensor.
static wan_status make_act(wan_vae_stream* st, Act& a, int F, int H, int W, int C, int ldc_mult = 64) {
  a.B = st->B;
  a.F = F;
  a.H = H;
  a.W = W;
  a.C = C;
  a.ldc = (int)rup(C, ldc_mult);
  a.lo = 0;
  if (st->m->split) {  // [hi | lo] halves per position
    a.lo = a.ldc;
    a.ldc *= 2;
  }
  if (!st->ws) {
    st->ws_used = rup(st->ws_used, 256) + a.bytes();
    return WAN_OK;
  }
  void* p = nullptr;
  WAN_TRY(ws_take(st, a.bytes(), &p));
  a.p = (bf16*)p;
  return WAN_OK;
}
static wan_status make_raw(wan_vae_stream* st, size_t bytes, void** p) {
  if (!st->ws) {
    st->ws_used = rup(st->ws_used, 256) + bytes;
    *p = nullptr;
    return WAN_OK;
  }
  return ws_take(st, bytes, p);
}

static wan_status plan_buffers(wan_vae_stream* st) {
  const int b = st->m->base, c4 = 4 * b, n = st->nmax;
  const int hA = st->h, wA = st->w;
  st->rings.clear();
  auto ring = [&](Act& a, int F, int H, int W, int C) -> wan_status {
    WAN_TRY(make_act(st, a, 2 + F, H, W, C));
    a.fmod = a.F;
    a.base = 0;
    a.zhist = 2;
    st->rings.push_back(&a);
    return WAN_OK;
  };
  const wan_vae_model* m = st->m;
  // level A
  WAN_TRY(ring(st->ringIn, n, hA, wA, m->zdim));
  for (auto& a : st->RA) WAN_TRY(make_act(st, a, n, hA, wA, c4));
  WAN_TRY(make_act(st, st->HA, n, hA, wA, c4));
  for (auto& a : st->ringA) WAN_TRY(ring(a, n, hA, wA, c4));
  WAN_TRY(ring(st->tcA, n, hA, wA, c4));
  WAN_TRY(make_act(st, st->tuA, 2 * n, hA, wA, c4));
  // attention
  AttnBufs& at = st->at;
  at.HW = hA * wA;
  at.HWs = (int)rup(at.HW, 16);
  at.HWp = (int)rup(at.HW, 64);
  at.Fmax = n;
  at.B = st->B;
  at.C = c4;
  at.sp = st->m->split ? 2 : 1;
  at.flash = attention_is_flash(st->m->split, c4);
  WAN_TRY(make_act(st, at.an, n, 1, at.HW, c4));
  WAN_TRY(make_act(st, at.qkv, n, 1, at.HW, 3 * c4));
  WAN_TRY(make_act(st, at.O, n, 1, at.HW, c4));
  void* p;
  if (!at.flash) {  // the HW x HW scores and probabilities
    WAN_TRY(make_raw(st, (size_t)st->B * at.s_bs() * sizeof(float), &p));
    at.S = (float*)p;
    WAN_TRY(make_raw(st, (size_t)st->B * at.p_bs() * sizeof(bf16), &p));
    at.P = (bf16*)p;
  }
  WAN_TRY(make_raw(st, (size_t)st->B * at.vt_bs() * sizeof(bf16), &p));
  at.Vt = (bf16*)p;
  // level B
  const int hB = 2 * hA, wB = 2 * wA;
  // levels B, C, D: R[0] holds the up block's input (the previous block's
  // resampler output, cin channels), R[1], R[2] and H its resnets' outputs
  // (cout); ring 0 feeds the first conv1 (cin), rings 1-5 the others (cout)
  const int ciB = m->up[1][0], coB = m->up[1][1];
  WAN_TRY(make_act(st, st->RB[0], 2 * n, hB, wB, ciB));
  for (int i = 1; i < 3; ++i) WAN_TRY(make_act(st, st->RB[i], 2 * n, hB, wB, coB));
  WAN_TRY(make_act(st, st->HB, 2 * n, hB, wB, coB));
  WAN_TRY(ring(st->ringB[0], 2 * n, hB, wB, ciB));
  for (int i = 1; i < 6; ++i) WAN_TRY(ring(st->ringB[i], 2 * n, hB, wB, coB));
  WAN_TRY(ring(st->tcB, 2 * n, hB, wB, coB));
  WAN_TRY(make_act(st, st->tuB, 4 * n, hB, wB, coB));
  // level C
  const int hC = 4 * hA, wC = 4 * wA;
  const int ciC = m->up[2][0], coC = m->up[2][1];
  WAN_TRY(make_act(st, st->RC[0], 4 * n, hC, wC, ciC));
  WAN_TRY(make_act(st, st->RC[1], 4 * n, hC, wC, coC));
  WAN_TRY(make_act(st, st->RC[2], 4 * n, hC, wC, coC));
  WAN_TRY(make_act(st, st->HC, 4 * n, hC, wC, coC));
  WAN_TRY(ring(st->ringC[0], 4 * n, hC, wC, ciC));
  for (int i = 1; i < 6; ++i) WAN_TRY(ring(st->ringC[i], 4 * n, hC, wC, coC));
  // level D
  const int hD = 8 * hA, wD = 8 * wA;
  const int ciD = m->up[3][0], coD = m->up[3][1];
  WAN_TRY(make_act(st, st->RD[0], 4 * n, hD, wD, ciD));
  WAN_TRY(make_act(st, st->RD[1], 4 * n, hD, wD, coD));
  WAN_TRY(make_act(st, st->RD[2], 4 * n, hD, wD, coD));
  WAN_TRY(make_act(st, st->HD, 4 * n, hD, wD, coD));
  WAN_TRY(ring(st->ringD[0], 4 * n, hD, wD, ciD));
  for (int i = 1; i < 6; ++i) WAN_TRY(ring(st->ringD[i], 4 * n, hD, wD, coD));
  WAN_TRY(ring(st->ringOut, 4 * n, hD, wD, coD));
  return WAN_OK;
}

// ------------------------------------------------------------ conv launches
struct OutSpec {
  void* p = nullptr;
  int f32 = 0;
  long long bs = 0, fs = 0;
  int ldc = 0, f0 = 0, fmul = 1, interleave = 0, lo = 0;
};
static OutSpec out_of(const Act& a, int f0 = 0) {
  OutSpec o;
  o.p = a.p;
  o.lo = a.lo;
  o.bs = a.bs();
  o.fs = a.fs();
  o.ldc = a.ldc;
  o.f0 = f0;
  return o;
}

// Appends the K slices of one kernel tap: cpad input channels of source
// `src` against B columns kb..kb+cpad.  In split mode a value is hi + lo in
// both operands and the tap becomes three slices, hi*hi + hi*lo + lo*hi
// (B's lo half follows its hi half at kb + cpad; A's at channel a_lo); the
// dropped lo*lo term is below 2^-16 of the product.
static wan_status add_tap(ConvArgs& A, int& nt, int src, int dt, int dy, int dx, int cpad, int a_lo, int kb,
                          int split) {
  const int parts = split ? 3 : 1;
  if (nt + parts > kMaxTaps) return fail(WAN_ERR_INTERNAL, "too many K slices");
  for (int q = 0; q < parts; ++q) {
    ConvTap& t = A.taps[nt++];
    t.src = (int8_t)src;
    t.dt = (int8_t)dt;
    t.dy = (int8_t)dy;
    t.dx = (int8_t)dx;
    t.a_c0 = (int16_t)(q == 2 ? a_lo : 0);
    t.nkb = (int16_t)(cpad / 64);
    t.b_k0 = kb + (q == 1 ? cpad : 0);
    A.total_kb += cpad / 64;
  }
  return WAN_OK;
}

// Fills the launch for conv `cw` reading A source 0 (`a0`, output frame 0 at
// frame coordinate a0_f0 for dt = 0) and optionally the shortcut source a1.
// Taps of source 0 with dt < dt_min are left out (they would read frames of
// zeros: the causal padding).  subpix_row: a sub-pixel conv with a plain
// store epilogue may take row mode.
static wan_status conv_setup(const ConvW& cw, const Act& a0, int a0_f0, const Act* a1, int a1_f0, int F, ConvLaunch& L,
                             int dt_min = 0, bool subpix_row = false) {
  memset(&L, 0, sizeof(L));
  ConvArgs& A = L.args;
  if (a0.ldc < cw.ci_pad || (a1 && a1->ldc < cw.sc_ci_pad))
    return fail(WAN_ERR_INTERNAL, "conv source narrower than its packed channels");
  // row mode (narrow N, 3x3 spatial taps, one source): 128-pixel row tiles,
  // one 130-pixel A box per (dt, dy) serving its three dx taps
  // (sub-pixel convs too, N tile 96, 128 or 192: each phase's two dx taps
  // read one 130-pixel box)
  const bool row = (!cw.split && !cw.subpix && cw.kh == 3 && cw.kw == 3 && !cw.sc_ci_pad && !a1 &&
                    (cw.bn == 96 || cw.bn == 128)) ||
                   (subpix_row && !cw.split && cw.subpix && cw.kh == 2 && cw.kw == 2 && !cw.sc_ci_pad && !a1 &&
                    (cw.bn == 96 || cw.bn == 128 || cw.bn == 192));
  // band mode (256-wide 3x3 convs, one source): a 16 x 10 A box per (dt, dx)
  // serving its three dy taps
  const bool band = !cw.split && !cw.subpix && cw.kh == 3 && cw.kw == 3 && !cw.sc_ci_pad && !a1 &&
                    (cw.bn == 192 || cw.bn == 256);
  if (band) {
    WAN_TRY(act_map(&L.a0, a0, 16, kBandBoxRows));
    L.a1 = L.a0;
    const uint64_t dims[3] = {(uint64_t)cw.ktot, (uint64_t)cw.co_pad, 1};
    const uint64_t strides[2] = {(uint64_t)cw.ktot * 2, (uint64_t)cw.ktot * cw.co_pad * 2};
    const uint32_t box[3] = {64, (uint32_t)(cw.bn / 2), 1};  // each CTA of a pair loads half
    WAN_TRY(encode(&L.b, 3, cw.w, dims, strides, box));
  } else if (row) {
    WAN_TRY(act_map(&L.a0, a0, 130, 1));
    L.a1 = L.a0;
    const uint64_t dims[3] = {(uint64_t)cw.ktot, (uint64_t)cw.co_pad, (uint64_t)(cw.subpix ? 4 : 1)};
    const uint64_t strides[2] = {(uint64_t)cw.ktot * 2, (uint64_t)cw.ktot * cw.co_pad * 2};
    const uint32_t box[3] = {64, (uint32_t)(cw.bn / 2), 1};  // each CTA of a pair loads half
    WAN_TRY(encode(&L.b, 3, cw.w, dims, strides, box));
  } else {
    WAN_TRY(act_map(&L.a0, a0));
    if (a1)
      WAN_TRY(act_map(&L.a1, *a1));
    else
      L.a1 = L.a0;
    WAN_TRY(b_map(&L.b, cw.w, cw.ktot, cw.co_pad, cw.subpix ? 4 : 1, cw.ktot, (long long)cw.ktot * cw.co_pad, cw.bn));
  }
  if (cw.split && (!a0.lo || (a1 && !a1->lo))) return fail(WAN_ERR_INTERNAL, "split conv on a plain tensor");
  A.subpix = cw.subpix;
  int nt = 0, k = 0;
  for (int dt = 0; dt < cw.kt; ++dt)
    for (int dy = 0; dy < cw.kh; ++dy)
      for (int dx = 0; dx < cw.kw; ++dx) {
        // sub-pixel taps carry source offsets 0/1; the kernel adds the phase's (i - 1, j - 1)
        const int oy = cw.subpix ? dy : dy - cw.kh / 2, ox = cw.subpix ? dx : dx - cw.kw / 2;
        if (dt < dt_min) {
          // the tap reads only causal zero padding
        } else if (band) {
          // taps (dt, dx) in that order, each standing for its three dy taps
          if (dy == 0) {
            const int kd = ((dt * cw.kh + 0) * cw.kw + dx) * cw.ci_pad;
            WAN_TRY(add_tap(A, nt, 0, dt, -1, ox, cw.ci_pad, a0.lo, kd, 0));
          }
        } else if (!row || dx == 0) {
          WAN_TRY(add_tap(A, nt, 0, dt, oy, ox, cw.ci_pad, a0.lo, k, cw.split));
        }
        k += (cw.split ? 2 : 1) * cw.ci_pad;
      }
  if (cw.sc_ci_pad) {
    if (!a1) return fail(WAN_ERR_INTERNAL, "shortcut conv without its source");
    WAN_TRY(add_tap(A, nt, 1, 0, 0, 0, cw.sc_ci_pad, a1->lo, k, cw.split));
    k += (cw.split ? 2 : 1) * cw.sc_ci_pad;
  }
  A.n_taps = nt;
  A.row = row ? 1 : 0;
  // the last 64-channel block of a tap with 96 (160, ...) input channels holds
  // 32 of them: two K16 steps (the source's channel extent ends there, so the
  // TMA fills the rest with zeros and those MMAs would add nothing)
  A.tail_k16 = (row && !a0.lo && cw.Ci % 64 == 32 && a0.chans() == cw.Ci) ? 2 : 0;
  A.band = band ? 1 : 0;
  A.row_bdk = row ? cw.ci_pad : band ? cw.kw * cw.ci_pad : 0;
  A.box_w = row ? 128 : 16;
  A.box_h = row ? 1 : 8;
  A.H = a0.H;
  A.W = a0.W;
  A.tiles_x = (int)cdiv(a0.W, A.box_w);
  A.tiles_y = (int)cdiv(a0.H, A.box_h);
  A.tiles_n = cw.co_pad / cw.bn;
  A.frames = F;
  A.batches = a0.B;
  A.src_f0[0] = a0.slot(a0_f0);
  A.src_fmod = a0.fmod;
  A.src_f0[1] = a1_f0;
  A.N = cw.Co;
  A.bias = cw.bias;
  L.bn = cw.bn;
  L.epi = kEpiStore;
  return WAN_OK;
}

static void set_out(ConvArgs& A, const OutSpec& o) {
  A.out = o.p;
  A.out_f32 = o.f32;
  A.out_bs = o.bs;
  A.out_fs = o.fs;
  A.out_ldc = o.ldc;
  A.out_f0 = o.f0;
  A.out_fmul = o.fmul;
  A.interleave_c = o.interleave;
  A.out_lo = o.lo;
}

// Enqueues a tensor-core launch; when profiling, brackets it with CUDA events
// on the same stream and records its nominal FLOPs (2 * M * N * K with the
// zero-padded taps included).
static wan_status run(ConvLaunch& L, Prof* prof, int kind, double flops, int* err, cudaStream_t s,
                      double exec_flops = -1.0) {
  L.args.err = err;
  if (L.args.N % 16 && L.epi != kEpiVideo) return fail(WAN_ERR_INTERNAL, "conv output channels not a multiple of 16");
  cudaEvent_t e1 = nullptr;
  if (prof) WAN_TRY(prof->begin(kind, flops, s, &e1, exec_flops));
  CUDA_TRY(launch_conv(L, s));
  if (e1) CUDA_TRY(cudaEventRecord(e1, s));
  if (prof) prof->launches++;
  return WAN_OK;
}

static double conv_flops(const ConvW& cw, const Act& a0, int F) {
  const double M = (double)a0.B * F * a0.H * a0.W;
  return 2.0 * M * cw.Co * ((double)cw.kt * cw.kh * cw.kw * cw.Ci + cw.sc_Ci);
}

// RMS norm (+ SiLU) of a conv's output fused into its epilogue, written to
// the current-frame slots of `ring`.
struct NormOut {
  const float* gs = nullptr;  // sqrt(C) * gamma
  bool silu = true;
  const Act* ring = nullptr;
};
// One N tile holds every output channel: the epilogue can normalise.
static bool single_tile(const ConvW& cw) { return cw.co_pad == cw.bn && !cw.subpix; }

// 3-frame causal conv over ring `in` (F current frames) into `out`.  While
// the ring's history holds the zero padding of a stream's start (in.zhist
// leading zero frames), output frame f < zhist reads zeros through its taps
// dt < zhist - f: those frames run as launches of their own without those
// taps (the zero padding is applied by leaving the taps out, not computed).
static wan_status ring_conv(wan_vae_stream* st, const ConvW& cw, Act& in, int F, const OutSpec& o, const Act* res,
                            const Act* sc, cudaStream_t s, int kind = kKindConv333, const NormOut* nrm = nullptr) {
  if (nrm && !single_tile(cw)) return fail(WAN_ERR_INTERNAL, "fused norm over several N tiles");
  const int z = cw.kt == 3 ? std::min(in.zhist, 2) : 0;
  const double kfull = (double)cw.kt * cw.kh * cw.kw * cw.Ci + cw.sc_Ci;
  for (int f0 = 0; f0 < F;) {
    // frames [f0, f1) share dt_min: one frame at a time while f0 < z
    const int dt_min = f0 < z ? z - f0 : 0;
    const int f1 = f0 < z ? f0 + 1 : F;
    const int nf = f1 - f0;
    ConvLaunch L;
    WAN_TRY(conv_setup(cw, in, f0, sc, f0, nf, L, dt_min));
    OutSpec of = o;
    of.f0 = o.f0 + f0 * o.fmul;
    set_out(L.args, of);
    if (nrm) {
      L.args.norm_gs = nrm->gs;
      L.args.norm_silu = nrm->silu ? 1 : 0;
      L.args.out2 = nrm->ring->p;
      L.args.out2_bs = nrm->ring->bs();
      L.args.out2_fs = nrm->ring->fs();
      L.args.out2_ldc = nrm->ring->ldc;
      L.args.out2_f0 = nrm->ring->slot(2 + f0);
      L.args.out2_fmod = nrm->ring->fmod;
      L.args.out2_lo = nrm->ring->lo;
    }
    if (res) {
      L.args.res = res->p;
      L.args.res_bs = res->bs();
      L.args.res_fs = res->fs();
      L.args.res_ldc = res->ldc;
      L.args.res_lo = res->lo;
      L.args.res_f0 = f0;
    }
    const double nominal = conv_flops(cw, in, nf);
    const double kept = (double)(cw.kt - dt_min) * cw.kh * cw.kw * cw.Ci + cw.sc_Ci;
    WAN_TRY(run(L, &st->prof, kind, nominal, st->err_dev, s, nominal * kept / kfull));
    f0 = f1;
  }
  st->advance.push_back({&in, F});
  return WAN_OK;
}

// Residual block (page "The parts", third bullet): x (F frames) -> y.
// normed: ring1 already holds SiLU(norm1(x)), written by the producer of x.
// next: the RMS norm that consumes y; when conv2 has one N tile it is fused
// into conv2's epilogue and *next_done is set.
static wan_status resnet(wan_vae_stream* st, const Resnet& r, const Act& x, Act& ring1, Act& ring2, Act& Ht, Act& y,
                         int F, cudaStream_t s, bool normed = false, const NormOut* next = nullptr,
                         bool* next_done = nullptr) {
  const int P = x.H * x.W;
  const double nb = 2.0 * 2 * x.B * F * (double)P * (x.lo ? 2 : 1);  // bytes per channel, read + write
  if (!normed)
    ELT(&st->prof, kKindNorm, nb * r.ci,
        launch_rms_norm(x.view(0), ring1.view(2), r.g1, r.ci, x.B, F, P, true, s, x.lo, ring1.lo));
  if (single_tile(r.c1)) {  // conv1 writes SiLU(norm2(h)) straight into conv2's ring
    NormOut n2;
    n2.gs = r.g2;
    n2.ring = &ring2;
    OutSpec none;
    WAN_TRY(ring_conv(st, r.c1, ring1, F, none, nullptr, nullptr, s, kKindConv333, &n2));
  } else {
    WAN_TRY(ring_conv(st, r.c1, ring1, F, out_of(Ht), nullptr, nullptr, s));
    ELT(&st->prof, kKindNorm, nb * r.co,
        launch_rms_norm(Ht.view(0), ring2.view(2), r.g2, r.co, x.B, F, P, true, s, Ht.lo, ring2.lo));
  }
  const bool fuse_next = next && single_tile(r.c2);
  if (next_done) *next_done = fuse_next;
  const NormOut* nx = fuse_next ? next : nullptr;
  if (r.ci != r.co)
    WAN_TRY(ring_conv(st, r.c2, ring2, F, out_of(y), nullptr, &x, s, kKindConv333, nx));
  else
    WAN_TRY(ring_conv(st, r.c2, ring2, F, out_of(y), &x, nullptr, s, kKindConv333, nx));
  return WAN_OK;
}

// Batched GEMM launch: A = rows of an activation tensor (HW positions per
// frame, `a_ldc` channels of which `K` are read, low halves at a_lo), B = a
// K-major operand whose columns b0.. (low halves at b0 + b_lo) are read.
static wan_status gemm_setup(ConvLaunch& L, const bf16* a_base, int a_ldc, int a_lo, int HW, int Fmax, int B,
                             long long a_fs, long long a_bs, int K, int b0, int b_lo, int split, int N_tiles_n, int bn,
                             int F) {
  memset(&L.args, 0, sizeof(L.args));
  WAN_TRY(act_map(&L.a0, a_base, a_ldc, a_ldc, HW, 1, Fmax, B, a_fs, a_bs, 128, 1));
  L.a1 = L.a0;
  ConvArgs& A = L.args;
  int nt = 0;
  if (split) {
    // hi*hi + hi*lo + lo*hi, with B's low half at b0 + b_lo
    WAN_TRY(add_tap(A, nt, 0, 0, 0, 0, K, a_lo, b0, 0));
    WAN_TRY(add_tap(A, nt, 0, 0, 0, 0, K, a_lo, b0 + b_lo, 0));
    WAN_TRY(add_tap(A, nt, 0, 0, 0, 0, K, a_lo, b0, 0));
    A.taps[2].a_c0 = (int16_t)a_lo;
  } else {
    WAN_TRY(add_tap(A, nt, 0, 0, 0, 0, K, 0, b0, 0));
  }
  A.n_taps = nt;
  A.box_w = 128;
  A.box_h = 1;
  A.H = 1;
  A.W = HW;
  A.tiles_x = (int)cdiv(HW, 128);
  A.tiles_y = 1;
  A.tiles_n = N_tiles_n;
  A.frames = F;
  A.batches = B;
  L.bn = bn;
  L.epi = kEpiStore;
  return WAN_OK;
}

// The flash kernel's launch for F frames of the buffers `at` (q, k in
// at.qkv channels [0, C) and [C, 2C), V^T in at.Vt, O into at.O).
static wan_status flash_setup(const AttnBufs& at, int F, int* err, FlashLaunch& FL) {
  const int C = at.C, HW = at.HW, B = at.B;
  memset(&FL, 0, sizeof(FL));
  const FlashBoxes fb = flash_attn_boxes(C);
  {
    const uint64_t dims[4] = {(uint64_t)at.qkv.chans(), (uint64_t)HW, (uint64_t)at.qkv.F, (uint64_t)B};
    const uint64_t strides[3] = {(uint64_t)at.qkv.ldc * 2, (uint64_t)at.qkv.fs() * 2, (uint64_t)at.qkv.bs() * 2};
    const uint32_t qbox[4] = {64, (uint32_t)fb.q_rows, 1, 1};
    WAN_TRY(encode(&FL.q, 4, at.qkv.p, dims, strides, qbox));
    const uint32_t kbox[4] = {64, (uint32_t)fb.k_rows, 1, 1};
    WAN_TRY(encode(&FL.k, 4, at.qkv.p, dims, strides, kbox));
  }
  {
    const uint64_t dims[4] = {(uint64_t)at.HWp, (uint64_t)C, (uint64_t)at.Fmax, (uint64_t)B};
    const uint64_t strides[3] = {(uint64_t)at.ldp() * 2, (uint64_t)at.vt_fs() * 2, (uint64_t)at.vt_bs() * 2};
    const uint32_t box[4] = {64, (uint32_t)fb.v_rows, 1, 1};
    WAN_TRY(encode(&FL.v, 4, at.Vt, dims, strides, box));
  }
  FlashArgs& a = FL.args;
  a.HW = HW;
  a.frames = F;
  a.batches = B;
  a.nkb = (HW + fb.key_block - 1) / fb.key_block;
  a.C = C;
  a.q_c0 = 0;
  a.k_c0 = C;
  a.scale_log2 = 1.4426950408889634f / std::sqrt((float)C);
  a.out = at.O.p;
  a.out_bs = at.O.bs();
  a.out_fs = at.O.fs();
  a.out_ldc = at.O.ldc;
  a.err = err;
  return WAN_OK;
}

// Mid-block attention over F frames of x (level A) into y = attn(x) + x
// (page "The parts", fourth bullet): RMS norm; qkv = 1x1 conv C -> 3C;
// S = q k^T per frame (fp32); P = softmax(S / sqrt(C)); O = P v; y = proj(O) + x.
static wan_status attention(const float* g, const ConvW& qkv, const ConvW& proj, AttnBufs& at, const Act& x, Act& y,
                            int F, Prof* prof, int* err, cudaStream_t s) {
  const double M = (double)at.B * F * at.HW;
  const int C = at.C, HW = at.HW, B = at.B, sp = at.sp - 1;
  ELT(prof, kKindNorm, 4.0 * M * C * at.sp, launch_rms_norm(x.view(0), at.an.view(0), g, C, B, F, HW, false, s, x.lo, at.an.lo));
  ConvLaunch L;
  // qkv = n Wqkv^T + b; split weights keep their low halves ci_pad after the high ones
  WAN_TRY(gemm_setup(L, at.an.p, at.an.ldc, at.an.lo, HW, at.an.F, B, at.an.fs(), at.an.bs(), qkv.ci_pad, 0,
                     qkv.ci_pad, sp, qkv.co_pad / qkv.bn, qkv.bn, F));
  WAN_TRY(b_map(&L.b, qkv.w, qkv.ktot, qkv.co_pad, 1, qkv.ktot, (long long)qkv.ktot * qkv.co_pad, qkv.bn));
  L.args.N = qkv.Co;
  L.args.bias = qkv.bias;
  set_out(L.args, out_of(at.qkv));
  WAN_TRY(run(L, prof, kKindAttention, 2.0 * M * 3 * C * C, err, s));
  if (at.flash) {
    // V^T per frame, then the flash kernel: O = softmax(q k^T / sqrt(C)) v
    for (int b = 0; b < B; ++b)
      ELT(prof, kKindMisc, 4.0 * F * HW * C,
          launch_transpose(at.qkv.p + b * at.qkv.bs() + 2 * C, at.qkv.fs(), at.qkv.ldc, at.Vt + b * at.vt_bs(),
                           at.vt_fs(), (int)at.ldp(), F, HW, C, s));
    FlashLaunch FL;
    WAN_TRY(flash_setup(at, F, err, FL));
    cudaEvent_t e1 = nullptr;
    const double nominal = 4.0 * M * HW * C;
    if (prof) WAN_TRY(prof->begin(kKindAttention, nominal, s, &e1, nominal * flash_attn_exec_ratio(C)));
    CUDA_TRY(launch_flash_attn(FL, s));
    if (e1) CUDA_TRY(cudaEventRecord(e1, s));
    if (prof) prof->launches++;
  } else {
    // S = q k^T: q = channels [0, C) of qkv, k = [C, 2C) (low halves 3C further on)
    // N tile: the largest power of two <= min(HW, 256), at least 16.  With
    // fewer than 16 positions the key box runs past the frame's rows: TMA reads
    // zeros there, the extra columns of S are never read by the softmax (n =
    // HW), and P and V^T keep zeros beyond HW from the workspace clear.
    int bnS = 16;
    while (bnS * 2 <= std::min(HW, 256)) bnS *= 2;
    WAN_TRY(gemm_setup(L, at.qkv.p, at.qkv.ldc, at.qkv.lo, HW, at.qkv.F, B, at.qkv.fs(), at.qkv.bs(), C, C, at.qkv.lo,
                       sp, (int)cdiv(at.HWs, bnS), bnS, F));
    WAN_TRY(b_map(&L.b, at.qkv.p, at.qkv.ldc, HW, (long long)B * at.Fmax, at.qkv.ldc, at.qkv.fs(), bnS));
    L.args.b_per_frame = 1;
    L.args.b_gstride = at.Fmax;
    L.args.N = at.HWs;
    {
      OutSpec o;
      o.p = at.S;
      o.f32 = 1;
      o.bs = at.s_bs();
      o.fs = (long long)HW * at.HWs;
      o.ldc = at.HWs;
      set_out(L.args, o);
    }
    WAN_TRY(run(L, prof, kKindAttention, 2.0 * M * HW * C, err, s));
    // P = softmax(S / sqrt(C)); V^T per frame
    const float scale = 1.0f / std::sqrt((float)C);
    for (int b = 0; b < B; ++b) {
      ELT(prof, kKindMisc, (4.0 * at.HWs + 2.0 * at.ldp()) * F * HW, launch_softmax_rows(at.S + b * at.s_bs(), at.HWs, at.P + b * at.p_bs(), at.ldp(), HW, (long long)F * HW,
                                    scale, s, sp ? at.HWp : 0));
      for (int part = 0; part <= sp; ++part)
        ELT(prof, kKindMisc, 4.0 * F * HW * C, launch_transpose(at.qkv.p + b * at.qkv.bs() + 2 * C + part * at.qkv.lo, at.qkv.fs(), at.qkv.ldc,
                                   at.Vt + b * at.vt_bs() + part * at.HWp, at.vt_fs(), (int)at.ldp(), F, HW, C, s));
    }
    // O = P V
    const int bnC = choose_bn(C);
    WAN_TRY(gemm_setup(L, at.P, (int)at.ldp(), sp ? at.HWp : 0, HW, at.Fmax, B, (long long)HW * at.ldp(), at.p_bs(),
                       at.HWp, 0, at.HWp, sp, (int)cdiv(C, bnC), bnC, F));
    WAN_TRY(b_map(&L.b, at.Vt, at.ldp(), C, (long long)B * at.Fmax, at.ldp(), at.vt_fs(), bnC));
    L.args.b_per_frame = 1;
    L.args.b_gstride = at.Fmax;
    L.args.N = C;
    set_out(L.args, out_of(at.O));
    WAN_TRY(run(L, prof, kKindAttention, 2.0 * M * HW * C, err, s));
  }
  // y = O Wp^T + b + x
  WAN_TRY(gemm_setup(L, at.O.p, at.O.ldc, at.O.lo, HW, at.O.F, B, at.O.fs(), at.O.bs(), proj.ci_pad, 0, proj.ci_pad,
                     sp, proj.co_pad / proj.bn, proj.bn, F));
  WAN_TRY(b_map(&L.b, proj.w, proj.ktot, proj.co_pad, 1, proj.ktot, (long long)proj.ktot * proj.co_pad, proj.bn));
  L.args.N = proj.Co;
  L.args.bias = proj.bias;
  set_out(L.args, out_of(y));
  L.args.res = x.p;
  L.args.res_bs = x.bs();
  L.args.res_fs = x.fs();
  L.args.res_ldc = x.ldc;
  L.args.res_lo = x.lo;
  WAN_TRY(run(L, prof, kKindAttention, 2.0 * M * C * C, err, s));
  return WAN_OK;
}

// ---------------------------------------------------------------- the chunk
static wan_status copy_frames(const Act& src, int sf0, const Act& dst, int df0, int F, Prof* prof, cudaStream_t s) {
  ELT(prof, kKindMisc, 4.0 * src.chans() * src.B * F * src.H * src.W,
      launch_copy_frames(src.view(sf0), dst.view(df0), src.chans(), src.B, F, src.H * src.W, s));
  return WAN_OK;
}

// upsample3d's time conv (page "The parts", fifth bullet; "The first latent
// frame yields one frame"): x has Fin frames; tu receives 2*Fin frames, or
// 2*Fin - 1 on the first chunk, whose first frame passes through.
static wan_status time_upsample(wan_vae_stream* st, const ConvW& tc, const Act& x, Act& ring, Act& tu, int Fin,
                                bool first, cudaStream_t s) {
  const int C = x.C;
  int fx0 = 0, fout0 = 0, Ft = Fin;
  if (first) {
    WAN_TRY(copy_frames(x, 0, tu, 0, 1, &st->prof, s));
    fx0 = 1;
    fout0 = 1;
    Ft = Fin - 1;
  }
  if (Ft <= 0) return WAN_OK;
  WAN_TRY(copy_frames(x, fx0, ring, 2, Ft, &st->prof, s));
  OutSpec o = out_of(tu, fout0);
  o.fmul = 2;
  o.interleave = C;
  return ring_conv(st, tc, ring, Ft, o, nullptr, nullptr, s, kKindTimeConv);
}

// upsample2d (nearest x2, 3x3 conv) of the low-resolution `x` (F frames),
// in the sub-pixel form, plus DupUp3D of the up block's input `blk` (page
// "The parts", fifth and sixth bullets); y is at twice x's resolution.  The
// Wan2.1 decoder has no DupUp3D: the conv's result is stored as it is.
static wan_status resample(wan_vae_stream* st, const ConvW& cw, const Act& x, const Act& blk, int ft, bool first,
                           Act& y, int F, cudaStream_t s) {
  ConvLaunch L;
  if (!cw.subpix || y.H != 2 * x.H || y.W != 2 * x.W) return fail(WAN_ERR_INTERNAL, "resample shapes");
  // Wan2.1's resamplers (plain store epilogue) may run in row mode
  WAN_TRY(conv_setup(cw, x, 0, nullptr, 0, F, L, 0, st->m->wan21));
  set_out(L.args, out_of(y));
  // nominal FLOPs: the 3x3 conv at the upsampled resolution; executed: the
  // four phases' 2x2 convs at the low resolution (4/9 of nominal)
  const double nominal = 2.0 * x.B * F * 4.0 * x.H * x.W * cw.Co * 9.0 * cw.Ci;
  const double executed = 2.0 * x.B * F * 4.0 * x.H * x.W * cw.Co * 4.0 * cw.Ci;
  if (st->m->wan21) return run(L, &st->prof, kKindResample, nominal, st->err_dev, s, executed);
  L.epi = kEpiDup;
  L.args.dup = blk.p;
  L.args.dup_bs = blk.bs();
  L.args.dup_fs = blk.fs();
  L.args.dup_ldc = blk.ldc;
  L.args.dup_W = blk.W;
  L.args.dup_ft = ft;
  L.args.dup_first = first ? 1 : 0;
  L.args.dup_lo = blk.lo;
  // r = out * ft * 4 / in: 4ft means channel c copies source channel c; r = 2
  // (ft = 1, in = 2 out) means source channel 2c + row parity.
  const int r = cw.Co * ft * 4 / blk.C;
  if (r == 4 * ft && blk.C == cw.Co)
    L.args.dup_pairs = 0;
  else if (ft == 1 && r == 2 && blk.C == 2 * cw.Co)
    L.args.dup_pairs = 1;
  else
    return fail(WAN_ERR_UNSUPPORTED, "DupUp3D with %d -> %d channels, ft %d", blk.C, cw.Co, ft);
  return run(L, &st->prof, kKindResample, nominal, st->err_dev, s, executed);
}

// The three residual blocks of an up block: R[0] -> R[1] -> R[2] -> R[1]
// (R[0], the block input, stays for DupUp3D), with each block's norm1 fused
// into the previous block's conv2 where possible.  `last` optionally names
// the norm that consumes the final output.
static wan_status resnet_chain(wan_vae_stream* st, const Resnet* r, Act* R, Act* rings, Act& Ht, int F,
                               const NormOut* last, cudaStream_t s, bool* last_done = nullptr) {
  const int io[3][2] = {{0, 1}, {1, 2}, {2, 1}};
  bool normed = false;
  for (int j = 0; j < 3; ++j) {
    NormOut nx;
    const NormOut* next = nullptr;
    if (j < 2) {
      nx.gs = r[j + 1].g1;
      nx.ring = &rings[2 * (j + 1)];
      next = &nx;
    } else {
      next = last;
    }
    bool done = false;
    WAN_TRY(resnet(st, r[j], R[io[j][0]], rings[2 * j], rings[2 * j + 1], Ht, R[io[j][1]], F, s, normed, next, &done));
    normed = done;
    if (j == 2 && last_done) *last_done = done;
  }
  return WAN_OK;
}

static wan_status run_chunk(wan_vae_stream* st, const void* z, int z_f32, long long Tz, long long t0, int n, void* out,
                            int out_f32, long long out_frames, long long out_f0, float* pre, cudaStream_t s) {
  const wan_vae_model* m = st->m;
  const bool first = st->first;
  const int FA = n, FB = first ? 2 * n - 1 : 2 * n, FC = first ? 4 * n - 3 : 4 * n;
  const int P = st->h * st->w;
  st->advance.clear();
  // 1. post_quant_conv into conv_in's ring
  ELT(&st->prof, kKindMisc, (double)st->B * FA * P * (m->zdim * (z_f32 ? 4 : 2) + 2 * st->ringIn.ldc),
      launch_post_quant(z, z_f32, m->zdim, st->B, (int)Tz, (int)t0, FA, P, m->pq_w, m->pq_b,
                        m->zstat_on ? m->zstat : nullptr, st->ringIn.view(2), m->split ? 0 : 1, s, st->ringIn.lo));
  // 2. conv_in, mid block
  WAN_TRY(ring_conv(st, m->conv_in, st->ringIn, FA, out_of(st->RA[0]), nullptr, nullptr, s));
  WAN_TRY(resnet(st, m->mid[0], st->RA[0], st->ringA[0], st->ringA[1], st->HA, st->RA[1], FA, s));
  WAN_TRY(attention(m->attn_g, m->qkv, m->proj, st->at, st->RA[1], st->RA[2], FA, &st->prof, st->err_dev, s));
  WAN_TRY(resnet(st, m->mid[1], st->RA[2], st->ringA[2], st->ringA[3], st->HA, st->RA[0], FA, s));
  // up block 0 (level A -> B); block input RA[0]
  WAN_TRY(resnet_chain(st, m->ups[0], st->RA, st->ringA + 4, st->HA, FA, nullptr, s));
  WAN_TRY(time_upsample(st, m->tconv[0], st->RA[1], st->tcA, st->tuA, FA, first, s));
  WAN_TRY(resample(st, m->resample[0], st->tuA, st->RA[0], 2, first, st->RB[0], FB, s));
  // up block 1 (level B -> C); block input RB[0]
  WAN_TRY(resnet_chain(st, m->ups[1], st->RB, st->ringB, st->HB, FB, nullptr, s));
  WAN_TRY(time_upsample(st, m->tconv[1], st->RB[1], st->tcB, st->tuB, FB, first, s));
  WAN_TRY(resample(st, m->resample[1], st->tuB, st->RB[0], 2, first, st->RC[0], FC, s));
  // up block 2 (level C -> D); block input RC[0]
  WAN_TRY(resnet_chain(st, m->ups[2], st->RC, st->ringC, st->HC, FC, nullptr, s));
  WAN_TRY(resample(st, m->resample[2], st->RC[1], st->RC[0], 1, first, st->RD[0], FC, s));
  // up block 3 (level D)
  NormOut nout;  // norm_out + SiLU, fused into the last conv2 when possible
  nout.gs = m->out_g;
  nout.ring = &st->ringOut;
  bool out_done = false;
  WAN_TRY(resnet_chain(st, m->ups[3], st->RD, st->ringD, st->HD, FC, &nout, s, &out_done));
  // norm_out, SiLU, conv_out with unpatchify + clamp in its epilogue
  if (!out_done) {
    ELT(&st->prof, kKindNorm, 4.0 * st->B * FC * st->RD[1].H * st->RD[1].W * m->base * (m->split ? 2 : 1),
        launch_rms_norm(st->RD[1].view(0), st->ringOut.view(2), m->out_g, m->base, st->B, FC,
                        st->RD[1].H * st->RD[1].W, true, s, st->RD[1].lo, st->ringOut.lo));
  }
  if (m->out_tf.w) {
    VideoConvLaunch V;
    WAN_TRY(video_conv_setup(m->out_tf, m->conv_out.bias, st->ringOut, FC, m->patch, V));
    VideoConvArgs& a = V.args;
    a.out = out;
    a.out_f32 = out_f32;
    a.out_f0 = (int)out_f0;
    a.preclamp = pre;
    a.vid_cs = out_frames * (long long)(m->patch * m->patch) * st->ringOut.H * st->ringOut.W;
    a.vid_bs = 3 * a.vid_cs;
    a.err = st->err_dev;
    cudaEvent_t e1 = nullptr;
    WAN_TRY(st->prof.begin(kKindConvOut, conv_flops(m->conv_out, st->ringOut, FC), s, &e1));
    CUDA_TRY(launch_video_conv(V, s));
    if (e1) CUDA_TRY(cudaEventRecord(e1, s));
    st->prof.launches++;
    st->advance.push_back({&st->ringOut, FC});
  } else {
    ConvLaunch L;
    const ConvW& co = m->conv_out;
    WAN_TRY(conv_setup(co, st->ringOut, 0, nullptr, 0, FC, L));
    L.epi = kEpiVideo;
    L.args.out = out;
    L.args.out_f32 = out_f32;
    L.args.out_f0 = (int)out_f0;
    L.args.preclamp = pre;
    L.args.vid_patch = m->patch;
    L.args.vid_cs = out_frames * (long long)(m->patch * m->patch) * st->ringOut.H * st->ringOut.W;
    L.args.vid_bs = 3 * L.args.vid_cs;
    WAN_TRY(run(L, &st->prof, kKindConvOut, conv_flops(m->conv_out, st->ringOut, FC), st->err_dev, s));
    st->advance.push_back({&st->ringOut, FC});
  }
  // 3. the causal caches: each ring's last two frames become its history
  for (auto& r : st->advance) {
    r.first->base = r.first->slot(r.second);
    r.first->zhist = std::max(0, r.first->zhist - r.second);
  }
  st->first = false;
  if (st->err_host) {
    CUDA_TRY(cudaMemcpyAsync(st->err_host, st->err_dev, sizeof(int), cudaMemcpyDeviceToHost, s));
    CUDA_TRY(cudaEventRecord(st->err_ev, s));
    st->err_pending = true;
  }
  return WAN_OK;
}

static wan_status stream_build(const wan_vae_model* m, int B, int h, int w, int nmax, bool async, cudaStream_t s,
                               wan_vae_stream* st) {
  st->m = m;
  st->B = B;
  st->h = h;
  st->w = w;
  st->nmax = nmax;
  st->mem.use_async = async;
  st->mem.async = s;
  st->ws = nullptr;
  st->ws_used = 0;
  WAN_TRY(plan_buffers(st));
  st->ws_bytes = rup(st->ws_used, 256) + 256;
  void* p;
  WAN_TRY(st->mem.alloc(&p, st->ws_bytes));
  st->ws = (char*)p;
  st->ws_used = 0;
  WAN_TRY(plan_buffers(st));
  WAN_TRY(st->mem.alloc(&p, 256));
  st->err_dev = (int*)p;
  if (async) {
    CUDA_TRY(cudaMemsetAsync(st->ws, 0, st->ws_bytes, s));
    CUDA_TRY(cudaMemsetAsync(st->err_dev, 0, 256, s));
  } else {
    CUDA_TRY(cudaMemset(st->ws, 0, st->ws_bytes));
    CUDA_TRY(cudaMemset(st->err_dev, 0, 256));
    CUDA_TRY(cudaMallocHost((void**)&st->err_host, sizeof(int)));
    *st->err_host = 0;
    CUDA_TRY(cudaEventCreateWithFlags(&st->err_ev, cudaEventDisableTiming));
    CUDA_TRY(cudaDeviceSynchronize());
  }
  st->first = true;
  return WAN_OK;
}

static void stream_free(wan_vae_stream* st) {
  if (!st) return;
  if (!st->mem.use_async) cudaDeviceSynchronize();
  for (int k = 0; k < 2; ++k) {
    if (st->dec_ev[k]) cudaEventDestroy(st->dec_ev[k]);
    if (st->d2h_ev[k]) cudaEventDestroy(st->d2h_ev[k]);
  }
  if (st->copy_stream) cudaStreamDestroy(st->copy_stream);
  st->mem.release();
  if (st->err_host) cudaFreeHost(st->err_host);
  if (st->err_ev) cudaEventDestroy(st->err_ev);
  delete st;
}

static wan_status check_pending_error(wan_vae_stream* st, bool block) {
  if (!st->err_pending) return WAN_OK;
  if (block) {
    CUDA_TRY(cudaEventSynchronize(st->err_ev));
  } else {
    const cudaError_t q = cudaEventQuery(st->err_ev);
    if (q == cudaErrorNotReady) return WAN_OK;
    if (q != cudaSuccess) return fail(WAN_ERR_CUDA, "earlier decode failed: %s", cudaGetErrorString(q));
  }
  st->err_pending = false;
  if (*st->err_host != 0)
    return fail(WAN_ERR_INTERNAL, "a decode kernel reported error %d (a bounded wait expired)", *st->err_host);
  return WAN_OK;
}

static wan_status dtype_ok(int d, const char* what) {
  if (d != WAN_F32 && d != WAN_BF16) return fail(WAN_ERR_DTYPE, "%s: dtype must be WAN_F32 or WAN_BF16, not %d", what, d);
  return WAN_OK;
}

static wan_status decode_chunk_impl(wan_vae_stream* st, const void* z, int z_dtype, long long z_frames, long long t0,
                                    int n, void* out, int out_dtype, long long out_frames, long long out_f0,
                                    float* pre, cudaStream_t s) {
  if (!st) return fail(WAN_ERR_INVALID_ARG, "null stream state");
  if (!z || !out) return fail(WAN_ERR_INVALID_ARG, "null latents or output");
  WAN_TRY(dtype_ok(z_dtype, "latents"));
  WAN_TRY(dtype_ok(out_dtype, "output"));
  if (n < 1 || n > st->nmax) return fail(WAN_ERR_INVALID_ARG, "chunk of %d frames (1..%d allowed)", n, st->nmax);
  if (t0 < 0 || t0 + n > z_frames) return fail(WAN_ERR_INVALID_ARG, "frames %lld..%lld outside z", t0, t0 + n - 1);
  const long long nf = st->first ? 4LL * n - 3 : 4LL * n;
  if (out_f0 < 0 || out_f0 + nf > out_frames)
    return fail(WAN_ERR_INVALID_ARG, "output frames %lld..%lld outside out (%lld frames)", out_f0, out_f0 + nf - 1,
                out_frames);
  WAN_TRY(check_pending_error(st, false));
  return run_chunk(st, z, z_dtype == WAN_F32, z_frames, t0, n, out, out_dtype == WAN_F32, out_frames, out_f0, pre, s);
}

static wan_status reset_impl(wan_vae_stream* st, cudaStream_t s) {
  for (Act* r : st->rings) {
    r->base = 0;
    r->zhist = 2;
    for (int b = 0; b < r->B; ++b) CUDA_TRY(cudaMemsetAsync(r->p + b * r->bs(), 0, 2 * r->fs() * sizeof(bf16), s));
  }
  st->first = true;
  return WAN_OK;
}

static wan_status clip_impl(wan_vae_stream* st, const void* z, int z_dtype, int T, void* out, int out_dtype,
                            float* pre, cudaStream_t s) {
  if (!st) return fail(WAN_ERR_INVALID_ARG, "null stream state");
  if (T < 1) return fail(WAN_ERR_INVALID_ARG, "T = %d", T);
  WAN_TRY(reset_impl(st, s));
  const long long F = 4LL * T - 3;
  long long f0 = 0;
  for (int t0 = 0; t0 < T;) {
    const int n = std::min(st->nmax, T - t0);
    WAN_TRY(decode_chunk_impl(st, z, z_dtype, T, t0, n, out, out_dtype, F, f0, pre, s));
    f0 += (t0 == 0) ? 4LL * n - 3 : 4LL * n;
    t0 += n;
  }
  return WAN_OK;
}

// ------------------------------------------------------------- tiled decode
// Tiles of equal latent size are decoded together as one batch (up to 64
// samples per stream); each batch's output lands in the tile buffer at the
// offsets of its tiles, which are consecutive.  Then the seams are blended
// and the blended tiles assembled into `out`.
static wan_status tiled_impl(const wan_vae_model* m, const void* z, int z_dtype, int B, int T, int h, int w,
                             int tile_h, int tile_w, int stride_h, int stride_w, int tile_batch, int max_chunk,
                             void* out, int out_dtype, cudaStream_t s) {
  const int P = 8 * m->patch;  // pixels per latent
  const int th = tile_h / P, tw = tile_w / P, sh = stride_h / P, sw = stride_w / P;
  std::vector<std::pair<int, int>> rows, cols;  // (origin, size) in latents
  for (int r = 0; r < h; r += sh) rows.push_back({r, std::min(th, h - r)});
  for (int c = 0; c < w; c += sw) cols.push_back({c, std::min(tw, w - c)});
  const int ni = (int)rows.size(), nj = (int)cols.size();
  if ((long long)ni * nj > kMaxTiles) return fail(WAN_ERR_UNSUPPORTED, "%d x %d tiles (at most %d)", ni, nj, kMaxTiles);
  const long long F = 4LL * T - 3, planes = 3LL * B * F;
  // tiles grouped by size, raster order inside a group
  std::vector<std::pair<std::pair<int, int>, int>> order;  // ((rows, cols), raster index)
  for (int i = 0; i < ni; ++i)
    for (int j = 0; j < nj; ++j) order.push_back({{rows[i].second, cols[j].second}, i * nj + j});
  std::stable_sort(order.begin(), order.end(),
                   [](const auto& a, const auto& b) { return a.first < b.first; });
  std::unique_ptr<TileTable> tab(new TileTable());
  tab->ni = ni;
  tab->nj = nj;
  tab->sh = stride_h;
  tab->sw = stride_w;
  long long total = 0;
  size_t zt_elems = 0;
  for (const auto& o : order) {
    TileDesc& t = tab->t[o.second];
    t.h = P * o.first.first;
    t.w = P * o.first.second;
    t.off = total;
    total += planes * t.h * t.w;
  }
  const int per_batch = std::max(1, std::min(tile_batch > 0 ? tile_batch : kMaxGather, std::min(kMaxGather, 64 / B)));
  for (const auto& o : order)
    zt_elems = std::max(zt_elems, (size_t)per_batch * B * m->zdim * T * o.first.first * o.first.second);
  const int zes = z_dtype == WAN_F32 ? 4 : 2;
  DevMem mem;
  mem.use_async = true;
  mem.async = s;
  wan_status r = WAN_OK;
  void *buf = nullptr, *zt = nullptr;
  wan_vae_stream* st = nullptr;
  auto drop_stream = [&]() {
    if (st) {
      st->mem.release();
      delete st;
      st = nullptr;
    }
  };
  do {
    if ((r = mem.alloc(&buf, (size_t)total * sizeof(float))) != WAN_OK) break;
    if ((r = mem.alloc(&zt, zt_elems * zes)) != WAN_OK) break;
    int sb = 0, sh_l = 0, sw_l = 0;  // the current stream's batch and tile size
    for (size_t g0 = 0; g0 < order.size() && r == WAN_OK;) {
      // the next batch: up to per_batch tiles of the same size
      size_t g1 = g0 + 1;
      while (g1 < order.size() && (int)(g1 - g0) < per_batch && order[g1].first == order[g0].first) ++g1;
      const int n = (int)(g1 - g0), rh = order[g0].first.first, cw = order[g0].first.second;
      if (!st || sb != n * B || sh_l != rh || sw_l != cw) {
        drop_stream();
        st = new wan_vae_stream();
        if ((r = stream_build(m, n * B, rh, cw, std::min(T, max_chunk), true, s, st)) != WAN_OK) break;
        sb = n * B;
        sh_l = rh;
        sw_l = cw;
      }
      TileGather gt;
      gt.n = n;
      gt.B = B;
      gt.h = h;
      gt.w = w;
      gt.th = rh;
      gt.tw = cw;
      gt.CT = (long long)m->zdim * T;
      for (int k = 0; k < n; ++k) {
        const int idx = order[g0 + k].second;
        gt.r0[k] = rows[idx / nj].first;
        gt.c0[k] = cols[idx % nj].first;
      }
      if (launch_gather_tiles(z, zes, zt, gt, s) != cudaSuccess) {
        r = fail(WAN_ERR_CUDA, "tile gather launch failed");
        break;
      }
      r = clip_impl(st, zt, z_dtype, T, (float*)buf + tab->t[order[g0].second].off, WAN_F32, nullptr, s);
      g0 = g1;
    }
    if (r != WAN_OK) break;
    if (launch_blend_tiles((float*)buf, *tab, planes, s) != cudaSuccess) {
      r = fail(WAN_ERR_CUDA, "tile blend launch failed");
      break;
    }
    if (launch_assemble_tiles((const float*)buf, *tab, out, out_dtype == WAN_F32, planes, P * h, P * w, s) !=
        cudaSuccess)
      r = fail(WAN_ERR_CUDA, "tile assembly launch failed");
  } while (false);
  drop_stream();
  mem.release();
  return r;
}

// ------------------------------------------------------------- C ABI
#define API_GUARD(...)                                               \
  try {                                                              \
    __VA_ARGS__                                                      \
  } catch (const std::bad_alloc&) {                                  \
    return fail(WAN_ERR_OOM, "host allocation failed");              \
  } catch (...) {                                                    \
    return fail(WAN_ERR_INTERNAL, "unexpected C++ exception");       \
  }

extern "C" {

int64_t wan_vae_out_frames(int64_t T) { return T >= 1 ? 4 * T - 3 : 0; }

const char* wan_vae_last_error(void) { return g_last_error.c_str(); }

const char* wan_vae_status_string(int32_t s) {
  switch (s) {
    case WAN_OK: return "WAN_OK";
    case WAN_ERR_INVALID_ARG: return "WAN_ERR_INVALID_ARG";
    case WAN_ERR_DTYPE: return "WAN_ERR_DTYPE";
    case WAN_ERR_MISSING_WEIGHT: return "WAN_ERR_MISSING_WEIGHT";
    case WAN_ERR_SHAPE: return "WAN_ERR_SHAPE";
    case WAN_ERR_UNSUPPORTED: return "WAN_ERR_UNSUPPORTED";
    case WAN_ERR_OOM: return "WAN_ERR_OOM";
    case WAN_ERR_CUDA: return "WAN_ERR_CUDA";
    case WAN_ERR_STATE: return "WAN_ERR_STATE";
    case WAN_ERR_INTERNAL: return "WAN_ERR_INTERNAL";
    case WAN_ERR_NOT_IMPLEMENTED: return "WAN_ERR_NOT_IMPLEMENTED";
  }
  return "unknown status";
}

wan_status wan_vae_model_create(const wan_tensor* weights, int32_t n_weights, int32_t dtype, wan_cuda_stream stream,
                                wan_vae_model** model) {
  API_GUARD({
    if (!model) return fail(WAN_ERR_INVALID_ARG, "null model output pointer");
    *model = nullptr;
    wan_vae_model* m = new wan_vae_model();
    const wan_status st = model_build_checked(weights, n_weights, dtype, (cudaStream_t)stream, m);
    if (st != WAN_OK) {
      if (!m->mem.ptrs.empty()) cudaStreamSynchronize((cudaStream_t)stream);
      m->mem.release();
      delete m;
      return st;
    }
    *model = m;
    return WAN_OK;
  })
}

void wan_vae_model_destroy(wan_vae_model* model) {
  if (!model) return;
  cudaDeviceSynchronize();
  model->mem.release();
  delete model;
}

int32_t wan_vae_model_base_dim(const wan_vae_model* model) { return model ? model->base : -1; }
int32_t wan_vae_model_z_dim(const wan_vae_model* model) { return model ? model->zdim : -1; }
int32_t wan_vae_model_scale(const wan_vae_model* model) { return model ? 8 * model->patch : -1; }

wan_status wan_vae_model_set_latent_stats(wan_vae_model* model, const float* mean, const float* std_dev, int32_t n) {
  API_GUARD({
    if (!model) return fail(WAN_ERR_INVALID_ARG, "null model");
    if (!mean && !std_dev) {
      model->zstat_on = false;
      return WAN_OK;
    }
    if (!mean || !std_dev) return fail(WAN_ERR_INVALID_ARG, "mean and std must both be given or both be NULL");
    const int zd = model->zdim;
    if (n != zd) return fail(WAN_ERR_SHAPE, "%d latent statistics given, %d expected", n, zd);
    float h[2 * kZdimMax];
    for (int c = 0; c < zd; ++c) {
      h[c] = mean[c];
      h[zd + c] = std_dev[c];
      if (!std::isfinite(h[c]) || !std::isfinite(h[zd + c]))
        return fail(WAN_ERR_INVALID_ARG, "latent statistic of channel %d is not finite", c);
    }
    if (!model->zstat) {
      void* p;
      WAN_TRY(model->mem.alloc(&p, sizeof(h)));
      model->zstat = (float*)p;
    }
    CUDA_TRY(cudaMemcpy(model->zstat, h, 2 * zd * sizeof(float), cudaMemcpyHostToDevice));
    model->zstat_on = true;
    return WAN_OK;
  })
}

wan_status wan_vae_stream_create(const wan_vae_model* model, int32_t B, int32_t h, int32_t w, int32_t max_chunk,
                                 wan_vae_stream** out) {
  API_GUARD({
    if (!out) return fail(WAN_ERR_INVALID_ARG, "null stream output pointer");
    *out = nullptr;
    if (!model) return fail(WAN_ERR_INVALID_ARG, "null model");
    if (B < 1 || h < 1 || w < 1 || max_chunk < 1)
      return fail(WAN_ERR_INVALID_ARG, "B=%d h=%d w=%d max_chunk=%d must be positive", B, h, w, max_chunk);
    if ((long long)8 * h > 65535 || (long long)8 * w > 65535 || max_chunk > 64 || B > 64)
      return fail(WAN_ERR_UNSUPPORTED, "latent %dx%d, batch %d, chunk %d too large", h, w, B, max_chunk);
    wan_vae_stream* st = new wan_vae_stream();
    const wan_status s = stream_build(model, B, h, w, max_chunk, false, nullptr, st);
    if (s != WAN_OK) {
      stream_free(st);
      return s;
    }
    *out = st;
    return WAN_OK;
  })
}

wan_status wan_vae_stream_reset(wan_vae_stream* st, wan_cuda_stream stream) {
  API_GUARD({
    if (!st) return fail(WAN_ERR_INVALID_ARG, "null stream state");
    return reset_impl(st, (cudaStream_t)stream);
  })
}

void wan_vae_stream_destroy(wan_vae_stream* st) { stream_free(st); }

int64_t wan_vae_stream_workspace_bytes(const wan_vae_stream* st) { return st ? (int64_t)st->ws_bytes : 0; }

wan_status wan_vae_stream_sync_status(wan_vae_stream* st, wan_cuda_stream stream) {
  API_GUARD({
    if (!st) return fail(WAN_ERR_INVALID_ARG, "null stream state");
    CUDA_TRY(cudaStreamSynchronize((cudaStream_t)stream));
    CUDA_TRY(cudaGetLastError());
    return check_pending_error(st, true);
  })
}

// ---- causal-cache checkpoint: header + the two history slots of every ring
struct StateHeader {
  uint64_t magic;
  int32_t base, split, B, h, w, first, n_rings;  // split: bit 0 fp32 split format, bit 1 Wan2.1
  int64_t payload;
};
static const uint64_t kStateMagic = 0x57414e5641453031ULL;  // "WANVAE01"

static int64_t state_payload(const wan_vae_stream* st) {
  int64_t n = 0;
  for (const Act* r : st->rings) n += (int64_t)r->B * 2 * r->fs() * (int64_t)sizeof(bf16);
  return n;
}

int64_t wan_vae_stream_state_bytes(const wan_vae_stream* st) {
  return st ? (int64_t)rup(sizeof(StateHeader), 256) + state_payload(st) : 0;
}

wan_status wan_vae_stream_save(wan_vae_stream* st, void* dst, int64_t bytes, wan_cuda_stream stream) {
  API_GUARD({
    if (!st || !dst) return fail(WAN_ERR_INVALID_ARG, "null argument");
    if (bytes < wan_vae_stream_state_bytes(st))
      return fail(WAN_ERR_INVALID_ARG, "state buffer of %lld bytes, %lld needed", (long long)bytes,
                  (long long)wan_vae_stream_state_bytes(st));
    cudaStream_t s = (cudaStream_t)stream;
    StateHeader hd{kStateMagic, st->m->base, (st->m->split ? 1 : 0) | (st->m->wan21 ? 2 : 0), st->B, st->h, st->w, st->first ? 1 : 0,
                   (int32_t)st->rings.size(), state_payload(st)};
    CUDA_TRY(cudaMemcpyAsync(dst, &hd, sizeof(hd), cudaMemcpyDefault, s));
    char* o = static_cast<char*>(dst) + rup(sizeof(StateHeader), 256);
    // each ring's two history frames (logical frames 0 and 1, which may sit
    // at the ring's last and first slots)
    for (const Act* r : st->rings)
      for (int b = 0; b < r->B; ++b)
        for (int f = 0; f < 2; ++f) {
          const size_t n = r->fs() * sizeof(bf16);
          CUDA_TRY(cudaMemcpyAsync(o, r->p + b * r->bs() + r->slot(f) * r->fs(), n, cudaMemcpyDefault, s));
          o += n;
        }
    return WAN_OK;
  })
}

wan_status wan_vae_stream_load(wan_vae_stream* st, const void* src, int64_t bytes, wan_cuda_stream stream) {
  API_GUARD({
    if (!st || !src) return fail(WAN_ERR_INVALID_ARG, "null argument");
    if (bytes < (int64_t)sizeof(StateHeader)) return fail(WAN_ERR_INVALID_ARG, "state buffer too small");
    cudaStream_t s = (cudaStream_t)stream;
    StateHeader hd;
    CUDA_TRY(cudaMemcpyAsync(&hd, src, sizeof(hd), cudaMemcpyDefault, s));
    CUDA_TRY(cudaStreamSynchronize(s));
    if (hd.magic != kStateMagic) return fail(WAN_ERR_INVALID_ARG, "not a decode state");
    if (hd.base != st->m->base || hd.split != ((st->m->split ? 1 : 0) | (st->m->wan21 ? 2 : 0)) || hd.B != st->B || hd.h != st->h ||
        hd.w != st->w || hd.n_rings != (int32_t)st->rings.size() || hd.payload != state_payload(st))
      return fail(WAN_ERR_STATE, "state of a different model, dtype or shape");
    if (bytes < wan_vae_stream_state_bytes(st)) return fail(WAN_ERR_INVALID_ARG, "state buffer truncated");
    const char* o = static_cast<const char*>(src) + rup(sizeof(StateHeader), 256);
    for (Act* r : st->rings) {
      r->base = 0;  // the history goes to slots 0 and 1
      r->zhist = hd.first ? 2 : 0;  // a state saved before the first chunk holds the zero history
      for (int b = 0; b < r->B; ++b) {
        const size_t n = 2 * r->fs() * sizeof(bf16);
        CUDA_TRY(cudaMemcpyAsync(r->p + b * r->bs(), o, n, cudaMemcpyDefault, s));
        o += n;
      }
    }
    st->first = hd.first != 0;
    return WAN_OK;
  })
}

wan_status wan_vae_stream_profile_begin(wan_vae_stream* st) {
  API_GUARD({
    if (!st) return fail(WAN_ERR_INVALID_ARG, "null stream state");
    st->prof.on = true;
    st->prof.launches = 0;
    st->prof.rec.clear();
    return WAN_OK;
  })
}

wan_status wan_vae_stream_profile_end(wan_vae_stream* st, wan_cuda_stream stream, wan_vae_profile* out) {
  API_GUARD({
    if (!st) return fail(WAN_ERR_INVALID_ARG, "null stream state");
    Prof& p = st->prof;
    wan_vae_profile r;
    memset(&r, 0, sizeof(r));
    r.launches = p.launches;

    if (p.on && !p.rec.empty()) {
      CUDA_TRY(cudaStreamSynchronize((cudaStream_t)stream));
      for (size_t i = 0; i < p.rec.size(); ++i) {
        float ms = 0.f;
        CUDA_TRY(cudaEventElapsedTime(&ms, p.ev[2 * i], p.ev[2 * i + 1]));
        const int k = p.rec[i].kind;
        if (k < kKindNorm) {
          r.tc_ms += ms;
          r.tc_flops += p.rec[i].work;
          r.tc_exec_flops += p.rec[i].exec;
          r.tc_launches += 1;
        }
        if (k >= 0 && k < kNumKinds) {
          r.kind_ms[k] += ms;
          r.kind_work[k] += p.rec[i].work;
          r.kind_exec[k] += p.rec[i].exec;
          r.kind_launches[k] += 1;
        }
      }
    }
    p.on = false;
    p.rec.clear();
    if (out) *out = r;
    return WAN_OK;
  })
}

wan_status wan_vae_decode_chunk(wan_vae_stream* st, const void* z, int32_t z_dtype, int64_t z_frames, int64_t t0,
                                int32_t n, void* out, int32_t out_dtype, int64_t out_frames, int64_t out_f0,
                                float* preclamp, wan_cuda_stream stream) {
  API_GUARD({
    return decode_chunk_impl(st, z, z_dtype, z_frames, t0, n, out, out_dtype, out_frames, out_f0, preclamp,
                             (cudaStream_t)stream);
  })
}

wan_status wan_vae_decode_clip(wan_vae_stream* st, const void* z, int32_t z_dtype, int32_t T, void* out,
                               int32_t out_dtype, float* preclamp, wan_cuda_stream stream) {
  API_GUARD({ return clip_impl(st, z, z_dtype, T, out, out_dtype, preclamp, (cudaStream_t)stream); })
}

wan_status wan_vae_decode_clip_host(wan_vae_stream* st, const void* z_host, int32_t z_dtype, int32_t T,
                                    void* out_host, int32_t out_dtype, wan_cuda_stream stream) {
  API_GUARD({
    if (!st || !z_host || !out_host) return fail(WAN_ERR_INVALID_ARG, "null argument");
    WAN_TRY(dtype_ok(z_dtype, "latents"));
    WAN_TRY(dtype_ok(out_dtype, "output"));
    if (T < 1) return fail(WAN_ERR_INVALID_ARG, "T = %d", T);
    cudaStream_t s = (cudaStream_t)stream;
    const size_t zes = z_dtype == WAN_F32 ? 4 : 2, oes = out_dtype == WAN_F32 ? 4 : 2;
    const int zd = st->m->zdim, ppl = 8 * st->m->patch;  // latent channels, pixels per latent
    const long long P = (long long)st->h * st->w, HW = (long long)ppl * ppl * P;
    const int n = st->nmax;
    const long long nfmax = 4LL * n;
    // staging: two latent chunks and two video chunks, kept by the stream
    const size_t zneed = (size_t)st->B * zd * n * P * 4, vneed = (size_t)st->B * 3 * nfmax * HW * 4;
    if (st->zb_bytes < zneed || st->vb_bytes < vneed) {
      for (int k = 0; k < 2; ++k) {
        WAN_TRY(st->mem.alloc(&st->zb[k], zneed));
        WAN_TRY(st->mem.alloc(&st->vb[k], vneed));
      }
      st->zb_bytes = zneed;
      st->vb_bytes = vneed;
    }
    if (!st->copy_stream) {
      CUDA_TRY(cudaStreamCreateWithFlags(&st->copy_stream, cudaStreamNonBlocking));
      for (int k = 0; k < 2; ++k) {
        CUDA_TRY(cudaEventCreateWithFlags(&st->dec_ev[k], cudaEventDisableTiming));
        CUDA_TRY(cudaEventCreateWithFlags(&st->d2h_ev[k], cudaEventDisableTiming));
      }
    }
    cudaStream_t cs = st->copy_stream;
    wan_status result = reset_impl(st, s);
    const long long F = 4LL * T - 3;
    long long f0 = 0;
    int i = 0;
    for (int t0 = 0; t0 < T && result == WAN_OK; ++i) {
      const int k = i & 1;
      const int nn = std::min(n, T - t0);
      const long long nf = t0 == 0 ? 4LL * nn - 3 : 4LL * nn;
      // buffer k is free once the download of chunk i - 2 is done
      if (i >= 2 && cudaStreamWaitEvent(s, st->d2h_ev[k], 0) != cudaSuccess) {
        result = fail(WAN_ERR_CUDA, "cudaStreamWaitEvent failed");
        break;
      }
      // latents of this chunk: rows (b, c) of nn*P values
      if (cudaMemcpy2DAsync(st->zb[k], nn * P * zes, (const char*)z_host + t0 * P * zes, (size_t)T * P * zes,
                            nn * P * zes, (size_t)st->B * zd, cudaMemcpyHostToDevice, s) != cudaSuccess) {
        result = fail(WAN_ERR_CUDA, "latent upload failed");
        break;
      }
      result = decode_chunk_impl(st, st->zb[k], z_dtype, nn, 0, nn, st->vb[k], out_dtype, nfmax, 0, nullptr, s);
      if (result != WAN_OK) break;
      // the download of this chunk's frames overlaps the next chunk's decode
      if (cudaEventRecord(st->dec_ev[k], s) != cudaSuccess || cudaStreamWaitEvent(cs, st->dec_ev[k], 0) != cudaSuccess ||
          cudaMemcpy2DAsync((char*)out_host + f0 * HW * oes, (size_t)F * HW * oes, st->vb[k], nfmax * HW * oes,
                            nf * HW * oes, (size_t)st->B * 3, cudaMemcpyDeviceToHost, cs) != cudaSuccess ||
          cudaEventRecord(st->d2h_ev[k], cs) != cudaSuccess) {
        result = fail(WAN_ERR_CUDA, "video download failed");
        break;
      }
      f0 += nf;
      t0 += nn;
    }
    cudaStreamSynchronize(cs);
    cudaStreamSynchronize(s);
    if (result != WAN_OK) return result;
    return check_pending_error(st, true);
  })
}

wan_status wan_vae_decode(const void* z, int32_t z_dtype, int32_t B, int32_t T, int32_t h, int32_t w,
                          const wan_tensor* weights, int32_t n_weights, void* out, int32_t dtype,
                          wan_cuda_stream stream) {
  API_GUARD({
    WAN_TRY(dtype_ok(dtype, "decode"));
    WAN_TRY(dtype_ok(z_dtype, "latents"));
    if (!z || !out) return fail(WAN_ERR_INVALID_ARG, "null latents or output");
    if (B < 1 || T < 1 || h < 1 || w < 1) return fail(WAN_ERR_INVALID_ARG, "B=%d T=%d h=%d w=%d", B, T, h, w);
    cudaStream_t s = (cudaStream_t)stream;
    wan_vae_model m;
    m.mem.use_async = true;
    m.mem.async = s;
    wan_status r = model_build_checked(weights, n_weights, dtype, s, &m);
    wan_vae_stream* st = nullptr;
    if (r == WAN_OK) {
      st = new wan_vae_stream();
      r = stream_build(&m, B, h, w, std::min(T, 4), true, s, st);
      if (r == WAN_OK) r = clip_impl(st, z, z_dtype, T, out, dtype, nullptr, s);
      st->mem.release();
      delete st;
    }
    m.mem.release();
    return r;
  })
}

wan_status wan_vae_decode_tiled(const wan_vae_model* model, const void* z, int32_t z_dtype, int32_t B, int32_t T,
                                int32_t h, int32_t w, int32_t tile_h, int32_t tile_w, int32_t stride_h,
                                int32_t stride_w, int32_t tile_batch, int32_t max_chunk, void* out, int32_t out_dtype,
                                wan_cuda_stream stream) {
  API_GUARD({
    for (int v : {tile_h, tile_w, stride_h, stride_w})
      if (v <= 0 || v % 16)
        return fail(WAN_ERR_INVALID_ARG, "tile %dx%d, stride %dx%d: positive multiples of 16 pixels needed", tile_h,
                    tile_w, stride_h, stride_w);
    if (stride_h > tile_h || stride_w > tile_w)
      return fail(WAN_ERR_INVALID_ARG, "tile stride %dx%d larger than the tile %dx%d", stride_h, stride_w, tile_h,
                  tile_w);
    if (tile_batch < 0 || max_chunk < 1)
      return fail(WAN_ERR_INVALID_ARG, "tile_batch=%d (>= 0) max_chunk=%d (>= 1)", tile_batch, max_chunk);
    WAN_TRY(dtype_ok(z_dtype, "latents"));
    WAN_TRY(dtype_ok(out_dtype, "output"));
    if (!model) return fail(WAN_ERR_INVALID_ARG, "null model");
    if (!z || !out) return fail(WAN_ERR_INVALID_ARG, "null latents or output");
    if ((uintptr_t)out % 16) return fail(WAN_ERR_INVALID_ARG, "output not 16-byte aligned");
    if (B < 1 || B > 64 || T < 1 || h < 1 || w < 1 || max_chunk > 64)
      return fail(WAN_ERR_INVALID_ARG, "B=%d (1..64) T=%d h=%d w=%d max_chunk=%d (<= 64)", B, T, h, w, max_chunk);
    if ((long long)8 * model->patch * h > 65535 || (long long)8 * model->patch * w > 65535)
      return fail(WAN_ERR_UNSUPPORTED, "frame of %dx%d latents too large", h, w);
    return tiled_impl(model, z, z_dtype, B, T, h, w, tile_h, tile_w, stride_h, stride_w, tile_batch, max_chunk, out,
                      out_dtype, (cudaStream_t)stream);
  })
}

}  // extern "C"

// Packed weights and workspace of the isolated attention block for N frames
// of H x W positions (the layer entry points below).
struct wan_attention {
  int N = 0, H = 0, W = 0, C = 0;
  float* g = nullptr;
  ConvW qkv, proj;
  AttnBufs at;
  int* err = nullptr;
  DevMem mem;
};

static wan_status attention_build(const wan_tensor* weights, int32_t n_weights, int32_t N, int32_t H, int32_t W,
                                  int32_t C, cudaStream_t s, wan_attention* A) {
  if (!weights) return fail(WAN_ERR_INVALID_ARG, "null weights");
  if (N < 1 || H < 1 || W < 1) return fail(WAN_ERR_INVALID_ARG, "N=%d H=%d W=%d", N, H, W);
  if (C % 64 || C < 64 || C > 1024) return fail(WAN_ERR_UNSUPPORTED, "C=%d (multiple of 64, <= 1024)", C);
  // pick the five tensors by suffix
  std::vector<wan_tensor> t;
  const char* suff[5] = {"norm.gamma", "to_qkv.weight", "to_qkv.bias", "proj.weight", "proj.bias"};
  for (const char* sfx : suff) {
    const wan_tensor* hit = nullptr;
    for (int i = 0; i < n_weights; ++i) {
      const char* nm = weights[i].name;
      if (!nm) continue;
      const size_t L = strlen(nm), Ls = strlen(sfx);
      if (L >= Ls && strcmp(nm + L - Ls, sfx) == 0) hit = &weights[i];
    }
    if (!hit) return fail(WAN_ERR_MISSING_WEIGHT, "missing weight '*%s'", sfx);
    wan_tensor c = *hit;
    c.name = sfx;
    t.push_back(c);
  }
  WeightTable wt{t.data(), (int)t.size()};
  A->N = N;
  A->H = H;
  A->W = W;
  A->C = C;
  DevMem& mem = A->mem;
  WAN_TRY(pack_gamma(wt, "norm.gamma", C, &A->g, mem, s));
  WAN_TRY(pack_conv(wt, "to_qkv", 3 * C, C, 1, 1, 1, true, "", 0, A->qkv, mem, s));
  WAN_TRY(pack_conv(wt, "proj", C, C, 1, 1, 1, true, "", 0, A->proj, mem, s));
  AttnBufs& at = A->at;
  at.HW = H * W;
  at.HWs = (int)rup(at.HW, 16);
  at.HWp = (int)rup(at.HW, 64);
  at.Fmax = N;
  at.B = 1;
  at.C = C;
  at.flash = attention_is_flash(false, C);
  auto mk = [&](Act& a, int ch) -> wan_status {
    a.B = 1;
    a.F = N;
    a.H = 1;
    a.W = at.HW;
    a.C = ch;
    a.ldc = ch;
    void* p;
    WAN_TRY(mem.alloc(&p, a.bytes()));
    a.p = (bf16*)p;
    return WAN_OK;
  };
  WAN_TRY(mk(at.an, C));
  WAN_TRY(mk(at.qkv, 3 * C));
  WAN_TRY(mk(at.O, C));
  void* p;
  if (!at.flash) {
    WAN_TRY(mem.alloc(&p, (size_t)at.s_bs() * sizeof(float)));
    at.S = (float*)p;
    WAN_TRY(mem.alloc(&p, (size_t)at.p_bs() * sizeof(bf16)));
    at.P = (bf16*)p;
    CUDA_TRY(cudaMemsetAsync(at.P, 0, (size_t)at.p_bs() * sizeof(bf16), s));
  }
  WAN_TRY(mem.alloc(&p, (size_t)at.vt_bs() * sizeof(bf16)));
  at.Vt = (bf16*)p;
  WAN_TRY(mem.alloc((void**)&A->err, 256));
  CUDA_TRY(cudaMemsetAsync(at.Vt, 0, (size_t)at.vt_bs() * sizeof(bf16), s));
  CUDA_TRY(cudaMemsetAsync(A->err, 0, 256, s));
  return WAN_OK;
}

static wan_status attention_run(wan_attention* A, const void* x, void* out, cudaStream_t s) {
  Act xa, ya;
  xa.p = (bf16*)x;
  ya.p = (bf16*)out;
  for (Act* a : {&xa, &ya}) {
    a->B = 1;
    a->F = A->N;
    a->H = 1;
    a->W = A->at.HW;
    a->C = A->C;
    a->ldc = A->C;
  }
  return attention(A->g, A->qkv, A->proj, A->at, xa, ya, A->N, nullptr, A->err, s);
}

extern "C" {

wan_status wan_attention_block(const void* x, int32_t N, int32_t H, int32_t W, int32_t C, const wan_tensor* weights,
                               int32_t n_weights, void* out, wan_cuda_stream stream) {
  API_GUARD({
    if (!x || !out || !weights) return fail(WAN_ERR_INVALID_ARG, "null argument");
    cudaStream_t s = (cudaStream_t)stream;
    wan_attention A;
    A.mem.use_async = true;
    A.mem.async = s;
    wan_status r = attention_build(weights, n_weights, N, H, W, C, s, &A);
    if (r == WAN_OK) r = attention_run(&A, x, out, s);
    A.mem.release();
    return r;
  })
}

wan_status wan_attention_create(const wan_tensor* weights, int32_t n_weights, int32_t N, int32_t H, int32_t W,
                                int32_t C, wan_cuda_stream stream, wan_attention** out) {
  API_GUARD({
    if (!out) return fail(WAN_ERR_INVALID_ARG, "null output handle");
    *out = nullptr;
    std::unique_ptr<wan_attention> A(new wan_attention());
    WAN_TRY(attention_build(weights, n_weights, N, H, W, C, (cudaStream_t)stream, A.get()));
    CUDA_TRY(cudaStreamSynchronize((cudaStream_t)stream));
    *out = A.release();
    return WAN_OK;
  })
}

wan_status wan_attention_run(wan_attention* A, const void* x, void* out, wan_cuda_stream stream) {
  API_GUARD({
    if (!A || !x || !out) return fail(WAN_ERR_INVALID_ARG, "null argument");
    return attention_run(A, x, out, (cudaStream_t)stream);
  })
}

wan_status wan_attention_status(wan_attention* A, wan_cuda_stream stream) {
  API_GUARD({
    if (!A) return fail(WAN_ERR_INVALID_ARG, "null attention block");
    int code = 0;
    CUDA_TRY(cudaMemcpyAsync(&code, A->err, sizeof(int), cudaMemcpyDeviceToHost, (cudaStream_t)stream));
    CUDA_TRY(cudaStreamSynchronize((cudaStream_t)stream));
    if (code) {
      CUDA_TRY(cudaMemsetAsync(A->err, 0, sizeof(int), (cudaStream_t)stream));
      return fail(WAN_ERR_INTERNAL, "an attention kernel reported error %d (a bounded wait expired)", code);
    }
    return WAN_OK;
  })
}

void wan_attention_destroy(wan_attention* A) {
  if (!A) return;
  cudaDeviceSynchronize();
  A->mem.release();
  delete A;
}

wan_status wan_causal_conv3d(const void* x, int32_t B, int32_t n_hist, int32_t F, int32_t H, int32_t W, int32_t Cin,
                             const void* weight, const void* bias, int32_t w_dtype, int32_t Cout, int32_t kt,
                             int32_t kh, int32_t kw, void* out, wan_cuda_stream stream) {
  API_GUARD({
    if (!x || !weight || !bias || !out) return fail(WAN_ERR_INVALID_ARG, "null argument");
    WAN_TRY(dtype_ok(w_dtype, "weights"));
    if (B < 1 || F < 1 || H < 1 || W < 1 || Cin < 8 || Cout < 16 || n_hist < 0 || n_hist > 2)
      return fail(WAN_ERR_INVALID_ARG, "B=%d F=%d H=%d W=%d Cin=%d Cout=%d n_hist=%d", B, F, H, W, Cin, Cout, n_hist);
    if (Cin % 8 || Cout % 16 || Cin > 4096 || Cout > 4096)
      return fail(WAN_ERR_UNSUPPORTED, "Cin %% 8 and Cout %% 16 must be 0 (Cin=%d Cout=%d)", Cin, Cout);
    for (int k : {kt, kh, kw})
      if (k != 1 && k != 3) return fail(WAN_ERR_UNSUPPORTED, "kernel extents must be 1 or 3");
    if (kt * kh * kw * (((Cin + 63) / 64)) > 0 && kt * kh * kw > kMaxTaps)
      return fail(WAN_ERR_UNSUPPORTED, "too many taps");
    cudaStream_t s = (cudaStream_t)stream;
    wan_tensor t[2] = {{"c.weight", weight, w_dtype, 5, {Cout, Cin, kt, kh, kw}}, {"c.bias", bias, w_dtype, 1, {Cout}}};
    WeightTable wt{t, 2};
    DevMem mem;
    mem.use_async = true;
    mem.async = s;
    wan_status r = WAN_OK;
    do {
      ConvW cw;
      if ((r = pack_conv(wt, "c", Cout, Cin, kt, kh, kw, false, "", 0, cw, mem, s)) != WAN_OK) break;
      // the input with two history slots in front, channels padded to 64
      Act xr;
      xr.B = B;
      xr.F = 2 + F;
      xr.H = H;
      xr.W = W;
      xr.C = Cin;
      xr.ldc = (int)rup(Cin, 64);
      void* p;
      if ((r = mem.alloc(&p, xr.bytes())) != WAN_OK) break;
      xr.p = (bf16*)p;
      int* err;
      if ((r = mem.alloc((void**)&err, 256)) != WAN_OK) break;
      if (cudaMemsetAsync(xr.p, 0, xr.bytes(), s) != cudaSuccess || cudaMemsetAsync(err, 0, 256, s) != cudaSuccess) {
        r = fail(WAN_ERR_CUDA, "memset failed");
        break;
      }
      const long long fs_in = (long long)H * W * Cin;
      FrameView vin{const_cast<void*>(x), (long long)(n_hist + F) * fs_in, fs_in, Cin, 0};
      if (launch_copy_frames(vin, xr.view(2 - n_hist), Cin, B, n_hist + F, H * W, s) != cudaSuccess) {
        r = fail(WAN_ERR_CUDA, "copy failed");
        break;
      }
      ConvLaunch L;
      if ((r = conv_setup(cw, xr, kt == 3 ? 0 : 2, nullptr, 0, F, L)) != WAN_OK) break;
      OutSpec o;
      o.p = out;
      o.fs = (long long)H * W * Cout;
      o.bs = (long long)F * o.fs;
      o.ldc = Cout;
      set_out(L.args, o);
      r = run(L, nullptr, 0, 0.0, err, s);
    } while (false);
    mem.release();
    return r;
  })
}

wan_status wan_conv_out_video(const void* x, int32_t B, int32_t n_hist, int32_t F, int32_t H, int32_t W, int32_t Cin,
                              const void* weight, const void* bias, int32_t w_dtype, int32_t Cout, void* out,
                              int32_t out_dtype, float* preclamp, wan_cuda_stream stream) {
  API_GUARD({
    if (!x || !weight || !bias || !out) return fail(WAN_ERR_INVALID_ARG, "null argument");
    WAN_TRY(dtype_ok(w_dtype, "weights"));
    WAN_TRY(dtype_ok(out_dtype, "output"));
    if (B < 1 || F < 1 || H < 1 || W < 1 || Cin < 8 || n_hist < 0 || n_hist > 2)
      return fail(WAN_ERR_INVALID_ARG, "B=%d F=%d H=%d W=%d Cin=%d n_hist=%d", B, F, H, W, Cin, n_hist);
    if (Cout != 12 && Cout != 3) return fail(WAN_ERR_UNSUPPORTED, "Cout must be 12 (2 x 2 patch) or 3, not %d", Cout);
    if (Cin % 8 || Cin > 1024) return fail(WAN_ERR_UNSUPPORTED, "Cin must be a multiple of 8 up to 1024, not %d", Cin);
    const int patch = Cout == 12 ? 2 : 1;
    cudaStream_t s = (cudaStream_t)stream;
    wan_tensor t[2] = {{"c.weight", weight, w_dtype, 5, {Cout, Cin, 3, 3, 3}}, {"c.bias", bias, w_dtype, 1, {Cout}}};
    WeightTable wt{t, 2};
    DevMem mem;
    mem.use_async = true;
    mem.async = s;
    wan_status r = WAN_OK;
    do {
      TapFoldW tf;
      if ((r = pack_tapfold(wt, "c", Cout, Cin, tf, mem, s)) != WAN_OK) break;
      float* bf;
      if ((r = mem.alloc((void**)&bf, 16 * sizeof(float))) != WAN_OK) break;
      if (cudaMemsetAsync(bf, 0, 16 * sizeof(float), s) != cudaSuccess ||
          launch_to_f32(bias, w_dtype == WAN_F32, nullptr, 0, bf, Cout, 1.0f, 1, s) != cudaSuccess) {
        r = fail(WAN_ERR_CUDA, "bias conversion failed");
        break;
      }
      // the input with two history slots in front, channels padded to 64
      Act xr;
      xr.B = B;
      xr.F = 2 + F;
      xr.H = H;
      xr.W = W;
      xr.C = Cin;
      xr.ldc = (int)rup(Cin, 64);
      void* p;
      if ((r = mem.alloc(&p, xr.bytes())) != WAN_OK) break;
      xr.p = (bf16*)p;
      int* err;
      if ((r = mem.alloc((void**)&err, 256)) != WAN_OK) break;
      if (cudaMemsetAsync(xr.p, 0, xr.bytes(), s) != cudaSuccess || cudaMemsetAsync(err, 0, 256, s) != cudaSuccess) {
        r = fail(WAN_ERR_CUDA, "memset failed");
        break;
      }
      const long long fs_in = (long long)H * W * Cin;
      FrameView vin{const_cast<void*>(x), (long long)(n_hist + F) * fs_in, fs_in, Cin, 0};
      if (launch_copy_frames(vin, xr.view(2 - n_hist), Cin, B, n_hist + F, H * W, s) != cudaSuccess) {
        r = fail(WAN_ERR_CUDA, "copy failed");
        break;
      }
      VideoConvLaunch V;
      if ((r = video_conv_setup(tf, bf, xr, F, patch, V)) != WAN_OK) break;
      V.args.out = out;
      V.args.out_f32 = out_dtype == WAN_F32;
      V.args.preclamp = preclamp;
      V.args.vid_cs = (long long)F * patch * patch * H * W;
      V.args.vid_bs = 3 * V.args.vid_cs;
      V.args.err = err;
      if (launch_video_conv(V, s) != cudaSuccess) {
        r = fail(WAN_ERR_CUDA, "conv_out launch failed: %s", cudaGetErrorString(cudaGetLastError()));
        break;
      }
    } while (false);
    mem.release();
    return r;
  })
}

}  // extern "C"

// ======================================================================
// Failure-detection self test
// ======================================================================
extern "C" wan_status wan_selftest_wait_timeout(int32_t cout, int32_t* device_code, wan_cuda_stream stream) {
  API_GUARD({
    if (device_code) *device_code = 0;
    if (cout != 64 && cout != 96 && cout != 256 && cout != 12)
      return fail(WAN_ERR_INVALID_ARG, "cout must be 64, 96, 256 or 12, not %d", cout);
    cudaStream_t s = (cudaStream_t)stream;
    DevMem mem;
    mem.use_async = true;
    mem.async = s;
    wan_status r = WAN_OK;
    int code = 0;
    if (cout == 12) do {
      // conv_out's tap-folded kernel: 64 -> 12 channels over one 16 x 32
      // frame (two history slots of zeros), the video 32 x 64
      TapFoldW tf;
      tf.Co = 12;
      tf.Ci = 64;
      tf.ci_pad = 64;
      tf.n = video_conv_n(12);
      Act x;
      x.B = 1;
      x.F = 3;
      x.H = 16;
      x.W = 32;
      x.C = 64;
      x.ldc = 64;
      void *pw, *pb, *px, *po, *pe;
      const size_t wb = (size_t)tf.n * 3 * tf.ci_pad * sizeof(bf16), bb = 16 * sizeof(float);
      const size_t ob = (size_t)3 * 4 * x.H * x.W * sizeof(bf16);
      if ((r = mem.alloc(&pw, wb)) || (r = mem.alloc(&pb, bb)) || (r = mem.alloc(&px, x.bytes())) ||
          (r = mem.alloc(&po, ob)) || (r = mem.alloc(&pe, 256)))
        break;
      if (cudaMemsetAsync(pw, 0, wb, s) || cudaMemsetAsync(pb, 0, bb, s) || cudaMemsetAsync(px, 0, x.bytes(), s) ||
          cudaMemsetAsync(pe, 0, 256, s)) {
        r = fail(WAN_ERR_CUDA, "memset failed");
        break;
      }
      tf.w = (bf16*)pw;
      x.p = (bf16*)px;
      VideoConvLaunch V;
      if ((r = video_conv_setup(tf, (const float*)pb, x, 1, 2, V)) != WAN_OK) break;
      V.args.out = po;
      V.args.vid_cs = (long long)4 * x.H * x.W;
      V.args.vid_bs = 3 * V.args.vid_cs;
      V.args.err = (int*)pe;
      V.args.wait_limit = 20000000;  // about 10 ms
      V.args.stall_at1 = 1;          // the first K stage is never loaded
      if (launch_video_conv(V, s) != cudaSuccess) {
        r = fail(WAN_ERR_CUDA, "conv_out launch failed: %s", cudaGetErrorString(cudaGetLastError()));
        break;
      }
      if (cudaMemcpyAsync(&code, pe, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
          cudaStreamSynchronize(s) != cudaSuccess) {
        r = fail(WAN_ERR_CUDA, "reading the error word failed: %s", cudaGetErrorString(cudaGetLastError()));
        break;
      }
    } while (false);
    else do {
      // a causal 3x3x3 conv 64 -> cout over one 16 x 32 frame (two history slots of zeros)
      ConvW cw;
      cw.Co = cout;
      cw.Ci = 64;
      cw.kt = cw.kh = cw.kw = 3;
      cw.ci_pad = 64;
      cw.ktot = 27 * 64;
      cw.bn = choose_bn(cout);
      cw.co_pad = (int)rup(cout, cw.bn);
      Act x;
      x.B = 1;
      x.F = 3;
      x.H = 16;
      x.W = 32;
      x.C = 64;
      x.ldc = 64;
      void *pw, *pb, *px, *po, *pe;
      const size_t wb = (size_t)cw.co_pad * cw.ktot * sizeof(bf16), bb = (size_t)cw.co_pad * sizeof(float);
      const size_t ob = (size_t)x.H * x.W * cout * sizeof(bf16);
      if ((r = mem.alloc(&pw, wb)) || (r = mem.alloc(&pb, bb)) || (r = mem.alloc(&px, x.bytes())) ||
          (r = mem.alloc(&po, ob)) || (r = mem.alloc(&pe, 256)))
        break;
      if (cudaMemsetAsync(pw, 0, wb, s) || cudaMemsetAsync(pb, 0, bb, s) || cudaMemsetAsync(px, 0, x.bytes(), s) ||
          cudaMemsetAsync(pe, 0, 256, s)) {
        r = fail(WAN_ERR_CUDA, "memset failed");
        break;
      }
      cw.w = (bf16*)pw;
      cw.bias = (float*)pb;
      x.p = (bf16*)px;
      ConvLaunch L;
      if ((r = conv_setup(cw, x, 0, nullptr, 0, 1, L)) != WAN_OK) break;
      OutSpec o;
      o.p = po;
      o.fs = (long long)x.H * x.W * cout;
      o.bs = o.fs;
      o.ldc = cout;
      set_out(L.args, o);
      L.args.wait_limit = 20000000;  // about 10 ms
      L.args.stall_at1 = 1;          // the first K stage is never loaded
      if ((r = run(L, nullptr, 0, 0.0, (int*)pe, s)) != WAN_OK) break;
      if (cudaMemcpyAsync(&code, pe, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
          cudaStreamSynchronize(s) != cudaSuccess) {
        r = fail(WAN_ERR_CUDA, "reading the error word failed: %s", cudaGetErrorString(cudaGetLastError()));
        break;
      }
    } while (false);
    mem.release();
    if (r != WAN_OK) return r;
    CUDA_TRY(cudaStreamSynchronize(s));
    if (device_code) *device_code = code;
    if (code) return fail(WAN_ERR_INTERNAL, "a conv kernel reported error %d (a bounded wait expired)", code);
    return WAN_OK;
  })
}

extern "C" wan_status wan_selftest_attention_timeout(int32_t C, int32_t* device_code, wan_cuda_stream stream) {
  API_GUARD({
    if (device_code) *device_code = 0;
    if (!flash_attn_supported(C)) return fail(WAN_ERR_INVALID_ARG, "no flash kernel takes head dim %d", C);
    cudaStream_t s = (cudaStream_t)stream;
    DevMem mem;
    mem.use_async = true;
    mem.async = s;
    wan_status r = WAN_OK;
    int code = 0;
    do {
      // one frame of 200 positions (two query blocks) of zeros
      AttnBufs at;
      at.HW = 200;
      at.HWs = (int)rup(at.HW, 16);
      at.HWp = (int)rup(at.HW, 64);
      at.Fmax = 1;
      at.B = 1;
      at.C = C;
      at.flash = true;
      auto mk = [&](Act& a, int ch) -> wan_status {
        a.B = 1;
        a.F = 1;
        a.H = 1;
        a.W = at.HW;
        a.C = ch;
        a.ldc = ch;
        void* p;
        WAN_TRY(mem.alloc(&p, a.bytes()));
        a.p = (bf16*)p;
        return cudaMemsetAsync(p, 0, a.bytes(), s) == cudaSuccess ? WAN_OK : fail(WAN_ERR_CUDA, "memset failed");
      };
      void *pv, *pe;
      if ((r = mk(at.qkv, 3 * C)) || (r = mk(at.O, C)) ||
          (r = mem.alloc(&pv, (size_t)at.vt_bs() * sizeof(bf16))) || (r = mem.alloc(&pe, 256)))
        break;
      at.Vt = (bf16*)pv;
      if (cudaMemsetAsync(pv, 0, (size_t)at.vt_bs() * sizeof(bf16), s) || cudaMemsetAsync(pe, 0, 256, s)) {
        r = fail(WAN_ERR_CUDA, "memset failed");
        break;
      }
      FlashLaunch FL;
      if ((r = flash_setup(at, 1, (int*)pe, FL)) != WAN_OK) break;
      FL.args.wait_limit = 20000000;  // about 10 ms
      FL.args.stall_at1 = 1;          // the first ring stage is never loaded
      if (launch_flash_attn(FL, s) != cudaSuccess) {
        r = fail(WAN_ERR_CUDA, "flash attention launch failed: %s", cudaGetErrorString(cudaGetLastError()));
        break;
      }
      if (cudaMemcpyAsync(&code, pe, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
          cudaStreamSynchronize(s) != cudaSuccess) {
        r = fail(WAN_ERR_CUDA, "reading the error word failed: %s", cudaGetErrorString(cudaGetLastError()));
        break;
      }
    } while (false);
    mem.release();
    if (r != WAN_OK) return r;
    CUDA_TRY(cudaStreamSynchronize(s));
    if (device_code) *device_code = code;
    if (code) return fail(WAN_ERR_INTERNAL, "the flash attention kernel reported error %d (a bounded wait expired)", code);
    return WAN_OK;
  })
}

// ======================================================================
// wan_causal_conv3d_noalloc: the causal conv with its scratch (packed
// weights, bias, the input copied behind two history slots, the error word)
// carved from a fixed device array instead of the stream-ordered allocator.
// ======================================================================
namespace {

// Scratch limit of the allocation-free entry point.  Every device that loads
// the library holds this array until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;  // 32 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the scratch array, cached per CUDA context.  In host
// code the array's name is only a stand-in: the address is looked up with
// cudaGetSymbolAddress while the calling thread's context is current, once
// per context.  Contexts are told apart by cuCtxGetId, whose ids are never
// reused within a process, so a context created after a cudaDeviceReset (or
// another context made current on the same device) gets its own lookup.
using PfnCtxGetCurrent = CUresult (*)(CUcontext*);
using PfnCtxGetId = CUresult (*)(CUcontext, unsigned long long*);
constexpr size_t kNoAllocMaxContexts = 64;
std::mutex g_noalloc_mu;
std::vector<std::pair<unsigned long long, void*>> g_noalloc_addr;  // (context id, address)

bool current_context_id(unsigned long long* id) {
  static PfnCtxGetCurrent get_current = nullptr;
  static PfnCtxGetId get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = (PfnCtxGetCurrent)fn;
    fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = (PfnCtxGetId)fn;
  });
  CUcontext ctx = nullptr;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
  return get_id(ctx, id) == CUDA_SUCCESS;
}

wan_status noalloc_scratch(char** out) {
  int dev = -1;
  CUDA_TRY(cudaGetDevice(&dev));
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  unsigned long long id = 0;
  if (current_context_id(&id))
    for (const auto& e : g_noalloc_addr)
      if (e.first == id) {
        *out = static_cast<char*>(e.second);
        return WAN_OK;
      }
  // set-up for this context (it also makes the device's primary context
  // current if the thread had none)
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess || !p)
    return fail(WAN_ERR_CUDA, "cudaGetSymbolAddress of the scratch array on device %d failed: %s", dev,
                cudaGetErrorString(e));
  if (current_context_id(&id) && g_noalloc_addr.size() < kNoAllocMaxContexts) g_noalloc_addr.push_back({id, p});
  *out = static_cast<char*>(p);
  return WAN_OK;
}

}  // namespace

extern "C" wan_status wan_causal_conv3d_noalloc(const void* x, int32_t B, int32_t n_hist, int32_t F, int32_t H,
                                                int32_t W, int32_t Cin, const void* weight, const void* bias,
                                                int32_t w_dtype, int32_t Cout, int32_t kt, int32_t kh, int32_t kw,
                                                void* out, wan_cuda_stream stream) {
  API_GUARD({
    if (!x || !weight || !bias || !out) return fail(WAN_ERR_INVALID_ARG, "null argument");
    WAN_TRY(dtype_ok(w_dtype, "weights"));
    if (B < 1 || F < 1 || H < 1 || W < 1 || Cin < 8 || Cout < 16 || n_hist < 0 || n_hist > 2)
      return fail(WAN_ERR_INVALID_ARG, "B=%d F=%d H=%d W=%d Cin=%d Cout=%d n_hist=%d", B, F, H, W, Cin, Cout, n_hist);
    if (Cin % 8 || Cout % 16 || Cin > 4096 || Cout > 4096)
      return fail(WAN_ERR_UNSUPPORTED, "Cin %% 8 and Cout %% 16 must be 0 (Cin=%d Cout=%d)", Cin, Cout);
    for (int k : {kt, kh, kw})
      if (k != 1 && k != 3) return fail(WAN_ERR_UNSUPPORTED, "kernel extents must be 1 or 3");
    if (kt * kh * kw > kMaxTaps) return fail(WAN_ERR_UNSUPPORTED, "too many taps");
    cudaStream_t s = (cudaStream_t)stream;
    // scratch plan: packed weights | bias | input with history slots | error word
    ConvW cw;
    cw.Co = Cout;
    cw.Ci = Cin;
    cw.kt = kt;
    cw.kh = kh;
    cw.kw = kw;
    cw.ci_pad = (int)rup(Cin, 64);
    const int taps = kt * kh * kw;
    cw.ktot = taps * cw.ci_pad;
    cw.bn = choose_bn(Cout);
    cw.co_pad = (int)rup(Cout, cw.bn);
    Act xr;
    xr.B = B;
    xr.F = 2 + F;
    xr.H = H;
    xr.W = W;
    xr.C = Cin;
    xr.ldc = cw.ci_pad;
    const size_t w_bytes = (size_t)cw.co_pad * cw.ktot * sizeof(bf16);
    const size_t off_b = rup(w_bytes, 256);
    const size_t off_x = off_b + rup((size_t)Cout * sizeof(float), 256);
    const size_t off_e = off_x + rup(xr.bytes(), 256);
    const size_t need = off_e + 256;
    if (need > kNoAllocScratchBytes)
      return fail(WAN_ERR_UNSUPPORTED, "this conv needs %zu bytes of scratch; the allocation-free entry point has %zu",
                  need, kNoAllocScratchBytes);
    char* base = nullptr;
    WAN_TRY(noalloc_scratch(&base));
    cw.w = reinterpret_cast<bf16*>(base);
    cw.bias = reinterpret_cast<float*>(base + off_b);
    xr.p = reinterpret_cast<bf16*>(base + off_x);
    int* err = reinterpret_cast<int*>(base + off_e);
    // The array keeps the previous call's contents: clear what must start at
    // zero (weight padding, history slots and channel padding, error word).
    CUDA_TRY(cudaMemsetAsync(cw.w, 0, w_bytes, s));
    CUDA_TRY(cudaMemsetAsync(xr.p, 0, xr.bytes(), s));
    CUDA_TRY(cudaMemsetAsync(err, 0, 256, s));
    CUDA_TRY(launch_pack_weight(weight, w_dtype == WAN_F32, Cout, Cin, taps, cw.w, cw.ktot, 0, cw.ci_pad, s));
    CUDA_TRY(launch_to_f32(bias, w_dtype == WAN_F32, nullptr, 0, cw.bias, Cout, 1.0f, 1, s));
    const long long fs_in = (long long)H * W * Cin;
    FrameView vin{const_cast<void*>(x), (long long)(n_hist + F) * fs_in, fs_in, Cin, 0};
    CUDA_TRY(launch_copy_frames(vin, xr.view(2 - n_hist), Cin, B, n_hist + F, H * W, s));
    ConvLaunch L;
    WAN_TRY(conv_setup(cw, xr, kt == 3 ? 0 : 2, nullptr, 0, F, L));
    OutSpec o;
    o.p = out;
    o.fs = (long long)H * W * Cout;
    o.bs = (long long)F * o.fs;
    o.ldc = Cout;
    set_out(L.args, o);
    return run(L, nullptr, 0, 0.0, err, s);
  })
}
