/*
 * wan_vae.h — C ABI of the GB300 (sm_103a) Wan2.2-TI2V-5B VAE decode.
 *
 * What it computes is defined on the page "wan22_vae_decode/reference.py"
 * (FastVideo; a standalone description of diffusers'
 * AutoencoderKLWan._decode): decode(z, weights, dtype) maps latents
 * z [B, 48, T, H/16, W/16] to a video [B, 3, 4T-3, H, W] in [-1, 1]:
 *   1. post_quant_conv, a 1x1x1 conv 48 -> 48 over all T frames
 *      (module docstring, "What is computed", item 1);
 *   2. the decoder run causally, chunk by chunk, each causal conv carrying the
 *      last two frames of its input to the next chunk (item 2; section
 *      "Causal caches"; section "The first latent frame yields one frame");
 *   3. unpatchify, video[b, k, f, 2y+i, 2x+j] = out[b, 4k+2j+i, f, y, x]
 *      (item 3);
 *   4. clamp to [-1, 1] (item 4).
 *
 * The same entry points decode with the Wan2.1 VAE (AutoencoderKLWan of the
 * Wan 2.1 and Wan 2.2 A14B pipelines; page "Fix the Wan VAE attention
 * block": z_dim 16, 8x spatial compression, the same attention block) when
 * given its weights: z [B, 16, T, H/8, W/8] -> video [B, 3, 4T-3, H, W], no
 * unpatchify.  Its remaining dimensions are not on the pages and follow that
 * model's published configuration (base dim 96; up blocks 4b -> 4b,
 * 2b -> 4b, 2b -> 2b, b -> b; resamplers halving the channels, no DupUp3D;
 * conv_out to 3 colours).  Below, "48" and "16h" read "16" and "8h" for it
 * (wan_vae_model_z_dim, wan_vae_model_scale).
 *
 * Conventions (all entry points):
 *  - Pointers named as device pointers are CUDA device memory owned by the
 *    caller; they must stay valid until the work enqueued on `stream`
 *    completes.  The library never frees caller memory.
 *  - All work is enqueued on the caller's stream; no entry point blocks the
 *    host unless its comment says so.
 *  - Every call returns a wan_status; nothing is thrown across the ABI.  The
 *    calling thread's last error message is available from
 *    wan_vae_last_error().
 *  - Arithmetic runs in the library's CUDA kernels; there is no CPU path.  If
 *    no CUDA device is present, calls that would launch work return
 *    WAN_ERR_CUDA.
 */
#ifndef WAN_VAE_H
#define WAN_VAE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream (cudaStream_t); NULL is the legacy default stream. */
typedef struct CUstream_st* wan_cuda_stream;

typedef enum {
  WAN_OK = 0,
  WAN_ERR_INVALID_ARG = 1,      /* null pointer, non-positive size, bad option */
  WAN_ERR_DTYPE = 2,            /* dtype not WAN_F32 / WAN_BF16 (the page's ValueError) */
  WAN_ERR_MISSING_WEIGHT = 3,   /* a required parameter name is absent */
  WAN_ERR_SHAPE = 4,            /* a tensor shape disagrees with the architecture */
  WAN_ERR_UNSUPPORTED = 5,      /* valid input this build does not handle */
  WAN_ERR_OOM = 6,              /* device allocation failed */
  WAN_ERR_CUDA = 7,             /* a CUDA runtime/driver call failed */
  WAN_ERR_STATE = 8,            /* handle used out of order */
  WAN_ERR_INTERNAL = 9,         /* a kernel reported an error (e.g. a bounded wait expired) */
  WAN_ERR_NOT_IMPLEMENTED = 10
} wan_status;

/* Element types.  WAN_F32: IEEE fp32.  WAN_BF16: bfloat16 (top half of an fp32). */
typedef enum { WAN_F32 = 0, WAN_BF16 = 1 } wan_dtype;

/* One parameter of the weight table, under diffusers' names ("decoder.*",
 * "post_quant_conv.*"; other names are ignored, as the page's decode keeps
 * only those two prefixes).  `data` is device memory, contiguous, in PyTorch
 * layout: conv3d weights [Cout, Cin, kt, kh, kw], conv2d weights
 * [Cout, Cin, kh, kw], biases [Cout], RMS-norm gammas any shape of C values. */
typedef struct {
  const char* name;
  const void* data;
  int32_t dtype;    /* wan_dtype */
  int32_t ndim;     /* 1..5 */
  int64_t shape[5];
} wan_tensor;

typedef struct wan_vae_model wan_vae_model;
typedef struct wan_vae_stream wan_vae_stream;

/* Output frames of a T-frame latent: 4T - 3 for T >= 1 (page section "The
 * first latent frame yields one frame"), 0 for T < 1.  Host only. */
int64_t wan_vae_out_frames(int64_t T);

/* Message of the calling thread's last failed call ("" if none). */
const char* wan_vae_last_error(void);

/* Name of a status code. */
const char* wan_vae_status_string(int32_t status);

/* Packs the 110 decoder + post_quant_conv tensors (Wan2.1: its decoder's
 * tensors, resamplers named up_blocks.i.upsamplers.0.*) into a library-owned model
 * (conv weights K-major with per-tap channel blocks padded to 64; biases and
 * sqrt(C)*gamma held as fp32; in WAN_BF16 mode every tensor is first rounded
 * to bf16, as the page's bf16 contract rounds the weights).  The
 * architecture is inferred from post_quant_conv.weight ([48, 48, 1, 1, 1]:
 * TI2V-5B; [16, 16, 1, 1, 1]: Wan2.1) and decoder.conv_in.weight
 * [4b, z, 3, 3, 3] (decoder base dim b); every other shape is checked
 * against them.  `dtype` is the decode precision: WAN_BF16 computes with bf16
 * operands and fp32 accumulation (the page's section "Precision", bf16
 * mode; every weight is rounded to bf16 first).  WAN_F32 keeps fp32 values
 * throughout: each weight and activation is held as a pair of bf16 halves
 * (hi = bf16(v), lo = bf16(v - hi)) and every product is formed as
 * hi*hi + hi*lo + lo*hi on the tensor cores with fp32 accumulation, about
 * 16 significant bits per operand (three times the MMA work of WAN_BF16).
 * The caller's tensors may be freed once the work enqueued on `stream` is
 * done.  Errors: WAN_ERR_INVALID_ARG, WAN_ERR_DTYPE, WAN_ERR_MISSING_WEIGHT,
 * WAN_ERR_SHAPE, WAN_ERR_OOM, WAN_ERR_CUDA. */
wan_status wan_vae_model_create(const wan_tensor* weights, int32_t n_weights, int32_t dtype,
                                wan_cuda_stream stream, wan_vae_model** model);
/* Frees the model (synchronises with the device; no work may be pending). */
void wan_vae_model_destroy(wan_vae_model* model);
/* Decoder base dim b of a model (256 for TI2V-5B, 96 for Wan2.1), or -1 for NULL. */
int32_t wan_vae_model_base_dim(const wan_vae_model* model);
/* Latent channels of a model: 48 (TI2V-5B) or 16 (Wan2.1); -1 for NULL. */
int32_t wan_vae_model_z_dim(const wan_vae_model* model);
/* Video pixels per latent along each spatial axis: 16 (TI2V-5B: 8x decoder
 * upsampling, then the 2x2 unpatchify) or 8 (Wan2.1); -1 for NULL. */
int32_t wan_vae_model_scale(const wan_vae_model* model);

/* Latent de-normalisation in front of the decode (the diffusers Wan VAE's
 * per-channel `latents_mean` / `latents_std` configuration lists, page
 * "[Feature] Implement tiled VAE encoding/decoding for Wan model. #11414";
 * the page gives neither values nor formula).  With statistics set, every
 * decode through this model (one-shot excepted: it has no model handle,
 * streams and tiled decodes included) first maps each latent to
 * z * std[c] + mean[c] in fp32, inside the post_quant_conv kernel, and then
 * applies the decode's own input rounding (bf16 models round the result).
 * mean, std_dev: HOST arrays of n = z_dim (48 or 16) finite fp32 values, copied before
 * return (synchronous copy); both NULL switches it off again.  Call it between
 * decodes, never while a decode that uses the model is in flight.
 * Errors: WAN_ERR_INVALID_ARG (null model, one of the two NULL, a value not
 * finite), WAN_ERR_SHAPE (n != z_dim), WAN_ERR_OOM, WAN_ERR_CUDA. */
wan_status wan_vae_model_set_latent_stats(wan_vae_model* model, const float* mean, const float* std_dev, int32_t n);

/* A decode stream: the causal caches (two frames per 3-frame conv, page
 * section "Causal caches") and the activation workspace for latents of
 * B x h x w, decoding at most `max_chunk` latent frames per call.  The
 * workspace is allocated here (one device allocation) and zero-filled; the
 * stream starts at the first chunk.  Errors: WAN_ERR_INVALID_ARG, WAN_ERR_OOM,
 * WAN_ERR_CUDA, WAN_ERR_UNSUPPORTED (h or w not representable). */
wan_status wan_vae_stream_create(const wan_vae_model* model, int32_t B, int32_t h, int32_t w, int32_t max_chunk,
                                 wan_vae_stream** stream_state);
/* Forgets all history (clears the caches on `stream`); the next chunk is a
 * first chunk again. */
wan_status wan_vae_stream_reset(wan_vae_stream* st, wan_cuda_stream stream);
/* Frees the stream state (synchronises with the device). */
void wan_vae_stream_destroy(wan_vae_stream* st);
/* Bytes of device workspace the stream holds. */
int64_t wan_vae_stream_workspace_bytes(const wan_vae_stream* st);
/* Blocks until the stream's enqueued work is done and reports any error a
 * kernel recorded (WAN_ERR_INTERNAL with a message) or a CUDA error. */
wan_status wan_vae_stream_sync_status(wan_vae_stream* st, wan_cuda_stream stream);

/* Checkpoint / resume of a decode.  A stream's state between chunks is the
 * causal caches (page section "Causal caches": the last two input frames of
 * every 3-frame conv) and whether the next chunk is a first chunk.
 * state_bytes: size of a saved state.  save: copies it, stream-ordered, to
 * `dst` (device or host memory, at least state_bytes).  load: restores a
 * state saved from a stream of the same model precision, base dim, B, h, w
 * (WAN_ERR_STATE otherwise); it blocks to read the header, then enqueues the
 * copies on `stream`.  A decode continued after load produces the frames the
 * saved stream would have produced. */
int64_t wan_vae_stream_state_bytes(const wan_vae_stream* st);
wan_status wan_vae_stream_save(wan_vae_stream* st, void* dst, int64_t bytes, wan_cuda_stream stream);
wan_status wan_vae_stream_load(wan_vae_stream* st, const void* src, int64_t bytes, wan_cuda_stream stream);

/* Device-side timing of the stream's work (for benchmarks).  Between
 * profile_begin and profile_end every launch is bracketed by CUDA events on
 * the launching stream; profile_end waits for the stream, sums the events and
 * reports them by kind with their algorithmic work: nominal FLOPs for the
 * tensor-core (implicit-GEMM) kinds (2*M*N*K per conv, zero-padded taps
 * included), bytes read + written for the memory-bound kinds.
 * kind index: 0 causal 3x3x3 convs (conv_in, residual blocks), 1 time convs,
 * 2 upsample2d convs (+DupUp3D), 3 attention GEMMs, 4 conv_out,
 * 5 RMS norm (+SiLU), 6 other memory-bound kernels (post_quant_conv, softmax,
 * transposes, frame copies).  Executed FLOPs count the arithmetic the
 * kernels run: equal to nominal except for the upsample2d convs, which run in
 * sub-pixel form (four 2x2 phase convs at the low resolution: 4/9 of the
 * nominal 3x3 conv at the high resolution), and the attention core at head
 * dims 512 and 1024, whose C / 256 CTAs per 128 queries each compute the
 * scores ((C / 256 + 1) / 2 of the nominal q k^T and P V FLOPs). */
typedef struct {
  int64_t launches;          /* all kernel launches enqueued */
  int64_t tc_launches;       /* tensor-core launches among them */
  double tc_ms;              /* their summed device time */
  double tc_flops;           /* their nominal FLOPs */
  double kind_ms[7];
  double kind_work[7];       /* nominal FLOPs (kinds 0-4) or bytes (kinds 5-6) */
  int64_t kind_launches[7];
  double tc_exec_flops;      /* executed FLOPs of the tensor-core launches */
  double kind_exec[7];       /* executed FLOPs (kinds 0-4; equal to kind_work for 5-6) */
} wan_vae_profile;
wan_status wan_vae_stream_profile_begin(wan_vae_stream* st);
wan_status wan_vae_stream_profile_end(wan_vae_stream* st, wan_cuda_stream stream, wan_vae_profile* out);

/* Decodes latent frames t0 .. t0+n-1 of z [B, 48, z_frames, h, w] (device,
 * NCDHW, z_dtype) as the next chunk of the stream (page functions decode /
 * decode_chunk; 1 <= n <= max_chunk).  Writes 4n - 3 video frames on the
 * stream's first chunk, 4n on later ones, into out [B, 3, out_frames, 16h, 16w]
 * (device, out_dtype) at frames out_f0 ... .  If `preclamp` is not NULL it
 * receives the same frames before the clamp, fp32, same layout as out.
 * Errors: WAN_ERR_INVALID_ARG (sizes, frame ranges), WAN_ERR_DTYPE, WAN_ERR_CUDA,
 * WAN_ERR_INTERNAL (an earlier chunk's kernel reported an error). */
wan_status wan_vae_decode_chunk(wan_vae_stream* st, const void* z, int32_t z_dtype, int64_t z_frames, int64_t t0,
                                int32_t n, void* out, int32_t out_dtype, int64_t out_frames, int64_t out_f0,
                                float* preclamp, wan_cuda_stream stream);

/* Resets the stream and decodes all T latent frames of z [B, 48, T, h, w]
 * into out [B, 3, 4T-3, 16h, 16w], in chunks of max_chunk frames. */
wan_status wan_vae_decode_clip(wan_vae_stream* st, const void* z, int32_t z_dtype, int32_t T, void* out,
                               int32_t out_dtype, float* preclamp, wan_cuda_stream stream);

/* As wan_vae_decode_clip, with z and out in HOST memory (page-locked memory
 * is recommended): copies each chunk's latents in, decodes, and copies each
 * chunk's frames out while the next chunk decodes.  Blocks the host until the
 * video is in `out_host`.  The first call allocates two latent and two video
 * staging chunks (fp32-sized, so either dtype fits) and a copy stream; the
 * stream keeps them for later calls and frees them in wan_vae_stream_destroy. */
wan_status wan_vae_decode_clip_host(wan_vae_stream* st, const void* z_host, int32_t z_dtype, int32_t T,
                                    void* out_host, int32_t out_dtype, wan_cuda_stream stream);

/* Tiled decode (the diffusers pull request "[Feature] Implement tiled VAE
 * encoding/decoding for Wan model. #11414": opt-in spatial tiling, tiles of a
 * sample-space size placed at a sample-space stride, defaults 256 and 192).
 * Decodes z [B, 48, T, h, w] (device, z_dtype) into out [B, 3, 4T-3, 16h, 16w]
 * (device, out_dtype) as overlapping tiles:
 *   - along each axis tiles start at 0, stride, 2*stride, ... (every start
 *     inside the frame) and hold min(tile, remaining) pixels;
 *   - each tile's latents are decoded on their own, exactly as
 *     wan_vae_decode_clip would decode them (own causal caches, chunks of
 *     max_chunk latent frames, unpatchify and clamp), into fp32;
 *   - in raster order each tile cross-fades its top rows with the tile above
 *     and then its left columns with the tile to its left, over the e pixels
 *     the two share: local row (column) k < e becomes
 *     earlier * (e - k) / e + this * k / e;
 *   - tile (i, j) supplies the pixels from its origin to the next origin.
 * The pages fix the interface, not the blend; this is the plainest reading.
 * tile_h, tile_w, stride_h, stride_w: video pixels, positive multiples of 16,
 * stride <= tile (stride == tile: no blending).  tile_batch: tiles of equal
 * size decoded together as one batch (0 = as many as fit in 64 samples);
 * smaller values lower the peak workspace.  At most 1024 tiles.
 * Memory: stream-ordered allocations released before return (fp32 tiles of
 * the whole video, plus one decode workspace at a time); no host
 * synchronisation.  `out` must be 16-byte aligned.  Errors: WAN_ERR_INVALID_ARG
 * (sizes, null pointers, alignment; the
 * tile arguments are checked first), WAN_ERR_DTYPE, WAN_ERR_UNSUPPORTED (too
 * many tiles), WAN_ERR_OOM, WAN_ERR_CUDA. */
wan_status wan_vae_decode_tiled(const wan_vae_model* model, const void* z, int32_t z_dtype, int32_t B, int32_t T,
                                int32_t h, int32_t w, int32_t tile_h, int32_t tile_w, int32_t stride_h,
                                int32_t stride_w, int32_t tile_batch, int32_t max_chunk, void* out, int32_t out_dtype,
                                wan_cuda_stream stream);

/* One-shot decode (the page's decode(z, weights, dtype)): packs the weights,
 * decodes z [B, 48, T, h, w] (device, z_dtype) into out [B, 3, 4T-3, 16h, 16w]
 * (device, `dtype`) and releases its temporaries, all stream-ordered
 * (stream-ordered allocator; no host synchronisation). */
wan_status wan_vae_decode(const void* z, int32_t z_dtype, int32_t B, int32_t T, int32_t h, int32_t w,
                          const wan_tensor* weights, int32_t n_weights, void* out, int32_t dtype,
                          wan_cuda_stream stream);

/* ---- layer entry points (the building blocks, exposed for testing) ----
 * The one-shot layer calls below are stream-ordered and do not wait for the
 * device: a bounded wait that runs out inside their kernels (about 2 s; it
 * does not happen in normal operation) is recorded in a temporary error word
 * that they do not read back.  The stream API reports such records
 * (wan_vae_stream_sync_status, and the next chunk), as does
 * wan_attention_status for a packed attention block. */

/* The mid-block attention (page section "What is computed", "The parts",
 * fourth bullet, WanAttentionBlock), per frame: n = RMS norm of x; q, k, v =
 * channels [0,C), [C,2C), [2C,3C) of a 1x1 conv C -> 3C of n; single-head
 * softmax(q k^T / sqrt(C)) v over the H*W positions; a 1x1 conv C -> C;
 * plus x.  x, out: [N][H*W][C] bf16 channels-last (device); weights: the
 * five tensors named *norm.gamma, *to_qkv.weight, *to_qkv.bias, *proj.weight,
 * *proj.bias.  C must be a multiple of 64 and at most 1024.  Temporaries come
 * from the stream-ordered allocator. */
wan_status wan_attention_block(const void* x, int32_t N, int32_t H, int32_t W, int32_t C, const wan_tensor* weights,
                               int32_t n_weights, void* out, wan_cuda_stream stream);

/* The same attention block with its weights packed once: create packs the
 * five tensors (as wan_attention_block names them) and sizes a workspace
 * for N frames of H x W positions at C channels (device memory owned by the
 * handle until destroy; blocks until the packing is done); run computes out =
 * block(x) for x, out [N][H*W][C] bf16 channels-last (device), stream-ordered,
 * no allocation; destroy waits for the device and frees.  Head dims up to
 * 384, 512 and 1024 run a flash kernel (online softmax; the HW x HW scores
 * never leave the SM); other head dims run a score GEMM, a row softmax and a
 * P V GEMM over an fp32 score workspace of N*HW*HW values.  Errors as
 * wan_attention_block. */
typedef struct wan_attention wan_attention;
wan_status wan_attention_create(const wan_tensor* weights, int32_t n_weights, int32_t N, int32_t H, int32_t W,
                                int32_t C, wan_cuda_stream stream, wan_attention** out);
wan_status wan_attention_run(wan_attention* block, const void* x, void* out, wan_cuda_stream stream);
/* Waits for `stream`, then reports a bounded-wait timeout that any earlier
 * run of this block recorded on the device (WAN_ERR_INTERNAL, and the record
 * is cleared), or WAN_OK. */
wan_status wan_attention_status(wan_attention* block, wan_cuda_stream stream);
void wan_attention_destroy(wan_attention* block);

/* One causal conv (page "The parts", first bullet, WanCausalConv3d): x
 * [B][n_hist + F][H][W][Cin] bf16 channels-last (device), its first n_hist
 * (0..2) frames being the conv's history; zero padding kh//2, kw//2 in space
 * and 2*(kt//2) frames in time (history first, zeros for the missing ones).
 * weight [Cout, Cin, kt, kh, kw] (w_dtype), bias [Cout] (w_dtype), kt, kh,
 * kw in {1, 3}.  out [B][F][H][W][Cout] bf16 (device).  Cout must be a
 * multiple of 16.  Temporaries come from the stream-ordered allocator. */
wan_status wan_causal_conv3d(const void* x, int32_t B, int32_t n_hist, int32_t F, int32_t H, int32_t W, int32_t Cin,
                             const void* weight, const void* bias, int32_t w_dtype, int32_t Cout, int32_t kt,
                             int32_t kh, int32_t kw, void* out, wan_cuda_stream stream);

/* The decoder's conv_out and what follows it (page section "What is
 * computed", item 2: norm_out, SiLU, then a causal 3x3x3 conv to 3 colours x
 * 2 x 2 patch channels; items 3-4: unpatchify and clamp), as the bf16 decode
 * runs it: the kernel that folds the nine spatial taps into the GEMM's N.
 * x [B][n_hist + F][H][W][Cin] bf16 channels-last (device), the conv's input
 * (already normalised), its first n_hist (0..2) frames being history; zero
 * padding 1 in space and zeros for the missing history frames.  weight
 * [Cout, Cin, 3, 3, 3], bias [Cout] (w_dtype, rounded to bf16).  Cout 12:
 * out [B][3][F][2H][2W], channel 4k + 2j + i -> colour k, row 2y + i, column
 * 2x + j; Cout 3: out [B][3][F][H][W].  Values clamped to [-1, 1] in
 * out_dtype; preclamp (optional, fp32, same shape) receives them before the
 * clamp.  Cin: a multiple of 8 up to 1024.  Temporaries come from the
 * stream-ordered allocator. */
wan_status wan_conv_out_video(const void* x, int32_t B, int32_t n_hist, int32_t F, int32_t H, int32_t W, int32_t Cin,
                              const void* weight, const void* bias, int32_t w_dtype, int32_t Cout, void* out,
                              int32_t out_dtype, float* preclamp, wan_cuda_stream stream);

/* Failure-detection self test (the pages have no counterpart: it exercises
 * this library's own bounded waits).  Runs one small causal conv (64 -> cout
 * channels: cout 64 for the one-CTA kernel, 256 for the two-CTA cluster
 * kernel, 96 for the row-tile kernel whose CTA pairs on adjacent rows share
 * B, 12 for conv_out's tap-folded kernel) whose TMA producer withholds its
 * first stage, with the wait limit
 * shortened to about 10 ms: the MMA issuer's wait runs out, every role of the
 * kernel drains its copies and exits, and the kernel leaves an error code in
 * its device error word.  Blocks until done.  Returns WAN_ERR_INTERNAL and
 * the code (1..3) in *device_code when the timeout was detected and reported,
 * WAN_OK if it was not; the CUDA context stays usable either way. */
wan_status wan_selftest_wait_timeout(int32_t cout, int32_t* device_code, wan_cuda_stream stream);

/* The same self test for the flash attention kernels: one frame of 200
 * positions at head dim C (up to 384: the one-CTA kernel; 512 or 1024: the
 * kernel with C / 256 CTAs per 128 queries), zeros in, the TMA producer
 * withholding its first ring stage, the wait limit about 10 ms.  Blocks until
 * done.  Returns WAN_ERR_INVALID_ARG if no flash kernel takes C,
 * WAN_ERR_INTERNAL and the code (1..3) in *device_code when the timeout was
 * detected and reported, WAN_OK if it was not; the context stays usable. */
wan_status wan_selftest_attention_timeout(int32_t C, int32_t* device_code, wan_cuda_stream stream);

/* wan_causal_conv3d without any device allocation.  The pages have no
 * counterpart: this is for callers that must not allocate device memory --
 * code that runs while a host framework owns all GPU memory through its own
 * pool, or that must not pay cudaMalloc's implicit device-wide
 * synchronisation on a latency-critical path.  Same arguments, layout and
 * result as wan_causal_conv3d; the caller still provides x, the weights and
 * out.  The scratch (packed weights, bias, a copy of x behind two history
 * slots, an error word) lives in one fixed 32 MiB device array inside the
 * library, which every GPU that loads the library holds until the process
 * exits; a conv whose scratch exceeds 32 MiB is rejected with
 * WAN_ERR_UNSUPPORTED before any work is enqueued.  The first call in a
 * CUDA context (per device, and again after a cudaDeviceReset) looks up the
 * array's device address with cudaGetSymbolAddress while that context is
 * current; make that first call before any stream capture.  All calls in one
 * context share that device's array: each call clears the parts that must
 * start at zero, and calls whose work overlaps on the same device (different
 * streams, or different host threads) race on it -- serialise them.  Calls on
 * different devices use different copies of the array and do not race. */
wan_status wan_causal_conv3d_noalloc(const void* x, int32_t B, int32_t n_hist, int32_t F, int32_t H, int32_t W,
                                     int32_t Cin, const void* weight, const void* bias, int32_t w_dtype,
                                     int32_t Cout, int32_t kt, int32_t kh, int32_t kw, void* out,
                                     wan_cuda_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* WAN_VAE_H */
