/*
 * wan_attn.h - C ABI of the B300 (sm_103a) attention library for Wan-style
 * video diffusion transformers.
 *
 * What the library computes (sources are the web pages about the Wan report,
 * arXiv 2503.20314, cited by page and section):
 *   - full, non-causal spatio-temporal self-attention over all latent tokens
 *     ("Wan Team, Alibaba (2025)" anthology note, Key takeaways; ctol.digital
 *     article, Engineering the Core);
 *   - 3D RoPE on Q and K with temporal / height / width bands (gojay.top
 *     "Wan2.1" paper reading, sections 费曼一分钟 and DiT 块);
 *   - tokens of a (1,2,2)-patchified latent grid, L = F * Hp * Wp (same page,
 *     DiT backbone);
 *   - cross-attention from video tokens to at most 512 umT5 text tokens (same
 *     page, config table ⑥ 1.3B vs 14B; aipaper.jasonlin.tech summary, Key
 *     contributions);
 *   - the backward pass used by rectified-flow training (gojay.top page,
 *     section 3 Training).
 * The pages fix no constants beyond these; the library's readings are: RoPE
 * pairs are adjacent dims (2j, 2j+1); the t, h, w bands are contiguous, of
 * widths d - 4*(d/6), 2*(d/6), 2*(d/6) (44/42/42 at d = 128); pair j of a band
 * of width w turns by pos * theta^(-2j/w); positions are the 0-based grid
 * coordinates; token l = (t*Hp + h)*Wp + w; logits are scale * <q_rot, k_rot>;
 * LSE is the natural log-sum-exp of the scaled logits.
 *
 * Conventions shared by every entry point
 *   - Tensors Q, K, V, O, dO, dQ, dK, dV are bf16 (raw 16-bit storage), layout
 *     [B, L, H, head_dim], contiguous, head_dim innermost. LSE is fp32 [B, H, L].
 *   - Every pointer argument except `tables`-free ones named below is a DEVICE
 *     pointer, 16-byte aligned, owned by the caller. The library never
 *     allocates or frees on these paths; outputs must not alias inputs.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream). All work is enqueued asynchronously on it; a return of WAN_OK
 *     means the work was launched, not that it finished.
 *   - Only head_dim == 128 and devices of compute capability 10.3 are
 *     supported (WAN_ERR_UNSUPPORTED otherwise).
 *   - Arguments are checked on the host before anything is enqueued; on any
 *     error nothing is launched. A device-side bounded wait that expires is
 *     reported later through wan_get_device_status().
 */
#ifndef WAN_ATTN_H
#define WAN_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  WAN_OK = 0,
  WAN_ERR_INVALID = 1,     /* null pointer, bad size, misalignment, small workspace */
  WAN_ERR_UNSUPPORTED = 2, /* head_dim != 128, or the device is not sm_103 */
  WAN_ERR_CUDA = 3,        /* a CUDA call or launch failed */
  WAN_ERR_TIMEOUT = 4,     /* a device-side bounded wait expired (reported by wan_get_device_status) */
  WAN_ERR_DEVICE_CHECK = 5 /* a debug build's device-side invariant check failed (likewise) */
};

enum { WAN_OP_FWD = 0, WAN_OP_BWD = 1, WAN_OP_FWD_FP8 = 2 };

/* Latent token grid: F latent frames x Hp x Wp patches, L = F * Hp * Wp. */
typedef struct {
  int F, Hp, Wp;
} wan_grid_t;

/* Human-readable name of a status code (static string). */
const char* wan_status_str(int status);

/* Library version, major * 10000 + minor * 100 + patch. */
int wan_version(void);

/*
 * 3D RoPE tables (gojay.top "Wan2.1" reading, 费曼一分钟 / DiT 块: 3D RoPE).
 * Bytes needed for the tables of grid g: (F*nt + Hp*nh + Wp*nw) * 8 with
 * nt, nh, nw the rotary pairs of the t, h, w bands (22, 21, 21 at d = 128).
 * Returns 0 for an invalid grid or head_dim.
 */
size_t wan_rope3d_tables_size(wan_grid_t g, int head_dim);

/*
 * Fill `tables_dev` (device, wan_rope3d_tables_size bytes) with float2
 * {cos, sin} of pos * theta^(-2j/w) for every position of each axis, computed
 * in double precision on the host and rounded to fp32: first the t table
 * [F][nt], then h [Hp][nh], then w [Wp][nw]. The copy is enqueued on
 * `stream`; the host staging buffer is released before return.
 */
int wan_rope3d_tables(wan_grid_t g, int head_dim, double theta, float* tables_dev, void* stream);

/*
 * Workspace bytes for op WAN_OP_FWD (self-attention forward: RoPE'd keys),
 * WAN_OP_BWD (backward: rotated Q and K, the fp32 dQ accumulator and the row
 * dot products D = rowsum(dO * O)) or WAN_OP_FWD_FP8 (FP8 forward: e4m3 Q, K,
 * transposed V and the per-head scales).
 */
size_t wan_attn_workspace_size(int op, int B, wan_grid_t g, int H, int head_dim);

/*
 * Self-attention forward with 3D RoPE (anthology note, Key takeaways: full
 * spatio-temporal self-attention; gojay.top reading, DiT 块: 3D RoPE).
 *   q, k, v : [B, L, H, 128] bf16 inputs (pre-RoPE q and k)
 *   o       : [B, L, H, 128] bf16 output, softmax(scale * q_rot k_rot^T) v
 *   lse     : [B, H, L] fp32 output, natural log-sum-exp of each row (may be NULL)
 *   tables  : device tables from wan_rope3d_tables for the same grid/head_dim
 *   scale   : logit scale (1/sqrt(128) for the Wan models)
 *   workspace, ws_bytes : device scratch of at least wan_attn_workspace_size(WAN_OP_FWD, ...)
 * B == 0 is a no-op returning WAN_OK. The call only enqueues kernels on
 * `stream` (no allocation, no synchronisation): after a first call on the
 * device it can be captured in a CUDA graph, whose replays compute on the
 * buffers' current contents.
 */
int wan_attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, wan_grid_t g, int H,
                 int head_dim, const float* tables, float scale, void* workspace, size_t ws_bytes,
                 void* stream);

/*
 * Cross-attention forward, video queries to padded text keys, no RoPE
 * (gojay.top reading, DiT backbone: text enters through cross-attention;
 * config table: umT5 with 512 tokens).
 *   q       : [B, Lq, H, 128] bf16, Lq = F * Hp * Wp of grid g
 *   k, v    : [B, Lk, H, 128] bf16, 1 <= Lk <= 512
 *   kv_lens : device int32 [B] valid key counts, or NULL for all Lk valid.
 *             Values are clamped to [0, Lk] on the device; a row with no
 *             valid key gets O = 0 and LSE = -inf.
 *   o, lse  : outputs as for wan_attn_fwd (lse may be NULL).
 */
int wan_xattn_fwd(const void* q, const void* k, const void* v, const int32_t* kv_lens, int Lk, void* o,
                  float* lse, int B, wan_grid_t g, int H, int head_dim, float scale, void* stream);

/*
 * Self-attention backward with 3D RoPE (gojay.top reading, 3 Training: the
 * rectified-flow step needs gradients through attention).
 *   q, k, v, o, lse : forward inputs and outputs (lse from wan_attn_fwd)
 *   dout            : [B, L, H, 128] bf16 upstream gradient
 *   dq, dk, dv      : [B, L, H, 128] bf16 gradients w.r.t. the pre-RoPE q, k and v
 *   workspace       : at least wan_attn_workspace_size(WAN_OP_BWD, ...) bytes
 * dQ is accumulated with fp32 atomics, so it is reproducible only to rounding.
 */
int wan_attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                 void* dq, void* dk, void* dv, int B, wan_grid_t g, int H, int head_dim, const float* tables,
                 float scale, void* workspace, size_t ws_bytes, void* stream);

/*
 * FP8 self-attention forward with 3D RoPE (anthology note, Key takeaways:
 * FP8 attention; ctol.digital article, "Speed, Scale, and Efficiency": FP8
 * quantisation among the inference speed-ups). Same arguments, layouts and
 * results as wan_attn_fwd; internally Q_rot, K_rot and V are quantised to
 * e4m3 with one scale per (b, h) and tensor (amax / 448), P to e4m3, and both
 * MMAs run as kind::f8f6f4 with fp32 accumulation. Accuracy is that of e4m3
 * (3 mantissa bits), about 7% relative RMS error on O for N(0,1) inputs.
 *   workspace: at least wan_attn_workspace_size(WAN_OP_FWD_FP8, B, g, H, 128) bytes
 * lse is required to be 4-byte aligned when given (it may be NULL).
 */
int wan_attn_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse, int B, wan_grid_t g, int H,
                     int head_dim, const float* tables, float scale, void* workspace, size_t ws_bytes,
                     void* stream);

/*
 * One step of Ring attention on one GPU: attention of a chunk of queries over
 * a chunk of keys of the same video, merged into a running result (anthology
 * note, Key takeaways, and ctol.digital article, "Speed, Scale, and
 * Efficiency": Wan trains long sequences with 2D context parallelism, Ring
 * Attention across devices and Ulysses inside; a Ring step attends to the
 * K/V chunk it holds and merges the partial result by log-sum-exp).
 *   q        : [B, q_len, H, 128] bf16, grid tokens q_start .. q_start+q_len-1 (pre-RoPE)
 *   k, v     : [B, kv_len, H, 128] bf16, grid tokens kv_start .. kv_start+kv_len-1 (k pre-RoPE)
 *   o, lse   : [B, q_len, H, 128] bf16 and [B, H, q_len] fp32 (lse required)
 *   accumulate = 0: o, lse <- attention over this K/V chunk.
 *   accumulate = 1: (o, lse) <- merge of the running (o, lse) with this
 *              chunk's (O_c, LSE_c): LSE = log(e^lse + e^LSE_c),
 *              O = (e^lse o + e^LSE_c O_c) / e^LSE. A running lse of -inf
 *              counts as empty.
 *   tables   : RoPE tables of grid g (positions are the tokens' grid coordinates)
 *   workspace: at least wan_attn_workspace_size(WAN_OP_FWD, B, g, H, 128)
 *              bytes (it holds the chunk's rotated keys).
 * 0 <= q_start, 1 <= q_len, q_start + q_len <= F*Hp*Wp, and the same for kv.
 * Stepping over all K/V chunks of a sequence reproduces wan_attn_fwd up to
 * rounding (o is rounded to bf16 after every step).
 */
int wan_attn_fwd_ring_step(const void* q, const void* k, const void* v, void* o, float* lse, int B, wan_grid_t g,
                           int H, int head_dim, const float* tables, float scale, int q_start, int q_len,
                           int kv_start, int kv_len, int accumulate, void* workspace, size_t ws_bytes,
                           void* stream);

/*
 * Decoupled cross-attention of image-to-video models: the video queries
 * attend separately to the text tokens and to the image tokens (a CLIP image
 * embedding projected to the model width) and the two results are added
 * (anthology note, Key takeaways: the CLIP image embedding enters through
 * decoupled cross-attention; gojay.top reading, section 6 Extended
 * Applications and code map ④ WanModel T2V / I2V: two attention paths, then
 * summed). The pages do not give the number of image tokens.
 *   q                : [B, Lq, H, 128] bf16, Lq = F*Hp*Wp
 *   k_txt, v_txt     : [B, Lk_txt, H, 128], lens_txt: device int32 [B] or NULL (all valid)
 *   k_img, v_img     : [B, Lk_img, H, 128], lens_img: device int32 [B] or NULL
 *   o                : softmax(q k_txt^T) v_txt + softmax(q k_img^T) v_img (bf16)
 *   lse              : optional [B, H, Lq], the log-sum-exp of the text path
 * 1 <= Lk_txt, Lk_img <= 512. No RoPE. Two launches on `stream`.
 */
int wan_xattn_fwd_dual(const void* q, const void* k_txt, const void* v_txt, const int32_t* lens_txt, int Lk_txt,
                       const void* k_img, const void* v_img, const int32_t* lens_img, int Lk_img, void* o,
                       float* lse, int B, wan_grid_t g, int H, int head_dim, float scale, void* stream);

/*
 * Synchronise `stream`, then return and clear the device error word of the
 * current device: WAN_OK, or WAN_ERR_TIMEOUT if a kernel gave up a bounded
 * wait since the last call (its outputs are then undefined), or WAN_ERR_CUDA
 * if the synchronisation itself failed.
 */
int wan_get_device_status(void* stream);

/*
 * Debug builds. The library built with -DWAN_DEBUG (libwan_attn_debug.so)
 * checks, inside its kernels, invariants they rely on: 1024-byte aligned
 * shared-memory bases, the TMEM allocation starting at lane 0 / column 0,
 * tile coordinates inside the problem, 16-byte aligned TMA inner
 * coordinates. The first failure is written to the device error word
 * without a trap; wan_get_device_status then returns WAN_ERR_DEVICE_CHECK
 * and wan_debug_check_line gives the source line of the failed check.
 *   wan_debug_build        : 1 for the debug library, 0 for the release one.
 *   wan_debug_inject_check : test hook; the next `count` kernel launches fail
 *                            their entry check (and skip no work). Debug
 *                            builds only: WAN_ERR_UNSUPPORTED otherwise,
 *                            WAN_ERR_INVALID for count < 0.
 *   wan_debug_check_line   : the line recorded by the last
 *                            WAN_ERR_DEVICE_CHECK status (0 if none yet).
 */
int wan_debug_build(void);
int wan_debug_inject_check(int count);
int wan_debug_check_line(void);

/*
 * Profiling hook: when `start` and `stop` (cudaEvent_t passed as void*) are
 * non-NULL, the next attention entry point records `start` on its stream
 * immediately before its main attention kernel and `stop` immediately after
 * it, so that cudaEventElapsedTime isolates that kernel from the pre- and
 * post-passes. The hook applies to one call and then clears itself; pass
 * NULL, NULL to clear it explicitly. The events stay owned by the caller.
 */
int wan_profile_set_events(void* start, void* stop);

/*
 * The same hook for one pass of an entry point: WAN_PASS_MAIN (the main
 * kernel, as wan_profile_set_events), WAN_PASS_ROPE (the K rotation
 * pre-pass of wan_attn_fwd, wan_attn_fwd_ring_step and wan_attn_bwd),
 * WAN_PASS_ROWS (the row pass of wan_attn_bwd: D = rowsum(dO * O) and
 * LSE * log2 e) or WAN_PASS_POST (the dQ post-pass of wan_attn_bwd:
 * R^T dQ_acc -> bf16). Events set for several passes are all consumed, and
 * cleared, by the next entry-point call; a pass that call does not run
 * leaves its events unrecorded. WAN_ERR_INVALID for an unknown pass or
 * exactly one NULL event.
 */
enum { WAN_PASS_MAIN = 0, WAN_PASS_ROPE = 1, WAN_PASS_ROWS = 2, WAN_PASS_POST = 3 };
int wan_profile_set_pass_events(int pass, void* start, void* stop);

/*
 * Test hook (not for production use): make the next `count` main-kernel
 * launches (attention forward, cross-attention, backward, FP8 forward or VAE
 * Conv3d) skip one producer arrival so that their consumers' bounded waits
 * expire after `timeout_ms`, exercising the timeout path without faulting.
 * count = 0 restores normal operation.
 */
int wan_debug_inject_stall(int count, int timeout_ms);

/*
 * Allocation-free variant of wan_attn_fwd. The Wan pages have no counterpart
 * of this entry point; it exists for callers that cannot allocate device
 * memory themselves: a host framework or plugin interface that hands the
 * library only its input and output buffers and offers no workspace, a
 * process whose device memory is entirely held by another allocator, or a
 * latency-critical caller that must not pay cudaMalloc's implicit device
 * synchronisation.
 *
 * Arguments, layout, results and errors are those of wan_attn_fwd, without
 * the workspace. The rotated keys go to a fixed scratch array that the
 * library keeps in device memory (a file-scope __device__ array of
 * WAN_NOALLOC_SCRATCH_BYTES = 64 MiB, held on every GPU that loads the
 * library until the process exits). So:
 *   - B * L * H must not exceed WAN_NOALLOC_MAX_ROW_HEADS (262,144, e.g. one
 *     32,760-token video with 8 heads); larger problems return
 *     WAN_ERR_INVALID before anything is enqueued;
 *   - the library itself allocates nothing here (no cudaMalloc, cudaFree or
 *     allocating library call);
 *   - every call on a device shares the same scratch, which keeps the last
 *     call's contents (each call overwrites all of the part it reads); two
 *     calls whose work overlaps on the GPU (e.g. on two streams without an
 *     ordering between them) race on it and give undefined results;
 *   - the first call on each device looks up the scratch array's device
 *     address (cudaGetSymbolAddress, with that device current), and so does
 *     the first call after the device's context has been re-created (e.g.
 *     by cudaDeviceReset); make that first call before any stream capture
 *     on the device.
 */
#define WAN_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)
#define WAN_NOALLOC_MAX_ROW_HEADS (WAN_NOALLOC_SCRATCH_BYTES / 256u)
int wan_attn_fwd_noalloc(const void* q, const void* k, const void* v, void* o, float* lse, int B, wan_grid_t g,
                         int H, int head_dim, const float* tables, float scale, void* stream);

/*
 * One causal 3D convolution layer of the Wan-VAE on one chunk of frames, with
 * its feature cache (gojay.top "Wan2.1" reading, Feature Cache section and
 * Fig. vae_cache (a): a time kernel of 3 reads frames t-2, t-1 and t; the
 * first chunk is padded with two zero frames in time, every later chunk is
 * prefixed with the previous chunk's last two input frames, so that chunked
 * processing equals one convolution over the whole video).
 *
 *   y[b,t,h,w,o] = bias[o] + sum_{kt,kh,kw,c} weight[o,kt,kh,kw,c] * xp[b, t+kt, h+kh-1, w+kw-1, c]
 *
 * with xp = (cache, or two zero frames) ++ x in time and zero outside the
 * picture (a cross-correlation, stride 1, 3 x 3 x 3 kernel).
 *   x         : [B, T, H, W, c_in]  bf16, channels last (device)
 *   cache     : [B, 2, H, W, c_in]  bf16, the previous chunk's last two input frames,
 *               or NULL for a first chunk (zeros)
 *   weight    : [c_out, 3, 3, 3, c_in] bf16
 *   bias      : [c_out] fp32, or NULL
 *   y         : [B, T, H, W, c_out] bf16 (output; must not overlap the inputs)
 *   cache_out : [B, 2, H, W, c_in] bf16, receives the last two frames of
 *               (cache or zeros) ++ x for the next chunk; may be NULL, and may
 *               be the same buffer as cache (it is written after the
 *               convolution has read cache, in stream order)
 * c_in and c_out must be multiples of 32 (WAN_ERR_UNSUPPORTED otherwise; a
 * C_in that is not a multiple of 64, such as the 96 channels of the VAE's
 * outer stages, is reduced in 32-channel steps); bf16 pointers 16-byte
 * aligned, bias 4-byte aligned. B = 0 is a no-op.
 * The reduction is accumulated in fp32 on tensor cores; y is rounded to bf16.
 */
int wan_vae_causal_conv3d(const void* x, const void* cache, const void* weight, const float* bias, void* y,
                          void* cache_out, int B, int T, int H, int W, int c_in, int c_out, void* stream);

/*
 * One time-downsampling layer of the Wan-VAE encoder on one chunk of frames,
 * with its one-frame feature cache (gojay.top "Wan2.1" reading, Feature
 * Cache section and Fig. vae_cache (b): a causal temporal convolution of
 * stride 2 whose cache holds the previous chunk's last input frame, so that
 * chunks of 1, 4, 4, ... frames give the same outputs as the whole video).
 * Readings: the kernel is 3 frames x 1 x 1 pixels with no padding; a first
 * chunk is one frame and passes through unchanged.
 *
 *   later chunk (cache given, T even):
 *     y[b,t,h,w,o] = bias[o] + sum_{kt,c} weight[o,kt,c] * xq[b, 2t+kt, h, w, c],
 *     t < T/2, xq = cache ++ x in time;
 *   first chunk (cache NULL): T must be 1 and c_out == c_in; y = x.
 *
 *   x         : [B, T, H, W, c_in]  bf16, channels last (device)
 *   cache     : [B, 1, H, W, c_in]  bf16, the previous chunk's last input
 *               frame, or NULL for a first chunk
 *   weight    : [c_out, 3, c_in] bf16 (not read for a first chunk; may be NULL there)
 *   bias      : [c_out] fp32, or NULL (not read for a first chunk)
 *   y         : [B, T/2, H, W, c_out] bf16 for a later chunk, [B, 1, H, W, c_in]
 *               for a first one (output; must not overlap the inputs)
 *   cache_out : [B, 1, H, W, c_in] bf16, receives x's last frame for the next
 *               chunk; may be NULL, and may be the same buffer as cache (it is
 *               written after the convolution has read cache, in stream order)
 * c_in and c_out must be multiples of 32 (WAN_ERR_UNSUPPORTED otherwise); an
 * odd T with a cache, or a first chunk of T != 1 or c_out != c_in, is
 * WAN_ERR_INVALID. bf16 pointers 16-byte aligned, bias 4-byte aligned. B = 0
 * is a no-op. fp32 accumulation on tensor cores; y is rounded to bf16.
 */
int wan_vae_time_downsample(const void* x, const void* cache, const void* weight, const float* bias, void* y,
                            void* cache_out, int B, int T, int H, int W, int c_in, int c_out, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* WAN_ATTN_H */
