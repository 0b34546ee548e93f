// Internal launch interface between the C ABI (api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "wan_attn.h"

namespace wan {

constexpr int kHeadDim = 128;
constexpr int kPairsT = 22;  // rotary pairs of the t band at head_dim 128 (44 dims)
constexpr int kPairsH = 21;  // h band (42 dims)
constexpr int kPairsW = 21;  // w band (42 dims)

// Device pointers to the three per-axis float2 {cos, sin} tables.
struct RopeTables {
  const float2* t;  // [F][kPairsT]
  const float2* h;  // [Hp][kPairsH]
  const float2* w;  // [Wp][kPairsW]
};

// Passes of an entry point that the profiling hook can bracket with events
// (the values of the WAN_PASS_* constants of the C ABI).
enum ProfPass : int {
  kPassMain = 0,  // the main kernel (attention, backward, FP8 attention, Conv3d)
  kPassRope = 1,  // the K rotation pre-pass (forward, Ring step, backward)
  kPassRows = 2,  // the backward's row pass (D and LSE * log2 e)
  kPassPost = 3,  // the backward's dQ post-pass (R^T dQ_acc -> bf16)
  kNumPasses = 4,
};

struct LaunchCommon {
  int* err;             // device error word
  uint64_t timeout_ns;  // bound of every device-side wait
  int stall;            // test hook: producer withholds one tile
  int force_check;      // test hook (debug builds): the kernel's entry check fails
  cudaEvent_t ev[kNumPasses][2];  // profiling hook: {start, stop} around each pass (may be null)
};

inline void record_pass(const LaunchCommon& lc, int pass, int which, cudaStream_t s) {
  if (lc.ev[pass][which]) cudaEventRecord(lc.ev[pass][which], s);
}
inline void record_start(const LaunchCommon& lc, cudaStream_t s) { record_pass(lc, kPassMain, 0, s); }
inline void record_stop(const LaunchCommon& lc, cudaStream_t s) { record_pass(lc, kPassMain, 1, s); }

// y = R(pos) x (or R(pos)^T x when inverse) for bf16 [B, L, H, 128]; y may equal x.
cudaError_t launch_rope_rotate_bf16(const void* x, void* y, int B, wan_grid_t g, int H, RopeTables tab,
                                    bool inverse, cudaStream_t s);

// Same for a chunk of L tokens per batch item starting at grid token pos0.
cudaError_t launch_rope_rotate_bf16_rows(const void* x, void* y, int B, int L, int pos0, wan_grid_t g, int H,
                                         RopeTables tab, bool inverse, cudaStream_t s);

// y(bf16) = R(pos)^T x(fp32) for [B, L, H, 128]; used for dQ.
cudaError_t launch_rope_unrotate_f32(const float* x, void* y, int B, wan_grid_t g, int H, RopeTables tab,
                                     cudaStream_t s);

// Backward row pass: D = rowsum(dO * O) and LSE * log2(e) into [B*H][Lpad]
// rows (pad: D = 0, LSE = +inf), for bf16 O, dO [B, L, H, 128] and fp32 LSE
// [B, H, L].
cudaError_t launch_bwd_rows(const void* o, const void* dout, const float* lse, float* lse2, float* drow, int B, int L,
                            int Lpad, int H, cudaStream_t s);

// How the forward epilogue combines this call's result with what o / lse hold.
enum FwdMerge : int {
  kMergeNone = 0,  // o, lse <- this call's attention
  kMergeLse = 1,   // o, lse <- log-sum-exp merge of (o, lse) with this call's (a ring step)
  kMergeAdd = 2,   // o <- o + this call's attention; lse untouched (summed attention paths)
};

// Forward attention. With rope = true (self-attention) q is rotated inside the
// kernel (query row r is grid token q_pos0 + r) and k_rot must already be
// rotated; with rope = false it is plain cross-attention over Lk keys with
// optional per-batch valid lengths.
int launch_attn_fwd(const void* q, const void* k_rot, const void* v, void* o, float* lse, int B, int Lq, int Lk,
                    int H, wan_grid_t g, RopeTables tab, bool rope, const int32_t* kv_lens, float scale,
                    const LaunchCommon& lc, cudaStream_t s, int q_pos0 = 0, int merge = kMergeNone);

// FP8 (e4m3) self-attention forward with per-head scales; the workspace
// holds Q8, K8, the transposed V8 and the per-head amax (attn_fwd_fp8.cu).
size_t attn_fwd_fp8_workspace_bytes(int B, int L, int H);
int launch_attn_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse, int B, wan_grid_t g, int H,
                        RopeTables tab, float scale, void* workspace, const LaunchCommon& lc, cudaStream_t s);

// Backward. Workspace layout is defined in attn_bwd.cu.
size_t attn_bwd_workspace_bytes(int B, int L, int H);
int launch_attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                    void* dq, void* dk, void* dv, int B, wan_grid_t g, int H, RopeTables tab, float scale,
                    void* workspace, const LaunchCommon& lc, cudaStream_t s);

// Causal 3 x 3 x 3 Conv3d of the Wan-VAE on one chunk (conv3d.cu). cache may
// be null (zeros before the chunk). c_in % 32 == 0; conv3d_n_tile(c_out) > 0.
// time_down: the 3 x 1 x 1, time-stride-2 downsampling layer instead (T even,
// a one-frame cache that must be given; T / 2 output frames).
int conv3d_n_tile(int c_out);
int launch_causal_conv3d(const void* x, const void* cache, const void* wt, const float* bias, void* y, int B, int T,
                         int H, int W, int c_in, int c_out, const LaunchCommon& lc, cudaStream_t s,
                         bool time_down = false);

}  // namespace wan
