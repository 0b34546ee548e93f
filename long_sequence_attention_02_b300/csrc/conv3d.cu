// Causal 3 x 3 x 3 Conv3d of the Wan-VAE with its feature cache, for sm_103a:
// an implicit GEMM on tcgen05 tensor cores.
//
// What is computed (gojay.top "Wan2.1" reading, Feature Cache section and
// Fig. vae_cache (a)): for one chunk of T frames,
//   y[b,t,h,w,o] = bias[o] + sum_{kt,kh,kw,c} wt[o,kt,kh,kw,c] * xp[b, t+kt, h+kh-1, w+kw-1, c],
// where xp is the chunk with its two past frames in front of it in time (the
// cache, i.e. the previous chunk's last two input frames, or zeros for the
// first chunk) and zero outside the picture. Activations are channels-last
// bf16 [B, T, H, W, C]; weights [C_out, 3, 3, 3, C_in] bf16; bias fp32.
//
// GEMM view: M = output positions, N = C_out, K = 27 taps x C_in. One CTA
// computes a tile of 128 positions x N channels, N = C_out when C_out <= 256,
// else the largest of 256, 192, 128, 64 and 32 that divides C_out. The
// positions are a strip of 128 consecutive pixels of one image row when the
// width is a multiple of 128 (or nearly so), else an 8 (h) x 16 (w) patch.
// When N <= 128 a strip tile holds two strips (rows h0 and h0 + 1), each
// with its own accumulator, so that every weight box feeds 256 positions.
// Per K step (one tap, kc = 64 input channels, or 32 when C_in is not a
// multiple of 64):
// - A = the 128 input pixels that tap reads, kc channels each, from a 5D TMA
//   box at the tap's offset. Its zero fill outside the tensor is the spatial
//   padding, and, for a first chunk, the causal padding too (a negative frame
//   coordinate). With a cache, taps that reach before the chunk read the cache
//   tensor instead. For a strip, one box of 130 pixels (the strip and one
//   pixel either side; one such row per strip of the tile) serves the three
//   taps kw = 0, 1, 2 of a row: the MMA descriptor of tap kw starts kw rows
//   into it. The swizzle is a function of the shared-memory address, so a
//   descriptor may start at any row.
// - B = the tap's N x kc weights: one 3D box {kc c, 1 tap, N}.
// Both land swizzled (rows of 2 kc bytes, 128- or 64-byte swizzle), and kc/16
// tcgen05.mma of kind::f16 (K = 16 each) accumulate into TMEM.
//
// Warps: 0 TMA producer of A, 6 TMA producer of B (A and B have rings of
// their own, since an A box may serve three taps), 1 MMA issuer and TMEM
// owner, 2-5 epilogue (TMEM -> + bias -> bf16 -> shared memory -> TMA stores
// of 32 channels, which write only the positions inside the picture).
// The CTAs are persistent (one per SM) and keep two sets of accumulators in
// TMEM (one accumulator per strip of a tile), so that one tile's epilogue
// runs under the next tile's MMAs.
// Every wait is bounded; on a timeout the device error word is set.
//
// The same kernel, instantiated for kModeTimeDown, runs the encoder's
// time-downsampling layer (Fig. vae_cache (b)): 3 x 1 x 1 taps, stride 2 in
// time, a one-frame cache, K = 3 taps x C_in; output frame t of a chunk
// reads its input frames 2t - 1 (the cache for t = 0), 2t and 2t + 1.
#include <climits>

#include "common.cuh"
#include "kernels.cuh"

namespace wan {

namespace {

constexpr int kConvThreads = 224;
constexpr int kMaxStages = 16;                // slots per ring (mbarrier arrays)
constexpr int kRingBytes = 208 * 1024;        // a strip's A and B rings together

// The epilogue stages 32 output channels of a tile (128 positions x 64 bytes,
// 64-byte swizzle) for one TMA store; two such buffers alternate.
constexpr int kOutStage = 128 * 64;

// Byte offset of 16-byte chunk `chunk` (0..3) of row `row` in a 64-byte-row
// tile in the SWIZZLE_64B layout: chunk bits 4-5 of the address XOR bits 7-8.
__device__ __forceinline__ uint32_t sw64_offset(uint32_t row, uint32_t chunk) {
  return row * 64u + ((chunk ^ ((row >> 1) & 3u)) << 4);
}

__device__ __forceinline__ void tma_store_5d(const CUtensorMap* map, const void* src, int c0, int c1, int c2, int c3,
                                             int c4) {
  asm volatile("cp.async.bulk.tensor.5d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3, %4, %5}], [%6];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(smem_u32(src))
               : "memory");
}

// One K step covers kC input channels of one tap: 64 (rows of 128 bytes,
// 128-byte swizzle) when C_in is a multiple of 64, else 32 (rows of 64 bytes,
// 64-byte swizzle) for layers such as the VAE's 96-channel ones.
//
// Patch tiles keep the {A, B} ring geometry fixed at compile time: stages of
// 128 A rows + 256 B rows (N up to 256), 4 of 48 KB or 8 of 24 KB. (The same
// layout with run-time stage count and strides measured about 8 % slower.)
// Strip rings depend on N, so the host sizes them.
template <int kC>
struct ConvCfg {
  static constexpr int kRow = kC * 2;                       // bytes per row of A and B
  static constexpr uint32_t kSwizzle = kC == 64 ? 2u : 4u;  // descriptor layout: SWIZZLE_128B / SWIZZLE_64B
  static constexpr uint32_t kPatchStage = (128 + 256) * kRow;
  static constexpr int kPatchStages = 192 * 1024 / kPatchStage;
};

struct ConvArgs {
  const float* bias;     // [C_out] or null
  int B, T, H, W, c_in, c_out, n_tile;  // T: output frames (half the input's for time downsampling)
  int ph, pw;            // positions of a tile: 1 or 2 x 128 (strips) or 8 x 16 (patch)
  int tiles_h, tiles_w, tiles_n;
  int n_tiles_total;     // B * tiles_h * tiles_w * T * tiles_n
  uint32_t tmem_cols;    // power of two >= 2 x (strips per tile) x n_tile
  int has_cache;
  // Rings in shared memory: A slot k at k * a_stride, B slot k at b_off +
  // k * b_stride, the two output staging buffers at out_off; all multiples
  // of 1024 bytes. For patches B slot k goes with A slot k (one {A, B}
  // stage), and a_full / a_empty cover both.
  int a_stages, b_stages;
  uint32_t a_bytes;      // bytes one A box brings (its rows x 2 kc)
  uint32_t a_stride, b_stride, b_off, out_off;
  LaunchCommon lc;
};

// Output tile index -> (b, t, tile row, tile column, channel tile). The
// channel tile runs fastest, then the frame, then the tile column: CTAs
// that run at the same time work on neighbouring tiles of all frames, so
// the input windows they share (the two past frames of a tap, the halo of a
// tile) are read from L2 rather than DRAM.
struct ConvTile {
  int b, t, h0, w0, n0;
};
__device__ __forceinline__ ConvTile conv_tile(int idx, const ConvArgs& a) {
  ConvTile x;
  const int nt = idx % a.tiles_n;
  idx /= a.tiles_n;
  x.t = idx % a.T;
  idx /= a.T;
  const int tw = idx % a.tiles_w;
  idx /= a.tiles_w;
  const int th = idx % a.tiles_h;
  x.b = idx / a.tiles_h;
  x.h0 = th * a.ph;
  x.w0 = tw * a.pw;
  x.n0 = nt * a.n_tile;
  return x;
}

__device__ __forceinline__ void tma_load_5d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1, int c2,
                                            int c3, int c4) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void conv_abort(volatile int* abort, int* err) {
  *abort = 1;
  atomicCAS(err, 0, kDevTimeout);
}

// Position in a ring of `stages` slots: the slot of the next fill and how
// many times the ring has wrapped (the parity of the barrier phase).
struct RingPos {
  int slot = 0, round = 0;
  __device__ __forceinline__ void next(int stages) {
    if (++slot == stages) {
      slot = 0;
      ++round;
    }
  }
};

// Every fill a producer issued lands before the CTA may exit: the last fill
// of each slot is that barrier's latest phase (a fill withheld by the test
// hook just lets its wait run out).
__device__ __forceinline__ void drain_ring(uint64_t* full, int fills, int stages, uint64_t to) {
  for (int k = fills - stages < 0 ? 0 : fills - stages; k < fills; ++k)
    mbar_wait(&full[k % stages], (k / stages) & 1, nullptr, to);
}

// Shared-memory matrix descriptor of a K-major tile with rows of kRow bytes
// in the swizzle matching the TMA box: bits [0,14) start >> 4, [16,30) LBO >> 4
// (unused for these K-major swizzled tiles), [32,46) SBO >> 4 (8 rows),
// [46,48) = 1 (tcgen05 descriptor version), [49,52) base offset = 0 (the
// swizzle follows the address bits, whatever row the descriptor starts at),
// [61,64) swizzle mode.
template <int kC>
__device__ __forceinline__ uint64_t conv_desc(uint32_t saddr) {
  constexpr uint32_t kSbo = 8 * ConvCfg<kC>::kRow;
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(kSbo >> 4) << 32) | (1ull << 46) |
         ((uint64_t)ConvCfg<kC>::kSwizzle << 61);
}

// Persistent: one CTA per SM walks the output tiles blockIdx.x,
// blockIdx.x + gridDim.x, ... The A and B rings run on across tiles, and
// TMEM holds two accumulators, so the epilogue of one tile overlaps the MMAs
// of the next.
//
// A tile's K loop: for each group of taps (the three kw of one (kt, kh) for
// a strip, one tap for a patch) and each kc-channel chunk, one A box, then
// one B box and kc/16 MMAs per tap of the group. For patches, A and B of a
// step travel together on one barrier (warp 6 idles); for strips they have
// producers and barriers of their own.
//
// kModeTimeDown selects the time-downsampling layer (Fig. vae_cache (b)):
// 3 x 1 x 1 taps with stride 2 in time; output frame t reads frames 2t - 1,
// 2t and 2t + 1 of the chunk, frame -1 being the one cached frame.
// kModeStrip2 stacks two strips (image rows h0 and h0 + 1) in one tile, with
// an accumulator each: a 2-row input box serves both, and each weight box
// feeds both strips' MMAs (for N <= 128, so that 2 x 2 accumulators fit TMEM).
enum ConvMode : int { kModePatch = 0, kModeStrip = 1, kModeTimeDown = 2, kModeStrip2 = 3 };

template <int kC, int kMode>
__global__ void __launch_bounds__(kConvThreads, 1)
    causal_conv3d_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_cache,
                         const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_y,
                         const ConvArgs a) {
  using Cfg = ConvCfg<kC>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  __shared__ __align__(8) uint64_t a_full[kMaxStages], a_empty[kMaxStages];
  __shared__ __align__(8) uint64_t b_full[kMaxStages], b_empty[kMaxStages];
  __shared__ __align__(8) uint64_t bar_acc_full[2], bar_acc_empty[2], bar_drain;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  __shared__ int epi_ok[4];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int* abort = &abort_sh;
  const uint64_t to = a.lc.timeout_ns;
  constexpr bool kTimeDown = kMode == kModeTimeDown;
  constexpr bool kStrip = kMode == kModeStrip || kMode == kModeStrip2;
  constexpr bool kFused = !kStrip;                 // A and B of a step on one barrier
  constexpr int kTapsPerA = kFused ? 1 : 3;        // taps one A box serves
  constexpr int kRows = kMode == kModeStrip2 ? 2 : 1;  // strips per tile, one accumulator each
  constexpr uint32_t kBoxRowLo = 130 * Cfg::kRow >> 4;  // one 130-pixel input row, in descriptor units
  constexpr int kTaps = kTimeDown ? 3 : 27;
  const int c_steps = a.c_in / kC;
  const int a_steps = kTaps / kTapsPerA * c_steps;  // A boxes per tile
  // ring geometry: compile-time for patches, the host's for strips
  const int a_stages = kFused ? Cfg::kPatchStages : a.a_stages;
  const int b_stages = kFused ? Cfg::kPatchStages : a.b_stages;
  const uint32_t a_stride = kFused ? Cfg::kPatchStage : a.a_stride;
  const uint32_t b_stride = kFused ? Cfg::kPatchStage : a.b_stride;
  const uint32_t b_off = kFused ? 128u * Cfg::kRow : a.b_off;

  if (threadIdx.x == 0) {
    for (int s = 0; s < a_stages; ++s) {
      mbar_init(&a_full[s], 1);
      mbar_init(&a_empty[s], 1);
    }
    for (int s = 0; s < b_stages; ++s) {
      mbar_init(&b_full[s], 1);
      mbar_init(&b_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bar_acc_full[b], 1);
      mbar_init(&bar_acc_empty[b], 4);  // one arrival per epilogue warp
    }
    mbar_init(&bar_drain, 1);
    abort_sh = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, a.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  // Debug builds: the accumulators start at TMEM lane 0 / column 0, the
  // swizzled rings need a 1024-byte aligned shared-memory base, and the ring
  // sizes fit their barrier arrays.
  if (threadIdx.x == 0) {
    WAN_DCHECK(!a.lc.force_check, a.lc.err);
    WAN_DCHECK(tmem == 0u, a.lc.err);
    WAN_DCHECK((smem_u32(smem) & 1023u) == 0u, a.lc.err);
    WAN_DCHECK(a_stages >= 1 && a_stages <= kMaxStages && b_stages >= 1 && b_stages <= kMaxStages &&
                   (!kFused || a.out_off == Cfg::kPatchStages * Cfg::kPatchStage),
               a.lc.err);
  }

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer of A
    if (lane == 0) {
      RingPos p;
      int fills = 0;  // A boxes issued, or withheld by the test hook
      bool ok = true;
      for (int idx = blockIdx.x; idx < a.n_tiles_total && ok; idx += gridDim.x) {
        const ConvTile x = conv_tile(idx, a);
        for (int s = 0; s < a_steps; ++s) {
          if (p.round > 0 && !mbar_wait(&a_empty[p.slot], (p.round - 1) & 1, abort, to)) {
            conv_abort(abort, a.lc.err);
            ok = false;
            break;
          }
          const int slot = p.slot;
          p.next(a_stages);
          ++fills;
          if (a.lc.stall && fills == 2) continue;  // test hook: the second A box never arrives
          const int tap = s / c_steps * kTapsPerA;  // first tap of the group (kw = 0 for a strip)
          const int c0 = (s % c_steps) * kC;
          const int kt = kTimeDown ? tap : tap / 9;
          const int kh = kTimeDown ? 1 : (tap / 3) % 3, kw = kTimeDown ? 1 : tap % 3;
          // input frame of this tap, < 0 before the chunk (the cache holds its last 2 or 1 frames)
          const int ti = kTimeDown ? 2 * x.t + kt - 1 : x.t + kt - 2;
          const int cache_frames = kTimeDown ? 1 : 2;
          // Debug builds: the tile lies in the output, and the TMA inner
          // coordinate (channels) starts on a 16-byte boundary.
          WAN_DCHECK(x.b < a.B && x.t < a.T && x.h0 < a.H && x.w0 < a.W && x.n0 + a.n_tile <= a.c_out &&
                         ((c0 * 2) & 15) == 0 && ti >= -cache_frames,
                     a.lc.err);
          uint8_t* sa = smem + slot * a_stride;
          mbar_arrive_expect_tx(&a_full[slot], kFused ? a.a_bytes + a.n_tile * Cfg::kRow : a.a_bytes);
          if (ti < 0 && a.has_cache)
            tma_load_5d(sa, &tm_cache, &a_full[slot], c0, x.w0 + kw - 1, x.h0 + kh - 1, ti + cache_frames, x.b);
          else  // before a first chunk (ti < 0) the box lies outside x and reads zeros
            tma_load_5d(sa, &tm_x, &a_full[slot], c0, x.w0 + kw - 1, x.h0 + kh - 1, ti, x.b);
          if (kFused) tma_load_3d(smem + b_off + slot * b_stride, &tm_w, &a_full[slot], c0, tap, x.n0);
        }
      }
      drain_ring(a_full, fills, a_stages, to);
    }
    __syncwarp();
  } else if (warp == 6) {
    // ------------------------------------------------------------ TMA producer of B (strips)
    if (!kFused && lane == 0) {
      const uint32_t tx = static_cast<uint32_t>(a.n_tile * Cfg::kRow);
      RingPos p;
      int fills = 0;
      bool ok = true;
      for (int idx = blockIdx.x; idx < a.n_tiles_total && ok; idx += gridDim.x) {
        const int n0 = idx % a.tiles_n * a.n_tile;
        for (int s = 0; s < a_steps && ok; ++s) {
          const int tap0 = s / c_steps * kTapsPerA;
          const int c0 = (s % c_steps) * kC;
          for (int j = 0; j < kTapsPerA; ++j) {
            if (p.round > 0 && !mbar_wait(&b_empty[p.slot], (p.round - 1) & 1, abort, to)) {
              conv_abort(abort, a.lc.err);
              ok = false;
              break;
            }
            uint8_t* sb = smem + b_off + p.slot * b_stride;
            mbar_arrive_expect_tx(&b_full[p.slot], tx);
            tma_load_3d(sb, &tm_w, &b_full[p.slot], c0, tap0 + j, n0);
            p.next(b_stages);
            ++fills;
          }
        }
      }
      drain_ring(b_full, fills, b_stages, to);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t idesc = idesc_bf16_f32(128, static_cast<uint32_t>(a.n_tile), 0, 0);
    const uint64_t d0 = conv_desc<kC>(smem_u32(smem));
    const uint32_t hi = static_cast<uint32_t>(d0 >> 32);
    const uint32_t lo0 = static_cast<uint32_t>(d0);
    bool ok = true;
    RingPos pa, pb;
    int i = 0;  // tiles of this CTA
    for (int idx = blockIdx.x; idx < a.n_tiles_total && ok; idx += gridDim.x, ++i) {
      const int ab = i & 1;
      const uint32_t acc = tmem + static_cast<uint32_t>(ab * kRows * a.n_tile);
      // The accumulators' previous tile has left TMEM.
      if (i >= 2) {
        ok = __all_sync(0xffffffffu, mbar_wait(&bar_acc_empty[ab], ((i >> 1) - 1) & 1, abort, to));
        if (!ok) {
          if (lane == 0) conv_abort(abort, a.lc.err);
          break;
        }
        tc_fence_after();
      }
      for (int s = 0; s < a_steps && ok; ++s) {
        ok = __all_sync(0xffffffffu, mbar_wait(&a_full[pa.slot], pa.round & 1, abort, to));
        if (!ok) {
          if (lane == 0) conv_abort(abort, a.lc.err);
          break;
        }
        const uint32_t a_lo = lo0 + ((static_cast<uint32_t>(pa.slot) * a_stride) >> 4);
#pragma unroll
        for (int j = 0; j < kTapsPerA; ++j) {
          if (!kFused) {
            ok = __all_sync(0xffffffffu, mbar_wait(&b_full[pb.slot], pb.round & 1, abort, to));
            if (!ok) {
              if (lane == 0) conv_abort(abort, a.lc.err);
              break;
            }
          }
          tc_fence_after();
          // tap kw = j of a strip: rows j .. j + 127 of the box's input row (one per strip)
          const uint32_t aj = a_lo + static_cast<uint32_t>(j * (Cfg::kRow >> 4));
          const int bslot = kFused ? pa.slot : pb.slot;  // for patches B came with A
          const uint32_t b_lo = lo0 + ((b_off + static_cast<uint32_t>(bslot) * b_stride) >> 4);
#pragma unroll
          for (int rr = 0; rr < kRows; ++rr)
#pragma unroll
            for (int kk = 0; kk < kC / 16; ++kk)  // 16 channels (32 bytes) per MMA
              umma_ss_elect_lo(acc + static_cast<uint32_t>(rr * a.n_tile), aj + rr * kBoxRowLo + kk * 2,
                               b_lo + kk * 2, hi, idesc, (s > 0 || j > 0 || kk > 0) ? 1u : 0u);
          if (!kFused) {
            umma_commit_elect(&b_empty[pb.slot]);
            pb.next(b_stages);
          }
        }
        if (!ok) break;
        umma_commit_elect(&a_empty[pa.slot]);
        pa.next(a_stages);
      }
      if (ok) umma_commit_elect(&bar_acc_full[ab]);
    }
    // Also on the failure path: every issued MMA completes before TMEM is freed.
    umma_commit_elect(&bar_drain);
    mbar_wait(&bar_drain, 0, nullptr, to);
  } else {
    // ------------------------------------------------------------ epilogue
    // Per 32 output channels of a tile: TMEM -> + bias -> bf16 -> a swizzled
    // staging buffer -> one TMA store, which also leaves out the positions
    // outside the picture. The bias arrives as one coalesced load per warp
    // (lane l holds channel l) and is spread with shuffles. The four warps
    // decide together whether to stop (flags written before a named barrier,
    // read after it), so none is left at a barrier.
    const int q = warp & 3;  // TMEM lanes 32q .. 32q+31
    const int r = q * 32 + lane;
    const bool leader = warp == 2 && lane == 0;  // issues the stores
    uint8_t* stage0 = smem + a.out_off;
    int i = 0, nchunk = 0;
    for (int idx = blockIdx.x; idx < a.n_tiles_total; idx += gridDim.x, ++i) {
      const int ab = i & 1;
      const bool done = __all_sync(0xffffffffu, mbar_wait(&bar_acc_full[ab], (i >> 1) & 1, abort, to));
      if (lane == 0) epi_ok[warp - 2] = done && !*abort ? 1 : 0;
      named_bar_sync(1, 128);
      const bool all_done = epi_ok[0] & epi_ok[1] & epi_ok[2] & epi_ok[3];
      if (!all_done) {
        if (!done && lane == 0) conv_abort(abort, a.lc.err);
        break;
      }
      tc_fence_after();
      const ConvTile x = conv_tile(idx, a);
      const uint32_t acc =
          tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(ab * kRows * a.n_tile);
      // Chunk c: TMEM columns 32c.. of the tile's accumulators, i.e. strip
      // c / nch, output channels 32 (c % nch).. A second strip below the
      // picture (odd H) is read but not stored.
      const int nch = a.n_tile / 32;
      for (int c = 0; c < kRows * nch; ++c) {
        const int rr = kRows == 1 ? 0 : c / nch, cc = c - rr * nch;
        const bool live = kRows == 1 || x.h0 + rr < a.H;  // the same for all four warps
        uint32_t v[32];
        if (live) {
          tmem_ld32(acc + static_cast<uint32_t>(c * 32), v);
          tmem_ld_wait_regs(v);
        }
        if (c == kRows * nch - 1) {
          // The accumulators may take the CTA's tile after next.
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bar_acc_empty[ab]);
        }
        if (!live) continue;
        const float bl = a.bias ? a.bias[x.n0 + cc * 32 + lane] : 0.f;
        uint32_t pk[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const float lo = __uint_as_float(v[2 * k]) + __shfl_sync(0xffffffffu, bl, 2 * k);
          const float hi2 = __uint_as_float(v[2 * k + 1]) + __shfl_sync(0xffffffffu, bl, 2 * k + 1);
          pk[k] = pack_bf16x2(lo, hi2);
        }
        uint8_t* st = stage0 + (nchunk & 1) * kOutStage;
        // This buffer's previous store (two chunks back) must have read it.
        if (leader) bulk_wait_group_read<1>();
        named_bar_sync(1, 128);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          *reinterpret_cast<uint4*>(st + sw64_offset(r, j)) = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2],
                                                                          pk[4 * j + 3]);
        fence_proxy_async_smem();
        named_bar_sync(1, 128);
        if (leader) {
          tma_store_5d(&tm_y, st, x.n0 + cc * 32, x.w0, x.h0 + rr, x.t, x.b);
          bulk_commit_group();
        }
        ++nchunk;
      }
    }
    if (leader) bulk_wait_group0();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, a.tmem_cols);
  }
}

// bf16 channels-last activations [B, frames, H, W, C] -> 5D tiled map, box
// {kc c, box_w w, box_h h, 1, 1}, 128-byte (kc = 64) or 64-byte (kc = 32)
// swizzle, zero fill outside.
bool make_tmap_act(CUtensorMap* map, const void* base, int B, int frames, int H, int W, int C, int kc, int box_w,
                   int box_h) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return false;
  const cuuint64_t c2 = (cuuint64_t)C * 2;
  cuuint64_t dims[5] = {(cuuint64_t)C, (cuuint64_t)W, (cuuint64_t)H, (cuuint64_t)frames, (cuuint64_t)B};
  cuuint64_t strides[4] = {c2, c2 * W, c2 * W * H, c2 * W * H * frames};
  cuuint32_t box[5] = {(cuuint32_t)kc, (cuuint32_t)box_w, (cuuint32_t)box_h, 1, 1};
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, kc == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Weights [C_out, taps, C_in] -> 3D tiled map, box {kc c, 1 tap, n_tile rows}.
bool make_tmap_wt(CUtensorMap* map, const void* base, int c_in, int c_out, int taps, int n_tile, int kc) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)c_in, (cuuint64_t)taps, (cuuint64_t)c_out};
  cuuint64_t strides[2] = {(cuuint64_t)c_in * 2, (cuuint64_t)c_in * 2 * taps};
  cuuint32_t box[3] = {(cuuint32_t)kc, 1, (cuuint32_t)n_tile};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, kc == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

uint32_t round_up_1k(uint32_t bytes) { return (bytes + 1023u) & ~1023u; }

// Strip tiles (1 x 128) when padding the width to a multiple of 128 wastes
// at most 1/16 of it; 8 x 16 patches otherwise and for time downsampling.
bool conv3d_uses_strips(int W, bool time_down) { return !time_down && ((W + 127) / 128 * 128 - W) * 16 <= W; }

}  // namespace

int conv3d_n_tile(int c_out) {
  if (c_out % 32 != 0) return 0;
  if (c_out <= 256) return c_out;  // one channel tile (an MMA N is any multiple of 16 up to 256)
  for (int n : {256, 192, 128, 64, 32})
    if (c_out % n == 0) return n;
  return 0;
}

int launch_causal_conv3d(const void* x, const void* cache, const void* wt, const float* bias, void* y, int B, int T,
                         int H, int W, int c_in, int c_out, const LaunchCommon& lc, cudaStream_t s, bool time_down) {
  const int n_tile = conv3d_n_tile(c_out);
  if (n_tile == 0 || c_in % 32 != 0) return WAN_ERR_UNSUPPORTED;
  const int kc = c_in % 64 == 0 ? 64 : 32;  // input channels per K step
  const uint32_t row = static_cast<uint32_t>(kc * 2);
  const bool strip = conv3d_uses_strips(W, time_down);
  const int rows = strip && 4 * n_tile <= 512 ? 2 : 1;  // strips per tile (2 x rows accumulators in TMEM)
  ConvArgs a;
  a.bias = bias;
  a.B = B;
  a.T = time_down ? T / 2 : T;  // output frames
  a.H = H;
  a.W = W;
  a.c_in = c_in;
  a.c_out = c_out;
  a.n_tile = n_tile;
  a.ph = strip ? rows : 8;
  a.pw = strip ? 128 : 16;
  a.tiles_h = (H + a.ph - 1) / a.ph;
  a.tiles_w = (W + a.pw - 1) / a.pw;
  a.tiles_n = c_out / n_tile;
  a.has_cache = cache != nullptr;
  a.lc = lc;
  // Rings: a strip's A box (130 rows) serves three taps, so its ring is short
  // and B takes the rest; a patch's A and B advance together in {A, B} stages.
  const int a_rows = strip ? (a.pw + 2) * rows : 128;
  a.a_bytes = static_cast<uint32_t>(a_rows) * row;
  const uint32_t a_slot = round_up_1k(a.a_bytes);
  const uint32_t b_slot = static_cast<uint32_t>(n_tile) * row;  // n_tile % 32 == 0: a multiple of 1024
  if (strip) {
    a.a_stages = kc == 64 ? 3 : 4;
    a.b_stages = static_cast<int>((kRingBytes - a.a_stages * a_slot) / b_slot);
    if (a.b_stages > kMaxStages) a.b_stages = kMaxStages;
    a.a_stride = a_slot;
    a.b_stride = b_slot;
    a.b_off = a.a_stages * a_slot;
    a.out_off = a.b_off + a.b_stages * b_slot;
  } else {
    a.a_stages = a.b_stages = kc == 64 ? ConvCfg<64>::kPatchStages : ConvCfg<32>::kPatchStages;
    a.a_stride = a.b_stride = kc == 64 ? ConvCfg<64>::kPatchStage : ConvCfg<32>::kPatchStage;
    a.b_off = 128 * row;
    a.out_off = a.a_stages * a.a_stride;
  }
  if (a.a_stages < 1 || a.b_stages < 2) return WAN_ERR_UNSUPPORTED;
  const int smem = static_cast<int>(a.out_off) + 2 * kOutStage + 1024;
  // Two accumulators of n_tile fp32 columns; TMEM is allocated in powers of two.
  const int cols = 2 * rows * n_tile;
  a.tmem_cols = cols <= 128 ? 128u : (cols <= 256 ? 256u : 512u);
  const long long total = (long long)B * a.T * a.tiles_h * a.tiles_w * a.tiles_n;
  if (total > INT_MAX) return WAN_ERR_INVALID;
  a.n_tiles_total = (int)total;
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return WAN_ERR_CUDA;
  const int grid = (int)(total < sms ? total : sms);  // persistent: one CTA per SM

  CUtensorMap tx, tc, tw, ty;
  const int cache_frames = time_down ? 1 : 2;
  // input box: {kc, 130, rows} for strips, {kc, 16, 8} for patches; output
  // box: 32 channels of one strip or patch, 64-byte swizzle
  const int in_w = strip ? a.pw + 2 : a.pw;
  if (!make_tmap_act(&tx, x, B, T, H, W, c_in, kc, in_w, a.ph) ||
      !make_tmap_act(&tc, cache ? cache : x, B, cache ? cache_frames : T, H, W, c_in, kc, in_w, a.ph) ||
      !make_tmap_wt(&tw, wt, c_in, c_out, time_down ? 3 : 27, n_tile, kc) ||
      !make_tmap_act(&ty, y, B, a.T, H, W, c_out, 32, a.pw, strip ? 1 : a.ph))
    return WAN_ERR_CUDA;
  auto kern = time_down ? (kc == 64 ? causal_conv3d_kernel<64, kModeTimeDown> : causal_conv3d_kernel<32, kModeTimeDown>)
              : rows == 2 ? (kc == 64 ? causal_conv3d_kernel<64, kModeStrip2> : causal_conv3d_kernel<32, kModeStrip2>)
              : strip   ? (kc == 64 ? causal_conv3d_kernel<64, kModeStrip> : causal_conv3d_kernel<32, kModeStrip>)
                        : (kc == 64 ? causal_conv3d_kernel<64, kModePatch> : causal_conv3d_kernel<32, kModePatch>);
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return WAN_ERR_CUDA;
  record_start(lc, s);
  kern<<<grid, kConvThreads, smem, s>>>(tx, tc, tw, ty, a);
  record_stop(lc, s);
  return cudaGetLastError() == cudaSuccess ? WAN_OK : WAN_ERR_CUDA;
}

}  // namespace wan
