// Attention backward for sm_103a (the gradient step of rectified-flow
// training - gojay.top "Wan2.1" reading, section 3 Training - through full
// 3D-RoPE self-attention).
//
// With P = softmax(scale * Q_rot K_rot^T) (recomputed from the forward LSE),
// D_i = dO_i . O_i and dS = scale * P o (dO V^T - D):
//   dV = P^T dO,  dK_rot = dS^T Q_rot,  dQ_rot = dS K_rot,
//   dK = R^T dK_rot,  dQ = R^T dQ_rot   (R = the 3D RoPE rotation of each token).
//
// Steps (all on the caller's stream):
//   1. prep: Q_rot, K_rot (RoPE pre-pass), D and LSE*log2(e) per row into
//      128-padded rows (pad: D = 0, LSE = +inf so padded queries get P = 0),
//      dQ accumulator := 0.
//   2. main: one CTA per 128-key tile of one (b, h), looping over all 128-row
//      query tiles. Everything is computed transposed (keys on TMEM lanes):
//        S^T  = K_rot Q_rot^T     dP^T = V dO^T         (tcgen05, A and B in smem)
//        P^T  = exp2(S^T*scale*log2e - LSE*log2e)      (threads, into TMEM)
//        dV  += P^T dO                                  (A = P^T from TMEM)
//        dS^T = scale * P^T o (dP^T - D)                (threads, into TMEM + smem)
//        dK  += dS^T Q_rot                              (A = dS^T from TMEM)
//        dQ_i = dS K_rot  (two N=64 halves)             (A = dS from smem, MN-major)
//      The dQ warpgroup reads dQ_i out of TMEM and stages it, as 128B-swizzled
//      128 x 32-float boxes, in the query tile's own {Q_rot, dO} stage: once
//      the dQ MMA is done, every MMA that reads that stage is done too (the
//      dQ MMAs come last in issue order), so d-half 0 goes where Q_rot was
//      and d-half 1 where dO was. A reduction warp adds the staged halves
//      into the fp32 accumulator with bulk tensor reductions and hands each
//      slot back to the producer as soon as its reduction has read it.
//      TMEM: dV [0,128) dK [128,256) S [256,384) dP [384,512); P^T, dS^T
//      (bf16) and the dQ halves reuse S and dP columns once the MMAs that read
//      them are ordered before (tcgen05 MMAs of one thread run in order).
//      Epilogue: dV -> bf16; dK -> R^T -> bf16.
//   3. post: dQ = R^T dQ_acc -> bf16.
//      The fp32 reduction of dQ into global memory is the costly part of the
//      backward (one 64 KB tile per query tile per CTA, bound by the L2's
//      reduction rate). Staging it in the consumed stage, instead of a buffer
//      that the next tile's dS must wait for, lets one tile's reduction run
//      under the next tile's MMAs and softmax; what it still gates is the
//      next-but-one tile's Q_rot and dO loads into that stage.
// Warps (register budgets moved with setmaxnreg):
//   0-7    compute (warp w: TMEM lanes 32*(w%4).., column half w/4)   152 regs
//   8      TMA producer; 9 MMA issuer (warp-converged, one elected lane
//          issues) and TMEM owner; 10 dQ reductions; 11 idle             96 regs
//   12-15  dQ writers (warp w: TMEM lanes 32*(w%4)..)                   112 regs
#include "common.cuh"
#include "kernels.cuh"

namespace wan {

namespace {

constexpr int kThreads = 512;
constexpr uint32_t kComputeRegs = 152;  // 2 x 128 x 152 + 128 x 96 + 128 x 112 = 512 x 128
constexpr uint32_t kControlRegs = 96;
constexpr uint32_t kDqRegs = 112;
constexpr int kDqWarp0 = 12;
constexpr int kLoadWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kReduceWarp = 10;
constexpr int kTile = 128;
constexpr int kTileBytes = 128 * 128 * 2;
constexpr int kHalfBytes = kTileBytes / 2;
// Dynamic shared memory map (bytes, from a 1024-aligned base).
constexpr int kOffK = 0;
constexpr int kOffV = kOffK + kTileBytes;
constexpr int kOffStage = kOffV + kTileBytes;  // 2 stages of {Q_rot, dO}
constexpr int kStageBytes = 2 * kTileBytes;
constexpr int kOffDS = kOffStage + 2 * kStageBytes;
constexpr int kOffRows = kOffDS + kTileBytes;  // 2 stages of {LSE*log2e[128], D[128]}
constexpr int kRowsBytes = 2 * kTile * 4;
constexpr int kOffBar = kOffRows + 2 * kRowsBytes;
constexpr int kSmemBytes = kOffBar + 256;  // barriers, TMEM base, abort word; dQ stop flags at 192

enum Bar {
  kBarKV = 0,
  kBarQFull0 = 1,   // +stage: Q_rot tile and the rows {LSE*log2e, D} landed
  kBarQEmpty0 = 3,  // +stage: the Q_rot slot (dQ half 0 staging) has been read by its reduction
  kBarS = 5,
  kBarDP = 6,
  kBarP = 7,
  kBarDS = 8,
  kBarDQ = 9,       // dQ (128 x 128 fp32) is in TMEM (dP columns)
  kBarDQFree = 10,  // ... and has been read: dP of the next tile may be written
  kBarAcc = 11,
  kBarDrain = 12,
  kBarDOFull0 = 13,  // +stage: dO tile landed
  kBarDOEmpty0 = 15,  // +stage: the dO slot (dQ half 1 staging) has been read by its reduction
  kBarStaged0 = 17,  // +stage: dQ half 0 written into the stage's Q_rot slot
  kBarStaged1 = 19,  // +stage: dQ half 1 written into the stage's dO slot
  kNumBars = 21
};
static_assert(kNumBars * 8 + 8 <= 192, "barrier area overlaps the dQ stop flags");

struct BwdArgs {
  const float* lse2;  // [B*H][Lpad] LSE * log2(e), pad +inf
  const float* drow;  // [B*H][Lpad] D, pad 0
  float* dq_acc;      // [B, L, H, 128] fp32
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  RopeTables tab;
  int L, Lpad, H, Hp, Wp;
  float scale_log2, scale;
  LaunchCommon lc;
};

__device__ __forceinline__ void raise_abort(volatile int* abort, int* err) {
  *abort = 1;
  atomicCAS(err, 0, kDevTimeout);
}

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort, int* err,
                                          uint64_t to) {
  bool ok = mbar_wait(bar, parity, abort, to);
  ok = __all_sync(0xffffffffu, ok);
  if (!ok && (threadIdx.x & 31) == 0) raise_abort(abort, err);
  return ok;
}

__device__ __forceinline__ void load32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  tmem_ld32(taddr, r);
  tmem_ld_wait_regs(r);
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_dq, const BwdArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint32_t* tmem_base_sh = reinterpret_cast<uint32_t*>(smem + kOffBar + kNumBars * 8);
  int* abort_sh = reinterpret_cast<int*>(smem + kOffBar + kNumBars * 8 + 4);
  volatile int* abort = abort_sh;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int h = blockIdx.y;
  const int b = blockIdx.z;
  const int kv0 = blockIdx.x * kTile;
  const int nq = (a.L + kTile - 1) / kTile;
  // Query tiles are visited from a per-CTA starting tile, so that the CTAs of
  // one head in flight add their dQ contributions into different rows
  // instead of all contending for the same L2 lines.
  const int q_start = static_cast<int>((static_cast<long long>(blockIdx.x) * nq) / gridDim.x);
  const uint64_t to = a.lc.timeout_ns;

  // The tile math below needs a 1024-byte aligned base (128B swizzle atoms).
  if (smem_u32(smem) & 1023u) {
    if (threadIdx.x == 0) atomicCAS(a.lc.err, 0, kDevTimeout);
    return;
  }

  if (threadIdx.x == 0) {
    mbar_init(&bars[kBarKV], 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars[kBarQFull0 + s], 1);
      mbar_init(&bars[kBarQEmpty0 + s], 1);
      mbar_init(&bars[kBarDOFull0 + s], 1);
      mbar_init(&bars[kBarDOEmpty0 + s], 1);
      mbar_init(&bars[kBarStaged0 + s], 4);  // one arrival per dQ warp
      mbar_init(&bars[kBarStaged1 + s], 4);
    }
    mbar_init(&bars[kBarS], 1);
    mbar_init(&bars[kBarDP], 1);
    mbar_init(&bars[kBarP], 8);
    mbar_init(&bars[kBarDS], 8);
    mbar_init(&bars[kBarDQ], 1);
    mbar_init(&bars[kBarDQFree], 4);
    mbar_init(&bars[kBarAcc], 1);
    mbar_init(&bars[kBarDrain], 1);
    *abort_sh = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_base_sh, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_base_sh;
  // Debug builds: the 512 TMEM columns start at lane 0 / column 0.
  if (threadIdx.x == 0) {
    WAN_DCHECK(!a.lc.force_check, a.lc.err);
    WAN_DCHECK(tmem == 0u, a.lc.err);
    WAN_DCHECK(kv0 < a.L && q_start >= 0 && q_start < nq, a.lc.err);
  }
  const uint32_t tDV = tmem, tDK = tmem + 128, tS = tmem + 256, tDP = tmem + 384;

  const size_t bh = static_cast<size_t>(b) * a.H + h;

  if (warp >= 8 && warp < kDqWarp0) {
   regs_shrink<kControlRegs>();
   if (warp == kLoadWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_do);
      mbar_arrive_expect_tx(&bars[kBarKV], 2 * kTileBytes);
      tma_load_4d(smem + kOffK, &tm_k, &bars[kBarKV], 0, h, kv0, b);
      tma_load_4d(smem + kOffK + kHalfBytes, &tm_k, &bars[kBarKV], 64, h, kv0, b);
      tma_load_4d(smem + kOffV, &tm_v, &bars[kBarKV], 0, h, kv0, b);
      tma_load_4d(smem + kOffV + kHalfBytes, &tm_v, &bars[kBarKV], 64, h, kv0, b);
      // Stage s holds query tile i = s, s + 2, ...; each of its two slots is
      // refilled as soon as the reduction of the dQ half staged in it has read it.
      int issued_q[2] = {0, 0}, issued_do[2] = {0, 0};
      for (int i = 0; i < nq; ++i) {
        const int s = i & 1, use = i >> 1;
        if (use > 0 && !mbar_wait(&bars[kBarQEmpty0 + s], (use - 1) & 1, abort, to)) {
          raise_abort(abort, a.lc.err);
          break;
        }
        if (a.lc.stall && i == 1) continue;  // test hook: query tile 1 never arrives
        uint8_t* st = smem + kOffStage + s * kStageBytes;
        uint8_t* rows = smem + kOffRows + s * kRowsBytes;
        const int q0 = (i + q_start < nq ? i + q_start : i + q_start - nq) * kTile;
        uint64_t* bar = &bars[kBarQFull0 + s];
        mbar_arrive_expect_tx(bar, kTileBytes + kRowsBytes);
        tma_load_4d(st, &tm_q, bar, 0, h, q0, b);
        tma_load_4d(st + kHalfBytes, &tm_q, bar, 64, h, q0, b);
        bulk_load(rows, a.lse2 + bh * a.Lpad + q0, kTile * 4, bar);
        bulk_load(rows + kTile * 4, a.drow + bh * a.Lpad + q0, kTile * 4, bar);
        issued_q[s] = use + 1;
        if (use > 0 && !mbar_wait(&bars[kBarDOEmpty0 + s], (use - 1) & 1, abort, to)) {
          raise_abort(abort, a.lc.err);
          break;
        }
        bar = &bars[kBarDOFull0 + s];
        mbar_arrive_expect_tx(bar, kTileBytes);
        tma_load_4d(st + kTileBytes, &tm_do, bar, 0, h, q0, b);
        tma_load_4d(st + kTileBytes + kHalfBytes, &tm_do, bar, 64, h, q0, b);
        issued_do[s] = use + 1;
      }
      // Every copy this warp issued lands before the CTA may exit.
      mbar_wait(&bars[kBarKV], 0, nullptr, to);
      for (int s = 0; s < 2; ++s) {
        if (issued_q[s] > 0) mbar_wait(&bars[kBarQFull0 + s], (issued_q[s] - 1) & 1, nullptr, to);
        if (issued_do[s] > 0) mbar_wait(&bars[kBarDOFull0 + s], (issued_do[s] - 1) & 1, nullptr, to);
      }
    }
    __syncwarp();
   } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    {
      const uint32_t id_kk = idesc_bf16_f32(128, 128, 0, 0);  // both operands K-major
      const uint32_t id_tm = idesc_bf16_f32(128, 128, 0, 1);  // A from TMEM, B MN-major
      const uint32_t id_dq = idesc_bf16_f32(128, 128, 1, 1);  // A and B MN-major
      const uint64_t dK = sdesc_sw128(smem_u32(smem + kOffK), 16, 1024);
      const uint64_t dV = sdesc_sw128(smem_u32(smem + kOffV), 16, 1024);
      const uint64_t dKmn = sdesc_sw128(smem_u32(smem + kOffK), kHalfBytes, 1024);
      const uint64_t dDS = sdesc_sw128(smem_u32(smem + kOffDS), kHalfBytes, 1024);
      const uint64_t dStage_k = sdesc_sw128(smem_u32(smem + kOffStage), 16, 1024);
      const uint64_t dStage_mn = sdesc_sw128(smem_u32(smem + kOffStage), kHalfBytes, 1024);
      bool ok = warp_wait(&bars[kBarKV], 0, abort, a.lc.err, to);
      for (int i = 0; i < nq && ok; ++i) {
        const int s = i & 1, use = i >> 1;
        const uint64_t so = static_cast<uint64_t>((s * kStageBytes) >> 4);   // Q tile of stage s
        const uint64_t sdo = so + static_cast<uint64_t>(kTileBytes >> 4);      // dO tile of stage s
        // S^T(i) goes into the S columns, whose last reader (dV(i-1)) was
        // issued earlier: no wait on the dQ warps.
        ok = warp_wait(&bars[kBarQFull0 + s], use & 1, abort, a.lc.err, to);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t off = static_cast<uint64_t>(((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4);
          umma_ss_elect(tS, dK + off, dStage_k + so + off, id_kk, kk > 0);
        }
        umma_commit_elect(&bars[kBarS]);
        if (!(ok = warp_wait(&bars[kBarDOFull0 + s], use & 1, abort, a.lc.err, to))) break;
        // dP^T(i) goes into the dP columns once dQ(i-1) has been read out of them.
        if (i > 0 && !(ok = warp_wait(&bars[kBarDQFree], (i - 1) & 1, abort, a.lc.err, to))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t off = static_cast<uint64_t>(((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4);
          umma_ss_elect(tDP, dV + off, dStage_k + sdo + off, id_kk, kk > 0);
        }
        umma_commit_elect(&bars[kBarDP]);
        if (!(ok = warp_wait(&bars[kBarP], i & 1, abort, a.lc.err, to))) break;
        tc_fence_after();
        // P^T sits in S columns [0,32) (queries 0..63) and [64,96) (queries 64..127).
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ts_elect(tDV, tS + (kk >> 2) * 64 + (kk & 3) * 8, dStage_mn + sdo + static_cast<uint64_t>(kk * 128),
                        id_tm, (i > 0 || kk > 0) ? 1u : 0u);
        if (!(ok = warp_wait(&bars[kBarDS], i & 1, abort, a.lc.err, to))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ts_elect(tDK, tDP + (kk >> 2) * 64 + (kk & 3) * 8, dStage_mn + so + static_cast<uint64_t>(kk * 128),
                        id_tm, (i > 0 || kk > 0) ? 1u : 0u);
        // dQ_i = dS K_rot (N = 128) into the dP columns: the fp32 dP there has
        // been read by the softmax, and the dS^T there by the dK MMAs issued
        // just before (tcgen05 MMAs of one thread run in order).
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ss_elect(tDP, dDS + static_cast<uint64_t>(kk * 128), dKmn + static_cast<uint64_t>((kk * 2048) >> 4),
                        id_dq, kk > 0);
        umma_commit_elect(&bars[kBarDQ]);
      }
      if (ok) umma_commit_elect(&bars[kBarAcc]);
      umma_commit_elect(&bars[kBarDrain]);
      mbar_wait(&bars[kBarDrain], 0, nullptr, to);
    }
   } else if (warp == kReduceWarp) {
    // ------------------------------------------------------------ dQ reductions
    // Adds each staged dQ half into the fp32 accumulator (two 128 x 32-float
    // boxes per half) and returns its slot to the producer once the bulk copy
    // has read it.
    if (lane == 0) {
      tma_prefetch_desc(&tm_dq);
      for (int i = 0; i < nq; ++i) {
        const int s = i & 1, use = i >> 1;
        const int qt = i + q_start < nq ? i + q_start : i + q_start - nq;
        WAN_DCHECK(qt >= 0 && qt < nq, a.lc.err);
        uint8_t* st = smem + kOffStage + s * kStageBytes;
        if (!mbar_wait(&bars[kBarStaged0 + s], use & 1, abort, to)) {
          raise_abort(abort, a.lc.err);
          break;
        }
        tma_reduce_add_4d(&tm_dq, st, 0, h, qt * kTile, b);
        tma_reduce_add_4d(&tm_dq, st + kTile * 128, 32, h, qt * kTile, b);
        bulk_commit_group();
        if (!mbar_wait(&bars[kBarStaged1 + s], use & 1, abort, to)) {
          raise_abort(abort, a.lc.err);
          break;
        }
        tma_reduce_add_4d(&tm_dq, st + kTileBytes, 64, h, qt * kTile, b);
        tma_reduce_add_4d(&tm_dq, st + kTileBytes + kTile * 128, 96, h, qt * kTile, b);
        bulk_commit_group();
        bulk_wait_group_read<1>();  // half 0's reductions have read the Q_rot slot
        mbar_arrive(&bars[kBarQEmpty0 + s]);
        bulk_wait_group_read<0>();
        mbar_arrive(&bars[kBarDOEmpty0 + s]);
      }
      bulk_wait_group0();  // every reduction is complete before the CTA exits
    }
    __syncwarp();
   }
  } else if (warp >= kDqWarp0) {
    regs_shrink<kDqRegs>();
    // ------------------------------------------------------------ dQ writers
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(wq * 32) << 16;
    // Per-warp stop flags (in the dynamic barrier area: a static __shared__
    // array would move the 1024-byte aligned dynamic base).
    volatile int* dq_fail = reinterpret_cast<volatile int*>(smem + kOffBar + 192);
    // Row r of the 128 x 64-float half in v -> two 128B-swizzled boxes of 32 floats.
    auto stage_half = [&](uint8_t* dst, const uint32_t (&v)[64]) {
#pragma unroll
      for (int c = 0; c < 16; ++c)  // box c/8, 16-byte chunk c%8 of row r
        *reinterpret_cast<uint4*>(dst + (c >> 3) * (kTile * 128) + sw128_offset(r, c & 7)) =
            make_uint4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
      fence_proxy_async_smem();  // visible to the bulk copies that read it
    };
    for (int i = 0; i < nq; ++i) {
      const int s = i & 1;
      const bool ok = warp_wait(&bars[kBarDQ], i & 1, abort, a.lc.err, to);
      // The four warps decide together whether to stop, so that none of
      // them is left waiting at the named barrier.
      if (lane == 0) dq_fail[wq] = ok ? 0 : 1;
      named_bar_sync(1, 128);
      if (dq_fail[0] | dq_fail[1] | dq_fail[2] | dq_fail[3]) break;
      tc_fence_after();
      // Half 0 (d 0..63) is staged before half 1 leaves TMEM (the next tile's
      // dP MMA waits for that). Each half goes to its slot of this tile's
      // stage: every MMA that read the stage completed before the dQ MMAs did.
      uint8_t* st = smem + kOffStage + s * kStageBytes;
      uint32_t v[64];
      tmem_ld32(tDP + lane_addr, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
      tmem_ld32(tDP + lane_addr + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
      tmem_ld_wait_regs(v);
      stage_half(st, v);
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kBarStaged0 + s]);
      tmem_ld32(tDP + lane_addr + 64, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
      tmem_ld32(tDP + lane_addr + 96, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
      tmem_ld_wait_regs(v);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kBarDQFree]);
      stage_half(st + kTileBytes, v);
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kBarStaged1 + s]);
    }
  } else {
    regs_grow<kComputeRegs>();
    // ------------------------------------------------------------ compute
    const int wq = warp & 3;
    const int ch = warp >> 2;  // column half
    const int r = wq * 32 + lane;
    const int key = kv0 + r;
    const bool key_ok = key < a.L;
    const uint32_t lane_addr = static_cast<uint32_t>(wq * 32) << 16;
    const float sl2 = a.scale_log2;
    bool ok = true;
    for (int i = 0; i < nq && ok; ++i) {
      const int s = i & 1, use = i >> 1;
      const float* lse2 = reinterpret_cast<const float*>(smem + kOffRows + s * kRowsBytes) + ch * 64;
      const float* drow = lse2 + kTile;
      ok = warp_wait(&bars[kBarQFull0 + s], use & 1, abort, a.lc.err, to);
      if (ok) ok = warp_wait(&bars[kBarS], i & 1, abort, a.lc.err, to);
      if (!ok) break;
      tc_fence_after();
      // P^T row of key r, queries ch*64 .. ch*64+63, two lanes of arithmetic
      // per f32x2 instruction. Keys past the end (zero K rows) get P = 0: a
      // warp decides once whether any of its keys is past the end.
      float p[64];
      {
        uint32_t sr[64];
        tmem_ld32(tS + lane_addr + ch * 64, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
        tmem_ld32(tS + lane_addr + ch * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
        tmem_ld_wait_regs(sr);
        const uint64_t sl2x2 = f2_pack(sl2, sl2);
#pragma unroll
        for (int k4 = 0; k4 < 16; ++k4) {  // the row values are the same for every lane: 16-byte broadcasts
          const float4 l4 = reinterpret_cast<const float4*>(lse2)[k4];
          const int k = 4 * k4;
          float x0, x1, x2, x3;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[k]), __uint_as_float(sr[k + 1])), sl2x2, f2_pack(-l4.x, -l4.y)),
                    x0, x1);
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[k + 2]), __uint_as_float(sr[k + 3])), sl2x2,
                           f2_pack(-l4.z, -l4.w)),
                    x2, x3);
          p[k] = ex2_approx(x0);
          p[k + 1] = ex2_approx(x1);
          p[k + 2] = ex2_approx(x2);
          p[k + 3] = ex2_approx(x3);
        }
        if (!__all_sync(0xffffffffu, key_ok) && !key_ok) {
#pragma unroll
          for (int k = 0; k < 64; ++k) p[k] = 0.f;
        }
      }
      {
        uint32_t pk[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) pk[k] = pack_bf16x2(p[2 * k], p[2 * k + 1]);
        tmem_st32(tS + lane_addr + ch * 64, pk);
        tmem_st_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kBarP]);

      if (!(ok = warp_wait(&bars[kBarDP], i & 1, abort, a.lc.err, to))) break;
      tc_fence_after();
      {
        uint32_t pk[32];
        // dS = scale * P o (dP - D), two lanes per f32x2 instruction, in two
        // 32-column chunks.
        const uint64_t sc2 = f2_pack(a.scale, a.scale);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t dr[32];
          tmem_ld32(tDP + lane_addr + ch * 64 + c * 32, dr);
          tmem_ld_wait_regs(dr);
#pragma unroll
          for (int k4 = 0; k4 < 8; ++k4) {
            const float4 d4 = reinterpret_cast<const float4*>(drow)[c * 8 + k4];
            const int k = 4 * k4, j = c * 32 + k;
            float s0, s1, s2, s3;
            f2_unpack(f2_mul(f2_sub(f2_pack(__uint_as_float(dr[k]), __uint_as_float(dr[k + 1])), f2_pack(d4.x, d4.y)),
                             f2_mul(f2_pack(p[j], p[j + 1]), sc2)),
                      s0, s1);
            f2_unpack(f2_mul(f2_sub(f2_pack(__uint_as_float(dr[k + 2]), __uint_as_float(dr[k + 3])),
                                    f2_pack(d4.z, d4.w)),
                             f2_mul(f2_pack(p[j + 2], p[j + 3]), sc2)),
                      s2, s3);
            pk[c * 16 + 2 * k4] = pack_bf16x2(s0, s1);
            pk[c * 16 + 2 * k4 + 1] = pack_bf16x2(s2, s3);
          }
        }
        tmem_st32(tDP + lane_addr + ch * 64, pk);
        // dS^T row r, queries ch*64 .. ch*64+63 -> half tile ch of the MN-major A operand.
        // The previous tile's dQ MMAs, the last readers of the dS buffer, were
        // issued before this tile's dP MMA, so they completed before DP fired.
        uint8_t* ds_row = smem + kOffDS + ch * kHalfBytes;
#pragma unroll
        for (int cc = 0; cc < 8; ++cc)
          *reinterpret_cast<uint4*>(ds_row + sw128_offset(r, cc)) =
              make_uint4(pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
        tmem_st_wait();
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kBarDS]);

    }
    // ------------------------------------------------------------ epilogue
    if (ok) ok = warp_wait(&bars[kBarAcc], 0, abort, a.lc.err, to);
    if (ok) {
      tc_fence_after();
      float v[64];
      {
        float t32[32];
        load32(tDV + lane_addr + ch * 64, t32);
#pragma unroll
        for (int k = 0; k < 32; ++k) v[k] = t32[k];
        load32(tDV + lane_addr + ch * 64 + 32, t32);
#pragma unroll
        for (int k = 0; k < 32; ++k) v[32 + k] = t32[k];
      }
      const size_t off = ((static_cast<size_t>(b) * a.L + key) * a.H + h) * 128 + ch * 64;
      if (key_ok) {
        uint4* dst = reinterpret_cast<uint4*>(a.dv + off);
#pragma unroll
        for (int q = 0; q < 8; ++q)
          dst[q] = make_uint4(pack_bf16x2(v[8 * q], v[8 * q + 1]), pack_bf16x2(v[8 * q + 2], v[8 * q + 3]),
                              pack_bf16x2(v[8 * q + 4], v[8 * q + 5]), pack_bf16x2(v[8 * q + 6], v[8 * q + 7]));
      }
      {
        float t32[32];
        load32(tDK + lane_addr + ch * 64, t32);
#pragma unroll
        for (int k = 0; k < 32; ++k) v[k] = t32[k];
        load32(tDK + lane_addr + ch * 64 + 32, t32);
#pragma unroll
        for (int k = 0; k < 32; ++k) v[32 + k] = t32[k];
      }
      if (key_ok) {
        const int w = key % a.Wp;
        const int hh = (key / a.Wp) % a.Hp;
        const int t = key / (a.Wp * a.Hp);
        uint32_t pk[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const int pair = ch * 32 + k;
          const float2 cs = pair < kPairsT ? a.tab.t[t * kPairsT + pair]
                                           : (pair < kPairsT + kPairsH ? a.tab.h[hh * kPairsH + pair - kPairsT]
                                                                       : a.tab.w[w * kPairsW + pair - kPairsT - kPairsH]);
          const float x0 = v[2 * k], x1 = v[2 * k + 1];
          pk[k] = pack_bf16x2(x0 * cs.x + x1 * cs.y, x1 * cs.x - x0 * cs.y);
        }
        uint4* dst = reinterpret_cast<uint4*>(a.dk + off);
#pragma unroll
        for (int q = 0; q < 8; ++q) dst[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

size_t align_up(size_t x) { return (x + 255) / 256 * 256; }

struct BwdWorkspace {
  void* q_rot;
  void* k_rot;
  float* dq_acc;
  float* lse2;
  float* drow;
  size_t bytes;
};

BwdWorkspace carve(void* base, int B, int L, int H) {
  const size_t n = (size_t)B * L * H;
  const int Lpad = (L + kTile - 1) / kTile * kTile;
  const size_t rows = (size_t)B * H * Lpad * 4;
  BwdWorkspace w;
  uint8_t* p = static_cast<uint8_t*>(base);
  size_t off = 0;
  w.q_rot = p + off;
  off += align_up(n * 256);
  w.k_rot = p + off;
  off += align_up(n * 256);
  w.dq_acc = reinterpret_cast<float*>(p + off);
  off += align_up(n * 512);
  w.lse2 = reinterpret_cast<float*>(p + off);
  off += align_up(rows);
  w.drow = reinterpret_cast<float*>(p + off);
  off += align_up(rows);
  w.bytes = off;
  return w;
}

}  // namespace

size_t attn_bwd_workspace_bytes(int B, int L, int H) { return carve(nullptr, B, L, H).bytes; }

int launch_attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                    void* dq, void* dk, void* dv, int B, wan_grid_t g, int H, RopeTables tab, float scale,
                    void* workspace, const LaunchCommon& lc, cudaStream_t s) {
  const int L = g.F * g.Hp * g.Wp;
  const int Lpad = (L + kTile - 1) / kTile * kTile;
  BwdWorkspace w = carve(workspace, B, L, H);
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);

  if (launch_rope_rotate_bf16(q, w.q_rot, B, g, H, tab, false, s) != cudaSuccess) return WAN_ERR_CUDA;
  record_pass(lc, kPassRope, 0, s);
  if (launch_rope_rotate_bf16(k, w.k_rot, B, g, H, tab, false, s) != cudaSuccess) return WAN_ERR_CUDA;
  record_pass(lc, kPassRope, 1, s);
  const long long n_rows = (long long)B * L * H;
  {
    record_pass(lc, kPassRows, 0, s);
    if (launch_bwd_rows(o, dout, lse, w.lse2, w.drow, B, L, Lpad, H, s) != cudaSuccess) return WAN_ERR_CUDA;
    record_pass(lc, kPassRows, 1, s);
  }
  if (cudaMemsetAsync(w.dq_acc, 0, (size_t)n_rows * 512, s) != cudaSuccess) return WAN_ERR_CUDA;

  CUtensorMap tq, tk, tv, tdo, tdq;
  if (!make_tmap_bld(&tq, w.q_rot, B, L, H, kHeadDim, 128) || !make_tmap_bld(&tk, w.k_rot, B, L, H, kHeadDim, 128) ||
      !make_tmap_bld(&tv, v, B, L, H, kHeadDim, 128) || !make_tmap_bld(&tdo, dout, B, L, H, kHeadDim, 128) ||
      !make_tmap_f32_bld(&tdq, w.dq_acc, B, L, H, kHeadDim, 128))
    return WAN_ERR_CUDA;
  BwdArgs a;
  a.lse2 = w.lse2;
  a.drow = w.drow;
  a.dq_acc = w.dq_acc;
  a.dk = static_cast<__nv_bfloat16*>(dk);
  a.dv = static_cast<__nv_bfloat16*>(dv);
  a.tab = tab;
  a.L = L;
  a.Lpad = Lpad;
  a.H = H;
  a.Hp = g.Hp;
  a.Wp = g.Wp;
  a.scale = scale;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.lc = lc;
  if (cudaFuncSetAttribute(attn_bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) != cudaSuccess)
    return WAN_ERR_CUDA;
  dim3 grid((L + kTile - 1) / kTile, H, B);
  record_start(lc, s);
  attn_bwd_kernel<<<grid, kThreads, kSmemBytes, s>>>(tq, tk, tv, tdo, tdq, a);
  record_stop(lc, s);
  if (cudaGetLastError() != cudaSuccess) return WAN_ERR_CUDA;
  record_pass(lc, kPassPost, 0, s);
  if (launch_rope_unrotate_f32(w.dq_acc, dq, B, g, H, tab, s) != cudaSuccess) return WAN_ERR_CUDA;
  record_pass(lc, kPassPost, 1, s);
  return WAN_OK;
}

}  // namespace wan
