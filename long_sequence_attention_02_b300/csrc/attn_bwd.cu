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
//      and the threads add dQ_i into the fp32 accumulator with vector atomics.
//      TMEM: dV [0,128) dK [128,256) S [256,384) dP [384,512); P^T, dS^T
//      (bf16) and the dQ halves reuse S and dP columns once the MMAs that read
//      them are ordered before (tcgen05 MMAs of one thread run in order).
//      Epilogue: dV -> bf16; dK -> R^T -> bf16.
//   3. post: dQ = R^T dQ_acc -> bf16.
// Warps: 0-7 compute (warp w: TMEM lanes 32*(w%4).., column half w/4),
// 8 TMA producer, 9 MMA issuer and TMEM owner.
#include "common.cuh"
#include "kernels.cuh"

namespace wan {

namespace {

constexpr int kThreads = 320;
constexpr int kLoadWarp = 8;
constexpr int kMmaWarp = 9;
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
constexpr int kSmemBytes = kOffBar + 256;

enum Bar {
  kBarKV = 0,
  kBarQFull0 = 1,   // +stage
  kBarQEmpty0 = 3,  // +stage
  kBarS = 5,
  kBarDP = 6,
  kBarP = 7,
  kBarDS = 8,
  kBarDQ = 9,
  kBarDQFree = 10,
  kBarAcc = 11,
  kBarDrain = 12,
  kNumBars = 13
};

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
  tmem_ld_wait();
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const BwdArgs a) {
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
    }
    mbar_init(&bars[kBarS], 1);
    mbar_init(&bars[kBarDP], 1);
    mbar_init(&bars[kBarP], 8);
    mbar_init(&bars[kBarDS], 8);
    mbar_init(&bars[kBarDQ], 1);
    mbar_init(&bars[kBarDQFree], 8);
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
  const uint32_t tDV = tmem, tDK = tmem + 128, tS = tmem + 256, tDP = tmem + 384;

  const size_t bh = static_cast<size_t>(b) * a.H + h;

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
      int issued[2] = {0, 0};
      for (int i = 0; i < nq; ++i) {
        const int s = i & 1, use = i >> 1;
        if (use > 0 && !mbar_wait(&bars[kBarQEmpty0 + s], (use - 1) & 1, abort, to)) {
          raise_abort(abort, a.lc.err);
          break;
        }
        if (a.lc.stall && i == 1) continue;  // test hook: query tile 1 never arrives
        uint8_t* st = smem + kOffStage + s * kStageBytes;
        uint8_t* rows = smem + kOffRows + s * kRowsBytes;
        uint64_t* bar = &bars[kBarQFull0 + s];
        mbar_arrive_expect_tx(bar, 2 * kTileBytes + kRowsBytes);
        const int q0 = i * kTile;
        tma_load_4d(st, &tm_q, bar, 0, h, q0, b);
        tma_load_4d(st + kHalfBytes, &tm_q, bar, 64, h, q0, b);
        tma_load_4d(st + kTileBytes, &tm_do, bar, 0, h, q0, b);
        tma_load_4d(st + kTileBytes + kHalfBytes, &tm_do, bar, 64, h, q0, b);
        bulk_load(rows, a.lse2 + bh * a.Lpad + q0, kTile * 4, bar);
        bulk_load(rows + kTile * 4, a.drow + bh * a.Lpad + q0, kTile * 4, bar);
        issued[s] = use + 1;
      }
      // Every copy this warp issued lands before the CTA may exit.
      mbar_wait(&bars[kBarKV], 0, nullptr, to);
      for (int s = 0; s < 2; ++s)
        if (issued[s] > 0) mbar_wait(&bars[kBarQFull0 + s], (issued[s] - 1) & 1, nullptr, to);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t id_kk = idesc_bf16_f32(128, 128, 0, 0);  // both operands K-major
      const uint32_t id_tm = idesc_bf16_f32(128, 128, 0, 1);  // A from TMEM, B MN-major
      const uint32_t id_dq = idesc_bf16_f32(128, 64, 1, 1);   // A and B MN-major, N = 64
      const uint32_t sK = smem_u32(smem + kOffK), sV = smem_u32(smem + kOffV);
      const uint32_t sDS = smem_u32(smem + kOffDS);
      bool ok = mbar_wait(&bars[kBarKV], 0, abort, to);
      for (int i = 0; i < nq && ok; ++i) {
        const int s = i & 1, use = i >> 1;
        const uint32_t sQ = smem_u32(smem + kOffStage + s * kStageBytes);
        const uint32_t sDO = sQ + kTileBytes;
        ok = mbar_wait(&bars[kBarQFull0 + s], use & 1, abort, to);
        if (ok && i > 0) ok = mbar_wait(&bars[kBarDQFree], (i - 1) & 1, abort, to);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
          umma_ss(tS, sdesc_sw128(sK + off, 16, 1024), sdesc_sw128(sQ + off, 16, 1024), id_kk, kk > 0);
        }
        umma_commit(&bars[kBarS]);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
          umma_ss(tDP, sdesc_sw128(sV + off, 16, 1024), sdesc_sw128(sDO + off, 16, 1024), id_kk, kk > 0);
        }
        umma_commit(&bars[kBarDP]);
        if (!(ok = mbar_wait(&bars[kBarP], i & 1, abort, to))) break;
        tc_fence_after();
        // P^T sits in S columns [0,32) (queries 0..63) and [64,96) (queries 64..127).
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ts(tDV, tS + (kk >> 2) * 64 + (kk & 3) * 8, sdesc_sw128(sDO + kk * 2048, kHalfBytes, 1024), id_tm,
                  (i > 0 || kk > 0) ? 1u : 0u);
        if (!(ok = mbar_wait(&bars[kBarDS], i & 1, abort, to))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ts(tDK, tDP + (kk >> 2) * 64 + (kk & 3) * 8, sdesc_sw128(sQ + kk * 2048, kHalfBytes, 1024), id_tm,
                  (i > 0 || kk > 0) ? 1u : 0u);
        // dQ_i = dS K_rot, d-halves into S[64,128) and dP[64,128).
#pragma unroll
        for (int half = 0; half < 2; ++half)
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma_ss((half ? tDP : tS) + 64, sdesc_sw128(sDS + kk * 2048, kHalfBytes, 1024),
                    sdesc_sw128(sK + half * kHalfBytes + kk * 2048, kHalfBytes, 1024), id_dq, kk > 0);
        umma_commit(&bars[kBarDQ]);
        umma_commit(&bars[kBarQEmpty0 + s]);
      }
      if (ok) umma_commit(&bars[kBarAcc]);
      if (!ok) raise_abort(abort, a.lc.err);
      umma_commit(&bars[kBarDrain]);
      mbar_wait(&bars[kBarDrain], 0, nullptr, to);
    }
    __syncwarp();
  } else {
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
      float p[64];
      {
        float sv[32];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          load32(tS + lane_addr + ch * 64 + c * 32, sv);
#pragma unroll
          for (int k = 0; k < 32; ++k) p[c * 32 + k] = key_ok ? ex2_approx(fmaf(sv[k], sl2, -lse2[c * 32 + k])) : 0.f;
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
        float dv[32];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          load32(tDP + lane_addr + ch * 64 + c * 32, dv);
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const int j0 = c * 32 + 2 * k;
            const float d0 = p[j0] * (dv[2 * k] - drow[j0]) * a.scale;
            const float d1 = p[j0 + 1] * (dv[2 * k + 1] - drow[j0 + 1]) * a.scale;
            pk[c * 16 + k] = pack_bf16x2(d0, d1);
          }
        }
        tmem_st32(tDP + lane_addr + ch * 64, pk);
        // dS^T row r, queries ch*64 .. ch*64+63 -> half tile ch of the MN-major A operand.
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

      if (!(ok = warp_wait(&bars[kBarDQ], i & 1, abort, a.lc.err, to))) break;
      tc_fence_after();
      float dq[64];
      {
        float t32[32];
        load32((ch ? tDP : tS) + lane_addr + 64, t32);
#pragma unroll
        for (int k = 0; k < 32; ++k) dq[k] = t32[k];
        load32((ch ? tDP : tS) + lane_addr + 96, t32);
#pragma unroll
        for (int k = 0; k < 32; ++k) dq[32 + k] = t32[k];
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kBarDQFree]);
      const int qrow = i * kTile + r;  // TMEM lane = query row of this tile
      if (qrow < a.L) {
        float4* dst = reinterpret_cast<float4*>(a.dq_acc + ((static_cast<size_t>(b) * a.L + qrow) * a.H + h) * 128 +
                                                ch * 64);
#pragma unroll
        for (int k = 0; k < 16; ++k)
          atomicAdd(dst + k, make_float4(dq[4 * k], dq[4 * k + 1], dq[4 * k + 2], dq[4 * k + 3]));
      }
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

// D_i = sum_d dO_id O_id and LSE_i * log2(e) into rows padded to a multiple
// of 128 (pad: D = 0, LSE = +inf). 16 threads per (b, l, h) row, 16 bytes each.
__global__ void __launch_bounds__(256) bwd_rows_kernel(const uint4* o, const uint4* dout, const float* lse,
                                                       float* lse2, float* drow, long long n_rows, int L, int Lpad,
                                                       int H) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n_rows * 16; i += stride) {
    const uint4 x = o[i], y = dout[i];
    const uint32_t xa[4] = {x.x, x.y, x.z, x.w}, ya[4] = {y.x, y.y, y.z, y.w};
    float acc = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      acc = fmaf(__uint_as_float(xa[k] << 16), __uint_as_float(ya[k] << 16), acc);
      acc = fmaf(__uint_as_float(xa[k] & 0xFFFF0000u), __uint_as_float(ya[k] & 0xFFFF0000u), acc);
    }
    // A row's 16 chunks are 16 aligned lanes that enter and leave the loop together.
    const unsigned group = 0xFFFFu << (threadIdx.x & 16);
#pragma unroll
    for (int m = 8; m >= 1; m >>= 1) acc += __shfl_xor_sync(group, acc, m, 16);
    if ((i & 15) == 0) {
      const long long row = i >> 4;  // (b*L + l)*H + h
      const int hh = (int)(row % H);
      const long long bl = row / H;
      const int l = (int)(bl % L);
      const long long bb = bl / L;
      const size_t dst = (size_t)(bb * H + hh) * Lpad + l;
      drow[dst] = acc;
      lse2[dst] = lse[(size_t)(bb * H + hh) * L + l] * 1.4426950408889634f;
    }
  }
}

__global__ void bwd_pad_kernel(float* lse2, float* drow, int BH, int L, int Lpad) {
  const int pad = Lpad - L;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < BH * pad; i += gridDim.x * blockDim.x) {
    const size_t dst = (size_t)(i / pad) * Lpad + L + (i % pad);
    lse2[dst] = INFINITY;
    drow[dst] = 0.f;
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
  if (launch_rope_rotate_bf16(k, w.k_rot, B, g, H, tab, false, s) != cudaSuccess) return WAN_ERR_CUDA;
  const long long n_rows = (long long)B * L * H;
  {
    long long want = (n_rows * 16 + 255) / 256, cap = (long long)sms * 8;
    bwd_rows_kernel<<<(int)(want < cap ? want : cap), 256, 0, s>>>((const uint4*)o, (const uint4*)dout, lse, w.lse2,
                                                                   w.drow, n_rows, L, Lpad, H);
    if (Lpad > L) bwd_pad_kernel<<<sms, 256, 0, s>>>(w.lse2, w.drow, B * H, L, Lpad);
  }
  if (cudaMemsetAsync(w.dq_acc, 0, (size_t)n_rows * 512, s) != cudaSuccess) return WAN_ERR_CUDA;

  CUtensorMap tq, tk, tv, tdo;
  if (!make_tmap_bld(&tq, w.q_rot, B, L, H, kHeadDim, 128) || !make_tmap_bld(&tk, w.k_rot, B, L, H, kHeadDim, 128) ||
      !make_tmap_bld(&tv, v, B, L, H, kHeadDim, 128) || !make_tmap_bld(&tdo, dout, B, L, H, kHeadDim, 128))
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
  attn_bwd_kernel<<<grid, kThreads, kSmemBytes, s>>>(tq, tk, tv, tdo, a);
  record_stop(lc, s);
  if (cudaGetLastError() != cudaSuccess) return WAN_ERR_CUDA;
  if (launch_rope_unrotate_f32(w.dq_acc, dq, B, g, H, tab, s) != cudaSuccess) return WAN_ERR_CUDA;
  return WAN_OK;
}

}  // namespace wan
