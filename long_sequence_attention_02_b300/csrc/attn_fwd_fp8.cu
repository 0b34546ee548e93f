// FP8 (e4m3) forward of 3D-RoPE self-attention for sm_103a.
//
// The Wan report lists FP8 attention among its inference speed-ups ("Wan Team,
// Alibaba (2025)" anthology note, Key takeaways: FP8 attention; ctol.digital
// article, "Speed, Scale, and Efficiency": diffusion cache, FP8 quantisation
// and activation offload give a 1.62x speed-up). The pages give no scheme;
// this file implements the plain per-head reading:
//   sq = amax|Q_rot| / 448, sk = amax|K_rot| / 448, sv = amax|V| / 448 for each (b, h);
//   Q8 = e4m3(Q_rot / sq), K8 = e4m3(K_rot / sk), V8 = e4m3(V / sv);
//   S = sq sk scale (Q8 K8^T);  P = 2^(S log2 e - m log2 e) with a running reference m;
//   P8 = e4m3(P) (P <= 256 < 448);  O = sv (P8 V8) / l,  l = sum of the fp32 P;
// every e4m3 rounding is to nearest even, saturating at +-448.
//
// Steps: fp8_amax_kernel (per-head amax of the rotated Q, K and of V),
// fp8_quant_kernel (Q8, K8 in the [B, L, H, 128] layout; V8 transposed to
// [B, H, 128, Lpad] so that both MMAs read K-major tiles), then the
// persistent attention kernel below. It has the roles, pipeline and TMEM
// layout of the bf16 kernel in attn_fwd.cu:
// - a tile is 128 rows x 128 bytes (one 128-byte swizzle atom across d);
// - each tcgen05.mma of kind::f8f6f4 covers K = 32, so QK and PV take 4
//   instructions per 128x128 tile instead of 8;
// - P is written to TMEM as e4m3, four per column, as the A operand of PV.
#include <climits>

#include "common.cuh"
#include "kernels.cuh"

namespace wan {

namespace {

constexpr int kTile = 128;
constexpr int kQTiles = 2;
constexpr int kTile8Bytes = 128 * 128;  // 16 KB
constexpr int kStages8 = 8;
constexpr int kThreads8 = 384;
constexpr uint32_t kSoftmaxRegs8 = 216;
constexpr uint32_t kControlRegs8 = 72;
constexpr int kLoadWarp8 = 8;
constexpr int kMmaWarp8 = 9;
constexpr int kQLoadWarp8 = 10;
constexpr int kSmemBytes8 = (kQTiles + kStages8) * kTile8Bytes + 1024;
constexpr float kTileSumBound = 256.0f;  // see the softmax's reference maximum
constexpr float kE4m3Max = 448.0f;

struct Fp8Args {
  const float* amax;  // [B*H][3]: amax of Q_rot, K_rot, V
  float* lse;
  int L, H, B;
  int n_qpairs;
  float scale_log2;  // logit scale * log2(e)
  LaunchCommon lc;
};

__device__ __forceinline__ void raise_abort8(volatile int* abort, int* err) {
  *abort = 1;
  atomicCAS(err, 0, kDevTimeout);
}

__device__ __forceinline__ bool warp_wait8(uint64_t* bar, uint32_t parity, volatile int* abort, int* err,
                                           uint64_t to) {
  bool ok = mbar_wait(bar, parity, abort, to);
  ok = __all_sync(0xffffffffu, ok);
  if (!ok && (threadIdx.x & 31) == 0) raise_abort8(abort, err);
  return ok;
}

__device__ __forceinline__ float rope_cs_axis(const RopeTables& tab, int pair, int t, int h, int w, float& sn) {
  float2 cs;
  if (pair < kPairsT) cs = tab.t[t * kPairsT + pair];
  else if (pair < kPairsT + kPairsH) cs = tab.h[h * kPairsH + (pair - kPairsT)];
  else cs = tab.w[w * kPairsW + (pair - kPairsT - kPairsH)];
  sn = cs.y;
  return cs.x;
}

// 8 consecutive elements (chunk c of a 128-wide row) of token l, rotated by
// the 3D RoPE angles of l.
__device__ __forceinline__ void load_rotated8(const uint4* src, int c, int l, int Hp, int Wp, const RopeTables& tab,
                                              float (&x)[8]) {
  const uint4 v = *src;
  const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
  const int w = l % Wp;
  const int hh = (l / Wp) % Hp;
  const int t = l / (Wp * Hp);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float sn;
    const float cs = rope_cs_axis(tab, c * 4 + k, t, hh, w, sn);
    const float a = __uint_as_float(wd[k] << 16), b = __uint_as_float(wd[k] & 0xFFFF0000u);
    x[2 * k] = a * cs - b * sn;
    x[2 * k + 1] = a * sn + b * cs;
  }
}

__device__ __forceinline__ void load_plain8(const uint4* src, float (&x)[8]) {
  const uint4 v = *src;
  const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    x[2 * k] = __uint_as_float(wd[k] << 16);
    x[2 * k + 1] = __uint_as_float(wd[k] & 0xFFFF0000u);
  }
}

// Per-(b, h) amax of |Q_rot|, |K_rot| and |V|. Block = 256 rows of one
// (b, h): 16 threads per row, 8 elements each; one atomicMax per block and
// tensor (non-negative floats order like their bit patterns).
__global__ void __launch_bounds__(256) fp8_amax_kernel(const uint4* q, const uint4* k, const uint4* v,
                                                       unsigned int* amax_bits, int L, int H, int Hp, int Wp,
                                                       RopeTables tab) {
  const int h = blockIdx.y, b = blockIdx.z;
  const int c = threadIdx.x & 15;
  float mq = 0.f, mk = 0.f, mv = 0.f;
  for (int r = threadIdx.x >> 4; r < 256; r += 16) {
    const int l = blockIdx.x * 256 + r;
    if (l >= L) break;
    const size_t chunk = ((static_cast<size_t>(b) * L + l) * H + h) * 16 + c;
    float x[8];
    load_rotated8(q + chunk, c, l, Hp, Wp, tab, x);
#pragma unroll
    for (int i = 0; i < 8; ++i) mq = fmaxf(mq, fabsf(x[i]));
    load_rotated8(k + chunk, c, l, Hp, Wp, tab, x);
#pragma unroll
    for (int i = 0; i < 8; ++i) mk = fmaxf(mk, fabsf(x[i]));
    load_plain8(v + chunk, x);
#pragma unroll
    for (int i = 0; i < 8; ++i) mv = fmaxf(mv, fabsf(x[i]));
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    mq = fmaxf(mq, __shfl_xor_sync(0xffffffffu, mq, o));
    mk = fmaxf(mk, __shfl_xor_sync(0xffffffffu, mk, o));
    mv = fmaxf(mv, __shfl_xor_sync(0xffffffffu, mv, o));
  }
  __shared__ float red[3][8];
  const int warp = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) {
    red[0][warp] = mq;
    red[1][warp] = mk;
    red[2][warp] = mv;
  }
  __syncthreads();
  if (threadIdx.x < 3) {
    float m = 0.f;
    for (int w = 0; w < 8; ++w) m = fmaxf(m, red[threadIdx.x][w]);
    atomicMax(amax_bits + (static_cast<size_t>(b) * H + h) * 3 + threadIdx.x, __float_as_uint(m));
  }
}

__device__ __forceinline__ float quant_mult(float amax) { return amax > 0.f ? kE4m3Max / amax : 1.0f; }

// Q8, K8 = e4m3 of the rotated, scaled rows ([B, L, H, 128] bytes); V8
// transposed per head into [B, H, 128, Lpad] bytes (zeros past L). Block =
// 128 tokens of one (b, h); V goes through shared memory in two passes of 64
// columns so that the transposed rows are written 16 bytes at a time.
__global__ void __launch_bounds__(256) fp8_quant_kernel(const uint4* q, const uint4* k, const uint4* v,
                                                        const float* amax, uint8_t* q8, uint8_t* k8, uint8_t* vt8,
                                                        int L, int Lpad, int H, int Hp, int Wp, RopeTables tab) {
  __shared__ float vs[128][65];  // [token][d within the pass], padded against bank conflicts
  const int h = blockIdx.y, b = blockIdx.z;
  const int l0 = blockIdx.x * 128;
  const float* am = amax + (static_cast<size_t>(b) * H + h) * 3;
  const float mq = quant_mult(am[0]), mk = quant_mult(am[1]), mv = quant_mult(am[2]);
  const int c = threadIdx.x & 15;
  for (int r = threadIdx.x >> 4; r < 128; r += 16) {
    const int l = l0 + r;
    if (l >= L) continue;
    const size_t chunk = ((static_cast<size_t>(b) * L + l) * H + h) * 16 + c;
    float x[8];
    load_rotated8(q + chunk, c, l, Hp, Wp, tab, x);
    uint2 o;
    o.x = pack_e4m3x4(x[0] * mq, x[1] * mq, x[2] * mq, x[3] * mq);
    o.y = pack_e4m3x4(x[4] * mq, x[5] * mq, x[6] * mq, x[7] * mq);
    *reinterpret_cast<uint2*>(q8 + chunk * 8) = o;
    load_rotated8(k + chunk, c, l, Hp, Wp, tab, x);
    o.x = pack_e4m3x4(x[0] * mk, x[1] * mk, x[2] * mk, x[3] * mk);
    o.y = pack_e4m3x4(x[4] * mk, x[5] * mk, x[6] * mk, x[7] * mk);
    *reinterpret_cast<uint2*>(k8 + chunk * 8) = o;
  }
  for (int pass = 0; pass < 2; ++pass) {
    // rows of 64 values: 8 threads per token, 8 values each
    const int cc = threadIdx.x & 7;
    for (int r = threadIdx.x >> 3; r < 128; r += 32) {
      const int l = l0 + r;
      float x[8];
      if (l < L) {
        load_plain8(v + ((static_cast<size_t>(b) * L + l) * H + h) * 16 + pass * 8 + cc, x);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) x[i] = 0.f;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) vs[r][cc * 8 + i] = x[i] * mv;
    }
    __syncthreads();
    // V^T rows: thread -> (d = 64 * pass + tid / 4, tokens 32 * (tid & 3) .. +32)
    const int dl = threadIdx.x >> 2;
    const int tb = (threadIdx.x & 3) * 32;
    uint8_t* dst = vt8 + ((static_cast<size_t>(b) * H + h) * 128 + pass * 64 + dl) * Lpad + l0 + tb;
#pragma unroll
    for (int g = 0; g < 2; ++g) {
      const int t0 = tb + g * 16;
      if (l0 + t0 >= Lpad) break;  // Lpad is a multiple of 16
      uint4 o;
      o.x = pack_e4m3x4(vs[t0 + 0][dl], vs[t0 + 1][dl], vs[t0 + 2][dl], vs[t0 + 3][dl]);
      o.y = pack_e4m3x4(vs[t0 + 4][dl], vs[t0 + 5][dl], vs[t0 + 6][dl], vs[t0 + 7][dl]);
      o.z = pack_e4m3x4(vs[t0 + 8][dl], vs[t0 + 9][dl], vs[t0 + 10][dl], vs[t0 + 11][dl]);
      o.w = pack_e4m3x4(vs[t0 + 12][dl], vs[t0 + 13][dl], vs[t0 + 14][dl], vs[t0 + 15][dl]);
      *reinterpret_cast<uint4*>(dst + g * 16) = o;
    }
    __syncthreads();
  }
}

__global__ void __launch_bounds__(kThreads8, 1)
    attn_fwd_fp8_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_vt, const __grid_constant__ CUtensorMap tm_o,
                        const Fp8Args a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;                               // 2 tiles of 128 x 128 bytes
  uint8_t* sKV = smem + kQTiles * kTile8Bytes;      // ring of K and V^T tiles

  __shared__ __align__(8) uint64_t bar_q_full, bar_q_empty;
  __shared__ __align__(8) uint64_t bar_kv_full[kStages8], bar_kv_empty[kStages8];
  __shared__ __align__(8) uint64_t bar_s_full[kQTiles], bar_p_full[kQTiles], bar_o_full[kQTiles];
  __shared__ __align__(8) uint64_t bar_drain;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  __shared__ int epi_ok[kQTiles][4];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t to = a.lc.timeout_ns;
  volatile int* abort = &abort_sh;
  const int n_items = a.n_qpairs * a.H * a.B;
  const int n_tiles = (a.L + kTile - 1) / kTile;

  struct Item {
    int b, h, q0, kv_start;
  };
  auto item_of = [&](int it) {
    Item x;
    const int qp = it % a.n_qpairs;
    const int bh = it / a.n_qpairs;
    x.h = bh % a.H;
    x.b = bh / a.H;
    x.q0 = qp * (kTile * kQTiles);
    x.kv_start = static_cast<int>((static_cast<long long>(qp) * n_tiles) / a.n_qpairs);
    WAN_DCHECK(x.b < a.B && x.h < a.H && x.q0 < a.L && x.kv_start < n_tiles, a.lc.err);
    return x;
  };

  if (threadIdx.x == 0) {
    mbar_init(&bar_q_full, 1);
    mbar_init(&bar_q_empty, kQTiles);
    for (int t = 0; t < kQTiles; ++t) {
      mbar_init(&bar_s_full[t], 1);
      mbar_init(&bar_p_full[t], 4);
      mbar_init(&bar_o_full[t], 1);
    }
    for (int s = 0; s < kStages8; ++s) {
      mbar_init(&bar_kv_full[s], 1);
      mbar_init(&bar_kv_empty[s], 1);
    }
    mbar_init(&bar_drain, 1);
    abort_sh = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp8) {
    tmem_alloc(&tmem_base_sh, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  // Debug builds: the 512 TMEM columns start at lane 0 / column 0, and the
  // swizzled tiles need a 1024-byte aligned shared-memory base.
  if (threadIdx.x == 0) {
    WAN_DCHECK(!a.lc.force_check, a.lc.err);
    WAN_DCHECK(tmem == 0u, a.lc.err);
    WAN_DCHECK((smem_u32(smem) & 1023u) == 0u, a.lc.err);
  }

  if (warp >= 8) {
   regs_shrink<kControlRegs8>();
   if (warp == kLoadWarp8) {
    // ------------------------------------------------------------ K / V^T producer
    if (lane == 0) {
      int ig = 0;
      bool ok = true;
      for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
        const Item x = item_of(it);
        for (int i = 0; i < 2 * n_tiles; ++i, ++ig) {
          const int slot = ig % kStages8;
          const int use = ig / kStages8;
          if (use > 0 && !mbar_wait(&bar_kv_empty[slot], (use - 1) & 1, abort, to)) {
            raise_abort8(abort, a.lc.err);
            ok = false;
            break;
          }
          if (a.lc.stall && ig == 1) continue;  // test hook: V_0 never arrives
          const int jt = (i >> 1) + x.kv_start;
          const int key0 = (jt < n_tiles ? jt : jt - n_tiles) * kTile;
          uint8_t* dst = sKV + slot * kTile8Bytes;
          mbar_arrive_expect_tx(&bar_kv_full[slot], kTile8Bytes);
          if (i & 1)
            tma_load_4d(dst, &tm_vt, &bar_kv_full[slot], key0, 0, x.h, x.b);   // V^T: 128 d rows x 128 keys
          else
            tma_load_4d(dst, &tm_k, &bar_kv_full[slot], 0, x.h, key0, x.b);   // K: 128 keys x 128 d
        }
      }
      for (int k = ig - kStages8 < 0 ? 0 : ig - kStages8; k < ig; ++k)
        mbar_wait(&bar_kv_full[k % kStages8], (k / kStages8) & 1, nullptr, to);
    }
    __syncwarp();
   } else if (warp == kQLoadWarp8) {
    // ------------------------------------------------------------ Q producer
    if (lane == 0) {
      int nq = 0;
      for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
        const Item x = item_of(it);
        if (nq > 0 && !mbar_wait(&bar_q_empty, (nq - 1) & 1, abort, to)) {
          raise_abort8(abort, a.lc.err);
          break;
        }
        mbar_arrive_expect_tx(&bar_q_full, kQTiles * kTile8Bytes);
        for (int t = 0; t < kQTiles; ++t)
          tma_load_4d(sQ + t * kTile8Bytes, &tm_q, &bar_q_full, 0, x.h, x.q0 + t * kTile, x.b);
        ++nq;
      }
      if (nq > 0) mbar_wait(&bar_q_full, (nq - 1) & 1, nullptr, to);
    }
    __syncwarp();
   } else if (warp == kMmaWarp8) {
    // ------------------------------------------------------------ MMA issuer
    {
      const uint32_t idesc = idesc_e4m3_f32(128, 128);
      const uint64_t dq = sdesc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t dkv = sdesc_sw128(smem_u32(sKV), 16, 1024);
      const uint32_t hi = static_cast<uint32_t>(dq >> 32);
      const uint32_t q_lo = static_cast<uint32_t>(dq), kv_lo = static_cast<uint32_t>(dkv);
      auto issue_qk = [&](int t, int slot) {
        const uint32_t qd = q_lo + static_cast<uint32_t>(t * (kTile8Bytes >> 4));
        const uint32_t kd = kv_lo + static_cast<uint32_t>(slot * (kTile8Bytes >> 4));
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)  // K = 32 bytes per MMA
          umma_ss_elect_lo_f8(tmem + t * 128, qd + kk * 2, kd + kk * 2, hi, idesc, kk > 0);
      };
      auto issue_pv = [&](int t, int slot, bool acc) {
        const uint32_t vd = kv_lo + static_cast<uint32_t>(slot * (kTile8Bytes >> 4));
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)  // P: 8 TMEM columns (32 keys) per MMA
          umma_ts_elect_lo_f8(tmem + 256 + t * 128, tmem + t * 128 + kk * 8, vd + kk * 2, hi, idesc,
                              (acc || kk > 0) ? 1u : 0u);
      };
      bool ok = true;
      int nq = 0, ig = 0, sp = 0;
      for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
        ok = warp_wait8(&bar_q_full, nq & 1, abort, a.lc.err, to);
        if (!ok) break;
        const int k0 = ig % kStages8;
        ok = warp_wait8(&bar_kv_full[k0], (ig / kStages8) & 1, abort, a.lc.err, to);
        if (!ok) break;
        tc_fence_after();
        issue_qk(0, k0);
        umma_commit_elect(&bar_s_full[0]);
        issue_qk(1, k0);
        umma_commit_elect(&bar_s_full[1]);
        umma_commit_elect(&bar_kv_empty[k0]);
        for (int j = 0; j < n_tiles && ok; ++j) {
          const int iv = ig + 2 * j + 1;
          const int vslot = iv % kStages8;
          ok = warp_wait8(&bar_kv_full[vslot], (iv / kStages8) & 1, abort, a.lc.err, to);
          const bool has_next = j + 1 < n_tiles;
          const int ik = ig + 2 * j + 2;
          const int kslot = ik % kStages8;
          if (ok && has_next) ok = warp_wait8(&bar_kv_full[kslot], (ik / kStages8) & 1, abort, a.lc.err, to);
          for (int t = 0; t < kQTiles && ok; ++t) {
            ok = warp_wait8(&bar_p_full[t], (sp + j) & 1, abort, a.lc.err, to);
            if (!ok) break;
            tc_fence_after();
            issue_pv(t, vslot, j > 0);
            if (t == kQTiles - 1) umma_commit_elect(&bar_kv_empty[vslot]);
            if (!has_next) {
              umma_commit_elect(&bar_o_full[t]);
            } else {
              issue_qk(t, kslot);
              umma_commit_elect(&bar_s_full[t]);
              if (t == kQTiles - 1) umma_commit_elect(&bar_kv_empty[kslot]);
            }
          }
        }
        ig += 2 * n_tiles;
        sp += n_tiles;
        ++nq;
      }
      umma_commit_elect(&bar_drain);
      mbar_wait(&bar_drain, 0, nullptr, to);
    }
   }
  } else {
    regs_grow<kSoftmaxRegs8>();
    // ------------------------------------------------------------ softmax
    // As in the bf16 kernel, a warp whose wait failed skips the work but keeps
    // walking the items, so the four warps of a tile pass the same barriers.
    const int t = warp >> 2;
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + lane_addr + t * 128;
    const uint32_t tO = tmem + lane_addr + 256 + t * 128;
    const int valid_last = a.L - (n_tiles - 1) * kTile;  // keys in the last key tile
    bool ok = true;
    int nq = 0, sp = 0;
    for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
      int kv_start, bh;
      {
        const Item x = item_of(it);
        kv_start = x.kv_start;
        bh = x.b * a.H + x.h;
      }
      const float* am = a.amax + static_cast<size_t>(bh) * 3;
      const float dq = am[0] / kE4m3Max, dk = am[1] / kE4m3Max;
      const float sl2 = a.scale_log2 * (am[0] > 0.f ? dq : 1.f) * (am[1] > 0.f ? dk : 1.f);
      float m_ref = -INFINITY;
      float l = 0.f;
      for (int j = 0; j < n_tiles && ok; ++j) {
        ok = warp_wait8(&bar_s_full[t], (sp + j) & 1, abort, a.lc.err, to);
        if (!ok) break;
        tc_fence_after();
        uint32_t sr[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, sr[c]);
        tmem_ld_wait_regs(sr);
#define WAN_S(e) __uint_as_float(sr[(e) >> 5][(e) & 31])
        const int jt = j + kv_start < n_tiles ? j + kv_start : j + kv_start - n_tiles;
        if (jt == n_tiles - 1 && valid_last < kTile) {
#pragma unroll
          for (int i = 0; i < 128; ++i)
            if (i >= valid_last) sr[i >> 5][i & 31] = __float_as_uint(-INFINITY);
        }
        // Reference maximum as in the bf16 kernel: the item's first key tile
        // sets m_ref; a later tile whose row sum of P stays <= kTileSumBound
        // has every P <= kTileSumBound < 448, inside the e4m3 range, and
        // needs no maximum of its own; a row above the bound moves m_ref to
        // the tile's maximum, rescales O and l, and the tile is recomputed.
        auto row_max = [&]() {
          float mc[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) mc[q] = WAN_S(q);
#pragma unroll
          for (int i = 4; i < 128; i += 8) {
#pragma unroll
            for (int q = 0; q < 4; ++q) mc[q] = max3f(mc[q], WAN_S(i + 2 * q), WAN_S(i + 2 * q + 1));
          }
          return max3f(mc[0], mc[1], fmaxf(mc[2], mc[3]));
        };
        if (j == 0) m_ref = row_max();
        float tsum = 0.f;
#pragma unroll 1
        for (int pass = 0; pass < 2; ++pass) {
          const float neg = -m_ref * sl2;
          const uint64_t sl2x2 = f2_pack(sl2, sl2);
          const uint64_t negx2 = f2_pack(neg, neg);
          uint64_t acc[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t pk[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {  // keys c*32 + 4i .. +3 -> one TMEM column
              const int e = c * 32 + 4 * i;
              float p[4];
#pragma unroll
              for (int u = 0; u < 2; ++u) {
                const uint64_t xx = f2_fma(f2_pack(WAN_S(e + 2 * u), WAN_S(e + 2 * u + 1)), sl2x2, negx2);
                float x0, x1;
                f2_unpack(xx, x0, x1);
                p[2 * u] = ex2_approx(x0);
                p[2 * u + 1] = ex2_approx(x1);
                acc[u] = f2_add(acc[u], f2_pack(p[2 * u], p[2 * u + 1]));
              }
              pk[i] = pack_e4m3x4(p[0], p[1], p[2], p[3]);
            }
            tmem_st8(tS + c * 8, pk);
          }
          float a0, a1, a2, a3;
          f2_unpack(acc[0], a0, a1);
          f2_unpack(acc[1], a2, a3);
          tsum = (a0 + a1) + (a2 + a3);
          const bool need = !(tsum <= kTileSumBound);
          if (pass == 1 || !__any_sync(0xffffffffu, need)) break;
          const float m_new = need ? fmaxf(m_ref, row_max()) : m_ref;
          const float alpha = ex2_approx((m_ref - m_new) * sl2);  // 1 where no new reference
          l *= alpha;
          m_ref = m_new;
          tmem_st_wait();
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            uint32_t ov[32];
            tmem_ld32(tO + c * 32, ov);
            tmem_ld_wait_regs(ov);
#pragma unroll
            for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
            tmem_st32(tO + c * 32, ov);
          }
        }
#undef WAN_S
        l += tsum;
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_p_full[t]);
      }

      // ---------------------------------------------------------- epilogue
      // O_t * sv / l -> bf16. Tile t's own 16 KB Q tile (free once O_t is
      // final: every QK MMA was issued before the last PV) stages the bf16
      // output in two rounds of 64 columns, each 128 rows x 128 bytes in the
      // 128-byte swizzled layout and written by one TMA store. The Q buffer
      // goes back to the Q producer after both tiles' stores have read it.
      if (ok) ok = warp_wait8(&bar_o_full[t], nq & 1, abort, a.lc.err, to);
      if (lane == 0) epi_ok[t][wq] = ok ? 1 : 0;
      named_bar_sync(1 + t, 128);
      const bool all_ok = epi_ok[t][0] & epi_ok[t][1] & epi_ok[t][2] & epi_ok[t][3];
      ok = ok && all_ok;
      const Item x = item_of(it);
      uint8_t* stage = sQ + t * kTile8Bytes;
      const int row = x.q0 + t * kTile + r;
      const float dv = a.amax[static_cast<size_t>(bh) * 3 + 2] / kE4m3Max;
      const float inv = (a.amax[static_cast<size_t>(bh) * 3 + 2] > 0.f ? dv : 1.f) / l;
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        if (all_ok) {
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t ov[32];
            tmem_ld32(tO + half * 64 + c * 32, ov);
            tmem_ld_wait_regs(ov);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int chunk = 4 * c + q;  // 16-byte chunk of the 64-column half row
              *reinterpret_cast<uint4*>(stage + sw128_offset(r, chunk)) =
                  make_uint4(pack_bf16x2(__uint_as_float(ov[8 * q]) * inv, __uint_as_float(ov[8 * q + 1]) * inv),
                             pack_bf16x2(__uint_as_float(ov[8 * q + 2]) * inv, __uint_as_float(ov[8 * q + 3]) * inv),
                             pack_bf16x2(__uint_as_float(ov[8 * q + 4]) * inv, __uint_as_float(ov[8 * q + 5]) * inv),
                             pack_bf16x2(__uint_as_float(ov[8 * q + 6]) * inv, __uint_as_float(ov[8 * q + 7]) * inv));
            }
          }
          if (half == 0 && a.lse && row < a.L)
            a.lse[static_cast<size_t>(bh) * a.L + row] = (m_ref * sl2 + __log2f(l)) * 0.69314718055994531f;
          fence_proxy_async_smem();
        }
        named_bar_sync(1 + t, 128);
        if (all_ok && wq == 0 && lane == 0) {
          tma_store_4d(&tm_o, stage, half * 64, x.h, x.q0 + t * kTile, x.b);
          bulk_commit_group();
          bulk_wait_group_read0();
          if (half == 1) mbar_arrive(&bar_q_empty);
        }
        named_bar_sync(1 + t, 128);
      }
      sp += n_tiles;
      ++nq;
    }
  }

  if (warp == 0 || warp == 4) bulk_wait_group0();
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp8) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

size_t attn_fwd_fp8_workspace_bytes(int B, int L, int H) {
  const size_t n = static_cast<size_t>(B) * L * H * 128;
  const size_t lpad = (static_cast<size_t>(L) + 15) / 16 * 16;
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  return up(n) + up(n) + up(static_cast<size_t>(B) * H * 128 * lpad) + up(static_cast<size_t>(B) * H * 3 * 4);
}

int launch_attn_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse, int B, wan_grid_t g, int H,
                        RopeTables tab, float scale, void* workspace, const LaunchCommon& lc, cudaStream_t s) {
  const int L = g.F * g.Hp * g.Wp;
  const int Lpad = (L + 15) / 16 * 16;
  const size_t n = static_cast<size_t>(B) * L * H * 128;
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  uint8_t* base = static_cast<uint8_t*>(workspace);
  uint8_t* q8 = base;
  uint8_t* k8 = q8 + up(n);
  uint8_t* vt8 = k8 + up(n);
  float* amax = reinterpret_cast<float*>(vt8 + up(static_cast<size_t>(B) * H * 128 * Lpad));

  if (cudaMemsetAsync(amax, 0, static_cast<size_t>(B) * H * 3 * 4, s) != cudaSuccess) return WAN_ERR_CUDA;
  fp8_amax_kernel<<<dim3((L + 255) / 256, H, B), 256, 0, s>>>(
      static_cast<const uint4*>(q), static_cast<const uint4*>(k), static_cast<const uint4*>(v),
      reinterpret_cast<unsigned int*>(amax), L, H, g.Hp, g.Wp, tab);
  fp8_quant_kernel<<<dim3((L + 127) / 128, H, B), 256, 0, s>>>(
      static_cast<const uint4*>(q), static_cast<const uint4*>(k), static_cast<const uint4*>(v), amax, q8, k8, vt8, L,
      Lpad, H, g.Hp, g.Wp, tab);
  if (cudaGetLastError() != cudaSuccess) return WAN_ERR_CUDA;

  CUtensorMap tq, tk, tvt, to;
  const cuuint64_t dqk[4] = {128, (cuuint64_t)H, (cuuint64_t)L, (cuuint64_t)B};
  const cuuint64_t sqk[3] = {128, (cuuint64_t)H * 128, (cuuint64_t)L * H * 128};
  const cuuint32_t bqk[4] = {128, 1, 128, 1};
  const cuuint64_t dvt[4] = {(cuuint64_t)Lpad, 128, (cuuint64_t)H, (cuuint64_t)B};
  const cuuint64_t svt[3] = {(cuuint64_t)Lpad, (cuuint64_t)Lpad * 128, (cuuint64_t)Lpad * 128 * H};
  const cuuint32_t bvt[4] = {128, 128, 1, 1};
  if (!make_tmap_u8(&tq, q8, dqk, sqk, bqk) || !make_tmap_u8(&tk, k8, dqk, sqk, bqk) ||
      !make_tmap_u8(&tvt, vt8, dvt, svt, bvt) || !make_tmap_bld(&to, o, B, L, H, kHeadDim, 128))
    return WAN_ERR_CUDA;

  Fp8Args a;
  a.amax = amax;
  a.lse = lse;
  a.L = L;
  a.H = H;
  a.B = B;
  a.n_qpairs = (L + kTile * kQTiles - 1) / (kTile * kQTiles);
  a.scale_log2 = scale * 1.4426950408889634f;
  a.lc = lc;
  const long long n_items = static_cast<long long>(a.n_qpairs) * H * B;
  if (n_items > INT_MAX) return WAN_ERR_INVALID;
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return WAN_ERR_CUDA;
  const int grid = static_cast<int>(n_items < sms ? n_items : sms);
  if (cudaFuncSetAttribute(attn_fwd_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes8) !=
      cudaSuccess)
    return WAN_ERR_CUDA;
  record_start(lc, s);
  attn_fwd_fp8_kernel<<<grid, kThreads8, kSmemBytes8, s>>>(tq, tk, tvt, to, a);
  record_stop(lc, s);
  return cudaGetLastError() == cudaSuccess ? WAN_OK : WAN_ERR_CUDA;
}

}  // namespace wan
