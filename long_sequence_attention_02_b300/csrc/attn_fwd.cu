// Attention forward for sm_103a: tcgen05 MMAs with TMEM accumulators, TMA
// K/V tiles, online softmax.
//
// What is computed: for each (b, h) and query row i,
//   O_i = sum_j softmax_j(scale * q_i . k_j) v_j,   LSE_i = log sum_j exp(scale * q_i . k_j)
// over all keys (self-attention: full, non-causal spatio-temporal attention
// over every latent token - "Wan Team, Alibaba (2025)" anthology note, Key
// takeaways) or over the valid text keys (cross-attention to at most 512 umT5
// tokens - gojay.top "Wan2.1" reading, DiT backbone and config table ⑥).
// With 3D RoPE (same page, DiT 块) the query tile is rotated in shared memory
// right after it lands; keys arrive already rotated.
//
// Persistent CTAs (one per SM) walk a static list of work items; an item is
// 2 query tiles of 128 rows of one (b, h), processed against all key tiles.
// Three warpgroups (register budgets moved with setmaxnreg):
//   warps 0-3   softmax of query tile 0 (one thread per row)      216 regs
//   warps 4-7   softmax of query tile 1                           216 regs
//   warp  8     TMA producer of K_j, V_j (ring)
//   warp  9     MMA issuer (warp-converged, one elected lane) and TMEM owner
//   warp  10    TMA producer of the items' Q tiles
//   warp  11    O store: TMA stores of the staged O tiles, Q buffer release  72 regs
// Cross-attention items are short (at most 4 key tiles), so there Q is
// double-buffered: the next item's Q load and first QK overlap the current
// item's output epilogue. Self-attention uses one Q buffer and a 4-slot ring.
// TMEM (512 columns x 128 lanes, fp32): S0 [0,128) S1 [128,256) O0 [256,384)
// O1 [384,512). P_t (bf16, two per column) overwrites the first 64 columns of
// S_t and is the A operand of O_t += P_t V_j straight from TMEM.
// Each item visits its key tiles cyclically from an item-dependent start.
// Per key tile the MMA order is PV0(j), QK0(j+1), PV1(j), QK1(j+1): softmax of
// tile 0 for j+1 overlaps the tensor work of tile 1 and vice versa. Because
// tcgen05 MMAs from one thread run in issue order, QK_t(j+1) never overwrites
// P_t(j) before PV_t(j) has read it, and O_t is final for iteration j once
// S_t(j+1) is signalled. The same ordering lets an item's first PV, which
// overwrites O_t, follow the previous item's epilogue: the softmax warps read
// O_t out of TMEM before they signal the new item's first P.
// Softmax keeps a per-row reference m: the row maximum of the item's first
// key tile. Later tiles are exponentiated against m without their own
// maximum; only a tile whose row sum of p exceeds 256 (its maximum grew by
// about 2^8) moves m, rescales O (in TMEM) and l, and is recomputed. The
// final O / l is exact for any reference, and p <= 256 stays well inside bf16.
#include <climits>

#include "common.cuh"
#include "kernels.cuh"

namespace wan {

namespace {

constexpr int kBlockM = 128;
constexpr int kQTiles = 2;
constexpr int kBlockN = 128;
constexpr int kTileBytes = 128 * 128 * 2;
constexpr int kHalfBytes = kTileBytes / 2;
constexpr int kThreads = 384;
constexpr uint32_t kSoftmaxRegs = 216;  // 2 x 128 x 216 + 128 x 72 = 384 x 168
constexpr uint32_t kControlRegs = 72;
constexpr int kLoadWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kQLoadWarp = 10;
constexpr int kStoreWarp = 11;
// Q buffers and K/V ring slots (self-attention: 1 + 4, cross-attention: 2 + 3).
template <bool kRope>
struct FwdCfg {
  static constexpr int kQBuf = kRope ? 1 : 2;
  static constexpr int kStages = kRope ? 4 : 3;
  static constexpr int kSmemBytes = (kQBuf * kQTiles + kStages) * kTileBytes + 1024;
};
constexpr float kTileSumBound = 256.0f;  // see the softmax's reference maximum

struct FwdArgs {
  __nv_bfloat16* o;
  float* lse;
  const int32_t* kv_lens;
  RopeTables tab;
  int Lq, Lk, H, Hp, Wp, B;
  int n_qpairs;  // 256-row query blocks per (b, h)
  int q_pos0;    // grid token of query row 0 (a chunk of a longer sequence)
  float scale_log2;
  LaunchCommon lc;
};

__device__ __forceinline__ void raise_abort(volatile int* abort, int* err) {
  *abort = 1;
  atomicCAS(err, 0, kDevTimeout);
}

// Warp-uniform bounded wait.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort, int* err,
                                          uint64_t to) {
  bool ok = mbar_wait(bar, parity, abort, to);
  ok = __all_sync(0xffffffffu, ok);
  if (!ok && (threadIdx.x & 31) == 0) raise_abort(abort, err);
  return ok;
}

// Rotate row r of a swizzled [128 x 128] bf16 tile in place by the 3D RoPE
// angles of token `row`.
__device__ __forceinline__ void rope_row_in_smem(uint8_t* tile, int r, int row, const FwdArgs& a) {
  const int tok = row + a.q_pos0;
  const int w = tok % a.Wp;
  const int tmp = tok / a.Wp;
  const int hh = tmp % a.Hp;
  const int t = tmp / a.Hp;
  const float2* ct = a.tab.t + t * kPairsT;
  const float2* ch = a.tab.h + hh * kPairsH;
  const float2* cw = a.tab.w + w * kPairsW;
#pragma unroll 4
  for (int c = 0; c < 16; ++c) {
    uint4* p = reinterpret_cast<uint4*>(tile + (c >> 3) * kHalfBytes + sw128_offset(r, c & 7));
    uint4 v = *p;
    uint32_t wd[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int pair = c * 4 + k;
      const float2 cs = pair < kPairsT ? ct[pair] : (pair < kPairsT + kPairsH ? ch[pair - kPairsT]
                                                                                : cw[pair - kPairsT - kPairsH]);
      const float x0 = __uint_as_float(wd[k] << 16);
      const float x1 = __uint_as_float(wd[k] & 0xFFFF0000u);
      wd[k] = pack_bf16x2(x0 * cs.x - x1 * cs.y, x0 * cs.y + x1 * cs.x);
    }
    *p = make_uint4(wd[0], wd[1], wd[2], wd[3]);
  }
}

template <bool kRope, int kMerge>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                    const FwdArgs a) {
  constexpr int kQBuf = FwdCfg<kRope>::kQBuf;
  constexpr int kStages = FwdCfg<kRope>::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;                                    // [kQBuf][2 tiles]
  uint8_t* sKV = smem + kQBuf * kQTiles * kTileBytes;    // [kStages] tiles

  __shared__ __align__(8) uint64_t bar_q_full[kQBuf], bar_q_ready[kQBuf], bar_q_empty[kQBuf];
  __shared__ __align__(8) uint64_t bar_kv_full[kStages], bar_kv_empty[kStages];
  __shared__ __align__(8) uint64_t bar_s_full[kQTiles], bar_p_full[kQTiles], bar_o_full[kQTiles];
  __shared__ __align__(8) uint64_t bar_drain;
  __shared__ __align__(8) uint64_t bar_oldo[kQTiles];  // previous O tile loaded (merging epilogues)
  // O tile t of the item in Q buffer q written to its staging area. One
  // barrier per buffer: its next phase needs that buffer's next Q load,
  // which waits for the store warp to have consumed this one.
  __shared__ __align__(8) uint64_t bar_o_staged[kQBuf][kQTiles];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh;
  __shared__ int epi_ok[kQTiles][4];  // per-warp epilogue go/stop flags
  __shared__ int store_ok[kQBuf][kQTiles];  // staged O tile is valid (read by the store warp)
  // The first key lengths, read once per CTA instead of at every item.
  constexpr int kLensCached = 64;
  __shared__ int lens_sh[kLensCached];
  if (a.kv_lens != nullptr && threadIdx.x < kLensCached && static_cast<int>(threadIdx.x) < a.B)
    lens_sh[threadIdx.x] = a.kv_lens[threadIdx.x];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t to = a.lc.timeout_ns;
  volatile int* abort = &abort_sh;
  const int n_items = a.n_qpairs * a.H * a.B;

  // Work item -> (b, h, first query row, key tiles, first key tile). Every
  // role walks the same items, so all derive the same counters from them.
  struct Item {
    int b, h, q0, n_valid, n_tiles, kv_start;
  };
  auto item_of = [&](int it) {
    Item x;
    const int qp = it % a.n_qpairs;
    const int bh = it / a.n_qpairs;
    x.h = bh % a.H;
    x.b = bh / a.H;
    x.q0 = qp * (kBlockM * kQTiles);
    x.n_valid = a.Lk;
    if (a.kv_lens != nullptr) {
      const int v = x.b < kLensCached ? lens_sh[x.b] : a.kv_lens[x.b];
      x.n_valid = v < 0 ? 0 : (v > a.Lk ? a.Lk : v);
    }
    x.n_tiles = (x.n_valid + kBlockN - 1) / kBlockN;
    // Key tiles are visited from a per-item offset (online softmax does not
    // depend on the order), so that the CTAs of one head in flight read
    // different K/V tiles.
    x.kv_start = x.n_tiles > 0 ? static_cast<int>((static_cast<long long>(qp) * x.n_tiles) / a.n_qpairs) : 0;
    WAN_DCHECK(x.b < a.B && x.h < a.H && x.q0 < a.Lq && x.n_tiles * kBlockN < a.Lk + kBlockN &&
                   (x.n_tiles == 0 || x.kv_start < x.n_tiles),
               a.lc.err);
    return x;
  };

  if (threadIdx.x == 0) {
    for (int q = 0; q < kQBuf; ++q) {
      mbar_init(&bar_q_full[q], 1);
      mbar_init(&bar_q_ready[q], kRope ? 8 : 1);
      mbar_init(&bar_q_empty[q], 1);  // the store warp, once both O tiles' stores have read it
      for (int t = 0; t < kQTiles; ++t) mbar_init(&bar_o_staged[q][t], 4);
    }
    for (int t = 0; t < kQTiles; ++t) {
      mbar_init(&bar_s_full[t], 1);
      mbar_init(&bar_p_full[t], 4);
      mbar_init(&bar_o_full[t], 1);
      mbar_init(&bar_oldo[t], 1);
    }
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bar_kv_full[s], 1);
      mbar_init(&bar_kv_empty[s], 1);
    }
    mbar_init(&bar_drain, 1);
    abort_sh = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
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
   regs_shrink<kControlRegs>();
   if (warp == kLoadWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      int ig = 0;  // K/V tiles issued (ring position)
      bool ok = true;
      for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
        const Item x = item_of(it);
        if (x.n_tiles == 0) continue;
        for (int i = 0; i < 2 * x.n_tiles; ++i, ++ig) {
          const int slot = ig % kStages;
          const int use = ig / kStages;
          if (use > 0 && !mbar_wait(&bar_kv_empty[slot], (use - 1) & 1, abort, to)) {
            raise_abort(abort, a.lc.err);
            ok = false;
            break;
          }
          if (a.lc.stall && ig == 1) continue;  // test hook: V_0 never arrives
          const CUtensorMap* m = (i & 1) ? &tm_v : &tm_k;
          const int jt = (i >> 1) + x.kv_start;
          const int row = (jt < x.n_tiles ? jt : jt - x.n_tiles) * kBlockN;
          uint8_t* dst = sKV + slot * kTileBytes;
          mbar_arrive_expect_tx(&bar_kv_full[slot], kTileBytes);
          tma_load_4d(dst, m, &bar_kv_full[slot], 0, x.h, row, x.b);
          tma_load_4d(dst + kHalfBytes, m, &bar_kv_full[slot], 64, x.h, row, x.b);
        }
      }
      // Every copy this warp issued lands before the CTA may exit (on the
      // normal path the consumers already waited for all of them). The last
      // fill of each slot / buffer is that barrier's latest phase.
      for (int k = ig - kStages < 0 ? 0 : ig - kStages; k < ig; ++k)
        mbar_wait(&bar_kv_full[k % kStages], (k / kStages) & 1, nullptr, to);
    }
    __syncwarp();
   } else if (warp == kQLoadWarp) {
    // ------------------------------------------------------------ Q producer
    // Q tiles of each item go into their buffer as soon as it is free, so a
    // Q prefetch never waits behind the K/V ring.
    if (lane == 0) {
      int nq = 0;  // items whose Q was loaded
      for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
        const Item x = item_of(it);
        if (x.n_tiles == 0) continue;
        const int qb = nq % kQBuf;
        if (nq >= kQBuf && !mbar_wait(&bar_q_empty[qb], ((nq / kQBuf) - 1) & 1, abort, to)) {
          raise_abort(abort, a.lc.err);
          break;
        }
        uint8_t* qdst = sQ + qb * (kQTiles * kTileBytes);
        mbar_arrive_expect_tx(&bar_q_full[qb], kQTiles * kTileBytes);
        for (int t = 0; t < kQTiles; ++t) {
          tma_load_4d(qdst + t * kTileBytes, &tm_q, &bar_q_full[qb], 0, x.h, x.q0 + t * kBlockM, x.b);
          tma_load_4d(qdst + t * kTileBytes + kHalfBytes, &tm_q, &bar_q_full[qb], 64, x.h, x.q0 + t * kBlockM, x.b);
        }
        ++nq;
      }
      // Every Q copy lands before the CTA may exit.
      for (int k = nq - kQBuf < 0 ? 0 : nq - kQBuf; k < nq; ++k)
        mbar_wait(&bar_q_full[k % kQBuf], (k / kQBuf) & 1, nullptr, to);
    }
    __syncwarp();
   } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs this loop (waits and descriptor arithmetic are
    // warp-uniform); one elected lane issues each MMA and commit.
    {
      const uint32_t idesc_s = idesc_bf16_f32(128, 128, 0, 0);  // Q (K-major) x K (K-major)
      const uint32_t idesc_o = idesc_bf16_f32(128, 128, 0, 1);  // P (TMEM) x V (MN-major)
      // Descriptors of the tiles' first K=16 slices; the others add a
      // constant to the start-address field (16-byte units, low word). All
      // of them share the high word.
      const uint64_t dq0 = sdesc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t dkv_k = sdesc_sw128(smem_u32(sKV), 16, 1024);
      const uint64_t dkv_v = sdesc_sw128(smem_u32(sKV), kHalfBytes, 1024);
      const uint32_t hi = static_cast<uint32_t>(dq0 >> 32);
      const uint32_t q_lo = static_cast<uint32_t>(dq0), k_lo = static_cast<uint32_t>(dkv_k),
                     v_lo = static_cast<uint32_t>(dkv_v);
      auto issue_qk = [&](int qb, int t, int slot) {
        const uint32_t qd = q_lo + static_cast<uint32_t>((qb * kQTiles + t) * (kTileBytes >> 4));
        const uint32_t kd = k_lo + static_cast<uint32_t>(slot * (kTileBytes >> 4));
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = static_cast<uint32_t>(((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4);
          umma_ss_elect_lo(tmem + t * 128, qd + off, kd + off, hi, idesc_s, kk > 0);
        }
      };
      auto issue_pv = [&](int t, int slot, bool acc) {
        const uint32_t vd = v_lo + static_cast<uint32_t>(slot * (kTileBytes >> 4));
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ts_elect_lo(tmem + 256 + t * 128, tmem + t * 128 + kk * 8, vd + static_cast<uint32_t>(kk * (2048 >> 4)),
                           hi, idesc_o, (acc || kk > 0) ? 1u : 0u);
      };
      bool ok = true;
      int nq = 0;   // items with key tiles so far (Q buffer use)
      int ig = 0;   // K/V ring position
      int sp = 0;   // S/P phases so far (per tile)
      for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
        const Item x = item_of(it);
        if (x.n_tiles == 0) continue;
        const int qb = nq % kQBuf;
        // Self-attention: the softmax warps rotate Q in shared memory first.
        ok = warp_wait(kRope ? &bar_q_ready[qb] : &bar_q_full[qb], (nq / kQBuf) & 1, abort, a.lc.err, to);
        if (!ok) break;
        const int k0 = ig % kStages;
        ok = warp_wait(&bar_kv_full[k0], (ig / kStages) & 1, abort, a.lc.err, to);
        if (!ok) break;
        tc_fence_after();
        issue_qk(qb, 0, k0);
        umma_commit_elect(&bar_s_full[0]);
        issue_qk(qb, 1, k0);
        umma_commit_elect(&bar_s_full[1]);
        umma_commit_elect(&bar_kv_empty[k0]);
        for (int j = 0; j < x.n_tiles && ok; ++j) {
          const int iv = ig + 2 * j + 1;
          const int vslot = iv % kStages;
          ok = warp_wait(&bar_kv_full[vslot], (iv / kStages) & 1, abort, a.lc.err, to);
          const bool has_next = j + 1 < x.n_tiles;
          const int ik = ig + 2 * j + 2;
          const int kslot = ik % kStages;
          if (ok && has_next) ok = warp_wait(&bar_kv_full[kslot], (ik / kStages) & 1, abort, a.lc.err, to);
          for (int t = 0; t < kQTiles && ok; ++t) {
            ok = warp_wait(&bar_p_full[t], (sp + j) & 1, abort, a.lc.err, to);
            if (!ok) break;
            tc_fence_after();
            issue_pv(t, vslot, j > 0);
            if (t == kQTiles - 1) umma_commit_elect(&bar_kv_empty[vslot]);
            if (!has_next) {
              umma_commit_elect(&bar_o_full[t]);
            } else {
              issue_qk(qb, t, kslot);
              umma_commit_elect(&bar_s_full[t]);
              if (t == kQTiles - 1) umma_commit_elect(&bar_kv_empty[kslot]);
            }
          }
        }
        ig += 2 * x.n_tiles;
        sp += x.n_tiles;
        ++nq;
      }
      // Every MMA of this CTA must be done before TMEM is released.
      umma_commit_elect(&bar_drain);
      mbar_wait(&bar_drain, 0, nullptr, to);
    }
   } else if (warp == kStoreWarp) {
    // ------------------------------------------------------------ O store
    // Writes each staged O tile with two TMA tensor stores and, once both
    // tiles' stores have read the staging area, hands the Q buffer back to
    // the Q producer. The softmax warps go on to their next item as soon as
    // their tile is staged. Rows past the end of the sequence fall outside
    // the tensor map and are not written.
    if (lane == 0) {
      int nq = 0;
      for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
        const Item x = item_of(it);
        if (x.n_tiles == 0) continue;
        const int qb = nq % kQBuf;
        bool ok = true;
        for (int t = 0; t < kQTiles && ok; ++t) {
          ok = mbar_wait(&bar_o_staged[qb][t], (nq / kQBuf) & 1, abort, to);
          if (ok && store_ok[qb][t]) {
            uint8_t* stage = sQ + (qb * kQTiles + t) * kTileBytes;
            tma_store_4d(&tm_o, stage, 0, x.h, x.q0 + t * kBlockM, x.b);
            tma_store_4d(&tm_o, stage + kHalfBytes, 64, x.h, x.q0 + t * kBlockM, x.b);
            bulk_commit_group();
          }
        }
        if (!ok) {
          raise_abort(abort, a.lc.err);
          break;
        }
        bulk_wait_group_read0();
        mbar_arrive(&bar_q_empty[qb]);
        ++nq;
      }
      bulk_wait_group0();
    }
    __syncwarp();
   }
  } else {
    regs_grow<kSoftmaxRegs>();
    // ------------------------------------------------------------ softmax
    const int t = warp >> 2;
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + lane_addr + t * 128;
    const uint32_t tO = tmem + lane_addr + 256 + t * 128;
    const float sl2 = a.scale_log2;
    // After a failed wait (ok = false) the warp skips all work but keeps
    // walking the items, so that the four warps of a tile always execute
    // the same sequence of named barriers.
    bool ok = true;
    int nq = 0;  // items with key tiles so far
    int sp = 0;  // S/P phases so far
    for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
      // Only the key-tile counts stay live through the softmax loop; the
      // output addresses are recomputed for the epilogue.
      int n_valid, n_tiles, kv_start;
      {
        const Item x = item_of(it);
        n_valid = x.n_valid;
        n_tiles = x.n_tiles;
        kv_start = x.kv_start;
      }
      if (n_tiles == 0) {  // no valid key: O = 0, LSE = -inf (a merge leaves o / lse as they are)
        if (kMerge != kMergeNone) continue;
        const Item x = item_of(it);
        const int row = x.q0 + t * kBlockM + r;
        if (row < a.Lq) {
          uint4* dst = reinterpret_cast<uint4*>(a.o + ((static_cast<size_t>(x.b) * a.Lq + row) * a.H + x.h) * kHeadDim);
          for (int c = 0; c < 16; ++c) dst[c] = make_uint4(0, 0, 0, 0);
          if (a.lse) a.lse[(static_cast<size_t>(x.b) * a.H + x.h) * a.Lq + row] = -INFINITY;
        }
        continue;
      }
      const int qb = nq % kQBuf;
      if (kRope) {
        if (ok) ok = warp_wait(&bar_q_full[qb], (nq / kQBuf) & 1, abort, a.lc.err, to);
        const int row = item_of(it).q0 + t * kBlockM + r;
        if (ok && row < a.Lq) rope_row_in_smem(sQ + (qb * kQTiles + t) * kTileBytes, r, row, a);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_q_ready[qb]);
      }

      float m_ref = -INFINITY;
      float l = 0.f;
      for (int j = 0; j < n_tiles && ok; ++j) {
        ok = warp_wait(&bar_s_full[t], (sp + j) & 1, abort, a.lc.err, to);
        if (!ok) break;
        tc_fence_after();
        uint32_t sr[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, sr[c]);
        tmem_ld_wait_regs(sr);
#define WAN_S(e) __uint_as_float(sr[(e) >> 5][(e) & 31])
        const int jt = j + kv_start < n_tiles ? j + kv_start : j + kv_start - n_tiles;
        const int valid = n_valid - jt * kBlockN;
        if (valid < kBlockN) {
#pragma unroll
          for (int i = 0; i < 128; ++i)
            if (i >= valid) sr[i >> 5][i & 31] = __float_as_uint(-INFINITY);
        }
        // Reference maximum. The item's first key tile sets m_ref to its row
        // maximum; later tiles are exponentiated against m_ref without taking
        // their own maximum. A tile whose row sum of P stays <= kTileSumBound
        // has every P <= kTileSumBound, so O and l stay well inside fp32; a
        // row whose sum exceeds it (its maximum grew by about 2^8 or more)
        // moves m_ref to the tile's maximum, rescales O and l, and the tile
        // is recomputed. The result is the same softmax for any m_ref.
        auto row_max = [&]() {
          float mc[4];  // four independent chains of three-input maxima
#pragma unroll
          for (int q = 0; q < 4; ++q) mc[q] = WAN_S(q);
#pragma unroll
          for (int i = 4; i < 128; i += 8) {
#pragma unroll
            for (int q = 0; q < 4; ++q)
              mc[q] = max3f(mc[q], WAN_S(i + 2 * q), WAN_S(i + 2 * q + 1));
          }
          return max3f(mc[0], mc[1], fmaxf(mc[2], mc[3]));
        };
        if (j == 0) m_ref = row_max();
        float lsum = 0.f;
#pragma unroll 1
        for (int pass = 0; pass < 2; ++pass) {
          // p = 2^(s * scale * log2(e) - m * scale * log2(e)), two lanes per f32x2 op.
          const float neg = -m_ref * sl2;
          const uint64_t sl2x2 = f2_pack(sl2, sl2);
          const uint64_t negx2 = f2_pack(neg, neg);
          uint64_t acc[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int e = c * 32 + 2 * i;
              const uint64_t xx = f2_fma(f2_pack(WAN_S(e), WAN_S(e + 1)), sl2x2, negx2);
              float x0, x1;
              f2_unpack(xx, x0, x1);
              const float p0 = ex2_approx(x0);
              const float p1 = ex2_approx(x1);
              const uint64_t pp = f2_pack(p0, p1);
              acc[i & 1] = f2_add(acc[i & 1], pp);
              pk[i] = pack_bf16x2(p0, p1);
            }
            tmem_st16(tS + c * 16, pk);
          }
          float a0, a1, a2, a3;
          f2_unpack(acc[0], a0, a1);
          f2_unpack(acc[1], a2, a3);
          lsum = (a0 + a1) + (a2 + a3);
          const bool need = !(lsum <= kTileSumBound);
          if (pass == 1 || !__any_sync(0xffffffffu, need)) break;
          // Rare path: new reference for the rows that need one (alpha = 1
          // for the others), O and l rescaled, then the tile again.
          const float m_new = need ? fmaxf(m_ref, row_max()) : m_ref;
          const float alpha = ex2_approx((m_ref - m_new) * sl2);
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
        l += lsum;
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_p_full[t]);
      }

      // ---------------------------------------------------------- epilogue
      // O_t is normalised into bf16 and staged in this tile's Q buffer (no
      // MMA reads it once O_t is final) in the 128-byte swizzled layout; the
      // store warp writes it out and hands the buffer back to the Q
      // producer. The four warps of the tile agree on stopping before the
      // named barrier.
      if (ok) ok = warp_wait(&bar_o_full[t], nq & 1, abort, a.lc.err, to);
      if (lane == 0) epi_ok[t][wq] = ok ? 1 : 0;
      named_bar_sync(1 + t, 128);
      const bool all_ok = epi_ok[t][0] & epi_ok[t][1] & epi_ok[t][2] & epi_ok[t][3];
      ok = ok && all_ok;
      const Item x = item_of(it);
      uint8_t* stage = sQ + (qb * kQTiles + t) * kTileBytes;
      if (all_ok) {
        tc_fence_after();
        const int row = x.q0 + t * kBlockM + r;
        float inv = 1.0f / l;
        const float lse_new = (m_ref * sl2 + __log2f(l)) * 0.69314718055994531f;  // natural log
        // Merging epilogues first bring the previous O tile into the staging
        // area (same swizzled layout as the store); rows past the end read 0.
        float w_old = 0.f;
        float lse_out = lse_new;
        if (kMerge != kMergeNone) {
          if (wq == 0 && lane == 0) {
            mbar_arrive_expect_tx(&bar_oldo[t], kTileBytes);
            tma_load_4d(stage, &tm_o, &bar_oldo[t], 0, x.h, x.q0 + t * kBlockM, x.b);
            tma_load_4d(stage + kHalfBytes, &tm_o, &bar_oldo[t], 64, x.h, x.q0 + t * kBlockM, x.b);
          }
          if (kMerge == kMergeLse && row < a.Lq) {
            // O = (e^lse_old O_old + e^lse_new O_new) / (e^lse_old + e^lse_new)
            const float lse_old = a.lse[(static_cast<size_t>(x.b) * a.H + x.h) * a.Lq + row];
            const float mx = fmaxf(lse_old, lse_new);
            const float eo = lse_old == -INFINITY ? 0.f : __expf(lse_old - mx);
            const float en = __expf(lse_new - mx);
            lse_out = mx + __logf(eo + en);
            w_old = eo / (eo + en);
            inv *= en / (eo + en);
          } else if (kMerge == kMergeAdd) {
            w_old = 1.f;
          }
          // Every warp of the tile waits for the copy (the TMA write of the
          // staging area happens-before the reads below).
          ok = warp_wait(&bar_oldo[t], nq & 1, abort, a.lc.err, to) && ok;
        }
        // O_t is read out of TMEM here; the next item's first PV overwrites it
        // only after this warp signals that item's first P (program order).
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t ov[32];
          tmem_ld32(tO + c * 32, ov);
          tmem_ld_wait_regs(ov);
#pragma unroll
          for (int q = 0; q < 4; ++q) {  // 16-byte chunk 4c+q of the row: half c/2, chunk (4c+q)%8
            const int chunk = 4 * c + q;
            uint4* dst = reinterpret_cast<uint4*>(stage + (chunk >> 3) * kHalfBytes + sw128_offset(r, chunk & 7));
            float vals[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) vals[i] = __uint_as_float(ov[8 * q + i]) * inv;
            if (kMerge != kMergeNone) {
              const uint4 old = *dst;
              const uint32_t ow[4] = {old.x, old.y, old.z, old.w};
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                vals[2 * i] = fmaf(w_old, __uint_as_float(ow[i] << 16), vals[2 * i]);
                vals[2 * i + 1] = fmaf(w_old, __uint_as_float(ow[i] & 0xFFFF0000u), vals[2 * i + 1]);
              }
            }
            *dst = make_uint4(pack_bf16x2(vals[0], vals[1]), pack_bf16x2(vals[2], vals[3]), pack_bf16x2(vals[4], vals[5]),
                              pack_bf16x2(vals[6], vals[7]));
          }
        }
        if (a.lse && row < a.Lq && kMerge != kMergeAdd)
          a.lse[(static_cast<size_t>(x.b) * a.H + x.h) * a.Lq + row] = lse_out;
        fence_proxy_async_smem();
      }
      // The store warp writes the staged tile out (store_ok[qb][t] is next
      // written for the item after the store warp has released buffer qb).
      if (wq == 0 && lane == 0) store_ok[qb][t] = all_ok ? 1 : 0;
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_o_staged[qb][t]);
      sp += n_tiles;
      ++nq;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

int launch_attn_fwd(const void* q, const void* k_rot, const void* v, void* o, float* lse, int B, int Lq, int Lk,
                    int H, wan_grid_t g, RopeTables tab, bool rope, const int32_t* kv_lens, float scale,
                    const LaunchCommon& lc, cudaStream_t s, int q_pos0, int merge) {
  CUtensorMap tq, tk, tv, to;
  if (!make_tmap_bld(&tq, q, B, Lq, H, kHeadDim, 128)) return WAN_ERR_CUDA;
  if (!make_tmap_bld(&to, o, B, Lq, H, kHeadDim, 128)) return WAN_ERR_CUDA;
  if (!make_tmap_bld(&tk, k_rot, B, Lk, H, kHeadDim, 128)) return WAN_ERR_CUDA;
  if (!make_tmap_bld(&tv, v, B, Lk, H, kHeadDim, 128)) return WAN_ERR_CUDA;
  FwdArgs a;
  a.o = static_cast<__nv_bfloat16*>(o);
  a.lse = lse;
  a.kv_lens = kv_lens;
  a.tab = tab;
  a.Lq = Lq;
  a.Lk = Lk;
  a.H = H;
  a.B = B;
  a.Hp = g.Hp;
  a.Wp = g.Wp;
  a.n_qpairs = (Lq + kBlockM * kQTiles - 1) / (kBlockM * kQTiles);
  a.q_pos0 = q_pos0;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.lc = lc;
  const long long n_items = static_cast<long long>(a.n_qpairs) * H * B;
  if (n_items > INT_MAX) return WAN_ERR_INVALID;
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return WAN_ERR_CUDA;
  const int grid = static_cast<int>(n_items < sms ? n_items : sms);  // persistent: one CTA per SM
  // Instantiations: self-attention (plain / Ring-step merge) and cross-
  // attention (plain / added second path).
  void (*kern)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const CUtensorMap, const FwdArgs) = nullptr;
  if (rope && merge == kMergeNone) kern = attn_fwd_kernel<true, kMergeNone>;
  if (rope && merge == kMergeLse) kern = attn_fwd_kernel<true, kMergeLse>;
  if (!rope && merge == kMergeNone) kern = attn_fwd_kernel<false, kMergeNone>;
  if (!rope && merge == kMergeAdd) kern = attn_fwd_kernel<false, kMergeAdd>;
  if (kern == nullptr) return WAN_ERR_INVALID;
  const int smem_bytes = rope ? FwdCfg<true>::kSmemBytes : FwdCfg<false>::kSmemBytes;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes) != cudaSuccess)
    return WAN_ERR_CUDA;
  record_start(lc, s);
  kern<<<grid, kThreads, smem_bytes, s>>>(tq, tk, tv, to, a);
  record_stop(lc, s);
  return cudaGetLastError() == cudaSuccess ? WAN_OK : WAN_ERR_CUDA;
}

}  // namespace wan
