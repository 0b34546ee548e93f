// 3D RoPE rotation of a bf16 [B, L, H, 128] tensor (an HBM-bound pass).
//
// gojay.top "Wan2.1" paper reading, 费曼一分钟 / DiT 块: Q and K carry 3D RoPE
// with separate temporal, height and width bands. Pairs (2j, 2j+1) of a band
// turn by the band's angle for the token's coordinate on that axis; the
// angles come from the caller's fp32 {cos, sin} tables.
//
// Loads and stores are 16-byte chunks (8 elements = 4 rotary pairs); the
// threads of a block cover contiguous bytes, so they are fully coalesced.
// The grids are multiples of the SM count and stride over the tensor.
#include "common.cuh"
#include "kernels.cuh"

namespace wan {

__device__ __forceinline__ float2 rope_cs(const RopeTables& tab, int pair, int t, int h, int w) {
  if (pair < kPairsT) return tab.t[t * kPairsT + pair];
  if (pair < kPairsT + kPairsH) return tab.h[h * kPairsH + (pair - kPairsT)];
  return tab.w[w * kPairsW + (pair - kPairsT - kPairsH)];
}

// x holds L consecutive tokens per batch item, the first one being token
// pos0 of the grid (pos0 > 0 for a chunk of a longer sequence).
//
// A block of 128 threads takes 8 tokens per step of a grid-stride loop, 16
// threads per token: thread c rotates the 16-byte chunk c (four rotary pairs)
// of every head of its token. The token's grid coordinates and the chunk's
// four {cos, sin} pairs are worked out once and serve all H heads; the 16
// threads of a token read and write 256 contiguous bytes per head, and up to
// kHeadsPerPass heads are loaded before the first is used.
template <bool kInverse>
__global__ void __launch_bounds__(128) rope_rotate_kernel(const uint4* x, uint4* y, long long n_tokens, int H,
                                                          int Hp, int Wp, int L, int pos0, RopeTables tab) {
  constexpr int kHeadsPerPass = 8;
  const int c = threadIdx.x & 15;
  int band[4], j[4], row[4];
  const float2* base[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int pair = c * 4 + k;
    band[k] = pair < kPairsT ? 0 : (pair < kPairsT + kPairsH ? 1 : 2);
    j[k] = band[k] == 0 ? pair : (band[k] == 1 ? pair - kPairsT : pair - kPairsT - kPairsH);
    row[k] = band[k] == 0 ? kPairsT : (band[k] == 1 ? kPairsH : kPairsW);
    base[k] = band[k] == 0 ? tab.t : (band[k] == 1 ? tab.h : tab.w);
  }
  for (long long tok = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 4); tok < n_tokens;
       tok += static_cast<long long>(gridDim.x) * 8) {
    const int l = static_cast<int>(tok % L) + pos0;
    const int w = l % Wp;
    const int hh = (l / Wp) % Hp;
    const int t = l / (Wp * Hp);
    float2 cs[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int pos = band[k] == 0 ? t : (band[k] == 1 ? hh : w);
      cs[k] = base[k][pos * row[k] + j[k]];
      if (kInverse) cs[k].y = -cs[k].y;
    }
    const size_t tok_chunk = static_cast<size_t>(tok) * H * 16 + c;
    for (int h0 = 0; h0 < H; h0 += kHeadsPerPass) {
      uint4 v[kHeadsPerPass];
#pragma unroll
      for (int u = 0; u < kHeadsPerPass; ++u)
        if (h0 + u < H) v[u] = x[tok_chunk + static_cast<size_t>(h0 + u) * 16];
#pragma unroll
      for (int u = 0; u < kHeadsPerPass; ++u) {
        if (h0 + u >= H) break;
        uint32_t wd[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float a = __uint_as_float(wd[k] << 16);
          const float b = __uint_as_float(wd[k] & 0xFFFF0000u);
          wd[k] = pack_bf16x2(a * cs[k].x - b * cs[k].y, a * cs[k].y + b * cs[k].x);
        }
        y[tok_chunk + static_cast<size_t>(h0 + u) * 16] = make_uint4(wd[0], wd[1], wd[2], wd[3]);
      }
    }
  }
}

// dQ path of the backward: fp32 [B, L, H, 128] -> R(pos)^T x -> bf16. A
// block of 128 threads takes 8 tokens per step of a grid-stride loop, 16
// threads per token: thread c rotates the 32-byte fp32 chunk c (8 elements)
// of every head of its token and writes 16 bytes per head. The token's grid
// coordinates and the chunk's four {cos, sin} pairs are worked out once and
// serve all H heads, and the 16 threads of a token read 512 contiguous bytes
// per head.
__global__ void __launch_bounds__(128) rope_unrotate_f32_kernel(const float4* x, uint4* y, long long n_tokens, int H,
                                                                int Hp, int Wp, int L, RopeTables tab) {
  constexpr int kHeadsPerPass = 4;
  const int c = threadIdx.x & 15;
  for (long long tok = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 4); tok < n_tokens;
       tok += static_cast<long long>(gridDim.x) * 8) {
    const int l = static_cast<int>(tok % L);
    const int w = l % Wp;
    const int hh = (l / Wp) % Hp;
    const int t = l / (Wp * Hp);
    float2 cs[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) cs[k] = rope_cs(tab, c * 4 + k, t, hh, w);
    const size_t tok_chunk = static_cast<size_t>(tok) * H * 16 + c;
    for (int h0 = 0; h0 < H; h0 += kHeadsPerPass) {
      float4 u0[kHeadsPerPass], u1[kHeadsPerPass];
#pragma unroll
      for (int u = 0; u < kHeadsPerPass; ++u)
        if (h0 + u < H) {
          const size_t i = tok_chunk + static_cast<size_t>(h0 + u) * 16;
          u0[u] = x[2 * i];
          u1[u] = x[2 * i + 1];
        }
#pragma unroll
      for (int u = 0; u < kHeadsPerPass; ++u) {
        if (h0 + u >= H) break;
        const float v[8] = {u0[u].x, u0[u].y, u0[u].z, u0[u].w, u1[u].x, u1[u].y, u1[u].z, u1[u].w};
        uint32_t wd[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float a = v[2 * k], b = v[2 * k + 1];
          wd[k] = pack_bf16x2(a * cs[k].x + b * cs[k].y, b * cs[k].x - a * cs[k].y);
        }
        y[tok_chunk + static_cast<size_t>(h0 + u) * 16] = make_uint4(wd[0], wd[1], wd[2], wd[3]);
      }
    }
  }
}

cudaError_t launch_rope_unrotate_f32(const float* x, void* y, int B, wan_grid_t g, int H, RopeTables tab,
                                     cudaStream_t s) {
  const int L = g.F * g.Hp * g.Wp;
  const long long n_tokens = (long long)B * L;
  if (n_tokens == 0 || H == 0) return cudaSuccess;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long cap = (long long)sms * 16;  // 16 resident blocks of 128 threads per SM
  const long long need = (n_tokens + 7) / 8;  // 8 tokens per block and step
  const int blocks = (int)(need < cap ? need : cap);
  rope_unrotate_f32_kernel<<<blocks, 128, 0, s>>>((const float4*)x, (uint4*)y, n_tokens, H, g.Hp, g.Wp, L, tab);
  return cudaGetLastError();
}

cudaError_t launch_rope_rotate_bf16(const void* x, void* y, int B, wan_grid_t g, int H, RopeTables tab,
                                    bool inverse, cudaStream_t s) {
  return launch_rope_rotate_bf16_rows(x, y, B, g.F * g.Hp * g.Wp, 0, g, H, tab, inverse, s);
}

cudaError_t launch_rope_rotate_bf16_rows(const void* x, void* y, int B, int L, int pos0, wan_grid_t g, int H,
                                         RopeTables tab, bool inverse, cudaStream_t s) {
  const long long n_tokens = (long long)B * L;
  if (n_tokens == 0 || H == 0) return cudaSuccess;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long cap = (long long)sms * 16;  // 16 resident blocks of 128 threads per SM
  const long long need = (n_tokens + 7) / 8;  // 8 tokens per block and step
  const int blocks = (int)(need < cap ? need : cap);
  const uint4* xs = static_cast<const uint4*>(x);
  uint4* ys = static_cast<uint4*>(y);
  if (inverse)
    rope_rotate_kernel<true><<<blocks, 128, 0, s>>>(xs, ys, n_tokens, H, g.Hp, g.Wp, L, pos0, tab);
  else
    rope_rotate_kernel<false><<<blocks, 128, 0, s>>>(xs, ys, n_tokens, H, g.Hp, g.Wp, L, pos0, tab);
  return cudaGetLastError();
}

}  // namespace wan
