// 3D RoPE rotation of a bf16 [B, L, H, 128] tensor (an HBM-bound pass).
//
// gojay.top "Wan2.1" paper reading, 费曼一分钟 / DiT 块: Q and K carry 3D RoPE
// with separate temporal, height and width bands. Pairs (2j, 2j+1) of a band
// turn by the band's angle for the token's coordinate on that axis; the
// angles come from the caller's fp32 {cos, sin} tables.
//
// One thread handles one 16-byte chunk (8 elements = 4 rotary pairs); a warp
// covers 512 contiguous bytes, so loads and stores are fully coalesced. The
// grid is a multiple of the SM count and strides over the tensor.
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
template <bool kInverse>
__global__ void __launch_bounds__(256) rope_rotate_kernel(const uint4* x, uint4* y,
                                                          long long n_chunks, int H, int Hp, int Wp, int L,
                                                          int pos0, RopeTables tab) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n_chunks; i += stride) {
    const int c = (int)(i & 15);          // chunk within the 128-wide head
    const long long rowhead = i >> 4;     // (b*L + l)*H + h
    const long long bl = rowhead / H;     // b*L + l
    const int l = (int)(bl % L) + pos0;
    const int w = l % Wp;
    const int hh = (l / Wp) % Hp;
    const int t = l / (Wp * Hp);
    uint4 v = x[i];
    uint32_t wd[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 cs = rope_cs(tab, c * 4 + k, t, hh, w);
      const float sn = kInverse ? -cs.y : cs.y;
      const float a = __uint_as_float(wd[k] << 16);
      const float b = __uint_as_float(wd[k] & 0xFFFF0000u);
      wd[k] = pack_bf16x2(a * cs.x - b * sn, a * sn + b * cs.x);
    }
    y[i] = make_uint4(wd[0], wd[1], wd[2], wd[3]);
  }
}

// dQ path of the backward: fp32 [B, L, H, 128] -> R(pos)^T x -> bf16.
// One thread per 8 elements (two 16-byte fp32 loads, one 16-byte bf16 store).
__global__ void __launch_bounds__(256) rope_unrotate_f32_kernel(const float4* x, uint4* y, long long n_chunks, int H,
                                                                int Hp, int Wp, int L, RopeTables tab) {
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n_chunks; i += stride) {
    const int c = (int)(i & 15);
    const long long bl = (i >> 4) / H;
    const int l = (int)(bl % L);
    const int w = l % Wp;
    const int hh = (l / Wp) % Hp;
    const int t = l / (Wp * Hp);
    const float4 u0 = x[2 * i];
    const float4 u1 = x[2 * i + 1];
    const float v[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
    uint32_t wd[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 cs = rope_cs(tab, c * 4 + k, t, hh, w);
      const float a = v[2 * k], b = v[2 * k + 1];
      wd[k] = pack_bf16x2(a * cs.x + b * cs.y, b * cs.x - a * cs.y);
    }
    y[i] = make_uint4(wd[0], wd[1], wd[2], wd[3]);
  }
}

cudaError_t launch_rope_unrotate_f32(const float* x, void* y, int B, wan_grid_t g, int H, RopeTables tab,
                                     cudaStream_t s) {
  const int L = g.F * g.Hp * g.Wp;
  const long long n_chunks = (long long)B * L * H * (kHeadDim / 8);
  if (n_chunks == 0) return cudaSuccess;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  long long want = (n_chunks + 255) / 256;
  long long cap = (long long)sms * 8;
  const int blocks = (int)(want < cap ? want : cap);
  rope_unrotate_f32_kernel<<<blocks, 256, 0, s>>>((const float4*)x, (uint4*)y, n_chunks, H, g.Hp, g.Wp, L, tab);
  return cudaGetLastError();
}

cudaError_t launch_rope_rotate_bf16(const void* x, void* y, int B, wan_grid_t g, int H, RopeTables tab,
                                    bool inverse, cudaStream_t s) {
  return launch_rope_rotate_bf16_rows(x, y, B, g.F * g.Hp * g.Wp, 0, g, H, tab, inverse, s);
}

cudaError_t launch_rope_rotate_bf16_rows(const void* x, void* y, int B, int L, int pos0, wan_grid_t g, int H,
                                         RopeTables tab, bool inverse, cudaStream_t s) {
  const long long n_chunks = (long long)B * L * H * (kHeadDim / 8);
  if (n_chunks == 0) return cudaSuccess;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  long long want = (n_chunks + 255) / 256;
  long long cap = (long long)sms * 8;  // 8 resident blocks of 256 threads per SM
  const int blocks = (int)(want < cap ? want : cap);
  if (inverse)
    rope_rotate_kernel<true><<<blocks, 256, 0, s>>>((const uint4*)x, (uint4*)y, n_chunks, H, g.Hp, g.Wp, L, pos0,
                                                     tab);
  else
    rope_rotate_kernel<false><<<blocks, 256, 0, s>>>((const uint4*)x, (uint4*)y, n_chunks, H, g.Hp, g.Wp, L, pos0,
                                                      tab);
  return cudaGetLastError();
}

}  // namespace wan
