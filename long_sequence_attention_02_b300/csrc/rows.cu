// Row pass of the attention backward (an HBM-bound pass): per (b, h) and
// query row i, D_i = dO_i . O_i and LSE_i * log2(e), into rows padded to a
// multiple of 128 (pad: D = 0, LSE = +inf, so padded queries get P = 0 in
// the backward kernel). The backward of attention needs D because
// dS = P o (dP - D) (the gradient of the softmax; gojay.top "Wan2.1"
// reading, section 3 Training, is the training step it serves).
#include "common.cuh"
#include "kernels.cuh"

namespace wan {

namespace {

// D_i = sum_d dO_id O_id and LSE_i * log2(e) into rows padded to a multiple
// of 128 (pad: D = 0, LSE = +inf). A block takes 32 consecutive tokens of one
// batch item (all H heads: 32 * H * 256 contiguous bytes of O and of dO) per
// step of a grid-stride loop. Its threads walk those bytes in 16-byte chunks,
// 16 lanes per (token, head) row, reduce each row with shuffles and leave
// the sums in shared memory; then D and LSE * log2 e go out along the token
// axis, so that the [B*H][Lpad] rows are read and written 128 bytes at a
// time rather than one float per row.
//
// The pass is short on instructions per byte: with all heads in one pass
// (H <= kRowsMaxH, every Wan shape) chunk q of the tile is simply chunk q of
// the tile's contiguous bytes and row q / 16 of its sums, so the loop does
// no division.
constexpr int kRowsTok = 32;
constexpr int kRowsMaxH = 64;  // heads per block tile held in shared memory (larger H: several passes)
__global__ void __launch_bounds__(256) bwd_rows_kernel(const uint4* o, const uint4* dout, const float* lse,
                                                       float* lse2, float* drow, int B, int L, int Lpad, int H) {
  __shared__ float dsum[kRowsTok * kRowsMaxH];  // [token][head of this pass]
  constexpr int kUnroll = 4;
  const int tiles_l = (L + kRowsTok - 1) / kRowsTok;
  const int c = threadIdx.x & 15;
  // A row's 16 chunks are 16 aligned lanes that enter and leave the loop together.
  const unsigned group = 0xFFFFu << (threadIdx.x & 16);
  for (long long tile = blockIdx.x; tile < (long long)B * tiles_l; tile += gridDim.x) {
    const int b = static_cast<int>(tile / tiles_l);
    const int l0 = static_cast<int>(tile % tiles_l) * kRowsTok;
    const int n_tok = L - l0 < kRowsTok ? L - l0 : kRowsTok;
    for (int h0 = 0; h0 < H; h0 += kRowsMaxH) {
      const int nh = H - h0 < kRowsMaxH ? H - h0 : kRowsMaxH;
      const bool whole = nh == H;  // the tile's rows are contiguous: row r of the pass is row r of the tile
      const size_t base = (static_cast<size_t>(b) * L + l0) * H * 16;
      const int n = n_tok * nh * 16;  // chunks of this pass
      for (int q0 = threadIdx.x; q0 < n; q0 += kUnroll * 256) {
        uint4 xo[kUnroll], yo[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int q = q0 + u * 256;
          if (q < n) {
            const int rh = q >> 4;  // (token, head) of this pass
            const size_t i = whole ? base + q
                                   : ((static_cast<size_t>(b) * L + l0 + rh / nh) * H + h0 + rh % nh) * 16 + c;
            xo[u] = o[i];
            yo[u] = dout[i];
          }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int q = q0 + u * 256;
          if (q >= n) break;
          const uint32_t xa[4] = {xo[u].x, xo[u].y, xo[u].z, xo[u].w}, ya[4] = {yo[u].x, yo[u].y, yo[u].z, yo[u].w};
          float acc = 0.f;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            acc = fmaf(__uint_as_float(xa[k] << 16), __uint_as_float(ya[k] << 16), acc);
            acc = fmaf(__uint_as_float(xa[k] & 0xFFFF0000u), __uint_as_float(ya[k] & 0xFFFF0000u), acc);
          }
#pragma unroll
          for (int m = 8; m >= 1; m >>= 1) acc += __shfl_xor_sync(group, acc, m, 16);
          if (c == 0) dsum[q >> 4] = acc;
        }
      }
      __syncthreads();
      for (int e = threadIdx.x; e < nh * kRowsTok; e += 256) {
        const int hh = e / kRowsTok, t = e % kRowsTok;
        if (t < n_tok) {
          const size_t bh = static_cast<size_t>(b) * H + h0 + hh;
          drow[bh * Lpad + l0 + t] = dsum[t * nh + hh];
          lse2[bh * Lpad + l0 + t] = lse[bh * L + l0 + t] * 1.4426950408889634f;
        }
      }
      __syncthreads();
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

}  // namespace

cudaError_t launch_bwd_rows(const void* o, const void* dout, const float* lse, float* lse2, float* drow, int B, int L,
                            int Lpad, int H, cudaStream_t s) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long tiles = (long long)B * ((L + kRowsTok - 1) / kRowsTok), cap = (long long)sms * 8;
  if (tiles > 0)
    bwd_rows_kernel<<<(int)(tiles < cap ? tiles : cap), 256, 0, s>>>(static_cast<const uint4*>(o),
                                                                     static_cast<const uint4*>(dout), lse, lse2, drow,
                                                                     B, L, Lpad, H);
  if (Lpad > L) bwd_pad_kernel<<<sms, 256, 0, s>>>(lse2, drow, B * H, L, Lpad);
  return cudaGetLastError();
}

}  // namespace wan
