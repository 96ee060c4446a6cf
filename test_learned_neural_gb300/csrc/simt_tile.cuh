// Register-tiled fp32 GEMM tile shared by the SIMT kernels.
#pragma once
#include "atlas_common.cuh"

namespace atlas {

// Block-wide 64x64 output tile of C = A * B with operand strides, 256 threads,
// each a 4x4 micro-tile; K streamed through shared memory in steps of 16.
struct TileOp {
  const float* p;
  long is, ks;  // element (i, k) at p[i * is + k * ks]
};

__device__ inline void tile_gemm(TileOp A, TileOp Bt, int M, int N, int K, int i0, int j0, float acc[4][4],
                          float* As, float* Bs) {
  // As[16][64] holds A(i0.., k0..), Bs[16][64] holds B(k0.., j0..), Bt(j, k) = B(k, j)
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  for (int a = 0; a < 4; ++a)
    for (int b = 0; b < 4; ++b) acc[a][b] = 0.f;
  for (int k0 = 0; k0 < K; k0 += 16) {
    for (int l = threadIdx.x; l < 16 * 64; l += blockDim.x) {
      const int kk = l / 64, ii = l % 64;
      const int gi = i0 + ii, gk = k0 + kk, gj = j0 + ii;
      As[kk * 64 + ii] = (gi < M && gk < K) ? A.p[gi * A.is + gk * A.ks] : 0.f;
      Bs[kk * 64 + ii] = (gj < N && gk < K) ? Bt.p[gj * Bt.is + gk * Bt.ks] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      float av[4], bv[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) av[a] = As[kk * 64 + ty * 4 + a];
#pragma unroll
      for (int b = 0; b < 4; ++b) bv[b] = Bs[kk * 64 + tx * 4 + b];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) acc[a][b] += av[a] * bv[b];
    }
    __syncthreads();
  }
}

}  // namespace atlas
